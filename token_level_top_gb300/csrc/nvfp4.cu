// nvfp4.cu -- expert GEMMs with 4-bit weights and activations (NVFP4):
// e2m1 values, one e4m3 scale per 16 consecutive elements of a row, one fp32
// scale per row.
//
// The pages quantise expert weights to 4-6 bits to move fewer bytes ([2kiu]
// §5.1) and warn that a dequantisation pass can eat the gain ([cnnetsun]
// §3.2).  Here the 4-bit codes go straight into the tensor cores:
// tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X multiplies packed e2m1
// tiles (K = 64 per instruction, 32 bytes of a 128-byte shared-memory row)
// and applies the e4m3 block scales itself; the epilogue applies the two row
// scales, as in the e4m3 path.
//
// Quantisation of a row x[0..n) (the weights once, token and activation rows
// on the fly), in fp32 steps:
//   scale = max|x| / 2688 (6 * 448: the largest e2m1 magnitude times the
//   largest e4m3 one; 1 for an all-zero row); for each block of 16,
//   b = e4m3(fl(fl(max|x_i| / scale) / 6)), den = fl(value(b) * scale),
//   code_i = e2m1(fl(x_i / den)) (round to nearest even, saturating), or 0
//   when den = 0.  Codes are packed two per byte, element 2m in the low
//   nibble; block scales are bytes, rows of them padded to 16 bytes.
//
// GEMM kernel: one persistent CTA per SM, 14 warps -- warp 0 TMA producer
// (per stage the block scales, 16 bytes a row, first and on a barrier of their
// own, then the codes of 128 rows x 256 values of A and of up to 256 rows of
// B), warp 1 allocates TMEM and issues
// the MMAs (M = 128, N = the tile width, up to 256), warps 2-5 and 10-13 the
// epilogue (two warps per lane quarter, each with half of the tile's columns),
// warps 6-9 copy each stage's block scales from shared memory into TMEM
// (tcgen05.st) as soon as they land, while the codes are still in flight, and
// arrive on the barrier the MMA thread waits on besides the codes': for each MMA, column i of lane l (in each of the four 32-lane
// quarters) holds the four scale bytes of row l + 32i of A (4 columns) and of
// B (N/32 columns, rounded up to 4; byte b: the scale of the MMA's b-th block
// of 16 along K).  Tiles of up to 128 columns have two TMEM accumulators
// (the epilogue of one tile overlaps the next tile's MMAs), wider tiles one.
// The W13 weights of this path are packed in 128-row blocks (64 W1 rows,
// then the 64 matching W3 rows), so that each 128 columns of a gate-up tile
// hold matching gate and up columns.  Every wait is bounded.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "quotient.cuh"

namespace moe {
namespace {

constexpr int kF4Threads = 448;   // 14 warps
constexpr int kF4MaxBN = 256;     // widest N tile
constexpr int kF4AccCols = 256;            // TMEM columns of the accumulator(s)
constexpr int kF4SfCol = kF4AccCols;       // first TMEM column of the block scales
constexpr int kF4MaxStages = 8;

// Rows of B a stage holds (128, or 256 for tiles wider than 128 columns).
__host__ __device__ constexpr int f4_b_alloc(int bn) { return bn <= 128 ? 128 : 256; }
// Bytes of one stage: A codes (a_rows rows of 128 bytes: 256 e2m1 values), B
// codes, A scales, B scales (16 bytes a row); a multiple of 1024.
__host__ __device__ constexpr uint32_t f4_stage_bytes(int a_rows, int bn)
{
    return (static_cast<uint32_t>(a_rows) * 144u + static_cast<uint32_t>(f4_b_alloc(bn)) * 144u + 1023u) / 1024u * 1024u;
}
// TMEM columns of the scales of one MMA's B rows: N/32 rounded up to 4.
__host__ __device__ constexpr int f4_sfb_cols(int bn) { return ((bn + 31) / 32 + 3) / 4 * 4; }
// TMEM columns of one stage's scales: 4 per MMA for A, f4_sfb_cols for B, 4 MMAs.
__host__ __device__ constexpr int f4_sf_stage_cols(int bn) { return 16 + 4 * f4_sfb_cols(bn); }

// ---------------------------------------------------------------- e2m1 codes
// Eight floats to eight e2m1 codes (round to nearest even, saturating),
// element 0 in the low nibble of the low byte.
__device__ __forceinline__ uint32_t e2m1x8(const float (&x)[8])
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]));
    return r;
}

// e4m3 code of a non-negative float (round to nearest even, saturating), and its value.
__device__ __forceinline__ uint32_t e4m3_code(float v)
{
    uint16_t two;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(two) : "f"(0.0f), "f"(v));
    return two & 0xFFu;
}

__device__ __forceinline__ float e4m3_value(uint32_t b)
{
    const uint32_t e = (b >> 3) & 15, m = b & 7;
    const float v = e == 0 ? static_cast<float>(m) * 0.001953125f   // m / 8 * 2^-6
                           : __uint_as_float(((e + 120u) << 23) | (m << 20));
    return (b & 0x80u) ? -v : v;
}

__device__ __forceinline__ void bf16x8(const uint4 v, float (&x)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[j]));
        x[2 * j] = f.x;
        x[2 * j + 1] = f.y;
    }
}

// Source row of output row r: the token rows of the kept slots (perm), the
// W13 re-packing into 128-row blocks (w13_F > 0: output block j of an expert
// holds W1 rows 64j.. and W3 rows 64j.. of the 256-row packed layout), or r.
__device__ __forceinline__ long long source_row(long long r, const int32_t* perm, int k, int w13_F)
{
    if (perm) return perm[r] / k;
    if (w13_F > 0) {
        const long long e = r / (2 * w13_F);
        const int l = static_cast<int>(r - e * 2 * w13_F);
        const int j = l / 128, w = l % 128;
        const int src = w < 64 ? 64 * j + w : 64 * j + (w - 64);   // row of W1 or of W3
        const int base = (src / 128) * 256 + (w < 64 ? 0 : 128) + src % 128;
        return e * 2 * w13_F + base;
    }
    return r;
}

constexpr int kQThreads = 256;
constexpr int kQMaxGroups = 4;   // 16-element groups per thread: rows up to 256 * 4 * 16 = 16384

// Threads per row (a power of two, 8..256): the fewest that hold the row's groups
// at up to kQMaxGroups each; a block of kQThreads quantises kQThreads / tpr rows.
int quant_threads_per_row(int cols)
{
    const int ng = cols / 16;
    int tpr = 8;
    while (tpr < kQThreads && tpr * kQMaxGroups < ng) tpr *= 2;
    return tpr;
}

// Each row's groups of 16 stay in registers; the row max is reduced over the
// row's threads (or given by amax_in), then each group is quantised.
__global__ void __launch_bounds__(kQThreads, 4) quantize_nvfp4_kernel(
    long long rows, int cols, int tpr, const uint4* __restrict__ w, const int32_t* __restrict__ perm, int k,
    int w13_F, const int32_t* __restrict__ nrows, const float* __restrict__ amax_in, uint2* __restrict__ codes,
    uint8_t* __restrict__ bscale, int sf_stride, float* __restrict__ scales, float* __restrict__ zero_rows)
{
    __shared__ float s_wmax[kQThreads / 32];
    const int lt = static_cast<int>(threadIdx.x) & (tpr - 1);   // thread within the row
    const long long row = static_cast<long long>(blockIdx.x) * (kQThreads / tpr) + threadIdx.x / tpr;
    const bool active = row < rows && !(nrows && row >= *nrows);
    const int ng = cols / 16;
    uint4 v[2 * kQMaxGroups];
    float gmax[kQMaxGroups];
    float amax = 0.0f;
    if (active) {
        const uint4* wr = w + source_row(row, perm, k, w13_F) * (cols / 8);
#pragma unroll
        for (int i = 0; i < kQMaxGroups; ++i) {
            const int g = lt + tpr * i;
            gmax[i] = 0.0f;
            if (g < ng) {
                v[2 * i] = __ldg(wr + 2 * g);
                v[2 * i + 1] = __ldg(wr + 2 * g + 1);
                float x[8];
                bf16x8(v[2 * i], x);
#pragma unroll
                for (int j = 0; j < 8; ++j) gmax[i] = fmaxf(gmax[i], fabsf(x[j]));
                bf16x8(v[2 * i + 1], x);
#pragma unroll
                for (int j = 0; j < 8; ++j) gmax[i] = fmaxf(gmax[i], fabsf(x[j]));
                amax = fmaxf(amax, gmax[i]);
            }
        }
    }
    if (amax_in) {
        if (active) amax = amax_in[row];
    } else {
        // over the row's lanes of this warp, then (rows wider than a warp) its warps
        for (int off = min(tpr, 32) / 2; off >= 1; off >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (tpr > 32) {
            if ((threadIdx.x & 31) == 0) s_wmax[threadIdx.x >> 5] = amax;
            __syncthreads();
            const int w0 = static_cast<int>(threadIdx.x / tpr) * (tpr / 32);
            for (int i = 0; i < tpr / 32; ++i) amax = fmaxf(amax, s_wmax[w0 + i]);
        }
    }
    if (!active) return;
    const float sc = amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
    if (lt == 0) {
        scales[row] = sc;
        if (zero_rows) zero_rows[row] = 0.0f;
    }
    uint2* cr = codes + row * (cols / 16);
    uint8_t* br = bscale + row * sf_stride;
#pragma unroll
    for (int i = 0; i < kQMaxGroups; ++i) {
        const int g = lt + tpr * i;
        if (g >= ng) continue;
        const uint32_t b = e4m3_code(__fdiv_rn(__fdiv_rn(gmax[i], sc), 6.0f));
        const float den = __fmul_rn(e4m3_value(b), sc);
        float x0[8], x1[8];
        bf16x8(v[2 * i], x0);
        bf16x8(v[2 * i + 1], x1);
        uint2 c = make_uint2(0u, 0u);
        if (den >= kFmaDivMin) {   // den and 1/den normal: the FMA quotient
            const float y = __frcp_rn(den);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                x0[j] = div_by(x0[j], den, y);
                x1[j] = div_by(x1[j], den, y);
            }
            c = make_uint2(e2m1x8(x0), e2m1x8(x1));
        } else if (den > 0.0f) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                x0[j] = __fdiv_rn(x0[j], den);
                x1[j] = __fdiv_rn(x1[j], den);
            }
            c = make_uint2(e2m1x8(x0), e2m1x8(x1));
        }
        cr[g] = c;
        br[g] = static_cast<uint8_t>(b);
    }
    // the padding of the scale row (never read as a scale: the tensor map ends at ng)
    for (int i = ng + lt; i < sf_stride; i += tpr) br[i] = 0;
}

// ---------------------------------------------------------------- the GEMM
struct F4Params {
    int kind, E, T, topk, d, F;
    int kb_total;   // K / 256 (stages of 128-byte rows), rounded up
    int bn;         // N tile: 256 (128 where N is not a multiple of 256); the down GEMM
                    // with one row tile per expert 64..256 (a multiple of 16)
    int a_rows;     // rows of A a stage has room for: 128, or 32 when every tile's rows fit 32
    int b_rows;     // rows of B a stage holds (f4_b_alloc(bn))
    uint32_t stage_bytes;
    int n_tiles;    // N tiles per expert
    int stages;
    int b_policy;   // 1: weight loads evict_first (every expert holds at most one row tile)
    const float* a_scale;   // per A row (slot order)
    const float* b_scale;   // per weight row
    float* act_amax;
    const int32_t* offsets;
    __nv_bfloat16* act;
    __nv_bfloat16* y_slots;
    int* status;
    long long budget;
};

// silu(x) = x sigmoid(x) = (x/2)(1 + tanh(x/2)), with the hardware tanh
// approximation: one MUFU operation instead of an exponential and a reciprocal
// (the epilogue of a 256-column gate-up tile is on the critical path: the next
// tile's MMAs wait for it); its error stays inside the bf16 rounding of the
// activation that follows.  Finite for every finite x (tanh saturates at +-1).
__device__ __forceinline__ float silu_f4(float x)
{
    float t;
    const float h = 0.5f * x;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return h * (1.0f + t);
}

// Named barrier 1 among the eight epilogue warps (256 threads); f4_epi_all also
// returns whether `pred` holds in all of them.
__device__ __forceinline__ void f4_epi_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool f4_epi_all(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}

// 16 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// 16 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
        "%13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
        "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D (+)= A . B^T with e2m1 A and B (K = 64), each 16-value block of A's rows and
// B's rows scaled by its e4m3 scale from TMEM.
__device__ __forceinline__ void mma_nvfp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}\n" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of kind::mxf4nvf4: e2m1 A and B (format 1), both
// K-major, e4m3 block scales (scale type 0), scale-factor ids 0, M x N.
__host__ __device__ constexpr uint32_t idesc_nvfp4(int M, int N)
{
    return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

struct F4Tile {
    int e, m, n;
};

__device__ __forceinline__ F4Tile f4_decode(const F4Params& p, int tile, const int* s_start, const int* s_offs)
{
    int lo = 0, hi = p.E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_start[mid] <= tile)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int mt = (s_offs[lo + 1] - s_offs[lo] + kBM - 1) / kBM;
    const int local = tile - s_start[lo];
    F4Tile t;
    t.e = lo;
    t.m = local % mt;   // row tiles fastest: they share the weight tile
    t.n = local / mt;
    return t;
}

// tmA / tmSA: the A codes and block scales in boxes of 128 rows; tmA32 / tmSA32
// the same in boxes of 32 rows, for tiles whose expert has at most 32 rows there
// (decode): the MMA still spans 128 rows, the rows past the box hold stale data
// and their results are not stored.  tmB / tmSB: boxes of bn weight rows.
__global__ void __launch_bounds__(kF4Threads, 1)
    moe_gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                          const __grid_constant__ CUtensorMap tmA32, const __grid_constant__ CUtensorMap tmSA32,
                          const F4Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int stages = p.stages;
    const uint32_t sb = p.stage_bytes;
    const uint32_t a_bytes = static_cast<uint32_t>(p.a_rows) * 128u;                 // A codes
    const uint32_t off_sfa = a_bytes + static_cast<uint32_t>(p.b_rows) * 128u;         // A scales
    const uint32_t off_sfb = off_sfa + static_cast<uint32_t>(p.a_rows) * 16u;          // B scales
    const int nacc = p.bn <= 128 ? 2 : 1;           // TMEM accumulators
    const int sfb_cols = f4_sfb_cols(p.bn);          // TMEM scale columns of one MMA's B rows
    const int sf_cols = f4_sf_stage_cols(p.bn);      // TMEM scale columns of one stage
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(stages) * sb);
    uint64_t* full_bar = bars;                 // the stage's codes (A and B) have landed
    uint64_t* empty_bar = bars + stages;
    uint64_t* sf_bar = bars + 2 * stages;      // the stage's block scales are in TMEM
    uint64_t* sfull_bar = bars + 3 * stages;   // the stage's block scales have landed
    uint64_t* tfull_bar = bars + 4 * stages;
    uint64_t* tempty_bar = bars + 4 * stages + 2;
    int* s_start = reinterpret_cast<int*>(bars + 4 * stages + 4);
    int* s_offs = s_start + (p.E + 1);
    volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(s_offs + (p.E + 1));
    float* s_bsc = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(s_tmem + 1) + 15) & ~uintptr_t(15));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSA);
        tma_prefetch_desc(&tmSB);
        tma_prefetch_desc(&tmA32);
        tma_prefetch_desc(&tmSA32);
        for (int i = 0; i < stages; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&sfull_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), 1);
            mbar_init(smem_u32(&sf_bar[i]), 4);   // the four scale-copying warps
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull_bar[b]), 1);
            mbar_init(smem_u32(&tempty_bar[b]), 8);   // the eight epilogue warps
        }
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(s_tmem)), 512);
        tmem_relinquish();
    }
    if (warp == 2) {
        int carry = 0;
        for (int base = 0; base <= p.E; base += 32) {
            const int e = base + lane;
            int o = 0, o1 = 0;
            if (e <= p.E) o = p.offsets[e];
            if (e < p.E) o1 = p.offsets[e + 1];
            if (e <= p.E) s_offs[e] = o;
            const int tiles = (e < p.E) ? (o1 - o + kBM - 1) / kBM * p.n_tiles : 0;
            int incl = tiles;
            for (int off = 1; off < 32; off <<= 1) {
                const int vv = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += vv;
            }
            if (e <= p.E) s_start[e] = carry + incl - tiles;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int total = s_start[p.E];
    const uint32_t idesc = idesc_nvfp4(kBM, p.bn);
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;
        const uint64_t pol_b = l2_policy_evict_first();
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            const F4Tile t = f4_decode(p, tile, s_start, s_offs);
            const int arow = s_offs[t.e] + t.m * kBM;
            const int brow = (p.kind == GK_GATEUP ? t.e * 2 * p.F : t.e * p.d) + t.n * p.bn;
            // the tile's rows fit a 32-row box (always so when the stages have room for 32)
            const bool few = p.a_rows == 32 || s_offs[t.e + 1] - arow <= 32;
            const uint32_t rows = (few ? 32u : 128u) + static_cast<uint32_t>(p.bn);   // A and B rows per stage
            for (int kb = 0; kb < p.kb_total; ++kb) {
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, p.budget))) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    // the block scales first, on their own barrier: the scale warps copy
                    // them into TMEM while the codes are still in flight
                    const uint32_t sfb = smem_u32(&sfull_bar[stage]);
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    uint8_t* st = smem + static_cast<size_t>(stage) * sb;
                    mbar_arrive_expect_tx(sfb, rows * 16u);
                    tma_load_2d(smem_u32(st + off_sfa), few ? &tmSA32 : &tmSA, kb * 16, arow, sfb);
                    if (p.b_policy)
                        tma_load_2d_hint(smem_u32(st + off_sfb), &tmSB, kb * 16, brow, sfb, pol_b);
                    else
                        tma_load_2d(smem_u32(st + off_sfb), &tmSB, kb * 16, brow, sfb);
                    mbar_arrive_expect_tx(fb, rows * 128u);
                    tma_load_2d(smem_u32(st), few ? &tmA32 : &tmA, kb * 128, arow, fb);
                    if (p.b_policy)
                        tma_load_2d_hint(smem_u32(st + a_bytes), &tmB, kb * 128, brow, fb, pol_b);
                    else
                        tma_load_2d(smem_u32(st + a_bytes), &tmB, kb * 128, brow, fb);
                }
                __syncwarp();
                issued_mask |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        if (!ok) {
            record_error(p.status, MOE_ERR_TIMEOUT);
            for (int s = 0; s < stages; ++s)
                if (issued_mask & (1u << s)) {
                    mbar_wait(smem_u32(&sfull_bar[s]), (issued_parity >> s) & 1, p.budget);
                    mbar_wait(smem_u32(&full_bar[s]), (issued_parity >> s) & 1, p.budget);
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int it = 0, last_b = -1;
            uint32_t last_par = 0;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
                const int b = it % nacc;
                const uint32_t acc_par = static_cast<uint32_t>(it / nacc) & 1u;
                if (!mbar_wait(smem_u32(&tempty_bar[b]), acc_par ^ 1, p.budget)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * 128);
                for (int kb = 0; kb < p.kb_total; ++kb) {
                    if (!mbar_wait(smem_u32(&full_bar[stage]), phase, p.budget) ||
                        !mbar_wait(smem_u32(&sf_bar[stage]), phase, p.budget)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(smem + static_cast<size_t>(stage) * sb);
                    const uint32_t b0 = a0 + a_bytes;   // (A rows past a_rows read B's bytes: not stored)
                    const uint32_t sf0 = tmem_base + static_cast<uint32_t>(kF4SfCol + sf_cols * stage);
#pragma unroll
                    for (int j = 0; j < 4; ++j)   // K = 64 per instruction: 32 bytes of each row
                        mma_nvfp4(d_tmem, sdesc_k_sw128(a0 + 32 * j), sdesc_k_sw128(b0 + 32 * j), idesc,
                                  sf0 + 4 * j, sf0 + 16 + sfb_cols * j, (kb > 0 || j > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&empty_bar[stage]));
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit(smem_u32(&tfull_bar[b]));
                last_b = b;
                last_par = acc_par;
            }
            if (!ok) record_error(p.status, MOE_ERR_TIMEOUT);
            if (last_b >= 0) mbar_wait(smem_u32(&tfull_bar[last_b]), last_par, p.budget);
        }
        __syncwarp();
    } else if (warp >= 6 && warp < 10) {
        // ------------------------------------------------------------ block scales into TMEM
        const int q = warp & 3;   // the TMEM lane quarter this warp may access
        int stage = 0;
        uint32_t phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            for (int kb = 0; kb < p.kb_total; ++kb) {
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sfull_bar[stage]), phase, p.budget))) {
                    record_error(p.status, MOE_ERR_TIMEOUT);
                    tile = total;
                    break;
                }
                // MMA j's scales: column 4j + i of lane 32q + l holds the four scale bytes
                // (word j) of A row l + 32i; column 16 + sfb_cols * j + i those of B row
                // l + 32i; the same in each of the four lane quarters
                const uint8_t* st = smem + static_cast<size_t>(stage) * sb;
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(kF4SfCol + sf_cols * stage);
                {
                    uint4 w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) w[i] = *reinterpret_cast<const uint4*>(st + off_sfa + (lane + 32 * i) * 16);
                    const uint32_t r[16] = {w[0].x, w[1].x, w[2].x, w[3].x, w[0].y, w[1].y, w[2].y, w[3].y,
                                            w[0].z, w[1].z, w[2].z, w[3].z, w[0].w, w[1].w, w[2].w, w[3].w};
                    tmem_st16(taddr, r);
                }
                if (sfb_cols == 4) {
                    uint4 w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) w[i] = *reinterpret_cast<const uint4*>(st + off_sfb + (lane + 32 * i) * 16);
                    const uint32_t r[16] = {w[0].x, w[1].x, w[2].x, w[3].x, w[0].y, w[1].y, w[2].y, w[3].y,
                                            w[0].z, w[1].z, w[2].z, w[3].z, w[0].w, w[1].w, w[2].w, w[3].w};
                    tmem_st16(taddr + 16, r);
                } else {   // 8 columns per MMA: rows l + 32i, i < 8 (the stage holds 256 rows)
                    uint4 w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) w[i] = *reinterpret_cast<const uint4*>(st + off_sfb + (lane + 32 * i) * 16);
                    uint32_t r[32];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        r[i] = w[i].x;
                        r[8 + i] = w[i].y;
                        r[16 + i] = w[i].z;
                        r[24 + i] = w[i].w;
                    }
                    tmem_st32(taddr + 16, r);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sf_bar[stage]));
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                    // TMEM lane quarter
        const int row = q * 32 + lane;
        const int eh = warp >= 10 ? 1 : 0;         // which half of the columns
        const int et = eh * 128 + (static_cast<int>(threadIdx.x) & 127);   // 0..255 over the eight warps
        int it = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
            const F4Tile t = f4_decode(p, tile, s_start, s_offs);
            const int b = it % nacc;
            const uint32_t acc_par = static_cast<uint32_t>(it / nacc) & 1u;
            // the tile's weight-row scales while its MMAs run; columns past the
            // expert's weight rows (the down GEMM's last tile) read no scale
            f4_epi_sync();
            {
                const int wrows = p.kind == GK_GATEUP ? 2 * p.F : p.d;
                const int col = t.n * p.bn + et;
                s_bsc[et] = (et < p.bn && col < wrows) ? __ldg(p.b_scale + static_cast<long long>(t.e) * wrows + col)
                                                       : 0.0f;
            }
            const bool got = f4_epi_all(mbar_wait(smem_u32(&tfull_bar[b]), acc_par, p.budget));
            if (!got) {
                record_error(p.status, MOE_ERR_TIMEOUT);
                break;
            }
            tc_fence_after();
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * 128);
            const int off = s_offs[t.e];
            const int cnt = s_offs[t.e + 1] - off;
            const int ri = t.m * kBM + row;
            const bool valid = ri < cnt;
            const float asc = valid ? p.a_scale[off + ri] : 0.0f;
            uint32_t v[32], u[32];
            if (p.kind == GK_GATEUP) {
                // each 128 columns: [0, 64) gate, [64, 128) the matching up columns;
                // this warp takes 32 of the 64 pairs
                __nv_bfloat16* dst = p.act + static_cast<size_t>(off + ri) * p.F + t.n * (p.bn / 2);
                float rmax = 0.0f;
                for (int h = 0; h < p.bn; h += 128) {
                    const int c = 32 * eh;
                    tmem_ld32(taddr + h + c, v);
                    tmem_ld32(taddr + h + 64 + c, u);
                    tmem_ld_wait2(v, u);
                    if (valid) {
                        const float* bg = s_bsc + h + c;
                        const float* bu = s_bsc + h + 64 + c;
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float g0 = __uint_as_float(v[2 * j]) * asc * bg[2 * j];
                            const float g1 = __uint_as_float(v[2 * j + 1]) * asc * bg[2 * j + 1];
                            const float u0 = __uint_as_float(u[2 * j]) * asc * bu[2 * j];
                            const float u1 = __uint_as_float(u[2 * j + 1]) * asc * bu[2 * j + 1];
                            const float a0 = silu_f4(g0) * u0, a1 = silu_f4(g1) * u1;
                            pk[j] = pack_bf16x2(a0, a1);
                            rmax = fmaxf(rmax, fmaxf(fabsf(a0), fabsf(a1)));
                        }
                        uint4* d4 = reinterpret_cast<uint4*>(dst + h / 2 + c);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            d4[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    }
                }
                if (valid && p.act_amax)
                    atomicMax(reinterpret_cast<unsigned int*>(p.act_amax + off + ri),
                              __float_as_uint(__bfloat162float(__float2bfloat16_rn(rmax))));
            } else {
                // 32-column pieces alternate between the two halves of the epilogue
                const int col0 = t.n * p.bn;
                const int ncols = min(p.bn, p.d - col0);   // a multiple of 16
                __nv_bfloat16* dst = p.y_slots + static_cast<size_t>(off + ri) * p.d + col0;
                for (int c = 32 * eh; c < ncols; c += 64) {
                    const int w = min(32, ncols - c);       // 32, or 16 for the last piece
                    if (w == 32)
                        tmem_ld32(taddr + c, v);
                    else
                        tmem_ld16(taddr + c, v);
                    tmem_ld_wait(v);
                    if (valid) {
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]) * asc * s_bsc[c + 2 * j],
                                                __uint_as_float(v[2 * j + 1]) * asc * s_bsc[c + 2 * j + 1]);
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (4 * j < w / 2) d4[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[b]));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// Byte matrix [rows, cols] (cols bytes a row, `stride` bytes apart), boxes of
// box_rows x box_cols bytes, 128-byte swizzle when the box is 128 bytes wide.
bool make_byte_map(CUtensorMap* tm, const void* ptr, uint64_t rows, uint64_t cols, uint64_t stride,
                   uint32_t box_rows, uint32_t box_cols)
{
    static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    if (!enc) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return false;
        enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {stride};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estride[2] = {1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE,
               box_cols == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// N tile of a launch: 256 columns (two 128-row blocks of the gate-up's
// packing; for the down GEMM the last tile of an expert may be partly past its
// rows), else 128.  Measured on the Mixtral-shaped prefill (4096 tokens, top-2):
// 256-wide tiles with one accumulator beat 128-wide tiles with two (the second
// accumulator hides the epilogue, the wider tile halves the reads of A per
// output column and a stage carries twice the MMA work per byte of A).
int f4_tile_width(int N) { return N % 256 == 0 ? 256 : 128; }

}  // namespace

int nvfp4_sf_stride(int cols) { return (cols / 16 + 15) / 16 * 16; }

cudaError_t launch_quantize_nvfp4(long long rows, int cols, const void* w, const int32_t* perm, int k,
                                  int w13_F, const int32_t* nrows, const float* amax_in, void* codes,
                                  void* bscale, float* scales, float* zero_rows, cudaStream_t s)
{
    if (rows <= 0) return cudaSuccess;
    if (cols % 32 != 0 || cols > kQThreads * kQMaxGroups * 16) return cudaErrorInvalidValue;
    const int tpr = quant_threads_per_row(cols);
    const long long blocks = (rows + kQThreads / tpr - 1) / (kQThreads / tpr);
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    quantize_nvfp4_kernel<<<static_cast<unsigned>(blocks), kQThreads, 0, s>>>(
        rows, cols, tpr, static_cast<const uint4*>(w), perm, k, w13_F, nrows, amax_in, static_cast<uint2*>(codes),
        static_cast<uint8_t*>(bscale), nvfp4_sf_stride(cols), scales, zero_rows);
    return cudaGetLastError();
}

cudaError_t launch_gemm_nvfp4(const F4Launch& g, cudaStream_t s)
{
    F4Params p{};
    p.kind = g.kind;
    p.E = g.E;
    p.T = g.T;
    p.topk = g.topk;
    p.d = g.d;
    p.F = g.F;
    p.a_scale = g.a_scale;
    p.b_scale = g.b_scale;
    p.act_amax = g.act_amax;
    p.offsets = g.offsets;
    p.act = static_cast<__nv_bfloat16*>(g.act);
    p.y_slots = static_cast<__nv_bfloat16*>(g.y_slots);
    p.status = g.status;
    p.budget = g.budget;
    const int K = g.kind == GK_GATEUP ? g.d : g.F;       // reduction length
    const int N = g.kind == GK_GATEUP ? 2 * g.F : g.d;   // weight rows of one expert
    if (K % 32 != 0 || N % 128 != 0) return cudaErrorInvalidValue;
    const int sms = num_sms();
    p.kb_total = (K + 255) / 256;
    // When no expert holds more than one row tile, each weight tile is read by one
    // tile only: its loads go first out of L2, and the down GEMM's column tile (a
    // multiple of 16, 64..256) is the one that needs the fewest passes over the
    // SMs times its width.
    const bool one_tile = g.rows_cap > 0 && std::min<long long>(g.rows_cap, static_cast<long long>(g.T)) <= kBM;
    p.b_policy = one_tile ? 1 : 0;
    p.bn = f4_tile_width(N);
    if (one_tile && g.kind != GK_GATEUP) {
        const long long mt = std::min<long long>(g.E, static_cast<long long>(g.T) * g.topk);
        long long best = -1;
        for (int bn = kF4MaxBN; bn >= 64; bn -= 16) {
            const long long cost = (mt * ((N + bn - 1) / bn) + sms - 1) / sms * bn;
            if (best < 0 || cost < best) {
                best = cost;
                p.bn = bn;
            }
        }
    }
    if (g.kind == GK_GATEUP && N % p.bn != 0) return cudaErrorInvalidValue;
    // with at most 32 rows per expert every tile loads a 32-row A box: the stages
    // keep room for 32 rows only, which leaves room for more stages
    p.a_rows = (one_tile && std::min<long long>(g.rows_cap, static_cast<long long>(g.T)) <= 32) ? 32 : 128;
    p.b_rows = f4_b_alloc(p.bn);
    p.stage_bytes = f4_stage_bytes(p.a_rows, p.bn);
    p.n_tiles = (N + p.bn - 1) / p.bn;
    const uint64_t arows = static_cast<uint64_t>(g.T) * g.topk;
    const uint64_t brows = static_cast<uint64_t>(g.E) * N;
    CUtensorMap tmA, tmB, tmSA, tmSB, tmA32, tmSA32;
    const int sfs = nvfp4_sf_stride(K);
    if (!make_byte_map(&tmA, g.a_codes, arows, K / 2, K / 2, kBM, 128) ||
        !make_byte_map(&tmB, g.b_codes, brows, K / 2, K / 2, p.bn, 128) ||
        !make_byte_map(&tmSA, g.a_sf, arows, K / 16, sfs, kBM, 16) ||
        !make_byte_map(&tmSB, g.b_sf, brows, K / 16, sfs, p.bn, 16) ||
        !make_byte_map(&tmA32, g.a_codes, arows, K / 2, K / 2, 32, 128) ||
        !make_byte_map(&tmSA32, g.a_sf, arows, K / 16, sfs, 32, 16))
        return cudaErrorInvalidValue;
    // shared memory: the stages (each with its four barriers), the two accumulator
    // barriers, the tile starts and offsets, the TMEM address, the weight-row scales
    const size_t fixed = 1024 + 64 + static_cast<size_t>(2 * (g.E + 1)) * 4 + 16 + 16 + 4 * kF4MaxBN;
    const int by_smem = static_cast<int>((227 * 1024 - fixed) / (p.stage_bytes + 32));
    const int by_tmem = (512 - kF4SfCol) / f4_sf_stage_cols(p.bn);
    const int stages = std::min(kF4MaxStages, std::min(by_smem, by_tmem));
    if (stages < 2) return cudaErrorInvalidValue;
    p.stages = stages;
    const size_t smem = fixed + static_cast<size_t>(stages) * (p.stage_bytes + 32);
    const cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(moe_gemm_nvfp4_kernel), 227 * 1024);
    if (e != cudaSuccess) return e;
    const long long mt_max = (static_cast<long long>(g.T) * g.topk + kBM - 1) / kBM + g.E;
    const int grid = static_cast<int>(std::min<long long>(mt_max * p.n_tiles, sms));
    if (grid <= 0) return cudaSuccess;
    moe_gemm_nvfp4_kernel<<<grid, kF4Threads, smem, s>>>(tmA, tmB, tmSA, tmSB, tmA32, tmSA32, p);
    return cudaGetLastError();
}

}  // namespace moe
