// bwd_gemm.cu -- the four per-expert products of the layer's backward pass on
// the tensor cores (tcgen05/TMEM, TMA-fed), over each expert's kept rows.
//
// The backward differentiates the expert FFN y = W2 (silu(W1 x) * W3 x) of
// "GPT-4稀疏激活真相…" §3.1 and the weighted combine of §4.3 for the routing
// the forward made.  With the kept rows of expert e stacked in a row block
// (bf16, padded with zero rows to a multiple of 128; see backward.cu):
//
//   BG_DGRAD   out[rows, N] = A[rows, K] . W_e[K, N]        (fp32 out)
//              dL/da = dL/dout . W2_e  (K = d, N = F)
//              dL/dx = (dg, du) . W13_e (K = 2F, N = d)
//   BG_WGRAD   out_e[Mw, N] = A_e[rows, Mw]^T . B_e[rows, N]  (fp32 out, K = the rows)
//              dW2_e  = dL/dout_e^T . (cw a)_e   (Mw = d, N = F)
//              dW13_e = (dg, du)_e^T . x_e       (Mw = 2F, N = d)
//
// Operands: the row blocks are K-major for BG_DGRAD's A (a row holds K
// contiguous values, loaded as 128-row x 64-column TMA boxes, as in the
// forward); the weights W_e[K, N] and both operands of BG_WGRAD are
// MN-major: a row of the stored matrix is one K index holding the M or N
// values contiguously.  Those are loaded as boxes of 64 K-rows x 64 M/N
// values (128 bytes, 128-byte swizzle) and described to tcgen05.mma as
// MN-major operands: 64-value blocks along M/N 8192 bytes apart (the
// descriptor's leading offset), groups of 8 K-rows 1024 bytes apart (its
// stride offset), instruction-descriptor bits 15 / 16 set for A / B.
//
// Same structure as the forward GEMM (gemm.cu): one persistent CTA per SM,
// 6 warps -- TMA producer, MMA issuer (one thread, M = 128, N = 256, K = 16
// per instruction, two TMEM accumulators), four epilogue warps that drain
// TMEM and store fp32 rows.  The tile table is built on the device from the
// forward's per-expert offsets; an expert with no kept rows gets zero weight
// gradients without MMAs.  Every wait is bounded.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kBN = 256;   // output tile columns
constexpr uint32_t kBoxBytes = 64 * 64 * 2;   // one 64 x 64 bf16 box

struct BwdGemmParams {
    int mode, E;
    int kb;          // BG_DGRAD: K / 64
    int wrows;       // BG_DGRAD: rows of one expert's weight matrix in the B map (= K)
    int N;           // output columns
    int n_tiles;     // ceil(N / 256)
    int Mw;          // BG_WGRAD: output rows per expert
    int m_tiles;     // BG_WGRAD: ceil(Mw / 128)
    int stages;
    const int32_t* offsets;   // [E + 1] the forward's kept slots per expert
    float* out;
    int* status;
    long long budget;
};

// MN-major operand, 128-byte swizzle: [0,14) start >> 4, [16,30) leading
// offset >> 4 = 8192 (the next 64-value block along M or N), [32,46) stride
// offset >> 4 = 1024 (the next 8 K-rows), [46,48) version 1, [61,64) swizzle 2.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(kBoxBytes >> 4) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

struct BTile {
    int e, m, n;
    int row0;   // BG_DGRAD: first padded row of the tile; BG_WGRAD: first padded row of expert e
    int nk;     // K blocks of 64
};

__device__ __forceinline__ BTile decode(const BwdGemmParams& p, int tile, const int* s_start, const int* s_poff,
                                        const int* s_offs)
{
    int lo = 0, hi = p.E - 1;   // largest e with s_start[e] <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_start[mid] <= tile)
            lo = mid;
        else
            hi = mid - 1;
    }
    BTile t;
    t.e = lo;
    const int local = tile - s_start[lo];
    if (p.mode == BG_DGRAD) {
        const int mt = (s_poff[lo + 1] - s_poff[lo]) / kBM;
        t.m = local % mt;
        t.n = local / mt;
        t.row0 = s_poff[lo] + t.m * kBM;
        t.nk = p.kb;
    } else {
        t.m = local % p.m_tiles;
        t.n = local / p.m_tiles;
        t.row0 = s_poff[lo];
        t.nk = (s_offs[lo + 1] - s_offs[lo] + 63) / 64;
    }
    return t;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_bwd_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const BwdGemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int stages = p.stages;
    constexpr uint32_t a_bytes = kBM * 64 * 2;    // 16 KB: 128 x 64 (K-major) or 2 boxes (MN-major)
    constexpr uint32_t b_bytes = kBN * 64 * 2;    // 32 KB: 4 boxes of 64 K-rows x 64 columns
    uint8_t* sA = smem;
    uint8_t* sB = sA + stages * a_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + stages * b_bytes);
    uint64_t* full_bar = bars;
    uint64_t* empty_bar = bars + stages;
    uint64_t* tfull_bar = bars + 2 * stages;
    uint64_t* tempty_bar = bars + 2 * stages + 2;
    int* s_start = reinterpret_cast<int*>(bars + 2 * stages + 4);
    int* s_poff = s_start + (p.E + 1);
    int* s_offs = s_poff + (p.E + 1);
    volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(s_offs + (p.E + 1));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        for (int i = 0; i < stages; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull_bar[b]), 1);
            mbar_init(smem_u32(&tempty_bar[b]), 4);
        }
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(s_tmem)), 2 * kBN);
        tmem_relinquish();
    }
    if (warp == 2) {
        // padded row offsets (each expert's kept rows rounded up to 128) and the
        // tile table: tiles of expert e start at s_start[e]
        int carry_rows = 0, carry_tiles = 0;
        for (int base = 0; base <= p.E; base += 32) {
            const int e = base + lane;
            int o = 0, o1 = 0;
            if (e <= p.E) o = p.offsets[e];
            if (e < p.E) o1 = p.offsets[e + 1];
            if (e <= p.E) s_offs[e] = o;
            const int prow = (e < p.E) ? (o1 - o + kBM - 1) / kBM * kBM : 0;
            int tiles = 0;
            if (e < p.E) tiles = (p.mode == BG_DGRAD ? prow / kBM : p.m_tiles) * p.n_tiles;
            int ir = prow, it = tiles;
            for (int off = 1; off < 32; off <<= 1) {
                const int vr = __shfl_up_sync(0xffffffffu, ir, off);
                const int vt = __shfl_up_sync(0xffffffffu, it, off);
                if (lane >= off) {
                    ir += vr;
                    it += vt;
                }
            }
            if (e <= p.E) {
                s_poff[e] = carry_rows + ir - prow;
                s_start[e] = carry_tiles + it - tiles;
            }
            carry_rows += __shfl_sync(0xffffffffu, ir, 31);
            carry_tiles += __shfl_sync(0xffffffffu, it, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int total = s_start[p.E];
    const bool a_mn = p.mode == BG_WGRAD;
    const uint32_t idesc = idesc_bf16_f32(kBM, kBN) | (a_mn ? (1u << 15) : 0u) | (1u << 16);
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            const BTile t = decode(p, tile, s_start, s_poff, s_offs);
            for (int kb = 0; kb < t.nk; ++kb) {
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, p.budget))) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    mbar_arrive_expect_tx(fb, a_bytes + b_bytes);
                    const uint32_t dA = smem_u32(sA + stage * a_bytes);
                    const uint32_t dB = smem_u32(sB + stage * b_bytes);
                    if (p.mode == BG_DGRAD) {
                        tma_load_2d(dA, &tmA, kb * 64, t.row0, fb);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tma_load_2d(dB + j * kBoxBytes, &tmB, t.n * kBN + 64 * j, t.e * p.wrows + kb * 64, fb);
                    } else {
                        const int y = t.row0 + kb * 64;
#pragma unroll
                        for (int j = 0; j < 2; ++j) tma_load_2d(dA + j * kBoxBytes, &tmA, t.m * kBM + 64 * j, y, fb);
#pragma unroll
                        for (int j = 0; j < 4; ++j) tma_load_2d(dB + j * kBoxBytes, &tmB, t.n * kBN + 64 * j, y, fb);
                    }
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
            for (int s = 0; s < stages; ++s)   // the copies issued land before the CTA exits
                if (issued_mask & (1u << s)) mbar_wait(smem_u32(&full_bar[s]), (issued_parity >> s) & 1, p.budget);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int it = 0, last_b = -1;
            uint32_t last_par = 0;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const BTile t = decode(p, tile, s_start, s_poff, s_offs);
                if (t.nk == 0) continue;   // no kept rows: the epilogue writes zeros
                const int b = it & 1;
                const uint32_t acc_par = (it >> 1) & 1;
                ++it;
                if (!mbar_wait(smem_u32(&tempty_bar[b]), acc_par ^ 1, p.budget)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * kBN);
                for (int kb = 0; kb < t.nk; ++kb) {
                    if (!mbar_wait(smem_u32(&full_bar[stage]), phase, p.budget)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * a_bytes);
                    const uint32_t b0 = smem_u32(sB + stage * b_bytes);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {   // K = 16 per instruction: 16 K-rows = 2048 bytes (MN-major)
                        const uint64_t ad = a_mn ? sdesc_mn_sw128(a0 + k * 2048) : sdesc_k_sw128(a0 + k * 32);
                        const uint64_t bd = sdesc_mn_sw128(b0 + k * 2048);
                        mma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    }
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
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int it = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const BTile t = decode(p, tile, s_start, s_poff, s_offs);
            const int orow = (p.mode == BG_DGRAD) ? t.row0 + row : t.m * kBM + row;
            const bool live = p.mode == BG_DGRAD || orow < p.Mw;
            float* dst = p.out + (p.mode == BG_DGRAD ? static_cast<size_t>(orow)
                                                     : static_cast<size_t>(t.e) * p.Mw + orow) * p.N + t.n * kBN;
            const int ncols = min(kBN, p.N - t.n * kBN);
            if (t.nk == 0) {
                if (live)
                    for (int c = 0; c < ncols; c += 4)
                        *reinterpret_cast<float4*>(dst + c) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                continue;
            }
            const int b = it & 1;
            const uint32_t acc_par = (it >> 1) & 1;
            ++it;
            if (!mbar_wait(smem_u32(&tfull_bar[b]), acc_par, p.budget)) {
                record_error(p.status, MOE_ERR_TIMEOUT);
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * kBN);
            uint32_t v[32];
            for (int c = 0; c < ncols; c += 32) {
                tmem_ld32(taddr + c, v);
                tmem_ld_wait(v);
                if (live) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
                    for (int j = 0; j < 8; ++j) d4[j] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
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
        tmem_dealloc(tmem_base, 2 * kBN);
    }
}

size_t bwd_gemm_fixed_smem(int E) { return 1024 + 6 * 8 + static_cast<size_t>(3 * (E + 1)) * 4 + 16; }

}  // namespace

cudaError_t launch_bwd_gemm(const BwdGemmLaunch& g, cudaStream_t s)
{
    BwdGemmParams p{};
    p.mode = g.mode;
    p.E = g.E;
    p.N = g.N;
    p.n_tiles = (g.N + kBN - 1) / kBN;
    p.offsets = g.offsets;
    p.out = g.out;
    p.status = g.status;
    p.budget = g.budget;
    if (g.N % 32 != 0 || g.K % 64 != 0 || g.N <= 0) return cudaErrorInvalidValue;
    CUtensorMap tmA, tmB;
    long long tiles = 0;
    if (g.mode == BG_DGRAD) {
        p.kb = g.K / 64;
        p.wrows = g.K;
        // A: the row block [rows, K] (K-major boxes); B: the weights [E*K, N] (64 x 64 boxes)
        if (!encode_bf16_map(&tmA, g.a, static_cast<uint64_t>(g.rows), static_cast<uint64_t>(g.K), kBM) ||
            !encode_bf16_map(&tmB, g.b, static_cast<uint64_t>(g.E) * g.K, static_cast<uint64_t>(g.N), 64))
            return cudaErrorInvalidValue;
        tiles = static_cast<long long>(g.rows / kBM + g.E) * p.n_tiles;
    } else {
        p.Mw = g.Mw;
        p.m_tiles = (g.Mw + kBM - 1) / kBM;
        if (g.Mw % 64 != 0) return cudaErrorInvalidValue;
        // A: the row block [rows, Mw]; B: the row block [rows, N] (both 64 x 64 boxes)
        if (!encode_bf16_map(&tmA, g.a, static_cast<uint64_t>(g.rows), static_cast<uint64_t>(g.Mw), 64) ||
            !encode_bf16_map(&tmB, g.b, static_cast<uint64_t>(g.rows), static_cast<uint64_t>(g.N), 64))
            return cudaErrorInvalidValue;
        tiles = static_cast<long long>(g.E) * p.m_tiles * p.n_tiles;
    }
    const size_t fixed = bwd_gemm_fixed_smem(g.E);
    const size_t per_stage = kBM * 64 * 2 + kBN * 64 * 2 + 16;
    p.stages = static_cast<int>(std::min<size_t>(6, (227 * 1024 - fixed) / per_stage));
    const size_t smem = fixed + static_cast<size_t>(p.stages) * per_stage;
    const cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(moe_bwd_gemm_kernel), 227 * 1024);
    if (e != cudaSuccess) return e;
    const int grid = static_cast<int>(std::min<long long>(tiles, num_sms()));
    if (grid <= 0) return cudaSuccess;
    moe_bwd_gemm_kernel<<<grid, kGemmThreads, smem, s>>>(tmA, tmB, p);
    return cudaGetLastError();
}

}  // namespace moe
