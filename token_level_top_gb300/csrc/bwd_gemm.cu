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
// TMEM and store fp32 rows.  With enough row tiles the CTAs run in clusters
// of two on tcgen05.mma.cta_group::2 (M = 256 over the pair, each CTA
// staging its 128 rows of A and half of B's 256 columns), which halves the
// shared-memory traffic per MMA.  The epilogue writes each warp's 32 x 32
// block through a padded shared-memory tile, so that every store
// instruction covers four whole 128-byte lines of a row-major output
// instead of 32 scattered pieces.  The tile table is built on the device
// from the forward's per-expert offsets; an expert with no kept rows gets
// zero weight gradients without MMAs.  Every wait is bounded.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kBN = 256;   // output tile columns
constexpr uint32_t kBoxBytes = 64 * 64 * 2;   // one 64 x 64 bf16 box
constexpr int kTrStride = 36;                 // floats per row of the epilogue's transpose tile

struct BwdGemmParams {
    int mode, E;
    int kb;          // BG_DGRAD: K / 64
    int wrows;       // BG_DGRAD: rows of one expert's weight matrix in the B map (= K)
    int N;           // output columns
    int n_tiles;     // ceil(N / 256)
    int Mw;          // BG_WGRAD: output rows per expert
    int m_tiles;     // BG_WGRAD: ceil(Mw / 128)
    int stages;
    int n_fast;      // BG_WGRAD: column tiles fastest within an expert (else row tiles)
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

// Tiles are numbered expert by expert.  Paired, a unit is two adjacent 128-row
// tiles, one per CTA of the cluster (rank), which share the unit's B tile.
template <bool PAIR>
__device__ __forceinline__ BTile decode(const BwdGemmParams& p, int tile, const int* s_start, const int* s_poff,
                                        const int* s_offs, int rank)
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
        const int units = PAIR ? (mt + 1) / 2 : mt;
        const int u = local % units;
        t.m = PAIR ? 2 * u + rank : u;
        t.n = local / units;
        t.row0 = s_poff[lo] + t.m * kBM;
        t.nk = p.kb;
    } else {
        const int units = PAIR ? (p.m_tiles + 1) / 2 : p.m_tiles;
        int u;
        if (p.n_fast) {
            u = local / p.n_tiles;
            t.n = local % p.n_tiles;
        } else {
            u = local % units;
            t.n = local / units;
        }
        t.m = PAIR ? 2 * u + rank : u;
        t.row0 = s_poff[lo];
        t.nk = (s_offs[lo + 1] - s_offs[lo] + 63) / 64;
    }
    return t;
}

// MN-major operand of the pair MMA: each CTA's part is `blocks` 64-column boxes.
constexpr uint32_t kStageTileBytes = kBoxBytes;

// Arrival on the first CTA's accumulator barrier with a CTA-scope release: the
// first CTA's MMAs depend only on this CTA's TMEM reads, complete before the
// arrival (tcgen05.wait::ld), not on the epilogue's fp32 row stores.
__device__ __forceinline__ void mbar_arrive_peer_cta(uint32_t cluster_bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

template <bool PAIR>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_bwd_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const BwdGemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int stages = p.stages;
    constexpr uint32_t a_bytes = kBM * 64 * 2;                   // 16 KB: 128 x 64 (K-major) or 2 boxes
    constexpr uint32_t b_bytes = (PAIR ? kBN / 2 : kBN) * 64 * 2;  // this CTA's boxes of the 256 B columns
    constexpr int b_boxes = (PAIR ? kBN / 2 : kBN) / 64;
    uint8_t* sA = smem;
    uint8_t* sB = sA + stages * a_bytes;
    float* s_tr = reinterpret_cast<float*>(sB + stages * b_bytes);   // 4 x [32][36] epilogue transpose
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_tr + 4 * 32 * kTrStride);
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
    const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
    const bool leader = rank == 0;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        for (int i = 0; i < stages; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull_bar[b]), 1);
            mbar_init(smem_u32(&tempty_bar[b]), PAIR ? 8 : 4);   // paired: both CTAs' epilogues
        }
        mbar_fence_init();
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(s_tmem)), 2 * kBN);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(const_cast<uint32_t*>(s_tmem)), 2 * kBN);
            tmem_relinquish();
        }
    }
    if (warp == 2) {
        // padded row offsets (each expert's kept rows rounded up to 128) and the
        // tile table: tiles of expert e start at s_start[e]
        const int units_w = PAIR ? (p.m_tiles + 1) / 2 : p.m_tiles;
        int carry_rows = 0, carry_tiles = 0;
        for (int base = 0; base <= p.E; base += 32) {
            const int e = base + lane;
            int o = 0, o1 = 0;
            if (e <= p.E) o = p.offsets[e];
            if (e < p.E) o1 = p.offsets[e + 1];
            if (e <= p.E) s_offs[e] = o;
            const int prow = (e < p.E) ? (o1 - o + kBM - 1) / kBM * kBM : 0;
            int tiles = 0;
            if (e < p.E) {
                const int mt = prow / kBM;
                tiles = (p.mode == BG_DGRAD ? (PAIR ? (mt + 1) / 2 : mt) : units_w) * p.n_tiles;
            }
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
    if (PAIR) cluster_sync_all();   // the peer's barriers exist before anything targets them
    const uint32_t tmem_base = *s_tmem;
    const int total = s_start[p.E];
    const bool a_mn = p.mode == BG_WGRAD;
    const uint32_t idesc = idesc_bf16_f32(PAIR ? 2 * kBM : kBM, kBN) | (a_mn ? (1u << 15) : 0u) | (1u << 16);
    // a cluster's two CTAs walk the same tile sequence
    const int tile0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int tile_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;
        for (int tile = tile0; tile < total && ok; tile += tile_step) {
            const BTile t = decode<PAIR>(p, tile, s_start, s_poff, s_offs, rank);
            const int bcol = t.n * kBN + (PAIR ? rank * (kBN / 2) : 0);   // this CTA's B columns
            for (int kb = 0; kb < t.nk; ++kb) {
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, p.budget))) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    // paired: both CTAs' copies count on the leader CTA's full barrier
                    const uint32_t fb = PAIR ? map_to_rank(smem_u32(&full_bar[stage]), 0) : smem_u32(&full_bar[stage]);
                    if (leader) mbar_arrive_expect_tx(smem_u32(&full_bar[stage]), (PAIR ? 2u : 1u) * (a_bytes + b_bytes));
                    const uint32_t dA = smem_u32(sA + stage * a_bytes);
                    const uint32_t dB = smem_u32(sB + stage * b_bytes);
                    auto load = [&](uint32_t dst, const CUtensorMap* tm, int x, int y) {
                        if (PAIR)
                            tma_load_2d_pair(dst, tm, x, y, fb);
                        else
                            tma_load_2d(dst, tm, x, y, fb);
                    };
                    if (p.mode == BG_DGRAD) {
                        load(dA, &tmA, kb * 64, t.row0);
#pragma unroll
                        for (int j = 0; j < b_boxes; ++j)
                            load(dB + j * kStageTileBytes, &tmB, bcol + 64 * j, t.e * p.wrows + kb * 64);
                    } else {
                        const int y = t.row0 + kb * 64;
#pragma unroll
                        for (int j = 0; j < 2; ++j) load(dA + j * kStageTileBytes, &tmA, t.m * kBM + 64 * j, y);
#pragma unroll
                        for (int j = 0; j < b_boxes; ++j) load(dB + j * kStageTileBytes, &tmB, bcol + 64 * j, y);
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
            // the copies issued land before the CTA exits (paired: the leader's full
            // barriers count both CTAs' copies; the final cluster barrier holds the peer)
            if (leader)
                for (int s = 0; s < stages; ++s)
                    if (issued_mask & (1u << s)) mbar_wait(smem_u32(&full_bar[s]), (issued_parity >> s) & 1, p.budget);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int it = 0, last_b = -1;
            uint32_t last_par = 0;
            for (int tile = tile0; tile < total && ok; tile += tile_step) {
                const BTile t = decode<PAIR>(p, tile, s_start, s_poff, s_offs, rank);
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
                        const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
                        if (PAIR)
                            mma_bf16_pair(d_tmem, ad, bd, idesc, acc);
                        else
                            mma_bf16(d_tmem, ad, bd, idesc, acc);
                    }
                    if (PAIR)   // frees the slot in both CTAs
                        mma_commit_pair(smem_u32(&empty_bar[stage]));
                    else
                        mma_commit(smem_u32(&empty_bar[stage]));
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if (PAIR)
                    mma_commit_pair(smem_u32(&tfull_bar[b]));
                else
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
        float* tr = s_tr + q * 32 * kTrStride;   // this warp's 32 x 32 transpose tile
        int it = 0;
        for (int tile = tile0; tile < total; tile += tile_step) {
            const BTile t = decode<PAIR>(p, tile, s_start, s_poff, s_offs, rank);
            // rows of this warp's 32-row quarter that are outputs: the tile belongs to the
            // expert's block (paired: the unit's second tile may lie past it) and, for the
            // weight gradients, lies within the Mw rows
            const int qrow0 = (p.mode == BG_DGRAD) ? t.row0 + q * 32 : t.m * kBM + q * 32;
            int live_rows;
            if (p.mode == BG_DGRAD)
                live_rows = (t.row0 < s_poff[t.e + 1]) ? 32 : 0;
            else
                live_rows = max(0, min(32, p.Mw - qrow0));
            float* dst = p.out + (p.mode == BG_DGRAD ? static_cast<size_t>(qrow0)
                                                     : static_cast<size_t>(t.e) * p.Mw + qrow0) * p.N + t.n * kBN;
            const int ncols = min(kBN, p.N - t.n * kBN);
            if (t.nk == 0) {
                for (int r = 0; r < live_rows; ++r)
                    for (int c = 4 * lane; c < ncols; c += 128)
                        *reinterpret_cast<float4*>(dst + static_cast<size_t>(r) * p.N + c) =
                            make_float4(0.0f, 0.0f, 0.0f, 0.0f);
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
                // this thread's row (lane) into the tile, then each store instruction
                // writes 4 rows x 32 columns (4 whole 128-byte lines)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<uint4*>(tr + lane * kTrStride + 4 * j) =
                        make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = 4 * i + (lane >> 3);
                    const float4 w = *reinterpret_cast<const float4*>(tr + r * kTrStride + 4 * (lane & 7));
                    if (r < live_rows)
                        *reinterpret_cast<float4*>(dst + static_cast<size_t>(r) * p.N + c + 4 * (lane & 7)) = w;
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR && !leader)   // the leader's MMAs wait for both CTAs' epilogues
                    mbar_arrive_peer_cta(map_to_rank(smem_u32(&tempty_bar[b]), 0));
                else
                    mbar_arrive(smem_u32(&tempty_bar[b]));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync_all();   // no CTA leaves while its peer may still target it
    if (warp == 1) {
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, 2 * kBN);
        else
            tmem_dealloc(tmem_base, 2 * kBN);
    }
}

size_t bwd_gemm_fixed_smem(int E)
{
    // alignment slack, the epilogue's transpose tiles, the 4 TMEM barriers, tile tables, TMEM address
    return 1024 + 4 * 32 * kTrStride * 4 + 6 * 8 + static_cast<size_t>(3 * (E + 1)) * 4 + 16;
}

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
    bool pair = false;
    if (g.mode == BG_DGRAD) {
        p.kb = g.K / 64;
        p.wrows = g.K;
        // paired when the experts average two or more row tiles and the tiles are short:
        // with a long K (the dx GEMM, K = 2F) a half-empty pair unit per expert and the
        // fewer, longer units cost more than the pairs save (Mixtral prefill, K = 28672:
        // 1138 us single, 1222 us paired; K = 4096: 673 us single, 594 us paired)
        pair = g.kept >= 2LL * kBM * g.E && g.K <= 8192;
        // A: the row block [rows, K] (K-major boxes); B: the weights [E*K, N] (64 x 64 boxes)
        if (!encode_bf16_map(&tmA, g.a, static_cast<uint64_t>(g.rows), static_cast<uint64_t>(g.K), kBM) ||
            !encode_bf16_map(&tmB, g.b, static_cast<uint64_t>(g.E) * g.K, static_cast<uint64_t>(g.N), 64))
            return cudaErrorInvalidValue;
        tiles = static_cast<long long>(g.rows / kBM + g.E) * p.n_tiles;
    } else {
        if (g.Mw % 64 != 0) return cudaErrorInvalidValue;
        p.Mw = g.Mw;
        p.m_tiles = (g.Mw + kBM - 1) / kBM;
        pair = p.m_tiles >= 2;
        // the larger operand is read once: column tiles fastest when A (Mw wide) is wider than B
        p.n_fast = g.Mw > g.N ? 1 : 0;
        // A: the row block [rows, Mw]; B: the row block [rows, N] (both 64 x 64 boxes)
        if (!encode_bf16_map(&tmA, g.a, static_cast<uint64_t>(g.rows), static_cast<uint64_t>(g.Mw), 64) ||
            !encode_bf16_map(&tmB, g.b, static_cast<uint64_t>(g.rows), static_cast<uint64_t>(g.N), 64))
            return cudaErrorInvalidValue;
        tiles = static_cast<long long>(g.E) * p.m_tiles * p.n_tiles;
    }
    const size_t fixed = bwd_gemm_fixed_smem(g.E);
    const size_t per_stage = kBM * 64 * 2 + (pair ? kBN / 2 : kBN) * 64 * 2 + 16;
    p.stages = static_cast<int>(std::min<size_t>(6, (227 * 1024 - fixed) / per_stage));
    const size_t smem = fixed + static_cast<size_t>(p.stages) * per_stage;
    const void* kfn = pair ? reinterpret_cast<const void*>(moe_bwd_gemm_kernel<true>)
                           : reinterpret_cast<const void*>(moe_bwd_gemm_kernel<false>);
    const cudaError_t e = ensure_smem_limit(kfn, 227 * 1024);
    if (e != cudaSuccess) return e;
    const int sms = num_sms();
    if (!pair) {
        const int grid = static_cast<int>(std::min<long long>(tiles, sms));
        if (grid <= 0) return cudaSuccess;
        moe_bwd_gemm_kernel<false><<<grid, kGemmThreads, smem, s>>>(tmA, tmB, p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // a persistent grid of no more clusters than can be resident at once
    int max_clusters = 0;
    cfg.gridDim = dim3(2 * 64, 1, 1);
    if (cudaOccupancyMaxActiveClusters(&max_clusters, moe_bwd_gemm_kernel<true>, &cfg) != cudaSuccess ||
        max_clusters <= 0)
        max_clusters = sms / 2;
    const long long units = (tiles + 1) / 2;
    const int clusters = static_cast<int>(std::max<long long>(1, std::min<long long>(units, max_clusters)));
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
    return cudaLaunchKernelEx(&cfg, moe_bwd_gemm_kernel<true>, tmA, tmB, p);
}

}  // namespace moe
