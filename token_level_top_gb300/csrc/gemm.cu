// gemm.cu -- persistent tcgen05/TMEM GEMM with TMA-fed operands for the
// three dense contractions of the MoE layer:
//
//   GK_ROUTER        logits partials  = h . W_r^T          (K split across CTAs)
//   GK_GATEUP        act = silu(x W1^T) * (x W3^T), x = the slot-ordered token rows
//                    (tiles of x_perm, the rows gathered by a separate pass)
//   GK_DOWN_SLOTS    y_slots     = act W2^T                 (slot order, bf16)
//
// The router is the linear map of the token's hidden state to expert logits
// ([coreui] §3.1 "Logits生成"; [csdn] §3.1 h @ W_gate); the experts are the
// SwiGLU FFNs W2(silu(W1 x) * W3 x) ([mhpn] §3.1; [2kiu] §1) run over each
// expert's group of tokens ([cnnetsun] §3.2 step 1), and the down projection
// is combined back to token order with the router weights ([mhpn] §4.3;
// [2kiu] §3 step 5).
//
// One CTA per SM (or two for the router), 6 warps:
//   warp 0    TMA producer: A tile 128 x 64 and B tile BN x 64, 128-byte
//             swizzle, into a ring of `stages` shared-memory slots;
//   warp 1    allocates TMEM; lane 0 issues tcgen05.mma (M=128, N=BN, K=16;
//             FP8: kind::f8f6f4, K=32) into one of two TMEM accumulators and
//             commits to mbarriers;
//   warps 2-5 epilogue: tcgen05.ld of their 32 TMEM lanes, fused math, store.
// Expert GEMMs whose experts average two or more row tiles run on clusters of
// two CTAs: each stages its own 128 rows of A and half of the BN weight rows,
// and CTA 0 issues tcgen05.mma.cta_group::2 (M=256) over both.
// Tiles are scheduled statically (tile += gridDim.x) from per-expert row
// counts read on the device, so no host synchronisation is needed.  Every
// wait is bounded; on expiry the CTA records MOE_ERR_TIMEOUT, drains what it
// issued and exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

struct GemmParams {
    int kind, E, T, topk, d, F;
    int kb_total;      // K / 64
    int bn;            // N tile
    int n_tiles;       // N tiles per expert
    int m_tiles;       // router: ceil(T / 128)
    int splits;        // router K splits
    int kb_per_split;  // router K blocks per split
    int stages;
    int b_policy;      // L2 policy of the weight loads: 0 default, 1 evict_first
    const float* b_scale;  // FP8: the scale of each weight row (output channel)
    const float* a_scale;  // FP8: the scale of each activation row (slot order)
    float* act_amax;       // FP8 gate-up: per activation row, atomically maxed with max |bf16 act|
    float* gu_save;          // gate-up, training: g and u of each kept row (fp32, packed W13 order)
    uint32_t tmem_cols;
    const int32_t* offsets;
    const int32_t* perm;
    __nv_bfloat16* act;
    __nv_bfloat16* y_slots;
    float* router_part;
    int* status;
    long long budget;
};

struct TileInfo {
    int e, m, n, kb0, kb1, split;
};

// Expert tiles are numbered expert by expert; within an expert, row units
// fastest (the row tiles that share a weight tile run together), then column
// tiles.  In paired mode a unit is two adjacent row tiles, one per CTA of the
// cluster; each CTA loads half of the unit's weight tile and the paired MMA
// reads both halves.
template <bool PAIR>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int tile,
                                                const int* s_tile_start, const int* s_offs,
                                                int rank)
{
    TileInfo ti;
    if (p.kind == GK_ROUTER) {
        ti.e = 0;
        ti.n = 0;
        ti.m = tile % p.m_tiles;
        ti.split = tile / p.m_tiles;
        ti.kb0 = ti.split * p.kb_per_split;
        ti.kb1 = min(p.kb_total, ti.kb0 + p.kb_per_split);
        return ti;
    }
    int lo = 0, hi = p.E - 1;  // largest e with tile_start[e] <= tile
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (s_tile_start[mid] <= tile)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int e = lo;
    const int cnt = s_offs[e + 1] - s_offs[e];
    const int mt = (cnt + kBM - 1) / kBM;
    const int units = PAIR ? (mt + 1) / 2 : mt;
    const int local = tile - s_tile_start[e];
    ti.e = e;
    ti.m = PAIR ? 2 * (local % units) + rank : local % units;
    ti.n = local / units;
    ti.kb0 = 0;
    ti.kb1 = p.kb_total;
    ti.split = 0;
    return ti;
}

// silu(x) = x sigmoid(x) = (x/2)(1 + tanh(x/2)), with the hardware tanh approximation
// (one MUFU operation; its error stays inside the bf16 rounding of the activation).
// Same box, alternating runs: e4m3 prefill gate-up 624 -> 609 us, bf16 1160 -> 1149 us.
__device__ __forceinline__ float silu_f(float x)
{
    float t;
    const float h = 0.5f * x;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return h * (1.0f + t);
}

// FP8: e4m3 activations and weights on tcgen05.mma.kind::f8f6f4.  A stage
// row is 128 bytes either way (64 bf16 or 128 e4m3 values), so the tiles,
// swizzle and descriptors are the bf16 ones; each MMA covers 32 bytes of K.
// The per-row activation scale and per-row weight scale multiply the
// accumulator in the epilogue.

// Arrival on the first CTA's accumulator barrier with a CTA-scope release: what
// the first CTA's MMAs depend on is this CTA's TMEM, whose reads are complete
// (tcgen05.wait::ld) before the arrival, so no cluster-wide fence over the
// epilogue's row stores is needed (a cluster-scope release waited for them: the
// e4m3 prefill gate-up took 637 us with it, 621 us without).
__device__ __forceinline__ void mbar_arrive_peer_cta(uint32_t cluster_bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

template <bool PAIR, bool FP8>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int stages = p.stages;
    const uint32_t a_bytes = kBM * kBK * 2;
    // paired: this CTA holds its 128 A rows and half of the BN weight rows
    const uint32_t b_bytes = static_cast<uint32_t>(PAIR ? p.bn / 2 : p.bn) * kBK * 2;
    uint8_t* sA = smem;
    uint8_t* sB = sA + stages * a_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + stages * b_bytes);
    uint64_t* full_bar = bars;
    uint64_t* empty_bar = bars + stages;
    uint64_t* tfull_bar = bars + 2 * stages;
    uint64_t* tempty_bar = bars + 2 * stages + 2;
    int* s_tile_start = reinterpret_cast<int*>(bars + 2 * stages + 4);
    int* s_offs = s_tile_start + (p.E + 1);
    volatile uint32_t* s_tmem = reinterpret_cast<volatile uint32_t*>(s_offs + (p.E + 1));
    // FP8: the current tile's weight-row scales, staged by the epilogue warps
    float* s_bsc = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(s_tmem + 1) + 15) & ~uintptr_t(15));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;

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
        if (PAIR) {   // one warp of each CTA of the pair, collectively
            tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(s_tmem)), p.tmem_cols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(const_cast<uint32_t*>(s_tmem)), p.tmem_cols);
            tmem_relinquish();
        }
    }
    if (p.kind != GK_ROUTER && warp == 2) {
        // tile_start[e] = sum over e' < e of ceil(count_e' / 128) * n_tiles
        int carry = 0;
        for (int base = 0; base <= p.E; base += 32) {
            const int e = base + lane;
            int o = 0, o1 = 0;
            if (e <= p.E) o = p.offsets[e];
            if (e < p.E) o1 = p.offsets[e + 1];
            if (e <= p.E) s_offs[e] = o;
            const int mt = (o1 - o + kBM - 1) / kBM;
            int tiles = (e < p.E) ? (PAIR ? (mt + 1) / 2 : mt) * p.n_tiles : 0;
            int incl = tiles;
            for (int off = 1; off < 32; off <<= 1) {
                int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            if (e <= p.E) s_tile_start[e] = carry + incl - tiles;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (PAIR) cluster_sync_all();   // the peer's barriers exist before anything targets them
    const uint32_t tmem_base = *s_tmem;
    const int total_tiles = (p.kind == GK_ROUTER) ? p.m_tiles * p.splits : s_tile_start[p.E];
    const uint32_t idesc = FP8 ? idesc_e4m3_f32(PAIR ? 2 * kBM : kBM, p.bn)
                               : idesc_bf16_f32(PAIR ? 2 * kBM : kBM, p.bn);
    const bool leader = rank == 0;   // the paired MMAs are issued by CTA 0 of the cluster
    // a cluster's two CTAs walk the same tile sequence
    const int tile0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int tile_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const uint64_t pol_b = l2_policy_evict_first();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;  // per stage: a load in flight + its parity
        for (int tile = tile0; tile < total_tiles && ok; tile += tile_step) {
            const TileInfo ti = decode_tile<PAIR>(p, tile, s_tile_start, s_offs, rank);
            int arow = 0, brow = 0;
            if (p.kind == GK_GATEUP) {
                arow = s_offs[ti.e] + ti.m * kBM;
                brow = ti.e * 2 * p.F + ti.n * kExpertBN;
            } else if (p.kind == GK_ROUTER) {
                arow = ti.m * kBM;
                brow = 0;
            } else {
                arow = s_offs[ti.e] + ti.m * kBM;
                brow = ti.e * p.d + ti.n * p.bn;
            }
            for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, p.budget))) {
                    ok = false;
                    break;
                }
                // paired: both CTAs' copies count on the leader CTA's full barrier
                const uint32_t fb = PAIR ? map_to_rank(smem_u32(&full_bar[stage]), 0)
                                         : smem_u32(&full_bar[stage]);
                if (lane == 0 && leader)
                    mbar_arrive_expect_tx(smem_u32(&full_bar[stage]),
                                          (PAIR ? 2u : 1u) * (a_bytes + b_bytes));
                __syncwarp();
                const int x = kb * (FP8 ? 2 * kBK : kBK);   // K elements of a 128-byte row
                const uint32_t dA = smem_u32(sA + stage * a_bytes);
                const uint32_t dB = smem_u32(sB + stage * b_bytes);
                if (PAIR) {
                    if (lane == 0) {
                        tma_load_2d_pair(dA, &tmA, x, arow, fb);
                        if (p.b_policy)
                            tma_load_2d_pair_hint(dB, &tmB, x, brow + rank * (p.bn / 2), fb, pol_b);
                        else
                            tma_load_2d_pair(dB, &tmB, x, brow + rank * (p.bn / 2), fb);
                    }
                } else {
                    if (lane == 0) {
                        tma_load_2d(dA, &tmA, x, arow, fb);
                        if (p.b_policy)
                            tma_load_2d_hint(dB, &tmB, x, brow, fb, pol_b);
                        else
                            tma_load_2d(dB, &tmB, x, brow, fb);
                    }
                }
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
            // let the copies issued land before the CTA exits (paired: the leader's
            // full barriers count both CTAs' copies; the final cluster barrier
            // holds the peer until the leader has drained)
            if (leader)
                for (int s = 0; s < stages; ++s)
                    if (issued_mask & (1u << s))
                        mbar_wait(smem_u32(&full_bar[s]), (issued_parity >> s) & 1, p.budget);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            int last_b = -1;
            uint32_t last_par = 0;
            for (int tile = tile0; tile < total_tiles && ok; tile += tile_step, ++it) {
                const TileInfo ti = decode_tile<PAIR>(p, tile, s_tile_start, s_offs, rank);
                const int b = it & 1;
                const uint32_t acc_par = (it >> 1) & 1;
                if (!mbar_wait(smem_u32(&tempty_bar[b]), acc_par ^ 1, p.budget)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * p.bn);
                for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&full_bar[stage]), phase, p.budget)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * a_bytes);
                    const uint32_t b0 = smem_u32(sB + stage * b_bytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        const uint64_t ad = sdesc_k_sw128(a0 + k * 32), bd = sdesc_k_sw128(b0 + k * 32);
                        const uint32_t acc = (kb > ti.kb0 || k > 0) ? 1u : 0u;
                        if (FP8) {
                            if (PAIR)
                                mma_e4m3_pair(d_tmem, ad, bd, idesc, acc);
                            else
                                mma_e4m3(d_tmem, ad, bd, idesc, acc);
                        } else {
                            if (PAIR)
                                mma_bf16_pair(d_tmem, ad, bd, idesc, acc);
                            else
                                mma_bf16(d_tmem, ad, bd, idesc, acc);
                        }
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
            // all MMAs issued must be complete before TMEM is released
            if (last_b >= 0) mbar_wait(smem_u32(&tfull_bar[last_b]), last_par, p.budget);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        int it = 0;
        for (int tile = tile0; tile < total_tiles; tile += tile_step, ++it) {
            const TileInfo ti = decode_tile<PAIR>(p, tile, s_tile_start, s_offs, rank);
            const int b = it & 1;
            const uint32_t acc_par = (it >> 1) & 1;
            const bool staged = FP8 && p.kind != GK_ROUTER;
            if (staged) {
                // the tile's weight-row scales into shared memory while its MMAs run
                // (the 128 epilogue threads, two scales each; named barrier 1)
                const int et = static_cast<int>(threadIdx.x) - 64;
                epilogue_sync();   // the previous tile's scales are no longer read
                for (int i = et; i < kExpertBN; i += 128) {
                    float v = 0.0f;
                    if (p.kind == GK_GATEUP)
                        v = __ldg(p.b_scale + static_cast<size_t>(ti.e) * 2 * p.F + ti.n * kExpertBN + i);
                    else if (i < p.bn && ti.n * p.bn + i < p.d)
                        v = __ldg(p.b_scale + static_cast<size_t>(ti.e) * p.d + ti.n * p.bn + i);
                    s_bsc[i] = v;
                }
            }
            bool got = mbar_wait(smem_u32(&tfull_bar[b]), acc_par, p.budget);
            // staged: one decision for the 128 threads (none is left at a barrier), and
            // the barrier that publishes the scales
            if (staged) got = epilogue_all(got);
            if (!got) {
                record_error(p.status, MOE_ERR_TIMEOUT);
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(b * p.bn);
            uint32_t v[32];
            if (p.kind == GK_ROUTER) {
                const int t = ti.m * kBM + row;
                float* dst = p.router_part + (static_cast<size_t>(ti.split) * p.T + t) * p.E;
                for (int c = 0; c < p.bn; c += 32) {
                    tmem_ld32(taddr + c, v);
                    tmem_ld_wait(v);
                    if (t < p.T) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (c + j < p.E) dst[c + j] = __uint_as_float(v[j]);
                    }
                }
            } else if (p.kind == GK_GATEUP) {
                const int off = s_offs[ti.e];
                const int cnt = s_offs[ti.e + 1] - off;
                const int ri = ti.m * kBM + row;
                uint32_t u[32];
                __nv_bfloat16* dst = p.act + static_cast<size_t>(off + ri) * p.F + ti.n * (kExpertBN / 2);
                // FP8: the tile's W1 and W3 row scales (packed rows of W13) are in
                // s_bsc; this thread's activation row scale
                const float asc = (FP8 && ri < cnt) ? p.a_scale[off + ri] : 0.0f;
                float rmax = 0.0f;   // FP8: max |act| over this thread's columns
                for (int c = 0; c < kExpertBN / 2; c += 32) {
                    tmem_ld32(taddr + c, v);                   // gate columns
                    tmem_ld32(taddr + kExpertBN / 2 + c, u);   // matching up columns
                    tmem_ld_wait2(v, u);
                    if (FP8) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            v[j] = __float_as_uint(__uint_as_float(v[j]) * asc * s_bsc[c + j]);
                            u[j] = __float_as_uint(__uint_as_float(u[j]) * asc * s_bsc[kExpertBN / 2 + c + j]);
                        }
                    }
                    if (ri < cnt && p.gu_save) {
                        // g and u kept for the backward pass, in the packed W13 column order
                        float* gs = p.gu_save + static_cast<size_t>(off + ri) * 2 * p.F + ti.n * kExpertBN + c;
                        uint4* g4 = reinterpret_cast<uint4*>(gs);
                        uint4* u4 = reinterpret_cast<uint4*>(gs + kExpertBN / 2);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            g4[j] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                            u4[j] = make_uint4(u[4 * j], u[4 * j + 1], u[4 * j + 2], u[4 * j + 3]);
                        }
                    }
                    if (ri < cnt) {
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float a0 = silu_f(__uint_as_float(v[2 * j])) * __uint_as_float(u[2 * j]);
                            const float a1 =
                                silu_f(__uint_as_float(v[2 * j + 1])) * __uint_as_float(u[2 * j + 1]);
                            pk[j] = pack_bf16x2(a0, a1);
                            if (FP8) rmax = fmaxf(rmax, fmaxf(fabsf(a0), fabsf(a1)));
                        }
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            d4[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    }
                }
                // The row maximum the activation quantiser needs, so that it
                // reads each row once: rounding to bf16 is monotone, so the
                // largest stored |value| is the rounded largest |value|; the
                // bits of non-negative floats order as the floats do.
                if (FP8 && p.act_amax && ri < cnt)
                    atomicMax(reinterpret_cast<unsigned int*>(p.act_amax + off + ri),
                              __float_as_uint(__bfloat162float(__float2bfloat16_rn(rmax))));
            } else {
                const int off = s_offs[ti.e];
                const int cnt = s_offs[ti.e + 1] - off;
                const int ri = ti.m * kBM + row;
                const bool valid = ri < cnt;
                const int slot = off + ri;
                const int col0 = ti.n * p.bn;
                __nv_bfloat16* dst = p.y_slots + static_cast<size_t>(slot) * p.d + col0;
                const float asc = (FP8 && valid) ? p.a_scale[slot] : 0.0f;
                for (int c = 0; c < p.bn; c += 32) {
                    if (col0 + c >= p.d) break;
                    tmem_ld32(taddr + c, v);
                    tmem_ld_wait(v);
                    if (FP8) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + c + j < p.d)
                                v[j] = __float_as_uint(__uint_as_float(v[j]) * asc * s_bsc[c + j]);
                    }
                    if (valid) {
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            d4[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    }
                }
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
            tmem_dealloc_pair(tmem_base, p.tmem_cols);
        else
            tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 2-D bf16 tensor [rows, cols] (row-major), box [box_rows, 64], 128-byte swizzle.
bool make_map(CUtensorMap* tm, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows)
{
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {cols * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), gdim, gstride,
                     box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D e4m3 (byte) tensor [rows, cols] (row-major), box [box_rows, 128]: the
// same 128-byte rows and swizzle as the bf16 boxes.
bool make_map_e4m3(CUtensorMap* tm, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows)
{
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {cols};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(2 * kBK), box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), gdim, gstride, box,
                     estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool encode_bf16_map(CUtensorMap* tm, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows)
{
    return make_map(tm, ptr, rows, cols, box_rows);
}

namespace {

uint32_t pow2_cols(int n)
{
    uint32_t c = 32;
    while (c < static_cast<uint32_t>(n)) c <<= 1;
    return c;
}

}  // namespace

namespace {

constexpr int kRouterStages = 4;

size_t gemm_fixed_smem(int E, bool fp8 = false)
{
    // alignment slack, barriers, tile table, TMEM address; FP8: the staged row scales
    return 1024 + 64 + static_cast<size_t>(2 * (E + 1)) * 4 + 16 + 6 * 8 + (fp8 ? 16 + 4 * kExpertBN : 0);
}

}  // namespace

int router_ctas_per_sm(int E)
{
    const size_t epad = static_cast<size_t>(std::max(32, (E + 31) / 32 * 32));
    const size_t smem = gemm_fixed_smem(E) + kRouterStages * (kBM * kBK * 2 + epad * kBK * 2 + 16);
    return smem <= 113 * 1024 ? 2 : 1;
}

cudaError_t launch_gemm(const GemmLaunch& g, cudaStream_t s)
{
    GemmParams p{};
    p.kind = g.kind;
    p.E = g.E;
    p.T = g.T;
    p.topk = g.topk;
    p.d = g.d;
    p.F = g.F;
    p.offsets = g.offsets;
    p.perm = g.perm;
    p.act = static_cast<__nv_bfloat16*>(g.act);
    p.y_slots = static_cast<__nv_bfloat16*>(g.y_slots);
    p.router_part = g.router_part;
    p.status = g.status;
    p.budget = g.budget;

    CUtensorMap tmA, tmB;
    // FP8: e4m3 activations and weights, each row with its scale
    const bool fp8 = g.fp8 && g.kind != GK_ROUTER;
    p.b_scale = fp8 ? g.b_scale : nullptr;
    p.a_scale = fp8 ? g.a_scale : nullptr;
    p.act_amax = fp8 ? g.act_amax : nullptr;
    p.gu_save = (!fp8 && g.kind == GK_GATEUP) ? static_cast<float*>(g.gu_save) : nullptr;
    const int kstep = fp8 ? 2 * kBK : kBK;   // K elements per 128-byte stage row
    // When no expert holds more than one row tile, every weight tile is read by
    // exactly one tile: its lines go first out of L2, ahead of the token rows.
    p.b_policy = (g.kind != GK_ROUTER && g.rows_cap > 0 && std::min<long long>(g.rows_cap, g.T) <= kBM) ? 1 : 0;
    auto map = [&](CUtensorMap* tm, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
        return fp8 ? make_map_e4m3(tm, ptr, rows, cols, box_rows) : make_map(tm, ptr, rows, cols, box_rows);
    };
    int grid = 0;
    const int sms = num_sms();
    // Row tiles are paired when the experts average at least two of them.
    const bool pair = (g.kind != GK_ROUTER) && static_cast<long long>(g.T) * g.topk >= 2LL * kBM * g.E;
    if (g.kind == GK_ROUTER) {
        p.bn = g.epad;
        p.kb_total = g.d / kBK;
        p.m_tiles = (g.T + kBM - 1) / kBM;
        p.splits = g.splits;
        p.kb_per_split = (p.kb_total + g.splits - 1) / g.splits;
        p.n_tiles = 1;
        if (!make_map(&tmA, g.a_ptr, g.T, g.d, kBM)) return cudaErrorInvalidValue;
        if (!make_map(&tmB, g.b_ptr, g.E, g.d, p.bn)) return cudaErrorInvalidValue;
        grid = std::min(p.m_tiles * p.splits, router_ctas_per_sm(g.E) * sms);
    } else if (g.kind == GK_GATEUP) {
        p.bn = kExpertBN;
        p.kb_total = g.d / kstep;
        p.n_tiles = g.F / (kExpertBN / 2);
        if (!map(&tmA, g.a_ptr, static_cast<uint64_t>(g.T) * g.topk, g.d, kBM))
            return cudaErrorInvalidValue;
        if (!map(&tmB, g.b_ptr, static_cast<uint64_t>(g.E) * 2 * g.F, g.d, pair ? kExpertBN / 2 : kExpertBN))
            return cudaErrorInvalidValue;
        const long long mt_max = (static_cast<long long>(g.T) * g.topk + kBM - 1) / kBM + g.E;
        grid = static_cast<int>(std::min<long long>(mt_max * p.n_tiles, sms));
    } else {
        p.bn = kExpertBN;
        if (!pair && g.rows_cap > 0 && g.rows_cap <= kBM) {
            // Every expert holds at most one row tile, so the tile count is
            // known: take the column tile (a multiple of 32, 128..256) that
            // needs the fewest passes over the SMs times its width.
            const long long mt = std::min<long long>(g.E, static_cast<long long>(g.T) * g.topk);
            long long best = -1;
            for (int bn = kExpertBN; bn >= 128; bn -= 32) {
                const long long tiles = mt * ((g.d + bn - 1) / bn);
                const long long cost = (tiles + sms - 1) / sms * bn;
                if (best < 0 || cost < best) {
                    best = cost;
                    p.bn = bn;
                }
            }
        }
        p.kb_total = g.F / kstep;
        p.n_tiles = (g.d + p.bn - 1) / p.bn;
        if (!map(&tmA, g.a_ptr, static_cast<uint64_t>(g.T) * g.topk, g.F, kBM))
            return cudaErrorInvalidValue;
        if (!map(&tmB, g.b_ptr, static_cast<uint64_t>(g.E) * g.d, g.F, pair ? p.bn / 2 : p.bn))
            return cudaErrorInvalidValue;
        const long long mt_max = (static_cast<long long>(g.T) * g.topk + kBM - 1) / kBM + g.E;
        grid = static_cast<int>(std::min<long long>(mt_max * p.n_tiles, sms));
    }
    const uint32_t a_bytes = kBM * kBK * 2;
    const uint32_t b_bytes = static_cast<uint32_t>(pair ? p.bn / 2 : p.bn) * kBK * 2;
    const size_t fixed = gemm_fixed_smem(g.E, fp8);
    const size_t budget_smem = 227 * 1024;
    int stages = static_cast<int>((budget_smem - fixed) / (a_bytes + b_bytes + 16));
    stages = std::max(2, std::min(stages, g.kind == GK_ROUTER ? kRouterStages : 8));
    p.stages = stages;
    p.tmem_cols = pow2_cols(2 * p.bn);
    const size_t smem = fixed + static_cast<size_t>(stages) * (a_bytes + b_bytes + 16);

    const void* kfn = pair ? (fp8 ? reinterpret_cast<const void*>(moe_gemm_kernel<true, true>)
                                  : reinterpret_cast<const void*>(moe_gemm_kernel<true, false>))
                           : (fp8 ? reinterpret_cast<const void*>(moe_gemm_kernel<false, true>)
                                  : reinterpret_cast<const void*>(moe_gemm_kernel<false, false>));
    const cudaError_t attr_err = ensure_smem_limit(kfn, 227 * 1024);
    if (attr_err != cudaSuccess) return attr_err;
    if (grid <= 0) return cudaSuccess;
    if (!pair) {
        if (fp8)
            moe_gemm_kernel<false, true><<<grid, kGemmThreads, smem, s>>>(tmA, tmB, p);
        else
            moe_gemm_kernel<false, false><<<grid, kGemmThreads, smem, s>>>(tmA, tmB, p);
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
    static int cached_clusters[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int max_clusters = (dev >= 0 && dev < 64) ? cached_clusters[dev] : 0;
    if (max_clusters <= 0) {
        cfg.gridDim = dim3(2 * 64, 1, 1);
        if (cudaOccupancyMaxActiveClusters(&max_clusters, fp8 ? moe_gemm_kernel<true, true> : moe_gemm_kernel<true, false>, &cfg) != cudaSuccess ||
            max_clusters <= 0)
            max_clusters = sms / 2;
        if (dev >= 0 && dev < 64) cached_clusters[dev] = max_clusters;
    }
    const int clusters = std::max(1, std::min(grid / 2, max_clusters));
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
    return fp8 ? cudaLaunchKernelEx(&cfg, moe_gemm_kernel<true, true>, tmA, tmB, p)
               : cudaLaunchKernelEx(&cfg, moe_gemm_kernel<true, false>, tmA, tmB, p);
}

}  // namespace moe
