// route_block.cuh -- the routing of one 256-token chunk by one 1024-thread
// block, or by a cluster of cs such blocks (each routes kChunk/cs of the
// chunk's tokens; their per-expert pick counts and probability sums meet
// through distributed shared memory).  Shared by the route kernel and the
// fused small-batch kernel.  (Semantics and citations: see route.cu.)
#pragma once

#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace detail {

constexpr int kRouteThreads = 1024;             // 32 warps share one chunk of tokens
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRankWarps = kChunk / 32;          // the rank pass: one token per thread

__device__ __forceinline__ float softmax_num(float s, float m)
{
    if (m == INFINITY) return (s == INFINITY) ? 1.0f : 0.0f;
    if (m == -INFINITY) return 1.0f;
    return expf(s - m);
}

// Tokens [cr*kChunk/cs, (cr+1)*kChunk/cs) of chunk `chunk`, by a block of
// kRouteThreads threads that is CTA cr of a cluster of cs (1, 2, 4 or 8)
// routing the same chunk.  With cs > 1 every CTA of the cluster must call it.
template <int EPL>
__device__ __forceinline__ void route_block(const RouteArgs& a, const int chunk, const int cs,
                                            const int cr)
{
    __shared__ int16_t s_ids[kChunk * 8];
    __shared__ int s_wcnt[kRankWarps][32 * EPL];
    __shared__ float s_wsum[kRouteWarps][32 * EPL];
    __shared__ int s_ctot[8][32 * EPL];   // per rank: this CTA's picks of each expert (cs > 1)
    __shared__ int16_t s_crl[kChunk * 8];   // rank of each pick among this CTA's (cs > 1)
    __shared__ float s_psum[32 * EPL];    // this CTA's probability sum of each expert
    __shared__ int s_nan;

    const int E = a.E, k = a.k, T = a.T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int G = 1;
    while (G < E && G < 32) G <<= 1;
    const int lg = lane & (G - 1);
    const int grp = lane / G;
    const int tpw = 32 / G;
    const int t_begin = chunk * kChunk;
    const int sub = kChunk / cs;          // tokens of this CTA
    const int tl0 = cr * sub;
    if (threadIdx.x == 0) s_nan = 0;

    float acc[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) acc[j] = 0.0f;
    bool saw_nan = false;

    for (int base = warp * tpw; base < sub; base += kRouteWarps * tpw) {
        const bool mine = base + grp < sub;   // a token slot of this CTA
        const int tl = tl0 + base + grp;
        const int t = t_begin + tl;
        const bool valid = mine && t < T;
        float s[EPL];
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int e = lg + G * j;
            s[j] = -INFINITY;
            if (valid && e < E) {
                float z;
                if (a.part) {
                    // partial sums in split order, loaded 8 at a time
                    z = 0.0f;
                    const float* pp = a.part + static_cast<size_t>(t) * E + e;
                    const size_t pstride = static_cast<size_t>(T) * E;
                    for (int sp0 = 0; sp0 < a.splits; sp0 += 8) {
                        float v[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            v[j] = (sp0 + j < a.splits) ? __ldg(pp + (sp0 + j) * pstride) : 0.0f;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (sp0 + j < a.splits) z += v[j];
                    }
                    if (a.bias) z += a.bias[e];
                } else {
                    z = a.logits_in[static_cast<size_t>(t) * E + e];
                }
                if (a.logits_out) a.logits_out[static_cast<size_t>(t) * E + e] = z;
                // the temperature divides the score before the penalty comes off
                float sc = (a.tau != 0.0f && a.tau != 1.0f) ? __fdiv_rn(z, a.tau) : z;
                if (a.usage && a.lambda != 0.0f) sc = __fsub_rn(sc, __fmul_rn(a.lambda, a.usage[e]));
                if (isnan(sc)) {
                    saw_nan = true;
                    sc = -INFINITY;  // ranks last; the call reports MOE_ERR_NONFINITE
                }
                if (a.scores_ws) a.scores_ws[static_cast<size_t>(t) * E + e] = sc;
                if (a.scores_user) a.scores_user[static_cast<size_t>(t) * E + e] = sc;
                s[j] = sc;
            }
        }
        // The token's preference order.  Up to 32 experts: each lane counts the
        // experts that rank before its own (all scores pass through the group by
        // shuffles).  More: a bitonic sort of the (score, index) keys across the
        // warp, element i = lane*EPL + j.
        int rank[EPL];
        float m = -INFINITY;
        float sv[EPL];
        int se[EPL];
        if (EPL == 1) {
            rank[0] = 0;
            for (int src = 0; src < G; ++src) {
                const float v = __shfl_sync(0xffffffffu, s[0], src, G);
                if (src < E) {
                    m = fmaxf(m, v);
                    rank[0] += ranks_before(v, src, s[0], lg) ? 1 : 0;
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                const int e = lg + G * j;
                sv[j] = (e < E) ? s[j] : -INFINITY;
                se[j] = (e < E) ? e : 0x7fff + e;   // absent experts sort last
                m = fmaxf(m, sv[j]);
            }
            for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            // network element i = lane*EPL + j (any starting placement sorts)
            constexpr int N = 32 * EPL;
#pragma unroll
            for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
                for (int stride = size >> 1; stride > 0; stride >>= 1) {
                    if (stride < EPL) {
#pragma unroll
                        for (int j = 0; j < EPL; ++j) {
                            const int pj = j ^ stride;
                            if (pj > j) {
                                const int i = lane * EPL + j;
                                const bool asc = (i & size) == 0;
                                const bool swap = asc ? ranks_before(sv[pj], se[pj], sv[j], se[j])
                                                      : ranks_before(sv[j], se[j], sv[pj], se[pj]);
                                if (swap) {
                                    const float tv = sv[j];
                                    sv[j] = sv[pj];
                                    sv[pj] = tv;
                                    const int te = se[j];
                                    se[j] = se[pj];
                                    se[pj] = te;
                                }
                            }
                        }
                    } else {
                        const int dl = stride / EPL;
#pragma unroll
                        for (int j = 0; j < EPL; ++j) {
                            const float ov = __shfl_xor_sync(0xffffffffu, sv[j], dl);
                            const int oe = __shfl_xor_sync(0xffffffffu, se[j], dl);
                            const int i = lane * EPL + j;
                            const bool asc = (i & size) == 0;
                            const bool low = (lane & dl) == 0;
                            const bool other_better = ranks_before(ov, oe, sv[j], se[j]);
                            if (other_better == (low == asc)) {
                                sv[j] = ov;
                                se[j] = oe;
                            }
                        }
                    }
                }
            }
        }
        // softmax over the token's experts
        float num[EPL];
        float part_sum = 0.0f;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int e = lg + G * j;
            num[j] = (e < E) ? softmax_num(s[j], m) : 0.0f;
            part_sum += num[j];
        }
        for (int off = G >> 1; off >= 1; off >>= 1)
            part_sum += __shfl_xor_sync(0xffffffffu, part_sum, off, G);
        const float zsum = part_sum;
        if (valid) {
            uint8_t* prow = a.prefs + static_cast<size_t>(t) * pref_stride(E);
#pragma unroll
            for (int j = 0; j < EPL; ++j) acc[j] += num[j] / zsum;
            if (EPL == 1) {
                for (int i = E + lg; i < kPrefLen; i += G) prow[i] = 255;   // pad short orders
                const int e = lg;
                if (e < E) {
                    prow[rank[0]] = static_cast<uint8_t>(e);
                    if (rank[0] < k) {
                        const size_t o = static_cast<size_t>(t) * k + rank[0];
                        a.ids_ws[o] = e;
                        if (a.ids_user) a.ids_user[o] = e;
                        if (a.topk_w) a.topk_w[o] = num[0] / zsum;
                        s_ids[tl * k + rank[0]] = static_cast<int16_t>(e);
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < EPL; ++j) {
                    const int pos = lane * EPL + j;   // sorted position
                    const int e = se[j];
                    if (pos < E) prow[pos] = static_cast<uint8_t>(e);
                    if (pos < k) {
                        const size_t o = static_cast<size_t>(t) * k + pos;
                        a.ids_ws[o] = e;
                        if (a.ids_user) a.ids_user[o] = e;
                        if (a.topk_w) a.topk_w[o] = softmax_num(sv[j], m) / zsum;
                        s_ids[tl * k + pos] = static_cast<int16_t>(e);
                    }
                }
            }
        } else if (mine && lg == 0) {
            for (int r = 0; r < k; ++r) s_ids[tl * k + r] = -1;
        }
    }
    if (saw_nan) s_nan = 1;

    // ---- P partial of this chunk: lanes -> warp (fixed order) -> chunk
#pragma unroll
    for (int j = 0; j < EPL; ++j)
        for (int off = G; off < 32; off <<= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], off);
    if (lane < G) {
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int e = lg + G * j;
            if (e < E) s_wsum[warp][e] = acc[j];
        }
    }
    for (int e = threadIdx.x; e < E; e += kRouteThreads)
        for (int w = 0; w < kRankWarps; ++w) s_wcnt[w][e] = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kRouteThreads) {
        float tot = 0.0f;
        for (int w = 0; w < kRouteWarps; ++w) tot += s_wsum[w][e];
        if (cs == 1)
            a.ppart[static_cast<size_t>(chunk) * E + e] = tot;
        else
            s_psum[e] = tot;
    }
    if (threadIdx.x == 0 && s_nan) record_error(a.status, MOE_ERR_NONFINITE);

    // ---- per rank: histogram of picks and stable rank within the chunk (the
    // first `sub` threads, one token each; the other warps only join the
    // barriers).  Within the CTA: in-warp rank + the earlier warps' counts;
    // across the cluster: + the picks of the chunk's earlier CTAs.
    const bool ranker = threadIdx.x < sub;
    const int tl = tl0 + threadIdx.x;
    const int t = t_begin + tl;
    for (int r = 0; r < k; ++r) {
        int e = -1, rnk = 0;
        if (ranker) {
            e = s_ids[tl * k + r];
            const uint32_t peers = __match_any_sync(0xffffffffu, e);
            rnk = __popc(peers & lanemask_lt());
            if (e >= 0 && lane == __ffs(peers) - 1) s_wcnt[warp][e] = __popc(peers);
        }
        __syncthreads();
        for (int ee = threadIdx.x; ee < E; ee += kRouteThreads) {
            int run = 0;
            for (int w = 0; w < kRankWarps; ++w) {
                const int c = s_wcnt[w][ee];
                s_wcnt[w][ee] = run;  // exclusive prefix over warps
                run += c;
            }
            if (cs == 1)
                a.hist[(static_cast<size_t>(r) * a.nchunks + chunk) * E + ee] = run;
            else
                s_ctot[r][ee] = run;
        }
        __syncthreads();
        if (ranker && e >= 0) {
            const int c = s_wcnt[warp][e] + rnk;   // rank among this CTA's picks
            if (cs == 1) {
                if (t < T) a.crank[static_cast<size_t>(t) * k + r] = c;
            } else {
                s_crl[threadIdx.x * 8 + r] = static_cast<int16_t>(c);
            }
        }
        __syncthreads();
        for (int ee = threadIdx.x; ee < E; ee += kRouteThreads)
            for (int w = 0; w < kRankWarps; ++w) s_wcnt[w][ee] = 0;
        __syncthreads();
    }
    if (cs == 1) return;
    cluster_sync_all();   // every CTA's totals are in place
    if (ranker && t < T) {
        for (int r = 0; r < k; ++r) {
            const int e = s_ids[tl * k + r];
            if (e < 0) continue;
            int base = 0;
            for (int c = 0; c < cr; ++c) base += ld_cluster_s32(map_to_rank(smem_u32(&s_ctot[r][e]), c));
            a.crank[static_cast<size_t>(t) * k + r] = base + s_crl[threadIdx.x * 8 + r];
        }
    }
    if (cr == cs - 1) {
        // the chunk's histogram: all CTAs' picks, in CTA order
        for (int i = threadIdx.x; i < k * E; i += kRouteThreads) {
            const int r = i / E, ee = i - r * E;
            int tot = 0;
            for (int c = 0; c < cs; ++c)
                tot += (c == cr) ? s_ctot[r][ee] : ld_cluster_s32(map_to_rank(smem_u32(&s_ctot[r][ee]), c));
            a.hist[(static_cast<size_t>(r) * a.nchunks + chunk) * E + ee] = tot;
        }
    }
    if (cr == 0) {
        // the chunk's probability sums, in CTA order
        for (int ee = threadIdx.x; ee < E; ee += kRouteThreads) {
            float tot = s_psum[ee];
            for (int c = 1; c < cs; ++c) tot += ld_cluster_f32(map_to_rank(smem_u32(&s_psum[ee]), c));
            a.ppart[static_cast<size_t>(chunk) * E + ee] = tot;
        }
    }
    cluster_sync_all();   // no CTA leaves while another reads its shared memory
}


}  // namespace detail
}  // namespace moe
