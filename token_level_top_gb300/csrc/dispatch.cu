// dispatch.cu -- capacity-capped dispatch with overflow reroute and drop.
//
// Semantics ([mhpn] §2.3, third check "硬性容量截断"; [2kiu] §2; [coreui]
// §3.3 and §5.2): entries (t, r) are placed in the order rank-major,
// token-minor -- every rank-0 pick before any rank-1 pick, tokens in index
// order.  Each entry takes the first expert of its token's preference order
// that is not full (fill < C) and not already serving the token; if none is
// left the entry is dropped.  Slot = the expert's fill count at that moment.
//
// Parallel form.  A full expert stays full, so between two "fill events" the
// set of full experts is constant and every entry's choice depends only on it
// and on its own token's earlier ranks.  Before the first event every entry
// takes its plain top-k pick, so its slot is (picks of that expert in earlier
// chunks) + (stable rank inside its chunk) -- both written by the route
// kernel.  Stage 1 (one CTA) scans the chunk histograms per expert, finds the
// first chunk q1 in which some expert's running count passes C, and leaves
// the per-chunk bases.  From chunk q1 on, 8 warps of the CTA (256 threads,
// synchronised on named barrier 1) replay the entries in windows of 256
// consecutive entries of one rank, one per thread, in rounds.  Each expert has
// a fill position in the window: the position of the entry that takes its last
// slot (-1 when it was full before the window, none when it does not fill).
// In a round every entry picks its expert with the experts whose fill position
// lies before it counted as full, __match_any_sync gives its rank among its
// warp's entries of that expert and each warp adds the earlier warps' counts
// (slot = fill + rank), and the entry with slot C-1 records the expert's new
// fill position.  Rounds repeat until the positions reproduce themselves; such a
// fixed point is the sequential fill, and each round settles the next fill in
// window order (every entry before it sees exactly the experts full at its
// turn, the other positions never lying before their true ones), so a window
// takes at most one round per fill in it, plus one; fills that do not interact
// settle in the same round.  The window then commits.  Stage 2 (grid-wide) writes the entries
// before q1, the permutation in slot order and the combine weights
// ([mhpn] §4.3: router probabilities renormalised over the experts used).
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "route_block.cuh"

namespace moe {
namespace {

constexpr int kSerialThreads = 1024;   // stage 1 and the staging
constexpr int kReplayThreads = 256;    // the replay: one window entry per thread
constexpr int kReplayWarps = kReplayThreads / 32;
static_assert(kSerialThreads >= 255, "stage 1 needs a thread per expert");
static_assert(kReplayThreads <= kSerialThreads && kReplayThreads % 32 == 0 && kReplayThreads >= 256,
              "replay warps; a thread per expert in the fill-position updates");
// dynamic shared memory of the standalone replay block (+ about 14 KB static)
constexpr size_t kSerialSmemCap = 208 * 1024;

// Barrier among the replay's threads only (named barrier 1).
__device__ __forceinline__ void replay_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kReplayThreads) : "memory");
}

// Barrier 1 among the replay's threads that also returns whether `pred` holds in any of them.
__device__ __forceinline__ bool replay_any(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "n"(kReplayThreads)
        : "memory");
    return r != 0;
}

struct SerialArgs {
    DispatchArgs a;
    int stage_cap;        // bytes of dynamic shared memory for the staged tail
    uint8_t* asg_global;  // [T*k] fallback when the staging does not fit in smem
};

// Read-only loads through the non-coherent cache, except where the data was
// written earlier in the same kernel (the fused small-batch kernel), which
// needs plain loads.
template <bool NC, typename V>
__device__ __forceinline__ V ld_in(const V* p)
{
    if constexpr (NC)
        return __ldg(p);
    else
        return *p;
}

// Experts already serving a token (its earlier ranks), one per byte in two
// words; unused bytes hold 0xFF.
struct Held {
    uint32_t lo = 0xFFFFFFFFu, hi = 0xFFFFFFFFu;
    int n = 0;
    __device__ __forceinline__ void add(int e)
    {
        const uint32_t sh = 8 * (n & 3), m = ~(0xFFu << sh), v = static_cast<uint32_t>(e & 0xFF) << sh;
        if (n < 4)
            lo = (lo & m) | v;
        else
            hi = (hi & m) | v;
        ++n;
    }
    __device__ __forceinline__ uint32_t get(int q) const { return ((q < 4 ? lo : hi) >> (8 * (q & 3))) & 0xFF; }
};

// Bit j of the result = bit 7 of byte j of x (the four products land on bits
// 28..31 without overlapping any other partial product).
__device__ __forceinline__ uint32_t byte_msbs(uint32_t x)
{
    return ((x & 0x80808080u) * 0x00204081u) >> 28;
}

// First of 16 order positions (the low n valid) whose expert is neither full
// for the entry at window position `pos` (s_fillpos[e] < pos: the entry taking
// the expert's last slot comes before it, -1 for experts full before the
// window) nor held, or -1.  Every position is looked at without an early exit,
// so the 16 loads overlap; the held test compares 4 positions at a time.
__device__ __forceinline__ int first_open16(const uint4 v, int n, const Held& held,
                                            const int16_t* s_fillpos, int pos)
{
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    uint32_t closed = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        closed |= static_cast<uint32_t>(s_fillpos[(wd[i >> 2] >> (8 * (i & 3))) & 0xFF] < pos) << i;
    for (int q = 0; q < held.n; ++q) {
        const uint32_t rep = held.get(q) * 0x01010101u;
#pragma unroll
        for (int j = 0; j < 4; ++j) closed |= byte_msbs(__vcmpeq4(wd[j], rep)) << (4 * j);
    }
    const uint32_t ok = ~closed & (n >= 16 ? 0xFFFFu : (1u << n) - 1u);
    if (!ok) return -1;
    const int i = __ffs(ok) - 1;
    const uint32_t w = i < 4 ? v.x : i < 8 ? v.y : i < 12 ? v.z : v.w;
    return (w >> (8 * (i & 3))) & 0xFF;
}

// First expert of the token's preference order that is neither full nor
// held.  prow holds the first nw 16-position words of the order (staged in
// shared memory, or the stored row itself); the rest is read from the stored
// order in global memory.
template <bool NC>
__device__ __forceinline__ int choose_expert(const DispatchArgs& a, int t, const uint4* prow, int nw,
                                             const Held& held, const int16_t* s_fillpos, int pos)
{
    const int E = a.E;
    for (int w = 0; w < nw; ++w) {
        const int p0 = 16 * w;
        if (p0 >= E) return -1;
        const int e = first_open16(prow[w], min(16, E - p0), held, s_fillpos, pos);
        if (e >= 0) return e;
    }
    const uint4* orow = reinterpret_cast<const uint4*>(a.prefs + static_cast<size_t>(t) * pref_stride(E));
    for (int p0 = 16 * nw; p0 < E; p0 += 16) {
        const int e = first_open16(ld_in<NC>(orow + p0 / 16), min(16, E - p0), held, s_fillpos, pos);
        if (e >= 0) return e;
    }
    return -1;
}

// Stage 1 and the replay, by one block of kSerialThreads threads (the replay
// itself by its first kReplayThreads); dsm is the block's dynamic shared
// memory (sa.stage_cap bytes for the staged tail).
template <bool NC>
__device__ __forceinline__ void dispatch_serial_block(const SerialArgs& sa, uint8_t* dsm)
{
    __shared__ int s_fill[256];
    __shared__ uint8_t s_isfull[256];       // 1 for a full expert (and for ids >= E)
    __shared__ int s_seg[kSerialThreads];   // stage 1: per (segment, expert) counts
    __shared__ int s_tot[256];
    __shared__ int s_cnt[kReplayWarps * 256];   // replay: per (warp, expert) window counts
    __shared__ int16_t s_fpos[256];        // replay: window position that fills each expert
    __shared__ int16_t s_fnext[256];       // the same from the current round's choices
    __shared__ int s_q1, s_nre, s_ndrop;
    const DispatchArgs& a = sa.a;
    const int E = a.E, T = a.T, k = a.k, nch = a.nchunks;
    const int Q = k * nch;
    const int cap = static_cast<int>(a.C);   // C <= T*k < 2^30
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- stage 1: running count per expert over the chunk rows q (rank-major
    // order).  Thread (j, e) = tid j*E + e sums rows [j*L, (j+1)*L) of expert e;
    // a scan over the segments gives each its start; a second pass writes the
    // bases and finds the first row whose running count passes C.
    const int S = min(min(32, kSerialThreads / E), Q);   // segments per expert
    const int L = (Q + S - 1) / S;
    const int seg = tid / E, se = tid - seg * E;
    const bool segt = seg < S;
    const int32_t* hist = a.hist;
    if (tid == 0) {
        s_q1 = Q;
        s_nre = 0;
        s_ndrop = 0;
    }
    for (int i = tid; i < kReplayWarps * E; i += kSerialThreads) s_cnt[i] = 0;
    int part = 0;
    if (segt) {
        const int q_end = min(Q, (seg + 1) * L);
        for (int q0 = seg * L; q0 < q_end; q0 += 8) {
            int c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                c[j] = (q0 + j < q_end) ? ld_in<NC>(hist + static_cast<size_t>(q0 + j) * E + se) : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) part += c[j];
        }
        s_seg[seg * E + se] = part;
    }
    __syncthreads();
    if (tid < E) {
        int run = 0;
        for (int j = 0; j < S; ++j) {
            const int c = s_seg[j * E + tid];
            s_seg[j * E + tid] = run;
            run += c;
        }
        s_tot[tid] = run;
    }
    __syncthreads();
    if (segt) {
        int32_t* __restrict__ basep = a.base;
        int cum = s_seg[seg * E + se], qe = Q;
        const int q_end = min(Q, (seg + 1) * L);
        for (int q0 = seg * L; q0 < q_end; q0 += 8) {
            int c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                c[j] = (q0 + j < q_end) ? ld_in<NC>(hist + static_cast<size_t>(q0 + j) * E + se) : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (q0 + j >= q_end) break;
                basep[static_cast<size_t>(q0 + j) * E + se] = cum;
                cum += c[j];
                if (qe == Q && cum > a.C) qe = q0 + j;
            }
        }
        if (qe < Q) atomicMin(&s_q1, qe);
    }
    __syncthreads();
    const int q1 = s_q1;
    if (tid < E) s_fill[tid] = (q1 < Q) ? a.base[static_cast<size_t>(q1) * E + tid] : s_tot[tid];
    if (tid < 256) s_isfull[tid] = (tid >= E || s_fill[tid] >= cap) ? 1 : 0;   // own s_fill entry

    // ---- stage the tail tokens' preference orders (as many leading 16-byte
    // words as fit) and their entries' experts in shared memory; when not even
    // one word fits, the orders stay in global memory and the experts go to
    // the global fallback
    const int r1 = q1 / nch;
    const int t1 = (q1 - r1 * nch) * kChunk;
    const int tbeg = (q1 < Q && r1 == k - 1) ? t1 : 0;   // first token with a tail entry
    const int ntail = (q1 < Q) ? T - tbeg : 0;
    const int pst16 = pref_stride(E) / 16;   // uint4 words per stored order
    const uint4* pfx = reinterpret_cast<const uint4*>(a.prefs) + static_cast<size_t>(tbeg) * pst16;
    int nw = pst16;                          // words of each order reachable through pfx
    uint8_t* asg = sa.asg_global;
    if (ntail > 0) {
        const int room = sa.stage_cap / ntail - k;   // bytes per token for its order
        const int fit = room >= 16 ? min(room / 16, pst16) : 0;
        if (fit > 0) {
            uint4* sp = reinterpret_cast<uint4*>(dsm);
            const int nwords = ntail * fit;
            for (int i0 = tid; i0 < nwords; i0 += 4 * kSerialThreads) {
                uint4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int i = i0 + j * kSerialThreads;
                    if (i < nwords) v[j] = pfx[static_cast<size_t>(i / fit) * pst16 + i % fit];
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int i = i0 + j * kSerialThreads;
                    if (i < nwords) sp[i] = v[j];
                }
            }
            pfx = sp;
            nw = fit;
            asg = dsm + static_cast<size_t>(nwords) * 16;
        }
        // entry (t, r) is placed before the tail when its chunk r*nch + t/kChunk < q1
        const int32_t* ids = a.ids;
        for (int r = 0; r < k; ++r) {
            for (int t0 = tbeg + tid; t0 < T; t0 += 4 * kSerialThreads) {
                uint8_t v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = t0 + j * kSerialThreads;
                    v[j] = 255;
                    if (t < T && r * nch + (t >> 8) < q1)
                        v[j] = static_cast<uint8_t>(ld_in<NC>(ids + static_cast<size_t>(t) * k + r));
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = t0 + j * kSerialThreads;
                    if (t < T) asg[static_cast<size_t>(t - tbeg) * k + r] = v[j];
                }
            }
        }
    }
    static_assert(kChunk == 256, "chunk index is t >> 8");
    __syncthreads();

    if (tid >= kReplayThreads) return;   // the replay and the totals belong to the first warps

    // ---- stage 2: replay from chunk q1, kReplayThreads consecutive entries of
    // one rank per window; see the file comment.
    int nre = 0, ndrop = 0;
    if (q1 < Q) {
        for (int r = r1; r < k; ++r) {
            for (int w0 = (r == r1 ? t1 : 0); w0 < T; w0 += kReplayThreads) {
                const int t = w0 + tid;
                const bool valid = t < T;
                const size_t ti = static_cast<size_t>(valid ? t - tbeg : 0);
                const uint4* prow = pfx + ti * nw;
                Held held;
                int want = -1;
                if (valid) {
                    for (int q = 0; q < r; ++q) held.add(asg[ti * k + q]);
                    const uint4 w = prow[0];   // r < k <= 8: the first word holds rank r's pick
                    want = ((r < 4 ? w.x : w.y) >> (8 * (r & 3))) & 0xFF;
                }
                // fill positions: -1 for experts full before the window, none yet for the rest
                if (tid < 256) {
                    s_fpos[tid] = s_isfull[tid] ? -1 : kReplayThreads;
                    s_fnext[tid] = kReplayThreads;
                }
                replay_sync();
                int e = -1, slot = 0;
                uint32_t peers = 0;
                bool leader = false;
                for (int round = 0;; ++round) {
                    // every entry chooses under the current fill positions
                    e = valid ? choose_expert<NC>(a, t, prow, nw, held, s_fpos, tid) : -1;
                    peers = __match_any_sync(0xffffffffu, valid ? e : -2);
                    const int rnk = __popc(peers & lanemask_lt());
                    leader = lane == __ffs(peers) - 1;
                    const bool placed = valid && e >= 0;
                    if (placed && leader) s_cnt[warp * E + e] = __popc(peers);
                    replay_sync();
                    // slot = fill + the earlier warps' entries of the expert + rank in the warp
                    slot = 0;
                    if (placed) {
                        slot = s_fill[e] + rnk;
#pragma unroll
                        for (int w = 0; w < kReplayWarps - 1; ++w)
                            if (w < warp) slot += s_cnt[w * E + e];
                        if (slot == cap - 1) s_fnext[e] = static_cast<int16_t>(tid);   // takes the last slot
                    }
                    replay_sync();
                    if (placed && leader) s_cnt[warp * E + e] = 0;   // all reads are done
                    bool moved = false;
                    if (tid < 256) {
                        if (s_fpos[tid] >= 0 && s_fnext[tid] != s_fpos[tid]) {
                            moved = true;
                            s_fpos[tid] = s_fnext[tid];
                        }
                        s_fnext[tid] = kReplayThreads;
                    }
                    if (!replay_any(moved)) break;   // the choices reproduce their own fill positions
                    if (round > E) {                 // unreachable: each round fixes the next fill in order
                        if (tid == 0) record_error(a.status, MOE_ERR_TIMEOUT);
                        break;
                    }
                }
                // commit the window
                if (valid) {
                    const size_t idx = static_cast<size_t>(t) * k + r;
                    const size_t li = static_cast<size_t>(t - tbeg) * k + r;
                    if (e >= 0) {
                        const int fl = (e != want) ? 1 : 0;
                        a.assign[idx] = e;
                        a.slot[idx] = slot;
                        a.flags[idx] = static_cast<uint8_t>(fl);
                        asg[li] = static_cast<uint8_t>(e);
                        nre += fl;
                    } else {
                        a.assign[idx] = -1;
                        a.slot[idx] = -1;
                        a.flags[idx] = 2;
                        asg[li] = 255;
                        ++ndrop;
                    }
                }
                if (valid && e >= 0 && leader) {
                    const int nc = __popc(peers);
                    if (atomicAdd(&s_fill[e], nc) + nc >= cap) s_isfull[e] = 1;
                }
                replay_sync();
            }
        }
    }
    for (int off = 16; off >= 1; off >>= 1) {
        nre += __shfl_xor_sync(0xffffffffu, nre, off);
        ndrop += __shfl_xor_sync(0xffffffffu, ndrop, off);
    }
    if (lane == 0) {
        atomicAdd(&s_nre, nre);
        atomicAdd(&s_ndrop, ndrop);
    }
    replay_sync();
    if (warp != 0) return;
    nre = s_nre;
    ndrop = s_ndrop;
    if (lane == 0) {
        a.ctrl[CTRL_Q1] = q1;
        a.ctrl[CTRL_NRE] = nre;
        a.ctrl[CTRL_NDROP] = ndrop;
        if (a.n_rerouted) *a.n_rerouted = nre;
        if (a.n_dropped) *a.n_dropped = ndrop;
    }
    // counts and exclusive offsets
    int carry = 0;
    for (int b = 0; b < E; b += 32) {
        const int e = b + lane;
        const int c = (e < E) ? s_fill[e] : 0;
        int incl = c;
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (e < E) {
            a.counts[e] = c;
            a.offsets[e] = carry + incl - c;
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) a.offsets[E] = carry;
}

__global__ void __launch_bounds__(kSerialThreads, 1) dispatch_serial_kernel(const SerialArgs sa)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    dispatch_serial_block<true>(sa, dsm);
}

// Token t's entries before the replay, its permutation entries and its
// combine weights.
__device__ __forceinline__ void dispatch_finish_token(const DispatchArgs& a, const int t)
{
    const int E = a.E, k = a.k;
    const int q1 = a.ctrl[CTRL_Q1];
    const int c = t / kChunk;
    int es[8];
    for (int r = 0; r < k; ++r) {
        const size_t idx = static_cast<size_t>(t) * k + r;
        const int q = r * a.nchunks + c;
        int e, sl;
        if (q < q1) {
            e = a.ids[idx];
            sl = a.base[static_cast<size_t>(q) * E + e] + a.crank[idx];
            a.assign[idx] = e;
            a.slot[idx] = sl;
            a.flags[idx] = 0;
        } else {
            e = a.assign[idx];
            sl = a.slot[idx];
        }
        es[r] = e;
        if (e >= 0) a.perm[a.offsets[e] + sl] = static_cast<int32_t>(idx);
    }
    // combine weights: p of each kept expert renormalised over the kept ones
    const float* srow = a.scores + static_cast<size_t>(t) * E;
    const int top = a.prefs[static_cast<size_t>(t) * pref_stride(E)];
    float mg = srow[top];
    if (isnan(mg)) mg = -INFINITY;
    float mk = -INFINITY;
    float sv[8];
    for (int r = 0; r < k; ++r) {
        sv[r] = -INFINITY;
        if (es[r] >= 0) {
            float s = srow[es[r]];
            if (isnan(s)) s = -INFINITY;
            sv[r] = s;
            mk = fmaxf(mk, s);
        }
    }
    float num[8];
    float tot = 0.0f;
    for (int r = 0; r < k; ++r) {
        float n = 0.0f;
        if (es[r] >= 0) {
            if (mg == INFINITY)
                n = (sv[r] == INFINITY) ? 1.0f : 0.0f;
            else if (mg == -INFINITY)
                n = 1.0f;
            else
                n = expf(sv[r] - mk);
        }
        num[r] = n;
        tot += n;
    }
    for (int r = 0; r < k; ++r)
        a.cw[static_cast<size_t>(t) * k + r] = (tot > 0.0f) ? num[r] / tot : 0.0f;
}

__global__ void dispatch_finish_kernel(const DispatchArgs a)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < a.T) dispatch_finish_token(a, t);
}

// A batch of one chunk (T <= kChunk) in one block: route, replay and finish
// with block barriers between them instead of three launches.
static_assert(detail::kRouteThreads == kSerialThreads, "one block runs both phases");
static_assert(kChunk <= detail::kRouteThreads, "one token per thread in the finish phase");

template <int EPL>
__global__ void __launch_bounds__(detail::kRouteThreads, 1)
    route_dispatch_small_kernel(const RouteArgs ra, const SerialArgs sa)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    detail::route_block<EPL>(ra, 0, 1, 0);
    __syncthreads();
    dispatch_serial_block<false>(sa, dsm);   // the replay warps return last
    __syncthreads();
    if (static_cast<int>(threadIdx.x) < sa.a.T) dispatch_finish_token(sa.a, threadIdx.x);
}

constexpr size_t kSmallSmemCap = 68 * 1024;   // >= kChunk*(pref_stride(255) + 8)

template <int EPL>
cudaError_t launch_small(const RouteArgs& ra, const SerialArgs& sa, size_t smem, cudaStream_t s)
{
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(route_dispatch_small_kernel<EPL>),
                                      static_cast<int>(kSmallSmemCap));
    if (e != cudaSuccess) return e;
    route_dispatch_small_kernel<EPL><<<1, detail::kRouteThreads, smem, s>>>(ra, sa);
    return cudaGetLastError();
}

}  // namespace

namespace {

// Without room in shared memory the replay keeps its per-entry experts in the
// (otherwise unused) tail of the rank-base table.
void set_fallback(SerialArgs& sa)
{
    const DispatchArgs& a = sa.a;
    uint8_t* b = reinterpret_cast<uint8_t*>(a.base);
    sa.asg_global = b + dispatch_asg_offset(a.k, a.nchunks, a.E);
}

}  // namespace

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s)
{
    if (a.T <= 0) return cudaSuccess;
    SerialArgs sa;
    sa.a = a;
    // room for the largest possible tail (every token), up to the cap; the
    // block decides from the actual tail whether it fits
    const size_t need = static_cast<size_t>(a.T) * (pref_stride(a.E) + a.k);
    const size_t smem = need < kSerialSmemCap ? need : kSerialSmemCap;
    sa.stage_cap = static_cast<int>(smem);
    set_fallback(sa);
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(dispatch_serial_kernel),
                                      static_cast<int>(kSerialSmemCap));
    if (e != cudaSuccess) return e;
    dispatch_serial_kernel<<<1, kSerialThreads, smem, s>>>(sa);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dispatch_finish_kernel<<<(a.T + 255) / 256, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_route_dispatch_small(const RouteArgs& ra, const DispatchArgs& a, cudaStream_t s)
{
    if (a.T <= 0) return cudaSuccess;
    if (a.T > kChunk || ra.nchunks != 1 || a.nchunks != 1) return cudaErrorInvalidValue;
    SerialArgs sa;
    sa.a = a;
    const size_t smem = static_cast<size_t>(a.T) * (pref_stride(a.E) + a.k);
    if (smem > kSmallSmemCap) return cudaErrorInvalidValue;
    sa.stage_cap = static_cast<int>(smem);
    set_fallback(sa);
    if (a.E <= 32) return launch_small<1>(ra, sa, smem, s);
    if (a.E <= 64) return launch_small<2>(ra, sa, smem, s);
    if (a.E <= 128) return launch_small<4>(ra, sa, smem, s);
    return launch_small<8>(ra, sa, smem, s);
}

}  // namespace moe
