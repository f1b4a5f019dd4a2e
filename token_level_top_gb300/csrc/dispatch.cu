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
// the per-chunk bases.  From chunk q1 on, the CTA replays the entries in
// windows of 256 consecutive entries of one rank, one per thread: each entry
// picks its expert under the current full set, __match_any_sync and a prefix
// over the warps give it its slot, a block minimum finds the first entry that
// takes an expert's last slot, everything up to it commits, and entries after
// it that chose the now-full expert choose again.  Stage 2 (grid-wide) writes the entries
// before q1, the permutation in slot order and the combine weights
// ([mhpn] §4.3: router probabilities renormalised over the experts used).
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "route_block.cuh"

namespace moe {
namespace {

constexpr int kSerialThreads = 1024;  // one replay window = one entry per thread
constexpr int kSerialWarps = kSerialThreads / 32;
constexpr size_t kSerialSmemCap = 224 * 1024;  // dynamic shared memory of the replay CTA

struct SerialArgs {
    DispatchArgs a;
    int use_smem;
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

// Experts already serving a token (its earlier ranks), packed one per byte
// into two words; unused bytes hold 0xFF, which is never an expert id.
struct Held {
    uint32_t lo = 0xFFFFFFFFu, hi = 0xFFFFFFFFu;
    __device__ __forceinline__ void set(int q, int e)
    {
        const uint32_t sh = 8 * (q & 3), m = ~(0xFFu << sh), v = static_cast<uint32_t>(e & 0xFF) << sh;
        if (q < 4)
            lo = (lo & m) | v;
        else
            hi = (hi & m) | v;
    }
    __device__ __forceinline__ bool has(int e) const
    {
        const uint32_t b = 0x01010101u * static_cast<uint32_t>(e);
        const uint32_t x = lo ^ b, y = hi ^ b;   // a zero byte marks a match
        return (((x - 0x01010101u) & ~x) | ((y - 0x01010101u) & ~y)) & 0x80808080u;
    }
};

// First expert of the preference order that is neither full nor held.  The
// first kPrefLen entries come from the token's staged prefix (16 bytes in
// registers); past it the stored order is read 16 entries at a time.
template <bool NC>
__device__ __forceinline__ int choose_expert(const DispatchArgs& a, int cap, int t, const uint4 pw,
                                             const Held& held, const int* s_fill)
{
    const int E = a.E;
    const int L = E < kPrefLen ? E : kPrefLen;
    const uint32_t words[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
    for (int i = 0; i < kPrefLen; ++i) {
        if (i >= L) break;
        const int e = (words[i >> 2] >> (8 * (i & 3))) & 0xFF;
        if (s_fill[e] < cap && !held.has(e)) return e;
    }
    if (L == E) return -1;
    const uint8_t* orow = a.prefs + static_cast<size_t>(t) * pref_stride(E);
    for (int p0 = kPrefLen; p0 < E; p0 += 16) {
        const uint4 w = ld_in<NC>(reinterpret_cast<const uint4*>(orow + p0));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (p0 + i >= E) return -1;
            const int e = (ww[i >> 2] >> (8 * (i & 3))) & 0xFF;
            if (s_fill[e] < cap && !held.has(e)) return e;
        }
    }
    return -1;
}

// The replay, by one block of kSerialThreads threads; dsm is the block's
// dynamic shared memory (sized by the launchers below).
template <bool NC>
__device__ __forceinline__ void dispatch_serial_block(const SerialArgs& sa, uint8_t* dsm)
{
    __shared__ int s_fill[256];
    __shared__ int s_q1, s_cut, s_estar, s_nre, s_ndrop;
    const DispatchArgs& a = sa.a;
    const int E = a.E, T = a.T, k = a.k, nch = a.nchunks;
    const int Q = k * nch;
    const int cap = static_cast<int>(a.C);   // C <= T*k < 2^30
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // dynamic shared memory: per expert and warp, the window's entry counts and
    // their exclusive prefix (+ fill); then the staged tail data
    int (*s_cnt)[kSerialWarps] = reinterpret_cast<int (*)[kSerialWarps]>(dsm);
    int (*s_base)[kSerialWarps] = reinterpret_cast<int (*)[kSerialWarps]>(dsm + E * kSerialWarps * 4);
    uint8_t* stage = dsm + 2 * E * kSerialWarps * 4;

    if (tid == 0) {
        s_q1 = Q;
        s_cut = kSerialThreads;
        s_nre = 0;
        s_ndrop = 0;
    }
    for (int i = tid; i < kSerialWarps * E; i += kSerialThreads) (&s_cnt[0][0])[i] = 0;
    static_assert(kSerialWarps == 32, "the cross-warp scan maps one warp count to each lane");
    __syncthreads();
    // ---- stage 1: running count per expert over chunks (rank-major order)
    int total = 0;
    if (tid < E) {
        const int32_t* hist = a.hist;
        int32_t* __restrict__ basep = a.base;
        int cum = 0, qe = Q;
        for (int q0 = 0; q0 < Q; q0 += 16) {
            int c[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                c[j] = (q0 + j < Q) ? ld_in<NC>(hist + static_cast<size_t>(q0 + j) * E + tid) : 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (q0 + j >= Q) break;
                basep[static_cast<size_t>(q0 + j) * E + tid] = cum;
                cum += c[j];
                if (qe == Q && cum > a.C) qe = q0 + j;
            }
        }
        total = cum;
        atomicMin(&s_q1, qe);
    }
    __syncthreads();
    const int q1 = s_q1;
    if (tid < E) s_fill[tid] = (q1 < Q) ? a.base[static_cast<size_t>(q1) * E + tid] : total;

    // ---- stage the tail tokens' preference prefixes and their entries' experts
    const int r1 = q1 / nch;
    const int t1 = (q1 - r1 * nch) * kChunk;
    const int tbeg = (q1 < Q && r1 == k - 1) ? t1 : 0;   // first token with a tail entry
    const int ntail = (q1 < Q) ? T - tbeg : 0;
    const int pst16 = pref_stride(E) / 16;   // uint4 words per stored order
    const uint4* pfx_g = reinterpret_cast<const uint4*>(a.prefs) +
                                      static_cast<size_t>(tbeg) * pst16;
    const uint4* pfx = pfx_g;
    int pfx_step = pst16;                    // staged copies keep only the first 16 bytes
    uint8_t* asg = sa.asg_global;
    if (sa.use_smem && ntail > 0) {
        uint4* sp = reinterpret_cast<uint4*>(stage);
        for (int i0 = tid; i0 < ntail; i0 += 4 * kSerialThreads) {
            uint4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * kSerialThreads;
                if (i < ntail) v[j] = pfx_g[static_cast<size_t>(i) * pst16];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * kSerialThreads;
                if (i < ntail) sp[i] = v[j];
            }
        }
        pfx = sp;
        pfx_step = 1;
        asg = stage + static_cast<size_t>(ntail) * kPrefLen;
    }
    if (ntail > 0) {
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

    // ---- stage 2: replay from chunk q1, kSerialThreads consecutive entries of one rank
    // per window; see the file comment.
    int nre = 0, ndrop = 0;
    if (q1 < Q) {
        for (int r = r1; r < k; ++r) {
            for (int w0 = (r == r1 ? t1 : 0); w0 < T; w0 += kSerialThreads) {
                const int t = w0 + tid;
                const bool valid = t < T;
                uint4 pw = make_uint4(0, 0, 0, 0);
                Held held;
                if (valid) {
                    pw = pfx[static_cast<size_t>(t - tbeg) * pfx_step];
                    for (int q = 0; q < r; ++q) held.set(q, asg[static_cast<size_t>(t - tbeg) * k + q]);
                }
                const int want = (valid && r < kPrefLen)
                                     ? (int)(((r < 4 ? pw.x : r < 8 ? pw.y : r < 12 ? pw.z : pw.w) >>
                                              (8 * (r & 3))) & 0xFF)
                                     : -1;
                int e = valid ? choose_expert<NC>(a, cap, t, pw, held, s_fill) : -1;
                bool active = valid;
                while (true) {
                    // ranks among the window's active entries that chose the same expert
                    const int key = active ? e : -2;
                    const uint32_t peers = __match_any_sync(0xffffffffu, key);
                    const int rnk = __popc(peers & lanemask_lt());
                    const bool leader = lane == __ffs(peers) - 1;
                    if (active && e >= 0 && leader) s_cnt[e][warp] = __popc(peers);
                    __syncthreads();
                    // per expert, exclusive prefix over the warps (lane w holds warp w)
                    for (int ee = warp; ee < E; ee += kSerialWarps) {
                        const int c = s_cnt[ee][lane];
                        int incl = c;
#pragma unroll
                        for (int off = 1; off < 32; off <<= 1) {
                            const int v = __shfl_up_sync(0xffffffffu, incl, off);
                            if (lane >= off) incl += v;
                        }
                        s_base[ee][lane] = s_fill[ee] + incl - c;
                    }
                    __syncthreads();
                    int slot = 0;
                    if (active && e >= 0) {
                        slot = s_base[e][warp] + rnk;
                        if (leader) s_cnt[e][warp] = 0;   // ready for the next round
                    }
                    // the first entry of the window that takes an expert's last slot
                    const bool last = active && e >= 0 && slot + 1 == cap;
                    const uint32_t evw = __ballot_sync(0xffffffffu, last);
                    if (evw && lane == 0) atomicMin(&s_cut, warp * 32 + __ffs(evw) - 1);
                    __syncthreads();
                    const int cut = s_cut;
                    const bool commit = active && tid <= cut;
                    if (commit) {
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
                    if (tid == cut) s_estar = e;
                    // new fill: each warp's leader adds its committed entries of the expert
                    const uint32_t cmask = __ballot_sync(0xffffffffu, commit);
                    if (active && e >= 0 && leader) {
                        const int nc = __popc(peers & cmask);
                        if (nc) atomicAdd(&s_fill[e], nc);
                    }
                    __syncthreads();
                    if (cut >= kSerialThreads) break;   // no expert filled in this window
                    const int estar = s_estar;
                    active = active && tid > cut;
                    if (active && e == estar) e = choose_expert<NC>(a, cap, t, pw, held, s_fill);
                    if (tid == 0) s_cut = kSerialThreads;   // read by all before the last barrier
                }
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
    __syncthreads();
    if (warp == 0) {
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
static_assert(kChunk <= kSerialThreads, "one token per thread in the finish phase");

template <int EPL>
__global__ void __launch_bounds__(kSerialThreads, 1)
    route_dispatch_small_kernel(const RouteArgs ra, const SerialArgs sa)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    detail::route_block<EPL>(ra, 0);
    __syncthreads();
    dispatch_serial_block<false>(sa, dsm);
    __syncthreads();
    if (static_cast<int>(threadIdx.x) < sa.a.T) dispatch_finish_token(sa.a, threadIdx.x);
}

constexpr size_t kSmallSmemCap = 96 * 1024;   // >= 2*255*32*4 + kChunk*(kPrefLen + 8)

template <int EPL>
cudaError_t launch_small(const RouteArgs& ra, const SerialArgs& sa, size_t smem, cudaStream_t s)
{
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(route_dispatch_small_kernel<EPL>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmallSmemCap));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    route_dispatch_small_kernel<EPL><<<1, kSerialThreads, smem, s>>>(ra, sa);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s)
{
    if (a.T <= 0) return cudaSuccess;
    SerialArgs sa;
    sa.a = a;
    // worst case: every token has a tail entry
    const size_t scan_bytes = 2 * static_cast<size_t>(a.E) * kSerialWarps * 4;
    const size_t need = static_cast<size_t>(a.T) * (kPrefLen + a.k);
    sa.use_smem = (scan_bytes + need) <= kSerialSmemCap ? 1 : 0;
    // without room in shared memory the replay keeps the entries' experts in
    // the (otherwise unused) tail of the rank table
    sa.asg_global = reinterpret_cast<uint8_t*>(a.base) +
                    static_cast<size_t>(a.k) * a.nchunks * a.E * sizeof(int32_t);
    const size_t smem = scan_bytes + (sa.use_smem ? need : 0);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(dispatch_serial_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSerialSmemCap));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dispatch_serial_kernel<<<1, kSerialThreads, smem, s>>>(sa);
    cudaError_t e = cudaGetLastError();
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
    sa.use_smem = 1;
    sa.asg_global = nullptr;
    const size_t smem = 2 * static_cast<size_t>(a.E) * kSerialWarps * 4 +
                        static_cast<size_t>(a.T) * (kPrefLen + a.k);
    if (smem > kSmallSmemCap) return cudaErrorInvalidValue;
    if (a.E <= 32) return launch_small<1>(ra, sa, smem, s);
    if (a.E <= 64) return launch_small<2>(ra, sa, smem, s);
    if (a.E <= 128) return launch_small<4>(ra, sa, smem, s);
    return launch_small<8>(ra, sa, smem, s);
}

}  // namespace moe
