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
// the per-chunk bases.  From chunk q1 on, one warp replays the entries 32 at a
// time: __match_any_sync gives each lane its rank among lanes choosing the
// same expert, a ballot finds the first lane that takes an expert's last
// slot, everything up to it commits, and lanes after it that chose the
// now-full expert choose again.  Stage 2 (grid-wide) writes the entries
// before q1, the permutation in slot order and the combine weights
// ([mhpn] §4.3: router probabilities renormalised over the experts used).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kSerialThreads = 1024;
constexpr size_t kSerialSmemCap = 200 * 1024;

struct SerialArgs {
    DispatchArgs a;
    int use_smem;
    uint8_t* asg_global;  // [T*k] fallback when the staging does not fit in smem
};

// First expert of the preference order that is neither full nor held.  The
// first kPrefLen entries come from the staged prefix; past it, the best
// remaining expert is found from the scores with the same order.
__device__ int choose_expert(const DispatchArgs& a, int t, int r, const uint8_t* pv,
                             const uint8_t* asg, const int* s_fill)
{
    const int E = a.E, k = a.k;
    const int L = E < kPrefLen ? E : kPrefLen;
    auto held = [&](int e) {
        for (int q = 0; q < r; ++q)
            if (asg[static_cast<size_t>(t) * k + q] == e) return true;
        return false;
    };
    for (int i = 0; i < L; ++i) {
        const int e = pv[i];
        if (s_fill[e] < a.C && !held(e)) return e;
    }
    if (L == E) return -1;
    float bv = -INFINITY;
    int bi = -1;
    const float* srow = a.scores + static_cast<size_t>(t) * E;
    for (int e = 0; e < E; ++e) {
        bool in_prefix = false;
        for (int i = 0; i < L; ++i) in_prefix |= (pv[i] == e);
        if (in_prefix || s_fill[e] >= a.C || held(e)) continue;
        float s = srow[e];
        if (isnan(s)) s = -INFINITY;
        if (bi < 0 || ranks_before(s, e, bv, bi)) {
            bv = s;
            bi = e;
        }
    }
    return bi;
}

__global__ void __launch_bounds__(kSerialThreads, 1) dispatch_serial_kernel(const SerialArgs sa)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ int s_fill[256];
    __shared__ int s_q1;
    const DispatchArgs& a = sa.a;
    const int E = a.E, T = a.T, k = a.k, nch = a.nchunks;
    const int Q = k * nch;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) s_q1 = Q;
    __syncthreads();
    // ---- stage 1: running count per expert over chunks (rank-major order)
    int total = 0;
    if (tid < E) {
        int cum = 0, qe = Q;
        for (int q = 0; q < Q; ++q) {
            const int c = a.hist[static_cast<size_t>(q) * E + tid];
            a.base[static_cast<size_t>(q) * E + tid] = cum;
            cum += c;
            if (qe == Q && cum > a.C) qe = q;
        }
        total = cum;
        atomicMin(&s_q1, qe);
    }
    __syncthreads();
    const int q1 = s_q1;
    if (tid < E) s_fill[tid] = (q1 < Q) ? a.base[static_cast<size_t>(q1) * E + tid] : total;

    // ---- stage the preference prefixes and the entries' experts
    const uint8_t* prefs = a.prefs;
    uint8_t* asg = sa.asg_global;
    if (sa.use_smem) {
        uint8_t* sp = dsm;
        const uint4* src = reinterpret_cast<const uint4*>(a.prefs);
        uint4* dst = reinterpret_cast<uint4*>(sp);
        const int n16 = (T * kPrefLen) / 16;
        for (int i = tid; i < n16; i += kSerialThreads) dst[i] = src[i];
        for (int i = n16 * 16 + tid; i < T * kPrefLen; i += kSerialThreads) sp[i] = a.prefs[i];
        prefs = sp;
        asg = sp + static_cast<size_t>(T) * kPrefLen;
    }
    for (int i = tid; i < T * k; i += kSerialThreads) {
        const int t = i / k, r = i - t * k;
        const int q = r * nch + t / kChunk;
        asg[i] = (q < q1) ? static_cast<uint8_t>(a.ids[i]) : static_cast<uint8_t>(255);
    }
    __syncthreads();
    if (warp != 0) return;

    // ---- stage 2: replay from chunk q1 with one warp
    int nre = 0, ndrop = 0;
    if (q1 < Q) {
        const int r1 = q1 / nch;
        const int t1 = (q1 - r1 * nch) * kChunk;
        for (int r = r1; r < k; ++r) {
            for (int t0 = (r == r1 ? t1 : 0); t0 < T; t0 += 32) {
                const int t = t0 + lane;
                const bool valid = t < T;
                uint8_t pv[kPrefLen];
                if (valid) {
                    const uint2 w = reinterpret_cast<const uint2*>(prefs)[t];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        pv[i] = static_cast<uint8_t>(w.x >> (8 * i));
                        pv[4 + i] = static_cast<uint8_t>(w.y >> (8 * i));
                    }
                }
                int e = valid ? choose_expert(a, t, r, pv, asg, s_fill) : -1;
                bool active = valid;
                while (true) {
                    const int key = active ? e : -2;
                    const uint32_t peers = __match_any_sync(0xffffffffu, key);
                    const int rnk = __popc(peers & lanemask_lt());
                    const bool takes = active && e >= 0;
                    const int before = takes ? s_fill[e] : 0;
                    const bool last = takes && (static_cast<long long>(before) + rnk + 1 == a.C);
                    const uint32_t ev = __ballot_sync(0xffffffffu, last);
                    const int cut = ev ? (__ffs(ev) - 1) : 31;
                    const bool commit = active && lane <= cut;
                    const uint32_t cmask = __ballot_sync(0xffffffffu, commit);
                    if (commit) {
                        const size_t idx = static_cast<size_t>(t) * k + r;
                        if (e >= 0) {
                            const int fl = (e != pv[r]) ? 1 : 0;
                            a.assign[idx] = e;
                            a.slot[idx] = before + rnk;
                            a.flags[idx] = static_cast<uint8_t>(fl);
                            asg[idx] = static_cast<uint8_t>(e);
                            nre += fl;
                        } else {
                            a.assign[idx] = -1;
                            a.slot[idx] = -1;
                            a.flags[idx] = 2;
                            asg[idx] = 255;
                            ++ndrop;
                        }
                    }
                    __syncwarp();
                    if (commit && e >= 0) {
                        const uint32_t cp = peers & cmask;
                        if (lane == __ffs(cp) - 1) s_fill[e] = before + __popc(cp);
                    }
                    __syncwarp();
                    if (!ev) break;
                    const int estar = __shfl_sync(0xffffffffu, e, cut);
                    active = active && lane > cut;
                    if (active && e == estar) e = choose_expert(a, t, r, pv, asg, s_fill);
                }
            }
        }
    }
    for (int off = 16; off >= 1; off >>= 1) {
        nre += __shfl_xor_sync(0xffffffffu, nre, off);
        ndrop += __shfl_xor_sync(0xffffffffu, ndrop, off);
    }
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

__global__ void dispatch_finish_kernel(const DispatchArgs a)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= a.T) return;
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
    const int top = a.prefs[static_cast<size_t>(t) * kPrefLen];
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

}  // namespace

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s)
{
    if (a.T <= 0) return cudaSuccess;
    SerialArgs sa;
    sa.a = a;
    const size_t need = static_cast<size_t>(a.T) * (kPrefLen + a.k);
    sa.use_smem = need <= kSerialSmemCap ? 1 : 0;
    // without room in shared memory the replay keeps the entries' experts in
    // the (otherwise unused) tail of the rank table
    sa.asg_global = reinterpret_cast<uint8_t*>(a.base) +
                    static_cast<size_t>(a.k) * a.nchunks * a.E * sizeof(int32_t);
    const size_t smem = sa.use_smem ? need : 0;
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

}  // namespace moe
