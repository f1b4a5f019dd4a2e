// route.cu -- router epilogue: scores, preference order, softmax, top-k and
// the load statistics, one group of lanes per token.
//
//   z = sum of the router GEMM's K-split partial sums (+ bias), or given logits
//   s = z - lambda*usage (two rounded fp32 ops)      [mhpn] §2.3; [cnnetsun] §3.1
//   p = softmax(s); top-k = the k best s, ties to the lower index   [coreui] §3.1
//   f_i = picks of i / T, P_i = mean p_i             [cnnetsun] §4.2; [coreui] §3.1
//
// Each chunk of kChunk consecutive tokens is routed by a cluster of 1-4
// blocks (as many as keep the grid within the SMs).  A token is owned
// by G = min(32, pow2(E)) lanes, each lane holding EPL experts (e = lane + G*j);
// each lane ranks its experts against all E scores (shuffled through the
// group), which gives the whole preference order, stored as expert bytes per
// token: the first k ranks are the top-k picks, the rest serve the
// dispatch's reroutes.  Per chunk the kernel also writes
// the per-rank histogram of picks and each pick's stable rank among equal
// picks in token order (warp __match_any_sync + a scan over warps): the
// dispatch uses them to place every entry before the first capacity event in
// parallel.  All reductions run in a fixed order, so results are
// deterministic.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "route_block.cuh"

namespace moe {
namespace {

// Clusters of `cs` blocks, one cluster per chunk.
template <int EPL>
__global__ void __launch_bounds__(detail::kRouteThreads) route_kernel(const RouteArgs a, const int cs)
{
    detail::route_block<EPL>(a, blockIdx.x / cs, cs, static_cast<int>(cluster_ctarank()));
}

template <int EPL>
cudaError_t launch_route_cs(const RouteArgs& a, int cs, cudaStream_t s)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(a.nchunks * cs));
    cfg.blockDim = dim3(detail::kRouteThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, route_kernel<EPL>, a, cs);
}

__global__ void route_stats_kernel(const StatsArgs a)
{
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
        long long cnt = 0;
        const int Q = a.k * a.nchunks;
        for (int q = 0; q < Q; ++q) cnt += a.hist[static_cast<size_t>(q) * a.E + e];
        float psum = 0.0f;
        for (int c = 0; c < a.nchunks; ++c) psum += a.ppart[static_cast<size_t>(c) * a.E + e];
        if (a.counts_pre) a.counts_pre[e] = static_cast<int32_t>(cnt);
        if (a.f) a.f[e] = static_cast<float>(static_cast<double>(cnt) / a.T);
        if (a.P) a.P[e] = psum / static_cast<float>(a.T);
    }
}

}  // namespace

static_assert(detail::kRouteThreads >= kChunk && kChunk % 32 == 0, "one token per thread in the rank pass");

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s)
{
    if (a.T <= 0) return cudaSuccess;
    // one SM per block: split each chunk over as many blocks (a power of two,
    // at most 4) as keep the grid within the SMs.  Clusters of 8 were slower:
    // the route stage of 16 chunks took 36.9 us with 8 CTAs per chunk, 28.7
    // with 4 and 28.6 with 2; with 32 chunks 4 beat 2 (35.2 against 38.2 us).
    int cs = 1;
    while (cs < 4 && a.nchunks * cs * 2 <= num_sms()) cs *= 2;
    cudaError_t e;
    if (a.E <= 32)
        e = launch_route_cs<1>(a, cs, s);
    else if (a.E <= 64)
        e = launch_route_cs<2>(a, cs, s);
    else if (a.E <= 128)
        e = launch_route_cs<4>(a, cs, s);
    else
        e = launch_route_cs<8>(a, cs, s);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_route_stats(const StatsArgs& a, cudaStream_t s)
{
    if (a.T <= 0) return cudaSuccess;
    route_stats_kernel<<<1, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
