// router.cu -- the router's front end around the router GEMM.
//
//   router_norm_kernel   x_t = LayerNorm(h_t) or h_t / max(||h_t||_2, eps), bf16,
//                        the input of the router GEMM (the 2kiu page §5.2: a
//                        LayerNorm before the router, or L2-normalised input
//                        embeddings, keeps rows of unusually large norm from
//                        distorting the logits; "GPT-4稀疏激活真相…" §3.1 lists
//                        a router that starts with a LayerNorm)
//   router_head_kernel   z_t = silu(u_t) . W2^T + bias, u_t the router GEMM's
//                        output for W1 (summed over its K splits): the two-layer
//                        router of "MoE稀疏激活原理…" §3.1 step 2 (W1 d x 2E,
//                        W2 2E x E, W1 -> silu -> W2)
//
// Both are HBM- or latency-bound row passes: the norm reads and writes T x d
// bf16 once; the head reads the splits x T x H partial sums and writes T x E
// logits.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kNormThreads = 256;

// Sum over a 256-thread block; every thread gets the same value (the eight
// warp sums are added in warp order).
__device__ __forceinline__ float block_sum256(float v, float* s_red)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.0f;
#pragma unroll
    for (int i = 0; i < kNormThreads / 32; ++i) t += s_red[i];
    __syncthreads();   // s_red is reused by the next call
    return t;
}

// One block per token row; each thread holds P 16-byte pieces (8 values) of
// the row, and for the LayerNorm their 8 gamma and beta values (loaded as
// float4 with the row).  mode 1: LayerNorm, mean and mean squared deviation
// over d, then (h - mean) / sqrt(var + eps) * gamma + beta.  mode 2:
// h / max(||h||, eps).
template <int P>
__global__ void __launch_bounds__(kNormThreads) router_norm_kernel(int d, int mode, float eps,
                                                                   const uint4* __restrict__ h,
                                                                   const float4* __restrict__ gamma,
                                                                   const float4* __restrict__ beta,
                                                                   uint4* __restrict__ x)
{
    __shared__ float s_red[kNormThreads / 32];
    const long long t = blockIdx.x;
    const int d8 = d / 8;
    const uint4* hr = h + t * d8;
    float v[P][8];
    float4 ga[P][2], be[P][2];
#pragma unroll
    for (int i = 0; i < P; ++i) {
        const int c = threadIdx.x + kNormThreads * i;
        const bool in = c < d8;
        const uint4 q = in ? __ldg(hr + c) : make_uint4(0u, 0u, 0u, 0u);
        const float4 one = make_float4(1.0f, 1.0f, 1.0f, 1.0f), zero = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        ga[i][0] = (in && gamma) ? __ldg(gamma + 2 * c) : one;
        ga[i][1] = (in && gamma) ? __ldg(gamma + 2 * c + 1) : one;
        be[i][0] = (in && beta) ? __ldg(beta + 2 * c) : zero;
        be[i][1] = (in && beta) ? __ldg(beta + 2 * c + 1) : zero;
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[j]);
            v[i][2 * j] = __bfloat162float(b.x);
            v[i][2 * j + 1] = __bfloat162float(b.y);
        }
    }
    float mean = 0.0f;
    if (mode == 1) {
        float sum = 0.0f;
#pragma unroll
        for (int i = 0; i < P; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) sum += v[i][j];
        mean = block_sum256(sum, s_red) / static_cast<float>(d);
    }
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < P; ++i) {
        if (threadIdx.x + kNormThreads * i < d8) {
#pragma unroll
            for (int j = 0; j < 8; ++j) ss += (v[i][j] - mean) * (v[i][j] - mean);
        }
    }
    ss = block_sum256(ss, s_red);
    float scale;
    if (mode == 1) {
        scale = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
    } else {
        const float den = fmaxf(sqrtf(ss), eps);
        scale = den > 0.0f ? 1.0f / den : 0.0f;
    }
    uint4* xr = x + t * d8;
#pragma unroll
    for (int i = 0; i < P; ++i) {
        const int c = threadIdx.x + kNormThreads * i;
        if (c >= d8) continue;
        const float g[8] = {ga[i][0].x, ga[i][0].y, ga[i][0].z, ga[i][0].w,
                            ga[i][1].x, ga[i][1].y, ga[i][1].z, ga[i][1].w};
        const float b[8] = {be[i][0].x, be[i][0].y, be[i][0].z, be[i][0].w,
                            be[i][1].x, be[i][1].y, be[i][1].z, be[i][1].w};
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            y[j] = (v[i][j] - mean) * scale;
            if (mode == 1) y[j] = y[j] * g[j] + b[j];
        }
        xr[c] = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                           pack_bf16x2(y[6], y[7]));
    }
}

constexpr int kHeadThreads = 256;
constexpr int kHeadWarps = kHeadThreads / 32;
constexpr int kHeadTokens = 4;                          // tokens per warp
constexpr int kHeadBlockTokens = kHeadWarps * kHeadTokens;

// A block takes kHeadBlockTokens tokens at a time (grid-stride over token
// groups).  W2 [E, H] bf16 is staged once per block in shared memory as fp32,
// transposed (w2t[j][e], rows padded to E + 1), so that for a fixed j the
// lanes read consecutive experts.  The whole block first forms a[t][j] = silu(u_tj) for the group's
// tokens (u summed over the splits in split order); then each warp takes
// kHeadTokens of them and each lane experts e = lane + 32 q (q < EPL), and sums
// a[t][j] * W2[e][j] over j in order, so that each staged weight serves
// kHeadTokens tokens; plus the bias.
template <int EPL>
__global__ void __launch_bounds__(kHeadThreads) router_head_kernel(int T, int E, int H, int splits,
                                                                   const float* __restrict__ part,
                                                                   const __nv_bfloat16* __restrict__ w2,
                                                                   const float* __restrict__ bias,
                                                                   float* __restrict__ z)
{
    extern __shared__ float s_dyn[];
    const int Ep = E + 1;                 // padded row: conflict-free transposed writes
    float* w2t = s_dyn;                   // [H][Ep]
    float* s_a = s_dyn + H * Ep;          // [kHeadBlockTokens][H]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int e = warp; e < E; e += kHeadWarps)
        for (int j = lane; j < H; j += 32) w2t[j * Ep + e] = __bfloat162float(w2[static_cast<size_t>(e) * H + j]);
    const size_t pstride = static_cast<size_t>(T) * H;
    for (int t0 = blockIdx.x * kHeadBlockTokens; t0 < T; t0 += gridDim.x * kHeadBlockTokens) {
        __syncthreads();   // w2t staged; s_a free again
        const int n = min(kHeadBlockTokens, T - t0) * H;
        const float* pp = part + static_cast<size_t>(t0) * H;   // the group's rows are contiguous
#pragma unroll 4
        for (int i = threadIdx.x; i < kHeadBlockTokens * H; i += kHeadThreads) {
            float u = 0.0f;
            if (i < n)
                for (int sp = 0; sp < splits; ++sp) u += __ldg(pp + sp * pstride + i);
            s_a[i] = u / (1.0f + expf(-u));
        }
        __syncthreads();
        const float* a = s_a + warp * kHeadTokens * H;
        float acc[kHeadTokens][EPL];
#pragma unroll
        for (int tt = 0; tt < kHeadTokens; ++tt)
#pragma unroll
            for (int q = 0; q < EPL; ++q) acc[tt][q] = 0.0f;
        for (int j = 0; j < H; ++j) {
            float w[EPL];
#pragma unroll
            for (int q = 0; q < EPL; ++q) {
                const int e = lane + 32 * q;
                w[q] = e < E ? w2t[j * Ep + e] : 0.0f;
            }
#pragma unroll
            for (int tt = 0; tt < kHeadTokens; ++tt) {
                const float av = a[tt * H + j];
#pragma unroll
                for (int q = 0; q < EPL; ++q) acc[tt][q] = fmaf(av, w[q], acc[tt][q]);
            }
        }
        const int tw = t0 + warp * kHeadTokens;
#pragma unroll
        for (int tt = 0; tt < kHeadTokens; ++tt) {
            if (tw + tt >= T) break;
#pragma unroll
            for (int q = 0; q < EPL; ++q) {
                const int e = lane + 32 * q;
                if (e < E) z[static_cast<size_t>(tw + tt) * E + e] = acc[tt][q] + (bias ? bias[e] : 0.0f);
            }
        }
    }
}

// z[t][e] = sum of the K-split partials in split order, plus the bias: the
// linear router's logits, summed as the route step sums them.
__global__ void router_sum_kernel(int T, int E, int splits, const float* __restrict__ part,
                                  const float* __restrict__ bias, float* __restrict__ z)
{
    const size_t n = static_cast<size_t>(T) * E;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        float u = 0.0f;
        for (int sp = 0; sp < splits; ++sp) u += __ldg(part + sp * n + i);
        if (bias) u += bias[i % E];
        z[i] = u;
    }
}

}  // namespace

cudaError_t launch_router_sum(int T, int E, int splits, const float* part, const float* bias, float* z,
                              cudaStream_t s)
{
    if (T <= 0) return cudaSuccess;
    const size_t n = static_cast<size_t>(T) * E;
    const int grid = static_cast<int>(std::min<size_t>((n + 255) / 256, static_cast<size_t>(num_sms()) * 8));
    router_sum_kernel<<<grid, 256, 0, s>>>(T, E, splits, part, bias, z);
    return cudaGetLastError();
}

size_t router_head_smem(int E, int H)
{
    return static_cast<size_t>(H) * (E + 1) * 4 + static_cast<size_t>(kHeadBlockTokens) * H * 4;
}

cudaError_t launch_router_norm(int T, int d, int mode, float eps, const void* h, const float* gamma,
                               const float* beta, void* x, cudaStream_t s)
{
    if (T <= 0) return cudaSuccess;
    const int d8 = d / 8;
    const uint4* h4 = static_cast<const uint4*>(h);
    uint4* x4 = static_cast<uint4*>(x);
    const float4* g4 = reinterpret_cast<const float4*>(gamma);
    const float4* b4 = reinterpret_cast<const float4*>(beta);
    const unsigned grid = static_cast<unsigned>(T);
    if (d8 <= kNormThreads)
        router_norm_kernel<1><<<grid, kNormThreads, 0, s>>>(d, mode, eps, h4, g4, b4, x4);
    else if (d8 <= 2 * kNormThreads)
        router_norm_kernel<2><<<grid, kNormThreads, 0, s>>>(d, mode, eps, h4, g4, b4, x4);
    else if (d8 <= 4 * kNormThreads)
        router_norm_kernel<4><<<grid, kNormThreads, 0, s>>>(d, mode, eps, h4, g4, b4, x4);
    else if (d8 <= 8 * kNormThreads)
        router_norm_kernel<8><<<grid, kNormThreads, 0, s>>>(d, mode, eps, h4, g4, b4, x4);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

template <int EPL>
cudaError_t head_launch(int T, int E, int H, int splits, const float* part, const void* w2, const float* bias,
                        float* z, cudaStream_t s)
{
    const size_t most = static_cast<size_t>(kMaxRouterWeights2 + kMaxRouterHidden) * 4 +
                        static_cast<size_t>(kHeadBlockTokens) * kMaxRouterHidden * 4;
    const cudaError_t attr_err =
        ensure_smem_limit(reinterpret_cast<const void*>(router_head_kernel<EPL>), static_cast<int>(most));
    if (attr_err != cudaSuccess) return attr_err;
    const int groups = (T + kHeadBlockTokens - 1) / kHeadBlockTokens;
    const int grid = std::min(groups, 2 * num_sms());
    router_head_kernel<EPL><<<grid, kHeadThreads, router_head_smem(E, H), s>>>(
        T, E, H, splits, part, static_cast<const __nv_bfloat16*>(w2), bias, z);
    return cudaGetLastError();
}

cudaError_t launch_router_head(int T, int E, int H, int splits, const float* part, const void* w2,
                               const float* bias, float* z, cudaStream_t s)
{
    if (T <= 0) return cudaSuccess;
    if (E <= 32) return head_launch<1>(T, E, H, splits, part, w2, bias, z, s);
    if (E <= 64) return head_launch<2>(T, E, H, splits, part, w2, bias, z, s);
    if (E <= 128) return head_launch<4>(T, E, H, splits, part, w2, bias, z, s);
    return head_launch<8>(T, E, H, splits, part, w2, bias, z, s);
}

}  // namespace moe
