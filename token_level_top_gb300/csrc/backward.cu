// backward.cu -- the layer's backward pass (training; not on the forward path).
//
// For the dispatch the forward made (read from its workspace) and dL/dout:
//   combine      out[t] = sum_r cw[t,r] y[t,r]  ->  dy = cw dout, dcw = dout . y
//   down         y = W2 a                        ->  da = W2^T dy, dW2 += dy a^T
//   SwiGLU       a = silu(g) u                   ->  dg = da u silu'(g), du = da silu(g)
//   gate / up    g = W1 x, u = W3 x              ->  dx = W1^T dg + W3^T du, dW1 += dg x^T, dW3 += du x^T
//   weights      cw_r = p_{e_r} / sum_kept p     ->  dp, then the softmax, the temperature and the
//                                                    router GEMM (dz, dh += dz W_r, dW_r = dz^T h)
// ("GPT-4稀疏激活真相…" §3.1 and §4.3 for the expert and the weighted combine; "MoE架构揭秘…"
// §3.1 for the router's softmax and the load-balancing term written from the mean
// probabilities, which enters as dL/dP).
//
// Layout: each expert's kept rows are copied into a zero-padded block of C rows (C the
// capacity), so that every per-expert product is one strided-batched GEMM of E uniform
// problems with no host synchronisation.  g and u are the ones the forward's gate-up epilogue
// kept (fp32) when its workspace was sized for the backward.  Those plain GEMMs go to cuBLAS (bf16 inputs, fp32
// accumulation); the gathers, the SwiGLU and softmax derivatives and the reductions are the
// kernels below.
#include <cublas_v2.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// One warp per padded row idx = e*C + j.  j < count_e: the kept slot s = offsets[e] + j of
// entry t*k + r = perm[s] -- the token row and dL/dout row, its combine weight, and the
// entry's padded row in map; else zeros.
__global__ void bwd_pad_kernel(int E, long long C, int d8, int k, const int32_t* __restrict__ offsets,
                               const int32_t* __restrict__ perm, const float* __restrict__ cw,
                               const uint4* __restrict__ h, const uint4* __restrict__ dout,
                               uint4* __restrict__ xp, uint4* __restrict__ dop, float* __restrict__ rcw,
                               int32_t* __restrict__ rslot, int32_t* __restrict__ map)
{
    const long long idx = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (idx >= E * C) return;
    const int e = static_cast<int>(idx / C);
    const long long j = idx - e * C;
    const int off = offsets[e];
    const int cnt = offsets[e + 1] - off;
    uint4* xr = xp + idx * d8;
    uint4* dr = dop + idx * d8;
    if (j < cnt) {
        const int ent = perm[off + j];
        const long long t = ent / k;
        const uint4* hs = h + t * d8;
        const uint4* ds = dout + t * d8;
        for (int c = lane; c < d8; c += 32) {
            xr[c] = __ldg(hs + c);
            dr[c] = __ldg(ds + c);
        }
        if (lane == 0) {
            rcw[idx] = cw[ent];
            rslot[idx] = off + static_cast<int>(j);
            map[ent] = static_cast<int32_t>(idx);
        }
    } else {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        for (int c = lane; c < d8; c += 32) {
            xr[c] = z;
            dr[c] = z;
        }
        if (lane == 0) {
            rcw[idx] = 0.0f;
            rslot[idx] = -1;
        }
    }
}

__global__ void fill_i32_kernel(int32_t* p, long long n, int32_t v)
{
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        p[i] = v;
}

__global__ void bf16_to_f32_kernel(const __nv_bfloat16* __restrict__ a, float* __restrict__ b, long long n)
{
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        b[i] = __bfloat162float(a[i]);
}

__device__ __forceinline__ uint2 pack4_bf16(float a, float b, float c, float d)
{
    return make_uint2(pack_bf16x2(a, b), pack_bf16x2(c, d));
}

// One block per padded row.  gu [T*k, 2F] holds the forward's g and u of each kept slot (bf16,
// packed W13 column order: block q of 256 columns has g of F-columns [128q, 128q+128), then
// their u); rslot gives the padded row's slot (-1: padding, g = u = 0).  dap [rows, F] =
// W2^T dout (bf16, before the combine weight).  Writes acw = cw * a (bf16, for dW2), dgu =
// (dg, du) in the packed order (bf16, for dx and dW13), and the row's dcw = sum_f dap_f a_f
// = dout . y.
__global__ void __launch_bounds__(256) swiglu_bwd_kernel(int F, const float* __restrict__ gu,
                                                         const int32_t* __restrict__ rslot,
                                                         const float* __restrict__ dap,
                                                         const float* __restrict__ rcw,
                                                         __nv_bfloat16* __restrict__ acw,
                                                         __nv_bfloat16* __restrict__ dgu,
                                                         float* __restrict__ dcw_row)
{
    __shared__ float s_red[8];
    const long long row = blockIdx.x;
    const float c = rcw[row];
    const int slot = rslot[row];
    const float* gr = gu + static_cast<long long>(slot < 0 ? 0 : slot) * 2 * F;
    const float* dr = dap + row * F;
    __nv_bfloat16* ar = acw + row * F;
    __nv_bfloat16* dgr = dgu + row * 2 * F;
    float part = 0.0f;
    for (int f = 4 * threadIdx.x; f < F; f += 4 * blockDim.x) {
        const int q = f >> 7, o = f & 127;
        float4 g4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), u4 = g4;
        if (slot >= 0) {
            g4 = *reinterpret_cast<const float4*>(gr + 256 * q + o);
            u4 = *reinterpret_cast<const float4*>(gr + 256 * q + 128 + o);
        }
        const float4 d4 = *reinterpret_cast<const float4*>(dr + f);
        const float g[4] = {g4.x, g4.y, g4.z, g4.w}, u[4] = {u4.x, u4.y, u4.z, u4.w};
        const float da[4] = {d4.x, d4.y, d4.z, d4.w};
        float a[4], dg[4], du[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float sg = 1.0f / (1.0f + expf(-g[i]));
            const float si = g[i] * sg;
            a[i] = si * u[i];
            part = fmaf(da[i], a[i], part);
            const float dd = c * da[i];
            dg[i] = dd * u[i] * sg * (1.0f + g[i] * (1.0f - sg));
            du[i] = dd * si;
        }
        *reinterpret_cast<uint2*>(ar + f) = pack4_bf16(c * a[0], c * a[1], c * a[2], c * a[3]);
        *reinterpret_cast<uint2*>(dgr + 256 * q + o) = pack4_bf16(dg[0], dg[1], dg[2], dg[3]);
        *reinterpret_cast<uint2*>(dgr + 256 * q + 128 + o) = pack4_bf16(du[0], du[1], du[2], du[3]);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = part;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int i = 0; i < (blockDim.x >> 5); ++i) t += s_red[i];
        dcw_row[row] = t;
    }
}

// One warp per token: p = softmax(s) (the forward's penalised scores), the kept ranks from
// map, cw_r = p_{e_r} / S, dp_e = dP_e / T + (dcw_r - sum_r' dcw_r' cw_r') / S on the kept
// experts, ds = p (dp - p . dp), dz = ds / tau.
template <int EPL>
__global__ void router_bwd_kernel(int T, int E, int k, long long C, float tau, const float* __restrict__ scores,
                                  const int32_t* __restrict__ map, const float* __restrict__ dcw_row,
                                  const float* __restrict__ dP, float* __restrict__ dz)
{
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const float* st = scores + static_cast<size_t>(t) * E;
    float s[EPL], p[EPL];
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
        const int e = lane + 32 * q;
        s[q] = e < E ? st[e] : -INFINITY;
        m = fmaxf(m, s[q]);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float sum = 0.0f;
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
        const int e = lane + 32 * q;
        if (m == INFINITY) p[q] = (s[q] == INFINITY) ? 1.0f : 0.0f;   // the limits of the forward
        else if (m == -INFINITY) p[q] = e < E ? 1.0f : 0.0f;
        else p[q] = e < E ? expf(s[q] - m) : 0.0f;
        sum += p[q];
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
#pragma unroll
    for (int q = 0; q < EPL; ++q) p[q] /= sum;
    // the kept ranks: expert, its probability (from the lane that holds it), dcw
    auto prob_of = [&](int e) {
        float v = 0.0f;
#pragma unroll
        for (int q = 0; q < EPL; ++q)
            if (q == (e >> 5)) v = p[q];
        return __shfl_sync(0xffffffffu, v, e & 31);
    };
    float S = 0.0f, mdot = 0.0f;
    for (int r = 0; r < k; ++r) {
        const int idx = map[static_cast<size_t>(t) * k + r];   // the same in every lane
        if (idx < 0) continue;
        S += prob_of(static_cast<int>(idx / C));
    }
    for (int r = 0; r < k; ++r) {
        const int idx = map[static_cast<size_t>(t) * k + r];
        if (idx < 0) continue;
        mdot += dcw_row[idx] * (prob_of(static_cast<int>(idx / C)) / S);
    }
    float dp[EPL];
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
        const int e = lane + 32 * q;
        dp[q] = (dP && e < E) ? dP[e] / static_cast<float>(T) : 0.0f;
    }
    for (int r = 0; r < k; ++r) {
        const int idx = map[static_cast<size_t>(t) * k + r];
        if (idx < 0) continue;
        const int e = static_cast<int>(idx / C);
        if ((e & 31) == lane) {
#pragma unroll
            for (int q = 0; q < EPL; ++q)
                if (q == (e >> 5)) dp[q] += (dcw_row[idx] - mdot) / S;
        }
    }
    float pd = 0.0f;
#pragma unroll
    for (int q = 0; q < EPL; ++q) pd += p[q] * dp[q];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) pd += __shfl_xor_sync(0xffffffffu, pd, off);
    const float inv = (tau != 0.0f) ? tau : 1.0f;
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
        const int e = lane + 32 * q;
        if (e < E) dz[static_cast<size_t>(t) * E + e] = p[q] * (dp[q] - pd) / inv;
    }
}

// dh[t] = sum over t's kept ranks, in rank order, of dx of that entry's padded row (fp32).
__global__ void bwd_dh_kernel(int T, int d, int k, const int32_t* __restrict__ map,
                              const float4* __restrict__ dx, float4* __restrict__ dh)
{
    const int d4 = d / 4;
    const long long n = static_cast<long long>(T) * d4;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long t = i / d4;
        const int c = static_cast<int>(i - t * d4);
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int r = 0; r < k; ++r) {
            const int idx = map[t * k + r];
            if (idx < 0) continue;
            const float4 v = dx[static_cast<long long>(idx) * d4 + c];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        dh[i] = acc;
    }
}

// dbias[e] = sum_t dz[t, e]: one block per expert.
__global__ void col_sum_kernel(int T, int E, const float* __restrict__ dz, float* __restrict__ out)
{
    __shared__ float s_red[8];
    const int e = blockIdx.x;
    float v = 0.0f;
    for (int t = threadIdx.x; t < T; t += blockDim.x) v += dz[static_cast<size_t>(t) * E + e];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int i = 0; i < (blockDim.x >> 5); ++i) t += s_red[i];
        out[e] = t;
    }
}

cublasHandle_t blas_handle()
{
    static std::mutex mu;
    static cublasHandle_t handles[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!handles[dev] && cublasCreate(&handles[dev]) != CUBLAS_STATUS_SUCCESS) handles[dev] = nullptr;
    return handles[dev];
}

// Row-major C[b] (M x N, ldc) = op(A[b]) (M x K) . op(B[b]) (K x N) + beta C[b], for b < batch.
// ta: A is stored K x M (else M x K); tb: B is stored N x K (else K x N).  As column-major
// cuBLAS sees it, C^T = op(B)^T op(A)^T.
bool gemm_rm(cublasHandle_t hd, bool ta, bool tb, int M, int N, int K, const void* A, cudaDataType at,
             int lda, long long sA, const void* B, cudaDataType bt, int ldb, long long sB, void* C,
             cudaDataType ct, int ldc, long long sC, int batch, float beta)
{
    const float alpha = 1.0f;
    return cublasGemmStridedBatchedEx(hd, tb ? CUBLAS_OP_T : CUBLAS_OP_N, ta ? CUBLAS_OP_T : CUBLAS_OP_N, N, M, K,
                                      &alpha, B, bt, ldb, sB, A, at, lda, sA, &beta, C, ct, ldc, sC, batch,
                                      CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) == CUBLAS_STATUS_SUCCESS;
}

int grid_of(long long n, int threads)
{
    const long long want = (n + threads - 1) / threads;
    const long long cap = static_cast<long long>(num_sms()) * 16;
    return static_cast<int>(std::max<long long>(1, std::min(want, cap)));
}

}  // namespace

size_t backward_bytes(long long T, int d, int E, int k, int F, long long C)
{
    const size_t EC = static_cast<size_t>(E) * static_cast<size_t>(C);
    const size_t per_row = static_cast<size_t>(d) * 2 * 2 + static_cast<size_t>(F) * 4 +
                           static_cast<size_t>(F) * 2 + static_cast<size_t>(F) * 2 * 2 +
                           static_cast<size_t>(d) * 4 + 12;
    return EC * per_row + static_cast<size_t>(T) * k * 4 + static_cast<size_t>(T) * E * 4 +
           static_cast<size_t>(T) * d * 4 + static_cast<size_t>(E) * d * 4 + 16 * 256;
}

cudaError_t run_backward(const BackwardArgs& a, cudaStream_t s)
{
    const int E = a.E, k = a.k, d = a.d, F = a.F, T = a.T;
    const long long C = a.C, EC = static_cast<long long>(E) * C;
    cublasHandle_t hd = blas_handle();
    if (!hd) return cudaErrorInitializationError;
    if (cublasSetStream(hd, s) != CUBLAS_STATUS_SUCCESS) return cudaErrorInvalidValue;
    // carve the scratch (16-byte aligned regions)
    char* p = static_cast<char*>(a.scratch);
    auto take = [&](size_t bytes) {
        char* o = p;
        p += (bytes + 255) / 256 * 256;
        return o;
    };
    auto* xp = reinterpret_cast<__nv_bfloat16*>(take(EC * d * 2));
    auto* dop = reinterpret_cast<__nv_bfloat16*>(take(EC * d * 2));
    auto* dap = reinterpret_cast<float*>(take(EC * F * 4));
    auto* acw = reinterpret_cast<__nv_bfloat16*>(take(EC * F * 2));
    auto* dgu = reinterpret_cast<__nv_bfloat16*>(take(EC * 2 * F * 2));
    auto* dx = reinterpret_cast<float*>(take(EC * d * 4));
    auto* rcw = reinterpret_cast<float*>(take(EC * 4));
    auto* dcw = reinterpret_cast<float*>(take(EC * 4));
    auto* rslot = reinterpret_cast<int32_t*>(take(EC * 4));
    auto* map = reinterpret_cast<int32_t*>(take(static_cast<size_t>(T) * k * 4));
    auto* dz = reinterpret_cast<float*>(take(static_cast<size_t>(T) * E * 4));
    auto* h32 = reinterpret_cast<float*>(take(static_cast<size_t>(T) * d * 4));
    auto* wr32 = reinterpret_cast<float*>(take(static_cast<size_t>(E) * d * 4));

    fill_i32_kernel<<<grid_of(static_cast<long long>(T) * k, 256), 256, 0, s>>>(map, static_cast<long long>(T) * k,
                                                                                 -1);
    bwd_pad_kernel<<<static_cast<unsigned>((EC + 7) / 8), 256, 0, s>>>(
        E, C, d / 8, k, a.offsets, a.perm, a.cw, static_cast<const uint4*>(a.h), static_cast<const uint4*>(a.dout),
        reinterpret_cast<uint4*>(xp), reinterpret_cast<uint4*>(dop), rcw, rslot, map);
    if (cudaGetLastError() != cudaSuccess) return cudaErrorLaunchFailure;
    const cudaDataType BF = CUDA_R_16BF, F32 = CUDA_R_32F;
    const long long W13 = 2LL * F * d, W2s = static_cast<long long>(d) * F;
    // dap = dout rows . W2_e  ([C, d] . [d, F]); g and u come from the forward
    if (!gemm_rm(hd, false, false, static_cast<int>(C), F, d, dop, BF, d, C * d, a.w2, BF, F, W2s, dap, F32, F,
                 C * F, E, 0.0f))
        return cudaErrorUnknown;
    swiglu_bwd_kernel<<<static_cast<unsigned>(EC), 256, 0, s>>>(F, a.gu, rslot, dap, rcw, acw, dgu, dcw);
    if (cudaGetLastError() != cudaSuccess) return cudaErrorLaunchFailure;
    // dx = (dg, du) . W13_e  ([C, 2F] . [2F, d])
    if (!gemm_rm(hd, false, false, static_cast<int>(C), d, 2 * F, dgu, BF, 2 * F, C * 2 * F, a.w13, BF, d, W13, dx,
                 F32, d, C * d, E, 0.0f))
        return cudaErrorUnknown;
    // dW2_e = dout_e^T (cw a)_e  ([d, C] . [C, F]);  dW13_e = (dg, du)_e^T x_e  ([2F, C] . [C, d])
    if (!gemm_rm(hd, true, false, d, F, static_cast<int>(C), dop, BF, d, C * d, acw, BF, F, C * F, a.dw2, F32, F,
                 W2s, E, 0.0f))
        return cudaErrorUnknown;
    if (!gemm_rm(hd, true, false, 2 * F, d, static_cast<int>(C), dgu, BF, 2 * F, C * 2 * F, xp, BF, d, C * d, a.dw13,
                 F32, d, W13, E, 0.0f))
        return cudaErrorUnknown;
    // the router
    const int warps = 8;
    const unsigned rgrid = static_cast<unsigned>((T + warps - 1) / warps);
    if (E <= 32)
        router_bwd_kernel<1><<<rgrid, 32 * warps, 0, s>>>(T, E, k, C, a.tau, a.scores, map, dcw, a.dP, dz);
    else if (E <= 64)
        router_bwd_kernel<2><<<rgrid, 32 * warps, 0, s>>>(T, E, k, C, a.tau, a.scores, map, dcw, a.dP, dz);
    else if (E <= 128)
        router_bwd_kernel<4><<<rgrid, 32 * warps, 0, s>>>(T, E, k, C, a.tau, a.scores, map, dcw, a.dP, dz);
    else
        router_bwd_kernel<8><<<rgrid, 32 * warps, 0, s>>>(T, E, k, C, a.tau, a.scores, map, dcw, a.dP, dz);
    bwd_dh_kernel<<<grid_of(static_cast<long long>(T) * d / 4, 256), 256, 0, s>>>(
        T, d, k, map, reinterpret_cast<const float4*>(dx), reinterpret_cast<float4*>(a.dh));
    bf16_to_f32_kernel<<<grid_of(static_cast<long long>(E) * d, 256), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a.w_router), wr32, static_cast<long long>(E) * d);
    if (cudaGetLastError() != cudaSuccess) return cudaErrorLaunchFailure;
    // dh += dz . W_r  ([T, E] . [E, d])
    if (!gemm_rm(hd, false, false, T, d, E, dz, F32, E, 0, wr32, F32, d, 0, a.dh, F32, d, 0, 1, 1.0f))
        return cudaErrorUnknown;
    if (a.dw_router) {
        bf16_to_f32_kernel<<<grid_of(static_cast<long long>(T) * d, 256), 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(a.h), h32, static_cast<long long>(T) * d);
        // dW_r = dz^T h  ([E, T] . [T, d])
        if (!gemm_rm(hd, true, false, E, d, T, dz, F32, E, 0, h32, F32, d, 0, a.dw_router, F32, d, 0, 1, 0.0f))
            return cudaErrorUnknown;
    }
    if (a.dbias) col_sum_kernel<<<E, 256, 0, s>>>(T, E, dz, a.dbias);
    return cudaGetLastError();
}

}  // namespace moe
