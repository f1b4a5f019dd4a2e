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
// Layout: each expert's kept rows are copied into a row block padded with zero rows to a
// multiple of 128 (the GEMM tile height), the blocks back to back in expert order.  The four
// per-expert products run on this library's tcgen05 GEMM (bwd_gemm.cu): the two input
// gradients as ragged grouped GEMMs over the blocks' row tiles, the two weight gradients with
// each expert's kept rows as the reduction dimension (64 rows per step; the zero rows fill the
// last step).  g and u are the ones the forward's gate-up epilogue kept (fp32) when its
// workspace was sized for the backward.  The gathers, the SwiGLU and softmax derivatives, the
// router's two small fp32 products and the reductions are the kernels below.  Nothing is
// padded beyond the tile; no library GEMM is called.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// One block: poff[e] = sum over e' < e of the kept rows of e' rounded up to 128 (the padded
// row blocks), poff[E] their total; map and emap (per entry t*k + r: its padded row and its
// expert) start as -1 (dropped entries keep it).
__global__ void bwd_prep_kernel(int E, long long n_ent, const int32_t* __restrict__ offsets,
                                int32_t* __restrict__ poff, int32_t* __restrict__ map, int32_t* __restrict__ emap)
{
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int carry = 0;
        for (int base = 0; base <= E; base += 32) {
            const int e = base + lane;
            const int rows = (e < E) ? (offsets[e + 1] - offsets[e] + kBM - 1) / kBM * kBM : 0;
            int incl = rows;
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            if (e <= E) poff[e] = carry + incl - rows;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    for (long long i = threadIdx.x; i < n_ent; i += blockDim.x) {
        map[i] = -1;
        emap[i] = -1;
    }
}

// The expert whose padded block holds row `row` (poff ascending, row < poff[E]).
__device__ __forceinline__ int block_of(const int32_t* __restrict__ poff, int E, int row)
{
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(poff + mid) <= row)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// One warp per padded row of the blocks.  Row j of expert e's block, j < count_e: the kept
// slot s = offsets[e] + j of entry t*k + r = perm[s] -- the token row and the dL/dout row, its
// combine weight, and the entry's row and expert in map / emap; j >= count_e: zeros.
__global__ void bwd_pad_kernel(int E, long long R, int d8, int k, const int32_t* __restrict__ offsets,
                               const int32_t* __restrict__ poff, const int32_t* __restrict__ perm,
                               const float* __restrict__ cw, const uint4* __restrict__ h,
                               const uint4* __restrict__ dout, uint4* __restrict__ xp, uint4* __restrict__ dop,
                               float* __restrict__ rcw, int32_t* __restrict__ rslot, int32_t* __restrict__ map,
                               int32_t* __restrict__ emap)
{
    const long long idx = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (idx >= R || idx >= __ldg(poff + E)) return;
    const int e = block_of(poff, E, static_cast<int>(idx));
    const long long j = idx - __ldg(poff + e);
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
            emap[ent] = e;
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

__device__ __forceinline__ uint2 pack4_bf16(float a, float b, float c, float d)
{
    return make_uint2(pack_bf16x2(a, b), pack_bf16x2(c, d));
}

// One block per padded row (rows past the blocks' total exit).  gu [T*k, 2F] holds the
// forward's g and u of each kept slot (fp32, packed W13 column order: block q of 256 columns
// has g of F-columns [128q, 128q+128), then their u); rslot gives the padded row's slot (-1:
// padding, g = u = 0).  dap [rows, F] = W2^T dout (fp32, before the combine weight).  Writes acw = cw * a (bf16, for dW2), dgu =
// (dg, du) in the packed order (bf16, for dx and dW13), and the row's dcw = sum_f dap_f a_f
// = dout . y.
__global__ void __launch_bounds__(256) swiglu_bwd_kernel(int F, int E, const int32_t* __restrict__ poff,
                                                         const float* __restrict__ gu,
                                                         const int32_t* __restrict__ rslot,
                                                         const float* __restrict__ dap,
                                                         const float* __restrict__ rcw,
                                                         __nv_bfloat16* __restrict__ acw,
                                                         __nv_bfloat16* __restrict__ dgu,
                                                         float* __restrict__ dcw_row)
{
    __shared__ float s_red[8];
    const long long row = blockIdx.x;
    if (row >= __ldg(poff + E)) return;
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
// map (padded row) and emap (expert), cw_r = p_{e_r} / S, dp_e = dP_e / T + (dcw_r - sum_r' dcw_r' cw_r') / S on the kept
// experts, ds = p (dp - p . dp), dz = ds / tau.
template <int EPL>
__global__ void router_bwd_kernel(int T, int E, int k, float tau, const float* __restrict__ scores,
                                  const int32_t* __restrict__ map, const int32_t* __restrict__ emap,
                                  const float* __restrict__ dcw_row, const float* __restrict__ dP,
                                  float* __restrict__ dz)
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
        S += prob_of(emap[static_cast<size_t>(t) * k + r]);
    }
    for (int r = 0; r < k; ++r) {
        const int idx = map[static_cast<size_t>(t) * k + r];
        if (idx < 0) continue;
        mdot += dcw_row[idx] * (prob_of(emap[static_cast<size_t>(t) * k + r]) / S);
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
        const int e = emap[static_cast<size_t>(t) * k + r];
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

// dh[t] = (sum over t's kept ranks, in rank order, of dx of that entry's padded row)
//         + sum_e dz[t, e] W_r[e] (expert order), fp32.  A block: kDhTokens tokens x 1024
// columns, each thread 4 columns of every token; dz of the block's tokens staged in shared
// memory, each W_r element read once per block.
constexpr int kDhTokens = 8;
__global__ void __launch_bounds__(256) bwd_dh_kernel(int T, int d, int E, int k, const int32_t* __restrict__ map,
                                                     const float4* __restrict__ dx, const float* __restrict__ dz,
                                                     const __nv_bfloat16* __restrict__ wr, float4* __restrict__ dh)
{
    extern __shared__ float s_dz[];   // [kDhTokens][E]
    const int t0 = blockIdx.x * kDhTokens;
    const int nt = min(kDhTokens, T - t0);
    for (int i = threadIdx.x; i < kDhTokens * E; i += blockDim.x) {
        const int tt = i / E;
        s_dz[i] = tt < nt ? dz[static_cast<size_t>(t0 + tt) * E + (i - tt * E)] : 0.0f;
    }
    __syncthreads();
    const int c4 = blockIdx.y * blockDim.x + threadIdx.x;   // float4 column
    if (4 * c4 >= d) return;
    float4 acc[kDhTokens];
#pragma unroll
    for (int tt = 0; tt < kDhTokens; ++tt) acc[tt] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int e = 0; e < E; ++e) {
        const uint2 w2 = __ldg(reinterpret_cast<const uint2*>(wr + static_cast<size_t>(e) * d) + c4);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w2.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w2.y));
#pragma unroll
        for (int tt = 0; tt < kDhTokens; ++tt) {
            const float z = s_dz[tt * E + e];
            acc[tt].x = fmaf(z, a.x, acc[tt].x);
            acc[tt].y = fmaf(z, a.y, acc[tt].y);
            acc[tt].z = fmaf(z, b.x, acc[tt].z);
            acc[tt].w = fmaf(z, b.y, acc[tt].w);
        }
    }
    const int d4 = d / 4;
    for (int tt = 0; tt < nt; ++tt) {
        const long long t = t0 + tt;
        float4 r = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int q = 0; q < k; ++q) {
            const int idx = map[t * k + q];
            if (idx < 0) continue;
            const float4 v = dx[static_cast<long long>(idx) * d4 + c4];
            r.x += v.x;
            r.y += v.y;
            r.z += v.z;
            r.w += v.w;
        }
        r.x += acc[tt].x;
        r.y += acc[tt].y;
        r.z += acc[tt].z;
        r.w += acc[tt].w;
        dh[t * d4 + c4] = r;
    }
}

// dW_r = dz^T h in two passes.  Pass 1: block (column block of 256, expert group of kWrE,
// token slice) -> part[slice][e][col] = sum over the slice's tokens, in token order, of
// dz[t, e] h[t, col].  Pass 2 sums the slices in order.
constexpr int kWrE = 16;
constexpr int kWrChunk = 64;
__global__ void __launch_bounds__(128) bwd_wr_part_kernel(int T, int d, int E, int slice,
                                                          const float* __restrict__ dz,
                                                          const __nv_bfloat16* __restrict__ h,
                                                          float* __restrict__ part)
{
    __shared__ float s_z[kWrChunk][kWrE];
    const int col = (blockIdx.x * blockDim.x + threadIdx.x) * 2;
    const int e0 = blockIdx.y * kWrE;
    const int ne = min(kWrE, E - e0);
    const int ta = blockIdx.z * slice, tb = min(T, ta + slice);
    float acc[kWrE][2];
#pragma unroll
    for (int q = 0; q < kWrE; ++q) acc[q][0] = acc[q][1] = 0.0f;
    for (int c0 = ta; c0 < tb; c0 += kWrChunk) {
        const int n = min(kWrChunk, tb - c0);
        __syncthreads();
        for (int i = threadIdx.x; i < kWrChunk * kWrE; i += blockDim.x) {
            const int tt = i / kWrE, q = i - tt * kWrE;
            s_z[tt][q] = (tt < n && q < ne) ? dz[static_cast<size_t>(c0 + tt) * E + e0 + q] : 0.0f;
        }
        __syncthreads();
        if (col < d) {
            for (int tt = 0; tt < n; ++tt) {
                const float2 hv =
                    __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(h + static_cast<size_t>(c0 + tt) * d + col));
#pragma unroll
                for (int q = 0; q < kWrE; ++q) {
                    acc[q][0] = fmaf(s_z[tt][q], hv.x, acc[q][0]);
                    acc[q][1] = fmaf(s_z[tt][q], hv.y, acc[q][1]);
                }
            }
        }
    }
    if (col >= d) return;
    for (int q = 0; q < ne; ++q)
        *reinterpret_cast<float2*>(part + (static_cast<size_t>(blockIdx.z) * E + e0 + q) * d + col) =
            make_float2(acc[q][0], acc[q][1]);
}

__global__ void bwd_wr_sum_kernel(long long n, int slices, const float* __restrict__ part, float* __restrict__ out)
{
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        float v = 0.0f;
        for (int z = 0; z < slices; ++z) v += part[static_cast<size_t>(z) * n + i];
        out[i] = v;
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

int grid_of(long long n, int threads)
{
    const long long want = (n + threads - 1) / threads;
    const long long cap = static_cast<long long>(num_sms()) * 16;
    return static_cast<int>(std::max<long long>(1, std::min(want, cap)));
}

}  // namespace

int wr_slices(long long T) { return static_cast<int>(std::max<long long>(1, std::min<long long>(32, (T + 127) / 128))); }

long long backward_block_rows(long long T, int E, int k, long long C)
{
    const long long per = (std::min(C, T) + kBM - 1) / kBM * kBM;
    return std::max<long long>(kBM, std::min(static_cast<long long>(E) * per, T * k + static_cast<long long>(kBM - 1) * E));
}

size_t backward_bytes(long long T, int d, int E, int k, int F, long long R)
{
    const size_t per_row = static_cast<size_t>(d) * 2 * 2 + static_cast<size_t>(F) * 4 +
                           static_cast<size_t>(F) * 2 + static_cast<size_t>(F) * 2 * 2 +
                           static_cast<size_t>(d) * 4 + 12;
    return static_cast<size_t>(R) * per_row + static_cast<size_t>(T) * k * 8 + static_cast<size_t>(T) * E * 4 +
           static_cast<size_t>(wr_slices(T)) * E * d * 4 + static_cast<size_t>(E + 1) * 4 + 16 * 256;
}

cudaError_t run_backward(const BackwardArgs& a, cudaStream_t s)
{
    const int E = a.E, k = a.k, d = a.d, F = a.F, T = a.T;
    const long long R = a.R;
    // carve the scratch (256-byte aligned regions)
    char* p = static_cast<char*>(a.scratch);
    auto take = [&](size_t bytes) {
        char* o = p;
        p += (bytes + 255) / 256 * 256;
        return o;
    };
    auto* poff = reinterpret_cast<int32_t*>(take(static_cast<size_t>(E + 1) * 4));
    auto* xp = reinterpret_cast<__nv_bfloat16*>(take(R * d * 2));
    auto* dop = reinterpret_cast<__nv_bfloat16*>(take(R * d * 2));
    auto* dap = reinterpret_cast<float*>(take(R * F * 4));
    auto* acw = reinterpret_cast<__nv_bfloat16*>(take(R * F * 2));
    auto* dgu = reinterpret_cast<__nv_bfloat16*>(take(R * 2 * F * 2));
    auto* dx = reinterpret_cast<float*>(take(R * d * 4));
    auto* rcw = reinterpret_cast<float*>(take(R * 4));
    auto* dcw = reinterpret_cast<float*>(take(R * 4));
    auto* rslot = reinterpret_cast<int32_t*>(take(R * 4));
    auto* map = reinterpret_cast<int32_t*>(take(static_cast<size_t>(T) * k * 4));
    auto* emap = reinterpret_cast<int32_t*>(take(static_cast<size_t>(T) * k * 4));
    auto* dz = reinterpret_cast<float*>(take(static_cast<size_t>(T) * E * 4));
    const int slices = wr_slices(T);
    auto* wr_part = reinterpret_cast<float*>(take(static_cast<size_t>(slices) * E * d * 4));

    bwd_prep_kernel<<<1, 1024, 0, s>>>(E, static_cast<long long>(T) * k, a.offsets, poff, map, emap);
    bwd_pad_kernel<<<static_cast<unsigned>((R + 7) / 8), 256, 0, s>>>(
        E, R, d / 8, k, a.offsets, poff, a.perm, a.cw, static_cast<const uint4*>(a.h),
        static_cast<const uint4*>(a.dout), reinterpret_cast<uint4*>(xp), reinterpret_cast<uint4*>(dop), rcw, rslot,
        map, emap);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;

    BwdGemmLaunch g{};
    g.E = E;
    g.rows = R;
    g.kept = static_cast<long long>(T) * k;
    g.offsets = a.offsets;
    g.status = a.status;
    g.budget = a.budget;
    // dL/da before the combine weight: dap = dL/dout rows . W2_e  ([rows, d] . [d, F])
    g.mode = BG_DGRAD;
    g.K = d;
    g.N = F;
    g.a = dop;
    g.b = a.w2;
    g.out = dap;
    if ((err = launch_bwd_gemm(g, s)) != cudaSuccess) return err;
    swiglu_bwd_kernel<<<static_cast<unsigned>(R), 256, 0, s>>>(F, E, poff, a.gu, rslot, dap, rcw, acw, dgu, dcw);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    // dx = (dg, du) . W13_e  ([rows, 2F] . [2F, d])
    g.K = 2 * F;
    g.N = d;
    g.a = dgu;
    g.b = a.w13;
    g.out = dx;
    if ((err = launch_bwd_gemm(g, s)) != cudaSuccess) return err;
    // dW2_e = dL/dout_e^T (cw a)_e  ([d, rows] . [rows, F]);  dW13_e = (dg, du)_e^T x_e  ([2F, rows] . [rows, d])
    g.mode = BG_WGRAD;
    g.K = 0;
    g.Mw = d;
    g.N = F;
    g.a = dop;
    g.b = acw;
    g.out = a.dw2;
    if ((err = launch_bwd_gemm(g, s)) != cudaSuccess) return err;
    g.Mw = 2 * F;
    g.N = d;
    g.a = dgu;
    g.b = xp;
    g.out = a.dw13;
    if ((err = launch_bwd_gemm(g, s)) != cudaSuccess) return err;
    // the router
    const int warps = 8;
    const unsigned rgrid = static_cast<unsigned>((T + warps - 1) / warps);
    if (E <= 32)
        router_bwd_kernel<1><<<rgrid, 32 * warps, 0, s>>>(T, E, k, a.tau, a.scores, map, emap, dcw, a.dP, dz);
    else if (E <= 64)
        router_bwd_kernel<2><<<rgrid, 32 * warps, 0, s>>>(T, E, k, a.tau, a.scores, map, emap, dcw, a.dP, dz);
    else if (E <= 128)
        router_bwd_kernel<4><<<rgrid, 32 * warps, 0, s>>>(T, E, k, a.tau, a.scores, map, emap, dcw, a.dP, dz);
    else
        router_bwd_kernel<8><<<rgrid, 32 * warps, 0, s>>>(T, E, k, a.tau, a.scores, map, emap, dcw, a.dP, dz);
    // dh = the experts' dx rows + dz . W_r
    const dim3 dgrid(static_cast<unsigned>((T + kDhTokens - 1) / kDhTokens), static_cast<unsigned>((d / 4 + 255) / 256));
    bwd_dh_kernel<<<dgrid, 256, static_cast<size_t>(kDhTokens) * E * 4, s>>>(
        T, d, E, k, map, reinterpret_cast<const float4*>(dx), dz, static_cast<const __nv_bfloat16*>(a.w_router),
        reinterpret_cast<float4*>(a.dh));
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (a.dw_router) {   // dW_r = dz^T h  ([E, T] . [T, d])
        const int slice = (T + slices - 1) / slices;
        const dim3 wgrid(static_cast<unsigned>((d / 2 + 127) / 128), static_cast<unsigned>((E + kWrE - 1) / kWrE),
                         static_cast<unsigned>(slices));
        bwd_wr_part_kernel<<<wgrid, 128, 0, s>>>(T, d, E, slice, dz, static_cast<const __nv_bfloat16*>(a.h), wr_part);
        const long long n = static_cast<long long>(E) * d;
        bwd_wr_sum_kernel<<<grid_of(n, 256), 256, 0, s>>>(n, slices, wr_part, a.dw_router);
    }
    if (a.dbias) col_sum_kernel<<<E, 256, 0, s>>>(T, E, dz, a.dbias);
    return cudaGetLastError();
}

}  // namespace moe
