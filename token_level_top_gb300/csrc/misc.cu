// misc.cu -- bandwidth kernels around the GEMMs: the gate/up weight
// re-layout, the row gather into slot order, the weighted combine of the
// expert outputs, and the bounded-wait failure probe.
#include "common.cuh"
#include "internal.h"
#include "quotient.cuh"

namespace moe {
namespace {

// w13[e][256 j + i] = i < 128 ? w1[e][128 j + i] : w3[e][128 j + i - 128]
// (rows of d bf16, copied 16 bytes per thread).
__global__ void pack_w13_kernel(int E, int F, int d, const uint4* __restrict__ w1,
                                const uint4* __restrict__ w3, uint4* __restrict__ w13)
{
    const size_t row16 = static_cast<size_t>(d) / 8;  // 16-byte words per row
    const size_t total = static_cast<size_t>(E) * 2 * F * row16;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t row = i / row16, col = i - row * row16;
        const size_t e = row / (2 * static_cast<size_t>(F));
        const int r = static_cast<int>(row - e * 2 * F);
        const int blk = r / 256, within = r - blk * 256;
        const bool up = within >= 128;
        const size_t src_row = e * F + static_cast<size_t>(blk) * 128 + (up ? within - 128 : within);
        w13[i] = (up ? w3 : w1)[src_row * row16 + col];
    }
}

// out[t] = sum over kept r (rank order, fp32) of cw[t,r] * y_slots[offsets[e]+slot], rounded
// to bf16 once.  One warp per (token, segment of 32*U 16-byte pieces of the
// row): lanes 0..k-1 fetch the token's rows and weights, then each lane
// streams U pieces per rank with all of them in flight.
template <int U>
__global__ void combine_kernel(int T, int d, int k, const uint4* __restrict__ y,
                               const int32_t* __restrict__ assign, const int32_t* __restrict__ slot,
                               const int32_t* __restrict__ offsets, const float* __restrict__ cw,
                               uint4* __restrict__ out)
{
    constexpr int kCombineUnroll = U;
    const int lane = threadIdx.x & 31;
    const int d8 = d / 8;
    const int nseg = (d8 + 32 * U - 1) / (32 * U);
    const long long wid = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (wid >= static_cast<long long>(T) * nseg) return;   // whole warps
    const int t = static_cast<int>(wid / nseg);
    const int seg = static_cast<int>(wid - static_cast<long long>(t) * nseg);
    int row = 0;
    float w = 0.0f;
    bool kept = false;
    if (lane < k) {
        const int e = assign[static_cast<size_t>(t) * k + lane];
        if (e >= 0) {
            row = offsets[e] + slot[static_cast<size_t>(t) * k + lane];
            w = cw[static_cast<size_t>(t) * k + lane];
            kept = true;
        }
    }
    const uint32_t kmask = __ballot_sync(0xffffffffu, kept);
    uint4* orow = out + static_cast<size_t>(t) * d8;
    {
        const int c0 = seg * 32 * U;
        float acc[kCombineUnroll][8];
#pragma unroll
        for (int u = 0; u < kCombineUnroll; ++u)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[u][j] = 0.0f;
        for (int r = 0; r < k; ++r) {
            if (!((kmask >> r) & 1u)) continue;   // uniform across the warp
            const uint4* yr = y + static_cast<size_t>(__shfl_sync(0xffffffffu, row, r)) * d8;
            const float wr = __shfl_sync(0xffffffffu, w, r);
            uint4 v[kCombineUnroll];
#pragma unroll
            for (int u = 0; u < kCombineUnroll; ++u) {
                const int c = c0 + u * 32 + lane;
                v[u] = c < d8 ? yr[c] : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kCombineUnroll; ++u) {
                const uint32_t words[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&words[j]);
                    acc[u][2 * j] += wr * __bfloat162float(b.x);
                    acc[u][2 * j + 1] += wr * __bfloat162float(b.y);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kCombineUnroll; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < d8)
                orow[c] = make_uint4(pack_bf16x2(acc[u][0], acc[u][1]), pack_bf16x2(acc[u][2], acc[u][3]),
                                     pack_bf16x2(acc[u][4], acc[u][5]), pack_bf16x2(acc[u][6], acc[u][7]));
        }
    }
}

__global__ void gather_rows_kernel(int rows_max, int d8, int k, int E, const uint4* __restrict__ h,
                                   const int32_t* __restrict__ perm,
                                   const int32_t* __restrict__ offsets, uint4* __restrict__ x)
{
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    const size_t i0 = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
    const int n = offsets[E];
    const size_t total = static_cast<size_t>(min(n, rows_max)) * d8;
    for (size_t i = i0; i < total; i += stride) {
        const size_t row = i / d8, c = i - row * d8;
        const int t = perm[row] / k;
        x[i] = h[static_cast<size_t>(t) * d8 + c];
    }
}

// Per-row FP8 (e4m3) quantisation:
//   s[r] = max_c |w[r,c]| / 448 (448: the largest finite e4m3; 1 for an all-zero row),
//   q[r,c] = e4m3(w[r,c] / s[r]), round to nearest even, saturated to +-448.
// Row r reads source row perm[r] / k when perm is given (the token rows of
// the kept slots), else row r; rows from *nrows on are skipped when nrows is
// given (a device-side count).

__device__ __forceinline__ float amax8(const uint4 v, float amax)
{
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&words[j]);
        amax = fmaxf(amax, fmaxf(fabsf(__bfloat162float(b.x)), fabsf(__bfloat162float(b.y))));
    }
    return amax;
}

// 1 / sc rounded, for div_by; 0 when sc is below kFmaDivMin (plain division).
__device__ __forceinline__ float recip_for_div(float sc) { return sc >= kFmaDivMin ? __frcp_rn(sc) : 0.0f; }

// Eight bf16 values to e4m3 codes of value / sc (y: recip_for_div(sc)).
__device__ __forceinline__ uint2 e4m3_8(const uint4 v, float sc, float y)
{
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
    uint32_t packed[2] = {0, 0};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&words[j]);
        const float v0 = __bfloat162float(b.x), v1 = __bfloat162float(b.y);
        const float x0 = y != 0.0f ? div_by(v0, sc, y) : __fdiv_rn(v0, sc);
        const float x1 = y != 0.0f ? div_by(v1, sc, y) : __fdiv_rn(v1, sc);
        uint16_t two;   // element x0 in the low byte
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(two) : "f"(x1), "f"(x0));
        packed[j >> 1] |= static_cast<uint32_t>(two) << (16 * (j & 1));
    }
    return make_uint2(packed[0], packed[1]);
}

// Each row's max |value| not yet known, longer rows: one warp per row, two
// passes over it (the second partly from L2).
__global__ void quantize_fp8_kernel(long long rows, int cols, const uint4* __restrict__ w,
                                    const int32_t* __restrict__ perm, int k,
                                    const int32_t* __restrict__ nrows, uint2* __restrict__ q,
                                    float* __restrict__ scales, float* __restrict__ zero_rows)
{
    const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= rows || (nrows && row >= *nrows)) return;   // whole warps
    const int lane = threadIdx.x & 31;
    const int c8 = cols / 8;
    const uint4* wr = w + (perm ? perm[row] / k : row) * c8;
    float amax = 0.0f;
#pragma unroll 4
    for (int c = lane; c < c8; c += 32) amax = amax8(__ldg(wr + c), amax);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
    if (lane == 0) {
        scales[row] = sc;
        if (zero_rows) zero_rows[row] = 0.0f;
    }
    uint2* qr = q + row * c8;
    const float y = recip_for_div(sc);
#pragma unroll 4
    for (int c = lane; c < c8; c += 32) qr[c] = e4m3_8(__ldg(wr + c), sc, y);
}

// Each row's max |value| not yet known, rows of at most 256 * 8 * P values:
// one 256-thread block per row, which holds the row in registers (P 16-byte
// pieces a thread), reduces its maximum and quantises it: one read.
template <int P>
__global__ void __launch_bounds__(256) quantize_fp8_block_kernel(
    int cols, const uint4* __restrict__ w, const int32_t* __restrict__ perm, int k,
    const int32_t* __restrict__ nrows, uint2* __restrict__ q, float* __restrict__ scales,
    float* __restrict__ zero_rows)
{
    __shared__ float s_wmax[8];
    const long long row = blockIdx.x;
    if (nrows && row >= *nrows) return;   // the whole block
    const int c8 = cols / 8;
    const uint4* wr = w + (perm ? perm[row] / k : row) * c8;
    uint4 v[P];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < P; ++i) {
        const int c = threadIdx.x + 256 * i;
        v[i] = c < c8 ? __ldg(wr + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < P; ++i) amax = amax8(v[i], amax);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((threadIdx.x & 31) == 0) s_wmax[threadIdx.x >> 5] = amax;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, s_wmax[i]);
    const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
    if (threadIdx.x == 0) {
        scales[row] = sc;
        if (zero_rows) zero_rows[row] = 0.0f;
    }
    uint2* qr = q + row * c8;
    const float y = recip_for_div(sc);
#pragma unroll
    for (int i = 0; i < P; ++i) {
        const int c = threadIdx.x + 256 * i;
        if (c < c8) qr[c] = e4m3_8(v[i], sc, y);
    }
}

// Each row's max |value| given: one pass, `parts` blocks per row (each a
// contiguous piece of it), so that a batch of few rows still spreads over the SMs.
__global__ void quantize_fp8_amax_kernel(int cols, int parts, const uint4* __restrict__ w,
                                         const int32_t* __restrict__ perm, int k,
                                         const int32_t* __restrict__ nrows,
                                         const float* __restrict__ amax_in, uint2* __restrict__ q,
                                         float* __restrict__ scales)
{
    const long long row = blockIdx.x / parts;
    const int part = static_cast<int>(blockIdx.x - row * parts);
    if (nrows && row >= *nrows) return;
    const float amax = amax_in[row];
    const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
    if (part == 0 && threadIdx.x == 0) scales[row] = sc;
    const int c8 = cols / 8;
    const int piece = (c8 + parts - 1) / parts;
    const int c_end = min(c8, (part + 1) * piece);
    const uint4* wr = w + (perm ? perm[row] / k : row) * c8;
    uint2* qr = q + row * c8;
    const float y = recip_for_div(sc);
#pragma unroll 4
    for (int c = part * piece + threadIdx.x; c < c_end; c += blockDim.x) qr[c] = e4m3_8(__ldg(wr + c), sc, y);
}

// One thread waits on an mbarrier that nothing will ever complete, with the
// library's bounded wait; when the budget runs out it records the timeout.
__global__ void timeout_probe_kernel(int* status, long long budget)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        mbar_fence_init();
        if (!mbar_wait(smem_u32(&bar), 0, budget)) record_error(status, MOE_ERR_TIMEOUT);
    }
}

int grid_for(size_t n, int threads)
{
    const size_t want = (n + threads - 1) / threads;
    const size_t cap = static_cast<size_t>(num_sms()) * 8;
    return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_pack_w13(int E, int F, int d, const void* w1, const void* w3, void* w13,
                            cudaStream_t s)
{
    const size_t total = static_cast<size_t>(E) * 2 * F * (d / 8);
    if (total == 0) return cudaSuccess;
    pack_w13_kernel<<<grid_for(total, 256), 256, 0, s>>>(E, F, d, static_cast<const uint4*>(w1),
                                                          static_cast<const uint4*>(w3),
                                                          static_cast<uint4*>(w13));
    return cudaGetLastError();
}

cudaError_t launch_gather_rows(int T, int d, int k, int E, const void* h, const int32_t* perm,
                               const int32_t* offsets, void* x_perm, cudaStream_t s)
{
    const int rows_max = T * k;
    const size_t total = static_cast<size_t>(rows_max) * (d / 8);
    if (total == 0) return cudaSuccess;
    gather_rows_kernel<<<grid_for(total, 256), 256, 0, s>>>(
        rows_max, d / 8, k, E, static_cast<const uint4*>(h), perm, offsets, static_cast<uint4*>(x_perm));
    return cudaGetLastError();
}

cudaError_t launch_combine(int T, int d, int k, const void* y_slots, const int32_t* assign,
                           const int32_t* slot, const int32_t* offsets, const float* cw, void* out,
                           cudaStream_t s)
{
    if (T <= 0 || d <= 0) return cudaSuccess;
    // longer pieces per warp for large batches, short ones (more warps) for
    // small; 2 pieces beat 4 by about 2 us at T = 4096-16384
    const int U = T >= 2048 ? 2 : 1;
    const long long warps = static_cast<long long>(T) * ((d / 8 + 32 * U - 1) / (32 * U));
    const int per_block = 8;
    const unsigned grid = static_cast<unsigned>((warps + per_block - 1) / per_block);
    if (U == 2)
        combine_kernel<2><<<grid, 32 * per_block, 0, s>>>(T, d, k, static_cast<const uint4*>(y_slots), assign,
                                                           slot, offsets, cw, static_cast<uint4*>(out));
    else
        combine_kernel<1><<<grid, 32 * per_block, 0, s>>>(T, d, k, static_cast<const uint4*>(y_slots), assign,
                                                           slot, offsets, cw, static_cast<uint4*>(out));
    return cudaGetLastError();
}

cudaError_t launch_quantize_fp8(long long rows, int cols, const void* w, const int32_t* perm, int k,
                                const int32_t* nrows, void* q, float* scales, cudaStream_t s,
                                const float* amax_in, float* zero_rows)
{
    if (rows <= 0) return cudaSuccess;
    if (amax_in) {
        if (zero_rows || rows > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
        // pieces of at least 256 vectors (one per thread), enough blocks for two per SM
        const long long c8 = cols / 8;
        long long parts = 1;
        while (parts < 8 && rows * parts < 2LL * num_sms() && c8 / (2 * parts) >= 256) parts *= 2;
        if (rows * parts > 0x7FFFFFFFLL) parts = 1;
        quantize_fp8_amax_kernel<<<static_cast<unsigned>(rows * parts), 256, 0, s>>>(
            cols, static_cast<int>(parts), static_cast<const uint4*>(w), perm, k, nrows, amax_in,
            static_cast<uint2*>(q), scales);
        return cudaGetLastError();
    }
    // a block per row while the rows fit one resident wave (a batch of a few
    // hundred tokens); beyond that, a warp per row schedules better
    const int c8 = cols / 8;
    if (c8 <= 256 * 4 && rows <= 8LL * num_sms()) {
        const unsigned grid = static_cast<unsigned>(rows);
        const uint4* w4 = static_cast<const uint4*>(w);
        uint2* q2 = static_cast<uint2*>(q);
        if (c8 <= 256)
            quantize_fp8_block_kernel<1><<<grid, 256, 0, s>>>(cols, w4, perm, k, nrows, q2, scales, zero_rows);
        else if (c8 <= 512)
            quantize_fp8_block_kernel<2><<<grid, 256, 0, s>>>(cols, w4, perm, k, nrows, q2, scales, zero_rows);
        else
            quantize_fp8_block_kernel<4><<<grid, 256, 0, s>>>(cols, w4, perm, k, nrows, q2, scales, zero_rows);
        return cudaGetLastError();
    }
    const int per_block = 8;
    quantize_fp8_kernel<<<static_cast<unsigned>((rows + per_block - 1) / per_block), 32 * per_block, 0, s>>>(
        rows, cols, static_cast<const uint4*>(w), perm, k, nrows, static_cast<uint2*>(q), scales, zero_rows);
    return cudaGetLastError();
}

cudaError_t launch_timeout_probe(int* status, long long budget, cudaStream_t s)
{
    timeout_probe_kernel<<<1, 32, 0, s>>>(status, budget);
    return cudaGetLastError();
}

}  // namespace moe
