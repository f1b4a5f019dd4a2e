// misc.cu -- bandwidth kernels around the GEMMs: the gate/up weight
// re-layout, the fp32 -> bf16 finalize of the fused combine, the slot-order
// combine used by moe_combine, and the bounded-wait failure probe.
#include "common.cuh"
#include "internal.h"

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

// out = bf16(acc), 4 values per thread.  Rows whose choices were all dropped
// received no contribution and stay 0.
__global__ void finalize_kernel(size_t n4, const float4* __restrict__ acc, uint2* __restrict__ out)
{
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const float4 v = acc[i];
        out[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    }
}

// out[t] = sum over kept r (rank order) of cw[t,r] * y_slots[offsets[e]+slot], 8 columns per thread.
__global__ void combine_kernel(int T, int d, int k, const uint4* __restrict__ y,
                               const int32_t* __restrict__ assign, const int32_t* __restrict__ slot,
                               const int32_t* __restrict__ offsets, const float* __restrict__ cw,
                               uint4* __restrict__ out)
{
    const int d8 = d / 8;
    const size_t total = static_cast<size_t>(T) * d8;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(i / d8);
        const int c8 = static_cast<int>(i - static_cast<size_t>(t) * d8);
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int r = 0; r < k; ++r) {
            const int e = assign[static_cast<size_t>(t) * k + r];
            if (e < 0) continue;
            const float w = cw[static_cast<size_t>(t) * k + r];
            const size_t srow = static_cast<size_t>(offsets[e]) + slot[static_cast<size_t>(t) * k + r];
            const uint4 v = y[srow * d8 + c8];
            const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&words[j]);
                acc[2 * j] += w * __bfloat162float(b.x);
                acc[2 * j + 1] += w * __bfloat162float(b.y);
            }
        }
        out[i] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                            pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
}

// x_perm[i] = h[perm[i] / k] for the kept slots i < offsets[E]: the token rows
// in slot order, so that the gate-up GEMM reads its A tiles with plain TMA
// tile loads.  16 bytes per thread, rows of d bf16.
__global__ void gather_rows_kernel(int rows_max, int d8, int k, int E, const uint4* __restrict__ h,
                                   const int32_t* __restrict__ perm,
                                   const int32_t* __restrict__ offsets, uint4* __restrict__ x,
                                   float4* __restrict__ zero, size_t zero4)
{
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    const size_t i0 = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
    // the fp32 output accumulator the down projection scatters into starts at zero
    for (size_t i = i0; i < zero4; i += stride) zero[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int n = offsets[E];
    const size_t total = static_cast<size_t>(min(n, rows_max)) * d8;
    for (size_t i = i0; i < total; i += stride) {
        const size_t row = i / d8, c = i - row * d8;
        const int t = perm[row] / k;
        x[i] = h[static_cast<size_t>(t) * d8 + c];
    }
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

cudaError_t launch_finalize(int T, int d, const float* acc, void* out, cudaStream_t s)
{
    const size_t n4 = static_cast<size_t>(T) * d / 4;
    if (n4 == 0) return cudaSuccess;
    finalize_kernel<<<grid_for(n4, 256), 256, 0, s>>>(n4, reinterpret_cast<const float4*>(acc),
                                                       static_cast<uint2*>(out));
    return cudaGetLastError();
}

cudaError_t launch_gather_rows(int T, int d, int k, int E, const void* h, const int32_t* perm,
                               const int32_t* offsets, void* x_perm, float* acc_zero,
                               cudaStream_t s)
{
    const int rows_max = T * k;
    const size_t total = static_cast<size_t>(rows_max) * (d / 8);
    const size_t zero4 = acc_zero ? static_cast<size_t>(T) * d / 4 : 0;
    if (total == 0) return cudaSuccess;
    gather_rows_kernel<<<grid_for(total, 256), 256, 0, s>>>(
        rows_max, d / 8, k, E, static_cast<const uint4*>(h), perm, offsets,
        static_cast<uint4*>(x_perm), reinterpret_cast<float4*>(acc_zero), zero4);
    return cudaGetLastError();
}

cudaError_t launch_combine(int T, int d, int k, const void* y_slots, const int32_t* assign,
                           const int32_t* slot, const int32_t* offsets, const float* cw, void* out,
                           cudaStream_t s)
{
    const size_t total = static_cast<size_t>(T) * (d / 8);
    if (total == 0) return cudaSuccess;
    combine_kernel<<<grid_for(total, 256), 256, 0, s>>>(T, d, k, static_cast<const uint4*>(y_slots),
                                                         assign, slot, offsets, cw,
                                                         static_cast<uint4*>(out));
    return cudaGetLastError();
}

cudaError_t launch_timeout_probe(int* status, long long budget, cudaStream_t s)
{
    timeout_probe_kernel<<<1, 32, 0, s>>>(status, budget);
    return cudaGetLastError();
}

}  // namespace moe
