// probes.cu -- roof probes and device self-tests for sm_103a.
//
// The probes follow the matrix-multiplication lab's Part 1 ("the two roofs, again"): the
// FP32 roof is measured with a kernel of nothing but independent multiply-adds held in
// registers, the memory roof with a streaming read.  A third probe measures the dense
// f16 tensor-core roof with tcgen05.mma on shared-memory operands and no global traffic.
// They exist to measure roofline denominators; they compute nothing anyone needs.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace phx {
namespace {

using namespace ptx;

// Eight independent multiply-add chains per thread (scalar) or eight chains of f32x2 pairs
// (packed): 16 (or 32) floating-point operations per thread per iteration.
template <bool PACKED>
__global__ void __launch_bounds__(256) ffma_probe_kernel(float* out, int iters) {
    const float seed = 1e-6f * static_cast<float>(threadIdx.x);
    const float b = 0.99999f;
    const float c = 1e-5f;
    if constexpr (!PACKED) {
        float a0 = seed, a1 = seed + 0.1f, a2 = seed + 0.2f, a3 = seed + 0.3f;
        float a4 = seed + 0.4f, a5 = seed + 0.5f, a6 = seed + 0.6f, a7 = seed + 0.7f;
#pragma unroll 8
        for (int k = 0; k < iters; ++k) {
            a0 = fmaf(a0, b, c); a1 = fmaf(a1, b, c); a2 = fmaf(a2, b, c); a3 = fmaf(a3, b, c);
            a4 = fmaf(a4, b, c); a5 = fmaf(a5, b, c); a6 = fmaf(a6, b, c); a7 = fmaf(a7, b, c);
        }
        out[blockIdx.x * blockDim.x + threadIdx.x] = a0 + a1 + a2 + a3 + a4 + a5 + a6 + a7;
    } else {
        const float2 b2 = make_float2(b, b);
        const float2 c2 = make_float2(c, c);
        float2 a0 = make_float2(seed, seed + 0.05f), a1 = make_float2(seed + 0.1f, seed + 0.15f);
        float2 a2 = make_float2(seed + 0.2f, seed + 0.25f), a3 = make_float2(seed + 0.3f, seed + 0.35f);
        float2 a4 = make_float2(seed + 0.4f, seed + 0.45f), a5 = make_float2(seed + 0.5f, seed + 0.55f);
        float2 a6 = make_float2(seed + 0.6f, seed + 0.65f), a7 = make_float2(seed + 0.7f, seed + 0.75f);
#pragma unroll 8
        for (int k = 0; k < iters; ++k) {
            a0 = __ffma2_rn(a0, b2, c2); a1 = __ffma2_rn(a1, b2, c2);
            a2 = __ffma2_rn(a2, b2, c2); a3 = __ffma2_rn(a3, b2, c2);
            a4 = __ffma2_rn(a4, b2, c2); a5 = __ffma2_rn(a5, b2, c2);
            a6 = __ffma2_rn(a6, b2, c2); a7 = __ffma2_rn(a7, b2, c2);
        }
        out[blockIdx.x * blockDim.x + threadIdx.x] = a0.x + a0.y + a1.x + a1.y + a2.x + a2.y +
                                                     a3.x + a3.y + a4.x + a4.y + a5.x + a5.y +
                                                     a6.x + a6.y + a7.x + a7.y;
    }
}

// Grid-stride float4 read of n floats (n % 4 == 0, x 16-byte aligned).
__global__ void __launch_bounds__(256) stream_read_kernel(const float4* __restrict__ x, int64_t n4,
                                                          float* sink) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    float acc = 0.f;
#pragma unroll 4
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 v = __ldcs(x + i);
        acc += v.x + v.y + v.z + v.w;
    }
    if (acc == 1234.5f) sink[0] = acc;
}

// Tensor-core probe: one thread per CTA issues `iters` rounds of four M=128 x N x K=16
// kind::f16 MMAs on zeroed shared-memory operands into one TMEM accumulator.
template <int N>
__global__ void __launch_bounds__(128, 1) mma_probe_kernel(int iters, float* sink, unsigned int* status) {
    constexpr uint32_t kA = 128 * 64 * 2;
    constexpr uint32_t kB = N * 64 * 2;
    constexpr uint32_t kCols = N < 32 ? 32 : N;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    uint32_t* words = reinterpret_cast<uint32_t*>(base_ptr);
    for (uint32_t i = threadIdx.x; i < (kA + kB) / 4; i += blockDim.x) words[i] = 0u;
    const uint32_t bar = base + kA + kB;
    uint32_t* slot = reinterpret_cast<uint32_t*>(base_ptr + kA + kB + 8);
    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
    }
    // make the zeroed operands visible to the tensor core (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 0) tmem_alloc(smem_u32(slot), kCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    if (threadIdx.x == 0) {
        constexpr uint32_t idesc = idesc_f16_f32acc(128, N);
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_f16_ss(tmem, sw128_kmajor_desc(base + k * 32), sw128_kmajor_desc(base + kA + k * 32),
                           idesc, (it | k) != 0 ? 1u : 0u);
        }
        mma_commit(bar);
    }
    __syncwarp();
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, 0, nullptr, status));
    tc_fence_after();
    if (warp == 0) {
        uint32_t r[32];
        if (ok) {
            tmem_ld_32x32b_x32(tmem, r);
            tmem_ld_wait();
            if (threadIdx.x == 0) sink[blockIdx.x] = __uint_as_float(r[0]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kCols);
    }
}

// One thread waits on a barrier that nothing arrives at; the bounded wait gives up after
// limit_ns and records the timeout.
__global__ void wait_selftest_kernel(uint64_t limit_ns, unsigned int* status) {
    __shared__ __align__(8) uint64_t bar_storage;
    const uint32_t bar = smem_u32(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
        mbar_wait(bar, 0, nullptr, status, limit_ns);
    }
}

}  // namespace

cudaError_t probe_ffma_launch(int packed, int64_t blocks, int iters, float* out, cudaStream_t stream) {
    if (packed)
        ffma_probe_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(out, iters);
    else
        ffma_probe_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(out, iters);
    return cudaGetLastError();
}

cudaError_t probe_stream_read_launch(const float* x, int64_t n, float* sink, int64_t blocks,
                                     cudaStream_t stream) {
    stream_read_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        reinterpret_cast<const float4*>(x), n / 4, sink);
    return cudaGetLastError();
}

cudaError_t probe_mma_f16_launch(int64_t ctas, int iters, int n, float* sink, unsigned int* status,
                                 cudaStream_t stream) {
    auto run = [&](auto kernel, uint32_t bytes) {
        cudaError_t err = cudaFuncSetAttribute(reinterpret_cast<const void*>(kernel),
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(bytes));
        if (err != cudaSuccess) return err;
        kernel<<<static_cast<unsigned>(ctas), 128, bytes, stream>>>(iters, sink, status);
        return cudaGetLastError();
    };
    const uint32_t extra = 1024 + 64;
    switch (n) {
        case 64: return run(mma_probe_kernel<64>, 128 * 64 * 2 + 64 * 64 * 2 + extra);
        case 128: return run(mma_probe_kernel<128>, 128 * 64 * 2 + 128 * 64 * 2 + extra);
        case 256: return run(mma_probe_kernel<256>, 128 * 64 * 2 + 256 * 64 * 2 + extra);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t selftest_wait_launch(uint64_t limit_ns, unsigned int* status, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
    return cudaGetLastError();
}

}  // namespace phx
