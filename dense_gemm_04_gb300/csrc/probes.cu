// probes.cu -- roof probes and device self-tests for sm_103a.
//
// The matrix-multiplication lab's Part 1 ("the two roofs, again") measures the FP32 roof
// with a kernel of nothing but register-resident multiply-adds and the memory roof with a
// kernel that only reads.  The two probes here measure the same two quantities on sm_103a
// with kernels designed for it; a third measures the dense f16 tensor-core roof with
// tcgen05.mma on shared-memory operands and no global traffic.  They exist to measure
// roofline denominators; they compute nothing anyone needs.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace phx {
namespace {

using namespace ptx;

// FP32 issue-rate probe.  Each SM of sm_103a has 4 sub-partitions of 32 FP32 lanes; a
// dependent multiply-add waits a few cycles for its predecessor, so each thread keeps
// kProbeLanes independent recurrences x <- x * rho + tau in registers, and the grid puts
// many warps on every SM.  rho and tau arrive as arguments, so the compiler can neither
// fold nor shorten the recurrences; with rho = 1 - 2^-12 and tau = 2^-13 every value stays
// in [0.5, 1) (the fixed point is 0.5).  PACKED runs the same recurrences two lanes per
// f32x2 instruction.  Both forms do 2 * kProbeLanes FLOPs per thread and iteration.  The
// lanes are folded by a pairwise tree and each thread stores its fold, so no recurrence is
// dead code.
constexpr int kProbeLanes = 12;

__device__ __forceinline__ float probe_seed(uint32_t g, int i) {
    uint32_t h = g * 0x85EBCA6Bu + static_cast<uint32_t>(i) * 0xC2B2AE35u;
    h ^= h >> 16;
    return __uint_as_float(0x3F000000u | (h & 0x007FFFFFu));  // [0.5, 1)
}

template <bool PACKED>
__global__ void __launch_bounds__(256) fp32_issue_probe_kernel(float* out, int iters, float rho, float tau) {
    const uint32_t g = blockIdx.x * blockDim.x + threadIdx.x;
    float v[kProbeLanes];
#pragma unroll
    for (int i = 0; i < kProbeLanes; ++i) v[i] = probe_seed(g, i);
    if constexpr (PACKED) {
        float2 w[kProbeLanes / 2];
#pragma unroll
        for (int i = 0; i < kProbeLanes / 2; ++i) w[i] = make_float2(v[2 * i], v[2 * i + 1]);
        const float2 r2 = make_float2(rho, rho), t2 = make_float2(tau, tau);
#pragma unroll 4
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int i = 0; i < kProbeLanes / 2; ++i) w[i] = __ffma2_rn(w[i], r2, t2);
        }
#pragma unroll
        for (int i = 0; i < kProbeLanes / 2; ++i) {
            v[2 * i] = w[i].x;
            v[2 * i + 1] = w[i].y;
        }
    } else {
#pragma unroll 4
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int i = 0; i < kProbeLanes; ++i) v[i] = fmaf(v[i], rho, tau);
        }
    }
#pragma unroll
    for (int step = 1; step < kProbeLanes; step *= 2) {
#pragma unroll
        for (int i = 0; i + step < kProbeLanes; i += 2 * step) v[i] += v[i + step];
    }
    out[g] = v[0];
}

// HBM read probe.  Block b reads its own contiguous slice of the buffer (16-byte words),
// each thread four words 4 KiB apart per step, so every warp keeps four 512-byte requests
// in flight and each block walks its slice front to back.  The words are folded with XOR
// (integer work, far below the load rate) and each block stores its fold in fold[b]: the
// XOR of all folds equals the XOR of every 32-bit word of the buffer, which the caller can
// check, so no load can be dropped.
__global__ void __launch_bounds__(256) hbm_read_probe_kernel(const uint4* __restrict__ x, int64_t words,
                                                             uint32_t* fold) {
    const int64_t per = (words + gridDim.x - 1) / gridDim.x;
    const int64_t begin = static_cast<int64_t>(blockIdx.x) * per;
    const int64_t end = begin + per < words ? begin + per : words;
    uint32_t f = 0;
    int64_t i = begin + threadIdx.x;
    for (; i + 3 * 256 < end; i += 4 * 256) {
        const uint4 a = __ldcs(x + i), b = __ldcs(x + i + 256);
        const uint4 c = __ldcs(x + i + 512), d = __ldcs(x + i + 768);
        f ^= (a.x ^ a.y ^ a.z ^ a.w) ^ (b.x ^ b.y ^ b.z ^ b.w) ^ (c.x ^ c.y ^ c.z ^ c.w) ^ (d.x ^ d.y ^ d.z ^ d.w);
    }
    for (; i < end; i += 256) {
        const uint4 a = __ldcs(x + i);
        f ^= a.x ^ a.y ^ a.z ^ a.w;
    }
    f = __reduce_xor_sync(0xffffffffu, f);
    __shared__ uint32_t warp_fold[8];
    if (threadIdx.x % 32 == 0) warp_fold[threadIdx.x / 32] = f;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
        for (int w = 0; w < 8; ++w) t ^= warp_fold[w];
        fold[blockIdx.x] = t;
    }
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
    const float rho = 1.0f - 1.0f / 4096.0f, tau = 1.0f / 8192.0f;
    if (packed)
        fp32_issue_probe_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(out, iters, rho, tau);
    else
        fp32_issue_probe_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(out, iters, rho, tau);
    return cudaGetLastError();
}

cudaError_t probe_stream_read_launch(const float* x, int64_t n, uint32_t* fold, int64_t blocks,
                                     cudaStream_t stream) {
    hbm_read_probe_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(reinterpret_cast<const uint4*>(x),
                                                                             n / 4, fold);
    return cudaGetLastError();
}

cudaError_t probe_mma_f16_launch(int64_t ctas, int iters, int n, float* sink, unsigned int* status,
                                 cudaStream_t stream) {
    auto run = [&](auto kernel, uint32_t bytes) {
        cudaError_t err = set_func_attr_once(reinterpret_cast<const void*>(kernel),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
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
