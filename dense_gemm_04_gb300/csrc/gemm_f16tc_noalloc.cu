// gemm_f16tc_noalloc.cu -- the f16 tensor-core GEMM for callers that cannot allocate device
// memory.
//
// phx_gemm_f16tc_f32acc needs scratch memory for the f16-rounded copies of A and B, and takes
// it from a device memory pool at every call.  Some callers cannot allocate device memory
// at all once they are running: code in a latency-critical loop that must never wait on
// the allocator (an allocation can block, grow the pool, or fail under memory pressure),
// and plug-ins inside a host application that owns the whole device-memory budget and
// forbids allocations behind its back.  phx_gemm_f16tc_f32acc_noalloc serves them: it runs
// the same cast pass and the same tensor-core kernel, but its scratch is the file-scope
// array below, which the CUDA runtime sets up with this library's device code, so the call
// itself allocates nothing.
//
// The array is 64 MiB (kNoAllocScratchBytes): the scratch of a 4096 x 4096 x 4096 problem,
// the f16 copies of A and B, fits exactly.  Every GPU that loads this part of the library
// holds those 64 MiB until the process exits.  All calls share the one array, on every
// stream, so calls whose work overlaps on the GPU race with each other: order them on one
// stream, or synchronise.  Each call rewrites every byte of scratch it reads (the cast pass
// writes the zero padding too; split-K slices write whole planes), so nothing has to be
// cleared between calls.  The array also holds the status word of the kernels' bounded
// waits, which phx_check_device_status reads and clears.
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>

#include "../../include/phx.h"
#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

// Status word for the kernels' bounded waits, then the operand scratch (256-byte aligned).
constexpr size_t kStatusBytes = 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kStatusBytes + kNoAllocScratchBytes];

struct NoAllocDevice {
    phx_status status = PHX_ERR_ARCH;
    unsigned char* base = nullptr;  // device address of g_noalloc_scratch on this device
    int sm_count = 0;
};

std::mutex g_noalloc_mu;
std::map<int, NoAllocDevice> g_noalloc_dev;

// Once per device, with that device current: check the architecture and look up the
// device address of the scratch array.  Only the address is used on the host; the array's
// name in host code is a host-side stand-in, never a device pointer.
phx_status noalloc_setup(const NoAllocDevice** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return PHX_ERR_ARCH;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    auto it = g_noalloc_dev.find(dev);
    if (it == g_noalloc_dev.end()) {
        NoAllocDevice d;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            d.status = PHX_ERR_ARCH;
        } else if (major != 10 || minor != 3) {
            d.status = PHX_ERR_ARCH;
        } else {
            void* p = nullptr;
            const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (err != cudaSuccess || p == nullptr) {
                cudaGetLastError();
                d.status = PHX_ERR_LAUNCH;
            } else {
                d.base = static_cast<unsigned char*>(p);
                d.status = PHX_OK;
            }
        }
        it = g_noalloc_dev.emplace(dev, d).first;
    }
    *out = &it->second;
    return it->second.status;
}

}  // namespace

namespace phx {

cudaError_t noalloc_take_status(unsigned int* word) {
    *word = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorNoDevice;
    unsigned char* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        auto it = g_noalloc_dev.find(dev);
        if (it == g_noalloc_dev.end() || it->second.status != PHX_OK) return cudaSuccess;
        base = it->second.base;
    }
    cudaError_t err = cudaMemcpy(word, base, sizeof *word, cudaMemcpyDeviceToHost);
    if (err == cudaSuccess) err = cudaMemset(base, 0, sizeof *word);
    return err;
}

}  // namespace phx

extern "C" phx_status phx_gemm_f16tc_f32acc_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                                    const float* A, const float* B, float beta,
                                                    float* C, phx_stream_t stream) {
    phx_status st = phx_validate_args(M, N, K, A, B, C);
    if (st != PHX_OK) return st;
    if (M == 0 || N == 0) return PHX_OK;
    const NoAllocDevice* d = nullptr;
    st = noalloc_setup(&d);
    if (st != PHX_OK) return st;
    if (K == 0 || alpha == 0.f) {
        if (beta == 1.f) return PHX_OK;
        return phx::scale_c_launch(M, N, beta, C, stream) == cudaSuccess ? PHX_OK : PHX_ERR_LAUNCH;
    }
    const int cfg = phx::choose_config_for(PHX_VARIANT_F16TC, M, N, K, d->sm_count);
    if (cfg < 0) return cfg == phx::kBadConfigPin ? PHX_ERR_CONFIG : PHX_ERR_INTERNAL;
    unsigned int* status_word = reinterpret_cast<unsigned int*>(d->base);
    void* workspace = d->base + kStatusBytes;
    if (phx::is_skinny_config(PHX_VARIANT_F16TC, cfg)) {
        // few rows of A (or few columns): no rounded copies; the scratch holds the K slices'
        // partial sums
        if (phx::skinny_run_bytes(PHX_VARIANT_F16TC, 0, 0, M, N, K, A, B, d->sm_count) > kNoAllocScratchBytes)
            return PHX_ERR_NOMEM;
        return phx::skinny_run(PHX_VARIANT_F16TC, 0, 0, M, N, K, alpha, A, B, beta, C, workspace, d->sm_count,
                               stream) == cudaSuccess
                   ? PHX_OK : PHX_ERR_LAUNCH;
    }
    // the same scratch layout and kernels as the pooled entry point (split-K planes included),
    // so the results are the same bit for bit
    if (phx::f16tc_run_bytes(cfg, M, N, K, d->sm_count) > kNoAllocScratchBytes) return PHX_ERR_NOMEM;
    return phx::f16tc_run(cfg, 0, 0, M, N, K, alpha, A, B, beta, C, workspace, status_word, d->sm_count,
                          stream) == cudaSuccess
               ? PHX_OK : PHX_ERR_LAUNCH;
}

extern "C" phx_status phx_selftest_bounded_wait_noalloc(uint64_t limit_ns, phx_stream_t stream) {
    const NoAllocDevice* d = nullptr;
    const phx_status st = noalloc_setup(&d);
    if (st != PHX_OK) return st;
    if (limit_ns < 1000) limit_ns = 1000;
    if (limit_ns > 1000000000ull) limit_ns = 1000000000ull;
    return phx::selftest_wait_launch(limit_ns, reinterpret_cast<unsigned int*>(d->base), stream) == cudaSuccess
               ? PHX_OK : PHX_ERR_LAUNCH;
}
