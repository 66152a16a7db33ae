// gemm_f16tc.cu -- f16 tensor cores with f32 accumulation on sm_103a (tcgen05 + TMA).
//
// C <- alpha * A @ B + beta * C, where every element of the f32 operands A and B is first
// rounded to the nearest f16 (ties to even) and the f16 x f16 products are summed in f32
// ("gemm on tensor cores", phobos-lang.dev/docs/examples/gemm-fp16tc-fp32acc/, section
// "What changes"; the tile structure is the same as "gemm, f32", sections "One output tile
// per CTA", "The k loop", "The epilogue").
//
// Two passes:
//   1. Cast (HBM-bound): A (M x K f32) -> Ah (M x Kp f16, row-major) and B (K x N f32) ->
//      Bt (N x Kp f16, B transposed) with cvt.rn (round to nearest even); Kp = K rounded up
//      to a multiple of 8 so every row starts on 16 bytes, the TMA stride rule; the pad
//      columns are written as zeros.  Both operands end up K-major, the layout the
//      tensor-core descriptors below describe.
//   2. GEMM: a persistent, warp-specialised kernel, one CTA per SM, 192 threads:
//        warp 4      TMA producer: loads 128 x 64 tiles of Ah and TILE_N x 64 tiles of Bt
//                    (128-byte swizzle) into a STAGES-deep shared-memory ring;
//        warp 5      MMA issuer: one thread issues tcgen05.mma.kind::f16 (M = 128,
//                    N = TILE_N, K = 16; four per 64-wide k block) into an f32 accumulator
//                    in tensor memory, and tcgen05.commit frees each ring slot;
//        warps 0-3   epilogue: tcgen05.ld of the accumulator (warp w owns TMEM lanes, i.e.
//                    rows, 32w..32w+31), alpha * acc + beta * c_old, store to C.
//      The accumulator is double-buffered in TMEM (2 x TILE_N columns), so the epilogue
//      of one tile overlaps the main loop of the next.  Edges: TMA fills rows and k
//      columns past the tensor with zeros; the epilogue skips stores past M and N.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace phx {
namespace {

using namespace ptx;

constexpr int kBM = 128;         // tcgen05 cta_group::1 M
constexpr int kBK = 64;          // 64 halves = 128 bytes = one swizzle row
constexpr int kUmmaK = 16;       // K of one kind::f16 MMA
constexpr int kEpiWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreadsTc = 192;

__host__ __device__ constexpr int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// ---------------------------------------------------------------------------------------
// Cast pass
// ---------------------------------------------------------------------------------------

// A (rows x K, f32) -> Ah (rows x Kp, f16), each thread writing 8 halves (16 bytes).
__global__ void cast_rows_kernel(const float* __restrict__ A, __half* __restrict__ Ah,
                                 int64_t rows, int64_t K, int64_t Kp, int vec) {
    const int64_t chunks = Kp / 8;
    const int64_t total = rows * chunks;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += stride) {
        const int64_t r = idx / chunks;
        const int64_t c = (idx - r * chunks) * 8;
        const float* src = A + r * K + c;
        float v[8];
        if (vec && c + 8 <= K) {
            const float4 x = __ldcs(reinterpret_cast<const float4*>(src));
            const float4 y = __ldcs(reinterpret_cast<const float4*>(src + 4));
            v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
            v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = (c + q < K) ? src[q] : 0.f;
        }
        uint4 out;
        __half2 h;
        h = __floats2half2_rn(v[0], v[1]); out.x = *reinterpret_cast<uint32_t*>(&h);
        h = __floats2half2_rn(v[2], v[3]); out.y = *reinterpret_cast<uint32_t*>(&h);
        h = __floats2half2_rn(v[4], v[5]); out.z = *reinterpret_cast<uint32_t*>(&h);
        h = __floats2half2_rn(v[6], v[7]); out.w = *reinterpret_cast<uint32_t*>(&h);
        *reinterpret_cast<uint4*>(Ah + r * Kp + c) = out;
    }
}

// B (K x N, f32) -> Bt (N x Kp, f16): 64 x 64 tiles through shared memory.
constexpr int kTT = 64;
__global__ void __launch_bounds__(256) cast_transpose_kernel(const float* __restrict__ B,
                                                             __half* __restrict__ Bt, int64_t K,
                                                             int64_t N, int64_t Kp) {
    __shared__ float tile[kTT][kTT + 1];  // [k][n]
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kTT;
    const int64_t k0 = static_cast<int64_t>(blockIdx.y) * kTT;
    const int tid = threadIdx.x;
#pragma unroll
    for (int i = 0; i < kTT * kTT / 256; ++i) {
        const int e = tid + i * 256;
        const int k = e / kTT;
        const int n = e % kTT;
        const int64_t gk = k0 + k;
        const int64_t gn = n0 + n;
        tile[k][n] = (gk < K && gn < N) ? __ldcs(B + gk * N + gn) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kTT * (kTT / 8) / 256; ++i) {
        const int e = tid + i * 256;
        const int n = e / (kTT / 8);
        const int kc = (e % (kTT / 8)) * 8;
        const int64_t gn = n0 + n;
        const int64_t gk = k0 + kc;
        if (gn < N && gk < Kp) {
            uint4 out;
            __half2 h;
            h = __floats2half2_rn(tile[kc + 0][n], tile[kc + 1][n]); out.x = *reinterpret_cast<uint32_t*>(&h);
            h = __floats2half2_rn(tile[kc + 2][n], tile[kc + 3][n]); out.y = *reinterpret_cast<uint32_t*>(&h);
            h = __floats2half2_rn(tile[kc + 4][n], tile[kc + 5][n]); out.z = *reinterpret_cast<uint32_t*>(&h);
            h = __floats2half2_rn(tile[kc + 6][n], tile[kc + 7][n]); out.w = *reinterpret_cast<uint32_t*>(&h);
            *reinterpret_cast<uint4*>(Bt + gn * Kp + gk) = out;
        }
    }
}

// ---------------------------------------------------------------------------------------
// GEMM kernel
// ---------------------------------------------------------------------------------------

// Tile order: groups of 8 tile rows, walked column by column, so the tiles the resident
// CTAs work on at one time share panels of A and B in L2.
__device__ __forceinline__ void tc_tile_coords(int t, int tiles_m, int tiles_n, int& pm, int& pn) {
    constexpr int kGroup = 8;
    const int per_group = kGroup * tiles_n;
    const int group = t / per_group;
    const int first_m = group * kGroup;
    const int rows = min(tiles_m - first_m, kGroup);
    const int r = t - group * per_group;
    pm = first_m + r % rows;
    pn = r / rows;
}

template <int BN, int STAGES>
struct TcLayout {
    static constexpr uint32_t kABytes = kBM * kBK * 2;
    static constexpr uint32_t kBBytes = BN * kBK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kTmemCols = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64
                                          : (2 * BN <= 128) ? 128 : (2 * BN <= 256) ? 256 : 512;
    // offsets from the 1024-byte aligned base
    static constexpr uint32_t kA = 0;
    static constexpr uint32_t kB = STAGES * kABytes;
    static constexpr uint32_t kBars = STAGES * kStageBytes;           // 8-byte aligned
    static constexpr uint32_t kNumBars = 2 * STAGES + 4 + 1;          // full, empty, tfull, tempty, done
    static constexpr uint32_t kTmemSlot = kBars + 8 * kNumBars;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kEnd = kAbort + 4;
    static constexpr uint32_t kDynSmem = kEnd + 1024;                 // + alignment slack
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "tcgen05 M=128 needs N % 16 == 0, N <= 256");
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "swizzle atoms stay 1024-aligned");
};

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreadsTc, 1)
gemm_f16tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  float* __restrict__ C, int M, int N, int num_kb, float alpha, float beta,
                  int tiles_m, int tiles_n, unsigned int* status) {
    using L = TcLayout<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);

    const uint32_t sA = base + L::kA;
    const uint32_t sB = base + L::kB;
    const uint32_t bars = base + L::kBars;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bars + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bars + 8u * (2 * STAGES + 2 + a); };
    const uint32_t done_bar = bars + 8u * (2 * STAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + L::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + L::kAbort);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int num_tiles = tiles_m * tiles_n;

    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), kEpiWarps);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            // issued[s]: bit 0 = a load was ever issued into slot s, bit 1 = its phase parity
            uint32_t issued_mask = 0, issued_phase = 0;
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                int pm, pn;
                tc_tile_coords(t, tiles_m, tiles_n, pm, pn);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, status)) { ok = false; break; }
                    mbar_arrive_expect_tx(full_bar(stage), L::kStageBytes);
                    tma_load_2d(sA + stage * L::kABytes, &tmA, kb * kBK, pm * kBM, full_bar(stage));
                    tma_load_2d(sB + stage * L::kBBytes, &tmB, kb * kBK, pn * BN, full_bar(stage));
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // Aborted: let every load this thread issued land before the CTA exits.
                for (int s = 0; s < STAGES; ++s)
                    if (issued_mask & (1u << s)) mbar_wait_drain(full_bar(s), (issued_phase >> s) & 1u);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32acc(kBM, BN);
            uint32_t stage = 0, phase = 0;
            uint32_t acc = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag, status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = sA + stage * L::kABytes;
                    const uint32_t b0 = sB + stage * L::kBBytes;
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        mma_f16_ss(d_tmem, sw128_kmajor_desc(a0 + k * kUmmaK * 2),
                                   sw128_kmajor_desc(b0 + k * kUmmaK * 2), idesc,
                                   (kb | k) != 0 ? 1u : 0u);
                    }
                    mma_commit(empty_bar(stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(tfull_bar(acc));
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            // Every MMA this thread issued has completed once done_bar fires.
            mma_commit(done_bar);
            mbar_wait_drain(done_bar, 0);
        }
    } else if (warp < kEpiWarps) {
        uint32_t acc = 0, acc_phase = 0;
        const bool read_c = beta != 0.f;
        const bool vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15u) == 0);
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            int pm, pn;
            tc_tile_coords(t, tiles_m, tiles_n, pm, pn);
            // warp-uniform outcome: the tcgen05.ld below is .sync.aligned
            if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), acc_phase, abort_flag, status))) break;
            tc_fence_after();
            const int row = pm * kBM + warp * 32 + lane;
            float* crow = C + static_cast<int64_t>(row) * N;
            const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + acc * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_addr + c * 32, r);
                tmem_ld_wait();
                const int col0 = pn * BN + c * 32;
                if (row < M) {
                    if (vec && col0 + 32 <= N) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            float4* p = reinterpret_cast<float4*>(crow + col0 + q * 4);
                            float4 o;
                            o.x = alpha * __uint_as_float(r[q * 4 + 0]);
                            o.y = alpha * __uint_as_float(r[q * 4 + 1]);
                            o.z = alpha * __uint_as_float(r[q * 4 + 2]);
                            o.w = alpha * __uint_as_float(r[q * 4 + 3]);
                            if (read_c) {
                                const float4 cv = *p;
                                o.x = fmaf(beta, cv.x, o.x);
                                o.y = fmaf(beta, cv.y, o.y);
                                o.z = fmaf(beta, cv.z, o.z);
                                o.w = fmaf(beta, cv.w, o.w);
                            }
                            *p = o;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            if (col0 + j < N) {
                                float o = alpha * __uint_as_float(r[j]);
                                if (read_c) o = fmaf(beta, crow[col0 + j], o);
                                crow[col0 + j] = o;
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, L::kTmemCols);
    }
}

// ---------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Tensor map of a row-major f16 matrix (rows x Kp) read in boxes of 64 halves x box_rows,
// 128-byte swizzle, zero fill outside the matrix.
bool make_map(CUtensorMap* map, const __half* ptr, int64_t rows, int64_t Kp, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(Kp), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(Kp) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(ptr), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

using TcKernelFn = void (*)(CUtensorMap, CUtensorMap, float*, int, int, int, float, float, int,
                            int, unsigned int*);

struct TcEntry {
    F16Config cfg;
    TcKernelFn fn;
    uint32_t smem;
};

template <int BN, int STAGES>
TcEntry make_tc_entry() {
    return TcEntry{F16Config{kBM, BN, kBK, STAGES}, &gemm_f16tc_kernel<BN, STAGES>,
                   TcLayout<BN, STAGES>::kDynSmem};
}

const TcEntry kTcEntries[] = {
    make_tc_entry<256, 4>(), make_tc_entry<256, 3>(), make_tc_entry<128, 6>(),
    make_tc_entry<128, 4>(), make_tc_entry<64, 8>(),
};
constexpr int kNumTc = sizeof(kTcEntries) / sizeof(kTcEntries[0]);

}  // namespace

int f16tc_num_configs() { return kNumTc; }

const F16Config& f16tc_config(int index) { return kTcEntries[index].cfg; }

size_t f16tc_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    const int64_t Kp = round_up(K, 8);
    return static_cast<size_t>(round_up(M * Kp * 2, 256) + round_up(N * Kp * 2, 256));
}

cudaError_t f16tc_cast_launch(int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                              void* workspace, int num_sms, cudaStream_t stream) {
    const int64_t Kp = round_up(K, 8);
    __half* Ah = static_cast<__half*>(workspace);
    __half* Bt = reinterpret_cast<__half*>(static_cast<char*>(workspace) + round_up(M * Kp * 2, 256));
    const int vec = (K % 4 == 0) && ((reinterpret_cast<uintptr_t>(A) & 15u) == 0);
    const int64_t total = M * (Kp / 8);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    cast_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(A, Ah, M, K, Kp, vec);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const dim3 grid(static_cast<unsigned>((N + kTT - 1) / kTT), static_cast<unsigned>((Kp + kTT - 1) / kTT));
    if (grid.y > 65535u) return cudaErrorInvalidValue;
    cast_transpose_kernel<<<grid, 256, 0, stream>>>(B, Bt, K, N, Kp);
    return cudaGetLastError();
}

cudaError_t f16tc_gemm_launch(int index, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                              float* C, const void* workspace, unsigned int* status, int num_sms,
                              cudaStream_t stream) {
    const TcEntry& e = kTcEntries[index];
    const int64_t Kp = round_up(K, 8);
    const __half* Ah = static_cast<const __half*>(workspace);
    const __half* Bt = reinterpret_cast<const __half*>(static_cast<const char*>(workspace) +
                                                       round_up(M * Kp * 2, 256));
    CUtensorMap mapA, mapB;
    if (!make_map(&mapA, Ah, M, Kp, kBM) || !make_map(&mapB, Bt, N, Kp, e.cfg.tile_n))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(reinterpret_cast<const void*>(e.fn),
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(e.smem));
    if (err != cudaSuccess) return err;
    const int tiles_m = static_cast<int>((M + kBM - 1) / kBM);
    const int tiles_n = static_cast<int>((N + e.cfg.tile_n - 1) / e.cfg.tile_n);
    const int64_t tiles = static_cast<int64_t>(tiles_m) * tiles_n;
    const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
    const int num_kb = static_cast<int>((K + kBK - 1) / kBK);
    e.fn<<<grid, kThreadsTc, e.smem, stream>>>(mapA, mapB, C, static_cast<int>(M),
                                               static_cast<int>(N), num_kb, alpha, beta, tiles_m,
                                               tiles_n, status);
    return cudaGetLastError();
}

}  // namespace phx
