// gemm_f16cvt.cu -- the f16 tensor-core GEMM with A rounded to f16 inside the kernel.
//
// The arithmetic is that of gemm_f16tc.cu: every element of A and B rounded to the nearest
// f16 (ties to even), the f16 x f16 products summed in f32 by tcgen05.mma.kind::f16, then
// alpha * acc + beta * c_old ("gemm on tensor cores", phobos-lang.dev/docs/examples/
// gemm-fp16tc-fp32acc/, section "What changes").  The difference is where A is rounded.
//
// For a problem with many rows and few columns (N within one or two tiles) A is most of the
// bytes, and the GEMM is bound by memory.  The separate rounding pass would read A, write
// its f16 copy (half of A's bytes), and the GEMM would read that copy back: 1.5 x A's f32
// bytes on top of the one read of A the problem needs.  Here the kernel reads A (f32) once,
// rounds it on the way into shared memory, in the layout the MMA reads.  Only B, which is
// small on such shapes, still goes through the rounding pass (N x Kp f16, K-major) and
// arrives by TMA.
//
// A persistent kernel, one CTA per SM, 320 threads (10 warps):
//   warp 4      TMA producer: per 64-wide k block of a 128-row tile, the 128 x 64 f32 box of A
//               (unswizzled, zeros past M and K) into a staging ring three k blocks deep, and
//               the TILE_N x 64 f16 tile of B into the MMA ring.
//   warps 6-9   converters: warp 6 + w takes rows 32w .. 32w+31 of the staged box; each lane
//               reads 8 (row, 16-byte chunk) pairs of 8 floats, hands the staging slot back,
//               rounds them with cvt.rn.f16x2.f32 and stores the 8 halves at chunk c ^ (r % 8)
//               of row r of the MMA ring's A slot: the 128-byte swizzle that TMA's
//               CU_TENSOR_MAP_SWIZZLE_128B writes.  (When A's rows do not start on 16 bytes
//               there is no tensor map of A: the converters then load A from global memory
//               themselves, 4 bytes at a time.)
//   warp 5      MMA issuer: tcgen05.mma.cta_group::1 (M = 128, N = TILE_N, K = 16).
//   warps 0-3   epilogue: tcgen05.ld of the accumulator (warp w: rows 32w..32w+31), through
//               a per-warp shared-memory buffer to coalesced rows of C.
// An MMA ring slot is full when B's bytes have landed and the four converter warps have
// arrived (after a proxy fence that makes their generic stores visible to the tensor cores).
// The accumulator is double-buffered in tensor memory.  Every wait is bounded (sm100_ptx.cuh).
//
// The kernel is launched as a programmatic dependent of the pass that rounds B.  A does not
// depend on that pass: the producer issues A's first staging load, then waits for the pass
// (griddepcontrol.wait) before its first load of B.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "debug_checks.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace phx {
namespace {

using namespace ptx;

constexpr int kBM = 128;        // tcgen05 cta_group::1 M
constexpr int kBK = 64;         // 64 halves = 128 bytes = one swizzle row
constexpr int kUmmaK = 16;      // K of one kind::f16 MMA
constexpr int kEpiWarps = 4;    // warps 0-3
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kFirstConvWarp = 6;
constexpr int kConvWarps = 4;   // warps 6-9
constexpr int kThreads = 32 * (kFirstConvWarp + kConvWarps);

// How the converters get A: 0 four bytes at a time from global memory, 1 sixteen bytes at a
// time from global memory (rows on 16 bytes), 2 from the TMA staging ring.
enum AMode : int { kAScalar = 0, kAVector = 1, kATma = 2 };

template <int BN, int STAGES, int STG>
struct CvtLayout {
    static constexpr uint32_t kABytes = kBM * kBK * 2;      // f16 A slot of the MMA ring
    static constexpr uint32_t kBBytes = BN * kBK * 2;       // f16 B slot
    static constexpr uint32_t kStgBytes = kBM * kBK * 4;    // f32 A slot of the staging ring
    // offsets from the 1024-byte aligned base
    static constexpr uint32_t kA = 0;
    static constexpr uint32_t kB = STAGES * kABytes;
    static constexpr uint32_t kStg = kB + STAGES * kBBytes;
    // per epilogue warp: a 32 x 32 f32 chunk, rows padded to 36 floats
    static constexpr uint32_t kEpiStride = 36;
    static constexpr uint32_t kEpiWarpFloats = 32 * kEpiStride;
    static constexpr uint32_t kEpi = kStg + STG * kStgBytes;
    static constexpr uint32_t kBars = kEpi + kEpiWarps * kEpiWarpFloats * 4;  // 8-byte aligned
    // full, empty, staging full, staging empty, tfull[2], tempty[2], done
    static constexpr uint32_t kNumBars = 2 * STAGES + 2 * STG + 5;
    static constexpr uint32_t kTmemSlot = kBars + 8 * kNumBars;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kDynSmem = kAbort + 4 + 1024;  // + alignment slack
    static constexpr uint32_t kTmemCols = 2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512);
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "tcgen05 N, and whole 32-column chunks");
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "swizzle atoms stay 1024-aligned");
    static_assert(kDynSmem <= 227 * 1024, "fits one CTA's shared memory");
};

__device__ __forceinline__ float4 ld_stream4(const float* p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t half2_bits(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

template <int BN, int STAGES, int STG>
__global__ void __launch_bounds__(kThreads, 1)
gemm_f16cvt_kernel(const float* __restrict__ A, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, float* __restrict__ C, int M, int N, int K, int num_kb,
                   float alpha, float beta, int tiles_m, int tiles_n, unsigned int* status, int a_mode) {
    using L = CvtLayout<BN, STAGES, STG>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);

    const uint32_t sA = base + L::kA;
    const uint32_t sB = base + L::kB;
    const uint32_t sStg = base + L::kStg;
    const uint32_t bars = base + L::kBars;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    auto sfull_bar = [&](int s) { return bars + 8u * (2 * STAGES + s); };
    auto sempty_bar = [&](int s) { return bars + 8u * (2 * STAGES + STG + s); };
    auto tfull_bar = [&](int a) { return bars + 8u * (2 * STAGES + 2 * STG + a); };
    auto tempty_bar = [&](int a) { return bars + 8u * (2 * STAGES + 2 * STG + 2 + a); };
    const uint32_t done_bar = bars + 8u * (2 * STAGES + 2 * STG + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + L::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + L::kAbort);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const bool staged = a_mode == kATma;
    const int num_items = tiles_m * tiles_n;
    // item w: tile row w % tiles_m, tile column w / tiles_m (the CTAs at work at one time
    // share B's tile)
    auto tile_of = [&](int w, int& pm, int& pn) {
        pn = w / tiles_m;
        pm = w - pn * tiles_m;
    };

    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tmB);
        if (staged) tma_prefetch_desc(&tmA);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1 + kConvWarps);  // the producer's expect_tx + the converters
            mbar_init(empty_bar(s), 1);
        }
        for (int s = 0; s < STG; ++s) {
            mbar_init(sfull_bar(s), 1);
            mbar_init(sempty_bar(s), kConvWarps);
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
            // per ring slot: a load was issued (mask) and the parity of its phase
            uint32_t issued_mask = 0, issued_phase = 0, sissued_mask = 0, sissued_phase = 0;
            uint32_t stage = 0, phase = 0, sstage = 0, sphase = 0;
            bool ok = true;
            bool b_ready = false;  // the rounding pass of B has been waited for
            for (int w = blockIdx.x; w < num_items && ok; w += gridDim.x) {
                int pm, pn;
                tile_of(w, pm, pn);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (staged) {
                        // A does not depend on the rounding pass: its first loads go out
                        // before the wait for that pass
                        if (!mbar_wait(sempty_bar(sstage), sphase ^ 1u, abort_flag, status)) { ok = false; break; }
                        PHX_DCHECK(sstage < STG && pm < tiles_m);
                        mbar_arrive_expect_tx(sfull_bar(sstage), L::kStgBytes);
                        tma_load_2d(sStg + sstage * L::kStgBytes, &tmA, kb * kBK, pm * kBM, sfull_bar(sstage));
                        sissued_mask |= 1u << sstage;
                        sissued_phase = (sissued_phase & ~(1u << sstage)) | (sphase << sstage);
                        if (++sstage == STG) { sstage = 0; sphase ^= 1u; }
                    }
                    if (!b_ready) {
                        // B comes from the rounding pass just before this kernel, which may
                        // still be running
                        asm volatile("griddepcontrol.wait;" ::: "memory");
                        b_ready = true;
                    }
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, status)) { ok = false; break; }
                    PHX_DCHECK(stage < STAGES && pn < tiles_n);
                    mbar_arrive_expect_tx(full_bar(stage), L::kBBytes);
                    tma_load_2d(sB + stage * L::kBBytes, &tmB, kb * kBK, pn * BN, full_bar(stage));
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // let every load issued into this CTA land before it exits
                for (int s = 0; s < STAGES; ++s)
                    if (issued_mask & (1u << s)) mbar_wait_drain(full_bar(s), (issued_phase >> s) & 1u);
                for (int s = 0; s < STG; ++s)
                    if (sissued_mask & (1u << s)) mbar_wait_drain(sfull_bar(s), (sissued_phase >> s) & 1u);
            }
        }
    } else if (warp >= kFirstConvWarp) {
        const int cw = warp - kFirstConvWarp;  // rows 32cw .. 32cw+31 of each tile
        const int chunk = lane & 7;             // 16-byte chunk of a 128-byte f16 row
        uint32_t stage = 0, phase = 0, sstage = 0, sphase = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < num_items && ok; w += gridDim.x) {
            int pm, pn;
            tile_of(w, pm, pn);
            const int64_t row_base = static_cast<int64_t>(pm) * kBM + cw * 32;
            for (int kb = 0; kb < num_kb; ++kb) {
                const int k = kb * kBK + chunk * 8;
                float4 v[8][2];
                if (staged) {
                    // the f32 box (zeros past M and K) from the staging slot, then the slot
                    // goes back to the producer
                    if (!__all_sync(0xffffffffu, mbar_wait(sfull_bar(sstage), sphase, abort_flag, status))) {
                        ok = false;
                        break;
                    }
                    const float* stg = reinterpret_cast<const float*>(base_ptr + L::kStg + sstage * L::kStgBytes);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = cw * 32 + 4 * i + (lane >> 3);
                        v[i][0] = *reinterpret_cast<const float4*>(stg + r * kBK + chunk * 8);
                        v[i][1] = *reinterpret_cast<const float4*>(stg + r * kBK + chunk * 8 + 4);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sempty_bar(sstage));
                    if (++sstage == STG) { sstage = 0; sphase ^= 1u; }
                } else {
                    // straight from global memory, all 8 chunks' loads in flight together
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int64_t grow = row_base + 4 * i + (lane >> 3);
                        const float* src = A + grow * K + k;
                        if (grow < M && a_mode == kAVector && k + 8 <= K) {
                            v[i][0] = ld_stream4(src);
                            v[i][1] = ld_stream4(src + 4);
                        } else {
                            float t[8];
#pragma unroll
                            for (int q = 0; q < 8; ++q) t[q] = (grow < M && k + q < K) ? __ldg(src + q) : 0.f;
                            v[i][0] = make_float4(t[0], t[1], t[2], t[3]);
                            v[i][1] = make_float4(t[4], t[5], t[6], t[7]);
                        }
                    }
                }
                if (!__all_sync(0xffffffffu, mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, status))) {
                    ok = false;
                    break;
                }
                uint8_t* a_stage = base_ptr + L::kA + stage * L::kABytes;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = cw * 32 + 4 * i + (lane >> 3);  // row within the tile
                    uint4 h;
                    h.x = half2_bits(v[i][0].x, v[i][0].y);
                    h.y = half2_bits(v[i][0].z, v[i][0].w);
                    h.z = half2_bits(v[i][1].x, v[i][1].y);
                    h.w = half2_bits(v[i][1].z, v[i][1].w);
                    PHX_DCHECK(r < kBM && chunk < 8);
                    *reinterpret_cast<uint4*>(a_stage + r * 128 + ((chunk ^ (r & 7)) << 4)) = h;
                }
                // the stores become visible to the tensor cores' reads of the slot
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_bar(stage));
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32acc(kBM, BN);
            uint32_t stage = 0, phase = 0;
            uint32_t acc = 0, acc_phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < num_items && ok; w += gridDim.x) {
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                PHX_DCHECK(acc * BN + BN <= L::kTmemCols);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag, status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = sA + stage * L::kABytes;
                    const uint32_t b0 = sB + stage * L::kBBytes;
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        const uint64_t ad = sw128_kmajor_desc(a0 + k * kUmmaK * 2);
                        const uint64_t bd = sw128_kmajor_desc(b0 + k * kUmmaK * 2);
                        mma_f16_ss(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                    }
                    mma_commit(empty_bar(stage));  // the slot is free once these MMAs are done
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(tfull_bar(acc));
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            // every MMA this thread issued has completed once done_bar fires
            mma_commit(done_bar);
            mbar_wait_drain(done_bar, 0);
        }
    } else {
        // epilogue, warps 0-3: warp w owns TMEM lanes (rows) 32w .. 32w+31
        float* epi = reinterpret_cast<float*>(base_ptr + L::kEpi) + warp * L::kEpiWarpFloats;
        const bool vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15u) == 0);
        const bool read_c = beta != 0.f;
        uint32_t acc = 0, acc_phase = 0;
        for (int w = blockIdx.x; w < num_items; w += gridDim.x) {
            int pm, pn;
            tile_of(w, pm, pn);
            // warp-uniform outcome: tcgen05.ld below is .sync.aligned
            if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), acc_phase, abort_flag, status))) break;
            tc_fence_after();
            const int row0 = pm * kBM + warp * 32;
            const uint32_t t_base = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + acc * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                const int col0 = pn * BN + c * 32;
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_base + c * 32, r);
                tmem_ld_wait();
                if (col0 >= N || row0 >= M) continue;  // warp-uniform: nothing of C here
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<float4*>(epi + lane * L::kEpiStride + q * 4) =
                        make_float4(__uint_as_float(r[q * 4 + 0]), __uint_as_float(r[q * 4 + 1]),
                                    __uint_as_float(r[q * 4 + 2]), __uint_as_float(r[q * 4 + 3]));
                __syncwarp();
                if (vec) {
                    // four rows of 128 bytes per instruction
                    const int cc = (lane % 8) * 4;
                    const int col = col0 + cc;
                    float4 cv[8];
                    if (read_c) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const int row = row0 + q * 4 + lane / 8;
                            cv[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (row < M && col < N)
                                cv[q] = *reinterpret_cast<const float4*>(C + static_cast<int64_t>(row) * N + col);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int rr = q * 4 + lane / 8;
                        const int row = row0 + rr;
                        if (row < M && col < N) {
                            const float4 a = *reinterpret_cast<const float4*>(epi + rr * L::kEpiStride + cc);
                            float4 o = make_float4(alpha * a.x, alpha * a.y, alpha * a.z, alpha * a.w);
                            if (read_c) {
                                o.x = fmaf(beta, cv[q].x, o.x);
                                o.y = fmaf(beta, cv[q].y, o.y);
                                o.z = fmaf(beta, cv[q].z, o.z);
                                o.w = fmaf(beta, cv[q].w, o.w);
                            }
                            PHX_DCHECK(col + 3 < N);
                            *reinterpret_cast<float4*>(C + static_cast<int64_t>(row) * N + col) = o;
                        }
                    }
                } else {
                    // one row of 32 columns per instruction; the 32 loads of C first
                    const int col = col0 + lane;
                    float cs[32];
                    if (read_c) {
#pragma unroll
                        for (int rr = 0; rr < 32; ++rr) {
                            const int row = row0 + rr;
                            cs[rr] = (row < M && col < N) ? C[static_cast<int64_t>(row) * N + col] : 0.f;
                        }
                    }
#pragma unroll
                    for (int rr = 0; rr < 32; ++rr) {
                        const int row = row0 + rr;
                        if (row < M && col < N) {
                            float o = alpha * epi[rr * L::kEpiStride + lane];
                            if (read_c) o = fmaf(beta, cs[rr], o);
                            C[static_cast<int64_t>(row) * N + col] = o;
                        }
                    }
                }
                __syncwarp();  // the buffer is rewritten by the next chunk
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));  // the accumulator buffer may be reused
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

using CvtKernelFn = void (*)(const float*, CUtensorMap, CUtensorMap, float*, int, int, int, int, float, float,
                             int, int, unsigned int*, int);

struct CvtEntry {
    F16Config cfg;
    CvtKernelFn fn;
    uint32_t smem;
};

template <int BN, int STAGES, int STG>
CvtEntry make_cvt_entry() {
    return CvtEntry{F16Config{kBM, BN, kBK, STAGES, 1, 1}, &gemm_f16cvt_kernel<BN, STAGES, STG>,
                    CvtLayout<BN, STAGES, STG>::kDynSmem};
}

// At each width 96 KB of MMA ring (4 slots of 24 KB, 3 of 32 KB, 2 of 48 KB) and 96 KB of
// f32 staging (3 k blocks of A in flight per SM).
const CvtEntry kCvtEntries[] = {
    make_cvt_entry<64, 4, 3>(),
    make_cvt_entry<128, 3, 3>(),
    make_cvt_entry<256, 2, 3>(),
};
constexpr int kNumCvt = sizeof(kCvtEntries) / sizeof(kCvtEntries[0]);

}  // namespace

int f16cvt_num_configs() { return kNumCvt; }

const F16Config& f16cvt_config(int index) { return kCvtEntries[index].cfg; }

int64_t debug_take_f16cvt() { return debug_take_local(); }

cudaError_t f16cvt_gemm_launch(int index, int64_t M, int64_t N, int64_t K, float alpha, float beta, float* C,
                               const float* A, const __half* Bt, int64_t ldb, unsigned int* status, int num_sms,
                               cudaStream_t stream) {
    if (index < 0 || index >= kNumCvt || M <= 0 || N <= 0 || K <= 0 || num_sms <= 0) return cudaErrorInvalidValue;
    const CvtEntry& e = kCvtEntries[index];
    const int bn = e.cfg.tile_n;
    const int64_t Kp = (K + 7) / 8 * 8;
    CUtensorMap mapB;
    if (!f16_operand_map(&mapB, Bt, N, Kp, bn, ldb)) return cudaErrorInvalidValue;
    const int64_t tiles_m = (M + kBM - 1) / kBM;
    const int64_t tiles_n = (N + bn - 1) / bn;
    const int64_t items = tiles_m * tiles_n;
    if (items > 0x7FFFFFFF || M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const int grid = static_cast<int>(items < num_sms ? items : num_sms);
    const int num_kb = static_cast<int>((K + kBK - 1) / kBK);
    // A through the TMA staging ring when its rows can be a tensor map (K % 4 == 0, 16-byte
    // aligned); else the converters load it themselves
    const bool a_al = (K % 4 == 0) && ((reinterpret_cast<uintptr_t>(A) & 15u) == 0);
    CUtensorMap mapA;
    std::memset(&mapA, 0, sizeof mapA);
    int a_mode = a_al ? kAVector : kAScalar;
    if (a_al && f32_rows_map(&mapA, A, M, K, kBK, kBM)) a_mode = kATma;
    cudaError_t err = set_func_attr_once(reinterpret_cast<const void*>(e.fn),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(e.smem));
    if (err != cudaSuccess) return err;
    // a programmatic dependent of the pass that rounds B (see the top of this file)
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(grid));
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = e.smem;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const int m32 = static_cast<int>(M), n32 = static_cast<int>(N), k32 = static_cast<int>(K);
    const int tm32 = static_cast<int>(tiles_m), tn32 = static_cast<int>(tiles_n);
    err = cudaLaunchKernelEx(&lc, e.fn, A, mapA, mapB, C, m32, n32, k32, num_kb, alpha, beta, tm32, tn32, status,
                             a_mode);
    if (err != cudaSuccess) {
        // a stream that does not take programmatic launches: launch normally
        cudaGetLastError();
        lc.numAttrs = 0;
        err = cudaLaunchKernelEx(&lc, e.fn, A, mapA, mapB, C, m32, n32, k32, num_kb, alpha, beta, tm32, tn32,
                                 status, a_mode);
    }
    return launched(err);
}

}  // namespace phx
