// gemm_f16cvt.cu -- the f16 tensor-core GEMM with operands rounded to f16 inside the kernel.
//
// The arithmetic is that of gemm_f16tc.cu: every element of A and B rounded to the nearest
// f16 (ties to even), the f16 x f16 products summed in f32 by tcgen05.mma.kind::f16, then
// alpha * acc + beta * c_old ("gemm on tensor cores", phobos-lang.dev/docs/examples/
// gemm-fp16tc-fp32acc/, section "What changes").  The difference is where the large operand
// is rounded.
//
// When one operand is most of a problem's bytes, the GEMM is bound by memory, and the
// separate rounding pass would read that operand, write its f16 copy (half its bytes) and
// the GEMM would read the copy back: 1.5 x its f32 bytes on top of the one read the problem
// needs.  Here the kernel reads that operand (f32) once and rounds it on the way into shared
// memory, in the layout the MMA reads; the other, small operand still goes through the
// rounding pass (K-major f16) and arrives by TMA.
//   CONVERT_A: many rows, few columns (N within a tile or two).  A is staged as 128 x 64 f32
//     boxes; B comes from the pass as N x Kp f16.
//   CONVERT_B: few rows (up to a tile or two), many columns.  B is staged as 64 x TILE_N f32
//     boxes (k rows of n) and transposed while it is rounded; A comes from the pass as M x Kp
//     f16.
//   CONVERT_A + CONVERT_B: both operands staged and rounded here, no pass at all: one launch,
//     no scratch unless K is split (for small problems, where the launches and the pass are
//     most of the time).
// In every mode, a grid whose tiles cannot give every SM work is split along K (at most 8
// slices of at least 8 k blocks) into slices that write f32 partial planes, added in slice
// order by a separate reduction.
//
// A persistent kernel, one CTA per SM, 320 threads (10 warps):
//   warp 4      TMA producer: per 64-deep k block, the f32 box of each converted operand into
//               a staging ring (unswizzled, zeros past the edges; one slot holds both boxes
//               when both are converted), and the f16 tile of the other operand, if any, into
//               the MMA ring.
//   warps 6-9   converters.  Each lane reads 8 (row, 16-byte chunk) pairs of 8 floats from
//               the staged box, hands the staging slot back, rounds them with
//               cvt.rn.f16x2.f32 and stores the 8 halves at chunk c ^ (r % 8) of row r of
//               the MMA ring's slot: the 128-byte swizzle TMA's CU_TENSOR_MAP_SWIZZLE_128B
//               writes, so the MMA descriptors are those of gemm_f16tc.cu.  For A a row of
//               the slot is a row of the box; for B a row of the slot (one n) is a column of
//               the box, read 8 k rows apart.  (Without a tensor map of the operand, rows not
//               on 16 bytes, the converters load it from global memory themselves.)
//   warp 5      MMA issuer: tcgen05.mma.cta_group::1 (M = 128, N = TILE_N, K = 16).
//   warps 0-3   epilogue: tcgen05.ld of the accumulator (warp w: rows 32w..32w+31), through
//               a per-warp shared-memory buffer to coalesced rows of C (or of a k slice's
//               partial plane).
// An MMA ring slot is full when the TMA bytes of the other operand (if any) have landed and
// the four converter warps have arrived (after a proxy fence that makes their generic stores
// visible to the tensor cores).
// The accumulator is double-buffered in tensor memory.  Every wait is bounded (sm100_ptx.cuh).
//
// With one operand converted, the kernel is launched as a programmatic dependent of the
// rounding pass.  The converted operand does not depend on that pass: the producer issues its
// first staging load, then waits for the pass (griddepcontrol.wait) before the first load of
// the other operand.
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
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kThreads = 32 * (kFirstConvWarp + kConvWarps);

// Which operands the kernel rounds itself.
enum CvtMode : int { kModeA = 0, kModeB = 1, kModeAB = 2 };

// How the converters get their operands: 0 from global memory (4 bytes at a time, A 16
// bytes at a time when its rows start on 16 bytes), 1 from the TMA staging ring.
enum SrcMode : int { kSrcGlobal = 0, kSrcTma = 1 };

template <int BN, int STAGES, int STG, int MODE>
struct CvtLayout {
    static constexpr bool kCvtA = MODE != kModeB;           // A rounded here
    static constexpr bool kCvtB = MODE != kModeA;           // B rounded here
    static constexpr uint32_t kABytes = kBM * kBK * 2;      // f16 A slot of the MMA ring
    static constexpr uint32_t kBBytes = BN * kBK * 2;       // f16 B slot
    // f32 part of a staging slot: 128 rows of A x 64 k, then 64 k x TILE_N columns of B
    static constexpr uint32_t kStgA = kCvtA ? kBM * kBK * 4 : 0;
    static constexpr uint32_t kStgB = kCvtB ? BN * kBK * 4 : 0;
    static constexpr uint32_t kStgBytes = kStgA + kStgB;
    // 16-byte chunks a converter thread writes per k block into each converted slot
    static constexpr int kChunksA = kABytes / 16 / kConvThreads;
    static constexpr int kChunksB = kBBytes / 16 / kConvThreads;
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
    static_assert(kChunksA == 8 && (!kCvtB || (kChunksB * 16 * kConvThreads == kBBytes && kChunksB <= 8)),
                  "the converters cover the slots, at most 8 chunks a thread");
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

// A (M x K) and B (K x N): the f32 operands, row-major.  tm_a32 / tm_b32: the tensor maps
// of the converted ones for the staging ring (src_mode kSrcTma); a_vec: A's rows start on 16
// bytes (loads from global memory).  tm_f16: the other operand's K-major f16 tensor map (B:
// N x Kp for CONVERT_A, A: M x Kp for CONVERT_B; unused when both are converted).  With
// ksplit > 1 the items are (tile, k slice) pairs and each writes its slice's partial products
// (alpha = 1, beta = 0) to plane `slice` of `partial` (M x N f32 each).
template <int BN, int STAGES, int STG, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
gemm_f16cvt_kernel(const float* __restrict__ A, const float* __restrict__ B,
                   const __grid_constant__ CUtensorMap tm_a32, const __grid_constant__ CUtensorMap tm_b32,
                   const __grid_constant__ CUtensorMap tm_f16, float* __restrict__ C, int M, int N, int K,
                   int num_kb, float alpha, float beta, int tiles_m, int tiles_n, unsigned int* status,
                   int src_mode, int a_vec, int ksplit, int kb_per_slice, float* __restrict__ partial) {
    using L = CvtLayout<BN, STAGES, STG, MODE>;
    constexpr bool kCvtA = L::kCvtA, kCvtB = L::kCvtB;
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
    const bool staged = src_mode == kSrcTma;
    const int num_items = tiles_m * tiles_n * ksplit;
    // item w: slice w % ksplit of tile t = w / ksplit, tile row t % tiles_m, tile column
    // t / tiles_m (the CTAs at work at one time share the column's tile of B); k blocks
    // kb0 .. kb0 + nkb - 1
    struct Item { int pm, pn, slice, kb0, nkb; };
    auto decode = [&](int w) {
        Item it;
        const int t = w / ksplit;
        it.slice = w - t * ksplit;
        it.pn = t / tiles_m;
        it.pm = t - it.pn * tiles_m;
        it.kb0 = it.slice * kb_per_slice;
        it.nkb = min(kb_per_slice, num_kb - it.kb0);
        return it;
    };

    if (warp == kProducerWarp && lane == 0) {
        if (MODE != kModeAB) tma_prefetch_desc(&tm_f16);
        if (staged && kCvtA) tma_prefetch_desc(&tm_a32);
        if (staged && kCvtB) tma_prefetch_desc(&tm_b32);
        for (int s = 0; s < STAGES; ++s) {
            // the converters, and the producer's expect_tx for the other operand's f16 tile
            mbar_init(full_bar(s), (MODE == kModeAB ? 0 : 1) + kConvWarps);
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
            bool pass_done = false;  // the rounding pass has been waited for
            (void)pass_done;         // (unused when both operands are rounded here)
            for (int w = blockIdx.x; w < num_items && ok; w += gridDim.x) {
                const Item it = decode(w);
                for (int kb = it.kb0; kb < it.kb0 + it.nkb; ++kb) {
                    if (staged) {
                        // the converted operands do not depend on the rounding pass: their
                        // first loads go out before the wait for that pass
                        if (!mbar_wait(sempty_bar(sstage), sphase ^ 1u, abort_flag, status)) { ok = false; break; }
                        PHX_DCHECK(sstage < STG && it.pm < tiles_m && it.pn < tiles_n && kb < num_kb);
                        mbar_arrive_expect_tx(sfull_bar(sstage), L::kStgBytes);
                        const uint32_t slot = sStg + sstage * L::kStgBytes;
                        if constexpr (kCvtA) tma_load_2d(slot, &tm_a32, kb * kBK, it.pm * kBM, sfull_bar(sstage));
                        if constexpr (kCvtB)
                            tma_load_2d(slot + L::kStgA, &tm_b32, it.pn * BN, kb * kBK, sfull_bar(sstage));
                        sissued_mask |= 1u << sstage;
                        sissued_phase = (sissued_phase & ~(1u << sstage)) | (sphase << sstage);
                        if (++sstage == STG) { sstage = 0; sphase ^= 1u; }
                    }
                    if constexpr (MODE != kModeAB) {
                        if (!pass_done) {
                            // the other operand comes from the rounding pass just before this
                            // kernel, which may still be running
                            asm volatile("griddepcontrol.wait;" ::: "memory");
                            pass_done = true;
                        }
                        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, status)) { ok = false; break; }
                        PHX_DCHECK(stage < STAGES);
                        if constexpr (MODE == kModeB) {
                            mbar_arrive_expect_tx(full_bar(stage), L::kABytes);
                            tma_load_2d(sA + stage * L::kABytes, &tm_f16, kb * kBK, it.pm * kBM, full_bar(stage));
                        } else {
                            mbar_arrive_expect_tx(full_bar(stage), L::kBBytes);
                            tma_load_2d(sB + stage * L::kBBytes, &tm_f16, kb * kBK, it.pn * BN, full_bar(stage));
                        }
                        issued_mask |= 1u << stage;
                        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
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
        const int ct = threadIdx.x - 32 * kFirstConvWarp;  // 0 .. 127
        // Chunk i of this thread in each converted slot: row r (a row of A, or one n of B) and
        // 16-byte chunk c (8 consecutive k).
        //   A: warp w owns rows 32w .. 32w+31; lane takes chunk lane % 8 of rows 4i + lane / 8.
        //   B: chunk id ct + 128 i: n = id % TILE_N, chunk = id / TILE_N, so the 32 lanes of a
        //      warp read 32 consecutive n of one staged k row (one 128-byte line).
        auto a_row = [&](int i) { return (ct / 32) * 32 + 4 * i + (lane >> 3); };
        auto a_chunk = [&](int) { return lane & 7; };
        auto b_row = [&](int i) { return (ct + kConvThreads * i) % BN; };
        auto b_chunk = [&](int i) { return (ct + kConvThreads * i) / BN; };
        // round chunk i (8 floats) to f16 and store it at chunk c ^ (r % 8) of row r of the slot
        auto store1 = [&](uint8_t* slot, const float (&x)[8], int r, int c) {
            uint4 h;
            h.x = half2_bits(x[0], x[1]);
            h.y = half2_bits(x[2], x[3]);
            h.z = half2_bits(x[4], x[5]);
            h.w = half2_bits(x[6], x[7]);
            PHX_DCHECK(r < 256 && c < 8);
            *reinterpret_cast<uint4*>(slot + r * 128 + ((c ^ (r & 7)) << 4)) = h;
        };
        uint32_t stage = 0, phase = 0, sstage = 0, sphase = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < num_items && ok; w += gridDim.x) {
            const Item it = decode(w);
            for (int kb = it.kb0; kb < it.kb0 + it.nkb; ++kb) {
                float v[8][8];
                const float* stg = nullptr;
                if (staged) {
                    // the f32 boxes (zeros past the edges) of the staging slot
                    if (!__all_sync(0xffffffffu, mbar_wait(sfull_bar(sstage), sphase, abort_flag, status))) {
                        ok = false;
                        break;
                    }
                    stg = reinterpret_cast<const float*>(base_ptr + L::kStg + sstage * L::kStgBytes);
                }
                // the staging slot goes back to the producer once this warp has read it all
                auto release = [&] {
                    if (!staged) return;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sempty_bar(sstage));
                    if (++sstage == STG) { sstage = 0; sphase ^= 1u; }
                };
                bool slot_free = false;  // the MMA ring's slot has been waited for
                auto wait_slot = [&] {
                    if (slot_free) return true;
                    slot_free = __all_sync(0xffffffffu, mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, status));
                    return slot_free;
                };
                if constexpr (kCvtA) {
#pragma unroll
                    for (int i = 0; i < L::kChunksA; ++i) {
                        const int r = a_row(i), c = a_chunk(i);
                        if (staged) {
                            const float4 x = *reinterpret_cast<const float4*>(stg + r * kBK + c * 8);
                            const float4 y = *reinterpret_cast<const float4*>(stg + r * kBK + c * 8 + 4);
                            v[i][0] = x.x; v[i][1] = x.y; v[i][2] = x.z; v[i][3] = x.w;
                            v[i][4] = y.x; v[i][5] = y.y; v[i][6] = y.z; v[i][7] = y.w;
                        } else {
                            const int k = kb * kBK + c * 8;
                            const int64_t grow = static_cast<int64_t>(it.pm) * kBM + r;
                            const float* p = A + grow * K + k;
                            if (grow < M && a_vec && k + 8 <= K) {
                                const float4 x = ld_stream4(p);
                                const float4 y = ld_stream4(p + 4);
                                v[i][0] = x.x; v[i][1] = x.y; v[i][2] = x.z; v[i][3] = x.w;
                                v[i][4] = y.x; v[i][5] = y.y; v[i][6] = y.z; v[i][7] = y.w;
                            } else {
#pragma unroll
                                for (int q = 0; q < 8; ++q) v[i][q] = (grow < M && k + q < K) ? __ldg(p + q) : 0.f;
                            }
                        }
                    }
                    if (!kCvtB) release();
                    if (!wait_slot()) { ok = false; break; }
#pragma unroll
                    for (int i = 0; i < L::kChunksA; ++i)
                        store1(base_ptr + L::kA + stage * L::kABytes, v[i], a_row(i), a_chunk(i));
                }
                if constexpr (kCvtB) {
#pragma unroll
                    for (int i = 0; i < L::kChunksB; ++i) {
                        const int r = b_row(i), c = b_chunk(i);
                        if (staged) {
                            // column r of the 64 x TILE_N box, k rows 8c .. 8c+7
                            const float* sb = stg + L::kStgA / 4;
#pragma unroll
                            for (int q = 0; q < 8; ++q) v[i][q] = sb[(8 * c + q) * BN + r];
                        } else {
                            const int k = kb * kBK + c * 8;
                            const int64_t n = static_cast<int64_t>(it.pn) * BN + r;
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                v[i][q] = (n < N && k + q < K) ? __ldg(B + static_cast<int64_t>(k + q) * N + n) : 0.f;
                        }
                    }
                    release();
                    if (!wait_slot()) { ok = false; break; }
#pragma unroll
                    for (int i = 0; i < L::kChunksB; ++i)
                        store1(base_ptr + L::kB + stage * L::kBBytes, v[i], b_row(i), b_chunk(i));
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
                const Item it = decode(w);
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                PHX_DCHECK(acc * BN + BN <= L::kTmemCols && it.nkb > 0);
                for (int kb = 0; kb < it.nkb; ++kb) {
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
        const bool vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15u) == 0) &&
                         (partial == nullptr || (reinterpret_cast<uintptr_t>(partial) & 15u) == 0);
        uint32_t acc = 0, acc_phase = 0;
        for (int w = blockIdx.x; w < num_items; w += gridDim.x) {
            const Item it = decode(w);
            // a k slice writes its plane of partial products; a whole tile writes C
            float* Cout = ksplit > 1 ? partial + static_cast<int64_t>(it.slice) * M * N : C;
            const float a_out = ksplit > 1 ? 1.f : alpha;
            const float b_out = ksplit > 1 ? 0.f : beta;
            const bool read_c = b_out != 0.f;
            // warp-uniform outcome: tcgen05.ld below is .sync.aligned
            if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), acc_phase, abort_flag, status))) break;
            tc_fence_after();
            const int row0 = it.pm * kBM + warp * 32;
            const uint32_t t_base = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + acc * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                const int col0 = it.pn * BN + c * 32;
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
                                cv[q] = *reinterpret_cast<const float4*>(Cout + static_cast<int64_t>(row) * N + col);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int rr = q * 4 + lane / 8;
                        const int row = row0 + rr;
                        if (row < M && col < N) {
                            const float4 a = *reinterpret_cast<const float4*>(epi + rr * L::kEpiStride + cc);
                            float4 o = make_float4(a_out * a.x, a_out * a.y, a_out * a.z, a_out * a.w);
                            if (read_c) {
                                o.x = fmaf(b_out, cv[q].x, o.x);
                                o.y = fmaf(b_out, cv[q].y, o.y);
                                o.z = fmaf(b_out, cv[q].z, o.z);
                                o.w = fmaf(b_out, cv[q].w, o.w);
                            }
                            PHX_DCHECK(col + 3 < N);
                            *reinterpret_cast<float4*>(Cout + static_cast<int64_t>(row) * N + col) = o;
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
                            cs[rr] = (row < M && col < N) ? Cout[static_cast<int64_t>(row) * N + col] : 0.f;
                        }
                    }
#pragma unroll
                    for (int rr = 0; rr < 32; ++rr) {
                        const int row = row0 + rr;
                        if (row < M && col < N) {
                            float o = a_out * epi[rr * L::kEpiStride + lane];
                            if (read_c) o = fmaf(b_out, cs[rr], o);
                            Cout[static_cast<int64_t>(row) * N + col] = o;
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

using CvtKernelFn = void (*)(const float*, const float*, CUtensorMap, CUtensorMap, CUtensorMap, float*, int, int, int,
                             int, float, float, int, int, unsigned int*, int, int, int, int, float*);

struct CvtEntry {
    F16Config cfg;
    int mode;
    CvtKernelFn fn;
    uint32_t smem;
};

template <int BN, int STAGES, int STG, int MODE>
CvtEntry make_cvt_entry() {
    return CvtEntry{F16Config{kBM, BN, kBK, STAGES, 1, MODE != kModeB ? 1 : 0, MODE != kModeA ? 1 : 0}, MODE,
                    &gemm_f16cvt_kernel<BN, STAGES, STG, MODE>, CvtLayout<BN, STAGES, STG, MODE>::kDynSmem};
}

// CONVERT_A: at each width 96 KB of MMA ring (4 slots of 24 KB, 3 of 32 KB, 2 of 48 KB) and
// 96 KB of f32 staging (3 k blocks of A in flight per SM).  CONVERT_B: the same at TILE_N = 64
// (3 staged k blocks of B are 48 KB) and 128 (96 KB).  Both: 2 staging slots of A and B
// (96 KB at TILE_N = 64, 128 KB at 128) and 3 or 2 MMA slots.
const CvtEntry kCvtEntries[] = {
    make_cvt_entry<64, 4, 3, kModeA>(),
    make_cvt_entry<128, 3, 3, kModeA>(),
    make_cvt_entry<256, 2, 3, kModeA>(),
    make_cvt_entry<64, 4, 3, kModeB>(),
    make_cvt_entry<128, 3, 3, kModeB>(),
    make_cvt_entry<64, 3, 2, kModeAB>(),
    make_cvt_entry<128, 2, 2, kModeAB>(),
};
constexpr int kNumCvt = sizeof(kCvtEntries) / sizeof(kCvtEntries[0]);

constexpr int kCvtMaxSplit = 8;
constexpr int kCvtMinKbPerSlice = 8;

// K blocks per slice: enough slices to give every SM an item when the tiles alone do not (at
// most 8, at least 8 k blocks each); num_kb when not split.
int cvt_kb_per_slice(const CvtEntry& e, int64_t M, int64_t N, int64_t K, int num_sms) {
    const int64_t num_kb = (K + kBK - 1) / kBK;
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + e.cfg.tile_n - 1) / e.cfg.tile_n);
    if (tiles <= 0 || 2 * tiles > num_sms) return static_cast<int>(num_kb);
    int64_t split = num_sms / tiles;
    if (split > kCvtMaxSplit) split = kCvtMaxSplit;
    if (split > num_kb / kCvtMinKbPerSlice) split = num_kb / kCvtMinKbPerSlice;
    if (split < 2) return static_cast<int>(num_kb);
    return static_cast<int>((num_kb + split - 1) / split);
}

}  // namespace

int f16cvt_num_configs() { return kNumCvt; }

const F16Config& f16cvt_config(int index) { return kCvtEntries[index].cfg; }

int64_t debug_take_f16cvt() { return debug_take_local(); }

size_t f16cvt_split_bytes(int index, int64_t M, int64_t N, int64_t K, int num_sms) {
    if (index < 0 || index >= kNumCvt) return 0;
    const int64_t num_kb = (K + kBK - 1) / kBK;
    const int kb = cvt_kb_per_slice(kCvtEntries[index], M, N, K, num_sms);
    if (kb >= num_kb) return 0;
    return static_cast<size_t>((num_kb + kb - 1) / kb) * static_cast<size_t>(M * N) * 4;
}

cudaError_t f16cvt_gemm_launch(int index, int64_t M, int64_t N, int64_t K, float alpha, float beta, float* C,
                               const float* A, const float* B, const __half* other, int64_t ld_other,
                               void* split_ws, unsigned int* status, int num_sms, cudaStream_t stream) {
    if (index < 0 || index >= kNumCvt || M <= 0 || N <= 0 || K <= 0 || num_sms <= 0) return cudaErrorInvalidValue;
    const CvtEntry& e = kCvtEntries[index];
    const int bn = e.cfg.tile_n;
    const int64_t Kp = (K + 7) / 8 * 8;
    if (M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF) return cudaErrorInvalidValue;
    // the f16 operand from the rounding pass: B (N x Kp) for CONVERT_A, A (M x Kp) for CONVERT_B
    CUtensorMap map_f16;
    std::memset(&map_f16, 0, sizeof map_f16);
    if (e.mode != kModeAB &&
        !f16_operand_map(&map_f16, other, e.mode == kModeB ? M : N, Kp, e.mode == kModeB ? kBM : bn, ld_other))
        return cudaErrorInvalidValue;
    const int64_t tiles_m = (M + kBM - 1) / kBM;
    const int64_t tiles_n = (N + bn - 1) / bn;
    const int64_t num_kb64 = (K + kBK - 1) / kBK;
    int kb_per = cvt_kb_per_slice(e, M, N, K, num_sms);
    if (split_ws == nullptr) kb_per = static_cast<int>(num_kb64);
    const int64_t ksplit = (num_kb64 + kb_per - 1) / kb_per;
    const int64_t items = tiles_m * tiles_n * ksplit;
    if (items > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const int grid = static_cast<int>(items < num_sms ? items : num_sms);
    // the converted operands through the TMA staging ring when their rows can be tensor maps
    // (16-byte aligned rows and bases, all of them); else the converters load them themselves
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const bool cvt_a = e.mode != kModeB, cvt_b = e.mode != kModeA;
    const bool a_al = K % 4 == 0 && al16(A), b_al = N % 4 == 0 && al16(B);
    CUtensorMap map_a32, map_b32;
    std::memset(&map_a32, 0, sizeof map_a32);
    std::memset(&map_b32, 0, sizeof map_b32);
    bool tma = (!cvt_a || a_al) && (!cvt_b || b_al);
    if (tma && cvt_a) tma = f32_rows_map(&map_a32, A, M, K, kBK, kBM);
    if (tma && cvt_b) tma = f32_rows_map(&map_b32, B, K, N, bn, kBK);
    const int src_mode = tma ? kSrcTma : kSrcGlobal;
    const int a_vec = a_al ? 1 : 0;
    float* partial = ksplit > 1 ? static_cast<float*>(split_ws) : nullptr;
    cudaError_t err = set_func_attr_once(reinterpret_cast<const void*>(e.fn),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(e.smem));
    if (err != cudaSuccess) return err;
    // with one operand from the rounding pass, a programmatic dependent of that pass (see the
    // top of this file)
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(grid));
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = e.smem;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = e.mode == kModeAB ? 0 : 1;
    const int m32 = static_cast<int>(M), n32 = static_cast<int>(N), k32 = static_cast<int>(K);
    const int tm32 = static_cast<int>(tiles_m), tn32 = static_cast<int>(tiles_n), nkb = static_cast<int>(num_kb64);
    const int ks32 = static_cast<int>(ksplit);
    err = cudaLaunchKernelEx(&lc, e.fn, A, B, map_a32, map_b32, map_f16, C, m32, n32, k32, nkb, alpha, beta, tm32,
                             tn32, status, src_mode, a_vec, ks32, kb_per, partial);
    if (err != cudaSuccess && lc.numAttrs > 0) {
        // a stream that does not take programmatic launches: launch normally
        cudaGetLastError();
        lc.numAttrs = 0;
        err = cudaLaunchKernelEx(&lc, e.fn, A, B, map_a32, map_b32, map_f16, C, m32, n32, k32, nkb, alpha, beta,
                                 tm32, tn32, status, src_mode, a_vec, ks32, kb_per, partial);
    }
    err = launched(err);
    if (err != cudaSuccess || ksplit == 1) return err;
    return splitk_reduce_launch(partial, ks32, M, N, alpha, beta, C, num_sms, stream);
}

}  // namespace phx
