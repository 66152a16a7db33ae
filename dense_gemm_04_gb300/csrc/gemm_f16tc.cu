// gemm_f16tc.cu -- f16 tensor cores with f32 accumulation on sm_103a (tcgen05 + TMA).
//
// C <- alpha * A @ B + beta * C, where every element of the f32 operands A and B is first
// rounded to the nearest f16 (ties to even) and the f16 x f16 products are summed in f32
// ("gemm on tensor cores", phobos-lang.dev/docs/examples/gemm-fp16tc-fp32acc/, section
// "What changes"; the tile structure is the same as "gemm, f32", sections "One output tile
// per CTA", "The k loop", "The epilogue").
//
// Two passes:
//   1. Cast (HBM-bound, one launch): A (M x K f32) -> Ah (M x Kp f16, row-major) and B
//      (K x N f32) -> Bt (N x Kp f16, B transposed) with cvt.rn (round to nearest even);
//      operands given transposed are read in their stored order; Kp = K rounded up
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
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "debug_checks.cuh"
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

// One launch casts both operands.  Each operand is a job: its f32 values, as rows x K,
// become rows x Kp halves (K-major), rounded to nearest even.  A job whose source is
// stored row by row (trans = 0) is cast 8 halves (16 bytes) per thread, grid-stride; a
// job whose source is stored transposed (trans = 1: K x rows) goes through 64 x 64 tiles
// of shared memory, one tile per block, with the tile's columns XOR-swizzled per band of
// 8 rows so that both the row-wise 16-byte stores of the loaded tile and the column-wise
// reads that build the output rows hit 32 different banks.  A of a plain GEMM is a row
// job and B a transposed one (B is K x N, its K-major form N x K).
constexpr int kTT = 64;

struct CastJob {
    const void* src;  // f32, or f16 when src_f16
    __half* dst;
    int64_t rows;     // rows of the K-major result
    int trans;        // source stored K x rows
    int src_f16;      // the source is already f16: the job only copies (and transposes)
    int vec;          // 16-byte source loads allowed
    int blocks;       // blocks of the launch this job takes (0: no job)
    int tiles_r;      // trans: 64-row tiles along rows
};

__device__ __forceinline__ int tt_swizzle(int k) { return ((k >> 3) & 7) << 2; }

// Four consecutive f16 values (8 bytes, 8-byte aligned) as floats, and back, rounded to
// nearest even.
__device__ __forceinline__ float4 load4_h(const __half* p) {
    const uint2 raw = *reinterpret_cast<const uint2*>(p);
    const __half2 lo = *reinterpret_cast<const __half2*>(&raw.x);
    const __half2 hi = *reinterpret_cast<const __half2*>(&raw.y);
    return make_float4(__low2float(lo), __high2float(lo), __low2float(hi), __high2float(hi));
}

__device__ __forceinline__ void store4_h(__half* p, float4 v) {
    const __half2 lo = __floats2half2_rn(v.x, v.y);
    const __half2 hi = __floats2half2_rn(v.z, v.w);
    uint2 raw;
    raw.x = *reinterpret_cast<const uint32_t*>(&lo);
    raw.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = raw;
}

__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
    uint4 out;
    __half2 h;
    h = __floats2half2_rn(v[0], v[1]); out.x = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2half2_rn(v[2], v[3]); out.y = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2half2_rn(v[4], v[5]); out.z = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2half2_rn(v[6], v[7]); out.w = *reinterpret_cast<uint32_t*>(&h);
    return out;
}

__global__ void __launch_bounds__(256) cast_kernel(CastJob j0, CastJob j1, int64_t K, int64_t Kp) {
    // let the GEMM that follows start its prologue while the cast finishes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x;
    int b = static_cast<int>(blockIdx.x);
    const CastJob j = b < j0.blocks ? j0 : j1;
    if (b >= j0.blocks) b -= j0.blocks;
    if (!j.trans) {
        const int64_t chunks = Kp / 8;
        const int64_t total = j.rows * chunks;
        const int64_t stride = static_cast<int64_t>(j.blocks) * 256;
        for (int64_t idx = static_cast<int64_t>(b) * 256 + tid; idx < total; idx += stride) {
            const int64_t r = idx / chunks;
            const int64_t c = (idx - r * chunks) * 8;
            if (j.src_f16) {
                const __half* hs = static_cast<const __half*>(j.src) + r * K + c;
                uint4 raw;
                if (j.vec && c + 8 <= K) {
                    raw = __ldcs(reinterpret_cast<const uint4*>(hs));
                } else {
                    __half h[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) h[q] = (c + q < K) ? hs[q] : __float2half_rn(0.f);
                    raw = *reinterpret_cast<const uint4*>(h);
                }
                *reinterpret_cast<uint4*>(j.dst + r * Kp + c) = raw;
                continue;
            }
            const float* src = static_cast<const float*>(j.src) + r * K + c;
            PHX_DCHECK(r < j.rows && c + 7 < Kp);
            float v[8];
            if (j.vec && c + 8 <= K) {
                const float4 x = __ldcs(reinterpret_cast<const float4*>(src));
                const float4 y = __ldcs(reinterpret_cast<const float4*>(src + 4));
                v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
                v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] = (c + q < K) ? src[q] : 0.f;
            }
            *reinterpret_cast<uint4*>(j.dst + r * Kp + c) = pack8(v);
        }
        return;
    }
    __shared__ __align__(16) float tile[kTT][kTT];  // [k][r ^ swizzle(k)]
    const int64_t R = j.rows;
    const int64_t r0 = static_cast<int64_t>(b % j.tiles_r) * kTT;
    const int64_t k0 = static_cast<int64_t>(b / j.tiles_r) * kTT;
    if (j.src_f16) {
        // f16 source: 8 halves (16 bytes) per load, 8 lanes per 128-byte row segment; the
        // values widen to f32 exactly and pack8 below rounds them back unchanged
#pragma unroll
        for (int i = 0; i < kTT * kTT / 8 / 256; ++i) {
            const int e = tid + i * 256;
            const int k = e / (kTT / 8);
            const int r8 = (e % (kTT / 8)) * 8;
            const int64_t gk = k0 + k;
            const int64_t gr = r0 + r8;
            const bool rk = gk < K;
            const __half* hs = static_cast<const __half*>(j.src) + gk * R + gr;
            float v[8];
            if (j.vec && rk && gr + 7 < R) {
                const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(hs));
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __half2 h2 = *reinterpret_cast<const __half2*>(&w[q]);
                    v[2 * q] = __low2float(h2);
                    v[2 * q + 1] = __high2float(h2);
                }
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] = (rk && gr + q < R) ? __half2float(hs[q]) : 0.f;
            }
            *reinterpret_cast<float4*>(&tile[k][r8 ^ tt_swizzle(k)]) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4*>(&tile[k][(r8 + 4) ^ tt_swizzle(k)]) = make_float4(v[4], v[5], v[6], v[7]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < kTT * kTT / 4 / 256; ++i) {
            const int e = tid + i * 256;
            const int k = e / (kTT / 4);
            const int r4 = (e % (kTT / 4)) * 4;
            const int64_t gk = k0 + k;
            const int64_t gr = r0 + r4;
            const bool rk = gk < K;
            const float* fs = static_cast<const float*>(j.src) + gk * R + gr;
            float4 v;
            if (j.vec && rk && gr + 3 < R) {
                v = __ldcs(reinterpret_cast<const float4*>(fs));
            } else {
                v.x = (rk && gr + 0 < R) ? fs[0] : 0.f;
                v.y = (rk && gr + 1 < R) ? fs[1] : 0.f;
                v.z = (rk && gr + 2 < R) ? fs[2] : 0.f;
                v.w = (rk && gr + 3 < R) ? fs[3] : 0.f;
            }
            *reinterpret_cast<float4*>(&tile[k][r4 ^ tt_swizzle(k)]) = v;
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kTT * (kTT / 8) / 256; ++i) {
        const int e = tid + i * 256;
        const int r = e / (kTT / 8);
        const int kc = (e % (kTT / 8)) * 8;
        const int64_t gr = r0 + r;
        const int64_t gk = k0 + kc;
        if (gr < R && gk < Kp) {
            PHX_DCHECK(gk + 7 < Kp && r < kTT && kc + 7 < kTT);
            const int col = r ^ tt_swizzle(kc);  // the same for the 8 rows kc .. kc+7
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = tile[kc + q][col];
            *reinterpret_cast<uint4*>(j.dst + gr * Kp + gk) = pack8(v);
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

// PAIR selects how CTAs cooperate:
//   0  one CTA per tile;
//   2  clusters of two CTAs run the 2-SM MMA (tcgen05.mma.cta_group::2, M = 256): each CTA
//      stages its own 128 rows of A and its own half of the B tile, and the even CTA's MMA
//      thread multiplies the pair's 256 x TILE_N tile, each CTA receiving its 128 rows of
//      the accumulator.  A CTA stages 2/3 of the bytes per k block that PAIR 0 does for the
//      same MMA work, so the same shared memory holds more k blocks in flight.
template <int BN, int STAGES, int PAIR>
struct TcLayout {
    static constexpr int kBRows = PAIR == 2 ? BN / 2 : BN;   // B rows a CTA stages per k block
    static constexpr uint32_t kABytes = kBM * kBK * 2;
    static constexpr uint32_t kBBytes = kBRows * kBK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kTmemCols = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64
                                          : (2 * BN <= 128) ? 128 : (2 * BN <= 256) ? 256 : 512;
    // offsets from the 1024-byte aligned base
    static constexpr uint32_t kA = 0;
    static constexpr uint32_t kB = STAGES * kABytes;
    // per epilogue warp: a 32 x 32 f32 chunk with rows padded to 36 floats (staging), or,
    // for the TMA epilogue, two 32 x 32 chunks in the 128-byte swizzled layout of a TMA box
    // (1024-byte aligned)
    static constexpr uint32_t kEpiStride = 36;
    static constexpr uint32_t kEpiWarpFloats = 2 * 32 * 32;
    static_assert(32 * kEpiStride <= kEpiWarpFloats, "the staging chunk fits the warp's region");
    static constexpr uint32_t kEpi = STAGES * kStageBytes;
    static constexpr uint32_t kEpiBytes = kEpiWarps * kEpiWarpFloats * 4;
    static constexpr uint32_t kBars = kEpi + kEpiBytes;               // 8-byte aligned
    // full, empty, tfull, tempty, done, and two c_old barriers per epilogue warp
    static constexpr uint32_t kNumBars = 2 * STAGES + 4 + 1 + 2 * kEpiWarps;
    static constexpr uint32_t kTmemSlot = kBars + 8 * kNumBars;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kEnd = kAbort + 4;
    static constexpr uint32_t kDynSmem = kEnd + 1024;                 // + alignment slack
    static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256, "tcgen05 needs N % 16 == 0, N <= 256");
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "swizzle atoms stay 1024-aligned");
};

template <int BN, int STAGES, int PAIR, bool OUT_H, bool EPI_TMA>
__global__ void __launch_bounds__(kThreadsTc, 1)
gemm_f16tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmB_half, const __grid_constant__ CUtensorMap tmB_quarter,
                  float* __restrict__ C, int M, int N, int num_kb, float alpha, float beta, int tiles_m,
                  int tiles_n, unsigned int* status, int full_tiles, int tail_split, int ksplit,
                  int kb_per_slice, float* __restrict__ partial, __half* __restrict__ Ch,
                  const __grid_constant__ CUtensorMap tmC, int epi_tma) {
    using L = TcLayout<BN, STAGES, PAIR>;
    constexpr bool kPair = PAIR != 0;
    constexpr bool kTwoSm = PAIR == 2;
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
    auto cold_bar = [&](int w, int b) { return bars + 8u * (2 * STAGES + 5 + 2 * w + b); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + L::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + L::kAbort);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;  // position in the CTA pair
    const bool leader = rank == 0;
    const int first_item = kPair ? static_cast<int>(blockIdx.x) / 2 : static_cast<int>(blockIdx.x);
    const int item_stride = kPair ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);
    // with a pair, a "tile" is two vertically adjacent tiles; CTA `rank` takes one of them
    const int tiles_rows = kPair ? (tiles_m + 1) / 2 : tiles_m;
    // Work items, dealt round-robin to the persistent CTAs (or pairs): every whole tile of
    // the full rounds, then each remaining (tail) tile as `tail_split` items of width
    // TILE_N / tail_split, so that a last round with few tiles keeps more SMs busy.  A
    // narrower item runs the same MMA sequence over K for each of its output elements.
    // With ksplit > 1 (a grid too small for the GPU) every tile is instead `ksplit` items,
    // one per k slice of kb_per_slice k blocks, each writing its partial product (alpha = 1,
    // beta = 0) to its own M x N plane of `partial` for a separate reduction.
    const int num_tiles = tiles_rows * tiles_n;
    const int num_items = ksplit > 1 ? num_tiles * ksplit : full_tiles + (num_tiles - full_tiles) * tail_split;
    constexpr int BN_HALF = BN / 2;
    struct Item { int pm, pn, n0, width, kb0, nkb, slice; };
    auto decode = [&](int w) {
        Item it;
        int tile = w;
        it.n0 = 0;
        it.width = BN;
        it.kb0 = 0;
        it.nkb = num_kb;
        it.slice = -1;
        if (ksplit > 1) {
            tile = w / ksplit;
            it.slice = w - tile * ksplit;
            it.kb0 = it.slice * kb_per_slice;
            it.nkb = min(kb_per_slice, num_kb - it.kb0);
        } else if (w >= full_tiles && tail_split > 1) {
            const int q = w - full_tiles;
            tile = full_tiles + q / tail_split;
            it.width = BN_HALF;
            it.n0 = (q % tail_split) * BN_HALF;
        }
        tc_tile_coords(tile, tiles_rows, tiles_n, it.pm, it.pn);
        if (kPair) it.pm = 2 * it.pm + static_cast<int>(rank);
        it.n0 += it.pn * BN;
        return it;
    };

    auto row0_of = [&](const Item& it) { return it.pm * kBM + warp * 32; };

    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmB_half);
        tma_prefetch_desc(&tmB_quarter);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), kTwoSm ? 2 * kEpiWarps : kEpiWarps);
        }
        mbar_init(done_bar, 1);
        for (int w = 0; w < kEpiWarps; ++w) {
            mbar_init(cold_bar(w, 0), 1);
            mbar_init(cold_bar(w, 1), 1);
        }
        if (epi_tma) tma_prefetch_desc(&tmC);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (kTwoSm) cluster_sync();  // both CTAs present before the pair allocates tensor memory
    if (warp == 0) {
        if (kTwoSm)
            tmem_alloc_2sm(smem_u32(tmem_slot), L::kTmemCols);
        else
            tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    }
    tc_fence_before();
    __syncthreads();
    if (kPair) cluster_sync();  // both CTAs' barriers exist before the other signals them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            // The operands come from the cast kernel just before this one, which may still be
            // running (programmatic dependent launch): wait for its writes before loading.
            asm volatile("griddepcontrol.wait;" ::: "memory");
            // issued[s]: bit 0 = a load was ever issued into slot s, bit 1 = its phase parity
            uint32_t issued_mask = 0, issued_phase = 0;
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int w = first_item; w < num_items && ok; w += item_stride) {
                const Item it = decode(w);
                const bool full = it.width == BN;
                for (int kb = it.kb0; kb < it.kb0 + it.nkb; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, status)) { ok = false; break; }
                    const uint32_t a_dst = sA + stage * L::kABytes;
                    const uint32_t b_dst = sB + stage * L::kBBytes;
                    PHX_DCHECK(stage < STAGES && kb < num_kb && it.pm * kBM < (kTwoSm ? 2 : 1) * tiles_rows * kBM &&
                               it.n0 < tiles_n * BN);
                    if constexpr (kTwoSm) {
                        // each CTA: its 128 rows of A and its share of B, counted on the even
                        // CTA's barrier, which expects the pair's bytes
                        const uint32_t cta_bytes = L::kABytes + (full ? L::kBBytes : L::kBBytes / 2);
                        const uint32_t lbar = map_to_rank(full_bar(stage), 0);
                        if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * cta_bytes);
                        tma_load_2d_2sm(a_dst, &tmA, kb * kBK, it.pm * kBM, lbar);
                        if (full)
                            tma_load_2d_2sm(b_dst, &tmB_half, kb * kBK, it.n0 + static_cast<int>(rank) * BN_HALF, lbar);
                        else
                            tma_load_2d_2sm(b_dst, &tmB_quarter, kb * kBK, it.n0 + static_cast<int>(rank) * (BN / 4), lbar);
                    } else {
                        mbar_arrive_expect_tx(full_bar(stage), L::kABytes + (full ? L::kBBytes : L::kBBytes / 2));
                        tma_load_2d(a_dst, &tmA, kb * kBK, it.pm * kBM, full_bar(stage));
                        tma_load_2d(b_dst, full ? &tmB : &tmB_half, kb * kBK, it.n0, full_bar(stage));
                    }
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok && (!kTwoSm || leader)) {
                // Aborted: let every load issued into this CTA land before the CTA exits (in
                // a 2-SM pair the even CTA's barriers count both CTAs' loads).
                for (int s = 0; s < STAGES; ++s)
                    if (issued_mask & (1u << s)) mbar_wait_drain(full_bar(s), (issued_phase >> s) & 1u);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0 && (!kTwoSm || leader)) {
            constexpr int kMmaM = kTwoSm ? 2 * kBM : kBM;
            constexpr uint32_t idesc_full = idesc_f16_f32acc(kMmaM, BN);
            constexpr uint32_t idesc_half = idesc_f16_f32acc(kMmaM, BN_HALF);
            uint32_t stage = 0, phase = 0;
            uint32_t acc = 0, acc_phase = 0;
            bool ok = true;
            for (int w = first_item; w < num_items && ok; w += item_stride) {
                const Item it = decode(w);
                const uint32_t idesc = it.width == BN ? idesc_full : idesc_half;
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
                        const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
                        if constexpr (kTwoSm)
                            mma_f16_ss_2sm(d_tmem, ad, bd, idesc, accum);
                        else
                            mma_f16_ss(d_tmem, ad, bd, idesc, accum);
                    }
                    // the slot is free again (in both CTAs of a pair)
                    if constexpr (kTwoSm)
                        mma_commit_2sm_multicast(empty_bar(stage), 0x3);
                    else
                        mma_commit(empty_bar(stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if constexpr (kTwoSm)
                    mma_commit_2sm_multicast(tfull_bar(acc), 0x3);
                else
                    mma_commit(tfull_bar(acc));
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            // Every MMA this thread issued has completed once done_bar fires.
            if constexpr (kTwoSm)
                mma_commit_2sm(done_bar);
            else
                mma_commit(done_bar);
            mbar_wait_drain(done_bar, 0);
        }
    } else if (warp < kEpiWarps) {
        float* epi = reinterpret_cast<float*>(base_ptr + L::kEpi) + warp * L::kEpiWarpFloats;
        uint32_t acc = 0, acc_phase = 0;
        const bool vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15u) == 0) &&
                         (partial == nullptr || (reinterpret_cast<uintptr_t>(partial) & 15u) == 0);
        // an f16 result (Ch) moves 4 halves = 8 bytes per lane on the vector path
        const bool vec_h = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(Ch) & 7u) == 0);
        // The TMA epilogue (whole tiles; an f32 C with N % 4 == 0 or an f16 C with N % 8 == 0,
        // 16-byte aligned): each 32 x 32 chunk's c_old arrives by TMA in one of the warp's two
        // buffers (the next chunk's while this one is finished), lane = row finishes the row in
        // place from the accumulator, and the chunk leaves by TMA store.  An f32 chunk is a
        // 128-byte swizzled box of 4 KB; an f16 chunk an unswizzled box of 2 KB (64-byte rows).
        const bool tma_c = EPI_TMA && epi_tma != 0 && ksplit == 1;
        constexpr uint32_t kChunkBytes = OUT_H ? 32 * 32 * 2 : 32 * 32 * 4;
        const bool load_c = tma_c && beta != 0.f;
        const uint32_t ebuf = smem_u32(epi);
        auto swz = [](int r, int u) { return r * 32 + ((u ^ (r & 7)) << 2); };
        uint32_t cph = 0;          // phase bit of each buffer's c_old barrier
        uint32_t cpend = 0;        // buffers with a c_old load in flight
        // a chunk with no element inside C is neither loaded nor stored
        auto live = [&](const Item& x, int c) { return x.pm * kBM + warp * 32 < M && x.n0 + c * 32 < N; };
        auto load_cold = [&](int w_req, int c_req, int b) {  // lane 0
            if (w_req >= num_items) return;
            const Item nx = decode(w_req);
            if (!live(nx, c_req)) return;
            mbar_arrive_expect_tx(cold_bar(warp, b), kChunkBytes);
            tma_load_2d(ebuf + b * 4096, &tmC, nx.n0 + c_req * 32, nx.pm * kBM + warp * 32, cold_bar(warp, b));
            cpend |= 1u << b;
        };
        int cc = 0;  // chunks finished by this warp, across items: buffer cc & 1
        bool prev_stored = false;  // chunk cc - 1 left by TMA store
        if (load_c && lane == 0) load_cold(first_item, 0, 0);
        for (int w = first_item; w < num_items; w += item_stride) {
            const Item it = decode(w);
            // a k slice writes its plane of partial products; a whole tile writes C
            float* Cout = it.slice >= 0 ? partial + static_cast<int64_t>(it.slice) * M * N : C;
            const float a_out = it.slice >= 0 ? 1.f : alpha;
            const float b_out = it.slice >= 0 ? 0.f : beta;
            const bool read_c = b_out != 0.f;
            // a whole tile of a half-precision result rounds alpha * acc + beta * c_old to f16
            // once (a k slice still writes f32 partial products)
            const bool out_h = OUT_H && it.slice < 0;
            // warp-uniform outcome: the tcgen05.ld below is .sync.aligned
            if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), acc_phase, abort_flag, status))) break;
            tc_fence_after();
            bool ok = true;
            const int nch = it.width / 32;
            const uint32_t t_base = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + acc * BN;
#pragma unroll 1
            for (int c = 0; tma_c && c < nch; ++c, ++cc) {
                const int b = cc & 1;
                if (lane == 0) {
                    if (load_c) {
                        // the other buffer's last store has read it: take the next chunk's c_old
                        bulk_wait_read<0>();
                        if (c + 1 < nch)
                            load_cold(w, c + 1, b ^ 1);
                        else
                            load_cold(w + item_stride, 0, b ^ 1);
                    } else if (prev_stored) {
                        bulk_wait_read<1>();  // this buffer's store (two chunks back) has read it
                    } else {
                        bulk_wait_read<0>();  // the last store may have come from this buffer
                    }
                }
                const bool chunk_live = live(it, c);
                __syncwarp();
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_base + c * 32, r);
                tmem_ld_wait();
                if (load_c && chunk_live) {
                    if (!__all_sync(0xffffffffu, mbar_wait(cold_bar(warp, b), (cph >> b) & 1u, abort_flag, status))) {
                        ok = false;
                        break;
                    }
                    cph ^= 1u << b;
                    if (lane == 0) cpend &= ~(1u << b);
                }
                __syncwarp();
                if (!chunk_live) {
                    prev_stored = false;
                    continue;
                }
                float* buf = epi + b * 32 * 32;
                if constexpr (OUT_H) {
                    // row `lane`: 32 halves = 4 x 16 bytes; alpha * acc + beta * c_old in f32,
                    // rounded to f16 once
                    uint4* row4 = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(buf) + lane * 64);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        float o[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) o[q] = alpha * __uint_as_float(r[u * 8 + q]);
                        if (load_c) {
                            const uint4 raw = row4[u];
                            const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const __half2 h2 = *reinterpret_cast<const __half2*>(&wv[q]);
                                o[2 * q] = fmaf(beta, __low2float(h2), o[2 * q]);
                                o[2 * q + 1] = fmaf(beta, __high2float(h2), o[2 * q + 1]);
                            }
                        }
                        row4[u] = pack8(o);
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        float4* p4 = reinterpret_cast<float4*>(buf + swz(lane, u));
                        float4 o;
                        o.x = alpha * __uint_as_float(r[u * 4 + 0]);
                        o.y = alpha * __uint_as_float(r[u * 4 + 1]);
                        o.z = alpha * __uint_as_float(r[u * 4 + 2]);
                        o.w = alpha * __uint_as_float(r[u * 4 + 3]);
                        if (load_c) {
                            const float4 co = *p4;
                            o.x = fmaf(beta, co.x, o.x);
                            o.y = fmaf(beta, co.y, o.y);
                            o.z = fmaf(beta, co.z, o.z);
                            o.w = fmaf(beta, co.w, o.w);
                        }
                        *p4 = o;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    PHX_DCHECK(it.n0 + c * 32 < N && row0_of(it) < M);
                    tma_store_2d(&tmC, ebuf + b * 4096, it.n0 + c * 32, row0_of(it));
                    bulk_commit();
                }
                prev_stored = true;
            }
            if (!ok) break;
            // Each chunk of 32 rows x 32 columns goes from TMEM (lane = row) through this
            // warp's shared-memory buffer, so that C is read and written along rows: four
            // rows of 128 bytes per float4 instruction, or one row of 128 bytes per scalar
            // instruction when N is not a multiple of 4.
            const int row0 = it.pm * kBM + warp * 32;
            const uint32_t t_addr = t_base;
#pragma unroll 1
            for (int c = 0; !tma_c && c < nch; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_addr + c * 32, r);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<float4*>(epi + lane * L::kEpiStride + q * 4) =
                        make_float4(__uint_as_float(r[q * 4 + 0]), __uint_as_float(r[q * 4 + 1]),
                                    __uint_as_float(r[q * 4 + 2]), __uint_as_float(r[q * 4 + 3]));
                __syncwarp();
                const int col0 = it.n0 + c * 32;
                // one code path for both result types: only the loads and stores of C differ
                if (out_h ? vec_h : vec) {
                    const int cc = (lane % 8) * 4;
                    const int col = col0 + cc;
                    float4 cv[8];
                    if (read_c) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const int row = row0 + q * 4 + lane / 8;
                            const int64_t off = static_cast<int64_t>(row) * N + col;
                            cv[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (row < M && col < N) cv[q] = out_h ? load4_h(Ch + off) : *reinterpret_cast<const float4*>(Cout + off);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int rr = q * 4 + lane / 8;
                        const int row = row0 + rr;
                        if (row < M && col < N) {
                            const float4 a = *reinterpret_cast<const float4*>(epi + rr * L::kEpiStride + cc);
                            float4 o;
                            o.x = a_out * a.x;
                            o.y = a_out * a.y;
                            o.z = a_out * a.z;
                            o.w = a_out * a.w;
                            if (read_c) {
                                o.x = fmaf(b_out, cv[q].x, o.x);
                                o.y = fmaf(b_out, cv[q].y, o.y);
                                o.z = fmaf(b_out, cv[q].z, o.z);
                                o.w = fmaf(b_out, cv[q].w, o.w);
                            }
                            const int64_t off = static_cast<int64_t>(row) * N + col;
                            PHX_DCHECK(col + 3 < N && c * 32 + cc + 3 < it.width);
                            if (out_h)
                                store4_h(Ch + off, o);
                            else
                                *reinterpret_cast<float4*>(Cout + off) = o;
                        }
                    }
                } else {
                    // all 32 rows' loads of C first, so they are in flight together
                    const int col = col0 + lane;
                    float cs[32];
                    if (read_c) {
#pragma unroll
                        for (int rr = 0; rr < 32; ++rr) {
                            const int row = row0 + rr;
                            const int64_t off = static_cast<int64_t>(row) * N + col;
                            cs[rr] = 0.f;
                            if (row < M && col < N) cs[rr] = out_h ? __half2float(Ch[off]) : Cout[off];
                        }
                    }
#pragma unroll
                    for (int rr = 0; rr < 32; ++rr) {
                        const int row = row0 + rr;
                        if (row < M && col < N) {
                            float o = a_out * epi[rr * L::kEpiStride + lane];
                            if (read_c) o = fmaf(b_out, cs[rr], o);
                            const int64_t off = static_cast<int64_t>(row) * N + col;
                            PHX_DCHECK(c * 32 + lane < it.width);
                            if (out_h)
                                Ch[off] = __float2half_rn(o);
                            else
                                Cout[off] = o;
                        }
                    }
                }
                __syncwarp();  // the buffer is rewritten by the next chunk
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                // the accumulator buffer may be reused (in a 2-SM pair, the even CTA's MMA
                // thread counts both CTAs' epilogue warps)
                if constexpr (kTwoSm)
                    mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
                else
                    mbar_arrive(tempty_bar(acc));
            }
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (tma_c && lane == 0) {
            bulk_wait<0>();  // every store of C has completed
            // a c_old load still in flight (one requested before an abandoned wait) lands
            // before the CTA's shared memory goes away
            for (int b = 0; b < 2; ++b)
                if (cpend & (1u << b)) mbar_wait_drain(cold_bar(warp, b), (cph >> b) & 1u);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // with a pair, neither CTA leaves while the other may still write into it or signal it
    if (kPair) cluster_sync();
    if (warp == 0) {
        tc_fence_after();
        if (kTwoSm)
            tmem_dealloc_2sm(tmem_base, L::kTmemCols);
        else
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

// A 2-D tiled tensor map (128-byte swizzle unless `swizzle` says otherwise, 256-byte L2
// promotion, zero fill), encoded once per (data type, address, extents, row stride, box,
// swizzle): a call of the same shape on the same (pooled, hence usually recurring) buffers
// finds its maps in this small cache.  The map depends on nothing else (not on the device:
// the address alone names the memory).
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, void* ptr, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    using Key = std::tuple<int, uintptr_t, uint64_t, uint64_t, uint64_t, uint32_t, uint32_t, int>;
    constexpr size_t kMaxEntries = 256;
    static std::mutex mu;
    static std::map<Key, CUtensorMap> cache;
    const Key key(static_cast<int>(dt), reinterpret_cast<uintptr_t>(ptr), inner, outer, row_bytes, box_inner,
                  box_outer, static_cast<int>(swizzle));
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *map = it->second;
            return true;
        }
    }
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(map, dt, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() >= kMaxEntries) cache.clear();
    cache.emplace(key, *map);
    return true;
}

// Tensor map of a K-major f16 operand: `rows` rows of `Kp` halves (a multiple of 8), `ld`
// halves apart, read in boxes of 64 halves x box_rows.
bool make_map(CUtensorMap* map, const __half* ptr, int64_t rows, int64_t Kp, int box_rows, int64_t ld) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, const_cast<__half*>(ptr), static_cast<uint64_t>(Kp),
                     static_cast<uint64_t>(rows), static_cast<uint64_t>(ld) * 2, kBK, static_cast<uint32_t>(box_rows));
}

using TcKernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, float*, int, int, int,
                            float, float, int, int, unsigned int*, int, int, int, int, float*, __half*,
                            CUtensorMap, int);

// C (M x N f32, rows N floats apart) as 32 x 32 boxes in the 128-byte swizzled layout, for
// the TMA epilogue.  Needs N % 4 == 0 and a 16-byte aligned C.
bool make_map_c(CUtensorMap* map, float* C, int64_t M, int64_t N) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                     static_cast<uint64_t>(N) * 4, 32, 32);
}

// An f16 C as 32 x 32 boxes of 64-byte rows, unswizzled.  Needs N % 8 == 0 and a 16-byte
// aligned C.
bool make_map_ch(CUtensorMap* map, __half* Ch, int64_t M, int64_t N) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Ch, static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                     static_cast<uint64_t>(N) * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
}

struct TcEntry {
    F16Config cfg;
    TcKernelFn fn;      // f32 result
    TcKernelFn fn_tma;  // f32 result through the TMA epilogue
    TcKernelFn fn_h;    // f16 result
    TcKernelFn fn_h_tma;  // f16 result through the TMA epilogue
    uint32_t smem;
};

// PAIR 0 runs in the configuration names as TILE_M=128 (one CTA per tile), PAIR 2 as
// TILE_M=256 (the pair's 2-SM tile).
template <int BN, int STAGES, int PAIR>
TcEntry make_tc_entry() {
    static_assert(PAIR == 0 || PAIR == 2, "one CTA per tile, or the 2-SM pair");
    return TcEntry{F16Config{PAIR == 2 ? 2 * kBM : kBM, BN, kBK, STAGES, PAIR == 0 ? 1 : 2},
                   &gemm_f16tc_kernel<BN, STAGES, PAIR, false, false>, &gemm_f16tc_kernel<BN, STAGES, PAIR, false, true>,
                   &gemm_f16tc_kernel<BN, STAGES, PAIR, true, false>, &gemm_f16tc_kernel<BN, STAGES, PAIR, true, true>,
                   TcLayout<BN, STAGES, PAIR>::kDynSmem};
}

const TcEntry kTcEntries[] = {
    make_tc_entry<256, 4, 0>(), make_tc_entry<256, 3, 0>(), make_tc_entry<128, 6, 0>(),
    make_tc_entry<128, 4, 0>(), make_tc_entry<64, 8, 0>(),  make_tc_entry<256, 6, 2>(),
    make_tc_entry<256, 5, 2>(), make_tc_entry<128, 8, 2>(),
};
constexpr int kNumTc = sizeof(kTcEntries) / sizeof(kTcEntries[0]);

}  // namespace

int f16tc_num_configs() { return kNumTc + f16cvt_num_configs(); }

const F16Config& f16tc_config(int index) {
    return index < kNumTc ? kTcEntries[index].cfg : f16cvt_config(index - kNumTc);
}

bool f16tc_is_convert_a(int index) {
    return index >= kNumTc && index < kNumTc + f16cvt_num_configs() && f16cvt_config(index - kNumTc).convert_a;
}

bool f16tc_is_convert_b(int index) {
    return index >= kNumTc && index < kNumTc + f16cvt_num_configs() && f16cvt_config(index - kNumTc).convert_b;
}

bool f16_operand_map(CUtensorMap* map, const __half* ptr, int64_t rows, int64_t Kp, int box_rows, int64_t ld) {
    return make_map(map, ptr, rows, Kp, box_rows, ld);
}

bool f32_rows_map(CUtensorMap* map, const float* ptr, int64_t rows, int64_t cols, int box_cols, int box_rows) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, const_cast<float*>(ptr), static_cast<uint64_t>(cols),
                     static_cast<uint64_t>(rows), static_cast<uint64_t>(cols) * 4, static_cast<uint32_t>(box_cols),
                     static_cast<uint32_t>(box_rows), CU_TENSOR_MAP_SWIZZLE_NONE);
}

int64_t debug_take_f16tc() { return debug_take_local(); }

size_t f16tc_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    const int64_t Kp = round_up(K, 8);
    return static_cast<size_t>(round_up(M * Kp * 2, 256) + round_up(N * Kp * 2, 256));
}

cudaError_t f16tc_prepare_launch(int in_f16, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                                 const void* A, const void* B, __half* Ah, __half* Bt, int num_sms,
                                 cudaStream_t stream) {
    const int64_t Kp = round_up(K, 8);
    auto aligned = [](const void* p, uintptr_t mask) { return (reinterpret_cast<uintptr_t>(p) & mask) == 0; };
    // K-major A is A itself unless A is given transposed; K-major B is the transpose of B
    // unless B is given transposed.
    auto make_job = [&](const void* src, __half* dst, int64_t rows, int trans) {
        CastJob j;
        j.src = src;
        j.dst = dst;
        j.rows = rows;
        j.trans = trans;
        j.src_f16 = in_f16 ? 1 : 0;
        if (trans)
            j.vec = rows % (in_f16 ? 8 : 4) == 0 && aligned(src, 15u);
        else
            j.vec = (in_f16 ? K % 8 == 0 : K % 4 == 0) && aligned(src, 15u);
        j.tiles_r = static_cast<int>((rows + kTT - 1) / kTT);
        int64_t blocks = 0;
        if (dst == nullptr) {
            blocks = 0;
        } else if (trans) {
            blocks = static_cast<int64_t>(j.tiles_r) * ((Kp + kTT - 1) / kTT);
        } else {
            blocks = (rows * (Kp / 8) + 255) / 256;
            const int64_t cap = static_cast<int64_t>(num_sms) * 8;
            if (blocks > cap) blocks = cap;
        }
        j.blocks = static_cast<int>(blocks < 0x3FFFFFFF ? blocks : 0x3FFFFFFF);
        return j;
    };
    const CastJob ja = make_job(A, Ah, M, trans_a ? 1 : 0);
    const CastJob jb = make_job(B, Bt, N, trans_b ? 0 : 1);
    const int64_t blocks = static_cast<int64_t>(ja.blocks) + jb.blocks;
    if (blocks > 0x7FFFFFFF || ja.blocks == 0x3FFFFFFF || jb.blocks == 0x3FFFFFFF) return cudaErrorInvalidValue;
    if (blocks == 0) return cudaSuccess;
    cast_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(ja, jb, K, Kp);
    return launched(cudaGetLastError());
}

cudaError_t f16tc_cast_launch_ex(int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                                 const float* A, const float* B, void* workspace, int num_sms,
                                 cudaStream_t stream) {
    const int64_t Kp = round_up(K, 8);
    __half* Ah = static_cast<__half*>(workspace);
    __half* Bt = reinterpret_cast<__half*>(static_cast<char*>(workspace) + round_up(M * Kp * 2, 256));
    return f16tc_prepare_launch(0, trans_a, trans_b, M, N, K, A, B, Ah, Bt, num_sms, stream);
}

cudaError_t f16tc_cast_launch(int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                              void* workspace, int num_sms, cudaStream_t stream) {
    return f16tc_cast_launch_ex(0, 0, M, N, K, A, B, workspace, num_sms, stream);
}

namespace {

constexpr int kTcMaxSplit = 8;
constexpr int kTcMinKbPerSlice = 16;

// K blocks per slice when a grid too small for the GPU is split along K; num_kb when not.
int tc_kb_per_slice(const TcEntry& e, int64_t M, int64_t N, int64_t K, int num_sms) {
    const bool mc = e.cfg.cluster == 2;
    const int64_t workers = mc ? num_sms / 2 : num_sms;
    const int64_t tiles_m = (M + kBM - 1) / kBM;
    const int64_t tiles = (mc ? (tiles_m + 1) / 2 : tiles_m) * ((N + e.cfg.tile_n - 1) / e.cfg.tile_n);
    const int64_t num_kb = (K + kBK - 1) / kBK;
    if (workers <= 0 || 2 * tiles > workers) return static_cast<int>(num_kb);
    int64_t split = workers / tiles;
    if (split > kTcMaxSplit) split = kTcMaxSplit;
    if (split > num_kb / kTcMinKbPerSlice) split = num_kb / kTcMinKbPerSlice;
    if (split < 2) return static_cast<int>(num_kb);
    return static_cast<int>((num_kb + split - 1) / split);
}

}  // namespace

size_t f16tc_split_bytes(int index, int64_t M, int64_t N, int64_t K, int num_sms) {
    if (index >= kNumTc) return f16cvt_split_bytes(index - kNumTc, M, N, K, num_sms);
    if (index < 0) return 0;
    const int64_t num_kb = (K + kBK - 1) / kBK;
    const int kb = tc_kb_per_slice(kTcEntries[index], M, N, K, num_sms);
    if (kb >= num_kb) return 0;
    return static_cast<size_t>((num_kb + kb - 1) / kb) * static_cast<size_t>(M * N) * 4;
}

cudaError_t f16tc_gemm_launch(int index, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                              float* C, const void* workspace, void* split_ws, unsigned int* status,
                              int num_sms, cudaStream_t stream) {
    const int64_t Kp = round_up(K, 8);
    const __half* Ah = static_cast<const __half*>(workspace);
    const __half* Bt = reinterpret_cast<const __half*>(static_cast<const char*>(workspace) +
                                                       round_up(M * Kp * 2, 256));
    return f16tc_gemm_launch_ops(index, M, N, K, alpha, beta, C, nullptr, Ah, Kp, Bt, Kp, split_ws, status,
                                 num_sms, stream);
}

cudaError_t f16tc_gemm_launch_ops(int index, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                                  float* C, __half* Ch, const __half* Ah, int64_t lda, const __half* Bt,
                                  int64_t ldb, void* split_ws, unsigned int* status, int num_sms,
                                  cudaStream_t stream) {
    if (index < 0 || index >= kNumTc) return cudaErrorInvalidValue;  // not this kernel's configuration
    const TcEntry& e = kTcEntries[index];
    const int64_t Kp = round_up(K, 8);
    CUtensorMap mapA, mapB, mapB_half, mapB_quarter;
    if (!make_map(&mapA, Ah, M, Kp, kBM, lda) || !make_map(&mapB, Bt, N, Kp, e.cfg.tile_n, ldb) ||
        !make_map(&mapB_half, Bt, N, Kp, e.cfg.tile_n / 2, ldb) ||
        !make_map(&mapB_quarter, Bt, N, Kp, e.cfg.tile_n / 4, ldb))
        return cudaErrorInvalidValue;
    // the TMA epilogue for an f32 C whose rows are 16-byte aligned, or an f16 C with N % 8 == 0
    // and a 16-byte aligned base (whole tiles: decided below, once the split is known)
    CUtensorMap mapC;
    std::memset(&mapC, 0, sizeof mapC);
    const bool c_tma_ok = Ch == nullptr ? N % 4 == 0 && (reinterpret_cast<uintptr_t>(C) & 15u) == 0 &&
                                              make_map_c(&mapC, C, M, N)
                                        : N % 8 == 0 && (reinterpret_cast<uintptr_t>(Ch) & 15u) == 0 &&
                                              make_map_ch(&mapC, Ch, M, N);
    TcKernelFn fn = Ch != nullptr ? e.fn_h : e.fn;
    cudaError_t err = cudaSuccess;
    const int tiles_m = static_cast<int>((M + kBM - 1) / kBM);  // 128-row tiles (one per CTA)
    const int tiles_n = static_cast<int>((N + e.cfg.tile_n - 1) / e.cfg.tile_n);
    // With clusters of two, work is counted in pairs of tiles and in CTA pairs.
    const bool mc = e.cfg.cluster == 2;  // CTA pairs running the 2-SM MMA
    const int64_t workers = mc ? num_sms / 2 : num_sms;
    const int64_t tiles = static_cast<int64_t>(mc ? (tiles_m + 1) / 2 : tiles_m) * tiles_n;
    // Whole tiles for the full rounds of the persistent grid; the tiles of a last, partial
    // round go out as two half-width items each when that still fits in one round.
    const int64_t full = tiles >= workers ? tiles / workers * workers : 0;
    const int64_t tail = tiles - full;
    int tail_split = (tail > 0 && 2 * tail <= workers) ? 2 : 1;
    // a grid too small for the GPU: split along K instead (when there is scratch for it)
    const int64_t num_kb64 = (K + kBK - 1) / kBK;
    int kb_per = tc_kb_per_slice(e, M, N, K, num_sms);
    if (split_ws == nullptr) kb_per = static_cast<int>(num_kb64);
    const int ksplit = static_cast<int>((num_kb64 + kb_per - 1) / kb_per);
    if (ksplit > 1) tail_split = 1;
    const int64_t items = ksplit > 1 ? tiles * ksplit : full + tail * tail_split;
    const int grid = static_cast<int>((items < workers ? items : workers) * (mc ? 2 : 1));
    const int num_kb = static_cast<int>((K + kBK - 1) / kBK);
    // Launched as a programmatic dependent of the cast kernel, so that its prologue (barrier
    // set-up, tensor-memory allocation, descriptor prefetch) overlaps the end of the cast;
    // the producer warp waits for the cast's writes before its first load.
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(grid));
    lc.blockDim = dim3(kThreadsTc);
    lc.dynamicSmemBytes = e.smem;
    lc.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = mc ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 2;
    const int m32 = static_cast<int>(M), n32 = static_cast<int>(N), full32 = static_cast<int>(full);
    float* partial = ksplit > 1 ? static_cast<float*>(split_ws) : nullptr;
    const int epi_tma = (c_tma_ok && ksplit == 1) ? 1 : 0;
    if (epi_tma) fn = Ch != nullptr ? e.fn_h_tma : e.fn_tma;
    err = set_func_attr_once(reinterpret_cast<const void*>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(e.smem));
    if (err != cudaSuccess) return err;
    err = cudaLaunchKernelEx(&lc, fn, mapA, mapB, mapB_half, mapB_quarter, C, m32, n32, num_kb, alpha,
                             beta, tiles_m, tiles_n, status, full32, tail_split, ksplit, kb_per, partial, Ch,
                             mapC, epi_tma);
    if (err != cudaSuccess) {
        // a stream that does not take programmatic launches: launch normally
        cudaGetLastError();
        lc.numAttrs = 1;
        err = cudaLaunchKernelEx(&lc, fn, mapA, mapB, mapB_half, mapB_quarter, C, m32, n32, num_kb,
                                 alpha, beta, tiles_m, tiles_n, status, full32, tail_split, ksplit, kb_per,
                                 partial, Ch, mapC, epi_tma);
    }
    err = launched(err);
    if (err != cudaSuccess || ksplit == 1) return err;
    if (Ch != nullptr) return splitk_reduce_launch_h(partial, ksplit, M, N, alpha, beta, Ch, num_sms, stream);
    return splitk_reduce_launch(partial, ksplit, M, N, alpha, beta, C, num_sms, stream);
}

}  // namespace phx
