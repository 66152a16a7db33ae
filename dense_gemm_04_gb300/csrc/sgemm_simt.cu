// sgemm_simt.cu -- f32 GEMM on the CUDA cores for sm_103a.
//
// C <- alpha * A @ B + beta * C, row-major f32 ("gemm, f32", phobos-lang.dev/docs/examples/
// gemm-fp32/: kernel listing; sections "One output tile per CTA", "The k loop",
// "The epilogue").
//
// Design (one CTA of 256 threads per TILE_M x TILE_N output tile, as in "One output tile
// per CTA" and @launch(256)):
//   * The k loop walks K in steps of TILE_K.  Each step copies a TILE_M x TILE_K panel of
//     A and a TILE_K x TILE_N panel of B into a STAGES-deep ring of shared-memory buffers
//     with cp.async, so the copies of the next STAGES-1 panels overlap the math on the
//     current one (the @pipeline double buffering, generalised to STAGES >= 2).
//   * Aligned path: both panels move as 16-byte cp.async.cg copies (the @aligned promise:
//     no masks, 16-byte vector loads).  Masked paths: when rows are still 16 bytes apart
//     (K % 4 == N % 4 == 0, aligned bases), 16-byte copies whose source size is 0 past an
//     edge; otherwise 4-byte cp.async.ca copies of that kind ("extra 128-byte lines, masked
//     elements").  Either writes zeros past an edge, and stores past an edge are skipped.
//     All paths compute the same values.
//   * The output tile is split over 8 warps (4 x 2) and each warp's tile over its 32 lanes
//     (4 x 8); every thread owns a TM x TN register micro-tile of accumulators, as the
//     lab's register-tiling rung does (Part 2, "register tiling"; Part 2, "The register
//     patch: reuse against occupancy").  The A panel lands row-major (as copied, 16 bytes
//     at a time) and is rewritten once per k tile into a k-major buffer, so that at each k
//     step a thread reads its TM values of A and its TN values of B as float4s.  The
//     copies of a later panel and the rewrite of the next one are issued part way through
//     the current panel's k steps, overlapping the multiply-adds.  Lanes that
//     share rows or columns read the same shared-memory words (broadcast), so one warp's
//     loads per k step touch 16 (or 32) rows of A and 64 (or 32) columns of B.
//   * Optionally (FMA2 = 1) the multiply-adds are issued as packed f32x2 FMAs (__ffma2_rn),
//     halving the FMA instructions the schedulers issue; each lane of the pair is an
//     ordinary IEEE f32 fused multiply-add, so the values are the same.
//   * Epilogue: C is read once (not at all when beta == 0) and written once, with 16-byte
//     accesses on the aligned path.
//   * A grid of more than one wave whose last wave would leave SMs idle spreads that wave's
//     k tiles evenly over one stream-K block per CTA slot (StreamK below).
// The tile body is in sgemm_tile_body.inc.
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <array>
#include <cstdint>
#include <map>
#include <mutex>
#include <vector>

#include "debug_checks.cuh"
#include "internal.h"

namespace phx {
namespace {

constexpr int kThreads = 256;
constexpr int kLanesM = 4;  // lanes of a warp along M
constexpr int kLanesN = 8;  // lanes of a warp along N

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 4-byte asynchronous copy; with pred false the source is not read and zeros are written.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const float* src, bool pred) {
    const int bytes = pred ? 4 : 0;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(bytes)
                 : "memory");
}

// 16-byte asynchronous copy, bypassing L1 (the panel is used once per CTA).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const float* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}

// 16-byte asynchronous copy that, with pred false, reads nothing and writes 16 zero bytes.
__device__ __forceinline__ void cp_async_16_zfill(uint32_t dst, const float* src, bool pred) {
    const int bytes = pred ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(bytes)
                 : "memory");
}

// How a kernel treats the edges of the matrices: every dimension a whole number of tiles and
// 16-byte rows (none); rows 16 bytes apart (K % 4 == N % 4 == 0, 16-byte aligned bases) and
// tiles past M, N or K (vec: 16-byte copies and stores, pieces past an edge zero or
// skipped); anything else (scalar: 4-byte copies and stores).
constexpr int kEdgeNone = 0;
constexpr int kEdgeScalar = 1;
constexpr int kEdgeVec = 2;

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Map a linear CTA index to (tile row, tile column), walking groups of 8 tile rows
// column by column so that CTAs running together share panels of A and B in L2.
__device__ __forceinline__ void tile_coords(int bid, int tiles_m, int tiles_n, int& pm, int& pn) {
    constexpr int kGroup = 8;
    const int per_group = kGroup * tiles_n;
    const int group = bid / per_group;
    const int first_m = group * kGroup;
    const int rows = min(tiles_m - first_m, kGroup);
    const int r = bid - group * per_group;
    pm = first_m + r % rows;
    pn = r / rows;
}

// Row stride (floats) of the k-major copy of the A panel: TILE_M plus 4, which keeps the
// 16-byte fragment reads aligned and spreads the transposing stores over the banks.
__host__ __device__ constexpr int at_row_stride(int bm) { return bm + 4; }

// Shared-memory floats one CTA uses: the A staging ring (row-major, as copied), two
// k-major A buffers, and the B ring.
__host__ __device__ constexpr int sgemm_smem_floats(int bm, int bn, int bk, int stages) {
    return stages * bm * bk + 2 * bk * at_row_stride(bm) + stages * bk * bn;
}

// Stream-K.  A grid whose last, partial wave would leave SMs idle -- or a grid of less than
// one wave -- runs its whole waves as tiles (sgemm_kernel over tiles [0, dp_tiles)) and
// spreads the k tiles of the remaining (tail) tiles evenly over `blocks` blocks of
// sgemm_streamk_kernel, at most one per CTA slot of the GPU, launched first so that they
// fill the GPU together: block s takes k tiles [s * work / blocks, (s + 1) * work / blocks)
// of the tail's k tiles laid end to end (tile after tile).  streamk_fixup_kernel then adds
// each tail tile's partial tiles in k order and applies alpha and beta, before the whole
// tiles run (while the partial tiles are still in L2).  The tail thus takes the same time
// on every block, instead of leaving SMs idle for a fraction of a wave.  (streamk_plan
// decides when, and how many blocks.)
struct StreamK {
    int dp_tiles;   // tiles [0, dp_tiles) are whole tiles; the rest are the tail
    int blocks;     // stream-K blocks (0: none)
    int64_t work;   // tail tiles x k tiles per tile
    float* slots;   // 2 * blocks tiles of BM x BN partial sums
};

// First k tile (of the tail's, end to end) of stream-K block s.
__host__ __device__ __forceinline__ int64_t streamk_begin(int64_t s, int64_t work, int64_t blocks) {
    return s * work / blocks;
}

// The stream-K block whose range contains k tile `lo` (of the tail's, end to end).
__host__ __device__ __forceinline__ int64_t streamk_first_block(int64_t lo, int64_t work, int64_t blocks) {
    int64_t b = lo * blocks / work;
    while (b > 0 && streamk_begin(b, work, blocks) > lo) --b;
    while (b + 1 < blocks && streamk_begin(b + 1, work, blocks) <= lo) ++b;
    return b;
}

// One output tile, or a k range of one: the CTA's whole computation, shared by the tile
// kernel and the stream-K kernel below.  Without LOCAL: tile blockIdx.x, whole K (or the
// k slice of a split grid), into C (or the slice's plane of `partial`).  With LOCAL: k
// tiles [kt0, kt1) of `tile`, alpha = 1 and beta = 0, into the BM x BN tile of partial sums
// at C (element (row, col) at C[(row - m0) * BN + col - n0]).
template <int BM, int BN, int BK, int STAGES, int TM, int TN, int EDGE, bool FMA2, bool LOCAL>
__device__ __forceinline__ void sgemm_tile(const float* __restrict__ A, const float* __restrict__ B,
                                           float* __restrict__ C, int M, int N, int K, int ldb, float alpha,
                                           float beta, int k_slice, float* __restrict__ partial, int tile, int kt0,
                                           int kt1) {
#include "sgemm_tile_body.inc"
}

template <int BM, int BN, int BK, int STAGES, int TM, int TN, int EDGE, bool FMA2, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
sgemm_kernel(const float* __restrict__ A, const float* __restrict__ B, float* __restrict__ C,
             int M, int N, int K, int ldb, float alpha, float beta, int k_slice, float* __restrict__ partial) {
    if constexpr (EDGE != kEdgeScalar) {
        sgemm_tile<BM, BN, BK, STAGES, TM, TN, EDGE, FMA2, false>(A, B, C, M, N, K, ldb, alpha, beta, k_slice, partial,
                                                                  0, 0, 0);
    } else {
        constexpr bool LOCAL = false;
        int tile = 0;
        const int kt0 = 0, kt1 = 0;
#include "sgemm_tile_body.inc"
    }
}

// Stream-K block s: k tiles [streamk_begin(s), streamk_begin(s + 1)) of the tail tiles'
// k tiles laid end to end, as at most two segments (the end of one tile, the start of the
// next), each written as a BM x BN tile of partial sums to slot 2s + segment.
template <int BM, int BN, int BK, int STAGES, int TM, int TN, int EDGE, bool FMA2, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
sgemm_streamk_kernel(const float* __restrict__ A, const float* __restrict__ B, int M, int N, int K, int ldb,
                     const StreamK sk) {
    const int k_tiles = (K + BK - 1) / BK;
    const int64_t s = blockIdx.x;
    int64_t it = streamk_begin(s, sk.work, sk.blocks);
    const int64_t end = streamk_begin(s + 1, sk.work, sk.blocks);
    int seg = 0;
#pragma unroll 1
    while (it < end) {
        const int t = static_cast<int>(it / k_tiles);
        const int kt0 = static_cast<int>(it - static_cast<int64_t>(t) * k_tiles);
        const int kt1 = static_cast<int>(min(static_cast<int64_t>(k_tiles), kt0 + (end - it)));
        if (seg > 0) __syncthreads();  // the first segment is done with the shared buffers
        sgemm_tile<BM, BN, BK, STAGES, TM, TN, EDGE, FMA2, true>(A, B, sk.slots + (2 * s + seg) * (BM * BN), M, N, K,
                                                                   ldb, 1.f, 0.f, 0, nullptr, sk.dp_tiles + t, kt0,
                                                                   kt1);
        it += kt1 - kt0;
        ++seg;
    }
}

// Finish the tail tiles of a stream-K launch: C <- alpha * sum + beta * C (beta == 0: C not
// read), where the sum adds, in k order, the partial tiles of the stream-K blocks whose k
// ranges meet the tile (a block that began in the tile before holds its part in its second
// slot; every block's range is at most one tile long, so it meets at most two tiles).
// bm * bn / 4096 blocks of 256 threads share a tile, each thread owning 4 float4s
// (thread x of part q: float4 q * 1024 + x + 256 i).  The partial tiles are read four at a
// time, all their loads in flight together, and added in k order; the segment bounds are
// the same for the whole block.
constexpr int kFixupVec = 4;      // float4s per thread and partial tile
constexpr int kFixupBatch = 4;    // partial tiles whose loads are in flight together
constexpr int kFixupThreads = 256;

__global__ void __launch_bounds__(kFixupThreads) streamk_fixup_kernel(StreamK sk, int k_tiles, int bm, int bn, int M,
                                                                      int N, float alpha, float beta,
                                                                      float* __restrict__ C, int vec) {
    const int parts = bm * bn / (4 * kFixupVec * kFixupThreads);
    const int t = static_cast<int>(blockIdx.x) / parts;
    const int part = static_cast<int>(blockIdx.x) - t * parts;
    const int64_t lo = static_cast<int64_t>(t) * k_tiles;
    const int64_t hi = lo + k_tiles;
    int64_t b = streamk_first_block(lo, sk.work, sk.blocks);
    int pm, pn;
    tile_coords(sk.dp_tiles + t, (M + bm - 1) / bm, (N + bn - 1) / bn, pm, pn);
    const int m0 = pm * bm, n0 = pn * bn;
    const int64_t tile_elems = static_cast<int64_t>(bm) * bn;
    const int first4 = part * (kFixupVec * kFixupThreads) + static_cast<int>(threadIdx.x);  // float4 index
    float4 acc[kFixupVec];
    bool first = true;
    int64_t s0 = streamk_begin(b, sk.work, sk.blocks);
    while (b < sk.blocks && s0 < hi) {
        // up to kFixupBatch non-empty partial tiles of this tile, in k order
        const float4* src[kFixupBatch];
        int n = 0;
        while (n < kFixupBatch && b < sk.blocks && s0 < hi) {
            const int64_t s1 = streamk_begin(b + 1, sk.work, sk.blocks);
            if (s1 > s0) {  // an empty range wrote nothing
                PHX_DCHECK(b < sk.blocks);
                src[n++] = reinterpret_cast<const float4*>(sk.slots + (2 * b + (s0 < lo ? 1 : 0)) * tile_elems);
            }
            s0 = s1;
            ++b;
        }
        float4 v[kFixupBatch][kFixupVec];
#pragma unroll
        for (int q = 0; q < kFixupBatch; ++q) {
            if (q < n) {
#pragma unroll
                for (int i = 0; i < kFixupVec; ++i) {
                    PHX_DCHECK(4 * (first4 + i * kFixupThreads) + 3 < tile_elems);
                    v[q][i] = __ldcs(src[q] + first4 + i * kFixupThreads);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kFixupBatch; ++q) {
            if (q < n) {
#pragma unroll
                for (int i = 0; i < kFixupVec; ++i) {
                    if (first) {
                        acc[i] = v[q][i];
                    } else {
                        acc[i].x += v[q][i].x; acc[i].y += v[q][i].y; acc[i].z += v[q][i].z; acc[i].w += v[q][i].w;
                    }
                }
                first = false;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kFixupVec; ++i) {
        const int e = 4 * (first4 + i * kFixupThreads);
        const int row = m0 + e / bn;
        const int col = n0 + e % bn;
        if (row >= M || col >= N) continue;
        PHX_DCHECK(!first && (!vec || col + 3 < N));  // every spread tile gets a partial sum
        float* c = C + static_cast<int64_t>(row) * N + col;
        const float a[4] = {acc[i].x, acc[i].y, acc[i].z, acc[i].w};
        if (vec) {
            float4 o = make_float4(alpha * a[0], alpha * a[1], alpha * a[2], alpha * a[3]);
            if (beta != 0.f) {
                const float4 co = *reinterpret_cast<const float4*>(c);
                o.x = fmaf(beta, co.x, o.x); o.y = fmaf(beta, co.y, o.y);
                o.z = fmaf(beta, co.z, o.z); o.w = fmaf(beta, co.w, o.w);
            }
            *reinterpret_cast<float4*>(c) = o;
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (col + q >= N) break;
                float o = alpha * a[q];
                if (beta != 0.f) o = fmaf(beta, c[q], o);
                c[q] = o;
            }
        }
    }
}

// C <- alpha * (P[0] + P[1] + ... + P[S-1]) + beta * C, the planes added in that order
// (beta == 0: C not read).  float4 when N % 4 == 0 and the pointers are 16-byte aligned.
__global__ void splitk_reduce_kernel(const float* __restrict__ P, int S, int64_t plane, float alpha,
                                     float beta, float* __restrict__ C, int vec) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t start = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (vec) {
        PHX_DCHECK(plane % 4 == 0);
        const int64_t n4 = plane / 4;
        for (int64_t i = start; i < n4; i += stride) {
            float4 acc = __ldcs(reinterpret_cast<const float4*>(P) + i);
            for (int s = 1; s < S; ++s) {
                const float4 v = __ldcs(reinterpret_cast<const float4*>(P + s * plane) + i);
                acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
            }
            float4 o = make_float4(alpha * acc.x, alpha * acc.y, alpha * acc.z, alpha * acc.w);
            if (beta != 0.f) {
                const float4 c = reinterpret_cast<const float4*>(C)[i];
                o.x = fmaf(beta, c.x, o.x); o.y = fmaf(beta, c.y, o.y);
                o.z = fmaf(beta, c.z, o.z); o.w = fmaf(beta, c.w, o.w);
            }
            reinterpret_cast<float4*>(C)[i] = o;
        }
        return;
    }
    for (int64_t i = start; i < plane; i += stride) {
        float acc = P[i];
        for (int s = 1; s < S; ++s) acc += P[s * plane + i];
        float o = alpha * acc;
        if (beta != 0.f) o = fmaf(beta, C[i], o);
        C[i] = o;
    }
}

// The split-K reduction into a half-precision C: the slices added in order in f32, then
// alpha * sum + beta * c_old rounded to f16 once.
__global__ void splitk_reduce_h_kernel(const float* __restrict__ P, int S, int64_t plane, float alpha, float beta,
                                       __half* __restrict__ C) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < plane; i += stride) {
        float acc = P[i];
        for (int s = 1; s < S; ++s) acc += P[s * plane + i];
        float o = alpha * acc;
        if (beta != 0.f) o = fmaf(beta, __half2float(C[i]), o);
        C[i] = __float2half_rn(o);
    }
}

__global__ void scale_c_h_kernel(__half* __restrict__ C, int64_t n, float beta) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        C[i] = __float2half_rn(beta == 0.f ? 0.f : beta * __half2float(C[i]));
}

// dst (cols x rows) <- src (rows x cols) transposed, through 32 x 32 tiles of shared
// memory padded by one column (conflict-free in both directions).
__global__ void __launch_bounds__(256) transpose_f32_kernel(const float* __restrict__ src, float* __restrict__ dst,
                                                            int64_t rows, int64_t cols, int64_t tiles_c) {
    __shared__ float t[32][33];
    const int64_t c0 = (static_cast<int64_t>(blockIdx.x) % tiles_c) * 32;
    const int64_t r0 = (static_cast<int64_t>(blockIdx.x) / tiles_c) * 32;
    const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;  // 32 x 8
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t r = r0 + ty + i * 8, c = c0 + tx;
        if (r < rows && c < cols) t[ty + i * 8][tx] = __ldcs(src + r * cols + c);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t c = c0 + ty + i * 8, r = r0 + tx;
        if (c < cols && r < rows) dst[c * rows + r] = t[tx][ty + i * 8];
    }
}

// C <- beta * C over M*N elements (beta == 0 writes zeros without reading C).
// dst[r][c] = src[r * sld + c] for r < srows and c < scols, else 0; one float4 of dst per
// thread and step (dcols % 4 == 0), grid-stride.
__global__ void __launch_bounds__(256) pad_copy_kernel(const float* __restrict__ src, int64_t srows, int64_t scols,
                                                       int64_t sld, float4* __restrict__ dst, int64_t rows,
                                                       int64_t dcols4) {
    const int64_t total = rows * dcols4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t r = i / dcols4;
        const int64_t c = (i - r * dcols4) * 4;
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = (r < srows && c + q < scols) ? __ldcs(src + r * sld + c + q) : 0.f;
        dst[i] = make_float4(v[0], v[1], v[2], v[3]);
    }
}

__global__ void scale_c_kernel(float* __restrict__ C, int64_t n, float beta) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        C[i] = beta == 0.f ? 0.f : beta * C[i];
}

// ---------------------------------------------------------------------------------------
// The compiled configurations.  The pages' search space is TILE_M, TILE_N in
// {32, 64, 128, 256} and TILE_K in {4, 8, 16, 32} ("gemm, f32", section "The attributes",
// @autotune row); this build compiles the part of it that a 256-thread CTA with
// 4x4..8x16 register micro-tiles covers, times STAGES in {3, 4} and the FMA2 switch.
// ---------------------------------------------------------------------------------------
using KernelFn = void (*)(const float*, const float*, float*, int, int, int, int, float, float, int, float*);
using StreamKFn = void (*)(const float*, const float*, int, int, int, int, StreamK);

struct Entry {
    SgemmConfig cfg;
    KernelFn fn[3];   // tile kernel by edge mode (kEdgeNone, kEdgeScalar, kEdgeVec)
    StreamKFn sk[3];  // the stream-K blocks of the same tile shape
    int smem_bytes;
};

template <int BM, int BN, int BK, int STAGES, int FMA2>
constexpr Entry make_entry() {
    constexpr int TM = BM / 16;  // 4 warps x 4 lanes along M
    constexpr int TN = BN / 16;  // 2 warps x 8 lanes along N
    // up to 64 accumulators a thread: two CTAs per SM (128 registers); 128: one CTA
    constexpr int MINB = TM * TN > 64 ? 1 : 2;
    return Entry{SgemmConfig{BM, BN, BK, STAGES, FMA2},
                 {&sgemm_kernel<BM, BN, BK, STAGES, TM, TN, kEdgeNone, FMA2 != 0, MINB>,
                  &sgemm_kernel<BM, BN, BK, STAGES, TM, TN, kEdgeScalar, FMA2 != 0, MINB>,
                  &sgemm_kernel<BM, BN, BK, STAGES, TM, TN, kEdgeVec, FMA2 != 0, MINB>},
                 {&sgemm_streamk_kernel<BM, BN, BK, STAGES, TM, TN, kEdgeNone, FMA2 != 0, MINB>,
                  &sgemm_streamk_kernel<BM, BN, BK, STAGES, TM, TN, kEdgeScalar, FMA2 != 0, MINB>,
                  &sgemm_streamk_kernel<BM, BN, BK, STAGES, TM, TN, kEdgeVec, FMA2 != 0, MINB>},
                 sgemm_smem_floats(BM, BN, BK, STAGES) * 4};
}

const Entry kEntries[] = {
    make_entry<128, 128, 8, 4, 0>(),  make_entry<128, 128, 8, 4, 1>(),
    make_entry<128, 128, 16, 3, 0>(), make_entry<128, 128, 16, 3, 1>(),
    make_entry<128, 128, 16, 4, 0>(), make_entry<128, 128, 16, 4, 1>(),
    make_entry<128, 128, 8, 3, 0>(),  make_entry<128, 128, 8, 3, 1>(),
    make_entry<128, 64, 8, 4, 0>(),   make_entry<128, 64, 16, 4, 1>(),
    make_entry<64, 128, 8, 4, 0>(),   make_entry<64, 128, 16, 4, 1>(),
    make_entry<64, 64, 8, 4, 0>(),    make_entry<64, 64, 16, 4, 0>(),
    make_entry<128, 256, 8, 4, 1>(),  make_entry<128, 256, 16, 3, 1>(),
    make_entry<128, 256, 16, 4, 1>(), make_entry<256, 128, 8, 4, 1>(),
    make_entry<256, 128, 16, 3, 1>(),
};
constexpr int kNumEntries = sizeof(kEntries) / sizeof(kEntries[0]);

}  // namespace

int sgemm_num_configs() { return kNumEntries; }

const SgemmConfig& sgemm_config(int index) { return kEntries[index].cfg; }

bool sgemm_is_aligned(int index, int64_t M, int64_t N, int64_t K, const float* A,
                      const float* B, const float* C) {
    const SgemmConfig& c = kEntries[index].cfg;
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    return M % c.tile_m == 0 && N % c.tile_n == 0 && K % c.tile_k == 0 && al16(A) && al16(B) &&
           al16(C);
}

namespace {

// The edge mode of config `index` for this problem with B's rows ldb floats apart: the aligned
// kernel for whole tiles; the 16-byte copies whenever the rows of A and B start on 16 bytes
// (C's rows decide only between 16- and 4-byte accesses in the epilogue); else 4-byte copies.
int sgemm_edge(int index, int64_t M, int64_t N, int64_t K, const float* A, const float* B, const float* C,
               int64_t ldb) {
    if (ldb == N && sgemm_is_aligned(index, M, N, K, A, B, C)) return kEdgeNone;
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    return (K % 4 == 0 && ldb % 4 == 0 && al16(A) && al16(B)) ? kEdgeVec : kEdgeScalar;
}

}  // namespace

namespace {

// CTAs of `fn` that fit on one SM at once (cached per device and kernel).
int ctas_per_sm(KernelFn fn, int smem) {
    static std::mutex mu;
    static std::map<std::pair<int, KernelFn>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_pair(dev, fn);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (set_func_attr_once(reinterpret_cast<const void*>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        n = 1;
    }
    if (n < 1) n = 1;
    cache[key] = n;
    return n;
}

constexpr int kMaxSplit = 8;
constexpr int kMinKTilesPerSlice = 16;

// Elements of K per slice when a grid too small for the GPU is split along K (the grid
// gets one row of CTAs per slice); K itself when it is not split.
// The split for `tiles` tiles of `k_tiles` k tiles on `slots` CTA slots, in elements of K
// per slice (K itself: no split).
int64_t k_per_slice_core(int64_t tiles, int64_t k_tiles, int64_t slots, int tile_k, int64_t K) {
    if (slots <= 0 || 2 * tiles > slots) return K;
    int64_t split = slots / tiles;
    if (split > kMaxSplit) split = kMaxSplit;
    if (split > k_tiles / kMinKTilesPerSlice) split = k_tiles / kMinKTilesPerSlice;
    if (split < 2) return K;
    return (k_tiles + split - 1) / split * tile_k;
}

int64_t k_per_slice(const Entry& e, int edge, int64_t M, int64_t N, int64_t K, int num_sms) {
    const int64_t tiles = ((M + e.cfg.tile_m - 1) / e.cfg.tile_m) * ((N + e.cfg.tile_n - 1) / e.cfg.tile_n);
    const int64_t slots = static_cast<int64_t>(ctas_per_sm(e.fn[edge], e.smem_bytes)) * num_sms;
    const int64_t k_tiles = (K + e.cfg.tile_k - 1) / e.cfg.tile_k;
    return k_per_slice_core(tiles, k_tiles, slots, e.cfg.tile_k, K);
}

// Stream-K plan (see StreamK).  The last, partial wave of the tile grid -- or the whole
// grid when it is less than one wave -- has T tiles of I k tiles each; its T * I k tiles go
// to P blocks, P = min(slots, T * I / kStreamKMinKTiles, kStreamKMaxSegments * T) and at
// least T (so that every block's range is at most one tile long and each block gets
// kStreamKMinKTiles or more; a tile is then split into at most about kStreamKMaxSegments
// partial tiles, which bounds the fix-up).
//   * Time in units of one tile computed by a CTA alone on its SM (the kernel is bound by
//     the SM's FMA rate, so CTAs sharing an SM share that rate): the T tiles as tiles take
//     ceil(T / SMs), the P blocks ceil(P / SMs) * T / P.  The plan is used when that saves
//     at least kStreamKMinGain of a wave (CTAs per SM tile times).
//   * Each segment costs a pipeline fill and a tile of partial sums, and the fix-up adds a
//     pass.  So blocks of fewer than kStreamKLongKTiles k tiles are used only where they
//     beat the alternative (the T tiles, or a grid split along K into slices) by a margin.
//     In k tiles of a lone CTA: n CTAs of k k-tiles each take ceil(n / SMs) * k.  The
//     blocks must take at most half of the alternative's time, or kStreamKOverheadKTiles
//     less.  Measured (f32, 128 x 128 tile, 152 SMs): 256^3 and 512^3 gain from blocks of
//     8 k tiles, 1024^3 and (300, 500, 3000) run faster split along K, and (2048, 2048,
//     256) as tiles.
constexpr double kStreamKMinGain = 0.05;
constexpr int64_t kStreamKMinKTiles = 8;
constexpr int64_t kStreamKLongKTiles = 64;
constexpr int64_t kStreamKMaxSegments = 8;
constexpr double kStreamKOverheadKTiles = 12.0;

// The plan for `tiles` tiles of `k_tiles` k tiles (of tile_k values of K) with `per_sm` CTAs
// per SM on `num_sms` SMs; no device queries, so it can be checked on the host.
StreamK streamk_plan_core(int64_t tiles, int64_t k_tiles, int64_t per_sm, int64_t num_sms, int tile_k, int64_t K) {
    StreamK sk{0, 0, 0, nullptr};
    const int64_t slots = per_sm * num_sms;
    if (num_sms <= 0 || per_sm <= 0 || tiles <= 0 || k_tiles <= 0) return sk;
    const int64_t tail = tiles > slots ? tiles % slots : tiles;
    if (tail == 0) return sk;
    const int64_t work = tail * k_tiles;
    int64_t blocks = slots;
    if (blocks > work / kStreamKMinKTiles) blocks = work / kStreamKMinKTiles;
    if (blocks > kStreamKMaxSegments * tail) blocks = kStreamKMaxSegments * tail;
    if (blocks < tail) return sk;
    const double as_tiles = static_cast<double>((tail + num_sms - 1) / num_sms);
    const double spread = static_cast<double>((blocks + num_sms - 1) / num_sms) * static_cast<double>(tail) /
                          static_cast<double>(blocks);
    if ((as_tiles - spread) / static_cast<double>(per_sm) < kStreamKMinGain) return sk;
    if (work / blocks < kStreamKLongKTiles) {
        int64_t alt_ctas = tail, alt_k = k_tiles;  // the alternative: CTAs, k tiles each
        if (tiles <= slots) {
            const int64_t ks = k_per_slice_core(tiles, k_tiles, slots, tile_k, K);
            alt_ctas = tiles * ((K + ks - 1) / ks);
            alt_k = (ks + tile_k - 1) / tile_k;
        }
        const double alt_t = static_cast<double>((alt_ctas + num_sms - 1) / num_sms) * static_cast<double>(alt_k);
        const double sk_t = static_cast<double>((blocks + num_sms - 1) / num_sms) * static_cast<double>(work) /
                            static_cast<double>(blocks);
        if (sk_t > 0.5 * alt_t && sk_t + kStreamKOverheadKTiles > alt_t) return sk;
    }
    sk.dp_tiles = static_cast<int>(tiles - tail);
    sk.blocks = static_cast<int>(blocks);
    sk.work = work;
    return sk;
}

StreamK streamk_plan(const Entry& e, int edge, int64_t M, int64_t N, int64_t K, int num_sms) {
    const int64_t tiles = ((M + e.cfg.tile_m - 1) / e.cfg.tile_m) * ((N + e.cfg.tile_n - 1) / e.cfg.tile_n);
    const int64_t k_tiles = (K + e.cfg.tile_k - 1) / e.cfg.tile_k;
    return streamk_plan_core(tiles, k_tiles, ctas_per_sm(e.fn[edge], e.smem_bytes), num_sms, e.cfg.tile_k, K);
}

}  // namespace

void sgemm_schedule_selftest(int index, int64_t M, int64_t N, int64_t K, int per_sm, int num_sms, int64_t out[6]) {
    const Entry& e = kEntries[index];
    const int64_t tiles = ((M + e.cfg.tile_m - 1) / e.cfg.tile_m) * ((N + e.cfg.tile_n - 1) / e.cfg.tile_n);
    const int64_t k_tiles = (K + e.cfg.tile_k - 1) / e.cfg.tile_k;
    const StreamK sk = streamk_plan_core(tiles, k_tiles, per_sm, num_sms, e.cfg.tile_k, K);
    const int64_t ks = sk.blocks > 0 ? K
                                     : k_per_slice_core(tiles, k_tiles, static_cast<int64_t>(per_sm) * num_sms,
                                                        e.cfg.tile_k, K);
    out[0] = sk.blocks > 0 ? sk.dp_tiles : tiles;
    out[1] = sk.blocks;
    out[2] = sk.work;
    out[3] = (K + ks - 1) / ks;
    out[4] = 0;
    out[5] = 1;
    if (sk.blocks == 0) return;
    // the segments the stream-K blocks write, walked as sgemm_streamk_kernel walks them:
    // (first k tile, end k tile, slot) per tail tile
    const int64_t tail = tiles - sk.dp_tiles;
    std::vector<std::vector<std::array<int64_t, 3>>> written(static_cast<size_t>(tail));
    for (int64_t b = 0; b < sk.blocks; ++b) {
        int64_t it = streamk_begin(b, sk.work, sk.blocks);
        const int64_t end = streamk_begin(b + 1, sk.work, sk.blocks);
        int64_t seg = 0;
        while (it < end) {
            const int64_t t = it / k_tiles;
            const int64_t kt0 = it - t * k_tiles;
            const int64_t kt1 = std::min(k_tiles, kt0 + (end - it));
            written[static_cast<size_t>(t)].push_back({kt0, kt1, 2 * b + seg});
            it += kt1 - kt0;
            ++seg;
        }
        out[4] = std::max(out[4], seg);
    }
    // the slots the fix-up reads, walked as streamk_fixup_kernel walks them
    for (int64_t t = 0; t < tail; ++t) {
        const int64_t lo = t * k_tiles, hi = lo + k_tiles;
        int64_t b = streamk_first_block(lo, sk.work, sk.blocks);
        int64_t s0 = streamk_begin(b, sk.work, sk.blocks);
        std::vector<int64_t> reads;
        for (; b < sk.blocks && s0 < hi; ++b) {
            const int64_t s1 = streamk_begin(b + 1, sk.work, sk.blocks);
            if (s1 > s0) reads.push_back(2 * b + (s0 < lo ? 1 : 0));
            s0 = s1;
        }
        const auto& w = written[static_cast<size_t>(t)];
        bool ok = reads.size() == w.size() && !w.empty() && w.front()[0] == 0 && w.back()[1] == k_tiles;
        for (size_t q = 0; ok && q < w.size(); ++q) {
            ok = reads[q] == w[q][2] && (q == 0 || w[q - 1][1] == w[q][0]);
        }
        if (!ok) out[5] = 0;
    }
}

size_t sgemm_workspace_bytes(int index, int64_t M, int64_t N, int64_t K, const float* A,
                             const float* B, const float* C, int num_sms, int64_t ldb) {
    const Entry& e = kEntries[index];
    const int edge = sgemm_edge(index, M, N, K, A, B, C, ldb < 0 ? N : ldb);
    const StreamK sk = streamk_plan(e, edge, M, N, K, num_sms);
    if (sk.blocks > 0) return static_cast<size_t>(2 * sk.blocks) * e.cfg.tile_m * e.cfg.tile_n * 4;
    const int64_t ks = k_per_slice(e, edge, M, N, K, num_sms);
    if (ks < K) return static_cast<size_t>((K + ks - 1) / ks) * static_cast<size_t>(M * N) * 4;
    return 0;
}

cudaError_t sgemm_launch(int index, int64_t M, int64_t N, int64_t K, float alpha,
                         const float* A, const float* B, float beta, float* C, void* workspace,
                         int num_sms, cudaStream_t stream, int64_t ldb) {
    if (ldb < 0) ldb = N;
    const Entry& e = kEntries[index];
    const int edge = sgemm_edge(index, M, N, K, A, B, C, ldb);
    KernelFn fn = e.fn[edge];
    cudaError_t err = set_func_attr_once(reinterpret_cast<const void*>(fn),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, e.smem_bytes);
    if (err != cudaSuccess) return err;
    const int64_t tiles = ((M + e.cfg.tile_m - 1) / e.cfg.tile_m) * ((N + e.cfg.tile_n - 1) / e.cfg.tile_n);
    if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
    // a stream-K spread of the last wave (or of the whole grid) first; else a grid too small
    // for the GPU split along K; else tiles only (no scratch: tiles only)
    StreamK sk{0, 0, 0, nullptr};
    if (workspace != nullptr) sk = streamk_plan(e, edge, M, N, K, num_sms);
    int64_t ks = sk.blocks > 0 ? K : k_per_slice(e, edge, M, N, K, num_sms);
    if (workspace == nullptr) ks = K;
    const int64_t slices = (K + ks - 1) / ks;
    float* partial = slices > 1 ? static_cast<float*>(workspace) : nullptr;
    if (sk.blocks > 0) {
        // the stream-K blocks first, one per CTA slot: they fill the GPU on their own
        StreamKFn skf = e.sk[edge];
        err = set_func_attr_once(reinterpret_cast<const void*>(skf), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 e.smem_bytes);
        if (err != cudaSuccess) return err;
        sk.slots = static_cast<float*>(workspace);
        skf<<<static_cast<unsigned>(sk.blocks), kThreads, e.smem_bytes, stream>>>(
            A, B, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), static_cast<int>(ldb), sk);
        err = launched(cudaGetLastError());
        if (err != cudaSuccess) return err;
        // then the tail tiles of C, while the partial tiles are still in L2 (the whole tiles
        // below write other elements of C)
        const int vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15u) == 0);
        const int parts = e.cfg.tile_m * e.cfg.tile_n / (4 * kFixupVec * kFixupThreads);
        streamk_fixup_kernel<<<static_cast<unsigned>((tiles - sk.dp_tiles) * parts), kFixupThreads, 0, stream>>>(
            sk, static_cast<int>((K + e.cfg.tile_k - 1) / e.cfg.tile_k), e.cfg.tile_m, e.cfg.tile_n,
            static_cast<int>(M), static_cast<int>(N), alpha, beta, C, vec);
        err = launched(cudaGetLastError());
        if (err != cudaSuccess) return err;
    }
    const int64_t grid = sk.blocks > 0 ? sk.dp_tiles : tiles;
    if (grid == 0) return cudaSuccess;  // the whole grid went to the stream-K blocks
    fn<<<dim3(static_cast<unsigned>(grid), static_cast<unsigned>(slices)), kThreads, e.smem_bytes, stream>>>(
        A, B, C, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), static_cast<int>(ldb), alpha, beta,
        static_cast<int>(ks), partial);
    err = launched(cudaGetLastError());
    if (err != cudaSuccess || slices == 1) return err;
    return splitk_reduce_launch(partial, static_cast<int>(slices), M, N, alpha, beta, C, num_sms, stream);
}

cudaError_t splitk_reduce_launch(const float* partial, int slices, int64_t M, int64_t N, float alpha,
                                 float beta, float* C, int num_sms, cudaStream_t stream) {
    const int64_t plane = M * N;
    const int vec = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15u) == 0) &&
                    ((reinterpret_cast<uintptr_t>(partial) & 15u) == 0);
    int64_t blocks = (plane / (vec ? 4 : 1) + 255) / 256;
    if (blocks > static_cast<int64_t>(num_sms) * 8) blocks = static_cast<int64_t>(num_sms) * 8;
    if (blocks < 1) blocks = 1;
    splitk_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(partial, slices, plane, alpha,
                                                                             beta, C, vec);
    return launched(cudaGetLastError());
}

cudaError_t splitk_reduce_launch_h(const float* partial, int slices, int64_t M, int64_t N, float alpha,
                                   float beta, __half* C, int num_sms, cudaStream_t stream) {
    const int64_t plane = M * N;
    int64_t blocks = (plane + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    splitk_reduce_h_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(partial, slices, plane, alpha,
                                                                               beta, C);
    return launched(cudaGetLastError());
}

cudaError_t scale_c_h_launch(int64_t M, int64_t N, float beta, __half* C, cudaStream_t stream) {
    const int64_t n = M * N;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    scale_c_h_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(C, n, beta);
    return launched(cudaGetLastError());
}

cudaError_t transpose_f32_launch(const float* src, float* dst, int64_t rows, int64_t cols,
                                 cudaStream_t stream) {
    const int64_t gx = (cols + 31) / 32, gy = (rows + 31) / 32;
    if (gx * gy > 0x7FFFFFFF) return cudaErrorInvalidValue;
    transpose_f32_kernel<<<static_cast<unsigned>(gx * gy), 256, 0, stream>>>(src, dst, rows, cols, gx);
    return launched(cudaGetLastError());
}

int64_t debug_take_sgemm() { return debug_take_local(); }

bool sgemm_scalar_edge(int index, int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                       const float* C) {
    return sgemm_edge(index, M, N, K, A, B, C, N) == kEdgeScalar;
}

cudaError_t pad_copy_launch(const float* src, int64_t srows, int64_t scols, int64_t sld, float* dst, int64_t rows,
                            int64_t dcols, int num_sms, cudaStream_t stream) {
    const int64_t n4 = rows * (dcols / 4);
    if (n4 == 0) return cudaSuccess;
    int64_t blocks = (n4 + 255) / 256;
    if (blocks > static_cast<int64_t>(num_sms) * 8) blocks = static_cast<int64_t>(num_sms) * 8;
    pad_copy_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(src, srows, scols, sld,
                                                                        reinterpret_cast<float4*>(dst), rows, dcols / 4);
    return launched(cudaGetLastError());
}

cudaError_t scale_c_launch(int64_t M, int64_t N, float beta, float* C, cudaStream_t stream) {
    const int64_t n = M * N;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    scale_c_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(C, n, beta);
    return launched(cudaGetLastError());
}

}  // namespace phx
