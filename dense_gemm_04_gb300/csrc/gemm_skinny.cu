// gemm_skinny.cu -- C <- alpha * A @ B + beta * C when A has only a few rows.
//
// The matrix-multiplication lab's last sweep (Part 5, the skinny-matrix sweep) multiplies an
// M x K matrix by a K x N one with M from 1 up: the least traffic any kernel can have is
// each input read once and C written once, s (MK + KN + MN) bytes, so with M small the
// intensity 2MKN / s (MK + KN + MN) is about M / s FLOP per byte and the operation sits on
// the bandwidth roof, not the compute roof.  A GEMM tile of 128 or 256 rows would mostly
// multiply zeros, and the tensor-core path's rounding pass would write and re-read B, so
// this file streams B exactly once from HBM with 16-byte loads and does the arithmetic on
// the CUDA cores, where it is not the bottleneck:
//
//   - A CTA owns 128 columns of C (32 lanes x 4), up to 16 rows of A (MT) and a slice of K.
//     Its 8 warps share the slice in groups of U = 4 rows: warp w takes groups w, w + 8, ...
//   - Each warp streams its groups through its own ring of S slots in shared memory with
//     asynchronous copies (cp.async): a slot holds the group's U rows of B (16 bytes per
//     lane and row, so a warp's copy of a row is one 512-byte segment) and the U x MT values
//     of A they meet.  S - 1 groups are in flight while one is multiplied, without holding
//     registers, and copies past an edge write zeros.  Only the warp's own lanes touch its
//     ring, so the main loop needs no CTA barrier.  A may be given stored K x M.
//   - The grid is sized to one wave: enough slices of K for every SM, no more.  The slices
//     of one output tile form a thread-block cluster (up to 8 CTAs); after each CTA has
//     added its warps' sums in warp order, the cluster adds its CTAs' tiles in rank order
//     through distributed shared memory, each CTA finishing 1/8 of the tile.  Only when a
//     tile needs more than 8 slices do whole clusters write partial planes, which the
//     split-K reduction adds in plane order.  The order of every sum is fixed by the shape,
//     so results do not depend on timing.
//
// The f16 variant ("gemm on tensor cores", section "What changes") rounds every element of
// A and B to the nearest f16 (ties to even) as it is loaded; the product of two f16 values
// is exact in f32, so the f32 multiply-adds here compute the same rounded products summed
// in f32 as the tensor cores do, only in another order.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "debug_checks.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace phx {
namespace {

constexpr int kSkThreads = 256;
constexpr int kSkWarps = kSkThreads / 32;
constexpr int kSkBN = 128;          // columns per CTA
constexpr int kSkMaxCluster = 8;    // portable cluster size
constexpr int kSkU = 4;             // B rows per group
constexpr int kSkStages = 5;        // ring slots per warp

// Floats of one ring slot: U rows x 128 columns of B, then U x MT values of A.
__host__ __device__ constexpr int sk_slot(int mt) { return kSkU * kSkBN + kSkU * mt; }

__host__ __device__ constexpr size_t sk_smem(int mt) {
    return static_cast<size_t>(kSkStages) * kSkWarps * sk_slot(mt) * 4;
}

__device__ __forceinline__ float round_f16(float x) { return __half2float(__float2half_rn(x)); }

// 16-byte asynchronous global -> shared copy (L2 only); with pred false it writes zeros and
// reads nothing.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const float* src, bool pred) {
    const int bytes = pred ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}

// 4-byte asynchronous global -> shared copy; with pred false it writes zero and reads nothing.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const float* src, bool pred) {
    const int bytes = pred ? 4 : 0;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ float ld_shared_cluster(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Grid: x = (tile, rank) with the cluster's ranks innermost (tile = column strip x row
// block of A, row blocks innermost so that CTAs sharing B rows run together); y = plane.
// The CTA's slice of K is slice = y * cs + rank, rows [slice * k_cta, +k_cta) clipped to K.
// Up to 8 rows a tile: 2 CTAs per SM.  16 rows: 1 CTA per SM, so that the 64 accumulators
// and the f32x2 operand pairs stay in registers (at 128 registers they spilled).
template <int MT, bool F16, bool VEC>
__global__ void __launch_bounds__(kSkThreads, MT > 8 ? 1 : 2) skinny_kernel(
    const float* __restrict__ A, const float* __restrict__ B, float* __restrict__ C, float* __restrict__ partial,
    int M, int64_t N, int K, int k_cta, int cs, int mchunks, int64_t strips, int a_trans, float alpha,
    float beta) {
    constexpr int U = kSkU;
    constexpr int S = kSkStages;
    constexpr int SLOT = sk_slot(MT);
    extern __shared__ float4 sk_smem4[];
    float* smem = reinterpret_cast<float*>(sk_smem4);  // [warps][S][SLOT]; after the loop: red
    float* red = smem;                                  // [warps][MT][128]; warp 0's part: the tile

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = cs > 1 ? static_cast<int>(ptx::cluster_ctarank()) : 0;
    const int64_t t = static_cast<int64_t>(blockIdx.x) / cs;
    const int mc = static_cast<int>(t % mchunks);
    const int64_t strip = t / mchunks;
    const int m0 = mc * MT;
    const int64_t n0 = strip * kSkBN;
    const int slice = static_cast<int>(blockIdx.y) * cs + rank;
    const int64_t k0 = static_cast<int64_t>(slice) * k_cta;
    const int kn = k0 >= K ? 0 : static_cast<int>(K - k0 < k_cta ? K - k0 : k_cta);

    float* ring = smem + warp * S * SLOT;
    const int64_t col = n0 + 4 * lane;
    // this warp's groups: rows warp*U + g*8U (relative to k0), g < G
    const int first = warp * U;
    const int G = kn > first ? (kn - first + kSkWarps * U - 1) / (kSkWarps * U) : 0;

    // Enqueue group g into its slot (no copies past G: an empty commit group keeps the count).
    auto issue = [&](int g) {
        if (g < G) {
            float* slot = ring + (g % S) * SLOT;
            const int kb = first + g * kSkWarps * U;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t k = k0 + kb + u;
                const bool rk = kb + u < kn;
                const float* src = B + k * N + col;
                const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(slot + u * kSkBN + 4 * lane));
                if (VEC) {
                    cp_async_16(dst, rk && col < N ? src : B, rk && col < N);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const bool ok = rk && col + q < N;
                        cp_async_4(dst + 4 * q, ok ? src + q : B, ok);
                    }
                }
            }
            // A: U x MT values, slot layout [u][m]
            float* as = slot + U * kSkBN;
            for (int e = lane; e < U * MT; e += 32) {
                const int u = e / MT, m = e - u * MT;
                const int64_t k = k0 + kb + u;
                const bool ok = kb + u < kn && m0 + m < M;
                const float* src = !ok ? A : a_trans ? A + k * M + m0 + m : A + static_cast<int64_t>(m0 + m) * K + k;
                cp_async_4(static_cast<uint32_t>(__cvta_generic_to_shared(as + e)), src, ok);
            }
        }
        asm volatile("cp.async.commit_group;\n" ::: "memory");
    };

    // Accumulators in pairs for packed f32x2 multiply-adds (the same IEEE fma in each half):
    //   MT <= 8: acc[m][h] = columns (2h, 2h+1) of the lane's four, row m (pairs along N, each
    //            A value duplicated into a register pair);
    //   MT > 8:  acc[p][c] = rows (2p, 2p+1), column c (pairs along M: the A pairs come straight
    //            from the 16-byte loads, and only the four B values are duplicated).
    constexpr int AR = MT <= 8 ? MT : MT / 2;
    constexpr int AC = MT <= 8 ? 2 : 4;
    float2 acc[AR][AC];
#pragma unroll
    for (int i = 0; i < AR; ++i)
#pragma unroll
        for (int j = 0; j < AC; ++j) acc[i][j] = make_float2(0.f, 0.f);

#pragma unroll
    for (int g = 0; g < S - 1; ++g) issue(g);
    for (int g = 0; g < G; ++g) {
        asm volatile("cp.async.wait_group %0;\n" ::"n"(S - 2) : "memory");
        __syncwarp();  // every lane's copies of group g have landed; group g-1's reads are done
        const float* slot = ring + (g % S) * SLOT;
        float* as = const_cast<float*>(slot) + U * kSkBN;
        if (F16) {
            for (int e = lane; e < U * MT; e += 32) as[e] = round_f16(as[e]);
            __syncwarp();
        }
        issue(g + S - 1);  // into the slot group g-1 used
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float4 bq = reinterpret_cast<const float4*>(slot + u * kSkBN)[lane];
            if (F16) {
                bq.x = round_f16(bq.x);
                bq.y = round_f16(bq.y);
                bq.z = round_f16(bq.z);
                bq.w = round_f16(bq.w);
            }
            const float* ak = as + u * MT;
            float av[MT];
            if (MT >= 4) {
#pragma unroll
                for (int q = 0; q < MT / 4; ++q) {
                    const float4 a4 = reinterpret_cast<const float4*>(ak)[q];
                    av[4 * q + 0] = a4.x;
                    av[4 * q + 1] = a4.y;
                    av[4 * q + 2] = a4.z;
                    av[4 * q + 3] = a4.w;
                }
            } else {
#pragma unroll
                for (int m = 0; m < MT; ++m) av[m] = ak[m];
            }
            if constexpr (MT <= 8) {
                const float2 bxy = make_float2(bq.x, bq.y), bzw = make_float2(bq.z, bq.w);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float2 aa = make_float2(av[m], av[m]);
                    acc[m][0] = __ffma2_rn(aa, bxy, acc[m][0]);
                    acc[m][1] = __ffma2_rn(aa, bzw, acc[m][1]);
                }
            } else {
                const float2 bc[4] = {make_float2(bq.x, bq.x), make_float2(bq.y, bq.y), make_float2(bq.z, bq.z),
                                      make_float2(bq.w, bq.w)};
#pragma unroll
                for (int p = 0; p < MT / 2; ++p) {
                    const float2 aa = make_float2(av[2 * p], av[2 * p + 1]);
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[p][c] = __ffma2_rn(aa, bc[c], acc[p][c]);
                }
            }
        }
    }
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();  // every warp is done with its ring: red may overwrite it

    // the warps' sums, added in warp order into warp 0's part of red
#pragma unroll
    for (int m = 0; m < MT; ++m)
        reinterpret_cast<float4*>(red + (warp * MT + m) * kSkBN)[lane] =
            MT <= 8 ? make_float4(acc[m % AR][0].x, acc[m % AR][0].y, acc[m % AR][1].x, acc[m % AR][1].y)
                    : (m % 2 == 0 ? make_float4(acc[(m / 2) % AR][0].x, acc[(m / 2) % AR][1].x,
                                                acc[(m / 2) % AR][2 % AC].x, acc[(m / 2) % AR][3 % AC].x)
                                  : make_float4(acc[(m / 2) % AR][0].y, acc[(m / 2) % AR][1].y,
                                                acc[(m / 2) % AR][2 % AC].y, acc[(m / 2) % AR][3 % AC].y));
    __syncthreads();
    constexpr int E = MT * kSkBN;
    for (int e = tid; e < E; e += kSkThreads) {
        float s = red[e];
#pragma unroll
        for (int w = 1; w < kSkWarps; ++w) s += red[w * E + e];
        red[e] = s;
    }

    // the cluster's tiles, added in rank order; rank r finishes elements [r E / cs, (r+1) E / cs)
    int e_begin = 0, e_end = E;
    if (cs > 1) {
        ptx::cluster_sync();
        e_begin = rank * E / cs;
        e_end = (rank + 1) * E / cs;
    } else {
        __syncthreads();
    }
    const uint32_t tile_addr = static_cast<uint32_t>(__cvta_generic_to_shared(red));
    for (int e = e_begin + tid; e < e_end; e += kSkThreads) {
        float s;
        if (cs > 1) {
            s = ld_shared_cluster(ptx::map_to_rank(tile_addr + 4u * e, 0));
            for (int q = 1; q < cs; ++q) s += ld_shared_cluster(ptx::map_to_rank(tile_addr + 4u * e, q));
        } else {
            s = red[e];
        }
        const int m = e / kSkBN, c = e - m * kSkBN;
        const int64_t n = n0 + c;
        const int mm = m0 + m;
        if (mm >= M || n >= N) continue;
        PHX_DCHECK(m < MT && cs <= 8);
        const int64_t idx = static_cast<int64_t>(mm) * N + n;
        if (partial != nullptr) {
            partial[static_cast<int64_t>(blockIdx.y) * M * N + idx] = s;
        } else {
            C[idx] = beta == 0.f ? alpha * s : fmaf(alpha, s, beta * C[idx]);
        }
    }
    // no CTA leaves while a peer may still read its tile
    if (cs > 1) ptx::cluster_sync();
}

using SkinnyFn = void (*)(const float*, const float*, float*, float*, int, int64_t, int, int, int, int,
                          int64_t, int, float, float);

template <int MT, bool F16>
SkinnyFn pick_vec(bool vec) {
    return vec ? skinny_kernel<MT, F16, true> : skinny_kernel<MT, F16, false>;
}

template <bool F16>
SkinnyFn pick(int mt, bool vec) {
    switch (mt) {
        case 1: return pick_vec<1, F16>(vec);
        case 2: return pick_vec<2, F16>(vec);
        case 4: return pick_vec<4, F16>(vec);
        case 8: return pick_vec<8, F16>(vec);
        default: return pick_vec<16, F16>(vec);
    }
}

size_t smem_for(int mt) {
    switch (mt) {
        case 1: return sk_smem(1);
        case 2: return sk_smem(2);
        case 4: return sk_smem(4);
        case 8: return sk_smem(8);
        default: return sk_smem(16);
    }
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Per device and kernel: the dynamic shared memory attribute is set once and the number
// of resident CTAs per SM measured once.
int prepared_occupancy(const void* fn, size_t smem) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, int> occ;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_pair(dev, fn);
    std::lock_guard<std::mutex> lock(mu);
    auto it = occ.find(key);
    if (it != occ.end()) return it->second;
    int blocks = 0;
    if (cudaFuncSetAttribute(key.second, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, key.second, kSkThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (blocks < 1) blocks = 1;
    occ.emplace(key, blocks);
    return blocks;
}

// Slices of K for `tiles` output tiles on `slots` resident CTAs: one wave, each slice at
// least `min_rows` long and a multiple of `align`, at most one cluster of 8 slices per tile
// once that gives every SM a CTA; beyond that the clusters of a tile write partial planes.
bool plan_slices(int64_t tiles, int64_t slots, int64_t K, int64_t min_rows, int64_t align, int num_sms, int* cs_out,
                 int* planes_out, int* k_cta_out) {
    int64_t slices = tiles >= slots ? 1 : slots / tiles;
    const int64_t by_k = cdiv(K, min_rows);
    if (slices > by_k) slices = by_k;
    if (slices > kSkMaxCluster && tiles * kSkMaxCluster >= num_sms) slices = kSkMaxCluster;
    if (slices < 1) slices = 1;
    const int64_t planes = cdiv(slices, kSkMaxCluster);
    const int64_t cs = cdiv(slices, planes);
    slices = cs * planes;
    const int64_t k_cta = cdiv(cdiv(K, slices), align) * align;
    if (k_cta > 0x7FFFFFFF || planes > 65535) return false;
    *cs_out = static_cast<int>(cs);
    *planes_out = static_cast<int>(planes);
    *k_cta_out = static_cast<int>(k_cta);
    return true;
}

struct SkinnyPlan {
    int mt = 1, mchunks = 1, cs = 1, planes = 1, k_cta = 1;
    int64_t strips = 1;
    size_t smem = 0;
    SkinnyFn fn = nullptr;
};

// One wave: tiles x slices <= SMs x resident CTAs, with at least one round of all warps'
// groups per slice, and no more than one cluster of 8 slices per tile once that gives every
// SM a CTA (each CTA keeps 2U rows of B in flight per thread, 64 KB, enough to stream at
// the HBM rate); beyond that the slices of a tile become planes of partial sums.
bool skinny_plan(int f16, int64_t M, int64_t N, int64_t K, const float* B, int num_sms, SkinnyPlan* p) {
    p->mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16;
    p->mchunks = static_cast<int>(cdiv(M, p->mt));
    p->strips = cdiv(N, kSkBN);
    const bool vec = N % 4 == 0 && (reinterpret_cast<uintptr_t>(B) & 15u) == 0;
    p->fn = f16 ? pick<true>(p->mt, vec) : pick<false>(p->mt, vec);
    p->smem = smem_for(p->mt);
    const int occ = prepared_occupancy(reinterpret_cast<const void*>(p->fn), p->smem);
    if (occ < 0) return false;
    return plan_slices(p->strips * p->mchunks, static_cast<int64_t>(num_sms) * occ, K,
                       static_cast<int64_t>(kSkWarps) * kSkU, 8, num_sms, &p->cs, &p->planes, &p->k_cta);
}

// ---------------------------------------------------------------------------------------
// B stored transposed (N x K, each output column one contiguous row of B): the layout of a
// weight matrix W in x @ W^T.  Every column is a dot product of one row of A with one row of
// W, both contiguous along k, so the CTA streams rows of W and reads A alongside:
//   - A CTA owns 32 columns (rows of W), up to 16 rows of A (MT) and a slice of K, which it
//     walks in chunks of 128.  A chunk of W (32 x 128) and of A (MT x 128) is one stage of
//     a CTA-wide cp.async ring (kNtStages deep, copies past an edge write zeros), and one
//     barrier per chunk makes it visible and frees the oldest slot.
//   - Warp w takes rows 4w .. 4w+3 of W; lane l takes k = 4l .. 4l+3 of every chunk (one
//     16-byte read per row), so each lane sums its own k's for the 4 x MT outputs, and the
//     32 lanes are added at the end with a butterfly of shuffles (a fixed order).
//   - The f16 variant rounds each element of W where it is used (every element is used by
//     one lane) and the A values in place once they land (all warps use them).
//   - The K slices of a tile are added through distributed shared memory in rank order, as
//     in the kernel above, or, past 8 slices, through partial planes.
//   - out_t: C (and the partial planes) stored transposed, N x M: output (m, n) at n * M + m.
//     With it the kernel also serves few columns against many rows: C = A @ B is
//     C^T = B^T @ A^T, a few-row product whose W is A itself, stored M x K.
// ---------------------------------------------------------------------------------------
constexpr int kNtRows = 32;    // rows of W (output columns) per CTA
constexpr int kNtKc = 128;     // k per chunk
constexpr int kNtStages = 4;   // chunks in the ring

__host__ __device__ constexpr int nt_stage_floats(int mt) { return (kNtRows + mt) * kNtKc; }

__host__ __device__ constexpr size_t nt_smem(int mt) {
    return static_cast<size_t>(kNtStages) * nt_stage_floats(mt) * 4 + static_cast<size_t>(mt) * kNtRows * 4;
}

template <int MT, bool F16, bool VEC>
__global__ void __launch_bounds__(kSkThreads, 2) skinny_nt_kernel(
    const float* __restrict__ A, const float* __restrict__ W, float* __restrict__ C, float* __restrict__ partial,
    int M, int N, int K, int k_cta, int cs, int mchunks, int strips, int a_trans, int out_t, float alpha,
    float beta) {
    constexpr int S = kNtStages;
    // A stored M x K with rows on 16-byte boundaries (the host passes a_trans = 2 for that)
    const bool a_vec = a_trans == 2;
    if (a_vec) a_trans = 0;
    constexpr int SF = nt_stage_floats(MT);
    constexpr int E = MT * kNtRows;
    extern __shared__ float4 nt_smem4[];
    float* ring = reinterpret_cast<float*>(nt_smem4);  // [S][32 + MT][64]: rows of W, then of A
    float* tile = ring + S * SF;                        // [MT][32] sums of this CTA

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = cs > 1 ? static_cast<int>(ptx::cluster_ctarank()) : 0;
    const int t = static_cast<int>(blockIdx.x) / cs;
    const int mc = t % mchunks;
    const int strip = t / mchunks;
    const int m0 = mc * MT;
    const int n0 = strip * kNtRows;
    const int slice = static_cast<int>(blockIdx.y) * cs + rank;
    const int64_t k0 = static_cast<int64_t>(slice) * k_cta;
    const int kn = k0 >= K ? 0 : static_cast<int>(K - k0 < k_cta ? K - k0 : k_cta);
    const int chunks = (kn + kNtKc - 1) / kNtKc;

    // Enqueue chunk c into slot c % S: 16-byte copies of W rows (4-byte ones when W's rows are
    // not 16-byte aligned), 4-byte copies of A.  An empty commit group past the last chunk
    // keeps the group count.  (A thread's copies of A are the ones it rounds in place.)
    auto issue = [&](int c) {
        if (c < chunks) {
            float* st = ring + (c % S) * SF;
            const int kb = c * kNtKc;
            for (int e = tid; e < kNtRows * (kNtKc / 4); e += kSkThreads) {
                const int r = e / (kNtKc / 4), k4 = (e % (kNtKc / 4)) * 4;
                const int n = n0 + r;
                const float* src = W + static_cast<int64_t>(n) * K + k0 + kb + k4;
                const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(st + r * kNtKc + k4));
                if (VEC) {
                    const bool ok = n < N && kb + k4 < kn;  // kn and the k offsets are multiples of 4
                    cp_async_16(dst, ok ? src : W, ok);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const bool ok = n < N && kb + k4 + q < kn;
                        cp_async_4(dst + 4 * q, ok ? src + q : W, ok);
                    }
                }
            }
            float* as = st + kNtRows * kNtKc;
            if (a_vec) {
                // A stored M x K with 16-byte rows: 16-byte copies (kn is a multiple of 4 then)
                for (int e = tid; e < MT * (kNtKc / 4); e += kSkThreads) {
                    const int m = e / (kNtKc / 4), k4 = (e % (kNtKc / 4)) * 4;
                    const bool ok = m0 + m < M && kb + k4 < kn;
                    const float* src = ok ? A + static_cast<int64_t>(m0 + m) * K + k0 + kb + k4 : A;
                    cp_async_16(static_cast<uint32_t>(__cvta_generic_to_shared(as + m * kNtKc + k4)), src, ok);
                }
            } else {
                for (int e = tid; e < MT * kNtKc; e += kSkThreads) {
                    const int m = e / kNtKc, k = e % kNtKc;
                    const bool ok = m0 + m < M && kb + k < kn;
                    const int64_t gk = k0 + kb + k;
                    const float* src = !ok ? A : a_trans ? A + gk * M + m0 + m : A + static_cast<int64_t>(m0 + m) * K + gk;
                    cp_async_4(static_cast<uint32_t>(__cvta_generic_to_shared(as + e)), src, ok);
                }
            }
        }
        asm volatile("cp.async.commit_group;\n" ::: "memory");
    };

    float acc[4][MT];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;

#pragma unroll
    for (int c = 0; c < S - 1; ++c) issue(c);
    for (int c = 0; c < chunks; ++c) {
        asm volatile("cp.async.wait_group %0;\n" ::"n"(S - 2) : "memory");
        if (F16) {
            // round, in place, the A values this thread copied (the same index sets as issue:
            // only a thread's own copies are known to have landed before the barrier)
            float* as = ring + (c % S) * SF + kNtRows * kNtKc;
            if (a_vec) {
                for (int e = tid; e < MT * (kNtKc / 4); e += kSkThreads) {
                    float4* p4 = reinterpret_cast<float4*>(as + (e / (kNtKc / 4)) * kNtKc + (e % (kNtKc / 4)) * 4);
                    float4 v = *p4;
                    v.x = round_f16(v.x);
                    v.y = round_f16(v.y);
                    v.z = round_f16(v.z);
                    v.w = round_f16(v.w);
                    *p4 = v;
                }
            } else {
                for (int e = tid; e < MT * kNtKc; e += kSkThreads) as[e] = round_f16(as[e]);
            }
        }
        __syncthreads();  // chunk c visible to all; chunk c-1's slot is free
        issue(c + S - 1);
        const float* st = ring + (c % S) * SF;
        float4 w4[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            w4[r] = reinterpret_cast<const float4*>(st + (4 * warp + r) * kNtKc)[lane];
            if (F16) {
                w4[r].x = round_f16(w4[r].x);
                w4[r].y = round_f16(w4[r].y);
                w4[r].z = round_f16(w4[r].z);
                w4[r].w = round_f16(w4[r].w);
            }
        }
        const float* as = st + kNtRows * kNtKc;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const float4 a4 = reinterpret_cast<const float4*>(as + m * kNtKc)[lane];
#pragma unroll
            for (int r = 0; r < 4; ++r)
                acc[r][m] = fmaf(a4.w, w4[r].w, fmaf(a4.z, w4[r].z, fmaf(a4.y, w4[r].y, fmaf(a4.x, w4[r].x, acc[r][m]))));
        }
    }
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");

    // the 32 lanes' sums: a butterfly, so every lane ends with every total
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float v = acc[r][m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[r][m] = v;
        }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) tile[m * kNtRows + 4 * warp + r] = acc[r][m];
    }

    int e_begin = 0, e_end = E;
    if (cs > 1) {
        ptx::cluster_sync();
        e_begin = rank * E / cs;
        e_end = (rank + 1) * E / cs;
    } else {
        __syncthreads();
    }
    const uint32_t tile_addr = static_cast<uint32_t>(__cvta_generic_to_shared(tile));
    for (int e = e_begin + tid; e < e_end; e += kSkThreads) {
        float v;
        if (cs > 1) {
            v = ld_shared_cluster(ptx::map_to_rank(tile_addr + 4u * e, 0));
            for (int q = 1; q < cs; ++q) v += ld_shared_cluster(ptx::map_to_rank(tile_addr + 4u * e, q));
        } else {
            v = tile[e];
        }
        const int m = e / kNtRows, cidx = e % kNtRows;
        const int mm = m0 + m, n = n0 + cidx;
        if (mm >= M || n >= N) continue;
        PHX_DCHECK(m < MT && cs <= 8);
        const int64_t idx = out_t ? static_cast<int64_t>(n) * M + mm : static_cast<int64_t>(mm) * N + n;
        if (partial != nullptr)
            partial[static_cast<int64_t>(blockIdx.y) * M * N + idx] = v;
        else
            C[idx] = beta == 0.f ? alpha * v : fmaf(alpha, v, beta * C[idx]);
    }
    if (cs > 1) ptx::cluster_sync();
}

using SkinnyNtFn = void (*)(const float*, const float*, float*, float*, int, int, int, int, int, int, int, int,
                            int, float, float);

template <int MT, bool F16>
SkinnyNtFn pick_nt_vec(bool vec) {
    return vec ? skinny_nt_kernel<MT, F16, true> : skinny_nt_kernel<MT, F16, false>;
}

template <bool F16>
SkinnyNtFn pick_nt(int mt, bool vec) {
    switch (mt) {
        case 1: return pick_nt_vec<1, F16>(vec);
        case 2: return pick_nt_vec<2, F16>(vec);
        case 4: return pick_nt_vec<4, F16>(vec);
        case 8: return pick_nt_vec<8, F16>(vec);
        default: return pick_nt_vec<16, F16>(vec);
    }
}

struct SkinnyNtPlan {
    int mt = 1, mchunks = 1, cs = 1, planes = 1, k_cta = 1, strips = 1;
    size_t smem = 0;
    SkinnyNtFn fn = nullptr;
};

bool skinny_nt_plan(int f16, int64_t M, int64_t N, int64_t K, const float* W, int num_sms, SkinnyNtPlan* p) {
    if (M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF) return false;
    p->mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16;
    p->mchunks = static_cast<int>(cdiv(M, p->mt));
    const int64_t strips = cdiv(N, kNtRows);
    if (strips * p->mchunks > 0x7FFFFFFF / kSkMaxCluster) return false;
    p->strips = static_cast<int>(strips);
    const bool vec = K % 4 == 0 && (reinterpret_cast<uintptr_t>(W) & 15u) == 0;
    p->fn = f16 ? pick_nt<true>(p->mt, vec) : pick_nt<false>(p->mt, vec);
    switch (p->mt) {
        case 1: p->smem = nt_smem(1); break;
        case 2: p->smem = nt_smem(2); break;
        case 4: p->smem = nt_smem(4); break;
        case 8: p->smem = nt_smem(8); break;
        default: p->smem = nt_smem(16); break;
    }
    const int occ = prepared_occupancy(reinterpret_cast<const void*>(p->fn), p->smem);
    if (occ < 0) return false;
    return plan_slices(strips * p->mchunks, static_cast<int64_t>(num_sms) * occ, K, 2 * kNtKc, kNtKc, num_sms,
                       &p->cs, &p->planes, &p->k_cta);
}

}  // namespace

size_t skinny_workspace_bytes(int f16, int64_t M, int64_t N, int64_t K, const float* B, int num_sms) {
    SkinnyPlan p;
    if (!skinny_plan(f16, M, N, K, B, num_sms, &p)) return 0;
    return p.planes > 1 ? static_cast<size_t>(p.planes) * static_cast<size_t>(M * N) * 4 : 0;
}

cudaError_t skinny_launch(int f16, int a_trans, int64_t M, int64_t N, int64_t K, float alpha,
                          const float* A, const float* B, float beta, float* C, void* workspace,
                          int num_sms, cudaStream_t stream) {
    SkinnyPlan p;
    if (!skinny_plan(f16, M, N, K, B, num_sms, &p)) return cudaErrorInvalidValue;
    if (p.planes > 1 && workspace == nullptr) return cudaErrorInvalidValue;
    const int64_t gx = p.strips * p.mchunks * p.cs;
    if (gx > 0x7FFFFFFF || p.planes > 65535 || M > 0x7FFFFFFF || K > 0x7FFFFFFF) return cudaErrorInvalidValue;
    float* partial = p.planes > 1 ? static_cast<float*>(workspace) : nullptr;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(p.planes), 1);
    cfg.blockDim = dim3(kSkThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err = cudaLaunchKernelEx(&cfg, p.fn, A, B, C, partial, static_cast<int>(M), N, static_cast<int>(K),
                                         p.k_cta, p.cs, p.mchunks, p.strips, a_trans ? 1 : 0, alpha, beta);
    err = launched(err);
    if (err != cudaSuccess || p.planes == 1) return err;
    return splitk_reduce_launch(partial, p.planes, M, N, alpha, beta, C, num_sms, stream);
}

size_t skinny_nt_workspace_bytes(int f16, int64_t M, int64_t N, int64_t K, const float* W, int num_sms) {
    SkinnyNtPlan p;
    if (!skinny_nt_plan(f16, M, N, K, W, num_sms, &p)) return 0;
    return p.planes > 1 ? static_cast<size_t>(p.planes) * static_cast<size_t>(M * N) * 4 : 0;
}

cudaError_t skinny_nt_launch(int f16, int a_trans, int64_t M, int64_t N, int64_t K, float alpha,
                             const float* A, const float* W, float beta, float* C, void* workspace,
                             int num_sms, cudaStream_t stream, int out_t) {
    SkinnyNtPlan p;
    if (!skinny_nt_plan(f16, M, N, K, W, num_sms, &p)) return cudaErrorInvalidValue;
    if (p.planes > 1 && workspace == nullptr) return cudaErrorInvalidValue;
    float* partial = p.planes > 1 ? static_cast<float*>(workspace) : nullptr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.strips) * p.mchunks * p.cs, static_cast<unsigned>(p.planes), 1);
    cfg.blockDim = dim3(kSkThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // a_trans = 2: A stored M x K with 16-byte aligned rows, copied 16 bytes at a time
    const int a_mode = a_trans ? 1 : (K % 4 == 0 && (reinterpret_cast<uintptr_t>(A) & 15u) == 0) ? 2 : 0;
    cudaError_t err = cudaLaunchKernelEx(&cfg, p.fn, A, W, C, partial, static_cast<int>(M), static_cast<int>(N),
                                         static_cast<int>(K), p.k_cta, p.cs, p.mchunks, p.strips, a_mode,
                                         out_t ? 1 : 0, alpha, beta);
    err = launched(err);
    if (err != cudaSuccess || p.planes == 1) return err;
    return splitk_reduce_launch(partial, p.planes, M, N, alpha, beta, C, num_sms, stream);
}

int64_t debug_take_skinny() { return debug_take_local(); }

}  // namespace phx
