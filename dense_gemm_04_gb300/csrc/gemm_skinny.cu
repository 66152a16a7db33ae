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
template <int MT, bool F16, bool VEC>
__global__ void __launch_bounds__(kSkThreads, 2) skinny_kernel(
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

    float2 acc[MT][2];  // columns (0, 1) and (2, 3) of the lane's four
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = make_float2(0.f, 0.f);

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
            if (MT <= 8) {
                // packed f32x2 multiply-adds: the same IEEE fma in each lane, half the issue
                // slots (with 16 rows the register pairs they need would spill)
                const float2 bxy = make_float2(bq.x, bq.y), bzw = make_float2(bq.z, bq.w);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float2 aa = make_float2(av[m], av[m]);
                    acc[m][0] = __ffma2_rn(aa, bxy, acc[m][0]);
                    acc[m][1] = __ffma2_rn(aa, bzw, acc[m][1]);
                }
            } else {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    acc[m][0].x = fmaf(av[m], bq.x, acc[m][0].x);
                    acc[m][0].y = fmaf(av[m], bq.y, acc[m][0].y);
                    acc[m][1].x = fmaf(av[m], bq.z, acc[m][1].x);
                    acc[m][1].y = fmaf(av[m], bq.w, acc[m][1].y);
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
            make_float4(acc[m][0].x, acc[m][0].y, acc[m][1].x, acc[m][1].y);
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
int prepared_occupancy(SkinnyFn fn, size_t smem) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, int> occ;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_pair(dev, reinterpret_cast<const void*>(fn));
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
    const int occ = prepared_occupancy(p->fn, p->smem);
    if (occ < 0) return false;
    const int64_t slots = static_cast<int64_t>(num_sms) * occ;
    const int64_t tiles = p->strips * p->mchunks;
    const int64_t min_rows = static_cast<int64_t>(kSkWarps) * kSkU;
    int64_t slices = tiles >= slots ? 1 : slots / tiles;
    const int64_t by_k = cdiv(K, min_rows);
    if (slices > by_k) slices = by_k;
    // one cluster per tile already gives every SM a CTA: no partial planes
    if (slices > kSkMaxCluster && tiles * kSkMaxCluster >= num_sms) slices = kSkMaxCluster;
    if (slices < 1) slices = 1;
    const int64_t planes = cdiv(slices, kSkMaxCluster);
    const int64_t cs = cdiv(slices, planes);
    slices = cs * planes;
    const int64_t k_cta = cdiv(cdiv(K, slices), 8) * 8;
    if (k_cta > 0x7FFFFFFF) return false;
    p->cs = static_cast<int>(cs);
    p->planes = static_cast<int>(planes);
    p->k_cta = static_cast<int>(k_cta);
    return true;
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
    if (err != cudaSuccess || p.planes == 1) return err;
    return splitk_reduce_launch(partial, p.planes, M, N, alpha, beta, C, num_sms, stream);
}

}  // namespace phx
