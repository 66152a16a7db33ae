// internal.h -- declarations shared by the translation units of libphx (not installed).
//
// The C ABI lives in include/phx.h; this header is the contract between phx_api.cu (argument
// checks, dispatch, configuration, tuning) and the kernel files sgemm_simt.cu,
// gemm_f16tc.cu and probes.cu.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace phx {

// Kernels this thread has enqueued through the library so far: every launch site adds its
// successful launches, and the event profile counts kernels per call from the difference.
void note_launches(int n);
int64_t noted_launches();

// cudaFuncSetAttribute(fn, attr, value) on the current device, once per (device, fn, attr,
// value): function attributes live with the device's context, so later calls skip the
// runtime call (phx_api.cu).
cudaError_t set_func_attr_once(const void* fn, cudaFuncAttribute attr, int value);

// Failed index checks of the bounds-checked build (-DPHX_DEBUG=1) in each translation unit's
// kernels since the last call, read and cleared (-1 if the read failed); always 0 otherwise.
int64_t debug_take_sgemm();
int64_t debug_take_f16tc();
int64_t debug_take_f16cvt();
int64_t debug_take_skinny();

// `err` of a kernel launch, noted as one launch when it succeeded.
inline cudaError_t launched(cudaError_t err) {
    if (err == cudaSuccess) note_launches(1);
    return err;
}

// Status codes written into the per-device status word by kernels (0 = nothing to report).
enum DeviceStatus : unsigned int {
    kDevOk = 0,
    kDevTimeout = 1,
};

// ---------------------------------------------------------------------------------------
// f32 SIMT GEMM (sgemm_simt.cu)
// ---------------------------------------------------------------------------------------
struct SgemmConfig {
    int tile_m, tile_n, tile_k, stages, fma2;
};

int sgemm_num_configs();
const SgemmConfig& sgemm_config(int index);

// True if the aligned (unmasked, 16-byte vector) kernel of config `index` may run on this
// problem: every dimension a whole number of tiles and A, B, C 16-byte aligned.
bool sgemm_is_aligned(int index, int64_t M, int64_t N, int64_t K, const float* A,
                      const float* B, const float* C);

// Scratch bytes config `index` uses for this problem on `num_sms` SMs: the partial
// products of the K slices when a grid too small for the GPU is split along K (0 if not).
size_t sgemm_workspace_bytes(int index, int64_t M, int64_t N, int64_t K, const float* A,
                             const float* B, const float* C, int num_sms, int64_t ldb = -1);

// Enqueue config `index` (the aligned kernel when sgemm_is_aligned; else the kernel with
// 16-byte edge copies when K % 4 == ldb % 4 == 0 and A, B are 16-byte aligned, which stores C
// 16 bytes at a time when N % 4 == 0 and C is 16-byte aligned and 4 bytes at a time otherwise;
// else the one with 4-byte edge copies).  B's rows are ldb floats apart (ldb = -1: N; a
// larger ldb for B in a padded copy, whose columns past N must be zero).  When sgemm_workspace_bytes is not 0 and `workspace` holds that
// many bytes, the last partial wave (or a grid of less than one wave) is spread as stream-K
// blocks and then fixed up, or a small grid is split along K and then reduced; with
// workspace == nullptr the grid runs as tiles only.
// Requires M, N > 0, K > 0 and alpha != 0 (the caller handles the degenerate cases).
cudaError_t sgemm_launch(int index, int64_t M, int64_t N, int64_t K, float alpha,
                         const float* A, const float* B, float beta, float* C, void* workspace,
                         int num_sms, cudaStream_t stream, int64_t ldb = -1);

// True if config `index` on this problem would copy operands 4 bytes at a time (rows of A or
// B not 16-byte aligned: K % 4 != 0, N % 4 != 0, or an unaligned base).
bool sgemm_scalar_edge(int index, int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                       const float* C);

// dst (rows x dcols, row-major, dcols % 4 == 0, 16-byte aligned) <- src (srows x scols, rows
// sld floats apart) with zeros past srows and scols: a copy of an operand whose rows start on
// 16 bytes.
cudaError_t pad_copy_launch(const float* src, int64_t srows, int64_t scols, int64_t sld, float* dst, int64_t rows,
                            int64_t dcols, int num_sms, cudaStream_t stream);

// Host check of the f32 GEMM's schedule for config `index` with `per_sm` CTAs per SM on
// `num_sms` SMs (no device involved): out[0] tiles that run whole (all of them without a
// stream-K part; each split into out[3] slices when the grid is split along K), out[1]
// stream-K blocks, out[2] their k tiles, out[3] K slices of a grid split along K (1: none),
// out[4] the most tile segments one stream-K block writes, out[5] 1 if, for every spread
// tile, the slots the fix-up reads are, in k order, exactly the segments the blocks write
// for it and those cover its k tiles once, else 0.
void sgemm_schedule_selftest(int index, int64_t M, int64_t N, int64_t K, int per_sm, int num_sms, int64_t out[6]);

// C <- alpha * (P[0] + ... + P[slices-1]) + beta * C, where P[s] is the s-th M x N plane of
// `partial`, added in that order (beta == 0: C not read).  Finishes a GEMM split along K.
cudaError_t splitk_reduce_launch(const float* partial, int slices, int64_t M, int64_t N, float alpha,
                                 float beta, float* C, int num_sms, cudaStream_t stream);

// The same reduction into an f16 C: C <- round_f16(alpha * sum + beta * C).
cudaError_t splitk_reduce_launch_h(const float* partial, int slices, int64_t M, int64_t N, float alpha,
                                   float beta, __half* C, int num_sms, cudaStream_t stream);

// C <- beta * C for an f16 C (beta == 0: zeros without reading C), rounded to nearest even.
cudaError_t scale_c_h_launch(int64_t M, int64_t N, float beta, __half* C, cudaStream_t stream);

// dst (cols x rows) <- the transpose of src (rows x cols), both row-major f32.
cudaError_t transpose_f32_launch(const float* src, float* dst, int64_t rows, int64_t cols,
                                 cudaStream_t stream);

// ---------------------------------------------------------------------------------------
// Few rows of A (gemm_skinny.cu): B streamed once, CUDA-core arithmetic, both precisions
// ---------------------------------------------------------------------------------------
// Scratch bytes skinny_launch needs for this problem (the partial planes of its K slices;
// 0 when it does not split K).
size_t skinny_workspace_bytes(int f16, int64_t M, int64_t N, int64_t K, const float* B, int num_sms);

// C <- alpha * op(A) @ B + beta * C for M, N, K > 0 and alpha != 0, A in blocks of 16 rows
// (meant for few rows: every block re-reads B, from L2 when it can); with f16
// both operands are rounded to f16 (ties to even) as they are loaded.  a_trans: A stored
// K x M.  `workspace` holds skinny_workspace_bytes bytes (may be null when that is 0).
cudaError_t skinny_launch(int f16, int a_trans, int64_t M, int64_t N, int64_t K, float alpha,
                          const float* A, const float* B, float beta, float* C, void* workspace,
                          int num_sms, cudaStream_t stream);

// The same with B stored transposed as W (N x K): C <- alpha * op(A) @ W^T + beta * C.
// out_t: C stored transposed (N x M, output (m, n) at n * M + m).
size_t skinny_nt_workspace_bytes(int f16, int64_t M, int64_t N, int64_t K, const float* W, int num_sms);
cudaError_t skinny_nt_launch(int f16, int a_trans, int64_t M, int64_t N, int64_t K, float alpha,
                             const float* A, const float* W, float beta, float* C, void* workspace,
                             int num_sms, cudaStream_t stream, int out_t = 0);

// C <- beta * C (beta == 0: C <- 0 without reading C).  Used for K == 0 or alpha == 0.
cudaError_t scale_c_launch(int64_t M, int64_t N, float beta, float* C, cudaStream_t stream);

// ---------------------------------------------------------------------------------------
// f16 tensor-core GEMM with f32 accumulation (gemm_f16tc.cu)
// ---------------------------------------------------------------------------------------
struct F16Config {
    int tile_m, tile_n, tile_k, stages;
    int cluster;        // 1: one CTA per 128-row tile; 2: CTA pairs running the 2-SM MMA (TILE_M = 256)
    int convert_a = 0;  // 1: A rounded to f16 inside the GEMM kernel (gemm_f16cvt.cu)
    int convert_b = 0;  // 1: B rounded to f16 inside the GEMM kernel (gemm_f16cvt.cu)
};

// The f16 configurations: the kernel of gemm_f16tc.cu (indices 0 .. n-1), then the kernel
// that rounds A or B itself (gemm_f16cvt.cu; f16tc_is_convert_a / _b).
int f16tc_num_configs();
const F16Config& f16tc_config(int index);
bool f16tc_is_convert_a(int index);
bool f16tc_is_convert_b(int index);
inline bool f16tc_is_convert(int index) { return f16tc_is_convert_a(index) || f16tc_is_convert_b(index); }

// Tensor map of a K-major f16 operand: `rows` rows of `Kp` halves (a multiple of 8), `ld`
// halves apart, read in 128-byte-swizzled boxes of 64 halves x box_rows (gemm_f16tc.cu).
bool f16_operand_map(CUtensorMap* map, const __half* ptr, int64_t rows, int64_t Kp, int box_rows, int64_t ld);

// Tensor map of a row-major f32 matrix (rows x cols, cols a multiple of 4, 16-byte aligned),
// read unswizzled in boxes of box_cols x box_rows; zeros past the edges (gemm_f16tc.cu).
bool f32_rows_map(CUtensorMap* map, const float* ptr, int64_t rows, int64_t cols, int box_cols, int box_rows);

// The kernel that rounds A or B itself (gemm_f16cvt.cu): its configurations, the scratch
// bytes of a CONVERT_B grid split along K (0 if not split), and one GEMM of configuration
// `index` (0 .. f16cvt_num_configs() - 1) on A (M x K f32) and B (K x N f32), row-major, with
// `other` the operand the kernel does not round, K-major f16 from the rounding pass (Bt,
// N x Kp, for CONVERT_A; Ah, M x Kp, for CONVERT_B), ld_other halves apart; split_ws holds
// the split's partial planes (nullptr: no split).  Launched as a programmatic dependent of
// the rounding pass.  Requires M, N, K > 0 and alpha != 0.
int f16cvt_num_configs();
const F16Config& f16cvt_config(int index);
size_t f16cvt_split_bytes(int index, int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t f16cvt_gemm_launch(int index, int64_t M, int64_t N, int64_t K, float alpha, float beta, float* C,
                               const float* A, const float* B, const __half* other, int64_t ld_other,
                               void* split_ws, unsigned int* status, int num_sms, cudaStream_t stream);

// Bytes of workspace for the rounded operands: A as M x Kp f16 and B transposed as
// N x Kp f16, Kp = K rounded up to a multiple of 8, each part 256-byte aligned.
size_t f16tc_workspace_bytes(int64_t M, int64_t N, int64_t K);

// Enqueue the cast pass: A -> rounded f16 A (M x Kp) and B -> rounded, transposed f16 B
// (N x Kp) in `workspace` (f16tc_workspace_bytes(M, N, K) bytes, 256-byte aligned).
cudaError_t f16tc_cast_launch(int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                              void* workspace, int num_sms, cudaStream_t stream);

// The general preparation pass: the K-major f16 operands Ah (M x Kp) and Bt (N x Kp) from A
// and B, which are f32 (rounded to nearest even) or, with in_f16, already f16 (copied).
// With trans_a, A is stored K x M; with trans_b, B is stored N x K.  A null Ah or Bt skips
// that operand (one the GEMM reads in place).
cudaError_t f16tc_prepare_launch(int in_f16, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                                 const void* A, const void* B, __half* Ah, __half* Bt, int num_sms,
                                 cudaStream_t stream);

// The same for operands given transposed: with trans_a, A is stored K x M; with trans_b, B
// is stored N x K.  The result in `workspace` is the same K-major pair.
cudaError_t f16tc_cast_launch_ex(int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                                 const float* A, const float* B, void* workspace, int num_sms,
                                 cudaStream_t stream);

// Scratch bytes config `index` uses on `num_sms` SMs for the partial products of the K
// slices when a grid too small for the GPU is split along K (0 if it is not split).
size_t f16tc_split_bytes(int index, int64_t M, int64_t N, int64_t K, int num_sms);

// Enqueue the tcgen05 GEMM of config `index` on the cast operands in `workspace`, split
// along K into `split_ws` (f16tc_split_bytes(...) bytes; nullptr: no split) and then
// reduced; `status` is the device status word; `num_sms` bounds the persistent grid.
// Requires M, N, K > 0 and alpha != 0.
cudaError_t f16tc_gemm_launch(int index, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                              float* C, const void* workspace, void* split_ws, unsigned int* status,
                              int num_sms, cudaStream_t stream);

// The GEMM on explicit K-major f16 operands: Ah (M rows, lda halves apart) and Bt (N rows,
// ldb apart), lda and ldb multiples of 8 and both 16-byte aligned.  The result goes to C
// (f32) or, when Ch is not null, to Ch (f16, alpha * acc + beta * c_old rounded once).
cudaError_t f16tc_gemm_launch_ops(int index, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                                  float* C, __half* Ch, const __half* Ah, int64_t lda, const __half* Bt,
                                  int64_t ldb, void* split_ws, unsigned int* status, int num_sms,
                                  cudaStream_t stream);

// One whole call of the f16 variant with configuration `cfg` (not the skinny kernel):
// the cast pass into `ws` and the tcgen05 GEMM (split along K into `ws` when the grid is too
// small for the GPU), both on `stream`; `ws` holds f16tc_run_bytes(...) bytes, 256-byte
// aligned.  The pooled and the allocation-free entry points both run this (phx_api.cu).
size_t f16tc_run_bytes(int cfg, int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t f16tc_run(int cfg, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K, float alpha,
                      const float* A, const float* B, float beta, float* C, void* ws, unsigned int* status,
                      int num_sms, cudaStream_t stream);

// The allocation-free entry point's status word on the current device (gemm_f16tc_noalloc.cu):
// copied to *word and cleared when that entry point has set up this device, else *word = 0.
cudaError_t noalloc_take_status(unsigned int* word);

// The configuration index a call of `variant` with this shape would use now (pinned, tuned
// or default), as phx_get_config reports it (phx_api.cu); kBadConfigPin when the variant's
// PHX_CONFIG_* environment pin does not parse (the call then returns PHX_ERR_CONFIG).
constexpr int kBadConfigPin = -2;
int choose_config_for(int variant, int64_t M, int64_t N, int64_t K, int sms);
// The skinny configuration's scratch and launch for a call (phx_api.cu): few rows of op(A),
// or few columns with A stored M x K (the transposed product on the kernel that streams
// rows).  f16 variant: both operands rounded to f16 as they are loaded.
size_t skinny_run_bytes(int variant, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K, const float* A,
                        const float* B, int num_sms);
cudaError_t skinny_run(int variant, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K, float alpha,
                       const float* A, const float* B, float beta, float* C, void* ws, int num_sms,
                       cudaStream_t stream);

// True if configuration `cfg` of `variant` is the skinny kernel rather than a GEMM tile.
bool is_skinny_config(int variant, int cfg);

// ---------------------------------------------------------------------------------------
// Probes and self-tests (probes.cu)
// ---------------------------------------------------------------------------------------
cudaError_t probe_ffma_launch(int packed, int64_t blocks, int iters, float* out,
                              cudaStream_t stream);
cudaError_t probe_stream_read_launch(const float* x, int64_t n, uint32_t* fold, int64_t blocks,
                                     cudaStream_t stream);
cudaError_t probe_mma_f16_launch(int64_t ctas, int iters, int n, float* sink,
                                 unsigned int* status, cudaStream_t stream);
cudaError_t selftest_wait_launch(uint64_t limit_ns, unsigned int* status,
                                 cudaStream_t stream);

}  // namespace phx
