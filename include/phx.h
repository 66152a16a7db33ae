/*
 * phx.h -- C ABI of libphx, a single-GPU GEMM library for GB300 (sm_103a).
 *
 * The one operation:   C <- alpha * A @ B + beta * C
 *
 * as stated in "gemm, f32" (phobos-lang.dev/docs/examples/gemm-fp32/): the kernel signature
 * gemm(A: tensor<f32>[M, K], B: tensor<f32>[K, N], C: tensor<f32>[M, N], alpha: f32,
 * beta: f32), section "The epilogue" (C is overwritten in place with alpha * acc +
 * beta * c_old), and in "gemm on tensor cores" (phobos-lang.dev/docs/examples/
 * gemm-fp16tc-fp32acc/), section "What changes" (operands rounded to f16, products summed
 * in f32).
 *
 * Conventions shared by every entry point below
 * ---------------------------------------------
 * Layout     A, B and C are row-major and contiguous: A is M x K with leading dimension K,
 *            B is K x N with leading dimension N, C is M x N with leading dimension N.
 *            Element (i, j) of C is C[i * N + j].  The _ex calls also take A or B stored
 *            transposed (see phx_op).
 * Pointers   A, B and C are DEVICE pointers (cudaMalloc, the caching allocator of a
 *            framework, managed memory) on the current device, 4-byte aligned, and not
 *            NULL whenever their matrix has at least one element.  The caller
 *            owns them; the library keeps no reference after the call.  C is read (unless
 *            beta == 0) and written in place.  A and B must not overlap C: an overlap is
 *            rejected with PHX_ERR_INVALID.  A and B may alias each other.
 * Stream     Work is enqueued on `stream` (NULL = the legacy default stream) and the call
 *            returns once it is enqueued; results are visible to later work on that
 *            stream.  The type phx_stream_t is cudaStream_t.
 * Sizes      M, N, K >= 0 and each below 2^31; M*K, K*N and M*N below 2^62.
 * Degenerate M == 0 or N == 0: nothing is read or written, PHX_OK.
 *            K == 0 or alpha == 0: A and B are not read and C <- beta * C.
 *            beta == 0: C is not read (NaN or Inf in C does not propagate), C <- alpha*A@B.
 * Errors     Arguments are checked before anything is launched; on an error return nothing
 *            was launched and no memory was touched.  The library never traps: a kernel
 *            whose internal wait runs out of time records PHX_ERR_TIMEOUT in a per-device
 *            status word and exits; phx_check_device_status() reports it.
 * Threads    Entry points may be called from several host threads; configuration pins
 *            and the tuning cache are process-wide and guarded by a lock.
 */
#ifndef PHX_H_
#define PHX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Every declaration below is part of the exported ABI, even when the library is built
 * with hidden default visibility. */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

typedef struct CUstream_st* phx_stream_t; /* identical to cudaStream_t */

typedef enum phx_status {
    PHX_OK = 0,
    PHX_ERR_INVALID = 1,  /* bad size, null or overlapping pointer, bad variant        */
    PHX_ERR_ARCH = 2,     /* no CUDA device, or the current device is not sm_103       */
    PHX_ERR_LAUNCH = 3,   /* a CUDA runtime call or a kernel launch failed             */
    PHX_ERR_TIMEOUT = 4,  /* a device-side bounded wait expired (see check_status)     */
    PHX_ERR_NOMEM = 5,    /* the f16 workspace could not be allocated                  */
    PHX_ERR_INTERNAL = 6, /* an invariant of the library itself failed                 */
    PHX_ERR_CONFIG = 7    /* config string unparsable or not among the compiled configs */
} phx_status;

/* Variants, for the configuration and tuning calls. */
enum { PHX_VARIANT_SGEMM = 0, PHX_VARIANT_F16TC = 1 };

/* ---------------------------------------------------------------------------------------
 * The GEMM calls
 * ------------------------------------------------------------------------------------- */

/* f32 GEMM on the CUDA cores ("gemm, f32", kernel listing and sections "One output tile
 * per CTA", "The k loop", "The epilogue").  Every product and sum is an f32 fused
 * multiply-add; the epilogue computes alpha * acc + beta * c_old in f32.  Tile-aligned
 * shapes with 16-byte aligned pointers take the aligned fast path, all others a masked
 * path (loads past an edge read zero, stores past an edge are skipped) that gives the
 * same result; the masked path keeps 16-byte copies when K % 4 == N % 4 == 0 and the
 * pointers are 16-byte aligned.
 * Two schedules use scratch taken, in stream order, from the library's pooled device
 * memory (PHX_ERR_NOMEM if that fails):
 *   - stream-K: the k steps of a last, partial wave of tiles -- or of a whole grid of less
 *     than one wave -- are shared evenly by one block per CTA slot, each writing partial
 *     tiles, which one more kernel adds in k order before applying the epilogue;
 *   - split-K: a grid too small to fill the GPU is split along K, each slice writing its
 *     partial products, which one more kernel adds in slice order.
 * The library picks between them and plain tiles by shape.  Either way the order of every
 * sum is fixed by the shape, so results do not depend on timing.  Other shapes allocate
 * nothing. */
phx_status phx_sgemm(int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                     const float* B, float beta, float* C, phx_stream_t stream);

/* f16 tensor cores with f32 accumulation ("gemm on tensor cores", section "What
 * changes"): every element of A and B is rounded to the nearest f16 (ties to even), the
 * f16 x f16 products are summed in f32 by tcgen05.mma into tensor memory, and the
 * epilogue computes alpha * acc + beta * c_old in f32.  The call's scratch -- the f16 copies
 * the rounding pass writes (at most phx_f16tc_workspace_bytes(M, N, K) bytes; none of an
 * operand the chosen configuration rounds itself) and, for a grid split along K, slices x
 * M x N x 4 bytes of f32 partial products -- is taken, in stream order, from a memory pool
 * the library owns for the current device, and returned to it after the GEMM
 * (PHX_ERR_NOMEM if that fails). */
phx_status phx_gemm_f16tc_f32acc(int64_t M, int64_t N, int64_t K, float alpha,
                                 const float* A, const float* B, float beta, float* C,
                                 phx_stream_t stream);

/* The same GEMM as phx_gemm_f16tc_f32acc for callers that cannot allocate device memory
 * while they run: code in a latency-critical loop that must never wait on an allocator (an
 * allocation can block, grow a pool or fail under memory pressure), or a plug-in whose host
 * application owns the whole device-memory budget.  The paper has no counterpart; this is
 * about this library's memory handling only.  Same arguments, rounding, kernels, schedule
 * and results (bit for bit, split-K included), but the scratch -- the f16 copies of A and B,
 * and the partial products of a grid split along K -- goes to one array of static device
 * memory inside the library, so the call allocates nothing:
 *   - Limit: the scratch of the call <= 64 MiB.  For shapes that do not split K that is
 *     phx_f16tc_workspace_bytes(M, N, K) (M = N = K = 4096 fits exactly); few rows of A need
 *     no copies, only the skinny kernel's partial sums.  A larger problem returns
 *     PHX_ERR_NOMEM before anything is launched.
 *   - Every GPU that loads this part of the library holds the 64 MiB until the process ends.
 *   - The first call on each device looks up the array's device address (once per device,
 *     with that device current); make that first call before any stream capture begins.
 *   - All calls share the array.  Calls whose GPU work overlaps (different streams, or no
 *     ordering between them) race and corrupt each other's results: keep them ordered.
 *     Nothing needs clearing between calls: each call rewrites all the scratch it reads.
 *   - A device-side wait that gives up records PHX_ERR_TIMEOUT in a status word inside that
 *     array; phx_check_device_status reads and clears it, like the pooled calls' word. */
phx_status phx_gemm_f16tc_f32acc_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                         const float* A, const float* B, float beta, float* C,
                                         phx_stream_t stream);

/* Storage order of an operand for the _ex calls, after the matrix-multiplication lab's
 * layout sweep (Part 5: the same products with A, B or both stored transposed).  The
 * product is always C (M x N) <- alpha * op(A) @ op(B) + beta * C with op(A) M x K and
 * op(B) K x N, both contiguous:
 *   PHX_OP_N   A stored M x K (A[i * K + k]);  B stored K x N (B[k * N + j]);
 *   PHX_OP_T   A stored K x M (A[k * M + i]);  B stored N x K (B[j * K + k]). */
typedef enum phx_op { PHX_OP_N = 0, PHX_OP_T = 1 } phx_op;

/* phx_sgemm with either operand stored transposed.  An operand given as PHX_OP_T is first
 * transposed into scratch taken, in stream order, from the library's pooled device memory
 * (M*K or K*N floats; PHX_ERR_NOMEM if that fails), then the same kernels run, so the
 * result is bit-identical to phx_sgemm on the transposed copy.  With PHX_OP_N for both
 * this is phx_sgemm.  An op outside {PHX_OP_N, PHX_OP_T} is PHX_ERR_INVALID. */
phx_status phx_sgemm_ex(phx_op op_a, phx_op op_b, int64_t M, int64_t N, int64_t K,
                        float alpha, const float* A, const float* B, float beta, float* C,
                        phx_stream_t stream);

/* phx_gemm_f16tc_f32acc with either operand stored transposed.  The rounding pass reads
 * each operand in its stored order and writes the same K-major f16 copies as for the plain
 * layout (a row-wise rounding for A as PHX_OP_N and B as PHX_OP_T, a tiled transposing
 * rounding for the other two), so no extra pass or workspace is needed and the result is
 * bit-identical to phx_gemm_f16tc_f32acc on op(A), op(B). */
phx_status phx_gemm_f16tc_f32acc_ex(phx_op op_a, phx_op op_b, int64_t M, int64_t N,
                                    int64_t K, float alpha, const float* A, const float* B,
                                    float beta, float* C, phx_stream_t stream);

/* An IEEE 754 binary16 value, as its bit pattern (the layout of __half and torch.float16). */
typedef uint16_t phx_f16;

/* Half-precision operands, after the matrix-multiplication lab's cuBLAS f16 GEMM (Part 4,
 * "precision", and Part 5): A and B are f16 already, so there is no rounding pass; the
 * f16 x f16 products are summed in f32 by tcgen05.mma exactly as in
 * phx_gemm_f16tc_f32acc, and the epilogue computes alpha * acc + beta * c_old in f32.
 *   phx_gemm_f16in_f32acc   C is f32 (M x N floats), as phx_gemm_f16tc_f32acc.
 *   phx_gemm_f16in_f16out   C is f16: c_old is read as f16 and alpha * acc + beta * c_old
 *                           is rounded to the nearest f16 (ties to even) once.  A grid split
 *                           along K adds its f32 partial sums first and rounds once too.
 * op_a / op_b give the storage order as for the _ex calls.  A, B (and an f16 C) must be
 * 2-byte aligned, an f32 C 4-byte aligned.  A stored M x K with K % 8 == 0 and 16-byte
 * alignment is read in place; otherwise it is copied into the K-major layout the tensor
 * cores read, and B always is (N x K halves, padded to a multiple of 8), in scratch taken in
 * stream order from the library's pooled device memory (PHX_ERR_NOMEM if that fails).  The
 * tile configuration is the f16 variant's (pins and tuning apply); where that is "SKINNY"
 * or a CONVERT_A=1 configuration, which read f32 operands, the default tile configuration
 * is used instead. */
phx_status phx_gemm_f16in_f32acc(phx_op op_a, phx_op op_b, int64_t M, int64_t N, int64_t K,
                                 float alpha, const phx_f16* A, const phx_f16* B, float beta,
                                 float* C, phx_stream_t stream);
phx_status phx_gemm_f16in_f16out(phx_op op_a, phx_op op_b, int64_t M, int64_t N, int64_t K,
                                 float alpha, const phx_f16* A, const phx_f16* B, float beta,
                                 phx_f16* C, phx_stream_t stream);

/* Bytes of the f16 copies the rounding pass of phx_gemm_f16tc_f32acc writes for this shape
 * when it rounds both operands: the rounded A (M rows) and the rounded, transposed B (N
 * rows), each row padded with zeros to a multiple of 8 halves, each part rounded up to 256
 * bytes.  That is the whole scratch of a call that neither splits K nor rounds an operand
 * inside the GEMM, and a bound on the copies of any call; a split along K takes its partial
 * products besides. */
phx_status phx_f16tc_workspace_bytes(int64_t M, int64_t N, int64_t K, size_t* bytes);

/* ---------------------------------------------------------------------------------------
 * Status
 * ------------------------------------------------------------------------------------- */

/* A static, human-readable name for a status code. */
const char* phx_status_string(phx_status s);

/* Synchronise `stream`, then read and clear the current device's status words -- the one
 * of the pooled entry points and the one inside phx_gemm_f16tc_f32acc_noalloc's static
 * array, each if that part of the library has run on this device: PHX_OK,
 * PHX_ERR_TIMEOUT if a kernel gave up a bounded wait since the last check, or
 * PHX_ERR_LAUNCH if the stream reported an error.  Allocates nothing. */
phx_status phx_check_device_status(phx_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * The bounds-checked build
 *
 * Built with PHX_DEBUG=1 (`python dense_gemm_04_gb300/build.py --debug` writes
 * _lib/libphx_debug.so; the binding loads it when the environment variable PHX_LIBRARY names
 * it), the kernels check their global-memory and shared-memory indices, tile coordinates and
 * tensor-memory columns as they go.  A failed check is counted in a device counter and the
 * kernel carries on (nothing traps; the kernel's own guards still decide what is accessed).
 * ------------------------------------------------------------------------------------- */

/* 1 if this library was built with the checks, else 0. */
int phx_debug_build(void);

/* Synchronise the current device, then write the number of failed checks since the last call
 * (0 in a library built without the checks) and clear it. */
phx_status phx_debug_violations(int64_t* count);

/* ---------------------------------------------------------------------------------------
 * Per-kernel timing, for roofline reports
 * ------------------------------------------------------------------------------------- */

/* Kernel kinds counted by the profile. */
enum { PHX_KIND_SGEMM = 0, PHX_KIND_F16_CAST = 1, PHX_KIND_TC_GEMM = 2, PHX_KIND_SCALE_C = 3,
       PHX_KIND_TRANSPOSE = 4, PHX_KIND_SKINNY = 5, PHX_NUM_KINDS = 6 };

/* Start a profile: from now on every GEMM call records CUDA events on its stream around
 * each kernel it launches (the f32 GEMM kernel; the f16 cast pass and the tensor-core GEMM
 * kernel separately; the C-scaling kernel of the degenerate cases).  Restarting discards the
 * previous marks. */
phx_status phx_profile_start(void);

/* Stop the profile: synchronise the recorded events and write, for each kind k in
 * [0, PHX_NUM_KINDS), the number of kernels launched[k] and their summed device time ms[k]
 * in milliseconds (one call may launch several kernels of its kind: a long f32 GEMM whose
 * last wave is spread as stream-K blocks launches those, the tiles and a fix-up; a grid
 * split along K adds its reduction).  Both arrays are caller-owned host arrays of
 * PHX_NUM_KINDS elements. */
phx_status phx_profile_stop(int64_t* launches, double* ms);

/* ---------------------------------------------------------------------------------------
 * Configurations and the autotuner
 *
 * A configuration is one compiled kernel shape, written as in "gemm, f32" section
 * "Tuning": "TILE_M=128 TILE_N=128 TILE_K=8 STAGES=4" (f32 variant; an optional
 * "FMA2=1" selects packed f32x2 multiply-adds) or "TILE_M=128 TILE_N=256 TILE_K=64
 * STAGES=4" (f16 variant).  The order of keys does not matter.  An f16 configuration
 * ending in "CONVERT_A=1" (TILE_M=128, TILE_N 64, 128 or 256) is the kernel that rounds A to
 * f16 itself as it stages A's f32 tiles, so that only B goes through the separate rounding
 * pass; it is the default where N <= 256 and A has 128-row tiles for at least half the SMs, or
 * M >= 1024, K >= 2048 and M * K >= 2^23 (K is then split to give every SM work).
 * One ending in "CONVERT_B=1" (TILE_M=128, TILE_N 64 or 128) rounds B itself the same way
 * (and splits K when its tiles cannot fill the SMs); it is the default for M <= 256, N >= 1024
 * and K * N >= 2^23.  One ending in "CONVERT_A=1 CONVERT_B=1" rounds both operands itself: one
 * launch, no rounding pass (the default for at most 2^25 multiply-adds).  All of them compute
 * the same rounded products, summed in f32 in the same order per tile.  An operand they round given transposed (op_a or op_b = PHX_OP_T), and the
 * half-precision entry points, take the default without them instead.  The last configuration of
 * each variant, "SKINNY", is the kernel for few rows of A (the lab's skinny-matrix sweep,
 * Part 5): B is streamed once from HBM with 16-byte loads and the products are summed with
 * f32 multiply-adds on the CUDA cores (for the f16 variant, of operands rounded to f16 as
 * they are loaded: the same rounded products, summed in f32).  It takes any M, in blocks
 * of 16 rows, and is the default for M <= 48 (f32) and M <= 16 (f16; M <= 8 where B has
 * 2^23 elements or more, N >= 1024, and the kernel that rounds B itself takes over).  For
 * f32 it is also the default for small problems (M <= 512 and M * N * K <= 2^27) and for
 * M <= 64 with K * N <= 2^22.  Few columns against many rows (M >= 1024 and N <= 16 for
 * f32, N <= 8 for f16), with A stored M x K, it runs as the transposed product
 * C^T = op(B)^T @ A^T, streaming A once and writing C^T transposed, which is C; that is the
 * default there when A has 2^22 elements or more (for f16 only up to 4 columns and 4096
 * rows, or an A below 2^23 elements, where the kernel that rounds A is slower).
 * ------------------------------------------------------------------------------------- */

/* Number of compiled configurations of a variant (or -1 for a bad variant). */
int phx_num_configs(int variant);

/* Canonical name of configuration `index` of `variant`, NUL-terminated in buf. */
phx_status phx_config_name(int variant, int index, char* buf, size_t buflen);

/* Pin one configuration for every later call of `variant` (spec as above), bypassing the
 * tuned and default choices; spec == NULL or "" removes the pin.  PHX_ERR_CONFIG if the
 * spec does not parse or names no compiled configuration. */
phx_status phx_set_config(int variant, const char* spec);

/* Name of the configuration a call of `variant` with this shape would use now. */
phx_status phx_get_config(int variant, int64_t M, int64_t N, int64_t K, char* buf,
                          size_t buflen);

/* Name of the configuration the last GEMM call of `variant` launched ("NONE" before the
 * first), for reports: phx_sgemm and phx_sgemm_ex for the f32 variant; phx_gemm_f16tc_f32acc,
 * its _ex form and the half-precision entry points for the f16 variant.  Degenerate calls
 * that launch no GEMM do not count. */
phx_status phx_last_config(int variant, char* buf, size_t buflen);

/* Tune `variant` for the shape (M, N, K), following "gemm, f32" section "Tuning":
 * stage 1 times every configuration briefly on scratch inputs and skips any that fails;
 * stage 2 runs the fastest `finalists` for `settle_ms` milliseconds to settle the clocks,
 * then times them over `rounds` rounds, one launch each per round in a freshly shuffled
 * order, and keeps the configuration with the lowest median.  The result goes into the
 * process-wide tuning cache, which later calls with this exact shape consult.  Scratch
 * inputs are allocated and freed inside the call; the call synchronises `stream`. */
phx_status phx_autotune(int variant, int64_t M, int64_t N, int64_t K, int finalists,
                        int rounds, int settle_ms, phx_stream_t stream);

/* The tuning cache is keyed by device as well as by variant and shape: a device's tag is
 * its name with spaces as underscores, a colon and its SM count ("NVIDIA_GB300:152"; "none"
 * without a device), and a tuned configuration is only used on a device with the tag it was
 * tuned on.  phx_device_tag writes the current device's tag to buf. */
phx_status phx_device_tag(char* buf, size_t buflen);

/* Save the tuning cache to a text file, one line per entry ("<tag> <variant> <M> <N> <K>
 * <configuration>"), or merge one in (PHX_ERR_CONFIG if a line does not parse; nothing is
 * merged then).  With the environment variable PHX_TUNE_CACHE=<path>, the first call of the
 * process merges that file in (if it exists) and every phx_autotune rewrites it. */
phx_status phx_tune_cache_save(const char* path);
phx_status phx_tune_cache_load(const char* path);

/* The record of the last phx_autotune of `variant`: the device, the shape, the pick, and
 * one line per finalist with the median of its second-stage timings and the median SM clock
 * read (through NVML queries; -1 where NVML is unavailable) right after each of them, as
 * NUL-terminated text ("NONE" before any tuning). */
phx_status phx_autotune_report(int variant, char* buf, size_t buflen);

/* ---------------------------------------------------------------------------------------
 * Roof probes: the two roofs of the matrix-multiplication lab's Part 1 (the FP32
 * multiply-add rate and the memory read rate), measured with kernels designed for sm_103a;
 * used for the denominators of the roofline.
 * ------------------------------------------------------------------------------------- */

/* FP32 multiply-add probe: `blocks` CTAs of 256 threads; each thread keeps 12 independent
 * recurrences x <- x * rho + tau in registers for `iters` iterations (packed = 1: the same
 * recurrences two per f32x2 instruction).  Floating-point operations performed:
 * blocks * 256 * iters * 24, packed or not.  `out` (device, blocks * 256 floats) receives
 * one value per thread, in [0.5, 1). */
phx_status phx_probe_ffma(int packed, int64_t blocks, int iters, float* out,
                          phx_stream_t stream);

/* HBM read probe: reads n floats of x (device, 16-byte aligned, n % 4 == 0; 4 * n bytes)
 * with `blocks` CTAs of 256 threads, each CTA one contiguous slice.  `fold` (device,
 * `blocks` 32-bit words) receives, per CTA, the XOR of every 32-bit word of its slice: the
 * XOR of all `blocks` words equals the XOR of every word of x, which proves the read. */
phx_status phx_probe_stream_read(const float* x, int64_t n, uint32_t* fold, int64_t blocks,
                                 phx_stream_t stream);

/* Tensor-core probe: `ctas` CTAs each issue `iters` rounds of 4 tcgen05.mma kind::f16
 * (M = 128, N = n, K = 16, f32 accumulate) on shared-memory operands, with no global
 * traffic.  Floating-point operations: ctas * iters * 4 * 2 * 128 * n * 16.  n is 64, 128
 * or 256.  `sink` (device, ctas floats) receives one accumulator value per CTA. */
phx_status phx_probe_mma_f16(int64_t ctas, int iters, int n, float* sink,
                             phx_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Self-tests of host and device machinery that cannot be reached through a correct GEMM.
 * ------------------------------------------------------------------------------------- */

/* Launch one CTA whose thread waits on a shared-memory mbarrier that nothing ever
 * arrives at, with a limit of `limit_ns` nanoseconds (clamped to [1e3, 1e9]).  The wait
 * gives up, records PHX_ERR_TIMEOUT in the status word and the kernel exits normally;
 * phx_check_device_status() then returns PHX_ERR_TIMEOUT.  No fault, trap or hang. */
phx_status phx_selftest_bounded_wait(uint64_t limit_ns, phx_stream_t stream);

/* The same self-test with the status word of phx_gemm_f16tc_f32acc_noalloc (inside its
 * static array; the first call on a device sets that device up as the GEMM call does):
 * phx_check_device_status() then returns PHX_ERR_TIMEOUT from that word.  Allocates nothing. */
phx_status phx_selftest_bounded_wait_noalloc(uint64_t limit_ns, phx_stream_t stream);

/* Run the autotuner's selection logic (stages 1 and 2 of phx_autotune) on a simulated
 * set of `n` candidates without any GPU: candidate i "takes" base_s[i] seconds scaled by
 * (1 + drift * calls_so_far) plus deterministic noise of relative size `noise`, and
 * fails if fail[i] != 0.  Writes the chosen index to *picked (-1 if every candidate
 * failed) and the number of simulated launches to *launches. */
phx_status phx_selftest_tuner(int n, const double* base_s, const int* fail, double noise,
                              double drift, int finalists, int rounds, uint64_t seed,
                              int* picked, int64_t* launches);

/* The f32 GEMM's schedule for configuration `config` (an index of phx_config_name for
 * PHX_VARIANT_SGEMM, not the skinny one) and shape (M, N, K), as it would be on a GPU with
 * `num_sms` SMs and `ctas_per_sm` CTAs of that configuration per SM, worked out on the host
 * without any GPU.  Writes six values to the caller's array out[6]:
 *   out[0]  tiles that run whole: all of them without a stream-K part (each split into
 *           out[3] K slices when the grid is split along K), else those before it;
 *   out[1]  stream-K blocks (0: no stream-K part);
 *   out[2]  the k tiles (TILE_K values of K each) those blocks share;
 *   out[3]  K slices of a grid split along K (1: not split);
 *   out[4]  the most tile segments one stream-K block writes (at most 2 by design);
 *   out[5]  1 if, for every spread tile, the partial tiles the fix-up adds are, in k order,
 *           exactly the ones the stream-K blocks write for it and cover its k tiles once;
 *           else 0.
 * PHX_ERR_INVALID for a bad configuration, shape or machine size. */
phx_status phx_selftest_sgemm_schedule(int config, int64_t M, int64_t N, int64_t K, int ctas_per_sm,
                                       int num_sms, int64_t* out);

/* Argument validation as the GEMM calls perform it, without launching anything and
 * without touching the device: PHX_OK if (M, N, K, A, B, C) would be accepted. */
phx_status phx_validate_args(int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                             const void* C);

/* Library version string. */
const char* phx_version(void);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif

#endif /* PHX_H_ */
