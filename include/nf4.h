/*
 * nf4.h -- C ABI of libnf4: NF4 weight-quantized projections on GB300 (sm_103a).
 *
 * The operation (source: "Decode V2 -- resident executor", section 6 "Linear
 * primitive" and section 3 "CPU oracle"): y = W_hat . x, where W_hat is an
 * NF4 block-quantized M x K matrix dequantized on the fly,
 *
 *     W_hat[m][k] = codebook[code(m, k)] * scales[m][k / 64]     (fp32)
 *
 * with the decode step's fused epilogues (residual add for o/down, SwiGLU over
 * paired gate/up projections, greedy argmax over lm_head rows) and the prefill
 * chunk (N <= 32 tokens read each weight once; section 0 "Goals" item 1).
 *
 * Data layout (all row-major, rows contiguous along K):
 *   codes  uint8 [M][K/2]   byte j of row m holds k = 2j in bits 0-3 and
 *                           k = 2j+1 in bits 4-7 ("low nibble = even k")
 *   scales fp32  [M][K/64]  one absmax scale per 64-weight block along K
 *   codebook                the 16 NormalFloat levels, ascending, cb[7] = 0,
 *                           cb[0] = -1, cb[15] = +1 (nf4_codebook)
 *   bf16 tensors are passed as uint16_t bit patterns.
 *
 * Conventions (section 4 "GPU state": arena allocated at load, no cudaMalloc,
 * .item() or host sync between layers; section 5: the step is captured in a
 * CUDA graph; "golang.design/x/accel/tensor", Overview: "you own the buffers
 * you named"):
 *   - Every tensor pointer is a DEVICE pointer owned by the caller.  The library
 *     allocates nothing per call, keeps no per-call host state, never
 *     synchronizes, and launches its kernels asynchronously on `stream`
 *     (a cudaStream_t; NULL is the legacy default stream).  Calls can be
 *     recorded into a CUDA graph.
 *   - Inputs are never written, except that nf4_gemv_residual's `y` may alias
 *     `residual`.  Any other overlap between an output and an input is
 *     undefined behaviour.
 *   - The N=1 kernels, the prefill-chunk kernel and nf4_rmsnorm use
 *     programmatic dependent launch: they may start, and read (or prefetch)
 *     the weights (nf4_rmsnorm: its gain), before the previous kernel on the
 *     stream has finished when that kernel allows it; activations, outputs and
 *     workspaces are touched only after it finishes.  So weights and gains must
 *     not be written by the kernel launched just before on the same stream if
 *     that kernel triggers its dependents early (no kernel of this library
 *     that writes weights does).  NF4_PDL=0 in the environment turns this off.
 *   - Arguments are validated on the host before any launch; a failed call
 *     launches nothing and returns a negative nf4_status.  nf4_last_error()
 *     gives a message for the calling thread's last failure.  Kernels report
 *     only a bounded wait that ran out and token ids outside their table,
 *     through nf4_check_device_errors; invalid device pointers are undefined
 *     behaviour.
 *   - Alignment: codes and x / X must be 16-byte aligned; scales, y, residual,
 *     logits and Y 4-byte aligned; out 2-byte; index and workspace 8-byte.
 *   - Sizes: K a positive multiple of 64 and at most NF4_MAX_K; 1 <= M < 2^31.
 *   - Weights and activations must be finite; NaN/Inf inputs give unspecified
 *     (but memory-safe) results.
 */
#ifndef NF4_H
#define NF4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Largest K the kernels accept (elements). */
#define NF4_MAX_K 65536
/* Largest token count of the prefill chunk (LIVE_MAX_N in the source page). */
#define NF4_MAX_CHUNK_N 32

typedef void* nf4_stream; /* a cudaStream_t */

/* One NF4 matrix: device pointers to its codes and scales, and its shape. */
typedef struct nf4_weight {
  const uint8_t* codes; /* [M][K/2] */
  const float* scales;  /* [M][K/64] */
  int64_t M;
  int64_t K;
} nf4_weight;

typedef enum nf4_status {
  NF4_OK = 0,
  NF4_EINVAL = -1, /* bad shape: K % 64, K > NF4_MAX_K, M < 1, N outside [1, 32], bad dtype */
  NF4_EALIGN = -2, /* a pointer is not aligned as stated above */
  NF4_ENULL = -3,  /* a required pointer is NULL */
  NF4_ECUDA = -4,  /* a CUDA runtime call or launch failed; see nf4_last_error() */
  NF4_EARCH = -5,  /* the current device is not compute capability 10.3 (sm_103a) */
  NF4_ETIMEOUT = -6, /* a kernel's bounded wait ran out (nf4_check_device_errors only) */
  NF4_ERANGE = -7    /* a token id was outside its table (nf4_check_device_errors only) */
} nf4_status;

/* Activation element type. */
typedef enum nf4_dtype { NF4_F32 = 0, NF4_BF16 = 1 } nf4_dtype;

/*
 * y[m] = sum_k W_hat[m][k] * x[k]   (N = 1 GEMV, fp32 out)
 * Source: "Decode V2 -- resident executor", section 6: the gemv backend, FP32
 * LUT x scale x x; N=1 passes a [K] view.
 *   W       weight (device codes/scales), shape M x K
 *   x       [K] activation, fp32 or bf16 (widened exactly to fp32)
 *   y       [M] fp32 output
 * Dequantization uses the 16 levels as exact fp32 values: each level * x
 * product is formed exactly inside a fused multiply-add, the block scale is
 * applied once per 32 weights, and the sums are fp32;
 * |y - y_exact| <= 2e-3 * sum_k |x_k * W_hat[m][k]|.
 * (Opt-in, not the default: with the environment variable NF4_LUT=1, bf16 x
 * takes a narrower loop with fp16-rounded levels, relative error up to 2^-12
 * per level, in which x values more than 2^31 below the largest magnitude of
 * their thread's 32- or 64-element slice lose bits or become zero.)
 * The result for a row depends only on that row's codes, scales and x (not on
 * its position), so identical rows give bit-identical outputs.
 */
nf4_status nf4_gemv(const nf4_weight* W, const void* x, nf4_dtype xt, float* y, nf4_stream stream);

/*
 * y[m] = sum_k W_hat[m][k] * x[k] + residual[m]
 * Source: same page, section 6: "o/down residual: gemv with add aliased to y".
 *   residual  [M] fp32; may be the same pointer as y (in-place residual add)
 */
nf4_status nf4_gemv_residual(const nf4_weight* W, const void* x, nf4_dtype xt, const float* residual,
                             float* y, nf4_stream stream);

/*
 * out[m] = bf16( silu(g_m) * u_m ),  g = Wg . x,  u = Wu . x,  silu(z) = z / (1 + e^-z)
 * Source: same page, section 6 ("gate+up pairs share x ... writes silu(g)*u")
 * and section 3 (SiLU after the full gate GEMM, never on a split-K partial);
 * SiLU evaluated in fp32 ("golang.design/x/accel/tensor", func SiLU).
 *   Wg, Wu  gate and up weights, identical M and K
 *   out     [M] bf16 bits, round to nearest even
 */
nf4_status nf4_gemv_swiglu(const nf4_weight* Wg, const nf4_weight* Wu, const void* x, nf4_dtype xt,
                           uint16_t* out, nf4_stream stream);

/*
 * SwiGLU over one matrix whose rows alternate gate and up:
 *   out[c] = bf16( silu(v[2c]) * v[2c + 1] ),  v = W . x
 * Source: "gizai:tensor/lazy", method Lazy.gluIn (a gate and an up projection
 * with their rows interleaved; output column c is silu of row 2c times row
 * 2c + 1, made as the product is stored, so v itself is never written).  The
 * arithmetic is that of nf4_gemv_swiglu.
 *   W       weight of 2 x outputs rows (W->M even, else NF4_EINVAL), M x K
 *   out     [W->M / 2] bf16 bits, round to nearest even
 */
nf4_status nf4_gemv_glu_interleaved(const nf4_weight* W, const void* x, nf4_dtype xt, uint16_t* out,
                                    nf4_stream stream);

/*
 * Fused q/k/v projection, one launch over the three matrices' rows sharing x:
 *   q[m] = sum_k Wq_hat[m][k] * x[k] + bq[m]   (likewise k with Wk, bk and v with Wv, bv)
 * Source: same page, section 6 ("one grid over q.M+k.M+v.M rows sharing x (no
 * packed copy)"; the q/k/v bias of Qwen2.5-style models is added in that
 * kernel, and dropping it changes the greedy ids).  The three weights stay in
 * their own buffers; the row space is q's rows, then k's, then v's, and a
 * block's range may span two matrices.
 *   Wq, Wk, Wv  weights with a common K (any M each; q.M + k.M + v.M < 2^31)
 *   bq, bk, bv  fp32 biases of length q.M, k.M, v.M, 4-byte aligned, or NULL
 *               for no bias; added once to the fp32 row sum
 *   q, k, v     fp32 outputs of length q.M, k.M, v.M (may be consecutive parts
 *               of one buffer)
 * Errors: as nf4_gemv, plus NF4_EINVAL when the K differ.
 */
nf4_status nf4_gemv_qkv(const nf4_weight* Wq, const nf4_weight* Wk, const nf4_weight* Wv, const float* bq,
                        const float* bk, const float* bv, const void* x, nf4_dtype xt, float* q, float* k, float* v,
                        nf4_stream stream);

/*
 * logits[m] = sum_k W_hat[m][k] * x[k];  *index = min{ m : logits[m] = max_j logits[j] }
 * Source: same page, section 5 (final lm_head -> next_token = argmax(logits),
 * the id stays on the device) and "golang.design/x/accel/tensor", func Argmax
 * ("Ties go to the lowest index").  One launch, no second pass over the logits:
 * every block folds its rows into a 64-bit (value, index) key with one atomic
 * max, and the last block to finish writes *index and re-zeroes the workspace.
 *   logits     [M] fp32 output (the values the argmax is taken over; +0 and
 *              -0 compare equal)
 *   index      one int64 on the device
 *   workspace  nf4_workspace_bytes(M, K, 1) bytes of device memory, zeroed by
 *              the caller ONCE before its first use; every call leaves it
 *              zeroed again.  Calls that share a workspace must not overlap in
 *              time (use one workspace per stream).
 */
nf4_status nf4_gemv_argmax(const nf4_weight* W, const void* x, nf4_dtype xt, float* logits,
                           int64_t* index, void* workspace, nf4_stream stream);

/*
 * Y[n][m] = sum_k X[n][k] * bf16(W_hat[m][k])   for n < N <= 32, fp32 accumulate
 * Source: same page, section 0 item 1 and section 5 (prefill walks the prompt
 * in chunks of LIVE_MAX_N = 32 through the tensor-core GEMM); each weight is
 * read once per chunk.  The dequantized weight is rounded to bf16 (nearest
 * even) and multiplied on the tcgen05 tensor cores with fp32 accumulation.
 *   X          [N][K] bf16 bits, K contiguous
 *   Y          [N][M] fp32
 *   workspace  nf4_workspace_bytes(M, K, N) bytes, zeroed once by the caller;
 *              every call leaves it zeroed again (same sharing rule as above)
 */
nf4_status nf4_gemm_chunk(const nf4_weight* W, const uint16_t* X, int N, float* Y, void* workspace,
                          nf4_stream stream);

/*
 * RMSNorm of `rows` rows of K values, as its own small kernel ahead of a
 * projection:  y[r][k] = x[r][k] * w[k] / sqrt(mean_k(x[r][k]^2) + eps)
 * Source: "Decode V2 -- resident executor", section 3 (x * rsqrt(mean(x^2) +
 * eps) * w, Qwen-style, no bias; RMS weights bf16 [hidden]), section 6 (RMS
 * writes in place) and its status table (RMS fused into the following
 * projections was a loss: every block repeats the reduction; RMS stays a
 * one-block kernel); "golang.design/x/accel/tensor", func RMSNorm (each row by
 * its own root mean square, computed in f32).
 *   x     [rows][K] fp32, 4-byte aligned
 *   w     [K] bf16 gain bits, 2-byte aligned
 *   eps   finite, >= 0
 *   y     [rows][K]: fp32 (yt = NF4_F32, 4-byte aligned; may be x itself, an
 *         in-place update) or bf16 bits (yt = NF4_BF16, rounded to nearest
 *         even; must not overlap x), ready as a projection's activation
 * One block per row; the sum of squares is fp32 in a fixed order (the result
 * depends only on the row), 1 / sqrt is IEEE-rounded.  Sizes: 1 <= K <=
 * NF4_MAX_K, 1 <= rows < 2^31.  Like the projections, the kernel uses
 * programmatic dependent launch: it lets the next kernel launch at once, and
 * reads x only after the previous kernel has finished.
 */
nf4_status nf4_rmsnorm(const float* x, const uint16_t* w, int64_t rows, int64_t K, float eps, void* y,
                       nf4_dtype yt, nf4_stream stream);

/*
 * nf4_gemm_chunk without a caller workspace, for callers that cannot allocate
 * device memory: a host program that owns every allocation and hands this
 * library only its inputs and outputs, or a loop that must not call
 * cudaMalloc (it synchronizes the device).  There is no counterpart on the
 * source pages; the arithmetic, arguments and errors are those of
 * nf4_gemm_chunk.
 *   Scratch: one 8 MiB array in the library's device memory, reserved on
 *   every GPU that loads the library until the process exits.  Shapes whose
 *   nf4_workspace_bytes(M, K, N) exceeds 8 MiB are rejected with NF4_EINVAL
 *   and a message; use nf4_gemm_chunk for them.  (The 13824 x 5120 weight at
 *   N = 32 needs about 7.1 MB.)
 *   The first call on a device looks the array's device address up, with that
 *   device current; make it before any stream capture.  The address is kept
 *   for the life of the process: after cudaDeviceReset, or anything else that
 *   destroys and recreates the device's primary context, it is stale, and
 *   this entry point must not be called again in that process.  Every call on a device
 *   shares the array: calls whose kernels may overlap on the GPU (different
 *   streams or host threads) race and must be serialized by the caller.  Each
 *   call clears the part of the scratch that must start at zero, then launches
 *   on `stream`.  Nothing is allocated.
 */
nf4_status nf4_gemm_chunk_noalloc(const nf4_weight* W, const uint16_t* X, int N, float* Y, nf4_stream stream);

/* Workspace bytes that nf4_gemv_argmax (N = 1) or nf4_gemm_chunk (N > 1) need
 * for an M x K weight; the caller allocates it once (arena). */
size_t nf4_workspace_bytes(int64_t M, int64_t K, int N);

/*
 * Quantize fp32 weights W [M][K] to NF4 on the device: per 64-block the scale
 * is max |w| (an all-zero block gets scale 0 and code 7, the exact-zero level);
 * each weight takes the level nearest to w / scale, ties to the lower level.
 * Source: "Decode V2 -- resident executor", section 2 (NF4 linears, 64-weight
 * groups, encode_nf4 as the one codec).  Not on the decode hot path; provided
 * so weights can be converted on the device.
 *   codes [M][K/2] uint8 out, scales [M][K/64] fp32 out
 */
nf4_status nf4_quantize(const float* W, int64_t M, int64_t K, uint8_t* codes, float* scales,
                        nf4_stream stream);

/*
 * Embedding rows kept as NF4, gathered and dequantized:
 *   out[i][k] = W_hat[ids[i]][k] = level(code) * scale   (one fp32 product)
 * Source: same page, section 10 (the embedding stays as NF4 rows and the rows
 * a step needs are dequantized into the arena; there is no dense [vocab,
 * hidden] table).
 *   E     the [V][K] NF4 table
 *   ids   [n] int64 token ids on the device, 8-byte aligned; n = 0 does nothing
 *   out   [n][K] on the device, 16-byte aligned: fp32 (ot = NF4_F32, exact
 *         products) or bf16 bits (ot = NF4_BF16, rounded to nearest even)
 * An id outside [0, V) cannot fault: its row is written as zeros and the
 * next nf4_check_device_errors() returns NF4_ERANGE.
 */
nf4_status nf4_dequant_rows(const nf4_weight* E, const int64_t* ids, int64_t n, void* out, nf4_dtype ot,
                            nf4_stream stream);

/*
 * Diagnostic, not for the hot path: synchronizes the current device, then
 * reads and clears the library's device-side error words.  Kernels that wait
 * on shared-memory barriers (bulk-copy pipelines, tensor-core commits) bound
 * every wait; a wait that runs out (which needs a broken device or library)
 * makes the block skip its remaining work and sets an error word instead of
 * hanging.  Returns NF4_ETIMEOUT if that happened since the last check (the
 * outputs of the calls in between are invalid), NF4_ERANGE if nf4_dequant_rows
 * met an id outside its table, NF4_OK otherwise.
 */
nf4_status nf4_check_device_errors(void);

/*
 * Diagnostic for failure-detection tests; never needed for correct results.
 * Sets how many times the bulk-copy GEMV and the TMA prefill-chunk kernels
 * poll a pipeline barrier (a producer waiting for a free stage, a consumer
 * for staged weights or, in the chunk, for the dequantized operand the
 * tensor core reads) before giving up (0 restores the default, 2^22 polls).
 * With a limit of a few polls a block's producer runs out as soon as its
 * ring is full (its consumers are still computing): the block stops issuing
 * copies, skips its remaining outputs, waits (with the full limit) for the
 * copies and tensor-core work it already issued, frees its tensor memory and
 * sets the error word that nf4_check_device_errors() reports as NF4_ETIMEOUT.
 * Outputs of such a call are invalid; workspaces are left zeroed as usual.
 * Process-wide; applies to calls launched afterwards.
 */
void nf4_debug_set_wait_limit(uint32_t polls);

/* Host copy of the 16 fp32 codebook levels the kernels use. Never fails. */
void nf4_codebook(float out[16]);

/* Message for the calling thread's most recent failed call ("" if none). */
const char* nf4_last_error(void);

/* Human-readable kernel configuration chosen for an M x K weight at N tokens
 * (block shape, rows per block, split), or a message if the shape is invalid.
 * The string is thread-local and valid until the next call on this thread. */
const char* nf4_describe_config(int64_t M, int64_t K, int N);

/* The same for one operation, whose epilogue can change the launch (its
 * register use sets how many row groups fit in a block): op is "gemv",
 * "residual", "swiglu", "glu", "qkv", "argmax" (N = 1, bf16 x; M counts all
 * rows of the launch: 2 x outputs for "glu", q + k + v rows for "qkv") or
 * "chunk" (N in [1, 32]).  nf4_describe_config(M, K, N) is "gemv" at N = 1
 * and "chunk" otherwise.  An unknown op gives a message saying so. */
const char* nf4_describe_launch(const char* op, int64_t M, int64_t K, int N);

#ifdef __cplusplus
}
#endif

#endif /* NF4_H */
