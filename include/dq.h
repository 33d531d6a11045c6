/*
 * dq.h -- C ABI of libdq: the single-token (M = 1) decode hot path of an LLM on
 * one NVIDIA GB300 (sm_103a): RMSNorm / LayerNorm, matrix-vector products over
 * bf16, Q4_K and Q6_K weights dequantised in registers, grouped-query decode
 * attention over an fp16 KV cache, and a whole decode token over a
 * Qwen3-8B-shaped layer stack.
 *
 * Conventions (every entry point):
 *   - Returns a dq_status: 0 (DQ_OK) or a negative code.  Arguments are checked
 *     before anything is launched; a failed check launches nothing.
 *   - Pointers are caller-owned DEVICE pointers unless marked "host".  The
 *     library never frees caller memory and allocates nothing in the compute
 *     calls (only dq_model_create allocates, and dq_model_destroy frees).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Work is enqueued asynchronously; nothing synchronises unless
 *     stated.  A CUDA error at launch returns DQ_ERR_CUDA and
 *     dq_last_cuda_error() gives the cudaError_t.
 *   - Kernels bound every internal wait by a wall-clock limit; a timeout sets a
 *     per-device error flag, readable with dq_device_error().
 *   - No exception or C++ type crosses this interface.
 *
 * Block formats (this library's canonical little-endian layouts; the pages fix
 * the sizes -- "The roofline holds on a second GPU", sections "The Math" and
 * "The search space": Q4_K is 4.5 bits per weight, 256 weights in 144 bytes;
 * Q6_K is 6.5625 bits per weight, 256 weights in 210 bytes -- but not the bit
 * positions, which are defined here):
 *
 *   Q4_K, 144 bytes, weights n = 32 j + i (j = 0..7):
 *     [0,2) d (binary16)  [2,4) dmin (binary16)
 *     [4,16) 96-bit little-endian bit string: sc_j at bits 6j..6j+5,
 *            m_j at bits 48+6j..53+6j (unsigned 6-bit)
 *     [16,144) byte 16+16j+i: low nibble = code of weight 32j+i,
 *              high nibble = code of weight 32j+16+i
 *     w_n = d * sc_j * q_n - dmin * m_j
 *   Q6_K, 210 bytes, weights n = 32 g + r (g = 0..7):
 *     [0,128) byte 16g+i: low nibble = low 4 bits of weight 32g+i,
 *             high nibble = low 4 bits of weight 32g+16+i
 *     [128,192) high 2 bits of weight 32g+16h+4t+e at bits 2t..2t+1 of byte
 *               128+8g+4h+e (h in {0,1}; t, e in 0..3)
 *     [192,208) int8 sc[16], sc[s] for weights 16s..16s+15
 *     [208,210) d (binary16)
 *     q_n = low4 | high2 << 4;  w_n = d * sc[n/16] * (q_n - 32)
 *   Q2_K, 84 bytes, weights n = 16 j + i (j = 0..15): 2-bit codes, the step
 *   below 4 bits that "The Mountain Runs" names (its closing section: the
 *   expert kernels dequantise 2/4-bit codes in registers) without a layout:
 *     [0,2) d (binary16)  [2,4) dmin (binary16)
 *     [4,20) byte 4+j: low nibble sc_j, high nibble m_j (unsigned 4-bit)
 *     [20,84) byte 20+4j+b (b = 0..3): the code of weight 16j+4k+b at bits
 *             2k..2k+1 (k = 0..3)
 *     w_n = d * sc_j * q_n - dmin * m_j      (2.625 bits per weight)
 *   A quantised matrix is row-major: row r is the K/256 blocks of that row,
 *   back to back.  The library requires 16-byte aligned rows, i.e. K % 256 == 0
 *   for Q4_K, K % 2048 == 0 for Q6_K and K % 1024 == 0 for Q2_K, and a
 *   16-byte aligned base pointer.
 *   bf16 matrices are row-major [rows][K], K % 8 == 0, 16-byte aligned.
 */
#ifndef DQ_H
#define DQ_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define DQ_API __declspec(dllexport)
#else
#define DQ_API __attribute__((visibility("default")))
#endif

typedef enum {
    DQ_OK = 0,
    DQ_ERR_NULL = -1,        /* a required pointer is NULL */
    DQ_ERR_SHAPE = -2,       /* a size is zero, negative or inconsistent */
    DQ_ERR_ALIGN = -3,       /* a pointer or row is not 16-byte aligned */
    DQ_ERR_UNSUPPORTED = -4, /* a shape this build has no kernel for */
    DQ_ERR_CUDA = -5,        /* a CUDA runtime call failed: see dq_last_cuda_error() */
    DQ_ERR_TIMEOUT = -6,     /* a kernel gave up a bounded wait (device flag) */
    DQ_ERR_ALLOC = -7        /* dq_model_create could not allocate its workspace */
} dq_status;

/* Weight formats. */
#define DQ_FMT_BF16 0
#define DQ_FMT_Q4K 1
#define DQ_FMT_Q6K 2
#define DQ_FMT_Q2K 3

/* Static text for a status code (never NULL). */
DQ_API const char* dq_status_string(int status);

/* cudaError_t of the most recent DQ_ERR_CUDA returned on this host thread. */
DQ_API int dq_last_cuda_error(void);

/* Synchronises `stream`, then reads and clears the current device's error flag:
 * 0 if no kernel gave up a bounded wait since the last call, else a bit mask
 * (1 consumer timeout, 2 producer timeout, 4 copies in flight at exit,
 * 8 bad argument seen on the device, 16 a fused-token wait for another
 * block's output ran out, 32 tensor-core completion timeout).  Returns DQ_ERR_CUDA on a
 * CUDA error. */
DQ_API int dq_device_error(void* stream);

/* The same check as a dq_status: synchronises `stream`, reads and clears the
 * current device's error flag, and returns DQ_OK when it was clear,
 * DQ_ERR_TIMEOUT when a kernel gave up a bounded wait since the last check
 * (any of the timeout bits above), DQ_ERR_SHAPE when the only bit is a bad
 * argument seen on the device, or DQ_ERR_CUDA.  Kernels that give up a wait
 * leave their outputs undefined but return, so the context stays usable. */
DQ_API int dq_check_device(void* stream);

/* ------------------------------------------------------------------- norms
 * "one-serial-kernel" (vocodex.ai), section "One thread": the normalisation
 * that runs twice per layer and once at the end, reduced by a block of threads
 * instead of one thread per row; the layer norm in two passes (mean, then the
 * variance of x - mean).
 *
 * dq_rmsnorm:   y[r][i] = x[r][i] / sqrt(mean_i(x[r][i]^2) + eps) * gamma[i]
 * dq_layernorm: y[r][i] = (x[r][i] - mu_r) / sqrt(var_r + eps) * gamma[i] + beta[i],
 *               mu_r = mean, var_r = population variance (divide by n).
 * x, y: fp32 [rows][n] row-major (y may equal x); gamma, beta: fp32 [n].
 * One thread block of 256 threads per row; fp32 arithmetic.
 * Errors: NULL pointer -> DQ_ERR_NULL; rows < 1, n < 1, or eps negative, NaN or
 * infinite -> DQ_ERR_SHAPE; gamma or beta not 16-byte aligned -> DQ_ERR_ALIGN. */
DQ_API int dq_rmsnorm(const float* x, const float* gamma, float* y, int rows, int n, float eps, void* stream);
DQ_API int dq_layernorm(const float* x, const float* gamma, const float* beta, float* y, int rows, int n,
                        float eps, void* stream);

/* Same computations with an explicit block size (1 .. 1024, a power of two):
 * threads = 1 is the one-thread-per-row kernel the page measured as the fault;
 * the sweep over thread counts is the page's "corner control" as a CUDA
 * block-size sweep.  Errors as above, plus DQ_ERR_SHAPE for a bad count. */
DQ_API int dq_rmsnorm_threads(const float* x, const float* gamma, float* y, int rows, int n, float eps,
                              int threads, void* stream);
DQ_API int dq_layernorm_threads(const float* x, const float* gamma, const float* beta, float* y, int rows,
                                int n, float eps, int threads, void* stream);

/* -------------------------------------------------------------------- GEMV
 * "The Mountain Runs" (coderlegion, S-MoE diary #5), section 3: one output per
 * weight row; the weight stream is read in wide consecutive chunks instead of
 * one thread per row.  Here rows are streamed into shared memory by bulk (TMA)
 * copies and dequantised in registers ("The roofline holds on a second GPU",
 * section "Hiding, fusing...": keep the weights packed, unpack in registers,
 * accumulate in 32 bits).
 *
 *   y[r] = sum_k W[r][k] * x[k],  r < rows, fp32 output.
 *
 * dq_gemv_bf16: W bf16 [rows][K], x bf16 [K] (both bit patterns), fp32
 *   accumulation.  K % 8 == 0, 8 <= K <= 24576.
 * dq_gemv_q4k / dq_gemv_q6k: W blocks (see the header comment), x fp32 [K].
 *   The activation is carried as a 15-bit fixed-point vector with one fp32
 *   scale per 32 elements (relative error <= 2^-15 of each group's largest
 *   |x|), products are exact 32-bit integer sums, the block scales are applied
 *   in fp32.  Q4_K: K % 256 == 0, 256 <= K <= 16384.  Q6_K: K % 2048 == 0,
 *   2048 <= K <= 16384.
 * dq_gemv_q2k: the same with Q2_K blocks (the min term uses the integer sums
 *   of the fixed-point activation over each 16-element sub-block).
 *   K % 1024 == 0, 1024 <= K <= 16384.
 * W, x 16-byte aligned (DQ_ERR_ALIGN otherwise).  y must not overlap W or x.
 * Ordering: each call is a programmatic dependent launch on `stream`.  Before
 * the previous kernel on the stream has completed it only sets up and asks L2
 * for the first weight tiles (a hint that reads nothing into the SMs); it
 * reads W and x and writes y only after that kernel's writes are visible, so
 * stream order holds as for a plain launch.
 * Errors: NULL -> DQ_ERR_NULL; rows < 1 or K outside the ranges -> DQ_ERR_SHAPE
 * or DQ_ERR_UNSUPPORTED. */
DQ_API int dq_gemv_bf16(const void* W_bf16, const void* x_bf16, float* y, int rows, int K, void* stream);
DQ_API int dq_gemv_q4k(const void* W_blocks, const float* x, float* y, int rows, int K, void* stream);
DQ_API int dq_gemv_q6k(const void* W_blocks, const float* x, float* y, int rows, int K, void* stream);
DQ_API int dq_gemv_q2k(const void* W_blocks, const float* x, float* y, int rows, int K, void* stream);

/* The same four products through one entry point, with flags.  fmt: DQ_FMT_BF16,
 * DQ_FMT_Q4K, DQ_FMT_Q6K or DQ_FMT_Q2K (x is bf16 for DQ_FMT_BF16, else fp32).
 * DQ_GEMV_STATIC_WEIGHTS: the kernel that precedes this call on the stream does
 * not write W (a model's weight table, say), so the GEMV may copy W into shared
 * memory before that kernel completes; x is still read, and y written, only after
 * it.  A caller that sets the flag while the preceding kernel writes W gets
 * undefined results.  flags = 0 is exactly dq_gemv_bf16/q4k/q6k/q2k.
 * Errors: as those, plus DQ_ERR_SHAPE for an unknown format or flag. */
#define DQ_GEMV_STATIC_WEIGHTS 1
DQ_API int dq_gemv_ex(int fmt, const void* W, const void* x, float* y, int rows, int K, int flags, void* stream);

/* Diagnostics: when `buffer` is not NULL, every later GEMV launch in this
 * process writes 8 unsigned 64-bit values per thread block at
 * buffer[8 * block]: global-timer ns at start, after set-up, after the
 * dependency wait, after the activation is staged, after it is quantised,
 * when the first weight stage is ready; then the latest warp end time and the
 * count of finished warps (both accumulated: zero the buffer before a launch).
 * Block 0 also writes SM clock stamps for its first 64 stages after the
 * per-block values, at buffer[8 * blocks + i]: [2t] stage t ready, [2t + 1]
 * thread 0 done with it, [128 + t] stage t's copy issued.  The i-th GEMV
 * launch after this call writes its values at word offset i (8 blocks + 192),
 * so the buffer needs (64 bytes per block + 1536 bytes) per traced launch.  A
 * dq_decode_step that runs the fused token kernel writes instead 8 values per
 * block and phase at buffer[8 (block * phases + phase)] (phases = 5 n_layers
 * + 1: per layer Q|K|V, attention, O, gate/up, down; then the vocabulary):
 * global-timer ns at [0] phase entered, [2] the block's warps done with the
 * previous phase, [4] phase done; SM clock cycles at [3] the same moment as
 * [2], [5] activation arrived and quantised, [7] activation in registers, [1]
 * first weight tile ready; [6] unused; 64 bytes per block and phase.  In an
 * attention phase the block's first item writes global-timer ns at [1] q ready,
 * [3] keys staged, [5] partial computed, [6] merge decided, [7] output
 * stored.  A tensor-core dq_matmul_q4k_path or dq_matmul_q4k_split writes, for
 * block 0 and its first 32 stages (one Q4_K block column each), 8 SM clock
 * stamps per stage at buffer[8 stage]: operands seen ready and MMAs issued
 * (control thread), stage start, weights landed, operand buffer free and stage
 * written (thread 0); then global-timer ns per block at buffer[256 + 4 block]:
 * [0] start, [1] first stage ready, [2] last stage's MMAs done, [3] end
 * (2304 bytes + 32 bytes per block).
 * NULL turns tracing off.  Not for use while
 * another thread launches kernels of the library. */
DQ_API int dq_debug_trace(void* buffer);

/* Dequantise nblocks consecutive blocks to fp32 (256 values per block), each
 * weight computed as the block formula above in fp32.  A test hook: with the
 * synthetic binades (Q4_K and Q2_K d in [2^-13, 2^-12), dmin in [2^-10, 2^-9);
 * Q6_K d in [2^-14, 2^-13)) every weight is exact, so the output is bit-exact.
 * blocks: any alignment; out: fp32 [nblocks * 256].  nblocks >= 1. */
DQ_API int dq_dequant_q4k(const void* blocks, float* out, long long nblocks, void* stream);
DQ_API int dq_dequant_q6k(const void* blocks, float* out, long long nblocks, void* stream);
DQ_API int dq_dequant_q2k(const void* blocks, float* out, long long nblocks, void* stream);

/* -------------------------------------------------------------- attention
 * Grouped-query decode attention for one token ("The roofline holds on a second
 * GPU", sections "Said before the run" and "Where the time goes": each new token
 * also reads the conversation's keys and values; 32 query heads share 8 KV heads
 * in the Qwen3-8B census).
 *
 *   for query head h (KV head g = h / (n_q / n_kv)) and keys j < n_keys:
 *     s_j = (q_h . k_gj) / sqrt(head_dim);  p = softmax(s);  out_h = sum_j p_j v_gj
 *
 * q: fp32 [n_q][head_dim]; k_plane, v_plane: fp16 [n_kv][max_ctx][head_dim]
 * (one layer of the cache); out: fp32 [n_q][head_dim].  The keys are split into
 * up to 32 chunks per KV head, one thread block each; the last block to finish
 * for a KV head merges the chunk partials (max-subtracted log-sum-exp).
 * workspace: device scratch of dq_attention_workspace_bytes(n_q, n_kv) bytes,
 * zero-filled by the caller before its first use; the kernel leaves it zeroed
 * again (its counters) so it can be reused.  Calls that share a workspace must
 * not overlap in time.
 * Limits: head_dim == 128, n_q % n_kv == 0, n_q / n_kv <= 8, 1 <= n_keys <= max_ctx.
 * Errors: NULL -> DQ_ERR_NULL; shapes -> DQ_ERR_SHAPE / DQ_ERR_UNSUPPORTED;
 * workspace too small -> DQ_ERR_SHAPE. */
DQ_API size_t dq_attention_workspace_bytes(int n_q, int n_kv);
DQ_API int dq_attention_decode(const float* q, const void* k_plane, const void* v_plane, float* out, int n_q,
                               int n_kv, int head_dim, int max_ctx, int n_keys, void* workspace,
                               size_t workspace_bytes, void* stream);

/* The same attention without any allocation.  The pages have no counterpart.
 * It serves callers that cannot call cudaMalloc: inference-server plugins
 * whose host process owns all device memory through its own pool, and
 * embedded or real-time deployments that fix their device memory at start-up
 * (where an allocation can fail, or would block the device, in the middle of
 * serving).  The scratch (merge counters and chunk partials) is one static
 * device array of the library, sized for n_q <= DQ_STATIC_ATT_MAX_Q and
 * n_kv <= DQ_STATIC_ATT_MAX_KV: 256 + 64 * 32 * 132 * 4 = 1,081,600 bytes,
 * held on every device that loads the library until the process exits.
 * The first call on a device, with that device current, looks up the array's
 * device address and keeps it for the process; make that first call before any
 * stream capture.  cudaDeviceReset invalidates the kept address: do not call
 * this entry point after a device reset.  Each call first clears the array's
 * merge counters with a cudaMemsetAsync on `stream` (not an allocation).  All
 * calls share the array, which keeps the last call's partials: calls whose
 * executions overlap in time (on any streams) race and give wrong results.
 * Arguments as dq_attention_decode without the workspace.
 * Errors: NULL -> DQ_ERR_NULL; shapes, and n_q > DQ_STATIC_ATT_MAX_Q or
 * n_kv > DQ_STATIC_ATT_MAX_KV -> DQ_ERR_SHAPE; head_dim != 128 or n_q / n_kv > 8
 * -> DQ_ERR_UNSUPPORTED, as is a current device index of 64 or more;
 * misaligned pointers -> DQ_ERR_ALIGN; a CUDA error -> DQ_ERR_CUDA. */
#define DQ_STATIC_ATT_MAX_Q 64
#define DQ_STATIC_ATT_MAX_KV 64
DQ_API int dq_attention_decode_static(const float* q, const void* k_plane, const void* v_plane, float* out, int n_q,
                                      int n_kv, int head_dim, int max_ctx, int n_keys, void* stream);

/* Qwen3 attention inputs.  The pages name the model (Qwen3-8B, "The roofline
 * holds on a second GPU", section "The Math") but not its attention's input
 * transforms; these are the model family's own:
 *   head_rmsnorm(v, w) = v / sqrt(mean(v^2) + eps) * w   (per 128-dim head)
 *   rope(v, pos): for i < 64, (v[i], v[i + 64]) turns by pos / theta^(i / 64)
 * with one weight vector for all query heads and one for all key heads.
 *
 * dq_rope_table fills table, fp32 (cos, sin) pairs [max_ctx][head_dim / 2][2]
 * (device, 16-byte aligned, written), with the angle p / theta^(2i / head_dim)
 * for row p and pair i, computed in double precision and rounded once to fp32.
 * Enqueued on `stream`.  Errors: NULL -> DQ_ERR_NULL; max_ctx < 1, head_dim
 * odd or < 2, theta <= 1 -> DQ_ERR_SHAPE; misaligned -> DQ_ERR_ALIGN. */
DQ_API int dq_rope_table(float* table, int max_ctx, int head_dim, double theta, void* stream);

/* dq_attention_decode with the Qwen3 inputs, for the token at pos = n_keys - 1:
 *   q_h <- rope(head_rmsnorm(q_h, q_norm), pos) for every query head;
 *   k_plane[g][pos] = fp16(rope(head_rmsnorm(k_new[g], k_norm), pos));
 * then the attention of q over keys 0..pos.  q: fp32 [n_q][128] as projected
 * (read, not modified); k_new: fp32 [n_kv][128] as projected (read); k_plane:
 * fp16 [n_kv][max_ctx][128] (row pos written, rows < pos read); v_plane as in
 * dq_attention_decode (row pos must already hold the token's value);
 * q_norm, k_norm: fp32 [128]; rope_table: a dq_rope_table of at least n_keys
 * rows for head_dim 128.  All device pointers, 16-byte aligned.  eps: the head
 * norm's epsilon, finite and >= 0 (else DQ_ERR_SHAPE).  Workspace, limits and
 * other errors as dq_attention_decode. */
DQ_API int dq_attention_decode_rope(const float* q, const float* k_new, void* k_plane, const void* v_plane, float* out,
                                    const float* q_norm, const float* k_norm, const float* rope_table, float eps,
                                    int n_q, int n_kv, int head_dim, int max_ctx, int n_keys, void* workspace,
                                    size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------ M-token sweep
 * "The roofline holds on a second GPU", section "The Math": M tokens share one
 * read of the weights; below M* = (w/16)(R/BW) memory bounds the product, above
 * it arithmetic does.  Y[m][r] = sum_k W[r][k] * X[m][k] for m < M.
 * W: Q4_K blocks [rows][K/256] (16-byte aligned); X fp32 [M][K] (16-byte
 * aligned); Y fp32 [M][rows].  1 <= M <= 64, K a positive multiple of 256.
 *
 * Paths: DQ_MATMUL_CUDA_CORE runs the streaming GEMV once per token (reads W
 * M times; K <= 16384).  DQ_MATMUL_TENSOR reads W once for all tokens on the
 * tensor cores (tcgen05.mma, fp16 operands: each weight and activation is
 * rounded to fp16, |X| must stay below 65504; fp32 accumulation).
 * DQ_MATMUL_AUTO picks CUDA cores for M <= 2 and tensor cores for M >= 3 (the
 * measured crossover on the 12288 x 4096 table).
 * Errors: NULL -> DQ_ERR_NULL; M, rows, K or path out of range ->
 * DQ_ERR_SHAPE; misaligned W or X -> DQ_ERR_ALIGN; CUDA-core path with
 * K > 16384 -> DQ_ERR_UNSUPPORTED; a CUDA error -> DQ_ERR_CUDA. */
#define DQ_MATMUL_AUTO 0
#define DQ_MATMUL_CUDA_CORE 1
#define DQ_MATMUL_TENSOR 2
DQ_API int dq_matmul_q4k_path(const void* W_blocks, const float* X, float* Y, int M, int rows, int K, int path,
                              void* stream);

/* dq_matmul_q4k_path with DQ_MATMUL_AUTO. */
DQ_API int dq_matmul_q4k(const void* W_blocks, const float* X, float* Y, int M, int rows, int K, void* stream);

/* The same product on the tensor cores with K split across blocks.  Without a
 * split every block takes whole rows: a share of rows / (SM count) rows that
 * fills only part of a 128-row tile (81 of 128 for 12288 rows on 152 SMs), over
 * all of K.  Here the (128-row tile, 256-column block) stages are shared out in
 * contiguous runs, so every tile is full and a block takes 10 or 11 stages
 * instead of 16 on that table.  A tile whose columns two or three blocks share
 * is summed from their partial tiles in block order (deterministic: the same
 * order whichever block finishes last).  For M > 16 a first kernel converts X
 * once into fp16 tiles in the workspace, which each stage then copies beside its
 * weights (instead of every block converting every token's activations).
 * Arguments, operand rounding and errors as dq_matmul_q4k_path with
 * DQ_MATMUL_TENSOR, with rows <= 524288 (else DQ_ERR_UNSUPPORTED); in addition
 * workspace: a device buffer of at least
 * dq_matmul_q4k_split_workspace_bytes(M, rows, K) bytes (else DQ_ERR_SHAPE),
 * 16-byte aligned (else DQ_ERR_ALIGN), owned by the caller, zero-filled before
 * its first use.  Its first 64 KB hold the tiles' counts, which every call
 * leaves at zero, the rest the fp16 activations (M > 16) and the partial tiles:
 * it serves later calls of any shape whose size fits.  Calls sharing one workspace must not run at the same time
 * (one workspace per stream).  After a call that reports a device error,
 * zero-fill it again. */
DQ_API int dq_matmul_q4k_split(const void* W_blocks, const float* X, float* Y, int M, int rows, int K,
                               void* workspace, long long workspace_bytes, void* stream);

/* Bytes of the workspace dq_matmul_q4k_split needs for this shape on the
 * current device (its SM count sets the split), or DQ_ERR_SHAPE /
 * DQ_ERR_UNSUPPORTED for a shape it does not take. */
DQ_API long long dq_matmul_q4k_split_workspace_bytes(int M, int rows, int K);

/* -------------------------------------------------------------- decode step
 * One decode token over a pre-norm decoder stack ("The roofline holds on a
 * second GPU", section "The Math": per layer a 4096x4096 attention table plus
 * 1024x4096 key and value tables, 12288x4096 gate and up tables, a 4096x12288
 * down table, then a 151936x4096 vocabulary table; "one-serial-kernel",
 * section "One thread": the norm twice per layer and once at the end).
 *
 * Per layer l, with x the fp32 residual vector:
 *   h = RMSNorm(x, attn_norm[l]);  [q|k|v] = Wqkv[l] h
 *   (Qwen3 inputs: each q and k head <- rope(head_rmsnorm(., q_norm/k_norm[l]), pos))
 *   cache[l][0][:, pos] = fp16(k);  cache[l][1][:, pos] = fp16(v)
 *   a = GQA attention of q over keys 0..pos;  x += Wo[l] a
 *   h = RMSNorm(x, ffn_norm[l]);  x += Wdown[l] (SiLU(Wgate[l] h) * (Wup[l] h))
 * then logits = Wvocab RMSNorm(x, out_norm).
 * Each layer runs as five kernels (norm+QKV with the cache append, attention
 * with its merge, O projection + residual, norm+gate/up+SwiGLU, down + residual)
 * chained with programmatic dependent launch and captured in one CUDA graph, so
 * each kernel streams its weights while the previous one finishes.
 */
typedef struct dq_model dq_model; /* opaque: owns workspace + graph, BORROWS weights */

typedef struct {
    int n_layers, hidden, ffn, n_q_heads, n_kv_heads, head_dim, vocab, max_ctx;
    float eps;                     /* every RMSNorm's epsilon: finite and >= 0 */
    /* host arrays of n_layers DEVICE pointers each (copied at create time): */
    const float* const* attn_norm; /* fp32 [hidden] */
    const void* const* wqkv;       /* Q4_K [(n_q + 2 n_kv) head_dim][hidden], rows q | k | v */
    const void* const* wo;         /* Q4_K [hidden][n_q head_dim] */
    const float* const* ffn_norm;  /* fp32 [hidden] */
    const void* const* wgate;      /* Q4_K [ffn][hidden] */
    const void* const* wup;        /* Q4_K [ffn][hidden] */
    const void* const* wdown;      /* DQ_FMT_Q4K or DQ_FMT_Q6K [hidden][ffn] */
    const int* down_fmt;           /* host int[n_layers]: format of wdown[l] */
    const float* out_norm;         /* device fp32 [hidden] */
    const void* wvocab;            /* device Q6_K [vocab][hidden] */
    void* kv_cache;                /* device fp16 [n_layers][2][n_kv][max_ctx][head_dim] */
    int use_graph;                 /* separate kernels only: 1 capture them in a CUDA graph, 0 eager launches */
    int flags;                     /* DQ_MODEL_* bits; 0 for the default behaviour */
    /* Qwen3 attention inputs (see dq_attention_decode_rope); q_norm NULL: plain
     * attention and the next two fields are ignored. */
    const float* const* q_norm;    /* host array of n_layers DEVICE pointers: fp32 [head_dim], query heads */
    const float* const* k_norm;    /* the same for the key heads */
    double rope_theta;             /* rotary base, > 1 (Qwen3: 1e6) */
} dq_model_desc;

/* dq_model_desc.flags: launch the token's kernels without programmatic
 * dependent launch (each kernel waits for the previous one to finish before it
 * starts streaming); for measuring what the overlap is worth. */
#define DQ_MODEL_NO_PDL 1
/* dq_model_desc.flags: run the token as one persistent cooperative kernel
 * (the fused token kernel) where the shape allows; otherwise the flag is
 * ignored and the separate kernels run.  See dq_model_create. */
#define DQ_MODEL_FUSED 2

/* Validates the description, allocates the workspace (activations, attention
 * scratch, the fused kernel's launch state) and prepares the token on the
 * current device.
 *
 * Two ways to run a token.  By default it is 5 n_layers + 1 kernels chained
 * by programmatic dependent launch, captured once in a CUDA graph when
 * use_graph is set.  With DQ_MODEL_FUSED, where the shape allows (at most 64
 * layers; hidden and n_q head_dim at most 4096, hidden a multiple of 2048;
 * ffn at most 12288 with a Q6_K down projection (a multiple of 2048), else as
 * far as the block's shared memory allows), it is
 * one cooperative launch of one block per SM that runs all phases while the
 * weights stream through each block's ring without a break; a phase starts on
 * each block as soon as the vector it reads is complete (every value carries a
 * tag of the write that made it, in its lowest mantissa bit: the activation
 * buffers of a fused model differ from the computed values by at most that one
 * fp32 ulp).  For contexts of at most 4 keys (pos <= 3) it skips the
 * attention phase and every block computes the attention at the start of
 * the O phase (and writes it to the model buffer of the attention output,
 * dq_model_buffer 2, one block per head).  With the Qwen3 inputs the workspace also holds the
 * rotary table (max_ctx x 512 bytes), computed here.  Host call;
 * synchronises the device.  *out receives the handle (NULL on error).
 * Errors: DQ_ERR_NULL, DQ_ERR_SHAPE, DQ_ERR_ALIGN, DQ_ERR_UNSUPPORTED,
 * DQ_ERR_ALLOC, DQ_ERR_CUDA. */
DQ_API int dq_model_create(const dq_model_desc* desc, dq_model** out);

/* Enqueues one token on `stream`: x_in fp32 [hidden] (read), position pos
 * (0 <= pos < max_ctx; the cache must hold keys 0..pos-1), logits fp32 [vocab]
 * (written).  Writes this token's k and v into the cache at pos.  Calls on one
 * model must not overlap in time.  The fused token kernel's arguments depend only
 * on this call's arguments (its launch state lives in the model's workspace and
 * the kernel's last block puts it back before it exits), so the call may be
 * captured into a CUDA graph and the graph replayed, one replay at a time per
 * model.
 * Errors: DQ_ERR_NULL, DQ_ERR_SHAPE, DQ_ERR_CUDA. */
DQ_API int dq_decode_step(dq_model* m, const float* x_in, int pos, float* logits, void* stream);

/* dq_decode_step from host memory: copies x_host (fp32 [hidden]) to the
 * model's own device buffer, enqueues the token on `stream`, copies the logits
 * (fp32 [vocab]) to logits_host and waits for the stream.  Page-locked host
 * buffers make the copies asynchronous; pageable ones work and are staged by the
 * driver.  Synchronises, so it cannot be captured into a CUDA graph.  Calls on one
 * model must not overlap in time.
 * Errors: DQ_ERR_NULL, DQ_ERR_SHAPE, DQ_ERR_CUDA. */
DQ_API int dq_decode_step_host(dq_model* m, const float* x_host, int pos, float* logits_host, void* stream);

/* Number of kernels one dq_decode_step launches. */
DQ_API int dq_model_launches_per_step(const dq_model* m);

/* 1 when dq_decode_step runs the fused token kernel, 0 when it runs separate
 * kernels, DQ_ERR_NULL for a NULL handle.  A fused token whose device wait ran
 * out (dq_check_device returns DQ_ERR_TIMEOUT) has undefined logits and cache
 * row, but the kernel still ends (its blocks stop working; blocks waiting on
 * their outputs run out in turn) and its last block resets the launch state
 * and the tagged activation buffers: the model stays usable, and the next token
 * at that position rewrites the cache row. */
DQ_API int dq_model_fused(const dq_model* m);

/* Diagnostics for the fused token kernel's failure path.  wait_limit_ns bounds
 * every wait of the model's later fused tokens (1e3 .. 6e10 ns; the default is
 * 4e9).  skew > 0 makes the NEXT fused token wait for something that never
 * comes: every read of an activation another block writes waits for a write
 * that is never made.  Every block's first such wait runs out after
 * wait_limit_ns, the kernel records the timeout (bit 16) and ends.  The skew
 * applies to one token only.
 * Errors: DQ_ERR_NULL; DQ_ERR_SHAPE (limit out of range, skew < 0 or > 1000);
 * DQ_ERR_UNSUPPORTED when the model does not run the fused kernel. */
DQ_API int dq_model_debug_waits(dq_model* m, unsigned long long wait_limit_ns, int skew);

/* Diagnostics: the next n workspace allocations of dq_model_create (in this
 * process) fail as if the device were out of memory, so the caller sees
 * DQ_ERR_ALLOC and no handle; n = 0 cancels.  Errors: DQ_ERR_SHAPE for n < 0. */
DQ_API int dq_debug_fail_next_allocs(int n);

/* Diagnostics for per-kernel timing: enqueues one of the token's kernels on
 * its own, launched as in the token (with programmatic dependent launch unless
 * the model has DQ_MODEL_NO_PDL: back-to-back calls overlap one kernel's
 * start-up with the previous one's end, as the token's kernels do), with the
 * position and logits pointer of the most recent dq_decode_step on this model.  kind: 0 norm+QKV+append,
 * 1 attention, 2 O projection + residual, 3 norm+gate/up+SwiGLU, 4 down +
 * residual, 5 final norm + vocabulary (layer ignored).  It updates the model's
 * activations and cache row like the token does.
 * Errors: DQ_ERR_NULL, DQ_ERR_SHAPE (layer or kind out of range), DQ_ERR_CUDA. */
DQ_API int dq_model_enqueue_kernel(dq_model* m, int layer, int kind, void* stream);

/* Diagnostics: device pointer of one of the model's activation buffers, for
 * checking a kernel's output in isolation.  which: 0 the fp32 residual x
 * [hidden], 1 q [n_q head_dim], 2 the attention output [n_q head_dim], 3 the
 * SwiGLU activation [ffn].  The buffers are owned by the model.
 * Errors: DQ_ERR_NULL, DQ_ERR_SHAPE. */
DQ_API int dq_model_buffer(const dq_model* m, int which, void** ptr);

/* Frees the workspace and graph (synchronises the device).  NULL is a no-op. */
DQ_API int dq_model_destroy(dq_model* m);

#ifdef __cplusplus
}
#endif

#endif /* DQ_H */
