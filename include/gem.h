/*
 * gem.h — C ABI of the GB300 (sm_103a) decoder-step library: Q4_0 dequantise-and-matvec,
 * RMSNorm / per-head QK-norm / RoPE / KV append, grouped-query split-K decode attention,
 * gated FFN activation, and one whole decoder layer step.
 *
 * Sources, cited by page title and section:
 *   [GEM]  "gem" engine research record (Gemma 4 native engine), sections "Verified model
 *          facts" and "Native Metal diagnostic: buffer ownership" and the decode-attention
 *          notes that follow them (split P*V partitions merged in ascending order).
 *   [GELO] "GELO LLM generation", sections 02 (definitions: decode, KV cache, QK-norm, GQA,
 *          sliding window, p-RoPE), 04 (Qwen3 family table), 05 (components: apply_qk_norm,
 *          cached attention with n_kv = n_cache + 1) and 06 (block topology).
 *
 * Conventions shared by every call
 *   - Every pointer argument is a DEVICE pointer owned by the caller.  The library never
 *     allocates device memory in a call (gem_step_plan_create, a set-up call, is the one
 *     exception); calls that need scratch take a caller-provided workspace whose size is
 *     returned by the matching *_workspace() query.  Two calls keep their scratch in arrays
 *     of the library instead, one per device: gem_q4_0_gemv with B >= 2 on matrices of more
 *     than 64M weights (its operand records, 4 MiB) and gem_gqa_decode_attn_noalloc (its split
 *     partials, 8 MiB).  Calls of the same
 *     one of these two that can run at the same time on one device (different streams) race
 *     on its array; calls issued in order on one stream are safe.  gem_q4_0_gemv_ws and
 *     gem_gqa_decode_attn take a caller workspace and share nothing.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).  Every
 *     call only enqueues work and returns; results are ready when the stream reaches them.
 *   - Activations are fp32, row-major [B][...] with the given row stride (in elements).
 *     KV caches hold IEEE binary16 bit patterns (uint16_t), laid out [B][n_kv][cap][d].
 *   - Q4_0 matrices are raw GGML bytes: N rows, each K/32 blocks of 18 bytes (binary16 scale
 *     d little endian, then 16 bytes of 4-bit codes q; byte j holds element j in its low
 *     nibble and element j + 16 in its high nibble); weight = (q - 8) * d.  [GEM]
 *   - The fast path needs K % 256 == 0 and a 16-byte aligned matrix; other matrices with
 *     K % 32 == 0 go through a slower general kernel.  K % 32 != 0 is rejected.
 *   - Batch B is 0..8 (0 = nothing to do).  Larger batches are GEM_ERR_UNSUPPORTED_SHAPE.
 *   - Arguments are checked on the host before anything is enqueued; a rejected call has
 *     no effect.  Values only the device can see (positions) are checked by the kernels,
 *     which then skip the offending sequence and OR a GEM_DEVFLAG_* bit into *status
 *     (when `status` is NULL, into the library's own per-device word, read with
 *     gem_device_status()).  Kernels never trap or assert.
 */
#ifndef GEM_H
#define GEM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GEM_API __attribute__((visibility("default")))
#else
#define GEM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gem_status {
    GEM_OK = 0,
    GEM_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad stride or enum */
    GEM_ERR_MISALIGNED = 2,         /* pointer or stride violates a stated alignment */
    GEM_ERR_UNSUPPORTED_SHAPE = 3,  /* K % 32 != 0, B > 8, head_dim not supported, ... */
    GEM_ERR_CUDA = 4,               /* a CUDA runtime call failed; see gem_last_cuda_error() */
    GEM_ERR_DEVICE_FLAG = 5,        /* gem_device_status() found a device-side flag set */
    GEM_ERR_TIMEOUT = 6,            /* a device-side wait gave up (GEM_DEVFLAG_TIMEOUT) */
    GEM_ERR_WORKSPACE = 7           /* workspace missing or smaller than the query returned */
} gem_status;

/* Device-side flag bits. */
#define GEM_DEVFLAG_POS_RANGE 1 /* pos[b] < 0, or pos[b] >= cache_cap for full attention */
#define GEM_DEVFLAG_TIMEOUT 2   /* a bounded wait on an asynchronous copy gave up */

/* Static description of a status code. */
GEM_API const char *gem_status_string(int status);
/* cudaError_t of the last CUDA failure seen by a gem_* call on this thread (0 = none). */
GEM_API int gem_last_cuda_error(void);
/* Library version, major * 10000 + minor * 100 + patch. */
GEM_API int gem_version(void);

/* Synchronously read (and, if reset != 0, clear) the library's device-side flag word on
 * the current device.  *flags receives the GEM_DEVFLAG_* bits.  Returns GEM_OK or
 * GEM_ERR_CUDA.  Not for use inside stream capture. */
GEM_API gem_status gem_device_status(int32_t *flags, int reset);

/* The status that a set of GEM_DEVFLAG_* bits (from gem_device_status() or a caller's own
 * status word) stands for: GEM_ERR_TIMEOUT when GEM_DEVFLAG_TIMEOUT is set, else
 * GEM_ERR_DEVICE_FLAG when any other bit is set, else GEM_OK.  Host only; no device call. */
GEM_API gem_status gem_status_from_flags(int32_t flags);

/*
 * Failure detection controls.  The pages have no counterpart of these calls: they let a
 * caller bound how long a kernel may wait for a copy or a grid barrier, and let tests make
 * one such wait run out without faulting or hanging the GPU.
 *
 * gem_set_wait_limit  sets the wall-time limit of every device-side wait (mbarrier waits on
 *         asynchronous copies, grid barriers of gem_decode_step) on the current device, in
 *         nanoseconds; 0 restores the default of 1 s.  Accepted range 1000 .. 60e9 ns, else
 *         GEM_ERR_INVALID_ARG.  A wait that runs out sets GEM_DEVFLAG_TIMEOUT, lets the
 *         copies it issued land (again bounded) and leaves the kernel; the outputs of that
 *         call are then unspecified.  Synchronous: call it while no library kernel runs on
 *         the device, outside stream capture.
 * gem_set_test_injection  sets GEM_INJECT_* bits on the current device (0 clears them),
 *         same synchronisation rules.  While set:
 *           GEM_INJECT_RING_SHORTFALL  the one-row Q4_0 GEMV (B = 1, K % 256 == 0) makes
 *             CTA 0 expect 16 bytes more than its last ring stage receives, so that stage's
 *             wait runs out after the wait limit (every copy still lands);
 *           GEM_INJECT_GRID_ARRIVAL  gem_decode_step makes CTA 0 leave out its arrival at
 *             the step's first grid barrier, so every CTA's barrier wait runs out and the
 *             step is aborted (the plan must then be destroyed and created again).
 *         Meant for tests of the timeout path only.
 */
#define GEM_INJECT_RING_SHORTFALL 1
#define GEM_INJECT_GRID_ARRIVAL 2
GEM_API gem_status gem_set_wait_limit(uint64_t ns);
GEM_API gem_status gem_set_test_injection(int mask);

/*
 * Q4_0 dequantise-and-matvec  [GEM] "Native Metal diagnostic: buffer ownership": the
 * SIMD-group Q4_0 matvec at the 31B FFN shape (5376 -> 21504) and the scalar C check.
 *
 *   y[b][n] = sum_{k<K} ((q[n][k] - 8) * d[n][k/32]) * x[b][k]  (+ residual[b][n])
 *
 *   W        N x (K/32) x 18 bytes, rows contiguous (row stride K/32*18 bytes).
 *   x        [B][ldx] fp32, ldx >= K.       y  [B][ldy] fp32, ldy >= N.
 *   residual nullable, [B][ldy] fp32; may alias y (read before write, element-wise).
 *   Accumulation is fp32 (on tensor cores where K % 256 == 0 and the inputs are aligned: exact
 *   weights times each activation as a binary16 hi + lo pair of about 22 significant bits,
 *   under power-of-two scales that are undone exactly).  y must not overlap W or x.
 *   For B >= 2 and more than 64M weights (N x K, both matrices in pair mode) on the tensor-core
 *   path the call converts x into tensor-core operand records first (a second launch on the
 *   same stream), kept in a library-owned array of 4 MiB per device (K <= 130816): calls on two
 *   streams of one device that may run at the same time must not both be such calls.  Use
 *   gem_q4_0_gemv_ws to give each call its own records instead.  Smaller 2..8-row calls build
 *   their operands inside one launch and use no records.
 */
GEM_API gem_status gem_q4_0_gemv(const void *W, int64_t N, int64_t K, const float *x, int64_t ldx,
                         int B, float *y, int64_t ldy, const float *residual, void *stream);

/*
 * gem_q4_0_gemv with a caller-provided workspace for the operand records of a 2..8-row call,
 * so calls on concurrently running streams share no state.  Same arithmetic, layout and
 * errors as gem_q4_0_gemv, plus:
 *   workspace  device scratch of gem_q4_0_gemv_workspace(B, K) bytes, 256-byte aligned
 *              (else GEM_ERR_MISALIGNED); contents need no initialisation.  When the query
 *              returns 0 (B = 1) workspace may be NULL; otherwise a missing or smaller
 *              workspace is GEM_ERR_WORKSPACE and nothing is launched.
 */
GEM_API size_t gem_q4_0_gemv_workspace(int B, int64_t K);
GEM_API gem_status gem_q4_0_gemv_ws(const void *W, int64_t N, int64_t K, const float *x,
                                    int64_t ldx, int B, float *y, int64_t ldy,
                                    const float *residual, void *workspace, size_t ws_bytes,
                                    void *stream);

/*
 * The Q4_0 GEMV with the pre-norm and the gated activation fused in: the form the layer step
 * runs for its QKV projection (norm), its gate/up pair (norm, two matrices, activation) and
 * its O / down projections (residual).  [GELO] 06 block topology (pre-norm before the merged
 * QKV and before the merged gate/up projections, gated activation); [GEM] "Native Metal
 * diagnostic: buffer ownership" (the gate+up two-matrix single launch).
 *
 *   xh[b]  = gamma ? x[b] / sqrt(mean_k x[b][k]^2 + eps) * gamma : x[b]
 *   W1 NULL:  y[b][n] = sum_k deq(W0)[n][k] xh[b][k]  (+ residual[b][n])
 *   W1 set:   y[b][n] = act(sum_k deq(W0)[n][k] xh[b][k]) * sum_k deq(W1)[n][k] xh[b][k]
 *             act 0: silu, 1: gelu_tanh (as gem_swiglu); residual must be NULL.
 *   W0, W1  N x K Q4_0 (same layout as gem_q4_0_gemv); gamma [K] fp32 or NULL; eps >= 0.
 *   Other arguments, the workspace (gem_q4_0_gemv_workspace(B, K) bytes for B >= 2) and the
 *   errors are those of gem_q4_0_gemv_ws.
 */
GEM_API gem_status gem_q4_0_gemv_fused(const void *W0, const void *W1, int64_t N, int64_t K,
                                       const float *x, int64_t ldx, int B, const float *gamma,
                                       float eps, int act, float *y, int64_t ldy,
                                       const float *residual, void *workspace, size_t ws_bytes,
                                       void *stream);

/*
 * Batched prefill Q4_0 GEMM: M = 1..32 activation rows (prompt tokens) through one matrix (or a
 * gate/up pair), each weight streamed from HBM once and reused by every row.  [GEM] "Native
 * Metal diagnostic: buffer ownership" (the batched-Q4 prefill operator: a dequantised weight tile
 * reused across up to 32 prompt rows with fp32 accumulation, measured in rows/s at the 31B FFN
 * shape).  Arithmetic, layouts and the optional norm / pair / activation / residual are those of
 * gem_q4_0_gemv_fused with B = M; the weights stay exact ((q - 8) * d, no rounding to half).
 *   M        0..32 (M <= 8 runs the decode kernels; 9..32 the column-tiled prefill kernel).
 *   workspace  gem_q4_0_gemm_workspace(M, K) bytes (0 for M = 1), 256-byte aligned, no
 *            initialisation: 4 * M * K bytes of operand records plus a row table.
 */
GEM_API size_t gem_q4_0_gemm_workspace(int M, int64_t K);
GEM_API gem_status gem_q4_0_gemm(const void *W0, const void *W1, int64_t N, int64_t K,
                                 const float *x, int64_t ldx, int M, const float *gamma, float eps,
                                 int act, float *y, int64_t ldy, const float *residual,
                                 void *workspace, size_t ws_bytes, void *stream);

/*
 * Q8_0 dequantise-and-matvec: the tied token embedding / output (logit) projection.
 * [GEM] "Verified model facts" (the published layout keeps the tied embedding as Q8_0) and
 * "Native Metal diagnostic: buffer ownership" (the Q8 logit matvec, one token, and the
 * fixed-eight-row form for a verifier at the 5,376 x 262,144 shape).
 *
 *   y[b][n] = sum_{k<K} (q[n][k] * d[n][k/32]) * x[b][k]
 *
 *   W   N rows of K/32 blocks of 34 bytes: binary16 scale d (little endian), then 32 int8
 *       codes q (element j of the block in byte 2 + j); 16-byte aligned (GEM_ERR_MISALIGNED).
 *   K   a multiple of 256 (GEM_ERR_UNSUPPORTED_SHAPE otherwise); B in 0..8.
 *   x   [B][ldx] fp32, ldx >= K, 16-byte aligned with ldx % 4 == 0 (GEM_ERR_MISALIGNED);
 *   y   [B][ldy] fp32, ldy >= N.  Accumulation is fp32: the products are formed on tensor
 *       cores from the exact codes and each activation as a binary16 hi + lo pair (about 22
 *       significant bits; each activation row is first scaled by a power of two, so any
 *       finite fp32 magnitude is kept).
 */
GEM_API gem_status gem_q8_0_gemv(const void *W, int64_t N, int64_t K, const float *x, int64_t ldx,
                                 int B, float *y, int64_t ldy, void *stream);

/*
 * Index of the largest value of each row: idx[b] = argmax_n y[b][n] (the next token of greedy
 * decoding).  [GEM] sampler note: equal logits go to the lowest token id.  Reading where the
 * pages are silent: a NaN is never chosen; a row of only NaN gives 0.
 *   y    [B][ldy] fp32 (ldy >= N, N < 2^31);  idx  [B] int32 device.
 *   workspace  gem_argmax_workspace(B, N) bytes, 256-byte aligned, contents need no
 *        initialisation (the call clears its arrival counters with a memset on the stream).
 *   Deterministic: chunk maxima are combined under a total order (value, then index).
 */
GEM_API size_t gem_argmax_workspace(int B, int64_t N);
GEM_API gem_status gem_argmax(const float *y, int64_t ldy, int B, int64_t N, int32_t *idx,
                              void *workspace, size_t ws_bytes, void *stream);

/*
 * Device top-k of logit rows: the sampler's candidate list.  [GEM] "Native Metal diagnostic:
 * buffer ownership" (the top-k sampler: a seeded test matches the full-sort token sequence,
 * equal logits broken by token id).
 *   idx[b][r], val[b][r] (r < k): the k largest entries of row b, largest first; equal values
 *   by lowest index; entries that are not numbers after every number, by index (so r = 0 is
 *   gem_argmax's index whenever the row holds a number).  val copies y bit for bit.
 *   y [B][ldy] fp32; 1 <= k <= 64, k <= N; N up to 2048 / k * 8192 (262,144 at k = 64), else
 *   GEM_ERR_UNSUPPORTED_SHAPE.  Workspace: gem_topk_workspace(B, N, k) bytes, 256-byte
 *   aligned, no initialisation (the call zeroes its arrival counters with a 4 * B-byte
 *   memset on the stream).  Deterministic.
 */
GEM_API size_t gem_topk_workspace(int B, int64_t N, int k);
GEM_API gem_status gem_topk(const float *y, int64_t ldy, int B, int64_t N, int k, int32_t *idx,
                            float *val, void *workspace, size_t ws_bytes, void *stream);

/*
 * Weighted RMSNorm  [GEM] "weighted RMSNorm over one or many heads"; [GELO] 06 pre-norm.
 *   out[b][i] = x[b][i] / sqrt(mean_i x[b][i]^2 + eps) * gamma[i]   (gamma NULL: 1)
 * x, out: [B][H] fp32 (may alias).
 */
GEM_API gem_status gem_rmsnorm(const float *x, int B, int64_t H, const float *gamma, float eps,
                       float *out, void *stream);

/*
 * Per-head QK-norm, RoPE and KV append for one new token per sequence.
 *   [GELO] 02/05 (QK-norm: each head's d-slice RMS-normalised with a shared gamma, before
 *   RoPE; p-RoPE rotates only the first rope_dim dims); [GEM] "NeoX/proportional RoPE",
 *   "Verified model facts" (full-attention V = unweighted RMSNorm of the K projection).
 *
 *   qkv      [B][ldqkv] fp32, in place.  Columns: Q heads [0, n_q*d), K heads
 *            [n_q*d, (n_q+n_kv)*d), then V heads (only when v_mode == 0).
 *   gamma_q, gamma_k  [d] fp32, nullable (NULL = no QK-norm for that tensor).
 *   v_mode   0: V rows come from qkv;  1: V = RMSNorm(raw K row) with no weight.
 *   pos      [B] int32 device: the new token's position p (= number of cached positions).
 *   RoPE     NeoX pairing (i, i + rope_dim/2), angle p * theta^(-2i/rope_dim), evaluated in
 *            fp64; rope_dim even, 2 <= rope_dim <= d.
 *   Caches   [B][n_kv][cache_cap][d] binary16; the new K and V rows are written, rounded to
 *            nearest even, at slot p (window == 0) or p mod window (window > 0, a ring of
 *            `window` slots; requires window <= cache_cap).  Q and K in qkv are replaced by
 *            their normalised, rotated fp32 values.
 *            v_mode 1 with k_cache NULL appends the V row only (a compact cache, see
 *            gem_gqa_decode_attn_compact); K in qkv is still normalised and rotated.
 *   status   nullable device int32: receives GEM_DEVFLAG_POS_RANGE for a bad pos[b].
 */
GEM_API gem_status gem_rmsnorm_qknorm_rope(float *qkv, int64_t ldqkv, int B, int n_q, int n_kv,
                                   int d, const float *gamma_q, const float *gamma_k,
                                   int v_mode, float eps, const int32_t *pos, float theta,
                                   int rope_dim, uint16_t *k_cache, uint16_t *v_cache,
                                   int64_t cache_cap, int window, int32_t *status,
                                   void *stream);

/*
 * Grouped-query decode attention, split-K over cache positions with an ordered merge.
 *   [GELO] 02 (GQA, sliding window of the last W tokens), 05 (decode attends
 *   n_kv = n_cache + 1 positions); [GEM] decode-attention notes (attention states over
 *   disjoint token ranges compose; partials summed in ascending partition order).
 *
 *   For sequence b with p = pos[b] and query head h (KV head g = h / (n_q / n_kv)):
 *     slots   S = {0 .. p} (window == 0) or {0 .. min(window, p + 1) - 1} (ring)
 *     out[b][h*d + i] = sum_{s in S} softmax_s(scale * q_h . K[b][g][s]) * V[b][g][s][i]
 *   q       [B][ldq] fp32, query heads contiguous (head h at column h*d); q 16-byte
 *           aligned and ldq % 4 == 0 (else GEM_ERR_MISALIGNED).
 *   caches  [B][n_kv][cache_cap][d] binary16, must already hold the new token's row.
 *   out     [B][ldo] fp32.
 *   d       64, 128, 256 or 512.  n_q % n_kv == 0 and n_q / n_kv <= 8.
 *   workspace  device scratch of gem_gqa_decode_attn_workspace() bytes (same B, n_q, n_kv,
 *           d, cache_cap, window), 256-byte aligned; contents need no initialisation (the
 *           call writes the split partials there and a second launch on the same stream
 *           combines them).  The query returns 0 (workspace may be NULL) where one split
 *           covers the range.
 *   Results are deterministic: the split count depends only on (p, shape, device), and
 *   partial states are merged in ascending split order (by whichever split finishes last).
 */
GEM_API size_t gem_gqa_decode_attn_workspace(int B, int n_q, int n_kv, int d, int64_t cache_cap,
                                     int window);
GEM_API gem_status gem_gqa_decode_attn(const float *q, int64_t ldq, const uint16_t *k_cache,
                               const uint16_t *v_cache, int B, int n_q, int n_kv, int d,
                               int64_t cache_cap, const int32_t *pos, int window, float scale,
                               float *out, int64_t ldo, void *workspace, size_t ws_bytes,
                               int32_t *status, void *stream);

/*
 * QK-norm, RoPE, KV append and decode attention in one call: the form the layer step runs.
 * [GELO] 02/05/06 and [GEM] as for gem_rmsnorm_qknorm_rope and gem_gqa_decode_attn.
 *   Same result as gem_rmsnorm_qknorm_rope(qkv, ...) followed by gem_gqa_decode_attn(q = qkv,
 *   ...): the caches receive the new rows and out the attention output.  For head_dim <= 256
 *   and n_q / n_kv <= 4 it is one launch (the attention kernel normalises and rotates its
 *   query heads and appends the new rows itself, leaving qkv unchanged); other shapes take
 *   the two launches (qkv's Q and K columns are then left normalised and rotated).  Treat
 *   qkv as unspecified after the call.  The workspace is gem_gqa_decode_attn_workspace()'s.
 */
GEM_API gem_status gem_gqa_decode_attn_fused(const float *qkv, int64_t ldqkv, int B, int n_q,
                                             int n_kv, int d, const float *gamma_q,
                                             const float *gamma_k, int v_mode, float eps,
                                             const int32_t *pos, float theta, int rope_dim,
                                             uint16_t *k_cache, uint16_t *v_cache,
                                             int64_t cache_cap, int window, float scale,
                                             float *out, int64_t ldo, void *workspace,
                                             size_t ws_bytes, int32_t *status, void *stream);

/*
 * Decode attention over a compact full-attention cache that keeps V rows only.
 *   [GEM] "Verified model facts": on a full-attention layer V is the unweighted RMSNorm of
 *   the K projection and K is the same normalised row times key_norm (gamma_k), then RoPE, so
 *   the cache can hold V alone and rebuild K inside the attention.  Reading (the record does
 *   not spell out the rotation): the rebuilt row is rotated at its own position,
 *     K_j = RoPE_j(V16_j * gamma_k)    (NeoX pairing on the first rope_dim dims, base theta),
 *   then out as gem_gqa_decode_attn with window 0: softmax over slots 0..p of scale * q.K_j,
 *   applied to V_j.  Half the cache bytes of the standard layout per position.
 *   q        [B][ldq] fp32, query heads normalised and rotated at p (gem_rmsnorm_qknorm_rope).
 *   v_cache  [B][n_kv][cache_cap][d] binary16, 16-byte aligned, already holding slot p.
 *   gamma_k  [d] fp32 device.  rope_dim a multiple of 16, 0 <= rope_dim <= d; theta > 0.
 *   d 64, 128, 256 or 512; n_q % n_kv == 0, n_q / n_kv <= 8.
 *   workspace  gem_gqa_decode_attn_compact_workspace() bytes (0: none needed), 256-byte
 *            aligned, no initialisation.  Splits are merged in ascending order (deterministic).
 *   GEM_ERR_UNSUPPORTED_SHAPE where no split layout fits shared memory.
 */
GEM_API size_t gem_gqa_decode_attn_compact_workspace(int B, int n_q, int n_kv, int d,
                                                     int64_t cache_cap, int rope_dim);
GEM_API gem_status gem_gqa_decode_attn_compact(const float *q, int64_t ldq, const uint16_t *v_cache,
                                               int B, int n_q, int n_kv, int d, int64_t cache_cap,
                                               const int32_t *pos, float scale, const float *gamma_k,
                                               int rope_dim, float theta, float *out, int64_t ldo,
                                               void *workspace, size_t ws_bytes, int32_t *status,
                                               void *stream);

/*
 * gem_gqa_decode_attn without a caller-supplied workspace: the split partials live in a
 * fixed array inside the library, so the call allocates no device memory at all (no
 * cudaMalloc/cudaFree, no allocating library routine).  The decode-attention pages have no
 * counterpart of this entry point; it exists for callers that cannot allocate:
 *   - programs that have handed all device memory to their own arena (weights plus a KV cache
 *     sized to fill HBM), where a new allocation could fail in the middle of decoding;
 *   - serving loops that must not call cudaMalloc/cudaFree per step, since those calls can
 *     synchronise the device and stall the other streams;
 *   - plain C callers that have no device allocator of their own for a scratch buffer.
 * Arguments, results and errors are those of gem_gqa_decode_attn (same kernels, same split
 * plan, so the output is bit-identical to that call's), except:
 *   - the split partials need gem_gqa_decode_attn_workspace() bytes for the same shape,
 *     B * n_q * ns * (d + 2) * 4 bytes where ns is the split count of the plan.  ns grows
 *     with the number of SMs (about SMs / (B * n_kv) splits for d = 512 or n_q / n_kv = 8,
 *     more for the other shapes) and, for d = 512 or n_q / n_kv = 8, with the attended range:
 *     each split covers at most 1024 positions, so ns >= ceil(min(window or cache_cap,
 *     cache_cap) / 1024).  When the need exceeds GEM_ATTN_NOALLOC_SCRATCH_BYTES (8 MiB) the
 *     call launches nothing and returns GEM_ERR_WORKSPACE.  Example on a 152-SM GPU: the
 *     4-KV-head, d = 512, n_q = 32 layer with cache_cap = 32769 fits at B = 1 (38 splits,
 *     2.5 MB) but not at B = 8 (33 splits, 17.4 MB); query gem_gqa_decode_attn_workspace() to
 *     know before calling.
 *   - the array exists once per device and every call on that device shares it.  Calls issued
 *     in order on one stream are safe; two calls that can run at the same time on one device
 *     (different streams, or different host threads with different streams) race on the
 *     array and corrupt each other's outputs.  No part of the array has to start at zero.
 *   - the first call on each device (with that device current) does the set-up: it looks up
 *     the array's device address and sets the kernels' shared-memory limit.  Make that first
 *     call before any stream capture begins.
 */
#define GEM_ATTN_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
GEM_API gem_status gem_gqa_decode_attn_noalloc(const float *q, int64_t ldq,
                                               const uint16_t *k_cache, const uint16_t *v_cache,
                                               int B, int n_q, int n_kv, int d,
                                               int64_t cache_cap, const int32_t *pos, int window,
                                               float scale, float *out, int64_t ldo,
                                               int32_t *status, void *stream);

/*
 * Gated FFN activation  [GELO] 04/05 (Qwen3 SwiGLU; Gemma gelu_pytorch_tanh).
 *   out = act(gate) * up,  act 0: silu(g) = g / (1 + e^-g);
 *                          act 1: 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))).
 *   gate, up, out: [B][F] fp32 contiguous (out may alias either input).
 */
GEM_API gem_status gem_swiglu(const float *gate, const float *up, int B, int64_t F, int act,
                      float *out, void *stream);

/*
 * One decoder layer step for B sequences (one new token each).
 *   [GELO] 06 block topology (pre-norm, merged QKV, QK-norm, RoPE, GQA over the cache,
 *   O projection + residual, pre-FFN norm, merged gate/up, gated activation, down
 *   projection + residual); [GEM] "Verified model facts" (Gemma 4 full-attention layers:
 *   no V projection, V = unweighted RMSNorm of the K projection).
 *
 *   Weight matrices are Q4_0 (see above):
 *     w_qkv  [(n_q + n_kv + (v_from_k ? 0 : n_kv)) * d] x H
 *     w_o    H x (n_q * d)        w_gate, w_up  F x H        w_down  H x F
 *   Norm weights are fp32: g_attn, g_ffn [H]; g_q, g_k [d] (used when qk_norm);
 *   g_post_attn, g_post_ffn [H] (used when post_norms: the O and down projection outputs
 *   are RMS-normalised before each residual add).
 *   act: 0 SiLU, 1 GELU-tanh.  scale: attention score scale.
 */
typedef struct gem_layer_desc {
    int64_t H, n_q, n_kv, d, F;
    float eps, theta, scale;
    int rope_dim, window, act;
    int qk_norm, v_from_k, post_norms;
    const void *w_qkv, *w_o, *w_gate, *w_up, *w_down;
    const float *g_attn, *g_ffn, *g_q, *g_k, *g_post_attn, *g_post_ffn;
    int compact_kv;   /* 1: compact full-attention cache (see gem_gqa_decode_attn_compact);
                         requires v_from_k, qk_norm and window == 0; k_cache may be NULL */
} gem_layer_desc;

/*   x        [B][H] fp32 in/out (the residual stream).
 *   k_cache, v_cache  this layer's caches [B][n_kv][cache_cap][d] binary16 (compact_kv: the
 *            V cache alone; k_cache is ignored and may be NULL).
 *   pos      [B] int32 device positions of the new tokens.
 *   workspace  gem_decode_layer_workspace(L, B, cache_cap) bytes, 256-byte aligned;
 *            contents need no initialisation.
 *   The step is enqueued as a short chain of kernels linked by programmatic dependent
 *   launch, so it can be captured into a CUDA graph for a stack of layers. */
GEM_API size_t gem_decode_layer_workspace(const gem_layer_desc *L, int B, int64_t cache_cap);
GEM_API gem_status gem_decode_layer(const gem_layer_desc *L, int B, float *x, uint16_t *k_cache,
                            uint16_t *v_cache, int64_t cache_cap, const int32_t *pos,
                            void *workspace, size_t ws_bytes, int32_t *status,
                            void *stream);

/*
 * A whole decode step (every layer, one new token per sequence) as ONE persistent launch.
 *   Same arithmetic and results as calling gem_decode_layer for layer 0, 1, ... in order
 *   (within the library's tolerance; summation orders differ).  One CTA per SM: a producer
 *   warp streams every stage of the CTA's weights and cached K/V rows by TMA through a
 *   shared-memory ring, running ahead across layer phases; consumer warps compute the
 *   phases (QKV, attention with QK-norm/RoPE/KV append fused, O, gate/up, down) separated
 *   by grid-wide barriers.  Every device-side wait is bounded: a wait that runs out sets
 *   GEM_DEVFLAG_TIMEOUT and makes every CTA leave the step (x is then unspecified).
 *
 *   gem_step_plan_create  validates the layers and prepares device-resident descriptors
 *            (tensor maps of every weight matrix and cache) and the step's scratch.  It
 *            allocates device memory and synchronises the device: call it once, outside any
 *            stream capture.  layers [nlayers] as for gem_decode_layer; k_caches[l],
 *            v_caches[l]: layer l's caches [B][n_kv][cache_caps[l]][d] binary16 (device
 *            pointers in host arrays; the plan keeps the pointers, not the arrays).
 *            Supported: every layer with the same head_dim d in {64, 128, 256},
 *            n_q / n_kv <= 4, no post_norms, no v_from_k, H, F and n_q * d multiples of
 *            256, B in 1..4, 16-byte aligned weights and caches; otherwise
 *            GEM_ERR_UNSUPPORTED_SHAPE (use gem_decode_layer for those layers).
 *   gem_decode_step  enqueues the step: x [B][H] fp32 in/out (16-byte aligned), pos [B]
 *            int32 device.  The plan's scratch (including grid-barrier and merge counters)
 *            is shared by every call with that plan: calls with one plan must not overlap
 *            (issue them in order on one stream).  Allocates nothing.
 *   gem_step_plan_destroy  frees the plan (after its last step has completed).
 */
typedef struct gem_step_plan gem_step_plan;
GEM_API gem_status gem_step_plan_create(const gem_layer_desc *layers, int nlayers, int B,
                                        uint16_t *const *k_caches, uint16_t *const *v_caches,
                                        const int64_t *cache_caps, gem_step_plan **plan);
GEM_API gem_status gem_decode_step(const gem_step_plan *plan, float *x, const int32_t *pos,
                                   int32_t *status, void *stream);
GEM_API void gem_step_plan_destroy(gem_step_plan *plan);

#ifdef __cplusplus
}
#endif
#endif /* GEM_H */
