/*
 * spec_verify -- batched verify-and-accept step of speculative decoding on
 * one GB300 GPU (sm_103a).
 *
 * The operation is the exact rejection rule of speculative decoding as the
 * lesson "Decodificação Especulativa e EAGLE" (ai-engineering.academy,
 * phase 10 lesson 25) states it in its sections "A Regra de Exatidão"
 * (the rule), "Caso ganancioso" (temperature 0) and "O Conceito / A
 * Configuração com Dois Modelos" (steps 1-4: K drafted tokens, one target
 * pass over K+1 positions, left-to-right acceptance, replacement or bonus
 * token).  For every row b of the batch, with T = temperature[b]:
 *
 *   p_t = softmax(target_logits[b, t, :] / T)   t = 0..K
 *   q_t = softmax(draft_logits[b, t, :] / T)    t = 0..K-1
 *   x_t = draft_tokens[b, t],  r_t = uniforms[b, t],  u = uniforms[b, K]
 *
 *   for t = 0..K-1: accept x_t iff r_t * q_t(x_t) < p_t(x_t); at the first
 *   rejection emit the smallest index i with C_i > u * W, C being the prefix
 *   sum of the residual w = max(p_t - q_t, 0) and W its total, and stop.
 *   If all K are accepted, emit the bonus token chosen the same way from p_K.
 *   T == 0 (greedy): accept iff argmax(target_logits[b, t, :]) == x_t
 *   (lowest index on ties); a rejection or the bonus emits that argmax.
 *
 * If the residual is zero everywhere (p == q to rounding) the replacement is
 * drawn from p_t with u.  Logits may be -inf; NaN and +inf are outside the
 * contract (no fault, unspecified tokens).
 *
 * Conventions for every entry point:
 *   - all array pointers are DEVICE pointers unless stated otherwise; arrays
 *     are dense, row-major, C-contiguous, owned by the caller;
 *   - the library allocates no memory and keeps no state beyond a per-device
 *     cache of the SM count and kernel attributes;
 *   - work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and runs asynchronously: spec_verify never synchronises the
 *     host; inputs must stay unchanged until the stream has run the call;
 *   - kernels are launched as programmatic dependents of the preceding
 *     kernel on the stream, so they may be scheduled while it drains.  Each
 *     waits (griddepcontrol.wait) for that kernel to complete before its
 *     first memory access, so stream order is kept for every read and write
 *     the caller can observe;
 *   - host-detectable errors return a status before anything is launched;
 *     row-level problems found on the device never fault or trap: the row is
 *     written as an error row (accepted_len = -1, all out_tokens -1) and a
 *     flag is OR-ed into the workspace (see spec_verify_device_errors);
 *   - the first call on a device fills the per-device cache (SM count,
 *     occupancy, kernel attributes).  After one such call, spec_verify,
 *     spec_verify_ragged, spec_verify_plug and spec_verify_and_plug make no
 *     call that CUDA stream capture forbids, so they may be captured into a CUDA graph and
 *     replayed (buffers and shapes fixed at capture).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* storage type of the logits */
#define SV_F32 0   /* IEEE float32 */
#define SV_BF16 1  /* bfloat16 (upper half of a float32) */

/* status codes returned by the host entry points */
#define SV_OK 0
#define SV_ERR_NULL 1       /* a required pointer is NULL */
#define SV_ERR_SHAPE 2      /* B < 0, K outside [1, SV_MAX_K], V outside [1, spec_verify_max_vocab(dtype)] */
#define SV_ERR_DTYPE 3      /* dtype is neither SV_F32 nor SV_BF16 */
#define SV_ERR_ALIGN 4      /* a pointer is not aligned to its element (workspace: 16 bytes) */
#define SV_ERR_WORKSPACE 5  /* workspace_bytes < spec_verify_workspace_bytes(B, K, V, dtype) */
#define SV_ERR_CUDA 6       /* a CUDA runtime call failed (launch, attribute, copy) */
#define SV_ERR_TOO_LARGE 7  /* spec_verify_static: the shape needs more than SV_STATIC_SCRATCH_BYTES */

/* device-side row flags, OR-ed into the workspace error word */
#define SV_DEV_BAD_TEMPERATURE 1u  /* T negative, NaN, infinite, or in (0, FLT_MIN) */
#define SV_DEV_BAD_TOKEN 2u        /* a drafted token outside [0, V) */
#define SV_DEV_NONFINITE 4u        /* a logit row without a finite maximum or sum */
#define SV_DEV_BAD_K 8u            /* spec_verify_ragged: k_per_row[b] outside [0, K] */
#define SV_DEV_PLUG_CLIPPED 16u    /* spec_verify_plug: a row's tokens did not all fit */
#define SV_DEV_BAD_LENGTH 32u      /* spec_verify_plug: seq_len[b] outside [0, max_len] */
#define SV_DEV_BAD_TREE 64u        /* spec_verify_tree: a parent or node token out of range */
#define SV_DEV_OUT_OF_BOUNDS 256u  /* checked build only (libspec_verify_checked.so, compiled with
                                      -DSV_CHECKED): an index failed its bounds test and the
                                      access was skipped */

#define SV_MAX_K 16
#define SV_MAX_TREE_NODES 128

/*
 * Bytes of scratch the caller must pass to spec_verify for this shape.
 * Pure host arithmetic; returns 0 for invalid arguments.
 */
size_t spec_verify_workspace_bytes(int B, int K, int V, int dtype);

/* Largest vocabulary accepted for `dtype` (0 for an unknown dtype). */
int spec_verify_max_vocab(int dtype);

/*
 * The verify-and-accept step for a batch of B rows.
 *
 *   target_logits  [B, K+1, V] of `dtype`; element-aligned.  Rows whose base
 *                  address and pitch (V * element size) are multiples of 16
 *                  bytes take the vectorised path, others a scalar path.
 *   draft_logits   [B, K, V] of `dtype` (not read for rows with T == 0).
 *   draft_tokens   [B, K] int32, the drafted ids x_0..x_{K-1}.
 *   uniforms       [B, K+1] float32 in [0, 1): r_0..r_{K-1}, then u.
 *                  Not read for rows with T == 0.
 *   temperature    [B] float32; 0 selects the greedy rule.
 *   accepted_len   [B] int32 out: accepted drafted tokens, 0..K (-1 = error row).
 *   out_tokens     [B, K+1] int32 out: x_0..x_{n-1}, then the replacement
 *                  or bonus token at slot n = accepted_len; later slots -1.
 *   logp_out       optional [B, K] float32 out (NULL to skip): log p_t(x_t)
 *                  for every drafted position of rows with T > 0; NaN on
 *                  greedy and error rows.
 *   logq_out       optional [B, K] float32 out: log q_t(x_t), same layout.
 *   workspace      device scratch, 16-byte aligned, at least
 *                  spec_verify_workspace_bytes(B, K, V, dtype) bytes; its
 *                  contents need no initialisation and are overwritten (the
 *                  4-byte word at offset 0 then holds the call's SV_DEV_*
 *                  flags).
 *   stream         cudaStream_t to enqueue on.
 *
 * B == 0 is a no-op (pointers may then be NULL).  Returns SV_OK or an
 * SV_ERR_* code; on an error code nothing has been launched.  Two calls
 * that share a workspace must be ordered on the device (same stream).
 *
 * Two launches: a persistent grid of (SM count x resident CTAs) whose warps
 * stream every logit row once and leave one partial per 2 KB tile, then G
 * CTAs per batch row that fold the row's statistics, run the acceptance
 * scan, weigh the sampled position's rows tile by tile and locate the
 * token.  No kernel waits on another's flags: the second launch waits for
 * the first (griddepcontrol.wait) and its CTAs meet through one atomic
 * ticket per row.
 */
int spec_verify(const void* target_logits, const void* draft_logits, int dtype,
                const int32_t* draft_tokens, const float* uniforms,
                const float* temperature, int B, int K, int V,
                int32_t* accepted_len, int32_t* out_tokens,
                float* logp_out, float* logq_out,
                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Adaptive verification: row b verifies only its first K_b = k_per_row[b]
 * drafted tokens (0 <= K_b <= K), as the stream transcript "IA local 202:
 * acelere muito a geração com speculative decoding" (44:15-45:16, "adaptive
 * verification") describes validating a different number of drafted
 * tokens per request.
 *
 * The arrays keep spec_verify's padded [B, K+1] / [B, K] layouts with K the
 * largest length.  Row b reads target rows 0..K_b, draft rows 0..K_b-1 (T > 0
 * only), tokens x_0..x_{K_b-1}, acceptance draws r_0..r_{K_b-1} and its
 * replacement/bonus draw u = uniforms[b, K_b]; nothing past its prefix is
 * read.  It is spec_verify's rule on that prefix:
 *   accepted_len[b]     0..K_b;
 *   out_tokens[b, :]    accepted_len + 1 tokens, then -1 up to slot K;
 *   logp_out / logq_out positions K_b..K-1 are NaN.
 * K_b outside [0, K] makes an error row (accepted_len = -1, all tokens -1)
 * and sets SV_DEV_BAD_K.
 *
 *   k_per_row   [B] int32, device, 4-byte aligned (NULL -> SV_ERR_NULL).
 * Every other argument and the return codes are those of spec_verify; the
 * workspace size is spec_verify_workspace_bytes(B, K, V, dtype).
 */
int spec_verify_ragged(const void* target_logits, const void* draft_logits, int dtype,
                       const int32_t* draft_tokens, const float* uniforms,
                       const float* temperature, const int32_t* k_per_row,
                       int B, int K, int V,
                       int32_t* accepted_len, int32_t* out_tokens,
                       float* logp_out, float* logq_out,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * The streaming launch of spec_verify alone.  Every logit row that
 * spec_verify (k_per_row == NULL) or spec_verify_ragged (k_per_row given)
 * reads is read once, and one partial per 2 KB tile of it is written to
 * `workspace` (at least spec_verify_workspace_bytes(B, K, V, dtype)
 * bytes); the flag word and the draw tickets are cleared.  The partials
 * are the library's internal intermediate, the ones spec_verify's second
 * launch folds: this call produces no output of the step and exists to
 * time or profile the streaming pass on its own.  Arguments as in
 * spec_verify_ragged; draft_tokens, uniforms and the outputs are not
 * needed.  Returns SV_OK, SV_ERR_DTYPE, SV_ERR_SHAPE, SV_ERR_NULL,
 * SV_ERR_ALIGN, SV_ERR_WORKSPACE or SV_ERR_CUDA.
 */
int spec_verify_row_stats(const void* target_logits, const void* draft_logits, int dtype,
                          const float* temperature, const int32_t* k_per_row, int B, int K, int V,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Reads the device-side row flags (SV_DEV_*) that the last spec_verify call
 * on this workspace OR-ed in.  Enqueues a 4-byte copy on `stream` and
 * SYNCHRONISES that stream; `flags` is a HOST pointer.  Returns SV_OK,
 * SV_ERR_NULL or SV_ERR_CUDA.
 */
int spec_verify_device_errors(const void* workspace, void* stream, uint32_t* flags);

/*
 * Bytes of the library's own device scratch used by spec_verify_static
 * (8 MiB, one array per device, part of the loaded module).
 */
#define SV_STATIC_SCRATCH_BYTES (8u << 20)

/*
 * spec_verify without a caller workspace and without any allocation.
 *
 * The lesson that states the rule has no counterpart of this call: it is a
 * convenience of this library for callers that cannot hand over, or must
 * not allocate, device scratch at call time.  Arguments, outputs and
 * return codes are those of spec_verify minus `workspace` and
 * `workspace_bytes`; the kernels and their arithmetic are the same, so the
 * results equal spec_verify's.
 *
 * The scratch is a file-scope device array of SV_STATIC_SCRATCH_BYTES bytes
 * (256-byte aligned) in this library.  Shapes whose
 * spec_verify_workspace_bytes(B, K, V, dtype) exceeds that size are
 * rejected with SV_ERR_TOO_LARGE before anything touches the device (at
 * V = 128256 bf16 and K = 4 that admits B up to 639).  Nothing in the
 * scratch must start at zero: the streaming launch resets its flag word and
 * tickets and writes every partial before the draw launch reads it.
 *
 * Setup: the first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it; a failed lookup returns
 * SV_ERR_CUDA.  Make that first call on each device before any stream
 * capture begins.  No call allocates memory (no cudaMalloc, no cudaFree,
 * no allocating library routine).
 *
 * There is ONE scratch per device: calls that may overlap on the device
 * (different streams without an ordering between them, or several host
 * threads) race on it and may return wrong tokens.  Order all calls on a
 * device, e.g. on one stream.  The device row flags of these calls are
 * kept in that scratch (error rows still show as accepted_len = -1); read
 * them with spec_verify_static_device_errors.
 */
int spec_verify_static(const void* target_logits, const void* draft_logits, int dtype,
                       const int32_t* draft_tokens, const float* uniforms,
                       const float* temperature, int B, int K, int V,
                       int32_t* accepted_len, int32_t* out_tokens,
                       float* logp_out, float* logq_out, void* stream);

/*
 * The SV_DEV_* flags of the last spec_verify_static call on the current
 * device: the 4-byte flag word of the static scratch, copied to the host
 * pointer `flags` on `stream` (which is then synchronised).  Call it on the
 * stream (or after the stream order) of the spec_verify_static call whose
 * flags are wanted; a later static call overwrites them.  Returns SV_OK,
 * SV_ERR_NULL (flags == NULL) or SV_ERR_CUDA.
 */
int spec_verify_static_device_errors(void* stream, uint32_t* flags);

/*
 * Greedy verification of a draft tree per row.  The lesson's section
 * "Verificação de Atenção em Árvore" checks every node of the tree in one
 * target pass and keeps the longest prefix along an accepted path.  Its
 * exercise 4 asks that the target accept the longest correct branch.
 *
 *   target_logits  [B, N+1, V] of dtype: slot 0 follows the context (the
 *                  root), slot i+1 follows node i.
 *   node_tokens    [B, N] int32: the token of every node.
 *   parents        [B, N] int32: -1 (a child of the root) or an earlier node
 *                  (parents[b, i] < i; breadth-first order satisfies this).
 *   accepted_len   [B] int32 out: depth of the accepted path, 0..N (-1 = error row).
 *   out_tokens     [B, N+1] int32 out: the tokens along the path, then the
 *                  target's argmax at its last node's slot (the root's slot
 *                  if no node is accepted), then -1.
 *   accepted_nodes [B, N] int32 out, may be NULL: the node indices along the
 *                  path, then -1.
 *   workspace      at least spec_verify_tree_workspace_bytes(B, N, V, dtype)
 *                  bytes, 16-byte aligned; needs no initialisation.
 *
 * Node i is accepted iff its parent is the root or accepted, and its token
 * equals argmax(target slot of the parent) (lowest index on ties).  The
 * deepest accepted node wins, with the lowest node index on ties.  A parent
 * outside [-1, i), a node token outside [0, V) or a slot with no finite
 * maximum makes an error row and sets SV_DEV_BAD_TREE / SV_DEV_NONFINITE
 * (read with spec_verify_device_errors).  1 <= N <= SV_MAX_TREE_NODES.
 * Returns the status codes of spec_verify.
 */
size_t spec_verify_tree_workspace_bytes(int B, int N, int V, int dtype);

int spec_verify_tree(const void* target_logits, int dtype, const int32_t* node_tokens,
                     const int32_t* parents, int B, int N, int V, int32_t* accepted_len,
                     int32_t* out_tokens, int32_t* accepted_nodes, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * The plug step: append each row's emitted tokens to its sequence buffer
 * and advance its length on the device.  The next decode step can then be
 * launched without reading the accepted lengths back to the host.  The page
 * "Accelerating Sonar through speculation" (single-token MTP schedule) plugs
 * the next target tokens into their places with a kernel, because the
 * accepted count otherwise forces a GPU-to-CPU sync.
 *
 *   accepted_len [B]        int32, device: spec_verify's output (-1 = error row).
 *   out_tokens   [B, K+1]   int32, device: spec_verify's output.
 *   tokens       [B, max_len] int32, device, in/out: each row's sequence.
 *   seq_len      [B]        int32, device, in/out: each row's current length.
 *   last_token   [B]        int32, device, out, may be NULL: the last emitted
 *                           token of each row (unchanged for rows not appended).
 *   flags        one uint32, device, may be NULL: OR-ed with SV_DEV_PLUG_CLIPPED
 *                or SV_DEV_BAD_LENGTH.
 *
 * For row b with n = accepted_len[b] >= 0 and L = seq_len[b] in
 * [0, max_len], out_tokens[b, 0..n] goes to tokens[b, L..L+n] and seq_len[b]
 * becomes L + n + 1.  Tokens that would land at or past max_len are dropped;
 * seq_len then stops at max_len and SV_DEV_PLUG_CLIPPED is set.  Error rows
 * are left unchanged; so are rows with L outside [0, max_len] or with
 * accepted_len[b] > K (not an output of spec_verify), which set
 * SV_DEV_BAD_LENGTH.  Enqueue it on spec_verify's stream, after the call; it
 * does not synchronise.  Returns SV_OK, SV_ERR_SHAPE (B < 0, K outside
 * [1, SV_MAX_K], max_len < 1), SV_ERR_NULL, SV_ERR_ALIGN or SV_ERR_CUDA.
 */
int spec_verify_plug(const int32_t* accepted_len, const int32_t* out_tokens, int B, int K,
                     int32_t* tokens, int32_t* seq_len, int max_len, int32_t* last_token,
                     uint32_t* flags, void* stream);

/*
 * spec_verify (or spec_verify_ragged) with the plug step fused into its
 * draw launch: one call, the same two launches as spec_verify, no third
 * launch for the plug.  The warp that writes a row's last token also appends the row's emitted tokens to
 * `tokens` and advances `seq_len`, with exactly
 * spec_verify_plug's rule: same arguments (tokens, seq_len, max_len,
 * last_token), same results.  Its SV_DEV_PLUG_CLIPPED / SV_DEV_BAD_LENGTH
 * flags go to the workspace word with the call's other device flags (read
 * them with spec_verify_device_errors).
 *
 *   k_per_row  [B] int32, device, or NULL (every row verifies K).
 * Every other argument is that of spec_verify or spec_verify_plug.  Returns
 * spec_verify's codes, SV_ERR_SHAPE for max_len < 1, SV_ERR_NULL for a NULL
 * tokens or seq_len, and SV_ERR_ALIGN for a misaligned int32 array.
 */
int spec_verify_and_plug(const void* target_logits, const void* draft_logits, int dtype,
                         const int32_t* draft_tokens, const float* uniforms,
                         const float* temperature, const int32_t* k_per_row,
                         int B, int K, int V,
                         int32_t* accepted_len, int32_t* out_tokens,
                         float* logp_out, float* logq_out,
                         int32_t* tokens, int32_t* seq_len, int max_len, int32_t* last_token,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Static, NUL-terminated description of a status code. */
const char* spec_verify_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
