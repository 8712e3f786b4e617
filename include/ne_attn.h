/*
 * ne_attn.h -- C ABI of the GB300 (sm_103a) causal grouped-query attention
 * library with rotary position embeddings: forward and backward.
 *
 * What is computed.  The attention of a NanoEuler-style decoder block
 * ("NanoEuler: a GPT-2-scale LLM built from scratch in C and CUDA",
 * technical specification: RoPE applied to queries and keys, grouped-query
 * attention sharing a smaller set of key/value heads, decoder-only; the
 * "CUDA engine" section: a hand-written FlashAttention kernel that tiles the
 * computation and uses an online softmax so the T x T matrix is never stored).
 * With G = Hq / Hkv and kv(h) = floor(h / G):
 *
 *   q'[t,h]  = R(t) q[t,h],  k'[s,j] = R(s) k[s,j]        (rotate-half RoPE:
 *              pairs (i, i + d/2) rotated by angle pos * theta^(-2i/d))
 *   S[t,s]   = <q'[t,h], k'[s,kv(h)]> / sqrt(d)  for s <= t (causal)
 *   lse[t]   = ln sum_{s<=t} exp S[t,s]
 *   O[t,h]   = sum_{s<=t} exp(S[t,s] - lse[t]) v[s,kv(h)]
 *
 * and the backward of L = sum(O * dO) with respect to the pre-RoPE q, k and
 * v; dk and dv are summed over the G query heads sharing each key/value head.
 * Variants below: a training pair that hands the rotated Q' and K' from the
 * forward to the backward, a sliding window (keys t-W+1 .. t), decode of one
 * new token per sequence against a key/value cache, and a backward that
 * allocates nothing.
 *
 * Layouts (all row-major, contiguous, no padding):
 *   q, o, dO, dq : bf16 [B][T][Hq][d]
 *   k, v, dk, dv : bf16 [B][T][Hkv][d]
 *   lse          : fp32 [B][Hq][T]     natural-log logsumexp of the scaled scores
 *
 * Ownership.  The caller allocates and owns every buffer (device memory for
 * tensors; the library allocates no memory).  Outputs are overwritten, never
 * accumulated into.  Calls are asynchronous on `stream` (a cudaStream_t
 * passed as void*, NULL = the legacy default stream); the caller keeps
 * buffers alive until the stream has passed the call.  The library is
 * reentrant; its only global state is one device status word per GPU that
 * records device-side errors (read and cleared by ne_attn_get_error).
 *
 * Preconditions: B, T >= 1 (T <= 2^24); Hq, Hkv >= 1 and Hq % Hkv == 0; d in
 * {32, 64, 128}; rope_theta > 0 and finite; tensor and workspace pointers
 * 16-byte aligned, lse 4-byte aligned; the current device is an sm_103 GPU.
 * Score-side operands (the rotated q and k, and the backward's dS) go
 * through the tensor cores as fp16, so elements of q and k,
 * and of dS = P (dP - D), must stay below 65504 in magnitude; a kernel that
 * sees a larger value records NE_ERR_RANGE in the status word.
 * RoPE angles are evaluated from each frequency rounded to a 64-bit
 * fixed-point fraction of a turn, times the position (exact modulo one turn
 * but for the dropped low word, under 2^-32 turn), so the angle is reduced
 * exactly into [-pi, pi) at every position and its error does not grow with
 * T: about 2e-7 radians from the float conversion, plus the hardware
 * sine/cosine error.
 *
 * Score precision.  The forward rounds q' and k' to fp16 for the tensor
 * cores, so a score carries a rounding error proportional to |q'| |k'|.  A
 * row whose rotated vector has mean square above 4 (|x'|^2 > 4 d, e.g. a row
 * drawn at several times the scale of the others; unit-variance rows reach
 * it with probability below 1e-12) is scored exactly instead: the forward
 * recomputes such a query row in fp32 from the bf16 inputs, and corrects
 * every row that sees such a key row by the exact softmax weight of that
 * pair.  The persistent forward runs one CTA per SM, each on a fixed share
 * of the query tiles; each CTA handles up to 48 such rows (the large query
 * rows of its tiles and the distinct large key rows they see).  Beyond that
 * the call records NE_WARN_PRECISION (the results are complete, with the
 * fp16 error on the pairs of the rows left over).  Within these limits lse
 * is within 1e-3 absolute of the exact result for unit-scale inputs, the
 * stated tolerance.  The backward uses the fp16 scores throughout.
 *
 * Errors.  Argument errors are returned synchronously and launch nothing.
 * Launch failures return NE_ERR_CUDA.  Device-side errors (a bounded wait
 * that ran out, a value out of fp16 range) and the precision warning are
 * recorded in the device status word and reported by ne_attn_get_error.  Nothing aborts, prints or
 * throws across this interface, and there is no CPU fallback.
 */
#ifndef NE_ATTN_H
#define NE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NE_OK = 0,
    NE_ERR_NULL = 1,        /* a required pointer is NULL */
    NE_ERR_SHAPE = 2,       /* B, T, Hq, Hkv out of range or Hq % Hkv != 0 */
    NE_ERR_UNSUPPORTED = 3, /* d not in {32, 64, 128}, or the device is not sm_103 */
    NE_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned */
    NE_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than ne_attn_bwd_workspace_size */
    NE_ERR_CUDA = 6,        /* a CUDA runtime / driver call or a launch failed */
    NE_ERR_TIMEOUT = 7,     /* a device-side bounded wait ran out (reported by get_error) */
    NE_ERR_RANGE = 8,       /* an fp16 tensor-core operand overflowed (reported by get_error) */
    NE_ERR_ARG = 9,         /* another invalid argument (rope_theta <= 0, NaN, a length
                               out of range, ...) */
    NE_ERR_TOO_LARGE = 10,  /* ne_attn_bwd_noalloc: shape exceeds its fixed scratch */
    NE_WARN_PRECISION = 11  /* a forward tile held more large-norm rows than it scores exactly
                               (reported by get_error; see "Score precision" above) */
} ne_status;

/*
 * Forward.  Reads q, k, v; writes o and lse.
 * Section "CUDA engine / kernel implementation" of the NanoEuler README page
 * (tiled FlashAttention with online softmax); RoPE and GQA from its
 * technical specification.
 */
int ne_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                int B, int T, int Hq, int Hkv, int d, float rope_theta, void *stream);

/*
 * Bytes of device workspace ne_attn_bwd needs for this shape: the per-row
 * dO.O dot products D (fp32 [B][Hq][T]), the rotated queries Q' = R(t) q
 * (fp16 [B][T][Hq][d]) and the rotated keys K' = R(s) k (fp16
 * [B][T][Hkv][d]), each rounded up to 256 bytes.
 * Returns 0 for a shape ne_attn_bwd would reject.
 */
size_t ne_attn_bwd_workspace_size(int B, int T, int Hq, int Hkv, int d);

/*
 * Backward of L = sum(O * dO).  Reads q, k, v, o, lse (as written by
 * ne_attn_fwd for the same inputs) and dO; writes dq, dk, dv (gradients with
 * respect to the pre-RoPE q and k, and v).  `workspace` is caller-owned
 * device memory of at least ne_attn_bwd_workspace_size(...) bytes; its
 * contents on entry do not matter.  Deterministic: no floating-point atomics,
 * so repeated calls on the same inputs give bitwise-equal results.
 * The pages validate the hand-written backward by central finite differences
 * in double precision (NanoEuler walkthrough, section 2.1).
 */
int ne_attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                const void *dO, void *dq, void *dk, void *dv, void *workspace,
                size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d,
                float rope_theta, void *stream);

/*
 * Training pair.  ne_attn_fwd_save is ne_attn_fwd that also leaves the
 * rotated Q' = R(t) q and K' = R(s) k (fp16) in `workspace` (at least
 * ne_attn_bwd_workspace_size(...) bytes, 16-byte aligned, caller-owned), in
 * the layout ne_attn_bwd uses; the forward rotates every Q and K tile in
 * shared memory anyway, so this saves the backward from reading q and k and
 * rotating them again.  ne_attn_bwd_saved is ne_attn_bwd for a workspace
 * filled that way: its preprocess computes D only.  q and k are validated
 * but not read by ne_attn_bwd_saved; the workspace must come from
 * ne_attn_fwd_save on the same q, k, shape and rope_theta, unchanged since
 * (the library cannot check this).  Results equal those of ne_attn_fwd
 * followed by ne_attn_bwd, bit for bit.  Errors as for ne_attn_fwd and
 * ne_attn_bwd (NE_ERR_WORKSPACE for a missing or short workspace).
 * `window` is the sliding window of ne_attn_fwd_window (0: causal); both
 * calls of a pair take the same value.
 */
/*
 * ne_attn_bwd_saved runs these three steps: ne_attn_bwd_preprocess_d (D only,
 * into the workspace; no rope_theta needed), then ne_attn_bwd_dq and
 * ne_attn_bwd_dkdv below, which read Q' and K' from the workspace.
 */
int ne_attn_bwd_preprocess_d(const void *o, const void *dO, void *workspace,
                             size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d,
                             void *stream);
int ne_attn_fwd_save(const void *q, const void *k, const void *v, void *o, float *lse,
                     void *workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv,
                     int d, float rope_theta, int window, void *stream);
int ne_attn_bwd_saved(const void *q, const void *k, const void *v, const void *o,
                      const float *lse, const void *dO, void *dq, void *dk, void *dv,
                      void *workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv,
                      int d, float rope_theta, int window, void *stream);

/*
 * The three steps ne_attn_bwd runs, in this order, exposed so a caller can
 * time them or run the two independent steps (dq, and dk/dv) on two streams
 * once the preprocess has finished.  Arguments mean what they mean for
 * ne_attn_bwd; `workspace` carries D from the preprocess to the other two.
 *
 * ne_attn_bwd_preprocess: D[b][h][t] = sum_c dO[b,t,h,c] * O[b,t,h,c] in fp32
 *   (the row dot product the backward of a softmax needs) and the rotated
 *   Q' = R(t) q and K' = R(s) k in fp16, all written into the workspace.
 * ne_attn_bwd_dq: dq from q, k, v, lse, dO and D (query-tile major: recomputes
 *   the scores and dP = dO v^T per key tile; dq = R(t)^T sum_s dS k' / sqrt(d)).
 * ne_attn_bwd_dkdv: dk and dv from v, lse, dO and the workspace's D, Q', K'
 *   (key-tile major: dk and dv summed over the query heads of each key/value
 *   head inside one CTA); `q` and `k` are validated, the kernel reads Q', K'.
 */
int ne_attn_bwd_preprocess(const void *q, const void *k, const void *o, const void *dO,
                           void *workspace, size_t workspace_bytes, int B, int T, int Hq,
                           int Hkv, int d, float rope_theta, void *stream);
int ne_attn_bwd_dq(const void *q, const void *k, const void *v, const float *lse,
                   const void *dO, void *dq, const void *workspace, size_t workspace_bytes,
                   int B, int T, int Hq, int Hkv, int d, float rope_theta, void *stream);
int ne_attn_bwd_dkdv(const void *q, const void *k, const void *v, const float *lse,
                     const void *dO, void *dk, void *dv, const void *workspace,
                     size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d,
                     float rope_theta, void *stream);

/*
 * Sliding-window variants (the per-layer window pattern of the nanochat
 * guide): query t attends to keys t-W+1 .. t only, W = `window` >= 1; W = 0
 * is the causal mask of ne_attn_fwd / ne_attn_bwd (W >= T gives the same
 * result).  Everything else (arguments, layouts, workspace, errors) as for
 * ne_attn_fwd and ne_attn_bwd; a negative window returns NE_ERR_ARG.  Key
 * tiles entirely outside every row's window are skipped.
 */
int ne_attn_fwd_window(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                       int T, int Hq, int Hkv, int d, float rope_theta, int window, void *stream);
int ne_attn_bwd_window(const void *q, const void *k, const void *v, const void *o,
                       const float *lse, const void *dO, void *dq, void *dk, void *dv,
                       void *workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv,
                       int d, float rope_theta, int window, void *stream);

/*
 * Decode against a key/value cache (the chat loop of the NanoEuler README's
 * KV-cache inference engine): one new token per sequence.  Its key and value
 * are the cache's last rows, so it sits at position Tk - 1 and every cached
 * key is visible to it; the result is, by definition, the last row of the
 * causal attention ne_attn_fwd computes over those Tk positions.
 *   q        bf16 [B][Hq][d]      the new tokens' queries, before RoPE
 *   k_cache  bf16 [B][Tk][Hkv][d] keys before RoPE (rotated at their positions)
 *   v_cache  bf16 [B][Tk][Hkv][d]
 *   o        bf16 [B][Hq][d]      written
 *   lse      fp32 [B][Hq]         written, natural log of the scaled scores
 *   workspace, workspace_bytes    caller-owned scratch of at least
 *                                 ne_attn_decode_workspace_size() bytes
 *                                 (16-byte aligned; no initial contents)
 * Preconditions as for ne_attn_fwd, and Hq / Hkv <= 16 (else
 * NE_ERR_UNSUPPORTED).  Asynchronous on `stream`; two kernels (the keys are
 * split into chunks of 128, each chunk's partial softmax is merged in chunk
 * order, so the result is deterministic).  Calls that share a workspace must
 * not overlap on the GPU.  ne_attn_decode_workspace_size returns 0 for an
 * invalid shape.
 */
size_t ne_attn_decode_workspace_size(int B, int Tk, int Hq, int Hkv, int d);
int ne_attn_decode(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                   void *workspace, size_t workspace_bytes, int B, int Tk, int Hq, int Hkv, int d,
                   float rope_theta, void *stream);

/*
 * Padded variable-length batches (the NanoEuler SFT stage pads each
 * instruction/response pair to the context and masks the loss on prompt and
 * padding: walkthrough section 3.2).  Sequence b holds its first
 * seqlens[b] tokens, 0 <= seqlens[b] <= T, at positions 0 .. seqlens[b]-1;
 * the rows after them are padding.  Each sequence is its own causal problem,
 * so its valid rows equal the same rows of ne_attn_fwd on the padded batch;
 * a padding row attends to nothing.
 *   seqlens    int32 [B], HOST memory, read during the call only
 *   workspace  caller-owned device memory (16-byte aligned, no initial
 *              contents) of at least ne_attn_varlen_workspace_size() bytes;
 *              the forward uses only its first part (the work-unit tables,
 *              with room for the device-side plan's counts and scratch)
 * ne_attn_fwd_varlen writes o and lse like ne_attn_fwd on valid rows, and
 * o = 0, lse = -inf on padding rows.  ne_attn_bwd_varlen takes o and lse
 * from ne_attn_fwd_varlen and writes the gradients of the sum of O * dO over
 * the valid rows: dq, dk, dv like ne_attn_bwd on valid positions (dO of
 * padding rows is never used) and 0 on padding positions.
 * Padding rows of q, k, v and dO must hold values the other entry points
 * accept (finite, within the fp16 range after rotation; zeros or a pad
 * token's activations do): tiles that straddle a sequence's end compute over
 * them, with zero weight, before the padding is overwritten.  Query tiles
 * (and, in the backward, key tiles) wholly past a sequence's end are
 * skipped, and the backward's preprocess does not read padding rows.  The library
 * builds the tables of live work units on the host and copies them into the
 * workspace with an asynchronous copy from pageable memory, so these calls
 * cannot be captured into a CUDA graph (the _dev variants below can); calls
 * that share a workspace must not overlap on the GPU.
 * Errors as for ne_attn_fwd / ne_attn_bwd; seqlens NULL gives NE_ERR_NULL, a
 * length outside [0, T] NE_ERR_ARG.  ne_attn_varlen_workspace_size returns 0
 * for an invalid shape.
 */
size_t ne_attn_varlen_workspace_size(int B, int T, int Hq, int Hkv, int d);
int ne_attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                       const int32_t *seqlens, void *workspace, size_t workspace_bytes, int B,
                       int T, int Hq, int Hkv, int d, float rope_theta, void *stream);
int ne_attn_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                       const float *lse, const void *dO, void *dq, void *dk, void *dv,
                       const int32_t *seqlens, void *workspace, size_t workspace_bytes, int B,
                       int T, int Hq, int Hkv, int d, float rope_theta, void *stream);

/*
 * The same with the lengths in DEVICE memory: seqlens_dev int32 [B], 4-byte
 * aligned, read by the GPU in stream order (so a preceding kernel may write
 * it).  A planning kernel builds the tables of live work units in the
 * workspace (the same tables, in the same order, as the host entry points)
 * and the persistent kernels read their unit counts from there, launching
 * one CTA per SM; the host never needs the lengths, so these calls can be
 * captured into a CUDA graph and the graph replayed with other lengths
 * written into the same buffer.  Results equal the host-length entry
 * points' bit for bit.  A length outside [0, T] is clamped into it and
 * reported as NE_ERR_ARG by ne_attn_get_error; seqlens_dev NULL gives
 * NE_ERR_NULL.  Workspace and everything else as above.
 */
int ne_attn_fwd_varlen_dev(const void *q, const void *k, const void *v, void *o, float *lse,
                           const int32_t *seqlens_dev, void *workspace, size_t workspace_bytes,
                           int B, int T, int Hq, int Hkv, int d, float rope_theta, void *stream);
int ne_attn_bwd_varlen_dev(const void *q, const void *k, const void *v, const void *o,
                           const float *lse, const void *dO, void *dq, void *dk, void *dv,
                           const int32_t *seqlens_dev, void *workspace, size_t workspace_bytes,
                           int B, int T, int Hq, int Hkv, int d, float rope_theta, void *stream);

/*
 * Packed variable-length batches: the sequences concatenated along the rows,
 * with no padding (the layout an SFT batch takes when its pairs are packed
 * instead of padded to the context).  Sequence b is rows cu_seqlens[b] ..
 * cu_seqlens[b+1]-1 of the pack, a causal problem of its own whose positions
 * (for RoPE) restart at 0.
 *   q, o, dO, dq  bf16 [total][Hq][d]
 *   k, v, dk, dv  bf16 [total][Hkv][d]
 *   lse           fp32 [Hq][total]
 *   cu_seqlens    int32 [nseq + 1], HOST memory, read during the call only:
 *                 cu_seqlens[0] = 0, non-decreasing, cu_seqlens[nseq] = total
 *                 (empty sequences are allowed)
 *   workspace     caller-owned device memory (16-byte aligned, no initial
 *                 contents) of at least ne_attn_packed_workspace_size() bytes;
 *                 the forward uses only its first part (the work-unit tables)
 * Results equal those of the padded entry points on the same sequences, row
 * for row; every row of the pack is a valid row.  The library builds the
 * tables of work units on the host and copies them into the workspace from
 * pageable memory, so these calls cannot be captured into a CUDA graph (the
 * _dev variants below can);
 * calls that share a workspace must not overlap on the GPU.  Errors as for
 * the padded entry points; cu_seqlens NULL gives NE_ERR_NULL, nseq < 1 or
 * total < 1 NE_ERR_SHAPE, an inconsistent cu_seqlens NE_ERR_ARG.
 * ne_attn_packed_workspace_size returns 0 for an invalid shape.
 */
size_t ne_attn_packed_workspace_size(int nseq, int total, int Hq, int Hkv, int d);
int ne_attn_fwd_packed(const void *q, const void *k, const void *v, void *o, float *lse,
                       const int32_t *cu_seqlens, void *workspace, size_t workspace_bytes,
                       int nseq, int total, int Hq, int Hkv, int d, float rope_theta,
                       void *stream);
int ne_attn_bwd_packed(const void *q, const void *k, const void *v, const void *o,
                       const float *lse, const void *dO, void *dq, void *dk, void *dv,
                       const int32_t *cu_seqlens, void *workspace, size_t workspace_bytes,
                       int nseq, int total, int Hq, int Hkv, int d, float rope_theta,
                       void *stream);

/*
 * The same with cu_seqlens in DEVICE memory (int32 [nseq + 1], 4-byte
 * aligned, read by the GPU in stream order), for CUDA graph capture: the
 * planning kernel of the _dev padded entry points builds the unit tables
 * from it, with the tile bound of one sequence of `total` rows (the host
 * never learns the longest sequence).  The kernels address rows through a
 * sanitised copy in the workspace: a prefix array that does not start at 0,
 * decreases or does not end at total is made monotone within [0, total]
 * and reported as NE_ERR_ARG by ne_attn_get_error.  Results equal the
 * host-array entry points' bit for bit for a valid prefix array.
 */
int ne_attn_fwd_packed_dev(const void *q, const void *k, const void *v, void *o, float *lse,
                           const int32_t *cu_seqlens_dev, void *workspace,
                           size_t workspace_bytes, int nseq, int total, int Hq, int Hkv, int d,
                           float rope_theta, void *stream);
int ne_attn_bwd_packed_dev(const void *q, const void *k, const void *v, const void *o,
                           const float *lse, const void *dO, void *dq, void *dk, void *dv,
                           const int32_t *cu_seqlens_dev, void *workspace,
                           size_t workspace_bytes, int nseq, int total, int Hq, int Hkv, int d,
                           float rope_theta, void *stream);

/*
 * The work units a padded variable-length batch launches (host only; no GPU
 * needed): per-sequence lengths seqlens[B] (host) give counts[0..2], the
 * live units of the forward, dq and dk/dv kernels, and each non-NULL table
 * receives up to `cap` of them as indices into that kernel's full unit
 * enumeration, in launch order (each table is the one the varlen entry
 * points copy into the workspace).  Returns NE_OK; NE_ERR_NULL if seqlens or
 * counts is NULL; NE_ERR_SHAPE / NE_ERR_UNSUPPORTED for a shape
 * ne_attn_fwd_varlen rejects; NE_ERR_ARG for a length outside [0, T].
 */
int ne_attn_varlen_plan(const int32_t *seqlens, int B, int T, int Hq, int Hkv, int d,
                        int32_t *fwd_units, int32_t *dq_units, int32_t *dkv_units, size_t cap,
                        int32_t *counts);

/*
 * Synchronises `stream`, then returns and clears the device-side status of
 * the current device: NE_ERR_TIMEOUT, NE_ERR_RANGE, NE_ERR_ARG (a length in
 * device memory out of range) or NE_WARN_PRECISION (in that order of
 * precedence) if a kernel recorded one since the last call,
 * NE_ERR_CUDA if the stream reports a CUDA error, else NE_OK.
 */
int ne_attn_get_error(void *stream);

/* Static, human-readable text for a status code. */
const char *ne_attn_status_string(int status);

/*
 * Upper bound, in nanoseconds, on every device-side wait of the launches the
 * calling host thread makes afterwards (default 2e9).  Each host thread has
 * its own value, so setting it never changes another thread's launches.  A
 * wait that runs out makes its kernel record NE_ERR_TIMEOUT, drain its own
 * in-flight work and return.
 */
void ne_attn_set_wait_limit_ns(uint64_t limit_ns);

/*
 * Check of the bounded-wait machinery: launches one block whose wait can
 * never be satisfied (a barrier nothing arrives on) under a wait limit of
 * `limit_ns`.  The launch itself returns NE_OK; a following
 * ne_attn_get_error(stream) must then report NE_ERR_TIMEOUT.
 */
int ne_attn_selftest_timeout(uint64_t limit_ns, void *stream);

/*
 * Backward that allocates nothing and takes no workspace.  (This entry point
 * has no counterpart on the pages; it exists for callers of this library.)
 *
 * Who needs it: callers that cannot call cudaMalloc -- code that runs with all
 * device memory already claimed by another allocator (a framework's caching
 * allocator, a fixed per-process memory budget) where a new allocation could
 * fail or fragment, and callers whose own interface gives them no place to
 * pass a workspace pointer through.
 *
 * Same arguments, results and errors as ne_attn_bwd, minus the workspace
 * (argument checks run in ne_attn_bwd's order; NE_ERR_TOO_LARGE takes the
 * place of NE_ERR_WORKSPACE).
 * The scratch ne_attn_bwd keeps in the workspace (D, Q', K') lives instead in
 * one fixed device array of ne_attn_bwd_noalloc_max_scratch() bytes (32 MiB)
 * compiled into the library: every GPU that loads the library holds it until
 * the process exits.  Shapes whose ne_attn_bwd_workspace_size exceeds that
 * return NE_ERR_TOO_LARGE and launch nothing.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  The address is kept for the rest of the process, like the status
 * word's: after cudaDeviceReset the library's device variables live at new
 * addresses, so do not call the library again in that process after a
 * reset.  All calls share the one array: calls that can overlap on the GPU
 * (different streams, or different host threads, on the same device) race on
 * it and must be serialised by the caller.  The array keeps the last call's
 * contents; every byte a call reads is written earlier in that same call, so
 * nothing needs clearing.  No memory is allocated or freed by this call.
 */
int ne_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                        const float *lse, const void *dO, void *dq, void *dk, void *dv, int B,
                        int T, int Hq, int Hkv, int d, float rope_theta, void *stream);

/* Size in bytes of ne_attn_bwd_noalloc's fixed scratch array. */
size_t ne_attn_bwd_noalloc_max_scratch(void);

#ifdef __cplusplus
}
#endif

#endif /* NE_ATTN_H */
