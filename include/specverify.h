/*
 * libspecverify: the verification sampler of speculative decoding on one
 * NVIDIA GB300 (sm_103a).
 *
 * What the library computes (page title, section):
 *   "Decodificación Especulativa y EAGLE" (Phase 10 - Lesson 25),
 *     section "El Concepto": the target scores K+1 positions in one pass; the
 *     drafted tokens are accepted or rejected left to right; a rejection
 *     draws a replacement and stops; if every draft is accepted a bonus token
 *     is drawn from the target at position K+1.
 *     section "La Regla de Exactitud": accept x_t iff r < p(x_t)/q(x_t) with
 *     r ~ U(0,1); otherwise draw from (p - q)+ / ||(p - q)+||_1 and stop.
 *     section "Caso codicioso": at temperature 0 accept iff argmax(p) = x_t,
 *     otherwise emit argmax(p) and stop.
 *   "Accelerating Sonar through speculation", section "Decodificación
 *     especulativa": n drafted tokens yield at most n+1 emitted tokens; the
 *     sampler's accepted lengths are what the scheduler reads back.
 *
 * Notation: request b in [0,B); n_b = draft_len[b] in [1,K]; T_b =
 * temperature[b]; p_{b,t} = softmax(target_logits[b,t,:] / T_b) for t <= n_b;
 * q_{b,t} = softmax(draft_logits[b,t,:] / T_b) for t < n_b.
 *
 * Readings fixed by this interface where the pages are silent:
 *   - uniforms[b,t] (t < n_b) drives the accept test at position t;
 *     uniforms[b,n_b] drives the bonus draw; uniforms_resample[b] drives the
 *     replacement draw at a rejected position.  One final draw per request.
 *   - The accept test is strict (u < p/q).  q(x) = 0 with p(x) > 0 accepts;
 *     p(x) = 0 rejects.
 *   - T_b = 0 selects the greedy rule on the raw target logits; the draft
 *     logits of that request are never read.  The same T_b divides target
 *     and draft logits.
 *   - argmax ties resolve to the lowest index.
 *   - Inverse CDF: the token is the smallest i with w_i > 0 and
 *     w_0 + ... + w_i > u * sum(w).  If rounding leaves none, the last i with
 *     w_i > 0.  A zero-weight token is never emitted.  A residual of exactly
 *     zero mass (possible only through rounding) falls back to drawing from p
 *     with the same uniform.
 *   - Rows t > n_b of the target and t >= n_b of the draft are never read.
 *   - out_tokens[b,:] = x_0 .. x_{j-1}, final token, then -1; accepted_len[b]
 *     = j in [0, n_b].
 *
 * Conventions for every call:
 *   - Ownership: every buffer is allocated and owned by the caller.  The
 *     library allocates nothing and keeps no state between calls besides
 *     what the caller's workspace holds.
 *   - Asynchrony: device calls only enqueue work on `stream` and never
 *     synchronise (except specv_read_device_status and
 *     spec_verify_sample_host, which say so).
 *   - Errors: problems visible on the host (null pointers, bad sizes,
 *     misalignment, a workspace that is too small) return a status before
 *     anything is enqueued.  Problems in the data (a draft length outside
 *     1..K, a token outside [0,V), a negative or non-finite temperature, a
 *     uniform outside [0,1), a sampled row without a finite maximum) are
 *     detected on the device: the request's accepted_len becomes -1, its
 *     out_tokens become -1, and a bit is set in the workspace's status word
 *     (specv_read_device_status).  Nothing traps.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* specv_stream_t;

typedef enum specv_status {
  SPECV_OK = 0,
  SPECV_ERR_INVALID_ARG = 1,  /* null pointer, size out of range, misalignment */
  SPECV_ERR_UNSUPPORTED = 2,  /* shape beyond the documented limits           */
  SPECV_ERR_WORKSPACE = 3,    /* workspace or staging buffer too small         */
  SPECV_ERR_CUDA = 4,         /* a CUDA call failed                            */
  SPECV_ERR_BAD_INPUT = 5     /* the device flagged bad data (status word)     */
} specv_status;

typedef enum specv_dtype {
  SPECV_F32 = 0,   /* IEEE float32 logits                          */
  SPECV_BF16 = 1   /* bfloat16 logits (raw 16-bit storage)          */
} specv_dtype;

/* Bits of the device status word. */
#define SPECV_DEV_BAD_DRAFT_LEN   0x01  /* draft_len[b] outside 1..K               */
#define SPECV_DEV_BAD_TOKEN       0x02  /* draft_tokens[b,t] outside [0,V), t<n_b  */
#define SPECV_DEV_BAD_TEMPERATURE 0x04  /* negative, NaN or infinite temperature   */
#define SPECV_DEV_BAD_UNIFORM     0x08  /* a value of uniforms[b,0..n_b] or
                                           uniforms_resample[b] outside [0,1), for
                                           greedy requests too                   */
#define SPECV_DEV_BAD_ROW         0x10  /* a row the request needs has no finite max */
#define SPECV_DEV_NO_DRAFT        0x20  /* T_b > 0 but draft_logits is NULL        */
#define SPECV_DEV_TIMEOUT         0x40  /* a bounded wait on a copy gave up        */
#define SPECV_DEV_BAD_TREE        0x80  /* a token tree whose parent of node i is not
                                           below i, or a node token outside [0,V) */

/* Limits. */
#define SPECV_MAX_DRAFT 16      /* K <= 16                               */
#define SPECV_MAX_BATCH 65535   /* B <= 65535                            */

/* Library version (major*10000 + minor*100 + patch). */
int specv_version(void);

/* Largest vocabulary supported for a dtype (2 MB rows, 342 chunks of 6 KB):
 * 1048576 for bf16, 524288 for f32. */
int specv_max_vocab(specv_dtype dtype);

/* Human-readable name of a status code (static string, never NULL). */
const char* specv_status_string(specv_status status);

/* Bytes of device workspace one call over B requests of up to K drafts of
 * a V-entry vocabulary needs: a header (status word, the residual and bonus
 * lists' lengths, which each launch sequence empties at its start), one
 * 32-byte draw record per request
 * (the residual and bonus lists), one 8-byte record per (row, 6 KB chunk),
 * the drafted tokens' logits, and one 32-byte record per (listed request,
 * 3 KB piece) holding the piece's residual sweep sums and total.  Batches
 * of more than 1024 requests run as consecutive launch sequences that share
 * it, so it is sized for at most 1024 requests.  Returns 0 for sizes out of
 * range. */
size_t specv_workspace_bytes(int B, int K, int V, specv_dtype dtype);

/* Zero a workspace on `stream` (cudaMemsetAsync).  Must run once before the
 * first call that uses the workspace; every call that completes leaves it
 * ready for the next (counters back at zero).  workspace must be 256-byte
 * aligned.  After a CUDA error inside a call, zero it again. */
specv_status specv_workspace_init(void* workspace, size_t workspace_bytes, specv_stream_t stream);

/*
 * The verification sampler.  All pointers are device pointers.
 *   target_logits     [B, K+1, V] of `dtype`, row-major, contiguous; the
 *                     base must be aligned to the element size (16-byte
 *                     alignment of every row enables bulk copies).
 *   draft_logits      [B, K, V] of `dtype`; may be NULL when every T_b is 0
 *                     (a request with T_b > 0 then fails with NO_DRAFT).
 *   draft_tokens      [B, K] int32, entries t < n_b in [0, V).
 *   draft_len         [B] int32 in 1..K, or NULL for "all K".
 *   temperature       [B] float32, >= 0 and finite; 0 selects greedy.
 *   uniforms          [B, K+1] float32 in [0,1).
 *   uniforms_resample [B] float32 in [0,1).
 *   accepted_len      [B] int32 output: j in [0, n_b], or -1 for bad data.
 *   out_tokens        [B, K+1] int32 output: accepted drafts, the final
 *                     token, then -1.
 *   workspace         specv_workspace_bytes(B, K, V, dtype) bytes, 256-byte aligned,
 *                     zeroed once with specv_workspace_init.  Calls that may
 *                     run concurrently need separate workspaces.
 *   stream            a stream of the current device (all buffers on it).
 * Enqueues four kernels on `stream` per 1024 requests (row statistics,
 * decisions, residual piece sums with the bonus draws, residual searches;
 * each as a programmatic dependent launch); no host synchronisation.
 */
specv_status spec_verify_sample(const void* target_logits, const void* draft_logits,
                                specv_dtype dtype, const int32_t* draft_tokens,
                                const int32_t* draft_len, const float* temperature,
                                const float* uniforms, const float* uniforms_resample,
                                int B, int K, int V, int32_t* accepted_len,
                                int32_t* out_tokens, void* workspace, size_t workspace_bytes,
                                specv_stream_t stream);

/*
 * Same as spec_verify_sample, and also writes per-row statistics for parity
 * checks: row_stats [B, K+1, 8] float32 (device), for the rows the request
 * needs (slots 6 and 7 only for the row of the final draw, t = accepted_len):
 *   0 max_i z^p_i (raw logit)    1 S_p = sum_i exp((z^p_i - max)/T)
 *   2 ln p(x_t)                  3 max_i z^q_i       4 S_q
 *   5 ln q(x_t)                  6 final-draw mass (below)
 *   7 the row's final-draw token (residual with uniforms_resample[b] at
 *     t < n_b, bonus with uniforms[b,n_b] at t = n_b; greedy: argmax)
 * Slot 6 is the normalised mass of the final draw's weights: sum_i (p_i - q_i)+
 * at a rejected position, sum_i p_i at the bonus position.  At T = 0 slot 0
 * is the row maximum and slot 7 the argmax for every row t <= n_b.  Unused
 * slots and rows are left untouched.
 */
specv_status spec_verify_sample_debug(const void* target_logits, const void* draft_logits,
                                      specv_dtype dtype, const int32_t* draft_tokens,
                                      const int32_t* draft_len, const float* temperature,
                                      const float* uniforms, const float* uniforms_resample,
                                      int B, int K, int V, int32_t* accepted_len,
                                      int32_t* out_tokens, void* workspace,
                                      size_t workspace_bytes, float* row_stats,
                                      specv_stream_t stream);

/* Copy the workspace's device status word to *status (host), then clear it.
 * Synchronises `stream`.  Returns SPECV_ERR_BAD_INPUT when the word was
 * non-zero, SPECV_OK when it was zero. */
specv_status specv_read_device_status(void* workspace, size_t workspace_bytes, int32_t* status,
                                      specv_stream_t stream);

/* Bytes of device staging spec_verify_sample_host needs (inputs and
 * outputs, each padded to 256 bytes).  with_draft = 0 when draft logits are
 * not passed. */
size_t specv_host_staging_bytes(int B, int K, int V, specv_dtype dtype, int with_draft);

/*
 * The sampler on HOST buffers: copies the inputs host->device into
 * `staging` (device, specv_host_staging_bytes bytes, 256-byte aligned),
 * runs spec_verify_sample, copies accepted_len and out_tokens back, and
 * synchronises `stream` before returning.  Of the logits only the rows the
 * kernels read cross the host link: a usable request's target rows
 * t <= draft_len[b] and, when temperature[b] > 0, its draft rows
 * t < draft_len[b].  Page-locked logits whose rows are a multiple of 16
 * bytes (16-byte-aligned bases) are gathered by one kernel that reads the
 * host memory through its device-visible address; other logits go as one
 * cudaMemcpyAsync per range of adjacent rows.  The other rows of `staging`
 * keep whatever they held and are never read.  draft_len and temperature are read on the host to decide
 * this, so they must be host-readable.  Every small input is copied whole.
 * Host buffers should be page-locked for asynchronous copies.  Same shapes
 * and readings as spec_verify_sample; draft_len and draft_logits may be NULL
 * as there.
 */
specv_status spec_verify_sample_host(const void* target_logits, const void* draft_logits,
                                     specv_dtype dtype, const int32_t* draft_tokens,
                                     const int32_t* draft_len, const float* temperature,
                                     const float* uniforms, const float* uniforms_resample,
                                     int B, int K, int V, int32_t* accepted_len,
                                     int32_t* out_tokens, void* staging, size_t staging_bytes,
                                     void* workspace, size_t workspace_bytes,
                                     specv_stream_t stream);

/* The launch shape the library picks for these sizes (diagnostics): out[0]
 * CTAs of the row-statistics kernel, out[1] vocabulary elements per chunk,
 * out[2] shared-memory copy slots per agent warp, out[3] chunks per row,
 * out[4] dynamic shared memory per CTA (bytes), out[5] threads per CTA
 * (32 per agent warp).  Queries the current device's occupancy; launches
 * nothing. */
specv_status specv_launch_plan(int B, int K, int V, specv_dtype dtype, int with_draft,
                               int32_t* out);

/* ------------------------------------------------------------------------
 * Steps around the verification (same conventions: device buffers, the
 * caller's workspace zeroed once with specv_workspace_init, asynchronous on
 * `stream`, data errors in the workspace's status word).
 * ---------------------------------------------------------------------- */

/* Bytes of workspace spec_sample_draft needs for R rows of V logits (0 for
 * sizes out of range). */
size_t specv_sample_workspace_bytes(int R, int V, specv_dtype dtype);

/*
 * The draft-side sampler ("Decodificación Especulativa y EAGLE", sections
 * "La Configuración de Dos Modelos" and "Desarrolla": the draft model
 * proposes each token by sampling softmax(z / T) of its logits):
 *   logits       [R, V] of `dtype`, one row per request.
 *   temperature  [R] float32 >= 0; 0 takes the row's argmax (lowest index).
 *   uniforms     [R] float32 in [0,1): tokens[r] is the smallest i with
 *                p_0 + ... + p_i > u * sum(p) and p_i > 0 (the same inverse
 *                CDF as the verification's final draws).
 *   tokens       [R] int32 output (-1 for a row flagged bad: temperature or
 *                uniform out of range, no finite maximum).
 *   workspace    specv_sample_workspace_bytes(R, V, dtype) bytes.
 *   row_stats    NULL, or [R, 8] float32: slot 0 the row maximum, 1 its
 *                normaliser sum exp((z - max)/T), 6 the drawn mass
 *                (sum of p, ~1), 7 the token; at T = 0 slots 0 and 7.
 * Enqueues two kernels per 1024 rows: the row statistics, then the
 * decisions of spec_verify_sample for requests with no drafts, whose bonus
 * draw (the sample) the decision kernel makes itself.
 */
specv_status spec_sample_draft(const void* logits, specv_dtype dtype, const float* temperature,
                               const float* uniforms, int R, int V, int32_t* tokens,
                               void* workspace, size_t workspace_bytes, float* row_stats,
                               specv_stream_t stream);

/*
 * Verification for a draft that proposes its top token ("Accelerating Sonar
 * through speculation", section "Objetivo-Borrador"): the distribution the
 * drafted token came from is the point mass q = 1{x}, so the rule of "La
 * Regla de Exactitud" accepts x_t iff u_t < p_t(x_t), and at the first
 * rejection j draws the replacement from (p_j - 1{x_j})+, i.e. from p_j with
 * x_j removed; every draft accepted draws the bonus from p_n.  No draft
 * logits.  Arguments, outputs, readings and errors as spec_verify_sample
 * without draft_logits (T = 0 is the greedy rule); workspace
 * specv_workspace_bytes(B, K, V, dtype); row_stats NULL or as
 * spec_verify_sample_debug (slots 3..5 unused; slot 6 at a rejected row is
 * 1 - p_j(x_j)).
 */
specv_status spec_verify_sample_onehot(const void* target_logits, specv_dtype dtype,
                                       const int32_t* draft_tokens, const int32_t* draft_len,
                                       const float* temperature, const float* uniforms,
                                       const float* uniforms_resample, int B, int K, int V,
                                       int32_t* accepted_len, int32_t* out_tokens,
                                       void* workspace, size_t workspace_bytes,
                                       float* row_stats, specv_stream_t stream);

/* Bytes of workspace spec_verify_tree_greedy needs (0 for sizes out of
 * range; N <= 64). */
size_t specv_tree_workspace_bytes(int B, int N, int V, specv_dtype dtype);

/*
 * Greedy verification of a token tree ("Decodificación Especulativa y EAGLE",
 * section "Verificación de Atención en Árvore"; "Accelerating Sonar through
 * speculation", section "EAGLE"): the target scores every node of a drafted
 * tree in one pass; node i is accepted iff its parent is accepted and the
 * target's argmax at the parent (lowest index) is node i's token; the root
 * (node 0, the last verified position) is always accepted.  The deepest
 * accepted node (lowest index among the deepest) ends the kept path.
 *   target_logits [B, N, V] of `dtype`: row i = the target's logits at node i.
 *   parents       [B, N] int32: parents[b,0] = -1, 0 <= parents[b,i] < i.
 *   tokens        [B, N] int32: node i's drafted token (tokens[b,0] unused).
 *   n_nodes       [B] int32 in 1..N: nodes >= n_nodes[b] are not read.
 *   accepted_len  [B] int32 output: the path's length (accepted drafts), or
 *                 -1 for a malformed tree (status SPECV_DEV_BAD_TREE) or bad
 *                 node count (SPECV_DEV_BAD_DRAFT_LEN).
 *   out_tokens    [B, N] int32 output: the path's tokens, then the argmax at
 *                 its last node, then -1.
 *   path_nodes    [B, N] int32 output: 0, then the path's node indices, then
 *                 -1 (the cache rows to keep).
 *   workspace     specv_tree_workspace_bytes(B, N, V, dtype) bytes.
 *   row_stats     NULL, or [B, N, 8] float32: slot 0 each node's maximum,
 *                 slot 7 its argmax.
 * The sampled (multi-branch) tree rule is not on the pages and not built.
 */
specv_status spec_verify_tree_greedy(const void* target_logits, specv_dtype dtype,
                                     const int32_t* parents, const int32_t* tokens,
                                     const int32_t* n_nodes, int B, int N, int V,
                                     int32_t* accepted_len, int32_t* out_tokens,
                                     int32_t* path_nodes, void* workspace,
                                     size_t workspace_bytes, float* row_stats,
                                     specv_stream_t stream);

/*
 * The post-accept insert ("Accelerating Sonar through speculation", sections
 * "Programación MTP para un solo token" and "Inferencia con decodificación
 * especulativa": a kernel writes the next step's tokens on the device, so
 * the host need not read the accepted lengths between steps).  For request
 * b with j = accepted_len[b] (as spec_verify_sample writes it):
 *   history[b, seq_lens[b] .. seq_lens[b] + j] = out_tokens[b, 0 .. j];
 *   seq_lens[b] += j + 1;  next_tokens[b] = out_tokens[b, j];
 *   cu_emitted[b + 1] = cu_emitted[b] + j + 1 (cu_emitted[0] = 0) and
 *   packed[cu_emitted[b] .. cu_emitted[b + 1]) = out_tokens[b, 0 .. j].
 * A request with j outside [0, K] emits nothing (status[b] = 1), one whose
 * history would pass L emits nothing (status[b] = 2); both keep their
 * history and length and get next_tokens[b] = -1.  status[b] = 0 otherwise.
 *   accepted_len [B], out_tokens [B, K+1], seq_lens [B] (in/out),
 *   history [B, L] (in/out), next_tokens [B], cu_emitted [B+1],
 *   packed [B*(K+1)] (only the first cu_emitted[B] written), status [B]:
 *   int32 device buffers.  One kernel of one CTA; no workspace.
 */
specv_status spec_insert_accepted(const int32_t* accepted_len, const int32_t* out_tokens, int B,
                                  int K, int32_t* seq_lens, int32_t* history, int L,
                                  int32_t* next_tokens, int32_t* cu_emitted, int32_t* packed,
                                  int32_t* status, specv_stream_t stream);

/*
 * The sampler without any allocation, for callers that cannot allocate
 * device memory where they run it: plugin interfaces that hand the plugin
 * only the tensors it declared, serving loops that forbid cudaMalloc after
 * start-up (it can synchronise the device and fragment a fixed budget), and
 * hosts whose device memory is owned by another allocator.  The pages have
 * no counterpart; this is a packaging variant of spec_verify_sample.
 *
 * Same inputs, outputs, readings and errors as spec_verify_sample, with no
 * workspace argument: the scratch (the workspace of spec_verify_sample)
 * lives in a module-scope device array of the library of
 * SPECV_NOALLOC_SCRATCH_BYTES (4 MiB); every GPU that loads the library
 * holds it until the process exits.  Shapes whose workspace
 * (specv_workspace_bytes) exceeds it return SPECV_ERR_UNSUPPORTED.
 *   - It calls no cudaMalloc, cudaFree or allocating library routine.
 *   - Every call looks up the array's device address in the current
 *     device's context (cudaGetSymbolAddress); the first call on a device
 *     may load the library's module there, so make it before any stream
 *     capture.  `stream` must belong to the current device.
 *   - Each call zeroes the part of the array it uses (cudaMemsetAsync on
 *     `stream`), then launches the kernels.  All calls on a device share the
 *     one array: calls that may overlap on the GPU (different streams, or
 *     concurrent host threads) race and must be serialised by the caller.
 *   - The device status word is not exposed: bad data shows as
 *     accepted_len[b] = -1 and out_tokens[b,:] = -1.
 */
#define SPECV_NOALLOC_SCRATCH_BYTES (4u << 20)

specv_status spec_verify_sample_noalloc(const void* target_logits, const void* draft_logits,
                                        specv_dtype dtype, const int32_t* draft_tokens,
                                        const int32_t* draft_len, const float* temperature,
                                        const float* uniforms, const float* uniforms_resample,
                                        int B, int K, int V, int32_t* accepted_len,
                                        int32_t* out_tokens, specv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
