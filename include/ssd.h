/*
 * ssd.h -- C ABI of libssd: the batched verify-and-sample step of speculative
 * decoding and the cache side of Saguaro (speculative speculative decoding),
 * as hand-written CUDA for sm_103a (GB300).
 *
 * Sources of the operations (page titles and sections):
 *   [SD]  "Speculative decoding" (brentwoodlivery.com): "The Algorithm
 *         (Step-by-Step)", "Derivation of Acceptance Criterion", "Temperature
 *         and Sampling", "Batching Speculation".
 *   [WHY] "Why does speculative decoding exist?" (til.phipham141.dev): "How it
 *         works" (Fix 2: longest accepted prefix plus one bonus token; greedy
 *         acceptance = draft token is the target argmax; Fix 3: min(1, p/q)
 *         acceptance and the residual (p - q)+).
 *   [SSD] "Speculative Speculative Decoding" notes (papernotes.org): "整体框架"
 *         (outcome v = (k, t*), speculation cache S_T, hit test), "关键设计" item 1
 *         (geometric and uniform fan-out F_k), item 2 (SAGUARO sampling
 *         sigma_{F,C}; cache keys from the draft logits) and item 3 (batch-size
 *         aware fallback; fast random-token backup).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Array arguments are DEVICE pointers owned by the caller, dense row-major,
 *   unless the argument name ends in _host.  The library never allocates or
 *   frees memory and never synchronises the stream: every device call only
 *   enqueues work on `stream` (a cudaStream_t; NULL = the legacy default
 *   stream) and returns.
 * - Shapes: B sequences, K drafted tokens per sequence, V vocabulary entries.
 *   Target logits  tgt [B, K+1, V]   (row i scores position i, row K is the
 *                                     extra row used when all K are accepted)
 *   Draft logits   drf [B, drf_rows, V], drf_rows in {K, K+1} (verification
 *                                     reads rows 0..K-1; ssd_draft_cache takes
 *                                     all K+1)
 *   Draft tokens   tokens [B, K] int32
 *   Uniforms       uniforms [B, K+1] fp32 in [0, 1): column i < K is the accept
 *                  draw of position i, column K draws the bonus token.
 *   Temperature    temperature [B] fp32 per sequence; 0 selects greedy
 *                  decoding; negative or NaN marks the sequence invalid.
 * - dtype is SSD_F32 or SSD_BF16 (storage type of both logit tensors).
 * - Every call returns an ssd status (SSD_OK = 0).  Host-side validation
 *   failures return before anything is enqueued.  SSD_ERR_CUDA reports a launch
 *   or attribute error from the CUDA runtime.
 * - Data errors found on the device (a drafted token outside [0, V), a bad
 *   temperature, non-finite logits, a bounded wait that ran out) do not abort
 *   the call: the affected sequence gets accept_len = -1 and bonus = -1, and
 *   the matching SSD_DEV_* bits are OR-ed into *dev_status when dev_status is
 *   not NULL (a device int32 the caller zeroes and reads).
 * - Workspace: calls that take one need ssd_workspace_size(B, K) bytes of
 *   device memory, 256-byte aligned, zero-filled before its first use (for
 *   example one cudaMemsetAsync after allocation).  Each completed call leaves
 *   its per-sequence counters at zero again, so the workspace is ready for the
 *   next call without another fill.  Calls sharing one workspace must not
 *   overlap on the GPU (use one workspace per stream).
 * - Limits: 1 <= K <= SSD_MAX_K, 2 <= V, 1 <= B, every cache segment and the
 *   reshape F at most SSD_MAX_F, and a row slice of at most SSD_MAX_V_F32 /
 *   SSD_MAX_V_BF16 vocabulary entries (larger V returns SSD_ERR_UNSUPPORTED).
 */
#ifndef SSD_H
#define SSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define SSD_OK 0
#define SSD_ERR_INVALID_ARG 1
#define SSD_ERR_DTYPE 2
#define SSD_ERR_CUDA 3
#define SSD_ERR_WORKSPACE 4
#define SSD_ERR_UNSUPPORTED 5

/* Logit storage types. */
#define SSD_F32 0
#define SSD_BF16 1

/* Device status bits. */
#define SSD_DEV_BAD_TOKEN 1
#define SSD_DEV_BAD_TEMPERATURE 2
#define SSD_DEV_NONFINITE 4
#define SSD_DEV_TIMEOUT 8

/* Limits. */
#define SSD_MAX_K 32
#define SSD_MAX_F 256
#define SSD_MAX_V_F32 400000
#define SSD_MAX_V_BF16 800000

/*
 * sigma_{F,C} descriptor of one draft row ([SSD] item 2).  Token t is in the
 * reshaped top-F set iff  z_t > thr_val  or  (z_t == thr_val and t <= thr_id),
 * compared on the raw stored logit z_t; thr_val/thr_id are the value and id of
 * the F-th largest logit (ties to the lowest id).  F == 0 is encoded as
 * thr_val = +inf, thr_id = -1 (empty set).  The reshaped draft distribution is
 * q'_t proportional to c_t * exp(z_t / tau), c_t = C inside the set, 1 outside.
 */
typedef struct ssd_reshape_desc {
    float thr_val;
    int32_t thr_id;
    int32_t F;
    float C;
} ssd_reshape_desc;

/* Kernel choice for rows on the 16-byte grid (process-wide; rows off the grid
 * always take the cluster kernel).  AUTO: for verification alone with fewer
 * units (sequences x (K+1)) than 8 per SM, the persistent streaming kernel in its
 * wide form (below); otherwise the streaming kernel when the batch has at least
 * as many units as the GPU has SMs -- in its wide form below twice as many -- or
 * when sigma_{F,C} is found in the pass, else the cluster kernel, which splits
 * each row across a thread-block cluster.  STREAM / CLUSTER / SLICE force
 * one.  SLICE, the slice kernel, splits every row into slices of 16 KB blocks
 * that the whole GPU works on at once and combines the slices' partial results
 * in the workspace; it applies to rows of whole 16-byte vectors (V a multiple of
 * the vector), without sigma found in the pass, B <= 2048 and a workspace of
 * ssd_workspace_size_v bytes; other calls fall back as under AUTO.  WIDE forces
 * the streaming kernel in its wide form, where both consumer groups of a CTA
 * work on each unit (half the units in flight, each at about twice the rate),
 * for rows of whole 16-byte vectors (V a multiple of the vector); other calls
 * fall back as under AUTO. */
#define SSD_DISPATCH_AUTO 0
#define SSD_DISPATCH_STREAM 1
#define SSD_DISPATCH_CLUSTER 2
#define SSD_DISPATCH_SLICE 3
#define SSD_DISPATCH_WIDE 4

/* Sets the kernel choice; returns the previous one, or -1 (and changes nothing)
 * for an unknown policy.  Calls already enqueued are not affected. */
int ssd_set_dispatch(int policy);

/* Name of the kernel that the most recent verify / cache / round call made on
 * the calling host thread launched ("stream" -- the persistent streaming kernel,
 * "stream-wide" -- the same kernel in its wide form,
 * "slice" -- the slice kernel, "cluster" -- the cluster kernel, "reshape+cluster"
 * -- the reshape kernel and then the cluster kernel for sigma found before the
 * pass), or "none" before any such call.  Plumbing for reporting (no counterpart on the pages); the string is
 * static, owned by the library. */
const char *ssd_last_kernel(void);

/* Check of the bounded waits (no counterpart on the pages): one warp waits on a
 * shared-memory mbarrier that nothing completes, with the same bounded wait
 * every kernel here uses but a limit of limit_ms milliseconds (1..10000); when
 * it gives up it ORs SSD_DEV_TIMEOUT into *dev_status (device int32, required)
 * and the launch ends normally, leaving the context usable.  The kernels' own
 * waits give up after 4 s. */
int ssd_check_wait_timeout(int32_t *dev_status, int limit_ms, void *stream);

/* Human-readable name of a status code (static string, never NULL). */
const char *ssd_strerror(int status);

/* Library version string. */
const char *ssd_version(void);

/* Bytes of workspace needed by ssd_verify / ssd_build_cache / ssd_round for a
 * batch of B sequences with K drafted tokens (0 when B or K is out of range). */
size_t ssd_workspace_size(int B, int K);

/* Workspace bytes that let every kernel serve a call with B sequences, K drafted
 * tokens, V-token rows of `dtype` and a cache budget (0 without a cache): the
 * ssd_workspace_size(B, K) regions plus the slice kernel's per-unit state,
 * per-slice partial results, per-group arrays of every unit (2 x ceil(V / 64)
 * floats) and its work queue.  A smaller workspace of at least
 * ssd_workspace_size(B, K) bytes is still valid: the slice kernel is then not
 * used.  Zero-filled once by the caller like the smaller one; each call leaves
 * it zeroed.  Returns 0 for invalid arguments. */
size_t ssd_workspace_size_v(int B, int K, int V, int dtype, int budget);

/*
 * ssd_verify -- [SD] "The Algorithm (Step-by-Step)" step 3 for a batch
 * ([SD] "Batching Speculation": every sequence accepts 0..K tokens
 * independently).  Per sequence b with temperature tau > 0 ([SD] "Temperature
 * and Sampling": p = softmax(target row / tau), q = softmax(draft row / tau),
 * or q = sigma_{F,C} when `reshape` is given):
 *   accept x~_i  iff  u_i * q_i(x~_i) < p_i(x~_i)        (min(1, p/q) against u_i)
 *   a = first rejected position, or K when none is rejected
 *   bonus = inverse CDF over ascending token id of max(0, p_a - q_a) / Z at
 *           u_K * Z (a < K; Z == 0 falls back to p_a), or of p_K (a == K).
 * tau == 0 ([WHY] Fix 2): accept iff x~_i is the target argmax (raw logits,
 * lowest id on ties); bonus = target argmax of row a.
 * Inputs: tgt, drf, tokens, uniforms, temperature as in the conventions;
 *   reshape: [B, K] descriptors from ssd_reshape_draft, or NULL.
 * Outputs: accept_len [B] int32 in [0, K] (-1 for an invalid sequence);
 *   bonus [B] int32 in [0, V); p_tok, q_tok [B, K] fp32 (may be NULL):
 *   p_i(x~_i) and q_i(x~_i) for i <= a, NaN for i > a (tau == 0: p_tok is 1
 *   when x~_i is the argmax else 0, q_tok is 1).
 * Rows after the first rejection are not needed; the kernel may skip them.
 */
int ssd_verify(const void *tgt, const void *drf, int dtype, int B, int K, int V, int drf_rows,
               const int32_t *tokens, const float *uniforms, const float *temperature,
               const ssd_reshape_desc *reshape, int32_t *accept_len, int32_t *bonus,
               float *p_tok, float *q_tok, void *workspace, size_t workspace_bytes,
               int32_t *dev_status, void *stream);

/*
 * ssd_fanout -- [SSD] item 1, host only.  F_k = F_0 a_p^{k/(1+r)} for k < K and
 * F_K = F_0 a_p^{K/(1+r)} (1 - a_p)^{-1/(1+r)}, with F_0 chosen so that the
 * real-valued F_k sum to `budget`; made integer by the largest-remainder
 * method (floor, then +1 to the largest fractional parts, lowest k on ties),
 * so the F_k sum to budget; each F_k is then clamped to V.
 * Outputs (host arrays): F_host [K+1], off_host [K+2] (off[0] = 0,
 * off[k+1] = off[k] + F_k).  Requires 0 < a_p < 1, r > -1, budget >= 0, V >= 1.
 */
int ssd_fanout(int K, int budget, double a_p, double r, int V, int32_t *F_host,
               int32_t *off_host);

/*
 * ssd_fanout_uniform -- the uniform fan-out that [SSD] item 1 compares the
 * geometric shape against: every accepted length k = 0..K gets the same share,
 * F_k = floor(budget / (K+1)), plus one for the first budget mod (K+1)
 * positions; each F_k is then clamped to V.  Outputs as ssd_fanout.
 * Requires budget >= 0, V >= 1.
 */
int ssd_fanout_uniform(int K, int budget, int V, int32_t *F_host, int32_t *off_host);

/*
 * ssd_backup_fill -- the fast random-token backup speculator of [SSD] item 3
 * (batch-size-aware fallback): for every sequence whose round missed the
 * cache (hit[b] == 0) the next round's K draft tokens are drawn uniformly
 * from the vocabulary, next_tokens[b, i] = min(V - 1, floor(u[b, i] * V))
 * with the caller's uniforms u [B, K] in [0, 1) (the product is taken exactly
 * in double; an fp32 uniform resolves 2^-24, so with V above 2^24 the top ids
 * are never drawn); rows of sequences that hit are left untouched.  hit [B] uint8, uniforms
 * [B, K] fp32, next_tokens [B, K] int32, all device pointers owned by the
 * caller.  Requires B >= 1, 1 <= K <= SSD_MAX_K, V >= 1.
 */
int ssd_backup_fill(const uint8_t *hit, const float *uniforms, int B, int K, int V,
                    int32_t *next_tokens, void *stream);

/*
 * ssd_reshape_draft -- [SSD] item 2 on `rows` independent draft rows
 * drf [rows, V]: the top-F set of each row (raw logits, lowest id on ties) and,
 * when q_out is not NULL, the reshaped distribution
 *   q_out[r, t] = c_t exp(z_t / tau_r) / sum_j c_j exp(z_j / tau_r),
 * c_t = C for the top-F tokens, 1 otherwise (tau_r = temperature_rows[r] > 0).
 * desc [rows] receives the descriptor (see ssd_reshape_desc).  Requires
 * 0 <= F <= SSD_MAX_F, 0 <= C <= 1, and not (C == 0 and F >= V).
 */
int ssd_reshape_draft(const void *drf, int dtype, int rows, int V, const float *temperature_rows,
                      int F, float C, ssd_reshape_desc *desc, float *q_out, int32_t *dev_status,
                      void *stream);

/*
 * ssd_draft_cache -- the draft side of a Saguaro round ([SSD] item 2: the
 * cache keys are chosen from the draft logits; sampling is reshaped by
 * sigma_{F,C} with F the position's fan-out).  drf [B, K+1, V] holds the draft
 * logits of positions 0..K of every sequence (row K: the draft's distribution
 * after all K drafted tokens, which the all-accepted outcome needs).
 * For each sequence b and position k = 0..K, segment k of cache_tok[b]
 * (columns off[k] .. off[k+1], off the prefix sums of F_host) receives the
 * F_k tokens of largest raw draft logit at row k, best first (ties to the
 * lowest id), leaving out the drafted token x~_k = tokens[b, k] for k < K;
 * a slot with no token left (F_k == V and x~_k excluded) holds -1.
 * tokens may be NULL (nothing left out).  desc [B, K] (may be NULL) receives
 * the sigma_{F_k,C} descriptor of draft row k < K (ssd_reshape_desc, same
 * set as ssd_reshape_draft with F = F_k); give it to ssd_verify / ssd_round
 * with drf_rows = K+1 so that verification uses the reshaped q.
 * At least one of cache_tok and desc must be non-NULL.  Requires
 * 1 <= K <= SSD_MAX_K, V >= 2, 0 <= F_k <= min(V, SSD_MAX_F),
 * budget >= sum F_k, and with desc: 0 <= C <= 1, not (C == 0 and F_k >= V).
 * One thread-block cluster per draft row; every row is read once.
 */
int ssd_draft_cache(const void *drf, int dtype, int B, int K, int V, const int32_t *tokens,
                    const int32_t *F_host, int budget, float C, int32_t *cache_tok,
                    ssd_reshape_desc *desc, int32_t *dev_status, void *stream);

/*
 * ssd_build_cache -- the speculation-cache keys of [SSD] "整体框架" / item 1:
 * for each sequence b and accepted length k = 0..K, the F_k bonus tokens most
 * likely to be drawn at outcome (k, t*), ranked by (score desc, id asc):
 *   tau > 0:  score = max(0, p_k - q_k) for k < K,  p_K for k = K;
 *   tau == 0: score = raw target logit of row k, x~_k ranked last (k < K).
 * F_host [K+1] (host) is the fan-out (ssd_fanout); segment k of a cache row is
 * cache_tok[b, off[k] .. off[k+1]) with off the prefix sums of F_host, and
 * budget >= off[K+1] is the row length of cache_tok [B, budget] int32.
 * Entries beyond off[K+1] are left untouched.
 */
int ssd_build_cache(const void *tgt, const void *drf, int dtype, int B, int K, int V,
                    int drf_rows, const int32_t *tokens, const float *temperature,
                    const ssd_reshape_desc *reshape, const int32_t *F_host, int budget,
                    int32_t *cache_tok, void *workspace, size_t workspace_bytes,
                    int32_t *dev_status, void *stream);

/*
 * ssd_cache_lookup -- [SSD] "整体框架": the true outcome (a, t*) hits iff t* is
 * in segment a of the sequence's cache row.  hit [B] uint8 (1 = hit),
 * slot [B] int32 = column of t* in cache_tok (-1 on a miss or when
 * accept_len[b] < 0).
 */
int ssd_cache_lookup(const int32_t *cache_tok, int B, int K, int budget, const int32_t *F_host,
                     const int32_t *accept_len, const int32_t *bonus, uint8_t *hit,
                     int32_t *slot, void *stream);

/*
 * ssd_round -- one fused launch of ssd_verify + ssd_build_cache +
 * ssd_cache_lookup: every logit row is read from HBM once.  Arguments and
 * outputs as in those three calls.
 */
int ssd_round(const void *tgt, const void *drf, int dtype, int B, int K, int V, int drf_rows,
              const int32_t *tokens, const float *uniforms, const float *temperature,
              const ssd_reshape_desc *reshape, const int32_t *F_host, int budget,
              int32_t *accept_len, int32_t *bonus, float *p_tok, float *q_tok,
              int32_t *cache_tok, uint8_t *hit, int32_t *slot, void *workspace,
              size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * ssd_verify_ld / ssd_round_ld -- ssd_verify / ssd_round on logit rows spaced
 * ld >= V elements apart (tgt row (b, i) starts at element (b (K+1) + i) ld,
 * drf row (b, i) at (b drf_rows + i) ld; both tensors share ld).  Entries V..ld-1
 * of a row are never used as logits.  A vocabulary whose rows are not a whole
 * number of 16-byte vectors (V * s not a multiple of 16) reaches the streaming
 * kernel this way when ld * s is a multiple of 16 and ld >= V rounded up to
 * 16 / s; other layouts take the cluster kernel.  ld = V is ssd_verify /
 * ssd_round.  Errors as those calls, and SSD_ERR_INVALID_ARG for ld < V.
 */
int ssd_verify_ld(const void *tgt, const void *drf, int dtype, int B, int K, int V, int ld,
                  int drf_rows, const int32_t *tokens, const float *uniforms, const float *temperature,
                  const ssd_reshape_desc *reshape, int32_t *accept_len, int32_t *bonus, float *p_tok,
                  float *q_tok, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                  void *stream);
int ssd_round_ld(const void *tgt, const void *drf, int dtype, int B, int K, int V, int ld,
                 int drf_rows, const int32_t *tokens, const float *uniforms, const float *temperature,
                 const ssd_reshape_desc *reshape, const int32_t *F_host, int budget,
                 int32_t *accept_len, int32_t *bonus, float *p_tok, float *q_tok, int32_t *cache_tok,
                 uint8_t *hit, int32_t *slot, void *workspace, size_t workspace_bytes,
                 int32_t *dev_status, void *stream);

/*
 * ssd_verify_sigma / ssd_round_sigma -- ssd_verify / ssd_round on the
 * sigma_{F_k,C}-reshaped draft ([SSD] item 2) without descriptors computed
 * beforehand: the top-F_k set of each sampled draft row is found while the
 * row streams through for verification, so the draft rows are read once.
 * sigma_F_host [K] (host): F_k of position k (0 = no reshape there), each
 * 0 <= F_k <= min(V, SSD_MAX_F); 0 <= sigma_C <= 1, and not (sigma_C == 0
 * and F_k >= V).  desc_out [B, K] (device, required) receives the
 * descriptor found for every position of every sampled sequence (the same
 * set ssd_reshape_draft gives with F = F_k); entries of greedy sequences,
 * and of sequences flagged invalid, may be left untouched, and so may, in
 * ssd_verify_sigma, the positions after a sequence's accepted length (their
 * rows are not needed once an earlier position rejected, and may be skipped).
 * Everything else as ssd_verify / ssd_round with reshape = the descriptors
 * found.
 * When the rows do not suit the streaming kernel (a row not on a 16-byte
 * boundary, or V too large for its shared memory) the descriptors are found
 * by a separate pass over the draft rows first.
 */
int ssd_verify_sigma(const void *tgt, const void *drf, int dtype, int B, int K, int V, int drf_rows,
                     const int32_t *tokens, const float *uniforms, const float *temperature,
                     const int32_t *sigma_F_host, float sigma_C, ssd_reshape_desc *desc_out,
                     int32_t *accept_len, int32_t *bonus, float *p_tok, float *q_tok,
                     void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);
int ssd_round_sigma(const void *tgt, const void *drf, int dtype, int B, int K, int V, int drf_rows,
                    const int32_t *tokens, const float *uniforms, const float *temperature,
                    const int32_t *sigma_F_host, float sigma_C, ssd_reshape_desc *desc_out,
                    const int32_t *F_host, int budget, int32_t *accept_len, int32_t *bonus,
                    float *p_tok, float *q_tok, int32_t *cache_tok, uint8_t *hit, int32_t *slot,
                    void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * ssd_round_noalloc -- ssd_round for callers that cannot allocate device
 * memory (no counterpart on the pages: this is plumbing of this library).
 * Some hosts own every device buffer and forbid allocation while they enqueue
 * work -- for example a plugin inside an inference server, where cudaMalloc
 * could block the device or fail under memory pressure while serving.  This
 * entry point takes no workspace: it keeps the round's scratch in a
 * file-scope device array of ssd_noalloc_max_scratch() bytes (1 MiB) that
 * every GPU loading the library holds until the process exits, and it calls
 * no allocating routine.
 * Arguments and outputs are those of ssd_round without the workspace.
 * Errors: SSD_ERR_UNSUPPORTED when ssd_workspace_size(B, K) exceeds the
 * array; otherwise as ssd_round.
 * The first call on a device looks up that device's address of the array
 * (with the device current); make that first call before any stream capture.
 * Each call clears the counters it needs on `stream` before the kernel.  All
 * calls share the one array per device: calls that overlap on the GPU (two
 * streams, or two host threads) race and must be serialised by the caller.
 */
size_t ssd_noalloc_max_scratch(void);
int ssd_round_noalloc(const void *tgt, const void *drf, int dtype, int B, int K, int V,
                      int drf_rows, const int32_t *tokens, const float *uniforms,
                      const float *temperature, const ssd_reshape_desc *reshape,
                      const int32_t *F_host, int budget, int32_t *accept_len, int32_t *bonus,
                      float *p_tok, float *q_tok, int32_t *cache_tok, uint8_t *hit,
                      int32_t *slot, int32_t *dev_status, void *stream);

/*
 * ssd_round_host -- ssd_round on inputs and outputs in host memory (no
 * counterpart on the pages: the transfer plumbing around [SSD] "整体框架").
 * Enqueues the copies of the inputs into `staging`, the round (ssd_round with
 * drf_rows = K, no reshape, no p/q outputs) and the copies of its results back.
 * A batch of B >= 128 runs in min(4, B / 64) chunks of consecutive sequences:
 * the input copies go on a copy stream the library keeps per device (made to
 * wait for the work already on `stream`), and each chunk's round and result
 * copies go on `stream` once that chunk's inputs have landed, so a round runs
 * while the next chunk is copied.  Everything is ordered before the work
 * enqueued on `stream` afterwards.  A sequence that does not sample (tau == 0 decides by the
 * target argmax, [WHY] Fix 2; an invalid tau is reported) never has its draft
 * logits read, so only the sampled sequences' draft rows are copied, each run
 * of consecutive sampled sequences as one copy: the host-to-device traffic is
 * the target logits, those draft rows, tokens, uniforms and temperatures.
 * Inputs (host memory; page-locked for the copies to run asynchronously):
 *   tgt [B, K+1, V] and drf [B, K, V] of `dtype`, contiguous; tokens [B, K];
 *   uniforms [B, K+1]; temperature [B] (also read by the host during the
 *   call); F_host [K+1] and budget as in ssd_build_cache.
 * Outputs (host memory, valid once `stream` has completed): accept_len [B],
 *   bonus [B], cache_tok [B, budget], hit [B], slot [B] as in ssd_round.
 * staging: device memory of at least ssd_host_staging_size(dtype, B, K, V,
 *   budget) bytes, owned by the caller, 256-byte aligned; workspace as in
 *   ssd_round.  h2d_bytes (host, may be NULL) receives the bytes copied to
 *   the device by this call.
 * Errors (before anything is enqueued): SSD_ERR_DTYPE for an unknown dtype;
 * SSD_ERR_INVALID_ARG for a NULL pointer, a size out of range, a fan-out that
 * ssd_build_cache would reject or a staging buffer that is too small.  Later:
 * SSD_ERR_CUDA when a copy cannot be enqueued; otherwise as ssd_round.
 */
size_t ssd_host_staging_size(int dtype, int B, int K, int V, int budget);
int ssd_round_host(const void *tgt, const void *drf, int dtype, int B, int K, int V,
                   const int32_t *tokens, const float *uniforms, const float *temperature,
                   const int32_t *F_host, int budget, int32_t *accept_len, int32_t *bonus,
                   int32_t *cache_tok, uint8_t *hit, int32_t *slot, void *staging,
                   size_t staging_bytes, void *workspace, size_t workspace_bytes,
                   int32_t *dev_status, size_t *h2d_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SSD_H */
