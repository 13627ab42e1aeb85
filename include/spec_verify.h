/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-decoding
 * verification library (libspecverify.so).
 *
 * The operation.  A target model has scored a block of K draft tokens in one
 * pass, giving logits for K+1 positions; the verifier accepts the longest valid
 * draft prefix and emits one more token of the target's own:
 *   - "Спекулятивный декодинг в проде" (kiosknews.app), opening section
 *     ("Откуда взялся спекулятивный декодинг"): the model accepts the longest
 *     correct prefix of the draft and places its own token at the first error;
 *     section "Немного теории", "Правило проверки": a drafted token x is
 *     accepted with probability min(1, p(x)/q(x)), p the target distribution
 *     after temperature and q the draft distribution; after a rejection the
 *     new token is sampled from the normalised residual max(0, p - q);
 *     "Утверждение 1": the emitted token is then distributed exactly as p.
 *   - "speculative decoding от черновика до проверки" (braintools.ru), "Как
 *     это работает", step 3 and the six-token remark: drafts are checked left
 *     to right, and when all K are accepted one more (bonus) token comes from
 *     position K+1 of the same pass; "Почему ответ не портится": at
 *     temperature 0 the check is a comparison with the target argmax.
 *   - "DSpark: ... верификацией по уверенности" (iitog.ru): the verify length
 *     of each request is chosen from the estimated survival probability of the
 *     draft prefix (spec_schedule_len below).
 *
 * Conventions (all entry points):
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *     caller owns every buffer.  The calls never allocate or free memory and
 *     never synchronise the device or the stream; all work is enqueued on
 *     `stream` (a cudaStream_t passed as void*, NULL = legacy default stream).
 *   - Host-detectable errors (null required pointers, sizes out of range,
 *     misaligned buffers, a workspace that is too small, an unknown dtype) are
 *     returned synchronously and nothing is launched.
 *   - Data-dependent problems never trap the GPU: they are clamped and
 *     reported through the optional device status word (SPEC_DEV_* bits,
 *     OR-ed into *dev_status; the caller zeroes it).
 *   - Identical inputs and seed give bit-identical outputs.  The random key is
 *     (seed, request index b, position k, draw); vary `seed` per decoding step.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1, /* null pointer, size out of range, misalignment */
    SPEC_ERR_UNSUPPORTED = 2, /* dtype or shape this build does not handle */
    SPEC_ERR_CUDA = 3,        /* a CUDA runtime call (launch) failed */
    SPEC_ERR_WORKSPACE = 4    /* workspace missing or smaller than required */
} spec_status_t;

typedef enum {
    SPEC_DTYPE_F32 = 0, /* IEEE float32 logits */
    SPEC_DTYPE_BF16 = 1 /* bfloat16 logits */
} spec_dtype_t;

/* Device status bits (OR-ed into *dev_status when dev_status != NULL). */
#define SPEC_DEV_BAD_TOKEN 1u /* a draft token outside [0, V): that request's verify
                                 length is cut to the first such position */
#define SPEC_DEV_BAD_LEN 2u   /* verify_len outside [0, K]: clamped */
#define SPEC_DEV_BAD_TREE    8u   /* a tree node whose parent is not an earlier node */
#define SPEC_DEV_TIMEOUT 4u   /* a bounded device-side wait gave up; outputs of the
                                 affected request are undefined */

#define SPEC_MAX_K 32          /* largest supported draft length K */
#define SPEC_MAX_TREE 64       /* largest candidate tree (nodes, root included) */
#define SPEC_MAX_V 0x40000000  /* largest supported vocabulary V (2^30) */

/*
 * Workspace size in bytes that spec_verify, spec_verify_debug,
 * spec_verify_early_exit, spec_verify_scheduled and spec_draft_confidence
 * need for the given problem (0 on invalid sizes).  The workspace is scratch
 * device memory owned by the caller; it must be 256-byte aligned, need not be
 * initialised, and must not be shared by calls that may run concurrently.
 */
size_t spec_verify_workspace_bytes(int B, int K, int V, spec_dtype_t dtype);

/*
 * spec_verify -- one verification step for a batch of B independent requests.
 *
 *   target_logits [B, K+1, V]  dtype, row-major contiguous.  Row k of request b
 *                              scores draft token k (k < K) or the bonus
 *                              position (k = verify length).
 *   draft_logits  [B, K, V]    dtype, row-major contiguous (never NULL; greedy
 *                              requests do not read it).
 *   draft_tokens  [B, K]       int32 drafted tokens x_k.
 *   verify_len    [B]          int32 number of drafts to verify per request,
 *                              L_b in [0, K]; NULL means K for every request.
 *                              Out-of-range values are clamped (SPEC_DEV_BAD_LEN).
 *   temperature   [B]          float32 per-request temperature T_b.  A request
 *                              is GREEDY when T_b is not a positive normal
 *                              float (T <= 0, NaN, inf, or below FLT_MIN):
 *                              draft token k is accepted iff it equals the
 *                              target argmax of row k (ties: lowest index),
 *                              and the emitted token is that argmax.
 *                              Otherwise SAMPLED: p = softmax(z/T) of the
 *                              target row, q = softmax(z'/T) of the draft row
 *                              (the same T), accept x_k iff u_k * q(x_k) <
 *                              p(x_k) with u_k a Philox uniform on a 2^-24
 *                              grid; at the first rejection a the emitted token
 *                              is drawn from max(0, p_a - q_a) (from p_a if that
 *                              mass is zero); if all L_b drafts are accepted it
 *                              is drawn from p at row L_b.  Draws are by
 *                              inverse CDF in ascending token order with a
 *                              Philox uniform on a 2^-53 grid.
 *   seed                       64-bit key of the Philox4x32-10 generator.
 *   B, K, V                    1 <= B < 2^24, 1 <= K <= SPEC_MAX_K,
 *                              2 <= V <= SPEC_MAX_V.
 *   out_tokens    [B, K+1]     int32, written: x_0..x_{a-1}, the emitted token
 *                              at position a, -1 after it.
 *   accept_len    [B]          int32, written: a (number of accepted drafts).
 *   workspace, workspace_bytes scratch of at least
 *                              spec_verify_workspace_bytes(B, K, V, dtype).
 *   dev_status                 nullable device uint32, see SPEC_DEV_*.
 *   stream                     cudaStream_t (as void*).
 *
 * Alignment: logits base pointers must be 16-byte aligned; rows whose byte
 * length V*sizeof(dtype) is not a multiple of 16 take a slower scalar path.
 * Logit values: -inf is legal (probability 0); NaN and +inf are not supported
 * (results unspecified, no fault); every row must hold a finite logit.
 */
spec_status_t spec_verify(const void *target_logits, const void *draft_logits,
                          spec_dtype_t dtype, const int32_t *draft_tokens,
                          const int32_t *verify_len, const float *temperature, uint64_t seed,
                          int B, int K, int V, int32_t *out_tokens, int32_t *accept_len,
                          void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                          void *stream);

/*
 * spec_verify_debug -- spec_verify plus the intermediates used for parity:
 *   row_stats [B, 2K+1, 2] float64: for target rows k = 0..K (index k) and draft
 *             rows k = 0..K-1 (index K+1+k): { max_v z_v/T, log sum_v exp(z_v/T - max) }.
 *             Rows the step did not read (beyond the verify length, draft rows of
 *             greedy requests, all rows of greedy requests) hold NaN.
 *   probs     [B, K, 2] float64: { p_k(x_k), q_k(x_k) } for sampled requests and
 *             k < L_b; NaN elsewhere.
 * Either pointer may be NULL.  Same contract otherwise.
 */
spec_status_t spec_verify_debug(const void *target_logits, const void *draft_logits,
                                spec_dtype_t dtype, const int32_t *draft_tokens,
                                const int32_t *verify_len, const float *temperature,
                                uint64_t seed, int B, int K, int V, int32_t *out_tokens,
                                int32_t *accept_len, void *workspace, size_t workspace_bytes,
                                uint32_t *dev_status, double *row_stats, double *probs,
                                void *stream);

/*
 * spec_verify_early_exit -- spec_verify with the positions verified in two
 * waves, [0, first_wave) and then [first_wave, K): a request whose first
 * rejection falls in the first wave (or whose verify length is at most
 * first_wave) needs no logit row of the second.  The outputs are bit-identical
 * to spec_verify's; the rows after a rejection are never read ("speculative
 * decoding от черновика до проверки" (braintools.ru), "Как это работает",
 * step 3: the drafts are checked left to right and the first mismatch ends the
 * step).  first_wave >= 1 (first_wave >= K is one wave, the spec_verify
 * path); otherwise SPEC_ERR_INVALID_ARG.  The workspace is the one
 * spec_verify_workspace_bytes gives.  Same contract as spec_verify otherwise;
 * it launches 8 kernels (5 with one wave).
 */
spec_status_t spec_verify_early_exit(const void *target_logits, const void *draft_logits,
                                     spec_dtype_t dtype, const int32_t *draft_tokens,
                                     const int32_t *verify_len, const float *temperature,
                                     uint64_t seed, int B, int K, int V, int first_wave,
                                     int32_t *out_tokens, int32_t *accept_len, void *workspace,
                                     size_t workspace_bytes, uint32_t *dev_status, void *stream);

/*
 * spec_verify_tree_greedy -- greedy verification of a candidate tree
 * ("speculative decoding от черновика до проверки" (braintools.ru), the Medusa
 * and EAGLE-2 passages: the draft is a tree of candidates the target checks in
 * one pass with tree attention; "Почему ответ не портится?": at temperature 0
 * a draft token is kept when it equals the target's argmax).
 *   Node 0 of each request is the root (the last committed token); node n >= 1
 *   carries node_tokens[b, n] and parent[b, n] < n.  target_logits [B, N, V]
 *   bf16/fp32 device, row n = the target's logits after node n's token (from
 *   tree attention).  Walk from the root: t = argmax of the current node's row
 *   (lowest index on ties); the next node is the lowest-index child carrying t;
 *   without one, t is emitted and the walk ends.
 *   Outputs (device int32): out_tokens [B, N] = the accepted tokens then the
 *   emitted one, -1 after; out_nodes [B, N] = the accepted node indices, -1
 *   after; accept_len [B] = the number of accepted nodes.
 *   1 <= N <= SPEC_MAX_TREE.  A node whose parent is not an earlier node
 *   belongs to no path (SPEC_DEV_BAD_TREE).  The workspace is
 *   spec_tree_workspace_bytes(B, N, V, dtype) bytes.  Errors as spec_verify.
 *   Sampled (T > 0) requests: spec_verify_tree.
 */
size_t spec_tree_workspace_bytes(int B, int N, int V, spec_dtype_t dtype);
spec_status_t spec_verify_tree_greedy(const void *target_logits, spec_dtype_t dtype,
                                      const int32_t *parent, const int32_t *node_tokens, int B,
                                      int N, int V, int32_t *out_tokens, int32_t *out_nodes,
                                      int32_t *accept_len, void *workspace, size_t workspace_bytes,
                                      uint32_t *dev_status, void *stream);

/*
 * spec_verify_tree -- verification of candidate trees at each request's
 * temperature: greedy requests (T not a positive normal float) take the walk
 * of spec_verify_tree_greedy; sampled requests apply the acceptance rule of
 * "Спекулятивный декодинг в проде" (kiosknews.app), "Правило проверки", to
 * every candidate of the tree, siblings in index order against successively
 * updated residuals (the multi-candidate form of the rule):
 *   at node u the weights r start as p_u = softmax(target row u / T); child c
 *   (token x; a token outside [0, V) is no candidate) is accepted iff
 *   u_acc * q_u(x) < r(x) / Z, q_u = softmax(draft row u / T); a rejection
 *   sets r = max(0, r / Z - q_u) with Z its sum (zero mass: r = p_u again).
 *   An accepted child becomes the current node; with none accepted the
 *   emitted token is the inverse CDF of r (smallest v whose inclusive prefix
 *   exceeds u_s * Z) and the walk ends.  With one child per node this is
 *   spec_verify's rule step for step; with the siblings of node u drawn
 *   independently from q_u the emitted tokens follow the target exactly.
 *   Uniforms: candidate node c uses the acceptance uniform of position c - 1
 *   and node u's emitted token the sampling uniform of position u (Philox keys
 *   as spec_verify), so a chain tree draws spec_verify's numbers.
 *   target_logits [B, N, V], draft_logits [B, N-1, V] (row n: the draft's
 *   logits after node n; the last node has no children; may be NULL when
 *   N = 1), both bf16/fp32 device and 16-byte aligned; parent, node_tokens
 *   [B, N] int32; temperature [B] float32 device.  Outputs as
 *   spec_verify_tree_greedy; the workspace is spec_tree_workspace_bytes.
 *   Each sampled request costs one pass over its vocabulary per rejected
 *   candidate, run by a thread-block cluster of up to 8 CTAs (as many as the
 *   batch leaves SMs free; one CTA each at large batches).  After a staging
 *   wait runs out (SPEC_DEV_TIMEOUT) the request's outputs are undefined but
 *   in range.  Errors as spec_verify.
 */
spec_status_t spec_verify_tree(const void *target_logits, const void *draft_logits,
                               spec_dtype_t dtype, const int32_t *parent,
                               const int32_t *node_tokens, const float *temperature, uint64_t seed,
                               int B, int N, int V, int32_t *out_tokens, int32_t *out_nodes,
                               int32_t *accept_len, void *workspace, size_t workspace_bytes,
                               uint32_t *dev_status, void *stream);

/*
 * spec_verify_tree_distinct -- spec_verify_tree for trees whose siblings are
 * DISTINCT tokens drawn one after another without replacement from their
 * parent's draft distribution q_u: the several candidates per position of
 * "Спекулятивное декодирование в vLLM и SGLang: MTP, EAGLE-3 и n-gram в 2026"
 * (alesha.pro; the EAGLE top-k tree of candidates) and of "Спекулятивный
 * декодинг в проде" (kiosknews.app), "7. DFlash 2" (16 candidates per
 * position).  The sibling checked after rejected siblings carrying tokens X
 * was drawn from q_u without X, renormalised by its remaining mass 1 - q_u(X);
 * the acceptance test and the residual update use that law (the residual keeps
 * the closed form of spec_verify_tree, its threshold step divided by the
 * remaining mass).  A sibling repeating a rejected sibling's token, or checked
 * when q_u has no mass left, could not have been drawn and is no candidate.
 * With the siblings drawn that way the emitted tokens follow the target
 * exactly.  Arguments, outputs, errors and workspace as spec_verify_tree;
 * chains give spec_verify_tree's (and spec_verify's) outputs.
 */
spec_status_t spec_verify_tree_distinct(const void *target_logits, const void *draft_logits,
                                        spec_dtype_t dtype, const int32_t *parent,
                                        const int32_t *node_tokens, const float *temperature,
                                        uint64_t seed, int B, int N, int V, int32_t *out_tokens,
                                        int32_t *out_nodes, int32_t *accept_len, void *workspace,
                                        size_t workspace_bytes, uint32_t *dev_status, void *stream);

/*
 * spec_draft_confidence -- the draft's confidence at every position, as the
 * confidence-scheduled verification of "DSpark: ... верификацией по
 * уверенности" (iitog.ru), "Ключевые факты", uses it: maxprob[b, k] =
 * max_v q_k(v) with q_k = softmax(draft_logits[b, k] / T_b), that is
 * 1 / sum_v exp((z_v - max z) / T_b); 1 for greedy requests (T_b not a
 * positive normal float: q is a point mass).  One pass over the draft rows of
 * the sampled requests.
 *   draft_logits [B, K, V] bf16/fp32 device (16-byte aligned), temperature [B]
 *   float32 device, maxprob [B, K] float32 device (written), relative accuracy
 *   ~1e-6.  The workspace is the one spec_verify_workspace_bytes gives for the
 *   same B, K, V.  Errors as spec_verify.
 */
spec_status_t spec_draft_confidence(const void *draft_logits, spec_dtype_t dtype,
                                    const float *temperature, int B, int K, int V,
                                    float *maxprob, void *workspace, size_t workspace_bytes,
                                    void *stream);

/*
 * spec_schedule_budget -- the load-aware side of the same schedule: the
 * verify length follows the prefix's survival probability and the engine's
 * current load.  Given the number of positions the engine verifies this step
 * (budget, from its load), keep the budget positions (b, k) with the largest
 * survival s[b, k] = c[b, 0] * ... * c[b, k] (c = draft_maxprob clamped to
 * [0, 1], NaN as 0; float32 products left to right, each rounded to nearest),
 * ties to the lower b, then the lower k.  Survival never grows along a
 * request, so the kept positions are a prefix of every request:
 * verify_len[b] is its length (budget <= 0: all 0; budget >= B*K: all K).
 *   draft_maxprob [B, K] float32 device, verify_len [B] int32 device (written).
 *   1 <= B < 2^24, 1 <= K <= SPEC_MAX_K, B * K <= 2^22 (else
 *   SPEC_ERR_UNSUPPORTED).  Bit-exact with a sort of the survival values.
 */
spec_status_t spec_schedule_budget(const float *draft_maxprob, int B, int K, long long budget,
                                   int32_t *verify_len, void *stream);

/*
 * spec_schedule_len -- confidence-scheduled verify length (DSpark, iitog.ru):
 *   verify_len[b] = number of leading positions k whose running product
 *   prod_{j<=k} draft_maxprob[b, j] stays >= threshold, the product taken left
 *   to right in float32 with every step rounded to nearest (no fused
 *   multiply-add).  The empty product is 1, so verify_len[b] >= 0; NaN stops
 *   the scan.
 *   draft_maxprob [B, K] float32 device, verify_len [B] int32 device (written).
 *   1 <= B < 2^24, 1 <= K <= SPEC_MAX_K.
 */
spec_status_t spec_schedule_len(const float *draft_maxprob, float threshold, int B, int K,
                                int32_t *verify_len, void *stream);

/*
 * spec_verify_scheduled -- confidence-scheduled verification in one call: the
 * draft's confidences, the verify lengths they give, and the verification
 * step, with every draft row read once.  "DSpark: ... верификацией по
 * уверенности" (iitog.ru), "Ключевые факты": the verify length of each request
 * follows the estimated survival of its draft prefix and the engine's load;
 * "Спекулятивный декодинг в проде" (kiosknews.app), "6. DSpark", "Грабли":
 * the scheduler cuts the draft where the drafter is unsure, and doing that
 * trimming on the GPU was the missing piece.
 *   draft_maxprob [B, K] float32 device, or NULL.  NULL: the confidences are
 *       computed from the draft rows, max_v q_k(v) as spec_draft_confidence
 *       gives them (1 for greedy requests), by one statistics pass over the
 *       sampled requests' draft rows whose per-row partials the step then reuses
 *       (its own statistics pass reads target rows only).  Given: they are
 *       used as they are and the step reads the draft rows it needs itself.
 *   mode SPEC_SCHED_THRESHOLD: verify_len[b] is the spec_schedule_len rule at
 *       `threshold` (formed per request inside the step's first kernel);
 *       SPEC_SCHED_BUDGET: the spec_schedule_budget rule with `budget`
 *       positions (B * K <= 2^22, else SPEC_ERR_UNSUPPORTED).
 *   maxprob_out [B, K] float32 device, nullable: receives the computed
 *       confidences (written only when draft_maxprob is NULL).
 *   verify_len_out [B] int32 device, nullable: receives the scheduled lengths
 *       (before the draft-token check of spec_verify, which may cut them).
 *   Everything else as spec_verify (the same workspace size).  The outputs
 *   are bit-identical to spec_draft_confidence (when draft_maxprob is NULL),
 *   then spec_schedule_len / spec_schedule_budget, then spec_verify on the
 *   same inputs.  Launches 5 kernels (threshold, confidences given), plus 3
 *   for the confidences and 1 for a budget.
 */
typedef enum {
    SPEC_SCHED_THRESHOLD = 0, /* survival product >= threshold */
    SPEC_SCHED_BUDGET = 1     /* the `budget` positions of highest survival */
} spec_sched_mode_t;
spec_status_t spec_verify_scheduled(const void *target_logits, const void *draft_logits,
                                    spec_dtype_t dtype, const int32_t *draft_tokens,
                                    const float *temperature, uint64_t seed, int B, int K, int V,
                                    const float *draft_maxprob, spec_sched_mode_t mode,
                                    float threshold, long long budget, float *maxprob_out,
                                    int32_t *verify_len_out, int32_t *out_tokens,
                                    int32_t *accept_len, void *workspace, size_t workspace_bytes,
                                    uint32_t *dev_status, void *stream);

/*
 * spec_verify_lmhead -- the verification step with its input side fused: the
 * logits come from the LM-head product of the hidden states, computed on the
 * tensor cores, and are consumed in that product's epilogue instead of being
 * written to memory ("speculative decoding от черновика до проверки"
 * (braintools.ru), "Как это работает", step 2: the target scores all drafts
 * in one pass, whose last step is the vocabulary projection; the same page
 * stresses that moving weights and activations through memory is the cost).
 *   hidden_target [B, K+1, d]  bf16, row (b, k) = the target's last hidden
 *                              state at position k; target logits row (b, k)
 *                              = hidden_target[b, k] . w_target^T.
 *   hidden_draft  [B, K, d]    bf16, the drafter's hidden states; draft logits
 *                              row (b, k) = hidden_draft[b, k] . w_draft^T.
 *   w_target, w_draft [V, d]   bf16 row-major LM-head weights (may be the same
 *                              buffer, as when the drafter shares the target's
 *                              head).  All four 16-byte aligned.
 *   d                          hidden size, a multiple of 64, at most 65536.
 *   V                          a multiple of 4.
 *   The logits are the fp32 accumulations of the bf16 products (tensor-core
 *   order); the step is then spec_verify's on those fp32 values: the same
 *   rule, outputs, uniforms, status bits and errors.  Every target row and
 *   every draft row is multiplied (the verify lengths and greedy requests do
 *   not shrink the product); the few rows the sampler draws from (one or two
 *   per sampled request) are multiplied again after the decisions, into the
 *   workspace.  row_stats / probs: as spec_verify_debug (nullable).
 *   workspace: spec_lmhead_workspace_bytes(B, K, V, d) bytes, 256-byte
 *   aligned (it holds 8 B V bytes of recomputed rows).  Launches 7 kernels when
 *   w_target == w_draft (the target and draft rows share one product launch
 *   and one recompute), 9 otherwise.
 */
size_t spec_lmhead_workspace_bytes(int B, int K, int V, int d);
spec_status_t spec_verify_lmhead(const void *hidden_target, const void *hidden_draft,
                                 const void *w_target, const void *w_draft, int d,
                                 const int32_t *draft_tokens, const int32_t *verify_len,
                                 const float *temperature, uint64_t seed, int B, int K, int V,
                                 int32_t *out_tokens, int32_t *accept_len, void *workspace,
                                 size_t workspace_bytes, uint32_t *dev_status, double *row_stats,
                                 double *probs, void *stream);

/*
 * spec_profile_events -- measurement hook.  When both events are non-NULL
 * (cudaEvent_t values passed as void*), every later spec_verify /
 * spec_verify_debug call records ev_start immediately before and ev_end
 * immediately after the launch of its dominant (logit-streaming) kernel, on
 * the call's stream, so a caller can time that kernel alone.  Pass NULL, NULL
 * to switch it off.  Process-global, not thread-safe; the events stay owned by
 * the caller.
 */
void spec_profile_events(void *ev_start, void *ev_end);

/* Number of kernels one spec_verify call launches (for launch accounting). */
int spec_verify_kernel_count(void);

/*
 * spec_verify_noalloc -- spec_verify without a caller-provided workspace, for
 * callers that cannot allocate device memory at the call site: code that runs
 * under a no-allocation rule (latency-critical serving loops, where cudaMalloc
 * can synchronise the device), plugins of frameworks that own every device
 * allocation, or callers that simply have no scratch buffer to hand.  The
 * pages have no counterpart to this entry point; it is a deployment aid.
 *
 * The scratch is a library-owned static device array of
 * SPEC_NOALLOC_SCRATCH_BYTES, resident on every GPU that loads the library
 * until the process exits.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.  The call itself allocates nothing
 * and frees nothing.  Problems whose workspace (spec_verify_workspace_bytes)
 * exceeds SPEC_NOALLOC_SCRATCH_BYTES are rejected with SPEC_ERR_WORKSPACE
 * before anything is launched.  Every call on a device shares the one array
 * and it keeps the last call's contents (no field needs to start at zero):
 * calls that may overlap on the GPU (different streams, no ordering) race and
 * must be serialised by the caller.  Arguments and results are otherwise those
 * of spec_verify.
 */
#define SPEC_NOALLOC_SCRATCH_BYTES (32u << 20)
spec_status_t spec_verify_noalloc(const void *target_logits, const void *draft_logits,
                                  spec_dtype_t dtype, const int32_t *draft_tokens,
                                  const int32_t *verify_len, const float *temperature,
                                  uint64_t seed, int B, int K, int V, int32_t *out_tokens,
                                  int32_t *accept_len, uint32_t *dev_status, void *stream);

/*
 * spec_verify_from_host -- spec_verify for inputs held in host memory, with
 * the copies over the host link limited to what the step reads.  The step of
 * "Спекулятивный декодинг в проде" (kiosknews.app), "Правило проверки", reads
 * for request b, with L_b its verify length clamped to [0, K], the target rows
 * 0..L_b and, when the request is sampled, the draft rows 0..L_b-1; a greedy
 * request reads no draft row.  The call, in stream order:
 *   1. copies draft_tokens, verify_len (when given) and temperature to their
 *      device buffers, and those rows of the logits to the same places of
 *      target_dev / draft_dev (one copy per run of adjacent rows);
 *   2. runs spec_verify on the device buffers;
 *   3. copies out_tokens_dev and accept_len_dev to out_tokens_host and
 *      accept_len_host.
 *   *_host inputs          host memory with spec_verify's layouts; the
 *                          greedy / sampled split and the clamp follow
 *                          spec_verify's rules (T not a finite value >=
 *                          FLT_MIN: greedy), read from verify_len_host and
 *                          temperature_host during the call.  verify_len_host
 *                          NULL: L_b = K (verify_len_dev is then unused).
 *   target_dev, draft_dev  device [B, K+1, V] / [B, K, V] buffers, 16-byte
 *                          aligned; rows the step does not read keep whatever
 *                          they held.
 *   draft_tokens_dev, verify_len_dev, temperature_dev, out_tokens_dev,
 *   accept_len_dev         device buffers of spec_verify's shapes.
 *   out_tokens_host, accept_len_host   host outputs [B, K+1], [B].
 *   workspace, dev_status  as spec_verify.
 *   h2d_bytes              nullable: the bytes copied host to device.
 * Everything is asynchronous on `stream` and nothing is allocated: the host
 * buffers must stay valid and unchanged until the stream has passed the
 * call (pinned host memory lets the copies run asynchronously).  Errors as
 * spec_verify, plus SPEC_ERR_INVALID_ARG for a missing buffer and
 * SPEC_ERR_CUDA when a copy cannot be enqueued (copies already enqueued may
 * then have run).
 */
spec_status_t spec_verify_from_host(
    const void *target_host, const void *draft_host, spec_dtype_t dtype,
    const int32_t *draft_tokens_host, const int32_t *verify_len_host,
    const float *temperature_host, uint64_t seed, int B, int K, int V, void *target_dev,
    void *draft_dev, int32_t *draft_tokens_dev, int32_t *verify_len_dev, float *temperature_dev,
    int32_t *out_tokens_dev, int32_t *accept_len_dev, int32_t *out_tokens_host,
    int32_t *accept_len_host, void *workspace, size_t workspace_bytes, uint32_t *dev_status,
    void *stream, size_t *h2d_bytes);

/*
 * spec_verify_scheduled_from_host -- spec_verify_from_host for lengths set by
 * a schedule of given draft confidences ("DSpark: спекулятивное
 * декодирование с верификацией по уверенности…" (iitog.ru), "Ключевые
 * факты"): the confidences go to the device, the schedule of mode (threshold:
 * spec_schedule_len; budget: spec_schedule_budget) runs there and writes
 * verify_len_dev, the lengths come back to verify_len_host, and the call
 * WAITS for them (one cudaStreamSynchronize of `stream`) before it copies
 * the logit rows those lengths need and runs the step as
 * spec_verify_from_host does.  Only that wait is synchronous.
 *   draft_maxprob_host [B, K] float32 host; maxprob_dev its device buffer.
 *   verify_len_dev, verify_len_host  [B] int32 device / host (written).
 *   Other arguments as spec_verify_from_host; h2d_bytes includes the
 *   confidences.
 * Errors as spec_verify_from_host and spec_verify_scheduled (mode, budget
 * size).
 */
spec_status_t spec_verify_scheduled_from_host(
    const void *target_host, const void *draft_host, spec_dtype_t dtype,
    const int32_t *draft_tokens_host, const float *temperature_host,
    const float *draft_maxprob_host, uint64_t seed, int B, int K, int V, spec_sched_mode_t mode,
    float threshold, long long budget, void *target_dev, void *draft_dev,
    int32_t *draft_tokens_dev, float *temperature_dev, float *maxprob_dev, int32_t *verify_len_dev,
    int32_t *out_tokens_dev, int32_t *accept_len_dev, int32_t *out_tokens_host,
    int32_t *accept_len_host, int32_t *verify_len_host, void *workspace, size_t workspace_bytes,
    uint32_t *dev_status, void *stream, size_t *h2d_bytes);

/*
 * spec_debug_force_wait_timeout -- diagnostics only: while enabled (1), every
 * warp of the bulk-copy kernels in later spec_verify calls (any device) first
 * waits on a barrier nothing completes; that bounded wait runs out after 1 ms
 * and the warp gives up as on a real timeout: SPEC_DEV_TIMEOUT in the status
 * word, its copies in flight drained (with the 2 s limit), its items skipped
 * (outputs then undefined but in range).  In spec_verify_tree calls, each
 * staging of node rows in the sampled walk first waits on such a barrier,
 * reports SPEC_DEV_TIMEOUT and then waits for its copies as usual (outputs
 * unchanged).  0 turns it off.  No counterpart on the pages: it exercises the
 * failure path of the bounded waits.
 */
spec_status_t spec_debug_force_wait_timeout(int enable);

/* Static description of a status code. */
const char *spec_status_str(spec_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
