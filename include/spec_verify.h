/*
 * spec_verify.h -- C ABI of libspecverify.so, the batched speculative-decoding verifier for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (pages: "投机解码" [Speculative decoding], rustineverything, sections
 * 目标模型怎么一次验证 [how the target verifies in one pass] and 接受规则为什么不改变分布 [why
 * the acceptance rule keeps the distribution]; "The speculative decoding zoo",
 * mlinterviewnotes 06-06, DFlash section and verification-method section):
 * the target model has produced, for each of B requests, logits for k+1 positions, where
 * position i conditions on the prefix and the first i drafts.  With p = softmax(logits / T),
 * drafts are accepted left to right with probability min(1, p(x) / q(x)); the first rejected
 * position is replaced by a draw from max(0, p - q) / Z; when all k are accepted one bonus
 * token is drawn from position k+1.  Each request therefore emits 1 to k+1 tokens, and
 * accept_len (the accepted draft count) tells the caller how many KV entries to keep.
 *
 * Conventions shared by every entry point
 *   - All array pointers are DEVICE pointers owned by the caller, contiguous, row-major.
 *     Logits must be aligned to their element size; any further alignment is optional
 *     (16-byte aligned rows take the vectorised path everywhere).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls only enqueue
 *     work on it; none synchronises the host, and none allocates memory.
 *   - The first call on a device (of any entry point, with that device current) reads its SM
 *     count and shared memory per SM and raises the dynamic shared-memory limits of the kernels
 *     that take more than the default (cudaFuncSetAttribute: the finalising kernels, which size
 *     their request so that at most ceil(B / SMs) of their CTAs share an SM, and the top-k / top-p
 *     ring kernel's 109 KiB); make it before any stream capture on that device.  The library keeps
 *     this per device for the life of the process, so it must not be used again after
 *     cudaDeviceReset.
 *   - The return value is a host status, known when the call returns:
 *       SPEC_VERIFY_OK, SPEC_VERIFY_EINVAL (bad argument), SPEC_VERIFY_EWORKSPACE
 *       (workspace too small or misaligned), SPEC_VERIFY_ECUDA (a launch failed).
 *     On a non-OK return nothing was enqueued (ECUDA: possibly part of it).
 *   - `dev_status` (optional, may be NULL) is a device int32.  The kernels raise it with an
 *     atomic maximum when they detect a fault in the data; they never clear it.  The caller
 *     zeroes it and reads it after the stream completes.  Codes: SPEC_VERIFY_DEV_*.
 *     A faulted request gets out_tokens = -1, accept_len = -1 (and accept_index = -1).
 *   - `workspace` is device scratch of at least spec_verify_workspace_bytes(...) bytes,
 *     256-byte aligned, ZERO-FILLED before its first use.  Every call leaves the part that
 *     must start at zero (per-request arrival counters, kept in a fixed region at the start of
 *     the workspace whatever the call's shape) zero again when it completes, so a workspace is
 *     zeroed once and reused by calls of any mode and shape.  Two calls in flight at the same
 *     time (different streams) must not share a workspace.
 *   - Random numbers: Philox4x32-10 (Salmon et al., SC'11) with key = (seed low word, seed
 *     high word) and counter = (slot, request, offset low word, offset high word).  Output
 *     word 0 gives u (the accept test, or the tree coin), word 1 gives v (the draw at the stop
 *     slot); a word x maps to (x >> 8) * 2^-24.  slot = draft position (chain) or depth (tree).
 *     A call uses only counters whose last two words equal `offset`: advance offset by one
 *     per call to get fresh randomness; the same (seed, offset) replays bit-exactly.
 *   - Draws use the inverse CDF in ascending token order: the smallest y whose running sum
 *     of the (unnormalised) weights exceeds v * Z.
 *   - Limits: 1 <= B <= 65536, 0 <= k <= 63 (chain), 1 <= N <= 64 (tree), 1 <= V < 2^31,
 *     B * rows * ceil((V + 7) / 4096) < 2^31 (bf16; fp32: 2048 in place of 4096), and
 *     |logit| / T must stay below 2^127 (the scaled logit is formed in fp32).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Logit element types. */
#define SPEC_VERIFY_BF16 0
#define SPEC_VERIFY_FP32 1

/* Host return codes. */
#define SPEC_VERIFY_OK 0
#define SPEC_VERIFY_EINVAL (-1)
#define SPEC_VERIFY_EWORKSPACE (-2)
#define SPEC_VERIFY_ECUDA (-3)
#define SPEC_VERIFY_ETOOBIG (-4) /* problem needs more than the built-in no-alloc scratch */

/* Device status codes (largest wins). */
#define SPEC_VERIFY_DEV_OK 0
#define SPEC_VERIFY_DEV_BAD_TOKEN 1   /* a draft / node token outside [-1, V) */
#define SPEC_VERIFY_DEV_BAD_ROW 2     /* a logit row holding NaN or +inf, or no finite value */
#define SPEC_VERIFY_DEV_BAD_TREE 3    /* parents[0] != -1, or parents[j] outside [0, j) */
#define SPEC_VERIFY_DEV_DUP_SIBLING 4 /* two children of one node share a token (target-only) */
#define SPEC_VERIFY_DEV_BAD_KV_POSITION 5 /* KV compaction: committed + N beyond the slot table,
                                             accept_len >= N, or a path entry outside [0, N) */
#define SPEC_VERIFY_DEV_BAD_KV_SLOT 6     /* KV compaction: a slot outside [0, num_slots) */

/* Modes for spec_verify_workspace_bytes. */
#define SPEC_VERIFY_MODE_GREEDY 0
#define SPEC_VERIFY_MODE_REJECTION 1
#define SPEC_VERIFY_MODE_TREE 2
#define SPEC_VERIFY_MODE_BLOCK 3

/*
 * Greedy chain verification ("The speculative decoding zoo", DFlash section: matches =
 * draft == argmax of the previous position, correct_len = cumprod(matches).sum, bonus =
 * argmax[correct_len]; "投机解码", subsection 贪心 [greedy]: a draft is accepted iff it equals
 * the target argmax, and on rejection the argmax is emitted without resampling).
 *   logits     [B][k+1][V], dtype SPEC_VERIFY_BF16 or SPEC_VERIFY_FP32
 *   draft_ids  [B][k] int32 in [-1, V); -1 means "no draft here" and ends the chain
 *   out_tokens [B][k+1] int32: accepted drafts, then the argmax at the stop position, then -1
 *   accept_len [B] int32: accepted drafts (0..k); emitted tokens = accept_len + 1
 * Argmax ties go to the lowest token index.  No temperature and no random numbers.
 */
int spec_verify_greedy(const void *logits, int dtype, const int32_t *draft_ids, int B, int k,
                       int V, int32_t *out_tokens, int32_t *accept_len, void *workspace,
                       size_t ws_bytes, int32_t *dev_status, void *stream);

/*
 * Sampled chain verification: standard rejection sampling when draft_probs is given, the
 * one-hot ("target-only") rule when it is NULL ("投机解码", subsections 采样：标准拒绝采样
 * [standard rejection] and 默认路径：草稿当 one-hot [default: one-hot draft]; "The speculative
 * decoding zoo", verification-method section: with a one-hot q, min(1, p/q) = p(x)).
 *   logits      [B][k+1][V] bf16 / fp32; p = softmax(logits / temperature)
 *   draft_ids   [B][k] int32 in [-1, V)
 *   draft_probs [B][k][V] fp32 draft distributions q, or NULL (q = one-hot at the draft)
 *   temperature > 0 and finite (use spec_verify_greedy for T = 0)
 *   out_tokens  [B][k+1] int32, accept_len [B] int32 (as for greedy)
 *   out_probs   optional [B][k+1][3] fp32 parity aid: for each position i < k with a draft,
 *               p_i(x_i) and q_i(x_i) (1 for one-hot); at the stop position j = accept_len,
 *               column 2 holds the normaliser Z of the distribution drawn from (the residual
 *               mass sum max(0, p - q), or 1 for a bonus or absent-draft draw); zeros elsewhere.
 * Accept test: u * q(x) < p(x) (so q(x) = 0 accepts iff p(x) > 0; p(x) = 0 never accepts).
 * If the residual mass underflows to zero the draw falls back to p.
 */
int spec_verify_rejection(const void *logits, int dtype, const int32_t *draft_ids,
                          const float *draft_probs, int B, int k, int V, float temperature,
                          uint64_t seed, uint64_t offset, int32_t *out_tokens,
                          int32_t *accept_len, float *out_probs, void *workspace,
                          size_t ws_bytes, int32_t *dev_status, void *stream);

/*
 * Block verification of a chain ("The speculative decoding zoo", mlinterviewnotes 06-06, the
 * block branch of the rejection sampler, citing Sun et al. 2024, arXiv:2403.10444): the prefix
 * of L drafts is judged as a whole.  With w_0 = 1 and w_{i+1} = min(1, w_i p_i(x)/q_i(x)) (q is
 * one-hot at the draft when draft_probs is NULL), candidate length L passes iff
 * u_L < h_L = r_L / (r_L + 1 - w_L), r_L = sum_y max(w_L p_L(y) - q_L(y), 0) (h_L = 1 when the
 * denominator is 0), and h = w at the last present draft; u_L is word 0 of Philox slot L - 1.
 * The accepted length j is the largest passing L (0 if none); the token after the prefix is
 * drawn by inverse CDF (v = word 1 of slot j) from max(w_j p_j - q_j, 0), or from p_j at the
 * last present draft (a bonus when all k are present), falling back to p_j if that mass is 0.
 *   Arguments, outputs and status codes as for spec_verify_rejection (no out_probs).
 *   Workspace: spec_verify_workspace_bytes(SPEC_VERIFY_MODE_BLOCK, B, k, V).
 * With draft_probs the residual masses need every row's softmax, so a third kernel re-reads
 * the logits and q of rows 0..j_max of each request; with one-hot drafts r_L is w_L times the
 * row's non-draft mass and no extra pass is made.
 */
int spec_verify_block(const void *logits, int dtype, const int32_t *draft_ids,
                      const float *draft_probs, int B, int k, int V, float temperature,
                      uint64_t seed, uint64_t offset, int32_t *out_tokens, int32_t *accept_len,
                      void *workspace, size_t ws_bytes, int32_t *dev_status, void *stream);

/*
 * Tree verification ("投机解码", subsection SGLang 默认：只看目标概率，可以验证一棵树
 * [SGLang default: target probabilities only, can verify a tree]: one coin per tree level,
 * siblings tried in order with a running sum of their target probabilities, residual =
 * p with the tried siblings zeroed; greedy trees follow the child equal to the argmax).
 *   logits       [B][N][V] bf16 / fp32: row n is the target distribution for node n's children
 *   node_tokens  [B][N] int32: token of each node; node 0 is the root (its token is ignored);
 *                -1 marks an absent node, which is never tried
 *   parents      [B][N] int32: parents[.][0] = -1 and 0 <= parents[.][j] < j for j >= 1;
 *                children of a node are tried in ascending node index
 *   mode         0 = greedy (temperature, seed, offset ignored), 1 = target-only sampling
 *   out_tokens   [B][N] int32: tokens of the accepted nodes, then the token drawn at the stop
 *                node (argmax in greedy mode; a bonus draw when the stop node is a leaf)
 *   accept_index [B][N] int32: node 0, then the accepted nodes in path order, then -1
 *   accept_len   [B] int32: accepted nodes (the root not counted)
 * Coin test at node n: the first child c with p_n(tok_c) > 0 and coin < sum of p_n over the
 * children tried so far (c included) is accepted.  Sibling tokens must be distinct in mode 1.
 */
int spec_verify_tree(const void *logits, int dtype, const int32_t *node_tokens,
                     const int32_t *parents, int B, int N, int V, int mode, float temperature,
                     uint64_t seed, uint64_t offset, int32_t *out_tokens, int32_t *accept_index,
                     int32_t *accept_len, void *workspace, size_t ws_bytes, int32_t *dev_status,
                     void *stream);

/*
 * Verify variants: a temperature per request and relaxed acceptance thresholds.
 *   temperatures    [B] float, device, or NULL.  Request b samples at temperatures[b] > 0 or is
 *                   greedy when temperatures[b] == 0: a batch may mix both ("The speculative
 *                   decoding zoo", DSpark section: the greedy rule for greedy requests, the
 *                   sampling rule for the others, merged).  NULL: every request uses
 *                   `temperature` (0 = all greedy).
 *   threshold_single, threshold_acc
 *                   in (0, 1]; 1 is the exact rule.  Target-only decisions (chain without draft
 *                   probabilities; tree) accept a candidate c with p(c) > 0 when the coin is below
 *                   (running sum of the tried candidates' p) / threshold_acc, or when
 *                   p(c) >= threshold_single ("投机解码", section 接受规则为什么不改变分布,
 *                   SGLang 默认 subsection and its remark on the two thresholds): values below 1
 *                   accept more and no longer preserve the target distribution.  With draft
 *                   probabilities both must be 1 (SPEC_VERIFY_EINVAL otherwise).
 *   top_k, top_p    [B] int32 / float, device, or NULL: p is the target distribution after
 *                   temperature, top-k and top-p ("投机解码", section 接受规则为什么不改变分布).
 *                   Top-k keeps every token whose logit reaches the k-th largest logit (ties kept
 *                   whole; k <= 0 or k >= V: off); top-p then keeps the fewest whole value levels
 *                   from the top whose probability, renormalised over the top-k set, reaches top_p
 *                   (>= 1: off; <= 0 keeps the top level).  p is renormalised over what is kept;
 *                   greedy requests are unaffected.  Two extra kernels find each row's logit
 *                   threshold first: one that reads each bf16 row once (top-k <= 256), then a
 *                   general one for the rows it leaves (top-p alone, larger k, fp32 logits; two
 *                   to five passes over a row).
 */
typedef struct spec_verify_options {
    const float *temperatures;
    float temperature;
    float threshold_single;
    float threshold_acc;
    const int32_t *top_k;
    const float *top_p;
} spec_verify_options;

/*
 * spec_verify_rejection with options: arguments, layouts, outputs and status codes as for
 * spec_verify_rejection (temperature taken from opt); a greedy request's out_probs row is 0.
 * Workspace: spec_verify_workspace_bytes(SPEC_VERIFY_MODE_REJECTION, B, k, V).
 * SPEC_VERIFY_EINVAL also for a NULL opt, a temperature that is negative or not finite (the
 * per-request temperatures are checked on the device: a negative or NaN entry is treated as
 * sampling with that value and yields a bad-row status), or thresholds outside (0, 1].
 */
int spec_verify_rejection_ex(const void *logits, int dtype, const int32_t *draft_ids,
                             const float *draft_probs, int B, int k, int V,
                             const spec_verify_options *opt, uint64_t seed, uint64_t offset,
                             int32_t *out_tokens, int32_t *accept_len, float *out_probs,
                             void *workspace, size_t ws_bytes, int32_t *dev_status, void *stream);

/*
 * spec_verify_tree with options: a request with temperature 0 walks by argmax (mode 0), the
 * others by the target-only rule at their temperature, with the relaxed thresholds.
 * Workspace: spec_verify_workspace_bytes(SPEC_VERIFY_MODE_TREE, B, N, V).
 */
int spec_verify_tree_ex(const void *logits, int dtype, const int32_t *node_tokens,
                        const int32_t *parents, int B, int N, int V, const spec_verify_options *opt,
                        uint64_t seed, uint64_t offset, int32_t *out_tokens, int32_t *accept_index,
                        int32_t *accept_len, void *workspace, size_t ws_bytes, int32_t *dev_status,
                        void *stream);

/*
 * Adaptive verification budget: which draft slots of a batch to verify ("The speculative
 * decoding zoo", section "The finer loop: DSpark's confidence budget"; "Inference Systems
 * Frontier: new models and speculative decoding", section "Deciding how much to verify by load").
 *   conf        [B][K] float, device: the drafter's confidence of each (request, position)
 *               slot; clamped to [0, 1], NaN read as 0.  Survival of slot (r, i) = the fp32
 *               running product conf[r][0..i].
 *   num_drafts  [B] int32, device, or NULL (all K): slots at positions >= num_drafts[r] never
 *               compete.
 *   cost        [B*K + 1] double, device: cost of a step that admits b draft slots (drafting
 *               plus verifying B + b tokens), any unit.
 * Slots are ranked by survival (equal survivals: the earlier position, then the lower request);
 * budget b scores (B + sum of the b best survivals) / cost[b] (the sum in 64-bit fixed point,
 * units of 2^-49; the rate to a relative 2^-45, so budgets whose rates agree to about 2^-44 may
 * be taken in either order); the first maximal b is chosen.  Outputs (device): admitted [B] (request r verifies its first admitted[r] drafts;
 * they sum to *budget), *budget, and *best_rate (or NULL).  cost must be positive.
 * B * K <= 16384, K <= 64.  workspace: device memory, 8-byte aligned, of
 * spec_verify_plan_budget_workspace_bytes(B, K) bytes (0 for unsupported sizes; 256, reserved:
 * the planner keeps its work in shared memory), caller-owned, no initialisation needed.  One
 * launch, asynchronous on `stream`: a cluster of 8 CTAs sorts the slots' survival scores (a
 * sort per CTA, then three merge rounds across the cluster through distributed shared memory),
 * sums them in 64-bit fixed point, picks the budget (rate keys in fp32 double-float arithmetic,
 * an integer maximum) and writes the admitted prefixes.  The first call on a device raises
 * the kernel's dynamic shared-memory limit (cudaFuncSetAttribute); make it before any stream
 * capture on that device.  SPEC_VERIFY_EINVAL for bad pointers, alignment or
 * sizes; SPEC_VERIFY_EWORKSPACE for a short or misaligned workspace; SPEC_VERIFY_ECUDA for a
 * failed launch.
 */
#define SPEC_VERIFY_BUDGET_MAX_SLOTS 16384
size_t spec_verify_plan_budget_workspace_bytes(int B, int K);
int spec_verify_plan_budget(const float *conf, const int32_t *num_drafts, int B, int K,
                            const double *cost, int32_t *admitted, int32_t *budget,
                            double *best_rate, void *workspace, size_t ws_bytes, void *stream);

/*
 * After tree verification: move each request's accepted-path KV rows to contiguous positions
 * after its committed prefix, and advance the committed length ("投机解码", section
 * 与调度、KV 的交互, SGLang part: the committed length grows by the accepted count, and with
 * topk > 1 the accepted path is moved to contiguous positions; "Draft sources: draft models,
 * n-gram, suffix decoding", section "SGLang's suffix automaton, in tree", NGRAM walk-through:
 * verification, then move_accept_tokens_to_target_kvcache).  The pages give the operation, not a
 * layout; ours:
 *   kv_pool       device memory, 16-byte aligned: `planes` planes (one per layer and K or V)
 *                 plane_stride_bytes apart, each [num_slots][row_bytes] (any element type;
 *                 row_bytes a multiple of 16; plane_stride_bytes a multiple of 16 and at least
 *                 num_slots * row_bytes; ignored when planes = 1)
 *   slot_table    [B][max_pos] int32: pool slot of each position of request b
 *   committed_in  [B] int32: committed positions; the verify forward wrote tree node j's KV at
 *                 position committed_in[b] + j (j < N)
 *   committed_out [B] int32 (must not alias committed_in): committed_in + accept_len + 1, or
 *                 committed_in unchanged for a request with accept_len = -1 or a fault
 *   accept_index  [B][N], accept_len [B]: as spec_verify_tree writes them
 * For i = 1..accept_len, in order, the row at position committed + accept_index[i] is copied to
 * position committed + i in every plane (skipped where both are the same slot).  Requests must
 * not share slots.  Device status codes 5 (committed + N beyond max_pos, accept_len >= N, or a
 * path entry outside [0, N)) and 6 (a slot outside [0, num_slots)) mark requests that are left
 * unchanged.  Host codes: SPEC_VERIFY_EINVAL for bad pointers or sizes (B > 65535, N > 64,
 * max_pos < N), SPEC_VERIFY_ECUDA for a failed launch.  Asynchronous on `stream`.
 */
int spec_verify_kv_compact(void *kv_pool, int64_t num_slots, size_t row_bytes, int planes,
                           size_t plane_stride_bytes, const int32_t *slot_table, int max_pos,
                           const int32_t *committed_in, int32_t *committed_out,
                           const int32_t *accept_index, const int32_t *accept_len, int B, int N,
                           int32_t *dev_status, void *stream);

/*
 * Workspace bytes needed by one call of the given mode (SPEC_VERIFY_MODE_*) with B requests,
 * k drafts (chain) or N nodes (tree) and vocabulary V.  A pure host function; 0 on bad input.
 * The size does not depend on dtype or on the device.
 */
size_t spec_verify_workspace_bytes(int mode, int B, int k_or_N, int V);

/* Static description of a status code (host or device code); never NULL. */
const char *spec_verify_strerror(int code);

/*
 * The library's Philox4x32-10 stream, exposed so that callers and tests can reproduce the
 * uniforms: out[((slot * n_req) + req) * 4 + w] = word w of counter (slot, req, offset_lo,
 * offset_hi) under key (seed_lo, seed_hi), for slot < n_slot, req < n_req.  `out` is a device
 * array of n_slot * n_req * 4 uint32.
 */
int spec_verify_philox(uint64_t seed, uint64_t offset, int n_slot, int n_req, uint32_t *out,
                       void *stream);

/*
 * Range checks of a debug build.  Compiled with -DSV_DEBUG, every kernel checks the index of each
 * global-memory access against the extent of the array it falls in (the inputs as sized by the
 * call's arguments, the outputs, the workspace); an index out of range is skipped, not followed,
 * and the first one is recorded.  This reads and clears that record: *fault = 0 when every access
 * was in range, else bit 63 set, the check's site number in bits 48..62 and the low 48 bits of the
 * offending index.  A release build makes no checks and always reports 0.  Synchronous: it
 * copies the record from the device (after the work already enqueued on the legacy default
 * stream; synchronise other streams first).  Returns SPEC_VERIFY_OK, SPEC_VERIFY_EINVAL for a
 * NULL fault, or SPEC_VERIFY_ECUDA.  Not a part of the pages' method: a test aid that stands in
 * for a memory checker.
 */
int spec_verify_debug_fault(uint64_t *fault);

/*
 * Waits that ran out of time in the top-k / top-p threshold kernel, read and cleared.  That
 * kernel streams rows through shared memory with asynchronous bulk copies and waits on each
 * copy's completion for at most 0.2 s; a wait that runs out (a copy should land in microseconds)
 * hands that CTA's remaining rows to the general threshold kernel, so the outputs are unaffected,
 * and adds one to this count.  *count = the waits that ran out since the last read (0 in normal
 * operation).  Synchronous (symbol copies after the work already enqueued on the legacy default
 * stream).  Returns SPEC_VERIFY_OK, SPEC_VERIFY_EINVAL for a NULL count, or SPEC_VERIFY_ECUDA.
 */
int spec_verify_wait_timeouts(uint64_t *count);

/*
 * Allocation-free variant of spec_verify_rejection.  The pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory when they verify (a step running
 * under an allocator that forbids new allocations, an engine whose device memory is owned by
 * another framework, or a thread that must not take the driver's allocation lock), and so have
 * no workspace to pass.  It computes exactly what spec_verify_rejection computes, with the same
 * arguments minus the workspace, using instead a scratch array built into the library: a
 * file-scope device array of SPEC_VERIFY_NOALLOC_SCRATCH_BYTES that every GPU loading the
 * library holds until the process exits.
 *   - Calls whose spec_verify_workspace_bytes(SPEC_VERIFY_MODE_REJECTION, B, k, V) exceeds
 *     SPEC_VERIFY_NOALLOC_SCRATCH_BYTES return SPEC_VERIFY_ETOOBIG and enqueue nothing.
 *   - The first call on a device looks up the array's device address (with that device
 *     current); make that first call before any stream capture on the device.
 *   - Every call on a device shares the one array and it keeps the last call's contents; each
 *     call clears the parts that must start at zero (on `stream`, with memsets).  Calls whose
 *     work overlaps on the GPU (different streams, no ordering between them) race on the array.
 *   - No cudaMalloc, cudaFree or other allocating routine is called.
 */
#define SPEC_VERIFY_NOALLOC_SCRATCH_BYTES (4u << 20)
int spec_verify_rejection_noalloc(const void *logits, int dtype, const int32_t *draft_ids,
                                  const float *draft_probs, int B, int k, int V,
                                  float temperature, uint64_t seed, uint64_t offset,
                                  int32_t *out_tokens, int32_t *accept_len, float *out_probs,
                                  int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
