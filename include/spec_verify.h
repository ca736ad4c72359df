/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) batched speculative-decoding verifier.
 *
 * The operation (accept-or-resample verification of drafted tokens) is the one defined on these
 * pages, cited by page title and section:
 *   [R] "Speculative decoding", rayaq.ca ml-models -- Mechanics, One round, steps 2-5 (accept left to
 *       right while u < min(1, p(x)/q(x)); replacement from max(0, p - q) / sum max(0, p - q) at the
 *       first rejection; bonus token from p at position gamma + 1 when every draft survives);
 *       Why the output is exactly the target's (alpha = sum_x min(p, q); the same temperature on p and
 *       q); The greedy case (argmax-prefix match, argmax correction and bonus); Implementation (p and q
 *       rows are softmax(logits / temp)).
 *   [B] "Inference: distillation and speculative decoding", brunomaga.github.io -- Draft-model
 *       speculative decoding (the greedy and the sampled acceptance rules; batched rows accept
 *       different counts, so lengths are tracked per row).
 *   [C] "Speculative decoding", cgnarendiran.github.io blog -- The correction that makes it exact.
 * Throughout, p is the TARGET distribution and q the DRAFT distribution (page [B] swaps the names).
 *
 * Shapes: B rows, G = gamma_max padded draft width, V vocabulary, s = element size of the logits.
 * Row b verifies gamma_b = draft_len[b] drafted tokens (0 <= gamma_b <= G). All tensors are dense,
 * row-major, contiguous.
 *
 * Sampling rule used for the library draws of the pages: inverse CDF in vocabulary-index order with
 * a strict '>' against u times the running total; tokens with zero weight are never chosen; if
 * rounding leaves no prefix above the threshold, the last token with positive weight is taken. A
 * rejection whose residual has zero total mass (possible only through rounding) draws from that
 * position's p with the residual uniform instead.
 *
 * Uniforms: u[b, i] (i < gamma_b) drives the accept test at position i, u[b, G] the residual draw,
 * u[b, G + 1] the bonus draw. Greedy rows (temperature exactly 0) read no uniforms and no draft
 * logits.
 *
 * Ownership: every pointer is caller-owned CUDA device memory (or host memory the device can address
 * directly). The library allocates nothing and holds no per-call state; all per-call scratch lives
 * in the caller's workspace.
 *
 * Asynchrony: calls validate their arguments on the host, enqueue work on `cuda_stream` (NULL = the
 * legacy default stream) and return. Outputs are valid once that stream has been synchronised.
 *
 * Row limits: rows whose byte length V * s is a multiple of 16, with 16-byte aligned logit bases,
 * run on the streaming kernel: bf16 V <= 1048576, fp32 V <= 311296. Any other V or alignment runs
 * on the element kernel: V <= 262144. Larger V returns SV_ERR_BAD_SHAPE.
 *
 * Errors: argument errors return a nonzero sv_status synchronously and enqueue nothing. Launch
 * errors return SV_ERR_CUDA. Data errors never trap: they mark the row (out_num_emitted[b] = -1,
 * out_tokens[b, :] = -1, out_alpha/p/q[b, :] = 0). Row data errors are: draft_len outside [0, G];
 * temperature NaN, negative, infinite or in (0, FLT_MIN); a drafted token outside [0, V) at
 * i < gamma_b; for sampled rows a used uniform outside [0, 1); a read logit row holding NaN or +inf,
 * or holding only -inf.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_NULL_POINTER = 1,        /* a required pointer is NULL                                   */
  SV_ERR_BAD_SHAPE = 2,           /* B < 1, gamma_max outside [0, SV_MAX_GAMMA], V < 1, V beyond
                                     the row limits below, or the launch grid overflows            */
  SV_ERR_BAD_DTYPE = 3,           /* dtype is not an sv_dtype                                     */
  SV_ERR_WORKSPACE_TOO_SMALL = 4, /* workspace_bytes < spec_verify_workspace_size(...), or NULL   */
  SV_ERR_MISALIGNED = 5,          /* a pointer is not aligned to its element type (workspace: 16 B) */
  SV_ERR_CUDA = 6,                /* a CUDA runtime call failed (device query or launch)          */
  SV_ERR_UNSUPPORTED_DEVICE = 7,  /* the current device is not compute capability 10.3           */
  SV_ERR_SCRATCH_TOO_SMALL = 8    /* spec_verify_noalloc: the sizes need more scratch than
                                     SV_NOALLOC_SCRATCH_BYTES                                     */
} sv_status;

typedef enum { SV_DTYPE_F32 = 0, SV_DTYPE_BF16 = 1 } sv_dtype;

#define SV_MAX_GAMMA 64
#define SV_VERSION 1
/* Size of the library's static device scratch used by spec_verify_noalloc (1 MiB per device). */
#define SV_NOALLOC_SCRATCH_BYTES (1u << 20)

/* Bytes of device workspace the verification calls need for these sizes (per-position records, one
 * arrival counter per row, a status word, then B * (2 * gamma_max + 1) fp32 row thresholds and a
 * row counter that only spec_verify_filtered uses), a multiple of 256. Returns 0 for invalid sizes.
 * The thresholds and the counter fill the last round_up(4 * (B * (2 * gamma_max + 1) + 1), 256)
 * bytes.
 *
 * The workspace must hold zeros before its first use (e.g. one cudaMemset after allocation). Every
 * call that runs to completion leaves it zeroed again, so it can be reused without clearing, also
 * by calls of other sizes. One workspace serves one call at a time: two calls in flight on the same
 * workspace race. */
size_t spec_verify_workspace_size(int32_t B, int32_t gamma_max, int32_t V, int32_t dtype);

/* Batched verification of one speculative round ([R] One round, steps 3-5; [R] The greedy case).
 *
 * target_logits   [B, G+1, V] dtype   target logits; row (b, i) gives p_{b,i} = softmax(z / T_b).
 *                                     Rows i > gamma_b are never read.
 * draft_logits    [B, G, V]   dtype   draft logits; q_{b,i} = softmax(z / T_b). Rows i >= gamma_b and
 *                                     all rows of greedy rows are never read. May be NULL if G == 0.
 * draft_tokens    [B, G]      int32   drafted tokens x_{b,i}; entries i >= gamma_b are ignored.
 * draft_len       [B]         int32   gamma_b in [0, G]; NULL means every row has gamma_b = G.
 * temperature     [B]         fp32    T_b; 0 selects greedy verification, > 0 sampled verification.
 * uniforms        [B, G+2]    fp32    caller-drawn uniforms in [0, 1) (layout above).
 * out_tokens      [B, G+1]    int32   emitted tokens: gamma accepted drafts, then the correction or
 *                                     bonus token, then -1 padding.
 * out_num_emitted [B]         int32   k_b + 1 in [1, gamma_b + 1]; -1 marks a row data error.
 * out_alpha       [B, G]      fp32    alpha_{b,i} = sum_v min(p_{b,i}(v), q_{b,i}(v)) for i < gamma_b
 *                                     (every verified position, also after the first rejection;
 *                                     greedy rows: 1 if x_i is the target argmax, else 0); 0 for
 *                                     i >= gamma_b. May be NULL.
 * B, gamma_max, V, dtype              sizes and the sv_dtype of both logit tensors.
 * workspace, workspace_bytes          zero-initialised device scratch of at least
 *                                     spec_verify_workspace_size(B, gamma_max, V, dtype) bytes,
 *                                     16-byte aligned.
 * cuda_stream                         a cudaStream_t, or NULL.
 * Returns an sv_status. */
int spec_verify(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                const int32_t* draft_len, const float* temperature, const float* uniforms,
                int32_t* out_tokens, int32_t* out_num_emitted, float* out_alpha,
                int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                void* workspace, size_t workspace_bytes, void* cuda_stream);

/* spec_verify with two more outputs, for probability-level checks:
 * out_p_draft [B, G] fp32  p_{b,i}(x_{b,i}) (greedy rows: 1 if x_i is the target argmax, else 0);
 * out_q_draft [B, G] fp32  q_{b,i}(x_{b,i}) (greedy rows: 1); both 0 for i >= gamma_b.
 * Either may be NULL. Everything else is as in spec_verify. */
int spec_verify_ex(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                   const int32_t* draft_len, const float* temperature, const float* uniforms,
                   int32_t* out_tokens, int32_t* out_num_emitted, float* out_alpha,
                   float* out_p_draft, float* out_q_draft,
                   int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                   void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Verification of one-hot drafts: the drafter decoded greedily, so its distribution at position i is
 * q_i = [v == x_i] and no draft logits exist. [B] "Inference: distillation and speculative decoding",
 * brunomaga.github.io -- Draft-model speculative decoding (a greedy draft is the one-hot case: the
 * target keeps it with probability p(x) and on a rejection draws from p without x); [R] One round,
 * steps 3-5 with that q. Per sampled position i < gamma_b:
 *   keep x_i while u[b,i] < p_i(x_i); alpha_i = sum_v min(p_i(v), q_i(v)) = p_i(x_i);
 *   at the first rejection the replacement is drawn with u[b,G] from max(0, p - q), i.e. p with x
 *   left out (inverse CDF in index order, strict '>' against u times its mass); a bonus token as in
 *   spec_verify. Greedy rows (temperature 0) are verified exactly as in spec_verify.
 * Arguments, layout, ownership, workspace and errors as in spec_verify_ex without draft_logits;
 * out_q_draft receives 1 for every verified position. Only rows of 16-byte multiples with a 16-byte
 * aligned target_logits are supported: other V return SV_ERR_BAD_SHAPE, a misaligned pointer
 * SV_ERR_MISALIGNED. Only the target rows 0..gamma_b of each row are read. */
int spec_verify_onehot(const void* target_logits, const int32_t* draft_tokens,
                       const int32_t* draft_len, const float* temperature, const float* uniforms,
                       int32_t* out_tokens, int32_t* out_num_emitted, float* out_alpha,
                       float* out_p_draft, float* out_q_draft,
                       int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                       void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Greedy verification of a tree of candidates (Medusa-style drafts): [B] "Inference: distillation
 * and speculative decoding", brunomaga.github.io -- Medusa (candidate continuations form a tree that
 * the target verifies in one pass with tree attention; the longest accepted path is kept).
 * Row b holds tree_size[b] nodes; node 0 is the root, the target's own next token, always kept.
 * A node j > 0 is accepted when its parent is accepted and tree_tokens[b,j] equals the target's
 * argmax at the parent (lowest index on ties). The path kept is the longest accepted one (the
 * lowest node index among the deepest), and the target's argmax at its last node is the next token.
 *
 * target_logits  [B, N, V] dtype   the target's logits at every node (rows j >= tree_size never read)
 * tree_tokens    [B, N]    int32   token of each node
 * tree_parents   [B, N]    int32   parent of each node: -1 at the root, 0 <= parent < j otherwise
 * tree_size      [B]       int32   nodes per row in [1, N]; NULL means N
 * out_path       [B, N]    int32   node indices of the kept path, root first, then -1
 * out_path_len   [B]       int32   nodes on the kept path (>= 1); -1 marks a row error
 * out_tokens     [B, N+1]  int32   tokens of the path's nodes, then the next token, then -1
 * out_pred       [B, N]    int32   the target's argmax at every node, -1 beyond tree_size (may be NULL)
 * B, N, V, dtype                   1 <= N <= SV_MAX_GAMMA + 1; dtype as in spec_verify
 * workspace                        as in spec_verify, sized spec_verify_workspace_size(B, N - 1, V,
 *                                  dtype)
 * Row errors (the row's outputs all -1): tree_size outside [1, N]; tree_parents[b,0] != -1 or a parent
 * outside [0, j); a node token outside [0, V); a node's logit row with NaN or +inf, or only -inf.
 * Only rows of 16-byte multiples with a 16-byte aligned target_logits are supported (other V:
 * SV_ERR_BAD_SHAPE; a misaligned base: SV_ERR_MISALIGNED). Other argument errors as in spec_verify. */
int spec_verify_tree_greedy(const void* target_logits, const int32_t* tree_tokens,
                            const int32_t* tree_parents, const int32_t* tree_size,
                            int32_t* out_path, int32_t* out_path_len, int32_t* out_tokens,
                            int32_t* out_pred, int32_t B, int32_t N, int32_t V, int32_t dtype,
                            void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Verification of filtered distributions: per-row top-k and top-p applied to p and q before the
 * test. [R] "Speculative decoding", rayaq.ca ml-models -- Why the output is exactly the target's
 * (temperature, top-p and any penalties are applied to p and q before the test; the rule then
 * preserves exactly the distribution it is given). For a sampled row, p_i and q_i are replaced by
 * filter(softmax(z / T)) with, in order:
 *   top-k (0 < top_k[b] < V): keep the tokens whose logit is at least the top_k-th largest logit
 *         (ties at the boundary all kept);
 *   top-p (top_p[b] < 1): on the renormalised top-k distribution, keep a token when the mass of
 *         the tokens with a strictly larger logit is below top_p[b] (tokens with equal logits go
 *         together; the largest logit is always kept);
 *   renormalise the kept probabilities.
 * Then the rule of spec_verify on the filtered p~, q~: keep x_i while u[b,i] < min(1, p~(x)/q~(x))
 * (where q~(x) = 0 the ratio is 1 if p~(x) > 0, else 0); at the first rejection draw from
 * max(0, p~ - q~) (from p~ when that has no mass) with u[b,G]; after gamma_b accepts draw the bonus
 * from the filtered target p~ with u[b,G+1]; alpha_i = sum_v min(p~, q~); out_p_draft /
 * out_q_draft are p~(x) and q~(x).
 * Greedy rows are verified as in spec_verify (filtering keeps the argmax).
 *
 * top_k  [B] int32  per-row k; <= 0 or >= V turns top-k off. NULL: off for every row.
 * top_p  [B] fp32   per-row nucleus mass; >= 1 turns top-p off; a sampled row with top_p NaN or
 *                   <= 0 is a row error (outputs -1 / 0). NULL: off for every row.
 * Both filters keep an upper set of the row's logits, so one threshold per row describes them: the
 * call enqueues on `cuda_stream` the threshold kernel of spec_verify_filter_thresholds (into the
 * workspace), with a workspace of spec_verify_filtered_workspace_size bytes the list kernel (below),
 * the streaming kernel of spec_verify_ex reading every logit below its row's threshold as -inf (it
 * skips the rows the list kernel verified), and a memset that clears the workspace's filter area.
 * Everything else (arguments, layout, ownership, workspace, errors) as in spec_verify_ex. Only rows
 * of 16-byte multiples are supported (else SV_ERR_BAD_SHAPE), with 16-byte aligned logit bases
 * (else SV_ERR_MISALIGNED), within the streaming kernel's row limits (bf16 V <= 1048576, fp32
 * V <= 311296; else SV_ERR_BAD_SHAPE). */
int spec_verify_filtered(const void* target_logits, const void* draft_logits,
                         const int32_t* draft_tokens, const int32_t* draft_len,
                         const float* temperature, const int32_t* top_k, const float* top_p,
                         const float* uniforms, int32_t* out_tokens, int32_t* out_num_emitted,
                         float* out_alpha, float* out_p_draft, float* out_q_draft,
                         int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                         void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Workspace bytes with which spec_verify_filtered also verifies from kept lists (0 for invalid
 * sizes): spec_verify_workspace_size(...) plus, per logit row, a count and 128 (index, logit)
 * entries, plus a flag per batch row (about 1 KB per logit row). With a workspace this large, a
 * sampled batch row with top-k on whose logit rows each keep at most 128 logits is verified from
 * those lists (the threshold kernel writes them; a list kernel runs the rule on them) instead of by
 * the streaming kernel; the outputs follow the same rule. A smaller workspace (at least
 * spec_verify_workspace_size) runs every row on the streaming kernel. Every call leaves the whole
 * workspace zeroed. */
size_t spec_verify_filtered_workspace_size(int32_t B, int32_t gamma_max, int32_t V, int32_t dtype);

/* The per-row thresholds of top-k / top-p filtering that spec_verify_filtered applies: for every
 * logit row the rule reads in a sampled batch row whose top_k or top_p is on, the smallest logit
 * the filters keep (defined as in spec_verify_filtered: the kept set is exactly the logits >= the
 * threshold); -inf for every other row (greedy rows, rows not read, rows whose filters are off, and
 * rows spec_verify_filtered reports as row errors: a bad draft_len, temperature or top_p, or a
 * logit row holding NaN or +inf, or only -inf). [R] "Speculative decoding", rayaq.ca ml-models --
 * Why the output is exactly the target's.
 *
 * target_logits, draft_logits, draft_len, temperature, top_k, top_p, B, gamma_max, V, dtype
 *                  as in spec_verify_filtered (device pointers; draft_len may be NULL).
 * out_thresholds   [B * (2 * gamma_max + 1)] fp32, device: target rows (b, i), i = 0..G, at
 *                  b * (G + 1) + i, then draft rows (b, i), i = 0..G-1, at B * (G + 1) + b * G + i.
 * One CTA per row at a time (a persistent grid), one launch on cuda_stream; nothing else is
 * written. Errors as in spec_verify_filtered (argument errors enqueue nothing). A top-p decision
 * within about 1e-6 of the nucleus boundary is taken with fp32 exponentials and 42-bit fixed-point
 * masses, not in exact arithmetic. */
int spec_verify_filter_thresholds(const void* target_logits, const void* draft_logits,
                                  const int32_t* draft_len, const float* temperature,
                                  const int32_t* top_k, const float* top_p, float* out_thresholds,
                                  int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                                  void* cuda_stream);

/* KV-cache rollback after a verified round, batched over ragged rows. [R] "Speculative decoding",
 * rayaq.ca ml-models -- Verification attention and the cache: the target's cache held n entries
 * before the round and n + gamma + 1 after verification; with k drafts accepted the first n + k + 1
 * are kept (the prefix, the last token, the accepted drafts) and the rest is dropped; the drafter's
 * cache is rolled back the same way ([B] Draft-model speculative decoding: the drafter keeps the
 * part of its cache that is still valid, which is one entry short on a full accept).
 *
 * prefix_len       [B] int32  n_b, target cache entries before the round
 * draft_len        [B] int32  gamma_b (NULL: gamma_max); clamped to [0, gamma_max]
 * out_num_emitted  [B] int32  k_b + 1 from spec_verify; -1 (a row error) commits nothing
 * drafter_len_in   [B] int32  the drafter cache's entries now (NULL: taken as n_b + k_b + 1)
 * target_len_out   [B] int32  n_b + k_b + 1 (n_b after a row error)
 * drafter_len_out  [B] int32  min(drafter_len_in, target_len_out) (may be NULL)
 * cache            optional contiguous target cache, row b at cache + b * cache_row_stride bytes,
 *                  cache_entries entries of entry_bytes each; when not NULL the dropped entries
 *                  [target_len_out, n_b + gamma_b + 1) of each row (clamped to cache_entries) are
 *                  set to zero bytes. entry_bytes and cache_row_stride multiples of 16, cache 16-byte
 *                  aligned (else SV_ERR_MISALIGNED); cache_row_stride >= entry_bytes * cache_entries.
 * All pointers are device pointers owned by the caller; one launch on cuda_stream; argument errors
 * return a status and launch nothing. */
int spec_verify_kv_rollback(const int32_t* prefix_len, const int32_t* draft_len,
                            const int32_t* out_num_emitted, const int32_t* drafter_len_in,
                            int32_t* target_len_out, int32_t* drafter_len_out, void* cache,
                            int64_t cache_row_stride, int32_t entry_bytes, int32_t cache_entries,
                            int32_t B, int32_t gamma_max, void* cuda_stream);

/* spec_verify_ex for callers that cannot allocate device memory. The pages have no counterpart:
 * this is a deployment convenience, not part of the method.
 *
 * Who needs it: engines whose device memory is fully planned at start-up and that forbid any
 * allocation on the serving path, host code that cannot afford the device-wide synchronisation of
 * cudaMalloc, and plugin interfaces that hand over only the input and output buffers. They pass the
 * same inputs and outputs as spec_verify_ex (the caller still owns those) but no workspace: the
 * kernels' scratch lives in a static device array of SV_NOALLOC_SCRATCH_BYTES inside the library,
 * which every GPU that loads the library holds until the process exits. The call allocates nothing
 * and frees nothing.
 *
 * Limit: sizes whose spec_verify_workspace_size(B, gamma_max, V, dtype) exceeds
 * SV_NOALLOC_SCRATCH_BYTES are rejected with SV_ERR_SCRATCH_TOO_SMALL before anything is enqueued.
 * Every other argument is checked as spec_verify_ex checks it, also before anything is enqueued,
 * and a rejected call returns the status spec_verify_ex would return.
 * Set-up: the first call on a device looks up the array's device address (cudaGetSymbolAddress)
 * with the current device, which must be the device of the buffers; make that first call before
 * any stream capture. Each call then clears the part of the array it uses (records, row counters
 * and status word: spec_verify_workspace_size bytes) on `cuda_stream` before its launch, so a
 * call never sees what an earlier one left. Every call shares the one array: calls whose
 * executions overlap on the GPU (other streams, other host threads) race and must be serialised
 * by the caller. Arguments, layout and errors otherwise as in spec_verify_ex. */
int spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                        const int32_t* draft_tokens, const int32_t* draft_len,
                        const float* temperature, const float* uniforms, int32_t* out_tokens,
                        int32_t* out_num_emitted, float* out_alpha, float* out_p_draft,
                        float* out_q_draft, int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                        void* cuda_stream);

/* spec_verify_ex from host buffers, copying in only what the rule reads. The pages have no
 * counterpart: this is the host side of a serving step whose logits sit in host memory.
 *
 * The rule reads target rows 0..gamma_b of row b and, for a sampled row (temperature not exactly
 * 0), draft rows 0..gamma_b - 1 ([R] "Speculative decoding", rayaq.ca ml-models -- Mechanics, One
 * round, steps 3-5; The greedy case: a greedy row compares with the target's argmax only). The
 * call enqueues on `cuda_stream` the host-to-device copies of draft_tokens, draft_len, temperature
 * and uniforms. The batch rows then go in up to four groups of at least 64 rows: the logit rows a
 * group's rule reads cross the host link on an internal stream of the library (one per device,
 * created on first use): a gather kernel reading page-locked, mapped host memory directly, else
 * one copy per run of contiguous rows (runs of consecutive rows b merge when row b has gamma_b =
 * gamma_max). After a group's rows (an event orders it) spec_verify_ex verifies that group on
 * `cuda_stream` while the next group's rows cross; p and q of the drafts are not returned. Last,
 * device-to-host copies of out_tokens, out_num_emitted and out_alpha on `cuda_stream`. Everything
 * the call enqueues is complete once `cuda_stream` is. Padding rows are never copied, and never
 * read by the kernels.
 *
 * h_*: host buffers in the layouts of spec_verify_ex (h_draft_len may be NULL = all gamma_max;
 * h_out_alpha may be NULL; with gamma_max = 0, h_draft_logits and h_draft_tokens may be NULL). The call reads h_draft_len and
 * h_temperature on the host before it returns; every h_* buffer must stay unchanged (inputs) and
 * untouched (outputs) until `cuda_stream` has been synchronised. Page-locked host memory makes the
 * copies asynchronous; pageable memory also works, at the copy speed of the driver's staging.
 * A row whose host draft_len lies outside [0, gamma_max] has no logits copied; the kernel marks
 * it as a row error from the staged copy of draft_len.
 * staging: caller-owned device memory of at least spec_verify_staging_size(B, gamma_max, V, dtype)
 * bytes, 256-byte aligned; it holds the staged inputs and outputs (its contents need no setup).
 * workspace: as in spec_verify_ex. h2d_bytes (may be NULL): set to the host-to-device bytes
 * enqueued. Errors: this call's own checks (dtype, sizes, NULL pointers, a staging buffer that is
 * not 256-byte aligned or too short, a workspace too short) return a status and enqueue nothing.
 * A status returned by the verification step (the checks of spec_verify_ex that concern the device
 * and the kernels' limits) or SV_ERR_CUDA from a failed copy comes after the input copies were
 * enqueued; the work enqueued before it may still run. */
size_t spec_verify_staging_size(int32_t B, int32_t gamma_max, int32_t V, int32_t dtype);
int spec_verify_staged(const void* h_target_logits, const void* h_draft_logits,
                       const int32_t* h_draft_tokens, const int32_t* h_draft_len,
                       const float* h_temperature, const float* h_uniforms,
                       int32_t* h_out_tokens, int32_t* h_out_num_emitted, float* h_out_alpha,
                       int32_t B, int32_t gamma_max, int32_t V, int32_t dtype, void* staging,
                       size_t staging_bytes, void* workspace, size_t workspace_bytes,
                       size_t* h2d_bytes, void* cuda_stream);
/* The host-to-device bytes spec_verify_staged enqueues for these host draft lengths and
 * temperatures (host arrays; h_draft_len may be NULL); 0 for invalid sizes. Host code only. */
size_t spec_verify_staged_h2d_bytes(const int32_t* h_draft_len, const float* h_temperature,
                                    int32_t B, int32_t gamma_max, int32_t V, int32_t dtype);

/* Reads the workspace's sticky status word into *status_out after synchronising `cuda_stream`
 * (B and gamma_max as in the call that used the workspace). 0 means every call so far completed
 * its protocol. A nonzero value means a kernel-internal wait gave up (every wait inside the
 * kernels is bounded; on a healthy device none gives up): that call stopped early and the rows it
 * had not finished keep stale outputs. The word stays set until the caller clears the workspace. */
int spec_verify_workspace_status(const void* workspace, int32_t B, int32_t gamma_max,
                                 int32_t* status_out, void* cuda_stream);

/* Static description of an sv_status value (never NULL). */
const char* spec_verify_status_string(int status);

/* SV_VERSION of the built library. */
int spec_verify_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
