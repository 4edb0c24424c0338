/*
 * specdec.h -- C ABI of the GB300 (sm_103a) speculative-decoding verification library.
 *
 * The library implements the verification step of speculative decoding: it turns
 * the target model's logits and the drafter's distributions into accepted tokens.
 * Sources, cited by page title and section:
 *   "Speculative decoding" (zerotofrontier.app, Chapter 20, Section 20.5)      -- SD 20.5
 *   "Speculative-Decoding / Medusa" (s1mplewind.github.io)                    -- Medusa notes
 *   "Speculative Decoding: The Art of Guessing Well" (astralord.github.io)    -- Art of Guessing
 *
 * Conventions shared by every entry point
 *   - Array arguments are caller-owned DEVICE pointers to contiguous row-major arrays;
 *     the library never allocates, frees or retains them.  Sizes are element counts.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Every call is asynchronous on `stream`; the caller synchronises before reading
 *     outputs.  Work is launched only on `stream`.
 *   - The return code covers host-side validation and launch errors only:
 *       SPECDEC_OK, SPECDEC_ERR_INVALID_ARG (a null required pointer, a non-positive
 *       size, an unknown dtype, misaligned workspace), SPECDEC_ERR_UNSUPPORTED (sizes the
 *       kernels do not handle), SPECDEC_ERR_CUDA (a launch failed), SPECDEC_ERR_WORKSPACE
 *       (workspace smaller than the matching *_workspace_bytes()).  On a non-OK return
 *       nothing was launched, except for SPECDEC_ERR_CUDA.
 *   - Problems in the DATA are reported per sequence in `out_status` (bit flags below).
 *     A sequence with any error bit set gets num_accepted = -1 and all its tokens -1.
 *     Warning bits leave the outputs valid.
 *   - Temperatures below SPECDEC_GREEDY_TEMPERATURE (including 0 and negatives) select
 *     greedy verification for that sequence (SD 20.5, "A round of greedy speculative
 *     decoding"; the special case "A greedy target" of the sampling rule).
 *   - Deterministic: the same inputs give bit-identical outputs on every call.
 *   - Workspaces: a call's workspace must hold at least the size the matching
 *     *_workspace_bytes() returns and be 256-byte aligned.  Its contents need no
 *     preparation: each call clears the counters it uses on its stream first.  One
 *     workspace can serve calls of any shape that fits, one call at a time; calls that
 *     overlap on the GPU must not share a workspace.
 */
#ifndef SPECDEC_H
#define SPECDEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SPECDEC_F32 = 0, SPECDEC_BF16 = 1 } specdec_dtype;

/* return codes */
#define SPECDEC_OK 0
#define SPECDEC_ERR_INVALID_ARG 1
#define SPECDEC_ERR_UNSUPPORTED 2
#define SPECDEC_ERR_CUDA 3
#define SPECDEC_ERR_WORKSPACE 4
#define SPECDEC_ERR_TOO_LARGE 5   /* the shape needs more scratch than the built-in array */

/* per-sequence status bits (errors: low byte; warnings: above) */
#define SPECDEC_STATUS_BAD_LOGIT 1          /* NaN or +inf logit in a row the call reads      */
#define SPECDEC_STATUS_EMPTY_ROW 2          /* a row whose logits are all -inf                */
#define SPECDEC_STATUS_BAD_TOKEN 4          /* draft / node token outside [0, V)              */
#define SPECDEC_STATUS_BAD_PROB 8           /* draft probability NaN, inf or negative         */
#define SPECDEC_STATUS_BAD_UNIFORM 16       /* uniform outside [0, 1) on a sampled sequence   */
#define SPECDEC_STATUS_BAD_TREE 32          /* parent not in [-1, i), or tree deeper than D   */
#define SPECDEC_STATUS_BAD_TEMPERATURE 64   /* temperature NaN or infinite                    */
#define SPECDEC_STATUS_TIMEOUT 128          /* a bounded wait inside a kernel gave up: not finished */
#define SPECDEC_STATUS_ERROR_MASK 0xFF
#define SPECDEC_STATUS_ZERO_Q 256           /* warning: q_i(x_i) == 0; accepted iff p_i(x_i) > 0 */
#define SPECDEC_STATUS_ZERO_RESIDUAL 512    /* warning: residual mass 0 after rounding; drew from p */

#define SPECDEC_GREEDY_TEMPERATURE 1e-3f

/* ------------------------------------------------------------------------------------
 * Chain verification: one round of speculative sampling per sequence.
 *
 * SD 20.5, "A round of speculative sampling" (Leviathan et al. Alg. 1) and the exercise
 * "Verify one round of speculative sampling"; Art of Guessing, "Speculative sampling".
 * For sequence b with temperature T = temperatures[b] >= SPECDEC_GREEDY_TEMPERATURE:
 *   p_i = softmax(logits[b, i, :] / T), i = 0..g
 *   draft i is accepted iff uniforms[b, i] * q_i(x_i) < p_i(x_i)   (u < p/q, min(1, .) implicit)
 *   J = number of leading accepted drafts
 *   the extra token y is the inverse-CDF draw with u = uniforms[b, g] from
 *   (p_J - q_J)+ (normalised), where q_g == 0 so that J == g draws the bonus from p_g:
 *   y = smallest k with C_k > u * S, C the running sum and S the total of the weights.
 * Greedy sequences accept while x_i == argmax_k logits[b, i, k] (lowest index on ties)
 * and emit the argmax of row J; draft_probs and uniforms are not read for them.
 *
 * logits          [B, g+1, V]  fp32 or bf16 (ldt)          row i: target after x_0..x_{i-1}
 * draft_probs     [B, g, V]    fp32, the distribution each draft was sampled from, as given
 * draft_tokens    [B, g]       int32
 * temperatures    [B]          fp32
 * uniforms        [B, g+1]     fp32 in [0, 1): slot i tests draft i, slot g drives y
 * out_tokens      [B, g+1]     int32: x_0..x_{J-1}, y, then -1
 * out_num_accepted[B]          int32: J (or -1 on a data error)
 * out_p_draft     [B, g]       fp32, optional (NULL): p_i(x_i) for i <= J; NaN after J,
 *                              for greedy sequences and on a data error
 * out_status      [B]          int32, optional (NULL): status bits
 * Positions are evaluated left to right, as the round itself runs: row i (its logits,
 * draft token, q_i(x_i) and uniform) counts only if drafts 0..i-1 were all accepted,
 * and the first data error or rejection ends the scan.  Rows after J therefore neither
 * change the outputs nor are validated (the default kernel does not read them at all),
 * and status bits describe rows 0..J plus uniforms[b, g] and q row J where the draw
 * uses them.  A non-finite temperature is an error whatever the rows hold.
 * Sizes: B >= 1, g >= 1, V >= 1, V < 2^31.
 * Host-resident rows: logits and draft_probs may be pinned host memory (cudaHostAlloc, or
 * registered with cudaHostRegister, mapped at its own address).  The left-to-right kernel
 * then reads only the rows the round needs, straight over the host link (no copy of the
 * whole batch); this needs 16-byte aligned rows, g + 1 <= 32 and V <= 1,048,576 (bf16) or
 * 786,432 (fp32), else SPECDEC_ERR_UNSUPPORTED.  Pageable host memory gives
 * SPECDEC_ERR_INVALID_ARG, and so does a device pointer on a device other than the current
 * one.  The other inputs, the outputs and the workspace are device memory.  The same holds
 * for specdec_verify_greedy and specdec_verify_chain_varlen.
 * Bounded waits: the left-to-right kernel's waits on its queues and copies give up after a
 * bound (one second); a sequence the kernel could not finish then comes back with
 * SPECDEC_STATUS_TIMEOUT, num_accepted -1 and tokens -1 (out_p_draft NaN).  The kernel
 * does not need its whole grid resident at once: while kernels on other streams hold SMs,
 * the part that is running takes every sequence in turn, and no running part waits on one
 * that has not started, so sharing the GPU slows a call but does not time it out.
 */
size_t specdec_chain_workspace_bytes(int B, int g, int V, specdec_dtype ldt);

/* Workspace for host-resident logits: specdec_chain_workspace_bytes plus room for one
 * device copy of a logits row per sequence (B * V * element size, rounded up to 256
 * bytes).  Given a workspace at least this large, with logits in pinned host memory, the
 * left-to-right kernel also writes each row it streams for a sequence's chain into that
 * sequence's copy, and a draw from that row (the residual at a rejection, or the bonus
 * row) reads the copy from device memory instead of reading the row a second time over
 * the host link.  A smaller workspace (at least specdec_chain_workspace_bytes) gives the
 * same results and reads drawn rows from the host again.  Device-resident logits, and
 * greedy-only calls, never use the copy.  The same sizes serve
 * specdec_verify_chain_varlen.  Returns 0 for invalid sizes or dtype. */
size_t specdec_chain_host_workspace_bytes(int B, int g, int V, specdec_dtype ldt);

int specdec_verify_chain(const void* logits, specdec_dtype ldt, const float* draft_probs,
                         const int32_t* draft_tokens, const float* temperatures,
                         const float* uniforms, int B, int g, int V, int32_t* out_tokens,
                         int32_t* out_num_accepted, float* out_p_draft, int32_t* out_status,
                         void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Chain verification with a per-request number of verified drafts (SD 20.5, "Choosing how
 * much to verify at every step": adaptive verification verifies l_r drafts of request r).
 *
 * The arguments of specdec_verify_chain, padded to g drafts, plus gammas [B] int32 with
 * 0 <= gammas[b] <= g: sequence b's round is the chain round on its first gammas[b] + 1
 * rows -- drafts 0..gammas[b]-1 tested with uniforms[b, 0..gammas[b]-1], the extra token
 * from row J (a rejection's residual, or the bonus row gammas[b]) with uniforms[b,
 * gammas[b]].  Rows, q rows and uniforms past gammas[b] are not read; out_tokens are -1
 * past J, out_p_draft NaN past J.  A count outside [0, g] gives SPECDEC_STATUS_BAD_TOKEN.
 * Exactness needs each count chosen without looking at the drafts it decides on (the
 * page's non-anticipating requirement, box "Trimming a draft can break exactness"); the
 * verifier cannot check it.  Needs 16-byte aligned rows, g + 1 <= 32 and V <= 1,048,576 (bf16)
 * or 786,432 (fp32) (the left-to-right kernel), else SPECDEC_ERR_UNSUPPORTED.  Workspace:
 * specdec_chain_workspace_bytes.
 */
int specdec_verify_chain_varlen(const void* logits, specdec_dtype ldt, const float* draft_probs,
                                const int32_t* draft_tokens, const float* temperatures,
                                const float* uniforms, const int32_t* gammas, int B, int g, int V,
                                int32_t* out_tokens, int32_t* out_num_accepted, float* out_p_draft,
                                int32_t* out_status, void* workspace, size_t workspace_bytes,
                                void* stream);

/* ------------------------------------------------------------------------------------
 * Block verification: one round per sequence, the draft judged jointly.
 *
 * Art of Guessing, "Block verification" (Sun et al.).  Same inputs, outputs and shapes as
 * specdec_verify_chain.  For a sampled sequence (T >= SPECDEC_GREEDY_TEMPERATURE), with
 * p_k = softmax(logits[b, k, :] / T) and q_k = draft_probs[b, k, :]:
 *   w_0 = 1, w_{k+1} = min(1, w_k * p_k(x_k) / q_k(x_k))       (q(x) = 0: ratio +inf, or 0
 *                                                              when p(x) = 0; 0 * inf = 0)
 *   mass_k = sum_v (w_k p_k(v) - q_k(v))+ (k < g), mass_g = w_g
 *   survival_k = mass_k / (mass_k + 1 - w_k) if w_k < 1, else 1
 *   prefix length k (1..g) survives iff uniforms[b, k-1] <= survival_k
 *   n = the longest surviving prefix (0 if none): out_num_accepted[b]
 *   the extra token is the inverse-CDF draw with uniforms[b, g] from (w_n p_n - q_n)+
 *   (q_g == 0): y = smallest v with C_v > u * S.  out_tokens = x_0..x_{n-1}, y, -1...
 * Greedy sequences are verified exactly as by specdec_verify_greedy (a one-hot target
 * reduces the rule to argmax matching).  The rule reads every row, every draft, every
 * q row and every uniform, so all are validated and every error found is reported
 * (status bits OR'd); an error gives J = -1, tokens -1 and p_draft NaN.  out_p_draft[b, k]
 * = p_k(x_k) for every k of a clean sampled sequence.  Warnings: SPECDEC_STATUS_ZERO_Q
 * (some q_k(x_k) == 0), SPECDEC_STATUS_ZERO_RESIDUAL (the residual of row n summed to 0
 * after rounding; the token is drawn from p_n).
 * Layout requirement: every logits row and q row starts on a 16-byte boundary (V * elem
 * size and V * 4 multiples of 16, bases aligned) and g + 1 <= 32; other shapes return
 * SPECDEC_ERR_UNSUPPORTED.  Sizes: B >= 1, g >= 1, V >= 1.
 */
size_t specdec_block_workspace_bytes(int B, int g, int V, specdec_dtype ldt);

int specdec_verify_block(const void* logits, specdec_dtype ldt, const float* draft_probs,
                         const int32_t* draft_tokens, const float* temperatures,
                         const float* uniforms, int B, int g, int V, int32_t* out_tokens,
                         int32_t* out_num_accepted, float* out_p_draft, int32_t* out_status,
                         void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Greedy verification (SD 20.5, "A round of greedy speculative decoding"; Art of
 * Guessing, "Draft and verify"): z_i = argmax logits[b, i, :] (lowest index on ties),
 * J = longest prefix with x_i == z_i, emit x_0..x_{J-1}, z_J.  Shapes as for the chain
 * call.  Every sequence is greedy whatever its temperature would be.
 */
size_t specdec_greedy_workspace_bytes(int B, int g, int V, specdec_dtype ldt);

int specdec_verify_greedy(const void* logits, specdec_dtype ldt, const int32_t* draft_tokens,
                          int B, int g, int V, int32_t* out_tokens, int32_t* out_num_accepted,
                          int32_t* out_status, void* workspace, size_t workspace_bytes,
                          void* stream);

/* ------------------------------------------------------------------------------------
 * Medusa tree verification: a walk of a candidate tree per sequence.
 *
 * Medusa notes, section "Attention Tree": at the current node the target draws a token
 * (inverse CDF of softmax(logits / T) with uniforms[b, d] at depth d, or the argmax for a
 * greedy sequence); if a child of the node carries that token the walk appends it and
 * descends, otherwise it emits the token and stops.  SD 20.5 gives the greedy walk after
 * the exercise "The tree attention mask".  Among children carrying the same token the
 * lowest node index is taken.
 *
 * logits        [B, N+1, V]  row 0: after the committed prefix (the root); row 1+i: after node i
 * node_tokens   [B, N]       int32
 * parents       [N]          int32, shared by the batch, parents[i] in [-1, i)
 * temperatures  [B]          fp32
 * uniforms      [B, D+1]     fp32 in [0, 1), D = max_depth
 * out_tokens    [B, D+1]     int32: the accepted node tokens then the final draw, -1 padded
 * out_path      [B, D]       int32: node ids of the accepted path, -1 padded
 * out_num_accepted [B]       int32: accepted nodes (or -1 on a data error)
 * out_status    [B]          int32, optional
 * max_depth D bounds the number of nodes on any root path (SPECDEC_STATUS_BAD_TREE if a
 * path is longer).  Only the rows the walk visits are read.  N >= 0, 1 <= D <= 64.
 */
size_t specdec_tree_workspace_bytes(int B, int N, int V, int max_depth, specdec_dtype ldt);

int specdec_verify_tree(const void* logits, specdec_dtype ldt, const int32_t* node_tokens,
                        const int32_t* parents, const float* temperatures, const float* uniforms,
                        int B, int N, int V, int max_depth, int32_t* out_tokens,
                        int32_t* out_path, int32_t* out_num_accepted, int32_t* out_status,
                        void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Sampled tree verification by recursive rejection (SD 20.5, box "Recursive rejection at
 * a node with several children"; the multi-step speculative sampling of SpecInfer).
 *
 * At the current node, whose children s_1..s_k were drafted independently from q, start
 * from R_1 = p = softmax(logits / T) at the node; try the children in node-index order:
 * accept s_i when uniforms[b, 1 + s_i's node id] * q(s_i) < R_i(s_i) and move to it;
 * otherwise R_{i+1} = (R_i - q)+ normalised and try the next child.  When every child is
 * rejected (or the node is a leaf) the extra token is the inverse-CDF draw of
 * uniforms[b, 0] from the last R (smallest v with C_v > u * S) and the walk ends.  The
 * emitted tokens follow the target exactly when every node's children are independent
 * draws from that node's q.  A greedy sequence descends into the lowest-index child
 * carrying the argmax and emits the argmax where none does.
 *
 * logits        [B, N+1, V]  row 0: after the committed prefix (the root); row 1+i: after node i
 * draft_probs   [B, N+1, V]  fp32: row 0: the distribution the root's children were drafted
 *                            from; row 1+i: node i's children's (leaf rows are not read)
 * node_tokens   [B, N]       int32
 * parents       [N]          int32, shared by the batch, parents[i] in [-1, i)
 * temperatures  [B]          fp32
 * uniforms      [B, N+1]     fp32 in [0, 1): slot 1+j tests node j, slot 0 the final draw
 * out_tokens    [B, D+1]     int32: the accepted node tokens then the final draw, -1 padded
 * out_path      [B, D]       int32: node ids of the accepted path, -1 padded
 * out_num_accepted [B]       int32: accepted nodes (or -1 on a data error)
 * out_status    [B]          int32, optional: the tree, every token, T and (sampled) every
 *                            uniform are checked first; then, along the walk, each visited
 *                            row (BAD_LOGIT, EMPTY_ROW), q(s) of each tried child and a q
 *                            row read whole at its node's first rejection (BAD_PROB).  An
 *                            error reports error bits only.  Warnings: ZERO_Q (a tried
 *                            child with q(s) = 0: accepted iff R(s) > 0), ZERO_RESIDUAL
 *                            (a residual summed to 0 after rounding; R_i is kept).
 * max_depth D bounds the number of nodes on any root path.  N >= 0, 1 <= D <= 64.  No
 * workspace is needed (specdec_tree_workspace_bytes applies and returns 0).
 *
 * flags: 0, or SPECDEC_TREE_WITHOUT_REPLACEMENT -- the children of every node were drawn
 * without replacement (Sequoia, Chen et al.; SD 20.5, the paragraph after the box's
 * proof): try i uses q_i, q with the tokens of the children already rejected at the node
 * set to zero and renormalised by Z_i = 1 - (q at those tokens), in the test
 * (u * q_i(s_i) < R_i(s_i)) and in the residual (R_{i+1} = (R_i - q_i)+ normalised).
 * When Z_i <= 0 (q's mass is used up) q_i is zero: the try follows the ZERO_Q rule and a
 * rejection leaves R_i.  Children drawn without replacement carry distinct tokens, so
 * two children of one node with the same token are an input error (BAD_TREE).  Other
 * flag bits: SPECDEC_ERR_INVALID_ARG.
 */
#define SPECDEC_TREE_WITHOUT_REPLACEMENT 1
int specdec_verify_tree_recursive(const void* logits, specdec_dtype ldt, const float* draft_probs,
                                  const int32_t* node_tokens, const int32_t* parents,
                                  const float* temperatures, const float* uniforms, int B, int N, int V,
                                  int max_depth, int flags, int32_t* out_tokens, int32_t* out_path,
                                  int32_t* out_num_accepted, int32_t* out_status, void* stream);

/* ------------------------------------------------------------------------------------
 * Gumbel-coupled verification (Art of Guessing, "Gumbel coupling", Daliri et al.).
 *
 * The drafter and the target use the same noise g_k at position k: the drafter proposed
 * x_k = argmax_i (log q_k(i) + g_k,i) (specdec_gumbel_draft below), the target samples
 * t_k = argmax_i (log p_k(i) + g_k,i) with p_k = softmax(logits[b, k, :] / T); the round keeps
 * x_0..x_{n-1} for the first n with x_n != t_n (n = g if none) and appends t_n.  The emitted
 * tokens are what the target alone samples with that noise, whatever the drafter.
 *
 * Noise: Philox4x32-10 (Salmon et al., SC 2011).  Entries 4j..4j+3 of row k of sequence b
 * use the outputs of counter (j, k, b, 0) under key (seed & 0xffffffff, seed >> 32); an
 * output x gives u = ((x >> 9) + 0.5) / 2^23.  Race in log2 units, float32:
 * score_i = a_i - log2(xi_i), xi_i = -log1p(u_i - 1), a_i = logit_i * log2(e) / T (target) or
 * log2(q_i) (drafter); ties go to the lowest index.  A greedy sequence (T < 1e-3) uses the
 * plain argmax of the logits.
 *
 * logits [B, g+1, V] (bf16/fp32), draft_tokens [B, g] int32, temperatures [B] fp32.
 * out_tokens [B, g+1] int32 (-1 padded), out_num_accepted [B] int32 (n, or -1 on an error),
 * out_status [B] int32 (optional).  Rows are evaluated left to right and the round stops at
 * n: rows after n are neither read nor validated.  Errors: BAD_TEMPERATURE (non-finite T),
 * then in row order BAD_LOGIT / EMPTY_ROW (row k) and BAD_TOKEN (draft k).
 * Sizes: B >= 1, g >= 1, V >= 1, B <= 65535; 16-byte aligned rows (V * element size a
 * multiple of 16, aligned base) take 16-byte loads, others scalar loads.  Workspace:
 * specdec_gumbel_workspace_bytes(B, g) bytes, 256-byte aligned, device memory (rows are
 * evaluated in waves of two across the GPU; the workspace holds each wave's partial races
 * and which rounds are still open).
 */
size_t specdec_gumbel_workspace_bytes(int B, int g);

int specdec_verify_gumbel(const void* logits, specdec_dtype ldt, const int32_t* draft_tokens,
                          const float* temperatures, uint64_t seed, int B, int g, int V,
                          int32_t* out_tokens, int32_t* out_num_accepted, int32_t* out_status,
                          void* workspace, size_t workspace_bytes, void* stream);

/* The drafter's side of Gumbel coupling: out_draft_tokens[b, k] = argmax_i (log q[b, k, i]
 * + g_{k,i}) with the noise above (same seed, counter (j, k, b, 0)).  draft_probs [B, g, V]
 * fp32; entries that are 0 are never chosen, nor are NaN or negative ones (-1 if no entry
 * qualifies). */
int specdec_gumbel_draft(const float* draft_probs, uint64_t seed, int B, int g, int V,
                         int32_t* out_draft_tokens, void* stream);

/* The shared noise itself, for a drafter that runs its race elsewhere:
 * out_noise[(b * rows + k) * V + i] = G = -log2(xi), xi = -ln(u), of entry i at row k of
 * sequence b (the race adds it to a_i).  out_noise [B, rows, V] fp32.  The library evaluates
 * G with its own approximation (absolute error below 4e-6 against the float64 definition). */
int specdec_gumbel_noise(uint64_t seed, int B, int rows, int V, float* out_noise, void* stream);

/* ------------------------------------------------------------------------------------
 * Accepted-branch KV compaction (SD 20.5, "Keeping the caches consistent after a
 * rejection": after a tree round the accepted branch's cache entries, scattered among
 * discarded siblings, are gathered into consecutive slots; a chain only moves a length).
 *
 * Node i of sequence b's candidates sits at logical slot prefix_len[b] + i; for
 * d < num_accepted[b] the entry of node path[b, d] moves to slot prefix_len[b] + d, in place.
 * A slot is row_bytes bytes:
 *   contiguous (block_table == NULL): slot s of sequence b at cache + b * seq_stride +
 *     s * slot_stride, num_slots slots per sequence;
 *   paged: at cache + block_table[b * max_blocks + s / block_size] * block_stride +
 *     (s % block_size) * slot_stride (num_slots = max_blocks * block_size).
 * Call it once per cache tensor (per layer, keys and values, or one call for a fused
 * layout).  path [B, max_depth] int32 (the tree verifier's out_path), num_accepted [B]
 * (its out_num_accepted; a negative count leaves the sequence alone).
 * out_new_len [B] int32 (optional): prefix_len + num_accepted, the entries to keep (the
 * extra token has no entry yet).  out_status [B] (optional): SPECDEC_STATUS_BAD_TREE when
 * a path does not climb the tree (path[d] >= d, strictly increasing) or leaves the cache;
 * that sequence is left alone.  Freeing emptied pages is the allocator's business.
 * 16-byte aligned layouts move 16-byte words, others bytes.  All pointers are device
 * pointers; strides and sizes in bytes.
 */
int specdec_compact_kv(void* cache, int64_t row_bytes, int64_t slot_stride, int64_t seq_stride,
                       int64_t num_slots, const int32_t* block_table, int block_size, int max_blocks,
                       int64_t block_stride, int B, const int32_t* prefix_len, const int32_t* path,
                       int max_depth, const int32_t* num_accepted, int32_t* out_new_len,
                       int32_t* out_status, void* stream);

/* ------------------------------------------------------------------------------------
 * Tree-attention mask and position ids (SD 20.5, box "Token tree and tree attention").
 *   out_mask          [N, P+N] uint8: row i is 1 on every prefix column j < P, on column
 *                     P+i and on column P+a for every ancestor a of node i; 0 elsewhere
 *   out_position_ids  [N] int64: P + depth(i), depth = number of ancestors
 *   out_depth         [N] int32, optional
 *   out_status        [1] int32: SPECDEC_STATUS_BAD_TREE if some parents[i] is not in
 *                     [-1, i); the other outputs are then unspecified
 * N >= 1, P >= 0, (P + N) * N < 2^31.
 */
int specdec_build_tree_mask(const int32_t* parents, int N, int prefix_len, uint8_t* out_mask,
                            int64_t* out_position_ids, int32_t* out_depth, int32_t* out_status,
                            void* stream);

/* ------------------------------------------------------------------------------------
 * Kernel timing for benchmarks.  While enabled, every kernel the library launches is
 * bracketed by a pair of CUDA events recorded on the launching stream.  The state is
 * process-global and not thread-safe; enable it only around single-threaded timing.
 *   specdec_profile_start(max_launches): creates the event pool; returns SPECDEC_OK.
 *   specdec_profile_read(total_ms, launches, n): synchronises the recorded events and
 *     writes per-kernel totals for kernel ids 0..n-1 (ids: SPECDEC_KERNEL_*); resets.
 *   specdec_profile_stop(): disables timing and destroys the events.
 */
#define SPECDEC_KERNEL_CHAIN_STATS 0   /* row statistics over every logits row      */
#define SPECDEC_KERNEL_CHAIN_SAMPLE 1  /* residual / bonus masses of the drawn rows */
#define SPECDEC_KERNEL_TREE_WALK 2
#define SPECDEC_KERNEL_TREE_MASK 3
#define SPECDEC_KERNEL_CHAIN_DECIDE 4  /* accept tests and first rejection          */
#define SPECDEC_KERNEL_CHAIN_FINISH 5  /* inverse-CDF search of the drawn rows      */
#define SPECDEC_KERNEL_CHAIN_SEQ 6     /* left-to-right chain verification          */
#define SPECDEC_KERNEL_BLOCK_DECIDE 7  /* block verification: weights per prefix    */
#define SPECDEC_KERNEL_BLOCK_FINISH 8  /* block verification: survival and the draw */
#define SPECDEC_KERNEL_BLOCK_FUSED 9   /* block verification in one launch           */
#define SPECDEC_KERNEL_TREE_RR 10      /* tree verification by recursive rejection   */
#define SPECDEC_KERNEL_GUMBEL 11       /* Gumbel-coupled verification                */
#define SPECDEC_KERNEL_GUMBEL_DRAFT 12 /* the drafter's shared-noise sampler          */
#define SPECDEC_KERNEL_KV_COMPACT 13   /* accepted-branch KV compaction              */
#define SPECDEC_NUM_KERNELS 14

int specdec_profile_start(int max_launches);
int specdec_profile_read(double* total_ms, int* launches, int n);
int specdec_profile_stop(void);

/* ------------------------------------------------------------------------------------
 * Chain verification without any allocation (no counterpart in the source pages; this is
 * a deployment convenience).
 *
 * Some callers cannot allocate device memory, or must not: code running under an
 * inference server's fixed memory plan that forbids allocations after start-up, plain C
 * hosts that link only this library and receive their tensors from elsewhere, and
 * latency-critical paths where cudaMalloc/cudaFree would synchronise the device.  This
 * entry point takes the same arguments as specdec_verify_chain minus the workspace and
 * uses scratch memory built into the library instead: one array of
 * SPECDEC_NOALLOC_SCRATCH_BYTES in device memory, which every GPU that loads the library
 * holds until the process exits.  It allocates nothing and calls no allocating routine.
 *
 *   - Set-up: the first call on each device (with that device current) looks up the
 *     array's device address; make that first call before any stream capture begins.
 *     The address is kept per device and primary context: after a device reset
 *     (cudaDeviceReset) the next call looks it up again.
 *   - Limit: a shape whose specdec_chain_workspace_bytes() exceeds
 *     SPECDEC_NOALLOC_SCRATCH_BYTES is rejected with SPECDEC_ERR_TOO_LARGE (nothing is
 *     launched; specdec_last_error() gives the sizes).  16 MiB covers, e.g., B=512, g=8,
 *     V=152064 fp32.
 *   - Sharing: every call on a device uses the same array and it keeps the last call's
 *     contents; each call clears the counters it needs on its own stream first.  Calls
 *     that overlap on the GPU (different streams, or host threads) race on the array and
 *     must be serialised by the caller.
 *   - Results are the same as specdec_verify_chain's for the same inputs.
 */
#define SPECDEC_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

int specdec_verify_chain_noalloc(const void* logits, specdec_dtype ldt, const float* draft_probs,
                                 const int32_t* draft_tokens, const float* temperatures,
                                 const float* uniforms, int B, int g, int V, int32_t* out_tokens,
                                 int32_t* out_num_accepted, float* out_p_draft, int32_t* out_status,
                                 void* stream);

/* ------------------------------------------------------------------------------------
 * Test hooks (the library's own tests and sweeps; not for production use).
 *
 * Process-global settings read by the calls issued after them (not thread-safe; set them
 * while no call is being issued).  Every hook defaults to 0, the production behaviour.
 *   SPECDEC_HOOK_CHAIN_ALL_ROWS    1: chain and greedy calls whose rows the left-to-right
 *                                  kernel takes run the all-rows streaming kernels instead
 *   SPECDEC_HOOK_BLOCK_TWO_PASS    1: block verification runs the statistics and mass
 *                                  kernels instead of the one-launch kernel
 *   SPECDEC_HOOK_TREE_CLUSTER      1, 2, 4 or 8: the tree walks' cluster size (where it fits)
 *   SPECDEC_HOOK_CHAIN_DROP_DRAWS  1: the left-to-right kernel never marks a queued draw
 *                                  as published, so the teams that take its ticket wait
 *                                  until the queue wait gives up (the sequences it belongs
 *                                  to come back with SPECDEC_STATUS_TIMEOUT)
 *   SPECDEC_HOOK_QUEUE_WAIT_US     >= 1: the left-to-right kernel's bound on waits for
 *                                  queued work, in microseconds (0: one second)
 * Returns SPECDEC_OK, or SPECDEC_ERR_INVALID_ARG for an unknown hook or value.
 */
#define SPECDEC_HOOK_CHAIN_ALL_ROWS 0
#define SPECDEC_HOOK_BLOCK_TWO_PASS 1
#define SPECDEC_HOOK_TREE_CLUSTER 2
#define SPECDEC_HOOK_CHAIN_DROP_DRAWS 3
#define SPECDEC_HOOK_QUEUE_WAIT_US 4
#define SPECDEC_NUM_HOOKS 5

int specdec_set_test_hook(int hook, int value);
int specdec_get_test_hook(int hook);

/* Library version string, e.g. "0.1.0". */
const char* specdec_version(void);

/* Description of the last SPECDEC_ERR_CUDA returned on the calling host thread: the step
 * that failed and the CUDA error.  The string stays valid until the thread's next call. */
const char* specdec_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECDEC_H */
