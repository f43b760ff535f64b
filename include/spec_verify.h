/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-decoding
 * verify-and-sample library (libspecverify.so).
 *
 * One call verifies a batch of B sequences after the target model's single
 * parallel forward over gamma+1 positions.  For every sequence b it
 *
 *   1. turns the target logits rows 1..gamma_b+1 and the draft logits rows
 *      1..gamma_b into the distributions actually sampled from, p and q, by
 *      temperature, then top-k, then top-p (each side with its own
 *      parameters)                               [wrblog §2.3, §7.2, §7.3];
 *   2. accepts draft token d_i with probability a_i = min(1, p_i(d_i)/q_i(d_i)),
 *      left to right, stopping at the first rejection  [wrblog §4.1, §6];
 *   3. draws the replacement from the residual (p_j - q_j)+ / Z at the
 *      rejected position j, or a bonus token from p_{gamma_b+1} when every
 *      draft was accepted                   [wrblog §5, §6; rainlin §1-§2];
 *
 * and, in greedy mode, emits the longest argmax-matching prefix plus the
 * target's argmax at the first mismatch (or the bonus position)
 *                                           [wrblog §7.1; baisen §2, §6].
 * Beyond that: lenient acceptance [magicnet §8], an end-of-sequence commit
 * and per-sequence sampling rules [wrblog §14.3, §15], early-exit greedy and
 * sampling verification [wrblog §6], and greedy verification of draft trees [baisen §8;
 * magicnet §7].
 *
 * Readings of points the sources leave open (the library and its tests use
 * exactly these):
 *   - transform order: temperature; top-k on the logits; renormalise; top-p
 *     on the renormalised probabilities; renormalise.
 *   - every ordering is (value descending, token index ascending): argmax and
 *     top-k ties go to the lower token index.  -0.0 equals +0.0.
 *   - top-p keeps the shortest prefix of that order whose cumulative
 *     probability reaches top_p (the crossing token is kept).
 *   - accept iff u < a (strict); uniforms lie in [0, 1).
 *   - a uniform u selects the smallest token x, in vocabulary order, whose
 *     cumulative weight C(x) exceeds u * Z.
 *   - q(d) == 0 gives a = 1 if p(d) > 0 else 0 and sets SPEC_SEQ_FLAG_ZERO_Q.
 *   - Z == 0 after a rejection (rounding only) draws from p_j instead and
 *     sets SPEC_SEQ_FLAG_Z_ZERO.
 *   - a NaN or +inf logit, or a row of only -inf, in any row a sequence uses
 *     fails that sequence: nothing is committed [wrblog §15].  -inf marks a
 *     banned token [wrblog §2.3].
 *
 * Sources cited above:
 *   [wrblog]  "推测解码：草稿模型、接受率、正确性与加速边界" (wrblog.cn)
 *   [rainlin] "投机解码" (rainlin-net.pages.dev, llm-inference/speculative-decoding)
 *   [baisen]  "投机采样 / 投机解码（Speculative Decoding）" (baisen.site)
 *   [magicnet] "投机解码到底能加速多少：把接受率、草稿成本与墙钟收益算清楚"
 *             (magicnetworld.com)
 *   [baisen]'s §8 and [magicnet]'s §7 describe draft trees verified in one forward.
 *
 * Conventions common to every entry point
 * ----------------------------------------
 * - Pointers named *_logits, draft_tokens, gamma_per_seq, draft_is_onehot,
 *   u_*, workspace and out_* are DEVICE pointers (cudaMalloc / torch CUDA
 *   tensors on the current device).  Sizes are host integers.
 * - The caller allocates and owns every buffer, including the workspace.  The
 *   library allocates nothing, keeps no state between calls and never
 *   synchronises: all work is enqueued on `stream` (a cudaStream_t; NULL is
 *   the legacy default stream) and the call returns immediately.  Two
 *   exceptions keep state: spec_verify_sample_noalloc (at the end of this
 *   header), whose scratch is a fixed array of the library's own device
 *   memory that keeps its contents between calls, shared by every call
 *   (overlapping calls race), plus a per-device cache of that array's address;
 *   and the process-wide switch of spec_set_early_logits_reads (below).
 * - Launch order.  The verifiers are launched as programmatic dependents of
 *   the previous kernel in the stream and wait for it to complete
 *   (griddepcontrol.wait) before they read or write anything -- results and
 *   ordering are those of plain stream order.  spec_set_early_logits_reads
 *   lets some of them read their logits before that wait (see there).
 * - Logits are row-major.  Element (b, i, x) of target_logits is at
 *   ((b * (gamma_max + 1) + i) * vocab + x); of draft_logits at
 *   ((b * gamma_max + i) * vocab + x).  Rows with i > gamma_b (target) or
 *   i >= gamma_b (draft) are never read.
 * - Full bandwidth needs vocab * sizeof(element) to be a multiple of 16 and
 *   16-byte aligned logits pointers; other layouts are accepted and run a
 *   slower element-wise load path.
 * - Host-checkable errors (NULL where a buffer is required, sizes out of
 *   range, temperature <= 0 or non-finite, top_p outside (0, 1], top_k < 0,
 *   element-misaligned pointers, a workspace that is too small or not
 *   256-byte aligned) return a non-zero spec_status_t and launch nothing.
 *   A failed launch returns SPEC_ERR_CUDA.  Data errors are reported per
 *   sequence through out_status / out_num_accepted (see SPEC_SEQ_*).  The
 *   library never traps the GPU.
 * - Calls that share a workspace must not overlap on the GPU.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SPEC_API __attribute__((visibility("default")))
#else
#define SPEC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1,   /* a NULL, size or parameter the contract excludes  */
    SPEC_ERR_UNSUPPORTED = 2,   /* a valid request this build does not handle       */
    SPEC_ERR_MISALIGNED = 3,    /* a pointer not aligned to its element / 256 bytes  */
    SPEC_ERR_WORKSPACE = 4,     /* workspace smaller than the *_workspace_size query */
    SPEC_ERR_CUDA = 5           /* the CUDA runtime reported an error at launch      */
} spec_status_t;

/* Per-sequence status written to out_status[b] (low byte: error code; high
 * bits: informational flags).  Any non-zero error code sets
 * out_num_accepted[b] = -1 and out_tokens[b][*] = -1: commit nothing. */
enum {
    SPEC_SEQ_OK = 0,
    SPEC_SEQ_BAD_LENGTH = 1,      /* gamma_per_seq[b] outside [0, gamma_max]          */
    SPEC_SEQ_BAD_TOKEN = 2,       /* a draft token d_i (i < gamma_b) outside [0, V)   */
    SPEC_SEQ_BAD_UNIFORM = 3,     /* a used uniform outside [0, 1) or NaN             */
    SPEC_SEQ_NONFINITE = 4,       /* NaN or +inf logit in a row the sequence uses     */
    SPEC_SEQ_EMPTY_SUPPORT = 5,   /* a used row whose logits are all -inf             */
    SPEC_SEQ_BAD_PARAMS = 6,      /* spec_verify_sample_ex: a per-sequence sampling
                                     rule the sequence uses is outside its domain     */
    SPEC_SEQ_BAD_TREE = 7,        /* spec_verify_greedy_tree: a node whose parent is
                                     not an earlier node                              */
    SPEC_SEQ_STALLED = 8,         /* a full-row draw's copies into shared memory did
                                     not arrive within its bounded wait (about a
                                     second): a device fault, not a data error       */
    SPEC_SEQ_ERROR_MASK = 0xFF,
    SPEC_SEQ_FLAG_ZERO_Q = 0x100, /* an evaluated draft token had q(d) == 0           */
    SPEC_SEQ_FLAG_Z_ZERO = 0x200, /* residual mass was 0 after a rejection            */
    SPEC_SEQ_FLAG_EOS = 0x400     /* spec_verify_sample_ex: the committed block ends
                                     with the end-of-sequence token                   */
};
/* Checks run in this order and the first failure is reported: length, draft
 * tokens, uniforms, per-sequence rules (spec_verify_sample_ex), then rows
 * i = 0..gamma_b (target row i, then draft row i) -- with early exit only up
 * to the sequence's first rejected draft. */

typedef enum { SPEC_BF16 = 0, SPEC_F32 = 1 } spec_dtype_t;

/* One side's production sampling rule [wrblog §2.3, §7.2-§7.3]:
 * temperature > 0 (finite); top_k == 0 or top_k >= vocab disables top-k;
 * top_p in (0, 1], 1 disables top-p. */
typedef struct {
    float temperature;
    int32_t top_k;
    float top_p;
} spec_sampling_params_t;

/* Bytes of workspace spec_verify_sample needs for this shape and these
 * parameters.  Returns SPEC_ERR_INVALID_ARG for sizes or parameters that
 * spec_verify_sample would reject, SPEC_ERR_UNSUPPORTED for gamma_max > 63
 * (the sampling verifier's limit).  The workspace must be zero-filled before
 * its first use; every call that returns SPEC_OK leaves its counter region
 * zero again, so a workspace is reusable without clearing. */
SPEC_API spec_status_t spec_verify_workspace_size(int32_t batch, int32_t gamma_max, int32_t vocab,
                                         spec_sampling_params_t target_params,
                                         spec_sampling_params_t draft_params,
                                         size_t* bytes);

/* Sampling-mode verification of `batch` sequences, asynchronous on `stream`:
 * one kernel launch, or two when the target's rows take the full-row path
 * (top_k off or above 128) -- the residual or bonus draw over a whole row
 * then runs in a second launch on the same stream, several CTAs per row.
 *
 * target_logits   [batch][gamma_max+1][vocab] of dtype.
 * draft_logits    [batch][gamma_max][vocab] of dtype, or NULL when every
 *                 sequence's draft is one-hot.
 * draft_tokens    [batch][gamma_max] int32, d_1..d_gamma_b per sequence
 *                 (may be NULL only when gamma_max == 0).
 * gamma_per_seq   [batch] int32 draft count per sequence, or NULL for
 *                 gamma_max everywhere (ragged batches pad to gamma_max).
 * draft_is_onehot [batch] uint8, non-zero = the draft proposed its tokens
 *                 with certainty (q is a delta at d_i, so a_i = p_i(d_i));
 *                 NULL = no one-hot sequence (ignored when draft_logits is
 *                 NULL).  One-hot sequences never read draft_logits.
 * u_accept        [batch][gamma_max] float, the uniform compared with a_i
 *                 (may be NULL only when gamma_max == 0).
 * u_sample        [batch] float, the uniform the residual or bonus draw uses.
 * out_tokens      [batch][gamma_max+1] int32: the accepted drafts, then the
 *                 replacement or bonus token, then -1.
 * out_num_accepted[batch] int32: accepted draft count A (0..gamma_b); the
 *                 sequence emits A+1 tokens; -1 = error, commit nothing.
 * out_accept_prob [batch][gamma_max] float a_i for i < gamma_b, -1 beyond;
 *                 or NULL.
 * out_residual_z  [batch] float, Z = sum (p_j - q_j)+ at the rejected
 *                 position, -1 when nothing was rejected; or NULL.
 * out_status      [batch] int32 SPEC_SEQ_* code, or NULL.
 * workspace       device buffer of at least spec_verify_workspace_size()
 *                 bytes, 256-byte aligned, zero-filled before first use. */
SPEC_API spec_status_t spec_verify_sample(const void* target_logits, const void* draft_logits,
                                 spec_dtype_t dtype, const int32_t* draft_tokens,
                                 const int32_t* gamma_per_seq, const uint8_t* draft_is_onehot,
                                 const float* u_accept, const float* u_sample,
                                 spec_sampling_params_t target_params,
                                 spec_sampling_params_t draft_params,
                                 int32_t batch, int32_t gamma_max, int32_t vocab,
                                 void* workspace, size_t workspace_bytes,
                                 int32_t* out_tokens, int32_t* out_num_accepted,
                                 float* out_accept_prob, float* out_residual_z,
                                 int32_t* out_status, void* stream);

/* Lenient sampling verification [magicnet §8]: spec_verify_sample with the
 * draft's distribution shrunk to lenience * q before it is compared with the
 * target, so draft token d_i is accepted with probability
 * a_i = min(1, p_i(d_i) / (lenience * q_i(d_i))), and at the first rejection
 * j the replacement is drawn from (p_j - lenience * q_j)+ / Z (the page gives
 * the acceptance rule; using lenience * q in the residual too is this
 * library's reading).  0 < lenience <= 1; lenience = 1 is spec_verify_sample
 * exactly.  Below 1 the output no longer follows the target's distribution:
 * the page's guarantee is that no token is emitted with more than
 * 1 / lenience times its target probability.  out_residual_z reports
 * Z = sum (p_j - lenience * q_j)+.  A lenience outside (0, 1] or NaN returns
 * SPEC_ERR_INVALID_ARG; everything else (arguments, workspace -- the same
 * spec_verify_workspace_size -- outputs, errors, launches) is as for
 * spec_verify_sample. */
SPEC_API spec_status_t spec_verify_sample_lenient(const void* target_logits, const void* draft_logits,
                                         spec_dtype_t dtype, const int32_t* draft_tokens,
                                         const int32_t* gamma_per_seq, const uint8_t* draft_is_onehot,
                                         const float* u_accept, const float* u_sample,
                                         spec_sampling_params_t target_params,
                                         spec_sampling_params_t draft_params, float lenience,
                                         int32_t batch, int32_t gamma_max, int32_t vocab,
                                         void* workspace, size_t workspace_bytes,
                                         int32_t* out_tokens, int32_t* out_num_accepted,
                                         float* out_accept_prob, float* out_residual_z,
                                         int32_t* out_status, void* stream);

/* Options of spec_verify_sample_ex.  {1.0f, -1, NULL, NULL, 0, 0} is
 * spec_verify_sample exactly.
 *
 * lenience           (0, 1]: as for spec_verify_sample_lenient [magicnet §8].
 * eos_token          -1, or an end-of-sequence token in [0, vocab): no token is
 *                    committed after it [wrblog §14.3].  When an accepted draft
 *                    d_t is the EOS, the sequence commits d_1..d_t only (no
 *                    replacement or bonus token; out_residual_z = -1);
 *                    SPEC_SEQ_FLAG_EOS marks a committed block that ends with
 *                    the EOS (also when the drawn token is the EOS).  The
 *                    acceptance scan and the draw are unchanged.
 * target_params_seq  [batch] DEVICE array of per-sequence target rules, or NULL
 * draft_params_seq   [batch] DEVICE array of per-sequence draft rules, or NULL:
 *                    requests batched together keep their own temperature,
 *                    top-k and top-p [wrblog §15].  When given, that side's
 *                    scalar rule is not used for sampling (it must still be
 *                    valid: it sizes nothing and is checked like the others).
 *                    A per-sequence rule outside its domain fails only its
 *                    sequence (SPEC_SEQ_BAD_PARAMS); a one-hot sequence's draft
 *                    rule is not used and not checked.  With per-sequence rules
 *                    the launch reserves the full-row path's extra shared
 *                    memory (fewer row CTAs per SM) and the draw kernel always
 *                    runs (its CTAs exit at once for sequences with kept-list
 *                    targets) -- unless kept_list_only is set.
 * kept_list_only     non-zero: the caller promises every per-sequence rule has
 *                    1 <= top_k <= 128 (top_k < vocab), the library's kept-list
 *                    path; the launch then keeps the plain call's occupancy and
 *                    workspace.  A per-sequence rule outside the promise fails
 *                    its sequence with SPEC_SEQ_BAD_PARAMS.  The scalar rules
 *                    must keep it too.  Ignored without per-sequence rules.
 * early_exit         non-zero: the sequential verifier of [wrblog §6] -- positions
 *                    are taken in order (target row i, draft row i, the decision
 *                    at i) and a sequence stops at its first failed row or
 *                    rejected draft.  The grid runs position-major, and a row
 *                    CTA that starts after an earlier position of its sequence
 *                    has stopped skips its row, so a launch of several waves
 *                    reads fewer rows.  Results: the same as without it on
 *                    valid rows; a NaN / +inf / all -inf row after the stop
 *                    does not fail the sequence, and out_accept_prob holds a_i
 *                    up to the stop and -1 after it.  Which rows are skipped
 *                    depends on timing, the results do not. */
typedef struct {
    float lenience;
    int32_t eos_token;
    const spec_sampling_params_t* target_params_seq;
    const spec_sampling_params_t* draft_params_seq;
    int32_t kept_list_only;
    int32_t early_exit;
} spec_verify_options_t;

/* Bytes of workspace spec_verify_sample_ex needs with these options (per-
 * sequence rules reserve room for both row paths).  options may be NULL. */
SPEC_API spec_status_t spec_verify_workspace_size_ex(int32_t batch, int32_t gamma_max, int32_t vocab,
                                            spec_sampling_params_t target_params,
                                            spec_sampling_params_t draft_params,
                                            const spec_verify_options_t* options, size_t* bytes);

/* spec_verify_sample with options (host pointer; NULL = the defaults):
 * lenience, the end-of-sequence commit and per-sequence sampling rules.
 * out_num_emitted [batch] int32, or NULL: tokens committed -- num_accepted + 1,
 * num_accepted when the block ends at an accepted EOS draft, -1 on error.
 * The workspace is spec_verify_workspace_size_ex() bytes.  An eos_token
 * outside [-1, vocab) or a lenience outside (0, 1] returns
 * SPEC_ERR_INVALID_ARG; everything else is as for spec_verify_sample. */
SPEC_API spec_status_t spec_verify_sample_ex(const void* target_logits, const void* draft_logits,
                                    spec_dtype_t dtype, const int32_t* draft_tokens,
                                    const int32_t* gamma_per_seq, const uint8_t* draft_is_onehot,
                                    const float* u_accept, const float* u_sample,
                                    spec_sampling_params_t target_params,
                                    spec_sampling_params_t draft_params,
                                    const spec_verify_options_t* options,
                                    int32_t batch, int32_t gamma_max, int32_t vocab,
                                    void* workspace, size_t workspace_bytes,
                                    int32_t* out_tokens, int32_t* out_num_accepted,
                                    float* out_accept_prob, float* out_residual_z,
                                    int32_t* out_status, int32_t* out_num_emitted, void* stream);

/* Bytes of workspace spec_verify_greedy needs (same zero-fill rule). */
SPEC_API spec_status_t spec_greedy_workspace_size(int32_t batch, int32_t gamma_max, size_t* bytes);

/* Greedy verification [wrblog §7.1; baisen §6]: g_i = argmax_x z_i(x)
 * (lowest index on ties) for i = 1..gamma_b+1; the sequence accepts
 * d_1..d_{j-1} where j is the first i with d_i != g_i and emits g_j, or
 * accepts every draft and emits g_{gamma_b+1}.  No sampling parameters and
 * no uniforms: argmax is unchanged by temperature, top-k and top-p.
 * Arguments as for spec_verify_sample. */
SPEC_API spec_status_t spec_verify_greedy(const void* target_logits, spec_dtype_t dtype,
                                 const int32_t* draft_tokens, const int32_t* gamma_per_seq,
                                 int32_t batch, int32_t gamma_max, int32_t vocab,
                                 void* workspace, size_t workspace_bytes,
                                 int32_t* out_tokens, int32_t* out_num_accepted,
                                 int32_t* out_status, void* stream);

/* Early-exit greedy verification [wrblog §6, §7.1]: the same outputs as
 * spec_verify_greedy on valid inputs, but a row is read only while the
 * sequence has not yet been decided: once row s of a sequence fails or
 * mismatches (d_s != g_s), rows after s are skipped, and the result depends
 * on rows 0..s alone.  The checks of a sequence run in the order length,
 * draft tokens, then rows 0..s; a NaN / +inf / all -inf row after the stop
 * does not fail the sequence (it would fail spec_verify_greedy).
 *
 * One launch over (position, sequence) pairs, positions first, so a row's
 * predecessors have usually finished when it starts; no CTA waits for
 * another.  A row whose predecessors are still running is read
 * speculatively (and abandoned part-way if an earlier row stops the sequence
 * meanwhile): out_rows_read can exceed (the stop + 1).
 * workspace     spec_greedy_workspace_size() bytes, same zero-fill rule
 *               (the kernel leaves it reusable).
 * out_rows_read [batch] int32: target rows read to the end (0 for a length or
 *               token error), or NULL.  Other arguments as for spec_verify_greedy. */
SPEC_API spec_status_t spec_verify_greedy_early(const void* target_logits, spec_dtype_t dtype,
                                       const int32_t* draft_tokens, const int32_t* gamma_per_seq,
                                       int32_t batch, int32_t gamma_max, int32_t vocab,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t* out_tokens, int32_t* out_num_accepted,
                                       int32_t* out_status, int32_t* out_rows_read, void* stream);

/* Workspace bytes spec_verify_greedy_tree needs (same zero-fill rule). */
SPEC_API spec_status_t spec_tree_workspace_size(int32_t batch, int32_t max_nodes, size_t* bytes);

/* Greedy verification of a draft tree per sequence [baisen §8; magicnet §7]:
 * several candidate continuations sharing prefixes, verified by one target
 * forward with tree attention.  Node 0 is the root (the position after the
 * committed prefix; its token is unused); node i > 0 carries draft token
 * tree_tokens[b][i] and parent tree_parents[b][i] < i.  Row i of target_logits
 * ([batch][max_nodes][vocab]) is the target's next-token logits after the path
 * root..i.  The accepted path starts at the root and moves to the child whose
 * token is the target's argmax at the current node (lowest index on argmax
 * ties; the first such child in node order if siblings repeat a token) until
 * no child matches; the argmax there is emitted (the correction, or the bonus
 * token at a leaf).  A chain tree (parent i - 1) is spec_verify_greedy.  The
 * pages give no multi-path acceptance rule for sampling mode; this library
 * has none.
 *
 * nodes_per_seq [batch] int32 in [1, max_nodes], or NULL (= max_nodes); nodes
 *               at or beyond it are never read.  Every node row below it is
 *               read, and a NaN / +inf / all -inf row fails the sequence.
 * out_tokens    [batch][max_nodes] int32: the accepted path's draft tokens, the
 *               emitted argmax, then -1.
 * out_num_accepted [batch]: accepted path length L (L + 1 tokens emitted), -1
 *               on error.
 * out_path      [batch][max_nodes] int32: the path's nodes, root first (L + 1
 *               entries), then -1; or NULL.
 * out_status    [batch] SPEC_SEQ_* (checks in order: length, node tokens,
 *               parents -> SPEC_SEQ_BAD_TREE, rows in node order), or NULL.
 * workspace     spec_tree_workspace_size() bytes, zero-filled before first use
 *               (left reusable).  One launch; other conventions as above. */
SPEC_API spec_status_t spec_verify_greedy_tree(const void* target_logits, spec_dtype_t dtype,
                                      const int32_t* tree_tokens, const int32_t* tree_parents,
                                      const int32_t* nodes_per_seq, int32_t batch, int32_t max_nodes,
                                      int32_t vocab, void* workspace, size_t workspace_bytes,
                                      int32_t* out_tokens, int32_t* out_num_accepted, int32_t* out_path,
                                      int32_t* out_status, void* stream);

/* Sampling-mode verification of a draft tree [baisen §8; magicnet §7]; the
 * acceptance rule is the plainest one that keeps the target's distribution,
 * since the pages give none for sampling mode.  Node 0 of each sequence's tree
 * is the root (the position after the committed prefix); node c > 0 carries
 * a draft token and a parent p_c < c.  The children of a node must be
 * independent draws from the draft distribution at that node (siblings may
 * repeat a token): that is what makes the result follow the target's law.
 * Walking from the root with the residual r = p_v (the target's distribution
 * at node v), the children are tried in node order: child c with token x is
 * accepted iff u_node[c] < min(1, r(x) / q_v(x)) [wrblog §4.1]; a rejection
 * replaces r by (r - q_v)+ / Z [wrblog §5] (Z == 0: r is kept and
 * SPEC_SEQ_FLAG_Z_ZERO set); an accepted child is entered with r = p_child.
 * When every child of the current node is rejected the token is drawn from r
 * with u_sample (inverse CDF in vocabulary order); at a node without children
 * it is drawn from p_v (the bonus) [wrblog §6].  With one child per node this
 * is spec_verify_sample.
 *
 * target_logits, draft_logits [batch][max_nodes][vocab] of dtype: row c is
 *               the target's / the draft's logits after the path root..c (the
 *               draft row of a node without children is not read).
 * tree_tokens, tree_parents [batch][max_nodes] int32 (entry 0 unused).
 * nodes_per_seq [batch] int32 in [1, max_nodes] (other values fail the
 *               sequence with SPEC_SEQ_BAD_LENGTH), or NULL (max_nodes).
 * u_node        [batch][max_nodes] float in [0, 1): node c's acceptance
 *               uniform (entry 0 unused; used only if c is tried).
 * u_sample      [batch] float in [0, 1).
 * target_params, draft_params: both with 1 <= top_k <= 128 and top_k < vocab
 *               (the kept-list path); other rules return SPEC_ERR_UNSUPPORTED.
 * max_nodes     1..32 (SPEC_ERR_UNSUPPORTED beyond).
 * workspace     spec_tree_sample_workspace_size() bytes, zero-filled before
 *               first use (left reusable).
 * out_tokens    [batch][max_nodes]: the accepted path's tokens, the drawn
 *               token, then -1.  out_num_accepted [batch]: the path length
 *               (-1 on error).  out_path [batch][max_nodes]: the path's nodes,
 *               root first, then -1, or NULL.  out_accept_prob
 *               [batch][max_nodes - 1]: entry c - 1 the acceptance probability
 *               of node c if it was tried, -1 otherwise, or NULL.
 *               out_residual_z [batch]: Z of the residual the token was drawn
 *               from (-1 for a bonus draw), or NULL.  out_status [batch]
 *               SPEC_SEQ_* (checks in order: length, node tokens, parents ->
 *               SPEC_SEQ_BAD_TREE, uniforms, rows in node order: target row c,
 *               then draft row c), or NULL.
 * One launch; every node's target row and the draft row of every node with
 * children are read; other conventions as above. */
SPEC_API spec_status_t spec_tree_sample_workspace_size(int32_t batch, int32_t max_nodes, int32_t vocab,
                                              spec_sampling_params_t target_params,
                                              spec_sampling_params_t draft_params, size_t* bytes);
SPEC_API spec_status_t spec_verify_sample_tree(const void* target_logits, const void* draft_logits,
                                      spec_dtype_t dtype, const int32_t* tree_tokens,
                                      const int32_t* tree_parents, const int32_t* nodes_per_seq,
                                      const float* u_node, const float* u_sample,
                                      spec_sampling_params_t target_params,
                                      spec_sampling_params_t draft_params, int32_t batch,
                                      int32_t max_nodes, int32_t vocab, void* workspace,
                                      size_t workspace_bytes, int32_t* out_tokens,
                                      int32_t* out_num_accepted, int32_t* out_path,
                                      float* out_accept_prob, float* out_residual_z,
                                      int32_t* out_status, void* stream);

/* The transform step alone [wrblog §7.2, §7.3]: writes the full probability
 * rows p = top_p(top_k(softmax(z / T))) the verifier samples from.
 * logits [rows][vocab] of dtype; out_probs [rows][vocab] float;
 * out_row_status [rows] int32 (SPEC_SEQ_OK, SPEC_SEQ_NONFINITE or
 * SPEC_SEQ_EMPTY_SUPPORT; a failed row is written as zeros), or NULL.
 * Needs no workspace. */
SPEC_API spec_status_t spec_transform_probs(const void* logits, spec_dtype_t dtype, int32_t rows,
                                   int32_t vocab, spec_sampling_params_t params,
                                   float* out_probs, int32_t* out_row_status, void* stream);

/* spec_verify_sample without a caller-provided workspace: for callers that
 * cannot allocate device memory themselves -- for example a plugin hosted by an
 * inference server whose device memory belongs to the server's own allocator,
 * or a latency-critical path that must not pay cudaMalloc's device-wide
 * synchronisation.  This entry point has no counterpart in the method's
 * description; it only changes where the scratch memory comes from.
 *
 * The scratch is a fixed 8 MiB array inside the library's device image; every
 * GPU that loads the library holds it until the process exits.  Requests whose
 * workspace (spec_verify_workspace_size) exceeds 8 MiB return
 * SPEC_ERR_WORKSPACE and launch nothing.  Nothing is allocated: no cudaMalloc,
 * cudaFree or allocating library routine is called.  Each call made outside
 * stream capture looks up the array's device address (cudaGetSymbolAddress)
 * with the current device and remembers it for that device; a call made while
 * `stream` is being captured uses the remembered address, so make a first call
 * on each device before any stream capture (under capture with none
 * remembered the call returns SPEC_ERR_CUDA).  After the host checks of
 * spec_verify_sample have passed, each call clears the scratch's counters with
 * cudaMemsetAsync on `stream` and then launches as spec_verify_sample does; a
 * call refused by those checks launches nothing and leaves the scratch alone.
 * All calls share the one array, which keeps the last call's contents: calls
 * that overlap on the GPU (other streams, other host threads) race and must
 * not be issued.  Other arguments, outputs and errors are as for
 * spec_verify_sample. */
SPEC_API spec_status_t spec_verify_sample_noalloc(const void* target_logits, const void* draft_logits,
                                                  spec_dtype_t dtype, const int32_t* draft_tokens,
                                                  const int32_t* gamma_per_seq,
                                                  const uint8_t* draft_is_onehot,
                                                  const float* u_accept, const float* u_sample,
                                                  spec_sampling_params_t target_params,
                                                  spec_sampling_params_t draft_params,
                                                  int32_t batch, int32_t gamma_max, int32_t vocab,
                                                  int32_t* out_tokens, int32_t* out_num_accepted,
                                                  float* out_accept_prob, float* out_residual_z,
                                                  int32_t* out_status, void* stream);

/* Static, NUL-terminated description of a spec_status_t. */
SPEC_API const char* spec_status_string(spec_status_t status);

/* Process-wide switch (default 0).  Non-zero: spec_verify_sample /
 * spec_verify_sample_lenient on the kept-list path (and the no-alloc call),
 * spec_verify_greedy and spec_verify_greedy_tree when no per-sequence lengths,
 * one-hot flags or node counts are given, and spec_verify_sample_tree without
 * node counts, stream their logits rows BEFORE they wait for the previous
 * kernel in the stream to complete, and wait only before they read any other
 * input or write anything (spec_verify_sample_tree also reads the tree's
 * parents early, to know which draft rows are used).  Back-to-back
 * calls then overlap one call's tail with the next call's stream (the serving
 * workload on GB300: 38.5 -> 26.8 us per call); results are unchanged.
 * The caller guarantees that the logits (and tree parents) a call reads are
 * completely written by the time the previous kernel in its stream allows its
 * dependents to launch: true when that kernel does not use programmatic dependent launch
 * (a kernel without griddepcontrol.launch_dependents allows it only when it
 * completes), when it is a call of this library (no kernel here writes
 * logits), or when a stream operation other than a kernel launch (a copy)
 * separates the producer from the call (the relaxed ordering applies only
 * between two consecutive kernel launches).
 * A producer of logits that signals its dependents before its last writes
 * must not directly precede a call while this switch is on.  The setting is
 * read when a call is made.  Always returns SPEC_OK. */
SPEC_API spec_status_t spec_set_early_logits_reads(int32_t enable);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
