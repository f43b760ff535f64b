"""Plain float64 CPU oracle for the batched speculative-decoding verify-and-sample step.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` are the only callers.  The CUDA
library never calls this module and shares no code, table or constant with it.

What it computes, in the pages' order (sources are listed at the end of this
docstring and cited as ``[tag §section]``):

1. The production transforms that turn logits into the distribution actually
   sampled from: temperature, then top-k, then top-p.  p (target) and q (draft)
   each use their own parameters.  [wrblog §2.3, §7.2, §7.3; magicnet §2]
2. Left-to-right verification: draft token d_i is accepted with probability
   a_i = min(1, p_i(d_i) / q_i(d_i)); the scan stops at the first rejection and
   every later draft is discarded.  [wrblog §4.1, §6; rainlin §1-§2; baisen §4]
3. At the first rejection j the replacement token is drawn from the residual
   (p_j - q_j)+ / Z with Z = sum (p_j - q_j)+.  If all drafts are accepted a
   bonus token is drawn from p_{gamma+1}.  [wrblog §5, §6; rainlin §2; baisen §4]
4. Greedy mode: accept while d_i equals argmax p_i; at the first mismatch emit
   argmax p_i; if every draft matches emit argmax p_{gamma+1}.
   [wrblog §7.1; baisen §2, §6; rainlin §2]

All arithmetic is float64 NumPy.  bf16 logits are widened exactly (bit shift).
Sorting, cumulative sums and ``searchsorted`` are library primitives; nothing
is blocked, fused or reordered beyond the definitions below.

Readings where the pages are silent (each is named where it is used):

* R1  transform order: temperature, top-k on the tempered logits, renormalise,
      top-p on the renormalised probabilities, renormalise.
* R2  ties: every ordering is (value descending, token index ascending).
* R3  top-p keeps the shortest prefix of that order whose cumulative
      probability is >= top_p; top_p == 1 keeps everything; top_k == 0 or
      top_k >= V keeps everything.
* R4  accept iff u < a (strict), u in [0, 1)  -- as in the demo of [wrblog §8].
* R5  a uniform u picks the smallest token x (vocabulary order) whose
      cumulative weight C(x) = sum_{y<=x} w(y) exceeds u * C(V-1).
* R6  q(d) == 0: a = 1 if p(d) > 0 else 0, and the sequence is flagged.
* R7  Z == 0 after a rejection (only reachable through rounding): draw from
      p_j instead and flag the sequence.
* R8  one uniform per draft position plus one uniform u_sample that the
      residual draw or the bonus draw consumes.
* R9  the bonus token is part of the output ([wrblog §6], [rainlin §1]).
* R10 a NaN or +inf logit in any row the sequence uses, or a row whose logits
      are all -inf, fails the whole sequence: nothing is committed
      ([wrblog §15]).  -inf marks a banned token ([wrblog §2.3]).
* R11 early-exit greedy: the rows are read in position order and reading
      stops at the first draft that differs from the target's argmax -- the
      sequential verifier of [wrblog §6], which never looks past the first
      rejection.  "The rows the sequence uses" in R10 are then the rows read.
* R13 per-sequence sampling rules [wrblog §15]: requests in one batch keep their
      own temperature / top-k / top-p, so each sequence may carry its own target
      and draft rules.  A rule outside its domain (temperature not finite or
      <= 0, top_k < 0, top_p outside (0, 1]) fails that sequence only, checked
      after the uniforms; a one-hot sequence's draft rule is not used, so not
      checked.
* R14 end-of-sequence commit [wrblog §14.3]: no token is committed after the
      end-of-sequence token.  The emitted block (accepted drafts, then the
      replacement or bonus token) is cut just after its first EOS; when an
      accepted draft is the EOS, the committed drafts end there and no
      replacement or bonus token follows.  The scan and the draw are unchanged
      (the same uniforms decide them); only the commit is cut.
* R15 greedy tree verification [baisen §8; magicnet §7]:
      the draft is a tree; node 0 is the root (the position after the
      committed prefix) and node i > 0 carries a draft token and a parent
      node p_i < i; the target row of node i scores the token after the path
      root..i.  The pages say the tree is verified in one forward and the best
      path is accepted, not how.  Greedy reading: from the root, move to the
      child whose token is the target's argmax at the current node -- the
      first such child in index order when siblings repeat a token -- until no
      child matches, then emit the argmax there (the correction, or the bonus
      at a leaf).  With distinct sibling tokens this is the deepest node whose
      whole path matches the argmaxes, and a chain (p_i = i - 1) is the linear
      greedy verifier.  Every node row is read, so any failed row fails the
      sequence (R10).  The sampling-mode counterpart is R17.
* R12 lenience beta in (0, 1] [magicnet §8]: the page shrinks the draft
      distribution to beta q and then compares it with the target; here beta q
      stands in for q throughout -- acceptance min(1, p / (beta q)) and, on a
      rejection, the residual (p - beta q)+ / Z_beta.  beta = 1 is the lossless
      path.  The page states only the acceptance rule and the guarantee that no
      token is drawn with more than 1 / beta times its true probability; the
      residual is this reading (it meets that guarantee, as the tests check).

Pins (tests/test_oracle_*.py): the worked examples of [wrblog §4.3, §5, §7.1]
and [baisen §2, §4, §6]; the identities Z = sum (p-q)+ = sum (q-p)+ =
1 - sum min(p,q) [rainlin §2; baisen §5; magicnet §3]; the exact single- and
multi-token output law by exhaustive enumeration; the truncated-geometric law
of tokens per round and its mean (1 - a^{g+1}) / (1 - a) [magicnet §4;
rainlin §3; wrblog §10]; the textbook softmax; brute-force top-k / top-p sets.
Parity unpinned: the tie rule R2 and the transform order R1 are readings, not
statements of the pages; only self-consistency and the brute-force set
definitions check them.

Sources:
  [wrblog]   "推测解码：草稿模型、接受率、正确性与加速边界" (wrblog.cn)
  [aiqz]     "投机解码：草稿小模型 + 大模型并行验证的无损加速" (aiqz.cc)
  [rainlin]  "投机解码" (rainlin-net.pages.dev, llm-inference/speculative-decoding)
  [baisen]   "投机采样 / 投机解码（Speculative Decoding）" (baisen.site)
  [magicnet] "投机解码到底能加速多少：把接受率、草稿成本与墙钟收益算清楚"
             (magicnetworld.com)
* R16 early-exit sampling (the sampling counterpart of R11): positions are
      read in order -- target row i, then draft row i -- and the scan stops at
      the first position whose rows fail or whose draft is rejected, the
      sequential verifier of [wrblog §6].  Rows after that position are never
      read, so they cannot fail the sequence, and their acceptance
      probabilities are reported as -1.  On inputs whose every row is valid
      the emitted tokens, counts, flags and residual mass equal R1-R10's.
* R17 sampling-mode tree verification [baisen §8; magicnet §7]: the pages verify a
      draft tree in one target forward and accept the best path, but give no
      acceptance rule for sampling mode.  Reading, the plainest one under which
      the output keeps the target's law: the children of a node are proposals
      drawn independently from the draft distribution q_v at that node (so
      siblings may repeat a token).  Walk from the root with the residual
      r = p_v: try the children in node order; child c with token x is accepted
      with probability min(1, r(x) / q_v(x)) (R4, R6 against its own uniform);
      after a rejection r becomes (r - q_v)+ / Z (R7 when Z == 0: r is kept and
      the sequence flagged).  An accepted child is entered with r = p_child.
      When every child of the current node is rejected, the token is drawn from
      r; at a node without children, from p_v (the bonus).  One uniform per
      non-root node (used only if the node is tried) and one u_sample for the
      final draw (R8).  A chain (each node one child) is the linear verifier
      R1-R10.  Every node's target row and the draft row of every node with
      children are read, so any failed row fails the sequence (R10).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

# Per-sequence status codes.  The numeric values are an interface convention
# that the C header states independently.
SEQ_OK = 0
SEQ_BAD_LENGTH = 1      # gamma_b outside [0, gamma_max]
SEQ_BAD_TOKEN = 2       # a draft token outside [0, V)
SEQ_BAD_UNIFORM = 3     # a uniform outside [0, 1) or NaN
SEQ_NONFINITE = 4       # NaN or +inf logit in a row the sequence uses
SEQ_EMPTY_SUPPORT = 5   # a row whose logits are all -inf
SEQ_BAD_PARAMS = 6      # a sampling rule the sequence uses is outside its domain (R13)
SEQ_BAD_TREE = 7        # a draft-tree node whose parent is not an earlier node (R15)
SEQ_ERROR_MASK = 0xFF
SEQ_FLAG_ZERO_Q = 0x100  # an evaluated draft token had q(d) == 0 (R6)
SEQ_FLAG_Z_ZERO = 0x200  # residual mass was 0 after a rejection (R7)
SEQ_FLAG_EOS = 0x400     # the committed block ends at the end-of-sequence token (R14)


# --------------------------------------------------------------------------
# Input widening
# --------------------------------------------------------------------------
def bf16_bits_to_float64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64 exactly.

    A bf16 value is the upper half of an IEEE float32, so shifting the 16 bits
    into the high half of a 32-bit word reproduces the value bit for bit.
    """
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def float32_to_float64(x: np.ndarray) -> np.ndarray:
    """Widen float32 logits to float64 exactly."""
    return np.asarray(x, dtype=np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Step 1: logits -> sampling distribution   [wrblog §2.3, §7.2, §7.3]
# --------------------------------------------------------------------------
def order_desc(z: np.ndarray) -> np.ndarray:
    """Token indices sorted by (logit descending, index ascending)  (R2).

    ``np.lexsort`` sorts by its last key first: -z ascending is z descending,
    ties fall back to the index key, ascending.  -0.0 and +0.0 compare equal,
    so they tie and the lower index wins.
    """
    idx = np.arange(z.size)
    return np.lexsort((idx, -z))


TOP_P_AMBIGUITY = 1e-6


@dataclass
class RowDist:
    """One transformed row: the distribution p (or q) over the vocabulary."""
    status: int
    probs: np.ndarray                  # (V,) float64; zeros unless status == SEQ_OK
    kept: np.ndarray                   # kept token ids in (value desc, index asc) order
    top_p_margin: float = np.inf       # distance of the top-p decision from top_p (R3)
    # Tokens whose membership in the top-p set turns on a cumulative probability
    # within TOP_P_AMBIGUITY of top_p (a token is kept iff the cumulative of the
    # tokens before it is < top_p), and their total probability before the cut.
    ambiguous: np.ndarray = field(default_factory=lambda: np.zeros(0, dtype=np.int64))
    ambiguous_mass: float = 0.0


def row_status(z: np.ndarray) -> int:
    """R10: NaN / +inf logits are invalid; a row of only -inf has no support."""
    if np.isnan(z).any() or np.isposinf(z).any():
        return SEQ_NONFINITE
    if np.all(np.isneginf(z)):
        return SEQ_EMPTY_SUPPORT
    return SEQ_OK


def transform_row(z: np.ndarray, temperature: float, top_k: int, top_p: float) -> RowDist:
    """p_T = softmax(z / T) restricted by top-k then top-p  [wrblog §7.2, §7.3] (R1-R3).

    Temperature is order preserving for T > 0, so the top-k set is taken on the
    raw logits.  The softmax over the kept set subtracts the largest kept logit
    (a constant shift that leaves softmax unchanged).
    """
    z = np.asarray(z, dtype=np.float64)
    V = z.size
    status = row_status(z)
    if status != SEQ_OK:
        return RowDist(status, np.zeros(V), np.zeros(0, dtype=np.int64))
    if not temperature > 0:
        raise ValueError("temperature must be > 0; use greedy verification for T -> 0")
    order = order_desc(z)
    kept = order if (top_k <= 0 or top_k >= V) else order[:top_k]
    zk = z[kept]
    m = zk[0]
    w = np.exp((zk - m) / temperature)          # -inf logits give weight 0
    p_tilde = w / w.sum()
    margin = np.inf
    ambiguous = np.zeros(0, dtype=np.int64)
    ambiguous_mass = 0.0
    if top_p < 1.0:
        cum = np.cumsum(p_tilde)
        reached = np.flatnonzero(cum >= top_p)
        n = int(reached[0]) + 1 if reached.size else kept.size
        above = cum[n - 1] - top_p
        below = top_p - cum[n - 2] if n >= 2 else np.inf
        margin = float(min(abs(above), abs(below)))
        before = np.concatenate([[0.0], cum[:-1]])        # cumulative of the tokens before each
        amb = np.abs(before - top_p) < TOP_P_AMBIGUITY
        ambiguous = kept[amb]
        ambiguous_mass = float(p_tilde[amb].sum())
        kept = kept[:n]
        w = w[:n]
    probs = np.zeros(V)
    probs[kept] = w / w.sum()
    return RowDist(SEQ_OK, probs, kept, margin, ambiguous, ambiguous_mass)


def one_hot_row(V: int, token: int) -> RowDist:
    """A draft that proposes one token with certainty (n-gram style, q = delta)."""
    probs = np.zeros(V)
    if 0 <= token < V:
        probs[token] = 1.0
    return RowDist(SEQ_OK, probs, np.array([token], dtype=np.int64))


# --------------------------------------------------------------------------
# Step 2: acceptance   [wrblog §4.1, §4.2, §6]
# --------------------------------------------------------------------------
def acceptance_probability(p_x: float, q_x: float, lenience: float = 1.0) -> tuple[float, bool]:
    """a(x) = min(1, p(x) / (beta q(x))) [wrblog §4.1; magicnet §8 (R12)], beta = 1 by
    default; returns (a, q_was_zero) (R6)."""
    if q_x > 0.0:
        return min(1.0, p_x / (lenience * q_x)), False
    return (1.0 if p_x > 0.0 else 0.0), True


def acceptance_rate(p: np.ndarray, q: np.ndarray) -> float:
    """Expected acceptance at one position: sum_x min(p(x), q(x))  [wrblog §4.2]."""
    return float(np.minimum(p, q).sum())


def residual_weights(p: np.ndarray, q: np.ndarray, lenience: float = 1.0) -> np.ndarray:
    """Unnormalised residual (p - beta q)+  [wrblog §5; magicnet §8 (R12)], beta = 1 by default."""
    return np.maximum(p - lenience * q, 0.0)


# --------------------------------------------------------------------------
# Step 3: draw one token from a weight vector (R5)
# --------------------------------------------------------------------------
def inverse_cdf(w: np.ndarray, u: float) -> tuple[int, float, float]:
    """Smallest x with C(x) > u * C(V-1), C the running sum in vocabulary order.

    Returns (token, lo, hi): the token's normalised CDF interval [lo, hi).
    """
    C = np.cumsum(np.asarray(w, dtype=np.float64))
    Z = C[-1]
    if not Z > 0:
        raise ValueError("cannot sample from an all-zero weight vector")
    x = int(np.searchsorted(C, u * Z, side="right"))
    x = min(x, C.size - 1)
    lo = C[x - 1] / Z if x > 0 else 0.0
    return x, float(lo), float(C[x] / Z)


# --------------------------------------------------------------------------
# One sequence
# --------------------------------------------------------------------------
@dataclass
class SeqResult:
    tokens: np.ndarray          # (gamma_max + 1,) int64; -1 after the last emitted token
    num_accepted: int           # -1 on error (commit nothing)
    status: int
    accept_prob: np.ndarray     # (gamma_max,) a_i for i < gamma_b, -1 elsewhere
    residual_Z: float           # Z at the rejected position, -1 when nothing was rejected
    accept_margin: float = np.inf   # min |u_i - a_i| over evaluated positions
    top_p_margin: float = np.inf    # min top-p margin over the rows used
    # evaluated draft tokens whose top-p membership (in p_i or q_i) is ambiguous
    draft_ambiguous: bool = False
    # tokens of the row(s) the final draw used whose top-p membership is ambiguous
    sample_ambiguous: np.ndarray = field(default_factory=lambda: np.zeros(0, dtype=np.int64))
    sample_u: float = np.nan
    sample_lo: float = np.nan
    sample_hi: float = np.nan
    sample_cdf: np.ndarray | None = field(default=None, repr=False)  # normalised CDF drawn from
    rows_read: int = -1             # early-exit greedy: target rows read (R11)
    num_emitted: int = -1           # tokens committed: num_accepted + 1, or fewer after an EOS cut (R14)
    path: list | None = None        # tree verification: the accepted path's nodes, root first (R15, R17)
    tree_trace: list | None = None  # sampling tree (R17): (node, a) of every tried node, in order


def _error_result(status: int, gamma_max: int) -> SeqResult:
    return SeqResult(np.full(gamma_max + 1, -1, dtype=np.int64), -1, status,
                     np.full(gamma_max, -1.0), -1.0)


def _valid_uniform(u: float) -> bool:
    return bool(0.0 <= u < 1.0)


def valid_params(params: tuple[float, int, float]) -> bool:
    """The domain of a sampling rule (R13): temperature finite and > 0, top_k >= 0, top_p in (0, 1]."""
    T, k, p = params
    return bool(np.isfinite(T) and T > 0.0 and k >= 0 and 0.0 < p <= 1.0)


def verify_sample_sequence(target: np.ndarray, draft: np.ndarray | None, tokens: np.ndarray,
                           u_accept: np.ndarray, u_sample: float,
                           target_params: tuple[float, int, float],
                           draft_params: tuple[float, int, float],
                           gamma_b: int, gamma_max: int, one_hot: bool,
                           keep_cdf: bool = False, lenience: float = 1.0,
                           early_exit: bool = False) -> SeqResult:
    """Verify one sequence in sampling mode  [wrblog §6; rainlin §1].

    target: (gamma_max+1, V) float64 logits; rows 0..gamma_b are used.
    draft:  (gamma_max, V) float64 logits, rows 0..gamma_b-1 used; ignored when one_hot.
    tokens: (gamma_max,) draft tokens d_1..d_gamma (0-based positions).
    early_exit: read the rows position by position and stop at the first
    failed row or rejected draft (R16).
    """
    V = target.shape[1]
    if not 0.0 < lenience <= 1.0:                                   # [magicnet §8]: 0 < beta <= 1
        raise ValueError("lenience must lie in (0, 1]")
    if not 0 <= gamma_b <= gamma_max:
        return _error_result(SEQ_BAD_LENGTH, gamma_max)
    d = [int(t) for t in tokens[:gamma_b]]
    if any(not 0 <= t < V for t in d):
        return _error_result(SEQ_BAD_TOKEN, gamma_max)
    if not all(_valid_uniform(float(u)) for u in u_accept[:gamma_b]) or not _valid_uniform(float(u_sample)):
        return _error_result(SEQ_BAD_UNIFORM, gamma_max)
    if not valid_params(target_params) or (not one_hot and not valid_params(draft_params)):    # R13
        return _error_result(SEQ_BAD_PARAMS, gamma_max)

    # Step 1: p_1..p_{gamma+1} and q_1..q_gamma, each with its own transform [wrblog §7.2].
    # Step 2: a_i for every draft position; the scan stops at the first rejection [wrblog §6].
    p_rows, q_rows = [], []
    a = np.full(gamma_max, -1.0)
    zero_q = np.zeros(gamma_max, dtype=bool)
    status = SEQ_OK
    rejected_at = None
    accept_margin = np.inf

    def draft_row(i):
        return one_hot_row(V, d[i]) if one_hot else transform_row(draft[i], *draft_params)

    def decide(i) -> bool:
        """a_i, the flags and the margin for position i; True if d_i is rejected."""
        nonlocal status, accept_margin
        a[i], zero_q[i] = acceptance_probability(p_rows[i].probs[d[i]], q_rows[i].probs[d[i]], lenience)
        if zero_q[i]:
            status |= SEQ_FLAG_ZERO_Q
        accept_margin = min(accept_margin, abs(float(u_accept[i]) - a[i]))
        return not float(u_accept[i]) < a[i]       # R4: strict comparison

    if early_exit:
        # R16: target row i, then draft row i, then the decision at i
        for i in range(gamma_b + 1):
            p_i = transform_row(target[i], *target_params)
            if p_i.status != SEQ_OK:
                res = _error_result(p_i.status, gamma_max)
                res.rows_read = i + 1
                return res
            p_rows.append(p_i)
            if i == gamma_b:
                break
            q_i = draft_row(i)
            if q_i.status != SEQ_OK:
                res = _error_result(q_i.status, gamma_max)
                res.rows_read = i + 1
                return res
            q_rows.append(q_i)
            if decide(i):
                rejected_at = i
                break
    else:
        for i in range(gamma_b + 1):
            p_i = transform_row(target[i], *target_params)
            if p_i.status != SEQ_OK:
                return _error_result(p_i.status, gamma_max)
            p_rows.append(p_i)
            if i < gamma_b:
                q_i = draft_row(i)
                if q_i.status != SEQ_OK:
                    return _error_result(q_i.status, gamma_max)
                q_rows.append(q_i)
        for i in range(gamma_b):                    # a_i for every position, then the scan
            a[i], zero_q[i] = acceptance_probability(p_rows[i].probs[d[i]], q_rows[i].probs[d[i]], lenience)
        for i in range(gamma_b):
            if zero_q[i]:
                status |= SEQ_FLAG_ZERO_Q
            accept_margin = min(accept_margin, abs(float(u_accept[i]) - a[i]))
            if not float(u_accept[i]) < a[i]:      # R4: strict comparison
                rejected_at = i
                break

    # Step 3: residual at the rejected position, else the bonus from p_{gamma+1}.
    residual_Z = -1.0
    if rejected_at is not None:
        j = rejected_at
        w = residual_weights(p_rows[j].probs, q_rows[j].probs, lenience)   # [wrblog §5] (R12)
        residual_Z = float(w.sum())
        if not residual_Z > 0:                                      # R7
            w = p_rows[j].probs
            status |= SEQ_FLAG_Z_ZERO
        n_acc = j
    else:
        w = p_rows[gamma_b].probs                                   # bonus [wrblog §6]
        n_acc = gamma_b
    tok, lo, hi = inverse_cdf(w, float(u_sample))

    out = np.full(gamma_max + 1, -1, dtype=np.int64)
    out[:n_acc] = d[:n_acc]
    out[n_acc] = tok
    used = p_rows[: n_acc + 1] + ([] if one_hot else q_rows[: min(n_acc + 1, gamma_b)])
    top_p_margin = min([r.top_p_margin for r in used] + [np.inf])
    evaluated = range(min(n_acc + 1, gamma_b))
    draft_amb = any(d[i] in p_rows[i].ambiguous or (not one_hot and d[i] in q_rows[i].ambiguous)
                    for i in evaluated)
    sample_rows = [p_rows[n_acc]] + ([q_rows[n_acc]] if (rejected_at is not None and not one_hot) else [])
    sample_amb = np.unique(np.concatenate([r.ambiguous for r in sample_rows]))
    res = SeqResult(out, n_acc, status, a, residual_Z, accept_margin, top_p_margin,
                    draft_ambiguous=draft_amb, sample_ambiguous=sample_amb,
                    sample_u=float(u_sample), sample_lo=lo, sample_hi=hi, num_emitted=n_acc + 1,
                    rows_read=n_acc + 1 if early_exit else -1)
    if keep_cdf:
        C = np.cumsum(w)
        res.sample_cdf = C / C[-1]
    return res


def commit_at_eos(res: SeqResult, eos_token: int) -> SeqResult:
    """Cut a sequence's committed block just after its first end-of-sequence token
    [wrblog §14.3] (R14).  eos_token < 0 and failed sequences are left unchanged."""
    if eos_token < 0 or res.num_accepted < 0:
        return res
    block = res.tokens[: res.num_accepted + 1]
    hits = np.flatnonzero(block == eos_token)
    if hits.size == 0:
        return res
    t = int(hits[0])
    tokens = res.tokens.copy()
    tokens[t + 1:] = -1
    cut = replace(res, tokens=tokens, status=res.status | SEQ_FLAG_EOS)
    if t < res.num_accepted:        # an accepted draft is the EOS: no replacement / bonus token
        cut.num_accepted = t + 1
        cut.num_emitted = t + 1
    return cut


def greedy_row(z: np.ndarray) -> tuple[int, int]:
    """argmax with the lowest index on ties (R2), and the row status (R10)."""
    status = row_status(z)
    if status != SEQ_OK:
        return -1, status
    return int(order_desc(z)[0]), SEQ_OK


def verify_greedy_sequence(target: np.ndarray, tokens: np.ndarray, gamma_b: int,
                           gamma_max: int) -> SeqResult:
    """Greedy verification: longest argmax-matching prefix plus one target token.

    [wrblog §7.1; baisen §2 (the "mat and the cat" walk-through), §6; rainlin §2]
    """
    V = target.shape[1]
    if not 0 <= gamma_b <= gamma_max:
        return _error_result(SEQ_BAD_LENGTH, gamma_max)
    d = [int(t) for t in tokens[:gamma_b]]
    if any(not 0 <= t < V for t in d):
        return _error_result(SEQ_BAD_TOKEN, gamma_max)
    g = []
    for i in range(gamma_b + 1):
        gi, st = greedy_row(target[i])
        if st != SEQ_OK:
            return _error_result(st, gamma_max)
        g.append(gi)
    n_acc = gamma_b
    for i in range(gamma_b):
        if d[i] != g[i]:
            n_acc = i
            break
    out = np.full(gamma_max + 1, -1, dtype=np.int64)
    out[:n_acc] = d[:n_acc]
    out[n_acc] = g[n_acc]
    return SeqResult(out, n_acc, SEQ_OK, np.full(gamma_max, -1.0), -1.0)


def verify_greedy_tree_sequence(target: np.ndarray, tokens: np.ndarray, parents: np.ndarray,
                                n_nodes: int, max_nodes: int) -> SeqResult:
    """Greedy verification of a draft tree (R15).

    target: (max_nodes, V) float64 logits, row i for node i (rows 0..n_nodes-1 used);
    tokens / parents: (max_nodes,) node tokens and parent indices (entry 0, the root, unused).
    Returns tokens = the accepted path's draft tokens then the correction / bonus token,
    num_accepted = the path length L, and the path's nodes (root first) in ``path``.
    """
    V = target.shape[1]
    if not 1 <= n_nodes <= max_nodes:
        return _error_result(SEQ_BAD_LENGTH, max_nodes - 1)
    if any(not 0 <= int(tokens[i]) < V for i in range(1, n_nodes)):
        return _error_result(SEQ_BAD_TOKEN, max_nodes - 1)
    if any(not 0 <= int(parents[i]) < i for i in range(1, n_nodes)):
        return _error_result(SEQ_BAD_TREE, max_nodes - 1)
    g = []
    for i in range(n_nodes):
        gi, st = greedy_row(target[i])
        if st != SEQ_OK:
            return _error_result(st, max_nodes - 1)
        g.append(gi)
    path = [0]
    while True:
        cur = path[-1]
        nxt = next((c for c in range(cur + 1, n_nodes)
                    if int(parents[c]) == cur and int(tokens[c]) == g[cur]), None)
        if nxt is None:
            break
        path.append(nxt)
    L = len(path) - 1
    out = np.full(max_nodes, -1, dtype=np.int64)
    out[:L] = [int(tokens[c]) for c in path[1:]]
    out[L] = g[path[-1]]
    res = SeqResult(out, L, SEQ_OK, np.full(max_nodes - 1, -1.0), -1.0, num_emitted=L + 1)
    res.path = path
    return res


def verify_greedy_tree(target: np.ndarray, tokens: np.ndarray, parents: np.ndarray,
                       nodes_per_seq: np.ndarray | None = None) -> BatchResult:
    """Batched greedy tree verification (R15), one sequence at a time."""
    B, N, _ = target.shape
    out = []
    for b in range(B):
        n = N if nodes_per_seq is None else int(nodes_per_seq[b])
        out.append(verify_greedy_tree_sequence(target[b], tokens[b], parents[b], n, N))
    return _collect(out)


def verify_sample_tree_sequence(target: np.ndarray, draft: np.ndarray, tokens: np.ndarray,
                                parents: np.ndarray, u_node: np.ndarray, u_sample: float,
                                n_nodes: int, max_nodes: int,
                                target_params: tuple[float, int, float],
                                draft_params: tuple[float, int, float]) -> SeqResult:
    """Sampling-mode verification of a draft tree (R17)  [baisen §8; magicnet §7; wrblog §4-§6].

    target, draft: (max_nodes, V) float64 logits; row v is the target's / the draft's
    distribution after the path root..v (draft rows of nodes without children are unused).
    tokens / parents: (max_nodes,) node tokens and parent indices (entry 0, the root, unused).
    u_node: (max_nodes,) the acceptance uniform of each node (entry 0 unused); u_sample: the
    final draw's uniform.  Returns tokens = the accepted path's tokens then the drawn token,
    num_accepted = the path length, accept_prob[v - 1] = a of node v if it was tried (-1
    otherwise), residual_Z = Z of the residual the final token was drawn from (-1 for a
    bonus draw), path = the accepted nodes (root first), tree_trace = the tried (node, a).
    """
    V = target.shape[1]
    G = max_nodes - 1
    if not 1 <= n_nodes <= max_nodes:
        return _error_result(SEQ_BAD_LENGTH, G)
    if any(not 0 <= int(tokens[i]) < V for i in range(1, n_nodes)):
        return _error_result(SEQ_BAD_TOKEN, G)
    if any(not 0 <= int(parents[i]) < i for i in range(1, n_nodes)):
        return _error_result(SEQ_BAD_TREE, G)
    if not all(_valid_uniform(float(u_node[i])) for i in range(1, n_nodes)) or not _valid_uniform(float(u_sample)):
        return _error_result(SEQ_BAD_UNIFORM, G)
    if not valid_params(target_params) or not valid_params(draft_params):
        return _error_result(SEQ_BAD_PARAMS, G)
    children = [[c for c in range(1, n_nodes) if int(parents[c]) == v] for v in range(n_nodes)]
    # every node's target row; the draft row of every node with children (R10)
    p_rows, q_rows = [], []
    for v in range(n_nodes):
        p_v = transform_row(target[v], *target_params)
        if p_v.status != SEQ_OK:
            return _error_result(p_v.status, G)
        p_rows.append(p_v)
        q_v = transform_row(draft[v], *draft_params) if children[v] else None
        if q_v is not None and q_v.status != SEQ_OK:
            return _error_result(q_v.status, G)
        q_rows.append(q_v)

    status = SEQ_OK
    a = np.full(G, -1.0)
    trace = []
    accept_margin = np.inf
    draft_amb = False
    path = [0]
    v = 0
    r = p_rows[0].probs                    # the residual target distribution at v
    w, residual_Z = r, -1.0                # what the final token is drawn from, and its mass
    while True:
        q_v = q_rows[v]
        entered = None
        for c in children[v]:
            x = int(tokens[c])
            a_c, zq = acceptance_probability(r[x], q_v.probs[x])
            a[c - 1] = a_c
            trace.append((c, a_c))
            if zq:
                status |= SEQ_FLAG_ZERO_Q
            accept_margin = min(accept_margin, abs(float(u_node[c]) - a_c))
            draft_amb = draft_amb or x in p_rows[v].ambiguous or x in q_v.ambiguous
            if float(u_node[c]) < a_c:                     # R4
                entered = c
                break
            res_w = residual_weights(r, q_v.probs)         # [wrblog §5]
            Z = float(res_w.sum())
            if Z > 0:
                w, residual_Z = res_w, Z
                r = res_w / Z
            else:                                          # R7: keep r
                status |= SEQ_FLAG_Z_ZERO
                w, residual_Z = r, Z
        if entered is None:
            if not children[v]:                            # a leaf: the bonus from p_v [wrblog §6]
                w, residual_Z = p_rows[v].probs, -1.0
            break
        path.append(entered)
        v = entered
        r = p_rows[v].probs
    tok, lo, hi = inverse_cdf(w, float(u_sample))
    L = len(path) - 1
    out = np.full(max_nodes, -1, dtype=np.int64)
    out[:L] = [int(tokens[c]) for c in path[1:]]
    out[L] = tok
    used = [p_rows[u] for u in range(n_nodes)] + [q for q in q_rows if q is not None]
    sample_rows = [p_rows[v]] + ([q_rows[v]] if children[v] else [])
    res = SeqResult(out, L, status, a, residual_Z, accept_margin,
                    min([row.top_p_margin for row in used] + [np.inf]),
                    draft_ambiguous=draft_amb,
                    sample_ambiguous=np.unique(np.concatenate([row.ambiguous for row in sample_rows])),
                    sample_u=float(u_sample), sample_lo=lo, sample_hi=hi, num_emitted=L + 1)
    res.path = path
    res.tree_trace = trace
    C = np.cumsum(w)
    res.sample_cdf = C / C[-1]
    return res


def verify_sample_tree(target: np.ndarray, draft: np.ndarray, tokens: np.ndarray, parents: np.ndarray,
                       u_node: np.ndarray, u_sample: np.ndarray,
                       target_params: tuple[float, int, float], draft_params: tuple[float, int, float],
                       nodes_per_seq: np.ndarray | None = None) -> BatchResult:
    """Batched sampling-mode tree verification (R17), one sequence at a time."""
    B, N, _ = target.shape
    out = []
    for b in range(B):
        n = N if nodes_per_seq is None else int(nodes_per_seq[b])
        out.append(verify_sample_tree_sequence(target[b], draft[b], tokens[b], parents[b], u_node[b],
                                               float(u_sample[b]), n, N, target_params, draft_params))
    return _collect(out)


def verify_greedy_sequence_early(target: np.ndarray, tokens: np.ndarray, gamma_b: int,
                                 gamma_max: int) -> SeqResult:
    """Greedy verification that stops reading rows at the first mismatch (R11).

    [wrblog §6] verifies position by position and stops at the first rejection;
    [wrblog §7.1] makes the greedy test d_i == argmax p_i.  Row i is read only
    once d_1..d_{i-1} all matched, so rows after the stop point are never read
    and their contents cannot fail the sequence.
    """
    V = target.shape[1]
    if not 0 <= gamma_b <= gamma_max:
        return _error_result(SEQ_BAD_LENGTH, gamma_max)
    d = [int(t) for t in tokens[:gamma_b]]
    if any(not 0 <= t < V for t in d):
        return _error_result(SEQ_BAD_TOKEN, gamma_max)
    out = np.full(gamma_max + 1, -1, dtype=np.int64)
    for i in range(gamma_b + 1):
        gi, st = greedy_row(target[i])
        if st != SEQ_OK:
            res = _error_result(st, gamma_max)
            res.rows_read = i + 1
            return res
        if i == gamma_b or d[i] != gi:
            out[:i] = d[:i]
            out[i] = gi
            return SeqResult(out, i, SEQ_OK, np.full(gamma_max, -1.0), -1.0, rows_read=i + 1)
    raise AssertionError("unreachable: the loop returns at i == gamma_b")


# --------------------------------------------------------------------------
# Batches  [aiqz "加速收益与工程" -- requests verified together as one batch]
# --------------------------------------------------------------------------
@dataclass
class BatchResult:
    tokens: np.ndarray
    num_accepted: np.ndarray
    status: np.ndarray
    accept_prob: np.ndarray
    residual_Z: np.ndarray
    seqs: list


def _collect(results: list[SeqResult]) -> BatchResult:
    return BatchResult(np.stack([r.tokens for r in results]),
                       np.array([r.num_accepted for r in results], dtype=np.int64),
                       np.array([r.status for r in results], dtype=np.int64),
                       np.stack([r.accept_prob for r in results]) if results else np.zeros((0, 0)),
                       np.array([r.residual_Z for r in results]),
                       results)


def verify_sample(target: np.ndarray, draft: np.ndarray | None, tokens: np.ndarray,
                  u_accept: np.ndarray, u_sample: np.ndarray,
                  target_params: tuple[float, int, float], draft_params: tuple[float, int, float],
                  gamma_per_seq: np.ndarray | None = None, one_hot: np.ndarray | None = None,
                  seqs: list[int] | None = None, keep_cdf: bool = False,
                  lenience: float = 1.0, params_per_seq: list | None = None,
                  eos_token: int = -1, early_exit: bool = False) -> BatchResult:
    """Batched sampling verification, one sequence at a time.

    target (B, gamma_max+1, V), draft (B, gamma_max, V) or None (all one-hot),
    tokens / u_accept (B, gamma_max), u_sample (B,), all float64 / int.
    ``seqs`` restricts the work to a subset of sequence indices.
    ``params_per_seq``: per sequence b, the pair (target rule, draft rule)
    replacing target_params / draft_params (R13).  ``eos_token`` >= 0 cuts
    each committed block after its first end-of-sequence token (R14).
    ``early_exit`` reads each sequence's rows in position order and stops at
    the first failed row or rejected draft (R16).
    """
    B, G1, _ = target.shape
    gamma_max = G1 - 1
    seqs = range(B) if seqs is None else seqs
    out = []
    for b in seqs:
        g = gamma_max if gamma_per_seq is None else int(gamma_per_seq[b])
        oh = draft is None or (one_hot is not None and bool(one_hot[b]))
        tp, dp = (target_params, draft_params) if params_per_seq is None else params_per_seq[b]
        res = verify_sample_sequence(target[b], None if oh else draft[b], tokens[b],
                                     u_accept[b], float(u_sample[b]), tp, dp, g, gamma_max, oh,
                                     keep_cdf, lenience, early_exit)
        out.append(commit_at_eos(res, eos_token))
    return _collect(out)


def verify_greedy(target: np.ndarray, tokens: np.ndarray,
                  gamma_per_seq: np.ndarray | None = None,
                  seqs: list[int] | None = None) -> BatchResult:
    """Batched greedy verification, one sequence at a time."""
    B, G1, _ = target.shape
    gamma_max = G1 - 1
    seqs = range(B) if seqs is None else seqs
    out = []
    for b in seqs:
        g = gamma_max if gamma_per_seq is None else int(gamma_per_seq[b])
        out.append(verify_greedy_sequence(target[b], tokens[b], g, gamma_max))
    return _collect(out)


def verify_greedy_early(target: np.ndarray, tokens: np.ndarray,
                        gamma_per_seq: np.ndarray | None = None,
                        seqs: list[int] | None = None) -> BatchResult:
    """Batched early-exit greedy verification (R11), one sequence at a time."""
    B, G1, _ = target.shape
    gamma_max = G1 - 1
    seqs = range(B) if seqs is None else seqs
    out = []
    for b in seqs:
        g = gamma_max if gamma_per_seq is None else int(gamma_per_seq[b])
        out.append(verify_greedy_sequence_early(target[b], tokens[b], g, gamma_max))
    return _collect(out)


def transform_rows(z: np.ndarray, temperature: float, top_k: int, top_p: float) -> tuple[np.ndarray, np.ndarray]:
    """Row-wise transform of a (rows, V) logits array: returns (probs, top_p_margin)."""
    probs = np.zeros(z.shape)
    margins = np.full(z.shape[0], np.inf)
    for r in range(z.shape[0]):
        rd = transform_row(z[r], temperature, top_k, top_p)
        probs[r] = rd.probs
        margins[r] = rd.top_p_margin
    return probs, margins


def transform_rows_detail(z: np.ndarray, temperature: float, top_k: int, top_p: float) -> list[RowDist]:
    """Row-wise transform keeping every row's full RowDist (ambiguity diagnostics included)."""
    return [transform_row(z[r], temperature, top_k, top_p) for r in range(z.shape[0])]
