"""Float64 CPU oracle of the batched lossless speculative-decoding verify step.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the package's
``smoke()`` check and the benchmark's CPU-baseline leg may import this.  It
shares no code with the CUDA path; both are fed from the seeded generator in
``speculative_decoding_verification_47_gb300.workloads``.

Sources (pages cited by title and section):
  [SD]  "Speculative decoding, the founding scheme" (hotelren.com), §2.1-§2.2
  [SSD] "Self-speculative decoding with layer skip and KV reuse" (xdnf.cn),
        §2.4, §3.2, §3.3, §3.4, §4.3
  [FS]  "FlashSpec speculative decoding in practice" (nzsm.cn), §2.3, §3.2, §5.4

Notation: p = target distribution, q = draft distribution ([SD §2.1],
[SSD §2.4]; the FlashSpec page swaps the letters, we do not).

Readings of points the pages leave open:
  R2  accept iff u < min(1, p(x)/q(x)), strict '<' (the comparison operator is
      lost in the extracted code of [SSD §4.3]); with u < 1 this equals u < r.
  R3  q(x) = 0 gives ratio 0, i.e. rejection ([SSD §4.3] code).
  R4  residual fallback: if sum(max(0, p - q)) <= 0 draw from p ([SSD §4.3]).
  R5  inverse CDF in index order: y = min{v : C(v) > u * sum(w)} with C the
      inclusive prefix; zero-weight tokens can never be drawn.
  R6  top-p: order tokens by (p desc, index asc); keep v iff the mass strictly
      before v is <= top_p; renormalise over the kept set ([FS §3.2] code).
  R7  top-p is applied identically to target and draft; the variant with
      ``topp_draft=False`` truncates only the target and leaves the draft
      untruncated (the option [SSD §3.4] prefers; NEXT-4 reading R28).
  R8  temperature: exp((z - m) / T) with m the row max, same T both sides
      ([SSD §2.4], [FS §2.3]).
  R9  one uniform per tested position (column i), one for the single
      resample / bonus draw (column K).
  R10 KV commit: seq_len_new = seq_len + n_accepted ([SSD §3.3], §4.3).
  R11 greedy: argmax with the lowest index on ties.
  R12 greedy bonus: the target argmax at position k_b.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

SAMPLED = 0
GREEDY = 1

# Device-flag bits (same meaning as the C ABI's SV_FLAG_* values, restated).
FLAG_BAD_K = 1
FLAG_BAD_TOKEN = 2
FLAG_NONFINITE = 4
FLAG_BAD_TEMPERATURE = 8
FLAG_BAD_UNIFORM = 16
FLAG_BAD_MODE = 32
FLAG_CAPACITY = 64
FLAG_BAD_N = 256


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def stored_to_f64(a, dtype: str) -> np.ndarray:
    return bf16_bits_to_f64(a) if dtype == "bf16" else np.asarray(a, np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Per-distribution processing: temperature softmax and optional top-p
# ----------------------------------------------------------------------------

@dataclass
class Processed:
    """A processed (tempered, optionally truncated) distribution of one row."""

    p: np.ndarray            # final probabilities over V (float64)
    m: float                 # row max of the raw logits
    S: float                 # sum_v exp((z_v - m) / T)
    M: float                 # kept mass before renormalisation (1 without top-p)
    kept: np.ndarray | None  # boolean keep mask (None without top-p)
    cut_margin: float        # distance of the top-p cut from top_p (inf if none)


def temperature_softmax(z: np.ndarray, T: float):
    """softmax(z / T) written as exp((z - m)/T) / sum, m = max z  [SSD §2.4,
    FS §2.3].  Returns (p, m, S)."""
    m = float(np.max(z))
    e = np.exp((z - m) / T)
    S = math.fsum(e.tolist())
    return e / S, m, S


def top_p_mask(p: np.ndarray, top_p: float):
    """Nucleus truncation [FS §3.2]: sort by probability (descending; equal
    probabilities by ascending index), exclusive running mass, keep a token
    iff the mass ranked strictly before it is <= top_p.  Returns
    (kept mask, kept mass, margin of the cut)."""
    V = p.shape[0]
    order = np.lexsort((np.arange(V), -p))
    ps = p[order]
    c_incl = np.cumsum(ps)
    c_excl = c_incl - ps
    keep_sorted = c_excl <= top_p
    kept = np.zeros(V, dtype=bool)
    kept[order[keep_sorted]] = True
    M = math.fsum(ps[keep_sorted].tolist())
    last = int(np.count_nonzero(keep_sorted)) - 1  # kept set is a prefix
    margin = top_p - c_excl[last]
    if last + 1 < V:
        margin = min(margin, c_excl[last + 1] - top_p)
    return kept, M, float(margin)


def process_row(z: np.ndarray, T: float, top_p: float) -> Processed:
    """Temperature softmax then, if top_p < 1, top-p with renormalisation.
    The same function serves target and draft rows (reading R7)."""
    p, m, S = temperature_softmax(z, T)
    if top_p >= 1.0:
        return Processed(p=p, m=m, S=S, M=1.0, kept=None, cut_margin=math.inf)
    kept, M, margin = top_p_mask(p, top_p)
    pp = np.where(kept, p / M, 0.0)
    return Processed(p=pp, m=m, S=S, M=M, kept=kept, cut_margin=margin)


# ----------------------------------------------------------------------------
# Sampling primitives
# ----------------------------------------------------------------------------

def inverse_cdf(w: np.ndarray, u: float):
    """Draw from norm(w) with one uniform u in [0, 1): the smallest index v
    whose inclusive prefix C(v) exceeds u * sum(w) (reading R5).  Returns
    (token, margin) where margin = min(t - C(y-1), C(y) - t) / sum(w)."""
    C = np.cumsum(w)
    total = float(C[-1])
    t = u * total
    y = int(np.searchsorted(C, t, side="right"))
    y = min(y, w.shape[0] - 1)
    lo = float(C[y - 1]) if y > 0 else 0.0
    margin = min(t - lo, float(C[y]) - t) / total
    return y, margin


def residual_weights(p: np.ndarray, q: np.ndarray):
    """max(0, p - q) [SD §2.1, SSD §2.4]; when it sums to 0 (p == q, or
    rounding) fall back to p [SSD §4.3] (reading R4).  Returns (w, sum, used
    the fallback)."""
    w = np.maximum(0.0, p - q)
    Sw = math.fsum(w.tolist())
    if Sw <= 0.0:
        return p, Sw, True
    return w, Sw, False


# ----------------------------------------------------------------------------
# Per-sequence verify
# ----------------------------------------------------------------------------

@dataclass
class Decision:
    kind: str        # "accept", "resample", "bonus", "greedy", "topp"
    position: int
    margin: float    # distance of the deciding quantity from its threshold


@dataclass
class SeqResult:
    n: int                      # accepted draft tokens
    out: list                   # out tokens, length K+1, -1 padded
    flags: int = 0
    decisions: list = field(default_factory=list)
    # per-position diagnostics for rows actually used
    m_t: dict = field(default_factory=dict)
    S_t: dict = field(default_factory=dict)
    M_t: dict = field(default_factory=dict)
    m_d: dict = field(default_factory=dict)
    S_d: dict = field(default_factory=dict)
    M_d: dict = field(default_factory=dict)
    px: dict = field(default_factory=dict)   # p'(x_i)
    qx: dict = field(default_factory=dict)   # q'(x_i)
    ratio: dict = field(default_factory=dict)
    argmax: dict = field(default_factory=dict)
    S_w: float = math.nan                    # residual mass at the cut
    fallback: bool = False


def _error(K: int, flags: int, res: SeqResult | None = None) -> SeqResult:
    r = res if res is not None else SeqResult(n=0, out=[-1] * (K + 1))
    r.n = 0
    r.out = [-1] * (K + 1)
    r.flags |= flags
    return r


def _finite_row(z: np.ndarray) -> bool:
    """NaN and +inf are errors; -inf marks a token with zero probability.
    A row whose entries are all -inf cannot be normalised."""
    if np.isnan(z).any() or np.isposinf(z).any():
        return False
    return bool(np.isfinite(z).any())


def _uniform_ok(u: float) -> bool:
    return 0.0 <= u < 1.0


def verify_from_distributions(P, Q, x, k: int, u, K: int):
    """The accept / reject chain on already-processed distributions
    [SD §2.1-§2.2, SSD §4.3].

    P: k+1 target distributions, Q: k draft distributions, x: k draft tokens,
    u: K+1 uniforms (column i tests position i, column K is the single
    resample / bonus draw).  Returns (n, y, decisions)."""
    decisions = []
    for i in range(k):
        p, q = P[i], Q[i]
        qx = q[x[i]]
        r = p[x[i]] / qx if qx > 0.0 else 0.0
        decisions.append(Decision("accept", i, abs(float(u[i]) - r)))
        if not (u[i] < r):
            w, _, _ = residual_weights(p, q)
            y, mg = inverse_cdf(w, float(u[K]))
            decisions.append(Decision("resample", i, mg))
            return i, y, decisions
    y, mg = inverse_cdf(P[k], float(u[K]))
    decisions.append(Decision("bonus", k, mg))
    return k, y, decisions


def verify_sequence(zt_rows, zd_rows, x, k: int, K: int, V: int, T: float,
                    top_p: float, u, mode: int, topp_draft: bool = True) -> SeqResult:
    """Verify one sequence.  zt_rows: K+1 target logit rows (float64, only rows
    0..k are looked at), zd_rows: K draft rows, x: K draft tokens, u: K+1
    uniforms.  Rows, tokens and uniforms are examined lazily in position
    order, so a problem past the first rejection has no effect (the same
    early exit the rule itself has)."""
    res = SeqResult(n=0, out=[-1] * (K + 1))
    if not (0 <= k <= K):
        return _error(K, FLAG_BAD_K, res)
    if mode not in (SAMPLED, GREEDY):
        return _error(K, FLAG_BAD_MODE, res)

    if mode == GREEDY:
        # Greedy branch [SSD §2.4]: accept while the draft token equals the
        # target argmax; emit the target argmax at the first mismatch or as
        # the bonus (readings R11, R12).
        for i in range(k + 1):
            zt = zt_rows[i]
            if not _finite_row(zt):
                return _error(K, FLAG_NONFINITE, res)
            a = int(np.argmax(zt))
            res.argmax[i] = a
            res.m_t[i] = float(zt[a])
            if i == k:
                res.decisions.append(Decision("greedy", i, math.inf))
                res.n, y = k, a
                break
            if not (0 <= x[i] < V):
                return _error(K, FLAG_BAD_TOKEN, res)
            res.decisions.append(Decision("greedy", i, math.inf))
            if x[i] != a:
                res.n, y = i, a
                break
        res.out = [int(v) for v in x[: res.n]] + [y] + [-1] * (K - res.n)
        return res

    if not (T > 0.0 and math.isfinite(T)):
        return _error(K, FLAG_BAD_TEMPERATURE, res)

    def target(i):
        zt = zt_rows[i]
        if not _finite_row(zt):
            return None
        pr = process_row(zt, T, top_p)
        res.m_t[i], res.S_t[i], res.M_t[i] = pr.m, pr.S, pr.M
        if pr.kept is not None:
            res.decisions.append(Decision("topp", i, pr.cut_margin))
        return pr

    for i in range(k):
        if not (0 <= x[i] < V):
            return _error(K, FLAG_BAD_TOKEN, res)
        if not _uniform_ok(float(u[i])):
            return _error(K, FLAG_BAD_UNIFORM, res)
        pt = target(i)
        zd = zd_rows[i]
        if pt is None or not _finite_row(zd):
            return _error(K, FLAG_NONFINITE, res)
        qd = process_row(zd, T, top_p if topp_draft else 1.0)
        res.m_d[i], res.S_d[i], res.M_d[i] = qd.m, qd.S, qd.M
        if qd.kept is not None:
            res.decisions.append(Decision("topp", i, qd.cut_margin))
        p, q = pt.p, qd.p
        px, qx = float(p[x[i]]), float(q[x[i]])
        r = px / qx if qx > 0.0 else 0.0          # reading R3
        res.px[i], res.qx[i], res.ratio[i] = px, qx, r
        res.decisions.append(Decision("accept", i, abs(float(u[i]) - r)))
        if not (float(u[i]) < r):                  # reading R2
            if not _uniform_ok(float(u[K])):
                return _error(K, FLAG_BAD_UNIFORM, res)
            w, Sw, fb = residual_weights(p, q)
            y, mg = inverse_cdf(w, float(u[K]))
            res.S_w, res.fallback = Sw, fb
            res.decisions.append(Decision("resample", i, mg))
            res.n = i
            res.out = [int(v) for v in x[:i]] + [y] + [-1] * (K - i)
            return res

    # All k accepted: bonus token from p at position k [SD §2.2, SSD §4.3].
    if not _uniform_ok(float(u[K])):
        return _error(K, FLAG_BAD_UNIFORM, res)
    pt = target(k)
    if pt is None:
        return _error(K, FLAG_NONFINITE, res)
    y, mg = inverse_cdf(pt.p, float(u[K]))
    res.decisions.append(Decision("bonus", k, mg))
    res.n = k
    res.out = [int(v) for v in x[:k]] + [y] + [-1] * (K - k)
    return res


class _LazyRows:
    """Rows of one sequence, widened to float64 only when looked at."""

    def __init__(self, arr, dtype):
        self.arr, self.dtype = arr, dtype

    def __getitem__(self, i):
        return stored_to_f64(self.arr[i], self.dtype)


@dataclass
class BatchResult:
    out_tokens: np.ndarray   # [B, K+1] int32
    n_accepted: np.ndarray   # [B] int32
    flags: int
    seqs: list


def spec_verify(target, draft, dtype: str, B: int, K: int, V: int, draft_tokens,
                k_per_row, temperature, top_p: float, uniforms, mode,
                rows=None, topp_draft: bool = True) -> BatchResult:
    """Batched verify: every sequence independently (reading R9 for the
    uniform layout).  ``target`` [B, K+1, V] and ``draft`` [B, K, V] hold the
    stored logits (bf16 bit patterns or float32).  ``rows`` optionally
    restricts the work to a subset of sequence indices (the others are
    returned as -1 / 0 and excluded from ``seqs``)."""
    out = np.full((B, K + 1), -1, dtype=np.int32)
    n = np.zeros(B, dtype=np.int32)
    flags = 0
    seqs = []
    kpr = np.full(B, K, np.int32) if k_per_row is None else np.asarray(k_per_row)
    sel = range(B) if rows is None else rows
    for b in sel:
        k = int(kpr[b])
        zt = _LazyRows(target[b], dtype)
        zd = _LazyRows(draft[b], dtype) if draft is not None else None
        r = verify_sequence(zt, zd, np.asarray(draft_tokens[b]), k, K, V,
                            float(temperature[b]), float(top_p),
                            np.asarray(uniforms[b], dtype=np.float64), int(mode[b]),
                            topp_draft=topp_draft)
        out[b] = r.out
        n[b] = r.n
        flags |= r.flags
        seqs.append((b, r))
    return BatchResult(out_tokens=out, n_accepted=n, flags=flags, seqs=seqs)


def kv_commit(seq_lens, n_accepted, capacity=None, K: int | None = None, k_per_row=None):
    """KV write-pointer rollback [SSD §3.3, §4.3; SD §4.3]: each sequence's
    pointer, which stood at the round-start length while the drafts were
    written speculatively, moves to seq_len + n_accepted; entries at and
    beyond it are discarded (reading R10).  A row that would pass its
    capacity, or whose n is negative (or above K when K is given, or above
    the round's k_b when k_per_row is given: more tokens accepted than
    drafted), is left unchanged and flagged.  Returns (new seq_lens, flags)."""
    s = np.asarray(seq_lens, dtype=np.int64).copy()
    flags = 0
    for b in range(s.shape[0]):
        nb = int(n_accepted[b])
        if nb < 0 or (K is not None and nb > K) or (k_per_row is not None and nb > int(k_per_row[b])):
            flags |= FLAG_BAD_N
            continue
        new = int(s[b]) + nb
        if capacity is not None and new > int(capacity[b]):
            flags |= FLAG_CAPACITY
            continue
        s[b] = new
    return s.astype(np.int32), flags
