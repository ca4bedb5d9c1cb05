"""Seeded synthetic workloads for the batched speculative-decoding verify step.

This module only draws inputs: logits, draft tokens, per-row knobs and the
uniform random numbers the verify rule consumes.  It holds none of the verify
arithmetic (no softmax normalisation, no acceptance test, no residual, no
top-p), so the CUDA path and the float64 oracle can both be fed from it
without sharing any of the method's steps.

Recipe (all NumPy PCG64; one child stream per sequence so generation can run
on a thread pool and any single sequence can be regenerated on its own):

* Target logits at every position: z_v = 2.0 * N(0,1) - 1.1 * ln(rank_v).
  ``rank`` is a per-sequence random permutation of 1..V (a Zipf(1.1) log-prior
  over a shuffled vocabulary), shared by all positions and both models.
* Draft logits at position i: the target row at i plus N(0, sigma_b^2) noise.
* Storage: bf16 (round-to-nearest-even via float32, as torch does) or float32.
* Draft tokens: sampled rows draw x_i from softmax(z_draft/T_b) with the
  Gumbel-max construction argmax_v(z_v/T + G_v); greedy rows take the draft
  argmax.  Gumbel-max is an independent way to draw from a softmax; the
  verify rule's own inverse-CDF draw is not used here.  When top-p is active,
  sampled rows still draw from the untruncated tempered draft softmax, so
  roughly (1 - kept mass) of the draws fall outside the draft's nucleus.
* Uniforms: integers in [0, 2^24) times 2^-24, exact in float32 and float64.
* Padding (positions at or beyond a row's k_b) is filled with canaries: NaN
  logits, token -1 and NaN uniforms.  A kernel that reads a padded slot
  trips its own input checks.

The pages' workloads (7B-class vocabularies 32000 / 128256 / 151936, k in
2..8, batched rows) are stood in for by these draws; no dataset item is used.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BF16 = "bf16"
F32 = "f32"

SAMPLED = 0
GREEDY = 1

BF16_NAN = np.uint16(0x7FC0)


# ----------------------------------------------------------------------------
# bf16 storage helpers (bit-level, no arithmetic of the method)
# ----------------------------------------------------------------------------

def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 bit patterns (uint16): first to float32
    (IEEE round-to-nearest-even), then RNE on the top 16 bits."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) >> 16
    out = u.astype(np.uint16)
    out[nan] = BF16_NAN
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# Workload description
# ----------------------------------------------------------------------------

@dataclass
class VerifyInputs:
    """One batch of verify inputs, laid out exactly as the C ABI reads them.

    target   [B, K+1, V]  uint16 (bf16 bits) or float32
    draft    [B, K, V]    same dtype
    draft_tokens [B, K]   int32 (-1 in padding)
    k_per_row    [B]      int32
    temperature  [B]      float32
    top_p        float
    uniforms [B, K+1]     float32; column i < k_b is the test of position i,
                          column K is the single resample / bonus draw
    mode     [B]          uint8 (0 sampled, 1 greedy)
    """

    name: str
    dtype: str
    B: int
    K: int
    V: int
    target: np.ndarray
    draft: np.ndarray
    draft_tokens: np.ndarray
    k_per_row: np.ndarray
    temperature: np.ndarray
    top_p: float
    uniforms: np.ndarray
    mode: np.ndarray
    sigma: np.ndarray
    seq_lens: np.ndarray | None = None
    capacity: np.ndarray | None = None
    meta: dict = field(default_factory=dict)

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == BF16 else 4

    def logits_f32(self, which: str) -> np.ndarray:
        """float32 view of the stored logits (exact widening for bf16)."""
        a = self.target if which == "target" else self.draft
        return bf16_bits_to_f32(a) if self.dtype == BF16 else a


def _stored(x: np.ndarray, dtype: str) -> np.ndarray:
    return f64_to_bf16_bits(x) if dtype == BF16 else x.astype(np.float32)


def _decoded(stored: np.ndarray, dtype: str) -> np.ndarray:
    return (bf16_bits_to_f32(stored) if dtype == BF16 else stored).astype(np.float64)


def gumbel_draft_token(z_draft: np.ndarray, T: float, rng: np.random.Generator) -> int:
    """Draw one token from softmax(z/T) by Gumbel-max: argmax(z/T + G)."""
    u = rng.random(z_draft.shape[0])
    # G = -log(-log U); U = 0 has probability 2^-53 and maps to -inf, harmless.
    with np.errstate(divide="ignore"):
        g = -np.log(-np.log(u))
    return int(np.argmax(z_draft / T + g))


def _gen_sequence(b, B, K, V, dtype, k_b, T_b, sigma_b, mode_b, seeds, draft_scale=1.0):
    logit_seed, token_seed, uniform_seed = seeds
    rl = np.random.Generator(np.random.PCG64(np.random.SeedSequence([logit_seed, b])))
    rt = np.random.Generator(np.random.PCG64(np.random.SeedSequence([token_seed, b])))
    ru = np.random.Generator(np.random.PCG64(np.random.SeedSequence([uniform_seed, b])))

    rank = rl.permutation(V).astype(np.float64) + 1.0
    prior = -1.1 * np.log(rank)

    tgt = np.empty((K + 1, V), dtype=np.uint16 if dtype == BF16 else np.float32)
    drf = np.empty((K, V), dtype=tgt.dtype)
    toks = np.full((K,), -1, dtype=np.int32)
    nan = BF16_NAN if dtype == BF16 else np.float32(np.nan)

    for i in range(K + 1):
        zt = 2.0 * rl.standard_normal(V) + prior
        if i <= k_b:
            tgt[i] = _stored(zt, dtype)
        else:
            tgt[i] = nan
        if i < K:
            zd = (zt if draft_scale == 1.0 else draft_scale * zt) + sigma_b * rl.standard_normal(V)
            if i < k_b:
                drf[i] = _stored(zd, dtype)
                zd_dec = _decoded(drf[i], dtype)
                if mode_b == GREEDY:
                    toks[i] = int(np.argmax(zd_dec))
                else:
                    toks[i] = gumbel_draft_token(zd_dec, T_b, rt)
            else:
                drf[i] = nan

    ui = ru.integers(0, 1 << 24, size=K + 1)
    u = (ui.astype(np.float64) * 2.0 ** -24).astype(np.float32)
    u[k_b:K] = np.nan
    return tgt, drf, toks, u


def synth_verify(
    name: str,
    B: int,
    K: int,
    V: int,
    dtype: str,
    k_per_row,
    temperature,
    sigma,
    mode,
    top_p: float = 1.0,
    seeds=(1000, 2000, 0),
    threads: int | None = None,
    draft_scale: float = 1.0,
) -> VerifyInputs:
    """Draw a verify batch.  ``k_per_row``, ``temperature``, ``sigma`` and
    ``mode`` are per-row arrays (or scalars broadcast over B).  ``top_p`` is
    kept as the float32 value the verify call receives, so that the oracle
    and the library cut at the same threshold.  ``draft_scale`` multiplies the
    target logits before the draft noise is added (1 = the plain recipe; below 1
    an under-confident draft)."""
    k_per_row = np.broadcast_to(np.asarray(k_per_row, dtype=np.int32), (B,)).copy()
    temperature = np.broadcast_to(np.asarray(temperature, dtype=np.float32), (B,)).copy()
    sigma = np.broadcast_to(np.asarray(sigma, dtype=np.float64), (B,)).copy()
    mode = np.broadcast_to(np.asarray(mode, dtype=np.uint8), (B,)).copy()

    sdt = np.uint16 if dtype == BF16 else np.float32
    target = np.empty((B, K + 1, V), dtype=sdt)
    draft = np.empty((B, K, V), dtype=sdt)
    tokens = np.empty((B, K), dtype=np.int32)
    uniforms = np.empty((B, K + 1), dtype=np.float32)

    def work(b):
        t, d, x, u = _gen_sequence(b, B, K, V, dtype, int(k_per_row[b]),
                                   float(temperature[b]), float(sigma[b]),
                                   int(mode[b]), seeds, draft_scale)
        target[b], draft[b], tokens[b], uniforms[b] = t, d, x, u

    nthreads = threads or min(16, os.cpu_count() or 1)
    if B * K * V < (1 << 20) or nthreads == 1:
        for b in range(B):
            work(b)
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(work, range(B)))

    return VerifyInputs(name=name, dtype=dtype, B=B, K=K, V=V, target=target,
                        draft=draft, draft_tokens=tokens, k_per_row=k_per_row,
                        temperature=temperature, top_p=float(np.float32(top_p)),
                        uniforms=uniforms, mode=mode, sigma=sigma)


# ----------------------------------------------------------------------------
# The five named workloads
# ----------------------------------------------------------------------------

CONFIG_NAMES = ("c0", "c1", "c2", "c3", "c4")


def config_c0(round_index: int = 0, V: int = 32000) -> VerifyInputs:
    """B=1, k=4, V=32000, fp32; draft noise 0.5; T=1; sampled.  One of 64
    independent rounds, selected by ``round_index`` (sequence index of the
    per-sequence streams)."""
    # Each round is sequence ``round_index`` of a 64-sequence draw, so the 64
    # rounds together equal ``config_c0_batched``.
    b = round_index
    t, d, x, u = _gen_sequence(b, 64, 4, V, F32, 4, 1.0, 0.5, SAMPLED, (1000, 2000, 0))
    return VerifyInputs(name=f"c0.r{b}", dtype=F32, B=1, K=4, V=V,
                        target=t[None], draft=d[None], draft_tokens=x[None],
                        k_per_row=np.array([4], np.int32),
                        temperature=np.array([1.0], np.float32), top_p=1.0,
                        uniforms=u[None], mode=np.zeros(1, np.uint8),
                        sigma=np.array([0.5]))


def config_c0_batched(rounds: int = 64, V: int = 32000) -> VerifyInputs:
    """The 64 rounds of c0 stacked as one B=64 batch (same draws as
    ``config_c0(r)`` for r in range(rounds))."""
    return synth_verify("c0x64", rounds, 4, V, F32, 4, 1.0, 0.5, SAMPLED,
                        seeds=(1000, 2000, 0))


@dataclass
class RowSpec:
    """Everything needed to regenerate any single sequence of a named batch
    workload with ``_gen_sequence`` (per-sequence random streams)."""

    name: str
    B: int
    K: int
    V: int
    dtype: str
    k_per_row: np.ndarray
    temperature: np.ndarray
    sigma: np.ndarray
    mode: np.ndarray
    top_p: float
    seeds: tuple

    def sequence(self, b: int):
        return _gen_sequence(b, self.B, self.K, self.V, self.dtype, int(self.k_per_row[b]),
                             float(self.temperature[b]), float(self.sigma[b]),
                             int(self.mode[b]), self.seeds)


def row_spec(name: str, B: int | None = None) -> RowSpec:
    """Row parameters of the batch workloads c1, c2, c3."""
    def full(v, n, dt):
        return np.broadcast_to(np.asarray(v, dtype=dt), (n,)).copy()

    if name == "c1":
        B = B or 64
        return RowSpec("c1", B, 5, 32000, BF16, full(5, B, np.int32), full(0.8, B, np.float32),
                       full(1.0, B, np.float64), full(SAMPLED, B, np.uint8), 1.0,
                       (1001, 2001, 1))
    if name == "c2":
        B = B or 256
        k, T, sg = c2_row_params(B)
        return RowSpec("c2", B, 8, 128256, BF16, k, T, sg, full(SAMPLED, B, np.uint8), 1.0,
                       (1002, 2002, 2))
    if name == "c3":
        B = B or 128
        mode = np.where(np.arange(B) < B // 2, GREEDY, SAMPLED).astype(np.uint8)
        return RowSpec("c3", B, 6, 151936, BF16, full(6, B, np.int32), full(0.7, B, np.float32),
                       full(0.5, B, np.float64), mode, float(np.float32(0.9)), (1003, 2003, 3))
    raise ValueError(f"no row spec for workload {name!r}")


def config_by_name(name: str, B: int | None = None) -> VerifyInputs:
    return {"c1": config_c1, "c2": config_c2, "c3": config_c3}[name](**({"B": B} if B else {}))


def config_c1(B: int = 64, V: int = 32000) -> VerifyInputs:
    """B=64, k=5, V=32000, bf16, draft noise 1.0, T=0.8, sampled; seq_lens
    ~U[128, 4096] for the KV write-pointer commit."""
    w = synth_verify("c1", B, 5, V, BF16, 5, 0.8, 1.0, SAMPLED, seeds=(1001, 2001, 1))
    r = np.random.Generator(np.random.PCG64(3001))
    w.seq_lens = r.integers(128, 4097, size=B).astype(np.int32)
    w.capacity = np.full(B, 4096 + 64, dtype=np.int32)
    return w


def c2_row_params(B: int = 256):
    """Per-row k_b ~ U{2..8}, T_b in {0.1, 0.7, 1.0}, sigma_b in {0.3, 1, 2}."""
    r = np.random.Generator(np.random.PCG64(4000))
    k = r.integers(2, 9, size=B).astype(np.int32)
    T = r.choice(np.array([0.1, 0.7, 1.0], dtype=np.float32), size=B)
    s = r.choice(np.array([0.3, 1.0, 2.0]), size=B)
    return k, T, s


def config_c2(B: int = 256, V: int = 128256) -> VerifyInputs:
    """B=256, K=8, V=128256, bf16, ragged k_b in 2..8, per-row temperature
    and draft noise; sampled."""
    k, T, s = c2_row_params(B)
    w = synth_verify("c2", B, 8, V, BF16, k, T, s, SAMPLED, seeds=(1002, 2002, 2))
    r = np.random.Generator(np.random.PCG64(3002))
    w.seq_lens = r.integers(128, 4097, size=B).astype(np.int32)
    w.capacity = np.full(B, 4096 + 64, dtype=np.int32)
    return w


def config_c3(B: int = 128, V: int = 151936) -> VerifyInputs:
    """B=128, k=6, V=151936, bf16, T=0.7, top_p=0.9 on both sides; rows
    0..B/2-1 greedy, the rest sampled; draft noise 0.5."""
    mode = np.where(np.arange(B) < B // 2, GREEDY, SAMPLED).astype(np.uint8)
    w = synth_verify("c3", B, 6, V, BF16, 6, 0.7, 0.5, mode, top_p=0.9,
                     seeds=(1003, 2003, 3))
    r = np.random.Generator(np.random.PCG64(3003))
    w.seq_lens = r.integers(128, 4097, size=B).astype(np.int32)
    w.capacity = np.full(B, 4096 + 64, dtype=np.int32)
    return w


@dataclass
class LMHeadInputs:
    """Layer-skip draft-logit producer inputs (bf16 bit patterns).

    hidden   [M, H]  layer-L hidden states ~ N(0, 1)
    hidden_t [M, H]  hidden + N(0, 0.5^2): a stand-in for the remaining
                     layers, so that target and draft logits differ
    norm_w   [H]     final RMSNorm weight ~ 1 + N(0, 0.02^2)
    W        [H, V]  LM head ~ N(0, 0.02^2), row-major (V contiguous)
    """

    M: int
    H: int
    V: int
    eps: float
    hidden: np.ndarray
    hidden_t: np.ndarray
    norm_w: np.ndarray
    W: np.ndarray


def lmhead_inputs(M: int = 512, H: int = 4096, V: int = 32000, seed: int = 1004,
                  hidden_scale: float = 1.0) -> LMHeadInputs:
    r = np.random.Generator(np.random.PCG64(seed))
    h = hidden_scale * r.standard_normal((M, H))
    ht = h + 0.5 * r.standard_normal((M, H))
    w = 1.0 + 0.02 * r.standard_normal(H)
    W = 0.02 * r.standard_normal((H, V))
    return LMHeadInputs(M=M, H=H, V=V, eps=1e-5, hidden=f64_to_bf16_bits(h),
                        hidden_t=f64_to_bf16_bits(ht), norm_w=f64_to_bf16_bits(w),
                        W=f64_to_bf16_bits(W))


def c4_verify_knobs(B: int = 64, K: int = 7, seed: int = 4):
    """Per-row knobs and uniforms for the verify step of the layer-skip
    workload (B=64, k=7, T=1, sampled).  Draft tokens are drawn later from
    whatever draft logits the caller produced (``gumbel_draft_token``)."""
    ru = np.random.Generator(np.random.PCG64(seed))
    u = (ru.integers(0, 1 << 24, size=(B, K + 1)).astype(np.float64) * 2.0 ** -24
         ).astype(np.float32)
    return dict(k_per_row=np.full(B, K, np.int32),
                temperature=np.ones(B, np.float32),
                mode=np.zeros(B, np.uint8), uniforms=u)


def draw_draft_tokens(draft_stored: np.ndarray, dtype: str, k_per_row, temperature,
                      mode, seed: int) -> np.ndarray:
    """Draft tokens for already-computed draft logits [B, K(+), V]: Gumbel-max
    for sampled rows, argmax for greedy rows, -1 in padding."""
    B, K = draft_stored.shape[0], draft_stored.shape[1]
    out = np.full((B, K), -1, dtype=np.int32)
    for b in range(B):
        r = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, b])))
        for i in range(int(k_per_row[b])):
            z = _decoded(draft_stored[b, i], dtype)
            out[b, i] = (int(np.argmax(z)) if int(mode[b]) == GREEDY
                         else gumbel_draft_token(z, float(temperature[b]), r))
    return out


# ----------------------------------------------------------------------------
# Round bookkeeping around the verify step: paged KV cache, dynamic k
# ----------------------------------------------------------------------------

@dataclass
class PagedRound:
    """One round's paged-KV state before the commit: sequence b holds
    seq_lens[b] committed tokens, its k_per_row[b] drafts were written after
    them, and block_table[b] lists the pages that cover all of those tokens
    (-1 past them); n_accepted[b] in [0, k_b] came back from verification."""
    seq_lens: np.ndarray
    n_accepted: np.ndarray
    k_per_row: np.ndarray
    block_table: np.ndarray
    page_size: int
    pool_pages: int


def paged_round(B: int = 1024, max_pages: int = 64, page_size: int = 16,
                seed: int = 4100) -> PagedRound:
    """Lengths ~U[100, max_pages*page_size/2), k_b ~U{2..8}, n_b ~U{0..k_b};
    page ids drawn without replacement from a pool of B*max_pages pages."""
    r = np.random.Generator(np.random.PCG64(seed))
    L = r.integers(100, max_pages * page_size // 2, size=B).astype(np.int32)
    k = r.integers(2, 9, size=B).astype(np.int32)
    n = np.array([r.integers(0, kb + 1) for kb in k], dtype=np.int32)
    ids = r.permutation(B * max_pages).astype(np.int32)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    for b in range(B):
        used = -(-(int(L[b]) + int(k[b])) // page_size)
        table[b, :used] = ids[b * max_pages: b * max_pages + used]
    return PagedRound(L, n, k, table, page_size, B * max_pages)


def dynk_history(B: int = 256, rounds: int = 64, seed: int = 4200):
    """A history of rounds for B controllers: k_used ~U{2..8} and
    n_accepted ~U{0..k_used} per (round, sequence), as int32
    [rounds, B] arrays."""
    r = np.random.Generator(np.random.PCG64(seed))
    k = r.integers(2, 9, size=(rounds, B)).astype(np.int32)
    n = (r.uniform(size=(rounds, B)) * (k + 1)).astype(np.int32)
    return n, k
