"""Float64 CPU oracle of the draft-side sampler: the k_b draft tokens of each
sequence drawn from already-computed draft logits, with the same temperature
and top-p processing the verify step applies.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the package's
``smoke()`` check and the benchmark's CPU-baseline leg may import this.  It
shares no code with the CUDA path.

Sources (pages cited by title and section):
  [FS]  "FlashSpec speculative decoding in practice" (nzsm.cn), §3.2: the
        draft stage samples each of its k tokens from the temperature softmax
        of its logits after top-p truncation, one position after another.
  [SSD] "Self-speculative decoding with layer skip and KV reuse" (xdnf.cn),
        §3.2, §4.2: the layer-skip draft produces k candidates the same way.

Readings (the points the pages leave open, and the reading taken):
  R22 one uniform per sampled position (column i of a [B, K] array); the token
      is the verify step's inverse CDF in index order (R5) over the processed
      row p' (R6, R8); greedy rows take the argmax, lowest index on ties (R11).
  R23 positions i >= k_b are padding (-1).  A bad k_b, mode or temperature
      gives -1 at every position of the sequence and its flag; a non-finite
      row or a uniform outside [0, 1) gives -1 at that position and its flag.
      Rows are independent: an error at one position does not stop the others
      (each draft step has its own logits).
"""

from __future__ import annotations

import math

import numpy as np

from oracle import verify as ov


def sample_row(z: np.ndarray, T: float, top_p: float, u: float, greedy: bool):
    """One token from one row of logits.  Returns (token, margin, flags);
    margin is the inverse-CDF margin of R13 (inf for greedy rows)."""
    if not ov._finite_row(z):  # NaN, +inf, or every logit -inf
        return -1, math.inf, ov.FLAG_NONFINITE
    if greedy:
        return int(np.argmax(z)), math.inf, 0
    if not (0.0 <= u < 1.0):
        return -1, math.inf, ov.FLAG_BAD_UNIFORM
    pr = ov.process_row(z, T, top_p)
    y, margin = ov.inverse_cdf(pr.p, u)
    return y, min(margin, pr.cut_margin), 0


def sample_tokens(logits, dtype: str, B: int, K: int, V: int, k_per_row, temperature,
                  top_p: float, uniforms, mode):
    """Draft tokens for a [B, K, V] block of stored logits.  Returns
    (tokens [B, K] int32, margins [B, K] float64, flags)."""
    tokens = np.full((B, K), -1, dtype=np.int32)
    margins = np.full((B, K), math.inf)
    flags = 0
    for b in range(B):
        k = int(k_per_row[b]) if k_per_row is not None else K
        md = int(mode[b]) if mode is not None else ov.SAMPLED
        T = float(temperature[b]) if temperature is not None else 1.0
        if not (0 <= k <= K):
            flags |= ov.FLAG_BAD_K
            continue
        if md not in (ov.SAMPLED, ov.GREEDY):
            flags |= ov.FLAG_BAD_MODE
            continue
        if md == ov.SAMPLED and not (T > 0.0 and math.isfinite(T)):
            flags |= ov.FLAG_BAD_TEMPERATURE
            continue
        for i in range(k):
            z = ov.stored_to_f64(logits[b, i], dtype)
            y, mg, f = sample_row(z, T, top_p, float(uniforms[b, i]), md == ov.GREEDY)
            tokens[b, i] = y
            margins[b, i] = mg
            flags |= f
    return tokens, margins, flags
