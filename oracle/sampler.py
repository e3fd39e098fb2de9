"""Binary64 CPU oracle for the per-row vocabulary sampling stage.

TEST INFRASTRUCTURE. Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import or run this module. It shares no code with the CUDA path (no kernels, headers, helpers or
constants) and never consumes anything the CUDA path produced.

Sources (page title -- section):

* [TOPP] "Split top-p numerical reference and conservative gate" -- "Independent binary64 numerical
  reference" (steps 1-6) and "Source basis" (probability-space mask, row maximum always kept,
  cumulative low-tail mask with the at-least-one-token rule).
* [GUMBEL] "[vLLM PR #45996] use log1p(-u) to improve FP32 Gumbel sampling precision" -- the
  implementation breakdown and the key source snippet: noise g = -log(-log1p(-u)), masked
  logits + g, arg-max that returns the lowest index among equal maxima; temperature 0 returns the
  arg-max.
* [TOPK] "[Kernel] Make persistent_topk deterministic" -- "Changes": exact top-k by (value descending,
  index ascending), output in ascending index order, -0.0 and +0.0 are the same key, unused output
  slots padded with -1.
* [LOGP] "[WS2][Logprob] Deterministic SM90 linear_logp ..." -- "Design: the numeric contract":
  m = max, S = sum exp(z - m), lse = m + log S, logp = min(z_t - lse, 0), temperature applied to the
  statistics rather than to stored logits; "Integration": transform order temperature -> top-k ->
  top-p -> min-p.
* [MINP] "Sorting-free top-k/top-p/min-p sampling with dual-pivot rejection kernels #901" --
  "Background": min-p pivot = max * p.

Readings where the pages are silent or leave a step open (the plainest one the rest supports):

* top-p is taken over the top-k-renormalised distribution (sequential transforms), target = p * S_k;
* min-p keeps v iff p_v >= min_p * p_max, i.e. exp(s_v) >= min_p on temperature-scaled weights;
* u = (b + 0.5) * 2^-32 for the 32-bit Philox word b, which is exact in binary64 and never 0 or 1;
* the perturbed score is s_v + g_v with s_v = (x_v - m) / T (max-subtracted);
* temperature <= 0 is greedy (the lowest-index maximum) and every filter then keeps one token; the
  reported log-probability then uses T = 1;
* the log-probability is over the full vocabulary at temperature T (not the filtered distribution).

Every function here is pinned by tests/test_oracle_pins.py (brute force on tiny rows with exact
rational arithmetic, closed forms, invariants, the published Philox known-answer vectors and a
chi-square test of the sampling law).
"""
from __future__ import annotations

import math
import struct
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

from .philox import token_words

STATUS_OK = 0
STATUS_INVALID_ARG = 1
STATUS_NONFINITE = 4

BAND_REL = 1e-6          # top-p / min-p exemption band, relative to S_k (resp. min_p)
TIE_REL = 1e-6           # near-tie draws: top-two perturbed scores closer than this, relative


def widen(row, dtype: str) -> np.ndarray:
    """Exact widening of stored logits to binary64 ([TOPP] step 1: keep the original values)."""
    if dtype == "bf16":
        bits = np.asarray(row, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    return np.asarray(row, dtype=np.float32).astype(np.float64)


def as_f32(v) -> float:
    """A runtime parameter as its fp32 value ([TOPP] step 1: p after fp32 conversion)."""
    return float(np.float32(v))


def order_key(value: float) -> int:
    """Order-preserving 32-bit key of an fp32 value; -0.0 and +0.0 share one key ([TOPK] Changes).

    Positive floats get the sign bit set, negative floats are bit-inverted, so unsigned key order is
    float order.
    """
    bits = struct.unpack("<I", struct.pack("<f", float(value)))[0]
    if bits == 0x80000000:
        bits = 0
    return (bits | 0x80000000) if (bits >> 31) == 0 else (~bits) & 0xFFFFFFFF


def canonical_order(x: np.ndarray) -> np.ndarray:
    """pi: token indices by (logit descending, token id ascending) -- [TOPP] step 2.

    A stable sort of -x keeps equal logits (including -0.0 == +0.0) in index order.
    """
    return np.argsort(-x, kind="stable")


def neumaier_scan(weights: np.ndarray, target: float) -> int:
    """Smallest count c whose compensated prefix sum reaches target ([TOPP] step 5); len if none.

    The test is (total - target) + comp >= 0 rather than total + comp >= target: near the crossing
    total - target is exact (Sterbenz), so the comparison is not lost to the rounding of the sum.
    """
    total = 0.0
    comp = 0.0
    for i, wi in enumerate(weights.tolist()):
        t = total + wi
        if abs(total) >= abs(wi):
            comp += (total - t) + wi
        else:
            comp += (wi - t) + total
        total = t
        if (total - target) + comp >= 0.0:
            return i + 1
    return len(weights)


def nucleus_count(weights_sorted: np.ndarray, target: float):
    """[TOPP] steps 5-6: scan, then certify the boundary with two math.fsum checks.

    Returns (count, ambiguous). ``ambiguous`` is the oracle_boundary_ambiguous flag: the compensated
    scan and the fsum certificate disagree (never tuned against; the parity band covers it).
    """
    c = neumaier_scan(weights_sorted, target)
    hi = math.fsum(weights_sorted[:c].tolist())
    lo = math.fsum(weights_sorted[:c - 1].tolist()) if c > 1 else 0.0
    ok = hi >= target and lo < target
    return c, (not ok)


@dataclass
class RowResult:
    status: int = STATUS_OK
    row_max: float = float("nan")       # m, the fp32 row maximum
    row_logsum: float = float("nan")    # log sum_v exp((x_v - m) / T) over the full row
    n: int = 0
    top_k_count: int = 0                # |K|
    kept: int = 0                       # final kept prefix length of pi
    kept_lo: int = 0                    # kept counts allowed by the 1e-6 band
    kept_hi: int = 0
    pivot_key: int = 0                  # key of the last kept token
    idx_cut: int = -1                   # index of the last kept token
    ambiguous: bool = False
    token: int = -1
    logprob: float = float("nan")
    best: float = float("nan")          # winning perturbed score
    second: float = float("nan")        # runner-up perturbed score (nan if one candidate)
    near_tie: bool = False
    order: Optional[np.ndarray] = field(default=None, repr=False)
    s: Optional[np.ndarray] = field(default=None, repr=False)


def _count_band(sorted_vals: np.ndarray, lo_thr: float, hi_thr: float):
    """Counts of a non-increasing sequence above lo_thr (strict) and at or above hi_thr."""
    return int(np.count_nonzero(sorted_vals > lo_thr)), int(np.count_nonzero(sorted_vals >= hi_thr))


def uniform_from_word(b) -> np.ndarray:
    """u = (b + 0.5) * 2^-32: the midpoint of the b-th of 2^32 equal cells, exact in binary64.

    It never returns 0 or 1, so no clamp is needed (the Gumbel precision page clamps its uniform at
    its smallest positive value instead).
    """
    return (np.asarray(b, dtype=np.float64) + 0.5) * 2.0 ** -32


def gumbel_from_uniform(u) -> np.ndarray:
    """g = -log(-log1p(-u)) ([GUMBEL]); P(G <= g) = exp(-exp(-g)) = 1 - u."""
    return -np.log(-np.log1p(-np.asarray(u, dtype=np.float64)))


def gumbel_scores(s: np.ndarray, cand: np.ndarray, seed: int, row_id: int, step) -> np.ndarray:
    """Perturbed scores s_v + g_v for the candidate tokens ([GUMBEL]); ``step`` scalar or 1-D."""
    u = uniform_from_word(token_words(cand, seed, row_id, step))
    return s[cand] + gumbel_from_uniform(u)


def argmax_lowest(scores: np.ndarray, cand: np.ndarray) -> np.ndarray:
    """Arg-max over the last axis of ``scores`` (aligned with ``cand``); equal maxima -> lowest index."""
    scores = np.atleast_2d(scores)
    best = scores.max(axis=1, keepdims=True)
    idx = np.where(scores == best, np.asarray(cand).reshape(1, -1), np.iinfo(np.int64).max)
    return idx.min(axis=1)


def draw_many(s: np.ndarray, cand: np.ndarray, seed: int, row_id: int, steps) -> np.ndarray:
    """Tokens drawn at each of ``steps`` (1-D) over the candidate set."""
    sc = gumbel_scores(s, cand, seed, row_id, np.asarray(steps, dtype=np.uint64).reshape(-1))  # [S, N]
    return argmax_lowest(sc, cand)


def draw(s: np.ndarray, cand: np.ndarray, seed: int, row_id: int, step: int):
    """(token, best score, runner-up score) of one draw over ``cand``."""
    sc = gumbel_scores(s, cand, seed, row_id, step)
    token = int(argmax_lowest(sc, cand)[0])
    best = float(sc.max())
    second = float(sc[cand != token].max()) if cand.size > 1 else float("nan")
    return token, best, second


def sample_row(row, dtype: str = "f32", temperature=1.0, top_k=0, top_p=1.0, min_p=0.0,
               seed: int = 0, row_id: int = 0, step: int = 0, keep_order: bool = False,
               kept_override: Optional[int] = None) -> RowResult:
    """One row of the stage: LSE, top-k, top-p, min-p, Gumbel-max draw, log-probability.

    ``kept_override`` re-draws over a different kept prefix length (used by the parity tests when the
    CUDA path kept a count inside the exemption band).
    """
    x = widen(row, dtype)
    n = int(x.size)
    res = RowResult(n=n)
    T = as_f32(temperature)
    p = as_f32(top_p)
    mp = as_f32(min_p)
    k = int(top_k)
    if n == 0:
        res.status = STATUS_INVALID_ARG
        return res
    if not np.all(np.isfinite(x)):                          # [TOPP]: reject non-finite inputs
        res.status = STATUS_NONFINITE
        return res
    if math.isnan(T) or math.isinf(T) or math.isnan(p) or p <= 0.0 or math.isnan(mp) or mp > 1.0:
        res.status = STATUS_INVALID_ARG
        return res

    order = canonical_order(x)                              # [TOPP] step 2
    m = float(x[order[0]])
    greedy = T <= 0.0
    t_eff = 1.0 if greedy else T
    s = (x - m) / t_eff                                     # [TOPP] step 3, [LOGP] temperature
    w = np.exp(s)
    S = math.fsum(w.tolist())                               # [LOGP] S, [TOPP] step 4 normaliser
    res.row_max = m
    res.row_logsum = math.log(S)

    nk = k if 0 < k < n else n                              # [TOPK]
    res.top_k_count = nk
    if greedy:
        kept = kept_lo = kept_hi = 1
    else:
        kept = kept_lo = kept_hi = nk
        if p < 1.0:                                         # [TOPP] steps 4-6 on the top-k set
            wk = w[order[:nk]]
            Sk = math.fsum(wk.tolist())
            target = p * Sk
            cp, amb = nucleus_count(wk, target)
            res.ambiguous = amb
            prefix = np.concatenate(([0.0], np.cumsum(wk)[:-1]))   # P_{j-1} for rank j
            band = BAND_REL * Sk
            # token at rank j is kept iff P_{j-1} < target; band tokens may go either way
            cp_lo = int(np.count_nonzero(prefix < target - band))
            cp_hi = int(np.count_nonzero(prefix <= target + band))
            kept, kept_lo, kept_hi = min(kept, cp), min(kept_lo, cp_lo), min(kept_hi, cp_hi)
        if mp > 0.0:                                        # [MINP] keep w_v >= min_p
            ws = w[order]
            cm = int(np.count_nonzero(ws >= mp))
            cm_lo, cm_hi = _count_band(ws, mp * (1.0 + BAND_REL), mp * (1.0 - BAND_REL))
            kept, kept_lo, kept_hi = min(kept, cm), min(kept_lo, cm_lo), min(kept_hi, cm_hi)
        kept, kept_lo, kept_hi = max(1, kept), max(1, kept_lo), max(1, kept_hi)   # at least one
    res.kept, res.kept_lo, res.kept_hi = kept, kept_lo, kept_hi
    last = int(order[kept - 1])
    res.pivot_key = order_key(x[last])
    res.idx_cut = last

    use = kept if kept_override is None else int(kept_override)
    if greedy:
        res.token = int(order[0])
        res.best = res.second = float("nan")
    else:
        cand = order[:use]
        res.token, res.best, res.second = draw(s, cand, seed, row_id, step)
        if not math.isnan(res.second):
            res.near_tie = (res.best - res.second) < TIE_REL * max(1.0, abs(res.best))
    res.logprob = min(float(s[res.token]) - res.row_logsum, 0.0)   # [LOGP] clamp
    if keep_order:
        res.order = order
        res.s = s
    return res


def kept_mask(res: RowResult, n: int) -> np.ndarray:
    """uint8 mask of the kept prefix of pi (1 = kept)."""
    mask = np.zeros(n, dtype=np.uint8)
    if res.order is not None and res.status == STATUS_OK:
        mask[res.order[:res.kept]] = 1
    return mask


def softmax_lse_row(row, dtype: str = "f32", temperature=1.0):
    """(m, log S) of one row at temperature T (T <= 0 reads as T = 1) -- [LOGP]."""
    r = sample_row(row, dtype, temperature=temperature if as_f32(temperature) > 0 else 1.0)
    return r.status, r.row_max, r.row_logsum


def logprob_row(row, dtype: str, temperature, token: int) -> float:
    """min((x_t - m)/T - log S, 0) over the full row -- [LOGP]."""
    x = widen(row, dtype)
    T = as_f32(temperature)
    t_eff = T if T > 0 else 1.0
    m = float(x.max())
    s = (x - m) / t_eff
    lse = math.log(math.fsum(np.exp(s).tolist()))
    return min(float(s[int(token)]) - lse, 0.0)


def topk_select_row(scores, length: int, k: int, k_max: int, dtype: str = "f32"):
    """[TOPK]: the k largest of scores[:length] by (value desc, index asc), in ascending index order.

    Returns (status, out[k_max]) with unused slots -1. NaN in the valid prefix is an error; +-inf are
    ordinary keys. k <= 0 selects nothing; k > k_max is an argument error. ``dtype`` "bf16" reads the
    scores as bfloat16 bit patterns, widened exactly ([TOPP] step 1), so equal bf16 values tie.
    """
    out = np.full(int(k_max), -1, dtype=np.int32)
    n = int(length)
    if n <= 0 or n > len(scores):
        return STATUS_INVALID_ARG, out
    x = widen(np.asarray(scores)[:n], dtype)
    if np.any(np.isnan(x)):                       # data errors are reported before parameter errors
        return STATUS_NONFINITE, out
    if k > k_max:
        return STATUS_INVALID_ARG, out
    if k <= 0:
        return STATUS_OK, out
    sel = np.sort(canonical_order(x)[:min(k, n)])
    out[:sel.size] = sel
    return STATUS_OK, out


def topn_logprobs_row(row, dtype: str, temperature, n_top: int):
    """The n_top most probable tokens of a row and their log-probabilities (a top-N logprob list).

    [LOGP] "Design: the numeric contract" gives the per-token log-probability min(z_t - lse, 0) with the
    temperature applied to the statistics; the list holds the first n_top tokens of the order (logit
    descending, token id ascending; [TOPP] step 2, [TOPK] Changes for ties), i.e. the most probable first.
    Returns (status, m, log S, idx[n_top], lp[n_top]); slots past the row length are -1 / NaN, and a row
    with a non-finite logit or temperature returns the error with every slot -1 / NaN.
    """
    x = widen(row, dtype)
    T = as_f32(temperature)
    idx = np.full(int(n_top), -1, dtype=np.int64)
    lp = np.full(int(n_top), np.nan, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        return STATUS_NONFINITE, math.nan, math.nan, idx, lp
    if math.isnan(T) or math.isinf(T):
        return STATUS_INVALID_ARG, math.nan, math.nan, idx, lp
    t_eff = T if T > 0 else 1.0
    m = float(x.max())
    s = (x - m) / t_eff
    log_s = math.log(math.fsum(np.exp(s).tolist()))
    order = canonical_order(x)
    take = min(int(n_top), x.size)
    for j in range(take):
        v = int(order[j])
        idx[j] = v
        lp[j] = min(float(s[v]) - log_s, 0.0)
    return STATUS_OK, m, log_s, idx, lp


def kept_logprob_row(row, dtype: str, temperature, top_k, top_p, min_p, token: int,
                     kept: Optional[int] = None):
    """Log-probability of ``token`` under the processed distribution: the softmax renormalised over the
    kept prefix of pi (temperature, then top-k, top-p, min-p, as in sample_row), -inf for a token outside
    it -- "[WS2][Logprob] ..." (Background: processed_logprobs derived from the rollout's logits, after
    the sampling transforms) with the clamp of [LOGP]: min(s_t - log sum_{kept} exp(s_v), 0).

    ``kept`` evaluates it for another kept prefix length (a parity test passes the CUDA path's count when
    that count lies in the 1e-6 band [kept_lo, kept_hi]). Greedy rows keep the first maximum alone.
    Returns (status, lp, kept_lo, kept_hi, rank of the token in pi).
    """
    res = sample_row(row, dtype, temperature, top_k, top_p, min_p, keep_order=True)
    if res.status != STATUS_OK:
        return res.status, math.nan, 0, 0, -1
    t = int(token)
    if not 0 <= t < res.n:
        return STATUS_INVALID_ARG, math.nan, 0, 0, -1
    c = res.kept if kept is None else int(kept)
    rank = int(np.flatnonzero(res.order == t)[0])
    if rank >= c:
        return STATUS_OK, -math.inf, res.kept_lo, res.kept_hi, rank
    log_sk = math.log(math.fsum(np.exp(res.s[res.order[:c]]).tolist()))
    return STATUS_OK, min(float(res.s[t]) - log_sk, 0.0), res.kept_lo, res.kept_hi, rank
