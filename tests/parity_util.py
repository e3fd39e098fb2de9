"""Helpers for the GPU parity tests: run the CUDA path on a workload and compare it with the oracle.

Tolerances (from the stage's contract):
* top-k index sets and their order: bit-exact;
* top-p / min-p kept prefix: exact, except that tokens whose binary64 prefix mass lies within 1e-6 * S_k
  of the target (min-p: weight within 1e-6 * min_p of min_p) may fall on either side -- the oracle
  returns the admissible range [kept_lo, kept_hi];
* log-probabilities and log-sum-exp: within 1e-5 absolute; row maxima exact;
* sampled tokens: identical on the same Philox counters, except draws whose two best perturbed scores
  differ by less than 1e-6 relative (near ties), which must stay below 1e-4 of all draws.

A compared row whose oracle boundary is ambiguous (the compensated scan and the fsum certificate disagree) fails
the comparison: "Split top-p numerical reference and conservative gate", Independent binary64 numerical
reference, step 6, reports oracle_boundary_ambiguous and stops there instead of comparing.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import sampler as osm

LOGP_TOL = 1e-5
# the entry point the sampling checks call: "vsamp_sample" (one cluster per row) or "vsamp_sample_ws"
# (split vocabulary, workspace)
SAMPLE_FN = "vsamp_sample"


def sample_fn(ts):
    return getattr(ts, SAMPLE_FN)


def to_device(batch_logits: np.ndarray, dtype: str, dev) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(batch_logits).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(batch_logits)).to(dev)


def t(arr, dev, dtype=None):
    a = np.asarray(arr)
    if a.dtype == np.uint64:
        a = a.view(np.int64)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    x = torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return x if dtype is None else x.to(dtype)


def run_sample(ts, batch, dev, V=None, row_id=None, x=None):
    x = to_device(batch.logits, batch.dtype, dev) if x is None else x
    tok, lp, st, stats = sample_fn(ts)(
        x, temperature=t(batch.temperature, dev), top_k=t(batch.top_k, dev), top_p=t(batch.top_p, dev),
        min_p=t(batch.min_p, dev), seed=t(batch.seed, dev), step=t(batch.step, dev),
        row_id=None if row_id is None else t(row_id, dev), V=V if V is not None else batch.V, want_stats=True)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), lp.cpu().numpy(), st.cpu().numpy(), stats.cpu().numpy()


def run_cut(ts, batch, dev, want_mask=True, x=None):
    x = to_device(batch.logits, batch.dtype, dev) if x is None else x
    cut, mask, stats = ts.vsamp_topp_minp_mask(
        x, temperature=t(batch.temperature, dev), top_k=t(batch.top_k, dev), top_p=t(batch.top_p, dev),
        min_p=t(batch.min_p, dev), V=batch.V, want_mask=want_mask)
    torch.cuda.synchronize()
    return cut.cpu().numpy(), None if mask is None else mask.cpu().numpy(), stats.cpu().numpy()


def oracle_row(batch, r, row_id=None, keep_order=True, kept_override=None):
    return osm.sample_row(batch.logits[r, :batch.V], batch.dtype, batch.temperature[r], batch.top_k[r],
                          batch.top_p[r], batch.min_p[r], int(batch.seed[r]), r if row_id is None else int(row_id),
                          int(batch.step[r]), keep_order=keep_order, kept_override=kept_override)


class TieCounter:
    def __init__(self):
        self.draws = 0
        self.near = 0

    def check(self, max_frac=1e-4):
        # below 1e4 draws a 1e-4 rate allows no near tie at all
        allowed = max_frac * self.draws if self.draws >= 10_000 else 0
        assert self.near <= allowed, f"near-tie draws {self.near} of {self.draws}"


def check_sample(batch, rows, tok, lp, st, stats, ties: TieCounter, row_ids=None):
    """Token, log-probability, status and kept count of each row against the oracle."""
    for r in rows:
        rid = None if row_ids is None else row_ids[r]
        ref = oracle_row(batch, r, row_id=rid)
        assert not ref.ambiguous, f"row {r}: oracle_boundary_ambiguous"
        assert st[r] == ref.status, f"row {r}: status {st[r]} != oracle {ref.status}"
        if ref.status != 0:
            assert tok[r] == -1 and math.isnan(lp[r]), f"row {r}: error row outputs {tok[r]}, {lp[r]}"
            continue
        kept = int(stats[r, 2])
        assert ref.kept_lo <= kept <= ref.kept_hi, f"row {r}: kept {kept} not in [{ref.kept_lo}, {ref.kept_hi}]"
        if kept != ref.kept:
            ref = oracle_row(batch, r, row_id=rid, kept_override=kept)
        ties.draws += 1
        if ref.near_tie:
            ties.near += 1
            assert tok[r] in set(ref.order[:kept].tolist())
        else:
            assert tok[r] == ref.token, f"row {r}: token {tok[r]} != oracle {ref.token} (kept {kept})"
        want_lp = osm.logprob_row(batch.logits[r, :batch.V], batch.dtype, batch.temperature[r], int(tok[r]))
        assert abs(float(lp[r]) - want_lp) <= LOGP_TOL, f"row {r}: logprob {lp[r]} vs {want_lp}"


def check_cut(batch, rows, cut, mask, stats):
    """Cut descriptor and mask of each row against the oracle's kept prefix."""
    for r in rows:
        ref = oracle_row(batch, r)
        assert not ref.ambiguous, f"row {r}: oracle_boundary_ambiguous"
        assert cut[r, 3] == ref.status, f"row {r}: status {cut[r, 3]} != {ref.status}"
        if ref.status != 0:
            assert cut[r, 2] == 0
            if mask is not None:
                assert not mask[r, :batch.V].any()
            continue
        kept = int(cut[r, 2])
        assert ref.kept_lo <= kept <= ref.kept_hi, f"row {r}: kept {kept} not in [{ref.kept_lo}, {ref.kept_hi}]"
        last = int(ref.order[kept - 1])
        assert int(cut[r, 1]) == last, f"row {r}: idx_cut {cut[r, 1]} != {last}"
        x64 = osm.widen(batch.logits[r, :batch.V], batch.dtype)
        assert (int(cut[r, 0]) & 0xFFFFFFFF) == osm.order_key(x64[last]), f"row {r}: pivot key"
        assert int(stats[r, 2]) == kept
        if mask is not None:
            want = np.zeros(batch.V, dtype=np.uint8)
            want[ref.order[:kept]] = 1
            assert np.array_equal(mask[r, :batch.V], want), f"row {r}: mask differs"
