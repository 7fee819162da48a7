"""Comparison rules shared by the GPU parity tests (CUDA path vs CPU oracle).

Expected values always come from the oracle's own run on the same seeded
inputs; CUDA outputs are only compared, never fed to the oracle.

Rules:
* integers decided by exact comparisons on identical inputs (greedy verify,
  schedule order/lengths) must match bit for bit;
* a token decided by a floating-point argmax must match wherever the oracle's
  top-2 margin exceeds `tol`; inside the margin the CUDA token must still be a
  maximiser within `tol` of the oracle's score, and the rest of that request's
  chain (which conditions on the token) is excused.  A sampled token is decided
  in two levels (oracle.dspark.gumbel_max): its margin is the smaller of the
  two, and a flagged token's block must be within `tol` of the best block
  score and the token within `tol` of the best entry of that block;
* confidences, log-sum-exps and log-probabilities within `rtol`.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import oracle


# Tie band of a token decision, relative to the score's magnitude.  The CUDA
# path and the oracle compute the same scores to about 1e-6 (f32 sums of the
# same bf16 products, f32 logarithms of the same Philox words), so a band of
# 1e-4 leaves a hundredfold margin and flags only genuine near-ties.
TOL_DRAFT = 1e-4


def flag_budget(compared: int) -> int:
    """Near-ties allowed among `compared` token decisions.  With a tie band of
    1e-4 of scores of order 1-10 and top-2 gaps of order 0.1 or more, fewer
    than one decision in a thousand falls in it; 1 % leaves room for the two
    levels of a sampled token and small shapes."""
    return max(1, compared // 100)


def host(x):
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu()
        if x.dtype == torch.bfloat16:
            x = x.float()
        return x.numpy()
    return np.asarray(x)


@dataclass
class DraftReport:
    compared: int = 0
    flagged: int = 0
    excused: int = 0
    max_conf_err: float = 0.0
    max_lse_err: float = 0.0
    notes: list = field(default_factory=list)


def _shift_band(shift_row, s, tau, cand):
    """Twice the largest logit difference (over the candidate entries `cand`)
    between the two sides' base logits, in score units."""
    if shift_row is None or not np.any(cand):
        return 0.0
    return 2.0 * float(np.max(shift_row[cand])) / (tau if tau > 0 else 1.0)


def compare_draft(gpu_tokens, gpu_conf, gpu_lse, gpu_logp, orc, tau, tol_rel=1e-3,
                  conf_rtol=1e-2, requests=None, shift=None) -> DraftReport:
    """Walk each request's chain; see module docstring.  `orc` from oracle.markov_draft(keep_scores).

    `shift` [requests, gamma, V], optional: where the two sides' base logits
    differ (|GPU - oracle|, e.g. one bf16 step of a value the LM head's f32 sum
    rounded the other way), a decision among the entries near the top can move
    by up to that much, so its tie band widens by twice the largest such
    difference among them."""
    gt = host(gpu_tokens).astype(np.int64)
    gc = host(gpu_conf).astype(np.float64)
    gl = None if gpu_lse is None else host(gpu_lse).astype(np.float64)
    gp = None if gpu_logp is None else host(gpu_logp).astype(np.float64)
    R, G = orc["tokens"].shape
    rows = range(R) if requests is None else requests
    rep = DraftReport()
    for oi, i in enumerate(rows):
        for k in range(G):
            c_o = orc["conf"][oi, k]
            err = abs(gc[i, k] - c_o)
            rep.max_conf_err = max(rep.max_conf_err, err / max(abs(c_o), 1e-30))
            assert err <= conf_rtol * abs(c_o) + 1e-6, (i, k, gc[i, k], c_o)
            s = orc["scores"][oi, k]
            smax = float(s.max())
            two_level = tau > 0 and "block_scores" in orc
            sh = None if shift is None else shift[oi, k]
            if two_level:
                bs = orc["block_scores"][oi, k]
                bmax = float(bs.max())
                tol = tol_rel * max(1.0, abs(smax), abs(bmax))
                if sh is not None:  # every entry of a block near the top
                    blk = orc["block"]
                    near = np.repeat(bs >= bmax - 0.5, blk)[:s.size]
                    tol += _shift_band(sh, s, tau, near)
            else:
                tol = tol_rel * max(1.0, abs(smax))
                if sh is not None:
                    tol += _shift_band(sh, s, tau, s >= smax - 0.5)
            g = int(gt[i, k])
            assert 0 <= g < s.size
            rep.compared += 1
            if orc["margin"][oi, k] > tol:
                assert g == orc["tokens"][oi, k], (i, k, g, orc["tokens"][oi, k],
                                                   orc["margin"][oi, k])
            elif two_level:
                rep.flagged += 1
                blk = orc["block"]
                b = g // blk
                assert bmax - bs[b] <= tol, (i, k, bmax - bs[b], tol)
                inner = s[b * blk:(b + 1) * blk]
                assert float(inner.max()) - s[g] <= tol, (i, k, float(inner.max()) - s[g], tol)
            else:
                rep.flagged += 1
                assert smax - s[g] <= tol, (i, k, smax - s[g], tol)
            if tau > 0 and gl is not None:
                e = abs(gl[i, k] - orc["lse"][oi, k])
                rep.max_lse_err = max(rep.max_lse_err, e)
                assert e <= conf_rtol * max(1.0, abs(orc["lse"][oi, k])), (i, k, e)
                if g == orc["tokens"][oi, k] and gp is not None:
                    assert abs(gp[i, k] - orc["logp"][oi, k]) <= conf_rtol * max(
                        1.0, abs(orc["logp"][oi, k])), (i, k, gp[i, k], orc["logp"][oi, k])
            if g != orc["tokens"][oi, k]:
                rep.excused += G - k - 1
                break
    return rep


# Tie band of a verify decision: the acceptance test's log-margin, a Gumbel
# draw's top-2 gap, a residual trial's |1 - p_d/p_t - u|.  The two sides take
# them from the same bf16 logits with f32 log-sum-exps and Gumbels (errors of
# order 1e-6), so 1e-4 leaves a hundredfold margin; a corrected token drawn by
# residual trials carries the smallest margin of all its trials, so a wider
# band would excuse most rows with many trials.
TOL_VERIFY = 1e-4


def compare_verify(gpu_acc, gpu_bonus, orc, tau, tol=TOL_VERIFY):
    """Accepted counts and bonus tokens; sampling decisions inside `tol` are flagged."""
    ga = host(gpu_acc).astype(np.int64)
    gb = host(gpu_bonus).astype(np.int64)
    flagged = 0
    R = orc["accepted"].size
    for i in range(R):
        if tau == 0.0:
            assert ga[i] == orc["accepted"][i], (i, ga[i], orc["accepted"][i])
            assert gb[i] == orc["bonus"][i], (i, gb[i], orc["bonus"][i])
            continue
        m = orc["accept_margin"][i]
        n_o = orc["accepted"][i]
        tested = m[:min(n_o + 1, m.size)]
        tested = tested[~np.isnan(tested)]
        if np.any(np.abs(tested) < tol):
            flagged += 1
            continue
        assert ga[i] == n_o, (i, ga[i], n_o)
        if orc["final_margin"][i] <= tol:
            flagged += 1
            continue
        assert gb[i] == orc["bonus"][i], (i, gb[i], orc["bonus"][i])
    return flagged


def sorted_order_ok(order, a):
    """order lists every id once, a non-increasing along it, ties by ascending id."""
    order = np.asarray(order)
    flat = a.reshape(-1)
    assert sorted(order.tolist()) == list(range(flat.size))
    for p in range(flat.size - 1):
        x, y = flat[order[p]], flat[order[p + 1]]
        assert x > y or (x == y and order[p] < order[p + 1])
    return True


def oracle_draft_inputs(inp):
    """Convert a workloads.make_inputs dict to the oracle's float64 view."""
    return {k: (oracle.dspark.to_f64(v) if isinstance(v, torch.Tensor) and v.is_floating_point()
                else v) for k, v in inp.items()}


def schedule_is_robust(o_s, rel=1e-4) -> bool:
    """True when perturbing the confidences by `rel` cannot change the oracle's
    schedule: distinct survival products are `rel` apart and the chosen Theta
    beats every other budget by `rel` (unconstrained) or every step is `rel`
    away from a tie (break)."""
    a = np.sort(o_s["a"].reshape(-1).astype(np.float64))
    d = np.diff(a)
    d = d[d > 0]
    if d.size and np.min(d / a[1:][np.diff(a) > 0]) < rel:
        return False
    th = o_s["thetas"]
    K = o_s["K"]
    others = np.delete(th, K)
    if others.size and np.max(others) > th[K] * (1 - rel):
        step = np.abs(np.diff(th)) / th[1:]
        return bool(np.min(step) > rel)
    return True
