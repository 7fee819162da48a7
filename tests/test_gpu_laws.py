"""The CUDA path against the plain laws of the method, not against the oracle.

Token-by-token parity compares the kernels with an oracle that takes the same
two-level sampler and the same random streams, so it cannot show that the
sampler itself is right.  These tests check what the pages and the mathematics
fix, on the CUDA path alone, by frequencies over many independent requests
(every request id keys its own Philox streams):

* the draft's tokens are distributed as softmax(l / tau) of their logits,
  with and without the Markov bias ("DSpark 深度解读" §二 设计一; plain
  Gumbel-max is an exact sampler of that law, and so must the kernel be);
* the verifier accepts position 1 with probability sum_v min(p_d, p_t) =
  1 - 1/2 ||p_d - p_t||_1, the confidence label of §二 设计二, and the token it
  emits first follows p_t (speculative sampling is lossless);
* a whole round, draft -> schedule -> verify, repeated, emits tokens that
  follow the target's own law in every admission mode that does not look at
  the token it admits (full length, random lengths, break, fixed K and the
  asynchronous mode of §三 挑战1).

Every chi-square test also shows its power: the same counts reject a plausible
slip (a wrong temperature, the reversed acceptance ratio, a perturbed target).
The seeds are fixed, so each outcome is deterministic.
"""
import math

import numpy as np
import pytest
import torch

import workloads

stats = pytest.importorskip("scipy.stats")

pytestmark = pytest.mark.gpu

dsp = pytest.importorskip("speculative_decoding_draft_02_gb300")

P_MIN = 1e-3    # a correct sampler must pass at this level
P_POWER = 1e-6  # a slipped law must be rejected at this level


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from speculative_decoding_draft_02_gb300 import build
    build.build()
    dsp.load_library()
    yield
    assert dsp.dspark_device_status() == 0


def _bf16(x):
    """float64 values of x rounded to bf16 (as the library receives them)."""
    return torch.as_tensor(x, dtype=torch.float64).to(torch.bfloat16).double().numpy()


def _softmax(l):
    l = np.asarray(l, dtype=np.float64)
    m = l.max(axis=-1, keepdims=True)
    e = np.exp(l - m)
    return e / e.sum(axis=-1, keepdims=True)


def _chisq(counts, probs):
    """Pearson chi-square p-value, cells of expected count below 5 pooled."""
    counts = np.asarray(counts, dtype=np.float64).reshape(-1)
    exp = np.asarray(probs, dtype=np.float64).reshape(-1) * counts.sum()
    keep = exp >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    ex = np.append(exp[keep], exp[~keep].sum())
    if ex[-1] == 0:
        obs, ex = obs[:-1], ex[:-1]
    return stats.chisquare(obs, ex * obs.sum() / ex.sum()).pvalue


def _head(R, G, V, r, d, W1, W2, w_conf=None):
    W_lm = torch.zeros((V, d), dtype=torch.float32)
    w = torch.zeros(d + r) if w_conf is None else w_conf
    return dsp.DraftHead.from_weights(R, G, W_lm, torch.as_tensor(W1, dtype=torch.float32),
                                      torch.as_tensor(W2, dtype=torch.float32), w,
                                      torch.ones(G))


def _draft(head, base, h, anchor, tau, seed):
    d = head.dims
    R, G = d.R, d.gamma
    out = dict(tokens=torch.empty((R, G), dtype=torch.int32, device="cuda"),
               conf=torch.empty((R, G), dtype=torch.float32, device="cuda"),
               logp=torch.empty((R, G), dtype=torch.float32, device="cuda"),
               lse=torch.empty((R, G), dtype=torch.float32, device="cuda"))
    ws = dsp.workspace(dsp.dspark_markov_workspace_bytes(d))
    dsp.dspark_markov_draft(d, base, h, anchor, head.W1, head.W2t, head.w_conf, head.T, tau,
                            seed, out["tokens"], out["conf"], out["logp"], out["lse"], ws)
    torch.cuda.synchronize()
    assert dsp.dspark_device_status() == 0
    return out


# V = 200: three whole sampler blocks of 64 ids and a ragged one of 8
V_LAW, R_LAW, D_LAW, RANK = 200, 8192, 64, 64


@pytest.mark.parametrize("tau", [0.6, 1.0, 1.6])
def test_draft_tokens_follow_softmax_without_bias(tau):
    """W2 = 0: every request and position draws from softmax(base / tau) of one
    shared base-logit row, R x gamma = 32768 independent draws."""
    R, G, V, r, d = R_LAW, 4, V_LAW, RANK, D_LAW
    rng = np.random.default_rng(70)
    row = _bf16(rng.standard_normal(V) * 1.3)
    W1 = rng.standard_normal((V, r)) / math.sqrt(r)
    head = _head(R, G, V, r, d, W1, np.zeros((r, V)))
    base = torch.tensor(row, dtype=torch.float64).to(torch.bfloat16).cuda().expand(R * G, V)
    out = _draft(head, base.contiguous(), torch.zeros((R * G, d), dtype=torch.bfloat16,
                                                      device="cuda"),
                 torch.zeros(R, dtype=torch.int32, device="cuda"), tau, 4242 + int(10 * tau))
    tok = out["tokens"].cpu().numpy().reshape(-1)
    assert tok.min() >= 0 and tok.max() < V
    counts = np.bincount(tok, minlength=V)
    p = _softmax(row / tau)
    assert _chisq(counts, p) > P_MIN
    assert _chisq(counts, _softmax(row / (1.15 * tau))) < P_POWER  # a wrong temperature
    # the log-sum-exp the draft reports is the plain one of l / tau
    lse = out["lse"].cpu().numpy()
    m = (row / tau).max()
    want = m + math.log(np.exp(row / tau - m).sum())
    assert np.all(np.abs(lse - want) <= 1e-4 * max(1.0, abs(want)))
    # and log p_d(x) is that token's plain log-probability
    logp = out["logp"].cpu().numpy().reshape(-1)
    assert np.all(np.abs(logp - np.log(p[tok])) <= 1e-4 * np.maximum(1.0, np.abs(np.log(p[tok]))))


@pytest.mark.parametrize("tau", [0.6, 1.0])
def test_draft_tokens_follow_softmax_with_markov_bias(tau):
    """Position 1 of every request, one shared anchor: the law is
    softmax((base + W1[anchor] W2) / tau) with the bias taken in float64 from
    the bf16 weights."""
    R, G, V, r, d = 2 * R_LAW, 1, V_LAW, RANK, D_LAW
    rng = np.random.default_rng(71)
    row = _bf16(rng.standard_normal(V) * 0.8)
    W1 = _bf16(rng.standard_normal((V, r)))
    W2 = _bf16(rng.standard_normal((r, V)) * 1.5 / math.sqrt(r))
    anchor = 17
    head = _head(R, G, V, r, d, W1, W2)
    base = torch.tensor(row, dtype=torch.float64).to(torch.bfloat16).cuda().expand(R * G, V)
    out = _draft(head, base.contiguous(), torch.zeros((R * G, d), dtype=torch.bfloat16,
                                                      device="cuda"),
                 torch.full((R,), anchor, dtype=torch.int32, device="cuda"), tau, 5151)
    tok = out["tokens"].cpu().numpy().reshape(-1)
    ell = row + W1[anchor] @ W2
    assert np.std(W1[anchor] @ W2) > 1.0  # the bias moves the law visibly
    counts = np.bincount(tok, minlength=V)
    assert _chisq(counts, _softmax(ell / tau)) > P_MIN
    assert _chisq(counts, _softmax(row / tau)) < P_POWER  # the bias left out


def _target_rows(rng, row, V, scale=0.9):
    return _bf16(row + rng.standard_normal(V) * scale)


def test_verify_acceptance_rate_is_the_confidence_label():
    """One draft position per request, drafted by the CUDA sampler from p_d and
    verified against a shared target row p_t: P(accept) = sum_v min(p_d, p_t);
    the first emitted token (the draft if accepted, else the residual draw)
    follows p_t; after an acceptance the bonus follows the second target row."""
    R, G, V, r, d, tau = 2 * R_LAW, 1, V_LAW, RANK, D_LAW, 1.0
    rng = np.random.default_rng(72)
    row = _bf16(rng.standard_normal(V) * 1.2)
    head = _head(R, G, V, r, d, rng.standard_normal((V, r)) / math.sqrt(r), np.zeros((r, V)))
    base = torch.tensor(row, dtype=torch.float64).to(torch.bfloat16).cuda().expand(R * G, V)
    base = base.contiguous()
    anchor = torch.zeros(R, dtype=torch.int32, device="cuda")
    out = _draft(head, base, torch.zeros((R * G, d), dtype=torch.bfloat16, device="cuda"),
                 anchor, tau, 909)
    t1, t2 = _target_rows(rng, row, V), _target_rows(rng, row, V)
    target = torch.tensor(np.stack([t1, t2]), dtype=torch.float64).to(torch.bfloat16)
    target = target.cuda().unsqueeze(0).expand(R, 2, V).contiguous()
    lens = torch.ones(R, dtype=torch.int32, device="cuda")
    acc = torch.empty(R, dtype=torch.int32, device="cuda")
    bonus = torch.empty(R, dtype=torch.int32, device="cuda")
    ws = dsp.workspace(dsp.dspark_verify_workspace_bytes(head.dims))
    dsp.dspark_verify(head.dims, anchor, out["tokens"], lens, base, head.W1, head.W2t,
                      out["lse"], out["logp"], target, tau, 31337, acc, bonus, ws)
    torch.cuda.synchronize()
    assert dsp.dspark_device_status() == 0
    a = acc.cpu().numpy()
    b = bonus.cpu().numpy()
    x = out["tokens"].cpu().numpy()[:, 0]
    assert set(np.unique(a)) <= {0, 1}
    pd, pt1, pt2 = _softmax(row / tau), _softmax(t1 / tau), _softmax(t2 / tau)
    label = float(np.minimum(pd, pt1).sum())
    assert label == pytest.approx(1.0 - 0.5 * np.abs(pd - pt1).sum(), abs=1e-12)
    sigma = math.sqrt(label * (1.0 - label) / R)
    assert abs(a.mean() - label) < 4.5 * sigma, (a.mean(), label, sigma)
    reversed_ratio = float(np.sum(pd * np.minimum(1.0, pd / pt1)))
    assert abs(reversed_ratio - label) > 8 * sigma  # that slip would be caught
    first = np.where(a == 1, x, b)
    assert _chisq(np.bincount(first, minlength=V), pt1) > P_MIN
    assert _chisq(np.bincount(first, minlength=V), pd) < P_POWER  # the draft's own law
    # after an acceptance the bonus comes from the second target row
    assert _chisq(np.bincount(b[a == 1], minlength=V), pt2) > P_MIN
    # after a rejection it comes from the normalised residual max(0, p_t - p_d)
    res = np.maximum(pt1 - pd, 0.0)
    assert _chisq(np.bincount(b[a == 0], minlength=V), res / res.sum()) > P_MIN


# ------------------------------------------------- a whole round, repeated ---

V_CH, G_CH, R_CH, BATCHES, L_CH = 128, 3, 4096, 8, 2


def _markov_target(rng, V):
    """A first-order Markov target whose mass sits on eight ids, four in each
    of the two sampler blocks (the rest share the remaining ~10 %)."""
    hot = np.array([3, 17, 40, 60, 64, 80, 101, 127])
    logPt = np.full((V, V), -3.5)
    logPt[:, hot] = rng.standard_normal((V, hot.size)) * 1.1
    return logPt


def _run_chain(mode, seed, logPt, start):
    """BATCHES x R_CH independent trials decode L_CH tokens each by repeated
    CUDA rounds (draft -> schedule -> verify) against the target chain."""
    rng = np.random.default_rng(seed)
    V, G, R, r, d = V_CH, G_CH, R_CH, 64, 64
    W1 = rng.standard_normal((V, r))
    W2 = rng.standard_normal((r, V)) * 0.9 / math.sqrt(r)
    base0 = rng.standard_normal((G, V)) * 0.8
    w_conf = torch.tensor(rng.standard_normal(d + r) * 0.4, dtype=torch.float32)
    head = _head(R, G, V, r, d, W1, W2, w_conf)
    rnd = dsp.Round(head)
    logPt_d = torch.tensor(logPt, dtype=torch.float32, device="cuda")
    sps = workloads.sps_table("concave", R * (G + 1)).cuda()
    first = np.full((BATCHES * R, L_CH), -1, dtype=np.int64)
    for bt in range(BATCHES):
        anchor = torch.full((R,), start, dtype=torch.int32, device="cuda")
        got = np.zeros(R, dtype=np.int64)
        ring = dsp.async_ring(R * G // 3, R * G // 2) if mode == "async" else None
        for t in range(8):
            s = seed * 100 + bt * 10 + t
            base = torch.tensor(np.tile(base0, (R, 1)), dtype=torch.float32).to(torch.bfloat16)
            rnd.base.copy_(base.cuda())
            h = workloads.random_normal((R * G, d), 1.0, s, device="cuda")
            dsp.dspark_markov_draft(head.dims, rnd.base, h, anchor, head.W1, head.W2t,
                                    head.w_conf, head.T, 1.0, 7000 + s, rnd.tokens, rnd.conf,
                                    rnd.logp_d, rnd.lse_d, rnd.ws_draft)
            prev = torch.cat([anchor[:, None], rnd.tokens], dim=1).long()   # x_0 .. x_G
            target = logPt_d[prev].to(torch.bfloat16).contiguous()         # row j | x_j
            if mode == "full":
                rnd.len.fill_(G)
            elif mode == "random":
                rnd.len.copy_(torch.tensor(rng.integers(0, G + 1, R), dtype=torch.int32))
            elif mode == "break":
                rnd.schedule(sps, dsp.SCHED_BREAK)
            elif mode == "fixed_k":
                rnd.schedule(sps, dsp.SCHED_FIXED_K, R * G // 2)
            elif mode == "async":
                rnd.schedule(sps, dsp.SCHED_ASYNC, k_ring=ring)
            rnd.verify(anchor, target, 1.0, 9000 + s)
            torch.cuda.synchronize()
            x = rnd.tokens.cpu().numpy()
            n = rnd.accepted.cpu().numpy().astype(np.int64)
            b = rnd.bonus.cpu().numpy()
            # this round's emitted tokens: x_1 .. x_n, then the bonus
            for q in range(G + 1):
                tok = np.where(q < n, x[:, min(q, G - 1)], b)
                emit = (q <= n) & (got < L_CH)
                first[bt * R + np.nonzero(emit)[0], got[emit]] = tok[emit]
                got += emit
            anchor = torch.tensor(b, dtype=torch.int32, device="cuda")
            if got.min() >= L_CH:
                break
        assert got.min() >= L_CH
    assert dsp.dspark_device_status() == 0
    return first


@pytest.mark.parametrize("mode", ["full", "random", "break", "fixed_k", "async"])
def test_round_emits_the_target_law(mode):
    """32768 trials, each decoding two tokens with CUDA rounds from one start
    token: the emitted pairs follow P_t(a | start) P_t(b | a), the target
    chain, in every non-anticipating admission mode."""
    rng = np.random.default_rng(73)
    logPt = _markov_target(rng, V_CH)
    start = 5
    first = _run_chain(mode, 11 + ["full", "random", "break", "fixed_k", "async"].index(mode),
                       logPt, start)
    Pt = _softmax(_bf16(logPt))
    joint = Pt[start][:, None] * Pt
    cells = first[:, 0] * V_CH + first[:, 1]
    counts = np.bincount(cells, minlength=V_CH * V_CH)
    assert _chisq(counts, joint) > P_MIN, mode
    assert _chisq(np.bincount(first[:, 0], minlength=V_CH), Pt[start]) > P_MIN
    # power: the chain at a slightly different temperature is rejected
    Pw = _softmax(_bf16(logPt) * 1.15)
    assert _chisq(counts, Pw[start][:, None] * Pw) < P_POWER
