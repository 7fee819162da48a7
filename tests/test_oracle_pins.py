"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties one oracle function to a closed form, a brute-force enumeration,
published known-answer vectors or a statistical law, so that a plausible
mistake (dropped term, wrong sign or index, transposed operand) fails here.
"""
import itertools
import math
import os
import zlib

import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import philox
from oracle.dspark import sigmoid

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- Philox ---

def test_philox_known_answers():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(x, 16) for x in line.split()])
    assert len(rows) == 3
    for row in rows:
        ctr, key, want = row[:4], row[4:6], row[6:]
        got = philox.philox4x32_10(*ctr, *key)
        assert [int(x) for x in got] == want


def test_uniform_is_exact_float32_in_open_interval():
    v = np.arange(4096, dtype=np.uint64)
    u = philox.uniform(12345, 3, 7, 0, v)
    assert np.all(u > 0) and np.all(u < 1)
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    # extremes of the map: word 0 -> 2^-24, word 2^32-1 -> 1 - 2^-24
    lo = ((0 >> 9) + 0.5) * 2.0 ** -23
    hi = (((2 ** 32 - 1) >> 9) + 0.5) * 2.0 ** -23
    assert lo == 2.0 ** -24 and hi == 1 - 2.0 ** -24
    # counter layout: slot v uses word v & 3 of counter (v >> 2, pos, req, stream)
    w = philox.philox4x32_10(5, 3, 7, 0, 12345 & 0xFFFFFFFF, 12345 >> 32)
    assert int(philox.words(12345, 3, 7, 0, 22)) == int(w[2])


def test_uniform_distribution():
    v = np.arange(200000, dtype=np.uint64)
    u = philox.uniform(99, 1, 2, 1, v)
    assert stats.kstest(u, "uniform").pvalue > 1e-4


# ------------------------------------------------------- a1: base logits ---

def test_base_logits_brute_force():
    rng = np.random.default_rng(1)
    h = rng.standard_normal((3, 5))
    W = rng.standard_normal((7, 5))
    want = np.zeros((3, 7))
    for m in range(3):
        for v in range(7):
            want[m, v] = sum(h[m, i] * W[v, i] for i in range(5))
    got = oracle.base_logits(h, W, bf16_out=False)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)
    # bf16 materialisation: representable, and within half a bf16 ulp (+fp32 step)
    gb = oracle.base_logits(h, W, bf16_out=True)
    assert np.array_equal(oracle.round_bf16(gb), gb)
    assert np.all(np.abs(gb - want) <= np.abs(want) * 2.0 ** -8 + 1e-30)


def test_round_bf16_known_values():
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: round to even -> 1
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38])
    got = oracle.round_bf16(x)
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == 1.0 + 2 ** -6 and got[3] == -2.5
    assert np.isfinite(got[4])


# ------------------------------------------- a2-a4: Markov head and conf ---

def _tiny_draft_inputs(R=3, G=4, V=11, r=3, d=5, seed=0, w2_zero=False):
    rng = np.random.default_rng(seed)
    base = rng.standard_normal((R, G, V))
    h = rng.standard_normal((R, G, d))
    anchor = rng.integers(0, V, R)
    W1 = rng.standard_normal((V, r))
    W2 = np.zeros((r, V)) if w2_zero else rng.standard_normal((r, V))
    w = rng.standard_normal(d + r)
    T = 1.0 + rng.random(G)
    return base, h, anchor, W1, W2, w, T


def test_markov_bias_is_row_of_explicit_transition_matrix():
    base, h, anchor, W1, W2, w, T = _tiny_draft_inputs()
    R, G, V = base.shape
    P = [[sum(W1[a, i] * W2[i, b] for i in range(W1.shape[1])) for b in range(V)]
         for a in range(V)]
    out = oracle.markov_draft(base, h, anchor, W1, W2, w, T, 0.0, 0, keep_logits=True)
    P = np.array(P)
    assert not np.allclose(P, P.T)
    prev = anchor.copy()
    for k in range(G):
        for rq in range(R):
            want = base[rq, k] + P[prev[rq]]          # row of x_{k-1}, not column
            np.testing.assert_allclose(out["logits"][rq, k], want, rtol=1e-12, atol=1e-12)
            assert out["tokens"][rq, k] == int(np.argmax(want))
        prev = out["tokens"][:, k]


def test_w2_zero_reduces_to_parallel_drafting():
    base, h, anchor, W1, W2, w, T = _tiny_draft_inputs(w2_zero=True, V=40)
    out = oracle.markov_draft(base, h, anchor, W1, W2, w, T, 0.0, 0)
    assert np.array_equal(out["tokens"], np.argmax(base, axis=2))


def test_fused_step_keeps_the_base_logit_unrounded():
    """One contraction per step gives h . W_lm exactly: 257.5 and 257.75 stay
    apart (the second wins), where the LM head's bf16 output rounds both to 258
    and the tie goes to the first id."""
    h = np.ones((1, 1, 2))
    W_lm = np.array([[256.0, 1.5], [256.0, 1.75]])   # every weight exact in bf16
    W1, W2 = np.zeros((2, 8)), np.zeros((8, 2))        # no Markov bias
    w, T, anchor = np.zeros(2 + 8), np.ones(1), np.zeros(1, dtype=np.int64)
    fused = oracle.fused_draft(h, anchor, W_lm, W1, W2, w, T, 0.0, 0)
    stored = oracle.markov_draft(oracle.base_logits(h, W_lm), h, anchor, W1, W2, w, T, 0.0, 0)
    assert fused["tokens"][0, 0] == 1 and stored["tokens"][0, 0] == 0


@pytest.mark.parametrize("tau", [0.0, 1.0])
def test_fused_step_equals_the_markov_head_when_base_logits_are_bf16_exact(tau):
    """Small-integer h and W_lm make every h . W_lm an integer below 256, exact in
    bf16: then the fused step and LM head + Markov head draw the same tokens and
    confidences (the same random streams)."""
    rng = np.random.default_rng(61)
    R, G, V, r, d = 3, 4, 130, 8, 6
    h = rng.integers(-2, 3, (R, G, d)).astype(np.float64)
    W_lm = rng.integers(-3, 4, (V, d)).astype(np.float64)
    W1 = rng.standard_normal((V, r))
    W2 = rng.standard_normal((r, V))
    w = rng.standard_normal(d + r)
    T = 1.0 + rng.random(G)
    anchor = rng.integers(0, V, R)
    base = oracle.base_logits(h, W_lm)
    assert np.array_equal(base, h @ W_lm.T)           # exact: the bf16 rounding is a no-op
    fused = oracle.fused_draft(h, anchor, W_lm, W1, W2, w, T, tau, 7)
    stored = oracle.markov_draft(base, h, anchor, W1, W2, w, T, tau, 7)
    assert np.array_equal(fused["tokens"], stored["tokens"])
    np.testing.assert_array_equal(fused["conf"], stored["conf"])


def _rnn_case(R=6, G=4, V=40, r=8, d=5, seed=51):
    rng = np.random.default_rng(seed)
    base = rng.standard_normal((R, G, V))
    h = rng.standard_normal((R, G, d))
    h[:, :, 0] = 1.0                                   # a constant feature
    anchor = rng.integers(0, V, R)
    W1 = rng.standard_normal((V, r))
    W2 = rng.standard_normal((r, V)) * 1.5
    w = rng.standard_normal(d + r)
    T = 1.0 + rng.random(G)
    return base, h, anchor, W1, W2, w, T


def test_rnn_head_without_weights_is_parallel_drafting():
    base, h, anchor, W1, W2, w, T = _rnn_case()
    r, d = W1.shape[1], h.shape[2]
    out = oracle.rnn_draft(base, h, anchor, W1, W2, np.zeros((2 * r, 2 * r + d)), w, T, 0.0, 0)
    assert np.array_equal(out["tokens"], np.argmax(base, axis=2))
    assert np.all(out["state"] == 0.0)
    # a closed gate (g -> 0 through the constant feature) keeps the zero state too
    W_gc = np.random.default_rng(3).standard_normal((2 * r, 2 * r + d))
    W_gc[:r, 2 * r] = -60.0
    out = oracle.rnn_draft(base, h, anchor, W1, W2, W_gc, w, T, 0.0, 0)
    assert np.array_equal(out["tokens"], np.argmax(base, axis=2))
    assert np.max(np.abs(out["state"])) < 1e-20


def test_rnn_head_with_open_gate_is_a_markov_head_on_tanh_embeddings():
    """g -> 1 and a candidate map that passes the embedding: s_k = tanh(W1[x_{k-1}]),
    so the draft is the Markov head's with W1 replaced by bf16(tanh(W1)) in the bias;
    the confidence head still sees W1 itself."""
    base, h, anchor, W1, W2, w, T = _rnn_case()
    r, d = W1.shape[1], h.shape[2]
    W_gc = np.zeros((2 * r, 2 * r + d))
    W_gc[:r, 2 * r] = 60.0                             # update gate open
    W_gc[r:, r:2 * r] = np.eye(r)                      # candidate = tanh(embedding)
    rnn = oracle.rnn_draft(base, h, anchor, W1, W2, W_gc, w, T, 0.0, 0)
    W1t = oracle.round_bf16(np.tanh(W1))
    mk = oracle.markov_draft(base, h, anchor, W1t, W2, w, T, 0.0, 0)
    assert np.array_equal(rnn["tokens"], mk["tokens"])
    assert np.all(mk["margin"] > 1e-9)                 # no tie decides the comparison
    mk_conf = oracle.markov_draft(base, h, anchor, W1, W2, w, T, 0.0, 0, forced=rnn["tokens"])
    np.testing.assert_allclose(rnn["conf"], mk_conf["conf"], rtol=1e-13)


def test_rnn_head_two_steps_in_closed_form():
    """One request, two steps, rank 1, worked by hand.  The gate row sees only
    the constant feature with weight ln 3, so g = sigmoid(ln 3) = 3/4; the
    candidate row takes 3/4 of the state (in bf16), the embedding and 1/4 of the
    constant feature.  With W1[anchor = 2] = 1/2 and W1[5] = -1/4:
      s_1 = 1/4 * 0   + 3/4 * tanh(0 + 1/2 + 1/4)            = 3/4 tanh(3/4)
      s_2 = 1/4 * s_1 + 3/4 * tanh(3/4 bf16(s_1) - 1/4 + 1/4)
    and the logit of id 0 at step k is bf16(s_k) * W2[0, 0] (its base logit is
    0).  A dropped carry, a swapped gate half, g and 1 - g exchanged, or an
    unrounded state would each give a different number."""
    import torch
    V, r, d = 8, 1, 1
    base = np.zeros((1, 2, V))
    base[0, 0, 5] = 10.0                               # x_1 = 5
    base[0, 1, 6] = 10.0                               # x_2 = 6
    h = np.ones((1, 2, d))
    W1 = np.zeros((V, r))
    W1[2, 0], W1[5, 0] = 0.5, -0.25
    W2 = np.zeros((r, V))
    W2[0, 0] = 0.375
    W_gc = np.array([[0.0, 0.0, math.log(3.0)],       # gate:      [state, embedding, h]
                     [0.75, 1.0, 0.25]])               # candidate: [state, embedding, h]
    out = oracle.rnn_draft(base, h, np.array([2]), W1, W2, W_gc, np.zeros(d + r), np.ones(2),
                           0.0, 0, keep_scores=True)
    bf = lambda x: torch.tensor(x, dtype=torch.float64).to(torch.bfloat16).double().item()
    s1 = 0.75 * math.tanh(0.75)
    s2 = 0.25 * s1 + 0.75 * math.tanh(0.75 * bf(s1))
    assert out["tokens"].tolist() == [[5, 6]]
    assert out["state"][0, 0] == pytest.approx(s2, abs=1e-15)
    assert out["scores"][0, 0, 0] == pytest.approx(bf(s1) * 0.375, abs=1e-15)
    assert out["scores"][0, 1, 0] == pytest.approx(bf(s2) * 0.375, abs=1e-15)
    # the slips this pin tells apart from the reading
    slips = {"no carry": 0.75 * math.tanh(0.75 * bf(s1)),
             "gate and 1 - gate exchanged": 0.75 * 0.25 * math.tanh(0.75)
             + 0.25 * math.tanh(0.75 * bf(0.25 * math.tanh(0.75))),
             "unrounded state": 0.25 * s1 + 0.75 * math.tanh(0.75 * s1)}
    sg = lambda x: 1.0 / (1.0 + math.exp(-x))
    w1 = sg(0.75) * math.tanh(math.log(3.0))           # rows exchanged: g from the
    slips["gate and candidate rows exchanged"] = (      # candidate row, tanh(ln 3) candidate
        (1 - sg(0.75 * bf(w1))) * w1 + sg(0.75 * bf(w1)) * math.tanh(math.log(3.0)))
    for name, wrong in slips.items():
        assert abs(wrong - s2) > 1e-6, name


def test_greedy_ties_pick_lowest_id():
    R, G, V = 2, 2, 9
    base = np.zeros((R, G, V))
    base[:, :, 3] = 1.0
    base[:, :, 6] = 1.0
    out = oracle.markov_draft(base, np.zeros((R, G, 2)), np.zeros(R, int),
                              np.zeros((V, 2)), np.zeros((2, V)), np.zeros(4), np.ones(G),
                              0.0, 0)
    assert np.all(out["tokens"] == 3)


def test_confidence_head_brute_force():
    base, h, anchor, W1, W2, w, T = _tiny_draft_inputs()
    R, G, V = base.shape
    d = h.shape[2]
    out = oracle.markov_draft(base, h, anchor, W1, W2, w, T, 0.0, 0)
    prev = anchor.copy()
    for k in range(G):
        for rq in range(R):
            cat = list(h[rq, k]) + list(W1[prev[rq]])   # [h_k; W1[x_{k-1}]]
            z = sum(wi * xi for wi, xi in zip(w, cat))
            c = 1.0 / (1.0 + math.exp(-z / T[k]))
            assert abs(out["conf"][rq, k] - c) < 1e-12
            assert abs(out["z"][rq, k] - z) < 1e-12
        prev = out["tokens"][:, k]
    # T = 1 is the plain sigmoid; a hotter temperature pulls c toward 1/2
    o1 = oracle.markov_draft(base, h, anchor, W1, W2, w, np.ones(G), 0.0, 0)
    np.testing.assert_allclose(o1["conf"], sigmoid(o1["z"]), rtol=0, atol=0)
    o3 = oracle.markov_draft(base, h, anchor, W1, W2, w, 3 * np.ones(G), 0.0, 0)
    assert np.all(np.abs(o3["conf"] - 0.5) <= np.abs(o1["conf"] - 0.5) + 1e-15)
    assert d == 5


@pytest.mark.parametrize("tau,block", [(0.7, 64), (1.0, 64), (1.6, 64), (1.0, 2), (0.7, 4)])
def test_gumbel_max_follows_softmax(tau, block):
    """Sampled draft tokens follow softmax(l / tau) (Gumbel-max law), with the
    vocabulary in one block (plain Gumbel-max) or cut into several."""
    V, N = 6, 60000
    logits = np.array([0.3, -1.0, 1.2, 0.0, 2.0, -0.4])
    base = np.broadcast_to(logits, (N, 1, V)).copy()
    out = oracle.markov_draft(base, np.zeros((N, 1, 1)), np.zeros(N, int),
                              np.zeros((V, 1)), np.zeros((1, V)), np.zeros(2), np.ones(1),
                              tau, seed=2024, block=block)
    counts = np.bincount(out["tokens"][:, 0], minlength=V)
    p = np.exp(logits / tau)
    p /= p.sum()
    assert stats.chisquare(counts, N * p).pvalue > 1e-4
    # log p_d of the sampled token is reported
    np.testing.assert_allclose(out["logp"][:, 0], np.log(p[out["tokens"][:, 0]]), atol=1e-12)


def test_two_level_gumbel_law_with_excluded_entries_and_ragged_block():
    """Blocks of 3 over V = 8 (last block of 2); one whole block and one more
    entry at -inf.  Frequencies follow softmax over the finite entries, the
    excluded ids never come up, and each token lies in its row's top block."""
    N, block = 90000, 3
    score = np.array([0.4, -0.7, 1.1, -np.inf, -np.inf, -np.inf, 0.9, -np.inf])
    smp = oracle.dspark.gumbel_max(np.broadcast_to(score, (N, 8)), 77, 3, np.arange(N), 0, block)
    tok = smp["token"]
    counts = np.bincount(tok, minlength=8)
    assert counts[3] == counts[4] == counts[5] == counts[7] == 0
    fin = np.isfinite(score)
    p = np.exp(score[fin] - score[fin].max())
    p /= p.sum()
    assert stats.chisquare(counts[fin], N * p).pvalue > 1e-4
    assert np.array_equal(tok // block, np.argmax(smp["block_scores"], axis=1))
    assert np.all(np.isneginf(smp["block_scores"][:, 1]))     # the empty block


def test_two_level_gumbel_in_one_block_is_plain_gumbel_max():
    """With one block the draw is the textbook argmax(score + g_v)."""
    rng = np.random.default_rng(41)
    N, V = 500, 50
    score = rng.standard_normal((N, V)) * 2.0
    req = np.arange(N) + 1000
    smp = oracle.dspark.gumbel_max(score, 5, 2, req, philox.STREAM_BONUS)  # V <= 64
    g = philox.gumbel(5, 2, req[:, None], philox.STREAM_BONUS, np.arange(V, dtype=np.uint64)[None, :])
    assert np.array_equal(smp["token"], np.argmax(score + g, axis=1))
    # an all -inf row has nothing to draw
    empty = oracle.dspark.gumbel_max(np.full((1, V), -np.inf), 5, 2, 0, 0)
    assert empty["token"][0] == -1


def test_two_level_gumbel_block_choice_follows_block_mass():
    """Block b* comes up with probability Z_b / Z (the first level alone)."""
    N, block = 80000, 4
    rng = np.random.default_rng(42)
    score = rng.standard_normal(16) * 1.5
    smp = oracle.dspark.gumbel_max(np.broadcast_to(score, (N, 16)), 9, 1, np.arange(N), 2, block)
    counts = np.bincount(smp["token"] // block, minlength=4)
    Z = np.exp(score).reshape(4, block).sum(axis=1)
    assert stats.chisquare(counts, N * Z / Z.sum()).pvalue > 1e-4
    # a max over the block instead of its mass (a plausible slip) is rejected here
    M = np.exp(score.reshape(4, block).max(axis=1))
    assert stats.chisquare(counts, N * M / M.sum()).pvalue < 1e-6


# ---------------------------------------- a5-a7: survival, sort, Theta ---

def test_survival_products_left_to_right_float32():
    rng = np.random.default_rng(3)
    c = rng.random((5, 6)).astype(np.float32)
    c[2, 3] = 1.0
    a = oracle.survival(c)
    for rq in range(5):
        acc = np.float32(1.0)
        for j in range(6):
            acc = np.float32(acc * c[rq, j]) if j else np.float32(c[rq, 0])
            assert a[rq, j] == acc
        assert np.all(np.diff(a[rq]) <= 0)


def test_global_order_matches_lexsort():
    rng = np.random.default_rng(4)
    c = rng.random((9, 4)).astype(np.float32)
    c[::3, 1:] = 1.0                     # equal survival products inside a request
    c[4] = c[1]                          # equal products across requests
    a = oracle.survival(c)
    flat = a.reshape(-1)
    idx = np.arange(flat.size)
    want = np.lexsort((idx, -flat.astype(np.float64)))
    assert np.array_equal(oracle.global_order(a), want)


def _sps_tables(n):
    B = np.arange(1, n + 1, dtype=np.float64)
    rng = np.random.default_rng(n)
    return {
        "linear": 1000 * (1 - (B - 1) / (2 * n)),
        "concave": 1000 * (1 - 0.75 * ((B - 1) / (n - 1)) ** 2),
        "stair": 1000 / (1 + 0.15 * np.floor((B - 1) / 3)),
        "noisy": np.sort(rng.uniform(100, 1000, n))[::-1] * (1 + 0.05 * rng.random(n)),
        "flat": np.full(n, 500.0),
    }


@pytest.mark.parametrize("R,G", [(1, 4), (2, 3), (3, 3), (4, 2), (3, 4)])
def test_unconstrained_theta_is_bruteforce_optimum(R, G):
    rng = np.random.default_rng(10 * R + G)
    for trial in range(4):
        c = (0.05 + 0.95 * rng.random((R, G))).astype(np.float32)
        if trial == 3:
            c[0, :] = 1.0
        for name, sps in _sps_tables(R * (G + 1)).items():
            sps32 = sps.astype(np.float32)
            s = oracle.schedule(c, sps32, oracle.UNCONSTRAINED)
            a = s["a"]
            best = max(oracle.theta_of_lengths(a, lens, sps32)
                       for lens in itertools.product(range(G + 1), repeat=R))
            assert s["theta"] == pytest.approx(best, rel=1e-12), name
            assert oracle.theta_of_lengths(a, s["len"], sps32) == pytest.approx(best, rel=1e-12)
            assert s["len"].sum() == s["K"]


def _bruteforce_best_theta(a, sps):
    """max over every allocation l in {0..G}^R of Theta(l), by enumeration."""
    R, G = a.shape
    best = -np.inf
    for lens in itertools.product(range(G + 1), repeat=R):
        B = sum(1 + l for l in lens)
        tau = sum(1.0 + float(np.sum(a[r, :l], dtype=np.float64)) for r, l in enumerate(lens))
        best = max(best, tau * float(sps[B - 1]))
    return best


def test_async_schedule_uses_the_prediction_of_two_rounds_back():
    """Round t admits the top K*_{t-2} by its own survival products; K*_t is the
    budget maximising Theta on round t alone."""
    rng = np.random.default_rng(21)
    R, G, T = 5, 3, 7
    sps = _sps_tables(R * (G + 1))["stair"].astype(np.float32)
    rounds = [(0.05 + 0.95 * rng.random((R, G))).astype(np.float32) for _ in range(T)]
    out = oracle.schedule_async(rounds, sps, 4, 9)
    assert out["K_used"][0] == 4 and out["K_used"][1] == 9
    for t in range(2, T):
        assert out["K_used"][t] == out["K_pred"][t - 2]
    for t, c in enumerate(rounds):
        a = oracle.survival(c)
        lens = out["len"][t]
        assert lens.sum() == out["K_used"][t]
        # the admitted set is the top-K of this round's products (prefix-closed per request)
        flat = a.reshape(-1).astype(np.float64)
        admitted = np.zeros(R * G, bool)
        for r in range(R):
            admitted[r * G:r * G + lens[r]] = True
        if admitted.any() and (~admitted).any():
            assert flat[admitted].min() >= flat[~admitted].max()
        # the prediction is that round's Theta optimum (brute force over allocations)
        best = _bruteforce_best_theta(a, sps)
        K_p = out["K_pred"][t]
        th_p = oracle.schedule(c, sps, oracle.FIXED_K, K_p)["theta"]
        assert th_p == pytest.approx(best, rel=1e-12)


def test_async_schedule_with_steady_confidences_reaches_the_optimum():
    rng = np.random.default_rng(22)
    R, G = 4, 3
    c = (0.05 + 0.95 * rng.random((R, G))).astype(np.float32)
    sps = _sps_tables(R * (G + 1))["concave"].astype(np.float32)
    out = oracle.schedule_async([c] * 5, sps, 0, R * G)
    best = _bruteforce_best_theta(oracle.survival(c), sps)
    assert out["theta"][0] <= best * (1 + 1e-12)       # any budget is at most the optimum
    for t in range(2, 5):
        assert out["theta"][t] == pytest.approx(best, rel=1e-12)


def test_ece_hand_worked_values():
    # one sample per bin: |0-0.05| + |0-0.15| + |1-0.95| + |1-0.85| over 4
    assert oracle.expected_calibration_error([0.05, 0.15, 0.95, 0.85], [0, 0, 1, 1], 10) == \
        pytest.approx(0.1, abs=1e-7)
    # one bin holding all three: |1 - (0.31 + 0.33 + 0.35)| / 3
    assert oracle.expected_calibration_error([0.31, 0.33, 0.35], [1, 0, 0], 10) == \
        pytest.approx(0.01 / 3, abs=1e-7)
    # 1.0 lands in the last bin, 0.0 in the first; perfectly calibrated extremes
    assert oracle.expected_calibration_error([1.0, 0.0], [1, 0], 15) == 0.0


def _planted_sts_data(T_star, N, seed):
    """Confidence logits and accepted counts drawn from a model whose prefix
    survival is exactly prod_j sigmoid(z_j / T*_j)."""
    rng = np.random.default_rng(seed)
    G = len(T_star)
    z = rng.normal(1.2, 2.0, (N, G)).astype(np.float32)
    p = 1.0 / (1.0 + np.exp(-z.astype(np.float64) / np.asarray(T_star)))
    ok = rng.random((N, G)) < p
    accepted = np.where(ok.all(axis=1), G, np.argmin(ok, axis=1))
    return z, accepted


def test_sts_recovers_planted_temperatures():
    T_star = [1.4, 0.7, 2.2, 1.0]
    z, accepted = _planted_sts_data(T_star, 200_000, 31)
    grid = np.linspace(0.5, 3.0, 51)
    fit = oracle.sts_fit(z, accepted, grid, 15)
    assert np.all(np.abs(fit["T"] - np.asarray(T_star)) <= 0.15), fit["T"]
    assert np.all(fit["ece"] < 0.01)
    # calibrating each conditional c_j against the prefix label (a plausible slip)
    # would pick far colder temperatures from position 2 on
    label2 = accepted >= 2
    c2 = 1.0 / (1.0 + np.exp(-z[:, 1].astype(np.float64) / fit["T"][1]))
    assert oracle.expected_calibration_error(c2, label2, 15) > 5 * fit["ece"][1]


def test_sts_is_equivariant_to_logit_scale():
    z, accepted = _planted_sts_data([1.1, 1.7, 0.9], 20_000, 32)
    grid = np.linspace(0.5, 3.0, 26)
    a = oracle.sts_fit(z, accepted, grid, 10)
    b = oracle.sts_fit(z * 2, accepted, grid * 2, 10)  # z/T unchanged, exactly in float32
    assert np.array_equal(b["T"], a["T"] * 2)
    assert np.array_equal(b["ece"], a["ece"])


def test_admitted_set_is_prefix_closed_and_top_k():
    rng = np.random.default_rng(7)
    c = (0.05 + 0.95 * rng.random((20, 5))).astype(np.float32)
    c[3, 1:4] = 1.0
    sps = _sps_tables(120)["stair"].astype(np.float32)
    for mode, kf in [(oracle.UNCONSTRAINED, 0), (oracle.BREAK, 0), (oracle.FIXED_K, 37)]:
        s = oracle.schedule(c, sps, mode, kf)
        a = s["a"]
        admitted = {(i // 5, i % 5) for i in s["order"][:s["K"]]}
        for (rq, j) in admitted:
            assert j == 0 or (rq, j - 1) in admitted
        assert sorted(admitted) == sorted((rq, j) for rq in range(20) for j in range(s["len"][rq]))
        # admitted products dominate the rejected ones
        if 0 < s["K"] < 100:
            amin = min(a[rq, j] for rq, j in admitted)
            amax = max(a[rq, j] for rq in range(20) for j in range(5) if (rq, j) not in admitted)
            assert amin >= amax
    assert oracle.schedule(c, sps, oracle.FIXED_K, 37)["K"] == 37
    assert oracle.schedule(c, sps, oracle.FIXED_K, 1000)["K"] == 100


def test_break_mode_first_local_maximum():
    rng = np.random.default_rng(8)
    for trial in range(20):
        R, G = 6, 4
        c = (0.05 + 0.95 * rng.random((R, G))).astype(np.float32)
        sps = _sps_tables(R * (G + 1))
        s = oracle.schedule(c, sps["stair"].astype(np.float32), oracle.BREAK)
        th = s["thetas"]
        K = s["K"]
        assert all(th[i + 1] > th[i] for i in range(K))
        assert K == R * G or th[K + 1] <= th[K]
        # with a linear SPS table Theta(K) is concave, so break = global search
        lin = sps["linear"].astype(np.float32)
        assert (oracle.schedule(c, lin, oracle.BREAK)["K"]
                == oracle.schedule(c, lin, oracle.UNCONSTRAINED)["K"])


def test_theta_closed_form_on_hand_example():
    # two requests, gamma 2: c = [[.5, .5], [.9, .1]]  -> a = [[.5,.25],[.9,.09]]
    c = np.array([[0.5, 0.5], [0.9, 0.1]], dtype=np.float32)
    sps = np.array([100, 100, 100, 90, 80, 10], dtype=np.float32)
    s = oracle.schedule(c, sps, oracle.UNCONSTRAINED)
    # sorted a: .9 (1,1), .5 (0,1), .25 (0,2), .09 (1,2)
    th = [2 * 100, 2.9 * 100, 3.4 * 90, 3.65 * 80, 3.74 * 10]
    np.testing.assert_allclose(s["thetas"], th, rtol=1e-7)
    assert s["K"] == 2 and list(s["len"]) == [1, 1]
    assert oracle.schedule(c, sps, oracle.BREAK)["K"] == 3 - 1


def test_theta_fixed_point_rounding_against_exact_rationals():
    """S_K counts the products in 2^-48 units, each rounded to nearest with halves
    up; Theta(K) is that sum times SPS, rounded once.  Pinned with exact
    rationals on the half-unit boundary (2^-49 rounds up, the float below it
    down), a product of 1 and one with a fraction of a unit."""
    from fractions import Fraction
    half = np.float32(2.0 ** -49)
    a = np.array([[1.0, half, np.nextafter(half, np.float32(0)), 0.3]], dtype=np.float32)
    sps = np.array([7.0, 3.0, 5.0, 2.0, 9.0], dtype=np.float32)
    order = oracle.global_order(a)
    got = oracle.dspark.theta_curve(a, order, sps)
    units = [int(Fraction(float(a.reshape(-1)[i])) * 2 ** 48 + Fraction(1, 2)) for i in order]
    assert units[2:] == [1, 0]                       # the boundary: half up, below half down
    RS = 1 << 48
    want = [float(Fraction(RS) * Fraction(float(sps[0])) / 2 ** 48)]
    for K, u in enumerate(units, start=1):
        RS += u
        want.append(float(Fraction(RS) * Fraction(float(sps[K])) / 2 ** 48))
    assert got.tolist() == want


def _exact_thetas(a, order, sps):
    """Theta(K) in exact rationals from the float32 products and table entries."""
    from fractions import Fraction
    R = a.shape[0]
    flat = a.reshape(-1)
    S = Fraction(0)
    out = [Fraction(R) * Fraction(float(sps[R - 1]))]
    for K, i in enumerate(order, start=1):
        S += Fraction(float(flat[i]))
        out.append((R + S) * Fraction(float(sps[R + K - 1])))
    return out


def test_fixed_point_theta_decides_as_exact_arithmetic_outside_its_rounding_band():
    """The fixed-point S_K moves R + S_K by at most gamma 2^-49 of itself, and
    the two float64 roundings add 2^-52.  Wherever the exact optimum beats every
    other budget by more than twice that, the fixed-point argmax (and the break
    mode's first drop) is the exact one.  Random confidences, some equal to 1
    and some repeated, over linear, concave, stepped and random tables."""
    from fractions import Fraction
    rng = np.random.default_rng(21)
    decided = 0
    for case in range(300):
        R = int(rng.integers(1, 30))
        G = int(rng.integers(1, 9))
        c = rng.uniform(0.3, 1.0, (R, G)).astype(np.float32)
        c[rng.random((R, G)) < 0.1] = 1.0
        if case % 3 == 0:                              # repeated values: ties in the sort
            c = np.round(c * 8) / 8
        n = R * (G + 1)
        B = np.arange(1, n + 1, dtype=np.float64)
        kind = case % 4
        if kind == 0:
            sps = 1000.0 * (1.0 - (B - 1) / (2.0 * n))
        elif kind == 1:
            sps = 1000.0 * (1.0 - 0.75 * ((B - 1) / n) ** 2)
        elif kind == 2:
            sps = 1000.0 / (1.0 + 0.15 * np.floor((B - 1) / max(1, n // 7)))
        else:
            sps = np.sort(rng.uniform(100, 1000, n))[::-1]
        sps = sps.astype(np.float32)
        o = oracle.schedule(c, sps, oracle.UNCONSTRAINED)
        ex = _exact_thetas(o["a"], o["order"], sps)
        k_exact = max(range(len(ex)), key=lambda K: (ex[K], -K))
        eps = Fraction(G, 2 ** 49) + Fraction(1, 2 ** 52)
        others = [ex[K] for K in range(len(ex)) if K != k_exact]
        if not others or all(ex[k_exact] > t * (1 + 2 * eps) for t in others):
            assert o["K"] == k_exact, case
            decided += 1
        # break mode: the first K whose next budget does not raise Theta
        steps = [ex[K + 1] / ex[K] - 1 for K in range(len(ex) - 1)]
        if all(abs(x) > 2 * eps for x in steps):
            kb = next((K for K, x in enumerate(steps) if x < 0), len(ex) - 1)
            assert oracle.schedule(c, sps, oracle.BREAK)["K"] == kb, case
    assert decided > 250


# ------------------------------------------------------------ a8: verify ---

def test_confidence_label_identity():
    rng = np.random.default_rng(11)
    for _ in range(50):
        V = rng.integers(2, 40)
        p = rng.dirichlet(np.ones(V) * rng.uniform(0.1, 3))
        q = rng.dirichlet(np.ones(V) * rng.uniform(0.1, 3))
        lab = oracle.confidence_label(p, q)
        assert lab == pytest.approx(np.minimum(p, q).sum(), abs=1e-12)
        assert 0.0 <= lab <= 1.0
    assert oracle.confidence_label(p, p) == pytest.approx(1.0)


def test_acceptance_rate_equals_confidence_label():
    """P(accept position 1) = sum_v min(p_d, p_t) = 1 - TV(p_d, p_t)."""
    V, N, tau = 7, 40000, 1.0
    rng = np.random.default_rng(12)
    ld = rng.standard_normal(V) * 1.3
    lt = rng.standard_normal(V) * 1.3
    base = np.broadcast_to(ld, (N, 1, V)).copy()
    dr = oracle.markov_draft(base, np.zeros((N, 1, 1)), np.zeros(N, int), np.zeros((V, 1)),
                             np.zeros((1, V)), np.zeros(2), np.ones(1), tau, seed=5)
    target = np.broadcast_to(np.stack([lt, lt]), (N, 2, V)).copy()
    res = oracle.verify(dr["tokens"], np.ones(N, int), base, target, tau, seed=6)
    pd = np.exp(ld - oracle.dspark.logsumexp(ld))
    pt = np.exp(lt - oracle.dspark.logsumexp(lt))
    label = oracle.confidence_label(pd, pt)
    rate = res["accepted"].mean()
    assert abs(rate - label) < 4 * math.sqrt(label * (1 - label) / N)
    # reversing the ratio (a plausible slip) would give a different rate here
    wrong = np.sum(pd * np.minimum(1, pd / pt))
    assert abs(wrong - label) > 8 * math.sqrt(label * (1 - label) / N)


def _one_position_verify(ld, lt, N, seed, block=64):
    """N requests of one admitted position: drafts sampled from softmax(ld),
    target row softmax(lt).  Returns the verify result and p_d, p_t."""
    V = ld.size
    base = np.broadcast_to(ld, (N, 1, V)).copy()
    dr = oracle.markov_draft(base, np.zeros((N, 1, 1)), np.zeros(N, int), np.zeros((V, 1)),
                             np.zeros((1, V)), np.zeros(2), np.ones(1), 1.0, seed=seed,
                             block=block)
    target = np.broadcast_to(np.stack([lt, lt]), (N, 2, V)).copy()
    res = oracle.verify(dr["tokens"], np.ones(N, int), base, target, 1.0, seed=seed + 1,
                        block=block)
    pd = np.exp(ld - oracle.dspark.logsumexp(ld))
    pt = np.exp(lt - oracle.dspark.logsumexp(lt))
    return res, pd, pt


@pytest.mark.parametrize("block,sup", [(1, 4), (2, 4)])
def test_three_level_trial_draw_follows_softmax(block, sup):
    """The residual trials' proposal (super-blocks, blocks, ids) samples
    softmax(score): V = 42 with ragged super-blocks and blocks and three ids at
    -inf, which never come up."""
    V, N = 42, 15000
    rng = np.random.default_rng(61)
    score = rng.standard_normal(V) * 1.1
    score[[3, 17, 41]] = -np.inf
    toks = np.array([oracle.dspark.gumbel_max_trial(score, 11, 2, n, 16, block, sup)["token"]
                     for n in range(N)])
    counts = np.bincount(toks, minlength=V)
    p = np.exp(score - oracle.dspark.logsumexp(score))
    assert counts[[3, 17, 41]].sum() == 0
    keep = p > 0
    assert stats.chisquare(counts[keep], N * p[keep]).pvalue > 1e-4


@pytest.mark.parametrize("sup", [16, 1])
def test_residual_draw_follows_the_residual_law(monkeypatch, sup):
    """On rejection the corrected token follows norm(max(0, p_t - p_d)) (the
    residual of speculative sampling), with the sampler's blocks of 3 ids over
    V = 7 (a ragged block; with super-blocks of one block, three of them), and
    the draws come from the trials."""
    monkeypatch.setattr(oracle.dspark, "TRIAL_SUPER", sup)
    ld = np.array([1.1, -0.3, 0.4, 2.0, -1.2, 0.0, 0.7])
    lt = np.array([0.2, 0.9, -0.5, 1.0, 0.3, 1.4, -0.8])
    res, pd, pt = _one_position_verify(ld, lt, 20000, 31, block=3)
    rej = res["accepted"] == 0
    q = np.maximum(pt - pd, 0.0)
    q /= q.sum()
    counts = np.bincount(res["bonus"][rej], minlength=ld.size)
    assert rej.sum() > 4000
    assert counts[q == 0].sum() == 0  # ids with p_d >= p_t are never the correction
    keep = q > 0
    assert stats.chisquare(counts[keep], rej.sum() * q[keep]).pvalue > 1e-4
    assert np.all(res["final_kind"][rej] == 4)
    # a trial that kept every proposal would give the target row itself
    assert stats.chisquare(counts, rej.sum() * pt).pvalue < 1e-8


def test_residual_trials_are_geometric_in_the_residual_mass():
    """Each trial keeps its proposal with probability sum(max(0, p_t - p_d)), so
    the trials of a rejected row are geometric with that mean inverse: a kept
    proposal that skipped the test, or a test with the ratio reversed, moves it."""
    ld = np.array([0.5, 0.1, -0.2, 0.8, 0.0])
    lt = np.array([0.6, -0.1, 0.1, 0.7, -0.2])
    res, pd, pt = _one_position_verify(ld, lt, 30000, 41)
    rej = res["accepted"] == 0
    z = np.maximum(pt - pd, 0.0).sum()
    n = res["trials"][rej]
    assert 0.05 < z < 0.2 and n.size > 1500
    sem = math.sqrt((1 - z) / z ** 2 / n.size)
    assert abs(n.mean() - 1 / z) < 4 * sem
    assert np.all(res["trials"][~rej] == 0)


def test_residual_without_trials_is_the_explicit_draw(monkeypatch):
    """With no trials every rejected row takes the explicit residual, drawn by
    Gumbel-max from log max(0, p_t - p_d): the same law."""
    monkeypatch.setattr(oracle.dspark, "RESIDUAL_TRIALS", 0)
    ld = np.array([1.1, -0.3, 0.4, 2.0, -1.2, 0.0, 0.7])
    lt = np.array([0.2, 0.9, -0.5, 1.0, 0.3, 1.4, -0.8])
    res, pd, pt = _one_position_verify(ld, lt, 15000, 51)
    rej = res["accepted"] == 0
    q = np.maximum(pt - pd, 0.0)
    q /= q.sum()
    counts = np.bincount(res["bonus"][rej], minlength=ld.size)
    keep = q > 0
    assert counts[~keep].sum() == 0
    assert stats.chisquare(counts[keep], rej.sum() * q[keep]).pvalue > 1e-4
    assert np.all(res["final_kind"][rej] == 1) and np.all(res["trials"] == 0)


def test_greedy_verify_accepts_own_argmax():
    rng = np.random.default_rng(13)
    R, G, V = 6, 4, 50
    target = rng.standard_normal((R, G + 1, V))
    tokens = np.argmax(target[:, :G], axis=2)
    lens = np.array([0, 1, 2, 3, 4, 4])
    res = oracle.verify(tokens, lens, None, target, 0.0, 0)
    assert list(res["accepted"]) == list(lens)
    for i in range(R):
        assert res["bonus"][i] == np.argmax(target[i, lens[i]])
    # corrupt one draft: rejected there, the correction is that row's argmax
    tokens2 = tokens.copy()
    tokens2[5, 1] = (tokens2[5, 1] + 1) % V
    res2 = oracle.verify(tokens2, lens, None, target, 0.0, 0)
    assert res2["accepted"][5] == 1 and res2["bonus"][5] == np.argmax(target[5, 1])


def test_sampling_verify_identical_distributions_always_accepts():
    rng = np.random.default_rng(14)
    R, G, V = 50, 3, 20
    logits = rng.standard_normal((R, G + 1, V))
    tokens = rng.integers(0, V, (R, G))
    lens = np.full(R, G)
    res = oracle.verify(tokens, lens, logits[:, :G], logits, 1.0, 9)
    assert np.all(res["accepted"] == G)


def _markov_target_rounds(mode, V=6, G=3, N=30000, L=3, seed=0, block=2):
    """Decode L tokens per trial by draft -> schedule -> verify rounds (oracle only).

    Target: a first-order Markov chain P_t(next | prev).  Draft: base logits per
    position plus a low-rank Markov bias; confidences from the confidence head.
    Every draw cuts the vocabulary into sampler blocks of `block` ids (three
    blocks over V = 6 by default), so both levels of the sampler take part.
    Returns the first L emitted tokens of each trial and the exact target joint.
    """
    rng = np.random.default_rng(seed)
    logPt = rng.standard_normal((V, V)) * 1.2
    Pt = np.exp(logPt - oracle.dspark.logsumexp(logPt, axis=1)[:, None])
    base0 = rng.standard_normal((G, V)) * 0.8
    r = 2
    W1 = rng.standard_normal((V, r))
    W2 = rng.standard_normal((r, V)) * 0.8
    d = 3
    h = rng.standard_normal((N, G, d))
    w = rng.standard_normal(d + r) * 1.5
    T = np.array([1.0, 1.3, 1.7])[:G]
    sps = 1000 * (1 - np.arange(N * (G + 1)) / (N * (G + 1) * 1.1))
    start = 2
    anchor = np.full(N, start)
    emitted = [[] for _ in range(N)]
    pending = [N * G // 3, N * G // 2]   # async mode: the first two rounds' capacities
    rnd = 0
    while min(len(e) for e in emitted) < L:
        base = np.broadcast_to(base0, (N, G, V)).copy()
        dr = oracle.markov_draft(base, h, anchor, W1, W2, w, T, 1.0, seed=1000 + rnd,
                                 keep_logits=True, block=block)
        x = dr["tokens"]
        prev = np.concatenate([anchor[:, None], x], axis=1)        # x_0..x_G
        target = logPt[prev]                                       # row j-1 | x_{j-1}
        if mode == "full":
            lens = np.full(N, G)
        elif mode == "random":
            lens = rng.integers(0, G + 1, N)
        elif mode == "break":
            lens = oracle.schedule(dr["conf"].astype(np.float32), sps, oracle.BREAK)["len"]
        elif mode == "fixed_k":
            lens = oracle.schedule(dr["conf"].astype(np.float32), sps, oracle.FIXED_K,
                                   N * G // 2)["len"]
        elif mode == "async":
            # capacity predicted two rounds earlier, top-K on this round's products
            c32 = dr["conf"].astype(np.float32)
            lens = oracle.schedule(c32, sps, oracle.FIXED_K, pending[rnd % 2])["len"]
            pending[rnd % 2] = oracle.schedule(c32, sps, oracle.UNCONSTRAINED)["K"]
        res = oracle.verify(x, lens, dr["logits"], target, 1.0, seed=5000 + rnd, block=block)
        for i in range(N):
            n = res["accepted"][i]
            emitted[i].extend(list(x[i, :n]) + [res["bonus"][i]])
            anchor[i] = emitted[i][-1]
        rnd += 1
    first = np.array([e[:L] for e in emitted])
    joint = np.ones([V] * L)
    for idx in itertools.product(range(V), repeat=L):
        p, prv = 1.0, start
        for t in idx:
            p *= Pt[prv, t]
            prv = t
        joint[idx] = p
    return first, joint


@pytest.mark.slow
@pytest.mark.parametrize("mode", ["full", "random", "break", "fixed_k", "async"])
def test_draft_schedule_verify_is_lossless(mode):
    """Chi-square: emitted tokens follow the target chain in non-anticipating modes."""
    V, L = 6, 3
    first, joint = _markov_target_rounds(mode, V=V, L=L, N=16000, seed=zlib.crc32(mode.encode()) % 1000)
    cells = np.ravel_multi_index(first.T, [V] * L)
    counts = np.bincount(cells, minlength=V ** L)
    exp = joint.reshape(-1) * first.shape[0]
    keep = exp >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    ex = np.append(exp[keep], exp[~keep].sum())
    assert stats.chisquare(obs, ex).pvalue > 1e-4
    # and marginally per position
    for t in range(L):
        m = np.bincount(first[:, t], minlength=V)
        pm = joint.sum(axis=tuple(i for i in range(L) if i != t))
        assert stats.chisquare(m, pm * first.shape[0]).pvalue > 1e-4


def test_zero_length_and_bonus_row():
    rng = np.random.default_rng(15)
    R, G, V = 30, 2, 12
    target = rng.standard_normal((R, G + 1, V))
    res = oracle.verify(np.zeros((R, G), int), np.zeros(R, int), None, target, 0.0, 0)
    assert np.all(res["accepted"] == 0)
    assert np.array_equal(res["bonus"], np.argmax(target[:, 0], axis=1))
    # sampling mode with nothing admitted: bonus is a plain sample from target row 1
    res = oracle.verify(np.zeros((R, G), int), np.zeros(R, int), np.zeros((R, G, V)),
                        target, 1.0, 3)
    assert np.all(res["accepted"] == 0)
    g = philox.gumbel(3, 1, np.arange(R)[:, None], philox.STREAM_BONUS,
                      np.arange(V, dtype=np.uint64)[None, :])
    assert np.array_equal(res["bonus"], np.argmax(target[:, 0] + g, axis=1))
