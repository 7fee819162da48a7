"""GPU parity: every stage of the CUDA path against the CPU oracle, through the C-ABI.

Sizes span several tiles with a ragged tail and finish in seconds on the oracle;
full-size checks at the benchmark's workload are in test_gpu_fullsize.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import (TOL_DRAFT, compare_draft, compare_verify, flag_budget, host,
                    schedule_is_robust, sorted_order_ok)

pytestmark = pytest.mark.gpu

dsp = pytest.importorskip("speculative_decoding_draft_02_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from speculative_decoding_draft_02_gb300 import build
    build.build()
    dsp.load_library()
    yield
    assert dsp.dspark_device_status() == 0


def dev(t, dtype=None):
    t = t.to("cuda")
    return t.to(dtype) if dtype is not None else t


SHAPES = [  # (R, gamma, V, r, d)
    (4, 5, 1024, 64, 256),       # the tiny workload
    (37, 4, 1000, 128, 320),     # ragged in rows and vocabulary
    (3, 3, 4104, 256, 512),      # vocabulary tail of 8
    (130, 2, 2056, 64, 192),     # rows past one 128-row tile
    (1, 1, 520, 64, 64),         # degenerate: one request, one position
]


def _weights(R, G, V, r, d, seed):
    w = workloads.WORKLOADS["tiny"].with_(R=R, gamma=G, V=V, r=r, d=d, anchor_hi=V)
    return workloads.make_inputs(w, seed=seed, with_target_noise=False)


# ------------------------------------------------------------------ a1 ----

# 17 and 5 row blocks of 128: the CTA-pair LM head (an odd count leaves the
# last pair's second half empty); 16 and 17 rows: the last size of the swapped-
# operand kernel and the first of the row-tiled one
@pytest.mark.parametrize("shape", SHAPES + [(520, 4, 1000, 64, 128), (160, 4, 1000, 64, 128),
                                            (4, 4, 4104, 64, 128), (17, 1, 4104, 64, 128)])
def test_lm_head_matches_oracle(shape):
    R, G, V, r, d = shape
    inp = _weights(R, G, V, r, d, seed=100 + V)
    h = inp["h"].reshape(R * G, d)
    want = oracle.base_logits(h, inp["W_lm"])                       # bf16-rounded
    dims = dsp.dims_of(R, G, V, r, d)
    out = torch.empty((R * G, V), dtype=torch.bfloat16, device="cuda")
    dsp.dspark_lm_head(dims, dev(h, torch.bfloat16), dev(inp["W_lm"], torch.bfloat16), out)
    got = host(out).astype(np.float64)
    exact = oracle.base_logits(h, inp["W_lm"], bf16_out=False)
    # within one bf16 rounding step of the exact value (1e-2 relative is the bar)
    err = np.abs(got - exact)
    assert np.all(err <= 2.0 ** -8 * np.abs(exact) + 1e-6), err.max()
    assert np.mean(got == want) > 0.999


def test_pack_w2_is_transpose():
    inp = _weights(2, 2, 1000, 128, 64, seed=7)
    dims = dsp.dims_of(2, 2, 1000, 128, 64)
    W2 = dev(inp["W2"], torch.bfloat16)
    W2t = torch.empty((1000, 128), dtype=torch.bfloat16, device="cuda")
    dsp.dspark_pack_w2(dims, W2, W2t)
    assert torch.equal(W2t, W2.t().contiguous())


# --------------------------------------------------------------- a2-a4 ----

def _draft_case(shape, tau, seed):
    R, G, V, r, d = shape
    inp = _weights(R, G, V, r, d, seed=seed)
    base = workloads.random_normal((R, G, V), 1.0, seed + 1)
    orc = oracle.markov_draft(base, inp["h"], inp["anchor"], inp["W1"], inp["W2"],
                              inp["w_conf"], inp["T"], tau, seed=12345 + seed, keep_scores=True)
    head = dsp.DraftHead.from_weights(R, G, inp["W_lm"], inp["W1"], inp["W2"], inp["w_conf"],
                                      inp["T"])
    rnd = dsp.Round(head)
    rnd.base.copy_(dev(base.reshape(R * G, V)))
    dsp.dspark_markov_draft(head.dims, rnd.base, dev(inp["h"], torch.bfloat16).contiguous(),
                            dev(inp["anchor"]), head.W1, head.W2t, head.w_conf, head.T, tau,
                            12345 + seed, rnd.tokens, rnd.conf, rnd.logp_d, rnd.lse_d,
                            rnd.ws_draft)
    return rnd, orc


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("tau", [0.0, 1.0, 0.6])
def test_markov_draft_matches_oracle(shape, tau):
    rnd, orc = _draft_case(shape, tau, seed=200 + shape[2])
    rep = compare_draft(rnd.tokens, rnd.conf, rnd.lse_d if tau > 0 else None,
                        rnd.logp_d if tau > 0 else None, orc, tau, tol_rel=TOL_DRAFT)
    print(f"{shape} tau={tau}: {rep.flagged} of {rep.compared} decisions in the tie band")
    assert rep.compared >= shape[0]
    assert rep.flagged <= flag_budget(rep.compared)
    assert dsp.dspark_device_status() == 0


def test_markov_zero_bias_is_parallel_argmax():
    """W2 = 0 gives plain parallel drafting: x_k = argmax of the base logits."""
    R, G, V, r, d = 9, 3, 1000, 64, 128
    inp = _weights(R, G, V, r, d, seed=31)
    inp["W2"] = torch.zeros_like(inp["W2"])
    base = workloads.random_normal((R, G, V), 1.0, 32)
    head = dsp.DraftHead.from_weights(R, G, inp["W_lm"], inp["W1"], inp["W2"], inp["w_conf"],
                                      inp["T"])
    rnd = dsp.Round(head)
    rnd.base.copy_(dev(base.reshape(R * G, V)))
    dsp.dspark_markov_draft(head.dims, rnd.base, dev(inp["h"], torch.bfloat16).contiguous(),
                            dev(inp["anchor"]), head.W1, head.W2t, head.w_conf, head.T, 0.0, 0,
                            rnd.tokens, rnd.conf, None, None, rnd.ws_draft)
    want = torch.argmax(base.float(), dim=2)  # first maximum on ties
    assert torch.equal(rnd.tokens.cpu().long(), want)


# --------------------------------------------------------------- a5-a7 ----

SPS_KINDS = ["linear", "concave", "stair"]


def sps_for(kind, n):
    """Positive SPS tables of n entries (the workloads' linear table is 64 long)."""
    if kind == "linear":
        B = torch.arange(1, n + 1, dtype=torch.float64)
        return (1000.0 * (1.0 - (B - 1.0) / (2.0 * n))).to(torch.float32)
    return workloads.sps_table(kind, n)


@pytest.mark.parametrize("R,G", [(4, 5), (1, 8), (64, 8), (256, 5), (1024, 7), (3, 1),
                                 (2047, 8)])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_schedule_matches_oracle(R, G, mode):
    for kind in SPS_KINDS:
        c = workloads.random_confidences(R, G, seed=R * 31 + G, ones_frac=0.05)
        n = R * (G + 1)
        sps = sps_for(kind, n)
        kf = (R * G) // 3
        o = oracle.schedule(c, sps, mode, kf)
        length = torch.empty(R, dtype=torch.int32, device="cuda")
        K = torch.empty(1, dtype=torch.int32, device="cuda")
        th = torch.empty(1, dtype=torch.float64, device="cuda")
        a = torch.empty((R, G), dtype=torch.float32, device="cuda")
        order = torch.empty(R * G, dtype=torch.int32, device="cuda")
        dsp.dspark_schedule(dev(c), R, G, dev(sps), mode, kf, length, K, th, a, order)
        assert np.array_equal(host(a), o["a"])                         # bit-exact f32 products
        assert np.array_equal(host(order), o["order"])                 # same total order
        # S_K in 2^-48 units and Theta in f64 on both sides: bit-exact
        assert int(K.item()) == o["K"], kind
        assert np.array_equal(host(length), o["len"]), kind
        assert float(th.item()) == o["theta"], kind


@pytest.mark.parametrize("R,G,kind", [(37, 4, "stair"), (64, 8, "concave"), (256, 5, "stair"),
                                        (1024, 7, "stair")])
def test_schedule_async_matches_oracle(R, G, kind):
    """Six rounds through one device ring: each round's admitted K is the
    optimum found two rounds earlier, its lengths the top-K of its own products."""
    T = 6
    rounds = [workloads.random_confidences(R, G, seed=1000 * R + 17 * t, ones_frac=0.02)
              for t in range(T)]
    sps = sps_for(kind, R * (G + 1))
    k0, k1 = (R * G) // 4, (R * G) // 2
    o = oracle.schedule_async(rounds, sps, k0, k1)
    ring = dsp.async_ring(k0, k1)
    length = torch.empty(R, dtype=torch.int32, device="cuda")
    K = torch.empty(1, dtype=torch.int32, device="cuda")
    th = torch.empty(1, dtype=torch.float64, device="cuda")
    for t, c in enumerate(rounds):
        before = host(ring).copy()
        dsp.dspark_schedule_async(dev(c), R, G, dev(sps), ring, length, K, th)
        after = host(ring)
        k_used = int(K.item())
        assert k_used == before[before[2] & 1]                 # the slot at the cursor
        assert after[2] == (before[2] ^ 1)                      # cursor flipped
        assert after[1 - (before[2] & 1)] == before[1 - (before[2] & 1)]
        assert k_used == o["K_used"][t]
        assert np.array_equal(host(length), o["len"][t])        # top-K: exact integers
        assert float(th.item()) == o["theta"][t]                 # same precision: bit-exact
        assert int(after[before[2] & 1]) == o["K_pred"][t]
    assert dsp.dspark_device_status() == 0


@pytest.mark.parametrize("shape", SHAPES)
def test_conf_logits_match_oracle(shape):
    R, G, V, r, d = shape
    inp = _weights(R, G, V, r, d, seed=400 + V)
    tokens = workloads.random_tokens(R, G, V, 401 + V)
    base = np.zeros((R, G, V))
    orc = oracle.markov_draft(base, inp["h"], inp["anchor"], inp["W1"], inp["W2"],
                              inp["w_conf"], inp["T"], 0.0, 0, forced=tokens)
    dims = dsp.dims_of(R, G, V, r, d)
    z = torch.empty((R, G), dtype=torch.float32, device="cuda")
    dsp.dspark_conf_logits(dims, dev(inp["h"], torch.bfloat16).contiguous(), dev(inp["anchor"]),
                           dev(tokens), dev(inp["W1"], torch.bfloat16),
                           dev(inp["w_conf"], torch.bfloat16), z)
    got = host(z).astype(np.float64)
    assert np.all(np.abs(got - orc["z"]) <= 1e-4 * np.maximum(1.0, np.abs(orc["z"])))
    assert dsp.dspark_device_status() == 0


def _planted_rounds(T_star, N, seed):
    g = torch.Generator().manual_seed(seed)
    G = len(T_star)
    z = (1.2 + 2.0 * torch.randn((N, G), generator=g)).float()
    p = torch.sigmoid(z.double() / torch.tensor(T_star, dtype=torch.float64))
    ok = torch.rand((N, G), generator=g, dtype=torch.float64) < p
    acc = torch.where(ok.all(dim=1), torch.full((N,), G), torch.argmin(ok.int(), dim=1))
    return z, acc.to(torch.int32)


@pytest.mark.parametrize("N,n_bins", [(1, 15), (777, 10), (100_000, 15), (400_000, 64)])
def test_sts_fit_matches_oracle(N, n_bins):
    T_star = [1.4, 0.7, 2.2, 1.0, 1.8]
    z, acc = _planted_rounds(T_star, N, seed=N + n_bins)
    grid = torch.linspace(0.5, 3.0, 51)
    o = oracle.sts_fit(z.numpy(), acc.numpy(), grid.numpy(), n_bins)
    G = len(T_star)
    T_out = torch.empty(G, dtype=torch.float32, device="cuda")
    ece = torch.empty(G, dtype=torch.float64, device="cuda")
    dsp.dspark_sts_fit(dev(z), dev(acc), dev(grid), n_bins, T_out, ece)
    got_T, got_e = host(T_out), host(ece)
    tol = 1e-4 + 8.0 / N  # f32 sigmoid rounding may move a sample across a bin edge
    for j in range(G):
        if got_T[j] != o["T"][j]:  # only a near tie of two grid values may separate them
            g = int(np.argmin(np.abs(grid.numpy() - got_T[j])))
            assert o["ece_grid"][j, g] - o["ece"][j] <= tol, (j, got_T[j], o["T"][j])
            break  # later positions build on a different (equally good) choice
        assert abs(got_e[j] - o["ece"][j]) <= tol, (j, got_e[j], o["ece"][j])
    assert dsp.dspark_device_status() == 0


def test_schedule_extremes():
    R, G = 50, 4
    c = workloads.random_confidences(R, G, seed=5)
    dec = torch.tensor(np.geomspace(1000, 1e-3, R * (G + 1)), dtype=torch.float32)
    flat = torch.full((R * (G + 1),), 500.0)
    neg = -torch.arange(1, R * (G + 1) + 1, dtype=torch.float32)  # meaningless but must be safe
    for sps, want_k in [(dec, 0), (flat, R * G), (neg, oracle.schedule(c, neg)["K"])]:
        length = torch.empty(R, dtype=torch.int32, device="cuda")
        K = torch.empty(1, dtype=torch.int32, device="cuda")
        th = torch.empty(1, dtype=torch.float64, device="cuda")
        dsp.dspark_schedule(dev(c), R, G, dev(sps), 0, 0, length, K, th)
        assert int(K.item()) == want_k
        assert int(length.sum().item()) == want_k
        assert sorted_order_ok(oracle.schedule(c, sps)["order"], oracle.survival(c))


def _schedule_gpu(c, R, G, sps, mode, kf=0):
    length = torch.empty(R, dtype=torch.int32, device="cuda")
    K = torch.empty(1, dtype=torch.int32, device="cuda")
    th = torch.empty(1, dtype=torch.float64, device="cuda")
    dsp.dspark_schedule(dev(c), R, G, dev(sps), mode, kf, length, K, th)
    return int(K.item()), host(length), float(th.item())


def test_schedule_at_the_size_limit_with_every_product_one():
    """R gamma = 16384 candidates, all survival products 1: the largest fixed-point
    sum, R + S_K = 2^15 units of 2^48 at K = n."""
    R, G = 16384, 1
    c = torch.ones((R, G), dtype=torch.float32)
    for kind in SPS_KINDS:
        sps = sps_for(kind, R * (G + 1))
        for mode in (0, 1):
            o = oracle.schedule(c, sps, mode)
            k, length, th = _schedule_gpu(c, R, G, sps, mode)
            assert k == o["K"] and th == o["theta"], (kind, mode)
            assert np.array_equal(length, o["len"])
    assert dsp.dspark_device_status() == 0


def test_schedule_with_nan_in_the_sps_table():
    """A NaN Theta never wins the argmax; break mode stops at it."""
    R, G = 40, 4
    c = workloads.random_confidences(R, G, seed=9)
    sps = sps_for("concave", R * (G + 1)).clone()
    best = oracle.schedule(c, sps)["K"]
    for at in (best, 3):
        bad = sps.clone()
        bad[R + at - 1] = float("nan")  # Theta(at) is NaN
        for mode in (0, 1):
            o = oracle.schedule(c, bad, mode)
            k, length, th = _schedule_gpu(c, R, G, bad, mode)
            assert k == o["K"], (at, mode)
            assert np.array_equal(length, o["len"])
            assert th == o["theta"] or (np.isnan(th) and np.isnan(o["theta"]))
    assert dsp.dspark_device_status() == 0


# ------------------------------------------------------------------ a8 ----

def _verify_case(shape, tau, seed, accept_bias=0.7, lens_kind="random", noise_std=0.3):
    R, G, V, r, d = shape
    inp = _weights(R, G, V, r, d, seed=seed)
    base = workloads.random_normal((R, G, V), 1.0, seed + 1)
    tokens = workloads.random_tokens(R, G, V, seed + 2)
    lens = workloads.random_lengths(R, G, seed + 3)
    if lens_kind == "full":
        lens = torch.full_like(lens, G)
    noise = workloads.random_normal((R, G + 1, V), noise_std, seed + 4, dtype=torch.float32)
    if tau == 0.0:
        target = workloads.random_normal((R, G + 1, V), 1.0, seed + 5)
        # make runs of accepted tokens likely: drafts equal the target argmax mostly
        am = torch.argmax(target[:, :G].float(), dim=2).to(torch.int32)
        pick = workloads.random_normal((R, G), 1.0, seed + 6, dtype=torch.float32) < accept_bias
        tokens = torch.where(pick, am, tokens)
        dl = None
        lse_d = logp_d = torch.zeros((R, G))
    else:
        orc_d = oracle.markov_draft(base, inp["h"], inp["anchor"], inp["W1"], inp["W2"],
                                    inp["w_conf"], inp["T"], tau, 0, forced=tokens,
                                    keep_logits=True)
        dl = orc_d["logits"]
        lse_d = torch.tensor(orc_d["lse"], dtype=torch.float32)
        logp_d = torch.tensor(orc_d["logp"], dtype=torch.float32)
        # target near the draft so that acceptance and rejection both happen
        t = np.concatenate([dl, dl[:, -1:]], axis=1) + noise.numpy()
        target = torch.tensor(t, dtype=torch.float32).to(torch.bfloat16)
    orc = oracle.verify(tokens, lens, dl, target, tau, seed=777 + seed)
    head = dsp.DraftHead.from_weights(R, G, inp["W_lm"], inp["W1"], inp["W2"], inp["w_conf"],
                                      inp["T"])
    rnd = dsp.Round(head)
    rnd.base.copy_(dev(base.reshape(R * G, V)))
    rnd.tokens.copy_(dev(tokens))
    rnd.len.copy_(dev(lens))
    rnd.lse_d.copy_(dev(lse_d))
    rnd.logp_d.copy_(dev(logp_d))
    rnd.verify(dev(inp["anchor"]), dev(target).contiguous(), tau, 777 + seed)
    return rnd, orc, lens


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("tau", [0.0, 1.0, 0.8])
def test_verify_matches_oracle(shape, tau):
    rnd, orc, lens = _verify_case(shape, tau, seed=300 + shape[2])
    flagged = compare_verify(rnd.accepted, rnd.bonus, orc, tau)
    print(f"verify {shape} tau={tau}: {flagged} of {shape[0]} requests in a tie band")
    assert flagged <= max(1, shape[0] // 50)
    acc = host(rnd.accepted)
    assert np.all(acc >= 0) and np.all(acc <= host(lens))
    assert dsp.dspark_device_status() == 0


def test_verify_rows_no_trial_settles_take_the_explicit_residual():
    """Target within a few hundredths of the draft: a rejected row's residual
    mass is about 1 %, so most of its 64 trials keep nothing and the row goes
    on to the explicit residual pass (the oracle's kind 1); the trials settle
    the rest (kind 4).  Both routes against the oracle."""
    shape = (768, 4, 1000, 128, 320)
    rnd, orc, lens = _verify_case(shape, 1.0, seed=351, noise_std=0.03)
    kinds = np.bincount(orc["final_kind"], minlength=5)
    print(f"oracle kinds (greedy, explicit, bonus, empty, trial): {kinds.tolist()}")
    assert kinds[1] >= 2 and kinds[4] >= 1
    flagged = compare_verify(rnd.accepted, rnd.bonus, orc, 1.0)
    print(f"verify {shape}: {flagged} of {shape[0]} requests in a tie band")
    assert flagged <= max(1, shape[0] // 50)
    assert dsp.dspark_device_status() == 0
    rejected, explicit = dsp.dspark_verify_residual_rows(rnd.head.dims, rnd.ws_verify)
    print(f"device: {rejected} rejected rows, {explicit} to the explicit pass")
    assert abs(rejected - int(kinds[1] + kinds[3] + kinds[4])) <= flagged
    assert abs(explicit - int(kinds[1] + kinds[3])) <= flagged


@pytest.mark.parametrize("shape,tau", [((37, 4, 1000, 128, 320), 1.0),
                                       ((37, 4, 1000, 128, 320), 0.0),
                                       ((3, 32, 520, 64, 64), 1.0),
                                       ((3, 32, 520, 64, 64), 0.0)])
def test_verify_full_lengths(shape, tau):
    """Every draft admitted (up to gamma = 32, the largest the library takes)."""
    rnd, orc, lens = _verify_case(shape, tau, seed=330 + shape[1], lens_kind="full")
    flagged = compare_verify(rnd.accepted, rnd.bonus, orc, tau)
    print(f"verify {shape} tau={tau}: {flagged} of {shape[0]} requests in a tie band")
    assert flagged <= max(1, shape[0] // 50)
    assert dsp.dspark_device_status() == 0


@pytest.mark.parametrize("tau", [0.0, 1.0])
def test_markov_draft_more_row_blocks_than_sms(tau):
    """153 blocks of 128 requests: more M blocks than a GB300 has SMs, so a CTA
    changes row block from one tile to the next and flushes a partial per tile."""
    shape = (153 * 128, 2, 520, 64, 64)
    rnd, orc = _draft_case(shape, tau, seed=280)
    rep = compare_draft(rnd.tokens, rnd.conf, rnd.lse_d if tau > 0 else None,
                        rnd.logp_d if tau > 0 else None, orc, tau, tol_rel=TOL_DRAFT)
    print(f"{shape} tau={tau}: {rep.flagged} of {rep.compared} in the tie band")
    assert rep.compared >= shape[0]
    assert rep.flagged <= flag_budget(rep.compared)
    assert dsp.dspark_device_status() == 0


@pytest.mark.parametrize("shape", [(4, 5, 1024, 64, 256), (37, 4, 1000, 128, 320),
                                   (130, 2, 2056, 64, 192)])
@pytest.mark.parametrize("tau", [0.0, 1.0])
def test_fused_draft_matches_oracle(shape, tau):
    """The fused single-contraction step against the oracle's statement of it
    (base logits h . W_lm exact, never rounded to bf16)."""
    R, G, V, r, d = shape
    seed = 240 + V
    inp = _weights(R, G, V, r, d, seed=seed)
    orc = oracle.fused_draft(inp["h"], inp["anchor"], inp["W_lm"], inp["W1"], inp["W2"],
                             inp["w_conf"], inp["T"], tau, seed=12345 + seed, keep_scores=True)
    head = dsp.DraftHead.from_weights(R, G, inp["W_lm"], inp["W1"], inp["W2"], inp["w_conf"],
                                      inp["T"])
    W_cat = torch.empty((V, d + r), dtype=torch.bfloat16, device="cuda")
    dsp.dspark_pack_fused(head.dims, head.W_lm, head.W2t, W_cat)
    assert torch.equal(W_cat[:, :d], head.W_lm) and torch.equal(W_cat[:, d:], head.W2t)
    rnd = dsp.Round(head)
    ws = dsp.workspace(dsp.dspark_fused_workspace_bytes(head.dims))
    dsp.dspark_fused_draft(head.dims, dev(inp["h"], torch.bfloat16).contiguous(),
                           dev(inp["anchor"]), W_cat, head.W1, head.w_conf, head.T, tau,
                           12345 + seed, rnd.tokens, rnd.conf, rnd.logp_d, rnd.lse_d, ws)
    rep = compare_draft(rnd.tokens, rnd.conf, rnd.lse_d if tau > 0 else None,
                        rnd.logp_d if tau > 0 else None, orc, tau, tol_rel=TOL_DRAFT)
    print(f"fused {shape} tau={tau}: {rep.flagged} of {rep.compared} in the tie band")
    assert rep.compared >= R
    assert rep.flagged <= flag_budget(rep.compared)
    assert dsp.dspark_device_status() == 0


@pytest.mark.parametrize("R", [200, 400])
def test_markov_draft_row_groups(R):
    """Sampling on a 152-CTA grid (two row blocks): 200 requests take groups of
    six warps per request in the row phase, 400 groups of four."""
    shape = (R, 2, 20000, 64, 64)
    rnd, orc = _draft_case(shape, 1.0, seed=290)
    rep = compare_draft(rnd.tokens, rnd.conf, rnd.lse_d, rnd.logp_d, orc, 1.0,
                        tol_rel=TOL_DRAFT)
    print(f"{shape}: {rep.flagged} of {rep.compared} in the tie band")
    assert rep.compared >= shape[0]
    assert rep.flagged <= flag_budget(rep.compared)
    assert dsp.dspark_device_status() == 0


@pytest.mark.parametrize("shape,tau", [((600, 3, 1000, 512, 64), 0.0),
                                       ((1100, 2, 20000, 256, 64), 0.0),
                                       ((1100, 2, 20000, 256, 64), 1.0),
                                       ((90, 3, 20000, 512, 64), 1.0)])
def test_markov_draft_with_resident_e(shape, tau):
    """Batches of four or more row blocks keep each CTA's E tile in shared memory
    for the step (5 row blocks on 20 CTAs at r = 512, 9 on 144 CTAs at r = 256;
    sampling with more than three requests per CTA).  Sampling at one row block
    keeps it too: eight k blocks of E at r = 512 here (four at r <= 256 in the
    small sampled cases of test_markov_draft_matches_oracle)."""
    rnd, orc = _draft_case(shape, tau, seed=295)
    rep = compare_draft(rnd.tokens, rnd.conf, rnd.lse_d if tau > 0 else None,
                        rnd.logp_d if tau > 0 else None, orc, tau, tol_rel=TOL_DRAFT)
    print(f"{shape}: {rep.flagged} of {rep.compared} in the tie band")
    assert rep.compared >= shape[0]
    assert rep.flagged <= flag_budget(rep.compared)
    assert dsp.dspark_device_status() == 0


@pytest.mark.parametrize("shape,tau", [((3, 32, 520, 64, 64), 0.0), ((3, 32, 520, 64, 64), 1.0),
                                       ((37, 4, 1000, 128, 320), 0.05),
                                       ((37, 4, 1000, 128, 320), 4.0)])
def test_markov_draft_edges(shape, tau):
    """gamma = 32; a very cold and a very hot sampling temperature."""
    rnd, orc = _draft_case(shape, tau, seed=260 + shape[1])
    rep = compare_draft(rnd.tokens, rnd.conf, rnd.lse_d if tau > 0 else None,
                        rnd.logp_d if tau > 0 else None, orc, tau, tol_rel=TOL_DRAFT)
    print(f"{shape} tau={tau}: {rep.flagged} of {rep.compared} in the tie band")
    assert rep.compared >= shape[0]
    assert rep.flagged <= flag_budget(rep.compared)
    assert dsp.dspark_device_status() == 0


def test_verify_zero_lengths_take_bonus_from_row_one():
    shape = (16, 3, 1000, 64, 64)
    R, G, V = shape[:3]
    for tau in (0.0, 1.0):
        inp = _weights(*shape, seed=41)
        target = workloads.random_normal((R, G + 1, V), 1.0, 42)
        head = dsp.DraftHead.from_weights(R, G, inp["W_lm"], inp["W1"], inp["W2"],
                                          inp["w_conf"], inp["T"])
        rnd = dsp.Round(head)
        rnd.tokens.zero_()
        rnd.len.zero_()
        rnd.lse_d.zero_()
        rnd.logp_d.zero_()
        rnd.base.zero_()
        rnd.verify(dev(inp["anchor"]), dev(target), tau, 9)
        orc = oracle.verify(np.zeros((R, G), int), np.zeros(R, int), np.zeros((R, G, V)),
                            target, tau, 9)
        assert np.all(host(rnd.accepted) == 0)
        compare_verify(rnd.accepted, rnd.bonus, orc, tau)


def test_device_status_reports_bad_tokens_and_lengths():
    shape = (4, 3, 1000, 64, 64)
    R, G, V = shape[:3]
    inp = _weights(*shape, seed=51)
    head = dsp.DraftHead.from_weights(R, G, inp["W_lm"], inp["W1"], inp["W2"], inp["w_conf"],
                                      inp["T"])
    rnd = dsp.Round(head)
    assert dsp.dspark_device_status() == 0
    bad_anchor = torch.tensor([0, 1, V + 5, 2], dtype=torch.int32, device="cuda")
    h = dev(inp["h"], torch.bfloat16).contiguous()
    rnd.base.zero_()
    dsp.dspark_markov_draft(head.dims, rnd.base, h, bad_anchor, head.W1, head.W2t, head.w_conf,
                            head.T, 0.0, 0, rnd.tokens, rnd.conf, None, None, rnd.ws_draft)
    assert dsp.dspark_device_status() == 5          # DSPARK_ERR_TOKEN, then cleared
    assert dsp.dspark_device_status() == 0
    rnd.len.copy_(torch.tensor([0, 1, G + 2, 1], dtype=torch.int32))
    target = torch.zeros((R, G + 1, V), dtype=torch.bfloat16, device="cuda")
    rnd.verify(dev(inp["anchor"]), target, 0.0, 1)
    assert dsp.dspark_device_status() == 6          # DSPARK_ERR_LENGTH
    with pytest.raises(dsp.DSparkError):
        dsp.dspark_verify(head.dims, None, rnd.tokens, rnd.len, None, None, None, None, None,
                          target, 1.0, 0, rnd.accepted, rnd.bonus, rnd.ws_verify)


# ------------------------------------------------------------ the round ---

# the Qwen3-8B-shaped case with its vocabulary cut to 4104 (a ragged 64-id
# block) and d to 256: tau = 1, T_k = 1 + 0.1 k, the concave SPS table
ROUND_CASES = {"tiny": workloads.WORKLOADS["tiny"],
               "qwen3_8b_small": workloads.WORKLOADS["qwen3_8b"].with_(V=4104, d=256,
                                                                       anchor_hi=4104)}


@pytest.mark.parametrize("name,tau,mode", [("tiny", 0.0, 0), ("tiny", 1.0, 1),
                                           ("tiny", 0.7, 2), ("qwen3_8b_small", 1.0, 0),
                                           ("qwen3_8b_small", 1.0, 1),
                                           ("qwen3_8b_small", 1.0, 2)])
def test_round_matches_oracle_end_to_end(name, tau, mode):
    """One whole round through Round.run, then each later stage on the oracle's
    own inputs: the scheduler on the oracle's confidences (bit-exact), and the
    verifier on the oracle's tokens and lengths (exact outside the tie bands).
    The oracle never sees a CUDA output; the CUDA stages see the oracle's."""
    w = ROUND_CASES[name]
    inp = workloads.make_inputs(w)
    R, G, V, d = w.R, w.gamma, w.V, w.d
    kf = R * G // 2
    orc_base = oracle.base_logits(inp["h"], inp["W_lm"])
    nxt = oracle.base_logits(inp["h_next"], inp["W_lm"])
    target_np = np.concatenate([orc_base, nxt[:, None, :]], axis=1) + host(inp["noise"])
    target = torch.tensor(target_np, dtype=torch.float32).to(torch.bfloat16)
    ds, vs = inp["draft_seed"], inp["verify_seed"]
    orc = oracle.markov_draft(orc_base, inp["h"], inp["anchor"], inp["W1"], inp["W2"],
                              inp["w_conf"], inp["T"], tau, ds, keep_scores=True,
                              keep_logits=True)
    head = dsp.DraftHead.from_weights(R, G, inp["W_lm"], inp["W1"], inp["W2"], inp["w_conf"],
                                      inp["T"])
    rnd = dsp.Round(head)
    h = dev(inp["h"], torch.bfloat16).contiguous()
    anchor = dev(inp["anchor"])
    sps = dev(inp["sps"])
    tgt = dev(target).contiguous()
    rnd.run(h, anchor, tgt, sps, tau, ds, vs, mode=mode, k_fixed=kf)
    torch.cuda.synchronize()
    assert dsp.dspark_device_status() == 0
    rep = compare_draft(rnd.tokens, rnd.conf, rnd.lse_d if tau > 0 else None,
                        rnd.logp_d if tau > 0 else None, orc, tau, tol_rel=TOL_DRAFT)
    print(f"{name} tau={tau} mode={mode}: draft {rep.flagged} of {rep.compared} in the tie band")
    assert rep.flagged <= flag_budget(rep.compared)
    c_o = orc["conf"].astype(np.float32)
    o_s = oracle.schedule(c_o, inp["sps"], mode, kf)
    acc = host(rnd.accepted)
    assert np.all(acc >= 0) and np.all(acc <= host(rnd.len))
    if np.array_equal(host(rnd.tokens), orc["tokens"]) and schedule_is_robust(o_s, rel=1e-4):
        assert np.array_equal(host(rnd.len), o_s["len"])  # the round's own schedule
    # the scheduler on the oracle's confidences: every output bit-exact
    dsp.dspark_schedule(dev(torch.tensor(c_o)), R, G, sps, mode, kf, rnd.len, rnd.K, rnd.theta)
    assert int(rnd.K.item()) == o_s["K"]
    assert np.array_equal(host(rnd.len), o_s["len"])
    assert float(rnd.theta.item()) == o_s["theta"]
    # the verifier on the oracle's base logits, tokens, lengths and draft
    # log-probabilities
    rnd.base.copy_(dev(torch.tensor(orc_base.reshape(R * G, V), dtype=torch.float32),
                       torch.bfloat16))
    rnd.tokens.copy_(dev(torch.tensor(orc["tokens"], dtype=torch.int32)))
    rnd.lse_d.copy_(dev(torch.tensor(orc["lse"], dtype=torch.float32)))
    rnd.logp_d.copy_(dev(torch.tensor(orc["logp"], dtype=torch.float32)))
    rnd.verify(anchor, tgt, tau, vs)
    torch.cuda.synchronize()
    ov = oracle.verify(orc["tokens"], o_s["len"], orc["logits"], target, tau, vs)
    flagged = compare_verify(rnd.accepted, rnd.bonus, ov, tau)
    print(f"  verify: {flagged} of {R} requests in a tie band")
    assert flagged <= max(1, R // 50)
    assert dsp.dspark_device_status() == 0


def test_run_host_matches_device_rounds():
    """Three back-to-back rounds from pinned host buffers (the target copied on a
    side stream under the draft) give the device-resident rounds' outputs."""
    w = workloads.WORKLOADS["tiny"].with_(R=37, V=1000, anchor_hi=1000, n_sps=256)
    inp = workloads.make_inputs(w)
    R, G, V, d = w.R, w.gamma, w.V, w.d
    head = dsp.DraftHead.from_weights(R, G, inp["W_lm"], inp["W1"], inp["W2"], inp["w_conf"],
                                      inp["T"])
    sps = dev(inp["sps"])
    tau = 1.0
    hs = [workloads.random_normal((R * G, d), 1.0, 700 + t) for t in range(3)]
    targets = [workloads.random_normal((R, G + 1, V), 1.5, 710 + t) for t in range(3)]
    want = []
    rnd = dsp.Round(head)
    for t in range(3):
        rnd.run(dev(hs[t], torch.bfloat16).contiguous(), dev(inp["anchor"]),
                dev(targets[t], torch.bfloat16).contiguous(), sps, tau, 11 + t, 21 + t)
        torch.cuda.synchronize()
        want.append({k: host(getattr(rnd, k)).copy() for k in ("tokens", "len", "accepted",
                                                             "bonus")})
    rnd2 = dsp.Round(head)
    dev_in = {"h": torch.empty((R * G, d), dtype=torch.bfloat16, device="cuda"),
              "anchor": torch.empty((R,), dtype=torch.int32, device="cuda"),
              "target": torch.empty((R, G + 1, V), dtype=torch.bfloat16, device="cuda")}
    a_host = inp["anchor"].to(torch.int32).pin_memory()
    h_host = [x.to(torch.bfloat16).pin_memory() for x in hs]      # alive until the end
    t_host = [x.to(torch.bfloat16).pin_memory() for x in targets]
    outs = []
    for t in range(3):  # no synchronisation between rounds
        out_host = {k: torch.empty(getattr(rnd2, k).shape, dtype=getattr(rnd2, k).dtype,
                                   pin_memory=True)
                    for k in ("tokens", "len", "accepted", "bonus")}
        rnd2.run_host(h_host[t], a_host, t_host[t], sps, tau, 11 + t, 21 + t, dev_in, out_host)
        outs.append(out_host)
    torch.cuda.synchronize()
    for t in range(3):
        for k in ("tokens", "len", "accepted", "bonus"):
            assert np.array_equal(outs[t][k].numpy(), want[t][k]), (t, k)
    assert dsp.dspark_device_status() == 0


# ------------------------------------------------------- the RNN head -----

def _rnn_weights(R, G, V, r, d, seed, scale=2.0):
    inp = _weights(R, G, V, r, d, seed=seed)
    g = torch.Generator().manual_seed(seed + 9)
    W_gc = (torch.randn((2 * r, 2 * r + d), generator=g) * (scale / math.sqrt(2 * r + d)))
    return inp, W_gc.to(torch.bfloat16)


@pytest.mark.parametrize("shape", [(4, 5, 1024, 64, 256), (37, 4, 1000, 128, 320),
                                   (130, 3, 2056, 64, 192)])
@pytest.mark.parametrize("tau", [0.0, 1.0])
def test_rnn_draft_matches_oracle(shape, tau):
    R, G, V, r, d = shape
    inp, W_gc = _rnn_weights(R, G, V, r, d, seed=500 + V)
    base = workloads.random_normal((R, G, V), 1.0, 501 + V)
    orc = oracle.rnn_draft(base, inp["h"], inp["anchor"], inp["W1"], inp["W2"], W_gc,
                           inp["w_conf"], inp["T"], tau, seed=4242, keep_scores=True)
    head = dsp.DraftHead.from_weights(R, G, inp["W_lm"], inp["W1"], inp["W2"], inp["w_conf"],
                                      inp["T"])
    rnd = dsp.Round(head)
    rnd.base.copy_(dev(base.reshape(R * G, V)))
    ws = dsp.workspace(dsp.dspark_rnn_workspace_bytes(head.dims))
    W_rec = dev(W_gc[:, :2 * r]).contiguous()
    W_hid = dev(W_gc[:, 2 * r:]).contiguous()
    dsp.dspark_rnn_draft(head.dims, rnd.base, dev(inp["h"], torch.bfloat16).contiguous(),
                         dev(inp["anchor"]), head.W1, head.W2t, W_rec, W_hid, head.w_conf, head.T,
                         tau, 4242, rnd.tokens, rnd.conf, rnd.logp_d, rnd.lse_d, ws)
    torch.cuda.synchronize()
    # the f32 state crosses bf16 roundings that the float64 oracle may take the
    # other way: a wider tie band than the Markov head's 1e-3
    rep = compare_draft(rnd.tokens, rnd.conf, rnd.lse_d if tau > 0 else None,
                        rnd.logp_d if tau > 0 else None, orc, tau, tol_rel=3e-3)
    assert rep.compared >= R
    assert rep.flagged <= max(3, rep.compared // 10)
    assert dsp.dspark_device_status() == 0


def test_rnn_draft_without_weights_is_parallel_drafting():
    R, G, V, r, d = 9, 3, 1000, 64, 128
    inp, W_gc = _rnn_weights(R, G, V, r, d, seed=77)
    base = workloads.random_normal((R, G, V), 1.0, 78)
    head = dsp.DraftHead.from_weights(R, G, inp["W_lm"], inp["W1"], inp["W2"], inp["w_conf"],
                                      inp["T"])
    rnd = dsp.Round(head)
    rnd.base.copy_(dev(base.reshape(R * G, V)))
    ws = dsp.workspace(dsp.dspark_rnn_workspace_bytes(head.dims))
    zero = torch.zeros((2 * r, 2 * r + d), dtype=torch.bfloat16, device="cuda")
    dsp.dspark_rnn_draft(head.dims, rnd.base, dev(inp["h"], torch.bfloat16).contiguous(),
                         dev(inp["anchor"]), head.W1, head.W2t, zero[:, :2 * r].contiguous(),
                         zero[:, 2 * r:].contiguous(), head.w_conf, head.T, 0.0, 0, rnd.tokens,
                         rnd.conf, None, None, ws)
    want = torch.argmax(base.float(), dim=2)  # first maximum on ties
    assert torch.equal(rnd.tokens.cpu().long(), want)
    assert dsp.dspark_device_status() == 0
