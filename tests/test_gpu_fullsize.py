"""Full-size parity at the benchmarked workload shapes, in the benchmark's launch
configuration (the package's DraftHead/Round objects, as bench.py drives them).

The oracle cannot run a whole V4-shaped round in seconds, so it recomputes a
few sampled requests one by one (their base-logit rows, Markov steps and
verification) and the scheduler in full.  Inputs come from the seeded
generators; nothing the CUDA path produces is fed to the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import TOL_DRAFT, compare_draft, compare_verify, flag_budget, host

pytestmark = pytest.mark.gpu

dsp = pytest.importorskip("speculative_decoding_draft_02_gb300")

SAMPLED = 16  # requests re-derived by the oracle per case (plus the first and last)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from speculative_decoding_draft_02_gb300 import build
    build.build()
    dsp.load_library()


def _sample_ids(R, seed):
    rng = np.random.default_rng(seed)
    pick = rng.choice(R, size=min(R, SAMPLED), replace=False)
    return np.array(sorted(set([0, R - 1] + pick.tolist())))


@pytest.mark.parametrize("name,tau", [("v4_dspark5", 1.0), ("qwen3_8b", 1.0), ("qwen3_4b", 0.0),
                                      ("qwen3_4b", 1.0), ("stress", 0.0)])
def test_draft_full_size_sampled_requests(name, tau):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, device="cuda", with_target_noise=False)
    R, G, V, d = w.R, w.gamma, w.V, w.d
    head = dsp.DraftHead.from_weights(R, G, inp["W_lm"], inp["W1"], inp["W2"], inp["w_conf"],
                                      inp["T"])
    rnd = dsp.Round(head)
    h = inp["h"].reshape(R * G, d).contiguous()
    rnd.draft(h, inp["anchor"], tau, inp["draft_seed"])
    torch.cuda.synchronize()
    assert dsp.dspark_device_status() == 0

    ids = _sample_ids(R, 11)
    W_lm = inp["W_lm"].cpu()
    h_s = inp["h"][ids].cpu()
    base_s = oracle.base_logits(h_s.reshape(-1, d), W_lm, vocab_chunk=16384).reshape(len(ids), G, V)
    orc = oracle.markov_draft(base_s, h_s, inp["anchor"][ids].cpu(), inp["W1"].cpu(),
                              inp["W2"].cpu(), inp["w_conf"].cpu(), inp["T"].cpu(), tau,
                              inp["draft_seed"], keep_scores=True, requests=ids)
    # the LM head sums in f32 and the oracle in f64, so a base logit near a bf16
    # rounding boundary can land one bf16 step away: the tie band of a decision
    # widens by the differences seen among the entries near its top
    got = host(rnd.base.view(R, G, V)[ids]).astype(np.float64)
    rep = compare_draft(rnd.tokens, rnd.conf, rnd.lse_d if tau > 0 else None,
                        rnd.logp_d if tau > 0 else None, orc, tau, tol_rel=TOL_DRAFT,
                        requests=ids, shift=np.abs(got - base_s))
    print(f"{name} tau={tau}: {rep.flagged} of {rep.compared} decisions in the tie band, "
          f"{int(np.sum(got != base_s))} of {got.size} base logits one bf16 step apart")
    assert rep.compared >= len(ids)
    assert rep.flagged <= flag_budget(rep.compared)
    # the base logits themselves, on the sampled rows
    exact = oracle.base_logits(h_s.reshape(-1, d), W_lm, bf16_out=False,
                               vocab_chunk=16384).reshape(len(ids), G, V)
    err = np.abs(got - exact)
    assert np.all(err <= 1e-2 * np.maximum(np.abs(exact), 1.0))  # the stated bar
    # fp32 accumulation over d terms can push a value to the neighbouring bf16
    assert np.mean(err <= 2.0 ** -8 * np.abs(exact) + 1e-5) > 0.999


@pytest.mark.parametrize("name", ["tiny", "qwen3_4b", "qwen3_8b", "v4_dspark5", "stress"])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_schedule_full_size(name, mode):
    w = workloads.WORKLOADS[name]
    R, G = w.R, w.gamma
    c = workloads.random_confidences(R, G, seed=w.seed, ones_frac=0.01)
    sps = workloads.sps_table(w.sps, w.n_sps)
    kf = (R * G) // 4
    o = oracle.schedule(c, sps, mode, kf)
    rnd_len = torch.empty(R, dtype=torch.int32, device="cuda")
    K = torch.empty(1, dtype=torch.int32, device="cuda")
    th = torch.empty(1, dtype=torch.float64, device="cuda")
    a = torch.empty((R, G), dtype=torch.float32, device="cuda")
    order = torch.empty(R * G, dtype=torch.int32, device="cuda")
    dsp.dspark_schedule(c.cuda(), R, G, sps.cuda(), mode, kf, rnd_len, K, th, a, order)
    assert np.array_equal(host(a), o["a"])
    assert np.array_equal(host(order), o["order"])
    # the same fixed-point sums and float64 products on both sides: bit-exact
    assert int(K.item()) == o["K"]
    assert np.array_equal(host(rnd_len), o["len"])
    assert float(th.item()) == o["theta"]
    if mode == 0 and name in ("v4_dspark5", "stress"):
        assert 0 < o["K"] < R * G  # the staircase tables give an interior optimum


@pytest.mark.parametrize("name,tau", [("v4_dspark5", 1.0), ("stress", 0.0), ("qwen3_8b", 1.0),
                                      ("qwen3_4b", 0.0), ("qwen3_4b", 1.0)])
def test_verify_full_size_sampled_requests(name, tau):
    w = workloads.WORKLOADS[name]
    R, G, V = w.R, w.gamma, w.V
    inp = workloads.make_inputs(w.with_(d=64), device="cuda", with_target_noise=False)
    base = workloads.random_normal((R, G, V), 1.0, w.seed + 1, device="cuda")
    tokens = workloads.random_tokens(R, G, V, w.seed + 2, device="cuda")
    lens = workloads.random_lengths(R, G, w.seed + 3, device="cuda")
    noise = workloads.random_normal((R, G + 1, V), 0.4, w.seed + 4, device="cuda",
                                    dtype=torch.float32)
    ids = _sample_ids(R, 13)
    # target near the drafts so that acceptance and rejection both occur; on the
    # sampled requests the drafts' own logits come from the oracle
    lse_d = torch.zeros((R, G), dtype=torch.float32)
    logp_d = torch.zeros((R, G), dtype=torch.float32)
    target = torch.cat([base.float(), base[:, -1:].float()], dim=1) + noise
    dl = None
    if tau > 0:
        od = oracle.markov_draft(base[ids].cpu(), np.zeros((len(ids), G, 1)), inp["anchor"][ids].cpu(),
                                 inp["W1"].cpu(), inp["W2"].cpu(), np.zeros(1 + w.r), np.ones(G),
                                 tau, 0, forced=tokens[ids].cpu(), keep_logits=True)
        dl = od["logits"]
        lse_d[ids] = torch.tensor(od["lse"], dtype=torch.float32)
        logp_d[ids] = torch.tensor(od["logp"], dtype=torch.float32)
        t_ids = np.concatenate([dl, dl[:, -1:]], axis=1) + host(noise[ids])
        target[ids] = torch.tensor(t_ids, dtype=torch.float32, device="cuda")
    else:  # make accepted runs likely: drafts equal the target argmax mostly
        am = torch.argmax(target[:, :G], dim=2).to(torch.int32)
        pick = workloads.random_normal((R, G), 1.0, w.seed + 5, device="cuda",
                                       dtype=torch.float32) < 1.0
        tokens = torch.where(pick, am, tokens)
    target = target.to(torch.bfloat16).contiguous()
    head = dsp.DraftHead.from_weights(R, G, inp["W_lm"], inp["W1"], inp["W2"], inp["w_conf"],
                                      inp["T"])
    rnd = dsp.Round(head)
    rnd.base.copy_(base.reshape(R * G, V))
    rnd.tokens.copy_(tokens)
    rnd.len.copy_(lens)
    rnd.lse_d.copy_(lse_d.cuda())
    rnd.logp_d.copy_(logp_d.cuda())
    rnd.verify(inp["anchor"], target, tau, w.seed + 77)
    torch.cuda.synchronize()
    assert dsp.dspark_device_status() == 0
    orc = oracle.verify(tokens[ids].cpu(), lens[ids].cpu(), dl, target[ids].cpu(), tau,
                        w.seed + 77, requests=ids)
    flagged = compare_verify(rnd.accepted[ids], rnd.bonus[ids], orc, tau)
    print(f"verify {name} tau={tau}: {flagged} of {len(ids)} requests in a tie band")
    assert flagged <= 1
    acc = host(rnd.accepted)
    assert np.all(acc >= 0) and np.all(acc <= host(lens))
