"""The allocation-free Markov draft entry point against the workspace one.

dspark_markov_draft_static serves callers that cannot allocate device memory
(a plugin interface that hands over only tensors, a serving loop that forbids
allocations after start-up): it keeps its scratch in a static device array of
the library.  Here it must give the same results as dspark_markov_draft with a
caller workspace, on two calls in a row, and refuse problems whose scratch
would not fit.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

dsp = pytest.importorskip("speculative_decoding_draft_02_gb300")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from speculative_decoding_draft_02_gb300 import build
    build.build()
    dsp.load_library()


def _case(R, G, V, r, d, seed):
    w = workloads.WORKLOADS["tiny"].with_(R=R, gamma=G, V=V, r=r, d=d, anchor_hi=V)
    inp = workloads.make_inputs(w, seed=seed, with_target_noise=False)
    base = workloads.random_normal((R * G, V), 1.0, seed + 1).to("cuda")
    head = dsp.DraftHead.from_weights(R, G, inp["W_lm"], inp["W1"], inp["W2"], inp["w_conf"],
                                      inp["T"])
    h = inp["h"].to("cuda", torch.bfloat16).reshape(R * G, d).contiguous()
    return head, base, h, inp["anchor"].to("cuda")


def _outputs(R, G):
    return [torch.full((R, G), -1, dtype=torch.int32, device="cuda")] + [
        torch.full((R, G), float("nan"), dtype=torch.float32, device="cuda") for _ in range(3)]


@pytest.mark.parametrize("tau", [0.0, 1.0])
@pytest.mark.parametrize("shape", [(37, 4, 1000, 128, 320), (256, 5, 4104, 512, 256)])
def test_static_scratch_matches_workspace_path(shape, tau):
    R, G, V, r, d = shape
    head, base, h, anchor = _case(R, G, V, r, d, seed=900 + V)
    dims = head.dims
    ws = dsp.workspace(dsp.dspark_markov_workspace_bytes(dims))
    ref = _outputs(R, G)
    dsp.dspark_markov_draft(dims, base, h, anchor, head.W1, head.W2t, head.w_conf, head.T, tau,
                            77, *ref, ws)
    torch.cuda.synchronize()
    for call in range(2):  # the static array keeps the previous call's contents
        got = _outputs(R, G)
        dsp.dspark_markov_draft_static(dims, base, h, anchor, head.W1, head.W2t, head.w_conf,
                                       head.T, tau, 77, *got)
        torch.cuda.synchronize()
        assert torch.equal(got[0], ref[0]), f"tokens differ on call {call}"
        for a, b in zip(got[1:], ref[1:]):
            np.testing.assert_allclose(a.cpu().numpy(), b.cpu().numpy(), rtol=1e-2, atol=1e-6)
    assert dsp.dspark_device_status() == 0


def test_static_scratch_rejects_problems_that_do_not_fit():
    dims = dsp.dims_of(1024, 7, 129280, 512, 7168)
    assert dsp.dspark_markov_workspace_bytes(dims) > dsp.STATIC_SCRATCH_BYTES
    t = torch.zeros(16, dtype=torch.int32, device="cuda")
    f = torch.zeros(16, dtype=torch.float32, device="cuda")
    b = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dsp.DSparkError, match="static scratch"):
        dsp.dspark_markov_draft_static(dims, b, b, t, b, b, b, f, 1.0, 0, t, f, f, f)
    lib = dsp.load_library()
    assert lib.dspark_markov_draft_static(None, None, None, None, None, None, None, None, 0.0, 0,
                                          None, None, None, None, None) == 1
