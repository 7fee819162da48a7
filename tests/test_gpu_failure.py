"""Failure detection on the GPU without a fault: a bounded wait runs out.

Every device-side wait of the library is an mbarrier wait bounded in time; on
expiry the kernel records DSPARK_ERR_TIMEOUT in the device status word and
returns.  The self-test entry point waits on a barrier nothing arrives on.
"""
import time

import numpy as np
import pytest
import torch

import speculative_decoding_draft_02_gb300 as dsp

pytestmark = pytest.mark.gpu

DSPARK_ERR_TIMEOUT = 7


def test_bounded_wait_reports_timeout_and_the_context_survives():
    dsp.dspark_device_status()  # start from a clear status word
    t0 = time.monotonic()
    dsp.dspark_selftest_wait_timeout(50_000_000)  # 50 ms
    assert dsp.dspark_device_status() == DSPARK_ERR_TIMEOUT
    assert time.monotonic() - t0 < 5.0
    assert dsp.dspark_device_status() == 0  # reading cleared it
    # the context still runs the path: a small LM head against torch
    g = torch.Generator().manual_seed(3)
    h = (torch.randn(20, 256, generator=g) / 4).to(torch.bfloat16)
    W = (torch.randn(1024, 256, generator=g) / 4).to(torch.bfloat16)
    out = torch.empty((20, 1024), dtype=torch.bfloat16, device="cuda")
    dsp.dspark_lm_head(dsp.dims_of(4, 5, 1024, 64, 256), h.cuda(), W.cuda(), out)
    ref = h.float() @ W.float().T
    assert np.abs(out.float().cpu().numpy() - ref.numpy()).max() < 0.05
    assert dsp.dspark_device_status() == 0
