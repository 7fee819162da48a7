"""Host-side checks of the C-ABI library: it loads without a GPU, exports every
symbol the header declares, and rejects bad arguments before launching."""
import ctypes
import os
import re

import pytest

import speculative_decoding_draft_02_gb300 as dsp
from speculative_decoding_draft_02_gb300 import build as dsp_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    dsp_build.build()
    return dsp.load_library()


def declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(dspark_[a-z0-9_]+)\s*\(", text))
    return names


def test_header_declares_the_boundary():
    names = declared_symbols()
    for must in ["dspark_lm_head", "dspark_markov_draft", "dspark_draft", "dspark_schedule",
                 "dspark_verify"]:
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(dsp.EXPORTS) <= declared_symbols()


def test_error_strings(lib):
    assert lib.dspark_error_string(0) == b"ok"
    assert b"SPS" in lib.dspark_error_string(2)
    assert lib.dspark_error_string(999) == b"unknown error"


def test_workspace_sizes(lib):
    d = dsp.dims_of(256, 5, 129280, 512, 7168)
    wm = dsp.dspark_markov_workspace_bytes(d)
    wv = dsp.dspark_verify_workspace_bytes(d)
    assert wm % 256 == 0 and wv % 256 == 0
    assert wm >= 256 * 512 * 2 and wv >= 256 * 512 * 2
    bad = dsp.dims_of(256, 5, 129281, 512, 7168)  # V not a multiple of 8
    assert dsp.dspark_markov_workspace_bytes(bad) == 0


@pytest.mark.parametrize("dims", [(0, 5, 1024, 64, 256), (4, 0, 1024, 64, 256),
                                  (4, 33, 1024, 64, 256), (4, 5, 1020, 64, 256),
                                  (4, 5, 1024, 48, 256), (4, 5, 1024, 64, 200)])
def test_bad_dims_rejected_without_launch(lib, dims):
    d = dsp.dims_of(*dims)
    fake = ctypes.c_void_p(256)
    rc = lib.dspark_lm_head(ctypes.byref(d), fake, fake, fake, None)
    assert rc == dsp.DSPARK_OK + 1  # DSPARK_ERR_ARG
    rc = lib.dspark_markov_draft(ctypes.byref(d), fake, fake, fake, fake, fake, fake, fake, 0.0,
                                 0, fake, fake, None, None, fake, 1 << 30, None)
    assert rc == 1


def test_null_pointers_and_short_tables_rejected(lib):
    d = dsp.dims_of(4, 5, 1024, 64, 256)
    fake = ctypes.c_void_p(256)
    assert lib.dspark_lm_head(ctypes.byref(d), None, fake, fake, None) == 1
    # schedule: SPS table shorter than R*(gamma+1)
    assert lib.dspark_schedule(fake, 4, 5, fake, 23, 0, 0, fake, fake, fake, None, None, None) == 2
    assert lib.dspark_schedule(fake, 4, 5, fake, 24, 7, 0, fake, fake, fake, None, None, None) == 1
    assert lib.dspark_schedule(fake, 4000, 5, fake, 1 << 20, 0, 0, fake, fake, fake, None, None,
                               None) == 1  # more than 16384 candidates
    # workspace too small / misaligned
    assert lib.dspark_markov_draft(ctypes.byref(d), fake, fake, fake, fake, fake, fake, fake, 0.0,
                                   0, fake, fake, None, None, fake, 16, None) == 4
    assert lib.dspark_markov_draft(ctypes.byref(d), fake, fake, fake, fake, fake, fake, fake, 0.0,
                                   0, fake, fake, None, None, ctypes.c_void_p(264), 1 << 30,
                                   None) == 4
    # sampling verify needs the draft operands
    assert lib.dspark_verify(ctypes.byref(d), fake, fake, fake, None, None, None, None, None,
                             fake, 1.0, 0, fake, fake, fake, 1 << 30, None) == 1
    # negative temperature
    assert lib.dspark_verify(ctypes.byref(d), fake, fake, fake, fake, fake, fake, fake, fake,
                             fake, -1.0, 0, fake, fake, fake, 1 << 30, None) == 1


def test_new_entry_points_check_arguments_without_launch(lib):
    d = dsp.dims_of(4, 5, 1024, 64, 256)
    fake = ctypes.c_void_p(256)
    # the bounded-wait self-test takes 1 ns .. 2 s
    assert lib.dspark_selftest_wait_timeout(0, None) == 1
    assert lib.dspark_selftest_wait_timeout(3_000_000_000, None) == 1
    # the RNN head needs its recurrent weights, and a large enough workspace
    assert lib.dspark_rnn_draft(ctypes.byref(d), fake, fake, fake, fake, fake, None, fake, fake,
                                fake, 0.0, 0, fake, fake, None, None, fake, 1 << 30, None) == 1
    assert lib.dspark_rnn_draft(ctypes.byref(d), fake, fake, fake, fake, fake, fake, fake, fake,
                                fake, 0.0, 0, fake, fake, None, None, fake, 16, None) == 4
    assert lib.dspark_rnn_workspace_bytes(ctypes.byref(d)) > lib.dspark_markov_workspace_bytes(
        ctypes.byref(d))
    # the fused single-contraction step needs the packed weights and its workspace
    assert lib.dspark_fused_draft(ctypes.byref(d), fake, fake, None, fake, fake, fake, 0.0, 0,
                                  fake, fake, None, None, fake, 1 << 30, None) == 1
    assert lib.dspark_fused_draft(ctypes.byref(d), fake, fake, fake, fake, fake, fake, 0.0, 0,
                                  fake, fake, None, None, fake, 16, None) == 4
    assert lib.dspark_pack_fused(ctypes.byref(d), fake, None, fake, None) == 1
    assert lib.dspark_fused_workspace_bytes(ctypes.byref(d)) > lib.dspark_markov_workspace_bytes(
        ctypes.byref(d))
    # STS: at most 64 bins; the asynchronous schedule needs its ring
    assert lib.dspark_sts_workspace_bytes(1000, 5, 51, 65) == 0
    assert lib.dspark_sts_fit(fake, fake, 1000, 5, fake, 51, 65, fake, fake, fake, 1 << 30,
                              None) == 1
    assert lib.dspark_schedule_async(fake, 4, 5, fake, 24, None, fake, fake, fake, None, None,
                                     None) == 1


def test_binding_refuses_host_tensors():
    import torch
    d = dsp.dims_of(4, 5, 1024, 64, 256)
    with pytest.raises(dsp.DSparkError):
        dsp.dspark_lm_head(d, torch.zeros(20, 256, dtype=torch.bfloat16),
                           torch.zeros(1024, 256, dtype=torch.bfloat16),
                           torch.zeros(20, 1024, dtype=torch.bfloat16))
