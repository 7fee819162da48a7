"""Python binding of libdspark.so — the DSpark draft-head round on one GB300.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  There is no fallback: if
the library is missing or a call fails, the call raises.

The functions carry the C-ABI names (see include/dspark.h) and take torch
tensors; `draft`, `schedule`, `verify` and `run_round` compose them.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Dict, Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdspark.so")

DSPARK_OK = 0
SCHED_UNCONSTRAINED = 0
SCHED_BREAK = 1
SCHED_FIXED_K = 2
SCHED_ASYNC = 3

EXPORTS = [
    "dspark_lm_head", "dspark_pack_w2", "dspark_markov_workspace_bytes", "dspark_markov_draft",
    "dspark_draft", "dspark_schedule", "dspark_verify_workspace_bytes", "dspark_verify",
    "dspark_device_status", "dspark_error_string", "dspark_launch_count",
    "dspark_markov_draft_static", "dspark_schedule_async", "dspark_conf_logits",
    "dspark_sts_workspace_bytes", "dspark_sts_fit", "dspark_rnn_workspace_bytes",
    "dspark_rnn_draft", "dspark_selftest_wait_timeout", "dspark_fused_workspace_bytes",
    "dspark_pack_fused", "dspark_fused_draft", "dspark_verify_residual_rows",
]
STATIC_SCRATCH_BYTES = 16 << 20


class DSparkError(RuntimeError):
    pass


class Dims(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int32), ("gamma", ctypes.c_int32), ("V", ctypes.c_int32),
                ("r", ctypes.c_int32), ("d", ctypes.c_int32)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load (once) the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise DSparkError(f"{path} not found: build it with "
                          "`python speculative_decoding_draft_02_gb300/build.py`")
    lib = ctypes.CDLL(path)
    P, I32, U64, SZ, F32 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64, ctypes.c_size_t,
                            ctypes.c_float)
    DP = ctypes.POINTER(Dims)
    sig = {
        "dspark_lm_head": (ctypes.c_int, [DP, P, P, P, P]),
        "dspark_pack_w2": (ctypes.c_int, [DP, P, P, P]),
        "dspark_markov_workspace_bytes": (SZ, [DP]),
        "dspark_markov_draft": (ctypes.c_int, [DP, P, P, P, P, P, P, P, F32, U64, P, P, P, P, P,
                                               SZ, P]),
        "dspark_draft": (ctypes.c_int, [DP, P, P, P, P, P, P, P, F32, U64, P, P, P, P, P, P, SZ,
                                        P]),
        "dspark_schedule": (ctypes.c_int, [P, I32, I32, P, I32, I32, I32, P, P, P, P, P, P]),
        "dspark_schedule_async": (ctypes.c_int, [P, I32, I32, P, I32, P, P, P, P, P, P, P]),
        "dspark_conf_logits": (ctypes.c_int, [DP, P, P, P, P, P, P, P]),
        "dspark_sts_workspace_bytes": (SZ, [I32, I32, I32, I32]),
        "dspark_sts_fit": (ctypes.c_int, [P, P, I32, I32, P, I32, I32, P, P, P, SZ, P]),
        "dspark_rnn_workspace_bytes": (SZ, [DP]),
        "dspark_fused_workspace_bytes": (SZ, [DP]),
        "dspark_pack_fused": (ctypes.c_int, [DP, P, P, P, P]),
        "dspark_fused_draft": (ctypes.c_int, [DP, P, P, P, P, P, P, F32, U64, P, P, P, P, P, SZ,
                                              P]),
        "dspark_selftest_wait_timeout": (ctypes.c_int, [U64, P]),
        "dspark_rnn_draft": (ctypes.c_int, [DP, P, P, P, P, P, P, P, P, P, F32, U64, P, P, P, P,
                                            P, SZ, P]),
        "dspark_verify_workspace_bytes": (SZ, [DP]),
        "dspark_verify": (ctypes.c_int, [DP, P, P, P, P, P, P, P, P, P, F32, U64, P, P, P, SZ,
                                         P]),
        "dspark_markov_draft_static": (ctypes.c_int, [DP, P, P, P, P, P, P, P, F32, U64, P, P, P,
                                                      P, P]),
        "dspark_verify_residual_rows": (ctypes.c_int, [DP, P, SZ, P, P, P]),
        "dspark_device_status": (ctypes.c_int, [P, ctypes.c_int]),
        "dspark_error_string": (ctypes.c_char_p, [ctypes.c_int]),
        "dspark_launch_count": (U64, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(rc: int, what: str):
    if rc != DSPARK_OK:
        msg = load_library().dspark_error_string(rc).decode()
        raise DSparkError(f"{what} failed: {msg} ({rc})")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise DSparkError("tensor must live on the GPU")
    if not t.is_contiguous():
        raise DSparkError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _bf16(t: torch.Tensor) -> torch.Tensor:
    return t if t.dtype == torch.bfloat16 else t.to(torch.bfloat16)


def dims_of(R: int, gamma: int, V: int, r: int, d: int) -> Dims:
    return Dims(R, gamma, V, r, d)


def _u64(seed: int) -> int:
    return int(seed) & 0xFFFFFFFFFFFFFFFF


# --------------------------------------------------------------- raw ABI ----

def dspark_lm_head(dims: Dims, h, W_lm, base_logits, stream=None):
    _check(load_library().dspark_lm_head(ctypes.byref(dims), _ptr(h), _ptr(W_lm),
                                         _ptr(base_logits), _stream(stream)), "dspark_lm_head")


def dspark_pack_w2(dims: Dims, W2, W2t, stream=None):
    _check(load_library().dspark_pack_w2(ctypes.byref(dims), _ptr(W2), _ptr(W2t), _stream(stream)),
           "dspark_pack_w2")


def dspark_markov_workspace_bytes(dims: Dims) -> int:
    return int(load_library().dspark_markov_workspace_bytes(ctypes.byref(dims)))


def dspark_verify_workspace_bytes(dims: Dims) -> int:
    return int(load_library().dspark_verify_workspace_bytes(ctypes.byref(dims)))


def dspark_markov_draft(dims, base_logits, h, anchor, W1, W2t, w_conf, T, tau, seed, tokens,
                        conf, logp_d, lse_d, workspace, stream=None):
    _check(load_library().dspark_markov_draft(
        ctypes.byref(dims), _ptr(base_logits), _ptr(h), _ptr(anchor), _ptr(W1), _ptr(W2t),
        _ptr(w_conf), _ptr(T), float(tau), _u64(seed), _ptr(tokens), _ptr(conf), _ptr(logp_d),
        _ptr(lse_d), _ptr(workspace), workspace.numel(), _stream(stream)), "dspark_markov_draft")


def dspark_markov_draft_static(dims, base_logits, h, anchor, W1, W2t, w_conf, T, tau, seed,
                               tokens, conf, logp_d, lse_d, stream=None):
    """dspark_markov_draft with the scratch kept inside the library (no workspace)."""
    _check(load_library().dspark_markov_draft_static(
        ctypes.byref(dims), _ptr(base_logits), _ptr(h), _ptr(anchor), _ptr(W1), _ptr(W2t),
        _ptr(w_conf), _ptr(T), float(tau), _u64(seed), _ptr(tokens), _ptr(conf), _ptr(logp_d),
        _ptr(lse_d), _stream(stream)), "dspark_markov_draft_static")


def dspark_draft(dims, h, anchor, W_lm, W1, W2t, w_conf, T, tau, seed, base_logits, tokens, conf,
                 logp_d, lse_d, workspace, stream=None):
    _check(load_library().dspark_draft(
        ctypes.byref(dims), _ptr(h), _ptr(anchor), _ptr(W_lm), _ptr(W1), _ptr(W2t), _ptr(w_conf),
        _ptr(T), float(tau), _u64(seed), _ptr(base_logits), _ptr(tokens), _ptr(conf),
        _ptr(logp_d), _ptr(lse_d), _ptr(workspace), workspace.numel(), _stream(stream)),
        "dspark_draft")


def dspark_schedule(conf, R, gamma, sps, mode, k_fixed, length, K_out, theta_out, a_out=None,
                    order_out=None, stream=None):
    _check(load_library().dspark_schedule(
        _ptr(conf), int(R), int(gamma), _ptr(sps), int(sps.numel()), int(mode), int(k_fixed),
        _ptr(length), _ptr(K_out), _ptr(theta_out), _ptr(a_out), _ptr(order_out),
        _stream(stream)), "dspark_schedule")


def dspark_schedule_async(conf, R, gamma, sps, k_ring, length, K_out, theta_out, a_out=None,
                          order_out=None, stream=None):
    _check(load_library().dspark_schedule_async(
        _ptr(conf), int(R), int(gamma), _ptr(sps), int(sps.numel()), _ptr(k_ring), _ptr(length),
        _ptr(K_out), _ptr(theta_out), _ptr(a_out), _ptr(order_out), _stream(stream)),
        "dspark_schedule_async")


def dspark_conf_logits(dims, h, anchor, tokens, W1, w_conf, z, stream=None):
    _check(load_library().dspark_conf_logits(
        ctypes.byref(dims), _ptr(h), _ptr(anchor), _ptr(tokens), _ptr(W1), _ptr(w_conf), _ptr(z),
        _stream(stream)), "dspark_conf_logits")


def dspark_rnn_workspace_bytes(dims) -> int:
    return int(load_library().dspark_rnn_workspace_bytes(ctypes.byref(dims)))


def dspark_rnn_draft(dims, base_logits, h, anchor, W1, W2t, W_rec, W_hid, w_conf, T, tau, seed,
                     tokens, conf, logp_d, lse_d, workspace, stream=None):
    _check(load_library().dspark_rnn_draft(
        ctypes.byref(dims), _ptr(base_logits), _ptr(h), _ptr(anchor), _ptr(W1), _ptr(W2t),
        _ptr(W_rec), _ptr(W_hid), _ptr(w_conf), _ptr(T), float(tau), _u64(seed), _ptr(tokens),
        _ptr(conf), _ptr(logp_d), _ptr(lse_d), _ptr(workspace), workspace.numel(),
        _stream(stream)), "dspark_rnn_draft")


def dspark_fused_workspace_bytes(dims) -> int:
    return int(load_library().dspark_fused_workspace_bytes(ctypes.byref(dims)))


def dspark_pack_fused(dims, W_lm, W2t, W_cat, stream=None):
    _check(load_library().dspark_pack_fused(ctypes.byref(dims), _ptr(W_lm), _ptr(W2t),
                                            _ptr(W_cat), _stream(stream)), "dspark_pack_fused")


def dspark_fused_draft(dims, h, anchor, W_cat, W1, w_conf, T, tau, seed, tokens, conf, logp_d,
                       lse_d, workspace, stream=None):
    _check(load_library().dspark_fused_draft(
        ctypes.byref(dims), _ptr(h), _ptr(anchor), _ptr(W_cat), _ptr(W1), _ptr(w_conf), _ptr(T),
        float(tau), _u64(seed), _ptr(tokens), _ptr(conf), _ptr(logp_d), _ptr(lse_d),
        _ptr(workspace), workspace.numel(), _stream(stream)), "dspark_fused_draft")


def dspark_sts_workspace_bytes(N: int, gamma: int, n_grid: int, n_bins: int) -> int:
    return int(load_library().dspark_sts_workspace_bytes(int(N), int(gamma), int(n_grid),
                                                         int(n_bins)))


def dspark_sts_fit(z, accepted, T_grid, n_bins, T_out, ece_out, workspace=None, stream=None):
    """Fit the per-position temperatures (see include/dspark.h); allocates the
    workspace when none is given."""
    N, G = z.shape
    need = load_library().dspark_sts_workspace_bytes(N, G, T_grid.numel(), int(n_bins))
    if need == 0:
        raise DSparkError("dspark_sts_fit: invalid sizes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=z.device)
    _check(load_library().dspark_sts_fit(
        _ptr(z), _ptr(accepted), int(N), int(G), _ptr(T_grid), int(T_grid.numel()), int(n_bins),
        _ptr(T_out), _ptr(ece_out), _ptr(workspace), workspace.numel(), _stream(stream)),
        "dspark_sts_fit")


def async_ring(k_round0: int, k_round1: int, device="cuda") -> torch.Tensor:
    """The device state of dspark_schedule_async: {K for round 0, K for round 1, cursor 0}."""
    return torch.tensor([int(k_round0), int(k_round1), 0], dtype=torch.int32, device=device)


def dspark_verify(dims, anchor, tokens, length, base_logits, W1, W2t, lse_d, logp_d, target, tau,
                  seed, accepted, bonus, workspace, stream=None):
    _check(load_library().dspark_verify(
        ctypes.byref(dims), _ptr(anchor), _ptr(tokens), _ptr(length), _ptr(base_logits),
        _ptr(W1), _ptr(W2t), _ptr(lse_d), _ptr(logp_d), _ptr(target), float(tau), _u64(seed),
        _ptr(accepted), _ptr(bonus), _ptr(workspace), workspace.numel(), _stream(stream)),
        "dspark_verify")


def dspark_verify_residual_rows(dims, workspace, stream=None):
    """(rejected, explicit_rows) of the last sampling dspark_verify on `workspace`."""
    rej, expl = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(load_library().dspark_verify_residual_rows(
        ctypes.byref(dims), _ptr(workspace), workspace.numel(), ctypes.byref(rej),
        ctypes.byref(expl), _stream(stream)), "dspark_verify_residual_rows")
    return int(rej.value), int(expl.value)


def dspark_device_status(stream=None, clear: bool = True) -> int:
    return int(load_library().dspark_device_status(_stream(stream), 1 if clear else 0))


def dspark_selftest_wait_timeout(limit_ns: int, stream=None):
    _check(load_library().dspark_selftest_wait_timeout(int(limit_ns), _stream(stream)),
           "dspark_selftest_wait_timeout")


def dspark_launch_count() -> int:
    return int(load_library().dspark_launch_count())


def check_device_status(stream=None):
    rc = dspark_device_status(stream)
    _check(rc, "device status")


# ------------------------------------------------------- tensor helpers ----

def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A byte buffer for the library's scratch (torch allocations are 256-B aligned)."""
    t = torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)
    assert t.data_ptr() % 256 == 0
    return t


@dataclass
class DraftHead:
    """Device-resident draft-head weights in the library's layouts."""
    dims: Dims
    W_lm: torch.Tensor    # bf16 [V, d]
    W1: torch.Tensor      # bf16 [V, r]
    W2t: torch.Tensor     # bf16 [V, r]  (W2 transposed once)
    w_conf: torch.Tensor  # bf16 [d + r]
    T: torch.Tensor       # f32 [gamma]

    @staticmethod
    def from_weights(R, gamma, W_lm, W1, W2, w_conf, T, device="cuda") -> "DraftHead":
        V, d = W_lm.shape
        r = W1.shape[1]
        dims = dims_of(R, gamma, V, r, d)
        W2d = _bf16(W2).to(device).contiguous()
        W2t = torch.empty((V, r), dtype=torch.bfloat16, device=device)
        dspark_pack_w2(dims, W2d, W2t)
        return DraftHead(dims, _bf16(W_lm).to(device).contiguous(), _bf16(W1).to(device).contiguous(),
                         W2t, _bf16(w_conf).to(device).contiguous(),
                         T.to(device=device, dtype=torch.float32).contiguous())


class Round:
    """Pre-allocated outputs and workspaces of one round (no allocation per call)."""

    def __init__(self, head: DraftHead, device="cuda"):
        d = head.dims
        self.head = head
        R, G, V = d.R, d.gamma, d.V
        self.base = torch.empty((R * G, V), dtype=torch.bfloat16, device=device)
        self.tokens = torch.empty((R, G), dtype=torch.int32, device=device)
        self.conf = torch.empty((R, G), dtype=torch.float32, device=device)
        self.logp_d = torch.empty((R, G), dtype=torch.float32, device=device)
        self.lse_d = torch.empty((R, G), dtype=torch.float32, device=device)
        self.len = torch.empty((R,), dtype=torch.int32, device=device)
        self.K = torch.empty((1,), dtype=torch.int32, device=device)
        self.theta = torch.empty((1,), dtype=torch.float64, device=device)
        self.accepted = torch.empty((R,), dtype=torch.int32, device=device)
        self.bonus = torch.empty((R,), dtype=torch.int32, device=device)
        self.ws_draft = workspace(dspark_markov_workspace_bytes(d), device)
        self.ws_verify = workspace(dspark_verify_workspace_bytes(d), device)
        # run_host: the target logits come in on a side stream during the draft
        self._copy_stream = torch.cuda.Stream(device=device)
        self._target_ready = torch.cuda.Event()

    def draft(self, h, anchor, tau, seed, stream=None):
        hd = self.head
        dspark_draft(hd.dims, h, anchor, hd.W_lm, hd.W1, hd.W2t, hd.w_conf, hd.T, tau, seed,
                     self.base, self.tokens, self.conf, self.logp_d, self.lse_d, self.ws_draft,
                     stream)

    def schedule(self, sps, mode=SCHED_UNCONSTRAINED, k_fixed=0, stream=None, k_ring=None):
        """mode SCHED_ASYNC takes the device ring of async_ring() and ignores k_fixed."""
        d = self.head.dims
        if mode == SCHED_ASYNC:
            if k_ring is None:
                raise DSparkError("SCHED_ASYNC needs k_ring (see async_ring)")
            dspark_schedule_async(self.conf, d.R, d.gamma, sps, k_ring, self.len, self.K,
                                  self.theta, stream=stream)
            return
        dspark_schedule(self.conf, d.R, d.gamma, sps, mode, k_fixed, self.len, self.K, self.theta,
                        stream=stream)

    def verify(self, anchor, target, tau, seed, stream=None):
        hd = self.head
        dspark_verify(hd.dims, anchor, self.tokens, self.len, self.base, hd.W1, hd.W2t,
                      self.lse_d, self.logp_d, target, tau, seed, self.accepted, self.bonus,
                      self.ws_verify, stream)

    def run(self, h, anchor, target, sps, tau, draft_seed, verify_seed,
            mode=SCHED_UNCONSTRAINED, k_fixed=0, stream=None, k_ring=None):
        """One whole round on device-resident inputs: draft -> schedule -> verify."""
        self.draft(h, anchor, tau, draft_seed, stream)
        self.schedule(sps, mode, k_fixed, stream, k_ring)
        self.verify(anchor, target, tau, verify_seed, stream)

    def run_host(self, h_host, anchor_host, target_host, sps, tau, draft_seed, verify_seed,
                 dev_in: Dict[str, torch.Tensor], out_host: Dict[str, torch.Tensor],
                 mode=SCHED_UNCONSTRAINED, k_fixed=0, stream=None, k_ring=None) -> None:
        """One round from pinned host inputs to pinned host outputs (copies included).

        h and the anchors are copied on `stream` ahead of the draft.  The target
        logits, read only by verify, are copied on a side stream that starts
        once everything already queued on `stream` (the previous round, whose
        verify reads the same buffer) is done, so the copy runs under the draft
        and the schedule; verify waits for it."""
        s = stream if stream is not None else torch.cuda.current_stream()
        c = self._copy_stream
        with torch.cuda.stream(s):
            dev_in["h"].copy_(h_host, non_blocking=True)
            dev_in["anchor"].copy_(anchor_host, non_blocking=True)
        c.wait_stream(s)
        with torch.cuda.stream(c):
            dev_in["target"].copy_(target_host, non_blocking=True)
        dev_in["target"].record_stream(c)
        self._target_ready.record(c)
        self.draft(dev_in["h"], dev_in["anchor"], tau, draft_seed, s)
        self.schedule(sps, mode, k_fixed, s, k_ring)
        s.wait_event(self._target_ready)
        self.verify(dev_in["anchor"], dev_in["target"], tau, verify_seed, s)
        with torch.cuda.stream(s):
            out_host["tokens"].copy_(self.tokens, non_blocking=True)
            out_host["len"].copy_(self.len, non_blocking=True)
            out_host["accepted"].copy_(self.accepted, non_blocking=True)
            out_host["bonus"].copy_(self.bonus, non_blocking=True)
