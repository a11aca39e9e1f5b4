"""dspark_markov_draft_noalloc against dspark_markov_draft, through the C-ABI.

The allocation-free entry point serves callers that cannot call cudaMalloc
(an engine whose pool owns all device memory, a plug-in that must not grow
the device footprint, code under a hard memory budget). It runs the same
CUDA-core draft kernels with scratch from an array built into the library,
so its output must match the workspace entry point's "simt" draft: token ids
exactly, probabilities, log-sum-exps and confidences within the 1e-4
relative tolerance of the other parity tests. Two calls in a row check that
the shared scratch left by one call does not leak into the next.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""

import ctypes as C

import numpy as np
import pytest
import torch

from speculative_decoding_head_gb300 import binding, build
from speculative_decoding_head_gb300.binding import Dims, Workspace
from speculative_decoding_head_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

RTOL = 1e-4


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else C.c_void_p(0)


def _noalloc(lib, wl, dev, seed, rnd, anchor):
    B, g = wl.B, wl.gamma
    out = {"tokens": torch.full((B, g), -1, dtype=torch.int32, device="cuda"),
           "pd_tok": torch.zeros((B, g), device="cuda"), "lse": torch.zeros((B, g), device="cuda"),
           "conf": torch.zeros((B, g), device="cuda")}
    status = torch.full((4,), 77, dtype=torch.int32, device="cuda")  # the call must clear it
    dims = Dims(B, g, wl.V, wl.r, wl.H, binding.WDTYPES[wl.wdtype], binding.MODES[wl.mode], 0)
    code = lib.dspark_markov_draft_noalloc(
        C.byref(dims), _ptr(dev["U"]), _ptr(dev["W1"]), _ptr(dev["W2"]), _ptr(anchor), _ptr(dev["h"]),
        _ptr(dev["w"]), _ptr(dev["T"]), C.c_uint64(seed), C.c_uint64(rnd), _ptr(out["tokens"]),
        _ptr(out["pd_tok"]), _ptr(out["lse"]), _ptr(out["conf"]), _ptr(status),
        C.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert code == 0, binding.status_string(code)
    assert int(status[0].item()) == 0
    return {k: v.cpu().numpy() for k, v in out.items()}


def _close(a, b):
    return np.all(np.abs(a.astype(np.float64) - b) <= RTOL * np.abs(b.astype(np.float64)) + 1e-30)


def test_noalloc_draft_matches_workspace_draft_on_two_calls():
    build.build()
    lib = binding.load()
    lib.dspark_markov_draft_noalloc.argtypes = [C.c_void_p] * 8 + [C.c_uint64, C.c_uint64] + [C.c_void_p] * 6
    lib.dspark_markov_draft_noalloc.restype = C.c_int
    wl = Workload("noalloc", B=48, gamma=4, V=5000, r=256, H=96, wdtype="bf16", mode="static", seed=41,
                  u_std=2.0, w_std=0.05)
    dev = {k: v.cuda().contiguous() for k, v in make_inputs(wl, with_target=False).items()}
    ws = Workspace.for_workload(wl, path="simt")
    anchors = [dev["anchor"], torch.roll(dev["anchor"], 7).contiguous()]
    for call, (rnd, anchor) in enumerate(zip((3, 4), anchors)):
        ref = ws.draft(dev["U"], dev["W1"], dev["W2"], anchor, dev["h"], dev["w"], dev["T"], 9, rnd)
        torch.cuda.synchronize()
        assert ws.device_status() == 0
        ref = {k: v.cpu().numpy() for k, v in ref.items()}
        got = _noalloc(lib, wl, dev, 9, rnd, anchor)
        assert (got["tokens"] == ref["tokens"]).all(), call
        for k in ("pd_tok", "lse", "conf"):
            assert _close(got[k], ref[k]), (call, k)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = binding.load()
    lib.dspark_markov_draft_noalloc.argtypes = [C.c_void_p] * 8 + [C.c_uint64, C.c_uint64] + [C.c_void_p] * 6
    lib.dspark_markov_draft_noalloc.restype = C.c_int
    big = Dims(4096, 5, 129280, 256, 0, 1, 0, 0)      # 4096 * 2020 block masses > 2^20 floats
    t = torch.zeros(64, device="cuda")
    p = C.c_void_p(t.data_ptr())
    code = lib.dspark_markov_draft_noalloc(C.byref(big), p, p, p, p, None, p, p, C.c_uint64(0), C.c_uint64(0),
                                           p, p, p, p, p, C.c_void_p(0))
    assert code == 5   # DSPARK_EUNSUPPORTED, nothing enqueued
