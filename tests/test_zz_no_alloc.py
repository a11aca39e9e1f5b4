"""dspark_markov_draft_noalloc against dspark_markov_draft, through the C-ABI.

The allocation-free entry point serves callers that cannot call cudaMalloc
(an engine whose pool owns all device memory, a plug-in that must not grow
the device footprint, code under a hard memory budget). It runs the same
CUDA-core draft kernels with scratch from an array built into the library,
so its output must match the workspace entry point's "simt" draft: token ids
exactly, probabilities, log-sum-exps and confidences within the 1e-4
relative tolerance of the other parity tests. It is also held to the fp64
oracle under the parity rule of the other draft tests (bit-exact tokens
except where the oracle calls a draw too close, where it adopts the GPU's
token). Two calls in a row check that the shared scratch left by one call
does not leak into the next. The cases cover bf16 and fp32 weights, no
hidden states (H = 0: the hidden half of each confidence logit is cleared,
not computed), and a shape whose scratch fills the array exactly.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""

import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_head_gb300 import binding, build
from speculative_decoding_head_gb300.binding import Dims, Workspace
from speculative_decoding_head_gb300.workloads import Workload, make_inputs

from parity import check_draft, np_inputs

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


def _lib():
    build.build()
    lib = binding.load()
    lib.dspark_markov_draft_noalloc.argtypes = [C.c_void_p] * 8 + [C.c_uint64, C.c_uint64] + [C.c_void_p] * 6
    lib.dspark_markov_draft_noalloc.restype = C.c_int
    return lib


# scratch floats of a shape: B * gamma rounded up to 64, plus B * ceil(V / 64)
LIMIT = 1 << 20
CASES = [
    Workload("noalloc_bf16", B=48, gamma=4, V=5000, r=256, H=96, wdtype="bf16", mode="static", seed=41,
             u_std=2.0, w_std=0.05),
    Workload("noalloc_f32", B=20, gamma=3, V=3001, r=32, H=40, wdtype="f32", mode="static", seed=42,
             u_std=2.0, w_std=0.1),
    Workload("noalloc_noh", B=16, gamma=5, V=2048, r=64, H=0, wdtype="bf16", mode="static", seed=43,
             u_std=2.0, w_std=0.05),
    # 256 * 4 = 1024 hidden halves plus 256 * 4092 block masses = 2^20 floats
    Workload("noalloc_full", B=256, gamma=4, V=4092 * 64, r=16, H=8, wdtype="bf16", mode="static", seed=44,
             u_std=2.0, w_std=0.05),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_noalloc_draft_matches_workspace_draft_and_oracle_on_two_calls(wl):
    lib = _lib()
    nblk = (wl.V + 63) // 64
    need = (wl.B * wl.gamma + 63) // 64 * 64 + wl.B * nblk
    assert need <= LIMIT
    if wl.name == "noalloc_full":
        assert need == LIMIT
    inp = make_inputs(wl, with_target=False)
    npi = np_inputs(inp)
    dev = {k: v.cuda().contiguous() for k, v in inp.items()}
    ws = Workspace.for_workload(wl, path="simt")
    anchors = [dev["anchor"], torch.roll(dev["anchor"], 7).contiguous()]
    # the oracle on every request of the small cases, on a sample of the full one
    reqs = list(range(wl.B)) if wl.B * wl.V <= 1 << 22 else [0, 1, 77, 128, 255]
    for call, (rnd, anchor) in enumerate(zip((3, 4), anchors)):
        ref = ws.draft(dev["U"], dev["W1"], dev["W2"], anchor, dev["h"], dev["w"], dev["T"], 9, rnd)
        torch.cuda.synchronize()
        assert ws.device_status() == 0
        ref = {k: v.cpu().numpy() for k, v in ref.items()}
        got = _noalloc(lib, wl, dev, 9, rnd, anchor)
        assert (got["tokens"] == ref["tokens"]).all(), call
        for k in ("pd_tok", "lse", "conf"):
            assert _close(got[k], ref[k]), (call, k)
        an = anchor.cpu().numpy()

        def draft_fn(rq, force, an=an, rnd=rnd):
            return oracle.draft(npi["U"], npi["W1"], npi["W2"], an, npi["h"], npi["w"], npi["T"], 9, rnd, reqs=rq,
                                force=force)

        t, _ = check_draft(got, draft_fn, reqs)
        t.check_rate()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = _lib()
    t = torch.zeros(64, device="cuda")
    p = C.c_void_p(t.data_ptr())
    for big in (Dims(4096, 5, 129280, 256, 0, 1, 0, 0),        # 4096 * 2020 block masses
                Dims(256, 4, 4092 * 64 + 1, 16, 0, 1, 0, 0)):  # one block past the exact fit
        code = lib.dspark_markov_draft_noalloc(C.byref(big), p, p, p, p, None, p, p, C.c_uint64(0),
                                               C.c_uint64(0), p, p, p, p, p, C.c_void_p(0))
        assert code == 5   # DSPARK_EUNSUPPORTED, nothing enqueued
