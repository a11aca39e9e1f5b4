"""The C-ABI library loads and exports every entry point include/dspark.h declares.

Runs without a GPU: only symbol lookup and host-only entry points are called.
"""

import ctypes
import os
import re

import pytest
import torch

from speculative_decoding_head_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    out = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            out |= set(re.findall(r"\b(dspark_[a-z_0-9]+)\s*\(", src))
    return out


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_library_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert {"dspark_markov_draft", "dspark_plan", "dspark_verify"} <= syms
    for s in sorted(syms):
        assert hasattr(lib, s), f"{s} declared in include/ but not exported"
    assert set(binding.SYMBOLS) <= syms


def test_status_strings_are_host_only(lib):
    for code, text in [(0, "ok"), (1, "invalid argument"), (3, "grid barrier timed out"), (99, "unknown status")]:
        assert binding.status_string(code) == text


def test_invalid_dims_are_rejected_before_touching_the_device(lib):
    h = ctypes.c_void_p()
    bad = [
        binding.Dims(0, 5, 1024, 16, 64, 0, 1, 0),      # B = 0
        binding.Dims(2, 0, 1024, 16, 64, 0, 1, 0),      # gamma = 0
        binding.Dims(2, 3, 1001, 16, 64, 1, 1, 0),      # bf16 needs V % 8 == 0
        binding.Dims(2, 3, 1024, 16, 64, 0, 2, 0),      # lagged needs lag >= 1
        binding.Dims(2, 3, 1024, 16, 64, 7, 1, 0),      # bad dtype
    ]
    for d in bad:
        assert lib.dspark_ws_create(ctypes.byref(d), ctypes.byref(h)) == 1
    assert lib.dspark_ws_create(None, ctypes.byref(h)) == 1
    # no workspace: every call is EINVAL
    assert lib.dspark_plan(None, None, None, None, None, None) == 1
    assert lib.dspark_last_launch_count(None) == -1


def test_workspace_creation_without_gpu_reports_cuda_error(lib):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    d = binding.Dims(2, 3, 1024, 16, 64, 0, 1, 0)
    assert lib.dspark_ws_create(ctypes.byref(d), ctypes.byref(h)) == 2


def test_binding_refuses_missing_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(binding.DsparkError):
        binding.load()


def test_sts_fit_arguments_are_checked_on_the_host(lib):
    """Bad sizes and null pointers are EINVAL / EUNSUPPORTED before any CUDA call."""
    fake = ctypes.c_void_p(16)   # never dereferenced: the checks come first
    args = dict(raw=fake, cstar=fake, N=100, g=4, Tgrid=fake, G=10, M=15, T=fake, ece=fake, scratch=fake, st=fake)

    def call(**kw):
        a = {**args, **kw}
        return lib.dspark_sts_fit(a["raw"], a["cstar"], a["N"], a["g"], a["Tgrid"], a["G"], a["M"], a["T"], a["ece"],
                                  a["scratch"], a["st"], None)

    assert call(M=0) == 1 and call(M=33) == 1            # 1 <= M <= 32
    assert call(N=0) == 1 and call(g=0) == 1 and call(G=0) == 1 and call(G=70000) == 1
    assert call(raw=None) == 1 and call(scratch=None) == 1 and call(st=None) == 1
    assert call(N=1 << 23) == 5                          # the fixed-point bin sums' range
    assert lib.dspark_sts_scratch_bytes(1000, 10) == 8 * 10 * 8 * 32 + 8 * 10 + 16 * 1000


def test_train_loss_arguments_are_checked_on_the_host(lib):
    """No workspace or a null pointer is EINVAL before any CUDA call."""
    fake = ctypes.c_void_p(256)
    assert lib.dspark_train_loss(None, *([fake] * 7), 4.0, *([fake] * 5), None) == 1
    assert lib.dspark_train_loss_scratch_bytes(None) == 0


def test_rnn_draft_arguments_are_checked_on_the_host(lib):
    fake = ctypes.c_void_p(256)
    assert lib.dspark_rnn_draft(None, *([fake] * 8), 0, 0, *([fake] * 6), None) == 1
    assert lib.dspark_rnn_draft_scratch_bytes(None) == 0


def test_rnn_verify_arguments_are_checked_on_the_host(lib):
    fake = ctypes.c_void_p(256)
    assert lib.dspark_verify_rnn(None, *([fake] * 10), 0, 0, fake, fake, None) == 1
