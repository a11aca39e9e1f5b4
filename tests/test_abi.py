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
