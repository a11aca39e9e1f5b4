"""Host-side pieces on CPU: the binding's argument marshalling checks and the
seeded input generators (shapes, dtypes, determinism, scales)."""

import numpy as np
import pytest
import torch

from speculative_decoding_head_gb300 import binding
from speculative_decoding_head_gb300.workloads import (STS_SETS, WORKLOADS, make_inputs, make_loss_inputs,
                                                       make_rnn_weights, make_sts_inputs, pack_rows, row_offsets)


def test_ptr_rejects_host_noncontiguous_and_wrong_dtype_tensors():
    assert binding._ptr(None).value in (None, 0)
    with pytest.raises(binding.DsparkError):
        binding._ptr(torch.zeros(4), name="x")                       # not a CUDA tensor
    if torch.cuda.is_available():
        with pytest.raises(binding.DsparkError):
            binding._ptr(torch.zeros(4, 4, device="cuda").t(), name="x")
        with pytest.raises(binding.DsparkError):
            binding._ptr(torch.zeros(4, device="cuda"), torch.int32, name="x")


def test_generators_are_deterministic_and_shaped():
    wl = WORKLOADS["tiny"]
    a, b = make_inputs(wl), make_inputs(wl)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    B, g, V, r, H = wl.B, wl.gamma, wl.V, wl.r, wl.H
    assert a["U"].shape == (B, g, V) and a["W1"].shape == (V, r) and a["W2"].shape == (r, V)
    assert a["h"].shape == (B, g, H) and a["w"].shape == (H + r,) and a["P_full"].shape == (B, g + 1, V)
    assert a["anchor"].dtype == torch.int32 and ((a["anchor"] >= 0) & (a["anchor"] < V)).all()


def test_loss_and_rnn_generators():
    wl = WORKLOADS["small"].with_(B=3, gamma=4, V=512, r=64, H=32)
    li = make_loss_inputs(wl)
    assert li["P"].shape == (3, 4, 512) and li["xstar"].dtype == torch.int32
    assert ((li["conf"] > 0.0) & (li["conf"] < 1.0)).all()
    assert torch.equal(li["P"], make_inputs(wl)["P_full"][:, :4])
    Wr = make_rnn_weights(wl)
    Z = 2 * wl.r + wl.H
    assert Wr.shape == (3, wl.r, Z) and Wr.dtype == torch.bfloat16
    assert abs(float(Wr.float().std()) * Z ** 0.5 - 1.0) < 0.05
    assert torch.equal(Wr, make_rnn_weights(wl))


def test_sts_sets_and_packing():
    c = STS_SETS["sts_small"]
    s = make_sts_inputs(1000, c["gamma"], c["seed"])
    assert s["raw"].shape == (1000, c["gamma"]) and ((s["cstar"] >= 0.02) & (s["cstar"] <= 0.98)).all()
    P = torch.arange(2 * 3 * 5, dtype=torch.float32).reshape(2, 3, 5)
    L = torch.tensor([2, 1], dtype=torch.int32)
    packed = pack_rows(P, L)
    assert torch.equal(packed, torch.stack([P[0, 0], P[0, 1], P[1, 0]]))
    assert row_offsets(L).tolist() == [0, 2, 3]
