"""The draft head's teacher-forced training objective on the GPU against the oracle.

Tolerances, from the arithmetic of the two vocabulary passes: z_d is an fp32
accumulation of r bf16 products (error ~1e-6 against the oracle's fp64), the
log-sum-exps combine fp32 (max, sum exp) pairs with ex2.approx (relative error
2^-22 per term), so lse and z_d at x* carry ~1e-6 relative error and ce, a
difference of two values of magnitude ~15, ~2e-5 absolute. l1 sums V terms of
|p_d - p_t| whose magnitudes add to at most 2, each with ~1e-6 relative error:
~2e-6 absolute plus fp32 summation. bce moves by |logit(c)| / 2 per unit of
l1. The loss is the weighted sum of the three, so its tolerance is the same
weighted sum of theirs.
"""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_head_gb300 import build
from speculative_decoding_head_gb300.binding import Workspace
from speculative_decoding_head_gb300.workloads import WORKLOADS, Workload, make_loss_inputs

from parity import np_inputs, to_device

pytestmark = pytest.mark.gpu

CE_ABS, CE_REL = 5e-5, 2e-6
L1_ABS = 2e-5
BCE_REL = 2e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _wl(name, B, gamma, V, r, seed=23):
    return Workload(name, B=B, gamma=gamma, V=V, r=r, H=0, wdtype="bf16", mode="static", seed=seed,
                    u_std=2.0, w_std=0.05)


def _tols(conf, ce_o, bce_o):
    tce = CE_ABS + CE_REL * np.abs(ce_o)
    c = conf.astype(np.float64)
    tbce = 0.5 * L1_ABS * np.abs(np.log(c / (1.0 - c))) + BCE_REL * np.abs(bce_o) + 1e-6
    return tce, tbce


def _gpu(wl, dev, tau):
    ws = Workspace.for_workload(wl)
    out = ws.train_loss(dev["U"], dev["W1"], dev["W2"], dev["anchor"], dev["xstar"], dev["P"], dev["conf"], tau)
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    assert ws.last_launches == 5
    return {k: out[k].cpu().numpy().astype(np.float64) for k in ("ce", "l1", "bce", "loss")}


def _compare(g, o, conf, rows, tau):
    ce_o, l1_o, bce_o = o["ce"], o["l1"], o["bce"]
    tce, tbce = _tols(conf[rows], ce_o, bce_o)
    assert (np.abs(g["ce"][rows] - ce_o) <= tce).all(), np.abs(g["ce"][rows] - ce_o).max()
    assert (np.abs(g["l1"][rows] - l1_o) <= L1_ABS).all(), np.abs(g["l1"][rows] - l1_o).max()
    assert (np.abs(g["bce"][rows] - bce_o) <= tbce).all(), np.abs(g["bce"][rows] - bce_o).max()
    k = np.arange(ce_o.shape[1])
    w = np.exp(-k / tau)
    tloss = float((w * (0.1 * tce + 0.9 * L1_ABS + tbce)).sum() / ce_o.shape[0])
    return tloss


@pytest.mark.parametrize("B,gamma,V,r,tau", [
    (2, 3, 1024, 64, 4.0),        # one column group, 8 tiles over 152 CTAs (most CTAs idle)
    (12, 5, 4104, 256, 4.0),      # two groups, the second ragged; a vocabulary ending inside a tile
    (7, 9, 33000, 128, 1.5),      # two groups of 32 and 31; several tiles per CTA
    (40, 4, 8192, 192, 100.0),    # five full groups, r = 192
])
def test_loss_parity(B, gamma, V, r, tau):
    wl = _wl(f"loss_{B}_{gamma}_{V}_{r}", B, gamma, V, r)
    inp = make_loss_inputs(wl)
    npi = np_inputs(inp)
    g = _gpu(wl, to_device(inp), tau)
    o = oracle.train_loss(npi["U"], npi["W1"], npi["W2"], npi["anchor"], npi["xstar"], npi["P"], npi["conf"], tau)
    tloss = _compare(g, o, npi["conf"], slice(None), tau)
    assert abs(g["loss"][0] - o["loss"]) <= tloss, (g["loss"][0], o["loss"], tloss)


def test_loss_full_size_sampled():
    """The prod shape (B=128, gamma=5, V=129280, r=256): the oracle on eight
    requests spread over the batch (positions are independent under teacher
    forcing), and the GPU's loss against the fp64 weighted sum of its own
    per-position values."""
    wl = WORKLOADS["prod"]
    tau = 4.0
    inp = make_loss_inputs(wl)
    npi = np_inputs(inp)
    g = _gpu(wl, to_device(inp), tau)
    rows = np.array([0, 17, 40, 63, 64, 99, 126, 127])
    sub = {k: npi[k][rows] for k in ("U", "anchor", "xstar", "P", "conf")}
    o = oracle.train_loss(sub["U"], npi["W1"], npi["W2"], sub["anchor"], sub["xstar"], sub["P"], sub["conf"], tau)
    _compare(g, o, npi["conf"], rows, tau)
    w = np.exp(-np.arange(wl.gamma) / tau)
    own = float((w * (0.1 * g["ce"] + 0.9 * g["l1"] + g["bce"])).sum() / wl.B)
    assert abs(g["loss"][0] - own) <= 1e-6 * abs(own) + 1e-6


def test_loss_identical_distributions_and_zero_head():
    """W1 = 0 and P = U: p_d = p_t, so l1 = 0 (c* = 1, bce = -log c) and ce
    is the target's own cross entropy at x*, whatever the draft would add."""
    wl = _wl("loss_ident", 6, 4, 5000, 64)
    inp = make_loss_inputs(wl)
    inp["W1"] = torch.zeros_like(inp["W1"])
    inp["P"] = inp["U"].clone()
    npi = np_inputs(inp)
    g = _gpu(wl, to_device(inp), 2.0)
    assert np.abs(g["l1"]).max() <= L1_ABS
    c = npi["conf"].astype(np.float64)
    assert np.allclose(g["bce"], -np.log(c), rtol=0, atol=1e-4)
    U = npi["U"].astype(np.float64)
    m = U.max(-1, keepdims=True)
    lse = (m + np.log(np.exp(U - m).sum(-1, keepdims=True)))[..., 0]
    ux = np.take_along_axis(U, npi["xstar"][..., None].astype(np.int64), -1)[..., 0]
    assert np.allclose(g["ce"], lse - ux, rtol=0, atol=CE_ABS)


def test_loss_bad_tokens_and_confidences_are_reported():
    wl = _wl("loss_bad", 3, 2, 1024, 64)
    inp = make_loss_inputs(wl)
    dev = to_device(inp)
    ws = Workspace.for_workload(wl)
    bad = dev["xstar"].clone()
    bad[1, 1] = wl.V                      # out of range: clamped to 0 in the kernel, reported
    ws.train_loss(dev["U"], dev["W1"], dev["W2"], dev["anchor"], bad, dev["P"], dev["conf"], 4.0)
    torch.cuda.synchronize()
    assert ws.device_status() == 6        # DSPARK_ERANGE
    ws.reset()
    conf = dev["conf"].clone()
    conf[0, 0] = 1.0
    ws.train_loss(dev["U"], dev["W1"], dev["W2"], dev["anchor"], dev["xstar"], dev["P"], conf, 4.0)
    torch.cuda.synchronize()
    assert ws.device_status() == 4        # DSPARK_ENUMERIC
