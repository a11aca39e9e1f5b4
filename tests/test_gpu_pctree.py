"""PCTree (the chain made a tree) on the GPU against the oracle.

The build is compared node by node: token, parent, depth and the node count
bit-exact, the path log-probability within 2e-5 + 1e-5 |lp| (fp32 sums of a
recomputed fp32 z minus an fp32 log-sum-exp along at most gamma levels),
for every request whose decisions the oracle does not call too close
(margin < oracle.MARGIN: a top-c choice or an admission decided by a
log-probability gap below 1e-5; such requests are counted). The verify walks
the same tree (the oracle's) on both sides: accepted path, accepted count and
next anchor bit-exact except at flagged requests.
"""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_head_gb300 import build
from speculative_decoding_head_gb300.binding import Workspace
from speculative_decoding_head_gb300.workloads import WORKLOADS, Workload, make_inputs, make_tree_targets

from parity import _record, np_inputs, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _wl(name, B, gamma, V, r, wdtype="bf16", seed=51):
    return Workload(name, B=B, gamma=gamma, V=V, r=r, H=8, wdtype=wdtype, mode="static", seed=seed, u_std=2.0,
                    w_std=0.05 if wdtype == "bf16" else 0.3)


def _check_build(g, o, reqs, N):
    flagged = compared = 0
    for b in reqs:
        if o["margin"][b] < oracle.MARGIN:
            flagged += 1
            continue
        assert g["n_nodes"][b] == o["n_nodes"][b], (b, g["n_nodes"][b], o["n_nodes"][b])
        n = int(o["n_nodes"][b]) + 1
        for k in ("tok", "par", "dep"):
            assert (g[k][b, :n] == o[k][b, :n]).all(), (k, b, g[k][b, :n], o[k][b, :n])
            assert (g[k][b, n:] == -1).all(), (k, b)
        d = np.abs(g["lp"][b, :n] - o["lp"][b, :n])
        assert (d <= 2e-5 + 1e-5 * np.abs(o["lp"][b, :n])).all(), (b, d.max())
        compared += 1
    _record("tree", compared * N, flagged)
    assert flagged <= 1 + 1e-4 * len(reqs) * N, flagged
    return compared


def _check_verify(gv, ov, reqs):
    flagged = compared = 0
    for b in reqs:
        if ov["margin"][b] < oracle.MARGIN:
            flagged += 1
            continue
        assert gv["n_acc"][b] == ov["n_acc"][b], (b, gv["n_acc"][b], ov["n_acc"][b])
        assert (gv["path"][b] == ov["path"][b]).all(), (b, gv["path"][b], ov["path"][b])
        assert gv["next_anchor"][b] == ov["next_anchor"][b], (b, gv["next_anchor"][b], ov["next_anchor"][b])
        compared += 1
    _record("treev", compared, flagged)
    assert flagged <= 1 + 1e-4 * len(reqs), flagged
    return compared


def _run(wl, c, N, path=None, reqs=None, sigma=0.5, rnd=3):
    inp = make_inputs(wl, with_target=False)
    dev, npi = to_device(inp), np_inputs(inp)
    ws = Workspace.for_workload(wl, path=path)
    gb = ws.pctree_build(dev["U"], dev["W1"], dev["W2"], dev["anchor"], c, N)
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    g = {k: v.cpu().numpy() for k, v in gb.items() if k != "scratch"}
    reqs = list(range(wl.B)) if reqs is None else list(reqs)
    o = oracle.pctree_build(npi["U"], npi["W1"], npi["W2"], npi["anchor"], c, N, reqs=reqs)
    assert _check_build(g, o, reqs, N) > 0
    # the verify walks the oracle's tree on both sides (the GPU's where they agree)
    P = make_tree_targets(wl, inp["U"], torch.from_numpy(o["dep"]), sigma=sigma)
    tok = torch.from_numpy(o["tok"]).cuda()
    par = torch.from_numpy(o["par"]).cuda()
    gv = ws.pctree_verify(P.cuda(), tok, par, N, wl.seed, rnd)
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    gv = {k: v.cpu().numpy() for k, v in gv.items()}
    ov = oracle.pctree_verify(o["tok"], o["par"], P.numpy(), wl.gamma, wl.seed, rnd, reqs=reqs)
    assert _check_verify(gv, ov, reqs) > 0
    return g, o, gv, ov


@pytest.mark.parametrize("wl,c,N", [
    (_wl("tree_tiny_f32", 2, 3, 1024, 16, "f32"), 2, 6),
    (_wl("tree_f32", 12, 4, 3000, 32, "f32", seed=52), 3, 12),
], ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_pctree_simt(wl, c, N):
    _run(wl, c, N)


@pytest.mark.parametrize("wl,c,N", [
    (_wl("tree_bf16", 40, 5, 4104, 256), 4, 16),      # a vocabulary ending inside a 128-wide tile
    (_wl("tree_deep", 20, 3, 2048, 64, seed=53), 2, 24),  # depth-limited: every path reaches gamma
    (_wl("tree_wide", 70, 5, 6000, 128, seed=54), 8, 8),
], ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_pctree_tcgen05(wl, c, N):
    g, o, gv, ov = _run(wl, c, N)
    assert (g["n_nodes"] <= N).all()


def test_pctree_both_paths_agree():
    wl = _wl("tree_paths", 16, 4, 2048, 64, seed=55)
    inp = to_device(make_inputs(wl, with_target=False))
    outs = []
    for path in ("tcgen05", "simt"):
        ws = Workspace.for_workload(wl, path=path)
        t = ws.pctree_build(inp["U"], inp["W1"], inp["W2"], inp["anchor"], 3, 10)
        torch.cuda.synchronize()
        assert ws.device_status() == 0
        outs.append({k: v.cpu().numpy() for k, v in t.items() if k != "scratch"})
    for k in ("tok", "par", "dep", "n_nodes"):
        assert (outs[0][k] == outs[1][k]).all(), k


def test_pctree_prod_shape_sampled():
    """B=128, gamma=5, V=129280, r=256, c=4, N=16: the GPU builds and verifies
    every request; the oracle checks six of them."""
    _run(WORKLOADS["prod"], 4, 16, reqs=[0, 1, 50, 64, 100, 127])
