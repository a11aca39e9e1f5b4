"""The persistent tcgen05 draft kernel against the oracle and the SIMT path.

Shapes cover one and several 128-row groups, a vocabulary that ends inside a
64-token tile (the last TMA boxes run out of bounds), every supported rank
(64..256) and batches smaller than one MMA tile.
"""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_head_gb300 import build
from speculative_decoding_head_gb300.binding import Workspace
from speculative_decoding_head_gb300.workloads import WORKLOADS, Workload, make_inputs

from parity import check_draft, gpu_np, np_inputs, rel_close, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _wl(name, B, gamma, V, r, H=32, seed=31):
    return Workload(name, B=B, gamma=gamma, V=V, r=r, H=H, wdtype="bf16", mode="static", seed=seed,
                    u_std=2.0, w_std=0.05)


def _draft(wl, dev, path, seed, rnd):
    ws = Workspace.for_workload(wl, path=path)
    assert ws.path == path
    d = ws.draft(dev["U"], dev["W1"], dev["W2"], dev["anchor"], dev["h"], dev["w"], dev["T"], seed, rnd)
    torch.cuda.synchronize()
    st = ws.device_status()
    assert st == 0, f"{path}: device status {st}"
    return gpu_np(d), ws


def _check(wl, rnd=0, reqs=None):
    inp = make_inputs(wl, with_target=False)
    dev, npi = to_device(inp), np_inputs(inp)
    tc, ws = _draft(wl, dev, "tcgen05", wl.seed, rnd)
    assert ws.last_launches == 1          # one persistent kernel
    simt, _ = _draft(wl, dev, "simt", wl.seed, rnd)
    reqs = range(wl.B) if reqs is None else reqs

    def draft_fn(rq, force):
        return oracle.draft(npi["U"], npi["W1"], npi["W2"], npi["anchor"], npi["h"], npi["w"], npi["T"], wl.seed,
                            rnd, reqs=rq, force=force)

    for name, g in (("tcgen05", tc), ("simt", simt)):
        t, od = check_draft(g, draft_fn, reqs)
        t.check_rate()
    # the two GPU paths agree on every value the oracle compared
    rr = list(reqs)
    assert rel_close(tc["lse"][rr], simt["lse"][rr]).all()
    assert rel_close(tc["conf"][rr], simt["conf"][rr]).all()
    return tc, simt, od


def test_tc_smallest():
    _check(_wl("tc_small", B=16, gamma=2, V=1024, r=64))


@pytest.mark.parametrize("B,gamma,V,r", [
    (1, 1, 64, 64),          # one row, one tile
    (5, 3, 1000, 128),       # vocabulary ends inside a tile
    (130, 2, 4104, 256),     # two row groups, the second nearly empty
    (200, 3, 2048, 192),     # two row groups, rank 192
    (256, 2, 6000, 256),     # two full row groups
    (64, 16, 2048, 128),     # a long block: sixteen steps, sixteen grid barriers
    (1000, 2, 1088, 64),     # eight row groups, the last one ragged
])
def test_tc_shapes(B, gamma, V, r):
    _check(_wl(f"tc_{B}_{V}_{r}", B=B, gamma=gamma, V=V, r=r, seed=B + V + r))


def test_tc_prod_full_size_sampled():
    wl = WORKLOADS["prod"]
    inp = make_inputs(wl, with_target=False)
    dev = to_device(inp)
    tc, _ = _draft(wl, dev, "tcgen05", wl.seed, 2)
    sub = np_inputs({k: inp[k] for k in ("W1", "W2")})

    def draft_fn(rq, force):
        return oracle.draft(inp["U"].numpy(), sub["W1"], sub["W2"], inp["anchor"].numpy(), inp["h"].numpy(),
                            inp["w"].numpy(), inp["T"].numpy(), wl.seed, 2, reqs=rq, force=force)

    t, _ = check_draft(tc, draft_fn, range(wl.B))     # every request of the batch
    t.check_rate()


def test_tc_repeatable_and_round_sensitive():
    wl = _wl("tc_rep", B=64, gamma=3, V=2048, r=256)
    dev = to_device(make_inputs(wl, with_target=False))
    a, _ = _draft(wl, dev, "tcgen05", 3, 7)
    b, _ = _draft(wl, dev, "tcgen05", 3, 7)
    c, _ = _draft(wl, dev, "tcgen05", 3, 8)
    for k in a:
        assert (a[k] == b[k]).all()
    assert not (a["tokens"] == c["tokens"]).all()


@pytest.mark.parametrize("B,gamma,V,r,sigma", [
    (24, 3, 1000, 128, 2.0),     # vocabulary ends inside a 128-wide tile
    (300, 2, 3000, 256, 3.0),    # most drafts rejected: three groups of 128 requests
    (128, 5, 8192, 192, 0.5),
])
def test_residual_paths_match_oracle(B, gamma, V, r, sigma):
    """Verify on the oracle's drafts with the tcgen05 and the SIMT residual pass."""
    from parity import Tally, compare_verify, pack_np, row_off_np
    wl = Workload(f"resid_{B}_{V}", B=B, gamma=gamma, V=V, r=r, H=16, wdtype="bf16", mode="static",
                  seed=B + V, u_std=2.0, w_std=0.05, noise="const", noise_args=(sigma,))
    inp = make_inputs(wl)
    dev, npi = to_device(inp), np_inputs(inp)
    od = oracle.draft(npi["U"], npi["W1"], npi["W2"], npi["anchor"], npi["h"], npi["w"], npi["T"], 3, 1)
    rng = np.random.default_rng(B)
    L = rng.integers(1, gamma + 2, B).astype(np.int32)
    ro = row_off_np(L)
    P = pack_np(npi["P_full"], L)
    ov = oracle.verify(P, ro, L, npi["anchor"], od["tokens"], npi["U"], npi["W1"], npi["W2"], 3, 1)
    assert ov["resid"].sum() > 0
    outs = {}
    for path in ("tcgen05", "simt"):
        ws = Workspace.for_workload(wl, path=path)
        out = ws.verify(torch.from_numpy(P).cuda(), torch.from_numpy(ro).cuda(), torch.from_numpy(L).cuda(),
                        dev["anchor"], torch.from_numpy(od["tokens"]).cuda(),
                        torch.from_numpy(od["pd_tok"].astype(np.float32)).cuda(),
                        torch.from_numpy(od["lse"].astype(np.float32)).cuda(), dev["U"], dev["W1"], dev["W2"], 3, 1)
        torch.cuda.synchronize()
        assert ws.device_status() == 0, path
        outs[path] = gpu_np(out)
        t = compare_verify(outs[path], ov, range(B))
        t.check_rate()
        assert t.compared > 0
