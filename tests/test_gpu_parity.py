"""GPU (C-ABI) vs fp64 oracle parity on seeded synthetic rounds.

Sizes: small enough for the oracle to finish in seconds yet spanning many
64-token blocks, a ragged last block, several 128-row groups; plus the
benchmark workloads at full size, every request, each in its own planner mode
(prod compact, long static, loaded lagged over chained rounds).

Rounds are chained under teacher forcing: where the oracle flags a decision
(a draw, a plan or a verify outcome too close to call in fp32) and the two
sides differ, the oracle adopts the GPU's outcome and both continue from it,
so every round of a chain is compared.
"""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_head_gb300 import build
from speculative_decoding_head_gb300.binding import Workspace
from speculative_decoding_head_gb300.workloads import WORKLOADS, Workload, make_inputs, pack_rows

from parity import (PLAN_CUT_TOL_OWN_INPUT, PLAN_THETA_TOL_OWN_INPUT, PLAN_THETA_TOL_SAME_INPUT, Tally,
                    _record, check_draft, compare_verify, gpu_np, np_inputs, oracle_plan, pack_np, row_off_np,
                    run_gpu_round, to_device)

pytestmark = pytest.mark.gpu

MID = {
    "tiny": WORKLOADS["tiny"],
    "mid_ragged": Workload("mid_ragged", B=16, gamma=5, V=4104, r=256, H=128, wdtype="bf16", mode="compact",
                           seed=11, u_std=2.0, w_std=0.05, temp_range=(0.8, 1.5), sps_knee=48.0),
    "mid_static_f32": Workload("mid_static_f32", B=8, gamma=4, V=3000, r=32, H=40, wdtype="f32",
                               mode="static", seed=12, u_std=2.0, w_std=0.1),
    "mid_b200": Workload("mid_b200", B=200, gamma=3, V=2048, r=128, H=64, wdtype="bf16", mode="compact",
                         seed=13, u_std=2.0, w_std=0.05, sps_knee=256.0),
    "mid_lagged": Workload("mid_lagged", B=40, gamma=4, V=1536, r=64, H=32, wdtype="bf16", mode="lagged",
                           seed=14, u_std=2.0, w_std=0.05, sps_knee=32.0, noise="per_request",
                           noise_args=(0.1, 0.5, 1.0), lag=2, rounds=5),
    "mid_oddV": Workload("mid_oddV", B=6, gamma=3, V=1001, r=16, H=24, wdtype="f32", mode="compact",
                         seed=15, u_std=2.0, w_std=0.1, sps_knee=8.0),
    "small": WORKLOADS["small"],
    # static rounds with more verified rows than two CTAs per SM can hold
    # partials for (256 x 8 rows): the bulk sweep runs one CTA per SM
    "mid_static_many_rows": Workload("mid_static_many_rows", B=256, gamma=7, V=2048, r=64, H=16, wdtype="bf16",
                                     mode="static", seed=16, u_std=2.0, w_std=0.05),
    # 129 blocks a row: the dynamic sweep, whose 128-block chunks and
    # 32-block groups then never line up with the rows
    "mid_dyn": Workload("mid_dyn", B=24, gamma=4, V=8256, r=128, H=64, wdtype="bf16", mode="compact",
                        seed=17, u_std=2.0, w_std=0.05, sps_knee=24.0),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def chained_rounds(wl, rounds=None):
    """Draft -> plan -> verify on both sides for ``rounds`` chained rounds of
    every request. Each round starts from the previous round's next anchors;
    the lagged planner's ring carries confidences across rounds on both
    sides. Returns (tally, rounds compared, plans compared, plans flagged)."""
    rounds = wl.rounds if rounds is None else rounds
    inp = make_inputs(wl)
    dev, npi = to_device(inp), np_inputs(inp)
    ws = Workspace.for_workload(wl)
    tally = Tally()
    plan_checked = plan_flagged = done = 0
    anchor = npi["anchor"].copy()
    confs = []
    for rnd in range(rounds):
        g = run_gpu_round(ws, dev, wl.seed, rnd, torch.from_numpy(anchor).cuda())

        def draft_fn(rq, force, anchor=anchor, rnd=rnd):
            return oracle.draft(npi["U"], npi["W1"], npi["W2"], anchor, npi["h"], npi["w"], npi["T"], wl.seed, rnd,
                                reqs=rq, force=force)

        t, od = check_draft(g, draft_fn, range(wl.B))
        tally = tally.add(t)
        conf32 = od["conf"].astype(np.float32)
        lag_conf = confs[rnd - wl.lag] if (wl.mode == "lagged" and rnd >= wl.lag) else None
        oL, pm = oracle_plan(wl, conf32, npi["sps"], lag_conf)
        if lag_conf is not None and pm.theta < PLAN_THETA_TOL_OWN_INPUT:
            # The lagged capacity K = argmax Theta_m sits on a flat top: its
            # best and runner-up Theta differ by less than the confidences'
            # fp32 differences can move them. The GPU's K (its admitted
            # count) must lie on that top; the oracle then adopts it and the
            # top-K selection on the current confidences is compared exactly.
            K_gpu = int((g["lengths"] - 1).sum())
            th = oracle.plan_theta_path(lag_conf, npi["sps"])
            assert th[K_gpu] >= th.max() * (1 - PLAN_THETA_TOL_OWN_INPUT), (rnd, K_gpu, int(th.argmax()))
            oL, cut = oracle.plan_topk(conf32, K_gpu)
            pm = oracle.PlanMargin(np.inf, cut)
        if pm.flagged(PLAN_THETA_TOL_OWN_INPUT, PLAN_CUT_TOL_OWN_INPUT):
            plan_flagged += 1
            L = g["lengths"]          # teacher forcing: the oracle adopts the GPU's lengths
        else:
            assert (g["lengths"] == oL).all(), (rnd, g["lengths"], oL, pm)
            plan_checked += 1
            L = oL
        assert (g["row_off"] == row_off_np(L)).all()
        _record("plan", 1, int(pm.flagged(PLAN_THETA_TOL_OWN_INPUT, PLAN_CUT_TOL_OWN_INPUT)))
        ov = oracle.verify(pack_np(npi["P_full"], L), row_off_np(L), L, anchor, od["tokens"], npi["U"], npi["W1"],
                           npi["W2"], wl.seed, rnd)
        tally = tally.add(compare_verify(g, ov, range(wl.B)))
        confs.append(conf32)
        # both sides continue from the GPU's next anchors, which are the
        # oracle's wherever its verify decisions were not flagged
        anchor = g["next_anchor"].astype(np.int32)
        done += 1
    tally.check_rate()
    assert tally.compared > 0
    return tally, done, plan_checked, plan_flagged


@pytest.mark.parametrize("name", list(MID))
def test_round_parity(name):
    """End to end: each side drafts, plans and verifies on its own outputs,
    every round of the chain compared (for mid_lagged, rounds t >= lag use
    the lagged capacity)."""
    wl = MID[name]
    _, done, checked, flagged = chained_rounds(wl)
    assert done == wl.rounds
    if wl.mode == "lagged":
        assert done >= wl.lag + 2
    assert checked + flagged == wl.rounds and checked >= wl.rounds - 1


@pytest.mark.parametrize("name,rounds", [("prod", 1), ("long", 1), ("loaded", 4)])
def test_full_size_rounds_in_own_mode(name, rounds):
    """The benchmark workloads at full size in their own planner modes, every
    request: prod compact (the planner on the head's own confidences, the
    ragged verify packed by the GPU's lengths), long static (16 verify rows),
    loaded lagged over four chained rounds (rounds 2 and 3 use the capacity
    of the confidences two rounds back), with per-request target noise."""
    wl = WORKLOADS[name]
    _, done, checked, flagged = chained_rounds(wl, rounds)
    assert done == rounds and checked >= rounds - 1


def _rand_conf(B, g, seed):
    rng = np.random.default_rng(seed)
    return (1.0 / (1.0 + np.exp(-rng.normal(0, 3.6, (B, g))))).astype(np.float32)


@pytest.mark.parametrize("name", ["prod", "loaded", "long", "tiny"])
def test_plan_parity_full_size(name):
    wl = WORKLOADS[name]
    sps = make_inputs(wl.with_(V=8, r=1, H=0), with_target=False)["sps"]   # sps depends on B, gamma only
    mode = "compact" if wl.mode == "static" else wl.mode
    wl = wl.with_(mode=mode)
    ws = Workspace(wl.B, wl.gamma, 64, 1, 0, "f32", mode, wl.lag or 2)
    sps_d = sps.cuda()
    confs = []
    flagged = 0
    for t in range(6 if mode == "lagged" else 3):
        c = _rand_conf(wl.B, wl.gamma, 1000 * wl.seed + t)
        confs.append(c)
        out = ws.plan(torch.from_numpy(c).cuda(), sps_d)
        torch.cuda.synchronize()
        assert ws.device_status() == 0
        lag = confs[t - wl.lag] if (mode == "lagged" and t >= wl.lag) else None
        oL, pm = oracle_plan(wl, c, sps.numpy(), lag)
        if pm.flagged(PLAN_THETA_TOL_SAME_INPUT, 0.0):
            flagged += 1
            continue
        assert (out["lengths"].cpu().numpy() == oL).all()
        assert (out["row_off"].cpu().numpy() == row_off_np(oL)).all()
    assert flagged <= 1


def test_plan_static_and_flat():
    ws = Workspace(5, 3, 64, 1, 0, "f32", "static")
    out = ws.plan(torch.zeros((5, 3), device="cuda"), torch.ones(1 + 5 * 4, dtype=torch.float64, device="cuda"))
    torch.cuda.synchronize()
    assert (out["lengths"].cpu() == 4).all() and out["row_off"].cpu().tolist() == [0, 4, 8, 12, 16, 20]
    ws = Workspace(5, 3, 64, 1, 0, "f32", "compact")
    c = torch.from_numpy(_rand_conf(5, 3, 1)).cuda()
    out = ws.plan(c, torch.full((21,), 400.0, dtype=torch.float64, device="cuda"))
    torch.cuda.synchronize()
    assert (out["lengths"].cpu() == 4).all()   # flat SPS table: full verify


@pytest.mark.parametrize("V", [4104, 8192], ids=["register_sweep", "dynamic_sweep"])
def test_verify_stagewise_on_oracle_drafts(V):
    """Both sides verify the oracle's drafts (rounded to fp32) under many length
    patterns: V % 64 != 0 takes the register sweep, 128 blocks a row (the
    smallest row the dynamic sweep takes) the dynamic sweep."""
    wl = MID["mid_ragged"].with_(B=48, V=V, seed=21)
    inp = make_inputs(wl)
    dev, npi = to_device(inp), np_inputs(inp)
    od = oracle.draft(npi["U"], npi["W1"], npi["W2"], npi["anchor"], npi["h"], npi["w"], npi["T"], 5, 9)
    ws = Workspace.for_workload(wl)
    rng = np.random.default_rng(3)
    tally = Tally()
    for trial in range(3):
        L = rng.integers(1, wl.gamma + 2, wl.B).astype(np.int32)
        ro = row_off_np(L)
        P = pack_np(npi["P_full"], L)
        out = ws.verify(torch.from_numpy(P).cuda(), torch.from_numpy(ro).cuda(), torch.from_numpy(L).cuda(),
                        dev["anchor"], torch.from_numpy(od["tokens"]).cuda(),
                        torch.from_numpy(od["pd_tok"].astype(np.float32)).cuda(),
                        torch.from_numpy(od["lse"].astype(np.float32)).cuda(), dev["U"], dev["W1"], dev["W2"],
                        5, 9 + trial)
        torch.cuda.synchronize()
        assert ws.device_status() == 0
        ov = oracle.verify(P, ro, L, npi["anchor"], od["tokens"], npi["U"], npi["W1"], npi["W2"], 5, 9 + trial)
        tally = tally.add(compare_verify(gpu_np(out), ov, range(wl.B)))
        assert (out["n_acc"].cpu().numpy() <= L - 1).all()
    tally.check_rate()
    assert tally.compared > 0


def test_determinism_and_launch_accounting():
    wl = MID["mid_b200"]
    dev = to_device(make_inputs(wl))
    ws = Workspace.for_workload(wl)
    a = run_gpu_round(ws, dev, 77, 5)
    b = run_gpu_round(ws, dev, 77, 5)
    for k in a:
        assert (a[k] == b[k]).all(), k
    c = run_gpu_round(ws, dev, 77, 6)
    assert not (a["tokens"] == c["tokens"]).all()   # another round draws other numbers
    assert ws.last_launches > 0


def test_device_errors_are_reported_not_faulted():
    wl = MID["tiny"]
    dev = to_device(make_inputs(wl))
    ws = Workspace.for_workload(wl)
    bad = dev["anchor"].clone()
    bad[1] = wl.V + 5                                  # out-of-range token id
    ws.draft(dev["U"], dev["W1"], dev["W2"], bad, dev["h"], dev["w"], dev["T"], 1, 0)
    torch.cuda.synchronize()
    assert ws.device_status() == 6
    ws.reset()
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    conf = torch.full((wl.B, wl.gamma), float("nan"), device="cuda")
    ws.plan(conf, dev["sps"])
    torch.cuda.synchronize()
    assert ws.device_status() == 4
    ws.reset()
    with pytest.raises(Exception):
        ws.plan(conf.cpu(), dev["sps"])               # host tensors are refused by the binding


@pytest.mark.parametrize("V", [4096, 16384], ids=["bulk", "dynamic"])
def test_verify_rejects_inconsistent_lengths(V):
    """Lengths outside [1, gamma + 1] or offsets that do not add up are reported
    as ERANGE, not faulted: by the bulk sweep (V % 64 == 0, 64 blocks a row)
    and by the dynamic sweep's finalize (256 blocks a row), which also leaves
    its chunk counter ready for the next call."""
    wl = MID["mid_ragged"].with_(B=16, V=V, seed=23)
    assert wl.V % 64 == 0
    inp = make_inputs(wl)
    dev, npi = to_device(inp), np_inputs(inp)
    od = oracle.draft(npi["U"], npi["W1"], npi["W2"], npi["anchor"], npi["h"], npi["w"], npi["T"], 5, 1)
    ws = Workspace.for_workload(wl)
    L = np.full(wl.B, 2, np.int32)
    P = pack_np(npi["P_full"], L)
    args = (torch.from_numpy(od["tokens"]).cuda(), torch.from_numpy(od["pd_tok"].astype(np.float32)).cuda(),
            torch.from_numpy(od["lse"].astype(np.float32)).cuda(), dev["U"], dev["W1"], dev["W2"], 5, 1)
    for bad_L, bad_ro in ((L.copy(), None), (L.copy(), "shift")):
        if bad_ro is None:
            bad_L[3] = 0                                   # a request with no verified row
        ro = row_off_np(bad_L)
        if bad_ro == "shift":
            ro[5] += 1                                     # offsets that do not add up
        out = ws.verify(torch.from_numpy(P).cuda(), torch.from_numpy(ro).cuda(), torch.from_numpy(bad_L).cuda(),
                        dev["anchor"], *args)
        torch.cuda.synchronize()
        assert ws.device_status() == 6, ws.device_status()
        ws.reset()
        torch.cuda.synchronize()
        assert ws.device_status() == 0
    # the workspace is usable again after the reset
    ro = row_off_np(L)
    out = ws.verify(torch.from_numpy(P).cuda(), torch.from_numpy(ro).cuda(), torch.from_numpy(L).cuda(),
                    dev["anchor"], *args)
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    ov = oracle.verify(P, ro, L, npi["anchor"], od["tokens"], npi["U"], npi["W1"], npi["W2"], 5, 1)
    compare_verify(gpu_np(out), ov, range(wl.B)).check_rate()


def test_gpu_losslessness_chi_square():
    """Replicated requests with token-independent rows: the first emitted token follows p_t."""
    from scipy import stats
    V, B = 100, 4096
    rng = np.random.default_rng(5)
    pt = rng.dirichlet(np.full(V, 0.5))
    pd = rng.dirichlet(np.full(V, 0.5))
    U = torch.from_numpy(np.broadcast_to(np.log(pd), (B, 1, V)).astype(np.float32).copy()).cuda()
    W1 = torch.zeros((V, 8), device="cuda")
    W2 = torch.zeros((8, V), device="cuda")
    anchor = torch.zeros(B, dtype=torch.int32, device="cuda")
    P = torch.from_numpy(np.broadcast_to(np.log(pt), (2 * B, V)).astype(np.float32).copy()).cuda()
    L = torch.full((B,), 2, dtype=torch.int32, device="cuda")
    ro = torch.arange(0, 2 * B + 1, 2, dtype=torch.int32, device="cuda")
    ws = Workspace(B, 1, V, 8, 0, "f32", "static")
    counts = np.zeros(V)
    acc = 0
    rounds = 12
    for rnd in range(rounds):
        d = ws.draft(U, W1, W2, anchor, None, torch.zeros(8, device="cuda"), torch.ones(1, device="cuda"), 9, rnd)
        v = ws.verify(P, ro, L, anchor, d["tokens"], d["pd_tok"], d["lse"], U, W1, W2, 9, rnd)
        torch.cuda.synchronize()
        n = v["n_acc"].cpu().numpy()
        tok = np.where(n > 0, d["tokens"].cpu().numpy()[:, 0], v["next_anchor"].cpu().numpy())
        counts += np.bincount(tok, minlength=V)
        acc += int(n.sum())
    N = rounds * B
    beta = np.minimum(pt, pd).sum()
    assert abs(acc / N - beta) < 5 * np.sqrt(beta * (1 - beta) / N)
    keep = pt > 0
    assert stats.chisquare(counts[keep], pt[keep] / pt[keep].sum() * N).pvalue > 1e-4
