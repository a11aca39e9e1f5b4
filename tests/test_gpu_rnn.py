"""The RNN head's draft tail (eq. (6)) on the GPU against the oracle.

Tokens are bit-exact except at positions the oracle flags (the same margins
as the Markov draft), where it adopts the GPU's token and continues (teacher
forcing); pd_tok, lse and conf within 1e-4 relative; the head vector o_k
within 2e-5 absolute (|o| < 1; its pre-activations are fp32 sums of 2r + H
terms) at every position.
"""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_head_gb300 import build
from speculative_decoding_head_gb300.binding import Workspace
from speculative_decoding_head_gb300.workloads import WORKLOADS, Workload, make_inputs, make_rnn_weights

from parity import check_draft, gpu_np, np_inputs, to_device

pytestmark = pytest.mark.gpu

OVEC_ATOL = 2e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _run(wl, rnd=0, reqs=None, path=None):
    inp = make_inputs(wl, with_target=False)
    inp["Wr"] = make_rnn_weights(wl)
    dev, npi = to_device(inp), np_inputs(inp)
    ws = Workspace.for_workload(wl, path=path)
    out = ws.rnn_draft(dev["U"], dev["W1"], dev["W2"], dev["Wr"], dev["anchor"], dev["h"], dev["w"], dev["T"],
                       wl.seed, rnd)
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    # hidden halves and the h projection (on tcgen05: the hi | lo split, then the GEMM), three per step
    tc_hproj = (ws.path == "tcgen05" and wl.wdtype == "bf16" and wl.H >= 64 and wl.H % 64 == 0 and wl.r % 64 == 0
                and wl.r <= 256)
    assert ws.last_launches == (3 if tc_hproj else 2 if wl.H > 0 else 0) + 3 * wl.gamma
    g = gpu_np({k: v for k, v in out.items() if k != "scratch"})
    reqs = list(range(wl.B)) if reqs is None else list(reqs)

    def draft_fn(rq, force):
        return oracle.rnn_draft(npi["U"], npi["W1"], npi["W2"], npi["Wr"], npi["anchor"], npi["h"], npi["w"],
                                npi["T"], wl.seed, rnd, reqs=rq, force=force)

    t, o = check_draft(g, draft_fn, reqs)
    t.check_rate()
    for b in reqs:
        d = np.abs(g["ovec"][b] - o["ovec"][b]).max()
        assert d <= OVEC_ATOL, (b, d)
    return g, o, t


def _wl(name, B, gamma, V, r, H, wdtype="bf16", seed=41):
    return Workload(name, B=B, gamma=gamma, V=V, r=r, H=H, wdtype=wdtype, mode="static", seed=seed, u_std=2.0,
                    w_std=0.05 if wdtype == "bf16" else 0.3)


@pytest.mark.parametrize("wl", [
    _wl("rnn_tiny", 2, 3, 1024, 16, 64, wdtype="f32"),
    _wl("rnn_small", 6, 4, 4104, 64, 96),            # a vocabulary ending inside a 64-token block
    _wl("rnn_noh", 5, 6, 2048, 32, 0, wdtype="f32"),  # no hidden states: z = [s; W1[x]]
    _wl("rnn_mid", 40, 5, 32000, 256, 1024),
    # the h projection on tcgen05 (H % 64 == 0): 3r in 192-wide tiles, K' = 2H
    # in fewer blocks than the ten slices (the rest write zeros), a partial
    # last 128-row tile
    _wl("rnn_tc_r128", 12, 3, 4104, 128, 128),
    _wl("rnn_tc_r64", 9, 4, 2048, 64, 192),
    # two row groups in the row pass (o_k's images per group of 128
    # requests; the second group's rows past B stay zero)
    _wl("rnn_two_groups", 160, 3, 8192, 64, 64),
], ids=lambda w: w.name)
def test_rnn_draft_parity(wl):
    _run(wl, rnd=1)


def test_rnn_h_projection_paths_agree():
    """The tcgen05 h projection (h as bf16 hi + lo, about 17 significant bits)
    against the CUDA-core one (fp32), through the whole RNN draft. o_1 depends
    on the projection and the anchor only; later steps also on the drawn
    tokens, so they are compared on the requests whose tokens agree. The
    bound: per product a relative error below 2^-18 of h, summed over H = 512
    terms with weights of std 1/32, is about 1.5e-6 rms; 2e-5 holds it at more
    than 10 sigma."""
    wl = _wl("rnn_hproj_paths", 24, 5, 8192, 256, 512, seed=47)
    inp = make_inputs(wl, with_target=False)
    dev = {k: v.cuda().contiguous() for k, v in inp.items()}
    Wr = make_rnn_weights(wl).cuda()
    outs = []
    for path in ("tcgen05", "simt"):
        ws = Workspace.for_workload(wl, path=path)
        o = ws.rnn_draft(dev["U"], dev["W1"], dev["W2"], Wr, dev["anchor"], dev["h"], dev["w"], dev["T"], 5, 1)
        torch.cuda.synchronize()
        assert ws.device_status() == 0
        outs.append({k: v.cpu().numpy() for k, v in o.items()})
    assert np.abs(outs[0]["ovec"][:, 0] - outs[1]["ovec"][:, 0]).max() < 2e-5
    same = (outs[0]["tokens"] == outs[1]["tokens"]).all(axis=1)
    assert same.sum() >= wl.B - 1  # the two block passes round differently: a flip is rare
    assert np.abs(outs[0]["ovec"][same] - outs[1]["ovec"][same]).max() < 2e-5


def test_rnn_draft_simt_block_pass():
    """The SIMT block pass (the fallback for shapes tcgen05 does not take) on
    a bf16 shape the tcgen05 pass also takes."""
    _run(_wl("rnn_small_simt", 6, 4, 4104, 64, 96), rnd=2, path="simt")


def test_rnn_draft_full_size():
    """The prod shape (B=128, gamma=5, V=129280, r=256, H=5120), every request."""
    _run(WORKLOADS["prod"], rnd=3)


def test_rnn_head_differs_from_markov_head():
    """Same inputs: the RNN head's tokens follow its own bias, not W1[x] W2."""
    wl = _wl("rnn_vs_markov", 8, 5, 4096, 64, 32)
    g, o, _ = _run(wl)
    inp = make_inputs(wl, with_target=False)
    npi = np_inputs(inp)
    m = oracle.draft(npi["U"], npi["W1"], npi["W2"], npi["anchor"], npi["h"], npi["w"], npi["T"], wl.seed, 0)
    assert not np.allclose(m["lse"], o["lse"])


@pytest.mark.parametrize("path", ["tcgen05", "simt"])
def test_rnn_verify_stagewise_on_oracle_drafts(path):
    """Both sides verify the oracle's RNN-head drafts: p_d of a rejected
    position from U + o W2 (the oracle's o_k, rounded to fp32 for the GPU),
    under several length patterns; most requests take a residual draw. The
    residual block pass runs on tcgen05 (o as bf16 hi + lo operands; the
    vocabulary ends 8 entries into its last tile) or on CUDA cores."""
    from parity import Tally, compare_verify, pack_np, row_off_np
    wl = _wl("rnn_verify", 24, 4, 4104, 64, 96, seed=43)
    inp = make_inputs(wl)
    inp["Wr"] = make_rnn_weights(wl)
    dev, npi = to_device(inp), np_inputs(inp)
    od = oracle.rnn_draft(npi["U"], npi["W1"], npi["W2"], npi["Wr"], npi["anchor"], npi["h"], npi["w"], npi["T"],
                          6, 4)
    ws = Workspace.for_workload(wl)
    ws.set_path(path)
    rng = np.random.default_rng(8)
    tally = Tally()
    resid = 0
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a).astype(np.float32)).cuda()
    for trial in range(3):
        L = rng.integers(1, wl.gamma + 2, wl.B).astype(np.int32)
        ro = row_off_np(L)
        P = pack_np(npi["P_full"], L)
        out = ws.verify_rnn(torch.from_numpy(P).cuda(), torch.from_numpy(ro).cuda(), torch.from_numpy(L).cuda(),
                            dev["anchor"], torch.from_numpy(od["tokens"]).cuda(), f32(od["pd_tok"]), f32(od["lse"]),
                            dev["U"], f32(od["ovec"]), dev["W2"], 6, 10 + trial)
        torch.cuda.synchronize()
        assert ws.device_status() == 0
        ov = oracle.verify(P, ro, L, npi["anchor"], od["tokens"], npi["U"], npi["W1"], npi["W2"], 6, 10 + trial,
                           ovec=od["ovec"])
        tally = tally.add(compare_verify(gpu_np(out), ov, range(wl.B)))
        resid += int(ov["resid"].sum())
        assert (out["n_acc"].cpu().numpy() <= L - 1).all()
    tally.check_rate()
    assert tally.compared > 0 and resid > 0


def test_rnn_verify_full_size():
    """The RNN verify at the prod shape (B=128, gamma=5, V=129280, r=256) on
    the oracle's drafts of sixteen sampled requests, each verifying two to
    gamma + 1 rows (most take a residual draw on tcgen05, whose CTAs then
    hold several requests each); the other requests verify their bonus row
    only."""
    from parity import compare_verify, pack_np, row_off_np
    wl = WORKLOADS["prod"]
    inp = make_inputs(wl)
    inp["Wr"] = make_rnn_weights(wl)
    npi = np_inputs(inp)
    reqs = [0, 1, 9, 23, 37, 42, 50, 64, 71, 88, 95, 101, 110, 117, 126, 127]
    od = oracle.rnn_draft(npi["U"], npi["W1"], npi["W2"], npi["Wr"], npi["anchor"], npi["h"], npi["w"], npi["T"],
                          7, 2, reqs=reqs)
    tokens = np.where(od["tokens"] < 0, 0, od["tokens"]).astype(np.int32)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(np.nan_to_num(a)).astype(np.float32)).cuda()
    L = np.ones(wl.B, np.int32)
    L[reqs] = np.random.default_rng(9).integers(2, wl.gamma + 2, len(reqs))
    ro = row_off_np(L)
    P = pack_np(npi["P_full"], L)
    ws = Workspace.for_workload(wl)
    assert ws.path == "tcgen05"
    out = ws.verify_rnn(torch.from_numpy(P).cuda(), torch.from_numpy(ro).cuda(), torch.from_numpy(L).cuda(),
                        inp["anchor"].cuda(), torch.from_numpy(tokens).cuda(), f32(od["pd_tok"]), f32(od["lse"]),
                        inp["U"].cuda(), f32(od["ovec"]), inp["W2"].cuda(), 7, 2)
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    ov = oracle.verify(P, ro, L, npi["anchor"], tokens, npi["U"], npi["W1"], npi["W2"], 7, 2, reqs=reqs,
                       ovec=np.nan_to_num(od["ovec"]))
    tally = compare_verify(gpu_np(out), ov, reqs)
    tally.check_rate()
    assert tally.compared > 0 and int(ov["resid"][reqs].sum()) > 0
    n = out["n_acc"].cpu().numpy()
    assert (n[L == 1] == 0).all()


def test_rnn_round_on_the_gpu_is_consistent():
    """The GPU's own RNN drafts through the planner and the RNN verify."""
    wl = _wl("rnn_round", 16, 5, 4096, 64, 32, seed=45).with_(mode="compact", sps_knee=32.0)
    inp = make_inputs(wl)
    Wr = make_rnn_weights(wl).cuda()
    dev = to_device(inp)
    ws = Workspace.for_workload(wl)
    d = ws.rnn_draft(dev["U"], dev["W1"], dev["W2"], Wr, dev["anchor"], dev["h"], dev["w"], dev["T"], 2, 0)
    p = ws.plan(d["conf"], dev["sps"])
    from speculative_decoding_head_gb300.workloads import pack_rows
    P = pack_rows(dev["P_full"], p["lengths"])
    v = ws.verify_rnn(P, p["row_off"], p["lengths"], dev["anchor"], d["tokens"], d["pd_tok"], d["lse"], dev["U"],
                      d["ovec"], dev["W2"], 2, 0)
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    L = p["lengths"].cpu().numpy()
    n = v["n_acc"].cpu().numpy()
    assert ((n >= 0) & (n <= L - 1)).all()
    na = v["next_anchor"].cpu().numpy()
    assert ((na >= 0) & (na < wl.V)).all()
