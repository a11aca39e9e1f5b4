"""A batch split by request, run as two shards on one GPU, against the unsplit batch.

Each shard has a workspace for its own requests (the draws keyed by batch
index through dspark_ws_set_shard) and plans the whole batch from the
concatenated confidences with dspark_plan_shard, which keeps its range of
lengths and row offsets. On a machine with several GPUs each shard runs in
its own process and the concatenation is an all-gather; here the shards run
one after the other on one GPU and the test concatenates (no kernel of one
shard waits on the other's). Over three chained rounds the shards must
return what one workspace returns for the whole batch: the same draft
tokens and confidences, the same lengths, the same accepted counts and next
anchors. The verify of a shard sums its target rows in a different launch
shape from the unsplit batch, so an accept test or a residual draw may fall
the other way where the fp64 oracle calls it too close to take in fp32;
only such requests may differ.
"""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_head_gb300.binding import Workspace
from speculative_decoding_head_gb300.shard import ShardedRound, shard_range
from speculative_decoding_head_gb300.workloads import WORKLOADS, make_inputs, pack_rows

from parity import np_inputs

pytestmark = pytest.mark.gpu

# 41 requests: shares of 21 and 20, the second starting at an index that is
# not a multiple of 4; the knee of the SPS table makes the planner cut
CASES = [
    ("compact_tc", WORKLOADS["prod"].with_(B=41, V=8192, H=256, sps_knee=24.0, mode="compact"), "tcgen05"),
    ("lagged_simt", WORKLOADS["prod"].with_(B=41, V=8192, H=256, sps_knee=24.0, mode="lagged", lag=2, seed=12),
     "simt"),
    ("three_way_static", WORKLOADS["small"].with_(B=10, V=4096, H=64), "tcgen05"),
]


@pytest.mark.parametrize("name,wl,path", CASES, ids=[c[0] for c in CASES])
def test_split_batch_rounds_match_the_unsplit_batch(name, wl, path):
    world = 3 if name.startswith("three") else 2
    inp = make_inputs(wl)
    npi = np_inputs(inp)
    dev = {k: v.cuda().contiguous() for k, v in inp.items()}
    whole = Workspace.for_workload(wl, path=path)
    ranks = [ShardedRound(wl.B, wl.gamma, wl.V, wl.r, wl.H, wl.wdtype, wl.mode, wl.lag or 2, rank=i, world=world,
                          path=path) for i in range(world)]
    seed = 5
    anchor = dev["anchor"]
    cut = 0
    for rnd in range(3):
        d = whole.draft(dev["U"], dev["W1"], dev["W2"], anchor, dev["h"], dev["w"], dev["T"], seed, rnd)
        p = whole.plan(d["conf"], dev["sps"])
        P = pack_rows(dev["P_full"], p["lengths"]).contiguous()
        v = whole.verify(P, p["row_off"], p["lengths"], anchor, d["tokens"], d["pd_tok"], d["lse"], dev["U"],
                         dev["W1"], dev["W2"], seed, rnd)
        parts = []
        for sr in ranks:
            b0, n = sr.b_begin, sr.b_count
            assert (b0, n) == shard_range(wl.B, sr.rank, world)
            sl = slice(b0, b0 + n)
            # each rank holds its own copies (16-byte aligned, as the library requires)
            ds = sr.draft(dev["U"][sl].clone(), dev["W1"], dev["W2"], anchor[sl].clone(), dev["h"][sl].clone(),
                          dev["w"], dev["T"], seed, rnd)
            parts.append((sr, sl, ds))
        conf_all = torch.cat([ds["conf"] for _, _, ds in parts]).contiguous()
        torch.cuda.synchronize()
        g = {k: v_.cpu().numpy() for k, v_ in d.items()}
        for sr, sl, ds in parts:
            assert sr.local.device_status() == 0
            assert (ds["tokens"].cpu().numpy() == g["tokens"][sl]).all(), (name, rnd, sr.rank)
            assert (ds["conf"].cpu().numpy() == g["conf"][sl]).all()
            for k in ("pd_tok", "lse"):
                np.testing.assert_allclose(ds[k].cpu().numpy(), g[k][sl], rtol=1e-6)
        L_whole = p["lengths"].cpu().numpy()
        got_L, got_n, got_a = [], [], []
        for sr, sl, ds in parts:
            ps = sr.planner.plan_shard(conf_all, dev["sps"], sr.b_begin, sr.b_count)
            Ls = ps["lengths_local"]
            assert (ps["lengths"].cpu().numpy() == L_whole).all()   # every rank plans the whole batch
            ro = ps["row_off_local"].cpu().numpy()
            assert ro[0] == 0 and (np.diff(ro) == Ls.cpu().numpy()).all()
            Ps = pack_rows(dev["P_full"][sl], Ls).contiguous()
            vs = sr.verify(Ps, ps["row_off_local"], Ls, anchor[sl].clone(), ds["tokens"], ds["pd_tok"], ds["lse"],
                           dev["U"][sl].clone(), dev["W1"], dev["W2"], seed, rnd)
            torch.cuda.synchronize()
            assert sr.local.device_status() == 0 and sr.planner.device_status() == 0
            got_L += Ls.cpu().tolist()
            got_n += vs["n_acc"].cpu().tolist()
            got_a += vs["next_anchor"].cpu().tolist()
        assert got_L == L_whole.tolist(), (name, rnd)
        cut += int((L_whole < wl.gamma + 1).sum())
        n_w, a_w = v["n_acc"].cpu().numpy(), v["next_anchor"].cpu().numpy()
        diff = [b for b in range(wl.B) if got_n[b] != n_w[b] or got_a[b] != a_w[b]]
        if diff:
            ro = np.zeros(wl.B + 1, np.int32)
            ro[1:] = np.cumsum(L_whole)
            oP = np.concatenate([npi["P_full"][b, :L_whole[b]] for b in range(wl.B)])
            o = oracle.verify(oP, ro, L_whole, anchor.cpu().numpy(), g["tokens"], npi["U"], npi["W1"], npi["W2"],
                              seed, rnd, reqs=diff)
            for b in diff:
                assert min(o["acc_margin"][b], o["smp_margin"][b]) < oracle.MARGIN, (name, rnd, b)
        anchor = v["next_anchor"].contiguous()
    if wl.mode != "static":
        assert cut > 0   # the planner shortened some requests
    for sr in ranks:
        sr.close()
