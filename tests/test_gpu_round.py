"""dspark_round (the whole round in one call, as the benchmark runs it)
against the three separate calls on the same inputs.

Inside dspark_round the planner also writes the packed-row table, the kernels
overlap their prologues with the previous kernel's tail, and the verify sweep
takes its chunks of P from a counter (the dynamic sweep, for rows of at
least 128 blocks) instead of fixed ranges. Over three chained rounds the
round must return what draft, plan and verify return: tokens, probabilities,
log-sum-exps and confidences bit-identical (the same kernels), the same
lengths and offsets, and the same accepted counts and next anchors, except
where the fp64 oracle calls an accept test or a residual draw too close to
take in fp32 (the two sweeps add a row's partials in different orders).
Both workspaces advance their own planner state (the lagged ring) in step.
"""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_head_gb300.binding import Workspace
from speculative_decoding_head_gb300.workloads import WORKLOADS, make_inputs, pack_rows

from parity import np_inputs

pytestmark = pytest.mark.gpu

CASES = [
    WORKLOADS["tiny"],                                       # 16 blocks a row: the fixed-range sweep with the row table
    WORKLOADS["small"].with_(B=20),                          # static lengths, 500 blocks a row
    WORKLOADS["prod"].with_(B=40, sps_knee=30.0),            # the compact planner at the prod vocabulary
    WORKLOADS["loaded"].with_(B=48, V=65536, sps_knee=40.0),  # the lagged planner
    WORKLOADS["long"].with_(B=16),                           # 16 rows a request
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_round_matches_separate_calls(wl):
    inp = make_inputs(wl)
    npi = np_inputs(inp)
    dev = {k: v.cuda().contiguous() for k, v in inp.items()}
    sep = Workspace.for_workload(wl)
    one = Workspace.for_workload(wl)
    seed = 11
    anchor = dev["anchor"]
    for rnd in range(3):
        d = sep.draft(dev["U"], dev["W1"], dev["W2"], anchor, dev["h"], dev["w"], dev["T"], seed, rnd)
        p = sep.plan(d["conf"], dev["sps"])
        P = pack_rows(dev["P_full"], p["lengths"]).contiguous()
        v = sep.verify(P, p["row_off"], p["lengths"], anchor, d["tokens"], d["pd_tok"], d["lse"], dev["U"],
                       dev["W1"], dev["W2"], seed, rnd)
        o = one.round(dev["U"], dev["W1"], dev["W2"], anchor, dev["h"], dev["w"], dev["T"], dev["sps"], P, seed, rnd)
        torch.cuda.synchronize()
        assert sep.device_status() == 0 and one.device_status() == 0, (sep.device_status(), one.device_status())
        for k in ("tokens", "pd_tok", "lse", "conf", "lengths", "row_off"):
            a = (d if k in d else p)[k].cpu().numpy()
            assert (o[k].cpu().numpy() == a).all(), (wl.name, rnd, k)
        n_s, a_s = v["n_acc"].cpu().numpy(), v["next_anchor"].cpu().numpy()
        n_o, a_o = o["n_acc"].cpu().numpy(), o["next_anchor"].cpu().numpy()
        diff = [b for b in range(wl.B) if n_s[b] != n_o[b] or a_s[b] != a_o[b]]
        if diff:
            L = p["lengths"].cpu().numpy()
            ro = np.zeros(wl.B + 1, np.int32)
            ro[1:] = np.cumsum(L)
            oP = np.concatenate([npi["P_full"][b, :L[b]] for b in range(wl.B)])
            ov = oracle.verify(oP, ro, L, anchor.cpu().numpy(), d["tokens"].cpu().numpy(), npi["U"], npi["W1"],
                               npi["W2"], seed, rnd, reqs=diff)
            for b in diff:
                assert min(ov["acc_margin"][b], ov["smp_margin"][b]) < oracle.MARGIN, (wl.name, rnd, b)
        anchor = v["next_anchor"].contiguous()
