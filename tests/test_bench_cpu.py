"""bench.py's reference arm (the oracle timed on host cores) and its JSON
contract, on CPU with the tiny workload and a short time budget."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2",
                        "--warmup", "1", "--cpu-seconds", "1"], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"].startswith("tiny")


def test_secondary_oracle_samples_run_on_cpu():
    """The oracle legs that sit beside the training-objective and RNN-draft
    timings (bench.py's cpu_baseline entries), on a small shape."""
    import sys as _s
    _s.path.insert(0, ROOT)
    import bench
    from speculative_decoding_head_gb300.workloads import WORKLOADS, make_inputs, make_loss_inputs, make_rnn_weights
    wl = WORKLOADS["small"].with_(B=4, gamma=3, V=1024, r=64, H=32)
    c = bench.oracle_loss_sample(wl, make_loss_inputs(wl), 0.2)
    assert c["value"] > 0 and c["kind"] == "oracle" and c["unit"] == "calls/s" and c["cores"] >= 1
    c = bench.oracle_rnn_sample(wl, make_inputs(wl, with_target=False), make_rnn_weights(wl), 0.2)
    assert c["value"] > 0 and c["kind"] == "oracle" and "RNN" in c["sample"]


def test_sts_oracle_sample_runs_on_cpu():
    import sys as _s
    _s.path.insert(0, ROOT)
    import bench
    from speculative_decoding_head_gb300.workloads import make_sts_inputs, sts_grid
    c = bench.oracle_sts_sample(make_sts_inputs(5000, 3, 1), sts_grid(8), 15, 0.1)
    assert c["value"] > 0 and c["unit"] == "fits/s" and c["kind"] == "oracle"
    assert bench.oracle_sts_sample(make_sts_inputs(100, 2, 1), sts_grid(4), 15, 0.0) is None


def test_round_parity_report_counts():
    """bench.py's oracle_parity entry: outputs equal to the oracle's give no
    mismatch; a changed draft token ends that request's draft comparison and
    drops it from the verify comparison; a changed next anchor counts once."""
    import sys as _s
    _s.path.insert(0, ROOT)
    import numpy as np
    import bench
    import oracle
    from speculative_decoding_head_gb300.workloads import WORKLOADS, make_inputs
    wl = WORKLOADS["small"].with_(B=6, V=4096, H=64)
    npi = bench._np_inputs(make_inputs(wl))
    od = oracle.draft(npi["U"], npi["W1"], npi["W2"], npi["anchor"], npi["h"], npi["w"], npi["T"], wl.seed, 0)
    L = bench.oracle_plan_lengths(wl, npi, wl.seed, 0, od)
    ro = np.zeros(wl.B + 1, np.int32)
    ro[1:] = np.cumsum(L)
    P = np.concatenate([npi["P_full"][b, :L[b]] for b in range(wl.B)]).reshape(-1, wl.V)
    ov = oracle.verify(P, ro, L, npi["anchor"], od["tokens"], npi["U"], npi["W1"], npi["W2"], wl.seed, 0)
    out = {"tokens": od["tokens"].copy(), "lengths": L, "n_acc": ov["n_acc"].copy(),
           "next_anchor": ov["next_anchor"].copy()}
    r = bench.oracle_round_parity(wl, npi, od, out, wl.seed, 0)
    assert r["draft"]["mismatched"] == 0 and r["draft"]["draws_compared"] + r["draft"]["flagged"] == wl.B * wl.gamma
    assert r["plan"]["lengths_equal"] and r["verify"]["mismatched"] == 0
    assert r["verify"]["requests_compared"] + r["verify"]["flagged"] == wl.B
    out["tokens"][0, 1] = (out["tokens"][0, 1] + 1) % wl.V
    out["next_anchor"][1] = (out["next_anchor"][1] + 1) % wl.V
    r = bench.oracle_round_parity(wl, npi, od, out, wl.seed, 0)
    assert r["draft"]["mismatched"] + r["draft"]["flagged"] >= 1
    assert r["draft"]["draws_compared"] + r["draft"]["flagged"] == wl.B * wl.gamma - (wl.gamma - 2)
    assert r["verify"]["requests_skipped_draft_differs"] == 1
    assert r["verify"]["mismatched"] + r["verify"]["flagged"] >= 1
