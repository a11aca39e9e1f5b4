"""GPU-vs-oracle parity helpers for the tests.

Parity rule: token ids, lengths, accepted counts and next anchors must be
bit-exact, except at decisions the fp64 oracle calls too close to take in
fp32 (margin < oracle.MARGIN); such "flagged" decisions are counted and must
stay below 1e-4 of the decisions compared. At a flagged position whose
outcome differs, the oracle adopts the GPU's choice and continues from it
(teacher forcing), so one flag does not end the comparison of a request or a
chained round. Draft probabilities, log-sum-exps and confidences must agree
within 1e-4 relative.

Expected flag rates. Every sample of the library is a two-level Gumbel-max
(block, then token inside the block); a level's decision is flagged when its
top two keys lie within MARGIN, which happens with probability about MARGIN
per level (the gap has density near 1 at zero: for 64 equal weights the law
is P(gap > t) = 64 / (1 + 63 e^t)), so about 2e-5 per draw. Accept tests are
flagged within MARGIN of the ratio, about 1e-5 per test. Each test allows
1e-4 of its decisions plus one stray flag (a sample of a few hundred draws
shows one flag in about 1% of runs); the session's totals are printed at the
end of the run.
"""

from __future__ import annotations

import dataclasses
import os
from typing import Dict, Optional, Sequence

import numpy as np
import torch

import oracle
from speculative_decoding_head_gb300 import workloads as wlmod

RTOL = 1e-4
# Planner flags. With identical fp32 confidences both sides form the same fp64
# survival products and sort order; only the prefix sums differ (the GPU sums
# them in 2^-50 fixed point: absolute error below M * 2^-51 < 4e-12 for
# M <= 8192, against tau >= 1), so a decision is flagged only when its
# relative Theta gap is below 1e-11.
PLAN_THETA_TOL_SAME_INPUT = 1e-11
# When each side computes its own confidences (fp32 on the GPU, fp64 rounded to
# fp32 in the oracle) they differ by ~1e-6 relative, survival products by up
# to gamma times that; decisions and the order across the cut are flagged
# below 1e-5 relative.
PLAN_THETA_TOL_OWN_INPUT = 1e-5
PLAN_CUT_TOL_OWN_INPUT = 1e-5


DRAFT_FLAG_RATE = 1e-4     # per draft draw (two Gumbel-max levels)
VERIFY_FLAG_RATE = 1e-4    # per verify decision (Gumbel keys, accept ratios)

# per test: (kind, compared, flagged), collected for the end-of-run summary
SESSION = []


def _record(kind: str, compared: int, flagged: int) -> None:
    name = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    SESSION.append((name, kind, compared, flagged))


@dataclasses.dataclass
class Tally:
    compared: int = 0
    flagged: int = 0
    excluded_requests: int = 0
    budget: float = 0.0    # flags allowed by the rates above
    slack: int = 1         # stray flags allowed on small samples

    def add(self, other: "Tally") -> "Tally":
        return Tally(self.compared + other.compared, self.flagged + other.flagged,
                     self.excluded_requests + other.excluded_requests, self.budget + other.budget,
                     max(self.slack, other.slack))

    def check_rate(self) -> None:
        assert self.flagged <= self.slack + int(self.budget), self


def np_inputs(inp: Dict[str, torch.Tensor]) -> Dict[str, np.ndarray]:
    out = {}
    for k, v in inp.items():
        if v.dtype == torch.bfloat16:
            out[k] = v.contiguous().view(torch.int16).cpu().numpy()
        else:
            out[k] = v.cpu().numpy()
    return out


def to_device(inp: Dict[str, torch.Tensor], device="cuda") -> Dict[str, torch.Tensor]:
    return {k: v.to(device).contiguous() for k, v in inp.items()}


def rel_close(a, b, rtol=RTOL) -> np.ndarray:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.abs(a - b) <= rtol * np.abs(b) + 1e-30


def compare_draft(g: Dict[str, np.ndarray], o: Dict[str, np.ndarray], reqs: Sequence[int]):
    """Compare draft outputs of the listed requests, position by position.

    ``o`` should come from ``forced_draft`` (the oracle already adopted the
    GPU's token at every flagged position where they differ); a flagged
    position is counted, an unflagged one must match bit for bit. Returns
    (tally, set of requests compared)."""
    t = Tally()
    for b in reqs:
        for k in range(o["tokens"].shape[1]):
            # lse_k and c_k depend on x_{k-1} only, which both sides share
            assert rel_close(g["lse"][b, k], o["lse"][b, k]), ("lse", b, k, g["lse"][b, k], o["lse"][b, k])
            assert rel_close(g["conf"][b, k], o["conf"][b, k]), ("conf", b, k, g["conf"][b, k], o["conf"][b, k])
            if o["margin"][b, k] < oracle.MARGIN:
                t.flagged += 1
            assert g["tokens"][b, k] == o["tokens"][b, k], ("token", b, k, g["tokens"][b, k], o["tokens"][b, k],
                                                             o["margin"][b, k])
            assert rel_close(g["pd_tok"][b, k], o["pd_tok"][b, k]), ("pd", b, k, g["pd_tok"][b, k], o["pd_tok"][b, k])
            t.compared += 1
    t.budget = DRAFT_FLAG_RATE * t.compared
    t.slack = 1
    _record("draft", t.compared, t.flagged)
    return t, set(reqs)


def forced_draft(g: Dict[str, np.ndarray], draft_fn, reqs: Sequence[int]) -> Dict[str, np.ndarray]:
    """The oracle's draft of ``reqs`` under teacher forcing.

    ``draft_fn(reqs, force)`` runs the oracle (force: [B, gamma] int32, -1 =
    draw). Wherever the oracle flags a position and its token differs from the
    GPU's, it adopts the GPU's token there and drafts the rest of that
    request again from it. A difference at an unflagged position is left in
    place for ``compare_draft`` to report."""
    reqs = list(reqs)
    B, gamma = g["tokens"].shape
    force = np.full((B, gamma), -1, np.int32)
    od = draft_fn(reqs, None)
    todo = reqs
    while todo:
        redo = []
        for b in todo:
            for k in range(gamma):
                if od["tokens"][b, k] == g["tokens"][b, k]:
                    continue
                if od["margin"][b, k] < oracle.MARGIN and force[b, k] < 0:
                    force[b, k] = g["tokens"][b, k]
                    redo.append(b)
                break
        if redo:
            o2 = draft_fn(redo, force)
            for key in od:
                od[key][redo] = o2[key][redo]
        todo = redo
    return od


def check_draft(g: Dict[str, np.ndarray], draft_fn, reqs: Sequence[int]):
    """forced_draft, then compare_draft; returns (tally, oracle outputs)."""
    od = forced_draft(g, draft_fn, reqs)
    t, _ = compare_draft(g, od, reqs)
    return t, od


def compare_verify(g: Dict[str, np.ndarray], o: Dict[str, np.ndarray], reqs: Sequence[int]) -> Tally:
    t = Tally()
    for b in reqs:
        if o["acc_margin"][b] < oracle.MARGIN or o["smp_margin"][b] < oracle.MARGIN:
            t.flagged += 1
            t.excluded_requests += 1
            continue
        assert g["n_acc"][b] == o["n_acc"][b], ("n_acc", b, g["n_acc"][b], o["n_acc"][b])
        assert g["next_anchor"][b] == o["next_anchor"][b], (
            "next_anchor", b, g["next_anchor"][b], o["next_anchor"][b], o["resid"][b], o["smp_margin"][b])
        t.compared += 2
    t.budget = VERIFY_FLAG_RATE * (t.compared + t.flagged)
    _record("verify", t.compared, t.flagged)
    return t


def oracle_plan(wl: wlmod.Workload, conf32: np.ndarray, sps: np.ndarray, lagged_conf=None):
    """Lengths the oracle assigns and its PlanMargin (infinite in static mode)."""
    B, g = conf32.shape
    if wl.mode == "static":
        return np.full(B, g + 1, np.int32), oracle.PlanMargin()
    if wl.mode == "compact" or lagged_conf is None:
        L, _, m = oracle.plan_sync(conf32, sps)
        return L, m
    L, _, m = oracle.plan_lagged(conf32, lagged_conf, sps)
    return L, m


def pack_np(P_full: np.ndarray, lengths: np.ndarray) -> np.ndarray:
    B, R, V = P_full.shape
    return np.concatenate([P_full[b, :lengths[b]] for b in range(B)]).reshape(-1, V)


def row_off_np(lengths: np.ndarray) -> np.ndarray:
    ro = np.zeros(len(lengths) + 1, np.int32)
    ro[1:] = np.cumsum(lengths)
    return ro


def gpu_np(d: Dict[str, torch.Tensor]) -> Dict[str, np.ndarray]:
    return {k: v.cpu().numpy() for k, v in d.items()}


def run_gpu_round(ws, dev: Dict[str, torch.Tensor], seed: int, rnd: int, anchor: Optional[torch.Tensor] = None):
    """draft -> plan -> (pack P by the GPU's lengths) -> verify, through the C-ABI."""
    anchor = dev["anchor"] if anchor is None else anchor
    d = ws.draft(dev["U"], dev["W1"], dev["W2"], anchor, dev["h"], dev["w"], dev["T"], seed, rnd)
    p = ws.plan(d["conf"], dev["sps"])
    P = wlmod.pack_rows(dev["P_full"], p["lengths"])
    v = ws.verify(P, p["row_off"], p["lengths"], anchor, d["tokens"], d["pd_tok"], d["lse"], dev["U"],
                  dev["W1"], dev["W2"], seed, rnd)
    torch.cuda.synchronize()
    st = ws.device_status()
    assert st == 0, f"device status {st}"
    return {**gpu_np(d), **gpu_np(p), **gpu_np(v)}
