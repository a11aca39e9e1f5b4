"""Seeded synthetic inputs for one DSpark round.

This module only draws random tensors with the shapes and value distributions
of the five synthetic workloads and marshals target-logit rows into the packed
ragged layout. It holds none of the method's arithmetic (no logits, no
softmax, no sampling, no planning), so both the CUDA path and the CPU oracle
may consume what it produces.

Workloads (sizes and distributions follow the configuration list that the
benchmark is quoted on):

  tiny   B=2   gamma=3  V=1024   r=16  H=64    fp32 weights, flat SPS table
  small  B=32  gamma=5  V=32000  r=256 H=1024  bf16 weights, static verify
  prod   B=128 gamma=5  V=129280 r=256 H=5120  bf16 weights, compact planner
  long   B=128 gamma=15 V=151936 r=256 H=4096  bf16 weights, full verify
  loaded B=256 gamma=7  V=129280 r=256 H=5120  bf16 weights, lagged planner

Target logits: row j of request b (j = 0..gamma) is the target's distribution
for the token after x_j. The configurations define it as the draft logits at
the drafted prefix plus Gaussian noise. A generator may not run the drafter,
so row j is drawn as the base logits U[b, j] plus noise (the Markov bias it
omits has standard deviation about sqrt(r) * std(W1) * std(W2), i.e. 0.006 for
the bf16 workloads and 0.04 for the tiny one, against std(U) >= 2); the bonus
row gamma has no draft position and is a fresh U-distributed draw plus noise.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    gamma: int
    V: int
    r: int
    H: int
    wdtype: str            # "f32" or "bf16" storage of W1 / W2
    mode: str              # "static" | "compact" | "lagged"
    seed: int
    u_std: float           # std of the base logits U
    w_std: float           # std of W1 and W2
    cw_std: float = 0.05   # std of the confidence weights w
    temp_range: Optional[tuple] = None   # STS temperatures ~ U[lo, hi]; None -> 1
    sps_knee: Optional[float] = None     # SPS(B) = 400 / (1 + B / knee); None -> flat
    noise: str = "const"   # "const" | "pos_linear" | "per_request"
    noise_args: tuple = (0.5,)
    lag: int = 0
    rounds: int = 1

    @property
    def n_sps(self) -> int:
        # SPS is indexed by the total number of verify tokens, 1 .. B*(gamma+1);
        # entry 0 is unused.
        return 1 + self.B * (self.gamma + 1)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", B=2, gamma=3, V=1024, r=16, H=64, wdtype="f32",
                     mode="compact", seed=0, u_std=2.0, w_std=0.1,
                     noise="const", noise_args=(0.5,)),
    "small": Workload("small", B=32, gamma=5, V=32000, r=256, H=1024, wdtype="bf16",
                      mode="static", seed=1, u_std=3.0, w_std=0.02,
                      noise="pos_linear", noise_args=(0.3, 1.0)),
    "prod": Workload("prod", B=128, gamma=5, V=129280, r=256, H=5120, wdtype="bf16",
                     mode="compact", seed=2, u_std=2.0, w_std=0.02,
                     temp_range=(0.8, 1.5), sps_knee=512.0,
                     noise="const", noise_args=(0.5,)),
    "long": Workload("long", B=128, gamma=15, V=151936, r=256, H=4096, wdtype="bf16",
                     mode="static", seed=3, u_std=2.0, w_std=0.02,
                     noise="pos_linear", noise_args=(0.2, 2.0)),
    "loaded": Workload("loaded", B=256, gamma=7, V=129280, r=256, H=5120, wdtype="bf16",
                       mode="lagged", seed=4, u_std=2.0, w_std=0.02,
                       sps_knee=128.0, noise="per_request", noise_args=(0.1, 0.5, 1.0),
                       lag=2, rounds=8),
}


def sps_table(wl: Workload) -> torch.Tensor:
    """SPS[n] for n = 0 .. B*(gamma+1) as float64 (entry 0 unused, set to SPS(1))."""
    n = torch.arange(wl.n_sps, dtype=torch.float64)
    n[0] = 1.0
    if wl.sps_knee is None:
        return torch.full((wl.n_sps,), 400.0, dtype=torch.float64)
    return 400.0 / (1.0 + n / wl.sps_knee)


def noise_std(wl: Workload, gen: torch.Generator) -> torch.Tensor:
    """Per (request, target row) noise std, shape [B, gamma+1] float32.

    Row j is the target distribution at draft position k = j + 1.
    """
    B, g = wl.B, wl.gamma
    k = torch.arange(1, g + 2, dtype=torch.float32)
    if wl.noise == "const":
        s = torch.full((B, g + 1), float(wl.noise_args[0]))
    elif wl.noise == "pos_linear":
        base, slope = wl.noise_args
        s = (base * (1.0 + slope * k / g)).expand(B, g + 1).clone()
    elif wl.noise == "per_request":
        choices = torch.tensor(wl.noise_args, dtype=torch.float32)
        idx = torch.randint(0, len(wl.noise_args), (B,), generator=gen)
        s = choices[idx].unsqueeze(1).expand(B, g + 1).clone()
    else:
        raise ValueError(wl.noise)
    return s


def _randn(shape, std, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std


def make_inputs(wl: Workload, device: str = "cpu", with_target: bool = True) -> Dict[str, torch.Tensor]:
    """Draw every input of one round for workload ``wl``.

    All tensors come from one ``torch.Generator`` seeded with ``wl.seed`` on
    ``device``; CPU and CUDA generators give different (each reproducible)
    streams, so parity tests draw on the CPU and copy to the GPU.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed)
    B, g, V, r, H = wl.B, wl.gamma, wl.V, wl.r, wl.H
    out: Dict[str, torch.Tensor] = {}
    out["U"] = _randn((B, g, V), wl.u_std, gen, device)
    w1 = _randn((V, r), wl.w_std, gen, device)
    w2 = _randn((r, V), wl.w_std, gen, device)
    if wl.wdtype == "bf16":
        w1, w2 = w1.to(torch.bfloat16), w2.to(torch.bfloat16)
    out["W1"], out["W2"] = w1.contiguous(), w2.contiguous()
    out["anchor"] = torch.randint(0, V, (B,), generator=gen, device=device, dtype=torch.int64).to(torch.int32)
    out["h"] = _randn((B, g, H), 1.0, gen, device)
    out["w"] = _randn((H + r,), wl.cw_std, gen, device)
    if wl.temp_range is None:
        out["T"] = torch.ones(g, dtype=torch.float32, device=device)
    else:
        lo, hi = wl.temp_range
        out["T"] = (lo + (hi - lo) * torch.rand(g, generator=gen, device=device)).to(torch.float32)
    out["sps"] = sps_table(wl).to(device)
    if with_target:
        cpu_gen = torch.Generator(device="cpu")
        cpu_gen.manual_seed(wl.seed + 7919)
        sig = noise_std(wl, cpu_gen).to(device)                      # [B, g+1]
        P = torch.empty((B, g + 1, V), dtype=torch.float32, device=device)
        P[:, :g] = out["U"]
        P[:, g] = _randn((B, V), wl.u_std, gen, device)
        P += _randn((B, g + 1, V), 1.0, gen, device) * sig.unsqueeze(-1)
        out["P_full"] = P
    return out


# Held-out calibration sets for the STS fit: confidence logits per position
# (mean falling along the block, as later positions are drafted with less
# context) and soft acceptance labels in [0, 1] that rise with the logit but
# are noisier and flatter than the logit's own sigmoid would be, so that the
# best temperatures differ from 1 and from position to position.
STS_SETS = {
    "sts_small": dict(N=20000, gamma=4, G=40, M=15, seed=49),
    "sts_prod": dict(N=262144, gamma=5, G=64, M=15, seed=41),
}


def sts_grid(G: int) -> torch.Tensor:
    """G temperatures from 0.1 upwards in steps of 0.1 (fp32)."""
    return (torch.arange(1, G + 1, dtype=torch.float64) * 0.1).to(torch.float32)


def make_sts_inputs(N: int, gamma: int, seed: int, device: str = "cpu") -> Dict[str, torch.Tensor]:
    gen = torch.Generator().manual_seed(seed)
    mu = torch.linspace(2.0, 0.5, gamma, dtype=torch.float64)
    raw = mu + 1.5 * torch.randn(N, gamma, generator=gen, dtype=torch.float64)
    # labels: a clipped affine function of the logit plus noise (no sigmoid)
    slope = torch.linspace(0.12, 0.2, gamma, dtype=torch.float64)
    lab = 0.55 + slope * raw + 0.08 * torch.randn(N, gamma, generator=gen, dtype=torch.float64)
    cstar = lab.clamp(0.02, 0.98)
    return {"raw": raw.to(torch.float32).to(device), "cstar": cstar.to(torch.float32).to(device)}


def make_rnn_weights(wl: Workload, seed_offset: int = 31337) -> torch.Tensor:
    """The RNN head's stacked weights Wr [3, r, 2r + H] (W_g, W_c, W_o) for
    workload ``wl`` (CPU), in the workload's weight dtype: entries
    N(0, 1 / (2r + H)), so that each pre-activation is of order one."""
    gen = torch.Generator().manual_seed(wl.seed + seed_offset)
    Z = 2 * wl.r + wl.H
    Wr = torch.randn((3, wl.r, Z), generator=gen, dtype=torch.float32) / Z ** 0.5
    return Wr.to(torch.bfloat16).contiguous() if wl.wdtype == "bf16" else Wr.contiguous()


def make_loss_inputs(wl: Workload, seed_offset: int = 104729) -> Dict[str, torch.Tensor]:
    """Inputs of the teacher-forced training objective for workload ``wl`` (CPU).

    U, W1, W2 and the anchors are the round's; P [B, gamma, V] is the target's
    logits at the gamma drafted positions (rows 0..gamma-1 of the round's
    target rows); the reference tokens x* are uniform over the vocabulary and
    the confidences uniform in [0.02, 0.98].
    """
    base = make_inputs(wl)
    gen = torch.Generator().manual_seed(wl.seed + seed_offset)
    B, g, V = wl.B, wl.gamma, wl.V
    return {"U": base["U"], "W1": base["W1"], "W2": base["W2"], "anchor": base["anchor"],
            "P": base["P_full"][:, :g].contiguous(),
            "xstar": torch.randint(0, V, (B, g), generator=gen, dtype=torch.int64).to(torch.int32),
            "conf": (0.02 + 0.96 * torch.rand(B, g, generator=gen)).to(torch.float32)}


def make_tree_targets(wl: Workload, U: torch.Tensor, dep: torch.Tensor, sigma: float = 0.5,
                      seed_offset: int = 7727) -> torch.Tensor:
    """Target logits of a draft tree's nodes, P [B, N+1, V] fp32 (CPU).

    Row i of request b is the target's distribution of the token after node
    i's path. As for the chain (module docstring), it is drawn as the base
    logits of the position that token takes, U[b, dep[b, i]], plus
    N(0, sigma^2) noise; a node at depth gamma is followed by the bonus
    position, a fresh U-distributed draw plus noise; empty node slots
    (dep < 0) are zeros.
    """
    gen = torch.Generator().manual_seed(wl.seed + seed_offset)
    B, N1 = dep.shape
    g, V = wl.gamma, wl.V
    P = torch.zeros(B, N1, V, dtype=torch.float32)
    d = dep.to(torch.int64).cpu()
    for b in range(B):
        for i in range(N1):
            k = int(d[b, i])
            if k < 0:
                continue
            base = U[b, k] if k < g else torch.randn(V, generator=gen) * wl.u_std
            P[b, i] = base + torch.randn(V, generator=gen) * sigma
    return P


def pack_rows(P_full: torch.Tensor, lengths: torch.Tensor) -> torch.Tensor:
    """Packed ragged target logits [sum(lengths), V]: rows 0..lengths[b]-1 of each request.

    This stands in for the target model, which writes its verify logits in
    the packed layout directly; it is a gather, not part of the method.
    """
    B, R, V = P_full.shape
    lengths = lengths.to(torch.int64).cpu()
    idx = torch.cat([b * R + torch.arange(int(lengths[b])) for b in range(B)])
    return P_full.reshape(B * R, V).index_select(0, idx.to(P_full.device)).contiguous()


def row_offsets(lengths: torch.Tensor) -> torch.Tensor:
    """Exclusive prefix sum of lengths, [B+1] int32 (marshalling helper for tests)."""
    l = lengths.to(torch.int64).cpu()
    off = torch.zeros(l.numel() + 1, dtype=torch.int64)
    off[1:] = torch.cumsum(l, 0)
    return off.to(torch.int32)


def bf16_bits(t: torch.Tensor) -> torch.Tensor:
    """Raw 16-bit patterns of a bfloat16 tensor (for consumers that read bits)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16)


def hbm_bytes(wl: Workload, sum_len: int) -> Dict[str, float]:
    """Algorithmic bytes of one round: U once, W2 once per draft step, verified P rows."""
    wb = 2 if wl.wdtype == "bf16" else 4
    u = wl.B * wl.gamma * wl.V * 4
    w2 = wl.r * wl.V * wb
    p = sum_len * wl.V * 4
    return {"U": float(u), "W2_per_step": float(w2), "P": float(p),
            "alg": float(u + wl.gamma * w2 + p), "alg_w2_once": float(u + w2 + p)}


__all__ = ["Workload", "WORKLOADS", "make_inputs", "pack_rows", "row_offsets",
           "sps_table", "noise_std", "bf16_bits", "hbm_bytes"]

