"""fp64 CPU oracle of one DSpark round (TEST INFRASTRUCTURE).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It wraps ``dspark_oracle.c`` (plain C,
fp64, its own Philox) through ctypes and numpy. It shares no code with the
CUDA library; see the C file's header for what each entry computes and which
passage of the pages it follows.

Sampling margins are returned so that callers can apply the parity rule:
decisions whose margin is below ``MARGIN`` are "flagged" (too close to call in
fp32) and are counted instead of compared.
"""

from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from typing import Dict, Optional, Sequence

import numpy as np

MARGIN = 1e-5          # parity margin on sampling keys, accept ratios and Theta

# purposes of the random stream (counter word 3, bits 24..31)
P_DRAFT_BLOCK, P_DRAFT_TOKEN, P_ACCEPT = 1, 2, 3
P_BONUS_BLOCK, P_BONUS_TOKEN, P_RESID_BLOCK, P_RESID_TOKEN = 4, 5, 6, 7
P_TREE_ACCEPT, P_TREE_BLOCK, P_TREE_TOKEN = 8, 9, 10

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libdspark_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp contraction off so x86 and Arm agree)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Dims(C.Structure):
    _fields_ = [("B", C.c_int), ("gamma", C.c_int), ("V", C.c_int), ("r", C.c_int),
                ("H", C.c_int), ("w_bf16", C.c_int)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            l = C.CDLL(build())
            P = C.c_void_p
            u32, u64, i32, dbl = C.c_uint32, C.c_uint64, C.c_int, C.c_double
            l.orc_philox4x32_10.argtypes = [P, P, P]
            l.orc_word.argtypes = [u64, u64, u32, u32, u32, u32]
            l.orc_word.restype = u32
            l.orc_uniform.argtypes = [u64, u64, u32, u32, u32, u32]
            l.orc_uniform.restype = dbl
            l.orc_gumbel.argtypes = [u64, u64, u32, u32, u32, u32]
            l.orc_gumbel.restype = dbl
            l.orc_logsumexp.argtypes = [P, C.c_long]
            l.orc_logsumexp.restype = dbl
            l.orc_draft.argtypes = [P, P, P, P, P, P, P, P, u64, u64, P, i32, P, P, P, P, P, P]
            l.orc_verify_head.argtypes = [P, P, P, P, P, P, P, P, P, P, u64, u64, P, i32,
                                          P, P, P, P, P]
            l.orc_pctree_build.argtypes = [P, P, P, P, P, i32, i32, P, i32, P, P, P, P, P, P]
            l.orc_pctree_verify.argtypes = [P, i32, P, P, P, u64, u64, P, i32, P, P, P, P]
            l.orc_rnn_draft.argtypes = [P, P, P, P, P, P, P, P, P, u64, u64, P, i32, P, P, P, P, P, P, P]
            l.orc_plan_sync.argtypes = [i32, i32, P, P, P, P]
            l.orc_plan_sync.restype = i32
            l.orc_plan_capacity.argtypes = [i32, i32, P, P, P]
            l.orc_plan_capacity.restype = i32
            l.orc_plan_topk.argtypes = [i32, i32, P, i32, P, P]
            l.orc_plan_theta_path.argtypes = [i32, i32, P, P, P]
            l.orc_survival.argtypes = [i32, i32, P, P]
            l.orc_verify.argtypes = [P, P, P, P, P, P, P, P, P, u64, u64, P, i32,
                                     P, P, P, P, P]
            l.orc_sample.argtypes = [P, C.c_long, u64, u64, u32, u32, u32, u32, P]
            l.orc_sample.restype = i32
            l.orc_sample_draft.argtypes = [P, C.c_long, u64, u64, u32, u32, P]
            l.orc_sample_draft.restype = i32
            l.orc_residual.argtypes = [P, P, C.c_long, u64, u64, u32, u32, P]
            l.orc_residual.restype = i32
            l.orc_markov_logits.argtypes = [P, P, P, P, i32, P]
            l.orc_sts_fit.argtypes = [i32, i32, P, P, i32, P, i32, P, P, P]
            l.orc_train_loss.argtypes = [P, P, P, P, P, P, P, P, dbl, P, P, P, P]
            l.orc_block_width.restype = i32
            l.orc_set_threads.argtypes = [i32]
            l.orc_get_threads.restype = i32
            _lib = l
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


def block_width() -> int:
    return int(lib().orc_block_width())


# ---------------------------------------------------------------- random stream
def philox(ctr: Sequence[int], key: Sequence[int]) -> np.ndarray:
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    o = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(o))
    return o


def word(seed, rnd, purpose, b, j, v) -> int:
    return int(lib().orc_word(seed, rnd, purpose, b, j, v))


def uniform(seed, rnd, purpose, b, j, v) -> float:
    return float(lib().orc_uniform(seed, rnd, purpose, b, j, v))


def gumbel(seed, rnd, purpose, b, j, v) -> float:
    return float(lib().orc_gumbel(seed, rnd, purpose, b, j, v))


def logsumexp(x) -> float:
    a = _c(x, np.float64)
    return float(lib().orc_logsumexp(_p(a), a.size))


def sample(logw, seed=0, rnd=0, pblk=P_DRAFT_BLOCK, ptok=P_DRAFT_TOKEN, b=0, j=0):
    """One two-level Gumbel-max draw from weights exp(logw). Returns (v, margin)."""
    a = _c(logw, np.float64)
    m = np.zeros(1, np.float64)
    v = lib().orc_sample(_p(a), a.size, seed, rnd, pblk, ptok, b, j, _p(m))
    return int(v), float(m[0])


def sample_draft(logw, seed=0, rnd=0, b=0, j=0):
    """One draw with the draft's random stream (block by Gumbel-max, token
    inside the block by Gumbel-max; purposes draft block / draft token).
    Returns (v, margin)."""
    a = _c(logw, np.float64)
    m = np.zeros(1, np.float64)
    v = lib().orc_sample_draft(_p(a), a.size, seed, rnd, b, j, _p(m))
    return int(v), float(m[0])


def train_loss(U, W1, W2, anchor, xstar, P, conf, tau: float) -> Dict[str, np.ndarray]:
    """Teacher-forced training objective (see ``orc_train_loss``): U and P are
    [B, gamma, V] fp32, xstar [B, gamma] int32, conf [B, gamma] fp32. Returns
    per-position ce, l1, bce [B, gamma] fp64 and the scalar loss."""
    U = _c(U, np.float32)
    B, g, V = U.shape
    W1a, bf = _weights(W1)
    W2a, _ = _weights(W2)
    d = _dims(B, g, V, W1a.shape[1], 0, bf)
    an = _c(anchor, np.int32)
    xs = _c(xstar, np.int32)
    Pa = _c(P, np.float32)
    cf = _c(conf, np.float32)
    ce = np.zeros((B, g), np.float64)
    l1 = np.zeros((B, g), np.float64)
    bce = np.zeros((B, g), np.float64)
    loss = np.zeros(1, np.float64)
    lib().orc_train_loss(C.byref(d), _p(U), _p(W1a), _p(W2a), _p(an), _p(xs), _p(Pa), _p(cf), float(tau),
                         _p(ce), _p(l1), _p(bce), _p(loss))
    return {"ce": ce, "l1": l1, "bce": bce, "loss": float(loss[0])}


def sts_fit(raw, cstar, Tgrid, M: int = 15):
    """Sequential temperature scaling (see ``orc_sts_fit``): raw and cstar are
    [N, gamma]; returns (T [gamma] float32, ece [gamma], margin [gamma])."""
    r = _c(raw, np.float32)
    c = _c(cstar, np.float32)
    t = _c(Tgrid, np.float32)
    N, g = r.shape
    T = np.zeros(g, np.float32)
    ece = np.zeros(g, np.float64)
    mg = np.zeros(g, np.float64)
    lib().orc_sts_fit(N, g, _p(r), _p(c), t.size, _p(t), M, _p(T), _p(ece), _p(mg))
    return T, ece, mg


def residual(pt, pd, seed=0, rnd=0, b=0, j=0):
    """One draw from norm(max(0, pt - pd)); v = -1 when there is no mass."""
    a, d = _c(pt, np.float64), _c(pd, np.float64)
    m = np.zeros(1, np.float64)
    v = lib().orc_residual(_p(a), _p(d), a.size, seed, rnd, b, j, _p(m))
    return int(v), float(m[0])


# ---------------------------------------------------------------- round stages
def _dims(B, gamma, V, r, H, w_bf16) -> _Dims:
    return _Dims(B, gamma, V, r, H, 1 if w_bf16 else 0)


def _weights(W) -> (np.ndarray, bool):
    """Accept fp32 arrays or raw bf16 bit patterns (uint16/int16)."""
    a = np.asarray(W)
    if a.dtype in (np.uint16, np.int16):
        return np.ascontiguousarray(a.view(np.uint16)), True
    return _c(a, np.float32), False


def _force(force, B, g):
    if force is None:
        return None
    f = _c(force, np.int32)
    if f.shape != (B, g):
        raise ValueError(f"force must be [{B}, {g}], got {f.shape}")
    return f


def draft(U, W1, W2, anchor, h, w, T, seed: int, rnd: int,
          reqs: Optional[Sequence[int]] = None, force=None) -> Dict[str, np.ndarray]:
    """Markov-head draft tail + confidence head, eq. (4), (5), (7).

    U [B, gamma, V] fp32, W1 [V, r], W2 [r, V] (fp32 or bf16 bits), anchor [B],
    h [B, gamma, H], w [H + r], T [gamma]. ``reqs`` restricts the work to a
    subset of requests (global indices keep their random streams). ``force``
    [B, gamma] int32 (optional): entries >= 0 are adopted in place of the
    draw at that position (teacher forcing at flagged positions).
    """
    U = _c(U, np.float32)
    B, g, V = U.shape
    w1, bf = _weights(W1)
    w2, _ = _weights(W2)
    r = w1.shape[1]
    h = _c(h, np.float32)
    H = h.shape[2]
    anchor = _c(anchor, np.int32)
    w = _c(w, np.float32)
    T = _c(T, np.float32)
    rq = _c(range(B) if reqs is None else reqs, np.int32)
    d = _dims(B, g, V, r, H, bf)
    out = {"tokens": np.full((B, g), -1, np.int32), "pd_tok": np.full((B, g), np.nan),
           "lse": np.full((B, g), np.nan), "conf": np.full((B, g), np.nan),
           "margin": np.full((B, g), np.inf)}
    f = _force(force, B, g)
    lib().orc_draft(C.byref(d), _p(U), _p(w1), _p(w2), _p(anchor), _p(h), _p(w), _p(T),
                    seed, rnd, _p(rq), rq.size, None if f is None else _p(f), _p(out["tokens"]), _p(out["pd_tok"]),
                    _p(out["lse"]), _p(out["conf"]), _p(out["margin"]))
    return out


def rnn_draft(U, W1, W2, Wr, anchor, h, w, T, seed: int, rnd: int,
              reqs: Optional[Sequence[int]] = None, force=None) -> Dict[str, np.ndarray]:
    """Draft tail with the RNN head, eq. (6) (see ``orc_rnn_draft``).

    As ``draft``, plus Wr [3, r, 2r + H] (W_g, W_c, W_o; same storage as W1)
    and the output ``ovec`` [B, gamma, r]: the head's vector o_k with
    z_k = U_k + o_k W2.
    """
    U = _c(U, np.float32)
    B, g, V = U.shape
    w1, bf = _weights(W1)
    w2, _ = _weights(W2)
    wr, bf_r = _weights(Wr)
    if bf_r != bf:
        raise ValueError("Wr must be stored like W1 and W2")
    r = w1.shape[1]
    h = _c(h, np.float32)
    H = h.shape[2]
    if wr.shape != (3, r, 2 * r + H):
        raise ValueError(f"Wr must be [3, {r}, {2 * r + H}], got {wr.shape}")
    anchor = _c(anchor, np.int32)
    w = _c(w, np.float32)
    T = _c(T, np.float32)
    rq = _c(range(B) if reqs is None else reqs, np.int32)
    d = _dims(B, g, V, r, H, bf)
    out = {"tokens": np.full((B, g), -1, np.int32), "pd_tok": np.full((B, g), np.nan),
           "lse": np.full((B, g), np.nan), "conf": np.full((B, g), np.nan),
           "margin": np.full((B, g), np.inf), "ovec": np.full((B, g, r), np.nan)}
    f = _force(force, B, g)
    lib().orc_rnn_draft(C.byref(d), _p(U), _p(w1), _p(w2), _p(wr), _p(anchor), _p(h), _p(w), _p(T),
                        seed, rnd, _p(rq), rq.size, None if f is None else _p(f), _p(out["tokens"]),
                        _p(out["pd_tok"]),
                        _p(out["lse"]), _p(out["conf"]), _p(out["margin"]), _p(out["ovec"]))
    return out


def pctree_build(U, W1, W2, anchor, c: int, N: int, reqs: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """PCTree's draft tree (see ``orc_pctree_build``): U [B, gamma, V], W1, W2
    as for ``draft``; c children per parent, N nodes besides the root. Returns
    tok, par, dep [B, N+1] int32, lp [B, N+1], n_nodes [B], margin [B] (only
    the rows of ``reqs`` are written when it is given)."""
    U = _c(U, np.float32)
    B, g, V = U.shape
    w1, bf = _weights(W1)
    w2, _ = _weights(W2)
    d = _dims(B, g, V, w1.shape[1], 0, bf)
    an = _c(anchor, np.int32)
    rq = _c(range(B) if reqs is None else reqs, np.int32)
    out = {"tok": np.full((B, N + 1), -1, np.int32), "par": np.full((B, N + 1), -1, np.int32),
           "dep": np.full((B, N + 1), -1, np.int32), "lp": np.full((B, N + 1), -np.inf),
           "n_nodes": np.zeros(B, np.int32), "margin": np.full(B, np.inf)}
    lib().orc_pctree_build(C.byref(d), _p(U), _p(w1), _p(w2), _p(an), int(c), int(N), _p(rq), rq.size,
                           _p(out["tok"]), _p(out["par"]), _p(out["dep"]), _p(out["lp"]), _p(out["n_nodes"]),
                           _p(out["margin"]))
    return out


def pctree_verify(tok, par, P, gamma: int, seed: int, rnd: int,
                  reqs: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """PCTree's lossless tree verify (see ``orc_pctree_verify``): tok, par
    [B, N+1] from ``pctree_build``, P [B, N+1, V] the target logits after each
    node's path. Returns path [B, gamma+1], n_acc, next_anchor, margin [B]
    (only the rows of ``reqs`` when it is given)."""
    tok = _c(tok, np.int32)
    par = _c(par, np.int32)
    P = _c(P, np.float32)
    B, N1, V = P.shape
    d = _dims(B, gamma, V, 0, 0, False)
    rq = _c(range(B) if reqs is None else reqs, np.int32)
    out = {"path": np.full((B, gamma + 1), -1, np.int32), "n_acc": np.full(B, -1, np.int32),
           "next_anchor": np.full(B, -1, np.int32), "margin": np.full(B, np.inf)}
    lib().orc_pctree_verify(C.byref(d), N1 - 1, _p(tok), _p(par), _p(P), seed, rnd, _p(rq), rq.size,
                            _p(out["path"]), _p(out["n_acc"]), _p(out["next_anchor"]), _p(out["margin"]))
    return out


def survival(conf) -> np.ndarray:
    c = _c(conf, np.float32)
    B, g = c.shape
    a = np.zeros((B, g), np.float64)
    lib().orc_survival(B, g, _p(c), _p(a))
    return a


class PlanMargin:
    """How close a planner outcome was to changing.

    theta: smallest relative Theta gap over the comparisons taken (flips only
           under rounding of that size: fp64 reassociation on identical
           inputs, fp32 differences of the confidences otherwise);
    cut:   relative gap between the survival values on both sides of the cut
           (two candidates closer than this may swap across it when their
           confidences differ in the last bits).
    """

    def __init__(self, theta=np.inf, cut=np.inf):
        self.theta, self.cut = float(theta), float(cut)

    def flagged(self, theta_tol: float, cut_tol: float) -> bool:
        return self.theta < theta_tol or self.cut < cut_tol

    def __repr__(self):
        return f"PlanMargin(theta={self.theta:.3g}, cut={self.cut:.3g})"


def plan_sync(conf, sps):
    """Algorithm 1 with early stop -> (lengths [B], admitted m, PlanMargin)."""
    c = _c(conf, np.float32)
    B, g = c.shape
    s = _c(sps, np.float64)
    assert s.size >= 1 + B * (g + 1)
    L = np.zeros(B, np.int32)
    m = np.zeros(2, np.float64)
    k = lib().orc_plan_sync(B, g, _p(c), _p(s), _p(L), _p(m))
    return L, int(k), PlanMargin(m[0], m[1])


def plan_capacity(conf, sps):
    """K = argmax_m Theta_m over the full admission path -> (K, theta margin)."""
    c = _c(conf, np.float32)
    B, g = c.shape
    s = _c(sps, np.float64)
    m = np.zeros(1, np.float64)
    K = lib().orc_plan_capacity(B, g, _p(c), _p(s), _p(m))
    return int(K), float(m[0])


def plan_theta_path(conf, sps) -> np.ndarray:
    """Theta_m = (B + sum of the m largest survival values) * SPS(B + m) for
    m = 0 .. B*gamma: the path whose first maximum is the lagged capacity."""
    c = _c(conf, np.float32)
    B, g = c.shape
    s = _c(sps, np.float64)
    th = np.zeros(B * g + 1, np.float64)
    lib().orc_plan_theta_path(B, g, _p(c), _p(s), _p(th))
    return th


def plan_topk(conf, K: int):
    """Lengths of the K best candidates -> (lengths, cut margin)."""
    c = _c(conf, np.float32)
    B, g = c.shape
    L = np.zeros(B, np.int32)
    m = np.zeros(1, np.float64)
    lib().orc_plan_topk(B, g, _p(c), int(K), _p(L), _p(m))
    return L, float(m[0])


def plan_lagged(conf_now, conf_lagged, sps):
    """Asynchronous planner: capacity from lagged confidences, top-K of current.

    Returns (lengths, K, PlanMargin(theta of the capacity argmax, cut of the top-K)).
    """
    K, m1 = plan_capacity(conf_lagged, sps)
    L, m2 = plan_topk(conf_now, K)
    return L, K, PlanMargin(m1, m2)


def verify(P_packed, row_off, lengths, anchor, tokens, U, W1, W2, seed: int, rnd: int,
           reqs: Optional[Sequence[int]] = None, ovec=None) -> Dict[str, np.ndarray]:
    """Lossless ragged verify. Returns n_acc, next_anchor, margins, resid flag.
    ``ovec`` [B, gamma, r]: the RNN head's vectors o_k (p_d from U + o W2)
    instead of the Markov head's W1[x_{k-1}]."""
    P = _c(P_packed, np.float32)
    U = _c(U, np.float32)
    B, g, V = U.shape
    w1, bf = _weights(W1)
    w2, _ = _weights(W2)
    r = w1.shape[1]
    ro = _c(row_off, np.int32)
    L = _c(lengths, np.int32)
    anchor = _c(anchor, np.int32)
    tokens = _c(tokens, np.int32)
    rq = _c(range(B) if reqs is None else reqs, np.int32)
    d = _dims(B, g, V, r, 0, bf)
    out = {"n_acc": np.full(B, -1, np.int32), "next_anchor": np.full(B, -1, np.int32),
           "acc_margin": np.full(B, np.inf), "smp_margin": np.full(B, np.inf),
           "resid": np.zeros(B, np.int32)}
    ov = None if ovec is None else _c(ovec, np.float64)
    if ov is not None and ov.shape != (B, g, r):
        raise ValueError(f"ovec must be [{B}, {g}, {r}], got {ov.shape}")
    lib().orc_verify_head(C.byref(d), _p(P), _p(ro), _p(L), _p(anchor), _p(tokens), _p(U),
                          _p(w1), _p(w2), None if ov is None else _p(ov), seed, rnd, _p(rq), rq.size,
                          _p(out["n_acc"]), _p(out["next_anchor"]), _p(out["acc_margin"]),
                          _p(out["smp_margin"]), _p(out["resid"]))
    return out


def markov_logits(Urow, W1, W2, x_prev: int) -> np.ndarray:
    u = _c(Urow, np.float32)
    w1, bf = _weights(W1)
    w2, _ = _weights(W2)
    V, r = w1.shape
    d = _dims(1, 1, V, r, 0, bf)
    z = np.zeros(V, np.float64)
    lib().orc_markov_logits(C.byref(d), _p(u), _p(w1), _p(w2), int(x_prev), _p(z))
    return z
