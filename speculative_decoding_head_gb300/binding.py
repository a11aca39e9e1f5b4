"""Python binding of libdspark.so (ctypes; argument marshalling only).

Every step of a round runs in the library's CUDA kernels. PyTorch supplies
device memory and the current stream. If the library has not been built the
binding raises; there is no CPU fallback.
"""

from __future__ import annotations

import ctypes as C
import os
import threading
from typing import Dict, Optional

import torch

from .build import LIB_PATH

MODES = {"static": 0, "compact": 1, "lagged": 2}
WDTYPES = {"f32": 0, "bf16": 1}

SYMBOLS = [
    "dspark_ws_create", "dspark_ws_destroy", "dspark_ws_reset", "dspark_last_error",
    "dspark_status_string", "dspark_last_launch_count", "dspark_path",
    "dspark_markov_draft", "dspark_plan", "dspark_verify", "dspark_round", "dspark_ws_set_path",
    "dspark_sts_fit", "dspark_sts_scratch_bytes", "dspark_train_loss", "dspark_train_loss_scratch_bytes",
    "dspark_rnn_draft", "dspark_rnn_draft_scratch_bytes", "dspark_verify_rnn",
    "dspark_pctree_scratch_bytes", "dspark_pctree_build", "dspark_pctree_verify",
    "dspark_ws_set_shard", "dspark_plan_shard",
]


class DsparkError(RuntimeError):
    pass


class Dims(C.Structure):
    _fields_ = [("B", C.c_int), ("gamma", C.c_int), ("V", C.c_int), ("r", C.c_int), ("H", C.c_int),
                ("wdtype", C.c_int), ("mode", C.c_int), ("lag", C.c_int)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB_PATH


def load() -> C.CDLL:
    """Load libdspark.so (built by __graft_entry__.build() or build.py)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise DsparkError(f"libdspark.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        lib = C.CDLL(LIB_PATH)
        P, i32, u64 = C.c_void_p, C.c_int, C.c_uint64
        lib.dspark_ws_create.argtypes = [C.POINTER(Dims), C.POINTER(P)]
        lib.dspark_ws_create.restype = i32
        lib.dspark_ws_destroy.argtypes = [P]
        lib.dspark_ws_destroy.restype = None
        lib.dspark_ws_reset.argtypes = [P, P]
        lib.dspark_ws_reset.restype = i32
        lib.dspark_last_error.argtypes = [P, C.POINTER(i32)]
        lib.dspark_last_error.restype = i32
        lib.dspark_status_string.argtypes = [i32]
        lib.dspark_status_string.restype = C.c_char_p
        lib.dspark_last_launch_count.argtypes = [P]
        lib.dspark_last_launch_count.restype = i32
        lib.dspark_path.argtypes = [P]
        lib.dspark_path.restype = C.c_char_p
        lib.dspark_ws_set_path.argtypes = [P, C.c_char_p]
        lib.dspark_ws_set_path.restype = i32
        lib.dspark_markov_draft.argtypes = [P, P, P, P, P, P, P, P, u64, u64, P, P, P, P, P]
        lib.dspark_markov_draft.restype = i32
        lib.dspark_plan.argtypes = [P, P, P, P, P, P]
        lib.dspark_plan.restype = i32
        lib.dspark_verify.argtypes = [P, P, P, P, P, P, P, P, P, P, P, u64, u64, P, P, P]
        lib.dspark_verify.restype = i32
        lib.dspark_round.argtypes = [P] * 10 + [u64, u64] + [P] * 9
        lib.dspark_round.restype = i32
        lib.dspark_sts_fit.argtypes = [P, P, i32, i32, P, i32, i32, P, P, P, P, P]
        lib.dspark_sts_fit.restype = i32
        lib.dspark_sts_scratch_bytes.argtypes = [i32, i32]
        lib.dspark_sts_scratch_bytes.restype = C.c_size_t
        lib.dspark_train_loss.argtypes = [P] * 8 + [C.c_double] + [P] * 6
        lib.dspark_train_loss.restype = i32
        lib.dspark_train_loss_scratch_bytes.argtypes = [P]
        lib.dspark_train_loss_scratch_bytes.restype = C.c_size_t
        lib.dspark_rnn_draft.argtypes = [P] * 9 + [u64, u64] + [P] * 7
        lib.dspark_rnn_draft.restype = i32
        lib.dspark_verify_rnn.argtypes = [P] * 11 + [u64, u64] + [P] * 3
        lib.dspark_verify_rnn.restype = i32
        lib.dspark_rnn_draft_scratch_bytes.argtypes = [P]
        lib.dspark_rnn_draft_scratch_bytes.restype = C.c_size_t
        lib.dspark_pctree_scratch_bytes.argtypes = [P, i32, i32]
        lib.dspark_pctree_scratch_bytes.restype = C.c_size_t
        lib.dspark_pctree_build.argtypes = [P] * 5 + [i32, i32] + [P] * 7
        lib.dspark_pctree_build.restype = i32
        lib.dspark_pctree_verify.argtypes = [P] * 4 + [i32, u64, u64] + [P] * 4
        lib.dspark_pctree_verify.restype = i32
        lib.dspark_ws_set_shard.argtypes = [P, i32]
        lib.dspark_ws_set_shard.restype = i32
        lib.dspark_plan_shard.argtypes = [P, P, P, i32, i32, P, P, P, P, P]
        lib.dspark_plan_shard.restype = i32
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load().dspark_status_string(int(code)).decode()


def _check(code: int, what: str) -> None:
    if code != 0:
        raise DsparkError(f"{what}: {status_string(code)} ({code})")


def _ptr(t: Optional[torch.Tensor], dtype=None, name="") -> C.c_void_p:
    if t is None:
        return C.c_void_p(0)
    if not t.is_cuda:
        raise DsparkError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise DsparkError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise DsparkError(f"{name} must be {dtype}, got {t.dtype}")
    return C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def sts_fit(raw: torch.Tensor, cstar: torch.Tensor, Tgrid: torch.Tensor, M: int = 15, stream=None):
    """Sequential temperature scaling (``dspark_sts_fit``): raw and cstar are
    [N, gamma] fp32 CUDA tensors, Tgrid [G] fp32. Returns (T [gamma] fp32,
    ece [gamma] fp64, device status [1] int32), all on the device."""
    lib = load()
    f32 = torch.float32
    if raw.dim() != 2 or cstar.shape != raw.shape:
        raise DsparkError("raw and cstar must be [N, gamma] of the same shape")
    N, g = raw.shape
    G = Tgrid.numel()
    dev = raw.device
    scratch = torch.empty(int(lib.dspark_sts_scratch_bytes(N, G)), dtype=torch.uint8, device=dev)
    T = torch.empty(g, dtype=f32, device=dev)
    ece = torch.empty(g, dtype=torch.float64, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    code = lib.dspark_sts_fit(_ptr(raw, f32, "raw"), _ptr(cstar, f32, "cstar"), N, g, _ptr(Tgrid, f32, "Tgrid"), G,
                              int(M), _ptr(T, f32, "T"), _ptr(ece, torch.float64, "ece"), _ptr(scratch, None, "scratch"),
                              _ptr(status, torch.int32, "status"), _stream(stream))
    _check(code, "dspark_sts_fit")
    return T, ece, status


class Workspace:
    """One DSpark workspace: the library's scratch arena for a fixed shape."""

    def __init__(self, B: int, gamma: int, V: int, r: int, H: int, wdtype: str = "bf16",
                 mode: str = "compact", lag: int = 2, path: Optional[str] = None):
        self.lib = load()
        self.dims = Dims(B, gamma, V, r, H, WDTYPES[wdtype], MODES[mode], lag if mode == "lagged" else 0)
        self.wdtype = torch.bfloat16 if wdtype == "bf16" else torch.float32
        self._h = C.c_void_p()
        _check(self.lib.dspark_ws_create(C.byref(self.dims), C.byref(self._h)), "dspark_ws_create")
        if path is not None:
            self.set_path(path)

    @classmethod
    def for_workload(cls, wl, path: Optional[str] = None) -> "Workspace":
        return cls(wl.B, wl.gamma, wl.V, wl.r, wl.H, wl.wdtype, wl.mode, wl.lag or 2, path)

    def close(self) -> None:
        if getattr(self, "_h", None) and self._h.value:
            self.lib.dspark_ws_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------ state
    @property
    def handle(self) -> C.c_void_p:
        return self._h

    @property
    def path(self) -> str:
        return self.lib.dspark_path(self._h).decode()

    def set_path(self, path: str) -> None:
        _check(self.lib.dspark_ws_set_path(self._h, path.encode()), "dspark_ws_set_path")

    @property
    def last_launches(self) -> int:
        return int(self.lib.dspark_last_launch_count(self._h))

    def reset(self, stream=None) -> None:
        _check(self.lib.dspark_ws_reset(self._h, _stream(stream)), "dspark_ws_reset")

    def device_status(self) -> int:
        v = C.c_int(0)
        _check(self.lib.dspark_last_error(self._h, C.byref(v)), "dspark_last_error")
        return int(v.value)

    # ------------------------------------------------------------ outputs
    def new_draft_outputs(self, device="cuda") -> Dict[str, torch.Tensor]:
        B, g = self.dims.B, self.dims.gamma
        return {"tokens": torch.empty((B, g), dtype=torch.int32, device=device),
                "pd_tok": torch.empty((B, g), dtype=torch.float32, device=device),
                "lse": torch.empty((B, g), dtype=torch.float32, device=device),
                "conf": torch.empty((B, g), dtype=torch.float32, device=device)}

    def new_plan_outputs(self, device="cuda") -> Dict[str, torch.Tensor]:
        B = self.dims.B
        return {"lengths": torch.empty(B, dtype=torch.int32, device=device),
                "row_off": torch.empty(B + 1, dtype=torch.int32, device=device)}

    def new_verify_outputs(self, device="cuda") -> Dict[str, torch.Tensor]:
        B = self.dims.B
        return {"n_acc": torch.empty(B, dtype=torch.int32, device=device),
                "next_anchor": torch.empty(B, dtype=torch.int32, device=device)}

    # ------------------------------------------------------------ calls
    def draft(self, U, W1, W2, anchor, h, w, T, seed: int, rnd: int, out=None, stream=None):
        out = out or self.new_draft_outputs(U.device)
        f32, i32 = torch.float32, torch.int32
        code = self.lib.dspark_markov_draft(
            self._h, _ptr(U, f32, "U"), _ptr(W1, self.wdtype, "W1"), _ptr(W2, self.wdtype, "W2"),
            _ptr(anchor, i32, "anchor"), _ptr(h, f32, "h") if self.dims.H > 0 else C.c_void_p(0),
            _ptr(w, f32, "w"), _ptr(T, f32, "T"), int(seed), int(rnd),
            _ptr(out["tokens"], i32, "tokens"), _ptr(out["pd_tok"], f32, "pd_tok"),
            _ptr(out["lse"], f32, "lse"), _ptr(out["conf"], f32, "conf"), _stream(stream))
        _check(code, "dspark_markov_draft")
        return out

    def plan(self, conf, sps, out=None, stream=None):
        out = out or self.new_plan_outputs(conf.device)
        code = self.lib.dspark_plan(self._h, _ptr(conf, torch.float32, "conf"),
                                    _ptr(sps, torch.float64, "sps"),
                                    _ptr(out["lengths"], torch.int32, "lengths"),
                                    _ptr(out["row_off"], torch.int32, "row_off"), _stream(stream))
        _check(code, "dspark_plan")
        return out

    def set_shard(self, b_offset: int):
        """This workspace holds requests b_offset .. b_offset + B - 1 of a
        batch split across devices (``dspark_ws_set_shard``)."""
        _check(self.lib.dspark_ws_set_shard(self._h, int(b_offset)), "dspark_ws_set_shard")

    def plan_shard(self, conf, sps, b_begin: int, b_count: int, out=None, stream=None):
        """Plan the whole batch (this workspace's B) from the gathered
        confidences and keep requests b_begin .. b_begin + b_count - 1
        (``dspark_plan_shard``). ``out`` gains lengths_local [b_count] and
        row_off_local [b_count + 1]."""
        dev = conf.device
        out = out or self.new_plan_outputs(dev)
        if "lengths_local" not in out:
            out["lengths_local"] = torch.zeros(b_count, dtype=torch.int32, device=dev)
            out["row_off_local"] = torch.zeros(b_count + 1, dtype=torch.int32, device=dev)
        i32 = torch.int32
        code = self.lib.dspark_plan_shard(self._h, _ptr(conf, torch.float32, "conf"),
                                          _ptr(sps, torch.float64, "sps"), int(b_begin), int(b_count),
                                          _ptr(out["lengths"], i32, "lengths"), _ptr(out["row_off"], i32, "row_off"),
                                          _ptr(out["lengths_local"], i32, "lengths_local"),
                                          _ptr(out["row_off_local"], i32, "row_off_local"), _stream(stream))
        _check(code, "dspark_plan_shard")
        return out

    def verify(self, P, row_off, lengths, anchor, tokens, pd_tok, lse, U, W1, W2, seed: int, rnd: int,
               out=None, stream=None):
        out = out or self.new_verify_outputs(P.device)
        f32, i32 = torch.float32, torch.int32
        code = self.lib.dspark_verify(
            self._h, _ptr(P, f32, "P"), _ptr(row_off, i32, "row_off"), _ptr(lengths, i32, "lengths"),
            _ptr(anchor, i32, "anchor"), _ptr(tokens, i32, "tokens"), _ptr(pd_tok, f32, "pd_tok"),
            _ptr(lse, f32, "lse"), _ptr(U, f32, "U"), _ptr(W1, self.wdtype, "W1"),
            _ptr(W2, self.wdtype, "W2"), int(seed), int(rnd), _ptr(out["n_acc"], i32, "n_acc"),
            _ptr(out["next_anchor"], i32, "next_anchor"), _stream(stream))
        _check(code, "dspark_verify")
        return out

    def rnn_draft(self, U, W1, W2, Wr, anchor, h, w, T, seed: int, rnd: int, out=None, stream=None):
        """Draft tail with the RNN head (``dspark_rnn_draft``): as ``draft``,
        plus Wr [3, r, 2r + H]; ``out`` also holds ovec [B, gamma, r] fp32."""
        if out is None:
            out = self.new_draft_outputs(U.device)
            B, g, r = self.dims.B, self.dims.gamma, self.dims.r
            out["ovec"] = torch.empty(B, g, r, dtype=torch.float32, device=U.device)
            out["scratch"] = torch.empty(int(self.lib.dspark_rnn_draft_scratch_bytes(self._h)), dtype=torch.uint8,
                                         device=U.device)
        f32, i32 = torch.float32, torch.int32
        code = self.lib.dspark_rnn_draft(
            self._h, _ptr(U, f32, "U"), _ptr(W1, self.wdtype, "W1"), _ptr(W2, self.wdtype, "W2"),
            _ptr(Wr, self.wdtype, "Wr"), _ptr(anchor, i32, "anchor"),
            _ptr(h, f32, "h") if self.dims.H > 0 else C.c_void_p(0), _ptr(w, f32, "w"), _ptr(T, f32, "T"),
            int(seed), int(rnd), _ptr(out["tokens"], i32, "tokens"), _ptr(out["pd_tok"], f32, "pd_tok"),
            _ptr(out["lse"], f32, "lse"), _ptr(out["conf"], f32, "conf"), _ptr(out["ovec"], f32, "ovec"),
            _ptr(out["scratch"], None, "scratch"), _stream(stream))
        _check(code, "dspark_rnn_draft")
        return out

    def pctree_build(self, U, W1, W2, anchor, c: int, N: int, out=None, stream=None):
        """PCTree's draft tree (``dspark_pctree_build``): tok, par, dep [B, N+1]
        int32, lp [B, N+1] fp32, n_nodes [B] int32."""
        B = self.dims.B
        if out is None:
            dev = U.device
            nbytes = int(self.lib.dspark_pctree_scratch_bytes(self._h, int(c), int(N)))
            if nbytes == 0:
                raise DsparkError(f"dspark_pctree_build: unsupported c={c}, N={N}")
            out = {k: torch.empty(B, N + 1, dtype=torch.int32, device=dev) for k in ("tok", "par", "dep")}
            out["lp"] = torch.empty(B, N + 1, dtype=torch.float32, device=dev)
            out["n_nodes"] = torch.empty(B, dtype=torch.int32, device=dev)
            out["scratch"] = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        f32, i32 = torch.float32, torch.int32
        code = self.lib.dspark_pctree_build(
            self._h, _ptr(U, f32, "U"), _ptr(W1, self.wdtype, "W1"), _ptr(W2, self.wdtype, "W2"),
            _ptr(anchor, i32, "anchor"), int(c), int(N), _ptr(out["tok"], i32, "tok"), _ptr(out["par"], i32, "par"),
            _ptr(out["dep"], i32, "dep"), _ptr(out["lp"], f32, "lp"), _ptr(out["n_nodes"], i32, "n_nodes"),
            _ptr(out["scratch"], None, "scratch"), _stream(stream))
        _check(code, "dspark_pctree_build")
        return out

    def pctree_verify(self, P, tok, par, N: int, seed: int, rnd: int, out=None, stream=None):
        """PCTree's lossless tree verify (``dspark_pctree_verify``): P [B, N+1, V]
        fp32. Returns path [B, gamma+1], n_acc [B], next_anchor [B] (int32)."""
        B, g = self.dims.B, self.dims.gamma
        if out is None:
            dev = P.device
            out = {"path": torch.empty(B, g + 1, dtype=torch.int32, device=dev),
                   "n_acc": torch.empty(B, dtype=torch.int32, device=dev),
                   "next_anchor": torch.empty(B, dtype=torch.int32, device=dev)}
        i32 = torch.int32
        code = self.lib.dspark_pctree_verify(
            self._h, _ptr(P, torch.float32, "P"), _ptr(tok, i32, "tok"), _ptr(par, i32, "par"), int(N), int(seed),
            int(rnd), _ptr(out["path"], i32, "path"), _ptr(out["n_acc"], i32, "n_acc"),
            _ptr(out["next_anchor"], i32, "next_anchor"), _stream(stream))
        _check(code, "dspark_pctree_verify")
        return out

    def verify_rnn(self, P, row_off, lengths, anchor, tokens, pd_tok, lse, U, ovec, W2, seed: int, rnd: int,
                   out=None, stream=None):
        """Verify of RNN-head drafts (``dspark_verify_rnn``): p_d of a rejected
        position from U + o W2 with ovec [B, gamma, r] fp32."""
        out = out or self.new_verify_outputs(P.device)
        f32, i32 = torch.float32, torch.int32
        code = self.lib.dspark_verify_rnn(
            self._h, _ptr(P, f32, "P"), _ptr(row_off, i32, "row_off"), _ptr(lengths, i32, "lengths"),
            _ptr(anchor, i32, "anchor"), _ptr(tokens, i32, "tokens"), _ptr(pd_tok, f32, "pd_tok"),
            _ptr(lse, f32, "lse"), _ptr(U, f32, "U"), _ptr(ovec, f32, "ovec"), _ptr(W2, self.wdtype, "W2"),
            int(seed), int(rnd), _ptr(out["n_acc"], i32, "n_acc"), _ptr(out["next_anchor"], i32, "next_anchor"),
            _stream(stream))
        _check(code, "dspark_verify_rnn")
        return out

    def new_loss_outputs(self, device="cuda") -> Dict[str, torch.Tensor]:
        B, g = self.dims.B, self.dims.gamma
        return {"ce": torch.empty(B, g, dtype=torch.float32, device=device),
                "l1": torch.empty(B, g, dtype=torch.float32, device=device),
                "bce": torch.empty(B, g, dtype=torch.float32, device=device),
                "loss": torch.empty(1, dtype=torch.float64, device=device),
                "scratch": torch.empty(int(self.lib.dspark_train_loss_scratch_bytes(self._h)), dtype=torch.uint8,
                                       device=device)}

    def train_loss(self, U, W1, W2, anchor, xstar, P, conf, tau: float, out=None, stream=None):
        """Teacher-forced training objective (``dspark_train_loss``): U and P
        [B, gamma, V] fp32, xstar and conf [B, gamma]; per-position ce, l1,
        bce and the scalar loss stay on the device."""
        out = out or self.new_loss_outputs(U.device)
        f32, i32 = torch.float32, torch.int32
        code = self.lib.dspark_train_loss(
            self._h, _ptr(U, f32, "U"), _ptr(W1, self.wdtype, "W1"), _ptr(W2, self.wdtype, "W2"),
            _ptr(anchor, i32, "anchor"), _ptr(xstar, i32, "xstar"), _ptr(P, f32, "P"), _ptr(conf, f32, "conf"),
            float(tau), _ptr(out["ce"], f32, "ce"), _ptr(out["l1"], f32, "l1"), _ptr(out["bce"], f32, "bce"),
            _ptr(out["loss"], torch.float64, "loss"), _ptr(out["scratch"], None, "scratch"), _stream(stream))
        _check(code, "dspark_train_loss")
        return out

    def round(self, U, W1, W2, anchor, h, w, T, sps, P, seed: int, rnd: int, out=None, stream=None):
        """draft -> plan -> verify on P packed for this round's lengths."""
        if out is None:
            out = {**self.new_draft_outputs(U.device), **self.new_plan_outputs(U.device),
                   **self.new_verify_outputs(U.device)}
        f32, i32 = torch.float32, torch.int32
        code = self.lib.dspark_round(
            self._h, _ptr(U, f32, "U"), _ptr(W1, self.wdtype, "W1"), _ptr(W2, self.wdtype, "W2"),
            _ptr(anchor, i32, "anchor"), _ptr(h, f32, "h") if self.dims.H > 0 else C.c_void_p(0),
            _ptr(w, f32, "w"), _ptr(T, f32, "T"), _ptr(sps, torch.float64, "sps"), _ptr(P, f32, "P"),
            int(seed), int(rnd), _ptr(out["tokens"], i32, "tokens"), _ptr(out["pd_tok"], f32, "pd_tok"),
            _ptr(out["lse"], f32, "lse"), _ptr(out["conf"], f32, "conf"),
            _ptr(out["lengths"], i32, "lengths"), _ptr(out["row_off"], i32, "row_off"),
            _ptr(out["n_acc"], i32, "n_acc"), _ptr(out["next_anchor"], i32, "next_anchor"),
            _stream(stream))
        _check(code, "dspark_round")
        return out
