"""Thin Python binding of libdustin.so (ctypes).

Argument marshalling only: every function here checks shapes and dtypes of
torch tensors, builds the C structs of ``include/dustin.h`` and calls the
entry point of the same name.  All work runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback.  If the library has not been built, or
a call returns an error status, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_int32, c_int64, c_size_t, c_void_p
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdustin.so")

STATUS = {0: "DUSTIN_OK", -1: "DUSTIN_EINVAL", -2: "DUSTIN_ERANGE", -3: "DUSTIN_ECUDA",
          -4: "DUSTIN_EDEVICE", -5: "DUSTIN_EWORKSPACE"}
DEV_INDEX, DEV_NAN, DEV_APPEND, DEV_TIMEOUT, DEV_SEQLEN = 1, 2, 4, 8, 16
MAX_SRH, MAX_PAIRS, MAX_LAYERS, MAX_QROWS, MAX_LCAP = 32, 32, 16, 128, 1 << 20

EXPORTS = ["dustin_version", "dustin_workspace_bytes", "dustin_workspace_init", "dustin_check",
           "dustin_score", "dustin_select", "dustin_verify_attn", "dense_verify_attn",
           "dustin_kv_append", "dustin_verify_step", "dustin_step_launches", "dustin_compact_kv",
           "dustin_score_noalloc", "dustin_score_noalloc_check", "dustin_wait_selftest",
           "dustin_verify_split"]


class DustinError(RuntimeError):
    def __init__(self, fn: str, status: int, flags: int = 0):
        self.status = status
        self.flags = flags
        msg = f"{fn} returned {STATUS.get(status, status)}"
        if flags:
            msg += f" (device flags 0x{flags:x})"
        super().__init__(msg)


# ------------------------------------------------------------------ structs


class CKV(ctypes.Structure):
    _fields_ = [("ptr", c_void_p), ("hkv", c_int32), ("d", c_int32),
                ("sb", c_int64), ("sh", c_int64), ("sl", c_int64)]


class CParams(ctypes.Structure):
    _fields_ = [("B", c_int32), ("Lcap", c_int32), ("gamma", c_int32), ("sinks", c_int32),
                ("window", c_int32), ("m", c_int32), ("k", c_int32)]


class CSignal(ctypes.Structure):
    _fields_ = [("n_layers", c_int32), ("hq", c_int32), ("nq", c_int32),
                ("q", POINTER(c_void_p)), ("k", POINTER(CKV))]


class CSRH(ctypes.Structure):
    _fields_ = [("channel", c_int32), ("layer", c_int32), ("q_head", c_int32)]


class CVerifyLayer(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", CKV), ("v", CKV), ("kb", c_void_p), ("vb", c_void_p),
                ("o", c_void_p)]


class CStep(ctypes.Structure):
    _fields_ = [("p", CParams), ("draft", POINTER(CSignal)), ("target", POINTER(CSignal)),
                ("srh", POINTER(CSRH)), ("n_srh", c_int32), ("hq", c_int32),
                ("n_layers", c_int32), ("layers", POINTER(CVerifyLayer)),
                ("seq_len", c_void_p), ("importance", c_void_p), ("i_verify", c_void_p),
                ("stage_events", POINTER(c_void_p))]


_lib_handle = None


def lib():
    """The loaded libdustin.so (raises if it has not been built)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m sparse_kv_verify_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        L.dustin_version.restype = c_char_p
        L.dustin_workspace_bytes.restype = c_size_t
        L.dustin_workspace_bytes.argtypes = [POINTER(CParams), POINTER(CSignal), POINTER(CSignal),
                                             POINTER(CSRH), c_int32, c_int32, c_int32, c_int32,
                                             c_int32]
        L.dustin_workspace_init.argtypes = [c_void_p, c_size_t, c_void_p]
        L.dustin_check.argtypes = [c_void_p, c_void_p, POINTER(c_int32)]
        L.dustin_score.argtypes = [POINTER(CParams), POINTER(CSignal), POINTER(CSignal),
                                   POINTER(CSRH), c_int32, c_void_p, c_void_p, c_void_p,
                                   c_size_t, c_void_p]
        L.dustin_select.argtypes = [POINTER(CParams), c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_size_t, c_void_p]
        L.dustin_verify_attn.argtypes = [POINTER(CParams), c_int32, c_void_p, CKV, CKV, c_void_p,
                                         c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_size_t, c_void_p]
        L.dense_verify_attn.argtypes = [POINTER(CParams), c_int32, c_void_p, CKV, CKV, c_void_p,
                                        c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                        c_void_p]
        L.dustin_kv_append.argtypes = [POINTER(CParams), c_int32, POINTER(CKV), POINTER(CKV),
                                       POINTER(c_void_p), POINTER(c_void_p), c_void_p, c_void_p,
                                       c_void_p, c_size_t, c_void_p]
        L.dustin_verify_step.argtypes = [POINTER(CStep), c_void_p, c_size_t, c_void_p]
        L.dustin_step_launches.argtypes = [POINTER(CStep), POINTER(c_int32), POINTER(c_int32)]
        L.dustin_compact_kv.argtypes = [POINTER(CParams), c_int32, POINTER(CKV), POINTER(CKV),
                                        c_void_p, c_void_p, POINTER(CKV), POINTER(CKV), c_void_p,
                                        c_void_p, c_size_t, c_void_p]
        L.dustin_score_noalloc.argtypes = [POINTER(CParams), POINTER(CSignal), POINTER(CSignal),
                                           POINTER(CSRH), c_int32, c_void_p, c_void_p, c_void_p]
        L.dustin_score_noalloc_check.argtypes = [c_void_p, POINTER(c_int32)]
        L.dustin_verify_split.argtypes = [POINTER(CParams), c_int32, c_int32, c_int32, c_int32,
                                          c_int32, POINTER(c_int32), POINTER(c_int32)]
        L.dustin_wait_selftest.argtypes = [ctypes.c_int64, c_void_p, c_void_p, c_size_t, c_void_p]
        for f in EXPORTS[1:]:
            if f != "dustin_workspace_bytes":
                getattr(L, f).restype = ctypes.c_int
        _lib_handle = L
    return _lib_handle


def version() -> str:
    return lib().dustin_version().decode()


# ------------------------------------------------------------------ python-side types


@dataclass
class Params:
    B: int
    Lcap: int
    gamma: int
    sinks: int
    window: int
    m: int
    k: int

    def c(self) -> CParams:
        return CParams(self.B, self.Lcap, self.gamma, self.sinks, self.window, self.m, self.k)


@dataclass
class Signal:
    """One scoring signal: per-layer queries ``[B][nq][hq][d]`` (None where a
    layer holds no SRH) and per-layer key caches ``[B][hkv][Lcap][d]``."""
    q: Sequence[Optional[torch.Tensor]]
    k: Sequence[torch.Tensor]

    def c(self):
        qs = next(t for t in self.q if t is not None)
        n = len(self.k)
        qarr = (c_void_p * n)(*[(_ptr(t, torch.bfloat16) if t is not None else None) for t in self.q])
        karr = (CKV * n)(*[kv_view(t) for t in self.k])
        s = CSignal(n, qs.shape[2], qs.shape[1], qarr, karr)
        s._keep = (qarr, karr)
        return s


def _ptr(t: torch.Tensor, dtype, contiguous: bool = True) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if contiguous and not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def kv_view(t: torch.Tensor) -> CKV:
    """C view of a bf16 cache tensor ``[B][hkv][Lcap][d]`` (rows contiguous)."""
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("cache must be [B][hkv][Lcap][d] with contiguous rows")
    _ptr(t, torch.bfloat16, contiguous=False)
    return CKV(t.data_ptr(), t.shape[1], t.shape[3], t.stride(0), t.stride(1), t.stride(2))


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(fn: str, st: int):
    if st != 0:
        raise DustinError(fn, st)


def _srh_array(srh):
    arr = (CSRH * len(srh))(*[CSRH(int(c), int(l), int(h)) for (c, l, h) in srh])
    return arr


class Workspace:
    """Caller-owned device scratch of ``dustin_workspace_bytes`` bytes."""

    def __init__(self, nbytes: int, device=None, stream=None):
        nbytes = max(256, int(nbytes))
        self.buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=device or "cuda")
        base = self.buf.data_ptr()
        self.off = (-base) % 256
        self.ptr = base + self.off
        self.nbytes = nbytes
        _check("dustin_workspace_init", lib().dustin_workspace_init(self.ptr, nbytes, _stream(stream)))


def workspace_bytes(p: Params, draft: Optional[Signal] = None, target: Optional[Signal] = None,
                    srh=(), verify=None) -> int:
    """Workspace bytes for scoring with ``srh`` and/or verifying with
    ``verify = (hq, hkv, d, n_layers)``."""
    cp = p.c()
    hq, hkv, d, nl = verify if verify is not None else (0, 0, 0, 0)
    if srh:
        dc = draft.c() if draft is not None else None
        tc = target.c() if target is not None else None
        arr = _srh_array(srh)
        n = lib().dustin_workspace_bytes(ctypes.byref(cp), ctypes.byref(dc) if dc else None,
                                         ctypes.byref(tc) if tc else None, arr, len(srh),
                                         hq, hkv, d, nl)
    else:
        n = lib().dustin_workspace_bytes(ctypes.byref(cp), None, None, None, 0, hq, hkv, d, nl)
    if n == 0:
        raise DustinError("dustin_workspace_bytes", -1)
    return int(n)


def workspace(p: Params, draft=None, target=None, srh=(), verify=None, device=None,
              stream=None) -> Workspace:
    return Workspace(workspace_bytes(p, draft, target, srh, verify), device=device, stream=stream)


def _verify_shape(q, k, n_layers=1):
    return (q.shape[2], k.shape[1], k.shape[3], n_layers)


def check(ws: Workspace, stream=None) -> int:
    """Synchronises the stream; returns the device error flags (and clears them)."""
    flags = c_int32(0)
    st = lib().dustin_check(ws.ptr, _stream(stream), ctypes.byref(flags))
    if st not in (0, -4):
        raise DustinError("dustin_check", st)
    return int(flags.value)


# ------------------------------------------------------------------ entry points


def dustin_score(p: Params, draft: Signal, target: Signal, srh, seq_len: torch.Tensor,
                 importance: Optional[torch.Tensor] = None, ws: Optional[Workspace] = None,
                 stream=None) -> torch.Tensor:
    dev = seq_len.device
    if importance is None:
        importance = torch.empty((p.B, 2, p.Lcap), dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(p, draft, target, srh, device=dev, stream=stream)
    d, t = draft.c(), target.c()
    arr = _srh_array(srh)
    st = lib().dustin_score(ctypes.byref(p.c()), ctypes.byref(d), ctypes.byref(t), arr, len(srh),
                            _ptr(seq_len, torch.int32), _ptr(importance, torch.float32),
                            ws.ptr, ws.nbytes, _stream(stream))
    _check("dustin_score", st)
    return importance


def dustin_score_noalloc(p: Params, draft: Signal, target: Signal, srh, seq_len: torch.Tensor,
                         importance: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """dustin_score with the library's own static scratch (no workspace).

    For callers that cannot allocate device memory when they score; the
    library keeps one 16 MiB scratch array per GPU, shared by all calls (calls
    that overlap on the GPU race on it)."""
    if importance is None:
        raise ValueError("pass a preallocated importance tensor [B][2][Lcap] fp32")
    d, t = draft.c(), target.c()
    arr = _srh_array(srh)
    st = lib().dustin_score_noalloc(ctypes.byref(p.c()), ctypes.byref(d), ctypes.byref(t), arr,
                                    len(srh), _ptr(seq_len, torch.int32),
                                    _ptr(importance, torch.float32), _stream(stream))
    _check("dustin_score_noalloc", st)
    return importance


def verify_split(p: Params, hq: int, hkv: int, d: int, n_layers: int = 1, dense: bool = False):
    """The verification kernel's stream-K split on the current device:
    (grid, tiles_per_unit); CTA c takes tiles [c*T/grid, (c+1)*T/grid) of the
    T = B * hkv * n_layers * tiles_per_unit tiles."""
    grid, tiles = c_int32(0), c_int32(0)
    st = lib().dustin_verify_split(ctypes.byref(p.c()), hq, hkv, d, n_layers, int(dense),
                                   ctypes.byref(grid), ctypes.byref(tiles))
    _check("dustin_verify_split", st)
    return int(grid.value), int(tiles.value)


def split_units(p: Params, hkv: int, n_layers: int, grid: int, tiles_per_unit: int):
    """Units u whose tiles the split gives to more than one CTA."""
    total = p.B * hkv * n_layers * tiles_per_unit

    def cta_of(x):   # the CTA c with c*total//grid <= x < (c+1)*total//grid
        return ((x + 1) * grid + total - 1) // total - 1

    return [u for u in range(p.B * hkv * n_layers)
            if cta_of(u * tiles_per_unit) != cta_of(u * tiles_per_unit + tiles_per_unit - 1)]


def wait_selftest(limit_ns: int, ws: "Workspace", stream=None) -> torch.Tensor:
    """Runs the bounded-wait self-test; returns the two waiters' times (ns)
    as a device int64 tensor.  Read the error word with check(ws)."""
    waited = torch.zeros(2, dtype=torch.int64, device=ws.buf.device)
    st = lib().dustin_wait_selftest(int(limit_ns), waited.data_ptr(), ws.ptr, ws.nbytes,
                                    _stream(stream))
    _check("dustin_wait_selftest", st)
    return waited


def noalloc_check(stream=None) -> int:
    """Synchronises the stream; returns (and clears) the device error flags
    that dustin_score_noalloc calls raised since the last check."""
    flags = c_int32(0)
    st = lib().dustin_score_noalloc_check(_stream(stream), ctypes.byref(flags))
    if st not in (0, -4):
        raise DustinError("dustin_score_noalloc_check", st)
    return int(flags.value)


def dustin_select(p: Params, importance: torch.Tensor, seq_len: torch.Tensor,
                  i_verify: Optional[torch.Tensor] = None, ws: Optional[Workspace] = None,
                  stream=None) -> torch.Tensor:
    if i_verify is None:
        i_verify = torch.empty((p.B, p.k), dtype=torch.int32, device=seq_len.device)
    if ws is None:
        ws = workspace(p, device=seq_len.device, stream=stream)
    st = lib().dustin_select(ctypes.byref(p.c()), _ptr(importance, torch.float32),
                             _ptr(seq_len, torch.int32), _ptr(i_verify, torch.int32), ws.ptr,
                             ws.nbytes, _stream(stream))
    _check("dustin_select", st)
    return i_verify


def _out(o, q):
    if o is None:
        o = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    return o


def dustin_verify_attn(p: Params, q, k, v, kb, vb, i_verify, seq_len, o=None, ws=None,
                       stream=None) -> torch.Tensor:
    o = _out(o, q)
    if ws is None:
        ws = workspace(p, verify=_verify_shape(q, k), device=q.device, stream=stream)
    st = lib().dustin_verify_attn(ctypes.byref(p.c()), q.shape[2], _ptr(q, torch.bfloat16),
                                  kv_view(k), kv_view(v), _ptr(kb, torch.bfloat16),
                                  _ptr(vb, torch.bfloat16), _ptr(i_verify, torch.int32),
                                  _ptr(seq_len, torch.int32), _ptr(o, torch.float32), ws.ptr,
                                  ws.nbytes, _stream(stream))
    _check("dustin_verify_attn", st)
    return o


def dense_verify_attn(p: Params, q, k, v, kb, vb, seq_len, o=None, ws=None,
                      stream=None) -> torch.Tensor:
    o = _out(o, q)
    if ws is None:
        ws = workspace(p, verify=_verify_shape(q, k), device=q.device, stream=stream)
    st = lib().dense_verify_attn(ctypes.byref(p.c()), q.shape[2], _ptr(q, torch.bfloat16),
                                 kv_view(k), kv_view(v), _ptr(kb, torch.bfloat16),
                                 _ptr(vb, torch.bfloat16), _ptr(seq_len, torch.int32),
                                 _ptr(o, torch.float32), ws.ptr, ws.nbytes, _stream(stream))
    _check("dense_verify_attn", st)
    return o


def dustin_compact_kv(p: Params, ks, vs, i_verify, seq_len, kcs=None, vcs=None, seq_len_c=None,
                      ws=None, stream=None):
    """Copies the selected rows of every layer's caches into compact caches
    [B][hkv][k][d]; returns (kcs, vcs, seq_len_c)."""
    n = len(ks)
    if kcs is None:
        kcs = [torch.empty((p.B, t.shape[1], p.k, t.shape[3]), dtype=t.dtype, device=t.device) for t in ks]
    if vcs is None:
        vcs = [torch.empty((p.B, t.shape[1], p.k, t.shape[3]), dtype=t.dtype, device=t.device) for t in vs]
    if seq_len_c is None:
        seq_len_c = torch.empty_like(seq_len)
    arr = lambda ts: (CKV * n)(*[kv_view(t) for t in ts])
    if ws is None:
        ws = workspace(p, device=seq_len.device, stream=stream)
    st = lib().dustin_compact_kv(ctypes.byref(p.c()), n, arr(ks), arr(vs), _ptr(i_verify, torch.int32),
                                 _ptr(seq_len, torch.int32), arr(kcs), arr(vcs),
                                 _ptr(seq_len_c, torch.int32), ws.ptr, ws.nbytes, _stream(stream))
    _check("dustin_compact_kv", st)
    return kcs, vcs, seq_len_c


def dustin_kv_append(p: Params, ks, vs, kbs, vbs, n_accept, seq_len, ws=None, stream=None):
    n = len(ks)
    karr = (CKV * n)(*[kv_view(t) for t in ks])
    varr = (CKV * n)(*[kv_view(t) for t in vs])
    kbarr = (c_void_p * n)(*[_ptr(t, torch.bfloat16) for t in kbs])
    vbarr = (c_void_p * n)(*[_ptr(t, torch.bfloat16) for t in vbs])
    if ws is None:
        ws = workspace(p, device=seq_len.device, stream=stream)
    st = lib().dustin_kv_append(ctypes.byref(p.c()), n, karr, varr, kbarr, vbarr,
                                _ptr(n_accept, torch.int32), _ptr(seq_len, torch.int32), ws.ptr,
                                ws.nbytes, _stream(stream))
    _check("dustin_kv_append", st)


class AppendCall:
    """Pre-marshalled arguments of dustin_kv_append, reusable across calls
    (the tensors it points to must stay alive and in place)."""

    def __init__(self, p: Params, ks, vs, kbs, vbs, n_accept, seq_len, ws=None, stream=None):
        n = len(ks)
        self._p = p.c()
        self._n = n
        self._k = (CKV * n)(*[kv_view(t) for t in ks])
        self._v = (CKV * n)(*[kv_view(t) for t in vs])
        self._kb = (c_void_p * n)(*[_ptr(t, torch.bfloat16) for t in kbs])
        self._vb = (c_void_p * n)(*[_ptr(t, torch.bfloat16) for t in vbs])
        self._acc = _ptr(n_accept, torch.int32)
        self._seq = _ptr(seq_len, torch.int32)
        self.ws = ws if ws is not None else workspace(p, device=seq_len.device, stream=stream)

    def __call__(self, stream=None):
        st = lib().dustin_kv_append(ctypes.byref(self._p), self._n, self._k, self._v, self._kb,
                                    self._vb, self._acc, self._seq, self.ws.ptr, self.ws.nbytes,
                                    _stream(stream))
        _check("dustin_kv_append", st)


@dataclass
class VerifyLayer:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    kb: torch.Tensor
    vb: torch.Tensor
    o: Optional[torch.Tensor] = None


class StepCall:
    """Pre-marshalled arguments of dustin_verify_step, reusable across calls
    (the tensors it points to must stay alive and in place)."""

    def __init__(self, p: Params, draft: Signal, target: Signal, srh, layers: Sequence[VerifyLayer],
                 seq_len, importance=None, i_verify=None, ws=None, events=None, stream=None):
        dev = seq_len.device
        self.importance = importance if importance is not None else torch.empty(
            (p.B, 2, p.Lcap), dtype=torch.float32, device=dev)
        self.i_verify = i_verify if i_verify is not None else torch.empty(
            (p.B, p.k), dtype=torch.int32, device=dev)
        for Lr in layers:
            Lr.o = _out(Lr.o, Lr.q)
        self.layers = list(layers)
        self.ws = ws if ws is not None else workspace(
            p, draft, target, srh, verify=_verify_shape(layers[0].q, layers[0].k, len(layers)),
            device=dev, stream=stream)
        self._d, self._t = draft.c(), target.c()
        self._srh = _srh_array(srh)
        self._larr = (CVerifyLayer * len(layers))(*[
            CVerifyLayer(_ptr(Lr.q, torch.bfloat16), kv_view(Lr.k), kv_view(Lr.v),
                         _ptr(Lr.kb, torch.bfloat16), _ptr(Lr.vb, torch.bfloat16),
                         _ptr(Lr.o, torch.float32)) for Lr in layers])
        self.step = CStep(p.c(), ctypes.pointer(self._d), ctypes.pointer(self._t), self._srh,
                          len(srh), layers[0].q.shape[2], len(layers), self._larr,
                          _ptr(seq_len, torch.int32), _ptr(self.importance, torch.float32),
                          _ptr(self.i_verify, torch.int32), None)
        self.events = events

    def launches(self):
        """(kernels one call launches, sequences per scoring group)."""
        n, g = c_int32(0), c_int32(0)
        _check("dustin_step_launches",
               lib().dustin_step_launches(ctypes.byref(self.step), ctypes.byref(n), ctypes.byref(g)))
        return n.value, g.value

    def __call__(self, stream=None, events=None):
        """Runs the step.  ``events``: optional 5 torch.cuda.Event(enable_timing=True)
        recorded before score, after the first scoring group's stream kernel,
        after all score kernels, after select and after verify."""
        ev = events if events is not None else self.events
        if ev is not None:
            for e in ev:
                if not e.cuda_event:      # torch creates the CUDA event on first record
                    e.record(stream if stream is not None else torch.cuda.current_stream())
            arr = (c_void_p * 5)(*[e.cuda_event for e in ev])
            self.step.stage_events = ctypes.cast(arr, POINTER(c_void_p))
        else:
            arr = None
            self.step.stage_events = None
        st = lib().dustin_verify_step(ctypes.byref(self.step), self.ws.ptr, self.ws.nbytes,
                                      _stream(stream))
        _check("dustin_verify_step", st)
        return self.importance, self.i_verify, [Lr.o for Lr in self.layers]


def dustin_verify_step(p: Params, draft: Signal, target: Signal, srh, layers, seq_len,
                       importance=None, i_verify=None, ws=None, events=None, stream=None):
    return StepCall(p, draft, target, srh, layers, seq_len, importance, i_verify, ws, events,
                    stream)(stream)
