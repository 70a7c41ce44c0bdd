"""ctypes binding of libgdn's C ABI (include/gdn.h), with the same entry-point names.

Argument marshalling only: every step of the prefill runs in libgdn's CUDA
kernels.  PyTorch supplies device memory (inputs, outputs, workspace) and the
stream.  If libgdn.so is missing or cannot be loaded, every call raises: there
is no CPU or library fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgdn.so")

GDN_BF16, GDN_F32 = 0, 1
SOLVERS = {"exact": 0, "block_adj": 1}
STATUS = {0: "GDN_OK", 1: "GDN_ERR_NULL", 2: "GDN_ERR_SHAPE", 3: "GDN_ERR_DTYPE", 4: "GDN_ERR_ALIGN",
          5: "GDN_ERR_WORKSPACE", 6: "GDN_ERR_UNSUPPORTED", 7: "GDN_ERR_CUDA", 8: "GDN_ERR_DEVICE",
          9: "GDN_ERR_CAPACITY", 10: "GDN_ERR_TIMEOUT"}
EXPORTS = ("gdn_workspace_bytes", "gdn_select_events", "gdn_events_status", "gdn_prefill_dense",
           "gdn_prefill_sparse", "gdn_workspace_status", "gdn_status_string", "gdn_version",
           "gdn_profile_enable", "gdn_profile_read", "gdn_prefill_sparse_noalloc", "gdn_selftest_wait_timeout",
           "gdn_prefill_sparse_online", "gdn_select_events_scored", "gdn_select_scored_workspace_bytes",
           "gdn_prefill_host", "gdn_prefill_host_workspace_bytes", "gdn_decode_step", "gdn_prefill_ex",
           "gdn_workspace_bytes_ex", "gdn_events_bytes", "gdn_events_carve", "gdn_noalloc_status",
           "gdn_select_events_gamma")
STAGES = ("select", "prefix", "intra", "wbuild", "scan_runs", "scan_chain", "scan", "output", "selector")


class GdnError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({msg})")
        self.status = status


class GdnShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("Nq", ctypes.c_int32), ("Nv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("dv", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class GdnOptions(ctypes.Structure):
    _fields_ = [("tail_window", ctypes.c_int32), ("w_deferred", ctypes.c_int32), ("scan_runs", ctypes.c_int32),
                ("scan_full", ctypes.c_int32), ("states_expanded", ctypes.c_int32), ("online_split", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 2)]


MODES = {"dense": 0, "sparse": 1, "online": 2}


class GdnEvents(ctypes.Structure):
    _fields_ = [("row_pair", ctypes.c_void_p), ("row_ptr", ctypes.c_void_p), ("ev_chunk", ctypes.c_void_p),
                ("grp_pred", ctypes.c_void_p), ("snap_slot", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("capacity", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def load(path: str | None = None):
    """Load libgdn.so (raises if it is absent: build it with gated_delta_rule_16_gb300.build)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libgdn.so not found at {p}; run `python -m gated_delta_rule_16_gb300.build`")
            lib = ctypes.CDLL(p)
            vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
            shp = ctypes.POINTER(GdnShape)
            evp = ctypes.POINTER(GdnEvents)
            lib.gdn_workspace_bytes.argtypes = [shp, i32, i32]
            lib.gdn_workspace_bytes.restype = sz
            lib.gdn_workspace_bytes_ex.argtypes = [shp, i32, i32, ctypes.POINTER(GdnOptions)]
            lib.gdn_workspace_bytes_ex.restype = sz
            lib.gdn_events_bytes.argtypes = [shp, ctypes.c_int32]
            lib.gdn_events_bytes.restype = sz
            lib.gdn_events_carve.argtypes = [shp, ctypes.c_int32, vp, evp]
            lib.gdn_events_carve.restype = i32
            lib.gdn_select_events.argtypes = [shp, vp, evp, vp]
            lib.gdn_select_events.restype = i32
            lib.gdn_events_status.argtypes = [evp, vp]
            lib.gdn_events_status.restype = i32
            lib.gdn_prefill_dense.argtypes = [shp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, vp]
            lib.gdn_prefill_dense.restype = i32
            lib.gdn_prefill_sparse.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, vp]
            lib.gdn_prefill_sparse.restype = i32
            lib.gdn_prefill_sparse_online.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp,
                                                      vp, sz, vp]
            lib.gdn_prefill_sparse_online.restype = i32
            lib.gdn_select_events_scored.argtypes = [shp, vp, vp, vp, vp, vp, vp, sz, vp]
            lib.gdn_select_events_scored.restype = i32
            lib.gdn_select_events_gamma.argtypes = [shp, vp, vp, vp, vp, vp, vp, sz, vp]
            lib.gdn_select_events_gamma.restype = i32
            lib.gdn_select_scored_workspace_bytes.argtypes = [shp]
            lib.gdn_select_scored_workspace_bytes.restype = sz
            lib.gdn_prefill_ex.argtypes = [shp, i32, vp, vp, vp, vp, vp, vp, vp, vp, i32, ctypes.POINTER(GdnOptions),
                                           vp, vp, vp, vp, vp, vp, sz, vp]
            lib.gdn_prefill_ex.restype = i32
            lib.gdn_decode_step.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.gdn_decode_step.restype = i32
            lib.gdn_prefill_host.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
            lib.gdn_prefill_host.restype = i32
            lib.gdn_prefill_host_workspace_bytes.argtypes = [shp, i32, i32]
            lib.gdn_prefill_host_workspace_bytes.restype = sz
            lib.gdn_prefill_sparse_noalloc.argtypes = [shp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp]
            lib.gdn_prefill_sparse_noalloc.restype = i32
            lib.gdn_noalloc_status.argtypes = [vp]
            lib.gdn_noalloc_status.restype = i32
            lib.gdn_selftest_wait_timeout.argtypes = [vp, i32, vp]
            lib.gdn_selftest_wait_timeout.restype = i32
            lib.gdn_workspace_status.argtypes = [vp, vp]
            lib.gdn_workspace_status.restype = i32
            lib.gdn_status_string.argtypes = [i32]
            lib.gdn_status_string.restype = ctypes.c_char_p
            lib.gdn_version.argtypes = []
            lib.gdn_version.restype = ctypes.c_int32
            lib.gdn_profile_enable.argtypes = [i32]
            lib.gdn_profile_enable.restype = i32
            lib.gdn_profile_read.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_int32,
                                             ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)]
            lib.gdn_profile_read.restype = i32
            _lib = lib
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        raise GdnError(fn, status, load().gdn_status_string(status).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def shape_of(q: torch.Tensor, v: torch.Tensor) -> GdnShape:
    B, T, Nq, d = q.shape
    return GdnShape(B, T, Nq, v.shape[2], d, v.shape[3], _dtype_code(q))


def _need(t, name, dtype=None, shape=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def gdn_workspace_bytes(shape: GdnShape, solver: str = "block_adj", sparse: int = 1) -> int:
    """sparse: 0 dense, 1 sparse with a given mask, 2 sparse with online selection."""
    return int(load().gdn_workspace_bytes(ctypes.byref(shape), SOLVERS[solver], int(sparse)))


class Workspace:
    """A reusable device workspace (a torch uint8 buffer) sized by gdn_workspace_bytes."""

    def __init__(self):
        self.buf = None

    def get(self, nbytes: int, device) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != torch.device(device):
            self.buf = None
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        return self.buf


_default_ws = {}


def _workspace(ws, nbytes, device):
    if ws is None:
        key = torch.device(device)
        ws = _default_ws.setdefault(key, Workspace())
    if isinstance(ws, Workspace):
        return ws.get(nbytes, device)
    return ws


def _prefill(fn, q, k, v, beta, g, mask, h0, solver, o, s_final, score, workspace, stream):
    B, T, Nq, d = q.shape
    Nv, dv = v.shape[2], v.shape[3]
    C = (T + 63) // 64
    _need(q, "q", shape=(B, T, Nq, d))
    _need(k, "k", dtype=q.dtype, shape=(B, T, Nq, d))
    _need(v, "v", dtype=q.dtype, shape=(B, T, Nv, dv))
    _need(beta, "beta", torch.float32, (B, T, Nv))
    _need(g, "g", torch.float32, (B, T, Nv))
    _need(h0, "h0", torch.float32, (B, Nv, d, dv))
    if mask is not None:
        _need(mask, "mask", torch.uint8, (B, Nv // 2, C))
    dev = q.device
    if o is None:
        o = torch.empty((B, T, Nv, dv), dtype=q.dtype, device=dev)
    if s_final is None:
        s_final = torch.empty((B, Nv, d, dv), dtype=torch.float32, device=dev)
    _need(o, "o", q.dtype, (B, T, Nv, dv))
    _need(s_final, "s_final", torch.float32, (B, Nv, d, dv))
    _need(score, "score", torch.float32, (B, Nv, C))
    shape = shape_of(q, v)
    nbytes = gdn_workspace_bytes(shape, solver, 1 if mask is not None else 0)
    ws = _workspace(workspace, nbytes, dev)
    lib = load()
    args = [ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0)]
    if fn == "gdn_prefill_sparse":
        args.append(_ptr(mask))
    args += [SOLVERS[solver], _ptr(o), _ptr(s_final), _ptr(score), _ptr(ws), ws.numel(), _stream(stream)]
    with torch.cuda.device(dev):
        _check(fn, getattr(lib, fn)(*args))
    return o, s_final


def gdn_prefill_dense(q, k, v, beta, g, *, h0=None, solver="exact", o=None, s_final=None, score=None,
                      workspace=None, stream=None):
    """Dense prefill through the C ABI; returns (o, s_final)."""
    return _prefill("gdn_prefill_dense", q, k, v, beta, g, None, h0, solver, o, s_final, score, workspace, stream)


def gdn_prefill_sparse(q, k, v, beta, g, mask, *, h0=None, solver="block_adj", o=None, s_final=None,
                       score=None, workspace=None, stream=None):
    """Event-sparse prefill through the C ABI; returns (o, s_final)."""
    if mask is None:
        raise ValueError("gdn_prefill_sparse needs an event mask")
    return _prefill("gdn_prefill_sparse", q, k, v, beta, g, mask, h0, solver, o, s_final, score, workspace,
                    stream)


def gdn_prefill_sparse_noalloc(q, k, v, beta, g, mask, *, h0=None, solver="block_adj", o=None, s_final=None,
                               score=None, stream=None):
    """Allocation-free event-sparse prefill (library-owned 64 MiB scratch); returns (o, s_final).

    For callers that cannot allocate device memory; see include/gdn.h.  The
    outputs must be passed in by such callers (o, s_final); when omitted here
    they are created with torch for convenience.
    """
    B, T, Nq, d = q.shape
    Nv, dv = v.shape[2], v.shape[3]
    C = (T + 63) // 64
    _need(q, "q", shape=(B, T, Nq, d))
    _need(k, "k", dtype=q.dtype, shape=(B, T, Nq, d))
    _need(v, "v", dtype=q.dtype, shape=(B, T, Nv, dv))
    _need(beta, "beta", torch.float32, (B, T, Nv))
    _need(g, "g", torch.float32, (B, T, Nv))
    _need(h0, "h0", torch.float32, (B, Nv, d, dv))
    _need(mask, "mask", torch.uint8, (B, Nv // 2, C))
    if o is None:
        o = torch.empty((B, T, Nv, dv), dtype=q.dtype, device=q.device)
    if s_final is None:
        s_final = torch.empty((B, Nv, d, dv), dtype=torch.float32, device=q.device)
    _need(o, "o", q.dtype, (B, T, Nv, dv))
    _need(s_final, "s_final", torch.float32, (B, Nv, d, dv))
    _need(score, "score", torch.float32, (B, Nv, C))
    shape = shape_of(q, v)
    with torch.cuda.device(q.device):
        _check("gdn_prefill_sparse_noalloc", load().gdn_prefill_sparse_noalloc(
            ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0), _ptr(mask),
            SOLVERS[solver], _ptr(o), _ptr(s_final), _ptr(score), _stream(stream)))
    return o, s_final


def gdn_prefill_sparse_online(q, k, v, beta, g, *, h0=None, eta=None, solver="block_adj", o=None,
                              s_final=None, score=None, mask_out=None, tier_out=None, workspace=None, stream=None):
    """Event-sparse prefill that selects its own events (Tail-16 scores, Eqs. 10-14).

    16 head pairs only.  Returns (o, s_final, mask [B,16,C] uint8, tier [B,16] int32).
    """
    B, T, Nq, d = q.shape
    Nv, dv = v.shape[2], v.shape[3]
    C = (T + 63) // 64
    _need(q, "q", shape=(B, T, Nq, d))
    _need(k, "k", dtype=q.dtype, shape=(B, T, Nq, d))
    _need(v, "v", dtype=q.dtype, shape=(B, T, Nv, dv))
    _need(beta, "beta", torch.float32, (B, T, Nv))
    _need(g, "g", torch.float32, (B, T, Nv))
    _need(h0, "h0", torch.float32, (B, Nv, d, dv))
    _need(eta, "eta", torch.float32, (B, Nv))
    dev = q.device
    if o is None:
        o = torch.empty((B, T, Nv, dv), dtype=q.dtype, device=dev)
    if s_final is None:
        s_final = torch.empty((B, Nv, d, dv), dtype=torch.float32, device=dev)
    if mask_out is None:
        mask_out = torch.empty((B, Nq, C), dtype=torch.uint8, device=dev)
    if tier_out is None:
        tier_out = torch.empty((B, Nq), dtype=torch.int32, device=dev)
    _need(o, "o", q.dtype, (B, T, Nv, dv))
    _need(s_final, "s_final", torch.float32, (B, Nv, d, dv))
    _need(score, "score", torch.float32, (B, Nv, C))
    _need(mask_out, "mask_out", torch.uint8, (B, Nq, C))
    _need(tier_out, "tier_out", torch.int32, (B, Nq))
    shape = shape_of(q, v)
    ws = _workspace(workspace, gdn_workspace_bytes(shape, solver, 2), dev)
    with torch.cuda.device(dev):
        _check("gdn_prefill_sparse_online", load().gdn_prefill_sparse_online(
            ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0), _ptr(eta),
            SOLVERS[solver], _ptr(o), _ptr(s_final), _ptr(score), _ptr(mask_out), _ptr(tier_out), _ptr(ws),
            ws.numel(), _stream(stream)))
    return o, s_final, mask_out, tier_out


def gdn_select_events_scored(score: torch.Tensor, g: torch.Tensor, eta=None, *, mask_out=None, tier_out=None,
                             workspace=None, stream=None):
    """Online selection from Tail-16 scores [B,32,C] and gates g [B,T,32]; returns (mask, tier)."""
    _need(score, "score", torch.float32)
    B, Nv, C = score.shape
    _need(g, "g", torch.float32, (B, C * 64, Nv))
    _need(eta, "eta", torch.float32, (B, Nv))
    dev = score.device
    if mask_out is None:
        mask_out = torch.empty((B, Nv // 2, C), dtype=torch.uint8, device=dev)
    if tier_out is None:
        tier_out = torch.empty((B, Nv // 2), dtype=torch.int32, device=dev)
    _need(mask_out, "mask_out", torch.uint8, (B, Nv // 2, C))
    _need(tier_out, "tier_out", torch.int32, (B, Nv // 2))
    shape = GdnShape(B, C * 64, Nv // 2, Nv, 128, 128, GDN_BF16)
    lib = load()
    ws = _workspace(workspace, int(lib.gdn_select_scored_workspace_bytes(ctypes.byref(shape))), dev)
    with torch.cuda.device(dev):
        _check("gdn_select_events_scored", lib.gdn_select_events_scored(
            ctypes.byref(shape), _ptr(score), _ptr(g), _ptr(eta), _ptr(mask_out), _ptr(tier_out), _ptr(ws),
            ws.numel(), _stream(stream)))
    return mask_out, tier_out


def gdn_select_events_gamma(score: torch.Tensor, gamma: torch.Tensor, eta=None, *, mask_out=None, tier_out=None,
                            workspace=None, stream=None):
    """Online selection from Tail-16 scores [B,32,C] and chunk gate tails gamma [B,32,C]
    (g at each chunk's last token); returns (mask, tier)."""
    _need(score, "score", torch.float32)
    B, Nv, C = score.shape
    _need(gamma, "gamma", torch.float32, (B, Nv, C))
    _need(eta, "eta", torch.float32, (B, Nv))
    dev = score.device
    if mask_out is None:
        mask_out = torch.empty((B, Nv // 2, C), dtype=torch.uint8, device=dev)
    if tier_out is None:
        tier_out = torch.empty((B, Nv // 2), dtype=torch.int32, device=dev)
    _need(mask_out, "mask_out", torch.uint8, (B, Nv // 2, C))
    _need(tier_out, "tier_out", torch.int32, (B, Nv // 2))
    shape = GdnShape(B, C * 64, Nv // 2, Nv, 128, 128, GDN_BF16)
    lib = load()
    ws = _workspace(workspace, int(lib.gdn_select_scored_workspace_bytes(ctypes.byref(shape))), dev)
    with torch.cuda.device(dev):
        _check("gdn_select_events_gamma", lib.gdn_select_events_gamma(
            ctypes.byref(shape), _ptr(score), _ptr(gamma), _ptr(eta), _ptr(mask_out), _ptr(tier_out), _ptr(ws),
            ws.numel(), _stream(stream)))
    return mask_out, tier_out


def _need_host(t, name, dtype=None, shape=None):
    if t is None:
        return
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def gdn_prefill_host(q, k, v, beta, g, mask=None, *, h0=None, solver="block_adj", o=None, s_final=None,
                     workspace=None, device="cuda:0", stream=None):
    """Prefill with host (CPU, preferably pinned) inputs and outputs; returns (o, s_final).

    The copies and kernels are enqueued on `stream`; the call does not wait, so
    synchronise the stream before reading the outputs.
    """
    B, T, Nq, d = q.shape
    Nv, dv = v.shape[2], v.shape[3]
    C = (T + 63) // 64
    _need_host(q, "q", shape=(B, T, Nq, d))
    _need_host(k, "k", dtype=q.dtype, shape=(B, T, Nq, d))
    _need_host(v, "v", dtype=q.dtype, shape=(B, T, Nv, dv))
    _need_host(beta, "beta", torch.float32, (B, T, Nv))
    _need_host(g, "g", torch.float32, (B, T, Nv))
    _need_host(h0, "h0", torch.float32, (B, Nv, d, dv))
    _need_host(mask, "mask", torch.uint8, (B, Nq, C))
    if o is None:
        o = torch.empty((B, T, Nv, dv), dtype=q.dtype).pin_memory()
    if s_final is None:
        s_final = torch.empty((B, Nv, d, dv), dtype=torch.float32).pin_memory()
    _need_host(o, "o", q.dtype, (B, T, Nv, dv))
    _need_host(s_final, "s_final", torch.float32, (B, Nv, d, dv))
    shape = shape_of(q, v)
    dev = torch.device(device)
    lib = load()
    nbytes = int(lib.gdn_prefill_host_workspace_bytes(ctypes.byref(shape), SOLVERS[solver], int(mask is not None)))
    ws = _workspace(workspace, nbytes, dev)
    with torch.cuda.device(dev):
        _check("gdn_prefill_host", lib.gdn_prefill_host(
            ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0), _ptr(mask),
            SOLVERS[solver], _ptr(o), _ptr(s_final), _ptr(ws), ws.numel(), _stream(stream)))
    return o, s_final


def gdn_prefill_ex(q, k, v, beta, g, *, mode="sparse", mask=None, h0=None, eta=None, solver="block_adj",
                   tail_window=0, w_deferred=False, scan_runs=False, scan_full=False, states_expanded=False,
                   online_split=0, o=None, s_final=None, score=None, mask_out=None,
                   tier_out=None, workspace=None, stream=None):
    """The general prefill with execution variants; returns (o, s_final, mask_out, tier_out)."""
    B, T, Nq, d = q.shape
    Nv, dv = v.shape[2], v.shape[3]
    C = (T + 63) // 64
    _need(q, "q", shape=(B, T, Nq, d))
    _need(k, "k", dtype=q.dtype, shape=(B, T, Nq, d))
    _need(v, "v", dtype=q.dtype, shape=(B, T, Nv, dv))
    _need(beta, "beta", torch.float32, (B, T, Nv))
    _need(g, "g", torch.float32, (B, T, Nv))
    _need(h0, "h0", torch.float32, (B, Nv, d, dv))
    _need(mask, "mask", torch.uint8, (B, Nq, C))
    _need(eta, "eta", torch.float32, (B, Nv))
    dev = q.device
    if o is None:
        o = torch.empty((B, T, Nv, dv), dtype=q.dtype, device=dev)
    if s_final is None:
        s_final = torch.empty((B, Nv, d, dv), dtype=torch.float32, device=dev)
    if mode == "online" and not online_split:
        if mask_out is None:
            mask_out = torch.empty((B, Nq, C), dtype=torch.uint8, device=dev)
        if tier_out is None:
            tier_out = torch.empty((B, Nq), dtype=torch.int32, device=dev)
    _need(score, "score", torch.float32, (B, Nv, C))
    shape = shape_of(q, v)
    opt = GdnOptions(int(tail_window), int(bool(w_deferred)), int(bool(scan_runs)), int(bool(scan_full)),
                     int(bool(states_expanded)), int(online_split))
    nbytes = int(load().gdn_workspace_bytes_ex(ctypes.byref(shape), SOLVERS[solver], MODES[mode], ctypes.byref(opt)))
    if nbytes == 0:
        raise GdnError("gdn_workspace_bytes_ex", 2, "invalid shape or options")
    ws = _workspace(workspace, nbytes, dev)
    with torch.cuda.device(dev):
        _check("gdn_prefill_ex", load().gdn_prefill_ex(
            ctypes.byref(shape), MODES[mode], _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0), _ptr(mask),
            _ptr(eta), SOLVERS[solver], ctypes.byref(opt), _ptr(o), _ptr(s_final), _ptr(score), _ptr(mask_out),
            _ptr(tier_out), _ptr(ws), ws.numel(), _stream(stream)))
    return o, s_final, mask_out, tier_out


def gdn_decode_step(q, k, v, beta, a, state, *, o=None, stream=None):
    """One decode step: q, k [B,Nq,d], v [B,Nv,dv], beta and a [B,Nv] fp32, state [B,Nv,d,dv] fp32
    (updated in place).  Returns o [B,Nv,dv] in q's dtype."""
    B, Nq, d = q.shape
    Nv, dv = v.shape[1], v.shape[2]
    _need(q, "q", shape=(B, Nq, d))
    _need(k, "k", dtype=q.dtype, shape=(B, Nq, d))
    _need(v, "v", dtype=q.dtype, shape=(B, Nv, dv))
    _need(beta, "beta", torch.float32, (B, Nv))
    _need(a, "a", torch.float32, (B, Nv))
    _need(state, "state", torch.float32, (B, Nv, d, dv))
    if o is None:
        o = torch.empty((B, Nv, dv), dtype=q.dtype, device=q.device)
    _need(o, "o", q.dtype, (B, Nv, dv))
    shape = GdnShape(B, 1, Nq, Nv, d, dv, _dtype_code(q))
    with torch.cuda.device(q.device):
        _check("gdn_decode_step", load().gdn_decode_step(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                                         _ptr(a), _ptr(state), _ptr(o), _stream(stream)))
    return o


def gdn_select_events(mask: torch.Tensor, Nq: int | None = None, capacity: int | None = None, stream=None):
    """Mask [B,P,C] uint8 -> CSR event lists on the device (dict of int32 tensors, views of one
    buffer sized by gdn_events_bytes and laid out by gdn_events_carve)."""
    _need(mask, "mask", torch.uint8)
    B, P, C = mask.shape
    G = (C + 1) // 2
    cap = B * P * C if capacity is None else int(capacity)
    dev = mask.device
    shape = GdnShape(B, C * 64, P, 2 * P, 128, 128, GDN_BF16)
    lib = load()
    nbytes = int(lib.gdn_events_bytes(ctypes.byref(shape), cap))
    if nbytes == 0:
        raise GdnError("gdn_events_bytes", 2, "invalid shape or capacity")
    buf = torch.zeros(nbytes + 256, dtype=torch.uint8, device=dev)
    base = buf.data_ptr()
    pad = (-base) % 256
    ev = GdnEvents()
    _check("gdn_events_carve", lib.gdn_events_carve(ctypes.byref(shape), cap, ctypes.c_void_p(base + pad),
                                                    ctypes.byref(ev)))
    view = lambda ptr, n: buf[ptr - base:ptr - base + 4 * n].view(torch.int32)
    out = {"row_pair": view(ev.row_pair, B * P), "row_ptr": view(ev.row_ptr, B * P + 1),
           "ev_chunk": view(ev.ev_chunk, cap), "grp_pred": view(ev.grp_pred, B * P * G),
           "snap_slot": view(ev.snap_slot, cap), "counts": view(ev.counts, 4), "_buf": buf}
    with torch.cuda.device(dev):
        _check("gdn_select_events", lib.gdn_select_events(ctypes.byref(shape), _ptr(mask), ctypes.byref(ev),
                                                          _stream(stream)))
    out["_struct"] = ev
    return out


def gdn_events_status(events: dict, stream=None) -> int:
    return int(load().gdn_events_status(ctypes.byref(events["_struct"]), _stream(stream)))


def gdn_noalloc_status(device="cuda:0", stream=None) -> int:
    """Status of the last allocation-free prefill on `device` (synchronises the stream)."""
    with torch.cuda.device(torch.device(device)):
        return int(load().gdn_noalloc_status(_stream(stream)))


def gdn_workspace_status(workspace, stream=None) -> int:
    buf = workspace.buf if isinstance(workspace, Workspace) else workspace
    return int(load().gdn_workspace_status(_ptr(buf), _stream(stream)))


def gdn_selftest_wait_timeout(limit_ms: int = 50, device="cuda:0", stream=None):
    """Run the bounded-wait self-test; returns (status code, milliseconds waited, status bits)."""
    st = torch.zeros(4, dtype=torch.int32, device=device)
    with torch.cuda.device(st.device):
        rc = int(load().gdn_selftest_wait_timeout(_ptr(st), int(limit_ms), _stream(stream)))
    host = st.cpu().tolist()
    return rc, host[3], host[2]


def gdn_version() -> int:
    return int(load().gdn_version())


def gdn_profile_enable(enable=True) -> None:
    """True / 1: record per-stage CUDA events in the following prefills (one-stream schedule);
    2: only count the kernels they launch (their normal schedule); False / 0: off (include/gdn.h)."""
    _check("gdn_profile_enable", load().gdn_profile_enable(int(enable)))


def gdn_profile_read(with_launches: bool = False):
    """Summed milliseconds per stage over the recorded prefills and their count
    (and, with_launches, the number of kernels they launched)."""
    ms = (ctypes.c_float * len(STAGES))()
    n = ctypes.c_int32(0)
    nl = ctypes.c_int64(0)
    _check("gdn_profile_read", load().gdn_profile_read(ms, len(STAGES), ctypes.byref(n), ctypes.byref(nl)))
    stages = {name: float(ms[i]) for i, name in enumerate(STAGES)}
    return (stages, int(n.value), int(nl.value)) if with_launches else (stages, int(n.value))
