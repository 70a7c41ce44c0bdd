"""CPU fp64 oracle of the chunkwise gated-delta prefill core (dense and event-sparse).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``.  The CUDA library never imports,
links or calls anything here, and this package never touches the CUDA library.

The arithmetic lives in ``gdn_oracle.c`` (plain C, fp64, one pthread per
(sequence, value head) unit); this module only compiles it with gcc, converts
inputs to fp64 and unpacks results.  Every formula's source is cited in that
file's header: SparseGDN reading notes, Secs. 2.1-2.7, Eqs. 1-25.

Parity status of each function (pins live in ``tests/test_oracle_pins.py``):
  prefill (exact solver, dense and sparse masks)  pinned: token-level brute force
  prefill (block-adjacent solver)                 pinned: kept blocks equal M^-1's
                                                  blocks; special inputs where it is exact
  events (CSR)                                    pinned: brute enumeration
  select (online selector, Eqs. 10-14)            pinned: nominal retention range and E bound of
                                                  the pages, constructed inputs with known tiers
  tail score                                      pinned: Frobenius norm by numpy
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

SOLVER_EXACT = 0
SOLVER_BLOCK_ADJ = 1
CHUNK = 64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags only: it also builds on Arm hosts)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-Wall", "-shared", "-fPIC",
                               "-o", tmp, _SRC, "-lpthread", "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            D = ctypes.POINTER(ctypes.c_double)
            I = ctypes.POINTER(ctypes.c_int)
            U8 = ctypes.POINTER(ctypes.c_uint8)
            lib.gdn_oracle_prefill_tail.restype = ctypes.c_int
            lib.gdn_oracle_prefill_tail.argtypes = ([ctypes.c_int] * 6 + [D] * 6 + [U8, ctypes.c_int, ctypes.c_int] +
                                                    [D] * 9 + [ctypes.c_int])
            lib.gdn_oracle_prefill.restype = ctypes.c_int
            lib.gdn_oracle_prefill.argtypes = [ctypes.c_int] * 6 + [D] * 6 + [U8, ctypes.c_int, ctypes.c_int] + [D] * 9
            lib.gdn_oracle_events.restype = ctypes.c_int
            lib.gdn_oracle_events.argtypes = [ctypes.c_int] * 3 + [U8, ctypes.c_int] + [I] * 7
            F = ctypes.POINTER(ctypes.c_float)
            lib.gdn_oracle_decode.restype = ctypes.c_int
            lib.gdn_oracle_decode.argtypes = [ctypes.c_int] * 5 + [D] * 7
            lib.gdn_oracle_select.restype = ctypes.c_int
            lib.gdn_oracle_select.argtypes = [ctypes.c_int] * 3 + [F, F, F, U8, I, I]
            _lib = lib
    return _lib


def _dptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def prefill(q, k, v, beta, g, mask=None, h0=None, solver=SOLVER_BLOCK_ADJ,
            nthreads=None, debug=False, tail=16):
    """Run the oracle on one batch of inputs.

    q, k [B,T,Nq,d]; v [B,T,Nv,dv]; beta, g [B,T,Nv]; mask [B,Nv/2,C] (uint8) or
    None for the dense path (every chunk selected); h0 [B,Nv,d,dv] or None.
    Returns a dict with ``o`` [B,T,Nv,dv] and ``s_final`` [B,Nv,d,dv]; with
    ``debug`` also ``o_chunk``, ``u``, ``u_prime``, ``w``, ``s_in``
    [B,Nv,C,d,dv], ``score`` [B,Nv,C] (Tail-``tail`` window) and ``cinv`` [B,Nv,C,64,64].
    """
    lib = _load()
    q, k, v, beta, g, h0 = map(_f64, (q, k, v, beta, g, h0))
    B, T, Nq, d = q.shape
    Nv, dv = v.shape[2], v.shape[3]
    C = (T + CHUNK - 1) // CHUNK
    o = np.zeros((B, T, Nv, dv))
    s_final = np.zeros((B, Nv, d, dv))
    out = {"o": o, "s_final": s_final}
    dbg = [None] * 7
    if debug:
        out.update(o_chunk=np.zeros((B, T, Nv, dv)), u=np.zeros((B, T, Nv, dv)),
                   u_prime=np.zeros((B, T, Nv, dv)), w=np.zeros((B, T, Nv, d)),
                   s_in=np.zeros((B, Nv, C, d, dv)), score=np.zeros((B, Nv, C)),
                   cinv=np.zeros((B, Nv, C, CHUNK, CHUNK)))
        dbg = [out[n] for n in ("o_chunk", "u", "u_prime", "w", "s_in", "score", "cinv")]
    m = None
    if mask is not None:
        m = np.ascontiguousarray(mask, dtype=np.uint8)
        if m.shape != (B, Nv // 2, C):
            raise ValueError(f"mask shape {m.shape} != {(B, Nv // 2, C)}")
    nthreads = nthreads or os.cpu_count() or 1
    rc = lib.gdn_oracle_prefill_tail(
        B, T, Nq, Nv, d, dv, _dptr(q), _dptr(k), _dptr(v), _dptr(beta), _dptr(g), _dptr(h0),
        None if m is None else m.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
        int(solver), int(nthreads), _dptr(o), _dptr(s_final), *[_dptr(x) for x in dbg], int(tail))
    if rc != 0:
        raise ValueError(f"gdn_oracle_prefill rejected its arguments (rc={rc})")
    return out


def events(mask, capacity=None):
    """CSR event lists of a [B,P,C] 0/1 mask (see gdn_oracle_events in gdn_oracle.c)."""
    lib = _load()
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    B, P, C = m.shape
    R, G = B * P, (C + 1) // 2
    cap = int(m.astype(np.int64).sum()) if capacity is None else int(capacity)
    I = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))
    row_pair = np.zeros(R, np.int32)
    row_ptr = np.zeros(R + 1, np.int32)
    ev_chunk = np.zeros(max(cap, 1), np.int32)
    grp_pred = np.zeros(max(R * G, 1), np.int32)
    snap_slot = np.zeros(max(cap, 1), np.int32)
    ne = np.zeros(1, np.int32)
    ns = np.zeros(1, np.int32)
    rc = lib.gdn_oracle_events(B, P, C, m.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), cap,
                               I(row_pair), I(row_ptr), I(ev_chunk), I(grp_pred), I(snap_slot), I(ne), I(ns))
    if rc < 0:
        raise ValueError("gdn_oracle_events rejected its arguments")
    E = int(ne[0])
    return {"overflow": rc == 1, "n_events": E, "n_snap": int(ns[0]),
            "row_pair": row_pair, "row_ptr": row_ptr, "ev_chunk": ev_chunk[:E] if rc == 0 else None,
            "grp_pred": grp_pred[:R * G].reshape(B, P, G), "snap_slot": snap_slot[:E] if rc == 0 else None}


def select(score, gamma, eta=None):
    """Online event selection (SparseGDN Sec. 2.4, Eqs. 10-14) for 16 head pairs.

    score, gamma: [B, Nv=32, C] fp32 (Tail-16 scores and chunk gate tails); eta: [B, Nv] or None.
    Returns dict: mask [B, 16, C] uint8, tier [B, 16] (0 L, 1 M, 2 H), k (k_L, k_M, k_H).
    """
    lib = _load()
    sc = np.ascontiguousarray(score, dtype=np.float32)
    gm = np.ascontiguousarray(gamma, dtype=np.float32)
    B, Nv, C = sc.shape
    et = None if eta is None else np.ascontiguousarray(eta, dtype=np.float32)
    mask = np.zeros((B, Nv // 2, C), np.uint8)
    tier = np.zeros((B, Nv // 2), np.int32)
    k = np.zeros(3, np.int32)
    F = lambda a: None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))
    I = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))
    rc = lib.gdn_oracle_select(B, Nv, C, F(sc), F(gm), F(et), mask.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
                               I(tier), I(k))
    if rc != 0:
        raise ValueError("gdn_oracle_select rejected its arguments (needs 16 head pairs)")
    return {"mask": mask, "tier": tier, "k": tuple(int(v) for v in k)}


def decode(q, k, v, beta, a, S):
    """One decode step (Eqs. 1-4 with a one-token chunk; see gdn_oracle.c).

    q, k [B, Nq, d]; v [B, Nv, dv]; beta, a [B, Nv] (a: the token's log2
    retention); S [B, Nv, d, dv].  Returns dict o [B, Nv, dv], s [B, Nv, d, dv].
    """
    lib = _load()
    q, k, v, beta, a = map(_f64, (q, k, v, beta, a))
    S = np.array(S, dtype=np.float64, order="C")
    B, Nq, d = q.shape
    Nv, dv = v.shape[1], v.shape[2]
    o = np.zeros((B, Nv, dv))
    rc = lib.gdn_oracle_decode(B, Nq, Nv, d, dv, _dptr(q), _dptr(k), _dptr(v), _dptr(beta), _dptr(a), _dptr(S),
                               _dptr(o))
    if rc != 0:
        raise ValueError("gdn_oracle_decode rejected its arguments")
    return {"o": o, "s": S}
