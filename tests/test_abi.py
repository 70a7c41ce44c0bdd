"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/gdn.h declares, sizes workspaces, and rejects bad arguments on the host
before anything is enqueued (only argument errors are exercised here, so no
pointer is ever dereferenced and no kernel is launched)."""
import ctypes
import os
import re

import pytest

import gated_delta_rule_16_gb300 as gdn
from gated_delta_rule_16_gb300 import _binding as bnd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_16_gb300 import build
    build.build()
    return gdn.load()


def declared_entry_points():
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    return sorted(set(re.findall(r"GDN_API\s+[\w\s\*]*?\b(gdn_\w+)\s*\(", text)))


def test_exports_match_header(lib):
    names = declared_entry_points()
    assert names == sorted(bnd.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert gdn.gdn_version() == 100
    for code in range(11):
        assert lib.gdn_status_string(code)
    assert lib.gdn_status_string(0) == b"ok"


def shape(B=1, T=4096, Nq=16, Nv=32, d=128, dv=128, dtype=bnd.GDN_BF16):
    return bnd.GdnShape(B, T, Nq, Nv, d, dv, dtype)


def test_workspace_bytes(lib):
    s = shape()
    n_ex = gdn.gdn_workspace_bytes(s, "exact")
    n_ba = gdn.gdn_workspace_bytes(s, "block_adj")
    assert n_ex == n_ba > 0   # bf16 defaults keep no solver blocks (W is built inside the intra step)
    s32 = shape(dtype=bnd.GDN_F32)  # fp32 storage keeps C-bar: 10 blocks (exact) vs 7 per chunk and head
    assert gdn.gdn_workspace_bytes(s32, "exact") - gdn.gdn_workspace_bytes(s32, "block_adj") == 4096 * 32 // 64 * 3 * 256 * 4
    # U alone is B*T*Nv*dv*2 bytes for bf16; the workspace holds at least that
    assert n_ba > 1 * 4096 * 32 * 128 * 2
    assert gdn.gdn_workspace_bytes(shape(d=64, dv=64)) == 0
    # a partial last chunk is allowed: C = ceil(T / 64)
    assert 0 < gdn.gdn_workspace_bytes(shape(T=100)) < gdn.gdn_workspace_bytes(shape(T=128))
    assert gdn.gdn_workspace_bytes(shape(Nv=31)) == 0
    assert gdn.gdn_workspace_bytes(shape(T=0)) > 0
    # grows linearly with the batch
    assert gdn.gdn_workspace_bytes(shape(B=2)) > 1.9 * n_ba


FAKE = 1 << 20  # aligned fake address: never dereferenced, every call below fails validation first


def call_dense(lib, s, ptrs=None, ws=FAKE, ws_bytes=1 << 40, solver=1):
    p = ptrs or {}
    get = lambda n: ctypes.c_void_p(p.get(n, FAKE))
    return lib.gdn_prefill_dense(ctypes.byref(s), get("q"), get("k"), get("v"), get("beta"), get("g"),
                                 ctypes.c_void_p(p.get("h0")), solver, get("o"), get("s"),
                                 ctypes.c_void_p(p.get("score")), ctypes.c_void_p(ws), ws_bytes, None)


def test_host_validation(lib):
    assert call_dense(lib, shape(d=64, dv=64)) == 6          # UNSUPPORTED
    assert call_dense(lib, shape(T=100)) == 8                 # a partial last chunk passes validation (no GPU here)
    assert call_dense(lib, shape(T=64 * 16385)) == 6          # UNSUPPORTED: more than 16384 chunks
    assert call_dense(lib, shape(Nv=31)) == 2                 # SHAPE
    assert call_dense(lib, shape(dtype=7)) == 3               # DTYPE
    assert call_dense(lib, shape(), solver=5) == 3            # DTYPE (solver)
    assert call_dense(lib, shape(), ptrs={"q": 0}) == 1       # NULL
    assert call_dense(lib, shape(), ptrs={"o": FAKE + 4}) == 4  # ALIGN
    assert call_dense(lib, shape(), ws=FAKE + 16) == 4        # ALIGN: workspace needs 256 bytes
    assert call_dense(lib, shape(), ws_bytes=1024) == 5       # WORKSPACE
    assert call_dense(lib, shape(), ws=0) == 1                # NULL workspace
    # B == 0 is a valid empty call: nothing to do, nothing touched
    assert call_dense(lib, shape(B=0), ptrs={n: 0 for n in ("q", "k", "v", "beta", "g", "o", "s")}, ws=0) == 0


def test_sparse_requires_mask(lib):
    s = shape()
    get = ctypes.c_void_p(FAKE)
    rc = lib.gdn_prefill_sparse(ctypes.byref(s), get, get, get, get, get, None, None, 1, get, get, None,
                                get, 1 << 40, None)
    assert rc == 1


def test_select_events_validation(lib):
    ev = bnd.GdnEvents(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 10)
    assert lib.gdn_select_events(ctypes.byref(shape()), None, ctypes.byref(ev), None) == 1
    ev2 = bnd.GdnEvents(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, -1)
    assert lib.gdn_select_events(ctypes.byref(shape()), ctypes.c_void_p(FAKE), ctypes.byref(ev2), None) == 2
    ev3 = bnd.GdnEvents(FAKE + 2, FAKE, FAKE, FAKE, FAKE, FAKE, 10)
    assert lib.gdn_select_events(ctypes.byref(shape()), ctypes.c_void_p(FAKE), ctypes.byref(ev3), None) == 4


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        bnd._lib, saved = None, bnd._lib
        try:
            bnd.load(str(tmp_path / "missing.so"))
        finally:
            bnd._lib = saved


def test_online_workspace_and_validation(lib):
    s = shape()
    assert gdn.gdn_workspace_bytes(s, "block_adj", 2) > gdn.gdn_workspace_bytes(s, "block_adj", 1)
    assert lib.gdn_select_scored_workspace_bytes(ctypes.byref(s)) > 16 * 64 * 4
    assert lib.gdn_select_scored_workspace_bytes(ctypes.byref(shape(Nq=2, Nv=4))) == 0
    f = ctypes.c_void_p(FAKE)

    def online(sh, ws_bytes=1 << 40, **kw):
        get = lambda n: ctypes.c_void_p(kw.get(n, FAKE))
        return lib.gdn_prefill_sparse_online(ctypes.byref(sh), get("q"), get("k"), get("v"), get("beta"),
                                             get("g"), None, None, 1, get("o"), get("s"), None, None, None,
                                             f, ws_bytes, None)

    assert online(shape(Nq=2, Nv=4)) == 6                     # UNSUPPORTED: the tier table is for 16 pairs
    assert online(shape(), q=0) == 1                          # NULL
    assert online(shape(), o=FAKE + 4) == 4                   # ALIGN
    assert online(shape(), ws_bytes=4096) == 5                # WORKSPACE

    def scored(sh, score=FAKE, g=FAKE, mask=FAKE, ws_bytes=1 << 40):
        return lib.gdn_select_events_scored(ctypes.byref(sh), ctypes.c_void_p(score), ctypes.c_void_p(g), None,
                                            ctypes.c_void_p(mask), None, f, ws_bytes, None)

    assert scored(shape(Nq=2, Nv=4)) == 6
    assert scored(shape(), score=0) == 1
    assert scored(shape(), mask=0) == 1
    assert scored(shape(), score=FAKE + 4) == 4
    assert scored(shape(), ws_bytes=64) == 5
    assert scored(shape(B=0), score=0, g=0, mask=0) == 0


def test_host_prefill_validation(lib):
    s = shape()
    dev_bytes = gdn.gdn_workspace_bytes(s, "block_adj", 1)
    host_bytes = lib.gdn_prefill_host_workspace_bytes(ctypes.byref(s), 1, 1)
    # staging holds q, k, v, beta, g, h0, mask, o and s_final on top of the workspace
    assert host_bytes > dev_bytes + 2 * (4096 * 16 * 128 * 2) + 2 * (4096 * 32 * 128 * 2)
    f = ctypes.c_void_p(FAKE)

    def host(sh, ws=FAKE, ws_bytes=1 << 40, q=FAKE):
        return lib.gdn_prefill_host(ctypes.byref(sh), ctypes.c_void_p(q), f, f, f, f, None, f, 1, f, f,
                                    ctypes.c_void_p(ws), ws_bytes, None)

    assert host(shape(d=64, dv=64)) == 6
    assert host(shape(), ws=0) == 1
    assert host(shape(), ws=FAKE + 16) == 4
    assert host(shape(), ws_bytes=dev_bytes) == 5     # the staging does not fit
    assert host(shape(), q=0) == 1
    assert host(shape(B=0), ws=0, q=0) == 0


def test_decode_validation(lib):
    f = ctypes.c_void_p(FAKE)

    def dec(sh, q=FAKE, st=FAKE):
        return lib.gdn_decode_step(ctypes.byref(sh), ctypes.c_void_p(q), f, f, f, f, ctypes.c_void_p(st), f, None)

    assert dec(shape(T=4096)) == 2                    # SHAPE: one token per sequence
    assert dec(shape(T=1, d=64, dv=64)) == 6          # UNSUPPORTED
    assert dec(shape(T=1, Nv=3)) == 2
    assert dec(shape(T=1), q=0) == 1
    assert dec(shape(T=1), st=FAKE + 8) == 4
    assert dec(shape(B=0, T=1), q=0, st=0) == 0


def test_prefill_ex_option_validation(lib):
    f = ctypes.c_void_p(FAKE)

    def ex(mode=1, opt=None, mask=FAKE):
        o = opt or bnd.GdnOptions()
        return lib.gdn_prefill_ex(ctypes.byref(shape()), mode, f, f, f, f, f, None, ctypes.c_void_p(mask), None, 1,
                                  ctypes.byref(o), f, f, None, None, None, f, 1 << 40, None)

    assert ex(opt=bnd.GdnOptions(12)) == 6                 # tail window must be 8, 16, 32 or 64
    assert ex(opt=bnd.GdnOptions(16, 2)) == 6              # w_deferred is 0 or 1
    r = bnd.GdnOptions(16, 0)
    r.reserved[1] = 1
    assert ex(opt=r) == 6                                  # reserved fields must be zero
    O = lambda **kw: bnd.GdnOptions(kw.get("tw", 0), kw.get("wd", 0), kw.get("runs", 0), kw.get("full", 0),
                                    kw.get("exp", 0))
    assert ex(opt=O(runs=1, full=1)) == 6                  # the full scan is a variant of the one-pass scan
    assert ex(opt=O(runs=1, exp=1)) == 6                   # so are the expanded states
    assert ex(opt=O(wd=1, full=1)) == 6                    # the full scan needs W of every chunk from intra
    assert ex(mode=2, opt=O(full=1)) == 6                  # not with online selection
    assert ex(opt=O(full=2)) == 6 and ex(opt=O(exp=3)) == 6
    assert ex(opt=O(full=1, exp=1)) == 8                   # valid together: stops at the device check here
    split = lambda v: bnd.GdnOptions(0, 0, 0, 0, 0, v)
    assert ex(opt=split(1)) == 6                           # two-call online selection: mode online only
    assert ex(mode=2, opt=split(3)) == 6
    assert ex(mode=2, opt=split(2), mask=0) == 1           # the second call takes the rank's mask
    assert ex(mode=2, opt=split(1)) == 1                   # the first call writes the scores (score=NULL here)
    assert ex(mode=7) == 6
    assert ex(mask=0) == 1                                 # sparse mode needs a mask
    assert ex(opt=bnd.GdnOptions(64, 1)) == 8              # valid: stops at the device check here


def test_workspace_bytes_ex_matches_and_orders_variants(lib):
    s = shape(T=32768)
    opt = lambda **kw: bnd.GdnOptions(kw.get("tw", 0), kw.get("wd", 0), kw.get("runs", 0))
    wsx = lambda mode, o=None: int(lib.gdn_workspace_bytes_ex(ctypes.byref(s), 1, mode,
                                                               None if o is None else ctypes.byref(o)))
    base = gdn.gdn_workspace_bytes(s, "block_adj", 1)
    assert wsx(1) == base == wsx(1, opt()) == wsx(0)       # defaults: dense and sparse share one layout
    assert wsx(2) == gdn.gdn_workspace_bytes(s, "block_adj", 2) > base
    # the compact C-bar blocks (bf16: 7 blocks of 16x16 per chunk and head, fp32 slots)
    assert wsx(1, opt(wd=1)) - base >= 32 * 512 * 7 * 256 * 4
    # the run maps: A (bf16), B and the entry states (fp32), 128 x 128 per run, head and pair
    assert wsx(1, opt(runs=1)) - base >= 16 * 2 * 32 * 128 * 128 * 10
    assert wsx(1, opt(runs=2)) == 0 and wsx(1, opt(tw=5)) == 0 and wsx(3) == 0
    # fp32 storage always keeps C-bar (its W is built after the intra step)
    s32 = shape(T=1024, dtype=bnd.GDN_F32)
    assert int(lib.gdn_workspace_bytes_ex(ctypes.byref(s32), 1, 1, None)) == gdn.gdn_workspace_bytes(s32)


def test_events_bytes_and_carve(lib):
    s = shape(B=2, T=1000, Nq=3, Nv=6)            # R = 6 rows, C = 16 chunks, G = 8 groups
    up = lambda n: (n + 255) // 256 * 256
    want = up(6 * 4) + up(7 * 4) + up(50 * 4) + up(6 * 8 * 4) + up(50 * 4) + up(16)
    assert int(lib.gdn_events_bytes(ctypes.byref(s), 50)) == want
    assert int(lib.gdn_events_bytes(ctypes.byref(s), -1)) == 0
    assert int(lib.gdn_events_bytes(ctypes.byref(shape(Nv=31)), 8)) == 0
    ev = bnd.GdnEvents()
    base = 1 << 20                                # never dereferenced: carving only computes addresses
    assert lib.gdn_events_carve(ctypes.byref(s), 50, ctypes.c_void_p(base), ctypes.byref(ev)) == 0
    offs = [p - base for p in (ev.row_pair, ev.row_ptr, ev.ev_chunk, ev.grp_pred, ev.snap_slot, ev.counts)]
    assert offs == [0, 256, 512, 768, 1024, 1280] and ev.capacity == 50
    assert offs[-1] + 16 <= want
    assert lib.gdn_events_carve(ctypes.byref(s), 50, ctypes.c_void_p(base + 16), ctypes.byref(ev)) == 4  # ALIGN
    assert lib.gdn_events_carve(ctypes.byref(s), 50, None, ctypes.byref(ev)) == 1                        # NULL
    assert lib.gdn_events_carve(ctypes.byref(s), -3, ctypes.c_void_p(base), ctypes.byref(ev)) == 2       # SHAPE
