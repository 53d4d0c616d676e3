"""The C-ABI library loads and exports every symbol include/epq.h declares;
host-side validation rejects bad arguments before anything is enqueued (no
GPU is needed for these: every call here fails its checks before touching
CUDA)."""
import ctypes
import os
import re

import pytest

import nvfp4_quantization_gb300 as nq
from nvfp4_quantization_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "epq.h")

FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails a host check first


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ep_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_exported_symbols():
    assert declared_functions() == sorted(_lib.SYMBOLS)


def test_library_exports_every_declared_symbol():
    L = nq.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_size_helpers():
    L = nq.lib()
    for H in (32, 1024, 1056, 4096, 7168):
        assert L.ep_nvfp4_row_bytes(H) == ((9 * H // 16 + 16 + 15) // 16) * 16
        assert L.ep_nvfp4_row_bytes(H) % 16 == 0
    assert L.ep_rows_capacity(4096, 2, 16, 128) == 4096 * 2 + 16 * 127
    assert L.ep_route_workspace_bytes(0, 2, 16) >= 16
    assert L.ep_route_workspace_bytes(16384, 8, 256) == 16 + 32 * 256 * 4
    # the largest batch the fixed scratch of ep_route_plan_noalloc holds at E = 256
    assert L.ep_route_workspace_bytes(130560, 8, 256) <= _lib.EP_ROUTE_STATIC_SCRATCH_BYTES
    assert L.ep_route_workspace_bytes(130561, 8, 256) > _lib.EP_ROUTE_STATIC_SCRATCH_BYTES


def test_status_strings():
    for s in range(0, -8, -1):
        assert _lib.status_string(s).startswith("EP_")


def test_host_memory_is_refused_with_ep_err_device():
    """Device guard, host side: pointers that are not device memory of the
    input's device (here plain host memory, which also holds on a machine
    without a GPU) return EP_ERR_DEVICE once the sizes are valid."""
    import numpy as np
    L = nq.lib()
    buf = np.zeros(1 << 20, np.int32)
    h = ctypes.c_void_p(buf.ctypes.data)
    T, k, E = 10, 2, 4
    R_cap = T * k + E * 127
    assert L.ep_route_plan(h, T, k, E, 128, R_cap, h, h, h, h, 1 << 20, h, None) == -6
    assert L.ep_nvfp4_pack(h, T, 1024, h, k, h, h, E, h, R_cap, None, 0, 0, h, None) == -6
    assert L.ep_nvfp4_unpack(h, R_cap, 1024, h, E, h, h, None) == -6
    g = _lib.EpGrouped(cw_codes=h.value, cw_scales=h.value, amax_row=h.value, amax_col=h.value, cw_scale_enc=h.value)
    assert L.ep_nvfp4_direct_receive(h, R_cap, 1024, h, E, None, ctypes.byref(g), 0, 0, 0, h, None) == -6
    assert L.ep_mxfp8_pack(h, T, 1024, h, k, h, h, E, h, R_cap, h, None) == -6
    assert buf.sum() == 0     # nothing was written


def test_route_plan_validation():
    L = nq.lib()
    f = L.ep_route_plan
    ok = dict(topk=FAKE, T=10, k=2, E=4, A=128, R_cap=10 * 2 + 4 * 127, off=FAKE, cnt=FAKE, dest=FAKE,
              ws=FAKE, ws_bytes=1 << 20, st=FAKE)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["topk"], a["T"], a["k"], a["E"], a["A"], a["R_cap"], a["off"], a["cnt"], a["dest"], a["ws"],
                 a["ws_bytes"], a["st"], None)
    assert call(off=None) == -1
    assert call(st=None) == -1
    assert call(k=0) == -2 and call(k=33) == -2 and call(E=0) == -2 and call(E=1025) == -2
    assert call(T=-1) == -2
    assert call(A=64) == -3 and call(A=0) == -3 and call(A=200) == -3
    assert call(R_cap=10 * 2 + 4 * 127 - 1) == -4
    assert call(ws_bytes=0) == -4


def test_pack_validation():
    L = nq.lib()

    def call(**kw):
        a = dict(tok=FAKE, T=4, H=1024, dest=FAKE, k=2, off=FAKE, cnt=FAKE, E=4, rows=FAKE, R_cap=600,
                 amax=None, rnd=0, seed=0, st=FAKE)
        a.update(kw)
        return L.ep_nvfp4_pack(a["tok"], a["T"], a["H"], a["dest"], a["k"], a["off"], a["cnt"], a["E"], a["rows"],
                               a["R_cap"], a["amax"], a["rnd"], a["seed"], a["st"], None)
    assert call(rows=None) == -1
    assert call(H=1000) == -2 and call(H=0) == -2 and call(k=40) == -2
    assert call(R_cap=-1) == -4
    assert call(tok=ctypes.c_void_p(0x10008)) == -3
    # MXFP8 shares the checks
    assert L.ep_mxfp8_pack(FAKE, 4, 48, FAKE, 2, FAKE, FAKE, 4, FAKE, 600, FAKE, None) == -2


def test_dispatch_validation():
    L = nq.lib()
    bad = ctypes.c_void_p(0x10002)
    args = [FAKE, FAKE, 4, 1024, 2, 4, 128, 600, FAKE, FAKE, FAKE, FAKE, 1 << 20, FAKE]
    assert L.ep_nvfp4_dispatch(*args, bad, 0, 0, FAKE, None) == -3        # misaligned expert_amax
    assert L.ep_nvfp4_dispatch(*args, None, 7, 0, FAKE, None) == -5       # unknown rounding
    args[6] = 64
    assert L.ep_nvfp4_dispatch(*args, None, 0, 0, FAKE, None) == -3       # alignment A not a multiple of 128


def test_receive_and_unpack_validation():
    L = nq.lib()
    g = _lib.EpGrouped()
    assert L.ep_nvfp4_direct_receive(FAKE, 128, 1024, FAKE, 4, None, ctypes.byref(g), 0, 0, 0, FAKE, None) == -1
    g = _lib.EpGrouped(rw_codes=FAKE.value, cw_codes=FAKE.value, cw_scales=FAKE.value, amax_row=FAKE.value,
                       amax_col=FAKE.value, cw_scale_enc=FAKE.value)
    # a partial rowwise group is rejected
    assert L.ep_nvfp4_direct_receive(FAKE, 128, 1024, FAKE, 4, None, ctypes.byref(g), 0, 0, 0, FAKE, None) == -1
    g.rw_codes = None
    assert L.ep_nvfp4_direct_receive(FAKE, 128, 1000, FAKE, 4, None, ctypes.byref(g), 0, 0, 0, FAKE, None) == -2
    assert L.ep_nvfp4_direct_receive(FAKE, 128, 1024, FAKE, 4, None, ctypes.byref(g), 7, 0, 0, FAKE, None) == -5
    # element positions (the stochastic-rounding counters) must stay below 2^36
    assert L.ep_nvfp4_direct_receive(FAKE, 1 << 26, 1024, FAKE, 4, None, ctypes.byref(g), 0, 0, 0, FAKE, None) != -4
    assert L.ep_nvfp4_direct_receive(FAKE, (1 << 26) + 1, 1024, FAKE, 4, None, ctypes.byref(g), 0, 0, 0, FAKE,
                                     None) == -4
    assert L.ep_nvfp4_direct_receive_swizzled(FAKE, (1 << 26) + 1, 1024, FAKE, 4, None, ctypes.byref(g), 0, 0, 0,
                                              FAKE, None) == -4
    # a supplied per-expert amax must be 4-byte aligned
    bad = ctypes.c_void_p(0x10002)
    assert L.ep_nvfp4_direct_receive(FAKE, 128, 1024, FAKE, 4, bad, ctypes.byref(g), 0, 0, 0, FAKE, None) == -3
    assert L.ep_nvfp4_direct_receive_swizzled(FAKE, 128, 1024, FAKE, 4, bad, ctypes.byref(g), 0, 0, 0, FAKE,
                                              None) == -3
    assert L.ep_nvfp4_unpack(FAKE, 128, 1000, FAKE, 4, FAKE, FAKE, None) == -2
    assert L.ep_nvfp4_unpack(None, 128, 1024, FAKE, 4, FAKE, FAKE, None) == -1


def test_bf16_quantizer_validation():
    L = nq.lib()
    bad = ctypes.c_void_p(0x10008)    # 8-byte aligned only

    def cw(**kw):
        a = dict(x=FAKE, R=256, H=1024, off=FAKE, E=4, amax=FAKE, codes=FAKE, scales=FAKE, ar=FAKE, ac=FAKE,
                 se=FAKE, rnd=0, st=FAKE)
        a.update(kw)
        return L.ep_nvfp4_colwise_rht_bf16(a["x"], a["R"], a["H"], a["off"], a["E"], a["amax"], a["codes"],
                                           a["scales"], a["ar"], a["ac"], a["se"], a["rnd"], 0, 0, a["st"], None)
    assert cw(amax=None) == -1 and cw(se=None) == -1 and cw(st=None) == -1
    assert cw(H=1000) == -2 and cw(E=0) == -2 and cw(E=1025) == -2
    assert cw(R=-1) == -4
    assert cw(rnd=2) == -5
    assert cw(x=bad) == -3 and cw(codes=bad) == -3

    def mx(**kw):
        a = dict(x=FAKE, R=256, H=1024, off=FAKE, E=4, buf=FAKE, st=FAKE)
        a.update(kw)
        return L.ep_mxfp8_colwise(a["x"], a["R"], a["H"], a["off"], a["E"], a["buf"], a["st"], None)
    assert mx(buf=None) == -1 and mx(off=None) == -1
    assert mx(H=48) == -2 and mx(E=0) == -2
    assert mx(R=-1) == -4
    assert mx(buf=bad) == -3


def test_route_plan_noalloc_validation():
    L = nq.lib()

    def call(**kw):
        a = dict(topk=FAKE, T=10, k=2, E=4, A=128, R=10 * 2 + 4 * 127, off=FAKE, cnt=FAKE, dest=FAKE, st=FAKE)
        a.update(kw)
        return L.ep_route_plan_noalloc(a["topk"], a["T"], a["k"], a["E"], a["A"], a["R"], a["off"], a["cnt"],
                                       a["dest"], a["st"], None)
    assert call(off=None) == -1 and call(st=None) == -1
    assert call(k=0) == -2 and call(E=1025) == -2
    assert call(A=64) == -3
    assert call(R=10 * 2 + 4 * 127 - 1) == -4
    # a plan larger than the fixed scratch is refused, not truncated
    T, k, E = 1 << 20, 8, 1024
    assert L.ep_route_workspace_bytes(T, k, E) > _lib.EP_ROUTE_STATIC_SCRATCH_BYTES
    assert call(T=T, k=k, E=E, R=T * k + E * 127) == -4


def test_static_scratch_size_matches_header():
    m = re.search(r"#define\s+EP_ROUTE_STATIC_SCRATCH_BYTES\s+(\d+)", open(HEADER).read())
    assert m and int(m.group(1)) == _lib.EP_ROUTE_STATIC_SCRATCH_BYTES
