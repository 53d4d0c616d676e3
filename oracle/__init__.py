"""Plain CPU oracle for the NVFP4 expert-parallel pack / direct-receive path.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The product package
never imports this module, and this module never imports the product package.

The arithmetic lives in plain C (``oracle/*.c``), compiled here with gcc with
floating-point contraction disabled so that every FP32 operation is one IEEE
binary32 operation rounded to nearest even.  This file only compiles the C
code, loads it with ctypes and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_BUILD = _HERE / "_build"
_LIB_PATH = _BUILD / "liboracle.so"
_SOURCES = ["formats.c", "route.c", "nvfp4.c", "receive.c", "mxfp8.c"]

ROUND_RNE = 0
ROUND_SR = 1
DEFAULT_SIGN_MASK = 0xA53C


def build(force: bool = False) -> Path:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (idempotent)."""
    srcs = [_HERE / s for s in _SOURCES] + [_HERE / "oracle.h"]
    if not force and _LIB_PATH.exists():
        newest = max(s.stat().st_mtime for s in srcs)
        if _LIB_PATH.stat().st_mtime >= newest:
            return _LIB_PATH
    _BUILD.mkdir(exist_ok=True)
    tmp = _BUILD / f"liboracle.{os.getpid()}.so"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", str(tmp)]
    cmd += [str(_HERE / s) for s in _SOURCES] + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(str(build()))
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int
_U64 = ctypes.c_uint64
_U16 = ctypes.c_uint16


def _declare(L):
    L.or_e2m1_value.argtypes = [_I32]; L.or_e2m1_value.restype = ctypes.c_double
    L.or_e2m1_rne.argtypes = [ctypes.c_double]; L.or_e2m1_rne.restype = _I32
    L.or_e2m1_sr.argtypes = [ctypes.c_double, ctypes.c_uint]; L.or_e2m1_sr.restype = _I32
    L.or_e4m3_value.argtypes = [_I32]; L.or_e4m3_value.restype = ctypes.c_double
    L.or_e4m3_rne_sat.argtypes = [ctypes.c_double]; L.or_e4m3_rne_sat.restype = _I32
    L.or_bf16_rne.argtypes = [ctypes.c_double]; L.or_bf16_rne.restype = ctypes.c_uint16
    L.or_token_scale_exp.argtypes = [ctypes.c_double]; L.or_token_scale_exp.restype = _I32
    L.or_mx_scale_exp.argtypes = [ctypes.c_double]; L.or_mx_scale_exp.restype = _I32
    L.or_e2m1_rne_batch.argtypes = [_P, _I64, _P]; L.or_e2m1_rne_batch.restype = None
    L.or_e2m1_sr_batch.argtypes = [_P, _P, _I64, _P]; L.or_e2m1_sr_batch.restype = None
    L.or_e4m3_rne_sat_batch.argtypes = [_P, _I64, _P]; L.or_e4m3_rne_sat_batch.restype = None
    L.or_sr_u16s.argtypes = [_U64, ctypes.c_uint32, _U64, _I64, _P]; L.or_sr_u16s.restype = None
    L.or_philox4x32_10.argtypes = [_P, _P, _P]; L.or_philox4x32_10.restype = None
    L.or_sr_u16.argtypes = [_U64, ctypes.c_uint32, _U64]; L.or_sr_u16.restype = ctypes.c_uint
    L.or_rht16_f32.argtypes = [_P, _U16, _P]; L.or_rht16_f32.restype = None
    L.or_row_bytes.argtypes = [_I64]; L.or_row_bytes.restype = ctypes.c_size_t
    L.or_route_plan.argtypes = [_P, _I64, _I32, _I32, _I32, _P, _P, _P]
    L.or_route_plan.restype = ctypes.c_uint32
    L.or_nvfp4_pack_token.argtypes = [_P, _I64, ctypes.c_uint32, _I32, _U64, _U64, _P]
    L.or_nvfp4_pack_token.restype = None
    L.or_scale_swizzle.argtypes = [_P, _I64, _I64, _P]; L.or_scale_swizzle.restype = None
    L.or_nvfp4_colwise_rht_bf16.argtypes = [_P, _I64, _I64, _P, _I32, _P, _P, _P, _P, _P, _P, _I32, _U64, _U16, _P]
    L.or_nvfp4_colwise_rht_bf16.restype = None
    L.or_mxfp8_colwise.argtypes = [_P, _I64, _I64, _P, _I32, _P]; L.or_mxfp8_colwise.restype = None
    L.or_nvfp4_pack.argtypes = [_P, _I64, _I64, _P, _I32, _P, _P, _I32, _P, _I64, _I32, _U64]
    L.or_nvfp4_pack.restype = None
    L.or_nvfp4_unpack.argtypes = [_P, _I64, _I64, _P, _I32, _P]
    L.or_nvfp4_unpack.restype = None
    L.or_expert_amax.argtypes = [_P, _I64, _P, _I32, _P, _P, _P]
    L.or_expert_amax.restype = None
    L.or_nvfp4_direct_receive.argtypes = [_P, _I64, _I64, _P, _I32, _P,
                                          _P, _P, _P, _P, _P, _P, _P, _P,
                                          _I32, _U64, _U16, _P]
    L.or_nvfp4_direct_receive.restype = None
    L.or_mxfp8_pack.argtypes = [_P, _I64, _I64, _P, _I32, _P, _P, _I32, _P, _I64]
    L.or_mxfp8_pack.restype = None


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _as(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- formats
def e2m1_value(code: int) -> float:
    return lib().or_e2m1_value(int(code))


def e2m1_rne(v: float) -> int:
    return lib().or_e2m1_rne(float(v))


def e2m1_sr(v: float, r16: int) -> int:
    return lib().or_e2m1_sr(float(v), int(r16))


def e4m3_value(code: int) -> float:
    return lib().or_e4m3_value(int(code))


def e4m3_rne_sat(v: float) -> int:
    return lib().or_e4m3_rne_sat(float(v))


def bf16_rne(v: float) -> int:
    return lib().or_bf16_rne(float(v))


def token_scale_exp(amax: float) -> int:
    return lib().or_token_scale_exp(float(amax))


def mx_scale_exp(bmax: float) -> int:
    return lib().or_mx_scale_exp(float(bmax))


def e2m1_rne_batch(v) -> np.ndarray:
    v = _as(v, np.float64).reshape(-1)
    out = np.zeros(v.shape[0], np.uint8)
    lib().or_e2m1_rne_batch(_ptr(v), v.shape[0], _ptr(out))
    return out


def e2m1_sr_batch(v, r16) -> np.ndarray:
    v = _as(v, np.float64).reshape(-1)
    r = _as(r16, np.uint16).reshape(-1)
    out = np.zeros(v.shape[0], np.uint8)
    lib().or_e2m1_sr_batch(_ptr(v), _ptr(r), v.shape[0], _ptr(out))
    return out


def e4m3_rne_sat_batch(v) -> np.ndarray:
    v = _as(v, np.float64).reshape(-1)
    out = np.zeros(v.shape[0], np.uint8)
    lib().or_e4m3_rne_sat_batch(_ptr(v), v.shape[0], _ptr(out))
    return out


def sr_u16s(seed: int, stream: int, idx0: int, n: int) -> np.ndarray:
    """The 16-bit random numbers of elements idx0 .. idx0+n-1 (reading R13)."""
    out = np.zeros(int(n), np.uint16)
    lib().or_sr_u16s(int(seed), int(stream), int(idx0), int(n), _ptr(out))
    return out


def philox4x32_10(ctr, key) -> np.ndarray:
    c = _as(ctr, np.uint32)
    k = _as(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().or_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def sr_u16(seed: int, stream: int, idx: int) -> int:
    return lib().or_sr_u16(int(seed), int(stream), int(idx))


def rht16_f32(d, sign_mask: int = DEFAULT_SIGN_MASK) -> np.ndarray:
    d = _as(d, np.float32)
    y = np.zeros(16, np.float32)
    lib().or_rht16_f32(_ptr(d), int(sign_mask), _ptr(y))
    return y


def row_bytes(H: int) -> int:
    return int(lib().or_row_bytes(int(H)))


def rows_capacity(T: int, k: int, E: int, A: int) -> int:
    """Upper bound on the number of received rows, sum_e ceil(c_e/A)*A."""
    return int(T) * int(k) + int(E) * (int(A) - 1)


# ---------------------------------------------------------------- the path
def route_plan(topk: np.ndarray, E: int, A: int):
    """Returns (offsets[E+1], counts[E], dest[T*k], status bits)."""
    topk = _as(topk, np.int32)
    T, k = topk.shape
    offsets = np.zeros(E + 1, np.int32)
    counts = np.zeros(E, np.int32)
    dest = np.zeros(T * k, np.int32)
    st = lib().or_route_plan(_ptr(topk), T, k, E, A, _ptr(offsets), _ptr(counts), _ptr(dest))
    return offsets, counts, dest, int(st)


def pack_token(x_bf16: np.ndarray, token_id: int = 0, rounding: int = ROUND_RNE,
               seed: int = 0, t_index: int | None = None) -> np.ndarray:
    x = _as(x_bf16, np.uint16)
    H = x.shape[0]
    row = np.zeros(row_bytes(H), np.uint8)
    ti = token_id if t_index is None else t_index
    lib().or_nvfp4_pack_token(_ptr(x), H, token_id, rounding, seed, ti, _ptr(row))
    return row


def nvfp4_pack(tokens_bf16: np.ndarray, dest, k, offsets, counts, E, R_cap,
               rounding: int = ROUND_RNE, seed: int = 0) -> np.ndarray:
    x = _as(tokens_bf16, np.uint16)
    T, H = x.shape
    dest = _as(dest, np.int32); offsets = _as(offsets, np.int32); counts = _as(counts, np.int32)
    rows = np.zeros((R_cap, row_bytes(H)), np.uint8)
    lib().or_nvfp4_pack(_ptr(x), T, H, _ptr(dest), k, _ptr(offsets), _ptr(counts), E,
                        _ptr(rows), R_cap, rounding, seed)
    return rows


def nvfp4_unpack(rows: np.ndarray, H: int, offsets, E) -> np.ndarray:
    rows = _as(rows, np.uint8)
    offsets = _as(offsets, np.int32)
    R_cap = rows.shape[0]
    out = np.zeros((R_cap, H), np.uint16)
    lib().or_nvfp4_unpack(_ptr(rows), R_cap, H, _ptr(offsets), E, _ptr(out))
    return out


def expert_amax(rows: np.ndarray, H: int, offsets, E):
    rows = _as(rows, np.uint8)
    offsets = _as(offsets, np.int32)
    a = np.zeros(E, np.float32); c = np.zeros(E, np.float32); s = np.zeros(E, np.float32)
    lib().or_expert_amax(_ptr(rows), H, _ptr(offsets), E, _ptr(a), _ptr(c), _ptr(s))
    return a, c, s


def scale_swizzle(lin: np.ndarray) -> np.ndarray:
    """Scale matrix [M, Kb] (uint8, M % 128 == 0, Kb % 4 == 0) -> its M*Kb
    bytes in the tiled block-scaled GEMM layout (reading R23)."""
    lin = _as(lin, np.uint8)
    M, Kb = lin.shape
    if M % 128 or Kb % 4:
        raise ValueError("scale_swizzle needs M % 128 == 0 and Kb % 4 == 0")
    out = np.zeros(M * Kb, np.uint8)
    lib().or_scale_swizzle(_ptr(lin), M, Kb, _ptr(out))
    return out


def swizzle_grouped_scales(dr: dict, H: int, offsets, E) -> dict:
    """The grouped operands of ``nvfp4_direct_receive`` with both scale
    tensors in the tiled layout (R23): the rowwise scales of rows [0, R) as one
    [R, H/16] matrix (expert slots are whole 128-row tiles), the columnwise
    scales of each expert as its own [H, n_e/16] matrix at byte
    offsets[e]*H/16.  Bytes past R*H/16 keep the linear values."""
    offsets = _as(offsets, np.int32)
    R = int(offsets[E])
    out = dict(dr)
    rw = dr["rw_scales"].copy()
    flat = rw.reshape(-1)
    flat[: R * H // 16] = scale_swizzle(dr["rw_scales"][:R])
    out["rw_scales"] = rw
    cw = dr["cw_scales"].copy()
    for e in range(E):
        a, n = int(offsets[e]), int(offsets[e + 1] - offsets[e])
        if n:
            blk = dr["cw_scales"][a * H // 16:(a + n) * H // 16].reshape(H, n // 16)
            cw[a * H // 16:(a + n) * H // 16] = scale_swizzle(blk)
    out["cw_scales"] = cw
    return out


def nvfp4_direct_receive(rows: np.ndarray, H: int, offsets, E, rounding: int = ROUND_RNE,
                         seed: int = 0, sign_mask: int = DEFAULT_SIGN_MASK,
                         experts=None):
    """Returns a dict of the grouped operands, metadata and the bound report.

    ``experts`` (iterable of expert ids) restricts the rowwise and columnwise
    outputs to those experts; the metadata always covers all experts."""
    rows = _as(rows, np.uint8)
    offsets = _as(offsets, np.int32)
    R_cap = rows.shape[0]
    mask = None
    if experts is not None:
        mask = np.zeros(E, np.uint8)
        mask[list(experts)] = 1
    out = dict(
        rw_codes=np.zeros((R_cap, H // 2), np.uint8),
        rw_scales=np.zeros((R_cap, H // 16), np.uint8),
        rw_row_scale=np.zeros(R_cap, np.float32),
        cw_codes=np.zeros(R_cap * H // 2, np.uint8),
        cw_scales=np.zeros(R_cap * H // 16, np.uint8),
        amax_row=np.zeros(E, np.float32),
        amax_col=np.zeros(E, np.float32),
        scale_enc=np.zeros(E, np.float32),
    )
    report = np.zeros(4, np.int64)
    lib().or_nvfp4_direct_receive(
        _ptr(rows), R_cap, H, _ptr(offsets), E,
        _ptr(mask) if mask is not None else None,
        _ptr(out["rw_codes"]), _ptr(out["rw_scales"]), _ptr(out["rw_row_scale"]),
        _ptr(out["cw_codes"]), _ptr(out["cw_scales"]), _ptr(out["amax_row"]),
        _ptr(out["amax_col"]), _ptr(out["scale_enc"]), rounding, seed, sign_mask,
        _ptr(report))
    out["report"] = dict(scale_saturated=int(report[0]), above_4x_rowwise_amax=int(report[1]),
                         element_saturated=int(report[2]), above_4x_block_input=int(report[3]))
    return out


def nvfp4_colwise_rht_bf16(x_bf16: np.ndarray, offsets, E, amax_in, rounding: int = ROUND_RNE, seed: int = 0,
                           sign_mask: int = DEFAULT_SIGN_MASK) -> dict:
    """BF16 rows [R_cap, H] (expert-grouped) + supplied per-expert amax ->
    the columnwise RHT operand and the per-expert metadata (reading R24)."""
    x = _as(x_bf16, np.uint16)
    R_cap, H = x.shape
    offsets = _as(offsets, np.int32)
    amax_in = _as(amax_in, np.float32)
    out = dict(cw_codes=np.zeros(R_cap * H // 2, np.uint8), cw_scales=np.zeros(R_cap * H // 16, np.uint8),
               amax_row=np.zeros(E, np.float32), amax_col=np.zeros(E, np.float32),
               scale_enc=np.zeros(E, np.float32))
    report = np.zeros(4, np.int64)
    lib().or_nvfp4_colwise_rht_bf16(_ptr(x), R_cap, H, _ptr(offsets), E, _ptr(amax_in), _ptr(out["cw_codes"]),
                                    _ptr(out["cw_scales"]), _ptr(out["amax_row"]), _ptr(out["amax_col"]),
                                    _ptr(out["scale_enc"]), rounding, seed, sign_mask, _ptr(report))
    out["report"] = dict(scale_saturated=int(report[0]), above_4x_rowwise_amax=int(report[1]),
                         element_saturated=int(report[2]), above_4x_block_input=int(report[3]))
    return out


def mxfp8_colwise(x_bf16: np.ndarray, offsets, E) -> np.ndarray:
    """Expert-grouped BF16 rows [R_cap, H] -> one buffer: the columnwise MXFP8
    data (expert e: [H][n_e] at offsets[e]*H) then scales (expert e:
    [H][n_e/32] at R_cap*H + offsets[e]*H/32) (reading R25)."""
    x = _as(x_bf16, np.uint16)
    R_cap, H = x.shape
    offsets = _as(offsets, np.int32)
    buf = np.zeros(R_cap * H + R_cap * (H // 32), np.uint8)
    lib().or_mxfp8_colwise(_ptr(x), R_cap, H, _ptr(offsets), E, _ptr(buf))
    return buf


def mxfp8_pack(tokens_bf16: np.ndarray, dest, k, offsets, counts, E, R_cap) -> np.ndarray:
    x = _as(tokens_bf16, np.uint16)
    T, H = x.shape
    dest = _as(dest, np.int32); offsets = _as(offsets, np.int32); counts = _as(counts, np.int32)
    buf = np.zeros(R_cap * H + R_cap * (H // 32), np.uint8)
    lib().or_mxfp8_pack(_ptr(x), T, H, _ptr(dest), k, _ptr(offsets), _ptr(counts), E,
                        _ptr(buf), R_cap)
    return buf
