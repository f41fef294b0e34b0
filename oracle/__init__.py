"""CPU oracle for the grouped FP8 quantizer and grouped expert GEMMs.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library: the arithmetic lives in ``gq_oracle.c`` (plain C, fp64
accumulation, fp32 op by op where the recipe fixes fp32), this module only
marshals numpy arrays.

Parity pins (tests/test_oracle_*.py) tie every function here to something
other than itself: brute-force nearest-code search, closed forms, the pages'
printed numbers, padding/grouping invariants and exact-arithmetic GEMMs.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_SPLITS, ERR_UNSUPPORTED = 0, -1, -2, -3, -4
RECIPE_MX, RECIPE_CHANNEL, RECIPE_NVFP4 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile gq_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            lib = C.CDLL(path)
            i64p = C.POINTER(C.c_int64)
            lib.or_e4m3_decode.restype = C.c_double
            lib.or_e4m3_decode.argtypes = [C.c_uint8]
            lib.or_e4m3_encode.restype = C.c_uint8
            lib.or_e4m3_encode.argtypes = [C.c_double]
            lib.or_mx_scale_exponent.restype = C.c_int
            lib.or_mx_scale_exponent.argtypes = [C.c_double]
            lib.or_split_scan.argtypes = [C.c_void_p, C.c_int, C.c_int64, C.c_int64, C.c_int,
                                          i64p, i64p, i64p]
            lib.or_quantize_mx.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_int,
                                           C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_int64,
                                           C.c_void_p, C.c_void_p, C.c_int64]
            lib.or_quantize_channel.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_void_p,
                                                C.c_int, C.c_float, C.c_void_p, C.c_void_p,
                                                C.c_int64]
            for f in (lib.or_gemm_fprop, lib.or_gemm_dgrad):
                f.argtypes = [C.c_void_p] * 4 + [C.c_void_p, C.c_int, C.c_int64, C.c_int64,
                                                 C.c_int64, C.c_void_p]
            for f in (lib.or_gemm_wgrad_mx, lib.or_gemm_wgrad_channel):
                f.argtypes = [C.c_void_p] * 4 + [C.c_void_p, C.c_int, C.c_int64, C.c_int64,
                                                 C.c_int64, C.c_int, C.c_void_p]
            lib.or_gemm_sample.argtypes = ([C.c_int] + [C.c_void_p] * 4 +
                                           [C.c_void_p, C.c_int, C.c_int64, C.c_int64, C.c_int64,
                                            C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p,
                                            C.c_void_p])
            lib.or_grouped_bias_add.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int64,
                                                C.c_int64]
            lib.or_grouped_bias_grad.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int64, C.c_int64,
                                                 C.c_void_p]
            lib.or_srelu_quantize_mx.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p,
                                                 C.c_int, C.c_void_p, C.c_void_p, C.c_int64, C.c_void_p,
                                                 C.c_void_p, C.c_int64]
            lib.or_e2m1_decode.restype = C.c_double
            lib.or_e2m1_decode.argtypes = [C.c_uint8]
            lib.or_e2m1_encode.restype = C.c_uint8
            lib.or_e2m1_encode.argtypes = [C.c_double]
            lib.or_nv_global_scale.restype = C.c_float
            lib.or_nv_global_scale.argtypes = [C.c_float]
            lib.or_quantize_nvfp4.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_int,
                                              C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_int64,
                                              C.c_void_p, C.c_void_p, C.c_int64, C.c_void_p]
            lib.or_gemm_nvfp4.argtypes = ([C.c_int] + [C.c_void_p] * 7 +
                                          [C.c_int, C.c_int64, C.c_int64, C.c_int64, C.c_int, C.c_void_p])
            lib.or_act_exp.restype = C.c_float
            lib.or_act_exp.argtypes = [C.c_float]
            lib.or_act_silu.restype = C.c_float
            lib.or_act_silu.argtypes = [C.c_float]
            lib.or_swiglu_quantize_mx.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p,
                                                  C.c_int, C.c_void_p, C.c_void_p, C.c_int64, C.c_void_p,
                                                  C.c_void_p, C.c_int64]
            lib.or_swiglu_quantize_mx.restype = C.c_int
            lib.or_gemm_nvfp4_sample.argtypes = ([C.c_int] + [C.c_void_p] * 7 +
                                                 [C.c_int, C.c_int64, C.c_int64, C.c_int64, C.c_int64,
                                                  C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p])
            for name in ("or_quantize_nvfp4", "or_gemm_nvfp4", "or_gemm_nvfp4_sample"):
                getattr(lib, name).restype = C.c_int
            for name in ("or_split_scan", "or_quantize_mx", "or_quantize_channel", "or_srelu_quantize_mx",
                         "or_gemm_fprop", "or_gemm_dgrad", "or_gemm_wgrad_mx",
                         "or_gemm_wgrad_channel", "or_gemm_sample", "or_grouped_bias_add",
                         "or_grouped_bias_grad"):
                getattr(lib, name).restype = C.c_int
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"oracle {what} failed with status {status}")
        self.status = status


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _splits(splits):
    return None if splits is None else np.ascontiguousarray(splits, dtype=np.int32)


def _check(st, what):
    if st != OK:
        raise OracleError(st, what)


# --------------------------------------------------------------------------- #
# element codecs                                                               #
# --------------------------------------------------------------------------- #

def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    b = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(b.shape, np.float64)
    lib.or_e4m3_decode_array(_p(b), C.c_int64(b.size), _p(out))
    return out


def e4m3_encode(values) -> np.ndarray:
    lib = _load()
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    lib.or_e4m3_encode_array(_p(v), C.c_int64(v.size), _p(out))
    return out


def mx_scale_exponent(amax: float) -> int:
    return int(_load().or_mx_scale_exponent(float(amax)))


# --------------------------------------------------------------------------- #
# split scan                                                                   #
# --------------------------------------------------------------------------- #

def split_scan(splits, num_groups: int, rows_cap: int, cols: int, recipe: int = RECIPE_MX):
    """Returns (row_offset[G+1], tile_prefix[G+1], scale_offset[G+1]) or raises."""
    lib = _load()
    G = num_groups
    off = np.zeros(G + 1, np.int64)
    tp = np.zeros(G + 1, np.int64)
    sb = np.zeros(G + 1, np.int64)
    s = _splits(splits)
    i64p = C.POINTER(C.c_int64)
    st = lib.or_split_scan(_p(s), G, rows_cap, cols, recipe, off.ctypes.data_as(i64p),
                           tp.ctypes.data_as(i64p), sb.ctypes.data_as(i64p))
    _check(st, "split_scan")
    return off, tp, sb


def scale_bytes_mx(splits, num_groups, rows_cap, cols) -> int:
    return int(split_scan(splits, num_groups, rows_cap, cols)[2][-1])


# --------------------------------------------------------------------------- #
# quantisers                                                                   #
# --------------------------------------------------------------------------- #

class MXQuantized:
    """Host copy of an MX-quantised buffer: codes [R, C] uint8 and swizzled
    E8M0 scale bytes for each enabled orientation."""

    def __init__(self, row_data, row_scale, col_data, col_scale, splits, rows_cap, cols):
        self.row_data, self.row_scale = row_data, row_scale
        self.col_data, self.col_scale = col_data, col_scale
        self.splits, self.rows_cap, self.cols = splits, rows_cap, cols


def quantize_mx(x_bits, splits, num_groups: int, rowwise=True, colwise=True,
                scale_capacity: int | None = None, data_fill: int = 0,
                scale_fill: int = 0) -> MXQuantized:
    """MXFP8 1x32 quantisation of a bf16 [R, C] buffer (uint16 bits).

    Code bytes of rows past the live total keep ``data_fill``; scale bytes past
    the grouped extent keep ``scale_fill`` (canaries for the tests)."""
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, Cc = x.shape
    s = _splits(splits)
    need = int(split_scan(s, num_groups, R, Cc)[2][-1])
    cap = need if scale_capacity is None else scale_capacity
    rd = np.full((R, Cc), data_fill, np.uint8) if rowwise else None
    cd = np.full((R, Cc), data_fill, np.uint8) if colwise else None
    rs = np.full(max(cap, 1), scale_fill, np.uint8) if rowwise else None
    cs = np.full(max(cap, 1), scale_fill, np.uint8) if colwise else None
    st = lib.or_quantize_mx(_p(x), R, Cc, _p(s), num_groups, int(rowwise), int(colwise),
                            _p(rd), _p(rs), cap, _p(cd), _p(cs), cap)
    _check(st, "quantize_mx")
    return MXQuantized(rd, rs, cd, cs, s, R, Cc)


def srelu_quantize_mx(y: np.ndarray, probs: np.ndarray, splits, num_groups: int, data_fill: int = 0,
                      scale_fill: int = 0) -> MXQuantized:
    """ScaledSReLU of an fp32 [R, C] buffer, a = probs[r] * relu(y)^2 in fp32,
    then MXFP8 1x32 quantisation rowwise and columnwise (as quantize_mx)."""
    lib = _load()
    yy = np.ascontiguousarray(y, np.float32)
    pr = np.ascontiguousarray(probs, np.float32)
    R, Cc = yy.shape
    s = _splits(splits)
    need = int(split_scan(s, num_groups, R, Cc)[2][-1])
    rd = np.full((R, Cc), data_fill, np.uint8)
    cd = np.full((R, Cc), data_fill, np.uint8)
    rs = np.full(max(need, 1), scale_fill, np.uint8)
    cs = np.full(max(need, 1), scale_fill, np.uint8)
    st = lib.or_srelu_quantize_mx(_p(yy), _p(pr), R, Cc, _p(s), num_groups, _p(rd), _p(rs), need, _p(cd),
                                  _p(cs), need)
    _check(st, "srelu_quantize_mx")
    return MXQuantized(rd, rs, cd, cs, s, R, Cc)


def act_exp(x: float) -> float:
    """The activation's own exp (fp32; see or_act_exp)."""
    return float(_load().or_act_exp(float(x)))


def act_silu(x: float) -> float:
    return float(_load().or_act_silu(float(x)))


def swiglu_quantize_mx(y: np.ndarray, probs: np.ndarray, splits, num_groups: int, data_fill: int = 0,
                       scale_fill: int = 0) -> MXQuantized:
    """ScaledSwiGLU of an fp32 [R, 2C] buffer (gate half, then linear half),
    a = (silu(gate) * linear) * probs[r] in fp32, then MXFP8 1x32 quantisation
    of the [R, C] activation rowwise and columnwise (as quantize_mx)."""
    lib = _load()
    yy = np.ascontiguousarray(y, np.float32)
    pr = np.ascontiguousarray(probs, np.float32)
    R, C2 = yy.shape
    Cc = C2 // 2
    s = _splits(splits)
    need = int(split_scan(s, num_groups, R, Cc)[2][-1])
    rd = np.full((R, Cc), data_fill, np.uint8)
    cd = np.full((R, Cc), data_fill, np.uint8)
    rs = np.full(max(need, 1), scale_fill, np.uint8)
    cs = np.full(max(need, 1), scale_fill, np.uint8)
    st = lib.or_swiglu_quantize_mx(_p(yy), _p(pr), R, Cc, _p(s), num_groups, _p(rd), _p(rs), need, _p(cd),
                                   _p(cs), need)
    _check(st, "swiglu_quantize_mx")
    return MXQuantized(rd, rs, cd, cs, s, R, Cc)


class ChannelQuantized:
    """Per-channel quantised buffer: codes [R, C] uint8 and fp32 scales
    [live_rows/128, C]."""

    def __init__(self, col_data, col_scale, splits, rows_cap, cols):
        self.col_data, self.col_scale = col_data, col_scale
        self.splits, self.rows_cap, self.cols = splits, rows_cap, cols


def quantize_channel(x_bits, splits, num_groups: int, zero_scale: float = 1e-30,
                     data_fill: int = 0) -> ChannelQuantized:
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, Cc = x.shape
    s = _splits(splits)
    off, _, _ = split_scan(s, num_groups, R, Cc, RECIPE_CHANNEL)
    L = int(off[-1])
    cd = np.full((R, Cc), data_fill, np.uint8)
    cs = np.zeros((max(L // 128, 1), Cc), np.float32)
    st = lib.or_quantize_channel(_p(x), R, Cc, _p(s), num_groups, C.c_float(zero_scale),
                                 _p(cd), _p(cs), cs.size)
    _check(st, "quantize_channel")
    return ChannelQuantized(cd, cs[:L // 128], s, R, Cc)


# --------------------------------------------------------------------------- #
# NVFP4                                                                        #
# --------------------------------------------------------------------------- #

def e2m1_decode(code: int) -> float:
    return float(_load().or_e2m1_decode(int(code)))


def e2m1_encode(value: float) -> int:
    return int(_load().or_e2m1_encode(float(value)))


def nv_global_scale(amax: float) -> float:
    """The second-level scale S_g of a group with this amax (fp32)."""
    return float(_load().or_nv_global_scale(float(amax)))


def scale_bytes_nvfp4(splits, num_groups, rows_cap, cols) -> int:
    """Bytes of the grouped NVFP4 scale regions: 512 (cols/64) sum_g T_g."""
    _, tp, _ = split_scan(splits, num_groups, rows_cap, cols)
    return int(512 * (cols // 64) * tp[-1])


class NVQuantized:
    """Host copy of an NVFP4-quantised buffer: rowwise codes [R, C/2] and
    transposed columnwise codes [C, R/2] (two E2M1 codes a byte), swizzled
    E4M3 scale bytes per orientation, and the per-group amax (fp32 [G])."""

    def __init__(self, row_data, row_scale, col_data, col_scale, amax, splits, rows_cap, cols):
        self.row_data, self.row_scale = row_data, row_scale
        self.col_data, self.col_scale = col_data, col_scale
        self.amax = amax
        self.splits, self.rows_cap, self.cols = splits, rows_cap, cols


def quantize_nvfp4(x_bits, splits, num_groups: int, rowwise=True, colwise=True,
                   data_fill: int = 0, scale_fill: int = 0) -> NVQuantized:
    """NVFP4 quantisation of a bf16 [R, C] buffer (uint16 bits); code bytes of
    rows past the live total keep ``data_fill``, scale bytes past the grouped
    extent ``scale_fill``."""
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, Cc = x.shape
    s = _splits(splits)
    need = scale_bytes_nvfp4(s, num_groups, R, Cc)
    rd = np.full((R, Cc // 2), data_fill, np.uint8) if rowwise else None
    cd = np.full((Cc, R // 2), data_fill, np.uint8) if colwise else None
    rs = np.full(max(need, 1), scale_fill, np.uint8) if rowwise else None
    cs = np.full(max(need, 1), scale_fill, np.uint8) if colwise else None
    amax = np.zeros(num_groups, np.float32)
    st = lib.or_quantize_nvfp4(_p(x), R, Cc, _p(s), num_groups, int(rowwise), int(colwise),
                               _p(rd), _p(rs), need, _p(cd), _p(cs), need, _p(amax))
    _check(st, "quantize_nvfp4")
    return NVQuantized(rd, rs, cd, cs, amax, s, R, Cc)


def gemm_nvfp4(kind: str, a: NVQuantized, b: NVQuantized, splits, num_groups, N, K,
               accumulate: bool = False, init: np.ndarray | None = None) -> np.ndarray:
    """Grouped GEMMs on NVFP4 operands, fp64:
    'fprop' Y = X_g W_g^T [R, N] (a = X rowwise, b = W rowwise);
    'dgrad' dX = dY_g W_g [R, K] (a = dY rowwise, b = W columnwise);
    'wgrad' dW[g] = (init[g] if accumulate) + dY_g^T X_g [G, N, K] (both columnwise).
    Rows past the live total of Y / dX are NaN."""
    lib = _load()
    R = a.rows_cap
    if kind == "fprop":
        k, ad, as_, bd, bs, y = 0, a.row_data, a.row_scale, b.row_data, b.row_scale, np.full((R, N), np.nan)
    elif kind == "dgrad":
        k, ad, as_, bd, bs, y = 1, a.row_data, a.row_scale, b.col_data, b.col_scale, np.full((R, K), np.nan)
    elif kind == "wgrad":
        k, ad, as_, bd, bs = 2, a.col_data, a.col_scale, b.col_data, b.col_scale
        y = (np.zeros((num_groups, N, K)) if init is None
             else np.ascontiguousarray(init, dtype=np.float64).copy())
    else:
        raise ValueError(kind)
    st = lib.or_gemm_nvfp4(k, _p(ad), _p(as_), _p(np.ascontiguousarray(a.amax, np.float32)), _p(bd), _p(bs),
                           _p(np.ascontiguousarray(b.amax, np.float32)), _p(_splits(splits)), num_groups, R,
                           N, K, int(accumulate), _p(y))
    _check(st, "gemm_nvfp4")
    return y


def gemm_nvfp4_sample(kind: str, a: NVQuantized, b: NVQuantized, splits, num_groups, N, K, i_idx, j_idx,
                      g_idx=None) -> np.ndarray:
    """Selected outputs of gemm_nvfp4, one fp64 dot product each: 'fprop'
    (row, n), 'dgrad' (row, k), 'wgrad' (g, n, k) without the accumulate term."""
    lib = _load()
    i_idx = np.ascontiguousarray(i_idx, np.int64)
    j_idx = np.ascontiguousarray(j_idx, np.int64)
    g = np.ascontiguousarray(np.zeros_like(i_idx) if g_idx is None else g_idx, np.int32)
    out = np.empty(i_idx.size, np.float64)
    if kind == "fprop":
        k, ad, as_, bd, bs = 0, a.row_data, a.row_scale, b.row_data, b.row_scale
    elif kind == "dgrad":
        k, ad, as_, bd, bs = 1, a.row_data, a.row_scale, b.col_data, b.col_scale
    elif kind == "wgrad":
        k, ad, as_, bd, bs = 2, a.col_data, a.col_scale, b.col_data, b.col_scale
    else:
        raise ValueError(kind)
    st = lib.or_gemm_nvfp4_sample(k, _p(ad), _p(as_), _p(np.ascontiguousarray(a.amax, np.float32)), _p(bd),
                                  _p(bs), _p(np.ascontiguousarray(b.amax, np.float32)), _p(_splits(splits)),
                                  num_groups, a.rows_cap, N, K, i_idx.size, _p(g), _p(i_idx), _p(j_idx), _p(out))
    _check(st, "gemm_nvfp4_sample")
    return out


# --------------------------------------------------------------------------- #
# grouped GEMMs                                                                #
# --------------------------------------------------------------------------- #

def gemm_fprop(xq: MXQuantized, wq: MXQuantized, splits, num_groups, N, K,
               out: np.ndarray | None = None) -> np.ndarray:
    """Y = X_g W_g^T per group, fp64 [R, N]; rows past the live total keep
    ``out``'s content (NaN by default)."""
    lib = _load()
    R = xq.rows_cap
    y = np.full((R, N), np.nan) if out is None else out
    st = lib.or_gemm_fprop(_p(xq.row_data), _p(xq.row_scale), _p(wq.row_data),
                           _p(wq.row_scale), _p(_splits(splits)), num_groups, R, N, K, _p(y))
    _check(st, "gemm_fprop")
    return y


def grouped_bias_add(y: np.ndarray, bias: np.ndarray, splits, num_groups) -> np.ndarray:
    """y[o_g + r, :] += bias[g] for the live rows of every group, in place on
    a C-contiguous fp64 [R, N] array; returns y."""
    lib = _load()
    assert y.dtype == np.float64 and y.flags.c_contiguous
    R, N = y.shape
    b = np.ascontiguousarray(bias, np.float64).reshape(num_groups, N)
    st = lib.or_grouped_bias_add(_p(y), _p(b), _p(_splits(splits)), num_groups, R, N)
    _check(st, "grouped_bias_add")
    return y


def grouped_bias_grad(dy_bits: np.ndarray, splits, num_groups) -> np.ndarray:
    """Per-group column sums of the live rows of a bf16 [R, C] buffer (given
    as uint16 bits), fp64 [G, C]."""
    lib = _load()
    dy = np.ascontiguousarray(dy_bits, np.uint16)
    R, Cc = dy.shape
    db = np.empty((num_groups, Cc))
    st = lib.or_grouped_bias_grad(_p(dy), _p(_splits(splits)), num_groups, R, Cc, _p(db))
    _check(st, "grouped_bias_grad")
    return db


def gemm_dgrad(dyq: MXQuantized, wq: MXQuantized, splits, num_groups, N, K,
               out: np.ndarray | None = None) -> np.ndarray:
    """dX = dY_g W_g per group (W columnwise), fp64 [R, K]."""
    lib = _load()
    R = dyq.rows_cap
    dx = np.full((R, K), np.nan) if out is None else out
    st = lib.or_gemm_dgrad(_p(dyq.row_data), _p(dyq.row_scale), _p(wq.col_data),
                           _p(wq.col_scale), _p(_splits(splits)), num_groups, R, N, K, _p(dx))
    _check(st, "gemm_dgrad")
    return dx


def gemm_wgrad(dyq, xq, splits, num_groups, N, K, accumulate: bool = False,
               init: np.ndarray | None = None) -> np.ndarray:
    """dW[g] = (init[g] if accumulate) + dY_g^T X_g over live rows, fp64 [G, N, K]."""
    lib = _load()
    R = dyq.rows_cap
    dw = (np.zeros((num_groups, N, K)) if init is None
          else np.ascontiguousarray(init, dtype=np.float64).copy())
    if isinstance(dyq, ChannelQuantized):
        st = lib.or_gemm_wgrad_channel(_p(dyq.col_data), _p(dyq.col_scale), _p(xq.col_data),
                                       _p(xq.col_scale), _p(_splits(splits)), num_groups, R, N,
                                       K, int(accumulate), _p(dw))
    else:
        st = lib.or_gemm_wgrad_mx(_p(dyq.col_data), _p(dyq.col_scale), _p(xq.col_data),
                                  _p(xq.col_scale), _p(_splits(splits)), num_groups, R, N, K,
                                  int(accumulate), _p(dw))
    _check(st, "gemm_wgrad")
    return dw


def gemm_sample(kind: str, a, b, splits, num_groups, N, K, i_idx, j_idx, g_idx=None):
    """Selected outputs, one fp64 dot product each.

    kind 'fprop': (row, n); 'dgrad': (row, k); 'wgrad': (g, n, k) -- the
    wgrad sample excludes any accumulate term."""
    lib = _load()
    i_idx = np.ascontiguousarray(i_idx, np.int64)
    j_idx = np.ascontiguousarray(j_idx, np.int64)
    g = np.ascontiguousarray(np.zeros_like(i_idx) if g_idx is None else g_idx, np.int32)
    out = np.empty(i_idx.size, np.float64)
    if kind == "fprop":
        k, ad, as_, bd, bs = 0, a.row_data, a.row_scale, b.row_data, b.row_scale
    elif kind == "dgrad":
        k, ad, as_, bd, bs = 1, a.row_data, a.row_scale, b.col_data, b.col_scale
    elif kind == "wgrad":
        k = 3 if isinstance(a, ChannelQuantized) else 2
        ad, as_, bd, bs = a.col_data, a.col_scale, b.col_data, b.col_scale
    else:
        raise ValueError(kind)
    st = lib.or_gemm_sample(k, _p(ad), _p(as_), _p(bd), _p(bs), _p(_splits(splits)),
                            num_groups, a.rows_cap, N, K, i_idx.size, _p(g), _p(i_idx),
                            _p(j_idx), _p(out))
    _check(st, "gemm_sample")
    return out
