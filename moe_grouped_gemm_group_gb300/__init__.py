"""Python binding of libgq: grouped FP8 quantizer and grouped expert GEMMs on GB300.

Argument marshalling only: every step of the path runs in the CUDA kernels of
libgq.so (built from csrc/ by ``moe_grouped_gemm_group_gb300.build``).  The
functions carry the C ABI's names (include/gq.h) and take torch CUDA tensors
for device buffers; torch supplies device memory and streams, nothing else.
There is no CPU fallback: if the library is missing or a tensor is not on a
CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

__all__ = [
    "GQError", "Recipe", "Quantized", "GroupedTensor", "load", "library_path",
    "gq_status_string", "gq_version", "gq_scale_bytes_bound", "gq_split_scan", "gq_quantize",
    "gq_gemm_fprop", "gq_gemm_dgrad", "gq_gemm_wgrad", "gq_gemm_wgrad_noalloc", "alloc_quantized",
    "gq_gemm_fprop_bias", "gq_quantize_dbias", "gq_dbias_workspace_bytes", "gq_gemm_fprop_srelu_quant",
    "gq_gemm_fprop_swiglu_quant", "gq_check_wait_limit",
    "RECIPE_MXFP8_1X32", "RECIPE_CHANNEL128_F32", "RECIPE_NVFP4_1X16", "DTYPE_F32", "DTYPE_BF16", "STATUS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libgq.so")

RECIPE_MXFP8_1X32, RECIPE_CHANNEL128_F32, RECIPE_NVFP4_1X16 = 0, 1, 2
DTYPE_F32, DTYPE_BF16 = 0, 1
STATUS = {0: "GQ_OK", -1: "GQ_ERR_INVALID_ARG", -2: "GQ_ERR_ALIGNMENT", -3: "GQ_ERR_SPLITS",
          -4: "GQ_ERR_UNSUPPORTED", -5: "GQ_ERR_CUDA", -6: "GQ_ERR_TIMEOUT",
          -7: "GQ_ERR_SHAPE_MISMATCH"}


class Recipe(C.Structure):
    _fields_ = [("kind", C.c_int32), ("rowwise", C.c_int32), ("colwise", C.c_int32),
                ("zero_scale", C.c_float)]


class Quantized(C.Structure):
    """Mirror of ``gq_quantized``."""
    _fields_ = [("num_groups", C.c_int32), ("reserved0", C.c_int32), ("rows_cap", C.c_int64),
                ("cols", C.c_int64), ("recipe", Recipe), ("row_data", C.c_void_p),
                ("row_scale", C.c_void_p), ("col_data", C.c_void_p), ("col_scale", C.c_void_p),
                ("row_scale_bytes", C.c_uint64), ("col_scale_bytes", C.c_uint64), ("amax", C.c_void_p)]


class GQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {gq_status_string(status)}")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libgq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"libgq.so is not built ({_LIB_PATH}); run "
                "`python -c 'import __graft_entry__ as g; g.build()'` or "
                "`python -m moe_grouped_gemm_group_gb300.build`")
        lib = C.CDLL(_LIB_PATH)
        vp, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
        qp = C.POINTER(Quantized)
        lib.gq_status_string.restype = C.c_char_p
        lib.gq_status_string.argtypes = [i32]
        lib.gq_version.restype = i32
        lib.gq_version.argtypes = []
        lib.gq_scale_bytes_bound.restype = C.c_uint64
        lib.gq_scale_bytes_bound.argtypes = [C.POINTER(Recipe), i32, i64, i64]
        lib.gq_split_scan.restype = i32
        lib.gq_split_scan.argtypes = [vp, i32, i64, i64, i32, vp, vp, vp]
        lib.gq_quantize.restype = i32
        lib.gq_quantize.argtypes = [vp, i64, i64, vp, i32, C.POINTER(Recipe), qp, vp, vp]
        for f in (lib.gq_gemm_fprop, lib.gq_gemm_dgrad):
            f.restype = i32
            f.argtypes = [qp, qp, vp, i32, i64, i64, vp, i32, vp, vp]
        lib.gq_gemm_wgrad.restype = i32
        lib.gq_gemm_wgrad.argtypes = [qp, qp, vp, i32, i64, i64, vp, i32, vp, C.c_uint64, vp, vp]
        lib.gq_gemm_fprop_bias.restype = i32
        lib.gq_gemm_fprop_bias.argtypes = [qp, qp, vp, i32, i64, i64, vp, i32, vp, i32, vp, vp]
        lib.gq_dbias_workspace_bytes.restype = C.c_uint64
        lib.gq_dbias_workspace_bytes.argtypes = [i32, i64, i64]
        lib.gq_quantize_dbias.restype = i32
        lib.gq_quantize_dbias.argtypes = [vp, i64, i64, vp, i32, C.POINTER(Recipe), qp, vp, vp, C.c_uint64,
                                          vp, vp]
        lib.gq_gemm_fprop_srelu_quant.restype = i32
        lib.gq_gemm_fprop_srelu_quant.argtypes = [qp, qp, vp, i32, i64, i64, vp, i32, vp, vp, i32, qp, vp, vp]
        lib.gq_gemm_fprop_swiglu_quant.restype = i32
        lib.gq_gemm_fprop_swiglu_quant.argtypes = [qp, qp, vp, i32, i64, i64, vp, i32, vp, vp, i32, qp, vp, vp]
        lib.gq_gemm_wgrad_noalloc.restype = i32
        lib.gq_gemm_wgrad_noalloc.argtypes = [qp, qp, vp, i32, i64, i64, vp, i32, vp, vp]
        lib.gq_check_wait_limit.restype = i32
        lib.gq_check_wait_limit.argtypes = [vp, vp, vp]
        _lib = lib
        return lib


# --------------------------------------------------------------------------- #
# marshalling helpers                                                          #
# --------------------------------------------------------------------------- #

def _ptr(t, name: str, required: bool = True):
    """Device address of a CUDA tensor (None -> NULL)."""
    if t is None:
        if required:
            raise ValueError(f"{name} is required")
        return None
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"{name} must be a CUDA tensor (device memory), got {getattr(t, 'device', type(t))}")
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


def _check(st: int, what: str):
    if st != 0:
        raise GQError(st, what)


class GroupedTensor:
    """A grouped quantised tensor: the torch buffers that back a
    ``gq_quantized`` descriptor, kept alive together with it."""

    def __init__(self, num_groups, rows_cap, cols, recipe: Recipe, row_data=None, row_scale=None,
                 col_data=None, col_scale=None, amax=None):
        self.row_data, self.row_scale = row_data, row_scale
        self.col_data, self.col_scale = col_data, col_scale
        self.amax = amax
        self.desc = Quantized()
        d = self.desc
        d.num_groups, d.rows_cap, d.cols = num_groups, rows_cap, cols
        d.recipe = Recipe(recipe.kind, recipe.rowwise, recipe.colwise, recipe.zero_scale)
        for name in ("row_data", "row_scale", "col_data", "col_scale", "amax"):
            t = getattr(self, name)
            setattr(d, name, None if t is None else _ptr(t, name).value)
        d.row_scale_bytes = 0 if row_scale is None else row_scale.numel() * row_scale.element_size()
        d.col_scale_bytes = 0 if col_scale is None else col_scale.numel() * col_scale.element_size()

    @property
    def num_groups(self):
        return self.desc.num_groups

    @property
    def rows_cap(self):
        return self.desc.rows_cap

    @property
    def cols(self):
        return self.desc.cols


def alloc_quantized(rows_cap: int, cols: int, num_groups: int, recipe: Recipe, device="cuda",
                    fill: int | None = None) -> GroupedTensor:
    """Allocate (with torch) the buffers of a grouped quantised tensor.

    NVFP4 codes take half a byte: rowwise [rows_cap, cols/2], columnwise
    stored transposed [cols, rows_cap/2], plus the fp32 [num_groups] amax.
    ``fill`` optionally pre-fills every byte (a canary for tests)."""
    import torch
    nbytes = gq_scale_bytes_bound(recipe, num_groups, rows_cap, cols)
    if nbytes == 0 and rows_cap > 0:
        raise ValueError("bad recipe or shape for gq_scale_bytes_bound")
    mk = torch.empty if fill is None else (lambda *a, **k: torch.full(*a, fill, **k))

    nv = recipe.kind == RECIPE_NVFP4_1X16

    def data(colwise=False):
        if nv:
            shape = (cols, rows_cap // 2) if colwise else (rows_cap, cols // 2)
            return mk(shape, dtype=torch.uint8, device=device)
        return mk((rows_cap, cols), dtype=torch.uint8, device=device)

    def scale():
        if recipe.kind == RECIPE_CHANNEL128_F32:
            t = torch.empty((max(nbytes, 4) // 4,), dtype=torch.float32, device=device)
            if fill is not None:
                t.view(torch.uint8).fill_(fill)
            return t
        return mk((max(nbytes, 16),), dtype=torch.uint8, device=device)

    rd = data() if recipe.rowwise else None
    rs = scale() if recipe.rowwise else None
    cd = data(True) if recipe.colwise else None
    cs = scale() if recipe.colwise else None
    am = None
    if nv:
        am = torch.empty((max(num_groups, 4),), dtype=torch.float32, device=device)
        if fill is not None:
            am.view(torch.uint8).fill_(fill)
    return GroupedTensor(num_groups, rows_cap, cols, recipe, rd, rs, cd, cs, am)


# --------------------------------------------------------------------------- #
# the C ABI                                                                    #
# --------------------------------------------------------------------------- #

def gq_status_string(status: int) -> str:
    try:
        return load().gq_status_string(int(status)).decode()
    except RuntimeError:
        return STATUS.get(int(status), "unknown gq_status")


def gq_version() -> int:
    return int(load().gq_version())


def gq_scale_bytes_bound(recipe: Recipe, num_groups: int, rows_cap: int, cols: int) -> int:
    return int(load().gq_scale_bytes_bound(C.byref(recipe), num_groups, rows_cap, cols))


def gq_split_scan(splits, num_groups: int, rows_cap: int, cols: int, recipe_kind: int, table,
                  status, stream=None) -> None:
    st = load().gq_split_scan(_ptr(splits, "splits", False), num_groups, rows_cap, cols,
                              recipe_kind, _ptr(table, "table"), _ptr(status, "status"),
                              _stream(stream))
    _check(st, "gq_split_scan")


def gq_quantize(x, splits, num_groups: int, recipe: Recipe, out: GroupedTensor, status,
                stream=None) -> None:
    """Quantise bf16 ``x`` [rows_cap, cols] into ``out``; ``splits`` is a CUDA
    int32 tensor of ``num_groups`` split sizes or None (uniform split)."""
    rows_cap, cols = (int(x.shape[0]), int(x.shape[1])) if x is not None else (0, out.cols)
    st = load().gq_quantize(_ptr(x, "x", rows_cap > 0), rows_cap, cols,
                            _ptr(splits, "splits", False), num_groups, C.byref(recipe),
                            C.byref(out.desc), _ptr(status, "status"), _stream(stream))
    _check(st, "gq_quantize")


def gq_gemm_fprop(x: GroupedTensor, w: GroupedTensor, splits, num_groups: int, n: int, k: int, y,
                  out_dtype: int, status, stream=None) -> None:
    st = load().gq_gemm_fprop(C.byref(x.desc), C.byref(w.desc), _ptr(splits, "splits", False),
                              num_groups, n, k, _ptr(y, "y"), out_dtype, _ptr(status, "status"),
                              _stream(stream))
    _check(st, "gq_gemm_fprop")


def gq_gemm_fprop_bias(x: GroupedTensor, w: GroupedTensor, splits, num_groups: int, n: int, k: int, bias,
                       y, out_dtype: int, status, stream=None) -> None:
    """gq_gemm_fprop plus the per-group bias ``bias`` ([num_groups, n], fp32
    or bf16 CUDA tensor) added in the GEMM's epilogue."""
    import torch
    bias_dtype = DTYPE_BF16 if bias.dtype == torch.bfloat16 else DTYPE_F32
    if bias.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError(f"bias must be fp32 or bf16, got {bias.dtype}")
    st = load().gq_gemm_fprop_bias(C.byref(x.desc), C.byref(w.desc), _ptr(splits, "splits", False),
                                   num_groups, n, k, _ptr(bias, "bias"), bias_dtype, _ptr(y, "y"), out_dtype,
                                   _ptr(status, "status"), _stream(stream))
    _check(st, "gq_gemm_fprop_bias")


def gq_gemm_fprop_srelu_quant(x: GroupedTensor, w: GroupedTensor, splits, num_groups: int, n: int, k: int,
                              probs, y, out_dtype: int, act_out: GroupedTensor, status, bias=None,
                              stream=None) -> None:
    """fc1 forward with ScaledSReLU (probs[r] * relu(y)^2) and the MXFP8 row +
    column quantisation of the activation fused into the epilogue; ``y``
    receives the pre-activation result, ``act_out`` the quantised activation."""
    import torch
    bias_dtype = 0
    if bias is not None:
        if bias.dtype not in (torch.bfloat16, torch.float32):
            raise ValueError(f"bias must be fp32 or bf16, got {bias.dtype}")
        bias_dtype = DTYPE_BF16 if bias.dtype == torch.bfloat16 else DTYPE_F32
    st = load().gq_gemm_fprop_srelu_quant(C.byref(x.desc), C.byref(w.desc), _ptr(splits, "splits", False),
                                          num_groups, n, k, _ptr(bias, "bias", False), bias_dtype,
                                          _ptr(probs, "probs"), _ptr(y, "y"), out_dtype, C.byref(act_out.desc),
                                          _ptr(status, "status"), _stream(stream))
    _check(st, "gq_gemm_fprop_srelu_quant")


def gq_gemm_fprop_swiglu_quant(x: GroupedTensor, w: GroupedTensor, splits, num_groups: int, n: int, k: int,
                               probs, y, out_dtype: int, act_out: GroupedTensor, status, bias=None,
                               stream=None) -> None:
    """fc1 forward with ScaledSwiGLU ((silu(gate) * linear) * probs[r], gate =
    y[:, :n/2], linear = y[:, n/2:]) and the MXFP8 row + column quantisation
    of the [R, n/2] activation fused into the epilogue."""
    import torch
    bias_dtype = 0
    if bias is not None:
        if bias.dtype not in (torch.bfloat16, torch.float32):
            raise ValueError(f"bias must be fp32 or bf16, got {bias.dtype}")
        bias_dtype = DTYPE_BF16 if bias.dtype == torch.bfloat16 else DTYPE_F32
    st = load().gq_gemm_fprop_swiglu_quant(C.byref(x.desc), C.byref(w.desc), _ptr(splits, "splits", False),
                                           num_groups, n, k, _ptr(bias, "bias", False), bias_dtype,
                                           _ptr(probs, "probs"), _ptr(y, "y"), out_dtype, C.byref(act_out.desc),
                                           _ptr(status, "status"), _stream(stream))
    _check(st, "gq_gemm_fprop_swiglu_quant")


def gq_dbias_workspace_bytes(num_groups: int, rows_cap: int, cols: int) -> int:
    return int(load().gq_dbias_workspace_bytes(num_groups, rows_cap, cols))


def gq_quantize_dbias(x, splits, num_groups: int, recipe: Recipe, out: GroupedTensor, dbias, workspace,
                      status, stream=None) -> None:
    """gq_quantize (MX) of a gradient ``x`` fused with its per-group column
    sums into ``dbias`` (fp32 [num_groups, cols]); ``workspace`` is a CUDA
    tensor of at least gq_dbias_workspace_bytes(...) bytes."""
    rows_cap, cols = (int(x.shape[0]), int(x.shape[1])) if x is not None else (0, out.cols)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = load().gq_quantize_dbias(_ptr(x, "x", rows_cap > 0), rows_cap, cols, _ptr(splits, "splits", False),
                                  num_groups, C.byref(recipe), C.byref(out.desc), _ptr(dbias, "dbias"),
                                  _ptr(workspace, "workspace"), ws_bytes, _ptr(status, "status"),
                                  _stream(stream))
    _check(st, "gq_quantize_dbias")


def gq_gemm_dgrad(dy: GroupedTensor, w: GroupedTensor, splits, num_groups: int, n: int, k: int,
                  dx, out_dtype: int, status, stream=None) -> None:
    st = load().gq_gemm_dgrad(C.byref(dy.desc), C.byref(w.desc), _ptr(splits, "splits", False),
                              num_groups, n, k, _ptr(dx, "dx"), out_dtype, _ptr(status, "status"),
                              _stream(stream))
    _check(st, "gq_gemm_dgrad")


WGRAD_WORKSPACE_BYTES = 256       # GQ_WGRAD_WORKSPACE_BYTES


def gq_gemm_wgrad(dy: GroupedTensor, x: GroupedTensor, splits, num_groups: int, n: int, k: int,
                  dw, accumulate: bool, status, stream=None, workspace="new") -> None:
    """`workspace`: a CUDA uint8 tensor of at least WGRAD_WORKSPACE_BYTES
    bytes (run-time tile order; not shared by calls that may overlap), None
    for the static order, or "new" (default) for a fresh one from torch's
    allocator on dw's device."""
    if isinstance(workspace, str):
        import torch
        workspace = torch.empty(WGRAD_WORKSPACE_BYTES, dtype=torch.uint8, device=dw.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().gq_gemm_wgrad(C.byref(dy.desc), C.byref(x.desc), _ptr(splits, "splits", False),
                              num_groups, n, k, _ptr(dw, "dw"), int(bool(accumulate)),
                              _ptr(workspace, "workspace", False), ws_bytes,
                              _ptr(status, "status"), _stream(stream))
    _check(st, "gq_gemm_wgrad")


def gq_gemm_wgrad_noalloc(dy: GroupedTensor, x: GroupedTensor, splits, num_groups: int, n: int, k: int,
                          dw, accumulate: bool, status, stream=None) -> None:
    """gq_gemm_wgrad without a caller workspace: the library's own per-device
    array serves as one (calls that may overlap on the GPU must not be
    issued; see include/gq.h)."""
    st = load().gq_gemm_wgrad_noalloc(C.byref(dy.desc), C.byref(x.desc), _ptr(splits, "splits", False),
                                      num_groups, n, k, _ptr(dw, "dw"), int(bool(accumulate)),
                                      _ptr(status, "status"), _stream(stream))
    _check(st, "gq_gemm_wgrad_noalloc")


def gq_check_wait_limit(status, report=None, stream=None) -> None:
    """Run the library's bounded-wait failure path once: a wait that never
    completes gives up after the limit and leaves GQ_ERR_TIMEOUT in
    ``status`` (int32 CUDA tensor); ``report`` is None or a CUDA int64
    tensor of 4 elements (per warp: nanoseconds waited, 1 if the wait
    completed)."""
    st = load().gq_check_wait_limit(_ptr(status, "status"), _ptr(report, "report", False), _stream(stream))
    _check(st, "gq_check_wait_limit")
