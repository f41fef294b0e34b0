"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports
every function include/gq.h declares, and its host-side checks answer before
anything is launched.  No call here reaches a kernel launch: every call either
fails a host check or touches no device pointer."""
import ctypes as C
import os
import re
import subprocess

import pytest

import moe_grouped_gemm_group_gb300 as gq
from moe_grouped_gemm_group_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gq.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return gq.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("gq_quantize", "gq_gemm_fprop", "gq_gemm_dgrad", "gq_gemm_wgrad", "gq_split_scan"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", gq.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in declared_functions():
        assert name in exported, f"{name} not exported (C linkage) by libgq.so"
        assert hasattr(lib, name)


def test_status_strings_and_version(lib):
    assert gq.gq_version() >> 16 == 1
    for code, name in gq.STATUS.items():
        assert gq.gq_status_string(code).startswith(name)
    assert "unknown" in gq.gq_status_string(12345)


def test_scale_bytes_bound(lib):
    mx = gq.Recipe(gq.RECIPE_MXFP8_1X32, 1, 1, 0.0)
    ch = gq.Recipe(gq.RECIPE_CHANNEL128_F32, 0, 1, 1e-30)
    assert gq.gq_scale_bytes_bound(mx, 64, 66560, 7168) == 512 * 56 * (520 + 64)
    assert gq.gq_scale_bytes_bound(ch, 4, 768, 2048) == 4 * 2048 * 6
    assert gq.gq_scale_bytes_bound(mx, 1, 128, 100) == 0          # cols % 128
    assert gq.gq_scale_bytes_bound(mx, 0, 128, 128) == 0          # no groups
    assert gq.gq_scale_bytes_bound(gq.Recipe(7, 1, 1, 0.0), 1, 128, 128) == 0


def _desc(G, R, Ccols, kind=0, row=1, col=1):
    d = gq.Quantized()
    d.num_groups, d.rows_cap, d.cols = G, R, Ccols
    d.recipe = gq.Recipe(kind, row, col, 0.0)
    return d


def test_quantize_host_checks_need_no_gpu(lib):
    """Each call fails a host check, so no pointer is dereferenced and
    nothing is launched (pointers below are never touched)."""
    fake = C.c_void_p(0x10000)
    st = C.c_void_p(0x20000)
    mx = gq.Recipe(gq.RECIPE_MXFP8_1X32, 1, 1, 0.0)
    d = _desc(2, 256, 256)
    assert lib.gq_quantize(fake, 256, 256, None, 2, C.byref(mx), C.byref(d), None, None) == -1  # no status
    assert lib.gq_quantize(fake, 256, 200, None, 2, C.byref(mx), C.byref(d), st, None) == -2    # cols % 128
    assert lib.gq_quantize(fake, 255, 256, None, 2, C.byref(mx), C.byref(d), st, None) == -2    # R % G
    assert lib.gq_quantize(fake, 256, 256, None, 0, C.byref(mx), C.byref(d), st, None) == -1    # G = 0
    assert lib.gq_quantize(fake, 256, 256, None, 2000, C.byref(mx), C.byref(d), st, None) == -1  # G > 1024
    big = _desc(1, 1 << 31, 256)
    assert lib.gq_quantize(fake, 1 << 31, 256, None, 1, C.byref(mx), C.byref(big), st, None) == -1  # rows >= 2^31
    assert lib.gq_quantize(fake, 256, 256, None, 4, C.byref(mx), C.byref(d), st, None) == -7    # descriptor G
    d2 = _desc(2, 256, 256)                                                                     # no buffers
    assert lib.gq_quantize(fake, 256, 256, None, 2, C.byref(mx), C.byref(d2), st, None) == -1
    d3 = _desc(2, 256, 256, kind=1, row=0, col=1)
    ch_row = gq.Recipe(gq.RECIPE_CHANNEL128_F32, 1, 1, 1e-30)
    assert lib.gq_quantize(fake, 256, 256, None, 2, C.byref(ch_row), C.byref(d3), st, None) == -4
    odd = C.c_void_p(0x10008)                                                                   # not 16B aligned
    assert lib.gq_quantize(odd, 256, 256, None, 2, C.byref(mx), C.byref(d), st, None) == -2


def test_gemm_host_checks_need_no_gpu(lib):
    st = C.c_void_p(0x20000)
    out = C.c_void_p(0x30000)
    x = _desc(1, 256, 256, row=1, col=0)
    x.row_data, x.row_scale, x.row_scale_bytes = 0x40000, 0x50000, 1 << 20
    w = _desc(1, 128, 256, row=1, col=0)
    w.row_data, w.row_scale, w.row_scale_bytes = 0x60000, 0x70000, 1 << 20
    # k disagrees with the descriptors
    assert lib.gq_gemm_fprop(C.byref(x), C.byref(w), None, 1, 128, 384, out, 0, st, None) == -7
    # n not a multiple of 128
    assert lib.gq_gemm_fprop(C.byref(x), C.byref(w), None, 1, 96, 256, out, 0, st, None) == -2
    # bad output dtype
    assert lib.gq_gemm_fprop(C.byref(x), C.byref(w), None, 1, 128, 256, out, 9, st, None) == -4
    # dgrad needs the weight columnwise
    dy = _desc(1, 256, 128, row=1, col=0)
    dy.row_data, dy.row_scale, dy.row_scale_bytes = 0x40000, 0x50000, 1 << 20
    assert lib.gq_gemm_dgrad(C.byref(dy), C.byref(w), None, 1, 128, 256, out, 0, st, None) in (-4, -7)
    # wgrad needs columnwise operands, same recipe, accumulate in {0, 1}
    assert lib.gq_gemm_wgrad(C.byref(dy), C.byref(x), None, 1, 128, 256, out, 0, None, 0, st, None) in (-4, -7)
    assert lib.gq_gemm_wgrad(C.byref(dy), C.byref(x), None, 1, 128, 256, out, 2, None, 0, st, None) == -1
    xc = _desc(1, 256, 256, kind=1, row=0, col=1)
    assert lib.gq_gemm_wgrad(C.byref(dy), C.byref(xc), None, 1, 128, 256, out, 0, None, 0, st, None) == -4
    # a workspace smaller than GQ_WGRAD_WORKSPACE_BYTES, or not 16-byte aligned
    ws = C.c_void_p(0x80000)
    assert lib.gq_gemm_wgrad(C.byref(dy), C.byref(x), None, 1, 128, 256, out, 0, ws, 255, st, None) == -1
    assert lib.gq_gemm_wgrad(C.byref(dy), C.byref(x), None, 1, 128, 256, out, 0, C.c_void_p(0x80008), 256,
                             st, None) == -2
    # scale capacity below the bound
    x2 = _desc(1, 256, 256, row=1, col=0)
    x2.row_data, x2.row_scale, x2.row_scale_bytes = 0x40000, 0x50000, 16
    assert lib.gq_gemm_fprop(C.byref(x2), C.byref(w), None, 1, 128, 256, out, 0, st, None) == -1


def test_noalloc_wgrad_refuses_too_many_tiles_without_a_gpu(lib):
    # 2^31 output tiles exceed the claim counter: refused on the host
    assert lib.gq_gemm_wgrad_noalloc(None, None, None, 1024, 1 << 17, 1 << 19, None, 1, None, None) == -1


def test_bias_entry_points_host_checks_need_no_gpu(lib):
    st = C.c_void_p(0x20000)
    out = C.c_void_p(0x30000)
    x = _desc(1, 256, 256, row=1, col=0)
    x.row_data, x.row_scale, x.row_scale_bytes = 0x40000, 0x50000, 1 << 20
    w = _desc(1, 128, 256, row=1, col=0)
    w.row_data, w.row_scale, w.row_scale_bytes = 0x60000, 0x70000, 1 << 20
    # no bias, a bias dtype that is neither fp32 nor bf16, a misaligned bias
    assert lib.gq_gemm_fprop_bias(C.byref(x), C.byref(w), None, 1, 128, 256, None, 0, out, 0, st, None) == -1
    assert lib.gq_gemm_fprop_bias(C.byref(x), C.byref(w), None, 1, 128, 256, C.c_void_p(0x80000), 5, out, 0,
                                  st, None) == -4
    assert lib.gq_gemm_fprop_bias(C.byref(x), C.byref(w), None, 1, 128, 256, C.c_void_p(0x80004), 0, out, 0,
                                  st, None) == -2
    # bias-grad workspace: the bound, and a refusal below it
    assert gq.gq_dbias_workspace_bytes(4, 1024, 256) == 4 * 256 * (8 + 4)
    assert gq.gq_dbias_workspace_bytes(4, 1024, 200) == 0
    mx = gq.Recipe(gq.RECIPE_MXFP8_1X32, 1, 1, 0.0)
    d = _desc(1, 256, 256)
    assert lib.gq_quantize_dbias(C.c_void_p(0x10000), 256, 256, None, 1, C.byref(mx), C.byref(d),
                                 C.c_void_p(0x90000), C.c_void_p(0xa0000), 16, st, None) == -1


def test_binding_refuses_host_tensors(lib):
    torch = pytest.importorskip("torch")
    x = torch.zeros((128, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        gq._ptr(x, "x")


def test_descriptor_mirror_matches_the_c_layout(tmp_path):
    """The ctypes mirror of gq_quantized has the C struct's size and field
    offsets (gcc compiles a probe against include/gq.h on the host)."""
    names = [f[0] for f in gq.Quantized._fields_]
    src = tmp_path / "probe.c"
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"gq.h\"\nint main(void){\n"
                   + "printf(\"%zu\\n\", sizeof(gq_quantized));\n"
                   + "".join(f"printf(\"%zu\\n\", offsetof(gq_quantized, {n}));\n" for n in names)
                   + "return 0;}\n")
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), "-o", str(exe), str(src)], check=True)
    vals = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert vals[0] == C.sizeof(gq.Quantized)
    for n, off in zip(names, vals[1:]):
        assert getattr(gq.Quantized, n).offset == off, n


def test_nvfp4_scale_bound_and_host_checks(lib):
    nv = gq.Recipe(gq.RECIPE_NVFP4_1X16, 1, 1, 0.0)
    assert gq.gq_scale_bytes_bound(nv, 64, 66560, 7168) == 512 * 112 * (520 + 64)
    fake = C.c_void_p(0x10000)
    st = C.c_void_p(0x20000)
    d = _desc(2, 256, 256, kind=gq.RECIPE_NVFP4_1X16)
    d.row_data = d.row_scale = d.col_data = d.col_scale = 0x30000
    d.row_scale_bytes = d.col_scale_bytes = 1 << 20
    # no amax buffer
    assert lib.gq_quantize(fake, 256, 256, None, 2, C.byref(nv), C.byref(d), st, None) == -1
    d.amax = 0x40002                                                     # not 4-byte aligned
    assert lib.gq_quantize(fake, 256, 256, None, 2, C.byref(nv), C.byref(d), st, None) == -2
    d.amax = 0x40000
    d2 = _desc(2, 240, 256, kind=gq.RECIPE_NVFP4_1X16)                   # colwise needs rows_cap % 32
    d2.row_data = d2.row_scale = d2.col_data = d2.col_scale = 0x30000
    d2.row_scale_bytes = d2.col_scale_bytes = 1 << 20
    d2.amax = 0x40000
    assert lib.gq_quantize(fake, 240, 256, None, 2, C.byref(nv), C.byref(d2), st, None) == -2
    d.row_scale_bytes = 16                                               # scale capacity
    assert lib.gq_quantize(fake, 256, 256, None, 2, C.byref(nv), C.byref(d), st, None) == -1
    # GEMMs: NVFP4 needs n and k multiples of 256, and both operands NVFP4
    x = _desc(2, 256, 128, kind=gq.RECIPE_NVFP4_1X16)
    w = _desc(2, 256, 128, kind=gq.RECIPE_NVFP4_1X16)
    for q in (x, w):
        q.row_data = q.row_scale = q.col_data = q.col_scale = 0x30000
        q.row_scale_bytes = q.col_scale_bytes = 1 << 20
        q.amax = 0x40000
    y = C.c_void_p(0x50000)
    assert lib.gq_gemm_fprop(C.byref(x), C.byref(w), None, 2, 128, 128, y, 0, st, None) == -4
    assert lib.gq_gemm_dgrad(C.byref(x), C.byref(w), None, 2, 128, 128, y, 0, st, None) == -4
    assert lib.gq_gemm_wgrad(C.byref(x), C.byref(x), None, 2, 128, 128, y, 0, None, 0, st, None) == -4
    mx = _desc(2, 256, 256)
    x256 = _desc(2, 256, 256, kind=gq.RECIPE_NVFP4_1X16)
    x256.row_data = x256.row_scale = 0x30000
    x256.row_scale_bytes = 1 << 20
    x256.amax = 0x40000
    assert lib.gq_gemm_fprop(C.byref(x256), C.byref(mx), None, 2, 128, 256, y, 0, st, None) in (-4, -7)
    # bias with NVFP4 operands is not provided
    assert lib.gq_gemm_fprop_bias(C.byref(x), C.byref(w), None, 2, 256, 256, y, 0, y, 0, st, None) == -4


def test_check_wait_limit_host_checks(lib):
    """A NULL status word and misaligned pointers are refused before launch."""
    st = C.c_void_p(0x20000)
    assert lib.gq_check_wait_limit(None, None, None) == -1
    assert lib.gq_check_wait_limit(C.c_void_p(0x20002), None, None) == -2
    assert lib.gq_check_wait_limit(st, C.c_void_p(0x10004), None) == -2


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without libgq.so every call raises: there is no fallback path."""
    monkeypatch.setattr(gq, "_LIB_PATH", str(tmp_path / "libgq.so"))
    monkeypatch.setattr(gq, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        gq.load()
    with pytest.raises(RuntimeError):
        gq.gq_version()
    with pytest.raises(RuntimeError):
        gq.gq_scale_bytes_bound(gq.Recipe(gq.RECIPE_MXFP8_1X32, 1, 1, 0.0), 1, 128, 128)
