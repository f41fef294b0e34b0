"""The C ABI driven from a plain C program, with no Python binding and no
torch: tests/c_abi_check.c is built with gcc against include/gq.h, linked to
libgq.so and the CUDA runtime, and run in its own process.  It allocates its
device buffers with cudaMalloc, quantises X, W and dY (MXFP8), runs the
grouped fprop and the k-grouped wgrad, and checks two host-side refusals;
its outputs are compared here with the oracle.  It then resets the device
(cudaDeviceReset), so that the library meets a new CUDA context: its cached
per-context set-up (kernel attributes, the no-alloc wgrad's array address)
must be redone there, and the no-alloc wgrad must give the same bits."""
import os
import subprocess

import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_grouped_gemm_group_gb300 as gq  # noqa: E402
from _gpu_util import REL_TOL  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime.h")):
            return cand
    pytest.skip("CUDA toolkit headers not found")


def test_c_program_quantize_fprop_wgrad(tmp_path):
    gq.load()
    lib = gq.library_path()
    cuda = _cuda_home()
    exe = tmp_path / "c_abi_check"
    subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), os.path.join(HERE, "c_abi_check.c"), "-o", str(exe),
                    lib, "-L", os.path.join(cuda, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{os.path.dirname(lib)}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"],
                   check=True)
    G, K, N, pad = 3, 256, 256, 96
    splits = np.array([128, 0, 96], np.int32)
    L = int(splits.sum())
    R = L + pad
    x = np.concatenate([W.normal_bf16((L, K), 81), W.uniform_bf16((pad, K), 82, -4, 4)])
    dy = np.concatenate([W.normal_bf16((L, N), 83), W.uniform_bf16((pad, N), 84, -4, 4)])
    w = W.normal_bf16((G * N, K), 85, scale=0.02)
    splits.tofile(tmp_path / "splits.bin")
    x.tofile(tmp_path / "x.bin")
    w.tofile(tmp_path / "w.bin")
    dy.tofile(tmp_path / "dy.bin")
    subprocess.run([str(exe), str(tmp_path), str(G), str(R), str(K), str(N)], check=True, timeout=300)

    status, refused_cols, refused_shape, reset_status, reset_equal = (
        int(v) for v in (tmp_path / "status.txt").read_text().split())
    assert status == 0
    assert reset_status == 0, "device status after cudaDeviceReset"
    assert reset_equal == 1, "the no-alloc wgrad changed after cudaDeviceReset"
    assert refused_cols == -2            # GQ_ERR_ALIGNMENT: cols % 128
    assert refused_shape == -7           # GQ_ERR_SHAPE_MISMATCH: descriptor cols
    xrow = np.fromfile(tmp_path / "xrow.bin", np.uint8).reshape(R, K)
    y = np.fromfile(tmp_path / "y.bin", np.float32).reshape(R, N)
    dw = np.fromfile(tmp_path / "dw.bin", np.float32).reshape(G, N, K)

    ox = O.quantize_mx(x, splits, G)
    assert np.array_equal(xrow[:L], ox.row_data[:L])
    want_y = O.gemm_fprop(O.quantize_mx(x, splits, G, colwise=False), O.quantize_mx(w, None, G, colwise=False),
                          splits, G, N, K)
    want_dw = O.gemm_wgrad(O.quantize_mx(dy, splits, G, rowwise=False), O.quantize_mx(x, splits, G, rowwise=False),
                           splits, G, N, K)
    off = np.concatenate([[0], np.cumsum(splits)])
    for g in range(G):
        a, b = int(off[g]), int(off[g + 1])
        if b == a:
            assert np.all(dw[g] == 0), f"group {g} is empty"
            continue
        e = np.linalg.norm(y[a:b] - want_y[a:b]) / np.linalg.norm(want_y[a:b])
        assert e <= REL_TOL, f"fprop group {g}: rel err {e}"
        e = np.linalg.norm(dw[g] - want_dw[g]) / np.linalg.norm(want_dw[g])
        assert e <= REL_TOL, f"wgrad group {g}: rel err {e}"
