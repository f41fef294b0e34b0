"""The largest group count the library takes (1024), with many empty and
32-row groups: the split scan held in every CTA's shared memory at its full
size, the tile-to-group search over it, and the wgrad's in-CTA sort of the
groups by size for its run-time tile order.  Quantisation bitwise against
the oracle; fprop (128-column tiles), dgrad and wgrad (256-column tiles, both
tile orders) at the GEMMs' tolerance; the same for the NVFP4 recipe."""
import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_grouped_gemm_group_gb300 as gq  # noqa: E402
from _gpu_util import (DEV, REL_TOL, check_status, host, mx_recipe, quantize, splits_dev,  # noqa: E402
                       status_dev)

G, N, K = 1024, 128, 256


@pytest.fixture(scope="module")
def data():
    rng = np.random.default_rng(91)
    splits = (rng.integers(0, 5, G) * 32).astype(np.int32)       # 0 .. 128 rows, about a fifth empty
    L = int(splits.sum())
    R = L + 64
    x = np.concatenate([W.normal_bf16((L, K), 92), W.uniform_bf16((64, K), 93, -4, 4)])
    dy = np.concatenate([W.normal_bf16((L, N), 94), W.uniform_bf16((64, N), 95, -4, 4)])
    w = W.normal_bf16((G * N, K), 96, scale=0.05)
    return splits, L, R, x, dy, w


def _close_groups(got, want, bounds, what):
    for g, (a, b) in enumerate(bounds):
        if b == a:
            continue
        e = np.linalg.norm(got[a:b].astype(np.float64) - want[a:b]) / np.linalg.norm(want[a:b])
        assert e <= REL_TOL, f"{what}: group {g} rel err {e}"


def test_quantize_1024_groups_bitwise(data):
    splits, L, R, x, _, _ = data
    q, st = quantize(x, splits, G, mx_recipe(True, True))
    check_status(st)
    ref = O.quantize_mx(x, splits, G)
    assert np.array_equal(host(q.row_data)[:L], ref.row_data[:L])
    assert np.array_equal(host(q.col_data)[:L], ref.col_data[:L])
    n = len(ref.row_scale)
    assert np.array_equal(host(q.row_scale)[:n], ref.row_scale)
    assert np.array_equal(host(q.col_scale)[:n], ref.col_scale)


def test_gemms_1024_groups(data):
    splits, L, R, x, dy, w = data
    off = np.concatenate([[0], np.cumsum(splits)])
    bounds = [(int(off[g]), int(off[g + 1])) for g in range(G)]
    st = status_dev()
    xq, _ = quantize(x, splits, G, mx_recipe(True, True), status=st)
    dq, _ = quantize(dy, splits, G, mx_recipe(True, True), status=st)
    wq, _ = quantize(w, None, G, mx_recipe(True, True), status=st)
    sp = splits_dev(splits)
    y = torch.empty((R, N), device=DEV)
    dx = torch.empty((R, K), device=DEV)
    gq.gq_gemm_fprop(xq, wq, sp, G, N, K, y, gq.DTYPE_F32, st)
    gq.gq_gemm_dgrad(dq, wq, sp, G, N, K, dx, gq.DTYPE_F32, st)
    dws = []
    for ws in ("new", None):                 # run-time tile order, static order
        dw = torch.full((G, N, K), float("nan"), device=DEV)
        gq.gq_gemm_wgrad(dq, xq, sp, G, N, K, dw, False, st, workspace=ws)
        dws.append(dw)
    check_status(st)
    assert torch.equal(dws[0].view(torch.int32), dws[1].view(torch.int32))

    oxr = O.quantize_mx(x, splits, G, colwise=False)
    odr = O.quantize_mx(dy, splits, G, colwise=False)
    owr = O.quantize_mx(w, None, G, colwise=False)
    owc = O.quantize_mx(w, None, G, rowwise=False)
    _close_groups(host(y), O.gemm_fprop(oxr, owr, splits, G, N, K), bounds, "fprop")
    _close_groups(host(dx), O.gemm_dgrad(odr, owc, splits, G, N, K), bounds, "dgrad")
    want = O.gemm_wgrad(O.quantize_mx(dy, splits, G, rowwise=False), O.quantize_mx(x, splits, G, rowwise=False),
                        splits, G, N, K)
    got = host(dws[0])
    for g in range(G):
        if splits[g] == 0:
            assert np.all(got[g] == 0), f"group {g} is empty"
        else:
            e = np.linalg.norm(got[g].astype(np.float64) - want[g]) / np.linalg.norm(want[g])
            assert e <= REL_TOL, f"wgrad group {g}: rel err {e}"


def test_nvfp4_1024_groups(data):
    """The NVFP4 recipe at the maximum group count: per-group amax, codes and
    scales bitwise; fprop, dgrad and wgrad (the last 64-row block of every
    32-row group half live) at the GEMMs' tolerance."""
    splits, L, R, x, _, _ = data
    N = 256                                  # NVFP4 GEMMs take n, k multiples of 256
    dy = np.concatenate([W.normal_bf16((L, N), 97), W.uniform_bf16((R - L, N), 98, -4, 4)])
    w = W.normal_bf16((G * N, K), 99, scale=0.05)
    off = np.concatenate([[0], np.cumsum(splits)])
    bounds = [(int(off[g]), int(off[g + 1])) for g in range(G)]
    nv = gq.Recipe(gq.RECIPE_NVFP4_1X16, 1, 1, 0.0)
    st = status_dev()

    def q(bits, sp):
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)
        out = gq.alloc_quantized(t.shape[0], t.shape[1], G, nv, DEV)
        gq.gq_quantize(t, splits_dev(sp), G, nv, out, st)
        return out

    xq, dq, wq = q(x, splits), q(dy, splits), q(w, None)
    sp = splits_dev(splits)
    y = torch.empty((R, N), device=DEV)
    dx = torch.empty((R, K), device=DEV)
    dw = torch.full((G, N, K), float("nan"), device=DEV)
    gq.gq_gemm_fprop(xq, wq, sp, G, N, K, y, gq.DTYPE_F32, st)
    gq.gq_gemm_dgrad(dq, wq, sp, G, N, K, dx, gq.DTYPE_F32, st)
    gq.gq_gemm_wgrad(dq, xq, sp, G, N, K, dw, False, st)
    check_status(st)
    ox, ody, ow = O.quantize_nvfp4(x, splits, G), O.quantize_nvfp4(dy, splits, G), O.quantize_nvfp4(w, None, G)
    assert np.array_equal(host(xq.amax)[:G], ox.amax)
    assert np.array_equal(host(xq.row_data)[:L], ox.row_data[:L])
    assert np.array_equal(host(xq.col_data)[:, :L // 2], ox.col_data[:, :L // 2])
    nb = O.scale_bytes_nvfp4(splits, G, R, K)
    assert np.array_equal(host(xq.row_scale)[:nb], ox.row_scale[:nb])
    assert np.array_equal(host(xq.col_scale)[:nb], ox.col_scale[:nb])
    _close_groups(host(y), O.gemm_nvfp4("fprop", ox, ow, splits, G, N, K), bounds, "nvfp4 fprop")
    _close_groups(host(dx), O.gemm_nvfp4("dgrad", ody, ow, splits, G, N, K), bounds, "nvfp4 dgrad")
    want = O.gemm_nvfp4("wgrad", ody, ox, splits, G, N, K)
    got = host(dw)
    for g in range(G):
        if splits[g] == 0:
            assert np.all(got[g] == 0), f"group {g} is empty"
        else:
            e = np.linalg.norm(got[g].astype(np.float64) - want[g]) / np.linalg.norm(want[g])
            assert e <= REL_TOL, f"nvfp4 wgrad group {g}: rel err {e}"
