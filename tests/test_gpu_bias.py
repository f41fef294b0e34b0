"""GPU parity of the grouped bias add fused into fprop and of the bias
gradient fused into the MX quantisation of dY, through the C ABI, against
the oracle (TransformerEngine PR 3224: launch_grouped_bias_add after the
grouped GEMM, with its zero-row guard; the backward's dbiases).

Bar: per-group relative Frobenius error <= 1e-5 (bf16 output: within one
bf16 ulp of the oracle rounded to bf16); codes and scales of the fused
quantisation bitwise equal to gq_quantize's; empty groups exactly 0; rows
past the live total untouched; repeated calls bitwise identical."""
import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_grouped_gemm_group_gb300 as gq  # noqa: E402
from _gpu_util import (DEV, REL_TOL, bf16_dev, check_status, host, mx_recipe, quantize,  # noqa: E402
                       splits_dev, status_dev)


def _bounds(splits):
    off = np.concatenate([[0], np.cumsum(splits)])
    return [(int(off[g]), int(off[g + 1])) for g in range(len(splits))]


def _close_rows(got, want, splits, what):
    for g, (a, b) in enumerate(_bounds(splits)):
        if b == a:
            continue
        e = np.linalg.norm(got[a:b].astype(np.float64) - want[a:b]) / np.linalg.norm(want[a:b])
        assert e <= REL_TOL, f"{what}: group {g} rel err {e}"


@pytest.mark.parametrize("N,bias_dtype", [(256, "f32"), (384, "f32"), (256, "bf16"), (384, "bf16")])
def test_fprop_bias_matches_oracle(N, bias_dtype):
    splits = np.array([96, 0, 160, 32, 256], np.int32)
    G, L, K, pad = len(splits), int(splits.sum()), 512, 64
    x = np.concatenate([W.normal_bf16((L, K), 61), W.uniform_bf16((pad, K), 62, -4, 4)])
    w = W.normal_bf16((G * N, K), 63, scale=0.02)
    b_bits = W.normal_bf16((G, N), 64, scale=0.5)
    b64 = W.bf16_bits_to_f32(b_bits).astype(np.float64)
    st = status_dev()
    xq, _ = quantize(x, splits, G, mx_recipe(True, False), status=st)
    wq, _ = quantize(w, None, G, mx_recipe(True, False), status=st)
    bias = bf16_dev(b_bits) if bias_dtype == "bf16" else torch.from_numpy(b64.astype(np.float32)).to(DEV)
    y = torch.full((L + pad, N), float("nan"), device=DEV)
    gq.gq_gemm_fprop_bias(xq, wq, splits_dev(splits), G, N, K, bias, y, gq.DTYPE_F32, st)
    check_status(st)
    got = host(y)
    want = O.grouped_bias_add(O.gemm_fprop(O.quantize_mx(x, splits, G, colwise=False),
                                           O.quantize_mx(w, None, G, colwise=False), splits, G, N, K),
                              b64, splits, G)
    _close_rows(got, want, splits, "fprop+bias")
    assert np.all(np.isnan(got[L:])), "wrote rows past the live total"

    # bf16 output: within one bf16 ulp of the oracle rounded to bf16
    yb = torch.full((L + pad, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    gq.gq_gemm_fprop_bias(xq, wq, splits_dev(splits), G, N, K, bias, yb, gq.DTYPE_BF16, st)
    check_status(st)
    gb = host(yb.float())[:L]
    wl = want[:L]
    wb = W.bf16_bits_to_f32(W.f32_to_bf16_bits(wl.astype(np.float32))).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(wl), 1e-30))) - 7)
    assert np.all(np.abs(gb - wb) <= ulp + 1e-30)


def test_fprop_bias_zero_bias_equals_fprop_bitwise():
    splits = np.array([128, 64], np.int32)
    G, N, K = 2, 256, 256
    x = W.normal_bf16((192, K), 65)
    w = W.normal_bf16((G * N, K), 66, scale=0.02)
    st = status_dev()
    xq, _ = quantize(x, splits, G, mx_recipe(True, False), status=st)
    wq, _ = quantize(w, None, G, mx_recipe(True, False), status=st)
    y0 = torch.empty((192, N), device=DEV)
    y1 = torch.empty((192, N), device=DEV)
    gq.gq_gemm_fprop(xq, wq, splits_dev(splits), G, N, K, y0, gq.DTYPE_F32, st)
    gq.gq_gemm_fprop_bias(xq, wq, splits_dev(splits), G, N, K, torch.zeros((G, N), device=DEV), y1,
                          gq.DTYPE_F32, st)
    check_status(st)
    assert torch.equal(y0.view(torch.int32), y1.view(torch.int32))


def _dbias_call(x_bits, splits, G, recipe, st):
    R, Cc = x_bits.shape
    q = gq.alloc_quantized(R, Cc, G, recipe, DEV, fill=0xAB)
    db = torch.full((G, Cc), float("nan"), device=DEV)
    ws = torch.empty(gq.gq_dbias_workspace_bytes(G, R, Cc), dtype=torch.uint8, device=DEV)
    gq.gq_quantize_dbias(bf16_dev(x_bits), splits_dev(splits), G, recipe, q, db, ws, st)
    return q, db


@pytest.mark.parametrize("splits,C", [([96, 0, 224, 32, 160], 384), ([512], 256), ([0, 0, 64], 128),
                                      ([1056, 32, 416], 512)])
def test_quantize_dbias_matches_oracle(splits, C):
    splits = np.array(splits, np.int32)
    G, L, pad = len(splits), int(splits.sum()), 96
    x = np.concatenate([W.normal_bf16((L, C), 67), W.uniform_bf16((pad, C), 68, -4, 4)])
    st = status_dev()
    rec = mx_recipe(True, True)
    q, db = _dbias_call(x, splits, G, rec, st)
    ref, _ = quantize(x, splits, G, rec, fill=0xAB, status=st)
    check_status(st)
    for a, b in (("row_data", "row_data"), ("col_data", "col_data")):
        assert torch.equal(getattr(q, a)[:L], getattr(ref, b)[:L]), a
    for a in ("row_scale", "col_scale"):
        assert torch.equal(getattr(q, a), getattr(ref, a)), a
    got = host(db)
    want = O.grouped_bias_grad(x, splits, G)
    for g in range(G):
        if splits[g] == 0:
            assert np.all(got[g] == 0), f"group {g} is empty: its bias grad must be 0"
        else:
            e = np.linalg.norm(got[g].astype(np.float64) - want[g]) / np.linalg.norm(want[g])
            assert e <= REL_TOL, f"group {g}: rel err {e}"
    # a second call gives the same bits
    _, db2 = _dbias_call(x, splits, G, rec, st)
    check_status(st)
    assert torch.equal(db.view(torch.int32), db2.view(torch.int32))


def test_quantize_dbias_all_empty_and_rowwise_only():
    st = status_dev()
    x = W.normal_bf16((128, 256), 69)
    _, db = _dbias_call(x, np.array([0, 0], np.int32), 2, mx_recipe(True, False), st)
    check_status(st)
    assert torch.all(db == 0)
    splits = np.array([64, 64], np.int32)
    _, db = _dbias_call(x, splits, 2, mx_recipe(True, False), st)
    check_status(st)
    want = O.grouped_bias_grad(x, splits, 2)
    got = host(db)
    for g in range(2):
        assert np.linalg.norm(got[g] - want[g]) / np.linalg.norm(want[g]) <= REL_TOL


def test_bias_host_checks():
    st = status_dev()
    x = W.normal_bf16((128, 256), 70)
    rec = mx_recipe(True, True)
    q = gq.alloc_quantized(128, 256, 1, rec, DEV)
    db = torch.empty((1, 256), device=DEV)
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(gq.GQError, match="GQ_ERR_INVALID_ARG"):
        gq.gq_quantize_dbias(bf16_dev(x), None, 1, rec, q, db, small, st)
    ch = gq.Recipe(gq.RECIPE_CHANNEL128_F32, 0, 1, 1e-30)
    qc = gq.alloc_quantized(128, 256, 1, ch, DEV)
    ws = torch.empty(gq.gq_dbias_workspace_bytes(1, 128, 256), dtype=torch.uint8, device=DEV)
    with pytest.raises(gq.GQError, match="GQ_ERR_UNSUPPORTED"):
        gq.gq_quantize_dbias(bf16_dev(x), None, 1, ch, qc, db, ws, st)


def test_bias_paths_moe_e64_zipf():
    """moe_e64_zipf sizes (64 experts, 65536 Zipf-routed tokens + 1024
    garbage rows, hidden 7168, fc1 width 2048).  fprop with a bf16 per-expert
    bias equals the plain fprop plus the bias bit for bit: the epilogue adds
    it to the fp32 accumulator once, and the plain fprop is held to the
    oracle at these shapes in test_gpu_fullsize.py.  The bias gradient fused
    into the quantisation of a [66560, 7168] dY: codes and scales bitwise
    equal to gq_quantize's, and 128 sampled columns of every group's column
    sums against the oracle per group at the GEMMs' tolerance."""
    w = W.workload("moe_e64_zipf")
    E, R, L, K, N = w.num_groups, w.rows_cap, w.live_rows, w.hidden, w.ffn
    splits = np.asarray(w.splits, np.int32)
    sp = torch.as_tensor(splits).to(DEV)
    st = status_dev()
    rec = mx_recipe(True, False)
    x = W.device_activation(w, K, 80, device=DEV)
    wt = W.device_normal_bf16((E * N, K), w.seed, 0.02, 81, DEV)
    b = W.device_normal_bf16((E, N), w.seed, 0.5, 82, DEV)
    qx = gq.alloc_quantized(R, K, E, rec, DEV)
    qw = gq.alloc_quantized(E * N, K, E, rec, DEV)
    gq.gq_quantize(x, sp, E, rec, qx, st)
    gq.gq_quantize(wt, None, E, rec, qw, st)
    del x, wt
    y0 = torch.full((R, N), float("nan"), device=DEV)
    y1 = torch.full((R, N), float("nan"), device=DEV)
    gq.gq_gemm_fprop(qx, qw, sp, E, N, K, y0, gq.DTYPE_F32, st)
    gq.gq_gemm_fprop_bias(qx, qw, sp, E, N, K, b, y1, gq.DTYPE_F32, st)
    check_status(st)
    rows_g = torch.repeat_interleave(torch.arange(E, device=DEV), sp.long())
    want = y0[:L] + b.float()[rows_g]
    assert torch.equal(y1[:L].view(torch.int32), want.view(torch.int32)), "fprop + bias != fprop, then + bias"
    assert bool(torch.isnan(y1[L:]).all()), "rows past the live total were written"
    del qx, qw, y0, y1, want

    dy = W.device_activation(w, K, 83, device=DEV)
    rec2 = mx_recipe(True, True)
    q = gq.alloc_quantized(R, K, E, rec2, DEV, fill=0xAB)
    db = torch.full((E, K), float("nan"), device=DEV)
    ws = torch.empty(gq.gq_dbias_workspace_bytes(E, R, K), dtype=torch.uint8, device=DEV)
    gq.gq_quantize_dbias(dy, sp, E, rec2, q, db, ws, st)
    ref = gq.alloc_quantized(R, K, E, rec2, DEV, fill=0xAB)
    gq.gq_quantize(dy, sp, E, rec2, ref, st)
    check_status(st)
    for name in ("row_data", "col_data"):
        assert torch.equal(getattr(q, name)[:L], getattr(ref, name)[:L]), name
    for name in ("row_scale", "col_scale"):
        assert torch.equal(getattr(q, name), getattr(ref, name)), name
    cols = np.sort(np.random.default_rng(84).choice(K, 128, replace=False))   # the oracle takes 128-column multiples
    idx = torch.as_tensor(cols, device=DEV)
    bits = dy[:L].index_select(1, idx).contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    want = O.grouped_bias_grad(bits, splits, E)
    got = host(db)[:, cols]
    for g in range(E):
        if splits[g] == 0:
            assert np.all(got[g] == 0), f"group {g} is empty: its bias grad must be 0"
        else:
            e = np.linalg.norm(got[g].astype(np.float64) - want[g]) / np.linalg.norm(want[g])
            assert e <= REL_TOL, f"group {g}: rel err {e}"
