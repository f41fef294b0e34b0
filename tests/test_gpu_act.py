"""GPU parity of the fc1 forward with ScaledSReLU and the MXFP8 quantisation
of fc2's input fused into the GEMM epilogue (gq_gemm_fprop_srelu_quant).

The pre-activation result Y is checked against the oracle's fprop (+ bias)
at the GEMMs' tolerance.  The codes and scales are decided from the fp32
accumulator, so the oracle takes that decision from the same fp32 values:
ScaledSReLU + MX quantisation of the GPU's own fp32 Y must give the kernel's
codes and scale bytes bit for bit.  The quantised activation does not depend
on Y's output dtype; rows past the live total are never written."""
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


def _run(x, w, splits, G, N, K, probs, out_dtype, bias=None):
    st = status_dev()
    xq, _ = quantize(x, splits, G, mx_recipe(True, False), status=st)
    wq, _ = quantize(w, None, G, mx_recipe(True, False), status=st)
    R = x.shape[0]
    act = gq.alloc_quantized(R, N, G, mx_recipe(True, True), DEV, fill=0xAB)
    tdt = torch.float32 if out_dtype == gq.DTYPE_F32 else torch.bfloat16
    y = torch.full((R, N), float("nan"), dtype=tdt, device=DEV)
    gq.gq_gemm_fprop_srelu_quant(xq, wq, splits_dev(splits), G, N, K, probs, y, out_dtype, act, st, bias=bias)
    check_status(st)
    return y, act


@pytest.mark.parametrize("splits,N,with_bias", [([96, 0, 160, 32, 256], 256, False),
                                                 ([128, 384, 0, 32], 512, True),
                                                 ([512], 256, True)])
def test_fused_srelu_quant_matches_oracle(splits, N, with_bias):
    splits = np.array(splits, np.int32)
    G, L, K, pad = len(splits), int(splits.sum()), 384, 64
    R = L + pad
    x = np.concatenate([W.normal_bf16((L, K), 81), W.uniform_bf16((pad, K), 82, -4, 4)])
    w = W.normal_bf16((G * N, K), 83, scale=0.05)
    rng = np.random.default_rng(84)
    probs_h = rng.uniform(0.0, 1.0, R).astype(np.float32)
    probs = torch.from_numpy(probs_h).to(DEV)
    b_bits = W.normal_bf16((G, N), 85, scale=0.5)
    bias = bf16_dev(b_bits) if with_bias else None

    y, act = _run(x, w, splits, G, N, K, probs, gq.DTYPE_F32, bias)
    yh = host(y)
    want = O.gemm_fprop(O.quantize_mx(x, splits, G, colwise=False), O.quantize_mx(w, None, G, colwise=False),
                        splits, G, N, K)
    if with_bias:
        want = O.grouped_bias_add(want, W.bf16_bits_to_f32(b_bits).astype(np.float64), splits, G)
    off = np.concatenate([[0], np.cumsum(splits)])
    for g in range(G):
        a, b = int(off[g]), int(off[g + 1])
        if b > a:
            e = np.linalg.norm(yh[a:b] - want[a:b]) / np.linalg.norm(want[a:b])
            assert e <= REL_TOL, f"Y group {g}: rel err {e}"
    assert np.all(np.isnan(yh[L:]))

    ref = O.srelu_quantize_mx(np.where(np.isnan(yh), 0, yh).astype(np.float32), probs_h, splits, G)
    assert np.array_equal(host(act.row_data)[:L], ref.row_data[:L]), "rowwise codes"
    assert np.array_equal(host(act.col_data)[:L], ref.col_data[:L]), "columnwise codes"
    n_scale = len(ref.row_scale)
    assert np.array_equal(host(act.row_scale)[:n_scale], ref.row_scale), "rowwise scales"
    assert np.array_equal(host(act.col_scale)[:n_scale], ref.col_scale), "columnwise scales"
    assert np.all(host(act.row_data)[L:] == 0xAB) and np.all(host(act.col_data)[L:] == 0xAB)

    # the quantised activation comes from the fp32 accumulator whatever Y's dtype
    yb, act_b = _run(x, w, splits, G, N, K, probs, gq.DTYPE_BF16, bias)
    for name in ("row_data", "col_data", "row_scale", "col_scale"):
        assert torch.equal(getattr(act_b, name), getattr(act, name)), name


def test_fused_srelu_quant_refuses_narrow_outputs():
    splits = np.array([128], np.int32)
    st = status_dev()
    x = W.normal_bf16((128, 256), 86)
    w = W.normal_bf16((384, 256), 87)
    xq, _ = quantize(x, splits, 1, mx_recipe(True, False), status=st)
    wq, _ = quantize(w, None, 1, mx_recipe(True, False), status=st)
    act = gq.alloc_quantized(128, 384, 1, mx_recipe(True, True), DEV)
    y = torch.empty((128, 384), device=DEV)
    probs = torch.ones(128, device=DEV)
    with pytest.raises(gq.GQError, match="GQ_ERR_UNSUPPORTED"):
        gq.gq_gemm_fprop_srelu_quant(xq, wq, splits_dev(splits), 1, 384, 256, probs, y, gq.DTYPE_F32, act, st)


# --------------------------------------------------------------------------- #
# ScaledSwiGLU (gq_gemm_fprop_swiglu_quant)                                    #
# --------------------------------------------------------------------------- #

def _run_glu(x, w, splits, G, N, K, probs, out_dtype, bias=None):
    st = status_dev()
    xq, _ = quantize(x, splits, G, mx_recipe(True, False), status=st)
    wq, _ = quantize(w, None, G, mx_recipe(True, False), status=st)
    R = x.shape[0]
    act = gq.alloc_quantized(R, N // 2, G, mx_recipe(True, True), DEV, fill=0xAB)
    tdt = torch.float32 if out_dtype == gq.DTYPE_F32 else torch.bfloat16
    y = torch.full((R, N), float("nan"), dtype=tdt, device=DEV)
    gq.gq_gemm_fprop_swiglu_quant(xq, wq, splits_dev(splits), G, N, K, probs, y, out_dtype, act, st, bias=bias)
    check_status(st)
    return y, act


@pytest.mark.parametrize("splits,N,with_bias", [([96, 0, 160, 32, 256], 256, False),
                                                 ([128, 384, 0, 32], 512, True),
                                                 ([512], 768, True)])
def test_fused_swiglu_quant_matches_oracle(splits, N, with_bias):
    """Y (both halves) at the GEMMs' tolerance; the [R, N/2] activation's codes
    and scales bit for bit against the oracle's ScaledSwiGLU + MX quantisation
    of the GPU's own fp32 Y (the oracle computes the same exp, fp32 op by op)."""
    splits = np.array(splits, np.int32)
    G, L, K, pad = len(splits), int(splits.sum()), 384, 64
    R = L + pad
    x = np.concatenate([W.normal_bf16((L, K), 181), W.uniform_bf16((pad, K), 182, -4, 4)])
    w = W.normal_bf16((G * N, K), 183, scale=0.08)
    rng = np.random.default_rng(184)
    probs_h = rng.uniform(0.0, 1.0, R).astype(np.float32)
    probs = torch.from_numpy(probs_h).to(DEV)
    b_bits = W.normal_bf16((G, N), 185, scale=0.5)
    bias = bf16_dev(b_bits) if with_bias else None

    y, act = _run_glu(x, w, splits, G, N, K, probs, gq.DTYPE_F32, bias)
    yh = host(y)
    want = O.gemm_fprop(O.quantize_mx(x, splits, G, colwise=False), O.quantize_mx(w, None, G, colwise=False),
                        splits, G, N, K)
    if with_bias:
        want = O.grouped_bias_add(want, W.bf16_bits_to_f32(b_bits).astype(np.float64), splits, G)
    off = np.concatenate([[0], np.cumsum(splits)])
    for g in range(G):
        a, b = int(off[g]), int(off[g + 1])
        if b > a:
            e = np.linalg.norm(yh[a:b] - want[a:b]) / np.linalg.norm(want[a:b])
            assert e <= REL_TOL, f"Y group {g}: rel err {e}"
    assert np.all(np.isnan(yh[L:]))

    ref = O.swiglu_quantize_mx(np.where(np.isnan(yh), 0, yh).astype(np.float32), probs_h, splits, G)
    assert np.array_equal(host(act.row_data)[:L], ref.row_data[:L]), "rowwise codes"
    assert np.array_equal(host(act.col_data)[:L], ref.col_data[:L]), "columnwise codes"
    n_scale = len(ref.row_scale)
    assert np.array_equal(host(act.row_scale)[:n_scale], ref.row_scale), "rowwise scales"
    assert np.array_equal(host(act.col_scale)[:n_scale], ref.col_scale), "columnwise scales"
    assert np.all(host(act.row_data)[L:] == 0xAB) and np.all(host(act.col_data)[L:] == 0xAB)

    yb, act_b = _run_glu(x, w, splits, G, N, K, probs, gq.DTYPE_BF16, bias)
    for name in ("row_data", "col_data", "row_scale", "col_scale"):
        assert torch.equal(getattr(act_b, name), getattr(act, name)), name
    assert torch.equal(yb[:L].float(), y[:L].to(torch.bfloat16).float())


def test_fused_swiglu_shape_checks():
    splits = np.array([128], np.int32)
    st = status_dev()
    x = W.normal_bf16((128, 256), 186)
    w = W.normal_bf16((512, 256), 187)
    xq, _ = quantize(x, splits, 1, mx_recipe(True, False), status=st)
    wq, _ = quantize(w, None, 1, mx_recipe(True, False), status=st)
    y = torch.empty((128, 512), device=DEV)
    probs = torch.ones(128, device=DEV)
    wrong = gq.alloc_quantized(128, 512, 1, mx_recipe(True, True), DEV)      # must be n / 2 = 256 wide
    with pytest.raises(gq.GQError, match="GQ_ERR_SHAPE_MISMATCH"):
        gq.gq_gemm_fprop_swiglu_quant(xq, wq, splits_dev(splits), 1, 512, 256, probs, y, gq.DTYPE_F32, wrong, st)


# --------------------------------------------------------------------------- #
# full size: moe_e64_zipf fc1 in the bench's launch configuration             #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("act_kind", ["srelu", "swiglu"])
def test_fused_activation_moe_e64_zipf_fc1(act_kind):
    """E = 64, hidden 7168, 65536 Zipf-routed tokens + 1024 garbage rows, fc1
    width 2048 (ScaledSReLU) or 2 x 2048 (ScaledSwiGLU): the fused kernel's
    fp32 Y equals the plain fprop's bit for bit (same tiles, same contraction
    order; the plain fprop is held to the oracle at these shapes in
    test_gpu_fullsize.py), and the activation's codes and scale regions equal
    the oracle's ScaledSReLU / ScaledSwiGLU + MX quantisation of that Y, byte
    for byte, over every live row."""
    w = W.workload("moe_e64_zipf")
    E, R, L, K = w.num_groups, w.rows_cap, w.live_rows, w.hidden
    N = w.ffn if act_kind == "srelu" else 2 * w.ffn
    x = W.device_activation(w, K, 60, device=DEV)
    wt = W.device_normal_bf16((E * N, K), w.seed, 0.02, 61, DEV)
    g = torch.Generator(device=DEV).manual_seed(62)
    probs = torch.rand(R, generator=g, device=DEV)
    sp = torch.as_tensor(w.splits).to(DEV)
    st = status_dev()
    rec = mx_recipe(True, False)
    qx = gq.alloc_quantized(R, K, E, rec, DEV)
    qw = gq.alloc_quantized(E * N, K, E, rec, DEV)
    gq.gq_quantize(x, sp, E, rec, qx, st)
    gq.gq_quantize(wt, None, E, rec, qw, st)
    del x, wt
    na = N if act_kind == "srelu" else N // 2
    act = gq.alloc_quantized(R, na, E, mx_recipe(True, True), DEV, fill=0xAB)
    y = torch.full((R, N), float("nan"), device=DEV)
    fused = gq.gq_gemm_fprop_srelu_quant if act_kind == "srelu" else gq.gq_gemm_fprop_swiglu_quant
    fused(qx, qw, sp, E, N, K, probs, y, gq.DTYPE_F32, act, st)
    y_plain = torch.full((R, N), float("nan"), device=DEV)
    gq.gq_gemm_fprop(qx, qw, sp, E, N, K, y_plain, gq.DTYPE_F32, st)
    torch.cuda.synchronize()
    check_status(st)
    assert torch.equal(y[:L], y_plain[:L]), "fused Y differs from the plain fprop"
    assert bool(torch.isnan(y[L:]).all()), "rows past the live total were written"

    yh = host(y[:L])
    ph = host(probs)
    yfull = np.zeros((R, N), np.float32)
    yfull[:L] = yh
    ref = (O.srelu_quantize_mx if act_kind == "srelu" else O.swiglu_quantize_mx)(yfull, ph, w.splits, E)
    for name in ("row_data", "col_data"):
        got = host(getattr(act, name))
        bad = np.flatnonzero((got[:L] != getattr(ref, name)[:L]).ravel())
        assert bad.size == 0, f"{name}: {bad.size} codes differ, first at {np.unravel_index(bad[0], (L, na))}"
        assert np.all(got[L:] == 0xAB), f"{name} written past the live rows"
    n_scale = len(ref.row_scale)
    for name in ("row_scale", "col_scale"):
        got = host(getattr(act, name))
        assert np.array_equal(got[:n_scale], getattr(ref, name)), name
        assert np.all(got[n_scale:] == 0xAB), f"{name} written past the grouped extent"
