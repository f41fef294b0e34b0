"""Pins for the oracle's grouped GEMMs (fprop, dgrad, k-grouped wgrad).

* Exact arithmetic: inputs built so that every 32-element block quantises
  without rounding (4-bit integers times a per-block power of two), so the
  grouped GEMM must equal numpy's fp64 matmul of the original values bit for
  bit; the per-block exponents make any misplaced scale or transposed operand
  visible.
* The pages' printed numbers: padded vs unpadded wgrad rel_err 0 with no
  non-finite values (TransformerEngine issue 3484), and the k-grouped wgrad
  reference norm 1.311e-03 with no blow-up (DeepGEMM issue 365).
* Closed forms and invariants: the expected wgrad norm sqrt(n*H*k)*s1*s2,
  <Y, dY> = <W, dW> = <X, dX>, accumulate semantics, empty groups.
"""
import json
import os

import numpy as np
import pytest

import oracle as O
import workloads as W
from workloads import bf16_bits_to_f32, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ints(rng, shape):
    return rng.integers(-14, 15, size=shape).astype(np.float64)


def rowwise_exact(rng, rows, cols, live_rows=None):
    """Values i * 2^s[r, c//32] with |i| <= 14: every rowwise 32-block is
    exactly representable after MX scaling."""
    s = rng.integers(-6, 7, size=(rows, cols // 32))
    return _ints(rng, (rows, cols)) * np.exp2(np.repeat(s, 32, axis=1))


def colwise_exact(rng, splits, rows, cols):
    """Values i * 2^s[32-row block, c]: every columnwise 32-block of every
    group (groups start on multiples of 32) is exactly representable."""
    s = rng.integers(-6, 7, size=(rows // 32, cols))
    return _ints(rng, (rows, cols)) * np.exp2(np.repeat(s, 32, axis=0))


def to_bits(v):
    b = f32_to_bf16_bits(v.astype(np.float32))
    assert np.array_equal(bf16_bits_to_f32(b).astype(np.float64), v)  # exact in bf16
    return b


SPLITS = [np.array(s, np.int32) for s in ([96], [64, 0, 160], [32, 128, 32, 0, 96])]


@pytest.mark.parametrize("splits", SPLITS)
def test_fprop_exact(splits):
    rng = np.random.default_rng(11)
    G, N, K = len(splits), 256, 384
    L = int(splits.sum())
    R = L + 32
    x = rowwise_exact(rng, R, K)
    w = rowwise_exact(rng, G * N, K)
    xq = O.quantize_mx(to_bits(x), splits, G, colwise=False)
    wq = O.quantize_mx(to_bits(w), None, G, colwise=False)
    y = O.gemm_fprop(xq, wq, splits, G, N, K)
    off = np.concatenate([[0], np.cumsum(splits)])
    for g in range(G):
        want = x[off[g]:off[g + 1]] @ w[g * N:(g + 1) * N].T
        np.testing.assert_array_equal(y[off[g]:off[g + 1]], want)
    assert np.all(np.isnan(y[L:]))                      # rows past L untouched


@pytest.mark.parametrize("splits", SPLITS)
def test_dgrad_exact(splits):
    rng = np.random.default_rng(12)
    G, N, K = len(splits), 256, 384
    L = int(splits.sum())
    R = L + 64
    dy = rowwise_exact(rng, R, N)
    w = colwise_exact(rng, None, G * N, K)
    dyq = O.quantize_mx(to_bits(dy), splits, G, colwise=False)
    wq = O.quantize_mx(to_bits(w), None, G, rowwise=False)
    dx = O.gemm_dgrad(dyq, wq, splits, G, N, K)
    off = np.concatenate([[0], np.cumsum(splits)])
    for g in range(G):
        want = dy[off[g]:off[g + 1]] @ w[g * N:(g + 1) * N]
        np.testing.assert_array_equal(dx[off[g]:off[g + 1]], want)
    assert np.all(np.isnan(dx[L:]))


@pytest.mark.parametrize("splits", SPLITS)
def test_wgrad_exact_live_rows_only(splits):
    rng = np.random.default_rng(13)
    G, N, K = len(splits), 256, 384
    L = int(splits.sum())
    R = L + 96
    dy = colwise_exact(rng, splits, R, N)
    x = colwise_exact(rng, splits, R, K)
    dyq = O.quantize_mx(to_bits(dy), splits, G, rowwise=False)
    xq = O.quantize_mx(to_bits(x), splits, G, rowwise=False)
    dw = O.gemm_wgrad(dyq, xq, splits, G, N, K)
    off = np.concatenate([[0], np.cumsum(splits)])
    for g in range(G):
        want = dy[off[g]:off[g + 1]].T @ x[off[g]:off[g + 1]]
        np.testing.assert_array_equal(dw[g], want)
        if splits[g] == 0:
            assert np.all(dw[g] == 0) and not np.any(np.signbit(dw[g]))


def test_wgrad_accumulate_and_empty_group():
    rng = np.random.default_rng(14)
    splits = np.array([64, 0, 96], np.int32)
    G, N, K = 3, 128, 256
    R = 192
    dyq = O.quantize_mx(W.normal_bf16((R, N), 1), splits, G, rowwise=False)
    xq = O.quantize_mx(W.normal_bf16((R, K), 2), splits, G, rowwise=False)
    init = rng.standard_normal((G, N, K))
    fresh = O.gemm_wgrad(dyq, xq, splits, G, N, K)
    acc = O.gemm_wgrad(dyq, xq, splits, G, N, K, accumulate=True, init=init)
    np.testing.assert_array_equal(acc, init + fresh)
    np.testing.assert_array_equal(acc[1], init[1])      # empty group left as it was
    assert np.all(fresh[1] == 0)


def test_cross_identity_fprop_dgrad_wgrad():
    """<Y, dY> = <W, dW> = <X, dX> with exactly quantisable inputs: ties the
    three contractions' operand orientations to one another."""
    rng = np.random.default_rng(15)
    splits = np.array([64, 32, 0, 128], np.int32)
    G, N, K = 4, 128, 256
    R = 256
    x = _ints(rng, (R, K)) * 2.0 ** -3
    w = _ints(rng, (G * N, K)) * 2.0 ** -5
    dy = _ints(rng, (R, N)) * 2.0 ** -4
    xq = O.quantize_mx(to_bits(x), splits, G)
    wq = O.quantize_mx(to_bits(w), None, G)
    dyq = O.quantize_mx(to_bits(dy), splits, G)
    y = O.gemm_fprop(xq, wq, splits, G, N, K)
    dx = O.gemm_dgrad(dyq, wq, splits, G, N, K)
    dw = O.gemm_wgrad(dyq, xq, splits, G, N, K)
    L = int(splits.sum())
    a = np.sum(y[:L] * dy[:L])
    b = np.sum(w.reshape(G, N, K) * dw)
    c = np.sum(dx[:L] * x[:L])
    assert a == b == c and a != 0


def test_accuracy_bound_on_random_data():
    """On N(0,1) data the fp64 result on dequantised operands stays within
    the e4m3 rounding bound of the bf16 product (each operand rounded to
    within 2^-4 relative, plus a subnormal floor)."""
    splits = np.array([128, 64, 96], np.int32)
    G, N, K = 3, 128, 512
    R = 320
    xb, wb = W.normal_bf16((R, K), 21), W.normal_bf16((G * N, K), 22)
    x, w = bf16_bits_to_f32(xb).astype(np.float64), bf16_bits_to_f32(wb).astype(np.float64)
    y = O.gemm_fprop(O.quantize_mx(xb, splits, G), O.quantize_mx(wb, None, G), splits, G, N, K)
    off = np.concatenate([[0], np.cumsum(splits)])
    for g in range(G):
        xs, ws = x[off[g]:off[g + 1]], w[g * N:(g + 1) * N]
        exact = xs @ ws.T
        bound = (2 * 2.0 ** -4 + 2.0 ** -8) * (np.abs(xs) @ np.abs(ws).T) + 1e-9
        err = np.abs(y[off[g]:off[g + 1]] - exact)
        assert np.all(err <= bound)
        assert np.linalg.norm(err) / np.linalg.norm(exact) < 0.05


def test_padded_single_group_wgrad_matches_unpadded():
    """TransformerEngine issue 3484: fills 0.0 and 3.0 past sum(split_sizes)
    must give rel_err 0 and no non-finite value against the unpadded wgrad."""
    gold = json.load(open(os.path.join(GOLDEN, "padded_wgrad_expected.json")))
    H = gold["hidden"]
    ref_w = W.workload("padded_single_group", rows_cap=gold["live_rows"], pad_kind="none")
    x0, dy0 = ref_w.activation(H, 0), ref_w.activation(H, 1)
    s = ref_w.splits
    ref = O.gemm_wgrad(O.quantize_mx(dy0, s, 1), O.quantize_mx(x0, s, 1), s, 1, H, H)
    for label, arm in gold["arms"].items():
        pad = W.fill_bf16((gold["pad_rows"], H), arm["fill"])
        x, dy = np.concatenate([x0, pad]), np.concatenate([dy0, pad])
        got = O.gemm_wgrad(O.quantize_mx(dy, s, 1), O.quantize_mx(x, s, 1), s, 1, H, H)
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel == arm["rel_err"], label
        assert int((~np.isfinite(got)).sum()) == arm["non_finite"] and got.size == arm["numel"]


@pytest.fixture(scope="module")
def kgrouped():
    gold = json.load(open(os.path.join(GOLDEN, "kgrouped_wgrad_reference_norm.json")))
    w = W.workload("kgrouped_zero_channel")
    dy, x = W.kgrouped_zero_channel_operands(w)
    outs = {}
    for sf in gold["sf_vals"]:
        dyq = O.quantize_channel(dy, w.splits, 4, zero_scale=sf)
        xq = O.quantize_channel(x, w.splits, 4, zero_scale=sf)
        outs[sf] = O.gemm_wgrad(dyq, xq, w.splits, 4, w.hidden, w.ffn)
    return gold, w, dy, x, outs


def test_kgrouped_reference_norm_from_the_page(kgrouped):
    """Max per-expert norm of the k-grouped wgrad lands on the page's printed
    reference max 1.311e-03; no expert exceeds max(100*||ref||, 1)."""
    gold, w, dy, x, outs = kgrouped
    for sf, dw in outs.items():
        norms = np.linalg.norm(dw.reshape(4, -1), axis=1)
        assert abs(norms.max() / gold["reference_max_norm"] - 1) < 0.02, (sf, norms)
        assert np.all(norms <= np.maximum(gold["blowup_factor"] * norms, gold["blowup_floor"]))
        assert np.all(np.isfinite(dw))


def test_kgrouped_closed_form_norms(kgrouped):
    """E||dY_e^T X_e||_F = sqrt(n*H*k) * s_dy * s_x for independent N(0, s^2)
    entries; each expert lands within 3 %."""
    gold, w, dy, x, outs = kgrouped
    norms = np.linalg.norm(outs[1e-30].reshape(4, -1), axis=1)
    for e, k in enumerate(gold["ks"]):
        want = np.sqrt(gold["hidden"] * gold["ffn"] * k) * gold["grad_scale"] * gold["act_scale"]
        assert abs(norms[e] / want - 1) < 0.03, (e, norms[e], want)


def test_kgrouped_zero_channel_and_sf_val_independence(kgrouped):
    """An all-zero gradient channel gives an exactly zero wgrad row, and the
    zero-amax scale value sf_val changes no output bit."""
    gold, w, dy, x, outs = kgrouped
    base = outs[gold["sf_vals"][-1]]
    for e, k in enumerate(gold["ks"]):
        if k == 128:
            assert np.all(base[e, 0] == 0)
    for sf, dw in outs.items():
        np.testing.assert_array_equal(dw, base)


def test_sampled_outputs_agree_with_dense():
    rng = np.random.default_rng(5)
    splits = np.array([96, 0, 64], np.int32)
    G, N, K = 3, 128, 256
    R = 192
    xb, wb, dyb = W.normal_bf16((R, K), 1), W.normal_bf16((G * N, K), 2), W.normal_bf16((R, N), 3)
    xq, wq, dyq = O.quantize_mx(xb, splits, G), O.quantize_mx(wb, None, G), O.quantize_mx(dyb, splits, G)
    y = O.gemm_fprop(xq, wq, splits, G, N, K)
    dx = O.gemm_dgrad(dyq, wq, splits, G, N, K)
    dw = O.gemm_wgrad(dyq, xq, splits, G, N, K)
    r, n, k = rng.integers(0, 160, 50), rng.integers(0, N, 50), rng.integers(0, K, 50)
    g = rng.integers(0, G, 50)
    np.testing.assert_allclose(O.gemm_sample("fprop", xq, wq, splits, G, N, K, r, n), y[r, n],
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(O.gemm_sample("dgrad", dyq, wq, splits, G, N, K, r, k), dx[r, k],
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(O.gemm_sample("wgrad", dyq, xq, splits, G, N, K, n, k, g),
                               dw[g, n, k], rtol=1e-12, atol=1e-12)
