"""Pins of the oracle's ScaledSwiGLU + MXFP8 quantisation of an fp32 buffer
(gate half g, linear half l: a = (silu(g) * l) * probs[r], then 1x32 MX
rowwise and columnwise) and of the activation's own exp.

Pinned against facts that do not restate its arithmetic:
  * the exp against the C library's exp (relative error below 2^-22 over
    its whole argument range) and exp(0) = 1;
  * silu(x) = x exactly once 1 + exp(-x) rounds to 1 (x >= 17), and
    silu(0) = 0;
  * where silu(g) = g and g * l * probs is exactly a bf16 value, the result
    equals quantize_mx of those bf16 values, codes and scales, bit for bit;
  * a zero linear half gives zero codes and zero scales;
  * scaling every prob by 2^k leaves the codes and shifts every non-zero
    scale byte by k; a row's prob moves only that row's rowwise scales;
  * rows past the live total are never written."""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W


def test_exp_against_the_c_library():
    xs = np.concatenate([np.linspace(-87.0, 88.0, 20001), np.linspace(-1.0, 1.0, 2001)]).astype(np.float32)
    worst = max(abs(O.act_exp(float(x)) / math.exp(float(x)) - 1.0) for x in xs)
    assert worst < 2.0 ** -22
    assert O.act_exp(0.0) == 1.0


def test_silu_special_values():
    assert O.act_silu(0.0) == 0.0
    for x in (17.0, 20.5, 64.0, 1000.0):
        assert O.act_silu(x) == x
    assert abs(O.act_silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-7
    assert -1e-6 < O.act_silu(-20.0) < 0.0


def _exact_case(splits, C, seed):
    """y with a gate half of values >= 17 (silu exact) and a linear half such
    that gate * linear * prob is exactly a bf16 value."""
    rng = np.random.default_rng(seed)
    L = int(np.sum(splits))
    gate = (rng.integers(17, 32, size=(L, C)) * 1.0).astype(np.float32)      # 5-bit integers
    lin = (rng.integers(-3, 4, size=(L, C)) * np.exp2(rng.integers(-4, 3, size=(L, 1)))).astype(np.float32)
    probs = np.exp2(rng.integers(-3, 2, size=L)).astype(np.float32)
    a = gate * lin * probs[:, None]
    bits = W.f32_to_bf16_bits(a)
    assert np.array_equal(W.bf16_bits_to_f32(bits), a)                       # exactly bf16
    return np.concatenate([gate, lin], axis=1), probs, bits


@pytest.mark.parametrize("splits", [[64, 0, 96], [128], [32, 32, 32, 32]])
def test_equals_bf16_quantiser_where_exact(splits):
    splits = np.array(splits, np.int32)
    G, L, C, pad = len(splits), int(splits.sum()), 256, 32
    y, probs, bits = _exact_case(splits, C, 91)
    y = np.concatenate([y, np.full((pad, 2 * C), np.nan, np.float32)])
    probs = np.concatenate([probs, np.full(pad, np.nan, np.float32)])
    bits = np.concatenate([bits, np.zeros((pad, C), np.uint16)])
    got = O.swiglu_quantize_mx(y, probs, splits, G, data_fill=0xCD)
    want = O.quantize_mx(bits, splits, G, data_fill=0xCD)
    for f in ("row_data", "col_data", "row_scale", "col_scale"):
        assert np.array_equal(getattr(got, f), getattr(want, f)), f
    assert np.all(got.row_data[L:] == 0xCD) and np.all(got.col_data[L:] == 0xCD)


def test_zero_linear_half_gives_zero():
    y = np.concatenate([W.bf16_bits_to_f32(W.normal_bf16((64, 128), 92)), np.zeros((64, 128), np.float32)], 1)
    q = O.swiglu_quantize_mx(y, np.ones(64, np.float32), np.array([64], np.int32), 1)
    assert np.all((q.row_data & 0x7F) == 0) and np.all((q.col_data & 0x7F) == 0)
    n = len(q.row_scale)
    assert np.all(q.row_scale[:n] == 0) and np.all(q.col_scale[:n] == 0)


def test_power_of_two_probs_shift_scales_only():
    splits = np.array([96, 32], np.int32)
    y = W.bf16_bits_to_f32(W.normal_bf16((128, 512), 93))
    base = O.swiglu_quantize_mx(y, np.ones(128, np.float32), splits, 2)
    for k in (-3, 5):
        q = O.swiglu_quantize_mx(y, np.full(128, 2.0 ** k, np.float32), splits, 2)
        assert np.array_equal(q.row_data, base.row_data) and np.array_equal(q.col_data, base.col_data)
        for got, ref in ((q.row_scale, base.row_scale), (q.col_scale, base.col_scale)):
            nz = ref != 0
            assert np.array_equal(got[nz].astype(int), ref[nz].astype(int) + k)


def test_a_rows_prob_moves_only_that_rows_rowwise_scales():
    y = np.abs(W.bf16_bits_to_f32(W.normal_bf16((64, 256), 94))) + 0.25
    probs = np.ones(64, np.float32)
    base = O.swiglu_quantize_mx(y, probs, np.array([64], np.int32), 1)
    probs[9] = 4.0
    q = O.swiglu_quantize_mx(y, probs, np.array([64], np.int32), 1)
    assert np.array_equal(q.row_data, base.row_data)
    diff = np.nonzero(q.row_scale != base.row_scale)[0]
    assert set(diff.tolist()) == {9 * 16 + j for j in range(4)}
    assert np.all(q.row_scale[diff].astype(int) == base.row_scale[diff].astype(int) + 2)
