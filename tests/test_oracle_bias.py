"""Pins of the oracle's grouped bias add and bias gradient (TransformerEngine
PR 3224: launch_grouped_bias_add after the grouped GEMM, with its zero-row
guard; the per-group dbiases of the backward).

The two are pinned against each other and against facts that do not restate
either formula:
  * adjointness: bias_grad is the transpose of bias_add seen as a linear map
    b -> Y, so <bias_add(0, b), dY> = <b, bias_grad(dY)> for any b, dY;
  * the per-group gradients sum to the column sums of all live rows, for
    every way of splitting them;
  * a tiny case written out by hand;
  * rows past the live total, empty groups and an all-empty split."""
import numpy as np
import pytest

import oracle as O
import workloads as W


def _f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


@pytest.mark.parametrize("splits", [[64, 0, 160, 32], [32], [0, 96, 0], [256, 256]])
def test_bias_grad_is_the_adjoint_of_bias_add(splits):
    splits = np.array(splits, np.int32)
    G, L, N, pad = len(splits), int(splits.sum()), 256, 64
    R = L + pad
    dy_bits = np.concatenate([W.normal_bf16((L, N), 51), W.uniform_bf16((pad, N), 52, -4, 4)])
    b = _f64(W.normal_bf16((G, N), 53))
    y = O.grouped_bias_add(np.zeros((R, N)), b, splits, G)
    lhs = float(np.sum(y * _f64(dy_bits)))
    rhs = float(np.sum(b * O.grouped_bias_grad(dy_bits, splits, G)))
    assert lhs == pytest.approx(rhs, rel=1e-12, abs=1e-9)


def test_group_gradients_sum_to_the_column_sums_for_any_split():
    N = 128
    dy_bits = W.normal_bf16((384, N), 54)
    total = _f64(dy_bits[:320]).sum(axis=0)
    for splits in ([320], [32, 288], [96, 0, 64, 160], [0, 0, 320]):
        db = O.grouped_bias_grad(dy_bits, np.array(splits, np.int32), len(splits))
        np.testing.assert_allclose(db.sum(axis=0), total, rtol=0, atol=1e-9)


def test_tiny_case_by_hand():
    # 2 groups of 32 rows over 128 columns: group 0 rows hold 1.0, group 1
    # rows hold -2.0, and 32 padding rows hold 100.0
    x = np.concatenate([np.full((32, 128), 1.0), np.full((32, 128), -2.0), np.full((32, 128), 100.0)])
    bits = W.f32_to_bf16_bits(x.astype(np.float32))
    db = O.grouped_bias_grad(bits, np.array([32, 32], np.int32), 2)
    assert np.all(db[0] == 32.0) and np.all(db[1] == -64.0)
    b = np.stack([np.full(128, 0.5), np.full(128, -0.25)])
    y = O.grouped_bias_add(np.full((96, 128), 10.0), b, np.array([32, 32], np.int32), 2)
    assert np.all(y[:32] == 10.5) and np.all(y[32:64] == 9.75) and np.all(y[64:] == 10.0)


def test_empty_groups_and_zero_rows():
    N = 128
    dy_bits = W.normal_bf16((64, N), 55)
    db = O.grouped_bias_grad(dy_bits, np.array([0, 64, 0], np.int32), 3)
    assert np.all(db[0] == 0) and np.all(db[2] == 0)
    # all-empty split: the bias add touches nothing, the gradient is zero
    y = np.full((64, N), 7.0)
    O.grouped_bias_add(y, np.ones((2, N)), np.array([0, 0], np.int32), 2)
    assert np.all(y == 7.0)
    assert np.all(O.grouped_bias_grad(dy_bits, np.array([0, 0], np.int32), 2) == 0)


def test_bad_splits_are_refused():
    with pytest.raises(O.OracleError):
        O.grouped_bias_grad(W.normal_bf16((64, 128), 56), np.array([48], np.int32), 1)   # not a multiple of 32
    with pytest.raises(O.OracleError):
        O.grouped_bias_add(np.zeros((64, 128)), np.zeros((1, 128)), np.array([96], np.int32), 1)  # past R
