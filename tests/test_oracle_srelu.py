"""Pins of the oracle's ScaledSReLU + MXFP8 quantisation of an fp32 buffer
(a = probs[r] * relu(y)^2, then 1x32 MX rowwise and columnwise).

Pinned against the independently pinned bf16 quantiser and against
invariances, not against a restatement of its own arithmetic:
  * where relu(y)^2 is exactly a bf16 value and probs = 1, the result equals
    quantize_mx of those bf16 values, codes and scales, bit for bit;
  * negative inputs give code +0 and drop out of every amax;
  * scaling every prob by 2^k leaves the codes and shifts every non-zero
    scale byte by k;
  * a row's prob scales that row's rowwise scale only;
  * rows past the live total are never written."""
import numpy as np
import pytest

import oracle as O
import workloads as W


def _exact_inputs(shape, seed):
    # small integers times powers of two: y^2 has at most 8 significant bits
    rng = np.random.default_rng(seed)
    mag = rng.integers(1, 16, size=shape).astype(np.float32)
    sign = np.where(rng.random(shape) < 0.3, -1.0, 1.0).astype(np.float32)
    scale = np.exp2(rng.integers(-6, 4, size=(shape[0], 1))).astype(np.float32)
    return mag * sign * scale


@pytest.mark.parametrize("splits", [[64, 0, 96], [128], [32, 32, 32, 32]])
def test_equals_bf16_quantiser_where_exact(splits):
    splits = np.array(splits, np.int32)
    G, L, C, pad = len(splits), int(splits.sum()), 256, 32
    y = np.concatenate([_exact_inputs((L, C), 71), np.full((pad, C), np.nan, np.float32)])
    probs = np.ones(L + pad, np.float32)
    a = np.square(np.maximum(y[:L], 0)).astype(np.float32)
    bits = np.concatenate([W.f32_to_bf16_bits(a), np.zeros((pad, C), np.uint16)])
    assert np.array_equal(W.bf16_bits_to_f32(bits[:L]), a)          # exactly bf16
    got = O.srelu_quantize_mx(y, probs, splits, G, data_fill=0xCD)
    want = O.quantize_mx(bits, splits, G, data_fill=0xCD)
    assert np.array_equal(got.row_data, want.row_data)
    assert np.array_equal(got.col_data, want.col_data)
    assert np.array_equal(got.row_scale, want.row_scale)
    assert np.array_equal(got.col_scale, want.col_scale)
    assert np.all(got.row_data[L:] == 0xCD) and np.all(got.col_data[L:] == 0xCD)


def test_negative_inputs_give_plus_zero():
    y = -np.abs(W.bf16_bits_to_f32(W.normal_bf16((64, 128), 72))) - 0.5
    y[5, 7] = 3.0                                        # one live value
    q = O.srelu_quantize_mx(y, np.ones(64, np.float32), np.array([64], np.int32), 1)
    live = np.zeros((64, 128), bool)
    live[5, 7] = True
    assert np.all(q.row_data[~live] == 0) and np.all(q.col_data[~live] == 0)
    assert q.row_data[5, 7] != 0 and q.col_data[5, 7] != 0


def test_power_of_two_probs_shift_scales_only():
    splits = np.array([96, 32], np.int32)
    y = W.bf16_bits_to_f32(W.normal_bf16((128, 256), 73))
    base = O.srelu_quantize_mx(y, np.ones(128, np.float32), splits, 2)
    for k in (-3, 5):
        q = O.srelu_quantize_mx(y, np.full(128, 2.0 ** k, np.float32), splits, 2)
        assert np.array_equal(q.row_data, base.row_data) and np.array_equal(q.col_data, base.col_data)
        for got, ref in ((q.row_scale, base.row_scale), (q.col_scale, base.col_scale)):
            nz = ref != 0
            assert np.array_equal(got[nz].astype(int), ref[nz].astype(int) + k)


def test_a_rows_prob_moves_only_that_rows_rowwise_scales():
    y = np.abs(W.bf16_bits_to_f32(W.normal_bf16((64, 128), 74))) + 0.25
    probs = np.ones(64, np.float32)
    base = O.srelu_quantize_mx(y, probs, np.array([64], np.int32), 1)
    probs[9] = 4.0
    q = O.srelu_quantize_mx(y, probs, np.array([64], np.int32), 1)
    assert np.array_equal(q.row_data, base.row_data)
    diff = np.nonzero(q.row_scale != base.row_scale)[0]
    # row 9 of the tile: atom bytes 9 * 16 + 0 * 4 + j for the 4 column blocks
    assert set(diff.tolist()) == {9 * 16 + j for j in range(4)}
    assert np.all(q.row_scale[diff].astype(int) == base.row_scale[diff].astype(int) + 2)
