"""Pins of the oracle's NVFP4 recipe (E2M1 codes, 16-element blocks with E4M3
scales, one fp32 second-level scale per group) and of its grouped GEMMs.

TransformerEngine PR 3224 names NVFP4 as a second quantiser of the same
grouped paths without defining it; the oracle follows the public NVFP4
format (the reading is written out in gq_oracle.c).  The pins
do not restate its arithmetic:
  * the E2M1 value table of the format, and a brute-force nearest-even
    search over it;
  * exact round trips: operands built so that every scale is exact
    dequantise to themselves, and each scale byte holds the scale known by
    construction at the position the [...][32][4][4] atom shape gives
    (numpy.ravel_multi_index over that shape);
  * invariances: padding content, scaling a group by 2^k, and
    columnwise(X) == rowwise(X^T) byte for byte;
  * an error bound: every element within one scale step of its input;
  * grouped GEMMs on exactly representable operands equal numpy matmuls of
    the inputs, with an empty and a 32-row group and NaN padding."""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W

E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # FP4 E2M1 magnitudes, codes 0..7
NAN_BF16 = 0x7FC0


def test_e2m1_decode_is_the_format_table():
    for c in range(16):
        v = O.e2m1_decode(c)
        assert abs(v) == E2M1_TABLE[c & 7]
        assert (math.copysign(1.0, v) < 0) == bool(c & 8)


def _nearest_even(v):
    a = abs(v)
    if a >= 6.0:
        idx = 7
    else:
        d = [abs(a - t) for t in E2M1_TABLE]
        best = min(d)
        cands = [i for i in range(8) if d[i] == best]
        idx = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
    return idx | (8 if math.copysign(1.0, v) < 0 else 0)


def test_e2m1_encode_is_nearest_even_with_saturation():
    mids = [(E2M1_TABLE[i] + E2M1_TABLE[i + 1]) / 2 for i in range(7)]
    vals = list(np.linspace(-7.5, 7.5, 3001)) + mids + [-m for m in mids]
    vals += [m + e for m in mids for e in (1e-9, -1e-9)] + [0.0, -0.0, 1e-30, -1e-30, 100.0, -1e9, np.inf]
    for v in vals:
        assert O.e2m1_encode(v) == _nearest_even(v), v


def test_global_scale_special_cases():
    assert O.nv_global_scale(2688.0) == 1.0
    assert O.nv_global_scale(0.0) == 1.0                   # empty or all-zero group
    assert O.nv_global_scale(2688.0 * 2.0 ** -5) == 32.0
    assert O.nv_global_scale(1e-38) == np.float32(np.finfo(np.float32).max)   # clamped


# --------------------------------------------------------------------------- #
# exactly representable operands                                               #
# --------------------------------------------------------------------------- #

def _exact_operand(splits, C, seed, pad):
    """bf16 bits [L + pad, C] whose NVFP4 round trip is exact, the values
    (fp64 [L, C]), and the scale each 16 x 16 tile's blocks must get.

    Per group: S_g = 2^p.  Every 16 x 16 tile holds E2M1 table values times
    one power of two, with +-6 on a permuted diagonal (so every row block and
    every column block of the tile has amax = 6 * that power).  Tile (0, 0)
    uses 448 * 2^-p, so amax_g = 2688 * 2^-p and its blocks get sf = 448;
    the others 2^(d - p), so their blocks get sf = 2^d, d in [-9, 8]."""
    rng = np.random.default_rng(seed)
    L = int(sum(splits))
    x = np.zeros((L, C))
    sf = {}
    o = 0
    for g, m in enumerate(splits):
        if m == 0:
            continue
        p = int(rng.integers(-4, 5))
        for a in range(0, m, 16):
            for b in range(0, C, 16):
                tile = rng.choice(E2M1_TABLE, size=(16, 16)) * rng.choice([-1.0, 1.0], size=(16, 16))
                tile[np.arange(16), rng.permutation(16)] = 6.0 * rng.choice([-1.0, 1.0], size=16)
                if a == 0 and b == 0:
                    scale, s = 448.0 * 2.0 ** -p, 448.0
                else:
                    d = int(rng.integers(-9, 9))
                    scale, s = 2.0 ** (d - p), 2.0 ** d
                x[o + a:o + a + 16, b:b + 16] = tile * scale
                sf[(o + a, b)] = s
        o += m
    bits = W.f32_to_bf16_bits(x.astype(np.float32))
    assert np.array_equal(W.bf16_bits_to_f32(bits).astype(np.float64), x)
    bits = np.concatenate([bits, np.full((pad, C), NAN_BF16, np.uint16)])
    return bits, x, sf


def _nib(data_row, i):
    byte = data_row[i // 2]
    return (byte >> 4) & 15 if i % 2 else byte & 15


def _code_value(code):
    return (-1.0 if code & 8 else 1.0) * E2M1_TABLE[code & 7]


def _tiles_prefix(splits):
    return np.concatenate([[0], np.cumsum([(m + 127) // 128 for m in splits])])


@pytest.mark.parametrize("splits,C", [([128, 64, 0, 96], 128), ([32], 256), ([256, 32], 128)])
def test_exact_round_trip_and_scale_positions(splits, C):
    bits, x, sf = _exact_operand(splits, C, 5, pad=32)
    R = bits.shape[0]
    G = len(splits)
    q = O.quantize_nvfp4(bits, np.array(splits, np.int32), G)
    tp = _tiles_prefix(splits)
    off = np.concatenate([[0], np.cumsum(splits)])
    for g in range(G):
        m, o = splits[g], int(off[g])
        if m == 0:
            continue
        T = int(tp[g + 1] - tp[g])
        base = 512 * (C // 64) * int(tp[g])
        S = O.nv_global_scale(float(q.amax[g]))
        assert S == 2688.0 / float(q.amax[g])
        for lr in range(m):
            r = o + lr
            for c in range(C):
                want_sf = sf[(o + 16 * (lr // 16), 16 * (c // 16))]
                # rowwise: block j = c // 16 of row lr
                j = c // 16
                pos = base + np.ravel_multi_index((lr // 128, j // 4, lr % 32, (lr % 128) // 32, j % 4),
                                                  (T, C // 64, 32, 4, 4))
                s_row = O.e4m3_decode([q.row_scale[pos]])[0]
                assert s_row == want_sf
                assert _code_value(_nib(q.row_data[r], c)) * s_row / S == x[r, c]
                # columnwise: block b = lr // 16 of column c, stored transposed
                b = lr // 16
                pos = base + np.ravel_multi_index((c // 128, b // 4, c % 32, (c % 128) // 32, b % 4),
                                                  (max(C // 128, 1), 2 * T, 32, 4, 4))
                s_col = O.e4m3_decode([q.col_scale[pos]])[0]
                assert s_col == want_sf
                assert _code_value(_nib(q.col_data[c], r)) * s_col / S == x[r, c]
    assert R % 2 == 0


def test_padding_content_never_matters():
    splits = np.array([96, 0, 32], np.int32)
    live = W.normal_bf16((128, 128), 11)
    outs = []
    for fill in (0.0, 3.0, np.nan):
        bits = np.concatenate([live, W.fill_bf16((64, 128), fill)])
        outs.append(O.quantize_nvfp4(bits, splits, 3, data_fill=0xA5))
    for q in outs[1:]:
        for a in ("row_data", "row_scale", "col_data", "col_scale", "amax"):
            assert np.array_equal(getattr(q, a), getattr(outs[0], a)), a
    # codes of padding rows are never written
    assert np.all(outs[0].row_data[128:] == 0xA5) and np.all(outs[0].col_data[:, 64:] == 0xA5)


@pytest.mark.parametrize("k", [-3, 4])
def test_power_of_two_scaling_leaves_codes_and_scales(k):
    splits = np.array([64, 32, 128], np.int32)
    x = W.normal_bf16((224, 256), 12)
    y = W.f32_to_bf16_bits(W.bf16_bits_to_f32(x) * np.float32(2.0 ** k))
    assert np.array_equal(W.bf16_bits_to_f32(y), W.bf16_bits_to_f32(x) * np.float32(2.0 ** k))
    a, b = O.quantize_nvfp4(x, splits, 3), O.quantize_nvfp4(y, splits, 3)
    for f in ("row_data", "row_scale", "col_data", "col_scale"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    assert np.array_equal(b.amax, a.amax * np.float32(2.0 ** k))


def test_columnwise_is_rowwise_of_the_transpose():
    x = W.normal_bf16((256, 384), 13)
    col = O.quantize_nvfp4(x, np.array([256], np.int32), 1, rowwise=False)
    row = O.quantize_nvfp4(np.ascontiguousarray(x.T), np.array([384], np.int32), 1, colwise=False)
    assert np.array_equal(col.col_data, row.row_data)
    assert np.array_equal(col.col_scale, row.row_scale)
    assert np.array_equal(col.amax, row.amax)


def test_every_element_within_one_scale_step():
    splits = np.array([128, 96], np.int32)
    x = W.normal_bf16((224, 256), 14, scale=3.0)
    q = O.quantize_nvfp4(x, splits, 2)
    xf = W.bf16_bits_to_f32(x).astype(np.float64)
    tp = _tiles_prefix(splits)
    off = [0, 128, 224]
    normal_blocks = 0
    for g in range(2):
        S = O.nv_global_scale(float(q.amax[g]))
        assert q.amax[g] == np.max(np.abs(W.bf16_bits_to_f32(x[off[g]:off[g + 1]])))
        T = int(tp[g + 1] - tp[g])
        base = 512 * 4 * int(tp[g])
        for lr in range(off[g + 1] - off[g]):
            r = off[g] + lr
            for j in range(16):
                pos = base + np.ravel_multi_index((lr // 128, j // 4, lr % 32, (lr % 128) // 32, j % 4),
                                                  (T, 4, 32, 4, 4))
                s = O.e4m3_decode([q.row_scale[pos]])[0]
                if s < 2.0 ** -6:
                    continue                            # subnormal scale: no bound claimed
                normal_blocks += 1
                for c in range(16 * j, 16 * j + 16):
                    deq = _code_value(_nib(q.row_data[r], c)) * s / S
                    assert abs(deq - xf[r, c]) <= s / S * (1 + 2.0 ** -20)   # fp32 rounding of x * m
    assert normal_blocks == 224 * 16


def test_zero_and_empty_groups():
    splits = np.array([0, 64, 32], np.int32)
    x = np.concatenate([np.zeros((64, 128), np.uint16), W.normal_bf16((32, 128), 15)])
    q = O.quantize_nvfp4(x, splits, 3, scale_fill=0x77)
    assert q.amax[0] == 0 and q.amax[1] == 0 and q.amax[2] > 0
    # group 1 (all zero): scale region (tiles 0..0) all zero, codes all zero
    assert np.all(q.row_scale[:512 * 2] == 0) and np.all(q.col_scale[:512 * 2] == 0)
    assert np.all(q.row_data[:64] == 0) and np.all(q.col_data[:, :32] == 0)


def test_bad_inputs_are_refused():
    with pytest.raises(O.OracleError):
        O.quantize_nvfp4(W.normal_bf16((64, 128), 16), np.array([48], np.int32), 1)     # split % 32
    with pytest.raises(O.OracleError):
        O.quantize_nvfp4(W.normal_bf16((64, 96), 16), np.array([64], np.int32), 1)      # cols % 128


# --------------------------------------------------------------------------- #
# grouped GEMMs                                                                #
# --------------------------------------------------------------------------- #

def test_gemms_on_exact_operands_equal_matmul():
    splits = [64, 0, 32, 160]
    G, N, K, pad = len(splits), 128, 256, 32
    s32 = np.array(splits, np.int32)
    off = np.concatenate([[0], np.cumsum(splits)])
    xb, x, _ = _exact_operand(splits, K, 21, pad)
    db, dy, _ = _exact_operand(splits, N, 22, pad)
    wb, w, _ = _exact_operand([N] * G, K, 23, 0)
    xq, dq, wq = O.quantize_nvfp4(xb, s32, G), O.quantize_nvfp4(db, s32, G), O.quantize_nvfp4(wb, None, G)
    y = O.gemm_nvfp4("fprop", xq, wq, s32, G, N, K)
    dx = O.gemm_nvfp4("dgrad", dq, wq, s32, G, N, K)
    init = np.random.default_rng(24).standard_normal((G, N, K))
    dw = O.gemm_nvfp4("wgrad", dq, xq, s32, G, N, K)
    dwa = O.gemm_nvfp4("wgrad", dq, xq, s32, G, N, K, accumulate=True, init=init)
    L = int(off[-1])
    for g in range(G):
        a, b = int(off[g]), int(off[g + 1])
        wg = w[g * N:(g + 1) * N]
        assert np.array_equal(y[a:b], x[a:b] @ wg.T)
        assert np.array_equal(dx[a:b], dy[a:b] @ wg)
        assert np.array_equal(dw[g], dy[a:b].T @ x[a:b])
        assert np.allclose(dwa[g], init[g] + dy[a:b].T @ x[a:b], rtol=1e-15, atol=0)
    assert np.all(dw[1] == 0)
    assert np.all(np.isnan(y[L:])) and np.all(np.isnan(dx[L:]))


def test_sampled_gemms_equal_the_full_gemms():
    """The one-dot-product-per-sample oracle (used at full size) against the
    pinned full GEMMs, at every sampled position, all three kinds."""
    splits = np.array([96, 0, 32, 160], np.int32)
    G, N, K, pad = 4, 256, 256, 32
    L = int(splits.sum())
    x = np.concatenate([W.normal_bf16((L, K), 25), W.uniform_bf16((pad, K), 26, -4, 4)])
    dy = np.concatenate([W.normal_bf16((L, N), 27), W.uniform_bf16((pad, N), 28, -4, 4)])
    w = W.normal_bf16((G * N, K), 29, scale=0.02)
    xq, dq, wq = O.quantize_nvfp4(x, splits, G), O.quantize_nvfp4(dy, splits, G), O.quantize_nvfp4(w, None, G)
    rng = np.random.default_rng(30)
    rows = rng.integers(0, L, 300)
    cn, ck = rng.integers(0, N, 300), rng.integers(0, K, 300)
    g = rng.choice(np.flatnonzero(splits > 0), 300)
    y = O.gemm_nvfp4("fprop", xq, wq, splits, G, N, K)
    dx = O.gemm_nvfp4("dgrad", dq, wq, splits, G, N, K)
    dw = O.gemm_nvfp4("wgrad", dq, xq, splits, G, N, K)
    np.testing.assert_allclose(O.gemm_nvfp4_sample("fprop", xq, wq, splits, G, N, K, rows, cn), y[rows, cn],
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(O.gemm_nvfp4_sample("dgrad", dq, wq, splits, G, N, K, rows, ck), dx[rows, ck],
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(O.gemm_nvfp4_sample("wgrad", dq, xq, splits, G, N, K, cn, ck, g), dw[g, cn, ck],
                               rtol=1e-12, atol=1e-12)
