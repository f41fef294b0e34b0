"""Pins for the oracle's split scan and quantisers.

Hand-derived values, the layout's stated structure, bijection of the scale
placement, padding invariance and grouping invariants -- none of them re-types
the oracle's own formula.
"""
import json
import os

import numpy as np
import pytest

import oracle as O
import workloads as W
from workloads import f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(a):
    return f32_to_bf16_bits(np.asarray(a, np.float32))


# --------------------------------------------------------------------------- #
# split scan                                                                   #
# --------------------------------------------------------------------------- #

def test_split_scan_is_a_prefix_sum():
    rng = np.random.default_rng(0)
    for G in (1, 2, 7, 64, 1024):
        s = (rng.integers(0, 20, G) * 32).astype(np.int32)
        s[rng.integers(0, G)] = 0
        off, tp, sb = O.split_scan(s, G, int(s.sum()) + 96, 256)
        np.testing.assert_array_equal(off, np.concatenate([[0], np.cumsum(s)]))
        tiles = -(-s.astype(np.int64) // 128)
        np.testing.assert_array_equal(tp, np.concatenate([[0], np.cumsum(tiles)]))
        np.testing.assert_array_equal(sb, tp * 512 * (256 // 128))


def test_split_scan_channel_offsets():
    s = np.array([256, 0, 128, 384], np.int32)
    off, _, sb = O.split_scan(s, 4, 1024, 512, O.RECIPE_CHANNEL)
    np.testing.assert_array_equal(sb, 4 * 512 * off // 128)


def test_split_scan_uniform():
    off, tp, _ = O.split_scan(None, 4, 4096, 128)
    np.testing.assert_array_equal(off, [0, 1024, 2048, 3072, 4096])
    np.testing.assert_array_equal(tp, [0, 8, 16, 24, 32])


@pytest.mark.parametrize("splits,rows,cols,recipe,status", [
    ([32, -32], 64, 128, O.RECIPE_MX, O.ERR_SPLITS),
    ([48], 64, 128, O.RECIPE_MX, O.ERR_SPLITS),
    ([64, 64], 96, 128, O.RECIPE_MX, O.ERR_SPLITS),
    ([64], 128, 128, O.RECIPE_CHANNEL, O.ERR_SPLITS),
    ([32], 64, 96, O.RECIPE_MX, O.ERR_ALIGNMENT),
    (None, 100, 128, O.RECIPE_MX, O.ERR_ALIGNMENT),
])
def test_split_scan_rejects(splits, rows, cols, recipe, status):
    G = 3 if splits is None else len(splits)
    s = None if splits is None else np.array(splits, np.int32)
    with pytest.raises(O.OracleError) as ei:
        O.split_scan(s, G, rows, cols, recipe)
    assert ei.value.status == status


# --------------------------------------------------------------------------- #
# MX: a hand-worked example                                                    #
# --------------------------------------------------------------------------- #

def test_mx_hand_worked_example():
    x = np.zeros((32, 128), np.float32)
    x[0, 0], x[0, 1], x[0, 2] = 1.0, -0.5, 3.0
    x[1, 40] = 2.0 ** -20
    q = O.quantize_mx(bf16(x), np.array([32], np.int32), 1)
    # rowwise: row 0 block 0 amax 3 -> e = 1 - 8 = -7 (byte 120); codes x*2^7
    assert q.row_data[0, :3].tolist() == [0x70, 0xE8, 0x7C]     # 128, -64, 384
    # row 1 block 1 amax 2^-20 -> e = -28 (byte 99); code 2^-20 * 2^28 = 256
    assert q.row_data[1, 40] == 0x78
    assert q.row_scale.size == 512
    want = np.zeros(512, np.uint8)
    want[0] = 120            # (row 0, block 0): byte 0
    want[17] = 99            # (row 1, block 1): 1*16 + 0*4 + 1
    np.testing.assert_array_equal(q.row_scale, want)
    # columnwise: col 0 amax 1 (e=-8, byte 119), col 1 amax .5 (e=-9, 118),
    # col 2 amax 3 (e=-7, 120), col 40 amax 2^-20 (e=-28, 99)
    assert q.col_data[0, :3].tolist() == [0x78, 0xF8, 0x7C]     # 256, -256, 384
    assert q.col_data[1, 40] == 0x78
    want = np.zeros(512, np.uint8)
    want[0] = 119            # column 0:  0*16 + 0*4 + block 0
    want[16] = 118           # column 1:  1*16
    want[32] = 120           # column 2:  2*16
    want[8 * 16 + 4] = 99    # column 40: (40%32)*16 + (40/32)*4
    np.testing.assert_array_equal(q.col_scale, want)
    assert np.count_nonzero(q.row_data) == 4 and np.count_nonzero(q.col_data) == 4


@pytest.mark.parametrize("r,j,byte", [(0, 0, 0), (1, 0, 16), (32, 0, 4), (0, 1, 1), (33, 2, 22),
                                      (127, 3, 511), (96, 3, 15)])
def test_mx_atom_positions(r, j, byte):
    """The [32][4][4] atom: a lone nonzero at (row r of the tile, 32-col block
    j) lights exactly one scale byte, at the hand-computed position."""
    x = np.zeros((128, 128), np.float32)
    x[r, 32 * j + 5] = 1.0
    q = O.quantize_mx(bf16(x), np.array([128], np.int32), 1)
    nz = np.flatnonzero(q.row_scale)
    assert nz.tolist() == [byte]
    # the same value seen columnwise: channel 32j+5, 32-row block r//32
    c, b = 32 * j + 5, r // 32
    assert np.flatnonzero(q.col_scale).tolist() == [(c % 32) * 16 + (c // 32) * 4 + b]


def test_mx_tile_order_rowwise_and_colwise():
    """Rowwise atoms run [row tile][col tile]; columnwise atoms run
    [col tile][row tile] with the row (m) tile as the inner stride, and a
    group's extent is its own tile count."""
    G, cols = 2, 384
    splits = np.array([96, 352], np.int32)          # T = 1 and 3 tiles
    R = int(splits.sum())
    off, tp, sb = O.split_scan(splits, G, R, cols)
    for g, t, ct in [(1, 2, 1), (1, 0, 2), (0, 0, 1), (1, 1, 0)]:
        x = np.zeros((R, cols), np.float32)
        x[off[g] + 128 * t, 128 * ct] = 1.0
        q = O.quantize_mx(bf16(x), splits, G)
        T = tp[g + 1] - tp[g]
        assert (np.flatnonzero(q.row_scale) // 512).tolist() == [(sb[g] // 512) + t * 3 + ct]
        assert (np.flatnonzero(q.col_scale) // 512).tolist() == [(sb[g] // 512) + ct * T + t]


def _live_blocks_all_nonzero(w_splits, cols, seed):
    """Input where every live 32-block has amax >= 1 (scale byte > 0)."""
    R = int(np.sum(w_splits)) + 64
    x = W.normal_bf16((R, cols), seed)
    x = x.copy()
    x[:, ::16] = bf16(np.full(1, 2.0))[0]       # two entries per 32-block ensure amax >= 2
    return x


@pytest.mark.parametrize("splits", [[32], [96, 0, 160, 32], [128, 256, 64], [0, 0, 32]])
def test_mx_scale_placement_is_a_bijection(splits):
    splits = np.array(splits, np.int32)
    G, cols = len(splits), 256
    x = _live_blocks_all_nonzero(splits, cols, 1)
    off, tp, sb = O.split_scan(splits, G, x.shape[0], cols)
    total = int(sb[-1])
    q = O.quantize_mx(x, splits, G, scale_capacity=total + 512, scale_fill=0xAB)
    live_blocks = int(splits.sum()) * (cols // 32)
    for s in (q.row_scale, q.col_scale):
        region = s[:total]
        assert np.count_nonzero(region) == live_blocks     # distinct bytes, one per block
        assert np.all(s[total:] == 0xAB)                    # nothing past the extent
    for g in range(G):                                      # each group's own extent
        T = int(tp[g + 1] - tp[g])
        assert sb[g + 1] - sb[g] == 512 * T * (cols // 128)


@pytest.mark.parametrize("splits", [[64, 160, 0, 32], [512], [32, 32, 32, 32, 32]])
def test_mx_grouped_equals_concatenation_of_single_group_quantizes(splits):
    splits = np.array(splits, np.int32)
    G, cols = len(splits), 384
    R = int(splits.sum()) + 32
    x = W.normal_bf16((R, cols), 2)
    q = O.quantize_mx(x, splits, G)
    off, _, sb = O.split_scan(splits, G, R, cols)
    rs, cs = [], []
    for g in range(G):
        part = x[off[g]:off[g + 1]]
        if part.shape[0] == 0:
            continue
        qg = O.quantize_mx(part, np.array([part.shape[0]], np.int32), 1)
        np.testing.assert_array_equal(q.row_data[off[g]:off[g + 1]], qg.row_data)
        np.testing.assert_array_equal(q.col_data[off[g]:off[g + 1]], qg.col_data)
        rs.append(qg.row_scale)
        cs.append(qg.col_scale)
    np.testing.assert_array_equal(q.row_scale[:sb[-1]], np.concatenate(rs))
    np.testing.assert_array_equal(q.col_scale[:sb[-1]], np.concatenate(cs))


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_mx_padding_content_never_matters(G):
    """Rows past sum(split_sizes) are outside every group (TransformerEngine
    issue 3484, 'Expected behavior'): fills 0.0, 3.0, uniform garbage and NaN
    give bitwise identical codes and scales; padding code rows are untouched."""
    cols, live = 256, 512
    splits = np.full(G, live // G, np.int32)
    live_x = W.normal_bf16((live, cols), 1)
    outs = []
    for fill in ("0", "3", "u", "nan"):
        if fill == "u":
            pad = W.uniform_bf16((256, cols), 9, -4, 4)
        elif fill == "nan":
            pad = np.full((256, cols), 0x7FC0, np.uint16)
        else:
            pad = W.fill_bf16((256, cols), float(fill))
        q = O.quantize_mx(np.concatenate([live_x, pad]), splits, G, data_fill=0x5A)
        assert np.all(q.row_data[live:] == 0x5A) and np.all(q.col_data[live:] == 0x5A)
        outs.append(q)
    for q in outs[1:]:
        for a in ("row_data", "col_data", "row_scale", "col_scale"):
            np.testing.assert_array_equal(getattr(q, a), getattr(outs[0], a))


def test_mx_single_group_padded_equals_unpadded():
    """num_groups == 1: a 768-row buffer with 512 live rows quantises exactly
    like the 512-row unpadded buffer (TransformerEngine issue 3484)."""
    w = W.workload("padded_single_group", pad_kind="fill3")
    x = w.activation(w.hidden, 0)
    qp = O.quantize_mx(x, w.splits, 1)
    qu = O.quantize_mx(x[:512], w.splits, 1)
    np.testing.assert_array_equal(qp.row_data[:512], qu.row_data)
    np.testing.assert_array_equal(qp.col_data[:512], qu.col_data)
    np.testing.assert_array_equal(qp.row_scale, qu.row_scale)
    np.testing.assert_array_equal(qp.col_scale, qu.col_scale)


def test_mx_block_max_code_in_top_binade():
    """With e = floor(log2 amax) - 8 the largest code of every nonzero block
    lies in [256, 448] (exponent field 15), unless the scale was clamped."""
    x = W.normal_bf16((256, 512), 3, scale=1e-3)
    q = O.quantize_mx(x, np.array([256], np.int32), 1)
    mags = O.e4m3_decode(q.row_data).reshape(256, 16, 32)
    mx = np.abs(mags).max(axis=2)
    assert np.all((mx >= 256) & (mx <= 448))
    mags = O.e4m3_decode(q.col_data).reshape(8, 32, 512)
    mx = np.abs(mags).max(axis=1)
    assert np.all((mx >= 256) & (mx <= 448))


# --------------------------------------------------------------------------- #
# per-channel 128-row recipe                                                   #
# --------------------------------------------------------------------------- #

def test_channel_hand_worked_example():
    x = np.zeros((128, 128), np.float32)
    x[0, 0], x[5, 0] = 56.0, -7.0                 # amax 56 = 448/8 -> sf = 1/8 exactly
    x[3, 1] = 448.0 * 2.0 ** -60                  # sf = 2^-60 exactly
    q = O.quantize_channel(bf16(x), np.array([128], np.int32), 1, zero_scale=1e-4)
    assert q.col_scale.shape == (1, 128)
    assert q.col_scale[0, 0] == np.float32(0.125)
    assert q.col_scale[0, 1] == np.float32(2.0 ** -60)
    assert q.col_scale[0, 2] == np.float32(1e-4)  # all-zero channel takes sf_val
    assert q.col_data[0, 0] == 0x7E and q.col_data[5, 0] == 0xE6      # 448, -56 = -1.75*2^5
    assert q.col_data[3, 1] == 0x7E
    assert np.count_nonzero(q.col_data) == 3


def test_channel_zero_scale_clamped():
    x = np.zeros((128, 128), np.uint16)
    q = O.quantize_channel(x, np.array([128], np.int32), 1, zero_scale=1e-38)
    assert np.all(q.col_scale == np.float32(1e-30))    # clamp_min(1e-30)


def test_channel_properties_on_random_data():
    """Every nonzero (block, channel) reaches a code of magnitude 448; the
    dequantised value is within half an e4m3 step of the input; an all-zero
    channel quantises to zeros with scale sf_val; sf_val changes nothing else."""
    w = W.workload("kgrouped_zero_channel")
    dy, _ = W.kgrouped_zero_channel_operands(w)
    outs = {}
    for sf in (1.0, 1e-4, 1e-8, 1e-30):
        outs[sf] = O.quantize_channel(dy, w.splits, 4, zero_scale=sf)
    q = outs[1e-30]
    codes = O.e4m3_decode(q.col_data).reshape(6, 128, 2048)
    amax_code = np.abs(codes).max(axis=1)
    x = W.bf16_bits_to_f32(dy).astype(np.float64).reshape(6, 128, 2048)
    zero = np.abs(x).max(axis=1) == 0
    assert zero.sum() == 2 and zero[2, 0] and zero[3, 0]     # experts 1 and 2, channel 0
    assert np.all(amax_code[~zero] == 448.0)
    deq = codes * q.col_scale.astype(np.float64)[:, None, :]
    err = np.abs(deq - x)
    bound = 2.0 ** -4 * (1 + 2.0 ** -20) * np.abs(x) + 2.0 ** -10 * q.col_scale[:, None, :]
    assert np.all(err <= bound)
    for sf, o in outs.items():
        np.testing.assert_array_equal(o.col_data, q.col_data)
        np.testing.assert_array_equal(o.col_scale[~zero], q.col_scale[~zero])
        assert np.all(o.col_scale[zero] == np.float32(max(np.float32(sf), np.float32(1e-30))))
