"""GPU parity of the grouped quantizer (gq_quantize, gq_split_scan) against the
CPU oracle: FP8 codes and scales bit-exact, padding never read, never written,
group-local scale extents, split errors and the noop flag on the device."""
import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_grouped_gemm_group_gb300 as gq  # noqa: E402
from _gpu_util import (assert_mx_equal, bf16_dev, ch_recipe, check_status, host, mx_recipe,  # noqa: E402
                       quantize, splits_dev, status_dev)


def _mx_case(bits, splits, G, rowwise=True, colwise=True):
    R, Cc = bits.shape
    gpu, st = quantize(bits, splits, G, mx_recipe(rowwise, colwise))
    check_status(st)
    ora = O.quantize_mx(bits, splits, G, rowwise=rowwise, colwise=colwise)
    off, _, sb = O.split_scan(splits, G, R, Cc)
    assert_mx_equal(gpu, ora, int(off[-1]), int(sb[-1]))
    return gpu, ora


SMALL = [
    ([512], 768, 1024),                        # one group, padded (TE issue 3484 geometry)
    ([512], 512, 1024),                        # unpadded
    ([32, 0, 96, 160, 0, 64], 480, 384),       # ragged tiles, empty groups, 32-row group
    ([0, 0, 32], 64, 128),
    ([128] * 8, 1024 + 64, 256),
    ([224, 32, 0, 416], 800, 640),
]


@pytest.mark.parametrize("splits,R,C", SMALL)
@pytest.mark.parametrize("orient", ["both", "row", "col"])
def test_mx_bit_exact_small(splits, R, C, orient):
    splits = np.array(splits, np.int32)
    L = int(splits.sum())
    bits = np.concatenate([W.normal_bf16((L, C), 7), W.uniform_bf16((R - L, C), 8, -4, 4)])
    _mx_case(bits, splits, len(splits), orient != "col", orient != "row")


def test_mx_value_range_extremes():
    """Tiny, huge, subnormal and exactly-representable magnitudes, zero blocks."""
    rng = np.random.default_rng(3)
    R, C = 256, 512
    x = rng.standard_normal((R, C)).astype(np.float32)
    x *= np.exp2(rng.integers(-130, 120, size=(R, 1))).astype(np.float32)
    x[:, :64] *= np.float32(2.0 ** -20)
    x[5, :] = 0.0
    x[:, 100] = 0.0
    x[7, 32:64] = np.float32(448.0)
    x[9, :32] = np.float32(1e-40)                 # fp32 subnormal -> bf16 subnormal
    bits = W.f32_to_bf16_bits(x)
    _mx_case(bits, np.array([128, 128], np.int32), 2)


@pytest.mark.parametrize("fill", ["zero", "three", "nan", "garbage"])
def test_mx_padding_never_read(fill):
    """Fills 0.0 / 3.0 / NaN / garbage past sum(split_sizes) give the same bytes
    (TransformerEngine issue 3484, 'Expected behavior')."""
    splits = np.array([96, 160], np.int32)
    live = W.normal_bf16((256, 512), 11)
    pad = {"zero": W.fill_bf16((128, 512), 0.0), "three": W.fill_bf16((128, 512), 3.0),
           "nan": np.full((128, 512), 0x7FC0, np.uint16),
           "garbage": W.uniform_bf16((128, 512), 12, -1e4, 1e4)}[fill]
    _mx_case(np.concatenate([live, pad]), splits, 2)


def test_mx_uniform_split_single_grouped_weight():
    """splits = NULL: uniform split of rows_cap / G (single grouped weight)."""
    bits = W.normal_bf16((8 * 512, 384), 5, scale=0.02)
    gpu, st = quantize(bits, None, 8, mx_recipe())
    check_status(st)
    ora = O.quantize_mx(bits, None, 8)
    _, _, sb = O.split_scan(None, 8, 8 * 512, 384)
    assert_mx_equal(gpu, ora, 8 * 512, int(sb[-1]))


def test_mx_output_reuse_and_determinism():
    """Quantising twice into the same preallocated output (PR 3224 output
    reuse) gives the same bytes; a different input then overwrites them."""
    splits = np.array([256, 0, 128], np.int32)
    a, b = W.normal_bf16((512, 256), 1), W.normal_bf16((512, 256), 2)
    out = gq.alloc_quantized(512, 256, 3, mx_recipe(), "cuda:0", fill=0xAB)
    st = status_dev()
    for bits in (a, a, b, a):
        gq.gq_quantize(bf16_dev(bits), splits_dev(splits), 3, mx_recipe(), out, st)
        check_status(st)
        ora = O.quantize_mx(bits, splits, 3)
        assert_mx_equal(out, ora, 384, int(O.split_scan(splits, 3, 512, 256)[2][-1]))


def test_mx_all_groups_empty():
    splits = np.zeros(4, np.int32)
    out, st = quantize(W.normal_bf16((256, 256), 1), splits, 4, mx_recipe())
    check_status(st)
    assert np.all(host(out.row_data) == 0xAB) and np.all(host(out.row_scale) == 0xAB)
    assert np.all(host(out.col_data) == 0xAB) and np.all(host(out.col_scale) == 0xAB)


@pytest.mark.parametrize("splits,why", [([64, -32], "negative"), ([48, 16], "misaligned"),
                                        ([256, 64], "overflow")])
def test_mx_bad_splits_set_status_and_write_nothing(splits, why):
    out, st = quantize(W.normal_bf16((288, 256), 1), np.array(splits, np.int32), 2, mx_recipe())
    check_status(st, -3)
    for t in (out.row_data, out.row_scale, out.col_data, out.col_scale):
        assert np.all(host(t) == 0xAB), why


def test_noop_flag_skips_every_kernel():
    st = status_dev(-3)
    out, _ = quantize(W.normal_bf16((128, 128), 1), np.array([128], np.int32), 1, mx_recipe(),
                      status=st)
    check_status(st, -3)
    assert np.all(host(out.row_data) == 0xAB) and np.all(host(out.col_scale) == 0xAB)


def test_host_checks():
    x = bf16_dev(W.normal_bf16((128, 256), 1))
    st = status_dev()
    out = gq.alloc_quantized(128, 256, 2, mx_recipe(), "cuda:0")
    with pytest.raises(gq.GQError) as e:       # descriptor declares 2 groups, call says 1
        gq.gq_quantize(x, splits_dev([128]), 1, mx_recipe(), out, st)
    assert e.value.status == -7
    with pytest.raises(gq.GQError) as e:       # rows_cap % G for the uniform split
        gq.gq_quantize(bf16_dev(W.normal_bf16((160, 256), 1)), None, 3, mx_recipe(),
                       gq.alloc_quantized(160, 256, 3, mx_recipe(), "cuda:0"), st)
    assert e.value.status == -2
    with pytest.raises(gq.GQError) as e:       # per-channel has no rowwise orientation
        r = gq.Recipe(gq.RECIPE_CHANNEL128_F32, 1, 1, 1e-30)
        gq.gq_quantize(x, splits_dev([128]), 1, r,
                       gq.alloc_quantized(128, 256, 1, ch_recipe(), "cuda:0"), st)
    assert e.value.status == -4
    with pytest.raises(ValueError):
        gq.gq_quantize(x.cpu(), None, 1, mx_recipe(), gq.alloc_quantized(128, 256, 1, mx_recipe()), st)
    check_status(st)


def test_split_scan_table():
    splits = np.array([96, 0, 160, 32, 0], np.int32)
    G = len(splits)
    table = torch.zeros(3 * (G + 1), dtype=torch.int64, device="cuda:0")
    st = status_dev()
    gq.gq_split_scan(splits_dev(splits), G, 512, 384, gq.RECIPE_MXFP8_1X32, table, st)
    check_status(st)
    off, tp, sb = O.split_scan(splits, G, 512, 384)
    np.testing.assert_array_equal(host(table), np.concatenate([off, tp, sb]))
    gq.gq_split_scan(splits_dev(np.array([128, 256], np.int32)), 2, 512, 384,
                     gq.RECIPE_CHANNEL128_F32, table, st)
    off, tp, sb = O.split_scan(np.array([128, 256], np.int32), 2, 512, 384, O.RECIPE_CHANNEL)
    np.testing.assert_array_equal(host(table)[:9], np.concatenate([off, tp, sb]))
    # NVFP4: the same partition, scale regions of 512 (cols/64) bytes per 128-row tile,
    # the last entry being the bytes the oracle's quantiser fills
    table.zero_()
    gq.gq_split_scan(splits_dev(splits), G, 512, 384, gq.RECIPE_NVFP4_1X16, table, st)
    check_status(st)
    off, tp, _ = O.split_scan(splits, G, 512, 384)
    got = host(table)
    np.testing.assert_array_equal(got[:2 * (G + 1)], np.concatenate([off, tp]))
    np.testing.assert_array_equal(got[2 * (G + 1):], 512 * (384 // 64) * tp)
    assert got[-1] == O.scale_bytes_nvfp4(splits, G, 512, 384)
    gq.gq_split_scan(splits_dev(np.array([128, 48], np.int32)), 2, 512, 384,
                     gq.RECIPE_MXFP8_1X32, table, st)
    check_status(st, -3)


def test_split_scan_many_groups():
    rng = np.random.default_rng(0)
    splits = (rng.integers(0, 5, 1024) * 32).astype(np.int32)
    table = torch.zeros(3 * 1025, dtype=torch.int64, device="cuda:0")
    st = status_dev()
    R = int(splits.sum()) + 32
    gq.gq_split_scan(splits_dev(splits), 1024, R, 256, gq.RECIPE_MXFP8_1X32, table, st)
    check_status(st)
    np.testing.assert_array_equal(host(table), np.concatenate(O.split_scan(splits, 1024, R, 256)))


# ------------------------------------------------------------- per-channel --

@pytest.mark.parametrize("sf", [1.0, 1e-4, 1e-8, 1e-30])
def test_channel_bit_exact_kgrouped_workload(sf):
    w = W.workload("kgrouped_zero_channel")
    dy, x = W.kgrouped_zero_channel_operands(w)
    for bits in (dy, x):
        gpu, st = quantize(bits, w.splits, 4, ch_recipe(sf))
        check_status(st)
        ora = O.quantize_channel(bits, w.splits, 4, zero_scale=sf)
        np.testing.assert_array_equal(host(gpu.col_data), ora.col_data)
        got = host(gpu.col_scale)[: ora.col_scale.size].reshape(ora.col_scale.shape)
        np.testing.assert_array_equal(got.view(np.uint32), ora.col_scale.view(np.uint32))


def test_channel_bit_exact_ragged():
    splits = np.array([256, 0, 128, 384], np.int32)
    R, C = 896, 640
    rng = np.random.default_rng(4)
    x = rng.standard_normal((R, C)).astype(np.float32) * np.exp2(rng.integers(-60, 60, (1, C)))
    x[:, 3] = 0.0
    x[128:256, 7] = 0.0
    bits = W.f32_to_bf16_bits(x.astype(np.float32))
    gpu, st = quantize(bits, splits, 4, ch_recipe(1e-4))
    check_status(st)
    ora = O.quantize_channel(bits, splits, 4, zero_scale=1e-4)
    np.testing.assert_array_equal(host(gpu.col_data)[:768], ora.col_data[:768])
    assert np.all(host(gpu.col_data)[768:] == 0xAB)
    got = host(gpu.col_scale)[: ora.col_scale.size].reshape(ora.col_scale.shape)
    np.testing.assert_array_equal(got.view(np.uint32), ora.col_scale.view(np.uint32))


def test_channel_misaligned_split_rejected():
    out, st = quantize(W.normal_bf16((256, 128), 1), np.array([96, 160], np.int32), 2, ch_recipe())
    check_status(st, -3)
    assert np.all(host(out.col_data) == 0xAB)


# --------------------------------------------------------------- full size --

@pytest.mark.parametrize("name", ["moe_e8", "moe_e64_zipf"])
def test_mx_full_size_activation(name):
    """The full-size token buffers (hidden width), bit-exact in full."""
    w = W.workload(name)
    bits = w.activation(w.hidden, 0)
    _mx_case(bits, w.splits, w.num_groups)


def test_mx_full_size_single_grouped_weight():
    """128 same-shape experts 4096 x 1536 in one buffer, quantised twice into
    the same preallocated output."""
    w = W.workload("single_grouped_weight")
    bits = W.normal_bf16((w.rows_cap, w.hidden), w.seed, scale=0.02)
    x = bf16_dev(bits)
    out = gq.alloc_quantized(w.rows_cap, w.hidden, 128, mx_recipe(), "cuda:0", fill=0xAB)
    st = status_dev()
    for _ in range(2):
        gq.gq_quantize(x, None, 128, mx_recipe(), out, st)
    check_status(st)
    ora = O.quantize_mx(bits, None, 128)
    assert_mx_equal(out, ora, w.rows_cap, int(O.split_scan(None, 128, w.rows_cap, w.hidden)[2][-1]))
