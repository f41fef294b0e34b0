"""GPU parity of the grouped GEMMs (fprop, dgrad, k-grouped wgrad) against the
CPU oracle, through the C ABI.

Bar: per-group relative Frobenius error <= 1e-5 against the oracle's fp64
result on the oracle's own quantisation of the same seeded inputs; bitwise
equality where the arithmetic is exact; padding rows, empty groups and
all-zero channels never affect a result; bitwise determinism.
"""
import json
import os

import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_grouped_gemm_group_gb300 as gq  # noqa: E402
from _gpu_util import (DEV, REL_TOL, bf16_dev, ch_recipe, check_status, host, mx_recipe,  # noqa: E402
                       quantize, rel_err_per_group, splits_dev, status_dev)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bounds(splits):
    off = np.concatenate([[0], np.cumsum(splits)])
    return [(int(off[g]), int(off[g + 1])) for g in range(len(splits))]


# --------------------------------------------------------------------------- #
# the three GEMMs, GPU side (C ABI) and oracle side                            #
# --------------------------------------------------------------------------- #

def gpu_fprop(x_bits, w_bits, splits, G, N, K, dtype=gq.DTYPE_F32):
    st = status_dev()
    xq, _ = quantize(x_bits, splits, G, mx_recipe(True, False), status=st)
    wq, _ = quantize(w_bits, None, G, mx_recipe(True, False), status=st)
    tdt = torch.float32 if dtype == gq.DTYPE_F32 else torch.bfloat16
    y = torch.full((x_bits.shape[0], N), float("nan"), dtype=tdt, device=DEV)
    gq.gq_gemm_fprop(xq, wq, splits_dev(splits), G, N, K, y, dtype, st)
    check_status(st)
    return host(y.float()) if dtype == gq.DTYPE_BF16 else host(y)


def ora_fprop(x_bits, w_bits, splits, G, N, K):
    return O.gemm_fprop(O.quantize_mx(x_bits, splits, G, colwise=False),
                        O.quantize_mx(w_bits, None, G, colwise=False), splits, G, N, K)


def gpu_dgrad(dy_bits, w_bits, splits, G, N, K, dtype=gq.DTYPE_F32):
    st = status_dev()
    dyq, _ = quantize(dy_bits, splits, G, mx_recipe(True, False), status=st)
    wq, _ = quantize(w_bits, None, G, mx_recipe(False, True), status=st)
    tdt = torch.float32 if dtype == gq.DTYPE_F32 else torch.bfloat16
    dx = torch.full((dy_bits.shape[0], K), float("nan"), dtype=tdt, device=DEV)
    gq.gq_gemm_dgrad(dyq, wq, splits_dev(splits), G, N, K, dx, dtype, st)
    check_status(st)
    return host(dx.float()) if dtype == gq.DTYPE_BF16 else host(dx)


def ora_dgrad(dy_bits, w_bits, splits, G, N, K):
    return O.gemm_dgrad(O.quantize_mx(dy_bits, splits, G, colwise=False),
                        O.quantize_mx(w_bits, None, G, rowwise=False), splits, G, N, K)


def gpu_wgrad(dy_bits, x_bits, splits, G, N, K, accumulate=False, init=None, recipe=None, workspace="new"):
    st = status_dev()
    recipe = recipe or mx_recipe(False, True)
    dyq, _ = quantize(dy_bits, splits, G, recipe, status=st)
    xq, _ = quantize(x_bits, splits, G, recipe, status=st)
    if init is None:
        dw = torch.full((G, N, K), float("nan"), dtype=torch.float32, device=DEV)
    else:
        dw = torch.from_numpy(np.ascontiguousarray(init, np.float32)).to(DEV)
    gq.gq_gemm_wgrad(dyq, xq, splits_dev(splits), G, N, K, dw, accumulate, st, workspace=workspace)
    check_status(st)
    return host(dw)


def ora_wgrad(dy_bits, x_bits, splits, G, N, K, accumulate=False, init=None, zero_scale=None):
    if zero_scale is None:
        dyq = O.quantize_mx(dy_bits, splits, G, rowwise=False)
        xq = O.quantize_mx(x_bits, splits, G, rowwise=False)
    else:
        dyq = O.quantize_channel(dy_bits, splits, G, zero_scale)
        xq = O.quantize_channel(x_bits, splits, G, zero_scale)
    return O.gemm_wgrad(dyq, xq, splits, G, N, K, accumulate,
                        None if init is None else np.asarray(init, np.float32).astype(np.float64))


def assert_rows_close(got, want, splits, what):
    errs = rel_err_per_group(got, want, bounds(splits))
    assert np.all(errs <= REL_TOL), f"{what}: per-group rel err {errs}"


def assert_groups_close(got, want, what):
    for g in range(got.shape[0]):
        nw = np.linalg.norm(want[g])
        if nw == 0:
            assert np.all(got[g] == 0), f"{what}: group {g} should be exactly zero"
        else:
            e = np.linalg.norm(got[g].astype(np.float64) - want[g]) / nw
            assert e <= REL_TOL, f"{what}: group {g} rel err {e}"


CASES = [
    # splits, pad rows, N, K
    ([512], 256, 256, 1024),
    ([96, 0, 160, 32], 64, 384, 256),
    ([128, 384, 0, 32, 224], 32, 256, 640),
    ([0, 0, 64], 0, 128, 128),
    ([1024, 32, 736], 96, 512, 512),
    ([32, 0, 96, 288, 160], 64, 256, 256),       # CTA-pair tiles with empty halves
    ([2048, 224], 0, 768, 512),
]


@pytest.mark.parametrize("splits,pad,N,K", CASES)
def test_fprop_matches_oracle(splits, pad, N, K):
    splits = np.array(splits, np.int32)
    G, L = len(splits), int(splits.sum())
    x = np.concatenate([W.normal_bf16((L, K), 1), W.uniform_bf16((pad, K), 2, -4, 4)])
    w = W.normal_bf16((G * N, K), 3, scale=0.02)
    got = gpu_fprop(x, w, splits, G, N, K)
    want = ora_fprop(x, w, splits, G, N, K)
    assert_rows_close(got, want, splits, "fprop")
    assert np.all(np.isnan(got[L:])), "fprop wrote rows past the live total"


@pytest.mark.parametrize("splits,pad,N,K", CASES)
def test_dgrad_matches_oracle(splits, pad, N, K):
    splits = np.array(splits, np.int32)
    G, L = len(splits), int(splits.sum())
    dy = np.concatenate([W.normal_bf16((L, N), 4), W.uniform_bf16((pad, N), 5, -4, 4)])
    w = W.normal_bf16((G * N, K), 6, scale=0.02)
    got = gpu_dgrad(dy, w, splits, G, N, K)
    want = ora_dgrad(dy, w, splits, G, N, K)
    assert_rows_close(got, want, splits, "dgrad")
    assert np.all(np.isnan(got[L:])), "dgrad wrote rows past the live total"


@pytest.mark.parametrize("splits,pad,N,K", CASES)
def test_wgrad_matches_oracle(splits, pad, N, K):
    splits = np.array(splits, np.int32)
    G, L = len(splits), int(splits.sum())
    dy = np.concatenate([W.normal_bf16((L, N), 7), W.uniform_bf16((pad, N), 8, -4, 4)])
    x = np.concatenate([W.normal_bf16((L, K), 9), W.uniform_bf16((pad, K), 10, -4, 4)])
    got = gpu_wgrad(dy, x, splits, G, N, K)
    want = ora_wgrad(dy, x, splits, G, N, K)
    assert_groups_close(got, want, "wgrad")


@pytest.mark.parametrize("K", [512, 384])
def test_wgrad_run_time_order_matches_static_order(K):
    """Skewed splits (one large group, empty and 32-row groups): the run-time
    tile order (claim workspace; both ends of the size-sorted group list) and
    the static order give the same bits, and match the oracle; a reused
    workspace is cleared by every call."""
    splits = np.array([32, 0, 1088, 96, 0, 32, 320, 64], np.int32)
    G, L, N = len(splits), int(splits.sum()), 256
    dy = np.concatenate([W.normal_bf16((L, N), 31), W.uniform_bf16((64, N), 32, -4, 4)])
    x = np.concatenate([W.normal_bf16((L, K), 33), W.uniform_bf16((64, K), 34, -4, 4)])
    init = W.bf16_bits_to_f32(W.normal_bf16((G, N, K), 35))
    ws = torch.empty(gq.WGRAD_WORKSPACE_BYTES, dtype=torch.uint8, device=DEV)
    stat = gpu_wgrad(dy, x, splits, G, N, K, True, init, workspace=None)
    dyn1 = gpu_wgrad(dy, x, splits, G, N, K, True, init, workspace=ws)
    dyn2 = gpu_wgrad(dy, x, splits, G, N, K, True, init, workspace=ws)
    assert np.array_equal(stat.view(np.uint32), dyn1.view(np.uint32))
    assert np.array_equal(dyn1.view(np.uint32), dyn2.view(np.uint32))
    want = ora_wgrad(dy, x, splits, G, N, K, True, init)
    for g in range(G):
        if splits[g] == 0:
            assert np.array_equal(dyn1[g].view(np.uint32), init[g].view(np.uint32))
    assert_groups_close(dyn1, want, "wgrad")
    # accumulate = 0: empty groups are written as +0.0 in either order
    z_stat = gpu_wgrad(dy, x, splits, G, N, K, False, None, workspace=None)
    z_dyn = gpu_wgrad(dy, x, splits, G, N, K, False, None, workspace=ws)
    assert np.array_equal(z_stat.view(np.uint32), z_dyn.view(np.uint32))
    assert np.all(z_dyn[splits == 0] == 0)


@pytest.mark.parametrize("kind,K", [("fprop", 384), ("dgrad", 384), ("fprop", 512), ("dgrad", 512)])
def test_bf16_output_within_one_ulp(kind, K):
    """bf16 output: 128- and 256-column tiles (dgrad's output width is K)."""
    splits = np.array([160, 96], np.int32)
    G, N = 2, 256
    a = W.normal_bf16((288, K if kind == "fprop" else N), 11)
    w = W.normal_bf16((G * N, K), 12, scale=0.05)
    if kind == "fprop":
        full = gpu_fprop(a, w, splits, G, N, K, gq.DTYPE_BF16)
        want = ora_fprop(a, w, splits, G, N, K)[:256]
    else:
        full = gpu_dgrad(a, w, splits, G, N, K, gq.DTYPE_BF16)
        want = ora_dgrad(a, w, splits, G, N, K)[:256]
    assert np.all(np.isnan(full[256:])), "wrote rows past the live total"
    got = full[:256]
    want_b = W.bf16_bits_to_f32(W.f32_to_bf16_bits(want.astype(np.float32))).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(want), 1e-30))) - 7)
    assert np.all(np.abs(got - want_b) <= ulp + 1e-30)


def test_exact_arithmetic_bitwise():
    """Integers times a per-tensor power of two quantise exactly and every
    fp32 partial sum is exact: the GPU must equal the oracle bit for bit."""
    rng = np.random.default_rng(21)
    splits = np.array([96, 0, 224, 32], np.int32)
    G, N, K = 4, 256, 512
    L = int(splits.sum())

    def ints(shape, p):
        return W.f32_to_bf16_bits((rng.integers(-14, 15, shape) * 2.0 ** p).astype(np.float32))

    x, w, dy = ints((L + 32, K), -3), ints((G * N, K), -5), ints((L + 32, N), -4)
    y = gpu_fprop(x, w, splits, G, N, K)
    np.testing.assert_array_equal(y[:L], ora_fprop(x, w, splits, G, N, K)[:L].astype(np.float32))
    dx = gpu_dgrad(dy, w, splits, G, N, K)
    np.testing.assert_array_equal(dx[:L], ora_dgrad(dy, w, splits, G, N, K)[:L].astype(np.float32))
    dw = gpu_wgrad(dy, x, splits, G, N, K)
    np.testing.assert_array_equal(dw, ora_wgrad(dy, x, splits, G, N, K).astype(np.float32))


def test_wgrad_accumulate_and_empty_groups():
    splits = np.array([0, 192, 0, 64], np.int32)
    G, N, K = 4, 128, 256
    dy, x = W.normal_bf16((320, N), 13), W.normal_bf16((320, K), 14)
    init = np.random.default_rng(15).standard_normal((G, N, K)).astype(np.float32)
    got = gpu_wgrad(dy, x, splits, G, N, K, accumulate=True, init=init)
    np.testing.assert_array_equal(got[0], init[0])          # empty: bit-unchanged
    np.testing.assert_array_equal(got[2], init[2])
    want = ora_wgrad(dy, x, splits, G, N, K, True, init)
    assert_groups_close(got, want, "wgrad accumulate")
    fresh = gpu_wgrad(dy, x, splits, G, N, K)                 # accumulate = 0: +0.0
    assert np.all(fresh[0] == 0) and not np.any(np.signbit(fresh[0]))


@pytest.mark.parametrize("splits", [
    [1536, 32, 0, 64, 32, 96],       # skewed: boxes 1 and 3 of each warp's share go by reduce-add
    [352, 320, 0, 288, 352, 320],    # even: every box by load + add + store
])
def test_wgrad_accumulate_skewed_and_even_splits(splits):
    """The accumulating wide wgrad (k % 256 == 0) adds its tiles into the main
    grad by two routes, chosen on the device from the split sizes: with
    skewed splits half of each warp's boxes go by TMA reduce-add, with even
    splits all by load + add + store.  Both match the oracle per group, give
    the same bits with the run-time and the static tile order, and leave an
    empty group bit-unchanged."""
    splits = np.array(splits, np.int32)
    G, N, K = len(splits), 256, 512
    L = int(splits.sum())
    dy = np.concatenate([W.normal_bf16((L, N), 16), W.uniform_bf16((64, N), 17, -4, 4)])
    x = np.concatenate([W.normal_bf16((L, K), 18), W.uniform_bf16((64, K), 19, -4, 4)])
    init = np.random.default_rng(20).standard_normal((G, N, K)).astype(np.float32)
    got = gpu_wgrad(dy, x, splits, G, N, K, accumulate=True, init=init)
    static = gpu_wgrad(dy, x, splits, G, N, K, accumulate=True, init=init, workspace=None)
    np.testing.assert_array_equal(got.view(np.uint32), static.view(np.uint32))
    np.testing.assert_array_equal(got[2], init[2])
    want = ora_wgrad(dy, x, splits, G, N, K, True, init)
    for g in range(G):
        if splits[g]:
            inc, ref = got[g].astype(np.float64) - init[g], want[g] - init[g]
            slack = 2.0 ** -24 * np.abs(got[g].astype(np.float64))
            resid = np.maximum(np.abs(inc - ref) - slack, 0.0)
            assert np.linalg.norm(resid) <= REL_TOL * np.linalg.norm(ref), f"group {g}"


def test_wgrad_empty_buffer_zero_fill():
    G, N, K = 3, 128, 128
    st = status_dev()
    r = mx_recipe(False, True)
    dyq = gq.alloc_quantized(0, N, G, r, DEV)
    xq = gq.alloc_quantized(0, K, G, r, DEV)
    dyq.desc.recipe.colwise = xq.desc.recipe.colwise = 1
    dw = torch.full((G, N, K), float("nan"), device=DEV)
    gq.gq_gemm_wgrad(dyq, xq, splits_dev([0, 0, 0]), G, N, K, dw, False, st)
    check_status(st)
    assert torch.all(dw == 0)


# ------------------------------------------------ the pages' own checks --

def test_padded_single_group_wgrad_rel_err_zero():
    """TransformerEngine issue 3484: G = 1, 512 live rows in a 768-row buffer;
    the wgrad with the tail zero-filled or 3.0-filled equals the unpadded
    wgrad exactly (rel_err 0, no non-finite value), and the fprop rows agree."""
    gold = json.load(open(os.path.join(GOLDEN, "padded_wgrad_expected.json")))
    H = gold["hidden"]
    live_x, live_dy = W.normal_bf16((512, H), 1, stream=0), W.normal_bf16((512, H), 1, stream=1)
    s = np.array([512], np.int32)
    ref = gpu_wgrad(live_dy, live_x, s, 1, H, H)
    w = W.normal_bf16((H, H), 1, scale=1 / 32, stream=2)
    ref_y = gpu_fprop(live_x, w, s, 1, H, H)
    for label, arm in gold["arms"].items():
        pad = W.fill_bf16((gold["pad_rows"], H), arm["fill"])
        got = gpu_wgrad(np.concatenate([live_dy, pad]), np.concatenate([live_x, pad]), s, 1, H, H)
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel == arm["rel_err"], label
        assert int((~np.isfinite(got)).sum()) == arm["non_finite"] and got.size == arm["numel"]
        y = gpu_fprop(np.concatenate([live_x, pad]), w, s, 1, H, H)
        np.testing.assert_array_equal(y[:512], ref_y)
    want = ora_wgrad(live_dy, live_x, s, 1, H, H)
    assert_groups_close(ref, want, "padded single group")


@pytest.fixture(scope="module")
def kgrouped():
    gold = json.load(open(os.path.join(GOLDEN, "kgrouped_wgrad_reference_norm.json")))
    w = W.workload("kgrouped_zero_channel")
    dy, x = W.kgrouped_zero_channel_operands(w)
    return gold, w, dy, x


@pytest.mark.parametrize("sf", [1.0, 1e-4, 1e-8, 1e-30])
def test_kgrouped_channel_wgrad(kgrouped, sf):
    """DeepGEMM issue 365 data: per-channel recipe, every sf_val: within 1e-5
    of the oracle, zero-channel rows exactly 0, no blow-up, and bitwise
    independent of sf_val."""
    gold, w, dy, x = kgrouped
    got = gpu_wgrad(dy, x, w.splits, 4, 2048, 2048, recipe=ch_recipe(sf))
    want = ora_wgrad(dy, x, w.splits, 4, 2048, 2048, zero_scale=sf)
    assert_groups_close(got, want, f"channel wgrad sf={sf}")
    for e, k in enumerate(gold["ks"]):
        if k == 128:
            assert np.all(got[e, 0] == 0)
    norms = np.linalg.norm(got.reshape(4, -1).astype(np.float64), axis=1)
    ref_norms = np.linalg.norm(want.reshape(4, -1), axis=1)
    assert np.all(norms <= np.maximum(gold["blowup_factor"] * ref_norms, gold["blowup_floor"]))
    assert abs(norms.max() / gold["reference_max_norm"] - 1) < 0.02
    base = gpu_wgrad(dy, x, w.splits, 4, 2048, 2048, recipe=ch_recipe(1e-30))
    np.testing.assert_array_equal(got, base)


def test_kgrouped_mx_wgrad(kgrouped):
    gold, w, dy, x = kgrouped
    got = gpu_wgrad(dy, x, w.splits, 4, 2048, 2048)
    want = ora_wgrad(dy, x, w.splits, 4, 2048, 2048)
    assert_groups_close(got, want, "mx wgrad")
    for e, k in enumerate(gold["ks"]):
        if k == 128:
            assert np.all(got[e, 0] == 0)


@pytest.mark.parametrize("recipe", ["channel", "mx"])
def test_kgrouped_wgrad_deterministic_10000_calls(kgrouped, recipe):
    """10,000 repeated calls on the same operands are bitwise identical and
    never blow up (the DeepGEMM issue 365 loop)."""
    gold, w, dy, x = kgrouped
    r = ch_recipe(1.0) if recipe == "channel" else mx_recipe(False, True)
    st = status_dev()
    dyq, _ = quantize(dy, w.splits, 4, r, status=st)
    xq, _ = quantize(x, w.splits, 4, r, status=st)
    sp = splits_dev(w.splits)
    ref = torch.empty((4, 2048, 2048), device=DEV)
    gq.gq_gemm_wgrad(dyq, xq, sp, 4, 2048, 2048, ref, False, st)
    out = torch.empty_like(ref)
    mismatches = torch.zeros((), dtype=torch.int64, device=DEV)
    for _ in range(10000):
        out.zero_()
        gq.gq_gemm_wgrad(dyq, xq, sp, 4, 2048, 2048, out, False, st)
        mismatches += (out != ref).any()
    check_status(st)
    assert int(mismatches.item()) == 0
    norms = torch.linalg.vector_norm(ref.reshape(4, -1), dim=1)
    assert float(norms.max()) < 1.0 and abs(float(norms.max()) / gold["reference_max_norm"] - 1) < 0.02


# ----------------------------------------------------- status and noop --

def test_gemm_bad_splits_and_noop():
    splits = np.array([128, 128], np.int32)
    G, N, K = 2, 128, 128
    x = W.normal_bf16((256, K), 1)
    st = status_dev()
    xq, _ = quantize(x, splits, G, mx_recipe(True, True), status=st)
    wq, _ = quantize(W.normal_bf16((G * N, K), 2), None, G, mx_recipe(True, True), status=st)
    check_status(st)
    y = torch.full((256, N), float("nan"), device=DEV)
    gq.gq_gemm_fprop(xq, wq, splits_dev([128, 48]), G, N, K, y, gq.DTYPE_F32, st)
    check_status(st, -3)                      # misaligned split: nothing written
    assert torch.all(torch.isnan(y))
    gq.gq_gemm_fprop(xq, wq, splits_dev(splits), G, N, K, y, gq.DTYPE_F32, st)
    assert torch.all(torch.isnan(y))          # status still set: the call is a no-op
    dw = torch.full((G, N, K), float("nan"), device=DEV)
    gq.gq_gemm_wgrad(xq, xq, splits_dev(splits), G, N, K, dw, False, st)
    assert torch.all(torch.isnan(dw))
    st.zero_()
    gq.gq_gemm_fprop(xq, wq, splits_dev([128, 256]), G, N, K, y, gq.DTYPE_F32, st)
    check_status(st, -3)                      # sum past rows_cap


def test_gemm_host_checks():
    st = status_dev()
    xq, _ = quantize(W.normal_bf16((256, 256), 1), [256], 1, mx_recipe(True, False), status=st)
    wq, _ = quantize(W.normal_bf16((128, 256), 2), None, 1, mx_recipe(True, False), status=st)
    y = torch.empty((256, 128), device=DEV)
    with pytest.raises(gq.GQError) as e:           # dgrad needs W columnwise
        gq.gq_gemm_dgrad(xq, wq, splits_dev([256]), 1, 256, 128, y, gq.DTYPE_F32, st)
    assert e.value.status in (-4, -7)
    with pytest.raises(gq.GQError) as e:           # k disagrees with the descriptor
        gq.gq_gemm_fprop(xq, wq, splits_dev([256]), 1, 128, 384, y, gq.DTYPE_F32, st)
    assert e.value.status == -7
    with pytest.raises(gq.GQError) as e:           # n not a multiple of 128
        gq.gq_gemm_fprop(xq, wq, splits_dev([256]), 1, 96, 256, y, gq.DTYPE_F32, st)
    assert e.value.status == -2
    check_status(st)


def test_fprop_repeat_bitwise():
    splits = np.array([224, 96, 0, 416], np.int32)
    G, N, K = 4, 256, 512
    st = status_dev()
    xq, _ = quantize(W.normal_bf16((800, K), 1), splits, G, mx_recipe(True, False), status=st)
    wq, _ = quantize(W.normal_bf16((G * N, K), 2), None, G, mx_recipe(True, False), status=st)
    ys = []
    for _ in range(20):
        y = torch.zeros((800, N), device=DEV)
        gq.gq_gemm_fprop(xq, wq, splits_dev(splits), G, N, K, y, gq.DTYPE_F32, st)
        ys.append(y)
    check_status(st)
    for y in ys[1:]:
        assert torch.equal(y, ys[0])
