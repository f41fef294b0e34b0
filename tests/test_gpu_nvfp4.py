"""GPU parity of the NVFP4 recipe (E2M1 codes, 16-element E4M3 block scales,
per-group fp32 second-level scale) through the C ABI, against the oracle.

Bar: codes, scale bytes and per-group amax bit-exact (the scale and code
decisions are taken in fp32 on both sides, op by op); rows past the live
total and scale bytes past the grouped extent untouched; GEMMs within 1e-5
relative Frobenius error per group of the oracle's fp64 result on its own
quantisation; empty groups exactly 0; repeated calls bitwise identical."""
import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_grouped_gemm_group_gb300 as gq  # noqa: E402
from _gpu_util import (DEV, REL_TOL, assert_sampled_groups_close,  # noqa: E402
                       assert_sampled_increments_close, bf16_dev, check_status, gather, host,
                       rel_err_per_group, splits_dev, status_dev, stratified_rows)

FILL = 0xAB


def nv_recipe(rowwise=True, colwise=True):
    return gq.Recipe(gq.RECIPE_NVFP4_1X16, int(rowwise), int(colwise), 0.0)


def quantize_nv(bits, splits, G, rowwise=True, colwise=True, status=None):
    x = bf16_dev(bits)
    R, Cc = x.shape
    rec = nv_recipe(rowwise, colwise)
    out = gq.alloc_quantized(R, Cc, G, rec, DEV, fill=FILL)
    st = status_dev() if status is None else status
    gq.gq_quantize(x, splits_dev(splits), G, rec, out, st)
    return out, st


def bounds(splits):
    off = np.concatenate([[0], np.cumsum(splits)])
    return [(int(off[g]), int(off[g + 1])) for g in range(len(splits))]


def operand(L, C, pad, seed, scale=1.0):
    return np.concatenate([W.normal_bf16((L, C), seed, scale=scale), W.uniform_bf16((pad, C), seed + 1, -4, 4)])


def assert_nv_equal(gpu, ora, L, extent):
    if gpu.row_data is not None:
        d = host(gpu.row_data)
        bad = np.argwhere(d[:L] != ora.row_data[:L])
        assert bad.size == 0, f"rowwise codes differ at {len(bad)} bytes, first {bad[0]}: " \
                              f"gpu {d[tuple(bad[0])]:#x} oracle {ora.row_data[tuple(bad[0])]:#x}"
        assert np.all(d[L:] == FILL), "rowwise codes written past the live rows"
        s = host(gpu.row_scale)
        bad = np.flatnonzero(s[:extent] != ora.row_scale[:extent])
        assert bad.size == 0, f"rowwise scales differ at {bad.size} bytes, first {bad[0]}"
        assert np.all(s[extent:] == FILL)
    if gpu.col_data is not None:
        d = host(gpu.col_data)
        bad = np.argwhere(d[:, :L // 2] != ora.col_data[:, :L // 2])
        assert bad.size == 0, f"columnwise codes differ at {len(bad)} bytes, first {bad[0]}: " \
                              f"gpu {d[tuple(bad[0])]:#x} oracle {ora.col_data[tuple(bad[0])]:#x}"
        assert np.all(d[:, L // 2:] == FILL), "columnwise codes written past the live rows"
        s = host(gpu.col_scale)
        bad = np.flatnonzero(s[:extent] != ora.col_scale[:extent])
        assert bad.size == 0, f"columnwise scales differ at {bad.size} bytes, first {bad[0]}"
        assert np.all(s[extent:] == FILL)
    assert np.array_equal(host(gpu.amax)[:len(ora.amax)].view(np.uint32), ora.amax.view(np.uint32))


@pytest.mark.parametrize("splits,C", [([256, 0, 96, 416, 32], 256), ([512], 384), ([0, 0, 64], 128),
                                      ([32] * 12 + [0, 160], 512)])
def test_quantize_matches_oracle_bitwise(splits, C):
    splits = np.array(splits, np.int32)
    G, L, pad = len(splits), int(splits.sum()), 64
    x = operand(L, C, pad, 31)
    q, st = quantize_nv(x, splits, G)
    check_status(st)
    ora = O.quantize_nvfp4(x, splits, G)
    assert_nv_equal(q, ora, L, O.scale_bytes_nvfp4(splits, G, L + pad, C))


@pytest.mark.parametrize("rowwise,colwise", [(True, False), (False, True)])
def test_quantize_one_orientation(rowwise, colwise):
    splits = np.array([128, 64, 0, 224], np.int32)
    G, L, C, pad = 4, 416, 256, 32
    x = operand(L, C, pad, 32, scale=0.01)
    q, st = quantize_nv(x, splits, G, rowwise, colwise)
    check_status(st)
    ora = O.quantize_nvfp4(x, splits, G, rowwise, colwise)
    assert_nv_equal(q, ora, L, O.scale_bytes_nvfp4(splits, G, L + pad, C))


def test_quantize_wide_range_and_ties():
    """Values spanning many binades, exact E2M1 ties after scaling, zero
    blocks and a zero group: subnormal E4M3 scales and round-to-even ties."""
    rng = np.random.default_rng(33)
    L, C = 256, 256
    v = rng.standard_normal((L, C)) * np.exp2(rng.integers(-20, 10, size=(L, 1)))
    v[:, :16] = 0.0                                      # an all-zero block in every row
    v[64:96] = 0.0                                       # group 1 below: all zero
    v[5, 16:32] = [6, 5, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25, -5, -3.5, -2.5, -1.75, -0.75, -0.25, 1e-3, 0]
    x = W.f32_to_bf16_bits(v.astype(np.float32))
    splits = np.array([64, 32, 160], np.int32)
    q, st = quantize_nv(x, splits, 3)
    check_status(st)
    assert_nv_equal(q, O.quantize_nvfp4(x, splits, 3), L, O.scale_bytes_nvfp4(splits, 3, L, C))


def test_quantize_uniform_weights_and_padding_invariance():
    G, N, K = 3, 256, 256
    w = W.normal_bf16((G * N, K), 34, scale=0.02)
    q, st = quantize_nv(w, None, G)
    check_status(st)
    assert_nv_equal(q, O.quantize_nvfp4(w, None, G), G * N, O.scale_bytes_nvfp4(None, G, G * N, K))
    # padding content never matters
    splits = np.array([96, 32], np.int32)
    live = W.normal_bf16((128, 128), 35)
    outs = []
    for fill in (0.0, 3.0, float("nan")):
        q, st = quantize_nv(np.concatenate([live, W.fill_bf16((64, 128), fill)]), splits, 2)
        check_status(st)
        outs.append(q)
    for q in outs[1:]:
        for a in ("row_data", "row_scale", "col_data", "col_scale", "amax"):
            assert torch.equal(getattr(q, a), getattr(outs[0], a)), a


# --------------------------------------------------------------------------- #
# GEMMs                                                                        #
# --------------------------------------------------------------------------- #

CASES = [
    ([256, 0, 96, 416, 32], 256, 512),      # empty, 32-row and ragged groups; half-live 64-row blocks
    ([512, 128], 512, 256),
    ([0, 0, 64], 256, 256),
]


@pytest.mark.parametrize("splits,N,K", CASES)
@pytest.mark.parametrize("dtype", [gq.DTYPE_F32, gq.DTYPE_BF16])
def test_fprop_dgrad_match_oracle(splits, N, K, dtype):
    splits = np.array(splits, np.int32)
    G, L, pad = len(splits), int(splits.sum()), 64
    R = L + pad
    x = operand(L, K, pad, 41)
    dy = operand(L, N, pad, 43)
    w = W.normal_bf16((G * N, K), 45, scale=0.02)
    st = status_dev()
    xq, _ = quantize_nv(x, splits, G, True, False, st)
    dq, _ = quantize_nv(dy, splits, G, True, False, st)
    wq, _ = quantize_nv(w, None, G, True, True, st)
    tdt = torch.float32 if dtype == gq.DTYPE_F32 else torch.bfloat16
    y = torch.full((R, N), float("nan"), dtype=tdt, device=DEV)
    dx = torch.full((R, K), float("nan"), dtype=tdt, device=DEV)
    sp = splits_dev(splits)
    gq.gq_gemm_fprop(xq, wq, sp, G, N, K, y, dtype, st)
    gq.gq_gemm_dgrad(dq, wq, sp, G, N, K, dx, dtype, st)
    check_status(st)
    oxq = O.quantize_nvfp4(x, splits, G, colwise=False)
    odq = O.quantize_nvfp4(dy, splits, G, colwise=False)
    owq = O.quantize_nvfp4(w, None, G)
    want_y = O.gemm_nvfp4("fprop", oxq, owq, splits, G, N, K)
    want_dx = O.gemm_nvfp4("dgrad", odq, owq, splits, G, N, K)
    tol = REL_TOL if dtype == gq.DTYPE_F32 else 2.0 ** -8
    live = [(a, b) for a, b in bounds(splits) if b > a]
    for got, want in ((host(y.float()), want_y), (host(dx.float()), want_dx)):
        errs = rel_err_per_group(got, want, live)
        assert np.all(errs <= tol), errs
        assert np.all(np.isnan(got[L:])), "rows past the live total written"


@pytest.mark.parametrize("splits,N,K", CASES + [([32] * 6 + [0, 224], 256, 256)])
def test_wgrad_matches_oracle(splits, N, K):
    splits = np.array(splits, np.int32)
    G, L, pad = len(splits), int(splits.sum()), 64
    dy = operand(L, N, pad, 51)
    x = operand(L, K, pad, 53)
    st = status_dev()
    dq, _ = quantize_nv(dy, splits, G, False, True, st)
    xq, _ = quantize_nv(x, splits, G, False, True, st)
    sp = splits_dev(splits)
    dw = torch.full((G, N, K), float("nan"), device=DEV)
    gq.gq_gemm_wgrad(dq, xq, sp, G, N, K, dw, False, st)
    init = torch.randn((G, N, K), generator=torch.Generator().manual_seed(55)).to(DEV)
    dwa = init.clone()
    gq.gq_gemm_wgrad(dq, xq, sp, G, N, K, dwa, True, st)
    check_status(st)
    odq = O.quantize_nvfp4(dy, splits, G, rowwise=False)
    oxq = O.quantize_nvfp4(x, splits, G, rowwise=False)
    want = O.gemm_nvfp4("wgrad", odq, oxq, splits, G, N, K)
    got, gota = host(dw), host(dwa)
    for g in range(G):
        if splits[g] == 0:
            assert np.all(got[g] == 0), f"group {g} is empty: dW must be 0"
            assert torch.equal(dwa[g], init[g]), f"group {g} is empty: accumulate must leave dW"
            continue
        e = np.linalg.norm(got[g] - want[g]) / np.linalg.norm(want[g])
        assert e <= REL_TOL, f"group {g}: rel err {e}"
        ea = np.linalg.norm(gota[g] - (host(init[g]) + want[g])) / np.linalg.norm(host(init[g]) + want[g])
        assert ea <= REL_TOL, f"group {g} (accumulate): rel err {ea}"


def test_repeated_calls_bitwise_identical():
    splits = np.array([256, 96, 0, 160], np.int32)
    G, L, N, K, pad = 4, 512, 256, 512, 32
    x = operand(L, K, pad, 61)
    dy = operand(L, N, pad, 62)
    w = W.normal_bf16((G * N, K), 63, scale=0.02)
    st = status_dev()
    sp = splits_dev(splits)
    outs = []
    for _ in range(3):
        xq, _ = quantize_nv(x, splits, G, True, True, st)
        dq, _ = quantize_nv(dy, splits, G, True, True, st)
        wq, _ = quantize_nv(w, None, G, True, True, st)
        y = torch.empty((L + pad, N), device=DEV)
        dx = torch.empty((L + pad, K), device=DEV)
        dw = torch.empty((G, N, K), device=DEV)
        gq.gq_gemm_fprop(xq, wq, sp, G, N, K, y, gq.DTYPE_F32, st)
        gq.gq_gemm_dgrad(dq, wq, sp, G, N, K, dx, gq.DTYPE_F32, st)
        gq.gq_gemm_wgrad(dq, xq, sp, G, N, K, dw, False, st)
        outs.append((xq.row_data.clone(), xq.col_data.clone(), y[:L].clone(), dx[:L].clone(), dw.clone()))
    check_status(st)
    for o in outs[1:]:
        for a, b in zip(o, outs[0]):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_bad_splits_make_every_call_a_noop():
    splits = np.array([48, 16], np.int32)                 # not multiples of 32
    x = operand(64, 256, 0, 71)
    q, st = quantize_nv(x, splits, 2)
    check_status(st, -3)                                  # GQ_ERR_SPLITS
    assert torch.all(q.row_data == FILL) and torch.all(q.col_data == FILL)
    assert torch.all(q.amax.view(torch.uint8) == FILL)


# --------------------------------------------------------------------------- #
# full size: the large MoE layer in the benchmark's launch configuration      #
# --------------------------------------------------------------------------- #

def _bits_of(t):
    return host(t.view(torch.int16)).view(np.uint16)


@pytest.mark.parametrize("fc", [1, 2])
def test_moe_e64_zipf_layer_nvfp4(fc):
    """E = 64, hidden 7168, ffn 2048, 65536 Zipf-routed tokens + 1024 garbage
    rows: every quantised buffer byte for byte against the oracle, and fprop,
    dgrad (fp32 and bf16 outputs) and wgrad (accumulate into an fp32 main
    grad) on sampled outputs: 64 in every non-empty expert plus 4096 over the
    layer, each expert's sampled relative error (of the wgrad's increment,
    with the fp32 rounding of the final add allowed per element) within
    1e-5."""
    w = W.workload("moe_e64_zipf")
    E, R, L = w.num_groups, w.rows_cap, w.live_rows
    K, N = (w.hidden, w.ffn) if fc == 1 else (w.ffn, w.hidden)
    s = 0 if fc == 1 else 1
    x = W.device_activation(w, K, 40 + s, device=DEV)
    dy = W.device_activation(w, N, 42 + s, device=DEV)
    wt = W.device_normal_bf16((E * N, K), w.seed, 0.02, 44 + s, DEV)
    main = W.device_normal_bf16((E, N, K), w.seed, 1e-3, 46 + s, DEV).float()
    main0 = main.clone()
    sp = torch.as_tensor(w.splits).to(DEV)
    st = status_dev()
    rec = nv_recipe()
    q = {k: gq.alloc_quantized(t.shape[0], t.shape[1], E, rec, DEV, fill=FILL)
         for k, t in (("x", x), ("dy", dy), ("w", wt))}
    gq.gq_quantize(x, sp, E, rec, q["x"], st)
    gq.gq_quantize(dy, sp, E, rec, q["dy"], st)
    gq.gq_quantize(wt, None, E, rec, q["w"], st)
    y = torch.empty((R, N), dtype=torch.float32, device=DEV)
    dx = torch.empty((R, K), dtype=torch.bfloat16, device=DEV)
    dx32 = torch.empty((R, K), dtype=torch.float32, device=DEV)
    gq.gq_gemm_fprop(q["x"], q["w"], sp, E, N, K, y, gq.DTYPE_F32, st)
    gq.gq_gemm_dgrad(q["dy"], q["w"], sp, E, N, K, dx, gq.DTYPE_BF16, st)
    gq.gq_gemm_dgrad(q["dy"], q["w"], sp, E, N, K, dx32, gq.DTYPE_F32, st)
    gq.gq_gemm_wgrad(q["dy"], q["x"], sp, E, N, K, main, True, st)
    torch.cuda.synchronize()
    check_status(st)

    ox = O.quantize_nvfp4(_bits_of(x), w.splits, E)
    ody = O.quantize_nvfp4(_bits_of(dy), w.splits, E)
    ow = O.quantize_nvfp4(_bits_of(wt), None, E)
    assert_nv_equal(q["x"], ox, L, O.scale_bytes_nvfp4(w.splits, E, R, K))
    assert_nv_equal(q["dy"], ody, L, O.scale_bytes_nvfp4(w.splits, E, R, N))
    assert_nv_equal(q["w"], ow, E * N, O.scale_bytes_nvfp4(None, E, E * N, K))

    rng = np.random.default_rng(98)
    n_s, per_group = 4096, 64
    rows, grp = stratified_rows(rng, w.splits, per_group, n_s)
    cn, ck = rng.integers(0, N, rows.size), rng.integers(0, K, rows.size)

    want = O.gemm_nvfp4_sample("fprop", ox, ow, w.splits, E, N, K, rows, cn)
    assert_sampled_groups_close(gather(y, rows, cn), want, grp, "fprop fp32")
    want = O.gemm_nvfp4_sample("dgrad", ody, ow, w.splits, E, N, K, rows, ck)
    assert_sampled_groups_close(gather(dx32, rows, ck), want, grp, "dgrad fp32")
    got = gather(dx, rows, ck)
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-6), "dgrad bf16"
    live = np.flatnonzero(w.splits > 0)
    g = np.concatenate([np.repeat(live, per_group), rng.choice(live, n_s)])
    cn, ck = rng.integers(0, N, g.size), rng.integers(0, K, g.size)
    want = O.gemm_nvfp4_sample("wgrad", ody, ox, w.splits, E, N, K, cn, ck, g)
    assert_sampled_increments_close(gather(main, g, cn, ck), gather(main0, g, cn, ck), want, g,
                                    "wgrad (accumulate)")
    for e in np.flatnonzero(w.splits == 0):
        assert torch.equal(main[e], main0[e]), f"empty expert {e} changed"


def test_buffer_past_2_31_elements_nvfp4():
    """X [300544, 7168] bf16 (R * K > 2^31; the last group's rows straddle
    element 2^31) on NVFP4 operands: quantisation of both orientations,
    fprop, dgrad (dX fp32, 8.6 GB) and the k-grouped wgrad.  Groups 0 and 2
    match the oracle run on that group alone (its amax and S_g come from the
    group's own rows): codes, scale regions and amax bit for bit, GEMMs
    within 1e-5; the middle group's outputs are finite."""
    K, N, G, R, pad = 7168, 256, 3, 300544, 128
    L = R - pad
    splits = np.array([1024, L - 2048, 1024], np.int32)
    assert R * K > 2 ** 31 and (L - 1024) * K < 2 ** 31 < L * K
    x = W.device_normal_bf16((R, K), 6, 1.0, 50, DEV)
    dy = W.device_normal_bf16((R, N), 6, 1.0, 51, DEV)
    wt = W.device_normal_bf16((G * N, K), 6, 0.02, 52, DEV)
    sp = torch.as_tensor(splits).to(DEV)
    st = status_dev()
    rec = nv_recipe()
    q = {k: gq.alloc_quantized(t.shape[0], t.shape[1], G, rec, DEV, fill=FILL)
         for k, t in (("x", x), ("dy", dy), ("w", wt))}
    gq.gq_quantize(x, sp, G, rec, q["x"], st)
    gq.gq_quantize(dy, sp, G, rec, q["dy"], st)
    gq.gq_quantize(wt, None, G, rec, q["w"], st)
    y = torch.empty((R, N), dtype=torch.float32, device=DEV)
    dx = torch.empty((R, K), dtype=torch.float32, device=DEV)
    dw = torch.empty((G, N, K), dtype=torch.float32, device=DEV)
    gq.gq_gemm_fprop(q["x"], q["w"], sp, G, N, K, y, gq.DTYPE_F32, st)
    gq.gq_gemm_dgrad(q["dy"], q["w"], sp, G, N, K, dx, gq.DTYPE_F32, st)
    gq.gq_gemm_wgrad(q["dy"], q["x"], sp, G, N, K, dw, False, st)
    torch.cuda.synchronize()
    check_status(st)

    def rel(got, want):
        return np.linalg.norm(got - want) / np.linalg.norm(want)

    off, tp, _ = O.split_scan(splits, G, R, K)
    for g in (0, 2):
        a, b = int(off[g]), int(off[g + 1])
        one = np.array([b - a], np.int32)
        xg, dyg, wg = _bits_of(x[a:b]), _bits_of(dy[a:b]), _bits_of(wt[g * N:(g + 1) * N])
        for key, bits, cols in (("x", xg, K), ("dy", dyg, N)):
            ora = O.quantize_nvfp4(bits, one, 1)
            sb, nbytes = 512 * (cols // 64) * int(tp[g]), 512 * (cols // 64) * ((b - a + 127) // 128)
            assert np.array_equal(host(q[key].row_data[a:b]), ora.row_data), f"{key} row codes, group {g}"
            assert np.array_equal(host(q[key].col_data[:, a // 2:b // 2]), ora.col_data), f"{key} col codes, group {g}"
            for t, o in ((q[key].row_scale, ora.row_scale), (q[key].col_scale, ora.col_scale)):
                assert np.array_equal(host(t[sb:sb + nbytes]), o[:nbytes]), f"{key} scales, group {g}"
            assert host(q[key].amax)[g:g + 1].view(np.uint32) == ora.amax.view(np.uint32), f"{key} amax, group {g}"
        ow = O.quantize_nvfp4(wg, None, 1)
        want = O.gemm_nvfp4("fprop", O.quantize_nvfp4(xg, one, 1, colwise=False), ow, one, 1, N, K)
        assert rel(host(y[a:b]), want) <= REL_TOL, f"fprop group {g}"
        want = O.gemm_nvfp4("dgrad", O.quantize_nvfp4(dyg, one, 1, colwise=False), ow, one, 1, N, K)
        assert rel(host(dx[a:b]), want) <= REL_TOL, f"dgrad group {g}"
        want = O.gemm_nvfp4("wgrad", O.quantize_nvfp4(dyg, one, 1, rowwise=False),
                            O.quantize_nvfp4(xg, one, 1, rowwise=False), one, 1, N, K)
        assert rel(host(dw[g]), want[0]) <= REL_TOL, f"wgrad group {g}"
    mid = slice(int(off[1]), int(off[2]))
    assert bool(torch.isfinite(y[mid]).all()) and bool(torch.isfinite(dx[mid]).all())
    assert bool(torch.isfinite(dw[1]).all())
    for key in ("x", "dy"):
        assert bool((q[key].row_data[L:] == FILL).all()) and bool((q[key].col_data[:, L // 2:] == FILL).all())
