"""Full-size parity in the launch configuration the benchmark times.

The large MoE layer (E = 64, hidden 7168, ffn 2048, 65536 Zipf-routed tokens
plus 1024 garbage rows) and the E = 8 layer (hidden 4096, ffn 2048, 16384
tokens): inputs drawn on the device by the seeded generators, every quantised
buffer compared byte for byte with the oracle, and fprop / dgrad / wgrad
(accumulate into a fp32 main grad) compared on sampled outputs that the
oracle computes one dot product at a time: 64 outputs in every non-empty
expert (so a 32-token expert is held to the bar as closely as the largest)
plus 4096 drawn over the whole layer.  fprop and dgrad are checked with fp32
outputs, per group, at 1e-5 relative Frobenius error of the samples (and
their bf16 outputs within one bf16 rounding); the accumulating wgrad's
increment main - main0 of every expert likewise, with only the fp32 rounding
of the final add allowed per element.

A buffer of more than 2^31 elements ([300544, 7168] bf16) runs the same
calls; its first and last groups are compared with the oracle run on each
group alone (a grouped quantisation equals the single-group quantisation of
each group's rows, bitwise: a pinned property of the oracle).
"""
import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_grouped_gemm_group_gb300 as gq  # noqa: E402
from _gpu_util import (DEV, REL_TOL, assert_mx_equal, assert_sampled_groups_close,  # noqa: E402
                       assert_sampled_increments_close, check_status, gather, host, mx_recipe, status_dev,
                       stratified_rows)

N_SAMPLES = 4096      # drawn uniformly over the live outputs
PER_GROUP = 64        # drawn in every non-empty group on top of those


def bits_of(t):
    return host(t.view(torch.int16)).view(np.uint16)


def run_layer(name, fc):
    w = W.workload(name)
    E, R, L = w.num_groups, w.rows_cap, w.live_rows
    K, N = (w.hidden, w.ffn) if fc == 1 else (w.ffn, w.hidden)     # fc: Y = X W^T, X [R, K], W_e [N, K]
    s = 0 if fc == 1 else 1
    x = W.device_activation(w, K, s, device=DEV)
    dy = W.device_activation(w, N, 2 + s, device=DEV)
    wt = W.device_normal_bf16((E * N, K), w.seed, 0.02, 10 + s, DEV)
    main = W.device_normal_bf16((E, N, K), w.seed, 1e-3, 20 + s, DEV).float()
    main0 = main.clone()
    sp = torch.as_tensor(w.splits).to(DEV)
    st = status_dev()
    mx = mx_recipe()
    q = {k: gq.alloc_quantized(t.shape[0], t.shape[1], E, mx, DEV, fill=0xAB)
         for k, t in (("x", x), ("dy", dy), ("w", wt))}
    gq.gq_quantize(x, sp, E, mx, q["x"], st)
    gq.gq_quantize(dy, sp, E, mx, q["dy"], st)
    gq.gq_quantize(wt, None, E, mx, q["w"], st)
    y = torch.empty((R, N), dtype=torch.bfloat16, device=DEV)
    dx = torch.empty((R, K), dtype=torch.bfloat16, device=DEV)
    gq.gq_gemm_fprop(q["x"], q["w"], sp, E, N, K, y, gq.DTYPE_BF16, st)
    gq.gq_gemm_dgrad(q["dy"], q["w"], sp, E, N, K, dx, gq.DTYPE_BF16, st)
    y32 = torch.empty((R, N), dtype=torch.float32, device=DEV)
    dx32 = torch.empty((R, K), dtype=torch.float32, device=DEV)
    gq.gq_gemm_fprop(q["x"], q["w"], sp, E, N, K, y32, gq.DTYPE_F32, st)
    gq.gq_gemm_dgrad(q["dy"], q["w"], sp, E, N, K, dx32, gq.DTYPE_F32, st)
    gq.gq_gemm_wgrad(q["dy"], q["x"], sp, E, N, K, main, True, st)
    torch.cuda.synchronize()
    check_status(st)

    xb, dyb, wb = bits_of(x), bits_of(dy), bits_of(wt)
    ox, ody, ow = O.quantize_mx(xb, w.splits, E), O.quantize_mx(dyb, w.splits, E), O.quantize_mx(wb, None, E)
    for key, ora, rows, cols, splits in (("x", ox, R, K, w.splits), ("dy", ody, R, N, w.splits),
                                         ("w", ow, E * N, K, None)):
        off, _, sb = O.split_scan(splits, E, rows, cols)
        assert_mx_equal(q[key], ora, int(off[-1]), int(sb[-1]))

    rng = np.random.default_rng(99)
    rows, grp = stratified_rows(rng, w.splits, PER_GROUP, N_SAMPLES)
    cn, ck = rng.integers(0, N, rows.size), rng.integers(0, K, rows.size)

    want = O.gemm_sample("fprop", ox, ow, w.splits, E, N, K, rows, cn)
    assert_sampled_groups_close(gather(y32, rows, cn), want, grp, "fprop fp32")
    got_b = gather(y, rows, cn)
    assert np.all(np.abs(got_b - want) <= np.abs(want) * 2.0 ** -8 + 1e-6), "fprop bf16"

    want = O.gemm_sample("dgrad", ody, ow, w.splits, E, N, K, rows, ck)
    assert_sampled_groups_close(gather(dx32, rows, ck), want, grp, "dgrad fp32")
    got_b = gather(dx, rows, ck)
    assert np.all(np.abs(got_b - want) <= np.abs(want) * 2.0 ** -8 + 1e-6), "dgrad bf16"

    # the wgrad: PER_GROUP outputs of every live expert plus N_SAMPLES more
    live = np.flatnonzero(w.splits > 0)
    g = np.concatenate([np.repeat(live, PER_GROUP), rng.choice(live, N_SAMPLES)])
    cn, ck = rng.integers(0, N, g.size), rng.integers(0, K, g.size)
    want = O.gemm_sample("wgrad", ody, ox, w.splits, E, N, K, cn, ck, g)
    assert_sampled_increments_close(gather(main, g, cn, ck), gather(main0, g, cn, ck), want, g,
                                    "wgrad (accumulate)")
    empty = np.flatnonzero(w.splits == 0)
    for e in empty:
        assert torch.equal(main[e], main0[e]), f"empty expert {e} changed"


@pytest.mark.parametrize("fc", [1, 2])
def test_moe_e64_zipf_layer(fc):
    run_layer("moe_e64_zipf", fc)


@pytest.mark.parametrize("fc", [1, 2])
def test_moe_e8_layer(fc):
    run_layer("moe_e8", fc)


def test_buffer_past_2_31_elements():
    """X [300544, 7168] bf16 (4.3 GB; R * K > 2^31, the last group's rows
    straddle element 2^31), dY [R, 256], three experts of width 256.  Both
    orientations of X and dY, fprop, dgrad (dX [R, 7168] fp32, 8.6 GB) and
    the k-grouped wgrad.  Groups 0 and 2 (1024 rows each) match the oracle on
    that group alone: codes and scale regions byte for byte, GEMMs within
    1e-5; the middle group's outputs are finite; the padding rows at the far
    end of the code buffers are never written."""
    K, N, G, R, pad = 7168, 256, 3, 300544, 128
    L = R - pad
    splits = np.array([1024, L - 2048, 1024], np.int32)
    assert R * K > 2 ** 31 and (L - 1024) * K < 2 ** 31 < L * K
    x = W.device_normal_bf16((R, K), 5, 1.0, 40, DEV)
    dy = W.device_normal_bf16((R, N), 5, 1.0, 41, DEV)
    wt = W.device_normal_bf16((G * N, K), 5, 0.02, 42, DEV)
    sp = torch.as_tensor(splits).to(DEV)
    st = status_dev()
    mx = mx_recipe()
    q = {k: gq.alloc_quantized(t.shape[0], t.shape[1], G, mx, DEV, fill=0xAB)
         for k, t in (("x", x), ("dy", dy), ("w", wt))}
    gq.gq_quantize(x, sp, G, mx, q["x"], st)
    gq.gq_quantize(dy, sp, G, mx, q["dy"], st)
    gq.gq_quantize(wt, None, G, mx, q["w"], st)
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

    off = np.concatenate([[0], np.cumsum(splits)])
    for g in (0, 2):
        a, b = int(off[g]), int(off[g + 1])
        one = np.array([b - a], np.int32)
        xg, dyg, wg = bits_of(x[a:b]), bits_of(dy[a:b]), bits_of(wt[g * N:(g + 1) * N])
        for key, bits, cols in (("x", xg, K), ("dy", dyg, N)):
            ora = O.quantize_mx(bits, one, 1)
            sb = O.split_scan(splits, G, R, cols)[2]
            nbytes = 512 * (cols // 128) * ((b - a + 127) // 128)
            assert np.array_equal(host(q[key].row_data[a:b]), ora.row_data), f"{key} row codes, group {g}"
            assert np.array_equal(host(q[key].col_data[a:b]), ora.col_data), f"{key} col codes, group {g}"
            for t, o in ((q[key].row_scale, ora.row_scale), (q[key].col_scale, ora.col_scale)):
                assert np.array_equal(host(t[int(sb[g]):int(sb[g]) + nbytes]), o[:nbytes]), f"{key} scales, group {g}"
        want = O.gemm_fprop(O.quantize_mx(xg, one, 1, colwise=False), O.quantize_mx(wg, None, 1, colwise=False),
                            one, 1, N, K)
        assert rel(host(y[a:b]), want) <= REL_TOL, f"fprop group {g}"
        want = O.gemm_dgrad(O.quantize_mx(dyg, one, 1, colwise=False), O.quantize_mx(wg, None, 1, rowwise=False),
                            one, 1, N, K)
        assert rel(host(dx[a:b]), want) <= REL_TOL, f"dgrad group {g}"
        want = O.gemm_wgrad(O.quantize_mx(dyg, one, 1, rowwise=False), O.quantize_mx(xg, one, 1, rowwise=False),
                            one, 1, N, K)
        assert rel(host(dw[g]), want[0]) <= REL_TOL, f"wgrad group {g}"
    mid = slice(int(off[1]), int(off[2]))
    assert bool(torch.isfinite(y[mid]).all()) and bool(torch.isfinite(dx[mid]).all())
    assert bool(torch.isfinite(dw[1]).all())
    for key in ("x", "dy"):
        assert bool((q[key].row_data[L:] == 0xAB).all()) and bool((q[key].col_data[L:] == 0xAB).all())
