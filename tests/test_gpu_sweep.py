"""GPU parity at the token-count sweep's shapes: 32 uniform experts, hidden
4096 (the contraction of fprop and the output width of dgrad), expert width
1536, in the launch configuration the sweep times (MXFP8 row + column
quantisation, fprop / dgrad, the wgrad accumulating into an fp32 main grad
with the run-time tile order).

The sweep stands beside the single grouped weight buffer of TransformerEngine
PR 3224 (its summary: one contiguous weight tensor for all experts, split
uniformly); the expert width 1536 is that buffer's.

* T = 1K tokens (32 rows an expert: every group is one 32-row block): every
  quantised byte and every output against the oracle's full result.
* T = 256K tokens (8192 rows an expert): every quantised byte, and sampled
  outputs (64 in every expert plus 4096 over the layer).
GEMM outputs: per group within 1e-5 relative Frobenius error (fp32 outputs;
bf16 outputs within one bf16 rounding; the wgrad's increment with the fp32
rounding of the final add allowed per element).
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
                       assert_sampled_increments_close, check_status, gather, host, mx_recipe,
                       rel_err_per_group, status_dev, stratified_rows)

E, H, N = 32, 4096, 1536


def bits_of(t):
    return host(t.view(torch.int16)).view(np.uint16)


@pytest.fixture(scope="module")
def weights():
    """The experts' weights [E * N, H] (as the sweep draws them), quantised
    once on the GPU and by the oracle."""
    st = status_dev()
    mx = mx_recipe()
    w = W.device_normal_bf16((E * N, H), 6, 0.02, 1, DEV)
    qw = gq.alloc_quantized(E * N, H, E, mx, DEV, fill=0xAB)
    gq.gq_quantize(w, None, E, mx, qw, st)
    torch.cuda.synchronize()
    check_status(st)
    ow = O.quantize_mx(bits_of(w), None, E)
    _, _, sb = O.split_scan(None, E, E * N, H)
    assert_mx_equal(qw, ow, E * N, int(sb[-1]))
    return qw, ow


def run(T, weights):
    qw, ow = weights
    wl = W.workload("token_sweep", tokens=T)
    assert wl.num_groups == E and wl.hidden == H and wl.ffn == N
    st = status_dev()
    mx = mx_recipe()
    sp = torch.as_tensor(wl.splits).to(DEV)
    x = W.device_normal_bf16((T, H), wl.seed, 1.0, 2, DEV)
    dy = W.device_normal_bf16((T, N), wl.seed, 1.0, 3, DEV)
    qx = gq.alloc_quantized(T, H, E, mx, DEV, fill=0xAB)
    qd = gq.alloc_quantized(T, N, E, mx, DEV, fill=0xAB)
    gq.gq_quantize(x, sp, E, mx, qx, st)
    gq.gq_quantize(dy, sp, E, mx, qd, st)
    y = torch.empty((T, N), dtype=torch.bfloat16, device=DEV)
    dx = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    y32 = torch.empty((T, N), dtype=torch.float32, device=DEV)
    dx32 = torch.empty((T, H), dtype=torch.float32, device=DEV)
    main = W.device_normal_bf16((E, N, H), wl.seed, 1e-3, 4, DEV).float()
    main0 = main.clone()
    gq.gq_gemm_fprop(qx, qw, sp, E, N, H, y, gq.DTYPE_BF16, st)
    gq.gq_gemm_dgrad(qd, qw, sp, E, N, H, dx, gq.DTYPE_BF16, st)
    gq.gq_gemm_fprop(qx, qw, sp, E, N, H, y32, gq.DTYPE_F32, st)
    gq.gq_gemm_dgrad(qd, qw, sp, E, N, H, dx32, gq.DTYPE_F32, st)
    gq.gq_gemm_wgrad(qd, qx, sp, E, N, H, main, True, st)
    torch.cuda.synchronize()
    check_status(st)
    ox, od = O.quantize_mx(bits_of(x), wl.splits, E), O.quantize_mx(bits_of(dy), wl.splits, E)
    for q, o, cols in ((qx, ox, H), (qd, od, N)):
        _, _, sb = O.split_scan(wl.splits, E, T, cols)
        assert_mx_equal(q, o, T, int(sb[-1]))
    return wl, ox, od, (y, dx, y32, dx32, main, main0)


def test_sweep_1k_tokens_full(weights):
    """T = 1K: 32 experts of 32 tokens, every output against the oracle."""
    T = 1024
    wl, ox, od, (y, dx, y32, dx32, main, main0) = run(T, weights)
    _, ow = weights
    off = np.concatenate([[0], np.cumsum(wl.splits)])
    bnds = [(int(off[g]), int(off[g + 1])) for g in range(E)]
    want_y = O.gemm_fprop(ox, ow, wl.splits, E, N, H)
    want_dx = O.gemm_dgrad(od, ow, wl.splits, E, N, H)
    want_dw = O.gemm_wgrad(od, ox, wl.splits, E, N, H)
    for what, got, want in (("fprop", host(y32), want_y), ("dgrad", host(dx32), want_dx)):
        errs = rel_err_per_group(got, want, bnds)
        assert np.all(errs <= REL_TOL), f"{what}: worst group {int(np.argmax(errs))} at {errs.max():.3e}"
    for what, got, want in (("fprop bf16", host(y.float()), want_y), ("dgrad bf16", host(dx.float()), want_dx)):
        assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-6), what
    for e in range(E):                       # expert by expert: every element of its increment
        new, old = host(main[e]).astype(np.float64).ravel(), host(main0[e]).astype(np.float64).ravel()
        assert_sampled_increments_close(new, old, want_dw[e].ravel(), np.zeros(new.size, np.int64),
                                        f"wgrad (accumulate), expert {e}")


def test_sweep_256k_tokens_sampled(weights):
    """T = 256K: 32 experts of 8192 tokens, every quantised byte, sampled
    GEMM outputs per expert."""
    T = 256 * 1024
    wl, ox, od, (y, dx, y32, dx32, main, main0) = run(T, weights)
    _, ow = weights
    rng = np.random.default_rng(256)
    rows, grp = stratified_rows(rng, wl.splits, 64, 4096)
    cn, ck = rng.integers(0, N, rows.size), rng.integers(0, H, rows.size)
    want = O.gemm_sample("fprop", ox, ow, wl.splits, E, N, H, rows, cn)
    assert_sampled_groups_close(gather(y32, rows, cn), want, grp, "fprop fp32")
    got = gather(y, rows, cn)
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-6), "fprop bf16"
    want = O.gemm_sample("dgrad", od, ow, wl.splits, E, N, H, rows, ck)
    assert_sampled_groups_close(gather(dx32, rows, ck), want, grp, "dgrad fp32")
    got = gather(dx, rows, ck)
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-6), "dgrad bf16"
    g = np.concatenate([np.repeat(np.arange(E), 64), rng.integers(0, E, 4096)])
    cn, ck = rng.integers(0, N, g.size), rng.integers(0, H, g.size)
    want = O.gemm_sample("wgrad", od, ox, wl.splits, E, N, H, cn, ck, g)
    assert_sampled_increments_close(gather(main, g, cn, ck), gather(main0, g, cn, ck), want, g,
                                    "wgrad (accumulate)")
