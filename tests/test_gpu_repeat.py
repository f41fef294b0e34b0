"""Bitwise determinism over 10,000 repeated calls, for every entry point of
the path.

DeepGEMM issue 365's unit test calls its k-grouped wgrad 10,000 times on
fixed operands and counts the calls whose result differs (1749 of 10,000
blew up).  The same loop runs here on the quantiser, fprop, dgrad and the
wgrad, with the data of TransformerEngine issue 3484's reproducer: one group
of 512 live tokens in a 768-row buffer whose padding rows hold 3.0, hidden =
ffn = 1024, X and dY ~N(0,1), W ~N(0,1)/32 (seed 1), on MXFP8 and on NVFP4
operands.  (The k-grouped wgrad at config 2's shapes has its own 10,000-call
loop in test_gpu_gemm.py.)

Before every call each output is refilled with a canary (0xFF bytes, or NaN
for fp32 outputs), so a call that failed to write a live byte would differ;
every call's live outputs are compared with the first call's on the device
and the mismatching calls counted, as the page's loop does.
"""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_grouped_gemm_group_gb300 as gq  # noqa: E402
from _gpu_util import DEV, bf16_dev, check_status, mx_recipe, splits_dev, status_dev  # noqa: E402

CALLS = 10000
L, R, H = 512, 768, 1024


def nv_recipe():
    return gq.Recipe(gq.RECIPE_NVFP4_1X16, 1, 1, 0.0)


@pytest.fixture(scope="module")
def data():
    w = W.workload("padded_single_group", pad_kind="fill3")
    assert (w.live_rows, w.rows_cap, w.hidden) == (L, R, H)
    x = bf16_dev(w.activation(H, 0))
    dy = bf16_dev(w.activation(H, 1))
    wt = bf16_dev(W.normal_bf16((H, H), 1, scale=1 / 32, stream=2))
    return x, dy, wt, splits_dev(w.splits)


def live_views(q: gq.GroupedTensor, nv: bool):
    """The bytes a quantisation of the 512 live rows writes: codes of the live
    rows and the group's scale region (and the NVFP4 amax)."""
    atoms = 4 * (H // (64 if nv else 128))          # 4 row tiles of 128
    v = [q.row_data[:L], q.row_scale[:512 * atoms], q.col_scale[:512 * atoms]]
    v.append(q.col_data[:, :L // 2] if nv else q.col_data[:L])
    if nv:
        v.append(q.amax[:1])
    return v


def refill(q: gq.GroupedTensor):
    for t in (q.row_data, q.row_scale, q.col_data, q.col_scale, q.amax):
        if t is not None:
            t.view(torch.uint8).fill_(0xFF)


@pytest.mark.parametrize("recipe", ["mx", "nvfp4"])
def test_quantize_10000_calls_bitwise(data, recipe):
    x, _, _, sp = data
    nv = recipe == "nvfp4"
    rec = nv_recipe() if nv else mx_recipe()
    st = status_dev()
    q = gq.alloc_quantized(R, H, 1, rec, DEV, fill=0xAB)
    gq.gq_quantize(x, sp, 1, rec, q, st)
    ref = [t.clone() for t in live_views(q, nv)]
    bad = torch.zeros((), dtype=torch.int64, device=DEV)
    for _ in range(CALLS):
        refill(q)
        gq.gq_quantize(x, sp, 1, rec, q, st)
        diff = torch.zeros((), dtype=torch.bool, device=DEV)
        for t, r in zip(live_views(q, nv), ref):
            diff |= (t != r).any()
        bad += diff
    check_status(st)
    assert int(bad.item()) == 0, f"{int(bad.item())} of {CALLS} quantisations differ"


@pytest.mark.parametrize("recipe", ["mx", "nvfp4"])
@pytest.mark.parametrize("kind", ["fprop", "dgrad", "wgrad"])
def test_gemm_10000_calls_bitwise(data, recipe, kind):
    x, dy, wt, sp = data
    nv = recipe == "nvfp4"
    rec = nv_recipe() if nv else mx_recipe()
    st = status_dev()
    qx, qd, qw = (gq.alloc_quantized(t.shape[0], H, 1, rec, DEV, fill=0xAB) for t in (x, dy, wt))
    gq.gq_quantize(x, sp, 1, rec, qx, st)
    gq.gq_quantize(dy, sp, 1, rec, qd, st)
    gq.gq_quantize(wt, None, 1, rec, qw, st)
    ws = torch.empty(gq.WGRAD_WORKSPACE_BYTES, dtype=torch.uint8, device=DEV)
    if kind == "wgrad":
        out = torch.empty((1, H, H), device=DEV)

        def call():
            gq.gq_gemm_wgrad(qd, qx, sp, 1, H, H, out, False, st, workspace=ws)

        def live():
            return out
    else:
        out = torch.empty((R, H), device=DEV)
        a = qx if kind == "fprop" else qd
        fn = gq.gq_gemm_fprop if kind == "fprop" else gq.gq_gemm_dgrad

        def call():
            fn(a, qw, sp, 1, H, H, out, gq.DTYPE_F32, st)

        def live():
            return out[:L]
    call()
    ref = live().clone()
    check_status(st)
    assert bool(torch.isfinite(ref).all())
    bad = torch.zeros((), dtype=torch.int64, device=DEV)
    for _ in range(CALLS):
        out.fill_(float("nan"))
        call()
        bad += (live() != ref).any()
    check_status(st)
    assert int(bad.item()) == 0, f"{int(bad.item())} of {CALLS} {kind} calls differ"
    if kind != "wgrad":
        assert bool(torch.isnan(out[L:]).all()), "rows past the live total were written"
