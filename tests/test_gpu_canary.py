"""Bytes past the live total can never reach a result.

TransformerEngine issue 3484 ('Expected behavior'): whatever the buffer holds
past sum(split_sizes) must not change any result.  The padding of the bf16
inputs is covered elsewhere (fills 0, 3.0, garbage, NaN); here the canary is
in the quantised buffers themselves.  Before quantising, every code and
scale byte is pre-filled with a NaN pattern: 0xFF and 0x7F for MXFP8 (both
e4m3 NaNs; 0xFF is also the E8M0 NaN scale), 0xFF and 0x7F for NVFP4 (E4M3
NaN scales; the E2M1 codes -6 / +6).  fprop and dgrad load the last 128-row
tile of a group whose rows run past the group into those bytes, the wgrad's
last k-tile of a ragged group holds them, and an NVFP4 64-row block can be
half past its group.  The GEMM results must be bitwise those of a run whose
buffers were pre-filled with a finite byte (0x00), and the output rows past
the live total must stay untouched.
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

# ragged groups: 32-row and empty ones, a last tile of 96 live rows, and the
# live total ending 32 rows into a 128-row tile; 64-row NVFP4 blocks half
# live at the ends of the 96- and 160-row groups
SPLITS = np.array([96, 0, 160, 32, 224, 0, 32], np.int32)
G, R, N, K = len(SPLITS), 768, 256, 512
L = int(SPLITS.sum())


def recipe(name):
    if name == "mx":
        return mx_recipe()
    return gq.Recipe(gq.RECIPE_NVFP4_1X16, 1, 1, 0.0)


def run(name, fill):
    """Quantise into buffers pre-filled with `fill`, then fprop, dgrad (fp32
    outputs pre-filled with a sentinel) and the wgrad, without and with
    accumulate; returns the outputs."""
    rec = recipe(name)
    st = status_dev()
    sp = splits_dev(SPLITS)
    x = bf16_dev(np.concatenate([W.normal_bf16((L, K), 11), W.uniform_bf16((R - L, K), 12, -4, 4)]))
    dy = bf16_dev(np.concatenate([W.normal_bf16((L, N), 13), W.uniform_bf16((R - L, N), 14, -4, 4)]))
    wt = bf16_dev(W.normal_bf16((G * N, K), 15, scale=0.02))
    q = {}
    for key, t, s in (("x", x, sp), ("dy", dy, sp), ("w", wt, None)):
        q[key] = gq.alloc_quantized(t.shape[0], t.shape[1], G, rec, DEV, fill=fill)
        gq.gq_quantize(t, s, G, rec, q[key], st)
    y = torch.full((R, N), 7.0, device=DEV)
    dx = torch.full((R, K), 7.0, device=DEV)
    dw = torch.full((G, N, K), float("nan"), device=DEV)
    main = torch.full((G, N, K), 0.5, device=DEV)
    gq.gq_gemm_fprop(q["x"], q["w"], sp, G, N, K, y, gq.DTYPE_F32, st)
    gq.gq_gemm_dgrad(q["dy"], q["w"], sp, G, N, K, dx, gq.DTYPE_F32, st)
    gq.gq_gemm_wgrad(q["dy"], q["x"], sp, G, N, K, dw, False, st)
    gq.gq_gemm_wgrad(q["dy"], q["x"], sp, G, N, K, main, True, st)
    torch.cuda.synchronize()
    check_status(st)
    return {"fprop": y, "dgrad": dx, "wgrad": dw, "wgrad accumulate": main}


@pytest.mark.parametrize("name", ["mx", "nvfp4"])
def test_nan_filled_quantised_buffers_change_nothing(name):
    base = run(name, 0x00)
    for what, t in base.items():
        assert bool(torch.isfinite(t).all()), f"{what}: non-finite with a finite fill"
    assert bool((base["fprop"][L:] == 7.0).all()) and bool((base["dgrad"][L:] == 7.0).all())
    for e in np.flatnonzero(SPLITS == 0):
        assert bool((base["wgrad"][e] == 0).all()) and bool((base["wgrad accumulate"][e] == 0.5).all())
    for fill in (0xFF, 0x7F):
        got = run(name, fill)
        for what, t in got.items():
            assert torch.equal(t, base[what]), f"{what} changed with quantised buffers pre-filled {fill:#x}"
