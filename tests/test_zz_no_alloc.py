"""gq_gemm_wgrad_noalloc: the k-grouped wgrad for callers that cannot hand the
library a workspace (no device allocator of their own, or no allocation
allowed on this path).  It must give what gq_gemm_wgrad gives with a
caller-owned workspace, call after call, even though every call reuses the
same library-owned array.

This file is collected last on purpose: the entry point keeps state inside
the library for the life of the process, so it runs after every other test
(and it must also pass alone, in a fresh process)."""
import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_grouped_gemm_group_gb300 as gq  # noqa: E402
from _gpu_util import DEV, REL_TOL, check_status, host, mx_recipe, quantize, splits_dev, status_dev  # noqa: E402


def _operands(splits, N, K, pad):
    L = int(np.sum(splits))
    dy = np.concatenate([W.normal_bf16((L, N), 41), W.uniform_bf16((pad, N), 42, -4, 4)])
    x = np.concatenate([W.normal_bf16((L, K), 43), W.uniform_bf16((pad, K), 44, -4, 4)])
    return dy, x


@pytest.mark.parametrize("K", [512, 384])
def test_noalloc_wgrad_matches_workspace_wgrad_twice(K):
    # skewed splits: long and short contractions, empty groups
    splits = np.array([32, 0, 1088, 96, 0, 32, 320, 64], np.int32)
    G, N = len(splits), 256
    dy, x = _operands(splits, N, K, 64)
    st = status_dev()
    dyq, _ = quantize(dy, splits, G, mx_recipe(False, True), status=st)
    xq, _ = quantize(x, splits, G, mx_recipe(False, True), status=st)
    sp = splits_dev(splits)
    init = torch.from_numpy(W.bf16_bits_to_f32(W.normal_bf16((G, N, K), 45))).to(DEV)

    ws = torch.empty(gq.WGRAD_WORKSPACE_BYTES, dtype=torch.uint8, device=DEV)
    want = init.clone()
    gq.gq_gemm_wgrad(dyq, xq, sp, G, N, K, want, True, st, workspace=ws)
    check_status(st)
    want_h = host(want)

    for _ in range(2):                       # the shared array must be reset by every call
        got = init.clone()
        gq.gq_gemm_wgrad_noalloc(dyq, xq, sp, G, N, K, got, True, st)
        check_status(st)
        got_h = host(got)
        err = np.linalg.norm((got_h - want_h).astype(np.float64)) / np.linalg.norm(want_h.astype(np.float64))
        assert err <= REL_TOL
        assert np.array_equal(got_h.view(np.uint32), want_h.view(np.uint32))

    # and both agree with the oracle
    ora = O.gemm_wgrad(O.quantize_mx(dy, splits, G, rowwise=False), O.quantize_mx(x, splits, G, rowwise=False),
                       splits, G, N, K, True, host(init).astype(np.float64))
    for g in range(G):
        e = np.linalg.norm(got_h[g].astype(np.float64) - ora[g]) / np.linalg.norm(ora[g])
        assert e <= REL_TOL, f"group {g}: rel err {e}"


def test_noalloc_wgrad_refuses_too_many_tiles():
    # 1024 groups x (2^17 / 128) x (2^19 / 256) = 2^31 tiles: refused before
    # any operand is looked at or anything is launched
    rc = gq.load().gq_gemm_wgrad_noalloc(None, None, None, 1024, 1 << 17, 1 << 19, None, 1, None, None)
    assert rc == -1
