"""The device-side failure path, run without a fault: gq_check_wait_limit
waits on an mbarrier that nothing arrives on, with the same bounded wait as
every kernel of the library.  The wait gives up after its limit (2 s of
%globaltimer), GQ_ERR_TIMEOUT lands in the status word, the second warp
leaves on the shared abort flag, and the CUDA context stays usable: the next
quantisation and GEMM on the same stream run and match the oracle."""
import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_grouped_gemm_group_gb300 as gq  # noqa: E402
from _gpu_util import (DEV, REL_TOL, check_status, host, mx_recipe, quantize, rel_err_per_group,  # noqa: E402
                       splits_dev, status_dev)

LIMIT_NS = 2_000_000_000


def test_wait_gives_up_with_timeout_status_and_context_survives():
    status = status_dev()
    report = torch.full((4,), -1, dtype=torch.int64, device=DEV)
    gq.gq_check_wait_limit(status, report)
    torch.cuda.synchronize()
    check_status(status, -6)                                 # GQ_ERR_TIMEOUT
    waited0, done0, waited1, done1 = (int(v) for v in host(report))
    assert done0 == 0 and done1 == 0                         # the phase never completed
    assert max(waited0, waited1) > LIMIT_NS                  # one warp ran out the limit ...
    assert min(waited0, waited1) > LIMIT_NS // 2             # ... the other left on the abort flag
    assert max(waited0, waited1) < 15 * LIMIT_NS

    # the context still runs work: quantise and fprop on the same stream
    G, N, K = 2, 256, 256
    splits = np.array([96, 160], np.int32)
    x = W.normal_bf16((256, K), 61)
    w = W.normal_bf16((G * N, K), 62, scale=0.02)
    st = status_dev()
    xq, _ = quantize(x, splits, G, mx_recipe(True, False), status=st)
    wq, _ = quantize(w, None, G, mx_recipe(True, False), status=st)
    y = torch.full((256, N), float("nan"), dtype=torch.float32, device=DEV)
    gq.gq_gemm_fprop(xq, wq, splits_dev(splits), G, N, K, y, gq.DTYPE_F32, st)
    check_status(st)
    ox = O.quantize_mx(x, splits, G, colwise=False)
    assert np.array_equal(host(xq.row_data), ox.row_data)
    want = O.gemm_fprop(ox, O.quantize_mx(w, None, G, colwise=False), splits, G, N, K)
    assert max(rel_err_per_group(host(y), want, [(0, 96), (96, 256)])) <= REL_TOL


def test_nonzero_status_makes_it_a_noop():
    status = status_dev(-3)
    report = torch.full((4,), -1, dtype=torch.int64, device=DEV)
    gq.gq_check_wait_limit(status, report)
    torch.cuda.synchronize()
    check_status(status, -3)
    assert np.all(host(report) == -1)
