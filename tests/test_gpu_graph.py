"""CUDA-graph capture of a whole grouped-linear step: fc1 and fc2 forward,
dgrad and wgrad (accumulating into fp32 main grads), every quantisation
included, with the split sizes on the device.  The step is captured once and
replayed with new split sizes and new inputs written into the same buffers;
each replay must give, bit for bit, what eager calls give on the same
inputs (TransformerEngine PR 3224: device split sizes, no host sync).  Both
the MXFP8 and the NVFP4 recipe."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_grouped_gemm_group_gb300 as gq  # noqa: E402
from _gpu_util import DEV, check_status  # noqa: E402

G, H, F, R = 4, 512, 256, 1024
SPLITS = [np.array([256, 0, 416, 288], np.int32), np.array([96, 512, 32, 320], np.int32)]


class Layer:
    def __init__(self, kind=gq.RECIPE_MXFP8_1X32):
        mx = gq.Recipe(kind, 1, 1, 0.0)
        self.mx = mx
        bf = torch.bfloat16
        self.inp = {"x1": torch.empty((R, H), dtype=bf, device=DEV), "x2": torch.empty((R, F), dtype=bf, device=DEV),
                    "dy1": torch.empty((R, F), dtype=bf, device=DEV), "dy2": torch.empty((R, H), dtype=bf, device=DEV),
                    "w1": torch.empty((G * F, H), dtype=bf, device=DEV),
                    "w2": torch.empty((G * H, F), dtype=bf, device=DEV)}
        shape = {"x1": (R, H), "x2": (R, F), "dy1": (R, F), "dy2": (R, H), "w1": (G * F, H), "w2": (G * H, F)}
        self.q = {k: gq.alloc_quantized(r, c, G, mx, DEV) for k, (r, c) in shape.items()}
        self.out = {"y1": torch.empty((R, F), dtype=bf, device=DEV), "y2": torch.empty((R, H), dtype=bf, device=DEV),
                    "dx2": torch.empty((R, F), dtype=bf, device=DEV), "dx1": torch.empty((R, H), dtype=bf, device=DEV),
                    "dw1": torch.empty((G, F, H), device=DEV), "dw2": torch.empty((G, H, F), device=DEV)}
        self.splits = torch.zeros(G, dtype=torch.int32, device=DEV)
        self.status = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.ws = torch.empty(gq.WGRAD_WORKSPACE_BYTES, dtype=torch.uint8, device=DEV)

    def load(self, seed, splits):
        gen = torch.Generator(device=DEV).manual_seed(seed)
        for k, t in self.inp.items():
            t.copy_(torch.randn(t.shape, generator=gen, device=DEV) * (0.02 if k.startswith("w") else 1.0))
        for k in ("dw1", "dw2"):
            self.out[k].copy_(torch.randn(self.out[k].shape, generator=gen, device=DEV) * 1e-3)
        for k in ("y1", "y2", "dx1", "dx2"):
            self.out[k].fill_(float("nan"))
        self.splits.copy_(torch.from_numpy(splits))

    def step(self):
        i, q, o, sp, st, mx = self.inp, self.q, self.out, self.splits, self.status, self.mx
        bf16 = gq.DTYPE_BF16
        gq.gq_quantize(i["x1"], sp, G, mx, q["x1"], st)
        gq.gq_quantize(i["w1"], None, G, mx, q["w1"], st)
        gq.gq_gemm_fprop(q["x1"], q["w1"], sp, G, F, H, o["y1"], bf16, st)
        gq.gq_quantize(i["x2"], sp, G, mx, q["x2"], st)
        gq.gq_quantize(i["w2"], None, G, mx, q["w2"], st)
        gq.gq_gemm_fprop(q["x2"], q["w2"], sp, G, H, F, o["y2"], bf16, st)
        gq.gq_quantize(i["dy2"], sp, G, mx, q["dy2"], st)
        gq.gq_gemm_dgrad(q["dy2"], q["w2"], sp, G, H, F, o["dx2"], bf16, st)
        gq.gq_gemm_wgrad(q["dy2"], q["x2"], sp, G, H, F, o["dw2"], True, st, workspace=self.ws)
        gq.gq_quantize(i["dy1"], sp, G, mx, q["dy1"], st)
        gq.gq_gemm_dgrad(q["dy1"], q["w1"], sp, G, F, H, o["dx1"], bf16, st)
        gq.gq_gemm_wgrad(q["dy1"], q["x1"], sp, G, F, H, o["dw1"], True, st, workspace=self.ws)

    def results(self):
        torch.cuda.synchronize()
        check_status(self.status)
        return {k: v.clone() for k, v in self.out.items()}


def _same_bits(a, b):
    ia = a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32)
    ib = b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32)
    return torch.equal(ia, ib)


@pytest.mark.parametrize("kind", [gq.RECIPE_MXFP8_1X32, gq.RECIPE_NVFP4_1X16])
def test_captured_step_replays_like_eager_calls(kind):
    layer = Layer(kind)
    layer.load(0, SPLITS[0])
    layer.step()                          # first calls on the device: set-up outside capture
    layer.results()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.step()

    for trial, splits in enumerate(SPLITS):
        layer.load(10 + trial, splits)
        graph.replay()
        got = layer.results()
        layer.load(10 + trial, splits)
        layer.step()
        want = layer.results()
        L = int(splits.sum())
        for k in want:
            g, w = (got[k][:L], want[k][:L]) if k in ("y1", "y2", "dx1", "dx2") else (got[k], want[k])
            assert _same_bits(g, w), f"replay {trial}: {k} differs from the eager result"
        # the live rows were written; the rows past the live total were not
        assert not torch.isnan(got["y1"][:L].float()).any()
        assert torch.isnan(got["y1"][L:].float()).all()


@pytest.mark.parametrize("kind", [gq.RECIPE_MXFP8_1X32, gq.RECIPE_NVFP4_1X16])
def test_weight_cache_reused_across_microbatches_in_a_graph(kind):
    """The weights are quantised once into a preallocated descriptor (the
    output reuse of TransformerEngine PR 3224's group_quantize) and that cache
    serves three microbatches, each with its own device split sizes and
    inputs: fprop, dgrad and a wgrad accumulating into one fp32 main grad.
    The whole sequence is captured once; replays give the eager bits."""
    rec = gq.Recipe(kind, 1, 1, 0.0)
    bf = torch.bfloat16
    nmb = 3
    w = torch.empty((G * F, H), dtype=bf, device=DEV)
    qw = gq.alloc_quantized(G * F, H, G, rec, DEV)
    xs = [torch.empty((R, H), dtype=bf, device=DEV) for _ in range(nmb)]
    dys = [torch.empty((R, F), dtype=bf, device=DEV) for _ in range(nmb)]
    sps = [torch.zeros(G, dtype=torch.int32, device=DEV) for _ in range(nmb)]
    qx = [gq.alloc_quantized(R, H, G, rec, DEV) for _ in range(nmb)]
    qd = [gq.alloc_quantized(R, F, G, rec, DEV) for _ in range(nmb)]
    ys = [torch.empty((R, F), dtype=bf, device=DEV) for _ in range(nmb)]
    dxs = [torch.empty((R, H), dtype=bf, device=DEV) for _ in range(nmb)]
    dw = torch.empty((G, F, H), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(gq.WGRAD_WORKSPACE_BYTES, dtype=torch.uint8, device=DEV)

    def load(seed):
        gen = torch.Generator(device=DEV).manual_seed(seed)
        w.copy_(torch.randn(w.shape, generator=gen, device=DEV) * 0.02)
        dw.copy_(torch.randn(dw.shape, generator=gen, device=DEV) * 1e-3)
        for m in range(nmb):
            xs[m].copy_(torch.randn(xs[m].shape, generator=gen, device=DEV))
            dys[m].copy_(torch.randn(dys[m].shape, generator=gen, device=DEV))
            sps[m].copy_(torch.from_numpy(SPLITS[(seed + m) % 2]))
            ys[m].fill_(float("nan"))
            dxs[m].fill_(float("nan"))

    def run():
        gq.gq_quantize(w, None, G, rec, qw, st)              # once per step: the weight cache
        for m in range(nmb):
            gq.gq_quantize(xs[m], sps[m], G, rec, qx[m], st)
            gq.gq_quantize(dys[m], sps[m], G, rec, qd[m], st)
            gq.gq_gemm_fprop(qx[m], qw, sps[m], G, F, H, ys[m], gq.DTYPE_BF16, st)
            gq.gq_gemm_dgrad(qd[m], qw, sps[m], G, F, H, dxs[m], gq.DTYPE_BF16, st)
            gq.gq_gemm_wgrad(qd[m], qx[m], sps[m], G, F, H, dw, True, st, workspace=ws)

    def snapshot():
        torch.cuda.synchronize()
        check_status(st)
        return [t.clone() for t in ys + dxs + [dw]]

    load(0)
    run()
    snapshot()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    for seed in (1, 2):
        load(seed)
        graph.replay()
        got = snapshot()
        load(seed)
        run()
        want = snapshot()
        for m in range(nmb):
            L = int(SPLITS[(seed + m) % 2].sum())
            assert _same_bits(got[m][:L], want[m][:L]), f"seed {seed}: y of microbatch {m}"
            assert _same_bits(got[nmb + m][:L], want[nmb + m][:L]), f"seed {seed}: dx of microbatch {m}"
        assert _same_bits(got[-1], want[-1]), f"seed {seed}: accumulated dW"


def test_captured_fc1_chain_moe_e64_zipf():
    """The moe_e64_zipf fc1 chain at full size (64 experts, 65536 Zipf-routed
    tokens + 1024 garbage rows, hidden 7168, width 2048): quantise X, W and
    dY, fprop, dgrad and a wgrad accumulating into the 3.8 GB fp32 main grad,
    captured once and replayed.  A replay gives the eager bits for the Zipf
    split sizes and for the same sizes in another expert order, written into
    the same device buffer between replays."""
    import workloads as W
    w = W.workload("moe_e64_zipf")
    E, R, L, H, F = w.num_groups, w.rows_cap, w.live_rows, w.hidden, w.ffn
    rec = gq.Recipe(gq.RECIPE_MXFP8_1X32, 1, 1, 0.0)
    bf = torch.bfloat16
    x = W.device_activation(w, H, 90, device=DEV)
    dy = W.device_activation(w, F, 91, device=DEV)
    wt = W.device_normal_bf16((E * F, H), w.seed, 0.02, 92, DEV)
    dw0 = W.device_normal_bf16((E, F, H), w.seed, 1e-3, 93, DEV).float()
    qx = gq.alloc_quantized(R, H, E, rec, DEV)
    qw = gq.alloc_quantized(E * F, H, E, rec, DEV)
    qd = gq.alloc_quantized(R, F, E, rec, DEV)
    y = torch.empty((R, F), dtype=bf, device=DEV)
    dx = torch.empty((R, H), dtype=bf, device=DEV)
    dw = torch.empty_like(dw0)
    sp = torch.zeros(E, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(gq.WGRAD_WORKSPACE_BYTES, dtype=torch.uint8, device=DEV)
    orders = [np.asarray(w.splits, np.int32),
              np.asarray(w.splits, np.int32)[np.random.default_rng(94).permutation(E)]]

    def chain():
        gq.gq_quantize(x, sp, E, rec, qx, st)
        gq.gq_quantize(wt, None, E, rec, qw, st)
        gq.gq_quantize(dy, sp, E, rec, qd, st)
        gq.gq_gemm_fprop(qx, qw, sp, E, F, H, y, gq.DTYPE_BF16, st)
        gq.gq_gemm_dgrad(qd, qw, sp, E, F, H, dx, gq.DTYPE_BF16, st)
        gq.gq_gemm_wgrad(qd, qx, sp, E, F, H, dw, True, st, workspace=ws)

    def reset(splits):
        sp.copy_(torch.from_numpy(splits))
        dw.copy_(dw0)
        y.fill_(float("nan"))
        dx.fill_(float("nan"))

    reset(orders[0])
    chain()                                   # first calls on the device: set-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chain()
    for trial, splits in enumerate(orders):
        reset(splits)
        graph.replay()
        torch.cuda.synchronize()
        check_status(st)
        got = (y.clone(), dx.clone(), dw.clone())
        reset(splits)
        chain()
        torch.cuda.synchronize()
        check_status(st)
        for name, g, e in zip(("y", "dx", "dw"), got, (y, dx, dw)):
            assert _same_bits(g, e), f"order {trial}: {name} differs from the eager result"
        assert not torch.isnan(got[0][:L].float()).any()
        assert torch.isnan(got[0][L:].float()).all()
