"""Seeded synthetic inputs for the grouped FP8 quantizer and the grouped GEMMs.

This module holds random draws, the bf16 rounding of those draws and the
split-size tables of the five MoE workloads; it holds none of the method's
arithmetic (no scaling, no FP8 encoding, no contraction). Both the CUDA path's
tests and benchmark and the CPU oracle's tests take their inputs from here, so
the two sides see the same bytes.

bf16 tensors are carried as ``numpy.uint16`` bit patterns (row-major).

Workloads (named after the bug reports they mirror):

* ``padded_single_group``: one group, hidden = ffn = 1024, 512 live rows in a
  768-row buffer whose tail is padding (TransformerEngine issue 3484,
  "Steps/Code to reproduce bug").
* ``kgrouped_zero_channel``: four experts with 256/128/128/256 tokens,
  n = H = 2048, gradient ~N(0,1)*1e-7 with channel 0 zeroed in both 128-token
  experts, activation ~N(0,1)*0.4 (DeepGEMM issue 365, the unit test).
* ``moe_e8``: E=8, hidden 4096, ffn 2048, 16384 routed tokens, Dirichlet
  splits in units of 128 with one expert empty, 1024 garbage padding rows.
* ``moe_e64_zipf``: E=64, hidden 7168, ffn 2048, 65536 tokens, Zipf(1.1)
  splits in units of 32 with empty and 32-token experts, 1024 garbage rows.
* ``single_grouped_weight``: 128 same-shape experts of 4096 x 1536 in one
  buffer (uniform split), plus a token-count sweep at hidden 4096 over 32
  experts (TransformerEngine PR 3224, single grouped weight).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "f32_to_bf16_bits", "bf16_bits_to_f32", "normal_bf16", "uniform_bf16",
    "fill_bf16", "dirichlet_splits", "zipf_splits", "Workload", "workload",
    "WORKLOADS", "SWEEP_TOKENS",
]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits.

    Only used to make bf16 inputs from float32 draws (finite values only).
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def normal_bf16(shape, seed: int, scale: float = 1.0, stream: int = 0) -> np.ndarray:
    """N(0, scale^2) draws rounded to bf16; PCG64 seeded by (seed, stream)."""
    rng = np.random.Generator(np.random.PCG64([seed, stream]))
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    chunk = 1 << 24
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        v = rng.standard_normal(e - s, dtype=np.float32)
        if scale != 1.0:
            v *= np.float32(scale)
        out[s:e] = f32_to_bf16_bits(v)
    return out.reshape(shape)


def uniform_bf16(shape, seed: int, lo: float, hi: float, stream: int = 0) -> np.ndarray:
    """Uniform[lo, hi) draws rounded to bf16 (the garbage tail of a padded buffer)."""
    rng = np.random.Generator(np.random.PCG64([seed, stream]))
    v = rng.uniform(lo, hi, size=int(np.prod(shape))).astype(np.float32)
    return f32_to_bf16_bits(v).reshape(shape)


def fill_bf16(shape, value: float) -> np.ndarray:
    """A constant bf16 buffer (e.g. a 0.0 / 3.0 / NaN padding fill)."""
    return np.full(shape, f32_to_bf16_bits(np.array([value], np.float32))[0]
                   if np.isfinite(value) else np.uint16(0x7FC0), dtype=np.uint16)


def _largest_remainder(weights: np.ndarray, units: int) -> np.ndarray:
    """Integer apportionment of ``units`` proportional to ``weights``."""
    w = np.asarray(weights, dtype=np.float64)
    quota = w / w.sum() * units
    base = np.floor(quota).astype(np.int64)
    short = units - int(base.sum())
    order = np.argsort(-(quota - base), kind="stable")
    base[order[:short]] += 1
    return base


def dirichlet_splits(num_groups: int, total: int, unit: int, seed: int,
                     empty: tuple[int, ...] = ()) -> np.ndarray:
    """Dirichlet(1,...,1) token shares rounded to multiples of ``unit``.

    Experts listed in ``empty`` get zero tokens; the other shares are
    renormalised and apportioned by largest remainder in units of ``unit``.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    p = rng.dirichlet(np.ones(num_groups))
    p[list(empty)] = 0.0
    units = _largest_remainder(p, total // unit)
    return (units * unit).astype(np.int32)


def zipf_splits(num_groups: int, total: int, unit: int, s: float, seed: int,
                n_empty: int = 3, n_min: int = 3) -> np.ndarray:
    """Zipf(s)-skewed token counts in multiples of ``unit``.

    Rank r gets a share proportional to r**-s, apportioned by largest
    remainder.  The ``n_empty`` lowest-ranked experts are then set to 0 tokens
    and the next ``n_min`` to one unit; the difference is absorbed by rank 1.
    Finally the expert order is permuted (seeded).
    """
    r = np.arange(1, num_groups + 1, dtype=np.float64)
    units = _largest_remainder(r ** -s, total // unit)
    units[num_groups - n_empty:] = 0
    units[num_groups - n_empty - n_min:num_groups - n_empty] = 1
    units[0] += total // unit - int(units.sum())
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(num_groups)
    return (units[perm] * unit).astype(np.int32)


SWEEP_TOKENS = tuple(1024 << i for i in range(9))  # 1K .. 256K


@dataclass
class Workload:
    """Shapes and split sizes of one synthetic MoE workload.

    ``rows_cap`` is the buffer row count R (>= sum(splits)); rows past the
    live total are padding.  ``hidden``/``ffn`` are the fc1 K and N.
    """
    name: str
    splits: np.ndarray
    rows_cap: int
    hidden: int
    ffn: int
    seed: int
    pad_kind: str = "none"          # none | fill3 | fill0 | uniform4
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def num_groups(self) -> int:
        return int(len(self.splits))

    @property
    def live_rows(self) -> int:
        return int(np.sum(self.splits))

    def padding(self, cols: int, stream: int) -> np.ndarray:
        """The padding rows [live_rows, rows_cap) of a bf16 buffer."""
        shape = (self.rows_cap - self.live_rows, cols)
        if self.pad_kind == "fill3":
            return fill_bf16(shape, 3.0)
        if self.pad_kind == "fill0" or self.pad_kind == "none":
            return fill_bf16(shape, 0.0)
        if self.pad_kind == "uniform4":
            return uniform_bf16(shape, self.seed, -4.0, 4.0, stream=1000 + stream)
        raise ValueError(self.pad_kind)

    def activation(self, cols: int, stream: int, scale: float = 1.0) -> np.ndarray:
        """A [rows_cap, cols] bf16 buffer: N(0, scale^2) live rows + padding."""
        live = normal_bf16((self.live_rows, cols), self.seed, scale, stream)
        return np.concatenate([live, self.padding(cols, stream)], axis=0)


def workload(name: str, **kw) -> Workload:
    """Build one of the named workloads (see the module docstring)."""
    if name == "padded_single_group":
        pad = kw.get("pad_kind", "fill3")
        rows = kw.get("rows_cap", 768)
        return Workload(name, np.array([512], np.int32), rows, 1024, 1024, seed=1,
                        pad_kind=pad)
    if name == "kgrouped_zero_channel":
        return Workload(name, np.array([256, 128, 128, 256], np.int32), 768, 2048, 2048,
                        seed=0, pad_kind="none")
    if name == "moe_e8":
        splits = dirichlet_splits(8, 16384, 128, seed=3, empty=(5,))
        return Workload(name, splits, 16384 + 1024, 4096, 2048, seed=3, pad_kind="uniform4")
    if name == "moe_e64_zipf":
        splits = zipf_splits(64, 65536, 32, 1.1, seed=4)
        return Workload(name, splits, 65536 + 1024, 7168, 2048, seed=4, pad_kind="uniform4")
    if name == "single_grouped_weight":
        return Workload(name, np.full(128, 4096, np.int32), 128 * 4096, 1536, 0, seed=5)
    if name == "token_sweep":
        t = int(kw["tokens"])
        return Workload(name, np.full(32, t // 32, np.int32), t, 4096, 1536, seed=6)
    raise KeyError(name)


WORKLOADS = ("padded_single_group", "kgrouped_zero_channel", "moe_e8", "moe_e64_zipf",
             "single_grouped_weight")


def kgrouped_zero_channel_operands(w: Workload):
    """The gradient / activation pair of the k-grouped wgrad repro.

    Gradient ~N(0,1)*1e-7 [768, 2048] with channel 0 zeroed for both
    128-token experts; activation ~N(0,1)*0.4 [768, 2048].
    """
    dy = normal_bf16((w.rows_cap, w.hidden), w.seed, 1e-7, stream=0)
    x = normal_bf16((w.rows_cap, w.ffn), w.seed, 0.4, stream=1)
    off = 0
    for m in w.splits:
        if m == 128:
            dy[off:off + m, 0] = 0
        off += int(m)
    return dy, x


def device_normal_bf16(shape, seed: int, scale: float = 1.0, stream: int = 0, device="cuda"):
    """N(0, scale^2) bf16 tensor drawn on the device (torch Philox generator
    seeded by (seed, stream)); used for full-size buffers that would take too
    long to draw on the host.  Returns a torch tensor."""
    import torch
    g = torch.Generator(device=device).manual_seed(int(seed) * 1000003 + int(stream))
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, float(scale), generator=g)
    return t.to(torch.bfloat16)


def device_uniform_bf16(shape, seed: int, lo: float, hi: float, stream: int = 0, device="cuda"):
    """Uniform[lo, hi) bf16 tensor drawn on the device (padding garbage)."""
    import torch
    g = torch.Generator(device=device).manual_seed(int(seed) * 1000003 + 7919 + int(stream))
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.uniform_(float(lo), float(hi), generator=g)
    return t.to(torch.bfloat16)


def device_activation(w: Workload, cols: int, stream: int, scale: float = 1.0, device="cuda"):
    """Device [rows_cap, cols] bf16 buffer: N(0, scale^2) live rows followed by
    the workload's padding rows (uniform[-4, 4] garbage or a constant fill)."""
    import torch
    out = torch.empty((w.rows_cap, cols), dtype=torch.bfloat16, device=device)
    L = w.live_rows
    out[:L] = device_normal_bf16((L, cols), w.seed, scale, stream, device)
    if w.rows_cap > L:
        if w.pad_kind == "uniform4":
            out[L:] = device_uniform_bf16((w.rows_cap - L, cols), w.seed, -4.0, 4.0, stream, device)
        else:
            out[L:] = 3.0 if w.pad_kind == "fill3" else 0.0
    return out
