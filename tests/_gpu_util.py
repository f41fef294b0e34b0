"""Helpers shared by the GPU parity tests: device copies of seeded inputs,
calls through the C ABI (via the Python binding), and comparisons against the
oracle's outputs."""
from __future__ import annotations

import numpy as np
import torch

import moe_grouped_gemm_group_gb300 as gq
import oracle as O

DEV = "cuda:0"
REL_TOL = 1e-5       # per-group relative Frobenius error of the GEMMs


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bits (host) -> bf16 CUDA tensor."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(DEV).view(torch.bfloat16)


def splits_dev(splits):
    return None if splits is None else torch.as_tensor(np.asarray(splits, np.int32)).to(DEV)


def status_dev(value: int = 0) -> torch.Tensor:
    return torch.full((1,), value, dtype=torch.int32, device=DEV)


def mx_recipe(rowwise=True, colwise=True) -> gq.Recipe:
    return gq.Recipe(gq.RECIPE_MXFP8_1X32, int(rowwise), int(colwise), 0.0)


def ch_recipe(zero_scale=1e-30) -> gq.Recipe:
    return gq.Recipe(gq.RECIPE_CHANNEL128_F32, 0, 1, float(zero_scale))


def quantize(bits, splits, G, recipe, fill=0xAB, status=None):
    """GPU quantisation through the C ABI; returns (GroupedTensor, status tensor)."""
    x = bf16_dev(bits) if isinstance(bits, np.ndarray) else bits
    R, Cc = x.shape
    out = gq.alloc_quantized(R, Cc, G, recipe, DEV, fill=fill)
    st = status_dev() if status is None else status
    gq.gq_quantize(x, splits_dev(splits), G, recipe, out, st)
    return out, st


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def check_status(st: torch.Tensor, want: int = 0):
    got = int(st.item())
    assert got == want, f"device status {got} ({gq.STATUS.get(got)}), want {want}"


def assert_mx_equal(gpu: gq.GroupedTensor, ora: O.MXQuantized, live_rows: int, scale_bytes: int,
                    fill=0xAB):
    """Codes of live rows and the grouped scale regions bit-exact; code rows
    past the live total and scale bytes past the grouped extent untouched."""
    for orient in ("row", "col"):
        gd = getattr(gpu, f"{orient}_data")
        if gd is None:
            continue
        d = host(gd)
        s = host(getattr(gpu, f"{orient}_scale"))
        od, os_ = getattr(ora, f"{orient}_data"), getattr(ora, f"{orient}_scale")
        bad = np.flatnonzero((d[:live_rows] != od[:live_rows]).ravel())
        assert bad.size == 0, (f"{orient} codes differ at {bad.size} places, first "
                               f"{np.unravel_index(bad[0], d[:live_rows].shape)}: "
                               f"gpu {d[:live_rows].ravel()[bad[0]]:#x} oracle "
                               f"{od[:live_rows].ravel()[bad[0]]:#x}")
        assert np.all(d[live_rows:] == fill), f"{orient} codes written past the live rows"
        bad = np.flatnonzero(s[:scale_bytes] != os_[:scale_bytes])
        assert bad.size == 0, (f"{orient} scales differ at {bad.size} bytes, first {bad[0]}: "
                               f"gpu {s[bad[0]]} oracle {os_[bad[0]]}")
        assert np.all(s[scale_bytes:] == fill), f"{orient} scales written past the grouped extent"


def rel_err_per_group(got: np.ndarray, want: np.ndarray, bounds):
    """Relative Frobenius error of each row range [a, b) of got vs want."""
    errs = []
    for a, b in bounds:
        w = want[a:b].astype(np.float64)
        g = got[a:b].astype(np.float64)
        nw = np.linalg.norm(w)
        if nw == 0:
            errs.append(0.0 if np.all(g == 0) else np.inf)
        else:
            errs.append(np.linalg.norm(g - w) / nw)
    return np.array(errs)


# --------------------------------------------------------------------------- #
# sampled full-size checks, held to the per-group bar                          #
# --------------------------------------------------------------------------- #

def gather(t: torch.Tensor, *idx) -> np.ndarray:
    """t[idx...] as fp64 on the host (idx: numpy index arrays)."""
    return host(t[tuple(torch.as_tensor(np.asarray(i)).to(t.device) for i in idx)].float()).astype(np.float64)


def stratified_rows(rng, splits, per_group: int, extra: int):
    """Token rows to sample: `per_group` rows drawn in every non-empty group
    (so a 32-row expert is checked as closely as the largest) plus `extra`
    drawn uniformly over all live rows; returns (rows, group of each row)."""
    splits = np.asarray(splits, np.int64)
    off = np.concatenate([[0], np.cumsum(splits)])
    rows, grp = [], []
    for g in np.flatnonzero(splits > 0):
        rows.append(rng.integers(off[g], off[g + 1], per_group))
        grp.append(np.full(per_group, g))
    if extra:
        r = rng.integers(0, off[-1], extra)
        rows.append(r)
        grp.append(np.searchsorted(off, r, side="right") - 1)
    return np.concatenate(rows), np.concatenate(grp)


def assert_sampled_groups_close(got, want, grp, what: str, tol: float = REL_TOL):
    """Per group: the relative Frobenius error of the sampled outputs within
    `tol`; a group whose sampled oracle values are all 0 must give exact 0."""
    worst = (0.0, -1)
    for g in np.unique(grp):
        m = grp == g
        nw = np.linalg.norm(want[m])
        if nw == 0:
            assert np.all(got[m] == 0), f"{what}: group {g} should be exactly 0"
            continue
        e = np.linalg.norm(got[m] - want[m]) / nw
        worst = max(worst, (e, int(g)))
    assert worst[0] <= tol, f"{what}: group {worst[1]} sampled relative error {worst[0]:.3e} > {tol:g}"
    return worst[0]


def assert_sampled_increments_close(new, old, want, grp, what: str, tol: float = REL_TOL):
    """Accumulating wgrad, per group: the increment new - old (exact in fp64
    from the two fp32 values) against the oracle's contraction.  The kernel
    computes new = fl32(old + acc), so |(new - old) - acc| <= 2^-24 |new|
    element by element; that rounding is allowed per element and what is
    left must meet the per-group bar: sum_e max(0, |new - old - want| -
    2^-24 |new|)^2 <= tol^2 sum_e want^2."""
    inc = new - old
    slack = 2.0 ** -24 * np.abs(new)
    resid = np.maximum(np.abs(inc - want) - slack, 0.0)
    worst = (0.0, -1)
    for g in np.unique(grp):
        m = grp == g
        nw = np.linalg.norm(want[m])
        if nw == 0:
            assert np.all(resid[m] == 0), f"{what}: group {g} increment should be exactly 0"
            continue
        e = np.linalg.norm(resid[m]) / nw
        worst = max(worst, (e, int(g)))
    assert worst[0] <= tol, f"{what}: group {worst[1]} sampled relative error {worst[0]:.3e} > {tol:g}"
    return worst[0]
