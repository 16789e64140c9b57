"""Comparison helpers shared by the GPU parity tests (tolerances of the problem statement)."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

# fp32 path: max |dO| <= 1e-4.  bf16 path: max |dO| <= 1.5e-2, mean |dO| <= 2e-3,
# |dLSE| <= 1e-3, gradients relative-L2 <= 2e-2 (each of dQ, dK, dV separately).
TOL_F32_O = 1e-4
TOL_F32_LSE = 1e-4
TOL_BF16_O_MAX = 1.5e-2
TOL_BF16_O_MEAN = 2e-3
TOL_BF16_LSE = 1e-3
TOL_GRAD_REL_L2 = 2e-2
TOL_F32_GRAD_REL_L2 = 1e-4


def f64(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float64).numpy()


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bfloat16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def check_fwd(o, lse, o_ref, lse_ref, dtype, what="", check_mean=True):
    """Element-wise comparison of O and LSE against the oracle; returns the statistics.
    The mean bound is a property of a whole output tensor; sampled rows pass
    check_mean=False and are held to the max bounds only."""
    o, lse, o_ref, lse_ref = f64(o), f64(lse), f64(o_ref), f64(lse_ref)
    assert o.shape == o_ref.shape and lse.shape == lse_ref.shape
    assert np.isfinite(o).all() and np.isfinite(lse).all(), f"non-finite output {what}"
    err = np.abs(o - o_ref)
    lerr = np.abs(lse - lse_ref)
    stats = {"max_abs_o": float(err.max()), "mean_abs_o": float(err.mean()),
             "max_abs_lse": float(lerr.max())}
    if dtype == torch.float32:
        assert stats["max_abs_o"] <= TOL_F32_O, (what, stats)
        assert stats["max_abs_lse"] <= TOL_F32_LSE, (what, stats)
        return stats
    # bf16: entries with |O_ref| >= 4 have a half-ulp of at least 2^-6 > 1.5e-2 in the bf16
    # output itself; there the bound is one bf16 ulp of O_ref (counted and reported).
    big = np.abs(o_ref) >= 4.0
    small_err = err[~big]
    stats["n_large_entries"] = int(big.sum())
    stats["max_abs_o_small"] = float(small_err.max()) if small_err.size else 0.0
    if big.any():
        stats["max_ulp_large"] = float((err[big] / bf16_ulp(o_ref[big])).max())
        assert stats["max_ulp_large"] <= 1.0, (what, stats)
    assert stats["max_abs_o_small"] <= TOL_BF16_O_MAX, (what, stats)
    if check_mean:
        assert stats["mean_abs_o"] <= TOL_BF16_O_MEAN, (what, stats)
    assert stats["max_abs_lse"] <= TOL_BF16_LSE, (what, stats)
    return stats


def rel_l2(x, ref) -> float:
    x, ref = f64(x), f64(ref)
    den = np.linalg.norm(ref.ravel())
    return float(np.linalg.norm((x - ref).ravel()) / max(den, 1e-30))


def check_grads(got: dict, ref: dict, dtype, what=""):
    """Relative L2 per gradient.  Where the exact gradient is zero (e.g. dQ and dK at N = 1,
    where P = 1 makes dS = 0) relative error is undefined; there the gradient must be zero
    to within the rounding of its inputs (max |x| <= tol)."""
    tol = TOL_F32_GRAD_REL_L2 if dtype == torch.float32 else TOL_GRAD_REL_L2
    stats = {}
    for n in ("dq", "dk", "dv"):
        g = f64(got[n])
        r = f64(ref[n])
        assert np.isfinite(g).all(), f"non-finite {n} {what}"
        if np.abs(r).max() <= 1e-12:
            stats[n] = ("abs", float(np.abs(g).max()))
            assert stats[n][1] <= tol, (what, n, stats)
            continue
        stats[n] = rel_l2(g, r)
        assert stats[n] <= tol, (what, n, stats)
    return stats


def guarded_empty(shape, dtype, device="cuda", pad=4096):
    """A tensor inside a larger buffer whose margins hold a sentinel (NaN for floating
    types, 0xAB for bytes); returns (view, check) where check() asserts that the margins
    are untouched."""
    n = int(np.prod(shape))
    floating = dtype.is_floating_point
    fill = float("nan") if floating else 0xAB
    buf = torch.full((n + 2 * pad,), fill, dtype=dtype, device=device)
    view = buf[pad:pad + n].view(shape)
    view.zero_()

    def check():
        for part in (buf[:pad].cpu(), buf[pad + n:].cpu()):
            ok = torch.isnan(part.float()).all() if floating else (part == 0xAB).all()
            assert ok, "write outside the output"

    return view, check


def oracle_threads(bytes_per_thread: float) -> int:
    """Host threads for an oracle call whose threads each hold ``bytes_per_thread`` of
    scratch (one head's S and P): every core, but no more than half of the memory the host
    reports available allows."""
    n = os.cpu_count() or 1
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    avail = int(line.split()[1]) * 1024
                    n = max(1, min(n, int(0.5 * avail // bytes_per_thread)))
                    break
    except OSError:
        pass
    return n


def record_stats(what: str, stats: dict) -> None:
    """Print the statistics of one comparison; with FA_PARITY_STATS set to a file path, also
    append them there as one JSON line."""
    print(what, stats)
    path = os.environ.get("FA_PARITY_STATS")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"what": what, **stats}) + "\n")
