"""Shared helpers for the GPU-vs-oracle parity tests.

Acceptance (the stated bar): the quantized state is bit-exact (codes,
scales/zeros, block token indices and counts, residual tokens, pool
membership, pool norms); the attention output, fp16 on the device, is
within max |d| <= 2e-3 and mean |d| <= 2e-4 of the oracle's double result.
"""
from __future__ import annotations

import numpy as np
import torch

MAX_ABS = 2e-3
MEAN_ABS = 2e-4
STATE_KEYS = ("bidx", "kcode", "ks", "kz", "vcode", "vs", "vz", "tk", "tv", "pidx", "pnorm", "pk", "pv")


def compare_state(gpu: dict, orc_cache, units=None):
    """Bit-exact comparison of the device export with the oracle, unit by unit."""
    U = gpu["bidx"].shape[0]
    units = range(U) if units is None else units
    for u in units:
        e = orc_cache.export_unit(u)
        assert (gpu["T"], gpu["nf"], gpu["tail"], gpu["npool"]) == (e["T"], e["nf"], e["tail"], e["npool"]), u
        assert np.array_equal(gpu["bcount"], e["bcount"]), u
        for k in STATE_KEYS:
            g = gpu[k][u]
            o = e[k]
            if not np.array_equal(g, o):
                bad = np.argwhere(g != o)
                raise AssertionError(f"unit {u} field {k}: {len(bad)} mismatches, first at {bad[:3].tolist()}: "
                                     f"gpu {g[tuple(bad[0])]} oracle {o[tuple(bad[0])]}")


def compare_out(out_gpu: torch.Tensor, ref: np.ndarray, where: str = ""):
    g = out_gpu.detach().float().cpu().numpy().astype(np.float64)
    d = np.abs(g - ref)
    assert np.all(np.isfinite(g)), f"non-finite output {where}"
    mx, mean = float(d.max()), float(d.mean())
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{where}: max|d|={mx:.3e} mean|d|={mean:.3e}"
    return mx, mean
