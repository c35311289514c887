"""Shared helpers of the GPU parity tests (host-side conversions; no method arithmetic)."""
from __future__ import annotations

import numpy as np
import pytest

from synth import inputs as I


def require_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    from dflash2_block_drafter_gb300 import _build
    import dflash2_block_drafter_gb300 as pkg
    _build.build()
    pkg.library()
    return torch


class OSite:
    """A conv site with float64 arrays (what the oracle reads)."""

    def __init__(self, s, blocks=None):
        sel = slice(None) if blocks is None else blocks
        self.w_kp = I.to_f64(s.w_kp)
        self.base = s.base.astype(np.float64)
        self.norm_w = I.to_f64(s.norm_w)
        self.y = I.to_f64(s.y)[sel]


def oracle_sites(wl, blocks=None):
    return [OSite(s, blocks) for s in wl.sites]


def dev_f64(t):
    """A device tensor back on the host as float64."""
    return t.detach().float().cpu().numpy().astype(np.float64)
