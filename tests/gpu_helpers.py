"""Helpers of the GPU parity tests: device copies of the seeded inputs and
bitwise comparisons."""
from __future__ import annotations

import numpy as np
import torch

from quantize_pack_gb300 import configs


def torch_dtype(code: int) -> torch.dtype:
    return torch.bfloat16 if code == configs.BF16 else torch.float16


def bits_to_dev(bits: np.ndarray, code: int, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch_dtype(code)).to(device)


def to_device(inp, device="cuda"):
    """(q, k, v shards [P, B, L, H, D], k_mean [B, H, D], v_scale [B, H, D])."""
    wl = inp.wl
    return (bits_to_dev(inp.shards("q"), wl.dtype, device),
            bits_to_dev(inp.shards("k"), wl.dtype, device),
            bits_to_dev(inp.shards("v"), wl.dtype, device),
            bits_to_dev(inp.k_mean, wl.dtype, device),
            torch.from_numpy(inp.v_scale).to(device))


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def assert_bits_equal(got, want, what=""):
    """Bit-for-bit equality (fp32 compared as raw words, so +-inf and the
    sign of zero count)."""
    g = np.ascontiguousarray(host(got) if isinstance(got, torch.Tensor) else got)
    w = np.ascontiguousarray(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    if g.dtype == np.float32:
        g, w = g.view(np.uint32), w.view(np.uint32)
    else:
        g, w = g.view(np.uint8), w.view(np.uint8)
    if not np.array_equal(g, w):
        bad = np.argwhere(g != w)
        raise AssertionError(f"{what}: {len(bad)} mismatches, first at {bad[:5].tolist()}: "
                             f"got {g[tuple(bad[0])]} want {w[tuple(bad[0])]}")
