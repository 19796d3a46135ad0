"""Pins of the oracle's k_mean_global production.

Page "k_grouped_amax" (k_mean_global parameter) asks only for the global K
mean rounded to the input dtype.  The oracle fixes one summation order (fp32
block sums of 64 rows, fp64 partials per rank and across ranks); these tests
pin it to the exact mean (math.fsum) within that order's error bound, check
round-half-even on exact midpoints, and the padding identities."""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantize_pack_gb300 import configs, synth
import helpers as hp


def _decode(bits, dtype):
    return hp.f32(bits, dtype).astype(np.float64)


def _ulp(x, dtype):
    """Spacing of the dtype at |x| (normal range)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return 2.0 ** (e - (7 if dtype == configs.BF16 else 10))


@pytest.mark.parametrize("wl", [hp.TINY, hp.PADDING_R, hp.LONG_R, hp.SIX, hp.B3, hp.CROSS_PAD],
                         ids=lambda w: w.name)
def test_mean_is_the_nearest_dtype_value_within_the_error_bound(wl):
    inp = synth.make_inputs(wl)
    got = _decode(O.k_mean_global(inp.shards("k"), wl.dtype, used_sequence=wl.used_sequence),
                  wl.dtype)
    kf = hp.f32(inp.k, wl.dtype)[:, :inp.used].astype(np.float64)        # [B, used, H, D]
    n = inp.used
    exact = np.empty(got.shape)
    absum = np.abs(kf).sum(axis=1)
    for b in range(wl.B):
        for hh in range(wl.H):
            for d in range(wl.D):
                exact[b, hh, d] = math.fsum(kf[b, :, hh, d]) / n
    # fp32 block sums of <= 64 terms: |error| <= 63 * 2^-24 * sum|x|; the mean's
    # fp32 rounding adds 2^-24 |mean|
    bound = (63 * 2.0 ** -24 * absum / n + 2.0 ** -23 * np.abs(exact)) * 1.01
    half = _ulp(exact, wl.dtype) / 2
    assert np.all(np.abs(got - exact) <= half + bound)
    # away from ties (by more than the bound) the result is the nearest value
    far = np.abs(np.abs(got - exact) - half) > bound
    assert np.all(np.abs(got - exact)[far] < half[far])


@pytest.mark.parametrize("dtype", [configs.BF16, configs.FP16])
def test_exact_midpoints_round_to_even(dtype):
    """Two ranks, one row each: the mean of two adjacent dtype values is their
    exact midpoint (representable in fp32) and must round to the even one."""
    rng = np.random.default_rng(5)
    D = 64
    if dtype == configs.BF16:
        base = torch.randn(D).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    else:
        base = (rng.standard_normal(D) * 4).astype(np.float16).view(np.uint16)
    base = np.where((base & 0x7FFF) < 0x0400, base | 0x0400, base).astype(np.uint16)  # normal
    nxt = (base + 1).astype(np.uint16)
    k_all = np.stack([base, nxt]).reshape(2, 1, 1, 1, D)
    got = O.k_mean_global(np.ascontiguousarray(k_all), dtype).reshape(D)
    even = np.where(base % 2 == 0, base, nxt)
    assert np.array_equal(got, even)


def test_used_none_equals_used_S_and_padding_only_changes_the_count():
    wl = hp.LONG_R
    inp = synth.make_inputs(wl.replace(pad_rows=0, name="long_nopad"))
    k = inp.shards("k")
    a = O.k_mean_global(k, wl.dtype)
    b = O.k_mean_global(k, wl.dtype, used_sequence=wl.S)
    assert a.tobytes() == b.tobytes()
    # a constant channel has that constant as its mean, padded or not
    const = np.full_like(k, synth.to_bits(np.array([1.5], np.float32), wl.dtype)[0])
    used = wl.S - 80
    flat = const.transpose(1, 0, 2, 3, 4).reshape(wl.B, wl.S, wl.H, wl.D).copy()
    flat[:, used:] = 0
    const = synth.shard(flat, wl.P)
    m = _decode(O.k_mean_global(const, wl.dtype, used_sequence=used), wl.dtype)
    assert np.all(m == 1.5)
