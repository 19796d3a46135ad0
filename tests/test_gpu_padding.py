"""GPU: the padding-row debug check (ulp_check_padding) against a plain numpy
count of the elements that are not +-0 in global rows >= used_sequence."""
import numpy as np
import pytest
import torch

from quantize_pack_gb300 import configs, synth, ulp
import gpu_helpers as gh
import helpers as hp

pytestmark = pytest.mark.gpu

PADDED = [configs.PADDING, hp.PADDING_R, hp.LONG_R]


def numpy_count(shards, wl, rank=None):
    """Elements of [P, B, L, H, D] 16-bit shards (or one shard of `rank`) in
    global rows t >= used whose magnitude bits are not zero."""
    P, B, L = shards.shape[0], shards.shape[1], shards.shape[2]
    ranks = range(P) if rank is None else [rank]
    total = 0
    for r in ranks:
        rows = np.arange(L) + r * L
        pad = shards[r][:, rows >= wl.used_sequence]
        total += int(np.count_nonzero(pad.view(np.uint16) & 0x7FFF))
    return total


@pytest.mark.parametrize("wl", PADDED, ids=[w.name for w in PADDED])
def test_seeded_inputs_have_zero_padding(wl):
    inp = synth.make_inputs(wl)
    q, k, v, _, _ = gh.to_device(inp)
    assert ulp.check_padding(q, k, v, rank=None, world_size=wl.P, used_sequence=wl.used_sequence) == 0
    for r in range(wl.P):
        assert ulp.check_padding(q[r], k[r], v[r], rank=r, world_size=wl.P,
                                 used_sequence=wl.used_sequence) == 0


@pytest.mark.parametrize("wl", PADDED, ids=[w.name for w in PADDED])
def test_planted_values_are_counted(wl):
    inp = synth.make_inputs(wl)
    rng = np.random.default_rng(11)
    shards = {x: np.array(inp.shards(x)) for x in "qkv"}
    P, B, L, H, D = shards["q"].shape
    S, used = P * L, wl.used_sequence
    planted = 0
    for x in "qkv":
        bits = shards[x].view(np.uint16)
        for _ in range(7):                     # nonzero values in padding rows
            t = int(rng.integers(used, S))
            bits[t // L, rng.integers(B), t % L, rng.integers(H), rng.integers(D)] = 0x3C00 | int(rng.integers(1, 255))
        # -0 in a padding row and a value in the last live row: not counted
        t = int(rng.integers(used, S))
        bits[t // L, 0, t % L, 0, 0] = 0x8000
        t = used - 1
        bits[t // L, 0, t % L, 0, 1] = 0x3C00
    want = sum(numpy_count(shards[x], wl) for x in "qkv")
    assert want > 0
    dev = [gh.bits_to_dev(shards[x], wl.dtype) for x in "qkv"]
    assert ulp.check_padding(*dev, rank=None, world_size=P, used_sequence=used) == want
    for r in range(P):
        want_r = sum(numpy_count(shards[x], wl, rank=r) for x in "qkv")
        got_r = ulp.check_padding(dev[0][r], dev[1][r], dev[2][r], rank=r, world_size=P, used_sequence=used)
        assert got_r == want_r, r


def test_no_padding_checks_nothing():
    wl = configs.TINY
    inp = synth.make_inputs(wl)
    q, k, v, _, _ = gh.to_device(inp)
    q.fill_(1.0)
    for used in (None, wl.P * wl.L):
        assert ulp.check_padding(q, k, v, rank=None, world_size=wl.P, used_sequence=used) == 0
