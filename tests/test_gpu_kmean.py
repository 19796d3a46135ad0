"""GPU parity of the k_mean_global production (the step before the path)
against the oracle, bit for bit, including the full-size workloads."""
import numpy as np
import pytest
import torch

import gpu_helpers as gh
import helpers as hp
from oracle import oracle as O
from quantize_pack_gb300 import configs, synth, ulp

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl", hp.CPU_WORKLOADS + [configs.PADDING, configs.LONG_NONALIGNED,
                                                   configs.HEAVY_TAIL],
                         ids=lambda w: w.name)
def test_k_mean_global_matches_oracle(wl):
    inp = synth.make_inputs(wl)
    k_sh = inp.shards("k")
    want = O.k_mean_global(k_sh, wl.dtype, used_sequence=wl.used_sequence)
    k = gh.bits_to_dev(k_sh, wl.dtype)
    got = ulp.k_mean_global(k, used_sequence=wl.used_sequence)
    torch.cuda.synchronize()
    assert got.dtype == gh.torch_dtype(wl.dtype) and tuple(got.shape) == (wl.B, wl.H, wl.D)
    g = got.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(g, want)


def test_k_mean_workspace_too_small_is_rejected():
    wl = hp.TINY
    k = gh.bits_to_dev(synth.make_inputs(wl).shards("k"), wl.dtype)
    need = ulp.k_mean_workspace_bytes(wl.B, wl.L, wl.H, wl.D, wl.P)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ulp.UlpError) as e:
        ulp.k_mean_global(k, workspace=ws)
    assert e.value.status == -1


@pytest.mark.parametrize("wl", [hp.TINY, hp.LONG_R, hp.SIX, hp.L1, hp.USED1, configs.LONG_NONALIGNED],
                         ids=lambda w: w.name)
def test_every_launch_shape_gives_the_same_bits(wl):
    """The first kernel's blocks per thread (1, 2, 4, 8) changes only the
    launch shape: every value reproduces the oracle bit for bit."""
    inp = synth.make_inputs(wl)
    k_sh = inp.shards("k")
    want = O.k_mean_global(k_sh, wl.dtype, used_sequence=wl.used_sequence)
    k = gh.bits_to_dev(k_sh, wl.dtype)
    for g in (1, 2, 4, 8):
        got = ulp.k_mean_global_grouped(k, g, used_sequence=wl.used_sequence)
        torch.cuda.synchronize()
        assert np.array_equal(got.view(torch.int16).cpu().numpy().view(np.uint16), want), g
    with pytest.raises(ulp.UlpError):
        ulp.k_mean_global_grouped(k, 3)
