"""Full-size parity: the three large workloads at their published sizes (and
the long one with 64-row Q groups, as `bench.py --q-group 64` runs it), run
exactly as bench.py times them (every rank in one launch per step, fused
amax+pack with the exchange folded into the stores, unpack of every
destination), compared bit for bit with the oracle over every output byte.
The oracle needs ~10-30 s per workload on one core."""
import numpy as np
import pytest
import torch

import gpu_helpers as gh
import helpers as hp
from quantize_pack_gb300 import configs, synth
from quantize_pack_gb300.path import UlyssesLowpPath

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl", [configs.VIDEO_DIT, configs.LONG_NONALIGNED, configs.HEAVY_TAIL,
                                configs.LONG_NONALIGNED.replace(
                                    q_group=64, name=configs.LONG_NONALIGNED.name + "_gq64")],
                         ids=lambda w: w.name)
def test_full_size_workload(wl):
    inp = synth.make_inputs(wl)
    q, k, v, km, vs = gh.to_device(inp)
    path = UlyssesLowpPath(B=wl.B, L=wl.L, H=wl.H, D=wl.D, world_size=wl.P,
                           dtype=gh.torch_dtype(wl.dtype), used_sequence=wl.used_sequence,
                           scale_sequence=wl.scale_sequence, aligned=wl.aligned,
                           q_group=wl.q_group)
    for _ in range(2):
        outs = path.run(q, k, v, km, vs)
    torch.cuda.synchronize()
    got = [gh.host(t) for t in outs]
    got_recv = gh.host(path.recv)
    got_amax = gh.host(path.k_amax)
    del q, k, v, path, outs
    torch.cuda.empty_cache()

    res = hp.run_oracle(inp)
    gh.assert_bits_equal(got_amax, res["amax"], "k_amax")
    gh.assert_bits_equal(got_recv, res["recv"], "chunks")
    for i, name in enumerate(["q8", "k8", "v8", "q_scale", "k_scale"]):
        want = np.stack([res["out"][p][i] for p in range(wl.P)])
        gh.assert_bits_equal(got[i], want, name)
    spad = (wl.S + 63) // 64 * 64
    assert got[2].shape[-1] == spad and not np.any(got[2][..., wl.S:])
