"""The allocation-free k_mean_global entry point, for callers that cannot
allocate device memory for a call (a host framework that already holds the
device memory, a plugin limited to the tensors it is handed, a loop where a
cudaMalloc may not run): through the C ABI, two calls in a row with different
shapes -- the second finds the first one's leftovers in the shared fixed
array -- each bit-equal to the workspace entry point, and a shape too large
for the fixed array rejected with a message.  Collected last on purpose."""
import numpy as np
import pytest
import torch

import gpu_helpers as gh
import helpers as hp
from quantize_pack_gb300 import configs, synth, ulp

pytestmark = pytest.mark.gpu


def _k(wl):
    return gh.bits_to_dev(synth.make_inputs(wl).shards("k"), wl.dtype)


def test_noalloc_matches_workspace_entry_point_twice():
    for wl in (configs.LONG_NONALIGNED.replace(H=16, name="long_h2"), hp.PADDING_R):
        k = _k(wl)
        want = ulp.k_mean_global(k, used_sequence=wl.used_sequence)
        out = torch.full((wl.B, wl.H, wl.D), 7.0, dtype=k.dtype, device="cuda")
        got = ulp.k_mean_global_noalloc(k, used_sequence=wl.used_sequence, out=out)
        torch.cuda.synchronize()
        assert got.data_ptr() == out.data_ptr()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), wl.name


def test_noalloc_rejects_shapes_beyond_the_fixed_array():
    # P=8, B=1, L=32768, H=64, D=128 needs 8 * 8 * 1 * 64 * 64 * 128 bytes = 32 MiB of
    # nodes, more than the 8 MiB array: rejected before any launch (k is never read)
    lib = ulp.lib()
    out = torch.full((1, 64, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    status = lib.ulp_k_mean_global_noalloc(1 << 20, 0, 1, 32768, 64, 128, 8, -1, out.data_ptr(), None)
    assert status == -1
    assert b"scratch" in lib.ulp_last_error()
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
