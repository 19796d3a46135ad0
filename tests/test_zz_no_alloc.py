"""The allocation-free k_mean_global entry point, for callers that cannot
allocate device memory for a call (a host framework that already holds the
device memory, a plugin limited to the tensors it is handed, a loop where a
cudaMalloc may not run).  Through the C ABI:
  - the full long workload, then a smaller one, in one test: the second call
    finds the first one's nodes in the shared fixed array; both are bit-equal
    to the oracle and to the workspace entry point;
  - a shape whose nodes fill the 8 MiB array exactly is bit-equal to the
    workspace entry point, and one 512-row group more is rejected;
  - a shape far beyond the array is rejected with a message, nothing written.
Collected last, so a run that stops at its first failure has run the rest."""
import numpy as np
import pytest
import torch

import gpu_helpers as gh
import helpers as hp
from oracle import oracle as O
from quantize_pack_gb300 import configs, synth, ulp

pytestmark = pytest.mark.gpu

ARRAY_BYTES = 8 << 20


def _node_bytes(P, B, L, H, D):
    """Scratch the entry point needs: 8-byte nodes over groups of 512 rows."""
    return 8 * P * B * ((L + 511) // 512) * H * D


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def test_noalloc_matches_oracle_large_then_small_shape():
    for wl in (configs.LONG_NONALIGNED, hp.PADDING_R):
        assert _node_bytes(wl.P, wl.B, wl.L, wl.H, wl.D) <= ARRAY_BYTES
        host_k = synth.make_inputs(wl).shards("k")
        k = gh.bits_to_dev(host_k, wl.dtype)
        out = torch.full((wl.B, wl.H, wl.D), 7.0, dtype=k.dtype, device="cuda")
        got = ulp.k_mean_global_noalloc(k, used_sequence=wl.used_sequence, out=out)
        want_ws = ulp.k_mean_global(k, used_sequence=wl.used_sequence)
        torch.cuda.synchronize()
        assert got.data_ptr() == out.data_ptr()
        want = O.k_mean_global(host_k, wl.dtype, used_sequence=wl.used_sequence)
        assert np.array_equal(_bits(got), want), f"{wl.name}: differs from the oracle"
        assert torch.equal(got.view(torch.int16), want_ws.view(torch.int16)), wl.name
        del k, host_k


def test_noalloc_fills_the_array_exactly_and_rejects_one_group_more():
    P, B, L, H, D = 8, 1, 32768, 16, 128
    assert _node_bytes(P, B, L, H, D) == ARRAY_BYTES
    g = torch.Generator(device="cuda").manual_seed(5)
    k = (torch.randn(P, B, L, H, D, device="cuda", generator=g) * 2 + 0.5).to(torch.bfloat16)
    for used in (None, P * L - 100):
        got = ulp.k_mean_global_noalloc(k, used_sequence=used)
        want = ulp.k_mean_global(k, used_sequence=used)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), used
    # one more 512-row group per rank: rejected before any launch (k is not read)
    assert _node_bytes(P, B, L + 1, H, D) > ARRAY_BYTES
    lib = ulp.lib()
    out = torch.full((B, H, D), 3.0, dtype=torch.bfloat16, device="cuda")
    assert lib.ulp_k_mean_global_noalloc(k.data_ptr(), 0, B, L + 1, H, D, P, -1, out.data_ptr(), None) == -1
    assert b"scratch" in lib.ulp_last_error()
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)


def test_noalloc_rejects_shapes_beyond_the_fixed_array():
    # P=8, B=1, L=32768, H=64, D=128 needs 32 MiB of nodes, four times the
    # array: rejected before any launch (k is never read)
    lib = ulp.lib()
    out = torch.full((1, 64, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    status = lib.ulp_k_mean_global_noalloc(1 << 20, 0, 1, 32768, 64, 128, 8, -1, out.data_ptr(), None)
    assert status == -1
    assert b"scratch" in lib.ulp_last_error()
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
