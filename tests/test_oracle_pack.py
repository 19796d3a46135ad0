"""Pins of the oracle's pack, exchange and unpack_for_sage.

P-invariance: the unpacked outputs over all destinations equal a one-rank
(global) quantisation of the unsharded tensors computed here by brute force
with library routines (numpy float32 division and rint, torch's E4M3 cast),
using no slots, chunks or ranks.  Page "unpack_for_sage": V is [B, D, h,
ceil(S/64)*64] with a zero global tail; scale_sequence emits the leading
slots of the full-width tensors byte for byte; extra Q scale slots are finite.
"""
import numpy as np
import pytest

from oracle import oracle as O
import helpers as hp


def _assemble(res, wl):
    """Per-destination outputs stitched back to global head order."""
    q8 = np.concatenate([res["out"][p][0] for p in range(wl.P)], axis=2)   # [B, S, H, D]
    k8 = np.concatenate([res["out"][p][1] for p in range(wl.P)], axis=2)
    v8 = np.concatenate([res["out"][p][2] for p in range(wl.P)], axis=2)   # [B, D, H, Spad]
    qs = np.concatenate([res["out"][p][3] for p in range(wl.P)], axis=1)   # [B, H, Wq]
    ks = np.concatenate([res["out"][p][4] for p in range(wl.P)], axis=1)
    return q8, k8, v8, qs, ks


@pytest.mark.parametrize("wl", hp.CPU_WORKLOADS, ids=lambda w: w.name)
def test_p_invariance_against_global_quantisation(wl):
    inp, res = hp.cached(wl)
    q8, k8, v8, qs, ks = _assemble(res, wl)
    S, used = wl.S, inp.used
    qf, kf, vf = (hp.f32(getattr(inp, n), wl.dtype) for n in "qkv")
    m = hp.f32(inp.k_mean, wl.dtype)

    # Q: scales and codes from the global q_group-row group amax
    qa = hp.global_q_amax(inp)
    q_scale = (qa / np.float32(127)).astype(np.float32)
    wq = qs.shape[2]
    assert np.array_equal(qs.view(np.uint32), q_scale[:, :, :wq].view(np.uint32))
    row_qs = np.repeat(q_scale, wl.q_group, axis=2)[:, :, :S]             # [B, H, S]
    assert np.array_equal(q8, hp.int8_codes(qf, row_qs.transpose(0, 2, 1)[..., None]))

    # K: live rows and live groups from the global group amax of live rows
    ka = hp.global_k_amax(inp)
    k_scale = (ka / np.float32(127)).astype(np.float32)
    n_live = (used + 63) // 64
    wk = ks.shape[2]
    assert np.array_equal(ks[:, :, :min(wk, n_live)].view(np.uint32),
                          k_scale[:, :, :min(wk, n_live)].view(np.uint32))
    row_ks = np.repeat(k_scale, 64, axis=2)[:, :, :S].transpose(0, 2, 1)[..., None]
    kc = (kf - m[:, None]).astype(np.float32)
    want_k = hp.int8_codes(kc, row_ks)
    assert np.array_equal(k8[:, :used], want_k[:, :used])

    # V: E4M3 of v / v_scale, transposed to [B, D, H, Spad], zero tail
    want_v = hp.e4m3_codes(vf / inp.v_scale[:, None])                     # [B, S, H, D]
    assert np.array_equal(v8[..., :S], want_v.transpose(0, 3, 2, 1))
    assert not np.any(v8[..., S:])


@pytest.mark.parametrize("wl", hp.CPU_WORKLOADS, ids=lambda w: w.name)
def test_unpack_shapes_tail_and_scale_prefix(wl):
    inp, res = hp.cached(wl)
    S = wl.S
    Spad = (S + 63) // 64 * 64
    for p in range(wl.P):
        q8, k8, v8, qs, ks = res["out"][p]
        assert q8.shape == (wl.B, S, wl.h, wl.D) and k8.shape == q8.shape
        assert v8.shape == (wl.B, wl.D, wl.h, Spad)
        assert not np.any(v8[..., S:])
        assert np.all(np.isfinite(qs)) and np.all(np.isfinite(ks))
        wq, wk = O.scale_widths(S if wl.scale_sequence is None else wl.scale_sequence, wl.q_group)
        assert qs.shape == (wl.B, wl.h, wq) and ks.shape == (wl.B, wl.h, wk)
        # scale_sequence narrows the scales to the leading slots of full width
        full = O.unpack_for_sage(np.ascontiguousarray(res["recv"][p]), batch_size=wl.B,
                                 local_sequence=wl.L, local_heads=wl.h, head_dim=wl.D,
                                 world_size=wl.P, scale_sequence=None, q_group=wl.q_group)
        assert np.array_equal(full[0], q8) and np.array_equal(full[1], k8)
        assert np.array_equal(full[2], v8)
        assert full[3][:, :, :wq].tobytes() == np.ascontiguousarray(qs).tobytes()
        assert full[4][:, :, :wk].tobytes() == np.ascontiguousarray(ks).tobytes()


@pytest.mark.parametrize("wl", hp.CPU_WORKLOADS, ids=lambda w: w.name)
def test_shared_boundary_scale_bytes_agree(wl):
    """A group touched by two ranks carries the same scale bytes in both
    sources' chunks (group-wide identical values)."""
    inp, res = hp.cached(wl)
    lay = O.chunk_layout(wl.B, wl.L, wl.h, wl.D, wl.q_group)
    G_Q = wl.q_group
    for G, key, n in ((64, "k_scale", O.slots(wl.L, 64)), (G_Q, "q_scale", O.slots(wl.L, G_Q))):
        for g in range((wl.S + G - 1) // G):
            rs = hp.ranks_touching(g, wl.L, wl.P, G)
            vals = []
            for r in rs:
                j = g - (r * wl.L) // G
                for p in range(wl.P):
                    chunk = res["send"][r, p]
                    arr = chunk[lay[key]:lay[key] + 4 * wl.B * wl.h * n].view(np.float32)
                    vals.append(arr.reshape(wl.B, wl.h, n)[:, :, j].copy())
            per_rank = [np.concatenate(vals[i * wl.P:(i + 1) * wl.P], axis=1) for i in range(len(rs))]
            for v in per_rank[1:]:
                assert v.tobytes() == per_rank[0].tobytes(), (key, g)


@pytest.mark.parametrize("wl", [hp.TINY, hp.LONG_R, hp.HEAVY_R, hp.G64[1]], ids=lambda w: w.name)
def test_dequantisation_error_bounds(wl):
    """|code * scale - x| <= scale/2 (within a binary32 rounding) wherever
    the code did not saturate, and each group's amax element maps to +-127."""
    inp, res = hp.cached(wl)
    q8, k8, v8, qs, ks = _assemble(res, wl)
    qf = hp.f32(inp.q, wl.dtype).astype(np.float64)
    row_qs = np.repeat(hp.global_q_amax(inp).astype(np.float64) / 127, wl.q_group,
                       axis=2)[:, :, :wl.S]
    s = row_qs.transpose(0, 2, 1)[..., None]
    err = np.abs(q8.astype(np.float64) * s - qf)
    ok = np.abs(q8) < 127
    assert np.all(err[ok] <= s.repeat(wl.D, axis=3)[ok] * (0.5 + 2.0 ** -20))
    assert np.abs(q8).max() == 127


def test_exchange_is_the_transpose_of_chunks():
    wl = hp.SIX
    inp, res = hp.cached(wl)
    for s in range(wl.P):
        for p in range(wl.P):
            assert np.array_equal(res["recv"][p, s], res["send"][s, p])
