"""Pins of the oracle's K amax, boundary min/max and derive steps.

Page "derive_k_boundary_amax": the derived slot equals the direct amax of
|rn(K - m)| over the whole group (monotone rn subtraction), a padding-only
slice contributes exactly 1e-7, a single-toucher boundary is bit-neutral.
Page "k_grouped_amax": used == S / None leave the output untouched; only the
partial live group (used-1)//64 changes under padding.
"""
import numpy as np
import pytest

from oracle import oracle as O
from quantize_pack_gb300 import synth
import helpers as hp


@pytest.mark.parametrize("wl", hp.CPU_WORKLOADS, ids=lambda w: w.name)
def test_derived_amax_equals_whole_group_amax(wl):
    """Every touched slot of every rank, after derive, is bit-equal to the
    direct amax over the global group's live rows (brute force on the
    unsharded tensor); groups with no live row follow the don't-care rule."""
    inp, res = hp.cached(wl)
    direct = hp.global_k_amax(inp)
    used = inp.used
    gu = (used - 1) // 64
    m_abs = np.maximum(np.abs(hp.f32(inp.k_mean, wl.dtype)).max(axis=2), hp.EPS)  # [B, H]
    for r in range(wl.P):
        groups = hp.touched_groups(r, wl.L, 64)
        for j, g in enumerate(groups):
            got = res["amax"][r][:, :, j]
            if g <= gu:
                assert np.array_equal(got.view(np.uint32), direct[:, :, g].view(np.uint32)), (r, g)
            elif j == 0 or j == len(groups) - 1:
                # fully padded boundary group: every slice is padding only
                assert np.all(got == hp.EPS), (r, g)
            else:
                # fully padded interior group: the kernel value over zero rows
                assert np.array_equal(got, m_abs), (r, g)
        for j in range(len(groups), O.slots(wl.L, 64)):
            assert np.all(res["amax"][r][:, :, j] == hp.EPS)


@pytest.mark.parametrize("wl", hp.CPU_WORKLOADS, ids=lambda w: w.name)
def test_kernel_amax_is_the_slice_partial(wl):
    """Before derive, slot j of rank r is the amax over r's own rows of the
    group (live rows only for the partial live group)."""
    inp, res = hp.cached(wl)
    kf = hp.f32(inp.k, wl.dtype)
    m = hp.f32(inp.k_mean, wl.dtype)
    c = np.abs(kf - m[:, None])
    used = inp.used
    gu = (used - 1) // 64 if used < wl.S else -1
    for r in range(wl.P):
        for j, g in enumerate(hp.touched_groups(r, wl.L, 64)):
            lo, hi = max(g * 64, r * wl.L), min(g * 64 + 64, (r + 1) * wl.L)
            if g == gu:
                hi = min(hi, used)
            want = np.full((wl.B, wl.H), hp.EPS, np.float32)
            if hi > lo:
                want = np.maximum(c[:, lo:hi].max(axis=(1, 3)), hp.EPS)
            assert np.array_equal(res["amax_kernel"][r][:, :, j], want), (r, g)


@pytest.mark.parametrize("wl", hp.CPU_WORKLOADS, ids=lambda w: w.name)
def test_minmax_and_q_partials(wl):
    inp, res = hp.cached(wl)
    kf = hp.f32(inp.k, wl.dtype)
    qa = np.abs(hp.f32(inp.q, wl.dtype))
    used = inp.used
    assert not np.any(np.signbit(res["minmax"]) & (res["minmax"] == 0))    # no -0 stored
    for r in range(wl.P):
        for e, G in ((0, 64), (1, 64)):
            groups = hp.touched_groups(r, wl.L, 64)
            g = groups[0] if e == 0 else groups[-1]
            lo, hi = max(g * 64, r * wl.L), min(g * 64 + 64, (r + 1) * wl.L, used)
            mn, mx = res["minmax"][r][:, :, e, 0], res["minmax"][r][:, :, e, 1]
            if hi <= lo:
                assert np.all(mn == np.inf) and np.all(mx == -np.inf)
            else:
                rows = kf[:, lo:hi] + np.float32(0)          # -0 -> +0
                assert np.array_equal(mn, rows.min(axis=1))
                assert np.array_equal(mx, rows.max(axis=1))
            G_Q = wl.q_group
            qg = hp.touched_groups(r, wl.L, G_Q)
            gq = qg[0] if e == 0 else qg[-1]
            lo, hi = max(gq * G_Q, r * wl.L), min(gq * G_Q + G_Q, (r + 1) * wl.L)
            want = np.maximum(qa[:, lo:hi].max(axis=(1, 3)), hp.EPS)
            assert np.array_equal(res["qb"][r][:, :, e], want)


@pytest.mark.parametrize("wl", [hp.TINY, hp.VIDEO_R, hp.HEAVY_R, hp.SPAN4], ids=lambda w: w.name)
def test_used_none_and_used_S_identical(wl):
    inp = synth.make_inputs(wl)
    k_sh = inp.shards("k")
    for r in range(wl.P):
        a = O.k_grouped_amax(k_sh[r], inp.k_mean, wl.dtype, rank=r, world_size=wl.P)
        b = O.k_grouped_amax(k_sh[r], inp.k_mean, wl.dtype, rank=r, world_size=wl.P,
                             used_sequence=wl.S)
        assert a.tobytes() == b.tobytes()


@pytest.mark.parametrize("wl", [hp.PADDING_R, hp.LONG_R, hp.SPAN4_PAD, hp.L1, hp.CROSS_PAD,
                                hp.SIX, hp.USED64], ids=lambda w: w.name)
def test_only_partial_live_group_changes(wl):
    """On zero-padded input, used vs None differ in the slot of (used-1)//64
    only, on the ranks whose slice holds that group."""
    inp = synth.make_inputs(wl)
    k_sh = inp.shards("k")
    gu = (inp.used - 1) // 64
    for r in range(wl.P):
        a = O.k_grouped_amax(k_sh[r], inp.k_mean, wl.dtype, rank=r, world_size=wl.P)
        b = O.k_grouped_amax(k_sh[r], inp.k_mean, wl.dtype, rank=r, world_size=wl.P,
                             used_sequence=inp.used)
        diff = np.nonzero(np.any(a != b, axis=(0, 1)))[0]
        first = (r * wl.L) // 64
        assert set(diff.tolist()) <= {gu - first}
        if inp.used % 64 == 0:
            assert diff.size == 0


def test_padding_only_slice_contributes_floor():
    wl = hp.CROSS_PAD                  # used = 80; rank 1 holds rows 96..127 of group 1
    inp, res = hp.cached(wl)
    assert np.all(res["minmax"][1][:, :, 0, 0] == np.inf)
    assert np.all(res["minmax"][1][:, :, 0, 1] == -np.inf)
    assert np.all(res["amax_kernel"][1][:, :, 0] == hp.EPS)
    # the derived slot of group 1 is rank 0's live partial on both ranks
    assert np.array_equal(res["amax"][0][:, :, 1], res["amax_kernel"][0][:, :, 1])
    assert np.array_equal(res["amax"][1][:, :, 0], res["amax_kernel"][0][:, :, 1])
    # a contribution built from sentinels alone is exactly 1e-7
    g = np.zeros((2, 1, 1, 2, 2, 4), np.float32)
    g[:, :, :, :, 0, :] = np.inf
    g[:, :, :, :, 1, :] = -np.inf
    km = synth.to_bits(np.array([[[1.0, -2.0, 3.0, 0.5]]], np.float32), 0)
    ga = np.full((1, 1, O.slots(96, 64)), 5.0, np.float32)
    O.derive_k_boundary_amax(ga, g, km, 0, rank=1, local_sequence=96, world_size=2)
    assert ga[0, 0, 0] == hp.EPS and ga[0, 0, 1] == hp.EPS and ga[0, 0, 2] == 5.0


@pytest.mark.parametrize("wl", [hp.VIDEO_R, hp.HEAVY_R], ids=lambda w: w.name)
def test_aligned_derive_is_bit_neutral(wl):
    inp, res = hp.cached(wl)
    assert res["amax"].tobytes() == res["amax_kernel"].tobytes()


def test_derive_hand_example():
    """A two-rank group worked by hand: m = (1.5, -2), rank 0 rows give
    K in [1, 2] x [-3, -2.5], rank 1 rows [0.25, 1.75] x [-1, -2]."""
    B, H, D, L, P = 1, 1, 2, 96, 2
    g = np.zeros((P, B, H, 2, 2, D), np.float32)
    # rank 0 touches groups 0, 1 (group 1 = its e=1); rank 1 touches 1, 2 (e=0)
    g[0, 0, 0, 1, 0] = [1.0, -3.0]      # min
    g[0, 0, 0, 1, 1] = [2.0, -2.5]      # max
    g[1, 0, 0, 0, 0] = [0.25, -2.0]
    g[1, 0, 0, 0, 1] = [1.75, -1.0]
    km = synth.to_bits(np.array([[[1.5, -2.0]]], np.float32), 0)
    ga = np.full((B, H, O.slots(L, 64)), 0.0, np.float32)
    O.derive_k_boundary_amax(ga, g, km, 0, rank=0, local_sequence=L, world_size=P)
    # rank 0: d0 max(2-1.5, 1.5-1) = 0.5; d1 max(-2.5+2, -2+3) = 1.0 -> 1.0
    # rank 1: d0 max(1.75-1.5, 1.5-0.25) = 1.25; d1 max(-1+2, -2+2) = 1.0 -> 1.25
    assert ga[0, 0, 1] == np.float32(1.25)
