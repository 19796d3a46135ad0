"""Pins of the oracle's geometry: slot counts, the chunk layout, the
consumer scale widths and which groups cross ranks."""
import os

import pytest

from oracle import oracle as O
from quantize_pack_gb300 import configs
import helpers as hp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "geometry.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_geometry_golden_matches_workloads():
    rows = _golden_rows()
    assert len(rows) == len(configs.ALL)
    for wl, row in zip(configs.ALL, rows):
        B, H, D, P, L, ks, qs, spad, wq, wk, wq2, wk2, cb = row
        assert (wl.B, wl.H, wl.D, wl.P, wl.L) == tuple(map(int, (B, H, D, P, L)))
        assert O.slots(wl.L, 64) == int(ks)
        assert O.slots(wl.L, 128) == int(qs)
        assert (wl.S + 63) // 64 * 64 == int(spad)
        assert O.scale_widths(wl.S) == (int(wq), int(wk))
        if wl.scale_sequence is not None:
            assert O.scale_widths(wl.scale_sequence) == (int(wq2), int(wk2))
        else:
            assert wq2 == wk2 == "-"
        assert O.chunk_layout(wl.B, wl.L, wl.h, wl.D)["chunk_bytes"] == int(cb)


@pytest.mark.parametrize("G", [64, 128])
def test_slots_bound_every_rank(G):
    # slots(L, G) must hold every group any rank touches, for every group size
    # of the Ulysses group, and is attained whenever L % G != 0 for some rank
    for P in (2, 4, 6, 8):
        for L in list(range(1, 300)) + [1000, 4096, 9360, 16384]:
            n = O.slots(L, G)
            touched = [len(hp.touched_groups(r, L, G)) for r in range(P)]
            assert max(touched) <= n, (P, L)
            if L % G == 0:
                assert max(touched) == n


@pytest.mark.parametrize("G_Q", [64, 128])
def test_chunk_sections_aligned_and_disjoint(G_Q):
    for B, L, h, D in [(1, 96, 4, 64), (1, 1000, 4, 128), (3, 17, 3, 64), (2, 1, 1, 128)]:
        lay = O.chunk_layout(B, L, h, D, G_Q)
        n = B * L * h * D
        assert lay["q"] == 0 and lay["k"] >= n and lay["v"] >= lay["k"] + n
        assert lay["q_scale"] >= lay["v"] + n
        assert lay["k_scale"] >= lay["q_scale"] + 4 * B * h * O.slots(L, G_Q)
        assert lay["chunk_bytes"] >= lay["k_scale"] + 4 * B * h * O.slots(L, 64)
        for key in ("k", "v", "q_scale", "k_scale", "chunk_bytes"):
            assert lay[key] % 16 == 0


@pytest.mark.parametrize("G_Q", [64, 128])
def test_scale_widths_cover_prefix(G_Q):
    for n in range(1, 2000):
        wq, wk = O.scale_widths(n, G_Q)
        assert (wq - 1) * G_Q < n <= wq * G_Q
        assert (wk - 1) * 64 < n <= wk * 64


def test_crossing_groups_of_the_workloads():
    # K groups touched by two ranks, by brute force over rows
    want = {
        "tiny": [1], "padding": [15, 31, 46], "video": [], "long": [146, 292, 438, 731, 877, 1023],
        "heavy": [],
    }
    for key, wl in zip(want, configs.ALL):
        got = [g for g in range((wl.S + 63) // 64) if len(hp.ranks_touching(g, wl.L, wl.P, 64)) > 1]
        assert got == want[key], key
