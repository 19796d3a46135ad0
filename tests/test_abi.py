"""The C ABI without a GPU: the library loads, exports every function the
header declares, its host geometry agrees with the oracle's (two independent
implementations), and argument checks reject bad calls before any launch."""
import ctypes
import os
import re

import pytest

from oracle import oracle as O
from quantize_pack_gb300 import build as B
from quantize_pack_gb300 import ulp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build_library()
    return ulp.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "ulp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ulp_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n


def test_geometry_agrees_with_oracle(lib):
    for L in list(range(1, 400)) + [1000, 4096, 9360, 16384]:
        for G in (64, 128):
            assert ulp.slots(L, G) == O.slots(L, G)
    for G_Q in (64, 128):
        for n in range(1, 1200):
            assert ulp.scale_widths(n, G_Q) == O.scale_widths(n, G_Q)
        for Bb, L, h, D in [(1, 96, 4, 64), (1, 1000, 4, 128), (2, 4096, 3, 128), (1, 9360, 5, 128),
                            (4, 16384, 16, 64), (3, 17, 3, 64), (2, 1, 1, 128)]:
            lay = O.chunk_layout(Bb, L, h, D, G_Q)
            assert ulp.chunk_bytes(Bb, L, h, D, G_Q) == lay["chunk_bytes"]
            assert ulp.chunk_offsets(Bb, L, h, D, G_Q) == (lay["q"], lay["k"], lay["v"],
                                                          lay["q_scale"], lay["k_scale"])
    for bad in (0, 32, 96, 256):
        with pytest.raises(ulp.UlpError):
            ulp.scale_widths(100, bad)
        with pytest.raises(ulp.UlpError):
            ulp.chunk_bytes(1, 96, 4, 64, bad)


FAKE = 1 << 20   # an aligned, never-dereferenced address: every call below fails validation


@pytest.mark.parametrize("args,status", [
    # dtype
    (dict(dtype=7), -2),
    # world size, rank, head dim, heads, used
    (dict(world_size=3), -1), (dict(world_size=16), -1), (dict(rank=2, world_size=2), -1),
    (dict(rank=-2), -1), (dict(D=96), -1), (dict(H=6, world_size=4), -1),
    (dict(used=0), -1), (dict(used=2 * 96 + 1), -1), (dict(L=0), -1), (dict(B=0), -1),
    (dict(pdl=3), -1),
    # alignment
    (dict(k=FAKE + 8), -3), (dict(k=0), -3), (dict(out=FAKE + 2), -3), (dict(km=FAKE + 4), -3),
])
def test_k_grouped_amax_rejects(lib, args, status):
    a = dict(k=FAKE, km=FAKE, dtype=0, B=1, L=96, H=8, D=64, rank=0, world_size=2, used=-1,
             out=FAKE, pdl=-1)
    a.update(args)
    got = lib.ulp_k_grouped_amax(a["k"], a["km"], a["dtype"], a["B"], a["L"], a["H"], a["D"],
                                 a["rank"], a["world_size"], a["used"], a["out"], a["pdl"], None)
    assert got == status
    assert lib.ulp_last_error() != b""


@pytest.mark.parametrize("args,status", [
    (dict(dtype=7), -2), (dict(world_size=3), -1), (dict(rank=2, world_size=2), -1),
    (dict(used=0), -1), (dict(used=2 * 96 + 1), -1),
    (dict(q=FAKE + 8), -3), (dict(v=FAKE + 4), -3), (dict(count=FAKE + 4), -3),
])
def test_check_padding_rejects(lib, args, status):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dtype=0, B=1, L=96, H=8, D=64, rank=-1, world_size=2, used=150,
             count=FAKE)
    a.update(args)
    got = lib.ulp_check_padding(a["q"], a["k"], a["v"], a["dtype"], a["B"], a["L"], a["H"], a["D"],
                                a["rank"], a["world_size"], a["used"], a["count"], None)
    assert got == status
    assert lib.ulp_last_error() != b""


def test_check_padding_without_padding_launches_nothing(lib):
    # used = -1 or S: no row to check, so the call returns before touching
    # the (fake) device pointers
    for used in (-1, 2 * 96):
        assert lib.ulp_check_padding(FAKE, FAKE, FAKE, 0, 1, 96, 8, 64, -1, 2, used, FAKE, None) == 0


def test_unpack_rejects(lib):
    ok = dict(recv=FAKE, B=1, L=96, h=4, D=64, P=2, aligned=-1, sseq=-1, gq=128, q8=FAKE,
              k8=FAKE, v8=FAKE, qs=FAKE, ks=FAKE, nd=1, pdl=-1)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.ulp_unpack_for_sage(a["recv"], a["B"], a["L"], a["h"], a["D"], a["P"],
                                       a["aligned"], a["sseq"], a["gq"], a["q8"], a["k8"], a["v8"],
                                       a["qs"], a["ks"], a["nd"], a["pdl"], None)
    assert call(aligned=1) == -1                       # L % 128 != 0
    assert b"aligned" in lib.ulp_last_error()
    assert call(sseq=0) == -1 and call(sseq=193) == -1
    assert call(P=5) == -1 and call(D=32) == -1 and call(nd=0) == -1
    assert call(v8=FAKE + 1) == -3
    assert call(gq=96) == -1 and b"q_group" in lib.ulp_last_error()


def test_pack_and_derive_reject(lib):
    base = [FAKE] * 8
    # fused must be 0/1, send_layout 0/1, q_group 64/128
    assert lib.ulp_pack(*base[:4], 0, *base[4:6], None, base[6], 1, 96, 8, 64, 0, 2, -1, 128, 2, FAKE, 0, -1, None) == -1
    assert lib.ulp_pack(*base[:4], 0, *base[4:6], None, base[6], 1, 96, 8, 64, 0, 2, -1, 128, 1, FAKE, 3, -1, None) == -1
    assert lib.ulp_pack(*base[:4], 0, *base[4:6], None, base[6], 1, 96, 8, 64, 0, 2, -1, 128, 1, FAKE + 2, 0, -1, None) == -3
    assert lib.ulp_pack(*base[:4], 0, *base[4:6], None, base[6], 1, 96, 8, 64, 0, 2, -1, 32, 1, FAKE, 0, -1, None) == -1
    # a misaligned gathered min/max buffer (the folded derive's input)
    assert lib.ulp_pack(*base[:4], 0, *base[4:6], FAKE + 2, base[6], 1, 96, 8, 64, 0, 2, -1, 128, 1, FAKE, 0, -1, None) == -3
    assert lib.ulp_derive_k_boundary_amax(FAKE, FAKE, FAKE, 1, 1, 8, 64, 2, 96, 2, None) == -1
    assert lib.ulp_boundary_minmax(FAKE, FAKE, 0, 1, 96, 8, 64, 0, 2, 500, 128, FAKE, FAKE, None) == -1
    assert lib.ulp_boundary_minmax(FAKE, FAKE, 0, 1, 96, 8, 64, 0, 2, -1, 0, FAKE, FAKE, None) == -1
    assert lib.ulp_alltoall_emulate(FAKE, FAKE, 2, 24, None) == -1
    assert lib.ulp_alltoall_emulate(FAKE, FAKE, 2, 32, None) == -1      # send == recv
    assert b"same buffer" in lib.ulp_last_error()


def test_group_step_rejects(lib):
    """ulp_group_step validates everything before it touches the device:
    pack's checks, unpack's, its own (the min/max and partial buffers, the
    barrier pair, the status word)."""
    ok = dict(q=FAKE, k=FAKE, v=FAKE, km=FAKE, dt=0, vs=FAKE, B=1, L=96, H=8, D=64, P=2, used=-1, gq=128,
              aligned=-1, sseq=-1, mm=FAKE, qp=FAKE, amax=FAKE, recv=FAKE, q8=FAKE, k8=FAKE, v8=FAKE, qs=FAKE,
              ks=FAKE, mode=1, bar=FAKE, st=FAKE)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.ulp_group_step(a["q"], a["k"], a["v"], a["km"], a["dt"], a["vs"], a["B"], a["L"], a["H"],
                                  a["D"], a["P"], a["used"], a["gq"], a["aligned"], a["sseq"], a["mm"],
                                  a["qp"], a["amax"], a["recv"], a["q8"], a["k8"], a["v8"], a["qs"], a["ks"],
                                  a["mode"], a["bar"], a["st"], None)
    assert call(bar=FAKE + 2) == -3 and b"barrier" in lib.ulp_last_error()
    assert call(bar=None) == -3
    assert call(st=FAKE + 1) == -3
    assert call(mm=None) == -1 and b"minmax" in lib.ulp_last_error()
    assert call(aligned=1) == -1 and b"aligned" in lib.ulp_last_error()     # L % 128 != 0
    assert call(gq=96) == -1 and b"q_group" in lib.ulp_last_error()
    assert call(q=FAKE + 8) == -3                                          # pack's alignment check
    assert call(v8=FAKE + 1) == -3                                         # unpack's
    assert call(P=5) == -1 and call(D=32) == -1 and call(dt=7) == -2
    assert call(used=193) == -1 and call(sseq=0) == -1
    # modes: unknown bits, the cooperative launch with another bit; the
    # separate launches validate everything before the first one
    assert call(mode=8) == -1 and call(mode=-1) == -1
    assert call(mode=3) == -1 and call(mode=5) == -1
    assert call(mode=0, bar=None, aligned=1) == -1 and b"aligned" in lib.ulp_last_error()
    assert call(mode=6, bar=None, mm=None) == -1 and b"minmax" in lib.ulp_last_error()
