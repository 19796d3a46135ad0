"""GPU parity: every output of the CUDA path, bit for bit, against the CPU
oracle on the same seeded inputs (reduced and small workloads spanning
several tiles, ragged tails, padding, groups across 2..8 ranks)."""
import numpy as np
import pytest
import torch

import helpers as hp
import gpu_helpers as gh
from quantize_pack_gb300 import configs, ulp
from quantize_pack_gb300.path import UlyssesLowpPath

pytestmark = pytest.mark.gpu

GPU_WORKLOADS = hp.CPU_WORKLOADS + [configs.PADDING]


def _setup(wl):
    inp, res = hp.cached(wl)
    return inp, res, gh.to_device(inp)


@pytest.mark.parametrize("wl", GPU_WORKLOADS, ids=lambda w: w.name)
def test_k_grouped_amax(wl):
    inp, res, (q, k, v, km, vs) = _setup(wl)
    got = ulp.k_grouped_amax(k, km, rank=None, world_size=wl.P, used_sequence=wl.used_sequence)
    gh.assert_bits_equal(got, res["amax_kernel"], "k_grouped_amax (all ranks)")
    for r in sorted({0, wl.P - 1}):
        one = ulp.k_grouped_amax(k[r].contiguous(), km, rank=r, world_size=wl.P,
                                 used_sequence=wl.used_sequence)
        gh.assert_bits_equal(one, res["amax_kernel"][r], f"k_grouped_amax rank {r}")


@pytest.mark.parametrize("wl", GPU_WORKLOADS, ids=lambda w: w.name)
def test_boundary_minmax(wl):
    inp, res, (q, k, v, km, vs) = _setup(wl)
    mm, qp = ulp.boundary_minmax(k, q, rank=None, world_size=wl.P, used_sequence=wl.used_sequence,
                                 q_group=wl.q_group)
    gh.assert_bits_equal(mm, res["minmax"], "minmax")
    gh.assert_bits_equal(qp, res["qb"], "q partial")
    r = wl.P - 1
    mm1, qp1 = ulp.boundary_minmax(k[r].contiguous(), q[r].contiguous(), rank=r, world_size=wl.P,
                                   used_sequence=wl.used_sequence, q_group=wl.q_group)
    gh.assert_bits_equal(mm1, res["minmax"][r], "minmax one rank")
    gh.assert_bits_equal(qp1, res["qb"][r], "q partial one rank")


@pytest.mark.parametrize("wl", GPU_WORKLOADS, ids=lambda w: w.name)
def test_derive(wl):
    inp, res, (q, k, v, km, vs) = _setup(wl)
    ga = ulp.k_grouped_amax(k, km, rank=None, world_size=wl.P, used_sequence=wl.used_sequence)
    mm, _ = ulp.boundary_minmax(k, q, rank=None, world_size=wl.P, used_sequence=wl.used_sequence,
                                 q_group=wl.q_group)
    ulp.derive_k_boundary_amax(ga, mm, km, rank=None, local_sequence=wl.L, world_size=wl.P)
    gh.assert_bits_equal(ga, res["amax"], "derived amax (all ranks)")
    # one rank at a time, from the oracle's own kernel output and gather
    for r in range(wl.P):
        one = torch.from_numpy(res["amax_kernel"][r].copy()).cuda()
        ulp.derive_k_boundary_amax(one, torch.from_numpy(res["minmax"]).cuda(), km, rank=r,
                                   local_sequence=wl.L, world_size=wl.P)
        gh.assert_bits_equal(one, res["amax"][r], f"derived amax rank {r}")


@pytest.mark.parametrize("derive", ["separate", "folded"])
@pytest.mark.parametrize("fused", [True, False], ids=["fused", "unfused"])
@pytest.mark.parametrize("wl", GPU_WORKLOADS, ids=lambda w: w.name)
def test_pack(wl, fused, derive):
    """Pack against the oracle: the chunk bytes (source-major, dest-major,
    one rank) and k_amax.  derive = "separate": derive_k_boundary_amax runs
    first and pack reads the boundary slots; "folded": pack derives them from
    the gathered min/max itself and writes them to k_amax."""
    inp, res, (q, k, v, km, vs) = _setup(wl)
    P = wl.P
    folded = derive == "folded"
    if fused:
        # the slots pack must not read are poisoned
        ga = torch.full((P, wl.B, wl.H, ulp.slots(wl.L, 64)), float("nan"), device="cuda")
    else:
        ga = ulp.k_grouped_amax(k, km, rank=None, world_size=P, used_sequence=wl.used_sequence)
    mm, qp = ulp.boundary_minmax(k, q, rank=None, world_size=P, used_sequence=wl.used_sequence,
                                 q_group=wl.q_group)
    ga0 = ga.clone()
    if not folded:
        ulp.derive_k_boundary_amax(ga, mm, km, rank=None, local_sequence=wl.L, world_size=P)
    extra = dict(gathered_minmax=mm if folded else None)
    send = ulp.pack(q, k, v, km, ga, qp, vs, rank=None, world_size=P,
                    used_sequence=wl.used_sequence, q_group=wl.q_group, fused=fused, **extra)
    gh.assert_bits_equal(send, res["send"], "send (source-major)")
    gh.assert_bits_equal(ga, res["amax"], "k_amax after pack")
    if folded:
        ga.copy_(ga0)
    recv = ulp.pack(q, k, v, km, ga, qp, vs, rank=None, world_size=P,
                    used_sequence=wl.used_sequence, q_group=wl.q_group, fused=fused,
                    send_layout=ulp.SEND_DEST_MAJOR, **extra)
    gh.assert_bits_equal(recv, res["recv"], "send (dest-major) = recv")
    # single-rank calls write the same chunks
    r = P - 1
    one_amax = (ga0 if folded else ga)[r].contiguous()
    one = ulp.pack(q[r].contiguous(), k[r].contiguous(), v[r].contiguous(), km,
                   one_amax, qp, vs, rank=r, world_size=P,
                   used_sequence=wl.used_sequence, q_group=wl.q_group, fused=fused, **extra)
    gh.assert_bits_equal(one, res["send"][r], f"send rank {r}")
    gh.assert_bits_equal(one_amax, res["amax"][r], f"k_amax rank {r} after pack")


@pytest.mark.parametrize("wl", GPU_WORKLOADS, ids=lambda w: w.name)
def test_alltoall_and_unpack(wl):
    inp, res, _ = _setup(wl)
    P = wl.P
    send = torch.from_numpy(res["send"]).cuda()
    recv = ulp.alltoall_emulate(send)
    gh.assert_bits_equal(recv, res["recv"], "recv")
    outs = ulp.unpack_for_sage(recv, batch_size=wl.B, local_sequence=wl.L, local_heads=wl.h,
                               head_dim=wl.D, world_size=P, aligned=wl.aligned,
                               scale_sequence=wl.scale_sequence, q_group=wl.q_group)
    names = ["q8", "k8", "v8", "q_scale", "k_scale"]
    for i, name in enumerate(names):
        want = np.stack([res["out"][p][i] for p in range(P)])
        gh.assert_bits_equal(outs[i], want, name)
    # one destination at a time, page signature
    for p in sorted({0, P - 1}):
        one = ulp.unpack_for_sage(recv[p].contiguous(), batch_size=wl.B, local_sequence=wl.L,
                                  local_heads=wl.h, head_dim=wl.D, world_size=P,
                                  scale_sequence=wl.scale_sequence, q_group=wl.q_group)
        for i, name in enumerate(names):
            gh.assert_bits_equal(one[i], res["out"][p][i], f"{name} dest {p}")


@pytest.mark.parametrize("mode", ["fused_folded", "unfused_copy", "fused_separate_derive", "single_launch"])
@pytest.mark.parametrize("wl", GPU_WORKLOADS, ids=lambda w: w.name)
def test_whole_path(wl, mode):
    """The step through UlyssesLowpPath: fused pack with the exchange and the
    derive folded in (three launches); the unfused pack, the derive folded,
    with the all-to-all as its own copy; the fused pack after a separate
    derive launch; the whole step as one cooperative launch (ulp.group_step),
    whose grid barrier must come back to a zero count after every step."""
    inp, res, (q, k, v, km, vs) = _setup(wl)
    path = UlyssesLowpPath(B=wl.B, L=wl.L, H=wl.H, D=wl.D, world_size=wl.P,
                           dtype=gh.torch_dtype(wl.dtype), used_sequence=wl.used_sequence,
                           scale_sequence=wl.scale_sequence, aligned=wl.aligned,
                           q_group=wl.q_group, fused=(mode != "unfused_copy"),
                           fold_exchange=(mode != "unfused_copy"),
                           fold_derive=(mode != "fused_separate_derive"),
                           single_launch=(mode == "single_launch"))
    assert path.launches_per_step == {"fused_folded": 3, "unfused_copy": 5, "fused_separate_derive": 4,
                                      "single_launch": 1}[mode]
    for step in range(2):                   # a second step on the same buffers
        outs = path.run(q, k, v, km, vs)
        torch.cuda.synchronize()
        for i, name in enumerate(["q8", "k8", "v8", "q_scale", "k_scale"]):
            want = np.stack([res["out"][p][i] for p in range(wl.P)])
            gh.assert_bits_equal(outs[i], want, name)
        gh.assert_bits_equal(path.recv, res["recv"], "recv")
        gh.assert_bits_equal(path.k_amax, res["amax"], "k_amax")
        if mode == "single_launch":
            path.check_status()
            # two barriers a step: the count is back at zero, the generation
            # advanced by two
            assert path.barrier.tolist() == [0, 2 * (step + 1)]
            gh.assert_bits_equal(path.minmax, res["minmax"], "minmax")
            gh.assert_bits_equal(path.q_partial, res["qb"], "q_partial")
