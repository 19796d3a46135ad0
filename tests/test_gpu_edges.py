"""GPU edge cases: guard bytes around every output stay untouched (no write
outside the documented extents), rejected calls leave their outputs
untouched, non-default streams, and repeated steps on changing inputs."""
import numpy as np
import pytest
import torch

import gpu_helpers as gh
import helpers as hp
from quantize_pack_gb300 import synth, ulp
from quantize_pack_gb300.path import UlyssesLowpPath

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side of an output
PATTERN = 0xA5


def guarded(shape, dtype):
    """A tensor of `shape` inside a byte buffer filled with PATTERN, with GUARD
    bytes on both sides (the inner tensor stays 16-byte aligned)."""
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    buf = torch.full((n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
    inner = buf[GUARD:GUARD + n].view(dtype).view(shape)
    return buf, inner


def guards_intact(buf):
    b = gh.host(buf)
    return bool(np.all(b[:GUARD] == PATTERN) and np.all(b[-GUARD:] == PATTERN))


@pytest.mark.parametrize("wl", [hp.TINY, hp.SPAN4_PAD, hp.SIX, hp.LONG_R, hp.B3, hp.G64[2], hp.G64[5]],
                         ids=lambda w: w.name)
def test_outputs_have_untouched_guards(wl):
    inp, res, (q, k, v, km, vs) = _setup(wl)
    P, B, L, H, D = wl.P, wl.B, wl.L, wl.H, wl.D
    nk = ulp.slots(L, 64)
    ga_buf, ga = guarded((P, B, H, nk), torch.float32)
    ulp.k_grouped_amax(k, km, rank=None, world_size=P, used_sequence=wl.used_sequence, out=ga)
    mm_buf, mm = guarded((P, B, H, 2, 2, D), torch.float32)
    qp_buf, qp = guarded((P, B, H, 2), torch.float32)
    G_Q = wl.q_group
    ulp.boundary_minmax(k, q, rank=None, world_size=P, used_sequence=wl.used_sequence, q_group=G_Q,
                        out=(mm, qp))
    ulp.derive_k_boundary_amax(ga, mm, km, rank=None, local_sequence=L, world_size=P)
    cb = ulp.chunk_bytes(B, L, wl.h, D, G_Q)
    send_buf, send = guarded((P, P, cb), torch.uint8)
    ulp.pack(q, k, v, km, ga, qp, vs, rank=None, world_size=P, used_sequence=wl.used_sequence,
             q_group=G_Q, fused=False, send=send)
    recv_buf, recv = guarded((P, P, cb), torch.uint8)
    ulp.alltoall_emulate(send, recv)
    shapes = [o.shape for o in ulp.unpack_outputs(B, L, wl.h, D, P, wl.scale_sequence, "cuda", P,
                                                  q_group=G_Q)]
    dts = [torch.int8, torch.int8, torch.uint8, torch.float32, torch.float32]
    outs = [guarded(s, d) for s, d in zip(shapes, dts)]
    ulp.unpack_for_sage(recv, batch_size=B, local_sequence=L, local_heads=wl.h, head_dim=D,
                        world_size=P, scale_sequence=wl.scale_sequence, q_group=G_Q,
                        out=[o[1] for o in outs])
    torch.cuda.synchronize()
    for name, buf in [("amax", ga_buf), ("minmax", mm_buf), ("q partial", qp_buf), ("send", send_buf),
                      ("recv", recv_buf)] + [(f"out{i}", o[0]) for i, o in enumerate(outs)]:
        assert guards_intact(buf), name
    gh.assert_bits_equal(ga, res["amax"], "amax")
    gh.assert_bits_equal(send, res["send"], "send")
    for i, o in enumerate(outs):
        gh.assert_bits_equal(o[1], np.stack([res["out"][p][i] for p in range(P)]), f"out{i}")


def _setup(wl):
    inp, res = hp.cached(wl)
    return inp, res, gh.to_device(inp)


def test_rejected_calls_leave_outputs_untouched():
    wl = hp.TINY
    inp, res, (q, k, v, km, vs) = _setup(wl)
    out = torch.full((wl.P, wl.B, wl.H, ulp.slots(wl.L, 64)), 7.0, device="cuda")
    for kw, status in [(dict(world_size=3), -1), (dict(used_sequence=0), -1),
                       (dict(used_sequence=wl.S + 1), -1)]:
        args = dict(rank=None, world_size=wl.P, used_sequence=None, out=out)
        args.update(kw)
        with pytest.raises(ulp.UlpError) as e:
            ulp.k_grouped_amax(k, km, **args)
        assert e.value.status == status
    send = torch.full((wl.P, wl.P, ulp.chunk_bytes(wl.B, wl.L, wl.h, wl.D)), 3, dtype=torch.uint8,
                      device="cuda")
    with pytest.raises(ulp.UlpError):
        ulp.pack(q, k, v, km, out, torch.zeros(wl.P, wl.B, wl.H, 2, device="cuda"), vs, rank=None,
                 world_size=wl.P, send=send, send_layout=7)
    outs = ulp.unpack_outputs(wl.B, wl.L, wl.h, wl.D, wl.P, None, "cuda")
    for o in outs:
        o.fill_(5)
    with pytest.raises(ulp.UlpError) as e:
        ulp.unpack_for_sage(send[0], batch_size=wl.B, local_sequence=wl.L, local_heads=wl.h,
                            head_dim=wl.D, world_size=wl.P, aligned=True, out=outs)
    assert "aligned" in str(e.value)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0) and torch.all(send == 3)
    assert all(torch.all(o == 5) for o in outs)


def test_non_default_stream_and_changing_inputs():
    wl = hp.LONG_R
    path = UlyssesLowpPath(B=wl.B, L=wl.L, H=wl.H, D=wl.D, world_size=wl.P,
                           dtype=gh.torch_dtype(wl.dtype), used_sequence=wl.used_sequence,
                           scale_sequence=wl.scale_sequence)
    side = torch.cuda.Stream()
    for seed in (21, 22):
        inp = synth.make_inputs(wl.replace(seed=seed, name=f"{wl.name}_s{seed}"))
        res = hp.run_oracle(inp)
        with torch.cuda.stream(side):
            q, k, v, km, vs = gh.to_device(inp)
            outs = path.run(q, k, v, km, vs)
        side.synchronize()
        for i, name in enumerate(["q8", "k8", "v8", "q_scale", "k_scale"]):
            gh.assert_bits_equal(outs[i], np.stack([res["out"][p][i] for p in range(wl.P)]), name)


@pytest.mark.parametrize("pdl", [False, True], ids=["pdl_off", "pdl_on"])
def test_programmatic_launch_on_and_off(pdl):
    wl = hp.PADDING_R
    inp, res, (q, k, v, km, vs) = _setup(wl)
    path = UlyssesLowpPath(B=wl.B, L=wl.L, H=wl.H, D=wl.D, world_size=wl.P,
                           dtype=gh.torch_dtype(wl.dtype), used_sequence=wl.used_sequence,
                           scale_sequence=wl.scale_sequence, pdl=pdl, pdl_unpack=pdl,
                           single_launch=False)
    for _ in range(3):
        outs = path.run(q, k, v, km, vs)
    torch.cuda.synchronize()
    for i, name in enumerate(["q8", "k8", "v8", "q_scale", "k_scale"]):
        gh.assert_bits_equal(outs[i], np.stack([res["out"][p][i] for p in range(wl.P)]), name)


@pytest.mark.parametrize("single", [False, True], ids=["three_launches", "single_launch"])
def test_cuda_graph_replay_with_new_inputs(single):
    wl = hp.SIX
    path = UlyssesLowpPath(B=wl.B, L=wl.L, H=wl.H, D=wl.D, world_size=wl.P,
                           dtype=gh.torch_dtype(wl.dtype), used_sequence=wl.used_sequence,
                           scale_sequence=wl.scale_sequence, single_launch=single)
    assert path.launches_per_step == (1 if single else 3)
    inp0 = synth.make_inputs(wl)
    q, k, v, km, vs = gh.to_device(inp0)
    graph = path.capture(q, k, v, km, vs)
    for seed in (31, 32):
        inp = synth.make_inputs(wl.replace(seed=seed, name=f"{wl.name}_g{seed}"))
        res = hp.run_oracle(inp)
        for dst, src in zip((q, k, v, km, vs), gh.to_device(inp)):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        for i, name in enumerate(["q8", "k8", "v8", "q_scale", "k_scale"]):
            gh.assert_bits_equal(path.out[i], np.stack([res["out"][p][i] for p in range(wl.P)]), name)
        path.check_status()


def test_host_pipeline_runs_consecutive_steps():
    """UlyssesLowpPath.run_host: three steps with different inputs, pinned
    host memory in and out, uploads overlapping the previous step's kernels
    and downloads; every step's outputs equal the oracle's."""
    wl = hp.PADDING_R
    path = UlyssesLowpPath(B=wl.B, L=wl.L, H=wl.H, D=wl.D, world_size=wl.P,
                           dtype=gh.torch_dtype(wl.dtype), used_sequence=wl.used_sequence,
                           scale_sequence=wl.scale_sequence)
    host_in, want = [], []
    for seed in (51, 52, 53):
        inp = synth.make_inputs(wl.replace(seed=seed, name=f"{wl.name}_h{seed}"))
        res = hp.run_oracle(inp)
        dev = gh.to_device(inp, device="cpu")
        host_in.append(tuple(t.pin_memory() for t in dev))
        want.append([np.stack([res["out"][p][i] for p in range(wl.P)]) for i in range(5)])
    host_out = [tuple(torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in path.out)
                for _ in host_in]
    path.run_host(host_in, host_out)
    torch.cuda.synchronize()
    for step, (got, exp) in enumerate(zip(host_out, want)):
        for i, name in enumerate(["q8", "k8", "v8", "q_scale", "k_scale"]):
            gh.assert_bits_equal(got[i], exp[i], f"step {step} {name}")


def test_group_step_barrier_timeout_reports_status():
    """The cooperative step's grid barrier gives up after its bound: with the
    arrival count preset far from any CTA's completing arrival, every CTA
    waits its 1 s, the kernel writes status 2 and returns (nothing hangs);
    check_status() raises, zeroes the barrier pair, and the next step is
    bit-exact again."""
    wl = hp.TINY
    inp, res, (q, k, v, km, vs) = _setup(wl)
    path = UlyssesLowpPath(B=wl.B, L=wl.L, H=wl.H, D=wl.D, world_size=wl.P,
                           dtype=gh.torch_dtype(wl.dtype), used_sequence=wl.used_sequence,
                           scale_sequence=wl.scale_sequence, single_launch=True)
    path.barrier[0] = 1 << 30                 # no arrival can make the count complete
    path.run(q, k, v, km, vs)
    torch.cuda.synchronize()
    assert int(path.status.item()) == 2
    with pytest.raises(RuntimeError, match="timed out"):
        path.check_status()
    assert path.barrier.tolist() == [0, 0] and int(path.status.item()) == 0
    outs = path.run(q, k, v, km, vs)
    torch.cuda.synchronize()
    path.check_status()
    for i, name in enumerate(["q8", "k8", "v8", "q_scale", "k_scale"]):
        gh.assert_bits_equal(outs[i], np.stack([res["out"][p][i] for p in range(wl.P)]), name)
