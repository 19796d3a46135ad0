"""The whole quantize -> pack -> exchange -> unpack path of an emulated Ulysses
group of P ranks held on one GPU.

Pack is a programmatic dependent launch: it loads its inputs while derive
finishes (derive writes none of them).  ``capture`` records one step as a
CUDA graph.

All P shards sit in device memory; the stats all-gather is the stacked
[P, ...] buffer the boundary kernel writes, and the all-to-all is folded into
the pack's store addresses (dest-major send buffer = every destination's
recv_u8) or, on request, run as a separate device copy.  One step is four
launches of the CUDA library: boundary min/max -> derive -> pack -> unpack; or
three when pack derives the K boundary slots from the gathered min/max itself
(``fold_derive``, the default for launch-bound workloads); plus
k_grouped_amax when the unfused pack is chosen, and the copy when the exchange
is not folded.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import ulp


FOLD_BELOW_BYTES = 256 << 20


class UlyssesLowpPath:
    def __init__(self, *, B: int, L: int, H: int, D: int, world_size: int, dtype: torch.dtype,
                 used_sequence: Optional[int] = None, scale_sequence: Optional[int] = None,
                 aligned: Optional[bool] = None, q_group: int = ulp.GQ, fused: bool = True,
                 fold_exchange: bool = True, fold_derive: Optional[bool] = None,
                 pdl: Optional[bool] = None, pdl_unpack: Optional[bool] = None,
                 single_launch: Optional[bool] = None, device="cuda"):
        P = world_size
        self.B, self.L, self.H, self.D, self.P = B, L, H, D, P
        self.h = H // P
        self.S = P * L
        self.dtype = dtype
        self.used_sequence = used_sequence
        self.scale_sequence = scale_sequence
        self.aligned = aligned
        self.q_group = q_group
        self.fused = fused
        self.fold_exchange = fold_exchange
        # fold_derive: pack derives the K boundary slots itself (one launch
        # fewer; its warp-0 derive costs the large workloads more than the
        # launch it saves).  None: fold when the step is launch-bound, i.e.
        # its Q, K, V inputs are under twice the 129 MB L2.
        launch_bound = 6 * P * B * L * H * D < FOLD_BELOW_BYTES
        self.fold_derive = launch_bound if fold_derive is None else fold_derive
        # pdl: programmatic launch of pack, which follows the boundary min/max
        # (or derive); neither writes pack's inputs, so pack loads them before
        # waiting;
        # pdl_unpack: of unpack.  None: on for launch-bound steps (its launch
        # overlaps pack's tail, about 3 us a step), off otherwise (its early
        # CTAs would sit on SMs through pack's last wave)
        self.pdl_pack = 2 if pdl is None or pdl else 0
        self.pdl = launch_bound if pdl_unpack is None else bool(pdl_unpack)
        # single_launch: the whole step as one cooperative launch
        # (ulp.group_step: boundary min/max, pack with the derive and the
        # exchange folded in, unpack).  Off unless asked for (None = off):
        # chained by programmatic launch, the separate launches take less GPU
        # time (each grid barrier costs about 2 us, and the fused kernel runs
        # one CTA per SM); the single launch wins only where the host's
        # launch rate bounds the step.  It needs the fused amax and the
        # folded exchange.
        can_single = fused and fold_exchange and fold_derive is not False
        if single_launch and not can_single:
            raise ValueError("single_launch needs fused=True, fold_exchange=True and fold_derive not False")
        self.single_launch = bool(single_launch)
        if self.single_launch:
            self.fold_derive = True
        self.device = torch.device(device)
        self.chunk_bytes = ulp.chunk_bytes(B, L, self.h, D, q_group)
        f32 = dict(dtype=torch.float32, device=self.device)
        self.k_amax = torch.empty((P, B, H, ulp.slots(L, ulp.GK)), **f32)
        self.minmax = torch.empty((P, B, H, 2, 2, D), **f32)
        self.q_partial = torch.empty((P, B, H, 2), **f32)
        u8 = dict(dtype=torch.uint8, device=self.device)
        self.recv = torch.empty((P, P, self.chunk_bytes), **u8)
        self.send = None if fold_exchange else torch.empty((P, P, self.chunk_bytes), **u8)
        self.out = ulp.unpack_outputs(B, L, self.h, D, P, scale_sequence, self.device, num_dests=P,
                                      q_group=q_group)
        # the single launch's grid barrier (zero before the first step; each
        # step leaves it ready for the next) and its status word
        i32 = dict(dtype=torch.int32, device=self.device)
        self.barrier = torch.zeros(2, **i32) if self.single_launch else None
        self.status = torch.zeros(1, **i32) if self.single_launch else None

    @property
    def launches_per_step(self) -> int:
        if self.single_launch:
            return 1
        return 3 + (0 if self.fold_derive else 1) + (0 if self.fused else 1) + (0 if self.fold_exchange else 1)

    def run(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, k_mean: torch.Tensor,
            v_scale: torch.Tensor, on_pack=None, out=None):
        """q, k, v: stacked shards [P, B, L, H, D]; k_mean [B, H, D] (input
        dtype); v_scale [B, H, D] fp32.  Returns the per-destination outputs
        (q8, k8, v8, q_scale, k_scale), each with a leading P axis, in
        ``out`` (a tuple from ``new_outputs()``) or ``self.out``.
        ``on_pack`` (optional) is a pair of callables run right before and
        after the pack launch (used to time it); with the single launch, around
        that launch."""
        P, L = self.P, self.L
        step = dict(world_size=P, minmax=self.minmax, q_partial=self.q_partial, k_amax=self.k_amax,
                    recv=self.recv, out=self.out if out is None else out,
                    used_sequence=self.used_sequence, q_group=self.q_group, aligned=self.aligned,
                    scale_sequence=self.scale_sequence)
        if self.single_launch:
            if on_pack is not None:
                on_pack[0]()
            res = ulp.group_step(q, k, v, k_mean, v_scale, mode=ulp.STEP_COOPERATIVE, barrier=self.barrier,
                                 status=self.status, **step)
            if on_pack is not None:
                on_pack[1]()
            return res
        if self.fused and self.fold_exchange and self.pdl_pack == 2 and on_pack is None:
            # the same launches from one call into the library (less host
            # time per step where the host's launch rate bounds it)
            mode = (0 if self.fold_derive else ulp.STEP_DERIVE_SEPARATE) | (ulp.STEP_UNPACK_PDL if self.pdl else 0)
            return ulp.group_step(q, k, v, k_mean, v_scale, mode=mode, **step)
        if not self.fused:
            ulp.k_grouped_amax(k, k_mean, rank=None, world_size=P,
                               used_sequence=self.used_sequence, out=self.k_amax)
        ulp.boundary_minmax(k, q, rank=None, world_size=P, used_sequence=self.used_sequence,
                            q_group=self.q_group, out=(self.minmax, self.q_partial))
        if not self.fold_derive:
            ulp.derive_k_boundary_amax(self.k_amax, self.minmax, k_mean, rank=None, local_sequence=L,
                                       world_size=P)
        if on_pack is not None:
            on_pack[0]()
        ulp.pack(q, k, v, k_mean, self.k_amax, self.q_partial, v_scale, rank=None,
                 world_size=P, used_sequence=self.used_sequence, q_group=self.q_group,
                 fused=self.fused, send=self.recv if self.fold_exchange else self.send,
                 send_layout=ulp.SEND_DEST_MAJOR if self.fold_exchange else ulp.SEND_SOURCE_MAJOR,
                 gathered_minmax=self.minmax if self.fold_derive else None, enable_pdl=self.pdl_pack)
        if on_pack is not None:
            on_pack[1]()
        if not self.fold_exchange:
            ulp.alltoall_emulate(self.send, self.recv)
        return ulp.unpack_for_sage(self.recv, batch_size=self.B, local_sequence=L,
                                   local_heads=self.h, head_dim=self.D, world_size=P,
                                   aligned=self.aligned, scale_sequence=self.scale_sequence,
                                   q_group=self.q_group, out=self.out if out is None else out,
                                   enable_pdl=self.pdl)

    def check_status(self):
        """Raise if a single-launch step gave up at a grid barrier (reads the
        status word, so it synchronises).  Zeroes the barrier and the status
        first, so the next step starts clean."""
        if self.status is None:
            return
        st = int(self.status.item())
        if st != 0:
            self.barrier.zero_()
            self.status.zero_()
            raise RuntimeError(f"group_step: a grid barrier timed out (status {st}); outputs undefined")

    def new_outputs(self):
        """A fresh set of device output tensors shaped like ``self.out``."""
        return tuple(torch.empty_like(o) for o in self.out)

    def new_inputs(self):
        """Device input tensors (q, k, v, k_mean, v_scale) for one step."""
        P, B, L, H, D = self.P, self.B, self.L, self.H, self.D
        dev = self.device
        x = dict(dtype=self.dtype, device=dev)
        return (torch.empty((P, B, L, H, D), **x), torch.empty((P, B, L, H, D), **x),
                torch.empty((P, B, L, H, D), **x), torch.empty((B, H, D), **x),
                torch.empty((B, H, D), dtype=torch.float32, device=dev))

    def run_host(self, host_inputs, host_outputs, pipe=None):
        """Run consecutive steps from pinned host memory to pinned host memory.

        host_inputs[i] = (q, k, v, k_mean, v_scale) and host_outputs[i] = the
        five outputs, all pinned CPU tensors shaped like ``new_inputs()`` /
        ``self.out``.  Step i's upload, its kernels and its download run on
        three streams with two device buffer sets, so step i + 1's upload
        overlaps step i's kernels and download (the two copy directions run
        concurrently).  Returns once every download has been issued; the
        caller synchronises (``torch.cuda.synchronize``) before reading.
        ``pipe`` (from ``host_pipe()``) holds the device buffers and streams;
        a new one is made when None."""
        pipe = self.host_pipe() if pipe is None else pipe
        compute = torch.cuda.current_stream(self.device)
        for i, (hin, hout) in enumerate(zip(host_inputs, host_outputs)):
            s = i % 2
            din, dout = pipe["inputs"][s], pipe["outputs"][s]
            up = pipe["up"]
            up.wait_event(pipe["in_free"][s])            # step i-2's kernels are done with din
            with torch.cuda.stream(up):
                for d, h in zip(din, hin):
                    d.copy_(h, non_blocking=True)
                pipe["in_ready"][s].record(up)
            compute.wait_event(pipe["in_ready"][s])
            compute.wait_event(pipe["out_free"][s])      # step i-2's download is done with dout
            self.run(*din, out=dout)
            pipe["in_free"][s].record(compute)
            pipe["out_ready"][s].record(compute)
            down = pipe["down"]
            down.wait_event(pipe["out_ready"][s])
            with torch.cuda.stream(down):
                for h, d in zip(hout, dout):
                    h.copy_(d, non_blocking=True)
                pipe["out_free"][s].record(down)
        compute.wait_stream(pipe["down"])

    def host_pipe(self):
        """Device buffers, streams and events of ``run_host``."""
        ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]
        pipe = {"inputs": [self.new_inputs(), self.new_inputs()],
                "outputs": [self.new_outputs(), self.new_outputs()],
                "up": torch.cuda.Stream(self.device), "down": torch.cuda.Stream(self.device),
                "in_ready": ev(), "in_free": ev(), "out_ready": ev(), "out_free": ev()}
        for e in pipe["in_free"] + pipe["out_free"]:      # nothing to wait for yet
            e.record(torch.cuda.current_stream(self.device))
        return pipe

    def capture(self, q, k, v, k_mean, v_scale):
        """Record one step on these input tensors as a CUDA graph; replay it
        with ``graph.replay()`` after refilling the same tensors.  The outputs
        are ``self.out``."""
        torch.cuda.synchronize(self.device)
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            self.run(q, k, v, k_mean, v_scale)        # warm the caches of the lazy loader
        torch.cuda.current_stream(self.device).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.run(q, k, v, k_mean, v_scale)
        return graph
