"""Python binding of libulp.so (ctypes): argument marshalling only.

Every step of the path runs in the CUDA library; this module turns torch
tensors into device pointers, sizes and the current CUDA stream, allocates
outputs with torch when the caller passes none, and raises ``UlpError`` on a
non-zero status.  There is no CPU fallback: without the built library every
call raises.

Function names and keyword arguments mirror the pages
"flashinfer.comm._ulysses_lowp.k_grouped_amax", "...derive_k_boundary_amax"
and "...unpack_for_sage"; ``rank=None`` runs every rank of an emulated
Ulysses group in one launch (per-rank tensors stacked on a leading axis).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libulp.so")

ULP_BF16, ULP_FP16, ULP_F32 = 0, 1, 2
ULP_ALL_RANKS = -1
SEND_SOURCE_MAJOR, SEND_DEST_MAJOR = 0, 1
PV_F16, PV_E4M3 = 0, 1   # precision of the attention's PV product
# group_step mode bits: one cooperative launch; else separate launches, with the
# derive as its own launch and/or unpack launched programmatically
STEP_COOPERATIVE, STEP_DERIVE_SEPARATE, STEP_UNPACK_PDL = 1, 2, 4
GK, GQ = 64, 128   # K group rows; default Q group rows (q_group=64 selects the other width)

_STATUS = {-1: "EINVAL", -2: "EDTYPE", -3: "EALIGN", -4: "ECUDA"}


class UlpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"ulp status {status} ({_STATUS.get(status, '?')}): {message}")
        self.status = status


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first (python -m quantize_pack_gb300.build or "
                "__graft_entry__.build()); the path has no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        L.ulp_last_error.restype = ctypes.c_char_p
        L.ulp_last_error.argtypes = []
        L.ulp_slots.argtypes = [_I, _I]
        L.ulp_scale_widths.argtypes = [_I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]
        L.ulp_chunk_bytes.argtypes = [_I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]
        L.ulp_chunk_offsets.argtypes = [_I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]
        L.ulp_k_mean_workspace_bytes.argtypes = [_I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]
        L.ulp_k_mean_global.argtypes = [_P, _I, _I, _I, _I, _I, _I, _I, _P, _SZ, _P, _P]
        L.ulp_k_mean_global_noalloc.argtypes = [_P, _I, _I, _I, _I, _I, _I, _I, _P, _P]
        L.ulp_k_mean_global_grouped.argtypes = [_P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _SZ, _P, _P]
        L.ulp_k_grouped_amax.argtypes = [_P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _I, _P]
        L.ulp_boundary_minmax.argtypes = [_P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P]
        L.ulp_derive_k_boundary_amax.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]
        L.ulp_check_padding.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P]
        L.ulp_pack.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                               _I, _P, _I, _I, _P]
        L.ulp_alltoall_emulate.argtypes = [_P, _P, _I, _SZ, _P]
        L.ulp_unpack_for_sage.argtypes = [_P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P,
                                          _I, _I, _P]
        L.ulp_sage_attention.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                         ctypes.c_float, _P, _SZ, _P, _I, _I, _P, _P]
        L.ulp_sage_attention_workspace_bytes.argtypes = [_I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]
        L.ulp_group_step.argtypes = [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                     _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P]
        for name in ("ulp_slots", "ulp_scale_widths", "ulp_chunk_bytes", "ulp_chunk_offsets",
                     "ulp_k_mean_workspace_bytes", "ulp_k_mean_global", "ulp_k_mean_global_noalloc",
                     "ulp_k_mean_global_grouped",
                     "ulp_k_grouped_amax", "ulp_boundary_minmax", "ulp_derive_k_boundary_amax",
                     "ulp_check_padding",
                     "ulp_pack", "ulp_alltoall_emulate", "ulp_unpack_for_sage", "ulp_group_step",
                     "ulp_sage_attention", "ulp_sage_attention_workspace_bytes"):
            getattr(L, name).restype = _I
        _lib = L
    return _lib


def _check(status: int) -> int:
    if status < 0:
        raise UlpError(status, lib().ulp_last_error().decode())
    return status


def _opt(x) -> int:
    return -1 if x is None else int(x)


def _tri(x: Optional[bool]) -> int:
    return -1 if x is None else int(bool(x))


def _pdl(x) -> int:
    """enable_pdl: None -> -1 (by device support), False/True -> 0/1, or 2 (pack
    may read its inputs before the preceding kernel completes)."""
    if x is None:
        return -1
    if isinstance(x, bool):
        return int(x)
    if int(x) in (0, 1, 2):
        return int(x)
    raise ValueError(f"enable_pdl must be None, a bool or 2, got {x!r}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ULP_BF16
    if t.dtype == torch.float16:
        return ULP_FP16
    raise TypeError(f"expected a bfloat16 or float16 tensor, got {t.dtype}")


def _ptr(t: torch.Tensor) -> int:
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


# ------------------------------------------------------------------ geometry

def slots(L: int, G: int) -> int:
    return _check(lib().ulp_slots(L, G))


def scale_widths(n: int, q_group: int = GQ) -> Tuple[int, int]:
    """(Q width, K width) of the consumer scale tensors for n rows."""
    q, k = _I(), _I()
    _check(lib().ulp_scale_widths(n, q_group, ctypes.byref(q), ctypes.byref(k)))
    return q.value, k.value


def chunk_bytes(B: int, L: int, h: int, D: int, q_group: int = GQ) -> int:
    n = _SZ()
    _check(lib().ulp_chunk_bytes(B, L, h, D, q_group, ctypes.byref(n)))
    return n.value


def chunk_offsets(B: int, L: int, h: int, D: int, q_group: int = GQ) -> Tuple[int, ...]:
    arr = (_SZ * 5)()
    _check(lib().ulp_chunk_offsets(B, L, h, D, q_group, arr))
    return tuple(int(x) for x in arr)


# ------------------------------------------------------------ path functions

def _rank_dims(x: torch.Tensor, rank: Optional[int]):
    """(rank code, number of stacked ranks, B, L, H, D) of a Q/K/V tensor."""
    if rank is None:
        if x.dim() != 5:
            raise ValueError("rank=None expects stacked shards [P, B, L, H, D]")
        return ULP_ALL_RANKS, x.shape[0], *x.shape[1:]
    if x.dim() != 4:
        raise ValueError("expected a shard [B, L, H, D]")
    return int(rank), 1, *x.shape


def k_mean_workspace_bytes(B: int, L: int, H: int, D: int, world_size: int) -> int:
    n = _SZ()
    _check(lib().ulp_k_mean_workspace_bytes(B, L, H, D, world_size, ctypes.byref(n)))
    return n.value


def k_mean_global(k: torch.Tensor, *, used_sequence: Optional[int] = None,
                  workspace: Optional[torch.Tensor] = None,
                  out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Global K mean [B, H, D] in k's dtype from every rank's shard
    k [P, B, L, H, D] (the all-reduce emulated in one call)."""
    P, B, L, H, D = k.shape
    need = k_mean_workspace_bytes(B, L, H, D, P)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=k.device)
    if out is None:
        out = torch.empty((B, H, D), dtype=k.dtype, device=k.device)
    _check(lib().ulp_k_mean_global(_ptr(k), _dtype_code(k), B, L, H, D, P, _opt(used_sequence),
                                   _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _ptr(out), _stream(k.device)))
    return out


def k_mean_global_grouped(k: torch.Tensor, blocks_per_thread: int, *,
                          used_sequence: Optional[int] = None,
                          workspace: Optional[torch.Tensor] = None,
                          out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """k_mean_global with the first kernel's blocks per thread fixed (1, 2, 4
    or 8) instead of chosen from the shape; the bits are the same for every
    value."""
    P, B, L, H, D = k.shape
    if workspace is None:
        workspace = torch.empty(k_mean_workspace_bytes(B, L, H, D, P), dtype=torch.uint8,
                                device=k.device)
    if out is None:
        out = torch.empty((B, H, D), dtype=k.dtype, device=k.device)
    _check(lib().ulp_k_mean_global_grouped(_ptr(k), _dtype_code(k), B, L, H, D, P,
                                           _opt(used_sequence), int(blocks_per_thread),
                                           _ptr(workspace),
                                           workspace.numel() * workspace.element_size(),
                                           _ptr(out), _stream(k.device)))
    return out


def k_mean_global_noalloc(k: torch.Tensor, *, used_sequence: Optional[int] = None,
                          out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """k_mean_global for callers that cannot allocate device memory for the
    call: the library keeps its intermediate sums in a fixed 8 MiB device
    array instead of a workspace (larger shapes raise).  Pass `out` to avoid
    any allocation on this side too.  Calls that can overlap on the GPU share
    that array and must be ordered by the caller."""
    P, B, L, H, D = k.shape
    if out is None:
        out = torch.empty((B, H, D), dtype=k.dtype, device=k.device)
    _check(lib().ulp_k_mean_global_noalloc(_ptr(k), _dtype_code(k), B, L, H, D, P,
                                           _opt(used_sequence), _ptr(out), _stream(k.device)))
    return out


def k_grouped_amax(k: torch.Tensor, k_mean_global: torch.Tensor, *, rank: Optional[int],
                   world_size: int, used_sequence: Optional[int] = None,
                   enable_pdl: Optional[bool] = None,
                   out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Per-touched-global-64-row-group fp32 amax of |K - k_mean_global|,
    [B, H, slots(L, 64)] (page "k_grouped_amax")."""
    rc, nr, B, L, H, D = _rank_dims(k, rank)
    shape = ((nr,) if rank is None else ()) + (B, H, slots(L, GK))
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=k.device)
    _check(lib().ulp_k_grouped_amax(_ptr(k), _ptr(k_mean_global), _dtype_code(k), B, L, H, D, rc,
                                    world_size, _opt(used_sequence), _ptr(out), _pdl(enable_pdl),
                                    _stream(k.device)))
    return out


def check_padding(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, rank: Optional[int],
                  world_size: int, used_sequence: Optional[int] = None) -> int:
    """Debug check of the precondition that input rows past used_sequence are
    zero (page "k_grouped_amax", used_sequence parameter): the number of Q, K
    and V elements in those rows that are not +-0 (0 when the inputs obey it).
    Waits for the count on the current stream."""
    rc, nr, B, L, H, D = _rank_dims(q, rank)
    count = torch.zeros(1, dtype=torch.int64, device=q.device)
    _check(lib().ulp_check_padding(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), B, L, H, D, rc, world_size,
                                   _opt(used_sequence), _ptr(count), _stream(q.device)))
    return int(count.item())


def boundary_minmax(k: torch.Tensor, q: torch.Tensor, *, rank: Optional[int], world_size: int,
                    used_sequence: Optional[int] = None, q_group: int = GQ,
                    out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None):
    """Raw-K boundary min/max [B, H, 2, 2, D] and Q boundary partial amax
    [B, H, 2] of a rank (stacked over ranks for rank=None: the gathered
    buffers)."""
    rc, nr, B, L, H, D = _rank_dims(k, rank)
    lead = (nr,) if rank is None else ()
    if out is None:
        mm = torch.empty(lead + (B, H, 2, 2, D), dtype=torch.float32, device=k.device)
        qp = torch.empty(lead + (B, H, 2), dtype=torch.float32, device=k.device)
    else:
        mm, qp = out
    _check(lib().ulp_boundary_minmax(_ptr(k), _ptr(q), _dtype_code(k), B, L, H, D, rc, world_size,
                                     _opt(used_sequence), q_group, _ptr(mm), _ptr(qp),
                                     _stream(k.device)))
    return mm, qp


def derive_k_boundary_amax(grouped_amax: torch.Tensor, gathered_minmax: torch.Tensor,
                           k_mean_global: torch.Tensor, *, rank: Optional[int],
                           local_sequence: int, world_size: int) -> torch.Tensor:
    """In place: the rank's first and last K group slots take the amax
    rebuilt from every touching rank's raw-K min/max (page
    "derive_k_boundary_amax")."""
    B, H, D = k_mean_global.shape
    _check(lib().ulp_derive_k_boundary_amax(_ptr(grouped_amax), _ptr(gathered_minmax),
                                            _ptr(k_mean_global), _dtype_code(k_mean_global), B, H,
                                            D, ULP_ALL_RANKS if rank is None else int(rank),
                                            local_sequence, world_size,
                                            _stream(grouped_amax.device)))
    return grouped_amax


def pack(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, k_mean_global: torch.Tensor,
         k_amax: torch.Tensor, gathered_q_partial: torch.Tensor, v_scale: torch.Tensor, *,
         rank: Optional[int], world_size: int, used_sequence: Optional[int] = None,
         q_group: int = GQ, fused: bool = True, send: Optional[torch.Tensor] = None,
         send_layout: int = SEND_SOURCE_MAJOR, gathered_minmax: Optional[torch.Tensor] = None,
         enable_pdl=None) -> torch.Tensor:
    """Quantise a rank's Q/K/V into its P chunks (INT8 Q/K, FP8 E4M3 V).

    With ``gathered_minmax`` (the [P, B, H, 2, 2, D] output of
    ``boundary_minmax``) the K boundary slots are derived inside the pack and
    written to ``k_amax`` (what ``derive_k_boundary_amax`` would write);
    without it they are read from ``k_amax``."""
    rc, nr, B, L, H, D = _rank_dims(q, rank)
    h = H // world_size
    cb = chunk_bytes(B, L, h, D, q_group)
    if send is None:
        if send_layout == SEND_DEST_MAJOR:
            shape = (world_size, world_size, cb)
        else:
            shape = ((nr,) if rank is None else ()) + (world_size, cb)
        send = torch.empty(shape, dtype=torch.uint8, device=q.device)
    _check(lib().ulp_pack(_ptr(q), _ptr(k), _ptr(v), _ptr(k_mean_global), _dtype_code(q),
                          _ptr(k_amax), _ptr(gathered_q_partial),
                          None if gathered_minmax is None else _ptr(gathered_minmax),
                          _ptr(v_scale), B, L, H, D, rc,
                          world_size, _opt(used_sequence), q_group, int(bool(fused)), _ptr(send),
                          int(send_layout), _pdl(enable_pdl), _stream(q.device)))
    return send


def alltoall_emulate(send: torch.Tensor, recv: Optional[torch.Tensor] = None) -> torch.Tensor:
    """recv[p][s] = send[s][p] over [P, P, chunk_bytes] buffers."""
    P, P2, cb = send.shape
    if recv is None:
        recv = torch.empty_like(send)
    _check(lib().ulp_alltoall_emulate(_ptr(send), _ptr(recv), P, cb, _stream(send.device)))
    return recv


def unpack_outputs(batch_size: int, local_sequence: int, local_heads: int, head_dim: int,
                   world_size: int, scale_sequence: Optional[int], device,
                   num_dests: Optional[int] = None, q_group: int = GQ):
    B, L, h, D, P = batch_size, local_sequence, local_heads, head_dim, world_size
    S = P * L
    Spad = (S + 63) // 64 * 64
    wq, wk = scale_widths(S if scale_sequence is None else scale_sequence, q_group)
    lead = () if num_dests is None else (num_dests,)
    return (torch.empty(lead + (B, S, h, D), dtype=torch.int8, device=device),
            torch.empty(lead + (B, S, h, D), dtype=torch.int8, device=device),
            torch.empty(lead + (B, D, h, Spad), dtype=torch.uint8, device=device),
            torch.empty(lead + (B, h, wq), dtype=torch.float32, device=device),
            torch.empty(lead + (B, h, wk), dtype=torch.float32, device=device))


def unpack_for_sage(recv_u8: torch.Tensor, *, batch_size: int, local_sequence: int,
                    local_heads: int, head_dim: int, world_size: int,
                    aligned: Optional[bool] = None, scale_sequence: Optional[int] = None,
                    q_group: int = GQ, out: Optional[Sequence[torch.Tensor]] = None,
                    enable_pdl: Optional[bool] = None):
    """Unpack source chunks onto the global grid (page "unpack_for_sage").

    recv_u8 [P, chunk_bytes] -> (q8, k8 [B, S, h, D] int8, v8 [B, D, h,
    ceil(S/64)*64] E4M3 bytes, q_scale, k_scale [B, h, width] fp32).
    recv_u8 [n, P, chunk_bytes] unpacks n destinations at once (outputs gain a
    leading n axis).  v8 is returned as uint8 bytes (E4M3 encoding); view it
    as torch.float8_e4m3fn where supported."""
    nd = None if recv_u8.dim() == 2 else recv_u8.shape[0]
    if out is None:
        out = unpack_outputs(batch_size, local_sequence, local_heads, head_dim, world_size,
                             scale_sequence, recv_u8.device, nd, q_group)
    q8, k8, v8, qs, ks = out
    v8b = v8.view(torch.uint8) if v8.dtype != torch.uint8 else v8
    _check(lib().ulp_unpack_for_sage(_ptr(recv_u8), batch_size, local_sequence, local_heads,
                                     head_dim, world_size, _tri(aligned), _opt(scale_sequence),
                                     q_group, _ptr(q8), _ptr(k8), _ptr(v8b), _ptr(qs), _ptr(ks),
                                     1 if nd is None else nd, _pdl(enable_pdl),
                                     _stream(recv_u8.device)))
    return tuple(out)


# ------------------------------------------------------------- the consumer

_OUT_CODES = {torch.float32: ULP_F32, torch.bfloat16: ULP_BF16, torch.float16: ULP_FP16}


def group_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, k_mean_global: torch.Tensor,
               v_scale: torch.Tensor, *, world_size: int, minmax: torch.Tensor,
               q_partial: torch.Tensor, k_amax: torch.Tensor, recv: torch.Tensor,
               out: Sequence[torch.Tensor], mode: int = 0, barrier: Optional[torch.Tensor] = None,
               used_sequence: Optional[int] = None, q_group: int = GQ,
               aligned: Optional[bool] = None, scale_sequence: Optional[int] = None,
               status: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, ...]:
    """One step of the whole emulated group from one call: ``boundary_minmax``
    (all ranks), ``pack`` fused, dest-major into ``recv`` (the derive folded
    in, or before it with STEP_DERIVE_SEPARATE), then ``unpack_for_sage`` of
    every destination into ``out`` (five tensors with a leading P axis, see
    ``unpack_outputs``).  q, k, v: stacked shards [P, B, L, H, D].
    ``mode``: 0 or STEP_DERIVE_SEPARATE | STEP_UNPACK_PDL bits for the
    separate launches; STEP_COOPERATIVE for one cooperative launch, which
    needs ``barrier`` (a 32-bit device tensor of two elements, zero before the
    first call; the kernel leaves it ready for the next one; zero it again
    after a non-zero ``status``)."""
    coop = bool(mode & STEP_COOPERATIVE)
    if coop and (barrier is None or barrier.numel() < 2 or barrier.dtype not in (torch.int32, torch.uint32)):
        raise ValueError("the cooperative launch needs barrier: a 32-bit tensor of at least two elements")
    P = world_size
    _, B, L, H, D = q.shape
    q8, k8, v8, qs, ks = out
    st = 0 if status is None else _ptr(status)
    bar = _ptr(barrier) if coop else None
    _check(lib().ulp_group_step(_ptr(q), _ptr(k), _ptr(v), _ptr(k_mean_global), _dtype_code(q),
                                _ptr(v_scale), B, L, H, D, P, _opt(used_sequence), q_group,
                                _tri(aligned), _opt(scale_sequence), _ptr(minmax), _ptr(q_partial),
                                _ptr(k_amax), _ptr(recv), _ptr(q8), _ptr(k8), _ptr(v8), _ptr(qs),
                                _ptr(ks), int(mode), bar, st, _stream(q.device)))
    return tuple(out)


def sage_attention(q8: torch.Tensor, k8: torch.Tensor, v8: torch.Tensor, q_scale: torch.Tensor,
                   k_scale: torch.Tensor, v_scale: torch.Tensor, *, n: Optional[int] = None,
                   q_group: int = GQ, sm_scale: Optional[float] = None,
                   out: Optional[torch.Tensor] = None, out_dtype: torch.dtype = torch.bfloat16,
                   workspace: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None, pv_fp8: bool = False) -> torch.Tensor:
    """Softmax attention over the unpacked tensors of one destination.

    q8, k8 [B, S, h, D] int8; v8 [B, D, h, Spad] E4M3 bytes (uint8 or
    float8_e4m3fn); q_scale [B, h, ceil(n/q_group)], k_scale [B, h,
    ceil(n/64)] fp32 (unpack_for_sage with scale_sequence=n gives exactly
    these); v_scale [B, h, D] fp32 (the caller's V scale of this
    destination's heads).  Attends over the live prefix of n rows (default S)
    and returns O [B, n, h, D] in out_dtype; sm_scale defaults to 1/sqrt(D).
    ``workspace``: optional uint8 device buffer of at least
    sage_attention_workspace_bytes(...) bytes (allocated when None).
    ``status``: optional int32 device tensor of one element, set non-zero by
    the kernel if a tensor-core product does not complete in time.
    ``pv_fp8``: the PV product in E4M3 (P rounded to E4M3, V read from v8
    as is) instead of fp16."""
    B, S, h, D = q8.shape
    n = S if n is None else int(n)
    if sm_scale is None:
        sm_scale = D ** -0.5
    if out is None:
        out = torch.empty((B, n, h, D), dtype=out_dtype, device=q8.device)
    if out.dtype not in _OUT_CODES:
        raise TypeError(f"out must be float32, bfloat16 or float16, got {out.dtype}")
    v8b = v8.view(torch.uint8) if v8.dtype != torch.uint8 else v8
    if workspace is None:
        workspace = torch.empty(sage_attention_workspace_bytes(B, S, h, D, n), dtype=torch.uint8,
                                device=q8.device)
    st = 0 if status is None else _ptr(status)
    _check(lib().ulp_sage_attention(_ptr(q8), _ptr(k8), _ptr(v8b), _ptr(q_scale), _ptr(k_scale),
                                    _ptr(v_scale), B, S, h, D, n, q_group, float(sm_scale),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _ptr(out), _OUT_CODES[out.dtype], PV_E4M3 if pv_fp8 else PV_F16, st,
                                    _stream(q8.device)))
    return out


def sage_attention_workspace_bytes(B: int, S: int, h: int, D: int, n: int) -> int:
    nb = _SZ()
    _check(lib().ulp_sage_attention_workspace_bytes(B, S, h, D, n, ctypes.byref(nb)))
    return nb.value
