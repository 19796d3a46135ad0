"""numpy front end of the C oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
bench's CPU-baseline leg, never by the library.  It imports nothing from the
CUDA package.  ``build()`` compiles oracle.c with gcc into ``_build/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")
SOURCES = [os.path.join(HERE, "oracle.c")]
HEADERS = [os.path.join(HERE, "oracle.h")]

GK = 64
GQ = 128       # default Q group rows; 64 selects the variant whose Q groups are the K groups

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (strict IEEE binary32: no contraction, no fast-math)."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    newest = max(os.path.getmtime(p) for p in SOURCES + HEADERS)
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < newest:
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", *SOURCES, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


def build_variant(source: str, path: str) -> str:
    """Compile an edited copy of oracle.c (the mutation tests plant mistakes
    in copies to check that the pins catch them) into `path`."""
    d = os.path.dirname(path)
    os.makedirs(d, exist_ok=True)
    src = os.path.join(d, "oracle_variant.c")
    with open(src, "w") as f:
        f.write(source)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-I", HERE, src, "-o", path, "-lm"], check=True)
    return path


class use_library:
    """Context manager: route every oracle call through another build of it."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = _lib
        _lib = ctypes.CDLL(self.path)
        _declare(_lib)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


def _declare(L):
    L.orc_bf16_to_f32.restype = ctypes.c_float
    L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_f16_to_f32.restype = ctypes.c_float
    L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_int8_code.restype = ctypes.c_int8
    L.orc_int8_code.argtypes = [ctypes.c_float]
    L.orc_e4m3.restype = ctypes.c_uint8
    L.orc_e4m3.argtypes = [ctypes.c_float]
    L.orc_e4m3_decode.restype = ctypes.c_float
    L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.orc_slots.restype = _I
    L.orc_slots.argtypes = [_I, _I]
    L.orc_chunk_layout.restype = None
    L.orc_chunk_layout.argtypes = [_I, _I, _I, _I, _I] + [ctypes.POINTER(_SZ)] * 6
    L.orc_scale_widths.restype = None
    L.orc_scale_widths.argtypes = [_I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]
    L.orc_k_mean_global.restype = None
    L.orc_k_mean_global.argtypes = [_P, _I, _I, _I, _I, _I, _I, _I, _P]
    L.orc_k_grouped_amax.restype = None
    L.orc_k_grouped_amax.argtypes = [_P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P]
    L.orc_boundary_minmax.restype = None
    L.orc_boundary_minmax.argtypes = [_P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P]
    L.orc_derive_k_boundary_amax.restype = None
    L.orc_derive_k_boundary_amax.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I]
    L.orc_pack.restype = None
    L.orc_pack.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]
    L.orc_alltoall.restype = None
    L.orc_alltoall.argtypes = [_P, _P, _I, _SZ]
    L.orc_unpack_for_sage.restype = None
    L.orc_unpack_for_sage.argtypes = [_P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]


def _ptr(a: np.ndarray, dtype) -> int:
    assert a.dtype == dtype, (a.dtype, dtype)
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _opt(x: Optional[int]) -> int:
    return -1 if x is None else int(x)


# ------------------------------------------------------------------ numbers

def bf16_to_f32(bits: int) -> float:
    return lib().orc_bf16_to_f32(bits)


def f16_to_f32(bits: int) -> float:
    return lib().orc_f16_to_f32(bits)


def int8_code(y: float) -> int:
    return lib().orc_int8_code(y)


def e4m3(x: float) -> int:
    return lib().orc_e4m3(x)


def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(code)


# ----------------------------------------------------------------- geometry

def slots(L: int, G: int) -> int:
    return lib().orc_slots(L, G)


def chunk_layout(B: int, L: int, h: int, D: int, q_group: int = GQ) -> dict:
    v = [_SZ() for _ in range(6)]
    lib().orc_chunk_layout(B, L, h, D, q_group, *[ctypes.byref(x) for x in v])
    keys = ["q", "k", "v", "q_scale", "k_scale", "chunk_bytes"]
    return {k: int(x.value) for k, x in zip(keys, v)}


def scale_widths(n: int, q_group: int = GQ) -> tuple:
    q, k = _I(), _I()
    lib().orc_scale_widths(n, q_group, ctypes.byref(q), ctypes.byref(k))
    return q.value, k.value


# ------------------------------------------------------------ path functions

def k_mean_global(k_all, dtype, *, used_sequence=None):
    """k_all: uint16 [P, B, L, H, D] -> uint16 [B, H, D] (dtype bits)."""
    P, B, L, H, D = k_all.shape
    out = np.empty((B, H, D), np.uint16)
    lib().orc_k_mean_global(_ptr(k_all, np.uint16), dtype, B, L, H, D, P, _opt(used_sequence),
                            _ptr(out, np.uint16))
    return out


def k_grouped_amax(k, k_mean, dtype, *, rank, world_size, used_sequence=None):
    """k: uint16 [B, L, H, D]; k_mean uint16 [B, H, D] -> float32 [B, H, slots(L,64)]."""
    B, L, H, D = k.shape
    out = np.empty((B, H, slots(L, GK)), np.float32)
    lib().orc_k_grouped_amax(_ptr(k, np.uint16), _ptr(k_mean, np.uint16), dtype, B, L, H, D,
                             rank, world_size, _opt(used_sequence), _ptr(out, np.float32))
    return out


def boundary_minmax(k, q, dtype, *, rank, world_size, used_sequence=None, q_group=GQ):
    """-> (minmax float32 [B, H, 2, 2, D], qb float32 [B, H, 2]) of one rank."""
    B, L, H, D = k.shape
    mm = np.empty((B, H, 2, 2, D), np.float32)
    qb = np.empty((B, H, 2), np.float32)
    lib().orc_boundary_minmax(_ptr(k, np.uint16), _ptr(q, np.uint16), dtype, B, L, H, D, rank,
                              world_size, _opt(used_sequence), q_group, _ptr(mm, np.float32),
                              _ptr(qb, np.float32))
    return mm, qb


def derive_k_boundary_amax(grouped_amax, gathered_minmax, k_mean, dtype, *, rank,
                           local_sequence, world_size):
    """Updates grouped_amax ([B, H, slots]) in place and returns it."""
    B, H, _ = grouped_amax.shape
    D = gathered_minmax.shape[-1]
    lib().orc_derive_k_boundary_amax(_ptr(grouped_amax, np.float32),
                                     _ptr(gathered_minmax, np.float32),
                                     _ptr(k_mean, np.uint16), dtype, B, H, D, rank,
                                     local_sequence, world_size)
    return grouped_amax


def pack(q, k, v, k_mean, dtype, k_amax, gathered_qb, v_scale, *, rank, world_size, q_group=GQ):
    """One rank's send buffer uint8 [P, chunk_bytes]."""
    B, L, H, D = q.shape
    h = H // world_size
    cb = chunk_layout(B, L, h, D, q_group)["chunk_bytes"]
    send = np.zeros((world_size, cb), np.uint8)
    lib().orc_pack(_ptr(q, np.uint16), _ptr(k, np.uint16), _ptr(v, np.uint16),
                   _ptr(k_mean, np.uint16), dtype, _ptr(k_amax, np.float32),
                   _ptr(gathered_qb, np.float32), _ptr(v_scale, np.float32), B, L, H, D, rank,
                   world_size, q_group, _ptr(send, np.uint8))
    return send


def alltoall(send_all):
    """send_all [P, P, chunk] (source-major) -> recv_all [P, P, chunk] (dest-major)."""
    P, P2, cb = send_all.shape
    recv = np.empty_like(send_all)
    lib().orc_alltoall(_ptr(send_all, np.uint8), _ptr(recv, np.uint8), P, cb)
    return recv


def unpack_for_sage(recv_u8, *, batch_size, local_sequence, local_heads, head_dim, world_size,
                    scale_sequence=None, q_group=GQ):
    B, L, h, D, P = batch_size, local_sequence, local_heads, head_dim, world_size
    S = P * L
    Spad = (S + 63) // 64 * 64
    wq, wk = scale_widths(S if scale_sequence is None else scale_sequence, q_group)
    q8 = np.empty((B, S, h, D), np.int8)
    k8 = np.empty((B, S, h, D), np.int8)
    v8 = np.empty((B, D, h, Spad), np.uint8)
    qs = np.empty((B, h, wq), np.float32)
    ks = np.empty((B, h, wk), np.float32)
    lib().orc_unpack_for_sage(_ptr(recv_u8, np.uint8), B, L, h, D, P, _opt(scale_sequence), q_group,
                              _ptr(q8, np.int8), _ptr(k8, np.int8), _ptr(v8, np.uint8),
                              _ptr(qs, np.float32), _ptr(ks, np.float32))
    return q8, k8, v8, qs, ks


# -------------------------------------------------- the whole emulated path

def forward(q_sh, k_sh, v_sh, k_mean, v_scale, dtype, *, used_sequence=None,
            scale_sequence=None, ranks=None, dests=None, q_group=GQ):
    """Every step of the path for an emulated Ulysses group of P ranks.

    q_sh, k_sh, v_sh: uint16 [P, B, L, H, D] shards.  Returns a dict with the
    per-rank kernel amax (before derive), minmax, qb, derived amax, the send
    buffers [P, P, chunk], the receive buffers [P, P, chunk] and the per-dest
    outputs (q8, k8, v8, q_scale, k_scale).  ``dests`` limits the unpack to
    some destinations (the sends of all ranks are always built).
    """
    P, B, L, H, D = q_sh.shape
    h = H // P
    ga0 = np.stack([k_grouped_amax(k_sh[r], k_mean, dtype, rank=r, world_size=P,
                                   used_sequence=used_sequence) for r in range(P)])
    mm, qb = zip(*[boundary_minmax(k_sh[r], q_sh[r], dtype, rank=r, world_size=P,
                                   used_sequence=used_sequence, q_group=q_group)
                   for r in range(P)])
    gathered = np.ascontiguousarray(np.stack(mm))
    gathered_qb = np.ascontiguousarray(np.stack(qb))
    ga = ga0.copy()
    for r in range(P):
        derive_k_boundary_amax(ga[r], gathered, k_mean, dtype, rank=r, local_sequence=L,
                               world_size=P)
    send = np.stack([pack(q_sh[r], k_sh[r], v_sh[r], k_mean, dtype, np.ascontiguousarray(ga[r]),
                          gathered_qb, v_scale, rank=r, world_size=P, q_group=q_group)
                     for r in range(P)])
    recv = alltoall(send)
    outs = {}
    for p in (range(P) if dests is None else dests):
        outs[p] = unpack_for_sage(np.ascontiguousarray(recv[p]), batch_size=B, local_sequence=L,
                                  local_heads=h, head_dim=D, world_size=P,
                                  scale_sequence=scale_sequence, q_group=q_group)
    return {"amax_kernel": ga0, "minmax": gathered, "qb": gathered_qb, "amax": ga,
            "send": send, "recv": recv, "out": outs}
