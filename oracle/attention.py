"""CPU oracle of the attention that consumes the unpacked tensors.

TEST INFRASTRUCTURE ONLY: imported by tests/ and the smoke check, never by
the library; it imports nothing from the CUDA package.

Page "flashinfer.comm._ulysses_lowp.unpack_for_sage" hands its outputs to a
Sage-style attention kernel: INT8 Q/K [B, S, h, D] with FP32 per-group scales
[B, h, width] whose width is derived from the rows the kernel is given
(scale_widths(n) for a live prefix of n rows), FP8 E4M3 V [B, D, h, Spad], and
the V scale, which stays with the caller.  The pages print no formula for
the attention itself; this oracle takes the plainest reading:

  Q[b,t,j,:] = q8[b,t,j,:] * q_scale[b,j,t // G_Q]
  K[b,u,j,:] = k8[b,u,j,:] * k_scale[b,j,u // 64]      (K centred by the mean:
               softmax over u is unchanged by subtracting k_mean, since
               q . m is the same for every key)
  V[b,u,j,d] = e4m3(v8[b,d,j,u]) * v_scale[b,j,d]
  O[b,t,j,:] = sum_u softmax_u(sm_scale * Q[b,t,j,:] . K[b,u,j,:]) V[b,u,j,:]

over the live prefix t, u < n, without a causal mask, in float64.  The
exact definition, written out: no blocking, no online softmax.
"""
from __future__ import annotations

import numpy as np

from . import oracle as _orc

GK = 64


def e4m3_table() -> np.ndarray:
    """float64 value of every E4M3 byte (the oracle's own decoder); NaN codes
    stay NaN."""
    return np.array([_orc.e4m3_decode(c) for c in range(256)], np.float64)


def dequantize(q8, k8, v8, q_scale, k_scale, v_scale, *, n: int, q_group: int = 128):
    """Dequantised Q, K, V [B, n, h, D] in float64 over the live prefix n."""
    B, S, h, D = q8.shape
    rows = np.arange(n)
    qs = q_scale.astype(np.float64)[:, :, rows // q_group]          # [B, h, n]
    ks = k_scale.astype(np.float64)[:, :, rows // GK]
    Q = q8[:, :n].astype(np.float64) * qs.transpose(0, 2, 1)[..., None]
    K = k8[:, :n].astype(np.float64) * ks.transpose(0, 2, 1)[..., None]
    tab = e4m3_table()
    Vc = tab[v8[..., :n]]                                          # [B, D, h, n]
    V = Vc.transpose(0, 3, 2, 1) * v_scale.astype(np.float64)[:, None]   # [B, n, h, D]
    return Q, K, V


def sage_attention(q8, k8, v8, q_scale, k_scale, v_scale, *, n: int, q_group: int = 128,
                   sm_scale: float | None = None, rows=None) -> np.ndarray:
    """O [B, n, h, D] float64 (or [B, len(rows), h, D] for the query rows
    ``rows`` only, each row by the same definition).

    q8, k8: int8 [B, S, h, D]; v8: uint8 (E4M3 bytes) [B, D, h, Spad];
    q_scale: [B, h, >= ceil(n/q_group)], k_scale: [B, h, >= ceil(n/64)] fp32;
    v_scale: [B, h, D] fp32 (the destination's heads); n: live rows;
    sm_scale defaults to 1/sqrt(D)."""
    B, S, h, D = q8.shape
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    Q, K, V = dequantize(q8, k8, v8, q_scale, k_scale, v_scale, n=n, q_group=q_group)
    if rows is not None:
        Q = Q[:, np.asarray(rows)]
    O = np.empty((B, Q.shape[1], h, D), np.float64)
    for b in range(B):
        for j in range(h):
            s = sm_scale * (Q[b, :, j] @ K[b, :, j].T)             # [queries, n]
            s -= s.max(axis=1, keepdims=True)
            p = np.exp(s)
            O[b, :, j] = (p @ V[b, :, j]) / p.sum(axis=1, keepdims=True)
    return O
