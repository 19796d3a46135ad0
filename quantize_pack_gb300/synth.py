"""Seeded synthetic inputs for the Ulysses low-precision quantize/pack path.

Serves both the CUDA path and the CPU oracle; it holds none of the method's
arithmetic (no amax, no scales of the path, no quantisation).  What it builds
is what a caller hands the path:

* Q, K, V on the global grid ``[B, S, H, D]`` as raw 16-bit patterns (bf16 or
  fp16), and the per-rank shards ``[P, B, L, H, D]`` cut from them;
* ``k_mean_global`` ``[B, H, D]``: the page "k_grouped_amax" (Parameters) says
  the caller passes the global K mean rounded to the input dtype.  Here it is
  the fp64 mean of the live rows ``[0, used)``, rounded to fp32, then to the
  dtype;
* ``v_scale`` ``[B, H, D]`` fp32: the page "unpack_for_sage" (Returns) leaves
  the V scale with the caller.  Here it is the per-(batch, head, channel)
  absolute maximum of V over the whole sequence (at least 1e-7) divided by
  448, the largest finite E4M3 magnitude.

Draw order (PCG64 ``default_rng(seed)``, float32 draws unless Student-t):
Q; K channel means ``[H, D]`` (shared over the batch); K deviations
``[B, S, H, D]``; V; then, when the workload has outliers, one uniform mask per
tensor for Q, K, V in that order, multiplying the selected entries by the
outlier factor.  Then the dtype cast (round to nearest even), the zero fill of
padding rows ``[used, S)``, then ``k_mean_global`` and ``v_scale``.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

from .configs import BF16, FP16, Workload


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return b.view(np.float16).astype(np.float32)


def to_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    return f32_to_bf16_bits(x) if dtype == BF16 else f32_to_f16_bits(x)


def from_bits(b: np.ndarray, dtype: int) -> np.ndarray:
    return bf16_bits_to_f32(b) if dtype == BF16 else f16_bits_to_f32(b)


@dataclasses.dataclass
class Inputs:
    wl: Workload
    q: np.ndarray          # uint16 [B, S, H, D]
    k: np.ndarray          # uint16 [B, S, H, D]
    v: np.ndarray          # uint16 [B, S, H, D]
    k_mean: np.ndarray     # uint16 [B, H, D]
    v_scale: np.ndarray    # float32 [B, H, D]

    @property
    def used(self) -> int:
        u = self.wl.used_sequence
        return self.wl.S if u is None else u

    def shards(self, name: str) -> np.ndarray:
        """Per-rank shards [P, B, L, H, D] (contiguous) of q, k or v."""
        return shard(getattr(self, name), self.wl.P)


def shard(x: np.ndarray, P: int) -> np.ndarray:
    B, S, H, D = x.shape
    L = S // P
    return np.ascontiguousarray(x.reshape(B, P, L, H, D).transpose(1, 0, 2, 3, 4))


def _draw(rng: np.random.Generator, dist: str, shape) -> np.ndarray:
    if dist == "normal":
        return rng.standard_normal(shape, dtype=np.float32)
    if dist == "t3":
        return rng.standard_t(3.0, shape).astype(np.float32)
    raise ValueError(dist)


def make_inputs(wl: Workload) -> Inputs:
    rng = np.random.default_rng(wl.seed)
    B, S, H, D = wl.B, wl.S, wl.H, wl.D
    shape = (B, S, H, D)

    q = _draw(rng, wl.qv_dist, shape)
    mu = rng.standard_normal((H, D), dtype=np.float32) * np.float32(wl.k_mean_std)
    kn = _draw(rng, wl.k_noise_dist, shape)
    kn *= np.float32(wl.k_noise_std)
    k = kn
    k += mu[None, None, :, :]
    del kn
    v = _draw(rng, wl.qv_dist, shape)
    if wl.outlier_frac > 0.0:
        for x in (q, k, v):
            m = rng.random(shape, dtype=np.float32) < np.float32(wl.outlier_frac)
            x[m] *= np.float32(wl.outlier_mult)
            del m

    qb = to_bits(q, wl.dtype); del q
    kb = to_bits(k, wl.dtype); del k
    vb = to_bits(v, wl.dtype); del v

    used = S if wl.used_sequence is None else wl.used_sequence
    if used < S:
        qb[:, used:] = 0
        kb[:, used:] = 0
        vb[:, used:] = 0

    kf = from_bits(kb[:, :used], wl.dtype)
    kmean64 = kf.mean(axis=1, dtype=np.float64)           # [B, H, D]
    del kf
    k_mean = to_bits(kmean64.astype(np.float32), wl.dtype)

    vabs = np.abs(from_bits(vb, wl.dtype)).max(axis=1)     # [B, H, D] float32
    v_scale = np.maximum(vabs, np.float32(1e-7)) / np.float32(448.0)
    v_scale = v_scale.astype(np.float32)

    return Inputs(wl=wl, q=qb, k=kb, v=vb, k_mean=np.ascontiguousarray(k_mean),
                  v_scale=np.ascontiguousarray(v_scale))


@dataclasses.dataclass
class AttentionOperands:
    """Quantised operands of the attention consumer, as unpack_for_sage
    returns them for one destination, plus the caller's V scale."""
    q8: np.ndarray        # int8 [B, S, h, D]
    k8: np.ndarray        # int8 [B, S, h, D]
    v8: np.ndarray        # uint8 E4M3 bytes [B, D, h, Spad]
    q_scale: np.ndarray   # fp32 [B, h, ceil(n / q_group)]
    k_scale: np.ndarray   # fp32 [B, h, ceil(n / 64)]
    v_scale: np.ndarray   # fp32 [B, h, D]
    n: int
    q_group: int


def attention_operands(seed: int, *, B: int, S: int, h: int, D: int, n: Optional[int] = None,
                       q_group: int = 128, spread: float = 1.0) -> AttentionOperands:
    """Seeded random codes and scales (PCG64 ``default_rng(seed)``, draws in
    this order): Q and K codes uniform in [-127, 127]; V bytes uniform over
    the finite E4M3 codes (the NaN codes 0x7F/0xFF are replaced by 0x3C, and
    the tail [S, Spad) is zero); Q and K scales uniform in
    [0.5, 2] * spread / (127 * 8) per group; V scales uniform in
    [0.01, 0.05] per channel.  ``spread`` widens the logits (peakier
    softmax).  Rows [n, S) of Q and K and keys [n, S) of V get extreme codes
    (+-127, 0x7E), which a consumer of the live prefix must ignore."""
    rng = np.random.default_rng(seed)
    n = S if n is None else n
    Spad = (S + 63) // 64 * 64
    q8 = rng.integers(-127, 128, size=(B, S, h, D), dtype=np.int8)
    k8 = rng.integers(-127, 128, size=(B, S, h, D), dtype=np.int8)
    v8 = rng.integers(0, 256, size=(B, D, h, Spad)).astype(np.uint8)
    v8[(v8 & 0x7F) == 0x7F] = 0x3C
    v8[..., S:] = 0
    wq, wk = (n + q_group - 1) // q_group, (n + 63) // 64
    qs = (spread * rng.uniform(0.5, 2.0, size=(B, h, wq)) / 127 / 8).astype(np.float32)
    ks = (spread * rng.uniform(0.5, 2.0, size=(B, h, wk)) / 127 / 8).astype(np.float32)
    vs = rng.uniform(0.01, 0.05, size=(B, h, D)).astype(np.float32)
    q8[:, n:] = 127
    k8[:, n:] = -127
    v8[..., n:S] = 0x7E
    return AttentionOperands(q8, k8, v8, qs, ks, vs, n, q_group)


def attention_operands_paired(seed: int, *, S: int, h: int, D: int, n: int, q_group: int = 128,
                              logit: float = 40.0) -> AttentionOperands:
    """Structured, peaky operands for one batch (B = 1): every query tile i
    (128 rows) has two dominant keys with identical codes, one in key tile
    i and one in key tile i + 1 (mod the tile count), so its softmax splits
    its weight about evenly between two values; a key tile that is dropped
    or counted twice moves those rows by a large fraction of max |V|.

    PCG64 ``default_rng(seed)``, draws in this order: one sign pattern
    p_i in {-127, 127}^D per query tile and head; Q rows = p_i plus integer
    noise in [-8, 8] (clipped to [-127, 127]); K codes uniform in [-24, 24];
    the dominant keys' places (uniform in the first half of a key tile's live
    rows for its own query tile, in the second half for the previous one); V
    bytes uniform over the finite E4M3 codes.  Q and K scales are one constant each, chosen so the
    dominant logits are about ``logit`` (natural units, 1/sqrt(D) softmax
    scale); V scales uniform in [0.01, 0.05].  Rows past n are set as in
    attention_operands."""
    rng = np.random.default_rng(seed)
    T = (n + 127) // 128                                   # tiles over the live prefix
    Spad = (S + 63) // 64 * 64
    pat = np.where(rng.integers(0, 2, size=(T, h, D)) == 1, 127, -127).astype(np.int32)
    q = np.repeat(pat, 128, axis=0)[:S]
    if q.shape[0] < S:
        q = np.concatenate([q, np.zeros((S - q.shape[0], h, D), np.int32)])
    q = np.clip(q + rng.integers(-8, 9, size=(S, h, D)), -127, 127)
    k = rng.integers(-24, 25, size=(S, h, D)).astype(np.int32)
    # key tile t holds query tile t's key in its first half and query tile
    # t - 1's in its second half (of its live rows), so no two collide
    u = rng.uniform(0.0, 1.0, size=(T, 2))
    for i in range(T):
        for which, t in ((0, i), (1, (i + 1) % T)):
            r = min(128, n - 128 * t)
            half = r // 2
            off = int(u[i, which] * half) if which == 0 else half + int(u[i, which] * (r - half))
            k[t * 128 + off] = pat[i]
    v8 = rng.integers(0, 256, size=(1, D, h, Spad)).astype(np.uint8)
    v8[(v8 & 0x7F) == 0x7F] = 0x3C
    v8[..., S:] = 0
    wq, wk = (n + q_group - 1) // q_group, (n + 63) // 64
    # logit = qs * ks * (127^2 D) / sqrt(D) for a dominant key
    qk = logit * np.sqrt(D) / (127.0 * 127.0 * D)
    qs = np.full((1, h, wq), np.sqrt(qk), np.float32)
    ks = np.full((1, h, wk), np.float32(qk) / qs[0, 0, 0], np.float32)
    vs = rng.uniform(0.01, 0.05, size=(1, h, D)).astype(np.float32)
    q8 = q.astype(np.int8)[None]
    k8 = k.astype(np.int8)[None]
    q8[:, n:] = 127
    k8[:, n:] = -127
    v8[..., n:S] = 0x7E
    return AttentionOperands(np.ascontiguousarray(q8), np.ascontiguousarray(k8), v8, qs, ks, vs, n, q_group)

