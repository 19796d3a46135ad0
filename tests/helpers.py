"""Shared test helpers: reduced workloads, brute-force global references.

The brute-force references here work on the unsharded global tensors with
numpy/torch library routines (float32 subtraction and division, numpy rint,
torch's float8_e4m3fn cast).  They know nothing of ranks, slots or chunks, so
they pin the oracle independently of its own loops.
"""
from __future__ import annotations

import numpy as np
import torch

from quantize_pack_gb300 import configs, synth

EPS = np.float32(1e-7)

# Geometry-preserving reductions of the five workloads (h = 1 head per
# destination, fewer rows) for the CPU suite, plus corner geometries.
TINY = configs.TINY
PADDING_R = configs.PADDING.replace(H=4, name="padding_h1")
VIDEO_R = configs.VIDEO_DIT.replace(H=8, L=256, name="video_dit_h1_L256")
LONG_R = configs.LONG_NONALIGNED.replace(H=8, L=585, name="long_nonaligned_h1_L585")
HEAVY_R = configs.HEAVY_TAIL.replace(H=2, L=1024, name="heavy_tail_h1_L1024")
# groups spanning four ranks; one group spanning all eight
SPAN4 = configs.Workload("span4_P8_L16", B=1, H=8, D=64, P=8, L=16, dtype=configs.BF16, seed=11,
                         k_mean_std=4.0, k_noise_std=0.05)
SPAN4_PAD = SPAN4.replace(pad_rows=37, scale_to_used=True, name="span4_P8_L16_used91")
L1 = configs.Workload("L1_P8", B=2, H=8, D=128, P=8, L=1, dtype=configs.FP16, seed=12,
                      k_mean_std=3.0, k_noise_std=0.1, pad_rows=3, scale_to_used=True)
# the partial live group crosses a rank boundary and the next rank's slice
# of it is padding only (used = 80, rows 64..127 span ranks 0 and 1)
CROSS_PAD = configs.Workload("cross_pad_P2_L96_used80", B=1, H=4, D=64, P=2, L=96,
                             dtype=configs.BF16, seed=13, pad_rows=112, scale_to_used=True,
                             k_mean_std=4.0, k_noise_std=0.05)
# world_size 6 (structurally supported), odd h with D = 64
SIX = configs.Workload("six_P6_L200_D64", B=2, H=18, D=64, P=6, L=200, dtype=configs.FP16,
                       seed=14, pad_rows=130, scale_to_used=True, k_mean_std=3.0,
                       k_noise_std=0.1)
# used a multiple of 64 (the partial group is fully live)
USED64 = configs.Workload("used_mult64_P4_L100", B=1, H=4, D=128, P=4, L=100, dtype=configs.BF16,
                          seed=15, pad_rows=16, scale_to_used=True, k_mean_std=2.0,
                          k_noise_std=0.2, outlier_frac=0.01)

# one live row; an odd batch with several heads per destination at D = 64
USED1 = configs.Workload("used1_P4_L50", B=1, H=8, D=64, P=4, L=50, dtype=configs.BF16, seed=16,
                         pad_rows=199, scale_to_used=True, k_mean_std=4.0, k_noise_std=0.05)
B3 = configs.Workload("b3_P2_L300_D64_fp16", B=3, H=6, D=64, P=2, L=300, dtype=configs.FP16,
                      seed=17, pad_rows=45, k_mean_std=3.0, k_noise_std=0.1, qv_dist="t3")

# the q_group = 64 variant (Q groups are the K groups) on the geometries with
# the most boundary cases: groups over 4 and 8 ranks, one-row shards, the
# partial live group across ranks, world_size 6, a ragged non-aligned shard
G64 = [w.replace(q_group=64, name=w.name + "_gq64") for w in (TINY, LONG_R, SPAN4_PAD, L1,
                                                              CROSS_PAD, SIX, B3)]

CPU_WORKLOADS = [TINY, PADDING_R, VIDEO_R, LONG_R, HEAVY_R, SPAN4, SPAN4_PAD, L1, CROSS_PAD, SIX,
                 USED64, USED1, B3] + G64


def f32(bits: np.ndarray, dtype: int) -> np.ndarray:
    return synth.from_bits(bits, dtype)


def touched_groups(r: int, L: int, G: int) -> list:
    """Brute force: distinct global groups holding some row of rank r."""
    return sorted({t // G for t in range(r * L, (r + 1) * L)})


def ranks_touching(g: int, L: int, P: int, G: int) -> list:
    return sorted({t // L for t in range(g * G, min(g * G + G, P * L))})


def global_k_amax(inp: synth.Inputs) -> np.ndarray:
    """Direct amax of |rn(K - m)| over each global 64-row group's live rows,
    floored at 1e-7 (the whole group at once, no ranks).  [B, H, ceil(S/64)];
    groups with no live row give 1e-7."""
    wl = inp.wl
    kf = f32(inp.k, wl.dtype)
    m = f32(inp.k_mean, wl.dtype)
    c = np.abs(kf - m[:, None, :, :])            # float32 subtraction: IEEE rn
    used = inp.used
    ng = (wl.S + 63) // 64
    out = np.full((wl.B, wl.H, ng), EPS, np.float32)
    for g in range(ng):
        hi = min(g * 64 + 64, used)
        if hi > g * 64:
            out[:, :, g] = np.maximum(c[:, g * 64:hi].max(axis=(1, 3)), EPS)
    return out


def global_q_amax(inp: synth.Inputs) -> np.ndarray:
    """max(1e-7, max |Q|) over each global G-row group, G = the workload's
    q_group.  [B, H, ceil(S/G)]."""
    wl = inp.wl
    G = wl.q_group
    qa = np.abs(f32(inp.q, wl.dtype))
    ng = (wl.S + G - 1) // G
    out = np.empty((wl.B, wl.H, ng), np.float32)
    for g in range(ng):
        out[:, :, g] = np.maximum(qa[:, g * G:g * G + G].max(axis=(1, 3)), EPS)
    return out


def int8_codes(x: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """clip(rint(rn(x / scale)), -128, 127) with numpy's float32 division."""
    y = (x.astype(np.float32) / scale.astype(np.float32)).astype(np.float32)
    return np.clip(np.rint(y), -128, 127).astype(np.int8)


def e4m3_codes(y: np.ndarray) -> np.ndarray:
    """torch's float8_e4m3fn cast (round to nearest even) after clamping to
    +-448, since torch's cast is not saturating."""
    t = torch.from_numpy(np.clip(y.astype(np.float32), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def run_oracle(inp: synth.Inputs, dests=None):
    from oracle import oracle as O
    wl = inp.wl
    return O.forward(inp.shards("q"), inp.shards("k"), inp.shards("v"), inp.k_mean, inp.v_scale,
                     wl.dtype, used_sequence=wl.used_sequence, scale_sequence=wl.scale_sequence,
                     dests=dests, q_group=wl.q_group)


_cache = {}


def cached(wl):
    """(inputs, oracle forward) for a workload, built once per session."""
    if wl.name not in _cache:
        inp = synth.make_inputs(wl)
        _cache[wl.name] = (inp, run_oracle(inp))
    return _cache[wl.name]
