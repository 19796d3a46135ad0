"""The five synthetic workloads of the Ulysses low-precision quantize/pack path.

Each workload fixes the shapes (B, H, D, Ulysses group size P, rows per shard L),
the input dtype, the padding (``used_sequence``) and the consumer scale width
(``scale_sequence``), plus the value distributions the seeded generator draws
(``quantize_pack_gb300.synth``).  Argument meaning follows the pages
"flashinfer.comm._ulysses_lowp.k_grouped_amax" (Parameters) and
"flashinfer.comm._ulysses_lowp.unpack_for_sage" (Parameters).

This module holds shapes and distribution parameters only: no arithmetic of
the method.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

BF16 = 0
FP16 = 1
DTYPE_NAMES = {BF16: "bf16", FP16: "fp16"}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    D: int
    P: int
    L: int
    dtype: int
    seed: int
    # rows [S - pad_rows, S) of Q/K/V are zero-filled and used_sequence = S - pad_rows
    pad_rows: int = 0
    # scale_sequence handed to unpack: None, or "used" (= used_sequence)
    scale_to_used: bool = False
    aligned: Optional[bool] = None
    # Q group rows: 128, or 64 (the variant whose Q groups are the K groups)
    q_group: int = 128
    # value recipe
    qv_dist: str = "normal"          # "normal" (N(0,1)) or "t3" (Student-t, nu=3)
    k_mean_std: float = 1.0          # std of the per-(head, channel) K mean
    k_noise_std: float = 0.1         # scale of the K deviation
    k_noise_dist: str = "normal"     # "normal" or "t3"
    outlier_frac: float = 0.0        # fraction of Q/K/V entries multiplied by outlier_mult
    outlier_mult: float = 20.0

    @property
    def S(self) -> int:
        return self.P * self.L

    @property
    def h(self) -> int:
        return self.H // self.P

    @property
    def used_sequence(self) -> Optional[int]:
        return None if self.pad_rows == 0 else self.S - self.pad_rows

    @property
    def scale_sequence(self) -> Optional[int]:
        return self.used_sequence if self.scale_to_used else None

    @property
    def N(self) -> int:
        """Elements per tensor over all ranks: B*S*H*D."""
        return self.B * self.S * self.H * self.D

    @property
    def tokens(self) -> int:
        return self.B * self.S

    def with_L(self, L: int, name: Optional[str] = None) -> "Workload":
        """Same recipe at a different shard length (pad rows kept when they fit)."""
        pad = self.pad_rows if self.pad_rows < self.P * L else 0
        return dataclasses.replace(self, L=L, pad_rows=pad,
                                   name=name or f"{self.name}@L{L}",
                                   aligned=(self.aligned if L % 128 == 0 else None))

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def describe(self) -> dict:
        return {
            "workload": self.name, "B": self.B, "H": self.H, "h": self.h,
            "D": self.D, "P": self.P, "L": self.L, "S": self.S,
            "dtype": DTYPE_NAMES[self.dtype],
            "used_sequence": self.used_sequence,
            "scale_sequence": self.scale_sequence,
            "aligned": self.aligned,
            "q_group": self.q_group,
        }


TINY = Workload("tiny_B1_H8_D64_P2_L96_bf16", B=1, H=8, D=64, P=2, L=96, dtype=BF16, seed=0,
                k_mean_std=4.0, k_noise_std=0.05)
PADDING = Workload("padding_B1_H16_D128_P4_L1000_fp16_used3900", B=1, H=16, D=128, P=4, L=1000,
                   dtype=FP16, seed=1, pad_rows=100, scale_to_used=True,
                   k_mean_std=3.0, k_noise_std=0.1)
VIDEO_DIT = Workload("video_dit_aligned_B2_H24_D128_P8_L4096_bf16", B=2, H=24, D=128, P=8, L=4096,
                     dtype=BF16, seed=2, aligned=True, k_mean_std=2.0, k_noise_std=0.2)
LONG_NONALIGNED = Workload("long_nonaligned_B1_H40_D128_P8_L9360_bf16_used74800", B=1, H=40, D=128,
                           P=8, L=9360, dtype=BF16, seed=3, pad_rows=80, scale_to_used=True,
                           k_mean_std=2.0, k_noise_std=0.2, outlier_frac=1e-3)
HEAVY_TAIL = Workload("heavy_tail_B4_H32_D64_P2_L16384_fp16", B=4, H=32, D=64, P=2, L=16384,
                      dtype=FP16, seed=4, aligned=True, qv_dist="t3", k_mean_std=4.0,
                      k_noise_std=0.05, k_noise_dist="t3")

ALL = [TINY, PADDING, VIDEO_DIT, LONG_NONALIGNED, HEAVY_TAIL]
BY_NAME = {w.name: w for w in ALL}
# The workload the throughput headline is quoted on: the largest, non-aligned one.
HEADLINE = LONG_NONALIGNED
