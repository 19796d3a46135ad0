"""Algorithmic byte counts of the path (what one pass must move at least),
used for effective-bandwidth figures.

N = B*S*H*D elements per tensor over all ranks.  One pass over every rank of
the emulated group reads Q, K, V once (2 bytes each), writes the packed
chunks (Q, K, V bytes + the scale sections), reads them back in the
receivers, and writes q8, k8, v8 (V padded to ceil(S/64)*64 rows) and the
consumer scales.  The emulated exchange and the boundary re-reads of at most
two groups per rank are not counted: the first is not part of the path on a
real Ulysses group, the second is a cost of the design.
"""
from __future__ import annotations

from .configs import Workload


def _slots(L: int, G: int) -> int:
    return (L + G - 1) // G + (L % G != 0)


def _a16(x: int) -> int:
    return (x + 15) // 16 * 16


def chunk_bytes(wl: Workload) -> int:
    n = wl.B * wl.L * wl.h * wl.D
    return (3 * _a16(n) + _a16(4 * wl.B * wl.h * _slots(wl.L, wl.q_group))
            + _a16(4 * wl.B * wl.h * _slots(wl.L, 64)))


def scale_section_bytes(wl: Workload) -> int:
    """Scale bytes of all P*P chunks."""
    return wl.P * wl.P * 4 * wl.B * wl.h * (_slots(wl.L, wl.q_group) + _slots(wl.L, 64))


def out_scale_bytes(wl: Workload) -> int:
    n = wl.S if wl.scale_sequence is None else wl.scale_sequence
    G = wl.q_group
    return wl.P * 4 * wl.B * wl.h * ((n + G - 1) // G + (n + 63) // 64)


def pack_bytes(wl: Workload) -> int:
    """Pack kernel: read Q, K, V; write codes and chunk scales."""
    return 6 * wl.N + 3 * wl.N + scale_section_bytes(wl)


def unpack_bytes(wl: Workload) -> int:
    """Unpack kernel: read codes and the scales used; write q8, k8, padded v8, scales."""
    spad = (wl.S + 63) // 64 * 64
    v_out = wl.B * wl.D * wl.H * spad
    return 3 * wl.N + 2 * wl.N + v_out + 2 * out_scale_bytes(wl)


def step_bytes(wl: Workload) -> int:
    """One pass of the whole path over every rank (~15 N)."""
    return pack_bytes(wl) + unpack_bytes(wl)


def input_bytes(wl: Workload) -> int:
    """Host -> device bytes of one step's inputs: Q, K, V, k_mean, v_scale."""
    return 6 * wl.N + 2 * wl.B * wl.H * wl.D + 4 * wl.B * wl.H * wl.D


def output_bytes(wl: Workload) -> int:
    """Device -> host bytes of one step's outputs: q8, k8, v8, scales of every destination."""
    spad = (wl.S + 63) // 64 * 64
    return 2 * wl.N + wl.B * wl.D * wl.H * spad + out_scale_bytes(wl)
