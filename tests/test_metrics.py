"""The byte counts behind the bench's effective-bandwidth figures
(quantize_pack_gb300/metrics.py), pinned to values derived by hand from the
chunk layout and to the library's own geometry."""
import pytest

from quantize_pack_gb300 import configs, metrics, ulp
from oracle import oracle as O

# chunk_bytes = 3 B L h D + a16(4 B h slots(L, 128)) + a16(4 B h slots(L, 64)),
# worked out per workload by hand (Tiny: 3*1*96*4*64 = 73728, Q slots 2 ->
# 32 B, K slots 3 -> 48 B: 73808)
HAND_CHUNK_BYTES = {
    configs.TINY.name: 73_808,
    configs.PADDING.name: 1_536_416,
    configs.VIDEO_DIT.name: 9_439_488,
    configs.LONG_NONALIGNED.name: 17_975_664,
    configs.HEAVY_TAIL.name: 201_424_896,
}


@pytest.mark.parametrize("wl", configs.ALL, ids=[w.name for w in configs.ALL])
def test_chunk_bytes_agree_with_hand_values_library_and_oracle(wl):
    want = HAND_CHUNK_BYTES[wl.name]
    assert metrics.chunk_bytes(wl) == want
    assert ulp.chunk_bytes(wl.B, wl.L, wl.h, wl.D) == want
    assert O.chunk_layout(wl.B, wl.L, wl.h, wl.D)["chunk_bytes"] == want


@pytest.mark.parametrize("wl", configs.ALL, ids=[w.name for w in configs.ALL])
def test_step_bytes_are_fifteen_n_plus_scales_and_v_padding(wl):
    n = wl.N
    spad = (wl.S + 63) // 64 * 64
    scales = metrics.scale_section_bytes(wl) + 2 * metrics.out_scale_bytes(wl)
    assert metrics.pack_bytes(wl) == 9 * n + metrics.scale_section_bytes(wl)
    assert metrics.unpack_bytes(wl) == 5 * n + wl.B * wl.D * wl.H * spad + 2 * metrics.out_scale_bytes(wl)
    assert metrics.step_bytes(wl) == 14 * n + wl.B * wl.D * wl.H * spad + scales
    # the scale terms and the V tail are small beside the 15 N payload
    assert 15 * n <= metrics.step_bytes(wl) <= 15 * n * 1.001


def test_long_workload_step_is_5_75_gb():
    # 15 N = 15 * 383,385,600 = 5,750,784,000 bytes (the figure the bench
    # divides by, plus 846,720 bytes of scales)
    wl = configs.LONG_NONALIGNED
    assert wl.N == 383_385_600
    assert metrics.step_bytes(wl) == 5_751_630_720
