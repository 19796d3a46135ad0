"""UlyssesLowpPath's launch plan, without a GPU: which launches a step makes
for each configuration (the size-based defaults and the explicit options),
and the combinations it rejects.  The path's buffers live on the CPU here;
nothing is launched."""
import pytest
import torch

from quantize_pack_gb300 import configs, ulp
from quantize_pack_gb300.path import FOLD_BELOW_BYTES, UlyssesLowpPath


def make(wl, **kw):
    dt = torch.bfloat16 if wl.dtype == configs.BF16 else torch.float16
    return UlyssesLowpPath(B=wl.B, L=wl.L, H=wl.H, D=wl.D, world_size=wl.P, dtype=dt,
                           used_sequence=wl.used_sequence, scale_sequence=wl.scale_sequence,
                           q_group=wl.q_group, device="cpu", **kw)


def test_launch_bound_threshold_is_the_input_size():
    for wl in configs.ALL:
        launch_bound = 6 * wl.P * wl.B * wl.L * wl.H * wl.D < FOLD_BELOW_BYTES
        p = make(wl)
        assert p.fold_derive == launch_bound and p.pdl == launch_bound, wl.name
        assert p.launches_per_step == (3 if launch_bound else 4), wl.name
        assert not p.single_launch and p.barrier is None and p.status is None


def test_explicit_options_and_launch_counts():
    wl = configs.TINY
    assert make(wl, fold_derive=False).launches_per_step == 4
    assert make(wl, fused=False).launches_per_step == 4             # + k_grouped_amax
    assert make(wl, fold_exchange=False).launches_per_step == 4     # + the all-to-all copy
    assert make(wl, fused=False, fold_exchange=False, fold_derive=False).launches_per_step == 6
    p = make(wl, single_launch=True)
    assert p.launches_per_step == 1 and p.fold_derive
    assert p.barrier.tolist() == [0, 0] and p.status.tolist() == [0]
    # a large workload may ask for the single launch too (the derive folds)
    big = make(configs.VIDEO_DIT.replace(L=256, name="vd_small_rows"), fold_derive=None, single_launch=True)
    assert big.fold_derive and big.launches_per_step == 1


@pytest.mark.parametrize("kw", [dict(fused=False), dict(fold_exchange=False), dict(fold_derive=False)])
def test_single_launch_needs_the_fused_folded_step(kw):
    with pytest.raises(ValueError, match="single_launch"):
        make(configs.TINY, single_launch=True, **kw)


def test_group_step_cooperative_needs_a_barrier():
    wl = configs.TINY
    p = make(wl)
    t = torch.zeros(1)
    with pytest.raises(ValueError, match="barrier"):
        ulp.group_step(t, t, t, t, t, world_size=wl.P, minmax=t, q_partial=t, k_amax=t, recv=t,
                       out=(t, t, t, t, t), mode=ulp.STEP_COOPERATIVE)
    with pytest.raises(ValueError, match="barrier"):
        ulp.group_step(t, t, t, t, t, world_size=wl.P, minmax=t, q_partial=t, k_amax=t, recv=t,
                       out=(t, t, t, t, t), mode=ulp.STEP_COOPERATIVE, barrier=torch.zeros(1, dtype=torch.int32))
    assert p.check_status() is None          # nothing to check without the single launch
