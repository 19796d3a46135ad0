"""GPU parity of the quantisation codecs on adversarial inputs.

The kernels take the int8 and E4M3 codes from a reciprocal multiply and fall
back to the IEEE quotient near rounding boundaries.  These inputs aim at that
decision: groups whose values are random 16-bit patterns below a chosen amax
(many scales, every binade), groups with power-of-two scales where x / s
lands exactly on half-integers (round-half-even ties), V values on E4M3
midpoints, and V scales spanning 2^-30..2^30 so that quotients are zero,
E4M3-subnormal, normal and saturating.  Everything goes through the public
path and is compared bit for bit with the oracle.
"""
import numpy as np
import pytest
import torch

import gpu_helpers as gh
import helpers as hp
from quantize_pack_gb300 import configs, synth
from quantize_pack_gb300.path import UlyssesLowpPath

pytestmark = pytest.mark.gpu


def _finite_patterns(dtype):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = synth.from_bits(bits, dtype)
    return bits[np.isfinite(f)], f[np.isfinite(f)]


def _group_fill(rng, dtype, n, amax_bits, tie=False):
    """n patterns with |value| <= the amax pattern, the amax itself first."""
    bits, vals = _finite_patterns(dtype)
    a = float(synth.from_bits(np.array([amax_bits], np.uint16), dtype)[0])
    if tie:
        # amax = 127 * 2^k -> scale 2^k exactly; values (n + 0.5) * 2^k and n * 2^k
        k = np.log2(a / 127.0)
        cand = np.concatenate([np.arange(-127, 127) + 0.5, np.arange(-127, 128)]) * 2.0 ** k
        cb = synth.to_bits(cand.astype(np.float32), dtype)
        keep = np.abs(synth.from_bits(cb, dtype)) <= a
        cb = cb[keep]
        out = rng.choice(cb, n)
    else:
        ok = np.abs(vals) <= a
        out = rng.choice(bits[ok], n)
    out[0] = amax_bits
    return out


def _adversarial(dtype, D, seed, P=2, L=512, H=8):
    wl = configs.Workload(f"codec_{configs.DTYPE_NAMES[dtype]}_D{D}_s{seed}", B=1, H=H, D=D, P=P,
                          L=L, dtype=dtype, seed=seed)
    rng = np.random.default_rng(1000 + seed)
    S = wl.S
    q = np.empty((1, S, H, D), np.uint16)
    k = np.empty((1, S, H, D), np.uint16)
    ng = S // 128
    for g in range(ng):
        for hh in range(H):
            tie = (g + hh) % 4 == 0
            if tie:
                # 127 * 2^e and (n + 1/2) * 2^e must be finite in the dtype
                e = int(rng.integers(-20, 20)) if dtype == configs.BF16 else int(rng.integers(-14, 8))
                amax = synth.to_bits(np.array([127.0 * 2.0 ** e], np.float32), dtype)[0]
            else:
                lim = 14 if dtype == configs.FP16 else 60
                amax = synth.to_bits(np.array([2.0 ** rng.uniform(-lim, lim)], np.float32), dtype)[0]
            vals = _group_fill(rng, dtype, 128 * D, amax, tie)
            q[0, g * 128:(g + 1) * 128, hh] = rng.permutation(vals).reshape(128, D)
            # K: two 64-row groups per Q group, each with its own amax around k_mean = 0
            for half in range(2):
                vals = _group_fill(rng, dtype, 64 * D, amax if half == 0 else
                                   synth.to_bits(np.array([2.0 ** rng.uniform(-12, 12)],
                                                          np.float32), dtype)[0], tie and half == 0)
                k[0, g * 128 + half * 64:g * 128 + half * 64 + 64, hh] = \
                    rng.permutation(vals).reshape(64, D)
    bits, _ = _finite_patterns(dtype)
    v = rng.choice(bits, (1, S, H, D)).astype(np.uint16)
    # E4M3 midpoints times a power-of-two scale on one head
    mids = np.array([(a + b) / 2 for a, b in zip(range(8, 15), range(9, 16))], np.float64)
    mid_vals = np.concatenate([mids * 2.0 ** e for e in range(-9, 8)])
    v[0, :, 0, :] = rng.choice(synth.to_bits(mid_vals.astype(np.float32), dtype), (S, D))
    v_scale = (2.0 ** rng.uniform(-30, 30, (1, H, D))).astype(np.float32)
    v_scale[0, 0, :] = (2.0 ** rng.integers(-3, 4, D)).astype(np.float32)
    k_mean = np.zeros((1, H, D), np.uint16)
    return synth.Inputs(wl=wl, q=q, k=k, v=v, k_mean=k_mean, v_scale=v_scale)


@pytest.mark.parametrize("dtype,D,seed", [(configs.BF16, 128, 0), (configs.BF16, 64, 1),
                                          (configs.FP16, 128, 2), (configs.FP16, 64, 3)])
def test_codec_adversarial(dtype, D, seed):
    inp = _adversarial(dtype, D, seed)
    wl = inp.wl
    res = hp.run_oracle(inp)
    q, k, v, km, vs = gh.to_device(inp)
    # the pack kernel of the three-launch step, and the same body inside the
    # single cooperative launch
    for single in (False, True):
        path = UlyssesLowpPath(B=wl.B, L=wl.L, H=wl.H, D=wl.D, world_size=wl.P,
                               dtype=gh.torch_dtype(wl.dtype), single_launch=single)
        outs = path.run(q, k, v, km, vs)
        torch.cuda.synchronize()
        gh.assert_bits_equal(path.recv, res["recv"], f"chunks (single launch {single})")
        for i, name in enumerate(["q8", "k8", "v8", "q_scale", "k_scale"]):
            want = np.stack([res["out"][p][i] for p in range(wl.P)])
            gh.assert_bits_equal(outs[i], want, f"{name} (single launch {single})")
