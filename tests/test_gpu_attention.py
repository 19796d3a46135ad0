"""GPU parity of the attention consumer (ulp_sage_attention) against the fp64
oracle (oracle/attention.py) on the same seeded operands.

Tolerance, from the kernel's arithmetic (per output element, relative to
Vmax = max over the live keys of |V[u, d]| for that batch, head and channel):
  * the integer logits q8 . k8 are exact (fp16 operands, fp32 accumulation of
    at most 128 products of magnitude <= 2^14);
  * the weight exponent fma(S, c, -m) with c = fl(fl(q_scale * fl(sm_scale *
    log2 e)) * k_scale): three roundings in c (3 2^-24 |x|) and one in the
    fma (2^-24 |x - m| <= 2^-23 xmax, xmax = the largest |x|); the error of m
    itself shifts every weight alike and cancels.  So each weight 2^(x - m)
    is off by at most ln2 * 6 * 2^-24 * xmax relative, plus the 2^-22 of the
    hardware exp2;
  * so the computed weights' mean is within 2 eps_e Vmax of the exact one,
    eps_e = 6 ln2 2^-24 xmax + 2^-22;
  * the numerator's weights are rounded to fp16 (2^-11 relative in the
    normal range, 2^-25 absolute below it) while the denominator sums the
    fp32 weights: at most 2^-11 Vmax more, plus n 2^-25 Vmax for the
    subnormal weights (the largest weight of a row is >= 1, so the sum is);
    with eps_w = 2^-11 + eps_e, 2 eps_e + 2^-11 <= 2 eps_w;
  * fp32 accumulation of the n products in the PV MMAs and the O rescales
    (numerator), and of the row's weights in eight partial sums per tile and
    one running sum across tiles (denominator): <= 2 (n + ntiles) 2^-23
    Vmax together; the final scaling by 1/l and v_scale: 3 2^-24.
bound(n, xmax) = 2 eps_w + n (2^-22 + 2^-25) + (2 ceil(n/128) + 3) 2^-23.
bf16 / fp16 outputs add one rounding of the result (2^-9 / 2^-12 relative).
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from quantize_pack_gb300 import synth, ulp
import helpers as hp
import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def bound(n: int, xmax: float) -> float:
    eps_w = 2.0 ** -11 + 6 * math.log(2) * 2.0 ** -24 * xmax + 2.0 ** -22
    return 2 * eps_w + n * (2.0 ** -22 + 2.0 ** -25) + (2 * math.ceil(n / 128) + 3) * 2.0 ** -23


def extent(c, sm_scale=None):
    """(Vmax [B, 1, h, D] = max over the live keys of |V|, xmax = the largest
    |logit| in log2 units)."""
    Q, K, V = A.dequantize(c.q8, c.k8, c.v8, c.q_scale, c.k_scale, c.v_scale, n=c.n,
                           q_group=c.q_group)
    D = c.q8.shape[3]
    sm = D ** -0.5 if sm_scale is None else sm_scale
    xmax = max(float(np.abs(Q[b, :, j] @ K[b, :, j].T).max())
               for b in range(Q.shape[0]) for j in range(Q.shape[2])) * sm / math.log(2)
    return np.abs(V).max(axis=1, keepdims=True), xmax


def run_gpu(c, out_dtype=torch.float32, sm_scale=None):
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ulp.sage_attention(dev(c.q8), dev(c.k8), dev(c.v8), dev(c.q_scale), dev(c.k_scale),
                             dev(c.v_scale), n=c.n, q_group=c.q_group, sm_scale=sm_scale,
                             out_dtype=out_dtype, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0, f"tensor-core wait timed out (code {status.item()})"
    return out.float().cpu().numpy().astype(np.float64)


def oracle(c, **kw):
    return A.sage_attention(c.q8, c.k8, c.v8, c.q_scale, c.k_scale, c.v_scale, n=c.n,
                            q_group=c.q_group, **kw)


def check(got, want, c, rel_out=0.0, sm_scale=None):
    vm, xmax = extent(c, sm_scale)
    tol = bound(c.n, xmax) * vm + rel_out * np.abs(want)
    err = np.abs(got - want)
    ratio = np.divide(err, tol, out=np.where(err > 0, np.inf, 0.0), where=tol > 0)
    worst = np.unravel_index(np.argmax(ratio), err.shape)
    assert np.all(err <= tol), (f"max err/tol {float(ratio[worst]):.3f} at {worst}: "
                                f"got {got[worst]} want {want[worst]}")
    return float(ratio.max())


CASES = [
    # B, S, h, D, n, q_group, spread
    (1, 200, 2, 64, 200, 128, 8.0),      # two query tiles, a ragged key tile
    (2, 333, 1, 128, 257, 64, 8.0),      # live prefix 257: one key past two tiles
    (1, 1000, 2, 128, 1000, 128, 16.0),  # 8 tiles, ragged tail of 104
    (1, 129, 3, 64, 65, 64, 4.0),        # one partial tile, odd head count
    (1, 64, 1, 128, 1, 128, 1.0),        # a single live row
    (1, 2048, 1, 128, 2048, 128, 16.0),  # tile-aligned, peaky softmax
    (1, 384, 2, 64, 300, 64, 32.0),      # very peaky: the running max moves often
]


@pytest.mark.parametrize("B,S,h,D,n,q_group,spread", CASES,
                         ids=[f"B{c[0]}_S{c[1]}_h{c[2]}_D{c[3]}_n{c[4]}_gq{c[5]}" for c in CASES])
def test_attention_matches_oracle(B, S, h, D, n, q_group, spread):
    c = synth.attention_operands(100 + S + n, B=B, S=S, h=h, D=D, n=n, q_group=q_group,
                                 spread=spread)
    got = run_gpu(c)
    assert got.shape == (B, n, h, D)
    check(got, oracle(c), c)


def test_explicit_softmax_scale():
    c = synth.attention_operands(7, B=1, S=300, h=2, D=128, n=280, q_group=128, spread=4.0)
    check(run_gpu(c, sm_scale=0.05), oracle(c, sm_scale=0.05), c, sm_scale=0.05)


@pytest.mark.parametrize("dtype,rel", [(torch.bfloat16, 2.0 ** -9), (torch.float16, 2.0 ** -12)],
                         ids=["bf16", "fp16"])
def test_half_precision_outputs(dtype, rel):
    c = synth.attention_operands(8, B=1, S=500, h=2, D=64, n=450, q_group=64, spread=8.0)
    check(run_gpu(c, out_dtype=dtype), oracle(c), c, rel_out=rel)


def test_rows_past_the_live_prefix_are_ignored():
    c = synth.attention_operands(9, B=1, S=400, h=1, D=128, n=250, q_group=128, spread=8.0)
    a = run_gpu(c)
    c.q8[:, 250:] = -128
    c.k8[:, 250:] = 127
    c.v8[..., 250:400] = 0x7F               # NaN codes past the prefix
    b = run_gpu(c)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("wl", [hp.PADDING_R, hp.G64[1]], ids=lambda w: w.name)
def test_on_the_unpacked_outputs_of_the_path(wl):
    """The oracle's own unpack outputs of a workload (bit-equal to the CUDA
    path's), fed to the consumer over the live prefix."""
    inp, res = hp.cached(wl)
    n = inp.used
    h = wl.h
    for p in sorted({0, wl.P - 1}):
        q8, k8, v8, qs, ks = res["out"][p]
        wq, wk = (n + wl.q_group - 1) // wl.q_group, (n + 63) // 64
        c = synth.AttentionOperands(q8, k8, v8, np.ascontiguousarray(qs[:, :, :wq]),
                                    np.ascontiguousarray(ks[:, :, :wk]),
                                    np.ascontiguousarray(inp.v_scale[:, p * h:(p + 1) * h]), n,
                                    wl.q_group)
        check(run_gpu(c), oracle(c), c)


def test_rejects_bad_arguments():
    c = synth.attention_operands(10, B=1, S=128, h=1, D=64, n=128)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    args = [dev(x) for x in (c.q8, c.k8, c.v8, c.q_scale, c.k_scale, c.v_scale)]
    for kw in (dict(n=0), dict(n=129), dict(q_group=32), dict(sm_scale=-1.0)):
        with pytest.raises(ulp.UlpError):
            ulp.sage_attention(*args, **kw)


def test_full_size_sampled_rows():
    """The long non-aligned workload's consumer shape (one destination: B=1,
    S = 8 x 9360, h = 5, D = 128, live prefix 74800), in the launch the bench
    times; sampled query rows of two heads against the oracle, row by row."""
    S, n, h, D = 8 * 9360, 74800, 5, 128
    c = synth.attention_operands(41, B=1, S=S, h=h, D=D, n=n, q_group=128, spread=8.0)
    got = run_gpu(c, out_dtype=torch.float32)
    rows = [0, 1, 127, 128, 4095, 37000, 74751, 74752, n - 2, n - 1]
    for j in (0, h - 1):
        cj = synth.AttentionOperands(
            np.ascontiguousarray(c.q8[:, :, j:j + 1]), np.ascontiguousarray(c.k8[:, :, j:j + 1]),
            np.ascontiguousarray(c.v8[:, :, j:j + 1]), np.ascontiguousarray(c.q_scale[:, j:j + 1]),
            np.ascontiguousarray(c.k_scale[:, j:j + 1]), np.ascontiguousarray(c.v_scale[:, j:j + 1]),
            n, 128)
        want = A.sage_attention(cj.q8, cj.k8, cj.v8, cj.q_scale, cj.k_scale, cj.v_scale, n=n,
                                q_group=128, rows=rows)[0, :, 0]            # [rows, D]
        Q, K, V = A.dequantize(cj.q8, cj.k8, cj.v8, cj.q_scale, cj.k_scale, cj.v_scale, n=n,
                               q_group=128)
        xmax = float(np.abs(Q[0, rows, 0] @ K[0, :, 0].T).max()) * D ** -0.5 / math.log(2)
        tol = bound(n, xmax) * np.abs(V[0, :, 0]).max(axis=0)              # [D]
        err = np.abs(got[0, rows, j] - want)
        assert np.all(err <= tol), (j, float((err / tol).max()))
