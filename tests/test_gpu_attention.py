"""GPU parity of the attention consumer (ulp_sage_attention) against the fp64
oracle (oracle/attention.py) on the same seeded operands, within the
tolerances of attention_check.py (the derived worst case everywhere; also the
typical bound at full size).  Each test prints its observed max error over
the worst-case tolerance (pytest -s shows it)."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from quantize_pack_gb300 import synth, ulp
import attention_check as ac
import helpers as hp
import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def run_gpu(c, out_dtype=torch.float32, sm_scale=None, pv_fp8=False):
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ulp.sage_attention(dev(c.q8), dev(c.k8), dev(c.v8), dev(c.q_scale), dev(c.k_scale),
                             dev(c.v_scale), n=c.n, q_group=c.q_group, sm_scale=sm_scale,
                             out_dtype=out_dtype, status=status, pv_fp8=pv_fp8)
    torch.cuda.synchronize()
    assert status.item() == 0, f"tensor-core wait timed out (code {status.item()})"
    return out.float().cpu().numpy().astype(np.float64)


def oracle(c, **kw):
    return A.sage_attention(c.q8, c.k8, c.v8, c.q_scale, c.k_scale, c.v_scale, n=c.n,
                            q_group=c.q_group, **kw)


def check(got, want, c, **kw):
    r = ac.check(got, want, c, **kw)
    print(f"max err / worst-case tolerance: {r:.4f}")
    return r


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


def test_paired_dominant_keys_within_the_typical_bound():
    """Structured peaky operands (every query tile's weight split between two
    equal dominant keys in neighbouring key tiles), ragged live prefix."""
    c = synth.attention_operands_paired(44, S=1100, h=2, D=128, n=1000)
    check(run_gpu(c), oracle(c), c, use_typical=True)


@pytest.mark.parametrize("B,S,h,D,n,q_group,spread", CASES,
                         ids=[f"B{c[0]}_S{c[1]}_h{c[2]}_D{c[3]}_n{c[4]}_gq{c[5]}" for c in CASES])
def test_e4m3_pv_matches_oracle(B, S, h, D, n, q_group, spread):
    """The E4M3 PV product (P rounded to E4M3, V straight from v8) against the
    exact fp64 attention, within the per-row bound of the weights' E4M3
    rounding (attention_check.e4m3_pv_tolerance); values past the live prefix
    (NaN codes among them) must not reach the output."""
    c = synth.attention_operands(100 + S + n, B=B, S=S, h=h, D=D, n=n, q_group=q_group,
                                 spread=spread)
    c.v8[..., n:] = 0x7F                     # NaN codes past the prefix (zero-filled keys
    got = run_gpu(c, pv_fp8=True)            # of the last tile must not read them)
    want = oracle(c)
    tol = ac.e4m3_pv_tolerance(c)
    err = np.abs(got - want)
    r = float(np.divide(err, tol, out=np.zeros_like(err), where=tol > 0).max())
    print(f"E4M3 PV: max err / its bound {r:.4f}; max err / max|V| "
          f"{float((err / np.abs(want).max()).max()):.2e}")
    assert np.all(np.isfinite(got)) and np.all(err <= tol), r


def test_e4m3_pv_paired_keys():
    c = synth.attention_operands_paired(45, S=1100, h=2, D=128, n=1000)
    got, want = run_gpu(c, pv_fp8=True), oracle(c)
    err = np.abs(got - want)
    assert np.all(err <= ac.e4m3_pv_tolerance(c)), float((err / ac.e4m3_pv_tolerance(c)).max())


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
        vmax = np.abs(V[0, :, 0]).max(axis=0)                               # [D]
        err = np.abs(got[0, rows, j] - want)
        assert np.all(err <= ac.worst(n, xmax) * vmax), (j, float((err / (ac.worst(n, xmax) * vmax)).max()))
        assert np.all(err <= ac.typical(n, xmax) * vmax), (j, float((err / (ac.typical(n, xmax) * vmax)).max()))
        print(f"head {j}: max err / worst-case tolerance {float((err / (ac.worst(n, xmax) * vmax)).max()):.4f}")


def test_full_size_every_row_paired_keys():
    """The bench's consumer shape (B=1, S = 8 x 9360, h = 5, D = 128, live
    prefix 74800) on structured operands: every query tile's softmax splits
    between two equal dominant keys, one in its own key tile and one in the
    next (synth.attention_operands_paired), so a key tile dropped or counted
    twice moves whole rows by a large part of max |V|.  Every query row of
    head 0 against the oracle (in chunks), within the typical bound, and the
    observed error at most a tenth of the worst-case tolerance."""
    S, n, h, D = 8 * 9360, 74800, 5, 128
    c = synth.attention_operands_paired(43, S=S, h=h, D=D, n=n)
    got = run_gpu(c, out_dtype=torch.float32)
    j = 0
    cj = synth.AttentionOperands(
        np.ascontiguousarray(c.q8[:, :, j:j + 1]), np.ascontiguousarray(c.k8[:, :, j:j + 1]),
        np.ascontiguousarray(c.v8[:, :, j:j + 1]), np.ascontiguousarray(c.q_scale[:, j:j + 1]),
        np.ascontiguousarray(c.k_scale[:, j:j + 1]), np.ascontiguousarray(c.v_scale[:, j:j + 1]),
        n, 128)
    want = np.empty((n, D))
    for r0 in range(0, n, 2048):
        rows = np.arange(r0, min(r0 + 2048, n))
        want[rows] = A.sage_attention(cj.q8, cj.k8, cj.v8, cj.q_scale, cj.k_scale, cj.v_scale, n=n,
                                      q_group=128, rows=rows)[0, :, 0]
    Q, K, V = A.dequantize(cj.q8, cj.k8, cj.v8, cj.q_scale, cj.k_scale, cj.v_scale, n=n, q_group=128)
    xmax = max(float(np.abs(Q[0, r0:r0 + 2048, 0] @ K[0, :, 0].T).max()) for r0 in range(0, n, 2048))
    xmax *= D ** -0.5 / math.log(2)
    vm = np.abs(V).max(axis=1, keepdims=True)
    r = check(got[:, :, j:j + 1], want[None, :, None, :], cj, use_typical=True, vm_xmax=(vm, xmax))
    assert r <= 0.1, f"observed max err is {r:.3f} of the worst-case tolerance (expected <= 0.1)"
