"""The tolerance of the attention consumer against the fp64 oracle, shared by
the GPU parity tests and the CPU check that the tolerance catches a dropped
or doubled key tile.

Two bounds, per output element, relative to Vmax = max over the live keys of
|V[u, d]| for that batch, head and channel:

worst(n, xmax): derived from the kernel's arithmetic, every rounding at its
  worst:
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
  worst = 2 eps_w + n (2^-22 + 2^-25) + (2 ceil(n/128) + 3) 2^-23.

typical(n, xmax): the same terms with the n-fold accumulation and subnormal
  terms taken as independent roundings, which grow like sqrt(n), with a
  margin of 16 (2 eps_w is kept whole: the fp16 rounding of the weights is
  per element, not a sum):
  typical = 2 eps_w + 16 sqrt(n) (2^-22 + 2^-25) + (2 sqrt(ceil(n/128)) + 3) 2^-23.
  At the bench's n = 74800 worst is 0.021 and typical 0.0023 of Vmax.

bf16 / fp16 outputs add one rounding of the result (2^-9 / 2^-12 relative).
"""
import math

import numpy as np

from oracle import attention as A


def worst(n: int, xmax: float) -> float:
    eps_w = 2.0 ** -11 + 6 * math.log(2) * 2.0 ** -24 * xmax + 2.0 ** -22
    return 2 * eps_w + n * (2.0 ** -22 + 2.0 ** -25) + (2 * math.ceil(n / 128) + 3) * 2.0 ** -23


def typical(n: int, xmax: float) -> float:
    eps_w = 2.0 ** -11 + 6 * math.log(2) * 2.0 ** -24 * xmax + 2.0 ** -22
    return (2 * eps_w + 16 * math.sqrt(n) * (2.0 ** -22 + 2.0 ** -25)
            + (2 * math.sqrt(math.ceil(n / 128)) + 3) * 2.0 ** -23)


def extent(c, sm_scale=None, rows=None):
    """(Vmax [B, 1, h, D] = max over the live keys of |V|, xmax = the largest
    |logit| in log2 units over the query rows `rows` (all when None))."""
    Q, K, V = A.dequantize(c.q8, c.k8, c.v8, c.q_scale, c.k_scale, c.v_scale, n=c.n,
                           q_group=c.q_group)
    if rows is not None:
        Q = Q[:, np.asarray(rows)]
    D = c.q8.shape[3]
    sm = D ** -0.5 if sm_scale is None else sm_scale
    xmax = max(float(np.abs(Q[b, :, j] @ K[b, :, j].T).max())
               for b in range(Q.shape[0]) for j in range(Q.shape[2])) * sm / math.log(2)
    return np.abs(V).max(axis=1, keepdims=True), xmax


def check(got, want, c, rel_out=0.0, sm_scale=None, use_typical=False, vm_xmax=None):
    """Assert |got - want| <= worst * Vmax (+ rel_out |want|) everywhere, and
    with use_typical also <= typical * Vmax; return max err / worst-tolerance."""
    vm, xmax = extent(c, sm_scale) if vm_xmax is None else vm_xmax
    err = np.abs(got - want)
    tol = worst(c.n, xmax) * vm + rel_out * np.abs(want)
    ratio = np.divide(err, tol, out=np.where(err > 0, np.inf, 0.0), where=tol > 0)
    w = np.unravel_index(np.argmax(ratio), err.shape)
    assert np.all(err <= tol), (f"max err/worst-case tolerance {float(ratio[w]):.3f} at {w}: "
                                f"got {got[w]} want {want[w]}")
    if use_typical:
        ttol = typical(c.n, xmax) * vm + rel_out * np.abs(want)
        tr = np.divide(err, ttol, out=np.where(err > 0, np.inf, 0.0), where=ttol > 0)
        t = np.unravel_index(np.argmax(tr), err.shape)
        assert np.all(err <= ttol), (f"max err/typical tolerance {float(tr[t]):.3f} at {t}: "
                                     f"got {got[t]} want {want[t]}")
    return float(ratio.max())


def perturbed(c, tile: int, mode: str, b: int = 0, j: int = 0) -> np.ndarray:
    """The attention of batch b, head j [n, D] with key tile `tile` (keys
    [128 tile, 128 tile + 128) of the live prefix) dropped ("drop") or
    counted twice ("double"): the error a kernel that skips or repeats one
    key tile would make, written out in float64 here to test the tolerance."""
    Q, K, V = A.dequantize(c.q8, c.k8, c.v8, c.q_scale, c.k_scale, c.v_scale, n=c.n,
                           q_group=c.q_group)
    D = c.q8.shape[3]
    s = D ** -0.5 * (Q[b, :, j] @ K[b, :, j].T)
    s -= s.max(axis=1, keepdims=True)
    p = np.exp(s)
    keys = slice(128 * tile, min(128 * tile + 128, c.n))
    p[:, keys] *= 0.0 if mode == "drop" else 2.0
    return (p @ V[b, :, j]) / p.sum(axis=1, keepdims=True)


def e4m3_pv_tolerance(c, sm_scale=None):
    """Per-element tolerance [B, n, h, D] of the E4M3 PV product (P rounded to
    E4M3, V read as E4M3), from the exact weights of every row.

    With w_u = 2^(x_u - x_max) the exact weight of key u relative to the
    row's maximum, the kernel rounds w_u * 2^(x_max - m) to E4M3, where its
    running m lies in [x_max - 8, x_max] (weights stay <= 2^8 < 448, no
    saturation).  E4M3 keeps 3 mantissa bits: a normal value (>= 2^-6) is
    off by at most 2^-4 of itself; below, by at most min(2^-10, the value)
    (half the 2^-9 subnormal step, or the value rounded to zero).  In units
    of w that is
        e_u = 2^-4 w_u                 if w_u >= 2^-6,
        e_u = min(2^-10, w_u)          otherwise.
    The denominator sums the fp32 weights, so the output moves by at most
    sum_u e_u |V[u, d]| / sum_u w_u, plus the weights' exponent error (2 eps_e
    Vmax, as in worst()) and the fp32 accumulation terms of worst()."""
    Q, K, V = A.dequantize(c.q8, c.k8, c.v8, c.q_scale, c.k_scale, c.v_scale, n=c.n,
                           q_group=c.q_group)
    B, n, h, D = Q.shape
    sm = D ** -0.5 if sm_scale is None else sm_scale
    tol = np.empty((B, n, h, D))
    for b in range(B):
        for j in range(h):
            x = sm * (Q[b, :, j] @ K[b, :, j].T) / math.log(2)          # log2 units
            xmax = float(np.abs(x).max())
            w = np.exp2(x - x.max(axis=1, keepdims=True))
            e = np.where(w >= 2.0 ** -6, 2.0 ** -4 * w, np.minimum(2.0 ** -10, w))
            vabs = np.abs(V[b, :, j])
            eps_e = 6 * math.log(2) * 2.0 ** -24 * xmax + 2.0 ** -22
            rest = 2 * eps_e + n * 2.0 ** -22 + (2 * math.ceil(n / 128) + 3) * 2.0 ** -23
            tol[b, :, j] = (e @ vabs) / w.sum(axis=1, keepdims=True) + rest * vabs.max(axis=0)
    return tol

