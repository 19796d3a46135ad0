"""Pins of the attention oracle (oracle/attention.py), the consumer of the
unpacked tensors (page "unpack_for_sage": INT8 Q/K with per-group scales of
the width the kernel derives from its rows, FP8 E4M3 V, the caller's V
scale).

Independent checks: a pure-Python brute force with math.exp / math.fsum and
torch's E4M3 cast, torch's scaled_dot_product_attention in float64 on
tensors dequantised here with torch ops, closed forms (zero queries give the
key mean; a dominant key gives its value row), invariances (key and query
permutations inside a scale group, rows past the live prefix), and planted
mistakes in copies of the oracle's source that these checks must reject."""
import inspect
import math

import numpy as np
import pytest
import torch

from oracle import attention as A

GK = 64


def make(seed, *, B=1, S=200, h=2, D=64, n=None, q_group=128, spread=1.0):
    """Seeded quantised operands: int8 codes, E4M3 bytes (finite, no NaN),
    positive per-group scales that vary from group to group."""
    rng = np.random.default_rng(seed)
    n = S if n is None else n
    Spad = (S + 63) // 64 * 64
    q8 = rng.integers(-127, 128, size=(B, S, h, D), dtype=np.int8)
    k8 = rng.integers(-127, 128, size=(B, S, h, D), dtype=np.int8)
    v8 = rng.integers(0, 256, size=(B, D, h, Spad)).astype(np.uint8)
    v8[(v8 & 0x7F) == 0x7F] = 0x3C                      # no NaN codes
    v8[..., S:] = 0
    wq, wk = (n + q_group - 1) // q_group, (n + GK - 1) // GK
    qs = (spread * rng.uniform(0.5, 2.0, size=(B, h, wq)) / 127 / 8).astype(np.float32)
    ks = (spread * rng.uniform(0.5, 2.0, size=(B, h, wk)) / 127 / 8).astype(np.float32)
    vs = rng.uniform(0.01, 0.05, size=(B, h, D)).astype(np.float32)
    return dict(q8=q8, k8=k8, v8=v8, q_scale=qs, k_scale=ks, v_scale=vs, n=n, q_group=q_group)


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    """Library decode: torch's float8_e4m3fn view of the bytes."""
    t = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def brute(c, b, t, j, sm_scale=None):
    """O[b, t, j, :] by pure-Python loops, from the definitions."""
    q8, k8, v8 = c["q8"], c["k8"], c["v8"]
    D = q8.shape[3]
    n, G = c["n"], c["q_group"]
    sm = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
    qsc = float(c["q_scale"][b, j, t // G])
    logits = []
    for u in range(n):
        ksc = float(c["k_scale"][b, j, u // GK])
        dot = math.fsum(int(q8[b, t, j, d]) * qsc * int(k8[b, u, j, d]) * ksc for d in range(D))
        logits.append(sm * dot)
    mx = max(logits)
    w = [math.exp(x - mx) for x in logits]
    tot = math.fsum(w)
    vals = e4m3_values(v8[b, :, j, :n])                     # [D, n]
    return [math.fsum(w[u] * float(vals[d, u]) * float(c["v_scale"][b, j, d]) for u in range(n)) / tot
            for d in range(D)]


def run(c, **kw):
    return A.sage_attention(c["q8"], c["k8"], c["v8"], c["q_scale"], c["k_scale"], c["v_scale"],
                            n=c["n"], q_group=c["q_group"], **kw)


@pytest.mark.parametrize("q_group", [64, 128])
def test_brute_force_on_a_few_rows(q_group):
    c = make(1, S=150, h=2, D=64, n=141, q_group=q_group)
    O = run(c)
    for b, t, j in [(0, 0, 0), (0, 70, 1), (0, 127, 0), (0, 128, 1), (0, 140, 0)]:
        want = np.array(brute(c, b, t, j))
        assert np.allclose(O[b, t, j], want, rtol=1e-12, atol=1e-15), (b, t, j)


def sdpa_reference(c, sm_scale=None):
    """torch's attention in float64 on operands dequantised with torch ops."""
    q8 = torch.from_numpy(c["q8"]).double()
    k8 = torch.from_numpy(c["k8"]).double()
    n, G = c["n"], c["q_group"]
    rows = torch.arange(n)
    qs = torch.from_numpy(c["q_scale"]).double().index_select(2, rows // G)     # [B, h, n]
    ks = torch.from_numpy(c["k_scale"]).double().index_select(2, rows // GK)
    Q = q8[:, :n].permute(0, 2, 1, 3) * qs[..., None]                            # [B, h, n, D]
    K = k8[:, :n].permute(0, 2, 1, 3) * ks[..., None]
    V = torch.from_numpy(e4m3_values(c["v8"][..., :n])).permute(0, 2, 3, 1)      # [B, h, n, D]
    V = V * torch.from_numpy(c["v_scale"]).double()[:, :, None, :]
    O = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=sm_scale)
    return O.permute(0, 2, 1, 3).numpy()                                          # [B, n, h, D]


@pytest.mark.parametrize("q_group", [64, 128])
@pytest.mark.parametrize("B,S,h,D,n", [(1, 300, 2, 64, 300), (2, 333, 1, 128, 257),
                                       (1, 129, 3, 64, 65), (1, 64, 1, 128, 1)])
def test_against_torch_attention(q_group, B, S, h, D, n):
    c = make(2 + S, B=B, S=S, h=h, D=D, n=n, q_group=q_group, spread=4.0)
    O = run(c)
    assert O.shape == (B, n, h, D)
    assert np.allclose(O, sdpa_reference(c), rtol=1e-11, atol=1e-14)
    # an explicit softmax scale
    assert np.allclose(run(c, sm_scale=0.3), sdpa_reference(c, sm_scale=0.3), rtol=1e-11,
                       atol=1e-14)


def test_selected_rows_equal_the_full_result():
    c = make(12, S=300, h=2, D=64, n=280, q_group=64)
    O = run(c)
    rows = [0, 63, 64, 200, 279]
    # the same values up to the library matmul's summation order
    assert np.allclose(run(c, rows=rows), O[:, rows], rtol=1e-13, atol=1e-16)


def test_zero_queries_average_the_values():
    c = make(3, S=200, h=2, D=64, n=190)
    c["q8"][:] = 0
    O = run(c)
    V = e4m3_values(c["v8"][..., :190]).transpose(0, 3, 2, 1) * c["v_scale"][:, None].astype(np.float64)
    assert np.allclose(O, np.broadcast_to(V.mean(axis=1, keepdims=True), O.shape), rtol=1e-13,
                       atol=1e-16)


def test_a_dominant_key_selects_its_value_row():
    c = make(4, S=128, h=1, D=64, n=128)
    c["q8"][:] = 0
    c["k8"][:] = 0
    c["q8"][0, :, 0, :] = 127
    c["k8"][0, 77, 0, :] = 127
    c["q_scale"][:] = 1.0
    c["k_scale"][:] = 1.0                              # logit gap 127^2 * 64 / 8: the rest vanish
    O = run(c)
    want = e4m3_values(c["v8"][0, :, 0, 77]) * c["v_scale"][0, 0].astype(np.float64)
    assert np.array_equal(O[0, :, 0], np.broadcast_to(want, (128, 64)))


def test_permutations_inside_scale_groups():
    c = make(5, S=256, h=2, D=64, n=256, q_group=128)
    O = run(c)
    rng = np.random.default_rng(9)
    # keys (with their values) permuted inside each 64-row K group
    perm = np.concatenate([g * 64 + rng.permutation(64) for g in range(4)])
    c2 = dict(c)
    c2["k8"] = np.ascontiguousarray(c["k8"][:, perm])
    c2["v8"] = np.ascontiguousarray(c["v8"][..., perm])
    assert np.allclose(run(c2), O, rtol=1e-12, atol=1e-15)
    # queries permuted inside each 128-row Q group permute the output rows
    qp = np.concatenate([g * 128 + rng.permutation(128) for g in range(2)])
    c3 = dict(c)
    c3["q8"] = np.ascontiguousarray(c["q8"][:, qp])
    assert np.array_equal(run(c3), O[:, qp])


def test_rows_past_the_live_prefix_do_not_matter():
    c = make(6, S=300, h=1, D=128, n=200)
    O = run(c)
    c2 = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in c.items()}
    c2["q8"][:, 200:] = 99
    c2["k8"][:, 200:] = -99
    c2["v8"][..., 200:] = 0x44
    assert np.array_equal(run(c2), O)


# ---------------------------------------------------------------- mutants

SRC = inspect.getsource(A)

MUTANTS = {
    "K scales per 128 rows": ("ks = k_scale.astype(np.float64)[:, :, rows // GK]",
                              "ks = k_scale.astype(np.float64)[:, :, rows // 128]"),
    "Q scales per 64 rows": ("qs = q_scale.astype(np.float64)[:, :, rows // q_group]",
                             "qs = q_scale.astype(np.float64)[:, :, rows // 64]"),
    "softmax scale dropped": ("s = sm_scale * (Q[b, :, j] @ K[b, :, j].T)",
                              "s = (Q[b, :, j] @ K[b, :, j].T)"),
    "softmax over queries": ("s -= s.max(axis=1, keepdims=True)\n            p = np.exp(s)\n            O[b, :, j] = (p @ V[b, :, j]) / p.sum(axis=1, keepdims=True)",
                             "s -= s.max(axis=0, keepdims=True)\n            p = np.exp(s)\n            O[b, :, j] = (p @ V[b, :, j]) / p.sum(axis=0, keepdims=True)[0][:, None]"),
    "V channel scale of the next channel": ("v_scale.astype(np.float64)[:, None]",
                                            "np.roll(v_scale.astype(np.float64), 1, axis=2)[:, None]"),
    "V codes read as integers": ("Vc = tab[v8[..., :n]]", "Vc = v8[..., :n].astype(np.float64)"),
    "V transposed": ("V = Vc.transpose(0, 3, 2, 1)", "V = Vc.transpose(0, 3, 2, 1)[:, ::-1]"),
}


def _checks_pass(mod) -> bool:
    try:
        for q_group in (64, 128):
            c = make(11, S=300, h=2, D=64, n=290, q_group=q_group, spread=4.0)
            O = mod.sage_attention(c["q8"], c["k8"], c["v8"], c["q_scale"], c["k_scale"],
                                   c["v_scale"], n=c["n"], q_group=q_group)
            if not np.allclose(O, sdpa_reference(c), rtol=1e-11, atol=1e-14):
                return False
            for b, t, j in [(0, 5, 0), (0, 200, 1)]:
                if not np.allclose(O[b, t, j], brute(c, b, t, j), rtol=1e-12, atol=1e-15):
                    return False
    except Exception:
        return False
    return True


def test_checks_accept_the_oracle():
    assert _checks_pass(A)


@pytest.mark.parametrize("name", list(MUTANTS))
def test_checks_reject_mutant(name):
    a, b = MUTANTS[name]
    assert SRC.count(a) == 1, name
    ns = {"__name__": "attention_mutant"}
    src = SRC.replace(a, b).replace("from . import oracle as _orc", "from oracle import oracle as _orc")
    exec(compile(src, "attention_mutant", "exec"), ns)

    class M:
        sage_attention = staticmethod(ns["sage_attention"])
    assert not _checks_pass(M), f"the checks did not catch: {name}"


@pytest.mark.parametrize("mode", ["drop", "double"])
def test_tolerance_rejects_a_key_tile_dropped_or_counted_twice(mode):
    """The GPU tests' tolerance (attention_check.check, worst case and
    typical) accepts the oracle's own result on structured operands and
    rejects the result of a kernel that drops one key tile or counts it twice
    (that result computed here in float64 by attention_check.perturbed)."""
    import attention_check as ac
    from quantize_pack_gb300 import synth
    c = synth.attention_operands_paired(3, S=1100, h=1, D=128, n=1000)
    want = A.sage_attention(c.q8, c.k8, c.v8, c.q_scale, c.k_scale, c.v_scale, n=c.n)
    assert ac.check(want, want, c, use_typical=True) == 0.0
    for tile in (0, 3, 7):                     # first, inner, the ragged last tile
        bad = ac.perturbed(c, tile, mode)[None, :, None, :]
        with pytest.raises(AssertionError, match="worst-case"):
            ac.check(bad, want, c)


def test_e4m3_pv_tolerance_holds_for_a_simulated_kernel_and_rejects_a_dropped_tile():
    """attention_check.e4m3_pv_tolerance, the bound of the E4M3 PV product:
    the attention with every weight (relative to the row max, and to a max
    8 log2 units above it, the two ends of the kernel's running max) rounded
    to E4M3 by torch's cast lies inside it; a dropped key tile does not."""
    import attention_check as ac
    from quantize_pack_gb300 import synth
    c = synth.attention_operands(5, B=1, S=600, h=1, D=64, n=520, q_group=64, spread=16.0)
    Q, K, V = A.dequantize(c.q8, c.k8, c.v8, c.q_scale, c.k_scale, c.v_scale, n=c.n, q_group=64)
    x = (Q[0, :, 0] @ K[0, :, 0].T) / 8.0 / math.log(2)
    want = A.sage_attention(c.q8, c.k8, c.v8, c.q_scale, c.k_scale, c.v_scale, n=c.n, q_group=64)
    tol = ac.e4m3_pv_tolerance(c)
    for lag in (0.0, 8.0):
        w = np.exp2(x - x.max(axis=1, keepdims=True) + lag)
        w8 = torch.from_numpy(w).to(torch.float8_e4m3fn).to(torch.float64).numpy()
        sim = (w8 @ V[0, :, 0]) / w.sum(axis=1, keepdims=True)
        assert np.all(np.abs(sim - want[0, :, 0]) <= tol[0, :, 0]), lag
    bad = ac.perturbed(c, 2, "drop")
    assert np.any(np.abs(bad - want[0, :, 0]) > tol[0, :, 0])

