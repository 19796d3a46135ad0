"""The pins catch plausible mistakes: each mutant below is a copy of the
oracle with one mistake planted (a dropped term, a wrong sign, index or
rounding rule, a transposed operand); the independent checks of the pin tests
must reject every mutant and accept the oracle itself."""
import os

import numpy as np
import pytest

from oracle import oracle as O
from quantize_pack_gb300 import synth
import helpers as hp

SRC = open(os.path.join(os.path.dirname(O.__file__), "oracle.c")).read()

MUTANTS = {
    "floor dropped": ("static float floor_eps(float x) { return x < EPS ? EPS : x; }",
                      "static float floor_eps(float x) { return x; }"),
    "ties away from zero": ("    return fmodf(n, 2.0f) == 0.0f ? n : n + 1.0f;", "    return n + 1.0f;"),
    "round up at half": ("    if (frac > 0.5f) return n + 1.0f;", "    if (frac >= 0.49f) return n + 1.0f;"),
    "int8 wraps instead of saturating": (
        "    if (y >= 128.0f) return 127;\n    if (y <= -129.0f) return -128;\n    float n = rne_int(y);\n"
        "    if (n > 127.0f) return 127;\n    if (n < -128.0f) return -128;\n    return (int8_t)n;",
        "    return (int8_t)(int)rne_int(fmaxf(fminf(y, 1e6f), -1e6f));"),
    "e4m3 saturates at 480": ("    if (a > 448.0f) return (uint8_t)(sign | 0x7E);",
                              "    if (a > 480.0f) return (uint8_t)(sign | 0x7E);"),
    "used correction dropped": ("                    if (g == gu && hi > used) hi = used;       /* live rows only */",
                                "                    (void)gu;"),
    "min/max ignores used": ("                if (hi > live) hi = live;", "                (void)live;"),
    "min/max takes max for min": ("                        mn = minf(mn, x);", "                        mn = maxf(mn, x);"),
    "derive wrong sign": ("                        float dn = m - gathered[base + d];        /* rn(m - minK) */",
                          "                        float dn = gathered[base + d] - m;"),
    "derive wrong e index": ("                    int ee = g == first_group(rr, L, GK) ? 0 : 1;",
                             "                    int ee = 0;"),
    "q merge ignores partner": ("                        amax = maxf(amax, gathered_qb[(((size_t)rr * B + b) * H + hh) * 2 + ee]);",
                                "                        if (rr == rank) amax = maxf(amax, gathered_qb[(((size_t)rr * B + b) * H + hh) * 2 + ee]);"),
    "scale divides by 128": ("                qs[jq] = amax / 127.0f;", "                qs[jq] = amax / 128.0f;"),
    "k not centred": ("                    float xk = in_f32(k, src, dtype) - in_f32(k_mean, ((size_t)b * H + hh) * D + d, dtype);",
                      "                    float xk = in_f32(k, src, dtype);"),
    "k centred with the wrong sign": ("                    float xk = in_f32(k, src, dtype) - in_f32(k_mean, ((size_t)b * H + hh) * D + d, dtype);",
                                      "                    float xk = in_f32(k_mean, ((size_t)b * H + hh) * D + d, dtype) - in_f32(k, src, dtype);"),
    "v not transposed": ("                    v8[vdst] = chunk[ov + src];",
                         "                    v8[(((size_t)b * Spad + t) * h + j) * D + d < (size_t)B * D * h * Spad ? (((size_t)b * Spad + t) * h + j) * D + d : vdst] = chunk[ov + src];"),
    "q scale from the next slot": ("                q_scale[((size_t)b * h + j) * wq + g] = src[((size_t)b * h + j) * nq + (g - first_group(s, L, gq))];",
                                   "                q_scale[((size_t)b * h + j) * wq + g] = src[((size_t)b * h + j) * nq + (g - first_group(s, L, gq)) + (g + 1 < wq)];"),
    "64-row Q groups coded with the 128-row slot": ("                float sq = qs[t / gq - fq], sk = ks[t / GK - fk];",
                                                    "                float sq = qs[t / gq - fq - (gq == 64 && (t / 64) % 2 == 1 && t / 64 > fq)], sk = ks[t / GK - fk];"),
    "Q partial over 128 rows in the 64-row variant": ("                int qhi = g_q * gq + gq < row0 + L ? g_q * gq + gq : row0 + L;",
                                                      "                int qhi = g_q * gq + 128 < row0 + L ? g_q * gq + 128 : row0 + L;"),
    "-0 kept in min/max": ("                        if (x == 0.0f) x = 0.0f;   /* -0 -> +0 */", ""),
}


def with_negative_zeros(inp):
    """The inputs with a few live K entries set to -0 (bits 0x8000)."""
    k = inp.k.copy()
    flat = k.reshape(-1)
    rows = min(inp.used, inp.wl.S)
    live = flat[: rows * inp.wl.H * inp.wl.D * inp.wl.B]
    live[::97] = 0x8000
    return synth.Inputs(wl=inp.wl, q=inp.q, k=k, v=inp.v, k_mean=inp.k_mean, v_scale=inp.v_scale)


def pins_pass(wl, negzero=False) -> bool:
    """The core pin checks of the oracle tests, on one workload."""
    inp = synth.make_inputs(wl)
    if negzero:
        inp = with_negative_zeros(inp)
    try:
        res = hp.run_oracle(inp)
        S, used = wl.S, inp.used
        gu = (used - 1) // 64
        direct = hp.global_k_amax(inp)
        m_abs = np.maximum(np.abs(hp.f32(inp.k_mean, wl.dtype)).max(axis=2), hp.EPS)
        for r in range(wl.P):                      # the derive identity and the don't-cares
            groups = hp.touched_groups(r, wl.L, 64)
            for j, g in enumerate(groups):
                got = res["amax"][r][:, :, j]
                if g <= gu:
                    want = direct[:, :, g]
                elif j == 0 or j == len(groups) - 1:
                    want = np.full_like(got, hp.EPS)
                else:
                    want = m_abs
                if got.tobytes() != np.ascontiguousarray(want).tobytes():
                    return False
            for j in range(len(groups), O.slots(wl.L, 64)):
                if not np.all(res["amax"][r][:, :, j] == hp.EPS):
                    return False
        kf = hp.f32(inp.k, wl.dtype)               # boundary min/max
        if np.any(np.signbit(res["minmax"]) & (res["minmax"] == 0)):
            return False
        for r in range(wl.P):
            groups = hp.touched_groups(r, wl.L, 64)
            for e, g in ((0, groups[0]), (1, groups[-1])):
                lo, hi = max(g * 64, r * wl.L), min(g * 64 + 64, (r + 1) * wl.L, used)
                mm = res["minmax"][r][:, :, e]
                if hi > lo:
                    rows = kf[:, lo:hi] + np.float32(0)
                    if mm[:, :, 0].tobytes() != rows.min(axis=1).tobytes():
                        return False
                    if mm[:, :, 1].tobytes() != rows.max(axis=1).tobytes():
                        return False
                elif not (np.all(mm[:, :, 0] == np.inf) and np.all(mm[:, :, 1] == -np.inf)):
                    return False
        q8 = np.concatenate([res["out"][p][0] for p in range(wl.P)], axis=2)
        k8 = np.concatenate([res["out"][p][1] for p in range(wl.P)], axis=2)
        v8 = np.concatenate([res["out"][p][2] for p in range(wl.P)], axis=2)
        qsc = np.concatenate([res["out"][p][3] for p in range(wl.P)], axis=1)
        ks = np.concatenate([res["out"][p][4] for p in range(wl.P)], axis=1)
        qs = (hp.global_q_amax(inp) / np.float32(127)).astype(np.float32)
        if qsc.tobytes() != np.ascontiguousarray(qs[:, :, :qsc.shape[2]]).tobytes():
            return False
        row_qs = np.repeat(qs, wl.q_group, axis=2)[:, :, :S].transpose(0, 2, 1)[..., None]
        if not np.array_equal(q8, hp.int8_codes(hp.f32(inp.q, wl.dtype), row_qs)):
            return False
        ksc = (direct / np.float32(127)).astype(np.float32)
        n_live = min(ks.shape[2], (used + 63) // 64)
        if ks[:, :, :n_live].tobytes() != np.ascontiguousarray(ksc[:, :, :n_live]).tobytes():
            return False
        # live rows, and the padding rows of the partial live group (saturating)
        lim = min(S, (gu + 1) * 64)
        row_ks = np.repeat(ksc, 64, axis=2)[:, :, :S].transpose(0, 2, 1)[..., None]
        kc = (kf - hp.f32(inp.k_mean, wl.dtype)[:, None]).astype(np.float32)
        if not np.array_equal(k8[:, :lim], hp.int8_codes(kc, row_ks)[:, :lim]):
            return False
        want_v = hp.e4m3_codes(hp.f32(inp.v, wl.dtype) / inp.v_scale[:, None])
        if not np.array_equal(v8[..., :S], want_v.transpose(0, 3, 2, 1)) or np.any(v8[..., S:]):
            return False
    except Exception:
        return False
    # number formats: ties to even, saturation, E4M3 against the library cast
    if any(O.int8_code(n + 0.5) % 2 for n in range(-120, 120)):
        return False
    if O.int8_code(300.0) != 127 or O.int8_code(-300.0) != -128:
        return False
    x = np.linspace(-470, 470, 4001, dtype=np.float32)
    if not np.array_equal(np.array([O.e4m3(float(v)) for v in x], np.uint8), hp.e4m3_codes(x)):
        return False
    return True


# small workloads whose geometry exercises every branch: crossing groups,
# padding with a partial live group, a padding-only slice, several heads
# the partial live group inside one rank (rows 448..511 of rank 1)
INNER_PAD = hp.configs.Workload("inner_pad_P2_L300_used500", B=1, H=4, D=64, P=2, L=300,
                                dtype=hp.configs.BF16, seed=18, pad_rows=100, scale_to_used=True,
                                k_mean_std=4.0, k_noise_std=0.05)
WORKLOADS = [hp.CROSS_PAD, hp.SPAN4_PAD, hp.USED64.replace(H=8, name="used64_h2"),
             hp.TINY, INNER_PAD, hp.SPAN4_PAD.replace(q_group=64, name="span4_pad_gq64"),
             INNER_PAD.replace(q_group=64, name="inner_pad_gq64")]


def _all_pass():
    return all(pins_pass(wl) for wl in WORKLOADS) and pins_pass(hp.TINY, negzero=True)


def test_pins_accept_the_oracle():
    assert _all_pass()


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    a, b = MUTANTS[name]
    assert SRC.count(a) == 1, name
    path = O.build_variant(SRC.replace(a, b), str(tmp_path / "liboracle_mutant.so"))
    with O.use_library(path):
        assert not _all_pass(), f"the pins did not catch: {name}"
