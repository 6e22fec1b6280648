"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against a closed form, an invariant, a library
routine, brute-force matrix algebra or hand-derived values in tests/golden/,
so that a dropped term, a wrong sign, a wrong index or a transposed operand in
the oracle fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from gated_deltanet_linear_04_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _frac(s: str) -> float:
    if s.startswith("log("):
        return math.log(float(Fraction(s[4:-1])))
    return float(Fraction(s))


# ----------------------------------------------------------------------------
# bf16 conversion: pinned to torch's float -> bfloat16 (round-to-nearest-even)
# ----------------------------------------------------------------------------
def test_bf16_rounding_matches_torch(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(0)
    mags = np.exp2(rng.uniform(-140, 128, 20000)).astype(np.float32)
    signs = np.where(rng.random(20000) < 0.5, -1.0, 1.0).astype(np.float32)
    x = mags * signs
    # exact ties: low 16 bits 0x8000 with odd and even kept parts
    tie_bits = (rng.integers(0x0080, 0x7F00, 2000, dtype=np.uint32) << 16) | 0x8000
    ties = tie_bits.view(np.float32)
    specials = np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, 3.39e38, -3.39e38, 1e-40, -1e-40,
                         2.0 ** -126, 2.0 ** -133, 2.0 ** -134, 1.5 * 2.0 ** -134, np.inf, -np.inf],
                        np.float32)
    allx = np.concatenate([x, ties, specials])
    ref = torch.from_numpy(allx).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = o.f64_to_bf16(allx.astype(np.float64))
    assert np.array_equal(got, ref)
    # and back: bf16 bits -> value, pinned to torch's bfloat16 -> float
    back = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(o.bf16_to_f64(ref), back, equal_nan=True)


def test_bf16_rounding_single_step_from_f64(oracle_mod):
    o = oracle_mod
    # just above a bf16 tie in f64 but a tie once rounded to f32: one RNE step
    # from f64 must round up (two steps through f32 would round to even = 1).
    x = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert o.bf16_to_f64(o.f64_to_bf16(x)) == 1.0 + 2.0 ** -7
    assert o.bf16_to_f64(o.f64_to_bf16(1.0 + 2.0 ** -8)) == 1.0            # tie -> even
    assert o.bf16_to_f64(o.f64_to_bf16(1.0 + 3 * 2.0 ** -8)) == 1.0 + 2.0 ** -6  # tie -> even (up)


# ----------------------------------------------------------------------------
# a4 gates
# ----------------------------------------------------------------------------
def test_gating_golden_points(oracle_mod):
    o = oracle_mod
    gold = json.load(open(os.path.join(GOLDEN, "gating_spot_values.json")))
    for p in gold["gate_points"]:
        a = np.array([_frac(p["a"])])
        bits = o.f64_to_bf16(a)
        assert o.bf16_to_f64(bits)[0] == a[0]          # exactly representable
        g, _ = o.gating(bits, o.f64_to_bf16(np.zeros(1)), np.array([_frac(p["A_log"])]),
                        np.array([_frac(p["dt_bias"])]))
        assert g[0] == pytest.approx(_frac(p["g"]), rel=1e-14)
    for p in gold["beta_points"]:
        _, beta = o.gating(o.f64_to_bf16(np.zeros(1)), o.f64_to_bf16(np.array([_frac(p["b"])])),
                           np.zeros(1), np.zeros(1))
        assert beta[0] == _frac(p["beta"])


def test_softplus_sigmoid_against_library(oracle_mod):
    from scipy.special import expit
    o = oracle_mod
    x = np.linspace(-60, 60, 4001)
    assert np.allclose(o.softplus(x), np.logaddexp(x, 0.0), rtol=1e-15, atol=0)
    assert np.allclose(o.softplus(x) - o.softplus(-x), x, rtol=0, atol=1e-13)
    assert np.allclose(o.sigmoid(x), expit(x), rtol=1e-15, atol=1e-300)


def test_gating_ranges_and_monotonicity(oracle_mod):
    o = oracle_mod
    d = wl.WORKLOADS["tiny"].dims.with_(T=64, Hv=8)
    p = wl.make_params(d, 5)
    acts = wl.make_activations(d, 6)
    g, beta = o.gating(wl.bf16_bits(acts["a"]), wl.bf16_bits(acts["b"]), p["A_log"].numpy(),
                       p["dt_bias"].numpy())
    assert g.shape == (d.B, d.T, d.Hv)
    assert np.all(g > 0) and np.all(g <= 1)
    assert np.all((beta > 0) & (beta < 1))
    # larger a -> more decay (smaller g); larger b -> larger beta
    xs = o.f64_to_bf16(np.linspace(-4, 4, 33))
    gg, bb = o.gating(xs, xs, np.full(1, 1.0), np.zeros(1))
    assert np.all(np.diff(gg) < 0) and np.all(np.diff(bb) > 0)


# ----------------------------------------------------------------------------
# a1-a3 conv window, conv + SiLU, q/k normalisation
# ----------------------------------------------------------------------------
def _silu_lib(u):
    from scipy.special import expit
    return u * expit(u)


def test_conv_against_numpy_correlate(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(1)
    K, T, Cs = 4, 37, 6
    st = rng.standard_normal((K - 1, Cs))
    x = rng.standard_normal((T, Cs))
    w = rng.standard_normal((Cs, K))
    out, new_st = o.conv_silu_channels(st, x, w)
    X = np.concatenate([st, x], 0)
    for c in range(Cs):
        ref = np.correlate(X[:, c], w[c], mode="valid")
        assert np.allclose(out[:, c], _silu_lib(ref), rtol=1e-13, atol=1e-15)
    assert np.array_equal(new_st, X[-(K - 1):])


@pytest.mark.parametrize("tap", [0, 1, 2, 3])
def test_conv_one_hot_tap_is_a_shift(oracle_mod, tap):
    o = oracle_mod
    rng = np.random.default_rng(2)
    K, T, Cs = 4, 10, 3
    st = rng.standard_normal((K - 1, Cs))
    x = rng.standard_normal((T, Cs))
    w = np.zeros((Cs, K))
    w[:, tap] = 1.0
    out, _ = o.conv_silu_channels(st, x, w)
    X = np.concatenate([st, x], 0)
    lag = K - 1 - tap           # tap K-1 is the current token
    for t in range(T):
        assert np.array_equal(out[t], _silu_lib(X[K - 1 + t - lag]))


def test_conv_prefix_consistency_and_mask_skip(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(3)
    K, T, Cs = 4, 40, 5
    st = rng.standard_normal((K - 1, Cs))
    x = rng.standard_normal((T, Cs))
    w = rng.standard_normal((Cs, K))
    full, st_full = o.conv_silu_channels(st, x, w)
    a, st_a = o.conv_silu_channels(st, x[:17], w)
    b, st_b = o.conv_silu_channels(st_a, x[17:], w)
    assert np.array_equal(np.concatenate([a, b]), full) and np.array_equal(st_b, st_full)
    valid = rng.random(T) < 0.6
    m, st_m = o.conv_silu_channels(st, x, w, valid)
    u, st_u = o.conv_silu_channels(st, x[valid], w)
    assert np.array_equal(m[valid], u) and np.all(m[~valid] == 0) and np.array_equal(st_m, st_u)
    # fewer valid tokens than K-1: the old state shifts by that many rows
    valid2 = np.zeros(T, bool)
    valid2[5] = True
    _, st2 = o.conv_silu_channels(st, x, w, valid2)
    assert np.array_equal(st2, np.concatenate([st[1:], x[5:6]]))


def test_qk_norm_and_scale(oracle_mod):
    o = oracle_mod
    d = wl.WORKLOADS["tiny"].dims.with_(T=16, Dk=64, Dv=32)
    inp = wl.workload_inputs(wl.WORKLOADS["tiny"], d)
    q, k, v, _ = o.conv_update(d, wl.bf16_bits(inp["qkv"]), wl.bf16_bits(inp["conv_w"]))
    qn = np.linalg.norm(o.bf16_to_f64(q), axis=-1)
    kn = np.linalg.norm(o.bf16_to_f64(k), axis=-1)
    # |rms(x)| = sqrt(Dk) up to eps; q scaled by 1/Dk, k by 1/sqrt(Dk); bf16 rounding 2^-8
    assert np.allclose(qn, d.Dk ** -0.5, rtol=4e-3)
    assert np.allclose(kn, 1.0, rtol=4e-3)
    # v is the SiLU output itself (no norm): compare with a direct SiLU of the conv
    X = o.bf16_to_f64(wl.bf16_bits(inp["qkv"]))[0]
    w = o.bf16_to_f64(wl.bf16_bits(inp["conv_w"]))
    c0 = 2 * d.Hk * d.Dk
    Xp = np.concatenate([np.zeros((d.K - 1, d.C)), X], 0)
    for c in range(c0, c0 + 5):
        ref = _silu_lib(np.correlate(Xp[:, c], w[c], mode="valid"))
        assert np.array_equal(o.bf16_to_f64(v[0, :, 0, c - c0]), o.round_bf16(ref))


# ----------------------------------------------------------------------------
# a5 recurrence
# ----------------------------------------------------------------------------
def test_scalar_recurrence_golden(oracle_mod):
    o = oracle_mod
    gold = json.load(open(os.path.join(GOLDEN, "scalar_recurrence.json")))
    st = gold["steps"]
    col = lambda key: np.array([[_frac(s[key])] for s in st])
    y, S = o.head_recurrence(col("q"), col("k"), col("v"), col("g")[:, 0], col("beta")[:, 0],
                             np.array([[_frac(gold["S0"])]]), np.array([s["mask"] for s in st]))
    assert np.array_equal(y[:, 0], np.array([_frac(s["y"]) for s in st]))
    assert S[0, 0] == _frac(st[-1]["S"])
    for n in range(1, len(st) + 1):       # every intermediate state too
        _, Sn = o.head_recurrence(col("q")[:n], col("k")[:n], col("v")[:n], col("g")[:n, 0],
                                  col("beta")[:n, 0], np.array([[_frac(gold["S0"])]]),
                                  np.array([s["mask"] for s in st[:n]]))
        assert Sn[0, 0] == _frac(st[n - 1]["S"])


def _rand_head(rng, T, Dk, Dv, unit_k=True):
    q = rng.standard_normal((T, Dk)) / math.sqrt(Dk)
    k = rng.standard_normal((T, Dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, Dv))
    g = rng.uniform(0.5, 1.0, T)
    beta = rng.uniform(0.0, 1.0, T)
    S0 = 0.05 * rng.standard_normal((Dv, Dk))
    return q, k, v, g, beta, S0


def test_identity_step_leaves_state_unchanged(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(4)
    q, k, v, g, beta, S0 = _rand_head(rng, 9, 32, 16)
    y, S = o.head_recurrence(q, k, v, np.ones(9), np.zeros(9), S0)
    assert np.array_equal(S, S0)
    assert np.allclose(y, q @ S0.T, rtol=1e-13, atol=1e-15)


def test_full_write_makes_state_map_k_to_v(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(5)
    q, k, v, g, beta, S0 = _rand_head(rng, 12, 32, 24, unit_k=True)
    S = S0
    for t in range(12):
        y, S = o.head_recurrence(k[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], np.ones(1), S)
        assert np.allclose(S @ k[t], v[t], rtol=0, atol=1e-12)
        assert np.allclose(y[0], v[t], rtol=0, atol=1e-12)   # y read from the updated state


def test_zero_decay_forgets_history(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(6)
    q, k, v, g, beta, S0 = _rand_head(rng, 5, 16, 8, unit_k=False)
    g[-1] = 0.0
    _, S = o.head_recurrence(q, k, v, g, beta, S0)
    assert np.allclose(S, beta[-1] * np.outer(v[-1], k[-1]), rtol=1e-14, atol=0)


def test_joint_linearity_in_state_and_values(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(7)
    q, k, v, g, beta, S0 = _rand_head(rng, 20, 16, 12)
    v2 = rng.standard_normal(v.shape)
    S02 = rng.standard_normal(S0.shape)
    y1, S1 = o.head_recurrence(q, k, v, g, beta, S0)
    y2, S2 = o.head_recurrence(q, k, v2, g, beta, S02)
    y3, S3 = o.head_recurrence(q, k, 2 * v - 3 * v2, g, beta, 2 * S0 - 3 * S02)
    assert np.allclose(y3, 2 * y1 - 3 * y2, atol=1e-11)
    assert np.allclose(S3, 2 * S1 - 3 * S2, atol=1e-11)


def _brute_force(q, k, v, g, beta, S0):
    """S_T = S0 P_1..P_T + sum_t beta_t v_t k_t^T P_{t+1}..P_T with
    P_t = g_t (I - beta_t k_t k_t^T); y_t = S_t q_t."""
    T, Dk = k.shape
    I = np.eye(Dk)
    P = [g[t] * (I - beta[t] * np.outer(k[t], k[t])) for t in range(T)]
    ys, Ss = [], []
    for n in range(1, T + 1):
        prod = I.copy()
        for t in range(n):
            prod = prod @ P[t]
        S = S0 @ prod
        for t in range(n):
            tail = I.copy()
            for s in range(t + 1, n):
                tail = tail @ P[s]
            S = S + beta[t] * np.outer(v[t], k[t]) @ tail
        Ss.append(S)
        ys.append(S @ q[n - 1])
    return np.array(ys), Ss[-1]


@pytest.mark.parametrize("Dk,Dv", [(4, 3), (3, 5), (6, 6)])
def test_brute_force_matrix_form(oracle_mod, Dk, Dv):
    o = oracle_mod
    rng = np.random.default_rng(8 + Dk)
    q, k, v, g, beta, S0 = _rand_head(rng, 6, Dk, Dv, unit_k=False)
    y, S = o.head_recurrence(q, k, v, g, beta, S0)
    yb, Sb = _brute_force(q, k, v, g, beta, S0)
    assert np.allclose(y, yb, rtol=1e-12, atol=1e-13)
    assert np.allclose(S, Sb, rtol=1e-12, atol=1e-13)


def test_prefix_consistency(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(9)
    q, k, v, g, beta, S0 = _rand_head(rng, 50, 32, 32)
    y, S = o.head_recurrence(q, k, v, g, beta, S0)
    ya, Sa = o.head_recurrence(q[:21], k[:21], v[:21], g[:21], beta[:21], S0)
    yb, Sb = o.head_recurrence(q[21:], k[21:], v[21:], g[21:], beta[21:], Sa)
    assert np.array_equal(np.concatenate([ya, yb]), y) and np.array_equal(Sb, S)


def test_mask_equals_unpadded_run(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(10)
    q, k, v, g, beta, S0 = _rand_head(rng, 40, 16, 8)
    m = (rng.random(40) < 0.5).astype(np.uint8)
    y, S = o.head_recurrence(q, k, v, g, beta, S0, m)
    sel = m != 0
    yu, Su = o.head_recurrence(q[sel], k[sel], v[sel], g[sel], beta[sel], S0)
    assert np.array_equal(y[sel], yu) and np.array_equal(S, Su)
    assert np.all(y[~sel] == 0.0)
    y0, S_none = o.head_recurrence(q, k, v, g, beta, S0, np.zeros(40, np.uint8))
    assert np.array_equal(S_none, S0) and np.all(y0 == 0.0)


def test_gqa_blocked_head_mapping(oracle_mod):
    """Hv = 4 on Hk = 2 must equal Hv = Hk = 4 with q, k repeated blockwise
    (numpy.repeat: k-head 0 serves v-heads 0, 1; k-head 1 serves 2, 3)."""
    o = oracle_mod
    d = wl.Dims(B=2, T=7, Hk=2, Hv=4, Dk=8, Dv=8)
    rng = np.random.default_rng(11)
    q = o.f64_to_bf16(rng.standard_normal((d.B, d.T, d.Hk, d.Dk)) * 0.1)
    k = o.f64_to_bf16(rng.standard_normal((d.B, d.T, d.Hk, d.Dk)) * 0.3)
    v = o.f64_to_bf16(rng.standard_normal((d.B, d.T, d.Hv, d.Dv)))
    g = rng.uniform(0.6, 1, (d.B, d.T, d.Hv))
    beta = rng.uniform(0, 1, (d.B, d.T, d.Hv))
    S0 = rng.standard_normal((d.B, d.Hv, d.Dv, d.Dk)) * 0.05
    y, S = o.recurrence(d, q, k, v, g, beta, S0, threads=1)
    d4 = d.with_(Hk=4)
    y4, S4 = o.recurrence(d4, np.repeat(q, 2, axis=2), np.repeat(k, 2, axis=2), v, g, beta, S0,
                          threads=1)
    assert np.array_equal(y, y4) and np.array_equal(S, S4)
    # the modulo mapping (hv % Hk) differs, so the pin can tell them apart
    y_mod, _ = o.recurrence(d4, np.tile(q, (1, 1, 2, 1)), np.tile(k, (1, 1, 2, 1)), v, g, beta, S0,
                            threads=1)
    assert not np.allclose(y, y_mod)


# ----------------------------------------------------------------------------
# a7 chunked form == sequential form (f64)
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [1, 16, 64])
@pytest.mark.parametrize("masked", [False, True])
def test_chunked_equals_sequential(oracle_mod, chunk, masked):
    o = oracle_mod
    rng = np.random.default_rng(12 + chunk)
    T = 150
    q, k, v, g, beta, S0 = _rand_head(rng, T, 32, 24)
    g = np.exp(-rng.uniform(0, 3, T))          # includes strong decay
    mask = (rng.random(T) < 0.7).astype(np.uint8) if masked else None
    y, S = o.head_recurrence(q, k, v, g, beta, S0, mask)
    yc, Sc = o.chunked_head(q, k, v, g, beta, S0, mask, chunk=chunk)
    assert np.linalg.norm(yc - y) <= 1e-12 * np.linalg.norm(y)
    assert np.linalg.norm(Sc - S) <= 1e-12 * np.linalg.norm(S)


# ----------------------------------------------------------------------------
# the composed core on the tiny workload
# ----------------------------------------------------------------------------
def test_core_tiny_and_pair_sampling_agree(oracle_mod):
    o = oracle_mod
    w = wl.WORKLOADS["tiny"]
    inp = wl.workload_inputs(w)
    d = inp["dims"]
    args = (d, wl.bf16_bits(inp["qkv"]), wl.bf16_bits(inp["conv_w"]), wl.bf16_bits(inp["a"]),
            wl.bf16_bits(inp["b"]), inp["A_log"].numpy(), inp["dt_bias"].numpy(),
            wl.bf16_bits(inp["conv_state"]), inp["state"].numpy().astype(np.float64))
    full = o.layer_core(*args)
    assert full["y"].shape == (1, 8, 2, 32) and full["state"].shape == (1, 2, 32, 32)
    assert np.all(np.isfinite(full["y"]))
    part = o.layer_core(*args, pairs=[(0, 1)])["heads"][(0, 1)]
    assert np.array_equal(part["y"], full["y"][0, :, 1])
    assert np.array_equal(part["state"], full["state"][0, 1])
    # sampled carried decode == full carried decode on the sampled head
    steps = [{k: wl.bf16_bits(v) for k, v in wl.decode_step_inputs(w, i, d.with_(T=1)).items()}
             for i in range(4)]
    d1 = d.with_(T=1)
    yf, sf, _ = o.decode(d1, steps, *args[2:3], *args[5:8], args[8])
    yp, sp, _ = o.decode(d1, steps, *args[2:3], *args[5:8], args[8], pairs=[(0, 1)])
    for i in range(4):
        assert np.array_equal(yp[i][(0, 1)], yf[i][0, 1])
    assert np.array_equal(sp[(0, 1)], sf[0, 1])


def test_decode_steps_equal_one_prefill(oracle_mod):
    """T single-token steps with carried states == one call over T tokens
    (state carried in f64 here so the comparison is exact)."""
    o = oracle_mod
    d = wl.Dims(B=2, T=6, Hk=1, Hv=2, Dk=32, Dv=32)
    inp = wl.workload_inputs(wl.WORKLOADS["tiny"], d)
    qkv, a, b = wl.bf16_bits(inp["qkv"]), wl.bf16_bits(inp["a"]), wl.bf16_bits(inp["b"])
    cw = wl.bf16_bits(inp["conv_w"])
    A_log, dt = inp["A_log"].numpy(), inp["dt_bias"].numpy()
    full = o.layer_core(d, qkv, cw, a, b, A_log, dt)
    cs, st = None, None
    d1 = d.with_(T=1)
    for t in range(d.T):
        out = o.layer_core(d1, qkv[:, t:t + 1], cw, a[:, t:t + 1], b[:, t:t + 1], A_log, dt, cs, st)
        assert np.array_equal(out["y"][:, 0], full["y"][:, t])
        cs, st = out["conv_state"], out["state"]
    assert np.array_equal(st, full["state"]) and np.array_equal(cs, full["conv_state"])


# ----------------------------------------------------------------------------
# f-1 RMSNormGated: pinned to torch's rms_norm and silu (float64 on the CPU)
# ----------------------------------------------------------------------------
def test_rmsnorm_gated_against_torch(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(21)
    Dv = 64
    y = o.f64_to_bf16(rng.standard_normal((3, 5, 4, Dv)) * 0.1)
    z = o.f64_to_bf16(rng.standard_normal((3, 5, 4, Dv)))
    w = rng.uniform(0.5, 1.5, Dv).astype(np.float32)
    eps = 1e-6
    got = o.rmsnorm_gated(y, z, w, eps)
    yt = torch.from_numpy(o.bf16_to_f64(y))
    zt = torch.from_numpy(o.bf16_to_f64(z))
    ref = torch.nn.functional.silu(zt) * torch.nn.functional.rms_norm(
        yt, (Dv,), weight=torch.from_numpy(w.astype(np.float64)), eps=eps)
    ref_bits = ref.to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # one rounding from f64 vs f64 -> f32 -> bf16: equal except on exact f32 ties
    assert np.mean(got == ref_bits) > 0.999


def test_rmsnorm_gated_closed_forms(oracle_mod):
    o = oracle_mod
    Dv = 32
    y = o.f64_to_bf16(np.full((1, Dv), -0.5))          # constant row: y / rms(y) = -1 (eps negligible)
    z = o.f64_to_bf16(np.full((1, Dv), 8.0))           # silu(8) = 8 sigmoid(8)
    w = np.linspace(0.5, 2.0, Dv).astype(np.float32)
    out = o.bf16_to_f64(o.rmsnorm_gated(y, z, w, 1e-6))
    expect = -(8.0 / (1.0 + math.exp(-8.0))) * w.astype(np.float64) / math.sqrt(1.0 + 4e-6)
    assert np.allclose(out, expect, rtol=2 ** -8)
    zero = o.bf16_to_f64(o.rmsnorm_gated(o.f64_to_bf16(np.zeros((2, Dv))), z.repeat(2, 0), w, 1e-6))
    assert np.all(zero == 0.0)                          # a zero row (masked step) stays zero


# ----------------------------------------------------------------------------
# f-3 vectorized gating (one decay factor per key channel)
# ----------------------------------------------------------------------------
def test_vec_gating_with_equal_channels_is_the_scalar_recurrence(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(31)
    q, k, v, g, beta, S0 = _rand_head(rng, 30, 16, 12)
    y, S = o.head_recurrence(q, k, v, g, beta, S0)
    yv, Sv = o.head_recurrence_vec(q, k, v, np.repeat(g[:, None], 16, axis=1), beta, S0)
    assert np.array_equal(y, yv) and np.array_equal(S, Sv)


@pytest.mark.parametrize("Dk,Dv", [(4, 3), (5, 6)])
def test_vec_gating_brute_force(oracle_mod, Dk, Dv):
    """S_T = S0 P_1..P_T + sum_t beta_t v_t k_t^T P_{t+1}..P_T with
    P_t = diag(g_t) (I - beta_t k_t k_t^T)."""
    o = oracle_mod
    rng = np.random.default_rng(32 + Dk)
    T = 6
    q, k, v, _, beta, S0 = _rand_head(rng, T, Dk, Dv, unit_k=False)
    G = rng.uniform(0.3, 1.0, (T, Dk))
    y, S = o.head_recurrence_vec(q, k, v, G, beta, S0)
    I = np.eye(Dk)
    P = [np.diag(G[t]) @ (I - beta[t] * np.outer(k[t], k[t])) for t in range(T)]
    Sb = S0.copy()
    for t in range(T):
        Sb = Sb @ P[t] + beta[t] * np.outer(v[t], k[t])
        assert np.allclose(y[t], Sb @ q[t], rtol=1e-12, atol=1e-13)
    assert np.allclose(S, Sb, rtol=1e-12, atol=1e-13)


def test_vec_gating_zero_channel_forgets_that_column(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(33)
    q, k, v, _, beta, S0 = _rand_head(rng, 1, 8, 5, unit_k=False)
    G = np.ones((1, 8))
    G[0, 3] = 0.0
    _, S = o.head_recurrence_vec(q, k, v, G, beta, S0)
    Sd = S0.copy()
    Sd[:, 3] = 0.0
    delta = beta[0] * (v[0] - Sd @ k[0])
    assert np.allclose(S, Sd + np.outer(delta, k[0]), rtol=1e-14, atol=1e-15)
