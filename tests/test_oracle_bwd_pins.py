"""Pins of the oracle's backward pass (the gradient of the recurrence), on
the CPU.  The pages define the forward recurrence only, so its derivative is
pinned against the forward oracle itself by central finite differences: a
random linear loss L = <y, Wy> + <S_T, WS> is differentiated with respect to
every scalar input of small cases and compared with the reverse pass given
dy = Wy and dS_T = WS.  A dropped term, a wrong sign or an index slip in the
reverse pass changes some gradient entry far beyond the finite-difference
error (~1e-9 here)."""
import numpy as np
import pytest


def _inputs(T, Dk, Dv, seed, masked, with_s0):
    rng = np.random.default_rng(seed)
    q = rng.normal(size=(T, Dk)) * 0.5
    k = rng.normal(size=(T, Dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.normal(size=(T, Dv))
    g = rng.uniform(0.3, 0.99, size=T)
    beta = rng.uniform(0.1, 0.9, size=T)
    S0 = rng.normal(size=(Dv, Dk)) * 0.3 if with_s0 else None
    mask = None
    if masked:
        mask = (rng.uniform(size=T) < 0.7).astype(np.uint8)
        mask[0] = 1
        mask[-1] = 0
    Wy = rng.normal(size=(T, Dv))
    WS = rng.normal(size=(Dv, Dk))
    return dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0, mask=mask), Wy, WS


def _loss(oracle_mod, x, Wy, WS):
    S0 = np.zeros((x["v"].shape[1], x["q"].shape[1])) if x["S0"] is None else x["S0"]
    y, S = oracle_mod.head_recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], S0, x["mask"])
    return float(np.sum(y * Wy) + np.sum(S * WS))


def _check_fd(oracle_mod, T, Dk, Dv, seed, masked, with_s0, h=1e-6, tol=1e-6):
    x, Wy, WS = _inputs(T, Dk, Dv, seed, masked, with_s0)
    grads = oracle_mod.head_recurrence_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], Wy, WS, x["mask"])
    names = [("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta")]
    if with_s0:
        names.append(("S0", "dS0"))
    for name, gname in names:
        base = x[name]
        fd = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = {kk: (vv.copy() if isinstance(vv, np.ndarray) else vv) for kk, vv in x.items()}
            xm = {kk: (vv.copy() if isinstance(vv, np.ndarray) else vv) for kk, vv in x.items()}
            xp[name][idx] += h
            xm[name][idx] -= h
            fd[idx] = (_loss(oracle_mod, xp, Wy, WS) - _loss(oracle_mod, xm, Wy, WS)) / (2 * h)
        got = grads[gname]
        err = np.abs(got - fd).max()
        scale = max(1.0, np.abs(fd).max())
        assert err <= tol * scale, "%s: max |analytic - finite difference| = %.3e" % (gname, err)
    if not with_s0:
        # the gradient of the (zero) initial state is still that of S0
        x0 = dict(x, S0=np.zeros((Dv, Dk)))
        g0 = oracle_mod.head_recurrence_bwd(x0["q"], x0["k"], x0["v"], x0["g"], x0["beta"], x0["S0"], Wy, WS,
                                            x0["mask"])
        assert np.allclose(g0["dS0"], grads["dS0"], rtol=0, atol=1e-12)
    return grads, x


@pytest.mark.parametrize("T,Dk,Dv,seed,masked,with_s0", [
    (5, 3, 2, 1, False, True),
    (6, 2, 3, 2, True, True),
    (4, 4, 1, 3, False, False),
    (7, 3, 3, 4, True, False),
])
def test_bwd_matches_finite_differences(T, Dk, Dv, seed, masked, with_s0, oracle_mod):
    _check_fd(oracle_mod, T, Dk, Dv, seed, masked, with_s0)


def test_bwd_masked_steps_have_zero_gradients(oracle_mod):
    grads, x = _check_fd(oracle_mod, 7, 3, 3, 4, True, True)
    off = x["mask"] == 0
    assert off.any()
    for gname in ("dq", "dk", "dv", "dg", "dbeta"):
        assert np.all(grads[gname][off] == 0.0), gname


def test_bwd_no_output_gradient_gives_zero(oracle_mod):
    x, _, _ = _inputs(5, 3, 2, 9, False, True)
    z = oracle_mod.head_recurrence_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], np.zeros((5, 2)),
                                       None, None)
    for gname, a in z.items():
        assert np.all(a == 0.0), gname


def test_bwd_sums_q_k_gradients_over_shared_heads(oracle_mod):
    # two v-heads read the same k-head: dq, dk of the k-head are the sums of
    # the per-head gradients (finite differences through both heads)
    from gated_deltanet_linear_04_gb300 import workloads as wl
    d = wl.Dims(B=1, T=4, Hk=1, Hv=2, Dk=3, Dv=2)
    rng = np.random.default_rng(5)
    qb = oracle_mod.f64_to_bf16(rng.normal(size=(1, 4, 1, 3)) * 0.5)
    kb = oracle_mod.f64_to_bf16(rng.normal(size=(1, 4, 1, 3)) * 0.5)
    vb = oracle_mod.f64_to_bf16(rng.normal(size=(1, 4, 2, 2)))
    g = rng.uniform(0.5, 0.95, size=(1, 4, 2))
    beta = rng.uniform(0.2, 0.8, size=(1, 4, 2))
    S0 = rng.normal(size=(1, 2, 2, 3)) * 0.2
    Wy = rng.normal(size=(1, 4, 2, 2))
    WS = rng.normal(size=(1, 2, 2, 3))
    out = oracle_mod.recurrence_bwd(d, qb, kb, vb, g, beta, S0, Wy, WS, threads=1)
    q, k, v = (oracle_mod.bf16_to_f64(a) for a in (qb, kb, vb))

    def loss(qq, kk):
        tot = 0.0
        for hv in range(2):
            y, S = oracle_mod.head_recurrence(qq, kk, v[0, :, hv], g[0, :, hv], beta[0, :, hv], S0[0, hv])
            tot += np.sum(y * Wy[0, :, hv]) + np.sum(S * WS[0, hv])
        return tot

    h = 1e-6
    for which in ("dq", "dk"):
        base_q, base_k = q[0, :, 0].copy(), k[0, :, 0].copy()
        fd = np.zeros((4, 3))
        for t in range(4):
            for j in range(3):
                qp, qm, kp, km = base_q.copy(), base_q.copy(), base_k.copy(), base_k.copy()
                if which == "dq":
                    qp[t, j] += h
                    qm[t, j] -= h
                else:
                    kp[t, j] += h
                    km[t, j] -= h
                fd[t, j] = (loss(qp, kp) - loss(qm, km)) / (2 * h)
        assert np.abs(out[which][0, :, 0] - fd).max() <= 1e-6 * max(1.0, np.abs(fd).max()), which


@pytest.mark.parametrize("T,Dk,Dv,chunk,seed,masked,with_s0", [
    (9, 4, 3, 4, 1, False, True),      # two full chunks and a one-step tail
    (20, 8, 6, 7, 2, True, True),      # chunk size that divides nothing
    (33, 16, 8, 64, 3, True, False),   # one partial chunk
    (50, 8, 8, 1, 4, False, True),     # chunks of one step: the sequential reverse itself
    (70, 8, 12, 16, 5, True, True),
])
def test_chunked_bwd_matches_sequential_reverse(T, Dk, Dv, chunk, seed, masked, with_s0, oracle_mod):
    """The chunked backward (the reverse of the chunk products, in numpy) and
    the step-by-step reverse (in C) are independent derivations of the same
    gradient; they agree to rounding."""
    x, Wy, WS = _inputs(T, Dk, Dv, seed, masked, with_s0)
    ref = oracle_mod.head_recurrence_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], Wy, WS, x["mask"])
    got = oracle_mod.chunked_head_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], Wy, WS, x["mask"],
                                      chunk=chunk)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dS0"):
        err = np.linalg.norm(got[name] - ref[name]) / max(np.linalg.norm(ref[name]), 1e-300)
        assert err < 1e-12, (name, err)
    if x["mask"] is not None:
        off = x["mask"] == 0
        for name in ("dq", "dk", "dv", "dg", "dbeta"):
            assert np.all(got[name][off] == 0.0), name


def test_chunked_bwd_strong_decay(oracle_mod):
    """Gates down to e^-32: every term of d(log g_t) carries the factor g_t,
    so dg = d(log g) / g stays accurate (a difference of prefix sums lost
    three digits here)."""
    rng = np.random.default_rng(9)
    T, Dk, Dv = 80, 8, 6
    q = rng.normal(size=(T, Dk))
    k = rng.normal(size=(T, Dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.normal(size=(T, Dv))
    g = np.exp(-rng.uniform(0.0, 32.0, size=T))
    beta = rng.uniform(0.1, 0.9, size=T)
    S0 = rng.normal(size=(Dv, Dk))
    dy = rng.normal(size=(T, Dv))
    dST = rng.normal(size=(Dv, Dk))
    ref = oracle_mod.head_recurrence_bwd(q, k, v, g, beta, S0, dy, dST)
    for chunk in (16, 64):
        got = oracle_mod.chunked_head_bwd(q, k, v, g, beta, S0, dy, dST, chunk=chunk)
        for name in ("dq", "dk", "dv", "dg", "dbeta", "dS0"):
            err = np.linalg.norm(got[name] - ref[name]) / np.linalg.norm(ref[name])
            assert err < 1e-12, (chunk, name, err)
        assert np.max(np.abs(got["dg"] - ref["dg"]) / np.abs(ref["dg"])) < 1e-11
