"""The pins must have teeth: plant plausible mistakes in a copy of the oracle
(on the CPU) and check that at least one pin fails for each of them."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle.core as oc
from tests import test_oracle_bwd_pins as bwd_pins
from tests import test_oracle_pins as pins

C_MUTATIONS = {
    "delta_sign": ("double delta = beta[t] * (vt[i] - kv);", "double delta = beta[t] * (kv - vt[i]);"),
    "no_decay": ("S[(size_t)i * Dk + j] *= g[t];", "S[(size_t)i * Dk + j] *= 1.0;"),
    "update_with_q": ("for (int j = 0; j < Dk; ++j) Si[j] += delta * kt[j];",
                      "for (int j = 0; j < Dk; ++j) Si[j] += delta * qt[j];"),
    "output_with_k": ("acc += Si[j] * qt[j];", "acc += Si[j] * kt[j];"),
    "mask_ignored": ("if (mask != NULL && mask[t] == 0) {", "if (mask != NULL && mask[t] == 2) {"),
    "beta_dropped": ("double delta = beta[t] * (vt[i] - kv);", "double delta = (vt[i] - kv);"),
}

VEC_MUTATION = ("S[(size_t)i * Dk + j] *= gt[j];", "S[(size_t)i * Dk + j] *= gt[i % Dk];")

C_PINS = [
    pins.test_scalar_recurrence_golden,
    pins.test_full_write_makes_state_map_k_to_v,
    pins.test_zero_decay_forgets_history,
    pins.test_identity_step_leaves_state_unchanged,
    pins.test_mask_equals_unpadded_run,
]


def _build_mutant(tmp_path, name, old, new):
    src = open(oc._SRC).read()
    # the scalar-gate function comes first in the file; plant the mistake there
    assert src.count(old) >= 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new, 1))
    so = tmp_path / f"lib{name}.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(path)])
    lib = ctypes.CDLL(str(so))
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_delta_rule_head.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp,
                                           ctypes.POINTER(ctypes.c_uint8), dp, dp]
    lib.oracle_delta_rule_head.restype = None
    lib.oracle_delta_rule_head_bwd.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp,
                                               ctypes.POINTER(ctypes.c_uint8), dp, dp, dp, dp, dp, dp, dp, dp, dp]
    lib.oracle_delta_rule_head_bwd.restype = ctypes.c_int
    return lib


def _some_pin_fails(pin_fns, **kw):
    for fn in pin_fns:
        try:
            fn(**kw)
        except AssertionError:
            return True
    return False


@pytest.mark.parametrize("name", sorted(C_MUTATIONS))
def test_c_mutation_is_caught(name, tmp_path, monkeypatch):
    old, new = C_MUTATIONS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    monkeypatch.setattr(oc, "_lib", lib)
    assert _some_pin_fails(C_PINS, oracle_mod=oc), name


# plausible mistakes in the backward pass (the forward stays intact, so the
# finite-difference pins expose them)
BWD_MUTATIONS = {
    "bwd_dq_dropped": ("dqt[j] += St[(size_t)i * Dk + j] * dyt[i];", "dqt[j] += 0.0 * dyt[i];"),
    "bwd_dk_sign": ("dkt[j] -= Sp[(size_t)i * Dk + j] * du[i];", "dkt[j] += Sp[(size_t)i * Dk + j] * du[i];"),
    "bwd_no_decay_carry": ("for (size_t e = 0; e < n; ++e) dS[e] *= g[t];",
                           "for (size_t e = 0; e < n; ++e) dS[e] *= 1.0;"),
    "bwd_dbeta_without_u": ("dbeta[t] += ddel[i] * u[(size_t)t * Dv + i];", "dbeta[t] += ddel[i];"),
    "bwd_dg_wrong_state": ("acc += dS[e] * Sprev[e];", "acc += dS[e] * St[e];"),
    "bwd_du_without_beta": ("du[i] = beta[t] * ddel[i];", "du[i] = ddel[i];"),
}

BWD_PINS = [lambda oracle_mod: bwd_pins._check_fd(oracle_mod, 5, 3, 2, 1, False, True),
            lambda oracle_mod: bwd_pins._check_fd(oracle_mod, 6, 2, 3, 2, True, True)]


@pytest.mark.parametrize("name", sorted(BWD_MUTATIONS))
def test_bwd_mutation_is_caught(name, tmp_path, monkeypatch):
    old, new = BWD_MUTATIONS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    monkeypatch.setattr(oc, "_lib", lib)
    assert _some_pin_fails(BWD_PINS, oracle_mod=oc), name


def _mut_gqa_modulo(d, hv):
    return hv % d.Hk


def _mut_softplus_sign(x):
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) - np.log1p(np.exp(-np.abs(x)))


PY_MUTATIONS = {
    "gqa_modulo": ("k_head_of", _mut_gqa_modulo, [pins.test_gqa_blocked_head_mapping]),
    "softplus_sign": ("softplus", _mut_softplus_sign,
                      [pins.test_gating_golden_points, pins.test_softplus_sigmoid_against_library]),
}


@pytest.mark.parametrize("name", sorted(PY_MUTATIONS))
def test_python_mutation_is_caught(name, monkeypatch):
    attr, fn, pin_fns = PY_MUTATIONS[name]
    oc.build_oracle()
    monkeypatch.setattr(oc, attr, fn)
    assert _some_pin_fails(pin_fns, oracle_mod=oc), name


def test_conv_tap_order_mutation_is_caught(monkeypatch):
    orig = oc.conv_silu_channels

    def flipped(state_rows, x_rows, w, valid=None):
        return orig(state_rows, x_rows, np.asarray(w)[:, ::-1], valid)

    monkeypatch.setattr(oc, "conv_silu_channels", flipped)
    assert _some_pin_fails([pins.test_conv_against_numpy_correlate], oracle_mod=oc)


def test_q_scale_mutation_is_caught(monkeypatch):
    orig = oc.rms_normalize

    def wrong_norm(x, eps):      # forgets the 1/sqrt(mean) factor
        return np.asarray(x, dtype=np.float64) * 0 + orig(x, eps) * 2.0

    monkeypatch.setattr(oc, "rms_normalize", wrong_norm)
    assert _some_pin_fails([pins.test_qk_norm_and_scale], oracle_mod=oc)


def test_vec_gating_row_instead_of_column_is_caught(tmp_path, monkeypatch):
    src = open(oc._SRC).read()
    old, new = VEC_MUTATION
    assert src.count(old) == 1
    path = tmp_path / "vec.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libvec.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(path)])
    lib = ctypes.CDLL(str(so))
    dp = ctypes.POINTER(ctypes.c_double)
    for name in ("oracle_delta_rule_head", "oracle_delta_rule_head_vec"):
        f = getattr(lib, name)
        f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_uint8),
                      dp, dp]
        f.restype = None
    monkeypatch.setattr(oc, "_lib", lib)
    assert _some_pin_fails([lambda oracle_mod: pins.test_vec_gating_brute_force(oracle_mod, 5, 6),
                            pins.test_vec_gating_zero_channel_forgets_that_column], oracle_mod=oc)
