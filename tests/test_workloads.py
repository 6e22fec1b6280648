"""The seeded synthetic inputs (no GPU): shapes and dtypes of the layouts the
ABI takes, the stated distributions, determinism per seed, and the ragged
batch's right-padded masks."""
import numpy as np
import torch

from gated_deltanet_linear_04_gb300 import workloads as wl


def test_every_workload_has_the_abi_shapes():
    for w in wl.WORKLOADS.values():
        d = w.dims.with_(T=min(w.dims.T, 64), B=min(w.dims.B, 4))
        inp = wl.workload_inputs(w, d)
        assert inp["qkv"].shape == (d.B, d.T, 2 * d.Hk * d.Dk + d.Hv * d.Dv) and inp["qkv"].dtype == torch.bfloat16
        assert inp["conv_w"].shape == (d.C, d.K) and inp["conv_w"].dtype == torch.bfloat16
        assert inp["a"].shape == inp["b"].shape == (d.B, d.T, d.Hv)
        assert inp["A_log"].shape == inp["dt_bias"].shape == (d.Hv,) and inp["A_log"].dtype == torch.float32
        assert inp["conv_state"].shape == (d.B, d.K - 1, d.C)
        assert inp["state"].shape == (d.B, d.Hv, d.Dv, d.Dk) and inp["state"].dtype == torch.float32
        assert d.Hv % d.Hk == 0


def test_inputs_are_deterministic_per_seed():
    w = wl.WORKLOADS["tiny"]
    a, b = wl.workload_inputs(w), wl.workload_inputs(w)
    for k in ("qkv", "conv_w", "a", "b", "A_log", "dt_bias", "conv_state", "state"):
        assert torch.equal(a[k], b[k]), k
    s0, s1 = wl.decode_step_inputs(w, 0), wl.decode_step_inputs(w, 1)
    assert not torch.equal(s0["qkv"], s1["qkv"])                   # fresh inputs every decode step


def test_stated_distributions():
    d = wl.Dims(B=4, T=512, Hk=2, Hv=8, Dk=128, Dv=128)
    p = wl.make_params(d, 5)
    A = torch.exp(p["A_log"])
    assert float(A.min()) >= 1.0 and float(A.max()) <= 16.0       # A_log = log U[1, 16]
    act = wl.make_activations(d, 6)
    x = act["qkv"].float()
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01
    w = p["conv_w"].float()
    assert abs(float(w.std()) - 0.5) < 0.02
    st = wl.make_states(d, 7, "normal", "normal")["state"]
    assert abs(float(st.std()) - 0.05) < 0.002
    z = wl.make_states(d, 7, "zeros", "zeros")
    assert not z["conv_state"].any() and not z["state"].any()


def test_ragged_rows_are_right_padded_within_the_stated_range():
    w = wl.WORKLOADS["prefill_ragged"]
    lens = wl.workload_lengths(w)
    assert lens.shape == (w.dims.B,)
    assert int(lens.min()) >= w.len_lo and int(lens.max()) <= w.len_hi <= w.dims.T
    m = wl.right_padded_mask(lens, w.dims.T).numpy()
    assert m.dtype == np.uint8
    for b, L in enumerate(lens.tolist()):
        assert m[b, :L].all() and not m[b, L:].any()
    assert torch.equal(lens, wl.workload_lengths(w))
