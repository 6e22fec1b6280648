"""Parity at the full workload sizes, in the launch configuration the
benchmark times.  The oracle recomputes sampled (b, hv) heads one by one; the
rest is checked through properties that hold at any size."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_04_gb300 import workloads as wl
from tests import _util as U

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def gdn():
    from gated_deltanet_linear_04_gb300.build import build_library
    build_library()
    from gated_deltanet_linear_04_gb300 import gdn as g
    torch.cuda.set_device(0)
    return g


def _decode_case(gdn, name, pairs, n_steps=None):
    w = wl.WORKLOADS[name]
    d = w.dims
    n = n_steps or w.steps
    inp = wl.workload_inputs(w)
    dev = lambda x: x.to(DEV)
    cs, st = dev(inp["conv_state"]).clone(), dev(inp["state"]).clone()
    conv_w, A_log, dt = dev(inp["conv_w"]), dev(inp["A_log"]), dev(inp["dt_bias"])
    steps = [wl.decode_step_inputs(w, i) for i in range(n)]
    ys = []
    y = torch.empty((d.B, d.Hv, d.Dv), dtype=torch.bfloat16, device=DEV)
    d1 = d.with_(T=1)
    for s in steps:
        gdn.gdn_recurrent_decode(d1, dev(s["qkv"][:, 0].contiguous()), conv_w, cs, dev(s["a"][:, 0].contiguous()),
                                 dev(s["b"][:, 0].contiguous()), A_log, dt, st, None, y)
        ys.append(torch.stack([y[b, hv] for (b, hv) in pairs]).float().cpu().numpy())
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    sbits = [{k: wl.bf16_bits(s[k]) for k in ("qkv", "a", "b")} for s in steps]
    yr, sr, _ = oracle.decode(d, sbits, wl.bf16_bits(inp["conv_w"]), inp["A_log"].numpy(), inp["dt_bias"].numpy(),
                              wl.bf16_bits(inp["conv_state"]), inp["state"].numpy().astype(np.float64), pairs=pairs)
    got = np.stack(ys)                                        # [n, P, Dv]
    ref = np.stack([np.stack([yr[i][p] for p in pairs]) for i in range(n)])
    U.assert_y_close(got, ref)
    st_h = st.cpu().numpy()
    for (b, hv) in pairs:
        U.assert_state_close(st_h[b, hv], sr[(b, hv)], "state (%d,%d)" % (b, hv))
    # property at any size: after >= K-1 steps the conv state holds the last
    # K-1 raw inputs of every channel, oldest first
    if n >= d.K - 1:
        last = torch.stack([steps[n - d.K + 1 + j]["qkv"][:, 0] for j in range(d.K - 1)], 1)
        assert torch.equal(cs.cpu(), last)


def test_decode_b1_1024_steps(gdn):
    _decode_case(gdn, "decode_b1", [(0, 0), (0, 17), (0, 31)])


def test_decode_b128_256_steps(gdn):
    _decode_case(gdn, "decode_b128", [(0, 0), (77, 12), (127, 31)])


def _prefill_case(gdn, name, pairs, chunk):
    w = wl.WORKLOADS[name]
    inp = wl.workload_inputs(w)
    d = inp["dims"]
    dev = lambda x: None if x is None else x.to(DEV)
    mask = inp["mask"]
    cs = dev(inp["conv_state"]).clone()
    y, s = gdn.core_prefill(d, dev(inp["qkv"]), dev(inp["conv_w"]), dev(inp["a"]), dev(inp["b"]), dev(inp["A_log"]),
                            dev(inp["dt_bias"]), cs, dev(inp["state"]), dev(mask), chunk)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    ref = oracle.layer_core(d, wl.bf16_bits(inp["qkv"]), wl.bf16_bits(inp["conv_w"]), wl.bf16_bits(inp["a"]),
                            wl.bf16_bits(inp["b"]), inp["A_log"].numpy(), inp["dt_bias"].numpy(),
                            wl.bf16_bits(inp["conv_state"]), inp["state"].numpy().astype(np.float64),
                            None if mask is None else mask.numpy(), pairs=pairs)["heads"]
    for (b, hv) in pairs:
        got = y[b, :, hv].float().cpu().numpy()
        U.assert_y_close(got, ref[(b, hv)]["y"], "y (%d,%d)" % (b, hv))
        U.assert_state_close(s[b, hv].cpu().numpy(), ref[(b, hv)]["state"], "state (%d,%d)" % (b, hv))
    if mask is not None:
        m = mask.to(DEV)
        pad = (m == 0)
        assert int(y[pad].abs().max().item() if pad.any() else 0) == 0, "padded y must be exactly zero"
    return y, s


@pytest.mark.parametrize("chunk", [0, 64])
def test_prefill_t8192(gdn, chunk):
    _prefill_case(gdn, "prefill_t8192", [(0, 0), (0, 13), (0, 31)], chunk)


@pytest.mark.parametrize("chunk", [0, 64])
def test_prefill_ragged(gdn, chunk):
    w = wl.WORKLOADS["prefill_ragged"]
    lens = wl.workload_lengths(w)
    order = np.argsort(lens.numpy())
    pairs = [(int(order[0]), 5), (int(order[-1]), 63), (int(order[len(order) // 2]), 30)]
    _prefill_case(gdn, "prefill_ragged", pairs, chunk)


@pytest.mark.parametrize("chunk", [0, 64])
def test_backward_t8192(gdn, chunk):
    """The backward pass at the single-sequence prefill workload's size (B=1,
    T=8192, 32 v-heads on 16 k-heads), q/k/v/g/beta from the workload's own
    conv and gates, dy and the final state's gradient seeded.  Sampled heads
    against the f64 reverse pass: dv, dg, dbeta, dstate_in of four v-heads and
    dq, dk of the two k-heads they share (sums over both v-heads)."""
    w = wl.WORKLOADS["prefill_t8192"]
    inp = wl.workload_inputs(w)
    d = inp["dims"]
    q, k, v, _ = oracle.conv_update(d, wl.bf16_bits(inp["qkv"]), wl.bf16_bits(inp["conv_w"]),
                                    wl.bf16_bits(inp["conv_state"]), None)
    g, beta = oracle.gating(wl.bf16_bits(inp["a"]), wl.bf16_bits(inp["b"]), inp["A_log"].numpy(),
                            inp["dt_bias"].numpy())
    g32, b32 = g.astype(np.float32), beta.astype(np.float32)
    t = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(DEV)
    gen = torch.Generator().manual_seed(4242)
    dy = (torch.randn((d.B, d.T, d.Hv, d.Dv), generator=gen) * 0.1).to(torch.bfloat16)
    dso = torch.randn((d.B, d.Hv, d.Dv, d.Dk), generator=gen) * 0.01
    s_in = inp["state"]
    out = gdn.prefill_backward(d, t(q), t(k), t(v), torch.from_numpy(g32).to(DEV), torch.from_numpy(b32).to(DEV),
                               dy.to(DEV), state_in=s_in.to(DEV), dstate_out=dso.to(DEV), chunk=chunk)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    G = d.Hv // d.Hk
    for hk in (0, 13):
        dq_ref = np.zeros((d.T, d.Dk))
        dk_ref = np.zeros((d.T, d.Dk))
        for hv in range(hk * G, hk * G + G):
            r = oracle.head_recurrence_bwd(oracle.bf16_to_f64(q[0, :, hk]), oracle.bf16_to_f64(k[0, :, hk]),
                                           oracle.bf16_to_f64(v[0, :, hv]), g32[0, :, hv].astype(np.float64),
                                           b32[0, :, hv].astype(np.float64), s_in[0, hv].numpy().astype(np.float64),
                                           U.bf16_dev_to_f64(dy[0, :, hv]), dso[0, hv].numpy().astype(np.float64))
            dq_ref += r["dq"]
            dk_ref += r["dk"]
            for name, rn, got in (("dv", "dv", out["dv"][0, :, hv]), ("dg", "dg", out["dg"][0, :, hv]),
                                  ("dbeta", "dbeta", out["dbeta"][0, :, hv]),
                                  ("dstate_in", "dS0", out["dstate_in"][0, hv])):
                U.assert_state_close(got.cpu().numpy(), r[rn], "%s (hv %d, chunk %d)" % (name, hv, chunk), tol=1e-3)
        U.assert_state_close(out["dq"][0, :, hk].cpu().numpy(), dq_ref, "dq (hk %d, chunk %d)" % (hk, chunk), tol=1e-3)
        U.assert_state_close(out["dk"][0, :, hk].cpu().numpy(), dk_ref, "dk (hk %d, chunk %d)" % (hk, chunk), tol=1e-3)
