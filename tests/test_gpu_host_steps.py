"""Decode steps fed from host memory (gdn_recurrent_decode_host_steps, the
end-to-end path of the benchmark) give the results of the same steps run on
device-resident inputs, bit for bit: the same kernel runs on the same bytes,
the copies only move them."""
import pytest
import torch

from gated_deltanet_linear_04_gb300 import workloads as wl
from tests.test_gpu_parity import gdn  # noqa: F401

pytestmark = pytest.mark.gpu


def _dev(t):
    return None if t is None else t.to("cuda:0")


@pytest.mark.parametrize("B,Hk,Hv,D,n,masked", [
    (4, 2, 4, 128, 5, False),
    (3, 1, 2, 32, 4, True),
    (128, 16, 32, 128, 3, False),     # the batched-decode workload's shape
])
def test_host_steps_equal_device_steps(gdn, B, Hk, Hv, D, n, masked):  # noqa: F811
    w = wl.WORKLOADS["decode_b128"]
    d = w.dims.with_(B=B, T=1, Hk=Hk, Hv=Hv, Dk=D, Dv=D)
    inp = wl.workload_inputs(w, d)
    steps = [wl.decode_step_inputs(w, i, d) for i in range(n)]
    qkv_h = torch.stack([s["qkv"][:, 0] for s in steps]).pin_memory()
    a_h = torch.stack([s["a"][:, 0] for s in steps]).pin_memory()
    b_h = torch.stack([s["b"][:, 0] for s in steps]).pin_memory()
    row_mask = None
    if masked:
        row_mask = torch.ones(B, dtype=torch.uint8)
        row_mask[1] = 0
    conv_w, A_log, dt_bias = _dev(inp["conv_w"]), _dev(inp["A_log"]), _dev(inp["dt_bias"])
    cs1, st1 = _dev(inp["conv_state"]).clone(), _dev(inp["state"]).clone()
    y_h = gdn.recurrent_decode_host_steps(d, qkv_h, a_h, b_h, conv_w, cs1, A_log, dt_bias, st1, _dev(row_mask))
    torch.cuda.synchronize()
    cs2, st2 = _dev(inp["conv_state"]).clone(), _dev(inp["state"]).clone()
    ys = [gdn.recurrent_decode(d, _dev(qkv_h[i]), conv_w, cs2, _dev(a_h[i]), _dev(b_h[i]), A_log, dt_bias, st2,
                               _dev(row_mask)) for i in range(n)]
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    assert torch.equal(y_h, torch.stack(ys).cpu())
    assert torch.equal(st1, st2) and torch.equal(cs1, cs2)


def test_host_steps_reject_device_tensors_as_host_buffers(gdn):  # noqa: F811
    w = wl.WORKLOADS["decode_b128"]
    d = w.dims.with_(B=2, T=1, Hk=1, Hv=2, Dk=32, Dv=32)
    inp = wl.workload_inputs(w, d)
    qkv = torch.zeros((1, 2, d.C), dtype=torch.bfloat16, device="cuda:0")
    ab = torch.zeros((1, 2, 2), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        gdn.recurrent_decode_host_steps(d, qkv, ab, ab, _dev(inp["conv_w"]), _dev(inp["conv_state"]),
                                        _dev(inp["A_log"]), _dev(inp["dt_bias"]), _dev(inp["state"]))
