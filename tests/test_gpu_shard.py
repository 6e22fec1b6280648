"""One call split across ranks by batch row (gdn.shard_rows) gives the whole
batch's results bit for bit: every (b, head) owns its state, conv channels
and outputs, so the kernels' results for a row do not depend on the other
rows.  The ranks are run one after the other on one GPU (they exchange
nothing; the gloo test in test_multirank.py covers the gathering on CPU)."""
import pytest
import torch

from gated_deltanet_linear_04_gb300 import workloads as wl
from tests.test_gpu_parity import gdn, inputs_for, make_mask, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world", [2, 3])
def test_decode_split_by_rows_is_bitwise(gdn, world):  # noqa: F811
    d = wl.Dims(B=7, T=1, Hk=2, Hv=4, Dk=128, Dv=128)
    inp = inputs_for(d, 901)
    steps = [inputs_for(d, 910 + i) for i in range(3)]

    def run(b0, b1):
        dl = d.with_(B=b1 - b0)
        cs = to_dev(inp["conv_state"][b0:b1]).clone()
        st = to_dev(inp["state"][b0:b1]).clone()
        ys = []
        for s in steps:
            ys.append(gdn.recurrent_decode(dl, to_dev(s["qkv"][b0:b1, 0].contiguous()), to_dev(inp["conv_w"]), cs,
                                           to_dev(s["a"][b0:b1, 0].contiguous()), to_dev(s["b"][b0:b1, 0].contiguous()),
                                           to_dev(inp["A_log"]), to_dev(inp["dt_bias"]), st))
        torch.cuda.synchronize()
        return torch.stack(ys), st, cs

    y_full, s_full, c_full = run(0, d.B)
    parts = [run(*gdn.shard_rows(d.B, world, r)) for r in range(world)]
    assert torch.equal(torch.cat([p[0] for p in parts], dim=1), y_full)
    assert torch.equal(torch.cat([p[1] for p in parts], dim=0), s_full)
    assert torch.equal(torch.cat([p[2] for p in parts], dim=0), c_full)


@pytest.mark.parametrize("chunk", [0, 64])
def test_prefill_split_by_rows_is_bitwise(gdn, chunk):  # noqa: F811
    d = wl.Dims(B=4, T=150, Hk=2, Hv=4, Dk=128, Dv=128)
    inp = inputs_for(d, 920)
    mask = make_mask("right", d.B, d.T, 921)

    def run(b0, b1):
        dl = d.with_(B=b1 - b0)
        cs = to_dev(inp["conv_state"][b0:b1]).clone()
        y, s = gdn.core_prefill(dl, to_dev(inp["qkv"][b0:b1]), to_dev(inp["conv_w"]), to_dev(inp["a"][b0:b1]),
                                to_dev(inp["b"][b0:b1]), to_dev(inp["A_log"]), to_dev(inp["dt_bias"]), cs,
                                to_dev(inp["state"][b0:b1]), to_dev(mask[b0:b1].contiguous()), chunk)
        torch.cuda.synchronize()
        return y, s, cs

    y_full, s_full, c_full = run(0, d.B)
    parts = [run(*gdn.shard_rows(d.B, 2, r)) for r in range(2)]
    assert torch.equal(torch.cat([p[0] for p in parts], dim=0), y_full)
    assert torch.equal(torch.cat([p[1] for p in parts], dim=0), s_full)
    assert torch.equal(torch.cat([p[2] for p in parts], dim=0), c_full)
