"""Parity of the backward pass (gdn_prefill_backward) with the oracle's
reverse pass, through the C ABI.  Tolerance: each gradient tensor within
1e-3 relative L2 of the float64 oracle (the f32 state's bound: the reverse
pass runs the same kind of f32 recurrence, backwards); masked steps exactly
zero."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_04_gb300 import workloads as wl
from tests import _util as U
from tests.test_gpu_parity import gdn, inputs_for, make_mask, np_mask, recurrence_inputs, to_dev  # noqa: F401

pytestmark = pytest.mark.gpu

GRAD_REL_L2 = 1e-3

BWD_CASES = [
    # B, T, Hk, Hv, Dk, Dv, mask, state_in, dstate_out
    (1, 40, 1, 1, 128, 128, None, True, True),
    (2, 77, 1, 2, 128, 128, "random", True, False),
    (1, 64, 2, 8, 64, 64, "right", False, True),
    (3, 33, 1, 4, 32, 32, "blocks", True, True),
    (2, 100, 2, 4, 128, 64, "allmasked_row", True, True),
    (1, 130, 1, 1, 64, 128, "sparse", False, False),
    (1, 1024, 1, 2, 128, 128, "random", True, True),     # long: error growth over many steps
    (2, 70, 16, 64, 128, 128, "random", True, True),     # 512 row slices: the single-launch form
    (1, 50, 16, 80, 64, 128, None, True, False),         # 320 row slices, no mask: single launch, Dk = 64
]


@pytest.mark.parametrize("B,T,Hk,Hv,Dk,Dv,mk,si,ds", BWD_CASES)
def test_backward_matches_oracle(gdn, B, T, Hk, Hv, Dk, Dv, mk, si, ds):  # noqa: F811
    d = wl.Dims(B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv)
    mask = make_mask(mk, B, T, 31 + T)
    r = recurrence_inputs(d, 3100 + T, mask)
    gen = torch.Generator().manual_seed(77 + T)
    dy = (torch.randn((B, T, Hv, Dv), generator=gen) * 0.1).to(torch.bfloat16)
    dso = torch.randn((B, Hv, Dv, Dk), generator=gen) * 0.01 if ds else None
    s_in = r["state"] if si else None
    out = gdn.prefill_backward(d, to_dev(r["q"]), to_dev(r["k"]), to_dev(r["v"]), to_dev(r["g"]), to_dev(r["beta"]),
                               to_dev(dy), state_in=to_dev(s_in), mask=to_dev(mask), dstate_out=to_dev(dso))
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    ref = oracle.recurrence_bwd(d, r["q_bits"], r["k_bits"], r["v_bits"], r["g"].numpy().astype(np.float64),
                                r["beta"].numpy().astype(np.float64),
                                None if s_in is None else s_in.numpy().astype(np.float64),
                                U.bf16_dev_to_f64(dy), None if dso is None else dso.numpy().astype(np.float64),
                                np_mask(mask))
    for name, rname in (("dq", "dq"), ("dk", "dk"), ("dv", "dv"), ("dg", "dg"), ("dbeta", "dbeta"),
                        ("dstate_in", "dstate_in")):
        got = out[name].cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), name
        if np.abs(ref[rname]).max() == 0.0:
            assert np.all(got == 0.0), name
            continue
        U.assert_state_close(got, ref[rname], name, tol=GRAD_REL_L2)
    if mask is not None:
        off = mask.numpy() == 0
        for name in ("dv", "dg", "dbeta"):
            assert np.all(out[name].cpu().numpy()[off] == 0.0), name + ": masked steps must be zero"


def test_backward_without_steps_passes_the_state_gradient(gdn):  # noqa: F811
    d = wl.Dims(B=2, T=0, Hk=1, Hv=2, Dk=32, Dv=32)
    dso = torch.randn((2, 2, 32, 32), generator=torch.Generator().manual_seed(3))
    empty_bf = torch.empty((2, 0, 1, 32), dtype=torch.bfloat16, device="cuda:0")
    out = gdn.prefill_backward(d, empty_bf, empty_bf, torch.empty((2, 0, 2, 32), dtype=torch.bfloat16,
                                                                  device="cuda:0"),
                               torch.empty((2, 0, 2), device="cuda:0"), torch.empty((2, 0, 2), device="cuda:0"),
                               torch.empty((2, 0, 2, 32), dtype=torch.bfloat16, device="cuda:0"),
                               dstate_out=to_dev(dso))
    torch.cuda.synchronize()
    assert torch.equal(out["dstate_in"].cpu(), dso)


# Chunked form (tensor cores; every head size on 128-wide tiles): the same
# oracle, the same bound.
BWD_CHUNKED_CASES = [
    # B, T, Hk, Hv, Dk, Dv, mask, state_in, dstate_out
    (1, 40, 1, 1, 128, 128, None, True, True),            # one partial chunk
    (1, 200, 1, 2, 128, 128, None, True, False),          # several chunks and a ragged tail
    (2, 77, 1, 2, 128, 128, "random", True, True),
    (2, 300, 2, 4, 128, 128, "blocks", False, True),      # wholly masked chunks skipped
    (2, 100, 2, 4, 128, 128, "allmasked_row", True, True),
    (1, 130, 1, 1, 128, 128, "sparse", False, False),
    (3, 129, 1, 3, 128, 128, "right", True, True),
    (1, 1024, 1, 2, 128, 128, "random", True, True),      # long: the carried gradient over 16 chunks
    (2, 70, 16, 80, 128, 128, None, True, True),          # 160 heads: the single-pass forward; a 9e-17 gate
    (3, 33, 1, 4, 32, 32, "blocks", True, True),          # small heads: padded tiles
    (1, 150, 2, 8, 64, 64, "right", False, True),
    (2, 100, 2, 4, 128, 64, "allmasked_row", True, True),
    (1, 130, 1, 1, 64, 128, "sparse", True, False),
    (2, 90, 1, 2, 32, 128, None, True, True),
]


@pytest.mark.parametrize("B,T,Hk,Hv,Dk,Dv,mk,si,ds", BWD_CHUNKED_CASES)
def test_backward_chunked_matches_oracle(gdn, B, T, Hk, Hv, Dk, Dv, mk, si, ds):  # noqa: F811
    d = wl.Dims(B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv)
    mask = make_mask(mk, B, T, 31 + T)
    r = recurrence_inputs(d, 3100 + T, mask)
    gen = torch.Generator().manual_seed(77 + T)
    dy = (torch.randn((B, T, Hv, Dv), generator=gen) * 0.1).to(torch.bfloat16)
    dso = torch.randn((B, Hv, Dv, Dk), generator=gen) * 0.01 if ds else None
    s_in = r["state"] if si else None
    out = gdn.prefill_backward(d, to_dev(r["q"]), to_dev(r["k"]), to_dev(r["v"]), to_dev(r["g"]), to_dev(r["beta"]),
                               to_dev(dy), state_in=to_dev(s_in), mask=to_dev(mask), dstate_out=to_dev(dso), chunk=64)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    ref = oracle.recurrence_bwd(d, r["q_bits"], r["k_bits"], r["v_bits"], r["g"].numpy().astype(np.float64),
                                r["beta"].numpy().astype(np.float64),
                                None if s_in is None else s_in.numpy().astype(np.float64),
                                U.bf16_dev_to_f64(dy), None if dso is None else dso.numpy().astype(np.float64),
                                np_mask(mask))
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dstate_in"):
        got = out[name].cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), name
        if np.abs(ref[name]).max() == 0.0:
            assert np.all(got == 0.0), name
            continue
        U.assert_state_close(got, ref[name], name + " (chunked)", tol=GRAD_REL_L2)
    if mask is not None:
        off = mask.numpy() == 0
        for name in ("dv", "dg", "dbeta"):
            assert np.all(out[name].cpu().numpy()[off] == 0.0), name + ": masked steps must be zero"
        offk = np.repeat(off[:, :, None], Hk, axis=2)
        for name in ("dq", "dk"):
            assert np.all(out[name].cpu().numpy()[offk] == 0.0), name + ": masked steps must be zero"


def test_backward_chunked_same_as_sequential_at_small_heads(gdn):  # noqa: F811
    # the chunked form at Dk = Dv = 32 agrees with the sequential form within
    # the tf32 bound on a masked batch (both against each other, not only the oracle)
    d = wl.Dims(B=2, T=160, Hk=2, Hv=4, Dk=32, Dv=32)
    mask = make_mask("random", 2, 160, 7)
    r = recurrence_inputs(d, 4321, mask)
    dy = (torch.randn((2, 160, 4, 32), generator=torch.Generator().manual_seed(5)) * 0.1).to(torch.bfloat16)
    outs = [gdn.prefill_backward(d, to_dev(r["q"]), to_dev(r["k"]), to_dev(r["v"]), to_dev(r["g"]),
                                 to_dev(r["beta"]), to_dev(dy), state_in=to_dev(r["state"]), mask=to_dev(mask),
                                 chunk=c) for c in (0, 64)]
    torch.cuda.synchronize()
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dstate_in"):
        U.assert_state_close(outs[1][name].cpu().numpy(), outs[0][name].cpu().numpy().astype(np.float64),
                             name + " chunked vs sequential", tol=GRAD_REL_L2)
