"""The binding compares every tensor's element count with the dims before it
passes the address to the library (which sees pointers only): on the CPU, a
call whose sizes all match gets as far as the device check, and one element
too many in any single argument is rejected by name.  No GPU needed."""
import pytest
import torch

from gated_deltanet_linear_04_gb300 import workloads as wl

D = wl.Dims(B=2, T=3, Hk=1, Hv=2, Dk=32, Dv=64, K=4)
D1 = wl.Dims(B=2, T=1, Hk=1, Hv=2, Dk=32, Dv=64, K=4)


@pytest.fixture(scope="module")
def gdn():
    from gated_deltanet_linear_04_gb300.build import build_library
    build_library()
    from gated_deltanet_linear_04_gb300 import gdn as g
    return g


def bf(*s):
    return torch.zeros(s, dtype=torch.bfloat16)


def f32(*s):
    return torch.zeros(s, dtype=torch.float32)


def u8(*s):
    return torch.ones(s, dtype=torch.uint8)


def i32(*s):
    return torch.ones(s, dtype=torch.int32)


def calls(g):
    """(function, dims, positional arguments) with the layouts of the ABI."""
    d, d1 = D, D1
    C = d.C
    qk = lambda dd: bf(dd.B, dd.T, dd.Hk, dd.Dk)
    vv = lambda dd: bf(dd.B, dd.T, dd.Hv, dd.Dv)
    gate = lambda dd: f32(dd.B, dd.T, dd.Hv)
    st = lambda dd: f32(dd.B, dd.Hv, dd.Dv, dd.Dk)
    return [
        (g.gdn_conv_update, d, [bf(d.B, d.T, C), bf(C, d.K), bf(d.B, d.K - 1, C), u8(d.B, d.T), qk(d), qk(d), vv(d)]),
        (g.gdn_gating, d, [bf(d.B, d.T, d.Hv), bf(d.B, d.T, d.Hv), f32(d.Hv), f32(d.Hv), gate(d), gate(d)]),
        (g.gdn_recurrent_decode, d1, [bf(d1.B, C), bf(C, d1.K), bf(d1.B, d1.K - 1, C), bf(d1.B, d1.Hv),
                                      bf(d1.B, d1.Hv), f32(d1.Hv), f32(d1.Hv), st(d1), u8(d1.B),
                                      bf(d1.B, d1.Hv, d1.Dv)]),
        (g.gdn_decode_window, d, [bf(d.B, d.T, C), bf(C, d.K), bf(d.B, d.K - 1, C), bf(d.B, d.T, d.Hv),
                                  bf(d.B, d.T, d.Hv), f32(d.Hv), f32(d.Hv), st(d), i32(d.B), vv(d)]),
        (g.gdn_prefill, d, [qk(d), qk(d), vv(d), gate(d), gate(d), st(d), st(d), u8(d.B, d.T), vv(d)]),
        (g.gdn_recurrent_decode_gated, d1, [bf(d1.B, C), bf(C, d1.K), bf(d1.B, d1.K - 1, C), bf(d1.B, d1.Hv),
                                            bf(d1.B, d1.Hv), f32(d1.Hv), f32(d1.Hv), st(d1), u8(d1.B),
                                            bf(d1.B, d1.Hv, d1.Dv), f32(d1.Dv), 1e-6, bf(d1.B, d1.Hv, d1.Dv)]),
        (g.gdn_prefill_gated, d, [qk(d), qk(d), vv(d), gate(d), gate(d), st(d), st(d), u8(d.B, d.T), vv(d),
                                  f32(d.Dv), 1e-6, vv(d)]),
        (g.gdn_prefill_backward, d, [qk(d), qk(d), vv(d), gate(d), gate(d), st(d), u8(d.B, d.T), vv(d), st(d),
                                     f32(d.B, d.T, d.Hk, d.Dk), f32(d.B, d.T, d.Hk, d.Dk),
                                     f32(d.B, d.T, d.Hv, d.Dv), gate(d), gate(d), st(d), None]),
        (g.gdn_prefill_noalloc, d, [qk(d), qk(d), vv(d), gate(d), gate(d), st(d), st(d), u8(d.B, d.T), vv(d)]),
        (g.gdn_rmsnorm_gated, d, [vv(d), vv(d), f32(d.Dv), 1e-6, vv(d)]),
        (g.gdn_prefill_vec, d, [qk(d), qk(d), vv(d), f32(d.B, d.T, d.Hv, d.Dk), gate(d), st(d), st(d),
                                u8(d.B, d.T), vv(d)]),
    ]


def _grown(t):
    """The same tensor with one element more (flattened)."""
    return torch.zeros(t.numel() + 1, dtype=t.dtype)


def test_matching_sizes_reach_the_device_check(gdn):
    for fn, dims, args in calls(gdn):
        with pytest.raises(ValueError, match="must be a CUDA tensor"):
            fn(dims, *args)


def test_one_element_too_many_is_rejected_by_name(gdn):
    n = 0
    for fn, dims, args in calls(gdn):
        for i, a in enumerate(args):
            if not isinstance(a, torch.Tensor):
                continue
            bad = list(args)
            bad[i] = _grown(a)
            with pytest.raises(ValueError, match="must hold %d elements" % a.numel()):
                fn(dims, *bad)
            n += 1
    assert n >= 90
