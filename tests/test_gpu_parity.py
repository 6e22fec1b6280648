"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small cases compare every output element; the full-size workloads compare
sampled (b, hv) heads, which the oracle computes one by one, plus properties
that hold at any size (padded outputs are exactly zero, the conv state holds
the last raw inputs).  Tolerances: y (bf16) max abs <= 2e-2 and rel L2 <= 1%;
f32 state rel L2 <= 1e-3; masks, zeros and conv_state copies bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_04_gb300 import workloads as wl
from tests import _util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_deltanet_linear_04_gb300.build import build_library
    build_library()
    from gated_deltanet_linear_04_gb300 import gdn as g
    assert torch.cuda.is_available(), "these tests need a GPU"
    torch.cuda.set_device(0)
    return g


DEV = "cuda:0"


def make_mask(kind, B, T, seed):
    g = torch.Generator().manual_seed(seed)
    if kind is None:
        return None
    if kind == "random":
        return (torch.rand((B, T), generator=g) < 0.6).to(torch.uint8)
    if kind == "sparse":
        return (torch.rand((B, T), generator=g) < 0.04).to(torch.uint8)
    if kind in ("left", "right"):
        lens = torch.randint(0, T + 1, (B,), generator=g)
        t = torch.arange(T)[None, :]
        m = (t < lens[:, None]) if kind == "right" else (t >= (T - lens)[:, None])
        return m.to(torch.uint8)
    if kind == "blocks":
        # about half of the 64-step chunks wholly masked, the rest partly
        nch = (T + 63) // 64
        keep = (torch.rand((B, nch), generator=g) < 0.5).repeat_interleave(64, dim=1)[:, :T]
        return ((torch.rand((B, T), generator=g) < 0.8) & keep).to(torch.uint8)
    if kind == "allmasked_row":
        m = (torch.rand((B, T), generator=g) < 0.5).to(torch.uint8)
        m[0] = 0
        return m
    raise ValueError(kind)


def inputs_for(d, seed, conv_state="normal", state="normal"):
    p = wl.make_params(d, seed)
    a = wl.make_activations(d, seed + 1)
    s = wl.make_states(d, seed + 2, "normal" if conv_state == "none" else conv_state, state)
    out = dict(p, **a, **s)
    if conv_state == "none":
        out["conv_state"] = None
    return out


def to_dev(x):
    return None if x is None else x.to(DEV)


def np_mask(m):
    return None if m is None else m.numpy()


# ---------------------------------------------------------------------------
# a4 gates
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B,T,Hv", [(1, 8, 2), (3, 77, 32), (2, 1, 64), (1, 1000, 5)])
def test_gating(gdn, B, T, Hv):
    d = wl.Dims(B=B, T=T, Hk=1, Hv=Hv, Dk=32, Dv=32)
    inp = inputs_for(d, 11 + T)
    a = (torch.randn((B, T, Hv), generator=torch.Generator().manual_seed(T)) * 4).to(torch.bfloat16)
    g, beta = gdn.gating(d, to_dev(a), to_dev(inp["b"]), to_dev(inp["A_log"]), to_dev(inp["dt_bias"]))
    gr, br = oracle.gating(U.bits(a), U.bits(inp["b"]), inp["A_log"].numpy(), inp["dt_bias"].numpy())
    # g = exp(-z), z = exp(A_log) softplus(a + dt_bias) is formed in f32 with a
    # few roundings of relative size 2^-24 each, so ln g carries an absolute
    # error of a few ulps of z: compare ln g against 1e-6 * max(1, z).
    gg = g.cpu().numpy().astype(np.float64)
    z = -np.log(gr)
    live = gr > 1e-36                       # below this f32 underflows
    assert np.all(np.abs(np.log(gg[live]) + z[live]) <= 1e-6 * np.maximum(1.0, z[live]))
    assert np.all(gg[~live] <= 1e-36)
    assert np.allclose(beta.cpu().numpy(), br, rtol=2e-6, atol=1e-30)


# ---------------------------------------------------------------------------
# a1-a3 conv window + conv + SiLU + q/k norm (+ a6 mask)
# ---------------------------------------------------------------------------
CONV_CASES = [
    # B, T, Hk, Hv, Dk, Dv, K, mask, conv_state
    (1, 8, 1, 2, 32, 32, 4, None, "zeros"),
    (2, 37, 2, 4, 64, 32, 4, "random", "normal"),
    (2, 65, 1, 1, 128, 128, 3, "left", "normal"),
    (3, 17, 2, 8, 32, 64, 2, "right", "none"),
    (1, 1, 4, 8, 128, 64, 4, None, "normal"),
    (2, 100, 2, 4, 128, 128, 4, "sparse", "normal"),
    (2, 33, 1, 2, 64, 64, 4, "allmasked_row", "normal"),
    (1, 300, 3, 6, 128, 32, 4, None, "normal"),
]


@pytest.mark.parametrize("B,T,Hk,Hv,Dk,Dv,K,mk,cs", CONV_CASES)
def test_conv_update(gdn, B, T, Hk, Hv, Dk, Dv, K, mk, cs):
    d = wl.Dims(B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, K=K)
    inp = inputs_for(d, 100 + T, conv_state=cs)
    mask = make_mask(mk, B, T, 7 + T)
    cs_dev = to_dev(inp["conv_state"])
    q, k, v = gdn.conv_update(d, to_dev(inp["qkv"]), to_dev(inp["conv_w"]), cs_dev, to_dev(mask))
    torch.cuda.synchronize()
    cs_bits = None if inp["conv_state"] is None else U.bits(inp["conv_state"])
    qr, kr, vr, csr = oracle.conv_update(d, U.bits(inp["qkv"]), U.bits(inp["conv_w"]), cs_bits, np_mask(mask))
    for name, got, ref in (("q", q, qr), ("k", k, kr), ("v", v, vr)):
        gb = U.bits(got)
        U.assert_bf16_within_one_ulp(gb, ref, name)
        if mask is not None:
            assert np.all(gb[mask.numpy() == 0] == 0), name + ": masked steps must be exactly zero"
    if cs_dev is not None:
        assert np.array_equal(U.bits(cs_dev), csr), "conv_state must equal the last K-1 valid raw inputs"


# ---------------------------------------------------------------------------
# a5/a6 recurrence, sequential prefill
# ---------------------------------------------------------------------------
def recurrence_inputs(d, seed, mask=None, conv_state="normal"):
    """q/k/v/g/beta produced by the oracle from synthetic layer inputs (the
    shapes and scales the recurrence sees in the model); g and beta rounded
    to f32, the device input type."""
    inp = inputs_for(d, seed, conv_state=conv_state)
    cs = None if inp["conv_state"] is None else U.bits(inp["conv_state"])
    q, k, v, _ = oracle.conv_update(d, U.bits(inp["qkv"]), U.bits(inp["conv_w"]), cs, np_mask(mask))
    g, beta = oracle.gating(U.bits(inp["a"]), U.bits(inp["b"]), inp["A_log"].numpy(), inp["dt_bias"].numpy())
    g32, b32 = g.astype(np.float32), beta.astype(np.float32)
    t = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    return {"q": t(q), "k": t(k), "v": t(v), "q_bits": q, "k_bits": k, "v_bits": v,
            "g": torch.from_numpy(g32), "beta": torch.from_numpy(b32), "state": inp["state"]}


SEQ_CASES = [
    # B, T, Hk, Hv, Dk, Dv, mask, state
    (1, 8, 1, 2, 32, 32, None, "zeros"),
    (1, 1, 1, 1, 128, 128, None, "normal"),
    (2, 63, 2, 4, 128, 128, "random", "normal"),
    (1, 64, 1, 2, 64, 128, None, "normal"),
    (2, 65, 2, 2, 128, 64, "right", "normal"),
    (1, 130, 1, 4, 32, 32, "left", "normal"),
    (2, 200, 4, 16, 128, 128, "allmasked_row", "normal"),
    (3, 129, 1, 3, 64, 32, "sparse", "zeros"),
    (3, 333, 1, 2, 128, 128, "blocks", "normal"),   # rows 1, 2 of the mask not 16-byte aligned
    (2, 640, 2, 4, 64, 64, "blocks", "zeros"),
]


@pytest.mark.parametrize("B,T,Hk,Hv,Dk,Dv,mk,st", SEQ_CASES)
def test_prefill_sequential(gdn, B, T, Hk, Hv, Dk, Dv, mk, st):
    d = wl.Dims(B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv)
    mask = make_mask(mk, B, T, 3 + T)
    r = recurrence_inputs(d, 200 + T, mask)
    state_in = r["state"] if st == "normal" else None
    y, s_out = gdn.prefill(d, to_dev(r["q"]), to_dev(r["k"]), to_dev(r["v"]), to_dev(r["g"]), to_dev(r["beta"]),
                           to_dev(state_in), to_dev(mask), chunk=0)
    torch.cuda.synchronize()
    s0 = None if state_in is None else state_in.numpy().astype(np.float64)
    yr, sr = oracle.recurrence(d, r["q_bits"], r["k_bits"], r["v_bits"], r["g"].numpy().astype(np.float64),
                               r["beta"].numpy().astype(np.float64), s0, np_mask(mask))
    yg = U.bf16_dev_to_f64(y)
    U.assert_y_close(yg, yr)
    U.assert_state_close(s_out.cpu().numpy(), sr)
    if mask is not None:
        assert np.all(U.bits(y)[mask.numpy() == 0] == 0), "padded y must be exactly zero"
        for b in range(B):
            if mask[b].sum() == 0:
                ref = np.zeros_like(sr[b]) if s0 is None else state_in[b].numpy()
                assert np.array_equal(s_out[b].cpu().numpy(), ref), "row without valid steps: state untouched"
    assert gdn.gdn_device_status() == gdn.GDN_OK


CHUNK_CASES = [
    # B, T, Hk, Hv, mask, state     (chunked form: Dk = Dv = 128)
    (1, 1, 1, 1, None, "normal"),
    (1, 63, 1, 2, None, "zeros"),
    (1, 64, 1, 2, None, "normal"),
    (2, 65, 2, 4, "random", "normal"),
    (1, 200, 1, 2, "right", "normal"),
    (3, 130, 1, 3, "left", "zeros"),
    (2, 257, 2, 4, "allmasked_row", "normal"),
    (2, 150, 1, 2, "sparse", "normal"),
    (3, 333, 1, 2, "blocks", "normal"),
    (2, 640, 1, 2, "blocks", "zeros"),
]


@pytest.mark.parametrize("B,T,Hk,Hv,mk,st", CHUNK_CASES)
def test_prefill_chunked(gdn, B, T, Hk, Hv, mk, st):
    d = wl.Dims(B=B, T=T, Hk=Hk, Hv=Hv, Dk=128, Dv=128)
    mask = make_mask(mk, B, T, 5 + T)
    r = recurrence_inputs(d, 500 + T, mask)
    state_in = r["state"] if st == "normal" else None
    y, s_out = gdn.prefill(d, to_dev(r["q"]), to_dev(r["k"]), to_dev(r["v"]), to_dev(r["g"]), to_dev(r["beta"]),
                           to_dev(state_in), to_dev(mask), chunk=64)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    s0 = None if state_in is None else state_in.numpy().astype(np.float64)
    yr, sr = oracle.recurrence(d, r["q_bits"], r["k_bits"], r["v_bits"], r["g"].numpy().astype(np.float64),
                               r["beta"].numpy().astype(np.float64), s0, np_mask(mask))
    U.assert_y_close(U.bf16_dev_to_f64(y), yr)
    U.assert_state_close(s_out.cpu().numpy(), sr)
    if mask is not None:
        assert np.all(U.bits(y)[mask.numpy() == 0] == 0), "padded y must be exactly zero"
        for b in range(B):
            if mask[b].sum() == 0:
                ref = np.zeros_like(sr[b]) if s0 is None else state_in[b].numpy()
                assert np.array_equal(s_out[b].cpu().numpy(), ref), "row without valid steps: state untouched"


@pytest.mark.parametrize("chunk", [0, 64])
def test_prefill_masked_chunks_across_scan_windows(gdn, chunk):
    # long rows that are mostly masked: the search for the next chunk with a
    # valid step crosses several windows of the chunk bitmap, and row 1's mask
    # starts off a 16-byte boundary
    B, T = 2, 17000
    d = wl.Dims(B=B, T=T, Hk=1, Hv=1, Dk=128, Dv=128)
    mask = torch.zeros((B, T), dtype=torch.uint8)
    for a, e in [(50, 120), (8300, 8400), (16500, 16600), (16990, 17000)]:
        mask[0, a:e] = 1
    mask[1, :200] = 1
    mask[1, 16900:] = 1
    mask[1, 12000] = 1
    r = recurrence_inputs(d, 4321, mask)
    y, s_out = gdn.prefill(d, to_dev(r["q"]), to_dev(r["k"]), to_dev(r["v"]), to_dev(r["g"]), to_dev(r["beta"]),
                           to_dev(r["state"]), to_dev(mask), chunk=chunk)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    yr, sr = oracle.recurrence(d, r["q_bits"], r["k_bits"], r["v_bits"], r["g"].numpy().astype(np.float64),
                               r["beta"].numpy().astype(np.float64), r["state"].numpy().astype(np.float64),
                               np_mask(mask))
    U.assert_y_close(U.bf16_dev_to_f64(y), yr)
    U.assert_state_close(s_out.cpu().numpy(), sr)
    assert np.all(U.bits(y)[mask.numpy() == 0] == 0), "masked y must be exactly zero"


@pytest.mark.parametrize("chunk", [0, 64])
def test_prefill_row_order(gdn, chunk):
    # right-padded rows of very different lengths: with a workspace the rows
    # are handed to CTAs longest first; that changes only which CTA takes which
    # row, so the outputs are bit-identical to index order (and match the oracle)
    B, T = 6, 700
    lens = [30, 700, 0, 333, 64, 699]
    d = wl.Dims(B=B, T=T, Hk=1, Hv=2, Dk=128, Dv=128)
    mask = (torch.arange(T)[None, :] < torch.tensor(lens)[:, None]).to(torch.uint8)
    r = recurrence_inputs(d, 77, mask)
    dev = [to_dev(r[n]) for n in ("q", "k", "v", "g", "beta")]
    s_in, m_dev = to_dev(r["state"]), to_dev(mask)
    y1, s1 = gdn.prefill(d, *dev, state_in=s_in, mask=m_dev, chunk=chunk, use_workspace=False)
    nws = gdn.gdn_prefill_workspace_size(d, chunk)
    ws = torch.full((nws,), 0xFF, dtype=torch.uint8, device=DEV)
    y2, s2 = torch.empty_like(y1), torch.empty_like(s1)
    gdn.gdn_prefill(d, *dev, s_in, s2, m_dev, y2, chunk, ws)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    assert torch.equal(y1, y2) and torch.equal(s1, s2), "row order must not change results"
    work = [(n + 63) // 64 for n in lens]
    assert ws[:4 * B].view(torch.int32).cpu().tolist() == sorted(range(B), key=lambda b: (-work[b], b))
    yr, sr = oracle.recurrence(d, r["q_bits"], r["k_bits"], r["v_bits"], r["g"].numpy().astype(np.float64),
                               r["beta"].numpy().astype(np.float64), r["state"].numpy().astype(np.float64),
                               np_mask(mask))
    U.assert_y_close(U.bf16_dev_to_f64(y2), yr)
    U.assert_state_close(s2.cpu().numpy(), sr)
    # a workspace below the row-order size is refused before any launch
    n_order = gdn.gdn_prefill_workspace_size(d, 0)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_prefill(d, *dev, s_in, s2, m_dev, y2, chunk, ws[:n_order - 16])
    assert e.value.status == gdn.GDN_ERR_INVALID_ARG


@pytest.mark.parametrize("chunk", [0, 64])
def test_prefill_zero_gates(gdn, chunk):
    # a gate of exactly 0 forgets everything before it; the chunked form works
    # with log g, so it must not turn the zero into -inf and NaN
    d = wl.Dims(B=2, T=150, Hk=1, Hv=2, Dk=128, Dv=128)
    r = recurrence_inputs(d, 777)
    g = r["g"].clone()
    g[0, [5, 64, 100], :] = 0.0
    g[1, 130, 1] = 0.0
    g[1, 63, 0] = 0.0
    dev = [to_dev(r[n]) for n in ("q", "k", "v")]
    y, s_out = gdn.prefill(d, *dev, to_dev(g), to_dev(r["beta"]), state_in=to_dev(r["state"]), chunk=chunk)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    yr, sr = oracle.recurrence(d, r["q_bits"], r["k_bits"], r["v_bits"], g.numpy().astype(np.float64),
                               r["beta"].numpy().astype(np.float64), r["state"].numpy().astype(np.float64))
    U.assert_y_close(U.bf16_dev_to_f64(y), yr)
    U.assert_state_close(s_out.cpu().numpy(), sr)


TWO_PASS_CASES = [
    # B, T, Hk, Hv, mask, state   (B * Hv below the SM count: the two-pass form)
    (1, 200, 1, 2, None, "normal"),
    (1, 64, 1, 1, None, "zeros"),
    (2, 333, 1, 3, "random", "normal"),
    (3, 700, 2, 4, "blocks", "normal"),
    (2, 257, 2, 4, "right", "zeros"),
    (2, 150, 1, 2, "allmasked_row", "normal"),
    (2, 100, 4, 24, "random", "normal"),     # 48 heads: the two passes as separate launches
    (1, 130, 8, 64, None, "zeros"),
]


@pytest.mark.parametrize("B,T,Hk,Hv,mk,st", TWO_PASS_CASES)
def test_prefill_two_pass_equals_single_pass(gdn, B, T, Hk, Hv, mk, st):
    # the two-pass chunked form runs the single pass's arithmetic on the same
    # operand bits: bit-identical y and state (and so the oracle's tolerance)
    d = wl.Dims(B=B, T=T, Hk=Hk, Hv=Hv, Dk=128, Dv=128)
    mask = make_mask(mk, B, T, 21 + T)
    r = recurrence_inputs(d, 2100 + T, mask)
    dev = [to_dev(r[n]) for n in ("q", "k", "v", "g", "beta")]
    s_in = to_dev(r["state"]) if st == "normal" else None
    n_full, n_order = gdn.gdn_prefill_workspace_size(d, 64), gdn.gdn_prefill_workspace_size(d, 0)
    assert n_full > n_order, "these sizes should ask for the two-pass workspace"
    y1, s1 = gdn.prefill(d, *dev, state_in=s_in, mask=to_dev(mask), chunk=64, use_workspace=False)
    ws = torch.full((n_full,), 0xAB, dtype=torch.uint8, device=DEV)
    y2 = torch.empty_like(y1)
    s2 = torch.empty_like(s1)
    gdn.gdn_prefill(d, *dev, s_in, s2, to_dev(mask), y2, 64, ws)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    assert torch.equal(y1, y2), "two-pass y differs from the single pass"
    assert torch.equal(s1, s2), "two-pass state differs from the single pass"
    s0 = None if s_in is None else r["state"].numpy().astype(np.float64)
    yr, sr = oracle.recurrence(d, r["q_bits"], r["k_bits"], r["v_bits"], r["g"].numpy().astype(np.float64),
                               r["beta"].numpy().astype(np.float64), s0, np_mask(mask))
    U.assert_y_close(U.bf16_dev_to_f64(y2), yr)
    U.assert_state_close(s2.cpu().numpy(), sr)


CHUNK_SMALL_HEAD_CASES = [
    # B, T, Hk, Hv, Dk, Dv, mask, state   (head sizes below 128: zero-padded 128-wide tiles)
    (1, 8, 1, 2, 32, 32, None, "zeros"),
    (2, 130, 1, 2, 64, 64, "right", "normal"),
    (1, 200, 2, 4, 32, 128, None, "normal"),
    (2, 97, 1, 3, 128, 64, "random", "normal"),
    (3, 333, 1, 2, 64, 32, "blocks", "normal"),
]


@pytest.mark.parametrize("B,T,Hk,Hv,Dk,Dv,mk,st", CHUNK_SMALL_HEAD_CASES)
def test_prefill_chunked_small_heads(gdn, B, T, Hk, Hv, Dk, Dv, mk, st):
    """The chunked form at Dk, Dv of 32 and 64 against the oracle, in the
    single pass and in the two-pass form, which agree bit for bit."""
    d = wl.Dims(B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv)
    mask = make_mask(mk, B, T, 9 + T)
    r = recurrence_inputs(d, 900 + T, mask)
    state_in = r["state"] if st == "normal" else None
    dev = [to_dev(r[n]) for n in ("q", "k", "v", "g", "beta")]
    y1, s1 = gdn.prefill(d, *dev, to_dev(state_in), to_dev(mask), chunk=64, use_workspace=False)
    y2, s2 = gdn.prefill(d, *dev, to_dev(state_in), to_dev(mask), chunk=64, use_workspace=True)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    assert gdn.gdn_prefill_workspace_size(d, 64) > gdn.gdn_prefill_workspace_size(d, 0), "two passes expected"
    s0 = None if state_in is None else state_in.numpy().astype(np.float64)
    yr, sr = oracle.recurrence(d, r["q_bits"], r["k_bits"], r["v_bits"], r["g"].numpy().astype(np.float64),
                               r["beta"].numpy().astype(np.float64), s0, np_mask(mask))
    U.assert_y_close(U.bf16_dev_to_f64(y1), yr)
    U.assert_state_close(s1.cpu().numpy(), sr)
    assert torch.equal(y1, y2) and torch.equal(s1, s2)
    if mask is not None:
        assert np.all(U.bits(y1)[mask.numpy() == 0] == 0), "padded y must be exactly zero"


def test_prefill_in_place_and_split_is_bitwise(gdn):
    """state_out may alias state_in; running T1 then T2 steps equals T1+T2
    steps bit for bit (the sequential form does the same arithmetic)."""
    d = wl.Dims(B=2, T=150, Hk=2, Hv=4, Dk=128, Dv=128)
    r = recurrence_inputs(d, 5)
    full_y, full_s = gdn.prefill(d, *(to_dev(r[x]) for x in ("q", "k", "v", "g", "beta")), to_dev(r["state"]))
    st = to_dev(r["state"]).clone()
    ys = []
    for lo, hi in ((0, 70), (70, 150)):
        dd = d.with_(T=hi - lo)
        sl = lambda x: to_dev(r[x][:, lo:hi].contiguous())
        y, _ = gdn.prefill(dd, sl("q"), sl("k"), sl("v"), sl("g"), sl("beta"), st, None, 0, state_out=st)
        ys.append(y)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(ys, 1), full_y)
    assert torch.equal(st, full_s)


@pytest.mark.parametrize("mk,use_ws", [(None, True), (None, False), ("random", True)])
def test_prefill_chunked_prefix_consistency(gdn, mk, use_ws):
    """prefill(T1) then prefill(T2) from the state it returns equals
    prefill(T1 + T2) in the chunked form, within the state and y bounds,
    with T1 not a multiple of the chunk length, so the second call's chunks
    start in the middle of the first call's chunk grid (the pages' serving
    loop replays a prefix and continues from its state)."""
    d = wl.Dims(B=2, T=333, Hk=2, Hv=4, Dk=128, Dv=128)
    T1 = 141
    mask = make_mask(mk, d.B, d.T, 88)
    r = recurrence_inputs(d, 88, mask)
    full_y, full_s = gdn.prefill(d, *(to_dev(r[x]) for x in ("q", "k", "v", "g", "beta")), to_dev(r["state"]),
                                 to_dev(mask), 64, use_workspace=use_ws)
    st = to_dev(r["state"]).clone()
    ys = []
    for lo, hi in ((0, T1), (T1, d.T)):
        dd = d.with_(T=hi - lo)
        sl = lambda x: to_dev(r[x][:, lo:hi].contiguous())
        m = None if mask is None else to_dev(mask[:, lo:hi].contiguous())
        y, _ = gdn.prefill(dd, sl("q"), sl("k"), sl("v"), sl("g"), sl("beta"), st, m, 64, state_out=st,
                           use_workspace=use_ws)
        ys.append(y)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    split_y = torch.cat(ys, 1)
    U.assert_y_close(U.bf16_dev_to_f64(split_y), U.bf16_dev_to_f64(full_y), "split y vs one call")
    U.assert_state_close(st.cpu().numpy(), full_s.cpu().numpy().astype(np.float64), "split state vs one call")
    yr, sr = oracle.recurrence(d, r["q_bits"], r["k_bits"], r["v_bits"], r["g"].numpy().astype(np.float64),
                               r["beta"].numpy().astype(np.float64), r["state"].numpy().astype(np.float64),
                               np_mask(mask))
    U.assert_y_close(U.bf16_dev_to_f64(split_y), yr, "split y vs oracle")
    U.assert_state_close(st.cpu().numpy(), sr, "split state vs oracle")
    if mask is not None:
        assert np.all(U.bits(split_y)[mask.numpy() == 0] == 0), "padded y must be exactly zero"


# ---------------------------------------------------------------------------
# the composed core (configuration "tiny" and masked variants)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mk", [None, "right", "random"])
def test_core_prefill_tiny(gdn, mk):
    w = wl.WORKLOADS["tiny"]
    inp = wl.workload_inputs(w)
    d = inp["dims"]
    mask = make_mask(mk, d.B, d.T, 1)
    cs = to_dev(inp["conv_state"]).clone()
    y, s = gdn.core_prefill(d, to_dev(inp["qkv"]), to_dev(inp["conv_w"]), to_dev(inp["a"]), to_dev(inp["b"]),
                            to_dev(inp["A_log"]), to_dev(inp["dt_bias"]), cs, to_dev(inp["state"]), to_dev(mask))
    torch.cuda.synchronize()
    ref = oracle.layer_core(d, U.bits(inp["qkv"]), U.bits(inp["conv_w"]), U.bits(inp["a"]), U.bits(inp["b"]),
                            inp["A_log"].numpy(), inp["dt_bias"].numpy(), U.bits(inp["conv_state"]),
                            inp["state"].numpy().astype(np.float64), np_mask(mask))
    U.assert_y_close(U.bf16_dev_to_f64(y), ref["y"])
    U.assert_state_close(s.cpu().numpy(), ref["state"])
    assert np.array_equal(U.bits(cs), ref["conv_state"])


@pytest.mark.parametrize("chunk,use_ws", [(0, True), (64, True), (64, False)])
def test_state_tolerance_after_4096_steps(gdn, chunk, use_ws):
    """The f32 state bound after T = 4096 from a nonzero initial state, in
    the sequential form and in both chunked forms (two passes when the
    workspace is given to these few heads, the single pass without it)."""
    d = wl.Dims(B=1, T=4096, Hk=1, Hv=2, Dk=128, Dv=128)
    inp = inputs_for(d, 4096)
    assert float(inp["state"].abs().max()) > 0
    y, s = gdn.core_prefill(d, to_dev(inp["qkv"]), to_dev(inp["conv_w"]), to_dev(inp["a"]), to_dev(inp["b"]),
                            to_dev(inp["A_log"]), to_dev(inp["dt_bias"]), to_dev(inp["conv_state"]).clone(),
                            to_dev(inp["state"]), None, chunk, None, use_ws)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    ref = oracle.layer_core(d, U.bits(inp["qkv"]), U.bits(inp["conv_w"]), U.bits(inp["a"]), U.bits(inp["b"]),
                            inp["A_log"].numpy(), inp["dt_bias"].numpy(), U.bits(inp["conv_state"]),
                            inp["state"].numpy().astype(np.float64))
    U.assert_y_close(U.bf16_dev_to_f64(y), ref["y"])
    U.assert_state_close(s.cpu().numpy(), ref["state"])


# ---------------------------------------------------------------------------
# fused decode
# ---------------------------------------------------------------------------
def run_decode_gpu(gdn, d, inp, steps, row_mask=None):
    cs = to_dev(inp["conv_state"]).clone()
    st = to_dev(inp["state"]).clone()
    ys = []
    for sin in steps:
        y = gdn.recurrent_decode(d.with_(T=1), to_dev(sin["qkv"][:, 0].contiguous()), to_dev(inp["conv_w"]), cs,
                                 to_dev(sin["a"][:, 0].contiguous()), to_dev(sin["b"][:, 0].contiguous()),
                                 to_dev(inp["A_log"]), to_dev(inp["dt_bias"]), st, to_dev(row_mask))
        ys.append(y)
    torch.cuda.synchronize()
    return ys, st, cs


DECODE_CASES = [
    # B, Hk, Hv, Dk, Dv, K, steps, row mask
    (1, 1, 2, 32, 32, 4, 6, False),
    (3, 2, 4, 128, 128, 4, 5, True),
    (2, 16, 32, 128, 128, 4, 3, False),
    (2, 1, 16, 64, 64, 3, 4, False),      # G = 16: cluster of 16 CTAs
    (5, 4, 8, 32, 128, 2, 4, True),
    (1, 2, 16, 128, 64, 4, 3, False),
]


@pytest.mark.parametrize("B,Hk,Hv,Dk,Dv,K,n,rm", DECODE_CASES)
def test_decode(gdn, B, Hk, Hv, Dk, Dv, K, n, rm):
    d = wl.Dims(B=B, T=1, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, K=K)
    inp = inputs_for(d, 300 + B * Hv)
    steps = [wl.make_activations(d, 400 + i) for i in range(n)]
    row_mask = None
    if rm:
        row_mask = torch.ones(B, dtype=torch.uint8)
        row_mask[1::2] = 0
    ys, st, cs = run_decode_gpu(gdn, d, inp, steps, row_mask)
    sbits = [{k: U.bits(s[k]) for k in ("qkv", "a", "b")} for s in steps]
    yr, sr, csr = oracle.decode(d, sbits, U.bits(inp["conv_w"]), inp["A_log"].numpy(), inp["dt_bias"].numpy(),
                                U.bits(inp["conv_state"]), inp["state"].numpy().astype(np.float64),
                                None if row_mask is None else row_mask.numpy())
    for i in range(n):
        U.assert_y_close(U.bf16_dev_to_f64(ys[i]), yr[i], "y step %d" % i)
    U.assert_state_close(st.cpu().numpy(), sr)
    assert np.array_equal(U.bits(cs), csr)
    if row_mask is not None:
        for b in range(B):
            if row_mask[b] == 0:
                assert torch.equal(st[b].cpu(), inp["state"][b]), "masked row: state untouched"
                assert all(int(y[b].abs().max()) == 0 for y in ys)
    assert gdn.gdn_device_status() == gdn.GDN_OK


def test_decode_steps_match_prefill(gdn):
    """n single-token decode steps == one prefill over the same n tokens."""
    d = wl.Dims(B=2, T=9, Hk=2, Hv=4, Dk=128, Dv=128)
    inp = inputs_for(d, 77)
    steps = [{k: inp[k][:, t:t + 1] for k in ("qkv", "a", "b")} for t in range(d.T)]
    ys, st, cs = run_decode_gpu(gdn, d, inp, steps)
    cs2 = to_dev(inp["conv_state"]).clone()
    y, s = gdn.core_prefill(d, to_dev(inp["qkv"]), to_dev(inp["conv_w"]), to_dev(inp["a"]), to_dev(inp["b"]),
                            to_dev(inp["A_log"]), to_dev(inp["dt_bias"]), cs2, to_dev(inp["state"]))
    torch.cuda.synchronize()
    U.assert_y_close(U.bf16_dev_to_f64(torch.stack(ys, 1)), U.bf16_dev_to_f64(y))
    U.assert_state_close(st.cpu().numpy(), s.cpu().numpy().astype(np.float64), tol=1e-5)
    assert torch.equal(cs, cs2)


# ---------------------------------------------------------------------------
# f-1 RMSNormGated output
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B,T,Hv,Dv", [(1, 8, 2, 32), (2, 37, 4, 64), (3, 65, 32, 128), (1, 1, 64, 128)])
def test_rmsnorm_gated(gdn, B, T, Hv, Dv):
    d = wl.Dims(B=B, T=T, Hk=1, Hv=Hv, Dk=32, Dv=Dv)
    gi = wl.make_gate_inputs(d, 600 + T)
    y = (torch.randn((B, T, Hv, Dv), generator=torch.Generator().manual_seed(T)) * 0.1).to(torch.bfloat16)
    y[0, 0] = 0                                       # a masked step's row
    out = gdn.rmsnorm_gated(d, to_dev(y), to_dev(gi["z"]), to_dev(gi["norm_w"]), 1e-6)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm_gated(U.bits(y), U.bits(gi["z"]), gi["norm_w"].numpy(), 1e-6)
    U.assert_bf16_within_one_ulp(U.bits(out), ref, "rmsnorm_gated")
    assert np.all(U.bf16_dev_to_f64(out[0, 0]) == 0.0)   # +0 or -0 (silu(z) < 0 times 0)


# f-1 fused: the gated norm in the decode and prefill epilogues
GATED_DECODE_CASES = [
    # B, Hk, Hv, Dk, Dv, K, row mask
    (3, 2, 4, 128, 128, 4, True),      # two row slices per head: sums exchanged in the cluster
    (2, 1, 16, 64, 64, 3, False),      # G = 16: one slice per head
    (4, 4, 4, 32, 32, 2, False),       # G = 1: several slices per head
    (2, 16, 32, 128, 128, 4, False),
]


@pytest.mark.parametrize("B,Hk,Hv,Dk,Dv,K,rm", GATED_DECODE_CASES)
def test_decode_gated(gdn, B, Hk, Hv, Dk, Dv, K, rm):
    d = wl.Dims(B=B, T=1, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, K=K)
    inp = inputs_for(d, 900 + B * Hv)
    gi = wl.make_gate_inputs(d, 950 + B)
    z, w, eps = gi["z"][:, 0].contiguous(), gi["norm_w"], 1e-6
    row_mask = None
    if rm:
        row_mask = torch.ones(B, dtype=torch.uint8)
        row_mask[1] = 0
    args = [to_dev(inp["qkv"][:, 0].contiguous()), to_dev(inp["conv_w"])]
    gates = [to_dev(inp["a"][:, 0].contiguous()), to_dev(inp["b"][:, 0].contiguous()), to_dev(inp["A_log"]),
             to_dev(inp["dt_bias"])]
    cs1, st1 = to_dev(inp["conv_state"]).clone(), to_dev(inp["state"]).clone()
    out = gdn.recurrent_decode_gated(d, *args, cs1, *gates, st1, to_dev(z), to_dev(w), eps, to_dev(row_mask))
    cs2, st2 = to_dev(inp["conv_state"]).clone(), to_dev(inp["state"]).clone()
    y = gdn.recurrent_decode(d, *args, cs2, *gates, st2, to_dev(row_mask))
    out2 = gdn.rmsnorm_gated(d, y, to_dev(z), to_dev(w), eps)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    assert torch.equal(st1, st2) and torch.equal(cs1, cs2), "the states are those of the plain step"
    U.assert_bf16_within_one_ulp(U.bits(out), U.bits(out2), "fused vs decode + rmsnorm_gated")
    sb = [{k: U.bits(inp[k]) for k in ("qkv", "a", "b")}]
    yr, _, _ = oracle.decode(d, sb, U.bits(inp["conv_w"]), inp["A_log"].numpy(), inp["dt_bias"].numpy(),
                             U.bits(inp["conv_state"]), inp["state"].numpy().astype(np.float64),
                             None if row_mask is None else row_mask.numpy())
    ref = oracle.rmsnorm_gated(oracle.f64_to_bf16(yr[0]), U.bits(z), w.numpy(), eps)
    U.assert_out_close(U.bf16_dev_to_f64(out), oracle.bf16_to_f64(ref), "gated decode output")
    if rm:
        assert np.all(U.bf16_dev_to_f64(out[1]) == 0.0), "a masked row gives zeros"


GATED_PREFILL_CASES = [
    # chunk, B, T, Hk, Hv, Dk, Dv, mask
    (64, 2, 200, 1, 2, 128, 128, "right"),
    (64, 3, 130, 2, 4, 128, 128, "random"),
    (64, 1, 64, 1, 1, 128, 128, None),
    (64, 3, 333, 1, 2, 128, 128, "blocks"),
    (64, 2, 70, 16, 80, 128, 128, "random"),     # B * Hv >= the SM count: the norm in the kernel's epilogue
    (64, 1, 160, 8, 160, 128, 128, "blocks"),
    (0, 2, 100, 2, 4, 64, 32, "random"),
    (0, 1, 77, 1, 2, 128, 128, None),
    (64, 2, 100, 80, 80, 64, 64, "random"),       # head size 64, the norm in the epilogue (mean over Dv)
    (64, 2, 90, 1, 2, 32, 64, "right"),
]


@pytest.mark.parametrize("chunk,B,T,Hk,Hv,Dk,Dv,mk", GATED_PREFILL_CASES)
def test_prefill_gated(gdn, chunk, B, T, Hk, Hv, Dk, Dv, mk):
    d = wl.Dims(B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv)
    mask = make_mask(mk, B, T, 11 + T)
    r = recurrence_inputs(d, 1500 + T, mask)
    gi = wl.make_gate_inputs(d, 1600 + T)
    eps = 1e-6
    dev = [to_dev(r[n]) for n in ("q", "k", "v", "g", "beta")]
    z, w = to_dev(gi["z"]), to_dev(gi["norm_w"])
    out, s1 = gdn.prefill_gated(d, *dev, z, w, eps, state_in=to_dev(r["state"]), mask=to_dev(mask), chunk=chunk)
    y, s2 = gdn.prefill(d, *dev, state_in=to_dev(r["state"]), mask=to_dev(mask), chunk=chunk)
    out2 = gdn.rmsnorm_gated(d, y, z, w, eps)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    assert torch.equal(s1, s2), "the state is that of the plain prefill"
    U.assert_bf16_within_one_ulp(U.bits(out), U.bits(out2), "fused vs prefill + rmsnorm_gated")
    yr, _ = oracle.recurrence(d, r["q_bits"], r["k_bits"], r["v_bits"], r["g"].numpy().astype(np.float64),
                              r["beta"].numpy().astype(np.float64), r["state"].numpy().astype(np.float64),
                              np_mask(mask))
    ref = oracle.rmsnorm_gated(oracle.f64_to_bf16(yr), U.bits(gi["z"]), gi["norm_w"].numpy(), eps)
    U.assert_out_close(U.bf16_dev_to_f64(out), oracle.bf16_to_f64(ref), "gated prefill output")
    if mask is not None:
        assert np.all(U.bf16_dev_to_f64(out)[mask.numpy() == 0] == 0.0), "masked steps give a zero"


def test_core_then_rmsnorm_gated_tiny(gdn):
    """The full layer core followed by the gated norm, against the oracle."""
    w = wl.WORKLOADS["tiny"]
    inp = wl.workload_inputs(w)
    d = inp["dims"]
    gi = wl.make_gate_inputs(d, 7)
    y, _ = gdn.core_prefill(d, to_dev(inp["qkv"]), to_dev(inp["conv_w"]), to_dev(inp["a"]), to_dev(inp["b"]),
                            to_dev(inp["A_log"]), to_dev(inp["dt_bias"]), to_dev(inp["conv_state"]).clone(),
                            to_dev(inp["state"]))
    out = gdn.rmsnorm_gated(d, y, to_dev(gi["z"]), to_dev(gi["norm_w"]), 1e-6)
    torch.cuda.synchronize()
    ref = oracle.layer_core(d, U.bits(inp["qkv"]), U.bits(inp["conv_w"]), U.bits(inp["a"]), U.bits(inp["b"]),
                            inp["A_log"].numpy(), inp["dt_bias"].numpy(), U.bits(inp["conv_state"]),
                            inp["state"].numpy().astype(np.float64))
    ref_out = oracle.rmsnorm_gated(ref["y_bf16"], U.bits(gi["z"]), gi["norm_w"].numpy(), 1e-6)
    U.assert_out_close(U.bf16_dev_to_f64(out), oracle.bf16_to_f64(ref_out), "gated output")


# ---------------------------------------------------------------------------
# f-2 multi-token decode window (speculative verify / accepted-prefix commit)
# ---------------------------------------------------------------------------
WINDOW_CASES = [
    # B, Hk, Hv, Dk, Dv, K, T, keep
    (2, 2, 4, 128, 128, 4, 4, None),
    (3, 1, 2, 64, 64, 3, 5, [0, 2, 5]),
    (2, 16, 32, 128, 128, 4, 8, [8, 3]),
    (1, 1, 16, 32, 128, 2, 1, [1]),
    (4, 2, 8, 128, 64, 4, 7, [7, 0, 1, 6]),
    (2, 1, 2, 32, 32, 3, 3, [1, 3]),          # keep < K-1: a kept row comes from the old conv_state
    (2, 2, 6, 64, 64, 3, 4, [4, 2]),          # G = 3: clusters of 6 CTAs, uneven q/k channel shares
    (1, 1, 16, 32, 32, 4, 6, [5]),            # clusters of 16 CTAs, 4 q/k channels each
]


@pytest.mark.parametrize("B,Hk,Hv,Dk,Dv,K,T,keep", WINDOW_CASES)
def test_decode_window(gdn, B, Hk, Hv, Dk, Dv, K, T, keep):
    d = wl.Dims(B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv, K=K)
    inp = inputs_for(d, 700 + B * T)
    keep_t = None if keep is None else torch.tensor(keep, dtype=torch.int32)
    cs = to_dev(inp["conv_state"]).clone()
    st = to_dev(inp["state"]).clone()
    y = gdn.decode_window(d, to_dev(inp["qkv"]), to_dev(inp["conv_w"]), cs, to_dev(inp["a"]), to_dev(inp["b"]),
                          to_dev(inp["A_log"]), to_dev(inp["dt_bias"]), st, to_dev(keep_t))
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    args = (U.bits(inp["qkv"]), U.bits(inp["conv_w"]), U.bits(inp["a"]), U.bits(inp["b"]), inp["A_log"].numpy(),
            inp["dt_bias"].numpy(), U.bits(inp["conv_state"]), inp["state"].numpy().astype(np.float64))
    full = oracle.layer_core(d, *args)
    U.assert_y_close(U.bf16_dev_to_f64(y), full["y"], "window y")
    st_h, cs_h = st.cpu().numpy(), U.bits(cs)
    for bb in range(B):
        kb = T if keep is None else keep[bb]
        if kb == 0:
            assert np.array_equal(st_h[bb], inp["state"][bb].numpy()), "keep 0: state untouched"
            assert np.array_equal(cs_h[bb], U.bits(inp["conv_state"])[bb]), "keep 0: conv_state untouched"
            continue
        dr = d.with_(B=1, T=kb)
        row = lambda x: np.ascontiguousarray(x[bb:bb + 1, :kb])
        ref = oracle.layer_core(dr, row(args[0]), args[1], row(args[2]), row(args[3]), args[4], args[5],
                                np.ascontiguousarray(args[6][bb:bb + 1]), args[7][bb:bb + 1])
        U.assert_state_close(st_h[bb], ref["state"][0], "state after %d kept tokens" % kb)
        assert np.array_equal(cs_h[bb], ref["conv_state"][0]), "conv_state after the kept prefix"


def test_decode_window_commit_equals_single_steps(gdn):
    """A window committed with keep = k gives the states that k single-token
    decode steps give (conv_state bit for bit, state within f32 rounding)."""
    d = wl.Dims(B=2, T=6, Hk=2, Hv=4, Dk=128, Dv=128)
    inp = inputs_for(d, 77)
    keep = [4, 6]
    cs_w, st_w = to_dev(inp["conv_state"]).clone(), to_dev(inp["state"]).clone()
    gdn.decode_window(d, to_dev(inp["qkv"]), to_dev(inp["conv_w"]), cs_w, to_dev(inp["a"]), to_dev(inp["b"]),
                      to_dev(inp["A_log"]), to_dev(inp["dt_bias"]), st_w, to_dev(torch.tensor(keep, dtype=torch.int32)))
    for bb, kb in enumerate(keep):
        d1 = d.with_(B=1)
        sub = {k: inp[k][bb:bb + 1] for k in ("qkv", "a", "b")}
        steps = [{k: sub[k][:, t:t + 1] for k in sub} for t in range(kb)]
        one = {"conv_state": inp["conv_state"][bb:bb + 1], "state": inp["state"][bb:bb + 1],
               "conv_w": inp["conv_w"], "A_log": inp["A_log"], "dt_bias": inp["dt_bias"]}
        _, st1, cs1 = run_decode_gpu(gdn, d1, one, steps)
        assert torch.equal(cs1[0], cs_w[bb])
        U.assert_state_close(st_w[bb].cpu().numpy(), st1[0].cpu().numpy().astype(np.float64), tol=1e-5)


# ---------------------------------------------------------------------------
# f-3 vectorized gating (one decay per key channel), sequential form
# ---------------------------------------------------------------------------
VEC_CASES = [
    # B, T, Hk, Hv, Dk, Dv, mask
    (1, 8, 1, 2, 32, 32, None),
    (2, 65, 2, 4, 128, 128, "random"),
    (1, 130, 1, 2, 64, 128, "right"),
    (3, 40, 1, 3, 128, 32, "allmasked_row"),
]


@pytest.mark.parametrize("B,T,Hk,Hv,Dk,Dv,mk", VEC_CASES)
def test_prefill_vec_gating(gdn, B, T, Hk, Hv, Dk, Dv, mk):
    d = wl.Dims(B=B, T=T, Hk=Hk, Hv=Hv, Dk=Dk, Dv=Dv)
    mask = make_mask(mk, B, T, 9 + T)
    r = recurrence_inputs(d, 800 + T, mask)
    gv = torch.rand((B, T, Hv, Dk), generator=torch.Generator().manual_seed(T)) * 0.7 + 0.3
    y, s = gdn.prefill_vec(d, to_dev(r["q"]), to_dev(r["k"]), to_dev(r["v"]), to_dev(gv), to_dev(r["beta"]),
                           to_dev(r["state"]), to_dev(mask))
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    yr, sr = oracle.recurrence_vec(d, r["q_bits"], r["k_bits"], r["v_bits"], gv.numpy().astype(np.float64),
                                   r["beta"].numpy().astype(np.float64), r["state"].numpy().astype(np.float64),
                                   np_mask(mask))
    U.assert_y_close(U.bf16_dev_to_f64(y), yr)
    U.assert_state_close(s.cpu().numpy(), sr)
    if mask is not None:
        assert np.all(U.bits(y)[mask.numpy() == 0] == 0)


def test_prefill_vec_with_equal_channels_matches_scalar(gdn):
    d = wl.Dims(B=2, T=100, Hk=2, Hv=4, Dk=128, Dv=128)
    r = recurrence_inputs(d, 5)
    gvec = r["g"][..., None].expand(d.B, d.T, d.Hv, d.Dk).contiguous()
    args = [to_dev(r[x]) for x in ("q", "k", "v")]
    y1, s1 = gdn.prefill(d, *args, to_dev(r["g"]), to_dev(r["beta"]), to_dev(r["state"]))
    y2, s2 = gdn.prefill_vec(d, *args, to_dev(gvec), to_dev(r["beta"]), to_dev(r["state"]))
    torch.cuda.synchronize()
    U.assert_y_close(U.bf16_dev_to_f64(y2), U.bf16_dev_to_f64(y1))
    U.assert_state_close(s2.cpu().numpy(), s1.cpu().numpy().astype(np.float64), tol=1e-5)
