"""Helpers shared by the GPU tests: tolerances, comparisons, conversions."""
import numpy as np
import torch

from gated_deltanet_linear_04_gb300 import workloads as wl

# Tolerances of the floating-point outputs (y in bf16, state in f32).
Y_MAX_ABS = 2e-2
Y_REL_L2 = 1e-2
STATE_REL_L2 = 1e-3


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def bf16_dev_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bits(t: torch.Tensor) -> np.ndarray:
    return wl.bf16_bits(t.detach().cpu())


def assert_y_close(y_gpu, y_ref, what="y"):
    y = np.asarray(y_gpu, np.float64)
    r = np.asarray(y_ref, np.float64)
    assert y.shape == r.shape, (y.shape, r.shape)
    assert np.all(np.isfinite(y)), what + ": non-finite output"
    err = np.abs(y - r).max() if y.size else 0.0
    rel = rel_l2(y, r) if y.size else 0.0
    assert err <= Y_MAX_ABS and rel <= Y_REL_L2, "%s: max abs %.3e (<= %.0e), rel L2 %.3e (<= %.0e)" % (
        what, err, Y_MAX_ABS, rel, Y_REL_L2)
    return err, rel


def assert_out_close(o_gpu, o_ref, what="out"):
    """The gated-norm output, y normalised to unit RMS per head row and
    scaled by silu(z) * w: values reach a few units, where one bf16 ulp is
    already 2^-6 .. 2^-5, so the y bound applies relative to max(1, |ref|)
    elementwise (an absolute bound for values below 1), with the same 1%
    relative L2 over the whole tensor."""
    o = np.asarray(o_gpu, np.float64)
    r = np.asarray(o_ref, np.float64)
    assert o.shape == r.shape, (o.shape, r.shape)
    assert np.all(np.isfinite(o)), what + ": non-finite output"
    err = (np.abs(o - r) / np.maximum(1.0, np.abs(r))).max() if o.size else 0.0
    rel = rel_l2(o, r) if o.size else 0.0
    assert err <= Y_MAX_ABS and rel <= Y_REL_L2, "%s: max scaled err %.3e (<= %.0e), rel L2 %.3e (<= %.0e)" % (
        what, err, Y_MAX_ABS, rel, Y_REL_L2)
    return err, rel


def assert_state_close(s_gpu, s_ref, what="state", tol=STATE_REL_L2):
    s = np.asarray(s_gpu, np.float64)
    r = np.asarray(s_ref, np.float64)
    assert s.shape == r.shape
    rel = rel_l2(s, r)
    assert rel <= tol, "%s: rel L2 %.3e (<= %.0e)" % (what, rel, tol)
    return rel


def assert_bf16_within_one_ulp(got_bits, ref_bits, what, max_frac=0.01):
    """bf16 outputs computed in f32 (device) vs f64 (oracle), each rounded once:
    equal except where the two pre-rounding values straddle a rounding
    boundary, which can move the result by one unit in the last place."""
    g = np.asarray(got_bits, np.uint16).astype(np.int32)
    r = np.asarray(ref_bits, np.uint16).astype(np.int32)
    # map sign-magnitude bf16 bit patterns to a monotone integer line
    def mono(x):
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    d = np.abs(mono(g) - mono(r))
    assert d.max(initial=0) <= 1, "%s: %d elements differ by > 1 ulp (max %d)" % (what, int((d > 1).sum()),
                                                                               int(d.max()))
    frac = float((d > 0).mean()) if d.size else 0.0
    assert frac <= max_frac, "%s: %.3f%% of elements differ by 1 ulp" % (what, 100 * frac)
    return frac
