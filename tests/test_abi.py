"""The C-ABI library loads, exports every entry point declared in
include/gdn.h, and rejects bad arguments on the host before any CUDA call
(no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    from gated_deltanet_linear_04_gb300.build import build_library
    build_library()
    from gated_deltanet_linear_04_gb300 import gdn
    return gdn.lib()


def declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return re.findall(r"GDN_API\s+[\w\s\*]+?\b(gdn_\w+)\s*\(", txt)


def test_header_declares_the_abi():
    names = set(declared_functions())
    for n in ("gdn_conv_update", "gdn_gating", "gdn_recurrent_decode", "gdn_prefill",
              "gdn_prefill_workspace_size", "gdn_status_string", "gdn_device_status", "gdn_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), "libgdn.so does not export " + n


def test_status_strings(lib):
    from gated_deltanet_linear_04_gb300 import gdn
    assert gdn.status_string(0) == "GDN_OK"
    for s in range(1, 5):
        assert gdn.status_string(s).startswith("GDN_ERR_")
    assert gdn.gdn_abi_version() == 1


def _dims(**kw):
    from gated_deltanet_linear_04_gb300 import gdn
    base = dict(B=1, T=8, Hk=1, Hv=2, Dk=32, Dv=32, K=4, eps_qk=1e-6)
    base.update(kw)
    return gdn.GdnDims(**base)


def _call(lib, name, d, n_ptrs, extra=()):
    f = getattr(lib, name)
    return f(ctypes.byref(d), *([None] * n_ptrs), *extra)


@pytest.mark.parametrize("kw,expect", [
    ({}, 1),                       # null pointers on non-empty tensors
    ({"Hv": 3}, 1),                # Hv % Hk != 0
    ({"T": -1}, 1),
    ({"Dk": 48}, 2),               # unsupported head size
    ({"Dv": 256}, 2),
    ({"K": 5}, 2),
    ({"K": 1}, 2),
])
def test_host_validation(lib, kw, expect):
    d = _dims(**kw)
    assert _call(lib, "gdn_gating", d, 6, (None,)) == expect
    assert _call(lib, "gdn_conv_update", d, 7, (None,)) == expect


def test_decode_requires_single_step_and_small_groups(lib):
    d = _dims(T=2)
    assert _call(lib, "gdn_recurrent_decode", d, 10, (None,)) == 1
    d = _dims(T=1, Hk=1, Hv=32)
    assert _call(lib, "gdn_recurrent_decode", d, 10, (None,)) == 2     # Hv/Hk > 16


def test_misaligned_pointer_rejected(lib):
    d = _dims(B=1, T=1)
    buf = ctypes.create_string_buffer(64)
    mis = ctypes.addressof(buf) | 1
    f = lib.gdn_gating
    assert f(ctypes.byref(d), mis, mis, mis, mis, mis, mis, None) == 1


def test_empty_sizes_are_noops(lib):
    d = _dims(B=0)
    assert _call(lib, "gdn_gating", d, 6, (None,)) == 0
    assert _call(lib, "gdn_conv_update", d, 7, (None,)) == 0
    d = _dims(T=0)
    assert _call(lib, "gdn_gating", d, 6, (None,)) == 0


def test_prefill_chunk_argument(lib):
    d = _dims()
    f = lib.gdn_prefill
    assert f(ctypes.byref(d), *([None] * 9), 32, None, 0, None) == 2    # unsupported chunk size
    # the optional row-order workspace: a few bytes per batch row, whole 256s
    n0 = lib.gdn_prefill_workspace_size(ctypes.byref(d), 0)
    assert n0 > 0 and n0 % 256 == 0 and n0 >= 8 * d.B
    # chunked with fewer heads than SMs: plus the two-pass images, one 145 KiB
    # blob per head and chunk of 64 steps and a ready flag each (any head size)
    n_blobs = d.B * d.Hv * ((d.T + 63) // 64)
    assert lib.gdn_prefill_workspace_size(ctypes.byref(d), 64) == n0 + n_blobs * 148480 + 256
    assert lib.gdn_prefill_workspace_size(ctypes.byref(d), 32) == 0
    assert lib.gdn_prefill_workspace_size(ctypes.byref(_dims(B=0)), 0) == 0


def test_decode_host_steps_staging_and_validation(lib):
    d = _dims(B=3, T=1)
    # four slots of qkv, a, b and y, each array rounded up to whole 256 bytes
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    C = 2 * d.Hk * d.Dk + d.Hv * d.Dv
    n = lib.gdn_decode_host_staging_size(ctypes.byref(d))
    assert n == 4 * (up(d.B * C * 2) + 2 * up(d.B * d.Hv * 2) + up(d.B * d.Hv * d.Dv * 2))
    assert lib.gdn_decode_host_staging_size(ctypes.byref(_dims(T=2))) == 0
    f = lib.gdn_recurrent_decode_host_steps
    none = [None] * 11
    assert f(ctypes.byref(d), -1, *none, 0, None) == 1            # negative step count
    assert f(ctypes.byref(_dims(T=2)), 1, *none, 0, None) == 1    # steps are single tokens
    assert f(ctypes.byref(d), 0, *none, 0, None) == 0             # no steps: nothing to do
    assert f(ctypes.byref(d), 3, *none, 0, None) == 1             # null host buffers
    # every pointer present and aligned, staging one byte short: rejected on
    # the host before any CUDA call
    buf = ctypes.create_string_buffer(4096)
    p = (ctypes.addressof(buf) + 15) // 16 * 16
    assert f(ctypes.byref(d), 3, *([p] * 11), n - 1, None) == 1


def test_binding_constants_match_the_header():
    from gated_deltanet_linear_04_gb300 import gdn
    txt = open(HEADER).read()
    m = re.search(r"#define\s+GDN_NOALLOC_MAX_ROWS\s+(\d+)", txt)
    assert m and int(m.group(1)) == gdn.GDN_NOALLOC_MAX_ROWS


def test_backward_chunked_workspace_sizes(lib):
    # per chunk of 64 steps of each (b, hv) head: 161 KiB of chain images,
    # 192 KiB of f32 records and a ready flag, after the row order
    d = _dims(B=2, T=130, Hk=1, Hv=2, Dk=128, Dv=128)
    n = 2 * 2 * 3
    order = lib.gdn_prefill_workspace_size(ctypes.byref(d), 0)
    flags = (n * 4 + 255) // 256 * 256
    assert lib.gdn_prefill_backward_chunked_workspace_size(ctypes.byref(d)) == order + n * (164864 + 196608) + flags
    # smaller heads run on the same 128-wide tiles and records: the same size
    for dk, dv in ((64, 128), (128, 64), (32, 32)):
        small = _dims(B=2, T=130, Hk=1, Hv=2, Dk=dk, Dv=dv)
        assert lib.gdn_prefill_backward_chunked_workspace_size(ctypes.byref(small)) == \
            order + n * (164864 + 196608) + flags
