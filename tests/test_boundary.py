"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

* libfab.so loads and exports every function include/fab.h declares;
* the packed layout matches the hand-worked offsets and the oracle's;
* argument validation returns the documented status before touching the GPU.
"""
import ctypes
import os
import re

import pytest

import oracle
from attention_backward_tcgen05_gb300 import binding
from attention_backward_tcgen05_gb300 import build as fab_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fab.h")


@pytest.fixture(scope="module")
def L():
    fab_build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FAB_EXPORT\s+[\w\s\*]+?\b(fab_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(names) == set(binding.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert binding.fab_version() >= 100


def test_status_strings(L):
    for s in range(6):
        assert binding.status_string(s)
    assert "unknown" in binding.status_string(99)


def read_golden():
    rows = []
    for line in open(os.path.join(ROOT, "tests", "golden", "packed_layout.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            a, b = line.split("|")
            rows.append((tuple(int(x) for x in a.split()), tuple(int(x) for x in b.split())))
    return rows


@pytest.mark.parametrize("dims,want", read_golden())
def test_packed_offsets_golden(L, dims, want):
    d = binding.make_dims(*dims)
    assert binding.fab_packed_offsets(d) == want
    assert binding.fab_packed_bytes(d) == want[2]


@pytest.mark.parametrize("dims", [(3, 5, 5, 7, 9, 3, 5), (2, 6, 3, 17, 1, 1, 2), (1, 1, 1, 1, 3, 13, 7)])
def test_packed_offsets_match_oracle(L, dims):
    assert binding.fab_packed_offsets(binding.make_dims(*dims)) == oracle.packed_layout(dims)


def test_workspace_bytes(L):
    d = binding.make_dims(4, 32, 8, 2048, 2048, 128, 128)
    ws = binding.fab_backward_workspace_bytes(d, binding.FAB_BF16)
    assert ws >= 4 * 32 * 2048 * 4 and ws % 256 == 0
    assert binding.fab_backward_workspace_bytes(binding.make_dims(1, 3, 2, 1, 1, 1, 1), 1) == 0
    assert binding.fab_backward_workspace_bytes(d, 7) == 0


def test_recompute_workspace_bytes(L):
    # without o and lse: D_i, the mask's live-tile maps (a byte per 128 x 128
    # tile, rows per query tile and rows per key tile, each row padded to 16
    # bytes), O (dtype) and LSE (f32), each rounded up to 256 bytes
    d = binding.make_dims(2, 4, 2, 100, 70, 64, 48)
    r256 = lambda x: (x + 255) // 256 * 256
    r16 = lambda x: (x + 15) // 16 * 16
    rows = 2 * 4 * 100
    bounds = r256(1 * r16(1) + 1 * r16(1))
    assert binding.fab_backward_workspace_bytes(d, binding.FAB_BF16) == r256(rows * 4) + bounds
    # 40 query tiles x 24 key tiles: 40 rows of 32 bytes, 24 rows of 48
    big = binding.make_dims(1, 2, 1, 5000, 3000, 128, 128)
    assert binding.fab_backward_workspace_bytes(big, binding.FAB_BF16) == r256(2 * 5000 * 4) + r256(40 * 32 + 24 * 48)
    for dt, elem in ((binding.FAB_BF16, 2), (binding.FAB_F16, 2), (binding.FAB_F32, 4)):
        want = r256(rows * 4) + bounds + r256(rows * 48 * elem) + r256(rows * 4)
        assert binding.fab_backward_recompute_workspace_bytes(d, dt) == want
        assert binding.fab_backward_recompute_workspace_bytes(d, dt) > binding.fab_backward_workspace_bytes(d, dt)
    assert binding.fab_backward_recompute_workspace_bytes(binding.make_dims(1, 3, 2, 1, 1, 1, 1), 1) == 0
    assert binding.fab_backward_recompute_workspace_bytes(d, 7) == 0


FAKE = 0x10000  # 16-byte-aligned non-null pointer; validation fails before it is used


def call_backward(L, dims, ptrs=None, dtype=binding.FAB_BF16, ws_bytes=1 << 30, mask=None):
    p = dict(q=FAKE, k=FAKE, v=FAKE, d=FAKE, o=FAKE, lse=FAKE, ws=FAKE, packed=FAKE)
    p.update(ptrs or {})
    vp = ctypes.c_void_p
    return L.fab_backward(vp(p["q"]), vp(p["k"]), vp(p["v"]), vp(p["d"]), vp(p["o"]), vp(p["lse"]), vp(mask), 0,
                          1.0, dtype, ctypes.byref(dims), vp(p["ws"]), ws_bytes, vp(p["packed"]), None)


def test_invalid_dims(L):
    for bad in [(1, 3, 2, 4, 4, 8, 8), (0, 1, 1, 4, 4, 8, 8), (1, 1, 1, -4, 4, 8, 8), (1, 1, 1, 4, 4, 0, 8)]:
        assert call_backward(L, binding.make_dims(*bad)) == binding.FAB_ERR_INVALID
        assert binding.fab_packed_bytes(binding.make_dims(*bad)) == 0
    nulls = [None] * 7 + [0, 1.0, 1, None, None, 0, None, None]  # every pointer null, dims null
    assert L.fab_backward(*nulls) == binding.FAB_ERR_INVALID


def test_null_and_misaligned_pointers(L):
    d = binding.make_dims(1, 2, 1, 64, 64, 64, 64)
    for key in ("q", "k", "v", "d", "o", "lse", "packed"):
        assert call_backward(L, d, {key: None}) == binding.FAB_ERR_INVALID, key
        assert call_backward(L, d, {key: FAKE + 4}) == binding.FAB_ERR_INVALID, key
    assert call_backward(L, d, mask=FAKE + 2) == binding.FAB_ERR_INVALID
    assert call_backward(L, d, dtype=5) == binding.FAB_ERR_INVALID
    assert call_backward(L, d, dtype=3) == binding.FAB_ERR_INVALID


def test_workspace_errors(L):
    d = binding.make_dims(1, 2, 1, 64, 64, 64, 64)
    assert call_backward(L, d, {"ws": None}) == binding.FAB_ERR_WORKSPACE
    assert call_backward(L, d, ws_bytes=16) == binding.FAB_ERR_WORKSPACE
    assert call_backward(L, d, {"ws": FAKE + 8}) == binding.FAB_ERR_WORKSPACE


def test_recompute_validation(L):
    # o and lse both NULL asks for the forward to be recomputed: the workspace
    # must then hold O and LSE as well; the other checks still apply first
    d = binding.make_dims(1, 2, 1, 64, 64, 64, 64)
    small = binding.fab_backward_workspace_bytes(d, binding.FAB_BF16)
    big = binding.fab_backward_recompute_workspace_bytes(d, binding.FAB_BF16)
    none = {"o": None, "lse": None}
    assert call_backward(L, d, none, ws_bytes=small) == binding.FAB_ERR_WORKSPACE
    assert call_backward(L, d, none, ws_bytes=big - 1) == binding.FAB_ERR_WORKSPACE
    assert call_backward(L, d, dict(none, q=None), ws_bytes=big) == binding.FAB_ERR_INVALID
    assert call_backward(L, d, dict(none, d=FAKE + 4), ws_bytes=big) == binding.FAB_ERR_INVALID
    assert call_backward(L, d, dict(none, packed=None), ws_bytes=big) == binding.FAB_ERR_INVALID
    assert call_backward(L, binding.make_dims(1, 3, 2, 4, 4, 8, 8), none, ws_bytes=big) == binding.FAB_ERR_INVALID
    vp = ctypes.c_void_p
    args = [vp(FAKE)] * 4 + [None, None, None, 0, 1.0, 1, ctypes.byref(d), vp(FAKE), None]
    assert L.fab_backward_noalloc(*args) == binding.FAB_ERR_INVALID  # no room for a recomputed O and LSE


def test_unsupported_width(L):
    d = binding.make_dims(1, 1, 1, 8, 8, 300, 8)
    assert call_backward(L, d) == binding.FAB_ERR_UNSUPPORTED
    vp = ctypes.c_void_p
    rc = L.fab_forward_lse(vp(FAKE), vp(FAKE), vp(FAKE), None, 0, 1.0, 1, ctypes.byref(d), vp(FAKE), vp(FAKE), None)
    assert rc == binding.FAB_ERR_UNSUPPORTED


def test_forward_validation(L):
    d = binding.make_dims(1, 3, 2, 8, 8, 8, 8)
    vp = ctypes.c_void_p
    rc = L.fab_forward_lse(vp(FAKE), vp(FAKE), vp(FAKE), None, 0, 1.0, 1, ctypes.byref(d), vp(FAKE), vp(FAKE), None)
    assert rc == binding.FAB_ERR_INVALID
    d = binding.make_dims(1, 2, 1, 8, 8, 8, 8)
    rc = L.fab_forward_lse(vp(FAKE), None, vp(FAKE), None, 0, 1.0, 1, ctypes.byref(d), vp(FAKE), vp(FAKE), None)
    assert rc == binding.FAB_ERR_INVALID


def test_binding_rejects_cpu_tensors(L):
    import torch

    q = torch.zeros(1, 1, 4, 8)
    with pytest.raises(ValueError):
        binding.fab_forward_lse(q, q, q, None, False, 1.0, q.new_empty(1, 4, 1, 8), q.new_empty(1, 1, 4), None)


def test_noalloc_validation_on_host(L):
    vp = ctypes.c_void_p
    # B*H*N beyond the fixed scratch: refused before any device work
    n = binding.NOALLOC_MAX_ROWS // 4 + 1
    d = binding.make_dims(1, 4, 4, n, 64, 64, 64)
    rc = L.fab_backward_noalloc(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None, 0, 1.0,
                                binding.FAB_BF16, ctypes.byref(d), vp(FAKE), None)
    assert rc == binding.FAB_ERR_WORKSPACE
    assert L.fab_backward_noalloc(*([None] * 7), 0, 1.0, 1, None, None, None) == binding.FAB_ERR_INVALID
