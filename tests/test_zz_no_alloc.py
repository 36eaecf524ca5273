"""fab_backward_noalloc, the backward entry point for callers that cannot
allocate device memory (their memory belongs to another allocator, or they must
not call cudaMalloc, which can synchronise the device, on their path).  Its
scratch is a fixed array inside libfab, so the caller passes only inputs and
outputs.  The results must match fab_backward's, call after call: the shared
array keeps the previous call's contents, and nothing may depend on them.

This file is collected last so that a run that stops at the first failure has
run every other test before it.
"""
import numpy as np
import pytest
import torch

from attention_backward_tcgen05_gb300 import binding, inputs
from parity import TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.lib()


CASES = [
    inputs.custom(2, 8, 2, 320, 384, 128, causal=True, mask="random", seed=42, name="tensor_core_masked"),
    inputs.custom(1, 4, 2, 130, 70, 64, seed=43, name="tensor_core_d64"),
    inputs.custom(1, 2, 1, 40, 50, 16, 24, dtype="f32", dist="uniform", causal=True, seed=44, name="cuda_core_f32"),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_noalloc_matches_fab_backward_on_consecutive_calls(w):
    x = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inputs.make(w).items()}
    o, lse = binding.forward(x["q"], x["k"], x["v"], x["mask"], w.causal, w.scale)
    dims = binding.dims_of(x["q"], x["k"], x["v"])
    ws, ref = binding.alloc_backward(dims, binding.dtype_code(x["q"]), x["q"].device)
    binding.fab_backward(x["q"], x["k"], x["v"], x["d"], o, lse, x["mask"], w.causal, w.scale, ws, ref)
    assert binding.fab_last_device_error() == binding.FAB_OK
    want = ref.double().cpu().numpy()
    off_k, off_v, end = (t // 4 for t in binding.fab_packed_offsets(dims))
    out = torch.empty_like(ref)
    for call in range(2):
        out.fill_(float("nan"))
        binding.fab_backward_noalloc(x["q"], x["k"], x["v"], x["d"], o, lse, x["mask"], w.causal, w.scale, out)
        assert binding.fab_last_device_error() == binding.FAB_OK
        got = out.double().cpu().numpy()
        assert np.all(np.isfinite(got)), call
        for lo, hi in ((0, off_k), (off_k, off_v), (off_v, end)):
            assert rel_err(got[lo:hi], want[lo:hi]) <= TOL[w.dtype], (call, lo)
        # the padding between and after the slices is written as zero on every call
        B, H, Hkv, N, M, DK, DV = dims.tuple()
        nq, nk, nv = DK * N * H * B, DK * M * Hkv * B, DV * M * Hkv * B
        assert np.all(got[nq:off_k] == 0) and np.all(got[off_k + nk:off_v] == 0) and np.all(got[off_v + nv:] == 0)


def test_noalloc_at_the_row_limit_with_a_mask():
    # B*H*N exactly FAB_NOALLOC_MAX_ROWS: D_i fills the whole fixed array, so
    # the mask's live-tile maps do not fit after it and the call computes
    # every tile; fab_backward on a caller workspace that holds the maps skips
    # the all -inf tiles.  A skipped tile only ever adds +0, so the two must
    # agree bit for bit, on two calls in a row.
    w = inputs.custom(1, 64, 8, binding.NOALLOC_MAX_ROWS // 64, 128, 64, mask="pad", mask_p=0.05, seed=45,
                      name="row_limit_masked")
    assert w.B * w.H * w.N == binding.NOALLOC_MAX_ROWS
    x = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inputs.make(w).items()}
    o, lse = binding.forward(x["q"], x["k"], x["v"], x["mask"], w.causal, w.scale)
    dims = binding.dims_of(x["q"], x["k"], x["v"])
    ws, want = binding.alloc_backward(dims, binding.dtype_code(x["q"]), x["q"].device)
    binding.fab_backward(x["q"], x["k"], x["v"], x["d"], o, lse, x["mask"], w.causal, w.scale, ws, want)
    assert binding.fab_last_device_error() == binding.FAB_OK
    assert torch.isfinite(want).all()
    out = torch.empty_like(want)
    for call in range(2):
        out.fill_(float("nan"))
        binding.fab_backward_noalloc(x["q"], x["k"], x["v"], x["d"], o, lse, x["mask"], w.causal, w.scale, out)
        assert binding.fab_last_device_error() == binding.FAB_OK
        assert torch.equal(out, want), call
