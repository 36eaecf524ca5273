"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small cases span several key/query tiles, ragged tails, GQA, batches, causal
and additive masks, D = 64 and 128 on the tensor-core path and odd widths /
f32 on the CUDA-core path.  The five measured workloads (and the two extra
masked ones) run at full size in the launch configuration the benchmark
times, and every element of dQ, dK, dV, O and LSE is compared with the
oracle's.
"""
import zlib

import numpy as np
import pytest
import torch

from attention_backward_tcgen05_gb300 import binding, inputs
from parity import TOL, check_pads_zero, compare, oracle_ref, rel_err, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.lib()
    yield


SMALL = [
    # name, B, H, Hkv, N, M, DK, DV, dtype, causal, mask
    ("tc128_causal_gqa_NltM", 2, 4, 2, 200, 300, 128, 128, "bf16", True, "none"),
    ("tc128_full_ragged", 1, 2, 2, 130, 257, 128, 128, "bf16", False, "none"),
    ("tc128_mask_gqa", 2, 4, 1, 96, 200, 128, 128, "bf16", False, "random"),
    ("tc128_causal_NgtM", 1, 2, 1, 300, 140, 128, 128, "bf16", True, "none"),
    ("tc128_causal_and_mask", 1, 3, 3, 190, 190, 128, 128, "bf16", True, "random"),
    ("tc64_causal", 2, 2, 2, 256, 256, 64, 64, "bf16", True, "none"),
    ("tc64_mask_gqa_ragged", 1, 4, 2, 70, 130, 64, 64, "bf16", False, "random"),
    ("tc128_single", 1, 1, 1, 1, 1, 128, 128, "bf16", False, "none"),
    # eight query heads per key/value head (the key pass walks all eight for
    # every query tile); one ragged query tile against eight key tiles; many
    # query tiles against one ragged key tile
    ("tc128_gqa8_causal", 1, 8, 1, 300, 300, 128, 128, "bf16", True, "none"),
    ("tc64_short_q_long_k", 1, 2, 1, 64, 1000, 64, 64, "bf16", False, "none"),
    ("tc128_long_q_short_k", 1, 2, 2, 1000, 64, 128, 128, "bf16", False, "none"),
    # more work units than SMs, so each persistent CTA walks several; causal
    # units of 1..5 tiles put short units back to back
    ("tc64_causal_many_units", 8, 8, 8, 640, 640, 64, 64, "bf16", True, "none"),
    ("tc128_gqa_mask_many_units", 16, 8, 4, 384, 384, 128, 128, "bf16", True, "random"),
    ("simt_f32_odd", 1, 2, 1, 40, 50, 16, 24, "f32", True, "none"),
    ("simt_f32_mask", 2, 2, 2, 33, 65, 64, 64, "f32", False, "random"),
    ("simt_bf16_odd", 1, 2, 1, 33, 47, 40, 24, "bf16", False, "random"),
    ("simt_f32_wide", 1, 1, 1, 20, 30, 256, 200, "f32", True, "none"),
    # padding masks: whole tiles of -inf past the last live key / query tile
    # are skipped (a query tile with no live key keeps one tile)
    ("tc128_pad_mask_gqa", 2, 4, 2, 700, 900, 128, 128, "bf16", False, "pad"),
    ("tc64_pad_mask_causal", 1, 2, 1, 700, 700, 64, 64, "bf16", True, "pad"),
    ("tc128_pad_many_units", 8, 8, 4, 512, 1024, 128, 128, "bf16", False, "pad"),
    ("tc128_f16_pad_mask", 2, 4, 2, 300, 600, 128, 128, "f16", True, "pad"),
    # block-diagonal (documents) and banded (sliding window) masks: -inf tiles
    # before and after each tile row's live span are skipped ("band:1": keys
    # within 128 of the scaled diagonal)
    ("tc128_docs_mask_gqa", 2, 4, 2, 900, 1100, 128, 128, "bf16", False, "docs:4"),
    ("tc64_docs_mask_causal", 1, 2, 1, 1000, 1000, 64, 64, "bf16", True, "docs:3"),
    ("tc128_band_mask", 1, 4, 4, 1000, 1000, 128, 128, "bf16", False, "band:1"),
    ("tc128_band_causal_NltM", 2, 2, 1, 600, 1300, 128, 128, "bf16", True, "band:2"),
    ("tc128_docs_many_units", 8, 8, 4, 640, 640, 128, 128, "bf16", False, "docs:5"),
    ("tc128_f16_band_mask", 2, 4, 2, 700, 700, 128, 128, "f16", False, "band:1"),
    ("simt_f32_docs", 1, 2, 1, 150, 170, 32, 32, "f32", False, "docs:3"),
    # float16 inputs: the tensor-core passes with f16 operands, the CUDA-core path
    ("tc128_f16_causal_gqa_mask", 2, 4, 2, 200, 300, 128, 128, "f16", True, "random"),
    ("tc64_f16_mask_ragged", 1, 4, 2, 96, 130, 64, 64, "f16", False, "random"),
    ("tc128_f16_many_units", 16, 8, 4, 384, 384, 128, 128, "f16", True, "none"),
    ("tc64_f16_causal_gqa", 2, 4, 2, 260, 260, 64, 64, "f16", True, "none"),
    ("simt_f16_odd", 1, 2, 1, 33, 47, 40, 24, "f16", False, "random"),
    # the pages' packing shape: widths below one 16-byte chunk, DK != DV
    ("simt_f32_dk3_dv5", 2, 4, 2, 37, 29, 3, 5, "f32", False, "random"),
    ("simt_bf16_dk3_dv5", 1, 2, 1, 33, 20, 3, 5, "bf16", True, "none"),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_cases(case):
    name, B, H, Hkv, N, M, DK, DV, dtype, causal, mask = case
    mask, _, parts = mask.partition(":")
    w = inputs.custom(B, H, Hkv, N, M, DK, DV, dtype=dtype, causal=causal, mask=mask, seed=zlib.crc32(name.encode()) % 1000,
                      dist="uniform" if dtype == "f32" else "normal", parts=int(parts or 4), name=name)
    x = inputs.make(w)
    gpu = run_gpu(w, x)
    ref = oracle_ref(w, x)
    errs = compare(w, gpu, ref)
    tol = TOL[dtype]
    for key in ("dq", "dk", "dv", "o"):
        assert errs[key] <= tol, (key, errs)
    assert errs["lse"] <= 1e-3 * max(1.0, float(np.nanmax(np.abs(ref["lse"][np.isfinite(ref["lse"])]))))
    check_pads_zero(w, gpu["packed"])


def test_masked_units_past_the_span_table():
    # more masked work units per CTA than the kernels' span tables hold (160
    # units each): units past the table walk their whole tile range instead
    # of the live span, which only adds exact zeros.  The padding mask makes
    # the second key tile (keys 128, 129) and the last query rows all -inf.
    # One query tile per head: the query pass and the forward run B*H =
    # 24,576 units, the key pass B*Hkv*2 = 24,576, so every persistent CTA
    # walks 161-162 units (152 SMs).
    B, H, Hkv, N, M, D = 16, 1536, 768, 16, 130, 64
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert B * H > 160 * sms and B * Hkv * 2 > 160 * sms, "the shape no longer passes the span tables"
    w = inputs.custom(B, H, Hkv, N, M, D, D, mask="pad", mask_p=0.05, seed=77, name="past_span_table")
    x = inputs.make(w)
    gpu = run_gpu(w, x)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    # o and lse NULL: the forward inside fab_backward walks its span table too
    recomputed = binding.backward(g["q"], g["k"], g["v"], g["d"], None, None, g["mask"], w.causal, w.scale)
    torch.cuda.synchronize()
    assert binding.fab_last_device_error() == binding.FAB_OK
    assert np.array_equal(recomputed.to("cpu", torch.float64).numpy(), gpu["packed"])
    del g, recomputed
    ref = oracle_ref(w, x)
    errs = compare(w, gpu, ref)
    for key in ("dq", "dk", "dv", "o"):
        assert errs[key] <= TOL["bf16"], (key, errs)
    check_pads_zero(w, gpu["packed"])


def test_unattended_keys_and_masked_rows_exact_zero():
    # causal with N < M leaves keys >= N unattended (a whole key tile of them);
    # a fully masked query row must get dQ exactly 0
    w = inputs.custom(1, 2, 1, 100, 400, 128, causal=True, mask="random", mask_p=0.05, seed=3)
    x = inputs.make(w)
    gpu = run_gpu(w, x)
    assert np.all(gpu["dk"][:, :, 100:] == 0) and np.all(gpu["dv"][:, :, 100:] == 0)
    n = x["masked_query"]
    assert np.all(gpu["dq"][:, :, n] == 0)
    assert np.all(gpu["o"][:, n] == 0) and np.all(np.isinf(gpu["lse"][:, :, n]))
    ref = oracle_ref(w, x)
    errs = compare(w, gpu, ref)
    assert max(errs["dq"], errs["dk"], errs["dv"]) <= TOL["bf16"], errs


def test_ones_upstream_positive_dv():
    # d = 1: dV of an attended key is the sum of its attention weights (> 0)
    w = inputs.custom(1, 2, 2, 128, 128, 128, seed=5)
    x = inputs.make(w)
    x["d"] = torch.ones_like(x["d"])
    gpu = run_gpu(w, x)
    assert np.all(gpu["dv"] > 0)


def test_linearity_in_upstream_gradient():
    w = inputs.custom(1, 2, 1, 192, 192, 128, causal=True, seed=9)
    x = inputs.make(w)
    a = run_gpu(w, x)
    x2 = dict(x)
    x2["d"] = (x["d"].float() * 2).to(x["d"].dtype)  # exact in bf16
    b = run_gpu(w, x2)
    for key in ("dq", "dk", "dv"):
        np.testing.assert_allclose(b[key], 2 * a[key], rtol=1e-5, atol=1e-6)


def test_repeat_calls_identical():
    # the packed buffer and workspace are fully rewritten on every call
    w = inputs.custom(2, 4, 2, 256, 256, 128, causal=True, seed=11)
    x = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inputs.make(w).items()}
    o, lse = binding.forward(x["q"], x["k"], x["v"], None, True, w.scale)
    dims = binding.dims_of(x["q"], x["k"], x["v"])
    ws, packed = binding.alloc_backward(dims, binding.FAB_BF16, x["q"].device)
    packed.fill_(float("nan"))
    ws.fill_(255)
    binding.fab_backward(x["q"], x["k"], x["v"], x["d"], o, lse, None, True, w.scale, ws, packed)
    first = packed.clone()
    binding.fab_backward(x["q"], x["k"], x["v"], x["d"], o, lse, None, True, w.scale, ws, packed)
    assert binding.fab_last_device_error() == binding.FAB_OK
    assert torch.isfinite(first).all()
    # dQ accumulation order may differ between calls; values agree to rounding
    torch.testing.assert_close(packed, first, rtol=1e-5, atol=1e-6)


# ----------------------------------------------------------------------------- the five workloads

@pytest.mark.parametrize("name", inputs.ORDER + inputs.EXTRA)
def test_workload_parity(name):
    w = inputs.WORKLOADS[name]
    x = inputs.make(w)
    gpu = run_gpu(w, x)
    # every unit and every row: the oracle runs one (batch, key/value head)
    # unit per host thread (long_seq: 16 units of one 16384-row head each)
    ref = oracle_ref(w, x)
    errs = compare(w, gpu, ref)
    tol = TOL[w.dtype]
    for key in ("dq", "dk", "dv", "o"):
        assert errs[key] <= tol, (name, key, errs)
    fin = np.isfinite(ref["lse"])
    assert errs["lse"] <= 1e-3 * max(1.0, float(np.max(np.abs(ref["lse"][fin])))), errs
    check_pads_zero(w, gpu["packed"])
    assert np.all(np.isfinite(gpu["packed"]))
    if w.mask == "random":
        n = x["masked_query"]
        assert np.all(gpu["dq"][:, :, n] == 0), "fully masked query must get zero gradient"


@pytest.mark.parametrize("dtype,DV", [("bf16", 128), ("bf16", 64), ("bf16", 40), ("f32", 128), ("f32", 30)])
def test_preprocess_di_and_zero_fill(dtype, DV):
    import oracle

    w = inputs.custom(2, 6, 3, 77, 50, 128 if DV in (64, 128) else DV, DV, dtype=dtype, seed=DV)
    x = inputs.make(w)
    dev = torch.device("cuda")
    d = x["d"].to(dev)
    o = inputs.make(inputs.custom(2, 6, 3, 77, 50, w.DK, DV, dtype=dtype, seed=DV + 1))["d"].to(dev)
    dims = binding.make_dims(*w.dims)
    ws, packed = binding.alloc_backward(dims, binding.dtype_code(d), dev)
    packed.fill_(7.0)
    binding.fab_backward_preprocess(d, o, dims, ws, packed)
    torch.cuda.synchronize()
    di = ws[: 2 * 6 * 77 * 4].view(torch.float32).view(2, 6, 77).double().cpu().numpy()
    want = oracle.di_rowdot(x["d"], o.cpu())
    np.testing.assert_allclose(di, want, rtol=1e-5, atol=1e-5)
    p = packed.double().cpu().numpy()
    off_k, off_v, end = (t // 4 for t in binding.fab_packed_offsets(dims))
    nq, nk, nv = w.DK * 77 * 6 * 2, w.DK * 50 * 3 * 2, DV * 50 * 3 * 2
    # the preprocess writes D_i and zeroes the padding only: every kernel
    # writes its gradient slice whole, so the slices keep the fill value
    assert np.all(p[:nq] == 7.0) and np.all(p[nq:off_k] == 0)
    assert np.all(p[off_k:off_k + nk] == 7.0) and np.all(p[off_k + nk:off_v] == 0)
    assert np.all(p[off_v:off_v + nv] == 7.0) and np.all(p[off_v + nv:] == 0)


@pytest.mark.parametrize("D,causal,mask", [(128, True, "none"), (64, False, "random")])
def test_every_slice_written_over_garbage(D, causal, mask):
    # the packed buffer starts as NaN: the preprocess zeroes only the padding,
    # so every gradient element must be written by the kernels themselves
    w = inputs.custom(2, 4, 2, 200, 300, D, D, causal=causal, mask=mask, seed=31 + D)
    x = inputs.make(w)
    dev = torch.device("cuda")
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o, lse = binding.forward(g["q"], g["k"], g["v"], g["mask"], w.causal, w.scale)
    dims = binding.make_dims(*w.dims)
    ws, packed = binding.alloc_backward(dims, binding.dtype_code(g["q"]), dev)
    packed.fill_(float("nan"))
    binding.fab_backward(g["q"], g["k"], g["v"], g["d"], o, lse, g["mask"], w.causal, w.scale, ws, packed)
    assert binding.fab_last_device_error() == binding.FAB_OK
    p = packed.double().cpu().numpy()
    assert np.all(np.isfinite(p))
    check_pads_zero(w, p)
    dq, dk, dv = (t.double().cpu().numpy() for t in binding.unpack(packed, dims))
    ref = oracle_ref(w, x)
    for key, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert rel_err(got, ref[key]) <= TOL["bf16"], key


@pytest.mark.parametrize("case", [("tc128_gqa_causal", 2, 4, 2, 200, 300, 128, 128, "bf16", True, "random"),
                                  ("simt_f32", 1, 2, 1, 40, 50, 16, 24, "f32", True, "none"),
                                  # the recomputed forward skips the mask's all -inf tiles too
                                  ("tc128_docs", 2, 4, 2, 700, 900, 128, 128, "bf16", False, "docs:4"),
                                  ("tc64_pad_causal", 1, 2, 1, 700, 700, 64, 64, "bf16", True, "pad:4"),
                                  ("tc128_f16_band", 2, 4, 2, 600, 600, 128, 128, "f16", False, "band:1")],
                         ids=lambda c: c[0])
def test_backward_without_o_and_lse(case):
    # o and lse NULL: the library recomputes the forward into the workspace;
    # the result is the explicit forward-then-backward result, bit for bit,
    # and meets the oracle at the usual tolerance
    name, B, H, Hkv, N, M, DK, DV, dtype, causal, mask = case
    mask, _, parts = mask.partition(":")
    w = inputs.custom(B, H, Hkv, N, M, DK, DV, dtype=dtype, causal=causal, mask=mask, seed=71,
                      dist="uniform" if dtype == "f32" else "normal", parts=int(parts or 4), name=name)
    x = inputs.make(w)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o, lse = binding.forward(g["q"], g["k"], g["v"], g["mask"], w.causal, w.scale)
    explicit = binding.backward(g["q"], g["k"], g["v"], g["d"], o, lse, g["mask"], w.causal, w.scale)
    recomputed = binding.backward(g["q"], g["k"], g["v"], g["d"], None, None, g["mask"], w.causal, w.scale)
    torch.cuda.synchronize()
    assert binding.fab_last_device_error() == binding.FAB_OK
    assert torch.equal(explicit, recomputed)
    dims = binding.dims_of(g["q"], g["k"], g["v"])
    ws = torch.full((binding.fab_backward_recompute_workspace_bytes(dims, binding.dtype_code(g["q"])),), 255,
                    dtype=torch.uint8, device="cuda")
    packed = torch.full((binding.fab_packed_bytes(dims) // 4,), float("nan"), device="cuda")
    binding.fab_backward(g["q"], g["k"], g["v"], g["d"], None, None, g["mask"], w.causal, w.scale, ws, packed)
    torch.cuda.synchronize()
    assert torch.equal(packed, explicit)
    # the O and LSE it recomputed (after D_i and the mask's live-tile maps)
    # are the forward's own, bit for bit
    aux = binding.fab_backward_workspace_bytes(dims, binding.dtype_code(g["q"]))
    ob = o.numel() * o.element_size()
    o_ws = ws[aux:aux + ob].view(o.dtype).view(o.shape)
    lse_at = aux + (ob + 255) // 256 * 256
    lse_ws = ws[lse_at:lse_at + lse.numel() * 4].view(torch.float32).view(lse.shape)
    assert torch.equal(o_ws, o)
    assert torch.equal(lse_ws, lse)
    ref = oracle_ref(w, x)
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
    dq, dk, dv = binding.unpack(recomputed, dims)
    gpu = dict(dq=f64(dq), dk=f64(dk), dv=f64(dv), o=f64(o), lse=f64(lse))
    errs = compare(w, gpu, ref)
    for key in ("dq", "dk", "dv", "o"):
        assert errs[key] <= TOL[dtype], (key, errs)


@pytest.mark.parametrize("D,dtype,causal,mask,parts", [(128, "bf16", False, "pad", 4), (64, "bf16", True, "pad", 4),
                                                       (128, "f16", True, "pad", 4), (128, "bf16", False, "docs", 4),
                                                       (64, "bf16", True, "band", 1), (128, "bf16", False, "band", 2)])
def test_mask_tile_skipping_is_exact(D, dtype, causal, mask, parts):
    # a tile whose mask entries are all -inf contributes P = 0 and dS = 0, so
    # skipping it adds nothing that was not +0: with the tile spans (the full
    # workspace) and without them (a workspace that ends after D_i) the
    # gradients agree bit for bit; padding, document and band masks leave
    # whole tiles -inf, after and before the live ones
    w = inputs.custom(2, 4, 2, 700, 900, D, D, dtype=dtype, causal=causal, mask=mask, mask_p=0.05, seed=83 + D,
                      parts=parts)
    x = inputs.make(w)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o, lse = binding.forward(g["q"], g["k"], g["v"], g["mask"], w.causal, w.scale)
    dims = binding.dims_of(g["q"], g["k"], g["v"])
    full = binding.fab_backward_workspace_bytes(dims, binding.dtype_code(g["q"]))
    di_only = (w.B * w.H * w.N * 4 + 255) // 256 * 256
    assert di_only < full
    outs = []
    for wsb in (full, di_only):
        ws = torch.full((wsb,), 255, dtype=torch.uint8, device="cuda")
        packed = torch.full((binding.fab_packed_bytes(dims) // 4,), float("nan"), device="cuda")
        binding.fab_backward(g["q"], g["k"], g["v"], g["d"], o, lse, g["mask"], w.causal, w.scale, ws, packed)
        outs.append(packed)
    torch.cuda.synchronize()
    assert binding.fab_last_device_error() == binding.FAB_OK
    assert torch.equal(outs[0], outs[1])
    assert not torch.isnan(outs[0]).any()


@pytest.mark.parametrize("D,causal,mask", [(128, True, "none"), (64, False, "random"), (128, False, "random")])
def test_two_phase_api_matches_fab_backward(D, causal, mask):
    # fab_backward_preprocess + fab_backward_main (D_i from the preprocess),
    # fab_backward_query_pass + fab_backward_key_pass and fab_backward (D_i
    # inside the query pass) must give the same gradients bit for bit: the
    # arithmetic per element is the same
    w = inputs.custom(2, 4, 2, 300, 260, D, D, causal=causal, mask=mask, seed=41 + D)
    x = inputs.make(w)
    dev = torch.device("cuda")
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o, lse = binding.forward(g["q"], g["k"], g["v"], g["mask"], w.causal, w.scale)
    dims = binding.make_dims(*w.dims)
    ws, a = binding.alloc_backward(dims, binding.dtype_code(g["q"]), dev)
    a.fill_(float("nan"))
    binding.fab_backward(g["q"], g["k"], g["v"], g["d"], o, lse, g["mask"], w.causal, w.scale, ws, a)
    ws2, b = binding.alloc_backward(dims, binding.dtype_code(g["q"]), dev)
    b.fill_(float("nan"))
    binding.fab_backward_preprocess(g["d"], o, dims, ws2, b)
    binding.fab_backward_main(g["q"], g["k"], g["v"], g["d"], lse, g["mask"], w.causal, w.scale, ws2, b)
    ws3, c = binding.alloc_backward(dims, binding.dtype_code(g["q"]), dev)
    c.fill_(float("nan"))
    binding.fab_backward_query_pass(g["q"], g["k"], g["v"], g["d"], o, lse, g["mask"], w.causal, w.scale, ws3, c)
    binding.fab_backward_key_pass(g["q"], g["k"], g["v"], g["d"], lse, g["mask"], w.causal, w.scale, ws3, c)
    assert binding.fab_last_device_error() == binding.FAB_OK
    n = w.B * w.H * w.N
    di_a = ws[: 4 * n].view(torch.float32).cpu()
    di_b = ws2[: 4 * n].view(torch.float32).cpu()
    # D_i: same products, summed in a different order by the two kernels
    torch.testing.assert_close(di_a, di_b, rtol=1e-5, atol=1e-5)
    assert torch.equal(a, c)
    ref = oracle_ref(w, x)
    for packed in (a, b):
        p = packed.double().cpu().numpy()
        assert np.all(np.isfinite(p))
        check_pads_zero(w, p)
        dq, dk, dv = (t.double().cpu().numpy() for t in binding.unpack(packed, dims))
        for key, got in (("dq", dq), ("dk", dk), ("dv", dv)):
            assert rel_err(got, ref[key]) <= TOL["bf16"], key


def test_many_tiles_repeatable_d128():
    # many query tiles per key tile (GQA group of 4, non-causal) exercises the
    # double-buffered score tiles and the shared lane quarters; no gradient
    # uses reductions, so repeated runs must agree bit for bit
    w = inputs.custom(1, 4, 1, 1024, 256, 128, seed=21)
    x = inputs.make(w)
    a = run_gpu(w, x)
    b = run_gpu(w, x)
    for key in ("dq", "dk", "dv"):
        assert np.array_equal(a[key], b[key]), key
    ref = oracle_ref(w, x)
    errs = compare(w, a, ref)
    assert max(errs["dq"], errs["dk"], errs["dv"]) <= TOL["bf16"], errs
