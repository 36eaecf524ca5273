"""Pins for the fp64 oracle, independent of the oracle itself (CPU only).

Each check is something the pages or the mathematics fix:
  * central differences of sum(d * attn(q, k, v)) on the ggmlR test shapes
    (test-flash-attn-back.R, num_grad: eps 1e-3, tolerance 2e-2);
  * a library attention routine in float64 (torch scaled_dot_product_attention
    and its autograd) on shapes with GQA, batches, masks;
  * closed forms: two keys (logistic weights), identical keys (uniform P),
    M = 1, identical value rows, scale = 0;
  * invariants: sum over keys of dK is 0, the two forms of D_i agree, fully
    masked rows and unattended keys get exactly zero, d = 1 gives positive
    dV, gradients are linear in d, GQA equals the group sum of replicated MHA;
  * the packed layout against hand-worked offsets and the ggmlR packing test.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from attention_backward_tcgen05_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
CONST = json.load(open(os.path.join(GOLDEN, "pages_constants.json")))
EPS = CONST["fd_eps"]["value"]
FD_TOL = CONST["fd_tolerance"]["value"]


def rand_case(rng, B, H, Hkv, N, M, DK, DV, lo=-1.0, hi=1.0):
    q = rng.uniform(lo, hi, (B, H, N, DK))
    k = rng.uniform(lo, hi, (B, Hkv, M, DK))
    v = rng.uniform(lo, hi, (B, Hkv, M, DV))
    d = rng.uniform(lo, hi, (B, N, H, DV))
    return q, k, v, d


def page_causal_mask(N, M):
    """ggmlR 'handles a mask': mask[(n+1):M, n] <- -Inf (R, 1-based) -> keys m > n masked."""
    mask = np.zeros((N, M))
    for n in range(N):
        mask[n, n + 1:] = -np.inf
    return mask


def num_grad(q, k, v, d, scale, mask, which, causal=False, eps=EPS):
    vals = {"q": q, "k": k, "v": v}
    x = vals[which]
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        hi = {kk: vv.copy() for kk, vv in vals.items()}
        lo = {kk: vv.copy() for kk, vv in vals.items()}
        hi[which][idx] += eps
        lo[which][idx] -= eps
        fh = np.sum(d * oracle.forward(hi["q"], hi["k"], hi["v"], mask, causal, scale)[0])
        fl = np.sum(d * oracle.forward(lo["q"], lo["k"], lo["v"], mask, causal, scale)[0])
        g[idx] = (fh - fl) / (2 * eps)
    return g


def mean_rel(a, b):
    """testthat / all.equal tolerance metric: mean |a-b| / mean |b|."""
    return float(np.mean(np.abs(a - b)) / np.mean(np.abs(b)))


# --------------------------------------------------------------------------- finite differences


@pytest.mark.parametrize("case", CONST["fd_cases"]["cases"], ids=lambda c: c["name"])
def test_fd_pages_shapes(case):
    rng = np.random.default_rng(case["seed_label"])
    B, H, Hkv, N, M, DK, DV = (case[x] for x in ("B", "H", "Hkv", "N", "M", "DK", "DV"))
    q, k, v, d = rand_case(rng, B, H, Hkv, N, M, DK, DV)
    scale = 1.0 / math.sqrt(DK)
    mask = page_causal_mask(N, M) if case["mask"] == "causal" else None
    g = oracle.backward(q, k, v, d, mask, False, scale)
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv")):
        fd = num_grad(q, k, v, d, scale, mask, name)
        assert mean_rel(g[key], fd) < FD_TOL, name
        # in fp64 the central difference is accurate to O(eps^2)
        assert np.max(np.abs(g[key] - fd)) < 1e-5, name
    assert np.all(np.isfinite(g["dk"]))


def test_fd_causal_flag_equals_page_mask():
    rng = np.random.default_rng(12)
    q, k, v, d = rand_case(rng, 1, 2, 1, 3, 4, 4, 4)
    scale = 0.5
    a = oracle.backward(q, k, v, d, page_causal_mask(3, 4), False, scale)
    b = oracle.backward(q, k, v, d, None, True, scale)
    for key in ("dq", "dk", "dv", "o", "lse", "di"):
        np.testing.assert_array_equal(a[key], b[key])
    # finite differences through the causal flag as well
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv")):
        fd = num_grad(q, k, v, d, scale, None, name, causal=True)
        assert np.max(np.abs(b[key] - fd)) < 1e-5


def test_fd_mask_and_asymmetric_dims():
    rng = np.random.default_rng(7)
    q, k, v, d = rand_case(rng, 2, 3, 1, 3, 5, 3, 5)
    mask = rng.uniform(-2, 2, (3, 5))
    mask[1, 2] = -np.inf
    scale = 0.7
    g = oracle.backward(q, k, v, d, mask, False, scale)
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv")):
        fd = num_grad(q, k, v, d, scale, mask, name)
        assert np.max(np.abs(g[key] - fd)) < 1e-5, name


# --------------------------------------------------------------------------- library routine (float64)


def sdpa_reference(q, k, v, d, mask, scale):
    """torch SDPA in float64 with autograd; K/V heads expanded to the query heads."""
    B, H, N, DK = q.shape
    Hkv = k.shape[1]
    rk2 = H // Hkv
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    kk = tk.repeat_interleave(rk2, dim=1)
    vv = tv.repeat_interleave(rk2, dim=1)
    am = None if mask is None else torch.tensor(mask)
    o = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, attn_mask=am, scale=scale)  # (B,H,N,DV)
    o_ours = o.permute(0, 2, 1, 3)  # (B,N,H,DV)
    (o_ours * torch.tensor(d)).sum().backward()
    s = torch.einsum("bhnd,bhmd->bhnm", tq.detach(), kk.detach()) * scale
    if am is not None:
        s = s + am
    lse = torch.logsumexp(s, dim=-1)
    return dict(o=o_ours.detach().numpy(), lse=lse.numpy(), dq=tq.grad.numpy(), dk=tk.grad.numpy(),
                dv=tv.grad.numpy())


@pytest.mark.parametrize("shape", [(1, 1, 1, 7, 9, 8, 8), (2, 4, 2, 5, 11, 6, 3), (2, 6, 3, 16, 16, 16, 16)])
@pytest.mark.parametrize("masked", [False, True])
def test_against_library_float64(shape, masked):
    rng = np.random.default_rng(sum(shape) + masked)
    B, H, Hkv, N, M, DK, DV = shape
    q, k, v, d = rand_case(rng, *shape, lo=-2, hi=2)
    mask = None
    if masked:
        mask = rng.uniform(-3, 3, (N, M))
        drop = rng.uniform(size=(N, M)) < 0.3
        drop[:, 0] = False  # keep one key per row so the library's softmax stays finite
        mask[drop] = -np.inf
    scale = 0.37
    ref = sdpa_reference(q, k, v, d, mask, scale)
    g = oracle.backward(q, k, v, d, mask, False, scale)
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(g[key], ref[key], rtol=1e-10, atol=1e-11, err_msg=key)


def test_causal_against_library_top_left():
    rng = np.random.default_rng(5)
    q, k, v, d = rand_case(rng, 1, 2, 2, 6, 9, 4, 4)  # N < M: top-left alignment matters
    ref = sdpa_reference(q, k, v, d, page_causal_mask(6, 9), 0.5)
    g = oracle.backward(q, k, v, d, None, True, 0.5)
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(g[key], ref[key], rtol=1e-10, atol=1e-11, err_msg=key)


# --------------------------------------------------------------------------- closed forms


def test_two_keys_logistic_closed_form():
    # one query, two keys, D = 1: p1 = sigmoid(s1 - s2); O = p1 v1 + p2 v2
    qv, k1, k2, v1, v2, dd, sc = 0.8, -0.3, 1.1, 0.25, -1.5, 0.6, 0.9
    q = np.array(qv).reshape(1, 1, 1, 1)
    k = np.array([k1, k2]).reshape(1, 1, 2, 1)
    v = np.array([v1, v2]).reshape(1, 1, 2, 1)
    d = np.array(dd).reshape(1, 1, 1, 1)
    g = oracle.backward(q, k, v, d, None, False, sc)
    p1 = 1.0 / (1.0 + math.exp(-(sc * qv * k1 - sc * qv * k2)))
    p2 = 1.0 - p1
    w = dd * p1 * p2 * (v1 - v2)
    assert g["o"].item() == pytest.approx(p1 * v1 + p2 * v2, rel=1e-14)
    assert g["lse"].item() == pytest.approx(math.log(math.exp(sc * qv * k1) + math.exp(sc * qv * k2)), rel=1e-14)
    assert g["dq"].item() == pytest.approx(sc * w * (k1 - k2), rel=1e-12)
    assert g["dk"][0, 0, 0, 0] == pytest.approx(sc * w * qv, rel=1e-12)
    assert g["dk"][0, 0, 1, 0] == pytest.approx(-sc * w * qv, rel=1e-12)
    assert g["dv"][0, 0, 0, 0] == pytest.approx(dd * p1, rel=1e-14)
    assert g["dv"][0, 0, 1, 0] == pytest.approx(dd * p2, rel=1e-14)


def test_identical_keys_uniform():
    rng = np.random.default_rng(3)
    B, H, Hkv, N, M, D = 2, 4, 2, 5, 7, 6
    q, k, v, d = rand_case(rng, B, H, Hkv, N, M, D, D)
    k[:] = k[:, :, :1, :]  # every key equal
    g = oracle.backward(q, k, v, d, None, False, 0.8)
    rk2 = H // Hkv
    for b in range(B):
        for h in range(H):
            hk = h // rk2
            np.testing.assert_allclose(g["o"][b, :, h, :], np.broadcast_to(v[b, hk].mean(0), (N, D)), rtol=1e-12)
    np.testing.assert_allclose(g["dq"], 0.0, atol=1e-14)
    for b in range(B):
        for hk in range(Hkv):
            want = d[b, :, hk * rk2:(hk + 1) * rk2, :].sum(axis=(0, 1)) / M
            np.testing.assert_allclose(g["dv"][b, hk], np.broadcast_to(want, (M, D)), rtol=1e-12)
    # dQ is still 0 with a mask: each row's dS sums to 0
    mask = rng.uniform(-1, 1, (N, M))
    g2 = oracle.backward(q, k, v, d, mask, False, 0.8)
    np.testing.assert_allclose(g2["dq"], 0.0, atol=1e-13)


def test_single_key():
    rng = np.random.default_rng(4)
    q, k, v, d = rand_case(rng, 1, 3, 1, 4, 1, 5, 3)
    g = oracle.backward(q, k, v, d, None, False, 1.3)
    np.testing.assert_allclose(g["o"], np.broadcast_to(v[0, 0, 0], (1, 4, 3, 3)), rtol=1e-14)
    np.testing.assert_allclose(g["dq"], 0.0, atol=1e-15)
    np.testing.assert_allclose(g["dk"], 0.0, atol=1e-15)
    np.testing.assert_allclose(g["dv"][0, 0, 0], d.sum(axis=(0, 1, 2)), rtol=1e-13)


def test_identical_value_rows():
    rng = np.random.default_rng(8)
    q, k, v, d = rand_case(rng, 1, 2, 2, 4, 6, 3, 3)
    v[:] = v[:, :, :1, :]
    g = oracle.backward(q, k, v, d, None, False, 0.9)
    np.testing.assert_allclose(g["dq"], 0.0, atol=1e-14)
    np.testing.assert_allclose(g["dk"], 0.0, atol=1e-14)


def test_zero_scale_uniform():
    rng = np.random.default_rng(9)
    q, k, v, d = rand_case(rng, 1, 1, 1, 3, 5, 4, 4)
    g = oracle.backward(q, k, v, d, None, False, 0.0)
    np.testing.assert_allclose(g["o"][0, :, 0, :], np.broadcast_to(v[0, 0].mean(0), (3, 4)), rtol=1e-13)
    np.testing.assert_allclose(g["lse"], math.log(5), rtol=1e-14)
    np.testing.assert_allclose(g["dq"], 0.0, atol=1e-15)
    np.testing.assert_allclose(g["dk"], 0.0, atol=1e-15)


# --------------------------------------------------------------------------- invariants


def test_invariants_random():
    rng = np.random.default_rng(21)
    B, H, Hkv, N, M, D = 2, 4, 2, 9, 12, 5
    q, k, v, d = rand_case(rng, B, H, Hkv, N, M, D, D)
    mask = rng.uniform(-1, 1, (N, M))
    mask[rng.uniform(size=(N, M)) < 0.2] = -np.inf
    mask[4, :] = -np.inf  # one fully masked query
    g = oracle.backward(q, k, v, d, mask, True, 0.6)
    # sum_m dS_nm = 0 for every row => sum over keys of dK is 0
    np.testing.assert_allclose(g["dk"].sum(axis=2), 0.0, atol=1e-13)
    # the two forms of D_i agree
    np.testing.assert_allclose(oracle.di_rowdot(d, g["o"]), g["di"], rtol=1e-12, atol=1e-14)
    # the fully masked query: output 0, LSE +inf, no gradient
    assert np.all(g["o"][:, 4] == 0) and np.all(np.isinf(g["lse"][:, :, 4]))
    assert np.all(g["dq"][:, :, 4] == 0)
    # linearity in d
    g2 = oracle.backward(q, k, v, 2.0 * d, mask, True, 0.6)
    for key in ("dq", "dk", "dv"):
        np.testing.assert_allclose(g2[key], 2.0 * g[key], rtol=1e-12, atol=1e-14)


def test_unattended_keys_zero():
    # causal with N < M: keys m >= N are attended by no query
    rng = np.random.default_rng(12)
    q, k, v, d = rand_case(rng, 1, 2, 1, 3, 6, 4, 4)
    g = oracle.backward(q, k, v, d, None, True, 0.5)
    assert np.all(g["dk"][:, :, 3:] == 0) and np.all(g["dv"][:, :, 3:] == 0)
    assert np.all(np.isfinite(g["dk"]))
    assert np.any(g["dk"][:, :, :3] != 0)


def test_ones_upstream_positive_dv():
    # ggmlR graph test: d(sum(softmax(qk)v))/dv is the summed attention weights
    rng = np.random.default_rng(14)
    q, k, v, _ = rand_case(rng, 1, 1, 1, 3, 4, 4, 4)
    g = oracle.backward(q, k, v, np.ones((1, 3, 1, 4)), None, False, 0.5)
    assert np.all(g["dv"] > 0)
    o, _ = oracle.forward(q, k, v, None, False, 0.5)
    # summed attention weights per key, replicated over DV
    s = np.einsum("nd,md->nm", q[0, 0], k[0, 0]) * 0.5
    p = np.exp(s - s.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    np.testing.assert_allclose(g["dv"][0, 0], np.repeat(p.sum(0)[:, None], 4, 1), rtol=1e-13)


def test_gqa_equals_group_sum_of_mha():
    rng = np.random.default_rng(13)
    B, H, Hkv, N, M, D = 2, 6, 2, 5, 7, 4
    q, k, v, d = rand_case(rng, B, H, Hkv, N, M, D, D)
    mask = rng.uniform(-1, 1, (N, M))
    g = oracle.backward(q, k, v, d, mask, True, 0.45)
    rk2 = H // Hkv
    kr = np.repeat(k, rk2, axis=1)
    vr = np.repeat(v, rk2, axis=1)
    m = oracle.backward(q, kr, vr, d, mask, True, 0.45)
    np.testing.assert_allclose(g["dq"], m["dq"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(g["o"], m["o"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(g["dk"], m["dk"].reshape(B, Hkv, rk2, M, D).sum(2), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(g["dv"], m["dv"].reshape(B, Hkv, rk2, M, D).sum(2), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_block_diagonal_mask_splits_into_documents(causal):
    # with -inf between documents (a block-diagonal mask), attention over the
    # whole sequence is attention over each document alone: every row of O,
    # LSE and dQ, and every row of dK and dV, equals the one-document run's.
    # Finite mask values inside the documents take part.  Causal: the
    # documents start at the same index on both axes, so the top-left
    # diagonal inside a document is the document's own.
    rng = np.random.default_rng(21)
    B, H, Hkv, D = 2, 4, 2, 5
    if causal:
        N = M = 10
        qdocs = kdocs = [(0, 4), (4, 10)]
    else:
        N, M = 9, 11
        qdocs, kdocs = [(0, 3), (3, 9)], [(0, 6), (6, 11)]
    q, k, v, d = rand_case(rng, B, H, Hkv, N, M, D, D)
    mask = np.full((N, M), -np.inf)
    for (n0, n1), (m0, m1) in zip(qdocs, kdocs):
        mask[n0:n1, m0:m1] = rng.uniform(-1, 1, (n1 - n0, m1 - m0))
    g = oracle.backward(q, k, v, d, mask, causal, 0.6)
    for (n0, n1), (m0, m1) in zip(qdocs, kdocs):
        r = oracle.backward(q[:, :, n0:n1], k[:, :, m0:m1], v[:, :, m0:m1], d[:, n0:n1],
                            mask[n0:n1, m0:m1], causal, 0.6)
        np.testing.assert_allclose(g["o"][:, n0:n1], r["o"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(g["lse"][:, :, n0:n1], r["lse"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(g["dq"][:, :, n0:n1], r["dq"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(g["dk"][:, :, m0:m1], r["dk"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(g["dv"][:, :, m0:m1], r["dv"], rtol=1e-12, atol=1e-14)


def test_units_subset_matches_full():
    rng = np.random.default_rng(2)
    q, k, v, d = rand_case(rng, 2, 4, 2, 6, 8, 4, 4)
    full = oracle.backward(q, k, v, d, None, True, 0.5)
    part = oracle.backward(q, k, v, d, None, True, 0.5, units=[3])  # b=1, hk=1 -> heads 2,3
    np.testing.assert_array_equal(part["dk"][1, 1], full["dk"][1, 1])
    np.testing.assert_array_equal(part["dv"][1, 1], full["dv"][1, 1])
    np.testing.assert_array_equal(part["dq"][1, 2:4], full["dq"][1, 2:4])
    assert np.all(part["dk"][0] == 0) and np.all(part["dq"][1, :2] == 0)


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(6)
    q, k, v, d = rand_case(rng, 3, 4, 2, 8, 8, 4, 4)
    a = oracle.backward(q, k, v, d, None, True, 0.5, threads=1)
    b = oracle.backward(q, k, v, d, None, True, 0.5, threads=5)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])


def test_rejects_bad_shapes():
    rng = np.random.default_rng(0)
    q, k, v, d = rand_case(rng, 1, 3, 2, 2, 2, 2, 2)  # H % Hkv != 0
    with pytest.raises(ValueError):
        oracle.backward(q, k, v, d)


# --------------------------------------------------------------------------- packed layout


def read_layout_golden():
    rows = []
    for line in open(os.path.join(GOLDEN, "packed_layout.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        a, b = line.split("|")
        rows.append((tuple(int(x) for x in a.split()), tuple(int(x) for x in b.split())))
    return rows


@pytest.mark.parametrize("dims,want", read_layout_golden())
def test_packed_layout_golden(dims, want):
    assert oracle.packed_layout(dims) == want


def test_packing_case_pages():
    c = CONST["packing_case"]
    dims = tuple(c[x] for x in ("B", "H", "Hkv", "N", "M", "DK", "DV"))
    rng = np.random.default_rng(c["seed_label"])
    q, k, v, d = rand_case(rng, *dims)
    g = oracle.backward(q, k, v, d, None, False, 1 / math.sqrt(c["DK"]))
    packed = oracle.pack(dims, g["dq"], g["dk"], g["dv"])
    B, H, Hkv, N, M, DK, DV = dims
    nq, nk, nv = DK * N * H * B, DK * M * Hkv * B, DV * M * Hkv * B
    off_k, off_v, end = (x // 4 for x in oracle.packed_layout(dims))
    assert len(packed) >= off_v + nv and nq <= off_k and off_k + nk <= off_v
    assert np.max(np.abs(packed[:nq])) > 0 and np.max(np.abs(packed[off_k:off_k + nk])) > 0
    assert np.max(np.abs(packed[off_v:off_v + nv])) > 0
    np.testing.assert_array_equal(packed[:nq], g["dq"].ravel())
    np.testing.assert_array_equal(packed[off_k:off_k + nk], g["dk"].ravel())
    np.testing.assert_array_equal(packed[off_v:off_v + nv], g["dv"].ravel())


def test_packing_pads_zero_ragged():
    dims = (1, 1, 1, 3, 5, 3, 5)
    rng = np.random.default_rng(1)
    q, k, v, d = rand_case(rng, *dims)
    g = oracle.backward(q, k, v, d, None, False, 0.5)
    packed = oracle.pack(dims, g["dq"], g["dk"], g["dv"])
    off_k, off_v, end = (x // 4 for x in oracle.packed_layout(dims))
    assert len(packed) == end
    assert np.all(packed[9:off_k] == 0) and np.all(packed[off_k + 15:off_v] == 0) and np.all(packed[off_v + 25:] == 0)


# --------------------------------------------------------------------------- workload generator


def test_workload_inputs_shapes_and_mask():
    w = inputs.custom(2, 4, 2, 16, 64, 8, mask="random", seed=5)
    x = inputs.make(w)
    assert x["q"].shape == (2, 4, 16, 8) and x["k"].shape == (2, 2, 64, 8) and x["d"].shape == (2, 16, 4, 8)
    assert x["q"].dtype == torch.bfloat16 and x["mask"].dtype == torch.float16
    n = x["masked_query"]
    assert torch.all(torch.isinf(x["mask"][n]))
    frac = torch.isinf(x["mask"]).float().mean().item()
    assert 0.05 < frac < 0.2
    y = inputs.make(w)
    assert torch.equal(x["q"], y["q"]) and torch.equal(x["mask"], y["mask"])


def test_row_range_exact_for_late_keys_under_causal():
    # under a causal mask only queries n >= m see key m, so visiting rows
    # [n0, N) gives exact dK/dV for keys >= n0 and exact rows n >= n0
    rng = np.random.default_rng(17)
    q, k, v, d = rand_case(rng, 1, 2, 1, 12, 12, 4, 4)
    full = oracle.backward(q, k, v, d, None, True, 0.5)
    part = oracle.backward(q, k, v, d, None, True, 0.5, rows=(7, 12))
    np.testing.assert_array_equal(part["dk"][:, :, 7:], full["dk"][:, :, 7:])
    np.testing.assert_array_equal(part["dv"][:, :, 7:], full["dv"][:, :, 7:])
    np.testing.assert_array_equal(part["dq"][:, :, 7:], full["dq"][:, :, 7:])
    assert np.all(part["dq"][:, :, :7] == 0)
    with pytest.raises(ValueError):
        oracle.backward(q, k, v, d, None, True, 0.5, rows=(5, 13))
