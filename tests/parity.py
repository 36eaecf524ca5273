"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the fp64 oracle on the same inputs, and compare slice by slice.

The metric is max|gpu - ref| / max|ref| per gradient slice (dQ, dK, dV),
gated at 1e-2 for bf16 operands and 2e-3 for f32 inputs.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from attention_backward_tcgen05_gb300 import binding, inputs

# max |gpu - oracle| / max |oracle| per slice.  bf16 (unit roundoff 2^-8) and
# f16 (2^-11) round P and dS to the input type for the tensor core; the f32
# path computes in f32 throughout.
TOL = {"bf16": 1e-2, "f16": 5e-3, "f32": 2e-3}


def run_gpu(w: inputs.Workload, x: dict):
    """Forward + backward on the current CUDA device; returns numpy float64
    (dq, dk, dv, packed, o, lse) and checks the device error word."""
    dev = torch.device("cuda")
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o, lse = binding.forward(g["q"], g["k"], g["v"], g["mask"], w.causal, w.scale)
    packed = binding.backward(g["q"], g["k"], g["v"], g["d"], o, lse, g["mask"], w.causal, w.scale)
    status = binding.fab_last_device_error()
    assert status == binding.FAB_OK, binding.status_string(status)
    dims = binding.make_dims(*w.dims)
    dq, dk, dv = binding.unpack(packed, dims)
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
    return dict(dq=f64(dq), dk=f64(dk), dv=f64(dv), packed=f64(packed), o=f64(o), lse=f64(lse))


def rel_err(got, ref):
    den = np.max(np.abs(ref))
    if den == 0:
        return float(np.max(np.abs(got)))
    return float(np.max(np.abs(got - ref)) / den)


def units_heads(w: inputs.Workload, units):
    rk2 = w.H // w.Hkv
    out = []
    for u in units:
        b, hk = divmod(u, w.Hkv)
        out.append((b, hk, list(range(hk * rk2, (hk + 1) * rk2))))
    return out


def compare(w: inputs.Workload, gpu: dict, ref: dict, units=None, check_forward=True, rows=None):
    """Returns {slice: rel_err}; with `units`, only those (b, hk) units.

    With `rows=(n0, N)` on a causal workload (the oracle visited query rows
    n >= n0 only) the comparison covers dQ/O rows n >= n0 and dK/dV keys
    m >= n0, which those rows determine exactly.
    """
    if rows is not None:
        assert w.causal and rows[1] == w.N
        n0 = rows[0]
        cut = lambda d: dict(dq=d["dq"][:, :, n0:], dk=d["dk"][:, :, n0:], dv=d["dv"][:, :, n0:],
                             o=d["o"][:, n0:], lse=d["lse"][:, :, n0:])
        gpu, ref = cut(gpu), cut(ref)
    errs = {}
    if units is None:
        for key in ("dq", "dk", "dv"):
            errs[key] = rel_err(gpu[key], ref[key])
        if check_forward:
            errs["o"] = rel_err(gpu["o"], ref["o"])
            fin = np.isfinite(ref["lse"])
            assert np.array_equal(np.isfinite(gpu["lse"]), fin), "LSE finiteness differs"
            errs["lse"] = float(np.max(np.abs(gpu["lse"][fin] - ref["lse"][fin]))) if fin.any() else 0.0
        return errs
    sel = units_heads(w, units)
    gq = np.concatenate([gpu["dq"][b, hs].ravel() for b, _, hs in sel])
    rq = np.concatenate([ref["dq"][b, hs].ravel() for b, _, hs in sel])
    gk = np.concatenate([gpu["dk"][b, hk].ravel() for b, hk, _ in sel])
    rk = np.concatenate([ref["dk"][b, hk].ravel() for b, hk, _ in sel])
    gv = np.concatenate([gpu["dv"][b, hk].ravel() for b, hk, _ in sel])
    rv = np.concatenate([ref["dv"][b, hk].ravel() for b, hk, _ in sel])
    errs = dict(dq=rel_err(gq, rq), dk=rel_err(gk, rk), dv=rel_err(gv, rv))
    if check_forward:
        go = np.concatenate([gpu["o"][b][:, hs].ravel() for b, _, hs in sel])
        ro = np.concatenate([ref["o"][b][:, hs].ravel() for b, _, hs in sel])
        errs["o"] = rel_err(go, ro)
    return errs


def check_pads_zero(w: inputs.Workload, packed: np.ndarray):
    B, H, Hkv, N, M, DK, DV = w.dims
    off_k, off_v, end = (t // 4 for t in oracle.packed_layout(w.dims))
    nq, nk, nv = DK * N * H * B, DK * M * Hkv * B, DV * M * Hkv * B
    assert len(packed) == end
    assert np.all(packed[nq:off_k] == 0) and np.all(packed[off_k + nk:off_v] == 0) and np.all(packed[off_v + nv:] == 0)


def oracle_ref(w: inputs.Workload, x: dict, units=None, threads=0, rows=None):
    return oracle.backward(x["q"], x["k"], x["v"], x["d"], x["mask"], w.causal, w.scale, units=units,
                           threads=threads, rows=rows)
