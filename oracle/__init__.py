"""fp64 CPU oracle for the fused attention backward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  It
shares no code with the CUDA library and the library never calls it.

Array convention (numpy, C order) -- the reverse of ggml's ne order:
    q    (B, H, N, DK)      == ne [DK, N, H, B]
    k    (B, Hkv, M, DK)    == ne [DK, M, Hkv, B]
    v    (B, Hkv, M, DV)    == ne [DV, M, Hkv, B]
    d, o (B, N, H, DV)      == ne [DV, H, N, B]  (the forward output's shape)
    mask (N, M)             == ne [M, N]; added to the score of (query n, key m)
    lse, di (B, H, N)       == ne [N, H, B]

The arithmetic lives in ``fab_oracle.cpp`` (plain loops in double precision);
this module only marshals arrays.  Sources are cited there: the ggmlR test
file's ``attn_ref`` for the forward, the labml "Flash Attention" page's
"Backward pass" section for the gradients, and the ggml
``ggml_flash_attn_back`` constructor for the packed layout.

Parity is pinned in ``tests/test_oracle.py`` against central differences,
a library attention routine in float64 (torch ``scaled_dot_product_attention``
and its autograd), closed forms and invariants.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_forward.argtypes = [dp, dp, dp, dp, ctypes.c_int, ctypes.c_double, ip, dp, dp, ctypes.c_int]
        lib.oracle_backward.argtypes = [dp, dp, dp, dp, dp, ctypes.c_int, ctypes.c_double, ip,
                                        dp, dp, dp, dp, dp, dp, ip, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int]
        lib.oracle_di_rowdot.argtypes = [dp, dp, ip, dp]
        lib.oracle_packed_layout.argtypes = [ip, ip, ip, ip]
        lib.oracle_pack.argtypes = [ip, dp, dp, dp, dp]
        for f in ("oracle_forward", "oracle_backward", "oracle_di_rowdot", "oracle_packed_layout", "oracle_pack"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    try:  # torch tensors (any dtype, any device) are widened exactly to float64
        import torch

        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def dims_of(q, k, v):
    """(B, H, Hkv, N, M, DK, DV) from array shapes."""
    B, H, N, DK = q.shape
    Bk, Hkv, M, DKk = k.shape
    Bv, Hv, Mv, DV = v.shape
    if (Bk, DKk) != (B, DK) or (Bv, Hv, Mv) != (B, Hkv, M):
        raise ValueError("inconsistent q/k/v shapes")
    return (B, H, Hkv, N, M, DK, DV)


def _dims_arr(dims):
    return np.ascontiguousarray(np.asarray(dims, dtype=np.int64))


def forward(q, k, v, mask=None, causal=False, scale=1.0, threads=0):
    """Returns (o (B,N,H,DV), lse (B,H,N)) in float64."""
    q, k, v, mask = _f64(q), _f64(k), _f64(v), _f64(mask)
    dims = dims_of(q, k, v)
    B, H, Hkv, N, M, DK, DV = dims
    if mask is not None and mask.shape != (N, M):
        raise ValueError("mask must be (N, M)")
    o = np.zeros((B, N, H, DV))
    lse = np.zeros((B, H, N))
    da = _dims_arr(dims)
    rc = _load().oracle_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), int(bool(causal)), float(scale),
                                da.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _ptr(o), _ptr(lse), int(threads))
    if rc:
        raise ValueError("oracle_forward rejected the shapes")
    return o, lse


def backward(q, k, v, d, mask=None, causal=False, scale=1.0, units=None, threads=0, rows=None):
    """Analytic gradients in float64.

    Returns a dict with dq (B,H,N,DK), dk (B,Hkv,M,DK), dv (B,Hkv,M,DV),
    o (B,N,H,DV), lse (B,H,N) and di (B,H,N).  With ``units`` (a list of
    b*Hkv + hk indices) only those units are computed; everything else is 0.
    With ``rows=(n_begin, n_end)`` only those query rows are visited: their
    o/lse/di/dq rows are exact and dk/dv hold those rows' contributions only.
    """
    q, k, v, d, mask = _f64(q), _f64(k), _f64(v), _f64(d), _f64(mask)
    dims = dims_of(q, k, v)
    B, H, Hkv, N, M, DK, DV = dims
    if d.shape != (B, N, H, DV):
        raise ValueError("d must be (B, N, H, DV)")
    if mask is not None and mask.shape != (N, M):
        raise ValueError("mask must be (N, M)")
    out = {
        "dq": np.zeros((B, H, N, DK)),
        "dk": np.zeros((B, Hkv, M, DK)),
        "dv": np.zeros((B, Hkv, M, DV)),
        "o": np.zeros((B, N, H, DV)),
        "lse": np.zeros((B, H, N)),
        "di": np.zeros((B, H, N)),
    }
    u = None if units is None else np.ascontiguousarray(np.asarray(units, dtype=np.int64))
    da = _dims_arr(dims)
    ip = ctypes.POINTER(ctypes.c_int64)
    rc = _load().oracle_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(d), _ptr(mask), int(bool(causal)), float(scale), da.ctypes.data_as(ip),
        _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["o"]), _ptr(out["lse"]), _ptr(out["di"]),
        None if u is None else u.ctypes.data_as(ip), 0 if u is None else len(u),
        0 if rows is None else int(rows[0]), N if rows is None else int(rows[1]), int(threads))
    if rc:
        raise ValueError("oracle_backward rejected the arguments")
    return out


def di_rowdot(d, o):
    """D = rowsum(dO * O) over DV for every (b, n, h); returns (B, H, N)."""
    d, o = _f64(d), _f64(o)
    B, N, H, DV = d.shape
    di = np.zeros((B, H, N))
    dims = _dims_arr((B, H, H, N, 1, 1, DV))
    rc = _load().oracle_di_rowdot(_ptr(d), _ptr(o), dims.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _ptr(di))
    if rc:
        raise ValueError("bad shapes")
    return di


def packed_layout(dims):
    """(off_k, off_v, end) in bytes for the packed f32 [dQ | dK | dV] result."""
    da = _dims_arr(dims)
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    rc = _load().oracle_packed_layout(da.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                      ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
    if rc:
        raise ValueError("bad dims")
    return a.value, b.value, c.value


def pack(dims, dq, dk, dv):
    """Packed result as float64 (end/4 entries), zero padding included."""
    dq, dk, dv = _f64(dq), _f64(dk), _f64(dv)
    _, _, end = packed_layout(dims)
    out = np.zeros(end // 4)
    da = _dims_arr(dims)
    rc = _load().oracle_pack(da.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _ptr(dq), _ptr(dk), _ptr(dv),
                             _ptr(out))
    if rc:
        raise ValueError("bad dims")
    return out
