"""fp64 CPU oracle for the differential-attention forward pass.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs are the only callers; the library
under ``transformer_attention_07_b300`` never imports this package and the
two share no code.

What it computes (the Differential Transformer pages):

* "How does Differential Attention work to suppress noise…" (iloveeagents.com),
  "Mathematical Formula": ``(softmax(Q1 K1^T/sqrt d) - lambda softmax(Q2 K2^T/sqrt d)) V``.
  One softmax per map (that page's Example snippet nests a second softmax on
  the second map; the formula and the llmbytes.dev steps do not).
* "Differential Transformer: How Noise-Canceling Attention Reinvents LLMs"
  (llmbytes.dev), "How Differential Attention Cancels Common-Mode Noise",
  steps 2-4: the two maps, the lambda-weighted subtraction, GroupNorm of the
  multi-head output and the ``(1 - lambda_init)`` scale.

The backward pass (``diffattn_bwd``) is the chain rule through the same
steps, one query row at a time; lambda is learnable on the pages, so its
gradient and that of the GroupNorm gain are returned with the input gradients.

The arithmetic lives in ``oracle.cpp`` (fp64, one row at a time, both
softmax rows materialised); this module only marshals arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import time

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

IN_F64, IN_F32, IN_BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile ``oracle.cpp`` into ``liboracle.so`` with the host compiler."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_diffattn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, f64, f64, i32,
                                            i32, i32, i32, i32, i32, i32,
                                            vp, f64, vp, i64, vp, vp, i32]
        lib.oracle_diffattn_fwd.restype = i32
        lib.oracle_diffattn_maps.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp]
        lib.oracle_diffattn_maps.restype = i32
        lib.oracle_diffattn_bwd.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, f64, f64, i32,
                                            i32, i32, i32, i32, i32, i32, vp, f64,
                                            vp, i64, vp, i64, vp, vp, vp, vp, vp, vp, vp, vp, i32]
        lib.oracle_diffattn_bwd.restype = i32
        _lib = lib
    return _lib


def _as_input(x):
    """Return (contiguous numpy array, oracle input-type code).

    Accepts numpy arrays (float64/float32) or torch CPU tensors (float64,
    float32, bfloat16 — the latter passed as raw 16-bit patterns)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), IN_BF16
            if x.dtype == torch.float32:
                return x.numpy(), IN_F32
            return x.to(torch.float64).numpy(), IN_F64
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, IN_F32
    return np.ascontiguousarray(x, dtype=np.float64), IN_F64


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def diffattn_fwd(q1, k1, q2, k2, v, lam, lam_init, causal=False, gamma=None, eps=1e-5,
                 rows=None, threads=0):
    """Forward pass in fp64.

    q1, q2: [B,H,Nq,d]; k1, k2: [B,H,Nk,d]; v: [B,H,Nk,dv]; all the same dtype.
    gamma: [H*dv] or None (ones).  rows: optional 1-D list of query indices
    computed for every (b,h).  Returns ``(o_pre, y)`` as float64 arrays of
    shape [B,H,R,dv] (R = Nq, or len(rows)): the pre-norm differential
    attention output and the GroupNorm-ed, (1 - lambda_init)-scaled output.
    """
    arrs = [_as_input(t) for t in (q1, k1, q2, k2, v)]
    types = {t for _, t in arrs}
    if len(types) != 1:
        raise TypeError("q1,k1,q2,k2,v must share one dtype")
    (aq1, ak1, aq2, ak2, av), in_type = [a for a, _ in arrs], types.pop()
    B, H, Nq, d = aq1.shape
    Nk, dv = ak1.shape[2], av.shape[3]
    g = _gamma_array(gamma, H, dv)
    r = None
    R = Nq
    if rows is not None:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        R = r.size
    o_pre = np.empty((B, H, R, dv), np.float64)
    y = np.empty((B, H, R, dv), np.float64)
    rc = _load().oracle_diffattn_fwd(
        _ptr(aq1), _ptr(ak1), _ptr(aq2), _ptr(ak2), _ptr(av), in_type,
        float(lam), float(lam_init), int(bool(causal)), B, H, Nq, Nk, d, dv,
        _ptr(g), float(eps), _ptr(r), R, _ptr(o_pre), _ptr(y), int(threads))
    if rc != 0:
        raise ValueError("oracle_diffattn_fwd rejected its arguments")
    return o_pre, y


def _gamma_array(gamma, H, dv):
    if gamma is None:
        return None
    g = np.ascontiguousarray(np.asarray(gamma.cpu() if hasattr(gamma, "cpu") else gamma,
                                        dtype=np.float64).reshape(-1))
    if g.size != H * dv:
        raise ValueError("gamma must have H*dv entries")
    return g


def diffattn_bwd(q1, k1, q2, k2, v, dy, lam, lam_init, causal=False, gamma=None, eps=1e-5,
                 rows=None, keys=None, threads=0):
    """Backward pass in fp64: gradients of ``sum(dy * y)``.

    Inputs as for ``diffattn_fwd``; dy is [B,H,Nq,dv] (any accepted dtype).
    ``rows`` / ``keys`` optionally restrict the query rows whose dq and the
    keys whose dk, dv are computed (the same indices for every (b,h)).
    Returns a dict of float64 arrays: dq1, dq2 [B,H,R,d]; dk1, dk2 [B,H,K,d];
    dv [B,H,K,dv]; and, only when neither rows nor keys is given, dlambda
    (a float), dlambda_rss (the root-sum-square of dlambda's per-row terms,
    the scale of its rounding error) and dgamma [H*dv].
    """
    arrs = [_as_input(t) for t in (q1, k1, q2, k2, v)]
    types = {t for _, t in arrs}
    if len(types) != 1:
        raise TypeError("q1,k1,q2,k2,v must share one dtype")
    (aq1, ak1, aq2, ak2, av), in_type = [a for a, _ in arrs], types.pop()
    ady, dy_type = _as_input(dy)
    B, H, Nq, d = aq1.shape
    Nk, dv = ak1.shape[2], av.shape[3]
    if ady.shape != (B, H, Nq, dv):
        raise ValueError("dy must be [B,H,Nq,dv]")
    g = _gamma_array(gamma, H, dv)
    r = k = None
    R, K = Nq, Nk
    if rows is not None:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        R = r.size
    if keys is not None:
        k = np.ascontiguousarray(np.asarray(keys, dtype=np.int64).reshape(-1))
        K = k.size
    full = rows is None and keys is None
    out = {"dq1": np.empty((B, H, R, d)), "dq2": np.empty((B, H, R, d)), "dk1": np.empty((B, H, K, d)),
           "dk2": np.empty((B, H, K, d)), "dv": np.empty((B, H, K, dv))}
    dlam = np.zeros(1) if full else None
    dlam_rss = np.zeros(1) if full else None
    dgam = np.empty(H * dv) if full else None
    rc = _load().oracle_diffattn_bwd(
        _ptr(aq1), _ptr(ak1), _ptr(aq2), _ptr(ak2), _ptr(av), in_type, _ptr(ady), dy_type,
        float(lam), float(lam_init), int(bool(causal)), B, H, Nq, Nk, d, dv, _ptr(g), float(eps),
        _ptr(r), R, _ptr(k), K, _ptr(out["dq1"]), _ptr(out["dq2"]), _ptr(out["dk1"]), _ptr(out["dk2"]),
        _ptr(out["dv"]), _ptr(dlam), _ptr(dgam), _ptr(dlam_rss), int(threads))
    if rc != 0:
        raise ValueError("oracle_diffattn_bwd rejected its arguments")
    if full:
        out["dlambda"] = float(dlam[0])
        out["dlambda_rss"] = float(dlam_rss[0])
        out["dgamma"] = dgam
    return out


def diffattn_maps(q1, k1, q2, k2, causal=False):
    """The two attention maps A1, A2 in full, [B,H,Nq,Nk] fp64 (masked = 0)."""
    arrs = [_as_input(t) for t in (q1, k1, q2, k2)]
    types = {t for _, t in arrs}
    if len(types) != 1:
        raise TypeError("q1,k1,q2,k2 must share one dtype")
    (aq1, ak1, aq2, ak2), in_type = [a for a, _ in arrs], types.pop()
    B, H, Nq, d = aq1.shape
    Nk = ak1.shape[2]
    a1 = np.empty((B, H, Nq, Nk), np.float64)
    a2 = np.empty((B, H, Nq, Nk), np.float64)
    rc = _load().oracle_diffattn_maps(_ptr(aq1), _ptr(ak1), _ptr(aq2), _ptr(ak2), in_type,
                                      int(bool(causal)), B, H, Nq, Nk, d, _ptr(a1), _ptr(a2))
    if rc != 0:
        raise ValueError("oracle_diffattn_maps rejected its arguments")
    return a1, a2


def timed_fwd(*args, **kwargs):
    """``diffattn_fwd`` plus its wall time in seconds (for the CPU baseline)."""
    t0 = time.perf_counter()
    out = diffattn_fwd(*args, **kwargs)
    return out, time.perf_counter() - t0
