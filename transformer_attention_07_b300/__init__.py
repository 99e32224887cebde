"""B300 (sm_103a) differential-attention forward: Python binding of libdiffattn.so.

The functions here marshal torch CUDA tensors into the C ABI declared in
``include/diffattn.h`` (pointers, sizes, the current stream) and do no
arithmetic: every step of the forward pass runs in the library's kernels.
If the shared library has not been built, every call raises; there is no
fallback implementation.

What the library computes (Differential Transformer pages — the DiffAttn
formula of the iloveeagents.com Q&A, "Mathematical Formula", and steps 2-4 of
llmbytes.dev "How Differential Attention Cancels Common-Mode Noise"):

    y = (1 - lambda_init) * GroupNorm_h( (softmax(Q1 K1^T/sqrt d) - lambda softmax(Q2 K2^T/sqrt d)) V )
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "fwd", "fwd_host", "fwd_host_workspace_bytes", "fwd_fp8", "fwd_train", "bwd", "bwd_workspace_bytes",
    "standard_fwd", "decode", "decode_paged", "decode_workspace_bytes", "decode_auto_splits", "prefill_plan", "PLAN_FORMS",
    "decode_partials", "decode_partials_bytes",
    "decode_merge", "gather_partials", "decode_sharded", "head_range", "gather_heads", "fwd_sharded",
    "status_string", "last_device_error", "selftest_wait_timeout", "load", "LIB_PATH",
    "DiffAttnError", "SUPPORTED_WIDTHS",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdiffattn.so")
SUPPORTED_WIDTHS = ((64, 128), (32, 64))

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE, ERR_TIMEOUT = range(6)

_lib = None


class DiffAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def load():
    """Load libdiffattn.so (built by ``python -m transformer_attention_07_b300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -m transformer_attention_07_b300.build` "
            "(there is no non-CUDA implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.diffattn_fwd.argtypes = [vp, vp, vp, vp, vp, f32, f32, i32, i32, i32, i32, i32, i32, i32, vp, f32, vp, vp]
    lib.diffattn_fwd.restype = i32
    lib.diffattn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, f32, f32, i32, i32, i32, i32, i32, i32, i32, vp, f32,
                                    vp, vp, vp]
    lib.diffattn_fwd_ex.restype = i32
    lib.diffattn_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.diffattn_decode_workspace_bytes.restype = sz
    lib.diffattn_decode_auto_splits.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.diffattn_decode_auto_splits.restype = i32
    lib.diffattn_prefill_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int),
                                          ctypes.POINTER(ctypes.c_longlong)]
    lib.diffattn_prefill_plan.restype = i32
    lib.diffattn_decode.argtypes = [vp, vp, vp, vp, vp, f32, f32, i32, i32, i32, i32, i32, vp, f32, i32, vp, sz,
                                    vp, vp, vp]
    lib.diffattn_decode.restype = i32
    lib.diffattn_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, f32, f32, i32, i32, i32, i32,
                                          vp, f32, i32, vp, sz, vp, vp, vp]
    lib.diffattn_decode_paged.restype = i32
    lib.diffattn_fwd_host_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.diffattn_fwd_host_workspace_bytes.restype = sz
    lib.diffattn_fwd_host.argtypes = [vp, vp, vp, vp, vp, f32, f32, i32, i32, i32, i32, i32, i32, i32, vp, f32, vp,
                                      i32, vp, sz, vp]
    lib.diffattn_fwd_host.restype = i32
    lib.diffattn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, f32, f32, i32, i32, i32, i32, i32, i32, i32, vp, f32,
                                     vp, vp, vp]
    lib.diffattn_fwd_fp8.restype = i32
    lib.diffattn_fwd_train.argtypes = [vp, vp, vp, vp, vp, f32, f32, i32, i32, i32, i32, i32, i32, i32, vp, f32,
                                       vp, vp, vp, vp, vp]
    lib.diffattn_fwd_train.restype = i32
    lib.diffattn_bwd_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.diffattn_bwd_workspace_bytes.restype = sz
    lib.diffattn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, f32, i32, i32, i32, i32, i32, i32, i32,
                                 vp, f32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.diffattn_bwd.restype = i32
    lib.diffattn_decode_partials_bytes.argtypes = [i32, i32, i32, i32]
    lib.diffattn_decode_partials_bytes.restype = sz
    lib.diffattn_decode_partials.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, sz, vp]
    lib.diffattn_decode_partials.restype = i32
    lib.diffattn_decode_merge.argtypes = [vp, i32, i32, i32, i32, i32, f32, f32, vp, f32, vp, vp, vp]
    lib.diffattn_decode_merge.restype = i32
    lib.diffattn_standard_fwd.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp]
    lib.diffattn_standard_fwd.restype = i32
    lib.diffattn_status_string.argtypes = [i32]
    lib.diffattn_status_string.restype = ctypes.c_char_p
    lib.diffattn_last_device_error.argtypes = [vp]
    lib.diffattn_last_device_error.restype = i32
    lib.diffattn_selftest_wait_timeout.argtypes = [vp]
    lib.diffattn_selftest_wait_timeout.restype = i32
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().diffattn_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check_bf16(name, t, ndim=4):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be a CUDA bf16 tensor")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D tensor [B,H,N,width]")


def _gamma(gamma, H, dv):
    import torch
    if gamma is None:
        return None
    if not gamma.is_cuda or gamma.dtype != torch.float32 or not gamma.is_contiguous() or gamma.numel() != H * dv:
        raise ValueError("gamma must be a contiguous CUDA float32 tensor with H*dv entries")
    return gamma


def fwd(q1, k1, q2, k2, v, lam, lam_init, causal=False, gamma=None, eps=1e-5, out=None, o_prenorm=None,
        stream=None):
    """Prefill forward.  q1,q2 [B,H,Nq,d]; k1,k2 [B,H,Nk,d]; v [B,H,Nk,dv] (CUDA bf16).

    Returns ``out`` (bf16 [B,H,Nq,dv], allocated if not given).  If
    ``o_prenorm`` (fp32 [B,H,Nq,dv]) is given, the pre-norm output is written
    there too.  Asynchronous on ``stream`` (default: torch's current stream)."""
    import torch
    for n, t in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2), ("v", v)):
        _check_bf16(n, t)
    B, H, Nq, d = q1.shape
    Nk, dv = k1.shape[2], v.shape[3]
    if out is None:
        out = torch.empty((B, H, Nq, dv), dtype=torch.bfloat16, device=q1.device)
    g = _gamma(gamma, H, dv)
    rc = load().diffattn_fwd_ex(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), float(lam), float(lam_init),
                                int(bool(causal)), B, H, Nq, Nk, d, dv, _ptr(g), float(eps), _ptr(out),
                                _ptr(o_prenorm), _stream(stream))
    if rc != OK:
        raise DiffAttnError(rc, "diffattn_fwd")
    return out


def fwd_host_workspace_bytes(B, H, Nq, Nk, d, dv, heads_per_chunk=0) -> int:
    return int(load().diffattn_fwd_host_workspace_bytes(B, H, Nq, Nk, d, dv, heads_per_chunk))


def fwd_host(q1, k1, q2, k2, v, lam, lam_init, causal=False, gamma=None, eps=1e-5, out=None, heads_per_chunk=0,
             workspace=None, stream=None, device=None):
    """Prefill with host-resident tensors: q1,q2 [B,H,Nq,d], k1,k2 [B,H,Nk,d],
    v [B,H,Nk,dv] are CPU bf16 tensors (page-locked for overlapped copies);
    returns ``out`` (CPU bf16 [B,H,Nq,dv]).  The library copies chunks of heads
    in, runs the kernel and copies the results out on its own streams.  The
    call is asynchronous: ``out`` is complete once ``stream`` (default: torch's
    current stream) has completed.  ``gamma`` is a CUDA tensor, as elsewhere."""
    import torch
    for n, t in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.bfloat16:
            raise TypeError(f"{n} must be a CPU bf16 tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous 4-D tensor [B,H,N,width]")
    B, H, Nq, d = q1.shape
    Nk, dv = k1.shape[2], v.shape[3]
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    if out is None:
        out = torch.empty((B, H, Nq, dv), dtype=torch.bfloat16).pin_memory()
    if workspace is None:
        workspace = torch.empty(max(fwd_host_workspace_bytes(B, H, Nq, Nk, d, dv, heads_per_chunk), 256),
                                dtype=torch.uint8, device=dev)
    g = _gamma(gamma, H, dv)
    rc = load().diffattn_fwd_host(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), float(lam), float(lam_init),
                                  int(bool(causal)), B, H, Nq, Nk, d, dv, _ptr(g), float(eps), _ptr(out),
                                  int(heads_per_chunk), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream))
    if rc != OK:
        raise DiffAttnError(rc, "diffattn_fwd_host")
    return out


def fwd_fp8(q1, k1, q2, k2, v, qk_scale, lam, lam_init, causal=False, gamma=None, eps=1e-5, out=None,
            o_prenorm=None, stream=None):
    """Prefill forward with fp8 (e4m3) queries and keys.  q1, q2 [B,H,Nq,d] and
    k1, k2 [B,H,Nk,d] are CUDA ``torch.float8_e4m3fn`` tensors; qk_scale is a
    CUDA float32 tensor of 4*H per-head dequantisation scales (rows q1, k1,
    q2, k2); v is bf16.  Returns out (bf16 [B,H,Nq,dv])."""
    import torch
    for n, t in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float8_e4m3fn:
            raise TypeError(f"{n} must be a CUDA float8_e4m3fn tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous 4-D tensor [B,H,N,d]")
    _check_bf16("v", v)
    B, H, Nq, d = q1.shape
    Nk, dv = k1.shape[2], v.shape[3]
    if (not qk_scale.is_cuda or qk_scale.dtype != torch.float32 or not qk_scale.is_contiguous()
            or qk_scale.numel() != 4 * H):
        raise ValueError("qk_scale must be a contiguous CUDA float32 tensor with 4*H entries")
    if out is None:
        out = torch.empty((B, H, Nq, dv), dtype=torch.bfloat16, device=q1.device)
    g = _gamma(gamma, H, dv)
    rc = load().diffattn_fwd_fp8(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), _ptr(qk_scale), float(lam),
                                 float(lam_init), int(bool(causal)), B, H, Nq, Nk, d, dv, _ptr(g), float(eps),
                                 _ptr(out), _ptr(o_prenorm), _stream(stream))
    if rc != OK:
        raise DiffAttnError(rc, "diffattn_fwd_fp8")
    return out


def fwd_train(q1, k1, q2, k2, v, lam, lam_init, causal=False, gamma=None, eps=1e-5, out=None, stream=None):
    """Training forward: returns ``(out, saved)`` where ``saved`` holds what
    ``bwd`` reads: ``o_prenorm`` and ``o2`` (fp32 [B,H,Nq,dv]: (A1 - lambda A2) V
    and A2 V) and ``lse`` (fp32 [2,B,H,Nq]: each map's log-sum-exp)."""
    import torch
    for n, t in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2), ("v", v)):
        _check_bf16(n, t)
    B, H, Nq, d = q1.shape
    Nk, dv = k1.shape[2], v.shape[3]
    dev = q1.device
    if out is None:
        out = torch.empty((B, H, Nq, dv), dtype=torch.bfloat16, device=dev)
    saved = {"o_prenorm": torch.empty((B, H, Nq, dv), dtype=torch.float32, device=dev),
             "o2": torch.empty((B, H, Nq, dv), dtype=torch.float32, device=dev),
             "lse": torch.empty((2, B, H, Nq), dtype=torch.float32, device=dev)}
    g = _gamma(gamma, H, dv)
    rc = load().diffattn_fwd_train(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), float(lam), float(lam_init),
                                   int(bool(causal)), B, H, Nq, Nk, d, dv, _ptr(g), float(eps), _ptr(out),
                                   _ptr(saved["o_prenorm"]), _ptr(saved["o2"]), _ptr(saved["lse"]), _stream(stream))
    if rc != OK:
        raise DiffAttnError(rc, "diffattn_fwd_train")
    return out, saved


def bwd_workspace_bytes(B, H, Nq, dv) -> int:
    return int(load().diffattn_bwd_workspace_bytes(B, H, Nq, dv))


def bwd(q1, k1, q2, k2, v, dy, saved, lam, lam_init, causal=False, gamma=None, eps=1e-5, workspace=None,
        grads=None, stream=None):
    """Backward pass.  ``saved`` is the dict ``fwd_train`` returned for these
    inputs; dy is the bf16 gradient of the output.  Returns a dict with dq1,
    dk1, dq2, dk2, dv (bf16, the inputs' shapes), dlambda (fp32 [1]) and
    dgamma (fp32 [H*dv]); ``grads`` may supply those tensors."""
    import torch
    for n, t in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2), ("v", v), ("dy", dy)):
        _check_bf16(n, t)
    B, H, Nq, d = q1.shape
    Nk, dv = k1.shape[2], v.shape[3]
    dev = q1.device
    if grads is None:
        grads = {"dq1": torch.empty_like(q1), "dk1": torch.empty_like(k1), "dq2": torch.empty_like(q2),
                 "dk2": torch.empty_like(k2), "dv": torch.empty_like(v),
                 "dlambda": torch.empty(1, dtype=torch.float32, device=dev),
                 "dgamma": torch.empty(H * dv, dtype=torch.float32, device=dev)}
    nbytes = bwd_workspace_bytes(B, H, Nq, dv)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    g = _gamma(gamma, H, dv)
    rc = load().diffattn_bwd(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), _ptr(dy), _ptr(saved["o_prenorm"]),
                             _ptr(saved["o2"]), _ptr(saved["lse"]), float(lam), float(lam_init), int(bool(causal)),
                             B, H, Nq, Nk, d, dv, _ptr(g), float(eps), _ptr(grads["dq1"]), _ptr(grads["dk1"]),
                             _ptr(grads["dq2"]), _ptr(grads["dk2"]), _ptr(grads["dv"]), _ptr(grads.get("dlambda")),
                             _ptr(grads.get("dgamma")), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != OK:
        raise DiffAttnError(rc, "diffattn_bwd")
    return grads


def standard_fwd(q, k, v, causal=False, out=None, out_f32=None, stream=None):
    """Standard softmax attention (the single-map baseline), d = dv = 128.
    q [B,H,Nq,128], k [B,H,Nk,128], v [B,H,Nk,128] CUDA bf16; returns out."""
    import torch
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_bf16(n, t)
    B, H, Nq, d = q.shape
    Nk, dv = k.shape[2], v.shape[3]
    if out is None:
        out = torch.empty((B, H, Nq, dv), dtype=torch.bfloat16, device=q.device)
    rc = load().diffattn_standard_fwd(_ptr(q), _ptr(k), _ptr(v), int(bool(causal)), B, H, Nq, Nk, d, dv,
                                      _ptr(out), _ptr(out_f32), _stream(stream))
    if rc != OK:
        raise DiffAttnError(rc, "diffattn_standard_fwd")
    return out


def decode_workspace_bytes(B, H, Nk, dv, num_splits=0) -> int:
    return int(load().diffattn_decode_workspace_bytes(B, H, Nk, dv, num_splits))


PLAN_FORMS = ("tile_grid", "tile_grouped", "persistent", "persistent_weight")


def prefill_plan(B, H, Nq, Nk, d=64, dv=128, causal=True, fp8=False, sms=148):
    """How the prefill entry points launch this shape on a device with ``sms``
    SMs (host arithmetic): returns (form, ctas), form one of PLAN_FORMS."""
    form, ctas = ctypes.c_int(-1), ctypes.c_longlong(-1)
    rc = load().diffattn_prefill_plan(B, H, Nq, Nk, d, dv, int(bool(causal)), int(bool(fp8)), sms,
                                      ctypes.byref(form), ctypes.byref(ctas))
    if rc != OK:
        raise DiffAttnError(rc, "diffattn_prefill_plan")
    return PLAN_FORMS[form.value], int(ctas.value)


def decode_auto_splits(B, H, Nk, d, dv, sms, max_splits=0) -> int:
    """Key ranges per (b, h) the decode entry points use with num_splits = 0 on
    a device with ``sms`` SMs (host arithmetic; 0 for invalid arguments)."""
    return int(load().diffattn_decode_auto_splits(B, H, Nk, d, dv, sms, max_splits))


def decode(q1, k1, q2, k2, v, lam, lam_init, gamma=None, eps=1e-5, num_splits=0, workspace=None, out=None,
           o_prenorm=None, stream=None):
    """Split-KV decode: q1,q2 [B,H,1,d]; k1,k2 [B,H,Nk,d]; v [B,H,Nk,dv] (CUDA bf16).

    ``workspace`` is a CUDA tensor of at least ``decode_workspace_bytes`` bytes
    (allocated here if not given).  Returns ``out`` (bf16 [B,H,1,dv])."""
    import torch
    for n, t in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2), ("v", v)):
        _check_bf16(n, t)
    B, H, Nq, d = q1.shape
    if Nq != 1:
        raise ValueError("decode takes one query per (b, h)")
    Nk, dv = k1.shape[2], v.shape[3]
    if workspace is None:   # (a given workspace is size-checked by the library)
        nbytes = decode_workspace_bytes(B, H, Nk, dv, num_splits)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q1.device)
    if out is None:
        out = torch.empty((B, H, 1, dv), dtype=torch.bfloat16, device=q1.device)
    g = _gamma(gamma, H, dv)
    rc = load().diffattn_decode(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), float(lam), float(lam_init),
                                B, H, Nk, d, dv, _ptr(g), float(eps), int(num_splits), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _ptr(out), _ptr(o_prenorm),
                                _stream(stream))
    if rc != OK:
        raise DiffAttnError(rc, "diffattn_decode")
    return out


def decode_paged(q1, q2, k1_pages, k2_pages, v_pages, block_table, seq_lens, lam, lam_init, gamma=None, eps=1e-5,
                 num_splits=0, workspace=None, out=None, o_prenorm=None, stream=None):
    """Paged split-KV decode.  q1, q2 [B,H,1,d]; k1_pages, k2_pages
    [num_pages,H,page_size,d]; v_pages [num_pages,H,page_size,dv] (CUDA bf16);
    block_table [B,max_pages] and seq_lens [B] CUDA int32.  Returns out."""
    import torch
    for n, t in (("q1", q1), ("q2", q2), ("k1_pages", k1_pages), ("k2_pages", k2_pages), ("v_pages", v_pages)):
        _check_bf16(n, t)
    for n, t in (("block_table", block_table), ("seq_lens", seq_lens)):
        if not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
            raise TypeError(f"{n} must be a contiguous CUDA int32 tensor")
    B, H, _, d = q1.shape
    num_pages, _, page_size, _ = k1_pages.shape
    dv = v_pages.shape[3]
    max_pages = block_table.shape[1]
    nbytes = decode_workspace_bytes(B, H, max_pages * page_size, dv, num_splits)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q1.device)
    if out is None:
        out = torch.empty((B, H, 1, dv), dtype=torch.bfloat16, device=q1.device)
    g = _gamma(gamma, H, dv)
    rc = load().diffattn_decode_paged(_ptr(q1), _ptr(q2), _ptr(k1_pages), _ptr(k2_pages), _ptr(v_pages),
                                      _ptr(block_table), _ptr(seq_lens), max_pages, page_size, num_pages,
                                      float(lam), float(lam_init), B, H, d, dv, _ptr(g), float(eps), int(num_splits),
                                      _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
                                      _ptr(o_prenorm), _stream(stream))
    if rc != OK:
        raise DiffAttnError(rc, "diffattn_decode_paged")
    return out


def decode_partials_bytes(B, H, dv, num_splits) -> int:
    return int(load().diffattn_decode_partials_bytes(B, H, dv, num_splits))


def decode_partials(q1, k1, q2, k2, v, num_splits, partials=None, stream=None):
    """Partial softmax states of this GPU's key range (see include/diffattn.h):
    returns an fp32 CUDA tensor [B*H, num_splits, 2, dv + 4]."""
    import torch
    for n, t in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2), ("v", v)):
        _check_bf16(n, t)
    B, H, _, d = q1.shape
    Nk, dv = k1.shape[2], v.shape[3]
    if partials is None:
        partials = torch.empty((B * H, num_splits, 2, dv + 4), dtype=torch.float32, device=q1.device)
    rc = load().diffattn_decode_partials(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), B, H, Nk, d, dv,
                                         int(num_splits), _ptr(partials),
                                         partials.numel() * partials.element_size(), _stream(stream))
    if rc != OK:
        raise DiffAttnError(rc, "diffattn_decode_partials")
    return partials


def decode_merge(partials, B, H, lam, lam_init, gamma=None, eps=1e-5, out=None, o_prenorm=None, stream=None):
    """Merge gathered partial states [num_parts, B*H, num_splits, 2, dv + 4]
    (or one part without the leading dimension); returns out [B,H,1,dv] bf16."""
    import torch
    if partials.dim() == 4:
        partials = partials.unsqueeze(0)
    if not partials.is_cuda or partials.dtype != torch.float32 or not partials.is_contiguous():
        raise TypeError("partials must be a contiguous CUDA float32 tensor")
    parts, bh, splits, two, w = partials.shape
    dv = w - 4
    if bh != B * H or two != 2:
        raise ValueError("partials must be [num_parts, B*H, num_splits, 2, dv + 4]")
    if out is None:
        out = torch.empty((B, H, 1, dv), dtype=torch.bfloat16, device=partials.device)
    g = _gamma(gamma, H, dv)
    rc = load().diffattn_decode_merge(_ptr(partials), parts, B, H, dv, splits, float(lam), float(lam_init), _ptr(g),
                                      float(eps), _ptr(out), _ptr(o_prenorm), _stream(stream))
    if rc != OK:
        raise DiffAttnError(rc, "diffattn_decode_merge")
    return out


def _all_gather(t, group):
    """All-gather ``t`` over ``group``: [world, *t.shape] in rank order, on
    t's device.  A gloo group exchanges host copies (gloo moves host memory);
    NCCL exchanges the device tensors directly."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    src = t.contiguous()
    if src.is_cuda and dist.get_backend(group) == "gloo":
        src = src.cpu()
    chunks = [torch.empty_like(src) for _ in range(world)]
    dist.all_gather(chunks, src, group=group)
    return torch.stack(chunks).to(t.device)


def gather_partials(partials, group=None):
    """All-gather the partial states of every rank of ``group`` (torch.distributed):
    returns [world, *partials.shape], rank order, the layout decode_merge reads.
    This is the one exchange step of sequence-sharded decode."""
    return _all_gather(partials, group)


def head_range(heads, world, rank):
    """The contiguous range [lo, hi) of flattened (b, h) heads that ``rank``
    of ``world`` computes in a head-partitioned prefill: sizes differ by at
    most one, every head belongs to exactly one rank, in rank order."""
    if world < 1 or not 0 <= rank < world or heads < 0:
        raise ValueError("need world >= 1, 0 <= rank < world and heads >= 0")
    return rank * heads // world, (rank + 1) * heads // world


def fwd_sharded(q1, k1, q2, k2, v, lam, lam_init, causal=False, gamma=None, eps=1e-5, group=None, gather=False,
                stream=None):
    """Prefill with the B*H independent heads partitioned over the ranks of
    ``group``: every rank passes the full inputs (or at least its heads) and
    computes the heads ``head_range(B*H, world, rank)`` of the flattened
    [B*H, N, width] view, with no exchange.  Returns this rank's slice of
    ``out`` as [hi - lo, Nq, dv]; with ``gather=True`` the slices of every
    rank are all-gathered into the full [B, H, Nq, dv] output on every rank
    (the only collective, needed only when one GPU consumes all heads)."""
    import torch
    import torch.distributed as dist
    B, H, Nq, _ = q1.shape
    dv = v.shape[3]
    world, rank = dist.get_world_size(group), dist.get_rank(group)
    lo, hi = head_range(B * H, world, rank)
    view = lambda t: t.reshape(1, B * H, t.shape[2], t.shape[3])[:, lo:hi]
    # Each flattened head keeps its own gain slice: gamma [H*dv] repeated over B.
    g = None if gamma is None else gamma.view(1, H * dv).expand(B, H * dv).reshape(B * H, dv)[lo:hi].reshape(-1)
    out = torch.empty((1, hi - lo, Nq, dv), dtype=torch.bfloat16, device=q1.device)
    if hi > lo:
        fwd(*(view(t).contiguous() for t in (q1, k1, q2, k2, v)), lam, lam_init, causal=causal,
            gamma=None if g is None else g.contiguous(), eps=eps, out=out, stream=stream)
    if not gather:
        return out[0]
    if stream is not None:
        torch.cuda.current_stream(q1.device).wait_stream(stream)
    return gather_heads(out[0], B, H, group).view(B, H, Nq, dv)


def gather_heads(mine, B, H, group=None):
    """All-gather the head slices of a head-partitioned prefill: ``mine`` is
    this rank's [hi - lo, ...] slice (``head_range``); returns the full
    [B*H, ...] tensor on every rank, heads in order.  Slices are padded to the
    largest share for the exchange and the padding is dropped after it."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    sizes = [hi - lo for lo, hi in (head_range(B * H, world, r) for r in range(world))]
    if mine.shape[0] != sizes[dist.get_rank(group)]:
        raise ValueError("mine must hold exactly this rank's heads")
    pad = torch.zeros((max(sizes),) + tuple(mine.shape[1:]), dtype=mine.dtype, device=mine.device)
    pad[: mine.shape[0]].copy_(mine)
    every = _all_gather(pad, group)
    return torch.cat([every[r, : sizes[r]] for r in range(world)])


def decode_sharded(q1, k1, q2, k2, v, lam, lam_init, num_splits=8, gamma=None, eps=1e-5, group=None, stream=None):
    """Split-KV decode with the key cache sharded over the ranks of ``group``:
    every rank passes the same queries and its own slice of K1, K2, V; the
    ranks' partial states are all-gathered and merged on every rank."""
    B, H = q1.shape[:2]
    part = decode_partials(q1, k1, q2, k2, v, num_splits, stream=stream)
    return decode_merge(gather_partials(part, group), B, H, lam, lam_init, gamma=gamma, eps=eps, stream=stream)


def last_device_error(stream=None) -> int:
    """Read and clear the device error word (synchronises ``stream``)."""
    return int(load().diffattn_last_device_error(_stream(stream)))


def selftest_wait_timeout(stream=None) -> None:
    """Launch the diagnostic kernel whose bounded wait runs out (about 2 s);
    afterwards ``last_device_error`` returns 0x601."""
    rc = load().diffattn_selftest_wait_timeout(_stream(stream))
    if rc != OK:
        raise DiffAttnError(rc, "diffattn_selftest_wait_timeout")
