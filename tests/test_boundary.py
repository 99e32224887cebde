"""C-ABI boundary checks that need no GPU: the library loads, exports every
entry point include/diffattn.h declares, and rejects bad arguments on the host
before any CUDA call (so these run on a machine without a device)."""
import ctypes
import os
import re

import pytest

import transformer_attention_07_b300 as da
from transformer_attention_07_b300 import build as dabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "diffattn.h")

OK, INVALID, UNSUPPORTED, CUDA, WORKSPACE, TIMEOUT = range(6)
FAKE = ctypes.c_void_p(0x10000)       # 16-byte aligned, never dereferenced on error paths
MISALIGNED = ctypes.c_void_p(0x10008)


@pytest.fixture(scope="module")
def lib():
    dabuild.build()
    return da.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(diffattn_\w+)\s*\(", text, re.M)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted([
        "diffattn_fwd", "diffattn_fwd_ex", "diffattn_fwd_host", "diffattn_fwd_host_workspace_bytes", "diffattn_fwd_fp8",
        "diffattn_fwd_train", "diffattn_bwd_workspace_bytes", "diffattn_bwd",
        "diffattn_decode_workspace_bytes", "diffattn_decode_auto_splits", "diffattn_prefill_plan", "diffattn_decode", "diffattn_decode_partials_bytes",
        "diffattn_decode_partials", "diffattn_decode_merge",
        "diffattn_decode_noalloc", "diffattn_decode_paged", "diffattn_standard_fwd", "diffattn_status_string",
        "diffattn_last_device_error", "diffattn_selftest_wait_timeout"])


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_is_built_for_sm103a_only():
    assert "arch=compute_103a,code=sm_103a" in " ".join(dabuild.FLAGS)


def fwd(lib, q=FAKE, out=FAKE, lam=0.5, lam_init=0.8, causal=0, B=1, H=1, Nq=4, Nk=4, d=64, dv=128,
        gamma=None, eps=1e-5, pre=None):
    return lib.diffattn_fwd_ex(q, q, q, q, q, lam, lam_init, causal, B, H, Nq, Nk, d, dv, gamma, eps, out, pre,
                               None)


def test_fwd_validation(lib):
    assert fwd(lib, q=None) == INVALID
    assert fwd(lib, out=None) == INVALID
    assert fwd(lib, B=-1) == INVALID
    assert fwd(lib, Nk=0) == INVALID
    assert fwd(lib, causal=2) == INVALID
    assert fwd(lib, causal=1, Nq=5, Nk=4) == INVALID
    assert fwd(lib, eps=-1.0) == INVALID
    assert fwd(lib, eps=float("nan")) == INVALID
    assert fwd(lib, lam=float("inf")) == INVALID
    assert fwd(lib, lam_init=float("nan")) == INVALID
    assert fwd(lib, d=128, dv=128) == UNSUPPORTED
    assert fwd(lib, d=64, dv=64) == UNSUPPORTED
    assert fwd(lib, q=MISALIGNED) == INVALID
    assert fwd(lib, pre=MISALIGNED) == INVALID
    assert fwd(lib, gamma=ctypes.c_void_p(0x10002)) == INVALID
    assert fwd(lib, H=70000) == INVALID


def test_fwd_empty_problems_return_ok_without_launch(lib):
    assert fwd(lib, B=0) == OK
    assert fwd(lib, H=0) == OK
    assert fwd(lib, Nq=0) == OK
    assert fwd(lib, Nq=0, causal=1) == OK


def test_fwd_host_validation(lib):
    hb = lib.diffattn_fwd_host_workspace_bytes
    # three slots of (q1, q2, k1, k2, v, out) for a chunk of heads, each tensor 256-byte aligned
    slot = lambda c, Nq, Nk, d, dv: sum((x + 255) // 256 * 256 for x in
                                        (c * Nq * d * 2, c * Nq * d * 2, c * Nk * d * 2, c * Nk * d * 2,
                                         c * Nk * dv * 2, c * Nq * dv * 2))
    assert hb(1, 16, 100, 100, 64, 128, 0) == 3 * slot(1, 100, 100, 64, 128)      # auto: 16 heads / 16 chunks
    assert hb(4, 16, 100, 100, 64, 128, 0) == 3 * slot(4, 100, 100, 64, 128)      # 64 heads / 16 chunks
    assert hb(2, 3, 64, 96, 32, 64, 5) == 3 * slot(3, 64, 96, 32, 64)             # capped at H
    assert hb(1, 0, 64, 64, 64, 128, 0) == 0
    fh = lambda q=FAKE, out=FAKE, ws=ctypes.c_void_p(0x10000), wsb=1 << 30, d=64, dv=128, chunk=0, B=1: \
        lib.diffattn_fwd_host(q, q, q, q, q, 0.5, 0.8, 0, B, 2, 64, 64, d, dv, None, 1e-5, out, chunk, ws, wsb, None)
    assert fh(q=None) == INVALID
    assert fh(out=None) == INVALID
    assert fh(chunk=-1) == INVALID
    assert fh(d=64, dv=64) == UNSUPPORTED
    assert fh(ws=None) == WORKSPACE
    assert fh(wsb=1024) == WORKSPACE
    assert fh(ws=ctypes.c_void_p(0x10010)) == INVALID
    assert fh(B=0) == OK


def test_fwd_fp8_validation(lib):
    f8 = lambda q=FAKE, sc=FAKE, d=64, dv=128, B=1, causal=0, Nq=4: lib.diffattn_fwd_fp8(
        q, q, q, q, FAKE, sc, 0.5, 0.8, causal, B, 1, Nq, 4, d, dv, None, 1e-5, FAKE, None, None)
    assert f8(sc=None) == INVALID
    assert f8(q=None) == INVALID
    assert f8(sc=ctypes.c_void_p(0x10002)) == INVALID
    assert f8(q=MISALIGNED) == INVALID
    assert f8(causal=1, Nq=5) == INVALID
    assert f8(d=64, dv=64) == UNSUPPORTED
    assert f8(B=0) == OK


def test_fwd_train_validation(lib):
    tr = lambda o2=FAKE, lse=FAKE, pre=FAKE, d=64, dv=128, B=1: lib.diffattn_fwd_train(
        FAKE, FAKE, FAKE, FAKE, FAKE, 0.5, 0.8, 0, B, 1, 4, 4, d, dv, None, 1e-5, FAKE, pre, o2, lse, None)
    assert tr(o2=None) == INVALID
    assert tr(lse=None) == INVALID
    assert tr(pre=None) == INVALID
    assert tr(o2=MISALIGNED) == INVALID
    assert tr(lse=ctypes.c_void_p(0x10002)) == INVALID
    assert tr(d=64, dv=64) == UNSUPPORTED
    assert tr(B=0) == OK


def test_bwd_workspace_bytes(lib):
    ws = lib.diffattn_bwd_workspace_bytes
    align = lambda x: (x + 255) // 256 * 256
    # do (bf16) + per-row constants in two layouts (Nq rounded up to 128) + partial sums per 64 rows
    B, H, Nq, dv = 2, 3, 200, 128
    pad = 256
    assert ws(B, H, Nq, dv) == (align(B * H * Nq * dv * 2) + 2 * align(B * H * pad * 16) +
                                align(B * H * (pad // 64) * dv * 4) + align(B * H * (pad // 64) * 4))
    assert ws(-1, 1, 1, 128) == 0


def test_bwd_validation(lib):
    def bwd(q=FAKE, d=64, dv=128, causal=0, Nq=4, Nk=4, ws=ctypes.c_void_p(0x10000), ws_bytes=1 << 20, dl=None,
            grad=FAKE, B=1):
        return lib.diffattn_bwd(q, q, q, q, q, q, q, q, q, 0.5, 0.8, causal, B, 1, Nq, Nk, d, dv, None, 1e-5,
                                grad, grad, grad, grad, grad, dl, None, ws, ws_bytes, None)
    assert bwd(q=None) == INVALID
    assert bwd(grad=None) == INVALID
    assert bwd(Nk=0) == INVALID
    assert bwd(causal=1, Nq=5, Nk=4) == INVALID
    assert bwd(d=32, dv=128) == UNSUPPORTED
    assert bwd(q=MISALIGNED) == INVALID
    assert bwd(dl=ctypes.c_void_p(0x10002)) == INVALID
    assert bwd(ws=None) == WORKSPACE
    assert bwd(ws_bytes=16) == WORKSPACE
    assert bwd(ws=ctypes.c_void_p(0x10010)) == INVALID     # not 256-byte aligned
    assert bwd(B=0) == OK


def test_standard_fwd_validation(lib):
    std = lambda q=FAKE, causal=0, Nq=4, Nk=4, d=128, dv=128, out=FAKE, f32=None: lib.diffattn_standard_fwd(
        q, q, q, causal, 1, 1, Nq, Nk, d, dv, out, f32, None)
    assert std(q=None) == INVALID
    assert std(out=None) == INVALID
    assert std(Nk=0) == INVALID
    assert std(causal=1, Nq=5, Nk=4) == INVALID
    assert std(d=64, dv=128) == UNSUPPORTED
    assert std(q=MISALIGNED) == INVALID
    assert std(f32=MISALIGNED) == INVALID
    assert std(Nq=0) == OK


def test_decode_paged_validation(lib):
    def pg(q=FAKE, table=FAKE, lens=FAKE, max_pages=4, page_size=64, num_pages=8, B=1, d=64, dv=128, splits=1,
           ws=FAKE, ws_bytes=1 << 20):
        return lib.diffattn_decode_paged(q, q, q, q, q, table, lens, max_pages, page_size, num_pages, 0.5, 0.8, B, 1,
                                         d, dv, None, 1e-5, splits, ws, ws_bytes, FAKE, None, None)
    assert pg(table=None) == INVALID
    assert pg(lens=None) == INVALID
    assert pg(page_size=48) == INVALID          # not a multiple of 32
    assert pg(page_size=0) == INVALID
    assert pg(max_pages=0) == INVALID
    assert pg(num_pages=0) == INVALID
    assert pg(d=32, dv=128) == UNSUPPORTED
    assert pg(table=ctypes.c_void_p(0x10002)) == INVALID
    assert pg(ws=None) == WORKSPACE
    assert pg(max_pages=2048, page_size=32, splits=1) == INVALID   # one range would span > 1024 pages
    assert pg(B=0) == OK


def test_decode_partials_and_merge_validation(lib):
    assert lib.diffattn_decode_partials_bytes(2, 3, 128, 4) == 2 * 3 * 4 * 2 * (128 + 4) * 4
    assert lib.diffattn_decode_partials_bytes(2, 3, 128, 0) == 0
    dp = lambda q=FAKE, splits=2, d=64, dv=128, buf=FAKE, nb=1 << 20, B=1: lib.diffattn_decode_partials(
        q, q, q, q, q, B, 2, 64, d, dv, splits, buf, nb, None)
    assert dp(q=None) == INVALID
    assert dp(splits=0) == INVALID
    assert dp(splits=65) == INVALID
    assert dp(d=32, dv=128) == UNSUPPORTED
    assert dp(buf=None) == WORKSPACE
    assert dp(nb=64) == WORKSPACE
    assert dp(buf=ctypes.c_void_p(0x10004)) == INVALID
    assert dp(B=0) == OK
    dm = lambda parts=2, splits=2, dv=128, out=FAKE, B=1, lam=0.5: lib.diffattn_decode_merge(
        FAKE, parts, B, 2, dv, splits, lam, 0.8, None, 1e-5, out, None, None)
    assert dm(parts=0) == INVALID
    assert dm(parts=100, splits=64) == INVALID     # more than 4096 partial states per head
    assert dm(out=None) == INVALID
    assert dm(dv=96) == UNSUPPORTED
    assert dm(lam=float("nan")) == INVALID
    assert dm(B=0) == OK


def test_decode_workspace_bytes(lib):
    ws = lib.diffattn_decode_workspace_bytes
    assert ws(32, 32, 32768, 128, 4) == 32 * 32 * 4 * 2 * (128 + 4) * 4
    assert ws(2, 3, 100, 64, 0) == 2 * 3 * 32 * 2 * (64 + 4) * 4
    assert ws(-1, 1, 1, 64, 0) == 0
    assert ws(1, 1, 0, 64, 0) == 0
    assert ws(1, 1, 10, 64, 65) == 0


def dec(lib, q=FAKE, ws=FAKE, ws_bytes=1 << 20, splits=1, B=1, H=1, Nk=64, d=64, dv=128, out=FAKE, eps=1e-5):
    return lib.diffattn_decode(q, q, q, q, q, 0.5, 0.8, B, H, Nk, d, dv, None, eps, splits, ws, ws_bytes, out,
                               None, None)


def test_decode_validation(lib):
    assert dec(lib, q=None) == INVALID
    assert dec(lib, out=None) == INVALID
    assert dec(lib, Nk=0) == INVALID
    assert dec(lib, splits=-1) == INVALID
    assert dec(lib, splits=65) == INVALID
    assert dec(lib, eps=-1.0) == INVALID
    assert dec(lib, d=32, dv=128) == UNSUPPORTED
    assert dec(lib, q=MISALIGNED) == INVALID
    assert dec(lib, ws=None) == WORKSPACE
    assert dec(lib, ws_bytes=16) == WORKSPACE
    assert dec(lib, ws=ctypes.c_void_p(0x10004)) == INVALID
    assert dec(lib, B=1 << 10, H=1 << 10, Nk=1 << 12) == INVALID   # > 2^31 cache rows
    assert dec(lib, B=0) == OK


def test_status_strings(lib):
    for s in range(6):
        assert da.status_string(s)
    assert da.status_string(99) == "unknown status"


def test_binding_raises_without_cuda_tensors():
    import torch
    x = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        da.fwd(x, x, x, x, torch.zeros(1, 1, 4, 128, dtype=torch.bfloat16), 0.5, 0.8)


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "transformer_attention_07_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "oracle.cpp" not in text and "liboracle" not in text, f
