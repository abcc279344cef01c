"""Host-side checks of the C ABI: the library builds, loads and exports every
symbol include/gpt2.h declares, and its host logic (sizes, validation, status
strings) behaves.  No GPU work is launched here."""
import ctypes as ct
import os
import re

import numpy as np
import pytest

from pretraining_step_train_b300 import binding, build
from oracle import gpt2_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gpt2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_header_declares_boundary_calls():
    names = declared_functions()
    for must in ("gpt2_create", "gpt2_forward", "gpt2_backward", "gpt2_clip_adamw", "attn_fwd",
                 "attn_bwd", "classifier_fwd_bwd"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in binding.SIGNATURES, name


def test_num_params_matches_oracle(lib):
    for (L, C, Vpad, T) in [(12, 768, 50304, 1024), (24, 1024, 50304, 1024), (48, 1600, 50304, 1024),
                            (4, 64, 256, 64), (0, 16, 48, 8)]:
        assert lib.gpt2_num_params(L, C, Vpad, T) == O.num_params(L, C, Vpad, T)


def test_arena_bytes_and_validation(lib):
    ok = lib.gpt2_arena_bytes(12, 12, 768, 50257, 50304, 1024, 16, binding.GPT2_BF16)
    assert ok > 0
    # params+grads bf16 and master/m/v fp32: at least 16 bytes per parameter
    assert ok > 16 * O.num_params(12, 768, 50304, 1024)
    assert ok < 60e9  # the 124M step at B=16 fits comfortably in one B300
    assert lib.gpt2_arena_bytes(4, 4, 64, 256, 256, 64, 4, binding.GPT2_FP32) > 0
    bad = [
        (12, 5, 768, 50257, 50304, 1024, 16, 1),   # C % H
        (12, 12, 768, 50257, 50000, 1024, 16, 1),  # Vpad < V
        (12, 12, 768, 50257, 50308, 1024, 16, 9),  # precision
        (12, 12, 768, 50257, 50304, 1024, 17, 1),  # B*T > 16384
        (12, 8, 768, 50257, 50304, 1024, 16, 1),   # bf16 needs head size 64
    ]
    for args in bad:
        assert lib.gpt2_arena_bytes(*args) == 0, args


def test_create_rejects_bad_arguments_on_host(lib):
    h = ct.c_void_p()
    n = lib.gpt2_arena_bytes(4, 4, 64, 256, 256, 64, 4, binding.GPT2_FP32)
    assert lib.gpt2_create(4, 4, 64, 256, 256, 64, 4, 0, None, n, None, ct.byref(h)) == binding.GPT2_E_INVAL
    assert lib.gpt2_create(4, 4, 64, 256, 256, 64, 4, 0, 256 * 7 + 1, n, None, ct.byref(h)) == binding.GPT2_E_INVAL
    assert lib.gpt2_create(4, 4, 64, 256, 256, 64, 4, 0, 4096, n - 1, None, ct.byref(h)) == binding.GPT2_E_INVAL
    assert lib.gpt2_create(4, 3, 64, 256, 256, 64, 4, 0, 4096, n, None, ct.byref(h)) == binding.GPT2_E_INVAL
    assert lib.gpt2_backward(None) == binding.GPT2_E_INVAL
    assert lib.gpt2_forward(None, None, None, None) == binding.GPT2_E_INVAL


def test_standalone_entry_points_validate_on_host(lib):
    assert lib.attn_fwd(None, None, None, None, None, 1, 1, 64, 64, 0, 0, 0, 0, 0, 0, 0.125, None) == binding.GPT2_E_INVAL
    assert lib.attn_fwd(16, 16, 16, 16, 16, 1, 1, 64, 32, 0, 0, 0, 0, 0, 0, 0.125, None) == binding.GPT2_E_UNSUPPORTED
    assert lib.classifier_fwd_bwd(None, None, None, 1, 8, 8, 8, None, None, None, None, 0, None) == binding.GPT2_E_INVAL
    assert lib.gemm_bf16(16, 16, 16, 64, 12, 64, 64, 64, 64, 0, 0, 0, 1, None, 0, None) == binding.GPT2_E_INVAL  # N % 8
    assert lib.attn_workspace_bytes(16, 12, 1024) == 16 * 12 * 1024 * 4
    assert lib.classifier_workspace_bytes(16384, 768, 50304) >= 16384 * 50304 * 2


def test_strerror(lib):
    for s in range(-7, 1):
        assert lib.gpt2_strerror(s)
    assert binding.GPT2Error(binding.GPT2_E_STATE, "x").status == binding.GPT2_E_STATE


def test_gemm_and_step_extensions_validate_on_host(lib):
    """The stream-K / epilogue GEMM entry points and the accumulation calls refuse
    bad arguments before any device work."""
    # splits -1 / -2 need a 16-byte aligned workspace of the stated size
    need = lib.gemm_bf16_sk_workspace_bytes()
    assert need > 0
    assert lib.gemm_bf16(16, 16, 16, 64, 64, 64, 64, 64, 64, 0, 0, 0, -1, None, need, None) == binding.GPT2_E_INVAL
    assert lib.gemm_bf16(16, 16, 16, 64, 64, 64, 64, 64, 64, 0, 0, 0, -1, 4096, need - 1, None) == binding.GPT2_E_INVAL
    assert lib.gemm_bf16(16, 16, 16, 64, 64, 64, 64, 64, 64, 0, 0, 0, -3, 4096, need, None) == binding.GPT2_E_INVAL
    # fused-epilogue entry: epilogue code, operands of the epilogue, splits range
    args = dict(A=16, B=16, D=16, D2=16, bias=16, X=16, col=None, M=64, N=64, K=64, lda=64, ldb=64, ldd=64)
    def epi(e, splits=1, **kw):
        a = dict(args, **kw)
        return lib.gemm_bf16_epilogue(a["A"], a["B"], a["D"], a["D2"], a["bias"], a["X"], a["col"], a["M"], a["N"],
                                      a["K"], a["lda"], a["ldb"], a["ldd"], 0, 0, e, splits, None, 0, None)
    assert epi(0) == binding.GPT2_E_INVAL      # 0 is not a fused epilogue
    assert epi(5) == binding.GPT2_E_INVAL
    assert epi(1, bias=None) == binding.GPT2_E_INVAL
    assert epi(2, X=None) == binding.GPT2_E_INVAL
    assert epi(3, D2=None) == binding.GPT2_E_INVAL
    assert epi(1, splits=2) == binding.GPT2_E_INVAL   # no K splits with a fused epilogue
    assert epi(1, splits=-1) == binding.GPT2_E_INVAL  # stream-K without a workspace
    assert lib.gpt2_grad_accumulate(None, 1, 0.5) == binding.GPT2_E_INVAL
    assert lib.gpt2_clip_adamw_accumulated(None, 6e-4, 0.9, 0.95, 1e-8, 0.1, 1.0, 1, None) == binding.GPT2_E_INVAL


def test_recompute_arena_savings(lib):
    """Activation recompute: level 1 keeps one gelu(h) buffer instead of L, level 2
    also keeps one LayerNorm output buffer instead of 2L; invalid levels are refused."""
    for (L, H, C, V, Vpad, T, B, prec) in [(12, 12, 768, 50257, 50304, 1024, 16, binding.GPT2_BF16),
                                           (4, 4, 64, 256, 256, 64, 4, binding.GPT2_FP32),
                                           (48, 25, 1600, 50257, 50304, 1024, 16, binding.GPT2_BF16)]:
        E = 2 if prec == binding.GPT2_BF16 else 4
        M = B * T
        r0, r1, r2 = (lib.gpt2_arena_bytes_r(L, H, C, V, Vpad, T, B, prec, r) for r in (0, 1, 2))
        assert r0 == lib.gpt2_arena_bytes(L, H, C, V, Vpad, T, B, prec)
        assert r0 - r1 == (L - 1) * M * 4 * C * E
        assert r1 - r2 == (2 * L - 1) * M * C * E
    assert lib.gpt2_arena_bytes_r(2, 2, 64, 256, 256, 64, 2, binding.GPT2_BF16, 3) == 0
    assert lib.gpt2_arena_bytes_r(2, 2, 64, 256, 256, 64, 2, binding.GPT2_BF16, -1) == 0
