"""Thin ctypes binding of libgpt2.so (argument marshalling only).

Every function of include/gpt2.h is exposed under the same name.  All compute
happens in the library's CUDA kernels; PyTorch serves only as the device
memory and stream provider (``Step`` allocates the arena as a uint8 CUDA
tensor and passes raw pointers).  Loading fails loudly when the library has
not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes as ct
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgpt2.so")

GPT2_OK, GPT2_E_INVAL, GPT2_E_STATE, GPT2_E_TOKEN = 0, -1, -2, -3
GPT2_E_CUDA, GPT2_E_TIMEOUT, GPT2_E_NONFINITE, GPT2_E_UNSUPPORTED = -4, -5, -6, -7
GPT2_FP32, GPT2_BF16 = 0, 1
GPT2_PARAMS, GPT2_GRADS, GPT2_ADAM_M, GPT2_ADAM_V, GPT2_MASTER, GPT2_GRAD_ACC = 0, 1, 2, 3, 4, 5
KERNEL_CLASSES = ["gemm", "splitk_reduce", "attn_fwd", "attn_bwd", "layernorm_fwd", "layernorm_bwd",
                  "cross_entropy", "encoder", "bias_grad", "grad_norm", "adamw", "recompute"]

_i, _ll, _sz, _f, _p = ct.c_int, ct.c_longlong, ct.c_size_t, ct.c_float, ct.c_void_p
_fp = ct.POINTER(ct.c_float)

# name -> (restype, argtypes), in header order
SIGNATURES = {
    "gpt2_num_params": (_sz, [_i, _i, _i, _i]),
    "gpt2_arena_bytes": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "gpt2_create": (_i, [_i, _i, _i, _i, _i, _i, _i, _i, _p, _sz, _p, ct.POINTER(_p)]),
    "gpt2_destroy": (None, [_p]),
    "gpt2_arena_bytes_r": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i, _i]),
    "gpt2_create_r": (_i, [_i, _i, _i, _i, _i, _i, _i, _i, _i, _p, _sz, _p, ct.POINTER(_p)]),
    "gpt2_set_stream": (_i, [_p, _p]),
    "gpt2_set_params": (_i, [_p, _p, _i]),
    "gpt2_get_tensor": (_i, [_p, _i, _p, _i]),
    "gpt2_forward": (_i, [_p, _p, _p, _fp]),
    "gpt2_backward": (_i, [_p]),
    "gpt2_clip_adamw": (_i, [_p, _f, _f, _f, _f, _f, _f, _i, _fp]),
    "gpt2_train_step_host": (_i, [_p, _p, _p, _f, _f, _f, _f, _f, _f, _i, _fp, _fp]),
    "gpt2_device_loss": (_p, [_p]),
    "gpt2_device_norm": (_p, [_p]),
    "gpt2_profile": (_i, [_p, _i]),
    "gpt2_profile_read": (_i, [_p, _i, ct.POINTER(_i), ct.POINTER(ct.c_double), ct.POINTER(ct.c_double),
                               ct.POINTER(ct.c_double)]),
    "gpt2_profile_regions": (_i, [_p]),
    "gpt2_profile_region": (_i, [_p, _i, ct.POINTER(_i), ct.POINTER(_i), ct.POINTER(ct.c_double),
                                 ct.POINTER(ct.c_double), ct.POINTER(ct.c_double)]),
    "gpt2_sync_status": (_i, [_p]),
    "gpt2_strerror": (ct.c_char_p, [_i]),
    "gpt2_last_cuda_error": (ct.c_char_p, []),
    "attn_fwd": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _ll, _ll, _ll, _ll, _ll, _ll, _f, _p]),
    "attn_bwd": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _ll, _ll, _ll, _ll, _ll,
                      _ll, _f, _p, _sz, _p]),
    "attn_workspace_bytes": (_sz, [_i, _i, _i]),
    "attn_bwd_noalloc": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _ll, _ll, _ll, _ll, _ll,
                              _ll, _f, _p]),
    "classifier_fwd_bwd": (_i, [_p, _p, _p, _i, _i, _i, _i, _p, _p, _p, _p, _sz, _p]),
    "classifier_workspace_bytes": (_sz, [_i, _i, _i]),
    "gpt2_encoder_fwd": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _i, _p, _p]),
    "gpt2_encoder_bwd": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _i, _p, _sz, _p]),
    "gemm_bf16": (_i, [_p, _p, _p, _i, _i, _i, _ll, _ll, _ll, _i, _i, _i, _i, _p, _sz, _p]),
    "gemm_bf16_sk_workspace_bytes": (_sz, []),
    "gemm_bf16_pairs": (_i, []),
    "gpt2_lr_schedule": (_f, [_i, _f, _i, _i, _f]),
    "gpt2_grad_accumulate": (_i, [_p, _i, _f]),
    "gpt2_clip_adamw_accumulated": (_i, [_p, _f, _f, _f, _f, _f, _f, _i, _p]),
    "gemm_bf16_epilogue": (_i, [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _ll, _ll, _ll, _i, _i, _i, _i, _p, _sz,
                                _p]),
    "gpt2_test_set_poison": (_i, [_i]),
    "gpt2_test_set_gemm_poison": (_i, [_i]),
    "gemm_bf16_status": (_i, [_p, _p, _p, _i, _i, _i, _ll, _ll, _ll, _i, _i, _i, _p, _sz, _p, _p]),
    "gpt2_set_guard": (_i, [_p, _f, _f, _i]),
    "gpt2_guard_read": (_i, [_p, _fp, _fp, ct.POINTER(_i), ct.POINTER(_i), ct.POINTER(_i)]),
}

_lib = None


def lib() -> ct.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m pretraining_step_train_b300.build`")
        L = ct.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


class GPT2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib().gpt2_strerror(status).decode()
        if status == GPT2_E_CUDA:
            msg += ": " + lib().gpt2_last_cuda_error().decode()
        super().__init__(f"{where}: {msg} ({status})")
        self.status = status


def check(status: int, where: str = "libgpt2") -> int:
    if status != GPT2_OK:
        raise GPT2Error(status, where)
    return status


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream_ptr(stream) -> int:
    return 0 if stream is None else int(stream.cuda_stream)


def __getattr__(name):
    # module-level access to the raw C functions under their C names
    if name in SIGNATURES:
        return getattr(lib(), name)
    raise AttributeError(name)


class Step:
    """One GPT-2 step driver over a torch-allocated device arena."""

    def __init__(self, L, H, C, V, Vpad, T, B, precision=GPT2_BF16, stream=None, device="cuda", recompute=0):
        import torch

        self.shape = dict(L=L, H=H, C=C, V=V, Vpad=Vpad, T=T, B=B)
        self.precision = precision
        self.recompute = recompute
        nbytes = lib().gpt2_arena_bytes_r(L, H, C, V, Vpad, T, B, precision, recompute)
        if nbytes == 0:
            raise GPT2Error(GPT2_E_INVAL, "gpt2_arena_bytes_r")
        self.arena = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.stream = stream
        h = _p()
        check(lib().gpt2_create_r(L, H, C, V, Vpad, T, B, precision, recompute, _ptr(self.arena), nbytes,
                                  _stream_ptr(stream), ct.byref(h)), "gpt2_create_r")
        self.h = h
        self.N = lib().gpt2_num_params(L, C, Vpad, T)

    def close(self):
        if getattr(self, "h", None):
            lib().gpt2_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_params(self, flat):
        """flat: float32 numpy array or CUDA tensor of N parameters (canonical order)."""
        import numpy as np

        if hasattr(flat, "data_ptr"):
            check(lib().gpt2_set_params(self.h, _ptr(flat), 1 if flat.is_cuda else 0), "gpt2_set_params")
        else:
            a = np.ascontiguousarray(flat, dtype=np.float32)
            assert a.size == self.N
            check(lib().gpt2_set_params(self.h, a.ctypes.data, 0), "gpt2_set_params")

    def get(self, which):
        import numpy as np

        out = np.empty(self.N, dtype=np.float32)
        check(lib().gpt2_get_tensor(self.h, which, out.ctypes.data, 0), "gpt2_get_tensor")
        return out

    def forward(self, tokens, targets, want_loss=True):
        loss = ct.c_float(0.0)
        check(lib().gpt2_forward(self.h, _ptr(tokens), _ptr(targets),
                                 ct.byref(loss) if want_loss else None), "gpt2_forward")
        return loss.value if want_loss else None

    def backward(self):
        check(lib().gpt2_backward(self.h), "gpt2_backward")

    def clip_adamw(self, lr=6e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=1.0,
                   t=1, want_norm=True):
        norm = ct.c_float(0.0)
        check(lib().gpt2_clip_adamw(self.h, lr, beta1, beta2, eps, weight_decay, max_norm, t,
                                    ct.byref(norm) if want_norm else None), "gpt2_clip_adamw")
        return norm.value if want_norm else None

    def grad_accumulate(self, first, scale):
        check(lib().gpt2_grad_accumulate(self.h, 1 if first else 0, scale), "gpt2_grad_accumulate")

    def clip_adamw_accumulated(self, lr=6e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1,
                               max_norm=1.0, t=1, want_norm=True):
        norm = ct.c_float(0.0)
        check(lib().gpt2_clip_adamw_accumulated(self.h, lr, beta1, beta2, eps, weight_decay, max_norm, t,
                                                ct.byref(norm) if want_norm else None),
              "gpt2_clip_adamw_accumulated")
        return norm.value if want_norm else None

    def train_step_host(self, tokens_np, targets_np, lr=6e-4, beta1=0.9, beta2=0.95, eps=1e-8,
                        weight_decay=0.1, max_norm=1.0, t=1):
        """Whole step from host int32 arrays (numpy or pinned CPU tensors); returns (loss, norm)."""
        loss, norm = ct.c_float(0.0), ct.c_float(0.0)

        def addr(a):
            return a.data_ptr() if hasattr(a, "data_ptr") else a.ctypes.data

        check(lib().gpt2_train_step_host(self.h, addr(tokens_np), addr(targets_np), lr, beta1, beta2,
                                         eps, weight_decay, max_norm, t, ct.byref(loss),
                                         ct.byref(norm)), "gpt2_train_step_host")
        return loss.value, norm.value

    def set_stream(self, stream):
        self.stream = stream
        check(lib().gpt2_set_stream(self.h, _stream_ptr(stream)), "gpt2_set_stream")

    def profile(self, on: bool):
        check(lib().gpt2_profile(self.h, 1 if on else 0), "gpt2_profile")

    def profile_read(self):
        """{class name: (regions, ms, flops, bytes)} of the regions recorded since profile(True)."""
        out = {}
        for i, name in enumerate(KERNEL_CLASSES):
            n, ms, fl, by = ct.c_int(), ct.c_double(), ct.c_double(), ct.c_double()
            check(lib().gpt2_profile_read(self.h, i, ct.byref(n), ct.byref(ms), ct.byref(fl), ct.byref(by)),
                  "gpt2_profile_read")
            out[name] = (n.value, ms.value, fl.value, by.value)
        return out

    def profile_regions(self):
        """[(class name, dims tuple, ms, flops, bytes)] of every recorded region in issue order."""
        out = []
        for i in range(lib().gpt2_profile_regions(self.h)):
            c, ms, fl, by = ct.c_int(), ct.c_double(), ct.c_double(), ct.c_double()
            dims = (ct.c_int * 6)()
            check(lib().gpt2_profile_region(self.h, i, ct.byref(c), dims, ct.byref(ms), ct.byref(fl),
                                            ct.byref(by)), "gpt2_profile_region")
            out.append((KERNEL_CLASSES[c.value], tuple(dims), ms.value, fl.value, by.value))
        return out

    def device_loss_ptr(self) -> int:
        return lib().gpt2_device_loss(self.h)

    def device_norm_ptr(self) -> int:
        return lib().gpt2_device_norm(self.h)

    def sync_status(self) -> int:
        return lib().gpt2_sync_status(self.h)

    def set_guard(self, loss_z=0.0, norm_z=0.0, window=128):
        check(lib().gpt2_set_guard(self.h, loss_z, norm_z, window), "gpt2_set_guard")

    def guard_read(self):
        """{z_loss, z_norm, skipped_spike, skipped_nonfinite, last_skipped} of the update guard."""
        zl, zn = ct.c_float(), ct.c_float()
        sp, nf, last = ct.c_int(), ct.c_int(), ct.c_int()
        check(lib().gpt2_guard_read(self.h, ct.byref(zl), ct.byref(zn), ct.byref(sp), ct.byref(nf),
                                    ct.byref(last)), "gpt2_guard_read")
        return dict(z_loss=zl.value, z_norm=zn.value, skipped_spike=sp.value, skipped_nonfinite=nf.value,
                    last_skipped=last.value)
