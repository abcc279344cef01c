"""attn_bwd_noalloc: the attention backward for callers that cannot allocate
device memory (a runtime that owns the whole device through its own pool, or
a loop that cannot afford cudaMalloc's device synchronisation).  It keeps its
scratch in a fixed array of the library's static device memory instead of a
caller workspace, and must give the same gradients as attn_bwd.

This file sorts last so that a run stopping at the first failure has already
run every other test; it passes alone in a fresh process too (the first call
looks the array's address up)."""
import ctypes as ct

import numpy as np
import pytest

from pretraining_step_train_b300 import binding, build, synth
from tests._helpers import rel_l2, to_dev, to_np

D = 64
SCALE = 1.0 / 8.0


def _grads(seed, B, H, T, noalloc):
    """attn_fwd, then attn_bwd (with a workspace) or attn_bwd_noalloc, on [B, H, T, 64] inputs."""
    import torch
    q, k, v, do = synth.attention_inputs(seed, B, H, T, D)
    qd, kd, vd, dod = (to_dev(x) for x in (q, k, v, do))
    strides = (H * T * D, T * D, D)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    L = binding.lib()
    views = (qd.data_ptr(), kd.data_ptr(), vd.data_ptr())
    binding.check(L.attn_fwd(*views, o.data_ptr(), lse.data_ptr(), B, H, T, D, *strides, *strides, SCALE,
                             None))
    dq, dk, dv = (torch.empty_like(qd) for _ in range(3))
    dviews = (dq.data_ptr(), dk.data_ptr(), dv.data_ptr())
    if noalloc:
        binding.check(L.attn_bwd_noalloc(*views, o.data_ptr(), lse.data_ptr(), dod.data_ptr(), *dviews,
                                         B, H, T, D, *strides, *strides, SCALE, None), "attn_bwd_noalloc")
    else:
        ws = torch.empty(L.attn_workspace_bytes(B, H, T), dtype=torch.uint8, device="cuda")
        binding.check(L.attn_bwd(*views, o.data_ptr(), lse.data_ptr(), dod.data_ptr(), *dviews, B, H, T, D,
                                 *strides, *strides, SCALE, ws.data_ptr(), ws.numel(), None), "attn_bwd")
    torch.cuda.synchronize()
    return [to_np(t) for t in (dq, dk, dv)]


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    """Two calls in a row (a larger then a smaller, ragged shape, so the second
    finds the first call's values in the shared array) against attn_bwd."""
    for seed, B, H, T in ((21, 2, 3, 256), (22, 1, 2, 200)):
        ref = _grads(seed, B, H, T, noalloc=False)
        got = _grads(seed, B, H, T, noalloc=True)
        for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
            assert np.isfinite(g).all(), name
            assert rel_l2(g, r) < 3e-2, (name, rel_l2(g, r))
            np.testing.assert_array_equal(g, r)  # same kernels, same order: identical bits


def test_noalloc_rejects_sizes_beyond_its_array_on_the_host():
    """B*H*T above the fixed array is refused before anything is enqueued."""
    build.build()
    L = binding.lib()
    fake = 1 << 20  # 16-byte aligned stand-in pointers: nothing is dereferenced on this path
    too_many = L.attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, 64, 16, 1025, D,
                                  1, 1, 1, 1, 1, 1, SCALE, None)
    assert too_many == binding.GPT2_E_UNSUPPORTED
    assert 64 * 16 * 1025 > 1048576
