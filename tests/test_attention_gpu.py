"""Parity of the fused causal attention kernels (attn_fwd / attn_bwd, through
the C ABI) with the oracle's materialised T x T masked softmax in float64."""
import numpy as np
import pytest

from oracle import gpt2_oracle as O
from pretraining_step_train_b300 import binding, synth
from tests._helpers import rel_l2, to_dev, to_np

pytestmark = pytest.mark.gpu

D = 64
SCALE = 1.0 / 8.0
LSE_TOL = 1e-4


def _run(q, k, v, do, layout):
    import torch
    B, H, T, d = q.shape
    if layout == "bhtd":
        dev = [to_dev(x) for x in (q, k, v, do)]
        qd, kd, vd, dod = dev
        strides = (H * T * d, T * d, d)
        ostr = strides
        o = torch.empty_like(qd)
        dq, dk, dv = (torch.empty_like(qd) for _ in range(3))
        views = (qd.data_ptr(), kd.data_ptr(), vd.data_ptr())
        dviews = (dq.data_ptr(), dk.data_ptr(), dv.data_ptr())
        get = lambda t: to_np(t)
        oget = lambda t: to_np(t)
    else:  # the step's packed qkv layout [B, T, 3C] and [B, T, C] outputs
        C = H * d
        packed = np.concatenate([x.transpose(0, 2, 1, 3).reshape(B, T, C) for x in (q, k, v)], axis=-1)
        qkv = to_dev(packed)
        dod = to_dev(do.transpose(0, 2, 1, 3).reshape(B, T, C))
        strides = (T * 3 * C, d, 3 * C)
        ostr = (T * C, d, C)
        o = torch.empty((B, T, C), dtype=torch.bfloat16, device="cuda")
        dqkv = torch.empty((B, T, 3 * C), dtype=torch.bfloat16, device="cuda")
        e = qkv.element_size()
        views = (qkv.data_ptr(), qkv.data_ptr() + C * e, qkv.data_ptr() + 2 * C * e)
        dviews = (dqkv.data_ptr(), dqkv.data_ptr() + C * e, dqkv.data_ptr() + 2 * C * e)
        unpack = lambda a, i: a[..., i * C:(i + 1) * C].reshape(B, T, H, d).transpose(0, 2, 1, 3)
        oget = lambda t: to_np(t).reshape(B, T, H, d).transpose(0, 2, 1, 3)
        dq = dk = dv = None
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    L = binding.lib()
    binding.check(L.attn_fwd(*views, o.data_ptr(), lse.data_ptr(), B, H, T, d, *strides, *ostr, SCALE, None))
    ws = torch.empty(L.attn_workspace_bytes(B, H, T), dtype=torch.uint8, device="cuda")
    binding.check(L.attn_bwd(*views, o.data_ptr(), lse.data_ptr(), dod.data_ptr(), *dviews, B, H, T, d,
                             *strides, *ostr, SCALE, ws.data_ptr(), ws.numel(), None))
    torch.cuda.synchronize()
    if layout == "bhtd":
        return oget(o), to_np(lse), get(dq), get(dk), get(dv)
    g = to_np(dqkv)
    return oget(o), to_np(lse), unpack(g, 0), unpack(g, 1), unpack(g, 2)


# The last two cases put about two work items on every CTA with an odd number of query
# tiles (5): each CTA walks a single-tile item before paired ones, so shared-memory sets,
# ring stages and the deferred releases after the tensor stores cycle across items.
@pytest.mark.parametrize("B,H,T,layout", [(2, 3, 128, "bhtd"), (1, 2, 200, "bhtd"), (2, 2, 64, "bhtd"),
                                          (2, 2, 192, "qkv"), (1, 1, 1, "bhtd"), (1, 2, 100, "qkv"),
                                          (8, 12, 640, "bhtd"), (8, 12, 640, "qkv")])
def test_attention_parity(B, H, T, layout):
    q, k, v, do = synth.attention_inputs(B * 100 + H * 10 + T, B, H, T, D)
    o, lse, dq, dk, dv = _run(q, k, v, do, layout)
    q64, k64, v64, do64 = (x.astype(np.float64) for x in (q, k, v, do))
    o_ref, p, lse_ref = O.attention_forward(q64, k64, v64, SCALE)
    dq_r, dk_r, dv_r = O.attention_backward(do64, q64, k64, v64, p, SCALE)
    assert rel_l2(o, o_ref) < 1e-2
    # lse is accumulated in fp32 from the fp32 scores (2^x by ex2.approx, ~2^-22 relative):
    # an off-by-one in the diagonal mask would move row i by about 1/(i+1)
    assert np.abs(lse - lse_ref).max() < LSE_TOL, np.abs(lse - lse_ref).max()
    for got, ref, nm in ((dq, dq_r, "dq"), (dk, dk_r, "dk"), (dv, dv_r, "dv")):
        assert rel_l2(got, ref) < 3e-2, (nm, rel_l2(got, ref))


@pytest.mark.parametrize("T", [1024, 2048, 4096])
def test_attention_microbench_shape_sampled_heads(T):
    """The attention microbench layout [16, 12, T, 64] up to the top of its T sweep;
    oracle on a few sampled (b, h)."""
    import torch
    B, H = 16, 12
    q, k, v, do = synth.attention_inputs(T, B, H, T, D)
    o, lse, dq, dk, dv = _run(q, k, v, do, "bhtd")
    rng = np.random.default_rng(T)
    for _ in range(3):
        b, h = int(rng.integers(B)), int(rng.integers(H))
        sl = lambda x: x[b:b + 1, h:h + 1].astype(np.float64)
        o_ref, p, lse_ref = O.attention_forward(sl(q), sl(k), sl(v), SCALE)
        dq_r, dk_r, dv_r = O.attention_backward(sl(do), sl(q), sl(k), sl(v), p, SCALE)
        assert rel_l2(o[b:b + 1, h:h + 1], o_ref) < 1e-2
        assert np.abs(lse[b:b + 1, h:h + 1] - lse_ref).max() < LSE_TOL
        for got, ref in ((dq, dq_r), (dk, dk_r), (dv, dv_r)):
            assert rel_l2(got[b:b + 1, h:h + 1], ref) < 3e-2


def test_attention_deterministic():
    q, k, v, do = synth.attention_inputs(5, 2, 2, 256, D)
    r1 = _run(q, k, v, do, "bhtd")
    r2 = _run(q, k, v, do, "bhtd")
    for a, b in zip(r1, r2):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("layout", ["bhtd", "qkv"])
def test_attention_causality_bit_identical(layout):
    """Keys and values after position t0 never reach a query at or before t0:
    perturbing them leaves those rows of O and lse bit-identical (forward), and
    dQ of those rows too (backward), while later rows do change.  t0 sits inside
    a 128-key tile, so the masked diagonal tile is exercised."""
    B, H, T = 2, 3, 384
    t0 = 200
    q, k, v, do = synth.attention_inputs(91, B, H, T, D)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, t0 + 1:] = synth.round_to_bf16(k2[:, :, t0 + 1:] * -3.0 + 0.5).reshape(k2[:, :, t0 + 1:].shape)
    v2[:, :, t0 + 1:] = synth.round_to_bf16(v2[:, :, t0 + 1:] * 2.0 - 1.0).reshape(v2[:, :, t0 + 1:].shape)
    o1, l1, dq1, _, _ = _run(q, k, v, do, layout)
    o2, l2, dq2, _, _ = _run(q, k2, v2, do, layout)
    np.testing.assert_array_equal(o1[:, :, :t0 + 1], o2[:, :, :t0 + 1])
    np.testing.assert_array_equal(l1[:, :, :t0 + 1], l2[:, :, :t0 + 1])
    np.testing.assert_array_equal(dq1[:, :, :t0 + 1], dq2[:, :, :t0 + 1])
    assert not np.array_equal(o1[:, :, t0 + 1:], o2[:, :, t0 + 1:])
    assert not np.array_equal(l1[:, :, t0 + 1:], l2[:, :, t0 + 1:])
