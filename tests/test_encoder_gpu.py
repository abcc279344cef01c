"""Bit-exactness of the embedding gather (forward) and the fixed-order
gradient scatter (backward) through the C ABI, against the oracle's float32
sequential references."""
import numpy as np
import pytest

from oracle import gpt2_oracle as O
from pretraining_step_train_b300 import binding, synth
from tests._helpers import to_dev, to_np

pytestmark = pytest.mark.gpu


def _tok(seed, B, T, V, dist="zipf"):
    return synth.token_batch(seed, B, T, V, dist)[0]


@pytest.mark.parametrize("prec", [binding.GPT2_FP32, binding.GPT2_BF16])
@pytest.mark.parametrize("B,T,C,V,Vpad", [(4, 64, 64, 256, 256), (16, 1024, 768, 50257, 50304), (1, 1, 8, 3, 8)])
def test_encoder_forward_bit_exact(prec, B, T, C, V, Vpad):
    import torch
    tok = _tok(B * T + C, B, T, V)
    wte = synth.normal(1, Vpad * C, 0.02).astype(np.float32).reshape(Vpad, C)
    wpe = synth.normal(2, T * C, 0.02).astype(np.float32).reshape(T, C)
    dt = "bf16" if prec == binding.GPT2_BF16 else "f32"
    if prec == binding.GPT2_BF16:
        wte, wpe = synth.round_to_bf16(wte).reshape(Vpad, C), synth.round_to_bf16(wpe).reshape(T, C)
    x0 = torch.empty((B, T, C), dtype=torch.bfloat16 if dt == "bf16" else torch.float32, device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    # keep every device tensor referenced until the kernel has run
    tok_d, wte_d, wpe_d = to_dev(tok, "i32"), to_dev(wte, dt), to_dev(wpe, dt)
    binding.check(binding.lib().gpt2_encoder_fwd(tok_d.data_ptr(), wte_d.data_ptr(), wpe_d.data_ptr(),
                                                 x0.data_ptr(), B, T, C, V, prec, st.data_ptr(), None))
    torch.cuda.synchronize()
    ref = O.encoder_forward_f32(tok, wte, wpe)
    if prec == binding.GPT2_BF16:
        ref = synth.round_to_bf16(ref).reshape(ref.shape)
    np.testing.assert_array_equal(to_np(x0), ref)
    assert int(st[0].item()) == 0


@pytest.mark.parametrize("prec", [binding.GPT2_FP32, binding.GPT2_BF16])
@pytest.mark.parametrize("B,T,C,V,Vpad", [(4, 64, 64, 256, 256), (16, 1024, 768, 50257, 50304), (1, 3, 8, 3, 8)])
def test_encoder_backward_bit_exact(prec, B, T, C, V, Vpad):
    import torch
    tok = _tok(B * T + 1, B, T, V)
    dx0 = synth.normal(3, B * T * C, 1e-3).astype(np.float32).reshape(B, T, C)
    din = synth.normal(4, Vpad * C, 1e-3).astype(np.float32).reshape(Vpad, C)
    dt = "bf16" if prec == binding.GPT2_BF16 else "f32"
    if prec == binding.GPT2_BF16:
        din = synth.round_to_bf16(din).reshape(Vpad, C)
    dwte = to_dev(din, dt)
    dwpe = torch.full((T, C), float("nan"), dtype=dwte.dtype, device="cuda")
    ws = torch.empty(8 * B * T, dtype=torch.uint8, device="cuda")
    tok_d, dx0_d = to_dev(tok, "i32"), to_dev(dx0, "f32")
    binding.check(binding.lib().gpt2_encoder_bwd(tok_d.data_ptr(), dx0_d.data_ptr(), dwte.data_ptr(),
                                                 dwpe.data_ptr(), B, T, C, V, prec, ws.data_ptr(), ws.numel(),
                                                 None))
    torch.cuda.synchronize()
    ref_wte, ref_wpe = O.encoder_backward_f32(tok, dx0, din, (T, C))
    if prec == binding.GPT2_BF16:
        ref_wte = synth.round_to_bf16(ref_wte).reshape(ref_wte.shape)
        ref_wpe = synth.round_to_bf16(ref_wpe).reshape(ref_wpe.shape)
    np.testing.assert_array_equal(to_np(dwte), ref_wte)
    np.testing.assert_array_equal(to_np(dwpe), ref_wpe)


def test_encoder_out_of_range_tokens_flagged_and_clamped():
    import torch
    B, T, C, V = 2, 8, 16, 10
    tok = _tok(5, B, T, V, "uniform")
    tok[0, 3] = -1
    tok[1, 7] = V
    wte = synth.normal(1, V * C).astype(np.float32).reshape(V, C)
    wpe = synth.normal(2, T * C).astype(np.float32).reshape(T, C)
    x0 = torch.empty((B, T, C), dtype=torch.float32, device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    tok_d, wte_d, wpe_d = to_dev(tok, "i32"), to_dev(wte, "f32"), to_dev(wpe, "f32")
    binding.check(binding.lib().gpt2_encoder_fwd(tok_d.data_ptr(), wte_d.data_ptr(), wpe_d.data_ptr(),
                                                 x0.data_ptr(), B, T, C, V, binding.GPT2_FP32, st.data_ptr(),
                                                 None))
    torch.cuda.synchronize()
    assert int(st[0].item()) & 1
    clamped = np.where((tok < 0) | (tok >= V), 0, tok)
    np.testing.assert_array_equal(to_np(x0), O.encoder_forward_f32(clamped, wte, wpe))
