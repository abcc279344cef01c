"""Every family of bounded waits in the pipelined kernels gives up after about
2 s, reports GPT2_E_TIMEOUT through the status word and leaves the context
usable.  The failure is made on the host: a test hook makes one producer skip
one transfer (no fault, trap or endless loop), and the next call on the same
context must match a fresh handle bit for bit."""
import numpy as np
import pytest

from oracle import gpt2_oracle as O
from pretraining_step_train_b300 import binding, synth
from tests._helpers import rel_l2, to_dev, to_np

pytestmark = pytest.mark.gpu

POISON_GEMM_FLAG, POISON_ATTN_FWD, POISON_ATTN_DQ, POISON_ATTN_DKDV, POISON_LN_BWD = 2, 4, 8, 16, 32
L, H, C, V, Vpad, T, B = 1, 2, 128, 1000, 1024, 256, 2


def _clean_step(s, batch):
    loss = s.forward(*batch)
    s.backward()
    norm = s.clip_adamw(t=1)
    return loss, norm, {w: s.get(w) for w in (binding.GPT2_GRADS, binding.GPT2_MASTER)}


@pytest.mark.parametrize("bit,phase", [(POISON_ATTN_FWD, "forward"), (POISON_ATTN_DQ, "backward"),
                                       (POISON_ATTN_DKDV, "backward"), (POISON_LN_BWD, "backward")])
def test_step_wait_expires_and_context_survives(bit, phase):
    """Attention forward, the two attention backward kernels and the streaming
    LayerNorm backward: a poisoned pass reports GPT2_E_TIMEOUT; the next step
    on the same handle equals a fresh handle's step bit for bit."""
    P = synth.init_params(111, L, C, V, Vpad, T, bf16_representable=True)
    flat = synth.flatten_params(P, L, C, Vpad, T)
    tok, tgt = synth.token_batch(112, B, T, V)
    batch = (to_dev(tok, "i32"), to_dev(tgt, "i32"))
    s = binding.Step(L, H, C, V, Vpad, T, B, precision=binding.GPT2_BF16)
    s.set_params(flat)
    lib = binding.lib()
    old = lib.gpt2_test_set_poison(bit)
    try:
        s.forward(*batch, want_loss=False)
        if phase == "backward":
            s.backward()
        st = s.sync_status()
    finally:
        lib.gpt2_test_set_poison(old)
    assert st == binding.GPT2_E_TIMEOUT
    assert s.sync_status() == binding.GPT2_OK  # read and cleared
    got = _clean_step(s, batch)
    f = binding.Step(L, H, C, V, Vpad, T, B, precision=binding.GPT2_BF16)
    f.set_params(flat)
    ref = _clean_step(f, batch)
    assert got[0] == ref[0] and got[1] == ref[1]
    for w in got[2]:
        np.testing.assert_array_equal(got[2][w], ref[2][w])
    oref = O.train_step(P, tok, tgt, O.Config(L, H, C, V, Vpad, T), lr=6e-4, t=1)
    assert abs(got[0] - oref["loss"]) / oref["loss"] < 1e-2
    s.close()
    f.close()


def test_stream_k_flag_wait_expires_and_workspace_stays_usable():
    """The stream-K schedule (10 output tiles cut along K over every SM): with
    the partial units' ready flags withheld, the finishing CTAs' flag waits run
    out; the call reports GPT2_E_TIMEOUT and the same workspace serves the next
    call, which is correct."""
    import torch
    M, N, K = 640, 264, 2112
    a = synth.round_to_bf16(synth.normal(121, M * K)).reshape(M, K)
    b = synth.round_to_bf16(synth.normal(122, N * K)).reshape(N, K)
    A, Bm = to_dev(a), to_dev(b)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    lib = binding.lib()
    ws = torch.zeros(lib.gemm_bf16_sk_workspace_bytes(), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (A.data_ptr(), Bm.data_ptr(), D.data_ptr(), M, N, K, K, K, N, 0, 0, -2, ws.data_ptr(), ws.numel(),
            st.data_ptr(), None)
    old = lib.gpt2_test_set_poison(POISON_GEMM_FLAG)
    try:
        r = lib.gemm_bf16_status(*args)
    finally:
        lib.gpt2_test_set_poison(old)
    assert r == binding.GPT2_E_TIMEOUT
    assert lib.gemm_bf16_status(*args) == binding.GPT2_OK
    ref = a.astype(np.float64) @ b.astype(np.float64).T
    assert rel_l2(to_np(D), ref) < 4e-3
