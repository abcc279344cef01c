"""Parity of the tcgen05 GEMM engine (through the C ABI) with the plain
definition D = A B^T evaluated in float64 on the same bf16 inputs."""
import ctypes as ct

import numpy as np
import pytest

from pretraining_step_train_b300 import binding, synth
from tests._helpers import rel_l2, to_dev, to_np

pytestmark = pytest.mark.gpu


def _operands(seed, M, N, K, a_mn, b_mn):
    a = synth.round_to_bf16(synth.normal(seed, M * K)).reshape(M, K)
    b = synth.round_to_bf16(synth.normal(seed + 1, N * K)).reshape(N, K)
    pad = lambda n: (n + 7) // 8 * 8
    if a_mn:
        lda = pad(M)
        As = np.zeros((K, lda), np.float32); As[:, :M] = a.T
    else:
        lda = pad(K)
        As = np.zeros((M, lda), np.float32); As[:, :K] = a
    if b_mn:
        ldb = pad(N)
        Bs = np.zeros((K, ldb), np.float32); Bs[:, :N] = b.T
    else:
        ldb = pad(K)
        Bs = np.zeros((N, ldb), np.float32); Bs[:, :K] = b
    return a, b, As, Bs, lda, ldb


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 520, 200), (1024, 768, 768), (64, 8, 16)])
def test_gemm_majors_fp32_out(a_mn, b_mn, M, N, K):
    import torch
    a, b, As, Bs, lda, ldb = _operands(M + N + K, M, N, K, a_mn, b_mn)
    A, B = to_dev(As), to_dev(Bs)
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    binding.check(binding.lib().gemm_bf16(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, lda, ldb, N,
                                          a_mn, b_mn, 1, 1, None, 0, None))
    torch.cuda.synchronize()
    ref = a.astype(np.float64) @ b.astype(np.float64).T
    got = to_np(D)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=0, atol=2e-5 * np.sqrt(K) * 4)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 1), (0, 1)])
def test_gemm_bf16_out_and_splitk(a_mn, b_mn):
    import torch
    M, N, K = 256, 512, 4096
    a, b, As, Bs, lda, ldb = _operands(7, M, N, K, a_mn, b_mn)
    A, B = to_dev(As), to_dev(Bs)
    ref = a.astype(np.float64) @ b.astype(np.float64).T
    for splits in (1, 4, 7):
        for f32 in (0, 1):
            D = torch.empty((M, N), dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")
            ws = torch.empty(splits * M * N * 4 + 256, dtype=torch.uint8, device="cuda")
            binding.check(binding.lib().gemm_bf16(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, lda, ldb,
                                                  N, a_mn, b_mn, f32, splits, ws.data_ptr(), ws.numel(), None))
            torch.cuda.synchronize()
            err = rel_l2(to_np(D), ref)
            # fp32 sums of K=4096 products: ~sqrt(K) * 2^-24 relative; bf16 output adds 2^-9
            assert err < (2e-5 if f32 else 4e-3), (splits, f32, err)


def test_gemm_deterministic():
    import torch
    M, N, K = 512, 768, 3072
    a, b, As, Bs, lda, ldb = _operands(9, M, N, K, 1, 1)
    A, B = to_dev(As), to_dev(Bs)
    outs = []
    for _ in range(2):
        D = torch.empty((M, N), dtype=torch.float32, device="cuda")
        ws = torch.empty(16 * M * N * 4, dtype=torch.uint8, device="cuda")
        binding.check(binding.lib().gemm_bf16(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, lda, ldb, N,
                                              1, 1, 1, 0, ws.data_ptr(), ws.numel(), None))
        outs.append(to_np(D))
    np.testing.assert_array_equal(outs[0], outs[1])


def _sk_workspace():
    import torch
    n = binding.lib().gemm_bf16_sk_workspace_bytes()
    assert n > 0
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (1024, 768, 768), (640, 264, 4160), (64, 8, 16)])
def test_gemm_in_kernel_partials(a_mn, b_mn, M, N, K):
    """The schedules that add partial sums inside the kernel.  -2 forces stream-K
    whenever the tiles leave a wave partly empty: with fewer tiles than SMs every
    tile is cut along K over many CTAs (down to one 64-wide k block each, several
    partial sums per tile, CTAs with no work).  -1 takes K splits with an
    in-kernel finish on these few-tile shapes (13 splits for K = 4160, 3 for
    K = 768, none where K is too short to split)."""
    import torch
    a, b, As, Bs, lda, ldb = _operands(M * 3 + N + K, M, N, K, a_mn, b_mn)
    A, B = to_dev(As), to_dev(Bs)
    ref = a.astype(np.float64) @ b.astype(np.float64).T
    ws = _sk_workspace()
    # the workspace is reused: each call leaves its flags lowered
    for mode, f32 in ((-2, 1), (-2, 0), (-1, 1), (-1, 0), (-2, 1)):
        D = torch.full((M, N), float("nan"), dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")
        binding.check(binding.lib().gemm_bf16(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, lda, ldb, N,
                                              a_mn, b_mn, f32, mode, ws.data_ptr(), ws.numel(), None))
        torch.cuda.synchronize()
        got = to_np(D)
        assert np.isfinite(got).all()
        if f32:
            np.testing.assert_allclose(got, ref, rtol=0, atol=2e-5 * np.sqrt(K) * 4)
        else:
            assert rel_l2(got, ref) < 4e-3
    # the flags sit in front of the partial-sum slots (three per SM, 128 x 256 fp32 each)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    flag_bytes = binding.lib().gemm_bf16_sk_workspace_bytes() - 3 * sms * 128 * 256 * 4
    flags = to_np(ws[:flag_bytes].view(torch.int32))
    assert not flags.any()


@pytest.mark.parametrize("M,N,K,a_mn,b_mn", [
    (16384, 768, 3072, 0, 1),   # 192 pair tiles on 74 pairs: two whole waves + 44 tiles cut along K
    (768, 3072, 16384, 1, 1),   # 36 pair tiles, two K splits finished in-kernel
])
def test_gemm_stream_k_step_shapes(M, N, K, a_mn, b_mn):
    """The schedule the training step takes (-1) on two of its GEMM shapes: equal to
    the float64 product within fp32 rounding, and bitwise repeatable."""
    import torch
    a, b, As, Bs, lda, ldb = _operands(11, M, N, K, a_mn, b_mn)
    A, B = to_dev(As), to_dev(Bs)
    ws = _sk_workspace()
    outs = []
    for _ in range(2):
        D = torch.empty((M, N), dtype=torch.float32, device="cuda")
        binding.check(binding.lib().gemm_bf16(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, lda, ldb, N,
                                              a_mn, b_mn, 1, -1, ws.data_ptr(), ws.numel(), None))
        outs.append(to_np(D))
    np.testing.assert_array_equal(outs[0], outs[1])
    rows = np.random.default_rng(0).choice(M, 256, replace=False)
    ref = a[rows].astype(np.float64) @ b.astype(np.float64).T
    np.testing.assert_allclose(outs[0][rows], ref, rtol=0, atol=2e-5 * np.sqrt(K) * 4)


def _epilogue_case(seed, M, N, K, a_mn, b_mn, epi, splits):
    """Run gemm_bf16_epilogue and its float64 reference on the same bf16 inputs."""
    import torch
    from oracle import gpt2_oracle as O
    a, b, As, Bs, lda, ldb = _operands(seed, M, N, K, a_mn, b_mn)
    A, B = to_dev(As), to_dev(Bs)
    bias = synth.round_to_bf16(synth.normal(seed + 2, N) * 0.5)
    X = synth.round_to_bf16(synth.normal(seed + 3, M * N).reshape(M, N))
    bias_d, X_d = to_dev(bias, "bf16"), to_dev(X, "bf16")
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    D2 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    G = (M + 31) // 32
    colpart = torch.full((G, N), float("nan"), dtype=torch.float32, device="cuda")
    ws = _sk_workspace()
    binding.check(binding.lib().gemm_bf16_epilogue(
        A.data_ptr(), B.data_ptr(), D.data_ptr(), D2.data_ptr(), bias_d.data_ptr(), X_d.data_ptr(),
        colpart.data_ptr() if epi == 4 else None, M, N, K, lda, ldb, N, a_mn, b_mn, epi, splits,
        ws.data_ptr(), ws.numel(), None))
    torch.cuda.synchronize()
    acc = a.astype(np.float64) @ b.astype(np.float64).T
    x = X.astype(np.float64)
    if epi == 1:
        ref = {"D": acc + bias}
    elif epi == 2:
        ref = {"D": acc + bias + x}
    elif epi == 3:
        h = acc + bias
        ref = {"D": O.gelu_grad(h), "D2": O.gelu(h)}
    else:
        dh = acc * x
        pad = np.zeros((G * 32, N)); pad[:M] = dh
        ref = {"D": dh, "colpart": pad.reshape(G, 32, N).sum(axis=1)}
    got = {"D": to_np(D), "D2": to_np(D2), "colpart": to_np(colpart)}
    return got, ref


@pytest.mark.parametrize("M,N,K,a_mn,b_mn,splits", [
    (640, 264, 2112, 0, 0, -2),     # 6 pair tiles cut along K over all pairs: 1-2 k blocks each, ragged N and K
    (640, 264, 2112, 0, 1, -1),     # fewer tiles than SMs: K splits finished in-kernel
    (4160, 1280, 2048, 0, 1, -1),   # 85 pair tiles: one whole wave + a stream-K tail of 11 tiles
    (300, 520, 200, 0, 0, 1),       # plain schedule, ragged M and K
])
@pytest.mark.parametrize("epi", [1, 2, 3, 4])
def test_gemm_fused_epilogues_under_each_schedule(M, N, K, a_mn, b_mn, splits, epi):
    """Bias, bias + residual, bias + GELU (gelu' and gelu from one tanh) and the
    GELU' backward with its per-32-row column sums, under the plain, in-kernel
    split and stream-K schedules: a partial-sum finish runs the same epilogue,
    and the epilogue's operand prefetch skips the partial-only fragments."""
    got, ref = _epilogue_case(M + N + K + epi, M, N, K, a_mn, b_mn, epi, splits)
    for k, r in ref.items():
        g = got[k]
        assert np.isfinite(g).all(), k
        if k == "colpart":
            # fp32 sums of fp32 products: rounding of K-long dot products and 32-row sums
            assert rel_l2(g, r) < 1e-5, (k, rel_l2(g, r))
        else:
            # bf16 output (2^-9) plus the hardware tanh (about 2^-11 relative)
            assert rel_l2(g, r) < 4e-3, (k, rel_l2(g, r))


def test_gemm_bounded_wait_expires_and_context_survives():
    """With the producer told to skip its first stage, the MMA thread's bounded
    wait runs out (about 2 s): the call reports GPT2_E_TIMEOUT, the kernel drains
    and returns, and the next GEMM on the same context is correct."""
    import torch
    M, N, K = 256, 512, 1024
    a, b, As, Bs, lda, ldb = _operands(17, M, N, K, 0, 0)
    A, B = to_dev(As), to_dev(Bs)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = binding.lib()
    old = lib.gpt2_test_set_gemm_poison(1)
    try:
        r = lib.gemm_bf16_status(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, lda, ldb, N, 0, 0,
                                 1, None, 0, st.data_ptr(), None)
    finally:
        lib.gpt2_test_set_gemm_poison(old)
    assert r == binding.GPT2_E_TIMEOUT
    r = lib.gemm_bf16_status(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, lda, ldb, N, 0, 0,
                             1, None, 0, st.data_ptr(), None)
    assert r == binding.GPT2_OK
    ref = a.astype(np.float64) @ b.astype(np.float64).T
    assert rel_l2(to_np(D), ref) < 4e-3
