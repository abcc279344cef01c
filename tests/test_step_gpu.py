"""Full training-step parity through the C ABI against the oracle:
forward + mean CE + backward + global-norm clip + AdamW.

fp32 mode (the tiny GPT step): loss within 1e-4 relative, every parameter
gradient within 1e-4 relative L2, post-AdamW weights within 1e-4.
bf16 mode: loss within 1e-2 relative, gradients within 3e-2 relative L2,
post-AdamW weights within 1e-2 relative L2 (the oracle runs in float64 on the
same bf16-rounded weights and tokens)."""
import numpy as np
import pytest

from oracle import gpt2_oracle as O
from pretraining_step_train_b300 import binding, synth
from tests._helpers import rel_l2, to_dev

pytestmark = pytest.mark.gpu

LR, B1, B2, EPS, WD, CLIP = 6e-4, 0.9, 0.95, 1e-8, 0.1, 1.0


def _gpu_step(cfg, B, prec, flat, tok, tgt, steps=1):
    s = binding.Step(cfg.L, cfg.H, cfg.C, cfg.V, cfg.Vpad, cfg.T, B, precision=prec)
    s.set_params(flat)
    td, gd = to_dev(tok, "i32"), to_dev(tgt, "i32")
    out = []
    for t in range(1, steps + 1):
        loss = s.forward(td, gd)
        s.backward()
        grads = s.get(binding.GPT2_GRADS)
        norm = s.clip_adamw(LR, B1, B2, EPS, WD, CLIP, t)
        out.append(dict(loss=loss, grads=grads, norm=norm, master=s.get(binding.GPT2_MASTER),
                        params=s.get(binding.GPT2_PARAMS), m=s.get(binding.GPT2_ADAM_M)))
    s.close()
    return out


ZERO_INIT = ("ln1b", "qkvb", "attprojb", "ln2b", "fcb", "fcprojb", "lnfb")


def _compare(cfg, P, res, ref, loss_tol, grad_tol, w_tol, flat):
    """Loss, every gradient tensor, the norm, and the post-AdamW weights.

    Weights: relative L2 over the whole parameter vector and over every tensor
    that does not start at zero.  A zero-initialised tensor holds only the
    first AdamW update, about -lr * sign(g), which is ill-conditioned where
    g sits at the rounding level (the key-bias gradient is exactly zero in
    exact arithmetic because softmax ignores a per-query shift); those
    tensors are compared on the elements whose gradient is well above it."""
    L, C, Vpad, T = cfg.L, cfg.C, cfg.Vpad, cfg.T
    assert abs(res["loss"] - ref["loss"]) / abs(ref["loss"]) < loss_tol, (res["loss"], ref["loss"])
    G = synth.unflatten_params(res["grads"], L, C, Vpad, T)
    worst = {k: rel_l2(G[k], ref["grads"][k]) for k in G}
    assert max(worst.values()) < grad_tol, worst
    assert abs(res["norm"] - ref["norm"]) / ref["norm"] < grad_tol
    ref_flat = np.concatenate([np.asarray(ref["params"][k]).reshape(-1) for k, _ in synth.param_shapes(L, C, Vpad, T)])
    assert rel_l2(res["master"], ref_flat) < w_tol
    W = synth.unflatten_params(res["master"], L, C, Vpad, T)
    for k in W:
        g = np.abs(ref["grads"][k])
        g_rms = np.sqrt(np.mean(g ** 2)) + 1e-30
        w_rms = np.sqrt(np.mean(np.asarray(P[k], np.float64) ** 2))
        if k in ZERO_INIT:
            big = g > 100 * grad_tol * g_rms
            if big.any():
                assert rel_l2(W[k][big], ref["params"][k][big]) < w_tol, k
        elif LR > 0.1 * w_rms:
            # the first update (about lr * sign(g)) is over a tenth of the weights: where |g|
            # sits near the rounding level its sign, and so the update, is not determined
            keep = g > 0.1 * g_rms
            assert rel_l2(W[k][keep], ref["params"][k][keep]) < w_tol, k
        else:
            assert rel_l2(W[k], ref["params"][k]) < w_tol, k
    return worst


def test_tiny_fp32_step_parity():
    """The tiny GPT step: L=4, H=4, C=64, V=256 (no padding), T=64, B=4, fp32."""
    L, H, C, V, Vpad, T, B = 4, 4, 64, 256, 256, 64, 4
    cfg = O.Config(L, H, C, V, Vpad, T)
    P = synth.init_params(0, L, C, V, Vpad, T)
    tok, tgt = synth.iid_token_batch(1, B, T, V)
    flat = synth.flatten_params(P, L, C, Vpad, T)
    res = _gpu_step(cfg, B, binding.GPT2_FP32, flat, tok, tgt)[0]
    ref = O.train_step(P, tok, tgt, cfg, lr=LR, t=1, beta1=B1, beta2=B2, eps=EPS, wd=WD, max_norm=CLIP)
    _compare(cfg, P, res, ref, 1e-4, 1e-4, 1e-4, flat)


def test_tiny_fp32_two_steps_moments():
    L, H, C, V, Vpad, T, B = 2, 2, 32, 64, 64, 16, 2
    cfg = O.Config(L, H, C, V, Vpad, T)
    P = synth.init_params(3, L, C, V, Vpad, T)
    tok, tgt = synth.iid_token_batch(4, B, T, V)
    flat = synth.flatten_params(P, L, C, Vpad, T)
    res = _gpu_step(cfg, B, binding.GPT2_FP32, flat, tok, tgt, steps=2)
    r1 = O.train_step(P, tok, tgt, cfg, lr=LR, t=1, beta1=B1, beta2=B2, eps=EPS, wd=WD, max_norm=CLIP)
    r2 = O.train_step(r1["params"], tok, tgt, cfg, lr=LR, t=2, M_=r1["m"], V_=r1["v"], beta1=B1, beta2=B2,
                      eps=EPS, wd=WD, max_norm=CLIP)
    _compare(cfg, r1["params"], res[1], r2, 1e-4, 1e-4, 1e-4, flat)


@pytest.mark.parametrize("L,H,C,V,Vpad,T,B", [(2, 2, 128, 1000, 1024, 128, 2), (1, 1, 64, 250, 256, 200, 1)])
def test_bf16_step_parity_small(L, H, C, V, Vpad, T, B):
    cfg = O.Config(L, H, C, V, Vpad, T)
    P = synth.init_params(5, L, C, V, Vpad, T, bf16_representable=True)
    tok, tgt = synth.token_batch(6, B, T, V)
    flat = synth.flatten_params(P, L, C, Vpad, T)
    res = _gpu_step(cfg, B, binding.GPT2_BF16, flat, tok, tgt)[0]
    ref = O.train_step(P, tok, tgt, cfg, lr=LR, t=1, beta1=B1, beta2=B2, eps=EPS, wd=WD, max_norm=CLIP)
    _compare(cfg, P, res, ref, 1e-2, 3e-2, 1e-2, flat)
    # the working bf16 copy is the round-to-nearest-even of the fp32 master copy
    np.testing.assert_array_equal(res["params"], synth.round_to_bf16(res["master"]))


@pytest.mark.slow
def test_bf16_step_parity_124m_shapes():
    """GPT-2 124M shapes (L=12, H=12, C=768, V=50257 -> 50304, T=1024) at B=1."""
    L, H, C, V, Vpad, T, B = 12, 12, 768, 50257, 50304, 1024, 1
    cfg = O.Config(L, H, C, V, Vpad, T)
    P = synth.init_params(7, L, C, V, Vpad, T, bf16_representable=True)
    tok, tgt = synth.token_batch(8, B, T, V)
    flat = synth.flatten_params(P, L, C, Vpad, T)
    res = _gpu_step(cfg, B, binding.GPT2_BF16, flat, tok, tgt)[0]
    ref = O.train_step(P, tok, tgt, cfg, lr=LR, t=1, beta1=B1, beta2=B2, eps=EPS, wd=WD, max_norm=CLIP,
                       dtype=np.float64)
    worst = _compare(cfg, P, res, ref, 1e-2, 3e-2, 1e-2, flat)
    print("worst grad rel L2:", max(worst.items(), key=lambda kv: kv[1]))


def _oracle_sequence_grads(args):
    """Oracle forward + backward of one sequence (float32), run in a worker."""
    shape, seed, b, tok, tgt = args
    L, H, C, V, Vpad, T = shape
    P = _worker_params(shape, seed)
    loss, cache = O.forward(P, tok, tgt, O.Config(L, H, C, V, Vpad, T), dtype=np.float32)
    return b, loss, O.backward(cache, O.Config(L, H, C, V, Vpad, T))


_WORKER_P = {}


def _worker_params(shape, seed):
    key = (shape, seed)
    if key not in _WORKER_P:
        L, H, C, V, Vpad, T = shape
        _WORKER_P.clear()
        _WORKER_P[key] = synth.init_params(seed, L, C, V, Vpad, T, bf16_representable=True)
    return _WORKER_P[key]


def _oracle_batch_step(shape, seed, tok, tgt, workers=4):
    """The oracle's step on B sequences, evaluated one sequence at a time.

    The loss is the mean over all B*T positions and every sequence has T of
    them, so the batch loss is the mean of the per-sequence losses and the batch
    gradient the mean of the per-sequence gradients (linearity of the mean); the
    clip and AdamW then run once on that gradient, as in the oracle's own step.
    The sequences run in a spawn-started process pool (no fork after CUDA)."""
    import multiprocessing as mp
    L, H, C, V, Vpad, T = shape
    B = tok.shape[0]
    jobs = [(shape, seed, b, tok[b:b + 1], tgt[b:b + 1]) for b in range(B)]
    G, losses = None, [0.0] * B
    with mp.get_context("spawn").Pool(min(workers, B)) as pool:
        for b, loss, g in pool.imap_unordered(_oracle_sequence_grads, jobs):
            losses[b] = loss
            if G is None:
                G = {k: np.zeros(v.shape, np.float64) for k, v in g.items()}
            for k in G:
                G[k] += g[k]
    G = {k: v / B for k, v in G.items()}
    P = synth.init_params(seed, L, C, V, Vpad, T, bf16_representable=True)
    zeros = {k: np.zeros(v.shape, np.float64) for k, v in G.items()}
    norm, nP, _, _ = O.clip_adamw({k: v.astype(np.float64) for k, v in P.items()}, G, zeros, zeros, 1, LR,
                                  beta1=B1, beta2=B2, eps=EPS, wd=WD, max_norm=CLIP)
    return dict(loss=float(np.mean(losses)), grads=G, norm=norm, params=nP), P


@pytest.mark.slow
def test_bf16_step_parity_124m_bench_batch():
    """The step the benchmark times: GPT-2 124M shapes at B=16, T=1024 (M = 16384,
    so every GEMM takes its production schedule: stream-K tails, in-kernel split
    finishes, 8-split weight gradients with the separate reduction, the
    persistent LayerNorm backward over 16384 rows, the CE merge over 786 column
    groups).  Loss, every gradient tensor, the norm and the post-AdamW master
    weights against the oracle (float32, per sequence, combined exactly)."""
    L, H, C, V, Vpad, T, B = 12, 12, 768, 50257, 50304, 1024, 16
    cfg = O.Config(L, H, C, V, Vpad, T)
    tok, tgt = synth.token_batch(42, B, T, V)
    ref, P = _oracle_batch_step((L, H, C, V, Vpad, T), 43, tok, tgt)
    flat = synth.flatten_params(P, L, C, Vpad, T)
    res = _gpu_step(cfg, B, binding.GPT2_BF16, flat, tok, tgt)[0]
    worst = _compare(cfg, P, res, ref, 1e-2, 3e-2, 1e-2, flat)
    print("worst grad rel L2:", max(worst.items(), key=lambda kv: kv[1]))


@pytest.mark.slow
@pytest.mark.parametrize("L,H,C,B", [(24, 16, 1024, 1), (2, 25, 1600, 1)])
def test_bf16_step_parity_350m_and_d48_shapes(L, H, C, B):
    """GPT-2 350M shapes (L=24, H=16, C=1024) and the d48 model's width (C=1600,
    H=25 heads of 64: N not a multiple of the 256-wide GEMM tile, 25 k blocks,
    LayerNorm rows of 200 vectors) at T=1024, against the oracle."""
    V, Vpad, T = 50257, 50304, 1024
    cfg = O.Config(L, H, C, V, Vpad, T)
    P = synth.init_params(71 + L, L, C, V, Vpad, T, bf16_representable=True)
    tok, tgt = synth.token_batch(72 + L, B, T, V)
    flat = synth.flatten_params(P, L, C, Vpad, T)
    res = _gpu_step(cfg, B, binding.GPT2_BF16, flat, tok, tgt)[0]
    ref = O.train_step(P, tok, tgt, cfg, lr=LR, t=1, beta1=B1, beta2=B2, eps=EPS, wd=WD, max_norm=CLIP,
                       dtype=np.float32)
    worst = _compare(cfg, P, res, ref, 1e-2, 3e-2, 1e-2, flat)
    print("worst grad rel L2:", max(worst.items(), key=lambda kv: kv[1]))


@pytest.mark.parametrize("prec,tol", [(binding.GPT2_BF16, (1e-2, 3e-2, 1e-2)), (binding.GPT2_FP32, (1e-4, 1e-4, 1e-4))])
def test_step_parity_without_clipping(prec, tol):
    """max_norm far above the gradient norm: the clip scale is exactly 1 and the
    update is AdamW on the raw gradient."""
    L, H, C, V, Vpad, T, B = (2, 2, 128, 1000, 1024, 128, 2) if prec == binding.GPT2_BF16 else (2, 2, 64, 256, 256, 64, 2)
    cfg = O.Config(L, H, C, V, Vpad, T)
    P = synth.init_params(81, L, C, V, Vpad, T, bf16_representable=prec == binding.GPT2_BF16)
    tok, tgt = synth.token_batch(82, B, T, V)
    flat = synth.flatten_params(P, L, C, Vpad, T)
    big = 1e4
    s = binding.Step(L, H, C, V, Vpad, T, B, precision=prec)
    s.set_params(flat)
    loss = s.forward(to_dev(tok, "i32"), to_dev(tgt, "i32"))
    s.backward()
    grads = s.get(binding.GPT2_GRADS)
    norm = s.clip_adamw(LR, B1, B2, EPS, WD, big, 1)
    res = dict(loss=loss, grads=grads, norm=norm, master=s.get(binding.GPT2_MASTER))
    s.close()
    ref = O.train_step(P, tok, tgt, cfg, lr=LR, t=1, beta1=B1, beta2=B2, eps=EPS, wd=WD, max_norm=big)
    assert O.clip_scale(ref["norm"], big) == 1.0 and ref["norm"] > CLIP
    _compare(cfg, P, res, ref, *tol, flat)


@pytest.mark.parametrize("rc", [1, 2])
@pytest.mark.parametrize("prec", [binding.GPT2_BF16, binding.GPT2_FP32])
def test_activation_recompute_step_parity(rc, prec):
    """Recompute levels 1 (GELU) and 2 (GELU and LayerNorm outputs): the step
    matches the oracle at the precision's tolerances, and matches the step that
    keeps every activation (to fp32 rounding in fp32 mode, where the recomputed
    values are the kept ones; within bf16 rounding in bf16 mode, where gelu and
    gelu' come from the rounded h)."""
    bf = prec == binding.GPT2_BF16
    L, H, C, V, Vpad, T, B = (2, 2, 128, 1000, 1024, 128, 2) if bf else (2, 2, 64, 256, 256, 64, 2)
    cfg = O.Config(L, H, C, V, Vpad, T)
    P = synth.init_params(91 + rc, L, C, V, Vpad, T, bf16_representable=bf)
    tok, tgt = synth.token_batch(92 + rc, B, T, V)
    flat = synth.flatten_params(P, L, C, Vpad, T)
    out = {}
    for r in (0, rc):
        s = binding.Step(L, H, C, V, Vpad, T, B, precision=prec, recompute=r)
        s.set_params(flat)
        loss = s.forward(to_dev(tok, "i32"), to_dev(tgt, "i32"))
        s.backward()
        grads = s.get(binding.GPT2_GRADS)
        norm = s.clip_adamw(LR, B1, B2, EPS, WD, CLIP, 1)
        out[r] = dict(loss=loss, grads=grads, norm=norm, master=s.get(binding.GPT2_MASTER))
        s.close()
    ref = O.train_step(P, tok, tgt, cfg, lr=LR, t=1, beta1=B1, beta2=B2, eps=EPS, wd=WD, max_norm=CLIP)
    tol = (1e-2, 3e-2, 1e-2) if bf else (1e-4, 1e-4, 1e-4)
    _compare(cfg, P, out[rc], ref, *tol, flat)
    if bf:
        assert abs(out[rc]["loss"] - out[0]["loss"]) < 1e-3 * abs(out[0]["loss"])
        assert rel_l2(out[rc]["grads"], out[0]["grads"]) < 1e-2
    else:
        assert out[rc]["loss"] == out[0]["loss"]  # the forward pass computes the same values
        assert rel_l2(out[rc]["grads"], out[0]["grads"]) < 1e-6


def test_bf16_step_deterministic():
    L, H, C, V, Vpad, T, B = 2, 2, 128, 1000, 1024, 128, 2
    cfg = O.Config(L, H, C, V, Vpad, T)
    P = synth.init_params(9, L, C, V, Vpad, T, bf16_representable=True)
    tok, tgt = synth.token_batch(10, B, T, V)
    flat = synth.flatten_params(P, L, C, Vpad, T)
    a = _gpu_step(cfg, B, binding.GPT2_BF16, flat, tok, tgt)[0]
    b = _gpu_step(cfg, B, binding.GPT2_BF16, flat, tok, tgt)[0]
    assert a["loss"] == b["loss"]
    np.testing.assert_array_equal(a["grads"], b["grads"])
    np.testing.assert_array_equal(a["master"], b["master"])


def test_call_order_and_host_step():
    L, H, C, V, Vpad, T, B = 1, 1, 64, 250, 256, 64, 2
    cfg = O.Config(L, H, C, V, Vpad, T)
    P = synth.init_params(11, L, C, V, Vpad, T, bf16_representable=True)
    tok, tgt = synth.token_batch(12, B, T, V)
    s = binding.Step(L, H, C, V, Vpad, T, B, precision=binding.GPT2_BF16)
    s.set_params(synth.flatten_params(P, L, C, Vpad, T))
    assert binding.lib().gpt2_backward(s.h) == binding.GPT2_E_STATE
    loss, norm = s.train_step_host(tok, tgt)
    ref = O.train_step(P, tok, tgt, cfg, lr=LR, t=1)
    assert abs(loss - ref["loss"]) / ref["loss"] < 1e-2
    assert abs(norm - ref["norm"]) / ref["norm"] < 3e-2
    assert binding.lib().gpt2_clip_adamw(s.h, LR, B1, B2, EPS, WD, CLIP, 1, None) == binding.GPT2_E_STATE
    # an out-of-range target is clamped and reported
    bad = tgt.copy()
    bad[0, 0] = V + 5
    import ctypes as ct
    lossv = ct.c_float()
    tok_d, bad_d = to_dev(tok, "i32"), to_dev(bad, "i32")
    r = binding.lib().gpt2_forward(s.h, tok_d.data_ptr(), bad_d.data_ptr(), ct.byref(lossv))
    assert r == binding.GPT2_E_TOKEN
    assert s.sync_status() == binding.GPT2_OK  # the status word was read and cleared
    s.close()


def test_host_step_graph_matches_device_steps():
    """gpt2_train_step_host replays one CUDA graph captured on its first call; its
    hyperparameters and tokens arrive through pinned staging copies inside the
    graph.  Three steps with a different learning rate, step index and batch each
    must equal, bit for bit, the same steps issued through forward / backward /
    clip_adamw; a clamped target is reported by the step that saw it and the
    status is clear again on the next."""
    L, H, C, V, Vpad, T, B = 2, 2, 128, 1000, 1024, 128, 2
    P = synth.init_params(21, L, C, V, Vpad, T, bf16_representable=True)
    flat = synth.flatten_params(P, L, C, Vpad, T)
    a = binding.Step(L, H, C, V, Vpad, T, B, precision=binding.GPT2_BF16)
    b = binding.Step(L, H, C, V, Vpad, T, B, precision=binding.GPT2_BF16)
    a.set_params(flat)
    b.set_params(flat)
    for i, lr in enumerate((LR, 0.5 * LR, 2.0 * LR)):
        tok, tgt = synth.token_batch(30 + i, B, T, V)
        la, na = a.train_step_host(tok, tgt, lr=lr, beta1=B1, beta2=B2, eps=EPS, weight_decay=WD,
                                   max_norm=CLIP, t=i + 1)
        lb = b.forward(to_dev(tok, "i32"), to_dev(tgt, "i32"))
        b.backward()
        nb = b.clip_adamw(lr=lr, beta1=B1, beta2=B2, eps=EPS, weight_decay=WD, max_norm=CLIP, t=i + 1)
        assert la == lb and na == nb, (i, la, lb, na, nb)
    for which in (0, 2, 3, 4):  # working and master parameters, AdamW m and v
        np.testing.assert_array_equal(a.get(which), b.get(which))
    tok, tgt = synth.token_batch(40, B, T, V)
    bad = tgt.copy()
    bad[1, 3] = V + 7
    with pytest.raises(binding.GPT2Error) as ei:
        a.train_step_host(tok, bad, t=4)
    assert ei.value.status == binding.GPT2_E_TOKEN
    a.train_step_host(tok, tgt, t=5)
    a.close()
    b.close()


@pytest.mark.parametrize("prec,grad_tol,w_tol", [(binding.GPT2_BF16, 3e-2, 1e-2), (binding.GPT2_FP32, 1e-4, 1e-4)])
def test_grad_accumulation_equals_the_large_batch(prec, grad_tol, w_tol):
    """Two micro-batches of B sequences, each gradient accumulated with scale 1/2,
    then one clip + AdamW, against the oracle's step on the 2B sequences at once:
    the gradient of the mean loss over 2B rows is the mean of the two
    micro-batch gradients."""
    L, H, C, V, Vpad, T, B = (2, 2, 128, 1000, 1024, 128, 2) if prec == binding.GPT2_BF16 else (2, 2, 64, 256, 256, 64, 2)
    cfg = O.Config(L, H, C, V, Vpad, T)
    P = synth.init_params(51, L, C, V, Vpad, T, bf16_representable=prec == binding.GPT2_BF16)
    tok, tgt = synth.token_batch(52, 2 * B, T, V)
    flat = synth.flatten_params(P, L, C, Vpad, T)
    s = binding.Step(L, H, C, V, Vpad, T, B, precision=prec)
    s.set_params(flat)
    # the accumulated step must follow backward; AdamW on the accumulator must follow an accumulate
    assert binding.lib().gpt2_grad_accumulate(s.h, 1, 0.5) == binding.GPT2_E_STATE
    losses = []
    for i in range(2):
        losses.append(s.forward(to_dev(tok[i * B:(i + 1) * B], "i32"), to_dev(tgt[i * B:(i + 1) * B], "i32")))
        s.backward()
        s.grad_accumulate(i == 0, 0.5)
    acc = s.get(binding.GPT2_GRAD_ACC)
    norm = s.clip_adamw_accumulated(LR, B1, B2, EPS, WD, CLIP, 1)
    assert binding.lib().gpt2_clip_adamw_accumulated(s.h, LR, B1, B2, EPS, WD, CLIP, 1, None) == binding.GPT2_E_STATE
    res = dict(loss=0.5 * (losses[0] + losses[1]), grads=acc, norm=norm, master=s.get(binding.GPT2_MASTER))
    s.close()
    ref = O.train_step(P, tok, tgt, cfg, lr=LR, t=1, beta1=B1, beta2=B2, eps=EPS, wd=WD, max_norm=CLIP)
    _compare(cfg, P, res, ref, 1e-2 if prec == binding.GPT2_BF16 else 1e-4, grad_tol, w_tol, flat)
