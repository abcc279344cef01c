"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against what the pages print, a closed form, an
invariant, brute force (finite differences) or an independent library routine
(torch CPU autograd / functional ops / torch.optim.AdamW), so that a dropped
term, a wrong sign or index, or a transposed operand fails at least one.
"""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import gpt2_oracle as O
from pretraining_step_train_b300 import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))


def tiny_case(seed=3, L=2, H=2, C=16, V=32, Vpad=48, T=8, B=2, zero_bias=False):
    cfg = O.Config(L, H, C, V, Vpad, T)
    P = synth.init_params(seed, L, C, V, Vpad, T)
    rng = np.random.default_rng(seed)
    # perturb biases and LN affine so every term of the backward is exercised
    if not zero_bias:
        for k in P:
            if k.endswith("b") or k in ("ln1w", "ln2w", "lnfw"):
                P[k] = (P[k] + 0.1 * rng.standard_normal(P[k].shape)).astype(np.float32)
    tok, tgt = synth.iid_token_batch(seed, B, T, V)
    return cfg, {k: v.astype(np.float64) for k, v in P.items()}, tok, tgt


# ----------------------------------------------------------- printed numbers
def test_param_count_matches_printed_d48():
    g = GOLD["d48_num_parameters"]
    c = g["config"]
    n = O.num_params(c["L"], c["C"], c["Vpad"], c["T"])
    assert n == g["value"]
    assert 2 * n == GOLD["d48_param_bytes_bf16"]["value"]


def test_param_count_124m_350m():
    assert O.num_params(12, 768, 50304, 1024) == 124475904
    assert O.num_params(12, 768, 50257, 1024) == 124439808
    assert O.num_params(24, 1024, 50304, 1024) == 354871296


def test_init_loss_closed_form_vs_printed():
    # E[loss] at init ~= ln V + C sigma^2 / 2 (logits ~ N(0, C sigma^2) after a unit LN)
    V = GOLD["vocab_padding"]["V"]
    assert abs(np.log(V) - GOLD["random_init_loss_small"]["value"]) < 0.01
    cf = np.log(V) + 1600 * 0.02 ** 2 / 2
    assert abs(cf - GOLD["d48_init_val_loss"]["value"]) < 0.03
    assert abs(cf - GOLD["d48_step1_loss"]["value"]) < 0.03


@pytest.mark.slow
def test_init_loss_124m_shapes():
    """Oracle forward at GPT-2 124M shapes lands on ln V + C sigma^2/2 = 10.977."""
    L, H, C, V, Vpad, T, B = 12, 12, 768, 50257, 50304, 256, 4
    P = synth.init_params(11, L, C, V, Vpad, 1024)
    tok, tgt = synth.iid_token_batch(12, B, T, V)
    loss, _ = O.forward(P, tok, tgt, O.Config(L, H, C, V, Vpad, 1024), dtype=np.float32)
    expect = np.log(V) + C * 0.02 ** 2 / 2
    assert abs(loss - expect) < 0.06, (loss, expect)
    assert abs(loss - np.log(V)) < 0.25


# ----------------------------------------------------------- init recipe
def test_init_recipe():
    L, C, V, Vpad, T = 4, 64, 250, 256, 64
    P = synth.init_params(5, L, C, V, Vpad, T)
    assert np.all(P["wte"][V:] == 0)
    assert abs(P["wte"][:V].std() - 0.02) < 0.001
    assert abs(P["qkvw"].std() - 0.02) < 0.001
    for k in ("attprojw", "fcprojw"):
        assert abs(P[k].std() - 0.02 / np.sqrt(2 * L)) < 0.0006
    assert np.all(P["ln1w"] == 1) and np.all(P["ln1b"] == 0) and np.all(P["lnfw"] == 1)
    assert np.all(P["qkvb"] == 0) and np.all(P["fcprojb"] == 0)


# ----------------------------------------------------------- gradients
def _loss(P, tok, tgt, cfg):
    return O.forward(P, tok, tgt, cfg)[0]


def test_finite_differences_all_tensors():
    """Central differences (h=1e-5, float64) along random directions and on
    random single elements of every tensor agree with the analytic gradient."""
    cfg, P, tok, tgt = tiny_case()
    loss, cache = O.forward(P, tok, tgt, cfg)
    G = O.backward(cache, cfg)
    rng = np.random.default_rng(0)
    h = 1e-5
    for name in P:
        if name == "wpe":
            pass
        for trial in range(2):
            d = rng.standard_normal(P[name].shape)
            if name == "wte":
                d[cfg.V:] = 0.0
            Pp = dict(P); Pp[name] = P[name] + h * d
            Pm = dict(P); Pm[name] = P[name] - h * d
            fd = (_loss(Pp, tok, tgt, cfg) - _loss(Pm, tok, tgt, cfg)) / (2 * h)
            an = float(np.sum(G[name] * d))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)) + 1e-9, (name, fd, an)
        flat = P[name].reshape(-1)
        for idx in rng.choice(flat.size, size=min(4, flat.size), replace=False):
            e = np.zeros(flat.size); e[idx] = 1.0
            e = e.reshape(P[name].shape)
            Pp = dict(P); Pp[name] = P[name] + h * e
            Pm = dict(P); Pm[name] = P[name] - h * e
            fd = (_loss(Pp, tok, tgt, cfg) - _loss(Pm, tok, tgt, cfg)) / (2 * h)
            an = G[name].reshape(-1)[idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)) + 1e-9, (name, idx, fd, an)


def _torch_model_loss(Pt, tok, tgt, cfg):
    """Independent GPT-2 forward from torch.nn.functional library ops (CPU)."""
    B, T = tok.shape
    C, H, d = cfg.C, cfg.H, cfg.d
    tok_t = torch.from_numpy(tok.astype(np.int64))
    x = F.embedding(tok_t, Pt["wte"]) + Pt["wpe"][:T]
    for l in range(cfg.L):
        h1 = F.layer_norm(x, (C,), Pt["ln1w"][l], Pt["ln1b"][l], eps=1e-5)
        qkv = F.linear(h1, Pt["qkvw"][l], Pt["qkvb"][l])
        q, k, v = qkv.split(C, dim=-1)
        q, k, v = (t.view(B, T, H, d).transpose(1, 2) for t in (q, k, v))
        y = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        y = y.transpose(1, 2).reshape(B, T, C)
        x = x + F.linear(y, Pt["attprojw"][l], Pt["attprojb"][l])
        h2 = F.layer_norm(x, (C,), Pt["ln2w"][l], Pt["ln2b"][l], eps=1e-5)
        x = x + F.linear(F.gelu(F.linear(h2, Pt["fcw"][l], Pt["fcb"][l]), approximate="tanh"),
                         Pt["fcprojw"][l], Pt["fcprojb"][l])
    x = F.layer_norm(x, (C,), Pt["lnfw"], Pt["lnfb"], eps=1e-5)
    logits = F.linear(x, Pt["wte"][: cfg.V])  # only the real vocab rows take part
    return F.cross_entropy(logits.reshape(B * T, cfg.V), torch.from_numpy(tgt.astype(np.int64)).reshape(-1))


def test_against_torch_autograd():
    cfg, P, tok, tgt = tiny_case(L=3, H=4, C=32, V=40, Vpad=64, T=12, B=3)
    loss, cache = O.forward(P, tok, tgt, cfg)
    G = O.backward(cache, cfg)
    Pt = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in P.items()}
    lt = _torch_model_loss(Pt, tok, tgt, cfg)
    lt.backward()
    assert abs(lt.item() - loss) < 1e-12 * abs(loss)
    for k in P:
        ref = Pt[k].grad.numpy()
        err = np.linalg.norm(G[k] - ref) / max(np.linalg.norm(ref), 1e-30)
        assert err < 1e-10, (k, err)


# ----------------------------------------------------------- invariants
def test_causality_bit_identical():
    cfg, P, tok, tgt = tiny_case(L=2, H=2, C=16, V=32, Vpad=48, T=10, B=2)
    _, c1 = O.forward(P, tok, tgt, cfg)
    t = 6
    tok2 = tok.copy()
    tok2[:, t + 1:] = (tok2[:, t + 1:] + 7) % cfg.V
    _, c2 = O.forward(P, tok2, tgt, cfg)
    z1 = c1["z"].reshape(2, 10, -1)[:, : t + 1]
    z2 = c2["z"].reshape(2, 10, -1)[:, : t + 1]
    np.testing.assert_allclose(z1, z2, rtol=1e-14, atol=0)
    assert not np.allclose(c1["z"].reshape(2, 10, -1)[:, t + 1:], c2["z"].reshape(2, 10, -1)[:, t + 1:])


def test_pad_rows_never_change_loss():
    cfg, P, tok, tgt = tiny_case()
    l1, c1 = O.forward(P, tok, tgt, cfg)
    G1 = O.backward(c1, cfg)
    P2 = dict(P)
    P2["wte"] = P["wte"].copy()
    P2["wte"][cfg.V:] = np.random.default_rng(1).standard_normal((cfg.Vpad - cfg.V, cfg.C))
    l2, c2 = O.forward(P2, tok, tgt, cfg)
    G2 = O.backward(c2, cfg)
    assert l1 == l2
    for k in G1:
        a, b = G1[k], G2[k]
        if k == "wte":
            a, b = a[: cfg.V], b[: cfg.V]
        np.testing.assert_array_equal(a, b)
    assert np.all(G1["wte"][cfg.V:] == 0)


def test_ce_and_ln_and_attention_invariants():
    cfg, P, tok, tgt = tiny_case()
    _, c = O.forward(P, tok, tgt, cfg)
    dz = O.cross_entropy_backward(c["probs"], tgt.reshape(-1))
    np.testing.assert_allclose(dz.sum(axis=1), 0, atol=1e-15)
    assert np.all(dz[:, cfg.V:] == 0)
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 24)); w = rng.standard_normal(24); b = rng.standard_normal(24)
    y, m, r = O.layernorm_forward(x, w, b)
    dy = rng.standard_normal(x.shape)
    dx, dw, db = O.layernorm_backward(dy, x, w, m, r)
    xhat = (x - m[:, None]) * r[:, None]
    np.testing.assert_allclose(dx.sum(axis=1), 0, atol=1e-12)
    # with eps > 0, mean(xhat^2) = var / (var + eps) < 1, so the identity carries that factor
    g = dy * w
    np.testing.assert_allclose((dx * xhat).sum(axis=1),
                               r * (g * xhat).sum(axis=1) * (1 - (xhat ** 2).mean(axis=1)), atol=1e-12)
    q, k, v = (rng.standard_normal((2, 3, 7, 4)) for _ in range(3))
    o, p, lse = O.attention_forward(q, k, v, 0.5)
    do = rng.standard_normal(o.shape)
    dp = np.einsum("bhid,bhjd->bhij", do, v)
    ds = p * (dp - (p * dp).sum(-1, keepdims=True))
    np.testing.assert_allclose(ds.sum(-1), 0, atol=1e-12)
    np.testing.assert_allclose((p * dp).sum(-1), (do * o).sum(-1), rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------- op-level library pins
def test_layernorm_vs_torch():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 40)) * 3 + 1; w = rng.standard_normal(40); b = rng.standard_normal(40)
    y, _, _ = O.layernorm_forward(x, w, b)
    yt = F.layer_norm(torch.tensor(x), (40,), torch.tensor(w), torch.tensor(b), eps=1e-5).numpy()
    np.testing.assert_allclose(y, yt, rtol=1e-12, atol=1e-12)


def test_attention_vs_torch_sdpa_and_lse():
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((2, 3, 9, 8)) for _ in range(3))
    o, p, lse = O.attention_forward(q, k, v, 1 / np.sqrt(8))
    ot = F.scaled_dot_product_attention(*(torch.tensor(a) for a in (q, k, v)), is_causal=True).numpy()
    np.testing.assert_allclose(o, ot, rtol=1e-12, atol=1e-12)
    s = np.einsum("bhid,bhjd->bhij", q, k) / np.sqrt(8)
    s = np.where(np.triu(np.ones((9, 9), bool), 1), -np.inf, s)
    lse_t = torch.logsumexp(torch.tensor(s), dim=-1).numpy()
    np.testing.assert_allclose(lse, lse_t, rtol=1e-12)


def test_attention_special_case_T1_is_v():
    rng = np.random.default_rng(6)
    q, k, v = (rng.standard_normal((2, 1, 1, 5)) for _ in range(3))
    o, p, lse = O.attention_forward(q, k, v, 0.3)
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(lse[..., 0], (q * k).sum(-1)[..., 0] * 0.3, rtol=1e-14)


def test_attention_backward_vs_torch():
    rng = np.random.default_rng(7)
    q, k, v, do = (rng.standard_normal((2, 2, 6, 4)) for _ in range(4))
    o, p, lse = O.attention_forward(q, k, v, 0.5)
    dq, dk, dv = O.attention_backward(do, q, k, v, p, 0.5)
    qt, kt, vt = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    F.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=0.5).backward(torch.tensor(do))
    for a, b in ((dq, qt), (dk, kt), (dv, vt)):
        np.testing.assert_allclose(a, b.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_cross_entropy_vs_torch():
    rng = np.random.default_rng(8)
    M, V, Vpad = 7, 11, 16
    z = rng.standard_normal((M, Vpad)) * 2
    tgt = rng.integers(0, V, M)
    loss, lse, probs = O.cross_entropy_forward(z, tgt, V)
    lt = F.cross_entropy(torch.tensor(z[:, :V]), torch.tensor(tgt)).item()
    assert abs(loss - lt) < 1e-13
    np.testing.assert_allclose(O.cross_entropy_backward(probs, tgt)[:, :V],
                               (torch.softmax(torch.tensor(z[:, :V]), 1).numpy() - np.eye(V)[tgt]) / M,
                               rtol=1e-12, atol=1e-15)


def test_classifier_fwd_bwd_vs_torch():
    rng = np.random.default_rng(9)
    M, C, V, Vpad = 10, 6, 13, 16
    x = rng.standard_normal((M, C)); w = rng.standard_normal((Vpad, C)) * 0.3
    w[V:] = rng.standard_normal((Vpad - V, C))  # pad rows must not matter
    tgt = rng.integers(0, V, M)
    loss, dx, dw, lse = O.classifier_forward_backward(x, w, tgt, V)
    xt = torch.tensor(x, requires_grad=True); wt = torch.tensor(w, requires_grad=True)
    lt = F.cross_entropy(xt @ wt[:V].T, torch.tensor(tgt))
    lt.backward()
    assert abs(loss - lt.item()) < 1e-13
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-11, atol=1e-14)
    assert np.all(dw[V:] == 0)


def test_gelu_form():
    x = np.linspace(-8, 8, 20001)
    import scipy.special as sp
    exact = 0.5 * x * (1 + sp.erf(x / np.sqrt(2)))
    assert np.abs(O.gelu(x) - exact).max() < 5e-4  # tanh form within its known error
    np.testing.assert_allclose(O.gelu(x) - O.gelu(-x), x, atol=1e-12)
    np.testing.assert_allclose(O.gelu(x), F.gelu(torch.tensor(x), approximate="tanh").numpy(), atol=1e-14)
    h = 1e-6
    np.testing.assert_allclose(O.gelu_grad(x), (O.gelu(x + h) - O.gelu(x - h)) / (2 * h), atol=1e-7)


def test_L0_reduces_to_linear_classifier():
    cfg, P, tok, tgt = tiny_case(L=0)
    loss, cache = O.forward(P, tok, tgt, cfg)
    x0 = P["wte"][tok] + P["wpe"][None, : tok.shape[1]]
    y, _, _ = O.layernorm_forward(x0, P["lnfw"], P["lnfb"])
    l2, _, _, _ = O.classifier_forward_backward(y.reshape(-1, cfg.C), P["wte"], tgt.reshape(-1), cfg.V)
    assert abs(loss - l2) < 1e-14


# ----------------------------------------------------------- optimizer
def test_adamw_vs_torch_optim_three_steps():
    rng = np.random.default_rng(10)
    w0 = rng.standard_normal((5, 4)); gs = [rng.standard_normal((5, 4)) for _ in range(3)]
    wt = torch.tensor(w0, requires_grad=True)
    opt = torch.optim.AdamW([wt], lr=6e-4, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    w, m, v = w0.copy(), np.zeros_like(w0), np.zeros_like(w0)
    for t, g in enumerate(gs, start=1):
        wt.grad = torch.tensor(g)
        opt.step()
        w, m, v = O.adamw_update(w, g, m, v, t, 6e-4, 0.9, 0.95, 1e-8, 0.1)
    np.testing.assert_allclose(w, wt.detach().numpy(), rtol=1e-13, atol=1e-15)


def test_adamw_closed_form_t1():
    rng = np.random.default_rng(11)
    w = rng.standard_normal(100); g = rng.standard_normal(100) * 1e-3
    nw, _, _ = O.adamw_update(w, g, 0 * w, 0 * w, 1, 1e-3, 0.9, 0.95, 1e-8, 0.1)
    np.testing.assert_allclose(nw - w, -1e-3 * (g / (np.abs(g) + 1e-8) + 0.1 * w), rtol=1e-9)


def test_clip_and_decay_set():
    cfg, P, tok, tgt = tiny_case()
    r = O.train_step(P, tok, tgt, cfg, lr=6e-4, t=1)
    G = r["grads"]
    n = O.global_norm(G)
    tt = []
    for g in G.values():
        t = torch.zeros(g.shape, dtype=torch.float64, requires_grad=True)
        t.grad = torch.tensor(g.copy())
        tt.append(t)
    tn = torch.nn.utils.clip_grad_norm_(tt, 1.0).item()
    assert abs(n - tn) < 1e-12 * n
    s = O.clip_scale(n)
    assert abs(np.sqrt(sum(float(np.sum((s * g) ** 2)) for g in G.values())) - min(n, 1.0)) < 1e-12
    # non-decayed tensors with zero gradient stay put; decayed ones shrink by lr*wd*w
    for k in P:
        expect_decay = k in ("wte", "wpe", "qkvw", "attprojw", "fcw", "fcprojw")
        assert (k in O.DECAYED) == expect_decay
    Gz = {k: np.zeros_like(v) for k, v in G.items()}
    Z = {k: np.zeros_like(v) for k, v in G.items()}
    _, nP, _, _ = O.clip_adamw(P, Gz, Z, Z, 1, 1e-2, wd=0.1)
    for k in P:
        expect = P[k] * (1 - 1e-2 * 0.1) if k in O.DECAYED else P[k]
        np.testing.assert_allclose(nP[k], expect, rtol=1e-14, atol=0)


# ----------------------------------------------------------- fp32 fixed-order encoder
def test_encoder_fp32_references():
    rng = np.random.default_rng(12)
    B, T, C, V, Vpad = 3, 5, 4, 6, 8
    tok = rng.integers(0, V, (B, T)).astype(np.int32)
    wte = rng.standard_normal((Vpad, C)).astype(np.float32)
    wpe = rng.standard_normal((T, C)).astype(np.float32)
    x0 = O.encoder_forward_f32(tok, wte, wpe)
    np.testing.assert_array_equal(x0, O.encoder_forward(tok, wte, wpe).astype(np.float32))
    # small-integer gradients make every float32 sum exact: compare with add.at exactly
    dx0 = rng.integers(-8, 9, (B, T, C)).astype(np.float32)
    din = rng.integers(-8, 9, (Vpad, C)).astype(np.float32)
    dwte, dwpe = O.encoder_backward_f32(tok, dx0, din, (T, C))
    ref = din.astype(np.float64).copy()
    np.add.at(ref, tok.reshape(-1), dx0.reshape(-1, C))
    np.testing.assert_array_equal(dwte, ref)
    np.testing.assert_array_equal(dwpe, dx0.sum(axis=0))


def test_encoder_backward_f32_real_data_within_rounding_bound():
    """The fixed-order float32 scatter (runs of 64 positions per id) on real
    values with heavy duplication, against the exact sum (float64 add.at, which
    fixes no order): n float32 additions of any order and grouping stay within
    n * 2^-24 * (|dwte_in| + sum |dx0|) of the exact result, per element, so a
    dropped, doubled or misplaced row fails while the grouping itself is free."""
    B, T, C, V, Vpad = 8, 128, 24, 50, 56
    tok = synth.token_batch(31, B, T, V)[0]
    counts = np.bincount(tok.reshape(-1), minlength=Vpad)
    assert counts.max() > 3 * 64  # the most frequent ids span several runs
    dx0 = synth.normal(32, B * T * C, 1e-3).astype(np.float32).reshape(B, T, C)
    din = synth.normal(33, Vpad * C, 1e-3).astype(np.float32).reshape(Vpad, C)
    dwte, dwpe = O.encoder_backward_f32(tok, dx0, din, (T, C))
    exact = din.astype(np.float64).copy()
    np.add.at(exact, tok.reshape(-1), dx0.reshape(-1, C).astype(np.float64))
    mag = np.abs(din).astype(np.float64)
    np.add.at(mag, tok.reshape(-1), np.abs(dx0).reshape(-1, C).astype(np.float64))
    n = (counts + 1)[:, None]
    err = np.abs(dwte.astype(np.float64) - exact)
    assert np.all(err <= n * 2.0 ** -24 * mag), float((err / (n * 2.0 ** -24 * mag + 1e-300)).max())
    assert np.all(dwte[counts == 0] == din[counts == 0])  # rows of absent ids are untouched
    exact_pe = dx0.astype(np.float64).sum(axis=0)
    err_pe = np.abs(dwpe.astype(np.float64) - exact_pe)
    assert np.all(err_pe <= B * 2.0 ** -24 * np.abs(dx0).astype(np.float64).sum(axis=0))
    # a row scattered to the wrong id is far outside the bound
    wrong = tok.copy()
    wrong[0, 0] = (wrong[0, 0] + 1) % V
    bad, _ = O.encoder_backward_f32(wrong, dx0, din, (T, C))
    assert np.any(np.abs(bad.astype(np.float64) - exact) > n * 2.0 ** -24 * mag)


def test_key_bias_gradient_vanishes():
    """Softmax is invariant to a per-query shift of the scores, so the key part
    of the QKV bias receives exactly zero gradient (up to rounding)."""
    cfg, P, tok, tgt = tiny_case()
    _, cache = O.forward(P, tok, tgt, cfg)
    G = O.backward(cache, cfg)
    C = cfg.C
    gk = G["qkvb"][:, C:2 * C]
    assert np.abs(gk).max() < 1e-14 * max(1.0, np.abs(G["qkvb"]).max()) + 1e-15
    assert np.abs(G["qkvb"][:, :C]).max() > 1e-8 and np.abs(G["qkvb"][:, 2 * C:]).max() > 1e-8
