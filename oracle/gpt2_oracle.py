"""CPU oracle for one GPT-2 pretraining step - TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
may import this module.  The product path never calls it and shares no code
with it.

It is a plain, slow, obviously-correct restatement of what the step computes,
in float64 by default (any numpy float dtype may be passed), written as
textbook numpy: one matmul per Linear, the full T x T masked softmax per
(batch, head), the full [rows, Vpad] logit matrix, closed-form backward rules
op by op, then the global-norm clip and AdamW.  No tiling, fusion or
reordering beyond the definitions.

Sources (pages on the subject, cited by title and section):
* "Let's reproduce GPT-2 (124M)" wiki page (nolimitkun.github.io),
  "Training recipe details": AdamW(0.9, 0.95, eps 1e-8), global clip 1.0,
  weight decay 0.1 on 2-D matrices only, residual projections scaled
  1/sqrt(2N), wte tied to lm_head; "GPU optimisation ladder": FlashAttention
  never materialises T x T (same result as this materialised form), vocab
  padded 50257 -> 50304.
* qntz.me nanoGPT news page: the block is multi-head attention + MLP +
  residual + LayerNorm; random-init loss 10.82 = ln(50257).
* dszhyy.com llm.c GPT-2 1558M article: GPT-2 hparams JSON (layer_norm_epsilon
  1e-5, initializer_range 0.02); "Reproduction setup" run log (parameter count
  1557686400 for d48, 4C MLP); "Parameter guide" (-c 0.1 decays 2-D weights
  only, GELU named by the -r / -ge flags).

Readings where the pages are silent (each listed in the design notes): pre-LN
block order with a final LayerNorm; tanh-form GELU; biased LayerNorm variance;
attention scale 1/sqrt(d), causal mask keeping j <= i; pad logit columns
excluded from the softmax; loss = mean over all B*T positions; clip norm over
every gradient with no epsilon; AdamW bias correction with step t and
decoupled decay.
"""
from __future__ import annotations

import numpy as np

LN_EPS = 1e-5  # GPT-2 hparams JSON, layer_norm_epsilon
GELU_K = np.sqrt(2.0 / np.pi)
GELU_C = 0.044715

DECAYED = ("wte", "wpe", "qkvw", "attprojw", "fcw", "fcprojw")  # the 2-D weight matrices


# ------------------------------------------------------------------ layout
def param_shapes(L, C, Vpad, T):
    """Canonical parameter order; Linear weights are [out, in]."""
    return [
        ("wte", (Vpad, C)), ("wpe", (T, C)),
        ("ln1w", (L, C)), ("ln1b", (L, C)),
        ("qkvw", (L, 3 * C, C)), ("qkvb", (L, 3 * C)),
        ("attprojw", (L, C, C)), ("attprojb", (L, C)),
        ("ln2w", (L, C)), ("ln2b", (L, C)),
        ("fcw", (L, 4 * C, C)), ("fcb", (L, 4 * C)),
        ("fcprojw", (L, C, 4 * C)), ("fcprojb", (L, C)),
        ("lnfw", (C,)), ("lnfb", (C,)),
    ]


def num_params(L, C, Vpad, T):
    """Padded wte + wpe + L blocks (12C^2 + 13C each) + final LN (2C)."""
    return sum(int(np.prod(s)) for _, s in param_shapes(L, C, Vpad, T))


# ------------------------------------------------------------------ ops
def encoder_forward(tok, wte, wpe):
    """x0[b, t, :] = wte[tok[b, t], :] + wpe[t, :]."""
    T = tok.shape[1]
    return wte[tok] + wpe[None, :T, :]


def layernorm_forward(x, w, b, eps=LN_EPS):
    """y = (x - mean) / sqrt(var + eps) * w + b over the last axis (biased var)."""
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mean) * rstd
    return xhat * w + b, mean[..., 0], rstd[..., 0]


def layernorm_backward(dy, x, w, mean, rstd):
    """Closed-form LayerNorm gradient; returns (dx, dw, db) summed over rows."""
    xhat = (x - mean[..., None]) * rstd[..., None]
    g = dy * w
    dx = rstd[..., None] * (g - g.mean(axis=-1, keepdims=True)
                            - xhat * (g * xhat).mean(axis=-1, keepdims=True))
    red = tuple(range(dy.ndim - 1))
    return dx, (dy * xhat).sum(axis=red), dy.sum(axis=red)


def gelu(x):
    """tanh-form GELU: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    return 0.5 * x * (1.0 + np.tanh(GELU_K * (x + GELU_C * x ** 3)))


def gelu_grad(x):
    """d gelu / dx of the tanh form."""
    u = GELU_K * (x + GELU_C * x ** 3)
    th = np.tanh(u)
    du = GELU_K * (1.0 + 3.0 * GELU_C * x ** 2)
    return 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th ** 2) * du


def attention_forward(q, k, v, scale):
    """Causal softmax attention per (b, h) on [B, H, T, d] arrays.

    S = q k^T * scale with S[i, j] = -inf for j > i; P = softmax_j(S);
    O = P v.  Returns (O, P, lse) where lse[b, h, i] = log sum_j exp S[i, j].
    """
    T = q.shape[2]
    s = np.matmul(q, np.swapaxes(k, -1, -2)) * scale
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)
    s = np.where(mask, -np.inf, s)
    smax = s.max(axis=-1, keepdims=True)
    e = np.exp(s - smax)
    ssum = e.sum(axis=-1, keepdims=True)
    p = e / ssum
    o = np.matmul(p, v)
    lse = (smax + np.log(ssum))[..., 0]
    return o, p, lse


def attention_backward(do, q, k, v, p, scale):
    """Gradients of O = softmax(mask(q k^T scale)) v w.r.t. q, k, v.

    dV = P^T dO; dP = dO v^T; dS = P * (dP - rowsum(P * dP)); dQ = dS k scale;
    dK = dS^T q scale.  (rowsum(P * dP) equals rowsum(dO * O).)
    """
    pt = np.swapaxes(p, -1, -2)
    dv = np.matmul(pt, do)
    dp = np.matmul(do, np.swapaxes(v, -1, -2))
    ds = p * (dp - (p * dp).sum(axis=-1, keepdims=True))
    dq = np.matmul(ds, k) * scale
    dk = np.matmul(np.swapaxes(ds, -1, -2), q) * scale
    return dq, dk, dv


def cross_entropy_forward(z, targets, V):
    """Mean CE over rows of logits z [M, Vpad]; columns >= V are excluded.

    Returns (loss, lse[M], probs[M, Vpad]) with probs 0 on the pad columns.
    """
    zz = z.copy()
    zz[:, V:] = -np.inf
    zmax = zz.max(axis=1, keepdims=True)
    e = np.exp(zz - zmax)
    ssum = e.sum(axis=1, keepdims=True)
    lse = (zmax + np.log(ssum))[:, 0]
    M = z.shape[0]
    loss = float(np.mean(lse - z[np.arange(M), targets]))
    return loss, lse, e / ssum


def cross_entropy_backward(probs, targets):
    """dz = (softmax - onehot(target)) / M for the mean loss."""
    M = probs.shape[0]
    dz = probs.copy()
    dz[np.arange(M), targets] -= 1.0
    return dz / M


def classifier_forward_backward(x, w, targets, V):
    """Tied lm_head + mean CE: z = x w^T; returns loss, dx, dw, and lse."""
    z = x @ w.T
    loss, lse, probs = cross_entropy_forward(z, targets, V)
    dz = cross_entropy_backward(probs, targets)
    return loss, dz @ w, dz.T @ x, lse


# ------------------------------------------------------------------ model
class Config:
    def __init__(self, L, H, C, V, Vpad, T):
        assert C % H == 0 and Vpad >= V
        self.L, self.H, self.C, self.V, self.Vpad, self.T = L, H, C, V, Vpad, T
        self.d = C // H
        self.scale = 1.0 / np.sqrt(self.d)


def forward(P, tok, tgt, cfg: Config, dtype=np.float64):
    """Forward pass of the pre-LN GPT-2 and its mean CE; returns (loss, cache)."""
    P = {k: np.asarray(v, dtype=dtype) for k, v in P.items()}
    B, T = tok.shape
    L, H, C, d = cfg.L, cfg.H, cfg.C, cfg.d
    x = encoder_forward(tok, P["wte"], P["wpe"])
    layers = []
    for l in range(L):
        c = {"x": x}
        c["ln1"], c["m1"], c["r1"] = layernorm_forward(x, P["ln1w"][l], P["ln1b"][l])
        qkv = c["ln1"] @ P["qkvw"][l].T + P["qkvb"][l]
        q, k, v = (qkv[..., i * C:(i + 1) * C].reshape(B, T, H, d).transpose(0, 2, 1, 3)
                   for i in range(3))
        o, p, lse = attention_forward(q, k, v, cfg.scale)
        c.update(q=q, k=k, v=v, p=p, lse=lse)
        c["y"] = o.transpose(0, 2, 1, 3).reshape(B, T, C)
        x1 = x + c["y"] @ P["attprojw"][l].T + P["attprojb"][l]
        c["x1"] = x1
        c["ln2"], c["m2"], c["r2"] = layernorm_forward(x1, P["ln2w"][l], P["ln2b"][l])
        c["h"] = c["ln2"] @ P["fcw"][l].T + P["fcb"][l]
        c["a"] = gelu(c["h"])
        x = x1 + c["a"] @ P["fcprojw"][l].T + P["fcprojb"][l]
        layers.append(c)
    lnf, mf, rf = layernorm_forward(x, P["lnfw"], P["lnfb"])
    M = B * T
    z = lnf.reshape(M, C) @ P["wte"].T
    loss, lse_ce, probs = cross_entropy_forward(z, tgt.reshape(M), cfg.V)
    cache = dict(P=P, tok=tok, tgt=tgt, layers=layers, xL=x, lnf=lnf, mf=mf, rf=rf,
                 z=z, probs=probs, lse_ce=lse_ce)
    return loss, cache


def backward(cache, cfg: Config):
    """Full backward pass; returns a dict of gradients keyed like the parameters."""
    P = cache["P"]
    tok, tgt = cache["tok"], cache["tgt"]
    B, T = tok.shape
    L, H, C, d = cfg.L, cfg.H, cfg.C, cfg.d
    M = B * T
    G = {k: np.zeros_like(v) for k, v in P.items()}
    dz = cross_entropy_backward(cache["probs"], tgt.reshape(M))
    lnf = cache["lnf"].reshape(M, C)
    G["wte"] += dz.T @ lnf
    dlnf = (dz @ P["wte"]).reshape(B, T, C)
    dx, G["lnfw"], G["lnfb"] = layernorm_backward(dlnf, cache["xL"], P["lnfw"], cache["mf"], cache["rf"])
    for l in reversed(range(L)):
        c = cache["layers"][l]
        # MLP: x2 = x1 + gelu(ln2 Wfc^T + bfc) Wfcp^T + bfcp
        G["fcprojw"][l] = dx.reshape(M, C).T @ c["a"].reshape(M, 4 * C)
        G["fcprojb"][l] = dx.sum(axis=(0, 1))
        da = dx @ P["fcprojw"][l]
        dh = da * gelu_grad(c["h"])
        G["fcw"][l] = dh.reshape(M, 4 * C).T @ c["ln2"].reshape(M, C)
        G["fcb"][l] = dh.sum(axis=(0, 1))
        dln2 = dh @ P["fcw"][l]
        dxl, G["ln2w"][l], G["ln2b"][l] = layernorm_backward(dln2, c["x1"], P["ln2w"][l], c["m2"], c["r2"])
        dx1 = dx + dxl
        # attention: x1 = x + y Wproj^T + bproj
        G["attprojw"][l] = dx1.reshape(M, C).T @ c["y"].reshape(M, C)
        G["attprojb"][l] = dx1.sum(axis=(0, 1))
        dy = dx1 @ P["attprojw"][l]
        do = dy.reshape(B, T, H, d).transpose(0, 2, 1, 3)
        dq, dk, dv = attention_backward(do, c["q"], c["k"], c["v"], c["p"], cfg.scale)
        dqkv = np.concatenate([g.transpose(0, 2, 1, 3).reshape(B, T, C) for g in (dq, dk, dv)], axis=-1)
        G["qkvw"][l] = dqkv.reshape(M, 3 * C).T @ c["ln1"].reshape(M, C)
        G["qkvb"][l] = dqkv.sum(axis=(0, 1))
        dln1 = dqkv @ P["qkvw"][l]
        dxl, G["ln1w"][l], G["ln1b"][l] = layernorm_backward(dln1, c["x"], P["ln1w"][l], c["m1"], c["r1"])
        dx = dx1 + dxl
    # encoder: tied wte receives the scatter of dx0 by token; wpe the sum over batch
    np.add.at(G["wte"], tok.reshape(M), dx.reshape(M, C))
    G["wpe"][:T] += dx.sum(axis=0)
    return G


def global_norm(G):
    """sqrt(sum of squares of every gradient element)."""
    return float(np.sqrt(sum(float(np.sum(np.asarray(g, dtype=np.float64) ** 2)) for g in G.values())))


def clip_scale(norm, max_norm=1.0):
    """Factor applied to every gradient: max_norm / norm when norm exceeds max_norm, else 1."""
    return max_norm / norm if norm > max_norm else 1.0


def adamw_update(w, g, m, v, t, lr, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.0):
    """One AdamW update (Loshchilov & Hutter, decoupled decay) at step t >= 1.

    Returns the new (w, m, v).
    """
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    mhat = m / (1.0 - beta1 ** t)
    vhat = v / (1.0 - beta2 ** t)
    w = w - lr * (mhat / (np.sqrt(vhat) + eps) + wd * w)
    return w, m, v


def clip_adamw(P, G, M_, V_, t, lr, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1, max_norm=1.0):
    """Global-norm clip of G then AdamW on every tensor (decay only on the 2-D matrices).

    Returns (norm, newP, newM, newV); inputs are not modified.
    """
    norm = global_norm(G)
    s = clip_scale(norm, max_norm)
    nP, nM, nV = {}, {}, {}
    for k in P:
        nP[k], nM[k], nV[k] = adamw_update(np.asarray(P[k], np.float64), s * np.asarray(G[k], np.float64),
                                           np.asarray(M_[k], np.float64), np.asarray(V_[k], np.float64),
                                           t, lr, beta1, beta2, eps, wd if k in DECAYED else 0.0)
    return norm, nP, nM, nV


def train_step(P, tok, tgt, cfg: Config, lr=6e-4, t=1, M_=None, V_=None, dtype=np.float64, **kw):
    """forward -> mean CE -> backward -> clip -> AdamW. Returns a dict of results."""
    loss, cache = forward(P, tok, tgt, cfg, dtype=dtype)
    G = backward(cache, cfg)
    if M_ is None:
        M_ = {k: np.zeros_like(v, dtype=np.float64) for k, v in G.items()}
    if V_ is None:
        V_ = {k: np.zeros_like(v, dtype=np.float64) for k, v in G.items()}
    norm, nP, nM, nV = clip_adamw(cache["P"], G, M_, V_, t, lr, **kw)
    return dict(loss=loss, grads=G, norm=norm, params=nP, m=nM, v=nV, cache=cache)


# ------------------------------------------------- fp32 sequential references
def encoder_forward_f32(tok, wte, wpe):
    """x0 = wte[tok] + wpe[t] with one IEEE float32 addition per element."""
    wte = np.asarray(wte, np.float32)
    wpe = np.asarray(wpe, np.float32)
    return (wte[tok] + wpe[None, : tok.shape[1], :]).astype(np.float32)


def encoder_backward_f32(tok, dx0, dwte_in, dwpe_shape, run=64):
    """Scatter of the encoder gradient in a fixed order, float32 throughout.

    For every vocab id v, its positions i = b*T + t in ascending order are cut
    into runs of `run`; each run is summed from zero in ascending order, the
    run sums are added in run order starting from zero, and
    dwte[v] = dwte_in[v] + total.  For every position t: dwpe[t] = sum over b
    ascending of dx0[b, t], starting from 0.  Returns (dwte, dwpe) as float32.
    (The pages fix no order; this one is the reading both sides implement.)
    """
    B, T = tok.shape
    C = dx0.shape[-1]
    flat = np.asarray(dx0, np.float32).reshape(B * T, C)
    ids = tok.reshape(-1)
    dwte = np.array(dwte_in, dtype=np.float32, copy=True)
    for vtok in np.unique(ids):
        pos = np.nonzero(ids == vtok)[0]  # ascending
        total = np.zeros(C, np.float32)
        for r0 in range(0, pos.size, run):
            acc = np.zeros(C, np.float32)
            for i in pos[r0:r0 + run]:
                acc = (acc + flat[i]).astype(np.float32)
            total = (total + acc).astype(np.float32)
        dwte[vtok] = (dwte[vtok] + total).astype(np.float32)
    dwpe = np.zeros(dwpe_shape, np.float32)
    acc = np.zeros((T, C), np.float32)
    for b in range(B):
        acc = (acc + np.asarray(dx0, np.float32)[b]).astype(np.float32)
    dwpe[:T] = acc
    return dwte, dwpe
