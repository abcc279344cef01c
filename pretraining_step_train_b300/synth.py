"""Seeded synthetic inputs for the GPT-2 training step.

This module only *produces data*: counter-based random numbers, the initial
parameter set and token streams.  It holds none of the training step's
arithmetic, so the CUDA path and the CPU oracle can both be fed from it
without sharing any computation.

Generators
----------
* ``splitmix64(seed, counter)`` - the counter-based 64-bit mixer of Steele,
  Lea and Flood ("Fast splittable pseudorandom number generators", 2014).
  Every draw is a pure function of (seed, index), so any slice of a stream can
  be regenerated independently.
* ``uniform`` - top 53 bits of a splitmix64 word scaled to [0, 1).
* ``normal`` - Box-Muller on pairs of uniforms.
* ``zipf_tokens`` - inverse-CDF sampling of p(k) proportional to (k+1)^-s over
  [0, V), the synthetic stand-in for the GPT-2-tokenised FineWeb-EDU shards
  the pages train on (the dataset itself is not used).

Initial parameters (``init_params``) follow the GPT-2 recipe the pages
describe (Let's reproduce GPT-2 (124M) wiki page, "training recipe" bullets;
GPT-2 hparams JSON "initializer_range": 0.02): every weight matrix plus wte
and wpe ~ N(0, 0.02), the two residual projections per block scaled by
1/sqrt(2L), biases 0, LayerNorm gamma 1 / beta 0, padded vocab rows of wte 0.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, counter: np.ndarray) -> np.ndarray:
    """splitmix64 output for each 64-bit counter value (vectorised, wraps mod 2^64)."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (counter.astype(np.uint64) + np.uint64(1)) * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniform(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """n float64 uniforms in [0, 1) from counters offset .. offset+n-1."""
    c = np.arange(offset, offset + n, dtype=np.uint64)
    return (splitmix64(seed, c) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal(seed: int, n: int, std: float = 1.0, chunk: int = 1 << 24) -> np.ndarray:
    """n float64 N(0, std^2) samples by Box-Muller (pairs of uniforms)."""
    out = np.empty(n, dtype=np.float64)
    npairs = (n + 1) // 2
    for p0 in range(0, npairs, chunk):
        p1 = min(npairs, p0 + chunk)
        u = uniform(seed, 2 * (p1 - p0), offset=2 * p0)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log1p(-u1))  # 1-u1 in (0, 1]
        ang = 2.0 * np.pi * u2
        z = np.empty(2 * (p1 - p0))
        z[0::2] = r * np.cos(ang)
        z[1::2] = r * np.sin(ang)
        lo = 2 * p0
        hi = min(n, 2 * p1)
        out[lo:hi] = z[: hi - lo]
    return out * std


def zipf_tokens(seed: int, rows: int, length: int, vocab: int, s: float = 1.1) -> np.ndarray:
    """int32 [rows, length] ids with p(k) ~ (k+1)^-s, k in [0, vocab), rank = id."""
    w = np.arange(1, vocab + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = uniform(seed, rows * length)
    ids = np.searchsorted(cdf, u, side="right")
    return np.minimum(ids, vocab - 1).astype(np.int32).reshape(rows, length)


def uniform_tokens(seed: int, rows: int, length: int, vocab: int) -> np.ndarray:
    """int32 [rows, length] ids i.i.d. uniform over [0, vocab)."""
    u = uniform(seed, rows * length)
    return np.minimum((u * vocab).astype(np.int64), vocab - 1).astype(np.int32).reshape(rows, length)


def token_batch(seed: int, B: int, T: int, V: int, dist: str = "zipf"):
    """(tokens, targets) int32 [B, T]; targets are the stream shifted by one."""
    if dist == "zipf":
        s = zipf_tokens(seed, B, T + 1, V)
    elif dist == "uniform":
        s = uniform_tokens(seed, B, T + 1, V)
    else:
        raise ValueError(dist)
    return np.ascontiguousarray(s[:, :T]), np.ascontiguousarray(s[:, 1:])


def iid_token_batch(seed: int, B: int, T: int, V: int):
    """Tokens and targets drawn independently and uniformly (the tiny fp32 case)."""
    tok = uniform_tokens(seed, B, T, V)
    tgt = uniform_tokens(seed ^ 0x5DEECE66D, B, T, V)
    return tok, tgt


# ----------------------------------------------------------------- parameters
def param_shapes(L: int, C: int, Vpad: int, T: int):
    """Canonical flat order of the parameter tensors (names follow GPT-2).

    Weight matrices are stored [out, in] (row-major), so a Linear computes
    y = x W^T + b.  Per-layer tensors are stacked along a leading L axis.
    """
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


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 value (round-to-nearest-even) of each element, returned as float32."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    r = r.astype(np.uint32)
    nan = np.isnan(a)
    out = r.view(np.float32).copy()
    out[nan] = np.nan
    return out


def init_params(seed: int, L: int, C: int, V: int, Vpad: int, T: int, std: float = 0.02,
                bf16_representable: bool = False) -> dict:
    """Initial GPT-2 parameters as float32 arrays, keyed by name (canonical order).

    With ``bf16_representable`` every value is rounded to the nearest bf16 so
    that a bf16 copy equals the fp32 master copy exactly.
    """
    out = {}
    for i, (name, shape) in enumerate(param_shapes(L, C, Vpad, T)):
        n = int(np.prod(shape))
        sub = seed * 1000003 + i * 7919
        if name.endswith("w") and name.startswith("ln"):
            a = np.ones(n)
        elif name in ("wte", "wpe", "qkvw", "attprojw", "fcw", "fcprojw"):
            s = std
            if name in ("attprojw", "fcprojw"):
                s = std / np.sqrt(2.0 * L)
            a = normal(sub, n, s)
            if name == "wte":
                a = a.reshape(Vpad, C)
                a[V:, :] = 0.0
                a = a.reshape(-1)
        else:
            a = np.zeros(n)
        a = a.astype(np.float32).reshape(shape)
        if bf16_representable:
            a = round_to_bf16(a).reshape(shape)
        out[name] = a
    return out


def flatten_params(params: dict, L: int, C: int, Vpad: int, T: int) -> np.ndarray:
    """Concatenate a parameter dict into one float32 vector in canonical order."""
    return np.concatenate([np.asarray(params[n], dtype=np.float32).reshape(-1)
                           for n, _ in param_shapes(L, C, Vpad, T)])


def unflatten_params(flat: np.ndarray, L: int, C: int, Vpad: int, T: int) -> dict:
    out, off = {}, 0
    for n, shape in param_shapes(L, C, Vpad, T):
        k = int(np.prod(shape))
        out[n] = flat[off:off + k].reshape(shape)
        off += k
    assert off == flat.size, (off, flat.size)
    return out


def attention_inputs(seed: int, B: int, H: int, T: int, d: int, bf16: bool = True):
    """q, k, v, dO ~ N(0, 1) as float32 [B, H, T, d] (bf16-representable if asked)."""
    outs = []
    for j in range(4):
        a = normal(seed * 31 + j, B * H * T * d).astype(np.float32).reshape(B, H, T, d)
        outs.append(round_to_bf16(a).reshape(a.shape) if bf16 else a)
    return tuple(outs)


def classifier_inputs(seed: int, M: int, C: int, V: int, Vpad: int, bf16: bool = True):
    """x ~ N(0,1) [M, C]; w ~ N(0, 0.02) [Vpad, C] with rows >= V zero; Zipf(1.1) targets [M]."""
    x = normal(seed * 17 + 1, M * C).astype(np.float32).reshape(M, C)
    w = normal(seed * 17 + 2, Vpad * C, 0.02).astype(np.float32).reshape(Vpad, C)
    w[V:] = 0.0
    if bf16:
        x = round_to_bf16(x).reshape(M, C)
        w = round_to_bf16(w).reshape(Vpad, C)
    tgt = zipf_tokens(seed * 17 + 3, 1, M, V).reshape(M)
    return x, w, tgt
