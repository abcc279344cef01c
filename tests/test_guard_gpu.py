"""The update guard of the step through the C ABI: a non-finite loss or
gradient norm, or (when thresholds are set) a loss or norm z-score above its
threshold, skips the AdamW update and leaves every weight and moment bit for
bit as it was (llm.c GPT-2 1558M article, "400B token run": updates are skipped
on momentary spikes, flags -sl 5.0 -sg 5.0; the run log's z-scores read "+nan"
until enough steps have passed).  The failures are made on the host: a NaN or
an outsized weight loaded through gpt2_set_params."""
import ctypes as ct

import numpy as np
import pytest

from oracle import gpt2_oracle as O
from pretraining_step_train_b300 import binding, synth
from tests._helpers import rel_l2, to_dev

pytestmark = pytest.mark.gpu

L, H, C, V, Vpad, T, B = 2, 2, 128, 1000, 1024, 128, 2
LR, B1, B2, EPS, WD, CLIP = 6e-4, 0.9, 0.95, 1e-8, 0.1, 1.0
STATE = (binding.GPT2_PARAMS, binding.GPT2_MASTER, binding.GPT2_ADAM_M, binding.GPT2_ADAM_V)


def _snapshot(s):
    return {w: np.ascontiguousarray(s.get(w), np.float32).view(np.uint32).copy() for w in STATE}


def _assert_same(a, b):
    for w in STATE:
        np.testing.assert_array_equal(a[w], b[w])


def _params(seed):
    P = synth.init_params(seed, L, C, V, Vpad, T, bf16_representable=True)
    return synth.flatten_params(P, L, C, Vpad, T), P


def _batch(seed):
    return tuple(to_dev(x, "i32") for x in synth.token_batch(seed, B, T, V))


def _clip_adamw(s, lr=LR, t=0):
    """gpt2_clip_adamw with a norm read-back: (status, norm)."""
    norm = ct.c_float()
    st = binding.lib().gpt2_clip_adamw(s.h, lr, B1, B2, EPS, WD, CLIP, t, ct.byref(norm))
    return st, norm.value


def _weight_index(name, *idx):
    """Flat index of one element of a named parameter tensor."""
    off = 0
    for n, shape in synth.param_shapes(L, C, Vpad, T):
        if n == name:
            return off + int(np.ravel_multi_index(idx, shape))
        off += int(np.prod(shape))
    raise KeyError(name)


def test_nonfinite_step_leaves_weights_untouched():
    """A NaN weight makes the loss and the norm NaN: the call reports
    GPT2_E_NONFINITE and master, working weights, m and v keep their bits; the
    next finite step runs normally and matches the oracle at t = 1 (the skipped
    step did not advance the device step counter)."""
    flat, P = _params(61)
    bad = flat.copy()
    bad[_weight_index("fcw", 1, 5, 7)] = np.nan
    s = binding.Step(L, H, C, V, Vpad, T, B, precision=binding.GPT2_BF16)
    s.set_params(bad)
    before = _snapshot(s)
    batch = _batch(62)
    s.forward(*batch, want_loss=False)
    s.backward()
    st, norm = _clip_adamw(s)
    assert st == binding.GPT2_E_NONFINITE and not np.isfinite(norm)
    _assert_same(before, _snapshot(s))
    g = s.guard_read()
    assert g["skipped_nonfinite"] == 1 and g["last_skipped"] == 1 and g["skipped_spike"] == 0
    # load finite weights again and take a normal step with the device counter
    s.set_params(flat)
    loss = s.forward(*batch)
    s.backward()
    st, norm = _clip_adamw(s)
    assert st == binding.GPT2_OK
    tok, tgt = synth.token_batch(62, B, T, V)
    ref = O.train_step(P, tok, tgt, O.Config(L, H, C, V, Vpad, T), lr=LR, t=1, beta1=B1, beta2=B2, eps=EPS,
                       wd=WD, max_norm=CLIP)
    assert abs(loss - ref["loss"]) / ref["loss"] < 1e-2
    ref_flat = synth.flatten_params({k: v.astype(np.float32) for k, v in ref["params"].items()}, L, C, Vpad, T)
    assert rel_l2(s.get(binding.GPT2_MASTER), ref_flat) < 1e-2
    assert s.guard_read()["last_skipped"] == 0
    s.close()


def test_spike_guard_skips_outlier_and_scores_match_the_window():
    """Window of 4: the z-scores are NaN until four finite values are held, then
    equal (x - mean) / std of the last four (population).  With thresholds of 3,
    an outsized LayerNorm gain makes the loss and the norm jump: the update is
    skipped (weights and moments keep their bits, the step counter stays), and
    with the checks off the same step is applied."""
    W = 4
    flat, P = _params(63)
    s = binding.Step(L, H, C, V, Vpad, T, B, precision=binding.GPT2_BF16)
    s.set_params(flat)
    s.set_guard(0.0, 3.0, W)
    losses, norms = [], []
    for i in range(W + 1):  # lr = 0: the weights stay put and the scores stay moderate
        losses.append(s.forward(*_batch(100 + i)))
        s.backward()
        st, n = _clip_adamw(s, lr=0.0)
        assert st == binding.GPT2_OK
        norms.append(n)
        g = s.guard_read()
        if i < W:
            assert np.isnan(g["z_loss"]) and np.isnan(g["z_norm"]), (i, g)
        else:
            for key, xs in (("z_loss", losses), ("z_norm", norms)):
                hist = np.array(xs[:W], np.float64)
                z = (xs[W] - hist.mean()) / hist.std()
                assert abs(g[key] - z) <= 1e-3 * max(1.0, abs(z)), (key, g[key], z)
        assert g["skipped_spike"] == 0 and g["last_skipped"] == 0
    # the final LayerNorm's gain scaled by 50: the logits, the loss and the gradients jump
    spiky = flat.copy()
    for c in range(C):
        spiky[_weight_index("lnfw", c)] *= 50.0
    s.set_guard(3.0, 3.0, W)  # both checks on; this empties the window, so refill it
    for i in range(W):
        s.forward(*_batch(150 + i))
        s.backward()
        assert _clip_adamw(s, lr=0.0)[0] == binding.GPT2_OK
    assert s.guard_read()["skipped_spike"] == 0
    s.set_params(spiky)  # zeroes m, v and the step counter; the guard's window stays
    before = _snapshot(s)
    batch = _batch(200)
    s.forward(*batch)
    s.backward()
    st, n = _clip_adamw(s)
    assert st == binding.GPT2_OK
    g = s.guard_read()
    assert max(g["z_loss"], g["z_norm"]) > 3.0 and g["skipped_spike"] == 1 and g["last_skipped"] == 1, (n, norms, g)
    _assert_same(before, _snapshot(s))
    # checks off (the window empties): the same step is applied, with t = 1 from the
    # counter that the skipped step left at 0; a second handle given t = 1 agrees bit for bit
    s.set_guard(0.0, 0.0, W)
    s.forward(*batch)
    s.backward()
    assert _clip_adamw(s)[0] == binding.GPT2_OK
    after = _snapshot(s)
    assert not np.array_equal(after[binding.GPT2_MASTER], before[binding.GPT2_MASTER])
    r = binding.Step(L, H, C, V, Vpad, T, B, precision=binding.GPT2_BF16)
    r.set_params(spiky)
    r.forward(*batch)
    r.backward()
    assert _clip_adamw(r, t=1)[0] == binding.GPT2_OK
    _assert_same(after, _snapshot(r))
    s.close()
    r.close()


def test_guard_settings_are_validated_on_the_host():
    s = binding.Step(1, 1, 64, 250, 256, 64, 1, precision=binding.GPT2_BF16)
    lib = binding.lib()
    assert lib.gpt2_set_guard(s.h, 5.0, 5.0, 1) == binding.GPT2_E_INVAL
    assert lib.gpt2_set_guard(s.h, 5.0, 5.0, 257) == binding.GPT2_E_INVAL
    assert lib.gpt2_set_guard(s.h, float("nan"), 5.0, 8) == binding.GPT2_E_INVAL
    assert lib.gpt2_set_guard(s.h, 5.0, 5.0, 256) == binding.GPT2_OK
    g = s.guard_read()
    assert np.isnan(g["z_loss"]) and g["skipped_spike"] == 0 and g["skipped_nonfinite"] == 0
    s.close()
