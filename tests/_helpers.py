"""Shared helpers of the test suites (device transfer, error metrics)."""
import numpy as np


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def to_dev(a, dtype="bf16"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype == "bf16":
        t = t.to(torch.float32).to(torch.bfloat16)
    elif dtype == "f32":
        t = t.to(torch.float32)
    elif dtype == "i32":
        t = t.to(torch.int32)
    return t.cuda()


def to_np(t):
    import torch
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def split_params(flat, L, C, Vpad, T):
    from pretraining_step_train_b300 import synth
    return synth.unflatten_params(np.asarray(flat), L, C, Vpad, T)
