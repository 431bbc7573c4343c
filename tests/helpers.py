"""Helpers shared by the tests: input conversion and error measures."""
import numpy as np


def weights_to_numpy(W):
    """synth.ExpertWeights (torch, any device) -> the oracle's dict of numpy arrays."""
    import torch
    cv = lambda t: None if t is None else t.detach().cpu().contiguous()
    out = dict(fmt=W.fmt, d=W.d, f=W.f)
    for name in ("gate", "up", "down"):
        t = cv(getattr(W, name))
        out[name] = bf16_bits(t) if t.dtype == torch.bfloat16 else t.numpy()
        s = cv(getattr(W, name + "_s"))
        out[name + "_s"] = None if s is None else s.numpy()
    out["glob"] = cv(W.glob).numpy()
    return out


def bf16_bits(t):
    """bf16 torch tensor -> numpy uint16 bit patterns."""
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


class LazySlots:
    """Slot-indexed view of a (device) tensor; slot s is copied to host on first use."""

    def __init__(self, t):
        self.t = t
        self.cache = {}

    def __getitem__(self, s):
        s = int(s)
        if s not in self.cache:
            self.cache[s] = self.t[s].detach().cpu().numpy()
        return self.cache[s]


def weights_lazy(W):
    """The oracle's weight dict over device tensors, fetching slots on demand."""
    import torch
    out = dict(fmt=W.fmt, d=W.d, f=W.f)
    for name in ("gate", "up", "down"):
        t = getattr(W, name)
        out[name] = _Bf16Slots(t) if t.dtype == torch.bfloat16 else LazySlots(t)
        s = getattr(W, name + "_s")
        out[name + "_s"] = None if s is None else LazySlots(s)
    out["glob"] = W.glob.detach().cpu().numpy()
    return out


class _Bf16Slots(LazySlots):
    def __getitem__(self, s):
        s = int(s)
        if s not in self.cache:
            self.cache[s] = bf16_bits(self.t[s])
        return self.cache[s]
