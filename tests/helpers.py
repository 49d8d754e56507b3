"""Small helpers shared by the GPU tests (data movement and error metrics
only; no arithmetic of the layer)."""

import numpy as np
import torch


def rel_frobenius(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def host(t):
    """Device tensor -> numpy (bf16 widened to fp32, exactly)."""
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


class ExpertView:
    """Indexable view of a [n, ...] weight tensor that hands the oracle one
    expert at a time as a host array (large weight sets never exist on the
    host in fp64 all at once)."""

    def __init__(self, t):
        self.t = t

    def __len__(self):
        return self.t.shape[0]

    def __getitem__(self, e):
        return host(self.t[e])
