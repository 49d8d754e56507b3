"""Small helpers shared by the GPU tests (data movement and error metrics
only; no arithmetic of the layer)."""

import numpy as np
import torch


def rel_frobenius(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def row_errors(a, b):
    """Relative error of every row (leading axis; the rest flattened):
    ||a_r - b_r|| / max(||b_r||, 1e-3 * median row norm of b).  The floor
    keeps a row whose reference is (nearly) zero from dividing by zero; it
    is far below any row a layer produces."""
    a = np.asarray(a, dtype=np.float64).reshape(len(a), -1)
    b = np.asarray(b, dtype=np.float64).reshape(len(b), -1)
    nb = np.linalg.norm(b, axis=1)
    floor = max(1e-3 * float(np.median(nb)), 1e-300)
    return np.linalg.norm(a - b, axis=1) / np.maximum(nb, floor)


def assert_close(a, b, tol, what=None, row_tol=None):
    """Both the whole tensor (relative Frobenius error) within `tol` and each
    row on its own (see row_errors) within `row_tol` (default `tol`): a
    single bad row of a large tensor hardly moves the Frobenius norm, so
    every row is bounded too."""
    row_tol = tol if row_tol is None else row_tol
    fro = rel_frobenius(a, b)
    if len(np.shape(b)) == 0 or np.size(b) == 0:
        assert fro < tol, (what, fro)
        return
    r = row_errors(a, b)
    worst = int(np.argmax(r))
    assert fro < tol and r[worst] < row_tol, (what, f"frobenius {fro:.3e}",
                                              f"worst row {worst}: {r[worst]:.3e}")


def host(t):
    """Device tensor -> numpy (bf16 widened to fp32, exactly)."""
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def tail_sample(offsets, token_of_row, T, n, seed=1):
    """Tokens to recompute with the oracle at a full-size shape, chosen so
    that the ragged ends of the grouped GEMMs' tiles are among them: the
    first and the last token; the tokens of the last 8 rows (the ragged last
    M tile) and of the first 4 rows of the most loaded expert's segment; the
    last row of up to 4 experts whose whole segment fits one 128-row tile;
    the last row of up to 4 experts with 2 to 4 tiles; then random tokens up
    to n.  Returns sorted unique token indices (at most n unless the
    required ones alone are more)."""
    off = np.asarray(offsets, dtype=np.int64)
    tor = np.asarray(token_of_row, dtype=np.int64)
    counts = np.diff(off)
    want = [0, T - 1]
    hot = int(np.argmax(counts))
    lo, hi = int(off[hot]), int(off[hot + 1])
    want += list(tor[max(lo, hi - 8):hi]) + list(tor[lo:min(hi, lo + 4)])
    one = np.nonzero((counts >= 1) & (counts <= 128))[0][:4]
    few = np.nonzero((counts > 128) & (counts <= 512))[0][:4]
    want += [int(tor[off[e + 1] - 1]) for e in list(one) + list(few)]
    chosen = sorted(set(int(t) for t in want))
    rng = np.random.default_rng(seed)
    rest = [t for t in rng.permutation(T) if t not in set(chosen)]
    chosen = sorted(set(chosen) | set(int(t) for t in rest[:max(0, n - len(chosen))]))
    return np.asarray(chosen, dtype=np.int64)


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
