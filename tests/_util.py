"""Shared test helpers: tolerance check, bf16 transfers, gap-separated routing inputs."""
from __future__ import annotations

import re

import numpy as np

import oracle
import workloads as wl

REL_TOL = 8e-3   # |y - y_ref| <= 8e-3 |y_ref| + 1e-3 * sum_k |x_k W_nk|
ABS_TOL = 1e-3
GAP = 1e-3       # minimum gap between adjacent top-(k+1) router scores


def to_f64(t) -> np.ndarray:
    """torch bf16/fp32 tensor -> float64 numpy (exact)."""
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def assert_within_tol(y, ref, absref, what="", rel=REL_TOL, absk=ABS_TOL):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - ref)
    bound = rel * np.abs(ref) + absk * absref
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        lines = ["%s: %d of %d elements outside |y-ref| <= %g|ref| + %g*A" %
                 (what, int(bad.sum()), bad.size, rel, absk)]
        for i in idx:
            i = tuple(i)
            lines.append("  at %s: y=%r ref=%r A=%r" % (i, y[i], ref[i], absref[i]))
        raise AssertionError("\n".join(lines))


def gap_rows(Wr_bits, M, H, k, *key, gap=GAP, max_tries=64):
    """Token rows ~N(0,1) whose fp64 router scores have adjacent gaps >= gap
    among the k+1 largest; a failing row is redrawn (its attempt number
    raised). Returns (x_bits, attempts)."""
    attempts = [0] * M
    for _ in range(max_tries):
        x = wl.token_rows(M, H, *key, attempts=attempts)
        logits, _ = oracle.linear(x, Wr_bits)
        g = oracle.sorted_gaps(logits, min(k + 1, logits.shape[1]))
        bad = np.where(~np.all(g >= gap, axis=1))[0] if g.shape[1] else np.array([], int)
        if bad.size == 0:
            return x, attempts
        for m in bad:
            attempts[m] += 1
    raise RuntimeError("could not draw gap-separated rows")


def header_functions(path) -> list:
    """Function names declared in a C header."""
    src = open(path).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:[A-Za-z_][A-Za-z0-9_]*[\s*]+)+([a-z_][a-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))
