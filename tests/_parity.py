"""Comparison helpers for GPU-vs-oracle parity (tie-aware code comparison)."""
import numpy as np

import oracle as O

TIE_TOL = 1e-5          # |d(gpu) - d(oracle)| in lattice units (1e-5 scale^2 in weight units)
MAX_TIE_FRACTION = 1e-4  # non-identical blocks allowed, as a fraction of all blocks


def compare_codes(gpu_codes, q, lattice, skip_rows_mask=None, max_fraction=MAX_TIE_FRACTION):
    """Codes must equal the oracle's except at certified near-ties.

    A differing block is accepted when its GPU code is a lattice code and its
    squared distance to the oracle's y (float64) is within TIE_TOL of the
    oracle's.  Returns (n_blocks, n_different).
    """
    n = O.LATTICE_DIM[lattice]
    g = np.asarray(gpu_codes).astype(np.int64)
    o = np.asarray(q.codes_wide)
    y = np.asarray(q.y)
    if skip_rows_mask is not None:
        keep = ~np.asarray(skip_rows_mask)
        g, o, y = g[keep], o[keep], y[keep]
    g = g.reshape(-1, n)
    o = o.reshape(-1, n)
    y = y.reshape(-1, n)
    diff = np.nonzero(np.any(g != o, axis=1))[0]
    if len(diff):
        member = O.code_membership_ok(lattice, g[diff])
        dg = O.block_sqdist(lattice, y[diff], g[diff])
        do = O.block_sqdist(lattice, y[diff], o[diff])
        ok = member & (np.abs(dg - do) <= TIE_TOL)
        if not ok.all():
            bad = diff[~ok][:5]
            raise AssertionError(
                f"{(~ok).sum()} of {len(g)} blocks differ beyond the tie band; first: "
                + "; ".join(f"block {b}: y={y[b]}, gpu={g[b]}, oracle={o[b]}" for b in bad))
        assert len(diff) <= max(2, max_fraction * len(g)), f"{len(diff)} tie blocks of {len(g)}"
    return len(g), len(diff)


def normwise_rel(a, ref):
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(a - ref) / (den if den > 0 else 1.0))
