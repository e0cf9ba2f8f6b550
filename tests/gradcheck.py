"""Per-slice comparison of backward results with the oracle.

A single norm over a whole gradient tensor averages an error confined to one
head or one short sequence away (one head in 256 with a 10 % error moves the
global relative L2 by about 0.6 %).  The backward is therefore judged slice
by slice -- one slice per (batch entry, head) of a dense [B, H, N, d] tensor,
or per (sequence, head) of a packed [total, H, d] one -- with two bounds:

* relative L2:   ||g_s - r_s||  <= REL_L2  * max(||r_s||,  FLOOR * rms * sqrt(n_s))
* element-wise:  max|g_s - r_s| <= ELEM    * max(max|r_s|, FLOOR * amax)

REL_L2 = 1e-2 is the stated tolerance for dQ, dK and dV.  ELEM = 2e-2 bounds
the worst element against the slice's largest one: bf16 output rounding alone
gives up to 2^-9 of an element, and the bf16 rounding of P and dS before the
products adds a few times that, so a correct kernel sits an order of magnitude
below it while a wrong row, column or tile does not.  FLOOR keeps slices whose
exact gradient vanishes (a single visible key: P = 1, dP - D = 0) from turning
fp64 rounding noise in the reference into a relative error: there the fp32
residue of the kernel is compared with 1e-3 of the gradients' typical size.
rms and amax are taken over all the gradients compared together (the largest
of the three), because a whole tensor can vanish -- with one key per row dQ
and dK are exactly zero everywhere -- while dV = P^T dO cannot while any key
is visible.
"""
from __future__ import annotations

import numpy as np

REL_L2 = 1e-2
ELEM = 2e-2
FLOOR = 1e-3


def slice_errors(g, r, rms_all, max_all):
    """(relative L2, element-wise ratio) of one slice, each already divided by
    its floored denominator, so a slice passes when both are <= 1."""
    g = np.asarray(g, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    n = r.size
    if n == 0:
        return 0.0, 0.0
    diff = g - r
    den_l2 = max(np.linalg.norm(r), FLOOR * rms_all * np.sqrt(n))
    den_el = max(np.abs(r).max(), FLOOR * max_all)
    rel = np.linalg.norm(diff) / den_l2 if den_l2 > 0 else float(np.linalg.norm(diff) > 0) * np.inf
    el = np.abs(diff).max() / den_el if den_el > 0 else float(np.abs(diff).max() > 0) * np.inf
    return rel / REL_L2, el / ELEM


def dense_slices(B, H):
    return [((b, h), (b, h)) for b in range(B) for h in range(H)]


def packed_slices(cu_seqlens, H):
    cu = [int(c) for c in cu_seqlens]
    out = []
    for s in range(len(cu) - 1):
        for h in range(H):
            out.append(((s, h), (slice(cu[s], cu[s + 1]), h)))
    return out


def check_grads(got, ref, slices, names=("dQ", "dK", "dV")):
    """Assert that every slice of every gradient meets both bounds; `slices`
    is a list of (label, index) pairs that select one slice from a tensor."""
    worst = {}
    rms_all = max((float(np.sqrt(np.mean(np.square(np.asarray(r, dtype=np.float64))))) for r in ref
                   if np.asarray(r).size), default=0.0)
    max_all = max((float(np.abs(np.asarray(r)).max()) for r in ref if np.asarray(r).size), default=0.0)
    for name, g, r in zip(names, got, ref):
        g = np.asarray(g)
        r = np.asarray(r)
        assert g.shape == r.shape, (name, g.shape, r.shape)
        assert np.isfinite(g).all(), f"{name}: non-finite values"
        bad = []
        w = (0.0, 0.0, None)
        for label, idx in slices:
            rel, el = slice_errors(g[idx], r[idx], rms_all, max_all)
            if max(rel, el) > max(w[0], w[1]):
                w = (rel, el, label)
            if rel > 1.0 or el > 1.0:
                bad.append((label, round(rel * REL_L2, 5), round(el * ELEM, 5)))
        worst[name] = w
        assert not bad, f"{name}: slices over tolerance (label, rel L2, max-abs / max|ref|): {bad[:8]}"
    return worst
