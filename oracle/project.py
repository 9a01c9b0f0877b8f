"""Projected-state oracle (test infrastructure only; nothing in the library
imports it).

RedKnot-MLA paper, first paragraphs (eqs. 2-4, the projected state) and the
TP8 fast-path paragraph (sliced W_a, Local restoration, row-wise replacement
into a contiguous projected state, W_b once); RedKnot blog, "The same idea
on DeepSeek-V4" (z = z_off + z_on, y = W_b z).  The first output projection
is bias free and sliced by the logical heads' channel ranges; heads act in
their native output groups of `group` consecutive heads, so W_a holds one
[d_g, group * d_v] block per group.  The inverse output rotation R^-1 is the
identity here (the value vectors carry no rotary part).  For every row t and
group g:

    z[t, g] = W_aG(g) O_G[t] + ( W_aL(g) O_L[t]  if row t is protected
                                 z_off[t, g]     otherwise )
    y[t]    = W_b z[t]

where W_aG(g) / W_aL(g) are the columns of group g's block that belong to its
Global / Local heads, O_G / O_L those heads' outputs, and z_off the cached
projected Local contribution of the document's offline pass.  Evaluated in
float64 from the given arrays.
"""
from __future__ import annotations

import numpy as np


def project_state(O: np.ndarray, z_off: np.ndarray, prot: np.ndarray, head_role: np.ndarray,
                  W_a: np.ndarray, W_b: np.ndarray, group: int = 8):
    """O [T, H, d_v]; z_off [T, G, d_g]; prot bool [T]; head_role [H] (1 Global);
    W_a [G, d_g, group * d_v]; W_b [d_model, G * d_g].  Returns (z [T, G, d_g],
    y [T, d_model]) in float64."""
    O = np.asarray(O, np.float64)
    T, H, dv = O.shape
    G = H // group
    dg = W_a.shape[1]
    z = np.zeros((T, G, dg))
    for g in range(G):
        Wg = np.asarray(W_a[g], np.float64)
        zg = np.zeros((T, dg))
        zl = np.zeros((T, dg))
        for i in range(group):
            h = g * group + i
            part = O[:, h, :] @ Wg[:, i * dv:(i + 1) * dv].T
            if head_role[h]:
                zg += part
            else:
                zl += part
        off = np.asarray(z_off[:, g, :], np.float64)
        z[:, g, :] = zg + np.where(prot[:, None], zl, off)
    y = z.reshape(T, G * dg) @ np.asarray(W_b, np.float64).T
    return z, y
