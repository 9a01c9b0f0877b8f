"""Pins of the projected-state oracle: special cases that reduce to one
library matmul (the unsplit projection, eq. 4's linear identity), the
replacement rule, and the second projection."""
import numpy as np

from oracle.project import project_state


def _case(seed=0, T=37, H=16, dv=24, dg=20, dm=18):
    rng = np.random.default_rng(seed)
    O = rng.standard_normal((T, H, dv))
    W_a = rng.standard_normal((H // 8, dg, 8 * dv))
    W_b = rng.standard_normal((dm, (H // 8) * dg))
    role = np.zeros(H, np.uint8)
    role[7::8] = 1
    role[2] = 1  # a group with two Global heads
    return rng, O, W_a, W_b, role


def _unsplit(O, W_a):
    T, H, dv = O.shape
    G = H // 8
    return np.stack([O.reshape(T, G, 8 * dv)[:, g, :] @ W_a[g].T for g in range(G)], axis=1)


def test_all_rows_protected_is_the_unsplit_projection():
    rng, O, W_a, W_b, role = _case()
    z_off = rng.standard_normal((O.shape[0], W_a.shape[0], W_a.shape[1]))
    z, y = project_state(O, z_off, np.ones(O.shape[0], bool), role, W_a, W_b)
    np.testing.assert_allclose(z, _unsplit(O, W_a), rtol=1e-12, atol=1e-10)


def test_exact_cache_gives_the_unsplit_projection_on_every_row():
    """Eq. 4: when the cached Local contribution is the full recomputation's,
    the split state equals the unsplit one whether a row is protected or not."""
    rng, O, W_a, W_b, role = _case(1)
    T, H, dv = O.shape
    O_L = O * (role == 0)[None, :, None]
    z_off = _unsplit(O_L, W_a)
    prot = rng.random(T) < 0.3
    z, y = project_state(O, z_off, prot, role, W_a, W_b)
    np.testing.assert_allclose(z, _unsplit(O, W_a), rtol=1e-12, atol=1e-10)
    np.testing.assert_allclose(y, _unsplit(O, W_a).reshape(T, -1) @ W_b.T, rtol=1e-12,
                               atol=1e-9)


def test_replacement_never_adds():
    rng, O, W_a, W_b, role = _case(2)
    T = O.shape[0]
    prot = rng.random(T) < 0.5
    z_off = rng.standard_normal((T, W_a.shape[0], W_a.shape[1]))
    z1, _ = project_state(O, z_off, prot, role, W_a, W_b)
    bump = rng.standard_normal(z_off.shape)
    z2, _ = project_state(O, z_off + bump, prot, role, W_a, W_b)
    np.testing.assert_array_equal(z1[prot], z2[prot])
    np.testing.assert_allclose(z2[~prot] - z1[~prot], bump[~prot], rtol=1e-12, atol=1e-12)


def test_unprotected_rows_are_global_part_plus_cache():
    rng, O, W_a, W_b, role = _case(3)
    T = O.shape[0]
    z_off = rng.standard_normal((T, W_a.shape[0], W_a.shape[1]))
    z, y = project_state(O, z_off, np.zeros(T, bool), role, W_a, W_b)
    O_G = O * (role == 1)[None, :, None]
    np.testing.assert_allclose(z, _unsplit(O_G, W_a) + z_off, rtol=1e-12, atol=1e-10)
    np.testing.assert_allclose(y, z.reshape(T, -1) @ W_b.T, rtol=1e-12, atol=1e-9)
