"""Pins of the oracle's projections (CPU): the in-projection's split follows the
pages' order (statecache.py, CacheQwen35._gdn: [mixed q|k|v, z, b, a]) --
checked with an identity weight, where each output must be a slice of the
input -- and both products are y[t][f] = sum_h x[t][h] w[f][h], checked
against a plain triple loop; the C-ABI rejects bad shapes on the host."""
import ctypes

import numpy as np
import pytest

from gated_deltanet_recurrence_delta_gb300 import build, gdn
from oracle import oracle


def test_in_proj_split_order_with_identity_weight():
    nk, nv, dk, dv = 2, 4, 8, 8
    kd, vd = nk * dk, nv * dv
    N = 2 * kd + 2 * vd + 2 * nv
    x = np.random.default_rng(0).standard_normal((5, N))
    out = oracle.in_proj(x, np.eye(N), nk, nv, dk, dv)
    o = 0
    for name, w in (("q", kd), ("k", kd), ("v", vd), ("z", vd), ("b", nv), ("a", nv)):
        assert np.array_equal(out[name], x[:, o:o + w]), name
        o += w
    assert o == N


def test_projections_against_a_triple_loop():
    rng = np.random.default_rng(1)
    M, H, nk, nv, dk, dv = 3, 5, 1, 2, 2, 2
    N = 2 * nk * dk + 2 * nv * dv + 2 * nv
    x, w = rng.integers(-3, 4, (M, H)).astype(float), rng.integers(-3, 4, (N, H)).astype(float)
    y = np.zeros((M, N))
    for t in range(M):
        for f in range(N):
            for h in range(H):
                y[t, f] += x[t, h] * w[f, h]
    out = oracle.in_proj(x, w, nk, nv, dk, dv)
    assert np.array_equal(np.concatenate([out[n] for n in ("q", "k", "v", "z", "b", "a")], 1), y)
    wo = rng.integers(-3, 4, (4, H)).astype(float)
    yo = np.array([[sum(x[t, h] * wo[f, h] for h in range(H)) for f in range(4)] for t in range(M)])
    assert np.array_equal(oracle.out_proj(x, wo), yo)


def test_projection_host_validation():
    build.build()
    lib = gdn.load_library()
    P = 1 << 30
    d = gdn.make_dims(B=1, T=1, nk=2, nv=4, dk=32, dv=32, n_slots=1)
    st = lib.gdn_in_proj(ctypes.byref(d), 4, 100, P, P, P, P, P, P, P, P, None)  # H not a multiple of 64
    assert gdn.STATUS[st] == "GDN_ERR_SHAPE"
    st = lib.gdn_in_proj(ctypes.byref(d), 4, 128, P, None, P, P, P, P, P, P, None)
    assert gdn.STATUS[st] == "GDN_ERR_ARG"
    assert lib.gdn_in_proj(ctypes.byref(d), 0, 128, P, P, P, P, P, P, P, P, None) == 0  # no tokens
    assert gdn.STATUS[lib.gdn_out_proj(4, 64, 100, P, P, P, None)] == "GDN_ERR_SHAPE"
    assert gdn.STATUS[lib.gdn_out_proj(4, 64, 128, P, P, P + 8, None)] == "GDN_ERR_ARG"
