"""Pins of the oracle's RMSNorm and context projection (CPU only).

"DFlash双实现对比" (hotelren.com) §4: selected target layers are concatenated
and projected; §1: the Qwen3 RMSNorm / rotary pieces are reused.
"""
import math

import numpy as np

from oracle.dflash_oracle import ctx_project, rms_norm
from tests.test_oracle_attention import rope_complex

EPS = 1e-6


def test_rms_norm_closed_forms():
    g = np.array([1.0, 2.0, -0.5, 3.0])
    for c in (0.0, 1e-4, 2.5, -7.0):
        x = np.full(4, c)
        np.testing.assert_allclose(rms_norm(x, g, EPS), c / math.sqrt(c * c + EPS) * g,
                                   rtol=1e-15, atol=0)
    x = np.array([3.0, 4.0])               # mean square 12.5
    np.testing.assert_allclose(rms_norm(x, None, 0.0), x / math.sqrt(12.5), rtol=1e-15)
    rng = np.random.default_rng(0)
    y = rng.standard_normal((3, 64))
    np.testing.assert_allclose(rms_norm(1e3 * y, None, 0.0), rms_norm(y, None, 0.0),
                               rtol=1e-13)


def brute_ctx_project(layers, w_fc, gh, wk, wv, gk, pos, Hkv, D, theta, eps):
    N = len(layers[0])
    H = w_fc.shape[0]
    out_k = np.zeros((N, Hkv, D))
    out_v = np.zeros((N, Hkv, D))
    for n in range(N):
        x = []
        for lay in layers:
            x.extend(lay[n])
        y = [sum(w_fc[o][i] * x[i] for i in range(len(x))) for o in range(H)]
        if gh is not None:
            r = math.sqrt(sum(t * t for t in y) / H + eps)
            y = [y[o] / r * gh[o] for o in range(H)]
        for hk in range(Hkv):
            kk = [sum(wk[hk * D + d][i] * y[i] for i in range(H)) for d in range(D)]
            vv = [sum(wv[hk * D + d][i] * y[i] for i in range(H)) for d in range(D)]
            if gk is not None:
                r = math.sqrt(sum(t * t for t in kk) / D + eps)
                kk = [kk[d] / r * gk[d] for d in range(D)]
            out_k[n, hk] = rope_complex(kk, pos[n], theta)
            out_v[n, hk] = vv
    return out_k, out_v


def _case(rng, N=5, nL=3, H=8, Hkv=2, D=4):
    layers = [rng.standard_normal((N, H)) for _ in range(nL)]
    w_fc = 0.3 * rng.standard_normal((H, nL * H))
    wk = 0.3 * rng.standard_normal((Hkv * D, H))
    wv = 0.3 * rng.standard_normal((Hkv * D, H))
    gh = 1 + 0.1 * rng.standard_normal(H)
    gk = 1 + 0.1 * rng.standard_normal(D)
    pos = rng.integers(0, 500, size=N)
    return layers, w_fc, gh, wk, wv, gk, pos


def test_ctx_project_brute_force_with_and_without_norms():
    rng = np.random.default_rng(1)
    layers, w_fc, gh, wk, wv, gk, pos = _case(rng)
    for use_norm in (False, True):
        a, b = (gh, gk) if use_norm else (None, None)
        r = ctx_project(layers, w_fc, a, wk, wv, b, pos, 2, 4, 1e4, EPS)
        k, v = brute_ctx_project(layers, w_fc, a, wk, wv, b, pos, 2, 4, 1e4, EPS)
        np.testing.assert_allclose(r["k"], k, atol=1e-12)
        np.testing.assert_allclose(r["v"], v, atol=1e-12)


def test_ctx_project_is_linear_without_norms():
    rng = np.random.default_rng(2)
    l1, w_fc, _, wk, wv, _, pos = _case(rng)
    l2 = [rng.standard_normal(x.shape) for x in l1]
    mix = [2.0 * a - 0.5 * b for a, b in zip(l1, l2)]
    r1 = ctx_project(l1, w_fc, None, wk, wv, None, pos, 2, 4, 1e4, EPS)
    r2 = ctx_project(l2, w_fc, None, wk, wv, None, pos, 2, 4, 1e4, EPS)
    rm = ctx_project(mix, w_fc, None, wk, wv, None, pos, 2, 4, 1e4, EPS)
    for key in ("y", "k", "v"):
        np.testing.assert_allclose(rm[key], 2.0 * r1[key] - 0.5 * r2[key], atol=1e-12)


def test_selecting_one_layer_block_returns_that_layer():
    """W_fc = [0 | I | 0] picks the middle target layer: Y equals its hidden state,
    which fixes the concatenation order of the layers."""
    rng = np.random.default_rng(3)
    layers, _, _, wk, wv, _, pos = _case(rng, nL=3, H=8)
    for j in range(3):
        w_fc = np.zeros((8, 24))
        w_fc[:, 8 * j:8 * j + 8] = np.eye(8)
        r = ctx_project(layers, w_fc, None, wk, wv, None, pos, 2, 4, 1e4, EPS)
        np.testing.assert_array_equal(r["y"], layers[j])
        np.testing.assert_allclose(r["v"].reshape(5, 8), layers[j] @ wv.T, atol=1e-13)


def test_identity_kv_weights_expose_the_norm_and_rope():
    """With W_k = W_v = I (H = Hkv*D), V is the normalised projection itself and
    K is its per-head norm followed by the rotation of each pair."""
    rng = np.random.default_rng(4)
    layers, w_fc, gh, _, _, gk, pos = _case(rng, nL=2, H=8, Hkv=2, D=4)
    eye = np.eye(8)
    r = ctx_project(layers, w_fc, gh, eye, eye, gk, pos, 2, 4, 1e4, EPS)
    y = np.concatenate(layers, -1) @ w_fc.T
    yh = y / np.sqrt((y * y).mean(-1, keepdims=True) + EPS) * gh
    np.testing.assert_allclose(r["v"].reshape(5, 8), yh, atol=1e-13)
    for n in range(5):
        for h in range(2):
            kk = yh[n, 4 * h:4 * h + 4]
            kk = kk / math.sqrt((kk * kk).mean() + EPS) * gk
            np.testing.assert_allclose(r["k"][n, h], rope_complex(list(kk), pos[n], 1e4),
                                       atol=1e-13)
