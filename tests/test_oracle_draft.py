"""Pins of the oracle's drafter-layer functions (CPU only): draft_qkv,
draft_out_mlp, draft_tokens.

"DFlash双实现对比" (hotelren.com) §1: the drafter is assembled from Qwen3
components (RMSNorm, rotary embedding, MLP); "dflash-mlx" (dpshk.com)
块扩散草稿: one forward over the block, every mask position predicts its own
token.  Each pin computes its value by a route other than the oracle's.
"""
import math

import numpy as np

from oracle.dflash_oracle import (draft_out_mlp, draft_qkv, draft_tokens, lm_head_argmax,
                                  silu)

EPS = 1e-6


def _rms(v):
    return math.sqrt(sum(t * t for t in v) / len(v) + EPS)


def brute_qkv(x, ln1, wq, wk, wv, qn, kn, Hq, Hkv, D):
    out = {"q": [], "k": [], "v": []}
    for row in x:
        r = _rms(row)
        h = [row[i] / r * ln1[i] for i in range(len(row))]
        for name, w, nh, gain in (("q", wq, Hq, qn), ("k", wk, Hkv, kn), ("v", wv, Hkv, None)):
            y = [sum(w[o][i] * h[i] for i in range(len(h))) for o in range(len(w))]
            heads = []
            for hh in range(nh):
                seg = y[hh * D:(hh + 1) * D]
                if gain is not None:
                    rs = _rms(seg)
                    seg = [seg[d] / rs * gain[d] for d in range(D)]
                heads.append(seg)
            out[name].append(heads)
    return {k: np.array(v) for k, v in out.items()}


def brute_out_mlp(x, o, wo, ln2, wg, wu, wd):
    x1s, x2s = [], []
    for row, orow in zip(x, o):
        x1 = [row[i] + sum(wo[i][j] * orow[j] for j in range(len(orow))) for i in range(len(row))]
        r = _rms(x1)
        h2 = [x1[i] / r * ln2[i] for i in range(len(x1))]
        m = []
        for f in range(len(wg)):
            a = sum(wg[f][i] * h2[i] for i in range(len(h2)))
            u = sum(wu[f][i] * h2[i] for i in range(len(h2)))
            m.append(a / (1.0 + math.exp(-a)) * u)
        x2 = [x1[i] + sum(wd[i][f] * m[f] for f in range(len(m))) for i in range(len(x1))]
        x1s.append(x1)
        x2s.append(x2)
    return np.array(x1s), np.array(x2s)


def _weights(rng, H=6, Hq=2, Hkv=1, D=4, F=5):
    return dict(ln1=1 + 0.1 * rng.standard_normal(H), wq=rng.standard_normal((Hq * D, H)),
                wk=rng.standard_normal((Hkv * D, H)), wv=rng.standard_normal((Hkv * D, H)),
                qn=1 + 0.1 * rng.standard_normal(D), kn=1 + 0.1 * rng.standard_normal(D),
                wo=rng.standard_normal((H, Hq * D)), ln2=1 + 0.1 * rng.standard_normal(H),
                wg=rng.standard_normal((F, H)), wu=rng.standard_normal((F, H)),
                wd=rng.standard_normal((H, F)))


def test_qkv_brute_force():
    rng = np.random.default_rng(0)
    w = _weights(rng)
    x = rng.standard_normal((3, 6))
    got = draft_qkv(x, w["ln1"], w["wq"], w["wk"], w["wv"], w["qn"], w["kn"], 2, 1, 4, EPS)
    ref = brute_qkv(x.tolist(), w["ln1"].tolist(), w["wq"].tolist(), w["wk"].tolist(),
                    w["wv"].tolist(), w["qn"].tolist(), w["kn"].tolist(), 2, 1, 4)
    for k in ("q", "k", "v"):
        np.testing.assert_allclose(got[k], ref[k], rtol=0, atol=1e-12)


def test_out_mlp_brute_force():
    rng = np.random.default_rng(1)
    w = _weights(rng)
    x = rng.standard_normal((3, 6))
    o = rng.standard_normal((3, 2, 4))
    got = draft_out_mlp(x, o, w["wo"], w["ln2"], w["wg"], w["wu"], w["wd"], EPS)
    x1, x2 = brute_out_mlp(x.tolist(), o.reshape(3, -1).tolist(), w["wo"].tolist(),
                           w["ln2"].tolist(), w["wg"].tolist(), w["wu"].tolist(),
                           w["wd"].tolist())
    np.testing.assert_allclose(got["x1"], x1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["x2"], x2, rtol=0, atol=1e-12)


def test_out_mlp_special_cases():
    rng = np.random.default_rng(2)
    w = _weights(rng)
    x = rng.standard_normal((4, 6))
    o = rng.standard_normal((4, 2, 4))
    # a zero gate projection switches the MLP off: silu(0) = 0
    r = draft_out_mlp(x, o, w["wo"], w["ln2"], 0 * w["wg"], w["wu"], w["wd"], EPS)
    np.testing.assert_array_equal(r["x2"], r["x1"])
    # a zero output projection leaves the residual stream unchanged
    r = draft_out_mlp(x, o, 0 * w["wo"], w["ln2"], w["wg"], w["wu"], w["wd"], EPS)
    np.testing.assert_array_equal(r["x1"], x)
    # the attention output enters linearly
    r1 = draft_out_mlp(np.zeros_like(x), o, w["wo"], w["ln2"], 0 * w["wg"], w["wu"], w["wd"], EPS)
    r2 = draft_out_mlp(np.zeros_like(x), 2 * o, w["wo"], w["ln2"], 0 * w["wg"], w["wu"], w["wd"],
                       EPS)
    np.testing.assert_allclose(r2["x1"], 2 * r1["x1"], atol=1e-12)


def test_silu_identities():
    x = np.linspace(-30, 30, 121)
    np.testing.assert_allclose(silu(x) - silu(-x), x, atol=1e-12)   # x s(x) + x s(-x) = x
    assert silu(np.array([0.0]))[0] == 0.0
    assert abs(silu(np.array([40.0]))[0] - 40.0) < 1e-12


def test_qk_norm_gives_unit_rms_heads():
    rng = np.random.default_rng(3)
    w = _weights(rng)
    x = rng.standard_normal((5, 6))
    r = draft_qkv(x, w["ln1"], w["wq"], w["wk"], w["wv"], np.ones(4), np.ones(4), 2, 1, 4, EPS)
    for t in ("q", "k"):
        ms = np.mean(r[t] ** 2, axis=-1)
        assert np.all(np.abs(ms - 1.0) < 1e-4)
    # v is not normalised and is linear in W_v
    r2 = draft_qkv(x, w["ln1"], w["wq"], w["wk"], 3 * w["wv"], None, None, 2, 1, 4, EPS)
    np.testing.assert_allclose(r2["v"], 3 * r["v"], atol=1e-12)


def test_draft_tokens_ignore_the_row_scale():
    """argmax(RMSNorm(x) g W^T) = argmax((x * g) W^T): the RMSNorm's per-row
    factor is positive, so the final norm only contributes its gains."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((32, 12))
    g = 1 + 0.1 * rng.standard_normal(12)
    w = rng.standard_normal((50, 12))
    r = draft_tokens(x, g, w, EPS, chunk=7)
    ref = lm_head_argmax(x * g, w, chunk=50)
    assert np.array_equal(r["posterior"], ref["posterior"])
    assert r["tokens"].shape == (2, 15)
    assert np.array_equal(r["tokens"], ref["posterior"].reshape(2, 16)[:, 1:])
    r3 = draft_tokens(3.5 * x, g, w, EPS)
    assert np.array_equal(r3["posterior"], r["posterior"])


def test_draft_tokens_planted():
    rng = np.random.default_rng(5)
    want = rng.integers(0, 40, size=16)
    x = rng.standard_normal((16, 10))
    w = 0.01 * rng.standard_normal((40, 10))
    for i, t in enumerate(want):
        w[t] += 4.0 * x[i] / np.linalg.norm(x[i]) ** 2
    r = draft_tokens(x, None, w, EPS)
    assert list(r["tokens"][0]) == list(want[1:])
