"""Pins of the oracle's RoPE and dual-source block attention (CPU only).

What the pages fix ("DFlash双实现对比" (hotelren.com) §2): Q from the block
only, K/V = context ⊕ block, no mask inside the block.  Each pin below is
computed by a route other than the oracle's own code.
"""
import cmath
import math

import numpy as np
import pytest
import torch

from oracle.dflash_oracle import apply_rope, block_attention, rope_inv_freq

THETA = 1.0e4


def rope_complex(vec, pos, theta=THETA):
    """RoPE written as a complex rotation of the pairs (x[d], x[d+D/2])."""
    D = len(vec)
    half = D // 2
    out = [0.0] * D
    for d in range(half):
        z = complex(vec[d], vec[d + half]) * cmath.exp(1j * pos * theta ** (-2.0 * d / D))
        out[d], out[d + half] = z.real, z.imag
    return out


def brute_block_attention(q_blk, k_blk, v_blk, ctx_k, ctx_v, seq_len, theta, scale):
    B, T, Hq, D = q_blk.shape
    Hkv = k_blk.shape[2]
    out = np.zeros((B, T, Hq, D))
    for b in range(B):
        L = int(seq_len[b])
        for h in range(Hq):
            g = h * Hkv // Hq
            keys, vals = [], []
            for j in range(L):
                keys.append(list(ctx_k[b][j, g]))
                vals.append(list(ctx_v[b][j, g]))
            for j in range(T):
                keys.append(rope_complex(list(k_blk[b, j, g]), L + j, theta))
                vals.append(list(v_blk[b, j, g]))
            for i in range(T):
                q = rope_complex(list(q_blk[b, i, h]), L + i, theta)
                s = [scale * sum(q[d] * kk[d] for d in range(D)) for kk in keys]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                z = sum(e)
                for d in range(D):
                    out[b, i, h, d] = sum(e[j] * vals[j][d] for j in range(len(vals))) / z
    return out


def _rand_case(rng, B=2, T=16, Hq=4, Hkv=2, D=8, lens=(5, 0)):
    q = rng.standard_normal((B, T, Hq, D))
    k = rng.standard_normal((B, T, Hkv, D))
    v = rng.standard_normal((B, T, Hkv, D))
    ck = [rng.standard_normal((L, Hkv, D)) for L in lens]
    cv = [rng.standard_normal((L, Hkv, D)) for L in lens]
    return q, k, v, ck, cv, np.array(lens)


def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 3, 8))
    pos = rng.integers(0, 1000, size=(5, 3))
    r = apply_rope(x, pos, THETA)
    for i in range(5):
        for j in range(3):
            np.testing.assert_allclose(r[i, j], rope_complex(list(x[i, j]), pos[i, j]),
                                       rtol=0, atol=1e-12)


def test_rope_invariants():
    rng = np.random.default_rng(2)
    q = rng.standard_normal(16)
    k = rng.standard_normal(16)
    # position 0 is the identity; norm is preserved
    np.testing.assert_allclose(apply_rope(q[None], np.array([0]), 1e6)[0], q, atol=0)
    for p in (1, 17, 8191):
        assert abs(np.linalg.norm(apply_rope(q[None], np.array([p]), 1e6)) -
                   np.linalg.norm(q)) < 1e-12
    # the q.k score depends on m - n only
    def score(m, n):
        return apply_rope(q[None], np.array([m]), 1e6)[0] @ apply_rope(k[None], np.array([n]), 1e6)[0]
    for m, n, s in [(5, 2, 100), (0, 9, 3), (40, 40, 7)]:
        assert abs(score(m, n) - score(m + s, n + s)) < 1e-10
    # first pair rotates by exactly pos radians (inv_freq[0] = 1)
    assert rope_inv_freq(16, 1e6)[0] == 1.0


def test_block_attention_brute_force():
    rng = np.random.default_rng(3)
    q, k, v, ck, cv, lens = _rand_case(rng)
    scale = 1 / math.sqrt(8)
    got = block_attention(q, k, v, ck, cv, lens, THETA, scale)
    ref = brute_block_attention(q, k, v, ck, cv, lens, THETA, scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_block_attention_reduces_to_textbook_mha():
    """No context, G = 1: plain non-causal multi-head attention over the block."""
    rng = np.random.default_rng(4)
    q, k, v, ck, cv, lens = _rand_case(rng, B=1, Hq=2, Hkv=2, D=8, lens=(0,))
    got = block_attention(q, k, v, ck, cv, lens, THETA, 1 / math.sqrt(8))
    qr = np.array([[rope_complex(list(q[0, i, h]), i) for i in range(16)] for h in range(2)])
    kr = np.array([[rope_complex(list(k[0, i, h]), i) for i in range(16)] for h in range(2)])
    vr = np.transpose(v[0], (1, 0, 2))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qr)[None], torch.from_numpy(kr)[None], torch.from_numpy(vr)[None],
        is_causal=False)[0].numpy()
    np.testing.assert_allclose(got[0], np.transpose(ref, (1, 0, 2)), rtol=0, atol=1e-12)


def test_zero_query_gives_mean_of_all_values():
    rng = np.random.default_rng(5)
    q, k, v, ck, cv, lens = _rand_case(rng, B=1, lens=(7,))
    q[:] = 0.0
    got = block_attention(q, k, v, ck, cv, lens, THETA, 0.3)
    for h in range(4):
        g = h // 2
        mean = (cv[0][:, g].sum(0) + v[0, :, g].sum(0)) / (7 + 16)
        np.testing.assert_allclose(got[0, :, h], np.broadcast_to(mean, (16, 8)), atol=1e-12)


def test_dominant_context_key_selects_its_value():
    rng = np.random.default_rng(6)
    q, k, v, ck, cv, lens = _rand_case(rng, B=1, Hq=2, Hkv=1, lens=(3,))
    u = rng.standard_normal(8)
    u /= np.linalg.norm(u)
    ck[0][1, 0] = 60.0 * u
    for i in range(16):        # choose q so that RoPE_{3+i}(q_i) = u for every row
        q[0, i, :, :] = rope_complex(list(u), -(3 + i))
    got = block_attention(q, k, v, ck, cv, lens, THETA, 1.0)
    np.testing.assert_allclose(got[0], np.broadcast_to(cv[0][1, 0], (16, 2, 8)), atol=1e-9)


def test_block_is_not_causal():
    rng = np.random.default_rng(7)
    q, k, v, ck, cv, lens = _rand_case(rng, B=1, lens=(4,))
    base = block_attention(q, k, v, ck, cv, lens, THETA, 0.35)
    v2 = v.copy()
    v2[0, 15] += 1.0          # the last block row
    changed = block_attention(q, k, v2, ck, cv, lens, THETA, 0.35)
    assert np.all(np.abs(changed[0, 0] - base[0, 0]).sum(-1) > 1e-6)   # row 0 sees row 15


def test_gqa_grouping_is_consecutive():
    rng = np.random.default_rng(8)
    q, k, v, ck, cv, lens = _rand_case(rng, B=1, Hq=4, Hkv=2, lens=(6,))
    base = block_attention(q, k, v, ck, cv, lens, THETA, 0.35)
    cv2 = [c.copy() for c in cv]
    cv2[0][:, 1] += 1.0
    changed = block_attention(q, k, v, ck, cv2, lens, THETA, 0.35)
    diff = np.abs(changed - base).reshape(16, 4, 8).max(axis=(0, 2))
    assert diff[0] == 0 and diff[1] == 0 and diff[2] > 0 and diff[3] > 0


@pytest.mark.parametrize("lens", [(0,), (1,), (33,)])
def test_context_lengths_edge_cases(lens):
    rng = np.random.default_rng(9)
    q, k, v, ck, cv, L = _rand_case(rng, B=1, D=4, lens=lens)
    got = block_attention(q, k, v, ck, cv, L, THETA, 0.5)
    ref = brute_block_attention(q, k, v, ck, cv, L, THETA, 0.5)
    np.testing.assert_allclose(got, ref, atol=1e-12)


# ---------------------------------------------------------------------------
# the target's verify attention (causal inside the block)
# ---------------------------------------------------------------------------
from oracle.dflash_oracle import verify_attention  # noqa: E402


def brute_verify_attention(q_blk, k_blk, v_blk, ctx_k, ctx_v, seq_len, theta, scale):
    B, T, Hq, D = q_blk.shape
    Hkv = k_blk.shape[2]
    out = np.zeros((B, T, Hq, D))
    for b in range(B):
        L = int(seq_len[b])
        for h in range(Hq):
            g = h * Hkv // Hq
            for i in range(T):
                keys = [list(ctx_k[b][j, g]) for j in range(L)]
                vals = [list(ctx_v[b][j, g]) for j in range(L)]
                for j in range(i + 1):                     # block rows 0..i only
                    keys.append(rope_complex(list(k_blk[b, j, g]), L + j, theta))
                    vals.append(list(v_blk[b, j, g]))
                q = rope_complex(list(q_blk[b, i, h]), L + i, theta)
                s = [scale * sum(q[d] * kk[d] for d in range(D)) for kk in keys]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                z = sum(e)
                for d in range(D):
                    out[b, i, h, d] = sum(e[j] * vals[j][d] for j in range(len(vals))) / z
    return out


def test_verify_attention_brute_force():
    rng = np.random.default_rng(21)
    q, k, v, ck, cv, lens = _rand_case(rng, lens=(5, 0))
    r = verify_attention(q, k, v, ck, cv, lens, THETA, 0.4)
    ref = brute_verify_attention(q, k, v, ck, cv, lens, THETA, 0.4)
    np.testing.assert_allclose(r["o"], ref, rtol=0, atol=1e-12)
    # the appended K rows are the block keys rotated at L + j
    for j in (0, 7, 15):
        np.testing.assert_allclose(r["k"][0, j, 1], rope_complex(list(k[0, j, 1]), 5 + j),
                                   atol=1e-12)
    np.testing.assert_array_equal(r["v"], v)


def test_verify_attention_last_row_is_the_block_attention():
    """Row 15 sees every block row, so it equals the non-causal block attention;
    row 0 sees the context and block row 0 only."""
    rng = np.random.default_rng(22)
    q, k, v, ck, cv, lens = _rand_case(rng, B=1, lens=(9,))
    causal = verify_attention(q, k, v, ck, cv, lens, THETA, 0.3)["o"]
    full = block_attention(q, k, v, ck, cv, lens, THETA, 0.3)
    np.testing.assert_allclose(causal[0, 15], full[0, 15], atol=1e-12)
    assert np.abs(causal[0, 0] - full[0, 0]).max() > 1e-6
    k2, v2 = k.copy(), v.copy()
    k2[0, 1:] = rng.standard_normal(k2[0, 1:].shape)        # later rows cannot reach row 0
    v2[0, 1:] += 5.0
    again = verify_attention(q, k2, v2, ck, cv, lens, THETA, 0.3)["o"]
    np.testing.assert_array_equal(again[0, 0], causal[0, 0])


# ---------------------------------------------------------------------------
# the target's prefill attention (causal over prompt chunks)
# ---------------------------------------------------------------------------
from oracle.dflash_oracle import prefill_attention, prefill_staged  # noqa: E402


def test_prefill_attention_brute_force_ragged_chunk():
    """A chunk of 37 rows (not a multiple of 16) after 5 and after 0 cached rows."""
    rng = np.random.default_rng(31)
    q, k, v, ck, cv, lens = _rand_case(rng, T=37, lens=(5, 0))
    r = prefill_attention(q, k, v, ck, cv, lens, THETA, 0.35)
    ref = brute_verify_attention(q, k, v, ck, cv, lens, THETA, 0.35)
    np.testing.assert_allclose(r["o"], ref, rtol=0, atol=1e-12)
    for j in (0, 16, 36):
        np.testing.assert_allclose(r["k"][1, j, 0], rope_complex(list(k[1, j, 0]), j),
                                   atol=1e-12)
    np.testing.assert_array_equal(r["v"], v)


def test_prefill_attention_chunked_equals_whole():
    """Feeding a 50-row prompt as chunks of 16, 7 and 27 rows, each appended to
    the cache before the next, gives the rows of one 50-row chunk."""
    rng = np.random.default_rng(32)
    q, k, v, ck, cv, lens = _rand_case(rng, B=2, T=50, lens=(3, 0))
    whole = prefill_attention(q, k, v, ck, cv, lens, THETA, 0.3)
    cache_k = [c.copy() for c in ck]
    cache_v = [c.copy() for c in cv]
    L = lens.copy()
    outs = []
    for a, b in ((0, 16), (16, 23), (23, 50)):
        r = prefill_attention(q[:, a:b], k[:, a:b], v[:, a:b], cache_k, cache_v, L, THETA, 0.3)
        outs.append(r["o"])
        for s in range(2):
            cache_k[s] = np.concatenate([cache_k[s][:L[s]], r["k"][s]])
            cache_v[s] = np.concatenate([cache_v[s][:L[s]], r["v"][s]])
        L = L + (b - a)
    np.testing.assert_allclose(np.concatenate(outs, axis=1), whole["o"], rtol=0, atol=1e-12)
    for s in range(2):
        np.testing.assert_allclose(cache_k[s][lens[s]:], whole["k"][s], rtol=0, atol=1e-13)


def test_prefill_attention_reduces_to_textbook_causal_mha():
    """No cached rows, G = 1: plain causal multi-head attention over the chunk."""
    rng = np.random.default_rng(33)
    T = 24
    q, k, v, ck, cv, lens = _rand_case(rng, B=1, T=T, Hq=2, Hkv=2, D=8, lens=(0,))
    got = prefill_attention(q, k, v, ck, cv, lens, THETA, 1 / math.sqrt(8))["o"]
    qr = np.array([[rope_complex(list(q[0, i, h]), i) for i in range(T)] for h in range(2)])
    kr = np.array([[rope_complex(list(k[0, i, h]), i) for i in range(T)] for h in range(2)])
    vr = np.transpose(v[0], (1, 0, 2))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qr)[None], torch.from_numpy(kr)[None], torch.from_numpy(vr)[None],
        is_causal=True)[0].numpy()
    np.testing.assert_allclose(got[0], np.transpose(ref, (1, 0, 2)), rtol=0, atol=1e-12)


def test_prefill_attention_of_16_rows_is_the_verify_attention():
    rng = np.random.default_rng(34)
    q, k, v, ck, cv, lens = _rand_case(rng, lens=(11, 4))
    a = prefill_attention(q, k, v, ck, cv, lens, THETA, 0.25)
    b = verify_attention(q, k, v, ck, cv, lens, THETA, 0.25)
    for key in ("o", "k", "v"):
        np.testing.assert_allclose(a[key], b[key], rtol=0, atol=1e-12)


def test_prefill_staged_is_the_argmax_at_the_last_row():
    """The staged token: the plain argmax of the logits, lowest index on exact ties."""
    rng = np.random.default_rng(35)
    h = rng.standard_normal((3, 16))
    w = rng.standard_normal((300, 16))
    w[57] *= 5.0                                     # row 1's maximum: the pair 57, 200
    w[200] = w[57]                                   # an exact tie: 57 must win
    h[1] = w[57]
    r = prefill_staged(h, w, chunk=64)
    logits = h @ w.T
    assert list(r["staged"]) == [int(np.argmax(x)) for x in logits]
    assert r["staged"][1] == 57
