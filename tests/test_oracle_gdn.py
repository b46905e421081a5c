"""Pins of the oracle's GatedDeltaNet tape-replay rollback (CPU only).

"dflash-mlx" (dpshk.com) 保证三 and "DFlash双实现对比" (hotelren.com) §7: the
recurrent state of a hybrid target cannot be cut back like a KV cache; the
verify forward records each step's innovation and the rollback replays only
the accepted steps.  Each pin below comes from the algebra of the delta rule,
not from the oracle's own code path.
"""
import numpy as np

from oracle.dflash_oracle import gdn_replay, gdn_step


def _tape(rng, B=2, T=16, NH=3, Dk=6, Dv=5, unit=True):
    k = rng.standard_normal((B, T, NH, Dk))
    if unit:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, NH, Dv))
    beta = rng.uniform(0.1, 0.9, size=(B, T, NH))
    g = -rng.uniform(0.0, 0.5, size=(B, T, NH))
    S0 = rng.standard_normal((B, NH, Dv, Dk))
    return S0, k, v, beta, g


def test_zero_steps_leave_the_state():
    rng = np.random.default_rng(0)
    S0, k, v, beta, g = _tape(rng)
    np.testing.assert_array_equal(gdn_replay(S0, k, v, beta, g, [0, 0]), S0)


def test_delta_rule_writes_v_at_k():
    """With no decay and beta = 1 the updated state maps the (unit) key to its
    value exactly: S (I - k k^T) k + v k^T k = v."""
    rng = np.random.default_rng(1)
    S = rng.standard_normal((5, 6))
    k = rng.standard_normal(6)
    k /= np.linalg.norm(k)
    v = rng.standard_normal(5)
    S1 = gdn_step(S, k, v, 1.0, 0.0)
    np.testing.assert_allclose(S1 @ k, v, atol=1e-12)
    # directions orthogonal to k are untouched
    w = rng.standard_normal(6)
    w -= (w @ k) * k
    np.testing.assert_allclose(S1 @ w, S @ w, atol=1e-12)


def test_pure_gate_scales_the_state():
    rng = np.random.default_rng(2)
    S0, k, v, beta, g = _tape(rng)
    beta[:] = 0.0
    out = gdn_replay(S0, k, v, beta, g, [4, 9])
    for b, n in enumerate((4, 9)):
        np.testing.assert_allclose(out[b], S0[b] * np.exp(g[b, :n].sum(0))[:, None, None],
                                   rtol=1e-12)


def test_rank_one_form_and_brute_force():
    """The update equals a*S - a*beta*(S k) k^T + beta v k^T written out by
    element, in plain Python."""
    rng = np.random.default_rng(3)
    S = rng.standard_normal((3, 4))
    k, v = rng.standard_normal(4), rng.standard_normal(3)
    beta, g = 0.37, -0.2
    a = float(np.exp(g))
    Sk = [sum(S[i][j] * k[j] for j in range(4)) for i in range(3)]
    ref = [[a * S[i][j] - a * beta * Sk[i] * k[j] + beta * v[i] * k[j] for j in range(4)]
           for i in range(3)]
    np.testing.assert_allclose(gdn_step(S, k, v, beta, g), ref, atol=1e-12)


def test_replay_composes():
    """Replaying n steps and then the next m equals replaying n + m steps."""
    rng = np.random.default_rng(4)
    S0, k, v, beta, g = _tape(rng, B=1)
    n, m = 5, 7
    mid = gdn_replay(S0, k, v, beta, g, [n])
    rest = gdn_replay(mid, k[:, n:], v[:, n:], beta[:, n:], g[:, n:], [m])
    np.testing.assert_allclose(rest, gdn_replay(S0, k, v, beta, g, [n + m]), atol=1e-12)
