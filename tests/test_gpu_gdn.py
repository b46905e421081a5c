"""GPU parity of dflash_gdn_replay (tape-replay rollback of GatedDeltaNet
states) against the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from oracle.dflash_oracle import gdn_replay as ref_replay
from synthetic import normal_bf16
from tests.gpu_helpers import dev_bf16, dev_i32

pytestmark = pytest.mark.gpu


def _case(rng, B, NH, Dk, Dv):
    k = rng.standard_normal((B, 16, NH, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)          # the layer L2-normalises its keys
    from synthetic import f32_to_bf16_bits
    k_bits = f32_to_bf16_bits(k.astype(np.float32))
    v_bits = normal_bf16(rng, (B, 16, NH, Dv))
    beta = rng.uniform(0.05, 0.95, size=(B, 16, NH)).astype(np.float32)
    g = (-rng.uniform(0.0, 0.3, size=(B, 16, NH))).astype(np.float32)
    S0 = (0.3 * rng.standard_normal((B, NH, Dv, Dk))).astype(np.float32)
    return S0, k_bits, v_bits, beta, g


@pytest.mark.parametrize("B,NH,Dk,Dv", [(1, 4, 128, 128), (3, 5, 64, 128), (2, 7, 128, 64),
                                        (4, 3, 64, 64)])
def test_gdn_replay(B, NH, Dk, Dv):
    import block_diffusion_speculative_02_gb300 as dfl
    rng = np.random.default_rng(B * 100 + NH)
    S0, kb, vb, beta, g = _case(rng, B, NH, Dk, Dv)
    acc = rng.integers(0, 16, size=B).astype(np.int32)
    acc[0] = 15
    state = torch.from_numpy(S0.copy()).cuda()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    dfl.dflash.dflash_gdn_replay(state, dev_bf16(kb), dev_bf16(vb), torch.from_numpy(beta).cuda(),
                                 torch.from_numpy(g).cuda(), dev_i32(acc), ws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    from oracle.dflash_oracle import bf16_to_f64
    ref = ref_replay(S0, bf16_to_f64(kb), bf16_to_f64(vb), beta.astype(np.float64),
                     g.astype(np.float64), acc + 1)
    got = state.cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert err.max() <= 1e-4 * max(1.0, np.abs(ref).max()), err.max()


@pytest.mark.parametrize("Dv", [64, 128])
@pytest.mark.parametrize("g_lo,g_hi", [(-40.0, -20.0), (-400.0, -100.0), (-60.0, 0.0)])
def test_gdn_replay_strong_decay(g_lo, g_hi, Dv):
    """Decays whose running product leaves the fp32 range of a scale factor
    (and, at -100 and below, exp(g) that underflows to zero): the replay must
    still follow the recurrence step by step."""
    import block_diffusion_speculative_02_gb300 as dfl
    from oracle.dflash_oracle import bf16_to_f64
    rng = np.random.default_rng(int(-g_lo) + Dv)
    B, NH, Dk = 2, 3, 128
    S0, kb, vb, beta, _ = _case(rng, B, NH, Dk, Dv)
    g = rng.uniform(g_lo, g_hi, size=(B, 16, NH)).astype(np.float32)
    g[:, ::4] = -0.01                  # some steps barely decay
    acc = np.array([15, 9], np.int32)
    state = torch.from_numpy(S0.copy()).cuda()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    dfl.dflash.dflash_gdn_replay(state, dev_bf16(kb), dev_bf16(vb), torch.from_numpy(beta).cuda(),
                                 torch.from_numpy(g).cuda(), dev_i32(acc), ws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    ref = ref_replay(S0, bf16_to_f64(kb), bf16_to_f64(vb), beta.astype(np.float64),
                     g.astype(np.float64), acc + 1)
    got = state.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    assert np.abs(got - ref).max() <= 1e-4 * max(1.0, np.abs(ref).max())


@pytest.mark.parametrize("Dk,Dv", [(128, 128), (64, 128), (128, 64)])
def test_gdn_replay_many_heads(Dk, Dv):
    """More 32-row blocks than can be resident at once (several waves of
    CTAs), over four sequences of which one has an invalid accept length and
    must keep its state as it was."""
    import block_diffusion_speculative_02_gb300 as dfl
    from oracle.dflash_oracle import bf16_to_f64
    rng = np.random.default_rng(Dk + Dv)
    B, NH = 4, 500
    S0, kb, vb, beta, g = _case(rng, B, NH, Dk, Dv)
    acc = np.array([5, 16, 15, 0], np.int32)
    state = torch.from_numpy(S0.copy()).cuda()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    dfl.dflash.dflash_gdn_replay(state, dev_bf16(kb), dev_bf16(vb), torch.from_numpy(beta).cuda(),
                                 torch.from_numpy(g).cuda(), dev_i32(acc), ws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) & dfl.dflash.STATUS_BITS["capacity"]
    got = state.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(got[1], S0[1])
    ok = [0, 2, 3]
    ref = ref_replay(S0[ok], bf16_to_f64(kb[ok]), bf16_to_f64(vb[ok]),
                     beta[ok].astype(np.float64), g[ok].astype(np.float64), acc[ok] + 1)
    assert np.abs(got[ok] - ref).max() <= 1e-4 * max(1.0, np.abs(ref).max())


def test_gdn_replay_bad_accept_length_is_flagged():
    import block_diffusion_speculative_02_gb300 as dfl
    rng = np.random.default_rng(9)
    S0, kb, vb, beta, g = _case(rng, 2, 3, 64, 64)
    state = torch.from_numpy(S0.copy()).cuda()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    dfl.dflash.dflash_gdn_replay(state, dev_bf16(kb), dev_bf16(vb), torch.from_numpy(beta).cuda(),
                                 torch.from_numpy(g).cuda(), dev_i32([16, 3]), ws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) & dfl.dflash.STATUS_BITS["capacity"]
    np.testing.assert_array_equal(state.cpu().numpy()[0], S0[0])    # untouched
    assert not np.array_equal(state.cpu().numpy()[1], S0[1])
