"""GPU parity of the drafter-layer calls (dflash_draft_qkv, dflash_draft_mlp,
dflash_draft_tokens) against the float64 oracle, through the C ABI, and of the
whole drafter layer composed with dflash_block_attention."""
import math

import numpy as np
import pytest
import torch

from oracle.dflash_oracle import bf16_to_f64
from oracle.dflash_oracle import block_attention as ref_attention
from oracle.dflash_oracle import draft_out_mlp, draft_qkv, draft_tokens
from synthetic import normal_bf16, pack_contiguous_heads, unit_rms_rows_bf16
from tests.gpu_helpers import (Guarded, assert_close_bf16, assert_close_bf16_wide, check_verify,
                               dev_bf16, dev_i32, host_bits, host_f64)

pytestmark = pytest.mark.gpu


def _dfl():
    import block_diffusion_speculative_02_gb300 as dfl
    return dfl


def layer_weights(rng, H, Hq, Hkv, D, F, norms=True):
    w = dict(ln1=normal_bf16(rng, (H,), 0.02, 1.0), wq=normal_bf16(rng, (Hq * D, H), 0.02),
             wk=normal_bf16(rng, (Hkv * D, H), 0.02), wv=normal_bf16(rng, (Hkv * D, H), 0.02),
             qn=normal_bf16(rng, (D,), 0.02, 1.0) if norms else None,
             kn=normal_bf16(rng, (D,), 0.02, 1.0) if norms else None,
             wo=normal_bf16(rng, (H, Hq * D), 0.02), ln2=normal_bf16(rng, (H,), 0.02, 1.0),
             wg=normal_bf16(rng, (F, H), 0.02), wu=normal_bf16(rng, (F, H), 0.02),
             wd=normal_bf16(rng, (H, F), 0.02), fn=normal_bf16(rng, (H,), 0.02, 1.0))
    return w


def _d(x):
    return None if x is None else dev_bf16(x)


def run_qkv(dfl, dims, x, w, Hq, Hkv, D, ws):
    n = x.shape[0]
    q = Guarded((n, Hq * D), torch.bfloat16)
    k = Guarded((n, Hkv * D), torch.bfloat16)
    v = Guarded((n, Hkv * D), torch.bfloat16)
    dfl.dflash.dflash_draft_qkv(dims, dev_bf16(x), dev_bf16(w["ln1"]), dev_bf16(w["wq"]),
                                dev_bf16(w["wk"]), dev_bf16(w["wv"]), _d(w["qn"]), _d(w["kn"]),
                                q.t, k.t, v.t, ws)
    torch.cuda.synchronize()
    for g in (q, k, v):
        g.check()
    return q.t, k.t, v.t


@pytest.mark.parametrize("B,H,Hq,Hkv,D,norms", [
    (1, 256, 4, 2, 64, True),
    (2, 256, 4, 2, 64, False),
    (17, 512, 8, 2, 128, True),      # 272 token rows: three 128-row chunks
    (32, 256, 4, 2, 64, True),       # the largest batch (512 token rows)
    (20, 512, 8, 2, 128, True),      # tiled: 256-feature tiles of q and k|v
    (24, 512, 8, 2, 128, False),
])
def test_draft_qkv(B, H, Hq, Hkv, D, norms):
    dfl = _dfl()
    rng = np.random.default_rng(B + H)
    w = layer_weights(rng, H, Hq, Hkv, D, 256, norms)
    x = unit_rms_rows_bf16(rng, (B * 16, H))
    dims = dfl.make_dims(B, H, Hq, Hkv, D, 1000, 1, 64)
    ws = dfl.dflash.alloc_draft_workspace(dims, 256)
    q, k, v = run_qkv(dfl, dims, x, w, Hq, Hkv, D, ws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    ref = draft_qkv(x, w["ln1"], w["wq"], w["wk"], w["wv"], w["qn"], w["kn"], Hq, Hkv, D, 1e-6)
    assert_close_bf16(host_f64(q).reshape(B * 16, Hq, D), ref["q"])
    assert_close_bf16(host_f64(k).reshape(B * 16, Hkv, D), ref["k"])
    assert_close_bf16(host_f64(v).reshape(B * 16, Hkv, D), ref["v"])


@pytest.mark.parametrize("B,H,Hq,D,F", [
    (1, 256, 4, 64, 512),
    (2, 384, 4, 128, 640),
    (17, 256, 4, 64, 384),           # 272 token rows: the tiled gate/up and down GEMMs
    (32, 256, 4, 64, 384),           # the largest batch (512 token rows)
    (20, 384, 4, 128, 640),          # tiled, hidden not a multiple of 256 (128-wide down tiles)
])
def test_draft_mlp(B, H, Hq, D, F):
    dfl = _dfl()
    rng = np.random.default_rng(B * 7 + F)
    w = layer_weights(rng, H, Hq, 2, D, F)
    x = unit_rms_rows_bf16(rng, (B * 16, H))
    o = normal_bf16(rng, (B * 16, Hq * D), 0.5)
    dims = dfl.make_dims(B, H, Hq, 2, D, 1000, 1, 64)
    ws = dfl.dflash.alloc_draft_workspace(dims, F)
    guarded = Guarded((B * 16, H), torch.bfloat16)
    out = guarded.t
    for _ in range(2):               # the second call finds the workspace as the first left it
        dfl.dflash.dflash_draft_mlp(dims, F, dev_bf16(x), dev_bf16(o), dev_bf16(w["wo"]),
                                    dev_bf16(w["ln2"]), dev_bf16(w["wg"]), dev_bf16(w["wu"]),
                                    dev_bf16(w["wd"]), out, ws)
        torch.cuda.synchronize()
        guarded.check()
        assert dfl.dflash_read_status(ws) == 0
        ref = draft_out_mlp(x, o, w["wo"], w["ln2"], w["wg"], w["wu"], w["wd"], 1e-6)
        assert np.abs(ref["x2"]).max() < 8          # bf16 half-ulp stays below the tolerance
        assert_close_bf16(host_f64(out), ref["x2"])


def test_draft_mlp_output_may_alias_input():
    dfl = _dfl()
    rng = np.random.default_rng(3)
    B, H, Hq, D, F = 1, 256, 4, 64, 256
    w = layer_weights(rng, H, Hq, 2, D, F)
    x = unit_rms_rows_bf16(rng, (B * 16, H))
    o = normal_bf16(rng, (B * 16, Hq * D), 0.5)
    dims = dfl.make_dims(B, H, Hq, 2, D, 1000, 1, 64)
    ws = dfl.dflash.alloc_draft_workspace(dims, F)
    xd = dev_bf16(x)
    dfl.dflash.dflash_draft_mlp(dims, F, xd, dev_bf16(o), dev_bf16(w["wo"]), dev_bf16(w["ln2"]),
                                dev_bf16(w["wg"]), dev_bf16(w["wu"]), dev_bf16(w["wd"]), xd, ws)
    torch.cuda.synchronize()
    ref = draft_out_mlp(x, o, w["wo"], w["ln2"], w["wg"], w["wu"], w["wd"], 1e-6)
    assert_close_bf16(host_f64(xd), ref["x2"])


@pytest.mark.parametrize("B,H,V", [(1, 256, 4096), (3, 512, 12345), (32, 256, 9001)])
def test_draft_tokens(B, H, V):
    dfl = _dfl()
    rng = np.random.default_rng(V)
    x = unit_rms_rows_bf16(rng, (B * 16, H))
    fn = normal_bf16(rng, (H,), 0.02, 1.0)
    w_lm = normal_bf16(rng, (V, H), 0.02)
    dims = dfl.make_dims(B, H, 4, 4, 128, V, 1, 64)
    ws = dfl.dflash.alloc_draft_workspace(dims, 128)
    staged = dev_i32(rng.integers(0, V, size=B))
    gblk = Guarded((B, 16), torch.int32, fill=-5)
    gpost = Guarded((B, 16), torch.int32, fill=0)
    blk, post = gblk.t, gpost.t
    for _ in range(2):
        dfl.dflash.dflash_draft_tokens(dims, dev_bf16(x), dev_bf16(fn), dev_bf16(w_lm), staged,
                                       blk, post, ws)
        torch.cuda.synchronize()
        gblk.check()
        gpost.check()
        assert dfl.dflash_read_status(ws) == 0
        ref = draft_tokens(x, fn, w_lm, 1e-6)
        got = post.cpu().numpy().reshape(-1)
        tie = (ref["gap"] <= 1e-3 * np.abs(ref["max"]))
        assert np.array_equal(got[~tie], ref["posterior"][~tie])
        b_np = blk.cpu().numpy()
        assert np.array_equal(b_np[:, 0], staged.cpu().numpy())
        assert np.array_equal(b_np[:, 1:], post.cpu().numpy()[:, 1:])
    # without a staged token, position 0 is left alone
    blk.fill_(-5)
    dfl.dflash.dflash_draft_tokens(dims, dev_bf16(x), None, dev_bf16(w_lm), None, blk, None, ws)
    torch.cuda.synchronize()
    assert np.all(blk.cpu().numpy()[:, 0] == -5)


def test_drafter_layer_composed():
    """x -> Q/K/V -> dual-source attention -> o-proj + MLP -> tokens on the
    GPU against the oracle chain in float64 from the same inputs."""
    dfl = _dfl()
    rng = np.random.default_rng(11)
    B, H, Hq, Hkv, D, F, V = 2, 256, 4, 2, 64, 512, 4096
    w = layer_weights(rng, H, Hq, Hkv, D, F)
    w_lm = normal_bf16(rng, (V, H), 0.02)
    L = np.array([70, 33], np.int32)
    cap = 128
    ctx_k = [normal_bf16(rng, (int(n), Hkv, D)) for n in L]
    ctx_v = [normal_bf16(rng, (int(n), Hkv, D)) for n in L]
    x = unit_rms_rows_bf16(rng, (B * 16, H))
    dims = dfl.make_dims(B, H, Hq, Hkv, D, V, 1, cap)
    ws = dfl.alloc_workspace(dims)
    dws = dfl.dflash.alloc_draft_workspace(dims, F)
    cache = dfl.KVView(dev_bf16(pack_contiguous_heads(ctx_k, cap, Hkv, D)),
                       dev_bf16(pack_contiguous_heads(ctx_v, cap, Hkv, D)), dev_i32(L),
                       capacity=cap)
    q, k, v = run_qkv(dfl, dims, x, w, Hq, Hkv, D, dws)
    attn = torch.empty((B, 16, Hq, D), dtype=torch.bfloat16, device="cuda")
    dfl.dflash_block_attention(dims, q.view(B, 16, Hq, D), k.view(B, 16, Hkv, D),
                               v.view(B, 16, Hkv, D), cache, 1 / math.sqrt(D), attn, ws)
    xo = torch.empty((B * 16, H), dtype=torch.bfloat16, device="cuda")
    dfl.dflash.dflash_draft_mlp(dims, F, dev_bf16(x), attn.view(B * 16, Hq * D), dev_bf16(w["wo"]),
                                dev_bf16(w["ln2"]), dev_bf16(w["wg"]), dev_bf16(w["wu"]),
                                dev_bf16(w["wd"]), xo, dws)
    blk = torch.zeros((B, 16), dtype=torch.int32, device="cuda")
    post = torch.zeros((B, 16), dtype=torch.int32, device="cuda")
    dfl.dflash.dflash_draft_tokens(dims, xo, dev_bf16(w["fn"]), dev_bf16(w_lm), None, blk, post,
                                   dws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0 and dfl.dflash_read_status(dws) == 0
    r = draft_qkv(x, w["ln1"], w["wq"], w["wk"], w["wv"], w["qn"], w["kn"], Hq, Hkv, D, 1e-6)
    o = ref_attention(r["q"].reshape(B, 16, Hq, D), r["k"].reshape(B, 16, Hkv, D),
                      r["v"].reshape(B, 16, Hkv, D), [bf16_to_f64(c) for c in ctx_k],
                      [bf16_to_f64(c) for c in ctx_v], L, 1e6, 1 / math.sqrt(D))
    assert_close_bf16(host_f64(attn), o)
    x2 = draft_out_mlp(x, o.reshape(B * 16, -1), w["wo"], w["ln2"], w["wg"], w["wu"], w["wd"],
                       1e-6)["x2"]
    assert_close_bf16(host_f64(xo), x2)
    # tokens: the oracle takes the GPU's bf16 layer output, as the GPU does
    t = draft_tokens(host_bits(xo), w["fn"], w_lm, 1e-6)
    tie = t["gap"] <= 1e-3 * np.abs(t["max"])
    got = post.cpu().numpy().reshape(-1)
    assert np.array_equal(got[~tie], t["posterior"][~tie])


@pytest.mark.parametrize("name", ["qwen3_8b_b1", "qwen3_32b_b4_32k"])
def test_drafter_layer_full_size(name):
    """Qwen3-8B / Qwen3-32B shapes (MLP width 12288 / 25600), batch 1 / 4, with
    the workload's weight distribution (std 0.02 throughout).  The layer output
    then passes 8 in places; there the bar is max-abs 2e-2 plus half a bf16 ulp
    of the float64 value (the rounding of the stored result alone), and the
    number of such elements is printed."""
    from synthetic import CONFIG_BY_NAME
    dfl = _dfl()
    cfg = CONFIG_BY_NAME[name]
    F = {4096: 12288, 5120: 25600}[cfg.hidden]
    rng = np.random.default_rng(5)
    B, H, Hq, Hkv, D = cfg.batch, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    w = layer_weights(rng, H, Hq, Hkv, D, F)
    x = unit_rms_rows_bf16(rng, (B * 16, H))
    o = normal_bf16(rng, (B * 16, Hq * D), 0.3)
    dims = dfl.make_dims(B, H, Hq, Hkv, D, cfg.vocab, 1, 64)
    dws = dfl.dflash.alloc_draft_workspace(dims, F)
    q, k, v = run_qkv(dfl, dims, x, w, Hq, Hkv, D, dws)
    xo = torch.empty((B * 16, H), dtype=torch.bfloat16, device="cuda")
    dfl.dflash.dflash_draft_mlp(dims, F, dev_bf16(x), dev_bf16(o), dev_bf16(w["wo"]),
                                dev_bf16(w["ln2"]), dev_bf16(w["wg"]), dev_bf16(w["wu"]),
                                dev_bf16(w["wd"]), xo, dws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(dws) == 0
    r = draft_qkv(x, w["ln1"], w["wq"], w["wk"], w["wv"], w["qn"], w["kn"], Hq, Hkv, D, 1e-6)
    assert_close_bf16_wide(host_f64(q).reshape(-1, Hq, D), r["q"])
    assert_close_bf16_wide(host_f64(k).reshape(-1, Hkv, D), r["k"])
    assert_close_bf16_wide(host_f64(v).reshape(-1, Hkv, D), r["v"])
    x2 = draft_out_mlp(x, o, w["wo"], w["ln2"], w["wg"], w["wu"], w["wd"], 1e-6)["x2"]
    info = assert_close_bf16_wide(host_f64(xo), x2)
    print(f"{name}: layer output max |x2| {info['max_ref']:.2f}, {info['n_wide']} of {x2.size} "
          f"elements at |x2| >= 8, max-abs error {info['max_abs']:.4f} "
          f"({info['max_abs_narrow']:.4f} below 8), rel-L2 {info['rel_l2']:.2e}")
