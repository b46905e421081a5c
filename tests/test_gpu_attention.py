"""GPU parity of dflash_block_attention against the float64 oracle, through
the C ABI: contiguous and paged caches, ragged and empty contexts, GQA group
sizes 1..8, head dims 64/128, and the full-size benchmark shapes."""
import math

import numpy as np
import pytest
import torch

from oracle.dflash_oracle import block_attention as ref_attention
from synthetic import (CONFIG_BY_NAME, make_cycle_inputs, make_paged_layout, normal_bf16,
                       pack_contiguous_heads, scatter_paged_heads)
from tests.gpu_helpers import Guarded, assert_close_bf16, dev_bf16, dev_i32, host_f64

pytestmark = pytest.mark.gpu


def _dfl():
    import block_diffusion_speculative_02_gb300 as dfl
    return dfl


def run_attention(q, k, v, ctx_k, ctx_v, lens, Hq, Hkv, D, theta, paged=False, capacity=None,
                  garbage=False, seed=0, max_ctx=None):
    dfl = _dfl()
    B = q.shape[0]
    rng = np.random.default_rng(seed)
    if max_ctx is None:
        max_ctx = int(max(lens)) + 16
    dims = dfl.make_dims(B, 128, Hq, Hkv, D, 1000, 1, max_ctx, rope_theta=theta)
    ws = dfl.alloc_workspace(dims)
    if paged:
        lay = make_paged_layout(rng, lens, reserve_tokens=16)
        kp = scatter_paged_heads(lay, ctx_k, Hkv, D)      # [pages, Hkv, 16, D]
        vp = scatter_paged_heads(lay, ctx_v, Hkv, D)
        if garbage:                       # NaN bit patterns in every unused row
            for b, L in enumerate(lens):
                pg = lay.page_table[b, int(L) // 16] if L % 16 else -1
                if pg >= 0:
                    kp[pg, :, L % 16:] = 0x7FC1
                    vp[pg, :, L % 16:] = 0x7FC1
        view = dfl.KVView(dev_bf16(kp), dev_bf16(vp), dev_i32(lens), capacity=lay.max_pages * 16,
                          page_table=dev_i32(lay.page_table), free_list=dev_i32(lay.free_list),
                          free_count=dev_i32([lay.free_count]), page_size=16)
    else:
        cap = capacity or int(max(lens)) + 16
        kc = pack_contiguous_heads(ctx_k, cap, Hkv, D)       # [B, Hkv, cap, D]
        vc = pack_contiguous_heads(ctx_v, cap, Hkv, D)
        if garbage:
            for b, L in enumerate(lens):
                kc[b, :, L:] = 0x7FC1
                vc[b, :, L:] = 0xFF80
        view = dfl.KVView(dev_bf16(kc), dev_bf16(vc), dev_i32(lens), capacity=cap)
    out = Guarded((B, 16, Hq, D), torch.bfloat16, fill=float("nan"))
    dfl.dflash_block_attention(dims, dev_bf16(q), dev_bf16(k), dev_bf16(v), view,
                               1.0 / math.sqrt(D), out.t, ws)
    torch.cuda.synchronize()
    out.check()
    status = dfl.dflash_read_status(ws)
    return host_f64(out.t), status


def _rand(seed, B, Hq, Hkv, D, lens):
    rng = np.random.default_rng(seed)
    q = normal_bf16(rng, (B, 16, Hq, D))
    k = normal_bf16(rng, (B, 16, Hkv, D))
    v = normal_bf16(rng, (B, 16, Hkv, D))
    ck = [normal_bf16(rng, (int(L), Hkv, D)) for L in lens]
    cv = [normal_bf16(rng, (int(L), Hkv, D)) for L in lens]
    return q, k, v, ck, cv


@pytest.mark.parametrize("B,Hq,Hkv,D,lens,paged", [
    (1, 4, 2, 64, [128], False),              # tiny cycle shapes
    (3, 8, 2, 128, [0, 37, 300], False),      # empty + ragged contexts
    (4, 8, 2, 128, [1, 16, 700, 1333], True),  # paged, shuffled pages
    (2, 16, 2, 128, [515, 64], False),        # G = 8 (128 query rows per KV head)
    (2, 2, 2, 64, [90, 5], True),             # G = 1, head_dim 64, paged
    (1, 4, 1, 128, [4000], False),            # many splits
    # more (sequence, KV head, split) CTAs than SMs (several waves) over
    # ragged lengths, empty and one-key contexts among them
    (20, 32, 8, 128, [9000, 0, 17, 4096, 4097, 300, 8191, 1, 5000, 2500,
                      16, 6000, 700, 8192, 3333, 64, 7777, 1200, 4500, 90], True),
    (24, 16, 8, 64, [5000, 4100, 12, 0, 900] * 4 + [8200, 33, 4096, 2], False),
])
def test_attention_parity_small(B, Hq, Hkv, D, lens, paged):
    q, k, v, ck, cv = _rand(sum(lens) + B, B, Hq, Hkv, D, lens)
    ref = ref_attention(q, k, v, ck, cv, np.array(lens), 1e6, 1 / math.sqrt(D))
    got, status = run_attention(q, k, v, ck, cv, np.array(lens, np.int32), Hq, Hkv, D, 1e6,
                                paged=paged)
    assert status == 0
    print(assert_close_bf16(got, ref))


@pytest.mark.parametrize("paged", [False, True])
def test_stale_rows_past_the_length_do_not_leak(paged):
    lens = [37, 200, 16]
    q, k, v, ck, cv = _rand(11, 3, 8, 2, 128, lens)
    ref = ref_attention(q, k, v, ck, cv, np.array(lens), 1e6, 1 / math.sqrt(128))
    got, status = run_attention(q, k, v, ck, cv, np.array(lens, np.int32), 8, 2, 128, 1e6,
                                paged=paged, garbage=True)
    assert status == 0 and np.isfinite(got).all()
    assert_close_bf16(got, ref)


def test_length_past_capacity_is_flagged():
    dfl = _dfl()
    lens = [20, 10]
    q, k, v, ck, cv = _rand(12, 2, 4, 2, 64, lens)
    got, status = run_attention(q, k, v, ck, cv, np.array([20, 10], np.int32), 4, 2, 64, 1e6,
                                capacity=21)
    assert status == 0
    bad = np.array([20, 40], np.int32)             # sequence 1 claims 40 rows of a 21-row cache
    ck2 = [ck[0], np.concatenate([ck[1], ck[1], ck[1], ck[1]])]
    cv2 = [cv[0], np.concatenate([cv[1], cv[1], cv[1], cv[1]])]
    got, status = run_attention(q, k, v, [ck2[0], ck2[1][:21]], [cv2[0], cv2[1][:21]], bad, 4,
                                2, 64, 1e6, capacity=21, max_ctx=48)
    assert status & dfl.dflash.STATUS_BITS["capacity"]
    ref = ref_attention(q[:1], k[:1], v[:1], ck[:1], cv[:1], np.array([20]), 1e6, 0.125)
    assert_close_bf16(got[:1], ref)
    assert np.isnan(got[1]).all()                 # left unwritten


@pytest.mark.parametrize("name", ["tiny_b1", "qwen3_4b_b1", "qwen3_8b_b1",
                                  "qwen3_8b_b32_paged", "qwen3_32b_b4_32k"])
def test_attention_parity_full_size(name):
    cfg = CONFIG_BY_NAME[name]
    inp = make_cycle_inputs(cfg, with_lm=False)
    lens = inp.ctx_len
    ref = ref_attention(inp.q_blk, inp.k_blk, inp.v_blk, inp.ctx_k, inp.ctx_v, lens,
                        cfg.rope_theta, 1 / math.sqrt(cfg.head_dim))
    got, status = run_attention(inp.q_blk, inp.k_blk, inp.v_blk, inp.ctx_k, inp.ctx_v, lens,
                                cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.rope_theta,
                                paged=cfg.paged)
    assert status == 0
    print(cfg.name, assert_close_bf16(got, ref))
