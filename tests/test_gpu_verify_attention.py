"""GPU parity of dflash_verify_attention (the target's attention in the verify
forward: causal inside the block, block K/V appended to the cache) against the
float64 oracle, through the C ABI, contiguous and paged."""
import math

import numpy as np
import pytest
import torch

from oracle.dflash_oracle import verify_attention as ref_verify_attention
from synthetic import make_paged_layout, normal_bf16, pack_contiguous_heads, scatter_paged_heads
from tests.gpu_helpers import Guarded, assert_close_bf16, dev_bf16, dev_i32, host_bits, host_f64

pytestmark = pytest.mark.gpu


def _dfl():
    import block_diffusion_speculative_02_gb300 as dfl
    return dfl


@pytest.mark.parametrize("B,Hq,Hkv,D,lens,paged", [
    (2, 4, 2, 64, [37, 0], False),
    (2, 8, 2, 128, [300, 17], True),
    (3, 32, 8, 128, [1000, 64, 5], False),
    (1, 4, 4, 64, [4096], True),
    (1, 32, 8, 128, [8192], False),        # the Qwen3-8B batch-1 shape the bench times
    # more CTAs than SMs (several waves) over ragged lengths
    (20, 16, 8, 128, [6000, 15, 0, 4097, 300, 9000, 64, 2000, 1, 5000] * 2, True),
    # G = 8 (the Qwen3-32B heads: 128 query rows per KV head, no doubled rows)
    (2, 16, 2, 128, [515, 64], False),
    (4, 64, 8, 128, [3000, 2500, 100, 0], True),
    (4, 64, 8, 128, [32768] * 4, False),   # the Qwen3-32B batch-4 long-context shape
])
def test_verify_attention(B, Hq, Hkv, D, lens, paged):
    dfl = _dfl()
    rng = np.random.default_rng(B + D + len(lens))
    lens = np.array(lens, np.int32)
    q = normal_bf16(rng, (B, 16, Hq, D))
    k = normal_bf16(rng, (B, 16, Hkv, D))
    v = normal_bf16(rng, (B, 16, Hkv, D))
    ck = [normal_bf16(rng, (int(L), Hkv, D)) for L in lens]
    cv = [normal_bf16(rng, (int(L), Hkv, D)) for L in lens]
    theta = 1e6
    max_ctx = int(lens.max()) + 32
    dims = dfl.make_dims(B, 128, Hq, Hkv, D, 1000, 1, max_ctx, rope_theta=theta)
    ws = dfl.alloc_workspace(dims)
    if paged:
        lay = make_paged_layout(rng, lens, reserve_tokens=16, slack_pages=8)
        view = dfl.KVView(dev_bf16(scatter_paged_heads(lay, ck, Hkv, D)),
                          dev_bf16(scatter_paged_heads(lay, cv, Hkv, D)), dev_i32(lens),
                          capacity=lay.max_pages * 16, page_table=dev_i32(lay.page_table),
                          free_list=dev_i32(lay.free_list), free_count=dev_i32([lay.free_count]),
                          page_size=16)
    else:
        cap = max_ctx
        view = dfl.KVView(dev_bf16(pack_contiguous_heads(ck, cap, Hkv, D)),
                          dev_bf16(pack_contiguous_heads(cv, cap, Hkv, D)), dev_i32(lens),
                          capacity=cap)
    out = Guarded((B, 16, Hq, D), torch.bfloat16)
    dfl.dflash.dflash_verify_attention(dims, dev_bf16(q), dev_bf16(k), dev_bf16(v), view,
                                       1.0 / math.sqrt(D), out.t, ws)
    torch.cuda.synchronize()
    out.check()
    assert dfl.dflash_read_status(ws) == 0
    ref = ref_verify_attention(q, k, v, ck, cv, lens, theta, 1.0 / math.sqrt(D))
    assert_close_bf16(host_f64(out.t), ref["o"])
    assert np.array_equal(view.seq_len.cpu().numpy(), lens + 16)
    kk, vv = host_f64(view.k), host_bits(view.v)
    table = view.page_table.cpu().numpy() if paged else None
    for b in range(B):
        for j in range(16):
            r = int(lens[b]) + j
            if paged:
                pg = table[b, r // 16]
                assert pg >= 0
                krow, vrow = kk[pg, :, r % 16], vv[pg, :, r % 16]
            else:
                krow, vrow = kk[b, :, r], vv[b, :, r]
            np.testing.assert_allclose(krow, ref["k"][b, j], atol=2e-2)
            np.testing.assert_array_equal(vrow, v[b, j])        # V is appended bit for bit
    if paged:
        fc = int(view.free_count.item())
        mapped = set(table[table >= 0].tolist())
        free = set(view.free_list.cpu().numpy()[:fc].tolist())
        assert mapped.isdisjoint(free) and len(mapped) + len(free) == lay.n_pages


def test_verify_attention_full_capacity_is_flagged():
    dfl = _dfl()
    rng = np.random.default_rng(3)
    B, Hq, Hkv, D = 1, 4, 2, 64
    lens = np.array([40], np.int32)
    q = normal_bf16(rng, (B, 16, Hq, D))
    k = normal_bf16(rng, (B, 16, Hkv, D))
    v = normal_bf16(rng, (B, 16, Hkv, D))
    ck = [normal_bf16(rng, (40, Hkv, D))]
    dims = dfl.make_dims(B, 128, Hq, Hkv, D, 1000, 1, 64)
    ws = dfl.alloc_workspace(dims)
    view = dfl.KVView(dev_bf16(pack_contiguous_heads(ck, 48, Hkv, D)),
                      dev_bf16(pack_contiguous_heads(ck, 48, Hkv, D)), dev_i32(lens), capacity=48)
    out = torch.empty((B, 16, Hq, D), dtype=torch.bfloat16, device="cuda")
    dfl.dflash.dflash_verify_attention(dims, dev_bf16(q), dev_bf16(k), dev_bf16(v), view, 0.125,
                                       out, ws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) & dfl.dflash.STATUS_BITS["capacity"]
    assert int(view.seq_len.item()) == 40                      # nothing appended
