"""GPU parity of the target's prefill ("dflash-mlx" (dpshk.com) 单次前向验证
①–②): dflash_prefill_attention (causal attention over a prompt chunk, its
K/V appended to the cache) and dflash_prefill_staged (the first staged token)
against the float64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

from oracle.dflash_oracle import apply_rope, bf16_to_f64, near_tie_mask
from oracle.dflash_oracle import prefill_attention as ref_prefill
from oracle.dflash_oracle import prefill_staged as ref_staged
from synthetic import (make_paged_layout, normal_bf16, pack_contiguous_heads, scatter_paged_heads,
                       unit_rms_rows_bf16)
from tests.gpu_helpers import Guarded, assert_close_bf16, dev_bf16, dev_i32, host_bits, host_f64

pytestmark = pytest.mark.gpu

THETA = 1e6


def _dfl():
    import block_diffusion_speculative_02_gb300 as dfl
    return dfl


def _view(dfl, paged, lay, ctx_k, ctx_v, L0, cap, Hkv, D):
    if paged:
        return dfl.KVView(dev_bf16(scatter_paged_heads(lay, ctx_k, Hkv, D)),
                          dev_bf16(scatter_paged_heads(lay, ctx_v, Hkv, D)), dev_i32(L0),
                          capacity=lay.max_pages * 16, page_table=dev_i32(lay.page_table),
                          free_list=dev_i32(lay.free_list), free_count=dev_i32([lay.free_count]))
    return dfl.KVView(dev_bf16(pack_contiguous_heads(ctx_k, cap, Hkv, D)),
                      dev_bf16(pack_contiguous_heads(ctx_v, cap, Hkv, D)), dev_i32(L0),
                      capacity=cap)


def _cache_rows(view, b, r0, r1):
    """Rows r0..r1-1 of sequence b as bf16 bits [n, Hkv, D] (k, v)."""
    k = view.k.view(torch.int16)
    v = view.v.view(torch.int16)
    if view.page_table is None:
        return (k[b, :, r0:r1].transpose(0, 1).cpu().numpy().view(np.uint16),
                v[b, :, r0:r1].transpose(0, 1).cpu().numpy().view(np.uint16))
    if r1 <= r0:
        shape = (0,) + tuple(view.k.shape[1:2]) + tuple(view.k.shape[3:])
        return np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    table = view.page_table.cpu().numpy()[b]
    ks, vs = [], []
    for r in range(r0, r1):
        pg = int(table[r // 16])
        ks.append(k[pg, :, r % 16].cpu().numpy())
        vs.append(v[pg, :, r % 16].cpu().numpy())
    return np.stack(ks).view(np.uint16), np.stack(vs).view(np.uint16)


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("Hq,Hkv,D,T,lens", [
    (4, 2, 64, 37, (33, 0)),       # ragged chunk, one sequence with no cached rows
    (32, 8, 128, 100, (70, 5)),    # Qwen3-8B heads
    (8, 1, 128, 16, (200, 17)),    # G = 8: 128 query rows per KV head
    (4, 4, 64, 1, (9, 40)),        # one-row chunk, G = 1
])
def test_prefill_attention_matches_oracle(paged, Hq, Hkv, D, T, lens):
    dfl = _dfl()
    rng = np.random.default_rng(100 + T + Hq + paged)
    B = len(lens)
    L0 = np.array(lens, np.int32)
    cap = int(L0.max()) + T + 24
    ctx_k = [normal_bf16(rng, (int(n), Hkv, D)) for n in L0]
    ctx_v = [normal_bf16(rng, (int(n), Hkv, D)) for n in L0]
    q = normal_bf16(rng, (B, T, Hq, D))
    k = normal_bf16(rng, (B, T, Hkv, D))
    v = normal_bf16(rng, (B, T, Hkv, D))
    lay = make_paged_layout(rng, L0, reserve_tokens=T + 8, max_len=cap)
    view = _view(dfl, paged, lay, ctx_k, ctx_v, L0, cap, Hkv, D)
    dims = dfl.make_dims(B, 128, Hq, Hkv, D, 1000, 1, cap)
    ws = dfl.alloc_prefill_workspace(dims, T)
    out = Guarded((B, T, Hq, D), torch.bfloat16)
    scale = 1 / math.sqrt(D)
    dfl.dflash_prefill_attention(dims, T, dev_bf16(q), dev_bf16(k), dev_bf16(v), view, scale,
                                 out.t, ws)
    torch.cuda.synchronize()
    out.check()
    assert dfl.dflash_read_status(ws) == 0
    ref = ref_prefill(q, k, v, [bf16_to_f64(c) for c in ctx_k], [bf16_to_f64(c) for c in ctx_v],
                      L0, THETA, scale)
    assert_close_bf16(host_f64(out.t), ref["o"])
    assert np.array_equal(view.seq_len.cpu().numpy(), L0 + T)
    for b in range(B):
        kk, vv = _cache_rows(view, b, int(L0[b]), int(L0[b]) + T)
        np.testing.assert_allclose(bf16_to_f64(kk), ref["k"][b], atol=2e-2)
        assert np.array_equal(vv, v[b])                    # V rows are stored as given
        pk, pv = _cache_rows(view, b, 0, int(L0[b]))       # the cached rows are untouched
        assert np.array_equal(pk, ctx_k[b]) and np.array_equal(pv, ctx_v[b])
    if paged:
        table = view.page_table.cpu().numpy()
        fc = int(view.free_count.item())
        mapped = set(table[table >= 0].tolist())
        free = set(view.free_list.cpu().numpy()[:fc].tolist())
        assert mapped.isdisjoint(free) and len(mapped) + len(free) == lay.n_pages
        for b in range(B):
            assert (table[b] >= 0).sum() == -(-int(L0[b] + T) // 16)


def test_prefill_attention_chunked_equals_whole():
    """A 200-row prompt fed as chunks of 64, 100 and 36 rows gives, within the
    float bar, the output and cache rows of one 200-row chunk (both against the
    oracle, and the cache V rows byte for byte)."""
    dfl = _dfl()
    rng = np.random.default_rng(7)
    B, Hq, Hkv, D, T = 2, 32, 8, 128, 200
    L0 = np.array([0, 48], np.int32)
    cap = 300
    ctx_k = [normal_bf16(rng, (int(n), Hkv, D)) for n in L0]
    ctx_v = [normal_bf16(rng, (int(n), Hkv, D)) for n in L0]
    q = normal_bf16(rng, (B, T, Hq, D))
    k = normal_bf16(rng, (B, T, Hkv, D))
    v = normal_bf16(rng, (B, T, Hkv, D))
    scale = 1 / math.sqrt(D)
    ref = ref_prefill(q, k, v, [bf16_to_f64(c) for c in ctx_k], [bf16_to_f64(c) for c in ctx_v],
                      L0, THETA, scale)
    whole = _view(dfl, False, None, ctx_k, ctx_v, L0, cap, Hkv, D)
    dims = dfl.make_dims(B, 128, Hq, Hkv, D, 1000, 1, cap)
    ws = dfl.alloc_prefill_workspace(dims, T)
    o_whole = torch.empty((B, T, Hq, D), dtype=torch.bfloat16, device="cuda")
    dfl.dflash_prefill_attention(dims, T, dev_bf16(q), dev_bf16(k), dev_bf16(v), whole, scale,
                                 o_whole, ws)
    chunked = _view(dfl, False, None, ctx_k, ctx_v, L0, cap, Hkv, D)
    o_chunks = []
    for a, b in ((0, 64), (64, 164), (164, 200)):
        n = b - a
        wsc = dfl.alloc_prefill_workspace(dims, n)
        o = torch.empty((B, n, Hq, D), dtype=torch.bfloat16, device="cuda")
        dfl.dflash_prefill_attention(dims, n, dev_bf16(np.ascontiguousarray(q[:, a:b])),
                                     dev_bf16(np.ascontiguousarray(k[:, a:b])),
                                     dev_bf16(np.ascontiguousarray(v[:, a:b])), chunked, scale, o,
                                     wsc)
        o_chunks.append(o)
        torch.cuda.synchronize()
        assert dfl.dflash_read_status(wsc) == 0
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    o_chunk = torch.cat(o_chunks, dim=1)
    assert_close_bf16(host_f64(o_whole), ref["o"])
    assert_close_bf16(host_f64(o_chunk), ref["o"])
    assert_close_bf16(host_f64(o_chunk), host_f64(o_whole), max_abs=1e-2)
    assert np.array_equal(whole.seq_len.cpu().numpy(), L0 + T)
    assert np.array_equal(chunked.seq_len.cpu().numpy(), L0 + T)
    for b in range(B):
        kw, vw = _cache_rows(whole, b, 0, int(L0[b]) + T)
        kc, vc = _cache_rows(chunked, b, 0, int(L0[b]) + T)
        assert np.array_equal(vw, vc)
        np.testing.assert_allclose(bf16_to_f64(kc), bf16_to_f64(kw), atol=2e-2)


def test_prefill_attention_capacity_is_refused_on_the_device():
    """L + T past the capacity: DFLASH_ST_CAPACITY, and that sequence's
    length, cache and output stay as they were; the other sequence runs."""
    dfl = _dfl()
    rng = np.random.default_rng(8)
    B, Hq, Hkv, D, T = 2, 4, 2, 64, 40
    L0 = np.array([30, 70], np.int32)              # 70 + 40 > 96
    cap = 96
    ctx_k = [normal_bf16(rng, (int(n), Hkv, D)) for n in L0]
    ctx_v = [normal_bf16(rng, (int(n), Hkv, D)) for n in L0]
    view = _view(dfl, False, None, ctx_k, ctx_v, L0, cap, Hkv, D)
    k_before = view.k.clone()
    dims = dfl.make_dims(B, 128, Hq, Hkv, D, 1000, 1, cap)
    ws = dfl.alloc_prefill_workspace(dims, T)
    out = torch.full((B, T, Hq, D), 7.0, dtype=torch.bfloat16, device="cuda")
    q = normal_bf16(rng, (B, T, Hq, D))
    k = normal_bf16(rng, (B, T, Hkv, D))
    v = normal_bf16(rng, (B, T, Hkv, D))
    dfl.dflash_prefill_attention(dims, T, dev_bf16(q), dev_bf16(k), dev_bf16(v), view,
                                 1 / math.sqrt(D), out, ws)
    torch.cuda.synchronize()
    st = dfl.dflash_read_status(ws)
    assert st & dfl.dflash.STATUS_BITS["capacity"]
    assert view.seq_len.cpu().numpy().tolist() == [30 + T, 70]
    assert torch.equal(view.k[1], k_before[1])
    assert bool((out[1] == 7.0).all())
    ref = ref_prefill(q[:1], k[:1], v[:1], [bf16_to_f64(ctx_k[0])], [bf16_to_f64(ctx_v[0])],
                      L0[:1], THETA, 1 / math.sqrt(D))
    assert_close_bf16(host_f64(out[:1]), ref["o"])


@pytest.mark.parametrize("chunk,paged,Hq", [(2048, False, 32), (512, True, 32), (2048, True, 64)])
def test_prefill_attention_full_size(chunk, paged, Hq):
    """Qwen3-8B heads (32 / 8, D 128; 32 prompt rows per CTA), one 8192-token
    prompt fed in chunks of 2048 (contiguous cache) or 512 (paged, shuffled
    pool), and the Qwen3-32B heads (64 / 8: 16 rows per CTA).  Sampled rows of
    every chunk are checked against the oracle computed one row at a time
    (a row's attention only needs the rows before it, which the chunked ==
    whole pin makes exact), and every appended K row against the rotation."""
    dfl = _dfl()
    rng = np.random.default_rng(81 + chunk + Hq)
    B, Hkv, D, P = 1, 8, 128, 8192
    q = normal_bf16(rng, (B, P, Hq, D))
    k = normal_bf16(rng, (B, P, Hkv, D))
    v = normal_bf16(rng, (B, P, Hkv, D))
    L0 = np.zeros(1, np.int32)
    cap = P + 64
    lay = make_paged_layout(rng, L0, reserve_tokens=cap, max_len=cap)
    view = _view(dfl, paged, lay, [np.zeros((0, Hkv, D), np.uint16)],
                 [np.zeros((0, Hkv, D), np.uint16)], L0, cap, Hkv, D)
    dims = dfl.make_dims(B, 4096, Hq, Hkv, D, 151936, 5, cap)
    ws = dfl.alloc_prefill_workspace(dims, chunk)
    scale = 1 / math.sqrt(D)
    out = torch.empty((B, P, Hq, D), dtype=torch.bfloat16, device="cuda")
    qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    for a in range(0, P, chunk):
        o = torch.empty((B, chunk, Hq, D), dtype=torch.bfloat16, device="cuda")
        dfl.dflash_prefill_attention(dims, chunk, qd[:, a:a + chunk].contiguous(),
                                     kd[:, a:a + chunk].contiguous(),
                                     vd[:, a:a + chunk].contiguous(), view, scale, o, ws)
        out[:, a:a + chunk] = o
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    assert int(view.seq_len.item()) == P
    # the appended cache against the rotation of the inputs
    kr = apply_rope(bf16_to_f64(k[0]), np.broadcast_to(np.arange(P)[:, None], (P, Hkv)), THETA)
    kc, vc = _cache_rows(view, 0, 0, P)
    assert np.array_equal(vc, v[0])
    err = np.abs(bf16_to_f64(kc) - kr).max()
    assert err <= 2e-2, err
    # sampled rows: the first and last of every chunk and a few inside
    rows = sorted({r for a in range(0, P, chunk) for r in (a, a + 1, a + chunk // 2, a + chunk - 1)}
                  | set(rng.integers(0, P, size=8).tolist()))
    vv = bf16_to_f64(v[0])
    got = host_f64(out[0, rows])
    for i, t in enumerate(rows):
        r = ref_prefill(q[:, t:t + 1], k[:, t:t + 1], v[:, t:t + 1], [kr[:t]], [vv[:t]],
                        np.array([t]), THETA, scale)
        assert_close_bf16(got[i][None, None], r["o"])


@pytest.mark.parametrize("B,H,V", [(1, 128, 1000), (5, 256, 4097), (32, 512, 3000),
                                   (4, 4096, 151936)])
def test_prefill_staged_matches_oracle(B, H, V):
    """The first staged token from the last prompt row of a [B, T, H] array
    (row stride T * H), with the near-tie rule; w_lm rows 3 and V - 1 are an
    exact tie planted as sequence 0's maximum, which must go to row 3."""
    dfl = _dfl()
    rng = np.random.default_rng(B + V)
    T = 5
    h = unit_rms_rows_bf16(rng, (B, T, H))
    w = normal_bf16(rng, (V, H), 0.02)
    w[3] = h[0, -1]
    w[V - 1] = w[3]
    dims = dfl.make_dims(B, H, 4, 2, 64, V, 1, 64)
    ws = dfl.alloc_workspace(dims)
    staged = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    hd = dev_bf16(h)
    dfl.dflash_prefill_staged(dims, hd[:, -1], dev_bf16(w), staged, ws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    ref = ref_staged(h[:, -1], w)
    got = staged.cpu().numpy()
    tie = near_tie_mask(ref["gap"], ref["max"])
    assert np.array_equal(got[~tie], ref["staged"][~tie]), (got, ref["staged"])
    assert got[0] == 3
    # a second call on the same workspace (its keys were cleared)
    staged.fill_(-1)
    dfl.dflash_prefill_staged(dims, hd[:, -1], dev_bf16(w), staged, ws)
    torch.cuda.synchronize()
    assert np.array_equal(staged.cpu().numpy(), got)
