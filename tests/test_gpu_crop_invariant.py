"""The crop invariant on the GPU ("DFlash双实现对比" (hotelren.com) §3 and
"dflash-mlx" (dpshk.com) 保证三): after every cycle the drafter context, cut
back to the committed length, holds exactly the rows that a fresh projection
of the committed tokens writes.

Cycles of the per-cycle projection (16 rows written at the drafter length)
followed by the crop to L + 1 + a are run on a context of prompt rows.  Two
fresh caches start from the same prompt rows and see only what was
committed:
  * "slots": per cycle, the same call with every uncommitted row of the block
    replaced by unrelated hidden states;
  * "packed": the committed rows of all cycles back to back, 16 per call,
    each call cropped to what is committed.
Every surviving row must be equal byte for byte.  That holds because the
projection of a row depends only on that row's hidden states and position,
and the cross-CTA sums of the stream-K GEMMs are added in a fixed order.
The shapes give tiles with up to 20 contributing CTAs (K = 5 x 1024)."""
import numpy as np
import pytest
import torch

from synthetic import (make_paged_layout, normal_bf16, pack_contiguous_heads, scatter_paged_heads,
                       unit_rms_rows_bf16)
from tests.gpu_helpers import dev_bf16, dev_i32

pytestmark = pytest.mark.gpu

B, H, HQ, HKV, D, V, NL = 2, 1024, 8, 2, 128, 4096, 5
CYCLES = 6


def _rows(view, b, n):
    """Rows 0..n-1 of sequence b as int16 bits [n, Hkv, D] (k, v)."""
    k = view.k.view(torch.int16)
    v = view.v.view(torch.int16)
    if view.page_table is None:
        return k[b, :, :n].transpose(0, 1).cpu().numpy(), v[b, :, :n].transpose(0, 1).cpu().numpy()
    table = view.page_table.cpu().numpy()[b]
    ks, vs = [], []
    for p in range((n + 15) // 16):
        m = min(16, n - 16 * p)
        ks.append(k[int(table[p]), :, :m].transpose(0, 1).cpu().numpy())
        vs.append(v[int(table[p]), :, :m].transpose(0, 1).cpu().numpy())
    return np.concatenate(ks), np.concatenate(vs)


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("sm_budget", [0, 37])
def test_cropped_context_equals_fresh_projection(paged, sm_budget):
    import block_diffusion_speculative_02_gb300 as dfl

    rng = np.random.default_rng(2024 + paged + sm_budget)
    L0 = np.array([150, 61], np.int32)
    cap = 400
    dims = dfl.make_dims(B, H, HQ, HKV, D, V, NL, cap, sm_budget=sm_budget)
    ws = dfl.alloc_workspace(dims)
    w = {n: dev_bf16(x) for n, x in dict(
        w_fc=normal_bf16(rng, (H, NL * H), 0.02), gh=normal_bf16(rng, (H,), 0.02, 1.0),
        wk=normal_bf16(rng, (HKV * D, H), 0.02), wv=normal_bf16(rng, (HKV * D, H), 0.02),
        gk=normal_bf16(rng, (D,), 0.02, 1.0)).items()}
    ctx_k = [normal_bf16(rng, (int(n), HKV, D)) for n in L0]
    ctx_v = [normal_bf16(rng, (int(n), HKV, D)) for n in L0]
    lay = make_paged_layout(rng, L0, reserve_tokens=cap - int(L0.max()), max_len=cap)

    def fresh():
        if paged:
            return dfl.KVView(dev_bf16(scatter_paged_heads(lay, ctx_k, HKV, D)),
                              dev_bf16(scatter_paged_heads(lay, ctx_v, HKV, D)), dev_i32(L0),
                              capacity=lay.max_pages * 16, page_table=dev_i32(lay.page_table),
                              free_list=dev_i32(lay.free_list),
                              free_count=dev_i32([lay.free_count]))
        return dfl.KVView(dev_bf16(pack_contiguous_heads(ctx_k, cap, HKV, D)),
                          dev_bf16(pack_contiguous_heads(ctx_v, cap, HKV, D)), dev_i32(L0),
                          capacity=cap)

    def project(view, layers):
        dfl.dflash_ctx_project(dims, [dev_bf16(x) for x in layers], w["w_fc"], w["gh"], w["wk"],
                               w["wv"], w["gk"], view.seq_len, view, ws)

    def crop(view, new_len):
        dfl.dflash_kv_crop([view], dev_i32(new_len), B, ws)

    # the cycles: project 16 rows at the drafter length, keep 1 + a of them
    blocks, accepts = [], []
    cyc = fresh()
    L = L0.copy()
    for _ in range(CYCLES):
        layers = [unit_rms_rows_bf16(rng, (B * 16, H)) for _ in range(NL)]
        a = rng.integers(0, 16, size=B)
        project(cyc, layers)
        L = L + 1 + a
        crop(cyc, L)
        blocks.append(layers)
        accepts.append(a)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    assert np.array_equal(cyc.seq_len.cpu().numpy(), L)

    # fresh, same slots: uncommitted rows of each block replaced
    slots = fresh()
    Ls = L0.copy()
    for layers, a in zip(blocks, accepts):
        other = []
        for x in layers:
            y = unit_rms_rows_bf16(rng, x.shape)
            for b in range(B):
                y[16 * b:16 * b + 1 + a[b]] = x[16 * b:16 * b + 1 + a[b]]
            other.append(y)
        project(slots, other)
        Ls = Ls + 1 + a
        crop(slots, Ls)

    # fresh, packed: the committed rows back to back, 16 per call
    committed = [[np.concatenate([layers[l][16 * b:16 * b + 1 + a[b]]
                                  for layers, a in zip(blocks, accepts)])
                  for b in range(B)] for l in range(NL)]
    n_commit = L - L0
    packed = fresh()
    done = np.zeros(B, np.int64)
    while (done < n_commit).any():
        layers = []
        for l in range(NL):
            x = unit_rms_rows_bf16(rng, (B * 16, H))
            for b in range(B):
                m = int(min(16, n_commit[b] - done[b]))
                x[16 * b:16 * b + m] = committed[l][b][done[b]:done[b] + m]
            layers.append(x)
        project(packed, layers)
        done = np.minimum(done + 16, n_commit)
        crop(packed, L0 + done)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    for view in (slots, packed):
        assert np.array_equal(view.seq_len.cpu().numpy(), L)
    for b in range(B):
        ref_k, ref_v = _rows(cyc, b, int(L[b]))
        for view in (slots, packed):
            got_k, got_v = _rows(view, b, int(L[b]))
            assert np.array_equal(got_k, ref_k), (b, np.argwhere(got_k != ref_k)[:4])
            assert np.array_equal(got_v, ref_v), (b, np.argwhere(got_v != ref_v)[:4])
    if paged:
        for view in (cyc, slots, packed):
            table = view.page_table.cpu().numpy()
            fc = int(view.free_count.item())
            mapped = set(table[table >= 0].tolist())
            free = set(view.free_list.cpu().numpy()[:fc].tolist())
            assert mapped.isdisjoint(free) and len(mapped) + len(free) == lay.n_pages
