"""Several consecutive draft/verify cycles on the GPU, state carried on the
device (write position aliasing the drafter length, committed length
aliasing the next cycle's len_before), against the oracle run through the
same sequence: ctx rows, lengths, pages, tokens and attention outputs."""
import math

import numpy as np
import pytest
import torch

from oracle.dflash_oracle import block_attention as ref_attention
from oracle.dflash_oracle import ctx_project as ref_project
from oracle.dflash_oracle import bf16_to_f64, kv_crop_lengths, near_tie_mask
from oracle.dflash_oracle import verify_accept as ref_verify
from synthetic import (draw_accept_lengths, make_block_ids, make_paged_layout, normal_bf16,
                       pack_contiguous_heads, scatter_paged_heads, unit_rms_rows_bf16)
from tests.gpu_helpers import assert_close_bf16, check_verify, dev_bf16, dev_i32, host_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("concurrent", [True, False])
@pytest.mark.parametrize("paged", [False, True])
def test_three_cycles_carry_state(paged, concurrent):
    import block_diffusion_speculative_02_gb300 as dfl
    from block_diffusion_speculative_02_gb300.cycle import CycleState, CycleWeights, run_cycle

    rng = np.random.default_rng(42 + paged)
    B, H, Hq, Hkv, D, V, nL = 2, 256, 4, 2, 64, 4096, 2
    theta, eps = 1e6, 1e-6
    L0 = np.array([100, 37], np.int32)
    w_lm = normal_bf16(rng, (V, H), 0.02)
    w_fc = normal_bf16(rng, (H, nL * H), 0.02)
    gh = normal_bf16(rng, (H,), 0.02, 1.0)
    wk = normal_bf16(rng, (Hkv * D, H), 0.02)
    wv = normal_bf16(rng, (Hkv * D, H), 0.02)
    gk = normal_bf16(rng, (D,), 0.02, 1.0)
    ctx_k = [normal_bf16(rng, (int(L), Hkv, D)) for L in L0]
    ctx_v = [normal_bf16(rng, (int(L), Hkv, D)) for L in L0]
    cap = 200
    dims = dfl.make_dims(B, H, Hq, Hkv, D, V, nL, cap, theta, eps)
    ws = dfl.alloc_workspace(dims)
    if paged:
        lay = make_paged_layout(rng, L0, reserve_tokens=64, max_len=cap)
        draft = dfl.KVView(dev_bf16(scatter_paged_heads(lay, ctx_k, Hkv, D)),
                           dev_bf16(scatter_paged_heads(lay, ctx_v, Hkv, D)), dev_i32(L0),
                           capacity=lay.max_pages * 16, page_table=dev_i32(lay.page_table),
                           free_list=dev_i32(lay.free_list), free_count=dev_i32([lay.free_count]))
    else:
        draft = dfl.KVView(dev_bf16(pack_contiguous_heads(ctx_k, cap, Hkv, D)),
                           dev_bf16(pack_contiguous_heads(ctx_v, cap, Hkv, D)), dev_i32(L0),
                           capacity=cap)
    target = dfl.KVView(None, None, dev_i32(L0 + 16), capacity=cap)
    w = CycleWeights(dev_bf16(w_lm), dev_bf16(w_fc), dev_bf16(gh), dev_bf16(wk), dev_bf16(wv),
                     dev_bf16(gk))
    commit = dev_i32(L0)                         # len_before of the next cycle aliases it
    out_tokens = torch.full((B, cap + 16), -1, dtype=torch.int32, device="cuda")
    ref_out = np.full((B, cap + 16), -1, np.int32)
    # oracle state: float64 context rows and lengths
    ref_k = [bf16_to_f64(x) for x in ctx_k]
    ref_v = [bf16_to_f64(x) for x in ctx_v]
    L = L0.copy()
    for cyc in range(3):
        # verify inputs without near ties (the rule would exclude them and the two
        # sides' states could then diverge in the next cycle)
        while True:
            hv = unit_rms_rows_bf16(rng, (B, 16, H))
            probe = ref_verify(hv, w_lm, np.zeros((B, 16), np.int32), L, out_cap=cap + 16)
            if not near_tie_mask(probe["gap"], probe["max"]).any():
                break
        layers = [unit_rms_rows_bf16(rng, (B * 16, H)) for _ in range(nL)]
        q = normal_bf16(rng, (B, 16, Hq, D))
        kb = normal_bf16(rng, (B, 16, Hkv, D))
        vb = normal_bf16(rng, (B, 16, Hkv, D))
        post0 = ref_verify(hv, w_lm, np.zeros((B, 16), np.int32), L, out_cap=cap + 16)
        blk = make_block_ids(rng, post0["posterior"], draw_accept_lengths(rng, ("uniform",), B), V)
        # ---- oracle cycle ----
        rv = ref_verify(hv, w_lm, blk, L, out_tokens=ref_out)
        ref_out = rv["out_tokens"]
        pos = np.repeat(L, 16) + np.tile(np.arange(16), B)
        rp = ref_project(layers, w_fc, gh, wk, wv, gk, pos, Hkv, D, theta, eps)
        for b in range(B):
            ref_k[b] = np.concatenate([ref_k[b][:L[b]], rp["k"][16 * b:16 * b + 16]])
            ref_v[b] = np.concatenate([ref_v[b][:L[b]], rp["v"][16 * b:16 * b + 16]])
        newL, bad = kv_crop_lengths(L + 16, rv["commit_len"])
        assert not bad.any()
        ro = ref_attention(q, kb, vb, ref_k, ref_v, newL, theta, 1 / math.sqrt(D))
        # ---- GPU cycle ----
        target.seq_len.copy_(commit + 16)        # the target's verify forward appended 16 rows
        st = CycleState(
            layer_hidden=[dev_bf16(x) for x in layers], verify_hidden=dev_bf16(hv.reshape(B * 16, H)),
            block_ids=dev_i32(blk), len_before=commit, write_pos=draft.seq_len,
            q_blk=dev_bf16(q), k_blk=dev_bf16(kb), v_blk=dev_bf16(vb), draft_cache=draft,
            target_view=target, posterior=torch.zeros((B, 16), dtype=torch.int32, device="cuda"),
            accept_len=torch.zeros(B, dtype=torch.int32, device="cuda"),
            next_staged=torch.zeros(B, dtype=torch.int32, device="cuda"), commit_len=commit,
            out_tokens=out_tokens,
            attn_out=torch.zeros((B, 16, Hq, D), dtype=torch.bfloat16, device="cuda"))
        run_cycle(dims, w, st, ws, concurrent=concurrent)
        torch.cuda.synchronize()
        assert dfl.dflash_read_status(ws) == 0
        got = {"posterior": st.posterior.cpu().numpy(), "accept": st.accept_len.cpu().numpy(),
               "next_staged": st.next_staged.cpu().numpy(),
               "commit_len": commit.cpu().numpy(), "out_tokens": out_tokens.cpu().numpy()}
        info = check_verify(rv, got, L)
        assert info["excluded_seqs"] == 0
        assert np.array_equal(draft.seq_len.cpu().numpy(), newL)
        assert np.array_equal(target.seq_len.cpu().numpy(), newL)
        assert_close_bf16(host_f64(st.attn_out), ro)
        # the block's context rows as written on the GPU (first 1 + a of them survive)
        kk = host_f64(draft.k)
        for b in range(B):
            for t in range(int(newL[b] - L[b])):
                r = int(L[b]) + t
                if paged:
                    pg = draft.page_table.cpu().numpy()[b, r // 16]
                    row = kk[pg, :, r % 16]
                else:
                    row = kk[b, :, r]
                np.testing.assert_allclose(row, ref_k[b][r], atol=2e-2)
        L = newL
        ref_k = [ref_k[b][:L[b]] for b in range(B)]
        ref_v = [ref_v[b][:L[b]] for b in range(B)]
    if paged:
        fc = int(draft.free_count.item())
        table = draft.page_table.cpu().numpy()
        mapped = set(table[table >= 0].tolist())
        free = set(draft.free_list.cpu().numpy()[:fc].tolist())
        assert mapped.isdisjoint(free) and len(mapped) + len(free) == lay.n_pages
        for b in range(B):
            assert (table[b] >= 0).sum() == -(-int(L[b]) // 16)


def test_cycle_graph_matches_direct_calls():
    """CycleGraph (copies in, the four calls, copies out, one CUDA graph) gives
    the same tokens, lengths and attention output as issuing the calls."""
    import block_diffusion_speculative_02_gb300 as dfl
    from block_diffusion_speculative_02_gb300.cycle import (CycleGraph, CycleState, CycleWeights,
                                                            run_cycle)

    rng = np.random.default_rng(7)
    B, H, Hq, Hkv, D, V, nL, cap = 2, 256, 4, 2, 64, 4096, 2, 200
    L0 = np.array([90, 41], np.int32)
    dims = dfl.make_dims(B, H, Hq, Hkv, D, V, nL, cap)
    w = CycleWeights(*(dev_bf16(x) for x in (
        normal_bf16(rng, (V, H), 0.02), normal_bf16(rng, (H, nL * H), 0.02),
        normal_bf16(rng, (H,), 0.02, 1.0), normal_bf16(rng, (Hkv * D, H), 0.02),
        normal_bf16(rng, (Hkv * D, H), 0.02), normal_bf16(rng, (D,), 0.02, 1.0))))
    ck = pack_contiguous_heads([normal_bf16(rng, (int(L), Hkv, D)) for L in L0], cap, Hkv, D)
    cv = pack_contiguous_heads([normal_bf16(rng, (int(L), Hkv, D)) for L in L0], cap, Hkv, D)
    host = {"verify_hidden": unit_rms_rows_bf16(rng, (B * 16, H)),
            "layers": [unit_rms_rows_bf16(rng, (B * 16, H)) for _ in range(nL)],
            "block_ids": rng.integers(0, V, size=(B, 16)).astype(np.int32),
            "q": normal_bf16(rng, (B, 16, Hq, D)), "k": normal_bf16(rng, (B, 16, Hkv, D)),
            "v": normal_bf16(rng, (B, 16, Hkv, D))}

    def state():
        draft = dfl.KVView(dev_bf16(ck), dev_bf16(cv), dev_i32(L0), capacity=cap)
        commit = dev_i32(L0)
        return CycleState(
            layer_hidden=[torch.zeros((B * 16, H), dtype=torch.bfloat16, device="cuda")
                          for _ in range(nL)],
            verify_hidden=torch.zeros((B * 16, H), dtype=torch.bfloat16, device="cuda"),
            block_ids=torch.zeros((B, 16), dtype=torch.int32, device="cuda"),
            len_before=commit, write_pos=draft.seq_len,
            q_blk=torch.zeros((B, 16, Hq, D), dtype=torch.bfloat16, device="cuda"),
            k_blk=torch.zeros((B, 16, Hkv, D), dtype=torch.bfloat16, device="cuda"),
            v_blk=torch.zeros((B, 16, Hkv, D), dtype=torch.bfloat16, device="cuda"),
            draft_cache=draft, target_view=dfl.KVView(None, None, dev_i32(L0 + 16), capacity=cap),
            posterior=torch.zeros((B, 16), dtype=torch.int32, device="cuda"),
            accept_len=torch.zeros(B, dtype=torch.int32, device="cuda"),
            next_staged=torch.zeros(B, dtype=torch.int32, device="cuda"), commit_len=commit,
            out_tokens=torch.full((B, cap + 16), -1, dtype=torch.int32, device="cuda"),
            attn_out=torch.zeros((B, 16, Hq, D), dtype=torch.bfloat16, device="cuda"))

    def inputs_of(st):
        dev = [st.verify_hidden, *st.layer_hidden, st.block_ids, st.q_blk, st.k_blk, st.v_blk]
        src = [host["verify_hidden"], *host["layers"], host["block_ids"], host["q"], host["k"],
               host["v"]]
        pairs = []
        for d, h in zip(dev, src):
            t = torch.from_numpy(np.ascontiguousarray(h).view(np.int16) if h.dtype == np.uint16
                                 else np.ascontiguousarray(h))
            pairs.append((t.view(d.dtype).pin_memory(), d))
        return pairs

    a = state()
    for h, d in inputs_of(a):
        d.copy_(h)
    run_cycle(dims, w, a, dfl.alloc_workspace(dims))
    b = state()
    outs = [b.accept_len, b.posterior, b.commit_len]
    host_out = [torch.empty_like(t, device="cpu").pin_memory() for t in outs]
    # the graph's warm-up run moves the state once: capture on a throw-away copy
    # of the lengths, then restore them and replay the captured cycle
    saved = [b.draft_cache.seq_len.clone(), b.commit_len.clone(), b.target_view.seq_len.clone()]
    g = CycleGraph(dims, w, b, dfl.alloc_workspace(dims), inputs_of(b), list(zip(outs, host_out)))
    for t, s in zip([b.draft_cache.seq_len, b.commit_len, b.target_view.seq_len], saved):
        t.copy_(s)
    b.out_tokens.fill_(-1)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(host_out[0].numpy(), a.accept_len.cpu().numpy())
    assert np.array_equal(host_out[1].numpy(), a.posterior.cpu().numpy())
    assert np.array_equal(host_out[2].numpy(), a.commit_len.cpu().numpy())
    assert np.array_equal(b.out_tokens.cpu().numpy(), a.out_tokens.cpu().numpy())
    assert np.array_equal(b.draft_cache.seq_len.cpu().numpy(), a.draft_cache.seq_len.cpu().numpy())
    # the projection adds its CTAs' partial sums in a fixed order and the
    # attention merges its splits in a fixed order: same inputs, same bits
    for x, y in ((b.attn_out, a.attn_out), (b.draft_cache.k, a.draft_cache.k),
                 (b.draft_cache.v, a.draft_cache.v)):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_pipelined_cycles_match_direct_calls():
    """PipelinedCycles (inputs of step k + 1 copied in while step k runs, two
    graphs over two input sets, shared state) gives, after three steps with
    different inputs, the tokens, lengths, results and attention output of
    issuing the calls step by step."""
    import dataclasses

    import block_diffusion_speculative_02_gb300 as dfl
    from block_diffusion_speculative_02_gb300.cycle import (CycleState, CycleWeights,
                                                            PipelinedCycles, packed_tensors,
                                                            run_cycle)

    rng = np.random.default_rng(17)
    B, H, Hq, Hkv, D, V, nL, cap = 2, 256, 4, 2, 64, 4096, 2, 260
    L0 = np.array([70, 33], np.int32)
    dims = dfl.make_dims(B, H, Hq, Hkv, D, V, nL, cap)
    w = CycleWeights(*(dev_bf16(x) for x in (
        normal_bf16(rng, (V, H), 0.02), normal_bf16(rng, (H, nL * H), 0.02),
        normal_bf16(rng, (H,), 0.02, 1.0), normal_bf16(rng, (Hkv * D, H), 0.02),
        normal_bf16(rng, (Hkv * D, H), 0.02), normal_bf16(rng, (D,), 0.02, 1.0))))
    ck = pack_contiguous_heads([normal_bf16(rng, (int(L), Hkv, D)) for L in L0], cap, Hkv, D)
    cv = pack_contiguous_heads([normal_bf16(rng, (int(L), Hkv, D)) for L in L0], cap, Hkv, D)
    specs = [((B * 16, H), torch.bfloat16)] * (1 + nL) + [((B, 16), torch.int32)] + \
        [((B, 16, Hq, D), torch.bfloat16), ((B, 16, Hkv, D), torch.bfloat16),
         ((B, 16, Hkv, D), torch.bfloat16)]
    steps = []
    for _ in range(3):
        flat, views = packed_tensors(specs, "cpu", pin=True)
        vals = [unit_rms_rows_bf16(rng, (B * 16, H)) for _ in range(1 + nL)] + \
            [rng.integers(0, V, size=(B, 16)).astype(np.int32), normal_bf16(rng, (B, 16, Hq, D)),
             normal_bf16(rng, (B, 16, Hkv, D)), normal_bf16(rng, (B, 16, Hkv, D))]
        for v_, x in zip(views, vals):
            v_.copy_(torch.from_numpy(x.view(np.int16) if x.dtype == np.uint16 else x)
                     .view(v_.dtype))
        steps.append(flat)

    def state(ins):
        draft = dfl.KVView(dev_bf16(ck), dev_bf16(cv), dev_i32(L0), capacity=cap)
        commit = dev_i32(L0)
        return CycleState(
            layer_hidden=list(ins[1:1 + nL]), verify_hidden=ins[0], block_ids=ins[1 + nL],
            len_before=commit, write_pos=draft.seq_len, q_blk=ins[2 + nL], k_blk=ins[3 + nL],
            v_blk=ins[4 + nL], draft_cache=draft,
            target_view=dfl.KVView(None, None, dev_i32(L0 + 16), capacity=cap + 64),
            posterior=torch.zeros((B, 16), dtype=torch.int32, device="cuda"),
            accept_len=torch.zeros(B, dtype=torch.int32, device="cuda"),
            next_staged=torch.zeros(B, dtype=torch.int32, device="cuda"), commit_len=commit,
            out_tokens=torch.full((B, cap + 64), -1, dtype=torch.int32, device="cuda"),
            attn_out=torch.zeros((B, 16, Hq, D), dtype=torch.bfloat16, device="cuda"))

    # step by step
    dev_a, ins_a = packed_tensors(specs, "cuda")
    a = state(ins_a)
    ws_a = dfl.alloc_workspace(dims)
    for flat in steps:
        dev_a.copy_(flat)
        run_cycle(dims, w, a, ws_a)
    torch.cuda.synchronize()

    # pipelined: two input slots, shared state
    dev0, ins0 = packed_tensors(specs, "cuda")
    dev1, ins1 = packed_tensors(specs, "cuda")
    dev0.copy_(steps[0])
    dev1.copy_(steps[0])
    b0 = state(ins0)
    b1 = dataclasses.replace(b0, layer_hidden=list(ins1[1:1 + nL]), verify_hidden=ins1[0],
                             block_ids=ins1[1 + nL], q_blk=ins1[2 + nL], k_blk=ins1[3 + nL],
                             v_blk=ins1[4 + nL])
    outs = [b0.accept_len, b0.posterior, b0.commit_len]
    host_out = [[torch.empty_like(t, device="cpu").pin_memory() for _ in range(2)] for t in outs]
    lens = [b0.draft_cache.seq_len, b0.commit_len, b0.target_view.seq_len]
    saved = [t.clone() for t in lens]
    pc = PipelinedCycles(dims, w, [b0, b1], dfl.alloc_workspace(dims), [dev0, dev1],
                         list(zip(outs, host_out)))
    for t, s in zip(lens, saved):          # undo the two warm-up cycles
        t.copy_(s)
    b0.out_tokens.fill_(-1)
    torch.cuda.synchronize()
    for flat in steps:
        pc.step(flat)
    s = pc.finish()
    assert np.array_equal(host_out[0][s].numpy(), a.accept_len.cpu().numpy())
    assert np.array_equal(host_out[1][s].numpy(), a.posterior.cpu().numpy())
    assert np.array_equal(host_out[2][s].numpy(), a.commit_len.cpu().numpy())
    assert np.array_equal(b0.out_tokens.cpu().numpy(), a.out_tokens.cpu().numpy())
    assert np.array_equal(b0.draft_cache.seq_len.cpu().numpy(),
                          a.draft_cache.seq_len.cpu().numpy())
    for x, y in ((b0.attn_out, a.attn_out), (b0.draft_cache.k, a.draft_cache.k),
                 (b0.draft_cache.v, a.draft_cache.v)):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
