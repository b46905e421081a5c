"""The lossless property on the GPU ("dflash-mlx" (dpshk.com) 什么是"无损"推测
解码 and 保证一–三): a draft/verify loop whose hot-path steps all run in
libdflash.so emits exactly the target's plain greedy decode.

The tiny random-weight target (bf16 embedding, LM head and LM-head input,
float64 body) runs its layers on the CPU; everything else goes through the
C ABI on the GPU:
  ② the first staged token (dflash_prefill_staged) and the prompt's drafter
    context (dflash_ctx_prefill);
  ③④ the drafter forward: dflash_draft_qkv, dflash_block_attention over the
    drafter cache, dflash_draft_mlp, dflash_draft_tokens;
  ⑤–⑧ verification, acceptance and commit (dflash_verify_accept);
  the block's drafter context (dflash_ctx_project) and ⑨ the crop of the
    target and drafter caches (dflash_kv_crop), whose new target length is
    what the CPU target keeps.
Two drafters: the GPU drafter's own tokens, and a peeking drafter that
overwrites them with the greedy continuation up to a planted first mistake,
so that every acceptance length 0..15 occurs.  The emitted tokens must equal
greedy decoding; positions where greedy decoding's top-2 logit gap is within
1e-3 of the maximum are counted and printed (an fp32 argmax may only differ
from float64 there)."""
import math

import numpy as np
import pytest
import torch

from oracle.dflash_oracle import round_bf16
from oracle.tiny_models import TinyDims, TinyDrafter, TinyTarget, greedy_decode
from tests.gpu_helpers import dev_bf16

pytestmark = pytest.mark.gpu

# shapes the kernels take: H a multiple of 128, Hkv * D a multiple of 128, D 64
DIMS = TinyDims(vocab=2048, hidden=128, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=256,
                n_layers=3, target_layer_ids=(1, 2), rope_theta=1.0e4, capacity=256)


def _dev_w(x):
    return dev_bf16(round_bf16(x))


def gpu_spec_loop(dfl, target, drafter, prompts, n_new, plant=None):
    """The cycle of 单次前向验证 ①–⑨ for a batch of prompts of one length, the
    hot-path steps on the GPU.  ``plant(b, cycle, committed)`` returns the
    acceptance length to plant for sequence b, or None for the GPU drafts."""
    d = target.d
    B, P = len(prompts), len(prompts[0])
    H, Hq, Hkv, D, V, F = d.hidden, d.n_q_heads, d.n_kv_heads, d.head_dim, d.vocab, d.ffn
    nL = len(d.target_layer_ids)
    cap = d.capacity
    dims = dfl.make_dims(B, H, Hq, Hkv, D, V, nL, cap, d.rope_theta, d.rms_eps)
    ws = dfl.alloc_workspace(dims)
    dws = dfl.dflash.alloc_draft_workspace(dims, F)
    pws = dfl.alloc_prefill_workspace(dims, P)
    lay = drafter.layer
    w = {n: _dev_w(x) for n, x in dict(
        w_lm=target.lm_head, embed=target.embed, w_fc=drafter.w_fc, gh=drafter.hidden_norm,
        ln1=lay.ln1, wq=lay.wq, wk=lay.wk, wv=lay.wv, qn=lay.q_norm, kn=lay.k_norm, wo=lay.wo,
        ln2=lay.ln2, wg=lay.w_gate, wu=lay.w_up, wd=lay.w_down, fn=drafter.final_norm).items()}
    i32 = dict(dtype=torch.int32, device="cuda")
    draft = dfl.KVView(torch.zeros((B, Hkv, cap, D), dtype=torch.bfloat16, device="cuda"),
                       torch.zeros((B, Hkv, cap, D), dtype=torch.bfloat16, device="cuda"),
                       torch.zeros(B, **i32), capacity=cap)
    tview = dfl.KVView(None, None, torch.zeros(B, **i32), capacity=cap)
    out_tokens = torch.full((B, cap), -1, **i32)
    caches = [target.new_cache() for _ in range(B)]

    # ① the target's prefill (CPU body); the prompt's drafter context
    hs, outs = zip(*[target.forward(p, c) for p, c in zip(prompts, caches)])
    layers = [dev_bf16(round_bf16(np.concatenate([o[i] for o in outs])))
              for i in d.target_layer_ids]
    dfl.dflash_ctx_prefill(dims, P, layers, w["w_fc"], w["gh"], w["wk"], w["wv"], w["kn"],
                           torch.zeros(B, **i32), draft, pws)
    # ② the first staged token from the last prompt row
    staged = torch.zeros(B, **i32)
    last = dev_bf16(round_bf16(np.stack([h[-1] for h in hs])))
    dfl.dflash_prefill_staged(dims, last, w["w_lm"], staged, ws)
    tview.seq_len.fill_(P)

    embed_bits = round_bf16(target.embed)
    q = torch.empty((B, 16, Hq, D), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((B, 16, Hkv, D), dtype=torch.bfloat16, device="cuda")
    v = torch.empty((B, 16, Hkv, D), dtype=torch.bfloat16, device="cuda")
    attn = torch.empty((B, 16, Hq, D), dtype=torch.bfloat16, device="cuda")
    x2 = torch.empty((B * 16, H), dtype=torch.bfloat16, device="cuda")
    block_ids = torch.zeros((B, 16), **i32)
    post = torch.zeros((B, 16), **i32)
    accept = torch.zeros(B, **i32)
    nxt = torch.zeros(B, **i32)
    commit = torch.full((B,), P, **i32)
    accepts, planted = [], []
    cycle = 0
    while True:
        torch.cuda.synchronize()
        lens = commit.cpu().numpy()
        if (lens - P >= n_new).all():
            break
        st = staged.cpu().numpy()
        # ③④ the drafter's forward over [staged, mask x 15]
        blk = np.full((B, 16), V - 1, np.int64)
        blk[:, 0] = st
        x = dev_bf16(embed_bits[blk.reshape(-1)])
        dfl.dflash.dflash_draft_qkv(dims, x, w["ln1"], w["wq"], w["wk"], w["wv"], w["qn"], w["kn"],
                                    q.view(B * 16, -1), k.view(B * 16, -1), v.view(B * 16, -1),
                                    dws)
        dfl.dflash_block_attention(dims, q, k, v, draft, 1 / math.sqrt(D), attn, ws)
        dfl.dflash.dflash_draft_mlp(dims, F, x, attn.view(B * 16, -1), w["wo"], w["ln2"], w["wg"],
                                    w["wu"], w["wd"], x2, dws)
        dfl.dflash.dflash_draft_tokens(dims, x2, w["fn"], w["w_lm"], staged, block_ids, None, dws)
        torch.cuda.synchronize()
        block = block_ids.cpu().numpy()
        assert np.array_equal(block[:, 0], st)
        want = np.full(B, -1)
        if plant is not None:
            for b in range(B):
                a = plant(b, cycle, int(lens[b] - P))
                if a is not None:
                    block[b, 1:] = plant.drafts(b, int(lens[b] - P), a, block[b, 1:])
                    want[b] = a
            block_ids.copy_(torch.from_numpy(block))
        # ⑤ one target forward over each block (CPU body)
        hv, layer_rows = [], [[] for _ in d.target_layer_ids]
        for b in range(B):
            h, o = target.forward(block[b], caches[b])
            hv.append(h)
            for j, i in enumerate(d.target_layer_ids):
                layer_rows[j].append(o[i])
        tview.seq_len.copy_(commit + 16)
        # ⑤–⑧ verification; the block's drafter context; ⑨ the crop of both caches
        dfl.dflash_verify_accept(dims, dev_bf16(round_bf16(np.concatenate(hv))), w["w_lm"],
                                 block_ids, commit, post, accept, nxt, commit, out_tokens, ws)
        dfl.dflash_ctx_project(dims, [dev_bf16(round_bf16(np.concatenate(r))) for r in layer_rows],
                               w["w_fc"], w["gh"], w["wk"], w["wv"], w["kn"], draft.seq_len, draft,
                               ws)
        dfl.dflash_kv_crop([tview, draft], commit, B, ws)
        staged.copy_(nxt)
        torch.cuda.synchronize()
        assert dfl.dflash_read_status(ws) == 0 and dfl.dflash_read_status(dws) == 0
        a_got = accept.cpu().numpy()
        new_len = tview.seq_len.cpu().numpy()
        assert np.array_equal(new_len, draft.seq_len.cpu().numpy())
        assert np.array_equal(new_len, lens + 1 + a_got)
        for b in range(B):
            caches[b].crop(int(new_len[b]))       # the target keeps the GPU-cropped length
            if want[b] >= 0:
                assert a_got[b] == want[b], (b, cycle, a_got[b], want[b])
        accepts.extend(a_got.tolist())
        planted.extend(int(x) for x in want if x >= 0)
        cycle += 1
        assert cycle < 4 * n_new
    toks = out_tokens.cpu().numpy()
    return [toks[b, P:P + n_new].tolist() for b in range(B)], accepts


def near_ties_of_greedy(target, prompt, tokens, rel=1e-3):
    """Positions of the greedy decode whose top-2 logit gap <= rel * |max|."""
    cache = target.new_cache()
    h, _ = target.forward(list(prompt) + list(tokens[:-1]), cache)
    lg = target.logits(h[len(prompt) - 1:])
    top = np.sort(lg, axis=1)
    gap = top[:, -1] - top[:, -2]
    return np.nonzero(gap <= rel * np.abs(top[:, -1]))[0].tolist()


class Planter:
    """Acceptance lengths on a schedule that covers 0..15 across sequences and
    seeds; the drafts are the greedy continuation with the first mistake at
    depth a."""

    def __init__(self, truths, seed, vocab):
        self.truths = truths
        self.seed = seed
        self.vocab = vocab
        self.rng = np.random.default_rng(seed)

    def __call__(self, b, cycle, done):
        return (5 * cycle + 7 * b + 3 * self.seed) % 16

    def drafts(self, b, done, a, current):
        truth = self.truths[b]
        out = np.array(truth[done + 1:done + 16], dtype=np.int64)
        if a < 15:
            out[a] = (out[a] + 1 + int(self.rng.integers(0, self.vocab - 3))) % (self.vocab - 1)
            out[a + 1:] = self.rng.integers(0, self.vocab - 1, size=15 - a - 1)
        return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gpu_loop_emits_the_greedy_decode(seed):
    import block_diffusion_speculative_02_gb300 as dfl
    target = TinyTarget(seed, DIMS, bf16_head=True)
    drafter = TinyDrafter(target, seed + 10, bf16_weights=True)
    rng = np.random.default_rng(300 + seed)
    n_new, P = 48, 24
    prompts = [rng.integers(0, DIMS.vocab - 1, size=P).tolist() for _ in range(2)]
    greedy = [greedy_decode(target, p, n_new) for p in prompts]
    ties = [near_ties_of_greedy(target, p, g) for p, g in zip(prompts, greedy)]
    print(f"seed {seed}: near-tie positions of the greedy decode {ties}")

    got, accepts = gpu_spec_loop(dfl, target, drafter, prompts, n_new)
    for b in range(2):
        assert got[b] == greedy[b], (b, ties[b], next(i for i, (x, y) in
                                                      enumerate(zip(got[b], greedy[b])) if x != y))
    print(f"seed {seed}: GPU drafter, acceptance lengths {sorted(set(accepts))}")

    truths = [greedy_decode(target, p, n_new + 40) for p in prompts]
    planter = Planter(truths, seed, DIMS.vocab)
    got, accepts = gpu_spec_loop(dfl, target, drafter, prompts, n_new, plant=planter)
    for b in range(2):
        assert got[b] == greedy[b], b
    print(f"seed {seed}: planted drafts, acceptance lengths {sorted(set(accepts))}")


def test_gpu_loop_every_acceptance_length():
    """Across three seeds and two sequences each, the planted schedule makes
    every acceptance length 0..15 occur on the GPU path, each committing
    1 + a greedy tokens."""
    import block_diffusion_speculative_02_gb300 as dfl
    seen = set()
    for seed in range(3):
        target = TinyTarget(seed, DIMS, bf16_head=True)
        drafter = TinyDrafter(target, seed + 10, bf16_weights=True)
        rng = np.random.default_rng(400 + seed)
        prompts = [rng.integers(0, DIMS.vocab - 1, size=20).tolist() for _ in range(2)]
        n_new = 64
        greedy = [greedy_decode(target, p, n_new) for p in prompts]
        truths = [greedy_decode(target, p, n_new + 40) for p in prompts]
        got, accepts = gpu_spec_loop(dfl, target, drafter, prompts, n_new,
                                     plant=Planter(truths, seed, DIMS.vocab))
        assert got == greedy
        seen |= set(accepts)
    assert seen == set(range(16)), sorted(seen)
