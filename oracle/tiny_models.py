"""Tiny random-weight target + drafter and the full speculative loop, float64.

TEST INFRASTRUCTURE ONLY (see dflash_oracle.py).  Used to pin the oracle's
hot-path steps as a whole: the draft/verify loop must emit exactly the
target's plain greedy decode (the lossless property of "dflash-mlx"
(dpshk.com), 什么是"无损"推测解码 and 保证一–三), and after every cycle the
cropped caches must equal a fresh prefill of the committed tokens (保证三).

The target is Qwen3-like (pre-norm decoder layers with per-head q/k RMSNorm,
rotate-half RoPE, GQA causal attention, SwiGLU MLP).  The drafter is one such
layer whose attention is the dual-source block attention of the oracle
(Q from the block; K/V = context projected from selected target layers ⊕
block), as "DFlash双实现对比" (hotelren.com) §2 and §4 describe.

All per-token arithmetic of the target is done one row at a time, so a token
processed inside a 16-token verify block and the same token processed alone
by greedy decoding go through identical floating-point operations.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .dflash_oracle import (BLOCK, acceptance_length, apply_rope, bf16_to_f64, block_attention,
                            ctx_project, draft_out_mlp, draft_qkv, draft_tokens,
                            kv_crop_lengths, rms_norm, round_bf16, verify_accept)


def _rows(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Row-by-row x @ w.T with a fixed per-row operation (one gemv per row)."""
    return np.stack([w @ np.ascontiguousarray(r) for r in x]) if len(x) else \
        np.zeros((0, w.shape[0]))


def _silu(x):
    return x / (1.0 + np.exp(-x))


def _bf16_values(x):
    """x rounded to the nearest bf16 values (float64 holding them exactly)."""
    return bf16_to_f64(round_bf16(x))


@dataclass
class TinyDims:
    vocab: int = 96
    hidden: int = 32
    n_q_heads: int = 4
    n_kv_heads: int = 2
    head_dim: int = 8
    ffn: int = 64
    n_layers: int = 3
    target_layer_ids: tuple = (1, 2)      # indices into the per-layer outputs
    rope_theta: float = 1.0e4
    rms_eps: float = 1.0e-6
    capacity: int = 512


class _Layer:
    def __init__(self, rng, d: TinyDims):
        H, Hq, Hkv, D, F = d.hidden, d.n_q_heads, d.n_kv_heads, d.head_dim, d.ffn
        s = 1.0 / np.sqrt(H)
        self.ln1 = 1.0 + 0.1 * rng.standard_normal(H)
        self.wq = s * rng.standard_normal((Hq * D, H))
        self.wk = s * rng.standard_normal((Hkv * D, H))
        self.wv = s * rng.standard_normal((Hkv * D, H))
        self.q_norm = 1.0 + 0.1 * rng.standard_normal(D)
        self.k_norm = 1.0 + 0.1 * rng.standard_normal(D)
        self.wo = (1.0 / np.sqrt(Hq * D)) * rng.standard_normal((H, Hq * D))
        self.ln2 = 1.0 + 0.1 * rng.standard_normal(H)
        self.w_gate = s * rng.standard_normal((F, H))
        self.w_up = s * rng.standard_normal((F, H))
        self.w_down = (1.0 / np.sqrt(F)) * rng.standard_normal((H, F))

    def mlp(self, x, eps):
        hn = rms_norm(x, self.ln2, eps)
        return x + _rows(_silu(_rows(hn, self.w_gate)) * _rows(hn, self.w_up), self.w_down)


class KVCache:
    """Per-layer contiguous K/V rows plus a length (the target's cache)."""

    def __init__(self, n_layers, capacity, n_kv_heads, head_dim):
        self.k = np.zeros((n_layers, capacity, n_kv_heads, head_dim))
        self.v = np.zeros((n_layers, capacity, n_kv_heads, head_dim))
        self.length = 0

    def crop(self, new_len: int):
        lens, bad = kv_crop_lengths([self.length], [new_len])
        assert not bad[0]
        self.length = int(lens[0])


class TinyTarget:
    """With ``bf16_head`` the target is a bf16 model at its boundaries: the
    embedding table and the LM head hold bf16 values, and the final hidden
    state reaches the LM head rounded to bf16 (as a bf16 model hands it over);
    the body still computes in float64.  Greedy decoding and the speculative
    loop both take logits through :meth:`logits` / :meth:`head_input`, so the
    loop stays exactly lossless."""

    def __init__(self, seed: int = 0, dims: TinyDims = TinyDims(), bf16_head: bool = False):
        rng = np.random.default_rng(seed)
        self.d = dims
        self.bf16_head = bf16_head
        self.embed = rng.standard_normal((dims.vocab, dims.hidden))
        self.layers = [_Layer(rng, dims) for _ in range(dims.n_layers)]
        self.final_norm = 1.0 + 0.1 * rng.standard_normal(dims.hidden)
        self.lm_head = (1.0 / np.sqrt(dims.hidden)) * rng.standard_normal((dims.vocab,
                                                                           dims.hidden))
        if bf16_head:
            self.embed = _bf16_values(self.embed)
            self.lm_head = _bf16_values(self.lm_head)

    def new_cache(self) -> KVCache:
        d = self.d
        return KVCache(d.n_layers, d.capacity, d.n_kv_heads, d.head_dim)

    def forward(self, tokens, cache: KVCache):
        """Process ``tokens`` at positions cache.length.. (causal), appending K/V.

        Returns (final-normed hidden [n,H], per-layer outputs list [n,H])."""
        d = self.d
        n = len(tokens)
        start = cache.length
        G = d.n_q_heads // d.n_kv_heads
        x = self.embed[np.asarray(tokens)]
        outs = []
        pos = start + np.arange(n)
        for li, lay in enumerate(self.layers):
            hn = rms_norm(x, lay.ln1, d.rms_eps)
            q = rms_norm(_rows(hn, lay.wq).reshape(n, d.n_q_heads, d.head_dim), lay.q_norm,
                         d.rms_eps)
            k = rms_norm(_rows(hn, lay.wk).reshape(n, d.n_kv_heads, d.head_dim), lay.k_norm,
                         d.rms_eps)
            v = _rows(hn, lay.wv).reshape(n, d.n_kv_heads, d.head_dim)
            q = apply_rope(q, np.broadcast_to(pos[:, None], q.shape[:2]), d.rope_theta)
            k = apply_rope(k, np.broadcast_to(pos[:, None], k.shape[:2]), d.rope_theta)
            cache.k[li, start:start + n] = k
            cache.v[li, start:start + n] = v
            att = np.zeros((n, d.n_q_heads, d.head_dim))
            scale = 1.0 / np.sqrt(d.head_dim)
            for i in range(n):
                p_i = start + i
                for h in range(d.n_q_heads):
                    g = h // G
                    kk = cache.k[li, :p_i + 1, g]
                    vv = cache.v[li, :p_i + 1, g]
                    s = (kk @ q[i, h]) * scale
                    s = s - s.max()
                    w = np.exp(s)
                    w = w / w.sum()
                    att[i, h] = w @ vv
            x = x + _rows(att.reshape(n, -1), lay.wo)
            x = lay.mlp(x, d.rms_eps)
            outs.append(x.copy())
        cache.length = start + n
        return rms_norm(x, self.final_norm, d.rms_eps), outs

    def head_input(self, final_hidden):
        """The final hidden rows as the LM head receives them."""
        return _bf16_values(final_hidden) if self.bf16_head else final_hidden

    def logits(self, final_hidden):
        return _rows(self.head_input(final_hidden), self.lm_head)


class TinyDrafter:
    """One-layer block-diffusion drafter sharing the target's embedding and LM head."""

    def __init__(self, target: TinyTarget, seed: int = 1, bf16_weights: bool = False):
        d = target.d
        rng = np.random.default_rng(seed)
        self.t = target
        self.d = d
        nL = len(d.target_layer_ids)
        self.w_fc = (1.0 / np.sqrt(nL * d.hidden)) * rng.standard_normal((d.hidden,
                                                                         nL * d.hidden))
        self.hidden_norm = 1.0 + 0.1 * rng.standard_normal(d.hidden)
        self.layer = _Layer(rng, d)
        self.final_norm = 1.0 + 0.1 * rng.standard_normal(d.hidden)
        if bf16_weights:         # every weight a bf16 value (a bf16 drafter's weights)
            self.w_fc = _bf16_values(self.w_fc)
            self.hidden_norm = _bf16_values(self.hidden_norm)
            self.final_norm = _bf16_values(self.final_norm)
            for name, w in vars(self.layer).items():
                setattr(self.layer, name, _bf16_values(w))
        self.mask_id = d.vocab - 1
        self.ctx_k = np.zeros((d.capacity, d.n_kv_heads, d.head_dim))
        self.ctx_v = np.zeros((d.capacity, d.n_kv_heads, d.head_dim))
        self.ctx_len = 0

    def write_ctx(self, layer_outs, pos0: int):
        """Project the selected target layers' rows into context K/V at pos0.."""
        d = self.d
        sel = [layer_outs[i] for i in d.target_layer_ids]
        n = sel[0].shape[0]
        r = ctx_project(sel, self.w_fc, self.hidden_norm, self.layer.wk, self.layer.wv,
                        self.layer.k_norm, pos0 + np.arange(n), d.n_kv_heads, d.head_dim,
                        d.rope_theta, d.rms_eps)
        self.ctx_k[pos0:pos0 + n] = r["k"]
        self.ctx_v[pos0:pos0 + n] = r["v"]
        self.ctx_len = pos0 + n

    def crop(self, new_len: int):
        lens, bad = kv_crop_lengths([self.ctx_len], [new_len])
        assert not bad[0]
        self.ctx_len = int(lens[0])

    def draft(self, staged: int) -> np.ndarray:
        """One parallel forward over [staged, mask x 15]; every mask position
        predicts its own token ("dflash-mlx" 块扩散草稿 steps 1–2)."""
        d = self.d
        lay = self.layer
        T = BLOCK
        blk = np.full(T, self.mask_id)
        blk[0] = staged
        x = self.t.embed[blk]
        r = draft_qkv(x, lay.ln1, lay.wq, lay.wk, lay.wv, lay.q_norm, lay.k_norm, d.n_q_heads,
                      d.n_kv_heads, d.head_dim, d.rms_eps)
        o = block_attention(r["q"][None], r["k"][None], r["v"][None], [self.ctx_k],
                            [self.ctx_v], [self.ctx_len], d.rope_theta,
                            1.0 / np.sqrt(d.head_dim))[0]
        x2 = draft_out_mlp(x, o, lay.wo, lay.ln2, lay.w_gate, lay.w_up, lay.w_down,
                           d.rms_eps)["x2"]
        return draft_tokens(x2, self.final_norm, self.t.lm_head, d.rms_eps)["tokens"][0]


def greedy_decode(target: TinyTarget, prompt, n_new: int) -> list:
    """Plain autoregressive greedy decoding, one token per target forward."""
    cache = target.new_cache()
    h, _ = target.forward(prompt, cache)
    tok = int(np.argmax(target.logits(h[-1:])[0]))
    out = [tok]
    while len(out) < n_new:
        h, _ = target.forward([tok], cache)
        tok = int(np.argmax(target.logits(h)[0]))
        out.append(tok)
    return out


def spec_loop(target: TinyTarget, drafter, prompt, n_new: int, on_cycle=None) -> dict:
    """The draft/verify cycle of "dflash-mlx" 单次前向验证 ①–⑨, greedy.

    ``drafter`` has ``draft(staged) -> 15 ids``, ``write_ctx(layer_outs, pos0)``
    and ``crop(new_len)``; ``on_cycle(state)`` is called after every cycle.
    """
    cache = target.new_cache()
    h, outs = target.forward(prompt, cache)                      # ① prefill
    staged = int(np.argmax(target.logits(h[-1:])[0]))            # ② staged first token
    drafter.write_ctx(outs, 0)
    committed = []
    accepts = []
    while len(committed) < n_new:
        L = cache.length
        drafts = drafter.draft(staged)                           # ③④
        block = np.concatenate([[staged], drafts]).astype(np.int32)
        hv, outs = target.forward(block, cache)                  # ⑤ one target forward
        r = verify_accept(target.head_input(hv)[None], target.lm_head, block[None],
                          np.array([len(committed)]), out_cap=len(committed) + BLOCK)
        a = int(r["accept"][0])                                   # ⑥
        committed.extend(int(t) for t in r["out_tokens"][0, len(committed):
                                                          int(r["commit_len"][0])])  # ⑦
        staged = int(r["next_staged"][0])                        # ⑧
        drafter.write_ctx(outs, L)                               # ctx rows of the block
        cache.crop(L + 1 + a)                                    # ⑨ crop both caches
        drafter.crop(L + 1 + a)
        accepts.append(a)
        if on_cycle is not None:
            on_cycle({"cache": cache, "drafter": drafter, "committed": list(committed),
                      "staged": staged, "accept": a, "prompt": list(prompt)})
    return {"tokens": committed[:n_new], "accepts": accepts}


def assert_acceptance_consistent(block, posterior, a):
    """Helper used by tests: the accepted drafts equal the posterior prefix."""
    assert a == acceptance_length(block[1:], posterior[:BLOCK - 1])
