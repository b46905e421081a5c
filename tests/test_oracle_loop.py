"""Pins of the whole cycle on a tiny random-weight target + drafter (CPU only).

* Lossless ("dflash-mlx" (dpshk.com) 什么是"无损"推测解码, 保证一–三): the
  draft/verify loop emits exactly the target's plain greedy decode.
* Crop invariant (保证三; "DFlash双实现对比" (hotelren.com) §3): after every
  cycle the cropped target cache equals a fresh prefill of the committed
  tokens, and the drafter's context equals the projection of that prefill.
* Paged crop: released pages are exactly those past the new length.
"""
import numpy as np
import pytest

from oracle.dflash_oracle import kv_crop_lengths, kv_crop_paged, pages_needed
from oracle.tiny_models import TinyDrafter, TinyTarget, greedy_decode, spec_loop


class PeekingDrafter(TinyDrafter):
    """A drafter that proposes the target's true greedy continuation with a
    planted first mistake at a random depth, so every acceptance length occurs."""

    def __init__(self, target, truth, prompt_len, seed=5):
        super().__init__(target, seed=seed)
        self.truth = truth
        self.prompt_len = prompt_len
        self.rng = np.random.default_rng(seed)

    def draft(self, staged):
        done = self.ctx_len - self.prompt_len            # committed tokens so far
        want = self.truth[done + 1:done + 16]
        want = list(want) + [0] * (15 - len(want))
        k = int(self.rng.integers(0, 16))                 # first wrong draft position
        out = np.array(want, dtype=np.int32)
        if k < 15:
            out[k] = (out[k] + 1 + int(self.rng.integers(0, self.d.vocab - 2))) % self.d.vocab
        return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_spec_loop_equals_greedy_decode(seed):
    t = TinyTarget(seed)
    prompt = list(np.random.default_rng(100 + seed).integers(0, 90, size=6))
    n = 48
    greedy = greedy_decode(t, prompt, n)
    real = spec_loop(t, TinyDrafter(t, seed + 10), prompt, n)
    assert real["tokens"] == greedy
    truth = greedy_decode(t, prompt, n + 40)
    peek = spec_loop(t, PeekingDrafter(t, truth, len(prompt), seed), prompt, n)
    assert peek["tokens"] == greedy
    assert max(peek["accepts"]) >= 5              # long acceptances exercised


@pytest.mark.parametrize("seed", [4, 5])
def test_spec_loop_equals_greedy_decode_with_bf16_boundaries(seed):
    """The same property for a target whose embedding, LM head and LM-head
    input are bf16 values (and a drafter with bf16 weights): the form a GPU
    loop consumes."""
    t = TinyTarget(seed, bf16_head=True)
    assert np.array_equal(t.lm_head.astype(np.float32).astype(np.float64), t.lm_head)
    prompt = list(np.random.default_rng(200 + seed).integers(0, 90, size=9))
    n = 40
    greedy = greedy_decode(t, prompt, n)
    assert spec_loop(t, TinyDrafter(t, seed + 20, bf16_weights=True), prompt, n)["tokens"] == greedy
    truth = greedy_decode(t, prompt, n + 40)
    assert spec_loop(t, PeekingDrafter(t, truth, len(prompt), seed), prompt, n)["tokens"] == greedy


def test_crop_invariant_after_every_cycle():
    t = TinyTarget(3)
    prompt = [4, 8, 15, 16, 23, 42]
    truth = greedy_decode(t, prompt, 120)
    checked = []

    def check(state):
        cache, dr = state["cache"], state["drafter"]
        toks = state["prompt"] + state["committed"]
        assert cache.length == len(toks) == dr.ctx_len
        fresh = t.new_cache()
        _, outs = t.forward(toks, fresh)
        L = cache.length
        np.testing.assert_array_equal(cache.k[:, :L], fresh.k[:, :L])
        np.testing.assert_array_equal(cache.v[:, :L], fresh.v[:, :L])
        ref = TinyDrafter(t, seed=5)
        ref.write_ctx(outs, 0)
        np.testing.assert_allclose(dr.ctx_k[:L], ref.ctx_k[:L], rtol=0, atol=1e-12)
        np.testing.assert_allclose(dr.ctx_v[:L], ref.ctx_v[:L], rtol=0, atol=1e-12)
        checked.append(state["accept"])

    spec_loop(t, PeekingDrafter(t, truth, len(prompt), seed=5), prompt, 60, on_cycle=check)
    assert len(checked) >= 4 and len(set(checked)) >= 3


def test_crop_lengths():
    lens, bad = kv_crop_lengths([10, 10, 0, 5], [3, 10, 0, 6])
    assert list(lens) == [3, 10, 0, 5] and list(bad) == [False, False, False, True]
    lens, bad = kv_crop_lengths([4], [-1])
    assert list(lens) == [4] and bad[0]


def test_paged_crop_releases_whole_pages_past_the_length():
    P = 16
    table = np.array([[7, 3, 9, 1, -1], [2, 5, -1, -1, -1]], dtype=np.int32)
    free = {0, 4, 6, 8}
    # seq 0: 64 -> 17 keeps pages 0,1 (page 1 holds token 16); seq 1: 32 -> 32 keeps both
    r = kv_crop_paged([64, 32], table, free, [17, 32], P)
    assert list(r["seq_len"]) == [17, 32]
    assert list(r["page_table"][0]) == [7, 3, -1, -1, -1]
    assert list(r["page_table"][1]) == [2, 5, -1, -1, -1]
    assert r["free"] == free | {9, 1}
    # page-aligned new length releases the page that starts there
    r = kv_crop_paged([64], table[:1], free, [32], P)
    assert list(r["page_table"][0]) == [7, 3, -1, -1, -1]
    r = kv_crop_paged([64], table[:1], free, [0], P)
    assert list(r["page_table"][0]) == [-1] * 5 and r["free"] == free | {7, 3, 9, 1}
    # an invalid grow leaves everything unchanged
    r = kv_crop_paged([20], table[:1], free, [40], P)
    assert r["bad"][0] and list(r["page_table"][0]) == list(table[0])
    # conservation: mapped + free is the same set before and after
    before = set(table[table >= 0].tolist()) | free
    r = kv_crop_paged([64, 32], table, free, [5, 0], P)
    after = set(r["page_table"][r["page_table"] >= 0].tolist()) | r["free"]
    assert before == after


def test_pages_needed_for_a_block():
    assert pages_needed([0, 15, 16, 33], 16, 16) == [[0], [0, 1], [1], [2, 3]]
