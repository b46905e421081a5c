"""The seeded input generators (CPU only): bf16 rounding, acceptance draws,
draft planting and the paged-cache layout."""
import numpy as np
import torch

from synthetic import (CONFIG_BY_NAME, CONFIGS, bf16_bits_to_f32, draw_accept_lengths, f32_to_bf16_bits,
                       geometric_ratio_for_mean, make_block_ids, make_paged_layout,
                       scatter_paged)


def test_bf16_rounding_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 3,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0,
                                  3.0e38, -1e-40], dtype=np.float32)])
    ours = f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(bf16_bits_to_f32(ours),
                                  torch.from_numpy(ours.view(np.int16)).view(torch.bfloat16)
                                  .float().numpy())


def test_truncated_geometric_ratio():
    for mean, q in ((13.0, 1.493549), (12.0, 1.311326)):
        got = geometric_ratio_for_mean(mean)
        assert abs(got - q) < 1e-5
        k = np.arange(16)
        w = got ** k
        assert abs((k * w).sum() / w.sum() - mean) < 1e-9
    rng = np.random.default_rng(1)
    a = draw_accept_lengths(rng, ("geometric", 13.0), 200000)
    assert abs(a.mean() - 13.0) < 0.02 and a.min() >= 0 and a.max() == 15
    u = draw_accept_lengths(rng, ("uniform",), 200000)
    assert abs(u.mean() - 7.5) < 0.03 and set(np.unique(u)) == set(range(16))


def test_make_block_ids_plants_exactly_a_matches():
    rng = np.random.default_rng(2)
    post = rng.integers(0, 50, size=(64, 16))
    acc = rng.integers(0, 16, size=64)
    blk = make_block_ids(rng, post, acc, 50)
    for b in range(64):
        a = acc[b]
        assert np.array_equal(blk[b, 1:1 + a], post[b, :a])
        if a < 15:
            assert blk[b, 1 + a] != post[b, a]
    assert blk.min() >= 0 and blk.max() < 50


def test_paged_layout_is_a_partition():
    rng = np.random.default_rng(3)
    lens = rng.integers(512, 16385, size=32)
    lay = make_paged_layout(rng, lens, reserve_tokens=32)
    mapped = lay.page_table[lay.page_table >= 0]
    free = lay.free_list[:lay.free_count]
    assert len(set(mapped.tolist())) == len(mapped)
    assert set(mapped.tolist()).isdisjoint(set(free.tolist()))
    assert len(mapped) + len(free) == lay.n_pages
    for b, L in enumerate(lens):
        assert (lay.page_table[b] >= 0).sum() == -(-L // 16)
    rows = [rng.integers(0, 60000, size=(int(L), 2)).astype(np.uint16) for L in lens[:3]]
    lay3 = make_paged_layout(rng, lens[:3], 16)
    pool = scatter_paged(lay3, rows, (2,))
    for b in range(3):
        for t in (0, 17, int(lens[b]) - 1):
            np.testing.assert_array_equal(pool[lay3.page_table[b, t // 16], t % 16], rows[b][t])


def test_config_shapes():
    names = [c.name for c in CONFIGS]
    assert names[2] == "qwen3_8b_b1"
    c = CONFIG_BY_NAME["qwen3_8b_b1"]
    assert (c.hidden, c.n_q_heads, c.n_kv_heads, c.head_dim, c.vocab, c.ctx_in) == \
        (4096, 32, 8, 128, 151936, 20480)
