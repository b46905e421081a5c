"""Seeded synthetic workloads for the DFlash per-cycle hot path.

This module only *generates* inputs: shapes, seeds, value distributions,
acceptance draws and paged-cache layouts.  It holds none of the method's
arithmetic (no projection, attention, argmax, acceptance or crop), so both
the float64 oracle (through the tests) and the CUDA path (through the tests
and the bench) can consume the very same bits without sharing any compute.

bf16 values are produced as raw uint16 bit patterns by round-to-nearest-even
done in integer arithmetic on float32 bits; the oracle reads those bits as
exact float64 values and the GPU receives the same bits as ``torch.bfloat16``.

Workload shapes follow the model families named on the DFlash pages: the
Qwen3 drafter reuses the Qwen3 building blocks (hotelren.com "DFlash双实现对比",
section 1), the block holds the staged token plus 15 mask tokens
(dpshk.com "dflash-mlx", 块扩散草稿 step 1), and the context features are the
concatenation of several target layers (hotelren.com, section 4).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

BLOCK = 16  # staged token + 15 mask positions


# --------------------------------------------------------------------------
# workload definitions
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class CycleConfig:
    """One synthetic draft+verify cycle workload."""

    name: str
    batch: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    vocab: int
    n_ctx_layers: int
    ctx_len: int                 # fixed context length (ignored when ctx_len_range is set)
    ctx_len_range: Optional[tuple] = None   # (lo, hi) inclusive, uniform per sequence
    paged: bool = False
    page_size: int = 16
    accept: tuple = ("uniform",)            # ("uniform",) or ("geometric", mean)
    block: int = BLOCK
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6
    seed_index: int = 0
    ffn: int = 0                 # MLP width of a drafter layer (the target's, Qwen3)

    @property
    def rows(self) -> int:
        return self.batch * self.block

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def ctx_in(self) -> int:
        return self.n_ctx_layers * self.hidden


CONFIGS = [
    CycleConfig("tiny_b1", batch=1, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                vocab=4096, n_ctx_layers=2, ctx_len=128, accept=("uniform",), seed_index=0,
                ffn=768),
    CycleConfig("qwen3_4b_b1", batch=1, hidden=2560, n_q_heads=32, n_kv_heads=8, head_dim=128,
                vocab=151936, n_ctx_layers=5, ctx_len=2048, accept=("geometric", 13.0),
                seed_index=1, ffn=9728),
    CycleConfig("qwen3_8b_b1", batch=1, hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
                vocab=151936, n_ctx_layers=5, ctx_len=8192, accept=("uniform",), seed_index=2,
                ffn=12288),
    CycleConfig("qwen3_8b_b32_paged", batch=32, hidden=4096, n_q_heads=32, n_kv_heads=8,
                head_dim=128, vocab=151936, n_ctx_layers=5, ctx_len=0,
                ctx_len_range=(512, 16384), paged=True, page_size=16,
                accept=("geometric", 13.0), seed_index=3, ffn=12288),
    CycleConfig("qwen3_32b_b4_32k", batch=4, hidden=5120, n_q_heads=64, n_kv_heads=8,
                head_dim=128, vocab=151936, n_ctx_layers=5, ctx_len=32768,
                accept=("geometric", 12.0), seed_index=4, ffn=25600),
]
CONFIG_BY_NAME = {c.name: c for c in CONFIGS}


def scaled(cfg: CycleConfig, **over) -> CycleConfig:
    """A copy of ``cfg`` with some fields replaced (small parity cases)."""
    d = dict(cfg.__dict__)
    d.update(over)
    return CycleConfig(**d)


# --------------------------------------------------------------------------
# bf16 bit handling (input preparation only)
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0, mean: float = 0.0,
                chunk: int = 1 << 24) -> np.ndarray:
    """i.i.d. N(mean, std^2) values rounded to bf16 (uint16 bits), generated in chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        x = rng.standard_normal(m, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        if mean != 0.0:
            x += np.float32(mean)
        out[s:s + m] = f32_to_bf16_bits(x)
    return out.reshape(shape)


def unit_rms_rows_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """Rows of i.i.d. N(0,1) values rescaled to unit root-mean-square, as bf16 bits.

    This is the input recipe "hidden states ~N(0,1) then RMS-normalised" (unit gain).
    """
    x = rng.standard_normal(shape)
    x = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True))
    return f32_to_bf16_bits(x.astype(np.float32))


# --------------------------------------------------------------------------
# acceptance draws
# --------------------------------------------------------------------------
def geometric_ratio_for_mean(mean: float, n_max: int = 15) -> float:
    """Ratio q of the truncated law p(a=k) ∝ q^k, k = 0..n_max, with the given mean.

    Solved by bisection on the (monotone in q) mean of the truncated law.
    """
    ks = np.arange(n_max + 1, dtype=np.float64)

    def mean_of(q):
        w = np.exp(ks * np.log(q))
        return float(np.sum(ks * w) / np.sum(w))

    lo, hi = 1e-6, 1e6
    for _ in range(200):
        mid = np.sqrt(lo * hi)
        if mean_of(mid) < mean:
            lo = mid
        else:
            hi = mid
    return float(np.sqrt(lo * hi))


def draw_accept_lengths(rng: np.random.Generator, spec: tuple, batch: int,
                        n_max: int = BLOCK - 1) -> np.ndarray:
    """Draft match lengths a_b in 0..15 for each sequence."""
    if spec[0] == "uniform":
        return rng.integers(0, n_max + 1, size=batch).astype(np.int32)
    if spec[0] == "geometric":
        q = geometric_ratio_for_mean(float(spec[1]), n_max)
        ks = np.arange(n_max + 1)
        w = q ** ks
        p = w / w.sum()
        return rng.choice(ks, size=batch, p=p).astype(np.int32)
    raise ValueError(spec)


def make_block_ids(rng: np.random.Generator, posterior: np.ndarray, accept: np.ndarray,
                   vocab: int) -> np.ndarray:
    """Blocks [B,16]: staged token, then drafts that copy ``posterior`` for the first
    ``accept[b]`` positions, then one token that differs from the posterior, then
    uniform random tokens.

    ``posterior[b, i]`` is the target's greedy token after block position i, so
    draft position 1+i is the one compared with it.
    """
    posterior = np.asarray(posterior)
    B, T = posterior.shape
    blk = rng.integers(0, vocab, size=(B, T)).astype(np.int32)
    for b in range(B):
        a = int(accept[b])
        for i in range(a):
            blk[b, 1 + i] = posterior[b, i]
        if a < T - 1:
            t = int(rng.integers(0, vocab - 1))
            if t >= posterior[b, a]:
                t += 1
            blk[b, 1 + a] = t
    return blk


# --------------------------------------------------------------------------
# whole-cycle inputs
# --------------------------------------------------------------------------
STREAMS = ["layer_hidden", "w_fc", "hidden_norm_w", "w_k", "w_v", "k_norm_w",
           "ctx_k", "ctx_v", "q_blk", "k_blk", "v_blk", "verify_hidden", "w_lm",
           "blocks", "accept", "ctx_lens", "pages", "draft_x", "draft_w"]


def streams_for(cfg: CycleConfig) -> dict:
    ss = np.random.SeedSequence(1000 + cfg.seed_index)
    children = ss.spawn(len(STREAMS))
    return {name: np.random.default_rng(c) for name, c in zip(STREAMS, children)}


@dataclass
class CycleInputs:
    cfg: CycleConfig
    layer_hidden: list          # nL x uint16 [B*16, H]
    w_fc: np.ndarray            # uint16 [H, nL*H]
    hidden_norm_w: np.ndarray   # uint16 [H]
    w_k: np.ndarray             # uint16 [Hkv*D, H]
    w_v: np.ndarray             # uint16 [Hkv*D, H]
    k_norm_w: np.ndarray        # uint16 [D]
    ctx_len: np.ndarray         # int32 [B]  context length L_b before the block
    ctx_k: list                 # per sequence uint16 [L_b, Hkv, D] (post-RoPE)
    ctx_v: list                 # per sequence uint16 [L_b, Hkv, D]
    q_blk: np.ndarray           # uint16 [B,16,Hq,D] (pre-RoPE)
    k_blk: np.ndarray           # uint16 [B,16,Hkv,D]
    v_blk: np.ndarray           # uint16 [B,16,Hkv,D]
    verify_hidden: np.ndarray   # uint16 [B,16,H] final-normed target hidden
    w_lm: np.ndarray            # uint16 [V,H]
    accept_draw: np.ndarray     # int32 [B] planted match lengths
    rng_blocks: np.random.Generator = field(repr=False, default=None)


def make_cycle_inputs(cfg: CycleConfig, with_lm: bool = True) -> CycleInputs:
    """All seeded inputs of one cycle except the draft tokens (those need the
    target's posterior; see :func:`make_block_ids`)."""
    r = streams_for(cfg)
    B, T, H = cfg.batch, cfg.block, cfg.hidden
    Hq, Hkv, D = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    layer_hidden = [unit_rms_rows_bf16(r["layer_hidden"], (B * T, H))
                    for _ in range(cfg.n_ctx_layers)]
    w_fc = normal_bf16(r["w_fc"], (H, cfg.n_ctx_layers * H), 0.02)
    hidden_norm_w = normal_bf16(r["hidden_norm_w"], (H,), 0.02, mean=1.0)
    w_k = normal_bf16(r["w_k"], (Hkv * D, H), 0.02)
    w_v = normal_bf16(r["w_v"], (Hkv * D, H), 0.02)
    k_norm_w = normal_bf16(r["k_norm_w"], (D,), 0.02, mean=1.0)
    if cfg.ctx_len_range is not None:
        lo, hi = cfg.ctx_len_range
        ctx_len = r["ctx_lens"].integers(lo, hi + 1, size=B).astype(np.int32)
    else:
        ctx_len = np.full(B, cfg.ctx_len, dtype=np.int32)
    ctx_k = [normal_bf16(r["ctx_k"], (int(L), Hkv, D)) for L in ctx_len]
    ctx_v = [normal_bf16(r["ctx_v"], (int(L), Hkv, D)) for L in ctx_len]
    q_blk = normal_bf16(r["q_blk"], (B, T, Hq, D))
    k_blk = normal_bf16(r["k_blk"], (B, T, Hkv, D))
    v_blk = normal_bf16(r["v_blk"], (B, T, Hkv, D))
    verify_hidden = unit_rms_rows_bf16(r["verify_hidden"], (B, T, H))
    w_lm = normal_bf16(r["w_lm"], (cfg.vocab, H), 0.02) if with_lm else None
    accept_draw = draw_accept_lengths(r["accept"], cfg.accept, B)
    return CycleInputs(cfg, layer_hidden, w_fc, hidden_norm_w, w_k, w_v, k_norm_w, ctx_len,
                       ctx_k, ctx_v, q_blk, k_blk, v_blk, verify_hidden, w_lm, accept_draw,
                       rng_blocks=r["blocks"])


# --------------------------------------------------------------------------
# cache layouts
# --------------------------------------------------------------------------
@dataclass
class PagedLayout:
    page_size: int
    n_pages: int
    max_pages: int              # page-table columns per sequence
    page_table: np.ndarray      # int32 [B, max_pages]; -1 = unmapped
    free_list: np.ndarray       # int32 [n_pages]; first free_count entries are free
    free_count: int


def make_paged_layout(rng: np.random.Generator, seq_lens, reserve_tokens: int,
                      page_size: int = 16, slack_pages: int = 64,
                      max_len: Optional[int] = None) -> PagedLayout:
    """Shuffled page pool: sequence b owns ceil(L_b / page) pages drawn from a random
    permutation of the pool; every sequence can grow by ``reserve_tokens``."""
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    B = len(seq_lens)
    if max_len is None:
        max_len = int(seq_lens.max()) + reserve_tokens
    max_pages = (max_len + page_size - 1) // page_size
    need = [(int(L) + page_size - 1) // page_size for L in seq_lens]
    grow = [((int(L) + reserve_tokens + page_size - 1) // page_size) for L in seq_lens]
    n_pages = int(sum(grow)) + slack_pages
    perm = rng.permutation(n_pages).astype(np.int32)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    k = 0
    for b in range(B):
        table[b, :need[b]] = perm[k:k + need[b]]
        k += need[b]
    free = perm[k:].copy()
    free_list = np.full(n_pages, -1, dtype=np.int32)
    free_list[:len(free)] = free
    return PagedLayout(page_size, n_pages, max_pages, table, free_list, len(free))


def scatter_paged(layout: PagedLayout, per_seq: list, row_shape) -> np.ndarray:
    """Pack per-sequence rows [L_b, ...] into a page pool [n_pages, page, ...] (bits)."""
    P = layout.page_size
    pool = np.zeros((layout.n_pages, P) + tuple(row_shape), dtype=np.uint16)
    for b, rows in enumerate(per_seq):
        L = rows.shape[0]
        for p in range((L + P - 1) // P):
            pg = layout.page_table[b, p]
            n = min(P, L - p * P)
            pool[pg, :n] = rows[p * P:p * P + n]
    return pool


def scatter_paged_heads(layout: PagedLayout, per_seq: list, n_heads: int,
                        head_dim: int) -> np.ndarray:
    """Head-major page pool [n_pages, Hkv, page, D] from per-sequence rows [L_b, Hkv, D]."""
    pool = scatter_paged(layout, per_seq, (n_heads, head_dim))
    return np.ascontiguousarray(pool.transpose(0, 2, 1, 3))


def pack_contiguous_heads(per_seq: list, capacity: int, n_heads: int,
                          head_dim: int) -> np.ndarray:
    """Head-major contiguous cache [B, Hkv, capacity, D] from rows [L_b, Hkv, D]."""
    out = pack_contiguous(per_seq, capacity, (n_heads, head_dim))
    return np.ascontiguousarray(out.transpose(0, 2, 1, 3))


def pack_contiguous(per_seq: list, capacity: int, row_shape) -> np.ndarray:
    """Pack per-sequence rows [L_b, ...] into a contiguous cache [B, capacity, ...] (bits)."""
    B = len(per_seq)
    out = np.zeros((B, capacity) + tuple(row_shape), dtype=np.uint16)
    for b, rows in enumerate(per_seq):
        out[b, :rows.shape[0]] = rows
    return out


# --------------------------------------------------------------------------
# device-side generation (bench workloads: same distributions, generated on
# the GPU with a seeded torch generator so that gigabytes of weights do not
# have to be drawn on the host)
# --------------------------------------------------------------------------
def device_generator(cfg: CycleConfig, stream_name: str, device="cuda"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(1000 * (1 + cfg.seed_index) + STREAMS.index(stream_name))
    return g


def device_normal_bf16(gen, shape, std: float = 1.0, mean: float = 0.0, device="cuda"):
    """i.i.d. N(mean, std^2) as a CUDA bf16 tensor (round to nearest even)."""
    import torch
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(torch.bfloat16)


def device_unit_rms_rows_bf16(gen, shape, device="cuda"):
    """Rows of N(0,1) values rescaled to unit root-mean-square, CUDA bf16."""
    import torch
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    x = x / x.pow(2).mean(dim=-1, keepdim=True).sqrt()
    return x.to(torch.bfloat16)
