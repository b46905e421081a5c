"""GPU parity of dflash_ctx_project against the float64 oracle, through the
C ABI: the K/V rows written into contiguous and paged drafter caches, the
length update, page reservation, and the rows that must stay untouched."""
import numpy as np
import pytest
import torch

from oracle.dflash_oracle import ctx_project as ref_project
from oracle.dflash_oracle import pages_needed
from synthetic import (CONFIG_BY_NAME, make_cycle_inputs, make_paged_layout, normal_bf16,
                       unit_rms_rows_bf16)
from tests.gpu_helpers import assert_close_bf16, dev_bf16, dev_i32, host_bits, host_f64

pytestmark = pytest.mark.gpu
SENTINEL = 0x3F80  # bf16 1.0


def _dfl():
    import block_diffusion_speculative_02_gb300 as dfl
    return dfl


def make_inputs(seed, B, H, nL, Hkv, D):
    rng = np.random.default_rng(seed)
    layers = [unit_rms_rows_bf16(rng, (B * 16, H)) for _ in range(nL)]
    w_fc = normal_bf16(rng, (H, nL * H), 0.02)
    gh = normal_bf16(rng, (H,), 0.02, mean=1.0)
    wk = normal_bf16(rng, (Hkv * D, H), 0.02)
    wv = normal_bf16(rng, (Hkv * D, H), 0.02)
    gk = normal_bf16(rng, (D,), 0.02, mean=1.0)
    return layers, w_fc, gh, wk, wv, gk


def run_project(layers, w_fc, gh, wk, wv, gk, write_pos, Hq, Hkv, D, theta, paged=False,
                capacity=None, alias=False, seed=0, pool_slack=8, sm_budget=0):
    dfl = _dfl()
    B = len(write_pos)
    H = w_fc.shape[0]
    nL = len(layers)
    write_pos = np.asarray(write_pos, np.int32)
    max_ctx = int(write_pos.max()) + 16
    dims = dfl.make_dims(B, H, Hq, Hkv, D, 1000, nL, max_ctx, rope_theta=theta)
    ws = dfl.alloc_workspace(dims)
    dims.sm_budget = sm_budget          # grid size only: the workspace does not depend on it
    rng = np.random.default_rng(seed)
    lay = None
    if paged:
        lay = make_paged_layout(rng, write_pos, reserve_tokens=16, slack_pages=pool_slack)
        kc = torch.full((lay.n_pages, Hkv, 16, D), 1.0, dtype=torch.bfloat16, device="cuda")
        vc = kc.clone()
        view = dfl.KVView(kc, vc, dev_i32(write_pos if alias else np.zeros(B, np.int32)),
                          capacity=lay.max_pages * 16, page_table=dev_i32(lay.page_table),
                          free_list=dev_i32(lay.free_list), free_count=dev_i32([lay.free_count]),
                          page_size=16)
    else:
        cap = capacity or max_ctx + 3
        kc = torch.full((B, Hkv, cap, D), 1.0, dtype=torch.bfloat16, device="cuda")
        vc = kc.clone()
        view = dfl.KVView(kc, vc, dev_i32(write_pos if alias else np.zeros(B, np.int32)),
                          capacity=cap)
    wp = view.seq_len if alias else dev_i32(write_pos)
    dfl.dflash_ctx_project(dims, [dev_bf16(x) for x in layers], dev_bf16(w_fc),
                           None if gh is None else dev_bf16(gh), dev_bf16(wk), dev_bf16(wv),
                           None if gk is None else dev_bf16(gk), wp, view, ws)
    torch.cuda.synchronize()
    return view, lay, dfl.dflash_read_status(ws)


def gather_rows(view, lay, write_pos, Hkv, D):
    """Rows pos..pos+15 of every sequence as [B*16, Hkv, D] float64 (k, v)."""
    k = host_f64(view.k)
    v = host_f64(view.v)
    ks, vs = [], []
    table = view.page_table.cpu().numpy() if lay is not None else None
    for b, pos in enumerate(write_pos):
        for t in range(16):
            r = int(pos) + t
            if table is not None:
                pg = table[b, r // 16]
                ks.append(k[pg, :, r % 16])
                vs.append(v[pg, :, r % 16])
            else:
                ks.append(k[b, :, r])
                vs.append(v[b, :, r])
    return np.stack(ks), np.stack(vs)


def check_project(layers, w_fc, gh, wk, wv, gk, write_pos, Hq, Hkv, D, theta=1e6, paged=False,
                  alias=False, sm_budget=0):
    B = len(write_pos)
    pos = np.repeat(np.asarray(write_pos), 16) + np.tile(np.arange(16), B)
    ref = ref_project(layers, w_fc, gh, wk, wv, gk, pos, Hkv, D, theta, 1e-6)
    view, lay, status = run_project(layers, w_fc, gh, wk, wv, gk, write_pos, Hq, Hkv, D, theta,
                                    paged=paged, alias=alias, sm_budget=sm_budget)
    assert status == 0, status
    k, v = gather_rows(view, lay, write_pos, Hkv, D)
    ek = assert_close_bf16(k, ref["k"])
    ev = assert_close_bf16(v, ref["v"])
    assert np.array_equal(view.seq_len.cpu().numpy(), np.asarray(write_pos) + 16)
    return view, lay, ek, ev


@pytest.mark.parametrize("norms", [False, True])
def test_project_tiny(norms):
    layers, w_fc, gh, wk, wv, gk = make_inputs(1, 1, 256, 2, 2, 64)
    if not norms:
        gh = gk = None
    view, _, ek, ev = check_project(layers, w_fc, gh, wk, wv, gk, [128], 4, 2, 64)
    # rows outside the block keep their old contents
    kb = host_bits(view.k)
    assert np.all(kb[0, :, :128] == SENTINEL) and np.all(kb[0, :, 144:] == SENTINEL)
    print(ek, ev)


@pytest.mark.parametrize("B,H,nL,Hkv,D,pos", [
    (3, 512, 3, 2, 128, [0, 13, 100]),
    (17, 256, 2, 2, 64, list(range(0, 17 * 5, 5))),    # 272 token rows: two token chunks
    (2, 1024, 5, 8, 128, [2048, 7]),
])
def test_project_contiguous(B, H, nL, Hkv, D, pos):
    layers, w_fc, gh, wk, wv, gk = make_inputs(B + H, B, H, nL, Hkv, D)
    check_project(layers, w_fc, gh, wk, wv, gk, pos, 4 * Hkv, Hkv, D)


@pytest.mark.parametrize("sm_budget", [1, 3, 20])
@pytest.mark.parametrize("B,H,nL,Hkv,D,pos", [
    (17, 256, 2, 2, 64, list(range(0, 17 * 5, 5))),    # on part of the device: the tiled path
    (2, 1024, 5, 8, 128, [2048, 7]),
])
def test_project_small_sm_budget(sm_budget, B, H, nL, Hkv, D, pos):
    """Few CTAs: each streams a long run of (tile, k-stage) units crossing many
    tile boundaries, so several CTAs add into every tile."""
    layers, w_fc, gh, wk, wv, gk = make_inputs(B + H + sm_budget, B, H, nL, Hkv, D)
    check_project(layers, w_fc, gh, wk, wv, gk, pos, 4 * Hkv, Hkv, D, sm_budget=sm_budget)


def test_cycle_sm_split():
    dfl = _dfl()
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    cfg = CONFIG_BY_NAME["qwen3_8b_b1"]
    dims = dfl.make_dims(1, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.vocab,
                         cfg.n_ctx_layers, 8192)
    v, p = dfl.dflash_cycle_sm_split(dims)
    assert v + p == nsm and p >= 1 and v >= 1
    proj = cfg.n_ctx_layers * cfg.hidden ** 2 + 2 * cfg.n_kv_heads * cfg.head_dim * cfg.hidden
    share = proj / (proj + cfg.vocab * cfg.hidden)
    assert abs(p - nsm * share) <= 0.5 + 1e-9


def test_project_paged_reserves_pages():
    B, H, nL, Hkv, D = 4, 512, 2, 2, 128
    pos = [5, 16, 40, 63]                     # blocks straddling one or two pages
    layers, w_fc, gh, wk, wv, gk = make_inputs(7, B, H, nL, Hkv, D)
    view, lay, _, _ = check_project(layers, w_fc, gh, wk, wv, gk, pos, 8, Hkv, D, paged=True)
    table = view.page_table.cpu().numpy()
    before_free = set(lay.free_list[:lay.free_count].tolist())
    newly = []
    for b, slots in enumerate(pages_needed(pos, 16, 16)):
        for s in slots:
            assert table[b, s] >= 0
            if lay.page_table[b, s] < 0:
                newly.append(int(table[b, s]))
            else:
                assert table[b, s] == lay.page_table[b, s]
    assert len(set(newly)) == len(newly) and set(newly) <= before_free
    fc = int(view.free_count.item())
    assert fc == lay.free_count - len(newly)
    assert set(view.free_list.cpu().numpy()[:fc].tolist()) == before_free - set(newly)


@pytest.mark.parametrize("norms", [False, True])
def test_project_tiled_path_paged_and_aliased(norms):
    """Past 256 token rows (here 20 sequences) on part of the device the tiled
    GEMMs project: a paged cache with blocks straddling pages, write positions
    aliasing the lengths, both norm settings; rows and newly mapped pages as on
    the streamed path."""
    B, H, nL, Hkv, D = 20, 512, 3, 2, 128
    rng = np.random.default_rng(31)
    pos = [int(x) for x in rng.integers(0, 90, size=B)]
    layers, w_fc, gh, wk, wv, gk = make_inputs(11, B, H, nL, Hkv, D)
    if not norms:
        gh = gk = None
    view, lay, _, _ = check_project(layers, w_fc, gh, wk, wv, gk, pos, 4 * Hkv, Hkv, D,
                                    paged=True, alias=True, sm_budget=40)
    table = view.page_table.cpu().numpy()
    for b, slots in enumerate(pages_needed(pos, 16, 16)):
        assert all(table[b, s] >= 0 for s in slots)
    mapped = table[table >= 0]
    assert len(set(mapped.tolist())) == len(mapped)


def test_project_tiled_path_flags_capacity():
    """The tiled path, like the streamed one, leaves a sequence without room
    for its 16 rows untouched and flags it."""
    dfl = _dfl()
    B = 18
    layers, w_fc, gh, wk, wv, gk = make_inputs(12, B, 256, 2, 2, 64)
    pos = [0] * (B - 1) + [30]
    view, _, status = run_project(layers, w_fc, gh, wk, wv, gk, pos, 4, 2, 64, 1e6, capacity=40,
                                  sm_budget=30)
    assert status & dfl.dflash.STATUS_BITS["capacity"]
    assert list(view.seq_len.cpu().numpy()) == [16] * (B - 1) + [0]
    assert np.all(host_bits(view.k)[B - 1] == SENTINEL)


def test_project_write_pos_aliases_seq_len():
    layers, w_fc, gh, wk, wv, gk = make_inputs(8, 2, 256, 2, 2, 64)
    check_project(layers, w_fc, gh, wk, wv, gk, [33, 0], 4, 2, 64, alias=True)


def test_project_flags_capacity():
    dfl = _dfl()
    layers, w_fc, gh, wk, wv, gk = make_inputs(9, 2, 256, 2, 2, 64)
    view, _, status = run_project(layers, w_fc, gh, wk, wv, gk, [0, 30], 4, 2, 64, 1e6,
                                  capacity=40)
    assert status & dfl.dflash.STATUS_BITS["capacity"]
    assert list(view.seq_len.cpu().numpy()) == [16, 0]          # second sequence untouched
    assert np.all(host_bits(view.k)[1] == SENTINEL)


def test_project_flags_an_exhausted_page_pool():
    dfl = _dfl()
    B, H, Hkv, D = 2, 256, 2, 64
    layers, w_fc, gh, wk, wv, gk = make_inputs(10, B, H, 2, Hkv, D)
    dims = dfl.make_dims(B, H, 4, Hkv, D, 1000, 2, 64)
    ws = dfl.alloc_workspace(dims)
    table = np.full((B, 4), -1, np.int32)
    table[0, 0], table[1, 0] = 0, 1          # each sequence owns one page, needs a second
    free = np.array([2, -1, -1, -1], np.int32)
    kc = torch.full((4, Hkv, 16, D), 1.0, dtype=torch.bfloat16, device="cuda")
    view = dfl.KVView(kc, kc.clone(), dev_i32([0, 0]), capacity=64, page_table=dev_i32(table),
                      free_list=dev_i32(free), free_count=dev_i32([1]), page_size=16)
    dfl.dflash_ctx_project(dims, [dev_bf16(x) for x in layers], dev_bf16(w_fc), dev_bf16(gh),
                           dev_bf16(wk), dev_bf16(wv), dev_bf16(gk), dev_i32([8, 8]), view, ws)
    torch.cuda.synchronize()
    status = dfl.dflash_read_status(ws)
    assert status & dfl.dflash.STATUS_BITS["pool_empty"]
    assert status & dfl.dflash.STATUS_BITS["page_missing"]
    t = view.page_table.cpu().numpy()
    assert sorted([t[0, 1], t[1, 1]]) == [-1, 2]         # exactly one sequence got the page
    assert int(view.free_count.item()) == 0


@pytest.mark.parametrize("name", ["qwen3_4b_b1", "qwen3_8b_b1", "qwen3_8b_b32_paged",
                                  "qwen3_32b_b4_32k"])
def test_project_full_size(name):
    cfg = CONFIG_BY_NAME[name]
    inp = make_cycle_inputs(cfg, with_lm=False)
    pos = inp.ctx_len
    _, _, ek, ev = check_project(inp.layer_hidden, inp.w_fc, inp.hidden_norm_w, inp.w_k, inp.w_v,
                                 inp.k_norm_w, pos, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                                 cfg.rope_theta, paged=cfg.paged)
    print(cfg.name, ek, ev)
