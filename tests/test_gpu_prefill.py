"""GPU parity of dflash_ctx_prefill (the whole-prompt context projection) against
the float64 oracle, through the C ABI: rows written into contiguous and paged
drafter caches at write_pos .. write_pos + T - 1, the lengths, page
reservation, capacity errors, and a sampled check at a full prompt size."""
import numpy as np
import pytest
import torch

from oracle.dflash_oracle import ctx_project as ref_project
from synthetic import make_paged_layout, normal_bf16, unit_rms_rows_bf16
from tests.gpu_helpers import assert_close_bf16, dev_bf16, dev_i32, host_bits, host_f64

pytestmark = pytest.mark.gpu
SENTINEL = 0x3F80  # bf16 1.0
THETA = 1e6


def _dfl():
    import block_diffusion_speculative_02_gb300 as dfl
    return dfl


def make_inputs(seed, rows, H, nL, Hkv, D, norms=True):
    rng = np.random.default_rng(seed)
    layers = [unit_rms_rows_bf16(rng, (rows, H)) for _ in range(nL)]
    w_fc = normal_bf16(rng, (H, nL * H), 0.02)
    gh = normal_bf16(rng, (H,), 0.02, mean=1.0) if norms else None
    wk = normal_bf16(rng, (Hkv * D, H), 0.02)
    wv = normal_bf16(rng, (Hkv * D, H), 0.02)
    gk = normal_bf16(rng, (D,), 0.02, mean=1.0) if norms else None
    return layers, w_fc, gh, wk, wv, gk


def run_prefill(inp, write_pos, T, Hq, Hkv, D, paged=False, capacity=None, alias=False,
                seed=0):
    dfl = _dfl()
    layers, w_fc, gh, wk, wv, gk = inp
    B = len(write_pos)
    H = w_fc.shape[0]
    nL = len(layers)
    write_pos = np.asarray(write_pos, np.int32)
    dims = dfl.make_dims(B, H, Hq, Hkv, D, 1000, nL, int(write_pos.max()) + T, rope_theta=THETA)
    ws = dfl.dflash.alloc_prefill_workspace(dims, T)
    lay = None
    if paged:
        lay = make_paged_layout(np.random.default_rng(seed), write_pos, reserve_tokens=T,
                                slack_pages=4)
        kc = torch.full((lay.n_pages, Hkv, 16, D), 1.0, dtype=torch.bfloat16, device="cuda")
        view = dfl.KVView(kc, kc.clone(), dev_i32(write_pos if alias else np.zeros(B, np.int32)),
                          capacity=lay.max_pages * 16, page_table=dev_i32(lay.page_table),
                          free_list=dev_i32(lay.free_list), free_count=dev_i32([lay.free_count]),
                          page_size=16)
    else:
        cap = capacity or int(write_pos.max()) + T + 5
        kc = torch.full((B, Hkv, cap, D), 1.0, dtype=torch.bfloat16, device="cuda")
        view = dfl.KVView(kc, kc.clone(), dev_i32(write_pos if alias else np.zeros(B, np.int32)),
                          capacity=cap)
    wp = view.seq_len if alias else dev_i32(write_pos)
    dfl.dflash.dflash_ctx_prefill(dims, T, [dev_bf16(x) for x in layers], dev_bf16(w_fc),
                                  None if gh is None else dev_bf16(gh), dev_bf16(wk),
                                  dev_bf16(wv), None if gk is None else dev_bf16(gk), wp, view, ws)
    torch.cuda.synchronize()
    return view, lay, dfl.dflash_read_status(ws)


def gather(view, lay, write_pos, T, rows_of_seq=None):
    """Rows (b, t) of the cache as [n, Hkv, D] float64 (k, v)."""
    k, v = host_f64(view.k), host_f64(view.v)
    table = view.page_table.cpu().numpy() if lay is not None else None
    ks, vs = [], []
    for b, pos in enumerate(write_pos):
        for t in (range(T) if rows_of_seq is None else rows_of_seq[b]):
            r = int(pos) + t
            if table is not None:
                pg = table[b, r // 16]
                ks.append(k[pg, :, r % 16])
                vs.append(v[pg, :, r % 16])
            else:
                ks.append(k[b, :, r])
                vs.append(v[b, :, r])
    return np.stack(ks), np.stack(vs)


def check(inp, write_pos, T, Hq, Hkv, D, paged=False, alias=False):
    layers, w_fc, gh, wk, wv, gk = inp
    pos = (np.repeat(np.asarray(write_pos), T) + np.tile(np.arange(T), len(write_pos)))
    ref = ref_project(layers, w_fc, gh, wk, wv, gk, pos, Hkv, D, THETA, 1e-6)
    view, lay, status = run_prefill(inp, write_pos, T, Hq, Hkv, D, paged=paged, alias=alias)
    assert status == 0, status
    k, v = gather(view, lay, write_pos, T)
    ek = assert_close_bf16(k, ref["k"])
    ev = assert_close_bf16(v, ref["v"])
    assert np.array_equal(view.seq_len.cpu().numpy(), np.asarray(write_pos) + T)
    return view, lay, ek, ev


@pytest.mark.parametrize("norms", [False, True])
def test_prefill_tiny(norms):
    """80 token rows: one ragged row tile; K/V tiles of 128 features (two
    heads of 64)."""
    inp = make_inputs(1, 2 * 40, 256, 2, 2, 64, norms=norms)
    view, _, ek, ev = check(inp, [0, 3], 40, 4, 2, 64)
    kb = host_bits(view.k)
    assert np.all(kb[0, :, 40:] == SENTINEL) and np.all(kb[1, :, :3] == SENTINEL)
    print(ek, ev)


@pytest.mark.parametrize("B,T,H,nL,Hkv,D,pos", [
    (3, 700, 512, 3, 2, 128, [0, 9, 130]),      # 17 row tiles: more than one raster band
    (1, 130, 2560, 5, 8, 128, [64]),            # Qwen3-4B widths, ragged tail of 2 rows
    (2, 129, 1024, 2, 4, 64, [1, 0]),           # 64-dim heads in 256-feature tiles
])
def test_prefill_contiguous(B, T, H, nL, Hkv, D, pos):
    inp = make_inputs(B * T + H, B * T, H, nL, Hkv, D)
    check(inp, pos, T, 4 * Hkv, Hkv, D)


def test_prefill_paged_reserves_pages():
    B, T, H, nL, Hkv, D = 2, 100, 512, 2, 2, 128
    pos = [5, 37]
    inp = make_inputs(7, B * T, H, nL, Hkv, D)
    view, lay, _, _ = check(inp, pos, T, 8, Hkv, D, paged=True)
    table = view.page_table.cpu().numpy()
    before_free = set(lay.free_list[:lay.free_count].tolist())
    newly = []
    for b, p0 in enumerate(pos):
        for s in range(p0 // 16, (p0 + T - 1) // 16 + 1):
            assert table[b, s] >= 0
            if lay.page_table[b, s] < 0:
                newly.append(int(table[b, s]))
            else:
                assert table[b, s] == lay.page_table[b, s]
    assert len(set(newly)) == len(newly) and set(newly) <= before_free
    assert int(view.free_count.item()) == lay.free_count - len(newly)


def test_prefill_write_pos_aliases_seq_len():
    inp = make_inputs(8, 2 * 50, 256, 2, 2, 64)
    check(inp, [33, 0], 50, 4, 2, 64, alias=True)


def test_prefill_flags_capacity():
    dfl = _dfl()
    inp = make_inputs(9, 2 * 40, 256, 2, 2, 64)
    view, _, status = run_prefill(inp, [0, 30], 40, 4, 2, 64, capacity=60)
    assert status & dfl.dflash.STATUS_BITS["capacity"]
    assert list(view.seq_len.cpu().numpy()) == [40, 0]          # second sequence untouched
    assert np.all(host_bits(view.k)[1] == SENTINEL)
    k, _ = gather(view, None, [0], 40)
    layers, w_fc, gh, wk, wv, gk = inp
    ref = ref_project([x[:40] for x in layers], w_fc, gh, wk, wv, gk, np.arange(40), 2, 64,
                      THETA, 1e-6)
    assert_close_bf16(k, ref["k"])


def test_prefill_flags_an_exhausted_page_pool():
    """Two 40-row prompts need three pages each; the pool holds four.  Every
    free page is handed out exactly once, the statuses are raised, the rows
    that got a page are correct and the others are skipped."""
    dfl = _dfl()
    B, T, H, nL, Hkv, D = 2, 40, 256, 2, 2, 64
    inp = make_inputs(12, B * T, H, nL, Hkv, D)
    layers, w_fc, gh, wk, wv, gk = inp
    dims = dfl.make_dims(B, H, 4, Hkv, D, 1000, nL, 64, rope_theta=THETA)
    ws = dfl.dflash.alloc_prefill_workspace(dims, T)
    n_pages = 4
    kc = torch.full((n_pages, Hkv, 16, D), 1.0, dtype=torch.bfloat16, device="cuda")
    table = np.full((B, 4), -1, np.int32)
    free = np.array([3, 0, 2, 1], np.int32)
    view = dfl.KVView(kc, kc.clone(), dev_i32([0, 0]), capacity=64, page_table=dev_i32(table),
                      free_list=dev_i32(free), free_count=dev_i32([4]), page_size=16)
    dfl.dflash.dflash_ctx_prefill(dims, T, [dev_bf16(x) for x in layers], dev_bf16(w_fc),
                                  dev_bf16(gh), dev_bf16(wk), dev_bf16(wv), dev_bf16(gk),
                                  dev_i32([0, 0]), view, ws)
    torch.cuda.synchronize()
    status = dfl.dflash_read_status(ws)
    assert status & dfl.dflash.STATUS_BITS["pool_empty"]
    assert status & dfl.dflash.STATUS_BITS["page_missing"]
    assert int(view.free_count.item()) == 0
    t = view.page_table.cpu().numpy()
    got = t[t >= 0]
    assert sorted(got.tolist()) == [0, 1, 2, 3]
    pos = np.tile(np.arange(T), B)
    ref = ref_project(layers, w_fc, gh, wk, wv, gk, pos, Hkv, D, THETA, 1e-6)
    k = host_f64(view.k)
    checked = 0
    for b in range(B):
        for r in range(T):
            pg = t[b, r // 16]
            if pg < 0:
                continue
            assert_close_bf16(k[pg, :, r % 16], ref["k"][b * T + r])
            checked += 1
    assert checked >= 48      # the four pages carry 64 rows, at most 16 of them past 40


def test_prefill_chunks_equal_one_call():
    """A prompt projected in two chunks (the second at write_pos = the first's
    length) lands where one call over the whole prompt puts it."""
    dfl = _dfl()
    H, nL, Hkv, D, T = 256, 2, 2, 64, 96
    inp = make_inputs(11, T, H, nL, Hkv, D)
    layers, w_fc, gh, wk, wv, gk = inp
    whole, _, st = run_prefill(inp, [0], T, 4, Hkv, D, capacity=T)
    assert st == 0
    dims = dfl.make_dims(1, H, 4, Hkv, D, 1000, nL, T, rope_theta=THETA)
    kc = torch.full((1, Hkv, T, D), 1.0, dtype=torch.bfloat16, device="cuda")
    view = dfl.KVView(kc, kc.clone(), dev_i32([0]), capacity=T)
    for lo, hi in ((0, 40), (40, T)):
        ws = dfl.dflash.alloc_prefill_workspace(dims, hi - lo)
        dfl.dflash.dflash_ctx_prefill(dims, hi - lo, [dev_bf16(x[lo:hi]) for x in layers],
                                      dev_bf16(w_fc), dev_bf16(gh), dev_bf16(wk), dev_bf16(wv),
                                      dev_bf16(gk), view.seq_len, view, ws)
        torch.cuda.synchronize()
        assert dfl.dflash_read_status(ws) == 0
    assert int(view.seq_len.item()) == T
    # rows are computed independently, so the chunked and whole results are
    # the same up to the order of fp32 additions (none here: same tiles)
    np.testing.assert_array_equal(host_bits(view.k), host_bits(whole.k))
    np.testing.assert_array_equal(host_bits(view.v), host_bits(whole.v))


def test_prefill_qwen3_8b_sampled_rows():
    """Qwen3-8B widths (H 4096, 5 layers, 8 KV heads of 128) at an 8192-token
    prompt, the size the bench times; the oracle checks 48 sampled rows (the
    projection is row-independent), plus the lengths."""
    dfl = _dfl()
    B, T, H, nL, Hkv, D = 1, 8192, 4096, 5, 8, 128
    rng = np.random.default_rng(2024)
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    layers_d = [torch.randn((T, H), generator=g, device="cuda").to(torch.bfloat16)
                for _ in range(nL)]
    w_fc = normal_bf16(rng, (H, nL * H), 0.02)
    gh = normal_bf16(rng, (H,), 0.02, mean=1.0)
    wk = normal_bf16(rng, (Hkv * D, H), 0.02)
    wv = normal_bf16(rng, (Hkv * D, H), 0.02)
    gk = normal_bf16(rng, (D,), 0.02, mean=1.0)
    dims = dfl.make_dims(B, H, 32, Hkv, D, 1000, nL, T, rope_theta=THETA)
    ws = dfl.dflash.alloc_prefill_workspace(dims, T)
    kc = torch.full((B, Hkv, T, D), 1.0, dtype=torch.bfloat16, device="cuda")
    view = dfl.KVView(kc, kc.clone(), dev_i32([0]), capacity=T)
    dfl.dflash.dflash_ctx_prefill(dims, T, layers_d, dev_bf16(w_fc), dev_bf16(gh), dev_bf16(wk),
                                  dev_bf16(wv), dev_bf16(gk), dev_i32([0]), view, ws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    assert int(view.seq_len.item()) == T
    rows = np.sort(np.concatenate([[0, 127, 128, T - 1], rng.choice(T, 44, replace=False)]))
    rows = np.unique(rows)
    idx = torch.from_numpy(rows).cuda()
    layers = [host_bits(x.index_select(0, idx)) for x in layers_d]
    ref = ref_project(layers, w_fc, gh, wk, wv, gk, rows, Hkv, D, THETA, 1e-6)
    k, v = gather(view, None, [0], T, rows_of_seq=[rows])
    print(assert_close_bf16(k, ref["k"]), assert_close_bf16(v, ref["v"]))
