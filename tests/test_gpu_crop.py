"""GPU parity of dflash_kv_crop (contiguous and paged views in one call)."""
import numpy as np
import pytest
import torch

from oracle.dflash_oracle import kv_crop_lengths, kv_crop_paged
from synthetic import make_paged_layout
from tests.gpu_helpers import dev_i32

pytestmark = pytest.mark.gpu


def _dfl():
    import block_diffusion_speculative_02_gb300 as dfl
    return dfl


def test_crop_contiguous_and_paged_views_together():
    dfl = _dfl()
    rng = np.random.default_rng(0)
    B = 32
    lens = rng.integers(512, 16385, size=B).astype(np.int32)
    lay = make_paged_layout(rng, lens, reserve_tokens=16)
    acc = rng.integers(0, 16, size=B)
    base = lens - 16                            # rows written by the last block end at lens
    new_len = (base + 1 + acc).astype(np.int32)
    new_len[3] = lens[3]                        # unchanged length
    new_len[4] = lens[4] + 1                    # invalid: would grow
    new_len[5] = 0                              # crop everything
    new_len[6] = (lens[6] // 16) * 16           # page-aligned: the page starting there goes
    dims = dfl.make_dims(B, 128, 1, 1, 128, 16, 1, 64)
    ws = dfl.alloc_workspace(dims)
    paged = dfl.KVView(None, None, dev_i32(lens), capacity=lay.max_pages * 16,
                       page_table=dev_i32(lay.page_table), free_list=dev_i32(lay.free_list),
                       free_count=dev_i32([lay.free_count]), page_size=16)
    contig_len = (lens + 5).astype(np.int32)
    contig_len[4] = lens[4]                     # keep the invalid one invalid in both views
    contig = dfl.KVView(None, None, dev_i32(contig_len), capacity=20000)
    dfl.dflash_kv_crop([paged, contig], dev_i32(new_len), B, ws)
    torch.cuda.synchronize()
    status = dfl.dflash_read_status(ws)
    assert status == dfl.dflash.STATUS_BITS["crop_grow"]

    ref = kv_crop_paged(lens, lay.page_table, set(lay.free_list[:lay.free_count].tolist()),
                        new_len, 16)
    assert np.array_equal(paged.seq_len.cpu().numpy(), ref["seq_len"])
    assert np.array_equal(paged.page_table.cpu().numpy(), ref["page_table"])
    fc = int(paged.free_count.item())
    fl = paged.free_list.cpu().numpy()
    assert fc == len(ref["free"])
    assert set(fl[:fc].tolist()) == ref["free"] and len(set(fl[:fc].tolist())) == fc
    cl, bad = kv_crop_lengths(contig_len, new_len)
    assert np.array_equal(contig.seq_len.cpu().numpy(), cl)
    assert bad[4] and not bad[:4].any()


def test_crop_rejects_bad_arguments():
    dfl = _dfl()
    dims = dfl.make_dims(1, 128, 1, 1, 128, 16, 1, 64)
    ws = dfl.alloc_workspace(dims)
    v = dfl.KVView(None, None, dev_i32([5]), capacity=8)
    with pytest.raises(dfl.DFlashError):
        dfl.dflash_kv_crop([v] * 5, dev_i32([1]), 1, ws)       # too many views
    with pytest.raises(dfl.DFlashError):
        dfl.dflash_kv_crop([v], dev_i32([1]), 0, ws)           # empty batch


def test_crop_keeps_a_page_that_would_overflow_a_full_free_list():
    """An inconsistent pool (free list already holding n_pages entries while a
    sequence still maps pages): the length is cut, the page that cannot be
    pushed stays mapped (nothing is lost or written past the list) and
    DFLASH_ST_CAPACITY is set."""
    dfl = _dfl()
    n_pages = 4
    table = np.array([[0, 1, -1, -1]], np.int32)          # sequence 0 maps pages 0 and 1
    free = np.array([0, 1, 2, 3], np.int32)               # ... and all four are listed free
    dims = dfl.make_dims(1, 128, 1, 1, 128, 16, 1, 64)
    ws = dfl.alloc_workspace(dims)
    view = dfl.KVView(None, None, dev_i32([30]), capacity=64, page_table=dev_i32(table),
                      free_list=dev_i32(free), free_count=dev_i32([n_pages]), page_size=16)
    dfl.dflash_kv_crop([view], dev_i32([5]), 1, ws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == dfl.dflash.STATUS_BITS["capacity"]
    assert int(view.seq_len.item()) == 5
    assert view.page_table.cpu().numpy().tolist() == [[0, 1, -1, -1]]
    assert int(view.free_count.item()) == n_pages
    assert view.free_list.cpu().numpy().tolist() == free.tolist()
