"""Host-side argument checks and workspace sizing of the later entry points,
exercised without a GPU: every case here is refused (or sized) before any
CUDA call, so nothing is launched."""
import ctypes

import pytest

E_ARG, E_ALIGN, E_UNSUPPORTED = -1, -2, -3


def _lib():
    import __graft_entry__
    __graft_entry__.build()
    from block_diffusion_speculative_02_gb300 import dflash
    return dflash, dflash.load_library()


def test_prefill_workspace_layout():
    """One workspace serves both prefill calls.  The context projection's:
    status (256 B) | write-position snapshot | per-tile sums of Y^2 |
    bf16(g_h * Y), each region 256-byte aligned, 256-feature tiles when the
    hidden size allows them.  The attention's: status (256 B) | split partials
    (O, then max and sum) when the chunk's (sequence, sub-block, KV head)
    units are fewer than 152, split ceil(152 / units) ways (at most 64, at
    most one per 16 context rows); a sub-block is 32 prompt rows when the G
    query heads of a KV head fill the 128 MMA rows with them (G <= 4), else
    16."""
    dflash, _ = _lib()
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for B, T, H in ((1, 8192, 4096), (2, 100, 512), (3, 7, 384)):
        dims = dflash.make_dims(B, H, 32, 8, 128, 1000, 5, T)
        rows = B * T
        tiles = H // 256 if H % 256 == 0 else H // 128
        proj = 256 + al(4 * B) + al(4 * tiles * rows) + al(2 * rows * H)
        G = 32 // 8
        sub = 32 if G * 32 <= 128 else 16             # prompt rows per CTA
        units = B * -(-T // sub) * 8
        splits = 1 if units >= 152 else min(-(-152 // units), -(-T // 16), 64)
        att = 256
        if splits > 1:
            n = units * splits * G * sub
            att = al(256 + 4 * n * 128 + 8 * n)
        assert dflash.dflash_prefill_workspace_bytes(dims, T) == max(proj, att), (B, T, H)


def test_prefill_rejects_bad_shapes_before_launching():
    dflash, lib = _lib()
    dims = dflash.make_dims(1, 4096, 32, 8, 128, 1000, 5, 64)
    with pytest.raises(dflash.DFlashError):
        dflash.dflash_prefill_workspace_bytes(dims, 0)           # no rows
    odd = dflash.make_dims(1, 4096, 32, 1, 64, 1000, 5, 64)     # K/V width 64: not a tile
    with pytest.raises(dflash.DFlashError):
        dflash.dflash_prefill_workspace_bytes(odd, 16)
    ptrs = (ctypes.c_void_p * 5)(*([0x1000] * 5))
    view = dflash.KVViewC()
    rc = lib.dflash_ctx_prefill(ctypes.byref(dims), 16, ptrs, 0x1000, None, 0x1000, 0x1000, None,
                                0x1000, ctypes.byref(view), 0x1000, 1 << 30, None)
    assert rc == E_ARG                                           # cache pointers missing


def test_gdn_replay_rejects_bad_arguments_before_launching():
    _, lib = _lib()
    p = 0x1000  # never dereferenced: every case fails a host check first
    f = lib.dflash_gdn_replay
    assert f(1, 4, 96, 128, p, p, p, p, p, p, p, 256, None) == E_UNSUPPORTED   # Dk 96
    assert f(1, 4, 128, 32, p, p, p, p, p, p, p, 256, None) == E_UNSUPPORTED   # Dv 32
    assert f(0, 4, 128, 128, p, p, p, p, p, p, p, 256, None) == E_ARG          # no sequences
    assert f(1, 4, 128, 128, None, p, p, p, p, p, p, 256, None) == E_ARG       # no state
    assert f(1, 4, 128, 128, p + 4, p, p, p, p, p, p, 256, None) == E_ALIGN    # misaligned state
    assert f(1, 4, 128, 128, p, p + 2, p, p, p, p, p, 256, None) == E_ALIGN    # misaligned keys


def test_fault_injection_returns_before_any_check(monkeypatch):
    """DFLASH_FAULT_INJECT makes the named entry point fail before it looks at
    its arguments (so even null pointers give the injected code), and leaves
    the other entry points alone."""
    _, lib = _lib()
    p = 0x1000
    monkeypatch.setenv("DFLASH_FAULT_INJECT", "dflash_gdn_replay")
    assert lib.dflash_gdn_replay(0, 0, 0, 0, None, None, None, None, None, None, None, 0,
                                 None) == -5
    assert lib.dflash_kv_crop(None, 0, None, 0, None, 0, None) == E_ARG     # not injected
    monkeypatch.setenv("DFLASH_FAULT_INJECT", "dflash_kv_crop:-4")
    assert lib.dflash_kv_crop(None, 0, None, 0, None, 0, None) == -4
    assert lib.dflash_gdn_replay(1, 4, 96, 128, p, p, p, p, p, p, p, 256, None) == E_UNSUPPORTED
    monkeypatch.setenv("DFLASH_FAULT_INJECT", "dflash_kv")                 # a prefix only
    assert lib.dflash_kv_crop(None, 0, None, 0, None, 0, None) == E_ARG
    monkeypatch.delenv("DFLASH_FAULT_INJECT")
    assert lib.dflash_selftest_wait(1, None, 0, None) == -4                 # no workspace
