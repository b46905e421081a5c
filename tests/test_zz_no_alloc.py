"""The allocation-free verify entry point, for callers that cannot allocate
device memory (plugins without an allocator, fixed memory budgets, code that
must not allocate during stream capture): called through the C ABI, its
results must equal those of dflash_verify_accept on the same inputs on every
one of two calls in a row, with the second call reusing the shared scratch
the first one left behind.

Collected last on purpose, so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from synthetic import draw_accept_lengths, make_block_ids, normal_bf16, unit_rms_rows_bf16
from tests.gpu_helpers import dev_bf16, dev_i32

pytestmark = pytest.mark.gpu


def _outputs(B, cap):
    return [torch.full((B, 16), -3, dtype=torch.int32, device="cuda"),
            torch.full((B,), -3, dtype=torch.int32, device="cuda"),
            torch.full((B,), -3, dtype=torch.int32, device="cuda"),
            torch.full((B,), -3, dtype=torch.int32, device="cuda"),
            torch.full((B, cap), -3, dtype=torch.int32, device="cuda")]


@pytest.mark.parametrize("B,H,V", [(1, 512, 30011), (4, 256, 20000), (32, 256, 9001)])
def test_noalloc_matches_workspace_entry_point_twice(B, H, V):
    import __graft_entry__
    __graft_entry__.build()
    from block_diffusion_speculative_02_gb300 import dflash as dfl

    lib = dfl.load_library()
    fn = lib.dflash_verify_accept_noalloc
    fn.restype = ctypes.c_int
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(dfl.Dims), vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int32,
                   vp]
    rng = np.random.default_rng(B * 7 + H)
    dims = dfl.make_dims(B, H, 4, 4, 128, V, 1, 64)
    ws = dfl.alloc_workspace(dims)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cap = 48
    for call in range(2):
        hidden = dev_bf16(unit_rms_rows_bf16(rng, (B * 16, H)))
        w = dev_bf16(normal_bf16(rng, (V, H), 0.02))
        # plant drafts from the workspace entry point's own posterior
        probe = _outputs(B, cap)
        zeros = dev_i32(np.zeros((B, 16)))
        lb = dev_i32(rng.integers(0, 20, size=B))
        dfl.dflash_verify_accept(dims, hidden, w, zeros, lb, *probe, ws)
        torch.cuda.synchronize()
        blk = dev_i32(make_block_ids(rng, probe[0].cpu().numpy(),
                                     draw_accept_lengths(rng, ("uniform",), B), V))
        ref = _outputs(B, cap)
        dfl.dflash_verify_accept(dims, hidden, w, blk, lb, *ref, ws)
        got = _outputs(B, cap)
        rc = fn(ctypes.byref(dims), hidden.data_ptr(), w.data_ptr(), blk.data_ptr(),
                lb.data_ptr(), *[t.data_ptr() for t in got], cap, stream)
        assert rc == 0, dfl.status_string(rc)
        torch.cuda.synchronize()
        # the workspace entry point's status (the variant reports none)
        assert dfl.dflash_read_status(ws) == 0
        for r, g in zip(ref, got):
            assert torch.equal(r, g), call


def test_noalloc_rejects_batches_past_its_scratch():
    import __graft_entry__
    __graft_entry__.build()
    from block_diffusion_speculative_02_gb300 import dflash as dfl

    lib = dfl.load_library()
    fn = lib.dflash_verify_accept_noalloc
    fn.restype = ctypes.c_int
    # 528 token rows > 512: refused by the shape check every entry point shares,
    # whose 512-row limit the scratch array covers (a static assertion in the
    # library ties the two), before anything is launched
    dims = dfl.make_dims(33, 256, 4, 4, 128, 1000, 1, 64)
    t = torch.zeros(16, dtype=torch.int32, device="cuda")
    rc = fn(ctypes.byref(dims), *([ctypes.c_void_p(t.data_ptr())] * 9), ctypes.c_int32(16),
            ctypes.c_void_p(0))
    assert rc != 0
