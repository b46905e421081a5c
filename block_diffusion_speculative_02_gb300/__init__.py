"""DFlash per-cycle hot path on GB300: hand-written sm_103a CUDA kernels behind a C ABI.

The four calls of one draft/verify cycle (context projection, dual-source
block attention, verification epilogue, KV-cache crop) live in
``libdflash.so``; :mod:`.dflash` is the ctypes binding that the tests and the
bench call.
"""
from . import dflash  # noqa: F401
from .dflash import (DFlashError, Dims, KVView, alloc_workspace, dflash_block_attention,  # noqa
                     dflash_ctx_project, dflash_cycle_sm_split, dflash_kv_crop,
                     dflash_read_status, dflash_verify_accept, dflash_workspace_bytes,
                     dflash_workspace_init, load_library, make_dims, with_sm_budget)
