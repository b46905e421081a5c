"""DFlash per-cycle hot path on GB300: hand-written sm_103a CUDA kernels behind a C ABI.

``libdflash.so`` holds the four calls of one draft/verify cycle (context
projection, dual-source block attention, verification epilogue, KV-cache
crop) and the calls around it: the rest of the drafter layer and its token
choice (``dflash_draft_qkv``, ``dflash_draft_mlp``, ``dflash_draft_tokens``),
the target's verify attention, the prefill (the target's attention over
prompt chunks, ``dflash_prefill_attention``, its first staged token,
``dflash_prefill_staged``, and the whole-prompt context projection,
``dflash_ctx_prefill``) and the GatedDeltaNet tape-replay rollback
(``dflash_gdn_replay``).  :mod:`.dflash` is the ctypes binding (argument
marshalling only); :mod:`.cycle` composes one cycle (``run_cycle``), captures
it as a CUDA graph (``CycleGraph``) and runs the serving loop with the input
copies overlapped (``PipelinedCycles``).
"""
from . import dflash  # noqa: F401
from .dflash import (DFlashError, Dims, KVView, alloc_draft_workspace,  # noqa: F401
                     alloc_prefill_workspace, alloc_workspace, dflash_block_attention,
                     dflash_ctx_prefill, dflash_ctx_project, dflash_cycle_sm_split,
                     dflash_draft_mlp, dflash_draft_qkv, dflash_draft_tokens, dflash_gdn_replay,
                     dflash_kv_crop, dflash_prefill_attention, dflash_prefill_staged,
                     dflash_read_status, dflash_verify_accept,
                     dflash_verify_attention, dflash_workspace_bytes, dflash_workspace_init,
                     load_library, make_dims, with_sm_budget)
