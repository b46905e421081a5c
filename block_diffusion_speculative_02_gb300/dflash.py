"""Thin ctypes binding of ``libdflash.so`` (the C ABI in include/dflash.h).

Argument marshalling only: every function takes torch tensors that already
live on the GPU, passes their device pointers and the current CUDA stream to
the library, and raises :class:`DFlashError` on a negative return code.  All
arithmetic happens in the CUDA kernels; there is no CPU fallback, and the
module refuses to load when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# DFLASH_LIBRARY may name another build of the same library (e.g. one compiled
# with different tile parameters); the default is the in-tree build.
LIB_PATH = os.environ.get("DFLASH_LIBRARY") or os.path.join(_PKG, "libdflash.so")

DFLASH_OK = 0
STATUS_BITS = {
    "crop_grow": 1 << 0,
    "out_overflow": 1 << 1,
    "page_missing": 1 << 2,
    "pool_empty": 1 << 3,
    "bad_token": 1 << 4,
    "capacity": 1 << 5,
    "timeout": 1 << 6,
}

EXPORTED = ["dflash_workspace_bytes", "dflash_workspace_init", "dflash_ctx_project",
            "dflash_block_attention", "dflash_verify_accept", "dflash_kv_crop",
            "dflash_read_status", "dflash_status_string", "dflash_version",
            "dflash_verify_accept_noalloc", "dflash_cycle_sm_split",
            "dflash_draft_workspace_bytes", "dflash_draft_qkv", "dflash_draft_mlp",
            "dflash_draft_tokens", "dflash_verify_attention", "dflash_gdn_replay",
            "dflash_prefill_workspace_bytes", "dflash_ctx_prefill", "dflash_selftest_wait",
            "dflash_prefill_attention", "dflash_prefill_staged"]


class DFlashError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


class Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("block", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("n_ctx_layers", ctypes.c_int32),
                ("max_ctx", ctypes.c_int32), ("rope_theta", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("sm_budget", ctypes.c_int32)]


class KVViewC(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("seq_len", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("free_list", ctypes.c_void_p), ("free_count", ctypes.c_void_p),
                ("capacity", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_pages", ctypes.c_int32), ("n_pages", ctypes.c_int32)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lib.dflash_workspace_bytes.restype = sz
    lib.dflash_workspace_bytes.argtypes = [ctypes.POINTER(Dims)]
    lib.dflash_workspace_init.restype = ctypes.c_int
    lib.dflash_workspace_init.argtypes = [vp, sz, vp]
    lib.dflash_ctx_project.restype = ctypes.c_int
    lib.dflash_ctx_project.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(vp), vp, vp, vp, vp,
                                       vp, vp, ctypes.POINTER(KVViewC), vp, sz, vp]
    lib.dflash_block_attention.restype = ctypes.c_int
    lib.dflash_block_attention.argtypes = [ctypes.POINTER(Dims), vp, vp, vp,
                                           ctypes.POINTER(KVViewC), ctypes.c_float, vp, vp, sz,
                                           vp]
    lib.dflash_verify_attention.restype = ctypes.c_int
    lib.dflash_verify_attention.argtypes = [ctypes.POINTER(Dims), vp, vp, vp,
                                            ctypes.POINTER(KVViewC), ctypes.c_float, vp, vp, sz,
                                            vp]
    lib.dflash_selftest_wait.restype = ctypes.c_int
    lib.dflash_selftest_wait.argtypes = [ctypes.c_int, vp, sz, vp]
    lib.dflash_prefill_workspace_bytes.restype = sz
    lib.dflash_prefill_workspace_bytes.argtypes = [ctypes.POINTER(Dims), i32]
    lib.dflash_ctx_prefill.restype = ctypes.c_int
    lib.dflash_ctx_prefill.argtypes = [ctypes.POINTER(Dims), i32, ctypes.POINTER(vp), vp, vp, vp,
                                       vp, vp, vp, ctypes.POINTER(KVViewC), vp, sz, vp]
    lib.dflash_prefill_attention.restype = ctypes.c_int
    lib.dflash_prefill_attention.argtypes = [ctypes.POINTER(Dims), i32, vp, vp, vp,
                                             ctypes.POINTER(KVViewC), ctypes.c_float, vp, vp, sz,
                                             vp]
    lib.dflash_prefill_staged.restype = ctypes.c_int
    lib.dflash_prefill_staged.argtypes = [ctypes.POINTER(Dims), vp, ctypes.c_int64, vp, vp, vp,
                                          sz, vp]
    lib.dflash_gdn_replay.restype = ctypes.c_int
    lib.dflash_gdn_replay.argtypes = [i32, i32, i32, i32] + [vp] * 6 + [vp, sz, vp]
    lib.dflash_verify_accept.restype = ctypes.c_int
    lib.dflash_verify_accept.argtypes = [ctypes.POINTER(Dims), vp, vp, vp, vp, vp, vp, vp, vp,
                                         vp, i32, vp, sz, vp]
    lib.dflash_verify_accept_noalloc.restype = ctypes.c_int
    lib.dflash_verify_accept_noalloc.argtypes = [ctypes.POINTER(Dims), vp, vp, vp, vp, vp, vp, vp,
                                                 vp, vp, i32, vp]
    lib.dflash_kv_crop.restype = ctypes.c_int
    lib.dflash_kv_crop.argtypes = [ctypes.POINTER(KVViewC), i32, vp, i32, vp, sz, vp]
    lib.dflash_read_status.restype = ctypes.c_int
    lib.dflash_read_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, vp]
    lib.dflash_status_string.restype = ctypes.c_char_p
    lib.dflash_status_string.argtypes = [ctypes.c_int]
    lib.dflash_version.restype = ctypes.c_int
    lib.dflash_version.argtypes = []
    lib.dflash_draft_workspace_bytes.restype = sz
    lib.dflash_draft_workspace_bytes.argtypes = [ctypes.POINTER(Dims), i32]
    lib.dflash_draft_qkv.restype = ctypes.c_int
    lib.dflash_draft_qkv.argtypes = [ctypes.POINTER(Dims)] + [vp] * 10 + [vp, sz, vp]
    lib.dflash_draft_mlp.restype = ctypes.c_int
    lib.dflash_draft_mlp.argtypes = [ctypes.POINTER(Dims), i32] + [vp] * 8 + [vp, sz, vp]
    lib.dflash_draft_tokens.restype = ctypes.c_int
    lib.dflash_draft_tokens.argtypes = [ctypes.POINTER(Dims)] + [vp] * 6 + [vp, sz, vp]
    lib.dflash_cycle_sm_split.restype = ctypes.c_int
    lib.dflash_cycle_sm_split.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(i32),
                                          ctypes.POINTER(i32)]
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().dflash_status_string(int(code)).decode()


def _check(rc: int, where: str):
    if rc != DFLASH_OK:
        raise DFlashError(rc, where)


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: Optional[torch.Tensor], dtype=None, name="tensor") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def make_dims(batch, hidden, n_q_heads, n_kv_heads, head_dim, vocab, n_ctx_layers, max_ctx,
              rope_theta=1.0e6, rms_eps=1.0e-6, block=16, sm_budget=0) -> Dims:
    return Dims(batch, block, hidden, n_q_heads, n_kv_heads, head_dim, vocab, n_ctx_layers,
                max_ctx, rope_theta, rms_eps, sm_budget)


def with_sm_budget(dims: Dims, sm_budget: int) -> Dims:
    """A copy of ``dims`` whose LM-head / projection grids use at most ``sm_budget`` SMs."""
    d = Dims.from_buffer_copy(dims)
    d.sm_budget = int(sm_budget)
    return d


def dflash_cycle_sm_split(dims: Dims):
    """(verify_sms, project_sms): SM budgets for running verify and the projection concurrently."""
    v, p = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(load_library().dflash_cycle_sm_split(ctypes.byref(dims), ctypes.byref(v),
                                                ctypes.byref(p)), "dflash_cycle_sm_split")
    return int(v.value), int(p.value)


@dataclass
class KVView:
    """A KV cache held in torch tensors (see dflash_kv_view in include/dflash.h)."""
    k: Optional[torch.Tensor]
    v: Optional[torch.Tensor]
    seq_len: torch.Tensor                      # int32 [B]
    capacity: int
    page_table: Optional[torch.Tensor] = None  # int32 [B, max_pages]
    free_list: Optional[torch.Tensor] = None   # int32 [n_pages]
    free_count: Optional[torch.Tensor] = None  # int32 [1]
    page_size: int = 16

    def c(self) -> KVViewC:
        paged = self.page_table is not None
        return KVViewC(
            _dev(self.k, torch.bfloat16, "k"), _dev(self.v, torch.bfloat16, "v"),
            _dev(self.seq_len, torch.int32, "seq_len"),
            _dev(self.page_table, torch.int32, "page_table"),
            _dev(self.free_list, torch.int32, "free_list"),
            _dev(self.free_count, torch.int32, "free_count"),
            int(self.capacity), int(self.page_size if paged else 0),
            int(self.page_table.shape[1]) if paged else 0,
            int(self.free_list.shape[0]) if paged else 0)


def dflash_workspace_bytes(dims: Dims) -> int:
    n = load_library().dflash_workspace_bytes(ctypes.byref(dims))
    if n == 0:
        raise DFlashError(-3, "dflash_workspace_bytes")
    return int(n)


def alloc_workspace(dims: Dims, device="cuda") -> torch.Tensor:
    """A zeroed workspace tensor of the size the library asks for."""
    return torch.zeros(dflash_workspace_bytes(dims), dtype=torch.uint8, device=device)


def dflash_workspace_init(ws: torch.Tensor, stream=None):
    _check(load_library().dflash_workspace_init(_dev(ws, name="ws"), ws.numel(), _stream(stream)),
           "dflash_workspace_init")


def dflash_ctx_project(dims: Dims, layer_hidden: Sequence[torch.Tensor], w_fc, hidden_norm_w,
                       w_k, w_v, k_norm_w, write_pos, cache: KVView, ws, stream=None):
    ptrs = (ctypes.c_void_p * len(layer_hidden))(
        *[_dev(h, torch.bfloat16, "layer_hidden") for h in layer_hidden])
    view = cache.c()
    _check(load_library().dflash_ctx_project(
        ctypes.byref(dims), ptrs, _dev(w_fc, torch.bfloat16, "w_fc"),
        _dev(hidden_norm_w, torch.bfloat16, "hidden_norm_w"), _dev(w_k, torch.bfloat16, "w_k"),
        _dev(w_v, torch.bfloat16, "w_v"), _dev(k_norm_w, torch.bfloat16, "k_norm_w"),
        _dev(write_pos, torch.int32, "write_pos"), ctypes.byref(view), _dev(ws, name="ws"),
        ws.numel(), _stream(stream)), "dflash_ctx_project")


def dflash_selftest_wait(arrive: bool, ws, stream=None):
    """One bounded wait: completed at once (arrive) or timed out after ~1 s (status bit)."""
    _check(load_library().dflash_selftest_wait(1 if arrive else 0, _dev(ws, name="ws"),
                                               ws.numel(), _stream(stream)),
           "dflash_selftest_wait")


def dflash_prefill_workspace_bytes(dims: Dims, tokens_per_seq: int) -> int:
    n = load_library().dflash_prefill_workspace_bytes(ctypes.byref(dims), int(tokens_per_seq))
    if n == 0:
        raise DFlashError(-3, "dflash_prefill_workspace_bytes")
    return int(n)


def alloc_prefill_workspace(dims: Dims, tokens_per_seq: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace for dflash_ctx_prefill with this many tokens per sequence."""
    return torch.zeros(dflash_prefill_workspace_bytes(dims, tokens_per_seq), dtype=torch.uint8,
                       device=device)


def dflash_ctx_prefill(dims: Dims, tokens_per_seq: int, layer_hidden: Sequence[torch.Tensor],
                       w_fc, hidden_norm_w, w_k, w_v, k_norm_w, write_pos, cache: KVView, ws,
                       stream=None):
    """Whole-prompt context projection: tokens_per_seq rows per sequence appended at write_pos."""
    ptrs = (ctypes.c_void_p * len(layer_hidden))(
        *[_dev(h, torch.bfloat16, "layer_hidden") for h in layer_hidden])
    view = cache.c()
    _check(load_library().dflash_ctx_prefill(
        ctypes.byref(dims), int(tokens_per_seq), ptrs, _dev(w_fc, torch.bfloat16, "w_fc"),
        _dev(hidden_norm_w, torch.bfloat16, "hidden_norm_w"), _dev(w_k, torch.bfloat16, "w_k"),
        _dev(w_v, torch.bfloat16, "w_v"), _dev(k_norm_w, torch.bfloat16, "k_norm_w"),
        _dev(write_pos, torch.int32, "write_pos"), ctypes.byref(view), _dev(ws, name="ws"),
        ws.numel(), _stream(stream)), "dflash_ctx_prefill")


def dflash_prefill_attention(dims: Dims, tokens_per_seq: int, q, k, v, cache: KVView,
                             scale: float, out, ws, stream=None):
    """The target's attention over a prompt chunk of tokens_per_seq rows per
    sequence (causal), the chunk's K/V appended to ``cache``."""
    view = cache.c()
    _check(load_library().dflash_prefill_attention(
        ctypes.byref(dims), int(tokens_per_seq), _dev(q, torch.bfloat16, "q"),
        _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"), ctypes.byref(view),
        float(scale), _dev(out, torch.bfloat16, "out"), _dev(ws, name="ws"), ws.numel(),
        _stream(stream)), "dflash_prefill_attention")


def dflash_prefill_staged(dims: Dims, last_hidden, w_lm, staged, ws, stream=None):
    """The first staged token per sequence: argmax of the LM head at the last
    prompt row.  ``last_hidden``: bf16 [B, H] whose rows may be strided (e.g.
    ``h[:, -1]`` of a [B, T, H] tensor); its row stride is passed on."""
    if not isinstance(last_hidden, torch.Tensor) or not last_hidden.is_cuda:
        raise ValueError("last_hidden must be a CUDA tensor")
    if last_hidden.dtype != torch.bfloat16 or last_hidden.dim() != 2 or last_hidden.stride(1) != 1:
        raise ValueError("last_hidden must be bf16 [B, H] with unit column stride")
    _check(load_library().dflash_prefill_staged(
        ctypes.byref(dims), last_hidden.data_ptr(), int(last_hidden.stride(0)),
        _dev(w_lm, torch.bfloat16, "w_lm"), _dev(staged, torch.int32, "staged"),
        _dev(ws, name="ws"), ws.numel(), _stream(stream)), "dflash_prefill_staged")


def dflash_block_attention(dims: Dims, q_blk, k_blk, v_blk, cache: KVView, scale: float, out,
                           ws, stream=None):
    view = cache.c()
    _check(load_library().dflash_block_attention(
        ctypes.byref(dims), _dev(q_blk, torch.bfloat16, "q_blk"),
        _dev(k_blk, torch.bfloat16, "k_blk"), _dev(v_blk, torch.bfloat16, "v_blk"),
        ctypes.byref(view), float(scale), _dev(out, torch.bfloat16, "out"), _dev(ws, name="ws"),
        ws.numel(), _stream(stream)), "dflash_block_attention")


def dflash_verify_attention(dims: Dims, q_blk, k_blk, v_blk, cache: KVView, scale: float, out,
                            ws, stream=None):
    """The target's verify attention: causal inside the block, block K/V appended to ``cache``."""
    view = cache.c()
    _check(load_library().dflash_verify_attention(
        ctypes.byref(dims), _dev(q_blk, torch.bfloat16, "q_blk"),
        _dev(k_blk, torch.bfloat16, "k_blk"), _dev(v_blk, torch.bfloat16, "v_blk"),
        ctypes.byref(view), float(scale), _dev(out, torch.bfloat16, "out"), _dev(ws, name="ws"),
        ws.numel(), _stream(stream)), "dflash_verify_attention")


def dflash_verify_accept(dims: Dims, hidden, w_lm, block_ids, len_before, posterior, accept_len,
                         next_staged, commit_len, out_tokens, ws, stream=None):
    _check(load_library().dflash_verify_accept(
        ctypes.byref(dims), _dev(hidden, torch.bfloat16, "hidden"),
        _dev(w_lm, torch.bfloat16, "w_lm"), _dev(block_ids, torch.int32, "block_ids"),
        _dev(len_before, torch.int32, "len_before"), _dev(posterior, torch.int32, "posterior"),
        _dev(accept_len, torch.int32, "accept_len"),
        _dev(next_staged, torch.int32, "next_staged"),
        _dev(commit_len, torch.int32, "commit_len"), _dev(out_tokens, torch.int32, "out_tokens"),
        int(out_tokens.shape[-1]), _dev(ws, name="ws"), ws.numel(), _stream(stream)),
        "dflash_verify_accept")


def dflash_verify_accept_noalloc(dims: Dims, hidden, w_lm, block_ids, len_before, posterior,
                                 accept_len, next_staged, commit_len, out_tokens, stream=None):
    """dflash_verify_accept without a workspace (library-owned static scratch)."""
    _check(load_library().dflash_verify_accept_noalloc(
        ctypes.byref(dims), _dev(hidden, torch.bfloat16, "hidden"),
        _dev(w_lm, torch.bfloat16, "w_lm"), _dev(block_ids, torch.int32, "block_ids"),
        _dev(len_before, torch.int32, "len_before"), _dev(posterior, torch.int32, "posterior"),
        _dev(accept_len, torch.int32, "accept_len"),
        _dev(next_staged, torch.int32, "next_staged"),
        _dev(commit_len, torch.int32, "commit_len"), _dev(out_tokens, torch.int32, "out_tokens"),
        int(out_tokens.shape[-1]), _stream(stream)), "dflash_verify_accept_noalloc")


def dflash_kv_crop(views: Sequence[KVView], new_len, batch: int, ws, stream=None):
    arr = (KVViewC * len(views))(*[v.c() for v in views])
    _check(load_library().dflash_kv_crop(arr, len(views), _dev(new_len, torch.int32, "new_len"),
                                         int(batch), _dev(ws, name="ws"), ws.numel(),
                                         _stream(stream)), "dflash_kv_crop")


def dflash_read_status(ws, clear: bool = True, stream=None) -> int:
    out = ctypes.c_uint32(0)
    _check(load_library().dflash_read_status(_dev(ws, name="ws"), ctypes.byref(out),
                                             1 if clear else 0, _stream(stream)),
           "dflash_read_status")
    return int(out.value)


def dflash_version() -> int:
    return int(load_library().dflash_version())


# ---------------------------------------------------------------------------
# the rest of one drafter layer and the drafter's tokens
# ---------------------------------------------------------------------------
def dflash_draft_workspace_bytes(dims: Dims, ffn: int) -> int:
    n = load_library().dflash_draft_workspace_bytes(ctypes.byref(dims), int(ffn))
    if n == 0:
        raise DFlashError(-3, "dflash_draft_workspace_bytes")
    return int(n)


def alloc_draft_workspace(dims: Dims, ffn: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace for the dflash_draft_* calls."""
    return torch.zeros(dflash_draft_workspace_bytes(dims, ffn), dtype=torch.uint8, device=device)


def dflash_draft_qkv(dims: Dims, x, ln1_w, w_q, w_k, w_v, q_norm_w, k_norm_w, q_out, k_out, v_out,
                     ws, stream=None):
    bf = torch.bfloat16
    _check(load_library().dflash_draft_qkv(
        ctypes.byref(dims), _dev(x, bf, "x"), _dev(ln1_w, bf, "ln1_w"), _dev(w_q, bf, "w_q"),
        _dev(w_k, bf, "w_k"), _dev(w_v, bf, "w_v"), _dev(q_norm_w, bf, "q_norm_w"),
        _dev(k_norm_w, bf, "k_norm_w"), _dev(q_out, bf, "q_out"), _dev(k_out, bf, "k_out"),
        _dev(v_out, bf, "v_out"), _dev(ws, name="ws"), ws.numel(), _stream(stream)),
        "dflash_draft_qkv")


def dflash_draft_mlp(dims: Dims, ffn: int, x, attn_out, w_o, ln2_w, w_gate, w_up, w_down, x_out,
                     ws, stream=None):
    bf = torch.bfloat16
    _check(load_library().dflash_draft_mlp(
        ctypes.byref(dims), int(ffn), _dev(x, bf, "x"), _dev(attn_out, bf, "attn_out"),
        _dev(w_o, bf, "w_o"), _dev(ln2_w, bf, "ln2_w"), _dev(w_gate, bf, "w_gate"),
        _dev(w_up, bf, "w_up"), _dev(w_down, bf, "w_down"), _dev(x_out, bf, "x_out"),
        _dev(ws, name="ws"), ws.numel(), _stream(stream)), "dflash_draft_mlp")


def dflash_draft_tokens(dims: Dims, x, final_norm_w, w_lm, staged, block_ids, posterior, ws,
                        stream=None):
    bf = torch.bfloat16
    _check(load_library().dflash_draft_tokens(
        ctypes.byref(dims), _dev(x, bf, "x"), _dev(final_norm_w, bf, "final_norm_w"),
        _dev(w_lm, bf, "w_lm"), _dev(staged, torch.int32, "staged"),
        _dev(block_ids, torch.int32, "block_ids"), _dev(posterior, torch.int32, "posterior"),
        _dev(ws, name="ws"), ws.numel(), _stream(stream)), "dflash_draft_tokens")


def dflash_gdn_replay(state, tape_k, tape_v, tape_beta, tape_g, accept_len, ws, stream=None):
    """Replay the committed 1 + a steps of the recorded tape onto ``state`` (in place)."""
    B, NH, Dv, Dk = state.shape
    _check(load_library().dflash_gdn_replay(
        int(B), int(NH), int(Dk), int(Dv), _dev(state, torch.float32, "state"),
        _dev(tape_k, torch.bfloat16, "tape_k"), _dev(tape_v, torch.bfloat16, "tape_v"),
        _dev(tape_beta, torch.float32, "tape_beta"), _dev(tape_g, torch.float32, "tape_g"),
        _dev(accept_len, torch.int32, "accept_len"), _dev(ws, name="ws"), ws.numel(),
        _stream(stream)), "dflash_gdn_replay")
