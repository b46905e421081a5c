"""One draft/verify cycle as a sequence of the four ABI calls.

"dflash-mlx" (dpshk.com) 单次前向验证 ⑤–⑨ and "DFlash双实现对比"
(hotelren.com) §2–§4: verify the block (LM head + greedy argmax +
acceptance + commit), project the block's target hidden states into the
drafter's context K/V, crop the target and drafter caches to the committed
length, then run the drafter's dual-source block attention for the next
block.  This module only holds device buffers and issues the calls; every
step runs in the CUDA library.

Verification and the projection do not depend on each other (the projection
reads the target's hidden states and the drafter's write position, not the
acceptance), so by default they run side by side: verify on the caller's
stream, the projection on a side stream, each on its own share of the SMs
(``dflash_cycle_sm_split``), joined before the crop.  The crop then runs on
the side stream beside the attention, which takes the drafter context's new
length from the commit length rather than waiting for the crop to write it.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass
from typing import List, Optional, Tuple

import torch

from .dflash import (Dims, KVView, dflash_block_attention, dflash_ctx_project,
                     dflash_cycle_sm_split, dflash_kv_crop, dflash_verify_accept, with_sm_budget)

_side_streams = {}


def side_stream(device) -> torch.cuda.Stream:
    """The side stream (one per device) that carries the projection."""
    idx = torch.device(device).index
    if idx is None:
        idx = torch.cuda.current_device()
    if idx not in _side_streams:
        _side_streams[idx] = torch.cuda.Stream(device=idx)
    return _side_streams[idx]


@dataclass
class CycleWeights:
    w_lm: torch.Tensor               # bf16 [V, H]
    w_fc: torch.Tensor               # bf16 [H, nL*H]
    hidden_norm_w: Optional[torch.Tensor]  # bf16 [H]
    w_k: torch.Tensor                # bf16 [Hkv*D, H]
    w_v: torch.Tensor                # bf16 [Hkv*D, H]
    k_norm_w: Optional[torch.Tensor]  # bf16 [D]


@dataclass
class CycleState:
    """Inputs, outputs and caches of one cycle for a batch of sequences."""
    layer_hidden: List[torch.Tensor]  # nL x bf16 [B*16, H]  (selected target layers)
    verify_hidden: torch.Tensor       # bf16 [B*16, H]        (final-normed target hidden)
    block_ids: torch.Tensor           # int32 [B, 16]
    len_before: torch.Tensor          # int32 [B] committed length before the cycle
    write_pos: torch.Tensor           # int32 [B] first context row of the block
    q_blk: torch.Tensor               # bf16 [B, 16, Hq, D]   (next block, pre-RoPE)
    k_blk: torch.Tensor               # bf16 [B, 16, Hkv, D]
    v_blk: torch.Tensor               # bf16 [B, 16, Hkv, D]
    draft_cache: KVView
    target_view: KVView
    posterior: torch.Tensor           # int32 [B, 16]
    accept_len: torch.Tensor          # int32 [B]
    next_staged: torch.Tensor         # int32 [B]
    commit_len: torch.Tensor          # int32 [B]
    out_tokens: torch.Tensor          # int32 [B, out_cap]
    attn_out: torch.Tensor            # bf16 [B, 16, Hq, D]


def _verify_and_project(dims_v: Dims, dims_p: Dims, w: CycleWeights, st: CycleState,
                        ws: torch.Tensor, main, side):
    """verify on ``main`` and the projection on ``side``, forked from and joined
    back into ``main``."""
    fork = torch.cuda.Event()
    fork.record(main)
    side.wait_event(fork)
    dflash_verify_accept(dims_v, st.verify_hidden, w.w_lm, st.block_ids, st.len_before,
                         st.posterior, st.accept_len, st.next_staged, st.commit_len,
                         st.out_tokens, ws, main)
    dflash_ctx_project(dims_p, st.layer_hidden, w.w_fc, w.hidden_norm_w, w.w_k, w.w_v,
                       w.k_norm_w, st.write_pos, st.draft_cache, ws, side)
    join = torch.cuda.Event()
    join.record(side)
    main.wait_event(join)


def tune_sm_split(dims: Dims, w: CycleWeights, states: List[CycleState], ws: torch.Tensor,
                  spread: Optional[int] = None, reps: int = 8,
                  rounds: int = 2) -> Tuple[int, int]:
    """Measure the verify || projection phase for SM splits around
    ``dflash_cycle_sm_split`` and return the fastest (verify_sms, project_sms).

    The proportional split is only a first guess: the two kernels' per-SM
    bandwidth shares and tile boundaries move the optimum by a few SMs (by
    more past 256 token rows, where both sides are bound by the tensor cores
    and run as tiled GEMMs: the default spread is then 8 SMs instead of 4).
    Runs ``rounds * (2 * spread + 1) * reps`` phases on the given states
    (their outputs are overwritten; lengths written by the projection are
    restored).
    """
    if spread is None:
        spread = 8 if dims.batch * dims.block > 256 else 4
    v0, p0 = dflash_cycle_sm_split(dims)
    nsm = v0 + p0
    main = torch.cuda.current_stream()
    side = side_stream(states[0].verify_hidden.device)
    saved = [s.draft_cache.seq_len.clone() for s in states]
    best = {}
    for _ in range(rounds):
        for p in range(max(1, p0 - spread), min(nsm - 1, p0 + spread) + 1):
            dv, dp = with_sm_budget(dims, nsm - p), with_sm_budget(dims, p)
            _verify_and_project(dv, dp, w, states[0], ws, main, side)   # warm
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(main)
            for i in range(reps):
                _verify_and_project(dv, dp, w, states[i % len(states)], ws, main, side)
            e1.record(main)
            e1.synchronize()
            t = e0.elapsed_time(e1) / reps
            best[p] = min(best.get(p, t), t)
    for s, L in zip(states, saved):
        s.draft_cache.seq_len.copy_(L)
    torch.cuda.synchronize()
    p = min(best, key=best.get)
    return nsm - p, p


def run_cycle(dims: Dims, w: CycleWeights, st: CycleState, ws: torch.Tensor,
              scale: Optional[float] = None, stream=None, concurrent: bool = True,
              sm_split: Optional[Tuple[int, int]] = None):
    """Issue one cycle on the current (or given) stream.

    With ``concurrent`` the verification and the projection run on disjoint
    SM budgets on two streams (``sm_split`` = (verify_sms, project_sms), by
    default ``dflash_cycle_sm_split``); otherwise all four calls queue on one
    stream.
    """
    if scale is None:
        scale = 1.0 / math.sqrt(dims.head_dim)
    main = torch.cuda.current_stream() if stream is None else stream
    if concurrent:
        verify_sms, project_sms = sm_split or dflash_cycle_sm_split(dims)
        side = side_stream(st.verify_hidden.device)
        _verify_and_project(with_sm_budget(dims, verify_sms), with_sm_budget(dims, project_sms),
                            w, st, ws, main, side)
        _crop_beside_attention(dims, st, ws, scale, main, side)
        return
    dflash_verify_accept(dims, st.verify_hidden, w.w_lm, st.block_ids, st.len_before,
                         st.posterior, st.accept_len, st.next_staged, st.commit_len,
                         st.out_tokens, ws, main)
    dflash_ctx_project(dims, st.layer_hidden, w.w_fc, w.hidden_norm_w, w.w_k, w.w_v,
                       w.k_norm_w, st.write_pos, st.draft_cache, ws, main)
    dflash_kv_crop([st.target_view, st.draft_cache], st.commit_len, dims.batch, ws, main)
    dflash_block_attention(dims, st.q_blk, st.k_blk, st.v_blk, st.draft_cache, scale,
                           st.attn_out, ws, main)


def _crop_beside_attention(dims: Dims, st: CycleState, ws: torch.Tensor, scale: float, main,
                           side):
    """The crop on ``side`` while the attention runs on ``main``, joined back.

    The crop sets the drafter context's length to the commit length; the
    attention reads that length from ``commit_len`` itself, so it need not
    wait for the crop.  The crop releases only pages at or past the new
    length, which the attention never reads, and it touches only the status
    word of the workspace.  The join keeps the next cycle (whose verification
    rewrites ``commit_len``) behind the crop."""
    fork = torch.cuda.Event()
    fork.record(main)
    side.wait_event(fork)
    dflash_kv_crop([st.target_view, st.draft_cache], st.commit_len, dims.batch, ws, side)
    dflash_block_attention(dims, st.q_blk, st.k_blk, st.v_blk,
                           dataclasses.replace(st.draft_cache, seq_len=st.commit_len), scale,
                           st.attn_out, ws, main)
    join = torch.cuda.Event()
    join.record(side)
    main.wait_event(join)


def packed_tensors(specs, device, pin: bool = False):
    """One flat buffer and views into it, one per (shape, dtype) in ``specs``
    (each view 256-byte aligned), so that a whole set of a step's inputs or
    outputs moves between host and device as a single copy."""
    offs, off = [], 0
    for shape, dtype in specs:
        off = (off + 255) // 256 * 256
        offs.append(off)
        n = 1
        for x in shape:
            n *= int(x)
        off += n * torch.empty((), dtype=dtype).element_size()
    flat = torch.empty(off, dtype=torch.uint8, device=device)
    if pin:
        flat = flat.pin_memory()
    views = []
    for (shape, dtype), o in zip(specs, offs):
        n = 1
        for x in shape:
            n *= int(x)
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        views.append(flat[o:o + nbytes].view(dtype).view(*shape))
    return flat, views


class CycleGraph:
    """One whole cycle -- the host-to-device copy of the step's inputs, the
    four calls, the device-to-host copy of its results -- captured once as a
    CUDA graph and replayed per step, so that the per-step host work is one
    graph launch (the serving loop of a fixed-shape batch).

    ``inputs``: (pinned host tensor, device tensor) pairs copied in every step;
    ``outputs``: (device tensor, pinned host tensor) pairs copied out.  The
    other arguments are those of :func:`run_cycle`.  Capturing runs the cycle
    once beforehand (outside the graph) to settle every lazy setup."""

    def __init__(self, dims: Dims, w: CycleWeights, st: CycleState, ws: torch.Tensor,
                 inputs, outputs, scale: Optional[float] = None, concurrent: bool = True,
                 sm_split: Optional[Tuple[int, int]] = None):
        self._args = (dims, w, st, ws, scale, concurrent, sm_split)
        self.inputs = list(inputs)
        self.outputs = list(outputs)
        warm = torch.cuda.Stream()
        warm.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(warm):
            self._body()
        torch.cuda.current_stream().wait_stream(warm)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._body()
        torch.cuda.synchronize()

    def _body(self):
        dims, w, st, ws, scale, concurrent, sm_split = self._args
        for h, d in self.inputs:
            d.copy_(h, non_blocking=True)
        run_cycle(dims, w, st, ws, scale, concurrent=concurrent, sm_split=sm_split)
        for d, h in self.outputs:
            h.copy_(d, non_blocking=True)

    def replay(self):
        """Launch one cycle on the current stream (asynchronous)."""
        self.graph.replay()


class PipelinedCycles:
    """The serving loop of a fixed-shape batch with the host-to-device copy of
    step k + 1's inputs overlapping step k's cycle.

    Two :class:`CycleGraph` s run over two device copies of the step inputs;
    the cache state and the results are shared by both, so consecutive steps
    still chain on the device.  A side stream copies the next step's inputs
    into the free copy while the current step runs, and at most two steps are
    in flight: :meth:`step` returns once the previous step's results have
    reached the host.

    ``states``: two CycleStates that differ only in their input tensors, which
    are views of ``dev_in[0]`` and ``dev_in[1]`` (one packed device buffer per
    slot, filled by one copy).  ``outputs``: (device tensor, (host tensor for
    slot 0, host tensor for slot 1)) pairs of pinned host destinations.
    Building the object runs the cycle twice (each graph's warm-up)."""

    def __init__(self, dims: Dims, w: CycleWeights, states, ws: torch.Tensor, dev_in, outputs,
                 scale: Optional[float] = None, concurrent: bool = True,
                 sm_split: Optional[Tuple[int, int]] = None):
        if len(states) != 2 or len(dev_in) != 2:
            raise ValueError("two slots of states and device inputs are needed")
        self.dev_in = list(dev_in)
        self.graphs = [CycleGraph(dims, w, st, ws, [], [(d, hs[s]) for d, hs in outputs], scale,
                                  concurrent, sm_split)
                       for s, st in enumerate(states)]
        self.copy_stream = torch.cuda.Stream()
        self.copied = [torch.cuda.Event(), torch.cuda.Event()]
        self.done = [torch.cuda.Event(), torch.cuda.Event()]
        self.k = 0

    def step(self, host_in: torch.Tensor) -> Optional[int]:
        """Queue one step whose inputs are the pinned host buffer ``host_in``
        (the layout of ``dev_in``; it must stay unchanged until the next call
        returns).  Returns the slot whose host outputs now hold the previous
        step's results (None on the first step)."""
        s = self.k & 1
        main = torch.cuda.current_stream()
        with torch.cuda.stream(self.copy_stream):
            if self.k >= 2:
                self.copy_stream.wait_event(self.done[s])   # step k-2 is done with this slot
            self.dev_in[s].copy_(host_in, non_blocking=True)
            self.copied[s].record(self.copy_stream)
        main.wait_event(self.copied[s])
        self.graphs[s].replay()
        self.done[s].record(main)
        prev = None
        if self.k >= 1:
            self.done[s ^ 1].synchronize()
            prev = s ^ 1
        self.k += 1
        return prev

    def finish(self) -> Optional[int]:
        """Wait for the last step queued; returns the slot holding its results."""
        if self.k == 0:
            return None
        s = (self.k - 1) & 1
        self.done[s].synchronize()
        return s
