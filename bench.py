#!/usr/bin/env python
"""Benchmark of the DFlash per-cycle hot path on GB300.

Metric: draft+verify cycles/s at Qwen3-8B shapes, block 16, and the fraction
of the HBM roofline.  One step = one whole cycle (dflash_verify_accept,
dflash_ctx_project, dflash_kv_crop over the target and drafter views,
dflash_block_attention) over one batch of synthetic inputs already resident
in HBM.  Every step replays the same cycle from the same state: the block is
written at a fixed context position, the crop trims it to the committed
length and the attention of the next block reads that length.  Verification
and the projection run side by side on two streams, each on its own share of
the SMs (the split is measured once before the warm-up; --sm-split fixes it,
--serial queues everything on one stream); the crop then runs on the side
stream beside the attention, which reads the committed length directly.
Beside `value` (calls issued step by step) the line reports the same cycle
replayed from CUDA graphs (`graph_replay`), and the same workload with its
draft match lengths drawn truncated-geometric with mean 13 instead of
uniform in 0..15 (`geometric_draw`).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
N > 1 runs under torchrun: every rank runs an independent replica (sequences
are independent; no collective on the data path) and rank 0 prints one JSON
line with the whole-job throughput over the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft+verify cycles/s at Qwen3-8B shapes, block 16; % of HBM roofline"
from synthetic import CONFIG_BY_NAME  # noqa: E402  (input generators only; no arithmetic)
UNIT = "cycles/s"
DEFAULT_CONFIG = "qwen3_8b_b1"
L2_BYTES = 129 * 1024 * 1024
PEAK_FALLBACK_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--breakdown-steps", type=int, default=100,
                    help="extra steps after the timed region with events around every call")
    ap.add_argument("--sets", type=int, default=0,
                    help="rotating input sets (0: enough to exceed twice the L2 size)")
    ap.add_argument("--prefill-tokens", type=int, default=8192,
                    help="prompt length of the prefill passes (0 = skip)")
    ap.add_argument("--prefill-chunk", type=int, default=2048,
                    help="prompt chunk of the prefill-attention pass")
    ap.add_argument("--alt-draw-steps", type=int, default=400,
                    help="timed cycles of the headline workload with the draft match lengths "
                         "drawn truncated-geometric with mean 13 (reported beside the "
                         "uniform headline; 0 = skip)")
    ap.add_argument("--b32-steps", type=int, default=50,
                    help="timed cycles of the batch-32 paged workload reported beside the "
                         "headline (0 = skip)")
    ap.add_argument("--draft-steps", type=int, default=100,
                    help="extra steps timing the rest of the drafter layer (Q/K/V, attention, "
                         "output projection + MLP, tokens), reported beside the cycle")
    ap.add_argument("--graph-replays", type=int, default=200,
                    help="cycles per rep of the graph-replay pass (5 reps; 0 = skip)")
    ap.add_argument("--sm-split", default="",
                    help="verify_sms,project_sms for the side-by-side phase (default: measured "
                         "around the proportional split before the warm-up)")
    ap.add_argument("--serial", action="store_true",
                    help="queue verify and the projection on one stream instead of running "
                         "them side by side on disjoint SM budgets")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# distributed plumbing (host logic; also exercised with gloo on CPU)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(backend: str):
    import torch.distributed as dist
    world, rank, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return world, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank: float, n_ranks: int, max_seconds: float) -> float:
    """Units processed by all ranks divided by the slowest rank's time."""
    return units_per_rank * n_ranks / max_seconds


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


PEAK_FALLBACK_TFLOPS = 1900.0


def measured_peak_tflops():
    """Dense bf16 tensor peak (burst) from MEASURED_PEAKS.json, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            if isinstance(d.get("bf16_tflops"), (int, float)):
                return float(d["bf16_tflops"]), "measured"
        except (OSError, ValueError):
            pass
    return PEAK_FALLBACK_TFLOPS, "fallback"


def measured_peak_gbs():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBs", "hbm"):
                if k in d and isinstance(d[k], (int, float)):
                    return float(d[k]), "measured"
        except (OSError, ValueError):
            pass
    return PEAK_FALLBACK_GBS, "fallback"


def profiled_traffic(profile_name: str, kernel: str = ""):
    """DRAM bytes per launch (read + write) and the algorithmic bytes per launch
    from a committed ncu summary under profiles/, while every source file it
    lists (`source_sha256: path=sha16 ...`, paths relative to the package)
    still has the SHA-256 it was captured on; else None.  `kernel` selects a
    `traffic_bytes_per_launch[kernel]` entry of a summary with several."""
    import hashlib
    p = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p, encoding="utf-8"):
        s = line.strip()
        if ":" in s and s.startswith(("source_sha256", "traffic_bytes_per_launch",
                                      "algorithmic_bytes_per_launch")):
            k, v = s.split(":", 1)
            vals[k.strip()] = v.strip()
    pairs = [x.split("=", 1) for x in vals.get("source_sha256", "").split()]
    if not pairs or any(len(x) != 2 for x in pairs):
        return None
    pkg = os.path.join(ROOT, "block_diffusion_speculative_02_gb300")
    for rel, sha in pairs:
        f = os.path.join(pkg, rel)
        if not os.path.exists(f) or hashlib.sha256(open(f, "rb").read()).hexdigest()[:16] != sha:
            return None
    tag = f"[{kernel}]" if kernel else ""
    t, a = vals.get("traffic_bytes_per_launch" + tag), vals.get("algorithmic_bytes_per_launch" + tag)
    if t is None or a is None:
        return None
    return {"traffic": float(t), "algorithmic": float(a), "ratio": float(t) / float(a),
            "profile": "profiles/" + profile_name}


def traffic_check():
    """DRAM traffic / algorithmic bytes per launch of the four kernels of the
    Qwen3-8B batch-1 cycle, from the committed ncu summaries (None where the
    kernel's sources changed since the capture)."""
    return {"lmhead_argmax_accept": profiled_traffic("lmhead_argmax_accept_qwen3_8b_b1.md"),
            "block_attention": profiled_traffic("block_attention_qwen3_8b_b1.md"),
            "streamk_gemm_fc": profiled_traffic("streamk_gemm_qwen3_8b_b1.md", "FcFin"),
            "streamk_gemm_kv": profiled_traffic("streamk_gemm_qwen3_8b_b1.md", "KvFin"),
            "note": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch (cold, "
                    "alone) over the algorithmic bytes of that launch; 1.0 = every byte once"}


# ---------------------------------------------------------------------------
# the workload on the GPU
# ---------------------------------------------------------------------------
def build_workload(cfg, n_sets: int, device="cuda"):
    import numpy as np
    import torch

    import block_diffusion_speculative_02_gb300 as dfl
    from block_diffusion_speculative_02_gb300.cycle import CycleState, CycleWeights
    from synthetic import (device_generator, device_normal_bf16, device_unit_rms_rows_bf16,
                           draw_accept_lengths, make_block_ids, make_paged_layout, streams_for)

    B, H, V = cfg.batch, cfg.hidden, cfg.vocab
    Hq, Hkv, D, nL = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.n_ctx_layers
    gen = {n: device_generator(cfg, n, device) for n in
           ("w_lm", "w_fc", "hidden_norm_w", "w_k", "w_v", "k_norm_w", "layer_hidden",
            "verify_hidden", "ctx_k", "ctx_v", "q_blk", "k_blk", "v_blk")}
    w = CycleWeights(
        w_lm=device_normal_bf16(gen["w_lm"], (V, H), 0.02, device=device),
        w_fc=device_normal_bf16(gen["w_fc"], (H, nL * H), 0.02, device=device),
        hidden_norm_w=device_normal_bf16(gen["hidden_norm_w"], (H,), 0.02, 1.0, device=device),
        w_k=device_normal_bf16(gen["w_k"], (Hkv * D, H), 0.02, device=device),
        w_v=device_normal_bf16(gen["w_v"], (Hkv * D, H), 0.02, device=device),
        k_norm_w=device_normal_bf16(gen["k_norm_w"], (D,), 0.02, 1.0, device=device))
    host = streams_for(cfg)
    if cfg.ctx_len_range is not None:
        lo, hi = cfg.ctx_len_range
        lens = host["ctx_lens"].integers(lo, hi + 1, size=B).astype(np.int32)
    else:
        lens = np.full(B, cfg.ctx_len, np.int32)
    max_ctx = int(lens.max()) + 16
    dims = dfl.make_dims(B, H, Hq, Hkv, D, V, nL, max_ctx, cfg.rope_theta, cfg.rms_eps)
    ws = dfl.alloc_workspace(dims, device)
    out_cap = max_ctx + 16
    states, accepts = [], []
    for r in range(n_sets):
        i32 = lambda a: torch.as_tensor(np.asarray(a, np.int32), device=device)  # noqa: E731
        if cfg.paged:
            # room for the cycle's 16 projected rows and, on top of the
            # committed length, the 16 rows the verify-attention pass appends
            lay = make_paged_layout(host["pages"], lens, reserve_tokens=32, slack_pages=64)
            n_rows = lay.n_pages * 16
            k = device_normal_bf16(gen["ctx_k"], (lay.n_pages, Hkv, 16, D), device=device)
            v = device_normal_bf16(gen["ctx_v"], (lay.n_pages, Hkv, 16, D), device=device)
            draft = dfl.KVView(k, v, i32(lens), capacity=lay.max_pages * 16,
                               page_table=i32(lay.page_table), free_list=i32(lay.free_list),
                               free_count=i32([lay.free_count]), page_size=16)
            tlay = make_paged_layout(host["pages"], lens + 16, reserve_tokens=16, slack_pages=64)
            target = dfl.KVView(None, None, i32(lens + 16), capacity=tlay.max_pages * 16,
                                page_table=i32(tlay.page_table), free_list=i32(tlay.free_list),
                                free_count=i32([tlay.free_count]), page_size=16)
            del n_rows
        else:
            cap = max_ctx + 16
            k = device_normal_bf16(gen["ctx_k"], (B, Hkv, cap, D), device=device)
            v = device_normal_bf16(gen["ctx_v"], (B, Hkv, cap, D), device=device)
            draft = dfl.KVView(k, v, i32(lens), capacity=cap)
            target = dfl.KVView(None, None, i32(lens + 16), capacity=cap)
        st = CycleState(
            layer_hidden=[device_unit_rms_rows_bf16(gen["layer_hidden"], (B * 16, H), device)
                          for _ in range(nL)],
            verify_hidden=device_unit_rms_rows_bf16(gen["verify_hidden"], (B * 16, H), device),
            block_ids=torch.zeros((B, 16), dtype=torch.int32, device=device),
            len_before=i32(lens), write_pos=i32(lens),
            q_blk=device_normal_bf16(gen["q_blk"], (B, 16, Hq, D), device=device),
            k_blk=device_normal_bf16(gen["k_blk"], (B, 16, Hkv, D), device=device),
            v_blk=device_normal_bf16(gen["v_blk"], (B, 16, Hkv, D), device=device),
            draft_cache=draft, target_view=target,
            posterior=torch.zeros((B, 16), dtype=torch.int32, device=device),
            accept_len=torch.zeros(B, dtype=torch.int32, device=device),
            next_staged=torch.zeros(B, dtype=torch.int32, device=device),
            commit_len=torch.zeros(B, dtype=torch.int32, device=device),
            out_tokens=torch.zeros((B, out_cap), dtype=torch.int32, device=device),
            attn_out=torch.zeros((B, 16, Hq, D), dtype=torch.bfloat16, device=device))
        # plant the drafts: the target's own posterior for the first a positions
        dfl.dflash_verify_accept(dims, st.verify_hidden, w.w_lm, st.block_ids, st.len_before,
                                 st.posterior, st.accept_len, st.next_staged, st.commit_len,
                                 st.out_tokens, ws)
        a = draw_accept_lengths(host["accept"], cfg.accept, B)
        blk = make_block_ids(host["blocks"], st.posterior.cpu().numpy(), a, V)
        st.block_ids.copy_(torch.as_tensor(blk, device=device))
        states.append(st)
        accepts.append(a)
    torch.cuda.synchronize()
    return dims, w, states, accepts, ws, lens


def lm_head_roofline(cfg, lm_bytes: int, lm_ms: float, hbm_peak, tensor_peak, traffic) -> dict:
    """The `roofline` entry for the LM-head launch: bound by the larger of its
    weight-stream time (bytes / HBM peak) and its tensor time (2 B 16 H V
    flops / bf16 peak) -- HBM at small batch, the tensor cores at batch 32 --
    with both fractions reported.  Peaks are (value, kind) pairs in GB/s and
    TFLOP/s; lm_ms is the mean launch duration in milliseconds."""
    peak, peak_kind = hbm_peak
    tpk, tpk_kind = tensor_peak
    lm_flops = 2.0 * cfg.batch * 16 * cfg.hidden * cfg.vocab
    lm_gbs = lm_bytes / (lm_ms / 1e3) / 1e9
    lm_tflops = lm_flops / (lm_ms / 1e3) / 1e12
    tensor_bound = lm_flops / (tpk * 1e12) > lm_bytes / (peak * 1e9)
    return {"bound": "tensor" if tensor_bound else "hbm", "kernel": "lmhead_argmax_accept",
            "achieved": lm_tflops if tensor_bound else lm_gbs,
            "peak": tpk if tensor_bound else peak,
            "peak_kind": tpk_kind if tensor_bound else peak_kind,
            "unit": "TFLOP/s" if tensor_bound else "GB/s",
            "frac": lm_tflops / tpk if tensor_bound else lm_gbs / peak,
            "traffic": traffic, "bytes_per_launch": lm_bytes, "flops_per_launch": lm_flops,
            "avg_launch_ms": lm_ms, "hbm_frac": lm_gbs / peak, "tensor_frac": lm_tflops / tpk}


def algorithmic_bytes(cfg, lens) -> dict:
    """Bytes one cycle must move at least: every weight once, the context KV of
    one drafter layer once, activations once."""
    B, H, V = cfg.batch, cfg.hidden, cfg.vocab
    Hq, Hkv, D, nL = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.n_ctx_layers
    T = 16
    lm = V * H * 2 + B * T * H * 2 + B * T * 4 * 4
    fc = H * nL * H * 2 + nL * B * T * H * 2
    kv = 2 * Hkv * D * H * 2 + 2 * B * T * Hkv * D * 2
    ctx_len_after = sum(int(L) + 1 for L in lens)  # attention reads L + 1 + a rows; a >= 0
    attn = 2 * Hkv * D * 2 * ctx_len_after + B * T * (Hq + 2 * Hkv) * D * 2 + B * T * Hq * D * 2
    return {"lm_head": lm, "ctx_project": fc + kv, "attention": attn,
            "total": lm + fc + kv + attn}


def draft_bytes(cfg) -> int:
    """Bytes one drafter layer plus its token choice must move at least: its
    weights and the LM head once, activations once (the attention's context
    KV is counted with the cycle)."""
    B, H, V, F = cfg.batch, cfg.hidden, cfg.vocab, cfg.ffn
    qd, kvd = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    T = 16
    weights = (qd + 2 * kvd) * H * 2 + H * qd * 2 + 3 * F * H * 2 + V * H * 2
    acts = B * T * (2 * H + qd + 2 * kvd + qd + H) * 2
    return weights + acts


def build_draft(cfg, device="cuda"):
    """Drafter-layer weights and activations of the workload's shapes (seeded)."""
    import torch

    from synthetic import device_generator, device_normal_bf16, device_unit_rms_rows_bf16
    B, H, F = cfg.batch, cfg.hidden, cfg.ffn
    qd, kvd = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    gw = device_generator(cfg, "draft_w", device)
    gx = device_generator(cfg, "draft_x", device)
    n = lambda shape, std=0.02, mean=0.0: device_normal_bf16(gw, shape, std, mean, device)  # noqa
    w = {"ln1": n((H,), 0.02, 1.0), "wq": n((qd, H)), "wk": n((kvd, H)), "wv": n((kvd, H)),
         "qn": n((cfg.head_dim,), 0.02, 1.0), "kn": n((cfg.head_dim,), 0.02, 1.0),
         "wo": n((H, qd)), "ln2": n((H,), 0.02, 1.0), "wg": n((F, H)), "wu": n((F, H)),
         "wd": n((H, F)), "fn": n((H,), 0.02, 1.0)}
    x = device_unit_rms_rows_bf16(gx, (B * 16, H), device)
    bufs = {"q": torch.empty((B * 16, qd), dtype=torch.bfloat16, device=device),
            "k": torch.empty((B * 16, kvd), dtype=torch.bfloat16, device=device),
            "v": torch.empty((B * 16, kvd), dtype=torch.bfloat16, device=device),
            "o": torch.empty((B, 16, cfg.n_q_heads, cfg.head_dim), dtype=torch.bfloat16,
                             device=device),
            "x_out": torch.empty((B * 16, H), dtype=torch.bfloat16, device=device),
            "block": torch.zeros((B, 16), dtype=torch.int32, device=device)}
    return w, x, bufs


# ---------------------------------------------------------------------------
# CPU oracle timing (bounded sample)
# ---------------------------------------------------------------------------
def oracle_inputs(cfg, frac: float = 1.0) -> dict:
    """Seeded inputs of the oracle's cycle (bf16 bit patterns), the whole
    workload when frac == 1, else a row sample: frac of the LM head's
    vocabulary rows and of the projection's output features, one KV head of
    the attention.  Weights are drawn with a seeded CPU torch generator (the
    same distributions as the GPU workload)."""
    import numpy as np
    import torch

    from synthetic import device_generator, device_normal_bf16, normal_bf16, unit_rms_rows_bf16

    def bits(t):
        return t.view(torch.int16).numpy().view(np.uint16)

    rng = np.random.default_rng(7)
    B, H, V = cfg.batch, cfg.hidden, cfg.vocab
    Hq, Hkv, D, nL = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.n_ctx_layers
    L = int(cfg.ctx_len or cfg.ctx_len_range[1])
    full = frac >= 1.0
    nv = V if full else max(64, int(V * frac))
    nf = H if full else max(D, int(H * frac) // D * D)
    hk = Hkv if full else 1
    g = device_generator(cfg, "w_lm", "cpu")
    inp = {
        "frac": frac, "nv": nv, "nf": nf, "hk": hk, "L": L,
        "hidden": unit_rms_rows_bf16(rng, (B, 16, H)),
        "w_lm": bits(device_normal_bf16(g, (nv, H), 0.02, device="cpu")),
        "layers": [unit_rms_rows_bf16(rng, (B * 16, H)) for _ in range(nL)],
        "w_fc": bits(device_normal_bf16(g, (nf, nL * H), 0.02, device="cpu")),
        "gh": normal_bf16(rng, (nf,), 0.02, 1.0),
        "wk": normal_bf16(rng, (hk * D, nf), 0.02), "wv": normal_bf16(rng, (hk * D, nf), 0.02),
        "gk": normal_bf16(rng, (D,), 0.02, 1.0),
        "q": normal_bf16(rng, (B, 16, hk * (Hq // Hkv), D)),
        "kb": normal_bf16(rng, (B, 16, hk, D)), "vb": normal_bf16(rng, (B, 16, hk, D)),
        "ck": [normal_bf16(rng, (L, hk, D)) for _ in range(B)],
        "cv": [normal_bf16(rng, (L, hk, D)) for _ in range(B)]}
    return inp


def oracle_cycle_seconds(cfg, inp: dict) -> dict:
    """Time the float64 oracle's four steps on `inp` (oracle_inputs).  On the
    whole workload (frac 1) the times are the cycle's own; on a row sample
    each step's time is scaled by the inverse of its sampled fraction (the
    steps are linear in the sampled rows and heads), and the result says it
    is extrapolated."""
    import numpy as np

    from oracle.dflash_oracle import block_attention, ctx_project, kv_crop_lengths, verify_accept

    B, H, V, D = cfg.batch, cfg.hidden, cfg.vocab, cfg.head_dim
    Hkv, L = cfg.n_kv_heads, inp["L"]
    nv, nf, hk = inp["nv"], inp["nf"], inp["hk"]
    blk = np.zeros((B, 16), np.int32)
    t = {}
    t0 = time.perf_counter()
    verify_accept(inp["hidden"], inp["w_lm"], blk, np.zeros(B, np.int32), out_cap=32)
    t["lm_head"] = (time.perf_counter() - t0) * (V / nv)
    t0 = time.perf_counter()
    ctx_project(inp["layers"], inp["w_fc"], inp["gh"], inp["wk"], inp["wv"], inp["gk"],
                np.arange(B * 16) + L, hk, D, cfg.rope_theta, cfg.rms_eps)
    t["ctx_project"] = (time.perf_counter() - t0) * (H / nf)
    t0 = time.perf_counter()
    block_attention(inp["q"], inp["kb"], inp["vb"], inp["ck"], inp["cv"], np.full(B, L),
                    cfg.rope_theta, 1 / math.sqrt(D))
    t["attention"] = (time.perf_counter() - t0) * (Hkv / hk)
    t0 = time.perf_counter()
    kv_crop_lengths(np.full(B, L + 16), np.full(B, L + 9))
    kv_crop_lengths(np.full(B, L + 16), np.full(B, L + 9))
    t["crop"] = time.perf_counter() - t0
    t["total"] = sum(t.values())
    t["extrapolated"] = nv < V or nf < H or hk < Hkv
    if t["extrapolated"]:
        t["sample"] = (f"extrapolated linearly from a row sample: LM head over {nv}/{V} vocab "
                       f"rows (x{V / nv:.1f}); projection over {nf}/{H} output features "
                       f"(x{H / nf:.1f}); attention of {hk}/{Hkv} KV heads (x{Hkv / hk:.0f}) "
                       f"at context {L}; crop in full; batch {B}")
    else:
        t["sample"] = (f"the whole cycle, no sampling: LM head over all {V} vocab rows, "
                       f"projection of all {H} features, attention of all {Hkv} KV heads at "
                       f"context {L}, crop; batch {B}")
    return t


def host_threads() -> dict:
    """The host threads the oracle may use: the CPU count, this process's
    affinity and the BLAS library's thread count (threadpoolctl when present,
    else the thread environment variables)."""
    info = {"os_cpu_count": os.cpu_count(), "affinity": cpu_cores()}
    try:
        from threadpoolctl import threadpool_info
        info["blas"] = [{"api": d.get("internal_api"), "threads": d.get("num_threads")}
                        for d in threadpool_info() if d.get("user_api") == "blas"]
    except ImportError:
        info["blas_env"] = {k: os.environ.get(k) for k in (
            "OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS") if os.environ.get(k)}
        info["blas"] = "threadpoolctl not installed; BLAS uses its default (all affinity cores)"
    return info


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, cfg):
    """The oracle, timed on the host cores: the whole cycle of the workload per
    step when the run fits the time budget, else a row sample per step
    (extrapolated, and said so)."""
    budget_s = 200.0
    n = args.steps + args.warmup
    inp = oracle_inputs(cfg, 1.0)
    first = oracle_cycle_seconds(cfg, inp)           # also the first warm-up step
    frac = 1.0
    while n * first["total"] * frac > budget_s and frac > 1 / 4096:
        frac /= 2
    if frac < 1.0:
        inp = oracle_inputs(cfg, frac)
    times = []
    wall0 = time.perf_counter()
    sample, extrap = first["sample"], first["extrapolated"]
    for i in range(1, n):
        r = oracle_cycle_seconds(cfg, inp)
        sample, extrap = r["sample"], r["extrapolated"]
        if i >= args.warmup:
            times.append(r["total"])
    while len(times) < args.steps:                  # steps > 0 and warmup == 0
        times.append(oracle_cycle_seconds(cfg, inp)["total"])
    measured_s = time.perf_counter() - wall0
    total = sum(times)
    value = args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": cfg.name, "batch": cfg.batch,
                                            "block": 16, "context": cfg.ctx_len},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample, "extrapolated": extrap,
                             "threads": host_threads(),
                             "host_seconds_of_timed_steps": measured_s},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# the timed cycle
# ---------------------------------------------------------------------------
def cycle_pass(cfg, steps, warmup, concurrent, sm_split_arg, sets, rank, local,
               sample_clocks=False):
    """Build the workload `cfg` on the GPU, fix the verify || projection SM
    split (measured around the proportional one unless given), run `warmup`
    untimed and `steps` timed cycles (CUDA events on the launching stream,
    events around every LM-head launch and the verify || projection phase),
    and return everything the other passes reuse."""
    import types

    import torch

    import block_diffusion_speculative_02_gb300 as dfl
    from block_diffusion_speculative_02_gb300.cycle import side_stream, tune_sm_split

    kv_bytes_per_set = 2 * cfg.n_kv_heads * cfg.head_dim * 2 * (
        cfg.batch * (cfg.ctx_len or cfg.ctx_len_range[1]) + 32)
    n_sets = sets or max(1, min(16, math.ceil(2 * L2_BYTES / max(1, kv_bytes_per_set))))
    dims, w, states, accepts, ws, lens = build_workload(cfg, n_sets)
    stream = torch.cuda.current_stream()
    if concurrent:
        # verify on this stream, the projection on a side stream, each on its
        # own share of the SMs (measured once around the proportional split,
        # before the warm-up); joined before the crop
        if sm_split_arg:
            verify_sms, project_sms = (int(x) for x in sm_split_arg.split(","))
        else:
            verify_sms, project_sms = tune_sm_split(dims, w, states, ws)
        side = side_stream(stream.device)
        fork, join = torch.cuda.Event(), torch.cuda.Event()
        fork2, join2 = torch.cuda.Event(), torch.cuda.Event()
    else:
        verify_sms = project_sms = 0
        side = stream
    dims_v = dfl.with_sm_budget(dims, verify_sms)
    dims_p = dfl.with_sm_budget(dims, project_sms)

    def step(i, ev=None):
        st = states[i % n_sets]
        if concurrent:
            fork.record(stream)
            side.wait_event(fork)
        if ev is not None:
            ev[0].record(stream)
        dfl.dflash_verify_accept(dims_v, st.verify_hidden, w.w_lm, st.block_ids, st.len_before,
                                 st.posterior, st.accept_len, st.next_staged, st.commit_len,
                                 st.out_tokens, ws, stream)
        if ev is not None:
            ev[1].record(stream)
        dfl.dflash_ctx_project(dims_p, st.layer_hidden, w.w_fc, w.hidden_norm_w, w.w_k, w.w_v,
                               w.k_norm_w, st.write_pos, st.draft_cache, ws, side)
        if concurrent:
            join.record(side)
            stream.wait_event(join)
        if ev is not None:
            ev[2].record(stream)
        if concurrent:
            # the crop beside the attention, which reads the drafter context's
            # new length from the commit length (as cycle.run_cycle does)
            fork2.record(stream)
            side.wait_event(fork2)
            dfl.dflash_kv_crop([st.target_view, st.draft_cache], st.commit_len, dims.batch, ws,
                               side)
            dfl.dflash_block_attention(dims, st.q_blk, st.k_blk, st.v_blk,
                                       dataclasses.replace(st.draft_cache, seq_len=st.commit_len),
                                       1.0 / math.sqrt(cfg.head_dim), st.attn_out, ws, stream)
            join2.record(side)
            stream.wait_event(join2)
        else:
            dfl.dflash_kv_crop([st.target_view, st.draft_cache], st.commit_len, dims.batch, ws,
                               stream)
            dfl.dflash_block_attention(dims, st.q_blk, st.k_blk, st.v_blk, st.draft_cache,
                                       1.0 / math.sqrt(cfg.head_dim), st.attn_out, ws, stream)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    status = dfl.dflash_read_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {status:#x} after warm-up")
    sampler = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0])
                           if os.environ.get("CUDA_VISIBLE_DEVICES", "").isdigit() else local)
    if sample_clocks and rank == 0:
        sampler.start()
        time.sleep(0.3)
    lm_events = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3))
                 for _ in range(steps)]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        step(warmup + i, lm_events[i])
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop() if (sample_clocks and rank == 0) else None
    elapsed_s = e0.elapsed_time(e1) / 1e3
    lm_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in lm_events)
    phase_ms = statistics.mean(a.elapsed_time(c) for a, _, c in lm_events)
    status = dfl.dflash_read_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {status:#x} after the timed region")
    return types.SimpleNamespace(
        dims=dims, w=w, states=states, accepts=accepts, ws=ws, lens=lens, n_sets=n_sets,
        concurrent=concurrent, verify_sms=verify_sms, project_sms=project_sms, stream=stream,
        clocks=clocks, elapsed_s=elapsed_s, lm_ms=lm_ms, phase_ms=phase_ms, steps=steps)


# ---------------------------------------------------------------------------
def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_env()
    cfg = CONFIG_BY_NAME[args.config]
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, cfg)
        return 0

    import numpy as np
    import torch

    import __graft_entry__
    torch.cuda.set_device(local)
    __graft_entry__.build()
    world, rank = init_dist("nccl")
    import block_diffusion_speculative_02_gb300 as dfl
    from block_diffusion_speculative_02_gb300.cycle import (CycleGraph, PipelinedCycles,
                                                            packed_tensors)

    cp = cycle_pass(cfg, args.steps, args.warmup, not args.serial, args.sm_split, args.sets,
                    rank, local, sample_clocks=True)
    dims, w, states, accepts, ws, lens = cp.dims, cp.w, cp.states, cp.accepts, cp.ws, cp.lens
    n_sets, concurrent = cp.n_sets, cp.concurrent
    verify_sms, project_sms = cp.verify_sms, cp.project_sms
    stream = cp.stream
    clocks, elapsed_s, lm_ms, phase_ms = cp.clocks, cp.elapsed_s, cp.lm_ms, cp.phase_ms
    max_s = max_over_ranks(elapsed_s, device="cuda")

    # launches of our kernels per step: verify 1, ctx_project 2, crop 1, attention 2
    launches_per_step = 6
    value = whole_job_value(args.steps, world, max_s)
    acc_mean = float(np.mean([np.mean(accepts[(args.warmup + i) % n_sets])
                              for i in range(args.steps)]))
    bytes_ = algorithmic_bytes(cfg, lens)
    peak, peak_kind = measured_peak_gbs()
    cycle_gbs = bytes_["total"] * args.steps / elapsed_s / 1e9
    # the committed DRAM captures are of the Qwen3-8B batch-1 launches only
    tchk = traffic_check() if cfg.name == "qwen3_8b_b1" else None
    traffic = tchk["lmhead_argmax_accept"]["traffic"] \
        if tchk and tchk["lmhead_argmax_accept"] else None

    lm_roofline = lm_head_roofline(cfg, bytes_["lm_head"], lm_ms, (peak, peak_kind),
                                   measured_peak_tflops(), traffic)

    # ---- the same cycles replayed from CUDA graphs (one per input set) ----
    graph_cycle = None
    if args.graph_replays > 0:
        scale = 1.0 / math.sqrt(cfg.head_dim)
        graphs = [CycleGraph(dims, w, states[i], ws, [], [], scale, concurrent=concurrent,
                             sm_split=(verify_sms, project_sms) if concurrent else None)
                  for i in range(n_sets)]
        for i in range(3 * n_sets):
            graphs[i % n_sets].replay()
        torch.cuda.synchronize()
        reps = []
        for _ in range(5):
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            for i in range(args.graph_replays):
                graphs[i % n_sets].replay()
            g1.record(stream)
            torch.cuda.synchronize()
            reps.append(1e3 * g0.elapsed_time(g1) / args.graph_replays)
        if dfl.dflash_read_status(ws) != 0:
            raise RuntimeError(f"device status {dfl.dflash_read_status(ws):#x} "
                               "set by the graph replays")
        del graphs
        us_c = statistics.median(reps)
        graph_cycle = {"value": 1e6 / us_c, "unit": UNIT, "us_per_cycle": us_c,
                       "reps_us": reps, "replays_per_rep": args.graph_replays,
                       "note": "the timed cycle replayed from CUDA graphs (one per rotating input "
                               "set), median of 5 reps"}

    # ---- per-call breakdown (separate pass, events between the calls) ----
    breakdown = None
    if args.breakdown_steps > 0:
        names = ["verify_accept", "ctx_project", "kv_crop", "block_attention"]
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)]
               for _ in range(args.breakdown_steps)]
        torch.cuda.synchronize()
        for i in range(args.breakdown_steps):
            st = states[i % n_sets]
            ev = evs[i]
            ev[0].record(stream)
            dfl.dflash_verify_accept(dims, st.verify_hidden, w.w_lm, st.block_ids, st.len_before,
                                     st.posterior, st.accept_len, st.next_staged, st.commit_len,
                                     st.out_tokens, ws)
            ev[1].record(stream)
            dfl.dflash_ctx_project(dims, st.layer_hidden, w.w_fc, w.hidden_norm_w, w.w_k,
                                   w.w_v, w.k_norm_w, st.write_pos, st.draft_cache, ws)
            ev[2].record(stream)
            dfl.dflash_kv_crop([st.target_view, st.draft_cache], st.commit_len, dims.batch, ws)
            ev[3].record(stream)
            dfl.dflash_block_attention(dims, st.q_blk, st.k_blk, st.v_blk, st.draft_cache,
                                       1.0 / math.sqrt(cfg.head_dim), st.attn_out, ws)
            ev[4].record(stream)
        torch.cuda.synchronize()
        breakdown = {n: 1e3 * statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs)
                     for j, n in enumerate(names)}
        breakdown["unit"] = "us per call (one stream, events between calls)"

    # ---- the rest of the drafter layer and its tokens (beside the cycle) ----
    draft = None
    if args.draft_steps > 0 and cfg.ffn:
        wd, xd, bd = build_draft(cfg)
        dws = dfl.dflash.alloc_draft_workspace(dims, cfg.ffn)
        F = cfg.ffn

        def draft_step(i):
            st = states[i % n_sets]
            dfl.dflash.dflash_draft_qkv(dims, xd, wd["ln1"], wd["wq"], wd["wk"], wd["wv"],
                                        wd["qn"], wd["kn"], bd["q"], bd["k"], bd["v"], dws)
            B_, Hq_, Hkv_, D_ = cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
            dfl.dflash_block_attention(dims, bd["q"].view(B_, 16, Hq_, D_),
                                       bd["k"].view(B_, 16, Hkv_, D_),
                                       bd["v"].view(B_, 16, Hkv_, D_), st.draft_cache,
                                       1.0 / math.sqrt(D_), bd["o"], ws)
            dfl.dflash.dflash_draft_mlp(dims, F, xd, bd["o"].view(B_ * 16, -1), wd["wo"],
                                        wd["ln2"], wd["wg"], wd["wu"], wd["wd"], bd["x_out"], dws)
            dfl.dflash.dflash_draft_tokens(dims, bd["x_out"], wd["fn"], w.w_lm, st.next_staged,
                                           bd["block"], None, dws)

        for i in range(3):
            draft_step(i)
        torch.cuda.synchronize()
        d0 = torch.cuda.Event(enable_timing=True)
        d1 = torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for i in range(args.draft_steps):
            draft_step(i)
        d1.record(stream)
        torch.cuda.synchronize()
        if dfl.dflash_read_status(dws) != 0:
            raise RuntimeError(f"device status {dfl.dflash_read_status(dws):#x} "
                               "set by the drafter calls")
        d_us_calls = 1e3 * d0.elapsed_time(d1) / args.draft_steps
        # the same steps replayed from CUDA graphs (one per rotating input set,
        # so the context caches still come from DRAM): no host work between
        # the launches
        graphs = []
        for i in range(n_sets):
            cap = torch.cuda.Stream()
            cap.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(cap):
                draft_step(i)
            torch.cuda.current_stream().wait_stream(cap)
            torch.cuda.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                draft_step(i)
            graphs.append(gr)
        torch.cuda.synchronize()
        for i in range(n_sets):
            graphs[i].replay()
        torch.cuda.synchronize()
        d0.record()
        for i in range(args.draft_steps):
            graphs[i % n_sets].replay()
        d1.record()
        torch.cuda.synchronize()
        if dfl.dflash_read_status(dws) != 0:
            raise RuntimeError(f"device status {dfl.dflash_read_status(dws):#x} "
                               "set by the drafter calls")
        d_us = 1e3 * d0.elapsed_time(d1) / args.draft_steps
        del graphs
        dbytes = draft_bytes(cfg) + bytes_["attention"]
        draft = {"us_per_block": d_us, "us_per_block_call_by_call": d_us_calls,
                 "bytes_per_block": dbytes,
                 "gbs": dbytes / (d_us / 1e6) / 1e9, "frac": dbytes / (d_us / 1e6) / 1e9 / peak,
                 "ffn": F, "launches_per_block": 9,
                 "note": "Q/K/V + block attention + output projection and SwiGLU MLP + "
                         "final-norm LM-head argmax, one drafter layer, not in the cycle metric"}

    # ---- the target's verify attention on a cache of the same shapes ----
    vatt = None
    if args.draft_steps > 0:
        st = states[0]
        dc = st.draft_cache
        L0 = dc.seq_len.clone()
        tview = dfl.KVView(dc.k, dc.v, dc.seq_len.clone(), capacity=dc.capacity,
                           page_table=dc.page_table, free_list=dc.free_list,
                           free_count=dc.free_count, page_size=dc.page_size)
        o_v = torch.empty_like(st.attn_out)
        D_ = cfg.head_dim

        # Each call appends 16 rows and moves the length, so every call starts
        # from the same length again (a 4-byte reset).  The calls are replayed
        # from CUDA graphs, so host-side work between them cannot stretch the
        # device time; the reset alone is timed the same way and subtracted.
        def reset():
            tview.seq_len.copy_(L0)

        def vcall():
            reset()
            dfl.dflash.dflash_verify_attention(dims, st.q_blk, st.k_blk, st.v_blk, tview,
                                               1.0 / math.sqrt(D_), o_v, ws)

        def graph_of(fn):
            cap = torch.cuda.Stream()
            cap.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(cap):
                for _ in range(3):
                    fn()
            torch.cuda.current_stream().wait_stream(cap)
            torch.cuda.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                fn()
            torch.cuda.synchronize()
            return gr

        def replay_us(gr, n):
            for _ in range(3):
                gr.replay()
            torch.cuda.synchronize()
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record()
            for _ in range(n):
                gr.replay()
            a1.record()
            torch.cuda.synchronize()
            return 1e3 * a0.elapsed_time(a1) / n

        g_v, g_r = graph_of(vcall), graph_of(reset)
        us_both = replay_us(g_v, args.draft_steps)
        us_reset = replay_us(g_r, args.draft_steps)
        us = us_both - us_reset
        if dfl.dflash_read_status(ws) != 0:
            raise RuntimeError(f"device status {dfl.dflash_read_status(ws):#x} "
                               "set by the verify attention")
        dc.seq_len.copy_(L0)
        vbytes = bytes_["attention"] + 2 * cfg.batch * 16 * cfg.n_kv_heads * D_ * 2
        vatt = {"us": us, "bytes": vbytes, "gbs": vbytes / (us / 1e6) / 1e9,
                "us_with_length_reset": us_both,
                "note": "one layer of the target's verify forward: causal-in-block attention "
                        "over the context plus the block K/V appended, replayed from a CUDA "
                        "graph; not in the cycle metric"}

    # ---- GatedDeltaNet tape-replay rollback (hybrid targets; synthetic states) ----
    gdn = None
    if args.draft_steps > 0:
        NH, DK, DV = 24 * 32, 128, 128           # 24 recurrent layers x 32 heads
        Bg = cfg.batch
        gg = torch.Generator(device="cuda")
        gg.manual_seed(7)
        states_g = [0.3 * torch.randn((Bg, NH, DV, DK), generator=gg, device="cuda")
                    for _ in range(3)]                # rotate: 3 x 48 MB > L2
        kt = torch.nn.functional.normalize(
            torch.randn((Bg, 16, NH, DK), generator=gg, device="cuda"), dim=-1).to(torch.bfloat16)
        vt = torch.randn((Bg, 16, NH, DV), generator=gg, device="cuda").to(torch.bfloat16)
        bt = torch.rand((Bg, 16, NH), generator=gg, device="cuda")
        gt = -0.3 * torch.rand((Bg, 16, NH), generator=gg, device="cuda")
        acc_g = states[0].accept_len
        gws = torch.zeros(256, dtype=torch.uint8, device="cuda")
        for i in range(3):
            dfl.dflash.dflash_gdn_replay(states_g[i % 3], kt, vt, bt, gt, acc_g, gws)
        torch.cuda.synchronize()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for i in range(args.draft_steps):
            dfl.dflash.dflash_gdn_replay(states_g[i % 3], kt, vt, bt, gt, acc_g, gws)
        g1.record(stream)
        torch.cuda.synchronize()
        if dfl.dflash_read_status(gws) != 0:
            raise RuntimeError(f"device status {dfl.dflash_read_status(gws):#x} "
                               "set by the GDN replay")
        us = 1e3 * g0.elapsed_time(g1) / args.draft_steps
        steps = int(acc_g.sum().item()) + Bg
        gbytes = Bg * NH * DV * DK * 4 * 2 + steps * NH * ((DK + DV) * 2 + 8)
        gdn = {"us": us, "bytes": gbytes, "gbs": gbytes / (us / 1e6) / 1e9,
               "frac": gbytes / (us / 1e6) / 1e9 / peak,
               "shape": f"B {Bg}, {NH} recurrent heads (24 layers x 32), Dk = Dv = {DK}, "
                        f"1 + a steps replayed",
               "note": "synthetic states; not in the cycle metric"}

    # ---- whole-prompt context projection (prefill), tensor-bound ----
    prefill = None
    if args.prefill_tokens > 0:
        T = args.prefill_tokens
        B_ = 1
        gp = torch.Generator(device="cuda")
        gp.manual_seed(11)
        pl_hidden = [torch.randn((B_ * T, cfg.hidden), generator=gp, device="cuda")
                     .to(torch.bfloat16) for _ in range(cfg.n_ctx_layers)]
        pdims = dfl.make_dims(B_, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                              cfg.vocab, cfg.n_ctx_layers, T, rope_theta=cfg.rope_theta)
        pws = dfl.dflash.alloc_prefill_workspace(pdims, T)
        pk = torch.empty((B_, cfg.n_kv_heads, T, cfg.head_dim), dtype=torch.bfloat16,
                         device="cuda")
        pview = dfl.KVView(pk, torch.empty_like(pk), torch.zeros(B_, dtype=torch.int32,
                                                                 device="cuda"), capacity=T)
        zero_pos = torch.zeros(B_, dtype=torch.int32, device="cuda")

        def prefill_call():
            dfl.dflash.dflash_ctx_prefill(pdims, T, pl_hidden, w.w_fc, w.hidden_norm_w, w.w_k,
                                          w.w_v, w.k_norm_w, zero_pos, pview, pws)

        for _ in range(3):
            prefill_call()
        torch.cuda.synchronize()
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        reps = 10
        p0.record(stream)
        for _ in range(reps):
            prefill_call()
        p1.record(stream)
        torch.cuda.synchronize()
        if dfl.dflash_read_status(pws) != 0:
            raise RuntimeError(f"device status {dfl.dflash_read_status(pws):#x} "
                               "set by the prefill projection")
        p_us = 1e3 * p0.elapsed_time(p1) / reps
        kvd = cfg.n_kv_heads * cfg.head_dim
        pflops = 2.0 * B_ * T * cfg.hidden * (cfg.n_ctx_layers * cfg.hidden + 2 * kvd)
        tpk, tpk_kind = measured_peak_tflops()
        prefill = {"tokens": B_ * T, "us": p_us, "tokens_per_s": B_ * T / (p_us / 1e6),
                   "roofline": {"bound": "tensor", "achieved": pflops / (p_us / 1e6) / 1e12,
                                "peak": tpk, "peak_kind": tpk_kind, "unit": "TFLOP/s",
                                "frac": pflops / (p_us / 1e6) / 1e12 / tpk,
                                "flops_per_call": pflops},
                   "note": "fc GEMM + K/V GEMM over a whole prompt (two launches), "
                           "not in the cycle metric"}
        del pl_hidden, pws, pk, pview

    # ---- the target's prefill attention: one layer over the prompt, in chunks ----
    prefill_att = None
    if args.prefill_tokens > 0:
        T, C = args.prefill_tokens, min(args.prefill_chunk, args.prefill_tokens)
        Hq_, Hkv_, D_ = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
        ga = torch.Generator(device="cuda")
        ga.manual_seed(13)
        qa = torch.randn((1, T, Hq_, D_), generator=ga, device="cuda").to(torch.bfloat16)
        ka = torch.randn((1, T, Hkv_, D_), generator=ga, device="cuda").to(torch.bfloat16)
        va = torch.randn((1, T, Hkv_, D_), generator=ga, device="cuda").to(torch.bfloat16)
        chunks = [(a, min(C, T - a)) for a in range(0, T, C)]
        qc = [qa[:, a:a + n].contiguous() for a, n in chunks]
        kc = [ka[:, a:a + n].contiguous() for a, n in chunks]
        vc = [va[:, a:a + n].contiguous() for a, n in chunks]
        oc = [torch.empty_like(x) for x in qc]
        adims = dfl.make_dims(1, cfg.hidden, Hq_, Hkv_, D_, cfg.vocab, cfg.n_ctx_layers, T,
                              rope_theta=cfg.rope_theta)
        aws = [dfl.dflash.alloc_prefill_workspace(adims, n) for _, n in chunks]
        ak = torch.empty((1, Hkv_, T, D_), dtype=torch.bfloat16, device="cuda")
        aview = dfl.KVView(ak, torch.empty_like(ak),
                           torch.zeros(1, dtype=torch.int32, device="cuda"), capacity=T)

        def prompt_pass():
            aview.seq_len.zero_()
            for j, (_, n) in enumerate(chunks):
                dfl.dflash.dflash_prefill_attention(adims, n, qc[j], kc[j], vc[j], aview,
                                                    1.0 / math.sqrt(D_), oc[j], aws[j])

        for _ in range(2):
            prompt_pass()
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        reps = 5
        a0.record(stream)
        for _ in range(reps):
            prompt_pass()
        a1.record(stream)
        torch.cuda.synchronize()
        for x in aws:
            if dfl.dflash_read_status(x) != 0:
                raise RuntimeError("device status set by the prefill attention")
        a_us = 1e3 * a0.elapsed_time(a1) / reps
        # causal attention: row t scores t + 1 keys; QK^T and PV, 2 flops per MAC each
        aflops = 4.0 * Hq_ * D_ * (T * (T + 1) / 2)
        # bytes it must move: Q, K, V in, O out, the appended K/V rows
        abytes = 2 * T * (2 * Hq_ + 4 * Hkv_) * D_
        tpk, tpk_kind = measured_peak_tflops()
        prefill_att = {
            "tokens": T, "chunk": C, "us": a_us,
            "roofline": {"bound": "tensor", "achieved": aflops / (a_us / 1e6) / 1e12,
                         "peak": tpk, "peak_kind": tpk_kind, "unit": "TFLOP/s",
                         "frac": aflops / (a_us / 1e6) / 1e12 / tpk, "flops_per_prompt": aflops,
                         "hbm_gbs": abytes / (a_us / 1e6) / 1e9, "bytes_per_prompt": abytes},
            "note": "one layer of the target's prefill: causal attention over the prompt fed in "
                    "chunks, each chunk's K/V appended to the cache (append + attention + "
                    "length launches per chunk); the query rows of a KV head (4 heads x 16 "
                    "rows) are staged twice in the 128-row MMA, so half the tensor issue "
                    "carries duplicates; not in the cycle metric"}
        del qa, ka, va, qc, kc, vc, oc, aws, ak, aview

    # ---- end to end: host buffers in, results out, every step ----
    e2e = None
    if args.e2e_steps > 0:
        # the step's inputs (verify hidden, selected layer hidden states, block
        # ids, block Q/K/V) live in one device buffer per slot and its results
        # (acceptance, next staged token, commit length, posterior) in one
        # device buffer, so that every step moves them with one host-to-device
        # and one device-to-host copy
        src = states[0]
        in_t = [src.verify_hidden, *src.layer_hidden, src.block_ids, src.q_blk, src.k_blk,
                src.v_blk]
        out_t = [src.accept_len, src.next_staged, src.commit_len, src.posterior]
        specs = [(t.shape, t.dtype) for t in in_t]
        slots = [packed_tensors(specs, "cuda") for _ in range(2)]
        dev_out, outs = packed_tensors([(t.shape, t.dtype) for t in out_t], "cuda")
        for _, ins in slots:
            for d_, t in zip(ins, in_t):
                d_.copy_(t)
        st_slots = [dataclasses.replace(
            src, verify_hidden=ins[0], layer_hidden=ins[1:1 + len(src.layer_hidden)],
            block_ids=ins[-4], q_blk=ins[-3], k_blk=ins[-2], v_blk=ins[-1],
            accept_len=outs[0], next_staged=outs[1], commit_len=outs[2], posterior=outs[3])
            for _, ins in slots]
        st_slots[0].commit_len.copy_(src.commit_len)
        host_in = slots[0][0].cpu().pin_memory()
        host_out = [torch.empty_like(dev_out, device="cpu").pin_memory() for _ in range(2)]
        h2d = host_in.numel()
        d2h = host_out[0].numel()
        # the serving loop of a fixed-shape batch: each step is one CUDA graph
        # (the whole cycle plus the copy of its results to the host); the copy
        # of the next step's inputs overlaps the current step
        pc = PipelinedCycles(dims, w, st_slots, ws, [d for d, _ in slots],
                             [(dev_out, host_out)], 1.0 / math.sqrt(cfg.head_dim),
                             concurrent=concurrent,
                             sm_split=(verify_sms, project_sms) if concurrent else None)
        for _ in range(3):
            pc.step(host_in)
        pc.finish()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            pc.step(host_in)
        pc.finish()
        e2e_s = time.perf_counter() - t0
        e2e_s = max_over_ranks(e2e_s, device="cuda")
        e2e = {"value": whole_job_value(args.e2e_steps, world, e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "loop": "PipelinedCycles: one graph per step; the next step's host-to-device "
                       "copy overlaps the current step; results read back every step"}

    # ---- the headline workload with the other draft-match draw (mean 13) ----
    alt = None
    if args.alt_draw_steps > 0 and cfg.accept[0] == "uniform" and cfg.name == DEFAULT_CONFIG:
        cfg_g = dataclasses.replace(cfg, accept=("geometric", 13.0))
        split = "%d,%d" % (verify_sms, project_sms) if concurrent else ""
        cg = cycle_pass(cfg_g, args.alt_draw_steps, 5, concurrent, split, args.sets, rank, local)
        sg = max_over_ranks(cg.elapsed_s, device="cuda")
        vg = whole_job_value(args.alt_draw_steps, world, sg)
        accg = float(np.mean([np.mean(a) for a in cg.accepts]))
        alt = {"draw": "truncated geometric, mean 13", "value": vg, "unit": UNIT,
               "steps": args.alt_draw_steps, "warmup": 5,
               "ms_per_step": 1e3 * sg / args.alt_draw_steps,
               "committed_tokens_per_s": vg * cfg.batch * (1 + accg),
               "tokens_per_cycle": cfg.batch * (1 + accg), "acceptance_rate": accg / 15.0,
               "note": "same workload, SM split and timing rules as the headline, whose "
                       "draft match lengths are uniform in 0..15"}
        del cg

    # ---- the batch-32 paged serving step, timed the same way (beside the headline) ----
    b32 = None
    if args.b32_steps > 0 and cfg.name == DEFAULT_CONFIG and not args.serial:
        cfg32 = CONFIG_BY_NAME["qwen3_8b_b32_paged"]
        c32 = cycle_pass(cfg32, args.b32_steps, 5, True, "", 0, rank, local)
        s32 = max_over_ranks(c32.elapsed_s, device="cuda")
        v32 = whole_job_value(args.b32_steps, world, s32)
        by32 = algorithmic_bytes(cfg32, c32.lens)
        acc32 = float(np.mean([np.mean(a) for a in c32.accepts]))
        rl32 = lm_head_roofline(cfg32, by32["lm_head"], c32.lm_ms, (peak, peak_kind),
                                measured_peak_tflops(), None)
        b32 = {"workload": cfg32.name, "value": v32, "unit": UNIT, "steps": args.b32_steps,
               "warmup": 5, "ms_per_step": 1e3 * s32 / args.b32_steps,
               "committed_tokens_per_s": v32 * cfg32.batch * (1 + acc32),
               "cycle_gbs": by32["total"] * args.b32_steps / c32.elapsed_s / 1e9,
               "cycle_roofline_frac": by32["total"] * args.b32_steps / c32.elapsed_s / 1e9 / peak,
               "verify_project_phase_us": 1e3 * c32.phase_ms,
               "roofline": rl32,
               "verify_project": "side by side, SM budgets %d + %d" % (c32.verify_sms,
                                                                        c32.project_sms),
               "note": "32 sequences, contexts U[512, 16384] in a shuffled paged cache, same "
                       "cycle, rotating-set and timing rules as the headline; the LM head and "
                       "the fc GEMM are bound by the tensor cores at this batch"}
        del c32

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp = oracle_inputs(cfg, 1.0)
        reps = [oracle_cycle_seconds(cfg, inp) for _ in range(3)]
        tot = statistics.median(r["total"] for r in reps)
        cpu = {"value": 1.0 / tot, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": reps[0]["sample"] + "; median of 3",
               "extrapolated": reps[0]["extrapolated"], "threads": host_threads()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * max_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": cfg.name, "batch": cfg.batch, "block": 16,
                       "hidden": cfg.hidden, "vocab": cfg.vocab, "context": int(lens.max()),
                       "ctx_layers": cfg.n_ctx_layers, "drafter_layers": 1,
                       "l2": f"{n_sets} rotating input sets (> L2)", "graph": False,
                       "verify_project": ("side by side, SM budgets %d + %d"
                                          % (verify_sms, project_sms)) if concurrent
                       else "one stream"},
            "committed_tokens_per_s": value * cfg.batch * (1 + acc_mean),
            "tokens_per_cycle": cfg.batch * (1 + acc_mean),
            "acceptance_rate": acc_mean / 15.0,
            "geometric_draw": alt,
            "cycle_gbs": cycle_gbs, "cycle_roofline_frac": cycle_gbs / peak,
            "algorithmic_bytes_per_cycle": bytes_,
            "verify_project_phase": {
                "us": 1e3 * phase_ms,
                "gbs": (bytes_["lm_head"] + bytes_["ctx_project"]) / (phase_ms / 1e3) / 1e9},
            "roofline": lm_roofline,
            "traffic_check": tchk,
            "gpu_launches": launches_per_step * args.steps,
            "graph_replay": graph_cycle,
            "breakdown": breakdown,
            "drafter_layer": draft,
            "verify_attention": vatt,
            "gdn_replay": gdn,
            "prefill_projection": prefill,
            "prefill_attention": prefill_att,
            "configs": {"qwen3_8b_b32_paged": b32} if b32 else None,
            "clocks": clocks,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    barrier()
    return 0


if __name__ == "__main__":
    sys.exit(main())
