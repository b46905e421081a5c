"""Float64 CPU oracle for the DFlash per-cycle hot path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module: only the test-suite, the smoke check and the bench's CPU-baseline
leg use it.  It shares no code with the CUDA library.

Everything is the plain definition written out in NumPy float64.  bf16 inputs
(uint16 bit patterns) are read as exact float64 values.  Where the pages leave
a step open, the reading taken is stated next to the function.

Sources (web pages on DFlash; cited by page and section):
  [P1] "DFlash双实现对比：PyTorch与MLX代码架构差异深度分析" (hotelren.com)
       §1 model definition (Qwen3 RMSNorm / rotary embedding reused),
       §2 attention (dual-source K/V: ctx ⊕ block, Q from the block only,
          non-causal inside the block), §3 KV-cache crop, §4 target-layer
          hidden states concatenated by target_layer_ids.
  [P2] "dflash-mlx" lossless speculative decoding (dpshk.com)
       块扩散草稿 (block = staged token + 15 masks; drafter reads target hidden),
       单次前向验证 (the nine-step cycle ①–⑨),
       保证二 (acceptance = sum(cumprod(draft == posterior)); prefix semantics;
          the first rejected position takes the target's own token),
       保证三 (caches cut back to the committed length).

Parity pins: see tests/test_oracle_*.py.  Every function below is pinned there
by something other than itself (brute force, closed forms, invariants,
worked cases from [P2]).
"""
from __future__ import annotations

import numpy as np

BLOCK = 16


# ---------------------------------------------------------------------------
# elementary pieces
# ---------------------------------------------------------------------------
def bf16_to_f64(bits) -> np.ndarray:
    """Exact float64 value of bf16 bit patterns (uint16)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def as_f64(x) -> np.ndarray:
    """uint16 arrays are bf16 bit patterns; everything else is converted to float64."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_to_f64(x)
    return x.astype(np.float64)


def rms_norm(x: np.ndarray, weight, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * weight.

    The Qwen3 RMSNorm the drafter reuses ([P1] §1).
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    y = x / np.sqrt(ms + eps)
    if weight is not None:
        y = y * as_f64(weight)
    return y


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """inv_freq[d] = theta^(-2d/D) for d < D/2 (Qwen3 rotary embedding, [P1] §1)."""
    d = np.arange(head_dim // 2, dtype=np.float64)
    return theta ** (-2.0 * d / head_dim)


def apply_rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE: for d < D/2 with angle = pos * inv_freq[d]
         x'[d]       = x[d] cos - x[d + D/2] sin
         x'[d + D/2] = x[d + D/2] cos + x[d] sin
    ``positions`` has the shape of ``x`` without its last axis.
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    half = D // 2
    pos = np.asarray(positions, dtype=np.float64)
    assert pos.shape == x.shape[:-1], (pos.shape, x.shape)
    ang = pos[..., None] * rope_inv_freq(D, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ---------------------------------------------------------------------------
# a1: context projection
# ---------------------------------------------------------------------------
def ctx_project(layer_hidden, w_fc, hidden_norm_w, w_k, w_v, k_norm_w, positions,
                n_kv_heads: int, head_dim: int, rope_theta: float, rms_eps: float) -> dict:
    """Context K/V for the drafter from the target's selected-layer hidden states.

    [P1] §4: the hidden states of the layers listed in target_layer_ids are
    concatenated; [P1] §2 / [P2] 块扩散草稿: the drafter's context K/V are
    projected from them.  Steps:
        X  = [h_l1 | h_l2 | ... | h_lnL]              (concat on the feature axis)
        Y  = X W_fc^T
        Y^ = RMSNorm(Y) * g_h            (if hidden_norm_w is given)
        K  = RoPE_pos(RMSNorm_head(Y^ W_k^T) * g_k)   (per-head norm if k_norm_w given)
        V  = Y^ W_v^T
    layer_hidden: nL arrays [N, H]; positions: [N] absolute token positions.
    Returns y, yhat [N, H]; k, v [N, Hkv, D].
    """
    xs = [as_f64(h) for h in layer_hidden]
    x = np.concatenate(xs, axis=-1)
    y = x @ as_f64(w_fc).T
    yhat = rms_norm(y, hidden_norm_w, rms_eps) if hidden_norm_w is not None else y
    N = y.shape[0]
    k = (yhat @ as_f64(w_k).T).reshape(N, n_kv_heads, head_dim)
    if k_norm_w is not None:
        k = rms_norm(k, k_norm_w, rms_eps)
    pos = np.broadcast_to(np.asarray(positions, dtype=np.float64)[:, None], (N, n_kv_heads))
    k = apply_rope(k, pos, rope_theta)
    v = (yhat @ as_f64(w_v).T).reshape(N, n_kv_heads, head_dim)
    return {"y": y, "yhat": yhat, "k": k, "v": v}


# ---------------------------------------------------------------------------
# a2: dual-source block attention
# ---------------------------------------------------------------------------
def block_attention(q_blk, k_blk, v_blk, ctx_k, ctx_v, seq_len, rope_theta: float,
                    scale: float) -> np.ndarray:
    """Drafter attention over ctx K/V concatenated with the block's own K/V.

    [P1] §2: Q comes only from the block tokens; K/V = concat(context K/V,
    block K/V); no causal mask inside the block.  GQA: query head h reads KV
    head floor(h / G) with G = Hq / Hkv.  Block token j sits at position
    L_b + j ([P2] 单次前向验证 ③: the staged token follows the context); ctx K
    is stored already rotated, block Q/K are rotated here.

    q_blk [B,T,Hq,D], k_blk/v_blk [B,T,Hkv,D] (pre-RoPE); ctx_k/ctx_v: per
    sequence arrays with at least L_b rows [.., Hkv, D]; seq_len [B] = L_b.
    Returns O [B,T,Hq,D] float64.
    """
    q_blk, k_blk, v_blk = as_f64(q_blk), as_f64(k_blk), as_f64(v_blk)
    B, T, Hq, D = q_blk.shape
    Hkv = k_blk.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    for b in range(B):
        L = int(seq_len[b])
        pos = L + np.arange(T, dtype=np.float64)
        q = apply_rope(q_blk[b], np.broadcast_to(pos[:, None], (T, Hq)), rope_theta)
        kb = apply_rope(k_blk[b], np.broadcast_to(pos[:, None], (T, Hkv)), rope_theta)
        keys = np.concatenate([as_f64(ctx_k[b][:L]).reshape(L, Hkv, D), kb], axis=0)
        vals = np.concatenate([as_f64(ctx_v[b][:L]).reshape(L, Hkv, D), v_blk[b]], axis=0)
        for h in range(Hq):
            g = h // G
            s = (q[:, h, :] @ keys[:, g, :].T) * scale        # [T, L+T], no mask
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=1, keepdims=True)
            out[b, :, h, :] = p @ vals[:, g, :]
    return out


# ---------------------------------------------------------------------------
# a3: verification epilogue
# ---------------------------------------------------------------------------
def lm_head_argmax(hidden, w_lm, chunk: int = 8192) -> dict:
    """Greedy argmax of logits = hidden W_lm^T, never materialising all logits.

    [P2] 保证一: every verify position's logits give their greedy argmax (the
    posterior).  Exact ties go to the lowest vocabulary index (the pages are
    silent; this reading is the one the kernels implement).
    Also returns, per row, the top-2 gap (max - second max, 0 on exact ties)
    and the max logit, which decide whether a position is a near tie.
    hidden [N, H]; w_lm [V, H].  Vocabulary rows are processed in chunks.
    """
    h = as_f64(hidden)
    N = h.shape[0]
    V = np.asarray(w_lm).shape[0]
    best = np.full(N, -np.inf)
    second = np.full(N, -np.inf)
    idx = np.zeros(N, dtype=np.int64)
    rows = np.arange(N)
    for v0 in range(0, V, chunk):
        w = as_f64(w_lm[v0:v0 + chunk])
        logits = h @ w.T                                   # [N, c]
        c_idx = np.argmax(logits, axis=1)                  # first maximum in the chunk
        c1 = logits[rows, c_idx]
        logits[rows, c_idx] = -np.inf
        c2 = logits.max(axis=1) if logits.shape[1] > 1 else np.full(N, -np.inf)
        new_second = np.maximum(np.maximum(np.minimum(best, c1), second), c2)
        take = c1 > best                                   # strictly greater: earlier chunk wins ties
        idx = np.where(take, v0 + c_idx, idx)
        best = np.maximum(best, c1)
        second = new_second
    return {"posterior": idx.astype(np.int32), "max": best, "gap": best - second}


# ---------------------------------------------------------------------------
# next: the target's attention in the verify forward
# ---------------------------------------------------------------------------
def verify_attention(q_blk, k_blk, v_blk, ctx_k, ctx_v, seq_len, rope_theta: float,
                     scale: float) -> dict:
    """The target's attention for the 16 verify rows of one layer.

    [P2] 单次前向验证 ⑤: the target runs one forward over the block
    [staged, d_1..d_15]; it is an ordinary causal decoder, so block row i sees
    the cached context rows 0..L_b-1 and the block rows 0..i, and the block's
    K/V join the target's cache (保证三 later cuts it back to the committed
    length).  Positions, GQA and RoPE as in block_attention.
    Returns O [B,T,Hq,D] and the rotated block K and the block V
    [B,T,Hkv,D] that are appended to the cache at rows L_b..L_b+15.
    """
    q_blk, k_blk, v_blk = as_f64(q_blk), as_f64(k_blk), as_f64(v_blk)
    B, T, Hq, D = q_blk.shape
    Hkv = k_blk.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    k_rot = np.zeros((B, T, Hkv, D), dtype=np.float64)
    for b in range(B):
        L = int(seq_len[b])
        pos = L + np.arange(T, dtype=np.float64)
        q = apply_rope(q_blk[b], np.broadcast_to(pos[:, None], (T, Hq)), rope_theta)
        kb = apply_rope(k_blk[b], np.broadcast_to(pos[:, None], (T, Hkv)), rope_theta)
        k_rot[b] = kb
        keys = np.concatenate([as_f64(ctx_k[b][:L]).reshape(L, Hkv, D), kb], axis=0)
        vals = np.concatenate([as_f64(ctx_v[b][:L]).reshape(L, Hkv, D), v_blk[b]], axis=0)
        mask = np.zeros((T, L + T), dtype=bool)
        for i in range(T):
            mask[i, L + i + 1:] = True                       # later block rows are hidden
        for h in range(Hq):
            g = h // G
            s = (q[:, h, :] @ keys[:, g, :].T) * scale
            s[mask] = -np.inf
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=1, keepdims=True)
            out[b, :, h, :] = p @ vals[:, g, :]
    return {"o": out, "k": k_rot, "v": v_blk.copy()}


# ---------------------------------------------------------------------------
# next: the target's prefill (attention over prompt chunks, staged token)
# ---------------------------------------------------------------------------
def prefill_attention(q, k, v, ctx_k, ctx_v, seq_len, rope_theta: float, scale: float) -> dict:
    """The target's attention over one chunk of the prompt, one layer.

    [P2] 单次前向验证 ①: the target prefills the prompt chunk by chunk, which
    initialises its KV cache.  A decoder is causal, so chunk row t of sequence
    b, at position L_b + t, attends to the rows already cached (0..L_b-1) and
    to the chunk rows 0..t; the chunk's rotated K and its V join the cache at
    rows L_b..L_b+T-1.  A whole prompt fed in chunks therefore gives the same
    rows as the prompt fed at once.  GQA, RoPE and positions as in
    block_attention.
    q [B,T,Hq,D], k/v [B,T,Hkv,D] (pre-RoPE), any T >= 1; ctx_k/ctx_v per
    sequence with at least L_b rows [.., Hkv, D] (stored rotated); seq_len [B].
    Returns o [B,T,Hq,D], the rotated chunk K and the chunk V [B,T,Hkv,D].
    """
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    k_rot = np.zeros((B, T, Hkv, D), dtype=np.float64)
    for b in range(B):
        L = int(seq_len[b])
        pos = L + np.arange(T, dtype=np.float64)
        qr = apply_rope(q[b], np.broadcast_to(pos[:, None], (T, Hq)), rope_theta)
        kr = apply_rope(k[b], np.broadcast_to(pos[:, None], (T, Hkv)), rope_theta)
        k_rot[b] = kr
        keys = np.concatenate([as_f64(ctx_k[b][:L]).reshape(L, Hkv, D), kr], axis=0)
        vals = np.concatenate([as_f64(ctx_v[b][:L]).reshape(L, Hkv, D), v[b]], axis=0)
        # row t sees keys 0 .. L + t
        hidden = np.arange(L + T)[None, :] > (L + np.arange(T))[:, None]
        for h in range(Hq):
            g = h // G
            s = (qr[:, h, :] @ keys[:, g, :].T) * scale
            s[hidden] = -np.inf
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=1, keepdims=True)
            out[b, :, h, :] = p @ vals[:, g, :]
    return {"o": out, "k": k_rot, "v": v.copy()}


def prefill_staged(last_hidden, w_lm, chunk: int = 8192) -> dict:
    """The first staged token ([P2] 单次前向验证 ②): the target's greedy token
    after the prompt, i.e. the argmax (lowest index on exact ties) of the LM
    head at the last prompt row.  last_hidden [B, H] (final-normed).  Returns
    the tokens [B] with the gap and max of lm_head_argmax."""
    r = lm_head_argmax(last_hidden, w_lm, chunk)
    r["staged"] = r["posterior"].copy()
    return r


def round_bf16(x) -> np.ndarray:
    """float64 -> bf16 bit patterns (uint16), rounding to nearest even via the
    float32 value (x rounded to float32, then its 16 low bits rounded away).
    Used where a float64 computation hands values to a bf16 consumer."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    r = ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16))
    r = np.where(nan, (u >> np.uint64(16)) | np.uint64(0x40), r)
    return r.astype(np.uint16)


# ---------------------------------------------------------------------------
# next: rollback of the recurrent (GatedDeltaNet) state of a hybrid target
# ---------------------------------------------------------------------------
def gdn_step(S, k, v, beta: float, g: float) -> np.ndarray:
    """One step of the gated delta rule on a state S [Dv, Dk]:
        S <- exp(g) * S (I - beta k k^T) + beta v k^T
    the recurrence of a GatedDeltaNet linear-attention layer (the layers whose
    state [P1] §7 and [P2] 保证三 say cannot simply be truncated)."""
    S = np.asarray(S, dtype=np.float64)
    k = as_f64(k)
    v = as_f64(v)
    Dk = k.shape[0]
    return np.exp(g) * S @ (np.eye(Dk) - beta * np.outer(k, k)) + beta * np.outer(v, k)


def gdn_replay(state, tape_k, tape_v, tape_beta, tape_g, n_steps) -> np.ndarray:
    """Tape-replay rollback ([P2] 保证三, [P1] §7): the verify forward recorded,
    per block step t, the innovation (k_t, v_t, beta_t, g_t) of every
    recurrent head; after acceptance only the first n_steps = 1 + a steps are
    replayed onto the state saved before the verify forward, which rebuilds the
    state exactly as if only the committed tokens had been processed.
    state [B, NH, Dv, Dk] (NH = recurrent heads over all such layers);
    tape_k [B, T, NH, Dk], tape_v [B, T, NH, Dv], tape_beta/tape_g [B, T, NH];
    n_steps [B].  Returns the new state [B, NH, Dv, Dk]."""
    out = np.array(state, dtype=np.float64, copy=True)
    B, NH = out.shape[:2]
    for b in range(B):
        for h in range(NH):
            S = out[b, h]
            for t in range(int(n_steps[b])):
                S = gdn_step(S, tape_k[b, t, h], tape_v[b, t, h], float(tape_beta[b, t, h]),
                             float(tape_g[b, t, h]))
            out[b, h] = S
    return out


# ---------------------------------------------------------------------------
# next: the rest of one drafter layer and the drafter's token choice
# ---------------------------------------------------------------------------
def draft_qkv(x, ln1_w, w_q, w_k, w_v, q_norm_w, k_norm_w, n_q_heads: int, n_kv_heads: int,
              head_dim: int, rms_eps: float) -> dict:
    """Block Q/K/V of one drafter layer, before the rotary embedding.

    [P1] §1: the drafter is built from Qwen3 components (RMSNorm, rotary
    embedding, MLP), i.e. a pre-norm decoder layer whose attention projections
    are followed by a per-head RMSNorm of q and k; [P2] 块扩散草稿 steps 1-2:
    the whole block (staged token + 15 masks) goes through one forward.
        h = RMSNorm(x) * ln1
        q = RMSNorm_head(h W_q^T) * q_norm,  k = RMSNorm_head(h W_k^T) * k_norm
        v = h W_v^T
    x [N, H] (the layer input rows, N = 16 per sequence).  Returns h [N, H],
    q [N, Hq, D], k, v [N, Hkv, D] (the attention rotates q and k itself).
    """
    h = rms_norm(as_f64(x), ln1_w, rms_eps)
    N = h.shape[0]
    q = (h @ as_f64(w_q).T).reshape(N, n_q_heads, head_dim)
    k = (h @ as_f64(w_k).T).reshape(N, n_kv_heads, head_dim)
    v = (h @ as_f64(w_v).T).reshape(N, n_kv_heads, head_dim)
    if q_norm_w is not None:
        q = rms_norm(q, q_norm_w, rms_eps)
    if k_norm_w is not None:
        k = rms_norm(k, k_norm_w, rms_eps)
    return {"h": h, "q": q, "k": k, "v": v}


def silu(x):
    """x * sigmoid(x), the activation of the Qwen3 MLP."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def draft_out_mlp(x, attn_out, w_o, ln2_w, w_gate, w_up, w_down, rms_eps: float) -> dict:
    """The rest of one drafter layer after its attention ([P1] §1, Qwen3
    decoder layer with the Qwen3 MLP):
        x1 = x + O W_o^T                       (O = attention output rows, [N, Hq*D])
        x2 = x1 + (silu(h2 W_gate^T) * (h2 W_up^T)) W_down^T,  h2 = RMSNorm(x1) * ln2
    Returns x1, x2 [N, H]."""
    x = as_f64(x)
    N = x.shape[0]
    x1 = x + as_f64(attn_out).reshape(N, -1) @ as_f64(w_o).T
    h2 = rms_norm(x1, ln2_w, rms_eps)
    m = silu(h2 @ as_f64(w_gate).T) * (h2 @ as_f64(w_up).T)
    x2 = x1 + m @ as_f64(w_down).T
    return {"x1": x1, "x2": x2}


def draft_tokens(x, final_norm_w, w_lm, rms_eps: float, chunk: int = 8192) -> dict:
    """The drafter's prediction for every block position: greedy argmax of
    RMSNorm(x) * final_norm W_lm^T (the drafter shares the target's LM head);
    the mask positions 1..15 are the drafted tokens ([P2] 块扩散草稿 step 2).
    x [B*16, H].  Returns the argmax, gap and max per row (as lm_head_argmax)
    and tokens [B, 15]."""
    hn = rms_norm(as_f64(x), final_norm_w, rms_eps)
    r = lm_head_argmax(hn, w_lm, chunk)
    r["tokens"] = r["posterior"].reshape(-1, BLOCK)[:, 1:].copy()
    return r


def acceptance_length(drafted, posterior) -> int:
    """[P2] 保证二: matches = (drafted == posterior); a = sum(cumprod(matches)).

    drafted = block[1:16] (the 15 drafts); posterior = post[0:15], where
    post[i] is the target's greedy token after block position i.
    """
    m = (np.asarray(drafted) == np.asarray(posterior)).astype(np.int64)
    return int(np.sum(np.cumprod(m)))


def verify_accept(hidden, w_lm, block_ids, len_before, out_tokens=None, out_cap=None,
                  chunk: int = 8192) -> dict:
    """Verification epilogue of one cycle ([P2] 单次前向验证 ⑤–⑧).

    hidden [B,T,H] final-normed target hidden states of [staged + 15 drafts];
    block_ids [B,T]; len_before [B] committed-token count before the cycle.
      posterior[b, i] = argmax_v logits[b, i, v]        (⑤, 保证一)
      a_b = sum(cumprod(block[b, 1:] == posterior[b, :15]))   (⑥, 保证二)
      commit block[b, 0..a_b] at out_tokens[b, len_before[b] + i]   (⑦)
      next_staged[b] = posterior[b, a_b]                (⑧; a_b = 15 is the bonus token)
      commit_len[b] = len_before[b] + 1 + a_b
    A sequence whose commit would pass ``out_cap`` is left uncommitted
    (flag ``overflow``), matching the library's error behaviour.
    """
    block_ids = np.asarray(block_ids)
    B, T = block_ids.shape
    H = np.asarray(hidden).shape[-1]
    am = lm_head_argmax(np.asarray(hidden).reshape(B * T, H), w_lm, chunk)
    post = am["posterior"].reshape(B, T)
    if out_tokens is None:
        cap = int(out_cap) if out_cap is not None else int(np.max(len_before)) + T
        out_tokens = np.zeros((B, cap), dtype=np.int32)
    out_tokens = np.array(out_tokens, dtype=np.int32, copy=True)
    cap = out_tokens.shape[1]
    accept = np.zeros(B, dtype=np.int32)
    next_staged = np.zeros(B, dtype=np.int32)
    commit_len = np.zeros(B, dtype=np.int32)
    overflow = np.zeros(B, dtype=bool)
    for b in range(B):
        a = acceptance_length(block_ids[b, 1:T], post[b, 0:T - 1])
        accept[b] = a
        start = int(len_before[b])
        if start + 1 + a > cap:
            overflow[b] = True
            commit_len[b] = start
            continue
        out_tokens[b, start:start + a + 1] = block_ids[b, 0:a + 1]
        next_staged[b] = post[b, a]
        commit_len[b] = start + 1 + a
    return {"posterior": post, "gap": am["gap"].reshape(B, T), "max": am["max"].reshape(B, T),
            "accept": accept, "next_staged": next_staged, "commit_len": commit_len,
            "out_tokens": out_tokens, "overflow": overflow}


def near_tie_mask(gap: np.ndarray, maxv: np.ndarray, rel: float = 1e-3) -> np.ndarray:
    """Positions whose top-2 gap is at most rel * |max logit| (excluded from the
    bit-exact comparison of token ids, and counted)."""
    return gap <= rel * np.abs(maxv)


# ---------------------------------------------------------------------------
# a4: KV-cache crop (and page reservation for the next block's rows)
# ---------------------------------------------------------------------------
def kv_crop_lengths(seq_len, new_len) -> tuple:
    """[P1] §3 / [P2] 保证三: after acceptance the cache keeps only the committed
    prefix: seq_len[b] <- new_len[b].  A request to grow (new_len > seq_len) or a
    negative length is invalid: that sequence is left unchanged and flagged."""
    seq_len = np.array(seq_len, dtype=np.int64, copy=True)
    new_len = np.asarray(new_len, dtype=np.int64)
    bad = (new_len > seq_len) | (new_len < 0)
    seq_len = np.where(bad, seq_len, new_len)
    return seq_len.astype(np.int32), bad


def kv_crop_paged(seq_len, page_table, free_pages: set, new_len, page_size: int) -> dict:
    """Paged crop: lengths as in :func:`kv_crop_lengths`; every mapped page whose
    first token index is >= new_len goes back to the free set and its table slot
    becomes -1.  The partially filled last page is kept.  (Reading: the pages do
    not describe paging; releasing whole pages beyond the length is the plain one.)"""
    table = np.array(page_table, dtype=np.int32, copy=True)
    free = set(free_pages)
    out_len, bad = kv_crop_lengths(seq_len, new_len)
    for b in range(table.shape[0]):
        if bad[b]:
            continue
        first_released = -(-int(out_len[b]) // page_size)
        for p in range(first_released, table.shape[1]):
            if table[b, p] >= 0:
                free.add(int(table[b, p]))
                table[b, p] = -1
    return {"seq_len": out_len, "page_table": table, "free": free, "bad": bad}


def pages_needed(write_pos, n_rows: int, page_size: int) -> list:
    """Page-table slots that must be mapped to write rows [pos, pos + n_rows)."""
    out = []
    for pos in np.asarray(write_pos):
        p0 = int(pos) // page_size
        p1 = (int(pos) + n_rows - 1) // page_size
        out.append(list(range(p0, p1 + 1)))
    return out
