"""GPU parity of dflash_verify_accept (LM head + argmax + acceptance + commit)
against the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from oracle.dflash_oracle import verify_accept as ref_verify
from synthetic import (CONFIG_BY_NAME, draw_accept_lengths, make_block_ids, make_cycle_inputs,
                       normal_bf16, unit_rms_rows_bf16)
from tests.gpu_helpers import Guarded, check_verify, dev_bf16, dev_i32

pytestmark = pytest.mark.gpu


def _dfl():
    import block_diffusion_speculative_02_gb300 as dfl
    return dfl


def gpu_verify(hidden_bits, w_bits, block_ids, len_before, out_cap, prev_out=None, calls=1,
               alias_len=False, sm_budget=0):
    dfl = _dfl()
    B = block_ids.shape[0]
    V, H = w_bits.shape
    dims = dfl.make_dims(B, H, 4, 4, 128, V, 1, 64, sm_budget=sm_budget)
    ws = dfl.alloc_workspace(dims)
    hid = dev_bf16(hidden_bits.reshape(B * 16, H))
    w = dev_bf16(w_bits)
    blk = dev_i32(block_ids)
    lb = dev_i32(len_before)
    guards = [Guarded((B, 16), torch.int32, fill=-5), Guarded((B,), torch.int32, fill=-5),
              Guarded((B,), torch.int32, fill=-5)]
    post, acc, nxt = (g.t for g in guards)
    cl = lb if alias_len else torch.full((B,), -5, dtype=torch.int32, device="cuda")
    out = dev_i32(prev_out if prev_out is not None else np.full((B, out_cap), -7, np.int32))
    results = []
    for _ in range(calls):
        if alias_len:
            cl.copy_(dev_i32(len_before))
        dfl.dflash_verify_accept(dims, hid, w, blk, cl if alias_len else lb, post, acc, nxt, cl,
                                 out, ws)
        torch.cuda.synchronize()
        for g in guards:
            g.check()
        results.append({"posterior": post.cpu().numpy(), "accept": acc.cpu().numpy(),
                        "next_staged": nxt.cpu().numpy(), "commit_len": cl.cpu().numpy(),
                        "out_tokens": out.cpu().numpy()})
    status = dfl.dflash_read_status(ws)
    return results, status


def _case(seed, B, H, V, accept_spec=("uniform",), len_before=None, out_cap=None):
    rng = np.random.default_rng(seed)
    hidden = unit_rms_rows_bf16(rng, (B, 16, H))
    w = normal_bf16(rng, (V, H), 0.02)
    ref0 = ref_verify(hidden, w, np.zeros((B, 16), np.int32), np.zeros(B, np.int32),
                      out_cap=64)
    acc = draw_accept_lengths(rng, accept_spec, B)
    blk = make_block_ids(rng, ref0["posterior"], acc, V)
    if len_before is None:
        len_before = rng.integers(0, 40, size=B).astype(np.int32)
    if out_cap is None:
        out_cap = int(len_before.max()) + 16
    return hidden, w, blk, len_before, out_cap


def _run_and_check(hidden, w, blk, len_before, out_cap, calls=1, alias_len=False):
    ref = ref_verify(hidden, w, blk, len_before, out_cap=out_cap,
                     out_tokens=np.full((blk.shape[0], out_cap), -7, np.int32))
    res, status = gpu_verify(hidden, w, blk, len_before, out_cap, calls=calls,
                             alias_len=alias_len)
    assert status == 0, status
    for r in res:
        info = check_verify(ref, r, len_before)
    for r in res[1:]:
        for k in r:
            assert np.array_equal(r[k], res[0][k]), k
    return ref, res[0], info


@pytest.mark.parametrize("seed,B,H,V", [
    (1, 1, 256, 4096),          # tiny cycle shapes
    (2, 3, 256, 50005),         # several 128-row tiles per CTA + partial tile + ragged vocab
    (3, 4, 512, 33000),         # 64 token columns
    (4, 17, 128, 9000),         # 272 token rows: the tiled path, a third row tile of 16
    (5, 32, 256, 20000),        # 512 token rows, ragged last vocabulary tile
    (6, 2, 128, 150),           # fewer vocabulary rows than SMs
])
def test_verify_parity_small(seed, B, H, V):
    hidden, w, blk, lb, cap = _case(seed, B, H, V)
    _, got, info = _run_and_check(hidden, w, blk, lb, cap, calls=2)
    print(info)


def test_verify_len_before_aliases_commit_len():
    hidden, w, blk, lb, cap = _case(7, 2, 256, 8192)
    _run_and_check(hidden, w, blk, lb, cap, alias_len=True)


def test_zero_hidden_picks_index_zero():
    B, H, V = 2, 256, 30000
    rng = np.random.default_rng(8)
    hidden = np.zeros((B, 16, H), np.uint16)
    w = normal_bf16(rng, (V, H), 0.02)
    blk = np.zeros((B, 16), np.int32)
    res, status = gpu_verify(hidden, w, blk, np.zeros(B, np.int32), 32)
    assert status == 0
    assert np.all(res[0]["posterior"] == 0)
    assert np.all(res[0]["accept"] == 15)          # every draft is token 0


def test_exact_tie_goes_to_the_lowest_index():
    """The row holding the maximum is duplicated far apart in the vocabulary
    (different CTAs): the lower copy must win."""
    B, H, V = 1, 256, 40000
    rng = np.random.default_rng(9)
    hidden = unit_rms_rows_bf16(rng, (B, 16, H))
    w = normal_bf16(rng, (V, H), 0.02)
    ref = ref_verify(hidden, w, np.zeros((B, 16), np.int32), np.zeros(B, np.int32), out_cap=32)
    for i, p in enumerate(ref["posterior"][0][:4]):
        lo = 100 + 7 * i
        w[lo] = w[p]
        w[V - 1 - i] = w[p]
    ref = ref_verify(hidden, w, np.zeros((B, 16), np.int32), np.zeros(B, np.int32), out_cap=32)
    res, _ = gpu_verify(hidden, w, np.zeros((B, 16), np.int32), np.zeros(B, np.int32), 32)
    for i in range(4):
        assert ref["posterior"][0][i] == 100 + 7 * i
        assert res[0]["posterior"][0][i] == 100 + 7 * i


def test_tiled_path_exact_ties_go_to_the_lowest_index():
    """Past 256 token rows the logits come from the tiled GEMM (256 vocabulary
    rows per tile).  Copies of a row's winner in an earlier tile, in the same
    tile and at the end of the vocabulary tie exactly; the lowest index wins."""
    B, H, V = 17, 256, 70001
    rng = np.random.default_rng(21)
    hidden = unit_rms_rows_bf16(rng, (B, 16, H))
    w = normal_bf16(rng, (V, H), 0.02)
    zeros, lb = np.zeros((B, 16), np.int32), np.zeros(B, np.int32)
    ref = ref_verify(hidden, w, zeros, lb, out_cap=32)
    want = {}
    for i in range(8):
        p = int(ref["posterior"][0][i])
        w[V - 1 - i] = w[p]                               # a later copy never wins
        if i < 4:
            lo = 100 + 7 * i                              # an earlier tile
        else:
            t0 = p // 256 * 256
            if p == t0:
                continue
            lo = t0 + (p - t0) // 2                       # earlier in the same tile
        w[lo] = w[p]
        want[i] = lo
    ref = ref_verify(hidden, w, zeros, lb, out_cap=32)
    res, status = gpu_verify(hidden, w, zeros, lb, 32)
    assert status == 0
    for i, lo in want.items():
        assert ref["posterior"][0][i] == lo
        assert res[0]["posterior"][0][i] == lo
    check_verify(ref, res[0], lb)


@pytest.mark.parametrize("B,H,V,budget", [(24, 256, 30011, 40), (32, 128, 9000, 7)])
def test_tiled_path_under_an_sm_budget(B, H, V, budget):
    """The tiled path confined to a few SMs (clusters of two within the
    budget) gives the same verification as on the whole device."""
    hidden, w, blk, lb, cap = _case(30 + B, B, H, V)
    full, st0 = gpu_verify(hidden, w, blk, lb, cap)
    part, st1 = gpu_verify(hidden, w, blk, lb, cap, sm_budget=budget)
    assert st0 == 0 and st1 == 0
    for k in full[0]:
        assert np.array_equal(full[0][k], part[0][k]), k
    ref = ref_verify(hidden, w, blk, lb, out_cap=cap,
                     out_tokens=np.full((B, cap), -7, np.int32))
    check_verify(ref, part[0], lb)


def test_overflow_and_bad_token_set_status_and_skip_commit():
    dfl = _dfl()
    hidden, w, blk, lb, cap = _case(10, 2, 256, 4096, accept_spec=("uniform",))
    blk[1, 5] = 10 ** 7                              # out of vocabulary
    lb = np.array([0, 30], np.int32)
    cap = 20                                         # sequence 1 cannot commit
    ref = ref_verify(hidden, w, blk, lb, out_tokens=np.full((2, cap), -7, np.int32))
    res, status = gpu_verify(hidden, w, blk, lb, cap)
    st = dfl.dflash.STATUS_BITS
    assert status & st["out_overflow"] and status & st["bad_token"]
    r = res[0]
    assert np.all(r["out_tokens"][1] == -7) and r["commit_len"][1] == -5 \
        and r["next_staged"][1] == -5
    assert r["accept"][1] == ref["accept"][1]
    check_verify({k: v[:1] for k, v in ref.items()}, {k: v[:1] for k, v in r.items()}, lb[:1])


@pytest.mark.parametrize("name", ["qwen3_4b_b1", "qwen3_8b_b1", "qwen3_8b_b32_paged",
                                  "qwen3_32b_b4_32k"])
def test_verify_parity_full_size(name):
    """The benchmark configurations at full size (vocabulary 151936)."""
    cfg = CONFIG_BY_NAME[name]
    inp = make_cycle_inputs(cfg)
    B = cfg.batch
    ref0 = ref_verify(inp.verify_hidden, inp.w_lm, np.zeros((B, 16), np.int32),
                      np.zeros(B, np.int32), out_cap=64)
    blk = make_block_ids(inp.rng_blocks, ref0["posterior"], inp.accept_draw, cfg.vocab)
    lb = np.full(B, 100, np.int32)
    ref, got, info = _run_and_check(inp.verify_hidden, inp.w_lm, blk, lb, 160)
    print(cfg.name, info, "accept", got["accept"])
