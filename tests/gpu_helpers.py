"""Helpers shared by the GPU parity tests: moving seeded host inputs to the
device and comparing token outputs under the near-tie rule."""
import numpy as np
import torch

from oracle.dflash_oracle import near_tie_mask


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> CUDA bfloat16 tensor with the same bits."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def dev_i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_verify(ref: dict, gpu: dict, len_before, rel: float = 1e-3) -> dict:
    """Token outputs must match the oracle exactly, except positions whose
    oracle top-2 gap is <= rel * |max logit| (counted).  A sequence whose first
    near-tie position lies within its accepted prefix (positions 0..a) has its
    acceptance, commit and next staged token excluded too (counted)."""
    tie = near_tie_mask(ref["gap"], ref["max"], rel)
    ok = ~tie
    assert np.array_equal(gpu["posterior"][ok], ref["posterior"][ok]), \
        np.argwhere((gpu["posterior"] != ref["posterior"]) & ok)[:10]
    B = tie.shape[0]
    excluded_seqs = 0
    for b in range(B):
        a = int(ref["accept"][b])
        ties = np.nonzero(tie[b])[0]
        if len(ties) and ties[0] <= a:
            excluded_seqs += 1
            continue
        assert gpu["accept"][b] == a, (b, gpu["accept"][b], a)
        assert gpu["next_staged"][b] == ref["next_staged"][b], b
        assert gpu["commit_len"][b] == ref["commit_len"][b], b
        lb = int(len_before[b])
        assert np.array_equal(gpu["out_tokens"][b, lb:lb + a + 1],
                              ref["out_tokens"][b, lb:lb + a + 1]), b
    return {"tie_positions": int(tie.sum()), "excluded_seqs": excluded_seqs}


def assert_close_bf16(got: np.ndarray, ref: np.ndarray, max_abs: float = 2e-2,
                      rel_l2: float = 1e-2) -> dict:
    """Float outputs: max-abs and relative-L2 error against the fp64 oracle."""
    err = np.abs(got - ref)
    mx = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(ref)) or 1.0
    rl2 = float(np.linalg.norm(got - ref)) / denom
    assert mx <= max_abs, (mx, np.unravel_index(int(err.argmax()), err.shape))
    assert rl2 <= rel_l2, rl2
    return {"max_abs": mx, "rel_l2": rl2, "max_ref": float(np.abs(ref).max()) if ref.size else 0}


def half_ulp_bf16(ref: np.ndarray) -> np.ndarray:
    """Half a bf16 unit in the last place at |ref| (7 fraction bits):
    2^(e - 8) for |ref| in [2^e, 2^(e + 1)); 0 where ref is 0."""
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def assert_close_bf16_wide(got: np.ndarray, ref: np.ndarray, max_abs: float = 2e-2,
                           rel_l2: float = 1e-2) -> dict:
    """The float bar for bf16 outputs that may pass 8 in magnitude: an element
    with |ref| < 8 is within max_abs of float64, one with |ref| >= 8 within
    max_abs plus half a bf16 ulp of ref (rounding the result to bf16 alone
    costs up to that much there); relative-L2 as usual.  Returns the error
    figures and how many elements took the wider bound."""
    err = np.abs(got - ref)
    wide = np.abs(ref) >= 8
    bound = max_abs + np.where(wide, half_ulp_bf16(ref), 0.0)
    bad = err > bound
    assert not bad.any(), (int(bad.sum()), float(err[bad].max()),
                           np.unravel_index(int(np.argmax(err - bound)), err.shape))
    denom = float(np.linalg.norm(ref)) or 1.0
    rl2 = float(np.linalg.norm(got - ref)) / denom
    assert rl2 <= rel_l2, rl2
    return {"max_abs": float(err.max()) if err.size else 0.0, "rel_l2": rl2,
            "max_ref": float(np.abs(ref).max()) if ref.size else 0.0,
            "n_wide": int(wide.sum()),
            "max_abs_narrow": float(err[~wide].max()) if (~wide).any() else 0.0}


class Guarded:
    """A device output buffer with guard bands on both sides (filled with the
    byte 0xA5); ``t`` is the buffer proper, ``check()`` asserts that nothing
    was written into the bands."""

    CANARY = 0xA5

    def __init__(self, shape, dtype, fill=None, guard_bytes=4096):
        es = torch.empty((), dtype=dtype).element_size()
        n = 1
        for x in shape:
            n *= int(x)
        self.g = guard_bytes // es
        self.n = n
        self.es = es
        self.raw = torch.empty(n + 2 * self.g, dtype=dtype, device="cuda")
        self.raw.view(torch.uint8).fill_(self.CANARY)
        self.t = self.raw[self.g:self.g + n].view(*shape)
        if fill is not None:
            self.t.fill_(fill)

    def check(self):
        b = self.raw.view(torch.uint8)
        head = b[:self.g * self.es]
        tail = b[(self.g + self.n) * self.es:]
        assert bool((head == self.CANARY).all()), "write before the output buffer"
        assert bool((tail == self.CANARY).all()), "write past the output buffer"
