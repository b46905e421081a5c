"""Host-side helpers of cycle.py (CPU only)."""
import torch

from block_diffusion_speculative_02_gb300.cycle import packed_tensors


def test_packed_tensors_are_aligned_disjoint_views():
    specs = [((3, 5), torch.bfloat16), ((7,), torch.int32), ((2, 16), torch.int32),
             ((1,), torch.float32)]
    flat, views = packed_tensors(specs, "cpu")
    assert [tuple(v.shape) for v in views] == [s for s, _ in specs]
    assert [v.dtype for v in views] == [d for _, d in specs]
    base = flat.data_ptr()
    spans = []
    for v in views:
        off = v.data_ptr() - base
        assert off % 256 == 0
        spans.append((off, off + v.numel() * v.element_size()))
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0
    assert spans[-1][1] <= flat.numel()
    for i, v in enumerate(views):          # writes through a view land in the flat buffer
        v.fill_(i + 1)
    for i, (v, (o0, o1)) in enumerate(zip(views, spans)):
        chunk = flat[o0:o1].view(v.dtype)
        assert torch.all(chunk == i + 1)
