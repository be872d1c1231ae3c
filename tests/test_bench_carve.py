"""The bench's single-buffer layout of a step's inputs and results (host
logic, no GPU): every tensor lies inside the buffer, 256-byte aligned, with
its own shape and dtype, and no two overlap."""
import torch

import bench


def test_carve_layout():
    specs = [((8, 1000), torch.bfloat16), ((8, 8), torch.float32), ((1000,), torch.uint8), ((3,), torch.float32),
             ((2, 5, 32), torch.uint8), ((1,), torch.bfloat16)]
    buf, views = bench.carve(torch, specs)
    assert buf.dtype == torch.uint8 and buf.dim() == 1
    base = buf.data_ptr()
    spans = []
    for v, (shape, dt) in zip(views, specs):
        assert tuple(v.shape) == shape and v.dtype == dt and v.is_contiguous()
        off = v.data_ptr() - base
        nbytes = v.numel() * v.element_size()
        assert off % 256 == 0 and off + nbytes <= buf.numel()
        spans.append((off, off + nbytes))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
    # writes through one view land in the buffer and nowhere else
    buf.zero_()
    views[2].fill_(7)
    off = views[2].data_ptr() - base
    assert int(buf[off:off + 1000].sum()) == 7000
    assert int(buf.sum()) == 7000
