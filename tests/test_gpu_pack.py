"""Packing MXFP8 weights with their scales into capped transfer buffers
with one copy launch per buffer, and unpacking them on the other side."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    import weight_transfer_gb300 as w
    return w


def test_pack_and_unpack_round_trip(w):
    rng = np.random.default_rng(3)
    shapes = [(768, 2048), (2048, 768), (512, 2048), (96, 64), (4096, 2048), (1, 32), (128, 4096)]
    codes = [torch.from_numpy(rng.integers(0, 256, m * k, dtype=np.uint8)).cuda() for m, k in shapes]
    scales = [torch.from_numpy(rng.integers(0, 256, w.mxfp8_swizzled_scale_bytes(1, m, k), dtype=np.uint8)).cuda()
              for m, k in shapes]
    pairs = [(c.numel(), s.numel()) for c, s in zip(codes, scales)]
    cap = 4 << 20
    slots, sizes = w.fp8q_pack_plan(pairs, cap)
    bufs = [torch.full((sz,), 0xEE, dtype=torch.uint8, device="cuda") for sz in sizes]
    for b in range(len(sizes)):
        segs = []
        for (bt, co, so), c, s in zip(slots, codes, scales):
            if bt == b:
                segs += [(c, bufs[b][co:co + c.numel()]), (s, bufs[b][so:so + s.numel()])]
        w.fp8q_copy_segments(segs)
    # the expected buffers, assembled on the host from the plan
    for b in range(len(sizes)):
        want = np.full(sizes[b], 0xEE, np.uint8)
        for (bt, co, so), c, s in zip(slots, codes, scales):
            if bt == b:
                want[co:co + c.numel()] = c.cpu().numpy()
                want[so:so + s.numel()] = s.cpu().numpy()
        assert np.array_equal(bufs[b].cpu().numpy(), want), f"buffer {b}"
    # receiver: scatter back into fresh tensors, all pairs of a batch in one launch
    out_c = [torch.zeros_like(c) for c in codes]
    out_s = [torch.zeros_like(s) for s in scales]
    for b in range(len(sizes)):
        segs = []
        for (bt, co, so), c, s, oc, os_ in zip(slots, codes, scales, out_c, out_s):
            if bt == b:
                segs += [(bufs[b][co:co + c.numel()], oc), (bufs[b][so:so + s.numel()], os_)]
        w.fp8q_copy_segments(segs)
    torch.cuda.synchronize()
    for c, s, oc, os_ in zip(codes, scales, out_c, out_s):
        assert torch.equal(c, oc) and torch.equal(s, os_)


def test_copy_segments_odd_sizes(w):
    src = torch.arange(300_017, dtype=torch.int32, device="cuda").to(torch.uint8)
    dst = torch.zeros(300_032, dtype=torch.uint8, device="cuda")
    w.fp8q_copy_segments([(src[:16 * 1000], dst[:16 * 1000]), (src[16 * 1000:], dst[16 * 1000:300_017])])
    torch.cuda.synchronize()
    assert torch.equal(dst[:300_017], src) and int(dst[300_017:].sum()) == 0
