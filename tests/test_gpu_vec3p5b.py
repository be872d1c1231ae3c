"""The 3.5e9-element gradient vector at full size: 4 shards quantized to
e4m3 in one launch each (64-bit indexing across 3.5e9 elements), then the
4-shard fused reduce streamed in 2^27-element (256 MiB of bf16) chunks.

The oracle checks sampled 128-blocks one by one: every zero block, the
blocks on both sides of each chunk boundary, the last block, and random
ones.  The generator is counter-based, so the oracle regenerates each sampled
block's inputs on the host on its own."""
import numpy as np
import pytest
import torch

import gen
from gpu_util import assert_same, assert_same_f32, bits16, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    import weight_transfer_gb300 as w
    return w


def test_vec3p5b_quantize_and_streamed_reduce(w, orc):
    n, k, chunk = gen.VEC_N, gen.VEC_K, gen.VEC_CHUNK
    nb = (n + 127) // 128
    dev = torch.device("cuda")
    free, _ = torch.cuda.mem_get_info()
    need = k * (2 * n + n + 4 * nb) + 2 * n
    if free < need * 1.1:
        pytest.skip(f"needs {need / 2**30:.1f} GiB of device memory, {free / 2**30:.1f} free")
    codes, scales = [], []
    for r in range(k):
        x = torch.empty(n, dtype=torch.bfloat16, device=dev)
        for c0 in range(0, n, chunk):
            cnt = min(chunk, n - c0)
            x[c0:c0 + cnt].copy_(gen.vec_chunk(r, c0, cnt))
        c, s = w.fp8q_quantize_blockwise(x, "e4m3")
        codes.append(c)
        scales.append(s)
        del x
    torch.cuda.synchronize()
    out = torch.empty(n, dtype=torch.bfloat16, device=dev)
    for c0 in range(0, n, chunk):
        cnt = min(chunk, n - c0)
        b0 = c0 // 128
        w.fp8q_dequant_reduce([c[c0:c0 + cnt] for c in codes], [s[b0:b0 + (cnt + 127) // 128] for s in scales],
                              "e4m3", out_bf16=out[c0:c0 + cnt], want_fp32=False, n=cnt)
    torch.cuda.synchronize()

    rng = np.random.default_rng(35)
    picks = [rng.integers(0, nb, 1500)]
    for r in range(k):
        picks.append(gen.vec_zero_blocks(r).astype(np.int64))
    bounds = np.arange(chunk // 128, nb, chunk // 128)
    picks += [bounds, bounds - 1, np.array([0, nb - 1])]
    blocks = np.unique(np.concatenate(picks))
    idx = torch.from_numpy((blocks[:, None] * 128 + np.arange(128)[None, :]).ravel()).to(dev)
    bidx = torch.from_numpy(blocks).to(dev)
    dev_codes = [u8(c[idx]).reshape(-1, 128) for c in codes]
    dev_scales = [s[bidx].cpu().numpy() for s in scales]
    dev_out = bits16(out[idx]).reshape(-1, 128)
    zero_seen = 0
    for t, b in enumerate(blocks):
        oq = [orc.quantize_blockwise(bits16(gen.vec_chunk(r, int(b) * 128, 128)), 0) for r in range(k)]
        for r in range(k):
            assert_same(dev_codes[r][t], oq[r][0], f"shard {r} block {b} codes")
            assert_same_f32(dev_scales[r][t:t + 1], oq[r][1], f"shard {r} block {b} scale")
            zero_seen += oq[r][1][0] == 0.0
        eb, _ = orc.dequant_reduce([c for c, _ in oq], [s for _, s in oq], 0)
        assert_same(dev_out[t], eb, f"block {b} reduce")
    assert zero_seen >= gen.VEC_ZERO_BLOCKS * k       # every zero block was checked
    del codes, scales, out
    torch.cuda.empty_cache()
