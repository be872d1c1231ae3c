"""(b) Fused dequant-reduce, single-shard dequantize and the unfused
comparator on the GPU, against the oracle, bit for bit (the stated bar of
1 bf16 ulp / 1e-6 relative is implied)."""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import gen
from gpu_util import Guarded, assert_same, assert_same_f32, bf16_from_bits, bits16, u8, varied_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    import weight_transfer_gb300 as w
    return w


def random_shards(k, n, fmt, seed):
    """Arbitrary finite codes and scales spread over many binades (incl. 0
    and subnormal scales) -- stresses every decode and rounding path."""
    rng = np.random.default_rng(seed)
    nb = (n + 127) // 128
    codes, scales = [], []
    for r in range(k):
        c = rng.integers(0, 256, n, dtype=np.uint8)
        if fmt == 0:
            c[(c & 0x7F) == 0x7F] = 0x11
        else:
            c[(c & 0x7C) == 0x7C] = 0x12
        s = (10.0 ** rng.uniform(-40, 30, nb)).astype(np.float32)
        s[rng.random(nb) < 0.05] = 0.0
        codes.append(c)
        scales.append(s)
    return codes, scales


def gpu_reduce(w, codes, scales, fmt, want_bf16=True, want_fp32=True, unfused=False):
    n = codes[0].size
    dc = [torch.from_numpy(c).cuda() for c in codes]
    ds = [torch.from_numpy(s).cuda() for s in scales]
    gb = Guarded(n, torch.bfloat16) if want_bf16 else None
    gf = Guarded(n, torch.float32) if want_fp32 else None
    fn = w.fp8q_dequant_reduce_unfused if unfused else w.fp8q_dequant_reduce
    fn(dc, ds, fmt, out_bf16=gb.t if gb else None, out_fp32=gf.t if gf else None,
       want_bf16=want_bf16, want_fp32=want_fp32)
    torch.cuda.synchronize()
    for g in (gb, gf):
        if g is not None:
            assert g.intact(), "write outside the output buffer"
    return (bits16(gb.t) if gb else None), (gf.t.cpu().numpy() if gf else None)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("k", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("n", [1, 15, 16, 17, 128, 129, 4096 + 17, 100_003])
def test_reduce_random_shards(w, orc, fmt, k, n):
    codes, scales = random_shards(k, n, fmt, seed=1000 * k + n + fmt)
    ob, of = gpu_reduce(w, codes, scales, fmt)
    eb, ef = orc.dequant_reduce(codes, scales, fmt)
    assert_same_f32(of, ef, "fp32")
    assert_same(ob, eb, "bf16")


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("mode", ["bf16", "fp32"])
def test_reduce_single_output(w, orc, fmt, mode):
    codes, scales = random_shards(4, 5000, fmt, seed=7 + fmt)
    ob, of = gpu_reduce(w, codes, scales, fmt, want_bf16=mode == "bf16", want_fp32=mode == "fp32")
    eb, ef = orc.dequant_reduce(codes, scales, fmt)
    if mode == "bf16":
        assert of is None
        assert_same(ob, eb, "bf16")
    else:
        assert ob is None
        assert_same_f32(of, ef, "fp32")


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("k", [2, 8])
def test_unfused_is_bit_identical(w, orc, fmt, k):
    codes, scales = random_shards(k, 50_001, fmt, seed=k + 50)
    fb, ff = gpu_reduce(w, codes, scales, fmt)
    ub, uf = gpu_reduce(w, codes, scales, fmt, unfused=True)
    assert_same_f32(uf, ff, "fp32")
    assert_same(ub, fb, "bf16")


@pytest.mark.parametrize("fmt", [0, 1])
def test_dequantize_single_shard(w, orc, fmt):
    codes, scales = random_shards(1, 70_001, fmt, seed=3 + fmt)
    c = torch.from_numpy(codes[0]).cuda()
    s = torch.from_numpy(scales[0]).cuda()
    ob, of = w.fp8q_dequantize(c, s, fmt, want_bf16=True, want_fp32=True)
    eb, ef = orc.dequantize(codes[0], scales[0], fmt)
    assert_same_f32(of.cpu().numpy(), ef, "fp32")
    assert_same(bits16(ob), eb, "bf16")


def test_pr1_config_end_to_end(w, orc):
    # two 1,048,576-value shards: e4m3 quantize then k = 2 reduce -> bf16
    xs = [gen.pr1_shard(r) for r in range(2)]
    dq = [w.fp8q_quantize_blockwise(x.cuda(), "e4m3") for x in xs]
    ob, _ = w.fp8q_dequant_reduce([c for c, _ in dq], [s for _, s in dq], "e4m3", want_fp32=False)
    oq = [orc.quantize_blockwise(bits16(x), 0) for x in xs]
    eb, _ = orc.dequant_reduce([c for c, _ in oq], [s for _, s in oq], 0)
    assert_same(bits16(ob), eb, "bf16")


@pytest.mark.parametrize("fmt", [0, 1])
def test_ddp_bucket_config_end_to_end(w, orc, fmt):
    # 8 shards of 13,107,200: quantize each, fused reduce -> bf16 and fp32,
    # and the unfused comparator on the same codes
    xs = [gen.ddp_shard(r) for r in range(gen.DDP_K)]
    dq = [w.fp8q_quantize_blockwise(x.cuda(), fmt) for x in xs]
    ob, of = w.fp8q_dequant_reduce([c for c, _ in dq], [s for _, s in dq], fmt)
    ub, uf = w.fp8q_dequant_reduce_unfused([c for c, _ in dq], [s for _, s in dq], fmt)
    with cf.ThreadPoolExecutor(8) as ex:
        oq = list(ex.map(lambda x: orc.quantize_blockwise(bits16(x), fmt), xs))
    for r in range(gen.DDP_K):
        assert_same(u8(dq[r][0]), oq[r][0], f"codes {r}")
    eb, ef = orc.dequant_reduce([c for c, _ in oq], [s for _, s in oq], fmt)
    assert_same_f32(of.cpu().numpy(), ef, "fp32")
    assert_same(bits16(ob), eb, "bf16")
    assert_same_f32(uf.cpu().numpy(), ef, "unfused fp32")
    assert_same(bits16(ub), eb, "unfused bf16")


def test_reduce_empty(w):
    c = torch.empty(0, dtype=torch.uint8, device="cuda")
    s = torch.empty(1, dtype=torch.float32, device="cuda")
    ob, of = w.fp8q_dequant_reduce([c, c], [s, s], "e4m3", n=0)
    assert ob.numel() == 0 and of.numel() == 0
