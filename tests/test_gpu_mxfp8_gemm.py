"""The 128 x 4-tiled E8M0 scale layout, read by a real consumer.

The prequantized weights of "perf: Reduce MXFP8 refit weight-transfer
overheads" (Summary: the MXFP8 "shuffle" buffers; Results: the batched MoE
shuffle) exist so that a Blackwell block-scaled GEMM can consume them as
they arrive.  This file hands the codes and swizzled scales that
mxfp8_quantize_swizzled writes to this GPU's own block-scaled MXFP8 GEMM
(cuBLASLt behind torch._scaled_mm: float8_e4m3fn operands, float8_e8m0fnu
scales) and compares the product, element by element, with a float64 GEMM
of the oracle's dequantized operands.  The GEMM reads the scale bytes by the
hardware's own layout and the oracle by its formula, so the two agree only
if the formula is that layout.

Tolerance.  Every product of two decoded E4M3 values times two powers of two
is exact in binary32; the GEMM sums K of them in fp32.  Whatever the order,
recursive summation stays within gamma_K * sum |a_k b_k| of the exact sum,
gamma_K = K u / (1 - K u) (Higham, "Accuracy and Stability of Numerical
Algorithms", 2nd ed., Thm 4.4 / eq. 4.4).  u is taken as 2^-23, twice the
binary32 unit roundoff, so that an accumulator that truncates instead of
rounding still passes; add 2^-24 |C| for the fp32 output.

Sensitivity.  In the selector cases the second operand's row n is non-zero
only in the 32-block n mod (K/32), so each output element is one block of
the first operand times one block of the second: a scale read from the wrong
place changes it by a power of two, with nothing else to hide behind.  The
first operand's blocks carry independent random powers of two, and the last
test shows that three near-miss tile layouts fail the same check.
"""
import numpy as np
import pytest
import torch

import gen

pytestmark = pytest.mark.gpu

U = 2.0 ** -23


@pytest.fixture(scope="module")
def w():
    import weight_transfer_gb300 as w
    return w


def blocky(rows, k, seed):
    """N(0, 1) values, each 1 x 32 block scaled by its own power of two in
    [2^-12, 2^12]: neighbouring scales differ, so a misplaced one shows."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((rows, k)).astype(np.float32)
    z *= np.repeat(np.exp2(rng.integers(-12, 13, size=(rows, k // 32))).astype(np.float32), 32, axis=1)
    return torch.from_numpy(z).to(torch.bfloat16)


def selector(rows, k, seed):
    """Row n non-zero only in the 32-block n mod (k / 32)."""
    x = blocky(rows, k, seed).float()
    kb = k // 32
    keep = torch.zeros(rows, kb, dtype=torch.bool)
    keep[torch.arange(rows), torch.arange(rows) % kb] = True
    return (x * keep.repeat_interleave(32, dim=1)).to(torch.bfloat16)


def qwen_like(rows, k, seed):
    """The stack's weight distribution: N(0, 0.02^2), 1% of rows x50."""
    return gen.normal_bf16(rows * k, 0.02, seed=seed, outlier_p=0.01, outlier_mult=50.0,
                           outlier_group=k).view(rows, k)


def dequant(orc, codes, scales, rows, k):
    """float64 [rows, k] from the oracle's MXFP8 dequantization (exact: a
    decoded E4M3 value times a power of two)."""
    bits = orc.mxfp8_dequantize(codes.cpu().numpy().ravel(), scales.cpu().numpy(), 1, rows, k)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(rows, k)


def gemm(a_codes, a_scales, b_codes, b_scales, m, n, k):
    """C [m, n] = A [m, k] x B [n, k]^T on the block-scaled MXFP8 path."""
    A = a_codes.reshape(m, k).view(torch.float8_e4m3fn)
    B = b_codes.reshape(n, k).view(torch.float8_e4m3fn)
    C = torch._scaled_mm(A, B.t(), scale_a=a_scales.view(torch.float8_e8m0fnu),
                         scale_b=b_scales.view(torch.float8_e8m0fnu), out_dtype=torch.float32)
    torch.cuda.synchronize()
    return C.double().cpu().numpy()


def within(C, Ad, Bd, k):
    ref = Ad @ Bd.T
    gamma = k * U / (1 - k * U)
    bound = gamma * (np.abs(Ad) @ np.abs(Bd).T) + 2.0 ** -24 * np.abs(ref)
    err = np.abs(C - ref)
    return err <= bound, err, bound


def check_product(w, orc, a, b):
    m, k = a.shape
    n = b.shape[0]
    ac, asc = w.mxfp8_quantize_swizzled(a.cuda())
    bc, bsc = w.mxfp8_quantize_swizzled(b.cuda())
    ok, err, bound = within(gemm(ac, asc, bc, bsc, m, n, k), dequant(orc, ac, asc, m, k),
                            dequant(orc, bc, bsc, n, k), k)
    bad = np.argwhere(~ok)
    assert bad.size == 0, f"{len(bad)} of {ok.size} outside the bound, first {tuple(bad[0])}: " \
                          f"err {err[tuple(bad[0])]:.3e} > {bound[tuple(bad[0])]:.3e}"


@pytest.mark.parametrize("m,n,k", [(128, 128, 32), (256, 128, 128), (4096, 128, 2048), (200, 128, 96),
                                   (384, 256, 2048)])
def test_gemm_reads_each_weight_scale_where_the_layout_puts_it(w, orc, m, n, k):
    # first operand: the scales under test; second: one block per row
    check_product(w, orc, blocky(m, k, seed=m + k), selector(n, k, seed=n + k + 1))


@pytest.mark.parametrize("m,n,k", [(128, 256, 32), (128, 4096, 2048), (128, 208, 96)])
def test_gemm_reads_each_second_operand_scale_where_the_layout_puts_it(w, orc, m, n, k):
    # the GEMM wants the second operand's row count divisible by 16 (208 still
    # pads its last 128-row scale tile)
    check_product(w, orc, selector(m, k, seed=m + k + 2), blocky(n, k, seed=n + k + 3))


@pytest.mark.parametrize("tokens,out,k", [(256, 768, 2048), (128, 4096, 2048), (256, 2048, 768), (4096, 512, 2048)])
def test_gemm_of_prequantized_qwen3_shaped_weights(w, orc, tokens, out, k):
    # y = x W^T with W [out, in] prequantized as the stack's tensors are
    check_product(w, orc, qwen_like(tokens, k, seed=out + 17), qwen_like(out, k, seed=k + 19))


def test_gemm_of_a_batched_expert_tensor_and_a_grouped_layer(w, orc):
    # one [4, 768, 2048] expert batch and one attention matrix quantized in
    # one grouped launch; each expert's scales are its slice of the batch's
    # buffer (matrices concatenated), consumed by one GEMM per expert
    E, M, K, tokens = 4, 768, 2048, 128
    experts = torch.stack([qwen_like(M, K, seed=40 + e) for e in range(E)])
    q = qwen_like(512, K, seed=50)
    (ec, qc), (es, qs) = w.mxfp8_quantize_swizzled_group([experts.cuda(), q.cuda()])
    x = blocky(tokens, K, seed=60)
    xc, xs = w.mxfp8_quantize_swizzled(x.cuda())
    Xd = dequant(orc, xc, xs, tokens, K)
    per = w.mxfp8_swizzled_scale_bytes(1, M, K)
    assert es.numel() == E * per
    for e in range(E):
        c_e, s_e = ec[e], es[e * per:(e + 1) * per]
        ok, _, _ = within(gemm(xc, xs, c_e, s_e, tokens, M, K), Xd, dequant(orc, c_e, s_e, M, K), K)
        assert ok.all(), f"expert {e}: {int((~ok).sum())} elements outside the bound"
    ok, _, _ = within(gemm(xc, xs, qc, qs, tokens, 512, K), Xd, dequant(orc, qc, qs, 512, K), K)
    assert ok.all()


def _relayout(nat, m, kb, order):
    """Row-major [m, kb] E8M0 bytes laid out in 128 x 4 tiles with the
    (row tile a, column tile b, row-in-32 i, row group g, column c) axes
    emitted in `order`."""
    mp, kp = -(-m // 128) * 128, -(-kb // 4) * 4
    pad = np.zeros((mp, kp), np.uint8)
    pad[:m, :kb] = nat
    t = pad.reshape(mp // 128, 4, 32, kp // 4, 4)       # axes a, g, i, b, c
    axes = {"a": 0, "g": 1, "i": 2, "b": 3, "c": 4}
    return torch.from_numpy(np.ascontiguousarray(t.transpose([axes[x] for x in order])).reshape(-1)).cuda()


def test_gemm_rejects_near_miss_tile_layouts(w, orc):
    # the same scale bytes in three other arrangements: the GEMM then reads
    # wrong scales and the product leaves the bound, while the library's
    # arrangement (a, b, i, g, c) passes
    m, n, k = 256, 128, 256                           # 2 x 2 tiles of the first operand's scales
    a, b = blocky(m, k, seed=71), selector(n, k, seed=72)
    ac, asc = w.mxfp8_quantize_swizzled(a.cuda())
    bc, bsc = w.mxfp8_quantize_swizzled(b.cuda())
    nat = orc.mxfp8_unswizzle(asc.cpu().numpy(), 1, m, k).reshape(m, k // 32)
    Ad, Bd = dequant(orc, ac, asc, m, k), dequant(orc, bc, bsc, n, k)
    same = _relayout(nat, m, k // 32, "abigc")
    assert torch.equal(same, asc)
    assert within(gemm(ac, same, bc, bsc, m, n, k), Ad, Bd, k)[0].all()
    for order in ("abgic", "abicg", "baigc"):         # row-major tile, swapped inner pair, column tiles first
        alt = _relayout(nat, m, k // 32, order)
        ok = within(gemm(ac, alt, bc, bsc, m, n, k), Ad, Bd, k)[0]
        assert not ok.all(), f"layout {order} was not told apart"
        # the column-tiles-first order moves half of the scales (2 of 4 tiles)
        assert (~ok).mean() > 0.25, f"layout {order}: only {(~ok).mean():.2%} of the outputs moved"
