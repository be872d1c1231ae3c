"""The seeded input generator: determinism, chunk independence, statistics."""
import numpy as np

import gen


def test_deterministic_and_chunk_independent():
    a = gen.normal_f32(100_001, 1.0, seed=3, outlier_p=0.01, outlier_mult=7.0)
    b = gen.normal_f32(100_001, 1.0, seed=3, outlier_p=0.01, outlier_mult=7.0)
    assert np.array_equal(a, b)
    for lo, n in [(1, 10), (77_777, 22_224), (50_000, 1)]:
        c = gen.normal_f32(n, 1.0, seed=3, offset=lo, outlier_p=0.01, outlier_mult=7.0)
        assert np.array_equal(c, a[lo:lo + n])
    assert not np.array_equal(a[:1000], gen.normal_f32(1000, 1.0, seed=4))


def test_thread_count_does_not_change_bytes():
    old = gen.NTHREADS
    try:
        gen.NTHREADS = 1
        a = gen.normal_f32(300_000, 2.0, seed=9)
        gen.NTHREADS = 7
        b = gen.normal_f32(300_000, 2.0, seed=9)
    finally:
        gen.NTHREADS = old
    assert np.array_equal(a, b)


def test_normal_statistics():
    x = gen.normal_f32(2_000_000, 1e-3, seed=0).astype(np.float64)
    assert abs(x.mean()) < 5e-6
    assert abs(x.std() / 1e-3 - 1) < 3e-3
    assert abs((np.abs(x) < 1e-3).mean() - 0.6827) < 2e-3


def test_outlier_fraction_and_row_groups():
    base = gen.normal_f32(1_000_000, 1.0, seed=5)
    out = gen.normal_f32(1_000_000, 1.0, seed=5, outlier_p=1e-3, outlier_mult=100.0)
    sel = out != base
    assert abs(sel.mean() - 1e-3) < 2e-4
    assert np.allclose(out[sel], base[sel] * 100.0, rtol=1e-6)
    rows = gen.normal_f32(512 * 256, 1.0, seed=6, outlier_p=0.1, outlier_mult=50.0, outlier_group=256)
    plain = gen.normal_f32(512 * 256, 1.0, seed=6)
    scaled_rows = (rows != plain).reshape(512, 256).any(axis=1)
    assert ((rows != plain).reshape(512, 256)[scaled_rows]).mean() > 0.99
    assert 0.05 < scaled_rows.mean() < 0.15


def test_distinct_zero_blocks():
    zb = gen.vec_zero_blocks(0)
    assert zb.size == 64 and np.unique(zb).size == 64
    assert zb.max() < (gen.VEC_N + 127) // 128
    b = int(zb[0])
    chunk = gen.vec_chunk(0, b * 128 - 64, 256)
    v = chunk.float().numpy()
    assert (v[64:192] == 0).all() and (v[:64] != 0).any()


def test_bf16_cast_and_recipe_shapes():
    t = gen.normal_bf16(1000, 1.0, seed=1)
    assert t.dtype.is_floating_point and t.element_size() == 2
    assert gen.qwen3_layer_elements() == 622_854_144
    assert gen.qwen3_layer_elements() * gen.QWEN3_LAYERS == 29_896_998_912
    assert 767 * 1024 in gen.RING_SIZES_BYTES and (1 << 26) in gen.RING_SIZES_BYTES
