"""The transfer-buffer planner (host only): every weight travels in the same
batch as its scale, batches respect the cap unless one pair alone exceeds it,
order and alignment are kept.  The case from the MXFP8 refit review -- a
weight about 32x its scale closing a batch -- must not split the pair."""
import random

import pytest

OK = 0


@pytest.fixture(scope="module")
def w():
    from conftest import build_lib
    build_lib()
    import weight_transfer_gb300 as w
    return w


def r16(x):
    return (x + 15) // 16 * 16


def check_plan(pairs, cap, slots, sizes):
    assert len(slots) == len(pairs)
    used = {}
    prev = (-1, -1)
    for (c, s), (b, co, so) in zip(pairs, slots):
        assert co % 16 == 0 and so % 16 == 0
        assert so == co + r16(c)                       # scale right after its own codes
        assert (b, co) > prev                          # order kept
        prev = (b, co)
        end = so + r16(s)
        assert end <= sizes[b]
        used.setdefault(b, []).append((co, end))
    for b, spans in used.items():
        spans.sort()
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            assert a1 <= b0                           # no overlap inside a batch
        if sizes[b] > cap:
            assert len(spans) == 1                    # only an oversized pair exceeds the cap
    assert sorted(used) == list(range(len(sizes)))


def test_weight_closing_a_batch_keeps_its_scale(w):
    # MXFP8 pairs: codes m*k bytes, scales m*k/32 bytes (about 32:1)
    m, k = 2048, 4096
    pair = (m * k, m * k // 32)
    cap = 3 * m * k                                   # the third weight fits, its scale would not
    slots, sizes = w.fp8q_pack_plan([pair] * 5, cap)
    check_plan([pair] * 5, cap, slots, sizes)
    assert [s[0] for s in slots] == [0, 0, 1, 1, 2]


def test_oversized_pair_travels_alone(w):
    pairs = [(1000, 40), (10_000_000, 312_500), (500, 20), (600, 20)]
    slots, sizes = w.fp8q_pack_plan(pairs, 1 << 20)
    check_plan(pairs, 1 << 20, slots, sizes)
    assert [s[0] for s in slots] == [0, 1, 2, 2]
    assert sizes[1] == r16(10_000_000) + r16(312_500)


def test_random_plans(w):
    rng = random.Random(7)
    for _ in range(200):
        n = rng.randint(1, 60)
        pairs = [(rng.randint(0, 5000), rng.randint(0, 300)) for _ in range(n)]
        cap = rng.randint(16, 12000)
        slots, sizes = w.fp8q_pack_plan(pairs, cap)
        check_plan(pairs, cap, slots, sizes)


def test_plan_argument_errors(w):
    import ctypes
    L = w.lib()
    nb = ctypes.c_int(-1)
    assert L.fp8q_pack_plan(None, 0, 1024, None, None, ctypes.byref(nb)) == OK and nb.value == 0
    assert L.fp8q_pack_plan(None, 3, 1024, None, None, ctypes.byref(nb)) == 1          # FP8Q_ERR_NULL
    items = (w.fp8q_pack_item_t * 1)(w.fp8q_pack_item_t(10, 1))
    slots = (w.fp8q_pack_slot_t * 1)()
    sizes = (ctypes.c_uint64 * 1)()
    assert L.fp8q_pack_plan(items, 1, 8, slots, sizes, ctypes.byref(nb)) == 2          # cap below 16: SIZE
    assert L.fp8q_copy_segments(None, 97, None) == 2
