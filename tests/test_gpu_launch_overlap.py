"""Programmatic dependent launch: long chains of launches, each reading what
the launch before it wrote, with no host synchronization in between.  The
results are byte-identical with the overlap on and off and equal the
oracle's, so every kernel waits for its predecessor before it reads."""
import numpy as np
import pytest
import torch

import gen
from gpu_util import assert_same, assert_same_f32, bits16, u8

pytestmark = pytest.mark.gpu

ROUNDS = 3


@pytest.fixture(scope="module")
def w():
    import weight_transfer_gb300 as w
    return w


def run_chain(w, parts, fmt):
    """ROUNDS rounds of: blockwise quantize of the running bf16 vector, a
    7-hop ring chain over the partials, the k = 8 reduce of the hop outputs,
    and a tensorwise quantize of the reduced bf16; the ring's bf16 result
    feeds the next round.  Returns every output, on the device."""
    outs = []
    x = parts[0]
    for _ in range(ROUNDS):
        c, s = w.fp8q_quantize_blockwise(x, fmt)
        hops = [(c, s)]
        b = None
        for h in range(1, len(parts)):
            c, s, b = w.fp8q_ring_hop(c, s, parts[h], fmt, want_bf16=h == len(parts) - 1)
            hops.append((c, s))
        rb, rf = w.fp8q_dequant_reduce([hc for hc, _ in hops], [hs for _, hs in hops], fmt)
        tc, tsa = w.fp8q_quantize_tensorwise(rb, fmt)
        outs.append((hops, b, rb, rf, tc, tsa))
        x = b
    return outs


def host(outs):
    res = []
    for hops, b, rb, rf, tc, tsa in outs:
        res.append(([(u8(c), s.cpu().numpy()) for c, s in hops], bits16(b), bits16(rb), rf.cpu().numpy(), u8(tc),
                    tsa.cpu().numpy()))
    return res


def oracle_chain(orc, parts, fmt):
    res = []
    x = parts[0]
    for _ in range(ROUNDS):
        c, s = orc.quantize_blockwise(x, fmt)
        hops = [(c, s)]
        for h in range(1, len(parts)):
            c, s, b = orc.ring_hop(c, s, parts[h], fmt)
            hops.append((c, s))
        rb, rf = orc.dequant_reduce([hc for hc, _ in hops], [hs for _, hs in hops], fmt)
        tc, tsc, tam = orc.quantize_tensorwise(rb, fmt)
        res.append((hops, b, rb, rf, tc, np.array([tsc, tam], np.float32)))
        x = b
    return res


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("n", [4096 * 3 + 77, 1 << 20, (1 << 22) + 4096])
def test_dependent_chain_overlap_on_off(w, orc, fmt, n):
    hparts = [gen.ring_partial(r, n) for r in range(gen.RING_PARTIALS)]
    parts = [p.cuda() for p in hparts]
    prev = w.fp8q_set_launch_overlap(True)
    try:
        on = host(run_chain(w, parts, fmt))
        w.fp8q_set_launch_overlap(False)
        off = host(run_chain(w, parts, fmt))
    finally:
        w.fp8q_set_launch_overlap(prev)
    ref = oracle_chain(orc, [bits16(p) for p in hparts], fmt)
    for r in range(ROUNDS):
        for got, tag in ((on[r], "on"), (off[r], "off")):
            hops, b, rb, rf, tc, tsa = got
            rhops, rb_b, rrb, rrf, rtc, rtsa = ref[r]
            for h, ((c, s), (oc, os_)) in enumerate(zip(hops, rhops)):
                assert_same(c, oc, f"{tag} round {r} hop {h} codes")
                assert_same_f32(s, os_, f"{tag} round {r} hop {h} scales")
            assert_same(b, rb_b, f"{tag} round {r} ring bf16")
            assert_same(rb, rrb, f"{tag} round {r} reduce bf16")
            assert_same_f32(rf, rrf, f"{tag} round {r} reduce f32")
            assert_same(tc, rtc, f"{tag} round {r} tensorwise codes")
            assert_same_f32(tsa, rtsa, f"{tag} round {r} tensorwise scale, amax")


def test_switch_returns_previous(w):
    prev = w.fp8q_set_launch_overlap(True)
    try:
        assert w.fp8q_set_launch_overlap(False) is True
        assert w.fp8q_set_launch_overlap(True) is False
    finally:
        w.fp8q_set_launch_overlap(prev)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("n", [4096 * 5 + 300, (1 << 21) + 128 * 7])
def test_hop_chain_local_ready(w, orc, fmt, n):
    # the 7-hop chain with each hop's local partial read before the previous
    # hop has finished (FP8Q_HOP_LOCAL_READY): the partials are written by
    # the host copy only; the incoming codes are the previous hop's output
    hparts = [gen.ring_partial(r, n) for r in range(gen.RING_PARTIALS)]
    parts = [p.cuda() for p in hparts]
    torch.cuda.synchronize()
    res = {}
    for flags in (w.FP8Q_HOP_LOCAL_READY, 0):
        c, s = w.fp8q_quantize_blockwise(parts[0], fmt)
        hops = []
        for h in range(1, len(parts)):
            (c, s, b), = w.fp8q_ring_hop_group_ex([{"in_codes": c, "in_scales": s, "local": parts[h],
                                                    "want_bf16": h == len(parts) - 1}], fmt, flags)
            hops.append((c, s))
        res[flags] = ([(u8(hc), hs.cpu().numpy()) for hc, hs in hops], bits16(b))     # read back after the chain
    c, s = orc.quantize_blockwise(bits16(hparts[0]), fmt)
    for h in range(1, gen.RING_PARTIALS):
        c, s, eb = orc.ring_hop(c, s, bits16(hparts[h]), fmt)
        for flags, (hops, _) in res.items():
            assert_same(hops[h - 1][0], c, f"flags {flags} hop {h} codes")
            assert_same_f32(hops[h - 1][1], s, f"flags {flags} hop {h} scales")
    for flags, (_, b) in res.items():
        assert_same(b, eb, f"flags {flags} final bf16")


def test_ddp_ring_chain_as_the_bench_launches_it(w, orc):
    # full size: the 8 DDP shards in one [8, n] allocation, hop 0 = the e4m3
    # quantize of shard 0 (part of the one-launch bucket quantize), hops 1..7
    # grouped calls of one with the early local copy, launched back to back,
    # the last with the bf16 output; every hop checked element by element
    n, k = gen.DDP_N, gen.DDP_K
    host = [gen.ddp_shard(r) for r in range(k)]
    bucket = torch.empty((k, n), dtype=torch.bfloat16, device="cuda")
    for r in range(k):
        bucket[r].copy_(host[r])
    qc, qs = w.fp8q_quantize_blockwise(bucket.view(-1), 0)
    prev = (qc[:n], qs[:n // 128])
    outs = []
    last = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    for h in range(1, k):
        hp = {"in_codes": prev[0], "in_scales": prev[1], "local": bucket[h],
              "out_bf16": last if h == k - 1 else None}
        (c, s, _), = w.fp8q_ring_hop_group_ex([hp], 0, w.FP8Q_HOP_LOCAL_READY)
        outs.append((c, s))
        prev = (c, s)
    got = [(u8(c), s.cpu().numpy()) for c, s in outs]
    c, s = orc.quantize_blockwise(bits16(host[0]), 0)
    for h in range(1, k):
        c, s, eb = orc.ring_hop(c, s, bits16(host[h]), 0)
        assert_same(got[h - 1][0], c, f"hop {h} codes")
        assert_same_f32(got[h - 1][1], s, f"hop {h} scales")
    assert_same(bits16(last), eb, "final bf16")


def test_step_with_inputs_ready(w, orc):
    # the bench step's order with FP8Q_INPUTS_READY wherever it holds: both
    # quantizes read the bucket (written by copies), each reduce reads codes
    # written two launches back, the MXFP8 group reads weights written by a
    # copy; results equal the unflagged run and the oracle
    k, n = 8, 4096 * 9 + 128 * 3 + 77
    host = [gen.normal_bf16(n, 1e-3, seed=900 + r, outlier_p=1e-3, outlier_mult=100.0) for r in range(k)]
    mx_shapes = [(2, 256, 768), (1, 384, 96)]
    mx_host = [gen.normal_bf16(b * m * kk, 0.02, seed=950 + i).view(b, m, kk) for i, (b, m, kk) in enumerate(mx_shapes)]
    shards = [h.cuda() for h in host]
    mx_in = [h.cuda() for h in mx_host]
    torch.cuda.synchronize()
    res = {}
    for flags in (w.FP8Q_INPUTS_READY, 0):
        q = {f: [w.fp8q_quantize_blockwise_ex(x, f, flags) for x in shards] for f in (0, 1)}
        red = {f: w.fp8q_dequant_reduce_ex([c for c, _ in q[f]], [s for _, s in q[f]], f, flags) for f in (0, 1)}
        mc, ms = w.mxfp8_quantize_swizzled_group_ex(mx_in, flags)
        torch.cuda.synchronize()
        res[flags] = ([u8(c) for f in (0, 1) for c, _ in q[f]], [bits16(red[f][0]) for f in (0, 1)],
                      [red[f][1].cpu().numpy() for f in (0, 1)], [u8(c) for c in mc], [u8(s) for s in ms])
    a, b = res[w.FP8Q_INPUTS_READY], res[0]
    for x, y in zip(a, b):
        for i, (p_, q_) in enumerate(zip(x, y)):
            assert np.array_equal(p_.view(np.uint8), q_.view(np.uint8)), f"flagged run differs ({i})"
    for f in (0, 1):
        oq = [orc.quantize_blockwise(bits16(h), f) for h in host]
        eb, ef = orc.dequant_reduce([c for c, _ in oq], [s for _, s in oq], f)
        assert_same(a[1][f], eb, f"reduce bf16 fmt {f}")
        assert_same_f32(a[2][f], ef, f"reduce fp32 fmt {f}")
    for i, (bb, m, kk) in enumerate(mx_shapes):
        ec, es = orc.mxfp8_quantize_swizzled(bits16(mx_host[i]).ravel(), bb, m, kk)
        assert_same(a[3][i].ravel(), ec, f"mxfp8 codes {i}")
        assert_same(a[4][i][:es.size], es, f"mxfp8 scales {i}")
