"""The library under CUDA-graph stream capture: a small step (both blockwise
formats, both fused reduces, the 7-hop ring chain with the early local copy,
a grouped MXFP8 launch and per-tensor scaling) is captured once, then
replayed on new inputs written in place.  Every replay equals an eager run
on the same inputs and the oracle."""
import numpy as np
import pytest
import torch

import gen
from gpu_util import assert_same, assert_same_f32, bits16, u8

pytestmark = pytest.mark.gpu

K = 8
N = 4096 * 5 + 77                 # several tiles and a ragged tail
MX = [(2, 256, 768), (1, 128, 96)]


@pytest.fixture(scope="module")
def w():
    import weight_transfer_gb300 as w
    return w


class Step:
    """Inputs and preallocated outputs of one small step, and its launches."""

    def __init__(self, w, dev):
        self.w = w
        nb = (N + 127) // 128
        self.bucket = [torch.empty(N, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        self.mx_in = [torch.empty((b, m, k), dtype=torch.bfloat16, device=dev) for b, m, k in MX]
        self.q = {f: [(torch.empty(N, dtype=torch.uint8, device=dev), torch.empty(nb, dtype=torch.float32, device=dev))
                      for _ in range(K)] for f in (0, 1)}
        self.red = {f: (torch.empty(N, dtype=torch.bfloat16, device=dev), torch.empty(N, dtype=torch.float32, device=dev))
                    for f in (0, 1)}
        self.hops = [(torch.empty(N, dtype=torch.uint8, device=dev), torch.empty(nb, dtype=torch.float32, device=dev))
                     for _ in range(K - 1)]
        self.ring_bf16 = torch.empty(N, dtype=torch.bfloat16, device=dev)
        self.mx_c = [torch.empty((b, m, k), dtype=torch.uint8, device=dev) for b, m, k in MX]
        self.mx_s = [torch.empty(max(w.mxfp8_swizzled_scale_bytes(b, m, k), 16), dtype=torch.uint8, device=dev)
                     for b, m, k in MX]
        self.tw_c = torch.empty(N, dtype=torch.uint8, device=dev)
        self.tw_sa = torch.empty(4, dtype=torch.float32, device=dev)

    def fill(self, seed):
        for r in range(K):
            self.bucket[r].copy_(gen.normal_bf16(N, 1e-3, seed=seed + r, outlier_p=1e-3, outlier_mult=100.0))
        for i, (b, m, k) in enumerate(MX):
            self.mx_in[i].copy_(gen.normal_bf16(b * m * k, 0.02, seed=seed + 50 + i).view(b, m, k))

    def launch(self):
        # the flags where they hold, as the bench's step uses them: the
        # bucket and the MXFP8 inputs are written by copies only; each reduce
        # reads codes from quantizes at least two launches back
        w = self.w
        ready = w.FP8Q_INPUTS_READY
        for f in (0, 1):
            for r in range(K):
                w.fp8q_quantize_blockwise_ex(self.bucket[r], f, ready, codes=self.q[f][r][0], scales=self.q[f][r][1])
        for f in (0, 1):
            w.fp8q_dequant_reduce_ex([c for c, _ in self.q[f]], [s for _, s in self.q[f]], f, ready,
                                     out_bf16=self.red[f][0], out_fp32=self.red[f][1])
        prev = self.q[0][0]
        for h in range(1, K):
            oc, os_ = self.hops[h - 1]
            hp = {"in_codes": prev[0], "in_scales": prev[1], "local": self.bucket[h], "out_codes": oc,
                  "out_scales": os_, "out_bf16": self.ring_bf16 if h == K - 1 else None}
            w.fp8q_ring_hop_group_ex([hp], 0, w.FP8Q_HOP_LOCAL_READY)
            prev = (oc, os_)
        w.mxfp8_quantize_swizzled_group_ex(self.mx_in, ready, codes=self.mx_c, scales=self.mx_s)
        w.fp8q_quantize_tensorwise(self.red[0][0], 0, codes=self.tw_c, scale_amax=self.tw_sa)

    def outputs(self):
        res = []
        for f in (0, 1):
            res += [u8(c) for c, _ in self.q[f]] + [s.cpu().numpy() for _, s in self.q[f]]
            res += [bits16(self.red[f][0]), self.red[f][1].cpu().numpy()]
        res += [u8(c) for c, _ in self.hops] + [s.cpu().numpy() for _, s in self.hops] + [bits16(self.ring_bf16)]
        res += [u8(c) for c in self.mx_c] + [s.cpu().numpy() for s in self.mx_s]
        res += [u8(self.tw_c), self.tw_sa[:2].cpu().numpy()]
        return res


def test_captured_step_replays_like_eager_and_oracle(w, orc):
    dev = torch.device("cuda")
    st = Step(w, dev)
    st.fill(1000)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):            # warm-up outside capture: first-call setup
        st.launch()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.launch()
    for seed in (2000, 3000):
        st.fill(seed)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        got = st.outputs()
        st.launch()                          # eager, same inputs
        torch.cuda.synchronize()
        eager = st.outputs()
        assert len(got) == len(eager)
        for i, (a, b) in enumerate(zip(got, eager)):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), f"output {i} differs from eager (seed {seed})"
        # and the oracle, on the ring chain, the reduces and MXFP8
        xs = [bits16(x) for x in st.bucket]
        for f in (0, 1):
            oq = [orc.quantize_blockwise(x, f) for x in xs]
            eb, ef = orc.dequant_reduce([c for c, _ in oq], [s for _, s in oq], f)
            assert_same(bits16(st.red[f][0]), eb, f"reduce bf16 fmt {f}")
            assert_same_f32(st.red[f][1].cpu().numpy(), ef, f"reduce fp32 fmt {f}")
        c, s = orc.quantize_blockwise(xs[0], 0)
        for h in range(1, K):
            c, s, b = orc.ring_hop(c, s, xs[h], 0)
            assert_same(u8(st.hops[h - 1][0]), c, f"hop {h} codes")
        assert_same(bits16(st.ring_bf16), b, "ring bf16")
        for i, (bb, m, k) in enumerate(MX):
            ec, es = orc.mxfp8_quantize_swizzled(bits16(st.mx_in[i]).ravel(), bb, m, k)
            assert_same(u8(st.mx_c[i]).ravel(), ec, f"mxfp8 codes {i}")
            assert_same(st.mx_s[i].cpu().numpy()[:es.size], es, f"mxfp8 scales {i}")


def test_captured_ring_allreduce_replays_like_eager_and_oracle(w, orc):
    # the simulated AllReduce (one grouped quantize, 7 grouped hops, the
    # all-gather decode: 9 launches from one C call) captured once, replayed
    # on new partials written in place; with and without the mean
    from test_gpu_ring_allreduce import oracle_allreduce
    P, n = 8, 8 * 512 * 11
    parts = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    res = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    ws = torch.empty(int(w.lib().fp8q_ring_allreduce_workspace_bytes(P, n)), dtype=torch.uint8, device="cuda")
    for mean in (False, True):
        def fill(seed):
            for r in range(P):
                parts[r].copy_(gen.normal_bf16(n, 1e-3, seed=seed + r, outlier_p=1e-3, outlier_mult=100.0))
        fill(10)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):        # first-call setup outside capture
            w.fp8q_ring_allreduce_sim(parts, "e4m3", results=res, workspace=ws, mean=mean)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            w.fp8q_ring_allreduce_sim(parts, "e4m3", results=res, workspace=ws, mean=mean)
        for seed in (20, 30):
            fill(seed)
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            got = [bits16(r) for r in res]
            want = oracle_allreduce(orc, [bits16(p) for p in parts], 0, mean)
            for r in range(P):
                assert_same(got[r], want, f"rank {r}, seed {seed}, mean {mean}")
        del g
