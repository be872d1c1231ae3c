// A ring AllReduce carried on the FP8 wire format, with all P ranks held on
// one GPU (host-side scheduling of the library's own kernels).
//
// "FP8 Transmission Optimization for VLA Training", section "FP8
// Transmission Optimization and Bottlenecks" (gradient collectives sent as
// blockwise e4m3/e5m2, ring-based approaches) and "How to Speed Up VLA
// Training Step by Step", PCIe paragraph (a ring AllReduce moves
// 2 (P-1)/P of the gradient bytes per GPU: 12.25 GB for 7 GB on 8 GPUs).
//
// Schedule (chunk c = elements [c m, (c+1) m), m = n / P):
//   reduce-scatter  step 0: rank i quantizes its chunk i and sends it on (the
//                   P quantizations are one grouped launch);
//                   step s = 1 .. P-1: rank i makes one ring hop on the
//                   message from rank i-1 (chunk (i-s) mod P) with its own
//                   chunk; the P hops of a step are one grouped launch.
//                   After step P-1 rank i holds chunk (i+1) mod P summed
//                   over all ranks, as codes and scales.
//   all-gather      the P reduced chunks travel the ring unchanged (codes and
//                   scales are the wire format); every rank dequantizes all
//                   of them, so every rank ends with the same bf16 vector
//                   (optionally divided by P: the mean).
// On one GPU the "send" is the next rank reading the sender's buffer; the
// bytes that would cross the wire are counted and returned.  The gathered
// codes are then one buffer that every rank reads, so the all-gather decode
// is one launch that decodes each tile once and writes all P results.
#include "fp8q_host.cuh"

namespace {

size_t round16(size_t b) { return (b + 15) & ~(size_t)15; }

// Workspace layout: message slots [2][P] (codes m, then scales) and the
// reduced vector (codes n, then scales n/128) in chunk order.
struct Layout {
    size_t m, slot, msg_codes, msg_scales, final_codes, final_scales, total;
};

Layout layout_of(int ranks, size_t n) {
    Layout L;
    L.m = n / (size_t)ranks;
    L.msg_codes = round16(L.m);
    L.msg_scales = round16(4 * (L.m / 128));
    L.slot = L.msg_codes + L.msg_scales;
    L.final_codes = 2 * (size_t)ranks * L.slot;
    L.final_scales = L.final_codes + round16(n);
    L.total = L.final_scales + round16(4 * (n / 128));
    return L;
}

}  // namespace

extern "C" size_t fp8q_ring_allreduce_workspace_bytes(int ranks, size_t n) {
    if (ranks < 2 || ranks > FP8Q_MAX_HOP_GROUP || n == 0 || n % (512 * (size_t)ranks) != 0) return 0;
    return layout_of(ranks, n).total;
}

extern "C" fp8q_status_t fp8q_ring_allreduce_sim_ex(const void* const* partials, void* const* results, int ranks,
                                                    size_t n, fp8q_format_t fmt, void* workspace,
                                                    size_t workspace_bytes, uint64_t* wire_bytes, unsigned int flags,
                                                    fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_ring_allreduce_sim_ex");
    using namespace fp8q;
    if (flags & ~FP8Q_ALLREDUCE_MEAN) return FP8Q_ERR_FLAGS;
    if (!valid_fmt(fmt)) return FP8Q_ERR_FORMAT;
    if (ranks < 2 || ranks > FP8Q_MAX_HOP_GROUP) return FP8Q_ERR_K;
    if (n > FP8Q_MAX_ELEMENTS) return FP8Q_ERR_SIZE;
    if (n == 0) {
        if (wire_bytes) *wire_bytes = 0;
        return FP8Q_OK;
    }
    if (n % (512 * (size_t)ranks) != 0) return FP8Q_ERR_SIZE;     // whole, 16-byte aligned chunks
    if (!partials || !results || !workspace) return FP8Q_ERR_NULL;
    const Layout L = layout_of(ranks, n);
    if (workspace_bytes < L.total) return FP8Q_ERR_SIZE;
    if (!aligned16(workspace)) return FP8Q_ERR_ALIGN;
    for (int r = 0; r < ranks; ++r) {
        if (!partials[r] || !results[r]) return FP8Q_ERR_NULL;
        if (!aligned16(partials[r]) || !aligned16(results[r])) return FP8Q_ERR_ALIGN;
        if (overlaps(results[r], 2 * n, workspace, L.total) || overlaps(partials[r], 2 * n, workspace, L.total))
            return FP8Q_ERR_ALIAS;
        for (int q = 0; q < ranks; ++q) {
            if (q != r && overlaps(results[r], 2 * n, results[q], 2 * n)) return FP8Q_ERR_ALIAS;
            // a rank's result may replace its own partial, but not another rank's
            if (q != r && overlaps(results[r], 2 * n, partials[q], 2 * n)) return FP8Q_ERR_ALIAS;
        }
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t m = L.m;
    auto msg_codes = [&](int buf, int r) { return ws + ((size_t)buf * ranks + r) * L.slot; };
    auto msg_scales = [&](int buf, int r) {
        return reinterpret_cast<float*>(ws + ((size_t)buf * ranks + r) * L.slot + L.msg_codes);
    };
    uint8_t* fin_codes = ws + L.final_codes;
    float* fin_scales = reinterpret_cast<float*>(ws + L.final_scales);
    auto chunk = [&](const void* base, int c) {
        return static_cast<const uint16_t*>(base) + (size_t)c * m;
    };

    // reduce-scatter, step 0: every rank quantizes its own chunk, all ranks
    // in one launch (the partials may have been written by the caller's last
    // kernel, so this launch waits for it before reading)
    {
        fp8q_quant_t items[FP8Q_MAX_QUANT_GROUP];
        for (int i = 0; i < ranks; ++i) items[i] = {chunk(partials[i], i), m, msg_codes(0, i), msg_scales(0, i)};
        const fp8q_status_t st = fp8q_quantize_blockwise_group(items, ranks, fmt, 0u, stream);
        if (st != FP8Q_OK) return st;
    }
    // steps 1 .. P-1: one hop per rank, all ranks in one launch
    for (int s = 1; s < ranks; ++s) {
        fp8q_hop_t hops[FP8Q_MAX_HOP_GROUP];
        for (int i = 0; i < ranks; ++i) {
            const int from = (i + ranks - 1) % ranks;
            const int c = ((i - s) % ranks + ranks) % ranks;        // the chunk the message carries
            fp8q_hop_t& hp = hops[i];
            hp.in_codes = msg_codes((s - 1) & 1, from);
            hp.in_scales = msg_scales((s - 1) & 1, from);
            hp.local_bf16 = chunk(partials[i], c);
            hp.n = m;
            if (s < ranks - 1) {
                hp.out_codes = msg_codes(s & 1, i);
                hp.out_scales = msg_scales(s & 1, i);
            } else {                                                 // chunk (i+1) mod P, fully reduced
                hp.out_codes = fin_codes + (size_t)c * m;
                hp.out_scales = fin_scales + (size_t)c * (m / 128);
            }
            hp.out_bf16 = nullptr;
        }
        // The local partials are the callers' inputs: no kernel of this call
        // writes them, and whatever wrote them had finished before the first
        // quantize above passed its grid-dependency wait, so each hop group
        // may start reading them while the previous group drains.
        const fp8q_status_t st = fp8q_ring_hop_group_ex(hops, ranks, fmt, FP8Q_HOP_LOCAL_READY, stream);
        if (st != FP8Q_OK) return st;
    }
    // all-gather of the reduced codes, then every rank decodes the whole
    // vector: one launch writes all P results
    {
        const int divisor = (flags & FP8Q_ALLREDUCE_MEAN) ? ranks : 0;
        const fp8q_status_t st = gather_decode_entry(fin_codes, fin_scales, n, fmt, results, ranks, divisor, stream);
        if (st != FP8Q_OK) return st;
    }
    if (wire_bytes) *wire_bytes = 2ull * (uint64_t)(ranks - 1) * (uint64_t)(m + 4 * (m / 128));
    return FP8Q_OK;
}

extern "C" fp8q_status_t fp8q_ring_allreduce_sim(const void* const* partials, void* const* results, int ranks,
                                                 size_t n, fp8q_format_t fmt, void* workspace,
                                                 size_t workspace_bytes, uint64_t* wire_bytes,
                                                 fp8q_stream_t stream) {
    FP8Q_NVTX_RANGE("fp8q_ring_allreduce_sim");
    return fp8q_ring_allreduce_sim_ex(partials, results, ranks, n, fmt, workspace, workspace_bytes, wire_bytes, 0u,
                                      stream);
}
