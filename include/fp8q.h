/* fp8q -- FP8 / MXFP8 transfer codec for GB300 (sm_103a).
 *
 * C ABI of libfp8q.so.  Every entry point takes plain pointers and sizes,
 * runs asynchronously on the caller's CUDA stream, allocates nothing, never
 * synchronizes and never frees.  Arguments are validated on the host before
 * anything is launched; a failed check returns its status synchronously and
 * launches nothing.  A launch that the CUDA runtime rejects returns
 * FP8Q_ERR_CUDA (the runtime's code is kept in fp8q_last_cuda_error()).
 * No C++ exception crosses this boundary.
 *
 * Pointer rules common to all entry points:
 *  - data pointers are DEVICE pointers owned by the caller, 16-byte aligned
 *    (FP8Q_ERR_ALIGN otherwise);
 *  - an output may not overlap an input or another output (FP8Q_ERR_ALIAS),
 *    except where an entry point says so;
 *  - bf16 arrays hold IEEE binary32 values truncated to their upper 16 bits
 *    (the usual bfloat16), passed as `void*`;
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *
 * Sources (web pages, cited by title and section):
 *  [P1] "FP8 Transmission Optimization for VLA Training: Byte Reduction Leads
 *       to Increased Latency" -- intro ("blockwise scaling", 48.4% fewer wire
 *       bytes than bf16) and "FP8 Transmission Optimization and Bottlenecks"
 *       (e4m3/e5m2 conversion kernels; fused dequantize-then-reduce that
 *       avoids the HBM traffic of the naive order; ring-based collectives).
 *  [P2] "How to Speed Up VLA Training Step by Step: 3x on Pi0.5" -- PCIe
 *       paragraph: bf16 gradients reduced by a ring AllReduce.
 *  [P3] "perf: Reduce MXFP8 refit weight-transfer overheads" -- Summary
 *       (trainer-side BF16->MXFP8 prequantization, MXFP8 shuffle buffers),
 *       Safety (each E4M3 tensor travels with its scale), self-review (E8M0
 *       zero-scale clamp; 2D/3D expert tensors), inline review (a K/32 scale
 *       dimension of size 1 must survive).
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* fp8q_stream_t; /* the same type as cudaStream_t */

typedef enum {
    FP8Q_E4M3 = 0, /* OFP8 E4M3 "fn": bias 7, max 448, no inf, 0x7F/0xFF NaN */
    FP8Q_E5M2 = 1  /* OFP8 E5M2: bias 15, max 57344, IEEE-style inf/NaN      */
} fp8q_format_t;

typedef enum {
    FP8Q_OK = 0,
    FP8Q_ERR_NULL = 1,   /* a required pointer is NULL                        */
    FP8Q_ERR_SIZE = 2,   /* a size is negative or beyond FP8Q_MAX_ELEMENTS    */
    FP8Q_ERR_ALIGN = 3,  /* a pointer is not 16-byte aligned                  */
    FP8Q_ERR_FORMAT = 4, /* unknown fp8q_format_t                             */
    FP8Q_ERR_K = 5,      /* shard count outside [1, FP8Q_MAX_SHARDS], or an
                            MXFP8 K that is not a positive multiple of 32     */
    FP8Q_ERR_CUDA = 6,   /* the CUDA runtime rejected a launch                */
    FP8Q_ERR_ALIAS = 7,  /* an output overlaps an input or another output     */
    FP8Q_ERR_FLAGS = 8   /* unknown bits in a flags argument                  */
} fp8q_status_t;

#define FP8Q_BLOCK 128                   /* elements per blockwise scale   */
#define FP8Q_MAX_SHARDS 16               /* k limit of fp8q_dequant_reduce */
#define FP8Q_MAX_ELEMENTS (1ull << 42)   /* n limit of every entry point   */
#define MXFP8_BLOCK 32                   /* elements per E8M0 scale        */

/* ---------------------------------------------------------------- (a) ----
 * Blockwise FP8 quantize ([P1] intro, "FP8 Transmission Optimization and
 * Bottlenecks").  For each block b of 128 consecutive elements (the last one
 * may be partial and covers only the valid elements):
 *     amax_b = max |x_i|,   scales[b] = RN_fp32(amax_b / Fmax)
 *     codes[i] = satfinite RNE_fp8(RN_fp32(x_i / scales[b]))
 * with Fmax = 448 (e4m3) or 57344 (e5m2); an all-zero block gets scale 0
 * and codes equal to the signed zero of each x_i.
 *   x_bf16 : n bf16 values (in)
 *   codes  : n bytes (out);  scales : fp8q_num_scales(n) floats (out)
 * n == 0 is a no-op returning FP8Q_OK. */
fp8q_status_t fp8q_quantize_blockwise(const void* x_bf16, size_t n, fp8q_format_t fmt,
                                      uint8_t* codes, float* scales, fp8q_stream_t stream);

/* Flag of the *_ex entry points (quantize, dequant-reduce, MXFP8 group):
 * the caller guarantees that no kernel that can still be running when this
 * call's kernel starts writes any of the call's inputs.  Every kernel of
 * this library lets its successor start only after its own grid-dependency
 * wait, so in a chain of these calls an input written two or more launches
 * back qualifies.  With programmatic dependent launch on (see
 * fp8q_set_launch_overlap) the kernel then starts copying its first tiles'
 * inputs while the previous kernel on the stream is finishing; every write
 * still waits for it.  Results are unchanged.  Unknown flag bits give
 * FP8Q_ERR_FLAGS. */
#define FP8Q_INPUTS_READY 1u

/* fp8q_quantize_blockwise with flags (FP8Q_INPUTS_READY). */
fp8q_status_t fp8q_quantize_blockwise_ex(const void* x_bf16, size_t n, fp8q_format_t fmt, uint8_t* codes,
                                         float* scales, unsigned int flags, fp8q_stream_t stream);

/* One item of a grouped quantize: the arguments of fp8q_quantize_blockwise. */
typedef struct {
    const void* x_bf16;        /* n bf16 (in)                                  */
    size_t n;
    uint8_t* codes;            /* n codes (out)                                */
    float* scales;             /* fp8q_num_scales(n) scales (out)              */
} fp8q_quant_t;

#define FP8Q_MAX_QUANT_GROUP 16

/* fp8q_quantize_blockwise for up to FP8Q_MAX_QUANT_GROUP independent arrays
 * in one launch (for instance every rank's chunk of a ring step, or several
 * gradient buckets).  `items` is a HOST array; every item is checked as by
 * fp8q_quantize_blockwise, no output may overlap any input or output of the
 * group (FP8Q_ERR_ALIAS), count must be in [1, FP8Q_MAX_QUANT_GROUP]
 * (FP8Q_ERR_SIZE), and flags may hold FP8Q_INPUTS_READY.  Empty items are
 * skipped.  Results are those of one fp8q_quantize_blockwise per item. */
fp8q_status_t fp8q_quantize_blockwise_group(const fp8q_quant_t* items, int count, fp8q_format_t fmt,
                                            unsigned int flags, fp8q_stream_t stream);

/* ---------------------------------------------------------------- (b) ----
 * Fused k-way dequantize-then-reduce ([P1] "FP8 Transmission Optimization
 * and Bottlenecks": the fused kernel never writes dequantized shards to
 * HBM).  For every element i, in rank order r = 0 .. k-1:
 *     acc = +0;  acc = RN(acc + RN(decode(codes[r][i]) * scales[r][i/128]))
 *     out_fp32[i] = acc,  out_bf16[i] = RNE_bf16(acc)
 * A sum, not a mean.
 *   codes, scales : HOST arrays of k device pointers (shard r: n codes and
 *                   fp8q_num_scales(n) scales); 1 <= k <= FP8Q_MAX_SHARDS
 *   out_bf16, out_fp32 : n elements each; either may be NULL, not both. */
fp8q_status_t fp8q_dequant_reduce(const uint8_t* const* codes, const float* const* scales, int k,
                                  size_t n, fp8q_format_t fmt, void* out_bf16, float* out_fp32,
                                  fp8q_stream_t stream);

/* fp8q_dequant_reduce with flags (FP8Q_INPUTS_READY, see above). */
fp8q_status_t fp8q_dequant_reduce_ex(const uint8_t* const* codes, const float* const* scales, int k,
                                     size_t n, fp8q_format_t fmt, void* out_bf16, float* out_fp32,
                                     unsigned int flags, fp8q_stream_t stream);

/* ---------------------------------------------------------------- (c) ----
 * One hop of a ring reduction carried on the FP8 wire format ([P1] ring-based
 * collectives; [P2] ring AllReduce of bf16 gradients).  At the receiver:
 *     y_i = RN(RN(decode(in_codes[i]) * in_scales[i/128]) + local_i)
 * then y is quantized blockwise exactly as in (a) (amax over |y|, the fp32
 * sum itself is requantized, not its bf16 rounding) into out_codes /
 * out_scales, and, when out_bf16 != NULL, out_bf16[i] = RNE_bf16(y_i).
 *   in_codes: n bytes; in_scales: fp8q_num_scales(n); local_bf16: n bf16 (in)
 *   out_codes, out_scales: as in (a) (out); out_bf16: n bf16 or NULL (out)
 * out_bf16 may be the same pointer as local_bf16 (in-place update of the
 * local partial); no other overlap is allowed. */
fp8q_status_t fp8q_ring_hop(const uint8_t* in_codes, const float* in_scales, const void* local_bf16,
                            size_t n, fp8q_format_t fmt, uint8_t* out_codes, float* out_scales,
                            void* out_bf16, fp8q_stream_t stream);

/* One hop of a grouped call: the arguments of fp8q_ring_hop. */
typedef struct {
    const uint8_t* in_codes;   /* n codes (in)                                 */
    const float* in_scales;    /* fp8q_num_scales(n) scales (in)               */
    const void* local_bf16;    /* n bf16 (in)                                  */
    size_t n;
    uint8_t* out_codes;        /* n codes (out)                                */
    float* out_scales;         /* fp8q_num_scales(n) scales (out)              */
    void* out_bf16;            /* n bf16 (out), or NULL                        */
} fp8q_hop_t;

#define FP8Q_MAX_HOP_GROUP 16

/* fp8q_ring_hop for up to FP8Q_MAX_HOP_GROUP independent hops in one launch
 * (for instance the hops every rank of a ring makes in one step).  `hops` is
 * a HOST array; every hop is checked as by fp8q_ring_hop, no output may
 * overlap any input or output of the group except a hop's out_bf16 written
 * in place over its own local_bf16, and count must be in
 * [1, FP8Q_MAX_HOP_GROUP] (FP8Q_ERR_SIZE).  Results are those of one
 * fp8q_ring_hop per hop. */
fp8q_status_t fp8q_ring_hop_group(const fp8q_hop_t* hops, int count, fp8q_format_t fmt, fp8q_stream_t stream);

/* Flags of fp8q_ring_hop_group_ex. */
#define FP8Q_HOP_LOCAL_READY 1u

/* fp8q_ring_hop_group with flags (unknown bits: FP8Q_ERR_FLAGS); the results
 * are those of fp8q_ring_hop_group.
 * FP8Q_HOP_LOCAL_READY: the caller guarantees that no kernel that can still
 * be running when this call's kernel starts writes any hop's local_bf16 (in
 * a ring the local partial is the rank's own gradient bucket, complete before
 * the incoming chunk arrives).  With programmatic dependent launch on (see
 * fp8q_set_launch_overlap) the kernel then starts copying the local partials
 * of its first tiles while the previous kernel on the stream is finishing;
 * the incoming codes and scales, and every write, still wait for it. */
fp8q_status_t fp8q_ring_hop_group_ex(const fp8q_hop_t* hops, int count, fp8q_format_t fmt, unsigned int flags,
                                     fp8q_stream_t stream);

/* ---------------------------------------------------- ring AllReduce ----
 * A ring AllReduce carried on the FP8 wire format, with all P ranks held on
 * one GPU ([P1] ring-based collectives on the FP8 wire; [P2] a ring
 * AllReduce moves 2 (P-1)/P of the bytes per GPU).  Chunk c of n elements is
 * [c n/P, (c+1) n/P).
 *   reduce-scatter: step 0, rank i quantizes its chunk i; steps 1..P-1,
 *     rank i makes one fp8q_ring_hop on the message of rank i-1 (chunk
 *     (i-s) mod P) with its own chunk, all P hops of a step in one launch;
 *     rank i ends with chunk (i+1) mod P summed over all ranks, as codes;
 *   all-gather: the reduced codes and scales travel unchanged, and every
 *     rank dequantizes the whole vector into results[r] (all ranks equal).
 *     The ranks share one GPU, so the gathered codes are one buffer: a
 *     single launch decodes it and writes all P results.
 * A sum; fp8q_ring_allreduce_sim_ex with FP8Q_ALLREDUCE_MEAN gives the mean.
 *   partials, results : HOST arrays of `ranks` device pointers to n bf16;
 *                       results[r] may be partials[r] (in place)
 *   ranks             : 2 .. FP8Q_MAX_HOP_GROUP (FP8Q_ERR_K otherwise)
 *   n                 : a multiple of 512 * ranks (FP8Q_ERR_SIZE otherwise)
 *   workspace         : fp8q_ring_allreduce_workspace_bytes(ranks, n) bytes of
 *                       device memory, caller-owned (message and result codes)
 *   wire_bytes        : if not NULL, the bytes one rank sends over the whole
 *                       collective: 2 (P-1) (n/P) (1 + 4/128). */
size_t fp8q_ring_allreduce_workspace_bytes(int ranks, size_t n);
fp8q_status_t fp8q_ring_allreduce_sim(const void* const* partials, void* const* results, int ranks, size_t n,
                                      fp8q_format_t fmt, void* workspace, size_t workspace_bytes,
                                      uint64_t* wire_bytes, fp8q_stream_t stream);

/* fp8q_ring_allreduce_sim with flags (0 = the sum, as above).
 * FP8Q_ALLREDUCE_MEAN: the all-gather decode divides each decoded value by
 * the rank count before the bf16 rounding,
 *     results[r][i] = RNE_bf16(RN(RN(decode(c_i) * s_b) / ranks))
 * with a true (correctly rounded) binary32 division; the codes on the wire
 * and wire_bytes are unchanged.  The pages reduce gradients over the ranks
 * without printing a mean; data-parallel training averages them, and this
 * is that average taken once, at the end, on the decoded sum.
 * Other flag bits: FP8Q_ERR_FLAGS. */
#define FP8Q_ALLREDUCE_MEAN 1u
fp8q_status_t fp8q_ring_allreduce_sim_ex(const void* const* partials, void* const* results, int ranks, size_t n,
                                         fp8q_format_t fmt, void* workspace, size_t workspace_bytes,
                                         uint64_t* wire_bytes, unsigned int flags, fp8q_stream_t stream);

/* The all-gather receiver step of the ring AllReduce above, on its own:
 * one FP8 vector (n codes and their fp8q_num_scales(n) block scales, the
 * fully reduced chunks in chunk order) decoded once and written as bf16 to
 * each of `count` outputs, outs[o][i] = RNE_bf16(RN(decode(c_i) * s_b)).
 * With FP8Q_ALLREDUCE_MEAN each decoded value is first divided by `count`
 * (a true binary32 division), as fp8q_ring_allreduce_sim_ex does.
 *   outs  : HOST array of `count` device pointers to n bf16 each
 *   count : 1 .. FP8Q_MAX_HOP_GROUP (FP8Q_ERR_K otherwise)
 * Outputs may not overlap each other or the inputs (FP8Q_ERR_ALIAS); other
 * flag bits: FP8Q_ERR_FLAGS. */
fp8q_status_t fp8q_gather_decode(const uint8_t* codes, const float* scales, size_t n, fp8q_format_t fmt,
                                 void* const* outs, int count, unsigned int flags, fp8q_stream_t stream);

/* ------------------------------------------------------------ variants ----
 * fp8q_quantize_tensorwise: one scale for the whole tensor (the tensorwise
 *   recipe of TorchAO's Float8Linear that [P2] uses for its FP8 GEMMs):
 *   amax = max |x_i|, s = RN(amax / Fmax), c_i = satfinite RNE_fp8(RN(x_i/s)),
 *   i.e. (a) with one block of n elements.  scale_amax: 2 device floats,
 *   [0] = s and [1] = amax on return (the call clears [1] first, with a
 *   cudaMemsetAsync on `stream`).
 * fp8q_ring_hop_bf16_requant: fp8q_ring_hop, but the block is requantized
 *   from RNE_bf16(y) -- the bf16 partial a receiver keeps -- instead of the
 *   fp32 sum y (the other reading of "adds it to the local bf16 partial and
 *   requantizes").  Same arguments and rules as fp8q_ring_hop. */
fp8q_status_t fp8q_quantize_tensorwise(const void* x_bf16, size_t n, fp8q_format_t fmt, uint8_t* codes,
                                       float* scale_amax, fp8q_stream_t stream);
fp8q_status_t fp8q_ring_hop_bf16_requant(const uint8_t* in_codes, const float* in_scales, const void* local_bf16,
                                         size_t n, fp8q_format_t fmt, uint8_t* out_codes, float* out_scales,
                                         void* out_bf16, fp8q_stream_t stream);

/* ---------------------------------------------------------------- (d) ----
 * BF16 -> MXFP8 weight prequantization ([P3] Summary, self-review).
 * w is [batch, m, k] row-major ([out, in] weights, batch = experts); every
 * row is cut into k/32 blocks of 32 along k.  Per block:
 *     amax = max |w|;  e = 0 if amax == 0 (zero-scale clamp), else
 *     e = clamp(floor(log2 amax) - 8 + 127, 0, 254)          (E8M0 byte)
 *     codes = satfinite RNE_e4m3(w * 2^(127 - e))             (row-major)
 * The E8M0 bytes are written in the 128x4-tiled layout of block-scaled GEMMs:
 * scale (r, j) of matrix bt lives at
 *     bt * R * C * 512 + ((r/128) * C + j/4) * 512
 *        + (r%32) * 16 + ((r%128)/32) * 4 + (j%4)
 * with R = ceil(m/128), C = ceil((k/32)/4); padding bytes are written as 0.
 *   codes: batch*m*k bytes; scales_swizzled: mxfp8_swizzled_scale_bytes()
 * k must be a positive multiple of 32 (FP8Q_ERR_K); k == 32 keeps its one
 * scale column (padded to 4).  batch == 0 or m == 0 is a no-op. */
fp8q_status_t mxfp8_quantize_swizzled(const void* w_bf16, int64_t batch, int64_t m, int64_t k,
                                      uint8_t* codes, uint8_t* scales_swizzled, fp8q_stream_t stream);

/* One weight tensor of a grouped MXFP8 call: the arguments of
 * mxfp8_quantize_swizzled for that tensor. */
typedef struct {
    const void* w_bf16;        /* [batch, m, k] bf16, row-major (in)        */
    int64_t batch, m, k;
    uint8_t* codes;            /* batch * m * k E4M3 codes (out)            */
    uint8_t* scales_swizzled;  /* mxfp8_swizzled_scale_bytes() bytes (out)  */
} mxfp8_tensor_t;

#define MXFP8_MAX_GROUP 16

/* mxfp8_quantize_swizzled for up to MXFP8_MAX_GROUP tensors in one launch
 * (for instance a decoder layer: the expert batches and the attention
 * matrices), the way [P3] batches its MXFP8 MoE shuffle over all experts of
 * a layer.  `tensors` is a HOST array of `count` descriptors; every tensor
 * is checked as by mxfp8_quantize_swizzled (same status codes), no output
 * may overlap any input or output of the group (FP8Q_ERR_ALIAS), and
 * count must be in [1, MXFP8_MAX_GROUP] (FP8Q_ERR_SIZE).  Empty tensors are
 * skipped.  Results are those of one mxfp8_quantize_swizzled per tensor. */
fp8q_status_t mxfp8_quantize_swizzled_group(const mxfp8_tensor_t* tensors, int count, fp8q_stream_t stream);

/* mxfp8_quantize_swizzled_group with flags (FP8Q_INPUTS_READY: no kernel
 * still running writes any tensor's w_bf16). */
fp8q_status_t mxfp8_quantize_swizzled_group_ex(const mxfp8_tensor_t* tensors, int count, unsigned int flags,
                                               fp8q_stream_t stream);

/* ------------------------------------------------------ MXFP8 receiver ----
 * The receiving side of [P3]'s prequantized transfer.
 *
 * mxfp8_dequantize_swizzled: w = RNE_bf16(decode_e4m3(c) * 2^(e - 127)) for
 *   codes [batch, m, k] and the swizzled E8M0 bytes of mxfp8_quantize_swizzled;
 *   the product is exact, only results below the bf16 range round.
 *   out_bf16: batch*m*k bf16 (out).  Same shape rules as the quantizer,
 *   and batch * ceil(m/128) * ceil(k/128) < 2^32 (FP8Q_ERR_SIZE).
 * mxfp8_unswizzle_scales: the E8M0 bytes in plain row-major order
 *   [batch, m, k/32] (the layout whose trailing k/32 dimension [P3]'s inline
 *   review insists on keeping, even when it is 1).
 * fp8q_count_mismatches: adds to the device counter *count the number of
 *   bytes where a and b differ (the bit-exact check [P3]'s reproductions
 *   ran on the shuffled MXFP8 buffers); the caller zeroes *count.  count must
 *   be 8-byte aligned device memory. */
fp8q_status_t mxfp8_dequantize_swizzled(const uint8_t* codes, const uint8_t* scales_swizzled, int64_t batch,
                                        int64_t m, int64_t k, void* out_bf16, fp8q_stream_t stream);
fp8q_status_t mxfp8_unswizzle_scales(const uint8_t* scales_swizzled, int64_t batch, int64_t m, int64_t k,
                                     uint8_t* scales_rowmajor, fp8q_stream_t stream);
fp8q_status_t fp8q_count_mismatches(const void* a, const void* b, size_t nbytes, unsigned long long* count,
                                    fp8q_stream_t stream);

/* ----------------------------------------------------- transfer packing ----
 * [P3] inline review: weights and their scales travel as separate entries
 * through size-capped transfer batches, a weight (~32x its scale) usually
 * closes a batch and its scale opens the next, and the receiver's per-batch
 * check then fails; oversized parameters travel alone.  The fix it names is
 * packing weight and scale atomically.
 *
 * fp8q_pack_plan (host only, no GPU): items[i] is the byte size of weight
 *   i's codes and of its scales.  Every pair goes whole into one batch:
 *   codes at slots[i].codes_offset, scales at slots[i].scales_offset of
 *   batch slots[i].batch (16-byte aligned offsets).  Pairs are taken in
 *   order; a pair that does not fit in the current batch (cap_bytes) opens
 *   the next one, and a pair larger than the cap gets a batch of its own.
 *   batch_bytes (room for `count` entries) receives each batch's size,
 *   *num_batches their number.
 * fp8q_copy_segments: one launch copying up to FP8Q_MAX_COPY_SEGMENTS
 *   device byte ranges (the gather of a plan's pairs into a transfer
 *   buffer, or the scatter out of it on the receiver).  src and dst 16-byte
 *   aligned, any byte count; destinations must not overlap each other or any
 *   source (FP8Q_ERR_ALIAS). */
typedef struct {
    uint64_t codes_bytes, scales_bytes;
} fp8q_pack_item_t;

typedef struct {
    int32_t batch;
    uint64_t codes_offset, scales_offset;
} fp8q_pack_slot_t;

typedef struct {
    const void* src;
    void* dst;
    uint64_t bytes;
} fp8q_copy_t;

#define FP8Q_MAX_COPY_SEGMENTS 96

fp8q_status_t fp8q_pack_plan(const fp8q_pack_item_t* items, int count, uint64_t cap_bytes, fp8q_pack_slot_t* slots,
                             uint64_t* batch_bytes, int* num_batches);
fp8q_status_t fp8q_copy_segments(const fp8q_copy_t* segs, int count, fp8q_stream_t stream);

/* ------------------------------------------------------------- helpers ---- */

/* ceil(n / 128): the number of fp32 scales of an n-element blockwise array. */
size_t fp8q_num_scales(size_t n);

/* Bytes of the swizzled E8M0 scale buffer of a [batch, m, k] weight
 * (0 for invalid arguments). */
size_t mxfp8_swizzled_scale_bytes(int64_t batch, int64_t m, int64_t k);

/* Static, NUL-terminated description of a status code. */
const char* fp8q_status_string(fp8q_status_t status);

/* cudaError_t of the most recent FP8Q_ERR_CUDA on the calling thread (0 if none). */
int fp8q_last_cuda_error(void);

/* Programmatic dependent launch, process-wide; on by default.  When on,
 * every kernel of this library is launched with programmatic stream
 * serialization: its blocks may be dispatched while the previous kernel on
 * the stream is still finishing, and each kernel waits on the device for
 * that kernel to complete, with its writes visible, before it touches global
 * memory.  Results and stream order are the same either way; only the gap
 * between dependent launches shrinks.  Returns the previous setting
 * (1 = on).  Takes effect for launches made after the call. */
int fp8q_set_launch_overlap(int enable);

/* Diagnostic, and the one call that synchronizes: waits for the current
 * device, then returns in *flags the error bits the kernels raised since the
 * last clear (0 = none; bit 0 = an input copy into shared memory did not land
 * within 2 s, after which the kernel stopped and its outputs are invalid).
 * Clears the bits when `clear` is non-zero. */
#define FP8Q_DEVICE_ERR_COPY_TIMEOUT 1u
fp8q_status_t fp8q_device_errors(unsigned int* flags, int clear);

/* Self-test of the bounded copy wait (a test hook, not a step of the codec).
 * Every staged kernel waits for its shared-memory copies with a wall-clock
 * limit of 2 s; when a wait runs out, the kernel raises
 * FP8Q_DEVICE_ERR_COPY_TIMEOUT and returns instead of hanging ([P3] Safety:
 * fail loudly).  This entry point launches one CTA of 64 threads that waits
 * on a shared-memory barrier armed for 16 transaction bytes, with the same
 * wait and the same give-up path, at a limit of `limit_ns`:
 *   - src == dst == NULL: no copy is issued, so the wait must run out after
 *     limit_ns; the CTA raises FP8Q_DEVICE_ERR_COPY_TIMEOUT (read back with
 *     fp8q_device_errors) and returns.  Nothing is in flight at any time, and
 *     the context stays usable for the calls that follow.
 *   - src, dst non-NULL (16-byte aligned device pointers, not overlapping):
 *     the 16 bytes at src are bulk-copied into the barrier's stage, the wait
 *     completes, and thread 0 writes them to dst; no error bit is raised.
 * limit_ns must lie in [FP8Q_SELFTEST_MIN_WAIT_NS, FP8Q_SELFTEST_MAX_WAIT_NS]
 * (FP8Q_ERR_SIZE otherwise); only one of src and dst NULL is FP8Q_ERR_NULL. */
#define FP8Q_SELFTEST_MIN_WAIT_NS 1000000ull      /* 1 ms */
#define FP8Q_SELFTEST_MAX_WAIT_NS 2000000000ull   /* 2 s, the kernels' own limit */
fp8q_status_t fp8q_selftest_copy_wait(const void* src, void* dst, uint64_t limit_ns, fp8q_stream_t stream);

/* Plain satfinite round-to-nearest-even conversion of n binary32 values to
 * FP8 codes, with no scale (the element conversion step of (a) and (c),
 * exposed for exhaustive checking and for per-tensor scaled callers).
 *   x: n floats (in);  codes: n bytes (out). */
fp8q_status_t fp8q_encode_f32(const float* x, size_t n, fp8q_format_t fmt, uint8_t* codes,
                              fp8q_stream_t stream);

/* Single-shard dequantize: d_i = RN(decode(codes[i]) * scales[i/128]), written
 * as fp32 and/or RNE bf16 (either output may be NULL, not both). */
fp8q_status_t fp8q_dequantize(const uint8_t* codes, const float* scales, size_t n, fp8q_format_t fmt,
                              void* out_bf16, float* out_fp32, fp8q_stream_t stream);

/* The naive order that (b) replaces ([P1]: "naive dequantize-then-reduce"),
 * kept as a comparator: each shard is dequantized to fp32 in `workspace`
 * (caller-owned, k * fp8q_unfused_stride(n) floats; shard r's slot starts at
 * float r * fp8q_unfused_stride(n)), then the k fp32 arrays are summed in
 * rank order.  Bit-identical to fp8q_dequant_reduce; it only moves more bytes. */
/* n rounded up to a multiple of 4: the per-shard fp32 slot of the workspace
 * of fp8q_dequant_reduce_unfused, which keeps every slot 16-byte aligned. */
size_t fp8q_unfused_stride(size_t n);

fp8q_status_t fp8q_dequant_reduce_unfused(const uint8_t* const* codes, const float* const* scales,
                                          int k, size_t n, fp8q_format_t fmt, float* workspace,
                                          void* out_bf16, float* out_fp32, fp8q_stream_t stream);

/* ----------------------------------------------- no-allocation variant ----
 * Not a step of the codec (the source pages have no counterpart): the
 * unfused comparator above with its scratch inside the library instead of
 * a caller-supplied workspace.
 *
 * Who needs it: callers that cannot call cudaMalloc.  An interception layer
 * slotted under a training framework runs in a process whose device memory
 * belongs to the framework's caching allocator, and it has no handle to that
 * allocator; and on a busy GPU a cudaMalloc / cudaFree pair can synchronize
 * the device and stall every stream.  Such a caller still passes its inputs
 * and outputs, but no workspace.
 *
 * The scratch is one static device array of FP8Q_STATIC_SCRATCH_FLOATS
 * floats (16 MiB) in the library.  It is reserved on a device when the
 * library's reduce module is loaded there -- under CUDA's default lazy
 * module loading, at the first use on that device of this call or of any
 * other reduce kernel of the library -- and held until the process exits.  Each shard uses fp8q_unfused_stride(n)
 * floats of it, so the call needs k * fp8q_unfused_stride(n) <=
 * FP8Q_STATIC_SCRATCH_FLOATS; larger calls return FP8Q_ERR_SIZE and launch
 * nothing.  The call allocates nothing: no cudaMalloc, no cudaFree.
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and keeps it; make that first call before any stream
 * capture.  All calls share the one array and it keeps whatever the last
 * call left there; nothing in it needs clearing, because every call writes
 * each scratch element it reads before reading it.  Calls whose work
 * overlaps on the GPU (different streams, or concurrent host threads) race
 * on the array: order them on one stream or with events.
 * Arguments and results are otherwise those of fp8q_dequant_reduce_unfused. */
#define FP8Q_STATIC_SCRATCH_FLOATS (1u << 22)

fp8q_status_t fp8q_dequant_reduce_unfused_static(const uint8_t* const* codes, const float* const* scales,
                                                 int k, size_t n, fp8q_format_t fmt, void* out_bf16,
                                                 float* out_fp32, fp8q_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H */
