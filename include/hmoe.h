/*
 * hmoe.h -- C ABI of libhmoe: the hybrid W4A16 mixture-of-experts layer on GB300 (sm_103a).
 *
 * The layer serves per-expert mixed-precision MoE checkpoints. Each expert
 * is a SwiGLU feed-forward block, W13 [2I, H] (gate rows, then up rows) and
 * W2 [H, I]. Its weights sit in one of two tiers, chosen per expert by a
 * bit map:
 *   4 = the kept tier, NVFP4 (or MXFP4 when kept_format says so),
 *   3 = the NF3 tier, 3-bit NormalFloat.
 * Activations are 16-bit throughout, bf16 or fp16 as the layer descriptor
 * says (act_dtype). Both tiers run off one shared route geometry (top-k ids,
 * gates, token permutation, expert offsets) and sum into one output.
 *   Cites: "quant: nvfp4_nf3_hybrid -- native serving for mixed NVFP4+NF3 MoE
 *   checkpoints", How it works (two prepared weight sets per layer, one
 *   shared route geometry and topk_sum, CUDA-graph-safe launches, an M<=8
 *   decode path). "quant: add native mixed NVFP4/MXFP4 plus NF3 MoE
 *   serving", Summary (hybrid_bit_map: 4 = kept, 3 = NF3; kept_format
 *   selects MXFP4; scratch sized from the maximum batched token count; no
 *   environment variables). "[Quantization][ModelOpt] W4A16 NVFP4 fused
 *   MoE", Summary (W4A16: 4-bit weights, 16-bit activations, no activation
 *   scales) and item 2 (the activation type may be bfloat16 or float16).
 *
 * Conventions
 *   - Every pointer argument named *_dev or documented "device" is device
 *     memory owned by the caller. The library never allocates device memory.
 *   - Host pointers are read during the call only.
 *   - hmoe_plan_routes and hmoe_forward enqueue work on the given stream and
 *     return. They never synchronise, allocate or copy to the host, so they
 *     may be captured in a CUDA graph. Grid sizes depend only on T and the
 *     layer descriptor, never on routing results.
 *   - Argument errors are found on the host. The call then returns a
 *     negative status before anything is enqueued, and hmoe_last_error()
 *     describes the error.
 *   - Faults the device finds (a route id or permutation entry out of
 *     range, inconsistent offsets, a bounded wait that timed out) do not
 *     trap. Kernels skip the bad access and record a code in the workspace.
 *     hmoe_check_device_status reads that code.
 *   - No C++ exceptions cross this boundary, and no environment variable
 *     configures the library. (Each entry point opens an NVTX range named
 *     after it, for profiler timelines; NVTX looks up its profiler-injection
 *     hook once, and without a profiler the ranges do nothing.)
 *   - Layout of the logical checkpoint tensors (the input to
 *     hmoe_pack_weights), for one matrix [N rows, K] of one expert:
 *       NVFP4: codes uint8 [N][K/2]. Element 2i is the low nibble, element
 *              2i+1 the high nibble. E2M1 is 1 sign, 2 exponent and 1
 *              mantissa bit. Scales are E4M3 uint8 [N][K/16] and there is one
 *              fp32 global scale. w = e2m1 * e4m3 * global.
 *       MXFP4: codes as NVFP4. Scales are E8M0 uint8 [N][K/32].
 *              w = e2m1 * 2^(b-127).
 *       NF3:   codes are an LSB-first 3-bit bitstream, uint8 [N][3K/8]. Code
 *              j is bits [3j, 3j+3) of the row's little-endian byte string.
 *              Scales are bf16 [N][K/64]. w = bf16_rne(cb[code] * scale),
 *              with the codebook cb (bf16 bits, index 0..7) =
 *              {BF80, BF09, BE7D, 0000, 3E3C, 3EC4, 3F1F, 3F80}, the 3-bit
 *              NormalFloat construction (Dettmers et al., QLoRA 2023).
 *     The pages fix none of these layouts. This library fixes them as above.
 */
#ifndef HMOE_H_
#define HMOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. NULL is the legacy default stream. */
typedef struct CUstream_st* hmoe_stream_t;

typedef enum {
  HMOE_OK = 0,
  HMOE_ERR_INVALID_ARG = -1,         /* NULL pointer, T < 0, bad enum value, ... */
  HMOE_ERR_UNSUPPORTED_SHAPE = -2,   /* H % 128, I % 64, E > 512, topk > 32, topk > E, T * topk > INT_MAX */
  HMOE_ERR_WORKSPACE_TOO_SMALL = -3, /* ws_bytes < hmoe_workspace_size(T) */
  HMOE_ERR_BAD_BITMAP = -4,          /* a bit_map entry other than 3 or 4 */
  HMOE_ERR_CUDA = -5,                /* a CUDA runtime call failed; see hmoe_last_error */
  HMOE_ERR_DEVICE_TIMEOUT = -6,      /* a bounded device wait ran out (from hmoe_check_device_status) */
  HMOE_ERR_BAD_ROUTE = -7            /* device found an out-of-range route entry */
} hmoe_status;

typedef enum { HMOE_FMT_NF3 = 3, HMOE_FMT_NVFP4 = 4, HMOE_FMT_MXFP4 = 5 } hmoe_fmt;

/* Activation type: x, the SwiGLU output h, the result, and the tensor-core
 * operands (the weights are dequantised to this type). Accumulation is fp32
 * either way.
 *   Cites: "[Quantization][ModelOpt] W4A16 NVFP4 fused MoE +
 *   --override-activation-dtype flag", Summary item 2 (bfloat16 or float16
 *   activations for the W4A16 path).
 * fp16 ranges (the weights are exact in fp16 only inside them; outside, a
 * value rounds to 0 or to infinity and the result is undefined): MXFP4
 * scale bytes b in 104..140 (2^-23 .. 2^13); NF3 scales in the fp16 normal
 * range 2^-14 .. 65504. Every NVFP4 value is exact in fp16. Activations
 * must fit fp16 like any fp16 model's. */
typedef enum { HMOE_ACT_BF16 = 0, HMOE_ACT_F16 = 1 } hmoe_act_dtype;

/* Activation quantisation: none (W4A16) or NVFP4 (W4A4).
 *   Cites: "[Quantization][ModelOpt] W4A16 NVFP4 fused MoE + ...", Summary
 *   (the W4A4 NVFP4 scheme: static NVFP4 weights, activations quantised to
 *   NVFP4 as they arrive).
 * With HMOE_ACT_QUANT_NVFP4 the forward quantises x before W13 and h (after
 * rounding to the activation type) before W2, each in blocks of 16 along the
 * row with the rule of hmoe_quantize_act_nvfp4 and the layer's static global
 * scale of that activation (act_global13, act_global2). The products are
 * computed exactly: e2m1 * e4m3 values are exact in bf16 and fp16, so the
 * same tensor-core and streaming kernels run on them, and the global scales
 * are applied to the fp32 sums. */
typedef enum { HMOE_ACT_QUANT_NONE = 0, HMOE_ACT_QUANT_NVFP4 = 1 } hmoe_act_quant;

/* One MoE layer's shape. kept_format is HMOE_FMT_NVFP4 or HMOE_FMT_MXFP4. */
typedef struct {
  int H;           /* hidden size, a multiple of 128 */
  int I;           /* expert intermediate size, a multiple of 64 */
  int E;           /* experts, 1..512 */
  int topk;        /* experts per token, 1..min(E, 32) */
  int kept_format; /* hmoe_fmt of the kept (bit 4) tier */
  int act_dtype;   /* hmoe_act_dtype; 0 (a zeroed struct) is bf16 */
  int act_quant;   /* hmoe_act_quant; 0 (a zeroed struct) is W4A16 */
  float act_global13; /* W4A4: static global scale of x (the W13 input), finite and > 0 */
  float act_global2;  /* W4A4: static global scale of h (the W2 input), finite and > 0 */
} hmoe_layer_desc;

/* One expert's logical checkpoint tensors (device pointers, layout above).
 * *_global is the NVFP4 fp32 global scale of that matrix. It is ignored
 * for MXFP4 and NF3. */
typedef struct {
  const void* w13_codes;
  const void* w13_scales;
  float w13_global;
  const void* w2_codes;
  const void* w2_scales;
  float w2_global;
} hmoe_expert_src;

typedef struct hmoe_layer hmoe_layer; /* opaque host handle: tier tables, no device memory */

/* Bytes of the two tier-local packed buffers for this bit map.
 *   Cites: "quant: nvfp4_nf3_hybrid -- native serving ...", How it works (two
 *   prepared weight objects per layer, one per tier); "quant: add native
 *   mixed NVFP4/MXFP4 plus NF3 MoE serving", Summary (compact tier-local
 *   storage).
 * bit_map: host int8 [E] with 4 or 3 per expert, or NULL for a uniform
 * layer (every expert in kept_format). The two outputs are the sizes of the
 * kept_buf and nf3_buf arguments of hmoe_pack_weights. Either may be 0. */
hmoe_status hmoe_packed_size(const hmoe_layer_desc* desc, const int8_t* bit_map,
                             size_t* kept_bytes, size_t* nf3_bytes);

/* Workspace bytes for hmoe_plan_routes and hmoe_forward at up to max_tokens
 * tokens per call.
 *   Cites: "quant: add native mixed NVFP4/MXFP4 plus NF3 MoE serving",
 *   Summary (scratch sized from the maximum batched token count).
 * The workspace holds the status word, the kernels' self-cleaning work
 * queues, the routing chunk counts, the quantised input (W4A4 only), the
 * gathered activation rows (T > 8),
 * the SwiGLU output h [T*k][I] (16-bit) and the per-slot W2 output [T*k][H]
 * fp32. Errors: the desc checks (HMOE_ERR_INVALID_ARG,
 * HMOE_ERR_UNSUPPORTED_SHAPE); max_tokens < 0 or bytes NULL is
 * HMOE_ERR_INVALID_ARG; max_tokens * topk above INT_MAX is
 * HMOE_ERR_UNSUPPORTED_SHAPE (the kernels index slots with 32-bit ints). */
hmoe_status hmoe_workspace_size(const hmoe_layer_desc* desc, int max_tokens, size_t* bytes);

/* The path hmoe_forward takes for T tokens when opts->path is HMOE_PATH_AUTO:
 * HMOE_PATH_STREAM while T * topk <= 8 * E (at most 8 routed slots per
 * expert on average; every T <= 8 included), HMOE_PATH_GROUPED above. Host
 * only: no device work, no GPU needed. The pages give the M <= 8 path
 * ("quant: nvfp4_nf3_hybrid ...", How it works) but no rule above it; the
 * factor 8 is this library's measured crossover between its two kernels.
 *   Cites: "quant: nvfp4_nf3_hybrid -- native serving ...", How it works
 *   (the M<=8 decode path beside the batched one).
 * Errors: HMOE_ERR_INVALID_ARG (NULL pointer, T < 0) and the desc checks of
 * hmoe_workspace_size. */
hmoe_status hmoe_auto_path(const hmoe_layer_desc* desc, int T, int* path);

/* Zero the workspace once, before its first use, on the stream. Every
 * completed hmoe_forward leaves the workspace's counters at zero again. Zero
 * it once more after a call reports HMOE_ERR_DEVICE_TIMEOUT.
 *   Cites: "quant: add native mixed NVFP4/MXFP4 plus NF3 MoE serving",
 *   Summary (scratch sized once, up front); "quant: nvfp4_nf3_hybrid --
 *   native serving ...", How it works (preplanned, CUDA-graph-safe launches:
 *   the scratch needs no per-call reset on the host).
 * ws_dev: device; all ws_bytes of it are zeroed. Errors:
 * HMOE_ERR_INVALID_ARG (NULL), HMOE_ERR_CUDA. */
hmoe_status hmoe_workspace_init(void* ws_dev, size_t ws_bytes, hmoe_stream_t stream);

/* Demultiplex the experts into tier-local packed buffers per the bit map. Each
 * tier's experts are stored contiguously in ascending expert id, in this
 * library's tile layout, which depends on act_dtype (NVFP4 codes are stored
 * for the decoder of that type). It then creates the layer handle.
 *   Cites: "quant: add native mixed NVFP4/MXFP4 plus NF3 MoE serving",
 *   Summary (demultiplex the expert weights into compact tier-local storage;
 *   the metadata is validated).
 * src: host array [E] of device pointers. kept_buf and nf3_buf are device
 * buffers of at least the hmoe_packed_size bytes (NULL if that size is 0),
 * and must stay alive while the handle is used. Kernels run on the stream.
 * The source tensors may be freed once the stream has passed this point.
 * Returns HMOE_ERR_BAD_BITMAP for an entry not in {3, 4}. *out receives the
 * handle. Free it with hmoe_layer_destroy. */
hmoe_status hmoe_pack_weights(const hmoe_layer_desc* desc, const int8_t* bit_map,
                              const hmoe_expert_src* src, void* kept_buf, void* nf3_buf,
                              hmoe_stream_t stream, hmoe_layer** out);

/* Route T tokens: softmax top-k with renormalised gates, then a stable
 * counting sort of the T*k slots by expert.
 *   Cites: "quant: nvfp4_nf3_hybrid -- native serving ...", How it works (the
 *   route geometry both tiers share).
 * logits: device fp32 [T][E] row-major. NaN logits are not supported.
 * ids:    device int32 [T][k]. The k largest logits, descending, with ties
 *         to the lower expert id; -0 and +0 count as equal.
 * gates:  device fp32 [T][k]. exp(l_j - l_max) / sum over the k chosen.
 * perm:   device int32 [T*k]. The flat slot indices s = t*k + j sorted by
 *         expert, ascending s within an expert.
 * offsets: device int32 [E+1]. The exclusive prefix sum of per-expert
 *         counts, with offsets[E] = T*k.
 * ws: the workspace (device). T = 0 is valid and writes offsets as zeros.
 * T * k above INT_MAX returns HMOE_ERR_UNSUPPORTED_SHAPE before anything is
 * enqueued. */
hmoe_status hmoe_plan_routes(const hmoe_layer* layer, const float* logits, int T, int32_t* ids,
                             float* gates, int32_t* perm, int32_t* offsets, void* ws,
                             size_t ws_bytes, hmoe_stream_t stream);

/* Forward options. Pass NULL to hmoe_forward_ex for the defaults. */
typedef enum {
  HMOE_TIERS_ONE_LAUNCH = 0,     /* both tiers in each launch, format chosen per expert */
  HMOE_TIERS_KEPT_FIRST = 1,     /* kept tier launch, then NF3 tier launch (per GEMM) */
  HMOE_TIERS_NF3_FIRST = 2       /* NF3 first, then kept */
} hmoe_tier_order;

typedef enum {
  HMOE_PATH_AUTO = 0,     /* streaming while T*topk <= 8*E (at most 8 routed slots per expert
                             on average, every T <= 8 included); the grouped path above */
  HMOE_PATH_STREAM = 1,   /* weight-streaming path at any T (tokens in groups of 8) */
  HMOE_PATH_GROUPED = 2   /* tensor-core grouped GEMM path (tcgen05) */
} hmoe_path;

typedef struct {
  int tier_order;    /* hmoe_tier_order */
  int path;          /* hmoe_path */
  int wait_limit_us; /* bound on every device-side wait; 0 = the default (2 s) */
  int debug_flags;   /* test hook: HMOE_DEBUG_NO_COPIES makes the weight producer issue nothing, so
                        the consumers' bounded waits run out and the call reports
                        HMOE_ERR_DEVICE_TIMEOUT through hmoe_check_device_status. 0 in normal use. */
  void* const* stage_events; /* optional cudaEvent_t[n_stage_events], recorded on the stream at
                                the stage boundaries: [0] before the W13 GEMM, [1] after it,
                                [2] after the W2 GEMM, [3] after the finalize. NULL = none.
                                Where one launch runs both GEMMs (the streaming path at
                                small T), [1] and [2] are both recorded after that launch. */
  int n_stage_events;
} hmoe_forward_opts;

#define HMOE_DEBUG_NO_COPIES 1
/* Comparison hook: the grouped path runs its CTA-pair tensor-core kernel
 * (tcgen05.mma.cta_group::2 over two SMs, 256-slot token tiles) instead of
 * the one-CTA kernel. Same results within the layer tolerance; for
 * measurements only; bf16 layers only. */
#define HMOE_DEBUG_GROUPED_PAIR 2

/* The layer: out[t] = sum_j gates[t,j] * W2_e (silu(W1_e x_t) * W3_e x_t) with
 * e = ids[t,j], fp32 accumulation and a result of the activation type
 * (h is rounded to that type too). Expert weights are dequantised from their
 * tier format to the activation type as they stream.
 *   Cites: "quant: nvfp4_nf3_hybrid -- native serving ...", How it works (both
 *   tiers run off one shared topk_sum; preplanned, CUDA-graph-safe launches;
 *   an M<=8 decode path); "[Quantization][ModelOpt] W4A16 NVFP4 fused MoE",
 *   Summary (W4A16: 4-bit weights, bf16 activations, fp32 accumulation).
 * Errors, all found on the host before anything is enqueued:
 * HMOE_ERR_INVALID_ARG (NULL layer or buffer, T < 0, x or out not 16-byte
 * aligned, a bad option, the grouped path forced at T <= 8,
 * HMOE_DEBUG_GROUPED_PAIR with fp16 activations),
 * HMOE_ERR_UNSUPPORTED_SHAPE (T * topk above INT_MAX),
 * HMOE_ERR_WORKSPACE_TOO_SMALL, and HMOE_ERR_CUDA if a launch fails. Faults
 * the kernels find are read later with hmoe_check_device_status.
 * x: device [T][H] of the activation type. out: device [T][H] of the same
 * type, fully overwritten.
 * ids, gates, perm, offsets: exactly as hmoe_plan_routes wrote them for
 * these T tokens.
 * The result does not depend on tier_order or on the order of the tokens:
 * each output element is summed in a fixed order. */
hmoe_status hmoe_forward(const hmoe_layer* layer, const void* x, int T, const int32_t* ids,
                         const float* gates, const int32_t* perm, const int32_t* offsets,
                         void* out, void* ws, size_t ws_bytes, hmoe_stream_t stream);

/* hmoe_forward with options (hmoe_forward_opts: tier order, path, wait
 * limit, stage events). opts NULL is the defaults. Arguments, results and
 * errors otherwise as hmoe_forward.
 *   Cites: "quant: nvfp4_nf3_hybrid -- native serving ...", How it works (a
 *   second launch for the other tier into the same topk_sum, or one launch
 *   for both: tier_order chooses). */
hmoe_status hmoe_forward_ex(const hmoe_layer* layer, const void* x, int T, const int32_t* ids,
                            const float* gates, const int32_t* perm, const int32_t* offsets,
                            void* out, void* ws, size_t ws_bytes, const hmoe_forward_opts* opts,
                            hmoe_stream_t stream);

/* The same layer forward as hmoe_forward, for callers that cannot allocate
 * device memory and so cannot provide a workspace. Examples are hosts that
 * give a library only its input and output buffers under a fixed
 * device-memory plan (some serving engines and plugin interfaces), and code
 * that must never reach the allocator or cudaFree's implicit device-wide
 * synchronisation.
 *   Cites: the same passages as hmoe_forward (the computation); the pages
 *   have no counterpart for the scratch arrangement, a library convenience.
 *
 * Instead of a caller workspace, the call uses a file-scope device array of
 * HMOE_STATIC_SCRATCH_BYTES (16 MiB). Every GPU that loads the library
 * holds that array until the process exits. The call allocates nothing: no
 * cudaMalloc, no cudaFree, and no allocating library routine.
 * - Set-up: the first call on each device looks up the array's device
 *   address while that device is current. Make that first call before any
 *   stream capture begins.
 * - Size limit: a batch whose scratch would exceed the array returns
 *   HMOE_ERR_WORKSPACE_TOO_SMALL before anything is enqueued. For the
 *   256-expert layer (H=6144, I=2048, top-8) every T <= 51 fits; for the
 *   128-expert layer (H=2048, I=768, top-8) every T <= 151 fits.
 * - Checks: every argument check of hmoe_forward runs first; a call that
 *   returns an error has enqueued nothing.
 * - Sharing: all calls share the one array per device, and it keeps the
 *   last call's contents. Each call first clears, on the stream, the work
 *   queues and counters that must start at zero. The device status word is
 *   not cleared by a call: a fault any earlier call recorded stays until
 *   hmoe_check_device_status_static reads (and clears) it. Calls that
 *   overlap on the GPU (other streams, other threads) race on the array.
 *   Serialise them.
 * - Arguments and results are as in hmoe_forward with the default options
 *   (automatic path, one launch per GEMM). */
#define HMOE_STATIC_SCRATCH_BYTES (16u << 20)
hmoe_status hmoe_forward_static(const hmoe_layer* layer, const void* x, int T, const int32_t* ids,
                                const float* gates, const int32_t* perm, const int32_t* offsets, void* out,
                                hmoe_stream_t stream);

/* hmoe_check_device_status for the array used by hmoe_forward_static on the
 * current device. It synchronises the stream.
 *   Cites: as hmoe_check_device_status. */
hmoe_status hmoe_check_device_status_static(hmoe_stream_t stream);

/* Synchronise the stream and read the device status word the kernels write
 * into the workspace. Returns HMOE_OK, HMOE_ERR_BAD_ROUTE or
 * HMOE_ERR_DEVICE_TIMEOUT, then clears the word.
 *   Cites: "quant: add native mixed NVFP4/MXFP4 plus NF3 MoE serving",
 *   Summary (the hybrid metadata is validated; here the route geometry the
 *   kernels read is checked on the device, and bad entries are reported
 *   instead of trapping).
 * This is the one call that synchronises; it is not for use inside a stream
 * capture. HMOE_ERR_CUDA if the copy or the synchronisation fails (for
 * example after a fault elsewhere in the context). */
hmoe_status hmoe_check_device_status(void* ws, size_t ws_bytes, hmoe_stream_t stream);

/* Test export of the tensor-core operand. It writes, for one expert matrix
 * and in logical row order, the operand tile (of the activation type) that
 * the grouped (tcgen05) kernel writes to shared memory, decoded by the same
 * device function. which = 13 gives [2I][H]; which = 2 gives [H][I]. dst is
 * device memory. The values are e2m1*e4m3 (NVFP4, without the global scale),
 * e2m1*2^(b-127) (MXFP4), or rne(cb*s) (NF3; in fp16 with s first converted
 * to fp16), exact or rounded once to the activation type. The weight-streaming
 * kernel uses the same values for NVFP4 and MXFP4 but not for NF3: see
 * hmoe_debug_decode_operand.
 *   Cites: "quant: nvfp4_nf3_hybrid -- native serving ...", How it works
 *   (the NVFP4 and NF3 tier weights); "quant: add native mixed NVFP4/MXFP4
 *   plus NF3 MoE serving", Summary (MXFP4 as the kept format); "[Quantization]
 *   [ModelOpt] W4A16 NVFP4 fused MoE", Summary item 2 (the activation type).
 * Errors: HMOE_ERR_INVALID_ARG (NULL layer or dst, expert out of range,
 * which not 13 or 2), HMOE_ERR_CUDA. */
hmoe_status hmoe_debug_dequant(const hmoe_layer* layer, int expert, int which, void* dst,
                               hmoe_stream_t stream);

/* Test export of the weight-streaming (decode) kernel's operand, decoded by
 * the same device function that kernel runs. dst: device [N][K] of the
 * activation type, as in
 * hmoe_debug_dequant; scales: device fp32 [N][K/64]. The kernel computes each
 * output row as the sum over 64-wide K groups g of scales[n][g] times the
 * fp32 sum over the group of dst[n][k] * x[k] (NVFP4 then times its global
 * scale). NF3: dst is the raw codebook entry cb[code] and scales the group's
 * bf16 scale as fp32 (for W4A4 layers, whose h the streaming kernel must form
 * from the same weights as the tensor-core kernel: the tile of
 * hmoe_debug_dequant and scales 1); NVFP4 and MXFP4: dst is the tile of hmoe_debug_dequant and
 * scales are 1.
 *   Cites: as hmoe_debug_dequant. Errors as hmoe_debug_dequant (scales NULL
 *   is HMOE_ERR_INVALID_ARG). */
hmoe_status hmoe_debug_decode_operand(const hmoe_layer* layer, int expert, int which, void* dst,
                                      float* scales, hmoe_stream_t stream);

/* Global scales and tier of one expert, as the handle holds them: *fmt is
 * the expert's format (HMOE_FMT_*), the globals are 1 for MXFP4 and NF3.
 *   Cites: "quant: add native mixed NVFP4/MXFP4 plus NF3 MoE serving",
 *   Summary (hybrid_bit_map: the tier of each expert).
 * Errors: HMOE_ERR_INVALID_ARG (NULL layer, expert out of range). */
hmoe_status hmoe_layer_expert_info(const hmoe_layer* layer, int expert, int* fmt,
                                   float* w13_global, float* w2_global);

/* Free the handle (host memory only; the caller's device buffers are left
 * as they are). NULL is ignored.
 *   Cites: "quant: nvfp4_nf3_hybrid -- native serving ...", How it works (the
 *   two prepared weight objects of a layer, which the handle describes). */
void hmoe_layer_destroy(hmoe_layer* layer);

/* ------------------------------------------------------------ dense Linear W4A16
 * One weight matrix W [N, K] stored as NVFP4, MXFP4 or NF3 (the logical
 * layouts at the top of this file), times bf16 or fp16 activations:
 *   y[t][n] = sum_k x[t][k] * W[n][k], fp32 accumulation, a result of the
 *   activation type.
 *   Cites: "[Quantization][ModelOpt] W4A16 NVFP4 fused MoE +
 *   --override-activation-dtype flag", Summary and Related (the fused-MoE
 *   W4A16 support follows a dense-Linear W4A16 method: 4-bit weights, 16-bit
 *   activations, no activation scales).
 * The same kernels as the MoE layer run it: the matrix is packed like an
 * expert's W2 (tile layout), and a forward is the W2 phase of the
 * weight-streaming kernel (T <= 8) or of the tensor-core grouped kernel
 * (above) over one expert with one slot per token, then the finalize.
 * Conventions as for the layer: caller-owned device memory, asynchronous on
 * the stream, no allocation, argument errors before anything is enqueued,
 * device faults in the workspace's status word (hmoe_check_device_status).
 * Zero the workspace once before its first use (hmoe_workspace_init). */
typedef struct {
  int N;   /* output features, a multiple of 128 */
  int K;   /* input features, a multiple of 64 */
  int fmt;       /* HMOE_FMT_NVFP4, HMOE_FMT_MXFP4 or HMOE_FMT_NF3 */
  int act_dtype; /* hmoe_act_dtype (fp16 ranges as for the layer); 0 is bf16 */
} hmoe_linear_desc;

typedef struct hmoe_linear hmoe_linear; /* opaque host handle: no device memory */

/* Bytes of the packed matrix (the packed argument of hmoe_linear_pack).
 *   Cites: the dense-Linear passage of this section. Errors:
 *   HMOE_ERR_INVALID_ARG, HMOE_ERR_UNSUPPORTED_SHAPE (N % 128, K % 64). */
hmoe_status hmoe_linear_packed_size(const hmoe_linear_desc* desc, size_t* bytes);

/* Workspace bytes for hmoe_linear_forward at up to max_tokens rows: the
 * status word, the kernels' work queues, the one-expert route geometry and
 * the fp32 product [max_tokens][N].
 *   Cites: the dense-Linear passage of this section. */
hmoe_status hmoe_linear_workspace_size(const hmoe_linear_desc* desc, int max_tokens, size_t* bytes);

/* Repack W into the tile layout and create the handle. codes, scales: device
 * tensors in the logical layout of desc->fmt; global_scale: the NVFP4 fp32
 * global scale (ignored otherwise). packed: device buffer of
 * hmoe_linear_packed_size bytes, 16-byte aligned, alive while the handle is
 * used. The sources may be freed once the stream has passed this point.
 *   Cites: the dense-Linear passage of this section. */
hmoe_status hmoe_linear_pack(const hmoe_linear_desc* desc, const void* codes, const void* scales,
                             float global_scale, void* packed, hmoe_stream_t stream, hmoe_linear** out);

/* out[t][n] = act(sum_k x[t][k] W[n][k]). x: device [T][K] and out: device
 * [T][N], both of the activation type (act), out fully overwritten; both
 * 16-byte aligned. T = 0 is valid.
 *   Cites: the dense-Linear passage of this section. */
hmoe_status hmoe_linear_forward(const hmoe_linear* linear, const void* x, int T, void* out, void* ws,
                                size_t ws_bytes, hmoe_stream_t stream);

/* With options: path (HMOE_PATH_AUTO chooses the streaming kernel for T <= 8),
 * wait_limit_us and debug_flags as for hmoe_forward_ex (HMOE_DEBUG_GROUPED_PAIR
 * with fp16 is HMOE_ERR_INVALID_ARG); tier_order and stage_events are
 * ignored.
 *   Cites: the dense-Linear passage of this section. */
hmoe_status hmoe_linear_forward_ex(const hmoe_linear* linear, const void* x, int T, void* out, void* ws,
                                   size_t ws_bytes, const hmoe_forward_opts* opts, hmoe_stream_t stream);

/* Free the handle (host memory only). NULL is ignored.
 *   Cites: the dense-Linear passage of this section. */
void hmoe_linear_destroy(hmoe_linear* linear);

/* NVFP4 activation quantisation, the rule the W4A4 forward applies:
 *   for each block of 16 consecutive values of a row, in fp32 arithmetic
 *   (each operation correctly rounded),
 *     s = E4M3_rne(min(amax / (6 g), 448)),  d = e4m3(s) * g,
 *     q_i = E2M1_rne_sat(a_i / d) (0 where d = 0; ties to the even mantissa
 *     bit, saturating at 6; a value that rounds to 0 gives code 0).
 *   Cites: "[Quantization][ModelOpt] W4A16 NVFP4 fused MoE + ...", Summary.
 * x: device [rows][K] of act_dtype, 16-byte aligned; K a multiple of 16.
 * codes: device uint8 [rows][K/2] (element 2i in the low nibble), 8-byte
 * aligned; scales: device uint8 [rows][K/16] E4M3 bytes. The logical NVFP4
 * layout of this header, so the output can be dequantised like weights with
 * global scale g. global_scale: finite and > 0. rows = 0 is valid.
 * Errors: HMOE_ERR_INVALID_ARG (NULL or misaligned pointer, rows < 0, K not a
 * positive multiple of 16, bad act_dtype or scale), HMOE_ERR_CUDA. */
hmoe_status hmoe_quantize_act_nvfp4(const void* x, int rows, int K, int act_dtype, float global_scale,
                                    void* codes, void* scales, hmoe_stream_t stream);

/* Message for the last failing call on this thread ("" if none). Part of
 * the error convention at the top of this file; no page defines it. */
const char* hmoe_last_error(void);

/* Number of kernels this library has launched in this process so far (all
 * entry points). A library utility for launch accounting; no page defines it. */
uint64_t hmoe_launch_count(void);

/* Library version, major*10000 + minor*100 + patch. A library utility; no
 * page defines it. */
int hmoe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HMOE_H_ */
