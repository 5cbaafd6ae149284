// internal.h -- launchers and host-side structures shared by the libhmoe translation units.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "common.cuh"

namespace hmoe {

// Count of kernel launches issued by the library (read by hmoe_launch_count).
void count_launches(int n);

// ---------------------------------------------------------------- routing
int route_chunks(int T);
cudaError_t launch_route(const float* logits, int T, int E, int k, int* ids, float* gates, int* perm,
                         int* offsets, int* chunk_cnt, int* chunk_base, cudaStream_t st);

// perm[t] = t, offsets = {0, T}, gates[t] = 1 (the dense Linear's route geometry).
cudaError_t launch_identity_route(int T, int* perm, int* offsets, float* gates, int num_sms, cudaStream_t st);

// ---------------------------------------------------------------- packing
// Geometry of one expert block inside a tier buffer: W13 tiles then W2 tiles.
struct ExpertGeom {
  int H, I;
  int rt13, kb13, rt2, kb2;  // row tiles / k-blocks of each matrix
  size_t tile;               // tile bytes of the format
  size_t w13_bytes, w2_bytes, expert_bytes;
};
ExpertGeom expert_geom(int H, int I, int fmt);

// nvfp4_nibbles: store NVFP4 codes in the nibble layout of MXFP4 (fp16 operand layers) instead of
// the shift-and-mask layout (bf16 operand layers).
cudaError_t launch_pack_matrix(int fmt, int which, const void* codes, const void* scales, int N, int K, int I,
                               uint8_t* dst, bool nvfp4_nibbles, cudaStream_t st);
// Test export of the dequantised operands (pack.cu): the tensor-core tile, or with
// decode_operand the weight-streaming kernel's operand plus its per-group scales.
cudaError_t launch_debug_dequant(int fmt, int which, const uint8_t* src, int N, int K, int I, void* dst,
                                 float* scales_out, bool decode_operand, int act_type, bool nf3_tile,
                                 cudaStream_t st);

// ---------------------------------------------------------------- streaming GEMM (any T; the decode path)
// Largest number of k-blocks per row tile in a pipeline stage of the
// streaming kernel (a stage holds two row tiles).
constexpr int STREAM_MAX_KBS = 4;
// The streaming kernel's work items are pairs of row tiles (one activation
// load serves both) when the batch can make at least this many W13 pair
// items per CTA, counting min(T * topk, E) token groups; else single row
// tiles, so that small batches keep more SMs busy. The choice depends only
// on the batch size and the layer, so every tier order of a forward makes
// the same choice and sums in the same order.
constexpr int STREAM_PAIR_MIN_ITEMS_PER_CTA = 2;
// One matrix of the expert FFN as the streaming kernel sees it.
struct StreamPhase {
  int rows, K;               // rows = 2I (W13) or H (W2); K = H or I
  int RT, KB;                // row tiles, k-blocks
  int kbs;                   // k-blocks per row tile and pipeline stage, items of two row tiles
  int kbs1;                  // k-blocks per pipeline stage, items of one row tile (up to 2 STREAM_MAX_KBS)
  const uint16_t* act;       // W13: x [T][H] by token; W2: h [S][I] by permuted position (operand type)
  int act_stride;
  size_t kept_off, nf3_off;  // byte offset of this matrix inside an expert's block
};

struct StreamParams {
  const uint8_t* kept_buf;
  const uint8_t* nf3_buf;
  int kept_fmt;
  int act_type;          // ACT_BF16 or ACT_F16: operand, h and output type
  float act_scale13;     // the W13 input's activation global scale (W4A4), else 1
  float act_scale2;      // the W2 input's activation global scale (W4A4), else 1
  int nf3_tile;          // 1: NF3 decoded to the tile values rne(cb * s) (W4A4 layers); 0: raw codes, scale on sums
  int H, I, E, topk, T;
  StreamPhase ph[2];     // [0] W13 (output h), [1] W2 (output y)
  int ph_begin, ph_end;  // phases this launch runs: [0,2) both (W2 items wait on done13), [0,1) or [1,2)
  int group_tokens;      // tokens per token group (<= 8)
  int pair_items;        // 1: work items are pairs of row tiles; 0: single row tiles
  int tier_mask;         // bit 0: kept experts, bit 1: NF3 experts
  size_t kept_expert_bytes, nf3_expert_bytes;
  const int* offsets;
  const int* perm;
  int* queue;                // [2] work-queue head and finished-CTA count, self-cleaning
  int* done13;               // [token groups] finished W13 warp-items per group, self-cleaning ([0,2) only)
  uint16_t* h_out;           // W13 output: [S][I] in the operand type (bf16 or fp16 bits), row = permuted position p
  float* y_out;              // W2 output:  [S][H] fp32, row = flat slot s
  int* status;
  unsigned long long wait_limit_ns;  // bound on every wait
  int debug_no_copies;               // test hook: the producer issues nothing
  ExpertTable tab;
};

int stream_grid(int num_sms);
cudaError_t launch_stream_gemm(const StreamParams& p, int grid, cudaStream_t st);

// ---------------------------------------------------------------- tensor-core grouped GEMM (large T)
struct GroupedParams {
  const uint8_t* kept_buf;
  const uint8_t* nf3_buf;
  int kept_fmt;
  int act_type;        // ACT_BF16 or ACT_F16
  float act_scale;     // this GEMM's input activation global scale (W4A4), else 1
  int which;           // 13: B = gathered x, output h;  2: B = h, output y
  int H, I, E, topk, T;
  int K, RT, KB;
  int tier_mask;
  size_t kept_expert_bytes, nf3_expert_bytes;
  size_t kept_w2_off, nf3_w2_off;
  const int* offsets;
  const int* perm;
  uint16_t* h_out;     // [S][I] in the operand type
  float* y_out;
  int* status;
  unsigned long long wait_limit_ns;
  int pair;            // 1: the CTA-pair kernel; 0: the one-CTA kernel (the default)
  ExpertTable tab;
};
cudaError_t launch_grouped_gemm(const GroupedParams& p, const uint16_t* b_src, int b_rows, int num_sms,
                                cudaStream_t st);
// xg[p] = x[perm[p] / k] for the S permuted slots (2-byte elements of either operand type).
cudaError_t launch_gather_rows(const uint16_t* x, const int* perm, int S, int k, int T, int H, uint16_t* xg,
                               int* status, int num_sms, cudaStream_t st);

// NVFP4 activation quantisation of n_values (a multiple of 16, rows of a
// multiple of 16 laid end to end) with global scale g (actquant.cu). With
// out set: the operand values e2m1 * e4m3 in the activation type (out may be
// x); else the codes (8 bytes per 16 values) and E4M3 scale bytes.
cudaError_t launch_act_quant(const uint16_t* x, long long n_values, float g, int act_type, uint16_t* out,
                             uint8_t* codes, uint8_t* scales, int num_sms, cudaStream_t st);

// out[t][c] = act(sum_j gates[t*k+j] * y[t*k+j][c]), act = bf16 or fp16 by act_type
cudaError_t launch_finalize(const float* y, const float* gates, int T, int k, int H, uint16_t* out, int act_type,
                            cudaStream_t st);

// Raises a kernel's dynamic shared-memory limit once per device: the
// attribute belongs to the current device, so a process that launches on
// several GPUs sets it on each. done is the kernel's bit mask of devices
// already set (ids 0..63; a higher id sets it on every call).
template <typename Kernel>
inline cudaError_t ensure_smem_attr(Kernel* kernel, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

}  // namespace hmoe
