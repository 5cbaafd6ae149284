// pack.cu -- repack one expert matrix from the logical checkpoint layout into tile layout,
// and the test-only export of the dequantised operand tiles.
//
// Cites: "quant: add native mixed NVFP4/MXFP4 plus NF3 MoE serving",
// Summary. Expert weights are demultiplexed into compact tier-local storage
// and repacked for the kernel. The tile layout is described in common.cuh.
// The pages' own kernel layout ("nf3_2p1", b12x #31) is for SM120 and is not
// reproduced.
#include "common.cuh"
#include "internal.h"

namespace hmoe {

ExpertGeom expert_geom(int H, int I, int fmt) {
  ExpertGeom g;
  g.H = H;
  g.I = I;
  g.rt13 = 2 * I / TILE_ROWS;
  g.kb13 = H / TILE_K;
  g.rt2 = H / TILE_ROWS;
  g.kb2 = I / TILE_K;
  g.tile = (size_t)tile_bytes(fmt);
  g.w13_bytes = (size_t)g.rt13 * g.kb13 * g.tile;
  g.w2_bytes = (size_t)g.rt2 * g.kb2 * g.tile;
  g.expert_bytes = g.w13_bytes + g.w2_bytes;
  return g;
}

// Logical row of tile-local row r (0..127) of row tile rt.
__device__ __forceinline__ int logical_row(int which, int I, int rt, int r) {
  if (which == 2) return rt * TILE_ROWS + r;
  const int w = r & 15, ch = rt * 64 + (r >> 4) * 8 + (w & 7);
  return (w < 8) ? ch : I + ch;
}

// NVFP4 code word: 8 codes laid out so that one AND (after a left shift of 0,
// 3 or 6 bits) puts a code pair's magnitude bits at bf16 bits 6..8 / 22..24
// and its sign at bit 15 / 31, i.e. a bf16 pair equal to 2^-126 times the
// E2M1 values (exponent field e, mantissa top bit m; e = 0 gives the
// subnormal m * 2^-127 = 0.5m * 2^-126). Pair (0,1) sits there unshifted,
// pair (2,3) 3 bits lower, pair (4,5) 6 bits lower; pair (6,7) fills the
// remaining bits: magnitude bits 0,1 at 10,11 / 26,27, bit 2 at 13 / 29,
// sign at 14 / 30.
__device__ __forceinline__ uint32_t e2m1s_word(const uint32_t* d) {
  uint32_t w = 0;
  const int base[3] = {6, 3, 0};
#pragma unroll
  for (int pr = 0; pr < 3; ++pr) {
    const uint32_t a = d[2 * pr], b = d[2 * pr + 1];
    w |= (a & 7u) << base[pr];
    w |= ((a >> 3) & 1u) << (base[pr] + 9);
    w |= (b & 7u) << (base[pr] + 16);
    w |= ((b >> 3) & 1u) << (base[pr] + 25);
  }
  const uint32_t a = d[6], b = d[7];
  w |= (a & 3u) << 10;
  w |= ((a >> 2) & 1u) << 13;
  w |= ((a >> 3) & 1u) << 14;
  w |= (b & 3u) << 26;
  w |= ((b >> 2) & 1u) << 29;
  w |= ((b >> 3) & 1u) << 30;
  return w;
}

__device__ __forceinline__ uint32_t e2m1_word(const uint32_t* d) {
  // d[0..7]: 4-bit codes. Layout: magnitudes in nibbles 0..7; signs of codes
  // 0..3 at bits 7,15,23,31 and of codes 4..7 at bits 3,11,19,27.
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w |= (d[i] & 7u) << (4 * i);
    w |= (d[4 + i] & 7u) << (16 + 4 * i);
    w |= ((d[i] >> 3) & 1u) << (8 * i + 7);
    w |= ((d[4 + i] >> 3) & 1u) << (8 * i + 3);
  }
  return w;
}

__global__ void pack_matrix_kernel(int fmt, int which, const uint8_t* __restrict__ codes,
                                   const uint8_t* __restrict__ scales, int N, int K, int I,
                                   uint8_t* __restrict__ dst, bool nvfp4_nibbles) {
  const int KB = K / TILE_K;
  const int rt = blockIdx.x / KB, kb = blockIdx.x % KB;
  const int tid = threadIdx.x, rg = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
  const int slot = rg * 32 + lane;
  const int R0 = rg * 16 + g, R1 = R0 + 8;
  const int L0 = logical_row(which, I, rt, R0), L1 = logical_row(which, I, rt, R1);
  const int k0 = kb * TILE_K + 16 * q;
  uint8_t* tile = dst + ((size_t)rt * KB + kb) * tile_bytes(fmt);
  if (fmt == FMT_NVFP4 || fmt == FMT_MXFP4) {
    uint32_t c0[16], c1[16];
    const uint8_t* s0 = codes + (size_t)L0 * (K / 2) + k0 / 2;
    const uint8_t* s1 = codes + (size_t)L1 * (K / 2) + k0 / 2;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      c0[2 * m] = s0[m] & 15u;
      c0[2 * m + 1] = s0[m] >> 4;
      c1[2 * m] = s1[m] & 15u;
      c1[2 * m + 1] = s1[m] >> 4;
    }
    uint4 v;
    if (fmt == FMT_NVFP4 && !nvfp4_nibbles) {
      v.x = e2m1s_word(c0);
      v.y = e2m1s_word(c0 + 8);
      v.z = e2m1s_word(c1);
      v.w = e2m1s_word(c1 + 8);
    } else {
      v.x = e2m1_word(c0);
      v.y = e2m1_word(c0 + 8);
      v.z = e2m1_word(c1);
      v.w = e2m1_word(c1 + 8);
    }
    *reinterpret_cast<uint4*>(tile + slot * 16) = v;
    if (fmt == FMT_NVFP4) {
      const uint32_t a = scales[(size_t)L0 * (K / 16) + k0 / 16];
      const uint32_t b = scales[(size_t)L1 * (K / 16) + k0 / 16];
      *reinterpret_cast<uint16_t*>(tile + 4096 + slot * 2) = (uint16_t)(a | (b << 8));
    } else if ((q & 1) == 0) {
      const uint32_t a = scales[(size_t)L0 * (K / 32) + k0 / 32];
      const uint32_t b = scales[(size_t)L1 * (K / 32) + k0 / 32];
      *reinterpret_cast<uint16_t*>(tile + 4096 + (rg * 16 + g * 2 + (q >> 1)) * 2) = (uint16_t)(a | (b << 8));
    }
  } else {
    // NF3: 16 codes = 48 bits starting at bit 3*k0 (a byte boundary: 6*q + 24*kb).
    uint64_t v0 = 0, v1 = 0;
    const uint8_t* s0 = codes + (size_t)L0 * (3 * K / 8) + 3 * k0 / 8;
    const uint8_t* s1 = codes + (size_t)L1 * (3 * K / 8) + 3 * k0 / 8;
#pragma unroll
    for (int m = 0; m < 6; ++m) {
      v0 |= (uint64_t)s0[m] << (8 * m);
      v1 |= (uint64_t)s1[m] << (8 * m);
    }
    uint32_t A = 0, B = 0, C = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t a0 = (uint32_t)(v0 >> (3 * j)) & 7u;
      const uint32_t b0 = (uint32_t)(v0 >> (3 * (8 + j))) & 7u;
      const uint32_t c0 = (uint32_t)(v1 >> (3 * j)) & 7u;
      const uint32_t d0 = (uint32_t)(v1 >> (3 * (8 + j))) & 7u;
      A |= (a0 | ((d0 & 1u) << 3)) << (4 * j);
      B |= (b0 | (((d0 >> 1) & 1u) << 3)) << (4 * j);
      C |= (c0 | (((d0 >> 2) & 1u) << 3)) << (4 * j);
    }
    *reinterpret_cast<uint32_t*>(tile + slot * 4) = A;
    *reinterpret_cast<uint32_t*>(tile + 1024 + slot * 4) = B;
    *reinterpret_cast<uint32_t*>(tile + 2048 + slot * 4) = C;
    if (q == 0) {
      const uint16_t* sc = reinterpret_cast<const uint16_t*>(scales);
      // the scales of R0 and R1 side by side: one 32-bit load per slot
      *reinterpret_cast<uint32_t*>(tile + 3072 + (rg * 8 + g) * 4) =
          (uint32_t)sc[(size_t)L0 * (K / 64) + kb] | ((uint32_t)sc[(size_t)L1 * (K / 64) + kb] << 16);
    }
  }
}

cudaError_t launch_pack_matrix(int fmt, int which, const void* codes, const void* scales, int N, int K, int I,
                               uint8_t* dst, bool nvfp4_nibbles, cudaStream_t st) {
  const int tiles = (N / TILE_ROWS) * (K / TILE_K);
  if (tiles == 0) return cudaSuccess;
  pack_matrix_kernel<<<tiles, 256, 0, st>>>(fmt, which, static_cast<const uint8_t*>(codes),
                                            static_cast<const uint8_t*>(scales), N, K, I, dst, nvfp4_nibbles);
  count_launches(1);
  return cudaGetLastError();
}

// ------------------------------------------------------------ debug export of operand tiles
// Both exports run dequant_slot, the decoder the GEMM kernels run, with the
// same shared tables the kernels build (E4M3; NF3 pairs in decode mode):
//   tile mode (WITH_NF3_SCALE = true): the operand tile (bf16 or fp16) the
//     tensor-core grouped kernel writes to shared memory. NVFP4 values in
//     bf16 are carried times 2^-63 inside the kernels (the factor returns
//     with the global scale), so the export multiplies 2^63 back, exactly.
//   decode mode (WITH_NF3_SCALE = false): the operand the weight-streaming
//     kernel feeds mma.sync. NVFP4 and MXFP4 are the tile values; NF3 values
//     are the raw codebook entries, and scales_out receives the fp32 factor
//     the kernel applies to each row's 64-wide group sum (1 for NVFP4/MXFP4).
template <int FMT, bool WITH_NF3_SCALE, int NLUT, int ACT>
__device__ __forceinline__ void debug_slot(const uint8_t* tile, int rg, int lane, const uint32_t* lut,
                                           uint32_t nf3_lut, uint32_t* r0, uint32_t* r1, float* s0, float* s1) {
  dequant_slot<FMT, WITH_NF3_SCALE, ACT, NLUT>(tile, rg, lane, r0, r1, s0, s1, lut, nf3_lut);
  if constexpr (FMT == FMT_NVFP4 && ACT == ACT_BF16) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      r0[i] = bf16x2_mul(r0[i], BF16X2_2P63);
      r1[i] = bf16x2_mul(r1[i], BF16X2_2P63);
    }
  }
}

template <bool WITH_NF3_SCALE, bool DECODE, int ACT>
__global__ void debug_dequant_kernel(int fmt, int which, const uint8_t* __restrict__ src, int N, int K, int I,
                                     uint16_t* __restrict__ dst, float* __restrict__ scales_out) {
  __shared__ uint32_t s_e4m3[256];
  __shared__ uint32_t s_nf3[NF3_LUT_WORDS];
  s_e4m3[threadIdx.x] = e4m3_lut_entry<ACT>(threadIdx.x);
  nf3_lut_fill<ACT>(s_nf3, threadIdx.x, blockDim.x);
  __syncthreads();
  const uint32_t nf3_lut = smem_u32(s_nf3) + 4u * (threadIdx.x & 31);
  const int KB = K / TILE_K;
  const int rt = blockIdx.x / KB, kb = blockIdx.x % KB;
  const int tid = threadIdx.x, rg = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
  const uint8_t* tile = src + ((size_t)rt * KB + kb) * tile_bytes(fmt);
  uint32_t r0[8], r1[8];
  float s0 = 1.0f, s1 = 1.0f;
  // The tensor-core kernel decodes NF3 with byte permutes only; the
  // weight-streaming kernel mixes the pair table and byte permutes.
  constexpr int NLUT = DECODE ? NF3_MIX_LUT : 0;
  if (fmt == FMT_NVFP4)
    debug_slot<FMT_NVFP4, WITH_NF3_SCALE, NLUT, ACT>(tile, rg, lane, s_e4m3, nf3_lut, r0, r1, &s0, &s1);
  else if (fmt == FMT_MXFP4)
    debug_slot<FMT_MXFP4, WITH_NF3_SCALE, NLUT, ACT>(tile, rg, lane, s_e4m3, nf3_lut, r0, r1, &s0, &s1);
  else debug_slot<FMT_NF3, WITH_NF3_SCALE, NLUT, ACT>(tile, rg, lane, s_e4m3, nf3_lut, r0, r1, &s0, &s1);
  const int L0 = logical_row(which, I, rt, rg * 16 + g), L1 = logical_row(which, I, rt, rg * 16 + g + 8);
  const int k0 = kb * TILE_K + 16 * q;
  uint4* d0 = reinterpret_cast<uint4*>(dst + (size_t)L0 * K + k0);
  uint4* d1 = reinterpret_cast<uint4*>(dst + (size_t)L1 * K + k0);
  d0[0] = make_uint4(r0[0], r0[1], r0[2], r0[3]);
  d0[1] = make_uint4(r0[4], r0[5], r0[6], r0[7]);
  d1[0] = make_uint4(r1[0], r1[1], r1[2], r1[3]);
  d1[1] = make_uint4(r1[4], r1[5], r1[6], r1[7]);
  if (scales_out && q == 0) {
    scales_out[(size_t)L0 * KB + kb] = s0;
    scales_out[(size_t)L1 * KB + kb] = s1;
  }
}

cudaError_t launch_debug_dequant(int fmt, int which, const uint8_t* src, int N, int K, int I, void* dst,
                                 float* scales_out, bool decode_operand, int act_type, bool nf3_tile,
                                 cudaStream_t st) {
  const int tiles = (N / TILE_ROWS) * (K / TILE_K);
  if (tiles == 0) return cudaSuccess;
  uint16_t* d = static_cast<uint16_t*>(dst);
  const bool f16 = act_type == ACT_F16;
  // decode mode: the streaming kernel's decoder (pair table and byte
  // permutes; NF3 tile values for W4A4 layers); tile mode: the tensor-core
  // kernel's.
  if (decode_operand && nf3_tile) {
    if (f16) debug_dequant_kernel<true, true, ACT_F16><<<tiles, 256, 0, st>>>(fmt, which, src, N, K, I, d, scales_out);
    else debug_dequant_kernel<true, true, ACT_BF16><<<tiles, 256, 0, st>>>(fmt, which, src, N, K, I, d, scales_out);
  } else if (decode_operand) {
    if (f16) debug_dequant_kernel<false, true, ACT_F16><<<tiles, 256, 0, st>>>(fmt, which, src, N, K, I, d, scales_out);
    else debug_dequant_kernel<false, true, ACT_BF16><<<tiles, 256, 0, st>>>(fmt, which, src, N, K, I, d, scales_out);
  } else {
    if (f16) debug_dequant_kernel<true, false, ACT_F16><<<tiles, 256, 0, st>>>(fmt, which, src, N, K, I, d, nullptr);
    else debug_dequant_kernel<true, false, ACT_BF16><<<tiles, 256, 0, st>>>(fmt, which, src, N, K, I, d, nullptr);
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace hmoe
