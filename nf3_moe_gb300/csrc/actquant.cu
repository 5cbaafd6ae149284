// actquant.cu -- NVFP4 activation quantisation for the W4A4 layer.
//
// Cites: "[Quantization][ModelOpt] W4A16 NVFP4 fused MoE +
// --override-activation-dtype flag", Summary: the W4A4 NVFP4 scheme takes
// static NVFP4 weights and activations quantised to NVFP4 as they arrive
// (per-16 block scales computed from the data, a static global scale g).
//
// Per block of 16 consecutive values of a row, every decision in fp32:
//   s = E4M3_rne(min(amax / (6 g), 448)),  d = e4m3(s) * g,
//   q_i = E2M1_rne_sat(a_i / d)  (0 where d = 0).
// The multiply and the divisions are the correctly rounded fp32 operations
// (no contraction), so the codes do not depend on the compiler.
//
// Two outputs:
//   logical: the codes (two per byte, even k in the low nibble) and the
//     E4M3 scale bytes, the NVFP4 layout of the weights;
//   operand: the values e2m1(q) * e4m3(s) written back in the activation
//     type (exact in bf16 and in fp16), g left out for the GEMM epilogue to
//     apply in fp32. The tensor-core and streaming kernels then compute
//     exactly the W4A4 products.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace hmoe {

// E2M1 code of an fp32 value: round to nearest, ties to the even mantissa
// bit, saturating at 6; a value that rounds to 0 gives code 0 whatever its
// sign.
__device__ __forceinline__ uint32_t e2m1_code_rne_sat(float v) {
  const float a = fabsf(v);
  const uint32_t m = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
                     (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) + (uint32_t)(a > 5.0f);
  return m | ((signbit(v) && m) ? 8u : 0u);
}

// The E2M1 value of a code: exponent field e (bias 1), mantissa bit m;
// e = 0 is the subnormal 0.5 m, else 2^(e-1) (1 + m/2), built as fp32 bits.
__device__ __forceinline__ float e2m1_code_value(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  const float mag = e == 0 ? 0.5f * (float)m : __uint_as_float(((126u + e) << 23) | (m << 22));
  return (c & 8u) ? -mag : mag;
}

template <int ACT>
__device__ __forceinline__ float act_to_f32(uint16_t b) {
  if constexpr (ACT == ACT_F16) return __half2float(__ushort_as_half(b));
  else return bf16_bits_to_float(b);
}

// One thread per block of 16 values. OPERAND: write the operand values back
// to out (which may alias x); else write codes and scales.
template <int ACT, bool OPERAND>
__global__ void act_quant_kernel(const uint16_t* x, long long n_blocks, float g,
                                 uint16_t* out, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  const float six_g = __fmul_rn(6.0f, g);
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < n_blocks;
       b += (long long)gridDim.x * blockDim.x) {
    const uint4 lo = reinterpret_cast<const uint4*>(x)[2 * b];
    const uint4 hi = reinterpret_cast<const uint4*>(x)[2 * b + 1];
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    float a[16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      a[2 * i] = act_to_f32<ACT>((uint16_t)(w[i] & 0xFFFFu));
      a[2 * i + 1] = act_to_f32<ACT>((uint16_t)(w[i] >> 16));
      amax = fmaxf(amax, fmaxf(fabsf(a[2 * i]), fabsf(a[2 * i + 1])));
    }
    const float t = fminf(__fdiv_rn(amax, six_g), 448.0f);
    const uint32_t s = (uint32_t)__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
    const float sv = bf16_bits_to_float(e4m3_to_bf16(s));
    const float d = __fmul_rn(sv, g);
    uint32_t q[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = d > 0.0f ? e2m1_code_rne_sat(__fdiv_rn(a[i], d)) : 0u;
    if constexpr (OPERAND) {
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        o[i] = f32x2_to_act<ACT>(e2m1_code_value(q[2 * i]) * sv, e2m1_code_value(q[2 * i + 1]) * sv);
      reinterpret_cast<uint4*>(out)[2 * b] = make_uint4(o[0], o[1], o[2], o[3]);
      reinterpret_cast<uint4*>(out)[2 * b + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    } else {
      uint32_t c0 = 0, c1 = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c0 |= q[i] << (4 * i);
        c1 |= q[8 + i] << (4 * i);
      }
      reinterpret_cast<uint2*>(codes)[b] = make_uint2(c0, c1);
      scales[b] = (uint8_t)s;
    }
  }
}

cudaError_t launch_act_quant(const uint16_t* x, long long n_values, float g, int act_type, uint16_t* out,
                             uint8_t* codes, uint8_t* scales, int num_sms, cudaStream_t st) {
  const long long nb = n_values / 16;
  if (nb == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (nb + threads - 1) / threads;
  const dim3 grid((unsigned)(blocks < (long long)num_sms * 8 ? blocks : (long long)num_sms * 8));
  const bool operand = out != nullptr;
  cudaError_t e;
  if (act_type == ACT_F16)
    e = operand ? launch_pdl(act_quant_kernel<ACT_F16, true>, grid, dim3(threads), 0, st, x, nb, g, out, codes, scales)
                : launch_pdl(act_quant_kernel<ACT_F16, false>, grid, dim3(threads), 0, st, x, nb, g, out, codes, scales);
  else
    e = operand ? launch_pdl(act_quant_kernel<ACT_BF16, true>, grid, dim3(threads), 0, st, x, nb, g, out, codes, scales)
                : launch_pdl(act_quant_kernel<ACT_BF16, false>, grid, dim3(threads), 0, st, x, nb, g, out, codes, scales);
  count_launches(1);
  return e;
}

}  // namespace hmoe
