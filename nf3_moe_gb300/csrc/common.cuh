// common.cuh -- device helpers shared by the libhmoe kernels (sm_103a).
//
// Packed tile layout (this library's choice; the pages leave it open, and the
// "nf3_2p1" layout of "quant: nvfp4_nf3_hybrid ...", Depends on, is prior art
// for SM120 only):
//
//   A tile is 128 weight rows x 64 K (one "k-block"). One expert matrix is
//   stored as tiles ordered (row tile rt, k-block kb) with kb fastest, so a
//   row tile's K extent is one contiguous byte range. Inside a tile, rows
//   form 8 groups of 16 (rg = 0..7). Thread slot (rg, lane), with
//   g = lane / 4 and q = lane % 4, owns rows R0 = 16 rg + g and R1 = R0 + 8,
//   and logical k = 16 q .. 16 q + 15 of the k-block. This is the A-fragment
//   ownership of an m16n8k16 MMA after permuting K inside each k-block. The
//   same slot also drives the tensor-core tile writer.
//
//   NVFP4 tile, 4608 B: codes [256 slots][16 B] = [R0 w0, R0 w1, R1 w0, R1 w1].
//     Each 32-bit word holds 8 E2M1 codes. The magnitude of code i (i<4) is
//     in nibble i bits 0..2, and code 4+i in nibble 4+i. The sign bits sit
//     in the nibbles' bit 3: code 0..3 at bits 7, 15, 23, 31 and code 4..7
//     at bits 3, 11, 19, 27. Then scales: [256 slots][2 B] = E4M3 of
//     (R0, group q) and (R1, group q).
//   MXFP4 tile, 4352 B: codes as NVFP4. Scales [8 rg][8 g][2 halves][2 B]
//     = E8M0 of (R0, q/2) and (R1, q/2).
//   NF3 tile, 3328 B: three words per slot, A at 0, B at 1024, C at 2048
//     (each [256 slots][4 B]). A's nibbles 0..7 hold R0 codes 0..7, B's hold
//     R0 codes 8..15, C's hold R1 codes 0..7, each in bits 0..2. Bit 3 of
//     nibble j in A, B and C holds bits 0, 1 and 2 of R1 code 8+j. Then bf16
//     scales at 3072: [8 rg][8 g][R0, R1][2 B], the two rows of a slot side
//     by side.
//   W13 rows are interleaved per 16-row group: group rows 0..7 are the gate
//   rows of 8 consecutive channels and rows 8..15 the up rows of the same
//   channels. So R0 and R1 of a thread slot are the gate and up rows of one
//   channel.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace hmoe {

constexpr int FMT_NF3 = 3, FMT_NVFP4 = 4, FMT_MXFP4 = 5;
constexpr int TILE_ROWS = 128;
constexpr int TILE_K = 64;
constexpr int MAX_E = 512;
constexpr int MAX_TOPK = 32;

__host__ __device__ constexpr int tile_bytes(int fmt) {
  return fmt == FMT_NVFP4 ? 4608 : (fmt == FMT_MXFP4 ? 4352 : 3328);
}

// Device status word codes (bit flags, OR-ed by kernels).
constexpr int DEV_TIMEOUT = 1;
constexpr int DEV_BAD_ROUTE = 2;

// Per-expert table passed by value in kernel parameters.
struct ExpertTable {
  uint16_t loc[MAX_E];        // tier-local index; bit 15 set = NF3 tier
  float g13[MAX_E];           // W13 global scale (NVFP4), else 1
  float g2[MAX_E];
};
constexpr uint16_t LOC_NF3 = 0x8000;

// NF3 codebook as bf16 bit patterns (kernel copy), index 0..7.
constexpr uint16_t NF3_CB[8] = {0xBF80, 0xBF09, 0xBE7D, 0x0000, 0x3E3C, 0x3EC4, 0x3F1F, 0x3F80};
// Byte tables for prmt lookups: low bytes and high bytes of the 8 entries.
constexpr uint32_t NF3_LO0 = 0x007D0980u, NF3_LO1 = 0x801FC43Cu;
constexpr uint32_t NF3_HI0 = 0x00BEBFBFu, NF3_HI1 = 0x3F3F3E3Eu;
// E2M1 magnitudes {0,.5,1,1.5,2,3,4,6} as bf16: low bytes and high bytes.
constexpr uint32_t E2M1_LO0 = 0xC0800000u, E2M1_LO1 = 0xC0804000u;
constexpr uint32_t E2M1_HI0 = 0x3F3F3F00u, E2M1_HI1 = 0x40404040u;

// Activation (operand) types: the MMA operands, h and the output are bf16 or
// fp16; the weights are decoded to the same type.
constexpr int ACT_BF16 = 0, ACT_F16 = 1;
// The same tables for fp16 operands. The E2M1 magnitudes in fp16 have zero
// low bytes ({0000, 3800, 3C00, 3E00, 4000, 4200, 4400, 4600}), so one table
// of high bytes serves; the NF3 entries in fp16 are the bf16 values exactly
// ({BC00, B848, B3E8, 0000, 31E0, 3620, 38F8, 3C00}).
constexpr uint32_t E2M1F_HI0 = 0x3E3C3800u, E2M1F_HI1 = 0x46444240u;
constexpr uint32_t NF3F_LO0 = 0x00E84800u, NF3F_LO1 = 0x00F820E0u;
constexpr uint32_t NF3F_HI0 = 0x00B3B8BCu, NF3F_HI1 = 0x3C383631u;

// ---------------------------------------------------------------- generic helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicOr(status, code);
}

// ---------------------------------------------------------------- mbarrier + bulk copy
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// The suspend-time hint lets a waiting thread sleep inside the instruction
// (up to the hint, in ns; the phase completing wakes it) instead of spinning
// on short polls that take issue slots from the working warps. Measured on
// the prefill kernel: 3.37 -> 3.30 ms at M=4096 for any hint of 20 ns to 2 us.
constexpr uint32_t MBAR_SUSPEND_HINT_NS = 500;
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(MBAR_SUSPEND_HINT_NS)
      : "memory");
  return ok != 0;
}

// Non-blocking probe: true if the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete. The wait is bounded:
// it returns false if *abort becomes non-zero or after limit_ns.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns = WAIT_LIMIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
}

// Orders this thread's generic-proxy global accesses with later (or, on
// the writing side, other threads' later) async-proxy accesses such as
// bulk copies.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Spins (bounded like mbar_wait) until the gpu-scope acquire load of *ctr
// is at least target. Returns false on abort or timeout.
__device__ __forceinline__ bool wait_count_at_least(const int* ctr, int target, volatile int* abort,
                                                    uint64_t limit_ns = WAIT_LIMIT_NS) {
  auto load = [ctr]() {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    return v;
  };
  if (load() >= target) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (load() >= target) return true;
    if ((it & 15u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
}

// 1D bulk copy (TMA engine, non-tensor form) global -> this CTA's shared memory.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Same, with an L2 evict-first policy for data read once (streamed weights).
__device__ __forceinline__ void bulk_g2s_stream(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// From a converged warp: one elected lane registers the expected bytes on the
// barrier and issues the weight copy (L2 evict-first policy), in one warp
// instruction sequence without a branch.
__device__ __forceinline__ void bulk_expect_and_copy_elect(void* dst, const void* src, uint32_t bytes,
                                                           uint32_t expect_bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%3], %4;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %5;\n\t}" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "r"(expect_bytes), "l"(policy)
      : "memory");
}
// Same with two weight ranges of the same size (the second only if second
// is set) under one expected byte count.
__device__ __forceinline__ void bulk_expect_and_copy2_elect(void* dst0, const void* src0, void* dst1, const void* src1,
                                                            uint32_t bytes, bool second, uint32_t expect_bytes,
                                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred e, t;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.and.b32 t, %7, 0, e;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%3], %4;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %5;\n\t"
      "@t cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%6], [%8], %2, [%3], %5;\n\t}" ::"r"(
          smem_u32(dst0)),
      "l"(src0), "r"(bytes), "r"(smem_u32(bar)), "r"(expect_bytes), "l"(policy), "r"(smem_u32(dst1)),
      "r"(second ? 1u : 0u), "l"(src1)
      : "memory");
}
// A bulk copy issued by every lane whose predicate is set, in one warp
// instruction (the lanes' copies are independent requests).
__device__ __forceinline__ void bulk_g2s_if(bool pred, void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred q;\n\t"
      "setp.ne.b32 q, %4, 0;\n\t"
      "@q cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "r"(pred ? 1u : 0u)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Programmatic dependent launch. A kernel launched with launch_pdl may start
// while its predecessor on the stream is still running. pdl_wait() blocks
// until the predecessor grid has completed and its writes are visible, so
// it must come before the kernel's first global read or write. Only
// shared-memory setup may precede it. pdl_trigger() lets the next kernel
// be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- bf16 helpers
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16_bcast(uint16_t b) { return (uint32_t)b | ((uint32_t)b << 16); }

// E4M3 byte -> bf16 bits. Exact: every E4M3 value is a bf16 value.
__device__ __forceinline__ uint16_t e4m3_to_bf16(uint32_t byte) {
  uint32_t s = (byte & 0x80u) << 8;
  uint32_t e = (byte >> 3) & 15u, m = byte & 7u;
  if (e == 0) {
    // subnormal m/8 * 2^-6 = m * 2^-9 -> normalise via float
    float f = (float)m * 0.001953125f;
    return (uint16_t)(s | (__float_as_uint(f) >> 16));
  }
  if (e == 15 && m == 7) return (uint16_t)(s | 0x7FC0u);  // NaN (never produced by encoders)
  return (uint16_t)(s | ((e + 120u) << 7) | (m << 4));
}
// E8M0 byte -> bf16 bits of 2^(b-127). b = 0 is the bf16 subnormal 2^-127.
__device__ __forceinline__ uint16_t e8m0_to_bf16(uint32_t byte) {
  if (byte == 0) return 0x0040;
  if (byte == 255) return 0x7FC0;
  return (uint16_t)(byte << 7);
}
__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <int ACT>
__device__ __forceinline__ uint32_t mul_x2(uint32_t a, uint32_t b) {
  if constexpr (ACT == ACT_F16) return f16x2_mul(a, b);
  else return bf16x2_mul(a, b);
}
// fp32 -> fp16 bits, round to nearest even (exact for the values used here).
__device__ __forceinline__ uint16_t f32_to_f16_bits(float f) { return __half_as_ushort(__float2half_rn(f)); }
// E4M3 byte -> fp16 bits (exact: every E4M3 value is an fp16 value).
__device__ __forceinline__ uint16_t e4m3_to_f16(uint32_t byte) {
  return f32_to_f16_bits(bf16_bits_to_float(e4m3_to_bf16(byte)));
}
// E8M0 byte -> fp16 bits of 2^(b-127). Exact for b in 103..142 (fp16
// subnormals included); outside that range the scale is unsupported for fp16
// operands (rounds to 0 or to infinity).
__device__ __forceinline__ uint16_t e8m0_to_f16(uint32_t byte) {
  if (byte == 0 || byte == 255) return byte ? 0x7E00 : 0;
  return f32_to_f16_bits(__uint_as_float(byte << 23));
}
// Output conversions of the fp32 results.
template <int ACT>
__device__ __forceinline__ uint16_t f32_to_act(float f) {
  if constexpr (ACT == ACT_F16) return __half_as_ushort(__float2half_rn(f));
  else return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
template <int ACT>
__device__ __forceinline__ uint32_t f32x2_to_act(float a, float b) {
  return (uint32_t)f32_to_act<ACT>(a) | ((uint32_t)f32_to_act<ACT>(b) << 16);
}

// ---------------------------------------------------------------- code word decoders
// 8 E2M1 codes (word layout in the header comment) -> 4 bf16x2 (codes 0,1 | 2,3 | 4,5 | 6,7).
__device__ __forceinline__ void e2m1x8_to_bf16x2(uint32_t w, uint32_t* p) {
  const uint32_t m = w & 0x77777777u;
  uint32_t lo = __byte_perm(E2M1_LO0, E2M1_LO1, m);
  uint32_t hi = __byte_perm(E2M1_HI0, E2M1_HI1, m) | (w & 0x80808080u);
  p[0] = __byte_perm(lo, hi, 0x5140);
  p[1] = __byte_perm(lo, hi, 0x7362);
  const uint32_t m2 = m >> 16;
  lo = __byte_perm(E2M1_LO0, E2M1_LO1, m2);
  hi = __byte_perm(E2M1_HI0, E2M1_HI1, m2) | ((w << 4) & 0x80808080u);
  p[2] = __byte_perm(lo, hi, 0x5140);
  p[3] = __byte_perm(lo, hi, 0x7362);
}

// 8 NVFP4 codes (the shift-and-mask word layout written by the packer) ->
// 4 bf16x2 holding 2^-126 times the E2M1 values. Multiplied by a scale that
// carries 2^63 (an exact bf16 product: at most 6 significant bits, never
// below the normal range), they give 2^-63 times the dequantised weights;
// the factor 2^63 returns with the global scale after the fp32 accumulation.
constexpr float NVFP4_UNSCALE = 9.223372036854775808e18f;  // 2^63
constexpr uint32_t BF16X2_2P63 = 0x5F005F00u;               // bf16 pair of 2^63
__device__ __forceinline__ void e2m1s_to_bf16x2(uint32_t w, uint32_t* p) {
  constexpr uint32_t M = 0x81C081C0u;
  p[0] = w & M;
  p[1] = (w << 3) & M;
  p[2] = (w << 6) & M;
  p[3] = ((w >> 4) & 0x00C000C0u) | ((w >> 5) & 0x01000100u) | ((w << 1) & 0x80008000u);
}

// 8 NF3 codes held as selector nibbles (bit 3 of each nibble clear) -> 4 bf16x2.
__device__ __forceinline__ void nf3x8_to_bf16x2(uint32_t sel, uint32_t* p) {
  uint32_t lo = __byte_perm(NF3_LO0, NF3_LO1, sel);
  uint32_t hi = __byte_perm(NF3_HI0, NF3_HI1, sel);
  p[0] = __byte_perm(lo, hi, 0x5140);
  p[1] = __byte_perm(lo, hi, 0x7362);
  sel >>= 16;
  lo = __byte_perm(NF3_LO0, NF3_LO1, sel);
  hi = __byte_perm(NF3_HI0, NF3_HI1, sel);
  p[2] = __byte_perm(lo, hi, 0x5140);
  p[3] = __byte_perm(lo, hi, 0x7362);
}

// 8 E2M1 codes (the nibble word layout of e2m1x8_to_bf16x2) -> 4 fp16x2.
// The fp16 values have zero low bytes: one lookup of high bytes, the sign
// OR-ed in, and two byte permutations that interleave zero low bytes.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t* p) {
  const uint32_t m = w & 0x77777777u;
  const uint32_t hi = __byte_perm(E2M1F_HI0, E2M1F_HI1, m) | (w & 0x80808080u);
  p[0] = __byte_perm(hi, 0u, 0x1404);
  p[1] = __byte_perm(hi, 0u, 0x3424);
  const uint32_t hi2 = __byte_perm(E2M1F_HI0, E2M1F_HI1, m >> 16) | ((w << 4) & 0x80808080u);
  p[2] = __byte_perm(hi2, 0u, 0x1404);
  p[3] = __byte_perm(hi2, 0u, 0x3424);
}

// 8 NF3 codes held as selector nibbles -> 4 fp16x2 (table values, unscaled).
__device__ __forceinline__ void nf3x8_to_f16x2(uint32_t sel, uint32_t* p) {
  uint32_t lo = __byte_perm(NF3F_LO0, NF3F_LO1, sel);
  uint32_t hi = __byte_perm(NF3F_HI0, NF3F_HI1, sel);
  p[0] = __byte_perm(lo, hi, 0x5140);
  p[1] = __byte_perm(lo, hi, 0x7362);
  sel >>= 16;
  lo = __byte_perm(NF3F_LO0, NF3F_LO1, sel);
  hi = __byte_perm(NF3F_HI0, NF3F_HI1, sel);
  p[2] = __byte_perm(lo, hi, 0x5140);
  p[3] = __byte_perm(lo, hi, 0x7362);
}

// NF3 pair table in shared memory, the lookup the kernels use instead of
// nf3x8_to_bf16x2 / nf3x8_to_f16x2 (measured 72 against 52 decoded weights
// per clock per SM: one byte extract on the ALU pipe, one multiply-add on
// the FMA pipe and one shared load per code pair, instead of about 2.25 ALU
// operations). Entry i, a byte of a selector word (code a in bits 0..2, code
// b in bits 4..6; bits 3 and 7 clear), holds the operand pair (cb[a], cb[b])
// of the operand type. The table is replicated once per bank: entry i of
// lane l is word i * 32 + l, so the lanes of a warp read 32 different banks
// whatever entries they look up.
constexpr int NF3_LUT_ENTRIES = 0x78;  // the largest selector byte is 0x77
constexpr int NF3_LUT_WORDS = NF3_LUT_ENTRIES * 32;
constexpr int NF3_LUT_BYTES = NF3_LUT_WORDS * 4;

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Fills the table (all threads of the block take part; a barrier must follow).
template <int ACT>
__device__ __forceinline__ void nf3_lut_fill(uint32_t* tab, int tid, int nthreads) {
  for (int w = tid; w < NF3_LUT_WORDS; w += nthreads) {
    uint32_t p[4];
    if constexpr (ACT == ACT_F16) nf3x8_to_f16x2((uint32_t)(w >> 5) & 0x77u, p);
    else nf3x8_to_bf16x2((uint32_t)(w >> 5) & 0x77u, p);
    tab[w] = p[0];
  }
}

// 8 NF3 codes held as selector nibbles -> 4 operand pairs, from the table.
// lut: the shared address of entry 0 of this lane (table base + 4 * lane).
__device__ __forceinline__ void nf3x8_lut(uint32_t sel, uint32_t lut, uint32_t* p) {
  p[0] = lds_u32(lut + __byte_perm(sel, 0u, 0x4440) * 128u);
  p[1] = lds_u32(lut + __byte_perm(sel, 0u, 0x4441) * 128u);
  p[2] = lds_u32(lut + __byte_perm(sel, 0u, 0x4442) * 128u);
  p[3] = lds_u32(lut + __byte_perm(sel, 0u, 0x4443) * 128u);
}

// The weight-streaming kernel's NF3 decode mix: selector words per slot
// taken through the pair table (of 4), the rest decoded with byte-table
// permutes. The table costs shared-memory bandwidth (one 128-byte wavefront
// per warp and code pair), the permutes ALU issue (about 2.25 operations
// per pair); with 16 consumer warps per SM sharing both, a mix keeps either
// from saturating. Measured per M=8 launch with single-tile items (table
// words of 4): 4: 249.0 us, 3 and 2 alternating: 242.6, 2: 242.1, 2 and 1:
// 245.4, 1: 249.3, 0: 257.4; with items of two row tiles, which load the
// activations once for both and leave more shared-memory bandwidth to the
// table: 4: 231.8, 3: 229.2 to 231.3, 2: 237.4, 1: 243.6. At M=2 (single-tile
// items) 3 words took 83.8 us, 2 words 90.0.
constexpr int NF3_MIX_LUT = 3;

// NF3 words A, B, C of one thread slot -> selector words for R0 codes 0..7,
// R0 8..15, R1 0..7 and R1 8..15.
__device__ __forceinline__ void nf3_selectors(uint32_t A, uint32_t B, uint32_t C, uint32_t* s) {
  s[0] = A & 0x77777777u;
  s[1] = B & 0x77777777u;
  s[2] = C & 0x77777777u;
  // Bits 4j+3 of A, B, C are bits 0, 1, 2 of code 8+j.
  s[3] = ((A >> 3) & 0x11111111u) | ((B >> 2) & 0x22222222u) | ((C >> 1) & 0x44444444u);
}

// Load one thread slot's packed data from a tile in shared memory and
// produce its dequantised operand pairs (bf16x2 or fp16x2 by ACT): r0[8] for
// row R0 (k pairs in order) and r1[8] for row R1. With with_nf3_scale ==
// false the NF3 values are raw codebook entries, and scale0/scale1 return the
// two row scales as floats for the caller to apply to fp32 sums. Otherwise
// every format's values come out multiplied by their scale (the "tile"
// values; NF3 rounded once to the operand type). NVFP4 tile values in bf16
// come out times 2^-63 (see e2m1s_to_bf16x2; nvfp4_unscale<ACT> returns the
// factor), in fp16 exactly.
// e4m3_lut: the 256-entry table of E4M3 scale pairs of the operand type,
// built by every kernel that decodes NVFP4 with e4m3_lut_entry<ACT>, indexed
// by the scale bytes directly (shared memory).
template <int ACT>
__device__ __forceinline__ uint32_t e4m3_lut_entry(uint32_t byte) {
  if constexpr (ACT == ACT_F16) return bf16_bcast(e4m3_to_f16(byte));
  else return bf16x2_mul(bf16_bcast(e4m3_to_bf16(byte)), BF16X2_2P63);
}
template <int ACT>
__host__ __device__ constexpr float nvfp4_unscale() {
  return ACT == ACT_F16 ? 1.0f : NVFP4_UNSCALE;
}
// NF3_LUT (0..4): how many of the slot's four NF3 selector words are looked
// up in the shared pair table whose lane address is nf3_lut (see
// nf3x8_lut); the others are decoded with byte-table permutes. The values
// are the same either way.
template <int FMT, bool WITH_NF3_SCALE, int ACT = ACT_BF16, int NF3_LUT = 0>
__device__ __forceinline__ void dequant_slot(const uint8_t* tile, int rg, int lane, uint32_t* r0, uint32_t* r1,
                                             float* scale0, float* scale1, const uint32_t* e4m3_lut,
                                             uint32_t nf3_lut = 0) {
  const int slot = rg * 32 + lane;
  if constexpr (FMT == FMT_NVFP4 || FMT == FMT_MXFP4) {
    const uint4 q = *reinterpret_cast<const uint4*>(tile + slot * 16);
    uint32_t s0, s1;
    if constexpr (FMT == FMT_NVFP4) {
      s0 = e4m3_lut[tile[4096 + slot * 2]];
      s1 = e4m3_lut[tile[4096 + slot * 2 + 1]];
    } else {
      const int g = lane >> 2, hq = (lane & 3) >> 1;
      const uint32_t sc = *reinterpret_cast<const uint16_t*>(tile + 4096 + (rg * 16 + g * 2 + hq) * 2);
      if constexpr (ACT == ACT_F16) {
        s0 = bf16_bcast(e8m0_to_f16(sc & 0xFFu));
        s1 = bf16_bcast(e8m0_to_f16(sc >> 8));
      } else {
        s0 = bf16_bcast(e8m0_to_bf16(sc & 0xFFu));
        s1 = bf16_bcast(e8m0_to_bf16(sc >> 8));
      }
    }
    if constexpr (ACT == ACT_F16) {
      // fp16 layers store NVFP4 codes in the nibble layout of MXFP4.
      e2m1x8_to_f16x2(q.x, r0);
      e2m1x8_to_f16x2(q.y, r0 + 4);
      e2m1x8_to_f16x2(q.z, r1);
      e2m1x8_to_f16x2(q.w, r1 + 4);
    } else if constexpr (FMT == FMT_NVFP4) {
      e2m1s_to_bf16x2(q.x, r0);
      e2m1s_to_bf16x2(q.y, r0 + 4);
      e2m1s_to_bf16x2(q.z, r1);
      e2m1s_to_bf16x2(q.w, r1 + 4);
    } else {
      e2m1x8_to_bf16x2(q.x, r0);
      e2m1x8_to_bf16x2(q.y, r0 + 4);
      e2m1x8_to_bf16x2(q.z, r1);
      e2m1x8_to_bf16x2(q.w, r1 + 4);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      r0[i] = mul_x2<ACT>(r0[i], s0);
      r1[i] = mul_x2<ACT>(r1[i], s1);
    }
    *scale0 = 1.0f;
    *scale1 = 1.0f;
  } else {
    const uint32_t A = *reinterpret_cast<const uint32_t*>(tile + slot * 4);
    const uint32_t B = *reinterpret_cast<const uint32_t*>(tile + 1024 + slot * 4);
    const uint32_t C = *reinterpret_cast<const uint32_t*>(tile + 2048 + slot * 4);
    const int g = lane >> 2;
    const uint32_t sbb = *reinterpret_cast<const uint32_t*>(tile + 3072 + (rg * 8 + g) * 4);
    const uint32_t sb0 = sbb & 0xFFFFu, sb1 = sbb >> 16;
    uint32_t s[4];
    nf3_selectors(A, B, C, s);
    static_assert(NF3_LUT >= 0 && NF3_LUT <= 4, "selector words through the table");
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t* p = (w < 2 ? r0 : r1) + 4 * (w & 1);  // s[0], s[1]: R0 codes 0..15; s[2], s[3]: R1
      if (w < NF3_LUT) nf3x8_lut(s[w], nf3_lut, p);
      else if constexpr (ACT == ACT_F16) nf3x8_to_f16x2(s[w], p);
      else nf3x8_to_bf16x2(s[w], p);
    }
    if constexpr (WITH_NF3_SCALE) {
      uint32_t S0, S1;
      if constexpr (ACT == ACT_F16) {
        // the bf16 scale as fp16 (exact for scales in the fp16 normal range)
        S0 = bf16_bcast(f32_to_f16_bits(bf16_bits_to_float(sb0)));
        S1 = bf16_bcast(f32_to_f16_bits(bf16_bits_to_float(sb1)));
      } else {
        S0 = bf16_bcast((uint16_t)sb0);
        S1 = bf16_bcast((uint16_t)sb1);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        r0[i] = mul_x2<ACT>(r0[i], S0);
        r1[i] = mul_x2<ACT>(r1[i], S1);
      }
      *scale0 = 1.0f;
      *scale1 = 1.0f;
    } else {
      *scale0 = bf16_bits_to_float(sb0);
      *scale1 = bf16_bits_to_float(sb1);
    }
  }
}

// ---------------------------------------------------------------- mma.sync (decode path)
template <int ACT = ACT_BF16>
__device__ __forceinline__ void mma_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                          uint32_t b1) {
  if constexpr (ACT == ACT_F16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same MMA with a zero accumulator input (d = a * b).
template <int ACT = ACT_BF16>
__device__ __forceinline__ void mma_16816_zc(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  if constexpr (ACT == ACT_F16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }
// silu with the fast exponential and divide intrinsics (relative error a few
// ulp of fp32; the result is rounded to bf16 right after).
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

}  // namespace hmoe
