// grouped.cu -- the tensor-core grouped GEMM for large batches (prefill): tcgen05 + TMEM + TMA.
//
// Cites: "quant: nvfp4_nf3_hybrid -- native serving for mixed NVFP4+NF3 MoE
// checkpoints", How it works. Both weight tiers feed one fused MoE GEMM
// over the shared route geometry. "[Quantization][ModelOpt] W4A16 NVFP4
// fused MoE", Summary. W4A16: weights dequantised to the 16-bit activation
// type, with no activation quantisation.
//
// One persistent CTA per SM takes work items (expert e, token tile nt of up
// to 128 permuted slots, a pair of weight row tiles rt, rt+1 of 128 rows
// each), with row-tile pairs fastest. The tokens sit on the MMA's M side
// (A = the activation tile, 128 x 64 per k-block) and the two dequantised
// weight row tiles on its N side (B, 256 x 64), so one MMA covers both row
// tiles and each activation tile is read from L2 once per 256 weight rows;
// the CTAs running together also share it through L2. An expert's token
// tiles follow each other, so its weight tiles are re-read from L2 rather
// than HBM.
//
// Operand type: bf16 or fp16 (template parameter ACT). Activations, the
// dequantised weights, h and the output are all of that type; tcgen05.mma
// kind::f16 takes A and B of the same type, so the instruction descriptor
// names it for both.
//
// Warp roles (24 warps; the role of warp w is chosen by its SM
// sub-partition w % 4, see GT_WARP_*):
//   warp 5       packed-weight producer. 1D bulk copies of each k-block's
//                two packed tiles (64 K each) into an 8-deep ring.
//   warp 9       activation producer. A 2D TMA tensor load (128 rows x 64,
//                128B swizzle) into the k-block's operand slot (a 3-deep
//                ring whose slots also hold the dequantised weight tiles),
//                completing on the slot's barrier, plus an L2 prefetch of
//                the tile needed 8 k-blocks later.
//   warp 1       MMA issuer (also allocates 512 TMEM columns). Per k-block:
//                one wait on the operand slot, 4 tcgen05.mma.kind::f16
//                (M = 128 tokens, N = 256 weight rows, K = 16) into a
//                double-buffered fp32 accumulator, one tcgen05.commit that
//                frees the slot.
//   16 warps     dequantisers, in two groups of 8 that take alternate
//                k-blocks. Per k-block each warp expands its 16-row group of
//                both row tiles: each thread turns one tile slot (2 rows x
//                16 K) of each into the operand type (E2M1 x E4M3,
//                E2M1 x 2^e, or the rounded product NF3 codebook x scale)
//                in the canonical K-major SWIZZLE_128B layout, then fences
//                the async proxy.
//   warps 12..15 epilogue. tcgen05.ld of the accumulator: TMEM lane = token,
//                column = weight row, so one thread holds one token's rows.
//                W13: gate and up rows of a 16-row group sit 8 columns
//                apart, so h = silu(g13*gate) * (g13*up) needs no shuffle
//                and 8 channels go out in one 16-byte store.
//                W2: y[s][row] = g2 * acc for the flat slot s = perm[p].
// Every mbarrier wait is bounded. On a timeout the CTA records
// DEV_TIMEOUT, drains its copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <algorithm>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace hmoe {

constexpr int GT_N = 128;                 // token tile
constexpr int GT_R = 2;                   // weight row tiles per item (they share the activation tile)
constexpr int GT_A_TILE = 128 * 128;      // one dequantised weight row tile, 128 x 64 2-byte values
constexpr int GT_A_BYTES = GT_R * GT_A_TILE;
constexpr int GT_B_BYTES = GT_N * 128;    // activation tile GT_N x 64 2-byte values
constexpr int GT_P_TILE = 4608;           // largest packed tile
constexpr int GT_P_BYTES = GT_R * GT_P_TILE;
constexpr int GT_PSTAGES = 8;             // packed weight tiles in flight (covers the L2/HBM latency)
// Operand stages: slot s holds one k-block's dequantised weight tiles (A)
// and its activation tile (B). One barrier per slot frees both, so each
// issuer commits once per k-block (measured 3.30 -> 3.21 ms at M=4096
// against separate A and B rings of depth 3 and 5).
constexpr int GT_OSTAGES = 3;
constexpr int GT_BPREFETCH = 8;           // B tiles prefetched into L2 ahead of the TMA loads
constexpr int GT_DQ_GROUPS = 2;           // dequant group g expands the k-blocks k with k % 2 == g
constexpr int GT_DQ_WARPS = 16;           // 8 per group, one per 16-row group of every row tile
constexpr int GT_DQ_PER_GROUP = GT_DQ_WARPS / GT_DQ_GROUPS;
// The waits track mbarrier phases by parity, which is only sound while a
// waiter is never two phases behind. A group revisits a ring slot after
// GT_DQ_GROUPS * (ring depth) k-blocks, and its own previous wait has already
// forced progress up to GT_DQ_GROUPS k-blocks back; with more than two groups
// a slot can be two phases behind the one awaited and the parity test passes
// early (measured: bounded waits timed out with four groups).
static_assert(GT_DQ_GROUPS <= 2, "parity-tracked waits need at most two dequant groups");
// That forced progress holds for the operand ring, whose slots are freed by
// MMA commits in issue order, but not for the packed ring: bulk copies may
// land out of order, so a group's earlier waits say nothing about a slot it
// did not wait on. With a depth that is a multiple of the group count each
// group owns its own packed slots and waits on each of them every time
// (measured: a 3-deep packed ring with two groups gave wrong results).
static_assert(GT_PSTAGES % GT_DQ_GROUPS == 0, "each dequant group owns its packed-ring slots");
constexpr int GT_EPI_WARPS = 4;
// Warp roles by SM sub-partition (a warp runs on sub-partition warp % 4).
// The MMA issuer's sub-partition (1) holds the light roles (the producers,
// one epilogue warp) and only one of the 16 ALU-bound dequant warps, so that
// the issuer gets issue slots at once: with four dequant warps beside it,
// its bookkeeping between two k-blocks took longer than the tensor core's
// queued work (measured with per-role timestamps) and left the tensor core
// idle. The epilogue warps are 12..15, one per sub-partition, because a
// warp reads the TMEM lanes 32 * (warp % 4) .. + 31.
constexpr int GT_WARP_MMA = 1, GT_WARP_PPROD = 5, GT_WARP_BPROD = 9, GT_WARP_EPI0 = 12;
constexpr int GT_WARPS = 24;
constexpr int GT_THREADS = GT_WARPS * 32;
// Dequant index of each warp (-1 for the other roles; warp 21 has none).
// Indices 0..7 (group 0) sit on warps 0, 2, 3, 4, 6, 7, 8, 17 and 8..15
// (group 1) on warps 10, 11, 16, 18, 19, 20, 22, 23: each group spread over
// the sub-partitions.
__device__ __constant__ const int8_t GT_DQ_INDEX[GT_WARPS] = {0,  -1, 1,  2,  3,  -1, 4,  5,  6,  -1, 8,  9,
                                                              -1, -1, -1, -1, 10, 7,  11, 12, 13, -1, 14, 15};
// Accumulator: TMEM lane = token (M = 128), column = weight row of the
// item's row-tile pair (N = 256), double-buffered.
constexpr int GT_ACC_COLS = GT_R * 128;
constexpr int GT_TMEM_COLS = 2 * GT_ACC_COLS;
// Shared memory map (offsets from the 1024-aligned base).
constexpr int GT_OFF_A = 0;
constexpr int GT_OFF_B = GT_OFF_A + GT_OSTAGES * GT_A_BYTES;
constexpr int GT_OFF_P = GT_OFF_B + GT_OSTAGES * GT_B_BYTES;
constexpr int GT_OFF_BAR = GT_OFF_P + GT_PSTAGES * GT_P_BYTES;
constexpr int GT_NBAR = 2 * GT_PSTAGES + 3 * GT_OSTAGES + 4 + 1;
constexpr int GT_OFF_MISC = GT_OFF_BAR + ((GT_NBAR * 8 + 16 + 127) / 128) * 128;
constexpr int GT_SMEM_BYTES = 1024 + GT_OFF_MISC + 2 * (MAX_E + 1) * 4 + 256 * 4;
static_assert(GT_SMEM_BYTES <= 232448, "shared memory budget");
static_assert(GT_OFF_P % 16 == 0 && GT_OFF_B % 1024 == 0, "alignment");
static_assert(GT_TMEM_COLS <= 512, "TMEM columns");

// ------------------------------------------------------------ tcgen05 / TMA wrappers
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// tcgen05.mma (kind::f16, A and B from shared memory, D in TMEM) and its
// commit, issued from a converged warp: every lane executes
// the instruction, and elect.sync predicates it to one lane (the lowest
// active one, so MMAs and their commits come from the same thread). Measured
// against issuing from inside an `if (lane == 0)` branch: a 128 x 128 x 16
// MMA takes 65 instead of 120 cycles of the tensor core's issue slot, the
// full rate of the tensor core, instead of half of it.
__device__ __forceinline__ void umma_kf16_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

// 16 lanes x 256 bits, four times along the columns: thread t gets rows
// base + t/4 (regs 4j, 4j+1) and base + t/4 + 8 (regs 4j+2, 4j+3) at
// columns 8j + 2(t % 4) and + 1 of repetition j.
__device__ __forceinline__ void tmem_ld16x256x4(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

// 256-bit global store of 8 words; the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8u(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
// 256-bit global store of 8 floats; the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8f(float* dst, const float* f) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "f"(f[0]), "f"(f[1]), "f"(f[2]),
               "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7])
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// The same TMA load from a converged warp: one elected lane registers the
// tile's bytes on the barrier and issues the load.
__device__ __forceinline__ void tma_expect_load_2d_elect(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                         uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%4], %5;\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n\t}" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "r"(bytes)
      : "memory");
}
// The same load without the expect_tx arrival (a second box on a barrier
// whose bytes an earlier tma_expect_load_2d_elect already registered).
__device__ __forceinline__ void tma_load_2d_elect(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n\t}" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_2d_elect(const CUtensorMap* map, int x, int y) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];\n\t}" ::"l"(map), "r"(x), "r"(y)
      : "memory");
}
// From a converged warp: an elected lane registers the bytes on the barrier,
// then every lane whose predicate is set issues its own 1D bulk copy (L2
// evict-first), all in one warp instruction.
__device__ __forceinline__ void mbar_expect_tx_elect(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s_stream_if(bool pred, void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                   uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred q;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n\t}" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy), "r"(pred ? 1u : 0u)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
               : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (SBO), version 1, base offset 0 (atoms 1024-aligned).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;                 // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024u >> 4) << 32;       // stride byte offset
  d |= (uint64_t)1u << 46;                 // descriptor version
  d |= (uint64_t)2u << 61;                 // SWIZZLE_128B
  return d;
}
// The descriptor above as (low word, high word). The low word holds the start
// address (>> 4) and the leading byte offset; the high word is constant.
// Advancing 32 bytes along K adds 2 to the low word.
constexpr uint32_t SW128_DESC_HI = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint32_t smem_desc_sw128_lo(uint32_t addr) { return ((addr >> 4) & 0x3FFFu) | (1u << 16); }
__device__ __forceinline__ uint64_t desc_from_lo(uint32_t lo) {
  return ((uint64_t)SW128_DESC_HI << 32) | (uint64_t)lo;
}

// Instruction descriptor, kind::f16: D fp32, A and B of the same type (bf16,
// type code 1, or fp16, code 0), both K-major.
template <int ACT = ACT_BF16>
__device__ __forceinline__ uint32_t idesc_kf16(int M, int N) {
  constexpr uint32_t ab = ACT == ACT_F16 ? 0u : 1u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// A work item: nt token tiles of 128 permuted slots from p0 (n slots in all)
// times nr weight row tiles from rt. Two shapes, both 512 cycles of tensor
// work per k-block and 256 accumulator columns:
//   nt = 1, nr = 1 or 2: one token tile (A, M = 128) times the row-tile pair
//     (B, N = 256): 4 MMAs of 128 x 256 x 16 per k-block;
//   nt = 2, nr = 1: two token tiles (two A operands) times one row tile (B,
//     N = 128): 8 MMAs of 128 x 128 x 16, into accumulator columns 0..127
//     (tile 0) and 128..255 (tile 1).
// An expert with more than 128 routed slots takes the second shape for each
// full 256-slot pair of token tiles (and for a remainder above 128), so each
// weight row tile is dequantised once per 256 slots instead of once per 128
// (measured 3.33 -> 3.22 ms at M=4096 with Zipf routing, where the 256
// experts need 379 token tiles); a remainder of at most 128 slots takes the
// first shape. (An N = 128 MMA issues in about 77 cycles against 64 of
// tensor work, so the second shape is bound by its issuing thread.)
struct GtItem {
  int e, p0, n, rt, nr, nt;
};

__host__ __device__ __forceinline__ int gt_items_of(int ne, int RT) {
  if (ne <= 0) return 0;
  const int RP = (RT + GT_R - 1) / GT_R;
  const int full = ne / (2 * GT_N), r = ne % (2 * GT_N);
  const int n2 = full + (r > GT_N ? 1 : 0);
  const int n1 = (r > 0 && r <= GT_N) ? 1 : 0;
  return n2 * RT + n1 * RP;
}

__device__ __forceinline__ int gt_expert_fmt(const GroupedParams& p, int e) {
  return (p.tab.loc[e] & LOC_NF3) ? FMT_NF3 : p.kept_fmt;
}

__device__ __forceinline__ GtItem gt_decode(const GroupedParams& p, const int* s_istart, const int* s_off, int i) {
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_istart[mid] <= i) lo = mid; else hi = mid;
  }
  GtItem it;
  it.e = lo;
  const int o0 = s_off[lo], ne = s_off[lo + 1] - o0;
  // Row tiles (or row-tile pairs) fastest: the CTAs that run together share
  // one activation tile through L2, and an expert's token tiles follow each
  // other, so its weight tiles are re-read from L2 rather than HBM.
  const int local = i - s_istart[lo];
  const int full = ne / (2 * GT_N), r = ne % (2 * GT_N);
  const int n2 = full + (r > GT_N ? 1 : 0);
  if (local < n2 * p.RT) {
    const int tp = local / p.RT;
    it.rt = local % p.RT;
    it.nr = 1;
    it.nt = 2;
    it.p0 = o0 + tp * 2 * GT_N;
    it.n = min(2 * GT_N, ne - tp * 2 * GT_N);
  } else {
    const int l1 = local - n2 * p.RT;
    it.rt = l1 * GT_R;
    it.nr = min(GT_R, p.RT - it.rt);
    it.nt = 1;
    it.p0 = o0 + n2 * 2 * GT_N;
    it.n = ne - n2 * 2 * GT_N;
  }
  return it;
}

// Writes one thread slot's dequantised rows (2 rows x 16 K) into the
// canonical K-major SWIZZLE_128B tile: row r of atom (r / 8) at (r % 8) * 128,
// 16-byte chunk c stored at chunk position c ^ (r % 8).
template <int FMT, int ACT = ACT_BF16>
__device__ __forceinline__ void gt_dequant_slot(const uint8_t* ptile, uint8_t* atile, int rg, int lane,
                                                const uint32_t* e4m3_lut) {
  uint32_t r0[8], r1[8];
  float s0, s1;
  dequant_slot<FMT, true, ACT>(ptile, rg, lane, r0, r1, &s0, &s1, e4m3_lut);
  const int g = lane >> 2, q = lane & 3;
  uint8_t* a0 = atile + (2 * rg) * 1024 + g * 128;
  uint8_t* a1 = atile + (2 * rg + 1) * 1024 + g * 128;
  const int c0 = ((2 * q) ^ g) * 16, c1 = ((2 * q + 1) ^ g) * 16;
  *reinterpret_cast<uint4*>(a0 + c0) = make_uint4(r0[0], r0[1], r0[2], r0[3]);
  *reinterpret_cast<uint4*>(a0 + c1) = make_uint4(r0[4], r0[5], r0[6], r0[7]);
  *reinterpret_cast<uint4*>(a1 + c0) = make_uint4(r1[0], r1[1], r1[2], r1[3]);
  *reinterpret_cast<uint4*>(a1 + c1) = make_uint4(r1[4], r1[5], r1[6], r1[7]);
}

// The k-block loop of one dequantising warp over one item, for one format
// (the format branch is taken once per item, not once per k-block). The
// groups of warps take turns by k-block (group par takes the k-blocks whose
// running count gk is par modulo the group count), and a warp expands its
// row groups rg, rg + 1, ... of every row tile of its k-blocks: the waits,
// fence and arrivals are paid once per several slots while all the warps
// stay busy. Returns false if a bounded wait gave up.
template <int FMT, int ACT>
__device__ __forceinline__ bool gt_dequant_item(int KB, int nr, int par, const uint8_t* p_base, uint8_t* a_base,
                                                uint64_t* pfull, uint64_t* pempty, uint64_t* afull,
                                                uint64_t* oempty, const uint32_t* s_e4m3, int rg, int lane,
                                                volatile int* s_flags, uint64_t lim, uint32_t& gk, int& ps,
                                                uint32_t& pph, int& as, uint32_t& aph) {
  for (int kb = 0; kb < KB; ++kb, ++gk) {
    if ((int)(gk % GT_DQ_GROUPS) == par) {
      if (!__all_sync(0xffffffffu, mbar_wait(&pfull[ps], pph, s_flags, lim)) ||
          !__all_sync(0xffffffffu, mbar_wait(&oempty[as], aph ^ 1u, s_flags, lim)))
        return false;
      const uint8_t* pt = p_base + ps * GT_P_BYTES;
      uint8_t* at = a_base + as * GT_A_BYTES;
#pragma unroll
      for (int h = 0; h < 8 / GT_DQ_PER_GROUP; ++h) {
        gt_dequant_slot<FMT, ACT>(pt, at, rg + h, lane, s_e4m3);
        if (nr > 1) gt_dequant_slot<FMT, ACT>(pt + GT_P_TILE, at + GT_A_TILE, rg + h, lane, s_e4m3);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&pempty[ps]);
        mbar_arrive(&afull[as]);
      }
    }
    if (++ps == GT_PSTAGES) {
      ps = 0;
      pph ^= 1u;
    }
    if (++as == GT_OSTAGES) {
      as = 0;
      aph ^= 1u;
    }
  }
  return true;
}

template <int ACT>
__global__ void __launch_bounds__(GT_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ GroupedParams p, const __grid_constant__ CUtensorMap tmap_b) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + GT_OFF_BAR);
  uint64_t* pfull = bars;                              // packed tile landed (tx)
  uint64_t* pempty = pfull + GT_PSTAGES;               // dequant warps done reading it
  // afull: the operand slot is complete: the group's 8 dequant warps wrote the
  // weight tiles (8 arrivals) and the activation tile landed (the TMA
  // producer's arrival and its bytes), so the issuer waits once per k-block.
  uint64_t* afull = pempty + GT_PSTAGES;
  uint64_t* oempty = afull + GT_OSTAGES;               // MMAs that read the slot completed
  uint64_t* acc_full = oempty + GT_OSTAGES;            // [2] accumulator ready for the epilogue
  uint64_t* acc_empty = acc_full + 2;                  // [2] epilogue drained it
  uint64_t* mma_done = acc_empty + 2;                  // final drain before TMEM release
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* s_flags = reinterpret_cast<volatile int*>(s_tmem + 1);  // [0] abort
  int* s_istart = reinterpret_cast<int*>(smem + GT_OFF_MISC);
  int* s_off = s_istart + MAX_E + 1;
  uint32_t* s_e4m3 = reinterpret_cast<uint32_t*>(s_off + MAX_E + 1);  // E4M3 -> operand-type pair

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < GT_PSTAGES; ++s) {
      mbar_init(&pfull[s], 1);
      mbar_init(&pempty[s], GT_DQ_PER_GROUP);
    }
    for (int s = 0; s < GT_OSTAGES; ++s) {
      mbar_init(&afull[s], GT_DQ_PER_GROUP + 1);
      mbar_init(&oempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], GT_EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
    s_flags[0] = 0;
  }
  if (warp == GT_WARP_MMA) {
    tmem_alloc(s_tmem, GT_TMEM_COLS);
    tmem_relinquish();
  }
  if (tid >= 96 && tid < 96 + 256)
    s_e4m3[tid - 96] = e4m3_lut_entry<ACT>((uint32_t)(tid - 96));
  pdl_wait();  // everything below reads or writes global memory
  pdl_trigger();
  for (int e = tid; e <= p.E; e += blockDim.x) s_off[e] = p.offsets[e];
  __syncthreads();
  if (warp == 0) {
    // Item prefix over the experts of the selected tiers.
    const int S = p.T * p.topk;
    bool bad = (s_off[0] != 0) || (s_off[p.E] != S);
    int run = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      int ni = 0;
      if (e < p.E) {
        const int ne = s_off[e + 1] - s_off[e];
        if (ne < 0) bad = true;
        const bool nf3 = (p.tab.loc[e] & LOC_NF3) != 0;
        const bool sel = nf3 ? (p.tier_mask & 2) : (p.tier_mask & 1);
        ni = sel ? gt_items_of(ne, p.RT) : 0;
      }
      int incl = ni;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int nb = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += nb;
      }
      if (e < p.E) s_istart[e] = run + incl - ni;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      s_istart[p.E] = bad ? 0 : run;
      if (bad && blockIdx.x == 0) set_status(p.status, DEV_BAD_ROUTE);
    }
    if (bad)
      for (int e = lane; e < p.E; e += 32) s_istart[e] = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int n_items = s_istart[p.E];
  const uint64_t lim = p.wait_limit_ns;

  if (warp == GT_WARP_PPROD) {
    // ------------------------------------------------ packed weight tiles (HBM)
    // Converged warp: lane r < nr copies row tile r, in one warp instruction.
    const uint64_t pol = l2_policy_evict_first();
    int slot = 0, issued = 0;
    uint32_t ph = 0;
    bool aborted = false;
    for (int i = blockIdx.x; i < n_items && !aborted; i += gridDim.x) {
      const GtItem it = gt_decode(p, s_istart, s_off, i);
      const int fmt = gt_expert_fmt(p, it.e);
      const uint32_t tb = (uint32_t)tile_bytes(fmt);
      const uint8_t* base = (fmt == FMT_NF3 ? p.nf3_buf : p.kept_buf) +
                            (size_t)(p.tab.loc[it.e] & 0x7FFF) *
                                (fmt == FMT_NF3 ? p.nf3_expert_bytes : p.kept_expert_bytes) +
                            (p.which == 2 ? (fmt == FMT_NF3 ? p.nf3_w2_off : p.kept_w2_off) : 0) +
                            (size_t)it.rt * p.KB * tb;
      const size_t rt_stride = (size_t)p.KB * tb;
      const int r = lane < it.nr ? lane : 0;
      for (int kb = 0; kb < p.KB; ++kb) {
        if (!__all_sync(0xffffffffu, mbar_wait(&pempty[slot], ph ^ 1u, s_flags, lim))) {
          aborted = true;
          break;
        }
        mbar_expect_tx_elect(&pfull[slot], tb * (uint32_t)it.nr);
        bulk_g2s_stream_if(lane < it.nr, smem + GT_OFF_P + slot * GT_P_BYTES + r * GT_P_TILE,
                           base + r * rt_stride + (size_t)kb * tb, tb, &pfull[slot], pol);
        ++issued;
        if (++slot == GT_PSTAGES) {
          slot = 0;
          ph ^= 1u;
        }
      }
    }
    if (aborted && lane == 0) {
      s_flags[0] = 1;
      set_status(p.status, DEV_TIMEOUT);
      volatile int never = 0;
      for (int b = 0; b < GT_PSTAGES && b < issued; ++b) {
        if (--slot < 0) {
          slot = GT_PSTAGES - 1;
          ph ^= 1u;
        }
        mbar_wait(&pfull[slot], ph, &never, lim);
      }
    }
    __syncwarp();
  } else if (warp == GT_WARP_BPROD) {
    // ------------------------------------------------ activation tiles (L2), TMA tensor loads
    int slot = 0, issued = 0;
    uint32_t ph = 0;
    bool aborted = false;
    for (int i = blockIdx.x; i < n_items && !aborted; i += gridDim.x) {
      const GtItem it = gt_decode(p, s_istart, s_off, i);
      for (int kb = 0; kb < p.KB; ++kb) {
        if (!__all_sync(0xffffffffu, mbar_wait(&oempty[slot], ph ^ 1u, s_flags, lim))) {
          aborted = true;
          break;
        }
        // Token tile 0 goes to the slot's activation tile; with two token
        // tiles, tile 1 goes to the second weight-tile half, unused by
        // one-row-tile items.
        tma_expect_load_2d_elect(smem + GT_OFF_B + slot * GT_B_BYTES, &tmap_b, kb * TILE_K, it.p0, &afull[slot],
                                 (uint32_t)(it.nt * GT_B_BYTES));
        if (it.nt == 2)
          tma_load_2d_elect(smem + GT_OFF_A + slot * GT_A_BYTES + GT_A_TILE, &tmap_b, kb * TILE_K, it.p0 + GT_N,
                            &afull[slot]);
        // Warm L2 with the tiles needed a few loads from now (same token tiles).
        if (kb + GT_BPREFETCH < p.KB) {
          tma_prefetch_2d_elect(&tmap_b, (kb + GT_BPREFETCH) * TILE_K, it.p0);
          if (it.nt == 2) tma_prefetch_2d_elect(&tmap_b, (kb + GT_BPREFETCH) * TILE_K, it.p0 + GT_N);
        }
        ++issued;
        if (++slot == GT_OSTAGES) {
          slot = 0;
          ph ^= 1u;
        }
      }
    }
    if (aborted && lane == 0) {
      s_flags[0] = 1;
      set_status(p.status, DEV_TIMEOUT);
      volatile int never = 0;
      for (int b = 0; b < GT_OSTAGES && b < issued; ++b) {
        if (--slot < 0) {
          slot = GT_OSTAGES - 1;
          ph ^= 1u;
        }
        mbar_wait(&afull[slot], ph, &never, lim);
      }
    }
    __syncwarp();
  } else if (warp == GT_WARP_MMA) {
    // ------------------------------------------------ MMA issuer
    // One tcgen05.mma occupies the tensor core for about 125 cycles whatever
    // its N up to 256 (measured), so the item's token tile is the M side
    // (M = 128) and its two weight row tiles the N side (N = 256): per
    // k-block 4 MMAs of 128 x 256 x 16, at the tensor core's full rate,
    // instead of 8 of 128 x tokens x 16. The whole warp runs the loop and
    // issues each MMA and commit from converged code (elect.sync).
    const uint32_t x_lo0 = smem_desc_sw128_lo(smem_u32(smem + GT_OFF_B));  // activation tile: A
    const uint32_t w_lo0 = smem_desc_sw128_lo(smem_u32(smem + GT_OFF_A));  // weight tiles: B
    int os = 0;
    uint32_t oph = 0;
    bool aborted = false;
    int j = 0;
    for (int i = blockIdx.x; i < n_items && !aborted; i += gridDim.x, ++j) {
      const GtItem it = gt_decode(p, s_istart, s_off, i);
      const int buf = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_empty[buf], ((uint32_t)(j >> 1) & 1u) ^ 1u, s_flags, lim))) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const uint32_t idesc = idesc_kf16<ACT>(128, it.nt == 2 ? 128 : it.nr * 128);
      const uint32_t d_tmem = tmem_base + (uint32_t)(buf * GT_ACC_COLS);
      // Operand slots are ordered by their barrier and the writers' proxy
      // fence; the tcgen05 fence after the accumulator hand-off covers TMEM.
      // The tensor core queues few MMAs, so the issuer must not stall between
      // k-blocks: the next slot's barrier is probed (non-blocking) between
      // this k-block's MMAs, while they execute, and only if it was not yet
      // complete does the issuer block on it after queueing them all.
      bool ready = false;
      for (int kb = 0; kb < p.KB; ++kb) {
        if (!ready && !__all_sync(0xffffffffu, mbar_wait(&afull[os], oph, s_flags, lim))) {
          aborted = true;
          break;
        }
        const uint32_t x_lo = x_lo0 + (uint32_t)os * (GT_B_BYTES >> 4);
        const uint32_t w_lo = w_lo0 + (uint32_t)os * (GT_A_BYTES >> 4);
        const int os_next = os + 1 == GT_OSTAGES ? 0 : os + 1;
        const uint32_t oph_next = os + 1 == GT_OSTAGES ? oph ^ 1u : oph;
        if (it.nt == 2) {
          // token tile 1's activations sit in the second weight-tile half
          const uint32_t x1_lo = w_lo + (GT_A_TILE >> 4);
          umma_kf16_warp(d_tmem, desc_from_lo(x_lo), desc_from_lo(w_lo), idesc, kb ? 1u : 0u);
          umma_kf16_warp(d_tmem, desc_from_lo(x_lo + 2), desc_from_lo(w_lo + 2), idesc, 1u);
          umma_kf16_warp(d_tmem, desc_from_lo(x_lo + 4), desc_from_lo(w_lo + 4), idesc, 1u);
          umma_kf16_warp(d_tmem, desc_from_lo(x_lo + 6), desc_from_lo(w_lo + 6), idesc, 1u);
          ready = kb + 1 < p.KB && __all_sync(0xffffffffu, mbar_test(&afull[os_next], oph_next));
          umma_kf16_warp(d_tmem + 128, desc_from_lo(x1_lo), desc_from_lo(w_lo), idesc, kb ? 1u : 0u);
          umma_kf16_warp(d_tmem + 128, desc_from_lo(x1_lo + 2), desc_from_lo(w_lo + 2), idesc, 1u);
          umma_kf16_warp(d_tmem + 128, desc_from_lo(x1_lo + 4), desc_from_lo(w_lo + 4), idesc, 1u);
          umma_kf16_warp(d_tmem + 128, desc_from_lo(x1_lo + 6), desc_from_lo(w_lo + 6), idesc, 1u);
        } else {
          umma_kf16_warp(d_tmem, desc_from_lo(x_lo), desc_from_lo(w_lo), idesc, kb ? 1u : 0u);
          umma_kf16_warp(d_tmem, desc_from_lo(x_lo + 2), desc_from_lo(w_lo + 2), idesc, 1u);
          ready = kb + 1 < p.KB && __all_sync(0xffffffffu, mbar_test(&afull[os_next], oph_next));
          umma_kf16_warp(d_tmem, desc_from_lo(x_lo + 4), desc_from_lo(w_lo + 4), idesc, 1u);
          umma_kf16_warp(d_tmem, desc_from_lo(x_lo + 6), desc_from_lo(w_lo + 6), idesc, 1u);
        }
        umma_commit_warp(&oempty[os]);
        os = os_next;
        oph = oph_next;
      }
      if (!aborted) umma_commit_warp(&acc_full[buf]);
    }
    if (aborted && lane == 0) {
      s_flags[0] = 1;
      set_status(p.status, DEV_TIMEOUT);
    }
    // Drain every MMA issued above before TMEM can be released.
    umma_commit_warp(mma_done);
    {
      volatile int never = 0;
      mbar_wait(mma_done, 0, &never, lim);
    }
    __syncwarp();
  } else if (GT_DQ_INDEX[warp] >= 0) {
    // ------------------------------------------------ dequantisers: packed tile -> operand tile
    // Group par expands the k-blocks k with k % GT_DQ_GROUPS == par, every
    // row tile; its warps split the 8 row groups. (Eight warps each expanding
    // both row tiles of every k-block was measured slower: 4.18 against 4.03
    // ms at M=4096.)
    const int dq = GT_DQ_INDEX[warp];
    const int par = dq / GT_DQ_PER_GROUP, rg = (dq % GT_DQ_PER_GROUP) * (8 / GT_DQ_PER_GROUP);
    int ps = 0, as = 0;
    uint32_t pph = 0, aph = 0, gk = 0;
    bool ok = true;
    const uint8_t* p_base = smem + GT_OFF_P;
    uint8_t* a_base = smem + GT_OFF_A;
    for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
      const GtItem it = gt_decode(p, s_istart, s_off, i);
      const int fmt = gt_expert_fmt(p, it.e);
      if (fmt == FMT_NVFP4)
        ok = gt_dequant_item<FMT_NVFP4, ACT>(p.KB, it.nr, par, p_base, a_base, pfull, pempty, afull, oempty, s_e4m3, rg,
                                        lane, s_flags, lim, gk, ps, pph, as, aph);
      else if (fmt == FMT_MXFP4)
        ok = gt_dequant_item<FMT_MXFP4, ACT>(p.KB, it.nr, par, p_base, a_base, pfull, pempty, afull, oempty, s_e4m3, rg,
                                        lane, s_flags, lim, gk, ps, pph, as, aph);
      else
        ok = gt_dequant_item<FMT_NF3, ACT>(p.KB, it.nr, par, p_base, a_base, pfull, pempty, afull, oempty, s_e4m3, rg,
                                      lane, s_flags, lim, gk, ps, pph, as, aph);
    }
    if (!ok && lane == 0) {
      s_flags[0] = 1;
      set_status(p.status, DEV_TIMEOUT);
    }
  } else if (warp >= GT_WARP_EPI0 && warp < GT_WARP_EPI0 + GT_EPI_WARPS) {
    // ------------------------------------------------ epilogue
    // TMEM lane = token column c of the item (each warp owns 32 lanes), TMEM
    // column = weight row of the row-tile pair. A thread reads 32 columns at
    // a time (32x32b.x32): two 16-row groups, i.e. W13 gate rows 0..7 and up
    // rows 8..15 of 8 channels each, or 32 consecutive W2 output rows.
    const int quarter = warp & 3;
    const int c = quarter * 32 + lane;
    const int S = p.T * p.topk;
    int j = 0;
    for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++j) {
      const GtItem it = gt_decode(p, s_istart, s_off, i);
      const int buf = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (uint32_t)(j >> 1) & 1u, s_flags, lim))) {
        if (lane == 0) {
          s_flags[0] = 1;
          set_status(p.status, DEV_TIMEOUT);
        }
        break;
      }
      tc_fence_after();
      // Thread c holds token c of each token tile: slot c (tile 0) and, for
      // two-tile items, slot 128 + c (tile 1, accumulator columns 128..255).
      int slot0 = -1, slot1 = -1;
      if (p.which != 13) {
        if (c < it.n) {
          const int sc = p.perm[it.p0 + c];
          if (sc >= 0 && sc < S) slot0 = sc;
          else set_status(p.status, DEV_BAD_ROUTE);
        }
        if (it.nt == 2 && GT_N + c < it.n) {
          const int sc = p.perm[it.p0 + GT_N + c];
          if (sc >= 0 && sc < S) slot1 = sc;
          else set_status(p.status, DEV_BAD_ROUTE);
        }
      }
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * GT_ACC_COLS);
      const int nchunk = it.nt == 2 ? 8 : it.nr * 4;
      for (int q = 0; q < nchunk; ++q) {
        uint32_t v[32];
        tmem_ld32(tbase + (uint32_t)(32 * q), v);
        tmem_wait_ld();
        const int tt = it.nt == 2 ? (q >> 2) : 0;             // token tile of the chunk
        const int rt = it.nt == 2 ? it.rt : it.rt + (q >> 2);  // row tile of the chunk
        const int r0 = (q & 3) * 32;  // first tile-local row of the chunk
        const int tok = tt * GT_N + c;
        if (p.which == 13) {
          if (tok >= it.n) continue;
          const float gsc =
              p.tab.g13[it.e] * (gt_expert_fmt(p, it.e) == FMT_NVFP4 ? nvfp4_unscale<ACT>() : 1.0f) * p.act_scale;
          // 16-row groups r0 / 16 and r0 / 16 + 1: rows 0..7 gate, 8..15 up, of
          // channels ch .. ch + 7 and ch + 8 .. ch + 15; the 16 channels go out
          // in one 32-byte store (one L2 sector).
          const int ch = rt * 64 + (r0 / 16) * 8;
          uint32_t hv[8];
#pragma unroll
          for (int g = 0; g < 2; ++g) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const float g0 = __uint_as_float(v[16 * g + 2 * w]) * gsc;
              const float g1 = __uint_as_float(v[16 * g + 2 * w + 1]) * gsc;
              const float u0 = __uint_as_float(v[16 * g + 8 + 2 * w]) * gsc;
              const float u1 = __uint_as_float(v[16 * g + 8 + 2 * w + 1]) * gsc;
              hv[4 * g + w] = f32x2_to_act<ACT>(silu_fast(g0) * u0, silu_fast(g1) * u1);
            }
          }
          st_global_v8u(p.h_out + (size_t)(it.p0 + tok) * p.I + ch, hv);
        } else {
          const int slot = tt ? slot1 : slot0;
          if (slot < 0) continue;
          const float gsc =
              p.tab.g2[it.e] * (gt_expert_fmt(p, it.e) == FMT_NVFP4 ? nvfp4_unscale<ACT>() : 1.0f) * p.act_scale;
          // 32-byte stores: each is one whole L2 sector of the slot's row (16-byte
          // stores wrote half sectors, and the W2 launch spent about a fifth of
          // its time on them: 1170 against 902 us without the stores at M=4096).
          float* dst = p.y_out + (size_t)slot * p.H + rt * 128 + r0;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            float f[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) f[u] = __uint_as_float(v[8 * w + u]) * gsc;
            st_global_v8f(dst + 8 * w, f);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == GT_WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem_base, GT_TMEM_COLS);
  }
}

// ============================================================ the CTA-pair kernel
// Two CTAs of a cluster (one per SM of a pair) run each work item together
// with tcgen05.mma.cta_group::2 (M = 256): the leader (cluster rank 0)
// dequantises row tile 2rp of the item's row pair and the peer row tile
// 2rp + 1; each CTA loads half of the item's token columns (B) into its own
// shared memory; one thread in the leader issues the MMAs for both SMs, and
// each CTA's TMEM receives its own 128 rows x N accumulator. Against the
// one-CTA kernel this halves, per SM and per k-block, the dequantised rows
// written to and read from shared memory for the same tensor work, and
// lets a token tile hold up to 256 slots.
//
// Warp roles, in both CTAs:
//   warp 0       packed-weight producer: 1D bulk copy of its row tile's
//                packed k-block into a 4-deep ring.
//   warp 1       TMEM allocation (collective over the pair); in the leader,
//                the MMA issuer.
//   warp 2       activation producer: 2D TMA loads (64-row boxes, 128B
//                swizzle) of its half of the token columns into its own
//                shared memory, completing on the leader's barrier.
//   warps 3..18  dequantisers (two groups of 8 taking alternate k-blocks;
//                warp w of a group expands 16-row group w of the row tile).
//   warps 19..22 epilogue (tcgen05.ld of the CTA's own accumulator).
// Hand-offs to the issuer go straight to the leader's barriers: the
// operand-slot barrier counts the dequant warps of both CTAs and the TMA
// bytes of both halves, and the accumulator-free barrier counts the
// epilogue warps of both CTAs. The leader's tcgen05.commit arrives on the
// same barrier in both CTAs (multicast), which frees the operand slot and
// hands over accumulators.
// Every wait is bounded; on a timeout the CTA records DEV_TIMEOUT, tells
// the other CTA to stop, and both drain before leaving through a final
// cluster barrier.
constexpr int G2_N = 256;                 // token tile of an item (both CTAs)
constexpr int G2_BH = G2_N / 2;           // B rows held by one CTA
constexpr int G2_BBOX = 64;               // rows per TMA box
constexpr int G2_A_BYTES = 128 * 128;     // one row tile's bf16 k-block (128 x 64)
constexpr int G2_B_BYTES = G2_BH * 128;   // bf16 128 x 64
constexpr int G2_P_TILE = 4608;
constexpr int G2_PSTAGES = 4;
constexpr int G2_OSTAGES = 4;
constexpr int G2_DQ_GROUPS = 2;
constexpr int G2_DQ_PER_GROUP = 8;        // one warp per 16-row group of the row tile
constexpr int G2_DQ_WARPS = G2_DQ_GROUPS * G2_DQ_PER_GROUP;
static_assert(G2_DQ_GROUPS <= 2, "parity-tracked waits need at most two dequant groups");
static_assert(G2_PSTAGES % G2_DQ_GROUPS == 0 && G2_OSTAGES % G2_DQ_GROUPS == 0,
              "each dequant group owns its ring slots");
constexpr int G2_EPI_WARPS = 4;
constexpr int G2_WARP_PPROD = 0, G2_WARP_MMA = 1, G2_WARP_BPROD = 2, G2_WARP_DQ0 = 3;
constexpr int G2_WARP_EPI0 = G2_WARP_DQ0 + G2_DQ_WARPS;
constexpr int G2_THREADS = (G2_WARP_EPI0 + G2_EPI_WARPS) * 32;
constexpr int G2_TMEM_COLS = 2 * G2_N;    // double-buffered 128 x 256 fp32 accumulators
constexpr int G2_OFF_A = 0;
constexpr int G2_OFF_B = G2_OFF_A + G2_OSTAGES * G2_A_BYTES;
constexpr int G2_OFF_P = G2_OFF_B + G2_OSTAGES * G2_B_BYTES;
constexpr int G2_OFF_BAR = G2_OFF_P + G2_PSTAGES * G2_P_TILE;
constexpr int G2_NBAR = 2 * G2_PSTAGES + 3 * G2_OSTAGES + 2 * 2 + 1;
constexpr int G2_OFF_MISC = G2_OFF_BAR + ((G2_NBAR * 8 + 16 + 127) / 128) * 128;
constexpr int G2_SMEM_BYTES = 1024 + G2_OFF_MISC + 2 * (MAX_E + 1) * 4 + 256 * 4;
static_assert(G2_SMEM_BYTES <= 232448, "shared memory budget");
static_assert(G2_OFF_B % 1024 == 0 && G2_OFF_P % 16 == 0 && G2_B_BYTES % 1024 == 0, "alignment");
static_assert(G2_TMEM_COLS <= 512, "TMEM columns");

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory object in the CTA of the given cluster rank.
__device__ __forceinline__ uint32_t mapa_shared(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// Arrive on a barrier in the other CTA of the pair (default release
// semantics, as for a local arrive). What it publishes is read by the tensor
// cores through the async proxy, after the usual proxy fence by the writers.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void st_remote_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// try_wait without a suspend-time hint: for the pair's latency-critical
// hand-offs (barriers completed from the other SM of the pair, and the
// issuer's waits).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
}
__device__ __forceinline__ void tmem_alloc2(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Commit of the pair's MMAs: arrives once on the barrier at this offset in
// both CTAs of the pair. Both are issued from a converged warp (elect.sync),
// like umma_kf16_warp.
__device__ __forceinline__ void umma2_commit_both(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void umma2_kf16_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 2D TMA load into this CTA's shared memory whose completion (bytes) is
// counted on a barrier of the pair given by its shared::cluster address.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t cluster_bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(cluster_bar)
      : "memory");
}

struct G2Item {
  int e, p0, n, rt, valid;  // rt: this CTA's row tile; valid = 0 for the peer of an odd last pair
};

__device__ __forceinline__ G2Item g2_decode(const GroupedParams& p, const int* s_istart, const int* s_off, int i,
                                            int rank) {
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_istart[mid] <= i) lo = mid; else hi = mid;
  }
  G2Item it;
  it.e = lo;
  const int o0 = s_off[lo], ne = s_off[lo + 1] - o0;
  const int RP = (p.RT + 1) / 2;
  const int local = i - s_istart[lo];
  const int rt = (local % RP) * 2 + rank;
  it.valid = rt < p.RT;
  it.rt = it.valid ? rt : p.RT - 1;  // a real tile keeps the pipeline uniform; its result is dropped
  const int nt = local / RP;
  it.p0 = o0 + nt * G2_N;
  it.n = min(G2_N, ne - nt * G2_N);
  return it;
}
// MMA width of an item: the token count rounded up to 32 (so each CTA's half
// is a whole number of 16-row groups).
__device__ __forceinline__ int g2_width(int n) { return max(32, (n + 31) & ~31); }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(G2_THREADS, 1)
    grouped_pair_kernel(const __grid_constant__ GroupedParams p, const __grid_constant__ CUtensorMap tmap_b) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G2_OFF_BAR);
  uint64_t* pfull = bars;                          // packed tile landed (tx)
  uint64_t* pempty = pfull + G2_PSTAGES;           // dequant warps done reading it
  uint64_t* bfull = pempty + G2_PSTAGES;           // leader: both B halves landed (tx of both CTAs)
  uint64_t* afull = bfull + G2_OSTAGES;            // leader: the dequant warps of both CTAs wrote A
  uint64_t* oempty = afull + G2_OSTAGES;           // the pair's MMAs on the slot completed (leader commit)
  uint64_t* acc_full = oempty + G2_OSTAGES;        // [2] accumulator complete (leader commit)
  uint64_t* acc_empty = acc_full + 2;              // [2] leader: the epilogues of both CTAs drained it
  uint64_t* mma_done = acc_empty + 2;              // final drain (leader commit)
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* s_flags = reinterpret_cast<volatile int*>(s_tmem + 1);  // [0] abort
  int* s_istart = reinterpret_cast<int*>(smem + G2_OFF_MISC);
  int* s_off = s_istart + MAX_E + 1;
  uint32_t* s_e4m3 = reinterpret_cast<uint32_t*>(s_off + MAX_E + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const uint32_t peer_flags = mapa_shared(const_cast<int*>(s_flags), rank ^ 1u);
  auto abort_pair = [&]() {
    s_flags[0] = 1;
    st_remote_u32(peer_flags, 1u);
    set_status(p.status, DEV_TIMEOUT);
  };
  if (tid == 0) {
    for (int s = 0; s < G2_PSTAGES; ++s) {
      mbar_init(&pfull[s], 1);
      mbar_init(&pempty[s], G2_DQ_PER_GROUP);
    }
    for (int s = 0; s < G2_OSTAGES; ++s) {
      mbar_init(&bfull[s], 1);
      mbar_init(&afull[s], 2 * G2_DQ_PER_GROUP);
      mbar_init(&oempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 2 * G2_EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    s_flags[0] = 0;
    fence_mbar_init();
  }
  if (warp == G2_WARP_MMA) {
    tmem_alloc2(s_tmem, G2_TMEM_COLS);
    tmem_relinquish2();
  }
  if (tid >= 96 && tid < 96 + 256)
    s_e4m3[tid - 96] = e4m3_lut_entry<ACT_BF16>((uint32_t)(tid - 96));
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated, before any remote access
  tc_fence_after();
  pdl_wait();      // everything below reads or writes global memory
  pdl_trigger();
  for (int e = tid; e <= p.E; e += blockDim.x) s_off[e] = p.offsets[e];
  __syncthreads();
  if (warp == 0) {
    const int S = p.T * p.topk;
    bool bad = (s_off[0] != 0) || (s_off[p.E] != S);
    int run = 0;
    const int RP = (p.RT + 1) / 2;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      int ni = 0;
      if (e < p.E) {
        const int ne = s_off[e + 1] - s_off[e];
        if (ne < 0) bad = true;
        const bool nf3 = (p.tab.loc[e] & LOC_NF3) != 0;
        const bool sel = nf3 ? (p.tier_mask & 2) : (p.tier_mask & 1);
        ni = (sel && ne > 0) ? ((ne + G2_N - 1) / G2_N) * RP : 0;
      }
      int incl = ni;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int nb = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += nb;
      }
      if (e < p.E) s_istart[e] = run + incl - ni;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      s_istart[p.E] = bad ? 0 : run;
      if (bad && blockIdx.x == 0) set_status(p.status, DEV_BAD_ROUTE);
    }
    if (bad)
      for (int e = lane; e < p.E; e += 32) s_istart[e] = 0;
  }
  __syncthreads();
  const uint32_t tmem_base = *s_tmem;
  const int n_items = s_istart[p.E];
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const uint64_t lim = p.wait_limit_ns;

  if (warp == G2_WARP_PPROD) {
    // ------------------------------------------------ packed weight tile of this CTA's row tile
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      int slot = 0, issued = 0;
      uint32_t ph = 0;
      bool aborted = false;
      for (int i = pair; i < n_items && !aborted; i += n_pairs) {
        const G2Item it = g2_decode(p, s_istart, s_off, i, (int)rank);
        const int fmt = gt_expert_fmt(p, it.e);
        const uint32_t tb = (uint32_t)tile_bytes(fmt);
        const uint8_t* base = (fmt == FMT_NF3 ? p.nf3_buf : p.kept_buf) +
                              (size_t)(p.tab.loc[it.e] & 0x7FFF) *
                                  (fmt == FMT_NF3 ? p.nf3_expert_bytes : p.kept_expert_bytes) +
                              (p.which == 2 ? (fmt == FMT_NF3 ? p.nf3_w2_off : p.kept_w2_off) : 0) +
                              (size_t)it.rt * p.KB * tb;
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!mbar_wait(&pempty[slot], ph ^ 1u, s_flags, lim)) {
            aborted = true;
            break;
          }
          mbar_arrive_expect_tx(&pfull[slot], tb);
          bulk_g2s_stream(smem + G2_OFF_P + slot * G2_P_TILE, base + (size_t)kb * tb, tb, &pfull[slot], pol);
          ++issued;
          if (++slot == G2_PSTAGES) {
            slot = 0;
            ph ^= 1u;
          }
        }
      }
      if (aborted) {
        abort_pair();
        volatile int never = 0;
        for (int b = 0; b < G2_PSTAGES && b < issued; ++b) {
          if (--slot < 0) {
            slot = G2_PSTAGES - 1;
            ph ^= 1u;
          }
          mbar_wait(&pfull[slot], ph, &never, lim);
        }
      }
    }
  } else if (warp == G2_WARP_BPROD) {
    // ------------------------------------------------ this CTA's half of the token columns
    if (lane == 0) {
      int slot = 0, issued = 0;
      uint32_t ph = 0;
      bool aborted = false;
      for (int i = pair; i < n_items && !aborted; i += n_pairs) {
        const G2Item it = g2_decode(p, s_istart, s_off, i, (int)rank);
        const int half = g2_width(it.n) / 2;
        const int row0 = it.p0 + (int)rank * half;
        const int nbox = (half + G2_BBOX - 1) / G2_BBOX;
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!mbar_wait_cluster(&oempty[slot], ph ^ 1u, s_flags, lim)) {
            aborted = true;
            break;
          }
          // The leader's barrier expects the bytes of both halves; each CTA's
          // loads land in its own shared memory and complete there.
          if (leader) mbar_arrive_expect_tx(&bfull[slot], (uint32_t)(2 * nbox * G2_BBOX * 128));
          const uint32_t bar = mapa_shared(&bfull[slot], 0);
          for (int b = 0; b < nbox; ++b)
            tma_load_2d_pair(smem + G2_OFF_B + slot * G2_B_BYTES + b * G2_BBOX * 128, &tmap_b, kb * TILE_K,
                             row0 + b * G2_BBOX, bar);
          if (kb + GT_BPREFETCH < p.KB)
            for (int b = 0; b < nbox; ++b)
              tma_prefetch_2d(&tmap_b, (kb + GT_BPREFETCH) * TILE_K, row0 + b * G2_BBOX);
          ++issued;
          if (++slot == G2_OSTAGES) {
            slot = 0;
            ph ^= 1u;
          }
        }
      }
      if (aborted) {
        // Loads in flight complete on the leader's barriers; the final
        // cluster barrier keeps both CTAs (and their shared memory) alive
        // until the leader has drained its waits.
        abort_pair();
        if (leader) {
          volatile int never = 0;
          for (int b = 0; b < G2_OSTAGES && b < issued; ++b) {
            if (--slot < 0) {
              slot = G2_OSTAGES - 1;
              ph ^= 1u;
            }
            mbar_wait(&afull[slot], ph, &never, lim);
          }
        }
      }
    }
  } else if (warp == G2_WARP_MMA) {
    if (leader) {
      // ------------------------------------------------ MMA issuer for the pair
      // The whole warp runs the loop, so that the MMA operands are computed in
      // converged code and are warp-uniform; lane 0 issues the MMAs and the
      // commits (a commit tracks the MMAs of the thread that issues it).
      int os = 0;
      uint32_t oph = 0;
      bool aborted = false;
      int j = 0;
      const uint32_t a_lo0 = smem_desc_sw128_lo(smem_u32(smem + G2_OFF_A));
      const uint32_t b_lo0 = smem_desc_sw128_lo(smem_u32(smem + G2_OFF_B));
      for (int i = pair; i < n_items && !aborted; i += n_pairs, ++j) {
        const G2Item it = g2_decode(p, s_istart, s_off, i, 0);
        const int buf = j & 1;
        const uint32_t par = ((uint32_t)(j >> 1) & 1u) ^ 1u;
        if (!__all_sync(0xffffffffu, mbar_wait_cluster(&acc_empty[buf], par, s_flags, lim))) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t idesc = idesc_kf16<ACT_BF16>(256, g2_width(it.n));
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * G2_N);
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait_cluster(&afull[os], oph, s_flags, lim) &&
                                           mbar_wait_cluster(&bfull[os], oph, s_flags, lim))) {
            aborted = true;
            break;
          }
          const uint32_t a_lo = a_lo0 + (uint32_t)os * (G2_A_BYTES >> 4);
          const uint32_t b_lo = b_lo0 + (uint32_t)os * (G2_B_BYTES >> 4);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma2_kf16_warp(d_tmem, desc_from_lo(a_lo + 2 * ks), desc_from_lo(b_lo + 2 * ks), idesc,
                            (kb | ks) ? 1u : 0u);
          umma2_commit_both(&oempty[os]);
          if (++os == G2_OSTAGES) {
            os = 0;
            oph ^= 1u;
          }
        }
        if (!aborted) umma2_commit_both(&acc_full[buf]);
      }
      if (aborted && lane == 0) abort_pair();
      umma2_commit_both(mma_done);  // completes once every MMA issued above has
    }
    // Both CTAs: wait for the leader's final commit, so that no MMA still
    // reads this CTA's shared memory or writes its TMEM (bounded; the leader
    // always commits it).
    if (lane == 0) {
      volatile int never = 0;
      if (!mbar_wait_cluster(mma_done, 0, &never, lim)) set_status(p.status, DEV_TIMEOUT);
    }
    __syncwarp();
  } else if (warp < G2_WARP_EPI0) {
    // ------------------------------------------------ dequantisers
    const int dq = warp - G2_WARP_DQ0;
    const int par = dq / G2_DQ_PER_GROUP, rg = dq % G2_DQ_PER_GROUP;
    const uint32_t r_afull = mapa_shared(afull, 0);
    int ps = 0, as = 0;
    uint32_t pph = 0, aph = 0, gk = 0;
    bool ok = true;
    for (int i = pair; i < n_items && ok; i += n_pairs) {
      const G2Item it = g2_decode(p, s_istart, s_off, i, (int)rank);
      const int fmt = gt_expert_fmt(p, it.e);
      for (int kb = 0; kb < p.KB && ok; ++kb, ++gk) {
        if ((int)(gk % G2_DQ_GROUPS) == par) {
          if (!__all_sync(0xffffffffu, mbar_wait(&pfull[ps], pph, s_flags, lim)) ||
              !__all_sync(0xffffffffu, mbar_wait_cluster(&oempty[as], aph ^ 1u, s_flags, lim))) {
            ok = false;
            break;
          }
          const uint8_t* pt = smem + G2_OFF_P + ps * G2_P_TILE;
          uint8_t* at = smem + G2_OFF_A + as * G2_A_BYTES;
          if (fmt == FMT_NVFP4) gt_dequant_slot<FMT_NVFP4>(pt, at, rg, lane, s_e4m3);
          else if (fmt == FMT_MXFP4) gt_dequant_slot<FMT_MXFP4>(pt, at, rg, lane, s_e4m3);
          else gt_dequant_slot<FMT_NF3>(pt, at, rg, lane, s_e4m3);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&pempty[ps]);
            if (leader) mbar_arrive(&afull[as]);
            else mbar_arrive_remote(r_afull + (uint32_t)(as * 8));
          }
        }
        if (++ps == G2_PSTAGES) {
          ps = 0;
          pph ^= 1u;
        }
        if (++as == G2_OSTAGES) {
          as = 0;
          aph ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) abort_pair();
  } else {
    // ------------------------------------------------ epilogue: this CTA's 128 rows x N accumulator
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int S = p.T * p.topk;
    const uint32_t r_acc_empty = mapa_shared(acc_empty, 0);
    int j = 0;
    for (int i = pair; i < n_items; i += n_pairs, ++j) {
      const G2Item it = g2_decode(p, s_istart, s_off, i, (int)rank);
      const int buf = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait_cluster(&acc_full[buf], (uint32_t)(j >> 1) & 1u, s_flags, lim))) {
        if (lane == 0) abort_pair();
        break;
      }
      tc_fence_after();
      const uint32_t col0 = (uint32_t)(buf * G2_N);
      if (it.valid && p.which == 13) {
        const float gsc = p.tab.g13[it.e] * (gt_expert_fmt(p, it.e) == FMT_NVFP4 ? NVFP4_UNSCALE : 1.0f) * p.act_scale;
        const int g = lane >> 2, qq = lane & 3;
        for (int h = 0; h < 2; ++h) {
          const int ch = it.rt * 64 + (2 * quarter + h) * 8 + g;
          const uint32_t ta = tmem_base + ((uint32_t)(quarter * 32 + 16 * h) << 16) + col0;
          for (int c0 = 0; c0 < it.n; c0 += 32) {
            uint32_t v[16];
            tmem_ld16x256x4(ta + (uint32_t)c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int rep = 0; rep < 4; ++rep) {
#pragma unroll
              for (int b = 0; b < 2; ++b) {
                const int col = c0 + 8 * rep + 2 * qq + b;
                const float gate = __uint_as_float(v[4 * rep + b]) * gsc;
                const float up = __uint_as_float(v[4 * rep + 2 + b]) * gsc;
                if (col < it.n) p.h_out[(size_t)(it.p0 + col) * p.I + ch] = f32_to_act<ACT_BF16>(silu_fast(gate) * up);
              }
            }
          }
        }
      } else if (it.valid) {
        const float gsc = p.tab.g2[it.e] * (gt_expert_fmt(p, it.e) == FMT_NVFP4 ? NVFP4_UNSCALE : 1.0f) * p.act_scale;
        const int orow = it.rt * 128 + row;
        const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + col0;
        for (int c0 = 0; c0 < it.n; c0 += 32) {
          int my_s = -1;
          if (c0 + lane < it.n) {
            const int sc = p.perm[it.p0 + c0 + lane];
            if (sc >= 0 && sc < S) my_s = sc;
            else set_status(p.status, DEV_BAD_ROUTE);
          }
          uint32_t v[32];
          tmem_ld32(taddr + (uint32_t)c0, v);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int sc = __shfl_sync(0xffffffffu, my_s, c);
            if (sc >= 0) p.y_out[(size_t)sc * p.H + orow] = __uint_as_float(v[c]) * gsc;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&acc_empty[buf]);
        else mbar_arrive_remote(r_acc_empty + (uint32_t)(buf * 8));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its partner may still touch its shared memory
  if (warp == G2_WARP_MMA) {
    tc_fence_after();
    tmem_dealloc2(tmem_base, G2_TMEM_COLS);
  }
}

// ------------------------------------------------------------ gather of activation rows
// xg[p] = x[perm[p] / k]: one warp per permuted row (perm read once per row),
// its lanes copying the row's 16-byte vectors with several loads in flight.
// (A flat index over rows x vectors needed a 64-bit division per vector.)
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x, const int* __restrict__ perm,
                                                          int S, int k, int H, uint16_t* __restrict__ xg, int* status) {
  pdl_wait();
  pdl_trigger();
  const int vec = H / 8;  // 16-byte vectors per row
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int pidx = blockIdx.x * wpb + (threadIdx.x >> 5); pidx < S; pidx += gridDim.x * wpb) {
    int s = perm[pidx];
    if (s < 0 || s >= S) {
      if (lane == 0) set_status(status, DEV_BAD_ROUTE);
      s = 0;
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(s / k) * H);
    uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)pidx * H);
#pragma unroll 8
    for (int c = lane; c < vec; c += 32) dst[c] = __ldg(src + c);
  }
}

cudaError_t launch_gather_rows(const uint16_t* x, const int* perm, int S, int k, int T, int H, uint16_t* xg,
                               int* status, int num_sms, cudaStream_t st) {
  (void)T;
  if (S == 0) return cudaSuccess;
  const long long blocks = ((long long)S + 7) / 8;
  const int grid = (int)(blocks < (long long)num_sms * 16 ? blocks : (long long)num_sms * 16);
  cudaError_t e = launch_pdl(gather_rows_kernel, dim3(grid), dim3(256), 0, st, x, perm, S, k, H, xg, status);
  count_launches(1);
  return e;
}

// ------------------------------------------------------------ host side
// The driver's tensor-map encoder. A successful lookup is cached; a failed
// one is retried on the next call (the atomic makes the cache safe with
// several host threads: each may look it up, all store the same pointer).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> cached{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 fn = cached.load(std::memory_order_acquire);
  if (fn) return fn;
  cudaDriverEntryPointQueryResult q;
  void* ptr = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !ptr)
    return nullptr;
  fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  cached.store(fn, std::memory_order_release);
  return fn;
}

// Clusters of two that can be resident at once on this device, for the
// pair kernel: its persistent grid must not exceed them, or the clusters that
// do not fit would start only after others had finished. Cached per device.
static int pair_clusters(int num_sms) {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_acquire);
    if (c > 0) return c;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_sms & ~1));
  cfg.blockDim = dim3(G2_THREADS);
  cfg.dynamicSmemBytes = G2_SMEM_BYTES;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, grouped_pair_kernel, &cfg) != cudaSuccess || n <= 0) return 0;
  n = std::min(n, num_sms / 2);
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_release);
  return n;
}

cudaError_t launch_grouped_gemm(const GroupedParams& p, const uint16_t* b_src, int b_rows, int num_sms,
                                cudaStream_t st) {
  static std::atomic<unsigned long long> attr1{0}, attr1h{0}, attr2{0};
  cudaError_t ea = ensure_smem_attr(grouped_gemm_kernel<ACT_BF16>, GT_SMEM_BYTES, attr1);
  if (ea == cudaSuccess) ea = ensure_smem_attr(grouped_gemm_kernel<ACT_F16>, GT_SMEM_BYTES, attr1h);
  if (ea == cudaSuccess) ea = ensure_smem_attr(grouped_pair_kernel, G2_SMEM_BYTES, attr2);
  if (ea != cudaSuccess) return ea;
  // The CTA-pair kernel takes bf16 operands only.
  if ((p.act_type != ACT_BF16 && p.act_type != ACT_F16) || (p.pair && p.act_type != ACT_BF16))
    return cudaErrorInvalidValue;
  if (b_rows <= 0) return cudaSuccess;
  if ((reinterpret_cast<uintptr_t>(b_src) & 15) != 0 || (p.K % TILE_K) != 0) return cudaErrorInvalidValue;
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)b_rows};
  const cuuint64_t strides[1] = {(cuuint64_t)p.K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)TILE_K, (cuuint32_t)(p.pair ? G2_BBOX : GT_N)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map, p.act_type == ACT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<uint16_t*>(b_src), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  cudaError_t e;
  if (!p.pair) {
    e = p.act_type == ACT_F16
            ? launch_pdl(grouped_gemm_kernel<ACT_F16>, dim3(num_sms), dim3(GT_THREADS), GT_SMEM_BYTES, st, p, map)
            : launch_pdl(grouped_gemm_kernel<ACT_BF16>, dim3(num_sms), dim3(GT_THREADS), GT_SMEM_BYTES, st, p, map);
  } else {
    const int pairs = pair_clusters(num_sms);
    if (pairs <= 0) return cudaErrorNotSupported;
    e = launch_pdl(grouped_pair_kernel, dim3(2 * pairs), dim3(G2_THREADS), G2_SMEM_BYTES, st, p, map);
  }
  count_launches(1);
  return e;
}

}  // namespace hmoe
