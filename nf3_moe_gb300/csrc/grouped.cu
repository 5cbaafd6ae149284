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
// each), with row-tile pairs fastest. Both row tiles of an item multiply
// the same activation tile, so each activation tile is read from L2 once per
// 256 weight rows; the CTAs running together also share it through L2. An
// expert's token tiles follow each other, so its weight tiles are re-read
// from L2 rather than HBM.
//
// Warp roles (24 warps):
//   warp 0       packed-weight producer. 1D bulk copies of each k-block's
//                two packed tiles (64 K each) into a 4-deep ring.
//   warp 2       activation producer. A 2D TMA tensor load (128 rows x 64
//                bf16, 128B swizzle) into the k-block's operand slot (a
//                3-deep ring whose slots also hold the dequantised weight
//                tiles), plus an L2 prefetch of the tile needed 8 k-blocks
//                later.
//   warps 1, 23  MMA issuers (warp 1 also allocates 512 TMEM columns).
//                Issuing a tcgen05.mma costs the issuing thread about 100
//                cycles, so each row tile has its own issuing lane: per
//                k-block it issues 4 tcgen05.mma.kind::f16 (M=128, N = token
//                count rounded up to 16, K=16) into its row tile's fp32
//                accumulator, double-buffered in TMEM. Both issuers'
//                tcgen05.commits free the operand slot (one commit each per
//                k-block).
//   warps 3..18  dequantisers, in two groups of 8 that take alternate
//                k-blocks. Per k-block each warp expands its 16-row group of
//                both row tiles: each thread turns one tile slot (2 rows x
//                16 K) of each into bf16 (E2M1 x E4M3, E2M1 x 2^e, or
//                bf16_rne(NF3 codebook x scale)) in the canonical K-major
//                SWIZZLE_128B operand layout, then fences the async proxy.
//   warps 19..22 epilogue. tcgen05.ld of the accumulators (each warp owns 32
//                TMEM lanes, i.e. 32 weight rows of each row tile).
//                W13: rows come in gate/up pairs 8 lanes apart, and one
//                16x256b load gives a thread both, so
//                h = bf16(silu(g13*gate) * (g13*up)) needs no shuffle.
//                W2: y[s][row] = g2 * acc for the flat slot s = perm[p].
// Every mbarrier wait is bounded. On a timeout the CTA records
// DEV_TIMEOUT, drains its copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace hmoe {

constexpr int GT_N = 128;                 // token tile
constexpr int GT_R = 2;                   // weight row tiles per item (they share the activation tile)
constexpr int GT_A_TILE = 128 * 128;      // bf16 A tile 128 x 64
constexpr int GT_A_BYTES = GT_R * GT_A_TILE;
constexpr int GT_B_BYTES = GT_N * 128;    // bf16 B tile GT_N x 64
constexpr int GT_P_TILE = 4608;           // largest packed tile
constexpr int GT_P_BYTES = GT_R * GT_P_TILE;
constexpr int GT_PSTAGES = 4;             // packed weight tiles in flight
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
constexpr int GT_WARP_PPROD = 0, GT_WARP_MMA = 1, GT_WARP_BPROD = 2, GT_WARP_DQ0 = 3;
constexpr int GT_WARP_EPI0 = GT_WARP_DQ0 + GT_DQ_WARPS;
// A second MMA-issuing warp: each issuer drives one row tile's accumulator.
constexpr int GT_WARP_MMA2 = GT_WARP_EPI0 + GT_EPI_WARPS;
constexpr int GT_MMA_ISSUERS = GT_R;
static_assert(GT_MMA_ISSUERS == 2, "issuer r drives row tile r");
constexpr int GT_THREADS = (GT_WARP_MMA2 + 1) * 32;
constexpr int GT_TMEM_COLS = 2 * GT_R * GT_N;   // [buffer][row tile] accumulators
// Shared memory map (offsets from the 1024-aligned base).
constexpr int GT_OFF_A = 0;
constexpr int GT_OFF_B = GT_OFF_A + GT_OSTAGES * GT_A_BYTES;
constexpr int GT_OFF_P = GT_OFF_B + GT_OSTAGES * GT_B_BYTES;
constexpr int GT_OFF_BAR = GT_OFF_P + GT_PSTAGES * GT_P_BYTES;
constexpr int GT_NBAR = 2 * GT_PSTAGES + 3 * GT_OSTAGES + 4 + GT_MMA_ISSUERS;
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
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same MMA with the accumulate flag known to be set (k-steps after the first).
__device__ __forceinline__ void umma_bf16_acc(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.eq.u32 p, 1, 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
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

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
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

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct GtItem {
  int e, p0, n, rt, nr;  // row tiles rt .. rt + nr - 1 (nr = 1 or 2)
};

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
  // Row-tile pairs fastest: the CTAs that run together share one activation
  // tile through L2, and an expert's token tiles follow each other, so its
  // weight tiles are re-read from L2 rather than HBM.
  const int RP = (p.RT + GT_R - 1) / GT_R;
  const int local = i - s_istart[lo];
  it.rt = (local % RP) * GT_R;
  it.nr = min(GT_R, p.RT - it.rt);
  const int nt = local / RP;
  it.p0 = o0 + nt * GT_N;
  it.n = min(GT_N, ne - nt * GT_N);
  return it;
}

// Writes one thread slot's dequantised rows (2 rows x 16 K) into the
// canonical K-major SWIZZLE_128B tile: row r of atom (r / 8) at (r % 8) * 128,
// 16-byte chunk c stored at chunk position c ^ (r % 8).
template <int FMT>
__device__ __forceinline__ void gt_dequant_slot(const uint8_t* ptile, uint8_t* atile, int rg, int lane,
                                                const uint32_t* e4m3_lut) {
  uint32_t r0[8], r1[8];
  float s0, s1;
  dequant_slot<FMT, true>(ptile, rg, lane, r0, r1, &s0, &s1, e4m3_lut);
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
template <int FMT>
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
        gt_dequant_slot<FMT>(pt, at, rg + h, lane, s_e4m3);
        if (nr > 1) gt_dequant_slot<FMT>(pt + GT_P_TILE, at + GT_A_TILE, rg + h, lane, s_e4m3);
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

__global__ void __launch_bounds__(GT_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ GroupedParams p, const __grid_constant__ CUtensorMap tmap_b) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + GT_OFF_BAR);
  uint64_t* pfull = bars;                              // packed tile landed (tx)
  uint64_t* pempty = pfull + GT_PSTAGES;               // dequant warps done reading it
  uint64_t* bfull = pempty + GT_PSTAGES;               // activation tile landed (tx)
  uint64_t* afull = bfull + GT_OSTAGES;                // dequant warps wrote the weight tiles
  uint64_t* oempty = afull + GT_OSTAGES;               // MMAs that read the slot completed
  uint64_t* acc_full = oempty + GT_OSTAGES;            // [2] accumulator ready for the epilogue
  uint64_t* acc_empty = acc_full + 2;                  // [2] epilogue drained it
  uint64_t* mma_done = acc_empty + 2;                  // [issuer] final drain before TMEM release
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(mma_done + GT_MMA_ISSUERS);
  volatile int* s_flags = reinterpret_cast<volatile int*>(s_tmem + 1);  // [0] abort
  int* s_istart = reinterpret_cast<int*>(smem + GT_OFF_MISC);
  int* s_off = s_istart + MAX_E + 1;
  uint32_t* s_e4m3 = reinterpret_cast<uint32_t*>(s_off + MAX_E + 1);  // E4M3 -> bf16 pair

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < GT_PSTAGES; ++s) {
      mbar_init(&pfull[s], 1);
      mbar_init(&pempty[s], GT_DQ_PER_GROUP);
    }
    for (int s = 0; s < GT_OSTAGES; ++s) {
      mbar_init(&bfull[s], 1);
      mbar_init(&afull[s], GT_DQ_PER_GROUP);
      mbar_init(&oempty[s], GT_MMA_ISSUERS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], GT_MMA_ISSUERS);
      mbar_init(&acc_empty[b], GT_EPI_WARPS);
    }
    for (int r = 0; r < GT_MMA_ISSUERS; ++r) mbar_init(&mma_done[r], 1);
    fence_mbar_init();
    s_flags[0] = 0;
  }
  if (warp == GT_WARP_MMA) {
    tmem_alloc(s_tmem, GT_TMEM_COLS);
    tmem_relinquish();
  }
  if (tid >= 96 && tid < 96 + 256)
    s_e4m3[tid - 96] = bf16x2_mul(bf16_bcast(e4m3_to_bf16((uint32_t)(tid - 96))), BF16X2_2P63);
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
        ni = (sel && ne > 0) ? ((ne + GT_N - 1) / GT_N) * ((p.RT + GT_R - 1) / GT_R) : 0;
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
    if (lane == 0) {
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
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!mbar_wait(&pempty[slot], ph ^ 1u, s_flags, lim)) {
            aborted = true;
            break;
          }
          mbar_arrive_expect_tx(&pfull[slot], tb * (uint32_t)it.nr);
          for (int r = 0; r < it.nr; ++r)
            bulk_g2s_stream(smem + GT_OFF_P + slot * GT_P_BYTES + r * GT_P_TILE, base + r * rt_stride + (size_t)kb * tb,
                            tb, &pfull[slot], pol);
          ++issued;
          if (++slot == GT_PSTAGES) {
            slot = 0;
            ph ^= 1u;
          }
        }
      }
      if (aborted) {
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
    }
  } else if (warp == GT_WARP_BPROD) {
    // ------------------------------------------------ activation tiles (L2), TMA tensor loads
    if (lane == 0) {
      int slot = 0, issued = 0;
      uint32_t ph = 0;
      bool aborted = false;
      for (int i = blockIdx.x; i < n_items && !aborted; i += gridDim.x) {
        const GtItem it = gt_decode(p, s_istart, s_off, i);
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!mbar_wait(&oempty[slot], ph ^ 1u, s_flags, lim)) {
            aborted = true;
            break;
          }
          mbar_arrive_expect_tx(&bfull[slot], GT_B_BYTES);
          tma_load_2d(smem + GT_OFF_B + slot * GT_B_BYTES, &tmap_b, kb * TILE_K, it.p0, &bfull[slot]);
          // Warm L2 with a tile needed a few loads from now (same token tile).
          if (kb + GT_BPREFETCH < p.KB) tma_prefetch_2d(&tmap_b, (kb + GT_BPREFETCH) * TILE_K, it.p0);
          ++issued;
          if (++slot == GT_OSTAGES) {
            slot = 0;
            ph ^= 1u;
          }
        }
      }
      if (aborted) {
        s_flags[0] = 1;
        set_status(p.status, DEV_TIMEOUT);
        volatile int never = 0;
        for (int b = 0; b < GT_OSTAGES && b < issued; ++b) {
          if (--slot < 0) {
            slot = GT_OSTAGES - 1;
            ph ^= 1u;
          }
          mbar_wait(&bfull[slot], ph, &never, lim);
        }
      }
    }
  } else if (warp == GT_WARP_MMA || warp == GT_WARP_MMA2) {
    // ------------------------------------------------ MMA issuers
    // Issuing one tcgen05.mma costs the issuing thread about 100 cycles, so
    // two threads in different warps (and SM sub-partitions) issue: issuer r
    // drives row tile r's accumulator. Both wait for the same operand stages
    // and both commit to the barriers that free them (two arrivals each).
    const int my_r = warp == GT_WARP_MMA ? 0 : 1;
    if (lane == 0) {
      const uint32_t a_lo0 = smem_desc_sw128_lo(smem_u32(smem + GT_OFF_A));
      const uint32_t b_lo0 = smem_desc_sw128_lo(smem_u32(smem + GT_OFF_B));
      int os = 0;
      uint32_t oph = 0;
      bool aborted = false;
      int j = 0;
      for (int i = blockIdx.x; i < n_items && !aborted; i += gridDim.x, ++j) {
        const GtItem it = gt_decode(p, s_istart, s_off, i);
        const int buf = j & 1;
        if (!mbar_wait(&acc_empty[buf], ((uint32_t)(j >> 1) & 1u) ^ 1u, s_flags, lim)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const int npad = max(16, (it.n + 15) & ~15);
        const uint32_t idesc = idesc_bf16(128, npad);
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * GT_R * GT_N);
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!mbar_wait(&afull[os], oph, s_flags, lim) || !mbar_wait(&bfull[os], oph, s_flags, lim)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          // Descriptor low words of this stage's A and B tiles (k-step 0).
          const uint32_t a_lo = a_lo0 + (uint32_t)os * (GT_A_BYTES >> 4);
          const uint32_t b_lo = b_lo0 + (uint32_t)os * (GT_B_BYTES >> 4);
          if (my_r < it.nr) {
            const uint32_t ar = a_lo + (uint32_t)my_r * (GT_A_TILE >> 4);
            const uint32_t dr = d_tmem + (uint32_t)(my_r * GT_N);
            umma_bf16(dr, desc_from_lo(ar), desc_from_lo(b_lo), idesc, kb ? 1u : 0u);
            umma_bf16_acc(dr, desc_from_lo(ar + 2), desc_from_lo(b_lo + 2), idesc);
            umma_bf16_acc(dr, desc_from_lo(ar + 4), desc_from_lo(b_lo + 4), idesc);
            umma_bf16_acc(dr, desc_from_lo(ar + 6), desc_from_lo(b_lo + 6), idesc);
          }
          umma_commit(&oempty[os]);
          if (++os == GT_OSTAGES) {
            os = 0;
            oph ^= 1u;
          }
        }
        if (!aborted) umma_commit(&acc_full[buf]);
      }
      if (aborted) {
        s_flags[0] = 1;
        set_status(p.status, DEV_TIMEOUT);
      }
      // Drain every MMA this thread issued before TMEM can be released.
      umma_commit(&mma_done[my_r]);
      volatile int never = 0;
      mbar_wait(&mma_done[my_r], 0, &never, lim);
    }
  } else if (warp < GT_WARP_EPI0) {
    // ------------------------------------------------ dequantisers: packed tile -> bf16 operand tile
    // Group par expands the k-blocks k with k % GT_DQ_GROUPS == par, every
    // row tile; its warps split the 8 row groups. (Eight warps each expanding
    // both row tiles of every k-block was measured slower: 4.18 against 4.03
    // ms at M=4096.)
    const int dq = warp - GT_WARP_DQ0;
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
        ok = gt_dequant_item<FMT_NVFP4>(p.KB, it.nr, par, p_base, a_base, pfull, pempty, afull, oempty, s_e4m3, rg,
                                        lane, s_flags, lim, gk, ps, pph, as, aph);
      else if (fmt == FMT_MXFP4)
        ok = gt_dequant_item<FMT_MXFP4>(p.KB, it.nr, par, p_base, a_base, pfull, pempty, afull, oempty, s_e4m3, rg,
                                        lane, s_flags, lim, gk, ps, pph, as, aph);
      else
        ok = gt_dequant_item<FMT_NF3>(p.KB, it.nr, par, p_base, a_base, pfull, pempty, afull, oempty, s_e4m3, rg,
                                      lane, s_flags, lim, gk, ps, pph, as, aph);
    }
    if (!ok && lane == 0) {
      s_flags[0] = 1;
      set_status(p.status, DEV_TIMEOUT);
    }
  } else {
    // ------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // tile row = TMEM lane
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
      // W2: the flat slot of each of the item's token columns (column
      // 32u + lane in item_slot[u]); -1 past the item or for a bad entry.
      int item_slot[GT_N / 32];
#pragma unroll
      for (int u = 0; u < GT_N / 32; ++u) {
        item_slot[u] = -1;
        if (p.which != 13 && 32 * u + lane < it.n) {
          const int sc = p.perm[it.p0 + 32 * u + lane];
          if (sc >= 0 && sc < S) item_slot[u] = sc;
          else set_status(p.status, DEV_BAD_ROUTE);
        }
      }
      for (int r = 0; r < it.nr; ++r) {
        const int rt = it.rt + r;
        const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)((buf * GT_R + r) * GT_N);
        if (p.which == 13) {
          // A 16-row group holds 8 gate rows then the 8 up rows of the same
          // channels, so the 16x256b load gives each thread gate and up of
          // one channel (row 16j + lane/4) for 8 token columns: SwiGLU in
          // registers, every lane busy. The quarter holds groups 2q, 2q + 1.
          const float gsc = p.tab.g13[it.e] * (gt_expert_fmt(p, it.e) == FMT_NVFP4 ? NVFP4_UNSCALE : 1.0f);
          const int g = lane >> 2, qq = lane & 3;
          for (int h = 0; h < 2; ++h) {
            const int grp16 = 2 * quarter + h;
            const int ch = rt * 64 + grp16 * 8 + g;
            const uint32_t ta = tmem_base + ((uint32_t)(quarter * 32 + 16 * h) << 16) +
                                (uint32_t)((buf * GT_R + r) * GT_N);
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
                  if (col < it.n)
                    p.h_out[(size_t)(it.p0 + col) * p.I + ch] = __float2bfloat16_rn(silu_fast(gate) * up);
                }
              }
            }
          }
        } else {
          // W2: lanes are output rows, so each column's store is one
          // coalesced row segment of slot s = perm[p0 + column].
          const float gsc = p.tab.g2[it.e] * (gt_expert_fmt(p, it.e) == FMT_NVFP4 ? NVFP4_UNSCALE : 1.0f);
          const int orow = rt * 128 + row;
#pragma unroll
          for (int u = 0; u < GT_N / 32; ++u) {
            if (32 * u >= it.n) break;
            uint32_t v[32];
            tmem_ld32(taddr + (uint32_t)(32 * u), v);
            tmem_wait_ld();
            const int my_s = item_slot[u];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const int sc = __shfl_sync(0xffffffffu, my_s, c);
              if (sc >= 0) p.y_out[(size_t)sc * p.H + orow] = __uint_as_float(v[c]) * gsc;
            }
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

// ------------------------------------------------------------ gather of activation rows
__global__ void gather_rows_kernel(const __nv_bfloat16* __restrict__ x, const int* __restrict__ perm, int S, int k,
                                   int T, int H, __nv_bfloat16* __restrict__ xg, int* status) {
  pdl_wait();
  pdl_trigger();
  const int vec = H / 8;  // 16-byte vectors per row
  const long long n = (long long)S * vec;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int pidx = (int)(i / vec), c = (int)(i % vec);
    int s = perm[pidx];
    if (s < 0 || s >= S) {
      if (c == 0) set_status(status, DEV_BAD_ROUTE);
      s = 0;
    }
    const int t = s / k;
    reinterpret_cast<uint4*>(xg + (size_t)pidx * H)[c] =
        __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H) + c);
  }
  (void)T;
}

cudaError_t launch_gather_rows(const __nv_bfloat16* x, const int* perm, int S, int k, int T, int H,
                               __nv_bfloat16* xg, int* status, int num_sms, cudaStream_t st) {
  if (S == 0) return cudaSuccess;
  const long long n = (long long)S * (H / 8);
  const long long blocks = (n + 255) / 256;
  const int grid = (int)(blocks < (long long)num_sms * 8 ? blocks : (long long)num_sms * 8);
  cudaError_t e = launch_pdl(gather_rows_kernel, dim3(grid), dim3(256), 0, st, x, perm, S, k, T, H, xg, status);
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

cudaError_t launch_grouped_gemm(const GroupedParams& p, const __nv_bfloat16* b_src, int b_rows, int num_sms,
                                cudaStream_t st) {
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t ea = ensure_smem_attr(grouped_gemm_kernel, GT_SMEM_BYTES, attr_done);
  if (ea != cudaSuccess) return ea;
  if (b_rows <= 0) return cudaSuccess;
  if ((reinterpret_cast<uintptr_t>(b_src) & 15) != 0 || (p.K % TILE_K) != 0) return cudaErrorInvalidValue;
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)b_rows};
  const cuuint64_t strides[1] = {(cuuint64_t)p.K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)TILE_K, (cuuint32_t)GT_N};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(b_src), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(grouped_gemm_kernel, dim3(num_sms), dim3(GT_THREADS), GT_SMEM_BYTES, st, p, map);
  count_launches(1);
  return e;
}

}  // namespace hmoe
