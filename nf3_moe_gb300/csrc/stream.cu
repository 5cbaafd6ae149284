// stream.cu -- the weight-streaming grouped GEMM (the M <= 8 decode path; valid at any T).
//
// Cites: "quant: nvfp4_nf3_hybrid -- native serving for mixed NVFP4+NF3 MoE
// checkpoints", How it works. An M<=8 decode path works on the top-k routed
// experts directly. Both tiers add into one shared output, and the second
// launch accumulates instead of zeroing. Here each routed expert's packed
// weights are streamed from HBM once per group of up to 8 of its tokens.
//
// One launch runs both matrices of the expert FFN. Work items are first
// every (token group, W13 rows), then every (token group, W2 rows), each
// over the whole K extent. The rows of an item are a pair of 128-row tiles
// when the batch makes at least two W13 pair items per CTA (the host
// decides from T * topk and E), else one tile, so that small batches keep
// more SMs busy. A token group is up to 8 consecutive permuted slots of one
// expert, so at T <= 8 there is exactly one group per touched expert.
// Persistent CTAs (2 per SM) pull items from a global work queue that
// resets itself. A W2 item reads the group's h rows, so its producer first
// waits (bounded) until every W13 item of that group has been written: each
// consumer warp counts its finished W13 items into a per-group counter with
// release semantics. W13 items never wait on anything, and every W13 item
// is dequeued before any W2 item, so the waits always end. The W13 tail
// overlaps the W2 start, and there is one launch instead of two. (Past the
// counter array's capacity the host runs the two phases as two launches of
// the same kernel.)
//
// The producer warp streams each item's packed tiles and the group's
// activation rows into a 2-stage shared-memory ring with 1D bulk copies
// (TMA engine), one warp instruction per stage: an elected lane copies the
// weight tiles and lane j the activation row of token j. A stage holds up
// to 8 k-block tiles: 4 k-blocks of each tile of a pair item, or 8 of a
// single-tile item. Eight k-blocks per stage instead of four halve the
// per-stage waits and bookkeeping of the consumers; measured 308 -> 284 us
// at M=8. It writes the item number into each stage header, and a
// terminator stage ends the consumers' loop. Eight consumer warps, one per
// 16-row group, dequantise in registers and issue m16n8k16 MMAs (bf16 or
// fp16 operands, template ACT) with the tokens as the N=8 side. Pair items
// decode the warp's slots of both tiles for one k-block and share one load
// of the activation fragments between them (the activation loads were a
// third of the kernel's shared-memory traffic); single-tile items decode
// two k-blocks' slots before their MMAs. The decoders:
//   NVFP4: shift-and-mask decode (bf16) or nibble-table decode (fp16), the
//     E4M3 scales from a shared table of operand-type pairs, one x2 multiply;
//   MXFP4: nibble-table decode, E8M0 scale multiply;
//   NF3: three of four selector words looked up in a bank-replicated shared
//     table of operand pairs, the fourth decoded with byte-table permutes
//     (the table is bound by shared-memory bandwidth, the permutes by ALU
//     issue; counters put the kernel's shared-memory wavefronts at 74% of
//     peak with the table alone), raw codebook values with the group scale
//     applied to the fp32 partial sums; for W4A4 layers (template TILE) the
//     tile values rne(cb * s), the weights the definition and the
//     tensor-core kernel use.
// Accumulation is fp32 with two accumulator sets per thread: the two tiles
// of a pair item, or alternate k-blocks of a single-tile item. The epilogue
// writes straight from registers:
//   W13: h[p][c] = act(silu(g13 * gate) * (g13 * up)), SwiGLU fused.
//   W2:  y[s][r] = g2 * sum, fp32, indexed by the flat slot s.
// The finalize kernel then applies the gates and sums each token's k slots
// in slot order, so every output element is summed in a fixed order.
// Splitting K across CTAs was measured slower at every batch size (the
// cross-CTA reduction costs more than the idle SMs it fills), so items
// always cover the whole K extent. Measured per M=8 launch: single-tile
// items 240.3 us, pair items 231.3 us; at M=1, pair items 85.4 us against
// 57.0 (too few items for 304 CTAs), hence the choice by batch size.
#include "common.cuh"
#include "internal.h"

namespace hmoe {

constexpr int SK_CONSUMER_WARPS = 8;
constexpr int SK_WARP_PRODUCER = SK_CONSUMER_WARPS;       // warp 8
constexpr int SK_THREADS = (SK_CONSUMER_WARPS + 1) * 32;
constexpr int SK_STAGES = 2;
constexpr int SK_TILES = 2;                                // row tiles per work item
constexpr int SK_MAX_KBS = STREAM_MAX_KBS;                 // k-blocks per tile and stage
// Two CTAs per SM: three (4 k-blocks per stage, 72 registers) measured
// slower, 252.3 against 249.5 us per M=8 launch, and 88.8 against 74.8 us at
// M=1.
constexpr int SK_CTAS_PER_SM = 2;
constexpr int SK_XROW = 2 * SK_MAX_KBS * 128 + 16;        // padded token row, bytes
constexpr int SK_W_BYTES = SK_TILES * SK_MAX_KBS * 4608;
constexpr int SK_X_BYTES = 8 * SK_XROW;
constexpr int SK_HDR_BYTES = 16;                           // {item, stage} written by the producer
constexpr int SK_STAGE_BYTES = SK_W_BYTES + SK_X_BYTES + SK_HDR_BYTES;
constexpr int SK_SMEM_DATA = SK_STAGES * SK_STAGE_BYTES;
constexpr int SK_NBAR = 2 * SK_STAGES;
constexpr int SK_SMEM_BYTES = SK_SMEM_DATA + SK_NBAR * 8 + 2 * (MAX_E + 1) * 4 + 4 * 4 + 256 * 4 + NF3_LUT_BYTES;
static_assert(SK_CTAS_PER_SM * (SK_SMEM_BYTES + 1024) <= 233472, "CTAs per SM");
static_assert(SK_STAGE_BYTES % 16 == 0, "stage alignment");

struct SkItem {
  int e, p0, n, rt, grp, ph;  // rt: row tile, or tile pair (row tiles 2 rt, 2 rt + 1); ph: 0 = W13, 1 = W2
  bool two;                   // pair items: row tile 2 rt + 1 exists (an odd tile count ends on one tile)
};

// Work items of one phase per token group: pairs of row tiles, or row tiles.
__device__ __forceinline__ int tile_pairs(const StreamPhase& P) { return (P.RT + 1) >> 1; }
__device__ __forceinline__ int phase_units(const StreamPhase& P, bool pair) { return pair ? tile_pairs(P) : P.RT; }

__device__ __forceinline__ int expert_fmt(const StreamParams& p, int e) {
  return (p.tab.loc[e] & LOC_NF3) ? FMT_NF3 : p.kept_fmt;
}

__device__ __forceinline__ SkItem decode_item(const StreamParams& p, const int* s_gstart, const int* s_off, int i,
                                              bool pair) {
  SkItem it;
  const int n13 = p.ph_begin == 0 ? s_gstart[p.E] * phase_units(p.ph[0], pair) : 0;
  it.ph = i >= n13 ? 1 : 0;
  const int local = it.ph ? i - n13 : i;
  const int PT = phase_units(p.ph[it.ph], pair);
  it.rt = local % PT;
  it.grp = local / PT;
  it.two = pair && 2 * it.rt + 1 < p.ph[it.ph].RT;
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_gstart[mid] <= it.grp) lo = mid; else hi = mid;
  }
  it.e = lo;
  const int c = it.grp - s_gstart[lo];
  const int o0 = s_off[lo], ne = s_off[lo + 1] - o0;
  it.p0 = o0 + c * p.group_tokens;
  it.n = min(p.group_tokens, ne - c * p.group_tokens);
  return it;
}

// Output of one thread's 2 rows x 2 tokens (v[0],v[1]: row R0; v[2],v[3]: row R1).
template <int ACT>
__device__ __forceinline__ void sk_emit(const StreamParams& p, const SkItem& it, int rt, int rg, int g, int q,
                                        const float* v) {
  const int S = p.T * p.topk;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = 2 * q + h;
    if (c >= it.n) continue;
    const int pp = it.p0 + c;
    if (it.ph == 0) {
      const float gsc =
          p.tab.g13[it.e] * (expert_fmt(p, it.e) == FMT_NVFP4 ? nvfp4_unscale<ACT>() : 1.0f) * p.act_scale13;
      const int ch = rt * 64 + rg * 8 + g;
      const float gate = v[h] * gsc, up = v[2 + h] * gsc;
      p.h_out[(size_t)pp * p.I + ch] = f32_to_act<ACT>(silu_f(gate) * up);
    } else {
      const float gsc =
          p.tab.g2[it.e] * (expert_fmt(p, it.e) == FMT_NVFP4 ? nvfp4_unscale<ACT>() : 1.0f) * p.act_scale2;
      const int s = p.perm[pp];
      if (s < 0 || s >= S) {
        set_status(p.status, DEV_BAD_ROUTE);
        continue;
      }
      const int row = rt * 128 + rg * 16 + g;
      p.y_out[(size_t)s * p.H + row] = v[h] * gsc;
      p.y_out[(size_t)s * p.H + row + 8] = v[2 + h] * gsc;
    }
  }
}

// Pair items. One k-block of one thread slot in both row tiles: dequantise
// through dequant_slot (the decoder hmoe_debug_decode_operand exports;
// NVFP4/MXFP4 scales applied in the operand type from the shared lookup
// table, NF3 values raw with the row scales applied to the fp32 sum of the
// k-block), both slots before any MMA, then 4 MMAs per tile. The two tiles
// share the activation fragments, so one load of the token rows serves 32
// weight rows. With TILE (W4A4 layers) NF3 is decoded to the tile values
// rne(cb * s) instead, the weights the definition and the tensor-core
// kernel use: W4A4 quantises h, so h must come from the same weights on
// both paths. Without TWO (the last item of a phase with an odd tile
// count) only tile 0 is computed.
template <int FMT, int ACT, bool TILE, bool TWO>
__device__ __forceinline__ void sk_kblock(const uint8_t* tile0, const uint8_t* tile1, const uint8_t* xrow, int rg,
                                          int lane, const uint32_t* s_e4m3, uint32_t nf3_lut, float* acc0,
                                          float* acc1) {
  uint32_t a0[8], a1[8], b0[8], b1[8];
  float sa0, sa1, sb0 = 1.0f, sb1 = 1.0f;
  dequant_slot<FMT, TILE, ACT, NF3_MIX_LUT>(tile0, rg, lane, a0, a1, &sa0, &sa1, s_e4m3, nf3_lut);
  if constexpr (TWO) dequant_slot<FMT, TILE, ACT, NF3_MIX_LUT>(tile1, rg, lane, b0, b1, &sb0, &sb1, s_e4m3, nf3_lut);
  const uint4 xa = *reinterpret_cast<const uint4*>(xrow);
  const uint4 xb = *reinterpret_cast<const uint4*>(xrow + 16);
  const uint32_t xr[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
  if constexpr (FMT == FMT_NVFP4 || FMT == FMT_MXFP4 || TILE) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      mma_16816<ACT>(acc0, a0[2 * s], a1[2 * s], a0[2 * s + 1], a1[2 * s + 1], xr[2 * s], xr[2 * s + 1]);
      if constexpr (TWO)
        mma_16816<ACT>(acc1, b0[2 * s], b1[2 * s], b0[2 * s + 1], b1[2 * s + 1], xr[2 * s], xr[2 * s + 1]);
    }
  } else {
    float d[4], e[4];
    mma_16816_zc<ACT>(d, a0[0], a1[0], a0[1], a1[1], xr[0], xr[1]);
    if constexpr (TWO) mma_16816_zc<ACT>(e, b0[0], b1[0], b0[1], b1[1], xr[0], xr[1]);
#pragma unroll
    for (int s = 1; s < 4; ++s) {
      mma_16816<ACT>(d, a0[2 * s], a1[2 * s], a0[2 * s + 1], a1[2 * s + 1], xr[2 * s], xr[2 * s + 1]);
      if constexpr (TWO)
        mma_16816<ACT>(e, b0[2 * s], b1[2 * s], b0[2 * s + 1], b1[2 * s + 1], xr[2 * s], xr[2 * s + 1]);
    }
    acc0[0] = fmaf(sa0, d[0], acc0[0]);
    acc0[1] = fmaf(sa0, d[1], acc0[1]);
    acc0[2] = fmaf(sa1, d[2], acc0[2]);
    acc0[3] = fmaf(sa1, d[3], acc0[3]);
    if constexpr (TWO) {
      acc1[0] = fmaf(sb0, e[0], acc1[0]);
      acc1[1] = fmaf(sb0, e[1], acc1[1]);
      acc1[2] = fmaf(sb1, e[2], acc1[2]);
      acc1[3] = fmaf(sb1, e[3], acc1[3]);
    }
  }
}

// All k-blocks of one stage: kbs tiles of row tile 0, then kbs of row tile 1.
template <int FMT, int ACT, bool TILE, bool TWO>
__device__ __forceinline__ void sk_stage(const uint8_t* sw, const uint8_t* sx, int kbs, int rg, int lane,
                                         const uint32_t* s_e4m3, uint32_t nf3_lut, float* acc0, float* acc1) {
  constexpr int TB = tile_bytes(FMT);
  if (kbs == SK_MAX_KBS) {
#pragma unroll
    for (int j = 0; j < SK_MAX_KBS; ++j)
      sk_kblock<FMT, ACT, TILE, TWO>(sw + j * TB, sw + (SK_MAX_KBS + j) * TB, sx + j * 128, rg, lane, s_e4m3, nf3_lut,
                                     acc0, acc1);
  } else {
    for (int j = 0; j < kbs; ++j)
      sk_kblock<FMT, ACT, TILE, TWO>(sw + j * TB, sw + (kbs + j) * TB, sx + j * 128, rg, lane, s_e4m3, nf3_lut, acc0,
                                     acc1);
  }
}

template <int FMT, int ACT, bool TILE>
__device__ __forceinline__ void sk_stage_any(bool two, const uint8_t* sw, const uint8_t* sx, int kbs, int rg, int lane,
                                             const uint32_t* s_e4m3, uint32_t nf3_lut, float* acc0, float* acc1) {
  if (two) sk_stage<FMT, ACT, TILE, true>(sw, sx, kbs, rg, lane, s_e4m3, nf3_lut, acc0, acc1);
  else sk_stage<FMT, ACT, TILE, false>(sw, sx, kbs, rg, lane, s_e4m3, nf3_lut, acc0, acc1);
}

// Single-tile items. One k-block of one thread slot: dequantise through dequant_slot (the
// decoder hmoe_debug_decode_operand exports; NVFP4/MXFP4 scales applied in
// the operand type from the shared lookup table, NF3 values raw with the row
// scales applied to the fp32 sum of the k-block) and 4 MMAs. With TILE (W4A4
// layers) NF3 is decoded to the tile values rne(cb * s) instead, the weights
// the definition and the tensor-core kernel use: W4A4 quantises h, so h must
// come from the same weights on both paths.
template <int FMT, int ACT, bool TILE>
__device__ __forceinline__ void sk1_kblock(const uint8_t* tile, const uint8_t* xrow, int rg, int lane,
                                          const uint32_t* s_e4m3, uint32_t nf3_lut, float* acc) {
  const uint4 xa = *reinterpret_cast<const uint4*>(xrow);
  const uint4 xb = *reinterpret_cast<const uint4*>(xrow + 16);
  const uint32_t xr[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
  uint32_t r0[8], r1[8];
  float sc0, sc1;
  dequant_slot<FMT, TILE, ACT, NF3_MIX_LUT>(tile, rg, lane, r0, r1, &sc0, &sc1, s_e4m3, nf3_lut);
  if constexpr (FMT == FMT_NVFP4 || FMT == FMT_MXFP4 || TILE) {
#pragma unroll
    for (int s = 0; s < 4; ++s)
      mma_16816<ACT>(acc, r0[2 * s], r1[2 * s], r0[2 * s + 1], r1[2 * s + 1], xr[2 * s], xr[2 * s + 1]);
  } else {
    float d[4];
    mma_16816_zc<ACT>(d, r0[0], r1[0], r0[1], r1[1], xr[0], xr[1]);
#pragma unroll
    for (int s = 1; s < 4; ++s)
      mma_16816<ACT>(d, r0[2 * s], r1[2 * s], r0[2 * s + 1], r1[2 * s + 1], xr[2 * s], xr[2 * s + 1]);
    acc[0] = fmaf(sc0, d[0], acc[0]);
    acc[1] = fmaf(sc0, d[1], acc[1]);
    acc[2] = fmaf(sc1, d[2], acc[2]);
    acc[3] = fmaf(sc1, d[3], acc[3]);
  }
}

// Two consecutive k-blocks of one thread slot: both slots decoded before
// either k-block's MMAs, so the warp has two independent decode chains to
// interleave (k-block j into accA, j + 1 into accB).
template <int FMT, int ACT, bool TILE>
__device__ __forceinline__ void sk1_kblock2(const uint8_t* tile, const uint8_t* xrow, int rg, int lane,
                                           const uint32_t* s_e4m3, uint32_t nf3_lut, float* accA, float* accB) {
  constexpr int TB = tile_bytes(FMT);
  uint32_t a0[8], a1[8], b0[8], b1[8];
  float sa0, sa1, sb0, sb1;
  dequant_slot<FMT, TILE, ACT, NF3_MIX_LUT>(tile, rg, lane, a0, a1, &sa0, &sa1, s_e4m3, nf3_lut);
  dequant_slot<FMT, TILE, ACT, NF3_MIX_LUT>(tile + TB, rg, lane, b0, b1, &sb0, &sb1, s_e4m3, nf3_lut);
  const uint4 xa = *reinterpret_cast<const uint4*>(xrow);
  const uint4 xb = *reinterpret_cast<const uint4*>(xrow + 16);
  const uint4 ya = *reinterpret_cast<const uint4*>(xrow + 128);
  const uint4 yb = *reinterpret_cast<const uint4*>(xrow + 144);
  const uint32_t xr[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
  const uint32_t yr[8] = {ya.x, ya.y, ya.z, ya.w, yb.x, yb.y, yb.z, yb.w};
  if constexpr (FMT == FMT_NVFP4 || FMT == FMT_MXFP4 || TILE) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      mma_16816<ACT>(accA, a0[2 * s], a1[2 * s], a0[2 * s + 1], a1[2 * s + 1], xr[2 * s], xr[2 * s + 1]);
      mma_16816<ACT>(accB, b0[2 * s], b1[2 * s], b0[2 * s + 1], b1[2 * s + 1], yr[2 * s], yr[2 * s + 1]);
    }
  } else {
    float d[4], e[4];
    mma_16816_zc<ACT>(d, a0[0], a1[0], a0[1], a1[1], xr[0], xr[1]);
    mma_16816_zc<ACT>(e, b0[0], b1[0], b0[1], b1[1], yr[0], yr[1]);
#pragma unroll
    for (int s = 1; s < 4; ++s) {
      mma_16816<ACT>(d, a0[2 * s], a1[2 * s], a0[2 * s + 1], a1[2 * s + 1], xr[2 * s], xr[2 * s + 1]);
      mma_16816<ACT>(e, b0[2 * s], b1[2 * s], b0[2 * s + 1], b1[2 * s + 1], yr[2 * s], yr[2 * s + 1]);
    }
    accA[0] = fmaf(sa0, d[0], accA[0]);
    accA[1] = fmaf(sa0, d[1], accA[1]);
    accA[2] = fmaf(sa1, d[2], accA[2]);
    accA[3] = fmaf(sa1, d[3], accA[3]);
    accB[0] = fmaf(sb0, e[0], accB[0]);
    accB[1] = fmaf(sb0, e[1], accB[1]);
    accB[2] = fmaf(sb1, e[2], accB[2]);
    accB[3] = fmaf(sb1, e[3], accB[3]);
  }
}

// All k-blocks of one stage, two accumulator sets to break the MMA chain.
template <int FMT, int ACT, bool TILE>
__device__ __forceinline__ void sk1_stage(const uint8_t* sw, const uint8_t* sx, int kbs, int rg, int lane,
                                         const uint32_t* s_e4m3, uint32_t nf3_lut, float* accA, float* accB) {
  constexpr int TB = tile_bytes(FMT);
  if (kbs == 2 * SK_MAX_KBS) {
#pragma unroll
    for (int j = 0; j < 2 * SK_MAX_KBS; j += 2)
      sk1_kblock2<FMT, ACT, TILE>(sw + j * TB, sx + j * 128, rg, lane, s_e4m3, nf3_lut, accA, accB);
  } else if (kbs == 4) {
    sk1_kblock2<FMT, ACT, TILE>(sw, sx, rg, lane, s_e4m3, nf3_lut, accA, accB);
    sk1_kblock2<FMT, ACT, TILE>(sw + 2 * TB, sx + 256, rg, lane, s_e4m3, nf3_lut, accA, accB);
  } else {
    for (int j = 0; j < kbs; ++j) sk1_kblock<FMT, ACT, TILE>(sw + j * TB, sx + j * 128, rg, lane, s_e4m3, nf3_lut, (j & 1) ? accB : accA);
  }
}

template <int ACT, bool TILE>
__global__ void __launch_bounds__(SK_THREADS, SK_CTAS_PER_SM) stream_gemm_kernel(const __grid_constant__ StreamParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SK_SMEM_DATA);
  uint64_t* empty = full + SK_STAGES;
  int* s_gstart = reinterpret_cast<int*>(empty + SK_STAGES);
  int* s_off = s_gstart + MAX_E + 1;             // the caller's offsets, copied once
  volatile int* s_flags = s_off + MAX_E + 1;     // [0] abort
  uint32_t* s_e4m3 = reinterpret_cast<uint32_t*>(const_cast<int*>(s_flags) + 4);  // E4M3 -> operand-type pair
  uint32_t* s_nf3 = s_e4m3 + 256;                                                // NF3 pair table
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t lim = p.wait_limit_ns;

  if (tid == 0) {
    for (int s = 0; s < SK_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], SK_CONSUMER_WARPS);
    }
    fence_mbar_init();
    s_flags[0] = 0;
  }
  if (tid < 256) s_e4m3[tid] = e4m3_lut_entry<ACT>((uint32_t)tid);
  nf3_lut_fill<ACT>(s_nf3, tid, blockDim.x);
  // Which experts this launch's tier selection covers, from the parameter
  // table, before the wait on the routing kernel (the prefix below reads it
  // from shared memory instead of indexing the parameter table per lane).
  for (int e = tid; e < p.E; e += blockDim.x) {
    const bool nf3 = (p.tab.loc[e] & LOC_NF3) != 0;
    s_gstart[e] = (nf3 ? (p.tier_mask & 2) : (p.tier_mask & 1)) ? 1 : 0;
  }
  pdl_wait();  // everything below reads or writes global memory
  pdl_trigger();
  for (int e = tid; e <= p.E; e += blockDim.x) s_off[e] = p.offsets[e];
  __syncthreads();
  // Group prefix over experts of the selected tiers, from the caller's offsets.
  if (warp == SK_WARP_PRODUCER) {
    const int S = p.T * p.topk;
    bool bad = (s_off[0] != 0) || (s_off[p.E] != S);
    int run = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      int ng = 0;
      if (e < p.E) {
        const int ne = s_off[e + 1] - s_off[e];
        if (ne < 0) bad = true;
        const bool sel = s_gstart[e] != 0;
        ng = (sel && ne > 0) ? (ne + p.group_tokens - 1) / p.group_tokens : 0;
      }
      int incl = ng;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int nb = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += nb;
      }
      if (e < p.E) s_gstart[e] = run + incl - ng;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      s_gstart[p.E] = bad ? 0 : run;
      if (bad && blockIdx.x == 0) set_status(p.status, DEV_BAD_ROUTE);
    }
    if (bad)
      for (int e = lane; e < p.E; e += 32) s_gstart[e] = 0;
  }
  __syncthreads();

  const int n_groups = s_gstart[p.E];
  const bool pair = p.pair_items != 0;
  int units = 0;
  for (int f = p.ph_begin; f < p.ph_end; ++f) units += phase_units(p.ph[f], pair);
  const int n_items = n_groups * units;
  const bool fused = p.ph_begin == 0 && p.ph_end == 2;

  if (warp == SK_WARP_PRODUCER) {
    // ------------------------------------------------ producer: dynamic work queue
    // With the test hook set the producer stays silent, so the consumers'
    // bounded waits run out and report DEV_TIMEOUT.
    // The whole warp runs the loop (converged), so that each bulk copy issues
    // as one warp instruction: one elected lane copies the weight tiles and
    // lane j the activation row of token j, all in the same instruction.
    if (!p.debug_no_copies) {
      const uint64_t pol = l2_policy_evict_first();
      const int S = p.T * p.topk;
      int slot = 0;
      uint32_t ph = 0;
      int issued = 0;
      bool aborted = false;
      while (!aborted) {
        int i = 0;
        if (lane == 0) i = atomicAdd(p.queue, 1);
        i = __shfl_sync(0xffffffffu, i, 0);
        if (i >= n_items) break;
        const SkItem it = decode_item(p, s_gstart, s_off, i, pair);
        const StreamPhase& P = p.ph[it.ph];
        const int fmt = expert_fmt(p, it.e);
        const size_t tb = (size_t)tile_bytes(fmt);
        const uint8_t* base = (fmt == FMT_NF3 ? p.nf3_buf : p.kept_buf) +
                              (size_t)(p.tab.loc[it.e] & 0x7FFF) *
                                  (fmt == FMT_NF3 ? p.nf3_expert_bytes : p.kept_expert_bytes) +
                              (fmt == FMT_NF3 ? P.nf3_off : P.kept_off);
        // Lane j < n: the activation row of the item's token j.
        int my_row = 0;
        if (lane < it.n) {
          if (it.ph == 0) {
            int s = p.perm[it.p0 + lane];
            if (s < 0 || s >= S) {
              set_status(p.status, DEV_BAD_ROUTE);
              s = 0;
            }
            my_row = s / p.topk;
          } else {
            my_row = it.p0 + lane;
          }
        }
        if (fused && it.ph == 1) {
          // The group's h rows come from its W13 items (any CTA): wait until
          // all of them are written, then order the bulk copies after.
          bool ok = true;
          if (lane == 0)
            ok = wait_count_at_least(p.done13 + it.grp, SK_CONSUMER_WARPS * phase_units(p.ph[0], pair), s_flags, lim);
          if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
            aborted = true;
            if (lane == 0) {
              s_flags[0] = 1;
              set_status(p.status, DEV_TIMEOUT);
            }
            break;
          }
          fence_proxy_async_global();
        }
        const int kbs = pair ? P.kbs : P.kbs1;
        const int nst = P.KB / kbs;
        for (int st = 0; st < nst; ++st) {
          if (!__all_sync(0xffffffffu, mbar_wait(&empty[slot], ph ^ 1u, s_flags, lim))) {
            aborted = true;
            if (lane == 0) {
              s_flags[0] = 1;
              set_status(p.status, DEV_TIMEOUT);
            }
            break;
          }
          const int kbA = st * kbs;
          const uint32_t wbytes = (uint32_t)(kbs * tb);
          const uint32_t xbytes = (uint32_t)(kbs * 128);
          uint8_t* sw = smem + slot * SK_STAGE_BYTES;
          uint8_t* sx = sw + SK_W_BYTES;
          if (lane == 0) {
            int* hdr = reinterpret_cast<int*>(sx + SK_X_BYTES);
            hdr[0] = i;
            hdr[1] = st;
          }
          __syncwarp();
          // Pair items: row tile 2 rt's k-blocks, then row tile 2 rt + 1's,
          // each one contiguous range of the tile layout. Single: row tile rt.
          const uint8_t* src0 = base + ((size_t)(pair ? 2 * it.rt : it.rt) * P.KB + kbA) * tb;
          bulk_expect_and_copy2_elect(sw, src0, sw + wbytes, src0 + (size_t)P.KB * tb, wbytes, it.two,
                                      (it.two ? 2u : 1u) * wbytes + (uint32_t)it.n * xbytes, &full[slot], pol);
          bulk_g2s_if(lane < it.n, sx + lane * SK_XROW, P.act + (size_t)my_row * P.act_stride + (size_t)kbA * 64,
                      xbytes, &full[slot]);
          ++issued;
          if (++slot == SK_STAGES) {
            slot = 0;
            ph ^= 1u;
          }
        }
      }
      if (lane == 0) {
        if (!aborted) {
          // Terminator stage: item -1, no bytes.
          if (mbar_wait(&empty[slot], ph ^ 1u, s_flags, lim)) {
            int* hdr = reinterpret_cast<int*>(smem + slot * SK_STAGE_BYTES + SK_W_BYTES + SK_X_BYTES);
            hdr[0] = -1;
            mbar_arrive(&full[slot]);
          } else {
            aborted = true;
            s_flags[0] = 1;
            set_status(p.status, DEV_TIMEOUT);
          }
        }
        if (aborted) {
          // Drain copies still in flight before the CTA may exit (bounded).
          volatile int never = 0;
          for (int b = 0; b < SK_STAGES && b < issued; ++b) {
            if (--slot < 0) {
              slot = SK_STAGES - 1;
              ph ^= 1u;
            }
            mbar_wait(&full[slot], ph, &never, lim);
          }
          s_flags[0] = 1;
        }
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------ consumers
    const int rg = warp, g = lane >> 2, q = lane & 3;
    const uint32_t nf3_lut = smem_u32(s_nf3) + 4u * (uint32_t)lane;
    int slot = 0;
    uint32_t ph = 0;
    SkItem it{};
    int fmt = FMT_NF3, kbs = 1, nst = 1;
    float acc0[4], acc1[4];
    while (true) {
      if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], ph, s_flags, lim))) {
        if (lane == 0) {
          s_flags[0] = 1;
          set_status(p.status, DEV_TIMEOUT);
        }
        break;
      }
      const uint8_t* sw = smem + slot * SK_STAGE_BYTES;
      const int* hdr = reinterpret_cast<const int*>(sw + SK_W_BYTES + SK_X_BYTES);
      const int i = hdr[0], st = hdr[1];
      if (i < 0) break;
      if (st == 0) {
        it = decode_item(p, s_gstart, s_off, i, pair);
        fmt = expert_fmt(p, it.e);
        kbs = pair ? p.ph[it.ph].kbs : p.ph[it.ph].kbs1;
        nst = p.ph[it.ph].KB / kbs;
#pragma unroll
        for (int r = 0; r < 4; ++r) acc0[r] = acc1[r] = 0.f;
      }
      const uint8_t* sx = sw + SK_W_BYTES + g * SK_XROW + q * 32;
      if (pair) {
        if (fmt == FMT_NVFP4)
          sk_stage_any<FMT_NVFP4, ACT, TILE>(it.two, sw, sx, kbs, rg, lane, s_e4m3, nf3_lut, acc0, acc1);
        else if (fmt == FMT_MXFP4)
          sk_stage_any<FMT_MXFP4, ACT, TILE>(it.two, sw, sx, kbs, rg, lane, s_e4m3, nf3_lut, acc0, acc1);
        else sk_stage_any<FMT_NF3, ACT, TILE>(it.two, sw, sx, kbs, rg, lane, s_e4m3, nf3_lut, acc0, acc1);
      } else {
        if (fmt == FMT_NVFP4) sk1_stage<FMT_NVFP4, ACT, TILE>(sw, sx, kbs, rg, lane, s_e4m3, nf3_lut, acc0, acc1);
        else if (fmt == FMT_MXFP4) sk1_stage<FMT_MXFP4, ACT, TILE>(sw, sx, kbs, rg, lane, s_e4m3, nf3_lut, acc0, acc1);
        else sk1_stage<FMT_NF3, ACT, TILE>(sw, sx, kbs, rg, lane, s_e4m3, nf3_lut, acc0, acc1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (++slot == SK_STAGES) {
        slot = 0;
        ph ^= 1u;
      }
      if (st != nst - 1) continue;
      // ---------------- item epilogue
      if (pair) {
        sk_emit<ACT>(p, it, 2 * it.rt, rg, g, q, acc0);
        if (it.two) sk_emit<ACT>(p, it, 2 * it.rt + 1, rg, g, q, acc1);
      } else {
        // single-tile items: acc0 and acc1 hold alternate k-blocks
#pragma unroll
        for (int r = 0; r < 4; ++r) acc0[r] += acc1[r];
        sk_emit<ACT>(p, it, it.rt, rg, g, q, acc0);
      }
      if (fused && it.ph == 0) {
        // Publish this warp's h rows to the W2 producers, whose bulk copies
        // (async proxy) may run on any SM: every lane fences its own stores
        // (proxy, then gpu scope), the warp synchronises, and lane 0 fences
        // again before one count per warp.
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          atomicAdd(p.done13 + it.grp, 1);
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    // The last CTA to leave resets the work queue and the group counters
    // for the next launch.
    if (atomicAdd(p.queue + 1, 1) == (int)gridDim.x - 1) {
      if (fused)
        for (int g = 0; g < n_groups; ++g) p.done13[g] = 0;
      p.queue[0] = 0;
      p.queue[1] = 0;
      __threadfence();
    }
  }
}

int stream_grid(int num_sms) { return SK_CTAS_PER_SM * num_sms; }

cudaError_t launch_stream_gemm(const StreamParams& p, int grid, cudaStream_t st) {
  static std::atomic<unsigned long long> attr[4] = {};
  cudaError_t ea = ensure_smem_attr(stream_gemm_kernel<ACT_BF16, false>, SK_SMEM_BYTES, attr[0]);
  if (ea == cudaSuccess) ea = ensure_smem_attr(stream_gemm_kernel<ACT_F16, false>, SK_SMEM_BYTES, attr[1]);
  if (ea == cudaSuccess) ea = ensure_smem_attr(stream_gemm_kernel<ACT_BF16, true>, SK_SMEM_BYTES, attr[2]);
  if (ea == cudaSuccess) ea = ensure_smem_attr(stream_gemm_kernel<ACT_F16, true>, SK_SMEM_BYTES, attr[3]);
  if (ea != cudaSuccess) return ea;
  if (p.act_type != ACT_BF16 && p.act_type != ACT_F16) return cudaErrorInvalidValue;
  if (p.ph_begin < 0 || p.ph_begin >= p.ph_end || p.ph_end > 2) return cudaErrorInvalidValue;
  if (p.ph_begin == 0 && p.ph_end == 2 && !p.done13) return cudaErrorInvalidValue;
  for (const StreamPhase& P : p.ph)
    if (P.kbs < 1 || P.kbs > SK_MAX_KBS || P.KB % P.kbs != 0 || P.kbs1 < 1 || P.kbs1 > 2 * SK_MAX_KBS ||
        P.KB % P.kbs1 != 0)
      return cudaErrorInvalidValue;
  if (p.group_tokens < 1 || p.group_tokens > 8) return cudaErrorInvalidValue;
  auto kern = p.act_type == ACT_F16 ? (p.nf3_tile ? stream_gemm_kernel<ACT_F16, true> : stream_gemm_kernel<ACT_F16, false>)
                                    : (p.nf3_tile ? stream_gemm_kernel<ACT_BF16, true> : stream_gemm_kernel<ACT_BF16, false>);
  cudaError_t e = launch_pdl(kern, dim3(grid), dim3(SK_THREADS), SK_SMEM_BYTES, st, p);
  count_launches(1);
  return e;
}

// ------------------------------------------------------------ finalize
// out[t][c] = act(sum_j gates[t*k+j] * y[t*k+j][c]) in slot order: blocks
// along x cover a row's column pairs, along y the tokens (grid-stride in
// both), so no index needs a division.
template <int ACT>
__global__ void finalize_kernel(const float* __restrict__ y, const float* __restrict__ gates, int T, int k, int H,
                                uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int half = H / 2;
  for (int t = blockIdx.y; t < T; t += gridDim.y) {
    const float* yt = y + (size_t)t * k * H;
    const float* gt = gates + (size_t)t * k;
    for (int c2 = blockIdx.x * blockDim.x + threadIdx.x; c2 < half; c2 += gridDim.x * blockDim.x) {
      float a = 0.f, b = 0.f;
      for (int j = 0; j < k; ++j) {
        const float g = gt[j];
        const float2 v = *reinterpret_cast<const float2*>(yt + (size_t)j * H + 2 * c2);
        a = fmaf(g, v.x, a);
        b = fmaf(g, v.y, b);
      }
      *reinterpret_cast<uint32_t*>(out + (size_t)t * H + 2 * c2) = f32x2_to_act<ACT>(a, b);
    }
  }
}

cudaError_t launch_finalize(const float* y, const float* gates, int T, int k, int H, uint16_t* out, int act_type,
                            cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int threads = 256;
  const int gx = (H / 2 + threads - 1) / threads;
  const int gy = T < 65535 ? T : 65535;
  const dim3 grid((unsigned)gx, (unsigned)gy);
  cudaError_t e = act_type == ACT_F16
                      ? launch_pdl(finalize_kernel<ACT_F16>, grid, dim3(threads), 0, st, y, gates, T, k, H, out)
                      : launch_pdl(finalize_kernel<ACT_BF16>, grid, dim3(threads), 0, st, y, gates, T, k, H, out);
  count_launches(1);
  return e;
}

}  // namespace hmoe
