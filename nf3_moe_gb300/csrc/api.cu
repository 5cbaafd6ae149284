// api.cu -- the C ABI of libhmoe (include/hmoe.h): validation, handle, workspace, launch order.
//
// Cites: "quant: nvfp4_nf3_hybrid -- native serving for mixed NVFP4+NF3 MoE
// checkpoints", How it works (two prepared weight objects per layer;
// preplanned, CUDA-graph-safe launches sharing one route geometry and one
// topk_sum; no environment variables; scratch sized from the maximum batched
// token count). "quant: add native mixed NVFP4/MXFP4 plus NF3 MoE serving",
// Summary (hybrid_bit_map 4 = kept, 3 = NF3; kept_format; the metadata is
// validated).
#include <algorithm>
#include <climits>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "../../include/hmoe.h"
#include "common.cuh"
#include "internal.h"

using namespace hmoe;

namespace hmoe {
static std::atomic<unsigned long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }
}  // namespace hmoe

struct hmoe_layer {
  hmoe_layer_desc d;
  uint8_t* kept_buf;
  uint8_t* nf3_buf;
  int n_kept, n_nf3;
  ExpertGeom gk, gn;
  ExpertTable tab;
  int num_sms;
};

namespace {

thread_local std::string g_err;

// An NVTX range over one library call, so that profilers (ncu --nvtx,
// Nsight Systems) label the launches it makes. With no tool attached a
// range costs a few nanoseconds and reads nothing from the environment but
// the profiler's own injection hook.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

hmoe_status fail(hmoe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

hmoe_status cuda_fail(cudaError_t e, const char* what) {
  return fail(HMOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

hmoe_status check_desc(const hmoe_layer_desc* d) {
  if (!d) return fail(HMOE_ERR_INVALID_ARG, "desc is NULL");
  if (d->kept_format != HMOE_FMT_NVFP4 && d->kept_format != HMOE_FMT_MXFP4)
    return fail(HMOE_ERR_INVALID_ARG, "kept_format must be NVFP4 (4) or MXFP4 (5), got %d", d->kept_format);
  if (d->H <= 0 || d->I <= 0 || d->E <= 0 || d->topk <= 0)
    return fail(HMOE_ERR_INVALID_ARG, "H, I, E, topk must be positive");
  if (d->H % 128 != 0 || d->I % 64 != 0)
    return fail(HMOE_ERR_UNSUPPORTED_SHAPE, "H must be a multiple of 128 and I of 64 (H=%d I=%d)", d->H, d->I);
  if (d->E > MAX_E) return fail(HMOE_ERR_UNSUPPORTED_SHAPE, "E=%d exceeds %d", d->E, MAX_E);
  if (d->topk > MAX_TOPK || d->topk > d->E)
    return fail(HMOE_ERR_UNSUPPORTED_SHAPE, "topk=%d must be <= min(E, %d)", d->topk, MAX_TOPK);
  if (d->act_dtype != HMOE_ACT_BF16 && d->act_dtype != HMOE_ACT_F16)
    return fail(HMOE_ERR_INVALID_ARG, "act_dtype must be HMOE_ACT_BF16 (0) or HMOE_ACT_F16 (1), got %d", d->act_dtype);
  if (d->act_quant != HMOE_ACT_QUANT_NONE && d->act_quant != HMOE_ACT_QUANT_NVFP4)
    return fail(HMOE_ERR_INVALID_ARG, "act_quant must be HMOE_ACT_QUANT_NONE (0) or HMOE_ACT_QUANT_NVFP4 (1), got %d",
                d->act_quant);
  if (d->act_quant == HMOE_ACT_QUANT_NVFP4 &&
      !(d->act_global13 > 0.0f && d->act_global13 < 3.0e38f && d->act_global2 > 0.0f && d->act_global2 < 3.0e38f))
    return fail(HMOE_ERR_INVALID_ARG, "W4A4 needs finite positive activation global scales (got %g, %g)",
                (double)d->act_global13, (double)d->act_global2);
  return HMOE_OK;
}

hmoe_status check_bitmap(const hmoe_layer_desc* d, const int8_t* bit_map) {
  if (!bit_map) return HMOE_OK;
  for (int e = 0; e < d->E; ++e)
    if (bit_map[e] != 3 && bit_map[e] != 4)
      return fail(HMOE_ERR_BAD_BITMAP, "bit_map[%d] = %d; entries must be 4 (kept) or 3 (NF3)", e, bit_map[e]);
  return HMOE_OK;
}

// The largest power of two up to max_kbs that divides the k-block count.
int pick_stage(int kbi, int max_kbs = STREAM_MAX_KBS) {
  for (int s = max_kbs; s > 1; s >>= 1)
    if (kbi % s == 0) return s;
  return 1;
}

constexpr int DECODE_MAX_T = 8;
// The automatic path streams weights (stream.cu) while the batch routes at
// most this many slots per expert on average, T * topk <= 8 * E, and uses the
// tensor-core grouped kernel above. The streaming kernel reads each touched
// expert once per group of 8 of its tokens, so its cost grows with the slots
// per expert; the grouped kernel costs about the same per k-block whatever
// its token count. Measured crossover (uniform routing, L2 flushed): at 8
// slots per expert streaming wins (256 experts, H=6144, I=2048, T=256: 1.69
// against 1.89 ms; 128 experts, H=2048, I=768, T=128: 146 against 164 us), at
// 12 to 16 the grouped kernel wins (T=384: 1.90 against 2.31 ms).
constexpr int STREAM_MAX_SLOTS_PER_EXPERT = 8;
// Token groups the fixed counter array holds. A stream-path forward whose
// group bound exceeds it runs W13 and W2 as two launches instead of one.
constexpr int STREAM_FUSED_MAX_GROUPS = 1024;

struct WsLayout {
  size_t status, queues, done13, chunk_cnt, chunk_base, xq, xg, h, y, total;
};

// Fixed prefix (status word, work queues) first, so that it stays at the
// same place for every T.
WsLayout ws_layout(const hmoe_layer_desc& d, int T) {
  WsLayout w{};
  size_t off = 0;
  w.status = off;
  off += 256;
  w.queues = off;                       // 4 launch slots x {head, finished}
  off += 256;
  w.done13 = off;                       // per-group W13 completion counts (fused stream launch)
  off += align256((size_t)STREAM_FUSED_MAX_GROUPS * 4);
  // T-dependent regions from here on.
  const size_t nch = (size_t)route_chunks(T);
  w.chunk_cnt = off;
  off += align256(nch * d.E * 4);
  w.chunk_base = off;
  off += align256(nch * d.E * 4);
  const size_t S = (size_t)T * d.topk;
  w.xq = off;                           // W4A4: the quantised layer input [T][H]
  off += align256(d.act_quant ? (size_t)T * d.H * 2 : 0);
  w.xg = off;
  off += align256(T > DECODE_MAX_T ? S * d.H * 2 : 0);
  w.h = off;
  off += align256(S * d.I * 2);
  w.y = off;
  off += align256(S * d.H * 4);
  w.total = off;
  return w;
}

hmoe_status check_ws(const hmoe_layer_desc& d, int T, void* ws, size_t ws_bytes, WsLayout* out) {
  if (!ws) return fail(HMOE_ERR_INVALID_ARG, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return fail(HMOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  *out = ws_layout(d, T);
  if (ws_bytes < out->total)
    return fail(HMOE_ERR_WORKSPACE_TOO_SMALL, "workspace holds %zu bytes, T=%d needs %zu", ws_bytes, T, out->total);
  return HMOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// The kernels index slots (s = t * topk + j) with 32-bit ints, so a batch
// may hold at most INT_MAX slots.
hmoe_status check_slots(const hmoe_layer_desc& d, int T) {
  const long long S = (long long)T * d.topk;
  if (S > (long long)INT_MAX)
    return fail(HMOE_ERR_UNSUPPORTED_SHAPE, "T*topk = %lld slots exceed the 32-bit slot index", S);
  return HMOE_OK;
}

}  // namespace

extern "C" {

int hmoe_version(void) { return 100; }

uint64_t hmoe_launch_count(void) { return (uint64_t)hmoe::g_launches.load(std::memory_order_relaxed); }

const char* hmoe_last_error(void) { return g_err.c_str(); }

hmoe_status hmoe_packed_size(const hmoe_layer_desc* desc, const int8_t* bit_map, size_t* kept_bytes,
                             size_t* nf3_bytes) {
  hmoe_status s = check_desc(desc);
  if (s != HMOE_OK) return s;
  if (!kept_bytes || !nf3_bytes) return fail(HMOE_ERR_INVALID_ARG, "output pointers are NULL");
  if ((s = check_bitmap(desc, bit_map)) != HMOE_OK) return s;
  int nk = 0, nn = 0;
  for (int e = 0; e < desc->E; ++e) {
    if (!bit_map || bit_map[e] == 4) ++nk; else ++nn;
  }
  *kept_bytes = (size_t)nk * expert_geom(desc->H, desc->I, desc->kept_format).expert_bytes;
  *nf3_bytes = (size_t)nn * expert_geom(desc->H, desc->I, FMT_NF3).expert_bytes;
  return HMOE_OK;
}

hmoe_status hmoe_workspace_size(const hmoe_layer_desc* desc, int max_tokens, size_t* bytes) {
  hmoe_status s = check_desc(desc);
  if (s != HMOE_OK) return s;
  if (!bytes || max_tokens < 0) return fail(HMOE_ERR_INVALID_ARG, "bytes NULL or max_tokens < 0");
  if ((s = check_slots(*desc, max_tokens)) != HMOE_OK) return s;
  // Every T <= max_tokens must fit (the layout grows with T; the loop keeps
  // that true however the layout changes).
  size_t need = ws_layout(*desc, max_tokens).total;
  for (int t = 0; t <= max_tokens && t <= DECODE_MAX_T; ++t) {
    const size_t n = ws_layout(*desc, t).total;
    if (n > need) need = n;
  }
  *bytes = need;
  return HMOE_OK;
}

static bool auto_is_grouped(const hmoe_layer_desc& d, int T) {
  return (long long)T * d.topk > (long long)STREAM_MAX_SLOTS_PER_EXPERT * d.E;
}

hmoe_status hmoe_auto_path(const hmoe_layer_desc* desc, int T, int* path) {
  hmoe_status s = check_desc(desc);
  if (s != HMOE_OK) return s;
  if (!path || T < 0) return fail(HMOE_ERR_INVALID_ARG, "path NULL or T < 0");
  *path = auto_is_grouped(*desc, T) ? HMOE_PATH_GROUPED : HMOE_PATH_STREAM;
  return HMOE_OK;
}

hmoe_status hmoe_workspace_init(void* ws, size_t ws_bytes, hmoe_stream_t stream) {
  if (!ws) return fail(HMOE_ERR_INVALID_ARG, "workspace is NULL");
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace)");
  return HMOE_OK;
}

hmoe_status hmoe_pack_weights(const hmoe_layer_desc* desc, const int8_t* bit_map, const hmoe_expert_src* src,
                              void* kept_buf, void* nf3_buf, hmoe_stream_t stream, hmoe_layer** out) {
  const NvtxRange nvtx("hmoe_pack_weights");
  hmoe_status s = check_desc(desc);
  if (s != HMOE_OK) return s;
  if ((s = check_bitmap(desc, bit_map)) != HMOE_OK) return s;
  if (!src || !out) return fail(HMOE_ERR_INVALID_ARG, "src or out is NULL");
  size_t kb = 0, nb = 0;
  hmoe_packed_size(desc, bit_map, &kb, &nb);
  if ((kb && !kept_buf) || (nb && !nf3_buf)) return fail(HMOE_ERR_INVALID_ARG, "a tier buffer is NULL");
  if ((kept_buf && !aligned16(kept_buf)) || (nf3_buf && !aligned16(nf3_buf)))
    return fail(HMOE_ERR_INVALID_ARG, "tier buffers must be 16-byte aligned");
  for (int e = 0; e < desc->E; ++e) {
    const hmoe_expert_src& x = src[e];
    if (!x.w13_codes || !x.w13_scales || !x.w2_codes || !x.w2_scales)
      return fail(HMOE_ERR_INVALID_ARG, "expert %d has a NULL source pointer", e);
  }
  hmoe_layer* L = new (std::nothrow) hmoe_layer();
  if (!L) return fail(HMOE_ERR_INVALID_ARG, "out of host memory");
  L->d = *desc;
  L->kept_buf = static_cast<uint8_t*>(kept_buf);
  L->nf3_buf = static_cast<uint8_t*>(nf3_buf);
  L->gk = expert_geom(desc->H, desc->I, desc->kept_format);
  L->gn = expert_geom(desc->H, desc->I, FMT_NF3);
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (ce != cudaSuccess) {
    delete L;
    return cuda_fail(ce, "device query");
  }
  int nk = 0, nn = 0;
  for (int e = 0; e < desc->E; ++e) {
    const bool kept = !bit_map || bit_map[e] == 4;
    const int fmt = kept ? desc->kept_format : FMT_NF3;
    uint8_t* dst;
    if (kept) {
      L->tab.loc[e] = (uint16_t)nk;
      dst = L->kept_buf + (size_t)nk * L->gk.expert_bytes;
      ++nk;
    } else {
      L->tab.loc[e] = (uint16_t)(nn | LOC_NF3);
      dst = L->nf3_buf + (size_t)nn * L->gn.expert_bytes;
      ++nn;
    }
    L->tab.g13[e] = fmt == FMT_NVFP4 ? src[e].w13_global : 1.0f;
    L->tab.g2[e] = fmt == FMT_NVFP4 ? src[e].w2_global : 1.0f;
    const ExpertGeom& g = kept ? L->gk : L->gn;
    const bool nibbles = desc->act_dtype == HMOE_ACT_F16;
    ce = launch_pack_matrix(fmt, 13, src[e].w13_codes, src[e].w13_scales, 2 * desc->I, desc->H, desc->I, dst,
                            nibbles, (cudaStream_t)stream);
    if (ce == cudaSuccess)
      ce = launch_pack_matrix(fmt, 2, src[e].w2_codes, src[e].w2_scales, desc->H, desc->I, desc->I,
                              dst + g.w13_bytes, nibbles, (cudaStream_t)stream);
    if (ce != cudaSuccess) {
      delete L;
      return cuda_fail(ce, "pack kernel launch");
    }
  }
  L->n_kept = nk;
  L->n_nf3 = nn;
  *out = L;
  return HMOE_OK;
}

void hmoe_layer_destroy(hmoe_layer* layer) { delete layer; }

hmoe_status hmoe_layer_expert_info(const hmoe_layer* L, int expert, int* fmt, float* g13, float* g2) {
  if (!L || expert < 0 || expert >= L->d.E) return fail(HMOE_ERR_INVALID_ARG, "bad layer or expert index");
  if (fmt) *fmt = (L->tab.loc[expert] & LOC_NF3) ? FMT_NF3 : L->d.kept_format;
  if (g13) *g13 = L->tab.g13[expert];
  if (g2) *g2 = L->tab.g2[expert];
  return HMOE_OK;
}

hmoe_status hmoe_plan_routes(const hmoe_layer* L, const float* logits, int T, int32_t* ids, float* gates,
                             int32_t* perm, int32_t* offsets, void* ws, size_t ws_bytes, hmoe_stream_t stream) {
  const NvtxRange nvtx("hmoe_plan_routes");
  if (!L) return fail(HMOE_ERR_INVALID_ARG, "layer is NULL");
  if (T < 0) return fail(HMOE_ERR_INVALID_ARG, "T=%d < 0", T);
  if (!offsets || (T > 0 && (!logits || !ids || !gates || !perm)))
    return fail(HMOE_ERR_INVALID_ARG, "a route buffer is NULL");
  hmoe_status s = check_slots(L->d, T);
  if (s != HMOE_OK) return s;
  WsLayout w{};
  if ((s = check_ws(L->d, T, ws, ws_bytes, &w)) != HMOE_OK) return s;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  cudaError_t e = launch_route(logits, T, L->d.E, L->d.topk, ids, gates, perm, offsets,
                               reinterpret_cast<int*>(wsb + w.chunk_cnt), reinterpret_cast<int*>(wsb + w.chunk_base),
                               (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "route kernel launch");
  return HMOE_OK;
}

// Records a caller's stage event. Inside a stream capture the record must
// become an event-record node (external flag); outside one, a plain record.
static cudaError_t record_stage_event(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal)
                                             : cudaEventRecord(ev, st);
}

static hmoe_status run_stream_path(const hmoe_layer* L, const void* x, int T, const float* gates,
                                   const int32_t* perm, const int32_t* offsets, void* out, uint8_t* wsb,
                                   const WsLayout& w, const hmoe_forward_opts& o, cudaStream_t st) {
  const int tier_order = o.tier_order;
  const hmoe_layer_desc& d = L->d;
  const int S = T * d.topk;
  StreamParams p{};
  p.kept_buf = L->kept_buf;
  p.nf3_buf = L->nf3_buf;
  p.kept_fmt = d.kept_format;
  p.act_type = d.act_dtype;
  const bool w4a4 = d.act_quant == HMOE_ACT_QUANT_NVFP4;
  p.act_scale13 = w4a4 ? d.act_global13 : 1.0f;
  p.act_scale2 = w4a4 ? d.act_global2 : 1.0f;
  p.nf3_tile = w4a4 ? 1 : 0;
  p.H = d.H;
  p.I = d.I;
  p.E = d.E;
  p.topk = d.topk;
  p.T = T;
  p.group_tokens = 8;
  p.kept_expert_bytes = L->gk.expert_bytes;
  p.nf3_expert_bytes = L->gn.expert_bytes;
  p.offsets = offsets;
  p.perm = perm;
  p.status = reinterpret_cast<int*>(wsb + w.status);
  p.done13 = reinterpret_cast<int*>(wsb + w.done13);
  p.h_out = reinterpret_cast<uint16_t*>(wsb + w.h);
  p.y_out = reinterpret_cast<float*>(wsb + w.y);
  p.tab = L->tab;
  p.wait_limit_ns = o.wait_limit_us > 0 ? (unsigned long long)o.wait_limit_us * 1000ull : WAIT_LIMIT_NS;
  p.debug_no_copies = (o.debug_flags & HMOE_DEBUG_NO_COPIES) ? 1 : 0;
  int masks[2] = {3, 0};
  if (tier_order == HMOE_TIERS_KEPT_FIRST) {
    masks[0] = 1;
    masks[1] = 2;
  } else if (tier_order == HMOE_TIERS_NF3_FIRST) {
    masks[0] = 2;
    masks[1] = 1;
  }
  const int grid = stream_grid(L->num_sms);
  auto mark = [&](int i) -> cudaError_t {
    if (o.stage_events && i < o.n_stage_events && o.stage_events[i])
      return record_stage_event((cudaEvent_t)o.stage_events[i], st);
    return cudaSuccess;
  };
  if (mark(0) != cudaSuccess) return cuda_fail(cudaGetLastError(), "stage event record");
  // W4A4: the layer input quantised to NVFP4 operand values (the global
  // scale goes to the W13 epilogue).
  const void* xin = x;
  if (w4a4) {
    uint16_t* xq = reinterpret_cast<uint16_t*>(wsb + w.xq);
    cudaError_t e = launch_act_quant(static_cast<const uint16_t*>(x), (long long)T * d.H, d.act_global13, d.act_dtype,
                                     xq, nullptr, nullptr, L->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "activation quantisation launch");
    xin = xq;
  }
  for (int f = 0; f < 2; ++f) {
    StreamPhase& P = p.ph[f];
    P.rows = f == 0 ? 2 * d.I : d.H;
    P.K = f == 0 ? d.H : d.I;
    P.RT = P.rows / TILE_ROWS;
    P.KB = P.K / TILE_K;
    P.kbs = pick_stage(P.KB);
    P.kbs1 = pick_stage(P.KB, 2 * STREAM_MAX_KBS);
    P.act = f == 0 ? static_cast<const uint16_t*>(xin) : p.h_out;
    P.act_stride = f == 0 ? d.H : d.I;
    P.kept_off = f == 0 ? 0 : L->gk.w13_bytes;
    P.nf3_off = f == 0 ? 0 : L->gn.w13_bytes;
  }
  {
    const long long groups = std::min<long long>(S, d.E);
    p.pair_items = groups * ((p.ph[0].RT + 1) / 2) >= (long long)STREAM_PAIR_MIN_ITEMS_PER_CTA * grid ? 1 : 0;
  }
  // Upper bound on the token groups of one launch: every slot of an expert
  // goes to one group of up to 8, so G <= min(S, ceil(S / 8) + E).
  const long long g_bound = std::min<long long>(S, (S + 7) / 8 + d.E);
  // W4A4 quantises h between the two GEMMs, so they run as two launches.
  const bool fused = g_bound <= STREAM_FUSED_MAX_GROUPS && !w4a4;
  // Fused: W13 and W2 run in one launch per tier selection, and the events
  // that follow W13 and W2 are both recorded after it.
  const int ranges[2][2] = {{0, fused ? 2 : 1}, {1, 2}};
  for (int r = 0; r < (fused ? 1 : 2); ++r) {
    p.ph_begin = ranges[r][0];
    p.ph_end = ranges[r][1];
    for (int li = 0; li < 2; ++li) {
      const int m = masks[li];
      if (!m) continue;
      p.tier_mask = m;
      p.queue = reinterpret_cast<int*>(wsb + w.queues) + 2 * (2 * r + li);
      cudaError_t e = launch_stream_gemm(p, grid, st);
      if (e != cudaSuccess) return cuda_fail(e, "stream GEMM launch");
    }
    if (r == 0 && w4a4) {
      cudaError_t eq = launch_act_quant(p.h_out, (long long)S * d.I, d.act_global2, d.act_dtype, p.h_out, nullptr,
                                        nullptr, L->num_sms, st);
      if (eq != cudaSuccess) return cuda_fail(eq, "activation quantisation launch");
    }
    cudaError_t e = mark(fused || r == 0 ? 1 : 2);
    if (e == cudaSuccess && fused) e = mark(2);
    if (e != cudaSuccess) return cuda_fail(e, "stage event record");
  }
  cudaError_t e = launch_finalize(p.y_out, gates, T, d.topk, d.H, static_cast<uint16_t*>(out), d.act_dtype, st);
  if (e != cudaSuccess) return cuda_fail(e, "finalize launch");
  if ((e = mark(3)) != cudaSuccess) return cuda_fail(e, "stage event record");
  return HMOE_OK;
}

static hmoe_status run_grouped_path(const hmoe_layer* L, const void* x, int T, const float* gates,
                                    const int32_t* perm, const int32_t* offsets, void* out, uint8_t* wsb,
                                    const WsLayout& w, const hmoe_forward_opts& o, cudaStream_t st) {
  const hmoe_layer_desc& d = L->d;
  const int S = T * d.topk;
  GroupedParams p{};
  p.kept_buf = L->kept_buf;
  p.nf3_buf = L->nf3_buf;
  p.kept_fmt = d.kept_format;
  p.act_type = d.act_dtype;
  const bool w4a4 = d.act_quant == HMOE_ACT_QUANT_NVFP4;
  p.H = d.H;
  p.I = d.I;
  p.E = d.E;
  p.topk = d.topk;
  p.T = T;
  p.kept_expert_bytes = L->gk.expert_bytes;
  p.nf3_expert_bytes = L->gn.expert_bytes;
  p.kept_w2_off = L->gk.w13_bytes;
  p.nf3_w2_off = L->gn.w13_bytes;
  p.offsets = offsets;
  p.perm = perm;
  p.status = reinterpret_cast<int*>(wsb + w.status);
  p.h_out = reinterpret_cast<uint16_t*>(wsb + w.h);
  p.y_out = reinterpret_cast<float*>(wsb + w.y);
  p.wait_limit_ns = o.wait_limit_us > 0 ? (unsigned long long)o.wait_limit_us * 1000ull : WAIT_LIMIT_NS;
  p.pair = (o.debug_flags & HMOE_DEBUG_GROUPED_PAIR) ? 1 : 0;
  p.tab = L->tab;
  uint16_t* xg = reinterpret_cast<uint16_t*>(wsb + w.xg);
  auto mark = [&](int i) -> cudaError_t {
    if (o.stage_events && i < o.n_stage_events && o.stage_events[i])
      return record_stage_event((cudaEvent_t)o.stage_events[i], st);
    return cudaSuccess;
  };
  int masks[2] = {3, 0};
  if (o.tier_order == HMOE_TIERS_KEPT_FIRST) {
    masks[0] = 1;
    masks[1] = 2;
  } else if (o.tier_order == HMOE_TIERS_NF3_FIRST) {
    masks[0] = 2;
    masks[1] = 1;
  }
  // W4A4: the layer input quantised to NVFP4 operand values first (the
  // global scale goes to the W13 epilogue).
  const uint16_t* xin = static_cast<const uint16_t*>(x);
  cudaError_t e = cudaSuccess;
  if (w4a4) {
    uint16_t* xq = reinterpret_cast<uint16_t*>(wsb + w.xq);
    e = launch_act_quant(xin, (long long)T * d.H, d.act_global13, d.act_dtype, xq, nullptr, nullptr, L->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "activation quantisation launch");
    xin = xq;
  }
  e = launch_gather_rows(xin, perm, S, d.topk, T, d.H, xg, p.status, L->num_sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "gather launch");
  if ((e = mark(0)) != cudaSuccess) return cuda_fail(e, "stage event record");
  for (int which : {13, 2}) {
    p.which = which;
    p.K = which == 13 ? d.H : d.I;
    p.RT = (which == 13 ? 2 * d.I : d.H) / TILE_ROWS;
    p.KB = p.K / TILE_K;
    const uint16_t* b = which == 13 ? xg : p.h_out;
    p.act_scale = !w4a4 ? 1.0f : (which == 13 ? d.act_global13 : d.act_global2);
    if (which == 2 && w4a4) {
      e = launch_act_quant(p.h_out, (long long)S * d.I, d.act_global2, d.act_dtype, p.h_out, nullptr, nullptr,
                           L->num_sms, st);
      if (e != cudaSuccess) return cuda_fail(e, "activation quantisation launch");
    }
    for (int m : masks) {
      if (!m) continue;
      p.tier_mask = m;
      e = launch_grouped_gemm(p, b, S, L->num_sms, st);
      if (e != cudaSuccess) return cuda_fail(e, "grouped GEMM launch");
    }
    if ((e = mark(which == 13 ? 1 : 2)) != cudaSuccess) return cuda_fail(e, "stage event record");
  }
  e = launch_finalize(p.y_out, gates, T, d.topk, d.H, static_cast<uint16_t*>(out), d.act_dtype, st);
  if (e != cudaSuccess) return cuda_fail(e, "finalize launch");
  if ((e = mark(3)) != cudaSuccess) return cuda_fail(e, "stage event record");
  return HMOE_OK;
}

}  // extern "C"

namespace {

// Every host-side check of a forward call except the workspace: run before
// anything is enqueued, by hmoe_forward_ex and hmoe_forward_static alike.
// *grouped receives the path the call takes.
hmoe_status check_forward(const hmoe_layer* L, const void* x, int T, const int32_t* ids, const float* gates,
                          const int32_t* perm, const int32_t* offsets, const void* out, const hmoe_forward_opts& o,
                          bool* grouped) {
  if (!L) return fail(HMOE_ERR_INVALID_ARG, "layer is NULL");
  if (T < 0) return fail(HMOE_ERR_INVALID_ARG, "T=%d < 0", T);
  if (check_slots(L->d, T) != HMOE_OK) return HMOE_ERR_UNSUPPORTED_SHAPE;
  if (o.tier_order < 0 || o.tier_order > 2) return fail(HMOE_ERR_INVALID_ARG, "bad tier_order %d", o.tier_order);
  if (o.path < 0 || o.path > 2) return fail(HMOE_ERR_INVALID_ARG, "bad path %d", o.path);
  if (o.wait_limit_us < 0) return fail(HMOE_ERR_INVALID_ARG, "wait_limit_us < 0");
  *grouped = o.path == HMOE_PATH_GROUPED || (o.path == HMOE_PATH_AUTO && auto_is_grouped(L->d, T));
  if (T == 0) return HMOE_OK;
  if (!x || !ids || !gates || !perm || !offsets || !out) return fail(HMOE_ERR_INVALID_ARG, "a buffer is NULL");
  if (!aligned16(x) || !aligned16(out)) return fail(HMOE_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
  if (*grouped && T <= DECODE_MAX_T)
    return fail(HMOE_ERR_INVALID_ARG, "the grouped path needs T > %d (the workspace holds no gather buffer below)",
                DECODE_MAX_T);
  if ((o.debug_flags & HMOE_DEBUG_GROUPED_PAIR) && L->d.act_dtype != HMOE_ACT_BF16)
    return fail(HMOE_ERR_INVALID_ARG, "the CTA-pair grouped kernel takes bf16 activations only");
  return HMOE_OK;
}

hmoe_status run_forward(const hmoe_layer* L, const void* x, int T, const float* gates, const int32_t* perm,
                        const int32_t* offsets, void* out, void* ws, const WsLayout& w, const hmoe_forward_opts& o,
                        bool grouped, cudaStream_t st) {
  if (T == 0) return HMOE_OK;
  if (grouped) return run_grouped_path(L, x, T, gates, perm, offsets, out, static_cast<uint8_t*>(ws), w, o, st);
  return run_stream_path(L, x, T, gates, perm, offsets, out, static_cast<uint8_t*>(ws), w, o, st);
}

const hmoe_forward_opts kDefaultOpts{HMOE_TIERS_ONE_LAUNCH, HMOE_PATH_AUTO, 0, 0, nullptr, 0};

}  // namespace

extern "C" {

hmoe_status hmoe_forward_ex(const hmoe_layer* L, const void* x, int T, const int32_t* ids, const float* gates,
                            const int32_t* perm, const int32_t* offsets, void* out, void* ws, size_t ws_bytes,
                            const hmoe_forward_opts* opts, hmoe_stream_t stream) {
  const NvtxRange nvtx("hmoe_forward");
  const hmoe_forward_opts o = opts ? *opts : kDefaultOpts;
  bool grouped = false;
  hmoe_status s = check_forward(L, x, T, ids, gates, perm, offsets, out, o, &grouped);
  if (s != HMOE_OK) return s;
  WsLayout w{};
  if ((s = check_ws(L->d, T, ws, ws_bytes, &w)) != HMOE_OK) return s;
  return run_forward(L, x, T, gates, perm, offsets, out, ws, w, o, grouped, (cudaStream_t)stream);
}

hmoe_status hmoe_forward(const hmoe_layer* L, const void* x, int T, const int32_t* ids, const float* gates,
                         const int32_t* perm, const int32_t* offsets, void* out, void* ws, size_t ws_bytes,
                         hmoe_stream_t stream) {
  return hmoe_forward_ex(L, x, T, ids, gates, perm, offsets, out, ws, ws_bytes, nullptr, stream);
}

hmoe_status hmoe_check_device_status(void* ws, size_t ws_bytes, hmoe_stream_t stream) {
  if (!ws || ws_bytes < 256) return fail(HMOE_ERR_INVALID_ARG, "workspace is NULL or too small");
  int word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, ws, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(int), (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  if (word & DEV_TIMEOUT) return fail(HMOE_ERR_DEVICE_TIMEOUT, "a bounded device wait timed out (status 0x%x)", word);
  if (word & DEV_BAD_ROUTE) return fail(HMOE_ERR_BAD_ROUTE, "device found an out-of-range route entry (status 0x%x)", word);
  return HMOE_OK;
}

namespace {
hmoe_status debug_export(const hmoe_layer* L, int expert, int which, void* dst, float* scales, bool decode_operand,
                         cudaStream_t st) {
  const bool nf3 = (L->tab.loc[expert] & LOC_NF3) != 0;
  const int fmt = nf3 ? FMT_NF3 : L->d.kept_format;
  const ExpertGeom& g = nf3 ? L->gn : L->gk;
  const uint8_t* base = (nf3 ? L->nf3_buf : L->kept_buf) + (size_t)(L->tab.loc[expert] & 0x7FFF) * g.expert_bytes;
  const int N = which == 13 ? 2 * L->d.I : L->d.H;
  const int K = which == 13 ? L->d.H : L->d.I;
  cudaError_t e = launch_debug_dequant(fmt, which, base + (which == 2 ? g.w13_bytes : 0), N, K, L->d.I, dst, scales,
                                       decode_operand, L->d.act_dtype, L->d.act_quant == HMOE_ACT_QUANT_NVFP4, st);
  if (e != cudaSuccess) return cuda_fail(e, "debug dequant launch");
  return HMOE_OK;
}
}  // namespace

hmoe_status hmoe_debug_dequant(const hmoe_layer* L, int expert, int which, void* dst, hmoe_stream_t stream) {
  if (!L || !dst || expert < 0 || expert >= L->d.E || (which != 13 && which != 2))
    return fail(HMOE_ERR_INVALID_ARG, "bad arguments to hmoe_debug_dequant");
  return debug_export(L, expert, which, dst, nullptr, false, (cudaStream_t)stream);
}

hmoe_status hmoe_debug_decode_operand(const hmoe_layer* L, int expert, int which, void* dst, float* scales,
                                      hmoe_stream_t stream) {
  if (!L || !dst || !scales || expert < 0 || expert >= L->d.E || (which != 13 && which != 2))
    return fail(HMOE_ERR_INVALID_ARG, "bad arguments to hmoe_debug_decode_operand");
  return debug_export(L, expert, which, dst, scales, true, (cudaStream_t)stream);
}

}  // extern "C"

// ------------------------------------------------------------ allocation-free forward
// The scratch of hmoe_forward_static: one file-scope device array per GPU
// that loads the library. Host code must not use the symbol as an address.
// The device address is looked up once per device with
// cudaGetSymbolAddress while that device is current, and passed to the
// kernels like any caller workspace.
static __device__ __align__(256) unsigned char g_hmoe_static_scratch[HMOE_STATIC_SCRATCH_BYTES];

namespace {
constexpr int STATIC_MAX_DEVICES = 64;
std::mutex g_static_mu;
void* g_static_ptr[STATIC_MAX_DEVICES] = {};

hmoe_status static_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= STATIC_MAX_DEVICES)
    return fail(HMOE_ERR_INVALID_ARG, "device ordinal %d beyond the %d supported", dev, STATIC_MAX_DEVICES);
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_hmoe_static_scratch);
    if (e != cudaSuccess || !p) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return HMOE_OK;
}
}  // namespace

extern "C" {

hmoe_status hmoe_forward_static(const hmoe_layer* L, const void* x, int T, const int32_t* ids, const float* gates,
                                const int32_t* perm, const int32_t* offsets, void* out, hmoe_stream_t stream) {
  const NvtxRange nvtx("hmoe_forward_static");
  // Every argument check runs before anything is enqueued.
  bool grouped = false;
  hmoe_status s = check_forward(L, x, T, ids, gates, perm, offsets, out, kDefaultOpts, &grouped);
  if (s != HMOE_OK) return s;
  const WsLayout w = ws_layout(L->d, T);
  if (w.total > (size_t)HMOE_STATIC_SCRATCH_BYTES)
    return fail(HMOE_ERR_WORKSPACE_TOO_SMALL,
                "T=%d needs %zu bytes of scratch; the static scratch of hmoe_forward_static holds %u", T, w.total,
                (unsigned)HMOE_STATIC_SCRATCH_BYTES);
  void* ws = nullptr;
  if ((s = static_scratch(&ws)) != HMOE_OK) return s;
  if (T == 0) return HMOE_OK;
  // The array keeps the previous call's contents. The kernels' work queues
  // and group counters must start at zero: clear them. The status word is
  // left alone, so a fault an earlier call recorded stays until
  // hmoe_check_device_status_static reads it.
  cudaError_t e = cudaMemsetAsync(static_cast<uint8_t*>(ws) + w.queues, 0, w.chunk_cnt - w.queues,
                                  (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the static scratch");
  return run_forward(L, x, T, gates, perm, offsets, out, ws, w, kDefaultOpts, grouped, (cudaStream_t)stream);
}

hmoe_status hmoe_check_device_status_static(hmoe_stream_t stream) {
  void* ws = nullptr;
  hmoe_status s = static_scratch(&ws);
  if (s != HMOE_OK) return s;
  return hmoe_check_device_status(ws, HMOE_STATIC_SCRATCH_BYTES, stream);
}

}  // extern "C"

// ------------------------------------------------------------ dense Linear W4A16
// One weight matrix W [N, K] (NVFP4, MXFP4 or NF3) times bf16 or fp16
// activations, run by the layer's own kernels: the matrix is packed like an
// expert's W2, and a forward is the W2 phase of the streaming kernel
// (T <= 8) or of the tensor-core grouped kernel (above) over a one-expert
// route geometry with one slot per token and gate 1, then the finalize to
// the activation type.
struct hmoe_linear {
  hmoe_linear_desc d;
  uint8_t* packed;
  size_t bytes;
  ExpertTable tab;
  int num_sms;
};

namespace {
struct LinWs {
  size_t status, queues, perm, offsets, gates, y, total;
};
LinWs lin_layout(const hmoe_linear_desc& d, int T) {
  LinWs w{};
  size_t off = 0;
  w.status = off;
  off += 256;
  w.queues = off;
  off += 256;
  w.perm = off;
  off += align256((size_t)T * 4);
  w.offsets = off;
  off += 256;
  w.gates = off;
  off += align256((size_t)T * 4);
  w.y = off;
  off += align256((size_t)T * d.N * 4);
  w.total = off;
  return w;
}
hmoe_status check_linear_desc(const hmoe_linear_desc* d) {
  if (!d) return fail(HMOE_ERR_INVALID_ARG, "desc is NULL");
  if (d->fmt != HMOE_FMT_NVFP4 && d->fmt != HMOE_FMT_MXFP4 && d->fmt != HMOE_FMT_NF3)
    return fail(HMOE_ERR_INVALID_ARG, "fmt must be NVFP4 (4), MXFP4 (5) or NF3 (3), got %d", d->fmt);
  if (d->N <= 0 || d->K <= 0) return fail(HMOE_ERR_INVALID_ARG, "N and K must be positive");
  if (d->N % 128 != 0 || d->K % 64 != 0)
    return fail(HMOE_ERR_UNSUPPORTED_SHAPE, "N must be a multiple of 128 and K of 64 (N=%d K=%d)", d->N, d->K);
  if (d->act_dtype != HMOE_ACT_BF16 && d->act_dtype != HMOE_ACT_F16)
    return fail(HMOE_ERR_INVALID_ARG, "act_dtype must be HMOE_ACT_BF16 (0) or HMOE_ACT_F16 (1), got %d", d->act_dtype);
  return HMOE_OK;
}
}  // namespace

extern "C" {

hmoe_status hmoe_linear_packed_size(const hmoe_linear_desc* desc, size_t* bytes) {
  hmoe_status s = check_linear_desc(desc);
  if (s != HMOE_OK) return s;
  if (!bytes) return fail(HMOE_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = (size_t)(desc->N / TILE_ROWS) * (desc->K / TILE_K) * tile_bytes(desc->fmt);
  return HMOE_OK;
}

hmoe_status hmoe_linear_workspace_size(const hmoe_linear_desc* desc, int max_tokens, size_t* bytes) {
  hmoe_status s = check_linear_desc(desc);
  if (s != HMOE_OK) return s;
  if (!bytes || max_tokens < 0) return fail(HMOE_ERR_INVALID_ARG, "bytes NULL or max_tokens < 0");
  *bytes = lin_layout(*desc, max_tokens).total;
  return HMOE_OK;
}

hmoe_status hmoe_linear_pack(const hmoe_linear_desc* desc, const void* codes, const void* scales, float global_scale,
                             void* packed, hmoe_stream_t stream, hmoe_linear** out) {
  const NvtxRange nvtx("hmoe_linear_pack");
  hmoe_status s = check_linear_desc(desc);
  if (s != HMOE_OK) return s;
  if (!codes || !scales || !packed || !out) return fail(HMOE_ERR_INVALID_ARG, "a pointer is NULL");
  if (!aligned16(packed)) return fail(HMOE_ERR_INVALID_ARG, "packed buffer must be 16-byte aligned");
  hmoe_linear* L = new (std::nothrow) hmoe_linear();
  if (!L) return fail(HMOE_ERR_INVALID_ARG, "out of host memory");
  L->d = *desc;
  L->packed = static_cast<uint8_t*>(packed);
  hmoe_linear_packed_size(desc, &L->bytes);
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (ce == cudaSuccess)
    ce = launch_pack_matrix(desc->fmt, 2, codes, scales, desc->N, desc->K, desc->K, L->packed,
                            desc->act_dtype == HMOE_ACT_F16, (cudaStream_t)stream);
  if (ce != cudaSuccess) {
    delete L;
    return cuda_fail(ce, "linear pack");
  }
  L->tab.loc[0] = desc->fmt == HMOE_FMT_NF3 ? LOC_NF3 : 0;
  L->tab.g13[0] = 1.0f;
  L->tab.g2[0] = desc->fmt == HMOE_FMT_NVFP4 ? global_scale : 1.0f;
  *out = L;
  return HMOE_OK;
}

void hmoe_linear_destroy(hmoe_linear* L) { delete L; }

hmoe_status hmoe_linear_forward_ex(const hmoe_linear* L, const void* x, int T, void* out, void* ws, size_t ws_bytes,
                                   const hmoe_forward_opts* opts, hmoe_stream_t stream) {
  const NvtxRange nvtx("hmoe_linear_forward");
  if (!L) return fail(HMOE_ERR_INVALID_ARG, "linear is NULL");
  if (T < 0) return fail(HMOE_ERR_INVALID_ARG, "T=%d < 0", T);
  const hmoe_forward_opts o = opts ? *opts : kDefaultOpts;
  if (o.path < 0 || o.path > 2) return fail(HMOE_ERR_INVALID_ARG, "bad path %d", o.path);
  if (o.wait_limit_us < 0) return fail(HMOE_ERR_INVALID_ARG, "wait_limit_us < 0");
  if ((o.debug_flags & HMOE_DEBUG_GROUPED_PAIR) && L->d.act_dtype != HMOE_ACT_BF16)
    return fail(HMOE_ERR_INVALID_ARG, "the CTA-pair grouped kernel takes bf16 activations only");
  if (!ws) return fail(HMOE_ERR_INVALID_ARG, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return fail(HMOE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const LinWs w = lin_layout(L->d, T);
  if (ws_bytes < w.total)
    return fail(HMOE_ERR_WORKSPACE_TOO_SMALL, "workspace holds %zu bytes, T=%d needs %zu", ws_bytes, T, w.total);
  if (T == 0) return HMOE_OK;
  if (!x || !out) return fail(HMOE_ERR_INVALID_ARG, "x or out is NULL");
  if (!aligned16(x) || !aligned16(out)) return fail(HMOE_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
  const bool grouped = o.path == HMOE_PATH_GROUPED || (o.path == HMOE_PATH_AUTO && T > DECODE_MAX_T);
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  int* perm = reinterpret_cast<int*>(wsb + w.perm);
  int* offsets = reinterpret_cast<int*>(wsb + w.offsets);
  float* gates = reinterpret_cast<float*>(wsb + w.gates);
  float* y = reinterpret_cast<float*>(wsb + w.y);
  int* status = reinterpret_cast<int*>(wsb + w.status);
  const unsigned long long lim =
      o.wait_limit_us > 0 ? (unsigned long long)o.wait_limit_us * 1000ull : WAIT_LIMIT_NS;
  const int kept_fmt = L->d.fmt == HMOE_FMT_NF3 ? FMT_NVFP4 : L->d.fmt;  // the unused tier's format
  cudaError_t e = launch_identity_route(T, perm, offsets, gates, L->num_sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "linear route launch");
  if (grouped) {
    GroupedParams p{};
    p.kept_buf = L->packed;
    p.nf3_buf = L->packed;
    p.kept_fmt = kept_fmt;
    p.act_type = L->d.act_dtype;
    p.act_scale = 1.0f;
    p.which = 2;
    p.H = L->d.N;
    p.I = L->d.K;
    p.E = 1;
    p.topk = 1;
    p.T = T;
    p.K = L->d.K;
    p.RT = L->d.N / TILE_ROWS;
    p.KB = L->d.K / TILE_K;
    p.tier_mask = 3;
    p.kept_expert_bytes = p.nf3_expert_bytes = L->bytes;
    p.offsets = offsets;
    p.perm = perm;
    p.y_out = y;
    p.status = status;
    p.wait_limit_ns = lim;
    p.pair = (o.debug_flags & HMOE_DEBUG_GROUPED_PAIR) ? 1 : 0;
    p.tab = L->tab;
    e = launch_grouped_gemm(p, static_cast<const uint16_t*>(x), T, L->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "linear grouped GEMM launch");
  } else {
    StreamParams p{};
    p.kept_buf = L->packed;
    p.nf3_buf = L->packed;
    p.kept_fmt = kept_fmt;
    p.act_type = L->d.act_dtype;
    p.act_scale13 = p.act_scale2 = 1.0f;
    p.H = L->d.N;
    p.I = L->d.K;
    p.E = 1;
    p.topk = 1;
    p.T = T;
    p.group_tokens = 8;
    p.tier_mask = 3;
    p.kept_expert_bytes = p.nf3_expert_bytes = L->bytes;
    p.offsets = offsets;
    p.perm = perm;
    p.queue = reinterpret_cast<int*>(wsb + w.queues);
    p.done13 = nullptr;
    p.y_out = y;
    p.status = status;
    p.wait_limit_ns = lim;
    p.debug_no_copies = (o.debug_flags & HMOE_DEBUG_NO_COPIES) ? 1 : 0;
    p.tab = L->tab;
    StreamPhase& P = p.ph[1];
    P.rows = L->d.N;
    P.K = L->d.K;
    P.RT = L->d.N / TILE_ROWS;
    P.KB = L->d.K / TILE_K;
    P.kbs = pick_stage(P.KB);
    P.kbs1 = pick_stage(P.KB, 2 * STREAM_MAX_KBS);
    P.act = static_cast<const uint16_t*>(x);
    P.act_stride = L->d.K;
    P.kept_off = P.nf3_off = 0;
    p.ph[0] = P;
    p.ph_begin = 1;
    p.ph_end = 2;
    p.pair_items = (long long)std::min(T, 1) * ((P.RT + 1) / 2) >=
                           (long long)STREAM_PAIR_MIN_ITEMS_PER_CTA * stream_grid(L->num_sms)
                       ? 1
                       : 0;
    e = launch_stream_gemm(p, stream_grid(L->num_sms), st);
    if (e != cudaSuccess) return cuda_fail(e, "linear stream GEMM launch");
  }
  e = launch_finalize(y, gates, T, 1, L->d.N, static_cast<uint16_t*>(out), L->d.act_dtype, st);
  if (e != cudaSuccess) return cuda_fail(e, "linear finalize launch");
  return HMOE_OK;
}

hmoe_status hmoe_linear_forward(const hmoe_linear* L, const void* x, int T, void* out, void* ws, size_t ws_bytes,
                                hmoe_stream_t stream) {
  return hmoe_linear_forward_ex(L, x, T, out, ws, ws_bytes, nullptr, stream);
}

hmoe_status hmoe_quantize_act_nvfp4(const void* x, int rows, int K, int act_dtype, float global_scale, void* codes,
                                    void* scales, hmoe_stream_t stream) {
  const NvtxRange nvtx("hmoe_quantize_act_nvfp4");
  if (rows < 0) return fail(HMOE_ERR_INVALID_ARG, "rows=%d < 0", rows);
  if (K <= 0 || K % 16 != 0) return fail(HMOE_ERR_INVALID_ARG, "K=%d must be a positive multiple of 16", K);
  if (act_dtype != HMOE_ACT_BF16 && act_dtype != HMOE_ACT_F16)
    return fail(HMOE_ERR_INVALID_ARG, "act_dtype must be HMOE_ACT_BF16 (0) or HMOE_ACT_F16 (1), got %d", act_dtype);
  if (!(global_scale > 0.0f && global_scale < 3.0e38f))
    return fail(HMOE_ERR_INVALID_ARG, "global_scale must be finite and > 0 (got %g)", (double)global_scale);
  if (rows == 0) return HMOE_OK;
  if (!x || !codes || !scales) return fail(HMOE_ERR_INVALID_ARG, "a pointer is NULL");
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(codes) & 7) != 0)
    return fail(HMOE_ERR_INVALID_ARG, "x must be 16-byte and codes 8-byte aligned");
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = launch_act_quant(static_cast<const uint16_t*>(x), (long long)rows * K, global_scale, act_dtype, nullptr,
                         static_cast<uint8_t*>(codes), static_cast<uint8_t*>(scales), sms, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "activation quantisation launch");
  return HMOE_OK;
}

}  // extern "C"
