// route.cu -- routing kernels: softmax top-k, renormalised gates, stable counting sort.
//
// Cites: "quant: nvfp4_nf3_hybrid -- native serving for mixed NVFP4+NF3 MoE
// checkpoints", How it works. Both tiers share one route geometry (top-k
// ids, gates, token permutation, expert offsets). The routing function is
// not given on the pages. The reading taken is softmax top-k, with the k
// chosen gates renormalised and ties going to the lower expert id.
//
// The sort is deterministic: the slots of an expert keep ascending flat
// slot index s = t*k + j. No result depends on atomic ordering. Small
// batches use one CTA. Large batches use three kernels: per-chunk top-k and
// counts, a column scan over chunks, and a stable placement per chunk.
#include "common.cuh"
#include "internal.h"

namespace hmoe {

constexpr int ROUTE_CHUNK_TOKENS = 32;  // tokens per chunk in the large-batch path

// Order-preserving map of fp32 to uint32 (a > b exactly when key(a) >
// key(b)), with -0 mapped like +0 so that the two compare equal, as they do
// as floats. NaN logits are not supported.
__device__ __forceinline__ uint32_t route_key(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float route_key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// One warp routes one token. Lane l holds logits of experts l, l+32, ...
// (E <= 512, so at most 16 per lane), as order-preserving keys. Each of the
// k rounds takes the lane's best remaining candidate (the lowest expert id
// among equal keys), then the warp's largest key and, among the lanes that
// hold it, the lowest expert id (two warp reductions), so the winners come
// in descending order with ties to the lower id. Lane r (r < k) returns the
// r-th winner's id and gate.
__device__ __forceinline__ void warp_route_token(const float* __restrict__ row, int E, int k, int lane,
                                                 int* my_id, float* my_gate) {
  uint32_t key[MAX_E / 32];
#pragma unroll
  for (int j = 0; j < MAX_E / 32; ++j) {
    const int e = lane + 32 * j;
    key[j] = (e < E) ? route_key(row[e]) : 0u;  // 0: below every real key
  }
  uint32_t taken = 0;
  int rid = 0;
  uint32_t rkey = 0;
  for (int r = 0; r < k; ++r) {
    uint32_t bk = 0;
    uint32_t be = 0xFFFFFFFFu;
#pragma unroll
    for (int j = 0; j < MAX_E / 32; ++j) {
      if (!((taken >> j) & 1u) && key[j] > bk) {  // j ascending: the first of equal keys has the lowest id
        bk = key[j];
        be = (uint32_t)(lane + 32 * j);
      }
    }
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t w = __reduce_min_sync(0xffffffffu, bk == m ? be : 0xFFFFFFFFu);
    if ((int)(w & 31u) == lane) taken |= 1u << (w >> 5);
    if (lane == r) {
      rid = (int)w;
      rkey = m;
    }
  }
  const float rval = route_key_value(rkey);
  const float lmax = __shfl_sync(0xffffffffu, rval, 0);
  const float z = (lane < k) ? expf(rval - lmax) : 0.0f;
  float sum = z;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  *my_id = rid;
  *my_gate = z / sum;
}

// ------------------------------------------------------------ small batches: one CTA
// Requires T*k <= 1024. Shared memory: ids[S] + counts[E] + offsets[E+1].
__global__ void __launch_bounds__(1024) route_small_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                           int* __restrict__ ids, float* __restrict__ gates,
                                                           int* __restrict__ perm, int* __restrict__ offsets) {
  extern __shared__ int sm[];
  pdl_wait();
  pdl_trigger();
  const int S = T * k;
  int* s_ids = sm;
  int* s_cnt = sm + S;
  int* s_off = s_cnt + E;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  for (int e = tid; e < E; e += blockDim.x) s_cnt[e] = 0;
  for (int t = warp; t < T; t += nwarps) {
    int id;
    float gt;
    warp_route_token(logits + (size_t)t * E, E, k, lane, &id, &gt);
    if (lane < k) {
      ids[t * k + lane] = id;
      gates[t * k + lane] = gt;
      s_ids[t * k + lane] = id;
    }
  }
  __syncthreads();
  for (int s = tid; s < S; s += blockDim.x) atomicAdd(&s_cnt[s_ids[s]], 1);
  __syncthreads();
  if (warp == 0) {
    // exclusive scan of E counts by one warp: lane owns a contiguous run
    const int per = (E + 31) / 32;
    const int e0 = lane * per;
    int local = 0;
    for (int e = e0; e < min(E, e0 + per); ++e) local += s_cnt[e];
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += n;
    }
    int run = incl - local;
    for (int e = e0; e < min(E, e0 + per); ++e) {
      s_off[e] = run;
      run += s_cnt[e];
    }
    if (lane == 31) s_off[E] = incl;
  }
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) offsets[e] = s_off[e];
  // Stable ranks (thread s holds slot s; S <= blockDim.x): inside a warp,
  // match_any ranks the slots of equal experts; the warps take turns in slot
  // order, each adding the running per-expert count (s_cnt, reused) of the
  // warps before it.
  for (int e = tid; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  const int e_mine = tid < S ? s_ids[tid] : -1 - lane;  // distinct dummies never match real ids
  const unsigned peers = __match_any_sync(0xffffffffu, e_mine);
  const int rank_w = __popc(peers & ((1u << lane) - 1u));
  const int nw = (S + 31) / 32;
  for (int w = 0; w < nw; ++w) {
    if (warp == w) {
      const int base = tid < S ? s_cnt[e_mine] : 0;
      __syncwarp();
      if (tid < S) {
        perm[s_off[e_mine] + base + rank_w] = tid;
        if (rank_w == 0) s_cnt[e_mine] = base + __popc(peers);
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------ large batches
// K1: 8 warps x 4 tokens per CTA = one chunk of 32 tokens. Writes ids,
// gates and the chunk's per-expert counts (every expert, zeros included).
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int* __restrict__ ids, float* __restrict__ gates,
                                                         int* __restrict__ chunk_cnt) {
  __shared__ int s_cnt[MAX_E];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += blockDim.x) s_cnt[e] = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  const int t0 = blockIdx.x * ROUTE_CHUNK_TOKENS;
  for (int i = 0; i < ROUTE_CHUNK_TOKENS / 8; ++i) {
    const int t = t0 + warp * (ROUTE_CHUNK_TOKENS / 8) + i;
    if (t >= T) break;
    int id;
    float gt;
    warp_route_token(logits + (size_t)t * E, E, k, lane, &id, &gt);
    if (lane < k) {
      ids[t * k + lane] = id;
      gates[t * k + lane] = gt;
      atomicAdd(&s_cnt[id], 1);
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) chunk_cnt[(size_t)blockIdx.x * E + e] = s_cnt[e];
}

// K2: one CTA. Column-wise exclusive scan over chunks gives chunk_base; the
// expert totals are scanned to offsets. The chunks are split into P ranges
// (P = blockDim / E threads per expert), each summed by one thread, so that
// every thread has few dependent round trips to L2: pass 1 sums the ranges,
// pass 2 writes each range's prefix from its base.
__global__ void __launch_bounds__(1024) route_scan_kernel(const int* __restrict__ chunk_cnt, int nchunks, int E,
                                                          int S, int* __restrict__ chunk_base,
                                                          int* __restrict__ offsets) {
  __shared__ int s_tot[MAX_E + 1];
  __shared__ int s_part[1024];
  __shared__ int s_wsum[32];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  const int P = max(1, (int)blockDim.x / E);
  const int e = tid % E, q = tid / E;
  const bool act = q < P;
  const int c0 = (int)((long long)q * nchunks / P), c1 = (int)((long long)(q + 1) * nchunks / P);
  int part = 0;
  if (act) {
#pragma unroll 8
    for (int c = c0; c < c1; ++c) part += chunk_cnt[(size_t)c * E + e];
    s_part[q * E + e] = part;
  }
  __syncthreads();
  if (act) {
    int run = 0;
    for (int qq = 0; qq < q; ++qq) run += s_part[qq * E + e];
#pragma unroll 8
    for (int c = c0; c < c1; ++c) {
      const int a = chunk_cnt[(size_t)c * E + e];
      chunk_base[(size_t)c * E + e] = run;
      run += a;
    }
    if (q == P - 1) s_tot[e] = run;
  }
  __syncthreads();
  // block exclusive scan of s_tot[0..E)
  const int lane = tid & 31, warp = tid >> 5;
  const int v = (tid < E) ? s_tot[tid] : 0;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += n;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? s_wsum[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += n;
    }
    s_wsum[lane] = wi - w;
  }
  __syncthreads();
  if (tid < E) offsets[tid] = s_wsum[warp] + incl - v;
  if (tid == 0) offsets[E] = S;
}

// K3: stable placement of one chunk's slots. Slots are taken in rounds of
// 256 in ascending order. Inside a round, a warp ranks equal experts with
// match_any, and earlier warps and rounds are added from shared counts.
__global__ void __launch_bounds__(256) route_place_kernel(const int* __restrict__ ids, int T, int E, int k,
                                                          const int* __restrict__ chunk_base,
                                                          const int* __restrict__ offsets,
                                                          int* __restrict__ perm) {
  __shared__ int s_run[MAX_E];
  __shared__ int s_w[8][MAX_E];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x;
  const int s_begin = c * ROUTE_CHUNK_TOKENS * k;
  const int s_end = min(T * k, s_begin + ROUTE_CHUNK_TOKENS * k);
  for (int e = tid; e < E; e += 256) {
    s_run[e] = 0;
    for (int w = 0; w < 8; ++w) s_w[w][e] = 0;
  }
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  for (int base = s_begin; base < s_end; base += 256) {
    const int s = base + tid;
    const bool valid = s < s_end;
    const int e = valid ? ids[s] : -1 - lane;  // distinct dummies never match real ids
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank_w = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank_w == 0) s_w[warp][e] = __popc(peers);
    __syncthreads();
    if (valid) {
      int rank = s_run[e] + rank_w;
      for (int w = 0; w < warp; ++w) rank += s_w[w][e];
      perm[offsets[e] + chunk_base[(size_t)c * E + e] + rank] = s;
    }
    __syncthreads();
    for (int ee = tid; ee < E; ee += 256) {
      int add = 0;
      for (int w = 0; w < 8; ++w) {
        add += s_w[w][ee];
        s_w[w][ee] = 0;
      }
      s_run[ee] += add;
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------ launcher
int route_chunks(int T) { return (T + ROUTE_CHUNK_TOKENS - 1) / ROUTE_CHUNK_TOKENS; }

cudaError_t launch_route(const float* logits, int T, int E, int k, int* ids, float* gates, int* perm,
                         int* offsets, int* chunk_cnt, int* chunk_base, cudaStream_t st) {
  const int S = T * k;
  if (S <= 1024) {
    const size_t smem = (size_t)(S + 2 * E + 1) * sizeof(int);
    cudaError_t e = launch_pdl(route_small_kernel, dim3(1), dim3(1024), smem, st, logits, T, E, k, ids, gates, perm,
                               offsets);
    count_launches(1);
    return e;
  }
  const int nch = route_chunks(T);
  cudaError_t e = launch_pdl(route_topk_kernel, dim3(nch), dim3(256), 0, st, logits, T, E, k, ids, gates, chunk_cnt);
  if (e == cudaSuccess)
    e = launch_pdl(route_scan_kernel, dim3(1), dim3(1024), 0, st, (const int*)chunk_cnt, nch, E, S, chunk_base,
                   offsets);
  if (e == cudaSuccess)
    e = launch_pdl(route_place_kernel, dim3(nch), dim3(256), 0, st, (const int*)ids, T, E, k,
                   (const int*)chunk_base, (const int*)offsets, perm);
  count_launches(3);
  return e;
}

// The route geometry of a dense Linear: one "expert", one slot per token.
// perm[t] = t, offsets = {0, T}, gates[t] = 1.
__global__ void identity_route_kernel(int T, int* perm, int* offsets, float* gates) {
  pdl_wait();
  pdl_trigger();
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
    perm[t] = t;
    gates[t] = 1.0f;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    offsets[0] = 0;
    offsets[1] = T;
  }
}

cudaError_t launch_identity_route(int T, int* perm, int* offsets, float* gates, int num_sms, cudaStream_t st) {
  const int blocks = (T + 255) / 256;
  const int grid = blocks < 1 ? 1 : (blocks < num_sms ? blocks : num_sms);
  cudaError_t e = launch_pdl(identity_route_kernel, dim3(grid), dim3(256), 0, st, T, perm, offsets, gates);
  count_launches(1);
  return e;
}

}  // namespace hmoe
