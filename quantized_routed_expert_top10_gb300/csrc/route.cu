// Router (steps 1-2) and token grouping (step 3) of the routed-expert MoE block, sm_103a.
//
// zwxr.cn news/242664, section "一次路由的完整旅程": moe_route projects the normalised activation
// with a BF16 GEMV to 512 expert logits; native_router_top10 does a softmax over all 512, a stable
// descending argsort, gathers the first 10 and renormalises with ggml's lower clamp.
// momoyeyu.github.io "ai-infra-strata", section "提示词处理": tokens are gathered per expert so a
// single read of an expert's weights serves every token routed to it.
#include "device_common.cuh"

namespace strata {
namespace {

// top-k of one token's logits (global memory written by other CTAs or kernels) by one warp.
__device__ void top_k_warp(const float* logits, int E, TopKScratch& sc, int32_t* ids, float* weights) {
  int id;
  float w;
  top_k_warp_fn([&](int e) { return __ldcg(logits + e); }, E, sc, &id, &w);
  const int lane = threadIdx.x & 31;
  if (lane < K) {
    ids[lane] = id;
    weights[lane] = w;
  }
}

// ---------------------------------------------------------------------------------------------
// Grouping: counting sort of pair numbers p = t*K + k by expert (stable), active experts.
// ---------------------------------------------------------------------------------------------

// From per-expert counts (shared) build expert_off, active and n_active.
// Whole CTA; cnt is shared [E]; sh_off, sh_flag shared [E]; scratch shared [>= 32].
__device__ void finish_grouping(const int* cnt, int E, int* sh_off, int* sh_flag, int* scratch,
                                int32_t* expert_off, int32_t* active, int32_t* n_active) {
  const int tid = threadIdx.x;
  const int total = cta_exclusive_scan(cnt, sh_off, E, scratch);
  for (int e = tid; e < E; e += blockDim.x) expert_off[e] = sh_off[e];
  if (tid == 0) expert_off[E] = total;
  // active list: exclusive scan of (cnt > 0) flags
  for (int e = tid; e < E; e += blockDim.x) sh_flag[e] = cnt[e] > 0 ? 1 : 0;
  __syncthreads();
  const int na = cta_exclusive_scan(sh_flag, sh_flag, E, scratch);
  for (int e = tid; e < E; e += blockDim.x)
    if (cnt[e] > 0) active[sh_flag[e]] = e;
  if (tid == 0) n_active[0] = na;
}

// ---------------------------------------------------------------------------------------------
// Decode routing: one kernel for T <= DECODE_T_MAX.  Every CTA computes 4 logits rows (one per
// warp) for all tokens and quantises a share of the expert input; the last CTA to finish runs
// top-k for every token, the grouping and the tile list.
// ---------------------------------------------------------------------------------------------
template <int TT>
__global__ void __launch_bounds__(128) route_decode_kernel(
    const float* __restrict__ x, int T, int apply_rmsnorm, const uint16_t* __restrict__ wr,
    const float* __restrict__ bias, int E, int q2_offset, float* __restrict__ logits,
    float* __restrict__ logits_user, int32_t* __restrict__ ids, float* __restrict__ weights,
    int32_t* __restrict__ expert_off, int32_t* __restrict__ pair, int32_t* __restrict__ active,
    int32_t* __restrict__ n_active, QBlock* __restrict__ qx,
    int* __restrict__ counter, int* __restrict__ status) {
  __shared__ float s_inv[TT];
  __shared__ float s_red[4][TT];
  __shared__ int32_t s_tmp[4][64];
  __shared__ int s_cnt[EMAX];
  __shared__ int s_off[EMAX];
  __shared__ int s_tile[EMAX];
  __shared__ int s_scratch[32];
  __shared__ int s_last;
  __shared__ TopKScratch s_topk[4];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // 1/rms per token (every CTA recomputes it; x is tiny and L2-resident).
  if (apply_rmsnorm) {
    float ss[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) ss[t] = 0.f;
    for (int h = tid; h < H; h += 128) {
#pragma unroll
      for (int t = 0; t < TT; ++t)
        if (t < T) { const float v = x[(size_t)t * H + h]; ss[t] += v * v; }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      const float r = warp_sum(ss[t]);
      if (lane == 0) s_red[warp][t] = r;
    }
    __syncthreads();
    if (tid < TT) {
      const float r = s_red[0][tid] + s_red[1][tid] + s_red[2][tid] + s_red[3][tid];
      s_inv[tid] = 1.f / sqrtf(r / (float)H + 1e-6f);
    }
  } else if (tid < TT) {
    s_inv[tid] = 1.f;
  }
  __syncthreads();

  // Router GEMV: warp -> expert row e; lane covers 8 columns per step, 10 steps.
  const int e = blockIdx.x * 4 + warp;
  if (e < E) {
    float acc[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t] = 0.f;
    const uint4* wrow = reinterpret_cast<const uint4*>(wr + (size_t)e * H);
#pragma unroll 5
    for (int i = 0; i < H / 256; ++i) {
      const int c = 8 * lane + 256 * i;
      const uint4 wv = __ldg(wrow + (c >> 3));
      float wf[8];
      wf[0] = __uint_as_float(wv.x << 16); wf[1] = __uint_as_float(wv.x & 0xffff0000u);
      wf[2] = __uint_as_float(wv.y << 16); wf[3] = __uint_as_float(wv.y & 0xffff0000u);
      wf[4] = __uint_as_float(wv.z << 16); wf[5] = __uint_as_float(wv.z & 0xffff0000u);
      wf[6] = __uint_as_float(wv.w << 16); wf[7] = __uint_as_float(wv.w & 0xffff0000u);
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        if (t < T) {
          const float4 a = __ldg(reinterpret_cast<const float4*>(x + (size_t)t * H + c));
          const float4 b = __ldg(reinterpret_cast<const float4*>(x + (size_t)t * H + c + 4));
          float s = acc[t];
          s = fmaf(wf[0], a.x, s); s = fmaf(wf[1], a.y, s); s = fmaf(wf[2], a.z, s); s = fmaf(wf[3], a.w, s);
          s = fmaf(wf[4], b.x, s); s = fmaf(wf[5], b.y, s); s = fmaf(wf[6], b.z, s); s = fmaf(wf[7], b.w, s);
          acc[t] = s;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      const float r = warp_sum(acc[t]);
      if (lane == 0 && t < T) {
        const float v = r * s_inv[t] + (bias ? bias[e] : 0.f);
        logits[(size_t)t * EMAX + e] = v;
        if (logits_user) logits_user[(size_t)t * E + e] = v;
      }
    }
  }

  // Quantise the expert input (rmsnorm(x) or x), one 64-block per warp.
  {
    const int nblk = T * KB_GU;
    for (int b = blockIdx.x * 4 + warp; b < nblk; b += gridDim.x * 4) {
      const int t = b / KB_GU, kb = b % KB_GU;
      const float2 v = *reinterpret_cast<const float2*>(x + (size_t)t * H + kb * QK + 2 * lane);
      quantise_block_warp(v.x * s_inv[t], v.y * s_inv[t], q2_offset, qx + b, s_tmp[warp]);
    }
  }

  // Last CTA: top-k for all tokens, then grouping.
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(counter, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int t = warp; t < T; t += 4)
    top_k_warp(logits + (size_t)t * EMAX, E, s_topk[warp], ids + t * K, weights + t * K);
  for (int i = tid; i < E; i += 128) s_cnt[i] = 0;
  __syncthreads();
  const int P = T * K;
  for (int p = tid; p < P; p += 128) {
    const int ee = ids[p];
    if (ee < 0 || ee >= E) set_status(status, ST_CORRUPT);
    else atomicAdd(&s_cnt[ee], 1);
  }
  __syncthreads();
  finish_grouping(s_cnt, E, s_off, s_tile, s_scratch, expert_off, active, n_active);
  __syncthreads();
  if (warp == 0) stable_scatter_warp(ids, 0, P, E, s_off, pair, 0);
  if (tid == 0) *counter = 0;
}

// ---------------------------------------------------------------------------------------------
// Prefill routing kernels.
// ---------------------------------------------------------------------------------------------
// Logits of token t = the router GEMM's ROUTER_KSPLIT partial sums added in a fixed order, plus the
// bias; then the top-10 of the token (one warp per token).
__global__ void __launch_bounds__(128) top_k_kernel(const float* __restrict__ parts, int T, int E,
                                                    const float* __restrict__ bias, float* __restrict__ logits_out,
                                                    int32_t* __restrict__ ids, float* __restrict__ weights) {
  static_assert(ROUTER_KSPLIT == 2, "the fixed summation order below assumes two slices");
  __shared__ TopKScratch s_topk[4];
  griddep_launch_dependents();
  griddep_wait();
  const int t = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;
  const size_t slice = (size_t)T * EMAX;
  const float* p = parts + (size_t)t * EMAX;
  // every load is issued before the first sum, so the warp waits for memory once, not once per j
  float a[16], b[16], lg[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int e = lane + 32 * j;
    a[j] = e < E ? __ldcg(p + e) : 0.f;
    b[j] = e < E ? __ldcg(p + slice + e) : 0.f;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int e = lane + 32 * j;
    float v = 0.f;
    if (e < E) {
      v = a[j] + b[j];
      if (bias) v += __ldg(bias + e);
      if (logits_out) logits_out[(size_t)t * E + e] = v;
    }
    lg[j] = v;
  }
  int id;
  float w;
  top_k_warp_fn([&](int e) { return lg[e >> 5]; }, E, s_topk[threadIdx.x >> 5], &id, &w);
  if (lane < K) {
    ids[t * K + lane] = id;
    weights[t * K + lane] = w;
  }
}

__global__ void __launch_bounds__(256) group_hist_kernel(const int32_t* __restrict__ ids, int P, int E,
                                                         int32_t* __restrict__ chunk_cnt, int* status) {
  __shared__ int cnt[EMAX];
  griddep_launch_dependents();
  griddep_wait();
  for (int i = threadIdx.x; i < E; i += 256) cnt[i] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * GROUP_CHUNK, p1 = min(P, p0 + GROUP_CHUNK);
  int ev[GROUP_CHUNK / 256];  // the thread's ids, loaded before any is counted
#pragma unroll
  for (int j = 0; j < GROUP_CHUNK / 256; ++j) {
    const int p = p0 + (int)threadIdx.x + 256 * j;
    ev[j] = p < p1 ? __ldg(ids + p) : 0;
  }
#pragma unroll
  for (int j = 0; j < GROUP_CHUNK / 256; ++j) {
    if (p0 + (int)threadIdx.x + 256 * j >= p1) break;
    const int e = ev[j];
    if (e < 0 || e >= E) set_status(status, ST_CORRUPT);
    else atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += 256) chunk_cnt[(size_t)blockIdx.x * EMAX + i] = cnt[i];
}

// One CTA of 512 threads: per-expert running base over chunks (chunk_cnt becomes exclusive bases
// within each expert; each thread reads its expert's counts of eight chunks at a time with independent
// loads), then offsets and the active list.
__global__ void __launch_bounds__(512) group_scan_kernel(int n_chunks, int E, int32_t* __restrict__ chunk_cnt,
                                                         int32_t* __restrict__ expert_off,
                                                         int32_t* __restrict__ active,
                                                         int32_t* __restrict__ n_active) {
  __shared__ int s_cnt[EMAX], s_off[EMAX], s_flag[EMAX], s_scratch[32];
  griddep_launch_dependents();
  griddep_wait();
  const int e = threadIdx.x;
  if (e < E) {
    int run = 0;
    for (int c0 = 0; c0 < n_chunks; c0 += 8) {
      int v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = c0 + j < n_chunks ? chunk_cnt[(size_t)(c0 + j) * EMAX + e] : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (c0 + j < n_chunks) {
          chunk_cnt[(size_t)(c0 + j) * EMAX + e] = run;
          run += v[j];
        }
    }
    s_cnt[e] = run;
  }
  __syncthreads();
  finish_grouping(s_cnt, E, s_off, s_flag, s_scratch, expert_off, active, n_active);
}

// One CTA of 8 warps per chunk: the chunk's ids staged in shared memory with independent loads; each
// warp counts its 256-pair slice, the slices' bases per expert are a prefix over the warps starting at
// expert_off[e] + the chunk's base, and each warp scatters its slice stably (the order is the
// chunk's, as one warp walking the whole chunk would give).
constexpr int SCATTER_WARPS = 8;
constexpr int SCATTER_SLICE = GROUP_CHUNK / SCATTER_WARPS;
__global__ void __launch_bounds__(32 * SCATTER_WARPS) group_scatter_kernel(const int32_t* __restrict__ ids, int P,
                                                                           int E, const int32_t* __restrict__ chunk_cnt,
                                                                           const int32_t* __restrict__ expert_off,
                                                                           int32_t* __restrict__ pair) {
  __shared__ int s_ids[GROUP_CHUNK];
  __shared__ int s_base[SCATTER_WARPS][EMAX];  // per-slice counts, then per-slice bases
  griddep_launch_dependents();
  griddep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p0 = blockIdx.x * GROUP_CHUNK, p1 = min(P, p0 + GROUP_CHUNK);
  for (int i = threadIdx.x; i < SCATTER_WARPS * EMAX; i += 32 * SCATTER_WARPS) (&s_base[0][0])[i] = 0;
  for (int p = p0 + (int)threadIdx.x; p < p1; p += 32 * SCATTER_WARPS) s_ids[p - p0] = __ldg(ids + p);
  __syncthreads();
  const int q0 = warp * SCATTER_SLICE, q1 = min(p1 - p0, q0 + SCATTER_SLICE);
  for (int q = q0 + lane; q < q1; q += 32) {
    const int e = s_ids[q];
    if (e >= 0 && e < E) atomicAdd(&s_base[warp][e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += 32 * SCATTER_WARPS) {
    int run = expert_off[e] + chunk_cnt[(size_t)blockIdx.x * EMAX + e];
#pragma unroll
    for (int w = 0; w < SCATTER_WARPS; ++w) {
      const int c = s_base[w][e];
      s_base[w][e] = run;
      run += c;
    }
  }
  __syncthreads();
  if (q0 < q1) stable_scatter_warp(s_ids, q0, q1, E, s_base[warp], pair, p0);
}

}  // namespace

cudaError_t launch_route_decode(const float* x, int T, int apply_rmsnorm, const uint16_t* w_router,
                                const float* bias, int E, int q2_offset, int32_t* ids, float* weights,
                                float* logits_out, const WsLayout& L, char* ws, cudaStream_t s) {
  const int grid = (E + 3) / 4;
#define STRATA_ROUTE_ARGS                                                                           \
  x, T, apply_rmsnorm, w_router, bias, E, q2_offset, (float*)(ws + L.logits), logits_out, ids, weights, \
      (int32_t*)(ws + L.expert_off), (int32_t*)(ws + L.pair), (int32_t*)(ws + L.active),              \
      (int32_t*)(ws + L.n_active), (QBlock*)(ws + L.qx),                                            \
      (int*)(ws + L.cnt_route), (int*)(ws + L.status)
  kernel_begin(KID_ROUTE_DECODE, s);
  if (T <= 1) route_decode_kernel<1><<<grid, 128, 0, s>>>(STRATA_ROUTE_ARGS);
  else if (T <= 2) route_decode_kernel<2><<<grid, 128, 0, s>>>(STRATA_ROUTE_ARGS);
  else if (T <= 4) route_decode_kernel<4><<<grid, 128, 0, s>>>(STRATA_ROUTE_ARGS);
  else route_decode_kernel<8><<<grid, 128, 0, s>>>(STRATA_ROUTE_ARGS);
  kernel_end(KID_ROUTE_DECODE, s);
#undef STRATA_ROUTE_ARGS
  return cudaGetLastError();
}

cudaError_t launch_top_k(const float* parts, int T, int E, const float* bias, float* logits_out, int32_t* ids,
                         float* weights, cudaStream_t s) {
  STRATA_LAUNCH(KID_TOP_K, s,
                launch_pdl(top_k_kernel, (T + 3) / 4, 128, 0, s, parts, T, E, bias, logits_out, ids, weights));
  return cudaGetLastError();
}

cudaError_t launch_group(const int32_t* ids, int T, int E, int32_t* expert_off, int32_t* pair, int32_t* active,
                         int32_t* n_active, const WsLayout& L, char* ws, cudaStream_t s) {
  const int P = T * K;
  int32_t* chunk_cnt = (int32_t*)(ws + L.chunk_cnt);
  int32_t* nat = (int32_t*)(ws + L.n_active);
  STRATA_LAUNCH(KID_GROUP_HIST, s,
                launch_pdl(group_hist_kernel, L.n_chunks, 256, 0, s, ids, P, E, chunk_cnt, (int*)(ws + L.status)));
  STRATA_LAUNCH(KID_GROUP_SCAN, s,
                launch_pdl(group_scan_kernel, 1, 512, 0, s, L.n_chunks, E, chunk_cnt, expert_off, active, nat));
  STRATA_LAUNCH(KID_GROUP_SCATTER, s,
                launch_pdl(group_scatter_kernel, L.n_chunks, 32 * SCATTER_WARPS, 0, s, ids, P, E, chunk_cnt, expert_off, pair));
  if (n_active && n_active != nat) cudaMemcpyAsync(n_active, nat, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
  return cudaGetLastError();
}

}  // namespace strata
