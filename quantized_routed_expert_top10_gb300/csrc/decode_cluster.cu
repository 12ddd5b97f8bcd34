// One-kernel MoE layer for small token counts (decode and verify windows, T <= 8), sm_103a,
// built on thread-block clusters.
//
// The layer -- router GEMV (zwxr.cn news/242664, "一次路由的完整旅程": BF16 projection to 512 logits,
// softmax, stable descending top-10, clamped renormalisation), grouping of tokens by expert
// (momoyeyu.github.io "ai-infra-strata", "提示词处理": one weight read serves every token routed to an
// expert), the Q2_0 SwiGLU experts (ai.thesatyajit.com "Strata engine", "The CPU kernels": codes
// {0,1,2,3} = {-1,0,1,2} x d, the offset removed once per block) and the weighted combine -- is one
// cooperative launch of 8-CTA clusters, two CTAs per SM:
//   1. every CTA computes a few router rows (two warps per row) and quantises a few 64-blocks of x;
//      the results are written to 16 replicas so that the next phase's reads spread over L2 slices;
//   2. one grid barrier (the last arriving CTA releases 16 replicated flags); every CTA then
//      computes the top-10 of all tokens and the grouping itself (identical everywhere);
//   3. cluster j takes distinct expert j (and j + #clusters, ...).  CTA rank r of the cluster
//      streams gate/up k-blocks [5r, 5r + 5) of all 640 rows and down row tiles r, r + 8, r + 16
//      through a ring of shared-memory stages (cp.async.bulk, L2 evict-first), so the expert's
//      1,382,400 bytes are split evenly over the cluster;
//   4. gate/up partial sums stay in each CTA's shared memory; after a cluster barrier, CTA r adds
//      the eight partials of the 64-row h blocks it owns (r and r + 8) through distributed shared
//      memory in rank order, applies silu(g) * u and quantises h; after a second cluster barrier
//      every CTA gathers the ten h blocks it needs for its down rows from their owners;
//   5. down rows go to parts[pair][row]; the last expert to finish an output row tile (a global
//      counter per tile) combines the ten weighted outputs of every token in k order (+ residual).
// All global waits are bounded by %globaltimer and record STRATA_E_TIMEOUT; cluster barriers are
// executed unconditionally by every CTA of a cluster, so a failed wait never strands a peer.  The
// last CTA to leave resets the counters for the next call.
#include "device_common.cuh"

namespace strata {
namespace {

constexpr int DC_THREADS = 256;
constexpr int DC_CLUSTER = 8;
constexpr int DC_UNIT = 23040;                 // bytes per streamed unit (5 gate/up k-blocks of a row tile,
                                               // or a whole 128-row down tile)
constexpr int DC_KBS = KB_GU / DC_CLUSTER;     // 5 gate/up k-blocks per CTA
constexpr int DC_MAXD = DECODE_T_MAX * K;      // at most 80 distinct experts
constexpr int DC_MAX_CLUSTERS = 64;
static_assert(DC_KBS * GU_CHUNK == DC_UNIT && KB_D * D_CHUNK == DC_UNIT, "equal unit sizes");
static_assert(FF / QK <= 2 * DC_CLUSTER, "each CTA owns at most two h blocks");

template <int TT>
struct DcCfg {
  static constexpr int NS = TT <= 4 ? 3 : 2;                          // ring stages
  static constexpr size_t RING = (size_t)NS * DC_UNIT;
  static constexpr size_t QX = sizeof(QBlock) * DC_KBS * TT;          // gate/up activation slice [5][TT]
  static constexpr size_t PBUF = sizeof(float2) * FF * TT;            // (g, u) partials [FF][TT]
  static constexpr size_t HQL = sizeof(QBlock) * 2 * TT;              // owned h blocks [2][TT]
  static constexpr size_t HQA = sizeof(QBlock) * KB_D * TT;           // gathered h blocks [10][TT]
  static constexpr size_t SMEM = RING + QX + PBUF + HQL + HQA;
};

struct DcParams {
  const float* x;  // [T][H] layer input (may alias out)
  float* out;      // [T][H]
  int T, E, q2_offset, residual;
  const uint16_t* wr;  // [E][H] bf16
  const float* bias;   // [E] or null
  const uint8_t* blobs;
  int64_t stride;
  int32_t* ids_out;  // [T][K]
  float* w_out;      // [T][K]
  float* dots;       // ws [WS_NREP][T][EMAX] router dot products, replicated
  float* sumsq;      // ws [WS_NREP][T][KB_GU] block sums of squares, replicated
  QBlock* qx;        // ws [T][KB_GU]
  float* parts;      // ws [T*K][H]
  int* sync;         // ws sync words
  int* status;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of `local` in the CTA of the given rank
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
  return a;
}
__device__ __forceinline__ float2 ld_dsmem_f2(uint32_t a) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_dsmem_u4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ int ld_dsmem_i32(uint32_t a) {
  int v;
  asm volatile("ld.shared::cluster.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ void qblock_words(const QBlock& a, uint32_t* hi, uint32_t* lo) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint4 h4 = reinterpret_cast<const uint4*>(a.hi)[w];
    const uint4 l4 = reinterpret_cast<const uint4*>(a.lo)[w];
    hi[4 * w] = h4.x; hi[4 * w + 1] = h4.y; hi[4 * w + 2] = h4.z; hi[4 * w + 3] = h4.w;
    lo[4 * w] = l4.x; lo[4 * w + 1] = l4.y; lo[4 * w + 2] = l4.z; lo[4 * w + 3] = l4.w;
  }
}

template <int TT>
__global__ void __launch_bounds__(DC_THREADS, 2) decode_cluster_kernel(const DcParams p) {
  using C = DcCfg<TT>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  QBlock* sqx = reinterpret_cast<QBlock*>(smem + C::RING);
  float2* pbuf = reinterpret_cast<float2*>(smem + C::RING + C::QX);
  QBlock* hql = reinterpret_cast<QBlock*>(smem + C::RING + C::QX + C::PBUF);
  QBlock* hqa = reinterpret_cast<QBlock*>(smem + C::RING + C::QX + C::PBUF + C::HQL);
  __shared__ uint64_t bars[C::NS];
  __shared__ int s_pending[C::NS];
  __shared__ float s_inv[TT];
  __shared__ int s_ids[TT * K];
  __shared__ float s_w[TT * K];
  __shared__ int s_te[DC_MAXD], s_tn[DC_MAXD], s_tq[DC_MAXD];
  __shared__ int s_first[TT * K];
  __shared__ int s_pair[TT * K];
  __shared__ float s_rpart[8][TT];
  __shared__ float s_bias[EMAX];
  __shared__ int32_t s_qtmp[8][64];
  __shared__ float s_h[TT][64];
  __shared__ float s_dn[TT][RT];
  __shared__ int s_flag, s_ok, s_nact, s_deff;

  const int G = gridDim.x, c = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T, E = p.E, P = T * K;
  const int rank = (int)cluster_rank(), cid = (int)cluster_index(), NCL = (int)cluster_count();
  int* bar = p.sync + WS_SYNC_BAR;
  int* exit_cnt = p.sync + WS_SYNC_EXIT;
  int* cnt_dn = p.sync + WS_SYNC_CNT_DN;

  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&bars[s], 1);
      s_pending[s] = -1;
    }
    fence_mbar_init();
    s_ok = 1;
    s_nact = 0;
  }
  for (int e = tid; e < E; e += DC_THREADS) s_bias[e] = p.bias ? __ldg(p.bias + e) : 0.f;

  // ---- 1. router dot products (two warps per row, four rows per CTA), x quantisation ----
  for (int e0 = c; e0 < E; e0 += 4 * G) {
    const int e = e0 + G * (warp >> 1);
    const int half = warp & 1;
    float acc[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t] = 0.f;
    if (e < E) {
      const uint4* wrow = reinterpret_cast<const uint4*>(p.wr + (size_t)e * H);
#pragma unroll
      for (int i = 0; i < H / 512; ++i) {
        const int col = half * (H / 2) + 8 * lane + 256 * i;
        float wf[8];
        bf16x8_to_f32(__ldg(wrow + (col >> 3)), wf);
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          if (t < T) {
            const float4 a4 = __ldg(reinterpret_cast<const float4*>(p.x + (size_t)t * H + col));
            const float4 b4 = __ldg(reinterpret_cast<const float4*>(p.x + (size_t)t * H + col + 4));
            float sa = acc[t];
            sa = fmaf(wf[0], a4.x, sa); sa = fmaf(wf[1], a4.y, sa); sa = fmaf(wf[2], a4.z, sa); sa = fmaf(wf[3], a4.w, sa);
            sa = fmaf(wf[4], b4.x, sa); sa = fmaf(wf[5], b4.y, sa); sa = fmaf(wf[6], b4.z, sa); sa = fmaf(wf[7], b4.w, sa);
            acc[t] = sa;
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      const float r = warp_sum(acc[t]);
      if (lane == 0) s_rpart[warp][t] = r;
    }
    __syncthreads();
    if (tid < 4 * TT) {
      const int slot = tid / TT, t = tid % TT;
      const int e2 = e0 + G * slot;
      if (e2 < E && t < T) {
        const float v = s_rpart[2 * slot][t] + s_rpart[2 * slot + 1][t];
#pragma unroll
        for (int r = 0; r < WS_NREP; ++r) p.dots[((size_t)r * T + t) * EMAX + e2] = v;
      }
    }
    __syncthreads();
  }
  for (int b = c + G * warp; b < T * KB_GU; b += 8 * G) {
    const int t = b / KB_GU, kb = b % KB_GU;
    const float2 v = __ldg(reinterpret_cast<const float2*>(p.x + (size_t)t * H + kb * QK + 2 * lane));
    const float ss = warp_sum(v.x * v.x + v.y * v.y);
    if (lane == 0)
#pragma unroll
      for (int r = 0; r < WS_NREP; ++r) p.sumsq[(size_t)r * T * KB_GU + b] = ss;
    quantise_block_warp(v.x, v.y, p.q2_offset, p.qx + b, s_qtmp[warp]);
  }

  // ---- grid barrier: last arriver releases replicated flags ----
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(bar, 1) == G - 1) {
      __threadfence();
#pragma unroll
      for (int r = 0; r < WS_NREP; ++r) st_relaxed(p.sync + WS_SYNC_REL + 32 * r, 1);
    }
    s_ok = spin_until_geq(p.sync + WS_SYNC_REL + 32 * (c % WS_NREP), 1, p.status) ? 1 : 0;
  }
  __syncthreads();

  // ---- 2. top-10 and grouping, in every CTA ----
  if (s_ok) {
    if (tid < T) {
      float inv = 1.f;
      if (p.residual) {
        const float* ssq = p.sumsq + ((size_t)(c % WS_NREP) * T + tid) * KB_GU;
        float s = 0.f;
        for (int kb = 0; kb < KB_GU; ++kb) s += __ldcg(ssq + kb);
        inv = 1.f / sqrtf(s / (float)H + 1e-6f);
      }
      s_inv[tid] = inv;
    }
    __syncthreads();
    for (int t = warp; t < T; t += 8) {
      const float inv = s_inv[t];
      const float* d = p.dots + ((size_t)(c % WS_NREP) * T + t) * EMAX;
      float lg[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int e = lane + 32 * j;
        lg[j] = (e < E) ? __ldcg(d + e) * inv + s_bias[e] : 0.f;
      }
      int id;
      float w;
      top_k_warp_fn([&](int e) { return lg[e >> 5]; }, E, &id, &w);
      if (lane < K) {
        s_ids[t * K + lane] = id;
        s_w[t * K + lane] = w;
      }
    }
    __syncthreads();
    // grouping of the P <= 80 pairs: slot of pair q = (pairs with a smaller expert id) + (earlier pairs
    // with the same expert); expert slot j = (distinct smaller ids).
    if (tid < P) {
      const int e = s_ids[tid];
      int first = 1;
      for (int q = 0; q < tid; ++q) first &= (s_ids[q] != e);
      s_first[tid] = first;
    }
    __syncthreads();
    if (tid < P) {
      const int e = s_ids[tid];
      int below = 0, same_before = 0, cnt = 0, dbelow = 0;
      for (int q = 0; q < P; ++q) {
        const int f = s_ids[q];
        below += (f < e);
        cnt += (f == e);
        same_before += (q < tid && f == e);
        dbelow += (s_first[q] && f < e);
      }
      s_pair[below + same_before] = tid;
      if (s_first[tid]) {
        s_te[dbelow] = e;
        s_tn[dbelow] = cnt;
        s_tq[dbelow] = below;
        atomicAdd(&s_nact, 1);
      }
    }
    if (c == 0)
      for (int q = tid; q < P; q += DC_THREADS) {
        p.ids_out[q] = s_ids[q];
        p.w_out[q] = s_w[q];
      }
    __syncthreads();
  }
  if (tid == 0) s_deff = s_ok ? s_nact : 0;
  __syncthreads();
  cluster_sync();
  // every CTA of the cluster follows rank 0's expert count, so cluster barriers always match
  const int D = ld_dsmem_i32(dsmem_addr(&s_deff, 0));
  cluster_sync();  // rank 0's shared memory stays valid until every peer has read it

  // ---- 3-5. experts: cluster cid takes distinct experts cid, cid + NCL, ... ----
  const uint64_t pol = policy_evict_first();
  const int n_dn = (rank + 2 * DC_CLUSTER < RT_D) ? 3 : 2;  // down tiles rank, rank + 8 (, rank + 16)
  const int n_units = RT_GU + n_dn;
  int ph[C::NS];  // next phase parity of each ring stage (persists across experts, like the barriers)
#pragma unroll
  for (int s = 0; s < C::NS; ++s) ph[s] = 0;
  for (int j = cid; j < D; j += NCL) {
    const int e = s_te[j], n = s_tn[j], q0 = s_tq[j];
    const uint8_t* blob = p.blobs + (int64_t)e * p.stride;
    auto unit_src = [&](int u) -> const uint8_t* {
      if (u < RT_GU) return blob + ((int64_t)u * KB_GU + rank * DC_KBS) * GU_CHUNK;
      const int rtd = rank + DC_CLUSTER * (u - RT_GU);
      return blob + D_REGION + (int64_t)rtd * KB_D * D_CHUNK;
    };
    if (tid == 0)
      for (int u = 0; u < C::NS && u < n_units; ++u) {
        s_pending[u] = ph[u];
        mbar_expect_tx(&bars[u], DC_UNIT);
        bulk_g2s_stream(ring + (size_t)u * DC_UNIT, unit_src(u), DC_UNIT, &bars[u], pol);
      }
    for (int idx = tid; idx < DC_KBS * TT * 9; idx += DC_THREADS) {
      const int blk = idx / 9, part = idx % 9;
      const int kb = blk / TT, ii = blk % TT;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (ii < n) {
        const int t = s_pair[q0 + ii] / K;
        v = __ldcg(reinterpret_cast<const uint4*>(p.qx + (size_t)t * KB_GU + rank * DC_KBS + kb) + part);
      }
      reinterpret_cast<uint4*>(sqx + blk)[part] = v;
    }
    __syncthreads();
    float tinv[TT];
#pragma unroll
    for (int ii = 0; ii < TT; ++ii) tinv[ii] = (ii < n) ? s_inv[s_pair[q0 + ii] / K] : 0.f;

    for (int u = 0; u < n_units; ++u) {
      const int st = u % C::NS;
      const bool ok = __syncthreads_and(s_ok && mbar_wait(&bars[st], (uint32_t)ph[st], p.status) ? 1 : 0);
      if (tid == 0) s_pending[st] = -1;
      ph[st] ^= 1;
      const uint8_t* stage = ring + (size_t)st * DC_UNIT;
      if (u < RT_GU) {
        // gate/up: thread = (row, matrix); 5 k-blocks
        const int row = tid & (RT - 1), mat = tid >> 7;
        float acc[TT];
#pragma unroll
        for (int ii = 0; ii < TT; ++ii) acc[ii] = 0.f;
        if (ok) {
#pragma unroll 1
          for (int kb = 0; kb < DC_KBS; ++kb) {
            const uint8_t* chunk = stage + kb * GU_CHUNK;
            const uint4 cw = *reinterpret_cast<const uint4*>(chunk + (mat ? 2048 : 0) + 16 * row);
            const float d = __half2float(*reinterpret_cast<const __half*>(chunk + 4096 + 4 * row + 2 * mat));
            const Masked m = mask_codes(cw);
#pragma unroll
            for (int ii = 0; ii < TT; ++ii) {
              if (ii < n) {
                const QBlock& a = sqx[kb * TT + ii];
                uint32_t hi[16], lo[16];
                qblock_words(a, hi, lo);
                const int v = dot64(m, hi, lo) - a.qoff;
                acc[ii] = fmaf(d * (a.s64 * tinv[ii]), (float)v, acc[ii]);
              }
            }
          }
        }
        float* pb = reinterpret_cast<float*>(pbuf + (size_t)(u * RT + row) * TT) + mat;
#pragma unroll
        for (int ii = 0; ii < TT; ++ii) pb[2 * ii] = acc[ii];
      } else {
        // down tile rtd: thread = (row, k-half); 5 k-blocks each, halves added in order
        const int rtd = rank + DC_CLUSTER * (u - RT_GU);
        const int row = tid & (RT - 1), kh = tid >> 7;
        float acc[TT];
#pragma unroll
        for (int ii = 0; ii < TT; ++ii) acc[ii] = 0.f;
        if (ok) {
#pragma unroll 1
          for (int k5 = 0; k5 < KB_D / 2; ++k5) {
            const int kb = kh * (KB_D / 2) + k5;
            const uint8_t* chunk = stage + kb * D_CHUNK;
            const uint4 cw = *reinterpret_cast<const uint4*>(chunk + 16 * row);
            const float d = __half2float(*reinterpret_cast<const __half*>(chunk + 2048 + 2 * row));
            const Masked m = mask_codes(cw);
#pragma unroll
            for (int ii = 0; ii < TT; ++ii) {
              if (ii < n) {
                const QBlock& a = hqa[kb * TT + ii];
                uint32_t hi[16], lo[16];
                qblock_words(a, hi, lo);
                const int v = dot64(m, hi, lo) - a.qoff;
                acc[ii] = fmaf(d * a.s64, (float)v, acc[ii]);
              }
            }
          }
        }
        if (kh == 1)
#pragma unroll
          for (int ii = 0; ii < TT; ++ii) s_dn[ii][row] = acc[ii];
        __syncthreads();
        if (kh == 0 && ok)
#pragma unroll
          for (int ii = 0; ii < TT; ++ii)
            if (ii < n) p.parts[(size_t)s_pair[q0 + ii] * H + rtd * RT + row] = acc[ii] + s_dn[ii][row];
        __threadfence();
        __syncthreads();
        if (tid == 0) s_flag = (atomicAdd(&cnt_dn[rtd], 1) == D - 1) ? 1 : 0;
        __syncthreads();
        if (s_flag) {
          // last expert for this output row tile: combine every token in k order (+ residual)
          __threadfence();
          if (tid < RT) {
            const int orow = rtd * RT + tid;
            for (int t = 0; t < T; ++t) {
              float a = 0.f;
#pragma unroll
              for (int k = 0; k < K; ++k) a = fmaf(s_w[t * K + k], __ldcg(p.parts + (size_t)(t * K + k) * H + orow), a);
              p.out[(size_t)t * H + orow] = p.residual ? p.x[(size_t)t * H + orow] + a : a;
            }
          }
          if (tid == 0) cnt_dn[rtd] = 0;
        }
      }
      __syncthreads();  // stage st and s_dn are free again
      if (tid == 0 && u + C::NS < n_units) {
        s_pending[st] = ph[st];
        mbar_expect_tx(&bars[st], DC_UNIT);
        bulk_g2s_stream(ring + (size_t)st * DC_UNIT, unit_src(u + C::NS), DC_UNIT, &bars[st], pol);
      }
      if (u == RT_GU - 1) {
        // all gate/up partials of the cluster are in shared memory: build the owned h blocks
        cluster_sync();
        for (int bi = 0; bi < 2; ++bi) {
          const int b = rank + DC_CLUSTER * bi;  // h block = down k-block b (rows 64b .. 64b + 63)
          if (b >= KB_D) break;
          for (int idx = tid; idx < 64 * n; idx += DC_THREADS) {
            const int r64 = idx & 63, ii = idx >> 6;
            const float2* src = pbuf + (size_t)(64 * b + r64) * TT + ii;
            float g = 0.f, uu = 0.f;
#pragma unroll
            for (int rr = 0; rr < DC_CLUSTER; ++rr) {
              const float2 v = ld_dsmem_f2(dsmem_addr(src, rr));
              g += v.x;
              uu += v.y;
            }
            s_h[ii][r64] = silu_mul(g, uu);
          }
          __syncthreads();
          if (warp < n) quantise_block_warp(s_h[warp][2 * lane], s_h[warp][2 * lane + 1], p.q2_offset,
                                            hql + bi * TT + warp, s_qtmp[warp]);
          __syncthreads();
        }
        cluster_sync();
        // gather the ten h blocks (x tokens) from their owners
        for (int idx = tid; idx < KB_D * TT * 9; idx += DC_THREADS) {
          const int blk = idx / 9, part = idx % 9;
          const int b = blk / TT, ii = blk % TT;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (ii < n) v = ld_dsmem_u4(dsmem_addr(hql + (b / DC_CLUSTER) * TT + ii, b % DC_CLUSTER) + 16 * part);
          reinterpret_cast<uint4*>(hqa + blk)[part] = v;
        }
        __syncthreads();
      }
    }
    // peers may still read this CTA's partials / h blocks: keep them until the whole cluster is done
    cluster_sync();
  }

  // ---- leave: drain copies still in flight (only after a failed wait), last CTA resets counters ----
  __syncthreads();
  if (tid == 0) {
    for (int st = 0; st < C::NS; ++st)
      if (s_pending[st] >= 0) mbar_wait(&bars[st], (uint32_t)s_pending[st], p.status);
    __threadfence();
    s_flag = (atomicAdd(exit_cnt, 1) == G - 1) ? 1 : 0;
  }
  __syncthreads();
  if (s_flag) {
    __threadfence();
    for (int w = tid; w < WS_SYNC_WORDS; w += DC_THREADS)
      if (w != WS_SYNC_EXIT) p.sync[w] = 0;
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      *exit_cnt = 0;
    }
  }
}

int g_clusters[DC_MAX_CLUSTERS][4];  // per device, per TT variant: clusters launched (0 = not queried)

template <int TT>
cudaError_t launch_tt(const DcParams& prm, cudaStream_t s) {
  using C = DcCfg<TT>;
  auto kern = decode_cluster_kernel<TT>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (err != cudaSuccess) return err;
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  const int vi = TT == 1 ? 0 : TT == 2 ? 1 : TT == 4 ? 2 : 3;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = DC_CLUSTER;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeCooperative;
  at[1].val.cooperative = 1;
  cfg.blockDim = dim3(DC_THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cfg.attrs = at;
  int ncl = (dev >= 0 && dev < DC_MAX_CLUSTERS) ? g_clusters[dev][vi] : 0;
  if (ncl == 0) {
    cfg.gridDim = dim3(DC_CLUSTER);
    cfg.numAttrs = 1;
    if ((err = cudaOccupancyMaxActiveClusters(&ncl, (void*)kern, &cfg)) != cudaSuccess) return err;
    if (ncl < 1) return cudaErrorInvalidConfiguration;
    if (ncl > DC_MAX_CLUSTERS) ncl = DC_MAX_CLUSTERS;
    if (dev >= 0 && dev < DC_MAX_CLUSTERS) g_clusters[dev][vi] = ncl;
  }
  cfg.gridDim = dim3(ncl * DC_CLUSTER);
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace

cudaError_t launch_decode_fused(const strata_experts_t& ex, const uint16_t* w_router, const float* bias,
                                const float* x, int T, int residual, float* out, int32_t* ids, float* weights,
                                const WsLayout& L, char* ws, cudaStream_t s) {
  DcParams prm;
  prm.x = x;
  prm.out = out;
  prm.T = T;
  prm.E = ex.n_expert;
  prm.q2_offset = ex.q2_offset;
  prm.residual = residual;
  prm.wr = w_router;
  prm.bias = bias;
  prm.blobs = (const uint8_t*)ex.blobs;
  prm.stride = ex.blob_stride;
  prm.ids_out = ids;
  prm.w_out = weights;
  prm.dots = (float*)(ws + L.dots_rep);
  prm.sumsq = (float*)(ws + L.sumsq);
  prm.qx = (QBlock*)(ws + L.qx);
  prm.parts = (float*)(ws + L.parts);
  prm.sync = (int*)(ws + WS_SYNC);
  prm.status = (int*)(ws + L.status);
  if (T <= 1) return launch_tt<1>(prm, s);
  if (T <= 2) return launch_tt<2>(prm, s);
  if (T <= 4) return launch_tt<4>(prm, s);
  return launch_tt<8>(prm, s);
}

}  // namespace strata
