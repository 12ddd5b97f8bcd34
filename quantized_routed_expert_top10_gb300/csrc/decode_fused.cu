// One-kernel MoE layer for small token counts (decode and verify windows, T <= 8), sm_103a.
//
// The whole layer -- router GEMV (zwxr.cn news/242664, "一次路由的完整旅程": BF16 projection to 512
// logits, softmax, stable descending top-10, clamped renormalisation), grouping of tokens by expert
// (momoyeyu.github.io "ai-infra-strata", "提示词处理": one weight read serves every token routed to an
// expert), the Q2_0 SwiGLU experts (ai.thesatyajit.com "Strata engine", "The CPU kernels": codes
// {0,1,2,3} = {-1,0,1,2} x d with the offset removed once per block) and the weighted combine -- runs
// as one cooperative launch of two 128-thread CTAs per SM:
//   1. every CTA computes a few router rows and quantises a few 64-blocks of x (16-bit integers split
//      into hi/lo bytes, see QBlock) and their sums of squares (for the rmsnorm of residual layers);
//   2. one grid barrier; then every CTA redundantly computes the top-10 of all tokens and the
//      grouping in shared memory (identical results everywhere, no second barrier);
//   3. the expert bytes are cut into equal 23,040-byte units -- gate/up units (expert, 128-row tile,
//      5 of the 40 k-blocks) and down units (expert, 128-row tile, all 10 k-blocks) -- dealt round
//      robin to the CTAs, gate/up units first.  Each CTA streams its units through a ring of shared
//      memory stages with cp.async.bulk (L2 evict-first) as soon as routing is known;
//   4. the last of the 8 CTAs of a gate/up row tile adds the partial sums in split order, applies
//      silu(g) * u, quantises h and bumps the expert's h counter; a down unit waits (bounded) until
//      its expert's five row tiles of h are ready; the last down unit of each output row tile
//      combines the ten weighted expert outputs of every token in k order (+ the residual).
// All waits are bounded by %globaltimer and record STRATA_E_TIMEOUT in the status word.  The last CTA
// to leave resets the counters, so the workspace is ready for the next call.
#include "device_common.cuh"

namespace strata {
namespace {

constexpr int DF_NS = 3;                       // ring stages per CTA
constexpr int DF_UNIT = 23040;                 // bytes per work unit
constexpr int DF_SGU = 8;                      // gate/up k-splits
constexpr int DF_KBU = KB_GU / DF_SGU;         // 5 k-blocks per gate/up unit
constexpr int DF_GU = RT_GU * DF_SGU;          // 40 gate/up units per expert
constexpr int DF_DN = RT_D;                    // 20 down units per expert
constexpr int DF_MAXD = DECODE_T_MAX * K;      // at most 80 distinct experts
constexpr int DF_THREADS = 128;
static_assert(DF_KBU * GU_CHUNK == DF_UNIT && KB_D * D_CHUNK == DF_UNIT, "equal unit sizes");

struct DecodeParams {
  const float* x;  // [T][H] layer input (may alias out)
  float* out;      // [T][H]
  int T, E, q2_offset, residual;
  const uint16_t* wr;  // [E][H] bf16
  const float* bias;   // [E] or null
  const uint8_t* blobs;
  int64_t stride;
  int32_t* ids_out;  // [T][K]
  float* w_out;      // [T][K]
  float* dots;       // ws [WS_NREP][T][EMAX] raw router dot products, replicated
  float* sumsq;      // ws [WS_NREP][T][KB_GU], replicated
  QBlock* qx;        // ws [T][KB_GU]
  QBlock* hq;        // ws [T*K][KB_D]
  float* partial;    // ws [RT_GU*DF_SGU][T*K][RT] float2
  float* parts;      // ws [T*K][H]
  int* sync;         // ws sync words (WS_SYNC)
  int* status;
};

__device__ __forceinline__ void unpack_words(const QBlock& a, uint32_t* hi, uint32_t* lo) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint4 h4 = reinterpret_cast<const uint4*>(a.hi)[w];
    const uint4 l4 = reinterpret_cast<const uint4*>(a.lo)[w];
    hi[4 * w] = h4.x; hi[4 * w + 1] = h4.y; hi[4 * w + 2] = h4.z; hi[4 * w + 3] = h4.w;
    lo[4 * w] = l4.x; lo[4 * w + 1] = l4.y; lo[4 * w + 2] = l4.z; lo[4 * w + 3] = l4.w;
  }
}

template <int TT>
__global__ void __launch_bounds__(DF_THREADS, 2) decode_layer_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;                                            // DF_NS * DF_UNIT
  QBlock* sq = reinterpret_cast<QBlock*>(smem + DF_NS * DF_UNIT);  // [KB_D][TT]
  __shared__ uint64_t bars[DF_NS];
  __shared__ int s_pending[DF_NS];
  __shared__ float s_inv[TT];
  __shared__ int s_ids[TT * K];
  __shared__ float s_w[TT * K];
  __shared__ int s_te[DF_MAXD];   // expert slot j -> expert id
  __shared__ int s_tn[DF_MAXD];   //               -> tokens routed to it
  __shared__ int s_tq[DF_MAXD];   //               -> first slot in s_pair
  __shared__ int s_first[TT * K];
  __shared__ int s_pair[TT * K];
  __shared__ float s_rpart[4][TT];
  __shared__ float s_bias[EMAX];
  __shared__ int32_t s_qtmp[4][64];
  __shared__ float s_h[TT][RT];
  __shared__ int s_flag, s_ok, s_nact;

  const int G = gridDim.x, c = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T, E = p.E, P = T * K;
  int* bar = p.sync + WS_SYNC_BAR;
  int* exit_cnt = p.sync + WS_SYNC_EXIT;
  int* cnt_gu = p.sync + WS_SYNC_CNT_GU;
  int* h_ready = p.sync + WS_SYNC_HREADY;
  int* cnt_dn = p.sync + WS_SYNC_CNT_DN;

  if (tid == 0) {
    for (int s = 0; s < DF_NS; ++s) {
      mbar_init(&bars[s], 1);
      s_pending[s] = -1;
    }
    fence_mbar_init();
    s_ok = 1;
  }
  for (int e = tid; e < E; e += DF_THREADS) s_bias[e] = p.bias ? __ldg(p.bias + e) : 0.f;

  // ---- 1. router dot products (two warps per row), x quantisation, block sums of squares ----
  for (int e0 = c; e0 < E; e0 += 2 * G) {
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
            float sacc = acc[t];
            sacc = fmaf(wf[0], a4.x, sacc); sacc = fmaf(wf[1], a4.y, sacc);
            sacc = fmaf(wf[2], a4.z, sacc); sacc = fmaf(wf[3], a4.w, sacc);
            sacc = fmaf(wf[4], b4.x, sacc); sacc = fmaf(wf[5], b4.y, sacc);
            sacc = fmaf(wf[6], b4.z, sacc); sacc = fmaf(wf[7], b4.w, sacc);
            acc[t] = sacc;
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
    if (tid < 2 * TT) {
      const int w2 = tid / TT, t = tid % TT;
      const int e2 = e0 + G * w2;
      if (e2 < E && t < T) {
        const float v = s_rpart[2 * w2][t] + s_rpart[2 * w2 + 1][t];
#pragma unroll
        for (int r = 0; r < WS_NREP; ++r) p.dots[((size_t)r * T + t) * EMAX + e2] = v;
      }
    }
    __syncthreads();
  }
  for (int b = c + G * warp; b < T * KB_GU; b += 4 * G) {
    const int t = b / KB_GU, kb = b % KB_GU;
    const float2 v = __ldg(reinterpret_cast<const float2*>(p.x + (size_t)t * H + kb * QK + 2 * lane));
    const float ss = warp_sum(v.x * v.x + v.y * v.y);
    if (lane == 0)
#pragma unroll
      for (int r = 0; r < WS_NREP; ++r) p.sumsq[(size_t)r * T * KB_GU + b] = ss;
    quantise_block_warp(v.x, v.y, p.q2_offset, p.qx + b, s_qtmp[warp]);
  }

  // ---- grid barrier ----
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(bar, 1) == G - 1) {
      __threadfence();  // release: every CTA's phase-1 writes happen before any flag is seen
#pragma unroll
      for (int r = 0; r < WS_NREP; ++r) st_relaxed(p.sync + WS_SYNC_REL + 32 * r, 1);
    }
    s_ok = spin_until_geq(p.sync + WS_SYNC_REL + 32 * (c % WS_NREP), 1, p.status) ? 1 : 0;
  }
  __syncthreads();

  // ---- 2. top-10 and grouping, redundantly in every CTA ----
  if (s_ok) {
    if (tid < T) {
      float inv = 1.f;
      if (p.residual) {
        float s = 0.f;
        const float* ssq = p.sumsq + ((size_t)(c % WS_NREP) * T + tid) * KB_GU;
        for (int kb = 0; kb < KB_GU; ++kb) s += __ldcg(ssq + kb);
        inv = 1.f / sqrtf(s / (float)H + 1e-6f);
      }
      s_inv[tid] = inv;
    }
    if (tid == 0) s_nact = 0;
    __syncthreads();
    for (int t = warp; t < T; t += 4) {
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
    // grouping of the P <= 80 pairs, directly on the pairs: slot of pair q = (pairs with a smaller
    // expert id) + (earlier pairs with the same expert); expert slot j = (distinct smaller ids).
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
      for (int q = tid; q < P; q += DF_THREADS) {
        p.ids_out[q] = s_ids[q];
        p.w_out[q] = s_w[q];
      }
    __syncthreads();
  }

  // ---- 3-4. expert units ----
  if (s_ok) {
    const int D = s_nact;
    const int n_gu = D * DF_GU, n_units = D * (DF_GU + DF_DN);
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int u, int i) {  // thread 0 only: unit u into stage i % DF_NS
      const int st = i % DF_NS;
      const uint8_t* src;
      if (u < n_gu) {
        const int j = u / DF_GU, r = u % DF_GU;
        const int rt = r / DF_SGU, s = r % DF_SGU;
        src = p.blobs + (int64_t)s_te[j] * p.stride + ((int64_t)rt * KB_GU + s * DF_KBU) * GU_CHUNK;
      } else {
        const int v = u - n_gu;
        const int j = v / DF_DN, rtd = v % DF_DN;
        src = p.blobs + (int64_t)s_te[j] * p.stride + D_REGION + (int64_t)rtd * KB_D * D_CHUNK;
      }
      s_pending[st] = (i / DF_NS) & 1;
      mbar_expect_tx(&bars[st], DF_UNIT);
      bulk_g2s_stream(ring + (size_t)st * DF_UNIT, src, DF_UNIT, &bars[st], pol);
    };
    if (tid == 0)
      for (int i = 0; i < DF_NS; ++i)
        if (c + G * i < n_units) issue(c + G * i, i);

    int i = 0;
    for (int u = c; u < n_units; u += G, ++i) {
      const int st = i % DF_NS;
      const uint32_t par = (uint32_t)((i / DF_NS) & 1);
      const uint8_t* stage = ring + (size_t)st * DF_UNIT;
      if (u < n_gu) {
        // -------- gate/up unit --------
        const int j = u / DF_GU, r = u % DF_GU;
        const int rt = r / DF_SGU, s = r % DF_SGU;
        const int n = s_tn[j], q0 = s_tq[j];
        for (int idx = tid; idx < DF_KBU * TT * 9; idx += DF_THREADS) {
          const int blk = idx / 9, part = idx % 9;
          const int kb = blk / TT, ii = blk % TT;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (ii < n) {
            const int t = s_pair[q0 + ii] / K;
            v = __ldcg(reinterpret_cast<const uint4*>(p.qx + (size_t)t * KB_GU + s * DF_KBU + kb) + part);
          }
          reinterpret_cast<uint4*>(sq + blk)[part] = v;
        }
        if (!__syncthreads_and(mbar_wait(&bars[st], par, p.status) ? 1 : 0)) {
          if (tid == 0) s_ok = 0;
          __syncthreads();
          break;
        }
        if (tid == 0) s_pending[st] = -1;
        float tinv[TT];
#pragma unroll
        for (int ii = 0; ii < TT; ++ii) tinv[ii] = (ii < n) ? s_inv[s_pair[q0 + ii] / K] : 0.f;
        float accg[TT], accu[TT];
#pragma unroll
        for (int ii = 0; ii < TT; ++ii) { accg[ii] = 0.f; accu[ii] = 0.f; }
#pragma unroll 1
        for (int kb = 0; kb < DF_KBU; ++kb) {
          const uint8_t* chunk = stage + kb * GU_CHUNK;
          const uint4 gc = *reinterpret_cast<const uint4*>(chunk + 16 * tid);
          const uint4 uc = *reinterpret_cast<const uint4*>(chunk + 2048 + 16 * tid);
          const __half2 sc = *reinterpret_cast<const __half2*>(chunk + 4096 + 4 * tid);
          const float dg = __low2float(sc), du = __high2float(sc);
          const Masked gm = mask_codes(gc), um = mask_codes(uc);
#pragma unroll
          for (int ii = 0; ii < TT; ++ii) {
            if (ii < n) {
              const QBlock& a = sq[kb * TT + ii];
              uint32_t hi[16], lo[16];
              unpack_words(a, hi, lo);
              const float f = a.s64 * tinv[ii];
              const int vg = dot64(gm, hi, lo) - a.qoff;
              const int vu = dot64(um, hi, lo) - a.qoff;
              accg[ii] = fmaf(dg * f, (float)vg, accg[ii]);
              accu[ii] = fmaf(du * f, (float)vu, accu[ii]);
            }
          }
        }
        float2* part = reinterpret_cast<float2*>(p.partial);
#pragma unroll
        for (int ii = 0; ii < TT; ++ii)
          if (ii < n) part[((size_t)(rt * DF_SGU + s) * P + q0 + ii) * RT + tid] = make_float2(accg[ii], accu[ii]);
        __threadfence();
        __syncthreads();
        if (tid == 0) s_flag = (atomicAdd(&cnt_gu[j * RT_GU + rt], 1) == DF_SGU - 1) ? 1 : 0;
        __syncthreads();
        if (s_flag) {
          __threadfence();
#pragma unroll
          for (int ii = 0; ii < TT; ++ii) {
            if (ii < n) {
              float g = 0.f, uu = 0.f;
              for (int ss = 0; ss < DF_SGU; ++ss) {
                const float2 v = __ldcg(part + ((size_t)(rt * DF_SGU + ss) * P + q0 + ii) * RT + tid);
                g += v.x;
                uu += v.y;
              }
              s_h[ii][tid] = silu_mul(g, uu);
            }
          }
          if (tid == 0) cnt_gu[j * RT_GU + rt] = 0;
          __syncthreads();
          for (int item = warp; item < 2 * n; item += 4) {
            const int ii = item >> 1, b = item & 1;
            quantise_block_warp(s_h[ii][64 * b + 2 * lane], s_h[ii][64 * b + 2 * lane + 1], p.q2_offset,
                                p.hq + (size_t)(q0 + ii) * KB_D + 2 * rt + b, s_qtmp[warp]);
          }
          __threadfence();
          __syncthreads();
          if (tid == 0) atomicAdd(&h_ready[j], 1);
        }
      } else {
        // -------- down unit --------
        const int v = u - n_gu;
        const int j = v / DF_DN, rtd = v % DF_DN;
        const int n = s_tn[j], q0 = s_tq[j];
        if (tid == 0) s_flag = spin_until_geq(&h_ready[j], RT_GU, p.status) ? 1 : 0;
        __syncthreads();
        if (!s_flag) { if (tid == 0) s_ok = 0; __syncthreads(); break; }
        for (int idx = tid; idx < KB_D * TT * 9; idx += DF_THREADS) {
          const int blk = idx / 9, part = idx % 9;
          const int kb = blk / TT, ii = blk % TT;
          uint4 w4 = make_uint4(0, 0, 0, 0);
          if (ii < n) w4 = __ldcg(reinterpret_cast<const uint4*>(p.hq + (size_t)(q0 + ii) * KB_D + kb) + part);
          reinterpret_cast<uint4*>(sq + blk)[part] = w4;
        }
        if (!__syncthreads_and(mbar_wait(&bars[st], par, p.status) ? 1 : 0)) {
          if (tid == 0) s_ok = 0;
          __syncthreads();
          break;
        }
        if (tid == 0) s_pending[st] = -1;
        float acc[TT];
#pragma unroll
        for (int ii = 0; ii < TT; ++ii) acc[ii] = 0.f;
#pragma unroll 1
        for (int kb = 0; kb < KB_D; ++kb) {
          const uint8_t* chunk = stage + kb * D_CHUNK;
          const uint4 cw = *reinterpret_cast<const uint4*>(chunk + 16 * tid);
          const float d = __half2float(*reinterpret_cast<const __half*>(chunk + 2048 + 2 * tid));
          const Masked m = mask_codes(cw);
#pragma unroll
          for (int ii = 0; ii < TT; ++ii) {
            if (ii < n) {
              const QBlock& a = sq[kb * TT + ii];
              uint32_t hi[16], lo[16];
              unpack_words(a, hi, lo);
              const int vv = dot64(m, hi, lo) - a.qoff;
              acc[ii] = fmaf(d * a.s64, (float)vv, acc[ii]);
            }
          }
        }
        const int row = rtd * RT + tid;
#pragma unroll
        for (int ii = 0; ii < TT; ++ii)
          if (ii < n) p.parts[(size_t)s_pair[q0 + ii] * H + row] = acc[ii];
        __threadfence();
        __syncthreads();
        if (tid == 0) s_flag = (atomicAdd(&cnt_dn[rtd], 1) == D - 1) ? 1 : 0;
        __syncthreads();
        if (s_flag) {
          __threadfence();
          for (int t = 0; t < T; ++t) {
            float a = 0.f;
#pragma unroll
            for (int k = 0; k < K; ++k) a = fmaf(s_w[t * K + k], __ldcg(p.parts + (size_t)(t * K + k) * H + row), a);
            p.out[(size_t)t * H + row] = p.residual ? p.x[(size_t)t * H + row] + a : a;
          }
          if (tid == 0) cnt_dn[rtd] = 0;
        }
      }
      __syncthreads();  // everyone is done with this stage and with sq
      if (tid == 0 && u + G * DF_NS < n_units) issue(u + G * DF_NS, i + DF_NS);
    }
  }

  // ---- leave: drain copies still in flight (only after a failed wait), last CTA resets counters ----
  __syncthreads();
  if (tid == 0) {
    for (int st = 0; st < DF_NS; ++st)
      if (s_pending[st] >= 0) mbar_wait(&bars[st], (uint32_t)s_pending[st], p.status);
    __threadfence();
    s_flag = (atomicAdd(exit_cnt, 1) == G - 1) ? 1 : 0;
  }
  __syncthreads();
  if (s_flag) {
    __threadfence();
    for (int w = tid; w < WS_SYNC_WORDS; w += DF_THREADS)
      if (w != WS_SYNC_EXIT) p.sync[w] = 0;
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      *exit_cnt = 0;
    }
  }
}

struct DeviceLaunchInfo {
  int grid[4] = {0, 0, 0, 0};  // per TT variant
};
DeviceLaunchInfo g_info[64];

template <int TT>
cudaError_t launch_tt(const DecodeParams& prm, cudaStream_t s) {
  const size_t smem = (size_t)DF_NS * DF_UNIT + sizeof(QBlock) * KB_D * TT;
  auto kern = decode_layer_kernel<TT>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  const int vi = TT == 1 ? 0 : TT == 2 ? 1 : TT == 4 ? 2 : 3;
  int grid = (dev >= 0 && dev < 64) ? g_info[dev].grid[vi] : 0;
  if (grid == 0) {
    int sms = 0, per_sm = 0;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, DF_THREADS, smem)) != cudaSuccess)
      return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    grid = sms * (per_sm < 2 ? per_sm : 2);
    if (dev >= 0 && dev < 64) g_info[dev].grid[vi] = grid;
  }
  void* args[] = {(void*)&prm};
  STRATA_LAUNCH(KID_DECODE_LAYER, s,
                err = cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(DF_THREADS), args, smem, s));
  return err;
}

}  // namespace

cudaError_t launch_decode_fused(const strata_experts_t& ex, const uint16_t* w_router, const float* bias,
                                const float* x, int T, int residual, float* out, int32_t* ids, float* weights,
                                const WsLayout& L, char* ws, cudaStream_t s) {
  DecodeParams prm;
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
  prm.hq = (QBlock*)(ws + L.hq);
  prm.partial = (float*)(ws + L.partial);
  prm.parts = (float*)(ws + L.parts);
  prm.sync = (int*)(ws + WS_SYNC);
  prm.status = (int*)(ws + L.status);
  if (T <= 1) return launch_tt<1>(prm, s);
  if (T <= 2) return launch_tt<2>(prm, s);
  if (T <= 4) return launch_tt<4>(prm, s);
  return launch_tt<8>(prm, s);
}

}  // namespace strata
