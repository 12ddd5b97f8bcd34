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
//   3. right after the barrier each CTA copies every token's quantised activations into shared
//      memory (one bulk copy, overlapping the top-k); the expert bytes are cut into equal
//      23,040-byte units -- gate/up units (expert, slab of 16 rows, all 40 k-blocks: contiguous in
//      the packed blob) and down units (expert, 128-row tile, all 10 k-blocks) -- dealt round robin
//      to the CTAs, gate/up units first.  Each CTA streams its units through a ring of shared memory
//      stages with cp.async.bulk (L2 evict-first) as soon as routing is known;
//   4. a gate/up unit finishes g and u of its 16 rows for the expert's tokens (8 thread groups of 5
//      k-blocks, added in group order), writes h = silu(g) * u and bumps the expert's h counter; a
//      down unit waits (bounded) until all 40 slabs of its expert are in, quantises h itself, and the
//      last down unit of each output row tile combines the ten weighted expert outputs of every
//      token in k order (+ the residual).
// All waits are bounded by %globaltimer and record STRATA_E_TIMEOUT in the status word.  The last CTA
// to leave resets the counters, so the workspace is ready for the next call.
#include "device_common.cuh"

namespace strata {
namespace {

constexpr int DF_UNIT = 23040;                 // bytes per work unit
constexpr int DF_GU = N_SLAB;                  // 40 gate/up units (slabs) per expert
constexpr int DF_DN = RT_D;                    // 20 down units per expert
constexpr int DF_MAXD = DECODE_T_MAX * K;      // at most 80 distinct experts
constexpr int DF_THREADS = 128;
constexpr int DF_KG = DF_THREADS / SLAB;       // 8 k-block groups per gate/up unit
constexpr int DF_KBG = KB_GU / DF_KG;          // 5 k-blocks per group
static_assert(SLAB_BYTES == DF_UNIT && KB_D * D_CHUNK == DF_UNIT, "equal unit sizes");
// Ring stages per CTA: three, or two when eight tokens' activations take the shared memory.
template <int TT>
__host__ __device__ constexpr int df_stages() { return TT <= 4 ? 3 : 2; }
template <int TT>
constexpr size_t df_smem() {
  return (size_t)df_stages<TT>() * DF_UNIT + sizeof(QBlock) * (size_t)(TT * KB_GU + KB_D * TT);
}

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
  float* hf;         // ws [T*K][FF] h of each pair, in slot order
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

// ---- two or more tokens: warp-level tensor-core products (mma.sync m16n8k16, fp16 x fp16 -> fp32) ----
// Weights are the A operand (16 rows x 16 k), the tokens (or an expert's pairs) the 8 columns of B.
// Within a 64-block the k order is free as long as A and B agree: k-step s of thread (g, t) -- g =
// lane / 4 owns rows g, g + 8 and column g, t = lane % 4 -- takes half2 number 2s (k = 2t, 2t + 1) and
// 2s + 1 (k = 2t + 8, 2t + 9) of code word t of its rows, where half2 number q = 4b + m holds field m of
// code bytes b and b + 2 (weights 16t + 4b + m and 16t + 8 + 4b + m).  Activations are stored once in
// that order ("fragment order": per (k-block, t, column) 16 halves, pair q at halves 2q, 2q + 1), so a
// thread's B operand for a whole k-block is two 16-byte loads.  A holds code - q2_offset exactly (the
// LOP3 / HSUB2 construction of the tensor-core prefill path); the scale d of each (row, k-block) is
// applied to the k-block's fp32 partial products.
__device__ __forceinline__ void mma_16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The 8 half2 (code - q2_offset) of one 16-code word, in half2 order q = 4b + m.
__device__ __forceinline__ void codes_to_half2(uint32_t word, const uint32_t* sub, uint32_t* h) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int b = q >> 2, m = q & 3;
    const uint32_t src = b ? (word >> 8) : word;
    const uint32_t bits = (src & (0x00030003u << (2 * m))) | ((uint32_t)((25 - 2 * m) << 10) * 0x00010001u);
    const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&bits), *reinterpret_cast<const __half2*>(&sub[m]));
    h[q] = *reinterpret_cast<const uint32_t*>(&v);
  }
}

// 16 consecutive values v[0..15] of a block (weights 16t ..) as the 8 fragment-order half2.
__device__ __forceinline__ void to_fragment_order(const float* v, uint32_t* h) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int b = q >> 2, m = q & 3;
    const __half2 x2 = __floats2half2_rn(v[4 * b + m], v[8 + 4 * b + m]);
    h[q] = *reinterpret_cast<const uint32_t*>(&x2);
  }
}

template <int TT>
__global__ void __launch_bounds__(DF_THREADS, 2) decode_layer_kernel(const DecodeParams p) {
  constexpr bool MMA = TT >= 2;  // one token: dp4a on the codes; more: tensor-core products
  constexpr int NS = df_stages<TT>();
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;                                                 // NS * DF_UNIT
  QBlock* sqx = reinterpret_cast<QBlock*>(smem + NS * DF_UNIT);         // [T][KB_GU] all tokens
  QBlock* sq = sqx + TT * KB_GU;                                        // [KB_D][TT] h of a down unit
  float2* red = reinterpret_cast<float2*>(sq);                          // [DF_KG][TT][SLAB] (gate/up)
  static_assert(sizeof(float2) * DF_KG * TT * SLAB <= sizeof(QBlock) * KB_D * TT, "reduction fits");
  __shared__ uint64_t bars[NS];
  __shared__ uint64_t bar_qx, bar_h;
  __shared__ int s_pending[NS];
  __shared__ int s_qx_pending, s_h_pending;
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
  __shared__ TopKScratch s_topk[DF_THREADS / 32];
  __shared__ int32_t s_qtmp[4][64];
  __shared__ int s_flag, s_ok, s_nact;

  const int G = gridDim.x, c = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T, E = p.E, P = T * K;
  int* exit_cnt = p.sync + WS_SYNC_EXIT;
  int* h_cnt = p.sync + WS_SYNC_HREADY;  // expert slot j at h_cnt[WS_SYNC_STRIDE * j]
  int* cnt_dn = p.sync + WS_SYNC_CNT_DN;  // row tile r at cnt_dn[WS_SYNC_STRIDE * r]

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars[s], 1);
      s_pending[s] = -1;
    }
    mbar_init(&bar_qx, 1);
    mbar_init(&bar_h, 1);
    s_qx_pending = 0;
    s_h_pending = -1;
    fence_mbar_init();
    s_ok = 1;
  }
  // loads for later steps, issued first so their latency hides under the router rows': the bias
  // (used by the top-k) and this warp's first block of x to quantise
  float bias_v[EMAX / DF_THREADS];
#pragma unroll
  for (int i = 0; i < EMAX / DF_THREADS; ++i) {
    const int e = tid + DF_THREADS * i;
    bias_v[i] = (p.bias && e < E) ? __ldg(p.bias + e) : 0.f;
  }
  const int t4x = lane >> 3, qx8 = lane & 7;  // fragment-order position of this lane's x pair (T >= 2)
  auto load_block = [&](int b, float2& v, float& xa, float& xb) {
    const int t = b / KB_GU, kb = b % KB_GU;
    v = __ldg(reinterpret_cast<const float2*>(p.x + (size_t)t * H + kb * QK + 2 * lane));
    if constexpr (MMA) {
      const float* src = p.x + (size_t)t * H + kb * QK + 16 * t4x + 4 * (qx8 >> 2) + (qx8 & 3);
      xa = __ldg(src);
      xb = __ldg(src + 8);
    }
  };
  float2 v0 = make_float2(0.f, 0.f);
  float xa0 = 0.f, xb0 = 0.f;
  if (c + G * warp < T * KB_GU) load_block(c + G * warp, v0, xa0, xb0);

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
    float2 v = v0;
    float xa = xa0, xb = xb0;
    if (b != c + G * warp) load_block(b, v, xa, xb);
    const float ss = warp_sum(v.x * v.x + v.y * v.y);
    if (lane == 0)
#pragma unroll
      for (int r = 0; r < WS_NREP; ++r) p.sumsq[(size_t)r * T * KB_GU + b] = ss;
    if constexpr (MMA) {  // fp16 x in fragment order: xs[kb][t4][token][16 halves]
      const __half2 x2 = __floats2half2_rn(xa, xb);
      reinterpret_cast<__half2*>(reinterpret_cast<uint8_t*>(p.qx) + ((size_t)(kb * 4 + t4x) * T + t) * 32)[qx8] = x2;
    } else {
      quantise_block_warp(v.x, v.y, p.q2_offset, p.qx + b, s_qtmp[warp]);
    }
  }

#pragma unroll
  for (int i = 0; i < EMAX / DF_THREADS; ++i)
    if (tid + DF_THREADS * i < E) s_bias[tid + DF_THREADS * i] = bias_v[i];

  // ---- grid barrier: each CTA makes its writes visible and counts into one of WS_NARR counters
  // (release add, no reply awaited), then polls all of them ----
  __syncthreads();
  if (tid == 0) {
    red_release_add(p.sync + WS_SYNC_ARR + 32 * (c % WS_NARR), 1);
    s_ok = spin_grid_arrivals<WS_NARR>(p.sync + WS_SYNC_ARR, 32, G, p.status) ? 1 : 0;
    if (s_ok) {
      // every token's quantised activations (written by all CTAs before the barrier) into shared
      // memory; the async-proxy copy is ordered after the acquire by the proxy fence
      fence_proxy_async_global();
      const uint32_t xbytes = MMA ? (uint32_t)(KB_GU * 4 * 32 * T) : (uint32_t)(sizeof(QBlock) * T * KB_GU);
      mbar_expect_tx(&bar_qx, xbytes);
      bulk_g2s(sqx, p.qx, xbytes, &bar_qx);
      s_qx_pending = 1;
    }
  }
  __syncthreads();

  // ---- 2. top-10 and grouping, redundantly in every CTA ----
  if (s_ok) {
    if (tid == 0) s_nact = 0;
    for (int t = warp; t < T; t += 4) {
      const float* d = p.dots + ((size_t)(c % WS_NREP) * T + t) * EMAX;
      float lg[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) lg[j] = (lane + 32 * j < E) ? __ldcg(d + lane + 32 * j) : 0.f;
      float inv = 1.f;  // rmsnorm of a residual layer: 1 / rms from the 40 block sums of squares
      if (p.residual) {
        const float* ssq = p.sumsq + ((size_t)(c % WS_NREP) * T + t) * KB_GU;
        float s = __ldcg(ssq + lane);
        if (lane + 32 < KB_GU) s += __ldcg(ssq + lane + 32);
        inv = 1.f / sqrtf(warp_sum(s) / (float)H + 1e-6f);
      }
      if (lane == 0) s_inv[t] = inv;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (lane + 32 * j < E) lg[j] = lg[j] * inv + s_bias[lane + 32 * j];
      int id;
      float w;
      top_k_warp_fn([&](int e) { return lg[e >> 5]; }, E, s_topk[warp], &id, &w);
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
    auto issue = [&](int u, int i) {  // thread 0 only: unit u into stage i % NS
      const int st = i % NS;
      const uint8_t* src;
      if (u < n_gu) {
        const int j = u / DF_GU, sl = u % DF_GU;
        src = p.blobs + (int64_t)s_te[j] * p.stride + (int64_t)sl * SLAB_BYTES;
      } else {
        const int v = u - n_gu;
        const int j = v / DF_DN, rtd = v % DF_DN;
        src = p.blobs + (int64_t)s_te[j] * p.stride + D_REGION + (int64_t)rtd * KB_D * D_CHUNK;
      }
      s_pending[st] = (i / NS) & 1;
      mbar_expect_tx(&bars[st], DF_UNIT);
      bulk_g2s_stream(ring + (size_t)st * DF_UNIT, src, DF_UNIT, &bars[st], pol);
    };
    if (tid == 0)
      for (int i = 0; i < NS; ++i)
        if (c + G * i < n_units) issue(c + G * i, i);

    int i = 0, n_dn = 0;
    for (int u = c; u < n_units; u += G, ++i) {
      const int st = i % NS;
      const uint32_t par = (uint32_t)((i / NS) & 1);
      const uint8_t* stage = ring + (size_t)st * DF_UNIT;
      if (u < n_gu) {
        // -------- gate/up unit: slab sl (rows 16 sl ..) of expert slot j, all k-blocks --------
        const int j = u / DF_GU, sl = u % DF_GU;
        const int n = s_tn[j], q0 = s_tq[j];
        bool ready = mbar_wait(&bars[st], par, p.status);
        if (s_qx_pending) ready = mbar_wait(&bar_qx, 0u, p.status) && ready;
        if (!__syncthreads_and(ready ? 1 : 0)) {
          if (tid == 0) s_ok = 0;
          __syncthreads();
          break;
        }
        if (tid == 0) {
          s_pending[st] = -1;
          s_qx_pending = 0;
        }
        if constexpr (MMA) {
          // warp w: k-blocks [10 w, 10 w + 10) of the 16-row slab, all T tokens as columns
          const int g = lane >> 2, t4 = lane & 3;
          uint32_t subq[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const __half2 s2 = __half2half2(__float2half_rn((float)((1024 >> (2 * m)) + p.q2_offset)));
            subq[m] = *reinterpret_cast<const uint32_t*>(&s2);
          }
          const uint8_t* xs = reinterpret_cast<const uint8_t*>(sqx);
          float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
          for (int kk = 0; kk < KB_GU / 4; ++kk) {
            const int kb = warp * (KB_GU / 4) + kk;
            const uint8_t* piece = stage + kb * SLAB_KB;
            const uint32_t wg0 = *reinterpret_cast<const uint32_t*>(piece + 16 * g + 4 * t4);
            const uint32_t wg1 = *reinterpret_cast<const uint32_t*>(piece + 16 * (g + 8) + 4 * t4);
            const uint32_t wu0 = *reinterpret_cast<const uint32_t*>(piece + 256 + 16 * g + 4 * t4);
            const uint32_t wu1 = *reinterpret_cast<const uint32_t*>(piece + 256 + 16 * (g + 8) + 4 * t4);
            const __half2 sc0 = *reinterpret_cast<const __half2*>(piece + 512 + 4 * g);
            const __half2 sc1 = *reinterpret_cast<const __half2*>(piece + 512 + 4 * (g + 8));
            uint4 x0 = make_uint4(0, 0, 0, 0), x1 = make_uint4(0, 0, 0, 0);
            if (g < T) {
              const uint4* xp = reinterpret_cast<const uint4*>(xs + ((size_t)(kb * 4 + t4) * T + g) * 32);
              x0 = xp[0];
              x1 = xp[1];
            }
            const uint32_t bq[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            uint32_t hg0[8], hg1[8], hu0[8], hu1[8];
            codes_to_half2(wg0, subq, hg0);
            codes_to_half2(wg1, subq, hg1);
            codes_to_half2(wu0, subq, hu0);
            codes_to_half2(wu1, subq, hu1);
            // even and odd k-steps into separate accumulators: two independent MMA chains per matrix
            float cg[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            float cu[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              const uint32_t a_g[4] = {hg0[2 * s], hg1[2 * s], hg0[2 * s + 1], hg1[2 * s + 1]};
              const uint32_t a_u[4] = {hu0[2 * s], hu1[2 * s], hu0[2 * s + 1], hu1[2 * s + 1]};
              mma_16816(cg[s & 1], a_g, bq[2 * s], bq[2 * s + 1]);
              mma_16816(cu[s & 1], a_u, bq[2 * s], bq[2 * s + 1]);
            }
            const float dg0 = __low2float(sc0), du0 = __high2float(sc0);
            const float dg1 = __low2float(sc1), du1 = __high2float(sc1);
            ag[0] = fmaf(dg0, cg[0][0] + cg[1][0], ag[0]); ag[1] = fmaf(dg0, cg[0][1] + cg[1][1], ag[1]);
            ag[2] = fmaf(dg1, cg[0][2] + cg[1][2], ag[2]); ag[3] = fmaf(dg1, cg[0][3] + cg[1][3], ag[3]);
            au[0] = fmaf(du0, cu[0][0] + cu[1][0], au[0]); au[1] = fmaf(du0, cu[0][1] + cu[1][1], au[1]);
            au[2] = fmaf(du1, cu[0][2] + cu[1][2], au[2]); au[3] = fmaf(du1, cu[0][3] + cu[1][3], au[3]);
          }
          // red[warp][mat][row][column]: the four warps' k ranges, added below in warp order
          float* rf = reinterpret_cast<float*>(red);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = g + 8 * (e >> 1), col = 2 * t4 + (e & 1);
            if (col < TT) {
              rf[((warp * 2 + 0) * SLAB + row) * TT + col] = ag[e];
              rf[((warp * 2 + 1) * SLAB + row) * TT + col] = au[e];
            }
          }
          __syncthreads();
          if (tid < SLAB * n) {
            const int r2 = tid % SLAB, ii = tid / SLAB;
            const int tk = s_pair[q0 + ii] / K;
            float gg = 0.f, uu = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              gg += rf[((w * 2 + 0) * SLAB + r2) * TT + tk];
              uu += rf[((w * 2 + 1) * SLAB + r2) * TT + tk];
            }
            const float inv = s_inv[tk];
            p.hf[(size_t)(q0 + ii) * FF + sl * SLAB + r2] = silu_mul(gg * inv, uu * inv);
          }
        } else {
        const int r = tid % SLAB, grp = tid / SLAB;  // row of the slab, group of DF_KBG k-blocks
        int tok[TT];
        float tinv[TT];
#pragma unroll
        for (int ii = 0; ii < TT; ++ii) {
          tok[ii] = (ii < n) ? s_pair[q0 + ii] / K : 0;
          tinv[ii] = (ii < n) ? s_inv[tok[ii]] : 0.f;
        }
        float accg[TT], accu[TT];
#pragma unroll
        for (int ii = 0; ii < TT; ++ii) { accg[ii] = 0.f; accu[ii] = 0.f; }
#pragma unroll 1
        for (int kk = 0; kk < DF_KBG; ++kk) {
          const int kb = grp * DF_KBG + kk;
          const uint8_t* piece = stage + kb * SLAB_KB;
          const uint4 gc = *reinterpret_cast<const uint4*>(piece + 16 * r);
          const uint4 uc = *reinterpret_cast<const uint4*>(piece + 256 + 16 * r);
          const __half2 sc = *reinterpret_cast<const __half2*>(piece + 512 + 4 * r);
          const float dg = __low2float(sc), du = __high2float(sc);
          const Masked gm = mask_codes(gc), um = mask_codes(uc);
#pragma unroll
          for (int ii = 0; ii < TT; ++ii) {
            if (ii < n) {
              const QBlock& a = sqx[tok[ii] * KB_GU + kb];
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
#pragma unroll
        for (int ii = 0; ii < TT; ++ii)
          if (ii < n) red[(grp * TT + ii) * SLAB + r] = make_float2(accg[ii], accu[ii]);
        __syncthreads();
        if (tid < SLAB * n) {  // (row, token): the 8 groups added in group order
          const int r2 = tid % SLAB, ii = tid / SLAB;
          float g = 0.f, uu = 0.f;
#pragma unroll
          for (int q = 0; q < DF_KG; ++q) {
            const float2 v = red[(q * TT + ii) * SLAB + r2];
            g += v.x;
            uu += v.y;
          }
          p.hf[(size_t)(q0 + ii) * FF + sl * SLAB + r2] = silu_mul(g, uu);
        }
        }
        __syncthreads();  // every h store issued; the stage and the reduction buffer are free
        if (tid == 0) {
          red_release_add(&h_cnt[WS_SYNC_STRIDE * j], 1);
          if (u + G * NS < n_units) issue(u + G * NS, i + NS);
        }
        continue;
      } else {
        // -------- down unit: row tile rtd of expert slot j --------
        const int v = u - n_gu;
        const int j = v / DF_DN, rtd = v % DF_DN;
        const int n = s_tn[j], q0 = s_tq[j];
        // h of the expert's n tokens (contiguous rows of hf) into shared memory with one bulk copy,
        // once all 40 slabs are in; the token activations' space is free (no gate/up unit follows)
        float* sh = reinterpret_cast<float*>(sqx);
        static_assert(sizeof(float) * TT * FF <= sizeof(QBlock) * TT * KB_GU, "h fits the activation space");
        if (tid == 0) {
          bool okh = spin_until_geq(&h_cnt[WS_SYNC_STRIDE * j], DF_GU, p.status);
          if (s_qx_pending) okh = mbar_wait(&bar_qx, 0u, p.status) && okh;  // (only if no gate/up unit ran)
          s_qx_pending = 0;
          if (okh) {
            fence_proxy_async_global();
            mbar_expect_tx(&bar_h, (uint32_t)(sizeof(float) * n * FF));
            bulk_g2s(sh, p.hf + (size_t)q0 * FF, (uint32_t)(sizeof(float) * n * FF), &bar_h);
            s_h_pending = n_dn & 1;
          }
          s_flag = okh ? 1 : 0;
        }
        __syncthreads();
        if (!s_flag) { if (tid == 0) s_ok = 0; __syncthreads(); break; }
        const bool hok = mbar_wait(&bar_h, (uint32_t)(n_dn & 1), p.status);
        ++n_dn;
        if (!__syncthreads_and(hok ? 1 : 0)) { if (tid == 0) s_ok = 0; __syncthreads(); break; }
        if (tid == 0) s_h_pending = -1;
        if constexpr (MMA) {  // h in fp16 fragment order: hx[kb][t4][slot][16 halves]
          uint8_t* hx = reinterpret_cast<uint8_t*>(sq);
          for (int idx = tid; idx < n * KB_D * 4; idx += DF_THREADS) {
            const int t4 = idx % 4, kb = (idx / 4) % KB_D, ii = idx / (4 * KB_D);
            const float4* v4 = reinterpret_cast<const float4*>(sh + ii * FF + kb * QK + 16 * t4);
            float f[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 a = v4[q];
              f[4 * q] = a.x; f[4 * q + 1] = a.y; f[4 * q + 2] = a.z; f[4 * q + 3] = a.w;
            }
            uint32_t hq[8];
            to_fragment_order(f, hq);
            uint4* dst = reinterpret_cast<uint4*>(hx + ((size_t)(kb * 4 + t4) * n + ii) * 32);
            dst[0] = make_uint4(hq[0], hq[1], hq[2], hq[3]);
            dst[1] = make_uint4(hq[4], hq[5], hq[6], hq[7]);
          }
        } else {
          for (int item = warp; item < n * KB_D; item += DF_THREADS / 32) {  // quantise h, one warp per block
            const int ii = item / KB_D, kb = item % KB_D;
            const float2 hv = reinterpret_cast<const float2*>(sh + ii * FF + kb * QK)[lane];
            quantise_block_warp(hv.x, hv.y, p.q2_offset, sq + kb * TT + ii, s_qtmp[warp]);
          }
        }
        if (!__syncthreads_and(mbar_wait(&bars[st], par, p.status) ? 1 : 0)) {
          if (tid == 0) s_ok = 0;
          __syncthreads();
          break;
        }
        if (tid == 0) s_pending[st] = -1;
        if constexpr (MMA) {
          // warp w: rows 32 w .. 32 w + 31 of the tile (two 16-row groups), all 10 k-blocks; columns =
          // the expert's pairs
          const int g = lane >> 2, t4 = lane & 3;
          uint32_t subq[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const __half2 s2 = __half2half2(__float2half_rn((float)((1024 >> (2 * m)) + p.q2_offset)));
            subq[m] = *reinterpret_cast<const uint32_t*>(&s2);
          }
          const uint8_t* hx = reinterpret_cast<const uint8_t*>(sq);
          float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 2
          for (int kb = 0; kb < KB_D; ++kb) {
            const uint8_t* chunk = stage + kb * D_CHUNK;
            uint4 x0 = make_uint4(0, 0, 0, 0), x1 = make_uint4(0, 0, 0, 0);
            if (g < n) {
              const uint4* xp = reinterpret_cast<const uint4*>(hx + ((size_t)(kb * 4 + t4) * n + g) * 32);
              x0 = xp[0];
              x1 = xp[1];
            }
            const uint32_t bq[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int rg = 0; rg < 2; ++rg) {
              const int R0 = 32 * warp + 16 * rg + g, R1 = R0 + 8;
              uint32_t h0[8], h1[8];
              codes_to_half2(*reinterpret_cast<const uint32_t*>(chunk + 16 * R0 + 4 * t4), subq, h0);
              codes_to_half2(*reinterpret_cast<const uint32_t*>(chunk + 16 * R1 + 4 * t4), subq, h1);
              const float d0 = __half2float(*reinterpret_cast<const __half*>(chunk + 2048 + 2 * R0));
              const float d1 = __half2float(*reinterpret_cast<const __half*>(chunk + 2048 + 2 * R1));
              float cc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
              for (int s = 0; s < 4; ++s) {
                const uint32_t a[4] = {h0[2 * s], h1[2 * s], h0[2 * s + 1], h1[2 * s + 1]};
                mma_16816(cc[s & 1], a, bq[2 * s], bq[2 * s + 1]);
              }
              acc[rg][0] = fmaf(d0, cc[0][0] + cc[1][0], acc[rg][0]); acc[rg][1] = fmaf(d0, cc[0][1] + cc[1][1], acc[rg][1]);
              acc[rg][2] = fmaf(d1, cc[0][2] + cc[1][2], acc[rg][2]); acc[rg][3] = fmaf(d1, cc[0][3] + cc[1][3], acc[rg][3]);
            }
          }
#pragma unroll
          for (int rg = 0; rg < 2; ++rg)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int col = 2 * t4 + (e & 1);
              const int row = rtd * RT + 32 * warp + 16 * rg + g + 8 * (e >> 1);
              if (col < n) p.parts[(size_t)s_pair[q0 + col] * H + row] = acc[rg][e];
            }
        } else {
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
        }
        const int row = rtd * RT + tid;  // combine: one output row per thread
        __syncthreads();
        if (tid == 0) s_flag = (atom_acq_rel_add(&cnt_dn[WS_SYNC_STRIDE * rtd], 1) == D - 1) ? 1 : 0;
        __syncthreads();
        if (s_flag) {
          float pv[TT * K], xv[TT];  // every load first, then the k-ordered sums
#pragma unroll
          for (int q = 0; q < TT * K; ++q) pv[q] = (q < T * K) ? __ldcg(p.parts + (size_t)q * H + row) : 0.f;
#pragma unroll
          for (int tt = 0; tt < TT; ++tt) xv[tt] = (tt < T && p.residual) ? p.x[(size_t)tt * H + row] : 0.f;
#pragma unroll
          for (int tt = 0; tt < TT; ++tt) {
            if (tt < T) {
              float a = 0.f;
#pragma unroll
              for (int k = 0; k < K; ++k) a = fmaf(s_w[tt * K + k], pv[tt * K + k], a);
              p.out[(size_t)tt * H + row] = p.residual ? xv[tt] + a : a;
            }
          }
          if (tid == 0) cnt_dn[WS_SYNC_STRIDE * rtd] = 0;
        }
      }
      __syncthreads();  // everyone is done with this stage and with sq / red
      if (tid == 0 && u + G * NS < n_units) issue(u + G * NS, i + NS);
    }
  }

  // ---- leave: drain copies still in flight (only after a failed wait), last CTA resets counters ----
  __syncthreads();
  if (tid == 0) {
    for (int st = 0; st < NS; ++st)
      if (s_pending[st] >= 0) mbar_wait(&bars[st], (uint32_t)s_pending[st], p.status);
    if (s_qx_pending) mbar_wait(&bar_qx, 0u, p.status);
    if (s_h_pending >= 0) mbar_wait(&bar_h, (uint32_t)s_h_pending, p.status);
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
  const size_t smem = df_smem<TT>();
  auto kern = decode_layer_kernel<TT>;
  cudaError_t err;
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  const int vi = TT == 1 ? 0 : TT == 2 ? 1 : TT == 4 ? 2 : 3;
  int grid = (dev >= 0 && dev < 64) ? g_info[dev].grid[vi] : 0;
  if (grid == 0) {  // first launch on this device: shared-memory opt-in and the co-resident grid
    if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return err;
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
  prm.hf = (float*)(ws + L.hf);
  prm.parts = (float*)(ws + L.parts);
  prm.sync = (int*)(ws + WS_SYNC);
  prm.status = (int*)(ws + L.status);
  if (T <= 1) return launch_tt<1>(prm, s);
  if (T <= 2) return launch_tt<2>(prm, s);
  if (T <= 4) return launch_tt<4>(prm, s);
  return launch_tt<8>(prm, s);
}

}  // namespace strata
