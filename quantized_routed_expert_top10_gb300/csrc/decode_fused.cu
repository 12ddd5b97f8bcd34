// One-kernel MoE layer for small token counts (decode and verify windows, T <= 8), sm_103a.
//
// The whole layer -- router GEMV (zwxr.cn news/242664, "一次路由的完整旅程": BF16 projection to 512
// logits, softmax, stable descending top-10, clamped renormalisation), grouping of tokens by expert
// (momoyeyu.github.io "ai-infra-strata", "提示词处理": one weight read serves every token routed to an
// expert), the Q2_0 SwiGLU experts (ai.thesatyajit.com "Strata engine", "The CPU kernels": codes
// {0,1,2,3} = {-1,0,1,2} x d with the offset removed once per block) and the weighted combine -- runs
// as one cooperative launch of two 256-thread CTAs per SM:
//   1. every CTA stages all tokens' activations in shared memory (up to four tokens' x arrive by
//      bulk copy; 16-bit integer blocks for one token, fp16 in MMA fragment order for more) with
//      their rmsnorm, then computes a few router rows and publishes them;
//   2. every CTA polls all router dot products and redundantly computes the top-10 of all tokens
//      and the grouping (identical results everywhere); in a decode stack its idle warps meanwhile
//      compute its rows of the next layer's router (the lookahead, step 5);
//   3. the expert bytes are cut into equal 23,040-byte units -- gate/up units (expert, slab of 16
//      rows, all 40 k-blocks: contiguous in the packed blob) and down units (expert, 128-row tile,
//      all 10 k-blocks) -- dealt round robin to the CTAs, gate/up units first.  Each CTA streams its
//      units through a ring of shared-memory stages with cp.async.bulk (L2 evict-first) as soon as
//      routing is known.  A gate/up unit publishes h = silu(g) * u of its 16 rows; a down unit polls
//      the h of its expert's tokens and publishes its 128 output rows per pair;
//   4. the CTA of down unit (expert slot j, row tile r) then polls the outputs of every pair for
//      share j of tile r's rows and writes their weighted sum in k order (+ the shared expert's
//      output, + the residual).  A layer's shared expert is one more expert slot holding every token
//      (pair slots K T + t, weight 1);
//   5. decode stacks: the last CTA takes the next layer's predicted top-10 (its router on this
//      layer's input) and publishes the distinct experts; at its start the next layer's CTAs
//      prefetch their share of those experts' units into L2 (a hint; results never depend on it).
// Every exchanged value travels as one 64-bit word (value bits, call tag) in the workspace's decode
// exchange area: a reader polls the words it needs until all carry this call's tag, so learning
// that a value is ready and fetching it take one round trip.  When the output aliases the input,
// the router publication is a release (after every read of x by its CTA) and its polling an
// acquire, which orders all reads of x before any write of the output.  Every wait is bounded by
// %globaltimer and records STRATA_E_TIMEOUT in the status word.  Every CTA advances the call epoch as
// it leaves (a max with no reply).
#include "device_common.cuh"

namespace strata {
namespace {

constexpr int DF_UNIT = 23040;                 // bytes per work unit
constexpr int DF_GU = N_SLAB;                  // 40 gate/up units (slabs) per expert
constexpr int DF_DN = RT_D;                    // 20 down units per expert
constexpr int DF_MAXD = DECODE_T_MAX * K;      // at most 80 distinct experts
constexpr int DF_THREADS = 256;
constexpr int DF_EARLY = 1;                    // unit copies issued as soon as routing is known
constexpr int DF_NW = DF_THREADS / 32;         // 8 warps
constexpr int DF_KG = DF_NW;                   // k-block groups per gate/up unit (one token: a warp each)
constexpr int DF_KBG = KB_GU / DF_KG;          // 5 k-blocks per group
static_assert(DF_KG * DF_KBG == KB_GU && 2 * SLAB * DF_KG == DF_THREADS, "gate/up unit split");
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
  int alias;           // out overlaps x: release/acquire around the router exchange (see step 1b)
  const uint16_t* wr;  // [E][H] bf16
  const float* bias;   // [E] or null
  const uint8_t* blobs;
  int64_t stride;
  const uint8_t* shared;  // the layer's shared expert (packed blob), or null
  int32_t* ids_out;  // [T][K]
  float* w_out;      // [T][K]
  uint64_t* dots;    // exchange area: router dot products [WS_NREP][DECODE_T_MAX][EMAX]
  uint64_t* htag;    //                h of each slot [DECODE_PAIRS][FF]
  uint64_t* ptag;    //                expert outputs of each pair [DECODE_PAIRS][H]
  uint64_t* pred;    //                next layer's predicted router logits [DECODE_T_MAX][EMAX]
  uint64_t* pred_ids;  //              [0]: D' predicted experts, [1 + j]: their ids, ascending
  const uint16_t* wr_next;  // next layer of a stack (lookahead), or null
  const float* bias_next;
  const uint8_t* blobs_next;
  int64_t stride_next;
  int* sync;         // ws sync words (WS_SYNC)
  int* status;
};

// Exchange words: (value bits, call tag).  A 64-bit aligned access is single-copy atomic, so a
// reader that sees the tag sees the value stored with it.
__device__ __forceinline__ void st_tagged(uint64_t* p, float v, uint32_t tag) {
  const uint64_t w = ((uint64_t)tag << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ uint64_t ld_tagged(const uint64_t* p) {
  uint64_t w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p));
  return w;
}
__device__ __forceinline__ bool has_tag(uint64_t w, uint32_t tag) { return (uint32_t)(w >> 32) == tag; }
__device__ __forceinline__ float tagged_value(uint64_t w) { return __uint_as_float((uint32_t)w); }

// Bounded poll (whole CTA) of `count` exchange words src[map(i)], i < count, into dst[i] (shared):
// each thread owns entries tid + DF_THREADS * k, k < KMAX (count <= KMAX * DF_THREADS), and re-reads
// the ones still missing, all in flight at once, until every entry of the CTA carries `tag`.  The
// verdicts are CTA-wide (barrier reductions), so every thread leaves on the same pass.  Between
// passes the CTA sleeps, 64 ns doubling up to 512 ns: a spinning CTA would take issue slots from the
// other CTA on its SM.  False (and ST_TIMEOUT) once limit_ns has passed (the layer uses the library's
// limit; the wait self-test passes a short one).
template <int KMAX, typename Map>
__device__ __forceinline__ bool poll_tagged(const uint64_t* src, Map map, int count, uint32_t tag, float* dst,
                                            int* status, unsigned long long limit_ns = kWaitLimitNs) {
  static_assert(KMAX <= 64, "one mask bit per entry");
  const int tid = threadIdx.x;
  uint64_t missing = 0;
#pragma unroll
  for (int k = 0; k < KMAX; ++k)
    if (tid + DF_THREADS * k < count) missing |= 1ull << k;
  const unsigned long long t0 = globaltimer();
  unsigned sleep_ns = 64;
  while (true) {
    uint64_t w[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      if ((missing >> k) & 1) w[k] = ld_tagged(src + map(tid + DF_THREADS * k));
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      if (((missing >> k) & 1) && has_tag(w[k], tag)) {
        dst[tid + DF_THREADS * k] = tagged_value(w[k]);
        missing &= ~(1ull << k);
      }
    if (__syncthreads_and(missing == 0 ? 1 : 0)) return true;
    if (__syncthreads_or(globaltimer() - t0 > limit_ns ? 1 : 0)) {
      if (tid == 0) set_status(status, ST_TIMEOUT);
      return false;
    }
    __nanosleep(sleep_ns);
    sleep_ns = min(2 * sleep_ns, 512u);
  }
}


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

// Quantise a 64-value block held as two halves in adjacent lanes (lane 2i + hb holds values
// 32 hb .. 32 hb + 31 in v, and its own max |v| in amax) into a QBlock: the same QBlock that
// quantise_block_warp builds, with one thread per half block instead of a warp per block.  Whole
// warps call it (the halves meet through shuffles); only `live` lanes store.
__device__ __forceinline__ void quantise_half_block(const float (&v)[32], float amax, bool live, int hb,
                                                    int q2_offset, QBlock* dst) {
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  int qv[32];
  int qs = 0;
  const float qinv = amax > 0.f ? 32767.f / amax : 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    qv[i] = amax > 0.f ? max(-32767, min(32767, __float2int_rn(v[i] * qinv))) : 0;
    qs += qv[i];
  }
  qs += __shfl_xor_sync(0xffffffffu, qs, 1);
  if (!live) return;
  // word (q4, m), q4 = 2 hb + g: bytes b' = 0..3 of the values 16 q4 + 4 b' + m
  uint32_t hw[8], lw[8];
#pragma unroll
  for (int g = 0; g < 2; ++g)
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      uint32_t hi = 0, lo = 0;
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const int val = qv[16 * g + 4 * bb + m];
        hi |= (uint32_t)((val >> 8) & 0xFF) << (8 * bb);
        lo |= (uint32_t)(val & 0xFF) << (8 * bb);
      }
      hw[4 * g + m] = hi;
      lw[4 * g + m] = lo;
    }
  uint4* dh = reinterpret_cast<uint4*>(dst->hi + 8 * hb);
  uint4* dl = reinterpret_cast<uint4*>(dst->lo + 8 * hb);
  dh[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  dh[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
  dl[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  dl[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
  if (hb == 0) {
    dst->s64 = amax > 0.f ? (amax / 32767.f) * (1.f / 64.f) : 0.f;
    dst->qoff = 64 * q2_offset * qs;
  }
}

// Bounded poll (one warp) of one token's E logit words src[e] (lane holds e = lane + 32 j) into lg
// until all carry `tag`; the warp leaves together.  False (and ST_TIMEOUT) once the wait limit passes.
__device__ __forceinline__ bool warp_poll_logits(const uint64_t* src, int E, uint32_t tag, float* lg, int* status) {
  const int lane = threadIdx.x & 31;
  uint32_t missing = (1u << (E >> 5)) - 1u;
  const unsigned long long t0 = globaltimer();
  while (true) {
    uint64_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if ((missing >> j) & 1) w[j] = ld_tagged(src + lane + 32 * j);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (((missing >> j) & 1) && has_tag(w[j], tag)) {
        lg[j] = tagged_value(w[j]);
        missing &= ~(1u << j);
      }
    if (__all_sync(0xffffffffu, missing == 0)) return true;
    if (__shfl_sync(0xffffffffu, globaltimer() - t0 > kWaitLimitNs ? 1 : 0, 0)) {
      if (lane == 0) set_status(status, ST_TIMEOUT);
      return false;
    }
    __nanosleep(100);  // back off: every CTA polls the same lines
  }
}

template <int TT>
__global__ void __launch_bounds__(DF_THREADS, 2) decode_layer_kernel(const DecodeParams p) {
  constexpr bool MMA = TT >= 2;  // one token: dp4a on the codes; more: tensor-core products
  constexpr int NS = df_stages<TT>();
  constexpr int ROWS_MAX = 16;   // router rows per CTA (grids of >= 32 CTAs)
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;                                                 // NS * DF_UNIT
  QBlock* sqx = reinterpret_cast<QBlock*>(smem + NS * DF_UNIT);         // [T][KB_GU] all tokens
  QBlock* sq = sqx + TT * KB_GU;                                        // [KB_D][TT] h of a down unit
  float* red = reinterpret_cast<float*>(sq);                            // gate/up partial sums
  static_assert(sizeof(float) * 2 * DF_NW * TT * SLAB <= sizeof(QBlock) * KB_D * TT, "reduction fits");
  __shared__ uint64_t bars[NS];
  __shared__ uint64_t bar_x;
  __shared__ int s_pending[NS];
  __shared__ float s_inv[TT];
  __shared__ float s_ssq[DF_NW];
  __shared__ float s_ssqt[DF_NW][TT];  // per warp and token (two or more tokens)
  __shared__ float s_dot[ROWS_MAX][TT];
  __shared__ __align__(16) int s_ids[(TT * K + 3) / 4 * 4];
  __shared__ float s_w[TT * (K + 1)];  // weight of each pair (a shared-expert pair K T + t: 1)
  __shared__ int s_te[DF_MAXD + 1];   // expert slot j -> expert id (-1: the shared expert)
  __shared__ int s_tn[DF_MAXD + 1];   //               -> tokens routed to it
  __shared__ int s_tq[DF_MAXD + 1];   //               -> first slot in s_pair
  __shared__ int s_first[TT * K];  // expert id of each slot (grouping)
  __shared__ int s_wcnt[DF_NW];
  __shared__ int s_pair[TT * (K + 1)];  // slot -> pair (routed t K + k; shared expert K T + t)
  __shared__ float s_rpart[DF_NW][TT];
  __shared__ float s_lpart[4][TT];  // lookahead rows' partial sums (warps 4-7)
  __shared__ float s_bias[EMAX];
  TopKScratch* s_topk = reinterpret_cast<TopKScratch*>(ring);  // [DF_NW], routing only (ring idle)
  static_assert(sizeof(TopKScratch) * DF_NW <= DF_UNIT, "top-k scratch fits the first stage");
  __shared__ int s_flag, s_ok, s_nact, s_dots0, s_tw0;

  const int G = gridDim.x, c = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T, E = p.E, P = T * K;
  int* exit_cnt = p.sync + WS_SYNC_EXIT;
  griddep_launch_dependents();

  // up to four tokens: every token's x (fp32) into the ring (idle until the units) with bulk copies,
  // read from there by the staging, the router rows and the lookahead
  constexpr bool XS = TT <= 4;
  constexpr int XSTR = H + 4;  // token stride of the ring copy (floats): rows start 4 banks apart
  const float* xs32 = reinterpret_cast<const float*>(ring + 8192);  // after the top-k scratch
  static_assert(!XS || 8192 + sizeof(float) * TT * XSTR <= (size_t)NS * DF_UNIT, "x fits the ring");
  static_assert(sizeof(TopKScratch) * DF_NW <= 8192, "top-k scratch before x");
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars[s], 1);
      s_pending[s] = -1;
    }
    mbar_init(&bar_x, 1);
    fence_mbar_init();
    s_ok = 1;
  }
  // loads for later steps, issued first (they read only the layer's constant router rows and bias, so
  // they may run while the previous kernel on the stream finishes): the bias (used by the top-k) and
  // this CTA's first router row (two warps per row, each over one half of the columns)
  float bias_v[EMAX / DF_THREADS];
#pragma unroll
  for (int i = 0; i < EMAX / DF_THREADS; ++i) {
    const int e = tid + DF_THREADS * i;
    bias_v[i] = (p.bias && e < E) ? __ldg(p.bias + e) : 0.f;
  }
  const int half = warp & 1;
  uint4 wq[H / 512];
  {
    const int e = c + G * (warp >> 1);
    if (e < E) {
      const uint4* wrow = reinterpret_cast<const uint4*>(p.wr + (size_t)e * H);
#pragma unroll
      for (int i = 0; i < H / 512; ++i) wq[i] = __ldg(wrow + ((half * (H / 2) + 8 * lane + 256 * i) >> 3));
    }
  }
  // everything else -- the call epoch, x, the exchange area -- only once the previous kernel is done
  griddep_wait();
  // this call's tag: one more than the previous call's (the CTAs advance the epoch as they leave)
  const uint32_t ep = (uint32_t)ld_relaxed(p.sync + WS_SYNC_EPOCH) + 1u;
  if (tid == 0) {
    if (XS) {
      mbar_expect_tx(&bar_x, (uint32_t)(sizeof(float) * T * H));
      for (int t = 0; t < T; ++t)
        bulk_g2s(ring + 8192 + sizeof(float) * t * XSTR, p.x + (size_t)t * H, (uint32_t)(sizeof(float) * H), &bar_x);
    }
    // the router words this CTA will poll into L2 now, so the publishers' stores and the polls meet
    // in L2 instead of each paying a miss later
    bulk_prefetch_l2(p.dots + (size_t)(c % WS_NREP) * DECODE_T_MAX * EMAX, (uint32_t)(sizeof(uint64_t) * T * EMAX));
  }
  // x of token t at column col: the ring copy (up to four tokens) or global memory
  auto x4 = [&](int t, int col) {
    return XS ? *reinterpret_cast<const float4*>(xs32 + (size_t)t * XSTR + col)
              : __ldg(reinterpret_cast<const float4*>(p.x + (size_t)t * H + col));
  };
  __syncthreads();  // the barriers are initialised before anyone waits on them
  if (XS) mbar_wait(&bar_x, 0u, p.status);  // bounded; a failure is in the status word

  // previous layer of a stack predicted this layer's experts (words tagged with the previous call's
  // tag): this CTA prefetches its share of their units into L2 while routing goes on.  A hint only.
  if (tid == DF_THREADS - 1) {
    // one or two tokens: the SM's two CTAs route on different warps (0-1, 2-3), hence on different
    // schedulers -- the top-10 is a latency chain that two warps on one scheduler would share
    s_tw0 = TT <= 2 ? 2 * (int)(atomicAdd(reinterpret_cast<unsigned*>(p.sync + WS_SYNC_SMRANK + (sm_id() & 255)), 1u) & 1u)
                    : 0;
    if (p.wr_next && TT <= 4)  // this CTA's rows of the next layer's router, for the lookahead below
      for (int e = c; e < E; e += G) bulk_prefetch_l2(p.wr_next + (size_t)e * H, (uint32_t)(sizeof(uint16_t) * H));
    const uint64_t w0 = ld_tagged(p.pred_ids);
    if (has_tag(w0, ep - 1u)) {
      const int D = min(__float_as_int(tagged_value(w0)), DF_MAXD);
      for (int u = c; u < D * (DF_GU + DF_DN); u += G) {
        const bool gu = u < D * DF_GU;
        const int j = gu ? u / DF_GU : (u - D * DF_GU) / DF_DN;
        const uint64_t wj = ld_tagged(p.pred_ids + 1 + j);
        const int e = __float_as_int(tagged_value(wj));
        if (!has_tag(wj, ep - 1u) || e < 0 || e >= E) continue;
        const uint8_t* b = p.blobs + (int64_t)e * p.stride;
        bulk_prefetch_l2(gu ? b + (int64_t)(u % DF_GU) * SLAB_BYTES
                            : b + D_REGION + (int64_t)((u - D * DF_GU) % DF_DN) * KB_D * D_CHUNK,
                         DF_UNIT);
      }
    }
  }

  // ---- 1a. every token's activations into shared memory, and their rmsnorm ----
  if constexpr (!MMA) {
    // one token: 40 blocks quantised to QBlocks, one thread per half block (32 values, the two
    // halves in adjacent lanes) -- the same QBlock as quantise_block_warp builds
    static_assert(2 * KB_GU <= DF_THREADS, "one thread per half block");
    const int b = tid >> 1, hb = tid & 1;
    const bool live = tid < 2 * KB_GU;
    float v[32];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 a = live ? x4(0, b * QK + 32 * hb + 4 * q) : make_float4(0.f, 0.f, 0.f, 0.f);
      v[4 * q] = a.x; v[4 * q + 1] = a.y; v[4 * q + 2] = a.z; v[4 * q + 3] = a.w;
    }
    float amax = 0.f, ss = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      amax = fmaxf(amax, fabsf(v[i]));
      ss = fmaf(v[i], v[i], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) s_ssq[warp] = ss;
    quantise_half_block(v, amax, live, hb, p.q2_offset, sqx + b);
  } else {
    // fp16 x in fragment order, xs[16-group][token][16 halves]: item = (16-group g, token t) with t
    // fastest, so consecutive threads write consecutive 32-byte fragments (conflict-free); thread tid
    // keeps token tid % TT throughout (256 is a multiple of TT), and each token's sum of squares is
    // reduced in a fixed order (lanes, then warps)
    static_assert(DF_THREADS % TT == 0, "a thread stays on one token");
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < (H / 16 * TT + DF_THREADS - 1) / DF_THREADS; ++k) {
      const int idx = tid + DF_THREADS * k, g = idx / TT, t = idx % TT;
      if (g < H / 16 && t < T) {
        float f[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 a = x4(t, 16 * g + 4 * q);
          f[4 * q] = a.x; f[4 * q + 1] = a.y; f[4 * q + 2] = a.z; f[4 * q + 3] = a.w;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) ss = fmaf(f[i], f[i], ss);
        uint32_t hq[8];
        to_fragment_order(f, hq);
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(sqx) + ((size_t)g * T + t) * 32);
        dst[0] = make_uint4(hq[0], hq[1], hq[2], hq[3]);
        dst[1] = make_uint4(hq[4], hq[5], hq[6], hq[7]);
      }
    }
#pragma unroll
    for (int o = TT; o < 32; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane < TT) s_ssqt[warp][lane] = ss;
    __syncthreads();
    if (tid < T) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < DF_NW; ++w) tot += s_ssqt[w][tid];
      s_inv[tid] = p.residual ? 1.f / sqrtf(tot / (float)H + 1e-6f) : 1.f;
    }
  }
#pragma unroll
  for (int i = 0; i < EMAX / DF_THREADS; ++i)
    if (tid + DF_THREADS * i < E) s_bias[tid + DF_THREADS * i] = bias_v[i];
  __syncthreads();

  // ---- 1b. router dot products: row c + G m, m = 0, 1, ... (two warps per row, DF_NW / 2 rows a round) ----
  int n_rows = 0;
  for (int e0 = c, it = 0; e0 < E; e0 += (DF_NW / 2) * G, ++it) {
    const int e = e0 + G * (warp >> 1);
    float acc[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t] = 0.f;
    if (e < E) {
      const uint4* wrow = reinterpret_cast<const uint4*>(p.wr + (size_t)e * H);
#pragma unroll
      for (int i = 0; i < H / 512; ++i) {
        const int col = half * (H / 2) + 8 * lane + 256 * i;
        float wf[8];
        bf16x8_to_f32(it == 0 ? wq[i] : __ldg(wrow + (col >> 3)), wf);
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          if (t < T) {
            const float4 a4 = x4(t, col), b4 = x4(t, col + 4);
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
    if (tid < (DF_NW / 2) * TT) {
      const int w2 = tid / TT, t = tid % TT, m = (DF_NW / 2) * it + w2;
      if (m < ROWS_MAX) s_dot[m][t] = s_rpart[2 * w2][t] + s_rpart[2 * w2 + 1][t];
    }
    __syncthreads();
    n_rows = min((DF_NW / 2) * (it + 1), ROWS_MAX);
  }
  // publish.  When out aliases x, the publication is a release (fence, then the tagged stores) after
  // every read of x by this CTA and the routing poll an acquire: every CTA's reads of x then happen
  // before any CTA's combine writes the output.  Otherwise the fences are left out.
  for (int idx = tid; idx < n_rows * T * WS_NREP; idx += DF_THREADS) {
    const int r = idx % WS_NREP, t = (idx / WS_NREP) % T, m = idx / (WS_NREP * T);
    const int e = c + G * m;
    if (e < E) {
      if (p.alias && idx == tid) fence_acq_rel_gpu();
      st_tagged(p.dots + ((size_t)r * DECODE_T_MAX + t) * EMAX + e, s_dot[m][t], ep);
    }
  }

  // ---- lookahead (decode stacks, T <= 4): while warps 0-3 route, warps 4-7 compute this CTA's rows of
  // the next layer's router on this layer's normalised input and publish them for the lookahead CTA
  // (step 5), which names the experts the next layer's CTAs prefetch into L2 ----
  if (TT <= 4 && p.wr_next && warp >= 4) {
    const int lw = warp - 4, lt = tid - 128;
    float inv1 = 1.f;  // one token: 1/rms from the staging's partial sums (as the routing computes it)
    if constexpr (!MMA) {
      float ssq = 0.f;
#pragma unroll
      for (int w = 0; w < DF_NW; ++w) ssq += s_ssq[w];
      inv1 = p.residual ? 1.f / sqrtf(ssq / (float)H + 1e-6f) : 1.f;
    }
    for (int e0 = c; e0 < E; e0 += 2 * G) {
      const int e = e0 + G * (lw >> 1);
      float acc[TT];
#pragma unroll
      for (int t = 0; t < TT; ++t) acc[t] = 0.f;
      if (e < E) {
        const uint4* wrow = reinterpret_cast<const uint4*>(p.wr_next + (size_t)e * H);
#pragma unroll
        for (int i = 0; i < H / 512; ++i) {
          const int col = (lw & 1) * (H / 2) + 8 * lane + 256 * i;
          float wf[8];
          bf16x8_to_f32(__ldg(wrow + (col >> 3)), wf);
#pragma unroll
          for (int t = 0; t < TT; ++t) {
            if (t < T) {
              const float4 a4 = x4(t, col), b4 = x4(t, col + 4);
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
        if (lane == 0) s_lpart[lw][t] = r;
      }
      named_barrier(1, 128);
      if (lt < 2 * TT) {
        const int w2 = lt / TT, t = lt % TT, e2 = e0 + G * w2;
        if (e2 < E && t < T) {
          const float inv = MMA ? s_inv[t] : inv1;
          const float v = (s_lpart[2 * w2][t] + s_lpart[2 * w2 + 1][t]) * inv + (p.bias_next ? __ldg(p.bias_next + e2) : 0.f);
          st_tagged(p.pred + (size_t)t * EMAX + e2, v, ep);
        }
      }
      named_barrier(1, 128);
    }
  }

  // ---- 2. top-10 and grouping, redundantly in every CTA ----
  if (tid == 0) {
    s_nact = 0;
    s_dots0 = 0;
  }
  __syncthreads();
  bool okr = true;
  for (int t = (warp - s_tw0 + DF_NW) % DF_NW; t < T; t += DF_NW) {
    // this token's dot products from replica c % WS_NREP: poll until all carry this call's tag.
    // Only token 0's warp polls from the start; the others wait (in shared memory) until token 0's
    // products are all in -- the publishers wrote every token's products together -- so the CTAs
    // do not flood the L2 with T times the polling reads.
    const uint64_t* src = p.dots + ((size_t)(c % WS_NREP) * DECODE_T_MAX + t) * EMAX;
    const int per = E >> 5;
    float lg[16];
    if (t > 0) {
      const unsigned long long t0 = globaltimer();
      while (*reinterpret_cast<volatile int*>(&s_dots0) == 0) {
        if (__shfl_sync(0xffffffffu, globaltimer() - t0 > kWaitLimitNs ? 1 : 0, 0)) break;
        __nanosleep(128);
      }
      __syncwarp();
    }
    okr = warp_poll_logits(src, E, ep, lg, p.status);
    if (t == 0 && lane == 0) *reinterpret_cast<volatile int*>(&s_dots0) = 1;
    if (!okr) break;
    if (p.alias) fence_acq_rel_gpu();  // acquire: pairs with every publisher's release
    float inv;
    if constexpr (MMA) {
      inv = s_inv[t];
    } else {
      float ssq = 0.f;
#pragma unroll
      for (int w = 0; w < DF_NW; ++w) ssq += s_ssq[w];
      inv = p.residual ? 1.f / sqrtf(ssq / (float)H + 1e-6f) : 1.f;
      if (lane == 0) s_inv[0] = inv;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < per) lg[j] = lg[j] * inv + s_bias[lane + 32 * j];
    int id;
    float w;
    top_k_warp_fn([&](int e) { return lg[e >> 5]; }, E, s_topk[warp], &id, &w);
    if (lane < K) {
      s_ids[t * K + lane] = id;
      s_w[t * K + lane] = w;
    }
    if constexpr (TT == 1) {
      // one token: its K ids are distinct, so expert slot = pair slot = the id's rank among them
      int below = 0;
#pragma unroll
      for (int q = 0; q < K; ++q) below += (__shfl_sync(0xffffffffu, id, q) < id) ? 1 : 0;
      if (lane < K) {
        s_pair[below] = lane;
        s_te[below] = id;
        s_tn[below] = 1;
        s_tq[below] = below;
      }
      if (lane == 0) s_nact = K;
    }
  }
  const bool routed = __syncthreads_and(okr ? 1 : 0);
  if (!routed) {
    if (tid == 0) s_ok = 0;
  } else if constexpr (TT > 1) {
    // grouping of the P <= 80 pairs by a counting sort: the slot of pair q is its rank by (expert id,
    // q); a slot whose id differs from the previous slot's starts the next expert slot
    for (int q = P + tid; q < (P + 3) / 4 * 4; q += DF_THREADS) s_ids[q] = EMAX;  // pad to whole int4
    __syncthreads();
    if (tid < P) {
      const int e = s_ids[tid];
      const int key = e * DF_MAXD + tid;
      int rank = 0;
      const int4* ids4 = reinterpret_cast<const int4*>(s_ids);
      for (int q4 = 0; q4 < (P + 3) / 4; ++q4) {
        const int4 f = ids4[q4];
        rank += (f.x * DF_MAXD + 4 * q4 < key) + (f.y * DF_MAXD + 4 * q4 + 1 < key) +
                (f.z * DF_MAXD + 4 * q4 + 2 < key) + (f.w * DF_MAXD + 4 * q4 + 3 < key);
      }
      s_pair[rank] = tid;
      s_first[rank] = e;  // the expert id of each slot
    }
    __syncthreads();
    const bool starts = tid < P && (tid == 0 || s_first[tid - 1] != s_first[tid]);
    const uint32_t bal = __ballot_sync(0xffffffffu, starts);
    if (lane == 0) s_wcnt[warp] = __popc(bal);
    __syncthreads();
    if (starts) {
      int j = __popc(bal & ((1u << lane) - 1u));
      for (int w = 0; w < warp; ++w) j += s_wcnt[w];
      const int id = s_first[tid];
      int n = 0;
      for (int q = tid; q < P && s_first[q] == id; ++q) ++n;
      s_te[j] = id;
      s_tn[j] = n;
      s_tq[j] = tid;
    }
    if (tid == 0) {
      int d = 0;
      for (int w = 0; w < DF_THREADS / 32; ++w) d += s_wcnt[w];
      s_nact = d;
    }
  }
  if (c == 0 && routed)
    for (int q = tid; q < P; q += DF_THREADS) {
      p.ids_out[q] = s_ids[q];
      p.w_out[q] = s_w[q];
    }
  __syncthreads();
  if (p.shared && routed) {  // the shared expert: one more expert slot, every token, weight 1
    if (tid < T) {
      s_pair[P + tid] = P + tid;
      s_w[P + tid] = 1.f;
    }
    if (tid == 0) {
      const int D = s_nact;
      s_te[D] = -1;
      s_tn[D] = T;
      s_tq[D] = P;
      s_nact = D + 1;
    }
    __syncthreads();
  }

  // ---- 3. expert units ----
  if (s_ok) {
    const int D = s_nact;
    const int n_gu = D * DF_GU, n_units = D * (DF_GU + DF_DN);
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int u, int i) {  // thread 0 only: unit u into stage i % NS
      const int st = i % NS;
      const uint8_t* src;
      if (u < n_gu) {
        const int j = u / DF_GU, sl = u % DF_GU;
        src = (s_te[j] >= 0 ? p.blobs + (int64_t)s_te[j] * p.stride : p.shared) + (int64_t)sl * SLAB_BYTES;
      } else {
        const int v = u - n_gu;
        const int j = v / DF_DN, rtd = v % DF_DN;
        src = (s_te[j] >= 0 ? p.blobs + (int64_t)s_te[j] * p.stride : p.shared) + D_REGION +
              (int64_t)rtd * KB_D * D_CHUNK;
      }
      s_pending[st] = (i / NS) & 1;
      mbar_expect_tx(&bars[st], DF_UNIT);
      bulk_g2s_stream(ring + (size_t)st * DF_UNIT, src, DF_UNIT, &bars[st], pol);
    };
    // the first DF_EARLY units' copies now, the rest once the first has arrived: not queued behind
    // every CTA's later stages, the first units start computing while the rest streams in
    if (tid == 0)
      for (int k = 0; k < DF_EARLY; ++k)
        if (c + G * k < n_units) issue(c + G * k, k);

    int i = 0;
    for (int u = c; u < n_units; u += G, ++i) {
      const int st = i % NS;
      const uint32_t par = (uint32_t)((i / NS) & 1);
      const uint8_t* stage = ring + (size_t)st * DF_UNIT;
      if (u < n_gu) {
        // -------- gate/up unit: slab sl (rows 16 sl ..) of expert slot j, all k-blocks --------
        const int j = u / DF_GU, sl = u % DF_GU;
        const int n = s_tn[j], q0 = s_tq[j];
        if (!__syncthreads_and(mbar_wait(&bars[st], par, p.status) ? 1 : 0)) {
          if (tid == 0) s_ok = 0;
          __syncthreads();
          break;
        }
        if (tid == 0) {
          s_pending[st] = -1;
          if (i == 0)
            for (int k = DF_EARLY; k < NS; ++k)
              if (c + G * k < n_units) issue(c + G * k, k);
        }
        if constexpr (MMA) {
          // warp w: k-blocks [5 w, 5 w + 5) of the 16-row slab, all T tokens as columns
          const int g = lane >> 2, t4 = lane & 3;
          uint32_t subq[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const __half2 s2 = __half2half2(__float2half_rn((float)((1024 >> (2 * m)) + p.q2_offset)));
            subq[m] = *reinterpret_cast<const uint32_t*>(&s2);
          }
          const uint8_t* xs = reinterpret_cast<const uint8_t*>(sqx);
          float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
          // software pipeline: the A fragments of k-block kb + 1 are built while kb's MMAs run
          uint32_t hg0[8], hg1[8], hu0[8], hu1[8];
          __half2 sc0, sc1;
          auto dequant = [&](int kb) {
            const uint8_t* piece = stage + kb * SLAB_KB;
            codes_to_half2(*reinterpret_cast<const uint32_t*>(piece + 16 * g + 4 * t4), subq, hg0);
            codes_to_half2(*reinterpret_cast<const uint32_t*>(piece + 16 * (g + 8) + 4 * t4), subq, hg1);
            codes_to_half2(*reinterpret_cast<const uint32_t*>(piece + 256 + 16 * g + 4 * t4), subq, hu0);
            codes_to_half2(*reinterpret_cast<const uint32_t*>(piece + 256 + 16 * (g + 8) + 4 * t4), subq, hu1);
            sc0 = *reinterpret_cast<const __half2*>(piece + 512 + 4 * g);
            sc1 = *reinterpret_cast<const __half2*>(piece + 512 + 4 * (g + 8));
          };
          constexpr int KPW = KB_GU / DF_NW;  // k-blocks per warp
          dequant(warp * KPW);
#pragma unroll
          for (int kk = 0; kk < KPW; ++kk) {
            const int kb = warp * KPW + kk;
            uint4 x0 = make_uint4(0, 0, 0, 0), x1 = make_uint4(0, 0, 0, 0);
            if (g < T) {
              const uint4* xp = reinterpret_cast<const uint4*>(xs + ((size_t)(kb * 4 + t4) * T + g) * 32);
              x0 = xp[0];
              x1 = xp[1];
            }
            const uint32_t bq[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            uint32_t a_g[4][4], a_u[4][4];
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              a_g[s][0] = hg0[2 * s]; a_g[s][1] = hg1[2 * s]; a_g[s][2] = hg0[2 * s + 1]; a_g[s][3] = hg1[2 * s + 1];
              a_u[s][0] = hu0[2 * s]; a_u[s][1] = hu1[2 * s]; a_u[s][2] = hu0[2 * s + 1]; a_u[s][3] = hu1[2 * s + 1];
            }
            const __half2 c0 = sc0, c1 = sc1;
            if (kk + 1 < KPW) dequant(kb + 1);
            // even and odd k-steps into separate accumulators: two independent MMA chains per matrix
            float cg[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            float cu[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              mma_16816(cg[s & 1], a_g[s], bq[2 * s], bq[2 * s + 1]);
              mma_16816(cu[s & 1], a_u[s], bq[2 * s], bq[2 * s + 1]);
            }
            const float dg0 = __low2float(c0), du0 = __high2float(c0);
            const float dg1 = __low2float(c1), du1 = __high2float(c1);
            ag[0] = fmaf(dg0, cg[0][0] + cg[1][0], ag[0]); ag[1] = fmaf(dg0, cg[0][1] + cg[1][1], ag[1]);
            ag[2] = fmaf(dg1, cg[0][2] + cg[1][2], ag[2]); ag[3] = fmaf(dg1, cg[0][3] + cg[1][3], ag[3]);
            au[0] = fmaf(du0, cu[0][0] + cu[1][0], au[0]); au[1] = fmaf(du0, cu[0][1] + cu[1][1], au[1]);
            au[2] = fmaf(du1, cu[0][2] + cu[1][2], au[2]); au[3] = fmaf(du1, cu[0][3] + cu[1][3], au[3]);
          }
          // red[warp][mat][row][column]: the warps' k ranges, added below in warp order
          float* rf = red;
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
            const int pq = s_pair[q0 + ii], tk = pq < P ? pq / K : pq - P;
            float gg = 0.f, uu = 0.f;
#pragma unroll
            for (int w = 0; w < DF_NW; ++w) {
              gg += rf[((w * 2 + 0) * SLAB + r2) * TT + tk];
              uu += rf[((w * 2 + 1) * SLAB + r2) * TT + tk];
            }
            const float inv = s_inv[tk];
            st_tagged(p.htag + (size_t)(q0 + ii) * FF + sl * SLAB + r2, silu_mul(gg * inv, uu * inv), ep);
          }
        } else {
          // thread: row r of the slab, matrix mat (gate, up), group grp = warp of DF_KBG k-blocks
          const int r = tid % SLAB, mat = (tid / SLAB) & 1, grp = warp;
          int tok[TT];
          float tinv[TT];
#pragma unroll
          for (int ii = 0; ii < TT; ++ii) {
            const int pq = (ii < n) ? s_pair[q0 + ii] : 0;
            tok[ii] = pq < P ? pq / K : pq - P;
            tinv[ii] = (ii < n) ? s_inv[tok[ii]] : 0.f;
          }
          float acc[TT];
#pragma unroll
          for (int ii = 0; ii < TT; ++ii) acc[ii] = 0.f;
#pragma unroll 1
          for (int kk = 0; kk < DF_KBG; ++kk) {
            const int kb = grp * DF_KBG + kk;
            const uint8_t* piece = stage + kb * SLAB_KB;
            const uint4 cw = *reinterpret_cast<const uint4*>(piece + 256 * mat + 16 * r);
            const float d = __half2float(*reinterpret_cast<const __half*>(piece + 512 + 4 * r + 2 * mat));
            const Masked cm = mask_codes(cw);
#pragma unroll
            for (int ii = 0; ii < TT; ++ii) {
              if (ii < n) {
                const QBlock& a = sqx[tok[ii] * KB_GU + kb];
                uint32_t hi[16], lo[16];
                unpack_words(a, hi, lo);
                const int vv = dot64(cm, hi, lo) - a.qoff;
                acc[ii] = fmaf(d * (a.s64 * tinv[ii]), (float)vv, acc[ii]);
              }
            }
          }
#pragma unroll
          for (int ii = 0; ii < TT; ++ii)
            if (ii < n) red[((grp * 2 + mat) * TT + ii) * SLAB + r] = acc[ii];
          __syncthreads();
          if (tid < SLAB * n) {  // (row, token): the groups added in group order
            const int r2 = tid % SLAB, ii = tid / SLAB;
            float g = 0.f, uu = 0.f;
#pragma unroll
            for (int q = 0; q < DF_KG; ++q) {
              g += red[((q * 2 + 0) * TT + ii) * SLAB + r2];
              uu += red[((q * 2 + 1) * TT + ii) * SLAB + r2];
            }
            st_tagged(p.htag + (size_t)(q0 + ii) * FF + sl * SLAB + r2, silu_mul(g, uu), ep);
          }
        }
      } else {
        // -------- down unit: row tile rtd of expert slot j --------
        const int v = u - n_gu;
        const int j = v / DF_DN, rtd = v % DF_DN;
        const int n = s_tn[j], q0 = s_tq[j];
        // h of the expert's n tokens (n * FF words from slot q0 on) into shared memory; the token
        // activations' space is free (no gate/up unit follows)
        float* sh = reinterpret_cast<float*>(sqx);
        static_assert(sizeof(float) * TT * FF <= sizeof(QBlock) * TT * KB_GU, "h fits the activation space");
        const uint64_t* hsrc = p.htag + (size_t)q0 * FF;
        if (!poll_tagged<(TT * FF + DF_THREADS - 1) / DF_THREADS>(hsrc, [](int x) { return x; }, n * FF, ep, sh,
                                                                 p.status)) {
          if (tid == 0) s_ok = 0;
          __syncthreads();
          break;
        }
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
          // quantise h: one thread per half block (T = 1 here: 10 blocks)
          static_assert(TT * KB_D * 2 <= DF_THREADS, "one thread per half block of h");
          const int blk = tid >> 1, hb = tid & 1;
          const bool live = blk < n * KB_D;
          const int ii = live ? blk / KB_D : 0, kb = live ? blk % KB_D : 0;
          float v[32];
          float amax = 0.f;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 a = live ? reinterpret_cast<const float4*>(sh + ii * FF + kb * QK + 32 * hb)[q]
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            v[4 * q] = a.x; v[4 * q + 1] = a.y; v[4 * q + 2] = a.z; v[4 * q + 3] = a.w;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
          if (warp * 32 < 2 * n * KB_D) quantise_half_block(v, amax, live, hb, p.q2_offset, sq + kb * TT + ii);
        }
        if (!__syncthreads_and(mbar_wait(&bars[st], par, p.status) ? 1 : 0)) {
          if (tid == 0) s_ok = 0;
          __syncthreads();
          break;
        }
        if (tid == 0) {
          s_pending[st] = -1;
          if (i == 0)
            for (int k = DF_EARLY; k < NS; ++k)
              if (c + G * k < n_units) issue(c + G * k, k);
        }
        if constexpr (MMA) {
          // warp w: rows 16 w .. 16 w + 15 of the tile, all 10 k-blocks; columns = the expert's pairs
          const int g = lane >> 2, t4 = lane & 3;
          uint32_t subq[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const __half2 s2 = __half2half2(__float2half_rn((float)((1024 >> (2 * m)) + p.q2_offset)));
            subq[m] = *reinterpret_cast<const uint32_t*>(&s2);
          }
          const uint8_t* hx = reinterpret_cast<const uint8_t*>(sq);
          constexpr int RG = RT / (16 * DF_NW);  // 16-row groups per warp
          float acc[RG][4] = {};
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
            for (int rg = 0; rg < RG; ++rg) {
              const int R0 = 16 * RG * warp + 16 * rg + g, R1 = R0 + 8;
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
          for (int rg = 0; rg < RG; ++rg)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int col = 2 * t4 + (e & 1);
              const int row = rtd * RT + 16 * RG * warp + 16 * rg + g + 8 * (e >> 1);
              if (col < n) st_tagged(p.ptag + (size_t)s_pair[q0 + col] * H + row, acc[rg][e], ep);
            }
        } else {
          // thread: row tid % RT, k-blocks [5 h, 5 h + 5) with h = tid / RT; the halves' sums meet in
          // the activation space (free once h is quantised)
          static_assert(DF_THREADS == 2 * RT, "two threads per down row");
          const int row = tid % RT, hh = tid / RT;
          float acc[TT];
#pragma unroll
          for (int ii = 0; ii < TT; ++ii) acc[ii] = 0.f;
#pragma unroll 1
          for (int kk = 0; kk < KB_D / 2; ++kk) {
            const int kb = hh * (KB_D / 2) + kk;
            const uint8_t* chunk = stage + kb * D_CHUNK;
            const uint4 cw = *reinterpret_cast<const uint4*>(chunk + 16 * row);
            const float d = __half2float(*reinterpret_cast<const __half*>(chunk + 2048 + 2 * row));
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
          float* rdn = reinterpret_cast<float*>(sqx);  // [2][TT][RT]
          static_assert(sizeof(float) * 2 * TT * RT <= sizeof(QBlock) * TT * KB_GU, "down halves fit");
#pragma unroll
          for (int ii = 0; ii < TT; ++ii)
            if (ii < n) rdn[(hh * TT + ii) * RT + row] = acc[ii];
          __syncthreads();
          if (tid < RT)
#pragma unroll
            for (int ii = 0; ii < TT; ++ii)
              if (ii < n)
                st_tagged(p.ptag + (size_t)s_pair[q0 + ii] * H + rtd * RT + tid,
                          rdn[ii * RT + tid] + rdn[(TT + ii) * RT + tid], ep);
        }
      }
      __syncthreads();  // everyone is done with this stage and with sq / red
      if (tid == 0 && u + G * NS < n_units) issue(u + G * NS, i + NS);
    }

    // ---- 4. combine: for each down unit (slot j, tile rtd) of this CTA, rows [j rp, (j + 1) rp) of
    // the tile: every pair's output polled into shared memory, then the k-ordered weighted sums ----
    const int rp = (RT + D - 1) / D;  // D >= K (K + 1 with a shared expert), so rp <= 13 (12)
    const int NPQ = P + (p.shared ? T : 0);  // pairs polled: the routed ones, then the shared expert's
    float* cs = reinterpret_cast<float*>(sqx);  // [pair][row of the share]
    constexpr int CS_MAX = TT * K * ((RT + K - 1) / K) > TT * (K + 1) * ((RT + K) / (K + 1))
                               ? TT * K * ((RT + K - 1) / K)
                               : TT * (K + 1) * ((RT + K) / (K + 1));
    static_assert(sizeof(float) * CS_MAX <= sizeof(QBlock) * TT * KB_GU, "share fits");
    for (int u = c; u < n_units && s_ok; u += G) {
      if (u < n_gu) continue;
      const int v = u - n_gu;
      const int j = v / DF_DN, rtd = v % DF_DN;
      const int r0 = j * rp, nr = min(RT, r0 + rp) - r0;
      if (nr <= 0) continue;
      const uint64_t* psrc = p.ptag + rtd * RT + r0;
      constexpr int KC = (CS_MAX + DF_THREADS - 1) / DF_THREADS;
      if (!poll_tagged<KC>(psrc, [nr](int x) { return (x / nr) * H + x % nr; }, NPQ * nr, ep, cs, p.status)) {
        if (tid == 0) s_ok = 0;
        __syncthreads();
        break;
      }
      if (tid < nr * T) {
        const int r = tid % nr, tt = tid / nr;
        const int row = rtd * RT + r0 + r;
        const float xv = p.residual ? p.x[(size_t)tt * H + row] : 0.f;
        float a = 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) a = fmaf(s_w[tt * K + k], cs[(tt * K + k) * nr + r], a);
        if (p.shared) a += cs[(P + tt) * nr + r];
        p.out[(size_t)tt * H + row] = p.residual ? xv + a : a;
      }
      __syncthreads();
    }

    // ---- 5. lookahead CTA (the last one, which has the fewest units): the next layer's predicted
    // top-10 of every token and the distinct experts among them ----
    if (p.wr_next && c == G - 1 && s_ok) {
      bool okp = true;
      for (int t = warp; t < T && okp; t += DF_NW) {
        float lg[16];
        okp = warp_poll_logits(p.pred + (size_t)t * EMAX, E, ep, lg, p.status);
        if (okp) {
          int id;
          float w;
          top_k_warp_fn([&](int e) { return lg[e >> 5]; }, E, s_topk[warp], &id, &w);
          if (lane < K) s_first[t * K + lane] = id;  // (grouping scratch, free now)
        }
      }
      // the distinct predicted experts in ascending id order (the order of expert slots), published
      // for the next layer's CTAs, which prefetch them into L2 while they route
      if (__syncthreads_and(okp ? 1 : 0)) {
        if (tid < P) {
          const int e = s_first[tid];
          int f = 1;
          for (int q = 0; q < tid; ++q) f &= (s_first[q] != e);
          s_pair[tid] = f;  // (grouping scratch, free now)
        }
        __syncthreads();
        if (tid < P && s_pair[tid]) {
          const int e = s_first[tid];
          int j = 0;
          for (int q = 0; q < P; ++q) j += (s_pair[q] && s_first[q] < e) ? 1 : 0;
          st_tagged(p.pred_ids + 1 + j, __int_as_float(e), ep);
        }
        if (tid == 0) {
          int d = 0;
          for (int q = 0; q < P; ++q) d += s_pair[q];
          st_tagged(p.pred_ids, __int_as_float(d), ep);
        }
      }
    }
  }

  // ---- leave: drain copies still in flight (only after a failed wait) and advance the epoch: every
  // CTA adds its max(epoch, tag) without waiting for a reply -- every CTA read the epoch before it
  // published anything, and the next call reads it after this one has ended.  At the last tag the CTAs
  // count out instead, and the last one clears the exchange area and restarts the epoch from 0. ----
  __syncthreads();
  if (tid == 0) {
    for (int st = 0; st < NS; ++st)
      if (s_pending[st] >= 0) mbar_wait(&bars[st], (uint32_t)s_pending[st], p.status);
    if (XS) mbar_wait(&bar_x, 0u, p.status);  // (returns at once unless its first wait failed)
  }
  if (ep != 0xffffffffu) {
    if (tid == 0) red_max_u32(reinterpret_cast<unsigned*>(p.sync + WS_SYNC_EPOCH), ep);
    return;
  }
  if (tid == 0) {
    __threadfence();
    s_flag = (atomicAdd(exit_cnt, 1) == G - 1) ? 1 : 0;
  }
  __syncthreads();
  if (s_flag) {
    __threadfence();
    uint4* area = reinterpret_cast<uint4*>(p.dots);
    for (size_t w = tid; w < (DX_END - DX_DOTS) / 16; w += DF_THREADS) area[w] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      p.sync[WS_SYNC_EPOCH] = 0;
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
    if (grid < 32) return cudaErrorInvalidConfiguration;  // router rows per CTA are bounded by 16
    if (dev >= 0 && dev < 64) g_info[dev].grid[vi] = grid;
  }
  // cooperative (every CTA resident: the layer's exchanges wait on one another), and with programmatic
  // stream serialisation: the kernel's constant-weight loads may overlap the previous kernel's tail;
  // it waits for that kernel (griddepcontrol.wait) before reading anything else
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(DF_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  STRATA_LAUNCH(KID_DECODE_LAYER, s, err = cudaLaunchKernelEx(&cfg, kern, prm));
  return err;
}

// Wait self-test: one CTA of the layer's shape runs the layer's two bounded waits on conditions that
// never hold -- a poll of an exchange word for a tag nothing writes, and an mbarrier phase nothing
// completes -- with a short limit; each expires, records ST_TIMEOUT in the status word and returns.
__global__ void __launch_bounds__(DF_THREADS) wait_selftest_kernel(const uint64_t* word, uint32_t tag,
                                                                   unsigned long long limit_ns, int* status) {
  __shared__ float s_dst[DF_THREADS];
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  poll_tagged<1>(word, [](int) { return 0; }, 1, tag, s_dst, status, limit_ns);
  if (threadIdx.x == 0) mbar_wait(&bar, 0u, status, limit_ns);  // no arrival ever comes
}

}  // namespace

cudaError_t launch_wait_selftest(const uint64_t* word, uint32_t tag, unsigned long long limit_ns, int* status,
                                 cudaStream_t s) {
  STRATA_LAUNCH(KID_WAIT_SELFTEST, s, wait_selftest_kernel<<<1, DF_THREADS, 0, s>>>(word, tag, limit_ns, status));
  return cudaGetLastError();
}

cudaError_t launch_decode_fused(const strata_experts_t& ex, const uint16_t* w_router, const float* bias,
                                const float* x, int T, int residual, int alias, float* out, int32_t* ids, float* weights,
                                const DecodeNext* next, const WsLayout& L, char* ws, cudaStream_t s) {
  DecodeParams prm;
  prm.x = x;
  prm.out = out;
  prm.T = T;
  prm.E = ex.n_expert;
  prm.q2_offset = ex.q2_offset;
  prm.residual = residual;
  prm.alias = alias;
  prm.wr = w_router;
  prm.bias = bias;
  prm.blobs = (const uint8_t*)ex.blobs;
  prm.stride = ex.blob_stride;
  prm.shared = (const uint8_t*)ex.shared_blob;
  prm.ids_out = ids;
  prm.w_out = weights;
  prm.dots = (uint64_t*)(ws + DX_DOTS);
  prm.htag = (uint64_t*)(ws + DX_H);
  prm.ptag = (uint64_t*)(ws + DX_PARTS);
  prm.pred = (uint64_t*)(ws + DX_PRED);
  prm.pred_ids = (uint64_t*)(ws + DX_PRED_IDS);
  prm.wr_next = next ? next->wr : nullptr;
  prm.bias_next = next ? next->bias : nullptr;
  prm.blobs_next = next ? next->blobs : nullptr;
  prm.stride_next = next ? next->stride : 0;
  prm.sync = (int*)(ws + WS_SYNC);
  prm.status = (int*)(ws + L.status);
  if (T <= 1) return launch_tt<1>(prm, s);
  if (T <= 2) return launch_tt<2>(prm, s);
  if (T <= 4) return launch_tt<4>(prm, s);
  return launch_tt<8>(prm, s);
}

}  // namespace strata
