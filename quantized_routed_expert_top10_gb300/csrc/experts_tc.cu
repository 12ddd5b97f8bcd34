// Q2_0 expert FFN on the tensor cores (tcgen05), for prefill chunks (T > 8), sm_103a.
//
// momoyeyu.github.io "ai-infra-strata", section "提示词处理": a prompt is cut into chunks, tokens are
// gathered per expert so one weight read serves all of them (W x becomes W X), and the kernel fuses
// the dequantisation with the matrix product.  ai.thesatyajit.com "Strata engine", "The CPU kernels":
// Q2_0 codes {0,1,2,3} mean {-1,0,1,2} x the block scale.  zwxr.cn news/242664, "一次路由的完整旅程":
// moe_combine adds the experts' outputs weighted by the router weights.
//
// Per expert e with n_e tokens (its slots in the grouping), two grouped GEMMs with the weights as the
// M = 128 operand ("swap AB") and the expert's tokens as N (up to 256 per tile):
//   gate/up:  [g; u] (2 x 128 rows x N) = [G_rt; U_rt] (128 x 2560) * X_e^T, h = silu(g) * u -> Hg (fp16)
//   down:     y_rt (128 rows x N) = D_rt (128 x 640) * H_e^T.  In a layer call the epilogue adds
//             w[t][k] * y into the layer output (fp32 reductions: the combine step, fused), so no
//             per-pair output is stored; strata_moe_experts stores y per pair instead.
// A tcgen05.mma costs its issuing thread about 100 cycles whatever N is, and one of N = 128 only ~70
// cycles of tensor time, so both kernels take the widest token tiles (N = 256): one MMA instruction
// then carries 128 x 256 x 16 multiply-adds.
// Warp roles in each persistent CTA (one per SM; work items = (tile, 128-row tile of the weights)):
//   warp 0      streams the token tile (gate/up: from Xg, the tokens copied once per layer into padded-slot
//               order by tc_gather_kernel; down: from Hg) and the Q2_0 code chunk of each 64-wide
//               k-block with cp.async.bulk into a 4-stage (gate/up) or 5-stage (down) ring;
//   warp 2      owns the TMEM allocation;
//   warps 4-11  dequantise the codes straight into the 128B-swizzled K-major shared-memory layout
//               (fp16: (c + 1024) built by one LOP3 per pair, minus (1024 + q2_offset), times d -- all
//               exact) in a 2-stage (gate/up) or 3-stage (down) ring of weight tiles, as two groups of
//               four warps taking alternate k-blocks;
//   warp 1      issues tcgen05.mma (fp16 x fp16 -> fp32) into TMEM (gate/up: one half for a tile of up to
//               128 tokens, both for a wider one; down: one half per item) and commits to the stages'
//               "empty" mbarriers;
//   warps 12-15 read the finished buffer with tcgen05.ld (one weight row per TMEM lane) and write the
//               epilogue while the next item accumulates into the other buffer; the down kernel runs
//               twelve more (warps 16-27, 896 threads), four warps per lane quadrant splitting the
//               columns.
// Every wait is bounded (STRATA_E_TIMEOUT).
//
// In-block order: the dequantiser emits the 64 weights of a block in the order pi (per 16 weights:
// 0,8,1,9,2,10,3,11,4,12,5,13,6,14,7,15), which is what one LOP3 per half2 produces from the packed
// codes; the token copy X16 and h (Hg) are stored in the same order, so every dot product is the
// same sum.
#include "tc_common.cuh"

namespace strata {
namespace {

constexpr int TCN = 256;        // max tokens per tile (MMA N)
constexpr int TCN_HALF = 128;   // tiles up to this wide take one half of TMEM (double-buffered)
constexpr uint32_t A_TILE = 128 * 128;      // 128 rows x 64 fp16

// Position in the emitted order (0..15) of weight j of a 16-group: the order is 0,8,1,9,..,7,15.
__host__ __device__ __forceinline__ int pi16_inv(int j) { return 2 * (j & 3) + 8 * ((j >> 2) & 1) + ((j >> 3) & 1); }

struct TcExpert { int32_t e, q0, n, q0pad; };    // grouping slots [q0, q0+n), padded rows from q0pad
struct TcTile { int32_t e, q0, n, q0pad; };      // <= 256 tokens of one expert

// ---------------------------------------------------------------------------------------------
// Tile list: experts' padded row ranges (multiples of 8) and tiles of at most 256 tokens.  The
// grouping may come from the caller, so it is checked before any tile is listed: every active entry
// must name an expert in [0, E) whose slot range lies in [0, P), the entries must be strictly
// increasing and their ranges in the same order without overlap (so the padded rows of all experts fit
// rows_cap).  Anything else sets ST_CORRUPT and lists no tile at all: the expert kernels then do
// nothing and every workspace offset they would derive stays unused.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(512) tc_prepare_kernel(const int32_t* __restrict__ expert_off,
                                                         const int32_t* __restrict__ active,
                                                         const int32_t* __restrict__ n_active, int E, int P,
                                                         TcExpert* __restrict__ exps, TcTile* __restrict__ tiles,
                                                         int32_t* __restrict__ counts, int max_tiles, int64_t rows_cap,
                                                         int shared_n, int* __restrict__ status) {
  __shared__ int s_pad[EMAX], s_full[EMAX], s_wide[EMAX], s_narrow[EMAX], s_scratch[32];
  __shared__ int s_e[EMAX], s_end[EMAX];
  __shared__ int s_bad;
  griddep_launch_dependents();
  griddep_wait();
  const int i = threadIdx.x;
  if (i == 0) s_bad = 0;
  const int na = max(0, min(*n_active, E));
  int e = -1, q0 = 0, n = 0;
  bool bad = false;
  if (i < na) {
    e = active[i];
    if (e >= 0 && e < E) {
      const int first = expert_off[e], end = expert_off[e + 1];
      if (first >= 0 && end >= first && end <= P) {
        q0 = first;
        n = end - first;
      } else {
        bad = true;
      }
    } else {
      bad = true;
    }
  }
  s_e[i] = e;
  s_end[i] = q0 + n;
  __syncthreads();
  if (i < na && i > 0 && (s_e[i - 1] >= e || s_end[i - 1] > q0)) bad = true;
  if (bad) s_bad = 1;
  __syncthreads();
  if (s_bad) {  // uniform over the CTA
    if (i == 0) {
      set_status(status, ST_CORRUPT);
      counts[0] = counts[1] = counts[2] = counts[3] = 0;
    }
    return;
  }
  s_pad[i] = (i < na) ? (n + 7) / 8 * 8 : 0;
  // gate/up tiles in three classes -- full (TCN tokens), other wide (> TCN_HALF), narrow -- listed in
  // that order, so each CTA's run of items changes between both-halves and one-half TMEM use once
  const int rem = n % TCN;
  s_full[i] = (i < na) ? n / TCN : 0;
  s_wide[i] = (i < na && rem > TCN_HALF) ? 1 : 0;
  s_narrow[i] = (i < na && rem > 0 && rem <= TCN_HALF) ? 1 : 0;
  __syncthreads();
  const int ppad = cta_exclusive_scan(s_pad, s_pad, EMAX, s_scratch);
  const int nfull = cta_exclusive_scan(s_full, s_full, EMAX, s_scratch);
  const int nwide = cta_exclusive_scan(s_wide, s_wide, EMAX, s_scratch);
  const int nnarrow = cta_exclusive_scan(s_narrow, s_narrow, EMAX, s_scratch);
  // a layer's shared expert (shared_n = T tokens, else 0): one more expert after the routed ones in
  // every list, marked e = -1, on virtual slots [P, P + T) (slot P + t = token t) and padded rows from ppad
  const int sfull = shared_n / TCN, srem = shared_n % TCN;
  const int swide = srem > TCN_HALF ? 1 : 0, snarrow = (srem > 0 && srem <= TCN_HALF) ? 1 : 0;
  const int wbase = nfull + sfull, nbase = wbase + nwide + swide;  // first wide / narrow tile
  const int ntiles = nbase + nnarrow + snarrow;
  const int ppad_all = ppad + (shared_n + 7) / 8 * 8;
  if ((int64_t)ppad_all + TCN > rows_cap) {  // cannot happen once the ranges are disjoint; kept as a bound
    if (i == 0) {
      set_status(status, ST_CORRUPT);
      counts[0] = counts[1] = counts[2] = counts[3] = 0;
    }
    return;
  }
  if (i < na) {
    exps[i] = TcExpert{e, q0, n, s_pad[i]};
    for (int t = 0; t < n / TCN; ++t) {
      const int idx = s_full[i] + t;
      if (idx < max_tiles) tiles[idx] = TcTile{e, q0 + t * TCN, TCN, s_pad[i] + t * TCN};
    }
    if (rem > 0) {
      const int t0 = n / TCN * TCN;
      const int idx = rem > TCN_HALF ? wbase + s_wide[i] : nbase + s_narrow[i];
      if (idx < max_tiles) tiles[idx] = TcTile{e, q0 + t0, rem, s_pad[i] + t0};
    }
  }
  if (i == 0 && shared_n > 0) {
    exps[na] = TcExpert{-1, P, shared_n, ppad};
    for (int t = 0; t < sfull; ++t)
      if (nfull + t < max_tiles) tiles[nfull + t] = TcTile{-1, P + t * TCN, TCN, ppad + t * TCN};
    if (srem > 0) {
      const int idx = swide ? wbase + nwide : nbase + nnarrow;
      if (idx < max_tiles) tiles[idx] = TcTile{-1, P + sfull * TCN, srem, ppad + sfull * TCN};
    }
  }
  if (i == 0) {
    counts[0] = na + (shared_n > 0 ? 1 : 0);
    counts[1] = min(ntiles, max_tiles);
    counts[2] = ppad_all;
    counts[3] = 0;  // unused (keeps slot_of, after the counts, 16-byte aligned)
  }
}

// X16 (see x16_store_chunk) of x for strata_moe_experts, times inv_rms[t] when given: one warp per
// token row.  A layer call gets X16 from the router's prep pass instead.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) tc_x16_kernel(const float* __restrict__ x, const float* __restrict__ inv_rms,
                                                     int T, uint8_t* __restrict__ x16) {
  griddep_launch_dependents();
  griddep_wait();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)t * H);
  const float sc = inv_rms ? __ldg(inv_rms + t) : 1.f;
#pragma unroll 4
  for (int i = 0; i < H / 128; ++i) tc::x16_store_chunk(__ldg(xr + lane + 32 * i), i, sc, t, T, x16);
}

// slot_of[p] = the grouping slot of pair p (the inverse of pair[]), -1 first for pairs a caller's
// grouping leaves out; a pair number outside [0, P) sets ST_CORRUPT and is skipped.
__global__ void __launch_bounds__(256) tc_slot_of_kernel(const int32_t* __restrict__ pair, int P,
                                                         int32_t* __restrict__ slot_of, int* __restrict__ status) {
  griddep_launch_dependents();
  griddep_wait();
  for (int j = blockIdx.x * 256 + threadIdx.x; j < P; j += gridDim.x * 256) {
    const int pr = pair[j];
    if (pr >= 0 && pr < P) slot_of[pr] = j;
    else set_status(status, ST_CORRUPT);
  }
}

// Xg[kb][row][128 B]: the padded-slot copy of the tokens the gate/up kernel bulk-copies its token tiles
// from (one contiguous run of rows per tile and k-block): row q0pad(e) + s of expert e holds X16 row
// (kb, token of the expert's slot s), its 16-byte chunks swizzled by row % 8 (the tensor core's 128B
// K-major layout, so a bulk copy of a row range is an MMA operand as it lands).  Token-major: one warp
// per token reads its 40 X16 rows once (lane = (k-block within a group of 4, chunk): 10 16-byte pieces)
// and writes them to the padded rows of its K slots (slot_of), and of its shared-expert slot P + t when
// the layer has one; each slot's expert comes from a binary search over the experts' first slots,
// staged in shared memory.  Rows of the 8-row padding between experts are not written: they only feed
// MMA columns the epilogues discard.
// ---------------------------------------------------------------------------------------------
constexpr int GATHER_THREADS = 256;
constexpr int GATHER_BLOCKS = 4 * 152;  // grid-stride over tokens; 4 CTAs per SM of a 152-SM GB300
__global__ void __launch_bounds__(GATHER_THREADS) tc_gather_kernel(const uint8_t* __restrict__ x16, int T,
                                                                   const int32_t* __restrict__ slot_of, int P,
                                                                   int shared, const TcExpert* __restrict__ exps,
                                                                   const int32_t* __restrict__ counts,
                                                                   uint8_t* __restrict__ xg, int64_t rows_cap) {
  __shared__ int s_q0[EMAX + 1], s_shift[EMAX + 1];  // the routed experts and a shared expert
  griddep_launch_dependents();
  griddep_wait();
  const int na = min(counts[0], EMAX + 1);
  for (int i = threadIdx.x; i < na; i += GATHER_THREADS) {
    const TcExpert ex = exps[i];
    s_q0[i] = ex.q0;
    s_shift[i] = ex.q0pad - ex.q0;  // padded row - slot
  }
  __syncthreads();
  if (na == 0) return;
  const int nslots = exps[na - 1].q0 + exps[na - 1].n;
  const int lane = threadIdx.x & 31, c = lane & 7, kb0 = lane >> 3;
  const int warps = gridDim.x * (GATHER_THREADS / 32);
  for (int t = blockIdx.x * (GATHER_THREADS / 32) + (threadIdx.x >> 5); t < T; t += warps) {
    uint4 v[KB_GU / 4];
    const uint8_t* src = x16 + (size_t)t * 128 + 16 * c;
#pragma unroll
    for (int i = 0; i < KB_GU / 4; ++i) v[i] = __ldg(reinterpret_cast<const uint4*>(src + (size_t)(kb0 + 4 * i) * T * 128));
    for (int k = 0; k < K + (shared ? 1 : 0); ++k) {
      const int slot = k < K ? __ldg(slot_of + (size_t)t * K + k) : P + t;
      if (slot < 0 || slot >= nslots) continue;  // a pair the caller's grouping leaves out
      int lo = 0, hi = na - 1;  // last expert whose first slot is <= slot
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_q0[mid] <= slot) lo = mid;
        else hi = mid - 1;
      }
      const int64_t row = (int64_t)slot + s_shift[lo];
      if (row < 0 || row >= rows_cap) continue;  // cannot happen for a checked grouping
      uint8_t* dst = xg + row * 128 + ((c ^ (int)(row & 7)) << 4);
#pragma unroll
      for (int i = 0; i < KB_GU / 4; ++i) *reinterpret_cast<uint4*>(dst + (int64_t)(kb0 + 4 * i) * rows_cap * 128) = v[i];
    }
  }
}

// Dequantise one 16-byte Q2_0 code row (64 weights, scale d) into the 8 swizzled 16-byte chunks of
// row r of a K-major tile.  Chunk c holds code bytes (c & 1) and 2 + (c & 1) of word c / 2, i.e.
// weights 4(c&1) .. +3 and 8 + 4(c&1) .. +3 of the 16-group c / 2; its half2 number m holds field m
// (bits 2m, 2m + 1) of both bytes.  OR-ing the field into the mantissa of M_m = 2^(10 - 2m), whose
// last-place unit sits at bit 2m, gives M_m + code in one LOP3; subtracting M_m + q2_offset and
// multiplying by d are exact.
struct DequantConsts {
  __half2 d2, sub[4];
  __device__ __forceinline__ DequantConsts(__half d, int q2_offset) : d2(__half2half2(d)) {
#pragma unroll
    for (int m = 0; m < 4; ++m) sub[m] = __half2half2(__float2half_rn((float)((1024 >> (2 * m)) + q2_offset)));
  }
};
// Chunk c of row r from the code word holding its bytes in bits 0..7 and 16..23.
__device__ __forceinline__ void dequant_chunk(uint32_t word, const DequantConsts& k, uint8_t* tile, int r, int c) {
  uint32_t out[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t magic = (uint32_t)((25 - 2 * m) << 10) * 0x00010001u;  // half2(2^(10 - 2m))
    const uint32_t bits = (word & (0x00030003u << (2 * m))) | magic;       // half2(M_m + code)
    __half2 h = *reinterpret_cast<const __half2*>(&bits);
    h = __hmul2(__hsub2(h, k.sub[m]), k.d2);                               // (code - q2_offset) * d
    out[m] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(tile + tc::swz_off(r, c)) = make_uint4(out[0], out[1], out[2], out[3]);
}
__device__ __forceinline__ void dequant_row(const uint4 codes, __half d, int q2_offset, uint8_t* tile, int r) {
  const DequantConsts k(d, q2_offset);
  const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
  for (int c = 0; c < 8; ++c) dequant_chunk((c & 1) ? (w[c >> 1] >> 8) : w[c >> 1], k, tile, r, c);
}
struct TcParams {
  const uint8_t* blobs;
  int64_t stride;
  const uint8_t* shared_blob;  // the layer's shared expert (tiles with e = -1), or null
  int q2_offset;
  const TcTile* tiles;
  const int32_t* counts;
  const uint8_t* act;   // gate/up: Xg [KB_GU][rows_cap][128 B]; down: Hg [KB_D][rows_cap][128 B]
  uint8_t* hg;          // gate/up output
  int64_t rows_cap;
  const int32_t* pair;  // slot -> pair
  int T;                // tokens
  int P;                // pairs (T * K)
  float* parts;         // down output per pair (strata_moe_experts), or null
  const float* wts;     // down, fused combine: router weights [T][K] (pair-indexed)
  float* out;           //                      layer output [T][H], already holding x (residual) or 0
  int* status;
};

// Kernel geometry.  Warp 0: copy producer; warp 1: MMA issuer; warp 2: TMEM owner; warps 4..11:
// dequantisers (two groups of 128 threads on alternate k-blocks, one weight row per thread: gate/up,
// that row of both matrices); warps 12..15 (down: 12..27): epilogue (one TMEM lane = one weight row
// per thread).
// gate/up (GU = true): item = (tile, row tile rt of gate and up): matrices gate_rt, up_rt.  TMEM: a
// tile of up to 128 tokens accumulates in half b (alternating) -- matrix j in columns [b*256 + j*128,
// +128) -- so its epilogue overlaps the next tile's main loop; a wider tile (up to 256 tokens, one
// dequantised weight tile serving all of them) takes both halves, matrix j in [j*256, +256).
// down (GU = false): item = (tile, row tile rt of down), one matrix in half b (alternating), columns
// [b*256, +256): every item's epilogue overlaps the next one's main loop.
// Threads per CTA: 16 warps for gate/up (its 125 registers per thread allow no more); the down kernel
// (at most 72 registers) runs 28, the last 16 of them epilogue warps, four per TMEM lane quadrant,
// because its epilogue -- 32k fp32 reductions per item, latency-bound -- is what it waits on.
template <bool GU>
constexpr int tc_epi_warps() { return GU ? 4 : 16; }
template <bool GU>
constexpr int tc_threads() { return 32 * (12 + tc_epi_warps<GU>()); }  // warps 0..11, then the epilogue
template <bool GU>
struct TcGeo {
  static constexpr int NMAT = GU ? 2 : 1;                 // weight matrices per item
  static constexpr int KBN = GU ? KB_GU : KB_D;          // k-blocks per item
  static constexpr int RTN = GU ? RT_GU : RT_D;          // weight row tiles per token tile
  static constexpr int CODE = GU ? GU_CHUNK : D_CHUNK;   // code bytes per k-block
  static constexpr uint32_t B_TILE = TCN * 128;          // token rows x 64 fp16
  static constexpr uint32_t TMA_STAGE = (B_TILE + CODE + 1023) / 1024 * 1024;  // token tile, then codes
  static constexpr int NS_TMA = GU ? 4 : 5;            // stages of (token tile, code chunks)
  // stages of dequantised weight tiles: down's k-block of MMAs is short, so it takes a third stage (the
  // dequantisers then work two k-blocks ahead of the tensor core)
  static constexpr int NS_A = GU ? 2 : 3;
  static constexpr uint32_t A_STAGE = NMAT * A_TILE;
  static constexpr uint32_t TMEM_COLS = 512;           // two halves of 256 columns
  static constexpr size_t SMEM = (size_t)NS_TMA * TMA_STAGE + (size_t)NS_A * A_STAGE + 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

// h = silu(g) * u for 16-column chunks [ch0, ch1) of a gate/up accumulator pair, by the warp of TMEM lane
// quadrant q (one weight row per thread): g in columns [0, mat_cols) of acc, u in [mat_cols, 2 mat_cols),
// written to Hg (fp16, the down kernel's operand layout).  The fast exponential and division (relative
// error ~1e-6) stay far below the fp16 rounding of h (2^-11).  The quadrant's 32 rows are half of one
// 64-wide k-block of h: 64 bytes of each token's Hg row.  Each chunk's 16 tokens x 64 bytes are put
// together in the warp's 1 KB of shared memory (stage) in Hg order, then written out as 16-byte pieces.
__device__ __forceinline__ void swiglu_chunks(const TcParams& p, const TcTile& tl, int rt, int q, uint32_t acc,
                                              uint32_t mat_cols, int ch0, int ch1, bool ok, uint8_t* stage) {
  const int lane = threadIdx.x & 31;
  const int pos = 16 * (lane >> 4) + pi16_inv(lane & 15);  // this row's place among the quadrant's 32
  uint8_t* hblk = p.hg + (int64_t)(2 * rt + (q >> 1)) * p.rows_cap * 128;  // the rows' k-block of Hg
  const int cbase = 4 * (q & 1);  // the quadrant's first 16-byte chunk in a 128-byte Hg row
#pragma unroll 1
  for (int ch = ch0; ch < ch1; ++ch) {
    uint32_t g[16], u[16];
    tc::tmem_ld16_async(acc + 16 * ch, g);
    tc::tmem_ld16_async(acc + mat_cols + 16 * ch, u);
    tc::tmem_wait_ld();
    if (ok) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float gv = __uint_as_float(g[i]), uv = __uint_as_float(u[i]);
        *reinterpret_cast<__half*>(stage + i * 64 + 2 * pos) = __float2half_rn(__fdividef(gv * uv, 1.f + __expf(-gv)));
      }
    }
    __syncwarp();
    if (ok) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {  // pieces lane and lane + 32: token i, chunk c
        const int i = (lane >> 2) + 8 * r, c = lane & 3;
        const int col = 16 * ch + i;
        if (col < tl.n) {
          const int hrow = tl.q0pad + col;
          *reinterpret_cast<uint4*>(hblk + (int64_t)hrow * 128 + ((((cbase + c) ^ hrow) & 7) << 4)) =
              *reinterpret_cast<const uint4*>(stage + i * 64 + 16 * c);
        }
      }
    }
    __syncwarp();
  }
}

// A 256-token gate/up tile takes both TMEM halves, so the next item's MMAs wait until its epilogue has
// drained them; the two dequantising warps of each lane quadrant (idle then: they have prepared the next
// item's first stages) take part of it.  Chunks of 16 columns are split in three: [0, a) for the epilogue
// warp, [a, b) for dequantiser warp 4 + q, [b, n) for warp 8 + q.
__device__ __forceinline__ void wide_split(int nch, int part, int& c0, int& c1) {
  const int a = (nch + 2) / 3, b = a + (nch - a + 1) / 2;
  c0 = part == 0 ? 0 : (part == 1 ? a : b);
  c1 = part == 0 ? a : (part == 1 ? b : nch);
}
constexpr int WIDE_BAR = 3;  // named barriers 3..6: epilogue warp 12 + q with dequantiser warps 4 + q, 8 + q

// Items so far in each TMEM half (two counters read and bumped by selects, so that a runtime half
// number never indexes a local array).
struct HalfUses {
  int u0 = 0, u1 = 0;
  __device__ __forceinline__ int operator[](int h) const { return h ? u1 : u0; }
  __device__ __forceinline__ void bump(int h) {
    u0 += h ? 0 : 1;
    u1 += h ? 1 : 0;
  }
};

// Item -> (token tile of up to 256 tokens, weight row tile rt): one dequantised weight tile serves all
// of the tile's tokens.
template <bool GU>
__device__ __forceinline__ TcTile item_tile(const TcParams& p, int item, int& rt) {
  rt = item % TcGeo<GU>::RTN;
  return p.tiles[item / TcGeo<GU>::RTN];
}

template <bool GU>
__global__ void __launch_bounds__(tc_threads<GU>(), 1) tc_expert_kernel(const TcParams p) {
  using G = TcGeo<GU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* tma_ring = smem;
  constexpr int NS_TMA = G::NS_TMA;
  constexpr uint32_t B_TILE = G::B_TILE;
  uint8_t* a_ring = smem + (size_t)NS_TMA * G::TMA_STAGE;
  constexpr int NS_A = G::NS_A;
  __shared__ uint64_t full_tma[NS_TMA], empty_tma[NS_TMA], full_a[NS_A], empty_a[NS_A];
  __shared__ uint64_t tmem_full[2], tmem_empty[2], mma_done;
  __shared__ uint32_t tmem_base;
  __shared__ int s_ep_pair[GU ? 1 : TCN];   // down epilogue: token (fused) or pair of each column
  __shared__ float s_ep_w[GU ? 1 : TCN];     //                router weight of that pair (fused combine)
  // gate/up: h staging, 1 KB per warp that runs swiglu_chunks (epilogue warps 12..15 -> 0..3, the
  // dequantising warps 4..11 helping with 256-token tiles -> 4..11)
  __shared__ __align__(16) uint8_t s_hstage[GU ? 12 : 1][1024];
  __shared__ int s_fail_flag;
  volatile int& s_fail = s_fail_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_launch_dependents();
  if (warp == 2) tc::tmem_alloc(&tmem_base, G::TMEM_COLS);
  if (tid == 0) {
    for (int s = 0; s < NS_TMA; ++s) {
      mbar_init(&full_tma[s], 1);
      mbar_init(&empty_tma[s], 1);
    }
    for (int s = 0; s < NS_A; ++s) {
      mbar_init(&full_a[s], 4);  // the four warps of the dequantising group that fills it
      mbar_init(&empty_a[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], tc_epi_warps<GU>());
    }
    mbar_init(&mma_done, 1);
    fence_mbar_init();
    s_fail = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  griddep_wait();  // tile lists, token and h copies come from the kernels before
  const uint32_t tmem = tmem_base;
  const int n_items = p.counts[1] * G::RTN;
  int* status = p.status;

  if (warp == 0) {
    // ---------------- producer: token tile + code chunk per k-block ----------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      for (int item = blockIdx.x; item < n_items && !s_fail; item += gridDim.x) {
        int rt;
        const TcTile tl = item_tile<GU>(p, item, rt);
        if (tl.n == 0) continue;
        const int nrows = (tl.n + 15) / 16 * 16;
        const uint8_t* blob = tl.e >= 0 ? p.blobs + (int64_t)tl.e * p.stride : p.shared_blob;
        for (int kb = 0; kb < G::KBN; ++kb, ++it) {
          const int s = it % NS_TMA;
          if (it >= NS_TMA && !mbar_wait(&empty_tma[s], (uint32_t)((it / NS_TMA - 1) & 1), status)) {
            s_fail = 1;
            break;
          }
          uint8_t* st = tma_ring + (size_t)s * G::TMA_STAGE;
          mbar_expect_tx(&full_tma[s], G::CODE + nrows * 128);
          bulk_g2s(st, p.act + ((int64_t)kb * p.rows_cap + tl.q0pad) * 128, nrows * 128, &full_tma[s]);
          if (GU) {
#pragma unroll
            for (int sl = 0; sl < RT / SLAB; ++sl)  // the tile's 8 slabs: one 576-byte piece each
              bulk_g2s_stream(st + B_TILE + sl * SLAB_KB,
                              blob + ((int64_t)(rt * (RT / SLAB) + sl) * KB_GU + kb) * SLAB_KB, SLAB_KB,
                              &full_tma[s], pol);
          } else {
            bulk_g2s_stream(st + B_TILE, blob + D_REGION + ((int64_t)rt * KB_D + kb) * D_CHUNK, D_CHUNK, &full_tma[s],
                            pol);
          }
        }
      }
      for (int back = 1; back <= NS_TMA && back <= it; ++back)  // copies still in flight after a failure
        mbar_wait(&full_tma[(it - back) % NS_TMA], (uint32_t)(((it - back) / NS_TMA) & 1), status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // One thread; its per-k-block work is all latency, so it waits only on full_a (every dequantiser
    // waits for the stage's copies before it arrives there, so full_a implies full_tma), keeps the
    // stage numbers, parities and descriptors incrementally and loads each item's tile one item ahead.
    if (lane == 0) {
      int n_small = 0;
      int s = 0, sa = 0;     // copy stage and weight stage of the next k-block
      uint32_t ph_a = 0;     // parity of sa's current use
      bool ready = false;    // the next k-block's full_a phase was seen complete
      HalfUses uses;  // items issued into each TMEM half so far
      const uint64_t bd0 = tc::smem_desc_sw128(smem_u32(tma_ring));
      const uint64_t ad00 = tc::smem_desc_sw128(smem_u32(a_ring));
      int rt_next = 0;
      TcTile tl_next = blockIdx.x < n_items ? item_tile<GU>(p, blockIdx.x, rt_next) : TcTile{0, 0, 0, 0};
      for (int item = blockIdx.x; item < n_items && !s_fail; item += gridDim.x) {
        const TcTile tl = tl_next;
        if (item + (int)gridDim.x < n_items) tl_next = item_tile<GU>(p, item + gridDim.x, rt_next);
        if (tl.n == 0) continue;
        const int nrows = (tl.n + 15) / 16 * 16;
        const uint32_t idesc = tc::idesc_f16_f32(128, nrows);
        // gate/up: a tile wider than 128 takes both halves (matrix j in half j); a narrower one takes
        // half b, alternating, matrix j at column b * 256 + 128 j.  down: half b, alternating.
        const bool wide = GU && nrows > TCN_HALF;
        const int b = wide ? 0 : (n_small++ & 1);
        bool okw = true;
        for (int h = 0; h < 2; ++h)
          if ((wide || h == b) && uses[h] >= 1)
            okw = okw && mbar_wait(&tmem_empty[h], (uint32_t)((uses[h] - 1) & 1), status);
        if (!okw) {
          s_fail = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t acc = tmem + (wide ? 0u : (uint32_t)b * 256u);
        const uint32_t mat_cols = wide ? 256u : 128u;
        for (int kb = 0; kb < G::KBN; ++kb) {
          if (!ready && !mbar_wait(&full_a[sa], ph_a, status)) {
            s_fail = 1;
            break;
          }
          tc::fence_after_sync();
          // descriptor address fields are (address >> 4) below 2^14: stage offsets add without carry
          const uint64_t bd = bd0 + (uint64_t)(s * (G::TMA_STAGE >> 4));
          const uint64_t ad0 = ad00 + (uint64_t)(sa * (G::A_STAGE >> 4));
          if (GU) {
            // the two matrices' MMAs alternate, so each accumulator's next MMA never waits on its last
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
              for (int mat = 0; mat < G::NMAT; ++mat)
                tc::mma_f16(acc + mat * mat_cols, ad0 + (uint64_t)((mat * A_TILE) >> 4) + 2 * kk, bd + 2 * kk, idesc,
                            (kb > 0 || kk > 0) ? 1u : 0u);
          } else {
            // down's k-block is four MMAs, shorter than the issuer's own loop: the next k-block's full_a
            // is tested while they issue
            const int sa1 = sa + 1 == NS_A ? 0 : sa + 1;
            const uint32_t ph1 = sa + 1 == NS_A ? (ph_a ^ 1u) : ph_a;
            ready = tc::mma_kblock_test_next(acc, ad0, bd, idesc, kb > 0 ? 1u : 0u, smem_u32(&full_a[sa1]), ph1) != 0;
          }
          tc::mma_commit(&empty_tma[s]);
          tc::mma_commit(&empty_a[sa]);
          if (++s == NS_TMA) s = 0;
          if (++sa == NS_A) {
            sa = 0;
            ph_a ^= 1u;
          }
        }
        if (s_fail) break;
        for (int h = 0; h < 2; ++h)
          if (wide || h == b) {
            tc::mma_commit(&tmem_full[h]);
            uses.bump(h);
          }
      }
      tc::mma_commit(&mma_done);  // every MMA this thread issued has finished before TMEM is released
      mbar_wait(&mma_done, 0u, status);
    }
  } else if (warp >= 4 && warp < 12) {
    // ---------------- dequantisers ----------------
    // Two groups of four warps take alternate k-blocks (items have an even number of them), so each
    // group's fixed cost per k-block -- its waits, the proxy fence, the arrival -- comes every other
    // k-block; each thread expands one weight row (gate/up: that row of both matrices).
    const int grp = (warp - 4) >> 2;
    const int row = (tid - 128) & 127;
    // the group's k-blocks are it = grp, grp + 2, ... (counted over all items): copy stage s = it % NS_TMA
    // and weight stage sa = it % NS_A, with the parities of it / NS_TMA and it / NS_A, kept incrementally
    // (a step of two k-blocks wraps each ring at most once: NS_A, NS_TMA >= 2)
    static_assert(NS_A >= 2 && NS_TMA >= 2 && G::KBN % 2 == 0, "two groups on alternate k-blocks");
    int it = grp, s = grp, sa = grp % NS_A;
    uint32_t ph_t = 0, ph_a = 0;
    bool ok = true;
    // gate/up: the TMEM use of every item, tracked as the issuer assigns it, so that a 256-token tile's
    // epilogue can be joined once the next item's first NS_A stages are dequantised (or after the last item)
    int n_small = 0;
    HalfUses uses;
    struct Pending { bool wide; TcTile tl; int rt; uint32_t par0, par1; };
    Pending pend{false, TcTile{0, 0, 0, 0}, 0, 0u, 0u};
    auto help_wide = [&](const Pending& pd) {
      ok = ok && mbar_wait(&tmem_full[0], pd.par0, status);
      ok = ok && mbar_wait(&tmem_full[1], pd.par1, status);
      tc::fence_after_sync();
      int c0, c1;
      wide_split((pd.tl.n + 15) / 16, warp < 8 ? 1 : 2, c0, c1);
      swiglu_chunks(p, pd.tl, pd.rt, warp & 3, tmem + ((uint32_t)(32 * (warp & 3)) << 16), 256u, c0, c1, ok,
                    s_hstage[warp]);
      tc::fence_before_sync();
      named_barrier(WIDE_BAR + (warp & 3), 96);
    };
    int rt_next = 0;
    TcTile tl_next = blockIdx.x < n_items ? item_tile<GU>(p, blockIdx.x, rt_next) : TcTile{0, 0, 0, 0};
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const int rt_cur = rt_next;
      const TcTile tl_cur = tl_next;  // loaded one item ahead
      if (item + (int)gridDim.x < n_items) tl_next = item_tile<GU>(p, item + gridDim.x, rt_next);
      if (tl_cur.n == 0) continue;
      Pending cur{false, tl_cur, rt_cur, (uint32_t)(uses[0] & 1), (uint32_t)(uses[1] & 1)};
      if (GU) {
        const bool wide = (tl_cur.n + 15) / 16 * 16 > TCN_HALF;
        const int b = wide ? 0 : (n_small++ & 1);
        cur.wide = wide;
        for (int h = 0; h < 2; ++h)
          if (wide || h == b) uses.bump(h);
      }
      for (int kb = grp; kb < G::KBN; kb += 2) {
        if (GU && kb >= NS_A && pend.wide) {  // the group's stages of this item are filled
          help_wide(pend);
          pend.wide = false;
        }
        if (it >= NS_A) ok = ok && mbar_wait(&empty_a[sa], ph_a ^ 1u, status);  // MMAs of k-block it - NS_A
        ok = ok && mbar_wait(&full_tma[s], ph_t, status);
        if (ok) {
          const uint8_t* code = tma_ring + (size_t)s * G::TMA_STAGE + B_TILE;
          uint8_t* ast = a_ring + (size_t)sa * G::A_STAGE;
          // gate/up: 8 slab pieces {gate codes, up codes, {gate d, up d} per row}; down: one chunk
          if (GU) {
            const uint8_t* pc = code + (row / SLAB) * SLAB_KB;
            const int rr = row % SLAB;
            const uint4 cg = *reinterpret_cast<const uint4*>(pc + 16 * rr);
            const uint4 cu = *reinterpret_cast<const uint4*>(pc + 256 + 16 * rr);
            const __half dg = *reinterpret_cast<const __half*>(pc + 512 + 4 * rr);
            const __half du = *reinterpret_cast<const __half*>(pc + 512 + 4 * rr + 2);
            dequant_row(cg, dg, p.q2_offset, ast, row);
            dequant_row(cu, du, p.q2_offset, ast + A_TILE, row);
          } else {
            const uint4 cw = *reinterpret_cast<const uint4*>(code + 16 * row);
            const __half d = *reinterpret_cast<const __half*>(code + 2048 + 2 * row);
            dequant_row(cw, d, p.q2_offset, ast, row);
          }
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_a[sa]);
        it += 2;
        s += 2;
        if (s >= NS_TMA) {
          s -= NS_TMA;
          ph_t ^= 1u;
        }
        sa += 2;
        if (sa >= NS_A) {
          sa -= NS_A;
          ph_a ^= 1u;
        }
      }
      if (GU) {
        if (pend.wide) help_wide(pend);  // an item shorter than NS_A k-blocks (never for gate/up)
        pend = cur;
      }
    }
    if (GU && pend.wide) help_wide(pend);
  } else if (warp >= 12) {
    // ---------------- epilogue ----------------
    constexpr int EPI = tc_epi_warps<GU>();
    const int q = warp & 3;
    const int epart = (warp - 12) >> 2;  // down: which part of each item's 16-column chunks this warp drains
    // down, fused combine: the layer output's lines stay in L2 while every expert adds into them
    const uint64_t keep = tc::policy_evict_last();
    const int etid = tid - 12 * 32;      // 0 .. 32 * EPI - 1
    int n_small = 0;
    HalfUses uses;  // items drained from each TMEM half so far (same assignment as the issuer)
    bool ok = true;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      int rt;
      const TcTile tl = item_tile<GU>(p, item, rt);
      if (tl.n == 0) continue;
      const int nrows = (tl.n + 15) / 16 * 16;
      const bool wide = GU && nrows > TCN_HALF;
      const int b = wide ? 0 : (n_small++ & 1);
      for (int h = 0; h < 2; ++h)
        if (wide || h == b) ok = ok && mbar_wait(&tmem_full[h], (uint32_t)(uses[h] & 1), status);
      tc::fence_after_sync();
      const uint32_t acc = tmem + (wide ? 0u : (uint32_t)b * 256u) + ((uint32_t)(32 * q) << 16);
      const uint32_t mat_cols = wide ? 256u : 128u;
      if (GU) {
        const int nch = nrows / 16;
        int c0 = 0, c1 = nch;
        if (wide) wide_split(nch, 0, c0, c1);
        swiglu_chunks(p, tl, rt, q, acc, mat_cols, c0, c1, ok, s_hstage[warp - 12]);
        if (wide) {  // the dequantising warps of this quadrant drain the rest
          tc::fence_before_sync();
          named_barrier(WIDE_BAR + q, 96);
        }
      } else {
        // the tile's pairs (and router weights) staged once per item by the epilogue threads
        named_barrier(2, 32 * EPI);  // every epilogue thread is done with the previous item's
        // fused combine: (token, router weight) of each column, the shared expert's slots P + t with
        // weight 1; strata_moe_experts: the pair number
        if (etid < tl.n) {
          const int slot = tl.q0 + etid;
          int pr = slot < p.P ? __ldg(p.pair + slot) : -1;
          if (slot < p.P && (pr < 0 || pr >= p.P)) pr = -1;
          if (p.out) {
            s_ep_pair[etid] = slot >= p.P ? slot - p.P : (pr >= 0 ? pr / K : -1);
            s_ep_w[etid] = slot >= p.P ? 1.f : (pr >= 0 ? __ldg(p.wts + pr) : 0.f);
          } else {
            s_ep_pair[etid] = pr;
          }
        }
        named_barrier(2, 32 * EPI);
        // each 4 x 4 block of (rows, columns) is transposed across 4 lanes, so that lane 4g + j writes
        // rows 4g .. 4g + 3 of column j: one 16-byte reduction (or store) instead of four
        const int j4 = lane & 3;
        const int orow = rt * 128 + 32 * q + 4 * (lane >> 2);
        constexpr int EPARTS = EPI / 4;  // warps per TMEM lane quadrant
        const int nch = nrows / 16, per = (nch + EPARTS - 1) / EPARTS;
#pragma unroll 1
        for (int ch = epart * per; ch < min(nch, (epart + 1) * per); ++ch) {
          uint32_t y[16];
          tc::tmem_ld16_async(acc + 16 * ch, y);
          tc::tmem_wait_ld();
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            uint32_t a[4] = {y[4 * m], y[4 * m + 1], y[4 * m + 2], y[4 * m + 3]};
            tc::transpose4_lanes(a, j4);
            const int col = 16 * ch + 4 * m + j4;
            const int pr = col < tl.n ? s_ep_pair[col] : -1;
            if (ok && pr >= 0 && pr < (p.out ? p.T : p.P)) {
              if (p.out) {  // fused combine: out[t] += w[t][k] * y (pr: the token here)
                const float w = s_ep_w[col];
                tc::red_add_v4_f32_hint(p.out + (size_t)pr * H + orow, w * __uint_as_float(a[0]),
                                        w * __uint_as_float(a[1]), w * __uint_as_float(a[2]),
                                        w * __uint_as_float(a[3]), keep);
              } else {
                *reinterpret_cast<uint4*>(p.parts + (size_t)pr * H + orow) = make_uint4(a[0], a[1], a[2], a[3]);
              }
            }
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0)
        for (int h = 0; h < 2; ++h)
          if (wide || h == b) mbar_arrive(&tmem_empty[h]);
      for (int h = 0; h < 2; ++h)
        if (wide || h == b) uses.bump(h);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc::tmem_dealloc(tmem, G::TMEM_COLS);
    tc::tmem_relinquish();
  }
}

int g_sms[64];

}  // namespace

// Rows of the padded h buffer Hg for a call with T tokens (every expert's slot range rounded up to 8
// rows, plus a tile's width of slack for the last tile's over-read).
int64_t tc_rows_cap(int T) { return (int64_t)T * (K + 1) + 8 * (EMAX + 1) + TCN; }
size_t tc_x16_bytes(int T) { return (size_t)KB_GU * T * 128; }
size_t tc_xg_bytes(int T) { return (size_t)KB_GU * tc_rows_cap(T) * 128; }
size_t tc_hg_bytes(int T) { return (size_t)KB_D * tc_rows_cap(T) * 128; }
// tile capacity: every expert's tiles plus the shared expert's (T more slots, one more expert)
inline int tc_max_tiles(int T) { return T * (K + 1) / TCN + EMAX + 1; }
size_t tc_meta_bytes(int T) {  // experts, tile list, counts [4], slot_of [T * K]
  return sizeof(TcExpert) * (EMAX + 1) + sizeof(TcTile) * (size_t)tc_max_tiles(T) +
         sizeof(int32_t) * (4 + (size_t)T * K) + 64;
}

cudaError_t launch_x16(const float* x, const float* inv_rms, int T, uint8_t* x16, cudaStream_t s) {
  STRATA_LAUNCH(KID_ROUTER_PREP, s, launch_pdl(tc_x16_kernel, (T + 7) / 8, 256, 0, s, x, inv_rms, T, x16));
  return cudaGetLastError();
}

cudaError_t launch_experts_tc(const strata_experts_t& ex, const uint8_t* x16, int T, const int32_t* expert_off,
                              const int32_t* pair, const int32_t* active, const int32_t* n_active, float* parts,
                              const float* weights, float* out, uint8_t* xg, uint8_t* hg, uint8_t* meta, int* status,
                              cudaStream_t s, const void* shared_blob) {
  const int max_tiles = tc_max_tiles(T);
  TcExpert* exps = reinterpret_cast<TcExpert*>(meta);
  TcTile* tiles = reinterpret_cast<TcTile*>(meta + sizeof(TcExpert) * (EMAX + 1));
  int32_t* counts = reinterpret_cast<int32_t*>(tiles + max_tiles);
  const int64_t rows_cap = tc_rows_cap(T);
  STRATA_LAUNCH(KID_TC_PREPARE, s,
                launch_pdl(tc_prepare_kernel, 1, 512, 0, s, expert_off, active, n_active, ex.n_expert, T * K, exps, tiles,
                                                    counts, max_tiles, rows_cap,
                                                    shared_blob ? T : 0, status));
  int32_t* slot_of = counts + 4;  // [T * K], after the counts in the tile-list area
  cudaError_t err = cudaSuccess;
  // a layer call (out set) groups every pair itself, so every slot_of entry is written; a caller's
  // grouping (strata_moe_experts) may leave pairs out, whose entries must read -1
  if (!out && (err = cudaMemsetAsync(slot_of, 0xFF, sizeof(int32_t) * (size_t)T * K, s)) != cudaSuccess) return err;
  STRATA_LAUNCH(KID_TC_GATHER, s, launch_pdl(tc_slot_of_kernel, GATHER_BLOCKS, 256, 0, s, pair, T * K, slot_of, status));
  STRATA_LAUNCH(KID_TC_GATHER, s,
                launch_pdl(tc_gather_kernel, GATHER_BLOCKS, GATHER_THREADS, 0, s, x16, T, slot_of, T * K, shared_blob ? 1 : 0,
                                                                          exps, counts, xg, rows_cap));
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  int sms = (dev >= 0 && dev < 64) ? g_sms[dev] : 0;
  if (sms == 0) {
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) g_sms[dev] = sms;
  }
  TcParams gp{(const uint8_t*)ex.blobs, ex.blob_stride, (const uint8_t*)shared_blob, ex.q2_offset, tiles, counts, xg,
              hg, rows_cap, pair, T,
              T * K, nullptr, nullptr, nullptr, status};
  if ((err = cudaFuncSetAttribute(tc_expert_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)TcGeo<true>::SMEM)) != cudaSuccess)
    return err;
  STRATA_LAUNCH(KID_TC_GATEUP, s, launch_pdl(tc_expert_kernel<true>, sms, tc_threads<true>(), TcGeo<true>::SMEM, s, gp));
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  TcParams dp = gp;
  dp.act = hg;
  dp.parts = out ? nullptr : parts;
  dp.wts = weights;
  dp.out = out;
  if ((err = cudaFuncSetAttribute(tc_expert_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)TcGeo<false>::SMEM)) != cudaSuccess)
    return err;
  STRATA_LAUNCH(KID_TC_DOWN, s, launch_pdl(tc_expert_kernel<false>, sms, tc_threads<false>(), TcGeo<false>::SMEM, s, dp));
  return cudaGetLastError();
}

}  // namespace strata
