// Q2_0 expert FFN on the tensor cores (tcgen05), for prefill chunks (T > 8), sm_103a.
//
// momoyeyu.github.io "ai-infra-strata", section "提示词处理": a prompt is cut into chunks, tokens are
// gathered per expert so one weight read serves all of them (W x becomes W X), and the kernel fuses
// the dequantisation with the matrix product.  ai.thesatyajit.com "Strata engine", "The CPU kernels":
// Q2_0 codes {0,1,2,3} mean {-1,0,1,2} x the block scale.
//
// Per expert e with n_e tokens (its slots in the grouping), two grouped GEMMs with the weights as the
// M = 128 operand ("swap AB") and the expert's tokens as N (up to 128 per tile):
//   gate/up:  [g; u] (2 x 128 rows x N) = [G_rt; U_rt] (128 x 2560) * X_e^T, h = silu(g) * u -> Hg (fp16)
//   down:     y (128 rows x N) = D_rt (128 x 640) * H_e^T -> parts[pair][row] (fp32)
// Warp roles in each persistent CTA (one per SM): warp 0 streams the Q2_0 code chunks and the token
// tile of each 64-wide k-block with cp.async.bulk; warps 4.. dequantise the codes straight into the
// 128B-swizzled K-major shared-memory layout (fp16: (c + 1024) built by one LOP3 per pair, minus
// (1024 + q2_offset), times d -- all exact); warp 1 issues tcgen05.mma (fp16 x fp16 -> fp32 in TMEM)
// and commits to the stage's "empty" mbarrier; after the last k-block the same dequant warps read the
// accumulators with tcgen05.ld for the epilogue.  Every wait is bounded (STRATA_E_TIMEOUT).
//
// In-block order: the dequantiser emits the 64 weights of a block in the order pi (per 16 weights:
// 0,8,1,9,2,10,3,11,4,12,5,13,6,14,7,15), which is what one LOP3 per half2 produces from the packed
// codes; the gathered tokens Xg and h (Hg) are stored in the same order, so every dot product is the
// same sum.
#include "tc_common.cuh"

namespace strata {
namespace {

constexpr int TCN = 128;        // max tokens per tile (MMA N)
constexpr int TC_NS = 4;        // ring stages
constexpr int GU_THREADS = 384; // warp 0 producer, warp 1 MMA, warps 4..11 dequant/epilogue
constexpr int DN_THREADS = 384;
constexpr uint32_t A_TILE = 128 * 128;      // 128 rows x 64 fp16
constexpr uint32_t B_TILE = TCN * 128;      // up to 128 token rows x 64 fp16

// position s (0..15) of the emitted order -> weight index within the 16; and its inverse
__host__ __device__ __forceinline__ int pi16(int s) { return ((s >> 1) & 3) + 4 * ((s >> 3) & 1) + 8 * (s & 1); }
__host__ __device__ __forceinline__ int pi16_inv(int j) { return 2 * (j & 3) + 8 * ((j >> 2) & 1) + ((j >> 3) & 1); }

struct TcExpert { int32_t e, q0, n, q0pad; };    // grouping slots [q0, q0+n), padded rows from q0pad
struct TcTile { int32_t e, q0, n, q0pad; };      // <= 128 tokens of one expert

// ---------------------------------------------------------------------------------------------
// Tile lists: experts' padded row ranges (multiples of 8) and tiles of at most 128 tokens.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(512) tc_prepare_kernel(const int32_t* __restrict__ expert_off,
                                                         const int32_t* __restrict__ active,
                                                         const int32_t* __restrict__ n_active, int E,
                                                         TcExpert* __restrict__ exps, TcTile* __restrict__ tiles,
                                                         int32_t* __restrict__ counts, int max_tiles) {
  __shared__ int s_pad[EMAX], s_nt[EMAX], s_scratch[32];
  const int i = threadIdx.x;
  const int na = min(*n_active, E);
  int e = 0, q0 = 0, n = 0;
  if (i < na) {
    e = active[i];
    q0 = expert_off[e];
    n = expert_off[e + 1] - q0;
  }
  s_pad[i] = (i < na) ? (n + 7) / 8 * 8 : 0;
  s_nt[i] = (i < na) ? (n + TCN - 1) / TCN : 0;
  __syncthreads();
  const int ppad = cta_exclusive_scan(s_pad, s_pad, EMAX, s_scratch);
  const int ntiles = cta_exclusive_scan(s_nt, s_nt, EMAX, s_scratch);
  if (i < na) {
    exps[i] = TcExpert{e, q0, n, s_pad[i]};
    for (int t = 0; t * TCN < n; ++t) {
      const int idx = s_nt[i] + t;
      if (idx < max_tiles) tiles[idx] = TcTile{e, q0 + t * TCN, min(TCN, n - t * TCN), s_pad[i] + t * TCN};
    }
  }
  if (i == 0) {
    counts[0] = na;
    counts[1] = min(ntiles, max_tiles);
    counts[2] = ppad;
  }
}

// ---------------------------------------------------------------------------------------------
// Xg[kb][row][128 B]: row = padded slot; fp16 x of the slot's token in pi order, swizzled by row % 8.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) tc_gather_kernel(const float* __restrict__ x, const int32_t* __restrict__ pair,
                                                        const TcExpert* __restrict__ exps,
                                                        const int32_t* __restrict__ counts, uint8_t* __restrict__ xg,
                                                        int64_t rows_cap) {
  const int kb = blockIdx.y;
  const int na = counts[0];
  for (int i = blockIdx.x; i < na; i += gridDim.x) {
    const TcExpert ex = exps[i];
    const int npad = (ex.n + 7) / 8 * 8;
    for (int idx = threadIdx.x; idx < npad * 8; idx += blockDim.x) {
      const int s = idx >> 3, c = idx & 7;
      uint4 out = make_uint4(0, 0, 0, 0);
      if (s < ex.n) {
        const int t = pair[ex.q0 + s] / K;
        const float* src = x + (size_t)t * H + kb * QK + 16 * (c >> 1);
        __half hv[8];
#pragma unroll
        for (int e8 = 0; e8 < 8; ++e8) hv[e8] = __float2half_rn(src[pi16(8 * (c & 1) + e8)]);
        out = *reinterpret_cast<uint4*>(hv);
      }
      const int64_t row = ex.q0pad + s;
      if (row < rows_cap)
        *reinterpret_cast<uint4*>(xg + ((int64_t)kb * rows_cap + row) * 128 + ((c ^ (row & 7)) << 4)) = out;
    }
  }
}

// Dequantise one 16-byte Q2_0 code row (64 weights, scale d) into 8 swizzled 16-byte chunks of row r.
// Chunks [c0, c0 + nc) only.
__device__ __forceinline__ void dequant_row(const uint4 codes, __half d, int q2_offset, uint8_t* tile, int r, int c0,
                                            int nc) {
  const __half2 magic_off = __half2half2(__float2half_rn(1024.f + (float)q2_offset));
  const __half2 d2 = __half2half2(d);
  const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    if (c < c0 || c >= c0 + nc) continue;
    const uint32_t word = w[c >> 1];
    const int base = (c & 1) ? 8 : 0;  // chunk 2q: pairs m = 0..3 (shift 2m); chunk 2q+1: shift 8 + 2m
    uint32_t out[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t bits = ((word >> (base + 2 * m)) & 0x00030003u) | 0x64006400u;  // half2(1024 + c)
      __half2 h = *reinterpret_cast<const __half2*>(&bits);
      h = __hmul2(__hsub2(h, magic_off), d2);                                         // (c - off) * d, exact
      out[m] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(tile + tc::swz_off(r, c)) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

struct TcGuParams {
  const uint8_t* blobs;
  int64_t stride;
  int q2_offset;
  const TcTile* tiles;
  const int32_t* counts;
  const uint8_t* xg;
  uint8_t* hg;
  int64_t rows_cap;
  int* status;
};

struct TcDnParams {
  const uint8_t* blobs;
  int64_t stride;
  int q2_offset;
  const TcTile* tiles;
  const int32_t* counts;
  const uint8_t* hg;
  int64_t rows_cap;
  const int32_t* pair;
  float* parts;
  int* status;
};

// Shared-memory plan of one stage (1024-aligned pieces): A tile(s), B tile, code chunk.
template <int NA, int CODE>
struct StagePlan {
  static constexpr uint32_t A_OFF = 0;
  static constexpr uint32_t B_OFF = NA * A_TILE;
  static constexpr uint32_t C_OFF = B_OFF + B_TILE;
  static constexpr uint32_t BYTES = (C_OFF + CODE + 1023) / 1024 * 1024;
};
using GuPlan = StagePlan<2, GU_CHUNK>;
using DnPlan = StagePlan<1, D_CHUNK>;

// ---------------------------------------------------------------------------------------------
// gate/up + SwiGLU.  Work item = (tile, row tile rt); TMEM: gate columns [0, 128), up [128, 256).
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(GU_THREADS, 1) gu_tc_kernel(const TcGuParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full_tma[TC_NS], full_a[TC_NS], empty[TC_NS], tmem_full, tmem_empty, mma_done;
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 2) tc::tmem_alloc(&tmem_base, 256);
  if (tid == 0) {
    for (int s = 0; s < TC_NS; ++s) {
      mbar_init(&full_tma[s], 1);
      mbar_init(&full_a[s], 8);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tmem_full, 1);
    mbar_init(&tmem_empty, 8);
    mbar_init(&mma_done, 1);
    fence_mbar_init();
    s_fail = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const int n_items = p.counts[1] * RT_GU;
  int* status = p.status;

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      for (int item = blockIdx.x; item < n_items && !s_fail; item += gridDim.x) {
        const TcTile tl = p.tiles[item / RT_GU];
        const int rt = item % RT_GU;
        const int nrows = (tl.n + 15) / 16 * 16;
        const uint8_t* codes = p.blobs + (int64_t)tl.e * p.stride + (int64_t)rt * KB_GU * GU_CHUNK;
        for (int kb = 0; kb < KB_GU; ++kb, ++it) {
          const int s = it % TC_NS;
          if (it >= TC_NS && !mbar_wait(&empty[s], (uint32_t)((it / TC_NS - 1) & 1), status)) { s_fail = 1; break; }
          uint8_t* st = smem + s * GuPlan::BYTES;
          mbar_expect_tx(&full_tma[s], GU_CHUNK + nrows * 128);
          bulk_g2s_stream(st + GuPlan::C_OFF, codes + (int64_t)kb * GU_CHUNK, GU_CHUNK, &full_tma[s], pol);
          bulk_g2s(st + GuPlan::B_OFF, p.xg + ((int64_t)kb * p.rows_cap + tl.q0pad) * 128, nrows * 128, &full_tma[s]);
        }
      }
      // copies still in flight (only after a failed wait): let them land before the CTA leaves
      for (int back = 1; back <= TC_NS && back <= it; ++back)
        mbar_wait(&full_tma[(it - back) % TC_NS], (uint32_t)(((it - back) / TC_NS) & 1), status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int it = 0, ti = 0;
      for (int item = blockIdx.x; item < n_items && !s_fail; item += gridDim.x, ++ti) {
        const TcTile tl = p.tiles[item / RT_GU];
        const int nrows = (tl.n + 15) / 16 * 16;
        const uint32_t idesc = tc::idesc_f16_f32(128, nrows);
        if (ti > 0 && !mbar_wait(&tmem_empty, (uint32_t)((ti - 1) & 1), status)) { s_fail = 1; break; }
        tc::fence_after_sync();
        for (int kb = 0; kb < KB_GU; ++kb, ++it) {
          const int s = it % TC_NS;
          const uint32_t par = (uint32_t)((it / TC_NS) & 1);
          if (!mbar_wait(&full_tma[s], par, status) || !mbar_wait(&full_a[s], par, status)) { s_fail = 1; break; }
          tc::fence_after_sync();
          uint8_t* st = smem + s * GuPlan::BYTES;
          const uint64_t ag = tc::smem_desc_sw128(smem_u32(st + GuPlan::A_OFF));
          const uint64_t au = tc::smem_desc_sw128(smem_u32(st + GuPlan::A_OFF + A_TILE));
          const uint64_t bd = tc::smem_desc_sw128(smem_u32(st + GuPlan::B_OFF));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
            tc::mma_f16(tmem, ag + 2 * kk, bd + 2 * kk, idesc, acc);
            tc::mma_f16(tmem + 128, au + 2 * kk, bd + 2 * kk, idesc, acc);
          }
          tc::mma_commit(&empty[s]);
        }
        if (s_fail) break;
        tc::mma_commit(&tmem_full);
      }
      // every MMA this thread issued has finished before TMEM is released
      tc::mma_commit(&mma_done);
      mbar_wait(&mma_done, 0u, status);
    }
  } else if (warp >= 4) {
    // ---------------- dequant + epilogue (256 threads: row, matrix) ----------------
    const int dt = tid - 128;
    const int row = dt & 127, mat = dt >> 7;
    const int ew = warp - 4;               // epilogue warp 0..7; TMEM lane quadrant = warp % 4
    const int erow = 32 * (warp & 3) + lane;
    const int ehalf = ew >> 2;
    int it = 0, ti = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++ti) {
      const TcTile tl = p.tiles[item / RT_GU];
      const int rt = item % RT_GU;
      const int nrows = (tl.n + 15) / 16 * 16;
      bool ok = true;
      for (int kb = 0; kb < KB_GU; ++kb, ++it) {
        const int s = it % TC_NS;
        uint8_t* st = smem + s * GuPlan::BYTES;
        if (it >= TC_NS) ok = ok && mbar_wait(&empty[s], (uint32_t)((it / TC_NS - 1) & 1), status);
        ok = ok && mbar_wait(&full_tma[s], (uint32_t)((it / TC_NS) & 1), status);
        if (ok) {
          const uint4 cw = *reinterpret_cast<const uint4*>(st + GuPlan::C_OFF + (mat ? 2048 : 0) + 16 * row);
          const __half d = *reinterpret_cast<const __half*>(st + GuPlan::C_OFF + 4096 + 4 * row + 2 * mat);
          dequant_row(cw, d, p.q2_offset, st + GuPlan::A_OFF + mat * A_TILE, row, 0, 8);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&full_a[s]);
      }
      // epilogue: h = silu(g) * u for this CTA's 128 rows and the tile's tokens
      ok = ok && mbar_wait(&tmem_full, (uint32_t)(ti & 1), status);
      tc::fence_after_sync();
      const int nch = nrows / 16;
      const int ch0 = ehalf ? (nch + 1) / 2 : 0, ch1 = ehalf ? nch : (nch + 1) / 2;
      const int k = rt * 128 + erow;  // h index = down's contraction index
      const int kbd = k >> 6, k64 = k & 63;
      const int pos = 16 * (k64 >> 4) + pi16_inv(k64 & 15);
      for (int ch = ch0; ch < ch1; ++ch) {
        float g[16], u[16];
        const uint32_t lane_addr = (uint32_t)(32 * (warp & 3)) << 16;
        tc::tmem_ld16(tmem + lane_addr + 16 * ch, g);
        tc::tmem_ld16(tmem + lane_addr + 128 + 16 * ch, u);
        if (ok) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = 16 * ch + i;
            if (col < tl.n) {
              const int64_t hrow = tl.q0pad + col;
              __half* dst = reinterpret_cast<__half*>(p.hg + ((int64_t)kbd * p.rows_cap + hrow) * 128 +
                                                      (((pos >> 3) ^ (hrow & 7)) << 4)) + (pos & 7);
              *dst = __float2half_rn(silu_mul(g[i], u[i]));
            }
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tmem_empty);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) tc::tmem_dealloc(tmem, 256);
  if (warp == 2) tc::tmem_relinquish();
}

// ---------------------------------------------------------------------------------------------
// down.  Work item = (tile, row tile rtd); TMEM columns [0, 128).
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(DN_THREADS, 1) down_tc_kernel(const TcDnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full_tma[TC_NS], full_a[TC_NS], empty[TC_NS], tmem_full, tmem_empty, mma_done;
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 2) tc::tmem_alloc(&tmem_base, 128);
  if (tid == 0) {
    for (int s = 0; s < TC_NS; ++s) {
      mbar_init(&full_tma[s], 1);
      mbar_init(&full_a[s], 8);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tmem_full, 1);
    mbar_init(&tmem_empty, 8);
    mbar_init(&mma_done, 1);
    fence_mbar_init();
    s_fail = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const int n_items = p.counts[1] * RT_D;
  int* status = p.status;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      for (int item = blockIdx.x; item < n_items && !s_fail; item += gridDim.x) {
        const TcTile tl = p.tiles[item / RT_D];
        const int rtd = item % RT_D;
        const int nrows = (tl.n + 15) / 16 * 16;
        const uint8_t* codes = p.blobs + (int64_t)tl.e * p.stride + D_REGION + (int64_t)rtd * KB_D * D_CHUNK;
        for (int kb = 0; kb < KB_D; ++kb, ++it) {
          const int s = it % TC_NS;
          if (it >= TC_NS && !mbar_wait(&empty[s], (uint32_t)((it / TC_NS - 1) & 1), status)) { s_fail = 1; break; }
          uint8_t* st = smem + s * DnPlan::BYTES;
          mbar_expect_tx(&full_tma[s], D_CHUNK + nrows * 128);
          bulk_g2s_stream(st + DnPlan::C_OFF, codes + (int64_t)kb * D_CHUNK, D_CHUNK, &full_tma[s], pol);
          bulk_g2s(st + DnPlan::B_OFF, p.hg + ((int64_t)kb * p.rows_cap + tl.q0pad) * 128, nrows * 128, &full_tma[s]);
        }
      }
      // copies still in flight (only after a failed wait): let them land before the CTA leaves
      for (int back = 1; back <= TC_NS && back <= it; ++back)
        mbar_wait(&full_tma[(it - back) % TC_NS], (uint32_t)(((it - back) / TC_NS) & 1), status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0, ti = 0;
      for (int item = blockIdx.x; item < n_items && !s_fail; item += gridDim.x, ++ti) {
        const TcTile tl = p.tiles[item / RT_D];
        const int nrows = (tl.n + 15) / 16 * 16;
        const uint32_t idesc = tc::idesc_f16_f32(128, nrows);
        if (ti > 0 && !mbar_wait(&tmem_empty, (uint32_t)((ti - 1) & 1), status)) { s_fail = 1; break; }
        tc::fence_after_sync();
        for (int kb = 0; kb < KB_D; ++kb, ++it) {
          const int s = it % TC_NS;
          const uint32_t par = (uint32_t)((it / TC_NS) & 1);
          if (!mbar_wait(&full_tma[s], par, status) || !mbar_wait(&full_a[s], par, status)) { s_fail = 1; break; }
          tc::fence_after_sync();
          uint8_t* st = smem + s * DnPlan::BYTES;
          const uint64_t ad = tc::smem_desc_sw128(smem_u32(st + DnPlan::A_OFF));
          const uint64_t bd = tc::smem_desc_sw128(smem_u32(st + DnPlan::B_OFF));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) tc::mma_f16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(&empty[s]);
        }
        if (s_fail) break;
        tc::mma_commit(&tmem_full);
      }
      // every MMA this thread issued has finished before TMEM is released
      tc::mma_commit(&mma_done);
      mbar_wait(&mma_done, 0u, status);
    }
  } else if (warp >= 4) {
    const int dt = tid - 128;
    const int row = dt & 127, half = dt >> 7;  // dequant: each thread writes 4 of the row's 8 chunks
    const int ew = warp - 4;
    const int erow = 32 * (warp & 3) + lane;
    const int ehalf = ew >> 2;
    int it = 0, ti = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++ti) {
      const TcTile tl = p.tiles[item / RT_D];
      const int rtd = item % RT_D;
      const int nrows = (tl.n + 15) / 16 * 16;
      bool ok = true;
      for (int kb = 0; kb < KB_D; ++kb, ++it) {
        const int s = it % TC_NS;
        uint8_t* st = smem + s * DnPlan::BYTES;
        if (it >= TC_NS) ok = ok && mbar_wait(&empty[s], (uint32_t)((it / TC_NS - 1) & 1), status);
        ok = ok && mbar_wait(&full_tma[s], (uint32_t)((it / TC_NS) & 1), status);
        if (ok) {
          const uint4 cw = *reinterpret_cast<const uint4*>(st + DnPlan::C_OFF + 16 * row);
          const __half d = *reinterpret_cast<const __half*>(st + DnPlan::C_OFF + 2048 + 2 * row);
          dequant_row(cw, d, p.q2_offset, st + DnPlan::A_OFF, row, 4 * half, 4);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&full_a[s]);
      }
      ok = ok && mbar_wait(&tmem_full, (uint32_t)(ti & 1), status);
      tc::fence_after_sync();
      const int nch = nrows / 16;
      const int ch0 = ehalf ? (nch + 1) / 2 : 0, ch1 = ehalf ? nch : (nch + 1) / 2;
      const int orow = rtd * 128 + erow;
      for (int ch = ch0; ch < ch1; ++ch) {
        float y[16];
        tc::tmem_ld16(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 16 * ch, y);
        if (ok) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = 16 * ch + i;
            if (col < tl.n) p.parts[(size_t)p.pair[tl.q0 + col] * H + orow] = y[i];
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tmem_empty);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) tc::tmem_dealloc(tmem, 128);
  if (warp == 2) tc::tmem_relinquish();
}

int g_sms[64];

}  // namespace

// Rows of the padded, gathered token buffers for a call with T tokens (every expert's slot range
// rounded up to 8 rows, plus 128 rows of slack for the last tile's over-read).
int64_t tc_rows_cap(int T) { return (int64_t)T * K + 8 * EMAX + TCN; }
size_t tc_xg_bytes(int T) { return (size_t)KB_GU * tc_rows_cap(T) * 128; }
size_t tc_hg_bytes(int T) { return (size_t)KB_D * tc_rows_cap(T) * 128; }
size_t tc_meta_bytes(int T) {
  return sizeof(TcExpert) * EMAX + sizeof(TcTile) * (size_t)(T * K / TCN + EMAX) + 64;
}

cudaError_t launch_experts_tc(const strata_experts_t& ex, const float* x, int T, const int32_t* expert_off,
                              const int32_t* pair, const int32_t* active, const int32_t* n_active, float* parts,
                              uint8_t* xg, uint8_t* hg, uint8_t* meta, int* status, cudaStream_t s) {
  const int max_tiles = T * K / TCN + EMAX;
  TcExpert* exps = reinterpret_cast<TcExpert*>(meta);
  TcTile* tiles = reinterpret_cast<TcTile*>(meta + sizeof(TcExpert) * EMAX);
  int32_t* counts = reinterpret_cast<int32_t*>(meta + sizeof(TcExpert) * EMAX + sizeof(TcTile) * max_tiles);
  const int64_t rows_cap = tc_rows_cap(T);
  tc_prepare_kernel<<<1, 512, 0, s>>>(expert_off, active, n_active, ex.n_expert, exps, tiles, counts, max_tiles);
  tc_gather_kernel<<<dim3(256, KB_GU), 256, 0, s>>>(x, pair, exps, counts, xg, rows_cap);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  int sms = (dev >= 0 && dev < 64) ? g_sms[dev] : 0;
  if (sms == 0) {
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) g_sms[dev] = sms;
  }
  TcGuParams gp{(const uint8_t*)ex.blobs, ex.blob_stride, ex.q2_offset, tiles, counts, xg, hg, rows_cap, status};
  const size_t gsmem = (size_t)TC_NS * GuPlan::BYTES + 1024;
  if ((err = cudaFuncSetAttribute(gu_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gsmem)) != cudaSuccess)
    return err;
  gu_tc_kernel<<<sms, GU_THREADS, gsmem, s>>>(gp);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  TcDnParams dp{(const uint8_t*)ex.blobs, ex.blob_stride, ex.q2_offset, tiles, counts, hg, rows_cap, pair, parts, status};
  const size_t dsmem = (size_t)TC_NS * DnPlan::BYTES + 1024;
  if ((err = cudaFuncSetAttribute(down_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dsmem)) !=
      cudaSuccess)
    return err;
  down_tc_kernel<<<sms, DN_THREADS, dsmem, s>>>(dp);
  return cudaGetLastError();
}

}  // namespace strata
