// Q2_0 expert FFN, GEMV-style path (step 4 of the block), sm_103a.
//
// ai.thesatyajit.com "Strata engine", section "The CPU kernels": Q2_0 codes {0,1,2,3} mean
// {-1,0,1,2} x scale, and a correction term removes the offset once per block instead of per
// weight.  Restated for the GPU: with activations quantised per 64-block to 16-bit integers
// q ~= v / s (split into a signed high and an unsigned low byte), a block contributes
//     d * s * (sum_i c_i q_i - q2_offset * sum_i q_i)
// and sum_i c_i q_i is formed exactly with dp4a on the raw code bytes: masking code word w with
// (3 << 2m) leaves c * 4^m in every byte, so four masks give four integer sums that recombine
// with shifts.  momoyeyu.github.io "ai-infra-strata", section "提示词处理": one read of an expert's
// weights serves every token routed to it -- a CTA handles up to NT tokens of one expert.
//
// Weights move global -> shared with cp.async.bulk into a ring of stages, each completed on an
// mbarrier; every wait is bounded by %globaltimer and reports STRATA_E_TIMEOUT via the status word.
#include "device_common.cuh"

namespace strata {
namespace {

constexpr int NSTAGE = 8;
// Ring of NSTAGE weight chunks of CHUNK bytes: stage i holds chunk i, i + NSTAGE, ...
template <int CHUNK>
struct Ring {
  uint8_t* buf;   // NSTAGE * CHUNK bytes, 16-aligned
  uint64_t* bar;  // NSTAGE barriers
  const uint8_t* src;
  int n;          // chunks to stream
};

template <int CHUNK>
__device__ __forceinline__ void ring_issue(const Ring<CHUNK>& r, int i) {
  const int s = i % NSTAGE;
  mbar_expect_tx(&r.bar[s], CHUNK);
  bulk_g2s(r.buf + (size_t)s * CHUNK, r.src + (size_t)i * CHUNK, CHUNK, &r.bar[s]);
}

// ---------------------------------------------------------------------------------------------
// gate/up + SwiGLU.  CTA = (tile, row tile rt, k split s); thread = one of the 128 rows.
// With S > 1 each CTA writes partial sums; the last of the S CTAs of (tile, rt) adds them in
// split order, applies silu(g) * u and quantises h for the down projection.
// ---------------------------------------------------------------------------------------------
template <int S>
__global__ void __launch_bounds__(128) gateup_kernel(const uint8_t* __restrict__ blobs, int64_t stride,
                                                     const Tile* __restrict__ tiles,
                                                     const int32_t* __restrict__ n_active_tiles,
                                                     const int32_t* __restrict__ pair,
                                                     const QBlock* __restrict__ qx, float* __restrict__ partial,
                                                     int* __restrict__ cnt_gu, QBlock* __restrict__ hq,
                                                     int q2_offset, int* __restrict__ status) {
  constexpr int KBS = KB_GU / S;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring_buf = smem;                                            // NSTAGE * GU_CHUNK
  QBlock* sq = reinterpret_cast<QBlock*>(smem + NSTAGE * GU_CHUNK);     // [KBS][NT]
  __shared__ uint64_t bars[NSTAGE];
  __shared__ float sh[NT][RT];
  __shared__ int32_t s_tmp[4][64];
  __shared__ int s_last;
  __shared__ int s_tok[NT];

  const int tile_idx = blockIdx.x / (RT_GU * S);
  const int rem = blockIdx.x % (RT_GU * S);
  const int rt = rem / S, sidx = rem % S;
  if (tile_idx >= n_active_tiles[1]) return;
  const Tile tl = tiles[tile_idx];
  const int n = tl.n;
  const int tid = threadIdx.x;
  const int kb0 = sidx * KBS;

  Ring<GU_CHUNK> ring{ring_buf, bars,
                      blobs + (int64_t)tl.e * stride + ((int64_t)rt * KB_GU + kb0) * GU_CHUNK, KBS};
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int i = 0; i < NSTAGE && i < KBS; ++i) ring_issue(ring, i);

  // tokens of this tile and their quantised activations for our k range
  if (tid < NT) s_tok[tid] = (tid < n) ? pair[tl.q0 + tid] / K : 0;
  __syncthreads();
  for (int i = tid; i < KBS * NT * 9; i += 128) {  // 144 B = 9 x 16 B per QBlock
    const int blk = i / 9, part = i % 9;
    const int kb = blk / NT, j = blk % NT;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (j < n) v = reinterpret_cast<const uint4*>(qx + (size_t)s_tok[j] * KB_GU + kb0 + kb)[part];
    reinterpret_cast<uint4*>(sq + blk)[part] = v;
  }
  __syncthreads();

  float accg[NT], accu[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) { accg[j] = 0.f; accu[j] = 0.f; }

  bool ok = true;
  for (int i = 0; i < KBS; ++i) {
    const int st = i % NSTAGE;
    if (!mbar_wait(&bars[st], (uint32_t)((i / NSTAGE) & 1), status)) { ok = false; break; }
    const uint8_t* chunk = ring_buf + (size_t)st * GU_CHUNK;
    const uint4 gc = *reinterpret_cast<const uint4*>(chunk + 16 * tid);
    const uint4 uc = *reinterpret_cast<const uint4*>(chunk + 2048 + 16 * tid);
    const __half2 sc = *reinterpret_cast<const __half2*>(chunk + 4096 + 4 * tid);
    const float dg = __low2float(sc), du = __high2float(sc);
    const Masked gm = mask_codes(gc), um = mask_codes(uc);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      if (j < n) {
        const QBlock& a = sq[i * NT + j];
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint4 h4 = reinterpret_cast<const uint4*>(a.hi)[w];
          const uint4 l4 = reinterpret_cast<const uint4*>(a.lo)[w];
          hi[4 * w] = h4.x; hi[4 * w + 1] = h4.y; hi[4 * w + 2] = h4.z; hi[4 * w + 3] = h4.w;
          lo[4 * w] = l4.x; lo[4 * w + 1] = l4.y; lo[4 * w + 2] = l4.z; lo[4 * w + 3] = l4.w;
        }
        const float s64 = a.s64;
        const int qoff = a.qoff;
        const int vg = dot64(gm, hi, lo) - qoff;
        const int vu = dot64(um, hi, lo) - qoff;
        accg[j] = fmaf(dg * s64, (float)vg, accg[j]);
        accu[j] = fmaf(du * s64, (float)vu, accu[j]);
      }
    }
    __syncthreads();  // every thread is done with stage st
    if (tid == 0 && i + NSTAGE < KBS) ring_issue(ring, i + NSTAGE);
  }
  if (!ok) return;

  if (S > 1) {
    float* pbase = partial + ((((size_t)tile_idx * RT_GU + rt) * S + sidx) * NT) * RT * 2;
#pragma unroll
    for (int j = 0; j < NT; ++j)
      if (j < n) reinterpret_cast<float2*>(pbase + (size_t)j * RT * 2)[tid] = make_float2(accg[j], accu[j]);
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&cnt_gu[tile_idx * RT_GU + rt], 1) == S - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      if (j < n) {
        float g = 0.f, u = 0.f;
        for (int s = 0; s < S; ++s) {
          const float2 v = __ldcg(reinterpret_cast<const float2*>(
              partial + ((((size_t)tile_idx * RT_GU + rt) * S + s) * NT + j) * RT * 2) + tid);
          g += v.x;
          u += v.y;
        }
        accg[j] = g;
        accu[j] = u;
      }
    }
    if (tid == 0) cnt_gu[tile_idx * RT_GU + rt] = 0;
  }
#pragma unroll
  for (int j = 0; j < NT; ++j)
    if (j < n) sh[j][tid] = silu_mul(accg[j], accu[j]);
  __syncthreads();
  // quantise h: (token j, half b) -> QBlock of slot q0 + j, down k-block 2*rt + b
  const int warp = tid >> 5, lane = tid & 31;
  for (int item = warp; item < 2 * n; item += 4) {
    const int j = item >> 1, b = item & 1;
    const float v0 = sh[j][64 * b + 2 * lane], v1 = sh[j][64 * b + 2 * lane + 1];
    quantise_block_warp(v0, v1, q2_offset, hq + (size_t)(tl.q0 + j) * KB_D + 2 * rt + b, s_tmp[warp]);
  }
}

// ---------------------------------------------------------------------------------------------
// down: CTA = (tile, row tile rt of 20); thread = one output row; parts[p][row] for every pair
// p of the tile.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(128) down_kernel(const uint8_t* __restrict__ blobs, int64_t stride,
                                                   const Tile* __restrict__ tiles,
                                                   const int32_t* __restrict__ n_active_tiles,
                                                   const int32_t* __restrict__ pair, const QBlock* __restrict__ hq,
                                                   float* __restrict__ parts, int* __restrict__ status) {
  __shared__ __align__(128) uint8_t ring_buf[KB_D * D_CHUNK];
  __shared__ __align__(16) QBlock sq[KB_D * NT];
  __shared__ uint64_t bars[KB_D];
  __shared__ int s_pair[NT];
  const int tile_idx = blockIdx.x / RT_D;
  const int rt = blockIdx.x % RT_D;
  if (tile_idx >= n_active_tiles[1]) return;
  const Tile tl = tiles[tile_idx];
  const int n = tl.n;
  const int tid = threadIdx.x;
  const uint8_t* src = blobs + (int64_t)tl.e * stride + D_REGION + (int64_t)rt * KB_D * D_CHUNK;
  if (tid == 0) {
    for (int s = 0; s < KB_D; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int i = 0; i < KB_D; ++i) {
      mbar_expect_tx(&bars[i], D_CHUNK);
      bulk_g2s(ring_buf + i * D_CHUNK, src + (size_t)i * D_CHUNK, D_CHUNK, &bars[i]);
    }
  if (tid < NT) s_pair[tid] = (tid < n) ? pair[tl.q0 + tid] : 0;
  for (int i = tid; i < KB_D * NT * 9; i += 128) {
    const int blk = i / 9, part = i % 9;
    const int kb = blk / NT, j = blk % NT;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (j < n) v = reinterpret_cast<const uint4*>(hq + (size_t)(tl.q0 + j) * KB_D + kb)[part];
    reinterpret_cast<uint4*>(sq + blk)[part] = v;
  }
  __syncthreads();
  float acc[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) acc[j] = 0.f;
  for (int kb = 0; kb < KB_D; ++kb) {
    if (!mbar_wait(&bars[kb], 0u, status)) return;
    const uint8_t* chunk = ring_buf + kb * D_CHUNK;
    const uint4 c = *reinterpret_cast<const uint4*>(chunk + 16 * tid);
    const float d = __half2float(*reinterpret_cast<const __half*>(chunk + 2048 + 2 * tid));
    const Masked m = mask_codes(c);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      if (j < n) {
        const QBlock& a = sq[kb * NT + j];
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint4 h4 = reinterpret_cast<const uint4*>(a.hi)[w];
          const uint4 l4 = reinterpret_cast<const uint4*>(a.lo)[w];
          hi[4 * w] = h4.x; hi[4 * w + 1] = h4.y; hi[4 * w + 2] = h4.z; hi[4 * w + 3] = h4.w;
          lo[4 * w] = l4.x; lo[4 * w + 1] = l4.y; lo[4 * w + 2] = l4.z; lo[4 * w + 3] = l4.w;
        }
        const int v = dot64(m, hi, lo) - a.qoff;
        acc[j] = fmaf(d * a.s64, (float)v, acc[j]);
      }
    }
  }
  const int row = rt * RT + tid;
#pragma unroll
  for (int j = 0; j < NT; ++j)
    if (j < n) parts[(size_t)s_pair[j] * H + row] = acc[j];
}

}  // namespace

cudaError_t launch_experts_gemv(const strata_experts_t& ex, int T, const int32_t* pair, const WsLayout& L,
                                char* ws, float* parts, cudaStream_t s) {
  const uint8_t* blobs = (const uint8_t*)ex.blobs;
  const Tile* tiles = (const Tile*)(ws + L.tiles);
  const int32_t* nat = (const int32_t*)(ws + L.n_active);
  const QBlock* qx = (const QBlock*)(ws + L.qx);
  QBlock* hq = (QBlock*)(ws + L.hq);
  int* status = (int*)(ws + L.status);
  const int max_tiles = L.max_tiles;
  // decode-sized calls only (T <= DECODE_T_MAX); larger calls take the tensor-core path
  (void)T;
  constexpr int S = S_SPLIT;
  const size_t smem = NSTAGE * GU_CHUNK + sizeof(QBlock) * (KB_GU / S) * NT;
  cudaFuncSetAttribute(gateup_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  STRATA_LAUNCH(KID_GEMV_GATEUP, s,
                gateup_kernel<S><<<max_tiles * RT_GU * S, 128, smem, s>>>(
                    blobs, ex.blob_stride, tiles, nat, pair, qx, (float*)(ws + L.partial), (int*)(ws + L.cnt_gu), hq,
                    ex.q2_offset, status));
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  STRATA_LAUNCH(KID_GEMV_DOWN, s,
                down_kernel<<<max_tiles * RT_D, 128, 0, s>>>(blobs, ex.blob_stride, tiles, nat, pair, hq, parts, status));
  return cudaGetLastError();
}

}  // namespace strata
