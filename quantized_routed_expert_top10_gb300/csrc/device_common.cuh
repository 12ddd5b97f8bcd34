// Device helpers shared by several kernels: bulk copies and mbarriers, bounded waits, top-k, scans.
#pragma once
#include "common.cuh"

namespace strata {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any wait in a correct run

// Programmatic dependent launch (launch_pdl): the next kernel on the stream may be scheduled once every
// CTA of this one has signalled; griddep_wait blocks until the previous kernel has completed and its
// memory is visible (at once for a kernel launched without the attribute).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t sm_id() {
  uint32_t v;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(v));
  return v;
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// Barrier among `threads` threads (whole warps) on hardware barrier `id` (0 is __syncthreads').
__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
// Bulk prefetch of global memory into L2 (16-byte aligned address, size % 16 == 0); no completion.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// global -> shared bulk copy completing on an mbarrier (16-byte aligned addresses, size % 16 == 0)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// the same with an L2 evict-first hint (data read exactly once)
__device__ __forceinline__ void bulk_g2s_stream(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// try_wait with a suspend-time hint: a thread whose phase has not completed sleeps until it does (or
// the hint runs out) instead of spinning, so waiting threads take no issue slots from their neighbours.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase; false (and ST_TIMEOUT recorded) if it never completed within
// limit_ns (the library's kernels use the default; the wait self-test passes a short one).  Each try
// sleeps at most 1 ms (or the limit, if shorter) before the clock is checked again.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  const uint32_t hint = (uint32_t)(limit_ns < 1000000ull ? limit_ns : 1000000ull);
  while (!mbar_try_wait_sleep(bar, parity, hint)) {
    if (globaltimer() - t0 > limit_ns) {
      set_status(status, ST_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Relaxed max with no reply.
__device__ __forceinline__ void red_max_u32(unsigned* p, unsigned v) {
  asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_relaxed(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// bf16 x 8 (one uint4) widened to fp32
__device__ __forceinline__ void bf16x8_to_f32(const uint4 w, float* f) {
  f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xffff0000u);
  f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xffff0000u);
  f[4] = __uint_as_float(w.z << 16); f[5] = __uint_as_float(w.z & 0xffff0000u);
  f[6] = __uint_as_float(w.w << 16); f[7] = __uint_as_float(w.w & 0xffff0000u);
}

// Orderable key of a logit: a larger float gets a larger unsigned key (-0 one below +0).  No number
// maps to 0, which marks an absent or removed entry.
__device__ __forceinline__ uint32_t logit_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

constexpr int TOPK_CAP = 64;  // candidates ranked directly; more (mass ties) take the round-by-round path
struct TopKScratch {          // one per warp, in shared memory
  uint2 cand[TOPK_CAP];       // (key, expert id)
  uint2 sel[K];               // rank k -> (key, expert id)
};

// top-k of one token by one warp.  logit(e) is the logit of expert e (E % 32 == 0, 32 <= E <= 512).
// The stable descending order of the softmax probabilities is the order of the logits (exp is
// increasing), equal logits by lower id; lane k (< K) returns the (id, weight) of rank k.
// Renormalisation: p_i / max(sum of the K selected p, 2^-14) with p_i = exp(l_i - max) / z.  The K
// largest of E probabilities sum to at least K / E >= 10 / 512 > 2^-14, so the clamp never binds and
// the weight is exp(l_i - l_0) / sum over the selected of exp(l_j - l_0); z is never needed.
// Selection: tau = the K-th largest of the 32 lane maxima; the K lanes whose maxima rank above it
// hold K keys >= tau, so every top-K key is >= tau.  The keys >= tau (typically 10-25) are compacted
// into shared memory and each is ranked by counting the candidates ahead of it (key, then lower id):
// a few short independent steps instead of K dependent warp-wide argmax rounds.
template <typename LogitFn>
__device__ __forceinline__ void top_k_warp_fn(LogitFn logit, int E, TopKScratch& sc, int* out_id, float* out_w) {
  const int lane = threadIdx.x & 31;
  const int per = E >> 5;
  uint32_t key[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) key[j] = (j < per) ? logit_key(logit(lane + 32 * j)) : 0u;
  uint32_t mk = key[0];
#pragma unroll
  for (int j = 1; j < 16; ++j) mk = max(mk, key[j]);
  int r = 0;  // rank of this lane's maximum among the lanes' (maximum, lane)
#pragma unroll
  for (int o = 1; o < 32; ++o) {
    const int src = (lane + o) & 31;
    const uint32_t v = __shfl_sync(0xffffffffu, mk, src);
    r += (v > mk || (v == mk && src < lane)) ? 1 : 0;
  }
  const uint32_t tau = __shfl_sync(0xffffffffu, mk, __ffs(__ballot_sync(0xffffffffu, r == K - 1)) - 1);
  const uint32_t below = (1u << lane) - 1u;
  int C = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const bool is = key[j] >= tau;
    const uint32_t bal = __ballot_sync(0xffffffffu, is);
    const int pos = C + __popc(bal & below);
    if (is && pos < TOPK_CAP) sc.cand[pos] = make_uint2(key[j], (uint32_t)(lane + 32 * j));
    C += __popc(bal);
  }
  __syncwarp();
  if (C <= TOPK_CAP) {
    for (int i = lane; i < C; i += 32) {
      const uint2 me = sc.cand[i];
      int rank = 0;
#pragma unroll 4
      for (int q = 0; q < C; ++q) {
        const uint2 o = sc.cand[q];
        rank += (o.x > me.x || (o.x == me.x && o.y < me.y)) ? 1 : 0;
      }
      if (rank < K) sc.sel[rank] = me;
    }
  } else {
    // more than TOPK_CAP keys tie around the threshold: K rounds of a warp argmax on (key, -id)
#pragma unroll 1
    for (int k = 0; k < K; ++k) {
      uint32_t bk = key[0];
      int bj = 0;
#pragma unroll
      for (int j = 1; j < 16; ++j)
        if (key[j] > bk) {
          bk = key[j];
          bj = j;
        }
      const uint32_t mx = __reduce_max_sync(0xffffffffu, bk);
      const uint32_t id = __reduce_min_sync(0xffffffffu, bk == mx ? (uint32_t)(lane + 32 * bj) : 0xffffffffu);
      if ((int)(id & 31u) == lane) {
        const int jw = (int)(id >> 5);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j == jw) key[j] = 0u;
      }
      if (lane == 0) sc.sel[k] = make_uint2(mx, id);
    }
  }
  __syncwarp();
  const uint2 me = sc.sel[lane < K ? lane : 0];
  const float l0 = key_logit(sc.sel[0].x);
  const float e = lane < K ? expf(key_logit(me.x) - l0) : 0.f;
  const float s = warp_sum(e);
  *out_id = (int)me.y;
  *out_w = e / s;
}

// Exclusive scan of cnt[0..E) (shared) by the whole CTA (blockDim multiple of 32, <= 1024); returns
// the total; out may alias cnt.  scratch: >= 32 shared ints.
__device__ __forceinline__ int cta_exclusive_scan(const int* cnt, int* out, int E, int* scratch) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int per = (E + nt - 1) / nt;
  const int b0 = tid * per;
  int local = 0;
  for (int i = 0; i < per; ++i)
    if (b0 + i < E) local += cnt[b0 + i];
  const int lane = tid & 31, warp = tid >> 5;
  int v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const int nw = nt >> 5;
    int w = (lane < nw) ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < nw) scratch[lane] = w;
  }
  __syncthreads();
  const int total = scratch[(nt >> 5) - 1];
  int run = v - local + (warp ? scratch[warp - 1] : 0);
  __syncthreads();
  for (int i = 0; i < per; ++i) {
    if (b0 + i < E) {
      const int c = cnt[b0 + i];
      out[b0 + i] = run;
      run += c;
    }
  }
  __syncthreads();
  return total;
}

// Stable scatter of pairs [p0, p1) by one warp: fill[e] (shared) holds the next slot of expert e, which
// receives pair number pair_base + p.  ids may be in shared or global memory; ids outside [0, E) are
// skipped.
__device__ __forceinline__ void stable_scatter_warp(const int32_t* ids, int p0, int p1, int E, int* fill,
                                                    int32_t* pair, int pair_base) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
  for (int base = p0; base < p1; base += 32) {
    const int p = base + lane;
    int e = (p < p1) ? ids[p] : -1;
    if (e >= E || e < 0) e = -1;
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & lt);
    int pos = 0;
    if (e >= 0) pos = fill[e] + rank;
    __syncwarp();
    if (e >= 0) {
      pair[pos] = pair_base + p;
      if ((same >> lane) == 1u) fill[e] += __popc(same);  // highest lane of the group
    }
    __syncwarp();
  }
}

}  // namespace strata
