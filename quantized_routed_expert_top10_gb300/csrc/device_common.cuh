// Device helpers shared by several kernels: bulk copies and mbarriers, bounded waits, top-k, scans.
#pragma once
#include "common.cuh"

namespace strata {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any wait in a correct run
constexpr float kRenormFloor = 6.103515625e-05f;            // 2^-14, ggml's lower clamp

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

// Bounded wait on an mbarrier phase; false (and ST_TIMEOUT recorded) if it never completed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      set_status(status, ST_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Orders this thread's earlier (generic-proxy) view of global memory before its later async-proxy
// accesses (cp.async.bulk reads of data that other threads wrote and released).
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Release reduction (fire and forget): every write this thread has observed -- its own, and the CTA's
// ordered before it by a barrier -- is visible device-wide before the add.
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Acquire-release add returning the old value.
__device__ __forceinline__ int atom_acq_rel_add(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void st_relaxed(int* p, int v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Bounded spin until *p >= target (one thread); false and ST_TIMEOUT if it never got there.
__device__ __forceinline__ bool spin_until_geq(const int* p, int target, int* status) {
  if (ld_acquire(p) >= target) return true;
  const unsigned long long t0 = globaltimer();
  while (ld_acquire(p) < target) {
    __nanosleep(64);
    if (globaltimer() - t0 > kWaitLimitNs) {
      set_status(status, ST_TIMEOUT);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// bf16 x 8 (one uint4) widened to fp32
__device__ __forceinline__ void bf16x8_to_f32(const uint4 w, float* f) {
  f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xffff0000u);
  f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xffff0000u);
  f[4] = __uint_as_float(w.z << 16); f[5] = __uint_as_float(w.z & 0xffff0000u);
  f[6] = __uint_as_float(w.w << 16); f[7] = __uint_as_float(w.w & 0xffff0000u);
}

// top-k of one token by one warp.  logit(e) is the logit of expert e (E % 32 == 0, E <= 512):
// softmax over E, the K largest probabilities in descending order (equal values: lower id first),
// renormalised as p / max(sum, 2^-14).  Lane k (< K) returns the (id, weight) of rank k.
// Each lane holds 16 candidates; every round takes a tree argmax over the lane's candidates and a
// butterfly argmax over the warp (a total order on (p, -id), so all lanes agree), then removes the
// winner.  The round loop is kept rolled so the code stays small.
template <typename LogitFn>
__device__ __forceinline__ void top_k_warp_fn(LogitFn logit, int E, int* out_id, float* out_w) {
  const int lane = threadIdx.x & 31;
  const int per = E >> 5;
  float p[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) p[j] = (j < per) ? logit(lane + 32 * j) : -INFINITY;
  float m = p[0];
#pragma unroll
  for (int j = 1; j < 16; ++j) m = fmaxf(m, p[j]);
  m = warp_max(m);
  float z = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    p[j] = (j < per) ? expf(p[j] - m) : 0.f;
    z += p[j];
  }
  z = warp_sum(z);
  const float rz = 1.f / z;
#pragma unroll
  for (int j = 0; j < 16; ++j) p[j] = (j < per) ? p[j] * rz : -1.f;
  // Keys: probability bits + 1 for live candidates (p >= 0, so bit order = value order), 0 for
  // removed or absent ones.  Each round: per-lane tree argmax (lower j on ties), warp max of the
  // keys with redux.sync, then the lowest expert id among the lanes holding that max.
  uint32_t key[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) key[j] = (j < per) ? __float_as_uint(p[j]) + 1u : 0u;
  float s = 0.f, my_p = 0.f;
  int my_id = 0;
#pragma unroll 1
  for (int k = 0; k < K; ++k) {
    uint32_t v8[8];
    int j8[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) {
      const bool r = key[2 * a + 1] > key[2 * a];
      v8[a] = r ? key[2 * a + 1] : key[2 * a];
      j8[a] = r ? 2 * a + 1 : 2 * a;
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const bool r = v8[2 * a + 1] > v8[2 * a];
      v8[a] = r ? v8[2 * a + 1] : v8[2 * a];
      j8[a] = r ? j8[2 * a + 1] : j8[2 * a];
    }
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const bool r = v8[2 * a + 1] > v8[2 * a];
      v8[a] = r ? v8[2 * a + 1] : v8[2 * a];
      j8[a] = r ? j8[2 * a + 1] : j8[2 * a];
    }
    const bool r = v8[1] > v8[0];
    const uint32_t bk = r ? v8[1] : v8[0];
    const uint32_t bid = (uint32_t)(lane + 32 * (r ? j8[1] : j8[0]));
    const uint32_t mx = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t id = __reduce_min_sync(0xffffffffu, bk == mx ? bid : 0xffffffffu);
    if ((int)(id & 31u) == lane) {
      const int jw = (int)(id >> 5);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j == jw) key[j] = 0u;
    }
    const float pv = __uint_as_float(mx - 1u);
    if (lane == k) {
      my_p = pv;
      my_id = (int)id;
    }
    s += pv;
  }
  *out_id = my_id;
  *out_w = my_p / fmaxf(s, kRenormFloor);
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
