// Launch accounting and caller-owned event timing of the library's kernels.
//
// Every launch site brackets its launch with kernel_begin / kernel_end (common.cuh).  kernel_end counts
// the launch in a process-wide counter; when the calling thread has armed timing of that kernel, the
// two calls record the caller's CUDA events on the launch's stream around the launch.
#include <atomic>

#include "common.cuh"

namespace strata {
namespace {

static_assert(KID_DECODE_LAYER == STRATA_KERNEL_DECODE_LAYER && KID_ROUTE_DECODE == STRATA_KERNEL_ROUTE_DECODE &&
                  KID_ROUTER_PREP == STRATA_KERNEL_ROUTER_PREP && KID_ROUTER_TC == STRATA_KERNEL_ROUTER_TC &&
                  KID_TOP_K == STRATA_KERNEL_TOP_K && KID_GROUP_HIST == STRATA_KERNEL_GROUP_HIST &&
                  KID_GROUP_SCAN == STRATA_KERNEL_GROUP_SCAN && KID_GROUP_SCATTER == STRATA_KERNEL_GROUP_SCATTER &&
                  KID_TC_PREPARE == STRATA_KERNEL_TC_PREPARE && KID_TC_GATHER == STRATA_KERNEL_TC_GATHER &&
                  KID_TC_GATEUP == STRATA_KERNEL_TC_GATEUP && KID_TC_DOWN == STRATA_KERNEL_TC_DOWN &&
                  KID_COMBINE == STRATA_KERNEL_COMBINE && KID_PACK == STRATA_KERNEL_PACK &&
                  KID_HOST_COPY == STRATA_KERNEL_HOST_COPY && KID_WAIT_SELFTEST == STRATA_KERNEL_WAIT_SELFTEST &&
                  KID_BLOB_CRC32 == STRATA_KERNEL_BLOB_CRC32 &&
                  KID_COUNT == STRATA_KERNEL_COUNT,
              "kernel ids of the ABI and the library differ");

std::atomic<unsigned long long> g_launches{0};
thread_local unsigned long long t_launches = 0;  // launches made by the calling thread

struct Armed {
  cudaEvent_t const* start = nullptr;
  cudaEvent_t const* stop = nullptr;
  int skip = 0;
  int n = 0;
  int used = 0;
};
thread_local Armed t_armed[KID_COUNT];

}  // namespace

void kernel_begin(int kid, cudaStream_t s) {
  Armed& a = t_armed[kid];
  if (a.skip == 0 && a.used < a.n) cudaEventRecord(a.start[a.used], s);
}

void kernel_end(int kid, cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  ++t_launches;
  Armed& a = t_armed[kid];
  if (a.skip > 0) {
    --a.skip;
  } else if (a.used < a.n) {
    cudaEventRecord(a.stop[a.used], s);
    ++a.used;
  }
}

bool profiling_armed() {
  for (int k = 0; k < KID_COUNT; ++k)
    if (t_armed[k].used < t_armed[k].n) return true;
  return false;
}

void count_launches(unsigned long long n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

unsigned long long launches_this_thread() { return t_launches; }

}  // namespace strata

extern "C" {

uint64_t strata_moe_launch_count(void) { return strata::g_launches.load(std::memory_order_relaxed); }

strata_status strata_moe_profile_arm(int32_t kernel, int32_t skip, void* const* start_events, void* const* stop_events,
                                     int32_t n) {
  if (kernel < 0 || kernel >= strata::KID_COUNT || n < 0 || skip < 0) return STRATA_E_INVAL;
  if (n > 0 && (!start_events || !stop_events)) return STRATA_E_INVAL;
  strata::Armed& a = strata::t_armed[kernel];
  a.start = reinterpret_cast<cudaEvent_t const*>(start_events);
  a.stop = reinterpret_cast<cudaEvent_t const*>(stop_events);
  a.skip = n > 0 ? skip : 0;
  a.n = n;
  a.used = 0;
  return STRATA_OK;
}

int32_t strata_moe_profile_recorded(int32_t kernel) {
  if (kernel < 0 || kernel >= strata::KID_COUNT) return -1;
  return strata::t_armed[kernel].used;
}

}  // extern "C"
