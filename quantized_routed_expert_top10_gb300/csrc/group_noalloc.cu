// strata_moe_group_noalloc: the grouping step for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all -- for example code running inside an engine whose
// device memory is owned by a custom pool or by another runtime, or a process that must not grow its
// footprint after start-up.  strata_moe_group needs a caller workspace for its per-chunk histograms;
// this variant takes that scratch from a fixed array in this library's own device memory instead, so
// the caller only passes its inputs and outputs.
//
// The array is a file-scope __device__ symbol of STRATA_MOE_GROUP_NOALLOC_SCRATCH_BYTES, sized for
// the largest call the ABI allows (T = 8192, 81,920 pairs).  Every GPU that loads the library holds
// it until the process exits.  Host code cannot use the symbol's name as a device address, so the
// first call on each device asks the runtime for the address (cudaGetSymbolAddress, with that device
// current) and caches it; that first call should therefore come before any stream capture.
// Every call shares the array: two calls whose GPU work overlaps race on it.  Nothing in it has to
// start at zero -- each call writes every word it later reads.
#include <mutex>

#include "common.cuh"

namespace strata {
namespace {

constexpr int64_t kNoAllocMaxPairs = (int64_t)TMAX * K;
constexpr int kNoAllocMaxChunks = (int)((kNoAllocMaxPairs + GROUP_CHUNK - 1) / GROUP_CHUNK);
constexpr size_t kOffStatus = 0;
constexpr size_t kOffNActive = 256;
constexpr size_t kOffChunks = 512;
constexpr size_t kScratchUsed = kOffChunks + sizeof(int32_t) * (size_t)kNoAllocMaxChunks * EMAX;
constexpr size_t kScratchBytes = 256 * 1024;
static_assert(kScratchBytes == STRATA_MOE_GROUP_NOALLOC_SCRATCH_BYTES, "header and library disagree");
static_assert(kScratchUsed <= kScratchBytes, "grouping scratch does not fit the static array");

static __device__ __align__(256) uint8_t g_group_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_group_scratch on the current device (looked up once per device).
strata_status scratch_for_current_device(char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return STRATA_E_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return STRATA_E_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_group_scratch) != cudaSuccess || !p) return STRATA_E_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = (char*)g_scratch_ptr[dev];
  return STRATA_OK;
}

}  // namespace
}  // namespace strata

using namespace strata;

extern "C" strata_status strata_moe_group_noalloc(const int32_t* ids, int32_t T, int32_t n_expert,
                                                  int32_t* expert_off, int32_t* pair, int32_t* active,
                                                  int32_t* n_active, void* stream) {
  if (T < 0 || (int64_t)T * K > kNoAllocMaxPairs) return STRATA_E_INVAL;
  if (n_expert < 32 || n_expert > EMAX || (n_expert % 32) != 0) return STRATA_E_INVAL;
  if (!ids || !expert_off || !pair || !active || !n_active) return STRATA_E_INVAL;
  if ((((uintptr_t)ids | (uintptr_t)expert_off | (uintptr_t)pair | (uintptr_t)active | (uintptr_t)n_active) & 3) != 0)
    return STRATA_E_ALIGN;
  if (T == 0) return STRATA_OK;
  char* scratch = nullptr;
  const strata_status st = scratch_for_current_device(&scratch);
  if (st != STRATA_OK) return st;
  WsLayout L{};
  L.status = kOffStatus;
  L.n_active = kOffNActive;
  L.chunk_cnt = kOffChunks;
  L.n_chunks = (T * K + GROUP_CHUNK - 1) / GROUP_CHUNK;
  const cudaError_t e = launch_group(ids, T, n_expert, expert_off, pair, active, n_active, L, scratch,
                                     (cudaStream_t)stream);
  return e == cudaSuccess ? STRATA_OK : STRATA_E_CUDA;
}
