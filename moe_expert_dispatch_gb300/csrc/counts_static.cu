// counts_static.cu - moe_counts_static: per-expert counts and offsets with
// no caller workspace and no device allocation.
//
// Some callers cannot allocate device memory when they call the library: a
// serving runtime that fixes its whole memory footprint at start-up and
// forbids allocation afterwards (cudaMalloc can synchronise the device and
// can fail under memory pressure in the middle of serving), or a plugin
// interface that gives an operator no scratch buffer. For them this entry
// point keeps the scratch of the counting step (the per-chunk histograms and
// per-chunk bases) in a fixed array of device memory that belongs to the
// library, instead of a workspace.
#include "common.cuh"
#include "internal.h"

namespace moe {

int* device_error_word();

namespace {

// int32 entries of each of the two scratch tables ([chunks, E] histograms and
// bases): chunks * E may not exceed this, i.e. n_ids <= 2048 * 65536 / E ids
// (16 M ids at E = 8, 1 M at E = 128, 131072 at E = 1024). 512 KB in total,
// held by every GPU that loads the library until the process exits.
constexpr int64_t kStaticEntries = 65536;

static __device__ __align__(256) int32_t g_static_counts_scratch[2 * kStaticEntries];

constexpr int kMaxDevices = 64;

// Device address of the array on the current device. Host code may not use
// the symbol itself (on the host it names a host-side stand-in), so the
// address is looked up once per device, with that device current.
int32_t* scratch_for_current_device() {
  static int32_t* addr[kMaxDevices] = {};
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return nullptr;
  if (!addr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_counts_scratch) != cudaSuccess || !p) return nullptr;
    addr[d] = static_cast<int32_t*>(p);
  }
  return addr[d];
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_counts_static(const int32_t* ids, int64_t n_ids, int E, int32_t* counts,
                                        int32_t* offsets, void* stream) {
  MOE_ENTRY_RANGE();
  if (n_ids < 0 || E < 1 || E > kMaxExperts || n_ids >= (static_cast<int64_t>(1) << 31))
    return MOE_ERR_INVALID_ARG;
  if ((n_ids > 0 && !ids) || !counts || !offsets) return MOE_ERR_INVALID_ARG;
  const int64_t chunks = route_chunks(n_ids > 0 ? n_ids : 1);
  if (chunks * E > kStaticEntries) return MOE_ERR_WORKSPACE;
  int32_t* scratch = scratch_for_current_device();
  if (!scratch) return MOE_ERR_CUDA;
  RouteScratch s;
  s.hist = scratch;
  s.base = scratch + kStaticEntries;
  s.chunks = chunks;
  return launch_counts(ids, n_ids, E, 1, counts, offsets, nullptr, s, device_error_word(),
                       static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
