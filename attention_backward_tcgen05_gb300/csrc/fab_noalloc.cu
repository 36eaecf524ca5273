// fab_noalloc.cu -- fab_backward_noalloc: the backward pass for callers that
// cannot allocate device memory.
//
// fab_backward needs a small device workspace (the per-row D_i terms, 4 bytes
// per query row and head, and with a mask its live-tile maps, a byte per
// 128 x 128 tile twice).  Some callers cannot provide one: code whose
// device memory belongs to another allocator that it may not bypass, or code
// that must not call cudaMalloc on its path because cudaMalloc can
// synchronise the device and stall other streams.  This entry point keeps that
// scratch in a fixed array in the library's own device memory instead, so the
// caller passes only inputs and outputs.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (FAB_NOALLOC_MAX_ROWS floats, 4 MiB) until the process
// exits.  Its device address is looked up once per device, with that device
// current, on the first call there, and kept for the rest of the process: a
// cudaDeviceReset (or any other teardown of the device's primary context)
// would leave that address stale, so the entry point must not be called on
// that device again afterwards.  All calls on a device share the array:
// two calls whose work overlaps on the GPU (different streams, no ordering
// between them) race on it.  Nothing in it has to start at zero: each call
// overwrites every D_i entry and map byte it reads before reading it.  When
// the maps do not fit after D_i, the call runs without them (every tile of
// a masked problem is computed; same results).
#include <mutex>

#include "fab.h"
#include "fab_internal.h"

namespace fab {
namespace {

constexpr int64_t kMaxRows = FAB_NOALLOC_MAX_ROWS;
constexpr int kMaxDevices = 64;

__device__ __align__(256) float g_noalloc_scratch[kMaxRows];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch on each device

// Device address of the scratch array on the current device; null on failure.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace fab

extern "C" FAB_EXPORT int fab_backward_noalloc(const void* q, const void* k, const void* v, const void* d,
                                               const void* o, const float* lse, const uint16_t* mask, int causal,
                                               float scale, int dtype, const fab_dims* dims, float* packed_out,
                                               fab_stream stream) {
  if (dims == nullptr || dims->B <= 0 || dims->H <= 0 || dims->N <= 0) return FAB_ERR_INVALID;
  if (o == nullptr || lse == nullptr) return FAB_ERR_INVALID;  // no room for a recomputed O and LSE
  // B*H*N rows of D_i must fit the fixed array (checked without overflow)
  if (dims->B > fab::kMaxRows || dims->H > fab::kMaxRows / dims->B || dims->N > fab::kMaxRows / (dims->B * dims->H))
    return FAB_ERR_WORKSPACE;
  void* scratch = fab::scratch_address();
  if (scratch == nullptr) return FAB_ERR_CUDA;
  return fab_backward(q, k, v, d, o, lse, mask, causal, scale, dtype, dims, scratch,
                      static_cast<size_t>(fab::kMaxRows) * sizeof(float), packed_out, stream);
}
