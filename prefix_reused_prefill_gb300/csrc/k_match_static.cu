// Fixed device scratch for kvr_slot_match_static.
//
// kvr_slot_match stages the prompt, the slot lengths and the match lengths in
// the scratch area the caller gave kvr_ctx_create.  kvr_slot_match_static
// stages them here instead: one array of fixed size inside the library, held
// by every GPU that loads it until the process exits, so that call needs no
// device memory from its caller at all.  Host code may not pass the array's
// name to a kernel (on the host it is only a stand-in symbol); the device
// address is looked up once per device with that device current.
#include <mutex>

#include "kvr_internal.cuh"

namespace kvr {

namespace {

constexpr int kStaticWords = KVR_STATIC_MATCH_MAX_TOKENS            // prompt copy
                             + KVR_MAX_SLOTS                        // slot lengths
                             + (KVR_MAX_SLOTS + 1) * KVR_MAX_SLOTS; // match lengths

static __device__ __align__(256) int32_t g_match_scratch[kStaticWords];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_addr[kMaxDevices] = {};

}  // namespace

// Device address of the static match scratch on the current device.  The
// first call on a device resolves it (cudaGetSymbolAddress), later calls reuse it.
cudaError_t static_match_scratch(int32_t** prompt, int** slot_len, int32_t** match_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int32_t* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_match_scratch);
      if (e != cudaSuccess) return e;
      g_addr[dev] = static_cast<int32_t*>(p);
    }
    base = g_addr[dev];
  }
  *prompt = base;
  *slot_len = base + KVR_STATIC_MATCH_MAX_TOKENS;
  *match_out = base + KVR_STATIC_MATCH_MAX_TOKENS + KVR_MAX_SLOTS;
  return cudaSuccess;
}

}  // namespace kvr
