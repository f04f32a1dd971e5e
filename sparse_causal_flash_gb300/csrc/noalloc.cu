// Allocation-free QK-sparse forward.
//
// Some callers cannot allocate device memory where they run attention:
// serving processes whose allocator hands out one fixed pool at start-up and
// refuses every later request (so a per-call workspace cannot be had), and
// plugins hosted by a framework that forbids allocation inside its callbacks
// (an allocation there can block or fail). For them scfa_qk_fwd_noalloc takes
// no workspace: its scratch (the live-tile metadata of the forward pass)
// lives in an array compiled into this library.
//
// The array has a fixed size, SCFA_NOALLOC_SCRATCH_BYTES; every GPU that
// loads the library holds it until the process exits. All calls on a device
// share it and it keeps the last call's contents: the metadata pass rewrites
// everything a call reads (the status word is cleared at its start), so no
// state leaks from one call to the next, but two calls whose work overlaps on
// the GPU (different streams, no ordering between them) race on the array.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SCFA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device. In host code
// the array's name is only a host-side stand-in, so the address is asked of
// the runtime, once per device, with that device current.
cudaError_t noalloc_scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" scfa_status scfa_qk_fwd_noalloc(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                           const int32_t* q_idx, const int32_t* k_idx, int B, int H, int Tq,
                                           int Tk, int D, float scale, uint16_t* o, float* lse, void* stream) {
  const size_t need = scfa_attn_workspace_size(SCFA_MODE_QK, 0, B, H, Tq, Tk, D);
  if (need == 0) return SCFA_ERR_INVALID;
  if (need > static_cast<size_t>(SCFA_NOALLOC_SCRATCH_BYTES)) return SCFA_ERR_WORKSPACE;
  void* ws = nullptr;
  if (noalloc_scratch_address(&ws) != cudaSuccess) return SCFA_ERR_CUDA;
  return scfa_qk_fwd(q, k, v, q_idx, k_idx, B, H, Tq, Tk, D, scale, o, lse, ws, SCFA_NOALLOC_SCRATCH_BYTES, 0,
                     stream);
}

// The status word of the array (its first int, as in every workspace), after
// the stream's work: SCFA_ERR_TIMEOUT, SCFA_ERR_WORKSPACE or SCFA_ERR_INVALID
// raised on the device by the last call, or SCFA_OK.
extern "C" scfa_status scfa_qk_fwd_noalloc_status(void* stream) {
  void* ws = nullptr;
  if (noalloc_scratch_address(&ws) != cudaSuccess) return SCFA_ERR_CUDA;
  return scfa_get_device_status(ws, stream);
}
