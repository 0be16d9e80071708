// fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.
//
// fa_bwd needs an fp32 dQ accumulator that the caller allocates and passes in.
// Some callers cannot do that at the point where they run the backward: code
// that works inside a memory budget owned by someone else (a host framework or
// serving runtime that has reserved the device memory up front and forbids
// allocations outside its own pool), or code that must not call cudaMalloc /
// cudaFree because those calls can synchronise the whole device.  This entry
// point takes its accumulator from a fixed array that is part of the library
// itself, so the call allocates nothing.
//
// The array is a file-scope static device array of kNoallocScratchBytes; every
// GPU that loads the library holds its own copy until the process exits.  All
// calls on one device share that copy and it keeps whatever the last call left
// in it: each call zeroes it before use (on the caller's stream).  Two calls on
// the same device whose work overlaps on the GPU (for example, issued to two
// streams with nothing ordering one after the other) race on it; the caller
// must serialise them.
#include <mutex>

#include "internal.h"

namespace fa {
namespace {

constexpr size_t kNoallocScratchBytes = 16u << 20;  // 16 MiB
static_assert(kNoallocScratchBytes == FA_NOALLOC_MAX_WORKSPACE_BYTES, "header and library disagree");

static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the array on the current device.  Host code cannot use the
// symbol itself (in host code it names a host-side stand-in), so the address is
// looked up once per device, with that device current, and cached.
fa_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                                    const float* L, const float* D, void* dQ, void* dK, void* dV, int B, int H,
                                    int N, int d, int causal, float scale, fa_stream_t stream) {
  // argument errors first, without touching the device
  if (fa_bwd_workspace_size(B, H, N, d, causal) == static_cast<size_t>(-1)) return FA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const fa_status st = fa::scratch_on_current_device(&scratch);
  if (st != FA_OK) return st;
  // fa_bwd picks the backward form and the accumulator it needs from one reading
  // of the form setting, rejects a problem whose accumulator is larger than the
  // array (FA_ERR_WORKSPACE), zeroes the part it uses on `stream`, then runs the
  // backward kernels with it.
  return fa_bwd(Q, K, V, O, dO, L, D, dQ, dK, dV, B, H, N, d, causal, scale, scratch, fa::kNoallocScratchBytes,
                stream);
}
