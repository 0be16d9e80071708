// C ABI of the exact tiled attention library: argument validation, tensor-map
// encoding and launch of the kernels in fwd.cu, bwd.cu and aux.cu.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace fa {

// One status word per device: kernels that give up on a wait record a site
// code here (first writer wins); launches skip their work while it is set.
__device__ int g_status_word;

namespace {

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {nullptr};
std::mutex g_mu;
// Process-wide debug settings.  Every entry point reads each one exactly once per
// call (a snapshot) and derives everything from that value, so a concurrent change
// takes effect on the next call, never halfway through one.
std::atomic<unsigned long long*> g_tile_counter{nullptr};
std::atomic<int> g_bwd_split{0};        // 0: the defaults below
std::atomic<int> g_fwd_form{0};         // 0: the default (fwd_form below)
// Caller-owned events recorded around the main kernel launch(es) of the forward
// ([0]) and the backward ([1]); both null when unset.
struct KernelEvents {
  cudaEvent_t start = nullptr, stop = nullptr;
};
KernelEvents g_kev[2];
std::mutex g_kev_mu;

KernelEvents kernel_events(int which) {
  std::lock_guard<std::mutex> lk(g_kev_mu);
  return g_kev[which];
}
constexpr int kDefaultBwdSplitD128 = 1;  // chosen by measurement on GB300 (then persistent: bwd_form_for)
// d = 64: the persistent one-kernel form once the problem has more visible tile
// pairs than this (about 20 per SM), else the two kernels, whose shorter steps and
// missing workspace passes (clear, dQ convert) win on small problems.  Measured on
// GB300, backward call in us (two kernels / persistent): 4x8x1024 causal, 1152 pairs,
// 43.9 / 47.9; 4x8x1024, 2048 pairs, 58.8 / 60.5; 4x8x2048 causal, 4352 pairs,
// 103.7 / 97.3; 8x16x1024 causal, 4608 pairs, 138.8 / 113.8; 1x32x8192 causal,
// 66560 pairs, 1058 / 957.
constexpr long long kD64PersistentMinPairs = 3072;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn get_encode() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

CUtensorMapSwizzle swizzle_for(int inner_bytes) {
  switch (inner_bytes) {
    case 128: return CU_TENSOR_MAP_SWIZZLE_128B;
    case 64: return CU_TENSOR_MAP_SWIZZLE_64B;
    case 32: return CU_TENSOR_MAP_SWIZZLE_32B;
    default: return CU_TENSOR_MAP_SWIZZLE_NONE;
  }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Shape checks shared by every entry point; *empty is set when there is no work.
fa_status check_shape(int B, int H, int N, int d, bool* empty) {
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long bh = static_cast<long long>(B) * H;
  *empty = (bh == 0 || N == 0);
  if (*empty) return FA_OK;
  if (bh > 65535) return FA_ERR_UNSUPPORTED;
  // element offsets are formed in 64 bits; keep rows within int range for tile indices
  if (static_cast<long long>(N) > (1LL << 30)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

}  // namespace

// Shape and mask checks of the general-mask entry points.  *empty: no query rows
// (or no heads), so no attention is computed.
fa_status check_mask_shape(int B, int H, int Nq, int Nk, int d, int causal, int window, bool* empty) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || window < 0) return FA_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (window > 0 && !causal) return FA_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(B) * H;
  *empty = (bh == 0 || Nq == 0);
  if (bh > 65535) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(Nq) > (1LL << 30) || static_cast<long long>(Nk) > (1LL << 30)) return FA_ERR_UNSUPPORTED;
  if (*empty) return FA_OK;
  if (Nk == 0) return FA_ERR_INVALID_ARG;  // a softmax over no keys
  if (causal && Nq > Nk) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

bool check_scale(float scale) { return std::isfinite(scale) && scale > 0.f; }

int* device_status_word() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

bool encode_bf16_3d(CUtensorMap* map, const void* base, int d, int N, int BH, int inner, int rows) {
  EncodeTiledFn enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(inner), static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  std::memset(map, 0, sizeof(*map));
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(inner * 2), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bf16_2d(CUtensorMap* map, const void* base, int inner_total, int rows_total, int box_inner,
                    int box_rows) {
  EncodeTiledFn enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner_total), static_cast<cuuint64_t>(rows_total)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner_total) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  std::memset(map, 0, sizeof(*map));
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(box_inner * 2), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 100; }

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
    default: return "FA_ERR_UNKNOWN";
  }
}

fa_status fa_get_tile_config(int d, int pass, int* Br, int* Bc) {
  if (Br == nullptr || Bc == nullptr) return FA_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (pass == 0) {
    *Br = kFwdBr;
    *Bc = kFwdBc;
  } else if (pass == 1) {
    *Br = bwd_br(d);
    *Bc = kBwdBc;
  } else {
    return FA_ERR_INVALID_ARG;
  }
  return FA_OK;
}

long long fa_tile_pairs_ex(int Nq, int Nk, int d, int causal, int window, int pass) {
  int Br = 0, Bc = 0;
  if (Nq < 0 || Nk < 0 || window < 0 || (window > 0 && !causal) || fa_get_tile_config(d, pass, &Br, &Bc) != FA_OK)
    return -1;
  if (Nq == 0 || Nk == 0) return 0;
  if (causal && Nq > Nk) return -1;
  const int Tq = (Nq + Br - 1) / Br;
  long long n = 0;
  for (int i = 0; i < Tq; ++i) {
    int lo = 0, hi = -1;
    key_tile_range(i, Br, Bc, Nq, Nk, causal != 0, window, &lo, &hi);
    if (hi >= lo) n += hi - lo + 1;
  }
  return n;
}

long long fa_tile_pairs(int N, int d, int causal, int pass) { return fa_tile_pairs_ex(N, N, d, causal, 0, pass); }

fa_status fa_debug_set_tile_counter(unsigned long long* dev_counter) {
  g_tile_counter.store(dev_counter);
  return FA_OK;
}

// Which forward kernel runs (fa_debug_set_fwd_form overrides).  Measured on GB300,
// forward TFLOP/s: the persistent kernel (form 3) hides most of the fixed cost of a
// CTA and wins unless query tiles see very many key tiles, e.g. at d = 128 the
// 1024-key window on 1 x 32 x 8192 807 against 689 (one tile per CTA) and 732 (two
// tiles per CTA), 8 x 16 x 2048 causal 946 against 804 and 840, 1 x 32 x 8192
// causal 1289 against 1238, 1 x 32 x 16384 causal (up to 128 key tiles) 1340-1392
// against 1304-1368, and at d = 64 every shape measured (2 x 16 x 4096 causal 652
// against 586); with up to 256 key tiles per query tile (1 x 32 x 32768 causal,
// 32768 non-causal, a 2048-query prefill chunk of 32768 keys) the one-tile kernel is
// 1-2% faster.
static int fwd_form_for(int d, int Nq, int Nk, bool causal, int window, int setting) {
  if (setting != 0) return (setting == 2 && d != 128) ? 1 : setting;
  if (d != 128) return 3;
  const int T = (Nq + kFwdBr - 1) / kFwdBr;
  for (int qt = T - 1; qt >= 0; --qt) {  // the widest ranges are at the end (causal) or inside (window)
    int lo = 0, hi = -1;
    key_tile_range(qt, kFwdBr, kFwdBc, Nq, Nk, causal, window, &lo, &hi);
    if (hi - lo + 1 > 128) return 1;
    if (window == 0) break;  // without a window the last query tile sees the most
  }
  return 3;
}

fa_status fa_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int Nq, int Nk,
                    int d, int causal, int window, float scale, fa_stream_t stream) {
  bool empty = false;
  fa_status st = check_mask_shape(B, H, Nq, Nk, d, causal, window, &empty);
  if (st != FA_OK) return st;
  if (!check_scale(scale)) return FA_ERR_INVALID_ARG;
  if (empty) return FA_OK;
  if (!Q || !K || !V || !O || !L) return FA_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(L, 4))
    return FA_ERR_INVALID_ARG;
  int* status = device_status_word();
  if (status == nullptr) return FA_ERR_CUDA;
  FwdLaunch a{Q, K, V, O, L, B * H, Nq, Nk, d, causal ? 1 : 0, window, scale, stream, status, g_tile_counter.load()};
  const int form = fwd_form_for(d, Nq, Nk, causal != 0, window, g_fwd_form.load());
  const KernelEvents ev = kernel_events(0);
  if (ev.start != nullptr && cudaEventRecord(ev.start, stream) != cudaSuccess) return FA_ERR_CUDA;
  st = form == 2 ? launch_fwd_pp(a) : form == 3 ? launch_fwd_persist(a) : launch_fwd(a);
  if (st == FA_OK && ev.stop != nullptr && cudaEventRecord(ev.stop, stream) != cudaSuccess) return FA_ERR_CUDA;
  return st;
}

fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int N, int d,
                 int causal, float scale, fa_stream_t stream) {
  return fa_fwd_ex(Q, K, V, O, L, B, H, N, N, d, causal, 0, scale, stream);
}

fa_status fa_bwd_preprocess(const void* O, const void* dO, float* D, int B, int H, int N, int d,
                            fa_stream_t stream) {
  bool empty = false;
  fa_status st = check_shape(B, H, N, d, &empty);
  if (st != FA_OK) return st;
  if (empty) return FA_OK;
  if (!O || !dO || !D) return FA_ERR_INVALID_ARG;
  if (!aligned(O, 16) || !aligned(dO, 16) || !aligned(D, 4)) return FA_ERR_INVALID_ARG;
  return launch_preprocess(O, dO, D, static_cast<long long>(B) * H * N, d, stream);
}

// Which backward form runs under the setting `setting` (a snapshot of
// fa_debug_set_bwd_split): 1 = one kernel over key tiles with dQ reduced in the
// fp32 workspace, 2 = two kernels (key tiles for dK, dV; query tiles for dQ).
static int bwd_split(int d, int setting) {
  if (d != 128 && d != 64) return 1;
  if (setting != 0) return setting;
  return kDefaultBwdSplitD128;
}

// The backward form that runs: the split (bwd_split), persistent at d = 128.  Measured
// on GB300 (backward TFLOP/s, one CTA per key tile -> persistent, both forms taking
// their per-step code from one header, calls of the two interleaved): 1 x 32 x 32768
// causal (256 query tiles per key tile) 1140 -> 1149, 1 x 32 x 8192 causal 1063 ->
// 1096, 2 x 16 x 4096 causal 898 -> 938.  (Mask and sizes no longer enter the choice;
// the arguments stay for the forward's rule and for callers.)
static int bwd_form_for(int BH, int d, int Nq, int Nk, bool causal, int window, int setting) {
  const int split = bwd_split(d, setting);
  if (setting != 0 || (d != 128 && d != 64)) return split;
  if (d == 128) return 3;
  const long long pairs = static_cast<long long>(BH) * fa_tile_pairs_ex(Nq, Nk, d, causal ? 1 : 0, window, 1);
  return pairs > kD64PersistentMinPairs ? 3 : 2;
}

// The backward form and the workspace it needs, both from one snapshot of the
// setting: a form that reduces dQ in the workspace (1, 3) always comes with the
// workspace size, the two-kernel form (2) with none.  Shape checked by the caller.
struct BwdPlan {
  int form;
  size_t need;
};
static BwdPlan bwd_plan(int B, int H, int Nq, int Nk, int d, bool causal, int window, bool empty, int setting) {
  BwdPlan p{bwd_form_for(B * H, d, Nq, Nk, causal, window, setting), 0};
  if (!empty && p.form != 2) p.need = static_cast<size_t>(B) * H * Nq * d * sizeof(float);
  return p;
}

size_t fa_bwd_workspace_size_ex(int B, int H, int Nq, int Nk, int d, int causal, int window) {
  bool empty = false;
  if (check_mask_shape(B, H, Nq, Nk, d, causal, window, &empty) != FA_OK) return static_cast<size_t>(-1);
  return bwd_plan(B, H, Nq, Nk, d, causal != 0, window, empty, g_bwd_split.load()).need;
}

fa_status fa_debug_bwd_plan(int B, int H, int Nq, int Nk, int d, int causal, int window, int* form,
                            size_t* workspace_bytes) {
  bool empty = false;
  if (!form || !workspace_bytes) return FA_ERR_INVALID_ARG;
  const fa_status st = check_mask_shape(B, H, Nq, Nk, d, causal, window, &empty);
  if (st != FA_OK) return st;
  const BwdPlan p = bwd_plan(B, H, Nq, Nk, d, causal != 0, window, empty, g_bwd_split.load());
  *form = p.form;
  *workspace_bytes = p.need;
  return FA_OK;
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d, int causal) {
  return fa_bwd_workspace_size_ex(B, H, N, N, d, causal, 0);
}

fa_status fa_selected_forms(int B, int H, int Nq, int Nk, int d, int causal, int window, int* fwd_form,
                            int* bwd_form) {
  bool empty = false;
  if (!fwd_form || !bwd_form) return FA_ERR_INVALID_ARG;
  const fa_status st = check_mask_shape(B, H, Nq, Nk, d, causal, window, &empty);
  if (st != FA_OK) return st;
  *fwd_form = fwd_form_for(d, Nq, Nk, causal != 0, window, g_fwd_form.load());
  *bwd_form = bwd_form_for(B * H, d, Nq, Nk, causal != 0, window, g_bwd_split.load());
  return FA_OK;
}

fa_status fa_debug_set_fwd_form(int form) {
  if (form < 0 || form > 3) return FA_ERR_INVALID_ARG;
  g_fwd_form.store(form);
  return FA_OK;
}

fa_status fa_debug_set_bwd_split(int split) {
  if (split < 0 || split > 3) return FA_ERR_INVALID_ARG;
  g_bwd_split.store(split);
  return FA_OK;
}

fa_status fa_debug_set_kernel_events(int which, void* start, void* stop) {
  if (which != 0 && which != 1) return FA_ERR_INVALID_ARG;
  if ((start == nullptr) != (stop == nullptr)) return FA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_kev_mu);
  g_kev[which].start = static_cast<cudaEvent_t>(start);
  g_kev[which].stop = static_cast<cudaEvent_t>(stop);
  return FA_OK;
}

fa_status fa_bwd_ex(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* L,
                    const float* D, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nk, int d, int causal,
                    int window, float scale, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  bool empty = false;
  fa_status st = check_mask_shape(B, H, Nq, Nk, d, causal, window, &empty);
  if (st != FA_OK) return st;
  if (!check_scale(scale)) return FA_ERR_INVALID_ARG;
  const size_t kv_bytes = static_cast<size_t>(B) * H * Nk * d * 2;
  if (empty) {
    // no query sees any key: the gradients of K and V are zero
    if (kv_bytes == 0) return FA_OK;
    if (!dK || !dV) return FA_ERR_INVALID_ARG;
    if (cudaMemsetAsync(dK, 0, kv_bytes, stream) != cudaSuccess || cudaMemsetAsync(dV, 0, kv_bytes, stream) != cudaSuccess)
      return FA_ERR_CUDA;
    return FA_OK;
  }
  (void)O;  // O enters only through D = rowsum(dO * O), formed by fa_bwd_preprocess
  if (!Q || !K || !V || !dO || !L || !D || !dQ || !dK || !dV) return FA_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(dO, 16) || !aligned(dQ, 16) ||
      !aligned(dK, 16) || !aligned(dV, 16) || !aligned(L, 4) || !aligned(D, 4))
    return FA_ERR_INVALID_ARG;
  // one snapshot of the setting gives both the form and the workspace it needs
  const BwdPlan plan = bwd_plan(B, H, Nq, Nk, d, causal != 0, window, false, g_bwd_split.load());
  const size_t need = plan.need;
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 16)))
    return FA_ERR_WORKSPACE;
  int* status = device_status_word();
  if (status == nullptr) return FA_ERR_CUDA;
  BwdLaunch a{Q,  K,  V,  dO, L,      D,     static_cast<float*>(workspace), dK,     dV,
              B * H, Nq, Nk, d, causal ? 1 : 0, window, scale, stream, status, g_tile_counter.load()};
  const KernelEvents ev = kernel_events(1);
  if (plan.form == 2) {
    if (ev.start != nullptr && cudaEventRecord(ev.start, stream) != cudaSuccess) return FA_ERR_CUDA;
    st = launch_bwd_two_kernel(a, dQ);
    if (st == FA_OK && ev.stop != nullptr && cudaEventRecord(ev.stop, stream) != cudaSuccess) return FA_ERR_CUDA;
    return st;
  }
  st = launch_zero(workspace, need, stream);
  if (st != FA_OK) return st;
  if (ev.start != nullptr && cudaEventRecord(ev.start, stream) != cudaSuccess) return FA_ERR_CUDA;
  st = plan.form == 3 ? launch_bwd_persist(a) : launch_bwd(a);
  if (st != FA_OK) return st;
  if (ev.stop != nullptr && cudaEventRecord(ev.stop, stream) != cudaSuccess) return FA_ERR_CUDA;
  return launch_dq_convert(static_cast<const float*>(workspace), dQ, static_cast<long long>(B) * H * Nq * d, scale,
                           stream);
}

fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* L,
                 const float* D, void* dQ, void* dK, void* dV, int B, int H, int N, int d, int causal, float scale,
                 void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return fa_bwd_ex(Q, K, V, O, dO, L, D, dQ, dK, dV, B, H, N, N, d, causal, 0, scale, workspace, workspace_bytes,
                   stream);
}

fa_status fa_poll_device_error(fa_stream_t stream, int* detail) {
  if (detail) *detail = 0;
  int* status = device_status_word();
  if (status == nullptr) return FA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (v == 0) return FA_OK;
  const int zero = 0;
  if (cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
  if (detail) *detail = v;
  return FA_ERR_TIMEOUT;
}

fa_status fa_debug_timeout_probe(int limit_us, fa_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return FA_ERR_INVALID_ARG;
  int* status = device_status_word();
  if (status == nullptr) return FA_ERR_CUDA;
  return launch_timeout_probe(limit_us, stream, status);
}

fa_status fa_selftest_umma(int mode, const void* A, const void* B, float* C, int K, int N, fa_stream_t stream) {
  if (mode < 0 || mode > 4) return FA_ERR_INVALID_ARG;
  if ((K != 32 && K != 64 && K != 128) || (N != 32 && N != 64 && N != 128)) return FA_ERR_INVALID_ARG;
  if (!A || !B || !C || !aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16)) return FA_ERR_INVALID_ARG;
  int* status = device_status_word();
  if (status == nullptr) return FA_ERR_CUDA;
  return launch_selftest(mode, A, B, C, K, N, stream, status);
}

}  // extern "C"
