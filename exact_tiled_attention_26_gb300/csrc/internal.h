// Internal host-side interface between the C ABI (api.cu) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include <utility>

#include "../../include/fa.h"

namespace fa {

// Tile shapes (see fa_get_tile_config).
constexpr int kFwdBr = 128, kFwdBc = 128;
constexpr int kBwdBc = 128;
constexpr int bwd_br(int) { return 128; }

// Visible tile ranges of the mask (FwdLaunch), shared by host counts and kernels.
// Key tiles [*lo, *hi] seen by query tile qt (Br rows), and query tiles seen by key
// tile kt (Bc keys); an empty range has *hi < *lo.
__host__ __device__ inline void key_tile_range(int qt, int Br, int Bc, int Nq, int Nk, bool causal, int window,
                                               int* lo, int* hi) {
  const int off = Nk - Nq;
  const int Tk = (Nk + Bc - 1) / Bc;
  const int p_first = qt * Br + off;
  const int p_last = (qt * Br + Br < Nq ? qt * Br + Br : Nq) - 1 + off;
  int h = Tk - 1;
  if (causal && p_last / Bc < h) h = p_last / Bc;
  int l = 0;
  if (window > 0) {
    const int first_key = p_first - window + 1;
    l = first_key > 0 ? first_key / Bc : 0;
  }
  *lo = l;
  *hi = h;
}
__host__ __device__ inline void query_tile_range(int kt, int Br, int Bc, int Nq, int Nk, bool causal, int window,
                                                 int* lo, int* hi) {
  const int off = Nk - Nq;
  const int Tq = (Nq + Br - 1) / Br;
  const int k_first = kt * Bc;
  const int k_last = (kt * Bc + Bc < Nk ? kt * Bc + Bc : Nk) - 1;
  int l = 0;
  if (causal) {
    const int first_row = k_first - off;  // first query whose position reaches this tile
    l = first_row > 0 ? first_row / Br : 0;
  }
  int h = Tq - 1;
  if (window > 0) {
    const int last_row = k_last - off + window - 1;  // last query whose window still reaches it
    h = last_row < 0 ? -1 : (last_row / Br < h ? last_row / Br : h);
  }
  *lo = l;
  *hi = h;
}

// Launch a kernel that may start before the previous kernel on the stream has
// ended (programmatic dependent launch): the kernel must call pdl_wait (ptx.cuh)
// before it touches anything that kernel writes, and everything it does before
// that must be safe to overlap with it.  It overlaps only if the kernel before it
// calls pdl_trigger (otherwise it starts when that kernel ends).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Shape and mask checks of the general-mask entry points (fa_fwd_ex's rules);
// *empty is set when there are no query rows or no heads.
fa_status check_mask_shape(int B, int H, int Nq, int Nk, int d, int causal, int window, bool* empty);
// scale finite and > 0.
bool check_scale(float scale);

// Launch order of (tile, head) work.  CTAs are dispatched in grid order; heads are
// interleaved in groups of `head_group` heads (within a group, the longest causal
// tiles of every head first), so that the heavy tiles of the last heads do not
// start late and leave a tail, while the K and V tiles the group's CTAs share stay
// in L2.  The group holds about 32 MiB of Q, K, V, dO: measured on GB300 (fwd / bwd
// TFLOP/s against one head at a time), 2 x 16 x 4096 x 128 causal with groups of 8:
// 1003 / 874 against 891 / 789; 1 x 32 x 8192 x 128 causal with 4: 1231 / 1053
// against 1166 / 1006; at 1 x 32 x 32768 x 128 one head at a time stays best.
inline int head_group(int BH, int Nq, int Nk, int d) {
  const long long per_head = 4LL * (static_cast<long long>(Nq) + Nk) * d;  // bytes of Q, K, V, dO
  long long g = per_head > 0 ? (32LL << 20) / per_head : BH;
  if (g > BH) g = BH;
  return g < 1 ? 1 : static_cast<int>(g);
}
// (tile, head) of the CTA at linear grid position `li` (x fastest) of a T x BH grid
// ordered as above; `tile` counts from the longest causal work.
__host__ __device__ inline void grouped_tile_head(int li, int T, int BH, int hg, int* tile, int* head) {
  const int g = li / (hg * T), r = li - g * hg * T;
  const int gs = (BH - g * hg) < hg ? (BH - g * hg) : hg;
  *tile = r / gs;
  *head = g * hg + r % gs;
}

// Device status word of the current device (see fa_poll_device_error).
int* device_status_word();

// Encodes a 3-D bf16 tensor map over a contiguous [BH, N, d] array: dims
// (d, N, BH), box (inner, rows, 1), swizzle width = inner * 2 bytes (<= 128).
bool encode_bf16_3d(CUtensorMap* map, const void* base, int d, int N, int BH, int inner, int rows);
// 2-D bf16 tensor map over a row-major [rows_total][inner_total] array.
bool encode_bf16_2d(CUtensorMap* map, const void* base, int inner_total, int rows_total, int box_inner,
                    int box_rows);

// Mask of every pass: Q (and O, L, dO, D, dQ) have Nq rows per head, K and V
// (and dK, dV) Nk rows; query row i sits at position i + Nk - Nq.  causal: keys
// j <= position; window > 0 (only with causal): also j > position - window.
struct FwdLaunch {
  const void *Q, *K, *V;
  void* O;
  float* L;
  int BH, Nq, Nk, d, causal, window;
  float scale;
  cudaStream_t stream;
  int* status;
  unsigned long long* counter;
};
fa_status launch_fwd(const FwdLaunch& a);
// d = 128 forward with two query tiles per CTA (fwd_pp.cu).
fa_status launch_fwd_pp(const FwdLaunch& a);
// Forward with one CTA per SM taking work units from a queue (fwd_persist.cu).
fa_status launch_fwd_persist(const FwdLaunch& a);

struct BwdLaunch {
  const void *Q, *K, *V, *dO;
  const float *L, *D;
  float* dQacc;
  void *dK, *dV;
  int BH, Nq, Nk, d, causal, window;
  float scale;
  cudaStream_t stream;
  int* status;
  unsigned long long* counter;
};
// One-kernel backward, one CTA per key tile: d = 32 (bwd.cu), d = 64 and 128 (bwd_tile.cu).
fa_status launch_bwd(const BwdLaunch& a);
fa_status launch_bwd_tile(const BwdLaunch& a);
// One-kernel backward, d = 64 and 128, one CTA per SM taking key tiles from a queue
// (bwd_persist.cu).
fa_status launch_bwd_persist(const BwdLaunch& a);
// Two-kernel backward (d = 64 or 128): dK, dV by key tile, then dQ by query tile,
// written directly to dQ (bf16); needs no workspace.
fa_status launch_bwd_two_kernel(const BwdLaunch& a, void* dQ);

fa_status launch_preprocess(const void* O, const void* dO, float* D, long long rows, int d, cudaStream_t s);
// Zero `bytes` (a multiple of 16) at 16-byte aligned `p`: an ordinary launch, so that a
// kernel launched after it with launch_pdl starts only once everything before it ended.
fa_status launch_zero(void* p, size_t bytes, cudaStream_t s);
fa_status launch_dq_convert(const float* dQacc, void* dQ, long long n, float scale, cudaStream_t s);
fa_status launch_timeout_probe(int limit_us, cudaStream_t s, int* status);
fa_status launch_selftest(int mode, const void* A, const void* B, float* C, int K, int N, cudaStream_t s,
                          int* status);

}  // namespace fa
