// Internal host-side interface between the C ABI (api.cu) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include "../../include/fa.h"

namespace fa {

// Tile shapes (see fa_get_tile_config).
constexpr int kFwdBr = 128, kFwdBc = 128;
constexpr int kBwdBc = 128;
constexpr int bwd_br(int) { return 128; }

// Device status word of the current device (see fa_poll_device_error).
int* device_status_word();

// Encodes a 3-D bf16 tensor map over a contiguous [BH, N, d] array: dims
// (d, N, BH), box (inner, rows, 1), swizzle width = inner * 2 bytes (<= 128).
bool encode_bf16_3d(CUtensorMap* map, const void* base, int d, int N, int BH, int inner, int rows);
// 2-D bf16 tensor map over a row-major [rows_total][inner_total] array.
bool encode_bf16_2d(CUtensorMap* map, const void* base, int inner_total, int rows_total, int box_inner,
                    int box_rows);

struct FwdLaunch {
  const void *Q, *K, *V;
  void* O;
  float* L;
  int BH, N, d, causal;
  float scale;
  cudaStream_t stream;
  int* status;
  unsigned long long* counter;
};
fa_status launch_fwd(const FwdLaunch& a);

struct BwdLaunch {
  const void *Q, *K, *V, *dO;
  const float *L, *D;
  float* dQacc;
  void *dK, *dV;
  int BH, N, d, causal;
  float scale;
  cudaStream_t stream;
  int* status;
  unsigned long long* counter;
};
fa_status launch_bwd(const BwdLaunch& a);
fa_status launch_bwd_d128(const BwdLaunch& a);
// Two-kernel backward (d = 128): dK, dV by key tile, then dQ by query tile,
// written directly to dQ (bf16); needs no workspace.
fa_status launch_bwd_two_kernel_d128(const BwdLaunch& a, void* dQ);

fa_status launch_preprocess(const void* O, const void* dO, float* D, long long rows, int d, cudaStream_t s);
fa_status launch_dq_convert(const float* dQacc, void* dQ, long long n, float scale, cudaStream_t s);
fa_status launch_timeout_probe(int limit_us, cudaStream_t s, int* status);
fa_status launch_selftest(int mode, const void* A, const void* B, float* C, int K, int N, cudaStream_t s,
                          int* status);

}  // namespace fa
