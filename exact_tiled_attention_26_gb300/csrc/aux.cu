// Bandwidth-bound kernels around the attention passes, and two diagnostics.
//
//  * preprocess: D_i = sum_k dO_ik O_ik ("CS336 Assignment 2 notes" §1.4,
//    Eq 17, D = rowsum(O * dO)); one pass over O and dO.
//  * dq_convert: scales the fp32 dQ accumulator and rounds it to bf16.
//  * timeout probe: one time-limited wait that can never complete.
//  * UMMA self-test: one 128 x N x K tile product through the operand paths
//    (K-major / M,N-major shared memory, tensor-memory A) of the attention kernels.
#include "internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float dot_bf16x8(uint4 a, uint4 b) {
  const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fx = __bfloat1622float2(x[i]);
    const float2 fy = __bfloat1622float2(y[i]);
    acc = fmaf(fx.x, fy.x, acc);
    acc = fmaf(fx.y, fy.y, acc);
  }
  return acc;
}

// LPR = D/8 lanes share one row (16 bytes each); each warp covers 32/LPR rows
// per step and UNR steps per loop trip so that several loads are in flight.
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const __nv_bfloat16* __restrict__ O,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         float* __restrict__ Dout, long long rows) {
  constexpr int LPR = D / 8, RPW = 32 / LPR, UNR = 4;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, part = lane % LPR;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  pdl_wait();  // O is the forward's output
  for (long long base = warp_id * RPW * UNR; base < rows; base += nwarps * RPW * UNR) {
    uint4 a[UNR], b[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const long long r = base + u * RPW + sub;
      if (r < rows) {
        a[u] = ld_stream_v4(O + r * D + part * 8);
        b[u] = ld_stream_v4(dO + r * D + part * 8);
      } else {
        a[u] = make_uint4(0, 0, 0, 0);
        b[u] = a[u];
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      float acc = dot_bf16x8(a[u], b[u]);
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      const long long r = base + u * RPW + sub;
      if (part == 0 && r < rows) Dout[r] = acc;
    }
  }
}

// dQ = bf16(scale * sum over key tiles of dS K): the softmax scale of Eq 18 is
// applied here, once per element, instead of to every dS element.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ src,
                                                         __nv_bfloat16* __restrict__ dst, long long n8,
                                                         float scale) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  pdl_wait();  // src is complete once the backward kernel has ended
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint4 lo = ld_stream_v4(src + 8 * i);
    const uint4 hi = ld_stream_v4(src + 8 * i + 4);
    uint4 out;
    out.x = pack_bf16x2(__uint_as_float(lo.x) * scale, __uint_as_float(lo.y) * scale);
    out.y = pack_bf16x2(__uint_as_float(lo.z) * scale, __uint_as_float(lo.w) * scale);
    out.z = pack_bf16x2(__uint_as_float(hi.x) * scale, __uint_as_float(hi.y) * scale);
    out.w = pack_bf16x2(__uint_as_float(hi.z) * scale, __uint_as_float(hi.w) * scale);
    *reinterpret_cast<uint4*>(dst + 8 * i) = out;
  }
}

// The fp32 dQ workspace cleared before the backward kernel reduces into it.
__global__ void __launch_bounds__(256) zero_kernel(uint4* __restrict__ p, long long n16) {
  pdl_trigger();  // the backward kernel may start its loads now; it waits before reducing
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

enum : int { SITE_PROBE = 0x301, SITE_SELFTEST = 0x401 };

__global__ void timeout_probe_kernel(uint64_t limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar_storage;
  __shared__ int abort_storage;
  const uint32_t bar = smem_u32(&bar_storage);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);  // nothing will ever arrive
    abort_storage = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const Guard g{status, &abort_storage};
  if (threadIdx.x == 0) mbar_wait(bar, 0, g, SITE_PROBE, limit_ns);
}

// ------------------------------------------------------------------ UMMA self-test
template <int MODE, int K, int N>
__global__ void __launch_bounds__(128, 1)
    umma_selftest_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __nv_bfloat16* __restrict__ Aglob, float* __restrict__ C, int* status) {
  constexpr bool A_MN = (MODE == 3 || MODE == 4);
  constexpr bool B_MN = (MODE == 1 || MODE == 2 || MODE == 4);
  constexpr bool A_TM = (MODE == 2);
  constexpr int A_INNER = A_MN ? 128 : K, A_ROWS = A_MN ? K : 128;
  constexpr int B_INNER = B_MN ? N : K, B_ROWS = B_MN ? K : N;
  constexpr int SWA = A_INNER * 2 >= 128 ? 128 : A_INNER * 2;
  constexpr int SWBB = B_INNER * 2 >= 128 ? 128 : B_INNER * 2;
  constexpr int A_BYTES = 128 * K * 2, B_BYTES = N * K * 2;
  constexpr int TM_C = 0, TM_A = 128, TM_COLS = 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const uint32_t sA = sb, sB = sb + A_BYTES;
  const uint32_t bar_load = sb + A_BYTES + B_BYTES, bar_mma = bar_load + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + A_BYTES + B_BYTES + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + A_BYTES + B_BYTES + 20);
  const Guard g{status, abort_flag};
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);

  if (threadIdx.x == 0) {
    mbar_expect_tx(bar_load, (A_TM ? 0 : A_BYTES) + B_BYTES);
    if (!A_TM)
      for (int c = 0; c < A_INNER / (SWA / 2); ++c) tma_load_2d(sA + c * A_ROWS * SWA, &tmA, bar_load, c * (SWA / 2), 0);
    for (int c = 0; c < B_INNER / (SWBB / 2); ++c) tma_load_2d(sB + c * B_ROWS * SWBB, &tmB, bar_load, c * (SWBB / 2), 0);
  }
  if constexpr (A_TM) {
    // row r of A (K elements) -> tensor-memory lane r, bf16 packed two per column
    const int r = threadIdx.x;
    for (int c = 0; c < K / 32; ++c) {
      uint32_t v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = *reinterpret_cast<const uint32_t*>(Aglob + r * K + 32 * c + 2 * i);
      tmem_st16(tl + TM_A + 16 * c, v);
    }
    tmem_st_wait();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    if (mbar_wait(bar_load, 0, g, SITE_SELFTEST)) {
      tc_fence_after();
      constexpr uint32_t id = idesc_bf16(128, N, A_MN, B_MN);
#pragma unroll
      for (int ks = 0; ks < K / 16; ++ks) {
        const uint64_t bd = B_MN ? sdesc_mnmajor<SWBB, B_ROWS>(sB, ks) : sdesc_kmajor<SWBB, B_ROWS>(sB, ks);
        if constexpr (A_TM) {
          mma_ts(tmem + TM_C, tmem + TM_A + ks * 8, bd, id, ks > 0);
        } else {
          const uint64_t ad = A_MN ? sdesc_mnmajor<SWA, A_ROWS>(sA, ks) : sdesc_kmajor<SWA, A_ROWS>(sA, ks);
          mma_ss(tmem + TM_C, ad, bd, id, ks > 0);
        }
      }
    }
    mma_commit(bar_mma);
  }
  const bool ok = mbar_wait_warp(bar_mma, 0, g, SITE_SELFTEST) && !*abort_flag;
  if (ok) {
    tc_fence_after();
    const int r = threadIdx.x;
    for (int c = 0; c < N / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(tl + TM_C + 32 * c, v);
      tmem_ld_wait<32>(v);
      for (int i = 0; i < 32; ++i) C[r * N + 32 * c + i] = __uint_as_float(v[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

template <int MODE, int K, int N>
fa_status launch_selftest_t(const void* A, const void* B, float* C, cudaStream_t s, int* status) {
  constexpr bool A_MN = (MODE == 3 || MODE == 4);
  constexpr bool B_MN = (MODE == 1 || MODE == 2 || MODE == 4);
  constexpr int A_INNER = A_MN ? 128 : K, A_ROWS = A_MN ? K : 128;
  constexpr int B_INNER = B_MN ? N : K, B_ROWS = B_MN ? K : N;
  constexpr int SWA = A_INNER * 2 >= 128 ? 128 : A_INNER * 2;
  constexpr int SWBB = B_INNER * 2 >= 128 ? 128 : B_INNER * 2;
  CUtensorMap mA, mB;
  if (!encode_bf16_2d(&mA, A, A_INNER, A_ROWS, SWA / 2, A_ROWS) || !encode_bf16_2d(&mB, B, B_INNER, B_ROWS, SWBB / 2, B_ROWS))
    return FA_ERR_CUDA;
  constexpr int smem = 128 * K * 2 + N * K * 2 + 64 + 1024;
  auto kern = umma_selftest_kernel<MODE, K, N>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return FA_ERR_CUDA;
  kern<<<1, 128, smem, s>>>(mA, mB, static_cast<const __nv_bfloat16*>(A), C, status);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int MODE, int K>
fa_status selftest_n(int N, const void* A, const void* B, float* C, cudaStream_t s, int* st) {
  switch (N) {
    case 32: return launch_selftest_t<MODE, K, 32>(A, B, C, s, st);
    case 64: return launch_selftest_t<MODE, K, 64>(A, B, C, s, st);
    case 128: return launch_selftest_t<MODE, K, 128>(A, B, C, s, st);
    default: return FA_ERR_INVALID_ARG;
  }
}

template <int MODE>
fa_status selftest_k(int K, int N, const void* A, const void* B, float* C, cudaStream_t s, int* st) {
  switch (K) {
    case 32: return selftest_n<MODE, 32>(N, A, B, C, s, st);
    case 64: return selftest_n<MODE, 64>(N, A, B, C, s, st);
    case 128: return selftest_n<MODE, 128>(N, A, B, C, s, st);
    default: return FA_ERR_INVALID_ARG;
  }
}

}  // namespace

fa_status launch_preprocess(const void* O, const void* dO, float* D, long long rows, int d, cudaStream_t s) {
  const int rpw = 32 / (d / 8);
  long long warps = (rows + rpw * 4 - 1) / (rpw * 4);
  long long blocks = (warps + 7) / 8;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  const auto* o = static_cast<const __nv_bfloat16*>(O);
  const auto* g = static_cast<const __nv_bfloat16*>(dO);
  const dim3 grid(static_cast<unsigned>(blocks));
  cudaError_t e = cudaSuccess;
  switch (d) {
    case 32: e = launch_pdl(preprocess_kernel<32>, grid, dim3(256), 0, s, o, g, D, rows); break;
    case 64: e = launch_pdl(preprocess_kernel<64>, grid, dim3(256), 0, s, o, g, D, rows); break;
    case 128: e = launch_pdl(preprocess_kernel<128>, grid, dim3(256), 0, s, o, g, D, rows); break;
    default: return FA_ERR_UNSUPPORTED;
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status launch_zero(void* p, size_t bytes, cudaStream_t s) {
  const long long n16 = static_cast<long long>(bytes / 16);
  long long blocks = (n16 + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  zero_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<uint4*>(p), n16);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status launch_dq_convert(const float* dQacc, void* dQ, long long n, float scale, cudaStream_t s) {
  const long long n8 = n / 8;
  long long blocks = (n8 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  const cudaError_t e = launch_pdl(dq_convert_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, dQacc,
                                   static_cast<__nv_bfloat16*>(dQ), n8, scale);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status launch_timeout_probe(int limit_us, cudaStream_t s, int* status) {
  timeout_probe_kernel<<<1, 32, 0, s>>>(static_cast<uint64_t>(limit_us) * 1000ull, status);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status launch_selftest(int mode, const void* A, const void* B, float* C, int K, int N, cudaStream_t s,
                          int* status) {
  switch (mode) {
    case 0: return selftest_k<0>(K, N, A, B, C, s, status);
    case 1: return selftest_k<1>(K, N, A, B, C, s, status);
    case 2: return selftest_k<2>(K, N, A, B, C, s, status);
    case 3: return selftest_k<3>(K, N, A, B, C, s, status);
    case 4: return selftest_k<4>(K, N, A, B, C, s, status);
    default: return FA_ERR_INVALID_ARG;
  }
}

}  // namespace fa
