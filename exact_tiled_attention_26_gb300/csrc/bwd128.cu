// Backward pass, head size 128: the software-pipelined main kernel.
//
// Same mathematics as bwd.cu ("CS336 Assignment 2 notes" §1.4, Equations 13-19,
// key/value tiles outer): one CTA owns 128 keys of one (batch, head), K_j and V_j
// stay in shared memory, and the CTA walks the visible 64-row query tiles i.
// With keys on the 128 tensor-memory lanes:
//
//   S^T(i)  = K Q_i^T,  dP^T(i) = V dO_i^T                          (UMMA)
//   P^T     = 2^(S^T c - L log2 e),  dS^T = P^T (dP^T - D)           (8 warps)
//   dV += P^T dO_i (P^T from tensor memory),  dK += dS^T Q_i,
//   dQ_i^T  = K^T dS^T  (into the dP^T columns of the same step)     (UMMA)
//   dQ_i   += dQ_i^T-tile, added into the fp32 workspace with one bulk reduce
//             per tile (performed in L2).  The softmax scale of Eq 18-19 is
//             applied to dK here at the end and to dQ by the convert pass.
//
// The UMMA issuer runs one step ahead: S^T(i+1) and dP^T(i+1) go to the other of
// two tensor-memory buffers while the element-wise warps work on step i, so the
// tensor pipe has work while P and dS are formed.  Tensor memory (512 columns):
// dK 128 | dV 128 | S^T x2 (64 each) | dP^T / dQ^T x2 (64 each).
//
// Warps: 0 TMA producer (all lanes also stage L*log2 e and D of each query tile
// in shared memory, two tiles ahead), 1 UMMA issuer (one thread), 2 dQ reducer
// (one thread issues the bulk adds), 4..11 element-wise (warp w: tensor-memory
// lane quarter w % 4, query half (w - 4) / 4; one key row per thread).
#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct B128 {
  static constexpr int D = 128, BN = 128, BM = 64;
  static constexpr int NTHREADS = 384;
  static constexpr int KV_BYTES = BN * D * 2;   // 32 KB
  static constexpr int QT_BYTES = BM * D * 2;   // 16 KB
  static constexpr int DS_BYTES = BN * BM * 2;  // 16 KB: dS^T [128 keys][64 queries], 128-byte rows
  static constexpr int DQ_BYTES = BM * D * 4;   // 32 KB: fp32 dQ tile [64][128]
  static constexpr int LD_BYTES = 2 * BM * 4;   // L*log2 e [64], D [64]
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_Q = OFF_V + KV_BYTES;        // 2 stages
  static constexpr int OFF_DO = OFF_Q + 2 * QT_BYTES;   // 2 stages
  static constexpr int OFF_DS = OFF_DO + 2 * QT_BYTES;  // 2 buffers
  static constexpr int OFF_DQ = OFF_DS + 2 * DS_BYTES;
  static constexpr int OFF_LD = OFF_DQ + DQ_BYTES;      // 2 stages
  static constexpr int OFF_BAR = OFF_LD + 2 * LD_BYTES;
  enum : int {
    B_KV = 0, B_QFULL = 1, B_QEMPTY = 3, B_SFULL = 5, B_DPFULL = 7, B_PREADY = 9, B_DVDONE = 11,
    B_DQFULL = 13, B_DQCONS = 15, B_DQSFULL = 17, B_DQSEMPTY = 18, B_FINAL = 19, NBAR = 20
  };
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static constexpr int TM_DK = 0, TM_DV = 128, TM_S = 256, TM_DP = 384, TM_COLS = 512;
  static constexpr int NCOMP = 256;  // element-wise threads
  static_assert(OFF_DS % 1024 == 0 && OFF_Q % 1024 == 0 && OFF_DO % 1024 == 0, "swizzled tiles need 1 KiB alignment");
  static_assert(SMEM <= 232448, "shared memory budget");
};

enum : int { SITE_PRODUCER = 0x211, SITE_MMA = 0x212, SITE_COMPUTE = 0x213, SITE_REDUCER = 0x214 };

template <bool CAUSAL>
__global__ void __launch_bounds__(B128::NTHREADS, 1)
    bwd_d128_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const float* __restrict__ Lg, const float* __restrict__ Dg, float* __restrict__ dQacc,
                    __nv_bfloat16* __restrict__ dK, __nv_bfloat16* __restrict__ dV, int N, float c_log2, float scale,
                    int* status, unsigned long long* tile_counter) {
  using C = B128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const Guard guard{status, abort_flag};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kt = blockIdx.x;  // key tile: with the causal mask the longest loops come first
  const int bh = blockIdx.y;
  const int Tq = (N + C::BM - 1) / C::BM;
  const int i0 = CAUSAL ? (kt * C::BN) / C::BM : 0;  // first query tile with a visible entry
  const int n_it = Tq - i0;
  const size_t row0 = static_cast<size_t>(bh) * N;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_KV), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::B_QFULL + b), 1 + 32);  // TMA bytes + the producer's 32 lanes (L, D)
      mbar_init(bar(C::B_QEMPTY + b), 1);
      mbar_init(bar(C::B_SFULL + b), 1);
      mbar_init(bar(C::B_DPFULL + b), 1);
      mbar_init(bar(C::B_PREADY + b), C::NCOMP);
      mbar_init(bar(C::B_DVDONE + b), 1);
      mbar_init(bar(C::B_DQFULL + b), 1);
      mbar_init(bar(C::B_DQCONS + b), C::NCOMP);
    }
    mbar_init(bar(C::B_DQSFULL), C::NCOMP);
    mbar_init(bar(C::B_DQSEMPTY), 1);
    mbar_init(bar(C::B_FINAL), 1);
    *abort_flag = (*reinterpret_cast<volatile int*>(status) != 0);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = *abort_flag != 0;

  if (warp == 0 && !skip) {
    // ---------------------------------------------------------------- producer (whole warp)
    if (lane == 0) {
      mbar_expect_tx(bar(C::B_KV), 2 * C::KV_BYTES);
      for (int c = 0; c < 2; ++c) {
        tma_load_3d(sb + C::OFF_K + c * C::BN * 128, &tmK, bar(C::B_KV), c * 64, kt * C::BN, bh);
        tma_load_3d(sb + C::OFF_V + c * C::BN * 128, &tmV, bar(C::B_KV), c * 64, kt * C::BN, bh);
      }
    }
    int last = -1;
    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1;
      if (!mbar_wait_warp(bar(C::B_QEMPTY + s), ((it >> 1) & 1) ^ 1, guard, SITE_PRODUCER)) break;
      const int q0 = (i0 + it) * C::BM;
      if (lane == 0) {
        mbar_expect_tx(bar(C::B_QFULL + s), 2 * C::QT_BYTES);
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(sb + C::OFF_Q + s * C::QT_BYTES + c * C::BM * 128, &tmQ, bar(C::B_QFULL + s), c * 64, q0, bh);
          tma_load_3d(sb + C::OFF_DO + s * C::QT_BYTES + c * C::BM * 128, &tmdO, bar(C::B_QFULL + s), c * 64, q0,
                      bh);
        }
      }
      // L (times log2 e) and D of this query tile; rows past N get L = +inf so that P = 0
      float* Ls = reinterpret_cast<float*>(smem + C::OFF_LD + s * C::LD_BYTES);
#pragma unroll
      for (int r = lane; r < C::BM; r += 32) {
        const int q = q0 + r;
        Ls[r] = q < N ? Lg[row0 + q] * kLog2e : INFINITY;
        Ls[C::BM + r] = q < N ? Dg[row0 + q] : 0.f;
      }
      mbar_arrive(bar(C::B_QFULL + s));
      last = it;
    }
    if (lane == 0 && *abort_flag) {
      mbar_drain(bar(C::B_KV), 0);
      for (int it = (last > 0 ? last - 1 : 0); it <= last; ++it)
        mbar_drain(bar(C::B_QFULL + (it & 1)), (it >> 1) & 1);
    }
  } else if (warp == 1 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- UMMA issuer
    constexpr uint32_t idS = idesc_bf16(128, C::BM, false, false);  // K|V (K-major) x Q|dO (K-major)
    constexpr uint32_t idDV = idesc_bf16(128, C::D, false, true);   // P^T (tensor memory) x dO (N-major)
    constexpr uint32_t idDK = idesc_bf16(128, C::D, false, true);   // dS^T (K-major) x Q (N-major)
    constexpr uint32_t idDQ = idesc_bf16(128, C::BM, true, true);   // K^T (M-major) x dS^T (N-major)
    const uint32_t kb = sb + C::OFF_K, vb = sb + C::OFF_V;
    auto issue_S = [&](int it) {
      const int b = it & 1;
      const uint32_t qb = sb + C::OFF_Q + b * C::QT_BYTES;
#pragma unroll
      for (int ks = 0; ks < C::D / 16; ++ks)
        mma_ss(tmem + C::TM_S + 64 * b, sdesc_kmajor<128, C::BN>(kb, ks), sdesc_kmajor<128, C::BM>(qb, ks), idS,
               ks > 0);
      mma_commit(bar(C::B_SFULL + b));
    };
    auto issue_dP = [&](int it) {
      const int b = it & 1;
      const uint32_t db = sb + C::OFF_DO + b * C::QT_BYTES;
#pragma unroll
      for (int ks = 0; ks < C::D / 16; ++ks)
        mma_ss(tmem + C::TM_DP + 64 * b, sdesc_kmajor<128, C::BN>(vb, ks), sdesc_kmajor<128, C::BM>(db, ks), idS,
               ks > 0);
      mma_commit(bar(C::B_DPFULL + b));
    };
    bool ok = mbar_wait(bar(C::B_KV), 0, guard, SITE_MMA);
    if (ok && n_it > 0) ok = mbar_wait(bar(C::B_QFULL), 0, guard, SITE_MMA);
    if (ok && n_it > 0) {
      tc_fence_after();
      issue_S(0);
      issue_dP(0);
    }
    for (int it = 0; ok && it < n_it; ++it) {
      const int b = it & 1, nb = b ^ 1;
      if (it + 1 < n_it) {
        if (!(ok = mbar_wait(bar(C::B_QFULL + nb), ((it + 1) >> 1) & 1, guard, SITE_MMA))) break;
        // S^T(it+1) overwrites the columns that held P^T(it-1): dV(it-1) must have read them
        if (it >= 1 && !(ok = mbar_wait(bar(C::B_DVDONE + nb), ((it - 1) >> 1) & 1, guard, SITE_MMA))) break;
        tc_fence_after();
        issue_S(it + 1);
        // dP^T(it+1) overwrites dQ^T(it-1): the element-wise warps must have read it
        if (it >= 1 && !(ok = mbar_wait(bar(C::B_DQCONS + nb), ((it - 1) >> 1) & 1, guard, SITE_MMA))) break;
        tc_fence_after();
        issue_dP(it + 1);
      }
      if (!(ok = mbar_wait(bar(C::B_PREADY + b), (it >> 1) & 1, guard, SITE_MMA))) break;
      tc_fence_after();
      const uint32_t qb = sb + C::OFF_Q + b * C::QT_BYTES;
      const uint32_t db = sb + C::OFF_DO + b * C::QT_BYTES;
      const uint32_t dsb = sb + C::OFF_DS + b * C::DS_BYTES;
      const uint32_t aP = tmem + C::TM_S + 64 * b;
      // dV += P^T dO_i: P^T of queries 0..31 sits in columns 0..15, of 32..63 in 32..47
#pragma unroll
      for (int ks = 0; ks < C::BM / 16; ++ks)
        mma_ts(tmem + C::TM_DV, aP + (ks >> 1) * 32 + (ks & 1) * 8, sdesc_mnmajor<128, C::BM>(db, ks), idDV,
               (it > 0 || ks > 0));
      mma_commit(bar(C::B_DVDONE + b));
      // dK += dS^T Q_i
#pragma unroll
      for (int ks = 0; ks < C::BM / 16; ++ks)
        mma_ss(tmem + C::TM_DK, sdesc_kmajor<128, C::BN>(dsb, ks), sdesc_mnmajor<128, C::BM>(qb, ks), idDK,
               (it > 0 || ks > 0));
      // dQ_i^T = K^T dS^T, into the dP^T columns of this step
#pragma unroll
      for (int ks = 0; ks < C::BN / 16; ++ks)
        mma_ss(tmem + C::TM_DP + 64 * b, sdesc_mnmajor<128, C::BN>(kb, ks), sdesc_mnmajor<128, C::BN>(dsb, ks), idDQ,
               ks > 0);
      mma_commit(bar(C::B_DQFULL + b));
      mma_commit(bar(C::B_QEMPTY + b));
    }
    mma_commit(bar(C::B_FINAL));
    if (ok && tile_counter != nullptr) atomicAdd(tile_counter, static_cast<unsigned long long>(n_it));
  } else if (warp == 2 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- dQ reducer
    const uint32_t dqs = sb + C::OFF_DQ;
    for (int j = 0; j < n_it; ++j) {
      if (!mbar_wait(bar(C::B_DQSFULL), j & 1, guard, SITE_REDUCER)) break;
      const int q0 = (i0 + j) * C::BM;
      const int rows = min(C::BM, N - q0);
      bulk_reduce_add_f32(dQacc + (row0 + q0) * C::D, dqs, static_cast<uint32_t>(rows * C::D * 4));
      bulk_commit();
      bulk_wait_read0();
      mbar_arrive(bar(C::B_DQSEMPTY));
    }
    bulk_wait0();
  } else if (warp >= 4 && !skip) {
    // ---------------------------------------------------------------- element-wise warps
    const int qw = warp & 3;        // tensor-memory lane quarter
    const int h = (warp - 4) >> 2;  // query half of each 64-row tile
    const int kr = qw * 32 + lane;  // key row (tensor-memory lane); also the d index of dQ^T
    const int key = kt * C::BN + kr;
    const uint32_t tl = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    float* dQs = reinterpret_cast<float*>(smem + C::OFF_DQ);
    bool ok = true;

    auto read_dq = [&](int j) -> bool {
      const int bj = j & 1;
      if (!mbar_wait_warp(bar(C::B_DQFULL + bj), (j >> 1) & 1, guard, SITE_COMPUTE)) return false;
      tc_fence_after();
      uint32_t r[32];
      tmem_ld32(tl + C::TM_DP + 64 * bj + 32 * h, r);
      tmem_ld_wait<32>(r);
      tc_fence_before();
      mbar_arrive(bar(C::B_DQCONS + bj));
      if (j >= 1 && !mbar_wait_warp(bar(C::B_DQSEMPTY), (j - 1) & 1, guard, SITE_COMPUTE)) return false;
#pragma unroll
      for (int x = 0; x < 32; ++x) dQs[(32 * h + x) * C::D + kr] = __uint_as_float(r[x]);
      fence_proxy_async_smem();
      mbar_arrive(bar(C::B_DQSFULL));
      return true;
    };

    for (int it = 0; it < n_it; ++it) {
      const int b = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!(ok = mbar_wait_warp(bar(C::B_QFULL + b), ph, guard, SITE_COMPUTE))) break;
      if (!(ok = mbar_wait_warp(bar(C::B_SFULL + b), ph, guard, SITE_COMPUTE))) break;
      if (!(ok = mbar_wait_warp(bar(C::B_DPFULL + b), ph, guard, SITE_COMPUTE))) break;
      tc_fence_after();
      uint32_t rs[32], rp[32];
      tmem_ld32(tl + C::TM_S + 64 * b + 32 * h, rs);
      tmem_ld32(tl + C::TM_DP + 64 * b + 32 * h, rp);
      tmem_ld_wait<32>(rs);
      tmem_ld_wait<32>(rp);
      const int qh = (i0 + it) * C::BM + 32 * h;  // first query of this half
      const float4* L4 = reinterpret_cast<const float4*>(smem + C::OFF_LD + b * C::LD_BYTES) + 8 * h;
      const float4* D4 = L4 + C::BM / 4;
      const bool masked = (CAUSAL && kt * C::BN + C::BN - 1 > qh) || (kt * C::BN + C::BN > N);
      uint32_t pk[16], dk[16];
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const float4 l = L4[v], dd = D4[v];
        const float lv[4] = {l.x, l.y, l.z, l.w}, dv[4] = {dd.x, dd.y, dd.z, dd.w};
        float p[4], ds[4];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int x = 4 * v + y;
          p[y] = ex2(fmaf(__uint_as_float(rs[x]), c_log2, -lv[y]));
          if (masked && ((CAUSAL && key > qh + x) || key >= N)) p[y] = 0.f;
          ds[y] = p[y] * (__uint_as_float(rp[x]) - dv[y]);
        }
        pk[2 * v] = pack_bf16x2(p[0], p[1]);
        pk[2 * v + 1] = pack_bf16x2(p[2], p[3]);
        dk[2 * v] = pack_bf16x2(ds[0], ds[1]);
        dk[2 * v + 1] = pack_bf16x2(ds[2], ds[3]);
      }
      // P^T of these 32 queries over this half's own S^T columns
      tmem_st16(tl + C::TM_S + 64 * b + 32 * h, pk);
      // dS^T row kr, queries 32h .. 32h+31: four 16-byte units of a 128-byte swizzled row
      uint8_t* row = smem + C::OFF_DS + b * C::DS_BYTES + kr * 128;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        *reinterpret_cast<uint4*>(row + (((4 * h + u) ^ (kr & 7)) << 4)) =
            make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::B_PREADY + b));
      if (it >= 1 && !(ok = read_dq(it - 1))) break;
    }
    if (ok && n_it > 0) ok = read_dq(n_it - 1);
    // dK (times scale) and dV: this warp's lane quarter, d columns 64h .. 64h+63
    if (ok) ok = mbar_wait_warp(bar(C::B_FINAL), 0, guard, SITE_COMPUTE);
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const float f = t == 0 ? scale : 1.f;
        __nv_bfloat16* dst = (t == 0 ? dK : dV) + (row0 + key) * C::D + 64 * h;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          tmem_ld32(tl + (t == 0 ? C::TM_DK : C::TM_DV) + 64 * h + 32 * c, r);
          tmem_ld_wait<32>(r);
          if (key < N) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * i]) * f, __uint_as_float(r[8 * i + 1]) * f),
                                 pack_bf16x2(__uint_as_float(r[8 * i + 2]) * f, __uint_as_float(r[8 * i + 3]) * f),
                                 pack_bf16x2(__uint_as_float(r[8 * i + 4]) * f, __uint_as_float(r[8 * i + 5]) * f),
                                 pack_bf16x2(__uint_as_float(r[8 * i + 6]) * f, __uint_as_float(r[8 * i + 7]) * f));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (!skip && *abort_flag) {
      if (lane == 0) mbar_drain(bar(C::B_FINAL), 0);
      __syncwarp();
    }
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

template <bool CAUSAL>
fa_status launch_t(const BwdLaunch& a) {
  using C = B128;
  CUtensorMap mQ, mK, mV, mdO;
  if (!encode_bf16_3d(&mQ, a.Q, C::D, a.N, a.BH, 64, C::BM) || !encode_bf16_3d(&mdO, a.dO, C::D, a.N, a.BH, 64, C::BM) ||
      !encode_bf16_3d(&mK, a.K, C::D, a.N, a.BH, 64, C::BN) || !encode_bf16_3d(&mV, a.V, C::D, a.N, a.BH, 64, C::BN))
    return FA_ERR_CUDA;
  auto kern = bwd_d128_kernel<CAUSAL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return FA_ERR_CUDA;
  const dim3 grid((a.N + C::BN - 1) / C::BN, a.BH);
  const float c_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  kern<<<grid, C::NTHREADS, C::SMEM, a.stream>>>(mQ, mK, mV, mdO, a.L, a.D, a.dQacc,
                                                 static_cast<__nv_bfloat16*>(a.dK), static_cast<__nv_bfloat16*>(a.dV),
                                                 a.N, c_log2, a.scale, a.status, a.counter);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status launch_bwd_d128(const BwdLaunch& a) { return a.causal ? launch_t<true>(a) : launch_t<false>(a); }

}  // namespace fa
