// Backward pass of exact tiled attention on sm_103a: main kernel for head size 32
// (head sizes 64 and 128 run the pipelined kernels of bwd_tile.cu and bwd_persist.cu).
//
// "CS336 Assignment 2 notes" §1.4, Equations 13-19, with the key/value tiles
// in the outer loop (kernel 1 of the notes' two-kernel scheme).  One CTA owns
// a 128-key tile of one (batch, head); K_j and V_j stay in shared memory while
// it walks the query tiles i that the causal mask leaves visible.  Everything
// is formed transposed so that keys sit on the 128 tensor-memory lanes:
//
//   S^T  = K_j Q_i^T                       (Eq 13, scale folded into exp2)
//   P^T  = exp(S^T - L_i)                   (Eq 14; L from the forward)
//   dV_j += P^T dO_i                        (Eq 15; P^T read from tensor memory)
//   dP^T = V_j dO_i^T                       (Eq 16)
//   dS^T = P^T * (dP^T - D_i)               (Eq 17; D from the preprocess; the scale
//                                            of Eq 18-19 is applied to dK and dQ at the end)
//   dK_j += dS^T Q_i                        (Eq 19; dS from shared memory)
//   dQ_i += dS K_j                          (Eq 18) formed per tile in tensor
//           memory and added into an fp32 [B,H,N,d] workspace with one bulk
//           reduce-add (performed in L2) per tile; a later pass rounds it.
//
// Tile shapes: 128 keys x 128 queries; dQ is formed as dQ = dS K (M = 128 queries).
//
// Warp roles: warp 0 TMA producer (K, V once; Q_i, dO_i 2-stage ring), warp 1
// UMMA issuer (one thread), warps 4..7 element-wise work (one thread per key
// lane) and the dQ hand-off, then the dK / dV epilogue.
#include "internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static_assert(D == 32, "head sizes 64 and 128 run bwd_tile.cu / bwd_persist.cu");
  static constexpr int BN = kBwdBc;  // keys per CTA (tensor-memory lanes)
  static constexpr int BM = 128;     // queries per inner step
  static constexpr int SWB = (D * 2 >= 128) ? 128 : D * 2;
  static constexpr int CE = SWB / 2, NCH = D / CE;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int QT_BYTES = BM * D * 2;
  static constexpr int DS_BYTES = BM * BN * 2;
  static constexpr int DQ_BYTES = BM * D * 4;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_Q = OFF_V + KV_BYTES;       // 2 stages
  static constexpr int OFF_DO = OFF_Q + 2 * QT_BYTES;  // 2 stages
  static constexpr int OFF_DS = OFF_DO + 2 * QT_BYTES;
  static constexpr int OFF_DQ = OFF_DS + DS_BYTES;
  static constexpr int OFF_LD = OFF_DQ + DQ_BYTES;     // L*log2e [BM], D [BM]
  static constexpr int OFF_BAR = OFF_LD + 2 * BM * 4;
  static constexpr int B_KV = 0, B_QFULL = 1, B_QEMPTY = 3, B_SFULL = 5, B_DPFULL = 6, B_PREADY = 7,
                       B_DQFULL = 8, B_DQFREE = 10, B_FINAL = 12, B_DVDONE = 13, NBAR = 14;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM = (SMEM_USED + 1024 > 120 * 1024) ? SMEM_USED + 1024 : 120 * 1024;
  // tensor memory columns
  static constexpr int DQC = D;  // columns of one dQ buffer
  static constexpr int TM_DK = 0, TM_DV = D, TM_S = 2 * D, TM_DP = 2 * D + BM, TM_DQ = 2 * D + 2 * BM;
  static constexpr int TM_COLS = 512;
  static_assert(TM_DQ + 2 * DQC <= TM_COLS, "tensor memory budget");
  static_assert(OFF_DS % 1024 == 0, "dS tile must be 1024-byte aligned");
};

enum : int { SITE_BWD_PRODUCER = 0x201, SITE_BWD_MMA = 0x202, SITE_BWD_COMPUTE = 0x203 };

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(256, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
               const float* __restrict__ Lg, const float* __restrict__ Dg, float* __restrict__ dQacc,
               __nv_bfloat16* __restrict__ dK, __nv_bfloat16* __restrict__ dV, int Nq, int Nk, int window, float c_log2, float scale,
               int* status, unsigned long long* tile_counter, int head_group) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const Guard guard{status, abort_flag};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int kt = 0, bh = 0;  // key tile (the longest causal loops first) and head, heads in groups (grouped_tile_head)
  grouped_tile_head(blockIdx.y * gridDim.x + blockIdx.x, gridDim.x, gridDim.y, head_group, &kt, &bh);
  const int off = Nk - Nq;  // position of query row i is i + off
  // visible query tiles i0 .. i0 + n_it - 1 (none: this CTA writes zero dK, dV)
  int i0 = 0, ilast = 0;
  query_tile_range(kt, C::BM, C::BN, Nq, Nk, CAUSAL, window, &i0, &ilast);
  const int n_it = ilast >= i0 ? ilast - i0 + 1 : 0;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_KV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_QFULL + s), 1);
      mbar_init(bar(C::B_QEMPTY + s), 1);
      mbar_init(bar(C::B_DQFULL + s), 1);
      mbar_init(bar(C::B_DQFREE + s), 128);
    }
    mbar_init(bar(C::B_SFULL), 1);
    mbar_init(bar(C::B_DPFULL), 1);
    mbar_init(bar(C::B_PREADY), 128);
    mbar_init(bar(C::B_FINAL), 1);
    mbar_init(bar(C::B_DVDONE), 1);
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

  if (warp == 0 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- producer
    mbar_expect_tx(bar(C::B_KV), 2 * C::KV_BYTES);
    for (int c = 0; c < C::NCH; ++c) {
      tma_load_3d(sb + C::OFF_K + c * C::BN * C::SWB, &tmK, bar(C::B_KV), c * C::CE, kt * C::BN, bh);
      tma_load_3d(sb + C::OFF_V + c * C::BN * C::SWB, &tmV, bar(C::B_KV), c * C::CE, kt * C::BN, bh);
    }
    int last = -1;
    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1;
      if (!mbar_wait(bar(C::B_QEMPTY + s), ((it >> 1) & 1) ^ 1, guard, SITE_BWD_PRODUCER)) break;
      const int q0 = (i0 + it) * C::BM;
      mbar_expect_tx(bar(C::B_QFULL + s), 2 * C::QT_BYTES);
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_3d(sb + C::OFF_Q + s * C::QT_BYTES + c * C::BM * C::SWB, &tmQ, bar(C::B_QFULL + s), c * C::CE, q0,
                    bh);
        tma_load_3d(sb + C::OFF_DO + s * C::QT_BYTES + c * C::BM * C::SWB, &tmdO, bar(C::B_QFULL + s), c * C::CE,
                    q0, bh);
      }
      last = it;
    }
    if (*abort_flag) {
      mbar_drain(bar(C::B_KV), 0);
      for (int it = (last > 0 ? last - 1 : 0); it <= last; ++it)
        mbar_drain(bar(C::B_QFULL + (it & 1)), (it >> 1) & 1);
    }
  } else if (warp == 1 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- UMMA issuer
    constexpr uint32_t idS = idesc_bf16(128, C::BM, false, false);  // K|V (K-major) x Q|dO (K-major)
    constexpr uint32_t idDV = idesc_bf16(128, D, false, true);      // P^T (tensor mem) x dO (N-major)
    constexpr uint32_t idDK = idesc_bf16(128, D, true, true);       // dS^T (M-major) x Q (N-major)
    constexpr uint32_t idDQ = idesc_bf16(128, D, false, true);      // dS (K-major) x K (N-major)
    bool ok = mbar_wait(bar(C::B_KV), 0, guard, SITE_BWD_MMA);
    for (int it = 0; ok && it < n_it; ++it) {
      const int s = it & 1;
      if (!(ok = mbar_wait(bar(C::B_QFULL + s), (it >> 1) & 1, guard, SITE_BWD_MMA))) break;
      // S^T is about to overwrite the columns that held P^T: dV(it-1) must have read them
      if (it > 0 && !(ok = mbar_wait(bar(C::B_DVDONE), (it - 1) & 1, guard, SITE_BWD_MMA))) break;
      tc_fence_after();
      const uint32_t qb = sb + C::OFF_Q + s * C::QT_BYTES;
      const uint32_t db = sb + C::OFF_DO + s * C::QT_BYTES;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_ss(tmem + C::TM_S, sdesc_kmajor<C::SWB, C::BN>(sb + C::OFF_K, ks), sdesc_kmajor<C::SWB, C::BM>(qb, ks),
               idS, ks > 0);
      mma_commit(bar(C::B_SFULL));
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_ss(tmem + C::TM_DP, sdesc_kmajor<C::SWB, C::BN>(sb + C::OFF_V, ks), sdesc_kmajor<C::SWB, C::BM>(db, ks),
               idS, ks > 0);
      mma_commit(bar(C::B_DPFULL));
      if (!(ok = mbar_wait(bar(C::B_PREADY), it & 1, guard, SITE_BWD_MMA))) break;
      if (it >= 2 && !(ok = mbar_wait(bar(C::B_DQFREE + s), ((it >> 1) & 1) ^ 1, guard, SITE_BWD_MMA))) break;
      tc_fence_after();
      // dV += P^T dO_i  (A = bf16 P^T over the S^T columns)
#pragma unroll
      for (int ks = 0; ks < C::BM / 16; ++ks)
        mma_ts(tmem + C::TM_DV, tmem + C::TM_S + ks * 8, sdesc_mnmajor<C::SWB, C::BM>(db, ks), idDV,
               (it > 0 || ks > 0));
      mma_commit(bar(C::B_DVDONE));
      // dK += dS^T Q_i  (dS stored [query][key]: M-major for A)
#pragma unroll
      for (int ks = 0; ks < C::BM / 16; ++ks)
        mma_ss(tmem + C::TM_DK, sdesc_mnmajor<128, C::BM>(sb + C::OFF_DS, ks), sdesc_mnmajor<C::SWB, C::BM>(qb, ks),
               idDK, (it > 0 || ks > 0));
      // dQ_i (this key tile's part)
      const uint32_t dq = tmem + C::TM_DQ + s * C::DQC;
#pragma unroll
      for (int ks = 0; ks < C::BN / 16; ++ks)
        mma_ss(dq, sdesc_kmajor<128, C::BM>(sb + C::OFF_DS, ks), sdesc_mnmajor<C::SWB, C::BN>(sb + C::OFF_K, ks),
               idDQ, ks > 0);
      mma_commit(bar(C::B_DQFULL + s));
      mma_commit(bar(C::B_QEMPTY + s));
    }
    mma_commit(bar(C::B_FINAL));
    if (ok && tile_counter != nullptr) atomicAdd(tile_counter, static_cast<unsigned long long>(n_it));
  } else if (warp >= 4 && !skip) {
    // ---------------------------------------------------------------- element-wise + dQ hand-off
    const int wq = warp & 3;
    const int kr = wq * 32 + lane;    // tensor-memory lane: key row (or d / query row for dQ)
    const int ct = threadIdx.x - 128;  // 0..127 within the group
    const int key = kt * C::BN + kr;
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    float* Ls = reinterpret_cast<float*>(smem + C::OFF_LD);
    float* Ds = Ls + C::BM;
    float* dQs = reinterpret_cast<float*>(smem + C::OFF_DQ);
    uint8_t* dSs = smem + C::OFF_DS;
    const size_t row0 = static_cast<size_t>(bh) * Nq, krow0 = static_cast<size_t>(bh) * Nk;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1;
      const int q0 = (i0 + it) * C::BM;
      // L (pre-multiplied by log2 e) and D of this query tile; rows past Nq get
      // L = +inf so that their P is exactly 0
      for (int t = ct; t < 2 * C::BM; t += 128) {
        const int r = t < C::BM ? t : t - C::BM;
        const int q = q0 + r;
        if (t < C::BM)
          Ls[r] = q < Nq ? Lg[row0 + q] * kLog2e : INFINITY;
        else
          Ds[r] = q < Nq ? Dg[row0 + q] : 0.f;
      }
      named_bar_sync(1, 128);
      if (!(ok = mbar_wait_warp(bar(C::B_SFULL), it & 1, guard, SITE_BWD_COMPUTE))) break;
      if (!(ok = mbar_wait_warp(bar(C::B_DPFULL), it & 1, guard, SITE_BWD_COMPUTE))) break;
      tc_fence_after();
      const bool masked = (CAUSAL && kt * C::BN + C::BN - 1 > q0 + off) ||
                          (window > 0 && kt * C::BN <= q0 + C::BM - 1 + off - window) || (kt * C::BN + C::BN > Nk);
      // queries of this tile (0 .. BM-1) that see this thread's key
      const int qlo = CAUSAL ? key - off - q0 : 0;
      const int qhi = key >= Nk ? -1 : (window > 0 ? key - off + window - 1 - q0 : C::BM - 1);
#pragma unroll
      for (int c = 0; c < C::BM / 32; ++c) {
        uint32_t rs[32], rp[32];
        tmem_ld32(tl + C::TM_S + 32 * c, rs);
        tmem_ld32(tl + C::TM_DP + 32 * c, rp);
        tmem_ld_wait<32>(rs);
        tmem_ld_wait<32>(rp);
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 32; x += 2) {
          float pv[2];
#pragma unroll
          for (int y = 0; y < 2; ++y) {
            const int ql = 32 * c + x + y;  // query within the tile
            float p = ex2(fmaf(__uint_as_float(rs[x + y]), c_log2, -Ls[ql]));
            if (masked && (ql < qlo || ql > qhi)) p = 0.f;
            const float ds = p * (__uint_as_float(rp[x + y]) - Ds[ql]);
            pv[y] = p;
            *reinterpret_cast<__nv_bfloat16*>(dSs + swz128_offset<C::BM>(ql, kr)) = __float2bfloat16_rn(ds);
          }
          pk[x >> 1] = pack_bf16x2(pv[0], pv[1]);
        }
        tmem_st16(tl + C::TM_S + 16 * c, pk);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::B_PREADY));

      // dQ of this tile pair: tensor memory -> shared fp32 [query][d] -> bulk add
      if (!(ok = mbar_wait_warp(bar(C::B_DQFULL + s), (it >> 1) & 1, guard, SITE_BWD_COMPUTE))) break;
      tc_fence_after();
      if (ct == 0) bulk_wait_read0();  // the previous tile's add has read dQs
      named_bar_sync(1, 128);
      const uint32_t dq = tl + C::TM_DQ + s * C::DQC;
      // lane = query row, columns = d
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(dq + 32 * c, r);
        tmem_ld_wait<32>(r);
        float4* rowp = reinterpret_cast<float4*>(dQs + kr * D + 32 * c);
#pragma unroll
        for (int v = 0; v < 8; ++v)
          rowp[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_DQFREE + s));
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (ct == 0) {
        const int rows = min(C::BM, Nq - q0);
        bulk_reduce_add_f32(dQacc + (row0 + q0) * D, smem_u32(dQs), static_cast<uint32_t>(rows * D * 4));
        bulk_commit();
      }
    }
    if (ct == 0) bulk_wait0();
    // dK, dV epilogue
    if (ok) ok = mbar_wait_warp(bar(C::B_FINAL), 0, guard, SITE_BWD_COMPUTE);
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const uint32_t col = t == 0 ? C::TM_DK : C::TM_DV;
        const float f = t == 0 ? scale : 1.f;  // Eq 19's scale, applied once to dK
        uint32_t r[32];
        tmem_ld32(tl + col, r);
        tmem_ld_wait<32>(r);
        // the row as packed bf16 (zero when no query sees these keys: the accumulators
        // were never written), then the warp's 32 rows with whole-row writes
        uint32_t pk[D / 2];
#pragma unroll
        for (int i = 0; i < D / 2; ++i)
          pk[i] = n_it == 0 ? 0u : pack_bf16x2(__uint_as_float(r[2 * i]) * f, __uint_as_float(r[2 * i + 1]) * f);
        const int w0 = kt * C::BN + wq * 32;  // the warp's first key row
        warp_store_rows<D / 8, 0>(pk, reinterpret_cast<uint8_t*>((t == 0 ? dK : dV) + (krow0 + w0) * D), D * 2,
                                  Nk - w0, lane);
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

template <int D, bool CAUSAL>
fa_status launch_bwd_t(const BwdLaunch& a) {
  using C = BwdCfg<D>;
  CUtensorMap mQ, mK, mV, mdO;
  if (!encode_bf16_3d(&mQ, a.Q, D, a.Nq, a.BH, C::CE, C::BM) ||
      !encode_bf16_3d(&mdO, a.dO, D, a.Nq, a.BH, C::CE, C::BM) ||
      !encode_bf16_3d(&mK, a.K, D, a.Nk, a.BH, C::CE, C::BN) || !encode_bf16_3d(&mV, a.V, D, a.Nk, a.BH, C::CE, C::BN))
    return FA_ERR_CUDA;
  auto kern = bwd_kernel<D, CAUSAL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return FA_ERR_CUDA;
  const dim3 grid((a.Nk + C::BN - 1) / C::BN, a.BH);
  const float c_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  kern<<<grid, 256, C::SMEM, a.stream>>>(mQ, mK, mV, mdO, a.L, a.D, a.dQacc, static_cast<__nv_bfloat16*>(a.dK),
                                         static_cast<__nv_bfloat16*>(a.dV), a.Nq, a.Nk, a.window, c_log2, a.scale, a.status,
                                         a.counter, head_group(a.BH, a.Nq, a.Nk, D));
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status launch_bwd(const BwdLaunch& a) {
  switch (a.d) {
    case 32: return a.causal ? launch_bwd_t<32, true>(a) : launch_bwd_t<32, false>(a);
    case 64:
    case 128: return launch_bwd_tile(a);  // the tensor-core pipeline of bwd_tile.cu
    default: return FA_ERR_UNSUPPORTED;
  }
}

}  // namespace fa
