// Forward pass, head size 128: two query tiles per CTA.
//
// The same computation as fwd.cu ("CS336 Assignment 2 notes" §1.2, with the
// whole-tile skip of §1.3 and the general mask), arranged so that the two
// query tiles A (rows 256 p .. 256 p + 127) and B (the next 128 rows) take
// turns on the tensor pipe: while the softmax warps of one tile work on its
// scores, the UMMAs of the other tile run.  The two softmax warpgroups share
// nothing (each keeps its own rows' running max and sums), so their work
// overlaps fully, and each K_j, V_j tile brought into shared memory serves both.
//
// Tensor memory (512 columns): S_A | S_B | O_A | O_B, 128 columns each; P_t is
// written as bf16 over the first 64 columns of S_t.  S_t of key tile j+1 is
// formed only after O_t += P_t V_j has read P_t, so O_t is never being written
// while its softmax warps rescale it.
//
// Warps: 0 TMA producer (Q_A, Q_B once; a 2-stage ring of K and V tiles over the
// union of the two tiles' visible key tiles), 1 UMMA issuer of S_A, S_B, 2 UMMA
// issuer of O_A += P_A V, O_B += P_B V (two issuing threads, as in fwd.cu), 3
// idle, 4..7 softmax and epilogue of tile A, 8..11 of tile B (one query row per
// thread, its tensor-memory lane).  Registers move from warpgroup 0 to the two
// softmax warpgroups with setmaxnreg: 56 + 2 x 224 = 3 x 168.
#include "fwd_softmax.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

struct PP {
  static constexpr int D = 128, BM = kFwdBr, BN = kFwdBc;
  static constexpr int NTHREADS = 384;
  static constexpr int TILE = BM * D * 2;  // 32 KiB: one 128 x 128 bf16 tile in two 64-column chunks
  static constexpr int OFF_Q = 0;          // Q_A, Q_B
  static constexpr int OFF_K = 2 * TILE;   // 2 stages
  static constexpr int OFF_V = 4 * TILE;   // 2 stages
  static constexpr int OFF_BAR = 6 * TILE;
  // barriers; [t] = query tile A (0) or B (1)
  static constexpr int B_Q = 0, B_KFULL = 2, B_KEMPTY = 4, B_VFULL = 6, B_VEMPTY = 8, B_SFULL = 10, B_PFULL = 12,
                       B_PFREE = 14, B_OFINAL = 16, B_SDONE = 17, NBAR = 18;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + alignment slack for the 1 KiB-aligned base
  static constexpr int TM_S = 0, TM_O = 256, TM_COLS = 512;  // S_t at 128 t, O_t at 256 + 128 t
};
static_assert(PP::SMEM <= 232448, "shared memory budget");

enum : int { SITE_PP_PRODUCER = 0x121, SITE_PP_MMA = 0x122, SITE_PP_SOFTMAX = 0x123 };

template <int MASK>
__global__ void __launch_bounds__(PP::NTHREADS, 1)
    fwd_pp_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O, float* __restrict__ Lout,
                  int Nq, int Nk, int window, float c_log2, int* status, unsigned long long* tile_counter,
                  int head_group) {
  using C = PP;
  constexpr bool CAUSAL = MASK >= 1, WINDOW = MASK == 2;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const Guard guard{status, abort_flag};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = (Nq + C::BM - 1) / C::BM;     // query tiles
  const int npair = (T + 1) / 2;
  int qp = 0, bh = 0;  // longest causal rows first, heads in groups (grouped_tile_head)
  grouped_tile_head(blockIdx.y * gridDim.x + blockIdx.x, npair, gridDim.y, head_group, &qp, &bh);
  qp = npair - 1 - qp;
  const int off = Nk - Nq;
  const int w = WINDOW ? window : 0;
  // visible key tiles of each query tile; tile B may not exist (odd T)
  int loA = 0, hiA = 0, loB = 1, hiB = 0;  // B empty unless it exists
  key_tile_range(2 * qp, C::BM, C::BN, Nq, Nk, CAUSAL, w, &loA, &hiA);
  const bool hasB = 2 * qp + 1 < T;
  if (hasB) key_tile_range(2 * qp + 1, C::BM, C::BN, Nq, Nk, CAUSAL, w, &loB, &hiB);
  auto lo_of = [&](int t) { return t == 0 ? loA : loB; };
  auto hi_of = [&](int t) { return t == 0 ? hiA : hiB; };
  // the union of the two intervals is itself an interval: B's rows follow A's
  const int jlo = loA, jhi = hasB ? max(hiA, hiB) : hiA;
  const int n_kv = jhi - jlo + 1;
  auto uses = [&](int t, int j) { return j >= lo_of(t) && j <= hi_of(t); };

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::B_Q + t), 1);
      mbar_init(bar(C::B_KFULL + t), 1);
      mbar_init(bar(C::B_KEMPTY + t), 1);
      mbar_init(bar(C::B_VFULL + t), 1);
      mbar_init(bar(C::B_VEMPTY + t), 1);
      mbar_init(bar(C::B_SFULL + t), 1);
      mbar_init(bar(C::B_PFULL + t), 128);
      mbar_init(bar(C::B_PFREE + t), 1);
    }
    mbar_init(bar(C::B_OFINAL), 1);
    mbar_init(bar(C::B_SDONE), 1);
    *abort_flag = (*reinterpret_cast<volatile int*>(status) != 0);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = *abort_flag != 0;

  if (warp < 4) {
    regs_dec<56>();
    if (warp == 0 && lane == 0 && !skip) {
      // ---------------------------------------------------------------- producer
      pdl_wait();  // Q, K, V (and the O, L rows written below) belong to earlier kernels
      for (int t = 0; t < (hasB ? 2 : 1); ++t) {
        mbar_expect_tx(bar(C::B_Q + t), C::TILE);
        for (int c = 0; c < 2; ++c)
          tma_load_3d(sb + C::OFF_Q + t * C::TILE + c * C::BM * 128, &tmQ, bar(C::B_Q + t), c * 64,
                      (2 * qp + t) * C::BM, bh);
      }
      int jk = -1, jv = -1;
      for (int u = 0; u < n_kv; ++u) {
        const int s = u & 1;
        const uint32_t par = ((u >> 1) & 1) ^ 1;
        if (!mbar_wait(bar(C::B_KEMPTY + s), par, guard, SITE_PP_PRODUCER)) break;
        mbar_expect_tx(bar(C::B_KFULL + s), C::TILE);
        for (int c = 0; c < 2; ++c)
          tma_load_3d(sb + C::OFF_K + s * C::TILE + c * C::BN * 128, &tmK, bar(C::B_KFULL + s), c * 64,
                      (jlo + u) * C::BN, bh);
        jk = u;
        if (!mbar_wait(bar(C::B_VEMPTY + s), par, guard, SITE_PP_PRODUCER)) break;
        mbar_expect_tx(bar(C::B_VFULL + s), C::TILE);
        for (int c = 0; c < 2; ++c)
          tma_load_3d(sb + C::OFF_V + s * C::TILE + c * C::BN * 128, &tmV, bar(C::B_VFULL + s), c * 64,
                      (jlo + u) * C::BN, bh);
        jv = u;
      }
      if (*abort_flag) {
        mbar_drain(bar(C::B_Q), 0);
        if (hasB) mbar_drain(bar(C::B_Q + 1), 0);
        for (int u = (jk > 0 ? jk - 1 : 0); u <= jk; ++u) mbar_drain(bar(C::B_KFULL + (u & 1)), (u >> 1) & 1);
        for (int u = (jv > 0 ? jv - 1 : 0); u <= jv; ++u) mbar_drain(bar(C::B_VFULL + (u & 1)), (u >> 1) & 1);
      }
    } else if (warp == 1 && lane == 0 && !skip) {
      // ---------------------------------------------------------------- UMMA issuer: S_A, S_B
      constexpr uint32_t idS = idesc_bf16(128, C::BN, false, false);
      bool ok = mbar_wait(bar(C::B_Q), 0, guard, SITE_PP_MMA) &&
                (!hasB || mbar_wait(bar(C::B_Q + 1), 0, guard, SITE_PP_MMA));
      int cnt[2] = {0, 0};  // key tiles each query tile has had so far
      for (int u = 0; ok && u < n_kv; ++u) {
        const int s = u & 1, j = jlo + u;
        if (!(ok = mbar_wait(bar(C::B_KFULL + s), (u >> 1) & 1, guard, SITE_PP_MMA))) break;
        const uint32_t kb = sb + C::OFF_K + s * C::TILE;
        for (int t = 0; t < 2; ++t) {
          if (!uses(t, j)) continue;
          // S_t is overwritten only after the previous O_t += P_t V has read P_t
          if (cnt[t] > 0 && !(ok = mbar_wait(bar(C::B_PFREE + t), (cnt[t] - 1) & 1, guard, SITE_PP_MMA))) break;
          tc_fence_after();
          const uint32_t qb = sb + C::OFF_Q + t * C::TILE;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ss(tmem + C::TM_S + 128 * t, sdesc_kmajor<128, 128>(qb, ks), sdesc_kmajor<128, 128>(kb, ks), idS,
                   ks > 0);
          mma_commit(bar(C::B_SFULL + t));
          ++cnt[t];
        }
        if (!ok) break;
        mma_commit(bar(C::B_KEMPTY + s));
      }
      mma_commit(bar(C::B_SDONE));
      if (ok && tile_counter != nullptr) atomicAdd(tile_counter, static_cast<unsigned long long>(cnt[0] + cnt[1]));
    } else if (warp == 2 && lane == 0 && !skip) {
      // ---------------------------------------------------------------- UMMA issuer: O_t += P_t V
      constexpr uint32_t idO = idesc_bf16(128, D, false, true);
      bool ok = true;
      int cnt[2] = {0, 0};
      for (int u = 0; ok && u < n_kv; ++u) {
        const int s = u & 1, j = jlo + u;
        if (!(ok = mbar_wait(bar(C::B_VFULL + s), (u >> 1) & 1, guard, SITE_PP_MMA))) break;
        const uint32_t vb = sb + C::OFF_V + s * C::TILE;
        for (int t = 0; t < 2; ++t) {
          if (!uses(t, j)) continue;
          if (!(ok = mbar_wait(bar(C::B_PFULL + t), cnt[t] & 1, guard, SITE_PP_MMA))) break;
          tc_fence_after();
          const uint32_t aP = tmem + C::TM_S + 128 * t;
#pragma unroll
          for (int ks = 0; ks < C::BN / 16; ++ks)
            mma_ts(tmem + C::TM_O + 128 * t, aP + ks * 8, sdesc_mnmajor<128, 128>(vb, ks), idO,
                   (cnt[t] > 0 || ks > 0));
          mma_commit(bar(C::B_PFREE + t));
          ++cnt[t];
        }
        if (!ok) break;
        mma_commit(bar(C::B_VEMPTY + s));
      }
      // every S_t completed before its P_t existed: this marks the end of all UMMAs
      mma_commit(bar(C::B_OFINAL));
    }
  } else {
    regs_inc<224>();
    const int t = (warp - 4) >> 2;  // query tile of this warpgroup
    if (!skip && (t == 0 || hasB)) {
      // ---------------------------------------------------------------- softmax + epilogue of tile t
      const int wq = warp & 3;
      const int row = wq * 32 + lane;
      const int qt = 2 * qp + t;
      const int q = qt * C::BM + row;
      const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
      const uint32_t tS = tl + C::TM_S + 128 * t, tO = tl + C::TM_O + 128 * t;
      const int jlo_t = lo_of(t), n_t = hi_of(t) - jlo_t + 1;
      SoftmaxRow st;
      bool ok = true;
      for (int j = 0; j < n_t; ++j) {
        if (!(ok = mbar_wait_warp(bar(C::B_SFULL + t), j & 1, guard, SITE_PP_SOFTMAX))) break;
        tc_fence_after();
        // O_t is at rest: its last product finished before S_t of this tile was formed
        // (that barrier has completed exactly j phases: the wait returns at once)
        auto wait_o = [&] { return mbar_wait_warp(bar(C::B_PFREE + t), (j - 1) & 1, guard, SITE_PP_SOFTMAX); };
        if (!(ok = softmax_tile<D, CAUSAL, WINDOW>(st, tS, tO, j == 0, (jlo_t + j) * C::BN, qt * C::BM, q, off, Nk,
                                                   window, c_log2, wait_o)))
          break;
        tc_fence_before();
        mbar_arrive(bar(C::B_PFULL + t));
      }
      // the last O_t += P_t V of this tile
      if (ok) ok = mbar_wait_warp(bar(C::B_PFREE + t), (n_t - 1) & 1, guard, SITE_PP_SOFTMAX);
      if (ok) {
        tc_fence_after();
        uint32_t pk[D / 2];
        softmax_epilogue_load<D>(st, tO, pk);
        if (q < Nq) {
          const size_t r0 = static_cast<size_t>(bh) * Nq + q;
          softmax_epilogue_store<D>(st, pk, O + r0 * D, Lout + r0);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (!skip && *abort_flag) {
      if (lane == 0) {
        mbar_drain(bar(C::B_SDONE), 0);
        mbar_drain(bar(C::B_OFINAL), 0);
      }
      __syncwarp();
    }
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

template <int MASK>
fa_status launch_pp_t(const FwdLaunch& a) {
  using C = PP;
  CUtensorMap mQ, mK, mV;
  if (!encode_bf16_3d(&mQ, a.Q, C::D, a.Nq, a.BH, 64, C::BM) || !encode_bf16_3d(&mK, a.K, C::D, a.Nk, a.BH, 64, C::BN) ||
      !encode_bf16_3d(&mV, a.V, C::D, a.Nk, a.BH, 64, C::BN))
    return FA_ERR_CUDA;
  auto kern = fwd_pp_kernel<MASK>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return FA_ERR_CUDA;
  const int T = (a.Nq + C::BM - 1) / C::BM;
  const dim3 grid((T + 1) / 2, a.BH);
  const float c_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  const cudaError_t e = launch_pdl(kern, grid, dim3(C::NTHREADS), C::SMEM, a.stream, mQ, mK, mV,
                                   static_cast<__nv_bfloat16*>(a.O), a.L, a.Nq, a.Nk, a.window, c_log2, a.status,
                                   a.counter, head_group(a.BH, a.Nq, a.Nk, C::D));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status launch_fwd_pp(const FwdLaunch& a) {
  if (a.d != 128) return FA_ERR_UNSUPPORTED;
  return a.window > 0 ? launch_pp_t<2>(a) : a.causal ? launch_pp_t<1>(a) : launch_pp_t<0>(a);
}

}  // namespace fa
