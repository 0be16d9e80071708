// Forward pass of exact tiled attention on sm_103a.
//
// "CS336 Assignment 2 notes" §1.2 (FlashAttention-2 forward): per query tile
// keep a running max m, running sum l and an unnormalised accumulator; per key
// tile S = Q K^T / sqrt(d), m_new = max(m, rowmax S), P = exp(S - m_new),
// rescale l and the accumulator by exp(m - m_new), add P V; finally O = acc / l
// and L = m + log l.  §1.3: a key tile whose first key lies after the query
// tile's last row is skipped.
//
// One CTA owns one 128-row query tile of one (batch, head).  Warp roles:
//   warp 0      TMA producer: Q once, then a 2-stage ring of K and V tiles
//   warp 1      UMMA issuer of S_j = Q K_j^T (one thread) into tensor memory
//               (three buffers)
//   warp 2      UMMA issuer of O += P_j V_j (one thread), P read from tensor
//               memory.  Two issuing threads keep the tensor pipe fed while
//               either waits on a barrier: a wait costs the issuing thread about
//               a hundred cycles even when the barrier is already complete, and
//               the pipe's queue of UMMAs is too short to cover that.
//   warps 4..7  softmax: one thread per query row (its tensor-memory lane);
//               online max/sum in base 2 with the scale folded into one FMA and
//               a lazily moved reference max, P written back as bf16 over its
//               own S columns; epilogue (fwd_softmax.cuh)
#include "fwd_softmax.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

template <int D>
struct FwdCfg {
  static constexpr int BM = kFwdBr, BN = kFwdBc;
  static constexpr int SWB = (D * 2 >= 128) ? 128 : D * 2;  // swizzle row bytes
  static constexpr int CE = SWB / 2;                        // bf16 per swizzle row
  static constexpr int NCH = D / CE;                        // chunks along d
  static constexpr int TILE = BM * D * 2;                   // one 128 x d bf16 tile
  static constexpr int STAGES = 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE;
  static constexpr int OFF_V = OFF_K + STAGES * TILE;
  static constexpr int OFF_BAR = OFF_V + STAGES * TILE;
  static constexpr int NSB = 3;  // S/P buffers in tensor memory
  // barriers
  static constexpr int B_Q = 0, B_KFULL = 1, B_KEMPTY = 3, B_VFULL = 5, B_VEMPTY = 7, B_SFULL = 9,
                       B_PFULL = 12, B_PFREE = 15, B_OFINAL = 18, B_SDONE = 19, NBAR = 20;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  // ask for enough that only one CTA fits per SM (each CTA holds all 512 TMEM columns)
  static constexpr int SMEM = (SMEM_USED + 1024 > 120 * 1024) ? SMEM_USED + 1024 : 120 * 1024;
  // tensor memory columns: S/P buffer b at b * 128, the O accumulator after them
  static constexpr int TM_S0 = 0, TM_O = NSB * 128, TM_COLS = 512;
  static_assert(TM_O + D <= TM_COLS, "tensor memory budget");
};

// wait-site codes recorded in the status word
enum : int { SITE_FWD_PRODUCER = 0x101, SITE_FWD_MMA = 0x102, SITE_FWD_SOFTMAX = 0x103 };

// MASK: 0 none, 1 causal, 2 causal with a sliding window (compile-time, so that
// the window's lower bound costs nothing in the other two).
template <int D, int MASK>
__global__ void __launch_bounds__(256, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O, float* __restrict__ Lout,
               int Nq, int Nk, int window, float c_log2, int* status, unsigned long long* tile_counter,
               int head_group) {
  using C = FwdCfg<D>;
  constexpr bool CAUSAL = MASK >= 1, WINDOW = MASK == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const Guard guard{status, abort_flag};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = (Nq + C::BM - 1) / C::BM;
  int qt = 0, bh = 0;  // longest causal rows first, heads in groups (grouped_tile_head)
  grouped_tile_head(blockIdx.y * gridDim.x + blockIdx.x, T, gridDim.y, head_group, &qt, &bh);
  qt = T - 1 - qt;
  const int off = Nk - Nq;  // position of query row i is i + off
  // visible key tiles jlo .. jlo + n_kv - 1 (whole-tile skip on both sides of the band)
  int jlo = 0, jhi = 0;
  key_tile_range(qt, C::BM, C::BN, Nq, Nk, CAUSAL, WINDOW ? window : 0, &jlo, &jhi);
  const int n_kv = jhi - jlo + 1;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_Q), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_KFULL + s), 1);
      mbar_init(bar(C::B_KEMPTY + s), 1);
      mbar_init(bar(C::B_VFULL + s), 1);
      mbar_init(bar(C::B_VEMPTY + s), 1);
    }
    for (int b = 0; b < C::NSB; ++b) {
      mbar_init(bar(C::B_SFULL + b), 1);
      mbar_init(bar(C::B_PFULL + b), 128);
      mbar_init(bar(C::B_PFREE + b), 1);
    }
    mbar_init(bar(C::B_OFINAL), 1);
    mbar_init(bar(C::B_SDONE), 1);
    // an earlier launch gave up: do no work until the host has polled the status
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

  if (warp == 0 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- producer
    pdl_wait();  // Q, K, V (and the O, L rows written below) belong to earlier kernels
    mbar_expect_tx(bar(C::B_Q), C::TILE);
    for (int c = 0; c < C::NCH; ++c)
      tma_load_3d(sb + C::OFF_Q + c * C::BM * C::SWB, &tmQ, bar(C::B_Q), c * C::CE, qt * C::BM, bh);
    int jk = -1, jv = -1;  // last K / V tile whose load was issued
    for (int j = 0; j < n_kv; ++j) {
      const int s = j & 1;
      const uint32_t par = ((j >> 1) & 1) ^ 1;
      if (!mbar_wait(bar(C::B_KEMPTY + s), par, guard, SITE_FWD_PRODUCER)) break;
      mbar_expect_tx(bar(C::B_KFULL + s), C::TILE);
      for (int c = 0; c < C::NCH; ++c)
        tma_load_3d(sb + C::OFF_K + s * C::TILE + c * C::BN * C::SWB, &tmK, bar(C::B_KFULL + s), c * C::CE,
                    (jlo + j) * C::BN, bh);
      jk = j;
      if (!mbar_wait(bar(C::B_VEMPTY + s), par, guard, SITE_FWD_PRODUCER)) break;
      mbar_expect_tx(bar(C::B_VFULL + s), C::TILE);
      for (int c = 0; c < C::NCH; ++c)
        tma_load_3d(sb + C::OFF_V + s * C::TILE + c * C::BN * C::SWB, &tmV, bar(C::B_VFULL + s), c * C::CE,
                    (jlo + j) * C::BN, bh);
      jv = j;
    }
    if (*abort_flag) {
      // gave up: let every load this thread started land before the CTA exits
      mbar_drain(bar(C::B_Q), 0);
      for (int j = (jk > 0 ? jk - 1 : 0); j <= jk; ++j) mbar_drain(bar(C::B_KFULL + (j & 1)), (j >> 1) & 1);
      for (int j = (jv > 0 ? jv - 1 : 0); j <= jv; ++j) mbar_drain(bar(C::B_VFULL + (j & 1)), (j >> 1) & 1);
    }
  } else if (warp == 1 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- UMMA issuer: S
    constexpr uint32_t idS = idesc_bf16(128, C::BN, false, false);  // Q (K-major) x K (K-major)
    bool ok = mbar_wait(bar(C::B_Q), 0, guard, SITE_FWD_MMA);
    for (int j = 0; ok && j < n_kv; ++j) {
      const int s = j & 1, b = j % C::NSB;
      // S buffer b last held P_{j-3}: the product that read it must be done
      if (j >= C::NSB && !(ok = mbar_wait(bar(C::B_PFREE + b), ((j / C::NSB) & 1) ^ 1, guard, SITE_FWD_MMA)))
        break;
      if (!(ok = mbar_wait(bar(C::B_KFULL + s), (j >> 1) & 1, guard, SITE_FWD_MMA))) break;
      tc_fence_after();
      const uint32_t kb = sb + C::OFF_K + s * C::TILE;
      const uint32_t dS = tmem + C::TM_S0 + b * 128;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_ss(dS, sdesc_kmajor<C::SWB, C::BM>(sb + C::OFF_Q, ks), sdesc_kmajor<C::SWB, C::BN>(kb, ks), idS, ks > 0);
      mma_commit(bar(C::B_SFULL + b));
      mma_commit(bar(C::B_KEMPTY + s));
    }
    mma_commit(bar(C::B_SDONE));  // drain point for teardown
    if (ok && tile_counter != nullptr) atomicAdd(tile_counter, static_cast<unsigned long long>(n_kv));
  } else if (warp == 2 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- UMMA issuer: P V
    constexpr uint32_t idO = idesc_bf16(128, D, false, true);  // P (tensor memory) x V (N-major)
    bool ok = true;
    for (int jj = 0; jj < n_kv; ++jj) {
      const int s = jj & 1, b = jj % C::NSB;
      if (!(ok = mbar_wait(bar(C::B_PFULL + b), (jj / C::NSB) & 1, guard, SITE_FWD_MMA))) break;
      if (!(ok = mbar_wait(bar(C::B_VFULL + s), (jj >> 1) & 1, guard, SITE_FWD_MMA))) break;
      tc_fence_after();
      const uint32_t vb = sb + C::OFF_V + s * C::TILE;
      const uint32_t aP = tmem + C::TM_S0 + b * 128;  // bf16 P packed two per column
#pragma unroll
      for (int ks = 0; ks < C::BN / 16; ++ks)
        mma_ts(tmem + C::TM_O, aP + ks * 8, sdesc_mnmajor<C::SWB, C::BN>(vb, ks), idO, (jj > 0 || ks > 0));
      mma_commit(bar(C::B_VEMPTY + s));
      mma_commit(bar(C::B_PFREE + b));
    }
    // every S_j completed before P_j existed, so this also marks the end of all UMMAs
    mma_commit(bar(C::B_OFINAL));
  } else if (warp >= 4 && !skip) {
    // ---------------------------------------------------------------- softmax + epilogue
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int q = qt * C::BM + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    SoftmaxRow st;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int b = j % C::NSB;
      if (!(ok = mbar_wait_warp(bar(C::B_SFULL + b), (j / C::NSB) & 1, guard, SITE_FWD_SOFTMAX))) break;
      tc_fence_after();
      // O holds P_0..P_{j-1} V: before a rescale, wait for the last of those products.
      // Its barrier is the one that frees S buffer (j-1) % 3; PV_{j-3} is already done
      // (S_j waited for it), so that barrier is at most one phase behind.
      auto wait_o = [&] {
        const int pb = (j - 1) % C::NSB;
        return mbar_wait_warp(bar(C::B_PFREE + pb), ((j - 1) / C::NSB) & 1, guard, SITE_FWD_SOFTMAX);
      };
      if (!(ok = softmax_tile<D, CAUSAL, WINDOW>(st, tl + C::TM_S0 + b * 128, tl + C::TM_O, j == 0,
                                                 (jlo + j) * C::BN, qt * C::BM, q, off, Nk, window, c_log2, wait_o)))
        break;
      tc_fence_before();
      mbar_arrive(bar(C::B_PFULL + b));
    }
    if (ok) ok = mbar_wait_warp(bar(C::B_OFINAL), 0, guard, SITE_FWD_SOFTMAX);
    if (ok) {
      tc_fence_after();
      uint32_t pk[D / 2];
      softmax_epilogue_load<D>(st, tl + C::TM_O, pk);
      const int w0 = qt * C::BM + wq * 32;  // the warp's first query row
      softmax_epilogue_store_rows<D>(st, pk, O, Lout, static_cast<size_t>(bh) * Nq + w0, Nq - w0, lane);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (!skip && *abort_flag) {
      // gave up: make sure no UMMA is still writing tensor memory before freeing it
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

template <int D, int MASK>
fa_status launch_fwd_t(const FwdLaunch& a) {
  using C = FwdCfg<D>;
  CUtensorMap mQ, mK, mV;
  if (!encode_bf16_3d(&mQ, a.Q, D, a.Nq, a.BH, C::CE, C::BM) ||
      !encode_bf16_3d(&mK, a.K, D, a.Nk, a.BH, C::CE, C::BN) || !encode_bf16_3d(&mV, a.V, D, a.Nk, a.BH, C::CE, C::BN))
    return FA_ERR_CUDA;
  auto kern = fwd_kernel<D, MASK>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return FA_ERR_CUDA;
  const dim3 grid((a.Nq + C::BM - 1) / C::BM, a.BH);
  const float c_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  const cudaError_t e = launch_pdl(kern, grid, dim3(256), C::SMEM, a.stream, mQ, mK, mV,
                                   static_cast<__nv_bfloat16*>(a.O), a.L, a.Nq, a.Nk, a.window, c_log2, a.status,
                                   a.counter, head_group(a.BH, a.Nq, a.Nk, D));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status launch_fwd(const FwdLaunch& a) {
  switch (a.d) {
#define FA_FWD_MASKS(D) \
  (a.window > 0 ? launch_fwd_t<D, 2>(a) : a.causal ? launch_fwd_t<D, 1>(a) : launch_fwd_t<D, 0>(a))
    case 32: return FA_FWD_MASKS(32);
    case 64: return FA_FWD_MASKS(64);
    case 128: return FA_FWD_MASKS(128);
#undef FA_FWD_MASKS
    default: return FA_ERR_UNSUPPORTED;
  }
}

}  // namespace fa
