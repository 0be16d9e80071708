// Forward pass, persistent: one CTA per SM takes (query tile, head) work units
// from a queue until none is left.
//
// The same computation as fwd.cu ("CS336 Assignment 2 notes" §1.2 with the
// whole-tile skip of §1.3 and the general mask) and the same warp roles; what
// changes is that a CTA runs many units back to back and overlaps their
// boundaries.  A CTA of fwd.cu pays a fixed cost of about 4 us (measured on GB300:
// launch, first loads, the first S before any softmax, the epilogue), which is
// 4-5 key tiles of work and, with short causal rows, a large share of its time.
// Here the next unit's Q and first K, V tiles load and its first S is formed while
// the current unit's last tiles and epilogue run, and units are taken from a
// counter in launch order (longest causal rows first, heads in groups, as in
// fwd.cu), so the SMs also finish together.
//
// Per CTA: warp 0 lane 0 takes a unit (atomicAdd on the launch's counter) and
// hands its index to the other roles through a two-slot ring in shared memory,
// then loads that unit's Q (two buffers) and K, V tiles (a 2-stage ring whose
// position runs on across units); warp 1 issues S = Q K_j^T into three 128-column
// tensor-memory buffers (position running on across units); warp 2 issues
// O += P_j V_j; warps 4..7 run the softmax and hand each unit's row state (running
// max and sums) to warps 8..11 through shared memory, then go straight on to the
// next unit; warps 8..11 wait for the unit's last P V product, take O out of
// tensor memory, release it to the next unit's first product and store O and L.
// Registers move with setmaxnreg: 56 (TMA, UMMA issue) + 232 (softmax) + 216
// (epilogue) = 3 x 168 at d = 128; 64 + 232 + 208 below.
#include <mutex>

#include "fwd_softmax.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fa {

// Work counters of the persistent launches: one pair per launch, taken in turn,
// each left zeroed by the launch that used it (queue_release), so launches that
// overlap on different streams never share one (up to kQueueSlots of them in
// flight at once).
constexpr int kQueueSlots = 1024;
__device__ unsigned int g_fwd_queue[2 * kQueueSlots];

namespace {

template <int D>
struct PCfg {
  static constexpr int BM = kFwdBr, BN = kFwdBc;
  static constexpr int SWB = (D * 2 >= 128) ? 128 : D * 2;
  static constexpr int CE = SWB / 2;
  static constexpr int NCH = D / CE;
  static constexpr int TILE = BM * D * 2;
  static constexpr int OFF_Q = 0;             // two Q buffers
  static constexpr int OFF_K = 2 * TILE;      // 2 stages
  static constexpr int OFF_V = OFF_K + 2 * TILE;
  static constexpr int OFF_BAR = OFF_V + 2 * TILE;
  static constexpr int NSB = 3;
  static constexpr int B_UFULL = 0, B_UEMPTY = 2, B_QFULL = 4, B_QEMPTY = 6, B_KFULL = 8, B_KEMPTY = 10,
                       B_VFULL = 12, B_VEMPTY = 14, B_SFULL = 16, B_PFULL = 19, B_PFREE = 22, B_OFULL = 25,
                       B_OFREE = 26, B_SDONE = 27, B_PVDONE = 28,
                       B_EREADY = 29,  // [unit parity] row state of the unit written by the softmax warps
                       B_EFREE = 31,   // [unit parity] read by the epilogue warps
                       NBAR = 33;
  static constexpr int NTHREADS = 384;
  // setmaxnreg shares of the launch's 3 x 168 registers per thread: TMA and UMMA issue,
  // softmax (232), epilogue.  At d <= 64 the issuing code needs a little more than 56
  // and the epilogue holds a narrower O.
  static constexpr int REG_ISSUE = D == 128 ? 56 : 64, REG_EPI = D == 128 ? 216 : 208;
  static_assert(REG_ISSUE + 232 + REG_EPI == 3 * 168, "register split");
  static constexpr int UEMPTY_COUNT = 1 + 1 + 4 + 4;  // S issuer, P V issuer, 4 softmax and 4 epilogue warps
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tensor-memory base, abort flag, unit ring
  static constexpr int OFF_ROWS = OFF_MISC + 16;       // [2][3][128] floats: m, l, l of the bf16 weights
  static constexpr int SMEM_USED = OFF_ROWS + 2 * 3 * BM * 4;
  static constexpr int SMEM = (SMEM_USED + 1024 > 120 * 1024) ? SMEM_USED + 1024 : 120 * 1024;
  static constexpr int TM_S0 = 0, TM_O = NSB * 128, TM_COLS = 512;
  static_assert(TM_O + D <= TM_COLS, "tensor memory budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

enum : int { SITE_PF_PRODUCER = 0x131, SITE_PF_MMA = 0x132, SITE_PF_SOFTMAX = 0x133 };

// Unit u -> query tile and head (grouped launch order, longest causal rows first)
// and its visible key tiles.
struct Unit {
  int qt, bh, jlo, n_kv;
};
FA_DEV Unit decode_unit(int u, int T, int BH, int hg, int Nq, int Nk, bool causal, int window) {
  Unit x;
  int tile = 0;
  grouped_tile_head(u, T, BH, hg, &tile, &x.bh);
  x.qt = T - 1 - tile;
  int hi = 0;
  key_tile_range(x.qt, kFwdBr, kFwdBc, Nq, Nk, causal, window, &x.jlo, &hi);
  x.n_kv = hi - x.jlo + 1;
  return x;
}

template <int D, int MASK>
__global__ void __launch_bounds__(PCfg<D>::NTHREADS, 1)
    fwd_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
                       float* __restrict__ Lout, int BH, int Nq, int Nk, int window, float c_log2, int head_group,
                       unsigned int* queue, int* status, unsigned long long* tile_counter) {
  using C = PCfg<D>;
  constexpr bool CAUSAL = MASK >= 1, WINDOW = MASK == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* unit_ring = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);  // two slots
  const Guard guard{status, abort_flag};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = (Nq + C::BM - 1) / C::BM;
  const int U = T * BH;
  const int off = Nk - Nq;
  const int w = WINDOW ? window : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::B_UFULL + i), 1);
      mbar_init(bar(C::B_UEMPTY + i), C::UEMPTY_COUNT);
      mbar_init(bar(C::B_QFULL + i), 1);
      mbar_init(bar(C::B_QEMPTY + i), 1);
      mbar_init(bar(C::B_KFULL + i), 1);
      mbar_init(bar(C::B_KEMPTY + i), 1);
      mbar_init(bar(C::B_VFULL + i), 1);
      mbar_init(bar(C::B_VEMPTY + i), 1);
    }
    for (int b = 0; b < C::NSB; ++b) {
      mbar_init(bar(C::B_SFULL + b), 1);
      mbar_init(bar(C::B_PFULL + b), 128);
      mbar_init(bar(C::B_PFREE + b), 1);
    }
    mbar_init(bar(C::B_OFULL), 1);
    mbar_init(bar(C::B_OFREE), 128);
    mbar_init(bar(C::B_SDONE), 1);
    mbar_init(bar(C::B_PVDONE), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::B_EREADY + i), 128);
      mbar_init(bar(C::B_EFREE + i), 128);
    }
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

  float* rows = reinterpret_cast<float*>(smem + C::OFF_ROWS);

  if (warp < 4) {
  regs_dec<PCfg<D>::REG_ISSUE>();
  if (warp == 0 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- producer
    pdl_wait();  // Q, K, V (and the O, L rows written below) belong to earlier kernels
    int kv = 0, jk = -1, jv = -1, kq = -1;  // K/V tiles issued; last K, V, Q load issued
    for (int k = 0;; ++k) {
      const int slot = k & 1;
      // the first unit is the CTA's own (no queue round trip before the first loads),
      // the rest come from the queue after the grid's first units
      int u = k == 0 ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x + atomicAdd(queue, 1u));
      if (u >= U) u = -1;
      // slot k % 2 last held unit k-2: every consumer has read it
      if (k >= 2 && !mbar_wait(bar(C::B_UEMPTY + slot), ((k >> 1) & 1) ^ 1, guard, SITE_PF_PRODUCER)) break;
      unit_ring[slot] = u;
      mbar_arrive(bar(C::B_UFULL + slot));
      if (u < 0) break;
      const Unit x = decode_unit(u, T, BH, head_group, Nq, Nk, CAUSAL, w);
      // Q buffer k % 2 last held unit k-2's Q: its last S product is done
      if (k >= 2 && !mbar_wait(bar(C::B_QEMPTY + slot), ((k >> 1) & 1) ^ 1, guard, SITE_PF_PRODUCER)) break;
      mbar_expect_tx(bar(C::B_QFULL + slot), C::TILE);
      for (int c = 0; c < C::NCH; ++c)
        tma_load_3d(sb + C::OFF_Q + slot * C::TILE + c * C::BM * C::SWB, &tmQ, bar(C::B_QFULL + slot), c * C::CE,
                    x.qt * C::BM, x.bh);
      kq = k;
      bool ok = true;
      for (int j = 0; j < x.n_kv; ++j, ++kv) {
        const int s = kv & 1;
        const uint32_t par = ((kv >> 1) & 1) ^ 1;
        if (!(ok = mbar_wait(bar(C::B_KEMPTY + s), par, guard, SITE_PF_PRODUCER))) break;
        mbar_expect_tx(bar(C::B_KFULL + s), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sb + C::OFF_K + s * C::TILE + c * C::BN * C::SWB, &tmK, bar(C::B_KFULL + s), c * C::CE,
                      (x.jlo + j) * C::BN, x.bh);
        jk = kv;
        if (!(ok = mbar_wait(bar(C::B_VEMPTY + s), par, guard, SITE_PF_PRODUCER))) break;
        mbar_expect_tx(bar(C::B_VFULL + s), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sb + C::OFF_V + s * C::TILE + c * C::BN * C::SWB, &tmV, bar(C::B_VFULL + s), c * C::CE,
                      (x.jlo + j) * C::BN, x.bh);
        jv = kv;
      }
      if (!ok) break;
    }
    if (*abort_flag) {
      // gave up: let every load this thread started land before the CTA exits
      for (int k = (kq > 0 ? kq - 1 : 0); k <= kq; ++k) mbar_drain(bar(C::B_QFULL + (k & 1)), (k >> 1) & 1);
      for (int j = (jk > 0 ? jk - 1 : 0); j <= jk; ++j) mbar_drain(bar(C::B_KFULL + (j & 1)), (j >> 1) & 1);
      for (int j = (jv > 0 ? jv - 1 : 0); j <= jv; ++j) mbar_drain(bar(C::B_VFULL + (j & 1)), (j >> 1) & 1);
    }
  } else if (warp == 1 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- UMMA issuer: S
    constexpr uint32_t idS = idesc_bf16(128, C::BN, false, false);
    bool ok = true;
    int kv = 0, gs = 0;  // K tiles and S buffers used so far, across units
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (!(ok = mbar_wait(bar(C::B_UFULL + slot), (k >> 1) & 1, guard, SITE_PF_MMA))) break;
      const int u = unit_ring[slot];
      mbar_arrive(bar(C::B_UEMPTY + slot));
      if (u < 0) break;
      const Unit x = decode_unit(u, T, BH, head_group, Nq, Nk, CAUSAL, w);
      if (!(ok = mbar_wait(bar(C::B_QFULL + slot), (k >> 1) & 1, guard, SITE_PF_MMA))) break;
      const uint32_t qb = sb + C::OFF_Q + slot * C::TILE;
      for (int j = 0; j < x.n_kv; ++j, ++kv, ++gs) {
        const int s = kv & 1, b = gs % C::NSB;
        // S buffer b last held P of S-tile gs-3: the product that read it is done
        if (gs >= C::NSB &&
            !(ok = mbar_wait(bar(C::B_PFREE + b), ((gs / C::NSB) & 1) ^ 1, guard, SITE_PF_MMA)))
          break;
        if (!(ok = mbar_wait(bar(C::B_KFULL + s), (kv >> 1) & 1, guard, SITE_PF_MMA))) break;
        tc_fence_after();
        const uint32_t kb = sb + C::OFF_K + s * C::TILE;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(tmem + C::TM_S0 + b * 128, sdesc_kmajor<C::SWB, C::BM>(qb, ks), sdesc_kmajor<C::SWB, C::BN>(kb, ks),
                 idS, ks > 0);
        mma_commit(bar(C::B_SFULL + b));
        mma_commit(bar(C::B_KEMPTY + s));
      }
      if (!ok) break;
      mma_commit(bar(C::B_QEMPTY + slot));  // this unit's Q has no later reader
    }
    mma_commit(bar(C::B_SDONE));  // drain point for teardown
    if (ok && tile_counter != nullptr) atomicAdd(tile_counter, static_cast<unsigned long long>(gs));
  } else if (warp == 2 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- UMMA issuer: P V
    constexpr uint32_t idO = idesc_bf16(128, D, false, true);
    bool ok = true;
    int kv = 0, gp = 0;
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (!(ok = mbar_wait(bar(C::B_UFULL + slot), (k >> 1) & 1, guard, SITE_PF_MMA))) break;
      const int u = unit_ring[slot];
      mbar_arrive(bar(C::B_UEMPTY + slot));
      if (u < 0) break;
      const Unit x = decode_unit(u, T, BH, head_group, Nq, Nk, CAUSAL, w);
      for (int j = 0; j < x.n_kv; ++j, ++kv, ++gp) {
        const int s = kv & 1, b = gp % C::NSB;
        if (!(ok = mbar_wait(bar(C::B_PFULL + b), (gp / C::NSB) & 1, guard, SITE_PF_MMA))) break;
        if (!(ok = mbar_wait(bar(C::B_VFULL + s), (kv >> 1) & 1, guard, SITE_PF_MMA))) break;
        // the first product of a unit overwrites O: the previous unit's epilogue has read it
        if (j == 0 && k > 0 && !(ok = mbar_wait(bar(C::B_OFREE), (k - 1) & 1, guard, SITE_PF_MMA))) break;
        tc_fence_after();
        const uint32_t vb = sb + C::OFF_V + s * C::TILE;
        const uint32_t aP = tmem + C::TM_S0 + b * 128;
#pragma unroll
        for (int ks = 0; ks < C::BN / 16; ++ks)
          mma_ts(tmem + C::TM_O, aP + ks * 8, sdesc_mnmajor<C::SWB, C::BN>(vb, ks), idO, (j > 0 || ks > 0));
        mma_commit(bar(C::B_VEMPTY + s));
        mma_commit(bar(C::B_PFREE + b));
      }
      if (!ok) break;
      mma_commit(bar(C::B_OFULL));  // O of this unit is complete
    }
    // every S completed before its P existed, so this marks the end of all UMMAs
    mma_commit(bar(C::B_PVDONE));
  }
  } else if (warp < 8) {
  regs_inc<232>();
  if (!skip) {
    // ---------------------------------------------------------------- softmax
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    bool ok = true;
    int gs = 0;
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (!(ok = mbar_wait_warp(bar(C::B_UFULL + slot), (k >> 1) & 1, guard, SITE_PF_SOFTMAX))) break;
      const int u = unit_ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_UEMPTY + slot));
      if (u < 0) break;
      const Unit x = decode_unit(u, T, BH, head_group, Nq, Nk, CAUSAL, w);
      const int q = x.qt * C::BM + row;
      SoftmaxRow st;
      for (int j = 0; j < x.n_kv; ++j, ++gs) {
        const int b = gs % C::NSB;
        if (!(ok = mbar_wait_warp(bar(C::B_SFULL + b), (gs / C::NSB) & 1, guard, SITE_PF_SOFTMAX))) break;
        tc_fence_after();
        // before a rescale: the last product into O (S-tile gs-1, same unit) is done;
        // that barrier is at most one phase behind
        auto wait_o = [&] {
          const int pb = (gs - 1) % C::NSB;
          return mbar_wait_warp(bar(C::B_PFREE + pb), ((gs - 1) / C::NSB) & 1, guard, SITE_PF_SOFTMAX);
        };
        if (!(ok = softmax_tile<D, CAUSAL, WINDOW>(st, tl + C::TM_S0 + b * 128, tl + C::TM_O, j == 0,
                                                   (x.jlo + j) * C::BN, x.qt * C::BM, q, off, Nk, window, c_log2,
                                                   wait_o)))
          break;
        tc_fence_before();
        mbar_arrive(bar(C::B_PFULL + b));
      }
      if (!ok) break;
      // the row state of this unit for the epilogue warps (slot k % 2 last held unit
      // k-2's, which they have read)
      if (k >= 2 && !(ok = mbar_wait_warp(bar(C::B_EFREE + slot), ((k >> 1) & 1) ^ 1, guard, SITE_PF_SOFTMAX)))
        break;
      float* rs = rows + slot * 3 * C::BM;
      rs[row] = st.m_run;
      rs[C::BM + row] = st.l_run;
      rs[2 * C::BM + row] = st.lr_run;
      mbar_arrive(bar(C::B_EREADY + slot));
    }
  }
  } else {
  regs_inc<PCfg<D>::REG_EPI>();  // from the launch's 168: an increase
  if (!skip) {
    // ---------------------------------------------------------------- epilogue
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (!(ok = mbar_wait_warp(bar(C::B_UFULL + slot), (k >> 1) & 1, guard, SITE_PF_SOFTMAX))) break;
      const int u = unit_ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_UEMPTY + slot));
      if (u < 0) break;
      const Unit x = decode_unit(u, T, BH, head_group, Nq, Nk, CAUSAL, w);
      const int q = x.qt * C::BM + row;
      if (!(ok = mbar_wait_warp(bar(C::B_EREADY + slot), (k >> 1) & 1, guard, SITE_PF_SOFTMAX))) break;
      const float* rs = rows + slot * 3 * C::BM;
      SoftmaxRow st;
      st.m_run = rs[row];
      st.l_run = rs[C::BM + row];
      st.lr_run = rs[2 * C::BM + row];
      mbar_arrive(bar(C::B_EFREE + slot));
      if (!(ok = mbar_wait_warp(bar(C::B_OFULL), k & 1, guard, SITE_PF_SOFTMAX))) break;
      tc_fence_after();
      uint32_t pk[D / 2];
      softmax_epilogue_load<D>(st, tl + C::TM_O, pk);
      tc_fence_before();
      mbar_arrive(bar(C::B_OFREE));  // the next unit's first P V may overwrite O
      if constexpr (!CAUSAL) {
        // whole-row writes: +2-3% where every unit ends at about the same time and the
        // stores come together, 2-3% slower on causal shapes (the longer epilogue)
        const int w0 = x.qt * C::BM + wq * 32;  // the warp's first query row
        softmax_epilogue_store_rows<D>(st, pk, O, Lout, static_cast<size_t>(x.bh) * Nq + w0, Nq - w0, lane);
      } else if (q < Nq) {
        const size_t r0 = static_cast<size_t>(x.bh) * Nq + q;
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
        mbar_drain(bar(C::B_PVDONE), 0);
      }
      __syncwarp();
    }
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
  if (threadIdx.x == 0) queue_release(queue);
}

std::mutex g_q_mu;
int g_q_next = 0;
unsigned int* g_q_base[64] = {nullptr};
int g_nsm[64] = {0};

template <int D, int MASK>
fa_status launch_persist_t(const FwdLaunch& a) {
  using C = PCfg<D>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_CUDA;
  unsigned int* counter = nullptr;
  int nsm = 0;
  {
    std::lock_guard<std::mutex> lk(g_q_mu);
    if (g_q_base[dev] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_fwd_queue) != cudaSuccess) return FA_ERR_CUDA;
      g_q_base[dev] = static_cast<unsigned int*>(p);
      if (cudaDeviceGetAttribute(&g_nsm[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FA_ERR_CUDA;
    }
    counter = g_q_base[dev] + 2 * g_q_next;
    g_q_next = (g_q_next + 1) % kQueueSlots;
    nsm = g_nsm[dev];
  }
  CUtensorMap mQ, mK, mV;
  if (!encode_bf16_3d(&mQ, a.Q, D, a.Nq, a.BH, C::CE, C::BM) ||
      !encode_bf16_3d(&mK, a.K, D, a.Nk, a.BH, C::CE, C::BN) || !encode_bf16_3d(&mV, a.V, D, a.Nk, a.BH, C::CE, C::BN))
    return FA_ERR_CUDA;
  auto kern = fwd_persist_kernel<D, MASK>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return FA_ERR_CUDA;
  const long long units = static_cast<long long>((a.Nq + C::BM - 1) / C::BM) * a.BH;
  const int grid = static_cast<int>(units < nsm ? units : nsm);
  const float c_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  const cudaError_t e = launch_pdl(kern, dim3(grid), dim3(C::NTHREADS), C::SMEM, a.stream, mQ, mK, mV,
                                   static_cast<__nv_bfloat16*>(a.O), a.L, a.BH, a.Nq, a.Nk, a.window, c_log2,
                                   head_group(a.BH, a.Nq, a.Nk, D), counter, a.status, a.counter);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status launch_fwd_persist(const FwdLaunch& a) {
  switch (a.d) {
#define FA_PF_MASKS(D) \
  (a.window > 0 ? launch_persist_t<D, 2>(a) : a.causal ? launch_persist_t<D, 1>(a) : launch_persist_t<D, 0>(a))
    case 32: return FA_PF_MASKS(32);
    case 64: return FA_PF_MASKS(64);
    case 128: return FA_PF_MASKS(128);
#undef FA_PF_MASKS
    default: return FA_ERR_UNSUPPORTED;
  }
}

}  // namespace fa
