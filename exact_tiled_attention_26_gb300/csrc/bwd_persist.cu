// Backward pass, head sizes 64 and 128, persistent: one CTA per SM takes (key tile,
// head) work units from a queue until none is left.
//
// Each unit is exactly the work of a bwd_tile.cu CTA ("CS336 Assignment 2 notes"
// §1.4, Equations 13-19, key/value tiles outer; the same roles, tensor-memory
// layout and per-step barriers, and the same per-step code, bwd_steps.cuh).  A
// bwd_tile.cu CTA pays a fixed cost of about 9 us at d = 128 (measured on GB300:
// launch, the K, V load, the first step before anything overlaps, the dK, dV
// epilogue, the last dQ drain), several steps' worth; here the next unit's first
// loads and its first S^T, dP^T overlap the current unit's epilogue and last drain,
// and units are taken from a counter in launch order (longest causal loops first,
// heads in groups, as in bwd_tile.cu), so the SMs also finish together.
//
// What runs on across units: the step count g (Q, dO stages, the two alternating
// tensor-memory regions and every per-step barrier phase), and the unit count k
// (K and V: NKV buffers, unit k in buffer k % NKV, reloaded once the last readers of
// unit k - NKV -- both UMMA issuers -- are done; dK and dV: the element-wise warps
// take them out of tensor memory and release them before the next unit's first dV,
// dK products).  At d = 128 shared memory holds one K, V buffer, so every unit
// boundary waits for the next unit's K and V to arrive (a few microseconds); at
// d = 64 it holds two, and the next unit's K and V load while the current unit
// runs.
#include <mutex>

#include "bwd_steps.cuh"
#include "internal.h"

namespace fa {

// Work counters of the persistent backward launches (as for the persistent
// forward: one pair per launch, left zeroed by it, up to kBwdQueueSlots in flight).
constexpr int kBwdQueueSlots = 1024;
__device__ unsigned int g_bwd_queue[2 * kBwdQueueSlots];

namespace {

using namespace bsteps;

// Barriers of this kernel beyond the per-step ones (bwd_steps.cuh).
enum : int {
  B_KVFULL = 0, B_FINAL = 17, B_ADONE = 18,
  B_KVFREE = 20,   // the unit's last readers of K and V are done (one commit from each issuer)
  B_DKVFULL = 21,  // the unit's dK, dV are complete in tensor memory
  B_DKVFREE = 22,  // the element-wise warps have taken them out
  B_UFULL = 23, B_UEMPTY = 25,  // unit ring, two slots
  B_KVFULL1 = 27, B_KVFREE1 = 28,  // the second K, V buffer's (d = 64)
  NBAR = 29
};
FA_DEV int kvfull(int b) { return b == 0 ? B_KVFULL : B_KVFULL1; }
FA_DEV int kvfree(int b) { return b == 0 ? B_KVFREE : B_KVFREE1; }
constexpr int UEMPTY_COUNT = 1 + 1 + 8 + 4;  // issuers A and B, 8 element-wise and 4 drain warps
constexpr int OFF_MISC = NBAR * 8;           // tensor-memory base, abort flag, unit ring
constexpr int NTHREADS = 512;
static_assert(OFF_MISC + 16 <= OFF_LD, "small region");

enum : int { SITE_P_PRODUCER = 0x231, SITE_P_MMA = 0x232, SITE_P_COMPUTE = 0x233, SITE_P_LAYOUT = 0x235 };

// Unit u -> key tile and head (grouped launch order) and the visible query tiles.
struct BUnit {
  int kt, bh, i0, n_it;
};
template <bool CAUSAL>
FA_DEV BUnit decode_bunit(int u, int Tk, int BH, int hg, int Nq, int Nk, int window) {
  BUnit x;
  grouped_tile_head(u, Tk, BH, hg, &x.kt, &x.bh);
  int ilast = 0;
  query_tile_range(x.kt, BM, BN, Nq, Nk, CAUSAL, window, &x.i0, &ilast);
  x.n_it = ilast >= x.i0 ? ilast - x.i0 + 1 : 0;
  return x;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(NTHREADS, 1)
    bwd_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                     const float* __restrict__ Lg, const float* __restrict__ Dg, float* __restrict__ dQacc,
                     __nv_bfloat16* __restrict__ dK, __nv_bfloat16* __restrict__ dV, int BH, int Nq, int Nk,
                     int window, float c_log2, float scale, int head_group, unsigned int* queue, int* status,
                     unsigned long long* tile_counter) {
  using LY = LayFor<D>;
  constexpr int NKV = LY::NKV;  // K, V buffers
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = align1024(smem_raw + SMALL);
  if (tiles + LY::TILES > smem_raw + LY::SMEM) {
    if (threadIdx.x == 0) {
      atomicCAS(status, 0, SITE_P_LAYOUT);
      queue_release(queue);
    }
    return;
  }
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + OFF_MISC + 4);
  volatile int* unit_ring = reinterpret_cast<volatile int*>(smem_raw + OFF_MISC + 8);
  Ctx x{smem_u32(smem_raw), smem_u32(tiles), smem_raw, tiles, 0u, Guard{status, abort_flag}};
  auto bar = [&](int i) -> uint32_t { return x.bar(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Tk = (Nk + BN - 1) / BN;
  const int U = Tk * BH;
  const int off = Nk - Nq;  // position of query row i is i + off
  auto decode = [&](int u) { return decode_bunit<CAUSAL>(u, Tk, BH, head_group, Nq, Nk, window); };

  if (threadIdx.x == 0) {
    for (int b = 0; b < NKV; ++b) {
      mbar_init(bar(kvfull(b)), 1);
      mbar_init(bar(kvfree(b)), 2);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_QFULL + s), 1 + 32);  // TMA bytes + the producer's 32 lanes (L, D)
      mbar_init(bar(B_QEMPTY + s), 1);
      mbar_init(bar(B_UFULL + s), 1);
      mbar_init(bar(B_UEMPTY + s), UEMPTY_COUNT);
    }
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_DPFULL), 1);
    for (int c = 0; c < 2; ++c) {
      mbar_init(bar(B_PREADY + c), NCOMP);
      mbar_init(bar(B_PREADY + 2 + c), NCOMP);
      mbar_init(bar(B_DSREADY + c), NCOMP);
    }
    mbar_init(bar(B_DPCONS), NCOMP);
    mbar_init(bar(B_DSSMEM), NCOMP);
    mbar_init(bar(B_DKDONE), 1);
    mbar_init(bar(B_DQFULL), 1);
    mbar_init(bar(B_DQCONS), NDQ);
    mbar_init(bar(B_FINAL), 1);
    mbar_init(bar(B_ADONE), 1);
    mbar_init(bar(B_DKVFULL), 1);
    mbar_init(bar(B_DKVFREE), NCOMP);
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
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  x.tmem = *tmem_slot;
  const bool skip = *abort_flag != 0;

  // Every role takes unit k from ring slot k % 2 and releases the slot.  `site`: the
  // role's wait-site code.
  auto take_unit = [&](int k, bool warp_wide, int site, int* u) -> bool {
    const int slot = k & 1;
    const bool ok = warp_wide ? mbar_wait_warp(bar(B_UFULL + slot), (k >> 1) & 1, x.guard, site)
                              : mbar_wait(bar(B_UFULL + slot), (k >> 1) & 1, x.guard, site);
    if (!ok) return false;
    *u = unit_ring[slot];
    if (warp_wide) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_UEMPTY + slot));
    } else {
      mbar_arrive(bar(B_UEMPTY + slot));
    }
    return true;
  };

  if (warp < 4) {
  regs_dec<72>();
  if (warp == 0 && !skip) {
    // ---------------------------------------------------------------- producer (whole warp)
    int g = 0, last = -1, kvk = -1;  // steps so far; last step and last unit whose loads were issued
    for (int k = 0;; ++k) {
      const int slot = k & 1;
      int u = 0;
      if (lane == 0) {  // the CTA's own first unit, then the queue after the grid's first units
        u = k == 0 ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x + atomicAdd(queue, 1u));
        if (u >= U) u = -1;
      }
      u = __shfl_sync(0xffffffffu, u, 0);
      // ring slot k % 2 last held unit k-2: every consumer has read it
      if (k >= 2 && !mbar_wait_warp(bar(B_UEMPTY + slot), ((k >> 1) & 1) ^ 1, x.guard, SITE_P_PRODUCER)) break;
      if (lane == 0) {
        unit_ring[slot] = u;
        mbar_arrive(bar(B_UFULL + slot));
      }
      if (u < 0) break;
      const BUnit w = decode(u);
      // K and V of this unit into buffer k % NKV, once the last readers of unit k - NKV
      // (which used it) are done
      const int b = k % NKV;
      if (lane == 0 && k >= NKV) {  // used once per unit: bring the descriptors back into their cache
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
      }
      if (k >= NKV && !mbar_wait_warp(bar(kvfree(b)), (k / NKV - 1) & 1, x.guard, SITE_P_PRODUCER)) break;
      if (lane == 0) {
        mbar_expect_tx(bar(kvfull(b)), LY::KVB);
        for (int c = 0; c < 2; ++c)  // at d = 64 the second K chunk is a copy of the first
          tma_load_3d(LY::k(x.tb, b) + c * CHUNK, &tmK, bar(kvfull(b)), D == 128 ? c * 64 : 0, w.kt * BN, w.bh);
        for (int c = 0; c < LY::TQ / CHUNK; ++c)
          tma_load_3d(LY::v(x.tb, b) + c * CHUNK, &tmV, bar(kvfull(b)), c * 64, w.kt * BN, w.bh);
      }
      kvk = k;
      bool ok = true;
      const size_t row0 = static_cast<size_t>(w.bh) * Nq;
      for (int it = 0; ok && it < w.n_it; ++it, ++g) {
        ok = produce_step<LY>(x, &tmQ, &tmdO, Lg, Dg, row0, Nq, (w.i0 + it) * BM, w.bh, g, lane, SITE_P_PRODUCER);
        if (ok) last = g;
      }
      if (!ok) break;
    }
    if (lane == 0 && *abort_flag) {
      for (int kk = (kvk >= NKV ? kvk - NKV + 1 : 0); kk <= kvk; ++kk)  // the K, V loads in flight
        mbar_drain(bar(kvfull(kk % NKV)), (kk / NKV) & 1);
      for (int it = (last > 0 ? last - 1 : 0); it <= last; ++it) mbar_drain(bar(B_QFULL + (it & 1)), (it >> 1) & 1);
    }
  } else if (warp == 1 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- UMMA issuer A: S^T, dP^T
    bool ok = true;
    int g = 0;
    for (int k = 0; ok; ++k) {
      int u = 0;
      if (!(ok = take_unit(k, false, SITE_P_MMA, &u)) || u < 0) break;
      const BUnit w = decode(u);
      const int b = k % NKV;
      if (!(ok = mbar_wait(bar(kvfull(b)), (k / NKV) & 1, x.guard, SITE_P_MMA))) break;
      for (int it = 0; ok && it < w.n_it; ++it, ++g) ok = issue_s_dp<LY>(x, g, b, SITE_P_MMA);
      if (!ok) break;
      mma_commit(bar(kvfree(b)));  // this unit's S^T, dP^T products (the readers of K, V here) are done
    }
    mma_commit(bar(B_ADONE));
    if (ok && tile_counter != nullptr) atomicAdd(tile_counter, static_cast<unsigned long long>(g));
  } else if (warp == 2 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- UMMA issuer B: dV, dK, dQ^T
    bool ok = true;
    int g = 0;
    for (int k = 0; ok; ++k) {
      int u = 0;
      if (!(ok = take_unit(k, false, SITE_P_MMA, &u)) || u < 0) break;
      const BUnit w = decode(u);
      // dK, dV of the previous unit are out of tensor memory (waited for every unit,
      // even one without steps, so that this barrier is never two phases behind)
      if (k > 0 && !(ok = mbar_wait(bar(B_DKVFREE), (k - 1) & 1, x.guard, SITE_P_MMA))) break;
      const int b = k % NKV;
      if (!(ok = mbar_wait(bar(kvfull(b)), (k / NKV) & 1, x.guard, SITE_P_MMA))) break;
      for (int it = 0; ok && it < w.n_it; ++it, ++g) ok = issue_dv_dk_dq<LY>(x, g, b, it == 0, SITE_P_MMA);
      if (!ok) break;
      mma_commit(bar(B_DKVFULL));  // this unit's dK, dV are complete
      mma_commit(bar(kvfree(b)));  // and its dQ^T products (the last readers of K) are done
    }
    mma_commit(bar(B_FINAL));
  }
  } else if (warp >= 12) {
    regs_inc<144>();
    if (!skip) {
    // ---------------------------------------------------------------- dQ drain
    pdl_wait();  // the workspace is cleared by the kernel before this one
    const int qw = warp & 3;
    bool ok = true;
    int g = 0;
    for (int k = 0; ok; ++k) {
      int u = 0;
      if (!(ok = take_unit(k, true, SITE_P_COMPUTE, &u)) || u < 0) break;
      const BUnit w = decode(u);
      const size_t row0 = static_cast<size_t>(w.bh) * Nq;
      for (int j = 0; ok && j < w.n_it; ++j, ++g) {
        const int q0 = (w.i0 + j) * BM;
        ok = drain_step<D>(x, g, dQacc + (row0 + q0) * D, min(BM, Nq - q0), qw, lane, SITE_P_COMPUTE);
      }
    }
    }
  } else {
    regs_inc<144>();
    if (!skip) {
    // ---------------------------------------------------------------- element-wise warps
    const int qw = warp & 3;
    const int h = (warp - 4) >> 2;
    bool ok = true;
    int g = 0;
    // dK, dV rows of the previous unit, held from its end until the next unit's K, V
    // are in shared memory, so that their stores do not compete with that load
    uint32_t outp[D / 2];
    size_t prow0 = 0;
    int pvalid = 0;
    bool pending = false;
    for (int k = 0; ok; ++k) {
      int u = 0;
      if (!(ok = take_unit(k, true, SITE_P_COMPUTE, &u))) break;
      if (pending) {
        if (u >= 0 && !(ok = mbar_wait_warp(bar(kvfull(k % NKV)), (k / NKV) & 1, x.guard, SITE_P_COMPUTE))) break;
        ew_store_dk_dv<D>(outp, dK, dV, prow0, pvalid, h, lane);
        pending = false;
      }
      if (u < 0) break;
      const BUnit w = decode(u);
      for (int it = 0; ok && it < w.n_it; ++it, ++g)
        ok = ew_step<LY, CAUSAL>(x, g, w.kt, w.i0 + it, Nk, off, window, c_log2, qw, h, lane, SITE_P_COMPUTE);
      if (!ok) break;
      // dK (times scale) and dV of this unit: taken out of tensor memory first and
      // released to the next unit
      if (!(ok = mbar_wait_warp(bar(B_DKVFULL), k & 1, x.guard, SITE_P_COMPUTE))) break;
      tc_fence_after();
      ew_load_dk_dv<D>(x, qw, h, scale, w.n_it == 0, outp);
      tc_fence_before();
      mbar_arrive(bar(B_DKVFREE));
      const int row0 = w.kt * BN + qw * 32;
      prow0 = static_cast<size_t>(w.bh) * Nk + row0;
      pvalid = Nk - row0;
      pending = true;
    }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (!skip && *abort_flag) {
      if (lane == 0) {
        mbar_drain(bar(B_ADONE), 0);
        mbar_drain(bar(B_FINAL), 0);
      }
      __syncwarp();
    }
    tc_fence_after();
    tmem_dealloc(x.tmem, TM_COLS);
  }
  if (threadIdx.x == 0) queue_release(queue);
}

std::mutex g_bq_mu;
int g_bq_next = 0;
unsigned int* g_bq_base[64] = {nullptr};
int g_bq_nsm[64] = {0};

template <int D, bool CAUSAL>
fa_status launch_p(const BwdLaunch& a) {
  using LY = LayFor<D>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_CUDA;
  unsigned int* counter = nullptr;
  int nsm = 0;
  {
    std::lock_guard<std::mutex> lk(g_bq_mu);
    if (g_bq_base[dev] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_bwd_queue) != cudaSuccess) return FA_ERR_CUDA;
      if (cudaDeviceGetAttribute(&g_bq_nsm[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FA_ERR_CUDA;
      g_bq_base[dev] = static_cast<unsigned int*>(p);
    }
    counter = g_bq_base[dev] + 2 * g_bq_next;
    g_bq_next = (g_bq_next + 1) % kBwdQueueSlots;
    nsm = g_bq_nsm[dev];
  }
  CUtensorMap mQ, mK, mV, mdO;
  if (!encode_bf16_3d(&mQ, a.Q, D, a.Nq, a.BH, 64, BM) || !encode_bf16_3d(&mdO, a.dO, D, a.Nq, a.BH, 64, BM) ||
      !encode_bf16_3d(&mK, a.K, D, a.Nk, a.BH, 64, BN) || !encode_bf16_3d(&mV, a.V, D, a.Nk, a.BH, 64, BN))
    return FA_ERR_CUDA;
  auto kern = bwd_persist_kernel<D, CAUSAL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM) != cudaSuccess)
    return FA_ERR_CUDA;
  const long long units = static_cast<long long>((a.Nk + BN - 1) / BN) * a.BH;
  const int grid = static_cast<int>(units < nsm ? units : nsm);
  const float c_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  // Launched so that it may start while the workspace is being cleared (as bwd_tile.cu).
  const cudaError_t e = launch_pdl(kern, dim3(grid), dim3(NTHREADS), LY::SMEM, a.stream, mQ, mK, mV, mdO, a.L,
                                   a.D, a.dQacc, static_cast<__nv_bfloat16*>(a.dK),
                                   static_cast<__nv_bfloat16*>(a.dV), a.BH, a.Nq, a.Nk, a.window, c_log2, a.scale,
                                   head_group(a.BH, a.Nq, a.Nk, D), counter, a.status, a.counter);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status launch_bwd_persist(const BwdLaunch& a) {
  if (a.d == 64) return a.causal ? launch_p<64, true>(a) : launch_p<64, false>(a);
  return a.causal ? launch_p<128, true>(a) : launch_p<128, false>(a);
}

}  // namespace fa
