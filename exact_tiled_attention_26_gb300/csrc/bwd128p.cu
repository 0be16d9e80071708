// Backward pass, head size 128, persistent: one CTA per SM takes (key tile, head)
// work units from a queue until none is left.
//
// Each unit is exactly the work of a bwd128.cu CTA ("CS336 Assignment 2 notes"
// §1.4, Equations 13-19, key/value tiles outer; the same roles, tensor-memory
// layout and per-step barriers).  A bwd128.cu CTA pays a fixed cost of about 9 us
// (measured on GB300: launch, the K, V load, the first step before anything
// overlaps, the dK, dV epilogue, the last dQ drain), several steps' worth; here the
// next unit's first loads and its first S^T, dP^T overlap the current unit's
// epilogue and last drain, and units are taken from a counter in launch order
// (longest causal loops first, heads in groups, as in bwd128.cu), so the SMs also
// finish together.
//
// What runs on across units: the step count g (Q, dO stages, the two alternating
// tensor-memory regions and every per-step barrier phase), and the unit count k
// (K and V: one buffer, reloaded once the unit's last readers -- both UMMA
// issuers -- are done; dK and dV: the element-wise warps take them out of tensor
// memory and release them before the next unit's first dV, dK products).
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace fa {

// Work counters of the persistent backward launches (as for the persistent
// forward: one per launch, zeroed on its stream, up to kBwdQueueSlots in flight).
constexpr int kBwdQueueSlots = 1024;
__device__ unsigned int g_bwd_queue[kBwdQueueSlots];

namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct B128P {
  static constexpr int D = 128, BN = 128, BM = 128;
  static constexpr int NTHREADS = 512;
  static constexpr int NCOMP = 256;  // element-wise threads
  static constexpr int NDQ = 128;    // dQ drain threads
  static constexpr int TILE = 128 * 128 * 2;
  enum : int {
    B_KVFULL = 0, B_QFULL = 1, B_QEMPTY = 3, B_SFULL = 5, B_DPFULL = 6,
    B_PREADY = 7,  // [step parity][sub-chunk]
    B_DSREADY = 11, B_DKDONE = 13, B_DQFULL = 14, B_DQCONS = 15, B_DPCONS = 16, B_FINAL = 17, B_ADONE = 18,
    B_DSSMEM = 19,
    B_KVFREE = 20,   // the unit's last readers of K and V are done (one commit from each issuer)
    B_DKVFULL = 21,  // the unit's dK, dV are complete in tensor memory
    B_DKVFREE = 22,  // the element-wise warps have taken them out
    B_UFULL = 23, B_UEMPTY = 25,  // unit ring, two slots
    NBAR = 27
  };
  static constexpr int UEMPTY_COUNT = 1 + 1 + 8 + 4;  // issuers A and B, 8 element-wise and 4 drain warps
  static constexpr int OFF_BAR = 0;
  static constexpr int OFF_MISC = NBAR * 8;  // tensor-memory base, abort flag, unit ring
  static constexpr int OFF_LD = 256;
  static constexpr int LD_BYTES = 2 * BM * 4;
  static constexpr int SMALL = OFF_LD + 2 * LD_BYTES;
  static constexpr int T_K = 0, T_V = TILE, T_Q = 2 * TILE, T_DO = 3 * TILE;
  static constexpr int T_DS = 6 * TILE;
  static constexpr int TILES = 7 * TILE;
  static constexpr int SMEM = 232448;
  static constexpr int TM_DK = 0, TM_DV = 128, TM_R = 256, TM_COLS = 512;
  static_assert(OFF_MISC + 16 <= OFF_LD, "small region");
  static_assert(SMALL <= 3072 && 3072 + TILES <= SMEM, "shared memory budget");
};

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
  query_tile_range(x.kt, B128P::BM, B128P::BN, Nq, Nk, CAUSAL, window, &x.i0, &ilast);
  x.n_it = ilast >= x.i0 ? ilast - x.i0 + 1 : 0;
  return x;
}

template <bool CAUSAL>
__global__ void __launch_bounds__(B128P::NTHREADS, 1)
    bwd_d128p_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                     const float* __restrict__ Lg, const float* __restrict__ Dg, float* __restrict__ dQacc,
                     __nv_bfloat16* __restrict__ dK, __nv_bfloat16* __restrict__ dV, int BH, int Nq, int Nk,
                     int window, float c_log2, float scale, int head_group, unsigned int* queue, int* status,
                     unsigned long long* tile_counter) {
  using C = B128P;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = align1024(smem_raw + C::SMALL);
  if (tiles + C::TILES > smem_raw + C::SMEM) {
    if (threadIdx.x == 0) atomicCAS(status, 0, SITE_P_LAYOUT);
    return;
  }
  const uint32_t sb = smem_u32(smem_raw);
  const uint32_t tb = smem_u32(tiles);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + C::OFF_MISC + 4);
  volatile int* unit_ring = reinterpret_cast<volatile int*>(smem_raw + C::OFF_MISC + 8);
  const Guard guard{status, abort_flag};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Tk = (Nk + C::BN - 1) / C::BN;
  const int U = Tk * BH;
  const int off = Nk - Nq;  // position of query row i is i + off
  auto decode = [&](int u) { return decode_bunit<CAUSAL>(u, Tk, BH, head_group, Nq, Nk, window); };

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_KVFULL), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_QFULL + s), 1 + 32);  // TMA bytes + the producer's 32 lanes (L, D)
      mbar_init(bar(C::B_QEMPTY + s), 1);
      mbar_init(bar(C::B_UFULL + s), 1);
      mbar_init(bar(C::B_UEMPTY + s), C::UEMPTY_COUNT);
    }
    mbar_init(bar(C::B_SFULL), 1);
    mbar_init(bar(C::B_DPFULL), 1);
    for (int c = 0; c < 2; ++c) {
      mbar_init(bar(C::B_PREADY + c), C::NCOMP);
      mbar_init(bar(C::B_PREADY + 2 + c), C::NCOMP);
      mbar_init(bar(C::B_DSREADY + c), C::NCOMP);
    }
    mbar_init(bar(C::B_DPCONS), C::NCOMP);
    mbar_init(bar(C::B_DSSMEM), C::NCOMP);
    mbar_init(bar(C::B_DKDONE), 1);
    mbar_init(bar(C::B_DQFULL), 1);
    mbar_init(bar(C::B_DQCONS), C::NDQ);
    mbar_init(bar(C::B_FINAL), 1);
    mbar_init(bar(C::B_ADONE), 1);
    mbar_init(bar(C::B_KVFREE), 2);
    mbar_init(bar(C::B_DKVFULL), 1);
    mbar_init(bar(C::B_DKVFREE), C::NCOMP);
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

  if (warp < 4) {
  regs_dec<72>();
  if (warp == 0 && !skip) {
    // ---------------------------------------------------------------- producer (whole warp)
    int g = 0, last = -1, kvk = -1;  // steps so far; last step and last unit whose loads were issued
    for (int k = 0;; ++k) {
      const int slot = k & 1;
      int u = 0;
      if (lane == 0) {
        u = static_cast<int>(atomicAdd(queue, 1u));
        if (u >= U) u = -1;
      }
      u = __shfl_sync(0xffffffffu, u, 0);
      // ring slot k % 2 last held unit k-2: every consumer has read it
      if (k >= 2 && !mbar_wait_warp(bar(C::B_UEMPTY + slot), ((k >> 1) & 1) ^ 1, guard, SITE_P_PRODUCER)) break;
      if (lane == 0) {
        unit_ring[slot] = u;
        mbar_arrive(bar(C::B_UFULL + slot));
      }
      if (u < 0) break;
      const BUnit x = decode(u);
      const size_t row0 = static_cast<size_t>(x.bh) * Nq;
      // K and V of this unit, once the previous unit's last readers are done
      if (k >= 1 && !mbar_wait_warp(bar(C::B_KVFREE), (k - 1) & 1, guard, SITE_P_PRODUCER)) break;
      if (lane == 0) {
        mbar_expect_tx(bar(C::B_KVFULL), 2 * C::TILE);
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(tb + C::T_K + c * 128 * 128, &tmK, bar(C::B_KVFULL), c * 64, x.kt * C::BN, x.bh);
          tma_load_3d(tb + C::T_V + c * 128 * 128, &tmV, bar(C::B_KVFULL), c * 64, x.kt * C::BN, x.bh);
        }
      }
      kvk = k;
      bool ok = true;
      for (int it = 0; it < x.n_it; ++it, ++g) {
        const int s = g & 1;
        const int q0 = (x.i0 + it) * C::BM;
        float lv[4], dv[4];
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
          const int q = q0 + lane + 32 * uu;
          lv[uu] = q < Nq ? -Lg[row0 + q] * kLog2e : -INFINITY;
          dv[uu] = q < Nq ? Dg[row0 + q] : 0.f;
        }
        if (!(ok = mbar_wait_warp(bar(C::B_QEMPTY + s), ((g >> 1) & 1) ^ 1, guard, SITE_P_PRODUCER))) break;
        if (lane == 0) {
          mbar_expect_tx(bar(C::B_QFULL + s), 2 * C::TILE);
          for (int c = 0; c < 2; ++c) {
            tma_load_3d(tb + C::T_Q + s * 2 * C::TILE + c * 128 * 128, &tmQ, bar(C::B_QFULL + s), c * 64, q0, x.bh);
            tma_load_3d(tb + C::T_DO + s * 2 * C::TILE + c * 128 * 128, &tmdO, bar(C::B_QFULL + s), c * 64, q0,
                        x.bh);
          }
        }
        float* Ls = reinterpret_cast<float*>(smem_raw + C::OFF_LD + s * C::LD_BYTES);
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
          Ls[lane + 32 * uu] = lv[uu];
          Ls[C::BM + lane + 32 * uu] = dv[uu];
        }
        mbar_arrive(bar(C::B_QFULL + s));
        last = g;
      }
      if (!ok) break;
    }
    if (lane == 0 && *abort_flag) {
      if (kvk >= 0) mbar_drain(bar(C::B_KVFULL), kvk & 1);
      for (int it = (last > 0 ? last - 1 : 0); it <= last; ++it)
        mbar_drain(bar(C::B_QFULL + (it & 1)), (it >> 1) & 1);
    }
  } else if (warp == 1 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- UMMA issuer A: S^T, dP^T
    constexpr uint32_t idKK = idesc_bf16(128, 128, false, false);
    const uint32_t kb = tb + C::T_K, vb = tb + C::T_V;
    bool ok = true;
    int g = 0;
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (!(ok = mbar_wait(bar(C::B_UFULL + slot), (k >> 1) & 1, guard, SITE_P_MMA))) break;
      const int u = unit_ring[slot];
      mbar_arrive(bar(C::B_UEMPTY + slot));
      if (u < 0) break;
      const BUnit x = decode(u);
      if (!(ok = mbar_wait(bar(C::B_KVFULL), k & 1, guard, SITE_P_MMA))) break;
      for (int it = 0; it < x.n_it; ++it, ++g) {
        const int s = g & 1;
        const uint32_t qb = tb + C::T_Q + s * 2 * C::TILE, db = tb + C::T_DO + s * 2 * C::TILE;
        const uint32_t rs = tmem + C::TM_R + 128 * s, rd = tmem + C::TM_R + 128 * (s ^ 1);
        if (!(ok = mbar_wait(bar(C::B_QFULL + s), (g >> 1) & 1, guard, SITE_P_MMA))) break;
        // region s held dP^T of the previous step: every element-wise thread has read it
        if (g > 0 && !(ok = mbar_wait(bar(C::B_DPCONS), (g - 1) & 1, guard, SITE_P_MMA))) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ss(rs, sdesc_kmajor<128, 128>(kb, ks), sdesc_kmajor<128, 128>(qb, ks), idKK, ks > 0);
        mma_commit(bar(C::B_SFULL));
        // region s^1 ended the previous step holding its dQ^T: the drain warps have read it
        if (g > 0 && !(ok = mbar_wait(bar(C::B_DQCONS), (g - 1) & 1, guard, SITE_P_MMA))) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ss(rd, sdesc_kmajor<128, 128>(vb, ks), sdesc_kmajor<128, 128>(db, ks), idKK, ks > 0);
        mma_commit(bar(C::B_DPFULL));
      }
      if (!ok) break;
      mma_commit(bar(C::B_KVFREE));  // this unit's S^T, dP^T products (the readers of K, V here) are done
    }
    mma_commit(bar(C::B_ADONE));
    if (ok && tile_counter != nullptr) atomicAdd(tile_counter, static_cast<unsigned long long>(g));
  } else if (warp == 2 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- UMMA issuer B: dV, dK, dQ^T
    constexpr uint32_t idTN = idesc_bf16(128, 128, false, true);
    constexpr uint32_t idMN = idesc_bf16(128, 128, true, true);
    const uint32_t kb = tb + C::T_K, dsb = tb + C::T_DS;
    bool ok = true;
    int g = 0;
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (!(ok = mbar_wait(bar(C::B_UFULL + slot), (k >> 1) & 1, guard, SITE_P_MMA))) break;
      const int u = unit_ring[slot];
      mbar_arrive(bar(C::B_UEMPTY + slot));
      if (u < 0) break;
      const BUnit x = decode(u);
      // dK, dV of the previous unit are out of tensor memory (waited for every unit,
      // even one without steps, so that this barrier is never two phases behind)
      if (k > 0 && !(ok = mbar_wait(bar(C::B_DKVFREE), (k - 1) & 1, guard, SITE_P_MMA))) break;
      if (!(ok = mbar_wait(bar(C::B_KVFULL), k & 1, guard, SITE_P_MMA))) break;
      for (int it = 0; it < x.n_it; ++it, ++g) {
        const int s = g & 1;
        const uint32_t qb = tb + C::T_Q + s * 2 * C::TILE, db = tb + C::T_DO + s * 2 * C::TILE;
        const uint32_t rs = tmem + C::TM_R + 128 * s;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (!(ok = mbar_wait(bar(C::B_PREADY + 2 * s + c), (g >> 1) & 1, guard, SITE_P_MMA))) break;
          tc_fence_after();
#pragma unroll
          for (int uu = 0; uu < 4; ++uu) {
            const int ks = 4 * (uu >> 1) + 2 * c + (uu & 1);
            mma_ts(tmem + C::TM_DV, rs + 64 * (ks >> 2) + (ks & 3) * 8, sdesc_mnmajor<128, 128>(db, ks), idTN,
                   (it > 0 || ks > 0));
          }
        }
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (!(ok = mbar_wait(bar(C::B_DSREADY + c), g & 1, guard, SITE_P_MMA))) break;
          tc_fence_after();
#pragma unroll
          for (int uu = 0; uu < 4; ++uu) {
            const int ks = 4 * (uu >> 1) + 2 * c + (uu & 1);
            mma_ts(tmem + C::TM_DK, rs + 64 * (ks >> 2) + 32 + (ks & 3) * 8, sdesc_mnmajor<128, 128>(qb, ks), idTN,
                   (it > 0 || ks > 0));
          }
        }
        if (!ok) break;
        mma_commit(bar(C::B_DKDONE));
        mma_commit(bar(C::B_QEMPTY + s));
        if (!(ok = mbar_wait(bar(C::B_DKDONE), g & 1, guard, SITE_P_MMA))) break;
        if (!(ok = mbar_wait(bar(C::B_DSSMEM), g & 1, guard, SITE_P_MMA))) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ss(rs, sdesc_mnmajor<128, 128>(kb, ks), sdesc_mnmajor<128, 128>(dsb, ks), idMN, ks > 0);
        mma_commit(bar(C::B_DQFULL));
      }
      if (!ok) break;
      mma_commit(bar(C::B_DKVFULL));  // this unit's dK, dV are complete
      mma_commit(bar(C::B_KVFREE));   // and its dQ^T products (the last readers of K) are done
    }
    mma_commit(bar(C::B_FINAL));
  }
  } else if (warp >= 12) {
    regs_inc<144>();
    if (!skip) {
    // ---------------------------------------------------------------- dQ drain
    const int qw = warp & 3;
    const int dd = qw * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    bool ok = true;
    int g = 0;
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (!(ok = mbar_wait_warp(bar(C::B_UFULL + slot), (k >> 1) & 1, guard, SITE_P_COMPUTE))) break;
      const int u = unit_ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_UEMPTY + slot));
      if (u < 0) break;
      const BUnit x = decode(u);
      const size_t row0 = static_cast<size_t>(x.bh) * Nq;
      for (int j = 0; j < x.n_it; ++j, ++g) {
        if (!(ok = mbar_wait_warp(bar(C::B_DQFULL), g & 1, guard, SITE_P_COMPUTE))) break;
        tc_fence_after();
        uint32_t r[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tl + C::TM_R + 128 * (g & 1) + 32 * c, r + 32 * c);
        tmem_ld_wait<128>(r);
        tc_fence_before();
        mbar_arrive(bar(C::B_DQCONS));
        const int q0 = (x.i0 + j) * C::BM;
        float* dst = dQacc + (row0 + q0) * C::D + dd;
        const int nq = min(C::BM, Nq - q0);
        if (nq >= C::BM) {
#pragma unroll
          for (int xx = 0; xx < C::BM; ++xx) atomicAdd(dst + static_cast<size_t>(xx) * C::D, __uint_as_float(r[xx]));
        } else {
#pragma unroll
          for (int xx = 0; xx < C::BM; ++xx)
            if (xx < nq) atomicAdd(dst + static_cast<size_t>(xx) * C::D, __uint_as_float(r[xx]));
        }
      }
    }
    }
  } else {
    regs_inc<144>();
    if (!skip) {
    // ---------------------------------------------------------------- element-wise warps
    const int qw = warp & 3;
    const int h = (warp - 4) >> 2;
    const int kr = qw * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    bool ok = true;
    int g = 0;
    for (int k = 0; ok; ++k) {
      const int slot = k & 1;
      if (!(ok = mbar_wait_warp(bar(C::B_UFULL + slot), (k >> 1) & 1, guard, SITE_P_COMPUTE))) break;
      const int u = unit_ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_UEMPTY + slot));
      if (u < 0) break;
      const BUnit x = decode(u);
      const int key = x.kt * C::BN + kr;
      for (int it = 0; it < x.n_it; ++it, ++g) {
        const int s = g & 1;
        if (!(ok = mbar_wait_warp(bar(C::B_QFULL + s), (g >> 1) & 1, guard, SITE_P_COMPUTE))) break;
        if (!(ok = mbar_wait_warp(bar(C::B_SFULL), g & 1, guard, SITE_P_COMPUTE))) break;
        tc_fence_after();
        const uint32_t rs = tl + C::TM_R + 128 * s, rd = tl + C::TM_R + 128 * (s ^ 1);
        const int qh = (x.i0 + it) * C::BM + 64 * h;
        const float4* L4 = reinterpret_cast<const float4*>(smem_raw + C::OFF_LD + s * C::LD_BYTES) + 16 * h;
        const float4* D4 = L4 + C::BM / 4;
        const bool masked = (CAUSAL && x.kt * C::BN + C::BN - 1 > qh + off) ||
                            (window > 0 && x.kt * C::BN <= qh + 63 + off - window) || (x.kt * C::BN + C::BN > Nk);
        const int qlo = CAUSAL ? key - off - qh : 0;
        const int qhi = key >= Nk ? -1 : (window > 0 ? key - off + window - 1 - qh : 63);
        const uint64_t cc = f2pack(c_log2, c_log2);
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          tmem_ld32(rs + 64 * h + 32 * c, r);
          tmem_ld_wait<32>(r);
          auto body = [&](auto mask_tag) {
            constexpr bool MASK = decltype(mask_tag)::value;
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const float4 l = L4[8 * c + v];
              float p[4];
#pragma unroll
              for (int y = 0; y < 4; y += 2) {
                const int xx = 4 * v + y;
                const uint64_t t = ffma2(f2pack(__uint_as_float(r[xx]), __uint_as_float(r[xx + 1])), cc,
                                         y == 0 ? f2pack(l.x, l.y) : f2pack(l.z, l.w));
                float t0, t1;
                f2unpack(t, t0, t1);
                p[y] = ex2(t0);
                p[y + 1] = ex2(t1);
                if (MASK) {
                  const int xs = 32 * c + xx;
                  if (xs < qlo || xs > qhi) p[y] = 0.f;
                  if (xs + 1 < qlo || xs + 1 > qhi) p[y + 1] = 0.f;
                }
              }
              pk[16 * c + 2 * v] = pack_bf16x2(p[0], p[1]);
              pk[16 * c + 2 * v + 1] = pack_bf16x2(p[2], p[3]);
            }
          };
          if (masked) body(std::true_type{}); else body(std::false_type{});
          tmem_st16(rs + 64 * h + 16 * c, pk + 16 * c);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(C::B_PREADY + 2 * s + c));
        }
        if (!(ok = mbar_wait_warp(bar(C::B_DPFULL), g & 1, guard, SITE_P_COMPUTE))) break;
        tc_fence_after();
        uint8_t* row = tiles + C::T_DS + h * (128 * 128) + kr * 128;
        uint32_t rdp[64];
        tmem_ld32(rd + 64 * h, rdp);
        tmem_ld32(rd + 64 * h + 32, rdp + 32);
        tmem_ld_wait<64>(rdp);
        tc_fence_before();
        mbar_arrive(bar(C::B_DPCONS));
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint32_t* r = rdp + 32 * c;
          uint32_t dk[16];
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const float4 dd = D4[8 * c + v];
#pragma unroll
            for (int y = 0; y < 4; y += 2) {
              const int xx = 4 * v + y;
              const uint32_t ww = pk[16 * c + (xx >> 1)];
              const uint64_t pp = f2pack(__uint_as_float(ww << 16), __uint_as_float(ww & 0xffff0000u));
              const uint64_t t = fadd2(f2pack(__uint_as_float(r[xx]), __uint_as_float(r[xx + 1])),
                                       y == 0 ? f2pack(-dd.x, -dd.y) : f2pack(-dd.z, -dd.w));
              float d0, d1;
              f2unpack(fmul2(pp, t), d0, d1);
              dk[xx >> 1] = pack_bf16x2(d0, d1);
            }
          }
          tmem_st16(rs + 64 * h + 32 + 16 * c, dk);
#pragma unroll
          for (int uu = 0; uu < 4; ++uu)
            *reinterpret_cast<uint4*>(row + (((4 * c + uu) ^ (kr & 7)) << 4)) =
                make_uint4(dk[4 * uu], dk[4 * uu + 1], dk[4 * uu + 2], dk[4 * uu + 3]);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(C::B_DSREADY + c));
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(C::B_DSSMEM));
      }
      if (!ok) break;
      // dK (times scale) and dV of this unit: this warp's lane quarter, d columns
      // 64h .. 64h+63, taken out of tensor memory first and released to the next unit
      if (!(ok = mbar_wait_warp(bar(C::B_DKVFULL), k & 1, guard, SITE_P_COMPUTE))) break;
      tc_fence_after();
      uint32_t outp[64];  // [dK | dV] x 32 bf16 pairs
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const float f = t == 0 ? scale : 1.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          tmem_ld32(tl + (t == 0 ? C::TM_DK : C::TM_DV) + 64 * h + 32 * c, r);
          tmem_ld_wait<32>(r);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            outp[32 * t + 16 * c + i] = x.n_it == 0 ? 0u  // no query sees these keys: dK = dV = 0
                                                    : pack_bf16x2(__uint_as_float(r[2 * i]) * f,
                                                                  __uint_as_float(r[2 * i + 1]) * f);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_DKVFREE));
      if (key < Nk) {
        const size_t krow0 = static_cast<size_t>(x.bh) * Nk;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          uint4* d4 = reinterpret_cast<uint4*>((t == 0 ? dK : dV) + (krow0 + key) * C::D + 64 * h);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            d4[i] = make_uint4(outp[32 * t + 4 * i], outp[32 * t + 4 * i + 1], outp[32 * t + 4 * i + 2],
                               outp[32 * t + 4 * i + 3]);
        }
      }
    }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (!skip && *abort_flag) {
      if (lane == 0) {
        mbar_drain(bar(C::B_ADONE), 0);
        mbar_drain(bar(C::B_FINAL), 0);
      }
      __syncwarp();
    }
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

std::mutex g_bq_mu;
int g_bq_next = 0;
unsigned int* g_bq_base[64] = {nullptr};
int g_bq_nsm[64] = {0};

template <bool CAUSAL>
fa_status launch_p(const BwdLaunch& a) {
  using C = B128P;
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
    counter = g_bq_base[dev] + g_bq_next;
    g_bq_next = (g_bq_next + 1) % kBwdQueueSlots;
    nsm = g_bq_nsm[dev];
  }
  CUtensorMap mQ, mK, mV, mdO;
  if (!encode_bf16_3d(&mQ, a.Q, C::D, a.Nq, a.BH, 64, C::BM) ||
      !encode_bf16_3d(&mdO, a.dO, C::D, a.Nq, a.BH, 64, C::BM) ||
      !encode_bf16_3d(&mK, a.K, C::D, a.Nk, a.BH, 64, C::BN) || !encode_bf16_3d(&mV, a.V, C::D, a.Nk, a.BH, 64, C::BN))
    return FA_ERR_CUDA;
  auto kern = bwd_d128p_kernel<CAUSAL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return FA_ERR_CUDA;
  if (cudaMemsetAsync(counter, 0, sizeof(unsigned int), a.stream) != cudaSuccess) return FA_ERR_CUDA;
  const long long units = static_cast<long long>((a.Nk + C::BN - 1) / C::BN) * a.BH;
  const int grid = static_cast<int>(units < nsm ? units : nsm);
  const float c_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  kern<<<grid, C::NTHREADS, C::SMEM, a.stream>>>(mQ, mK, mV, mdO, a.L, a.D, a.dQacc,
                                                 static_cast<__nv_bfloat16*>(a.dK), static_cast<__nv_bfloat16*>(a.dV),
                                                 a.BH, a.Nq, a.Nk, a.window, c_log2, a.scale,
                                                 head_group(a.BH, a.Nq, a.Nk, C::D), counter, a.status, a.counter);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status launch_bwd_d128_persist(const BwdLaunch& a) { return a.causal ? launch_p<true>(a) : launch_p<false>(a); }

}  // namespace fa
