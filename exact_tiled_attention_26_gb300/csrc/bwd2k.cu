// Backward pass, head sizes 64 and 128 (templated on d; the default form at d = 64,
// selectable at d = 128): the two-kernel form of "CS336 Assignment 2 notes" §1.4 (kernel 1
// iterates key/value tiles in its outer loop and forms dK, dV; kernel 2 iterates query tiles
// and forms dQ; S and P are computed in both).  No atomics and no workspace: each output is written once.
//
// bwd_kv_kernel: one CTA per 128 keys (keys on the 128 tensor-memory lanes),
//   S^T = K Q_i^T, dP^T = V dO_i^T (UMMA), P^T, dS^T (16 element-wise warps, 32
//   queries each), dV += P^T dO_i, dK += dS^T Q_i (UMMA, A from tensor
//   memory).  Tensor memory: dK | dV | two regions that take turns holding S^T
//   (then P^T | dS^T) and dP^T.
// bwd_q_kernel: one CTA per 128 queries (queries on the lanes; L and D of the
//   row kept in registers), S = Q K_j^T (two buffers), dP = dO V_j^T (UMMA),
//   P = 2^(S c - L log2 e), dS = P (dP - D) (16 warps, four per lane quarter, one
//   per 32-key quarter), dQ += dS K_j (UMMA, A = dS in tensor memory), then
//   dQ * scale -> bf16.  Tensor memory: S x2 | dP | dQ.
// Both kernels split UMMA issue over two threads, as the other kernels do.
#include <type_traits>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int SMEM_MAX = 232448;

enum : int { SITE_KV = 0x221, SITE_Q = 0x222 };

// ============================================================================ dK, dV
template <int D>
struct KVC {
  static constexpr int TD = 128 * D * 2, NCH = D / 64;  // a 128 x D bf16 tile, in 64-column chunks
  static constexpr int NTHREADS = 640, NCOMP = 512;  // 4 + 16 element-wise warps
  enum : int {
    B_KV = 0, B_QFULL = 1, B_QEMPTY = 3, B_SFULL = 5, B_DPFULL = 6,
    B_PREADY = 7,  // [step parity][sub-chunk]: the element-wise warps may be a step ahead of issuer B
    B_DSREADY = 11, B_DKDONE = 13, B_DPCONS = 14, B_FINAL = 15, B_ADONE = 16, NBAR = 17
  };
  static constexpr int OFF_MISC = NBAR * 8, OFF_LD = 256, LD_BYTES = 2 * 128 * 4;
  static constexpr int SMALL = OFF_LD + 2 * LD_BYTES;
  static constexpr int T_K = 0, T_V = TD, T_Q = 2 * TD, T_DO = 3 * TD;  // Q, dO: + s * 2 TD
  static constexpr int TILES = 6 * TD;
  static constexpr int SMEM = SMALL + 1024 + TILES;
  // Two 128-column regions alternate: step i keeps S^T (then P^T | dS^T) in region
  // i % 2 and dP^T in region (i + 1) % 2, so S^T of step i+1 can be formed as soon
  // as dP^T of step i has been read, while dK of step i is still being accumulated.
  static constexpr int TM_DK = 0, TM_DV = 128, TM_R = 256;  // dK, dV use D columns each
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(KVC<D>::NTHREADS, 1)
    bwd_kv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const float* __restrict__ Lg, const float* __restrict__ Dg, __nv_bfloat16* __restrict__ dK,
                  __nv_bfloat16* __restrict__ dV, int Nq, int Nk, int window, float c_log2, float scale, int* status,
                  unsigned long long* tile_counter, int head_group) {
  using C = KVC<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = align1024(smem_raw + C::SMALL);
  const uint32_t sb = smem_u32(smem_raw), tb = smem_u32(tiles);
  auto bar = [&](int i) -> uint32_t { return sb + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + C::OFF_MISC + 4);
  const Guard guard{status, abort_flag};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int kt = 0, bh = 0;  // longest causal loops first, heads in groups (grouped_tile_head)
  grouped_tile_head(blockIdx.y * gridDim.x + blockIdx.x, gridDim.x, gridDim.y, head_group, &kt, &bh);
  const int off = Nk - Nq;  // position of query row i is i + off
  int i0 = 0, ilast = 0;
  query_tile_range(kt, 128, 128, Nq, Nk, CAUSAL, window, &i0, &ilast);
  const int n_it = ilast >= i0 ? ilast - i0 + 1 : 0;  // none: this CTA writes zero dK, dV
  const size_t row0 = static_cast<size_t>(bh) * Nq, krow0 = static_cast<size_t>(bh) * Nk;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_KV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_QFULL + s), 1 + 32);
      mbar_init(bar(C::B_QEMPTY + s), 1);
      // sub-chunk c = query quarters c and 2 + c: half of the element-wise threads
      mbar_init(bar(C::B_PREADY + 2 * s), C::NCOMP / 2);
      mbar_init(bar(C::B_PREADY + 2 * s + 1), C::NCOMP / 2);
      mbar_init(bar(C::B_DSREADY + s), C::NCOMP / 2);
    }
    mbar_init(bar(C::B_SFULL), 1);
    mbar_init(bar(C::B_DPFULL), 1);
    mbar_init(bar(C::B_DKDONE), 1);
    mbar_init(bar(C::B_DPCONS), C::NCOMP);
    mbar_init(bar(C::B_FINAL), 1);
    mbar_init(bar(C::B_ADONE), 1);
    *abort_flag = (*reinterpret_cast<volatile int*>(status) != 0);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = *abort_flag != 0;

  if (warp == 0 && !skip) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      mbar_expect_tx(bar(C::B_KV), 2 * C::TD);
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_3d(tb + C::T_K + c * 128 * 128, &tmK, bar(C::B_KV), c * 64, kt * 128, bh);
        tma_load_3d(tb + C::T_V + c * 128 * 128, &tmV, bar(C::B_KV), c * 64, kt * 128, bh);
      }
    }
    int last = -1;
    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1, q0 = (i0 + it) * 128;
      float lv[4], dv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = q0 + lane + 32 * u;
        lv[u] = q < Nq ? -Lg[row0 + q] * kLog2e : -INFINITY;
        dv[u] = q < Nq ? Dg[row0 + q] : 0.f;
      }
      if (!mbar_wait_warp(bar(C::B_QEMPTY + s), ((it >> 1) & 1) ^ 1, guard, SITE_KV)) break;
      if (lane == 0) {
        mbar_expect_tx(bar(C::B_QFULL + s), 2 * C::TD);
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_3d(tb + C::T_Q + s * 2 * C::TD + c * 128 * 128, &tmQ, bar(C::B_QFULL + s), c * 64, q0, bh);
          tma_load_3d(tb + C::T_DO + s * 2 * C::TD + c * 128 * 128, &tmdO, bar(C::B_QFULL + s), c * 64, q0, bh);
        }
      }
      float* Ls = reinterpret_cast<float*>(smem_raw + C::OFF_LD + s * C::LD_BYTES);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        Ls[lane + 32 * u] = lv[u];
        Ls[128 + lane + 32 * u] = dv[u];
      }
      mbar_arrive(bar(C::B_QFULL + s));
      last = it;
    }
    if (lane == 0 && *abort_flag) {
      mbar_drain(bar(C::B_KV), 0);
      for (int it = (last > 0 ? last - 1 : 0); it <= last; ++it) mbar_drain(bar(C::B_QFULL + (it & 1)), (it >> 1) & 1);
    }
  } else if (warp == 1 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- issuer A: S^T, dP^T
    constexpr uint32_t idKK = idesc_bf16(128, 128, false, false);
    const uint32_t kb = tb + C::T_K, vb = tb + C::T_V;
    bool ok = mbar_wait(bar(C::B_KV), 0, guard, SITE_KV);
    for (int it = 0; ok && it < n_it; ++it) {
      const int s = it & 1;
      const uint32_t qb = tb + C::T_Q + s * 2 * C::TD, db = tb + C::T_DO + s * 2 * C::TD;
      const uint32_t rs = tmem + C::TM_R + 128 * s, rd = tmem + C::TM_R + 128 * (s ^ 1);
      if (!(ok = mbar_wait(bar(C::B_QFULL + s), (it >> 1) & 1, guard, SITE_KV))) break;
      // region s held dP^T of the last step: every element-wise thread has read it
      if (it > 0 && !(ok = mbar_wait(bar(C::B_DPCONS), (it - 1) & 1, guard, SITE_KV))) break;
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_ss(rs, sdesc_kmajor<128, 128>(kb, ks), sdesc_kmajor<128, 128>(qb, ks), idKK, ks > 0);
      mma_commit(bar(C::B_SFULL));
      // region s^1 held P^T and dS^T of the last step until dV and dK read them
      if (it > 0 && !(ok = mbar_wait(bar(C::B_DKDONE), (it - 1) & 1, guard, SITE_KV))) break;
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_ss(rd, sdesc_kmajor<128, 128>(vb, ks), sdesc_kmajor<128, 128>(db, ks), idKK, ks > 0);
      mma_commit(bar(C::B_DPFULL));
    }
    mma_commit(bar(C::B_ADONE));
    if (ok && tile_counter != nullptr) atomicAdd(tile_counter, static_cast<unsigned long long>(n_it));
  } else if (warp == 2 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- issuer B: dV, dK
    constexpr uint32_t idTN = idesc_bf16(128, D, false, true);
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it) {
      const int s = it & 1;
      const uint32_t qb = tb + C::T_Q + s * 2 * C::TD, db = tb + C::T_DO + s * 2 * C::TD;
      const uint32_t rs = tmem + C::TM_R + 128 * s;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (!(ok = mbar_wait(bar(C::B_PREADY + 2 * s + c), (it >> 1) & 1, guard, SITE_KV))) break;
        tc_fence_after();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ks = 4 * (u >> 1) + 2 * c + (u & 1);
          // query block ks (16 queries) is in quarter ks/2: P^T at 32 (ks/2) + 8 (ks%2)
          mma_ts(tmem + C::TM_DV, rs + 32 * (ks >> 1) + 8 * (ks & 1), sdesc_mnmajor<128, 128>(db, ks), idTN,
                 (it > 0 || ks > 0));
        }
      }
      if (!ok) break;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (!(ok = mbar_wait(bar(C::B_DSREADY + c), it & 1, guard, SITE_KV))) break;
        tc_fence_after();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ks = 4 * (u >> 1) + 2 * c + (u & 1);
          mma_ts(tmem + C::TM_DK, rs + 32 * (ks >> 1) + 16 + 8 * (ks & 1), sdesc_mnmajor<128, 128>(qb, ks), idTN,
                 (it > 0 || ks > 0));
        }
      }
      if (!ok) break;
      mma_commit(bar(C::B_DKDONE));
      mma_commit(bar(C::B_QEMPTY + s));
    }
    mma_commit(bar(C::B_FINAL));
  } else if (warp >= 4 && !skip) {
    // ---------------------------------------------------------------- element-wise warps
    // warp w: tensor-memory lane quarter w % 4 (32 keys), query quarter (w - 4) / 4
    // (32 queries); P^T and dS^T of a query quarter go over its own 32 S^T columns
    const int qw = warp & 3, qq = (warp - 4) >> 2, c = qq & 1, kr = qw * 32 + lane, key = kt * 128 + kr;
    const uint32_t tl = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    const uint64_t cc = f2pack(c_log2, c_log2);
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1;
      if (!(ok = mbar_wait_warp(bar(C::B_QFULL + s), (it >> 1) & 1, guard, SITE_KV))) break;
      if (!(ok = mbar_wait_warp(bar(C::B_SFULL), it & 1, guard, SITE_KV))) break;
      tc_fence_after();
      const uint32_t rs = tl + C::TM_R + 128 * s + 32 * qq, rd = tl + C::TM_R + 128 * (s ^ 1) + 32 * qq;
      const int q0 = (i0 + it) * 128 + 32 * qq;  // first query of this quarter
      const float4* L4 = reinterpret_cast<const float4*>(smem_raw + C::OFF_LD + s * C::LD_BYTES) + 8 * qq;
      const float4* D4 = L4 + 32;
      const bool masked = (CAUSAL && kt * 128 + 127 > q0 + off) || (window > 0 && kt * 128 <= q0 + 31 + off - window) ||
                          (kt * 128 + 128 > Nk);
      // queries of this quarter (0..31) that see this thread's key
      const int qlo = CAUSAL ? key - off - q0 : 0;
      const int qhi = key >= Nk ? -1 : (window > 0 ? key - off + window - 1 - q0 : 31);
      uint32_t pk[16];
      {
        uint32_t r[32];
        tmem_ld32(rs, r);
        tmem_ld_wait<32>(r);
        auto body = [&](auto mask_tag) {
          constexpr bool MASK = decltype(mask_tag)::value;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const float4 l = L4[v];
            float p[4];
#pragma unroll
            for (int y = 0; y < 4; y += 2) {
              const int x = 4 * v + y;
              float t0, t1;
              f2unpack(ffma2(f2pack(__uint_as_float(r[x]), __uint_as_float(r[x + 1])), cc,
                             y == 0 ? f2pack(l.x, l.y) : f2pack(l.z, l.w)),
                       t0, t1);
              p[y] = ex2(t0);
              p[y + 1] = ex2(t1);
              if (MASK) {  // visible iff qlo <= x <= qhi
                if (x < qlo || x > qhi) p[y] = 0.f;
                if (x + 1 < qlo || x + 1 > qhi) p[y + 1] = 0.f;
              }
            }
            pk[2 * v] = pack_bf16x2(p[0], p[1]);
            pk[2 * v + 1] = pack_bf16x2(p[2], p[3]);
          }
        };
        if (masked) body(std::true_type{}); else body(std::false_type{});
      }
      tmem_st16(rs, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::B_PREADY + 2 * s + c));
      if (!(ok = mbar_wait_warp(bar(C::B_DPFULL), it & 1, guard, SITE_KV))) break;
      tc_fence_after();
      // this thread's dP^T out of tensor memory first, so that S^T of the next step
      // can be formed in its region while dS is computed
      uint32_t r[32];
      tmem_ld32(rd, r);
      tmem_ld_wait<32>(r);
      tc_fence_before();
      mbar_arrive(bar(C::B_DPCONS));
      uint32_t dk[16];
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const float4 dd = D4[v];
#pragma unroll
        for (int y = 0; y < 4; y += 2) {
          const int x = 4 * v + y;
          const uint32_t w = pk[x >> 1];
          float d0, d1;
          f2unpack(fmul2(f2pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)),
                         fadd2(f2pack(__uint_as_float(r[x]), __uint_as_float(r[x + 1])),
                               y == 0 ? f2pack(-dd.x, -dd.y) : f2pack(-dd.z, -dd.w))),
                   d0, d1);
          dk[x >> 1] = pack_bf16x2(d0, d1);
        }
      }
      tmem_st16(rs + 16, dk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::B_DSREADY + c));
    }
    if (ok) ok = mbar_wait_warp(bar(C::B_FINAL), 0, guard, SITE_KV);
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const float f = t == 0 ? scale : 1.f;
        // this warp's D / 4 columns of d
        uint32_t r[32];
        if constexpr (D == 128) tmem_ld32(tl + (t == 0 ? C::TM_DK : C::TM_DV) + 32 * qq, r);
        else tmem_ld16(tl + (t == 0 ? C::TM_DK : C::TM_DV) + 16 * qq, r);
        tmem_ld_wait<32>(r);
        // this warp's D / 4 columns of its 32 key rows, as packed bf16 (zero when no query
        // sees these keys: the accumulators were never written)
        uint32_t pk[D / 8];
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
          pk[i] = n_it == 0 ? 0u : pack_bf16x2(__uint_as_float(r[2 * i]) * f, __uint_as_float(r[2 * i + 1]) * f);
        const int w0 = kt * 128 + qw * 32;  // the warp's first key row
        warp_store_rows<D / 32, 0>(pk, reinterpret_cast<uint8_t*>((t == 0 ? dK : dV) + (krow0 + w0) * D + (D / 4) * qq),
                                   D * 2, Nk - w0, lane);
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
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================ dQ
template <int D>
struct QC {
  static constexpr int TD = 128 * D * 2, NCH = D / 64;
  static constexpr int NTHREADS = 640, NCOMP = 512;  // 4 + 16 element-wise warps
  // K_j lives until dQ_j is done, V_j only until dP_j is: three K stages and two
  // V stages let each load start two steps ahead of its use.
  static constexpr int KST = 3, VST = 2;
  enum : int {
    B_QDO = 0, B_KFULL = 1, B_KEMPTY = 4, B_VFULL = 7, B_VEMPTY = 9, B_SFULL = 11, B_SFREE = 13, B_DPFULL = 15,
    B_DSREADY = 16,  // [S buffer][sub-chunk]
    B_FINAL = 20, B_ADONE = 21, B_DPCONS = 22, NBAR = 23
  };
  static constexpr int OFF_MISC = NBAR * 8;
  static constexpr int SMALL = 256;
  static constexpr int T_Q = 0, T_DO = TD, T_K = 2 * TD, T_V = (2 + KST) * TD;  // stage k: + k TD
  static constexpr int TILES = (2 + KST + VST) * TD;
  static constexpr int SMEM = SMALL + 1024 + TILES;
  static constexpr int TM_S = 0, TM_DP = 256, TM_DQ = 384;  // S buffer b at TM_S + 128 b
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(QC<D>::NTHREADS, 1)
    bwd_q_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                 const float* __restrict__ Lg, const float* __restrict__ Dg, __nv_bfloat16* __restrict__ dQ, int Nq, int Nk, int window,
                 float c_log2, float scale, int* status, int head_group) {
  using C = QC<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = align1024(smem_raw + C::SMALL);
  const uint32_t sb = smem_u32(smem_raw), tb = smem_u32(tiles);
  auto bar = [&](int i) -> uint32_t { return sb + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + C::OFF_MISC + 4);
  const Guard guard{status, abort_flag};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = (Nq + 127) / 128;
  int qt = 0, bh = 0;  // longest causal rows first, heads in groups (grouped_tile_head)
  grouped_tile_head(blockIdx.y * gridDim.x + blockIdx.x, T, gridDim.y, head_group, &qt, &bh);
  qt = T - 1 - qt;
  const int off = Nk - Nq;
  int jlo = 0, jhi = 0;  // visible key tiles (every query row sees at least one key)
  key_tile_range(qt, 128, 128, Nq, Nk, CAUSAL, window, &jlo, &jhi);
  const int n_kv = jhi - jlo + 1;
  const size_t row0 = static_cast<size_t>(bh) * Nq;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_QDO), 1);
    for (int k = 0; k < C::KST; ++k) {
      mbar_init(bar(C::B_KFULL + k), 1);
      mbar_init(bar(C::B_KEMPTY + k), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::B_VFULL + b), 1);
      mbar_init(bar(C::B_VEMPTY + b), 1);
      mbar_init(bar(C::B_SFULL + b), 1);
      mbar_init(bar(C::B_SFREE + b), 1);
      // sub-chunk c = key quarters c and 2 + c: half of the element-wise threads
      for (int c = 0; c < 2; ++c) mbar_init(bar(C::B_DSREADY + 2 * b + c), C::NCOMP / 2);
    }
    mbar_init(bar(C::B_DPFULL), 1);
    mbar_init(bar(C::B_DPCONS), C::NCOMP);
    mbar_init(bar(C::B_FINAL), 1);
    mbar_init(bar(C::B_ADONE), 1);
    *abort_flag = (*reinterpret_cast<volatile int*>(status) != 0);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = *abort_flag != 0;

  if (warp == 0 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- producer
    mbar_expect_tx(bar(C::B_QDO), 2 * C::TD);
    for (int c = 0; c < C::NCH; ++c) {
      tma_load_3d(tb + C::T_Q + c * 128 * 128, &tmQ, bar(C::B_QDO), c * 64, qt * 128, bh);
      tma_load_3d(tb + C::T_DO + c * 128 * 128, &tmdO, bar(C::B_QDO), c * 64, qt * 128, bh);
    }
    int lastk = -1, lastv = -1;
    for (int j = 0; j < n_kv; ++j) {
      const int k = j % C::KST, v = j & 1;
      if (!mbar_wait(bar(C::B_KEMPTY + k), ((j / C::KST) & 1) ^ 1, guard, SITE_Q)) break;
      mbar_expect_tx(bar(C::B_KFULL + k), C::TD);
      for (int c = 0; c < C::NCH; ++c)
        tma_load_3d(tb + C::T_K + k * C::TD + c * 128 * 128, &tmK, bar(C::B_KFULL + k), c * 64, (jlo + j) * 128, bh);
      lastk = j;
      if (!mbar_wait(bar(C::B_VEMPTY + v), ((j >> 1) & 1) ^ 1, guard, SITE_Q)) break;
      mbar_expect_tx(bar(C::B_VFULL + v), C::TD);
      for (int c = 0; c < C::NCH; ++c)
        tma_load_3d(tb + C::T_V + v * C::TD + c * 128 * 128, &tmV, bar(C::B_VFULL + v), c * 64, (jlo + j) * 128, bh);
      lastv = j;
    }
    if (*abort_flag) {
      mbar_drain(bar(C::B_QDO), 0);
      for (int j = max(lastk - (C::KST - 1), 0); j <= lastk; ++j)
        mbar_drain(bar(C::B_KFULL + j % C::KST), (j / C::KST) & 1);
      for (int j = max(lastv - 1, 0); j <= lastv; ++j) mbar_drain(bar(C::B_VFULL + (j & 1)), (j >> 1) & 1);
    }
  } else if (warp == 1 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- issuer A: S, dP
    constexpr uint32_t idKK = idesc_bf16(128, 128, false, false);
    const uint32_t qb = tb + C::T_Q, db = tb + C::T_DO;
    bool ok = mbar_wait(bar(C::B_QDO), 0, guard, SITE_Q);
    for (int j = 0; ok && j < n_kv; ++j) {
      const int s = j & 1, k = j % C::KST;
      const uint32_t kb = tb + C::T_K + k * C::TD, vb = tb + C::T_V + s * C::TD;
      if (!(ok = mbar_wait(bar(C::B_KFULL + k), (j / C::KST) & 1, guard, SITE_Q))) break;
      // S buffer s last held dS_{j-2}: dQ_{j-2} must have read it
      if (j >= 2 && !(ok = mbar_wait(bar(C::B_SFREE + s), ((j >> 1) & 1) ^ 1, guard, SITE_Q))) break;
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_ss(tmem + C::TM_S + 128 * s, sdesc_kmajor<128, 128>(qb, ks), sdesc_kmajor<128, 128>(kb, ks), idKK, ks > 0);
      mma_commit(bar(C::B_SFULL + s));
      // the dP columns are free once every element-wise thread has read dP_{j-1}
      if (j > 0 && !(ok = mbar_wait(bar(C::B_DPCONS), (j - 1) & 1, guard, SITE_Q))) break;
      if (!(ok = mbar_wait(bar(C::B_VFULL + s), (j >> 1) & 1, guard, SITE_Q))) break;
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_ss(tmem + C::TM_DP, sdesc_kmajor<128, 128>(db, ks), sdesc_kmajor<128, 128>(vb, ks), idKK, ks > 0);
      mma_commit(bar(C::B_DPFULL));
      mma_commit(bar(C::B_VEMPTY + s));
    }
    mma_commit(bar(C::B_ADONE));
  } else if (warp == 2 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- issuer B: dQ
    constexpr uint32_t idTN = idesc_bf16(128, D, false, true);  // dS (tensor memory) x K (N-major)
    bool ok = true;
    for (int j = 0; ok && j < n_kv; ++j) {
      const int s = j & 1, k = j % C::KST;
      const uint32_t kb = tb + C::T_K + k * C::TD;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (!(ok = mbar_wait(bar(C::B_DSREADY + 2 * s + c), (j >> 1) & 1, guard, SITE_Q))) break;
        tc_fence_after();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ks = 4 * (u >> 1) + 2 * c + (u & 1);  // key block ks: quarter ks/2, dS at 32 (ks/2) + 8 (ks%2)
          mma_ts(tmem + C::TM_DQ, tmem + C::TM_S + 128 * s + 32 * (ks >> 1) + 8 * (ks & 1),
                 sdesc_mnmajor<128, 128>(kb, ks), idTN, (j > 0 || ks > 0));
        }
      }
      if (!ok) break;
      mma_commit(bar(C::B_SFREE + s));
      mma_commit(bar(C::B_KEMPTY + k));  // S_j completed before dS_j existed
    }
    mma_commit(bar(C::B_FINAL));
  } else if (warp >= 4 && !skip) {
    // ---------------------------------------------------------------- element-wise warps
    // warp w: tensor-memory lane quarter w % 4 (32 query rows), key quarter (w - 4) / 4
    // (32 keys); the bf16 dS of a key quarter goes over its own 32 S columns
    const int qw = warp & 3, kq = (warp - 4) >> 2, c = kq & 1, row = qw * 32 + lane, q = qt * 128 + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    const float nl = q < Nq ? -Lg[row0 + q] * kLog2e : -INFINITY;  // rows past Nq: P = 0
    const float dq = q < Nq ? Dg[row0 + q] : 0.f;
    const int p = q + off;  // this row's position
    const uint64_t cc = f2pack(c_log2, c_log2), nl2 = f2pack(nl, nl), nd2 = f2pack(-dq, -dq);
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int s = j & 1;
      if (!(ok = mbar_wait_warp(bar(C::B_SFULL + s), (j >> 1) & 1, guard, SITE_Q))) break;
      tc_fence_after();
      const int k0 = (jlo + j) * 128 + 32 * kq;  // first key of this quarter
      const bool masked = (CAUSAL && k0 + 31 > qt * 128 + off) || (window > 0 && k0 <= qt * 128 + 127 + off - window) ||
                          (k0 + 32 > Nk);
      // keys of this quarter (0..31) this row sees: position p, keys below Nk
      const int khi = min(CAUSAL ? p - k0 : 31, Nk - 1 - k0);
      const int klo = window > 0 ? p - window + 1 - k0 : 0;
      const uint32_t sc = tl + C::TM_S + 128 * s + 32 * kq;
      uint32_t pk[16];
      {
        uint32_t r[32];
        tmem_ld32(sc, r);
        tmem_ld_wait<32>(r);
        auto body = [&](auto mask_tag) {
          constexpr bool MASK = decltype(mask_tag)::value;
#pragma unroll
          for (int x = 0; x < 32; x += 2) {
            float t0, t1;
            f2unpack(ffma2(f2pack(__uint_as_float(r[x]), __uint_as_float(r[x + 1])), cc, nl2), t0, t1);
            float p0 = ex2(t0), p1 = ex2(t1);
            if (MASK) {  // visible iff klo <= x <= khi
              if (x < klo || x > khi) p0 = 0.f;
              if (x + 1 < klo || x + 1 > khi) p1 = 0.f;
            }
            pk[x >> 1] = pack_bf16x2(p0, p1);
          }
        };
        if (masked) body(std::true_type{}); else body(std::false_type{});
      }
      if (!(ok = mbar_wait_warp(bar(C::B_DPFULL), j & 1, guard, SITE_Q))) break;
      tc_fence_after();
      uint32_t r[32];
      tmem_ld32(tl + C::TM_DP + 32 * kq, r);
      tmem_ld_wait<32>(r);
      tc_fence_before();
      mbar_arrive(bar(C::B_DPCONS));
      uint32_t dk[16];
#pragma unroll
      for (int x = 0; x < 32; x += 2) {
        const uint32_t w = pk[x >> 1];
        float d0, d1;
        f2unpack(fmul2(f2pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)),
                       fadd2(f2pack(__uint_as_float(r[x]), __uint_as_float(r[x + 1])), nd2)),
                 d0, d1);
        dk[x >> 1] = pack_bf16x2(d0, d1);
      }
      tmem_st16(sc, dk);  // over this quarter's own S columns, already read
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::B_DSREADY + 2 * s + c));
    }
    if (ok) ok = mbar_wait_warp(bar(C::B_FINAL), 0, guard, SITE_Q);
    if (ok) {
      tc_fence_after();
      uint32_t r[32];
      if constexpr (D == 128) tmem_ld32(tl + C::TM_DQ + 32 * kq, r);
      else tmem_ld16(tl + C::TM_DQ + 16 * kq, r);
      tmem_ld_wait<32>(r);
      uint32_t pk[D / 8];
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
        pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * scale, __uint_as_float(r[2 * i + 1]) * scale);
      const int w0 = qt * 128 + qw * 32;  // the warp's first query row
      warp_store_rows<D / 32, 0>(pk, reinterpret_cast<uint8_t*>(dQ + (row0 + w0) * D + (D / 4) * kq), D * 2, Nq - w0,
                                 lane);
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
    tmem_dealloc(tmem, 512);
  }
}

// Side streams for the query-tile kernel, created on first use per device and kept
// for the process (round robin over a few, so calls on different caller streams
// rarely share one); each with its own fork and join events.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kSideStreams = 4, kMaxSideDevices = 64;
SideStream g_side[kMaxSideDevices][kSideStreams];
int g_side_next[kMaxSideDevices] = {0};
std::mutex g_side_mu;  // held for a whole fork/join enqueue: the events are shared

fa_status side_stream(SideStream** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxSideDevices) return FA_ERR_CUDA;
  SideStream& ss = g_side[dev][g_side_next[dev]];
  g_side_next[dev] = (g_side_next[dev] + 1) % kSideStreams;
  if (ss.s == nullptr && cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess) return FA_ERR_CUDA;
  if (ss.fork == nullptr && cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess)
    return FA_ERR_CUDA;
  if (ss.join == nullptr && cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess)
    return FA_ERR_CUDA;
  *out = &ss;
  return FA_OK;
}

template <int D, bool CAUSAL>
fa_status launch_t(const BwdLaunch& a, void* dQ) {
  CUtensorMap mQ, mK, mV, mdO;
  if (!encode_bf16_3d(&mQ, a.Q, D, a.Nq, a.BH, 64, 128) || !encode_bf16_3d(&mdO, a.dO, D, a.Nq, a.BH, 64, 128) ||
      !encode_bf16_3d(&mK, a.K, D, a.Nk, a.BH, 64, 128) || !encode_bf16_3d(&mV, a.V, D, a.Nk, a.BH, 64, 128))
    return FA_ERR_CUDA;
  static_assert(KVC<D>::SMEM <= SMEM_MAX && QC<D>::SMEM <= SMEM_MAX, "shared memory budget");
  auto kkv = bwd_kv_kernel<D, CAUSAL>;
  auto kq = bwd_q_kernel<D, CAUSAL>;
  // Each CTA takes all 512 tensor-memory columns, so no two CTAs may share an SM
  // (a second allocation would wait for the first CTA to exit).  Asking for more
  // than half of the SM's shared memory guarantees it whatever the register counts.
  constexpr int kExclusive = 120 * 1024;
  const int smem_kv = KVC<D>::SMEM > kExclusive ? KVC<D>::SMEM : kExclusive;
  const int smem_q = QC<D>::SMEM > kExclusive ? QC<D>::SMEM : kExclusive;
  if (cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_kv) != cudaSuccess ||
      cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_q) != cudaSuccess)
    return FA_ERR_CUDA;
  const int Tq = (a.Nq + 127) / 128, Tk = (a.Nk + 127) / 128;
  const float c_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  // The two kernels are independent (both read Q, K, V, dO, L, D; they write different
  // outputs), so the query-tile kernel runs on a side stream forked from the caller's:
  // its CTAs take the SMs that the key-tile kernel's last, partial wave leaves idle
  // (a CTA of either kernel fills an SM's registers, so they never share one).
  std::lock_guard<std::mutex> lk(g_side_mu);
  SideStream* ss = nullptr;
  const fa_status st = side_stream(&ss);
  if (st != FA_OK) return st;
  if (cudaEventRecord(ss->fork, a.stream) != cudaSuccess || cudaStreamWaitEvent(ss->s, ss->fork, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  kkv<<<dim3(Tk, a.BH), KVC<D>::NTHREADS, smem_kv, a.stream>>>(
      mQ, mK, mV, mdO, a.L, a.D, static_cast<__nv_bfloat16*>(a.dK), static_cast<__nv_bfloat16*>(a.dV), a.Nq, a.Nk,
      a.window, c_log2, a.scale, a.status, a.counter, head_group(a.BH, a.Nq, a.Nk, D));
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  kq<<<dim3(Tq, a.BH), QC<D>::NTHREADS, smem_q, ss->s>>>(mQ, mK, mV, mdO, a.L, a.D,
                                                        static_cast<__nv_bfloat16*>(dQ), a.Nq, a.Nk, a.window,
                                                        c_log2, a.scale, a.status,
                                                        head_group(a.BH, a.Nq, a.Nk, D));
  // the caller's stream continues only once both kernels are done
  if (cudaGetLastError() != cudaSuccess || cudaEventRecord(ss->join, ss->s) != cudaSuccess ||
      cudaStreamWaitEvent(a.stream, ss->join, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace

fa_status launch_bwd_two_kernel(const BwdLaunch& a, void* dQ) {
  switch (a.d) {
    case 64: return a.causal ? launch_t<64, true>(a, dQ) : launch_t<64, false>(a, dQ);
    case 128: return a.causal ? launch_t<128, true>(a, dQ) : launch_t<128, false>(a, dQ);
    default: return FA_ERR_UNSUPPORTED;
  }
}

}  // namespace fa
