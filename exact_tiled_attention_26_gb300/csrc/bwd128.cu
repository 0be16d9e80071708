// Backward pass, head size 128: the main kernel.
//
// Same mathematics as bwd.cu ("CS336 Assignment 2 notes" §1.4, Equations 13-19,
// key/value tiles outer): one CTA owns 128 keys of one (batch, head); K_j and
// V_j stay in shared memory while the CTA walks the visible 128-row query tiles
// i.  With keys on the 128 tensor-memory lanes, per step:
//
//   S^T  = K Q_i^T                       (UMMA, M=N=128)          Eq 13
//   P^T  = 2^(S^T c - L log2 e) -> bf16, kept in tensor memory     Eq 14
//   dP^T = V dO_i^T                      (UMMA)                   Eq 16
//   dV  += P^T dO_i                      (UMMA, A = P^T in TMEM)   Eq 15
//   dS^T = P^T (dP^T - D) -> bf16, in tensor memory and in shared memory (Eq 17)
//   dK  += dS^T Q_i                      (UMMA, A = dS^T in TMEM)  Eq 19
//   dQ_i^T = K^T dS^T                    (UMMA, over the dP^T columns)
//   dQ_i += dQ_i^T, added from registers into the fp32 workspace with
//           coalesced reductions in L2                             Eq 18
// The softmax scale of Eq 18-19 is applied to dK at the end and to dQ by the
// convert pass.
//
// Every UMMA is M = 128, N = 128 (narrower UMMAs do not reach the tensor pipe's
// rate).  Tensor memory (512 columns): dK 128 | dV 128 | two 128-column regions
// that take turns.  Step i keeps S^T in region i % 2; there query half h (64
// queries) overwrites its own S^T with its bf16 P^T (columns 64h .. 64h+31) and
// dS^T (64h+32 .. 64h+63), and once dV and dK have read those, dQ_i^T is formed
// over the whole region.  dP^T of step i goes to region (i + 1) % 2, which held
// dQ^T of step i-1.  The element-wise warps take all of dP^T into registers before
// forming dS, so S^T of step i+1 is formed in that region while dS of step i is
// computed and dK of step i accumulates.
//
// Warps: 0 TMA producer (its 32 lanes also stage L*log2 e and D of each query
// tile in shared memory, two tiles ahead), 1 and 2 UMMA issuers (one thread
// each: S^T and dP^T; dV, dK and dQ^T -- two issuing threads keep the tensor pipe
// fed while either one waits on a barrier), 4..11
// element-wise (warp w: tensor-memory lane quarter w % 4, query half (w - 4) / 4;
// one key row per thread), 12..15 dQ drain (warp w: lane quarter w % 4, i.e. 32
// values of d; each takes all 128 columns of dQ^T out of tensor memory at once,
// frees the columns, then issues the reductions while the next step runs).  L2
// absorbs fp32 reductions at about 20 bytes per clock per SM, so the 64 KiB of
// dQ per step are drained off the element-wise warps' path.  Registers move from
// the producer/UMMA warpgroup to the others with setmaxnreg: 72 + 3 x 144 <= 4 x 128.
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct B128 {
  static constexpr int D = 128, BN = 128, BM = 128;
  static constexpr int NTHREADS = 512;
  static constexpr int NCOMP = 256;             // element-wise threads
  static constexpr int NDQ = 128;               // dQ drain threads
  static constexpr int TILE = 128 * 128 * 2;    // one 128 x 128 bf16 tile (two 64-column chunks)
  // small region at the start of dynamic shared memory
  enum : int {
    B_KV = 0, B_QFULL = 1, B_QEMPTY = 3, B_SFULL = 5, B_DPFULL = 6,
    B_PREADY = 7,  // [step parity][sub-chunk]: the element-wise warps may be a step ahead of issuer B
    B_DSREADY = 11, B_DKDONE = 13, B_DQFULL = 14, B_DQCONS = 15, B_DPCONS = 16, B_FINAL = 17, B_ADONE = 18,
    B_DSSMEM = 19,  // dS^T of the step is in shared memory (for dQ^T)
    NBAR = 20
  };
  static constexpr int OFF_BAR = 0;
  static constexpr int OFF_MISC = NBAR * 8;     // tensor-memory base, abort flag
  static constexpr int OFF_LD = 256;            // 2 stages x (-L*log2 e [128], D [128])
  static constexpr int LD_BYTES = 2 * BM * 4;
  static constexpr int SMALL = OFF_LD + 2 * LD_BYTES;
  // 1 KiB-aligned tiles after it
  static constexpr int T_K = 0, T_V = TILE, T_Q = 2 * TILE, T_DO = 3 * TILE;  // Q, dO: stage s adds s * 2 * TILE
  static constexpr int T_DS = 6 * TILE;         // dS^T [128 keys][128 queries]
  static constexpr int TILES = 7 * TILE;        // 224 KiB
  static constexpr int SMEM = 232448;           // the per-block maximum
  // Two 128-column regions take turns: step i keeps S^T, then P^T | dS^T, then dQ^T
  // in region i % 2, and dP^T in region (i + 1) % 2.
  static constexpr int TM_DK = 0, TM_DV = 128, TM_R = 256, TM_COLS = 512;
  // with a 1 KiB-aligned base the tiles start at 3 KiB and end exactly at the limit
  static_assert(SMALL <= 3072 && 3072 + TILES <= SMEM, "shared memory budget");
};

enum : int { SITE_PRODUCER = 0x211, SITE_MMA = 0x212, SITE_COMPUTE = 0x213, SITE_LAYOUT = 0x215 };

template <bool CAUSAL>
__global__ void __launch_bounds__(B128::NTHREADS, 1)
    bwd_d128_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const float* __restrict__ Lg, const float* __restrict__ Dg, float* __restrict__ dQacc,
                    __nv_bfloat16* __restrict__ dK, __nv_bfloat16* __restrict__ dV, int Nq, int Nk, int window, float c_log2, float scale,
                    int* status, unsigned long long* tile_counter, int head_group) {
  using C = B128;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = align1024(smem_raw + C::SMALL);
  if (tiles + C::TILES > smem_raw + C::SMEM) {
    // the dynamic shared memory base is too badly aligned for this layout: report, do nothing
    if (threadIdx.x == 0) atomicCAS(status, 0, SITE_LAYOUT);
    return;
  }
  const uint32_t sb = smem_u32(smem_raw);
  const uint32_t tb = smem_u32(tiles);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + C::OFF_MISC + 4);
  const Guard guard{status, abort_flag};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // key tile (with the causal mask the longest loops come first) and head, heads in
  // groups (grouped_tile_head)
  int kt = 0, bh = 0;
  grouped_tile_head(blockIdx.y * gridDim.x + blockIdx.x, gridDim.x, gridDim.y, head_group, &kt, &bh);
  const int off = Nk - Nq;  // position of query row i is i + off
  // visible query tiles i0 .. i0 + n_it - 1 (none: this CTA writes zero dK, dV)
  int i0 = 0, ilast = 0;
  query_tile_range(kt, C::BM, C::BN, Nq, Nk, CAUSAL, window, &i0, &ilast);
  const int n_it = ilast >= i0 ? ilast - i0 + 1 : 0;
  const size_t row0 = static_cast<size_t>(bh) * Nq;   // Q, dO, L, D, dQ rows
  const size_t krow0 = static_cast<size_t>(bh) * Nk;  // K, V, dK, dV rows

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_KV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_QFULL + s), 1 + 32);  // TMA bytes + the producer's 32 lanes (L, D)
      mbar_init(bar(C::B_QEMPTY + s), 1);
    }
    mbar_init(bar(C::B_SFULL), 1);
    mbar_init(bar(C::B_DPFULL), 1);
    for (int c = 0; c < 2; ++c) {  // the two 32-query sub-chunks of each thread's 64 queries
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
  // warpgroup 0 (producer and UMMA issuers) gives registers to the others
  regs_dec<72>();
  if (warp == 0 && !skip) {
    // ---------------------------------------------------------------- producer (whole warp)
    if (lane == 0) {
      mbar_expect_tx(bar(C::B_KV), 2 * C::TILE);
      for (int c = 0; c < 2; ++c) {
        tma_load_3d(tb + C::T_K + c * 128 * 128, &tmK, bar(C::B_KV), c * 64, kt * C::BN, bh);
        tma_load_3d(tb + C::T_V + c * 128 * 128, &tmV, bar(C::B_KV), c * 64, kt * C::BN, bh);
      }
    }
    int last = -1;
    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1;
      const int q0 = (i0 + it) * C::BM;
      // -L log2 e and D of this query tile, read before waiting for the stage; rows
      // past Nq get -L log2 e = -inf so that their P is exactly 0
      float lv[4], dv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = q0 + lane + 32 * u;
        lv[u] = q < Nq ? -Lg[row0 + q] * kLog2e : -INFINITY;
        dv[u] = q < Nq ? Dg[row0 + q] : 0.f;
      }
      if (!mbar_wait_warp(bar(C::B_QEMPTY + s), ((it >> 1) & 1) ^ 1, guard, SITE_PRODUCER)) break;
      if (lane == 0) {
        mbar_expect_tx(bar(C::B_QFULL + s), 2 * C::TILE);
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(tb + C::T_Q + s * 2 * C::TILE + c * 128 * 128, &tmQ, bar(C::B_QFULL + s), c * 64, q0, bh);
          tma_load_3d(tb + C::T_DO + s * 2 * C::TILE + c * 128 * 128, &tmdO, bar(C::B_QFULL + s), c * 64, q0, bh);
        }
      }
      float* Ls = reinterpret_cast<float*>(smem_raw + C::OFF_LD + s * C::LD_BYTES);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        Ls[lane + 32 * u] = lv[u];
        Ls[C::BM + lane + 32 * u] = dv[u];
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
    // ---------------------------------------------------------------- UMMA issuer A: S^T, dP^T
    constexpr uint32_t idKK = idesc_bf16(128, 128, false, false);  // S^T, dP^T: K-major x K-major
    const uint32_t kb = tb + C::T_K, vb = tb + C::T_V;
    bool ok = mbar_wait(bar(C::B_KV), 0, guard, SITE_MMA);
    for (int it = 0; ok && it < n_it; ++it) {
      const int s = it & 1;
      const uint32_t qb = tb + C::T_Q + s * 2 * C::TILE, db = tb + C::T_DO + s * 2 * C::TILE;
      const uint32_t rs = tmem + C::TM_R + 128 * s, rd = tmem + C::TM_R + 128 * (s ^ 1);
      if (!(ok = mbar_wait(bar(C::B_QFULL + s), (it >> 1) & 1, guard, SITE_MMA))) break;
      // region s held dP^T of the previous step: every element-wise thread has read it
      if (it > 0 && !(ok = mbar_wait(bar(C::B_DPCONS), (it - 1) & 1, guard, SITE_MMA))) break;
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_ss(rs, sdesc_kmajor<128, 128>(kb, ks), sdesc_kmajor<128, 128>(qb, ks), idKK, ks > 0);
      mma_commit(bar(C::B_SFULL));
      // region s^1 ended the previous step holding its dQ^T: the drain warps have read it
      if (it > 0 && !(ok = mbar_wait(bar(C::B_DQCONS), (it - 1) & 1, guard, SITE_MMA))) break;
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_ss(rd, sdesc_kmajor<128, 128>(vb, ks), sdesc_kmajor<128, 128>(db, ks), idKK, ks > 0);
      mma_commit(bar(C::B_DPFULL));
    }
    mma_commit(bar(C::B_ADONE));  // drain point for teardown
    if (ok && tile_counter != nullptr) atomicAdd(tile_counter, static_cast<unsigned long long>(n_it));
  } else if (warp == 2 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- UMMA issuer B: dV, dK, dQ^T
    // S^T and dP^T of a step are complete before the element-wise warps can signal
    // P and dS ready, so this thread's commits cover every reader of Q_i and dO_i.
    constexpr uint32_t idTN = idesc_bf16(128, 128, false, true);  // dV, dK: A in TMEM x N-major B
    constexpr uint32_t idMN = idesc_bf16(128, 128, true, true);   // dQ^T: K^T (M-major) x dS^T (N-major)
    const uint32_t kb = tb + C::T_K, dsb = tb + C::T_DS;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1;
      const uint32_t qb = tb + C::T_Q + s * 2 * C::TILE, db = tb + C::T_DO + s * 2 * C::TILE;
      const uint32_t rs = tmem + C::TM_R + 128 * s;
      // dV += P^T dO_i.  Query block ks (16 queries) is in half ks/4, sub-chunk (ks%4)/2;
      // its bf16 P^T sits in columns 64 (ks/4) + 8 (ks%4).  Sub-chunk 0 (blocks 0,1,4,5)
      // is ready before sub-chunk 1 (blocks 2,3,6,7).
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (!(ok = mbar_wait(bar(C::B_PREADY + 2 * s + c), (it >> 1) & 1, guard, SITE_MMA))) break;
        tc_fence_after();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ks = 4 * (u >> 1) + 2 * c + (u & 1);
          mma_ts(tmem + C::TM_DV, rs + 64 * (ks >> 2) + (ks & 3) * 8, sdesc_mnmajor<128, 128>(db, ks), idTN,
                 (it > 0 || ks > 0));
        }
      }
      if (!ok) break;
      // dK += dS^T Q_i (dS^T of block ks in columns 64 (ks/4) + 32 + 8 (ks%4))
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (!(ok = mbar_wait(bar(C::B_DSREADY + c), it & 1, guard, SITE_MMA))) break;
        tc_fence_after();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ks = 4 * (u >> 1) + 2 * c + (u & 1);
          mma_ts(tmem + C::TM_DK, rs + 64 * (ks >> 2) + 32 + (ks & 3) * 8, sdesc_mnmajor<128, 128>(qb, ks), idTN,
                 (it > 0 || ks > 0));
        }
      }
      if (!ok) break;
      mma_commit(bar(C::B_DKDONE));
      mma_commit(bar(C::B_QEMPTY + s));  // Q_i, dO_i have no later reader
      // dQ_i^T = K^T dS^T (both from shared memory) over region s, once dV and dK have
      // read its P^T and dS^T
      if (!(ok = mbar_wait(bar(C::B_DKDONE), it & 1, guard, SITE_MMA))) break;
      if (!(ok = mbar_wait(bar(C::B_DSSMEM), it & 1, guard, SITE_MMA))) break;
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_ss(rs, sdesc_mnmajor<128, 128>(kb, ks), sdesc_mnmajor<128, 128>(dsb, ks), idMN, ks > 0);
      mma_commit(bar(C::B_DQFULL));
    }
    mma_commit(bar(C::B_FINAL));
  }
  } else if (warp >= 12) {
    regs_inc<144>();
    if (!skip) {
    // ---------------------------------------------------------------- dQ drain
    // dQ_j^T (lane = d, columns = queries) -> dQ workspace rows; each warp access
    // covers 32 consecutive d of one query row (128 bytes).
    const int qw = warp & 3;
    const int dd = qw * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    for (int j = 0; j < n_it; ++j) {
      if (!mbar_wait_warp(bar(C::B_DQFULL), j & 1, guard, SITE_COMPUTE)) break;
      tc_fence_after();
      uint32_t r[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tl + C::TM_R + 128 * (j & 1) + 32 * c, r + 32 * c);
      tmem_ld_wait<128>(r);
      tc_fence_before();
      mbar_arrive(bar(C::B_DQCONS));
      const int q0 = (i0 + j) * C::BM;
      float* dst = dQacc + (row0 + q0) * C::D + dd;
      const int nq = min(C::BM, Nq - q0);
      if (nq >= C::BM) {
#pragma unroll
        for (int x = 0; x < C::BM; ++x) atomicAdd(dst + static_cast<size_t>(x) * C::D, __uint_as_float(r[x]));
      } else {
#pragma unroll
        for (int x = 0; x < C::BM; ++x)
          if (x < nq) atomicAdd(dst + static_cast<size_t>(x) * C::D, __uint_as_float(r[x]));
      }
    }
    }
  } else {
    regs_inc<144>();
    if (!skip) {
    // ---------------------------------------------------------------- element-wise warps
    const int qw = warp & 3;        // tensor-memory lane quarter
    const int h = (warp - 4) >> 2;  // query half (64 queries) of each tile
    const int kr = qw * 32 + lane;  // key row (tensor-memory lane); also the d index of dQ^T
    const int key = kt * C::BN + kr;
    const uint32_t tl = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    bool ok = true;

    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1;
      if (!(ok = mbar_wait_warp(bar(C::B_QFULL + s), (it >> 1) & 1, guard, SITE_COMPUTE))) break;
      if (!(ok = mbar_wait_warp(bar(C::B_SFULL), it & 1, guard, SITE_COMPUTE))) break;
      tc_fence_after();
      const uint32_t rs = tl + C::TM_R + 128 * s, rd = tl + C::TM_R + 128 * (s ^ 1);
      const int qh = (i0 + it) * C::BM + 64 * h;  // first query of this half
      const float4* L4 = reinterpret_cast<const float4*>(smem_raw + C::OFF_LD + s * C::LD_BYTES) + 16 * h;
      const float4* D4 = L4 + C::BM / 4;
      const bool masked = (CAUSAL && kt * C::BN + C::BN - 1 > qh + off) ||
                          (window > 0 && kt * C::BN <= qh + 63 + off - window) || (kt * C::BN + C::BN > Nk);
      // queries of this half (0..63) that see this thread's key: key <= q + off (causal),
      // key > q + off - window (window), and none at all past Nk
      const int qlo = CAUSAL ? key - off - qh : 0;
      const int qhi = key >= Nk ? -1 : (window > 0 ? key - off + window - 1 - qh : 63);
      const uint64_t cc = f2pack(c_log2, c_log2);
      // ---- P^T = 2^(S^T c - L log2 e), two sub-chunks of 32 queries, each released
      // to the dV product as soon as it is in tensor memory
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
              const int x = 4 * v + y;  // within the sub-chunk
              const uint64_t t = ffma2(f2pack(__uint_as_float(r[x]), __uint_as_float(r[x + 1])), cc,
                                       y == 0 ? f2pack(l.x, l.y) : f2pack(l.z, l.w));
              float t0, t1;
              f2unpack(t, t0, t1);
              p[y] = ex2(t0);
              p[y + 1] = ex2(t1);
              if (MASK) {
                const int xs = 32 * c + x;  // query of the half: visible iff qlo <= xs <= qhi
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
      // ---- dS^T = P^T (dP^T - D), from the same bf16 P that enters dV; two sub-chunks
      if (!(ok = mbar_wait_warp(bar(C::B_DPFULL), it & 1, guard, SITE_COMPUTE))) break;
      tc_fence_after();
      uint8_t* row = tiles + C::T_DS + h * (128 * 128) + kr * 128;
      // all of this thread's dP^T out of tensor memory first, so that S^T of the next
      // step can be formed in its region while dS is computed
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
            const int x = 4 * v + y;
            const uint32_t w = pk[16 * c + (x >> 1)];
            const uint64_t pp = f2pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
            const uint64_t t = fadd2(f2pack(__uint_as_float(r[x]), __uint_as_float(r[x + 1])),
                                     y == 0 ? f2pack(-dd.x, -dd.y) : f2pack(-dd.z, -dd.w));
            float d0, d1;
            f2unpack(fmul2(pp, t), d0, d1);
            dk[x >> 1] = pack_bf16x2(d0, d1);
          }
        }
        tmem_st16(rs + 64 * h + 32 + 16 * c, dk);
        // dS^T row kr, queries 64h + 32c .. +31: four 16-byte units of the swizzled row
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4*>(row + (((4 * c + u) ^ (kr & 7)) << 4)) =
              make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_DSREADY + c));  // dK reads dS^T from tensor memory
      }
      // dQ^T reads dS^T from shared memory: one proxy fence for both sub-chunks
      fence_proxy_async_smem();
      mbar_arrive(bar(C::B_DSSMEM));

    }
    // dK (times scale) and dV: this warp's lane quarter, d columns 64h .. 64h+63
    if (ok) ok = mbar_wait_warp(bar(C::B_FINAL), 0, guard, SITE_COMPUTE);
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const float f = t == 0 ? scale : 1.f;
        __nv_bfloat16* dst = (t == 0 ? dK : dV) + (krow0 + key) * C::D + 64 * h;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          tmem_ld32(tl + (t == 0 ? C::TM_DK : C::TM_DV) + 64 * h + 32 * c, r);
          tmem_ld_wait<32>(r);
          if (n_it == 0) {  // no query sees these keys: the accumulators were never written
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          }
          if (key < Nk) {
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

template <bool CAUSAL>
fa_status launch_t(const BwdLaunch& a) {
  using C = B128;
  CUtensorMap mQ, mK, mV, mdO;
  if (!encode_bf16_3d(&mQ, a.Q, C::D, a.Nq, a.BH, 64, C::BM) ||
      !encode_bf16_3d(&mdO, a.dO, C::D, a.Nq, a.BH, 64, C::BM) ||
      !encode_bf16_3d(&mK, a.K, C::D, a.Nk, a.BH, 64, C::BN) || !encode_bf16_3d(&mV, a.V, C::D, a.Nk, a.BH, 64, C::BN))
    return FA_ERR_CUDA;
  auto kern = bwd_d128_kernel<CAUSAL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return FA_ERR_CUDA;
  const dim3 grid((a.Nk + C::BN - 1) / C::BN, a.BH);
  const float c_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  kern<<<grid, C::NTHREADS, C::SMEM, a.stream>>>(mQ, mK, mV, mdO, a.L, a.D, a.dQacc,
                                                 static_cast<__nv_bfloat16*>(a.dK), static_cast<__nv_bfloat16*>(a.dV),
                                                 a.Nq, a.Nk, a.window, c_log2, a.scale, a.status, a.counter,
                                                 head_group(a.BH, a.Nq, a.Nk, C::D));
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status launch_bwd_d128(const BwdLaunch& a) { return a.causal ? launch_t<true>(a) : launch_t<false>(a); }

}  // namespace fa
