// Backward pass, head sizes 64 and 128: one CTA per key tile.
//
// "CS336 Assignment 2 notes" §1.4, Equations 13-19, key/value tiles outer: one CTA
// owns 128 keys of one (batch, head); K_j and V_j stay in shared memory while the CTA
// walks the visible 128-row query tiles i.  The per-step work of every role (the five
// UMMAs, the element-wise P^T and dS^T, the dQ drain) is in bwd_steps.cuh, shared with
// the persistent kernel (bwd_persist.cu); this file walks a single unit of work per
// CTA.  The softmax scale of Eq 18-19 is applied to dK at the end and to dQ by the
// convert pass.
//
// Every UMMA is M = 128, N = 128 (narrower UMMAs do not reach the tensor pipe's rate).
//
// Warps: 0 TMA producer (its 32 lanes also stage L*log2 e and D of each query tile in
// shared memory, two tiles ahead), 1 and 2 UMMA issuers (one thread each: S^T and
// dP^T; dV, dK and dQ^T -- two issuing threads keep the tensor pipe fed while either
// one waits on a barrier), 4..11 element-wise (warp w: tensor-memory lane quarter
// w % 4, query half (w - 4) / 4; one key row per thread), 12..15 dQ drain (warp w:
// lane quarter w % 4, i.e. 32 values of d; each takes its columns of dQ^T out of
// tensor memory at once, frees them, then issues the reductions while the next step
// runs).  L2 absorbs fp32 reductions at about 20 bytes per clock per SM, so the
// 64 KiB of dQ per step are drained off the element-wise warps' path.  Registers move
// from the producer/UMMA warpgroup to the others with setmaxnreg: 72 + 3 x 144 <= 4 x 128.
#include "bwd_steps.cuh"
#include "internal.h"

namespace fa {
namespace {

using namespace bsteps;

// Barriers of this kernel beyond the per-step ones (bwd_steps.cuh).
enum : int { B_KV = 0, B_FINAL = 17, B_ADONE = 18, NBAR = 20 };
constexpr int OFF_MISC = NBAR * 8;  // tensor-memory base, abort flag
constexpr int NTHREADS = 512;
static_assert(OFF_MISC + 8 <= OFF_LD, "small region");

enum : int { SITE_PRODUCER = 0x211, SITE_MMA = 0x212, SITE_COMPUTE = 0x213, SITE_LAYOUT = 0x215 };

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(NTHREADS, 1)
    bwd_tile_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const float* __restrict__ Lg, const float* __restrict__ Dg, float* __restrict__ dQacc,
                    __nv_bfloat16* __restrict__ dK, __nv_bfloat16* __restrict__ dV, int Nq, int Nk, int window,
                    float c_log2, float scale, int* status, unsigned long long* tile_counter, int head_group) {
  using LY = Lay<D, 1>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = align1024(smem_raw + SMALL);
  if (tiles + LY::TILES > smem_raw + LY::SMEM) {
    // the dynamic shared memory base is too badly aligned for this layout: report, do nothing
    if (threadIdx.x == 0) atomicCAS(status, 0, SITE_LAYOUT);
    return;
  }
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + OFF_MISC + 4);
  Ctx x{smem_u32(smem_raw), smem_u32(tiles), smem_raw, tiles, 0u, Guard{status, abort_flag}};
  auto bar = [&](int i) -> uint32_t { return x.bar(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // key tile (with the causal mask the longest loops come first) and head, heads in
  // groups (grouped_tile_head)
  int kt = 0, bh = 0;
  grouped_tile_head(blockIdx.y * gridDim.x + blockIdx.x, gridDim.x, gridDim.y, head_group, &kt, &bh);
  const int off = Nk - Nq;  // position of query row i is i + off
  // visible query tiles i0 .. i0 + n_it - 1 (none: this CTA writes zero dK, dV)
  int i0 = 0, ilast = 0;
  query_tile_range(kt, BM, BN, Nq, Nk, CAUSAL, window, &i0, &ilast);
  const int n_it = ilast >= i0 ? ilast - i0 + 1 : 0;
  const size_t row0 = static_cast<size_t>(bh) * Nq;   // Q, dO, L, D, dQ rows
  const size_t krow0 = static_cast<size_t>(bh) * Nk;  // K, V, dK, dV rows

  if (threadIdx.x == 0) {
    mbar_init(bar(B_KV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_QFULL + s), 1 + 32);  // TMA bytes + the producer's 32 lanes (L, D)
      mbar_init(bar(B_QEMPTY + s), 1);
    }
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_DPFULL), 1);
    for (int c = 0; c < 2; ++c) {  // the two 32-query sub-chunks of each thread's 64 queries
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

  if (warp < 4) {
  // warpgroup 0 (producer and UMMA issuers) gives registers to the others
  regs_dec<72>();
  if (warp == 0 && !skip) {
    // ---------------------------------------------------------------- producer (whole warp)
    if (lane == 0) {
      mbar_expect_tx(bar(B_KV), LY::KVB);
      for (int c = 0; c < 2; ++c)  // at d = 64 the second K chunk is a copy of the first
        tma_load_3d(LY::k(x.tb, 0) + c * CHUNK, &tmK, bar(B_KV), D == 128 ? c * 64 : 0, kt * BN, bh);
      for (int c = 0; c < LY::TQ / CHUNK; ++c)
        tma_load_3d(LY::v(x.tb, 0) + c * CHUNK, &tmV, bar(B_KV), c * 64, kt * BN, bh);
    }
    int last = -1;
    for (int it = 0; it < n_it; ++it) {
      if (!produce_step<LY>(x, &tmQ, &tmdO, Lg, Dg, row0, Nq, (i0 + it) * BM, bh, it, lane, SITE_PRODUCER)) break;
      last = it;
    }
    if (lane == 0 && *abort_flag) {
      mbar_drain(bar(B_KV), 0);
      for (int it = (last > 0 ? last - 1 : 0); it <= last; ++it) mbar_drain(bar(B_QFULL + (it & 1)), (it >> 1) & 1);
    }
  } else if (warp == 1 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- UMMA issuer A: S^T, dP^T
    bool ok = mbar_wait(bar(B_KV), 0, x.guard, SITE_MMA);
    for (int it = 0; ok && it < n_it; ++it) ok = issue_s_dp<LY>(x, it, 0, SITE_MMA);
    mma_commit(bar(B_ADONE));  // drain point for teardown
    if (ok && tile_counter != nullptr) atomicAdd(tile_counter, static_cast<unsigned long long>(n_it));
  } else if (warp == 2 && lane == 0 && !skip) {
    // ---------------------------------------------------------------- UMMA issuer B: dV, dK, dQ^T
    for (int it = 0; it < n_it; ++it)
      if (!issue_dv_dk_dq<LY>(x, it, 0, it == 0, SITE_MMA)) break;
    mma_commit(bar(B_FINAL));
  }
  } else if (warp >= 12) {
    regs_inc<D == 64 ? 136 : 144>();
    if (!skip) {
    // ---------------------------------------------------------------- dQ drain
    pdl_wait();  // the workspace is cleared by the kernel before this one
    const int qw = warp & 3;
    for (int j = 0; j < n_it; ++j) {
      const int q0 = (i0 + j) * BM;
      if (!drain_step<D>(x, j, dQacc + (row0 + q0) * D, min(BM, Nq - q0), qw, lane, SITE_COMPUTE)) break;
    }
    }
  } else {
    regs_inc<D == 64 ? 152 : 144>();  // 72 + 152 x 2 + 136 = 4 x 128 at d = 64
    if (!skip) {
    // ---------------------------------------------------------------- element-wise warps
    const int qw = warp & 3;        // tensor-memory lane quarter
    const int h = (warp - 4) >> 2;  // query half (64 queries) of each tile
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it)
      ok = ew_step<LY, CAUSAL>(x, it, kt, i0 + it, Nk, off, window, c_log2, qw, h, lane, SITE_COMPUTE);
    // dK (times scale) and dV: this warp's lane quarter, d columns (D/2) h .. (D/2) h + D/2 - 1
    if (ok) ok = mbar_wait_warp(bar(B_FINAL), 0, x.guard, SITE_COMPUTE);
    if (ok) {
      tc_fence_after();
      uint32_t outp[D / 2];
      ew_load_dk_dv<D>(x, qw, h, scale, n_it == 0, outp);
      const int row0 = kt * BN + qw * 32;
      ew_store_dk_dv<D>(outp, dK, dV, krow0 + row0, Nk - row0, h, lane);
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
}

template <int D, bool CAUSAL>
fa_status launch_t(const BwdLaunch& a) {
  using LY = Lay<D, 1>;
  CUtensorMap mQ, mK, mV, mdO;
  if (!encode_bf16_3d(&mQ, a.Q, D, a.Nq, a.BH, 64, BM) || !encode_bf16_3d(&mdO, a.dO, D, a.Nq, a.BH, 64, BM) ||
      !encode_bf16_3d(&mK, a.K, D, a.Nk, a.BH, 64, BN) || !encode_bf16_3d(&mV, a.V, D, a.Nk, a.BH, 64, BN))
    return FA_ERR_CUDA;
  auto kern = bwd_tile_kernel<D, CAUSAL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM) != cudaSuccess)
    return FA_ERR_CUDA;
  const dim3 grid((a.Nk + BN - 1) / BN, a.BH);
  const float c_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  // Launched so that it may start while the workspace is being cleared: only the dQ
  // drain touches the workspace, and it waits for the clearing kernel's end first;
  // everything else it reads was complete before that kernel started.
  const cudaError_t e = launch_pdl(kern, grid, dim3(NTHREADS), LY::SMEM, a.stream, mQ, mK, mV, mdO, a.L, a.D,
                                   a.dQacc, static_cast<__nv_bfloat16*>(a.dK), static_cast<__nv_bfloat16*>(a.dV),
                                   a.Nq, a.Nk, a.window, c_log2, a.scale, a.status, a.counter,
                                   head_group(a.BH, a.Nq, a.Nk, D));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status launch_bwd_tile(const BwdLaunch& a) {
  if (a.d == 64) return a.causal ? launch_t<64, true>(a) : launch_t<64, false>(a);
  return a.causal ? launch_t<128, true>(a) : launch_t<128, false>(a);
}

}  // namespace fa
