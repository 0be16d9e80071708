// The per-step work of every role of the tensor-core backward at head sizes 64 and 128
// ("CS336 Assignment 2 notes" §1.4, Equations 13-19, key/value tiles outer), shared by
// the kernel with one CTA per key tile (bwd_tile.cu) and the persistent kernel
// (bwd_persist.cu).  Both kernels lay out shared and tensor memory the same way and
// number the per-step barriers the same way (the constants below); they differ only in
// how they walk units of work.
//
// One step processes query tile i against the CTA's key tile j, keys on the 128
// tensor-memory lanes:
//   S^T  = K Q_i^T                       (UMMA, M=N=128)          Eq 13
//   P^T  = 2^(S^T c - L log2 e) -> bf16, kept in tensor memory     Eq 14
//   dP^T = V dO_i^T                      (UMMA)                   Eq 16
//   dV  += P^T dO_i                      (UMMA, A = P^T in TMEM)   Eq 15
//   dS^T = P^T (dP^T - D) -> bf16, in tensor memory and in shared memory (Eq 17)
//   dK  += dS^T Q_i                      (UMMA, A = dS^T in TMEM)  Eq 19
//   dQ_i^T = K^T dS^T                    (UMMA, over the dP^T columns)
//   dQ_i += dQ_i^T, added from registers into the fp32 workspace with
//           coalesced reductions in L2                             Eq 18
// Every UMMA has M = 128 and N = 128 or d.  At d = 64 the dQ^T product keeps M = 128:
// its A operand K^T is read from a K tile stored twice (the second 64-column chunk a
// copy of the first), so tensor-memory lanes 64..127 repeat d = 0..63 -- the
// tensor pipe takes an M = 64 product no faster, and the result keeps the
// M = 128 lane layout.
// Tensor memory (512 columns): dK 128 | dV 128 (d columns of each used) | two
// 128-column regions that take turns.  Step g keeps S^T in region g % 2; there query half h (64 queries) overwrites
// its own S^T with its bf16 P^T (columns 64h .. 64h+31) and dS^T (64h+32 .. 64h+63),
// and once dV and dK have read those, dQ_g^T is formed over the whole region.  dP^T of
// step g goes to region (g + 1) % 2, which held dQ^T of step g-1.
//
// `g` is the CTA's step count: it picks the Q, dO stage, the tensor-memory regions and
// every barrier phase, and runs on across units in the persistent kernel.  `kvb` is the
// K, V buffer of the step's unit (the persistent kernel keeps two at d = 64).
#pragma once

#include <type_traits>

#include "ptx.cuh"

namespace fa {
namespace bsteps {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int BN = 128, BM = 128;
constexpr int NCOMP = 256;  // element-wise threads (warps 4..11)
constexpr int NDQ = 128;    // dQ drain threads (warps 12..15)
constexpr int CHUNK = 128 * 64 * 2;  // 128 rows x 64 bf16 columns (one 128-byte swizzle span)
// Per-step barriers (the kernels add their own from 17 on).
enum : int {
  B_QFULL = 1, B_QEMPTY = 3, B_SFULL = 5, B_DPFULL = 6,
  B_PREADY = 7,  // [step parity][sub-chunk]: the element-wise warps may be a step ahead of issuer B
  B_DSREADY = 11, B_DKDONE = 13, B_DQFULL = 14, B_DQCONS = 15, B_DPCONS = 16,
  B_DSSMEM = 19,  // dS^T of the step is in shared memory (for dQ^T)
};
constexpr int OFF_BAR = 0;
constexpr int OFF_LD = 256;  // 2 stages x (-L*log2 e [128], D [128])
constexpr int LD_BYTES = 2 * BM * 4;
constexpr int SMALL = OFF_LD + 2 * LD_BYTES;
constexpr int SMEM_MAX = 232448;  // the per-block maximum
constexpr int TM_DK = 0, TM_DV = 128, TM_R = 256, TM_COLS = 512;

// Shared-memory layout at head size D with NKV K, V buffers, 1 KiB-aligned tiles after
// the small region.  Every 128-row tile is stored in 64-column chunks of CHUNK bytes.
template <int D, int NKV_>
struct Lay {
  static_assert(D == 64 || D == 128, "head size");
  static constexpr int NKV = NKV_;
  static constexpr int TQ = 128 * D * 2;  // a Q, dO or V tile
  static constexpr int TK = 2 * CHUNK;    // K: two chunks (at D = 64 the second is a copy)
  static constexpr int KVB = TK + TQ;     // one K, V buffer
  static constexpr int T_Q = NKV_ * KVB;   // Q, dO of stage s at T_Q + s * 2 TQ (+ TQ for dO)
  static constexpr int T_DS = T_Q + 4 * TQ;  // dS^T [128 keys][128 queries]
  static constexpr int TILES = T_DS + 2 * CHUNK;
  static constexpr int SMEM = 3072 + TILES;  // with a 1 KiB-aligned base the tiles start at 3 KiB
  static_assert(SMALL <= 3072 && SMEM <= SMEM_MAX, "shared memory budget");
  static FA_DEV uint32_t k(uint32_t tb, int b) { return tb + b * KVB; }
  static FA_DEV uint32_t v(uint32_t tb, int b) { return tb + b * KVB + TK; }
  static FA_DEV uint32_t q(uint32_t tb, int s) { return tb + T_Q + s * 2 * TQ; }
  static FA_DEV uint32_t dO(uint32_t tb, int s) { return tb + T_Q + s * 2 * TQ + TQ; }
};
// The layouts the kernels use: one K, V buffer at d = 128 (224 KiB of tiles), two at
// d = 64 (192 KiB).
template <int D>
using LayFor = Lay<D, D == 128 ? 1 : 2>;

// What every role needs: shared-window addresses of the small region and the tiles,
// generic pointers to the same, the tensor-memory base and the wait guard.
struct Ctx {
  uint32_t sb, tb;
  uint8_t* small;
  uint8_t* tiles;
  uint32_t tmem;
  Guard guard;
  FA_DEV uint32_t bar(int i) const { return sb + OFF_BAR + 8 * i; }
};

// Producer (whole warp): Q_i, dO_i of query tile rows q0 .. q0+127 of head bh into
// stage g % 2 (once the dK product of step g-2 has released it), and -L log2 e, D of
// those rows into shared memory (rows past Nq get -L log2 e = -inf, so their P is 0).
template <class LY>
FA_DEV bool produce_step(const Ctx& x, const CUtensorMap* tmQ, const CUtensorMap* tmdO, const float* Lg,
                         const float* Dg, size_t row0, int Nq, int q0, int bh, int g, int lane, int site) {
  const int s = g & 1;
  // read before waiting for the stage
  float lv[4], dv[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int q = q0 + lane + 32 * u;
    lv[u] = q < Nq ? -Lg[row0 + q] * kLog2e : -INFINITY;
    dv[u] = q < Nq ? Dg[row0 + q] : 0.f;
  }
  if (!mbar_wait_warp(x.bar(B_QEMPTY + s), ((g >> 1) & 1) ^ 1, x.guard, site)) return false;
  if (lane == 0) {
    mbar_expect_tx(x.bar(B_QFULL + s), 2 * LY::TQ);
    for (int c = 0; c < LY::TQ / CHUNK; ++c) {
      tma_load_3d(LY::q(x.tb, s) + c * CHUNK, tmQ, x.bar(B_QFULL + s), c * 64, q0, bh);
      tma_load_3d(LY::dO(x.tb, s) + c * CHUNK, tmdO, x.bar(B_QFULL + s), c * 64, q0, bh);
    }
  }
  float* Ls = reinterpret_cast<float*>(x.small + OFF_LD + s * LD_BYTES);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    Ls[lane + 32 * u] = lv[u];
    Ls[BM + lane + 32 * u] = dv[u];
  }
  mbar_arrive(x.bar(B_QFULL + s));
  return true;
}

// UMMA issuer A (one thread): S^T = K Q^T into region g % 2, dP^T = V dO^T into the
// other region.  K and V (buffer kvb) must be in shared memory.
template <class LY>
FA_DEV bool issue_s_dp(const Ctx& x, int g, int kvb, int site) {
  constexpr uint32_t idKK = idesc_bf16(128, 128, false, false);  // K-major x K-major
  constexpr int KS = LY::TQ / (128 * 32);                         // k-steps of 16 over d
  const int s = g & 1;
  const uint32_t kb = LY::k(x.tb, kvb), vb = LY::v(x.tb, kvb);
  const uint32_t qb = LY::q(x.tb, s), db = LY::dO(x.tb, s);
  const uint32_t rs = x.tmem + TM_R + 128 * s, rd = x.tmem + TM_R + 128 * (s ^ 1);
  if (!mbar_wait(x.bar(B_QFULL + s), (g >> 1) & 1, x.guard, site)) return false;
  // region s held dP^T of the previous step: every element-wise thread has read it
  if (g > 0 && !mbar_wait(x.bar(B_DPCONS), (g - 1) & 1, x.guard, site)) return false;
  tc_fence_after();
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
    mma_ss(rs, sdesc_kmajor<128, 128>(kb, ks), sdesc_kmajor<128, 128>(qb, ks), idKK, ks > 0);
  mma_commit(x.bar(B_SFULL));
  // region s^1 ended the previous step holding its dQ^T: the drain warps have read it
  if (g > 0 && !mbar_wait(x.bar(B_DQCONS), (g - 1) & 1, x.guard, site)) return false;
  tc_fence_after();
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
    mma_ss(rd, sdesc_kmajor<128, 128>(vb, ks), sdesc_kmajor<128, 128>(db, ks), idKK, ks > 0);
  mma_commit(x.bar(B_DPFULL));
  return true;
}

// UMMA issuer B (one thread): dV += P^T dO, dK += dS^T Q (both A operands in tensor
// memory), then dQ^T = K^T dS^T (both from shared memory) over region g % 2 once dV
// and dK have read its P^T and dS^T.  first: the unit's first step (the accumulators
// start from zero).  S^T and dP^T of the step are complete before the element-wise
// warps signal P and dS ready, so this thread's commits cover every reader of Q, dO.
template <class LY>
FA_DEV bool issue_dv_dk_dq(const Ctx& x, int g, int kvb, bool first, int site) {
  constexpr uint32_t idTN = idesc_bf16(128, LY::TQ / 256, false, true);  // A in TMEM x N-major B (N = d)
  constexpr uint32_t idMN = idesc_bf16(128, 128, true, true);            // K^T (M-major) x dS^T (N-major)
  const int s = g & 1;
  const uint32_t kb = LY::k(x.tb, kvb), dsb = x.tb + LY::T_DS;
  const uint32_t qb = LY::q(x.tb, s), db = LY::dO(x.tb, s);
  const uint32_t rs = x.tmem + TM_R + 128 * s;
  // dV += P^T dO.  Query block ks (16 queries) is in half ks/4, sub-chunk (ks%4)/2; its
  // bf16 P^T sits in columns 64 (ks/4) + 8 (ks%4).  Sub-chunk 0 (blocks 0,1,4,5) is
  // ready before sub-chunk 1 (blocks 2,3,6,7).
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    if (!mbar_wait(x.bar(B_PREADY + 2 * s + c), (g >> 1) & 1, x.guard, site)) return false;
    tc_fence_after();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int ks = 4 * (u >> 1) + 2 * c + (u & 1);
      mma_ts(x.tmem + TM_DV, rs + 64 * (ks >> 2) + (ks & 3) * 8, sdesc_mnmajor<128, 128>(db, ks), idTN,
             (!first || ks > 0));
    }
  }
  // dK += dS^T Q (dS^T of block ks in columns 64 (ks/4) + 32 + 8 (ks%4))
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    if (!mbar_wait(x.bar(B_DSREADY + c), g & 1, x.guard, site)) return false;
    tc_fence_after();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int ks = 4 * (u >> 1) + 2 * c + (u & 1);
      mma_ts(x.tmem + TM_DK, rs + 64 * (ks >> 2) + 32 + (ks & 3) * 8, sdesc_mnmajor<128, 128>(qb, ks), idTN,
             (!first || ks > 0));
    }
  }
  mma_commit(x.bar(B_DKDONE));
  mma_commit(x.bar(B_QEMPTY + s));  // Q, dO of this stage have no later reader
  if (!mbar_wait(x.bar(B_DKDONE), g & 1, x.guard, site)) return false;
  if (!mbar_wait(x.bar(B_DSSMEM), g & 1, x.guard, site)) return false;
  tc_fence_after();
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    mma_ss(rs, sdesc_mnmajor<128, 128>(kb, ks), sdesc_mnmajor<128, 128>(dsb, ks), idMN, ks > 0);
  mma_commit(x.bar(B_DQFULL));
  return true;
}

// dQ drain (warp qw of warps 12..15, lane quarter qw): takes its columns of dQ_g^T out
// of tensor memory at once, frees them, then adds them into the fp32 workspace from
// registers (each warp access covers 32 consecutive d of one query row, 128 bytes).
// d = 128: d = 32 qw + lane, all 128 queries.  d = 64 (lanes 64..127 repeat 0..63):
// d = 32 (qw % 2) + lane, queries 64 (qw / 2) .. +63.  tile: workspace row q0 of the
// step's query tile (nq <= 128 valid rows).
template <int D>
FA_DEV bool drain_step(const Ctx& x, int g, float* tile, int nq, int qw, int lane, int site) {
  constexpr int NQ = D == 128 ? 128 : 64;  // queries per drain thread
  const int qb = D == 128 ? 0 : 64 * (qw >> 1);
  float* dst = tile + static_cast<size_t>(qb) * D + (D == 128 ? qw : (qw & 1)) * 32 + lane;
  const int nv = nq - qb;  // valid queries of this thread's range
  const uint32_t tl = x.tmem + (static_cast<uint32_t>(qw * 32) << 16);
  if (!mbar_wait_warp(x.bar(B_DQFULL), g & 1, x.guard, site)) return false;
  tc_fence_after();
  uint32_t r[NQ];
#pragma unroll
  for (int c = 0; c < NQ / 32; ++c) tmem_ld32(tl + TM_R + 128 * (g & 1) + qb + 32 * c, r + 32 * c);
  tmem_ld_wait<NQ>(r);
  tc_fence_before();
  mbar_arrive(x.bar(B_DQCONS));
  if (nv >= NQ) {
#pragma unroll
    for (int q = 0; q < NQ; ++q) atomicAdd(dst + static_cast<size_t>(q) * D, __uint_as_float(r[q]));
  } else {
#pragma unroll
    for (int q = 0; q < NQ; ++q)
      if (q < nv) atomicAdd(dst + static_cast<size_t>(q) * D, __uint_as_float(r[q]));
  }
  return true;
}

// Element-wise warps (warp w of 4..11: lane quarter qw = w % 4, query half h = (w-4)/4;
// one key row per thread): P^T and dS^T of step g, key tile kt (this thread's key
// row kr), query tile qt.  off = Nk - Nq (query q sits at q + off).
template <class LY, bool CAUSAL>
FA_DEV bool ew_step(const Ctx& x, int g, int kt, int qt, int Nk, int off, int window, float c_log2, int qw, int h,
                    int lane, int site) {
  // d = 128: P^T goes to the dV product only after dP^T is out of tensor memory, so that
  // the dV product (a TS UMMA, whose tensor-memory reads slow tcgen05.ld down) does not
  // run under that load (measured +0.4-1.2% at d = 128; at d = 64, where dV is shorter
  // and its early start matters more, releasing each half of P^T at once is 2% faster).
  constexpr bool DP_FIRST = LY::TQ == 128 * 128 * 2;
  const int s = g & 1;
  const int kr = qw * 32 + lane;  // key row (tensor-memory lane)
  const int key = kt * BN + kr;
  const uint32_t tl = x.tmem + (static_cast<uint32_t>(qw * 32) << 16);
  if (!mbar_wait_warp(x.bar(B_QFULL + s), (g >> 1) & 1, x.guard, site)) return false;
  if (!mbar_wait_warp(x.bar(B_SFULL), g & 1, x.guard, site)) return false;
  tc_fence_after();
  const uint32_t rs = tl + TM_R + 128 * s, rd = tl + TM_R + 128 * (s ^ 1);
  const int qh = qt * BM + 64 * h;  // first query of this half
  const float4* L4 = reinterpret_cast<const float4*>(x.small + OFF_LD + s * LD_BYTES) + 16 * h;
  const float4* D4 = L4 + BM / 4;
  const bool masked = (CAUSAL && kt * BN + BN - 1 > qh + off) || (window > 0 && kt * BN <= qh + 63 + off - window) ||
                      (kt * BN + BN > Nk);
  // queries of this half (0..63) that see this thread's key: key <= q + off (causal),
  // key > q + off - window (window), and none at all past Nk
  const int qlo = CAUSAL ? key - off - qh : 0;
  const int qhi = key >= Nk ? -1 : (window > 0 ? key - off + window - 1 - qh : 63);
  const uint64_t cc = f2pack(c_log2, c_log2);
  // ---- P^T = 2^(S^T c - L log2 e), two sub-chunks of 32 queries, each released to the
  // dV product as soon as it is in tensor memory
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
          const int xx = 4 * v + y;  // within the sub-chunk
          const uint64_t t = ffma2(f2pack(__uint_as_float(r[xx]), __uint_as_float(r[xx + 1])), cc,
                                   y == 0 ? f2pack(l.x, l.y) : f2pack(l.z, l.w));
          float t0, t1;
          f2unpack(t, t0, t1);
          p[y] = ex2(t0);
          p[y + 1] = ex2(t1);
          if (MASK) {
            const int xs = 32 * c + xx;  // query of the half: visible iff qlo <= xs <= qhi
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
    if (!DP_FIRST) {
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(x.bar(B_PREADY + 2 * s + c));
    }
  }
  if (DP_FIRST) tmem_st_wait();
  // ---- dS^T = P^T (dP^T - D), from the same bf16 P that enters dV; two sub-chunks
  if (!mbar_wait_warp(x.bar(B_DPFULL), g & 1, x.guard, site)) return false;
  tc_fence_after();
  uint8_t* row = x.tiles + LY::T_DS + h * CHUNK + kr * 128;
  // all of this thread's dP^T out of tensor memory first, so that S^T of the next step
  // can be formed in its region while dS is computed
  uint32_t rdp[64];
  tmem_ld32(rd + 64 * h, rdp);
  tmem_ld32(rd + 64 * h + 32, rdp + 32);
  tmem_ld_wait<64>(rdp);
  tc_fence_before();
  if (DP_FIRST) {
    mbar_arrive(x.bar(B_PREADY + 2 * s));
    mbar_arrive(x.bar(B_PREADY + 2 * s + 1));
  }
  mbar_arrive(x.bar(B_DPCONS));
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
        const uint32_t w = pk[16 * c + (xx >> 1)];
        const uint64_t pp = f2pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
        const uint64_t t = fadd2(f2pack(__uint_as_float(r[xx]), __uint_as_float(r[xx + 1])),
                                 y == 0 ? f2pack(-dd.x, -dd.y) : f2pack(-dd.z, -dd.w));
        float d0, d1;
        f2unpack(fmul2(pp, t), d0, d1);
        dk[xx >> 1] = pack_bf16x2(d0, d1);
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
    mbar_arrive(x.bar(B_DSREADY + c));  // dK reads dS^T from tensor memory
  }
  // dQ^T reads dS^T from shared memory: one proxy fence for both sub-chunks
  fence_proxy_async_smem();
  mbar_arrive(x.bar(B_DSSMEM));
  return true;
}

// Element-wise epilogue, first half: this thread's key row of dK (times scale) and dV,
// d columns (D/2) h .. (D/2) h + D/2 - 1, out of tensor memory as packed bf16
// ([dK | dV] x D/4 pairs); zero when no query saw these keys (the accumulators were
// never written).
template <int D>
FA_DEV void ew_load_dk_dv(const Ctx& x, int qw, int h, float scale, bool none, uint32_t (&outp)[D / 2]) {
  constexpr int HW = D / 2;  // d columns per query half
  const uint32_t tl = x.tmem + (static_cast<uint32_t>(qw * 32) << 16);
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const float f = t == 0 ? scale : 1.f;
#pragma unroll
    for (int c = 0; c < HW / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tl + (t == 0 ? TM_DK : TM_DV) + HW * h + 32 * c, r);
      tmem_ld_wait<32>(r);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        outp[(HW / 2) * t + 16 * c + i] =
            none ? 0u : pack_bf16x2(__uint_as_float(r[2 * i]) * f, __uint_as_float(r[2 * i + 1]) * f);
    }
  }
}

// Second half: the warp's 32 key rows (rows row0 .. row0+31 of [B*H*Nk, D], the first
// nvalid of them below Nk) into dK and dV, d columns (D/2) h .. (D/2) h + D/2 - 1, with
// whole-row writes.  Every lane of the warp must call it.
template <int D>
FA_DEV void ew_store_dk_dv(uint32_t (&outp)[D / 2], __nv_bfloat16* dK, __nv_bfloat16* dV, size_t row0, int nvalid,
                           int h, int lane) {
  constexpr int HW = D / 2;  // d columns per query half
  warp_store_rows<HW / 8, 0>(outp, reinterpret_cast<uint8_t*>(dK + row0 * D + HW * h), D * 2, nvalid, lane);
  warp_store_rows<HW / 8, HW / 2>(outp, reinterpret_cast<uint8_t*>(dV + row0 * D + HW * h), D * 2, nvalid, lane);
}

}  // namespace bsteps
}  // namespace fa
