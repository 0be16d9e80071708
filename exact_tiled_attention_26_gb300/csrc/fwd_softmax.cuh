// The forward's per-row softmax work, shared by the one-tile (fwd.cu) and the
// two-tile (fwd_pp.cu) forward kernels: "CS336 Assignment 2 notes" §1.2 for one
// query row, one key tile at a time, in base 2 with the softmax scale folded into
// one FMA.  The thread owns one query row: its tensor-memory lane.
//
// The reference max m is moved lazily, with hysteresis.  O / l and L = m + log l do
// not depend on which m is used, so m only has to keep P = 2^(S c - m) inside the
// range of fp32 and bf16: it starts kFwdMaxHeadroom above the first tile's max and
// is moved (to kFwdMaxHeadroom above the new tile's max, with O and l multiplied by
// 2^(m_old - m_new)) only when a tile's max passes it by more than
// kFwdRescaleThreshold.  Between moves P <= 2^24 and each row's largest weight is
// >= 2^-24, so sums over up to 2^30 keys stay far inside fp32 for any |V| < 2^70.
// Every row's max grows as more keys are seen (by about 30 in base 2 over 8192 keys
// when the scores have a standard deviation of 16); starting above it makes moves
// rare: with Q, K scaled by 4 on the 1 x 32 x 8192 x 128 causal shape, a move on
// about 2.5% of (warp, key tile) steps against 57% for "start at the first tile's
// max, move past 8" (simulated from the same score distribution).
#pragma once

#include "ptx.cuh"

namespace fa {

constexpr float kFwdRescaleThreshold = 24.0f;  // base-2 units
constexpr float kFwdMaxHeadroom = 24.0f;       // base-2 units
constexpr float kFwdLn2 = 0.6931471805599453f;

// Running state of one query row.
struct SoftmaxRow {
  float m_run = -INFINITY;  // running (reference) max of S * scale * log2(e)
  float l_run = 0.f;        // running sum of P (for L)
  float lr_run = 0.f;       // running sum of P as rounded to bf16 for the P V product (for O)
};

// One 128-key tile for the calling thread's query row q: S (128 fp32 columns at
// tS, already complete) is masked, the running max updated, and P = 2^(S c - m)
// written back as bf16 over the first 64 columns at tS (the tensor-memory stores
// are complete on return).  When the max moves, O (D columns at tO) is rescaled
// after wait_o() reports that the product that last wrote O is complete.
//   first: the row's first key tile; k0: its first key; row0: first query row of
//   the query tile (for the edge test); off = Nk - Nq (query q sits at q + off).
// Returns false only if wait_o() gave up.
template <int D, bool CAUSAL, bool WINDOW, class WaitO>
FA_DEV bool softmax_tile(SoftmaxRow& st, uint32_t tS, uint32_t tO, bool first, int k0, int row0, int q, int off,
                         int Nk, int window, float c_log2, WaitO&& wait_o) {
  constexpr int BM = 128, BN = 128;
  uint32_t r[128];
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, r + 32 * c);
  tmem_ld_wait<128>(r);
  float s[128];
#pragma unroll
  for (int k = 0; k < 128; ++k) s[k] = __uint_as_float(r[k]);
  if ((CAUSAL && k0 + BN - 1 > row0 + off) || (WINDOW && k0 <= row0 + BM - 1 + off - window) || k0 + BN > Nk) {
    // this row sees tile columns lo .. hi (position q + off; keys below Nk)
    const int hi = min(CAUSAL ? q + off - k0 : BN - 1, Nk - 1 - k0);
    const int lo = WINDOW ? q + off - window + 1 - k0 : 0;
#pragma unroll
    for (int k = 0; k < 128; ++k)
      if (k > hi || k < lo) s[k] = -INFINITY;
  }
  // row max as eight independent chains of 3-input maxes (depth ~10, not 127)
  float m8[8];
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    m8[a] = fmax3(s[16 * a], s[16 * a + 1], s[16 * a + 2]);
#pragma unroll
    for (int b = 3; b < 15; b += 2) m8[a] = fmax3(m8[a], s[16 * a + b], s[16 * a + b + 1]);
    m8[a] = fmaxf(m8[a], s[16 * a + 15]);
  }
  const float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
  const float m_tile = mx * c_log2;
  if (first) {
    st.m_run = m_tile + kFwdMaxHeadroom;  // -inf stays -inf (a window's fully masked first tile)
  } else {
    const bool move = m_tile > st.m_run + kFwdRescaleThreshold;
    if (__any_sync(0xffffffffu, move)) {
      const float m_new = m_tile + kFwdMaxHeadroom;
      const float alpha = move ? ex2(st.m_run - m_new) : 1.f;
      if (move) {
        st.l_run *= alpha;
        st.lr_run *= alpha;
        st.m_run = m_new;
      }
      if (!wait_o()) return false;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_ld_wait<32>(o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st32(tO + 32 * c, o);
      }
      tmem_st_wait();
    }
  }
  // a row whose keys so far were all masked (a window's first tile) keeps
  // m = -inf; its P is 0 and the first visible tile rescales by 0
  const float neg_m = (WINDOW && st.m_run == -INFINITY) ? 0.f : -st.m_run;
  // two columns per packed f32x2 instruction: exponent argument and running sum of
  // P (for L); the sum of P as rounded to bf16 (for O's normaliser) adds the packed
  // bf16 pair itself, one mixed-precision add per column; two chains each
  const uint64_t cc2 = f2pack(c_log2, c_log2), nm2 = f2pack(neg_m, neg_m);
  uint64_t ls[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
  float rl[2] = {0.f, 0.f}, rh[2] = {0.f, 0.f};
  uint32_t p[64];
#pragma unroll
  for (int k = 0; k < 128; k += 2) {
    float t0, t1;
    f2unpack(ffma2(f2pack(s[k], s[k + 1]), cc2, nm2), t0, t1);
    const float p0 = ex2(t0), p1 = ex2(t1);
    ls[(k >> 1) & 1] = fadd2(ls[(k >> 1) & 1], f2pack(p0, p1));
    const uint32_t pk = pack_bf16x2(p0, p1);
    p[k >> 1] = pk;
    add_bf16x2_f32(pk, rl[(k >> 1) & 1], rh[(k >> 1) & 1]);
  }
  float a0, a1, a2, a3;
  f2unpack(fadd2(ls[0], ls[1]), a0, a1);
  a2 = rl[0] + rl[1];
  a3 = rh[0] + rh[1];
  st.l_run += a0 + a1;
  st.lr_run += a2 + a3;
  tmem_st32(tS, p);
  tmem_st32(tS + 32, p + 32);
  tmem_st_wait();
  return true;
}

// The epilogue in two halves, for a caller that must release O's columns before the
// global stores: load O / l into packed bf16 registers (the tensor-memory loads are
// complete on return), then store them and L.
template <int D>
FA_DEV void softmax_epilogue_load(const SoftmaxRow& st, uint32_t tO, uint32_t (&pk)[D / 2]) {
  const float inv_l = 1.f / st.lr_run;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(tO + 32 * c, o);
    tmem_ld_wait<32>(o);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[16 * c + i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
  }
}
template <int D>
FA_DEV void softmax_epilogue_store(const SoftmaxRow& st, const uint32_t (&pk)[D / 2], __nv_bfloat16* orow,
                                   float* lrow) {
  uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
  for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
  *lrow = (st.m_run + lg2(st.l_run)) * kFwdLn2;
}

// Second half for a whole warp: its 32 query rows (rows row0 .. row0+31 of [B*H*Nq, D],
// the first nvalid of them below Nq) of O with whole-row writes, and this thread's L
// (row row0 + lane, if below Nq).  Every lane of the warp must call it.
template <int D>
FA_DEV void softmax_epilogue_store_rows(const SoftmaxRow& st, uint32_t (&pk)[D / 2], __nv_bfloat16* O, float* Lout,
                                        size_t row0, int nvalid, int lane) {
  warp_store_rows<D / 8, 0>(pk, reinterpret_cast<uint8_t*>(O + row0 * D), D * 2, nvalid, lane);
  if (lane < nvalid) Lout[row0 + lane] = (st.m_run + lg2(st.l_run)) * kFwdLn2;
}

}  // namespace fa
