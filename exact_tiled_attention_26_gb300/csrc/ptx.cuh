// Thin inline-PTX wrappers for sm_103a: mbarrier (with time-limited waits),
// TMA tile loads, bulk reductions, and the tcgen05 tensor-memory / UMMA
// instructions.  Written from the PTX ISA's descriptions of these instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#define FA_DEV __device__ __forceinline__

namespace fa {

// A kernel gives up on any single wait after this long and records an error.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

FA_DEV uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

FA_DEV uint64_t gtimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------------------
// mbarrier
// ----------------------------------------------------------------------------
FA_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
FA_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
FA_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
FA_DEV void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
FA_DEV bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Where a kernel records that it gave up.  `status` is a device word shared by
// all launches (sticky until the host polls it); `abort` is a per-CTA shared
// flag so that the other roles of the CTA stop waiting at once.
struct Guard {
  int* status;
  volatile int* abort;
};

// Wait for the phase of parity `parity` of barrier `bar` to complete.  Returns
// false (and records `site`) if it has not completed within the limit, or if
// another role of this CTA already gave up.
FA_DEV bool mbar_wait(uint32_t bar, uint32_t parity, const Guard& g, int site,
                      uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = gtimer_ns();
  for (;;) {
    if (mbar_try(bar, parity)) return true;
    if (*g.abort) return false;
    if (gtimer_ns() - t0 > limit_ns) {
      *g.abort = 1;
      atomicCAS(g.status, 0, site);
      __threadfence();
      return false;
    }
  }
}

// Same, taken by a whole warp: the result is uniform across the warp so that
// warp-collective instructions that follow are executed by all lanes or none.
FA_DEV bool mbar_wait_warp(uint32_t bar, uint32_t parity, const Guard& g, int site) {
  const bool ok = mbar_wait(bar, parity, g, site);
  return __all_sync(0xffffffffu, ok);
}

// Used only on the way out of a CTA that gave up: wait (bounded, ignoring the
// abort flag) for asynchronous work this CTA started, so nothing is still
// writing its shared or tensor memory when it exits.
FA_DEV void mbar_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  const uint64_t t0 = gtimer_ns();
  while (!mbar_try(bar, parity)) {
    if (gtimer_ns() - t0 > limit_ns) return;
  }
}

// Move registers between warpgroups (all four warps of a warpgroup execute it).
template <uint32_t N>
FA_DEV void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
template <uint32_t N>
FA_DEV void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }

FA_DEV void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ----------------------------------------------------------------------------
// TMA (tensor-map tile loads) and bulk copies
// ----------------------------------------------------------------------------
FA_DEV void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
FA_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
FA_DEV void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
// Element-wise fp32 add of `bytes` contiguous bytes of shared memory into global
// memory (both 16-byte aligned, bytes a multiple of 16), performed in L2.
FA_DEV void bulk_reduce_add_f32(float* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(gdst),
               "r"(ssrc), "r"(bytes)
               : "memory");
}
FA_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
FA_DEV void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
FA_DEV void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's ordinary shared-memory writes before later reads of the
// same memory by the async proxy (tensor cores, bulk copies).
FA_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ----------------------------------------------------------------------------
// tcgen05: tensor memory and UMMA
// ----------------------------------------------------------------------------
FA_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
FA_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
FA_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
FA_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
FA_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]
FA_DEV void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accum)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
FA_DEV void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accum)
      : "memory");
}
// Arrive once on `bar` when every tcgen05.mma issued so far by this thread is done.
FA_DEV void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulation.
// Bit layout: [4,6) D format (1 = f32), [7,10) A format (1 = bf16),
// [10,13) B format (1 = bf16), 15 A major (1 = M-major), 16 B major
// (1 = N-major), [17,23) N/8, [24,29) M/16.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets (all >> 4), the fixed version bits (0b001 at [46,49)) and the
// swizzle mode at [61,64) (2 = 128 B, 4 = 64 B, 6 = 32 B).
FA_DEV uint64_t make_sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (static_cast<uint64_t>(swz) << 61);
}

template <int SWB>
struct SwzCode;
template <>
struct SwzCode<128> { static constexpr uint32_t v = 2; };
template <>
struct SwzCode<64> { static constexpr uint32_t v = 4; };
template <>
struct SwzCode<32> { static constexpr uint32_t v = 6; };

// Operand tiles in shared memory are stored the way a TMA load with swizzle
// width SWB bytes writes them: the contiguous ("inner") dimension is cut into
// chunks of SWB/2 bf16 elements; chunk c holds those elements for all ROWS outer
// indices, one SWB-byte row per outer index, and chunks follow one another.
//
// K-major operand (outer = M or N, inner = K): descriptor for k-step ks (16 K).
template <int SWB, int ROWS>
FA_DEV uint64_t sdesc_kmajor(uint32_t base, int ks) {
  constexpr int CE = SWB / 2;
  const int k0 = ks * 16;
  const uint32_t addr = base + static_cast<uint32_t>((k0 / CE) * (ROWS * SWB) + (k0 % CE) * 2);
  return make_sdesc(addr, 16, 8 * SWB, SwzCode<SWB>::v);
}
// M/N-major operand (outer = K, inner = M or N): k-step ks covers outer rows
// [16 ks, 16 ks + 16); the next SWB/2 M/N elements live one chunk further on.
template <int SWB, int ROWS>
FA_DEV uint64_t sdesc_mnmajor(uint32_t base, int ks) {
  const uint32_t addr = base + static_cast<uint32_t>(ks * 16 * SWB);
  return make_sdesc(addr, ROWS * SWB, 8 * SWB, SwzCode<SWB>::v);
}

// The same descriptors as a base (k-step 0) plus a per-k-step byte offset, so
// that an issuing loop adds a compile-time constant to the start-address field
// (bits [0,14), address >> 4) instead of rebuilding the descriptor.
template <int SWB, int ROWS>
FA_DEV uint64_t sdesc_kmajor_base(uint32_t base) {
  return make_sdesc(base, 16, 8 * SWB, SwzCode<SWB>::v);
}
template <int SWB, int ROWS>
FA_DEV uint64_t sdesc_mnmajor_base(uint32_t base) {
  return make_sdesc(base, ROWS * SWB, 8 * SWB, SwzCode<SWB>::v);
}
template <int SWB, int ROWS>
__host__ __device__ constexpr uint32_t kmajor_off(int ks) {
  return static_cast<uint32_t>(((ks * 16) / (SWB / 2)) * (ROWS * SWB) + ((ks * 16) % (SWB / 2)) * 2);
}
template <int SWB>
__host__ __device__ constexpr uint32_t mnmajor_off(int ks) {
  return static_cast<uint32_t>(ks * 16 * SWB);
}
FA_DEV uint64_t desc_at(uint64_t base_desc, uint32_t byte_off) { return base_desc + (byte_off >> 4); }

// Byte offset of bf16 element (row, col) in a SWB=128 tile written as above
// (ROWS rows per chunk), including the 128-byte swizzle (16-byte unit index
// XOR row % 8).  The tile base must be 1024-byte aligned.
template <int ROWS>
FA_DEV uint32_t swz128_offset(int row, int col) {
  const int chunk = col >> 6, c = col & 63;
  return static_cast<uint32_t>(chunk * (ROWS * 128) + row * 128 + ((((c >> 3) ^ (row & 7)) << 4) | ((c & 7) << 1)));
}

// tcgen05.ld / st, 32 data-path lanes x 32-bit, N consecutive columns per lane.
#define FA_R8(b) "=r"(r[b + 0]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), "=r"(r[b + 4]), "=r"(r[b + 5]), "=r"(r[b + 6]), "=r"(r[b + 7])
#define FA_W8(b) "r"(r[b + 0]), "r"(r[b + 1]), "r"(r[b + 2]), "r"(r[b + 3]), "r"(r[b + 4]), "r"(r[b + 5]), "r"(r[b + 6]), "r"(r[b + 7])

FA_DEV void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24)
      : "r"(taddr));
}
FA_DEV void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : FA_R8(0), FA_R8(8)
      : "r"(taddr));
}
FA_DEV void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      FA_W8(0), FA_W8(8), FA_W8(16), FA_W8(24)
      : "memory");
}
FA_DEV void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      FA_W8(0), FA_W8(8)
      : "memory");
}
#undef FA_R8
#undef FA_W8

// Wait for this thread's outstanding tcgen05.ld; the registers listed are tied
// to the wait so that no use of them is scheduled before it.
template <int NR>
FA_DEV void tmem_ld_wait(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < NR; ++i) asm volatile("" : "+r"(r[i]));
}
FA_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ----------------------------------------------------------------------------
// Arithmetic helpers (PTX instructions, not library functions)
// ----------------------------------------------------------------------------
FA_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
FA_DEV float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
FA_DEV float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed pairs of fp32 (Blackwell's two-wide FP32 instructions).
FA_DEV uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
FA_DEV void f2unpack(uint64_t v, float& lo, float& hi) { asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v)); }
FA_DEV uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
FA_DEV uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
FA_DEV uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

FA_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// lo += the low bf16 of pk, hi += its high bf16: two mixed-precision adds (sm_100
// and later), each widening its bf16 operand exactly and rounding the f32 sum to
// nearest, so the same as adding the two halves unpacked to f32.
FA_DEV void add_bf16x2_f32(uint32_t pk, float& lo, float& hi) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n add.rn.f32.bf16 %0, l, %0;\n add.rn.f32.bf16 %1, h, %1;\n}"
      : "+f"(lo), "+f"(hi)
      : "r"(pk));
}

// Stores a warp's 32 rows with whole-row writes.  Lane l holds row l's NC 16-byte
// chunks in words v[OFF .. OFF + 4 NC); row l goes to `base + l * stride` (bytes).  A
// butterfly of shuffles over groups of NC lanes hands lane i chunk i % NC of its
// group's NC rows, so that each store instruction writes 32 / NC whole rows of 16 NC
// bytes instead of 32 scattered 16-byte pieces.  Only rows below nvalid are written.
// Every lane of the warp must call it; v is left permuted.
template <int NC, int OFF, int N>
FA_DEV void warp_store_rows(uint32_t (&v)[N], uint8_t* base, size_t stride, int nvalid, int lane) {
  static_assert(NC >= 1 && NC <= 32 && (NC & (NC - 1)) == 0 && OFF + 4 * NC <= N, "chunks");
#pragma unroll
  for (int m = NC / 2; m >= 1; m >>= 1) {
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int k0 = 0; k0 < NC; ++k0) {
      if (k0 & m) continue;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t& a0 = v[OFF + 4 * k0 + w];
        uint32_t& a1 = v[OFF + 4 * (k0 | m) + w];
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, hi ? a0 : a1, m);
        if (hi) a0 = recv; else a1 = recv;
      }
    }
  }
  const int c = lane & (NC - 1), g0 = lane & ~(NC - 1);
#pragma unroll
  for (int j = 0; j < NC; ++j)
    if (g0 + j < nvalid)
      *reinterpret_cast<uint4*>(base + static_cast<size_t>(g0 + j) * stride + 16 * c) =
          make_uint4(v[OFF + 4 * j], v[OFF + 4 * j + 1], v[OFF + 4 * j + 2], v[OFF + 4 * j + 3]);
}

// Programmatic dependent launch (a kernel launched with launch_pdl, internal.h, may
// start while the kernel before it on the stream is still running).  pdl_wait:
// block until that kernel has completed and its memory writes are visible (a no-op
// when the launch was an ordinary one).  pdl_trigger: let the next kernel on the
// stream, if launched with launch_pdl, start now (its own pdl_wait still orders
// its reads after this kernel's end).  Only the workspace clear triggers early: its
// dependent, the backward kernel, has loads and products to do before it waits.
// A dependent that could only wait (the dQ convert, the preprocess, the forward)
// would hold SMs that another stream's kernels could use, so kernels followed by
// one of those never trigger: their dependents start when they end.
FA_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
FA_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// End of a persistent launch, one thread per CTA after the CTA's last unit fetch:
// q[0] counts the units taken from the queue, q[1] the CTAs finished.  The last CTA to finish
// zeroes both, so the slot is ready for the next launch that takes it (every
// launch starts from zeroes, and a launch that never ran left them untouched).
FA_DEV void queue_release(unsigned int* q) {
  __threadfence();
  if (atomicAdd(q + 1, 1u) == gridDim.x * gridDim.y * gridDim.z - 1) {
    q[0] = 0u;
    q[1] = 0u;
    __threadfence();
  }
}

// Round a dynamic shared-memory pointer up so that its shared-window address is
// 1024-byte aligned (swizzled operand tiles need it).
FA_DEV uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

}  // namespace fa
