/*
 * Exact tiled attention (FlashAttention-2 forward and recompute backward) for
 * NVIDIA GB300 (sm_103a): the C ABI of libfa_gb300.so.
 *
 * What is computed (sources: "CS336 Assignment 2 notes: FlashAttention & DDP",
 * Part 1 §1.2-§1.4; "CS324 lecture 8: 03_online_softmax_and_flash.py";
 * "CS349E lecture 11: 03_flash_backward.py"):
 *
 *   S = Q K^T * scale, P = softmax(S) row by row, O = P V          (§1.1, §1.2)
 *   L = m + ln(l): the natural-log logsumexp of each row of S        (§1.2)
 *   D = rowsum(dO * O)                                               (§1.4 Eq 17)
 *   P = exp(S - L), dV = P^T dO, dP = dO V^T, dS = P * (dP - D),
 *   dQ = dS K * scale, dK = dS^T Q * scale                           (§1.4 Eq 13-19)
 *
 * With `causal` != 0, query row i sees keys 0..i (top-left alignment) and a
 * key tile whose first key lies after a query tile's last row is skipped
 * entirely (§1.3; CS349E lecture 11 demo4_causal).
 *
 * Common conventions for every entry point below:
 *   - Q, K, V, O, dO, dQ, dK, dV are bf16 (__nv_bfloat16) device arrays laid
 *     out contiguously as [B, H, N, d] (row stride d elements).  L and D are
 *     fp32 device arrays [B, H, N].  Every pointer must be 16-byte aligned
 *     (L and D: 4-byte aligned).
 *   - d must be 32, 64 or 128; B, H, N >= 0 and B*H <= 65535.  A call with
 *     B*H*N == 0 does nothing and returns FA_OK (pointers may then be NULL).
 *   - scale must be finite and > 0 (normally 1/sqrt(d)).
 *   - The caller owns every buffer.  The library allocates no device memory.
 *   - All work is enqueued asynchronously on `stream` (NULL = the legacy
 *     default stream); entry points return after launch.  Argument errors are
 *     reported before anything is enqueued; a failed launch returns
 *     FA_ERR_CUDA.  Kernels never trap: each wait inside a kernel has a time
 *     limit, and on expiry the kernel records an error in a device status word
 *     and exits; fa_poll_device_error() reads it.
 *   - No N x N buffer is ever allocated or written.
 *   - The library keeps a few device addresses per device for the life of the
 *     process (the status word, the work counters of the persistent kernels,
 *     the array of fa_bwd_noalloc), looked up on first use.  Do not use it
 *     across cudaDeviceReset() or any other teardown of a device's primary
 *     context: those addresses would be stale.
 *   - The debug settings below (fa_debug_*) are process-wide.  Each entry point
 *     reads each setting once per call and takes every decision of that call
 *     from that one reading, so a setting changed from another thread applies
 *     from the next call on.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* fa_stream_t;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or scale       */
    FA_ERR_UNSUPPORTED = 2,  /* d not in {32,64,128}, B*H too large, no sm_103a  */
    FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed                */
    FA_ERR_TIMEOUT = 4,      /* a kernel gave up waiting (see fa_poll_device_error) */
    FA_ERR_WORKSPACE = 5     /* workspace missing or smaller than required       */
} fa_status;

/*
 * Forward pass: O = softmax(Q K^T * scale) V and L = logsumexp of each score row.
 * "CS336 Assignment 2 notes" §1.2 (FlashAttention-2 forward: per query tile,
 * running max m, running sum l, deferred normalisation O/l, L = m + log l)
 * and §1.3 (whole-tile causal skip).
 *   Q, K, V : in,  bf16 [B,H,N,d]
 *   O       : out, bf16 [B,H,N,d]
 *   L       : out, fp32 [B,H,N], natural log, in units of the scaled scores
 */
fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* L,
                 int B, int H, int N, int d, int causal, float scale, fa_stream_t stream);

/*
 * Forward pass with a general mask ("_ex" forms take Nq and Nk separately and a
 * sliding window; fa_fwd is fa_fwd_ex with Nq = Nk = N and window = 0).
 *   Q       : in,  bf16 [B,H,Nq,d]      K, V : in, bf16 [B,H,Nk,d]
 *   O       : out, bf16 [B,H,Nq,d]      L    : out, fp32 [B,H,Nq]
 * Query row i sits at sequence position i + Nk - Nq: the queries are the last
 * Nq positions of the key sequence, so a decoded token (Nq = 1) sees every key
 * ("CS349E lecture 11: 03_flash_backward.py" demo4_causal, observation 3);
 * with Nq = Nk this is the top-left alignment of fa_fwd.
 *   causal : query i sees keys j <= i + Nk - Nq; needs Nq <= Nk
 *            (FA_ERR_UNSUPPORTED otherwise).
 *   window : 0 for none; w > 0 (only with causal, else FA_ERR_INVALID_ARG):
 *            query i also sees only keys j > i + Nk - Nq - w, i.e. itself and
 *            the w - 1 positions before it ("CS324 lecture 8:
 *            03_online_softmax_and_flash.py" window_attention_torch).  Key
 *            tiles wholly outside the band are skipped on both sides.
 * Nq = 0 is a no-op; Nk = 0 with Nq > 0 is FA_ERR_INVALID_ARG (a softmax over
 * no keys).  Every other argument as in fa_fwd.
 */
fa_status fa_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* L,
                    int B, int H, int Nq, int Nk, int d, int causal, int window, float scale,
                    fa_stream_t stream);

/*
 * Backward preprocessing: D_i = sum_k dO_ik * O_ik (fp32 accumulation).
 * "CS336 Assignment 2 notes" §1.4 Eq 17 (D = rowsum(O * dO)); the identity
 * D_i = sum_j dP_ij P_ij that lets D be formed once before the backward is
 * the one of "CS349E lecture 11" demo1_gradcheck.
 *   O, dO : in,  bf16 [B,H,N,d]
 *   D     : out, fp32 [B,H,N]
 */
fa_status fa_bwd_preprocess(const void* O, const void* dO, float* D,
                            int B, int H, int N, int d, fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd needs: an fp32 [B,H,N,d] accumulator for
 * dQ (key tiles add their dS K contributions into it) when the one-kernel
 * backward runs; 0 when the two-kernel backward runs (see
 * fa_debug_set_bwd_split) or for empty inputs; (size_t)-1 for invalid sizes.
 * Query it after any change of the backward split.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d, int causal);

/*
 * Backward pass from the saved O and L: dQ, dK, dV.
 * "CS336 Assignment 2 notes" §1.4 Equations 13-19, key/value tiles in the
 * outer loop (kernel 1 of the notes' two-kernel backward) with dQ accumulated
 * across key tiles in the fp32 workspace, then rounded to bf16.
 *   Q, K, V, O, dO : in,  bf16 [B,H,N,d]
 *   L              : in,  fp32 [B,H,N]  (from fa_fwd)
 *   D              : in,  fp32 [B,H,N]  (from fa_bwd_preprocess)
 *   dQ, dK, dV     : out, bf16 [B,H,N,d]
 *   workspace      : scratch, >= fa_bwd_workspace_size() bytes, 16-byte
 *                    aligned; overwritten (zeroed first) on every call, so
 *                    calls that overlap on the GPU must not share it.
 */
fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* L, const float* D, void* dQ, void* dK, void* dV,
                 int B, int H, int N, int d, int causal, float scale,
                 void* workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Backward pass with the general mask of fa_fwd_ex (same Nq, Nk, causal,
 * window; L, D, dQ are [B,H,Nq], [B,H,Nq], [B,H,Nq,d]; dK, dV [B,H,Nk,d]).
 * Keys that no query sees get dK = dV = 0; Nq = 0 writes zeros to dK and dV.
 * The workspace is fa_bwd_workspace_size_ex() bytes.  fa_bwd is fa_bwd_ex with
 * Nq = Nk = N and window = 0.
 */
size_t fa_bwd_workspace_size_ex(int B, int H, int Nq, int Nk, int d, int causal, int window);
fa_status fa_bwd_ex(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                    const float* L, const float* D, void* dQ, void* dK, void* dV,
                    int B, int H, int Nq, int Nk, int d, int causal, int window, float scale,
                    void* workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Largest workspace fa_bwd_noalloc can provide: B*H*N*d*4 bytes must not exceed
 * it (16 MiB, e.g. B*H*N = 32768 rows at d = 128).
 */
#define FA_NOALLOC_MAX_WORKSPACE_BYTES (16u << 20)

/*
 * fa_bwd for callers that cannot allocate device memory when they run the
 * backward: for example, code working inside device memory that a host
 * framework or serving runtime has reserved up front (no allocations outside
 * its pool), or code that must not call cudaMalloc/cudaFree because those can
 * synchronise the device.  The pages have no counterpart: this entry point
 * exists only for such callers.
 *
 * Same arguments, results and errors as fa_bwd, without the workspace: the fp32
 * dQ accumulator is a fixed array inside the library (one per device that
 * loads it, held until the process exits), so the call allocates nothing.
 *   - Returns FA_ERR_WORKSPACE, without enqueuing anything, when the backward
 *     that runs needs an accumulator larger than the array:
 *     fa_bwd_workspace_size() > FA_NOALLOC_MAX_WORKSPACE_BYTES, i.e.
 *     B*H*N*d*4 bytes for the one-kernel form (d = 32, d = 128 by default).
 *     The two-kernel form (d = 64 by default) uses no accumulator and no
 *     array, and has no such limit.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - All calls on a device share the array, which keeps the last call's
 *     contents; each call zeroes it on `stream` first.  Calls on the same device
 *     whose work overlaps on the GPU race on it: serialise them.
 */
fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                         const float* L, const float* D, void* dQ, void* dK, void* dV,
                         int B, int H, int N, int d, int causal, float scale, fa_stream_t stream);

/*
 * One forward + backward step of exact attention on HOST-resident tensors: O,
 * L, dQ, dK, dV from Q, K, V, dO, exactly as fa_fwd_ex, fa_bwd_preprocess and
 * fa_bwd_ex compute them (same mask rules, same kernels), with every host <->
 * device copy inside the call.  The pages run both passes on device arrays; this
 * entry point is for callers whose tensors live in host memory, and it hides the
 * copies behind the kernels: the B*H heads go through in chunks, and while one
 * chunk computes, the next chunk's inputs come in and the previous chunk's
 * results go out, on streams internal to the library.
 *
 *   Q, dO: bf16 host [B,H,Nq,d]; K, V: bf16 host [B,H,Nk,d]; outputs O, dQ: bf16
 *   host [B,H,Nq,d]; dK, dV: bf16 host [B,H,Nk,d]; L: fp32 host [B,H,Nq].  Host
 *   arrays should be page-locked (cudaHostAlloc, cudaHostRegister) for the copies
 *   to run asynchronously and overlap the kernels; pageable arrays give the same
 *   results with the copies serialised.
 *   heads_per_chunk: heads of the flattened B*H per chunk; 0 lets the library
 *   choose (fa_fwd_bwd_host_chunk_heads tells which).
 *   workspace: fa_fwd_bwd_host_workspace_size() bytes of device memory, 256-byte
 *   aligned (FA_ERR_WORKSPACE otherwise): device copies of up to four chunks and
 *   two dQ accumulators.  Calls that share a workspace must be ordered (the same
 *   stream, or synchronised).
 *   stream: the step is ordered after the work already on `stream`, and work
 *   enqueued on `stream` later is ordered after the last copy back.  The call
 *   returns once all of it is enqueued; the host outputs are valid, and the host
 *   inputs may change again, after `stream` is synchronised.
 * Argument errors return before anything is enqueued.  A failure midway (a CUDA
 * call, or an error from one chunk's fa_fwd_ex / fa_bwd_ex) returns that status
 * with part of the step enqueued; `stream` is still ordered after every copy
 * that was enqueued, so once `stream` is synchronised the library no longer
 * reads or writes the host arrays.
 * fa_fwd_bwd_host_chunk_heads and fa_fwd_bwd_host_workspace_size are host only
 * (no GPU needed) and return -1 (as size_t for the second) on bad arguments.
 */
int fa_fwd_bwd_host_chunk_heads(int B, int H, int Nq, int Nk, int d, int heads_per_chunk);
size_t fa_fwd_bwd_host_workspace_size(int B, int H, int Nq, int Nk, int d, int causal, int window,
                                      int heads_per_chunk);
fa_status fa_fwd_bwd_host(const void* Q, const void* K, const void* V, const void* dO,
                          void* O, float* L, void* dQ, void* dK, void* dV,
                          int B, int H, int Nq, int Nk, int d, int causal, int window, float scale,
                          int heads_per_chunk, void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* fa_status_string(fa_status s);

/*
 * Tile shape used by a pass: pass 0 = forward (Br query rows x Bc keys),
 * pass 1 = backward main kernel (Br query rows per inner step x Bc keys per
 * CTA).  Host only; needs no GPU.
 */
fa_status fa_get_tile_config(int d, int pass, int* Br, int* Bc);

/*
 * Number of (query tile, key tile) pairs one head computes in a pass, from
 * the closed form for the tiles of fa_get_tile_config (with the causal mask:
 * query tile i sees key tiles 0 .. floor((min((i+1) Br, N) - 1) / Bc);
 * "CS349E lecture 11" demo4_causal).  Host only; -1 on bad arguments.
 */
long long fa_tile_pairs(int N, int d, int causal, int pass);

/*
 * The same count for the mask of fa_fwd_ex: query tile i (positions p_first ..
 * p_last) sees key tiles max(0, floor((p_first - w + 1) / Bc)) .. floor(p_last /
 * Bc) (the first bound only with a window w, the second only when causal).
 * Host only; -1 on bad arguments.
 */
long long fa_tile_pairs_ex(int Nq, int Nk, int d, int causal, int window, int pass);

/*
 * Debug: when `dev_counter` is non-NULL, every later fa_fwd / fa_bwd launch
 * adds the number of tile pairs it computed to *dev_counter (a device
 * unsigned long long the caller owns and zeroes).  NULL switches it off.
 * Process-wide setting.
 */
fa_status fa_debug_set_tile_counter(unsigned long long* dev_counter);

/*
 * Debug: which form of the backward fa_bwd runs for d = 64 and 128 ("CS336
 * Assignment 2 notes" §1.4 leaves the split open):
 *   1: one kernel, key/value tiles outer; dQ accumulated in the fp32 workspace
 *      and rounded to bf16 by a second pass;
 *   2: two kernels, key/value tiles outer for dK and dV, then query tiles outer
 *      for dQ (S and P recomputed in both); no workspace, no reductions;
 *   3: form 1 with one CTA per SM taking key tiles from a queue, consecutive
 *      tiles overlapped (d = 64 and 128; the same 1024 work counters rule as
 *      fa_debug_set_fwd_form's form 3);
 *   0: the library's default, chosen by measurement on GB300: form 3 at
 *      d = 128; at d = 64 form 3 when B*H times the visible 128 x 128 tile
 *      pairs per head (fa_tile_pairs_ex) exceeds 3072, else form 2.
 * d = 32 always runs form 1.  Process-wide setting; FA_ERR_INVALID_ARG for
 * other values.
 */
fa_status fa_debug_set_bwd_split(int split);

/*
 * Debug: which forward kernel fa_fwd runs (the same computation, "CS336
 * Assignment 2 notes" §1.2; form 2 exists for d = 128 only, other d run form 1
 * in its place):
 *   1: one 128-row query tile per CTA;
 *   2: two query tiles per CTA whose softmax and tensor-core work take turns;
 *   3: one CTA per SM taking query tiles from a queue, consecutive tiles
 *      overlapped (any d).  Each launch takes the next of 1024 work counters in
 *      a static device array (no allocation), which its last CTA leaves zeroed
 *      for the counter's next launch; at most 1024 such launches may be in
 *      flight at once across streams;
 *   0: the library's default, chosen by measurement on GB300: form 3 for d <= 64,
 *      and for d = 128 when no query tile sees more than 128 key tiles; else 1.
 * Process-wide setting; FA_ERR_INVALID_ARG for other values.
 */
fa_status fa_debug_set_fwd_form(int form);

/*
 * Which backward form fa_bwd_ex would run for these sizes and mask, and the
 * workspace it would need, both taken from one reading of the
 * fa_debug_set_bwd_split setting, exactly as fa_bwd_ex takes them: a form that
 * reduces dQ in the workspace (1, 3) always comes with B*H*Nq*d*4 bytes, the
 * two-kernel form (2) with 0.  Host only; the argument checks of fa_bwd_ex.
 */
fa_status fa_debug_bwd_plan(int B, int H, int Nq, int Nk, int d, int causal, int window, int* form,
                            size_t* workspace_bytes);

/*
 * Debug: times the main kernels from the caller's side.  `start` and `stop` are
 * CUDA events (cudaEvent_t, created and owned by the caller); later calls of
 * fa_fwd_ex (which = 0) or fa_bwd_ex (which = 1) record `start` on their
 * stream just before launching their main kernel (the forward kernel; the
 * backward main kernel, or both kernels of the two-kernel form) and `stop` just
 * after it, so cudaEventElapsedTime(start, stop) is that launch's device time
 * (the backward's workspace clear and dQ conversion are outside it).  Both NULL
 * switch it off; exactly one NULL is FA_ERR_INVALID_ARG.  Process-wide setting.
 */
fa_status fa_debug_set_kernel_events(int which, void* start, void* stop);

/*
 * Which forms fa_fwd_ex and fa_bwd_ex would run for these sizes and mask under
 * the current settings (the numbers of fa_debug_set_fwd_form and
 * fa_debug_set_bwd_split).  Host only; the argument checks of fa_fwd_ex.
 */
fa_status fa_selected_forms(int B, int H, int Nq, int Nk, int d, int causal, int window, int* fwd_form,
                            int* bwd_form);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device.  FA_OK if no kernel has given up since the last poll;
 * FA_ERR_TIMEOUT otherwise, with the failing wait site in *detail (may be NULL).
 * While the word is set, later launches skip their work.
 */
fa_status fa_poll_device_error(fa_stream_t stream, int* detail);

/*
 * Diagnostic: runs one wait on a barrier that nothing ever completes, with a
 * limit of `limit_us` microseconds (1..1000000), on `stream`.  The kernel
 * must give up, record FA_ERR_TIMEOUT and exit; a following
 * fa_poll_device_error() returns it.  Exercises the bounded-wait path that
 * every kernel uses, without faulting or hanging the GPU.
 */
fa_status fa_debug_timeout_probe(int limit_us, fa_stream_t stream);

/*
 * Diagnostic: one 128 x N x K tile product on the tensor cores through the
 * same shared-memory / tensor-memory operand paths the attention kernels use.
 *   mode 0: C = A B^T, A [128][K], B [N][K]          (both K-major)
 *   mode 1: C = A B,   A [128][K], B [K][N]          (B N-major)
 *   mode 2: C = A B,   A [128][K] staged in tensor memory, B [K][N]
 *   mode 3: C = A^T B^T, A [K][128], B [N][K]        (A M-major)
 *   mode 4: C = A^T B, A [K][128], B [K][N]          (both M/N-major)
 * A, B: bf16 device arrays (row-major as shown); C: fp32 [128][N] device.
 * K and N in {32, 64, 128}.  Not part of attention; used by the tests.
 */
fa_status fa_selftest_umma(int mode, const void* A, const void* B, float* C, int K, int N,
                           fa_stream_t stream);

/* Library version: major*10000 + minor*100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
