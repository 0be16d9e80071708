// Forward + backward on host-resident tensors (fa_fwd_bwd_host): the flattened
// B*H heads go through in chunks, each chunk's inputs copied in on one stream,
// computed on one of two compute streams (so that one chunk's last wave overlaps
// the next chunk's first), and its results copied out on a third; the device
// side holds up to four chunks at once.  Only plumbing lives here: the
// attention itself is the same fa_fwd_ex / fa_bwd_preprocess / fa_bwd_ex calls
// on each chunk's device copies.
#include <cstdint>
#include <mutex>

#include "internal.h"

namespace fa {
namespace {

constexpr int kSlots = 4;           // chunks whose device copies are live at once
constexpr int kComputeStreams = 2;  // chunks computed alternately on two streams
// Small chunks keep the first copy in and the last copy out short; each launch
// should still fill the 152 SMs once.  Measured on the 1 x 32 x 32768 x 128 causal
// step: 1, 2, 4 and 8 heads per chunk gave about 1170, 1156, 1128 and 1077 TFLOP/s.
constexpr int kTargetChunks = 32;
constexpr int kMinTilesPerChunk = 152;
constexpr int kMaxDevices = 64;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Byte offsets of one chunk's device arrays inside its slot.
struct SlotLayout {
  size_t q, k, v, dO, o, L, D, dQ, dK, dV, bytes;
};

SlotLayout slot_layout(int hc, int Nq, int Nk, int d) {
  const size_t rq = static_cast<size_t>(hc) * Nq * d * 2, rk = static_cast<size_t>(hc) * Nk * d * 2;
  const size_t rl = static_cast<size_t>(hc) * Nq * 4;
  SlotLayout s{};
  size_t at = 0;
  auto put = [&](size_t* off, size_t bytes) {
    *off = at;
    at += align256(bytes);
  };
  put(&s.q, rq);
  put(&s.k, rk);
  put(&s.v, rk);
  put(&s.dO, rq);
  put(&s.o, rq);
  put(&s.L, rl);
  put(&s.D, rl);
  put(&s.dQ, rq);
  put(&s.dK, rk);
  put(&s.dV, rk);
  s.bytes = at;
  return s;
}

struct Plan {
  int hc = 0, chunks = 0, slots = 0, streams = 0;
  SlotLayout slot{};
  size_t acc_bytes = 0;  // one dQ accumulator (fa_bwd_workspace_size_ex of a full chunk)
  size_t total = 0;
};

int chunk_heads(int BH, int Nq, int Nk, int heads_per_chunk) {
  if (BH <= 0) return 0;
  if (heads_per_chunk > 0) return heads_per_chunk < BH ? heads_per_chunk : BH;
  // at least one wave of tiles per chunk, in the shorter of the query and key directions
  const int tq = (Nq + kFwdBr - 1) / kFwdBr, tk = (Nk + kBwdBc - 1) / kBwdBc;
  const int tiles = (tq < tk ? tq : tk) > 0 ? (tq < tk ? tq : tk) : 1;
  int hc = (kMinTilesPerChunk + tiles - 1) / tiles;
  const int by_count = (BH + kTargetChunks - 1) / kTargetChunks;
  if (hc < by_count) hc = by_count;
  if (hc >= BH) return BH;
  const int chunks = (BH + hc - 1) / hc;
  return (BH + chunks - 1) / chunks;  // even chunks: no short last one
}

Plan make_plan(int BH, int Nq, int Nk, int d, int causal, int window, int heads_per_chunk) {
  Plan p;
  p.hc = chunk_heads(BH, Nq, Nk, heads_per_chunk);
  if (p.hc == 0) return p;
  p.chunks = (BH + p.hc - 1) / p.hc;
  p.slots = p.chunks < kSlots ? p.chunks : kSlots;
  p.streams = p.chunks < kComputeStreams ? p.chunks : kComputeStreams;
  p.slot = slot_layout(p.hc, Nq, Nk, d);
  p.acc_bytes = align256(fa_bwd_workspace_size_ex(1, p.hc, Nq, Nk, d, causal, window));
  p.total = p.slot.bytes * p.slots + p.acc_bytes * p.streams;
  return p;
}

// Streams and events of one device, created on first use and kept for the process.
struct Pipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr, comp[kComputeStreams] = {};
  // per slot: Q, K, V in; dO in; forward done (O, L ready); backward done; every output out
  cudaEvent_t start = nullptr, end = nullptr, in_qkv[kSlots] = {}, in[kSlots] = {}, fwd[kSlots] = {}, done[kSlots] = {},
              out[kSlots] = {};
  cudaEvent_t drain[1 + kComputeStreams] = {};  // the tails of h2d and the compute streams, on an error
};
Pipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu;  // held for a whole enqueue: the slot events are shared

bool make_pipe(Pipe* p) {
  if (p->ready) return true;
  // handles made by an earlier, failed attempt are kept; only the missing ones are made
  auto stream = [](cudaStream_t* s) { return *s != nullptr || cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) == cudaSuccess; };
  auto event = [](cudaEvent_t* e) { return *e != nullptr || cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
  bool ok = stream(&p->h2d) && stream(&p->d2h) && event(&p->start) && event(&p->end);
  for (int i = 0; ok && i < kComputeStreams; ++i) ok = stream(&p->comp[i]);
  for (int i = 0; ok && i < 1 + kComputeStreams; ++i) ok = event(&p->drain[i]);
  for (int i = 0; ok && i < kSlots; ++i)
    ok = event(&p->in_qkv[i]) && event(&p->in[i]) && event(&p->fwd[i]) && event(&p->done[i]) && event(&p->out[i]);
  p->ready = ok;
  return ok;
}

bool copy(void* dst, const void* src, size_t bytes, cudaMemcpyKind kind, cudaStream_t s) {
  return bytes == 0 || cudaMemcpyAsync(dst, src, bytes, kind, s) == cudaSuccess;
}

// After a failure midway through an enqueue: copies from or to the caller's host
// arrays may already be queued on the internal streams.  Order the caller's stream
// after all of them (best effort: a call that fails here too is skipped), so that
// synchronising `caller` still means the library no longer touches those arrays.
void drain_into(Pipe& p, cudaStream_t caller) {
  cudaStream_t tails[1 + kComputeStreams] = {p.h2d};
  for (int i = 0; i < kComputeStreams; ++i) tails[1 + i] = p.comp[i];
  for (int i = 0; i < 1 + kComputeStreams; ++i)
    if (cudaEventRecord(p.drain[i], tails[i]) == cudaSuccess) cudaStreamWaitEvent(p.d2h, p.drain[i], 0);
  if (cudaEventRecord(p.end, p.d2h) == cudaSuccess) cudaStreamWaitEvent(caller, p.end, 0);
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

int fa_fwd_bwd_host_chunk_heads(int B, int H, int Nq, int Nk, int d, int heads_per_chunk) {
  bool empty = false;
  if (heads_per_chunk < 0 || check_mask_shape(B, H, Nq, Nk, d, 0, 0, &empty) != FA_OK) return -1;
  return chunk_heads(B * H, Nq, Nk, heads_per_chunk);
}

size_t fa_fwd_bwd_host_workspace_size(int B, int H, int Nq, int Nk, int d, int causal, int window,
                                      int heads_per_chunk) {
  bool empty = false;
  if (heads_per_chunk < 0 || check_mask_shape(B, H, Nq, Nk, d, causal, window, &empty) != FA_OK)
    return static_cast<size_t>(-1);
  return make_plan(B * H, Nq, Nk, d, causal, window, heads_per_chunk).total;
}

fa_status fa_fwd_bwd_host(const void* Q, const void* K, const void* V, const void* dO, void* O, float* L, void* dQ,
                          void* dK, void* dV, int B, int H, int Nq, int Nk, int d, int causal, int window, float scale,
                          int heads_per_chunk, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  bool empty = false;
  fa_status st = check_mask_shape(B, H, Nq, Nk, d, causal, window, &empty);
  if (st != FA_OK) return st;
  if (heads_per_chunk < 0 || !check_scale(scale)) return FA_ERR_INVALID_ARG;
  const int BH = B * H;
  if (BH == 0) return FA_OK;
  const size_t nq = static_cast<size_t>(Nq) * d, nk = static_cast<size_t>(Nk) * d;  // elements per head
  if (Nq > 0 && (!Q || !dO || !O || !L || !dQ)) return FA_ERR_INVALID_ARG;
  if (Nk > 0 && (!K || !V || !dK || !dV)) return FA_ERR_INVALID_ARG;
  const Plan p = make_plan(BH, Nq, Nk, d, causal, window, heads_per_chunk);
  if (p.total > 0 && (workspace == nullptr || workspace_bytes < p.total ||
                      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0))
    return FA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;

  std::lock_guard<std::mutex> lk(g_pipe_mu);
  Pipe& pp = g_pipe[dev];
  if (!make_pipe(&pp)) return FA_ERR_CUDA;
  auto* ws = static_cast<char*>(workspace);
  auto* acc = ws + p.slot.bytes * p.slots;
  const auto* hQ = static_cast<const char*>(Q);
  const auto* hK = static_cast<const char*>(K);
  const auto* hV = static_cast<const char*>(V);
  const auto* hdO = static_cast<const char*>(dO);
  auto* hO = static_cast<char*>(O);
  auto* hL = reinterpret_cast<char*>(L);
  auto* hdQ = static_cast<char*>(dQ);
  auto* hdK = static_cast<char*>(dK);
  auto* hdV = static_cast<char*>(dV);

  // every internal stream starts after the caller's earlier work
  if (cudaEventRecord(pp.start, stream) != cudaSuccess) return FA_ERR_CUDA;
  bool ok = cudaStreamWaitEvent(pp.h2d, pp.start, 0) == cudaSuccess && cudaStreamWaitEvent(pp.d2h, pp.start, 0) == cudaSuccess;
  for (int i = 0; ok && i < p.streams; ++i) ok = cudaStreamWaitEvent(pp.comp[i], pp.start, 0) == cudaSuccess;
  if (!ok) return FA_ERR_CUDA;

  // from here on part of the step may be enqueued: an error leaves the caller's
  // stream ordered after whatever was
  auto fail = [&](fa_status e) {
    drain_into(pp, stream);
    return e;
  };
  for (int c = 0; c < p.chunks; ++c) {
    const int h0 = c * p.hc, hn = (BH - h0) < p.hc ? (BH - h0) : p.hc;
    const int slot = c % p.slots;
    cudaStream_t cs = pp.comp[c % p.streams];
    char* sb = ws + p.slot.bytes * slot;
    const size_t bq = nq * 2 * hn, bk = nk * 2 * hn, bl = static_cast<size_t>(Nq) * 4 * hn;
    const size_t off_q = nq * 2 * h0, off_k = nk * 2 * h0, off_l = static_cast<size_t>(Nq) * 4 * h0;
    // in: this slot's inputs were last read by the chunk `slots` earlier.  Q, K, V
    // first (the forward needs only those), then dO.
    ok = (c < p.slots || cudaStreamWaitEvent(pp.h2d, pp.done[slot], 0) == cudaSuccess) &&
         copy(sb + p.slot.q, hQ + off_q, bq, cudaMemcpyHostToDevice, pp.h2d) &&
         copy(sb + p.slot.k, hK + off_k, bk, cudaMemcpyHostToDevice, pp.h2d) &&
         copy(sb + p.slot.v, hV + off_k, bk, cudaMemcpyHostToDevice, pp.h2d) &&
         cudaEventRecord(pp.in_qkv[slot], pp.h2d) == cudaSuccess &&
         copy(sb + p.slot.dO, hdO + off_q, bq, cudaMemcpyHostToDevice, pp.h2d) &&
         cudaEventRecord(pp.in[slot], pp.h2d) == cudaSuccess;
    if (!ok) return fail(FA_ERR_CUDA);
    // compute: the forward after Q, K, V arrived and the slot's previous outputs
    // left; the backward after dO arrived
    if (cudaStreamWaitEvent(cs, pp.in_qkv[slot], 0) != cudaSuccess ||
        (c >= p.slots && cudaStreamWaitEvent(cs, pp.out[slot], 0) != cudaSuccess))
      return fail(FA_ERR_CUDA);
    st = fa_fwd_ex(sb + p.slot.q, sb + p.slot.k, sb + p.slot.v, sb + p.slot.o, reinterpret_cast<float*>(sb + p.slot.L),
                   1, hn, Nq, Nk, d, causal, window, scale, cs);
    if (st != FA_OK) return fail(st);
    if (cudaEventRecord(pp.fwd[slot], cs) != cudaSuccess || cudaStreamWaitEvent(cs, pp.in[slot], 0) != cudaSuccess)
      return fail(FA_ERR_CUDA);
    st = fa_bwd_preprocess(sb + p.slot.o, sb + p.slot.dO, reinterpret_cast<float*>(sb + p.slot.D), 1, hn, Nq, d, cs);
    if (st != FA_OK) return fail(st);
    st = fa_bwd_ex(sb + p.slot.q, sb + p.slot.k, sb + p.slot.v, sb + p.slot.o, sb + p.slot.dO,
                   reinterpret_cast<const float*>(sb + p.slot.L), reinterpret_cast<const float*>(sb + p.slot.D),
                   sb + p.slot.dQ, sb + p.slot.dK, sb + p.slot.dV, 1, hn, Nq, Nk, d, causal, window, scale,
                   acc + p.acc_bytes * (c % p.streams), p.acc_bytes, cs);
    if (st != FA_OK) return fail(st);
    if (cudaEventRecord(pp.done[slot], cs) != cudaSuccess) return fail(FA_ERR_CUDA);
    // out: O and L once the forward is done, the gradients once the backward is
    ok = cudaStreamWaitEvent(pp.d2h, pp.fwd[slot], 0) == cudaSuccess &&
         copy(hO + off_q, sb + p.slot.o, bq, cudaMemcpyDeviceToHost, pp.d2h) &&
         copy(hL + off_l, sb + p.slot.L, bl, cudaMemcpyDeviceToHost, pp.d2h) &&
         cudaStreamWaitEvent(pp.d2h, pp.done[slot], 0) == cudaSuccess &&
         copy(hdQ + off_q, sb + p.slot.dQ, bq, cudaMemcpyDeviceToHost, pp.d2h) &&
         copy(hdK + off_k, sb + p.slot.dK, bk, cudaMemcpyDeviceToHost, pp.d2h) &&
         copy(hdV + off_k, sb + p.slot.dV, bk, cudaMemcpyDeviceToHost, pp.d2h) &&
         cudaEventRecord(pp.out[slot], pp.d2h) == cudaSuccess;
    if (!ok) return fail(FA_ERR_CUDA);
  }
  // every chunk's copy out follows its compute, which follows its copy in: the
  // copy-out stream's last event covers the whole step
  if (cudaEventRecord(pp.end, pp.d2h) != cudaSuccess || cudaStreamWaitEvent(stream, pp.end, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // extern "C"
