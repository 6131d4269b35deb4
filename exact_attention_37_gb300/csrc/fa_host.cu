// Host-buffer entry points: the attention step with its inputs and outputs in
// host memory, pipelined over chunks of heads on three library-owned streams so
// that the host-to-device copies of chunk c + 1, the kernels of chunk c and the
// device-to-host copies of chunk c - 1 overlap.  Within a chunk the forward pass
// starts once Q, K and V are on the device (dO follows); O and L go back as soon
// as the forward pass has written them, and dK and dV as soon as the kernel that
// writes them has run (while the dQ kernel runs), so the pipeline's fill and
// drain carry only part of a chunk's copies.  Heads are independent in both
// passes, so a chunk of heads is a complete problem of its own; each chunk runs
// through fa_fwd_ex / fa_bwd_ex on a slice of one device scratch region that
// the caller provides (the library allocates no device memory).
#include <algorithm>
#include <mutex>
#include <vector>

#include "../../include/fa_attention.h"
#include "fa_internal.h"
#include "fa_marks.h"
#include "fa_nvtx.h"

namespace fa {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 64;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Offsets of the tensors inside the device scratch (each 256-byte aligned).
struct ScratchLayout {
  size_t q, k, v, dout, o, lse, dq, dk, dv, ws, ws_bytes, total;
};

ScratchLayout layout(long long BH, int N, int d, bool bwd, int max_chunk_heads) {
  const size_t t = (size_t)BH * N * d * 2;  // one [B*H, N, d] 16-bit tensor
  ScratchLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  L.q = take(t);
  L.k = take(t);
  L.v = take(t);
  L.o = take(t);
  L.lse = take((size_t)BH * N * 4);
  if (bwd) {
    L.dout = take(t);
    L.dq = take(t);
    L.dk = take(t);
    L.dv = take(t);
    // The chunks' kernels run one after another on one stream, so a workspace
    // sized for the largest chunk serves them all.
    L.ws_bytes = fa_bwd_workspace_size(1, max_chunk_heads, N, d);
    L.ws = take(L.ws_bytes);
  }
  L.total = off;
  return L;
}

// Library-owned streams and events of one device, created on first use.
struct Pipeline {
  cudaStream_t up = nullptr, comp = nullptr, down = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t qkv_up[kMaxChunks] = {}, dout_up[kMaxChunks] = {};
  cudaEvent_t fwd_done[kMaxChunks] = {}, dkdv_done[kMaxChunks] = {}, comp_done[kMaxChunks] = {};
  bool ready = false;
};

std::mutex g_mu;
Pipeline g_pipe[kMaxDevices];

bool pipeline_for_device(Pipeline** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  Pipeline& p = g_pipe[dev];
  if (!p.ready) {
    const unsigned sf = cudaStreamNonBlocking;
    const unsigned ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.up, sf) != cudaSuccess || cudaStreamCreateWithFlags(&p.comp, sf) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.down, sf) != cudaSuccess || cudaEventCreateWithFlags(&p.start, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.end, ef) != cudaSuccess)
      return false;
    for (int c = 0; c < kMaxChunks; ++c)
      if (cudaEventCreateWithFlags(&p.qkv_up[c], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.dout_up[c], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.fwd_done[c], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.dkdv_done[c], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.comp_done[c], ef) != cudaSuccess)
        return false;
    p.ready = true;
  }
  *out = &p;
  return true;
}

// Heads per chunk.  An explicit count gives equal chunks (the last may be
// smaller); the default (chunks <= 0) gives middle chunks of about B*H / 4 heads
// with first and last chunks of half that, so the pipeline's fill (the first
// upload) and drain (the last download) are short.  Every chunk but the last is a
// multiple of `align` heads.  Returns the number of chunks.
int chunk_plan(long long BH, int chunks, int align, int (&plan)[kMaxChunks]) {
  auto up = [&](long long x) { return std::max<long long>(align, (x + align - 1) / align * align); };
  auto down = [&](long long x) { return std::max<long long>(align, x / align * align); };
  long long mid, first;
  if (chunks > 0) {
    chunks = (int)std::min<long long>(std::min(chunks, kMaxChunks), BH);
    mid = first = up((BH + chunks - 1) / chunks);
  } else {
    mid = up((BH + 3) / 4);
    first = up(mid / 2);
  }
  int n = 0;
  long long h = 0;
  while (h < BH && n < kMaxChunks - 1) {
    long long c = n == 0 ? first : mid;
    // Default plan: when what would remain after this chunk is shorter than a
    // first chunk, take less now (still a multiple of `align`), so the last chunk
    // stays about as short as the first.
    if (chunks <= 0 && BH - h - c < first && BH - h - c > 0) c = down(BH - h - first);
    c = std::min(c, BH - h);  // only the last chunk can be cut short here
    plan[n++] = (int)c;
    h += c;
  }
  if (h < BH) plan[n++] = (int)(BH - h);
  return n;
}

fa_status enqueue_chunks(Pipeline* P, const ScratchLayout& L, char* s, const void* q, const void* k, const void* v,
                         const void* dout, void* o, float* lse, void* dq, void* dk, void* dv, const int* plan,
                         int chunks, int N, int d, float scale, int causal, fa_dtype dtype, bool bwd);

fa_status run_host(const void* q, const void* k, const void* v, const void* dout, void* o, float* lse, void* dq,
                   void* dk, void* dv, void* scratch, size_t scratch_bytes, int B, int H, int N, int d, float scale,
                   int causal, fa_dtype dtype, int chunks, fa_stream_t stream, bool bwd) {
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  const long long BH = (long long)B * H;
  if (BH * N == 0) return FA_OK;
  if (!q || !k || !v || !o || !lse || (bwd && (!dout || !dq || !dk || !dv))) return FA_ERR_INVALID_ARG;
  // Each chunk's L starts on a 16-byte boundary: chunk starts are multiples of m
  // heads with m * N a multiple of 4.
  const int m = N % 4 == 0 ? 1 : (N % 2 == 0 ? 2 : 4);
  int plan[kMaxChunks];
  chunks = chunk_plan(BH, chunks, m, plan);
  int per = 0;  // heads of the largest chunk
  for (int c = 0; c < chunks; ++c) per = std::max(per, plan[c]);
  const size_t need = fa_host_scratch_size(B, H, N, d, bwd ? 1 : 0);
  if (need == 0) return FA_ERR_INVALID_ARG;  // invalid sizes (d, limits)
  if (!scratch || scratch_bytes < need) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(scratch) & 255u) != 0) return FA_ERR_MISALIGNED;

  std::lock_guard<std::mutex> lock(g_mu);
  Pipeline* P = nullptr;
  if (!pipeline_for_device(&P)) return FA_ERR_CUDA;
  const ScratchLayout L = layout(BH, N, d, bwd, per);
  char* s = static_cast<char*>(scratch);
  cudaStream_t caller = reinterpret_cast<cudaStream_t>(stream);
  // Everything starts after the work already queued on the caller's stream.
  if (cudaEventRecord(P->start, caller) != cudaSuccess || cudaStreamWaitEvent(P->up, P->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(P->comp, P->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(P->down, P->start, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  fa_status st = enqueue_chunks(P, L, s, q, k, v, dout, o, lse, dq, dk, dv, plan, chunks, N, d, scale, causal,
                                dtype, bwd);
  // The caller's stream continues after everything enqueued (also after a failure
  // part-way, so no copy is still in flight when the caller's stream moves on).
  // (The event is re-recorded in turn: each wait captures its state at the call.)
  if (cudaEventRecord(P->end, P->up) != cudaSuccess || cudaStreamWaitEvent(P->comp, P->end, 0) != cudaSuccess ||
      cudaEventRecord(P->end, P->comp) != cudaSuccess || cudaStreamWaitEvent(P->down, P->end, 0) != cudaSuccess ||
      cudaEventRecord(P->end, P->down) != cudaSuccess || cudaStreamWaitEvent(caller, P->end, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  return st;
}

fa_status enqueue_chunks(Pipeline* P, const ScratchLayout& L, char* s, const void* q, const void* k, const void* v,
                         const void* dout, void* o, float* lse, void* dq, void* dk, void* dv, const int* plan,
                         int chunks, int N, int d, float scale, int causal, fa_dtype dtype, bool bwd) {
  const size_t head_t = (size_t)N * d * 2;  // bytes of one head of a 16-bit tensor
  const size_t head_l = (size_t)N * 4;      // bytes of one head of L
  auto H2D = [&](size_t dev_off, const void* host, size_t off, size_t bytes) {
    return cudaMemcpyAsync(s + dev_off + off, static_cast<const char*>(host) + off, bytes, cudaMemcpyHostToDevice,
                           P->up) == cudaSuccess;
  };
  auto D2H = [&](void* host, size_t dev_off, size_t off, size_t bytes) {
    return cudaMemcpyAsync(static_cast<char*>(host) + off, s + dev_off + off, bytes, cudaMemcpyDeviceToHost,
                           P->down) == cudaSuccess;
  };
  long long h0 = 0;
  for (int c = 0; c < chunks; h0 += plan[c++]) {
    const int hc = plan[c];
    const size_t ot = (size_t)h0 * head_t, bt = (size_t)hc * head_t;
    const size_t ol = (size_t)h0 * head_l, bl = (size_t)hc * head_l;
    // ---- upload: Q, K, V, then dO (needed only by the backward pass)
    if (!H2D(L.q, q, ot, bt) || !H2D(L.k, k, ot, bt) || !H2D(L.v, v, ot, bt)) return FA_ERR_CUDA;
    if (cudaEventRecord(P->qkv_up[c], P->up) != cudaSuccess) return FA_ERR_CUDA;
    if (bwd && (!H2D(L.dout, dout, ot, bt) || cudaEventRecord(P->dout_up[c], P->up) != cudaSuccess))
      return FA_ERR_CUDA;
    // ---- compute (one chunk of heads is a problem with B = 1, H = hc)
    if (cudaStreamWaitEvent(P->comp, P->qkv_up[c], 0) != cudaSuccess) return FA_ERR_CUDA;
    fa_stream_t cs = reinterpret_cast<fa_stream_t>(P->comp);
    fa_status st = fa_fwd_ex(s + L.q + ot, s + L.k + ot, s + L.v + ot, s + L.o + ot,
                             reinterpret_cast<float*>(s + L.lse + ol), 1, hc, hc, N, N, d, scale, causal, dtype, cs);
    if (st != FA_OK) return st;
    if (cudaEventRecord(P->fwd_done[c], P->comp) != cudaSuccess) return FA_ERR_CUDA;
    if (bwd) {
      if (cudaStreamWaitEvent(P->comp, P->dout_up[c], 0) != cudaSuccess) return FA_ERR_CUDA;
      arm_dkdv_mark(P->dkdv_done[c]);  // recorded right after the kernel that writes dK and dV
      st = fa_bwd_ex(s + L.q + ot, s + L.k + ot, s + L.v + ot, s + L.o + ot, s + L.dout + ot,
                     reinterpret_cast<const float*>(s + L.lse + ol), s + L.dq + ot, s + L.dk + ot, s + L.dv + ot,
                     s + L.ws, L.ws_bytes, 1, hc, hc, N, N, d, scale, causal, dtype, cs);
      const bool marked = take_dkdv_mark();
      if (st != FA_OK) return st;
      if (cudaEventRecord(P->comp_done[c], P->comp) != cudaSuccess) return FA_ERR_CUDA;
      if (!marked && cudaEventRecord(P->dkdv_done[c], P->comp) != cudaSuccess) return FA_ERR_CUDA;
    }
    // ---- download: O and L once the forward pass has written them, dK and dV once
    // their kernel has run, then dQ
    if (cudaStreamWaitEvent(P->down, P->fwd_done[c], 0) != cudaSuccess) return FA_ERR_CUDA;
    if (!D2H(o, L.o, ot, bt) || !D2H(lse, L.lse, ol, bl)) return FA_ERR_CUDA;
    if (bwd && (cudaStreamWaitEvent(P->down, P->dkdv_done[c], 0) != cudaSuccess || !D2H(dk, L.dk, ot, bt) ||
                !D2H(dv, L.dv, ot, bt) || cudaStreamWaitEvent(P->down, P->comp_done[c], 0) != cudaSuccess ||
                !D2H(dq, L.dq, ot, bt)))
      return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

int fa_host_chunk_plan(int B, int H, int N, int chunks, int* plan, int capacity) {
  if (B < 0 || H < 0 || N < 0 || capacity < 0) return -1;
  const long long BH = (long long)B * H;
  if (BH * N == 0) return 0;
  const int m = N % 4 == 0 ? 1 : (N % 2 == 0 ? 2 : 4);
  int p[kMaxChunks];
  const int n = chunk_plan(BH, chunks, m, p);
  if (plan && capacity >= n)
    for (int c = 0; c < n; ++c) plan[c] = p[c];
  return n;
}

size_t fa_host_scratch_size(int B, int H, int N, int d, int with_backward) {
  if (B < 0 || H < 0 || N < 0 || (d != 64 && d != 128 && d != 256)) return 0;
  const long long BH = (long long)B * H;
  if (BH * N == 0) return 0;
  if (with_backward && fa_bwd_workspace_size(1, (int)std::min<long long>(BH, 1 << 24), N, d) == 0) return 0;
  return layout(BH, N, d, with_backward != 0, (int)std::min<long long>(BH, 1 << 24)).total;
}

fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, void* dev_scratch,
                      size_t scratch_bytes, int B, int H, int N, int d, float scale, int causal, fa_dtype dtype,
                      int chunks, fa_stream_t stream) {
  const fa::NvtxRange range("fa_fwd_host");
  return run_host(q, k, v, nullptr, o, lse, nullptr, nullptr, nullptr, dev_scratch, scratch_bytes, B, H, N, d,
                  scale, causal, dtype, chunks, stream, false);
}

fa_status fa_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dout, void* o, float* lse,
                          void* dq, void* dk, void* dv, void* dev_scratch, size_t scratch_bytes, int B, int H, int N,
                          int d, float scale, int causal, fa_dtype dtype, int chunks, fa_stream_t stream) {
  const fa::NvtxRange range("fa_fwd_bwd_host");
  return run_host(q, k, v, dout, o, lse, dq, dk, dv, dev_scratch, scratch_bytes, B, H, N, d, scale, causal, dtype,
                  chunks, stream, true);
}

}  // extern "C"
