// C-ABI entry points of the exact-attention library (declared in include/fa_attention.h).
//
// This layer validates arguments on the host (nothing is launched for a bad
// call), encodes the TMA descriptors of the [B*H, N, d] tensors, lays out the
// backward workspace, and owns the device error word that the kernels' bounded
// waits write.  It allocates no device memory.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/fa_attention.h"
#include "fa_internal.h"
#include "fa_marks.h"
#include "fa_nvtx.h"
#include "ptx.cuh"

namespace fa {

// Device error record the kernels write when a bounded wait gives up (one per
// device that loads the library): bits, first failure code, its CTA, its barrier.
__device__ uint32_t g_error_word[4];

namespace {

constexpr int kMaxDevices = 64;
uint32_t g_last_detail[4] = {0, 0, 0, 0};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// The current CUDA context (driver API, looked up through the runtime's entry-point
// query so the library needs no link against libcuda), or nullptr.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  CUcontext c = nullptr;
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

// Device address of a __device__ symbol on the current device, cached per device
// and keyed on the device's current context: after cudaDeviceReset (a new primary
// context) the address is looked up again instead of reusing a stale one.
struct SymbolCache {
  std::mutex mu;
  CUcontext ctx[kMaxDevices] = {};
  void* ptr[kMaxDevices] = {};
  void* get(const void* symbol) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    // (before the first runtime call on a thread no context may be current yet: the
    // lookup below makes it current, and the next call re-keys the cache once)
    const CUcontext c = current_context();
    std::lock_guard<std::mutex> lock(mu);
    if (!ptr[dev] || c != ctx[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess) return nullptr;
      ptr[dev] = p;
      ctx[dev] = c;
    }
    return ptr[dev];
  }
};

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  return sms > 0 ? sms : 1;
}

// Address of the error word on the current device.
uint32_t* error_word_ptr() {
  static SymbolCache cache;
  return static_cast<uint32_t*>(cache.get(g_error_word));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks shared by both passes.  Returns FA_OK or the first problem found.
fa_status check_common(int B, int H, int H_kv, int Nq, int Nk, int d, float scale, int dtype) {
  if (B < 0 || H < 0 || H_kv < 0 || Nq < 0 || Nk < 0) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (H > 0 && (H_kv < 1 || H % H_kv != 0)) return FA_ERR_INVALID_ARG;
  const long long BH = (long long)B * H;
  // grid size and 32-bit index limits of the kernels
  if (BH > (1LL << 24) || Nq > (1 << 28) || Nk > (1 << 28)) return FA_ERR_UNSUPPORTED;
  if (BH * ((Nq + 127) / 128) * 2 > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if ((long long)B * H_kv * ((Nk + 127) / 128) * 2 > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  // the d = 256 backward launches both kinds of CTA in one grid
  if (BH * ((Nq + 127) / 128) + (long long)B * H_kv * ((Nk + 127) / 128) * 2 > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  // Queries with an empty key set are not a supported problem.
  if (BH * Nq > 0 && Nk == 0) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

fa_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return FA_ERR_CUDA;
  if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;  // the kernels are built for sm_103a only
  return FA_OK;
}

// TMA descriptor of a [BH, N, d] 16-bit tensor read or written in boxes of
// 64 columns (128 B, 128-byte swizzle) x `box_rows` rows of one head.
bool make_map(CUtensorMap* m, const void* ptr, long long BH, int N, int d, bool bf16, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

constexpr float kLog2e = 1.4426950408889634f;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Library-owned events for the measurement hook.
struct Profile {
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev;
  std::vector<int> kind;
  int used = 0;
  bool on = false;
  bool open = false;  // a begin mark is waiting for its end mark
  void release() {
    for (auto& e : ev) {
      if (e.first) cudaEventDestroy(e.first);
      if (e.second) cudaEventDestroy(e.second);
    }
    ev.clear();
    kind.clear();
    used = 0;
    on = false;
    open = false;
  }
};
Profile& profile() {
  static Profile p;
  return p;
}

}  // namespace

void profile_mark_begin(cudaStream_t stream) {
  Profile& p = profile();
  if (!p.on || p.used >= (int)p.ev.size()) return;
  if (cudaEventRecord(p.ev[p.used].first, stream) == cudaSuccess) p.open = true;
}

namespace {
// The host-buffer pipeline's dK/dV mark (one per thread: calls on other threads
// are not affected).
thread_local cudaEvent_t t_dkdv_mark = nullptr;
thread_local bool t_dkdv_recorded = false;
}  // namespace

void arm_dkdv_mark(cudaEvent_t ev) {
  t_dkdv_mark = ev;
  t_dkdv_recorded = false;
}

bool take_dkdv_mark() {
  const bool r = t_dkdv_recorded;
  t_dkdv_mark = nullptr;
  t_dkdv_recorded = false;
  return r;
}

void profile_mark_end(cudaStream_t stream, int kind) {
  if (t_dkdv_mark && (kind == kProfileBwdKV || kind == kProfileBwdFused)) {
    t_dkdv_recorded = cudaEventRecord(t_dkdv_mark, stream) == cudaSuccess;
    t_dkdv_mark = nullptr;
  }
  Profile& p = profile();
  if (!p.on || !p.open) return;
  p.open = false;
  if (cudaEventRecord(p.ev[p.used].second, stream) == cudaSuccess) p.kind[p.used++] = kind;
}

size_t bwd_delta_offset(long long BH, int N) { return round_up((size_t)BH * bwd_npad(N) * sizeof(float), 256); }
size_t bwd_workspace_bytes(long long BH, int N) {
  return bwd_delta_offset(BH, N) + round_up((size_t)BH * bwd_npad(N) * sizeof(float), 256);
}

}  // namespace fa

using namespace fa;

namespace fa {

// cta_head_group for a given number of SMs (also the host query fa_cta_head_group).
static int cta_head_group_for(long long nheads, int nblocks, size_t bytes_per_head, bool causal, int num_sms) {
  if (nheads <= 1 || nblocks <= 0) return 1;
  const long long sms = std::max(num_sms, 1);
  const long long nb = nblocks;
  const long long work = causal ? nb * (nb + 1) / 2 : nb * nb;  // steps per head; the longest CTA takes nb
  const long long g_tail = (sms * nb + work - 1) / work;
  const long long g_l2 = std::max<long long>(1, (48ll << 20) / (long long)std::max<size_t>(bytes_per_head, 1));
  const long long g = std::min(std::max(g_tail, g_l2), nheads);
  // Equal groups: a short last group would hold heavy CTAs with too little work
  // around them.  Take the smallest divisor of nheads in [g, 2g] if there is one.
  for (long long c = g; c <= std::min(2 * g, nheads); ++c)
    if (nheads % c == 0) return (int)c;
  return (int)g;
}

int cta_head_group(long long nheads, int nblocks, size_t bytes_per_head, bool causal) {
  return cta_head_group_for(nheads, nblocks, bytes_per_head, causal, sm_count());
}

}  // namespace fa

extern "C" {

fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv,
                    int N_q, int N_k, int d, float scale, int causal, fa_dtype dtype, fa_stream_t stream) {
  const fa::NvtxRange range("fa_fwd_ex");
  fa_status st = check_common(B, H, H_kv, N_q, N_k, d, scale, (int)dtype);
  if (st != FA_OK) return st;
  if ((long long)B * H * N_q == 0) return FA_OK;  // empty problem
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_MISALIGNED;
  if ((st = check_device()) != FA_OK) return st;
  const bool bf16 = dtype == FA_BF16;
  const long long BH = (long long)B * H, BHkv = (long long)B * H_kv;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, q, BH, N_q, d, bf16, 128) || !make_map(&mk, k, BHkv, N_k, d, bf16, 128) ||
      !make_map(&mv, v, BHkv, N_k, d, bf16, 128) || !make_map(&mo, o, BH, N_q, d, bf16, 128))
    return FA_ERR_CUDA;
  FwdArgs a{};
  a.lse = lse;
  a.N = N_q;
  a.Nk = N_k;
  a.BH = (int)BH;
  a.H = H;
  a.group = H / H_kv;
  const int rows = fwd_rows_per_cta(d, BH, N_q, sm_count());
  a.num_qblocks = (N_q + rows - 1) / rows;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.causal = causal ? 1 : 0;
  a.head_group = cta_head_group(BH, a.num_qblocks, (size_t)4 * (N_q + N_k) * d, causal != 0);
  a.err = error_word_ptr();
  if (!a.err) return FA_ERR_CUDA;
  cudaError_t e = launch_fwd(d, bf16, rows, mq, mk, mv, mo, a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, fa_dtype dtype, fa_stream_t stream) {
  return fa_fwd_ex(q, k, v, o, lse, B, H, H, N, N, d, scale, causal, dtype, stream);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (check_common(B, H, H > 0 ? 1 : 0, N, N, d, 1.f, FA_FP16) != FA_OK) return 0;
  if ((size_t)B * H * N == 0) return 0;
  return bwd_workspace_bytes((long long)B * H, N);
}

fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                    void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int H_kv,
                    int N_q, int N_k, int d, float scale, int causal, fa_dtype dtype, fa_stream_t stream) {
  const fa::NvtxRange range("fa_bwd_ex");
  fa_status st = check_common(B, H, H_kv, N_q, N_k, d, scale, (int)dtype);
  if (st != FA_OK) return st;
  if ((long long)B * H * N_q == 0) {
    // No query rows: nothing flows back, so dK = dV = 0.
    const size_t kv_bytes = (size_t)B * H_kv * N_k * d * 2;
    if (kv_bytes == 0) return FA_OK;
    if (!dk || !dv) return FA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(dk, 0, kv_bytes, s) != cudaSuccess || cudaMemsetAsync(dv, 0, kv_bytes, s) != cudaSuccess)
      return FA_ERR_CUDA;
    return FA_OK;
  }
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_MISALIGNED;
  const size_t need = fa_bwd_workspace_size(B, H, N_q, d);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_MISALIGNED;
  if ((st = check_device()) != FA_OK) return st;
  const bool bf16 = dtype == FA_BF16;
  const long long BH = (long long)B * H, BHkv = (long long)B * H_kv;
  const int rows = bwd_box_rows(d);
  CUtensorMap mq, mk, mv, mdo;
  if (!make_map(&mq, q, BH, N_q, d, bf16, rows) || !make_map(&mk, k, BHkv, N_k, d, bf16, rows) ||
      !make_map(&mv, v, BHkv, N_k, d, bf16, rows) || !make_map(&mdo, dout, BH, N_q, d, bf16, rows))
    return FA_ERR_CUDA;
  BwdArgs a{};
  a.q = q;
  a.k = k;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.lse_log2 = static_cast<float*>(workspace);
  a.delta = reinterpret_cast<float*>(static_cast<char*>(workspace) + bwd_delta_offset(BH, N_q));
  a.Npad = bwd_npad(N_q);
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.N = N_q;
  a.Nk = N_k;
  a.d = d;
  a.BH = (int)BH;
  a.BHkv = (int)BHkv;
  a.H = H;
  a.group = H / H_kv;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.causal = causal ? 1 : 0;
  a.head_group_kv = cta_head_group(BHkv, (N_k + 127) / 128, (size_t)4 * ((size_t)a.group * N_q + N_k) * d, causal != 0);
  a.head_group_q = cta_head_group(BH, (N_q + 127) / 128, (size_t)4 * (N_q + N_k) * d, causal != 0);
  a.err = error_word_ptr();
  if (!a.err) return FA_ERR_CUDA;
  cudaError_t e = launch_bwd(d, bf16, mq, mk, mv, mdo, a, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                 float scale, int causal, fa_dtype dtype, fa_stream_t stream) {
  return fa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, H, N, N, d, scale, causal,
                   dtype, stream);
}

}  // extern "C"

namespace fa {
namespace {
// Fixed scratch of fa_bwd_noalloc (the backward workspace: fp32 L log2 e and D
// rows).  Its name in host code is only a host-side stand-in; the device address
// comes from cudaGetSymbolAddress on each device.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch on the current device.
void* noalloc_scratch_ptr() {
  static SymbolCache cache;
  return cache.get(g_noalloc_scratch);
}
}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                         int causal, fa_dtype dtype, fa_stream_t stream) {
  const fa::NvtxRange range("fa_bwd_noalloc");
  fa_status st = check_common(B, H, H, N, N, d, scale, (int)dtype);
  if (st != FA_OK) return st;
  if ((long long)B * H * N == 0) return FA_OK;
  if (fa_bwd_workspace_size(B, H, N, d) > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if ((st = check_device()) != FA_OK) return st;
  void* scratch = noalloc_scratch_ptr();
  if (!scratch) return FA_ERR_CUDA;
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch, kNoAllocScratchBytes, B, H, N, d, scale, causal, dtype,
                stream);
}

int fa_cta_head_group(long long nheads, int nblocks, size_t bytes_per_head, int causal, int num_sms) {
  if (nheads < 1 || nblocks < 0) return -1;
  return cta_head_group_for(nheads, nblocks, bytes_per_head, causal != 0, num_sms > 0 ? num_sms : sm_count());
}

fa_status fa_check_device_status(fa_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  uint32_t rec[4] = {0, 0, 0, 0};
  if (cudaMemcpyFromSymbol(rec, g_error_word, sizeof(rec)) != cudaSuccess) return FA_ERR_CUDA;
  for (int i = 0; i < 4; ++i) g_last_detail[i] = rec[i];
  if (rec[0] != 0) {
    const uint32_t zero[4] = {0, 0, 0, 0};
    if (cudaMemcpyToSymbol(g_error_word, zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
    // the first failure decides: a debug-build check (code kDbgBase | kind) or a wait
    return (rec[1] & kDbgBase) ? FA_ERR_DEVICE_CHECK : FA_ERR_DEVICE_TIMEOUT;
  }
  return FA_OK;
}

fa_status fa_selftest_device_check(int kind, fa_stream_t stream) {
#ifdef FA_DEBUG
  if (kind < (int)kDbgTmaCol || kind > (int)kDbgPhase) return FA_ERR_INVALID_ARG;
  fa_status st = check_device();
  if (st != FA_OK) return st;
  uint32_t* err = error_word_ptr();
  if (!err) return FA_ERR_CUDA;
  return launch_selftest_check(err, kind, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                                  : FA_ERR_CUDA;
#else
  (void)kind;
  (void)stream;
  return FA_ERR_UNSUPPORTED;  // the checks are compiled out of this build
#endif
}

fa_status fa_selftest_wait_timeout(uint32_t limit_us, fa_stream_t stream) {
  if (limit_us == 0 || limit_us > 1000000u) return FA_ERR_INVALID_ARG;
  fa_status st = check_device();
  if (st != FA_OK) return st;
  uint32_t* err = error_word_ptr();
  if (!err) return FA_ERR_CUDA;
  return launch_selftest_wait(err, 1000ull * limit_us, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

uint32_t fa_last_device_error_bits(void) { return g_last_detail[0]; }

void fa_last_device_error_detail(uint32_t* out4) {
  if (!out4) return;
  for (int i = 0; i < 4; ++i) out4[i] = g_last_detail[i];
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
    case FA_ERR_DEVICE_CHECK: return "FA_ERR_DEVICE_CHECK";
  }
  return "FA_ERR_UNKNOWN";
}

fa_status fa_profile_begin(int n) {
  if (n < 0 || n > 65536) return FA_ERR_INVALID_ARG;
  Profile& p = profile();
  p.release();
  p.ev.resize((size_t)n);
  p.kind.assign((size_t)n, 0);
  for (auto& e : p.ev) {
    if (cudaEventCreate(&e.first) != cudaSuccess || cudaEventCreate(&e.second) != cudaSuccess) {
      p.release();
      return FA_ERR_CUDA;
    }
  }
  p.used = 0;
  p.open = false;
  p.on = n > 0;
  return FA_OK;
}

int fa_profile_end(float* out_ms, int* out_kind, int max_out) {
  Profile& p = profile();
  int written = 0;
  bool failed = false;
  for (int i = 0; i < p.used && i < max_out; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.ev[i].second) != cudaSuccess ||
        cudaEventElapsedTime(&ms, p.ev[i].first, p.ev[i].second) != cudaSuccess) {
      failed = true;
      break;
    }
    if (out_ms) out_ms[i] = ms;
    if (out_kind) out_kind[i] = p.kind[i];
    ++written;
  }
  p.release();
  return failed ? -1 : written;
}

uint32_t fa_version(void) { return (1u << 16) | 0u; }

}  // extern "C"
