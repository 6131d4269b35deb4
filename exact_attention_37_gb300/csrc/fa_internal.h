// Host-side declarations shared by the C-ABI layer and the kernel translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Arguments of the forward kernel that are not TMA descriptors.
struct FwdArgs {
  float* lse;            // [B*H, N] fp32 logsumexp output
  int N;                 // query rows per head (N_q)
  int Nk;                // key/value rows per head (N_k)
  int BH;                // batch * query heads
  int H;                 // query heads per batch entry
  int group;             // query heads per key/value head (H / H_kv)
  int num_qblocks;       // ceil(N / rows per CTA)
  float scale;           // softmax scale
  float scale_log2;      // scale * log2(e): scores go to base 2 with one multiply
  int causal;            // key j hidden from query i when j > i + (Nk - N)
  int head_group;        // heads per group of the CTA order (cta_head_group)
  uint32_t* err;         // device error word
};

// Arguments of the backward kernels that are not TMA descriptors.
struct BwdArgs {
  const void* q;         // [B*H, N, d] queries (16-bit)
  const void* k;         // [B*H_kv, Nk, d] keys (16-bit)
  const void* o;         // [B*H, N, d] forward output (16-bit)
  const void* dout;      // [B*H, N, d] upstream gradient (16-bit)
  const float* lse;      // [B*H, N] logsumexp from the forward pass
  float* lse_log2;       // [B*H, Npad] L * log2(e), +inf on padding rows (workspace)
  float* delta;          // [B*H, Npad] fp32 D = rowsum(dO o O), 0 on padding rows (workspace)
  void* dq;              // [B*H, N, d] 16-bit dQ output
  void* dk;              // [B*H_kv, Nk, d] 16-bit dK output
  void* dv;              // [B*H_kv, Nk, d] 16-bit dV output
  int N;                 // query rows per head (N_q)
  int Npad;              // N rounded up to a multiple of 128 (row stride of lse_log2 and delta)
  int Nk;                // key/value rows per head (N_k)
  int d;
  int BH;                // batch * query heads
  int BHkv;              // batch * key/value heads
  int H;                 // query heads per batch entry
  int group;             // query heads per key/value head
  float scale;
  float scale_log2;
  int causal;
  int head_group_kv;     // key/value heads per group of the dK/dV kernel's CTA order
  int head_group_q;      // query heads per group of the dQ kernel's CTA order
  uint32_t* err;
};

// Heads per group of a kernel's CTA order (grouped_tile): the blocks of G heads are
// launched before those of the next G, so the tiles that concurrently running CTAs
// read stay in L2.  G is the smallest count whose group gives every SM at least as
// much work as the group's longest CTA (no tail inside a group), raised until the
// group's tensors (bytes_per_head each) fill about 48 MB, at most nheads, and
// then rounded up to a divisor of nheads (within a factor of two) so that every
// group is equally long.
// nblocks is the number of CTA blocks per head, each doing up to nblocks steps.
int cta_head_group(long long nheads, int nblocks, size_t bytes_per_head, bool causal);

// Rows of Q handled by one forward CTA: 128 at d = 256; at d = 64 and 128, 256 (two
// 128-row sub-tiles a CTA) unless that grid (BH x ceil(N / 256) CTAs) would fill less
// than one wave of the num_sms SMs, then 128 (one sub-tile a CTA, twice the CTAs).
int fwd_rows_per_cta(int d, long long BH, int N, int num_sms);

// Forward launch; `rows` is fwd_rows_per_cta's answer for the same problem.
cudaError_t launch_fwd(int d, bool bf16, int rows, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& o, const FwdArgs& a, cudaStream_t stream);

// Measurement hook: events around each main kernel launch while profiling is on
// (no-ops otherwise).  Kinds, as fa_profile_end reports them:
enum : int {
  kProfileFwd = 0,       // the fused forward kernel
  kProfileBwdKV = 1,     // the dK/dV kernel (d = 64, 128)
  kProfileBwdQ = 2,      // the dQ kernel (d = 64, 128)
  kProfileBwdFused = 3,  // the one backward launch of d = 256
};
void profile_mark_begin(cudaStream_t stream);
void profile_mark_end(cudaStream_t stream, int kind);

// Workspace layout of the backward pass (bytes): L*log2(e) and D rows padded per
// head to a multiple of 128, each part 256-byte aligned.  The same for every head
// dimension: no kernel keeps a gradient accumulator in device memory.
size_t bwd_workspace_bytes(long long BH, int N);
size_t bwd_delta_offset(long long BH, int N);
inline int bwd_npad(int N) { return (N + 127) / 128 * 128; }

// Rows per TMA box of the backward pass's Q, K, V, dO descriptors for head dimension d.
inline int bwd_box_rows(int d) { return d == 256 ? 64 : 128; }

// Main kernels of the backward pass with 128 x 128 tiles (d = 64, 128): dK/dV, then dQ.
cudaError_t launch_bwd_main_sq(int d, bool bf16, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& dout, const BwdArgs& a, cudaStream_t stream);

// Main kernel of the backward pass for d = 256 (dK, dV and dQ CTAs in one launch).
cudaError_t launch_bwd_main_256(bool bf16, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& dout, const BwdArgs& a, cudaStream_t stream);

// Failure-detection self-test: one bounded wait that nothing completes.
cudaError_t launch_selftest_wait(uint32_t* err, uint64_t limit_ns, cudaStream_t stream);

#ifdef FA_DEBUG
// FA_DEBUG builds: one device-side check of the given kind handed a value that breaks it.
cudaError_t launch_selftest_check(uint32_t* err, int kind, cudaStream_t stream);
#endif

cudaError_t launch_bwd(int d, bool bf16, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& dout, const BwdArgs& a, cudaStream_t stream);

}  // namespace fa
