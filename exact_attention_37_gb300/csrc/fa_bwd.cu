// Backward pass of exact attention for sm_103a: the D pre-pass and the launch
// sequence for every head dimension.  The main kernels are in fa_bwd_sq.cu
// (d = 64, 128: a dK/dV kernel and a dQ kernel) and fa_bwd256.cu (d = 256: one
// launch of dK, dV and dQ CTAs); none of them uses atomics.
//
// The pages say the method serves training (page "FlashAttention-2 —
// فلاش أتنشن-2", section "Performance and efficiency") and that no N x N matrix
// is kept in device memory (page "FlashAttention — فلاش أتنشن", section
// "Tiling and block processing"); the backward pass therefore rebuilds the
// probabilities block by block from Q, K and the forward pass's logsumexp L:
//
//   D_i  = sum_c dO_ic O_ic                       (pre-pass, one value per row)
//   P    = exp(scale * q_i.k_j - L_i)             (recomputed, never stored globally)
//   dV_j = sum_i P_ij dO_i
//   dS   = P o (dO_i . v_j - D_i)
//   dK_j = scale * sum_i dS_ij q_i
//   dQ_i = scale * sum_j dS_ij k_j
#include <algorithm>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// D_i = sum_c dO_ic O_ic per row, and L_i * log2(e) copied next to it.  Both row
// vectors are padded per head to Npad rows (a multiple of 128) so the main
// kernels read whole aligned blocks; padding rows
// get L = +inf (P = 0) and D = 0.  D / 8 lanes share a row, each loading 16 bytes
// of O and of dO, so a warp covers 256 / D rows per step; two steps are in flight
// per iteration to keep enough loads outstanding for the memory system.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdArgs args, long long slots) {
  constexpr int kLpr = D / 8;            // lanes per row
  constexpr int kRpw = 32 / kLpr;        // rows per warp step
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLpr, part = lane % kLpr;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const uint16_t* o = reinterpret_cast<const uint16_t*>(args.o);
  const uint16_t* g = reinterpret_cast<const uint16_t*>(args.dout);
  const long long steps = (slots + kRpw - 1) / kRpw;
  for (long long st0 = warp0; st0 < steps; st0 += 2 * nwarps) {
    uint4 ov[2], gv[2];
    long long slot[2], row[2];
    bool valid[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const long long st = st0 + k * nwarps;
      slot[k] = st * kRpw + sub;
      const long long head = slot[k] / args.Npad;
      const int i = (int)(slot[k] - head * args.Npad);
      valid[k] = st < steps && slot[k] < slots && i < args.N;
      row[k] = head * args.N + i;
      if (valid[k]) {
        const size_t base = (size_t)row[k] * D + part * 8;
        ov[k] = *reinterpret_cast<const uint4*>(o + base);
        gv[k] = *reinterpret_cast<const uint4*>(g + base);
      } else {
        ov[k] = make_uint4(0, 0, 0, 0);
        gv[k] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint32_t ow[4] = {ov[k].x, ov[k].y, ov[k].z, ov[k].w};
      const uint32_t gw[4] = {gv[k].x, gv[k].y, gv[k].z, gv[k].w};
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        acc = fmaf(widen16<BF16>((uint16_t)(ow[w] & 0xFFFFu)), widen16<BF16>((uint16_t)(gw[w] & 0xFFFFu)), acc);
        acc = fmaf(widen16<BF16>((uint16_t)(ow[w] >> 16)), widen16<BF16>((uint16_t)(gw[w] >> 16)), acc);
      }
#pragma unroll
      for (int off = kLpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (st0 + k * nwarps < steps && slot[k] < slots && part == 0) {
        if (valid[k]) {
          args.delta[slot[k]] = acc;
          args.lse_log2[slot[k]] = args.lse[row[k]] * kLog2e;
        } else {
          args.lse_log2[slot[k]] = INFINITY;  // padding row
          args.delta[slot[k]] = 0.f;
        }
      }
    }
  }
}

int num_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

// D and L log2(e), both padded per head.
template <int D, bool BF16>
cudaError_t launch_pre(const BwdArgs& a, cudaStream_t stream) {
  const long long slots = (long long)a.BH * a.Npad;
  const long long want = (slots * D / 256 + 7) / 8;  // warp steps / warps per block
  const int grid = (int)std::max<long long>(1, std::min<long long>(want, (long long)num_sms() * 16));
  fa_bwd_pre_kernel<D, BF16><<<grid, 256, 0, stream>>>(a, slots);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(int d, bool bf16, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& dout, const BwdArgs& a, cudaStream_t stream) {
  cudaError_t e;
  switch (d) {
    case 64:
      e = bf16 ? launch_pre<64, true>(a, stream) : launch_pre<64, false>(a, stream);
      return e != cudaSuccess ? e : launch_bwd_main_sq(d, bf16, q, k, v, dout, a, stream);
    case 128:
      e = bf16 ? launch_pre<128, true>(a, stream) : launch_pre<128, false>(a, stream);
      return e != cudaSuccess ? e : launch_bwd_main_sq(d, bf16, q, k, v, dout, a, stream);
    case 256:
      e = bf16 ? launch_pre<256, true>(a, stream) : launch_pre<256, false>(a, stream);
      return e != cudaSuccess ? e : launch_bwd_main_256(bf16, q, k, v, dout, a, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace fa
