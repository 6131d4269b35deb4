// Backward pass of exact attention for sm_103a.
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
//   dQ_i = scale * sum_j dS_ij k_j                (fp32 accumulator, atomics)
//
// Work is split over (batch*head, key block of 128 keys) -- the key-block
// parallelism of page "FlashAttention-2 — فلاش أتنشن-2", section "Technical
// architecture", item 2 -- and, for d = 256, over two 128-column halves of the
// gradients.  Each CTA keeps K_j and V_j in shared memory and the dK_j, dV_j
// accumulators in TMEM, and streams the query blocks it needs (under the causal
// mask only those at or after the diagonal).
//
// Everything is computed transposed, keys on TMEM lanes: S^T = K_j Q_i^T and
// dP^T = V_j dO_i^T give every softmax thread one key row, so P^T and dS^T can
// be written as the K-major A operands of dV += P^T dO and dK += dS^T Q.  dQ
// uses the same dS^T tile read MN-major: dQ_i = dS K_j (keys on the K side) for
// 128-row query blocks, or dQ_i^T = K_j^T dS^T for 64-row query blocks so that
// the accumulator keeps M = 128.
//
// Warp roles: warps 0-7 (two warpgroups, half of the query columns each) turn
// S^T and dP^T into P^T and dS^T, releasing the S^T/dP^T accumulators as soon
// as they have read them so the next block's scores overlap this block's
// exponentials; warps 8-11 drain dQ from TMEM into the fp32 accumulator and
// write dK, dV at the end; warp 12 issues TMA loads; warp 13 issues the tcgen05
// MMAs.
#include <algorithm>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBN = 128;   // keys per CTA (= TMEM lanes)
// Warp roles: 0-7 elementwise (two warpgroups), 8-11 dQ drain and epilogue, 12 TMA, 13 MMA.
constexpr int kWarpTma = 12;
constexpr int kWarpMma = 13;
constexpr int kBwdThreads = 14 * 32;
constexpr float kLog2e = 1.4426950408889634f;

// D, DH: head dim and gradient columns per CTA; BM: query rows per block;
// DQT: compute dQ^T (M = DH) instead of dQ (M = BM); STG: Q/dO pipeline depth;
// NPB: P^T/dS^T tile buffers (2 lets the softmax warps write block i+1 while the
// tensor cores still read block i).
template <int D, int DH, int BM, bool DQT, int STG, int NPB>
struct BwdLayout {
  static constexpr uint32_t kKVPanel = kBN * 128;                 // 128 key rows x 128 B
  static constexpr uint32_t kQPanel = BM * 128;                   // BM query rows x 128 B
  static constexpr uint32_t kKVTile = (D / 64) * kKVPanel;
  static constexpr uint32_t kQTile = (D / 64) * kQPanel;
  static constexpr uint32_t kPdsPanel = kBN * 128;                // 128 key rows x 64 queries
  static constexpr uint32_t kPdsTile = (BM / 64) * kPdsPanel;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + kKVTile;
  static constexpr uint32_t kQ = kV + kKVTile;                    // STG stages of (Q, dO)
  static constexpr uint32_t kPds = kQ + STG * 2 * kQTile;         // NPB x (P^T, dS^T)
  static constexpr uint32_t pt(int b) { return kPds + 2u * kPdsTile * b; }
  static constexpr uint32_t dst(int b) { return kPds + 2u * kPdsTile * b + kPdsTile; }
  static constexpr uint32_t kLD = kPds + 2u * kPdsTile * NPB;     // 2 buffers x (L, D) x BM floats
  static constexpr uint32_t kBar = kLD + 2 * 2 * BM * 4;
  static constexpr int kKVFull = 0;
  static constexpr int kQFull = 1;
  static constexpr int kQEmpty = kQFull + STG;
  static constexpr int kSFull = kQEmpty + STG;
  static constexpr int kSdpFree = kSFull + 1;
  static constexpr int kPdsFull = kSdpFree + 1;                   // two, used alternately
  static constexpr int kGrads = kPdsFull + 2;                     // one per P^T/dS^T buffer
  static constexpr int kDqFree = kGrads + NPB;
  static constexpr int kDrain = kDqFree + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr uint32_t kTmemSlot = kBar + kNumBars * 8;
  static constexpr uint32_t kBytes = kTmemSlot + 16;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  // TMEM columns
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColDP = BM;
  static constexpr uint32_t kColDV = 2 * BM;
  static constexpr uint32_t kColDK = 2 * BM + DH;
  static constexpr uint32_t kColDQ = 2 * BM + 2 * DH;
  static constexpr uint32_t kDqCols = DQT ? BM : DH;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kColDQ + kDqCols <= 512, "TMEM budget");
  static_assert(kBytes + 1024 <= 232448, "shared memory budget");
  static_assert(!DQT || DH == 128, "dQ^T needs M = 128");
  static_assert(DQT || BM == 128, "dQ needs M = 128");
};

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void red_add(float* addr, float a) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(a) : "memory");
}
__device__ __forceinline__ void st_global_v4(void* addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <int D, int DH, int BM, bool DQT, int STG, int NPB, bool BF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdArgs args) {
  using L = BwdLayout<D, DH, BM, DQT, STG, NPB>;
  constexpr int kHalves = D / DH;
  constexpr int kCW = BM / 2;        // query columns per elementwise warpgroup
  constexpr int kNCh = kCW / 32;     // 32-column TMEM chunks per elementwise thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
  auto sQ = [&](int s) -> uint32_t { return sbase + L::kQ + 2u * L::kQTile * s; };
  auto sDO = [&](int s) -> uint32_t { return sbase + L::kQ + 2u * L::kQTile * s + L::kQTile; };
  const uint32_t sK = sbase + L::kK, sV = sbase + L::kV;
  auto sPt = [&](int b) -> uint32_t { return sbase + L::pt(b); };
  auto sDSt = [&](int b) -> uint32_t { return sbase + L::dst(b); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = args.N;

  // Work tile: the lowest key blocks first across all heads (under the causal mask
  // they have the most query blocks), so the last wave holds the lightest work.
  const int tiles_per_kb = args.BH * kHalves;
  const int kb = (int)(blockIdx.x / tiles_per_kb);
  const int rem = (int)(blockIdx.x % tiles_per_kb);
  const int bh = rem / kHalves;
  const int half = rem % kHalves;
  const int key0 = kb * kBN;
  const int nqb = (N + BM - 1) / BM;
  const int i_begin = args.causal ? key0 / BM : 0;
  const int nit = nqb - i_begin;  // query blocks this CTA visits (>= 1)

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kKVFull), 1);
    for (int s = 0; s < STG; ++s) {
      mbar_init(bar(L::kQFull + s), 1);
      mbar_init(bar(L::kQEmpty + s), 1);
    }
    mbar_init(bar(L::kSFull), 1);
    mbar_init(bar(L::kSdpFree), 256);
    mbar_init(bar(L::kPdsFull + 0), 256);
    mbar_init(bar(L::kPdsFull + 1), 256);
    for (int b = 0; b < NPB; ++b) mbar_init(bar(L::kGrads + b), 1);
    mbar_init(bar(L::kDqFree), 128);
    mbar_init(bar(L::kDrain), 1);
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(sbase + L::kTmemSlot, L::kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_expect_tx(bar(L::kKVFull), 2 * L::kKVTile);
#pragma unroll
      for (int p = 0; p < D / 64; ++p) {
        tma_load_3d(sK + p * L::kKVPanel, &tm_k, bar(L::kKVFull), 64 * p, key0, bh);
        tma_load_3d(sV + p * L::kKVPanel, &tm_v, bar(L::kKVFull), 64 * p, key0, bh);
      }
      for (int it = 0; it < nit; ++it) {
        const int s = it % STG, u = it / STG;
        if (u > 0 && !mbar_wait(bar(L::kQEmpty + s), (u - 1) & 1, args.err, kErrTimeoutRing)) break;
        mbar_expect_tx(bar(L::kQFull + s), 2 * L::kQTile);
        const int q0 = (i_begin + it) * BM;
#pragma unroll
        for (int p = 0; p < D / 64; ++p) {
          tma_load_3d(sQ(s) + p * L::kQPanel, &tm_q, bar(L::kQFull + s), 64 * p, q0, bh);
          tma_load_3d(sDO(s) + p * L::kQPanel, &tm_do, bar(L::kQFull + s), 64 * p, q0, bh);
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = make_idesc_f16(BF16, kBN, BM, false, false);     // S^T, dP^T: M=128 keys, N=BM
      constexpr uint32_t kIdG = make_idesc_f16(BF16, kBN, DH, false, true);      // dV, dK: M=128 keys, N=DH
      constexpr uint32_t kIdQ = DQT ? make_idesc_f16(BF16, DH, BM, true, true)   // dQ^T: M=DH, N=BM, A=K^T
                                    : make_idesc_f16(BF16, BM, DH, true, true);  // dQ: M=BM, N=DH, A=dS
      const uint32_t hp = (uint32_t)(half * (DH / 64));  // first 64-column panel of this CTA's half
      auto issue_sdp = [&](int s) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t a_off = (kk >> 2) * L::kKVPanel + (kk & 3) * 32;
          const uint32_t b_off = (kk >> 2) * L::kQPanel + (kk & 3) * 32;
          mma_ss(tmem + L::kColS, make_sdesc_sw128(sK + a_off, 16, 1024), make_sdesc_sw128(sQ(s) + b_off, 16, 1024),
                 kIdS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t a_off = (kk >> 2) * L::kKVPanel + (kk & 3) * 32;
          const uint32_t b_off = (kk >> 2) * L::kQPanel + (kk & 3) * 32;
          mma_ss(tmem + L::kColDP, make_sdesc_sw128(sV + a_off, 16, 1024),
                 make_sdesc_sw128(sDO(s) + b_off, 16, 1024), kIdS, kk > 0);
        }
      };
      auto issue_grads = [&](int s, int it) {
        const int pb = it % NPB;
        // dV += P^T dO, dK += dS^T Q: A K-major over the BM queries, B MN-major (DH columns).
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk) {
          const uint32_t a_off = (kk >> 2) * L::kPdsPanel + (kk & 3) * 32;
          const uint32_t b_off = hp * L::kQPanel + kk * 2048;
          mma_ss(tmem + L::kColDV, make_sdesc_sw128(sPt(pb) + a_off, 16, 1024),
                 make_sdesc_sw128(sDO(s) + b_off, L::kQPanel, 1024), kIdG, (it > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk) {
          const uint32_t a_off = (kk >> 2) * L::kPdsPanel + (kk & 3) * 32;
          const uint32_t b_off = hp * L::kQPanel + kk * 2048;
          mma_ss(tmem + L::kColDK, make_sdesc_sw128(sDSt(pb) + a_off, 16, 1024),
                 make_sdesc_sw128(sQ(s) + b_off, L::kQPanel, 1024), kIdG, (it > 0 || kk > 0) ? 1u : 0u);
        }
        // dQ (or dQ^T) over the 128 keys of this block; both operands MN-major.
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t k_off = hp * L::kKVPanel + kk * 2048;
          const uint32_t ds_off = kk * 2048;
          if constexpr (DQT) {
            mma_ss(tmem + L::kColDQ, make_sdesc_sw128(sK + k_off, L::kKVPanel, 1024),
                   make_sdesc_sw128(sDSt(pb) + ds_off, L::kPdsPanel, 1024), kIdQ, kk > 0);
          } else {
            mma_ss(tmem + L::kColDQ, make_sdesc_sw128(sDSt(pb) + ds_off, L::kPdsPanel, 1024),
                   make_sdesc_sw128(sK + k_off, L::kKVPanel, 1024), kIdQ, kk > 0);
          }
        }
      };
      auto next_scores = [&](int it) -> bool {
        const int s1 = (it + 1) % STG;
        if (!mbar_wait(bar(L::kQFull + s1), ((it + 1) / STG) & 1, args.err, kErrTimeoutTma)) return false;
        tc_fence_after();
        issue_sdp(s1);
        mma_commit(bar(L::kSFull));
        return true;
      };
      bool ok = mbar_wait(bar(L::kKVFull), 0, args.err, kErrTimeoutTma);
      if (ok) ok = mbar_wait(bar(L::kQFull + 0), 0, args.err, kErrTimeoutTma);
      if (ok) {
        tc_fence_after();
        issue_sdp(0);
        mma_commit(bar(L::kSFull));
      }
      for (int it = 0; ok && it < nit; ++it) {
        const int s = it % STG;
        // Scores of the next block as soon as this block's S^T/dP^T have been read
        // out of TMEM, so they run while the elementwise warps exponentiate.
        // (With one Q/dO stage the next tile only arrives after this block's
        // gradients release the stage, so they go after the gradients.)
        if (STG > 1 && it + 1 < nit) {
          ok = mbar_wait(bar(L::kSdpFree), it & 1, args.err, kErrTimeoutSoftmax);
          if (!ok || !(ok = next_scores(it))) break;
        }
        ok = mbar_wait(bar(L::kPdsFull + (it & 1)), (it >> 1) & 1, args.err, kErrTimeoutSoftmax);
        if (!ok) break;
        tc_fence_after();
        if (it > 0) {
          ok = mbar_wait(bar(L::kDqFree), (it - 1) & 1, args.err, kErrTimeoutSoftmax);
          if (!ok) break;
          tc_fence_after();
        }
        issue_grads(s, it);
        mma_commit(bar(L::kGrads + it % NPB));
        mma_commit(bar(L::kQEmpty + s));
        if (STG == 1 && it + 1 < nit && !(ok = next_scores(it))) break;
      }
      mma_commit(bar(L::kDrain));
      mbar_wait(bar(L::kDrain), 0, args.err, kErrTimeoutMma);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ P^T and dS^T
    // Two warpgroups; warpgroup e handles query columns [e*kCW, (e+1)*kCW) of the block.
    const int e = warp >> 2;
    const int wq = warp & 3;
    const int r = (wq << 5) + lane;  // key row inside the block == TMEM lane
    const int key = key0 + r;
    const int cbeg = e * kCW;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const float c = args.scale_log2;
    float* sL = reinterpret_cast<float*>(smem + L::kLD);  // [2][2][BM]: (L*log2e, D) per buffer
    const size_t row_base = (size_t)bh * N;
    // L and D of query column (block it, column cbeg + r) are fetched one block
    // ahead, so the global-memory latency overlaps the previous block's work.
    float pf_l = 0.f, pf_d = 0.f;
    bool pf_in = false;
    auto prefetch = [&](int it) {
      const int q = (i_begin + it) * BM + cbeg + r;
      pf_in = (r < kCW) && (it < nit) && (q < N);
      if (pf_in) {
        pf_l = __ldg(args.lse + row_base + q);
        pf_d = __ldg(args.delta + row_base + q);
      }
    };
    prefetch(0);
    for (int it = 0; it < nit; ++it) {
      const int q0 = (i_begin + it) * BM;
      float* bufL = sL + (it & 1) * 2 * BM;
      float* bufD = bufL + BM;
      if (r < kCW) {
        bufL[cbeg + r] = pf_in ? pf_l * kLog2e : INFINITY;  // rows past N get P = 0
        bufD[cbeg + r] = pf_in ? pf_d : 0.f;
      }
      prefetch(it + 1);
      named_bar_sync(1 + e, 128);
      if (!mbar_wait(bar(L::kSFull), it & 1, args.err, kErrTimeoutMma)) break;
      tc_fence_after();
      const bool diag = args.causal && (key0 + kBN - 1 > q0);  // some key of the block is after some query
      const int pb = it % NPB;
      // The P^T/dS^T buffer pb is free once the gradients of block it-NPB (its last reader) are done.
      auto wait_buffer = [&]() -> bool {
        if (it < NPB) return true;
        if (!mbar_wait(bar(L::kGrads + pb), ((it / NPB) - 1) & 1, args.err, kErrTimeoutMma)) return false;
        tc_fence_after();
        return true;
      };
      uint32_t pw[kCW / 2], dw[kCW / 2];
      bool ok = true;
      if constexpr (kNCh > 1) ok = wait_buffer();  // wide blocks write chunk by chunk
      if (!ok) break;
#pragma unroll
      for (int ch = 0; ch < kNCh; ++ch) {
        uint32_t sv[32], dv[32];
        tmem_ld_32x32b_x32(tmem + lane_base + L::kColS + cbeg + 32 * ch, sv);
        tmem_ld_32x32b_x32(tmem + lane_base + L::kColDP + cbeg + 32 * ch, dv);
        tmem_wait_ld();
        reg_fence32(sv);
        reg_fence32(dv);
        if (ch == kNCh - 1) {
          tc_fence_before();  // this thread is done reading S^T and dP^T from TMEM
          mbar_arrive(bar(L::kSdpFree));
        }
        float p[32], ds[32];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const int col = cbeg + 32 * ch + 4 * e4;
          const float4 l4 = *reinterpret_cast<const float4*>(bufL + col);
          const float4 d4 = *reinterpret_cast<const float4*>(bufD + col);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
          const float dd[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int x = 4 * e4 + u;
            float pe = ex2_approx(fmaf(__uint_as_float(sv[x]), c, -lv[u]));
            if (diag && key > q0 + col + u) pe = 0.f;
            p[x] = pe;
            ds[x] = pe * (__uint_as_float(dv[x]) - dd[u]);
          }
        }
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          pw[16 * ch + x] = pack2<BF16>(p[2 * x], p[2 * x + 1]);
          dw[16 * ch + x] = pack2<BF16>(ds[2 * x], ds[2 * x + 1]);
        }
        if constexpr (kNCh > 1) {
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int chunk = (cbeg + 32 * ch) / 8 + k4;  // 16-byte chunk index along the row
            const uint32_t off = (chunk >> 3) * L::kPdsPanel + sw128_offset(r, chunk & 7);
            const int w = 16 * ch + 4 * k4;
            st_shared_v4(sPt(pb) + off, pw[w], pw[w + 1], pw[w + 2], pw[w + 3]);
            st_shared_v4(sDSt(pb) + off, dw[w], dw[w + 1], dw[w + 2], dw[w + 3]);
          }
        }
      }
      if constexpr (kNCh == 1) {
        if (!wait_buffer()) break;
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int chunk = cbeg / 8 + k4;
          const uint32_t off = (chunk >> 3) * L::kPdsPanel + sw128_offset(r, chunk & 7);
          st_shared_v4(sPt(pb) + off, pw[4 * k4], pw[4 * k4 + 1], pw[4 * k4 + 2], pw[4 * k4 + 3]);
          st_shared_v4(sDSt(pb) + off, dw[4 * k4], dw[4 * k4 + 1], dw[4 * k4 + 2], dw[4 * k4 + 3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(L::kPdsFull + (it & 1)));
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ dQ drain + dK/dV epilogue
    const int wq = warp - 8;
    const int r = (wq << 5) + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    float* dq_acc = args.dq_acc + (size_t)bh * N * D;
    bool ok = true;
    for (int it = 0; it < nit; ++it) {
      const int q0 = (i_begin + it) * BM;
      ok = mbar_wait(bar(L::kGrads + it % NPB), (it / NPB) & 1, args.err, kErrTimeoutMma);
      if (!ok) break;
      tc_fence_after();
      constexpr int kCh = L::kDqCols / 32;
      uint32_t v[kCh][32];
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) tmem_ld_32x32b_x32(tmem + lane_base + L::kColDQ + 32 * ch, v[ch]);
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) reg_fence32(v[ch]);
      tc_fence_before();
      mbar_arrive(bar(L::kDqFree));
      if constexpr (DQT) {
        // lane r holds dQ^T row r: column half*DH + r of query rows q0 .. q0+BM-1
        const int col = half * DH + r;
#pragma unroll
        for (int ch = 0; ch < kCh; ++ch)
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int q = q0 + 32 * ch + x;
            if (q < N) red_add(dq_acc + (size_t)q * D + col, __uint_as_float(v[ch][x]));
          }
      } else {
        // lane r holds dQ row q0 + r, columns half*DH .. half*DH+DH-1
        const int q = q0 + r;
        if (q < N) {
          float* dst = dq_acc + (size_t)q * D + half * DH;
#pragma unroll
          for (int ch = 0; ch < kCh; ++ch)
#pragma unroll
            for (int x = 0; x < 32; x += 4)
              red_add_v4(dst + 32 * ch + x, __uint_as_float(v[ch][x]), __uint_as_float(v[ch][x + 1]),
                         __uint_as_float(v[ch][x + 2]), __uint_as_float(v[ch][x + 3]));
        }
      }
    }
    if (ok) {
      // Final gradients of this key block; lane r holds key row key0 + r.
      const int key = key0 + r;
      const size_t out_row = ((size_t)bh * N + key) * D + half * DH;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t col0 = which == 0 ? L::kColDV : L::kColDK;
        const float mul = which == 0 ? 1.f : args.scale;
        uint16_t* dst = reinterpret_cast<uint16_t*>(which == 0 ? args.dv : args.dk) + out_row;
#pragma unroll 1
        for (int ch = 0; ch < DH / 32; ++ch) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem + lane_base + col0 + 32 * ch, v);
          tmem_wait_ld();
          reg_fence32(v);
          if (key < N) {
#pragma unroll
            for (int x = 0; x < 32; x += 8)
              st_global_v4(dst + 32 * ch + x,
                           pack2<BF16>(__uint_as_float(v[x]) * mul, __uint_as_float(v[x + 1]) * mul),
                           pack2<BF16>(__uint_as_float(v[x + 2]) * mul, __uint_as_float(v[x + 3]) * mul),
                           pack2<BF16>(__uint_as_float(v[x + 4]) * mul, __uint_as_float(v[x + 5]) * mul),
                           pack2<BF16>(__uint_as_float(v[x + 6]) * mul, __uint_as_float(v[x + 7]) * mul));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// D_i = sum_c dO_ic O_ic per row, and the fp32 dQ accumulator set to zero.
// One warp per row, grid-stride; each lane handles D/32 consecutive elements.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdArgs args, long long rows) {
  constexpr int kPer = D / 32;  // 2, 4 or 8 elements per lane
  const int lane = threadIdx.x & 31;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const uint16_t* o = reinterpret_cast<const uint16_t*>(args.o);
  const uint16_t* g = reinterpret_cast<const uint16_t*>(args.dout);
  for (long long row = warp0; row < rows; row += nwarps) {
    const size_t base = (size_t)row * D + lane * kPer;
    float acc = 0.f;
    uint16_t ov[kPer], gv[kPer];
    if constexpr (kPer == 8) {
      *reinterpret_cast<uint4*>(ov) = *reinterpret_cast<const uint4*>(o + base);
      *reinterpret_cast<uint4*>(gv) = *reinterpret_cast<const uint4*>(g + base);
    } else if constexpr (kPer == 4) {
      *reinterpret_cast<uint2*>(ov) = *reinterpret_cast<const uint2*>(o + base);
      *reinterpret_cast<uint2*>(gv) = *reinterpret_cast<const uint2*>(g + base);
    } else {
      *reinterpret_cast<uint32_t*>(ov) = *reinterpret_cast<const uint32_t*>(o + base);
      *reinterpret_cast<uint32_t*>(gv) = *reinterpret_cast<const uint32_t*>(g + base);
    }
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      acc = fmaf(widen16<BF16>(ov[e]), widen16<BF16>(gv[e]), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) args.delta[row] = acc;
    float* z = args.dq_acc + base;
#pragma unroll
    for (int e = 0; e < kPer; e += 2) *reinterpret_cast<float2*>(z + e) = make_float2(0.f, 0.f);
  }
}

// dQ = scale * dQ_acc rounded to 16 bits; 8 elements per thread, grid-stride.
template <bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_dq_convert_kernel(const BwdArgs args, long long n8) {
  const float4* src = reinterpret_cast<const float4*>(args.dq_acc);
  uint4* dst = reinterpret_cast<uint4*>(args.dq);
  const float s = args.scale;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
    const float4 a = src[2 * i], b = src[2 * i + 1];
    dst[i] = make_uint4(pack2<BF16>(a.x * s, a.y * s), pack2<BF16>(a.z * s, a.w * s), pack2<BF16>(b.x * s, b.y * s),
                        pack2<BF16>(b.z * s, b.w * s));
  }
}

template <int D, int DH, int BM, bool DQT, int STG, int NPB, bool BF16>
cudaError_t launch_bwd_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout,
                         const BwdArgs& a, cudaStream_t stream) {
  using L = BwdLayout<D, DH, BM, DQT, STG, NPB>;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long rows = (long long)a.BH * a.N;
  // 1) D and zeroed dQ accumulator
  {
    const long long want = (rows + 7) / 8;
    const int grid = (int)std::min<long long>(want, (long long)sms * 16);
    fa_bwd_pre_kernel<D, BF16><<<grid, 256, 0, stream>>>(a, rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // 2) main kernel
  {
    auto kern = fa_bwd_kernel<D, DH, BM, DQT, STG, NPB, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kAlloc);
    if (e != cudaSuccess) return e;
    const long long nkb = (a.N + kBN - 1) / kBN;
    const long long grid = nkb * a.BH * (D / DH);
    profile_mark_begin(stream);
    kern<<<(unsigned)grid, kBwdThreads, L::kAlloc, stream>>>(q, k, v, dout, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    profile_mark_end(stream, 1);
  }
  // 3) dQ conversion
  {
    const long long n8 = rows * D / 8;
    const int grid = (int)std::min<long long>((n8 + 255) / 256, (long long)sms * 16);
    fa_bwd_dq_convert_kernel<BF16><<<grid, 256, 0, stream>>>(a, n8);
    return cudaGetLastError();
  }
}

}  // namespace

int bwd_query_rows(int d) { return d == 64 ? 128 : 64; }

cudaError_t launch_bwd(int d, bool bf16, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& dout, const BwdArgs& a, cudaStream_t stream) {
  switch (d) {
    case 64:
      return bf16 ? launch_bwd_t<64, 64, 128, false, 3, 1, true>(q, k, v, dout, a, stream)
                  : launch_bwd_t<64, 64, 128, false, 3, 1, false>(q, k, v, dout, a, stream);
    case 128:
      return bf16 ? launch_bwd_t<128, 128, 64, true, 3, 2, true>(q, k, v, dout, a, stream)
                  : launch_bwd_t<128, 128, 64, true, 3, 2, false>(q, k, v, dout, a, stream);
    case 256:
      return bf16 ? launch_bwd_t<256, 128, 64, true, 1, 1, true>(q, k, v, dout, a, stream)
                  : launch_bwd_t<256, 128, 64, true, 1, 1, false>(q, k, v, dout, a, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace fa
