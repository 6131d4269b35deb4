// Backward pass of exact attention for sm_103a: the pre-pass and dQ conversion
// kernels, the launch sequence for every head dimension, and the fused main
// kernel used for d = 256 (d = 64 and 128 run the two deterministic main
// kernels of fa_bwd_sq.cu instead).
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
// exponentials; warps 8-11 drain dQ from TMEM into the fp32 accumulator (lane =
// head-dimension index: each reduction instruction covers 32 consecutive columns
// of one query row) and write dK, dV at the end; warp 12 issues TMA loads; warp 13
// issues the tcgen05 MMAs.
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
  static constexpr uint32_t kDs = kQ + STG * 2 * kQTile;          // NPB x dS^T
  static constexpr uint32_t dst(int b) { return kDs + kPdsTile * b; }
  static constexpr uint32_t kLD = kDs + kPdsTile * NPB;           // 2 buffers x (L, D) x BM floats
  static constexpr uint32_t kBar = kLD + 2 * 2 * BM * 4;
  static constexpr int kKVFull = 0;
  static constexpr int kQFull = 1;
  static constexpr int kQEmpty = kQFull + STG;
  static constexpr int kSReady = kQEmpty + STG;                   // S^T of the block is in TMEM
  static constexpr int kDpReady = kSReady + 1;                    // dP^T of the block is in TMEM
  static constexpr int kSdpFree = kDpReady + 1;                   // S^T and dP^T have been read out
  static constexpr int kPFull = kSdpFree + 1;                     // two, used alternately: P^T in TMEM
  static constexpr int kDsFull = kPFull + 2;                      // two, used alternately: dS^T in smem
  static constexpr int kGrads = kDsFull + 2;                      // one per P^T/dS^T buffer
  static constexpr int kDqFree = kGrads + NPB;
  static constexpr int kDrain = kDqFree + 1;
  static constexpr int kEwSync = kDrain + 1;                      // two: one per elementwise warpgroup
  static constexpr int kNumBars = kEwSync + 2;
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
  static constexpr uint32_t kColPt = kColDQ + kDqCols;            // NPB x P^T (16-bit pairs, BM/2 columns)
  static constexpr uint32_t pt_col(int b) { return kColPt + (uint32_t)(BM / 2) * b; }
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kColPt + NPB * (BM / 2) <= 512, "TMEM budget");
  static_assert(kBytes + 1024 <= 232448, "shared memory budget");
  static_assert(!DQT || DH == 128, "dQ^T needs M = 128");
  static_assert(DQT || BM == 128, "dQ needs M = 128");
};

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
  auto sDSt = [&](int b) -> uint32_t { return sbase + L::dst(b); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = args.N;

  // Work tile: the lowest key blocks first (under the causal mask they have the
  // most query blocks), so the last wave holds the lightest work; key/value heads
  // in groups of args.head_group_kv (both column halves of a head in one group), so
  // the tiles of the running CTAs stay in L2.  One CTA per (key/value head, key
  // block, column half); it visits the query blocks of every query head of its
  // group, so dK and dV of a shared key/value head are summed in TMEM without any
  // cross-CTA reduction.
  int kb, rem;
  grouped_tile(blockIdx.x, args.BHkv * kHalves, (args.Nk + kBN - 1) / kBN, args.head_group_kv * kHalves, kb, rem);
  const int bh_kv = rem / kHalves;
  const int half = rem % kHalves;
  const int Nk = args.Nk;
  const int koff = Nk - N;  // causal mask: key j visible to query i iff j <= i + koff
  const int key0 = kb * kBN;
  const int nqb = (N + BM - 1) / BM;
  const int i_begin = args.causal ? max(0, key0 - koff) / BM : 0;
  const int nit_h = nqb - i_begin;    // query blocks per query head (>= 1)
  const int nit = nit_h * args.group;  // over the whole group
  const int h_kv = bh_kv % (args.H / args.group);
  const int bh_q0 = (bh_kv / (args.H / args.group)) * args.H + h_kv * args.group;  // first query head of the group
  // query head and query block of iteration it
  auto q_head = [&](int it) { return bh_q0 + it / nit_h; };
  auto q_block = [&](int it) { return i_begin + it % nit_h; };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kKVFull), 1);
    for (int s = 0; s < STG; ++s) {
      mbar_init(bar(L::kQFull + s), 1);
      mbar_init(bar(L::kQEmpty + s), 1);
    }
    mbar_init(bar(L::kSReady), 1);
    mbar_init(bar(L::kDpReady), 1);
    mbar_init(bar(L::kSdpFree), 256);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(L::kPFull + b), 256);
      mbar_init(bar(L::kDsFull + b), 256);
    }
    for (int b = 0; b < NPB; ++b) mbar_init(bar(L::kGrads + b), 1);
    mbar_init(bar(L::kDqFree), 128);
    mbar_init(bar(L::kDrain), 1);
    mbar_init(bar(L::kEwSync + 0), 128);
    mbar_init(bar(L::kEwSync + 1), 128);
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
        tma_load_3d(sK + p * L::kKVPanel, &tm_k, bar(L::kKVFull), 64 * p, key0, bh_kv);
        tma_load_3d(sV + p * L::kKVPanel, &tm_v, bar(L::kKVFull), 64 * p, key0, bh_kv);
      }
      for (int it = 0; it < nit; ++it) {
        const int s = it % STG, u = it / STG;
        if (u > 0 && !mbar_wait(bar(L::kQEmpty + s), (u - 1) & 1, args.err, kErrTimeoutRing)) break;
        mbar_expect_tx(bar(L::kQFull + s), 2 * L::kQTile);
        const int q0 = q_block(it) * BM, bq = q_head(it);
#pragma unroll
        for (int p = 0; p < D / 64; ++p) {
          tma_load_3d(sQ(s) + p * L::kQPanel, &tm_q, bar(L::kQFull + s), 64 * p, q0, bq);
          tma_load_3d(sDO(s) + p * L::kQPanel, &tm_do, bar(L::kQFull + s), 64 * p, q0, bq);
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
      constexpr uint32_t kHi = sdesc_hi_sw128(1024);  // every operand here: 8-row groups 1024 B apart
      auto issue_sdp = [&](int s) {
        const uint32_t k0 = sdesc_lo(sK, 16), v0 = sdesc_lo(sV, 16);
        const uint32_t q0 = sdesc_lo(sQ(s), 16), o0 = sdesc_lo(sDO(s), 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t a_off = ((kk >> 2) * L::kKVPanel + (kk & 3) * 32) >> 4;
          const uint32_t b_off = ((kk >> 2) * L::kQPanel + (kk & 3) * 32) >> 4;
          mma_ss_lohi(tmem + L::kColS, k0 + a_off, kHi, q0 + b_off, kHi, kIdS, kk > 0);
        }
        mma_commit(bar(L::kSReady));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t a_off = ((kk >> 2) * L::kKVPanel + (kk & 3) * 32) >> 4;
          const uint32_t b_off = ((kk >> 2) * L::kQPanel + (kk & 3) * 32) >> 4;
          mma_ss_lohi(tmem + L::kColDP, v0 + a_off, kHi, o0 + b_off, kHi, kIdS, kk > 0);
        }
        mma_commit(bar(L::kDpReady));
      };
      // dV += P^T dO: A (P^T) from TMEM, B (dO) MN-major over the DH columns.
      auto issue_dv = [&](int s, int it) {
        const int pb = it % NPB;
        const uint32_t o0 = sdesc_lo(sDO(s) + hp * L::kQPanel, L::kQPanel);
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          mma_ts_lohi(tmem + L::kColDV, tmem + L::pt_col(pb) + 8 * kk, o0 + ((kk * 2048) >> 4), kHi, kIdG,
                      (it > 0 || kk > 0) ? 1u : 0u);
      };
      // dK += dS^T Q (A K-major from smem), then dQ (or dQ^T) over the block's 128 keys.
      auto issue_dk_dq = [&](int s, int it) {
        const int pb = it % NPB;
        const uint32_t ds0 = sdesc_lo(sDSt(pb), 16), q0 = sdesc_lo(sQ(s) + hp * L::kQPanel, L::kQPanel);
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk) {
          const uint32_t a_off = ((kk >> 2) * L::kPdsPanel + (kk & 3) * 32) >> 4;
          mma_ss_lohi(tmem + L::kColDK, ds0 + a_off, kHi, q0 + ((kk * 2048) >> 4), kHi, kIdG,
                      (it > 0 || kk > 0) ? 1u : 0u);
        }
        const uint32_t kmn0 = sdesc_lo(sK + hp * L::kKVPanel, L::kKVPanel);
        const uint32_t dsmn0 = sdesc_lo(sDSt(pb), L::kPdsPanel);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t off = (kk * 2048) >> 4;
          if constexpr (DQT) {
            mma_ss_lohi(tmem + L::kColDQ, kmn0 + off, kHi, dsmn0 + off, kHi, kIdQ, kk > 0);
          } else {
            mma_ss_lohi(tmem + L::kColDQ, dsmn0 + off, kHi, kmn0 + off, kHi, kIdQ, kk > 0);
          }
        }
      };
      auto next_scores = [&](int it) -> bool {
        const int s1 = (it + 1) % STG;
        if (!mbar_wait(bar(L::kQFull + s1), ((it + 1) / STG) & 1, args.err, kErrTimeoutTma)) return false;
        tc_fence_after();
        issue_sdp(s1);
        return true;
      };
      bool ok = mbar_wait(bar(L::kKVFull), 0, args.err, kErrTimeoutTma);
      if (ok) ok = mbar_wait(bar(L::kQFull + 0), 0, args.err, kErrTimeoutTma);
      if (ok) {
        tc_fence_after();
        issue_sdp(0);
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
        ok = mbar_wait(bar(L::kPFull + (it & 1)), (it >> 1) & 1, args.err, kErrTimeoutSoftmax);
        if (!ok) break;
        tc_fence_after();
        issue_dv(s, it);
        ok = mbar_wait(bar(L::kDsFull + (it & 1)), (it >> 1) & 1, args.err, kErrTimeoutSoftmax);
        if (!ok) break;
        if (it > 0) ok = mbar_wait(bar(L::kDqFree), (it - 1) & 1, args.err, kErrTimeoutSoftmax);
        if (!ok) break;
        tc_fence_after();
        issue_dk_dq(s, it);
        mma_commit(bar(L::kGrads + it % NPB));
        mma_commit(bar(L::kQEmpty + s));
        if (STG == 1 && it + 1 < nit && !(ok = next_scores(it))) break;
      }
      mma_commit(bar(L::kDrain));
      mbar_wait(bar(L::kDrain), 0, args.err, kErrTimeoutMma, false);
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
    // L and D of query column (block it, column cbeg + r) are fetched one block
    // ahead, so the global-memory latency overlaps the previous block's work.
    float pf_l = 0.f, pf_d = 0.f;
    bool pf_in = false;
    auto prefetch = [&](int it) {
      if (it >= nit) {
        pf_in = false;
        return;
      }
      const int q = q_block(it) * BM + cbeg + r;
      const size_t row_base = (size_t)q_head(it) * args.Npad;
      pf_in = (r < kCW) && (q < N);
      if (pf_in) {
        pf_l = __ldg(args.lse_log2 + row_base + q);
        pf_d = __ldg(args.delta + row_base + q);
      }
    };
    prefetch(0);
    SmemSync wg_sync{bar(L::kEwSync + e), 0u};
    for (int it = 0; it < nit; ++it) {
      const int q0 = q_block(it) * BM;
      float* bufL = sL + (it & 1) * 2 * BM;
      float* bufD = bufL + BM;
      if (r < kCW) {
        // Rows past N get P = 0 through L = +inf; rows that see no key (L = -inf)
        // get P = 0 through the causal mask below.
        bufL[cbeg + r] = pf_in ? pf_l : INFINITY;
        bufD[cbeg + r] = pf_in ? pf_d : 0.f;
      }
      prefetch(it + 1);
      if (!wg_sync.sync(args.err)) break;
      const bool diag = args.causal && (key0 + kBN - 1 > q0 + koff);  // some key is hidden from some query
      const int pb = it % NPB;
      // P^T of block it-NPB (TMEM buffer pb) and dS^T (smem buffer pb) are free once
      // that block's gradients are done.
      if (it >= NPB) {
        if (!mbar_wait(bar(L::kGrads + pb), ((it / NPB) - 1) & 1, args.err, kErrTimeoutMma)) break;
        tc_fence_after();
      }
      // ---- P^T = 2^(S^T c - L log2 e), as soon as S^T is in TMEM (dP^T may still be running)
      if (!mbar_wait(bar(L::kSReady), it & 1, args.err, kErrTimeoutMma)) break;
      tc_fence_after();
      float p[kCW];
#pragma unroll
      for (int ch = 0; ch < kNCh; ++ch) {
        uint32_t sv[32];
        tmem_ld_32x32b_x32(tmem + lane_base + L::kColS + cbeg + 32 * ch, sv);
        tmem_wait_ld();
        reg_fence32(sv);
        uint32_t pw[16];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const int col = cbeg + 32 * ch + 4 * e4;
          const float4 l4 = *reinterpret_cast<const float4*>(bufL + col);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int x = 4 * e4 + u;
            float pe = ex2_approx(fmaf(__uint_as_float(sv[x]), c, -lv[u]));
            if (diag && key > q0 + col + u + koff) pe = 0.f;
            p[32 * ch + x] = pe;
          }
        }
#pragma unroll
        for (int x = 0; x < 16; ++x) pw[x] = pack2<BF16>(p[32 * ch + 2 * x], p[32 * ch + 2 * x + 1]);
        tmem_st_32x32b_x16(tmem + lane_base + L::pt_col(pb) + (cbeg + 32 * ch) / 2, pw);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(L::kPFull + (it & 1)));
      // ---- dS^T = P^T o (dP^T - D)
      if (!mbar_wait(bar(L::kDpReady), it & 1, args.err, kErrTimeoutMma)) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < kNCh; ++ch) {
        uint32_t dv[32];
        tmem_ld_32x32b_x32(tmem + lane_base + L::kColDP + cbeg + 32 * ch, dv);
        tmem_wait_ld();
        reg_fence32(dv);
        if (ch == kNCh - 1) {
          tc_fence_before();  // this thread is done reading S^T and dP^T from TMEM
          mbar_arrive(bar(L::kSdpFree));
        }
        uint32_t dw[16];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const int col = cbeg + 32 * ch + 4 * e4;
          const float4 d4 = *reinterpret_cast<const float4*>(bufD + col);
          const float dd[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            const int x = 4 * e4 + u;
            const float ds0 = p[32 * ch + x] * (__uint_as_float(dv[x]) - dd[u]);
            const float ds1 = p[32 * ch + x + 1] * (__uint_as_float(dv[x + 1]) - dd[u + 1]);
            dw[x >> 1] = pack2<BF16>(ds0, ds1);
          }
        }
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int chunk = (cbeg + 32 * ch) / 8 + k4;  // 16-byte chunk index along the row
          const uint32_t off = (chunk >> 3) * L::kPdsPanel + sw128_offset(r, chunk & 7);
          st_shared_v4(sDSt(pb) + off, dw[4 * k4], dw[4 * k4 + 1], dw[4 * k4 + 2], dw[4 * k4 + 3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(L::kDsFull + (it & 1)));
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ dQ drain + dK/dV epilogue
    const int wq = warp - 8;
    const int r = (wq << 5) + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    bool ok = true;
    for (int it = 0; it < nit; ++it) {
      const int q0 = q_block(it) * BM;
      float* dq_acc = args.dq_acc + (size_t)q_head(it) * N * D;
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
      const size_t out_row = ((size_t)bh_kv * Nk + key) * D + half * DH;
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
          if (key < Nk) {
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

// D_i = sum_c dO_ic O_ic per row, L_i * log2(e) copied next to it, and the fp32
// dQ accumulator set to zero.  Both row vectors are padded per head to Npad rows
// (a multiple of 128) so the main kernels read whole aligned blocks; padding rows
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
      if (args.dq_acc && valid[k]) {
        float4* z = reinterpret_cast<float4*>(args.dq_acc + (size_t)row[k] * D + part * 8);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
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

int num_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

// D, L log2(e) (both padded per head) and the zeroed dQ accumulator.
template <int D, bool BF16>
cudaError_t launch_pre(const BwdArgs& a, cudaStream_t stream) {
  const long long slots = (long long)a.BH * a.Npad;
  const long long want = (slots * D / 256 + 7) / 8;  // warp steps / warps per block
  const int grid = (int)std::max<long long>(1, std::min<long long>(want, (long long)num_sms() * 16));
  fa_bwd_pre_kernel<D, BF16><<<grid, 256, 0, stream>>>(a, slots);
  return cudaGetLastError();
}

// dQ = scale * dQ accumulator, rounded to the input type.
template <int D, bool BF16>
cudaError_t launch_convert(const BwdArgs& a, cudaStream_t stream) {
  const long long n8 = (long long)a.BH * a.N * D / 8;
  const int grid = (int)std::min<long long>((n8 + 255) / 256, (long long)num_sms() * 16);
  fa_bwd_dq_convert_kernel<BF16><<<grid, 256, 0, stream>>>(a, n8);
  return cudaGetLastError();
}

template <int D, int DH, int BM, bool DQT, int STG, int NPB, bool BF16>
cudaError_t launch_main(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout,
                        const BwdArgs& a, cudaStream_t stream) {
  using L = BwdLayout<D, DH, BM, DQT, STG, NPB>;
  auto kern = fa_bwd_kernel<D, DH, BM, DQT, STG, NPB, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kAlloc);
  if (e != cudaSuccess) return e;
  const long long nkb = (a.Nk + kBN - 1) / kBN;
  const long long grid = nkb * a.BHkv * (D / DH);
  profile_mark_begin(stream);
  kern<<<(unsigned)grid, kBwdThreads, L::kAlloc, stream>>>(q, k, v, dout, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  profile_mark_end(stream, 1);
  return cudaSuccess;
}

// The three launches of the backward pass, in order on `stream`.
template <int D, bool BF16, typename Main>
cudaError_t launch_all(const BwdArgs& a, cudaStream_t stream, Main main) {
  cudaError_t e = launch_pre<D, BF16>(a, stream);
  if (e != cudaSuccess) return e;
  if ((e = main()) != cudaSuccess) return e;
  return launch_convert<D, BF16>(a, stream);
}

}  // namespace

int bwd_query_rows(int d) { return d == 256 ? 64 : 128; }

bool bwd_needs_dq_acc(int d) { return d == 256; }

cudaError_t launch_bwd(int d, bool bf16, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& dout, const BwdArgs& a, cudaStream_t stream) {
  switch (d) {
    case 64:
    case 128: {
      // No dQ accumulator: the dQ kernel writes dQ itself, so the pre-pass only
      // computes D and L log2(e) and no conversion pass follows.
      BwdArgs a2 = a;
      a2.dq_acc = nullptr;
      cudaError_t e = d == 64 ? (bf16 ? launch_pre<64, true>(a2, stream) : launch_pre<64, false>(a2, stream))
                              : (bf16 ? launch_pre<128, true>(a2, stream) : launch_pre<128, false>(a2, stream));
      if (e != cudaSuccess) return e;
      return launch_bwd_main_sq(d, bf16, q, k, v, dout, a2, stream);
    }
    case 256:
      return bf16 ? launch_all<256, true>(a, stream, [&] {
        return launch_main<256, 128, 64, true, 1, 1, true>(q, k, v, dout, a, stream);
      })
                  : launch_all<256, false>(a, stream, [&] {
                      return launch_main<256, 128, 64, true, 1, 1, false>(q, k, v, dout, a, stream);
                    });
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace fa
