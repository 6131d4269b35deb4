// Forward pass of exact attention for sm_103a: O = softmax(Q K^T * scale + mask) V and
// the per-row logsumexp L, in one fused kernel.
//
// The method is the one of the page "FlashAttention — فلاش أتنشن": Q, K and V are
// split into tiles held on chip (section "Tiling and block processing"), every
// query row keeps a running maximum and a running sum of exponentials that are
// updated block by block and give the exact softmax (section "Online softmax"),
// and the matrix products, the mask, the softmax and the product with V happen
// in one kernel that writes only the final output (section "Fusion of the
// operations into one CUDA kernel").  Work is split over (batch*head, query
// block) so that one head spreads over many SMs (page "FlashAttention-2 —
// فلاش أتنشن-2", section "Technical architecture", item 2).
//
// GB300 mapping (one CTA per 128*NQ query rows):
//   warp 4*NQ     TMA producer: Q sub-tiles once, then K_0, V_0, K_1, V_1, ...
//                 through a ring of STAGES shared-memory slots.
//   warp 4*NQ+1   MMA issuer (one thread): S_t = Q_t K_j^T into TMEM, then
//                 O_t += P_t V_j with P_t read straight from TMEM (tcgen05.mma
//                 with the A operand in tensor memory), so P never touches
//                 shared memory.  Per block the order is P_0 V_j, S_0(j+1),
//                 P_1 V_j, S_1(j+1): the tensor pipe runs in order, so S_t(j+1)
//                 overwrites the TMEM columns of P_t only after P_t V_j has read
//                 them, and while softmax warpgroup t works on one block the
//                 tensor cores work on the other sub-tile.
//   warp 4*NQ+2   (d = 64 only) second MMA issuer.  One thread issues a
//                 tcgen05.mma only about every 50 cycles, more than the 32 an
//                 N = 64 product takes, so at d = 64, where P has TMEM columns of
//                 its own, warp 4*NQ+1 issues the score products and this warp the
//                 P V products; the two share no TMEM columns.
//   warps 4t..4t+3  softmax for query sub-tile t: thread r owns query row r and
//                 TMEM lane r, so every row reduction stays inside one thread.
//                 Scores are taken to base 2 with one FMA (scale*log2 e folded in),
//                 exponentiated with ex2, summed, rounded to 16 bits and stored
//                 back into the first half of the row's S columns as P.  The
//                 row's reference maximum only moves when the new maximum exceeds
//                 it by more than 8 (base 2); otherwise the old one is kept, which
//                 leaves the result exact (all terms share one reference) and
//                 skips the rescale of O.  When it moves, the thread rescales its
//                 O row in TMEM before releasing P.
//   epilogue      O / l rounded to 16 bits, staged in the dead Q tile, stored by TMA;
//                 L = m*scale + ln(l) written per row.
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;                 // query rows per sub-tile (= TMEM lanes)
constexpr int kBN = 128;                 // keys per block
constexpr uint32_t kPanelBytes = 16384;  // 128 rows x 128 B: one 64-column swizzled panel

template <int D, int NQ, int STAGES>
struct FwdLayout {
  static constexpr int kPanels = D / 64;
  static constexpr uint32_t kTileBytes = kPanels * kPanelBytes;  // 128 rows x D 16-bit values
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kRing = kQ + NQ * kTileBytes;
  static constexpr uint32_t kBar = kRing + STAGES * kTileBytes;
  // One sub-tile (NQ = 1) keeps two score buffers, used by alternate key blocks, so
  // the scores of block j+1 are computed while the softmax works on block j.
  static constexpr int kSBufs = NQ == 1 ? 2 : NQ;
  // Two sub-tiles at d = 64 leave 128 TMEM columns free: each sub-tile's P goes to
  // its own 64 columns there instead of into its S columns, so S(j+1) may overwrite
  // S(j) as soon as the softmax has read it, not only after P(j) V has run.
  static constexpr bool kSepP = NQ == 2 && D == 64;
  // MMA issuers.  One thread issues a tcgen05.mma only about every 50 cycles, and
  // an N = 64 product executes in 32, so with separate P buffers (which leave the
  // score products and the P V products no TMEM columns in common) one warp issues
  // the score products and another the P V products.
  static constexpr int kIssuers = kSepP ? 2 : 1;
  static constexpr int kThreads = (4 * NQ + 1 + kIssuers) * 32;
  // barrier indices
  static constexpr int kQFull = 0;
  static constexpr int kFull = 1;
  static constexpr int kEmpty = kFull + STAGES;
  static constexpr int kSFull = kEmpty + STAGES;  // one per score buffer
  static constexpr int kPFull = kSFull + kSBufs;  // one per score buffer
  static constexpr int kODone = kPFull + kSBufs;  // one per sub-tile
  static constexpr int kDrain = kODone + NQ;
  static constexpr int kSFree = kDrain + 1;        // kSepP: one per sub-tile, S read out
  static constexpr int kNumBars = kSFree + (kSepP ? NQ : 0);
  static constexpr uint32_t kTmemSlot = kBar + kNumBars * 8;
  static constexpr uint32_t kBytes = kTmemSlot + 16;
  static constexpr uint32_t kAlloc = kBytes + 1024;  // room to align the base to 1024 B
  // TMEM columns: score buffer b (P in its first 64 columns) at 128*b, O_t after all
  // score buffers.  With NQ = 2 sub-tile t owns buffer t.
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t s_col(int b) { return 128u * b; }
  static constexpr uint32_t o_col(int t) { return 128u * kSBufs + (uint32_t)D * t; }
  // where P of sub-tile t is packed: its S columns, or (kSepP) 64 columns after O
  static constexpr uint32_t p_col(int t) { return kSepP ? 128u * kSBufs + (uint32_t)D * NQ + 64u * t : s_col(t); }
  static_assert(128 * kSBufs + D * NQ + (kSepP ? 64 * NQ : 0) <= 512, "TMEM budget");
  static_assert(kBytes + 1024 <= 232448, "shared memory budget");
};

template <int D, int NQ, int STAGES, bool BF16>
__global__ void __launch_bounds__(FwdLayout<D, NQ, STAGES>::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdArgs args) {
  using L = FwdLayout<D, NQ, STAGES>;
  constexpr int kWarpTma = 4 * NQ;
  constexpr int kWarpMma = 4 * NQ + 1;  // MMA issuer (separate P buffers: score products; P V in the next warp)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
  auto sQ = [&](int t) -> uint32_t { return sbase + L::kQ + L::kTileBytes * t; };
  auto sRing = [&](int s) -> uint32_t { return sbase + L::kRing + L::kTileBytes * s; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = args.N;

  // Heaviest query blocks first (under the causal mask the last blocks see the most
  // keys), so the last wave holds the lightest work; heads in groups of
  // args.head_group, so the K/V tiles of the running CTAs stay in L2.
  int qb, bh;
  grouped_tile(blockIdx.x, args.BH, args.num_qblocks, args.head_group, qb, bh);
  qb = args.num_qblocks - 1 - qb;
  // Key/value head of this query head (grouped-query attention).
  const int bh_kv = (bh / args.H) * (args.H / args.group) + (bh % args.H) / args.group;
  const int row0 = qb * (kBM * NQ);
  const int Nk = args.Nk;
  const int koff = Nk - N;  // causal mask: key j visible to query i iff j <= i + koff

  // Key blocks each sub-tile visits (0 for a sub-tile past the end or with no visible key).
  int nblk[NQ];
  int nb = 0;
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    const int r0 = row0 + kBM * t;
    const int last_key = args.causal ? min(r0 + kBM - 1 + koff, Nk - 1) : Nk - 1;
    nblk[t] = (r0 >= N || last_key < 0) ? 0 : last_key / kBN + 1;
    nb = max(nb, nblk[t]);
  }

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kQFull), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(L::kFull + s), 1);
      mbar_init(bar(L::kEmpty + s), 1);
    }
    for (int b = 0; b < L::kSBufs; ++b) {
      mbar_init(bar(L::kSFull + b), 1);
      mbar_init(bar(L::kPFull + b), kBM / 32);  // one arrival per softmax warp
    }
    for (int t = 0; t < NQ; ++t) mbar_init(bar(L::kODone + t), 1);
    if constexpr (L::kSepP)
      for (int t = 0; t < NQ; ++t) mbar_init(bar(L::kSFree + t), kBM / 32);
    mbar_init(bar(L::kDrain), L::kIssuers);
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
    tma_prefetch_desc(&tm_o);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);
  debug_context(tmem, args.err);
  const Extent3 ext_q{D, N, args.BH}, ext_kv{D, Nk, args.BH / args.group};

  // Ring items in the order the MMA warp consumes them.  Two sub-tiles: K_0, V_0,
  // K_1, V_1, ...  One sub-tile (two score buffers), or two with separate P buffers:
  // K_0, K_1, V_0, K_2, V_1, K_3, ..., V_{nb-1}, the next block's K before this
  // block's V.
  auto ring_item = [&](int e, bool& is_v) -> int {
    if constexpr (NQ != 1 && !L::kSepP) {
      is_v = e & 1;
      return e >> 1;
    } else {
      if (e == 0) { is_v = false; return 0; }
      if (e == 2 * nb - 1) { is_v = true; return nb - 1; }
      is_v = !(e & 1);
      return (e & 1) ? (e + 1) >> 1 : (e >> 1) - 1;
    }
  };

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_expect_tx(bar(L::kQFull), NQ * L::kTileBytes);
#pragma unroll
      for (int t = 0; t < NQ; ++t)
#pragma unroll
        for (int p = 0; p < L::kPanels; ++p)
          tma_load_box(sQ(t) + p * kPanelBytes, &tm_q, bar(L::kQFull), 64 * p, row0 + kBM * t, bh, ext_q, args.err);
      int n = 0;  // ring loads issued
      for (int e = 0; e < 2 * nb; ++e) {
        const int s = e % STAGES, u = e / STAGES;
        if (u > 0 && !mbar_wait(bar(L::kEmpty + s), (u - 1) & 1, args.err, kErrTimeoutRing)) break;
        mbar_expect_tx(bar(L::kFull + s), L::kTileBytes);
        bool is_v;
        const int blk = ring_item(e, is_v);
        const CUtensorMap* m = is_v ? &tm_v : &tm_k;
#pragma unroll
        for (int p = 0; p < L::kPanels; ++p)
          tma_load_box(sRing(s) + p * kPanelBytes, m, bar(L::kFull + s), 64 * p, kBN * blk, bh_kv, ext_kv, args.err);
        ++n;
      }
      // Every copy this thread issued lands before the CTA exits, even when the
      // consumers gave up after a timeout elsewhere (bounded waits, abort ignored).
      mbar_wait(bar(L::kQFull), 0, args.err, kErrTimeoutTma, false);
      for (int s = 0; s < STAGES; ++s)
        if (n > s) mbar_wait(bar(L::kFull + s), ((n - 1 - s) / STAGES) & 1, args.err, kErrTimeoutTma, false);
    }
  } else if (warp >= kWarpMma) {
    // ------------------------------------------------------------ MMA issuer(s)
    if (lane == 0) {
      constexpr uint32_t kIdS = make_idesc_f16(BF16, kBM, kBN, false, false);
      constexpr uint32_t kIdPV = make_idesc_f16(BF16, kBM, D, false, true);
      constexpr uint32_t kHi = sdesc_hi_sw128(1024);  // every operand here: 8-row groups 1024 B apart
      // S of sub-tile t into score buffer `buf`, K from ring slot s
      auto issue_s = [&](int t, int buf, int s) {
        const uint32_t a0 = sdesc_lo(sQ(t), 16), b0 = sdesc_lo(sRing(s), 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4;
          mma_ss_lohi(tmem + L::s_col(buf), a0 + off, kHi, b0 + off, kHi, kIdS, kk > 0);
        }
      };
      // O_t += P V_j, P packed in score buffer `buf`, V from ring slot s
      auto issue_pv = [&](int t, int buf, int s, int j) {
        const uint32_t b0 = sdesc_lo(sRing(s), kPanelBytes);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)  // P: 8 TMEM columns (16 keys) per step
          mma_ts_lohi(tmem + L::o_col(t), tmem + (L::kSepP ? L::p_col(t) : L::s_col(buf)) + 8 * kk,
                      b0 + ((kk * 2048) >> 4), kHi, kIdPV, (j > 0 || kk > 0) ? 1u : 0u);
      };
      auto wait_full = [&](int e) -> bool {
        return mbar_wait(bar(L::kFull + e % STAGES), (e / STAGES) & 1, args.err, kErrTimeoutTma);
      };
      if constexpr (L::kSepP) {
        // Two issuers.  Warp kWarpMma: S_0(0), S_1(0), then S_t(j+1) once the softmax
        // has read S_t(j), and it releases the K items.  Warp kWarpMma + 1: P_t(j) V_j
        // once P_t(j) is packed, and it releases the V items.  Ring item of K(j+1):
        // 2j + 1; of V_j: 2j + 2, or 2nb - 1 for the last.  The P V issuer's test of a
        // V item's slot is never two phases stale: the slot last held either one of
        // its own V items (seen in order) or a K item that an S(j') read before the
        // P(j') this issuer has already waited for.
        bool ok = nb > 0;
        if (warp == kWarpMma) {
          ok = ok && mbar_wait(bar(L::kQFull), 0, args.err, kErrTimeoutTma) && wait_full(0);
          if (ok) {
            tc_fence_after();
            for (int t = 0; t < NQ; ++t)
              if (nblk[t] > 0) {
                issue_s(t, t, 0);
                mma_commit(bar(L::kSFull + t));
              }
            mma_commit(bar(L::kEmpty + 0));
          }
          for (int j = 0; ok && j + 1 < nb; ++j) {
            const int ek = 2 * j + 1;
            if (!(ok = wait_full(ek))) break;
            for (int t = 0; t < NQ; ++t)
              if (j + 1 < nblk[t]) {
                if (!(ok = mbar_wait(bar(L::kSFree + t), j & 1, args.err, kErrTimeoutSoftmax))) break;
                tc_fence_after();
                issue_s(t, t, ek % STAGES);
                mma_commit(bar(L::kSFull + t));
              }
            if (!ok) break;
            mma_commit(bar(L::kEmpty + ek % STAGES));
          }
        } else {
          for (int j = 0; ok && j < nb; ++j) {
            const int ev = (j == nb - 1) ? 2 * nb - 1 : 2 * j + 2;
            if (!(ok = wait_full(ev))) break;
            for (int t = 0; t < NQ; ++t)
              if (j < nblk[t]) {
                if (!(ok = mbar_wait(bar(L::kPFull + t), j & 1, args.err, kErrTimeoutSoftmax))) break;
                tc_fence_after();
                issue_pv(t, t, ev % STAGES, j);
                mma_commit(bar(L::kODone + t));
              }
            if (!ok) break;
            mma_commit(bar(L::kEmpty + ev % STAGES));
          }
        }
      } else if constexpr (NQ == 1) {
        bool ok = nb > 0 && mbar_wait(bar(L::kQFull), 0, args.err, kErrTimeoutTma) && wait_full(0);
        // S(0) S(1) | P(j) V_j, S(j+2) | ...: S(j+2) overwrites buffer j & 1 only after
        // P(j) V_j has read it (one thread's MMAs execute in issue order).  Ring item
        // of S(j): 0 for j = 0, else 2j - 1; of P(j) V_j: 2j + 2, or 2nb - 1 for the last.
        if (ok) {
          tc_fence_after();
          issue_s(0, 0, 0);
          mma_commit(bar(L::kSFull + 0));
          mma_commit(bar(L::kEmpty + 0));
          if (nb > 1 && (ok = wait_full(1))) {
            tc_fence_after();
            issue_s(0, 1, 1 % STAGES);
            mma_commit(bar(L::kSFull + 1));
            mma_commit(bar(L::kEmpty + 1 % STAGES));
          }
        }
        for (int j = 0; ok && j < nb; ++j) {
          const int b = j & 1;
          const int ev = (j == nb - 1) ? 2 * nb - 1 : 2 * j + 2;
          if (!(ok = mbar_wait(bar(L::kPFull + b), (j >> 1) & 1, args.err, kErrTimeoutSoftmax) && wait_full(ev)))
            break;
          tc_fence_after();
          issue_pv(0, b, ev % STAGES, j);
          mma_commit(bar(L::kODone + 0));
          mma_commit(bar(L::kEmpty + ev % STAGES));
          if (j + 2 < nb) {
            const int ek = 2 * j + 3;
            if (!(ok = wait_full(ek))) break;
            tc_fence_after();
            issue_s(0, b, ek % STAGES);
            mma_commit(bar(L::kSFull + b));
            mma_commit(bar(L::kEmpty + ek % STAGES));
          }
        }
      } else {
      bool ok = nb > 0 && mbar_wait(bar(L::kQFull), 0, args.err, kErrTimeoutTma) && wait_full(0);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < NQ; ++t)
          if (nblk[t] > 0) {
            issue_s(t, t, 0);
            mma_commit(bar(L::kSFull + t));
          }
        mma_commit(bar(L::kEmpty + 0));
      }
      for (int j = 0; ok && j < nb; ++j) {
        const int ev = 2 * j + 1, ek = 2 * j + 2;  // ring items of V_j and K_{j+1}
        const bool next = j + 1 < nb;
        ok = wait_full(ev) && (!next || wait_full(ek));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
          if (j < nblk[t]) {
            ok = mbar_wait(bar(L::kPFull + t), j & 1, args.err, kErrTimeoutSoftmax);
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, t, ev % STAGES, j);
            mma_commit(bar(L::kODone + t));
          }
          if (t == NQ - 1) mma_commit(bar(L::kEmpty + ev % STAGES));  // last reader of V_j issued
          if (j + 1 < nblk[t]) {
            issue_s(t, t, ek % STAGES);  // in order after P_t V_j, which read these columns
            mma_commit(bar(L::kSFull + t));
          }
        }
        if (!ok) break;
        if (next) mma_commit(bar(L::kEmpty + ek % STAGES));
      }
      }
      // Every MMA must have finished before TMEM can be released.
      mma_commit(bar(L::kDrain));
      mbar_wait(bar(L::kDrain), 0, args.err, kErrTimeoutMma, false);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int t = warp >> 2;
    const int r = ((warp & 3) << 5) + lane;  // row inside the sub-tile == TMEM lane
    const int q_row = row0 + kBM * t + r;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + lane_base + L::o_col(t);
    const float c = args.scale_log2;
    const int key_limit = args.causal ? min(q_row + koff, Nk - 1) : Nk - 1;  // last key this row sees
    float m = -INFINITY;  // reference maximum (raw score units)
    float l = 0.f;        // running sum of 2^((s - m) c)
    bool ok = true;
    const int my_blocks = nblk[t];
    for (int j = 0; j < my_blocks; ++j) {
      // score buffer of this block and the parity of its barriers' phase
      const int buf = NQ == 1 ? (j & 1) : t;
      const uint32_t par = NQ == 1 ? ((j >> 1) & 1) : (j & 1);
      const uint32_t tS = tmem + lane_base + L::s_col(buf);
      ok = warp_wait(bar(L::kSFull + buf), par, args.err, kErrTimeoutMma);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int h = 0; h < 4; ++h) tmem_ld_32x32b_x32(tS + 32 * h, sr[h]);
      tmem_wait_ld();
#pragma unroll
      for (int h = 0; h < 4; ++h) reg_fence32(sr[h]);
      if constexpr (L::kSepP) {
        tc_fence_before();
        warp_arrive(bar(L::kSFree + t));  // S_t may be overwritten by the next block's scores
      }

      float s[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(sr[i >> 5][i & 31]);
      const int nvalid = key_limit - kBN * j + 1;  // keys kBN*j .. kBN*j+nvalid-1 are visible
      if (nvalid < kBN) {
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = (i < nvalid) ? s[i] : -INFINITY;
      }
      // Row maximum: four independent chains of 3-input max.
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int i = 4; i < 124; i += 8) {
        mx0 = max3f(mx0, s[i], s[i + 1]);
        mx1 = max3f(mx1, s[i + 2], s[i + 3]);
        mx2 = max3f(mx2, s[i + 4], s[i + 5]);
        mx3 = max3f(mx3, s[i + 6], s[i + 7]);
      }
      mx0 = max3f(mx0, s[124], s[125]);
      mx1 = max3f(mx1, s[126], s[127]);
      const float m_new = max3f(m, max3f(mx0, mx1, mx2), mx3);
      // Keep the old reference unless the maximum grew by more than 8 (base 2).
      const float m_use = (m == -INFINITY || (m_new - m) * c > 8.f) ? m_new : m;
      const float mc = (m_use == -INFINITY) ? 0.f : m_use * c;
      const float alpha = ex2_approx(fmaf(m, c, -mc));  // 0 when m = -inf
      // p = 2^(s c - m c): packed FMA for the exponent, ex2, packed adds for the row
      // sum.  P (two 16-bit values per column) goes into its own 64 columns (separate
      // P buffers) or into the first 64 columns of S_t, half a row at a time so the
      // packed words do not all stay live.
      bool o_done = false;
      const uint32_t tP = L::kSepP ? tmem + lane_base + L::p_col(t) : tS;
      float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
      if constexpr (L::kSepP) {
        // P(j) overwrites P(j-1) in its own columns: wait until P(j-1) V has run,
        // but only after the first half row of exponentials, which overlap that
        // product.  (P(j) V cannot be issued before P(j) is packed, so ODone is at
        // most one phase ahead of this wait: its parity is unambiguous.)
        uint32_t pa[32], pb[32];
#pragma unroll
        for (int i = 0; i < 64; i += 4) {
          float x0, x1, x2, x3;
          fma2(s[i], s[i + 1], c, -mc, x0, x1);
          fma2(s[i + 2], s[i + 3], c, -mc, x2, x3);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
          add2(l0, l1, p0, p1);
          add2(l2, l3, p2, p3);
          pa[i >> 1] = pack2<BF16>(p0, p1);
          pa[(i >> 1) + 1] = pack2<BF16>(p2, p3);
        }
        if (j > 0) {
          ok = warp_wait(bar(L::kODone + t), (j - 1) & 1, args.err, kErrTimeoutMma);
          if (!ok) break;
          tc_fence_after();
          o_done = true;
        }
        tmem_st_32x32b_x32(tP, pa);
#pragma unroll
        for (int i = 64; i < 128; i += 4) {
          float x0, x1, x2, x3;
          fma2(s[i], s[i + 1], c, -mc, x0, x1);
          fma2(s[i + 2], s[i + 3], c, -mc, x2, x3);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
          add2(l0, l1, p0, p1);
          add2(l2, l3, p2, p3);
          pb[(i - 64) >> 1] = pack2<BF16>(p0, p1);
          pb[((i - 64) >> 1) + 1] = pack2<BF16>(p2, p3);
        }
        tmem_st_32x32b_x32(tP + 32, pb);
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pw[32];
#pragma unroll
          for (int i = 64 * h; i < 64 * h + 64; i += 4) {
            float x0, x1, x2, x3;
            fma2(s[i], s[i + 1], c, -mc, x0, x1);
            fma2(s[i + 2], s[i + 3], c, -mc, x2, x3);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            add2(l0, l1, p0, p1);
            add2(l2, l3, p2, p3);
            pw[(i % 64) >> 1] = pack2<BF16>(p0, p1);
            pw[((i % 64) >> 1) + 1] = pack2<BF16>(p2, p3);
          }
          tmem_st_32x32b_x32(tP + 32 * h, pw);
        }
      }
      l = l * alpha + ((l0 + l1) + (l2 + l3));
      tmem_wait_st();
      // O_t is rescaled only when the reference moved, after the previous P V is done.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        if (!o_done) {
          ok = warp_wait(bar(L::kODone + t), (j - 1) & 1, args.err, kErrTimeoutMma);
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tO + 32 * ch, o);
          tmem_wait_ld();
          reg_fence32(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st_32x32b_x32(tO + 32 * ch, o);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      warp_arrive(bar(L::kPFull + buf));
      m = m_use;
    }
    const bool has_rows = row0 + kBM * t < N;
    if (ok && has_rows) {
      // A sub-tile whose rows see no key at all writes O = 0 and L = -inf; it still
      // waits for its Q tile to land before reusing that shared memory.
      // With two score buffers (NQ = 1) up to two P V products can still be in flight
      // here, so the parity of ODone would be ambiguous: wait for the one-phase
      // drain barrier the MMA warp commits after its last product instead.
      if (my_blocks == 0)
        ok = warp_wait(bar(L::kQFull), 0, args.err, kErrTimeoutTma);
      else if constexpr (NQ == 1)
        ok = warp_wait(bar(L::kDrain), 0, args.err, kErrTimeoutMma);
      else
        ok = warp_wait(bar(L::kODone + t), (my_blocks - 1) & 1, args.err, kErrTimeoutMma);
      if (ok) {
        tc_fence_after();
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        if (q_row < N) {
          args.lse[(size_t)bh * N + q_row] = (l > 0.f) ? m * args.scale + logf(l) : -INFINITY;
        }
        // O / l -> 16-bit, staged in the Q tile of this sub-tile (its last use is over).
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          if (my_blocks > 0) {
            tmem_ld_32x32b_x32(tO + 32 * ch, o);
            tmem_wait_ld();
            reg_fence32(o);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
          }
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int chunk = ch * 4 + k4;  // 16-byte chunk index along the row
            const int b = k4 * 8;
            st_shared_v4(sQ(t) + (chunk >> 3) * kPanelBytes + sw128_offset(r, chunk & 7),
                         pack2<BF16>(__uint_as_float(o[b]) * inv_l, __uint_as_float(o[b + 1]) * inv_l),
                         pack2<BF16>(__uint_as_float(o[b + 2]) * inv_l, __uint_as_float(o[b + 3]) * inv_l),
                         pack2<BF16>(__uint_as_float(o[b + 4]) * inv_l, __uint_as_float(o[b + 5]) * inv_l),
                         pack2<BF16>(__uint_as_float(o[b + 6]) * inv_l, __uint_as_float(o[b + 7]) * inv_l));
          }
        }
        fence_proxy_async_smem();
      }
    }
    // All 128 threads of this sub-tile reach the barrier (ok or not), then one stores.
    named_bar_sync(1 + t, kBM);
    if (ok && has_rows && r == 0) {
#pragma unroll
      for (int p = 0; p < L::kPanels; ++p)
        tma_store_box(&tm_o, sQ(t) + p * kPanelBytes, 64 * p, row0 + kBM * t, bh, ext_q, args.err);
      tma_store_commit();
      tma_store_wait0();
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (kDebug) {
    // every barrier completed as many phases as the protocol says
    if (threadIdx.x == 0 && no_abort(args.err)) {
      check_phase(bar(L::kQFull), 1, args.err, L::kQFull);
      for (int s = 0; s < STAGES; ++s) {
        check_phase(bar(L::kFull + s), count_mod(2 * nb, s, STAGES), args.err, L::kFull + s);
        check_phase(bar(L::kEmpty + s), count_mod(2 * nb, s, STAGES), args.err, L::kEmpty + s);
      }
      for (int b = 0; b < L::kSBufs; ++b) {
        const uint32_t n_s = NQ == 1 ? count_mod(nb, b, 2) : (uint32_t)nblk[b];
        check_phase(bar(L::kSFull + b), n_s, args.err, L::kSFull + b);
        check_phase(bar(L::kPFull + b), n_s, args.err, L::kPFull + b);
      }
      for (int t = 0; t < NQ; ++t) check_phase(bar(L::kODone + t), nblk[t], args.err, L::kODone + t);
      check_phase(bar(L::kDrain), 1, args.err, L::kDrain);
      if constexpr (L::kSepP)
        for (int t = 0; t < NQ; ++t) check_phase(bar(L::kSFree + t), nblk[t], args.err, L::kSFree + t);
    }
  }
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int D, int NQ, int STAGES, bool BF16>
cudaError_t launch_fwd_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                         const FwdArgs& a, cudaStream_t stream) {
  using L = FwdLayout<D, NQ, STAGES>;
  auto kern = fa_fwd_kernel<D, NQ, STAGES, BF16>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kAlloc);
  if (err != cudaSuccess) return err;
  const long long grid = (long long)a.num_qblocks * a.BH;
  profile_mark_begin(stream);
  kern<<<(unsigned)grid, L::kThreads, L::kAlloc, stream>>>(q, k, v, o, a);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  profile_mark_end(stream, kProfileFwd);
  return cudaSuccess;
}

}  // namespace

int fwd_rows_per_cta(int d, long long BH, int N, int num_sms) {
  if (d == 256) return kBM;
  const long long ctas = BH * (((long long)N + 2 * kBM - 1) / (2 * kBM));
  return ctas < num_sms ? kBM : 2 * kBM;
}

// Two 128-row sub-tiles a CTA (eight softmax warps keep the MUFU and the tensor pipe
// busy) unless the problem is too small to fill the GPU with such CTAs; then one
// sub-tile a CTA with two score buffers, as at d = 256 (measured: faster for grids
// under one wave, much slower for larger ones).
cudaError_t launch_fwd(int d, bool bf16, int rows, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& o, const FwdArgs& a, cudaStream_t stream) {
  const bool one = rows == kBM;
  switch (d) {
    case 64:
      if (one)
        return bf16 ? launch_fwd_t<64, 1, 8, true>(q, k, v, o, a, stream)
                    : launch_fwd_t<64, 1, 8, false>(q, k, v, o, a, stream);
      return bf16 ? launch_fwd_t<64, 2, 8, true>(q, k, v, o, a, stream)
                  : launch_fwd_t<64, 2, 8, false>(q, k, v, o, a, stream);
    case 128:
      if (one)
        return bf16 ? launch_fwd_t<128, 1, 5, true>(q, k, v, o, a, stream)
                    : launch_fwd_t<128, 1, 5, false>(q, k, v, o, a, stream);
      return bf16 ? launch_fwd_t<128, 2, 5, true>(q, k, v, o, a, stream)
                  : launch_fwd_t<128, 2, 5, false>(q, k, v, o, a, stream);
    case 256:
      return bf16 ? launch_fwd_t<256, 1, 2, true>(q, k, v, o, a, stream)
                  : launch_fwd_t<256, 1, 2, false>(q, k, v, o, a, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace fa
