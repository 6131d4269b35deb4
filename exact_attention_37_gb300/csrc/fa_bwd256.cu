// Backward pass for head dimension 256: one launch of three kinds of CTA, no
// atomics, so dQ, dK and dV are bitwise reproducible.
//
// Like the d = 64 / 128 kernels it rebuilds the probabilities block by block from
// Q, K and the forward pass's logsumexp (page "FlashAttention — فلاش أتنشن",
// section "Tiling and block processing") and applies the chain-rule derivatives
// of the attention formula (same page, section "The problem of standard
// attention"):
//
//   P = 2^(S scale log2 e - L log2 e),   dP = dO V^T,   dS = P o (dP - D),
//   dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K.
//
// At d = 256 a 128-row accumulator of one gradient fills half of the tensor
// memory (256 of 512 columns) and a 128-row operand tile takes 64 KB of shared
// memory, so dK and dV cannot both stay in one CTA next to the score tiles.  The
// work is therefore split by output:
//
//   dK CTA  (key/value head, 128-key block): keys on TMEM lanes.  K is copied once
//           into tensor memory and is the A operand of S^T = K Q^T; V stays in
//           shared memory for dP^T = V dO^T; Q and dO stream in 64-row tiles;
//           dK += dS^T Q with dS^T packed in tensor memory.
//   dV CTA  (same block): only S^T = K Q^T and dV += P^T dO, so it streams
//           128-row Q and dO tiles (N = 128 score products) with K in shared
//           memory, and keeps P^T apart from S^T in tensor memory so the next
//           block's scores run while the elementwise warps exponentiate.
//   dQ CTA  (query head, 128-row query block): queries on TMEM lanes.  Q in tensor
//           memory is the A operand of S = Q K^T; dO stays in shared memory for
//           dP = dO V^T; K and V stream in 64-key tiles; dQ += dS K.
//
// The dK and dQ CTAs run the same program on swapped operands (K, V, Q, dO) <->
// (Q, dO, K, V), with the per-column (dK) or per-row (dQ) L and D.  The key-block
// CTAs are the key-block parallelism of page "FlashAttention-2 — فلاش أتنشن-2",
// section "Technical architecture", item 2; each visits the query blocks of every
// query head of its key/value head's group, so the group sums of dK and dV stay
// in tensor memory.  The dK and dV CTAs of one key block are adjacent in the
// grid (they stream the same Q and dO tiles), and the dQ CTAs follow them.
//
// dK and dQ CTAs: tensor memory columns 0-127 hold the resident operand (K or Q,
// 16-bit pairs), 128-191 and 192-255 the S and dP buffers, 256-511 the gradient
// accumulator; shared memory holds the stationary 128-row tile (64 KB), three
// 64-row stages of the operand read by the score and gradient products, two of
// the operand read by the second product (32 KB each), and the L, D values of
// each query stage.  dV CTAs lay out their own (below).  Warps: 0-7 elementwise
// (two warpgroups, half of the tile columns each), 8 TMA, 9 MMA, 10 a second MMA
// issuer in dK and dQ CTAs.  One thread issues a tcgen05.mma only about every 50
// cycles, more than the 32 an N = 64 score product takes, so there warp 9 issues
// the score products (S buffer, read only by the elementwise warps) and warp 10
// the dP and gradient products (dP buffer, where dS is packed for the gradient).
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kRoleDK = 0, kRoleDV = 1, kRoleDQ = 2;
constexpr int kRes = 128;                    // rows of the resident operand (= TMEM lanes)
constexpr int kBlk = 64;                     // rows of a streamed tile
constexpr uint32_t kP64 = 64 * 128;          // one 64-column panel of 64 rows (8 KB)
constexpr uint32_t kP128 = 128 * 128;        // one 64-column panel of 128 rows (16 KB)
constexpr uint32_t kT64 = 4 * kP64;          // 64 rows x 256 columns (32 KB)
constexpr uint32_t kT128 = 4 * kP128;        // 128 rows x 256 columns (64 KB)
constexpr int kZStages = 3, kWStages = 2;
constexpr int kEwWarps = 8;
constexpr int kWarpTma = 8, kWarpMma = 9;
constexpr int kWarpMma2 = 10;  // dK and dQ CTAs: the second MMA issuer (idle in dV CTAs)
constexpr int kThreads = 11 * 32;

// shared memory
constexpr uint32_t kSmY = 0;
constexpr uint32_t kSmZ = kT128;
constexpr uint32_t kSmW = kSmZ + kZStages * kT64;
constexpr uint32_t kSmLD = kSmW + kWStages * kT64;          // per Z stage: 64 L log2 e, then 64 D
constexpr uint32_t kSmBar = kSmLD + kZStages * 512;
enum : int {
  kYFull = 0,
  kAReady = 1,                 // the resident operand is in tensor memory
  kZFull = 2,                  // three
  kZEmpty = kZFull + kZStages,
  kWFull = kZEmpty + kZStages, // two
  kWEmpty = kWFull + kWStages,
  kSReady = kWEmpty + kWStages,  // two (the dV CTA alternates; the others use the first)
  kSFree = kSReady + 2,        // the scores have been read out of tensor memory
  kDpReady = kSFree + 1,
  kDsFull = kDpReady + 1,      // dS packed into the dP buffer
  kPFull = kDsFull + 1,        // two: P^T packed into its score buffer (dV CTA)
  kDone = kPFull + 2,          // the last gradient product has completed
  kNumBars
};
constexpr uint32_t kSmTmemSlot = kSmBar + kNumBars * 8;
constexpr uint32_t kSmAlloc = kSmTmemSlot + 16 + 1024;  // + alignment of the dynamic base
static_assert(kSmAlloc <= 232448, "shared memory budget");

// tensor memory columns
constexpr uint32_t kTmA = 0;
constexpr uint32_t kTmBuf0 = 128;
constexpr uint32_t kTmBuf1 = 192;
constexpr uint32_t kTmG = 256;

constexpr uint32_t kHi = sdesc_hi_sw128(1024);  // every operand: 8-row groups 1024 B apart
constexpr uint32_t idesc_score(bool bf16) { return make_idesc_f16(bf16, 128, kBlk, false, false); }
constexpr uint32_t idesc_grad(bool bf16) { return make_idesc_f16(bf16, 128, 256, false, true); }

// Column (relative to a score buffer) of the packed 16-bit pairs of K step kk:
// warpgroup e packs its 32 columns into the first 16 columns of its own range, so
// no warpgroup writes where the other still reads.
__device__ __forceinline__ uint32_t packed_col(int kk) { return 32u * (kk >> 1) + 8u * (kk & 1); }

// Acc (128 x 64) = A B^T, A the resident 128 x 256 operand in tensor memory,
// B a 64-row K-major tile in shared memory.
__device__ __forceinline__ void score_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem, uint32_t idesc) {
  const uint32_t b0 = sdesc_lo(b_smem, 16);
#pragma unroll
  for (int kk = 0; kk < 16; ++kk)
    mma_ts_lohi(d_tmem, a_tmem + 8 * kk, b0 + (((kk >> 2) * kP64 + (kk & 3) * 32) >> 4), kHi, idesc, kk > 0);
}
// Acc (128 x 64) = A B^T, A a 128-row and B a 64-row K-major tile in shared memory.
__device__ __forceinline__ void score_ss(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem, uint32_t idesc) {
  const uint32_t a0 = sdesc_lo(a_smem, 16), b0 = sdesc_lo(b_smem, 16);
#pragma unroll
  for (int kk = 0; kk < 16; ++kk)
    mma_ss_lohi(d_tmem, a0 + (((kk >> 2) * kP128 + (kk & 3) * 32) >> 4), kHi,
                b0 + (((kk >> 2) * kP64 + (kk & 3) * 32) >> 4), kHi, idesc, kk > 0);
}
// Acc (128 x 256) (+)= A B, A (128 x 64) packed in a score buffer, B a 64-row tile
// read MN-major (rows = K, four 64-column panels of N).
__device__ __forceinline__ void grad_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem, uint32_t idesc, bool acc) {
  const uint32_t b0 = sdesc_lo(b_smem, kP64);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_ts_lohi(d_tmem, a_tmem + packed_col(kk), b0 + ((kk * 2048) >> 4), kHi, idesc, (acc || kk > 0) ? 1u : 0u);
}

// TMA load of a 64-row tile (four 64-column boxes) completing `bar`.
__device__ __forceinline__ void load_tile64(uint32_t dst, const CUtensorMap* m, uint32_t bar, int row, int plane,
                                            const Extent3& ext, uint32_t* err) {
#pragma unroll
  for (int p = 0; p < 4; ++p) tma_load_box(dst + p * kP64, m, bar, 64 * p, row, plane, ext, err);
}
// A 128-row tile as two 64-row boxes per panel (the same 128-byte-swizzled layout
// a 128-row box gives: the second box starts 64 rows = 8 KB into the panel).
__device__ __forceinline__ void load_tile128(uint32_t dst, const CUtensorMap* m, uint32_t bar, int row, int plane,
                                             const Extent3& ext, uint32_t* err) {
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    tma_load_box(dst + p * kP128, m, bar, 64 * p, row, plane, ext, err);
    tma_load_box(dst + p * kP128 + kP64, m, bar, 64 * p, row + 64, plane, ext, err);
  }
}

__device__ __forceinline__ void st_global_v4(void* addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void ld_shared_f4(uint32_t addr, float4& v) {
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
}

// First 64-row query block a key block starting at key0 sees (all of them without
// the causal mask).  The last query row sees every key, so it is always a block.
__device__ __forceinline__ int first_qblock(const BwdArgs& a, int key0) {
  return a.causal ? max(0, key0 - (a.Nk - a.N)) / kBlk : 0;
}
// Blocks a CTA streams: for a dK CTA the 64-row query blocks from its first
// visible one, over every query head of its group; for a dQ CTA the 64-key blocks
// its rows see (0 when none: then it writes dQ = 0).
__device__ __forceinline__ int cta_blocks(const BwdArgs& a, int role, int blk) {
  if (role != kRoleDQ) return ((a.N + kBlk - 1) / kBlk - first_qblock(a, blk * kRes)) * a.group;
  const int last = a.causal ? min(a.Nk - 1, blk * kRes + kRes - 1 + (a.Nk - a.N)) : a.Nk - 1;  // last key any row sees
  return last < 0 ? 0 : last / kBlk + 1;
}

template <int ROLE, bool BF16>
__device__ __forceinline__ void bwd256_cta(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                           const CUtensorMap* tm_do, const BwdArgs& args, int blk, int head,
                                           uint8_t* smem, uint32_t sbase, uint32_t tmem) {
  static_assert(ROLE != kRoleDV, "dV CTAs run bwd256_dv_cta");
  constexpr bool kKeyRows = ROLE == kRoleDK;  // keys on TMEM lanes (dK CTA)
  auto bar = [&](int i) -> uint32_t { return sbase + kSmBar + 8u * i; };
  auto sZ = [&](int s) -> uint32_t { return sbase + kSmZ + kT64 * s; };
  auto sW = [&](int s) -> uint32_t { return sbase + kSmW + kT64 * s; };
  auto sLD = [&](int s) -> uint32_t { return sbase + kSmLD + 512u * s; };
  const uint32_t sY = sbase + kSmY;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = args.N, Nk = args.Nk;
  const int koff = Nk - N;  // key j visible to query i iff j <= i + koff

  // ---- this CTA's rows and the blocks it streams
  const int row0 = blk * kRes;  // first key (dK, dV) or query (dQ)
  const int plane_a = head;     // key/value plane (dK, dV) or query plane (dQ)
  const int nit = cta_blocks(args, ROLE, blk);
  const int i_begin = kKeyRows ? first_qblock(args, row0) : 0;
  const int nit_h = kKeyRows ? (N + kBlk - 1) / kBlk - i_begin : 1;  // query blocks per query head (>= 1)
  const int hpb = args.H / args.group;                               // key/value heads per batch entry
  const int bh_q0 = kKeyRows ? (head / hpb) * args.H + (head % hpb) * args.group : 0;  // first query head of the group
  const int bh_kv = kKeyRows ? head : (head / args.H) * (args.H / args.group) + (head % args.H) / args.group;
  // streamed block it: its first row and plane
  auto z_row = [&](int it) { return kKeyRows ? (i_begin + it % nit_h) * kBlk : it * kBlk; };
  auto z_plane = [&](int it) { return kKeyRows ? bh_q0 + it / nit_h : bh_kv; };
  const CUtensorMap* mZ = kKeyRows ? tm_q : tm_k;
  const CUtensorMap* mW = kKeyRows ? tm_do : tm_v;
  const CUtensorMap* mY = kKeyRows ? tm_v : tm_do;
  const Extent3 ext_q{256, N, args.BH}, ext_kv{256, Nk, args.BHkv};
  const Extent3& ext_zw = kKeyRows ? ext_q : ext_kv;  // streamed tiles
  const Extent3& ext_y = kKeyRows ? ext_kv : ext_q;   // the stationary tile

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && nit > 0) {
      mbar_expect_tx(bar(kYFull), kT128);
      load_tile128(sY, mY, bar(kYFull), row0, kKeyRows ? bh_kv : head, ext_y, args.err);
      int n_z = 0, n_w = 0;  // loads issued
      for (int it = 0; it < nit; ++it) {
        const int s = it % kZStages, u = it / kZStages;
        if (u > 0 && !mbar_wait(bar(kZEmpty + s), (u - 1) & 1, args.err, kErrTimeoutRing)) break;
        const int zr = z_row(it), zp = z_plane(it);
        mbar_expect_tx(bar(kZFull + s), kT64 + (kKeyRows ? 512u : 0u));
        load_tile64(sZ(s), mZ, bar(kZFull + s), zr, zp, ext_zw, args.err);
        if constexpr (kKeyRows) {
          const long long nrows = (long long)args.BH * args.Npad, first = (long long)zp * args.Npad + zr;
          bulk_load_rows(sLD(s), args.lse_log2, first, 256, nrows, bar(kZFull + s), args.err);
          bulk_load_rows(sLD(s) + 256, args.delta, first, 256, nrows, bar(kZFull + s), args.err);
        }
        ++n_z;
        const int sw = it % kWStages, uw = it / kWStages;
        if (uw > 0 && !mbar_wait(bar(kWEmpty + sw), (uw - 1) & 1, args.err, kErrTimeoutRing)) break;
        mbar_expect_tx(bar(kWFull + sw), kT64);
        load_tile64(sW(sw), mW, bar(kWFull + sw), zr, zp, ext_zw, args.err);
        ++n_w;
      }
      // Every copy this thread issued lands before the CTA exits, even when the
      // consumers gave up after a timeout elsewhere (bounded waits, abort ignored).
      mbar_wait(bar(kYFull), 0, args.err, kErrTimeoutTma, false);
      for (int s = 0; s < kZStages; ++s)
        if (n_z > s) mbar_wait(bar(kZFull + s), ((n_z - 1 - s) / kZStages) & 1, args.err, kErrTimeoutTma, false);
      for (int s = 0; s < kWStages; ++s)
        if (n_w > s) mbar_wait(bar(kWFull + s), ((n_w - 1 - s) / kWStages) & 1, args.err, kErrTimeoutTma, false);
    }
  } else if (warp == kWarpMma || warp == kWarpMma2) {
    // ------------------------------------------------------------ MMA issuers
    // Warp kWarpMma: S(0) | S(i+1) once S(i) has been read out; it reads only the
    // resident operand and Z.  Warp kWarpMma2: dP(0) | G(i) once dS(i) is packed,
    // dP(i+1); dP(i+1) overwrites the packed dS(i) only after G(i) has read it (one
    // thread's tcgen05.mma operations execute in issue order).  Z(i) is read by
    // S(i) and G(i): its slot is free once both issuers have released it (each
    // waits for Z(i) to land first, so its arrival belongs to that item's phase).
    if (lane == 0 && nit > 0) {
      constexpr uint32_t kIdS = idesc_score(BF16), kIdG = idesc_grad(BF16);
      const uint32_t tA = tmem + kTmA, tB0 = tmem + kTmBuf0, tB1 = tmem + kTmBuf1, tG = tmem + kTmG;
      auto zfull = [&](int it) { return mbar_wait(bar(kZFull + it % kZStages), (it / kZStages) & 1, args.err, kErrTimeoutTma); };
      auto wfull = [&](int it) { return mbar_wait(bar(kWFull + it % kWStages), (it / kWStages) & 1, args.err, kErrTimeoutTma); };
      bool ok = true;
      if (warp == kWarpMma) {
        ok = mbar_wait(bar(kAReady), 0, args.err, kErrTimeoutSoftmax);
        for (int it = 0; ok && it < nit; ++it) {
          if (it > 0 && !(ok = mbar_wait(bar(kSFree), (it - 1) & 1, args.err, kErrTimeoutSoftmax))) break;
          if (!(ok = zfull(it))) break;
          tc_fence_after();
          score_ts(tB0, tA, sZ(it % kZStages), kIdS);
          mma_commit(bar(kSReady));
          mma_commit(bar(kZEmpty + it % kZStages));
        }
      } else {
        ok = mbar_wait(bar(kYFull), 0, args.err, kErrTimeoutTma) && wfull(0);
        if (ok) {
          tc_fence_after();
          score_ss(tB1, sY, sW(0), kIdS);
          mma_commit(bar(kDpReady));
          mma_commit(bar(kWEmpty + 0));  // W(0): read by dP(0) only
        }
        for (int it = 0; ok && it < nit; ++it) {
          if (!(ok = mbar_wait(bar(kDsFull), it & 1, args.err, kErrTimeoutSoftmax) && zfull(it))) break;
          tc_fence_after();
          grad_ts(tG, tB1, sZ(it % kZStages), kIdG, it > 0);
          mma_commit(bar(kZEmpty + it % kZStages));  // Z(it): last read by G(it)
          if (it + 1 < nit) {
            if (!(ok = wfull(it + 1))) break;
            tc_fence_after();
            score_ss(tB1, sY, sW((it + 1) % kWStages), kIdS);
            mma_commit(bar(kDpReady));
            mma_commit(bar(kWEmpty + (it + 1) % kWStages));
          }
        }
      }
      mma_commit(bar(kDone));  // also ends the epilogue's wait after a failure (result discarded)
      mbar_wait(bar(kDone), 0, args.err, kErrTimeoutMma, false);
    }
  } else if (warp < kEwWarps) {
    // ------------------------------------------------------------ elementwise warps + epilogue
    const int e = warp >> 2;                 // warpgroup: tile columns [32 e, 32 e + 32)
    const int r = ((warp & 3) << 5) + lane;  // TMEM lane: key row (dK, dV) or query row (dQ)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int row = row0 + r;
    const int nrows = kKeyRows ? Nk : N;
    const float c = args.scale_log2;
    bool ok = nit > 0;
    if (ok) {
      // ---- the resident operand (K or Q) into tensor memory: this thread's row,
      // warpgroup e's 128 of the 256 columns, as 16-bit pairs (zeros past the end)
      const uint16_t* src = reinterpret_cast<const uint16_t*>(kKeyRows ? args.k : args.q) +
                            ((size_t)plane_a * nrows + row) * 256 + 128 * e;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t a[32];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (row < nrows) v = *reinterpret_cast<const uint4*>(src + 64 * h + 8 * x);
          a[4 * x] = v.x;
          a[4 * x + 1] = v.y;
          a[4 * x + 2] = v.z;
          a[4 * x + 3] = v.w;
        }
        tmem_st_32x32b_x32(tmem + lane_base + kTmA + 64 * e + 32 * h, a);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(bar(kAReady));
    }
    // per-row L log2 e and D (dQ CTA): +inf and 0 on padding rows, so P = 0 there
    float Lr = 0.f, Dr = 0.f;
    if constexpr (!kKeyRows) {
      Lr = args.lse_log2[(size_t)head * args.Npad + row];
      Dr = args.delta[(size_t)head * args.Npad + row];
    }
    const int cbeg = 32 * e;
    for (int it = 0; ok && it < nit; ++it) {
      const int c0 = z_row(it);  // first query (dK) or key (dQ) of the block
      // some visible (key, query) pair hidden in this block: causal diagonal, or (dQ)
      // keys past N_k in the last block (their K, V rows are zero, but P would not be)
      const bool diag = kKeyRows ? (args.causal && row0 + kRes - 1 > c0 + koff)
                                 : ((args.causal && c0 + kBlk - 1 > row0 + koff) || c0 + kBlk > Nk);
      float l4v[32], d4v[32];
      if constexpr (kKeyRows) {
        // L log2 e and D of the block's queries arrive with its Q tile
        const int s = it % kZStages;
        if (!(ok = warp_wait(bar(kZFull + s), (it / kZStages) & 1, args.err, kErrTimeoutTma))) break;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float4 t;
          ld_shared_f4(sLD(s) + 4u * (cbeg + 4 * i), t);
          l4v[4 * i] = t.x, l4v[4 * i + 1] = t.y, l4v[4 * i + 2] = t.z, l4v[4 * i + 3] = t.w;
          ld_shared_f4(sLD(s) + 256u + 4u * (cbeg + 4 * i), t);
          d4v[4 * i] = t.x, d4v[4 * i + 1] = t.y, d4v[4 * i + 2] = t.z, d4v[4 * i + 3] = t.w;
        }
      }
      // ---- P = 2^(S c - L log2 e)
      const uint32_t tS = tmem + lane_base + kTmBuf0 + cbeg;
      if (!(ok = warp_wait(bar(kSReady), it & 1, args.err, kErrTimeoutMma))) break;
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld_32x32b_x32(tS, sv);
      tmem_wait_ld();
      reg_fence32(sv);
      float p[32];
#pragma unroll
      for (int x = 0; x < 32; x += 2) {
        float x0, x1;
        if constexpr (kKeyRows)
          fma2v(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1]), c, -l4v[x], -l4v[x + 1], x0, x1);
        else
          fma2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1]), c, -Lr, x0, x1);
        p[x] = ex2_approx(x0);
        p[x + 1] = ex2_approx(x1);
      }
      if (diag) {
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const int col = c0 + cbeg + x;
          const bool hidden = kKeyRows ? (args.causal && row > col + koff)
                                       : ((args.causal && col > row + koff) || col >= Nk);
          if (hidden) p[x] = 0.f;
        }
      }
      {
        tc_fence_before();
        warp_arrive(bar(kSFree));  // the scores may be overwritten by the next block's now
        // ---- dS = P o (dP - D), packed into the dP buffer
        const uint32_t tDP = tmem + lane_base + kTmBuf1 + cbeg;
        if (!(ok = warp_wait(bar(kDpReady), it & 1, args.err, kErrTimeoutMma))) break;
        tc_fence_after();
        uint32_t dv[32];
        tmem_ld_32x32b_x32(tDP, dv);
        tmem_wait_ld();
        reg_fence32(dv);
        uint32_t dw[16];
#pragma unroll
        for (int x = 0; x < 32; x += 2) {
          float ds0, ds1;
          if constexpr (kKeyRows)
            submul2(p[x], p[x + 1], __uint_as_float(dv[x]), __uint_as_float(dv[x + 1]), d4v[x], d4v[x + 1], ds0, ds1);
          else
            submul2(p[x], p[x + 1], __uint_as_float(dv[x]), __uint_as_float(dv[x + 1]), Dr, Dr, ds0, ds1);
          dw[x >> 1] = pack2<BF16>(ds0, ds1);
        }
        tmem_st_32x32b_x16(tDP, dw);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(bar(kDsFull));
      }
    }
    // ---- the gradient rows: lane r holds row `row`; warpgroup e writes columns
    // [128 e, 128 e + 128).  A dQ CTA whose rows see no key writes dQ = 0.
    if (nit == 0 || (ok && warp_wait(bar(kDone), 0, args.err, kErrTimeoutMma))) {
      tc_fence_after();
      const float mul = args.scale;
      void* out = ROLE == kRoleDK ? args.dk : args.dq;
      uint16_t* dst = reinterpret_cast<uint16_t*>(out) + ((size_t)plane_a * nrows + row) * 256 + 128 * e;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t v[32];
        if (nit > 0) {
          tmem_ld_32x32b_x32(tmem + lane_base + kTmG + 128 * e + 32 * ch, v);
          tmem_wait_ld();
          reg_fence32(v);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] = 0u;
        }
        if (row < nrows) {
#pragma unroll
          for (int x = 0; x < 32; x += 8)
            st_global_v4(dst + 32 * ch + x, pack2<BF16>(__uint_as_float(v[x]) * mul, __uint_as_float(v[x + 1]) * mul),
                         pack2<BF16>(__uint_as_float(v[x + 2]) * mul, __uint_as_float(v[x + 3]) * mul),
                         pack2<BF16>(__uint_as_float(v[x + 4]) * mul, __uint_as_float(v[x + 5]) * mul),
                         pack2<BF16>(__uint_as_float(v[x + 6]) * mul, __uint_as_float(v[x + 7]) * mul));
        }
      }
    }
  }
}

// ---------------------------------------------------------------- dV CTAs
// A dV CTA has only the score product and dV, so it can stream 128-row query tiles:
// K stays in shared memory (64 KB) as the A operand of S^T = K Q^T (N = 128), and
// tensor memory holds S^T (columns 0-127), P^T packed (128-191) and dV (256-511).
// With P^T apart from S^T, S^T(i+1) is issued as soon as the elementwise warps have
// read S^T(i) and runs while they exponentiate; P^T(i+1) waits only for dV(i).  The
// ring of two 64 KB slots is filled in the order the products read it: Q_0, Q_1,
// dO_0, Q_2, dO_1, ..., dO_last; the L log2 e values of each query tile go through
// two stages of their own (their reader, not the ring, decides when they are free).
constexpr int kDvRows = 128;                  // query rows per streamed tile
constexpr uint32_t kSmDvRing = kSmZ;          // two 64 KB slots
constexpr uint32_t kTmDvS = 0, kTmDvP = 128;  // S^T fp32, P^T packed
// barrier indices of the dV program (its own set in the same barrier array)
enum : int {
  kDvKFull = 0,    // K tile
  kDvFull = 1,     // two ring slots
  kDvEmpty = 3,    // two
  kDvLFull = 5,    // two: L log2 e of block i in stage i & 1
  kDvLEmpty = 7,   // two: the elementwise warps have read that stage
  kDvSReady = 9,   // S^T in TMEM
  kDvSFree = 10,   // S^T read out
  kDvPFull = 11,   // P^T packed
  kDvDone = 12,    // dV(i) has run: P^T may be overwritten
  kDvDrain = 13,   // the last dV product has completed
  kDvNumBars
};
static_assert(kDvNumBars <= kNumBars, "dV barriers inside the barrier array");
static_assert(kSmDvRing + 2 * kT128 <= kSmLD, "dV ring inside the streamed-tile region");
__device__ __forceinline__ void init_dv_barriers(uint32_t sbase) {
  auto bar = [&](int i) -> uint32_t { return sbase + kSmBar + 8u * i; };
  mbar_init(bar(kDvKFull), 1);
  for (int s = 0; s < 2; ++s) {
    mbar_init(bar(kDvFull + s), 1);
    mbar_init(bar(kDvEmpty + s), 1);
    mbar_init(bar(kDvLFull + s), 1);
    mbar_init(bar(kDvLEmpty + s), kEwWarps);
  }
  mbar_init(bar(kDvSReady), 1);
  mbar_init(bar(kDvSFree), kEwWarps);
  mbar_init(bar(kDvPFull), kEwWarps);
  mbar_init(bar(kDvDone), 1);
  mbar_init(bar(kDvDrain), 1);
}

__device__ __forceinline__ int dv_first_qblock(const BwdArgs& a, int key0) {
  return a.causal ? max(0, key0 - (a.Nk - a.N)) / kDvRows : 0;
}
__device__ __forceinline__ int dv_blocks(const BwdArgs& a, int blk) {
  return ((a.N + kDvRows - 1) / kDvRows - dv_first_qblock(a, blk * kRes)) * a.group;
}
// Ring item e: is it a dO tile, and of which block.  Q_0 | Q_{i+1}, dO_i | dO_last.
__device__ __forceinline__ int dv_item(int e, int nit, bool& is_do) {
  if (e == 0) { is_do = false; return 0; }
  if (e == 2 * nit - 1) { is_do = true; return nit - 1; }
  is_do = !(e & 1);
  return (e & 1) ? (e + 1) >> 1 : (e >> 1) - 1;
}
// Acc (128 x 128) = A B^T, A and B 128-row K-major tiles in shared memory (d = 256).
__device__ __forceinline__ void score_ss128(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem, uint32_t idesc) {
  const uint32_t a0 = sdesc_lo(a_smem, 16), b0 = sdesc_lo(b_smem, 16);
#pragma unroll
  for (int kk = 0; kk < 16; ++kk) {
    const uint32_t off = ((kk >> 2) * kP128 + (kk & 3) * 32) >> 4;
    mma_ss_lohi(d_tmem, a0 + off, kHi, b0 + off, kHi, idesc, kk > 0);
  }
}
// Acc (128 x 256) (+)= A B, A (128 x 128) packed in TMEM, B a 128-row tile read MN-major.
__device__ __forceinline__ void grad_ts128(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem, uint32_t idesc, bool acc) {
  const uint32_t b0 = sdesc_lo(b_smem, kP128);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts_lohi(d_tmem, a_tmem + 8 * kk, b0 + ((kk * 2048) >> 4), kHi, idesc, (acc || kk > 0) ? 1u : 0u);
}

template <bool BF16>
__device__ __forceinline__ void bwd256_dv_cta(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                              const CUtensorMap* tm_do, const BwdArgs& args, int blk, int head,
                                              uint32_t sbase, uint32_t tmem) {
  auto bar = [&](int i) -> uint32_t { return sbase + kSmBar + 8u * i; };
  auto sRing = [&](int s) -> uint32_t { return sbase + kSmDvRing + kT128 * s; };
  auto sL = [&](int i) -> uint32_t { return sbase + kSmLD + 512u * (i & 1); };  // L log2 e of block i
  const uint32_t sK = sbase + kSmY;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = args.N, Nk = args.Nk;
  const int koff = Nk - N;
  const int key0 = blk * kRes;
  const int nit = dv_blocks(args, blk);  // >= 1: the last query row sees every key
  const int i_begin = dv_first_qblock(args, key0);
  const int nit_h = (N + kDvRows - 1) / kDvRows - i_begin;
  const int hpb = args.H / args.group;
  const int bh_q0 = (head / hpb) * args.H + (head % hpb) * args.group;
  auto q_row = [&](int i) { return (i_begin + i % nit_h) * kDvRows; };
  auto q_plane = [&](int i) { return bh_q0 + i / nit_h; };
  const Extent3 ext_q{256, N, args.BH}, ext_kv{256, Nk, args.BHkv};

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_expect_tx(bar(kDvKFull), kT128);
      load_tile128(sK, tm_k, bar(kDvKFull), key0, head, ext_kv, args.err);
      int n = 0, nl = 0;  // ring loads and L loads issued
      for (int e = 0; e < 2 * nit; ++e) {
        const int s = e & 1, u = e >> 1;
        if (u > 0 && !mbar_wait(bar(kDvEmpty + s), (u - 1) & 1, args.err, kErrTimeoutRing)) break;
        bool is_do;
        const int i = dv_item(e, nit, is_do);
        mbar_expect_tx(bar(kDvFull + s), kT128);
        load_tile128(sRing(s), is_do ? tm_do : tm_q, bar(kDvFull + s), q_row(i), q_plane(i), ext_q, args.err);
        ++n;
        if (!is_do) {
          // L log2 e of block i into stage i & 1, once the elementwise warps have read block i - 2's
          const int b = i & 1;
          if (i >= 2 && !mbar_wait(bar(kDvLEmpty + b), ((i >> 1) - 1) & 1, args.err, kErrTimeoutRing)) break;
          const long long nrows = (long long)args.BH * args.Npad, first = (long long)q_plane(i) * args.Npad + q_row(i);
          mbar_expect_tx(bar(kDvLFull + b), 512);
          bulk_load_rows(sL(i), args.lse_log2, first, 512, nrows, bar(kDvLFull + b), args.err);
          ++nl;
        }
      }
      // Every copy this thread issued lands before the CTA exits (bounded waits, abort ignored).
      mbar_wait(bar(kDvKFull), 0, args.err, kErrTimeoutTma, false);
      for (int s = 0; s < 2; ++s) {
        if (n > s) mbar_wait(bar(kDvFull + s), ((n - 1 - s) >> 1) & 1, args.err, kErrTimeoutTma, false);
        if (nl > s) mbar_wait(bar(kDvLFull + s), ((nl - 1 - s) >> 1) & 1, args.err, kErrTimeoutTma, false);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // S^T(0) | S^T(i+1) once S^T(i) has been read, then dV(i) once P^T(i) is packed | ...
    // S^T(i+1) is issued after dV(i-1), so a dV(i) commit is at most one phase ahead
    // of the elementwise warps that wait for it.
    if (lane == 0) {
      constexpr uint32_t kIdS = make_idesc_f16(BF16, 128, kDvRows, false, false);
      constexpr uint32_t kIdG = idesc_grad(BF16);
      auto full = [&](int e) { return mbar_wait(bar(kDvFull + (e & 1)), (e >> 1) & 1, args.err, kErrTimeoutTma); };
      bool ok = mbar_wait(bar(kDvKFull), 0, args.err, kErrTimeoutTma) && full(0);
      if (ok) {
        tc_fence_after();
        score_ss128(tmem + kTmDvS, sK, sRing(0), kIdS);
        mma_commit(bar(kDvSReady));
        mma_commit(bar(kDvEmpty + 0));
      }
      for (int i = 0; ok && i < nit; ++i) {
        if (i + 1 < nit) {
          const int e = 2 * i + 1;  // Q_{i+1}
          if (!(ok = mbar_wait(bar(kDvSFree), i & 1, args.err, kErrTimeoutSoftmax) && full(e))) break;
          tc_fence_after();
          score_ss128(tmem + kTmDvS, sK, sRing(e & 1), kIdS);
          mma_commit(bar(kDvSReady));
          mma_commit(bar(kDvEmpty + (e & 1)));
        }
        const int e = (i == nit - 1) ? 2 * nit - 1 : 2 * i + 2;  // dO_i
        if (!(ok = full(e) && mbar_wait(bar(kDvPFull), i & 1, args.err, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        grad_ts128(tmem + kTmG, tmem + kTmDvP, sRing(e & 1), kIdG, i > 0);
        mma_commit(bar(kDvDone));
        mma_commit(bar(kDvEmpty + (e & 1)));
      }
      mma_commit(bar(kDvDrain));  // also ends the epilogue's wait after a failure (result discarded)
      mbar_wait(bar(kDvDrain), 0, args.err, kErrTimeoutMma, false);
    }
  } else if (warp < kEwWarps) {
    // ------------------------------------------------------------ P^T, epilogue
    const int e = warp >> 2;                 // warpgroup: query columns [64 e, 64 e + 64)
    const int r = ((warp & 3) << 5) + lane;  // TMEM lane: key row
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int key = key0 + r;
    const float c = args.scale_log2;
    bool ok = true;
    for (int i = 0; ok && i < nit; ++i) {
      const int q0 = q_row(i);
      const bool diag = args.causal && key0 + kRes - 1 > q0 + koff;  // some key hidden from some query
      // L log2 e of the block's queries, in stage i & 1 (the stage's barrier is at most
      // one phase ahead: block i + 2's copy waits for this block's LEmpty)
      if (!(ok = warp_wait(bar(kDvLFull + (i & 1)), (i >> 1) & 1, args.err, kErrTimeoutTma))) break;
      float lv[64];
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        float4 t;
        ld_shared_f4(sL(i) + 4u * (64 * e + 4 * x), t);
        lv[4 * x] = t.x, lv[4 * x + 1] = t.y, lv[4 * x + 2] = t.z, lv[4 * x + 3] = t.w;
      }
      warp_arrive(bar(kDvLEmpty + (i & 1)));
      if (!(ok = warp_wait(bar(kDvSReady), i & 1, args.err, kErrTimeoutMma))) break;
      tc_fence_after();
      uint32_t sv[2][32];
      tmem_ld_32x32b_x32(tmem + lane_base + kTmDvS + 64 * e, sv[0]);
      tmem_ld_32x32b_x32(tmem + lane_base + kTmDvS + 64 * e + 32, sv[1]);
      tmem_wait_ld();
      reg_fence32(sv[0]);
      reg_fence32(sv[1]);
      tc_fence_before();
      warp_arrive(bar(kDvSFree));  // S^T may be overwritten by the next block's scores now
      float p[64];
#pragma unroll
      for (int x = 0; x < 64; x += 2) {
        float x0, x1;
        fma2v(__uint_as_float(sv[x >> 5][x & 31]), __uint_as_float(sv[x >> 5][(x & 31) + 1]), c, -lv[x], -lv[x + 1],
              x0, x1);
        p[x] = ex2_approx(x0);
        p[x + 1] = ex2_approx(x1);
      }
      if (diag) {
#pragma unroll
        for (int x = 0; x < 64; ++x)
          if (key > q0 + 64 * e + x + koff) p[x] = 0.f;
      }
      // P^T(i) overwrites P^T(i-1): wait until dV(i-1) has read it
      if (i > 0) {
        if (!(ok = warp_wait(bar(kDvDone), (i - 1) & 1, args.err, kErrTimeoutMma))) break;
        tc_fence_after();
      }
      uint32_t pw[32];
#pragma unroll
      for (int x = 0; x < 32; ++x) pw[x] = pack2<BF16>(p[2 * x], p[2 * x + 1]);
      tmem_st_32x32b_x32(tmem + lane_base + kTmDvP + 32 * e, pw);
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(bar(kDvPFull));
    }
    // ---- dV rows: lane r holds key row `key`; warpgroup e writes columns [128 e, 128 e + 128)
    if (ok && warp_wait(bar(kDvDrain), 0, args.err, kErrTimeoutMma)) {
      tc_fence_after();
      uint16_t* dst = reinterpret_cast<uint16_t*>(args.dv) + ((size_t)head * Nk + key) * 256 + 128 * e;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem + lane_base + kTmG + 128 * e + 32 * ch, v);
        tmem_wait_ld();
        reg_fence32(v);
        if (key < Nk) {
#pragma unroll
          for (int x = 0; x < 32; x += 8)
            st_global_v4(dst + 32 * ch + x, pack2<BF16>(__uint_as_float(v[x]), __uint_as_float(v[x + 1])),
                         pack2<BF16>(__uint_as_float(v[x + 2]), __uint_as_float(v[x + 3])),
                         pack2<BF16>(__uint_as_float(v[x + 4]), __uint_as_float(v[x + 5])),
                         pack2<BF16>(__uint_as_float(v[x + 6]), __uint_as_float(v[x + 7])));
        }
      }
    }
  }
}

__device__ __forceinline__ void check_phases_dv(uint32_t sbase, int nit, uint32_t* err) {
  auto bar = [&](int i) -> uint32_t { return sbase + kSmBar + 8u * i; };
  check_phase(bar(kDvKFull), 1, err, kDvKFull);
  for (int s = 0; s < 2; ++s) {
    check_phase(bar(kDvFull + s), nit, err, kDvFull + s);  // 2 nit items alternate the two slots
    check_phase(bar(kDvEmpty + s), nit, err, kDvEmpty + s);
    check_phase(bar(kDvLFull + s), count_mod(nit, s, 2), err, kDvLFull + s);
    check_phase(bar(kDvLEmpty + s), count_mod(nit, s, 2), err, kDvLEmpty + s);
  }
  for (int b : {kDvSReady, kDvSFree, kDvPFull, kDvDone}) check_phase(bar(b), nit, err, b);
  check_phase(bar(kDvDrain), 1, err, kDvDrain);
}

// FA_DEBUG builds: the phases every barrier of a dK or dQ CTA completed, against
// its protocol (thread 0, after the CTA's final barrier, when no wait gave up).
template <int ROLE>
__device__ __forceinline__ void check_phases(uint32_t sbase, int nit, uint32_t* err) {
  auto bar = [&](int i) -> uint32_t { return sbase + kSmBar + 8u * i; };
  check_phase(bar(kYFull), nit > 0, err, kYFull);
  check_phase(bar(kAReady), nit > 0, err, kAReady);
  for (int s = 0; s < kZStages; ++s) {
    check_phase(bar(kZFull + s), count_mod(nit, s, kZStages), err, kZFull + s);
    check_phase(bar(kZEmpty + s), count_mod(nit, s, kZStages), err, kZEmpty + s);
  }
  for (int s = 0; s < kWStages; ++s) {
    check_phase(bar(kWFull + s), count_mod(nit, s, kWStages), err, kWFull + s);
    check_phase(bar(kWEmpty + s), count_mod(nit, s, kWStages), err, kWEmpty + s);
  }
  for (int b : {kSReady, kSFree, kDpReady, kDsFull}) check_phase(bar(b), nit, err, b);
  check_phase(bar(kDone), nit > 0, err, kDone);
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // CTA -> (role, block, head), by groups of G key/value heads (args.head_group_kv):
  // a group's dK and dV CTAs (the pair of one key block side by side, lowest key
  // blocks first: under the causal mask they see the most query blocks), then the
  // dQ CTAs of its G * group query heads (the last query blocks first).  The query
  // heads of key/value heads [a, a + G) are [a * group, (a + G) * group), so a
  // group's dQ CTAs read the same K, V, Q, dO its key-block CTAs have just brought
  // into L2, and the light CTAs that end one group run beside the heavy ones that
  // start the next.
  const int nkb = (args.Nk + kRes - 1) / kRes;
  const int nqb = (args.N + kRes - 1) / kRes;
  const int grp = args.group;
  const int G = max(1, min(args.head_group_kv, args.BHkv));
  const unsigned per_full = (unsigned)G * (2u * (unsigned)nkb + (unsigned)nqb * (unsigned)grp);
  const int g = (int)(blockIdx.x / per_full);
  const int h0 = g * G;                        // first key/value head of the group
  const int Gg = min(G, args.BHkv - h0);       // heads in this group (the last may be short)
  unsigned t = blockIdx.x - (unsigned)g * per_full;
  const unsigned n_kv = 2u * (unsigned)nkb * (unsigned)Gg;
  int role, blk, head;
  if (t < n_kv) {
    role = (t & 1) ? kRoleDV : kRoleDK;
    t >>= 1;
    blk = (int)(t / (unsigned)Gg);
    head = h0 + (int)(t % (unsigned)Gg);
  } else {
    t -= n_kv;
    const unsigned nq_heads = (unsigned)Gg * (unsigned)grp;
    role = kRoleDQ;
    blk = nqb - 1 - (int)(t / nq_heads);
    head = h0 * grp + (int)(t % nq_heads);
  }

  if (threadIdx.x == 0 && role == kRoleDV) {
    init_dv_barriers(sbase);
    fence_mbar_init();
  } else if (threadIdx.x == 0) {
    mbar_init(sbase + kSmBar + 8u * kYFull, 1);
    mbar_init(sbase + kSmBar + 8u * kAReady, kEwWarps);
    for (int s = 0; s < kZStages; ++s) {
      mbar_init(sbase + kSmBar + 8u * (kZFull + s), 1);
      mbar_init(sbase + kSmBar + 8u * (kZEmpty + s), 2);  // read by both issuers' products
    }
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(sbase + kSmBar + 8u * (kWFull + s), 1);
      mbar_init(sbase + kSmBar + 8u * (kWEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sbase + kSmBar + 8u * (kSReady + b), 1);
      mbar_init(sbase + kSmBar + 8u * (kPFull + b), kEwWarps);
    }
    mbar_init(sbase + kSmBar + 8u * kSFree, kEwWarps);
    mbar_init(sbase + kSmBar + 8u * kDpReady, 1);
    mbar_init(sbase + kSmBar + 8u * kDsFull, kEwWarps);
    mbar_init(sbase + kSmBar + 8u * kDone, 2);  // both issuers
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(sbase + kSmTmemSlot, 512);
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
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kSmTmemSlot);
  debug_context(tmem, args.err);

  if (role == kRoleDK)
    bwd256_cta<kRoleDK, BF16>(&tm_q, &tm_k, &tm_v, &tm_do, args, blk, head, smem, sbase, tmem);
  else if (role == kRoleDV)
    bwd256_dv_cta<BF16>(&tm_q, &tm_k, &tm_do, args, blk, head, sbase, tmem);
  else
    bwd256_cta<kRoleDQ, BF16>(&tm_q, &tm_k, &tm_v, &tm_do, args, blk, head, smem, sbase, tmem);

  tc_fence_before();
  __syncthreads();
  if constexpr (kDebug) {
    if (threadIdx.x == 0 && no_abort(args.err)) {
      if (role == kRoleDK) check_phases<kRoleDK>(sbase, cta_blocks(args, role, blk), args.err);
      else if (role == kRoleDV) check_phases_dv(sbase, dv_blocks(args, blk), args.err);
      else check_phases<kRoleDQ>(sbase, cta_blocks(args, role, blk), args.err);
    }
  }
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool BF16>
cudaError_t launch_256(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout,
                       const BwdArgs& a, cudaStream_t stream) {
  auto kern = fa_bwd256_kernel<BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmAlloc);
  if (e != cudaSuccess) return e;
  const long long grid = 2LL * ((a.Nk + kRes - 1) / kRes) * a.BHkv + (long long)((a.N + kRes - 1) / kRes) * a.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  profile_mark_begin(stream);
  kern<<<(unsigned)grid, kThreads, kSmAlloc, stream>>>(q, k, v, dout, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  profile_mark_end(stream, kProfileBwdFused);
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd_main_256(bool bf16, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& dout, const BwdArgs& a, cudaStream_t stream) {
  return bf16 ? launch_256<true>(q, k, v, dout, a, stream) : launch_256<false>(q, k, v, dout, a, stream);
}

}  // namespace fa
