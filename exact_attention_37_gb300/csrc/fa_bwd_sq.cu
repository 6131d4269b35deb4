// Backward pass for head dimensions 64 and 128 as two kernels on 128 x 128 tiles,
// with no atomics: every gradient element is summed in a fixed order inside one
// CTA, so dQ, dK and dV are bitwise reproducible.
//
// Both kernels rebuild the probabilities block by block from Q, K and the forward
// pass's logsumexp (page "FlashAttention — فلاش أتنشن", section "Tiling and block
// processing") and apply the chain-rule derivatives of the attention formula
// (same page, section "The problem of standard attention"):
//
//   P = 2^(S scale log2 e - L log2 e),   dP = dO V^T,   dS = P o (dP - D),
//   dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K.
//
// fa_bwd_kv_kernel: one CTA per (key/value head, 128-key block), looping over the
//   query blocks of every query head of the group (the key-block parallelism of
//   page "FlashAttention-2 — فلاش أتنشن-2", section "Technical architecture",
//   item 2).  Keys sit on TMEM lanes: S^T = K Q^T, dP^T = V dO^T.  P^T is written
//   back as packed 16-bit pairs into the columns of S^T and feeds dV += P^T dO as
//   the tensor-memory A operand; dS^T likewise goes into the columns of dP^T and
//   feeds dK += dS^T Q.  Only the B operands (dO, Q) are read from shared memory
//   by the gradient products.
// fa_bwd_q_kernel: one CTA per (query head, 128-row query block), looping over the
//   key blocks its rows see.  Queries sit on TMEM lanes: S = Q K^T and dP = dO V^T
//   (two dP buffers, so dP runs two key blocks ahead); dS goes back into its dP
//   buffer as packed pairs and feeds dQ += dS K; dQ stays in TMEM until the CTA
//   writes it once, scaled and rounded.
//
// The second kernel recomputes S and dP (7 products per tile pair instead of 5);
// in exchange no fp32 reductions leave the SM, and the dQ accumulator, its
// zeroing and its conversion pass disappear.
//
// The score products have M = N = 128, the gradient products N = d.  Warps: 4 NWG
// elementwise warps (NWG warpgroups, 128 / NWG tile columns each; every warp
// arrives once on the barriers it signals), one TMA warp, one MMA warp, and in the
// dQ kernel a second MMA warp.  One thread issues a tcgen05.mma only about every
// 50 cycles, so the dQ kernel splits its products by the tensor-memory columns
// they touch: S on one issuer, dP and dQ (which reads dS from the dP buffers) on
// the other, so every product that overwrites columns another reads stays in the
// same thread as its reader.  (The same split of the dK/dV kernel, S^T and dV |
// dP^T and dK, interleaves the two streams so that S^T(i+1) lands later; it was
// slower.)
#include <algorithm>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr uint32_t kPanel = 128 * 128;    // 128 rows x 128 B (64 16-bit columns)
// A 128-row tile of Q, K, V or dO with head dimension D: D / 64 panels.
template <int D>
constexpr uint32_t tile_bytes() { return (uint32_t)(D / 64) * kPanel; }

template <int NWG>
struct SqCfg {
  static constexpr int kCols = 128 / NWG;      // tile columns per elementwise thread
  static constexpr int kCh = kCols / 32;       // 32-column TMEM chunks per thread
  static constexpr int kEw = 128 * NWG;        // elementwise threads
  static constexpr int kWarpTma = 4 * NWG;
  static constexpr int kWarpMma = 4 * NWG + 1;
  static constexpr int kWarpMma2 = 4 * NWG + 2;  // dQ kernel: the second MMA issuer
  static constexpr int kThreadsKV = kEw + 64;
  static constexpr int kThreadsQ = kEw + 96;
  // TMEM column, relative to a packed region, of the 16 K elements of step kk:
  // warpgroup e packs its kCols columns into kCols / 2 columns starting at kCols e.
  static constexpr uint32_t packed_col(int kk) { return kCols * ((16 * kk) / kCols) + ((16 * kk) % kCols) / 2; }
};

__device__ __forceinline__ void st_global_v4(void* addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void ld_shared_f4(uint32_t addr, float4& v) {
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
}

constexpr uint32_t kIdSS(bool bf16) { return make_idesc_f16(bf16, 128, 128, false, false); }  // both K-major
// N = D, A K-major (from TMEM or shared memory), B MN-major
constexpr uint32_t kIdTS(bool bf16, int d) { return make_idesc_f16(bf16, 128, d, false, true); }
constexpr uint32_t kHi = sdesc_hi_sw128(1024);  // every operand: 8-row groups 1024 B apart

// Acc (128 x 128, fp32) = A B^T with A, B 128 x D K-major tiles in shared memory
// (D / 64 panels each): S^T = K Q^T, dP^T = V dO^T, S = Q K^T, dP = dO V^T.
template <int D>
__device__ __forceinline__ void mma_scores(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem, uint32_t idesc) {
  const uint32_t a0 = sdesc_lo(a_smem, 16), b0 = sdesc_lo(b_smem, 16);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * kPanel + (kk & 3) * 32) >> 4;
    mma_ss_lohi(d_tmem, a0 + off, kHi, b0 + off, kHi, idesc, kk > 0);
  }
}
// Acc (+)= A B with A (128 x 128) packed in TMEM by NWG warpgroups and B a 128-row
// tile in shared memory read MN-major (rows = K, 64-column panels of N).
template <int NWG>
__device__ __forceinline__ void mma_packed(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem, uint32_t idesc,
                                           bool acc) {
  const uint32_t b0 = sdesc_lo(b_smem, kPanel);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts_lohi(d_tmem, a_tmem + SqCfg<NWG>::packed_col(kk), b0 + ((kk * 2048) >> 4), kHi, idesc,
                (acc || kk > 0) ? 1u : 0u);
}

// TMA load of one 128-row tile (D / 64 boxes of 64 columns) completing `bar`.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* m, uint32_t bar, int row, int plane,
                                          const Extent3& ext, uint32_t* err) {
#pragma unroll
  for (int p = 0; p < D / 64; ++p) tma_load_box(dst + p * kPanel, m, bar, 64 * p, row, plane, ext, err);
}

// Stores 32 fp32 values (times mul) as 16-bit to dst (64 contiguous bytes).
template <bool BF16>
__device__ __forceinline__ void store_row32(uint16_t* dst, const uint32_t (&v)[32], float mul) {
#pragma unroll
  for (int x = 0; x < 32; x += 8)
    st_global_v4(dst + x, pack2<BF16>(__uint_as_float(v[x]) * mul, __uint_as_float(v[x + 1]) * mul),
                 pack2<BF16>(__uint_as_float(v[x + 2]) * mul, __uint_as_float(v[x + 3]) * mul),
                 pack2<BF16>(__uint_as_float(v[x + 4]) * mul, __uint_as_float(v[x + 5]) * mul),
                 pack2<BF16>(__uint_as_float(v[x + 6]) * mul, __uint_as_float(v[x + 7]) * mul));
}

// ============================================================================ dK, dV
namespace kv {
template <int D>
struct Smem {
  static constexpr uint32_t T = tile_bytes<D>();
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = T;
  static constexpr uint32_t kQ = 2 * T;    // two stages
  static constexpr uint32_t kDO = 4 * T;   // two stages
  static constexpr uint32_t kLD = 6 * T;   // two stages of L log2 e (512 B) and D (512 B) of a query block
  static constexpr uint32_t kBar = 6 * T + 2048;
};
enum : int {
  kKVFull = 0,
  kQFull = 1,    // two: a Q tile with the L log2 e and D rows of its query block
  kQEmpty = 3,   // two
  kDOFull = 5,   // two
  kDOEmpty = 7,  // two
  kSReady = 9,   // S^T of the block is in TMEM
  kPFull,        // S^T read out and P^T written back packed into its columns
  kDpReady,      // dP^T of the block is in TMEM
  kDsFull,       // dS^T written
  kDone,         // the last dK product has completed
  kNumBars
};
template <int D>
constexpr uint32_t tmem_slot() { return Smem<D>::kBar + kNumBars * 8; }
template <int D>
constexpr uint32_t smem_alloc() { return tmem_slot<D>() + 16 + 1024; }  // + alignment of the dynamic base
static_assert(smem_alloc<128>() <= 232448, "shared memory budget");
constexpr uint32_t kTmS = 0;     // S^T fp32, then P^T packed
constexpr uint32_t kTmDP = 128;  // dP^T fp32, then dS^T packed
constexpr uint32_t kTmDV = 256;
template <int D>
constexpr uint32_t tm_dk() { return 256 + D; }
}  // namespace kv

template <int D, int NWG, bool BF16>
__global__ void __launch_bounds__(SqCfg<NWG>::kThreadsKV, 1)
    fa_bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdArgs args) {
  using namespace kv;
  using C = SqCfg<NWG>;
  using M = Smem<D>;
  constexpr int kCols = C::kCols, kCh = C::kCh;
  constexpr uint32_t kTile = M::T, kSmTmemSlot = tmem_slot<D>(), kTmDK = tm_dk<D>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + M::kBar + 8u * i; };
  auto sQ = [&](int s) -> uint32_t { return sbase + M::kQ + kTile * s; };
  auto sDO = [&](int s) -> uint32_t { return sbase + M::kDO + kTile * s; };
  const uint32_t sK = sbase + M::kK, sV = sbase + M::kV;
  auto sLD = [&](int s) -> uint32_t { return sbase + M::kLD + 1024u * s; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = args.N;
  const int Nk = args.Nk;

  // Work tile: lowest key blocks first (under the causal mask they see the most
  // query blocks), key/value heads in groups of args.head_group_kv so the Q and dO
  // tiles of the running CTAs stay in L2.  The CTA visits the query blocks of every
  // query head of its key/value head's group, so dK, dV of the group sum in TMEM.
  int kb, bh_kv;
  grouped_tile(blockIdx.x, args.BHkv, (Nk + 127) / 128, args.head_group_kv, kb, bh_kv);
  const int koff = Nk - N;  // key j visible to query i iff j <= i + koff
  const int key0 = kb * 128;
  const int nqb = (N + 127) / 128;
  const int i_begin = args.causal ? max(0, key0 - koff) / 128 : 0;
  const int nit_h = nqb - i_begin;  // >= 1: the last query row sees every key
  const int nit = nit_h * args.group;
  const int hpb = args.H / args.group;  // key/value heads per batch entry
  const int bh_q0 = (bh_kv / hpb) * args.H + (bh_kv % hpb) * args.group;
  auto q_head = [&](int it) { return bh_q0 + it / nit_h; };
  auto q_block = [&](int it) { return i_begin + it % nit_h; };

  if (threadIdx.x == 0) {
    mbar_init(bar(kKVFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kQFull + s), 1);
      mbar_init(bar(kQEmpty + s), 1);
      mbar_init(bar(kDOFull + s), 1);
      mbar_init(bar(kDOEmpty + s), 1);
    }
    mbar_init(bar(kSReady), 1);
    mbar_init(bar(kPFull), C::kEw / 32);  // one arrival per elementwise warp
    mbar_init(bar(kDpReady), 1);
    mbar_init(bar(kDsFull), C::kEw / 32);
    mbar_init(bar(kDone), 1);
    fence_mbar_init();
  }
  if (warp == C::kWarpMma) {
    tmem_alloc(sbase + kSmTmemSlot, 512);
    tmem_relinquish();
  }
  if (warp == C::kWarpTma && lane == 0) {
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
  const Extent3 ext_q{D, N, args.BH}, ext_kv{D, Nk, args.BHkv};

  if (warp == C::kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_expect_tx(bar(kKVFull), 2 * kTile);
      load_tile<D>(sK, &tm_k, bar(kKVFull), key0, bh_kv, ext_kv, args.err);
      load_tile<D>(sV, &tm_v, bar(kKVFull), key0, bh_kv, ext_kv, args.err);
      int n_do = 0, n_q = 0;  // loads issued
      for (int it = 0; it < nit; ++it) {
        const int s = it & 1, u = it >> 1;
        const int q0 = q_block(it) * 128, bq = q_head(it);
        // Q first: S^T of a block is issued before its dP^T.
        if (u > 0 && !mbar_wait(bar(kQEmpty + s), (u - 1) & 1, args.err, kErrTimeoutRing)) break;
        mbar_expect_tx(bar(kQFull + s), kTile + 1024);
        load_tile<D>(sQ(s), &tm_q, bar(kQFull + s), q0, bq, ext_q, args.err);
        const long long nrows = (long long)args.BH * args.Npad, first = (long long)bq * args.Npad + q0;
        bulk_load_rows(sLD(s), args.lse_log2, first, 512, nrows, bar(kQFull + s), args.err);
        bulk_load_rows(sLD(s) + 512, args.delta, first, 512, nrows, bar(kQFull + s), args.err);
        ++n_q;
        if (u > 0 && !mbar_wait(bar(kDOEmpty + s), (u - 1) & 1, args.err, kErrTimeoutRing)) break;
        mbar_expect_tx(bar(kDOFull + s), kTile);
        load_tile<D>(sDO(s), &tm_do, bar(kDOFull + s), q0, bq, ext_q, args.err);
        ++n_do;
      }
      // Every copy this thread issued lands before the CTA exits, even when the
      // consumers gave up after a timeout elsewhere (bounded waits, abort ignored).
      mbar_wait(bar(kKVFull), 0, args.err, kErrTimeoutTma, false);
      for (int s = 0; s < 2; ++s) {
        if (n_q > s) mbar_wait(bar(kQFull + s), ((n_q - 1 - s) >> 1) & 1, args.err, kErrTimeoutTma, false);
        if (n_do > s) mbar_wait(bar(kDOFull + s), ((n_do - 1 - s) >> 1) & 1, args.err, kErrTimeoutTma, false);
      }
    }
  } else if (warp == C::kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // Order: S(0) dP(0) | dV(i) S(i+1) dK(i) dP(i+1) | ...  S(i+1) overwrites the
    // packed P^T(i) only after dV(i) has read it, and dP(i+1) overwrites dS^T(i)
    // only after dK(i) has read it, because one thread's tcgen05.mma operations
    // execute in issue order.  dO(i) is free once dV(i) completes, Q(i) once dK(i)
    // completes.
    if (lane == 0) {
      bool ok = mbar_wait(bar(kKVFull), 0, args.err, kErrTimeoutTma);
      if (ok) ok = mbar_wait(bar(kQFull + 0), 0, args.err, kErrTimeoutTma);
      if (ok) {
        tc_fence_after();
        mma_scores<D>(tmem + kTmS, sK, sQ(0), kIdSS(BF16));
        mma_commit(bar(kSReady));
        ok = mbar_wait(bar(kDOFull + 0), 0, args.err, kErrTimeoutTma);
      }
      if (ok) {
        tc_fence_after();
        mma_scores<D>(tmem + kTmDP, sV, sDO(0), kIdSS(BF16));
        mma_commit(bar(kDpReady));
      }
      for (int it = 0; ok && it < nit; ++it) {
        const int s = it & 1, s1 = (it + 1) & 1;
        if (!(ok = mbar_wait(bar(kPFull), it & 1, args.err, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        mma_packed<NWG>(tmem + kTmDV, tmem + kTmS, sDO(s), kIdTS(BF16, D), it > 0);
        mma_commit(bar(kDOEmpty + s));  // dO(it): last read by dV(it)
        if (it + 1 < nit) {
          if (!(ok = mbar_wait(bar(kQFull + s1), ((it + 1) >> 1) & 1, args.err, kErrTimeoutTma))) break;
          tc_fence_after();
          mma_scores<D>(tmem + kTmS, sK, sQ(s1), kIdSS(BF16));
          mma_commit(bar(kSReady));
        }
        if (!(ok = mbar_wait(bar(kDsFull), it & 1, args.err, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        mma_packed<NWG>(tmem + kTmDK, tmem + kTmDP, sQ(s), kIdTS(BF16, D), it > 0);
        mma_commit(bar(kQEmpty + s));   // Q(it): last read by dK(it)
        if (it + 1 < nit) {
          if (!(ok = mbar_wait(bar(kDOFull + s1), ((it + 1) >> 1) & 1, args.err, kErrTimeoutTma))) break;
          tc_fence_after();
          mma_scores<D>(tmem + kTmDP, sV, sDO(s1), kIdSS(BF16));
          mma_commit(bar(kDpReady));
        } else {
          mma_commit(bar(kDone));
        }
      }
      if (!ok) mma_commit(bar(kDone));  // lets the epilogue wait end; its result is discarded
      mbar_wait(bar(kDone), 0, args.err, kErrTimeoutMma, false);
    }
  } else if (warp < 4 * NWG) {
    // ------------------------------------------------------------ P^T, dS^T, epilogue
    const int e = warp >> 2;                 // warpgroup: query columns [kCols e, kCols (e + 1))
    const int r = ((warp & 3) << 5) + lane;  // TMEM lane: key row
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int cbeg = kCols * e;
    const int key = key0 + r;
    const float c = args.scale_log2;
    bool ok = true;
    for (int it = 0; it < nit; ++it) {
      const int q0 = q_block(it) * 128;
      const bool diag = args.causal && (key0 + 127 > q0 + koff);  // some key hidden from some query
      // ---- P^T = 2^(S^T c - L log2 e), packed into the S^T columns.  L log2 e and
      // D of the block's queries arrive with its Q tile.
      const uint32_t sl = sLD(it & 1) + 4u * cbeg, sd = sl + 512;
      if (!(ok = warp_wait(bar(kQFull + (it & 1)), (it >> 1) & 1, args.err, kErrTimeoutTma))) break;
      float4 l4[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) ld_shared_f4(sl + 16 * i, l4[i]);
      if (!(ok = warp_wait(bar(kSReady), it & 1, args.err, kErrTimeoutMma))) break;
      tc_fence_after();
      float p[kCols];
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) {
        uint32_t sv[32];
        tmem_ld_32x32b_x32(tmem + lane_base + kTmS + cbeg + 32 * ch, sv);
        if (ch > 0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) ld_shared_f4(sl + 128 * ch + 16 * i, l4[i]);
        }
        tmem_wait_ld();
        reg_fence32(sv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int x = 4 * i;
          float x0, x1, x2, x3;
          fma2v(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1]), c, -l4[i].x, -l4[i].y, x0, x1);
          fma2v(__uint_as_float(sv[x + 2]), __uint_as_float(sv[x + 3]), c, -l4[i].z, -l4[i].w, x2, x3);
          p[32 * ch + x] = ex2_approx(x0);
          p[32 * ch + x + 1] = ex2_approx(x1);
          p[32 * ch + x + 2] = ex2_approx(x2);
          p[32 * ch + x + 3] = ex2_approx(x3);
        }
        if (diag) {
#pragma unroll
          for (int x = 0; x < 32; ++x)
            if (key > q0 + cbeg + 32 * ch + x + koff) p[32 * ch + x] = 0.f;
        }
      }
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) {
        uint32_t pw[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) pw[x] = pack2<BF16>(p[32 * ch + 2 * x], p[32 * ch + 2 * x + 1]);
        tmem_st_32x32b_x16(tmem + lane_base + kTmS + cbeg + 16 * ch, pw);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(bar(kPFull));
      // ---- dS^T = P^T o (dP^T - D), packed into the dP^T columns
      if (!(ok = warp_wait(bar(kDpReady), it & 1, args.err, kErrTimeoutMma))) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) {
        uint32_t dv[32];
        tmem_ld_32x32b_x32(tmem + lane_base + kTmDP + cbeg + 32 * ch, dv);
        float4 d4[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) ld_shared_f4(sd + 128 * ch + 16 * i, d4[i]);
        tmem_wait_ld();
        reg_fence32(dv);
        uint32_t dw[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int x = 4 * i;
          float ds0, ds1, ds2, ds3;
          submul2(p[32 * ch + x], p[32 * ch + x + 1], __uint_as_float(dv[x]), __uint_as_float(dv[x + 1]), d4[i].x,
                  d4[i].y, ds0, ds1);
          submul2(p[32 * ch + x + 2], p[32 * ch + x + 3], __uint_as_float(dv[x + 2]), __uint_as_float(dv[x + 3]),
                  d4[i].z, d4[i].w, ds2, ds3);
          dw[x >> 1] = pack2<BF16>(ds0, ds1);
          dw[(x >> 1) + 1] = pack2<BF16>(ds2, ds3);
        }
        tmem_st_32x32b_x16(tmem + lane_base + kTmDP + cbeg + 16 * ch, dw);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(bar(kDsFull));
    }
    // ---- dV, dK of this key block once the last dK product has completed:
    // lane r holds key row key0 + r; the D / 32 column chunks go round-robin to the
    // warpgroups.
    if (ok && warp_wait(bar(kDone), 0, args.err, kErrTimeoutMma)) {
      tc_fence_after();
      const size_t out_row = ((size_t)bh_kv * Nk + key) * D;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t col0 = which == 0 ? kTmDV : kTmDK;
        const float mul = which == 0 ? 1.f : args.scale;
        uint16_t* dst = reinterpret_cast<uint16_t*>(which == 0 ? args.dv : args.dk) + out_row;
#pragma unroll 1
        for (int ch = e; ch < D / 32; ch += NWG) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem + lane_base + col0 + 32 * ch, v);
          tmem_wait_ld();
          reg_fence32(v);
          if (key < Nk) store_row32<BF16>(dst + 32 * ch, v, mul);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (kDebug) {
    if (threadIdx.x == 0 && no_abort(args.err)) {
      check_phase(bar(kKVFull), 1, args.err, kKVFull);
      for (int s = 0; s < 2; ++s)
        for (int b : {kQFull, kQEmpty, kDOFull, kDOEmpty}) check_phase(bar(b + s), count_mod(nit, s, 2), args.err, b + s);
      for (int b : {kSReady, kPFull, kDpReady, kDsFull}) check_phase(bar(b), nit, args.err, b);
      check_phase(bar(kDone), 1, args.err, kDone);
    }
  }
  if (warp == C::kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================ dQ
namespace qk {
template <int D>
struct Smem {
  static constexpr uint32_t T = tile_bytes<D>();
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kDO = T;
  static constexpr uint32_t kK = 2 * T;   // three stages (K is read by S and by dQ)
  static constexpr uint32_t kV = 5 * T;   // two stages (V is read by dP only)
  static constexpr uint32_t kBar = 7 * T;
};
enum : int {
  kQFull = 0,    // Q and dO tiles in shared memory
  kKFull = 1,    // three
  kKEmpty = 4,   // three
  kVFull = 7,    // two
  kVEmpty = 9,   // two
  kSReady = 11,  // S of the block is in TMEM
  kPDone = 12,   // S read out
  kDpReady = 13, // two, one per dP buffer: dP of the block is in the buffer
  kDsFull = 15,  // two: dS written into the buffer's first columns
  kDone = 17,    // the last dQ product has completed
  kNumBars
};
template <int D>
constexpr uint32_t tmem_slot() { return Smem<D>::kBar + kNumBars * 8; }
template <int D>
constexpr uint32_t smem_alloc() { return tmem_slot<D>() + 16 + 1024; }
static_assert(smem_alloc<128>() <= 232448, "shared memory budget");
// TMEM: S (fp32), two dP buffers (fp32, then dS packed into the first columns
// of its buffer), and the dQ accumulator.
constexpr uint32_t kTmS = 0;
constexpr uint32_t kTmDP = 128;  // buffer b at 128 + 128 b
constexpr uint32_t kTmDQ = 384;
}  // namespace qk

template <int D, int NWG, bool BF16>
__global__ void __launch_bounds__(SqCfg<NWG>::kThreadsQ, 1)
    fa_bwd_q_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdArgs args) {
  using namespace qk;
  using C = SqCfg<NWG>;
  using M = Smem<D>;
  constexpr int kCols = C::kCols, kCh = C::kCh;
  constexpr uint32_t kTile = M::T, kSmTmemSlot = tmem_slot<D>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + M::kBar + 8u * i; };
  auto sK = [&](int s) -> uint32_t { return sbase + M::kK + kTile * s; };
  auto sV = [&](int s) -> uint32_t { return sbase + M::kV + kTile * s; };
  const uint32_t sQ = sbase + M::kQ, sDO = sbase + M::kDO;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = args.N;
  const int Nk = args.Nk;

  // Work tile: the last query blocks first (under the causal mask they see the most
  // keys), so the final wave holds the lightest work; heads in groups of
  // args.head_group_q.
  const int nqb = (N + 127) / 128;
  int qb, bh;
  grouped_tile(blockIdx.x, args.BH, nqb, args.head_group_q, qb, bh);
  qb = nqb - 1 - qb;
  const int bh_kv = (bh / args.H) * (args.H / args.group) + (bh % args.H) / args.group;
  const int koff = Nk - N;  // key j visible to query i iff j <= i + koff
  const int q0 = qb * 128;
  int nkv = (Nk + 127) / 128;
  if (args.causal) {
    const int last = min(Nk - 1, q0 + 127 + koff);  // last key any row of the block sees
    nkv = last < 0 ? 0 : last / 128 + 1;
  }

  if (threadIdx.x == 0) {
    mbar_init(bar(kQFull), 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(bar(kKFull + s), 1);
      mbar_init(bar(kKEmpty + s), 2);  // K: read by S and dQ, one issuer each
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVEmpty + s), 1);
    }
    mbar_init(bar(kSReady), 1);
    mbar_init(bar(kPDone), C::kEw / 32);  // one arrival per elementwise warp
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kDpReady + b), 1);
      mbar_init(bar(kDsFull + b), C::kEw / 32);
    }
    mbar_init(bar(kDone), 2);  // both issuers
    fence_mbar_init();
  }
  if (warp == C::kWarpMma) {
    tmem_alloc(sbase + kSmTmemSlot, 512);
    tmem_relinquish();
  }
  if (warp == C::kWarpTma && lane == 0) {
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
  const Extent3 ext_q{D, N, args.BH}, ext_kv{D, Nk, args.BHkv};

  if (warp == C::kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && nkv > 0) {
      mbar_expect_tx(bar(kQFull), 2 * kTile);
      load_tile<D>(sQ, &tm_q, bar(kQFull), q0, bh, ext_q, args.err);
      load_tile<D>(sDO, &tm_do, bar(kQFull), q0, bh, ext_q, args.err);
      int n_k = 0, n_v = 0;  // loads issued
      for (int j = 0; j < nkv; ++j) {
        const int sk = j % 3, uk = j / 3, sv = j & 1, uv = j >> 1;
        if (uk > 0 && !mbar_wait(bar(kKEmpty + sk), (uk - 1) & 1, args.err, kErrTimeoutRing)) break;
        mbar_expect_tx(bar(kKFull + sk), kTile);
        load_tile<D>(sK(sk), &tm_k, bar(kKFull + sk), 128 * j, bh_kv, ext_kv, args.err);
        ++n_k;
        if (uv > 0 && !mbar_wait(bar(kVEmpty + sv), (uv - 1) & 1, args.err, kErrTimeoutRing)) break;
        mbar_expect_tx(bar(kVFull + sv), kTile);
        load_tile<D>(sV(sv), &tm_v, bar(kVFull + sv), 128 * j, bh_kv, ext_kv, args.err);
        ++n_v;
      }
      // Every copy this thread issued lands before the CTA exits.
      mbar_wait(bar(kQFull), 0, args.err, kErrTimeoutTma, false);
      for (int s = 0; s < 3; ++s)
        if (n_k > s) mbar_wait(bar(kKFull + s), ((n_k - 1 - s) / 3) & 1, args.err, kErrTimeoutTma, false);
      for (int s = 0; s < 2; ++s)
        if (n_v > s) mbar_wait(bar(kVFull + s), ((n_v - 1 - s) >> 1) & 1, args.err, kErrTimeoutTma, false);
    }
  } else if (warp == C::kWarpMma || warp == C::kWarpMma2) {
    // ------------------------------------------------------------ MMA issuers
    // Warp kWarpMma: S(j), as soon as S(j-1) has been read out.  Warp kWarpMma2:
    // dP(0) dP(1) | dQ(j) dP(j+2) | ...: dP(j+2) goes into the buffer of block j,
    // whose dS(j) dQ(j) has just read (one thread's operations execute in issue
    // order).  K(j) is read by S(j) and dQ(j): its slot is free once both issuers
    // have released it (each waits for it to land first).
    if (lane == 0 && nkv > 0) {
      bool ok = mbar_wait(bar(kQFull), 0, args.err, kErrTimeoutTma);
      auto kfull = [&](int j) { return mbar_wait(bar(kKFull + j % 3), (j / 3) & 1, args.err, kErrTimeoutTma); };
      if (warp == C::kWarpMma) {
        for (int j = 0; ok && j < nkv; ++j) {
          if (j > 0 && !(ok = mbar_wait(bar(kPDone), (j - 1) & 1, args.err, kErrTimeoutSoftmax))) break;
          if (!(ok = kfull(j))) break;
          tc_fence_after();
          mma_scores<D>(tmem + kTmS, sQ, sK(j % 3), kIdSS(BF16));
          mma_commit(bar(kSReady));
          mma_commit(bar(kKEmpty + j % 3));
        }
      } else {
        constexpr uint32_t kIdG = kIdTS(BF16, D);
        auto issue_dp = [&](int j) -> bool {
          if (!mbar_wait(bar(kVFull + (j & 1)), (j >> 1) & 1, args.err, kErrTimeoutTma)) return false;
          tc_fence_after();
          mma_scores<D>(tmem + kTmDP + 128 * (j & 1), sDO, sV(j & 1), kIdSS(BF16));
          mma_commit(bar(kDpReady + (j & 1)));
          mma_commit(bar(kVEmpty + (j & 1)));
          return true;
        };
        if (ok) ok = issue_dp(0);
        if (ok && nkv > 1) ok = issue_dp(1);
        for (int j = 0; ok && j < nkv; ++j) {
          const int b = j & 1;
          if (!(ok = mbar_wait(bar(kDsFull + b), (j >> 1) & 1, args.err, kErrTimeoutSoftmax) && kfull(j))) break;
          tc_fence_after();
          mma_packed<NWG>(tmem + kTmDQ, tmem + kTmDP + 128 * b, sK(j % 3), kIdG, j > 0);
          mma_commit(bar(kKEmpty + j % 3));
          if (j + 2 < nkv && !(ok = issue_dp(j + 2))) break;
        }
      }
      mma_commit(bar(kDone));
      mbar_wait(bar(kDone), 0, args.err, kErrTimeoutMma, false);
    }
  } else if (warp < 4 * NWG) {
    // ------------------------------------------------------------ P, dS, epilogue
    const int e = warp >> 2;                 // warpgroup: key columns [kCols e, kCols (e + 1))
    const int r = ((warp & 3) << 5) + lane;  // TMEM lane: query row
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int cbeg = kCols * e;
    const int q = q0 + r;
    const float c = args.scale_log2;
    const float Lr = args.lse_log2[(size_t)bh * args.Npad + q];  // +inf on padding rows: P = 0
    const float Dr = args.delta[(size_t)bh * args.Npad + q];
    bool ok = nkv > 0;
    for (int j = 0; ok && j < nkv; ++j) {
      const int k0 = 128 * j;
      // some key of the block hidden from some query: the causal diagonal, or keys past
      // N_k in the last block (their K, V rows are zero-filled, but P would not be:
      // 2^(-L) can overflow when a row's scores are all very negative)
      const bool diag = (args.causal && k0 + 127 > q0 + koff) || k0 + 128 > Nk;
      // ---- P = 2^(S c - L log2 e), kept in registers
      if (!(ok = warp_wait(bar(kSReady), j & 1, args.err, kErrTimeoutMma))) break;
      tc_fence_after();
      float p[kCols];
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) {
        uint32_t sv[32];
        tmem_ld_32x32b_x32(tmem + lane_base + kTmS + cbeg + 32 * ch, sv);
        tmem_wait_ld();
        reg_fence32(sv);
#pragma unroll
        for (int x = 0; x < 32; x += 2) {
          float x0, x1;
          fma2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1]), c, -Lr, x0, x1);
          p[32 * ch + x] = ex2_approx(x0);
          p[32 * ch + x + 1] = ex2_approx(x1);
        }
        if (diag) {
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int key = k0 + cbeg + 32 * ch + x;
            if ((args.causal && key > q + koff) || key >= Nk) p[32 * ch + x] = 0.f;
          }
        }
      }
      tc_fence_before();
      warp_arrive(bar(kPDone));  // S may be overwritten by the next block's scores now
      // ---- dS = P o (dP - D), packed into the first columns of this warpgroup's part
      // of the block's dP buffer
      const int b = j & 1;
      const uint32_t dpb = tmem + lane_base + kTmDP + 128 * b + cbeg;
      if (!(ok = warp_wait(bar(kDpReady + b), (j >> 1) & 1, args.err, kErrTimeoutMma))) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < kCh; ++ch) {
        uint32_t dv[32];
        tmem_ld_32x32b_x32(dpb + 32 * ch, dv);
        tmem_wait_ld();
        reg_fence32(dv);
        uint32_t dw[16];
#pragma unroll
        for (int x = 0; x < 32; x += 2) {
          float ds0, ds1;
          submul2(p[32 * ch + x], p[32 * ch + x + 1], __uint_as_float(dv[x]), __uint_as_float(dv[x + 1]), Dr, Dr,
                  ds0, ds1);
          dw[x >> 1] = pack2<BF16>(ds0, ds1);
        }
        tmem_st_32x32b_x16(dpb + 16 * ch, dw);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(bar(kDsFull + b));
    }
    // ---- dQ rows: lane r holds query row q; the D / 32 column chunks go round-robin
    // to the warpgroups.
    if (nkv == 0 || (ok && warp_wait(bar(kDone), 0, args.err, kErrTimeoutMma))) {
      tc_fence_after();
      uint16_t* dst = reinterpret_cast<uint16_t*>(args.dq) + ((size_t)bh * N + q) * D;
#pragma unroll 1
      for (int ch = e; ch < D / 32; ch += NWG) {
        uint32_t v[32];
        if (nkv > 0) {
          tmem_ld_32x32b_x32(tmem + lane_base + kTmDQ + 32 * ch, v);
          tmem_wait_ld();
          reg_fence32(v);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] = 0u;  // rows that see no key: dQ = 0
        }
        if (q < N) store_row32<BF16>(dst + 32 * ch, v, args.scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (kDebug) {
    if (threadIdx.x == 0 && no_abort(args.err)) {
      check_phase(bar(kQFull), nkv > 0, args.err, kQFull);
      for (int s = 0; s < 3; ++s) {
        check_phase(bar(kKFull + s), count_mod(nkv, s, 3), args.err, kKFull + s);
        check_phase(bar(kKEmpty + s), count_mod(nkv, s, 3), args.err, kKEmpty + s);
      }
      for (int s = 0; s < 2; ++s)
        for (int b : {kVFull, kVEmpty, kDpReady, kDsFull}) check_phase(bar(b + s), count_mod(nkv, s, 2), args.err, b + s);
      check_phase(bar(kSReady), nkv, args.err, kSReady);
      check_phase(bar(kPDone), nkv, args.err, kPDone);
      check_phase(bar(kDone), nkv > 0, args.err, kDone);
    }
  }
  if (warp == C::kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Two elementwise warpgroups (64 tile columns a thread): measured 4-6 % faster than
// four (fewer warps moving scores through tensor memory beside the products) and
// than one, at d = 64 and 128 alike.
constexpr int kBwdSqWarpgroups = 2;

template <int D, bool BF16>
cudaError_t launch_sq(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout,
                      const BwdArgs& a, cudaStream_t stream) {
  constexpr int kNwg = kBwdSqWarpgroups;
  constexpr int kThreadsKV = SqCfg<kNwg>::kThreadsKV, kThreadsQ = SqCfg<kNwg>::kThreadsQ;
  constexpr uint32_t kKvSmem = kv::smem_alloc<D>(), kQSmem = qk::smem_alloc<D>();
  auto kkv = fa_bwd_kv_kernel<D, kNwg, BF16>;
  auto kq = fa_bwd_q_kernel<D, kNwg, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kKvSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQSmem);
  if (e != cudaSuccess) return e;
  const long long grid_kv = (long long)((a.Nk + 127) / 128) * a.BHkv;
  const long long grid_q = (long long)((a.N + 127) / 128) * a.BH;
  profile_mark_begin(stream);
  kkv<<<(unsigned)grid_kv, kThreadsKV, kKvSmem, stream>>>(q, k, v, dout, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  profile_mark_end(stream, kProfileBwdKV);
  profile_mark_begin(stream);
  kq<<<(unsigned)grid_q, kThreadsQ, kQSmem, stream>>>(q, k, v, dout, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  profile_mark_end(stream, kProfileBwdQ);
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd_main_sq(int d, bool bf16, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& dout, const BwdArgs& a, cudaStream_t stream) {
  switch (d) {
    case 64:
      return bf16 ? launch_sq<64, true>(q, k, v, dout, a, stream) : launch_sq<64, false>(q, k, v, dout, a, stream);
    case 128:
      return bf16 ? launch_sq<128, true>(q, k, v, dout, a, stream) : launch_sq<128, false>(q, k, v, dout, a, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace fa
