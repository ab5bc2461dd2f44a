// fwd_kernel.cuh -- exact flash-attention forward for sm_103a (TMA + tcgen05 + TMEM).
//
// Work partition ("From-scratch CUDA attention kernel reaches 94.4% of
// FlashAttention-4 on NVIDIA B200", section "How the kernel partitions its
// work"): Q, K, V and O are cut into 128-row tiles; a work unit is one
// (batch, query head) and TWO consecutive 128-row Q tiles, loaded once, whose
// K/V tiles stream through a shared-memory ring.  One CTA per unit, except
// in the split-key mode with more units than SMs (PERSIST): there at most one
// CTA per SM walks its share of the units (see unit_index), so barriers and
// TMEM are set up once per CTA and the next unit's Q and K/V loads overlap the
// current unit's last steps and epilogue.  For each K/V tile: S = Q K^T (tensor cores, fp32 in TMEM), an online
// softmax update (running row max m and running row sum l, FlashStieltjes
// page, "The challenge"), P (bf16, written back over S in TMEM), and
// O += P V (tensor cores, fp32 in TMEM).  At the end O / l is written as bf16
// and LSE = ln 2 * (m + log2 l).
//
// Warp roles (12 warps, three warpgroups):
//   warps 0-3   softmax for Q tile 0 (one thread per row, TMEM lanes 0-127)
//   warps 4-7   softmax for Q tile 1
//   warp  8     TMA producer: Q tiles, then K_0, V_0, K_1, V_1, ... into the ring
//   warp  9     TMEM allocator and tcgen05.mma issuer
//   warps 10-11 idle; they complete the third warpgroup for the register split
// Registers: launched at 168 per thread (the cap when 3 warps share an SM
// sub-partition); the third warpgroup gives registers back (setmaxnreg.dec to
// 56) and the softmax warpgroups take them (224): 2*224 + 56 = 3*168.  With
// 128 scores live per row, the extra registers let many exp2 chains be in
// flight at once; at 168 the compiler could keep only a few.
// MMA issue order per K/V tile j (two Q tiles ping-pong so that one tile's
// softmax overlaps the other tile's matmuls):
//   S0_j = Q0 K_j^T ; O1 += P1_{j-1} V_{j-1} ; S1_j = Q1 K_j^T ; O0 += P0_j V_j
// P_t aliases S_t; tcgen05.mma operations issued by one thread execute in
// order, so S_t(j+1) never overwrites P_t(j) before O_t += P_t(j) V_j read it.
//
// Softmax is computed in base 2 with c = scale * log2(e):  p = 2^(s*c - m).
// The reference maximum m is raised only when the new row maximum exceeds it
// by more than kRescaleThreshold (2^8); then O and l are rescaled by
// 2^(m_old - m_new).  O and l always share the same m, so O / l and the LSE
// are unchanged by the choice; p <= 2^8 keeps bf16/fp32 far from overflow.
//
// Causal (FlashAttention for Tesla P100 page, "What it supports"): tiles
// entirely above the diagonal are skipped, not masked; only the diagonal
// tile is masked (key > query -> -inf).  Ragged N: TMA zero-fills rows past N
// inside each (batch, head) plane, key columns >= N are masked to -inf, and
// rows >= N are never stored.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "ptx.cuh"
#include "kernels.h"

namespace attn {

constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct FwdCfg {
  static constexpr int kTileRows = 128;
  static constexpr int kTileBytes = kTileRows * D * 2;  // one Q/K/V tile in bf16
  static constexpr int kBoxBytes = kTileRows * 128;     // one 64-column TMA box (128 B rows)
  static constexpr int kBoxes = D / 64;
  static constexpr int kStages = (D == 128) ? 4 : 6;
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = 2 * kTileBytes;
  static constexpr int kBarOff = kRingOff + kStages * kTileBytes;
  // barriers: q_full, full[kStages], empty[kStages], s_full[2], p_full[2], o_final,
  // q_empty, o_free[2]
  static constexpr int kNumBars = 1 + 2 * kStages + 8;
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;  // + misc + alignment slack
  static constexpr int kThreads = 384;
  // Register split (per thread): 8 softmax warps, 4 other warps.
  static constexpr int kRegSoftmax = 224, kRegOther = 56;
  static_assert(8 * kRegSoftmax + 4 * kRegOther == 12 * launch_regs(kThreads),
                "the register split must add up to the launch allocation");
  static constexpr uint32_t kTmemCols = 512;
};

// Position in the K/V ring: stage and the parity of its current use,
// advanced one entry at a time (no division by the stage count).
struct RingPos {
  int s = 0;
  uint32_t ph = 0;
  template <int ST>
  __device__ __forceinline__ void advance() {
    if (++s == ST) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// One work unit: query tiles t0 (slot 0) and t1 (slot 1) of one (batch, query
// head); n0 / n1 key tiles for the two slots (KVSPLIT: t0 == t1, slot 0 takes
// key tiles [0, h0), slot 1 [h0, h0 + n1)).
struct FwdUnit {
  int bh, b, h, bh_kv;
  int seq0, N;  // first token and length of the unit's sequence
  int t0, t1, h0, n0, n1, nkv;
  bool has_t1;
};

// VARLEN: a batch of sequences of different lengths packed token-major,
// q/o [total, Hq, D], k/v [total, Hkv, D], lse [Hq, total]; sequence b is
// rows cu_seqlens[b] .. cu_seqlens[b+1]-1.  The grid is that of a batch of
// max_seqlen-long sequences (p.N = max_seqlen), one unit per CTA; CTAs past
// their sequence's end leave at once.  The TMA maps address a head's rows
// with a stride of H*D elements (box 64 x 1 head x 128 tokens), which lands in
// shared memory exactly as a dense tile; key rows past the sequence are masked
// like a ragged tail and query rows past it are not written.
//
// KVSPLIT: one 128-row query tile per unit, its key range cut in two halves
// that the two tile slots (TMEM S/O pairs, softmax warpgroups) process side
// by side -- slot 0 key tiles [0, n/2), slot 1 [n/2, n) -- and merged at the
// end from each slot's (max, sum, O).  For grids of less than one wave of
// tile pairs: every step keeps both slots busy and the longest unit runs
// about n/2 steps, where pairing query tiles t and T-1-t (so that every unit
// runs T+1 steps) leaves one slot idle in most steps.
//
// PERSIST (split-key mode only): at most one CTA per SM, each walking its
// units (see unit_index); the host uses it when there are more units than
// SMs, so that a CTA's second unit's set-up and first loads hide under its
// first unit's last steps.  Otherwise every CTA runs one unit.
template <int D, bool CAUSAL, bool F16, bool VARLEN = false, bool KVSPLIT = false,
          bool PERSIST = false>
__global__ void __launch_bounds__(384, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using Cfg = FwdCfg<D>;
  static_assert(!KVSPLIT || !VARLEN, "KVSPLIT is a mode of the dense kernel");
  static_assert(!PERSIST || KVSPLIT, "persistent CTAs are used in the split-key mode");
  constexpr int ST = Cfg::kStages;

  // ---- work units, in the order of their index u:
  //  * Non-causal: adjacent tiles (2qb, 2qb+1); the units of one head are
  //    consecutive so that those in flight at one time share its K/V in L2.
  //  * Causal: adjacent tiles, longest blocks of all heads first (both tiles
  //    are active in almost every step, so the MMAs of one overlap the
  //    softmax of the other).
  //  * KVSPLIT: qb is the unit's one query tile, longest first when causal.
  const int BH = p.B * p.Hq;
  const int nqb = KVSPLIT ? p.num_kv_tiles : p.num_qblocks;
  const int units = nqb * BH;
  const int G = (int)gridDim.x;
  // Units per CTA: several only with PERSIST, in the split-key mode (grids
  // of tile pairs under one wave), where each CTA has one or two units.
  // Grids of tile pairs keep one unit per CTA: with several units per CTA
  // the static assignment measured 2-4 % slower than the hardware's dispatch
  // of whole CTAs to the SMs that free up first.
  constexpr bool kPersist = PERSIST;
  constexpr int kMaxUnits = kPersist ? 0x7FFFFFFF : 1;
  // The k-th unit of this CTA: rounds of G consecutive units, walked forwards
  // in even rounds and backwards in odd ones, so that (longest first) the
  // CTA that took a round's longest unit takes the next round's shortest.
  // A packed batch (VARLEN) keeps one unit per CTA: its lengths are known on
  // the device only.
  auto unit_index = [&](int k) -> int {
    if (!kPersist) return k == 0 ? (int)blockIdx.x : -1;
    const int r = k * G + ((k & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
    return r < units ? r : -1;
  };
  auto decode = [&](int u) {
    FwdUnit U;
    const int qb = CAUSAL ? nqb - 1 - u / BH : u % nqb;
    U.bh = CAUSAL ? u % BH : u / nqb;
    U.b = U.bh / p.Hq;
    U.h = U.bh % p.Hq;
    U.bh_kv = U.b * p.Hkv + U.h / p.G;
    U.seq0 = 0;
    U.N = p.N;
    if constexpr (VARLEN) {
      U.seq0 = p.cu_seqlens[U.b];
      U.N = p.cu_seqlens[U.b + 1] - U.seq0;
    }
    const int T = VARLEN ? (U.N + 127) / 128 : p.num_kv_tiles;
    U.t0 = KVSPLIT ? qb : 2 * qb;
    U.t1 = KVSPLIT ? qb : 2 * qb + 1;
    U.has_t1 = KVSPLIT || U.t1 * 128 < U.N;
    const int n_all = CAUSAL ? qb + 1 : T;  // KVSPLIT: the query tile's key tiles
    U.h0 = KVSPLIT ? n_all / 2 : 0;
    U.n0 = KVSPLIT ? U.h0 : (CAUSAL ? U.t0 + 1 : T);
    U.n1 = KVSPLIT ? n_all - U.h0 : (U.has_t1 ? (CAUSAL ? U.t1 + 1 : T) : 0);
    U.nkv = max(U.n0, U.n1);
    return U;
  };
  // The CTA's first unit, decoded by every thread before the set-up (the
  // integer divisions overlap it); later units are decoded by each role.
  const FwdUnit U0 = decode((int)blockIdx.x);
  if constexpr (VARLEN) {
    // lengths must lie in [0, max_seqlen] and sequences inside [0, total)
    if (U0.seq0 < 0 || U0.N < 0 || U0.N > p.N || U0.seq0 > p.total - U0.N) {
      if (threadIdx.x == 0) atomicOr(p.err, kErrSeqlen);
      return;
    }
    if (U0.t0 * 128 >= U0.N) return;  // past this sequence's end
  }
  // TMA coordinates of a 128-row tile: (column, row, plane) of the dense
  // (D, N, B*H) map, or (column, head, token) of the packed (D, H, total) map
  auto load_tile = [&](uint32_t dst, const CUtensorMap* tm, uint32_t bar, int c, int tile,
                       int plane, int head, int seq0) {
    if constexpr (VARLEN)
      tma_load_3d(dst, tm, bar, c * 64, head, seq0 + tile * 128);
    else
      tma_load_3d(dst, tm, bar, c * 64, tile * 128, plane);
  };
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_base + pad;

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = (int)(threadIdx.x & 31);

  const uint32_t bar0 = sbase + Cfg::kBarOff;
  auto bar_q = [&]() { return bar0; };
  auto bar_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_empty = [&](int s) { return bar0 + 8u * (1 + ST + s); };
  auto bar_s = [&](int t) { return bar0 + 8u * (1 + 2 * ST + t); };
  auto bar_p = [&](int t) { return bar0 + 8u * (3 + 2 * ST + t); };
  auto bar_o = [&]() { return bar0 + 8u * (5 + 2 * ST); };       // a unit's MMAs all done
  auto bar_qe = [&]() { return bar0 + 8u * (6 + 2 * ST); };      // a unit's S MMAs all done
  auto bar_of = [&](int t) { return bar0 + 8u * (7 + 2 * ST + t); };  // O_t read out
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kBarOff + Cfg::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    mbar_init(bar_q(), 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s(t), 1);
      mbar_init(bar_p(t), 4);
      // KVSPLIT: both warpgroups read both O accumulators in the merge
      mbar_init(bar_of(t), KVSPLIT ? 8 : 4);
    }
    mbar_init(bar_o(), 1);
    mbar_init(bar_qe(), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{p.timeout_ns, p.err, abort_flag};

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    regs_decrease<Cfg::kRegOther>();
    if (lane == 0) {
      uint32_t it = 0;  // ring entries issued (over all units)
      RingPos rp;       // ring position of entry `it`
      int nql = 0;      // Q loads issued
      bool ok = true;
      for (int k = 0; k < kMaxUnits && ok; ++k) {
        const int u = unit_index(k);
        if (u < 0) break;
        const FwdUnit U = k == 0 ? U0 : decode(u);
        // The unit's Q tiles replace the previous unit's once its S MMAs are done.
        if (k > 0 && !(ok = mbar_wait_tested_inl(bar_qe(), (uint32_t)(k - 1) & 1u, wc))) break;
        const int nq = (U.has_t1 && !KVSPLIT) ? 2 : 1;
        mbar_arrive_expect_tx(bar_q(), nq * Cfg::kTileBytes);
        for (int t = 0; t < nq; ++t)
          for (int c = 0; c < Cfg::kBoxes; ++c)
            load_tile(sbase + Cfg::kQOff + t * Cfg::kTileBytes + c * Cfg::kBoxBytes, &tm_q,
                      bar_q(), c, t ? U.t1 : U.t0, U.bh, U.h, U.seq0);
        ++nql;
        for (int j = 0; j < U.nkv && ok; ++j) {
          // Ring entries of step j: K_j, V_j; with KVSPLIT K of slot 0 (while it
          // is active) and of slot 1, then V of slot 0 and of slot 1.
          for (int e = 0; e < (KVSPLIT ? 4 : 2) && ok; ++e) {
            const int kv = KVSPLIT ? (e >> 1) : e;
            const int slot = e & 1;
            if (KVSPLIT && slot == 0 && j >= U.n0) continue;
            const int tile = (KVSPLIT && slot) ? U.h0 + j : j;
            const int s = rp.s;
            ok = mbar_wait_inl(bar_empty(s), rp.ph ^ 1u, wc);
            if (!ok) break;
            mbar_arrive_expect_tx(bar_full(s), Cfg::kTileBytes);
            const CUtensorMap* tm = kv ? &tm_v : &tm_k;
            for (int c = 0; c < Cfg::kBoxes; ++c)
              load_tile(sbase + Cfg::kRingOff + s * Cfg::kTileBytes + c * Cfg::kBoxBytes, tm,
                        bar_full(s), c, tile, U.bh_kv, U.h / p.G, U.seq0);
            ++it;
            rp.advance<ST>();
          }
        }
      }
      if (!ok) {
        // Let every copy already issued land before the CTA can exit.
        for (uint32_t f = (it > (uint32_t)ST ? it - ST : 0); f < it; ++f)
          mbar_wait_drain_inl(bar_full((int)(f % ST)), (f / ST) & 1u, wc);
        if (nql > 0) mbar_wait_drain_inl(bar_q(), (uint32_t)(nql - 1) & 1u, wc);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    regs_decrease<Cfg::kRegOther>();
    if (lane == 0) {
      constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, 0, 0, F16);
      constexpr uint32_t kIdescO = make_idesc_bf16(128, D, 1, 0, F16);
      const uint32_t q_addr[2] = {sbase + Cfg::kQOff, sbase + Cfg::kQOff + Cfg::kTileBytes};
      const uint32_t tS[2] = {tmem_base, tmem_base + 128};
      const uint32_t tO[2] = {tmem_base + 256, tmem_base + 384};
      auto ring = [&](int s) { return sbase + Cfg::kRingOff + s * Cfg::kTileBytes; };
      // Descriptors as an address word per tile plus a K-step offset added inside
      // the MMA's asm (one register per tile; nothing hoisted per K step).
      constexpr uint32_t kHi = sdesc_sw128_hi(1024);
      // (KVSPLIT: both slots multiply the one Q tile)
      const uint32_t q_lo[2] = {sdesc_sw128_lo(q_addr[0], 16),
                                sdesc_sw128_lo(q_addr[KVSPLIT ? 0 : 1], 16)};
      auto koff = [](int kk) {  // K-major: 32-byte steps inside a 64-column box, then a box
        return (uint32_t)(((kk / 4) * Cfg::kBoxBytes + (kk % 4) * 32) >> 4);
      };
      auto issue_qk = [&](int t, uint32_t kaddr) {
        const uint32_t k_lo = sdesc_sw128_lo(kaddr, 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_w(tS[t], q_lo[t], koff(kk), k_lo, koff(kk), kHi, kIdescS, kk > 0);
      };
      auto issue_pv = [&](int t, uint32_t vaddr, bool acc) {
        const uint32_t v_lo = sdesc_sw128_lo(vaddr, Cfg::kBoxBytes);  // MN-major: 16 rows per step
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_w(tO[t], tS[t] + kk * 8, v_lo, (uint32_t)((kk * 2048) >> 4), kHi, kIdescO,
                   (acc || kk > 0) ? 1u : 0u);
      };

      bool ok = true;
      uint32_t np0 = 0, np1 = 0;
      RingPos rp;  // next ring entry to consume
      int k = 0;
      for (; k < kMaxUnits && ok; ++k) {
        const int u = unit_index(k);
        if (u < 0) break;
        const FwdUnit U = k == 0 ? U0 : decode(u);
        const int n0 = U.n0, n1 = U.n1, nkv = U.nkv;
        if (!(ok = mbar_wait_inl(bar_q(), (uint32_t)k & 1u, wc))) break;
        // A unit's first P.V MMA of slot t overwrites O_t: the softmax warps must
        // have read the previous unit's O_t out of TMEM (phase k-1 of bar_of(t)).
        const uint32_t of_ph = (uint32_t)(k - 1) & 1u;
        bool of0 = k == 0, of1 = k == 0;
        int sv_prev = 0;
        bool a1_prev = false;
        if constexpr (KVSPLIT) {
          // Order per step j, consuming the ring entries in the producer's order
          // K_0(j), K_1(j), V_0(j), V_1(j): S_0(j); O_1 += P_1(j-1) V_1(j-1);
          // S_1(j); O_0 += P_0(j) V_0(j) -- each softmax gets the duration of
          // the other slot's two MMAs, as with two query tiles.
          auto next = [&](int& s, uint32_t& ph) {
            s = rp.s;
            ph = rp.ph;
            rp.advance<ST>();
          };
          int svb = 0;
          uint32_t phvb = 0;
          for (int j = 0; j < nkv && ok; ++j) {
            const bool a0 = j < n0;
            int s;
            uint32_t ph;
            if (a0) {
              next(s, ph);
              if (!(ok = mbar_wait_inl(bar_full(s), ph, wc))) break;
              tc_fence_after();
              issue_qk(0, ring(s));
              mma_commit(bar_s(0));
              mma_commit(bar_empty(s));
            }
            if (j > 0) {
              if (!(ok = mbar_wait_inl(bar_full(svb), phvb, wc))) break;
              if (!(ok = mbar_wait_inl(bar_p(1), np1 & 1u, wc))) break;
              if (!of1 && !(ok = mbar_wait_inl(bar_of(1), of_ph, wc))) break;
              of1 = true;
              ++np1;
              tc_fence_after();
              issue_pv(1, ring(svb), j - 1 > 0);
              mma_commit(bar_empty(svb));
            }
            next(s, ph);
            if (!(ok = mbar_wait_inl(bar_full(s), ph, wc))) break;
            tc_fence_after();
            issue_qk(1, ring(s));
            mma_commit(bar_s(1));
            mma_commit(bar_empty(s));
            if (a0) {
              next(s, ph);
              if (!(ok = mbar_wait_inl(bar_full(s), ph, wc))) break;
              if (!(ok = mbar_wait_inl(bar_p(0), np0 & 1u, wc))) break;
              if (!of0 && !(ok = mbar_wait_inl(bar_of(0), of_ph, wc))) break;
              of0 = true;
              ++np0;
              tc_fence_after();
              issue_pv(0, ring(s), j > 0);
              mma_commit(bar_empty(s));
            }
            next(svb, phvb);  // V_1(j): waited for where it is used
          }
          if (ok) mma_commit(bar_qe());  // every S MMA of the unit is issued
          if (ok && nkv > 0) {
            ok = mbar_wait_inl(bar_full(svb), phvb, wc) && mbar_wait_inl(bar_p(1), np1 & 1u, wc) &&
                 (of1 || mbar_wait_inl(bar_of(1), of_ph, wc));
            if (ok) {
              ++np1;
              tc_fence_after();
              issue_pv(1, ring(svb), nkv - 1 > 0);
              mma_commit(bar_empty(svb));
            }
          }
        }
        for (int j = 0; j < (KVSPLIT ? 0 : nkv) && ok; ++j) {
          const bool a0 = j < n0, a1 = j < n1;
          const int sk = rp.s;
          const uint32_t phk = rp.ph;
          rp.advance<ST>();
          const int sv = rp.s;
          const uint32_t phv = rp.ph;
          rp.advance<ST>();
          if (!(ok = mbar_wait_inl(bar_full(sk), phk, wc))) break;
          tc_fence_after();
          if (a0) {
            issue_qk(0, ring(sk));
            mma_commit(bar_s(0));
          }
          if (j > 0 && a1_prev) {
            if (!(ok = mbar_wait_inl(bar_p(1), np1 & 1u, wc))) break;
            if (!of1 && !(ok = mbar_wait_inl(bar_of(1), of_ph, wc))) break;
            of1 = true;
            ++np1;
            tc_fence_after();
            issue_pv(1, ring(sv_prev), j - 1 > 0);
          }
          if (j > 0) mma_commit(bar_empty(sv_prev));
          if (a1) {
            issue_qk(1, ring(sk));
            mma_commit(bar_s(1));
          }
          mma_commit(bar_empty(sk));
          if (!(ok = mbar_wait_inl(bar_full(sv), phv, wc))) break;
          tc_fence_after();
          if (a0) {
            if (!(ok = mbar_wait_inl(bar_p(0), np0 & 1u, wc))) break;
            if (!of0 && !(ok = mbar_wait_inl(bar_of(0), of_ph, wc))) break;
            of0 = true;
            ++np0;
            tc_fence_after();
            issue_pv(0, ring(sv), j > 0);
          }
          sv_prev = sv;
          a1_prev = a1;
        }
        if (!KVSPLIT && ok) {
          mma_commit(bar_qe());  // every S MMA of the unit is issued
          if (a1_prev) {
            if ((ok = mbar_wait_inl(bar_p(1), np1 & 1u, wc) &&
                      (of1 || mbar_wait_inl(bar_of(1), of_ph, wc)))) {
              ++np1;
              tc_fence_after();
              issue_pv(1, ring(sv_prev), nkv - 1 > 0);
            }
          }
          // the last V tile: no S MMA of this unit reads the ring after it
          if (ok && nkv > 0) mma_commit(bar_empty(sv_prev));
        }
        if (ok) mma_commit(bar_o());
      }
      // On an aborted run nobody else may wait for the final commit: wait here
      // so that no MMA is in flight when TMEM is released.
      if (!ok) {
        mma_commit(bar_o());
        mbar_wait_drain_inl(bar_o(), (uint32_t)k & 1u, wc);
      }
    }
  } else if (warp >= 10) {
    regs_decrease<Cfg::kRegOther>();
  } else {
    // ------------------------------------------------------------ softmax
    regs_increase<Cfg::kRegSoftmax>();
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem_base + lane_off + (uint32_t)(t * 128);
    const uint32_t tO = tmem_base + lane_off + 256u + (uint32_t)(t * 128);
    const float C = p.scale_log2;
    uint32_t ns = 0;  // S tiles of this slot waited for (over all units)
    bool ok = true;
    for (int k = 0; k < kMaxUnits && ok; ++k) {
      const int u = unit_index(k);
      if (u < 0) break;
      const FwdUnit U = k == 0 ? U0 : decode(u);
      const int n_t = t ? U.n1 : U.n0;
      const int qtile = t ? U.t1 : U.t0;
      const int grow = qtile * 128 + row;
      const int N = U.N;
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < n_t; ++j) {
        // tcgen05.ld/st are warp-collective: keep the decision warp-uniform.
        ok = __all_sync(0xffffffffu, mbar_wait_inl(bar_s(t), ns & 1u, wc));
        ++ns;
        if (!ok) break;
        tc_fence_after();
        float s[128];
        {
          uint32_t r[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, r[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[c][i]);
        }
        const int kvt = (KVSPLIT && t) ? U.h0 + j : j;  // key tile of this step
        const int kv0 = kvt * 128;
        if ((CAUSAL && kvt == qtile) || kv0 + 128 > N) {
          int lim = N - kv0;  // columns >= lim are past the sequence end
          if (CAUSAL) lim = min(lim, grow - kv0 + 1);  // causal: key <= query
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim) s[c] = -INFINITY;
        }
        float mp[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mp[q] = fmaxf(s[q], s[q + 8]);
#pragma unroll
        for (int c = 16; c < 128; c += 16)
#pragma unroll
          for (int q = 0; q < 8; ++q) mp[q] = fmax3(mp[q], s[c + q], s[c + 8 + q]);
        const float mx = fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]),
                               fmaxf(mp[6], mp[7]));
        const float m_new = fmaxf(m_used, mx * C);
        const bool need = (m_new - m_used) > kRescaleThreshold;
        const float corr = need ? ex2_approx(m_used - m_new) : 1.f;
        if (need) m_used = m_new;
        l *= corr;
        const float2 c2 = make_float2(C, C);
        const float2 nm2 = make_float2(-m_used, -m_used);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), c2, nm2);
          const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          acc[(c >> 1) & 3] = __fadd2_rn(acc[(c >> 1) & 3], pp);
          pk[c / 2] = pack2<F16>(pp.x, pp.y);
          if (c == 62) tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        }
        tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
        const float2 a = __fadd2_rn(a01, a23);
        l += a.x + a.y;
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // O_t is stable here: its last update was committed before S_t(j).
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t r[32];
            tmem_ld32(tO + c, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
            tmem_st32(tO + c, r);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p(t));
      }
      // Every warp waits for the unit's MMAs, with or without steps of its own,
      // so that all roles move from unit to unit together.
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait_inl(bar_o(), (uint32_t)k & 1u, wc));
      if constexpr (KVSPLIT) {
        // Merge the two slots' partial results of the same rows: each thread
        // publishes its (m, l) through the unused second Q buffer; then
        // warpgroup t writes output columns [t D/2, (t+1) D/2) and warpgroup 0
        // the LSE.  Both warpgroups pass this named barrier once per unit, the
        // shared decision included, so they leave the unit loop together.
        float* xm = reinterpret_cast<float*>(smem + Cfg::kQOff + Cfg::kTileBytes);
        xm[(2 * t) * 128 + row] = m_used;
        xm[(2 * t + 1) * 128 + row] = l;
        ok = named_bar_and(1, 256, ok);
        if (ok) {
          tc_fence_after();
          const int n0 = U.n0;
          const float m0 = xm[row], l0 = xm[128 + row], m1 = xm[256 + row], l1 = xm[384 + row];
          const float m = n0 > 0 ? fmaxf(m0, m1) : m1;
          const float a0 = n0 > 0 ? ex2_approx(m0 - m) : 0.f;
          const float a1 = ex2_approx(m1 - m);
          const float L = a0 * l0 + a1 * l1;
          const float s0 = a0 / L, s1 = a1 / L;
          const bool live = grow < N;
          uint4* orow = reinterpret_cast<uint4*>(
              static_cast<uint16_t*>(p.o) + ((size_t)U.bh * p.N + (size_t)(live ? grow : 0)) * D);
          const uint32_t tO0 = tmem_base + lane_off + 256u, tO1 = tmem_base + lane_off + 384u;
#pragma unroll
          for (int c = t * (D / 2); c < (t + 1) * (D / 2); c += 32) {
            uint32_t r0[32], r1[32];
            tmem_ld32(tO1 + c, r1);
            if (n0 > 0) tmem_ld32(tO0 + c, r0);
            tmem_ld_wait();
            float o[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
              o[i] = __uint_as_float(r1[i]) * s1 + (n0 > 0 ? __uint_as_float(r0[i]) * s0 : 0.f);
            if (live) {
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 w;
                w.x = pack2<F16>(o[8 * v + 0], o[8 * v + 1]);
                w.y = pack2<F16>(o[8 * v + 2], o[8 * v + 3]);
                w.z = pack2<F16>(o[8 * v + 4], o[8 * v + 5]);
                w.w = pack2<F16>(o[8 * v + 6], o[8 * v + 7]);
                orow[c / 8 + v] = w;
              }
            }
          }
          if (t == 0 && live)
            p.lse[(size_t)U.bh * p.N + grow] = (m + log2f(L)) * 0.69314718055994530942f;
        }
      }
      if (!KVSPLIT && ok && n_t > 0) {
        tc_fence_after();
        const float inv_l = 1.f / l;
        const bool live = grow < N;
        // row grow of the output: dense [B*Hq, N, D], or packed [total, Hq, D]
        const size_t orow_idx = VARLEN ? ((size_t)(U.seq0 + (live ? grow : 0)) * p.Hq + U.h)
                                       : ((size_t)U.bh * p.N + (size_t)(live ? grow : 0));
        uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + orow_idx * D);
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t r[32];
          tmem_ld32(tO + c, r);
          tmem_ld_wait();
          if (live) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 w;
              w.x = pack2<F16>(__uint_as_float(r[8 * v + 0]) * inv_l, __uint_as_float(r[8 * v + 1]) * inv_l);
              w.y = pack2<F16>(__uint_as_float(r[8 * v + 2]) * inv_l, __uint_as_float(r[8 * v + 3]) * inv_l);
              w.z = pack2<F16>(__uint_as_float(r[8 * v + 4]) * inv_l, __uint_as_float(r[8 * v + 5]) * inv_l);
              w.w = pack2<F16>(__uint_as_float(r[8 * v + 6]) * inv_l, __uint_as_float(r[8 * v + 7]) * inv_l);
              orow[c / 8 + v] = w;
            }
          }
        }
        // LSE: dense [B*Hq, N], packed [Hq, total]
        const size_t lse_idx =
            VARLEN ? (size_t)U.h * p.total + U.seq0 + grow : (size_t)U.bh * p.N + grow;
        if (live) p.lse[lse_idx] = (m_used + log2f(l)) * 0.69314718055994530942f;
      }
      // This warp has read O out of TMEM: the next unit's first P.V may
      // overwrite it (KVSPLIT: both accumulators, read by both warpgroups).
      if (ok) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (KVSPLIT) {
            mbar_arrive(bar_of(0));
            mbar_arrive(bar_of(1));
          } else {
            mbar_arrive(bar_of(t));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace attn
