// bwd_kernel.cuh -- exact flash-attention backward for sm_103a (TMA + tcgen05 + TMEM).
//
// P is recomputed from the forward's row log-sum-exp, never stored; dS = P o (dP - Delta)
// with Delta_i = dO_i . O_i is formed in fp32 (FlashAttention for Tesla P100
// page, "Documentation": dS is a cancellation, dV = P^T dO is not).  Gradients
// accumulate in fp32 ("What it supports": fp32 gradient accumulation).
//
// Three kernels per call:
//   bwd_preprocess  Delta_i = sum_d dO_id O_id and LSE2_i = LSE_i log2(e), written
//                   to row-padded buffers (rows past N: LSE2 = +inf so P = 0,
//                   Delta = 0); zeroes the fp32 dQ accumulator.  Memory-bound:
//                   16-byte loads, several rows per warp in flight.
//   bwd_kernel      one CTA per (batch, kv head, 128-key tile j).  It loops over
//                   the query heads of its group and over the query tiles i
//                   (i >= j when causal: tiles above the diagonal are skipped):
//                     S^T  = K_j Q_i^T            (tcgen05, TMEM, keys on lanes)
//                     dP^T = V_j dO_i^T           (tcgen05, TMEM)
//                     P^T  = 2^(S^T c - LSE2_i), dS^T = P^T o (dP^T - Delta_i)
//                     dV_j += P^T dO_i            (A = P^T from TMEM)
//                     dK_j += dS^T Q_i            (A = dS^T from TMEM)
//                     dQ_i  = dS K_j              (A = the dS^T tile in shared
//                                                  memory, read MN-major)
//                   dK/dV stay in TMEM across the whole group (no GQA reduction
//                   pass).  The tensor cores run, per query tile i,
//                     dP_i, dV_i, S_{i+1}, dK_i, dQ_i
//                   so that P_{i+1} is computed while dK_i, dQ_i and dP_{i+1}
//                   run, and dS_i while dV_i and S_{i+1} run.  dQ_i goes TMEM ->
//                   registers of a dedicated warpgroup (freeing the columns for
//                   dP_{i+1} at once) -> a two-slot shared staging ring -> TMA
//                   tensor reduce-add into the fp32 accumulator.
//   bwd_postprocess dQ = scale * dQacc -> bf16.
//
// Group split (p.gsplit > 1, chosen by the host when one CTA per (key tile,
// batch, kv head) would not fill the GPU): the query heads of a group are
// divided over gsplit CTAs; each adds its fp32 dK/dV partials into fp32
// accumulators by TMA reduce-add, and bwd_post_kv converts them to bf16.
//
// Warp roles of bwd_kernel (16 warps):
//   0-7   compute warps.  Warp w covers TMEM lanes 32*(w%4).. (32 keys) and
//         query half w/4: P for 64 queries of its key rows (kept in registers,
//         written to TMEM as bf16 for the dV MMA), then dS for the same
//         queries; at the end it writes dV (half 0) or dK (half 1).
//   8-11  dQ warpgroup (thread = query row): dQ_i out of TMEM, staged 32
//         columns (16 KB) at a time, reduce-adds issued by its first thread.
//   12    TMA producer: K_j, V_j once; Q_i with LSE2_i and Delta_i into a
//         2-stage ring; dO_i into a single buffer (reloaded once dV_i is done).
//   13    TMEM allocator and MMA issuer.
//   14-15 idle (they complete the fourth warpgroup for the register split).
// Registers: launched at 128 per thread; setmaxnreg moves them to the compute
// warps (144: P of 64 queries stays live across the dS step) and the dQ
// warpgroup (168: a whole fp32 dQ row), 8*144 + 4*168 + 4*56 = 16*128.
//
// TMEM columns: [0,128) S^T, with P^T (bf16) of queries 0-63 written over
// columns [0,32) and of queries 64-127 over [64,96) (each half stays inside the
// S^T columns its own warps read); [128,256) dP^T, with dS^T (bf16) written
// the same way over [128,160) and [192,224) for the dK MMA; [256,256+D) dV;
// [256+D,256+2D) dK; dQ_i at [256+2D,256+3D) when D=64, else over dP^T.
// dS^T read from TMEM spares shared-memory bandwidth: a 128 x 128 x 16 MMA
// with both operands in shared memory reads 8 KB in ~70 cycles, close to the
// 128 B/clk an SM's shared memory delivers, and the TMA loads, dS stores and
// dQ staging share it (measured: +1.3 % at D=128, nothing at D=64).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "ptx.cuh"
#include "kernels.h"

namespace attn {

constexpr unsigned kErrSmemAlign = 2u;  // device error bit: shared memory base misaligned

template <int V>
struct IntConst {
  static constexpr int value = V;
};

template <int D>
struct BwdCfg {
  static constexpr int kTile = 128 * D * 2;  // one 128-row bf16 tile
  static constexpr int kBox = 128 * 128;     // one 128-row box of 128-byte rows
  static constexpr int kBoxes = D / 64;      // bf16 boxes per tile
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kQ0 = 2 * kTile;        // Q stage s at kQ0 + s * kTile
  static constexpr int kdO = 4 * kTile;
  static constexpr int kdS = 5 * kTile;        // dS^T tile: 128 keys x 128 queries bf16
  static constexpr int kdQ = kdS + 2 * kBox;   // dQ staging: 2 slots of 128 rows x 32 fp32
  static constexpr int kVec = kdQ + 2 * kBox;  // stage s: LSE2[128] then Delta[128]
  static constexpr int kBar = kVec + 2 * 1024;
  static constexpr int kNumBars = 16;
  static constexpr int kSmemBytes = kBar + kNumBars * 8 + 16;
  static constexpr int kThreads = 512;
  static constexpr uint32_t kTmemCols = 512;
  // Register split (per thread): 8 compute warps, 4 dQ warps, 4 other warps.
  static constexpr int kRegCompute = 144, kRegDq = 168, kRegOther = 56;
  static_assert(8 * kRegCompute + 4 * kRegDq + 4 * kRegOther == 16 * launch_regs(kThreads),
                "the register split must add up to the launch allocation");
  // Group split: the fp32 dV / dK partials (D/32 boxes each) are staged over
  // the Q ring and over dO + dS, all free once the last MMA has completed.
  static_assert(2 * kTile >= (D / 32) * kBox, "dV partial staging");
  static_assert(kTile + 2 * kBox >= (D / 32) * kBox, "dK partial staging");
};

// DQ = false: dK and dV only (the deterministic backward computes dQ in bwd_dq_kernel).
// VARLEN: sequences packed token-major (BwdParams::cu_seqlens); the grid is
// that of a batch of max_seqlen-long sequences and CTAs whose key tile lies
// past their sequence's end leave at once.  The TMA maps are the packed
// (D, H, total) ones (box 64 x 1 head x 128 tokens; the fp32 dQ map 32 x 1 x
// 128), whose tiles land in shared memory exactly as dense ones.  Key rows
// past the sequence are masked like a ragged tail; query rows past it have
// LSE2 = +inf, so their P, dS and dQ rows are zero (their dQ reduce-adds add
// zeros to the next sequence's rows).  No group split.
template <int D, bool CAUSAL, bool F16, bool DQ = true, bool VARLEN = false>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
               const __grid_constant__ CUtensorMap tm_dv, const BwdParams p) {
  using Cfg = BwdCfg<D>;
  static_assert(!(VARLEN && !DQ), "the packed backward has no deterministic variant");

  // ---- work unit: (key tile j, batch, kv head).  Non-causal: the key tiles of
  // one head are consecutive, so the CTAs resident at one time share a few
  // heads' Q, dO and dQ accumulator in L2, and each starts its query loop at
  // tile j so that they add into different dQ tiles at any one time.  Causal:
  // heaviest key tiles (smallest j) first for load balance, in bands of units
  // when there are many (a working set of a few heads; see BwdParams::band).
  const int BHkv = p.B * p.Hkv;
  const int GS = VARLEN ? 1 : p.gsplit;  // CTAs per (key tile, batch, kv head)
  int j, unit;
  if (CAUSAL) {
    // Key tiles in p.jchunks ranges [c T / K, (c+1) T / K), heaviest range
    // first; inside a range, bands of p.band units; inside a band, key tile j
    // ascending (the heaviest CTAs of the band first).
    const int NU = BHkv * GS, T = p.num_kv_tiles, K = p.jchunks;
    int c = 0;
    while (c + 1 < K && (int)blockIdx.x >= ((c + 1) * T / K) * NU) ++c;
    const int ja = c * T / K, w = (c + 1) * T / K - ja;
    const int r = (int)blockIdx.x - ja * NU;
    const int per = p.band * w;
    const int band = r / per;
    const int u0 = band * p.band;
    const int ub = min(p.band, NU - u0);
    const int r2 = r - band * per;
    j = ja + r2 / ub;
    unit = u0 + r2 % ub;
  } else {
    j = (int)blockIdx.x % p.num_kv_tiles;
    unit = (int)blockIdx.x / p.num_kv_tiles;
  }
  const int bhkv = unit / GS;
  const int gi = unit % GS;  // which slice of the group's query heads
  const int b = bhkv / p.Hkv, hkv = bhkv % p.Hkv;
  int seq0 = 0, N = p.N;  // first token and length of this CTA's sequence
  if constexpr (VARLEN) {
    seq0 = p.cu_seqlens[b];
    N = p.cu_seqlens[b + 1] - seq0;
    if (seq0 < 0 || N < 0 || N > p.N || seq0 > p.total - N) {  // not a valid sequence
      if (threadIdx.x == 0) atomicOr(p.err, kErrSeqlen);
      return;
    }
    if (j * 128 >= N) return;  // past this sequence's end
  }
  const int T = VARLEN ? (N + 127) / 128 : p.num_kv_tiles;
  const int Gs = p.G / GS;  // query heads of this CTA
  const int i0 = CAUSAL ? j : 0;
  const int n_i = T - i0;
  const int n_it = Gs * n_i;
  auto q_head = [&](int it) {  // flat b*Hq + h
    return b * p.Hq + hkv * p.G + gi * Gs + it / n_i;
  };
  auto q_tile = [&](int it) {
    const int r = it % n_i;
    return CAUSAL ? i0 + r : (r + j) % T;
  };
  // TMA load of the 128 rows from `row` of one (batch, head): (column, row,
  // plane) of a dense (D, N, B*H) map, or (column, head, token) of a packed
  // (D, H, total) one.
  auto load_rows = [&](uint32_t dst, const CUtensorMap* tm, uint32_t bar, int col, int row,
                       int plane, int head) {
    if constexpr (VARLEN)
      tma_load_3d(dst, tm, bar, col, head, seq0 + row);
    else
      tma_load_3d(dst, tm, bar, col, row, plane);
  };
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  // The 128-byte swizzle atoms need a 1024-byte aligned base; there is no room
  // for padding at D=128, so refuse (and report) instead of computing garbage.
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemAlign);
    return;
  }
  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = (int)(threadIdx.x & 31);

  const uint32_t bar0 = sbase + Cfg::kBar;
  const uint32_t bar_kv = bar0;
  auto bar_q_full = [&](int s) { return bar0 + 8u * (1 + s); };  // Q, LSE2, Delta of stage s
  auto bar_q_free = [&](int s) { return bar0 + 8u * (3 + s); };  // dK MMA done with stage s
  const uint32_t bar_do_full = bar0 + 8u * 5;
  const uint32_t bar_do_free = bar0 + 8u * 6;   // dV MMA done with dO
  const uint32_t bar_s = bar0 + 8u * 7;         // S^T complete
  const uint32_t bar_p = bar0 + 8u * 8;         // P^T in TMEM (8 compute warps)
  const uint32_t bar_dp = bar0 + 8u * 9;        // dP^T complete
  const uint32_t bar_ds = bar0 + 8u * 10;       // dS^T in shared memory (8 compute warps)
  const uint32_t bar_dq = bar0 + 8u * 11;       // dQ complete in TMEM
  const uint32_t bar_dq_free = bar0 + 8u * 12;  // dQ read out of TMEM (4 dQ warps)
  const uint32_t bar_done = bar0 + 8u * 13;     // every MMA complete
  auto bar_epi = [&](int h) { return bar0 + 8u * (14 + h); };  // group split: partial staged
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kBar + Cfg::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_q_full(s), 1);
      mbar_init(bar_q_free(s), 1);
      mbar_init(bar_epi(s), 4);
    }
    mbar_init(bar_do_full, 1);
    mbar_init(bar_do_free, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_p, 8);
    mbar_init(bar_dp, 1);
    mbar_init(bar_ds, 8);
    mbar_init(bar_dq, 1);
    mbar_init(bar_dq_free, 4);
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 13) tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
  if (warp == 12 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    if (DQ) tma_prefetch_desc(&tm_dq);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const WaitCtl wc{p.timeout_ns, p.err, abort_flag};
  // At D=64 dQ has columns of its own, so dP_{it+1} need not wait for dQ_it to
  // be read out; at D=128 the 512 columns are full and dQ reuses dP's.
  constexpr bool kOwnDq = 256 + 3 * D <= (int)Cfg::kTmemCols;
  const uint32_t tS = tmem_base, tdP = tmem_base + 128, tdV = tmem_base + 256,
                 tdK = tmem_base + 256 + D, tdQ = kOwnDq ? tmem_base + 256 + 2 * D : tdP;

  if (warp >= 12) {
    regs_decrease<Cfg::kRegOther>();
    if (warp == 12 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      mbar_arrive_expect_tx(bar_kv, 2 * Cfg::kTile);
      for (int c = 0; c < Cfg::kBoxes; ++c) {
        load_rows(sbase + Cfg::kK + c * Cfg::kBox, &tm_k, bar_kv, c * 64, j * 128, bhkv, hkv);
        load_rows(sbase + Cfg::kV + c * Cfg::kBox, &tm_v, bar_kv, c * 64, j * 128, bhkv, hkv);
      }
      auto load_q = [&](int it) {  // Q_i, LSE2_i, Delta_i into stage it&1
        const int s = it & 1;
        const int bhq = q_head(it), i = q_tile(it);
        const uint32_t qs = sbase + Cfg::kQ0 + s * Cfg::kTile;
        mbar_arrive_expect_tx(bar_q_full(s), Cfg::kTile + 1024);
        for (int c = 0; c < Cfg::kBoxes; ++c)
          load_rows(qs + c * Cfg::kBox, &tm_q, bar_q_full(s), c * 64, i * 128, bhq, bhq - b * p.Hq);
        const size_t voff = (size_t)bhq * p.Npad + (size_t)i * 128;
        bulk_load(sbase + Cfg::kVec + s * 1024, p.lse2 + voff, 512, bar_q_full(s));
        bulk_load(sbase + Cfg::kVec + s * 1024 + 512, p.delta + voff, 512, bar_q_full(s));
      };
      auto load_do = [&](int it) {
        mbar_arrive_expect_tx(bar_do_full, Cfg::kTile);
        const int bhq = q_head(it);
        for (int c = 0; c < Cfg::kBoxes; ++c)
          load_rows(sbase + Cfg::kdO + c * Cfg::kBox, &tm_do, bar_do_full, c * 64,
                    q_tile(it) * 128, bhq, bhq - b * p.Hq);
      };
      load_q(0);
      load_do(0);
      if (n_it > 1) load_q(1);
      int nq = n_it > 1 ? 2 : 1, ndo = 1;  // loads issued
      bool ok = true;
      for (int it = 0; it < n_it && ok; ++it) {
        if (it + 1 < n_it) {
          if (!(ok = mbar_wait_tested_inl(bar_do_free, (uint32_t)it & 1u, wc))) break;
          load_do(it + 1);
          ++ndo;
        }
        if (it + 2 < n_it) {
          if (!(ok = mbar_wait_tested_inl(bar_q_free(it & 1), (uint32_t)(it >> 1) & 1u, wc))) break;
          load_q(it + 2);
          ++nq;
        }
      }
      if (!ok) {
        // Let every load already issued land before the CTA can exit.
        for (int f = (nq > 2 ? nq - 2 : 0); f < nq; ++f)
          mbar_wait_drain_inl(bar_q_full(f & 1), (uint32_t)(f >> 1) & 1u, wc);
        mbar_wait_drain_inl(bar_do_full, (uint32_t)(ndo - 1) & 1u, wc);
        mbar_wait_drain_inl(bar_kv, 0, wc);
      }
    } else if (warp == 13 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdescSS = make_idesc_bf16(128, 128, 0, 0, F16);
      constexpr uint32_t kIdescB_MN = make_idesc_bf16(128, D, 1, 0, F16);  // dV, dK
      constexpr uint32_t kIdescDQ = make_idesc_bf16(128, D, 1, 1, F16);    // dQ: A, B MN-major
      constexpr uint32_t kHi = sdesc_sw128_hi(1024);  // 8-row groups 1024 bytes apart
      // Address words of every operand, K-major (K advances inside a 128-byte
      // row, then by a 64-column box) or MN-major (K advances by 16 rows; the
      // 64-element MN chunks are one box apart).
      const uint32_t kK = sdesc_sw128_lo(sbase + Cfg::kK, 16);
      const uint32_t kV = sdesc_sw128_lo(sbase + Cfg::kV, 16);
      const uint32_t kdO = sdesc_sw128_lo(sbase + Cfg::kdO, 16);
      const uint32_t kdS = sdesc_sw128_lo(sbase + Cfg::kdS, 16);
      const uint32_t mdO = sdesc_sw128_lo(sbase + Cfg::kdO, Cfg::kBox);
      const uint32_t mdS = sdesc_sw128_lo(sbase + Cfg::kdS, Cfg::kBox);
      const uint32_t mK = sdesc_sw128_lo(sbase + Cfg::kK, Cfg::kBox);
      const uint32_t kQ0 = sdesc_sw128_lo(sbase + Cfg::kQ0, 16);
      const uint32_t mQ0 = sdesc_sw128_lo(sbase + Cfg::kQ0, Cfg::kBox);
      constexpr uint32_t kQs = Cfg::kTile >> 4;  // stage stride in address units
      // K-step kk of a K-major operand: (kk/4) boxes + (kk%4) 32-byte steps;
      // of an MN-major operand: kk * 16 rows of 128 bytes.
      auto koff = [](int kk) { return (uint32_t)(((kk / 4) * Cfg::kBox + (kk % 4) * 32) >> 4); };
      auto moff = [](int kk) { return (uint32_t)((kk * 2048) >> 4); };
      // X^T = A B^T with A a [128 x D] K-major tile (K or V), B a [128 x D] K-major tile.
      auto issue_t = [&](uint32_t dst, uint32_t a, uint32_t bb) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_w(dst, a, koff(kk), bb, koff(kk), kHi, kIdescSS, kk > 0);
      };
      // One query tile: dP_it, dV_it, S_{it+1}, dK_it, dQ_it.  The stage s = it & 1
      // is a compile-time constant, so every descriptor is a register plus an
      // immediate.
      auto step = [&](int it, auto stage) -> bool {
        constexpr int s = decltype(stage)::value;
        const uint32_t mQs_ = mQ0 + s * kQs, kQn = kQ0 + (s ^ 1) * kQs;
        // dP_it over the dP^T columns, once dQ_{it-1} has been read out of them.
        if (!mbar_wait_tested_inl(bar_do_full, (uint32_t)it & 1u, wc)) return false;
        if (DQ && !kOwnDq && it > 0 &&
            !mbar_wait_tested_inl(bar_dq_free, (uint32_t)(it - 1) & 1u, wc))
          return false;
        tc_fence_after();
        issue_t(tdP, kV, kdO);
        mma_commit(bar_dp);
        // dV += P^T dO  (K = 128 queries; A = P^T from TMEM)
        if (!mbar_wait_tested_inl(bar_p, (uint32_t)it & 1u, wc)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_w(tdV, tS + (kk / 4) * 64 + (kk % 4) * 8, mdO, moff(kk), kHi, kIdescB_MN,
                   (it > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar_do_free);
        // S_{it+1} over the S^T columns (P^T_it has been consumed by dV, in order).
        if (it + 1 < n_it) {
          if (!mbar_wait_tested_inl(bar_q_full(s ^ 1), (uint32_t)((it + 1) >> 1) & 1u, wc)) return false;
          tc_fence_after();
          issue_t(tS, kK, kQn);
          mma_commit(bar_s);
        }
        if (!mbar_wait_tested_inl(bar_ds, (uint32_t)it & 1u, wc)) return false;
        tc_fence_after();
        // dK += dS^T Q first: it frees Q stage s for the producer one MMA group
        // earlier.  A = dS^T (bf16) from TMEM, where the compute warps wrote it
        // over the dP^T columns they had read (dQ_it and dP_{it+1}, the next
        // writers of those columns, are issued after this).
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_w(tdK, tdP + (kk / 4) * 64 + (kk % 4) * 8, mQs_, moff(kk), kHi, kIdescB_MN,
                   (it > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar_q_free(s));
        if (DQ) {
          if (kOwnDq && it > 0 &&
              !mbar_wait_tested_inl(bar_dq_free, (uint32_t)(it - 1) & 1u, wc))
            return false;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dQ = dS K  (K = 128 keys)
            mma_ss_w(tdQ, mdS, moff(kk), mK, moff(kk), kHi, kIdescDQ, kk > 0);
          mma_commit(bar_dq);
        }
        return true;
      };
      bool ok = mbar_wait_tested_inl(bar_kv, 0, wc) && mbar_wait_tested_inl(bar_q_full(0), 0, wc);
      if (ok) {
        tc_fence_after();
        issue_t(tS, kK, kQ0);
        mma_commit(bar_s);
      }
      for (int it = 0; it < n_it && ok; it += 2) {
        ok = step(it, IntConst<0>{});
        if (ok && it + 1 < n_it) ok = step(it + 1, IntConst<1>{});
      }
      mma_commit(bar_done);
      if (!ok) mbar_wait_drain_inl(bar_done, 0, wc);
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ warpgroup
    regs_increase<Cfg::kRegDq>();
    const int wq = warp & 3;
    const int qrow = wq * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const bool leader = warp == 8 && lane == 0;
    const uint32_t swz = (uint32_t)(qrow & 7);
    const uint32_t st_row = sbase + Cfg::kdQ + (uint32_t)qrow * 128u;
    int chunk = 0;
    bool ok = true;
    for (int it = 0; it < (DQ ? n_it : 0); ++it) {
      // One decision for the whole warpgroup: its named barriers need all 4 warps.
      ok = named_bar_and(1, 128, mbar_wait_tested_inl(bar_dq, (uint32_t)it & 1u, wc));
      if (!ok) break;
      tc_fence_after();
      uint32_t r[D / 32][32];
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(tdQ + lane_off + cc * 32, r[cc]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dq_free);
      const int qt = q_tile(it), qh = q_head(it);
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc, ++chunk) {
        const uint32_t slot = (uint32_t)(chunk & 1) * Cfg::kBox;
        // The slot's previous reduce-add (two chunks ago) must have read it.
        if (leader) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        named_bar_sync(1, 128);
        // 128-byte rows, 16-byte chunks swizzled by row & 7 (the map's 128B swizzle).
#pragma unroll
        for (int v = 0; v < 8; ++v)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                           st_row + slot + ((((uint32_t)v) ^ swz) << 4)),
                       "r"(r[cc][4 * v]), "r"(r[cc][4 * v + 1]), "r"(r[cc][4 * v + 2]),
                       "r"(r[cc][4 * v + 3])
                       : "memory");
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader) {
          if constexpr (VARLEN)
            tma_reduce_add_3d(&tm_dq, sbase + Cfg::kdQ + slot, cc * 32, qh - b * p.Hq,
                              seq0 + qt * 128);
          else
            tma_reduce_add_3d(&tm_dq, sbase + Cfg::kdQ + slot, cc * 32, qt * 128, qh);
          bulk_commit();
        }
      }
    }
    if (ok && GS > 1) {
      // Group split: add the fp32 dV / dK partials the compute warps stage.
      ok = named_bar_and(1, 128, mbar_wait_tested_inl(bar_epi(0), 0, wc) &&
                                     mbar_wait_tested_inl(bar_epi(1), 0, wc));
      if (ok && leader) {
        for (int c = 0; c < D / 32; ++c) {
          tma_reduce_add_3d(&tm_dv, sbase + Cfg::kQ0 + c * Cfg::kBox, c * 32, j * 128, bhkv);
          tma_reduce_add_3d(&tm_dk, sbase + Cfg::kdO + c * Cfg::kBox, c * 32, j * 128, bhkv);
        }
        bulk_commit();
      }
    }
    if (leader) bulk_wait_all();
  } else {
    // ------------------------------------------------------------ compute warps 0-7
    regs_increase<Cfg::kRegCompute>();
    const int wq = warp & 3;   // TMEM lane quadrant
    const int ch = warp >> 2;  // query half
    const int row = wq * 32 + lane;  // key row
    const int kj = j * 128 + row;
    const bool key_live = kj < N;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float C = p.scale_log2;
    const float2 c2 = make_float2(C, C);
    const uint32_t swz = (uint32_t)(row & 7);
    const uint32_t ds_row = sbase + Cfg::kdS + (uint32_t)ch * Cfg::kBox + (uint32_t)row * 128u;
    const uint32_t ts = tS + lane_off + (uint32_t)ch * 64u;
    const uint32_t tp = tdP + lane_off + (uint32_t)ch * 64u;
    bool ok = true;
    for (int it = 0; it < n_it && ok; ++it) {
      const int s = it & 1;
      // ---- P = 2^(S c - LSE2) for queries [64ch, 64ch + 64) of this key row
      ok = __all_sync(0xffffffffu, mbar_wait_tested_inl(bar_s, (uint32_t)it & 1u, wc) &&
                                       mbar_wait_tested_inl(bar_q_full(s), (uint32_t)(it >> 1) & 1u, wc));
      if (!ok) break;
      tc_fence_after();
      const float* lse2 = reinterpret_cast<const float*>(smem + Cfg::kVec + s * 1024) + ch * 64;
      const float* delta = lse2 + 128;
      const bool diag = CAUSAL && q_tile(it) == j;
      float pf[64];
      // The masks (causal: query < key on the diagonal tile; ragged: key rows
      // past N) apply to few tiles; the others take a copy of the loop without
      // them (a warp-uniform choice), which saves issue slots on every pair.
      auto p_phase = [&](auto masked) {
        constexpr bool kMasked = decltype(masked)::value != 0;
        uint32_t sr[2][16];
        tmem_ld16(ts, sr[0]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // 16 query columns per chunk, the next one in flight
          const int bb = c & 1;
          tmem_ld_wait();
          if (c + 1 < 4) tmem_ld16(ts + (c + 1) * 16, sr[bb ^ 1]);
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            const int qc = c * 16 + e;  // query within this half
            const float4 l4 = *reinterpret_cast<const float4*>(lse2 + qc);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int ee = e + 2 * h;
              const float2 nl = h ? make_float2(-l4.z, -l4.w) : make_float2(-l4.x, -l4.y);
              const float2 x = __ffma2_rn(
                  make_float2(__uint_as_float(sr[bb][ee]), __uint_as_float(sr[bb][ee + 1])), c2,
                  nl);
              float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              if constexpr (kMasked) {
                if (diag) {  // causal: query < key is masked
                  const int q = ch * 64 + qc + 2 * h;
                  if (q < row) pp.x = 0.f;
                  if (q + 1 < row) pp.y = 0.f;
                }
                if (!key_live) pp = make_float2(0.f, 0.f);
              }
              pf[c * 16 + ee] = pp.x;
              pf[c * 16 + ee + 1] = pp.y;
              pk[ee / 2] = pack2<F16>(pp.x, pp.y);
            }
          }
          // P^T (bf16) over S^T columns this warp has already read.
          tmem_st8(ts + c * 8, pk);
        }
      };
      if (__any_sync(0xffffffffu, diag || !key_live))
        p_phase(IntConst<1>{});
      else
        p_phase(IntConst<0>{});
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p);

      // ---- dS = P o (dP - Delta) for the same queries, to shared memory
      ok = __all_sync(0xffffffffu, mbar_wait_tested_inl(bar_dp, (uint32_t)it & 1u, wc));
      if (!ok) break;
      tc_fence_after();
      {
        // dP in two 32-column halves (fewer live registers next to the 64 P
        // values; the dS^T written below only covers columns of the first half).
        uint32_t dr[32];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
        tmem_ld32(tp + hf * 32, dr);
        tmem_ld_wait();
        auto dpv = [&](int q) { return __uint_as_float(dr[q - 32 * hf]); };
#pragma unroll
        for (int c = 2 * hf; c < 2 * hf + 2; ++c) {
          uint32_t dk[8];
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            const int qc = c * 16 + e;
            const float4 d4 = *reinterpret_cast<const float4*>(delta + qc);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int ee = e + 2 * h;
              const float2 nd = h ? make_float2(-d4.z, -d4.w) : make_float2(-d4.x, -d4.y);
              const float2 dd =
                  __fadd2_rn(make_float2(dpv(c * 16 + ee), dpv(c * 16 + ee + 1)), nd);
              const float2 ds = __fmul2_rn(make_float2(pf[c * 16 + ee], pf[c * 16 + ee + 1]), dd);
              dk[ee / 2] = pack2<F16>(ds.x, ds.y);
            }
          }
          // dS^T over the dP^T columns just read (A of the dK MMA) and, for the
          // dQ MMA, to shared memory (box ch) in the 128-byte swizzled layout.
          tmem_st8(tp + c * 8, dk);
#pragma unroll
          for (int v = 0; v < (DQ ? 2 : 0); ++v) {
            const uint32_t chunk = ((uint32_t)(c * 2 + v)) ^ swz;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(ds_row + chunk * 16),
                         "r"(dk[4 * v]), "r"(dk[4 * v + 1]), "r"(dk[4 * v + 2]), "r"(dk[4 * v + 3])
                         : "memory");
          }
        }
        }
      }
      tmem_st_wait();
      if constexpr (DQ) fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait_tested_inl(bar_done, 0, wc));
    if (ok && GS > 1) {
      // Group split: stage this row's fp32 dV (half 0) or unscaled dK (half 1)
      // partial for the dQ warpgroup's reduce-add.
      tc_fence_after();
      const uint32_t src = (ch ? tdK : tdV) + lane_off;
      const uint32_t stage = sbase + (ch ? Cfg::kdO : Cfg::kQ0) + (uint32_t)row * 128u;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(src + c * 32, rr);
        tmem_ld_wait();
#pragma unroll
        for (int v = 0; v < 8; ++v)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                           stage + c * Cfg::kBox + ((((uint32_t)v) ^ swz) << 4)),
                       "r"(rr[4 * v]), "r"(rr[4 * v + 1]), "r"(rr[4 * v + 2]), "r"(rr[4 * v + 3])
                       : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_epi(ch));
    } else if (ok) {
      // Epilogue: half 0 writes dV, half 1 writes dK (scaled) of this key row.
      tc_fence_after();
      const size_t krow = key_live ? (size_t)kj : 0;
      const size_t orow = (VARLEN ? ((size_t)seq0 + krow) * p.Hkv + hkv
                                  : (size_t)bhkv * p.N + krow) * D;
      uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(ch ? p.dk : p.dv) + orow);
      const float mul = ch ? p.scale : 1.f;
      const uint32_t src = (ch ? tdK : tdV) + lane_off;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(src + c * 32, rr);
        tmem_ld_wait();
        if (key_live) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack2<F16>(__uint_as_float(rr[8 * v + 0]) * mul, __uint_as_float(rr[8 * v + 1]) * mul);
            w.y = pack2<F16>(__uint_as_float(rr[8 * v + 2]) * mul, __uint_as_float(rr[8 * v + 3]) * mul);
            w.z = pack2<F16>(__uint_as_float(rr[8 * v + 4]) * mul, __uint_as_float(rr[8 * v + 5]) * mul);
            w.w = pack2<F16>(__uint_as_float(rr[8 * v + 6]) * mul, __uint_as_float(rr[8 * v + 7]) * mul);
            out[c * 4 + v] = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// Rows of the preprocessing kernel per CTA: D/8 lanes per padded row (16
// bytes of O and of dO each), 32*8/D rows per warp and pass, kPrePasses
// passes with all loads issued before the first reduction (several KB in
// flight per warp: one 128-byte row per warp left the kernel latency-bound
// at a third of the copy bandwidth).
constexpr int kPrePasses = 4;
template <int D>
constexpr int pre_rows_per_cta() { return 8 * (32 * 8 / D) * kPrePasses; }

// dO . O of one row from its D/8 lanes (8 elements each, lane l the elements
// [8l, 8l+8)), summed over those lanes; both preprocessing kernels use it, so
// a packed batch of equal lengths gets the dense batch's Delta bit for bit.
template <int D, bool F16>
__device__ __forceinline__ float pre_row_dot(const uint4& a, const uint4& g) {
  auto dot2 = [](uint32_t u, uint32_t v) {
    const float2 x = unpack2<F16>(u), y = unpack2<F16>(v);
    return x.x * y.x + x.y * y.y;
  };
  float acc = dot2(a.x, g.x) + dot2(a.y, g.y) + dot2(a.z, g.z) + dot2(a.w, g.w);
#pragma unroll
  for (int off = D / 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  return acc;
}

// Delta and LSE2 into row-padded buffers; zero the dQ accumulator (and, with
// the group split, the dK/dV accumulators).  Padded row r = (b*Hq + h, i),
// i < Npad; rows past N get LSE2 = +inf, Delta = 0.
template <int D, bool F16>
__global__ void __launch_bounds__(256)
    bwd_preprocess(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                   const float* __restrict__ lse, float* __restrict__ lse2,
                   float* __restrict__ delta, float* __restrict__ dq_acc, long long rows, int N,
                   int Npad, float* __restrict__ dk_acc, float* __restrict__ dv_acc,
                   long long kv_rows) {
  constexpr int L = D / 8;       // lanes per row
  constexpr int RPW = 32 / L;    // rows per warp and pass
  static_assert(128 % (RPW * kPrePasses) == 0, "a warp's rows lie in one (batch, head)");
  const int lane = threadIdx.x & 31;
  const int sub = lane / L, l = lane % L;
  // The warp's rows: RPW * kPrePasses consecutive padded rows of one (batch,
  // head) plane (Npad is a multiple of 128).
  const long long rw = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * (RPW * kPrePasses);
  const long long bh = rw / Npad;
  const int iw = (int)(rw - bh * Npad);
  uint4 a[kPrePasses], g[kPrePasses];
#pragma unroll
  for (int ps = 0; ps < kPrePasses; ++ps) {
    const int i = iw + ps * RPW + sub;
    a[ps] = make_uint4(0u, 0u, 0u, 0u);
    g[ps] = make_uint4(0u, 0u, 0u, 0u);
    if (rw < rows && i < N) {
      const size_t base = ((size_t)bh * N + i) * D + (size_t)l * 8;
      a[ps] = *reinterpret_cast<const uint4*>(o + base);
      g[ps] = *reinterpret_cast<const uint4*>(dout + base);
    }
  }
#pragma unroll
  for (int ps = 0; ps < kPrePasses; ++ps) {
    const float acc = pre_row_dot<D, F16>(a[ps], g[ps]);
    if (rw >= rows) continue;
    const int i = iw + ps * RPW + sub;
    const long long r = rw + ps * RPW + sub;
    if (l == 0) {
      lse2[r] = i < N ? lse[(size_t)bh * N + i] * 1.4426950408889634f : INFINITY;
      delta[r] = acc;
    }
    // D fp32 per accumulator row: two 16-byte stores per lane
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    if (dq_acc != nullptr) {  // none in the deterministic backward
      float4* zq = reinterpret_cast<float4*>(dq_acc + (size_t)r * D) + 2 * l;
      zq[0] = z;
      zq[1] = z;
    }
    if (r < kv_rows) {  // group split: zero the dK/dV accumulators too
      float4* zk = reinterpret_cast<float4*>(dk_acc + (size_t)r * D) + 2 * l;
      float4* zv = reinterpret_cast<float4*>(dv_acc + (size_t)r * D) + 2 * l;
      zk[0] = z;
      zk[1] = z;
      zv[0] = z;
      zv[1] = z;
    }
  }
}

// Packed variable-length batches: Delta and LSE2 of padded row (b*Hq + h, i),
// i < Npad, from token cu_seqlens[b] + i of o/dout [total, Hq, D] and lse
// [Hq, total]; rows past the sequence's end (or of a sequence whose offsets
// are not valid, which the main kernel reports) get LSE2 = +inf, Delta = 0.
// The lane and row layout of bwd_preprocess.
template <int D, bool F16>
__global__ void __launch_bounds__(256)
    bwd_preprocess_varlen(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                          const float* __restrict__ lse, const int* __restrict__ cu_seqlens,
                          float* __restrict__ lse2, float* __restrict__ delta, long long rows,
                          int Hq, int Npad, int max_seqlen, int total) {
  constexpr int L = D / 8;       // lanes per row
  constexpr int RPW = 32 / L;    // rows per warp and pass
  const int lane = threadIdx.x & 31;
  const int sub = lane / L, l = lane % L;
  const long long rw = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * (RPW * kPrePasses);
  if (rw >= rows) return;
  const long long bh = rw / Npad;  // the warp's rows share one (sequence, head)
  const int iw = (int)(rw - bh * Npad);
  const int b = (int)(bh / Hq), h = (int)(bh % Hq);
  const int seq0 = cu_seqlens[b];
  const int len = cu_seqlens[b + 1] - seq0;
  const bool valid = seq0 >= 0 && len >= 0 && len <= max_seqlen && seq0 <= total - len;
  uint4 a[kPrePasses], g[kPrePasses];
#pragma unroll
  for (int ps = 0; ps < kPrePasses; ++ps) {
    const int i = iw + ps * RPW + sub;
    a[ps] = make_uint4(0u, 0u, 0u, 0u);
    g[ps] = make_uint4(0u, 0u, 0u, 0u);
    if (valid && i < len) {
      const size_t base = ((size_t)(seq0 + i) * Hq + h) * D + (size_t)l * 8;
      a[ps] = *reinterpret_cast<const uint4*>(o + base);
      g[ps] = *reinterpret_cast<const uint4*>(dout + base);
    }
  }
#pragma unroll
  for (int ps = 0; ps < kPrePasses; ++ps) {
    const float acc = pre_row_dot<D, F16>(a[ps], g[ps]);
    const int i = iw + ps * RPW + sub;
    const bool live = valid && i < len;
    if (l == 0) {
      const long long r = rw + ps * RPW + sub;
      lse2[r] = live ? lse[(size_t)h * total + seq0 + i] * 1.4426950408889634f : INFINITY;
      delta[r] = live ? acc : 0.f;
    }
  }
}

// dQ = scale * dQacc (rows < N) -> bf16.  8 elements per thread.
template <int D, bool F16>
__global__ void __launch_bounds__(256)
    bwd_postprocess(const float* __restrict__ dq_acc, uint16_t* __restrict__ dq,
                    long long rows, int N, int Npad, float scale) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // 8-element group
  constexpr int kGroups = D / 8;
  const long long r = idx / kGroups;  // output row (b*Hq + h)*N + i
  if (r >= rows) return;
  const int g = (int)(idx % kGroups);
  const long long bh = r / N;
  const int i = (int)(r % N);
  const float4* src = reinterpret_cast<const float4*>(dq_acc + ((size_t)bh * Npad + i) * D + g * 8);
  const float4 a = src[0], c = src[1];
  uint4 w;
  w.x = pack2<F16>(a.x * scale, a.y * scale);
  w.y = pack2<F16>(a.z * scale, a.w * scale);
  w.z = pack2<F16>(c.x * scale, c.y * scale);
  w.w = pack2<F16>(c.z * scale, c.w * scale);
  reinterpret_cast<uint4*>(dq + (size_t)r * D)[g] = w;
}

// Group split: dK = scale * dKacc, dV = dVacc (rows < N) -> bf16.  8 elements
// per thread; rows are (b*Hkv + h)*N + i.
template <int D, bool F16>
__global__ void __launch_bounds__(256)
    bwd_post_kv(const float* __restrict__ dk_acc, const float* __restrict__ dv_acc,
                uint16_t* __restrict__ dk, uint16_t* __restrict__ dv, long long rows,
                int N, int Npad, float scale) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  constexpr int kGroups = D / 8;
  const long long r = idx / kGroups;
  if (r >= rows) return;
  const int g = (int)(idx % kGroups);
  const long long bh = r / N;
  const int i = (int)(r % N);
  const size_t off = ((size_t)bh * Npad + i) * D + g * 8;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const float4* src = reinterpret_cast<const float4*>((which ? dk_acc : dv_acc) + off);
    const float m = which ? scale : 1.f;
    const float4 a = src[0], c = src[1];
    uint4 w;
    w.x = pack2<F16>(a.x * m, a.y * m);
    w.y = pack2<F16>(a.z * m, a.w * m);
    w.z = pack2<F16>(c.x * m, c.y * m);
    w.w = pack2<F16>(c.z * m, c.w * m);
    reinterpret_cast<uint4*>((which ? dk : dv) + (size_t)r * D)[g] = w;
  }
}

}  // namespace attn
