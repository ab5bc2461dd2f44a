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
//                   Delta = 0); zeroes the fp32 dQ accumulator.
//   bwd_kernel      one CTA per (batch, kv head, 128-key tile j).  It loops over
//                   the query heads of its group and over the query tiles i
//                   (i >= j when causal: tiles above the diagonal are skipped):
//                     S^T  = K_j Q_i^T            (tcgen05, TMEM, keys on lanes)
//                     dP^T = V_j dO_i^T           (tcgen05, TMEM)
//                     P^T  = 2^(S^T c - LSE2_i), dS^T = P^T o (dP^T - Delta_i)
//                     dV_j += P^T dO_i            (A = P^T from TMEM)
//                     dK_j += dS^T Q_i            (A = dS^T from shared memory)
//                     dQ_i  = dS K_j              (A = the same dS^T tile read MN-major)
//                   dK/dV stay in TMEM across the whole group (no GQA reduction
//                   pass).  dQ_i goes TMEM -> registers -> the Q_i/dO_i ring
//                   stage (dead once the dQ MMA has finished) -> TMA tensor
//                   reduce-add into the fp32 accumulator, issued by the producer
//                   thread, which reloads the stage as soon as the reduce-add has
//                   read it.
//   bwd_postprocess dQ = scale * dQacc -> bf16.
//
// Group split (p.gsplit > 1, chosen by the host when one CTA per (key tile,
// batch, kv head) would not fill the GPU): the query heads of a group are
// divided over gsplit CTAs; each adds its fp32 dK/dV partials into fp32
// accumulators by TMA reduce-add, and bwd_post_kv converts them to bf16.
//
// Warp roles of bwd_kernel (10 warps):
//   0-7  compute warps.  Warp w covers TMEM lanes 32*(w%4).. and column half
//        w/4: it computes dS for 64 of the 128 queries of its 32 key rows, then
//        stages half of the dQ columns of its 32 query rows, and at the end
//        writes dV (half 0) or dK (half 1) of its key rows.
//   8    TMA producer (K_j, V_j once; Q_i, dO_i, LSE2, Delta per iteration into a
//        2-stage ring) and issuer of the dQ reduce-adds.  Q and dO of a stage
//        have separate barriers: the dQ half staged in the Q area is added
//        first, so Q of step it+2 starts loading (D=128) while the dO-area
//        half is still being read.
//   9    TMEM allocator and MMA issuer.
//
// TMEM columns: [0,128) S^T, with P^T (bf16) of queries 0-63 written over
// columns [0,32) and of queries 64-127 over [64,96) (each half stays inside the
// S^T columns its own warps read); [128,256) dP^T, later overwritten by dQ_i;
// [256,256+D) dV; [256+D,256+2D) dK.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "ptx.cuh"
#include "kernels.h"

namespace attn {

constexpr unsigned kErrSmemAlign = 2u;  // device error bit: shared memory base misaligned

template <int D>
struct BwdCfg {
  static constexpr int kTile = 128 * D * 2;  // one 128-row bf16 tile
  static constexpr int kBox = 128 * 128;     // one 64-column box (128-byte rows)
  static constexpr int kBoxes = D / 64;
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kQ0 = 2 * kTile;      // stage s: Q at kQ0 + s*2*kTile, dO right after
  static constexpr int kdS = 6 * kTile;      // dS^T tile: 128 keys x 128 queries bf16
  static constexpr int kVec = kdS + 2 * kBox;  // stage s: LSE2[128] then Delta[128]
  static constexpr int kBar = kVec + 2 * 1024;
  // kv_full, qd_full[2] (dO, LSE2, Delta), staged[2], s_ready, ds_ready, dq_ready,
  // dq_free, all_done, red_go, prod_done, epi_staged[2] (group split only), q_full[2]
  static constexpr int kNumBars = 16;
  static constexpr int kSmemBytes = kBar + kNumBars * 8 + 16;
  static constexpr int kThreads = 320;
  static constexpr uint32_t kTmemCols = 512;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(320, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
               const __grid_constant__ CUtensorMap tm_dv, const BwdParams p) {
  using Cfg = BwdCfg<D>;
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
  auto bar_qd_full = [&](int s) { return bar0 + 8u * (1 + s); };   // dO_i, LSE2, Delta landed
  auto bar_q_full = [&](int s) { return bar0 + 8u * (14 + s); };   // Q_i landed
  auto bar_staged = [&](int h) { return bar0 + 8u * (3 + h); };  // dQ column half h staged
  const uint32_t bar_s = bar0 + 8u * 5;
  const uint32_t bar_ds = bar0 + 8u * 6;
  const uint32_t bar_dq = bar0 + 8u * 7;
  const uint32_t bar_dq_free = bar0 + 8u * 8;
  const uint32_t bar_done = bar0 + 8u * 9;
  // The producer has taken step it's staged dQ: the compute warps may signal
  // the next step's staging (keeps staged[] from running a phase ahead).
  const uint32_t bar_red_go = bar0 + 8u * 10;
  // Group split only: the producer has finished with every ring stage, and the
  // compute warps have staged their dV (half 0) / dK (half 1) partials.
  const uint32_t bar_prod_done = bar0 + 8u * 11;
  auto bar_epi = [&](int h) { return bar0 + 8u * (12 + h); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kBar + Cfg::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_qd_full(s), 1);
      mbar_init(bar_q_full(s), 1);
      mbar_init(bar_staged(s), 4);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_ds, 8);
    mbar_init(bar_dq, 1);
    mbar_init(bar_dq_free, 8);
    mbar_init(bar_done, 1);
    mbar_init(bar_red_go, 1);
    mbar_init(bar_prod_done, 1);
    mbar_init(bar_epi(0), 4);
    mbar_init(bar_epi(1), 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dq);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // ---- work unit: (key tile j, batch, kv head).  Non-causal: the key tiles of
  // one head are consecutive, so the CTAs resident at one time share a few
  // heads' Q, dO and dQ accumulator in L2.  Causal: the heaviest key tiles
  // (smallest j) of all heads go first, for load balance.
  const int T = p.num_kv_tiles;
  const int BHkv = p.B * p.Hkv;
  const int GS = p.gsplit;  // CTAs per (key tile, batch, kv head)
  const int j = CAUSAL ? (int)blockIdx.x / (BHkv * GS) : (int)blockIdx.x % T;
  const int unit = CAUSAL ? (int)blockIdx.x % (BHkv * GS) : (int)blockIdx.x / T;
  const int bhkv = unit / GS;
  const int gi = unit % GS;  // which slice of the group's query heads
  const int b = bhkv / p.Hkv, hkv = bhkv % p.Hkv;
  const int Gs = p.G / GS;  // query heads of this CTA
  const int i0 = CAUSAL ? j : 0;
  const int n_i = T - i0;
  const int n_it = Gs * n_i;
  auto q_head = [&](int it) {  // flat b*Hq + h
    return b * p.Hq + hkv * p.G + gi * Gs + it / n_i;
  };
  auto q_tile = [&](int it) { return i0 + it % n_i; };
  const WaitCtl wc{p.timeout_ns, p.err, abort_flag};
  const uint32_t tS = tmem_base, tdP = tmem_base + 128, tdV = tmem_base + 256,
                 tdK = tmem_base + 256 + D;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer + dQ reduce
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_kv, 2 * Cfg::kTile);
      for (int c = 0; c < Cfg::kBoxes; ++c) {
        tma_load_3d(sbase + Cfg::kK + c * Cfg::kBox, &tm_k, bar_kv, c * 64, j * 128, bhkv);
        tma_load_3d(sbase + Cfg::kV + c * Cfg::kBox, &tm_v, bar_kv, c * 64, j * 128, bhkv);
      }
      auto load_q = [&](int it) {
        const int s = it & 1;
        const uint32_t qs = sbase + Cfg::kQ0 + s * 2 * Cfg::kTile;
        mbar_arrive_expect_tx(bar_q_full(s), Cfg::kTile);
        for (int c = 0; c < Cfg::kBoxes; ++c)
          tma_load_3d(qs + c * Cfg::kBox, &tm_q, bar_q_full(s), c * 64, q_tile(it) * 128, q_head(it));
      };
      auto load_do = [&](int it) {
        const int s = it & 1;
        const int bhq = q_head(it), i = q_tile(it);
        const uint32_t qs = sbase + Cfg::kQ0 + s * 2 * Cfg::kTile;
        mbar_arrive_expect_tx(bar_qd_full(s), Cfg::kTile + 1024);
        for (int c = 0; c < Cfg::kBoxes; ++c)
          tma_load_3d(qs + Cfg::kTile + c * Cfg::kBox, &tm_do, bar_qd_full(s), c * 64, i * 128,
                      bhq);
        const size_t voff = (size_t)bhq * p.Npad + (size_t)i * 128;
        bulk_load(sbase + Cfg::kVec + s * 1024, p.lse2 + voff, 512, bar_qd_full(s));
        bulk_load(sbase + Cfg::kVec + s * 1024 + 512, p.delta + voff, 512, bar_qd_full(s));
      };
      auto load_stage = [&](int it) {
        load_q(it);
        load_do(it);
      };
      int loaded = 0;
      for (; loaded < 2 && loaded < n_it; ++loaded) load_stage(loaded);
      bool ok = true;
      for (int it = 0; it < n_it && ok; ++it) {
        // dQ_it was staged in stage it&1 (its MMAs are all complete by then):
        // add it to the accumulator half by half, then reuse the stage.
        // Half 0 of dQ_it was staged in the Q area of the stage, half 1 in the
        // dO area: as soon as half 0 has been read, Q for step it+2 can load.
        const uint32_t stage = sbase + Cfg::kQ0 + (it & 1) * 2 * Cfg::kTile;
        for (int h = 0; h < 2 && ok; ++h) {
          if (!(ok = mbar_wait(bar_staged(h), (uint32_t)it & 1u, wc))) break;
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc) {
            const int c = h * (D / 64) + cc;  // 32-column box
            tma_reduce_add_3d(&tm_dq, stage + c * Cfg::kBox, c * 32, q_tile(it) * 128,
                              q_head(it));
          }
          bulk_commit();
        }
        if (ok) mbar_arrive(bar_red_go);
        if constexpr (D == 128) {
          asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          if (ok && loaded < n_it) load_q(loaded);
          bulk_wait_read_all();
          if (ok && loaded < n_it) load_do(loaded++);
        } else {  // at D=64 reloading the whole stage at once measured faster
          bulk_wait_read_all();
          if (ok && loaded < n_it) load_stage(loaded++);
        }
      }
      bulk_wait_all();
      if (ok && GS > 1) {
        // Group split: every stage is free now; take the dV / dK partials the
        // compute warps stage there and add them into the fp32 accumulators.
        mbar_arrive(bar_prod_done);
        for (int h = 0; h < 2 && ok; ++h) {
          if (!(ok = mbar_wait(bar_epi(h), 0, wc))) break;
          const uint32_t src = sbase + Cfg::kQ0 + h * 2 * Cfg::kTile;
          for (int c = 0; c < D / 32; ++c)
            tma_reduce_add_3d(h ? &tm_dk : &tm_dv, src + c * Cfg::kBox, c * 32, j * 128, bhkv);
        }
        bulk_commit();
        bulk_wait_all();
      }
      if (!ok) {
        // Let every load already issued land before the CTA can exit.
        for (int f = (loaded > 2 ? loaded - 2 : 0); f < loaded; ++f) {
          mbar_wait_drain(bar_q_full(f & 1), (uint32_t)(f >> 1) & 1u, wc);
          mbar_wait_drain(bar_qd_full(f & 1), (uint32_t)(f >> 1) & 1u, wc);
        }
        mbar_wait_drain(bar_kv, 0, wc);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescSS = make_idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t kIdescB_MN = make_idesc_bf16(128, D, 1, 0);  // dV, dK
      constexpr uint32_t kIdescDQ = make_idesc_bf16(128, D, 1, 1);    // dQ: A and B MN-major
      const uint32_t k_addr = sbase + Cfg::kK, v_addr = sbase + Cfg::kV, ds_addr = sbase + Cfg::kdS;
      auto q_addr = [&](int s) { return sbase + Cfg::kQ0 + s * 2 * Cfg::kTile; };
      auto do_addr = [&](int s) { return sbase + Cfg::kQ0 + s * 2 * Cfg::kTile + Cfg::kTile; };
      // X^T = A B^T with A a [128 x D] K-major tile (K or V), B a [128 x D] K-major tile.
      auto issue_t = [&](uint32_t dst, uint32_t a, uint32_t bb) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * Cfg::kBox + (kk % 4) * 32;
          mma_ss(dst, make_sdesc_sw128(a + off, 16, 1024), make_sdesc_sw128(bb + off, 16, 1024),
                 kIdescSS, kk > 0);
        }
      };
      auto issue_grads = [&](int s, bool acc) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // dV += P^T dO  (K = 128 queries)
          mma_ts(tdV, tS + (kk / 4) * 64 + (kk % 4) * 8,
                 make_sdesc_sw128(do_addr(s) + kk * 2048, Cfg::kBox, 1024), kIdescB_MN,
                 (acc || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // dK += dS^T Q  (K = 128 queries)
          const uint32_t off = (kk / 4) * Cfg::kBox + (kk % 4) * 32;
          mma_ss(tdK, make_sdesc_sw128(ds_addr + off, 16, 1024),
                 make_sdesc_sw128(q_addr(s) + kk * 2048, Cfg::kBox, 1024), kIdescB_MN,
                 (acc || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // dQ = dS K  (K = 128 keys), into the dP^T columns
          mma_ss(tdP, make_sdesc_sw128(ds_addr + kk * 2048, Cfg::kBox, 1024),
                 make_sdesc_sw128(k_addr + kk * 2048, Cfg::kBox, 1024), kIdescDQ, kk > 0);
      };

      bool ok = mbar_wait(bar_kv, 0, wc) && mbar_wait(bar_q_full(0), 0, wc) &&
                mbar_wait(bar_qd_full(0), 0, wc);
      if (ok) {
        tc_fence_after();
        issue_t(tS, k_addr, q_addr(0));
        issue_t(tdP, v_addr, do_addr(0));
        mma_commit(bar_s);
      }
      for (int it = 0; it < n_it && ok; ++it) {
        const int s = it & 1;
        if (!(ok = mbar_wait(bar_ds, (uint32_t)it & 1u, wc))) break;
        tc_fence_after();
        issue_grads(s, it > 0);
        mma_commit(bar_dq);  // the dQ warps release stage s after staging dQ in it
        if (it + 1 < n_it) {
          const int s1 = (it + 1) & 1;
          if (!(ok = mbar_wait(bar_q_full(s1), (uint32_t)((it + 1) >> 1) & 1u, wc))) break;
          tc_fence_after();
          issue_t(tS, k_addr, q_addr(s1));
          if (!(ok = mbar_wait(bar_dq_free, (uint32_t)it & 1u, wc))) break;
          if (!(ok = mbar_wait(bar_qd_full(s1), (uint32_t)((it + 1) >> 1) & 1u, wc))) break;
          tc_fence_after();
          issue_t(tdP, v_addr, do_addr(s1));
          mma_commit(bar_s);
        }
      }
      mma_commit(bar_done);
      if (!ok) mbar_wait_drain(bar_done, 0, wc);
    }
  } else {
    // ------------------------------------------------------------ compute warps 0-7
    const int wq = warp & 3;   // TMEM lane quadrant
    const int ch = warp >> 2;  // column half
    const int row = wq * 32 + lane;  // key row (dS, epilogue) / query row (dQ staging)
    const int kj = j * 128 + row;
    const bool key_live = kj < p.N;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float C = p.scale_log2;
    const float2 c2 = make_float2(C, C);
    const uint32_t swz = (uint32_t)(row & 7);
    const uint32_t ds_row = sbase + Cfg::kdS + (uint32_t)ch * Cfg::kBox + (uint32_t)row * 128u;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1;
      // ---- dS = P o (dP - Delta) for queries [64ch, 64ch + 64) of this key row
      ok = __all_sync(0xffffffffu, mbar_wait(bar_s, (uint32_t)it & 1u, wc) &&
                                       mbar_wait(bar_qd_full(s), (uint32_t)(it >> 1) & 1u, wc));
      if (!ok) break;
      tc_fence_after();
      const float* lse2 = reinterpret_cast<const float*>(smem + Cfg::kVec + s * 1024) + ch * 64;
      const float* delta = lse2 + 128;
      const bool diag = CAUSAL && q_tile(it) == j;
      const uint32_t ts = tS + lane_off + (uint32_t)ch * 64u;
      const uint32_t tp = tdP + lane_off + (uint32_t)ch * 64u;
      uint32_t sr[2][16], dr[2][16];
      tmem_ld16(ts, sr[0]);
      tmem_ld16(tp, dr[0]);
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 16 query columns per chunk, the next one in flight
        const int bb = c & 1;
        tmem_ld_wait();
        if (c + 1 < 4) {
          tmem_ld16(ts + (c + 1) * 16, sr[bb ^ 1]);
          tmem_ld16(tp + (c + 1) * 16, dr[bb ^ 1]);
        }
        uint32_t pk[8], dk[8];
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const int qc = c * 16 + e;  // query within this half
          const float4 l4 = *reinterpret_cast<const float4*>(lse2 + qc);
          const float4 d4 = *reinterpret_cast<const float4*>(delta + qc);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int ee = e + 2 * h;
            const float2 nl = h ? make_float2(-l4.z, -l4.w) : make_float2(-l4.x, -l4.y);
            const float2 nd = h ? make_float2(-d4.z, -d4.w) : make_float2(-d4.x, -d4.y);
            const float2 x = __ffma2_rn(
                make_float2(__uint_as_float(sr[bb][ee]), __uint_as_float(sr[bb][ee + 1])), c2, nl);
            float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            if (diag) {  // causal: query < key is masked
              const int q = ch * 64 + qc + 2 * h;
              if (q < row) pp.x = 0.f;
              if (q + 1 < row) pp.y = 0.f;
            }
            if (!key_live) pp = make_float2(0.f, 0.f);
            const float2 dd = __fadd2_rn(
                make_float2(__uint_as_float(dr[bb][ee]), __uint_as_float(dr[bb][ee + 1])), nd);
            const float2 ds = __fmul2_rn(pp, dd);
            pk[ee / 2] = pack_bf16x2(pp.x, pp.y);
            dk[ee / 2] = pack_bf16x2(ds.x, ds.y);
          }
        }
        // P^T (bf16) over S^T columns this warp has already read.
        tmem_st8(ts + c * 8, pk);
        // dS^T row to shared memory (box ch) in the 128-byte swizzled layout.
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          const uint32_t chunk = ((uint32_t)(c * 2 + v)) ^ swz;
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(ds_row + chunk * 16),
                       "r"(dk[4 * v]), "r"(dk[4 * v + 1]), "r"(dk[4 * v + 2]), "r"(dk[4 * v + 3])
                       : "memory");
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds);

      // ---- dQ_it: TMEM -> registers -> stage `s` (all MMAs reading it are done)
      ok = __all_sync(0xffffffffu, mbar_wait(bar_dq, (uint32_t)it & 1u, wc));
      if (!ok) break;
      tc_fence_after();
      uint32_t r[D / 64][32];  // this warp's D/2 dQ columns of its query row
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) tmem_ld32(tdP + lane_off + (ch * (D / 64) + cc) * 32, r[cc]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dq_free);
      // Boxes of [128 rows x 32 fp32], 128-byte rows, 16-byte chunks swizzled by row & 7.
      const uint32_t stage = sbase + Cfg::kQ0 + s * 2 * Cfg::kTile + (uint32_t)row * 128u;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc)
#pragma unroll
        for (int v = 0; v < 8; ++v)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                           stage + (ch * (D / 64) + cc) * Cfg::kBox + ((((uint32_t)v) ^ swz) << 4)),
                       "r"(r[cc][4 * v]), "r"(r[cc][4 * v + 1]), "r"(r[cc][4 * v + 2]),
                       "r"(r[cc][4 * v + 3])
                       : "memory");
      fence_proxy_async_smem();
      if (it > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar_red_go, (uint32_t)(it - 1) & 1u, wc));
        if (!ok) break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_staged(ch));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_done, 0, wc));
    if (ok && GS > 1) {
      // Group split: stage this row's fp32 dV (half 0) or unscaled dK (half 1)
      // partial into ring stage `ch` for the producer's reduce-add.
      ok = __all_sync(0xffffffffu, mbar_wait(bar_prod_done, 0, wc));
      if (ok) {
        tc_fence_after();
        const uint32_t src = (ch ? tdK : tdV) + lane_off;
        const uint32_t stage = sbase + Cfg::kQ0 + ch * 2 * Cfg::kTile + (uint32_t)row * 128u;
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
      }
    } else if (ok) {
      // Epilogue: half 0 writes dV, half 1 writes dK (scaled) of this key row.
      tc_fence_after();
      const size_t orow = ((size_t)bhkv * p.N + (size_t)(key_live ? kj : 0)) * D;
      uint4* out = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(ch ? p.dk : p.dv) + orow);
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
            w.x = pack_bf16x2(__uint_as_float(rr[8 * v + 0]) * mul, __uint_as_float(rr[8 * v + 1]) * mul);
            w.y = pack_bf16x2(__uint_as_float(rr[8 * v + 2]) * mul, __uint_as_float(rr[8 * v + 3]) * mul);
            w.z = pack_bf16x2(__uint_as_float(rr[8 * v + 4]) * mul, __uint_as_float(rr[8 * v + 5]) * mul);
            w.w = pack_bf16x2(__uint_as_float(rr[8 * v + 6]) * mul, __uint_as_float(rr[8 * v + 7]) * mul);
            out[c * 4 + v] = w;
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

// Delta and LSE2 into row-padded buffers; zero the dQ accumulator.  One warp per
// padded row (b*Hq + h, i), i < Npad.
template <int D>
__global__ void __launch_bounds__(256)
    bwd_preprocess(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                   const float* __restrict__ lse, float* __restrict__ lse2,
                   float* __restrict__ delta, float* __restrict__ dq_acc, long long rows, int N,
                   int Npad, float* __restrict__ dk_acc, float* __restrict__ dv_acc,
                   long long kv_rows) {
  const long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const long long bh = r / Npad;
  const int i = (int)(r % Npad);
  float acc = 0.f;
  if (i < N) {
    constexpr int kPer = D / 32;  // elements per lane: 2 or 4
    const size_t base = ((size_t)bh * N + i) * D + (size_t)lane * kPer;
    if (kPer == 2) {
      const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(o + base);
      const __nv_bfloat162 g = *reinterpret_cast<const __nv_bfloat162*>(dout + base);
      acc = __bfloat162float(a.x) * __bfloat162float(g.x) + __bfloat162float(a.y) * __bfloat162float(g.y);
    } else {
      const uint2 a = *reinterpret_cast<const uint2*>(o + base);
      const uint2 g = *reinterpret_cast<const uint2*>(dout + base);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
      for (int t = 0; t < 2; ++t)
        acc += __bfloat162float(a2[t].x) * __bfloat162float(g2[t].x) +
               __bfloat162float(a2[t].y) * __bfloat162float(g2[t].y);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  }
  if (lane == 0) {
    lse2[r] = i < N ? lse[(size_t)bh * N + i] * 1.4426950408889634f : INFINITY;
    delta[r] = acc;
  }
  float4* z = reinterpret_cast<float4*>(dq_acc + (size_t)r * D);
#pragma unroll
  for (int t = lane; t < D / 4; t += 32) z[t] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (r < kv_rows) {  // group split: zero the dK/dV accumulators too
    float4* zk = reinterpret_cast<float4*>(dk_acc + (size_t)r * D);
    float4* zv = reinterpret_cast<float4*>(dv_acc + (size_t)r * D);
#pragma unroll
    for (int t = lane; t < D / 4; t += 32) {
      zk[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      zv[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// dQ = scale * dQacc (rows < N) -> bf16.  8 elements per thread.
template <int D>
__global__ void __launch_bounds__(256)
    bwd_postprocess(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq,
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
  w.x = pack_bf16x2(a.x * scale, a.y * scale);
  w.y = pack_bf16x2(a.z * scale, a.w * scale);
  w.z = pack_bf16x2(c.x * scale, c.y * scale);
  w.w = pack_bf16x2(c.z * scale, c.w * scale);
  reinterpret_cast<uint4*>(dq + (size_t)r * D)[g] = w;
}

// Group split: dK = scale * dKacc, dV = dVacc (rows < N) -> bf16.  8 elements
// per thread; rows are (b*Hkv + h)*N + i.
template <int D>
__global__ void __launch_bounds__(256)
    bwd_post_kv(const float* __restrict__ dk_acc, const float* __restrict__ dv_acc,
                __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, long long rows,
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
    w.x = pack_bf16x2(a.x * m, a.y * m);
    w.y = pack_bf16x2(a.z * m, a.w * m);
    w.z = pack_bf16x2(c.x * m, c.y * m);
    w.w = pack_bf16x2(c.z * m, c.w * m);
    reinterpret_cast<uint4*>((which ? dk : dv) + (size_t)r * D)[g] = w;
  }
}

}  // namespace attn
