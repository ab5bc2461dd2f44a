// bwd_dq_kernel.cuh -- dQ of the backward computed per query tile, in a fixed
// order, for the deterministic backward (attn_bwd_deterministic).
//
// The main backward kernel adds each key tile's dQ partial into an fp32
// accumulator with TMA reduce-adds, whose arrival order (and so the rounding of
// the sum) changes from run to run.  Here one CTA owns query tile i of one
// (batch, query head) and walks the key tiles j in order (j <= i when causal),
// recomputing what dQ needs (FlashAttention for Tesla P100 page,
// "Documentation": dS = P o (dP - D)):
//     S_j  = Q_i K_j^T,  P_j = 2^(S_j c - LSE2_i)         (tcgen05, TMEM)
//     dP_j = dO_i V_j^T, dS_j = P_j o (dP_j - Delta_i)    (tcgen05, TMEM)
//     dQ_i += dS_j K_j                                    (fp32 in TMEM, in j order)
// and writes dQ_i = scale * dQ_i once.  Queries sit on the TMEM lanes, so
// LSE2_i and Delta_i are per-thread constants; dS_j goes to shared memory as
// the K-major A operand of the dQ MMA.
//
// Warp roles (12 warps): 0-7 compute (warp w: query rows 32*(w%4).., key half
// w/4), 8 TMA producer (Q_i and dO_i once, K_j and V_j into a 2-stage ring), 9
// TMEM allocator and MMA issuer, 10-11 idle.  The compute warps release S_j and
// dP_j as soon as they have read them into registers, so S_{j+1} and dP_{j+1}
// run while they work on step j.  TMEM columns: [0,128) S, [128,256) dP,
// [256,256+D) dQ.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "ptx.cuh"
#include "kernels.h"

namespace attn {

template <int D>
struct DqCfg {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kBox = 128 * 128;
  static constexpr int kBoxes = D / 64;
  static constexpr int kQ = 0;
  static constexpr int kdO = kTile;
  static constexpr int kKV0 = 2 * kTile;  // stage s: K at kKV0 + 2 s kTile, V right after
  static constexpr int kdS = 6 * kTile;   // dS_j: 128 queries x 128 keys bf16, K-major
  static constexpr int kBar = kdS + 2 * kBox;
  // qd_full, kv_full[2], kv_free[2], s_full, s_used, dp_full, dp_used, ds_full,
  // ds_free, done
  static constexpr int kNumBars = 12;
  static constexpr int kSmemBytes = kBar + kNumBars * 8 + 16;
  static_assert(kSmemBytes <= 227 * 1024, "more shared memory than one CTA may have");
  static constexpr int kThreads = 384;
  static constexpr uint32_t kTmemCols = 512;
};

template <int D, bool CAUSAL, bool F16>
__global__ void __launch_bounds__(384, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p, uint16_t* __restrict__ dq) {
  using Cfg = DqCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.err, 2u);
    return;
  }
  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = (int)(threadIdx.x & 31);

  const uint32_t bar0 = sbase + Cfg::kBar;
  const uint32_t bar_qd = bar0;
  auto bar_kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_kv_free = [&](int s) { return bar0 + 8u * (3 + s); };
  const uint32_t bar_s = bar0 + 8u * 5;        // S_j complete
  const uint32_t bar_s_used = bar0 + 8u * 6;   // S_j read out of TMEM (8 compute warps)
  const uint32_t bar_dp = bar0 + 8u * 7;       // dP_j complete
  const uint32_t bar_dp_used = bar0 + 8u * 8;  // dP_j read out of TMEM (8 compute warps)
  const uint32_t bar_ds = bar0 + 8u * 9;       // dS_j in shared memory (8 compute warps)
  const uint32_t bar_ds_free = bar0 + 8u * 10;  // the dQ MMA has read dS_j
  const uint32_t bar_done = bar0 + 8u * 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kBar + Cfg::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    mbar_init(bar_qd, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_free(s), 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_s_used, 8);
    mbar_init(bar_dp, 1);
    mbar_init(bar_dp_used, 8);
    mbar_init(bar_ds, 8);
    mbar_init(bar_ds_free, 1);
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // ---- work unit: (query tile i, batch, query head).  Causal: the heaviest
  // tiles (largest i) first; non-causal: the tiles of one head consecutive.
  const int T = p.num_kv_tiles;
  const int BH = p.B * p.Hq;
  const int i = CAUSAL ? T - 1 - (int)blockIdx.x / BH : (int)blockIdx.x % T;
  const int bh = CAUSAL ? (int)blockIdx.x % BH : (int)blockIdx.x / T;
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int bhkv = b * p.Hkv + hq / p.G;
  const int n_j = CAUSAL ? i + 1 : T;
  const WaitCtl wc{p.timeout_ns, p.err, abort_flag};
  const uint32_t tS = tmem_base, tdP = tmem_base + 128, tdQ = tmem_base + 256;

  if (warp == 8) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      mbar_arrive_expect_tx(bar_qd, 2 * Cfg::kTile);
      for (int c = 0; c < Cfg::kBoxes; ++c) {
        tma_load_3d(sbase + Cfg::kQ + c * Cfg::kBox, &tm_q, bar_qd, c * 64, i * 128, bh);
        tma_load_3d(sbase + Cfg::kdO + c * Cfg::kBox, &tm_do, bar_qd, c * 64, i * 128, bh);
      }
      auto load_kv = [&](int j) {
        const int s = j & 1;
        const uint32_t st = sbase + Cfg::kKV0 + s * 2 * Cfg::kTile;
        mbar_arrive_expect_tx(bar_kv_full(s), 2 * Cfg::kTile);
        for (int c = 0; c < Cfg::kBoxes; ++c) {
          tma_load_3d(st + c * Cfg::kBox, &tm_k, bar_kv_full(s), c * 64, j * 128, bhkv);
          tma_load_3d(st + Cfg::kTile + c * Cfg::kBox, &tm_v, bar_kv_full(s), c * 64, j * 128,
                      bhkv);
        }
      };
      int loaded = 0;
      for (; loaded < 2 && loaded < n_j; ++loaded) load_kv(loaded);
      bool ok = true;
      for (int j = 0; j + 2 < n_j && ok; ++j) {
        if (!(ok = mbar_wait_tested_inl(bar_kv_free(j & 1), (uint32_t)(j >> 1) & 1u, wc))) break;
        load_kv(j + 2);
        ++loaded;
      }
      if (!ok) {
        for (int f = (loaded > 2 ? loaded - 2 : 0); f < loaded; ++f)
          mbar_wait_drain_inl(bar_kv_full(f & 1), (uint32_t)(f >> 1) & 1u, wc);
        mbar_wait_drain_inl(bar_qd, 0, wc);
      }
    }
  } else if (warp == 9) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t kIdescSS = make_idesc_bf16(128, 128, 0, 0, F16);
      constexpr uint32_t kIdescDQ = make_idesc_bf16(128, D, 1, 0, F16);  // B = K_j MN-major
      constexpr uint32_t kHi = sdesc_sw128_hi(1024);
      const uint32_t kQ = sdesc_sw128_lo(sbase + Cfg::kQ, 16);
      const uint32_t kdO = sdesc_sw128_lo(sbase + Cfg::kdO, 16);
      const uint32_t kdS = sdesc_sw128_lo(sbase + Cfg::kdS, 16);
      auto kK = [&](int s) { return sdesc_sw128_lo(sbase + Cfg::kKV0 + s * 2 * Cfg::kTile, 16); };
      auto kV = [&](int s) {
        return sdesc_sw128_lo(sbase + Cfg::kKV0 + s * 2 * Cfg::kTile + Cfg::kTile, 16);
      };
      auto mK = [&](int s) {
        return sdesc_sw128_lo(sbase + Cfg::kKV0 + s * 2 * Cfg::kTile, Cfg::kBox);
      };
      auto koff = [](int kk) { return (uint32_t)(((kk / 4) * Cfg::kBox + (kk % 4) * 32) >> 4); };
      auto issue_t = [&](uint32_t dst, uint32_t a, uint32_t bb) {  // X = A B^T, K = D
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_w(dst, a, koff(kk), bb, koff(kk), kHi, kIdescSS, kk > 0);
      };
      bool ok = mbar_wait_tested_inl(bar_qd, 0, wc) && mbar_wait_tested_inl(bar_kv_full(0), 0, wc);
      if (ok) {
        tc_fence_after();
        issue_t(tS, kQ, kK(0));
        mma_commit(bar_s);
        issue_t(tdP, kdO, kV(0));
        mma_commit(bar_dp);
      }
      for (int j = 0; j < n_j && ok; ++j) {
        const int s = j & 1;
        if (j + 1 < n_j) {
          const int s1 = s ^ 1;
          if (!(ok = mbar_wait_tested_inl(bar_kv_full(s1), (uint32_t)((j + 1) >> 1) & 1u, wc))) break;
          if (!(ok = mbar_wait_tested_inl(bar_s_used, (uint32_t)j & 1u, wc))) break;
          tc_fence_after();
          issue_t(tS, kQ, kK(s1));
          mma_commit(bar_s);
          if (!(ok = mbar_wait_tested_inl(bar_dp_used, (uint32_t)j & 1u, wc))) break;
          tc_fence_after();
          issue_t(tdP, kdO, kV(s1));
          mma_commit(bar_dp);
        }
        if (!(ok = mbar_wait_tested_inl(bar_ds, (uint32_t)j & 1u, wc))) break;
        tc_fence_after();
        const uint32_t mKs = mK(s);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // dQ += dS_j K_j  (K = 128 keys)
          mma_ss_w(tdQ, kdS, koff(kk), mKs, (uint32_t)((kk * 2048) >> 4), kHi, kIdescDQ,
                   (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar_ds_free);
        mma_commit(bar_kv_free(s));
      }
      mma_commit(bar_done);
      if (!ok) mbar_wait_drain_inl(bar_done, 0, wc);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ compute warps 0-7
    const int wq = warp & 3;
    const int ch = warp >> 2;  // key half
    const int row = wq * 32 + lane;
    const int qi = i * 128 + row;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const size_t vrow = (size_t)bh * p.Npad + (size_t)i * 128 + row;
    const float nlse2 = -p.lse2[vrow];  // +inf rows (past N) give P = 0
    const float ndelta = -p.delta[vrow];
    const float C = p.scale_log2;
    const uint32_t swz = (uint32_t)(row & 7);
    const uint32_t ds_row = sbase + Cfg::kdS + (uint32_t)ch * Cfg::kBox + (uint32_t)row * 128u;
    const uint32_t ts = tS + lane_off + (uint32_t)ch * 64u;
    const uint32_t tp = tdP + lane_off + (uint32_t)ch * 64u;
    bool ok = true;
    for (int j = 0; j < n_j; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait_tested_inl(bar_s, (uint32_t)j & 1u, wc));
      if (!ok) break;
      tc_fence_after();
      float pv[64];
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(ts, ra);
        tmem_ld32(ts + 32, rb);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          pv[c] = __uint_as_float(ra[c]);
          pv[c + 32] = __uint_as_float(rb[c]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_s_used);
      // P = 2^(S c - LSE2) with keys past N or (causal) above the query masked.
      const int k0 = j * 128 + ch * 64;
      const int lim = CAUSAL ? min(p.N - k0, qi - k0 + 1) : p.N - k0;  // keys < lim are live
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float x = ex2_approx(fmaf(pv[c], C, nlse2));
        pv[c] = c < lim ? x : 0.f;
      }
      ok = __all_sync(0xffffffffu, mbar_wait_tested_inl(bar_dp, (uint32_t)j & 1u, wc));
      if (!ok) break;
      tc_fence_after();
      uint32_t dk[32];
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(tp, ra);
        tmem_ld32(tp + 32, rb);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_dp_used);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float d0 = __uint_as_float(c < 32 ? ra[c] : rb[c - 32]);
          const float d1 = __uint_as_float(c < 32 ? ra[c + 1] : rb[c - 31]);
          dk[c / 2] = pack2<F16>(pv[c] * (d0 + ndelta), pv[c + 1] * (d1 + ndelta));
        }
      }
      // dS_j (query row, 64 keys) into the K-major tile once dQ_{j-1} has read it.
      if (j > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait_tested_inl(bar_ds_free, (uint32_t)(j - 1) & 1u, wc));
        if (!ok) break;
      }
#pragma unroll
      for (int v = 0; v < 8; ++v)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                         ds_row + ((((uint32_t)v) ^ swz) << 4)),
                     "r"(dk[4 * v]), "r"(dk[4 * v + 1]), "r"(dk[4 * v + 2]), "r"(dk[4 * v + 3])
                     : "memory");
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait_tested_inl(bar_done, 0, wc));
    if (ok) {
      // Epilogue: dQ = scale * acc, this warp's half of the columns of its row.
      tc_fence_after();
      const bool live = qi < p.N;
      uint4* out = reinterpret_cast<uint4*>(dq + ((size_t)bh * p.N + (size_t)(live ? qi : 0)) * D);
#pragma unroll
      for (int c = ch * (D / 2); c < (ch + 1) * (D / 2); c += 32) {
        uint32_t rr[32];
        tmem_ld32(tdQ + lane_off + c, rr);
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack2<F16>(__uint_as_float(rr[8 * v + 0]) * p.scale, __uint_as_float(rr[8 * v + 1]) * p.scale);
            w.y = pack2<F16>(__uint_as_float(rr[8 * v + 2]) * p.scale, __uint_as_float(rr[8 * v + 3]) * p.scale);
            w.z = pack2<F16>(__uint_as_float(rr[8 * v + 4]) * p.scale, __uint_as_float(rr[8 * v + 5]) * p.scale);
            w.w = pack2<F16>(__uint_as_float(rr[8 * v + 6]) * p.scale, __uint_as_float(rr[8 * v + 7]) * p.scale);
            out[c / 8 + v] = w;
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
