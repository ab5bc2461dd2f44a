// stj_kernel.cuh -- Stieltjes attention forward for sm_103a, on the forward's
// TMA + tcgen05 + TMEM tile pipeline.
//
// FlashStieltjes page ("Why touch softmax", "The challenge", "The kernel"):
// the weights are p_j = (lambda - s_j)^-q with the pole lambda placed above the
// row's best score so that they add up to 1; it is found per row by
// Newton-Raphson from lambda = 1.1 after subtracting the row maximum, and since
// lambda depends on every score the keys are streamed several times, with the
// scores recomputed each time and only two numbers per row kept in between:
//   sweep 0           m = max_j s_j  (s = scale * q.k over the allowed keys)
//   sweeps 1..steps   one Newton step each:  with a_j = pole - s_j,
//                     f = sum_j a_j^-q, g = sum_j a_j^-(q+1),
//                     pole <- pole + (f - 1) / (q g)   (pole = m + lambda)
//   last sweep        p_j = a_j^-q (bf16, over S in TMEM), O += P V (tcgen05)
// O is written as bf16 and the pole (m + lambda, score units) as fp32.
//
// Same CTA layout as the softmax forward: two consecutive 128-row Q tiles of one
// (batch, head), warps 0-3 / 4-7 one tile each (thread = row = TMEM lane), warp
// 8 the TMA producer (Q once; K_j for the first sweeps, K_j and V_j for the
// last, through one shared-memory ring), warp 9 the MMA issuer, 10-11 idle.
// TMEM: S0, S1 (P over them in the last sweep), O0, O1.  The compute warps
// release S_t as soon as they have read it, so S_t(j+1) overlaps their work on
// S_t(j); in the last sweep the order is that of the softmax forward,
//   S0_j ; O1 += P1_{j-1} V_{j-1} ; S1_j ; O0 += P0_j V_j.
// Causal tiles above the diagonal are skipped; keys past N or (causal) above
// the query get no weight.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "ptx.cuh"
#include "kernels.h"
#include "fwd_kernel.cuh"

namespace attn {

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The softmax forward's tiles, ring and register split, with two more barriers.
template <int D>
struct StjCfg : FwdCfg<D> {
  static constexpr int kNumBars = FwdCfg<D>::kNumBars + 2;
  static constexpr int kSmemBytes = FwdCfg<D>::kBarOff + kNumBars * 8 + 16 + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "more shared memory than one CTA may have");
};

template <int D, bool CAUSAL, int ORDER>
__global__ void __launch_bounds__(384, 1)
    stj_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using Cfg = StjCfg<D>;
  constexpr int ST = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_base + pad;

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = (int)(threadIdx.x & 31);

  // Barriers: q_full, full[ST], empty[ST], s_full[2], p_full[2] (4 warps),
  // o_final, s_free[2] (4 warps).
  const uint32_t bar0 = sbase + Cfg::kBarOff;
  auto bar_q = [&]() { return bar0; };
  auto bar_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_empty = [&](int s) { return bar0 + 8u * (1 + ST + s); };
  auto bar_s = [&](int t) { return bar0 + 8u * (1 + 2 * ST + t); };
  auto bar_p = [&](int t) { return bar0 + 8u * (3 + 2 * ST + t); };
  auto bar_o = [&]() { return bar0 + 8u * (5 + 2 * ST); };
  auto bar_sfree = [&](int t) { return bar0 + 8u * (6 + 2 * ST + t); };
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
      mbar_init(bar_sfree(t), 4);
    }
    mbar_init(bar_o(), 1);
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

  // ---- work unit: adjacent query tiles (2qb, 2qb+1) of one (batch, head);
  // causal: the longest blocks of all heads first.
  const int T = p.num_kv_tiles;
  const int BH = p.B * p.Hq;
  const int qb = CAUSAL ? p.num_qblocks - 1 - (int)blockIdx.x / BH : (int)blockIdx.x % p.num_qblocks;
  const int bh = CAUSAL ? (int)blockIdx.x % BH : (int)blockIdx.x / p.num_qblocks;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int bh_kv = b * p.Hkv + h / p.G;
  const int t0 = 2 * qb, t1 = 2 * qb + 1;
  const bool has_t1 = t1 * 128 < p.N;
  const int n0 = CAUSAL ? t0 + 1 : T;
  const int n1 = has_t1 ? (CAUSAL ? t1 + 1 : T) : 0;
  const int nkv = max(n0, n1);
  const int nsw = p.steps + 2;  // max sweep, Newton sweeps, weights sweep
  const WaitCtl wc{p.timeout_ns, p.err, abort_flag};

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    regs_decrease<Cfg::kRegOther>();
    if (lane == 0) {
      const int nq = has_t1 ? 2 : 1;
      mbar_arrive_expect_tx(bar_q(), nq * Cfg::kTileBytes);
      for (int t = 0; t < nq; ++t)
        for (int c = 0; c < Cfg::kBoxes; ++c)
          tma_load_3d(sbase + Cfg::kQOff + t * Cfg::kTileBytes + c * Cfg::kBoxBytes, &tm_q, bar_q(),
                      c * 64, (t ? t1 : t0) * 128, bh);
      uint32_t it = 0;
      bool ok = true;
      for (int sw = 0; sw < nsw && ok; ++sw) {
        const int nkind = (sw == nsw - 1) ? 2 : 1;  // K only, or K and V
        for (int j = 0; j < nkv && ok; ++j) {
          for (int kv = 0; kv < nkind && ok; ++kv, ++it) {
            const int s = (int)(it % ST);
            const uint32_t ph = (it / ST) & 1u;
            ok = mbar_wait_inl(bar_empty(s), ph ^ 1u, wc);
            if (!ok) break;
            mbar_arrive_expect_tx(bar_full(s), Cfg::kTileBytes);
            const CUtensorMap* tm = kv ? &tm_v : &tm_k;
            for (int c = 0; c < Cfg::kBoxes; ++c)
              tma_load_3d(sbase + Cfg::kRingOff + s * Cfg::kTileBytes + c * Cfg::kBoxBytes, tm,
                          bar_full(s), c * 64, j * 128, bh_kv);
          }
        }
      }
      if (!ok) {
        for (uint32_t f = (it > (uint32_t)ST ? it - ST : 0); f < it; ++f)
          mbar_wait_drain_inl(bar_full((int)(f % ST)), (f / ST) & 1u, wc);
        mbar_wait_drain_inl(bar_q(), 0, wc);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    regs_decrease<Cfg::kRegOther>();
    if (lane == 0) {
      constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t kIdescO = make_idesc_bf16(128, D, 1, 0);
      constexpr uint32_t kHi = sdesc_sw128_hi(1024);
      const uint32_t tS[2] = {tmem_base, tmem_base + 128};
      const uint32_t tO[2] = {tmem_base + 256, tmem_base + 384};
      const uint32_t q_lo[2] = {sdesc_sw128_lo(sbase + Cfg::kQOff, 16),
                                sdesc_sw128_lo(sbase + Cfg::kQOff + Cfg::kTileBytes, 16)};
      auto ring = [&](int s) { return sbase + Cfg::kRingOff + s * Cfg::kTileBytes; };
      auto koff = [](int kk) {
        return (uint32_t)(((kk / 4) * Cfg::kBoxBytes + (kk % 4) * 32) >> 4);
      };
      auto issue_qk = [&](int t, uint32_t kaddr) {
        const uint32_t k_lo = sdesc_sw128_lo(kaddr, 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_w(tS[t], q_lo[t], koff(kk), k_lo, koff(kk), kHi, kIdescS, kk > 0);
      };
      auto issue_pv = [&](int t, uint32_t vaddr, bool acc) {
        const uint32_t v_lo = sdesc_sw128_lo(vaddr, Cfg::kBoxBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_w(tO[t], tS[t] + kk * 8, v_lo, (uint32_t)((kk * 2048) >> 4), kHi, kIdescO,
                   (acc || kk > 0) ? 1u : 0u);
      };
      uint32_t ns[2] = {0, 0}, np[2] = {0, 0};
      // S_t into its TMEM columns once the compute warps have read the previous S_t.
      auto issue_s = [&](int t, int sk) -> bool {
        if (ns[t] > 0 && !mbar_wait_inl(bar_sfree(t), (ns[t] - 1) & 1u, wc)) return false;
        tc_fence_after();
        issue_qk(t, ring(sk));
        mma_commit(bar_s(t));
        ++ns[t];
        return true;
      };
      bool ok = mbar_wait_inl(bar_q(), 0, wc);
      uint32_t it = 0;
      for (int sw = 0; sw < nsw && ok; ++sw) {
        const bool last = sw == nsw - 1;
        int sv_prev = 0;
        bool a1_prev = false;
        for (int j = 0; j < nkv && ok; ++j) {
          const bool a0 = j < n0, a1 = j < n1;
          const int sk = (int)(it % ST);
          const uint32_t phk = (it / ST) & 1u;
          ++it;
          int sv = 0;
          uint32_t phv = 0;
          if (last) {
            sv = (int)(it % ST);
            phv = (it / ST) & 1u;
            ++it;
          }
          if (!(ok = mbar_wait_inl(bar_full(sk), phk, wc))) break;
          tc_fence_after();
          if (a0 && !(ok = issue_s(0, sk))) break;
          if (last && j > 0 && a1_prev) {
            if (!(ok = mbar_wait_inl(bar_p(1), np[1] & 1u, wc))) break;
            ++np[1];
            tc_fence_after();
            issue_pv(1, ring(sv_prev), j - 1 > 0);
          }
          if (last && j > 0) mma_commit(bar_empty(sv_prev));
          if (a1 && !(ok = issue_s(1, sk))) break;
          mma_commit(bar_empty(sk));
          if (last) {
            if (!(ok = mbar_wait_inl(bar_full(sv), phv, wc))) break;
            tc_fence_after();
            if (a0) {
              if (!(ok = mbar_wait_inl(bar_p(0), np[0] & 1u, wc))) break;
              ++np[0];
              tc_fence_after();
              issue_pv(0, ring(sv), j > 0);
            }
            sv_prev = sv;
            a1_prev = a1;
          }
        }
        if (ok && last && a1_prev) {
          if ((ok = mbar_wait_inl(bar_p(1), np[1] & 1u, wc))) {
            ++np[1];
            tc_fence_after();
            issue_pv(1, ring(sv_prev), nkv - 1 > 0);
          }
        }
      }
      mma_commit(bar_o());
      if (!ok) mbar_wait_drain_inl(bar_o(), 0, wc);
    }
  } else if (warp >= 10) {
    regs_decrease<Cfg::kRegOther>();
  } else {
    // ------------------------------------------------------------ compute warps
    regs_increase<Cfg::kRegSoftmax>();
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int n_t = t ? n1 : n0;
    const int qtile = t ? t1 : t0;
    const int grow = qtile * 128 + row;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem_base + lane_off + (uint32_t)(t * 128);
    const uint32_t tO = tmem_base + lane_off + 256u + (uint32_t)(t * 128);
    const float scale = p.scale;
    float m = -INFINITY, pole = 0.f;
    uint32_t cnt = 0;
    bool ok = true;
    for (int sw = 0; sw < nsw && ok; ++sw) {
      const bool last = sw == nsw - 1;
      float f = 0.f, g = 0.f;
      for (int j = 0; j < n_t; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait_inl(bar_s(t), cnt & 1u, wc));
        ++cnt;
        if (!ok) break;
        tc_fence_after();
        float s[128];  // raw q.k; the scale is folded into the uses below
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
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sfree(t));
        const int kv0 = j * 128;
        int lim = p.N - kv0;  // keys >= lim get no weight
        if (CAUSAL) lim = min(lim, grow - kv0 + 1);
        // Only the diagonal tile and the ragged last tile have keys to mask
        // (a warp-uniform test); the others take the unmasked loops.
        const bool masked = (CAUSAL && j == qtile) || kv0 + 128 > p.N;
        if (sw == 0) {
          float mx = -INFINITY;
          if (masked) {
#pragma unroll
            for (int c = 0; c < 128; ++c) mx = c < lim ? fmaxf(mx, s[c]) : mx;
          } else {
            float mp[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mp[k] = fmaxf(s[k], s[k + 8]);
#pragma unroll
            for (int c = 16; c < 128; c += 16)
#pragma unroll
              for (int k = 0; k < 8; ++k) mp[k] = fmax3(mp[k], s[c + k], s[c + 8 + k]);
            mx = fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
          }
          m = fmaxf(m, mx * scale);  // scale > 0: the max commutes with it
        } else {
          // a = pole - scale s in one fused step per pair; w = a^-q; Newton
          // sweeps sum w and w / a, the last sweep writes w as P.
          const float2 ns = make_float2(-scale, -scale), pp = make_float2(pole, pole);
          auto weights = [&](int c, float2& w, float2& r) {
            const float2 a = __ffma2_rn(make_float2(s[c], s[c + 1]), ns, pp);
            r = make_float2(rcp_approx(a.x), rcp_approx(a.y));
            w = __fmul2_rn(r, r);
            if (ORDER == 4) w = __fmul2_rn(w, w);
            if (masked) w = make_float2(c < lim ? w.x : 0.f, c + 1 < lim ? w.y : 0.f);
          };
          if (!last) {
            float2 fa = make_float2(0.f, 0.f), ga = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < 128; c += 2) {
              float2 w, r;
              weights(c, w, r);
              fa = __fadd2_rn(fa, w);
              ga = __ffma2_rn(w, r, ga);
            }
            f += fa.x + fa.y;
            g += ga.x + ga.y;
          } else {
            uint32_t pk[64];
#pragma unroll
            for (int c = 0; c < 128; c += 2) {
              float2 w, r;
              weights(c, w, r);
              pk[c / 2] = pack_bf16x2(w.x, w.y);
            }
            tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
            tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_p(t));
          }
        }
      }
      if (!ok) break;
      if (sw == 0)
        pole = m + 1.1f;  // Newton's start, 1.1 above the row max
      else if (!last)
        pole += (f - 1.f) / ((float)ORDER * g);
    }
    if (ok && n_t > 0) ok = __all_sync(0xffffffffu, mbar_wait_inl(bar_o(), 0, wc));
    if (ok && n_t > 0) {
      tc_fence_after();
      const bool live = grow < p.N;
      uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) +
                                             ((size_t)bh * p.N + (size_t)(live ? grow : 0)) * D);
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t r[32];
        tmem_ld32(tO + c, r);
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
            w.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
            w.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
            w.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
            orow[c / 8 + v] = w;
          }
        }
      }
      if (live) p.lse[(size_t)bh * p.N + grow] = pole;
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
