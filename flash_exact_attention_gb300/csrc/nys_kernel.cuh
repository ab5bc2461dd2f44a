// nys_kernel.cuh -- Nystrom attention forward for sm_103a.
//
// FlashNystrom page, "Scope": O = softmax(Q Kt^T) pinv(softmax(Qt Kt^T))
// softmax(Qt K^T) V, with the landmarks Qt, Kt the means of m consecutive
// segments of Q and K and the pseudo-inverse taken by unrolled Newton-Schulz
// steps in fp32; "Configuration": the Tikhonov ridge (M = A^T A + lambda I,
// lambda = |A|_1 |A|_inf / kappa*).  Every score matrix is scaled by the
// caller's scale.  Six kernels, all O(N m D) but for the m x m algebra:
//
//   1 nys_pool_kernel   partial segment sums of the Q rows (HBM stream, 16-byte
//                       loads; one CTA per (head, segment, split))
//   2 nys_qt_kernel     per query head: Qt = the segment means (fp32), and its
//                       bf16 hi/lo tiles for the tensor cores
//   3 nys_kv_kernel     per (query head, key chunk): softmax(scale Qt K^T) V
//                       over the chunk, flash-style on tcgen05 (Qt padded to a
//                       128-row A tile, K/V streamed by TMA), written as
//                       unnormalised partials with row max and row sum; two
//                       otherwise idle warps sum the K rows of each segment out
//                       of the same shared-memory tiles (K is read from HBM once)
//   4 nys_merge_kernel  per (query head, landmark): W = merge of the chunk
//                       partials (fp32)
//   5 nys_lmy_kernel    per query head: Kt, A2 = softmax(scale Qt Kt^T), the
//                       ridge, Newton-Schulz, pinv(A2) and Y = pinv(A2) W, all in
//                       shared memory (fp32, register-tiled); Kt and Y leave as
//                       bf16 hi/lo tiles
//   6 nys_out_kernel    persistent over 128-row query tiles: S = Q Kt^T
//                       (tcgen05, N = mp), softmax over the m landmarks,
//                       O = P Y (tcgen05, K = mp), bf16 out through a swizzled
//                       staging tile and a TMA store; two warp groups take
//                       alternate tiles
//
// HBM traffic: Q twice (kernels 1 and 6), K and V once (kernel 3), O once.
//
// The landmarks and Y are fp32 values that enter bf16 tensor-core products.
// Each is split as x = hi + lo with hi = bf16(x), lo = bf16(x - hi) (16
// significant bits together) and its product taken as the sum of the two
// (the reduction dimension doubled, the other operand used twice): S = Qt K^T
// in kernel 3, S = Q Kt^T and O = P Y in kernel 6.  Those passes are bound by
// HBM, so the extra MMAs cost no time; the softmax weights P stay single bf16
// as in exact flash attention.
#pragma once
#include <cuda.h>
#include <type_traits>
#include <cuda_runtime.h>
#include "ptx.cuh"
#include "kernels.h"

namespace attn {

// bf16 pair of an fp32 value: hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void split_bf16(float x, uint16_t& hi, uint16_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  hi = __bfloat16_as_ushort(h);
  lo = __bfloat16_as_ushort(__float2bfloat16_rn(x - __bfloat162float(h)));
}

// First row of landmark segment i: floor(i N / m).
__device__ __forceinline__ long long seg_lo(int i, int N, int m) {
  return (long long)i * N / m;
}

// ============================================================ 1: pooling
// grid (pool_splits, m, B*Hq), 256 threads.  CTA (s, i, z) sums rows
// lo + L*s/S .. lo + L*(s+1)/S - 1 of segment i = [floor(iN/m), floor((i+1)N/m))
// of query plane z into pool_part.
template <int D>
__global__ void __launch_bounds__(256) nys_pool_kernel(const NysParams p) {
  constexpr int CG = D / 8;     // 16-byte column groups of a row
  constexpr int RG = 256 / CG;  // rows read per pass
  __shared__ float red[RG][D];
  const int split = (int)blockIdx.x, i = (int)blockIdx.y, z = (int)blockIdx.z;
  const uint16_t* src = static_cast<const uint16_t*>(p.q) + (size_t)z * p.N * D;
  const long long lo = seg_lo(i, p.N, p.m), hi = seg_lo(i + 1, p.N, p.m);
  const long long L = hi - lo;
  const long long r0 = lo + L * split / p.pool_splits;
  const long long r1 = lo + L * (split + 1) / p.pool_splits;
  const int t = (int)threadIdx.x, cg = t % CG, rg = t / CG;
  const uint4* base = reinterpret_cast<const uint4*>(src) + cg;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  auto add = [&](const uint4& u) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc[2 * e] += __uint_as_float(w[e] << 16);
      acc[2 * e + 1] += __uint_as_float(w[e] & 0xffff0000u);
    }
  };
  long long r = r0 + rg;
  for (; r + 3 * RG < r1; r += 4 * RG) {
    uint4 u[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) u[k] = __ldg(base + (r + (long long)k * RG) * CG);
#pragma unroll
    for (int k = 0; k < 4; ++k) add(u[k]);
  }
  for (; r < r1; r += RG) add(__ldg(base + r * CG));
#pragma unroll
  for (int e = 0; e < 8; ++e) red[rg][cg * 8 + e] = acc[e];
  __syncthreads();
  if (t < D) {
    float s = 0.f;
#pragma unroll 8
    for (int g = 0; g < RG; ++g) s += red[g][t];
    p.pool_part[(((size_t)z * p.m + i) * p.pool_splits + split) * D + t] = s;
  }
}

// ============================================================ 2: Qt
// grid (128 D / W / T, B*Hq), T threads: thread (i, g) of head bh takes row i
// of Qt, columns W g .. W g + W - 1 (the mean of segment i: fp32 copy and bf16
// hi/lo pair in two 128-row tiles; rows >= m zero), the split partial sums
// added in order, two chains (even and odd splits) per column.  W = 4 (16-byte
// loads, T = 256) when there are few splits; W = 1 (T = D) when there are
// many, where the longer chains of loads want more threads and more SMs.
constexpr int kNysSmallThreads = 256;
template <int D, int W>
__global__ void __launch_bounds__(W == 4 ? kNysSmallThreads : D) nys_qt_kernel(const NysParams p) {
  static_assert(W == 1 || W == 4, "one or four columns per thread");
  using V = typename std::conditional<W == 4, float4, float>::type;
  constexpr int G = D / W;
  const int idx = (int)(blockIdx.x * blockDim.x + threadIdx.x);
  const int i = idx / G, d0 = (idx % G) * W, bh = (int)blockIdx.y;
  if (i >= 128) return;
  const int m = p.m, S = p.pool_splits;
  auto add = [](V& acc, const V& a) {
    if constexpr (W == 4) {
      acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
    } else {
      acc += a;
    }
  };
  float x[W];
#pragma unroll
  for (int e = 0; e < W; ++e) x[e] = 0.f;
  if (i < m) {
    const V* pq = reinterpret_cast<const V*>(p.pool_part + ((size_t)bh * m + i) * S * D + d0);
    V s0, s1;
    memset(&s0, 0, sizeof(V));
    memset(&s1, 0, sizeof(V));
    int k = 0;
#pragma unroll 4
    for (; k + 1 < S; k += 2) {
      const V a = pq[(size_t)k * G], c = pq[(size_t)(k + 1) * G];
      add(s0, a);
      add(s1, c);
    }
    if (k < S) add(s0, pq[(size_t)k * G]);
    const float len = (float)(seg_lo(i + 1, p.N, m) - seg_lo(i, p.N, m));
    const float* f0 = reinterpret_cast<const float*>(&s0);
    const float* f1 = reinterpret_cast<const float*>(&s1);
#pragma unroll
    for (int e = 0; e < W; ++e) x[e] = (f0[e] + f1[e]) / len;
    V xv;
    memcpy(&xv, x, sizeof(V));
    *reinterpret_cast<V*>(p.qt32 + ((size_t)bh * m + i) * D + d0) = xv;
  }
  uint16_t* q16 = p.qt16 + (size_t)bh * 2 * 128 * D + (size_t)i * D + d0;
  if constexpr (W == 4) {
    uint16_t hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split_bf16(x[e], hi[e], lo[e]);
    *reinterpret_cast<uint2*>(q16) = make_uint2(hi[0] | ((uint32_t)hi[1] << 16),
                                                hi[2] | ((uint32_t)hi[3] << 16));
    *reinterpret_cast<uint2*>(q16 + 128 * D) = make_uint2(lo[0] | ((uint32_t)lo[1] << 16),
                                                          lo[2] | ((uint32_t)lo[3] << 16));
  } else {
    split_bf16(x[0], q16[0], q16[128 * D]);
  }
}

// ============================================================ 5: landmarks, pinv, Y
// C (MR x NC, both multiples of 16) = A B with A given as its transpose At
// (At[k][i] = A[i][k], row stride lda) and B (row stride ldb), every entry
// summed over k in order.  Each warp takes (8 TRL) x 16 blocks of C
// (grid-stride over the CTA's warps); lane (rg, cg) = (lane / 4, lane % 4)
// holds the TRL x 4 entries at rows TRL rg .. TRL rg + TRL - 1 and columns
// 4 cg .. 4 cg + 3 of the block, and per K-step reads TRL values of At's row k
// and 4 of B's with vector loads and issues 2 TRL packed fp32x2
// multiply-adds.  These products are bound by shared-memory wavefronts: a
// warp's vector load costs one wavefront per 32 floats it delivers, broadcast
// or not, so larger register tiles (fewer loads per multiply-add) beat more
// warps.  store(i, j, value) writes the result.
template <int TRL, class Store>
__device__ __forceinline__ void mm_blocks_t(const float* At, int lda, const float* B, int ldb, int K,
                                            int MR, int NC, Store store) {
  constexpr int BR = 8 * TRL;
  const int warp = (int)(threadIdx.x >> 5), lane = (int)(threadIdx.x & 31);
  const int nwarps = (int)(blockDim.x >> 5);
  const int bcols = NC / 16, blocks = (MR / BR) * bcols;
  const int ro = TRL * (lane >> 2), co = 4 * (lane & 3);
  for (int blk = warp; blk < blocks; blk += nwarps) {
    const int r0 = (blk / bcols) * BR + ro, c0 = (blk % bcols) * 16 + co;
    const float* a = At + r0;
    const float* bb = B + c0;
    float2 acc[TRL][2];
#pragma unroll
    for (int x = 0; x < TRL; ++x) acc[x][0] = acc[x][1] = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
      float av[TRL];
      if constexpr (TRL == 8) {
        const float4 v4 = *reinterpret_cast<const float4*>(a + k * lda);
        const float4 w4 = *reinterpret_cast<const float4*>(a + k * lda + 4);
        av[0] = v4.x; av[1] = v4.y; av[2] = v4.z; av[3] = v4.w;
        av[4] = w4.x; av[5] = w4.y; av[6] = w4.z; av[7] = w4.w;
      } else if constexpr (TRL == 4) {
        const float4 v4 = *reinterpret_cast<const float4*>(a + k * lda);
        av[0] = v4.x; av[1] = v4.y; av[2] = v4.z; av[3] = v4.w;
      } else {
        const float2 v2 = *reinterpret_cast<const float2*>(a + k * lda);
        av[0] = v2.x; av[1] = v2.y;
      }
      const float4 bv = *reinterpret_cast<const float4*>(bb + k * ldb);
      const float2 b01 = make_float2(bv.x, bv.y), b23 = make_float2(bv.z, bv.w);
#pragma unroll
      for (int x = 0; x < TRL; ++x) {
        const float2 ax = make_float2(av[x], av[x]);
        acc[x][0] = __ffma2_rn(ax, b01, acc[x][0]);
        acc[x][1] = __ffma2_rn(ax, b23, acc[x][1]);
      }
    }
#pragma unroll
    for (int x = 0; x < TRL; ++x) {
      store(r0 + x, c0, acc[x][0].x);
      store(r0 + x, c0 + 1, acc[x][0].y);
      store(r0 + x, c0 + 2, acc[x][1].x);
      store(r0 + x, c0 + 3, acc[x][1].y);
    }
  }
}

// The register tile for a shape: 8 x 4 for the 64 x 64 products over 64 steps
// (4 warps; 12 wavefronts per 1024 multiply-adds), 4 x 4 for the other
// products of at least 64 x 64 entries with MR a multiple of 32, else 2 x 4
// (the smaller products, where more warps matter more).
template <class Store>
__device__ __forceinline__ void mm_blocks(const float* At, int lda, const float* B, int ldb, int K,
                                          int MR, int NC, Store store) {
  if (MR == 64 && NC == 64 && K <= 64)
    mm_blocks_t<8>(At, lda, B, ldb, K, MR, NC, store);
  else if (MR % 32 == 0 && MR * NC >= 64 * 64)
    mm_blocks_t<4>(At, lda, B, ldb, K, MR, NC, store);
  else
    mm_blocks_t<2>(At, lda, B, ldb, K, MR, NC, store);
}

// mp x mp result (mp in {16, 32, 48, 64}) over K steps into C (row stride mp);
// ends with a __syncthreads.
__device__ __forceinline__ void mm_sq(int mp, const float* At, int lda, const float* B, int ldb,
                                      int K, float* C) {
  mm_blocks(At, lda, B, ldb, K, mp, mp, [&](int i, int j, float v) { C[i * mp + j] = v; });
  __syncthreads();
}

// max over columns of the column |sums| times max over rows of the row |sums|
// of an mp x mp matrix (zero padding does not change either); every thread
// gets the result.  `red` holds 2 * 64 + 1 floats.  512 threads.
__device__ __forceinline__ float norm1_norminf(const float* A, int mp, float* red) {
  const int t = (int)threadIdx.x, warp = t >> 5, lane = t & 31;
  if (t < mp) {
    float s = 0.f;
    for (int r = 0; r < mp; ++r) s += fabsf(A[r * mp + t]);
    red[t] = s;
  }
  for (int r = warp; r < mp; r += 16) {
    float s = (lane < mp ? fabsf(A[r * mp + lane]) : 0.f) +
              (lane + 32 < mp ? fabsf(A[r * mp + lane + 32]) : 0.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) red[64 + r] = s;
  }
  __syncthreads();
  if (warp == 0) {  // the two maxima over (at most) 64 entries each
    float n1 = 0.f, ninf = 0.f;
    for (int e = lane; e < mp; e += 32) {
      n1 = fmaxf(n1, red[e]);
      ninf = fmaxf(ninf, red[64 + e]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      n1 = fmaxf(n1, __shfl_xor_sync(0xffffffffu, n1, o));
      ninf = fmaxf(ninf, __shfl_xor_sync(0xffffffffu, ninf, o));
    }
    if (lane == 0) red[128] = n1 * ninf;
  }
  __syncthreads();
  const float r = red[128];
  __syncthreads();
  return r;
}

// Dst = Src^T for mp x mp matrices.  At mp = 64 a warp moves 32 entries along
// a diagonal, (i, j) = (32 h + lane, (c + lane) mod 64) for its piece (h, c),
// so that both its reads (banks j mod 32) and its writes (banks i mod 32) hit
// 32 different banks.
__device__ __forceinline__ void smem_transpose(const float* src, float* dst, int mp) {
  if (mp == 64) {
    const int lane = (int)(threadIdx.x & 31);
    for (int pc = (int)(threadIdx.x >> 5); pc < 128; pc += (int)(blockDim.x >> 5)) {
      const int i = (pc & 1) * 32 + lane, j = ((pc >> 1) + lane) & 63;
      dst[j * 64 + i] = src[i * 64 + j];
    }
    return;
  }
  for (int idx = (int)threadIdx.x; idx < mp * mp; idx += (int)blockDim.x)
    dst[(idx % mp) * mp + idx / mp] = src[idx];
}

template <int D>
struct NysLyCfg {
  static constexpr int kThreads = 512;
  // row stride of the transposed landmark tiles: a multiple of 4 (vector
  // loads), not of 32 (the transposed writes spread over 8 banks)
  static constexpr int kLd = 68;
  // shared floats: R0 = qtT [D][kLd] (then W [64][D]), R1 = ktT [D][kLd],
  // eight 64 x 64 matrices (A, At, M, Mt, X, Xt, T1, T2), red [132]
  static constexpr int kR = D * kLd > 64 * D ? D * kLd : 64 * D;
  static constexpr int kFloats = 2 * kR + 8 * 64 * 64 + 132;
  static constexpr int kSmemBytes = kFloats * 4;
  static_assert(kSmemBytes <= 227 * 1024, "more shared memory than one CTA may have");
};

// One CTA (512 threads) per query head (b, h).
template <int D>
__global__ void __launch_bounds__(512, 1) nys_lmy_kernel(const NysParams p) {
  using Cfg = NysLyCfg<D>;
  constexpr int LD = Cfg::kLd;
  extern __shared__ __align__(16) float ly[];
  const int m = p.m, mp = p.mp, P = p.kparts;
  float* qtT = ly;            // [D][LD]
  float* W = ly;              // [64][D], after A2
  float* ktT = ly + Cfg::kR;  // [D][LD]
  float* A = ktT + Cfg::kR;   // [mp][mp] each
  float* At = A + 64 * 64;
  float* M = At + 64 * 64;
  float* Mt = M + 64 * 64;
  float* X = Mt + 64 * 64;
  float* Xt = X + 64 * 64;
  float* T1 = Xt + 64 * 64;
  float* T2 = T1 + 64 * 64;
  float* red = T2 + 64 * 64;
  const int t = (int)threadIdx.x;
  const int bh = (int)blockIdx.x, b = bh / p.Hq, h = bh % p.Hq;
  const int bhk = b * p.Hkv + h / p.G;

  // Qt from its fp32 copy, Kt from the key-chunk partial sums of its segments
  // (chunk c_first(i) + k, share s of its tiles wrote slot k * shares + s;
  // slots of no (chunk, share) pair stay zero).  Per landmark first: the
  // number of slots and 1 / segment length.
  int* seg_parts = reinterpret_cast<int*>(red);  // red[0..63]
  float* seg_inv = red + 64;                     // red[64..127]
  if (t < m) {
    const long long chunk_rows = (long long)p.kv_tpc * 128;
    const long long lo = seg_lo(t, p.N, m), hi = seg_lo(t + 1, p.N, m);
    seg_parts[t] = ((int)((hi - 1) / chunk_rows - lo / chunk_rows) + 1) * (4 / (D / 64));
    seg_inv[t] = 1.f / (float)(hi - lo);
  }
  __syncthreads();
  {
    // Thread t: column d = t % D of rows i0, i0 + di, ... (all its loads
    // issued before the sums that need them: one round trip per partial).
    constexpr int kU = D * 64 / 512, di = 512 / D;
    const int d = t % D, i0 = t / D;
    float qv[kU], s0[kU], s1[kU];
    int np[kU];
    int maxp = 0;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * di;
      qv[u] = 0.f;
      s0[u] = 0.f;
      s1[u] = 0.f;
      np[u] = 0;
      if (i < m) {
        qv[u] = p.qt32[((size_t)bh * m + i) * D + d];
        np[u] = seg_parts[i];
        maxp = max(maxp, np[u]);
      }
    }
    // two chains per entry (even and odd partials), added at the end
    for (int k = 0; k < maxp; k += 2) {
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const float* pk = p.kpart + (((size_t)bhk * m + i0 + u * di) * P + k) * D + d;
        if (k < np[u]) s0[u] += pk[0];
        if (k + 1 < np[u]) s1[u] += pk[D];
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * di;
      if (i < mp) {
        qtT[d * LD + i] = qv[u];
        ktT[d * LD + i] = i < m ? (s0[u] + s1[u]) * seg_inv[i] : 0.f;
      }
    }
  }
  for (int idx = t; idx < mp * mp; idx += 512) A[idx] = 0.f;
  __syncthreads();  // (also: red is free again)
  if (h % p.G == 0) {  // Kt as a bf16 hi/lo pair of mp-row tiles, once per key head
    uint16_t* dk = p.kt16 + (size_t)bhk * 2 * mp * D;
    for (int idx = t; idx < mp * D; idx += 512) {
      const int r = idx / D, d = idx % D;
      split_bf16(ktT[d * LD + r], dk[idx], dk[mp * D + idx]);
    }
  }

  // A2 = softmax(scale Qt Kt^T) over the m landmarks (zero outside m x m)
  {
    auto st = [&](int i, int j, float v) {
      if (i < m && j < m) A[i * mp + j] = v * p.scale;
    };
    mm_blocks(qtT, LD, ktT, LD, D, mp, mp, st);
  }
  __syncthreads();
  {
    const int warp = t >> 5, lane = t & 31;
    for (int i = warp; i < m; i += 16) {
      const float a0 = lane < m ? A[i * mp + lane] : -INFINITY;
      const float a1 = lane + 32 < m ? A[i * mp + lane + 32] : -INFINITY;
      float mx = fmaxf(a0, a1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float e0 = lane < m ? expf(a0 - mx) : 0.f;
      const float e1 = lane + 32 < m ? expf(a1 - mx) : 0.f;
      float sum = e0 + e1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      const float inv = 1.f / sum;
      if (lane < m) A[i * mp + lane] = e0 * inv;
      if (lane + 32 < m) A[i * mp + lane + 32] = e1 * inv;
    }
  }
  __syncthreads();
  smem_transpose(A, At, mp);
  // W (rows >= m zero) into the region Qt occupied
  {
    const float4* wsrc = reinterpret_cast<const float4*>(p.w + (size_t)bh * m * D);
    float4* wdst = reinterpret_cast<float4*>(W);
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 64 * D / 4 / 512; ++u) {  // 16-byte pieces, rows >= m zero
      const int idx = t + u * 512;
      if (idx < mp * D / 4) wdst[idx] = idx < m * D / 4 ? wsrc[idx] : z;
    }
  }
  __syncthreads();

  // Newton-Schulz on M = A^T A + lambda I (ridge) or on A itself.  With the
  // ridge M is symmetric, and so is every iterate (X_0 = M / c0 and each step
  // is a polynomial in M): the transposed operands are the matrices themselves.
  const bool ridge = p.kappa > 0.f;
  const float* Mtp = Mt;
  const float* Xtp = Xt;
  if (ridge) {
    const float lambda = norm1_norminf(A, mp, red) / p.kappa;
    mm_sq(mp, A, mp, A, mp, mp, M);  // (A^T)^T = A
    for (int i = t; i < m; i += 512) M[i * mp + i] += lambda;
    Mtp = M;
    Xtp = X;
  } else {
    for (int idx = t; idx < mp * mp; idx += 512) {
      M[idx] = A[idx];
      Mt[idx] = At[idx];
    }
  }
  __syncthreads();
  const float c0 = norm1_norminf(M, mp, red);
  const float inv_c0 = c0 > 0.f ? 1.f / c0 : 0.f;
  for (int idx = t; idx < mp * mp; idx += 512) {  // X = M^T / c0
    X[idx] = Mtp[idx] * inv_c0;
    if (!ridge) Xt[idx] = M[idx] * inv_c0;
  }
  __syncthreads();
  for (int it = 0; it < p.iters; ++it) {
    mm_sq(mp, Mtp, mp, X, mp, mp, T1);  // M X
    mm_sq(mp, Xtp, mp, T1, mp, mp, T2);  // X M X
    for (int idx = t; idx < mp * mp; idx += 512) {
      const float x = 2.f * X[idx] - T2[idx];
      X[idx] = x;
      if (!ridge) Xt[(idx % mp) * mp + idx / mp] = x;
    }
    __syncthreads();
  }
  // pinv(A2)^T: (X A^T)^T = A X^T = A X with the ridge, X^T without
  const float* Pt = Xt;
  if (ridge) {
    mm_sq(mp, At, mp, X, mp, mp, T1);
    Pt = T1;
  }

  // Y = pinv(A2) W as a bf16 hi/lo pair (rows >= m zero: W's are)
  {
    uint16_t* y = p.y16 + (size_t)bh * 2 * mp * D;
    auto st = [&](int i, int j, float v) { split_bf16(v, y[i * D + j], y[(mp + i) * D + j]); };
    mm_blocks(Pt, mp, W, D, mp, mp, D, st);
  }
}

// ============================================================ 3: softmax(Qt K^T) V
template <int D>
struct NysKvCfg {
  static constexpr int kTileBytes = 128 * D * 2;  // one 128-row bf16 tile
  static constexpr int kBoxBytes = 128 * 128;     // one 64-column TMA box
  static constexpr int kBoxes = D / 64;
  // ring slots of one tile each, filled K_0, V_0, K_1, V_1, ...; a K slot is
  // released when S_j has read it, a V slot when O += P_j V_j has
  static constexpr int kSlots = (D == 128) ? 5 : 8;
  static constexpr int kQOff = 0;                      // Qt hi tile, then Qt lo tile
  static constexpr int kRingOff = 2 * kTileBytes;
  static constexpr int kBarOff = kRingOff + kSlots * kTileBytes;
  // barriers: q_full, full[slots], empty[slots], s_full[2], p_full[2], pv_done[2], done
  static constexpr int kNumBars = 1 + 2 * kSlots + 7;
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "more shared memory than one CTA may have");
  static constexpr int kThreads = 256;  // softmax warps 0-1, K-sum warps 2-3 and 6-7, producer, MMA
  static constexpr uint32_t kTmemCols = 512;  // S0, S1 (128 each), O (D)
};

// grid (kv_chunks, B*Hq).  Warps 0-1: thread = landmark row = TMEM lane (rows
// >= m are the zero padding of the A tile; m <= 64, so warps 2-3 hold none);
// warp 4: TMA producer (Qt once, K_j and V_j through the ring); warp 5: MMA;
// K-sum warps 2, 3, 6, 7: in the CTA of the first query head of each
// key/value head, the K row sums of each landmark segment, read from the K
// tiles in shared memory and written per (segment, chunk, warp): K-sum warp w
// (0-3) takes the 64-column box w % (D / 64) of the rows in its share
// w / (D / 64) of each tile.  A ring slot is free again once the MMA has read
// it and the four K-sum warps have passed it.
// Order of the tensor work: S_0, S_1, O += P_0 V_0, S_2, O += P_1 V_1, ...;
// S_j overwrites the TMEM columns that P_{j-2} occupied only after the
// (in-order) O += P_{j-2} V_{j-2} was issued.
// The running max is kept lazily: O and l are rescaled (after the previous
// P V has completed) only when the tile max exceeds the max in use by more
// than 8 (log2 units), so the weights in use stay below 2^8.
// P V completions are signalled on pv_done[u % 2]; the softmax warps observe
// every phase of each in order (O += P_{j-2} V_{j-2} at tile j, already done by
// then), because a parity wait on a barrier two phases behind would pass at
// once, and nothing orders the arrivals of two different commits.
template <int D>
__global__ void __launch_bounds__(256, 1)
    nys_kv_kernel(const __grid_constant__ CUtensorMap tm_qt, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const NysParams p) {
  using Cfg = NysKvCfg<D>;
  constexpr int ST = Cfg::kSlots;
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
  auto bar_s = [&](int b) { return bar0 + 8u * (1 + 2 * ST + b); };
  auto bar_p = [&](int b) { return bar0 + 8u * (3 + 2 * ST + b); };
  auto bar_pv = [&](int b) { return bar0 + 8u * (5 + 2 * ST + b); };
  auto bar_done = [&]() { return bar0 + 8u * (7 + 2 * ST); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kBarOff + Cfg::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int m = p.m;
  const int nw = (m + 31) / 32;  // softmax warps holding landmark rows
  if (threadIdx.x == 0) {
    mbar_init(bar_q(), 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 5);  // MMA commit + the four K-sum warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_s(b), 1);
      mbar_init(bar_p(b), nw);
    }
    mbar_init(bar_pv(0), 1);
    mbar_init(bar_pv(1), 1);
    mbar_init(bar_done(), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_qt);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int chunk = (int)blockIdx.x, bh = (int)blockIdx.y;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int bhk = b * p.Hkv + h / p.G;
  const int j0 = chunk * p.kv_tpc;
  const int n = min(p.kv_tpc, p.num_kv_tiles - j0);
  const WaitCtl wc{p.timeout_ns, p.err, abort_flag};
  auto slot = [&](int s) { return sbase + Cfg::kRingOff + s * Cfg::kTileBytes; };

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_q(), 2 * Cfg::kTileBytes);
      for (int u = 0; u < 2; ++u)
        for (int c = 0; c < Cfg::kBoxes; ++c)
          tma_load_3d(sbase + Cfg::kQOff + u * Cfg::kTileBytes + c * Cfg::kBoxBytes, &tm_qt, bar_q(),
                      c * 64, u * 128, bh);
      bool ok = true;
      int it = 0;
      for (; it < 2 * n; ++it) {
        const int s = it % ST;
        if (!(ok = mbar_wait_inl(bar_empty(s), ((uint32_t)(it / ST) & 1u) ^ 1u, wc))) break;
        mbar_arrive_expect_tx(bar_full(s), Cfg::kTileBytes);
        const CUtensorMap* tm = (it & 1) ? &tm_v : &tm_k;
        for (int c = 0; c < Cfg::kBoxes; ++c)
          tma_load_3d(slot(s) + c * Cfg::kBoxBytes, tm, bar_full(s), c * 64, (j0 + it / 2) * 128, bhk);
      }
      if (!ok) {
        for (int f = (it > ST ? it - ST : 0); f < it; ++f)
          mbar_wait_drain_inl(bar_full(f % ST), (uint32_t)(f / ST) & 1u, wc);
        mbar_wait_drain_inl(bar_q(), 0, wc);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t kIdescO = make_idesc_bf16(128, D, 1, 0);
      constexpr uint32_t kHi = sdesc_sw128_hi(1024);
      const uint32_t tS[2] = {tmem_base, tmem_base + 128};
      const uint32_t tO = tmem_base + 256;
      const uint32_t qh_lo = sdesc_sw128_lo(sbase + Cfg::kQOff, 16);
      const uint32_t ql_lo = sdesc_sw128_lo(sbase + Cfg::kQOff + Cfg::kTileBytes, 16);
      auto koff = [](int kk) {
        return (uint32_t)(((kk / 4) * Cfg::kBoxBytes + (kk % 4) * 32) >> 4);
      };
      // O += P_u V_u, once P_u is in TMEM and V_u in its slot
      auto issue_pv = [&](int u) -> bool {
        const int iv = 2 * u + 1, sv = iv % ST;
        if (!mbar_wait_inl(bar_p(u & 1), (uint32_t)(u >> 1) & 1u, wc)) return false;
        if (!mbar_wait_inl(bar_full(sv), (uint32_t)(iv / ST) & 1u, wc)) return false;
        tc_fence_after();
        const uint32_t v_lo = sdesc_sw128_lo(slot(sv), Cfg::kBoxBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_w(tO, tS[u & 1] + kk * 8, v_lo, (uint32_t)((kk * 2048) >> 4), kHi, kIdescO,
                   (u > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar_pv(u & 1));
        mma_commit(bar_empty(sv));
        return true;
      };
      bool ok = mbar_wait_inl(bar_q(), 0, wc);
      for (int jj = 0; jj < n && ok; ++jj) {
        const int ik = 2 * jj, s = ik % ST;
        if (!(ok = mbar_wait_inl(bar_full(s), (uint32_t)(ik / ST) & 1u, wc))) break;
        tc_fence_after();
        const uint32_t k_lo = sdesc_sw128_lo(slot(s), 16);
        // S = Qt_hi K^T + Qt_lo K^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_w(tS[jj & 1], qh_lo, koff(kk), k_lo, koff(kk), kHi, kIdescS, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_w(tS[jj & 1], ql_lo, koff(kk), k_lo, koff(kk), kHi, kIdescS, 1u);
        mma_commit(bar_s(jj & 1));
        mma_commit(bar_empty(s));
        if (jj > 0 && !(ok = issue_pv(jj - 1))) break;
      }
      if (ok && n > 0) ok = issue_pv(n - 1);
      // after an abort, let every tcgen05 op already issued finish before TMEM is freed
      mma_commit(bar_done());
      if (!ok) mbar_wait_drain_inl(bar_done(), 0, wc);
    }
  } else if (warp == 2 || warp == 3 || warp >= 6) {
    // ------------------------------------------------------------ K segment sums
    constexpr int kShares = 4 / Cfg::kBoxes;  // row shares of a tile
    const int ks = warp < 6 ? warp - 2 : warp - 4;  // 0..3
    const int box = ks % Cfg::kBoxes, share = ks / Cfg::kBoxes;
    const int r_lo = share * (128 / kShares), r_hi = r_lo + 128 / kShares;
    const bool pools = h % p.G == 0;
    const long long chunk_rows = (long long)p.kv_tpc * 128;
    float s0 = 0.f, s1 = 0.f;
    int seg = -1;
    long long next_lo = 0;  // first row of segment seg + 1
    auto flush = [&]() {
      if (seg >= 0) {
        const int k = chunk - (int)(seg_lo(seg, p.N, m) / chunk_rows);
        float2* dst = reinterpret_cast<float2*>(
            p.kpart + (((size_t)bhk * m + seg) * p.kparts + k * kShares + share) * D + box * 64);
        dst[lane] = make_float2(s0, s1);
      }
      s0 = s1 = 0.f;
    };
    bool ok = true;
    for (int it = 0; it < 2 * n; ++it) {
      const int s = it % ST;
      ok = __all_sync(0xffffffffu, mbar_wait_inl(bar_full(s), (uint32_t)(it / ST) & 1u, wc));
      if (!ok) break;
      if (pools && (it & 1) == 0) {
        const long long g0 = (long long)(j0 + it / 2) * 128;
        const int rows = (int)min((long long)r_hi, (long long)p.N - g0);  // this share's end
        if (seg < 0 && r_lo < rows) {
          seg = (int)(((g0 + r_lo + 1) * m - 1) / p.N);  // the segment holding row g0 + r_lo
          next_lo = seg_lo(seg + 1, p.N, m);
        }
        const uint32_t base = slot(s) + box * Cfg::kBoxBytes + (uint32_t)(lane & 3) * 4u;
        // row r of the 128-byte-swizzled box: 16-byte chunk (lane / 4) ^ (r % 8)
        auto word = [&](int r) {
          uint32_t v;
          asm volatile("ld.shared.b32 %0, [%1];"
                       : "=r"(v)
                       : "r"(base + (uint32_t)r * 128u + (uint32_t)(((lane >> 2) ^ (r & 7)) << 4)));
          return v;
        };
        int r = r_lo;
        while (r < rows) {
          // segments may also have ended in rows of the other shares: each
          // one passed gets its (possibly empty) sum written
          while (g0 + r >= next_lo) {
            flush();
            ++seg;
            next_lo = seg_lo(seg + 1, p.N, m);
          }
          const int r_end = (int)min((long long)rows, next_lo - g0);  // rows of this segment
          float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
          for (; r + 8 <= r_end; r += 8) {
            uint32_t v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = word(r + e);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              a0 += __uint_as_float(v[e] << 16);
              a1 += __uint_as_float(v[e] & 0xffff0000u);
              b0 += __uint_as_float(v[e + 1] << 16);
              b1 += __uint_as_float(v[e + 1] & 0xffff0000u);
            }
          }
          for (; r < r_end; ++r) {
            const uint32_t v = word(r);
            a0 += __uint_as_float(v << 16);
            a1 += __uint_as_float(v & 0xffff0000u);
          }
          s0 += a0 + b0;
          s1 += a1 + b1;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty(s));
    }
    if (ok && pools) flush();
  } else if (warp < nw) {
    // ------------------------------------------------------------ softmax warps
    const int row = warp * 32 + lane;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float c = p.scale_log2;
    float mu = -INFINITY, l = 0.f;
    bool ok = true;
    for (int jj = 0; jj < n; ++jj) {
      const int bb = jj & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_inl(bar_s(bb), (uint32_t)(jj >> 1) & 1u, wc));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = tmem_base + lane_off + (uint32_t)(bb * 128);
      float x[128];
      {
        uint32_t r[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, r[q]);
        tmem_ld_wait();
        const int lim = p.N - (j0 + jj) * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            x[q * 32 + e] = (q * 32 + e < lim) ? __uint_as_float(r[q][e]) * c : -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int e = 0; e < 128; ++e) mx = fmaxf(mx, x[e]);
      // O += P_{jj-2} V_{jj-2} (observed in turn; see above)
      if (jj >= 2) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait_inl(bar_pv(jj & 1), (uint32_t)((jj - 2) >> 1) & 1u, wc));
        if (!ok) break;
      }
      const bool raise = mx > mu + 8.f;
      if (__any_sync(0xffffffffu, raise)) {
        const float mnew = raise ? mx : mu;
        if (jj > 0) {
          // O += P_{jj-1} V_{jj-1} must have landed before O is rescaled
          ok = __all_sync(0xffffffffu, mbar_wait_inl(bar_pv((jj - 1) & 1),
                                                     (uint32_t)((jj - 1) >> 1) & 1u, wc));
          if (!ok) break;
          tc_fence_after();
          const float f = ex2_approx(mu - mnew);
          const uint32_t tO = tmem_base + lane_off + 256u;
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t r[32];
            tmem_ld32(tO + q * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
            tmem_st32(tO + q * 32, r);
          }
          tmem_st_wait();
          l *= f;
        }
        mu = mnew;
      }
      uint32_t pk[64];
      float ls = 0.f;
#pragma unroll
      for (int e = 0; e < 128; e += 2) {
        const float p0 = ex2_approx(x[e] - mu), p1 = ex2_approx(x[e + 1] - mu);
        ls += p0 + p1;
        pk[e / 2] = pack_bf16x2(p0, p1);
      }
      l += ls;
      tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p(bb));
    }
    // every MMA of the CTA, the last P V included, has completed
    if (ok && n > 0) ok = __all_sync(0xffffffffu, mbar_wait_inl(bar_done(), 0, wc));
    if (ok && n > 0) {
      tc_fence_after();
      const size_t prow = ((size_t)bh * p.kv_chunks + chunk) * m + row;
      float4* dst = reinterpret_cast<float4*>(p.kv_o + prow * D);
      const uint32_t tO = tmem_base + lane_off + 256u;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t r[32];
        tmem_ld32(tO + q * 32, r);
        tmem_ld_wait();
        if (row < m) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[q * 8 + e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                                         __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
        }
      }
      if (row < m) *reinterpret_cast<float2*>(p.kv_ml + prow * 2) = make_float2(mu, l);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// ============================================================ 4: merge
// grid (m D / 4 / (256 / R), B*Hq), 256 threads = R chunk groups x 256 / R
// (row, column quad) pairs: landmark row i of head bh, columns 4g .. 4g + 3,
// W_i = sum_c 2^(mu_c - M) O_c / sum_c 2^(mu_c - M) l_c over the key chunks
// (M the largest mu_c), each sum kept as four partial sums over the chunks
// c = r mod 4 (r = 0..3) in order, added in that order at the end.  R = 1: one
// thread keeps all four (few chunks); R = 4: group r keeps the r-th and the
// four meet in shared memory (many chunks, four times the threads on them).
template <int D, int R>
__global__ void __launch_bounds__(kNysSmallThreads) nys_merge_kernel(const NysParams p) {
  static_assert(R == 1 || R == 4, "one or four chunk groups");
  constexpr int G = D / 4, PAIRS = kNysSmallThreads / R;
  __shared__ float4 part[R == 4 ? 4 : 1][PAIRS];
  __shared__ float dpart[R == 4 ? 4 : 1][PAIRS];
  const int pr = (int)threadIdx.x % PAIRS, r = (int)threadIdx.x / PAIRS;
  const int idx = (int)blockIdx.x * PAIRS + pr;
  const int m = p.m, C = p.kv_chunks;
  const int i = idx / G, d0 = (idx % G) * 4, bh = (int)blockIdx.y;
  const bool live = i < m;
  const int il = live ? i : 0;
  const float2* ml = reinterpret_cast<const float2*>(p.kv_ml) + (size_t)bh * C * m + il;
  const float4* ob = reinterpret_cast<const float4*>(p.kv_o + ((size_t)bh * C * m + il) * D + d0);
  const size_t ostep = (size_t)m * G;  // one chunk, in float4
  __shared__ float mpart[R == 4 ? 4 : 1][PAIRS];
  float M = -INFINITY;
  if constexpr (R == 1) {
#pragma unroll 4
    for (int c = 0; c < C; ++c) M = fmaxf(M, ml[(size_t)c * m].x);
  } else {  // each group the maximum over its chunks, then the four meet
#pragma unroll 4
    for (int c = r; c < C; c += 4) M = fmaxf(M, ml[(size_t)c * m].x);
    mpart[r][pr] = M;
    __syncthreads();
    M = fmaxf(fmaxf(mpart[0][pr], mpart[1][pr]), fmaxf(mpart[2][pr], mpart[3][pr]));
  }
  auto step = [&](int c, float4& nr, float& dr) {
    const float2 v = ml[(size_t)c * m];
    const float4 o = ob[(size_t)c * ostep];
    const float f = exp2f(v.x - M);
    nr.x = fmaf(f, o.x, nr.x);
    nr.y = fmaf(f, o.y, nr.y);
    nr.z = fmaf(f, o.z, nr.z);
    nr.w = fmaf(f, o.w, nr.w);
    dr = fmaf(f, v.y, dr);
  };
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 n0 = z, n1 = z, n2 = z, n3 = z;
  float e0 = 0.f, e1 = 0.f, e2 = 0.f, e3 = 0.f;
  if constexpr (R == 1) {
    int c = 0;
    for (; c + 3 < C; c += 4) {
      step(c, n0, e0);
      step(c + 1, n1, e1);
      step(c + 2, n2, e2);
      step(c + 3, n3, e3);
    }
    if (c < C) step(c, n0, e0);
    if (c + 1 < C) step(c + 1, n1, e1);
    if (c + 2 < C) step(c + 2, n2, e2);
  } else {
#pragma unroll 4
    for (int c = r; c < C; c += 4) step(c, n0, e0);
    part[r][pr] = n0;
    dpart[r][pr] = e0;
    __syncthreads();
    if (r != 0) return;
    n0 = part[0][pr];
    n1 = part[1][pr];
    n2 = part[2][pr];
    n3 = part[3][pr];
    e0 = dpart[0][pr];
    e1 = dpart[1][pr];
    e2 = dpart[2][pr];
    e3 = dpart[3][pr];
  }
  if (!live) return;
  const float dn = e0 + e1 + e2 + e3;
  *reinterpret_cast<float4*>(p.w + ((size_t)bh * m + i) * D + d0) =
      make_float4((n0.x + n1.x + n2.x + n3.x) / dn, (n0.y + n1.y + n2.y + n3.y) / dn,
                  (n0.z + n1.z + n2.z + n3.z) / dn, (n0.w + n1.w + n2.w + n3.w) / dn);
}

// ============================================================ 6: output pass
template <int D>
struct NysOutCfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kBoxBytes = 128 * 128;
  static constexpr int kBoxes = D / 64;
  static constexpr int kStages = (D == 128) ? 3 : 6;  // Q tiles in flight
  static constexpr int kQOff = 0;
  static constexpr int kKtOff = kStages * kTileBytes;  // Kt hi, lo: up to 2 x 64 rows x D
  static constexpr int kYOff = kKtOff + 128 * D * 2;    // Y hi, lo: up to 2 x 64 rows x D
  static constexpr int kStOff = kYOff + 128 * D * 2;    // two O staging tiles (TMA store)
  static constexpr int kBarOff = kStOff + 2 * kTileBytes;
  // barriers: q_full[ST], q_empty[ST], ky_full, ky_empty, s_full[2], p_full[2],
  // o_full[2], o_free[2], done
  static constexpr int kNumBars = 2 * kStages + 11;
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "more shared memory than one CTA may have");
  static constexpr int kThreads = 320;  // two groups of 4 softmax warps, producer, MMA
  // S0, S1 (64 columns each), O0, O1 (D each)
  static constexpr uint32_t kTmemCols = (128 + 2 * D) <= 256 ? 256 : 512;
};

// Persistent: CTA c owns query tiles [c*W/G, (c+1)*W/G) of the B*Hq*T tiles,
// head-major, so consecutive tiles mostly share Kt and Y.  Warps 0-3 and 4-7
// are two groups that take the CTA's tiles in turn (group g the tiles t with
// t % 2 == g, TMEM buffers S_g, O_g, staging tile g): thread = query row =
// TMEM lane, softmax over the landmarks, then the epilogue of the same tile,
// while the other group works on its neighbour.  Warp 8: TMA (Kt and Y on a
// head change, Q tiles through a ring); warp 9: MMA, in the order S_0, S_1,
// O_0 = P_0 Y, S_2, O_1 = P_1 Y, ... with the previous head's last P Y issued
// before Kt and Y are replaced.
template <int D>
__global__ void __launch_bounds__(320, 1)
    nys_out_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kt,
                   const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ CUtensorMap tm_o,
                   const NysParams p) {
  using Cfg = NysOutCfg<D>;
  constexpr int ST = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_base & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_base + pad;
  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = (int)(threadIdx.x & 31);

  const uint32_t bar0 = sbase + Cfg::kBarOff;
  auto bar_qf = [&](int s) { return bar0 + 8u * s; };
  auto bar_qe = [&](int s) { return bar0 + 8u * (ST + s); };
  auto bar_kyf = [&]() { return bar0 + 8u * (2 * ST); };
  auto bar_kye = [&]() { return bar0 + 8u * (2 * ST + 1); };
  auto bar_s = [&](int b) { return bar0 + 8u * (2 * ST + 2 + b); };
  auto bar_p = [&](int b) { return bar0 + 8u * (2 * ST + 4 + b); };
  auto bar_of = [&](int b) { return bar0 + 8u * (2 * ST + 6 + b); };
  auto bar_oe = [&](int b) { return bar0 + 8u * (2 * ST + 8 + b); };
  auto bar_done = [&]() { return bar0 + 8u * (2 * ST + 10); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kBarOff + Cfg::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(bar_qf(s), 1);
      mbar_init(bar_qe(s), 1);
    }
    mbar_init(bar_kyf(), 1);
    mbar_init(bar_kye(), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_s(b), 1);
      mbar_init(bar_p(b), 4);
      mbar_init(bar_of(b), 1);
      mbar_init(bar_oe(b), 4);
    }
    mbar_init(bar_done(), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kt);
    tma_prefetch_desc(&tm_y);
    tma_prefetch_desc(&tm_o);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int T = p.num_kv_tiles;
  const long long total = (long long)p.B * p.Hq * T;
  const long long w0 = total * blockIdx.x / gridDim.x, w1 = total * (blockIdx.x + 1) / gridDim.x;
  const int nt = (int)(w1 - w0);
  const int m = p.m, mp = p.mp;
  const WaitCtl wc{p.timeout_ns, p.err, abort_flag};

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int cur = -1;
      uint32_t nky = 0;
      bool ok = true;
      int t = 0;
      for (; t < nt; ++t) {
        const long long w = w0 + t;
        const int bh = (int)(w / T), qt = (int)(w % T);
        if (bh != cur) {
          if (nky > 0 && !(ok = mbar_wait_inl(bar_kye(), (nky - 1) & 1u, wc))) break;
          const int bhk = (bh / p.Hq) * p.Hkv + (bh % p.Hq) / p.G;
          // hi then lo, each as D/64 boxes of mp rows
          mbar_arrive_expect_tx(bar_kyf(), 4u * (uint32_t)mp * D * 2);
          for (int u = 0; u < 2; ++u)
            for (int c = 0; c < Cfg::kBoxes; ++c) {
              const uint32_t off = (uint32_t)((u * Cfg::kBoxes + c) * mp * 128);
              tma_load_3d(sbase + Cfg::kKtOff + off, &tm_kt, bar_kyf(), c * 64, u * mp, bhk);
              tma_load_3d(sbase + Cfg::kYOff + off, &tm_y, bar_kyf(), c * 64, u * mp, bh);
            }
          ++nky;
          cur = bh;
        }
        const int s = t % ST;
        if (!(ok = mbar_wait_inl(bar_qe(s), ((uint32_t)(t / ST) & 1u) ^ 1u, wc))) break;
        mbar_arrive_expect_tx(bar_qf(s), Cfg::kTileBytes);
        for (int c = 0; c < Cfg::kBoxes; ++c)
          tma_load_3d(sbase + Cfg::kQOff + s * Cfg::kTileBytes + c * Cfg::kBoxBytes, &tm_q, bar_qf(s),
                      c * 64, qt * 128, bh);
      }
      if (!ok) {
        for (int f = (t > ST ? t - ST : 0); f < t; ++f)
          mbar_wait_drain_inl(bar_qf(f % ST), (uint32_t)(f / ST) & 1u, wc);
        if (nky > 0) mbar_wait_drain_inl(bar_kyf(), (nky - 1) & 1u, wc);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = make_idesc_bf16(128, (uint32_t)mp, 0, 0);
      constexpr uint32_t kIdescO = make_idesc_bf16(128, D, 1, 0);
      constexpr uint32_t kHi = sdesc_sw128_hi(1024);
      const uint32_t tS[2] = {tmem_base, tmem_base + 64};
      const uint32_t tO[2] = {tmem_base + 128, tmem_base + 128 + D};
      const uint32_t half = (uint32_t)(Cfg::kBoxes * mp * 128);  // hi tile -> lo tile
      const uint32_t kth_lo = sdesc_sw128_lo(sbase + Cfg::kKtOff, 16);
      const uint32_t ktl_lo = sdesc_sw128_lo(sbase + Cfg::kKtOff + half, 16);
      const uint32_t yh_lo = sdesc_sw128_lo(sbase + Cfg::kYOff, (uint32_t)mp * 128);
      const uint32_t yl_lo = sdesc_sw128_lo(sbase + Cfg::kYOff + half, (uint32_t)mp * 128);
      int pv_next = 0;
      bool ok = true;
      auto issue_pv = [&](int u) -> bool {
        if (u != pv_next) return true;
        if (!mbar_wait_inl(bar_p(u & 1), (uint32_t)(u >> 1) & 1u, wc)) return false;
        if (u >= 2 && !mbar_wait_inl(bar_oe(u & 1), (uint32_t)((u - 2) >> 1) & 1u, wc)) return false;
        tc_fence_after();
        // O = P Y_hi + P Y_lo
        for (int kk = 0; kk < mp / 16; ++kk)
          mma_ts_w(tO[u & 1], tS[u & 1] + kk * 8, yh_lo, (uint32_t)((kk * 2048) >> 4), kHi, kIdescO,
                   kk > 0 ? 1u : 0u);
        for (int kk = 0; kk < mp / 16; ++kk)
          mma_ts_w(tO[u & 1], tS[u & 1] + kk * 8, yl_lo, (uint32_t)((kk * 2048) >> 4), kHi, kIdescO,
                   1u);
        mma_commit(bar_of(u & 1));
        ++pv_next;
        return true;
      };
      int cur = -1;
      uint32_t nky = 0;
      for (int t = 0; t < nt && ok; ++t) {
        const int bh = (int)((w0 + t) / T);
        if (bh != cur) {
          if (t > 0) {
            if (!(ok = issue_pv(t - 1))) break;
            mma_commit(bar_kye());
          }
          if (!(ok = mbar_wait_inl(bar_kyf(), nky & 1u, wc))) break;
          ++nky;
          cur = bh;
        }
        const int s = t % ST;
        if (!(ok = mbar_wait_inl(bar_qf(s), (uint32_t)(t / ST) & 1u, wc))) break;
        tc_fence_after();
        const uint32_t q_lo = sdesc_sw128_lo(sbase + Cfg::kQOff + s * Cfg::kTileBytes, 16);
        // S = Q Kt_hi^T + Q Kt_lo^T
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t a_off = (uint32_t)(((kk / 4) * Cfg::kBoxBytes + (kk % 4) * 32) >> 4);
          const uint32_t b_off = (uint32_t)(((kk / 4) * mp * 128 + (kk % 4) * 32) >> 4);
          mma_ss_w(tS[t & 1], q_lo, a_off, kth_lo, b_off, kHi, idS, kk > 0 ? 1u : 0u);
          mma_ss_w(tS[t & 1], q_lo, a_off, ktl_lo, b_off, kHi, idS, 1u);
        }
        mma_commit(bar_s(t & 1));
        mma_commit(bar_qe(s));
        if (t > 0 && !(ok = issue_pv(t - 1))) break;
      }
      if (ok && nt > 0) ok = issue_pv(nt - 1);
      mma_commit(bar_done());
      if (!ok) mbar_wait_drain_inl(bar_done(), 0, wc);
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int g = warp >> 2, wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t bar_id = 1u + (uint32_t)g;  // named barrier of the group (128 threads)
    const bool leader = threadIdx.x == (unsigned)(g * 128);
    const float c = p.scale_log2;
    const uint32_t tS = tmem_base + lane_off + (uint32_t)(g * 64);
    const uint32_t tO = tmem_base + lane_off + 128u + (uint32_t)(g * D);
    // staging tile g, row `row` (128-byte swizzle, the TMA layout)
    const uint32_t st_base = sbase + Cfg::kStOff + (uint32_t)g * Cfg::kTileBytes;
    const uint32_t st_row = st_base + (uint32_t)row * 128u;
    // O_u / l -> bf16 -> staging tile -> TMA store (rows past N are left out).
    // The leader first waits until its previous store has read the tile; every
    // wait outcome is ANDed over the group's warps at its named barrier, so that
    // they leave together.
    auto epilogue = [&](int u, float linv) -> bool {
      const bool got = __all_sync(0xffffffffu, mbar_wait_inl(bar_of(g), (uint32_t)(u >> 1) & 1u, wc));
      if (leader) bulk_wait_read_all();
      if (!named_bar_and(bar_id, 128, got)) return false;
      tc_fence_after();
      const long long w = w0 + u;
      const int bh = (int)(w / T), qt = (int)(w % T);
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t r[32];
        tmem_ld32(tO + q * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t x0 = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * linv, __uint_as_float(r[8 * v + 1]) * linv);
          const uint32_t x1 = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * linv, __uint_as_float(r[8 * v + 3]) * linv);
          const uint32_t x2 = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * linv, __uint_as_float(r[8 * v + 5]) * linv);
          const uint32_t x3 = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * linv, __uint_as_float(r[8 * v + 7]) * linv);
          const int chunk = (q & 1) * 4 + v;  // 16-byte chunk of the 128-byte row
          const uint32_t addr = st_row + (uint32_t)(q >> 1) * Cfg::kBoxBytes +
                                (uint32_t)((chunk ^ (row & 7)) * 16);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x0), "r"(x1),
                       "r"(x2), "r"(x3)
                       : "memory");
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_oe(g));
      fence_proxy_async_smem();
      named_bar_sync(bar_id, 128);
      if (leader) {
        for (int cb = 0; cb < Cfg::kBoxes; ++cb)
          tma_store_3d(&tm_o, st_base + cb * Cfg::kBoxBytes, cb * 64, qt * 128, bh);
        bulk_commit();
      }
      return true;
    };
    bool ok = true;
    for (int t = g; t < nt && ok; t += 2) {
      ok = named_bar_and(bar_id, 128,
                         __all_sync(0xffffffffu, mbar_wait_inl(bar_s(g), (uint32_t)(t >> 1) & 1u, wc)));
      if (!ok) break;
      tc_fence_after();
      float x[64];
      {
        uint32_t r[4][16];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q * 16 < mp) tmem_ld16(tS + q * 16, r[q]);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int e = 0; e < 16; ++e)
            x[q * 16 + e] = (q * 16 + e < m) ? __uint_as_float(r[q][e]) * c : -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int e = 0; e < 64; ++e) mx = fmaxf(mx, x[e]);
      uint32_t pk[32];
      float l = 0.f;
#pragma unroll
      for (int e = 0; e < 64; e += 2) {
        const float p0 = ex2_approx(x[e] - mx), p1 = ex2_approx(x[e + 1] - mx);
        l += p0 + p1;
        pk[e / 2] = pack_bf16x2(p0, p1);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q * 16 < mp) tmem_st8(tS + q * 8, *reinterpret_cast<uint32_t(*)[8]>(&pk[q * 8]));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p(g));
      ok = epilogue(t, 1.f / l);
    }
    if (leader) bulk_wait_all();
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
