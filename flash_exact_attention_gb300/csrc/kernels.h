// kernels.h -- internal interface between the C-ABI layer (attn_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

// Forward kernel parameters (everything but the tensor maps).
struct FwdParams {
  void* o;              // bf16 [B, Hq, N, D]
  float* lse;           // fp32 [B, Hq, N]
  int B, Hq, Hkv, N;
  int G;                // Hq / Hkv
  int num_qblocks;      // ceil(ceil(N / 128) / 2): CTAs per (batch, head)
  int kvsplit;          // one query tile per CTA, key range split over the two slots
  int num_kv_tiles;     // ceil(N / 128)
  float scale_log2;     // scale * log2(e)
  uint64_t timeout_ns;  // limit of every device-side wait
  unsigned int* err;    // device error word
  int ctas;             // persistent CTAs of the dense forward (0: one CTA per work unit)
  // Stieltjes forward only (lse then holds the pole): the softmax scale and
  // the number of Newton steps.
  float scale;
  int steps;
  // Packed variable-length forward only: sequence b is tokens
  // cu_seqlens[b] .. cu_seqlens[b+1]-1 of `total`; N above is max_seqlen.
  const int* cu_seqlens;
  int total;
};

// Nystrom attention forward (six kernels; nys_kernel.cuh).  Landmark rows are
// padded to mp (m rounded up to a multiple of 16, at least 16) wherever they
// are a tensor-core operand dimension.
struct NysParams {
  const void* q;        // bf16 [B, Hq, N, D]
  const void* k;        // bf16 [B, Hkv, N, D]
  void* o;              // bf16 [B, Hq, N, D]
  int B, Hq, Hkv, N, G;
  int m, mp;            // landmarks, and m padded for the tensor cores
  int iters;            // Newton-Schulz steps
  float kappa;          // ridge target condition number (0 = no ridge)
  float scale;          // score scale
  float scale_log2;     // scale * log2(e)
  int num_kv_tiles;     // ceil(N / 128)
  // Q pooling: partial segment sums [B*Hq, m, pool_splits, D]
  int pool_splits;
  float* pool_part;
  float* qt32;          // fp32 [B*Hq, m, D]: Qt
  // bf16 hi/lo pairs (x = hi + lo, rows >= m zero) of the tensor-core operands:
  uint16_t* qt16;       // [B*Hq, 2, 128, D]: Qt as two 128-row A tiles
  uint16_t* kt16;       // [B*Hkv, 2, mp, D]: Kt
  uint16_t* y16;        // [B*Hq, 2, mp, D]: Y = pinv(A2) W
  // split-key pass: chunk c of a head covers key tiles [c*kv_tpc, (c+1)*kv_tpc)
  int kv_chunks, kv_tpc;
  float* kv_o;          // fp32 [B*Hq, kv_chunks, m, D]: unnormalised partial W
  float* kv_ml;         // fp32 [B*Hq, kv_chunks, m, 2]: row max (log2 units), row sum
  float* w;             // fp32 [B*Hq, m, D]: W = softmax(scale Qt K^T) V
  // K segment sums from the split-key pass: slot k of segment i holds the sum
  // over its rows in chunk floor(first row of i / chunk rows) + k
  int kparts;
  float* kpart;         // fp32 [B*Hkv, m, kparts, D]
  int out_ctas;         // persistent CTAs of the output pass
  uint64_t timeout_ns;
  unsigned int* err;
};

// Enqueues the six Nystrom kernels (tq, to: q and o; tk, tv: k and v; tqt,
// tkt, ty: the landmark and Y operand tiles in scratch).
cudaError_t launch_nys_d64(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tqt, const CUtensorMap& tkt, const CUtensorMap& ty,
                           const CUtensorMap& to, const NysParams& p, cudaStream_t stream);
cudaError_t launch_nys_d128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tqt, const CUtensorMap& tkt, const CUtensorMap& ty,
                            const CUtensorMap& to, const NysParams& p, cudaStream_t stream);

// Backward parameters of the main kernel (everything but the tensor maps).
struct BwdParams {
  void* dk;             // bf16 [B, Hkv, N, D]
  void* dv;             // bf16 [B, Hkv, N, D]
  float* dq_acc;        // fp32 [B*Hq, Npad, D], zeroed by bwd_preprocess
  const float* lse2;    // fp32 [B*Hq, Npad]: LSE * log2(e); +inf for rows >= N
  const float* delta;   // fp32 [B*Hq, Npad]: rowsum(dO * O); 0 for rows >= N
  int B, Hq, Hkv, N;
  int Npad;             // N rounded up to a multiple of 128
  int G;                // Hq / Hkv
  int num_kv_tiles;     // ceil(N / 128)
  float scale;          // softmax scale
  float scale_log2;     // scale * log2(e)
  uint64_t timeout_ns;
  unsigned int* err;
  // Query heads of a group are split over `gsplit` CTAs (1 = one CTA owns the
  // whole group and writes dK/dV directly).  With gsplit > 1 each CTA adds its
  // fp32 dK/dV partials into dk_acc / dv_acc ([B*Hkv, Npad, D], zeroed by the
  // preprocess, converted by the postprocess).
  int gsplit;
  float* dk_acc;
  float* dv_acc;
  // Causal CTA order.  The key tiles are split into `jchunks` ranges run one
  // after the other (heaviest first); within a range the work units (one
  // (batch, kv head[, group slice]) each) go in bands of `band`, key tile j
  // ascending inside a band.  With many units, bands keep the CTAs resident
  // at one time on the Q, dO and dQ rows of a few heads (L2) instead of all
  // of them (HBM); the ranges keep the heaviest CTAs of the last band from
  // starting at the very end.  band = all units, jchunks = 1: plain j order.
  int band;
  int jchunks;
  // Packed variable-length backward only (else nullptr / 0): sequence b is
  // tokens cu_seqlens[b] .. cu_seqlens[b+1]-1 of q/o/dO/dQ [total, Hq, D] and
  // k/v/dK/dV [total, Hkv, D]; N is max_seqlen, and lse2/delta are
  // [B*Hq, Npad] with rows past a sequence's end at +inf / 0.
  const int* cu_seqlens;
  int total;
};

// Device pointers of the backward's fp32 scratch.
struct BwdScratch {
  float* dq_acc;
  float* lse2;
  float* delta;
  float* dk_acc;  // only with gsplit > 1
  float* dv_acc;
};

// Causal CTA order (BwdParams::band, ::jchunks) for `units` work units of
// `tiles` key tiles each, whose query-side rows (Q, dO bf16 and the fp32 dQ
// accumulator) take `unit_bytes`.
void bwd_order(BwdParams* p, long long units, int tiles, double unit_bytes, int sms);

// Bytes of fp32 scratch the backward needs for these sizes.
size_t bwd_scratch_bytes(int B, int Hq, int N, int D);

// Bytes of fp32 scratch for a given group split (adds the dK/dV accumulators).
size_t bwd_scratch_bytes_split(int B, int Hq, int Hkv, int N, int D, int gsplit);

// Splits one scratch block of bwd_scratch_bytes() into its three arrays.
BwdScratch carve_scratch(void* base, int B, int Hq, int N, int D);

// Same, with the dK/dV accumulators of a group split after them.
BwdScratch carve_scratch_split(void* base, int B, int Hq, int Hkv, int N, int D, int gsplit);

// Host-side validation and set-up of a backward call (tensor maps and every
// parameter except the scratch pointers).  Returns ATTN_OK, an error code, or
// -1 when there is nothing to compute.
int bwd_prepare(const void* q, const void* k, const void* v, const void* o, const float* lse,
                int B, int Hq, int Hkv, int N, int D, float scale, const void* dout, void* dq,
                void* dk, void* dv, BwdParams* p, CUtensorMap* tq, CUtensorMap* tk,
                CUtensorMap* tv, CUtensorMap* tdo, bool allow_split = false,
                bool f16 = false);

// Enqueues the three backward kernels with the scratch already in `p`.
int bwd_launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& tdo, const BwdParams& p, const void* o, const void* dout,
               const float* lse, void* dq, int D, int causal, cudaStream_t s,
               bool f16 = false, bool det = false);

// Enqueues preprocess, main and postprocess kernels of the backward.
cudaError_t launch_bwd_d64(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, const BwdParams& p, const void* o,
                           const void* dout, const float* lse, void* dq, bool causal,
                           cudaStream_t stream);
cudaError_t launch_bwd_d128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdParams& p, const void* o,
                            const void* dout, const float* lse, void* dq, bool causal,
                            cudaStream_t stream);
// The deterministic backward (bf16): dK/dV kernel without dQ, then dQ per query tile.
cudaError_t launch_bwd_det_d64(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& tdo, const BwdParams& p, const void* o,
                               const void* dout, const float* lse, void* dq, bool causal,
                               cudaStream_t stream);
cudaError_t launch_bwd_det_d128(const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                                const void* o, const void* dout, const float* lse, void* dq,
                                bool causal, cudaStream_t stream);
// The same for fp16 inputs and gradients.
cudaError_t launch_bwd_d64_f16(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& tdo, const BwdParams& p, const void* o,
                               const void* dout, const float* lse, void* dq, bool causal,
                               cudaStream_t stream);
cudaError_t launch_bwd_d128_f16(const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                                const void* o, const void* dout, const float* lse, void* dq,
                                bool causal, cudaStream_t stream);

// Host helpers shared by the entry points (attn_api.cu).
int validate_shape(int B, int Hq, int Hkv, int N, int D, float scale);
int device_setup(int* dev_out, unsigned int** err_out);
int device_sm_count(int dev);
int encode_tile_map(CUtensorMap* map, const void* base, int D, int N, int BH, bool f16 = false,
                    int box_rows = 128);
int encode_f32_rows_map(CUtensorMap* map, const void* base, int D, int rows, int BH);
int encode_packed_map(CUtensorMap* map, const void* base, int D, int H, int total,
                      bool f32 = false);
uint64_t wait_timeout_ns();
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Each launcher enqueues one forward kernel; returns the launch's cudaError_t.
cudaError_t launch_fwd_d64(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const FwdParams& p, bool causal, cudaStream_t stream);
cudaError_t launch_fwd_d128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, bool causal, cudaStream_t stream);
cudaError_t launch_fwd_d64_f16(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const FwdParams& p, bool causal, cudaStream_t stream);
cudaError_t launch_fwd_d128_f16(const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const FwdParams& p, bool causal,
                                cudaStream_t stream);

// Packed variable-length forward (bf16), one kernel per call.
cudaError_t launch_fwd_varlen_d64(const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const FwdParams& p, bool causal,
                                  cudaStream_t stream);
cudaError_t launch_fwd_varlen_d128(const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const FwdParams& p, bool causal,
                                   cudaStream_t stream);

// fp16 versions of the packed variable-length forward.
cudaError_t launch_fwd_varlen_d64_f16(const CUtensorMap& tq, const CUtensorMap& tk,
                                      const CUtensorMap& tv, const FwdParams& p, bool causal,
                                      cudaStream_t stream);
cudaError_t launch_fwd_varlen_d128_f16(const CUtensorMap& tq, const CUtensorMap& tk,
                                       const CUtensorMap& tv, const FwdParams& p, bool causal,
                                       cudaStream_t stream);

// Packed variable-length backward (bf16; _f16: fp16): preprocess, main kernel, dQ
// conversion.  tdq is the packed fp32 map of p.dq_acc [total, Hq, D].
cudaError_t launch_bwd_varlen_d64(const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const CUtensorMap& tdo,
                                  const CUtensorMap& tdq, const BwdParams& p, const void* o,
                                  const void* dout, const float* lse, void* dq, bool causal,
                                  cudaStream_t stream);
cudaError_t launch_bwd_varlen_d128(const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const CUtensorMap& tdo,
                                   const CUtensorMap& tdq, const BwdParams& p, const void* o,
                                   const void* dout, const float* lse, void* dq, bool causal,
                                   cudaStream_t stream);
cudaError_t launch_bwd_varlen_d64_f16(const CUtensorMap& tq, const CUtensorMap& tk,
                                      const CUtensorMap& tv, const CUtensorMap& tdo,
                                      const CUtensorMap& tdq, const BwdParams& p, const void* o,
                                      const void* dout, const float* lse, void* dq, bool causal,
                                      cudaStream_t stream);
cudaError_t launch_bwd_varlen_d128_f16(const CUtensorMap& tq, const CUtensorMap& tk,
                                       const CUtensorMap& tv, const CUtensorMap& tdo,
                                       const CUtensorMap& tdq, const BwdParams& p, const void* o,
                                       const void* dout, const float* lse, void* dq, bool causal,
                                       cudaStream_t stream);

// Stieltjes attention forward (order 2 or 4), one kernel per call.
cudaError_t launch_stj_d64(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const FwdParams& p, bool causal, int order, cudaStream_t stream);
cudaError_t launch_stj_d128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, bool causal, int order, cudaStream_t stream);

// Entry points behind the C ABI (attn_api.cu, bwd.cu).
int bwd_entry(const void* q, const void* k, const void* v, const void* o, const float* lse, int B,
              int Hq, int Hkv, int N, int D, int causal, float scale, void* stream,
              const void* dout, void* dq, void* dk, void* dv, bool f16 = false,
              bool det = false);
int fwd_entry(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
              int Hkv, int N, int D, int causal, float scale, void* stream, bool f16 = false);
int bwd_varlen_entry(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const int* cu_seqlens, int B, int Hq, int Hkv, int total,
                     int max_seqlen, int D, int causal, float scale, void* stream,
                     const void* dout, void* dq, void* dk, void* dv, bool f16 = false);
int fwd_varlen_entry(const void* q, const void* k, const void* v, void* o, float* lse,
                     const int* cu_seqlens, int B, int Hq, int Hkv, int total, int max_seqlen,
                     int D, int causal, float scale, void* stream, bool f16 = false);

}  // namespace attn
