/*
 * attn.h -- C ABI of libattn.so: exact flash attention on one NVIDIA GB300 (sm_103a).
 *
 * Operation (forward).  For every batch b, query head h and query row i,
 *     O_i   = sum_j softmax_j(scale * q_i . k_j) v_j
 *     LSE_i = ln sum_j exp(scale * q_i . k_j)
 * over the allowed keys j (all N keys, or j <= i when causal), computed
 * flash-style: K/V stream through on-chip tiles with a running row maximum
 * and running row sum, and the N x N score matrix is never stored.
 *   - exact attention and the tiling: "From-scratch CUDA attention kernel
 *     reaches 94.4% of FlashAttention-4 on NVIDIA B200", section "How the
 *     kernel partitions its work"; FlashNystrom page, "Scope";
 *   - the running max / running sum: FlashStieltjes page, "The challenge";
 *   - MHA/GQA/MQA (Hq a multiple of Hkv), causal with the upper triangle
 *     skipped, ragged N, head dims 64 and 128, shapes (B,H,N,D):
 *     FlashAttention for Tesla P100 page, "What it supports", "Quick start";
 *   - LSE, the tiled softmax's running log-sum-exp state: FlashNystrom page,
 *     "Scope" and "References".
 * Query head h reads key/value head h / (Hq / Hkv).
 *
 * Operation (backward).  Given dO = dL/dO, with P recomputed from LSE:
 *     Delta_i = dO_i . O_i,   dS_ij = P_ij (dO_i . v_j - Delta_i)
 *     dQ_i = scale sum_j dS_ij k_j
 *     dK_j = scale sum_{h in group} sum_i dS_ij q_i
 *     dV_j = sum_{h in group} sum_i P_ij dO_i
 *   (FlashAttention for Tesla P100 page, "Documentation": dS = P(dP - D) is a
 *   cancellation and is kept in fp32; fp32 gradient accumulation: "What it
 *   supports".)
 *
 * Common conventions for every entry point.
 *   - All tensor pointers are DEVICE pointers owned by the caller, 16-byte
 *     aligned, to contiguous row-major arrays:
 *       q, o, dout, dq : bf16 [B, Hq, N, D]
 *       k, v, dk, dv   : bf16 [B, Hkv, N, D]
 *       lse            : fp32 [B, Hq, N]   (natural log)
 *     bf16 means IEEE bfloat16 bit patterns (uint16 storage).
 *   - Outputs must not alias inputs or each other.
 *   - D must be 64 or 128; Hq must be a positive multiple of Hkv; B, N >= 0.
 *     B*Hq*N == 0 returns ATTN_OK and launches nothing.
 *   - scale is the softmax scale (1/sqrt(D) in the usual case); it must be
 *     finite and positive.
 *   - stream is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous: they enqueue work on the stream and never synchronise.
 *     Argument errors are detected on the host before anything is enqueued.
 *   - Device-side waits are bounded; a wait that runs out sets a device flag
 *     that attn_device_status() reports (ATTN_ERR_DEVICE_TIMEOUT).
 *   - The library keeps no per-call state; it caches the driver entry point
 *     and kernel attributes.  It is safe to call from several host threads.
 */
#ifndef FLASH_EXACT_ATTENTION_GB300_ATTN_H
#define FLASH_EXACT_ATTENTION_GB300_ATTN_H

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum attn_status_code {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,    /* bad size, null pointer, misalignment, bad scale */
  ATTN_ERR_UNSUPPORTED = 2,    /* head dim not in {64, 128} */
  ATTN_ERR_CUDA = 3,           /* a CUDA runtime/driver call or launch failed */
  ATTN_ERR_DEVICE_TIMEOUT = 4, /* a bounded device wait ran out (see attn_device_status) */
  ATTN_ERR_ARCH = 5,           /* the current device is not compute capability 10.3 */
  ATTN_ERR_SCRATCH_LIMIT = 6   /* attn_bwd_noalloc: the problem needs more scratch than
                                  its fixed array holds */
};

/*
 * Forward: writes o (bf16 [B,Hq,N,D]) and lse (fp32 [B,Hq,N]).
 * Inputs q, k, v are read only.  Returns an attn_status_code.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int Hq, int Hkv, int N, int D, int causal, float scale,
             void* stream);

/*
 * Backward: the forward's arguments with o and lse as INPUTS (the outputs of
 * attn_fwd on the same q, k, v, causal, scale), then dout (bf16 [B,Hq,N,D],
 * input) and the outputs dq (bf16 [B,Hq,N,D]), dk, dv (bf16 [B,Hkv,N,D]).
 * Scratch: fp32 workspaces (Delta [B,Hq,N] and a dQ accumulator
 * [B,Hq,N,D]) are taken stream-ordered from the current device's default
 * memory pool (cudaMallocAsync/cudaFreeAsync on `stream`).
 * Returns an attn_status_code.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o,
             const float* lse, int B, int Hq, int Hkv, int N, int D, int causal,
             float scale, void* stream, const void* dout, void* dq, void* dk,
             void* dv);

/*
 * The same two calls for IEEE fp16 (binary16) q, k, v, o, dout, dq, dk, dv
 * instead of bf16 (FlashAttention for Tesla P100, "What it supports": fp16
 * inputs with fp32 accumulation).  Arguments, layouts, scratch, results and
 * error codes are those of attn_fwd / attn_bwd; lse stays fp32.  P and dS are
 * rounded to fp16 for the tensor cores (P <= 2^8 and |dS| well inside fp16's
 * range for attention inputs); every accumulation is fp32.  Results that
 * exceed fp16's range (|x| > 65504) become +-inf.
 */
int attn_fwd_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int Hq, int Hkv, int N, int D, int causal, float scale,
                 void* stream);
int attn_bwd_f16(const void* q, const void* k, const void* v, const void* o,
                 const float* lse, int B, int Hq, int Hkv, int N, int D, int causal,
                 float scale, void* stream, const void* dout, void* dq, void* dk,
                 void* dv);

/*
 * Stieltjes attention forward (bf16; FlashStieltjes page, "Why touch softmax",
 * "The challenge", "The kernel"): weights p_j = (lambda - s_j)^-order over the
 * allowed keys, s = scale * q.k, with the pole lambda found per row by
 * newton_steps Newton-Raphson steps on sum_j (lambda - s_j)^-order = 1 from
 * 1.1 above the row maximum (the page's kernel runs 3); o = sum_j p_j v_j
 * (bf16 [B,Hq,N,D]), pole = lambda in score units (fp32 [B,Hq,N]).  The keys
 * are streamed newton_steps + 2 times.  Other arguments, layouts and errors as
 * attn_fwd; order must be 2 or 4 (else ATTN_ERR_UNSUPPORTED), 1 <= newton_steps
 * <= 64 (else ATTN_ERR_INVALID_ARG).  Weights are used as the last step leaves
 * them: rows whose Newton iteration has not converged are not renormalised.
 */
int attn_stieltjes_fwd(const void* q, const void* k, const void* v, void* o, float* pole,
                       int B, int Hq, int Hkv, int N, int D, int causal, float scale, int order,
                       int newton_steps, void* stream);

/*
 * Forward over a batch of sequences of different lengths, packed without
 * padding (bf16).  Each sequence b is an independent attention problem over
 * its own tokens, exactly as attn_fwd computes for one sequence (causal means
 * key j <= query i within the sequence).  Token-major packed layout:
 *   q, o : bf16 [total, Hq, D];  k, v : bf16 [total, Hkv, D];
 *   lse  : fp32 [Hq, total]  (natural log, as attn_fwd)
 *   cu_seqlens : int32 DEVICE array [B + 1], cu_seqlens[0] = 0,
 *                nondecreasing, cu_seqlens[B] = total; sequence b is tokens
 *                cu_seqlens[b] .. cu_seqlens[b+1] - 1.
 *   max_seqlen : at least the longest sequence (it sizes the grid).
 * Ragged sequences without padding: FlashAttention for Tesla P100 page, "What
 * it supports".  D in {64, 128}; Hq a multiple of Hkv; B, total, max_seqlen
 * >= 0 (any of them 0: ATTN_OK, nothing launched); pointers 16-byte aligned
 * (cu_seqlens 4-byte).  Empty sequences are allowed.  The lengths live on the
 * device, so they are checked there: a decreasing entry, a sequence longer
 * than max_seqlen or one reaching past total leaves that sequence's rows
 * unwritten and makes attn_device_status() return ATTN_ERR_INVALID_ARG.  One
 * kernel launch.
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* cu_seqlens, int B, int Hq, int Hkv, int total, int max_seqlen,
                    int D, int causal, float scale, void* stream);

/*
 * Backward of attn_fwd_varlen (bf16): dq, dk, dv of sum(dout * O), each
 * sequence independently, from the forward's o and lse (the P recomputation
 * of attn_bwd: FlashAttention for Tesla P100 page, "Documentation").
 *   q, o, dout, dq : bf16 [total, Hq, D];  k, v, dk, dv : bf16 [total, Hkv, D];
 *   lse : fp32 [Hq, total] as attn_fwd_varlen wrote it;
 *   cu_seqlens, max_seqlen, causal, scale : as given to attn_fwd_varlen.
 * Sizes, alignment and the device-side check of cu_seqlens as for
 * attn_fwd_varlen (an invalid sequence leaves its dk/dv rows unwritten and
 * its dq rows zero; attn_device_status() then returns ATTN_ERR_INVALID_ARG).
 * Tokens outside every sequence (when cu_seqlens[0] > 0 or cu_seqlens[B] <
 * total) get dq = 0 and unwritten dk/dv.  dQ is summed in fp32 with atomic
 * reduce-adds, so its last bits vary from run to run.  Scratch: fp32
 * total*Hq*D (dQ accumulator) + 2*B*Hq*ceil(max_seqlen/128)*128 (LSE2, Delta),
 * cudaMallocAsync / cudaFreeAsync on `stream`.  A memset and three kernel
 * launches.
 */
int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const int* cu_seqlens, int B, int Hq, int Hkv, int total, int max_seqlen,
                    int D, int causal, float scale, void* stream, const void* dout, void* dq,
                    void* dk, void* dv);

/*
 * attn_fwd_varlen / attn_bwd_varlen with fp16 tensors (q, k, v, o, dout, dq,
 * dk, dv fp16; lse fp32): the same arguments, layouts, checks and errors, and
 * the arithmetic of attn_fwd_f16 / attn_bwd_f16 (P and dS rounded to fp16 for
 * the tensor cores, fp32 accumulation).
 */
int attn_fwd_varlen_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int* cu_seqlens, int B, int Hq, int Hkv, int total, int max_seqlen,
                        int D, int causal, float scale, void* stream);
int attn_bwd_varlen_f16(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const int* cu_seqlens, int B, int Hq, int Hkv,
                        int total, int max_seqlen, int D, int causal, float scale, void* stream,
                        const void* dout, void* dq, void* dk, void* dv);

/*
 * Nystrom attention forward (bf16 in and out).  FlashNystrom page, "Scope":
 *     O = softmax(s Q Kt^T) . pinv(softmax(s Qt Kt^T)) . softmax(s Qt K^T) . V
 * per (batch, query head), s = scale, every softmax over its rows.  Qt and Kt
 * are the m = num_landmarks landmarks: landmark i is the mean of rows
 * floor(i N / m) .. floor((i+1) N / m) - 1 of Q (of that query head) and of K
 * (of its key/value head h / (Hq / Hkv)).  pinv is newton_iters unrolled
 * Newton-Schulz steps X <- 2X - X A X from X = A^T / (|A|_1 |A|_inf), in fp32;
 * with kappa > 0 ("Configuration": the Tikhonov ridge) they run on
 * A^T A + lambda I, lambda = |A|_1 |A|_inf / kappa, and pinv(A) = X A^T;
 * kappa = 0 runs them on A itself.  No causal mask, no value convolution.
 *   q, o : bf16 [B, Hq, N, D];  k, v : bf16 [B, Hkv, N, D]  (device, 16-byte
 *   aligned, contiguous).  D in {64, 128}; 1 <= num_landmarks <= 64 (larger:
 *   ATTN_ERR_UNSUPPORTED); N >= num_landmarks; 0 <= newton_iters <= 100;
 *   kappa finite and >= 0; B * (Hq + Hkv) <= 65535.  B * Hq == 0 returns
 *   ATTN_OK without launching.
 * Landmarks, the landmark softmax, W = softmax(s Qt K^T) V and pinv(A) W are
 * fp32; Qt, Kt, P and pinv(A) W enter the tensor cores as bf16.  Scratch of
 * about (B*Hq + B*Hkv) * m * D * 4 * splits + B*Hq*(chunks*m*(D+2)*4 + ...)
 * bytes is taken with cudaMallocAsync / cudaFreeAsync on `stream`.  A memset
 * and six kernel launches.
 */
int attn_nystrom_fwd(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                     int Hkv, int N, int D, int num_landmarks, int newton_iters, float kappa,
                     float scale, void* stream);

/*
 * Deterministic backward (bf16): the arguments, layouts and error codes of
 * attn_bwd, with results that are bitwise identical from run to run.
 * attn_bwd adds each key tile's fp32 dQ partial into an accumulator in
 * arrival order, so dQ's last bits vary between runs; here dK and dV come from
 * the same kernel without those adds, and dQ from a second kernel that owns a
 * query tile and sums its key tiles in a fixed order (recomputing S and dP:
 * 7 MMAs per (query, key) tile pair instead of 5).  A GQA group is never split
 * across CTAs on this path.  Scratch: fp32 LSE2 and Delta only
 * (cudaMallocAsync/cudaFreeAsync on `stream`).
 */
int attn_bwd_deterministic(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, int B, int Hq, int Hkv, int N, int D, int causal,
                           float scale, void* stream, const void* dout, void* dq, void* dk,
                           void* dv);

/*
 * Backward without any device allocation.  No counterpart in the paper: this
 * is a deployment variant of attn_bwd for callers that cannot call the CUDA
 * allocator -- a process whose device memory is owned by its own pool, or a
 * serving loop that allows no allocation after start-up.
 * Arguments, layouts, results and error codes are those of attn_bwd.  The fp32
 * scratch lives in one fixed array in device memory of
 * attn_bwd_noalloc_scratch_limit() bytes (32 MiB), which must hold
 * B*Hq*roundup(N,128)*(D+2)*4 bytes; larger problems return
 * ATTN_ERR_SCRATCH_LIMIT before any device work.
 *   - Every call on a device shares that array.  Calls that can overlap on the
 *     GPU (other streams, unordered host threads) race and give wrong results.
 *   - The array keeps the previous call's contents; each call rewrites all it
 *     reads before reading it.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it: make it before any stream capture.
 *   - The array occupies device memory until the process exits: from the
 *     first call into this library on a device under lazy module loading (the
 *     CUDA default), or from context creation on every device when
 *     CUDA_MODULE_LOADING=EAGER, even if attn_bwd_noalloc is never called.
 *   - The library caches per-device addresses (this array, its error word):
 *     do not use it across cudaDeviceReset.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, int B, int Hq, int Hkv, int N, int D, int causal,
                     float scale, void* stream, const void* dout, void* dq, void* dk, void* dv);

/* Size in bytes of attn_bwd_noalloc's fixed scratch array. */
long long attn_bwd_noalloc_scratch_limit(void);

/* Static, human-readable text for a status code (never NULL). */
const char* attn_status_string(int status);

/*
 * Synchronises `stream`, then reports and clears the device-side error flag
 * of the current device: ATTN_ERR_DEVICE_TIMEOUT if a bounded wait ran out in
 * any kernel since the last call, ATTN_ERR_CUDA if the synchronisation
 * failed, ATTN_OK otherwise.
 */
int attn_device_status(void* stream);

/*
 * Sets the limit, in milliseconds, on every device-side wait of kernels
 * launched afterwards by this process (default 2000; values < 1 are rejected
 * with ATTN_ERR_INVALID_ARG).
 */
int attn_set_wait_timeout_ms(int ms);

/*
 * Failure-detection self-test (diagnostic; not part of the attention method).
 * Enqueues on `stream` a one-thread kernel whose bounded device wait can never
 * be satisfied, so the wait runs out after `timeout_ms` (1..10000) and sets the
 * device error word: the next attn_device_status() returns
 * ATTN_ERR_DEVICE_TIMEOUT (and clears it).  Nothing faults or hangs; the
 * context stays usable.  Returns ATTN_ERR_INVALID_ARG for a limit out of range.
 */
int attn_selftest_wait_timeout(int timeout_ms, void* stream);

/* Library ABI version: (major << 16) | minor. */
int attn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FLASH_EXACT_ATTENTION_GB300_ATTN_H */
