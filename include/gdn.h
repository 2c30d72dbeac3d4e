/*
 * gdn.h -- C ABI of the GB300 Gated DeltaNet library (libgdn_gb300.so).
 *
 * The method. For every sequence and head, with a d_v x d_k state S, scalar
 * gates alpha_t = exp(g_t) in (0, 1] and write strengths beta_t:
 *
 *     S~_t = alpha_t S_{t-1}                       (forget first)
 *     u_t  = beta_t (v_t - S~_t k_t)               (error of the prediction)
 *     S_t  = S~_t + u_t k_t^T                      (delta-rule write)
 *     o_t  = S_t q_t                               (read after the write)
 *
 * This is the Gated DeltaNet update as the illustrated DeltaNet walk-through
 * (stay-hungry-time.github.io/deltanet) states it in its GDN paragraph (worked
 * example 3 -> 2.4 -> 3.7), with the read after the write and the diagonal
 * included as in its DeltaNet output paragraphs. alpha = 1 gives plain
 * DeltaNet. GDN_GATE_AFTER_PREDICT selects the other placement, u_t =
 * beta_t (v_t - S_{t-1} k_t), S_t = alpha_t S_{t-1} + u_t k_t^T, the form of
 * the lqnn.cn "GPU parallelisation of Gated DeltaNet" page, section 1.2.
 *
 * The library evaluates it chunkwise (chunks of C tokens): a gated UT/WY
 * transform per chunk (the walk-through's "UT transform" and "WY
 * representation" pages), the serial state recurrence across chunks and the
 * chunk output (its chunkwise DeltaNet state/output paragraphs), and for long
 * sequences the incremental-state / scaling-matrix correction of "How to
 * Implement Sequence Parallelism in DeltaNet" (papercache.org, A2). Results
 * equal the token recurrence up to floating-point rounding.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, row-major
 *     and contiguous, and must not alias each other (except where stated).
 *   - States are stored transposed: h0, hT and state are [N, H, dk, dv] fp32
 *     and element (i, j) of a head's dk x dv block is S[j][i].
 *   - Work is enqueued on `stream` (NULL = legacy default stream) and runs
 *     asynchronously; no entry point synchronises the host. Argument checks
 *     run on the host first: a failing check returns a negative status and
 *     enqueues nothing.
 *   - Workspace, when a path needs it, is taken with cudaMallocAsync on
 *     `stream` and released with cudaFreeAsync on the same stream.
 *   - Thread safety: entry points may be called concurrently from several
 *     host threads on different streams.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* gdn_stream_t;

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = -1,  /* null pointer, bad size, bad packing */
  GDN_ERR_UNSUPPORTED = -2,  /* valid request this build does not serve */
  GDN_ERR_MISALIGNED = -3,   /* pointer not 16-byte aligned */
  GDN_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed */
  GDN_ERR_TIMEOUT = -5       /* a bounded device wait gave up */
} gdn_status_t;

/* Gate placement (see the top of this file). */
#define GDN_GATE_BEFORE_PREDICT 0 /* default */
#define GDN_GATE_AFTER_PREDICT 1

/* Element type of q, k, v and out for gdn_chunk_fwd_ex. */
#define GDN_DTYPE_BF16 0
#define GDN_DTYPE_F32 1

/* Kernel family for gdn_chunk_fwd_ex (GDN_PATH_AUTO picks the fastest one
 * that serves the request). */
#define GDN_PATH_AUTO 0
#define GDN_PATH_SIMT 1   /* fp32 CUDA-core arithmetic; any supported shape */
#define GDN_PATH_TCGEN05 2 /* bf16 tcgen05/TMEM tensor-core path */
/* The tensor-core path with its chain kernel fixed (GDN_PATH_TCGEN05 picks
 * the one that needs fewer waves of CTAs, the split one on a tie): */
#define GDN_PATH_TCGEN05_SPLIT 3 /* 64 state rows per CTA (two CTAs per
                                    (sequence, head) when dv = 128) */
#define GDN_PATH_TCGEN05_WHOLE 4 /* 128 state rows per CTA, state in TMEM
                                    lanes (zero-padded when dv = 64) */
#define GDN_PATH_TCGEN05_FUSED 5 /* one launch: clusters of two preparation
                                    and two whole-state chain CTAs, the
                                    chunks handed over through a small ring
                                    in global memory that stays in L2 (a few
                                    chunks per (sequence, head)); no
                                    sequence-parallel split (sp_parts must be
                                    0 or 1); never chosen by GDN_PATH_AUTO */
/* How the sub-sequences of a sequence-parallel split are combined, OR-ed into
 * `path` of gdn_chunk_fwd_ex (default: the library's choice by a cost model,
 * in practice the serial chain): */
#define GDN_SP_CHAIN 0x100 /* serial chain, P - 2 dependent steps */
#define GDN_SP_SCAN 0x200  /* associative (Hillis-Steele) scan over the
                              sub-sequence maps, ceil(log2(P - 2)) rounds */

/*
 * gdn_chunk_fwd -- chunkwise forward pass, bf16 q/k/v/out.
 *
 *   q, k        bf16 [B, T, H, dk]; k (and usually q) L2-normalised per row
 *   v           bf16 [B, T, H, dv]
 *   g           fp32 [B, T, H], log alpha (<= 0)
 *   beta        fp32 [B, T, H]
 *   h0          fp32 [N, H, dk, dv] initial states, or NULL for zero states
 *   out         bf16 [B, T, H, dv] (written)
 *   hT          fp32 [N, H, dk, dv] final states (written), or NULL
 *   cu_seqlens  NULL for a dense batch (N = B sequences of T tokens), or a
 *               DEVICE int32 [B + 1] array of packed sequence offsets: then
 *               the tensors are [1, T, H, ...], B = N is the number of
 *               sequences, cu_seqlens[0] = 0, non-decreasing, and
 *               cu_seqlens[B] = T. Chunks never cross a sequence boundary;
 *               each sequence starts from its own h0 (or zero) state. The
 *               host never reads this array; a kernel that finds an
 *               inconsistent entry skips that sequence and records
 *               GDN_ERR_INVALID_ARG, returned by gdn_device_status.
 *   B, H, T     sizes; T may be any value >= 0 (no multiple of C needed)
 *   dk, dv      64 or 128 each
 *   C           chunk size; 64
 * Returns GDN_OK or a negative gdn_status_t.
 */
int gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                  const float* beta, const float* h0, void* out, float* hT,
                  const int32_t* cu_seqlens, int B, int H, int T, int dk,
                  int dv, int C, gdn_stream_t stream);

/* gdn_chunk_fwd_f32 -- the same with fp32 q, k, v and out (fp32 CUDA-core
 * arithmetic throughout). */
int gdn_chunk_fwd_f32(const float* q, const float* k, const float* v,
                      const float* g, const float* beta, const float* h0,
                      float* out, float* hT, const int32_t* cu_seqlens, int B,
                      int H, int T, int dk, int dv, int C,
                      gdn_stream_t stream);

/*
 * gdn_chunk_fwd_ex -- gdn_chunk_fwd with explicit options.
 *   dtype      GDN_DTYPE_BF16 or GDN_DTYPE_F32 (q, k, v, out)
 *   variant    GDN_GATE_BEFORE_PREDICT or GDN_GATE_AFTER_PREDICT
 *   path       GDN_PATH_* (the GDN_PATH_TCGEN05* paths require bf16;
 *              they serve dk = 64 on the dk = 128 kernels with the keys'
 *              and queries' second 64 columns read as zeros),
 *              optionally OR GDN_SP_CHAIN or GDN_SP_SCAN (not both)
 *   sp_parts   sequence-parallel split: 0 = automatic, 1 = never split,
 *              P >= 2 = split every sequence into P sub-sequences of whole
 *              chunks (incremental state from zero + scaling matrix, then the
 *              correction of the start states, by the serial chain or the
 *              associative scan, and the fused corrected output)
 * Other arguments as gdn_chunk_fwd.
 */
int gdn_chunk_fwd_ex(const void* q, const void* k, const void* v,
                     const float* g, const float* beta, const float* h0,
                     void* out, float* hT, const int32_t* cu_seqlens, int B,
                     int H, int T, int dk, int dv, int C, int dtype,
                     int variant, int path, int sp_parts,
                     gdn_stream_t stream);

/*
 * gdn_chunk_fwd_fused -- the forward pass with the steps either side of the
 * recurrence done in the same kernels (illustrated DeltaNet page, the
 * architecture table and its L2 Norm / RMSNorm paragraphs; its GDN section
 * for the output gate):
 *   in:  q <- q / |q|, k <- k / |k| per (token, head) over d_k (a zero vector
 *        stays zero); log alpha g = -softplus(a); beta = sigmoid(b)
 *   out: o <- o / sqrt(mean_{d_v}(o^2) + eps) * norm_weight, per (token,
 *        head), when norm_weight is given; then o <- o * sigmoid(gate)
 *        elementwise when gate is given
 *   q, k        bf16 [B, T, H, dk], raw (not normalised)
 *   a, b        fp32 [B, T, H] gate and step logits
 *   norm_weight fp32 [dv] (device) or NULL: no output normalisation
 *   gate        bf16 [B, T, H, dv] (device) or NULL: no output gate
 *   eps         >= 0, added to the mean of squares
 *   path        GDN_PATH_AUTO or GDN_PATH_TCGEN05 (the same here),
 *               GDN_PATH_TCGEN05_SPLIT, GDN_PATH_TCGEN05_WHOLE or
 *               GDN_PATH_TCGEN05_FUSED
 * Other arguments as gdn_chunk_fwd (decay before the prediction, automatic
 * sequence-parallel split). Served by the bf16 tensor-core path only:
 * dk = 128 and dv in {64, 128}; other shapes (and GDN_PATH_SIMT) return
 * GDN_ERR_UNSUPPORTED. The pages print no interface; this one is the
 * library's.
 */
int gdn_chunk_fwd_fused(const void* q, const void* k, const void* v,
                        const float* a, const float* b, const float* h0,
                        void* out, float* hT, const int32_t* cu_seqlens,
                        const float* norm_weight, const void* gate, float eps,
                        int B, int H, int T, int dk, int dv, int C, int path,
                        gdn_stream_t stream);

/*
 * gdn_recurrent_step -- one decode token per (sequence, head), state updated
 * in place (the token recurrence above applied once).
 *   q, k   bf16 [N, H, dk]      v, out  bf16 [N, H, dv]
 *   g      fp32 [N, H] (log alpha)       beta  fp32 [N, H]
 *   state  fp32 [N, H, dk, dv], read and overwritten
 *   dk, dv 64 or 128 each
 * The state is streamed from HBM once and written once (16-byte vectors).
 */
int gdn_recurrent_step(const void* q, const void* k, const void* v,
                       const float* g, const float* beta, float* state,
                       void* out, int N, int H, int dk, int dv,
                       gdn_stream_t stream);

/*
 * gdn_kda_fwd -- the delta rule with a per-channel decay (KDA; illustrated
 * DeltaNet walk-through, KDA paragraphs of its hybrid-architecture section),
 * token by token, state in fp32:
 *   S_bar = S_{t-1} diag(exp(g_t))          (key channel c of the d_v x d_k
 *                                             state scaled by exp(g_{t,c}))
 *   S_t = S_bar + beta_t (v_t - S_bar k_t) k_t^T,   o_t = S_t q_t
 * With every g_{t,c} equal this is gdn_chunk_fwd's recurrence.
 *   q, k   bf16 [B, T, H, dk]     v, out  bf16 [B, T, H, dv]   (device)
 *   g      fp32 [B, T, H, dk] log-decays (<= 0 for a decay; any value is
 *          evaluated as given, no rescaling is involved)
 *   beta   fp32 [B, T, H]
 *   h0     fp32 [N, H, dk, dv] or NULL (zero); hT likewise or NULL; element
 *          (i, j) is S[j][i]; hT may be the same buffer as h0, which makes a
 *          call with T = 1 a decode step that updates the state in place
 *   cu_seqlens  as for gdn_chunk_fwd (B = N sequences, T = total tokens)
 *   dk, dv 64 or 128
 * One CTA per (32 value rows, head, sequence); the call is asynchronous on
 * `stream`; an invalid packing is recorded in the status word
 * (gdn_device_status). Returns GDN_OK, GDN_ERR_INVALID_ARG,
 * GDN_ERR_UNSUPPORTED, GDN_ERR_MISALIGNED or GDN_ERR_CUDA.
 */
int gdn_kda_fwd(const void* q, const void* k, const void* v, const float* g,
                const float* beta, const float* h0, void* out, float* hT,
                const int32_t* cu_seqlens, int B, int H, int T, int dk, int dv,
                gdn_stream_t stream);

/*
 * gdn_kda_fwd_ex -- gdn_kda_fwd with a choice of kernels. Arguments and
 * results as for gdn_kda_fwd, plus:
 *   path      GDN_PATH_SIMT: the token-by-token kernel of gdn_kda_fwd.
 *             GDN_PATH_TCGEN05 (or GDN_PATH_TCGEN05_WHOLE): the chunk form
 *             on the tensor cores (walk-through: UT transform and WY
 *             sections with the per-channel gates of the GLA section;
 *             chunks of 64 tokens, bf16 operands, fp32 state and
 *             accumulation), dk = 128 and dv in {64, 128} only (otherwise
 *             GDN_ERR_UNSUPPORTED). Inside a chunk the decay of token r
 *             relative to token s is factored through 16-token blocks; a
 *             chunk in which some channel decays by more than 2^120 within
 *             one such block takes an exact pairwise sum instead (slower,
 *             same result).
 *             GDN_PATH_AUTO: the chunk form where it applies (at least one
 *             token, dk = 128, dv in {64, 128}), else the token-by-token
 *             kernel. GDN_PATH_TCGEN05_SPLIT: GDN_ERR_UNSUPPORTED.
 *             GDN_SP_CHAIN / GDN_SP_SCAN may be or-ed in as for
 *             gdn_chunk_fwd_ex.
 *   sp_parts  sequence-parallel split of the chunk form as for
 *             gdn_chunk_fwd_ex (0: automatic); ignored by GDN_PATH_SIMT.
 * The chunk form allocates its workspace with cudaMallocAsync on `stream`
 * (about 65 KB per chunk and head).
 */
int gdn_kda_fwd_ex(const void* q, const void* k, const void* v, const float* g,
                   const float* beta, const float* h0, void* out, float* hT,
                   const int32_t* cu_seqlens, int B, int H, int T, int dk,
                   int dv, int path, int sp_parts, gdn_stream_t stream);

/*
 * gdn_kda_bwd -- gradients of gdn_kda_fwd (walk-through: cost table and
 * memory paragraphs, a chunked model keeps only chunk-boundary states and
 * recomputes the rest; the lqnn.cn page: block recompute). For the loss
 * L = sum(dout * out) + sum(dhT * hT) it returns dL/dq, dk, dv, dg, dbeta and
 * dL/dh0. One token's adjoint, for the gradient dS arriving at S_t:
 *   dq_t = S_t^T do_t;  dS += do_t q_t^T;  du = dS k_t;
 *   dk_t = dS^T u - beta_t S_bar^T du;  dbeta_t = du . (v_t - S_bar k_t);
 *   dv_t = beta_t du;  dS_bar = dS - beta_t du k_t^T;
 *   dg_t = column sums of dS_bar (.) S_bar;  dS_{t-1} = dS_bar diag(e^{g_t}).
 * Inputs as gdn_kda_fwd (q, k, v bf16; g fp32 [B, T, H, dk]; beta fp32;
 * h0 fp32 [N, H, dk, dv] or NULL), plus
 *   dout   bf16 [B, T, H, dv], the gradient of out (device)
 *   dhT    fp32 [N, H, dk, dv] or NULL (zero), the gradient of hT
 * Outputs (device, fp32, written completely): dq, dk [B, T, H, dk]; dv
 * [B, T, H, dv]; dg [B, T, H, dk]; dbeta [B, T, H]; dh0 [N, H, dk, dv] or
 * NULL (not wanted; may be the dhT buffer). No output may alias an input
 * other than dh0 = dhT.
 * The forward state is recomputed on the GPU in fp32: a forward sweep keeps
 * the state every 16 tokens, then each 16-token block is recomputed from its
 * checkpoint and swept backwards. Scratch (cudaMallocAsync on `stream`):
 * about 1 KB per token and 32 value rows for the checkpoints (dk = 128; half
 * for dk = 64), 3 dk + 1 floats per token, head and 32 value rows of partial
 * sums, and a window of the recomputed 16-token block (256 KB per sequence,
 * head and 32 value rows at dk = 128). Asynchronous on
 * `stream`; an invalid packing is recorded in the status word. Returns GDN_OK,
 * GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED (head dims other than 64 / 128,
 * more than 65535 sequences), GDN_ERR_MISALIGNED or GDN_ERR_CUDA.
 */
int gdn_kda_bwd(const void* q, const void* k, const void* v, const float* g,
                const float* beta, const float* h0, const void* dout,
                const float* dhT, float* dq, float* dk, float* dv, float* dg,
                float* dbeta, float* dh0, const int32_t* cu_seqlens, int B,
                int H, int T, int dk_dim, int dv_dim, gdn_stream_t stream);

/*
 * gdn_chunk_bwd -- the same for gdn_chunk_fwd_ex's scalar gate: g and dg are
 * fp32 [B, T, H] (every key channel shares the token's log-decay; dg is the
 * sum of the per-channel gradient over the channels), and `variant` is the
 * gate placement of the forward pass: GDN_GATE_BEFORE_PREDICT (gdn_chunk_fwd's
 * default) or GDN_GATE_AFTER_PREDICT (predict with the undecayed state, then
 * decay; the adjoint's last steps become dk_t = dS^T u - beta_t S^T du,
 * dg_t = sum(dS (.) S) e^{g_t}, dS_{t-1} = e^{g_t} dS - beta_t du k_t^T with
 * S = S_{t-1}); anything else returns GDN_ERR_INVALID_ARG. Everything else
 * as gdn_kda_bwd.
 */
int gdn_chunk_bwd(const void* q, const void* k, const void* v, const float* g,
                  const float* beta, const float* h0, const void* dout,
                  const float* dhT, float* dq, float* dk, float* dv, float* dg,
                  float* dbeta, float* dh0, const int32_t* cu_seqlens, int B,
                  int H, int T, int dk_dim, int dv_dim, int variant,
                  gdn_stream_t stream);

/*
 * gdn_chunk_bwd_fused -- gradients of gdn_chunk_fwd_fused (the recurrence with
 * the steps either side: q, k L2-normalised, g = -softplus(a), beta =
 * sigmoid(b); out = RMSNorm(o) * norm_weight (when given) * sigmoid(gate)
 * (when given)) for L = sum(dout * out) + sum(dhT * hT). The steps' adjoints,
 * per (token, head): dgate = dout * y * s (1 - s) with y the normalised,
 * weighted output and s = sigmoid(gate); dweight = sum over rows of
 * dout * s * o r; do = r (dn - n mean(dn * n)) with n = o r, dn = dout * s *
 * w, r = (mean(o^2) + eps)^(-1/2); then the recurrence's backward
 * (gdn_chunk_bwd); then dq_raw = (dq - q (q . dq)) / |q_raw| (k alike;
 * zero rows get zero), da = -dg sigmoid(a), db = dbeta beta (1 - beta).
 * Inputs as gdn_chunk_fwd_fused (q, k, v, gate, dout bf16; a, b, norm_weight,
 * h0, dhT fp32; eps >= 0); outputs fp32: dq, dk [B, T, H, dk], dv
 * [B, T, H, dv], da, db [B, T, H], dh0 [N, H, dk, dv] or NULL, dweight
 * [dv] (only with norm_weight) or NULL, dgate like v (only with gate) or
 * NULL. The recurrence runs on the fp32 normalised inputs: the backward
 * kernel's forward sweep (a launch of its own) forms o in fp32 with its
 * checkpoints, the epilogue's adjoint turns dout into do, and the reverse
 * sweep follows; so these are the gradients of the exact (unrounded) map.
 * dk, dv in {64, 128}. Scratch (cudaMallocAsync on `stream`): about 4 (4 dk
 * + 3 dv + 6) bytes per token and head, plus gdn_chunk_bwd's. Returns as
 * gdn_chunk_bwd.
 */
int gdn_chunk_bwd_fused(const void* q, const void* k, const void* v,
                        const float* a, const float* b, const float* h0,
                        const int32_t* cu_seqlens, const float* norm_weight,
                        const void* gate, float eps, const void* dout,
                        const float* dhT, float* dq, float* dk, float* dv,
                        float* da, float* db, float* dh0, float* dweight,
                        float* dgate, int B, int H, int T, int dk_dim,
                        int dv_dim, gdn_stream_t stream);

/*
 * gdn_chunk_bwd_chunked -- gdn_chunk_bwd (decay before the prediction) through
 * the chunk form instead of the token-by-token reverse sweep (the
 * walk-through's chunkwise form and memory paragraphs: the state is kept at
 * chunk boundaries and everything inside a chunk is recomputed in parallel).
 * Per chunk of 64 tokens: the UT/WY quantities, the chunks' entry states by a
 * forward chain, their exit gradients by a reverse chain
 *   dU = P^T dO + K_bar dS'^T,  dS = e^{G_L} dS' + dO^T diag(e^G) Q - dU^T W,
 * then dq, dk, dv, dbeta, dg of every chunk in parallel (the adjoint of each
 * step of the chunk form; all fp32). Arguments, layouts, outputs and error
 * codes as gdn_chunk_bwd; cu_seqlens must be NULL (dense batches; otherwise
 * GDN_ERR_UNSUPPORTED). Scratch: about 650 KB per 64-token chunk and head at
 * d_k = d_v = 128 (cudaMallocAsync on `stream`).
 */
int gdn_chunk_bwd_chunked(const void* q, const void* k, const void* v,
                          const float* g, const float* beta, const float* h0,
                          const void* dout, const float* dhT, float* dq,
                          float* dk, float* dv, float* dg, float* dbeta,
                          float* dh0, const int32_t* cu_seqlens, int B, int H,
                          int T, int dk_dim, int dv_dim, gdn_stream_t stream);

/* gdn_chunk_bwd_f32 -- gdn_chunk_bwd for fp32 q, k, v and dout (the inputs
 * of gdn_chunk_fwd_f32 / gdn_chunk_fwd_ex with GDN_DTYPE_F32); everything
 * else, outputs included, as gdn_chunk_bwd. */
int gdn_chunk_bwd_f32(const float* q, const float* k, const float* v,
                      const float* g, const float* beta, const float* h0,
                      const float* dout, const float* dhT, float* dq, float* dk,
                      float* dv, float* dg, float* dbeta, float* dh0,
                      const int32_t* cu_seqlens, int B, int H, int T,
                      int dk_dim, int dv_dim, int variant, gdn_stream_t stream);

/*
 * gdn_chunk_fwd_sp_noalloc -- the sequence-parallel forward pass of
 * gdn_chunk_fwd_ex (path GDN_PATH_SIMT, sp_parts >= 2) for callers that may
 * not allocate device memory while they enqueue work (for example a plugin
 * of an inference engine whose memory plan is fixed in advance, or a serving
 * loop under a fixed memory budget). The pages describe no such variant; it
 * exists for this library's callers only.
 *
 * Instead of cudaMallocAsync it uses one fixed scratch array in device memory
 * owned by the library: GDN_NOALLOC_SCRATCH_BYTES per device, held by every
 * device that loads the library until the process exits. It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   - Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and caches it; make
 *     that first call before any stream capture on that device. The cache
 *     is keyed on the current driver context: after a device reset (or
 *     with another context current on the device) the next call looks the
 *     address up again, so that call too should precede any capture.
 *   - Size limit: the request needs gdn_noalloc_scratch_bytes(B, H, dk, dv,
 *     sp_parts) bytes; a request above GDN_NOALLOC_SCRATCH_BYTES returns
 *     GDN_ERR_UNSUPPORTED and enqueues nothing. sp_parts < 2 returns
 *     GDN_ERR_INVALID_ARG.
 *   - Sharing: all calls on a device use the same array, which keeps the last
 *     call's contents (every entry a call reads is written earlier in that
 *     call). Calls that overlap on the GPU (different streams, or host
 *     threads without ordering) race on it; the caller must serialise them.
 * Arguments and results are those of gdn_chunk_fwd_ex (dtype, variant,
 * sp_parts); other status codes as there.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (32u << 20)
int gdn_chunk_fwd_sp_noalloc(const void* q, const void* k, const void* v,
                             const float* g, const float* beta,
                             const float* h0, void* out, float* hT,
                             const int32_t* cu_seqlens, int B, int H, int T,
                             int dk, int dv, int C, int dtype, int variant,
                             int sp_parts, gdn_stream_t stream);

/* Scratch bytes gdn_chunk_fwd_sp_noalloc needs for these sizes (0 when
 * sp_parts < 2, B or H is not positive, or dk / dv is not 64 or 128). */
unsigned long long gdn_noalloc_scratch_bytes(int B, int H, int dk, int dv,
                                             int sp_parts);

/* gdn_device_status -- waits for `stream`, then returns and clears the
 * status recorded by kernels on the current device (GDN_OK, or the first
 * GDN_ERR_INVALID_ARG / GDN_ERR_TIMEOUT recorded since the last call). */
int gdn_device_status(gdn_stream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* gdn_status_string(int status);

/* Library version as MAJOR * 10000 + MINOR * 100 + PATCH. */
int gdn_version(void);

/* Number of kernels this library has enqueued in this process so far (all
 * devices, all streams). Lets a caller count the launches inside a timed
 * region. */
unsigned long long gdn_kernel_launches(void);

/* Kernel families, for per-kernel timing (no paper counterpart: a
 * measurement aid). */
typedef enum {
  GDN_KERNEL_CHUNK_PREP = 0,    /* tensor-core path: state-independent part
                                   of every (chunk, head) */
  GDN_KERNEL_CHUNK_CHAIN = 1,   /* tensor-core path: chunk-to-chunk state
                                   chain and outputs, 64 rows per CTA */
  GDN_KERNEL_CHUNK_SIMT = 2,    /* fp32-arithmetic chunk kernel */
  GDN_KERNEL_SP_CHAIN = 3,      /* sequence-parallel start-state chain */
  GDN_KERNEL_DECODE = 4,        /* single-token recurrent step */
  GDN_KERNEL_CHUNK_OFFSETS = 5, /* chunk offsets of packed sequences */
  GDN_KERNEL_CHUNK_CHAIN_WHOLE = 6, /* the same chain, 128 rows per CTA */
  GDN_KERNEL_KDA = 7,           /* per-channel-decay recurrence, token by
                                   token */
  GDN_KERNEL_KDA_PREP = 8,      /* chunked KDA: state-independent part of
                                   every chunk (its chain is kernel 6) */
  GDN_KERNEL_BWD = 9,           /* backward pass: checkpoints, recomputation
                                   and the reverse sweep */
  GDN_KERNEL_BWD_FINALIZE = 10, /* backward pass: sums over row blocks */
  GDN_KERNEL_CBWD_PREP = 11,    /* chunk-form backward: per-chunk T, W, U0, P */
  GDN_KERNEL_CBWD_FWD = 12,     /* chunk-form backward: entry states, U */
  GDN_KERNEL_CBWD_REV = 13,     /* chunk-form backward: exit gradients, dU */
  GDN_KERNEL_CBWD_GRAD = 14,    /* chunk-form backward: per-chunk gradients */
  GDN_KERNEL_CHUNK_FUSED = 15,  /* tensor-core path in one launch: the
                                   preparation and the chain of each
                                   (sequence, head) in one cluster */
  GDN_KERNEL_COUNT = 16
} gdn_kernel_t;

/* gdn_timing_enable -- per-kernel device timing on (nonzero) or off (0).
 * While on, every kernel the library enqueues is bracketed by two CUDA
 * events recorded on its stream (no synchronisation is added). Switching
 * discards all accumulated and pending timings. Returns GDN_OK or
 * GDN_ERR_CUDA. Events belong to the device current at launch time. */
int gdn_timing_enable(int on);

/* gdn_timing_read -- waits for the events recorded so far, folds their
 * elapsed times into per-kernel totals and writes, for `kernel` (a
 * gdn_kernel_t), the number of timed launches and their summed device time
 * in milliseconds since timing was last enabled. Either pointer may be NULL.
 * Returns GDN_OK, GDN_ERR_INVALID_ARG (unknown kernel) or GDN_ERR_CUDA. */
int gdn_timing_read(int kernel, unsigned long long* launches,
                    double* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_H */
