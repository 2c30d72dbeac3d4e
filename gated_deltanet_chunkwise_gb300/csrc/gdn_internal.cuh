// Internal declarations shared by the library's translation units.
#pragma once

#include <functional>

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// One chunked forward request after host validation.
//
// Sequence-parallel passes (parts > 1) split each sequence's chunks into
// `parts` contiguous sub-sequences. `mode` selects what a launch does:
//   kModeOutput : state rows start from h0 / zero (part 0) or from
//                 ws_start (part p >= 1); outputs are written; the last part
//                 writes hT.
//   kModeSplit  : part 0 runs the true recurrence from h0 and writes both its
//                 outputs and its end state (the start of part 1, into
//                 ws_start); parts p >= 1 run from a zero state (rows
//                 [0, dv): the incremental state) and from the identity
//                 (rows [dv, dv + dk): the scaling matrix) and write both end
//                 values into ws_end.
// Workspace layouts (math orientation, row-major, dk columns):
//   ws_end   [N, H, parts, dv + dk, dk]
//   ws_start [N, H, parts, dv, dk]   (entry p holds the true start of part p)
enum { kModeOutput = 0, kModeSplit = 1 };

struct ChunkParams {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* h0;
  void* out;
  float* hT;
  const int32_t* cu_seqlens;
  int N, H, T, dk, dv, C;
  int variant;     // GDN_GATE_BEFORE_PREDICT / GDN_GATE_AFTER_PREDICT
  int parts;       // sequence-parallel split (>= 1)
  int part_begin;  // first part covered by this launch
  int part_count;  // parts covered by this launch (grid.z = N * part_count)
  int mode;
  float* ws_end;
  float* ws_start;
  int* status;     // device status word (first error wins)
  // tensor-core path: per-(chunk, head) operands written by the preparation
  // kernel (index chunk * H + head) and, for packed calls, chunk offsets
  const int32_t* chunk_off;  // [N + 1] first chunk of each sequence
  void* wneg;                // [chunks, H, 64, dk] bf16, -W = -T_W K
  void* pm;                  // [chunks, H, 64, 64] bf16, (Q K^T) (.) D (.) M
  void* tu;                  // [chunks, H, 64, 64] bf16, T diag(beta)
  float* cv;                 // [chunks, H, 132] fp32, e^G, e^{G_L-G}, gamma
                             // (KDA: [chunks, H, 256], gamma per key channel)
  // KDA (gdn_kda_fwd_ex on the tensor-core path): per-channel decays, so the
  // preparation also writes Q_g = Q (.) e^G and K_d = K (.) e^{G_L - G} as
  // bf16 tile images, and the chain decays the state column by column
  int kda;
  void* qg;                  // [chunks, H, 64, dk] bf16
  void* kd;                  // [chunks, H, 64, dk] bf16
  // steps either side of the recurrence (gdn_chunk_fwd_fused; tensor-core
  // path only): with `prologue` set, q and k are raw (normalised in the
  // kernels), g holds the gate logits a (g = -softplus(a)) and beta the step
  // logits b (beta = sigmoid(b)); with `epilogue` set, each output row is
  // RMS-normalised over d_v (times norm_w when given) and gated by
  // sigmoid(gate_z) when given
  int chain_rows;  // state rows per chain CTA: 64 (chunk_tc_kernel) or 128
  int prologue;
  int epilogue;
  const float* norm_w;       // [dv] fp32 or null
  const void* gate_z;        // like out (bf16) or null
  float eps;
  // fused single-launch path: per (sequence, head) a ring of hand-off
  // slots in global memory (launch_chunk_fused, fused_ring_bytes)
  void* ring;
};

struct DecodeParams {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  float* state;
  void* out;
  int N, H, dk, dv;
  int variant;
};

// The delta rule with a per-channel decay (gdn_kda_fwd).
struct KdaParams {
  const void* q;        // bf16 [tokens, H, dk]
  const void* k;        // bf16 [tokens, H, dk]
  const void* v;        // bf16 [tokens, H, dv]
  const float* g;       // fp32 [tokens, H, dk] log-decays
  const float* beta;    // fp32 [tokens, H]
  const float* h0;      // fp32 [N, H, dk, dv] or null
  void* out;            // bf16 [tokens, H, dv]
  float* hT;            // fp32 [N, H, dk, dv] or null (may be h0)
  const int32_t* cu_seqlens;
  int N, H, T, dk, dv;
  int* status;          // device status word
};

// Launchers (return a cudaError_t from the launch itself).
cudaError_t launch_chunk_simt(const ChunkParams& p, bool bf16,
                              cudaStream_t stream);
cudaError_t launch_sp_chain(const ChunkParams& p, cudaStream_t stream);
// The same correction by an associative scan over the sub-sequence maps;
// `buf` holds as many bytes as ws_end.
cudaError_t launch_sp_scan(const ChunkParams& p, float* buf,
                           cudaStream_t stream, int* launches);
// Tensor-core (tcgen05) path: bf16, dk in {64, 128} (64 on the 128 layout,
// the keys' and queries' second block read as zeros), dv in {64, 128}
// (KDA: dk = 128). A call takes
// chunk_tc_workspace_bytes of workspace (bound with chunk_tc_bind_workspace),
// runs launch_ut_prep once, then launch_chunk_tc for each pass.
bool chunk_tc_supported(int dk, int dv, long long tokens, int N, int H);
size_t chunk_tc_workspace_bytes(const ChunkParams& p);
void chunk_tc_bind_workspace(ChunkParams& p, void* ws);
cudaError_t launch_ut_prep(const ChunkParams& p, cudaStream_t stream,
                           int* launches);
// Chunk offsets of a packed call (part of launch_ut_prep / launch_kda_prep).
cudaError_t launch_chunk_offsets(const ChunkParams& p, cudaStream_t stream,
                                 int* launches);
// KDA on the tensor-core path (p.kda set; workspace bound as above): the
// preparation of every (chunk, head), then launch_chunk_tc with 128 rows.
cudaError_t launch_kda_prep(const ChunkParams& p, cudaStream_t stream,
                            int* launches);
long long chunk_tc_chunks_bound(const ChunkParams& p);
// Exclusive prefix of ceil(len_n / L) over the sequences of a packed call,
// out[N] the total (one launch).
cudaError_t launch_block_offsets(const int32_t* cu_seqlens, int N, int T,
                                 int L, int32_t* out, int* status,
                                 cudaStream_t stream);
int chunk_tc_nch_dense(const ChunkParams& p);
cudaError_t launch_chunk_tc(const ChunkParams& p, cudaStream_t stream);
// The same path in one launch with no workspace (one sub-sequence): a
// cluster per (sequence, head) of a preparation CTA and a whole-state chain
// CTA (bf16, dk in {64, 128}, dv in {64, 128}; not KDA).
cudaError_t launch_chunk_fused(const ChunkParams& p, cudaStream_t stream);
// Bytes of the hand-off ring the fused path needs (p.ring).
size_t fused_ring_bytes(const ChunkParams& p);
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_kda(const KdaParams& p, cudaStream_t stream);

// Backward pass (bwd.cu): gradients of the recurrence; per_channel: KDA's
// g [tokens, H, dk] (else the scalar gate); f32: fp32 q, k, v, dout (else
// bf16); variant: the gate placement. With `between`, the kernel's forward
// sweep (writing o_t to o_out when not null) and its reverse sweep are two
// launches with `between` enqueued between them (dout may be produced there).
int run_bwd(const void* q, const void* k, const void* v, const float* g,
            const float* beta, const float* h0, const void* dout,
            const float* dhT, float* dq, float* dk, float* dvo, float* dg,
            float* dbeta, float* dh0, const int32_t* cu_seqlens, int B, int H,
            int T, int dk_, int dv, bool per_channel, int variant, bool f32,
            cudaStream_t stream, float* o_out,
            const std::function<cudaError_t()>* between);

// Backward of the steps either side of the recurrence (fused_bwd.cu):
// scratch buffers, fp32, per (token, head) row.
struct FusedBwdBufs {
  float *qh, *kh, *vf, *g, *beta, *invq, *invk;  // prologue outputs
  float *o, *dO;                                 // recurrence output, its gradient
  float *dqh, *dkh, *dg, *dbeta;                 // the recurrence's gradients
  float* wpart;                                  // weight-gradient partials
};
size_t fused_bwd_bind(FusedBwdBufs& f, void* ws, long long rows, int dk, int dv);
cudaError_t launch_sub_prologue(const FusedBwdBufs& f, const void* q,
                                const void* k, const void* v, const float* a,
                                const float* b, long long rows, int dk, int dv,
                                cudaStream_t stream);
cudaError_t launch_sub_epilogue_bwd(const FusedBwdBufs& f, const void* dout,
                                    const float* w, const void* z, float eps,
                                    long long rows, int dv, float* dgate,
                                    float* dweight, cudaStream_t stream);
cudaError_t launch_sub_prologue_bwd(const FusedBwdBufs& f, const float* a,
                                    long long rows, int dk, float* dq,
                                    float* dk_out, float* da, float* db,
                                    cudaStream_t stream);

// Host helpers owned by gdn_abi.cu.
int validate_chunk_args(const void* q, const void* k, const void* v,
                        const float* g, const float* beta, const float* h0,
                        const void* out, const float* hT,
                        const int32_t* cu_seqlens, int B, int H, int T,
                        int dk, int dv, int C, int dtype, int variant,
                        int path, int sp_parts);
int device_status_ptr(int** out);
cudaError_t count_launches(cudaError_t e, int launches);
// Per-kernel timing (gdn_timing_enable): timing_start records the opening
// event of a launch of `kernel` on `stream` and returns a token (-1 while
// timing is off); timing_stop records the closing event, or drops the
// record when the launch itself failed.
int timing_start(int kernel, cudaStream_t stream);
void timing_stop(int token, cudaStream_t stream, cudaError_t launch_result);

// Device-side helpers --------------------------------------------------------

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Token range [bos, eos) of sequence n; false (and a recorded error) when the
// packing is inconsistent.
__device__ __forceinline__ bool sequence_range(const ChunkParams& p, int n,
                                               long long& bos,
                                               long long& eos) {
  if (p.cu_seqlens) {
    const int b = p.cu_seqlens[n], e = p.cu_seqlens[n + 1];
    if (b < 0 || e < b || e > p.T) {
      record_status(p.status, GDN_ERR_INVALID_ARG);
      return false;
    }
    bos = b;
    eos = e;
  } else {
    bos = (long long)n * p.T;
    eos = bos + p.T;
  }
  return true;
}

// Chunk range [c_begin, c_end) of part `part` of a sequence with nch chunks.
__device__ __forceinline__ void part_range(int nch, int parts, int part,
                                           int& c_begin, int& c_end) {
  const int per = (nch + parts - 1) / parts;
  c_begin = min(nch, part * per);
  c_end = min(nch, c_begin + per);
}

}  // namespace gdn
