// Single-token recurrent step (decode), state updated in place.
//
// Per (sequence, head) the fp32 state Z = S^T (dk x dv, dv contiguous) is
// streamed from HBM once and written once. With a = alpha, b = beta:
//   sk = Z^T k, sq = Z^T q                                  (old state)
//   u  = b (v - a sk)          [gate before the prediction]
//   u  = b (v - sk)            [gate after the prediction]
//   Z <- a Z + k u^T,  o = a sq + u (k . q)
// which is one step of the token recurrence (the GDN paragraph of the
// illustrated DeltaNet walk-through; read after the write). The bound is HBM:
// 8 dk dv bytes of state traffic against ~7 dk dv flops.
//
// Layout of the work: one CTA of 128 threads per (sequence, head). A thread
// owns 4 consecutive state columns (one float4) of DK * DV / 512 rows; a warp
// reads whole 512-byte rows, so every access is a coalesced 16-byte vector.
// Partial dot products are combined across the threads sharing a column
// group through shared memory.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 128;

template <typename InT, int DK, int DV, int VARIANT>
__global__ void __launch_bounds__(kThreads)
    decode_kernel(const DecodeParams p) {
  constexpr int TPR = DV / 4;              // threads per state row
  constexpr int RPP = kThreads / TPR;      // rows per pass
  constexpr int PASSES = DK / RPP;         // rows per thread
  __shared__ float sk_q[2][DK];
  __shared__ float red[2][RPP][DV];
  __shared__ float s_kq;

  const int tid = threadIdx.x;
  const int cg = tid % TPR;                // column group
  const int ro = tid / TPR;                // row offset
  const size_t nh = blockIdx.x;
  const InT* q = static_cast<const InT*>(p.q) + nh * DK;
  const InT* k = static_cast<const InT*>(p.k) + nh * DK;
  const InT* v = static_cast<const InT*>(p.v) + nh * DV;
  float4* Z = reinterpret_cast<float4*>(p.state + nh * DK * DV);

  // Issue the whole state tile first so its loads overlap the token reads.
  float4 z[PASSES];
#pragma unroll
  for (int e = 0; e < PASSES; ++e) z[e] = Z[(ro + e * RPP) * TPR + cg];

  for (int i = tid; i < DK; i += kThreads) {
    sk_q[0][i] = to_f32(k[i]);
    sk_q[1][i] = to_f32(q[i]);
  }
  const float a = expf(p.g[nh]);
  const float b = p.beta[nh];
  __syncthreads();
  if (tid < 32) {
    float s = 0.f;
    for (int i = tid; i < DK; i += 32) s = fmaf(sk_q[0][i], sk_q[1][i], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (tid == 0) s_kq = s;
  }

  float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
  for (int e = 0; e < PASSES; ++e) {
    const int i = ro + e * RPP;
    const float ki = sk_q[0][i], qi = sk_q[1][i];
    pk.x = fmaf(z[e].x, ki, pk.x); pk.y = fmaf(z[e].y, ki, pk.y);
    pk.z = fmaf(z[e].z, ki, pk.z); pk.w = fmaf(z[e].w, ki, pk.w);
    pq.x = fmaf(z[e].x, qi, pq.x); pq.y = fmaf(z[e].y, qi, pq.y);
    pq.z = fmaf(z[e].z, qi, pq.z); pq.w = fmaf(z[e].w, qi, pq.w);
  }
  reinterpret_cast<float4*>(red[0][ro])[cg] = pk;
  reinterpret_cast<float4*>(red[1][ro])[cg] = pq;
  __syncthreads();

  // Every thread needs u for its 4 columns: reduce the RPP partials.
  float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sq = sk;
#pragma unroll
  for (int r = 0; r < RPP; ++r) {
    const float4 x = reinterpret_cast<const float4*>(red[0][r])[cg];
    const float4 y = reinterpret_cast<const float4*>(red[1][r])[cg];
    sk.x += x.x; sk.y += x.y; sk.z += x.z; sk.w += x.w;
    sq.x += y.x; sq.y += y.y; sq.z += y.z; sq.w += y.w;
  }
  const float pa = VARIANT == GDN_GATE_BEFORE_PREDICT ? a : 1.f;
  float u[4];
  const float vv[4] = {to_f32(v[cg * 4 + 0]), to_f32(v[cg * 4 + 1]),
                       to_f32(v[cg * 4 + 2]), to_f32(v[cg * 4 + 3])};
  const float skv[4] = {sk.x, sk.y, sk.z, sk.w};
  const float sqv[4] = {sq.x, sq.y, sq.z, sq.w};
#pragma unroll
  for (int c = 0; c < 4; ++c) u[c] = b * (vv[c] - pa * skv[c]);

  if (ro == 0) {
    InT* o = static_cast<InT*>(p.out) + nh * DV;
    const float kq = s_kq;
#pragma unroll
    for (int c = 0; c < 4; ++c) o[cg * 4 + c] = from_f32<InT>(fmaf(a, sqv[c], u[c] * kq));
  }

#pragma unroll
  for (int e = 0; e < PASSES; ++e) {
    const int i = ro + e * RPP;
    const float ki = sk_q[0][i];
    float4 w;
    w.x = fmaf(a, z[e].x, ki * u[0]);
    w.y = fmaf(a, z[e].y, ki * u[1]);
    w.z = fmaf(a, z[e].z, ki * u[2]);
    w.w = fmaf(a, z[e].w, ki * u[3]);
    Z[i * TPR + cg] = w;
  }
}

template <typename InT, int VARIANT>
cudaError_t launch_shape(const DecodeParams& p, cudaStream_t stream) {
  const unsigned grid = (unsigned)((size_t)p.N * p.H);
  const int t = timing_start(GDN_KERNEL_DECODE, stream);
  if (p.dk == 128 && p.dv == 128)
    decode_kernel<InT, 128, 128, VARIANT><<<grid, kThreads, 0, stream>>>(p);
  else if (p.dk == 128 && p.dv == 64)
    decode_kernel<InT, 128, 64, VARIANT><<<grid, kThreads, 0, stream>>>(p);
  else if (p.dk == 64 && p.dv == 128)
    decode_kernel<InT, 64, 128, VARIANT><<<grid, kThreads, 0, stream>>>(p);
  else
    decode_kernel<InT, 64, 64, VARIANT><<<grid, kThreads, 0, stream>>>(p);
  const cudaError_t e = cudaGetLastError();
  timing_stop(t, stream, e);
  return e;
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.variant == GDN_GATE_AFTER_PREDICT)
    return launch_shape<__nv_bfloat16, GDN_GATE_AFTER_PREDICT>(p, stream);
  return launch_shape<__nv_bfloat16, GDN_GATE_BEFORE_PREDICT>(p, stream);
}

}  // namespace gdn
