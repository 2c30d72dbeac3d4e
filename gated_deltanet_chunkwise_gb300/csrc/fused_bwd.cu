// Backward of the steps either side of the recurrence (gdn_chunk_bwd_fused).
//
// Illustrated DeltaNet walk-through, architecture table and its L2 Norm /
// RMSNorm paragraphs; its GDN section for the output gate. The forward
// (gdn_chunk_fwd_fused) is q = q_raw / |q_raw|, k alike, g = -softplus(a),
// beta = sigmoid(b), o = recurrence, out = (o r) w sigmoid(z) with
// r = (mean(o^2) + eps)^(-1/2). Its backward, per (token, head) row, around
// the recurrence's own (fp32 backward kernel):
//   epilogue:  dz = dout * (n w) * s (1 - s),  dy = dout * s,  dw += dy * n,
//              do = r (dn - n mean(dn * n)),  dn = dy * w     (n = o r)
//   prologue:  dq_raw = (dq - q (q . dq)) / |q_raw|  (k alike),
//              da = -dg sigmoid(a),  db = dbeta beta (1 - beta).
// Three row kernels (one warp per (token, head) row, d / 32 values per lane)
// and a fixed-order sum of the weight gradient's per-CTA partials. The
// recurrence's forward output o comes in fp32 from the forward sweep of the
// backward kernel (a launch of its own; the epilogue's adjoint runs between
// it and the reverse sweep), so the gradients are those of the exact
// (unrounded) map.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kRowThreads = 256;  // 8 warps, one row each at a time

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float sigm(float x) { return 1.f / (1.f + expf(-x)); }

// A lane's N consecutive values of a row (N = d / 32), one vector access.
template <int N>
__device__ __forceinline__ void ldv(const float* p, float (&x)[N]) {
  if constexpr (N == 4) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else {
    const float2 v = *reinterpret_cast<const float2*>(p);
    x[0] = v.x; x[1] = v.y;
  }
}
template <int N>
__device__ __forceinline__ void ldv(const __nv_bfloat16* p, float (&x)[N]) {
  if constexpr (N == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xffff0000u);
    x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xffff0000u);
  } else {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
    x[0] = __uint_as_float(v << 16); x[1] = __uint_as_float(v & 0xffff0000u);
  }
}
template <int N>
__device__ __forceinline__ void stv(float* p, const float (&x)[N]) {
  if constexpr (N == 4)
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  else
    *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
}

// q, k normalised (fp32), v widened to fp32, g = -softplus(a), beta =
// sigmoid(b), and the inverse lengths of q and k (0 for a zero row).
template <int DK, int DV>
__global__ void __launch_bounds__(kRowThreads)
    sub_prologue_kernel(const __nv_bfloat16* __restrict__ q,
                        const __nv_bfloat16* __restrict__ k,
                        const __nv_bfloat16* __restrict__ v,
                        const float* __restrict__ a, const float* __restrict__ b,
                        long long rows, float* qh, float* kh, float* vf,
                        float* g, float* beta, float* invq, float* invk) {
  constexpr int NK = DK / 32, NV = DV / 32;
  const int lane = threadIdx.x & 31;
  const long long w0 = ((long long)blockIdx.x * kRowThreads + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * kRowThreads) >> 5;
  for (long long row = w0; row < rows; row += nw) {
    const long long ek = row * DK + NK * lane, ev = row * DV + NV * lane;
    float xq[NK], xk[NK], xv[NV], sq = 0.f, sk = 0.f;
    ldv<NK>(q + ek, xq);
    ldv<NK>(k + ek, xk);
    ldv<NV>(v + ev, xv);
#pragma unroll
    for (int j = 0; j < NK; ++j) {
      sq = fmaf(xq[j], xq[j], sq);
      sk = fmaf(xk[j], xk[j], sk);
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    const float iq = sq > 0.f ? rsqrtf(sq) : 0.f, ik = sk > 0.f ? rsqrtf(sk) : 0.f;
#pragma unroll
    for (int j = 0; j < NK; ++j) {
      xq[j] *= iq;
      xk[j] *= ik;
    }
    stv<NK>(qh + ek, xq);
    stv<NK>(kh + ek, xk);
    stv<NV>(vf + ev, xv);
    if (lane == 0) {
      const float x = a[row];
      g[row] = -(fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))));
      beta[row] = sigm(b[row]);
      invq[row] = iq;
      invk[row] = ik;
    }
  }
}

// do (fp32) from dout through the output gate and the RMSNorm; dgate; the
// weight gradient's partial sum of this CTA (wpart[blockIdx.x][DV]).
template <int DV>
__global__ void __launch_bounds__(kRowThreads)
    sub_epilogue_bwd_kernel(const float* __restrict__ o,
                            const __nv_bfloat16* __restrict__ dout,
                            const float* __restrict__ w,
                            const __nv_bfloat16* __restrict__ z, float eps,
                            long long rows, float* dO, float* dgate,
                            float* wpart) {
  constexpr int NV = DV / 32;
  __shared__ float red[kRowThreads / 32][DV];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long w0 = ((long long)blockIdx.x * kRowThreads + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * kRowThreads) >> 5;
  float dwacc[NV], wv[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    dwacc[j] = 0.f;
    wv[j] = w ? w[NV * lane + j] : 1.f;
  }
  for (long long row = w0; row < rows; row += nw) {
    const long long e = row * DV + NV * lane;
    float x[NV], dy[NV], zz[NV], ss = 0.f;
    ldv<NV>(o + e, x);
    ldv<NV>(dout + e, dy);
    if (z) ldv<NV>(z + e, zz);
#pragma unroll
    for (int j = 0; j < NV; ++j) ss = fmaf(x[j], x[j], ss);
    const float r = w ? rsqrtf(warp_sum(ss) * (1.f / DV) + eps) : 1.f;
    float dz[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const float n = x[j] * r, pre = w ? n * wv[j] : x[j];
      if (z) {
        const float sg = sigm(zz[j]);
        dz[j] = dy[j] * pre * sg * (1.f - sg);
        dy[j] *= sg;
      }
      if (w) {
        dwacc[j] = fmaf(dy[j], n, dwacc[j]);
        dy[j] *= wv[j];  // now dn
      }
    }
    if (z && dgate) stv<NV>(dgate + e, dz);
    if (w) {
      float t = 0.f;
#pragma unroll
      for (int j = 0; j < NV; ++j) t = fmaf(dy[j], x[j] * r, t);
      const float m = warp_sum(t) * (1.f / DV);
#pragma unroll
      for (int j = 0; j < NV; ++j) dy[j] = r * (dy[j] - x[j] * r * m);
    }
    stv<NV>(dO + e, dy);
  }
  if (!w) return;
#pragma unroll
  for (int j = 0; j < NV; ++j) red[warp][NV * lane + j] = dwacc[j];
  __syncthreads();
  for (int c = threadIdx.x; c < DV; c += kRowThreads) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kRowThreads / 32; ++i) s += red[i][c];
    wpart[(size_t)blockIdx.x * DV + c] = s;
  }
}

// dweight[c] = sum of the CTAs' partials in a fixed order: one CTA of 1024
// threads, 1024 / dv groups; group j adds the partials i = j mod groups in
// increasing i (many loads in flight per thread), then the group sums are
// added in group order.
constexpr int kWsumThreads = 1024;
__global__ void __launch_bounds__(kWsumThreads)
    sub_weight_sum_kernel(const float* __restrict__ wpart, int parts, int dv,
                          float* dw) {
  __shared__ float gs[kWsumThreads];
  const int ng = kWsumThreads / dv, c = threadIdx.x % dv, j = threadIdx.x / dv;
  float s = 0.f;
  if (j < ng) {
    int i = j;
    for (; i + 3 * ng < parts; i += 4 * ng) {
      const float x0 = wpart[(size_t)i * dv + c];
      const float x1 = wpart[(size_t)(i + ng) * dv + c];
      const float x2 = wpart[(size_t)(i + 2 * ng) * dv + c];
      const float x3 = wpart[(size_t)(i + 3 * ng) * dv + c];
      s += x0; s += x1; s += x2; s += x3;
    }
    for (; i < parts; i += ng) s += wpart[(size_t)i * dv + c];
  }
  gs[threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.x < dv) {
    float t = 0.f;
    for (int g = 0; g < ng; ++g) t += gs[g * dv + threadIdx.x];
    dw[threadIdx.x] = t;
  }
}

// dq_raw, dk_raw from the normalised vectors' gradients; da, db.
template <int DK>
__global__ void __launch_bounds__(kRowThreads)
    sub_prologue_bwd_kernel(const float* __restrict__ qh,
                            const float* __restrict__ kh,
                            const float* __restrict__ dqh,
                            const float* __restrict__ dkh,
                            const float* __restrict__ invq,
                            const float* __restrict__ invk,
                            const float* __restrict__ a,
                            const float* __restrict__ beta,
                            const float* __restrict__ dg,
                            const float* __restrict__ dbeta, long long rows,
                            float* dq, float* dk, float* da, float* db) {
  constexpr int NK = DK / 32;
  const int lane = threadIdx.x & 31;
  const long long w0 = ((long long)blockIdx.x * kRowThreads + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * kRowThreads) >> 5;
  for (long long row = w0; row < rows; row += nw) {
    const long long e = row * DK + NK * lane;
    float xq[NK], xk[NK], gq[NK], gk[NK], tq = 0.f, tk = 0.f;
    ldv<NK>(qh + e, xq);
    ldv<NK>(kh + e, xk);
    ldv<NK>(dqh + e, gq);
    ldv<NK>(dkh + e, gk);
#pragma unroll
    for (int j = 0; j < NK; ++j) {
      tq = fmaf(xq[j], gq[j], tq);
      tk = fmaf(xk[j], gk[j], tk);
    }
    tq = warp_sum(tq);
    tk = warp_sum(tk);
    const float iq = invq[row], ik = invk[row];
#pragma unroll
    for (int j = 0; j < NK; ++j) {
      gq[j] = (gq[j] - xq[j] * tq) * iq;
      gk[j] = (gk[j] - xk[j] * tk) * ik;
    }
    stv<NK>(dq + e, gq);
    stv<NK>(dk + e, gk);
    if (lane == 0) {
      da[row] = -dg[row] * sigm(a[row]);
      const float bt = beta[row];
      db[row] = dbeta[row] * bt * (1.f - bt);
    }
  }
}

int row_grid(long long rows) {
  const long long need = (rows * 32 + kRowThreads - 1) / kRowThreads;
  return (int)std::max<long long>(1, std::min<long long>(need, 152ll * 8));
}

}  // namespace

cudaError_t launch_sub_prologue(const FusedBwdBufs& f, const void* q,
                                const void* k, const void* v, const float* a,
                                const float* b, long long rows, int dk, int dv,
                                cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  auto go = [&](auto kern) {
    kern<<<row_grid(rows), kRowThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(v), a, b, rows, f.qh, f.kh, f.vf, f.g,
        f.beta, f.invq, f.invk);
  };
  if (dk == 64 && dv == 64) go(sub_prologue_kernel<64, 64>);
  else if (dk == 64) go(sub_prologue_kernel<64, 128>);
  else if (dv == 64) go(sub_prologue_kernel<128, 64>);
  else go(sub_prologue_kernel<128, 128>);
  return cudaGetLastError();
}

cudaError_t launch_sub_epilogue_bwd(const FusedBwdBufs& f, const void* dout,
                                    const float* w, const void* z, float eps,
                                    long long rows, int dv, float* dgate,
                                    float* dweight, cudaStream_t stream) {
  if (rows <= 0) {
    if (dweight) return cudaMemsetAsync(dweight, 0, (size_t)dv * sizeof(float), stream);
    return cudaSuccess;
  }
  const int grid = row_grid(rows);
  auto go = [&](auto kern) {
    kern<<<grid, kRowThreads, 0, stream>>>(
        f.o, static_cast<const __nv_bfloat16*>(dout), w,
        static_cast<const __nv_bfloat16*>(z), eps, rows, f.dO, dgate, f.wpart);
  };
  if (dv == 64) go(sub_epilogue_bwd_kernel<64>); else go(sub_epilogue_bwd_kernel<128>);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !dweight) return e;
  sub_weight_sum_kernel<<<1, kWsumThreads, 0, stream>>>(f.wpart, grid, dv, dweight);
  return cudaGetLastError();
}

cudaError_t launch_sub_prologue_bwd(const FusedBwdBufs& f, const float* a,
                                    long long rows, int dk, float* dq,
                                    float* dk_out, float* da, float* db,
                                    cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  auto go = [&](auto kern) {
    kern<<<row_grid(rows), kRowThreads, 0, stream>>>(
        f.qh, f.kh, f.dqh, f.dkh, f.invq, f.invk, a, f.beta, f.dg, f.dbeta,
        rows, dq, dk_out, da, db);
  };
  if (dk == 64) go(sub_prologue_bwd_kernel<64>); else go(sub_prologue_bwd_kernel<128>);
  return cudaGetLastError();
}

// The scratch buffers, each rounded up to 256 bytes; with ws = null only
// the total size is computed.
size_t fused_bwd_bind(FusedBwdBufs& f, void* ws, long long rows, int dk, int dv) {
  size_t off = 0;
  const size_t r = (size_t)rows;
  auto take = [&](size_t n) {
    float* x = ws ? reinterpret_cast<float*>(static_cast<char*>(ws) + off) : nullptr;
    off += ((n * sizeof(float) + 255) & ~(size_t)255);
    return x;
  };
  f.qh = take(r * dk); f.kh = take(r * dk); f.dqh = take(r * dk); f.dkh = take(r * dk);
  f.vf = take(r * dv); f.o = take(r * dv); f.dO = take(r * dv);
  f.g = take(r); f.beta = take(r); f.invq = take(r); f.invk = take(r);
  f.dg = take(r); f.dbeta = take(r);
  f.wpart = take((size_t)152 * 8 * dv);
  return off;
}

}  // namespace gdn
