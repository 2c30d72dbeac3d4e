// gdn_chunk_bwd_chunked: the backward pass of the scalar-gate recurrence
// (decay before the prediction) through the chunk form, in four launches:
//   cbwd_prep_kernel   per (chunk, head): G, T = (I + A)^{-1}, W, U0, P
//   cbwd_fwd_kernel    per (32 value rows, head, sequence): the chunks in
//                      order; each chunk's entry state S and its U
//   cbwd_rev_kernel    the same grid, the chunks in reverse; each chunk's
//                      exit gradient dS' and dU, and dh0
//   cbwd_grad_kernel   per (chunk, head): dq, dk, dv, dbeta, dg
// The arithmetic (fp32 throughout; the adjoint of each step of the chunk
// form) is in bwd_chunked_body.cuh. The per-chunk intermediates live in a
// stream-ordered workspace (about 650 KB per chunk and head at
// d_k = d_v = 128).
#include "gdn_internal.cuh"
#include "bwd_chunked_body.cuh"

namespace gdn {
namespace {

constexpr int kCbThreads = 256;
// value rows per chain CTA: with 64 the chain grids (d_v / 64 per head and
// sequence) of a 4-sequence, 16-head problem run in one wave at one CTA per
// SM (32 rows took two)
constexpr int kCbRows = 64;

struct DevX {
  int tid, nt;
  float* smem;
  __device__ void sync() { __syncthreads(); }
};

template <int DK, int DV, bool BF>
__global__ void __launch_bounds__(kCbThreads) cbwd_prep_kernel(const cbwd::Args a) {
  extern __shared__ float4 sm4[];
  DevX x{(int)threadIdx.x, kCbThreads, reinterpret_cast<float*>(sm4)};
  cbwd::prep_body<DK, DV, BF>(x, a, (int)blockIdx.x);
}

template <int DK, int DV, bool BF>
__global__ void __launch_bounds__(kCbThreads) cbwd_fwd_kernel(const cbwd::Args a) {
  extern __shared__ float4 sm4[];
  DevX x{(int)threadIdx.x, kCbThreads, reinterpret_cast<float*>(sm4)};
  cbwd::fwd_body<DK, DV, kCbRows, BF>(x, a, (int)blockIdx.x, (int)blockIdx.y, (int)blockIdx.z);
}

template <int DK, int DV, bool BF>
__global__ void __launch_bounds__(kCbThreads) cbwd_rev_kernel(const cbwd::Args a) {
  extern __shared__ float4 sm4[];
  DevX x{(int)threadIdx.x, kCbThreads, reinterpret_cast<float*>(sm4)};
  cbwd::rev_body<DK, DV, kCbRows, BF>(x, a, (int)blockIdx.x, (int)blockIdx.y, (int)blockIdx.z);
}

template <int DK, int DV, bool BF>
__global__ void __launch_bounds__(kCbThreads, 3) cbwd_grad_kernel(const cbwd::Args a) {
  extern __shared__ float4 sm4[];
  DevX x{(int)threadIdx.x, kCbThreads, reinterpret_cast<float*>(sm4)};
  cbwd::grad_body<DK, DV, BF>(x, a, (int)blockIdx.x);
}

bool al16c(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <int DK, int DV>
cudaError_t launch_all(const cbwd::Args& a, long long zc, cudaStream_t st, int* launches) {
  using namespace cbwd;
  const int s_prep = prep_smem<DK, DV, true>() * 4, s_fwd = fwd_smem<DK, kCbRows>() * 4,
            s_rev = rev_smem<DK, kCbRows>() * 4, s_grad = grad_smem<DK, DV, true>(kCbThreads) * 4;
  auto kp = cbwd_prep_kernel<DK, DV, true>;
  auto kf = cbwd_fwd_kernel<DK, DV, true>;
  auto kr = cbwd_rev_kernel<DK, DV, true>;
  auto kg = cbwd_grad_kernel<DK, DV, true>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, s_prep)) ||
      (e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, s_fwd)) ||
      (e = cudaFuncSetAttribute(kr, cudaFuncAttributeMaxDynamicSharedMemorySize, s_rev)) ||
      (e = cudaFuncSetAttribute(kg, cudaFuncAttributeMaxDynamicSharedMemorySize, s_grad)))
    return e;
  const dim3 chain(DV / kCbRows, a.H, a.N);
  int t = timing_start(GDN_KERNEL_CBWD_PREP, st);
  kp<<<(unsigned)zc, kCbThreads, s_prep, st>>>(a);
  e = cudaGetLastError();
  timing_stop(t, st, e);
  if (e) return e;
  t = timing_start(GDN_KERNEL_CBWD_FWD, st);
  kf<<<chain, kCbThreads, s_fwd, st>>>(a);
  e = cudaGetLastError();
  timing_stop(t, st, e);
  if (e) return e;
  t = timing_start(GDN_KERNEL_CBWD_REV, st);
  kr<<<chain, kCbThreads, s_rev, st>>>(a);
  e = cudaGetLastError();
  timing_stop(t, st, e);
  if (e) return e;
  t = timing_start(GDN_KERNEL_CBWD_GRAD, st);
  kg<<<(unsigned)zc, kCbThreads, s_grad, st>>>(a);
  e = cudaGetLastError();
  timing_stop(t, st, e);
  if (e == cudaSuccess) *launches += 4;
  return e;
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_chunk_bwd_chunked(const void* q, const void* k, const void* v,
                                     const float* g, const float* beta, const float* h0,
                                     const void* dout, const float* dhT, float* dq,
                                     float* dk, float* dv, float* dg, float* dbeta,
                                     float* dh0, const int32_t* cu_seqlens, int B, int H,
                                     int T, int dk_dim, int dv_dim, gdn_stream_t stream) {
  using namespace gdn;
  if (B < 0 || H <= 0 || T < 0) return GDN_ERR_INVALID_ARG;
  if ((dk_dim != 64 && dk_dim != 128) || (dv_dim != 64 && dv_dim != 128))
    return GDN_ERR_UNSUPPORTED;
  if (cu_seqlens && B == 0) return GDN_ERR_INVALID_ARG;
  if (cu_seqlens) return GDN_ERR_UNSUPPORTED;  // dense batches only
  if (B > 65535 || H > 65535) return GDN_ERR_UNSUPPORTED;
  const long long tokens = (long long)B * T;
  if (B == 0) return GDN_OK;
  if (tokens > 0 && (!q || !k || !v || !g || !beta || !dout || !dq || !dk || !dv || !dg ||
                     !dbeta))
    return GDN_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, g, beta, h0, dout, dhT, dq, dk, dv, dg, dbeta, dh0};
  for (const void* p : ptrs)
    if (p && !al16c(p)) return GDN_ERR_MISALIGNED;
  const void* outs[] = {dq, dk, dv, dg, dbeta};
  for (const void* o : outs)
    if (o && (o == q || o == k || o == v || o == g || o == beta || o == dout))
      return GDN_ERR_INVALID_ARG;
  int* status = nullptr;
  int rc = device_status_ptr(&status);
  if (rc != GDN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t sdd = (size_t)B * H * dk_dim * dv_dim;
  if (T == 0) {  // nothing to sweep: dh0 = dhT
    cudaError_t e = cudaSuccess;
    if (dh0 && dh0 != dhT)
      e = dhT ? cudaMemcpyAsync(dh0, dhT, sdd * 4, cudaMemcpyDeviceToDevice, st)
              : cudaMemsetAsync(dh0, 0, sdd * 4, st);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  }
  const int nch = (T + cbwd::C - 1) / cbwd::C;
  const long long zc = (long long)B * nch * H;
  if (zc > 0x7fffffffll) return GDN_ERR_UNSUPPORTED;
  const size_t C = cbwd::C, DK = dk_dim, DV = dv_dim;
  // per chunk and head, in floats
  const size_t per = C + 2 * C * C + C * DK + 2 * C * DV + 2 * DV * DK + C * DV +  // G T P W U0 U S dSx dU
                     5 * C * DK + C * DV + 5 * C * C;  // dOS dKbar dW dKb dKs, dVb, dP dT X dA KK
  float* ws = nullptr;
  if (cudaMallocAsync(reinterpret_cast<void**>(&ws), per * zc * sizeof(float), st) != cudaSuccess)
    return GDN_ERR_CUDA;
  float* cur = ws;
  auto take = [&](size_t n) { float* p = cur; cur += n * (size_t)zc; return p; };
  cbwd::Args a{};
  a.q = q; a.k = k; a.v = v; a.dout = dout;
  a.g = g; a.beta = beta; a.h0 = h0; a.dhT = dhT;
  a.N = B; a.H = H; a.T = T; a.nch = nch;
  a.G = take(C); a.Tm = take(C * C); a.P = take(C * C); a.W = take(C * DK);
  a.U0 = take(C * DV); a.U = take(C * DV); a.S = take(DV * DK); a.dSx = take(DV * DK);
  a.dU = take(C * DV);
  a.dOS = take(C * DK); a.dKbar = take(C * DK); a.dW = take(C * DK); a.dKb = take(C * DK);
  a.dKs = take(C * DK); a.dVb = take(C * DV);
  a.dP = take(C * C); a.dT = take(C * C); a.X = take(C * C); a.dA = take(C * C);
  a.KK = take(C * C);
  a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta; a.dh0 = dh0;
  int launches = 0;
  cudaError_t e;
  if (dk_dim == 128 && dv_dim == 128) e = launch_all<128, 128>(a, zc, st, &launches);
  else if (dk_dim == 128) e = launch_all<128, 64>(a, zc, st, &launches);
  else if (dv_dim == 128) e = launch_all<64, 128>(a, zc, st, &launches);
  else e = launch_all<64, 64>(a, zc, st, &launches);
  count_launches(e, launches);
  const cudaError_t f = cudaFreeAsync(ws, st);
  return (e == cudaSuccess && f == cudaSuccess) ? GDN_OK : GDN_ERR_CUDA;
}
