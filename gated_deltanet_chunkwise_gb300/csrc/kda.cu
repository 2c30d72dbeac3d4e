// KDA: the delta rule with a per-channel decay, token by token on the GPU.
//
// Illustrated DeltaNet walk-through, KDA paragraphs: each token scales
// column c of the d_v x d_k state by alpha_{t,c} = exp(g_{t,c}) ("decay
// first"), then corrects it with the delta rule on the forgotten state and
// reads it with q after the write:
//   S_bar = S diag(alpha_t);  u = beta_t (v_t - S_bar k_t);
//   S_t = S_bar + u k_t^T;    o_t = S_t q_t.
// Rows of the state never mix (row a's prediction and read use row a
// only), so the work spreads over (32-row blocks, heads, sequences): one CTA
// of 8 warps per block, each warp 4 state rows, each lane d_k / 32 channels
// of those 4 rows in fp32 registers (a token's q, k, alpha slice is read
// once per lane and used for 4 rows). Tokens go through in blocks of 16:
// their q, k, alpha (exp taken once, when staged), the block's v rows and
// beta in shared memory, fetched into registers a block ahead. The warp's
// four row sums per token (prediction, read) take a transposing shuffle
// butterfly (6 shuffles) and the four corrections 4 broadcasts; outputs
// leave per block, 64 contiguous bytes per token. Exact for any log-decay
// (no rescaling).
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kKdaRpw = 4;  // state rows per warp (and per thread)
constexpr int kKdaRows = 8 * kKdaRpw;  // state rows per CTA (8 warps)
constexpr int kKdaThreads = 256;
constexpr int kKdaTok = 16;      // tokens per staged block

// N (2 or 4) consecutive floats from shared memory in one vector load.
template <int N>
__device__ __forceinline__ void load_slice(const float* p, float (&x)[N]) {
  if constexpr (N == 4) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else {
    const float2 v = *reinterpret_cast<const float2*>(p);
    x[0] = v.x; x[1] = v.y;
  }
}

__device__ __forceinline__ void unpack_bf16x8_f(uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <int DK>
__global__ void __launch_bounds__(kKdaThreads)
    kda_kernel(const __nv_bfloat16* __restrict__ q,
               const __nv_bfloat16* __restrict__ k,
               const __nv_bfloat16* __restrict__ v,
               const float* __restrict__ g, const float* __restrict__ beta,
               const float* h0, __nv_bfloat16* __restrict__ out, float* hT,
               const int32_t* __restrict__ cu_seqlens, int H, int T, int dv,
               int* status) {
  constexpr int CPT = DK / 32;  // channels per thread
  __shared__ float sk[kKdaTok][DK], sq[kKdaTok][DK], sa[kKdaTok][DK];
  __shared__ float sv[kKdaTok][kKdaRows], sb[kKdaTok];
  __shared__ __nv_bfloat16 so[kKdaTok][kKdaRows];
  const int tid = threadIdx.x;
  const int lane = tid & 31, w = tid >> 5;
  const int h = blockIdx.y, n = blockIdx.z;
  const int row0 = blockIdx.x * kKdaRows, a0 = row0 + kKdaRpw * w;
  long long bos, eos;
  if (cu_seqlens) {
    // packed: T is the total token count; an invalid packing is recorded
    bos = cu_seqlens[n];
    eos = cu_seqlens[n + 1];
    if (bos < 0 || eos < bos || eos > T) {
      if (threadIdx.x == 0) record_status(status, GDN_ERR_INVALID_ARG);
      return;
    }
  } else {
    bos = (long long)n * T;
    eos = bos + T;
  }
  const size_t nh = (size_t)n * H + h;
  // Lane l of warp w holds channels CPT l .. CPT l + CPT - 1 of the warp's
  // rows a0 .. a0 + 3: each token's q, k, alpha slice is read once (one
  // vector load each, the warp's reads contiguous) and used for four rows.
  float S[kKdaRpw][CPT];
  // state element (c, a) of h0 / hT is S[a][c]
#pragma unroll
  for (int r = 0; r < kKdaRpw; ++r)
#pragma unroll
    for (int j = 0; j < CPT; ++j)
      S[r][j] = h0 ? h0[(nh * DK + CPT * lane + j) * dv + a0 + r] : 0.f;
  // Staging: the next block's q, k, g, v rows and beta are fetched into
  // registers (16-byte loads, all in flight together) while the current
  // block is processed, then converted into shared memory.
  constexpr int KTOT = kKdaTok * DK / 8, GTOT = kKdaTok * DK / 4;
  constexpr int KCH = (KTOT + kKdaThreads - 1) / kKdaThreads;  // q/k chunks of 8
  constexpr int GCH = (GTOT + kKdaThreads - 1) / kKdaThreads;  // g chunks of 4
  uint4 rk[KCH], rq[KCH], rv = make_uint4(0, 0, 0, 0);
  float4 rg[GCH];
  float rb = 0.f;
  auto fetch = [&](long long t0) {
    const int nt = (int)max(0ll, min((long long)kKdaTok, eos - t0));
#pragma unroll
    for (int j = 0; j < KCH; ++j) {
      const int e = tid + j * kKdaThreads, tt = e / (DK / 8), c8 = e % (DK / 8);
      rk[j] = rq[j] = make_uint4(0, 0, 0, 0);
      if (e < KTOT && tt < nt) {
        const size_t r = ((size_t)(t0 + tt) * H + h) * DK + 8 * c8;
        rk[j] = *reinterpret_cast<const uint4*>(k + r);
        rq[j] = *reinterpret_cast<const uint4*>(q + r);
      }
    }
#pragma unroll
    for (int j = 0; j < GCH; ++j) {
      const int e = tid + j * kKdaThreads, tt = e / (DK / 4), c4 = e % (DK / 4);
      rg[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < GTOT && tt < nt)
        rg[j] = *reinterpret_cast<const float4*>(
            g + ((size_t)(t0 + tt) * H + h) * DK + 4 * c4);
    }
    if (tid < kKdaTok * kKdaRows / 8) {
      const int tt = tid / (kKdaRows / 8), r8 = tid % (kKdaRows / 8);
      rv = make_uint4(0, 0, 0, 0);
      if (tt < nt)
        rv = *reinterpret_cast<const uint4*>(
            v + ((size_t)(t0 + tt) * H + h) * dv + row0 + 8 * r8);
    }
    if (tid < kKdaTok)
      rb = tid < nt ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
  };
  auto stage = [&]() {
#pragma unroll
    for (int j = 0; j < KCH; ++j) {
      const int e = tid + j * kKdaThreads, tt = e / (DK / 8), c8 = e % (DK / 8);
      if (e >= KTOT) continue;
      float f[8];
      unpack_bf16x8_f(rk[j], f);
#pragma unroll
      for (int x = 0; x < 8; ++x) sk[tt][8 * c8 + x] = f[x];
      unpack_bf16x8_f(rq[j], f);
#pragma unroll
      for (int x = 0; x < 8; ++x) sq[tt][8 * c8 + x] = f[x];
    }
#pragma unroll
    for (int j = 0; j < GCH; ++j) {
      const int e = tid + j * kKdaThreads, tt = e / (DK / 4), c4 = e % (DK / 4);
      if (e >= GTOT) continue;
      // exp(0) = 1 on the padding past a sequence's end
      *reinterpret_cast<float4*>(&sa[tt][4 * c4]) =
          make_float4(expf(rg[j].x), expf(rg[j].y), expf(rg[j].z), expf(rg[j].w));
    }
    if (tid < kKdaTok * kKdaRows / 8) {
      const int tt = tid / (kKdaRows / 8), r8 = tid % (kKdaRows / 8);
      float f[8];
      unpack_bf16x8_f(rv, f);
#pragma unroll
      for (int x = 0; x < 8; ++x) sv[tt][8 * r8 + x] = f[x];
    }
    if (tid < kKdaTok) sb[tid] = rb;
  };
  fetch(bos);
  for (long long t0 = bos; t0 < eos; t0 += kKdaTok) {
    const int nt = (int)min((long long)kKdaTok, eos - t0);
    __syncthreads();  // previous block consumed and written out
    stage();
    __syncthreads();
    if (t0 + kKdaTok < eos) fetch(t0 + kKdaTok);
    for (int tt = 0; tt < nt; ++tt) {
      float av[CPT], kv[CPT], qv[CPT];
      load_slice<CPT>(&sa[tt][CPT * lane], av);  // contiguous over the warp
      load_slice<CPT>(&sk[tt][CPT * lane], kv);
      load_slice<CPT>(&sq[tt][CPT * lane], qv);
      float p[kKdaRpw];
#pragma unroll
      for (int r = 0; r < kKdaRpw; ++r) {
        p[r] = 0.f;
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          S[r][j] *= av[j];
          p[r] = fmaf(S[r][j], kv[j], p[r]);
        }
      }
      // lane l ends with the warp's sum for row rr(l) (the lane's top bits):
      // halving exchanges (xor 16, then 8 for four rows) leave one value,
      // the remaining offsets add it up over the lane's group
      const int rr = lane / (32 / kKdaRpw);
      auto rowsum = [&](float (&x)[kKdaRpw]) {
#pragma unroll
        for (int nv = kKdaRpw, off = 16; nv > 1; nv >>= 1, off >>= 1) {
          const bool up = (lane & off) != 0;
#pragma unroll
          for (int j = 0; j < nv / 2; ++j) {
            const float give = up ? x[j] : x[j + nv / 2];
            const float keep = up ? x[j + nv / 2] : x[j];
            x[j] = keep + __shfl_xor_sync(0xffffffffu, give, off);
          }
        }
        float y = x[0];
#pragma unroll
        for (int off = 16 / kKdaRpw; off >= 1; off >>= 1)
          y += __shfl_xor_sync(0xffffffffu, y, off);
        return y;
      };
      const float pred = rowsum(p);
      const float ur = sb[tt] * (sv[tt][kKdaRpw * w + rr] - pred);
      float o[kKdaRpw];
#pragma unroll
      for (int r = 0; r < kKdaRpw; ++r) {
        const float u = __shfl_sync(0xffffffffu, ur, (32 / kKdaRpw) * r);
        o[r] = 0.f;
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          S[r][j] = fmaf(u, kv[j], S[r][j]);
          o[r] = fmaf(S[r][j], qv[j], o[r]);
        }
      }
      const float orow = rowsum(o);
      if (lane % (32 / kKdaRpw) == 0)
        so[tt][kKdaRpw * w + rr] = __float2bfloat16_rn(orow);
    }
    __syncthreads();
    // the block's outputs: 32 rows (64 bytes) per token
    for (int idx = tid; idx < nt * kKdaRows; idx += kKdaThreads) {
      const int tt = idx / kKdaRows, rr = idx % kKdaRows;
      out[((size_t)(t0 + tt) * H + h) * dv + row0 + rr] = so[tt][rr];
    }
  }
  if (hT) {
#pragma unroll
    for (int r = 0; r < kKdaRpw; ++r)
#pragma unroll
      for (int j = 0; j < CPT; ++j)
        hT[(nh * DK + CPT * lane + j) * dv + a0 + r] = S[r][j];
  }
}

}  // namespace

cudaError_t launch_kda(const KdaParams& p, cudaStream_t stream) {
  dim3 grid(p.dv / kKdaRows, p.H, p.N);
  const int t = timing_start(GDN_KERNEL_KDA, stream);
  auto go = [&](auto kern) {
    kern<<<grid, kKdaThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(p.q),
        static_cast<const __nv_bfloat16*>(p.k),
        static_cast<const __nv_bfloat16*>(p.v), p.g, p.beta, p.h0,
        static_cast<__nv_bfloat16*>(p.out), p.hT, p.cu_seqlens, p.H, p.T, p.dv,
        p.status);
  };
  if (p.dk == 64) go(kda_kernel<64>); else go(kda_kernel<128>);
  const cudaError_t e = cudaGetLastError();
  timing_stop(t, stream, e);
  return e;
}

}  // namespace gdn
