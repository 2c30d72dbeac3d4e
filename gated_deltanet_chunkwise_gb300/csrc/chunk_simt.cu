// Chunkwise Gated DeltaNet forward pass in fp32 CUDA-core arithmetic.
//
// Serves fp32 inputs (tensor cores at TF32 would not hold a 1e-3 bound after
// the triangular solve) and any bf16 request the tensor-core path does not
// take. One CTA owns (sequence, head, a DVT-row tile of the d_v x d_k state)
// and walks the sequence's chunks in order; per chunk it performs
//   (a) the gated UT/WY transform: A = strict_lower(diag(beta)(K K^T) (.) D'),
//       then W = (I + A)^{-1} diag(beta e^{G'}) K and U0 = (I + A)^{-1}
//       diag(beta) V by forward substitution, one column per thread
//       ("UT transform" page of the illustrated DeltaNet walk-through: the
//       unit-lower-triangular system solved by structure, no inverse);
//   (b) U = U0 - W S^T and S <- gamma S + U^T Kbar with Kbar = diag(e^{G_L-G})K
//       (its chunkwise state-passing paragraph, gated with the Gamma/gamma
//       prefixes of its GLA section);
//   (c) O = diag(e^G) Q S^T + ((Q K^T) (.) D (.) M_incl) U (its chunkwise
//       output paragraph; the diagonal is kept because the read follows the
//       write).
// D_rj = exp(G_r - G_j) with G the chunk-local cumulative log gate; D' uses
// G_{r-1} instead of G_r for GDN_GATE_AFTER_PREDICT. All exponents are <= 0.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kDVT = 32;  // state rows per CTA

template <int DK, int C>
struct SimtSmem {
  static constexpr int KP = DK + 1;        // padded K/Q row
  static constexpr int XW = DK + kDVT;     // solve width: W | U
  static constexpr int XP = XW + 1;
  static constexpr int CP = C + 1;
  static constexpr int kFloats = C * KP * 2 + C * XP + C * CP * 2 +
                                 kDVT * KP + C * kDVT + 5 * C;
  static constexpr size_t kBytes = sizeof(float) * kFloats;
};

template <typename InT, int DK, int C, int VARIANT>
__global__ void __launch_bounds__(kThreads)
    chunk_simt_kernel(const ChunkParams p) {
  using L = SimtSmem<DK, C>;
  extern __shared__ float smem[];
  float* sK = smem;                 // [C][KP]
  float* sQ = sK + C * L::KP;       // [C][KP]
  float* sX = sQ + C * L::KP;       // [C][XP]  W | U0 -> U
  float* sA = sX + C * L::XP;       // [C][CP]  strict-lower system matrix
  float* sP = sA + C * L::CP;       // [C][CP]  gated causal scores
  float* sS = sP + C * L::CP;       // [DVT][KP] state rows (fp32)
  float* sV = sS + kDVT * L::KP;    // [C][DVT] V tile, then history read
  float* sG = sV + C * kDVT;        // [C] cumulative log gate
  float* sGp = sG + C;              // [C] prediction exponent base
  float* sB = sGp + C;              // [C] beta
  float* sRaw = sB + C;             // [C] raw g
  float* sDec = sRaw + C;           // [C] exp(G_last - G_r)

  const int tid = threadIdx.x;
  const int H = p.H, dv = p.dv;
  const int h = blockIdx.y;
  const int n = blockIdx.z / p.part_count;
  const int part = p.part_begin + blockIdx.z % p.part_count;
  const int row0 = blockIdx.x * kDVT;

  // Role of this CTA.
  const bool value_rows = row0 < dv;
  const bool split_tail = (p.mode == kModeSplit) && part > 0;
  if (!value_rows && !(split_tail && row0 < dv + DK)) return;
  const bool scale_rows = !value_rows;              // rows of M
  const bool emit = (p.mode == kModeOutput) || part == 0;

  long long bos, eos;
  if (!sequence_range(p, n, bos, eos)) return;
  const int nch = (int)((eos - bos + C - 1) / C);
  int c_begin, c_end;
  part_range(nch, p.parts, part, c_begin, c_end);

  const InT* q = static_cast<const InT*>(p.q);
  const InT* k = static_cast<const InT*>(p.k);
  const InT* v = static_cast<const InT*>(p.v);
  InT* out = static_cast<InT*>(p.out);
  const size_t nh = (size_t)n * H + h;

  // ---- initial state rows ----
  for (int idx = tid; idx < kDVT * DK; idx += kThreads) {
    const int i = idx / kDVT, c = idx % kDVT;  // c fastest: coalesced h0 read
    float s = 0.f;
    if (scale_rows) {
      s = (i == row0 - dv + c) ? 1.f : 0.f;
    } else if (split_tail) {
      s = 0.f;
    } else if (part > 0) {
      s = p.ws_start[((nh * p.parts + part) * dv + row0 + c) * DK + i];
    } else if (p.h0) {
      s = p.h0[(nh * DK + i) * dv + row0 + c];
    }
    sS[c * L::KP + i] = s;
  }

  for (int ch = c_begin; ch < c_end; ++ch) {
    const long long t0 = bos + (long long)ch * C;
    const int len = (int)min((long long)C, eos - t0);
    __syncthreads();  // previous chunk done with the tiles

    // ---- load K, Q (zero past the sequence end), V tile, g, beta ----
    for (int idx = tid; idx < C * DK; idx += kThreads) {
      const int r = idx / DK, i = idx % DK;
      float kv = 0.f, qv = 0.f;
      if (r < len) {
        const size_t row = (size_t)(t0 + r) * H + h;
        kv = to_f32(k[row * DK + i]);
        qv = to_f32(q[row * DK + i]);
      }
      sK[r * L::KP + i] = kv;
      sQ[r * L::KP + i] = qv;
    }
    for (int idx = tid; idx < C * kDVT; idx += kThreads) {
      const int r = idx / kDVT, c = idx % kDVT;
      float vv = 0.f;
      if (r < len && value_rows) {
        const size_t row = (size_t)(t0 + r) * H + h;
        vv = to_f32(v[row * dv + row0 + c]);
      }
      sV[r * kDVT + c] = vv;
    }
    if (tid < C) {
      float gg = 0.f, bb = 0.f;
      if (tid < len) {
        const size_t row = (size_t)(t0 + tid) * H + h;
        gg = p.g[row];
        bb = p.beta[row];
      }
      sRaw[tid] = gg;
      sB[tid] = bb;
    }
    __syncthreads();
    if (tid == 0) {
      float acc = 0.f;
      for (int r = 0; r < C; ++r) {
        acc += sRaw[r];
        sG[r] = acc;
        sGp[r] = VARIANT == GDN_GATE_BEFORE_PREDICT ? acc : acc - sRaw[r];
      }
    }
    __syncthreads();
    const float Glast = sG[C - 1];
    if (tid < C) sDec[tid] = expf(Glast - sG[tid]);

    // ---- system matrix A and gated scores P ----
    for (int idx = tid; idx < C * C; idx += kThreads) {
      const int r = idx / C, j = idx % C;
      float a = 0.f, pp = 0.f;
      if (j <= r) {
        float kk = 0.f, qk = 0.f;
#pragma unroll 8
        for (int i = 0; i < DK; ++i) {
          const float kj = sK[j * L::KP + i];
          kk = fmaf(sK[r * L::KP + i], kj, kk);
          qk = fmaf(sQ[r * L::KP + i], kj, qk);
        }
        pp = expf(sG[r] - sG[j]) * qk;
        if (j < r) a = sB[r] * expf(sGp[r] - sG[j]) * kk;
      }
      sA[r * L::CP + j] = a;
      sP[r * L::CP + j] = pp;
    }
    __syncthreads();

    // ---- forward substitution: (I + A) X = [diag(beta e^G') K | diag(beta) V]
    if (tid < L::XW) {
      const int col = tid;
      for (int r = 0; r < C; ++r) {
        float x = col < DK ? sB[r] * expf(sGp[r]) * sK[r * L::KP + col]
                           : sB[r] * sV[r * kDVT + (col - DK)];
        for (int j = 0; j < r; ++j)
          x = fmaf(-sA[r * L::CP + j], sX[j * L::XP + col], x);
        sX[r * L::XP + col] = x;
      }
    }
    __syncthreads();

    // ---- U = U0 - W S^T ; history read e^{G} Q S^T (into sV) ----
    for (int idx = tid; idx < C * kDVT; idx += kThreads) {
      const int r = idx / kDVT, c = idx % kDVT;
      float ws = 0.f, qs = 0.f;
#pragma unroll 8
      for (int i = 0; i < DK; ++i) {
        const float s = sS[c * L::KP + i];
        ws = fmaf(sX[r * L::XP + i], s, ws);
        qs = fmaf(sQ[r * L::KP + i], s, qs);
      }
      sX[r * L::XP + DK + c] -= ws;
      sV[r * kDVT + c] = expf(sG[r]) * qs;
    }
    __syncthreads();

    // ---- output rows (read after the write: j <= r) ----
    if (emit) {
      for (int idx = tid; idx < C * kDVT; idx += kThreads) {
        const int r = idx / kDVT, c = idx % kDVT;
        if (r < len) {
          float o = sV[r * kDVT + c];
          for (int j = 0; j <= r; ++j)
            o = fmaf(sP[r * L::CP + j], sX[j * L::XP + DK + c], o);
          const size_t row = (size_t)(t0 + r) * H + h;
          out[row * dv + row0 + c] = from_f32<InT>(o);
        }
      }
    }
    // ---- state: S <- gamma S + U^T Kbar ----
    const float gam = expf(Glast);
    for (int idx = tid; idx < kDVT * DK; idx += kThreads) {
      const int c = idx / DK, i = idx % DK;
      float acc = 0.f;
#pragma unroll 8
      for (int r = 0; r < C; ++r)
        acc = fmaf(sX[r * L::XP + DK + c] * sDec[r], sK[r * L::KP + i], acc);
      sS[c * L::KP + i] = fmaf(gam, sS[c * L::KP + i], acc);
    }
  }
  __syncthreads();

  // ---- final state ----
  if (p.mode == kModeSplit) {
    if (part == 0) {
      if (p.parts > 1)
        for (int idx = tid; idx < kDVT * DK; idx += kThreads) {
          const int c = idx / DK, i = idx % DK;
          p.ws_start[((nh * p.parts + 1) * dv + row0 + c) * DK + i] =
              sS[c * L::KP + i];
        }
    } else {
      for (int idx = tid; idx < kDVT * DK; idx += kThreads) {
        const int c = idx / DK, i = idx % DK;
        p.ws_end[((nh * p.parts + part) * (dv + DK) + row0 + c) * DK + i] =
            sS[c * L::KP + i];
      }
    }
  } else if (p.hT && part == p.parts - 1) {
    for (int idx = tid; idx < kDVT * DK; idx += kThreads) {
      const int i = idx / kDVT, c = idx % kDVT;
      p.hT[(nh * DK + i) * dv + row0 + c] = sS[c * L::KP + i];
    }
  }
}

// Serial correction chain over sub-sequences (the CP=4 chain of the sequence
// parallelism note): S_start(p + 1) = dS_end(p) + S_start(p) M_end(p) for
// p = 1 .. parts - 2; S_start(1) was written by part 0 of the split pass.
// One CTA per (sequence, head, kSpRows state rows); M_end(p) (dk x dk) is staged
// in shared memory by asynchronous copies, the next part's while this one is
// multiplied, and each thread forms a RPT x 4 block of the product in fp32
// registers (rows from a broadcast, four columns per 16-byte load).
constexpr int kSpRows = 16;
template <int DK>
struct SpChainSmem {
  static constexpr int kS = kSpRows * (DK + 4);  // start rows, padded
  static constexpr size_t kBytes = (size_t)(kS + 2 * DK * DK) * sizeof(float);
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(smem)),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int DK>
__global__ void __launch_bounds__(kThreads) sp_chain_kernel(const ChunkParams p) {
  constexpr int CG = DK / 4;             // column groups of four
  constexpr int RG = kThreads / CG;      // row groups
  constexpr int RPT = kSpRows / RG;         // rows per thread
  static_assert(RG * RPT == kSpRows && CG * RG == kThreads, "sp chain tiling");
  constexpr int SP = DK + 4;             // padded pitch of the start rows
  extern __shared__ float sp_smem[];
  float* sS = sp_smem;                   // [kSpRows][SP]
  float* sM0 = sp_smem + SpChainSmem<DK>::kS;  // [2][DK][DK]
  const int tid = threadIdx.x;
  const int cg = tid % CG, rg = tid / CG;
  const int h = blockIdx.y, n = blockIdx.z;
  const int row0 = blockIdx.x * kSpRows;
  const int dv = p.dv;
  const size_t nh = (size_t)n * p.H + h;
  if (p.cu_seqlens) {
    long long bos, eos;
    if (!sequence_range(p, n, bos, eos)) return;
  }
  for (int idx = tid; idx < kSpRows * DK / 4; idx += kThreads) {
    const int c = idx / (DK / 4), i4 = idx % (DK / 4);
    *reinterpret_cast<float4*>(sS + c * SP + 4 * i4) =
        reinterpret_cast<const float4*>(
            p.ws_start + ((nh * p.parts + 1) * dv + row0 + c) * DK)[i4];
  }
  auto stage_m = [&](int part) {
    const float4* M4 = reinterpret_cast<const float4*>(
        p.ws_end + (nh * p.parts + part) * (size_t)(dv + DK) * DK + (size_t)dv * DK);
    float4* dst = reinterpret_cast<float4*>(sM0 + (part & 1) * DK * DK);
    for (int idx = tid; idx < DK * DK / 4; idx += kThreads)
      cp_async16(dst + idx, M4 + idx);
    cp_async_commit();
  };
  if (p.parts > 2) stage_m(1);
  for (int part = 1; part + 1 < p.parts; ++part) {
    const float* end = p.ws_end + (nh * p.parts + part) * (size_t)(dv + DK) * DK;
    const float* sM = sM0 + (part & 1) * DK * DK;
    // the other buffer was last read before the barrier that ended the
    // previous part
    if (part + 2 < p.parts) {
      stage_m(part + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    float acc[RPT][4];
#pragma unroll
    for (int a = 0; a < RPT; ++a) {
      const float4 d4 = reinterpret_cast<const float4*>(
          end + (size_t)(row0 + rg * RPT + a) * DK)[cg];
      acc[a][0] = d4.x; acc[a][1] = d4.y; acc[a][2] = d4.z; acc[a][3] = d4.w;
    }
    __syncthreads();  // M staged (and the start rows of this part)
#pragma unroll 4
    for (int i = 0; i < DK; ++i) {
      const float4 m = reinterpret_cast<const float4*>(sM + i * DK)[cg];
#pragma unroll
      for (int a = 0; a < RPT; ++a) {
        const float sv = sS[(rg * RPT + a) * SP + i];
        acc[a][0] = fmaf(sv, m.x, acc[a][0]);
        acc[a][1] = fmaf(sv, m.y, acc[a][1]);
        acc[a][2] = fmaf(sv, m.z, acc[a][2]);
        acc[a][3] = fmaf(sv, m.w, acc[a][3]);
      }
    }
    __syncthreads();  // every thread done with S and M of this part
#pragma unroll
    for (int a = 0; a < RPT; ++a) {
      const int c = rg * RPT + a;
      const float4 v4 = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
      *reinterpret_cast<float4*>(sS + c * SP + 4 * cg) = v4;
      reinterpret_cast<float4*>(
          p.ws_start + ((nh * p.parts + part + 1) * dv + row0 + c) * DK)[cg] = v4;
    }
  }
}

// Associative-scan alternative to the serial chain ([lqnn] section 3.4: the
// chunk-level prefix scan, Hillis-Steele). Sub-sequence p >= 1 of the split
// pass is the affine map f_p(S) = S M_p + dS_p (ws_end entry p: dS rows
// 0 .. dv-1, M rows dv .. dv+dk-1). Maps compose associatively,
//   f_b after f_a = (M_a M_b, dS_a M_b + dS_b),
// so the inclusive prefixes G_p = f_p after ... after f_1, p = 1 .. L = P-2,
// take ceil(log2 L) rounds: in the round with offset d every map p > d
// becomes G_{p-d}-part after it. Then S_start(p + 1) = S_start(1) M^G_p +
// dS^G_p. One kernel does both: rows of X times M plus an added row, for
// kScanRows rows of one map per CTA (every CTA stages the map's whole M, so
// the rows per CTA set how often M is read).
//   combine: X = src[p - d] (all dv + dk rows), M = src[p].M, added row =
//            src[p].dS (dS rows only); maps p <= d are copied
//   apply:   X = ws_start[1] (dv rows), M = src[p].M, added row = src[p].dS,
//            written to ws_start[p + 1]
constexpr int kScanRows = 64;
template <int DK>
struct SpAffineSmem {
  static constexpr int kS = kScanRows * (DK + 4);
  static constexpr size_t kBytes = (size_t)(kS + DK * DK) * sizeof(float);
};

template <int DK>
__global__ void __launch_bounds__(kThreads)
    sp_affine_kernel(const ChunkParams p, const float* src, float* dst, int d,
                     int apply) {
  constexpr int CG = DK / 4, RG = kThreads / CG, RPT = kScanRows / RG;
  static_assert(RG * RPT == kScanRows && CG * RG == kThreads, "tiling");
  constexpr int SP = DK + 4;
  extern __shared__ float af_smem[];
  float* sX = af_smem;                          // [kScanRows][SP]
  float* sM = af_smem + SpAffineSmem<DK>::kS;   // [DK][DK]
  const int tid = threadIdx.x;
  const int cg = tid % CG, rg = tid / CG;
  const int dv = p.dv, L = p.parts - 2;
  const int h = blockIdx.y, n = blockIdx.z / L, m = blockIdx.z % L + 1;
  const int row0 = blockIdx.x * kScanRows;
  if (p.cu_seqlens) {
    long long bos, eos;
    if (!sequence_range(p, n, bos, eos)) return;
  }
  const size_t nh = (size_t)n * p.H + h;
  const size_t entry = (size_t)(dv + DK) * DK;
  const float* sp = src + (nh * p.parts + m) * entry;  // map m
  float* out;
  const float* xr;
  if (apply) {
    out = p.ws_start + ((nh * p.parts + m + 1) * dv + row0) * DK;
    xr = p.ws_start + ((nh * p.parts + 1) * dv + row0) * DK;
  } else {
    out = dst + (nh * p.parts + m) * entry + (size_t)row0 * DK;
    if (m <= d) {
      // already a full prefix: carried over
      for (int idx = tid; idx < kScanRows * DK / 4; idx += kThreads)
        reinterpret_cast<float4*>(out)[idx] =
            reinterpret_cast<const float4*>(sp + (size_t)row0 * DK)[idx];
      return;
    }
    xr = src + (nh * p.parts + m - d) * entry + (size_t)row0 * DK;
  }
  for (int idx = tid; idx < kScanRows * DK / 4; idx += kThreads) {
    const int c = idx / (DK / 4), i4 = idx % (DK / 4);
    *reinterpret_cast<float4*>(sX + c * SP + 4 * i4) =
        reinterpret_cast<const float4*>(xr + (size_t)c * DK)[i4];
  }
  const float4* M4 = reinterpret_cast<const float4*>(sp + (size_t)dv * DK);
  for (int idx = tid; idx < DK * DK / 4; idx += kThreads)
    reinterpret_cast<float4*>(sM)[idx] = M4[idx];
  float acc[RPT][4];
#pragma unroll
  for (int a = 0; a < RPT; ++a) {
    const int r = row0 + rg * RPT + a;  // row of the map (dS rows first)
    float4 d4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < dv) d4 = reinterpret_cast<const float4*>(sp + (size_t)r * DK)[cg];
    acc[a][0] = d4.x; acc[a][1] = d4.y; acc[a][2] = d4.z; acc[a][3] = d4.w;
  }
  __syncthreads();
#pragma unroll 4
  for (int i = 0; i < DK; ++i) {
    const float4 mv = reinterpret_cast<const float4*>(sM + i * DK)[cg];
#pragma unroll
    for (int a = 0; a < RPT; ++a) {
      const float xv = sX[(rg * RPT + a) * SP + i];
      acc[a][0] = fmaf(xv, mv.x, acc[a][0]);
      acc[a][1] = fmaf(xv, mv.y, acc[a][1]);
      acc[a][2] = fmaf(xv, mv.z, acc[a][2]);
      acc[a][3] = fmaf(xv, mv.w, acc[a][3]);
    }
  }
#pragma unroll
  for (int a = 0; a < RPT; ++a)
    reinterpret_cast<float4*>(out + (size_t)(rg * RPT + a) * DK)[cg] =
        make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
}

template <typename InT, int DK, int VARIANT>
cudaError_t launch_typed(const ChunkParams& p, cudaStream_t stream) {
  constexpr int C = 64;
  auto kern = chunk_simt_kernel<InT, DK, C, VARIANT>;
  const size_t bytes = SimtSmem<DK, C>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  const int rows = p.mode == kModeSplit ? p.dv + DK : p.dv;
  dim3 grid(rows / kDVT, p.H, p.N * p.part_count);
  const int t = timing_start(GDN_KERNEL_CHUNK_SIMT, stream);
  kern<<<grid, kThreads, bytes, stream>>>(p);
  e = cudaGetLastError();
  timing_stop(t, stream, e);
  return e;
}

template <typename InT>
cudaError_t launch_dk(const ChunkParams& p, cudaStream_t stream) {
  const bool after = p.variant == GDN_GATE_AFTER_PREDICT;
  if (p.dk == 64)
    return after ? launch_typed<InT, 64, GDN_GATE_AFTER_PREDICT>(p, stream)
                 : launch_typed<InT, 64, GDN_GATE_BEFORE_PREDICT>(p, stream);
  return after ? launch_typed<InT, 128, GDN_GATE_AFTER_PREDICT>(p, stream)
               : launch_typed<InT, 128, GDN_GATE_BEFORE_PREDICT>(p, stream);
}

}  // namespace

cudaError_t launch_chunk_simt(const ChunkParams& p, bool bf16,
                              cudaStream_t stream) {
  return bf16 ? launch_dk<__nv_bfloat16>(p, stream)
              : launch_dk<float>(p, stream);
}

cudaError_t launch_sp_chain(const ChunkParams& p, cudaStream_t stream) {
  if (p.parts < 3) return cudaSuccess;
  dim3 grid(p.dv / kSpRows, p.H, p.N);
  const int t = timing_start(GDN_KERNEL_SP_CHAIN, stream);
  cudaError_t e = cudaSuccess;
  if (p.dk == 64) {
    e = cudaFuncSetAttribute(sp_chain_kernel<64>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SpChainSmem<64>::kBytes);
    if (e == cudaSuccess)
      sp_chain_kernel<64><<<grid, kThreads, SpChainSmem<64>::kBytes, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(sp_chain_kernel<128>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SpChainSmem<128>::kBytes);
    if (e == cudaSuccess)
      sp_chain_kernel<128><<<grid, kThreads, SpChainSmem<128>::kBytes, stream>>>(p);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  timing_stop(t, stream, e);
  return e;
}

// The associative-scan combination (sp_affine_kernel): ceil(log2 L) combine
// rounds ping-ponging between ws_end and `buf` (same size as ws_end), then
// the apply launch. Returns the launch result; *launches counts launches.
cudaError_t launch_sp_scan(const ChunkParams& p, float* buf,
                           cudaStream_t stream, int* launches) {
  *launches = 0;
  if (p.parts < 3) return cudaSuccess;
  const int L = p.parts - 2;
  auto kern = p.dk == 64 ? sp_affine_kernel<64> : sp_affine_kernel<128>;
  const size_t bytes = p.dk == 64 ? SpAffineSmem<64>::kBytes
                                  : SpAffineSmem<128>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  const float* src = p.ws_end;
  float* dst = buf;
  for (int d = 1; d < L; d *= 2) {
    const int t = timing_start(GDN_KERNEL_SP_CHAIN, stream);
    kern<<<dim3((p.dv + p.dk) / kScanRows, p.H, p.N * L), kThreads, bytes,
           stream>>>(p, src, dst, d, 0);
    e = cudaGetLastError();
    timing_stop(t, stream, e);
    if (e != cudaSuccess) return e;
    ++*launches;
    src = dst;
    dst = dst == buf ? p.ws_end : buf;
  }
  const int t = timing_start(GDN_KERNEL_SP_CHAIN, stream);
  kern<<<dim3(p.dv / kScanRows, p.H, p.N * L), kThreads, bytes, stream>>>(
      p, src, nullptr, 0, 1);
  e = cudaGetLastError();
  timing_stop(t, stream, e);
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace gdn
