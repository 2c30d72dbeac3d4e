// Chunk-form backward of the scalar-gate recurrence (decay before the
// prediction), fp32 arithmetic: the adjoint of the UT/WY chunk form (the
// illustrated DeltaNet walk-through: UT transform, WY representation,
// chunkwise state passing; its cost table and memory paragraphs and the
// chunk form of "GPU parallelisation of Gated DeltaNet", m.lqnn.cn: keep the
// state at chunk boundaries, recompute inside). Per chunk of L <= 64 tokens
// with entry state S (d_v x d_k), G the chunk-local cumulative gate,
// E = e^G, D_rs = e^{G_r - G_s}:
//   A = strict_lower(diag(beta) K K^T (.) D),  T = (I + A)^{-1}
//   W = T diag(beta E) K,  U0 = T diag(beta) V,  U = U0 - W S^T
//   P = (Q K^T) (.) D (.) M_incl,  K_bar = diag(e^{G_L - G}) K
//   O = diag(E) Q S^T + P U,  S' = e^{G_L} S + U^T K_bar
// and, for the gradient dS' arriving at the exit state,
//   dU = P^T dO + K_bar dS'^T,  dS = e^{G_L} dS' + dO^T diag(E) Q - dU^T W
// (a reverse chain of the forward chain's shape) and, in parallel over
// chunks, dQ, dK, dV, dbeta, dG from S, dS', U, dU, T, P (the terms are
// written out in grad_body). Four bodies: prep (per chunk and head), the
// forward chain and the reverse chain (per 32 value rows, head, sequence),
// grad (per chunk and head). They are written over an execution context X
// (x.tid, x.nt, x.smem, x.sync()) so that the kernels instantiate them with
// one CUDA thread per tid; every loop bound is uniform across a CTA, so
// every thread reaches every x.sync().
#pragma once
#include <cstring>
#include <type_traits>
#ifdef __CUDACC__
#define GDN_HD __host__ __device__
#else
#define GDN_HD
#include <cmath>
#endif

namespace gdn {
namespace cbwd {

constexpr int C = 64;

// q, k, v, dout: bf16 (BF = true) or fp32 rows, read through ldin
struct Args {
  const void *q, *k, *v, *dout;
  const float *g, *beta, *h0, *dhT;
  int N, H, T, nch;  // nch = ceil(T / C)
  // workspace per chunk-head z = (n * nch + c) * H + h
  float *G, *Tm, *W, *U0, *P, *U, *S, *dSx, *dU;
  // per-chunk-head scratch of the gradient body
  float *dOS, *dKbar, *dW, *dKb, *dVb, *dP, *dT, *X, *dA, *KK, *dKs;
  // outputs
  float *dq, *dk, *dv, *dg, *dbeta, *dh0;
};

template <bool BF>
GDN_HD inline float ldin(const void* p, size_t i) {
  if (BF) {
    const unsigned int w = (unsigned int)static_cast<const unsigned short*>(p)[i] << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return f;
  }
  return static_cast<const float*>(p)[i];
}

// Shared-memory copies of the inputs: bf16 inputs stay bf16 bit patterns
// (exact, half the bytes), fp32 inputs stay fp32. tv reads either as fp32.
template <bool BF>
using tile_t = typename std::conditional<BF, unsigned short, float>::type;
GDN_HD inline float tv(float v) { return v; }
GDN_HD inline float tv(unsigned short u) {
  const unsigned int w = (unsigned int)u << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return f;
}
#ifdef __CUDA_ARCH__
// Eight consecutive bf16 values at element i of p (16-byte aligned), times s,
// into dst[0..7] (16-byte aligned); zeros without a read when !in.
__device__ __forceinline__ void ld8_bf16_scaled(float* dst, const void* p, size_t i,
                                                float s, bool in = true) {
  if (!in) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    reinterpret_cast<float4*>(dst)[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(p) + i);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  float f[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = __uint_as_float(w[e] << 16) * s;
    f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u) * s;
  }
  reinterpret_cast<float4*>(dst)[0] = make_float4(f[0], f[1], f[2], f[3]);
  reinterpret_cast<float4*>(dst)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
#endif

#ifdef __CUDA_ARCH__
// p[0], p[s], p[2s], p[3s] (four consecutive k) as fp32: one 16-byte (fp32)
// or 8-byte (bf16) load when s == 1 and the address allows it.
template <class T>
__device__ __forceinline__ void ld4k(const T* p, int s, float (&v)[4]) {
  if constexpr (std::is_same<T, unsigned short>::value) {
    if (s == 1 && (reinterpret_cast<uintptr_t>(p) & 7u) == 0) {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      v[0] = __uint_as_float(u.x << 16);
      v[1] = __uint_as_float(u.x & 0xffff0000u);
      v[2] = __uint_as_float(u.y << 16);
      v[3] = __uint_as_float(u.y & 0xffff0000u);
      return;
    }
  } else {
    if (s == 1 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
      const float4 f = *reinterpret_cast<const float4*>(p);
      v[0] = f.x;
      v[1] = f.y;
      v[2] = f.z;
      v[3] = f.w;
      return;
    }
  }
  v[0] = tv(p[0]);
  v[1] = tv(p[s]);
  v[2] = tv(p[2 * s]);
  v[3] = tv(p[3 * s]);
}
#endif

// Row padding of the shared-memory tiles, in elements: the products' fragment
// loads read 8 rows x 4 elements or 4 rows x 8 elements at a time, and a pad
// of 16 bytes (bf16) or 4 floats puts those rows in distinct banks.
template <bool BF>
constexpr int kPad = BF ? 8 : 4;
constexpr int kPadF = 4;  // fp32 state tiles

template <bool BF>
GDN_HD inline tile_t<BF> ldtile(const void* p, size_t i) {
  if constexpr (BF) return static_cast<const unsigned short*>(p)[i];
  else return static_cast<const float*>(p)[i];
}

#ifdef __CUDA_ARCH__
// fp32 x as a tf32 pair hi + lo (hi rounded to nearest, lo the rounded
// remainder): products of the pairs keep about fp32 accuracy.
__device__ __forceinline__ void tf32_split(float v, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(v));
  const float rest = v - __uint_as_float(hi);
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(rest));
}
// d += a b for one m16n8k8 tile (tf32 operands, fp32 accumulate).
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
#endif

// C[M][N] via epi(i, j, sum_k A(i,k) B(k,j)), A(i,k) = A[i*ars + k*acs],
// B(k,j) = B[k*brs + j*bcs]. Every output element is passed to epi exactly
// once, by one thread.
template <class X, class TA, class TB, class F>
GDN_HD void gemm(X& x, int M, int N, int K, const TA* A, int ars, int acs,
                 const TB* B, int brs, int bcs, F epi) {
#ifdef __CUDA_ARCH__
  // a bf16 operand is exact in tf32: its low part is zero and its two
  // products with it are skipped
  constexpr bool a_exact = std::is_same<TA, unsigned short>::value;
  constexpr bool b_exact = std::is_same<TB, unsigned short>::value;
  if (M % 16 == 0 && N % 32 == 0 && K % 8 == 0 && x.nt % 32 == 0) {
    // Tensor cores: each warp a 16 x 32 tile of C (four m16n8k8 tiles
    // sharing the A fragment), operands split into tf32 pairs and
    // multiplied as hi*hi + hi*lo + lo*hi, accumulated in fp32.
    // Fragment layout (m16n8k8, tf32): lane = 4 g + t; A rows g, g + 8 and
    // columns t, t + 4; B rows t, t + 4 and column g; C rows g, g + 8 and
    // columns 2t, 2t + 1.
    const int warp = x.tid >> 5, lane = x.tid & 31, nw = x.nt >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int tn = N / 32, ntiles = (M / 16) * tn;
    for (int tile = warp; tile < ntiles; tile += nw) {
      const int m0 = (tile / tn) * 16, n0 = (tile % tn) * 32;
      float acc[4][4];
      for (int q = 0; q < 4; ++q)
        for (int e = 0; e < 4; ++e) acc[q][e] = 0.f;
      if (K % 16 == 0) {
        // Sixteen k per step, two products: thread t takes k0 + 4t .. k0 +
        // 4t + 3, the first product 4t and 4t + 1 (fragment columns / rows
        // t and t + 4), the second 4t + 2 and 4t + 3. A and B take the same
        // k in the same slot, so the sums are those of the plain order, and
        // an operand contiguous in k is read with one vector load per row.
#pragma unroll 1
        for (int k0 = 0; k0 < K; k0 += 16) {
          float ar0[4], ar1[4];
          ld4k(A + (m0 + g) * ars + (k0 + 4 * t) * acs, acs, ar0);
          ld4k(A + (m0 + g + 8) * ars + (k0 + 4 * t) * acs, acs, ar1);
          uint32_t ah1[4], al1[4], ah2[4], al2[4];
          tf32_split(ar0[0], ah1[0], al1[0]);
          tf32_split(ar1[0], ah1[1], al1[1]);
          tf32_split(ar0[1], ah1[2], al1[2]);
          tf32_split(ar1[1], ah1[3], al1[3]);
          tf32_split(ar0[2], ah2[0], al2[0]);
          tf32_split(ar1[2], ah2[1], al2[1]);
          tf32_split(ar0[3], ah2[2], al2[2]);
          tf32_split(ar1[3], ah2[3], al2[3]);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int n = n0 + 8 * q + g;
            float br[4];
            ld4k(B + (k0 + 4 * t) * brs + n * bcs, brs, br);
            uint32_t bh[4], bl[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) tf32_split(br[e], bh[e], bl[e]);
            if (!a_exact) mma_tf32(acc[q], al1, bh[0], bh[1]);
            if (!b_exact) mma_tf32(acc[q], ah1, bl[0], bl[1]);
            mma_tf32(acc[q], ah1, bh[0], bh[1]);
            if (!a_exact) mma_tf32(acc[q], al2, bh[2], bh[3]);
            if (!b_exact) mma_tf32(acc[q], ah2, bl[2], bl[3]);
            mma_tf32(acc[q], ah2, bh[2], bh[3]);
          }
        }
      } else
#pragma unroll 4
      for (int k0 = 0; k0 < K; k0 += 8) {
        uint32_t ah[4], al[4];
        tf32_split(tv(A[(m0 + g) * ars + (k0 + t) * acs]), ah[0], al[0]);
        tf32_split(tv(A[(m0 + g + 8) * ars + (k0 + t) * acs]), ah[1], al[1]);
        tf32_split(tv(A[(m0 + g) * ars + (k0 + t + 4) * acs]), ah[2], al[2]);
        tf32_split(tv(A[(m0 + g + 8) * ars + (k0 + t + 4) * acs]), ah[3], al[3]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int n = n0 + 8 * q + g;
          uint32_t bh0, bl0, bh1, bl1;
          tf32_split(tv(B[(k0 + t) * brs + n * bcs]), bh0, bl0);
          tf32_split(tv(B[(k0 + t + 4) * brs + n * bcs]), bh1, bl1);
          if (!a_exact) mma_tf32(acc[q], al, bh0, bh1);
          if (!b_exact) mma_tf32(acc[q], ah, bl0, bl1);
          mma_tf32(acc[q], ah, bh0, bh1);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = n0 + 8 * q + 2 * t;
        epi(m0 + g, c, acc[q][0]);
        epi(m0 + g, c + 1, acc[q][1]);
        epi(m0 + g + 8, c, acc[q][2]);
        epi(m0 + g + 8, c + 1, acc[q][3]);
      }
    }
    return;
  }
#endif
  // thread (ti, tj) owns rows ti + m*M/4 and columns tj + n*N/4: neighbouring
  // threads read neighbouring columns of B (coalesced, and conflict-free in
  // shared memory when B's column stride is 1 or an odd number of floats)
  const int tm = M / 4, tn = N / 4, ntiles = tm * tn;
  for (int tile = x.tid; tile < ntiles; tile += x.nt) {
    const int ti = tile / tn, tj = tile % tn;
    float acc[4][4];
    for (int i = 0; i < 4; ++i)
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int kk = 0; kk < K; ++kk) {
      float a[4], b[4];
      for (int i = 0; i < 4; ++i) a[i] = tv(A[(ti + i * tm) * ars + kk * acs]);
      for (int j = 0; j < 4; ++j) b[j] = tv(B[kk * brs + (tj + j * tn) * bcs]);
      for (int i = 0; i < 4; ++i)
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    for (int i = 0; i < 4; ++i)
      for (int j = 0; j < 4; ++j) epi(ti + i * tm, tj + j * tn, acc[i][j]);
  }
}

GDN_HD inline int chunk_len(const Args& a, int c) {
  const int L = a.T - c * C;
  return L < C ? L : C;
}

// ---- 1. per (chunk, head): G, T = (I + A)^{-1}, W, U0, P -----------------
// smem floats: K, Q [C][DK], V [C][DV], A [C][C], T [C][C], G, beta [C]
template <int DK, int DV, bool BF>
constexpr int prep_smem() {
  return (2 * C * (DK + kPad<BF>) + C * (DV + kPad<BF>)) * (int)sizeof(tile_t<BF>) / 4 +
         2 * C * C + 2 * C;
}

template <int DK, int DV, bool BF, class X>
GDN_HD void prep_body(X& x, const Args& a, int z) {
  const int h = z % a.H, nc = z / a.H, c = nc % a.nch, n = nc / a.nch;
  const int L = chunk_len(a, c);
  const long long t0 = (long long)n * a.T + (long long)c * C;
  constexpr int LK = DK + kPad<BF>, LQ = DK + kPad<BF>, LV = DV + kPad<BF>;
  using TT = tile_t<BF>;
  TT* sK = reinterpret_cast<TT*>(x.smem);
  TT* sQ = sK + C * LK;
  TT* sV = sQ + C * LQ;
  float* sA = reinterpret_cast<float*>(sV + C * LV);
  float* sT = sA + C * C;
  float* sG = sT + C * C;
  float* sB = sG + C;
  for (int i = x.tid; i < C * DK; i += x.nt) {
    const int t = i / DK, cc = i % DK;
    const bool in = t < L;
    const size_t r = ((size_t)(t0 + t) * a.H + h) * DK + cc;
    sK[t * LK + cc] = in ? ldtile<BF>(a.k, r) : TT(0);
    sQ[t * LQ + cc] = in ? ldtile<BF>(a.q, r) : TT(0);
  }
  for (int i = x.tid; i < C * DV; i += x.nt) {
    const int t = i / DV, cc = i % DV;
    sV[t * LV + cc] = t < L ? ldtile<BF>(a.v, ((size_t)(t0 + t) * a.H + h) * DV + cc) : TT(0);
  }
  for (int t = x.tid; t < C; t += x.nt) {
    sB[t] = t < L ? a.beta[(size_t)(t0 + t) * a.H + h] : 0.f;
    sG[t] = t < L ? a.g[(size_t)(t0 + t) * a.H + h] : 0.f;
  }
  x.sync();
  if (x.tid == 0)
    for (int t = 1; t < C; ++t) sG[t] += sG[t - 1];  // padded g = 0
  x.sync();
  float* G = a.G + (size_t)z * C;
  for (int t = x.tid; t < C; t += x.nt) G[t] = sG[t];
  // A and P
  float* P = a.P + (size_t)z * C * C;
  gemm(x, C, C, DK, sK, LK, 1, sK, 1, LK, [&](int r, int s, float kk) {
    sA[r * C + s] = r > s ? sB[r] * kk * expf(sG[r] - sG[s]) : 0.f;
  });
  gemm(x, C, C, DK, sQ, LQ, 1, sK, 1, LK, [&](int r, int s, float qk) {
    P[r * C + s] = r >= s ? qk * expf(sG[r] - sG[s]) : 0.f;
  });
  x.sync();
  // T = (I + A)^{-1} (unit lower triangular) by 16 x 16 blocks: the four
  // diagonal blocks by substitution side by side (16 steps), then the
  // blocks below the diagonal one sub-diagonal at a time:
  //   T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj   (i > j)
  for (int i = x.tid; i < C * C; i += x.nt) {
    const int r = i / C, c2 = i % C;
    if (r / 16 != c2 / 16) sT[i] = 0.f;
  }
  for (int r = 0; r < 16; ++r) {
    for (int e = x.tid; e < 64; e += x.nt) {
      const int b = e / 16, j = e % 16, R = 16 * b + r, J = 16 * b + j;
      float t = r == j ? 1.f : 0.f;
      for (int s = j; s < r; ++s) t = fmaf(-sA[R * C + 16 * b + s], sT[(16 * b + s) * C + J], t);
      sT[R * C + J] = j <= r ? t : 0.f;
    }
    x.sync();
  }
  float* sM = sA;  // scratch rows: A's blocks on and above the diagonal are
                   // not read again (A_ik with k < i only)
  for (int dd = 1; dd < 4; ++dd) {
    // M_ij = sum_k A_ik T_kj for the blocks (i, j = i - dd), into the
    // (j, i) block of the scratch (above the diagonal)
    for (int e = x.tid; e < (4 - dd) * 256; e += x.nt) {
      const int bi = dd + e / 256, bj = bi - dd, r = (e % 256) / 16, c2 = e % 16;
      const int R = 16 * bi + r, J = 16 * bj + c2;
      float m = 0.f;
      for (int k = 16 * bj; k < 16 * bi; ++k) m = fmaf(sA[R * C + k], sT[k * C + J], m);
      sM[(16 * bj + r) * C + 16 * bi + c2] = m;
    }
    x.sync();
    // T_ij = -T_ii M_ij
    for (int e = x.tid; e < (4 - dd) * 256; e += x.nt) {
      const int bi = dd + e / 256, bj = bi - dd, r = (e % 256) / 16, c2 = e % 16;
      const int R = 16 * bi + r;
      float t = 0.f;
      for (int k = 0; k <= r; ++k)
        t = fmaf(sT[R * C + 16 * bi + k], sM[(16 * bj + k) * C + 16 * bi + c2], t);
      sT[R * C + 16 * bj + c2] = -t;
    }
    x.sync();
  }
  float* Tg = a.Tm + (size_t)z * C * C;
  for (int i = x.tid; i < C * C; i += x.nt) Tg[i] = sT[i];
  // W = (T diag(beta e^G)) K, U0 = (T diag(beta)) V: the factors scale the
  // columns of copies of T (T itself is stored above), so that K and V keep
  // their exact input values
  x.sync();
  float* sTW = sA;  // A and the merge scratch are not read again
  for (int i = x.tid; i < C * C; i += x.nt) {
    const int s2 = i % C;
    const float tt = sT[i];
    sTW[i] = tt * (sB[s2] * expf(sG[s2]));
    sT[i] = tt * sB[s2];
  }
  x.sync();
  float* W = a.W + (size_t)z * C * DK;
  float* U0 = a.U0 + (size_t)z * C * DV;
  gemm(x, C, DK, C, sTW, C, 1, sK, LK, 1, [&](int t, int cc, float s) { W[t * DK + cc] = s; });
  gemm(x, C, DV, C, sT, C, 1, sV, LV, 1, [&](int t, int cc, float s) { U0[t * DV + cc] = s; });
}

// ---- 2. forward chain: entry state S and U of every chunk ----------------
// one CTA per (RB value rows, head, sequence); smem: W, Kbar [C][DK],
// U0 [C][RB], S [RB][DK], U [C][RB], Snew [RB][DK]
template <int DK, int RB>
constexpr int fwd_smem() {
  return C * (DK + 4) + C * (DK + 8) + C * RB + 2 * RB * (DK + kPadF) + C * (RB + 8);
}

template <int DK, int DV, int RB, bool BF, class X>
GDN_HD void fwd_body(X& x, const Args& a, int rb, int h, int n) {
  // padded rows: a tile read as 8 rows x 4 elements by the products' fragment
  // loads gets 4 floats, one read as 4 rows x 8 elements 8 floats
  constexpr int LS = DK + kPadF, LW = DK + 4, LKb = DK + 8, LU = RB + 8;
  float* sW = x.smem;
  float* sKb = sW + C * LW;
  float* sU0 = sKb + C * LKb;
  float* sS = sU0 + C * RB;
  float* sU = sS + RB * LS;
  float* sSn = sU + C * LU;
  const int row0 = rb * RB;
  for (int i = x.tid; i < RB * DK; i += x.nt) {
    const int j = i / DK, cc = i % DK;
    sS[j * LS + cc] = a.h0 ? a.h0[(((size_t)n * a.H + h) * DK + cc) * DV + row0 + j] : 0.f;
  }
  for (int c = 0; c < a.nch; ++c) {
    const int z = (n * a.nch + c) * a.H + h, L = chunk_len(a, c);
    const long long t0 = (long long)n * a.T + (long long)c * C;
    const float* G = a.G + (size_t)z * C;
    const float GL = G[L - 1];
    x.sync();  // the previous chunk is done with the buffers
    // e^{G_L - G_t} once per token, in sU until U overwrites it
    for (int t = x.tid; t < C; t += x.nt) sU[t] = t < L ? expf(GL - G[t]) : 0.f;
    x.sync();
#ifdef __CUDA_ARCH__
    if constexpr (BF) {
      // 16-byte loads: W and U0 as float4, K eight bf16 at a time
      const float4* W4 = reinterpret_cast<const float4*>(a.W + (size_t)z * C * DK);
      for (int i = x.tid; i < C * DK / 4; i += x.nt)
        *reinterpret_cast<float4*>(sW + (4 * i / DK) * LW + 4 * i % DK) = W4[i];
      for (int i = x.tid; i < C * DK / 8; i += x.nt) {
        const int t = 8 * i / DK, cc = 8 * i % DK;
        ld8_bf16_scaled(sKb + t * LKb + cc, a.k, ((size_t)(t0 + t) * a.H + h) * DK + cc,
                        sU[t], t < L);
      }
      for (int i = x.tid; i < C * RB / 4; i += x.nt) {
        const int t = 4 * i / RB, j = 4 * i % RB;
        reinterpret_cast<float4*>(sU0)[i] =
            *reinterpret_cast<const float4*>(a.U0 + (size_t)z * C * DV + t * DV + row0 + j);
      }
    } else
#endif
    {
      for (int i = x.tid; i < C * DK; i += x.nt) {
        const int t = i / DK, cc = i % DK;
        sW[t * LW + cc] = a.W[(size_t)z * C * DK + i];
        sKb[t * LKb + cc] =
            t < L ? sU[t] * ldin<BF>(a.k, ((size_t)(t0 + t) * a.H + h) * DK + cc) : 0.f;
      }
      for (int i = x.tid; i < C * RB; i += x.nt) {
        const int t = i / RB, j = i % RB;
        sU0[i] = a.U0[(size_t)z * C * DV + t * DV + row0 + j];
      }
    }
    float* Sg = a.S + (size_t)z * DV * DK;
    for (int i = x.tid; i < RB * DK; i += x.nt)
      Sg[(size_t)row0 * DK + i] = sS[(i / DK) * LS + i % DK];
    x.sync();
    // U = U0 - W S^T (C x RB)
    float* Ug = a.U + (size_t)z * C * DV;
    gemm(x, C, RB, DK, sW, LW, 1, sS, 1, LS, [&](int t, int j, float ws) {
      const float u = sU0[t * RB + j] - ws;
      sU[t * LU + j] = u;
      Ug[t * DV + row0 + j] = u;
    });
    x.sync();
    // S <- gamma S + U^T Kbar (RB x DK)
    const float gam = expf(GL);
    gemm(x, RB, DK, C, sU, 1, LU, sKb, LKb, 1, [&](int j, int cc, float s) {
      sSn[j * LS + cc] = fmaf(gam, sS[j * LS + cc], s);
    });
    x.sync();
    for (int i = x.tid; i < RB * LS; i += x.nt) sS[i] = sSn[i];
  }
}

// ---- 3. reverse chain: exit gradient dS' and dU of every chunk -----------
// smem: P [C][C], dO [C][RB], Kbar, Qg, W [C][DK], dS, dSn [RB][DK], dU [C][RB]
template <int DK, int RB>
constexpr int rev_smem() {
  return C * (C + 8) + C * (RB + 8) + C * (DK + 4) + 2 * C * (DK + 8) + 2 * RB * (DK + kPadF) +
         C * (RB + 8);
}

template <int DK, int DV, int RB, bool BF, class X>
GDN_HD void rev_body(X& x, const Args& a, int rb, int h, int n) {
  // padded rows: a tile read as 8 rows x 4 elements by the products' fragment
  // loads gets 4 floats, one read as 4 rows x 8 elements 8 floats
  constexpr int LD = DK + kPadF, LP = C + 8, LO = RB + 8, LKb = DK + 4, LQg = DK + 8,
                LW = DK + 8, LdU = RB + 8;
  float* sP = x.smem;
  float* sO = sP + C * LP;
  float* sKb = sO + C * LO;
  float* sQg = sKb + C * LKb;
  float* sW = sQg + C * LQg;
  float* sD = sW + C * LW;
  float* sDn = sD + RB * LD;
  float* sdU = sDn + RB * LD;
  const int row0 = rb * RB;
  for (int i = x.tid; i < RB * DK; i += x.nt) {
    const int j = i / DK, cc = i % DK;
    sD[j * LD + cc] = a.dhT ? a.dhT[(((size_t)n * a.H + h) * DK + cc) * DV + row0 + j] : 0.f;
  }
  for (int c = a.nch - 1; c >= 0; --c) {
    const int z = (n * a.nch + c) * a.H + h, L = chunk_len(a, c);
    const long long t0 = (long long)n * a.T + (long long)c * C;
    const float* G = a.G + (size_t)z * C;
    const float GL = G[L - 1];
    x.sync();
    // e^{G_L - G_t} and e^{G_t} once per token, in sdU until dU overwrites it
    for (int t = x.tid; t < C; t += x.nt) {
      sdU[t] = t < L ? expf(GL - G[t]) : 0.f;
      sdU[C + t] = t < L ? expf(G[t]) : 0.f;
    }
    x.sync();
#ifdef __CUDA_ARCH__
    if constexpr (BF) {
      // 16-byte loads: P and W as float4, dO, K and Q eight bf16 at a time
      const float4* P4 = reinterpret_cast<const float4*>(a.P + (size_t)z * C * C);
      for (int i = x.tid; i < C * C / 4; i += x.nt)
        *reinterpret_cast<float4*>(sP + (4 * i / C) * LP + 4 * i % C) = P4[i];
      for (int i = x.tid; i < C * RB / 8; i += x.nt) {
        const int t = 8 * i / RB, j = 8 * i % RB;
        ld8_bf16_scaled(sO + t * LO + j, a.dout, ((size_t)(t0 + t) * a.H + h) * DV + row0 + j,
                        1.f, t < L);
      }
      for (int i = x.tid; i < C * DK / 8; i += x.nt) {
        const int t = 8 * i / DK, cc = 8 * i % DK;
        const bool in = t < L;
        const size_t r = ((size_t)(t0 + t) * a.H + h) * DK + cc;
        ld8_bf16_scaled(sKb + t * LKb + cc, a.k, r, sdU[t], in);
        ld8_bf16_scaled(sQg + t * LQg + cc, a.q, r, sdU[C + t], in);
      }
      const float4* W4 = reinterpret_cast<const float4*>(a.W + (size_t)z * C * DK);
      for (int i = x.tid; i < C * DK / 4; i += x.nt)
        *reinterpret_cast<float4*>(sW + (4 * i / DK) * LW + 4 * i % DK) = W4[i];
    } else
#endif
    {
      for (int i = x.tid; i < C * C; i += x.nt) sP[(i / C) * LP + i % C] = a.P[(size_t)z * C * C + i];
      for (int i = x.tid; i < C * RB; i += x.nt) {
        const int t = i / RB, j = i % RB;
        sO[t * LO + j] =
            t < L ? ldin<BF>(a.dout, ((size_t)(t0 + t) * a.H + h) * DV + row0 + j) : 0.f;
      }
      for (int i = x.tid; i < C * DK; i += x.nt) {
        const int t = i / DK, cc = i % DK;
        const bool in = t < L;
        const size_t r = ((size_t)(t0 + t) * a.H + h) * DK + cc;
        sKb[t * LKb + cc] = in ? sdU[t] * ldin<BF>(a.k, r) : 0.f;
        sQg[t * LQg + cc] = in ? sdU[C + t] * ldin<BF>(a.q, r) : 0.f;
        sW[t * LW + cc] = a.W[(size_t)z * C * DK + i];
      }
    }
    float* dSg = a.dSx + (size_t)z * DV * DK;
    for (int i = x.tid; i < RB * DK; i += x.nt)
      dSg[(size_t)row0 * DK + i] = sD[(i / DK) * LD + i % DK];
    x.sync();
    // dU = P^T dO + Kbar dS'^T (C x RB)
    float* dUg = a.dU + (size_t)z * C * DV;
    gemm(x, C, RB, DK, sKb, LKb, 1, sD, 1, LD, [&](int t, int j, float s) {
      sdU[t * LdU + j] = s;
    });
    x.sync();
    gemm(x, C, RB, C, sP, 1, LP, sO, LO, 1, [&](int t, int j, float s) {
      const float u = sdU[t * LdU + j] + s;
      sdU[t * LdU + j] = u;
      dUg[t * DV + row0 + j] = u;
    });
    x.sync();
    // dS = gamma dS' + dO^T Qg - dU^T W (RB x DK)
    const float gam = expf(GL);
    gemm(x, RB, DK, C, sO, 1, LO, sQg, LQg, 1, [&](int j, int cc, float s) {
      sDn[j * LD + cc] = fmaf(gam, sD[j * LD + cc], s);
    });
    x.sync();
    gemm(x, RB, DK, C, sdU, 1, LdU, sW, LW, 1, [&](int j, int cc, float s) {
      sDn[j * LD + cc] -= s;
    });
    x.sync();
    for (int i = x.tid; i < RB * LD; i += x.nt) sD[i] = sDn[i];
  }
  x.sync();
  if (a.dh0)
    for (int i = x.tid; i < RB * DK; i += x.nt) {
      const int j = i / DK, cc = i % DK;
      a.dh0[(((size_t)n * a.H + h) * DK + cc) * DV + row0 + j] = sD[j * LD + cc];
    }
}

// ---- 4. per (chunk, head): dq, dk, dv, dbeta, dg -------------------------
// smem: K, Q [C][DK], V, dO [C][DV], G, beta, E, ebar, dG [C], red [nt + 1]
template <int DK, int DV, bool BF>
constexpr int grad_smem(int nt) {
  return (2 * C * (DK + kPad<BF>) + 2 * C * (DV + kPad<BF>)) * (int)sizeof(tile_t<BF>) / 4 +
         5 * C + nt + 1;
}

template <int DK, int DV, bool BF, class X>
GDN_HD void grad_body(X& x, const Args& a, int z) {
  const int h = z % a.H, nc = z / a.H, c = nc % a.nch, n = nc / a.nch;
  const int L = chunk_len(a, c);
  const long long t0 = (long long)n * a.T + (long long)c * C;
  constexpr int LK = DK + kPad<BF>, LQ = DK + kPad<BF>, LV = DV + kPad<BF>,
                LO = DV + kPad<BF>;  // padded rows (fragment loads)
  using TT = tile_t<BF>;
  TT* sK = reinterpret_cast<TT*>(x.smem);
  TT* sQ = sK + C * LK;
  TT* sV = sQ + C * LQ;
  TT* sO = sV + C * LV;
  float* sG = reinterpret_cast<float*>(sO + C * LO);
  float* sB = sG + C;
  float* sE = sB + C;
  float* sEb = sE + C;
  float* sdG = sEb + C;
  float* red = sdG + C;
  for (int i = x.tid; i < C * DK; i += x.nt) {
    const int t = i / DK, cc = i % DK;
    const bool in = t < L;
    const size_t r = ((size_t)(t0 + t) * a.H + h) * DK + cc;
    sK[t * LK + cc] = in ? ldtile<BF>(a.k, r) : TT(0);
    sQ[t * LQ + cc] = in ? ldtile<BF>(a.q, r) : TT(0);
  }
  for (int i = x.tid; i < C * DV; i += x.nt) {
    const int t = i / DV, cc = i % DV;
    const bool in = t < L;
    const size_t r = ((size_t)(t0 + t) * a.H + h) * DV + cc;
    sV[t * LV + cc] = in ? ldtile<BF>(a.v, r) : TT(0);
    sO[t * LO + cc] = in ? ldtile<BF>(a.dout, r) : TT(0);
  }
  const float* G = a.G + (size_t)z * C;
  const float GL = G[L - 1];
  for (int t = x.tid; t < C; t += x.nt) {
    sG[t] = G[t];
    sB[t] = t < L ? a.beta[(size_t)(t0 + t) * a.H + h] : 0.f;
    sE[t] = t < L ? expf(G[t]) : 0.f;
    sEb[t] = t < L ? expf(GL - G[t]) : 0.f;
  }
  x.sync();
  const size_t zCK = (size_t)z * C * DK, zCV = (size_t)z * C * DV, zCC = (size_t)z * C * C;
  const float* S = a.S + (size_t)z * DV * DK;
  const float* dSx = a.dSx + (size_t)z * DV * DK;
  const float* U = a.U + zCV;
  const float* dU = a.dU + zCV;
  const float* Tm = a.Tm + zCC;
  const float* P = a.P + zCC;
  float *dOS = a.dOS + zCK, *dKbar = a.dKbar + zCK, *dW = a.dW + zCK;
  float *dKb = a.dKb + zCK, *dKs = a.dKs + zCK, *dVb = a.dVb + zCV;
  float *dP = a.dP + zCC, *dT = a.dT + zCC, *Xm = a.X + zCC, *dA = a.dA + zCC;
  float* KK = a.KK + zCC;
  // contractions over the value rows; K K^T
  gemm(x, C, DK, DV, sO, LO, 1, S, DK, 1, [&](int t, int cc, float s) { dOS[t * DK + cc] = s; });
  gemm(x, C, DK, DV, U, DV, 1, dSx, DK, 1, [&](int t, int cc, float s) { dKbar[t * DK + cc] = s; });
  gemm(x, C, DK, DV, dU, DV, 1, S, DK, 1, [&](int t, int cc, float s) { dW[t * DK + cc] = -s; });
  gemm(x, C, C, DV, sO, LO, 1, U, 1, DV, [&](int t, int s, float d) { dP[t * C + s] = t >= s ? d : 0.f; });
  gemm(x, C, C, DK, sK, LK, 1, sK, 1, LK, [&](int r, int s, float d) { KK[r * C + s] = d; });
  float part = 0.f;  // sum(dS' (.) S)
  for (int i = x.tid; i < DV * DK; i += x.nt) part = fmaf(dSx[i], S[i], part);
  red[x.tid] = part;
  x.sync();
  if (x.tid == 0) {
    float sd = 0.f;
    for (int i = 0; i < x.nt; ++i) sd += red[i];
    red[x.nt] = sd;
  }
  // dKb = T^T dW, dVb = T^T dU
  gemm(x, C, DK, C, Tm, 1, C, dW, DK, 1, [&](int t, int cc, float s) { dKb[t * DK + cc] = s; });
  gemm(x, C, DV, C, Tm, 1, C, dU, DV, 1, [&](int t, int cc, float s) { dVb[t * DV + cc] = s; });
  // dT = dW Kb^T + dU Vb^T, Kb = diag(beta E) K, Vb = diag(beta) V
  gemm(x, C, C, DK, dW, DK, 1, sK, 1, LK, [&](int r, int s, float d) { dT[r * C + s] = d * sB[s] * sE[s]; });
  x.sync();
  gemm(x, C, C, DV, dU, DV, 1, sV, 1, LV, [&](int r, int s, float d) { dT[r * C + s] += d * sB[s]; });
  x.sync();
  // X = T^T dT; dA = strict_lower(-X T^T)
  gemm(x, C, C, C, Tm, 1, C, dT, C, 1, [&](int r, int s, float d) { Xm[r * C + s] = d; });
  x.sync();
  gemm(x, C, C, C, Xm, C, 1, Tm, 1, C, [&](int r, int s, float d) { dA[r * C + s] = r > s ? -d : 0.f; });
  x.sync();
  // dbeta and dG per token t: on the device four lanes per token, each a
  // quarter of every sum, combined by shuffles; on the host one thread per
  // token
#ifdef __CUDA_ARCH__
  if (x.nt == 4 * C) {
    const int t = x.tid >> 2, q = x.tid & 3;
    float kdkb = 0.f, vdvb = 0.f, qdos = 0.f, kdkbar = 0.f, dbp = 0.f, dGp = 0.f;
    for (int cc = q; cc < DK; cc += 4) {
      kdkb = fmaf(tv(sK[t * LK + cc]), dKb[t * DK + cc], kdkb);
      qdos = fmaf(tv(sQ[t * LQ + cc]), dOS[t * DK + cc], qdos);
      kdkbar = fmaf(tv(sK[t * LK + cc]), dKbar[t * DK + cc], kdkbar);
    }
    for (int cc = q; cc < DV; cc += 4) vdvb = fmaf(tv(sV[t * LV + cc]), dVb[t * DV + cc], vdvb);
    for (int s = q; s < C; s += 4) {
      const float kk = KK[t * C + s];
      if (s < t) {
        const float D = expf(sG[t] - sG[s]);
        dbp = fmaf(dA[t * C + s] * D, kk, dbp);
        dGp = fmaf(dA[t * C + s], sB[t] * kk * D, dGp);
      }
      if (s > t) dGp -= dA[s * C + t] * sB[s] * kk * expf(sG[s] - sG[t]);
      if (s <= t) dGp = fmaf(dP[t * C + s], P[t * C + s], dGp);
      if (s >= t) dGp -= dP[s * C + t] * P[s * C + t];
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      kdkb += __shfl_xor_sync(0xffffffffu, kdkb, o);
      vdvb += __shfl_xor_sync(0xffffffffu, vdvb, o);
      qdos += __shfl_xor_sync(0xffffffffu, qdos, o);
      kdkbar += __shfl_xor_sync(0xffffffffu, kdkbar, o);
      dbp += __shfl_xor_sync(0xffffffffu, dbp, o);
      dGp += __shfl_xor_sync(0xffffffffu, dGp, o);
    }
    if (q == 0) {
      const float db = sE[t] * kdkb + vdvb + dbp;
      const float dG = sB[t] * sE[t] * kdkb + sE[t] * qdos - sEb[t] * kdkbar + dGp;
      if (t < L) a.dbeta[(size_t)(t0 + t) * a.H + h] = db;
      sdG[t] = dG;
      red[t] = sEb[t] * kdkbar;  // the partials above were summed into red[nt]
    }
  } else
#endif
  {
  for (int t = x.tid; t < C; t += x.nt) {
    float kdkb = 0.f, vdvb = 0.f, qdos = 0.f, kdkbar = 0.f;
    for (int cc = 0; cc < DK; ++cc) {
      kdkb = fmaf(tv(sK[t * LK + cc]), dKb[t * DK + cc], kdkb);
      qdos = fmaf(tv(sQ[t * LQ + cc]), dOS[t * DK + cc], qdos);
      kdkbar = fmaf(tv(sK[t * LK + cc]), dKbar[t * DK + cc], kdkbar);
    }
    for (int cc = 0; cc < DV; ++cc) vdvb = fmaf(tv(sV[t * LV + cc]), dVb[t * DV + cc], vdvb);
    float db = sE[t] * kdkb + vdvb;
    float dG = sB[t] * sE[t] * kdkb + sE[t] * qdos - sEb[t] * kdkbar;
    for (int s = 0; s < C; ++s) {
      const float kk = KK[t * C + s];
      if (s < t) {
        const float D = expf(sG[t] - sG[s]);
        db = fmaf(dA[t * C + s] * D, kk, db);
        dG = fmaf(dA[t * C + s], sB[t] * kk * D, dG);
      }
      if (s > t) dG -= dA[s * C + t] * sB[s] * kk * expf(sG[s] - sG[t]);
      if (s <= t) dG = fmaf(dP[t * C + s], P[t * C + s], dG);
      if (s >= t) dG -= dP[s * C + t] * P[s * C + t];
    }
    if (t < L) a.dbeta[(size_t)(t0 + t) * a.H + h] = db;
    sdG[t] = dG;
    red[t] = sEb[t] * kdkbar;  // the partials above were summed into red[nt]
  }
  }
  x.sync();
  if (x.tid == 0) {
    float kb = 0.f;
    for (int t = 0; t < L; ++t) kb += red[t];
    sdG[L - 1] += kb + expf(GL) * red[x.nt];
    float acc = 0.f;
    for (int t = L - 1; t >= 0; --t) {
      acc += sdG[t];
      a.dg[(size_t)(t0 + t) * a.H + h] = acc;
    }
  }
  // dP (.) D into X, B = diag(beta) (dA (.) D) into dT
  for (int i = x.tid; i < C * C; i += x.nt) {
    const int r = i / C, s = i % C;
    const float D = r >= s ? expf(sG[r] - sG[s]) : 0.f;
    Xm[i] = dP[i] * D;
    dT[i] = sB[r] * dA[i] * D;
  }
  x.sync();
  // dQ = diag(E) dOS + (dP (.) D) K
  gemm(x, C, DK, C, Xm, C, 1, sK, LK, 1, [&](int t, int cc, float s) {
    if (t < L) a.dq[((size_t)(t0 + t) * a.H + h) * DK + cc] = fmaf(sE[t], dOS[t * DK + cc], s);
  });
  // dK = (dP (.) D)^T Q + B K + B^T K + diag(ebar) dKbar + diag(beta E) dKb
  gemm(x, C, DK, C, Xm, 1, C, sQ, LQ, 1, [&](int s, int cc, float v) { dKs[s * DK + cc] = v; });
  x.sync();
  gemm(x, C, DK, C, dT, C, 1, sK, LK, 1, [&](int s, int cc, float v) { dKs[s * DK + cc] += v; });
  x.sync();
  gemm(x, C, DK, C, dT, 1, C, sK, LK, 1, [&](int s, int cc, float v) {
    const float r = dKs[s * DK + cc] + v + sEb[s] * dKbar[s * DK + cc] +
                    sB[s] * sE[s] * dKb[s * DK + cc];
    if (s < L) a.dk[((size_t)(t0 + s) * a.H + h) * DK + cc] = r;
  });
  // dV = diag(beta) dVb
  for (int i = x.tid; i < C * DV; i += x.nt) {
    const int t = i / DV, cc = i % DV;
    if (t < L) a.dv[((size_t)(t0 + t) * a.H + h) * DV + cc] = sB[t] * dVb[i];
  }
}

}  // namespace cbwd
}  // namespace gdn
