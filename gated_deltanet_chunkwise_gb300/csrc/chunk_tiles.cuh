// Pieces shared by the tensor-core preparation kernels (Gated DeltaNet and
// KDA) and the chain kernels: chunk geometry, the layout of the per-(chunk,
// head) workspace images, the chunk-to-sequence lookup, the small tf32
// products and the blocked unit-lower-triangular inverse (illustrated
// DeltaNet walk-through, UT transform section), and the bf16 tile writers.
#pragma once

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {
using namespace tc;

constexpr int C = 64;
constexpr int DK = 128;
constexpr int DVT = 64;
constexpr int AP = 68;  // fp32 row pitch of the solve buffer

// Gate vectors of one chunk (written by one warp): cumulative log gate G,
// alpha = e^g, e^G, beta e^{G'}, beta, e^{G_L - G}, e^{-G}, gamma = e^{G_L},
// and whether e^{G_r} e^{-G_j} stays in the normal fp32 range; then the
// inverse lengths of the chunk's k and q rows (1 when they come normalised).
constexpr int VEC_G = 0, VEC_ALPHA = 64, VEC_EG = 128, VEC_EGPB = 192,
              VEC_BETA = 256, VEC_DEC = 320, VEC_IEG = 384, VEC_GAMMA = 448,
              VEC_SAFE = 449, VEC_SK = 452, VEC_SQ = 516, VEC_FLOATS = 580;
// The part of them the chain kernel reads, per (chunk, head) in the
// workspace: e^G, e^{G_L - G}, gamma (padded to a multiple of 16 bytes).
constexpr int CV_EG = 0, CV_DEC = 64, CV_GAMMA = 128, CV_FLOATS = 132;
constexpr uint32_t CV_BYTES = CV_FLOATS * 4;

// Chunk `c` of the whole call -> (sequence n, chunk index within n).
__device__ __forceinline__ void locate_chunk(const ChunkParams& p, int c,
                                             int nch_dense, int& n, int& lc) {
  if (!p.chunk_off) {
    n = c / nch_dense;
    lc = c - n * nch_dense;
    return;
  }
  int lo = 0, hi = p.N;  // chunk_off[lo] <= c < chunk_off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.chunk_off[mid] <= c) lo = mid; else hi = mid;
  }
  n = lo;
  lc = c - p.chunk_off[lo];
}

__device__ __forceinline__ int chunk_base(const ChunkParams& p, int n,
                                          int nch_dense) {
  return p.chunk_off ? p.chunk_off[n] : n * nch_dense;
}

// AND of `v` over the threads of named barrier `id` (also a barrier).

__device__ __forceinline__ bool bar_and(int id, int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q, p;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ bool wait_ignoring_abort(uint64_t* bar,
                                                    uint32_t parity) {
  int local = 0;
  return mbar_wait(bar, parity, &local);
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&x)[64]) {
  float (&lo)[32] = *reinterpret_cast<float(*)[32]>(&x[0]);
  float (&hi)[32] = *reinterpret_cast<float(*)[32]>(&x[32]);
  tmem_ld32(taddr, lo);
  tmem_ld32(taddr + 32, hi);
  tmem_ld_wait();
}

// ---------------------------------------------------------------------------
// Small tensor-core products for the triangular solve: mma.sync m16n8k8 with
// tf32 inputs and fp32 accumulation, fragments loaded from row-major fp32
// tiles of pitch AP (conflict-free for the A fragment since AP = 4 mod 32).
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

struct FragA { uint32_t a[4]; };
struct FragB { uint32_t b[2]; };

// 16 x 8 tile of a row-major matrix at (r0, c0).
__device__ __forceinline__ FragA load_frag_a(const float* X, int r0, int c0,
                                             int lane) {
  const int g = lane >> 2, t = lane & 3;
  FragA f;
  f.a[0] = to_tf32(X[(r0 + g) * AP + c0 + t]);
  f.a[1] = to_tf32(X[(r0 + g + 8) * AP + c0 + t]);
  f.a[2] = to_tf32(X[(r0 + g) * AP + c0 + t + 4]);
  f.a[3] = to_tf32(X[(r0 + g + 8) * AP + c0 + t + 4]);
  return f;
}

// 8 x 8 tile (k rows, n columns) of a row-major matrix at (k0, n0).
__device__ __forceinline__ FragB load_frag_b(const float* X, int k0, int n0,
                                             int lane) {
  const int g = lane >> 2, t = lane & 3;
  FragB f;
  f.b[0] = to_tf32(X[(k0 + t) * AP + n0 + g]);
  f.b[1] = to_tf32(X[(k0 + t + 4) * AP + n0 + g]);
  return f;
}

__device__ __forceinline__ void mma_tf32(float (&c)[4], const FragA& a,
                                         const FragB& b) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a.a[0]), "r"(a.a[1]), "r"(a.a[2]), "r"(a.a[3]), "r"(b.b[0]),
        "r"(b.b[1]));
}

// Store s * C (16 x 8 accumulator tile) at (r0, c0) of a row-major matrix.
__device__ __forceinline__ void store_frag_c(float* X, int r0, int c0,
                                             const float (&c)[4], float s,
                                             int lane) {
  const int g = lane >> 2, t = lane & 3;
  *reinterpret_cast<float2*>(X + (r0 + g) * AP + c0 + 2 * t) =
      make_float2(s * c[0], s * c[1]);
  *reinterpret_cast<float2*>(X + (r0 + g + 8) * AP + c0 + 2 * t) =
      make_float2(s * c[2], s * c[3]);
}

// D(16 x 16 at (dr, dc)) = s * X(16 x K at (xr, xc)) Y(K x 16 at (yr, yc)).
template <int K>
__device__ __forceinline__ void mm16x16(float* D, int dr, int dc, const float* X,
                                        int xr, int xc, const float* Y, int yr,
                                        int yc, float s, int lane) {
  float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < K; k += 8) {
    const FragA a = load_frag_a(X, xr, xc + k, lane);
    mma_tf32(c0, a, load_frag_b(Y, yr + k, yc, lane));
    mma_tf32(c1, a, load_frag_b(Y, yr + k, yc + 8, lane));
  }
  store_frag_c(D, dr, dc, c0, s, lane);
  store_frag_c(D, dr, dc + 8, c1, s, lane);
}

// (I + A)^{-1} for the strictly lower 64 x 64 A, in place: on entry AT holds
// A row-major (zeros on and above the diagonal), on exit its lower triangle
// holds T with a unit diagonal, and its 16 x 16 blocks above the diagonal
// blocks are zero except the upper-right 32 x 32 block, which is scratch.
// Blocked in powers of two: the four 16 x 16 diagonal blocks by substitution,
// then T_10 = -T_11 A_10 T_00 at 16 and at 32 with the products on the tensor
// cores (tf32). All 128 prep threads take part (tid 0..127); they meet at
// named barrier `bar`.
__device__ __forceinline__ void solve_unit_lower(float* AT, int tid,
                                                 int bar = 1) {
  const int warp = tid >> 5, lane = tid & 31;
  // 1. diagonal 16 x 16 blocks: one per warp, lane l < 16 owns column l,
  //    x_m = delta_ml - sum_{j<m} A_mj x_j
  {
    const int b = 16 * warp;
    float xs[16];
    if (lane < 16) {
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float4* arow = reinterpret_cast<const float4*>(AT + (b + m) * AP + b);
        // four partial sums, so that the dependent chain of a row is m / 4
        // multiply-adds long rather than m
        float acc0 = (m == lane) ? 1.f : 0.f, acc1 = 0.f, acc2 = 0.f,
              acc3 = 0.f;
#pragma unroll
        for (int q = 0; q < (m + 3) / 4; ++q) {
          const float4 a = arow[q];  // one broadcast load for four terms
          if (4 * q < m) acc0 = fmaf(-a.x, xs[4 * q], acc0);
          if (4 * q + 1 < m) acc1 = fmaf(-a.y, xs[4 * q + 1], acc1);
          if (4 * q + 2 < m) acc2 = fmaf(-a.z, xs[4 * q + 2], acc2);
          if (4 * q + 3 < m) acc3 = fmaf(-a.w, xs[4 * q + 3], acc3);
        }
        xs[m] = (acc0 + acc1) + (acc2 + acc3);
      }
    }
    __syncwarp();  // the whole block is read before it is overwritten
    if (lane < 16) {
#pragma unroll
      for (int m = 0; m < 16; ++m) AT[(b + m) * AP + b + lane] = xs[m];
    }
  }
  named_bar(bar, 128);
  // 2. 16 -> 32: warp p in {0, 1} merges diagonal blocks (2p, 2p+1); the
  //    product X = A_10 T_00 goes to rows 16p.., columns 32+16p.. (scratch)
  if (warp < 2) {
    const int kb = 32 * warp, xr = 16 * warp, xc = 32 + 16 * warp;
    mm16x16<16>(AT, xr, xc, AT, kb + 16, kb, AT, kb, kb, 1.f, lane);
    __syncwarp();
    mm16x16<16>(AT, kb + 16, kb, AT, kb + 16, kb + 16, AT, xr, xc, -1.f,
                lane);
  }
  named_bar(bar, 128);
  // 3. 32 -> 64: X = A_21 T_11 into rows 0-31, columns 32-63, then
  //    T_21 = -T_22 X; warp w owns rows 16 (w >> 1), columns 16 (w & 1)
  {
    const int mr = 16 * (warp >> 1), nc = 16 * (warp & 1);
    mm16x16<32>(AT, mr, 32 + nc, AT, 32 + mr, 0, AT, 0, nc, 1.f, lane);
    named_bar(bar, 128);
    mm16x16<32>(AT, 32 + mr, nc, AT, 32 + mr, 32, AT, 0, 32 + nc, -1.f, lane);
  }
  named_bar(bar, 128);
}



// Write 32 fp32 values as bf16 into 16-byte chunks 4 hf .. 4 hf + 3 of row r
// of a 128-byte-row swizzled tile.
__device__ __forceinline__ void store_half_bf16(uint8_t* tile, int r, int hf,
                                                const float (&x)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 w;
    w.x = pack_bf16x2(x[8 * c + 0], x[8 * c + 1]);
    w.y = pack_bf16x2(x[8 * c + 2], x[8 * c + 3]);
    w.z = pack_bf16x2(x[8 * c + 4], x[8 * c + 5]);
    w.w = pack_bf16x2(x[8 * c + 6], x[8 * c + 7]);
    *reinterpret_cast<uint4*>(tile + sw128(r, 4 * hf + c)) = w;
  }
}

// kN fp32 values as bf16 into 16-byte chunks c0 .. c0 + kN / 8 - 1 of row r
// of a 128-byte-row swizzled tile.
template <int kN>
__device__ __forceinline__ void store_cols_bf16(uint8_t* tile, int r, int c0,
                                                const float (&x)[kN]) {
#pragma unroll
  for (int c = 0; c < kN / 8; ++c) {
    uint4 w;
    w.x = pack_bf16x2(x[8 * c + 0], x[8 * c + 1]);
    w.y = pack_bf16x2(x[8 * c + 2], x[8 * c + 3]);
    w.z = pack_bf16x2(x[8 * c + 4], x[8 * c + 5]);
    w.w = pack_bf16x2(x[8 * c + 6], x[8 * c + 7]);
    *reinterpret_cast<uint4*>(tile + sw128(r, c0 + c)) = w;
  }
}

// As store_half_bf16, scaled by s.
__device__ __forceinline__ void store_half_bf16_scaled(uint8_t* tile, int r,
                                                       int hf,
                                                       const float (&x)[32],
                                                       float s) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 w;
    w.x = pack_bf16x2(s * x[8 * c + 0], s * x[8 * c + 1]);
    w.y = pack_bf16x2(s * x[8 * c + 2], s * x[8 * c + 3]);
    w.z = pack_bf16x2(s * x[8 * c + 4], s * x[8 * c + 5]);
    w.w = pack_bf16x2(s * x[8 * c + 6], s * x[8 * c + 7]);
    *reinterpret_cast<uint4*>(tile + sw128(r, 4 * hf + c)) = w;
  }
}

// Per-(chunk, head) operands the preparation writes for the chain kernel,
// each the exact image of a 1024-byte-aligned shared-memory tile (64 rows of
// 128 bytes, 128-byte swizzle) so that both sides move them with plain bulk
// copies: -W as two 64-column blocks, P, T_U.
constexpr uint32_t TILE_BYTES = 8192;
constexpr uint32_t WS_W_BYTES = 2 * TILE_BYTES;
constexpr uint32_t WS_P_BYTES = TILE_BYTES;
constexpr uint32_t WS_TU_BYTES = TILE_BYTES;
// KDA adds Q_g and K_d (two 64-column blocks each) and a longer decay record:
// e^G (ones: the decay is inside Q_g), an unused block, gamma per key channel.
constexpr uint32_t WS_QG_BYTES = 2 * TILE_BYTES;
constexpr uint32_t WS_KD_BYTES = 2 * TILE_BYTES;
constexpr int KCV_FLOATS = 256;
constexpr uint32_t KCV_BYTES = KCV_FLOATS * 4;

}  // namespace

// Tensor map over a [d2][d1][d0] row-major tensor (bf16, or fp32 when
// `fp32`) whose box is b0 x 1 x b2 elements with no swizzle: the box lands
// in shared memory as b2 rows of b0 contiguous elements (host side).
bool make_rows_map(CUtensorMap* map, const void* ptr, bool fp32, long long d0,
                   long long d1, long long d2, uint32_t b0, uint32_t b2);

}  // namespace gdn
