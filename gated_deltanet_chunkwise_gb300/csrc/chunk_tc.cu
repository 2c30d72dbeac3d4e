// Chunkwise Gated DeltaNet forward pass on the sm_103a tensor cores.
//
// One CTA owns (sequence, head, a 64-row tile of the state's d_v rows) and
// walks the sequence's chunks (C = 64, d_k = 128) in order. The state is kept
// transposed, S^T (d_k x 64), in fp32 registers of the "chain" warpgroup (one
// d_k row per thread) and mirrored as bf16 in shared memory for the MMAs.
// Per chunk (illustrated DeltaNet walk-through: UT transform, WY
// representation, chunkwise state passing and output; scalar gate prefixes
// of its GLA section), with D_rj = exp(G_r - G_j), G the chunk-local
// cumulative log gate, G' = G (decay first) or G_{r-1} (decay after the
// prediction), and every gate factor folded into an operand that is written
// anyway (all such factors lie in (0, 1]):
//
//   prep   MMA0  [K;Q] K^T -> K K^T, Q K^T
//          A = strict_lower(diag(beta) K K^T (.) D'),  T = (I + A)^{-1},
//          P = (Q K^T) (.) D (.) M_incl,
//          T_W = T diag(beta e^{G'}),  T_U = T diag(beta)
//          MMA   [T_W;T_W] K -> W (twice);  [0;T_U] V -> U0 starts the
//                chunk's accumulator (rows 64-127);  -W is stored after Q
//   chain  MMA1  accumulator += [Q;-W] S^T -> H = Q S^T (rows 0-63),
//                U = U0 - W S^T (rows 64-127)
//          MMA2  K^T (diag(e^{G_L - G}) U) -> Delta;  S^T <- gamma S^T + Delta
//          MMA3  [P;0] U -> P U;   O = diag(e^G) H + P U at read-out
//
// The serial chain per chunk is two MMA round trips and two short register
// phases; everything else overlaps it.
//
// Warp roles (352 threads): warps 0-3 prep, 4-7 chain, 8 TMA producer (also
// the chunk's gate vectors), 9 issues the chain's MMAs, 10 the prep's MMAs.
// Operand tiles are bf16 with the 128-byte swizzle; K/Q/V arrive by TMA in a
// two-stage ring. Every wait is bounded; a CTA that gives up records
// GDN_ERR_TIMEOUT, drains its MMAs, frees its TMEM and exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_internal.cuh"
#include "gdn_selftest.h"
#include "tc_ptx.cuh"

namespace gdn {
namespace {
using namespace tc;

constexpr int C = 64;
constexpr int DK = 128;
constexpr int DVT = 64;
constexpr int kThreads = 352;

// Stage: per 64-column block of d_k, three 64-row groups K | Q | -W (the
// first two by TMA, -W by the prep); [K;Q] and [Q;-W] are 128-row K-major
// tiles and K alone is the N-major operand of the W and Delta products. The
// V tile (64 x 64) follows the two column blocks.
constexpr uint32_t ST_K = 0;
constexpr uint32_t ST_Q = 8192;
constexpr uint32_t ST_W = 16384;
constexpr uint32_t ST_CB = 24576;
constexpr uint32_t ST_V = 49152;
constexpr uint32_t STAGE_BYTES = 57344;
constexpr uint32_t STAGE_TMA_BYTES = 40960;
// T buffer: T_W twice, P (even chunks), zeros, T_U, P (odd chunks), zeros;
// [T_W;T_W], [P0;0], [0;T_U] and [P1;0] are 128-row K-major tiles.
constexpr uint32_t TB_TW = 0, TB_TW2 = 8192, TB_P0 = 16384, TB_Z = 24576,
                   TB_TU = 32768, TB_P1 = 40960, TB_Z2 = 49152,
                   TB_BYTES = 57344;

constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_TB = 2 * STAGE_BYTES;               // 114688
constexpr uint32_t OFF_S = OFF_TB + TB_BYTES;              // S^T, bf16
constexpr uint32_t OFF_U = OFF_S + 16384;                  // U, bf16
constexpr uint32_t OFF_UD = OFF_U + 8192;                  // diag(e^{G_L-G}) U
constexpr int AP = 68;  // fp32 row pitch of the solve buffer
constexpr uint32_t OFF_AT = OFF_UD + 8192;                 // A, then T (fp32)
// Per-stage gate vectors written by the producer warp: cumulative log gate G,
// alpha = e^g, e^G, beta e^{G'}, beta, e^{G_L - G}, e^{-G}, gamma = e^{G_L},
// and whether e^{G_r} e^{-G_j} stays in the normal fp32 range.
constexpr int VEC_G = 0, VEC_ALPHA = 64, VEC_EG = 128, VEC_EGPB = 192,
              VEC_BETA = 256, VEC_DEC = 320, VEC_IEG = 384, VEC_GAMMA = 448,
              VEC_SAFE = 449, VEC_FLOATS = 452;
constexpr uint32_t OFF_VEC = OFF_AT + 64 * AP * 4;
constexpr uint32_t OFF_BAR = OFF_VEC + 2 * VEC_FLOATS * 4;

enum {
  B_FULL0, B_FULL1, B_EMPTY0, B_EMPTY1, B_MMA0, B_D0FREE, B_PREPT, B_WDONE,
  B_PREPD0, B_PREPD1, B_SREADY, B_D1FULL0, B_D1FULL1, B_UREADY, B_D2FULL,
  B_D3FULL0, B_D3FULL1, B_D1FREE0, B_D1FREE1, B_TPFREE0, B_TPFREE1,
  B_DRAIN_C, B_DRAIN_P, NBARS
};
constexpr uint32_t OFF_MISC = OFF_BAR + NBARS * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// TMEM columns (fp32 accumulators, 128 lanes each).
constexpr uint32_t TM_D0 = 0, TM_D1 = 64, TM_DW = 192, TM_D2 = 320,
                   TM_D3 = 384;
constexpr uint32_t TMEM_COLS = 512;

constexpr uint32_t ID_KK = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_KMN = idesc_bf16(128, 64, false, true);
constexpr uint32_t ID_KMN128 = idesc_bf16(128, 128, false, true);
constexpr uint32_t ID_MNMN = idesc_bf16(128, 64, true, true);

__device__ __forceinline__ uint32_t bar_count(int b) {
  switch (b) {
    case B_FULL0: case B_FULL1: return 2;
    case B_D0FREE: case B_PREPT: case B_PREPD0: case B_PREPD1: case B_SREADY:
      return 128;
    case B_UREADY: case B_D1FREE0: case B_D1FREE1: return 64;
    default: return 1;
  }
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

// Write a 64-value fp32 row as bf16 into row r of a 128-byte-row swizzled tile.
__device__ __forceinline__ void store_row_bf16(uint8_t* tile, int r,
                                               const float (&x)[64]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint4 w;
    w.x = pack_bf16x2(x[8 * c + 0], x[8 * c + 1]);
    w.y = pack_bf16x2(x[8 * c + 2], x[8 * c + 3]);
    w.z = pack_bf16x2(x[8 * c + 4], x[8 * c + 5]);
    w.w = pack_bf16x2(x[8 * c + 6], x[8 * c + 7]);
    *reinterpret_cast<uint4*>(tile + sw128(r, c)) = w;
  }
}

__device__ __forceinline__ void load_vec64(const float* src, float (&x)[64]) {
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const float4 v = reinterpret_cast<const float4*>(src)[c];
    x[4 * c] = v.x; x[4 * c + 1] = v.y; x[4 * c + 2] = v.z; x[4 * c + 3] = v.w;
  }
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
// cores (tf32). All 128 prep threads take part.
__device__ __forceinline__ void solve_unit_lower(float* AT, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  // 1. diagonal 16 x 16 blocks: one per warp, lane l < 16 owns column l,
  //    x_m = delta_ml - sum_{j<m} A_mj x_j
  {
    const int b = 16 * warp;
    float xs[16];
    if (lane < 16) {
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float* arow = AT + (b + m) * AP + b;
        float acc = (m == lane) ? 1.f : 0.f;
#pragma unroll
        for (int j = 0; j < m; ++j) acc = fmaf(-arow[j], xs[j], acc);
        xs[m] = acc;
      }
    }
    __syncwarp();  // the whole block is read before it is overwritten
    if (lane < 16) {
#pragma unroll
      for (int m = 0; m < 16; ++m) AT[(b + m) * AP + b + lane] = xs[m];
    }
  }
  named_bar(1, 128);
  // 2. 16 -> 32: warp p in {0, 1} merges diagonal blocks (2p, 2p+1); the
  //    product X = A_10 T_00 goes to rows 16p.., columns 32+16p.. (scratch)
  if (warp < 2) {
    const int kb = 32 * warp, xr = 16 * warp, xc = 32 + 16 * warp;
    mm16x16<16>(AT, xr, xc, AT, kb + 16, kb, AT, kb, kb, 1.f, lane);
    __syncwarp();
    mm16x16<16>(AT, kb + 16, kb, AT, kb + 16, kb + 16, AT, xr, xc, -1.f,
                lane);
  }
  named_bar(1, 128);
  // 3. 32 -> 64: X = A_21 T_11 into rows 0-31, columns 32-63, then
  //    T_21 = -T_22 X; warp w owns rows 16 (w >> 1), columns 16 (w & 1)
  {
    const int mr = 16 * (warp >> 1), nc = 16 * (warp & 1);
    mm16x16<32>(AT, mr, 32 + nc, AT, 32 + mr, 0, AT, 0, nc, 1.f, lane);
    named_bar(1, 128);
    mm16x16<32>(AT, 32 + mr, nc, AT, 32 + mr, 32, AT, 0, 32 + nc, -1.f, lane);
  }
  named_bar(1, 128);
}

template <int VARIANT>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_tc_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap tmq,
                    const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H, dv = p.dv;
  const int h = blockIdx.y;
  const int n = blockIdx.z / p.part_count;
  const int part = p.part_begin + blockIdx.z % p.part_count;
  const int row0 = blockIdx.x * DVT;
  const bool value_rows = row0 < dv;
  const bool split_tail = (p.mode == kModeSplit) && part > 0;
  if (!value_rows && !(split_tail && row0 < dv + DK)) return;
  const bool scale_rows = !value_rows;
  const bool emit = (p.mode == kModeOutput) || part == 0;
  long long bos, eos;
  if (!sequence_range(p, n, bos, eos)) return;
  const int nch = (int)((eos - bos + C - 1) / C);
  int c_begin, c_end;
  part_range(nch, p.parts, part, c_begin, c_end);
  const int nloc = c_end - c_begin;
  const size_t nh = (size_t)n * H + h;

  // ---- set-up ----
  if (tid == 0) {
    for (int b = 0; b < NBARS; ++b) mbar_init(&bars[b], bar_count(b));
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < 128) {
    // the two zero blocks of the T buffer
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int i = tid; i < 1024; i += 128) {
      const uint32_t off = (i < 512 ? TB_Z : TB_Z2) + (uint32_t)(i & 511) * 16;
      *reinterpret_cast<uint4*>(sm + OFF_TB + off) = z;
    }
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto stage = [&](int i) { return base + OFF_STAGE + (i & 1) * STAGE_BYTES; };

  if (warp == 8) {
    // ================= TMA producer + gate vectors =================
    int issued = 0;
    for (int i = 0; i < nloc; ++i) {
      const int s = i & 1;
      if (i >= 2 && !mbar_wait(&bars[B_EMPTY0 + s], ((i >> 1) - 1) & 1,
                               abort_flag))
        break;
      const long long t0 = bos + (long long)(c_begin + i) * C;
      const int len = (int)min((long long)C, eos - t0);
      uint8_t* st = sm + OFF_STAGE + s * STAGE_BYTES;
      uint64_t* full = &bars[B_FULL0 + s];
      if (lane == 0) {
        mbar_arrive_expect_tx(full, STAGE_TMA_BYTES);
        const int tok = (int)t0;
        tma_load_3d(st + ST_K, &tmk, full, 0, h, tok);
        tma_load_3d(st + ST_K + ST_CB, &tmk, full, 64, h, tok);
        tma_load_3d(st + ST_Q, &tmq, full, 0, h, tok);
        tma_load_3d(st + ST_Q + ST_CB, &tmq, full, 64, h, tok);
        tma_load_3d(st + ST_V, &tmv, full, value_rows ? row0 : 0, h, tok);
      }
      {
        // gate vectors (tokens past the end: g = 0, beta = 0)
        const unsigned fm = 0xffffffffu;
        float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
        const size_t rbase = (size_t)t0 * H + h;
        if (lane < len) {
          g0 = p.g[rbase + (size_t)lane * H];
          b0 = p.beta[rbase + (size_t)lane * H];
        }
        if (lane + 32 < len) {
          g1 = p.g[rbase + (size_t)(lane + 32) * H];
          b1 = p.beta[rbase + (size_t)(lane + 32) * H];
        }
        float s0 = g0, s1 = g1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float u0 = __shfl_up_sync(fm, s0, o);
          const float u1 = __shfl_up_sync(fm, s1, o);
          if (lane >= o) {
            s0 += u0;
            s1 += u1;
          }
        }
        s1 += __shfl_sync(fm, s0, 31);
        const float Gl = __shfl_sync(fm, s1, 31);
        const float p0 = VARIANT == GDN_GATE_BEFORE_PREDICT ? s0 : s0 - g0;
        const float p1 = VARIANT == GDN_GATE_BEFORE_PREDICT ? s1 : s1 - g1;
        const bool in_range = __all_sync(
            fm, s0 >= -87.f && s0 <= 87.f && s1 >= -87.f && s1 <= 87.f);
        float* vec = reinterpret_cast<float*>(sm + OFF_VEC) + s * VEC_FLOATS;
        vec[VEC_G + lane] = s0;
        vec[VEC_G + 32 + lane] = s1;
        vec[VEC_ALPHA + lane] = expf(g0);
        vec[VEC_ALPHA + 32 + lane] = expf(g1);
        vec[VEC_EG + lane] = expf(s0);
        vec[VEC_EG + 32 + lane] = expf(s1);
        vec[VEC_EGPB + lane] = expf(p0) * b0;
        vec[VEC_EGPB + 32 + lane] = expf(p1) * b1;
        vec[VEC_BETA + lane] = b0;
        vec[VEC_BETA + 32 + lane] = b1;
        vec[VEC_DEC + lane] = expf(Gl - s0);
        vec[VEC_DEC + 32 + lane] = expf(Gl - s1);
        vec[VEC_IEG + lane] = expf(-s0);
        vec[VEC_IEG + 32 + lane] = expf(-s1);
        if (lane == 0) {
          vec[VEC_GAMMA] = expf(Gl);
          vec[VEC_SAFE] = in_range ? 1.f : 0.f;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(full);
      issued = i + 1;
    }
    // never leave with a TMA copy still landing in shared memory
    if (lane == 0)
      for (int i = max(0, issued - 2); i < issued; ++i)
        wait_ignoring_abort(&bars[B_FULL0 + (i & 1)], (i >> 1) & 1);
  } else if (warp == 10) {
    // ================= prep MMAs: K K^T / Q K^T, W and U0 =================
    if (lane == 0 && nloc > 0) {
      const uint32_t tb = base + OFF_TB;
      auto mma0 = [&](int j) {
        const uint32_t st = stage(j);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t a =
              sdesc(st + ST_K + (k >> 2) * ST_CB + (k & 3) * 32, 16, 1024);
          mma_bf16(tmem + TM_D0, a, a, ID_KK, k > 0);
        }
        mma_commit(&bars[B_MMA0]);
      };
      bool ok = mbar_wait(&bars[B_FULL0], 0, abort_flag);
      if (ok) {
        tc_fence_after();
        mma0(0);
      }
      for (int j = 0; ok && j < nloc; ++j) {
        if (j + 1 < nloc) {
          ok = mbar_wait(&bars[B_D0FREE], j & 1, abort_flag) &&
               mbar_wait(&bars[B_FULL0 + ((j + 1) & 1)], ((j + 1) >> 1) & 1,
                         abort_flag);
          if (!ok) break;
          tc_fence_after();
          mma0(j + 1);
        }
        ok = mbar_wait(&bars[B_PREPT], j & 1, abort_flag) &&
             (j < 2 || mbar_wait(&bars[B_D1FREE0 + (j & 1)],
                                 ((j >> 1) - 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const uint32_t st = stage(j);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // W (twice) = [T_W;T_W] K
          mma_bf16(tmem + TM_DW, sdesc(tb + TB_TW + k * 32, 16, 1024),
                   sdesc(st + ST_K + k * 2048, ST_CB, 1024), ID_KMN128, k > 0);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // U0 = [0;T_U] V starts the accumulator
          mma_bf16(tmem + TM_D1 + 64 * (j & 1), sdesc(tb + TB_Z + k * 32, 16, 1024),
                   sdesc(st + ST_V + k * 2048, 8192, 1024), ID_KMN, k > 0);
        mma_commit(&bars[B_WDONE]);
      }
      mma_commit(&bars[B_DRAIN_P]);
      wait_ignoring_abort(&bars[B_DRAIN_P], 0);
    }
  } else if (warp == 9) {
    // ================= chain MMAs =================
    if (lane == 0 && nloc > 0) {
      const uint32_t tb = base + OFF_TB;
      for (int i = 0; i < nloc; ++i) {
        const int b = i & 1;
        bool ok = mbar_wait(&bars[B_SREADY], i & 1, abort_flag) &&
                  mbar_wait(&bars[B_PREPD0 + b], (i >> 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t st = stage(i);
#pragma unroll
        for (int k = 0; k < 8; ++k)  // += [Q;-W] S^T
          mma_bf16(tmem + TM_D1 + 64 * b,
                   sdesc(st + ST_Q + (k >> 2) * ST_CB + (k & 3) * 32, 16, 1024),
                   sdesc(base + OFF_S + k * 2048, 8192, 1024), ID_KMN, 1);
        mma_commit(&bars[B_D1FULL0 + b]);
        ok = mbar_wait(&bars[B_UREADY], i & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)  // Delta = K^T diag(e^{G_L-G}) U
          mma_bf16(tmem + TM_D2, sdesc(st + ST_K + k * 2048, ST_CB, 1024),
                   sdesc(base + OFF_UD + k * 2048, 8192, 1024), ID_MNMN, k > 0);
        mma_commit(&bars[B_D2FULL]);
        mma_commit(&bars[B_EMPTY0 + b]);
        const uint32_t pz = tb + (b ? TB_P1 : TB_P0);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // P U
          mma_bf16(tmem + TM_D3 + 64 * b, sdesc(pz + k * 32, 16, 1024),
                   sdesc(base + OFF_U + k * 2048, 8192, 1024), ID_KMN, k > 0);
        mma_commit(&bars[B_D3FULL0 + b]);
        mma_commit(&bars[B_TPFREE0 + b]);
      }
      mma_commit(&bars[B_DRAIN_C]);
      wait_ignoring_abort(&bars[B_DRAIN_C], 0);
    }
  } else if (warp < 4) {
    // ================= prep warpgroup =================
    float* AT = reinterpret_cast<float*>(sm + OFF_AT);
    uint8_t* tbuf = sm + OFF_TB;
    const uint32_t lanes = (uint32_t)(32 * warp) << 16;
    for (int j = 0; j < nloc; ++j) {
      const int s = j & 1;
      const float* vec =
          reinterpret_cast<const float*>(sm + OFF_VEC) + s * VEC_FLOATS;
      uint8_t* st = sm + OFF_STAGE + s * STAGE_BYTES;
      // stage data and gate vectors (full), K K^T and Q K^T (MMA0)
      bool ok = mbar_wait(&bars[B_FULL0 + s], (j >> 1) & 1, abort_flag) &&
                mbar_wait(&bars[B_MMA0], j & 1, abort_flag);
      if (!bar_and(1, 128, ok)) break;
      tc_fence_after();
      float x[64];
      tmem_ld64(tmem + TM_D0 + lanes, x);
      tc_fence_before();
      mbar_arrive(&bars[B_D0FREE]);
      // P buffer of chunk j-2 consumed
      ok = j < 2 ||
           mbar_wait(&bars[B_TPFREE0 + s], ((j >> 1) - 1) & 1, abort_flag);
      if (!bar_and(1, 128, ok)) break;
      const bool safe = vec[VEC_SAFE] != 0.f;
      // w = e^{-G} (factored decays) or alpha (running products)
      float w[64];
      load_vec64(vec + (safe ? VEC_IEG : VEC_ALPHA), w);
      if (tid < 64) {
        // row r of A: beta_r exp(G'_r - G_j) k_r.k_j for j < r
        const int r = tid;
        if (safe) {
          const float er = vec[VEC_EGPB + r];
#pragma unroll
          for (int jj = 0; jj < 64; ++jj) x[jj] = jj < r ? er * w[jj] * x[jj] : 0.f;
        } else {
          const float br = vec[VEC_BETA + r];
          float d = 1.f;
          x[63] = 0.f;
#pragma unroll
          for (int jj = 62; jj >= 0; --jj) {
            float a = 0.f;
            if (jj < r) {
              if (VARIANT == GDN_GATE_BEFORE_PREDICT) {
                d *= w[jj + 1];
                a = br * d * x[jj];
              } else {
                a = br * d * x[jj];
                d *= w[jj];
              }
            }
            x[jj] = a;
          }
        }
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4)
          *reinterpret_cast<float4*>(AT + r * AP + 4 * c4) =
              make_float4(x[4 * c4], x[4 * c4 + 1], x[4 * c4 + 2], x[4 * c4 + 3]);
      } else {
        // row r of P: exp(G_r - G_j) q_r.k_j for j <= r
        const int r = tid - 64;
        if (safe) {
          const float er = vec[VEC_EG + r];
#pragma unroll
          for (int jj = 0; jj < 64; ++jj) x[jj] = jj <= r ? er * w[jj] * x[jj] : 0.f;
        } else {
          float d = 1.f;
#pragma unroll
          for (int jj = 63; jj >= 0; --jj) {
            float pv = 0.f;
            if (jj <= r) {
              pv = d * x[jj];
              d *= w[jj];
            }
            x[jj] = pv;
          }
        }
        store_row_bf16(tbuf + (s ? TB_P1 : TB_P0), r, x);
      }
      named_bar(1, 128);
      solve_unit_lower(AT, tid);
      {
        // T_W = T diag(beta e^{G'}) (two copies), T_U = T diag(beta)
        const int r = tid >> 1, hh = tid & 1;
        float f[32], fw[32], fu[32];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 t4 =
              *reinterpret_cast<const float4*>(AT + r * AP + hh * 32 + 4 * c4);
          const float4 w4 = *reinterpret_cast<const float4*>(
              vec + VEC_EGPB + hh * 32 + 4 * c4);
          // rows of the scaling matrix see V = 0, so U0 = 0 for them
          const float4 u4 = scale_rows
                                ? make_float4(0.f, 0.f, 0.f, 0.f)
                                : *reinterpret_cast<const float4*>(
                                      vec + VEC_BETA + hh * 32 + 4 * c4);
          f[4 * c4] = t4.x; f[4 * c4 + 1] = t4.y;
          f[4 * c4 + 2] = t4.z; f[4 * c4 + 3] = t4.w;
          fw[4 * c4] = w4.x; fw[4 * c4 + 1] = w4.y;
          fw[4 * c4 + 2] = w4.z; fw[4 * c4 + 3] = w4.w;
          fu[4 * c4] = u4.x; fu[4 * c4 + 1] = u4.y;
          fu[4 * c4 + 2] = u4.z; fu[4 * c4 + 3] = u4.w;
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = hh * 32 + e;
          f[e] = col < r ? f[e] : (col == r ? 1.f : 0.f);
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 a, c;
          a.x = pack_bf16x2(f[8 * q4 + 0] * fw[8 * q4 + 0], f[8 * q4 + 1] * fw[8 * q4 + 1]);
          a.y = pack_bf16x2(f[8 * q4 + 2] * fw[8 * q4 + 2], f[8 * q4 + 3] * fw[8 * q4 + 3]);
          a.z = pack_bf16x2(f[8 * q4 + 4] * fw[8 * q4 + 4], f[8 * q4 + 5] * fw[8 * q4 + 5]);
          a.w = pack_bf16x2(f[8 * q4 + 6] * fw[8 * q4 + 6], f[8 * q4 + 7] * fw[8 * q4 + 7]);
          c.x = pack_bf16x2(f[8 * q4 + 0] * fu[8 * q4 + 0], f[8 * q4 + 1] * fu[8 * q4 + 1]);
          c.y = pack_bf16x2(f[8 * q4 + 2] * fu[8 * q4 + 2], f[8 * q4 + 3] * fu[8 * q4 + 3]);
          c.z = pack_bf16x2(f[8 * q4 + 4] * fu[8 * q4 + 4], f[8 * q4 + 5] * fu[8 * q4 + 5]);
          c.w = pack_bf16x2(f[8 * q4 + 6] * fu[8 * q4 + 6], f[8 * q4 + 7] * fu[8 * q4 + 7]);
          const uint32_t off = sw128(r, hh * 4 + q4);
          *reinterpret_cast<uint4*>(tbuf + TB_TW + off) = a;
          *reinterpret_cast<uint4*>(tbuf + TB_TW2 + off) = a;
          *reinterpret_cast<uint4*>(tbuf + TB_TU + off) = c;
        }
      }
      fence_proxy_async();
      mbar_arrive(&bars[B_PREPT]);
      // -W after Q in the stage: warps 0-1 columns 0-63 (lanes 0-63),
      // warps 2-3 columns 64-127 (lanes 64-127 hold the second copy of W)
      ok = mbar_wait(&bars[B_WDONE], j & 1, abort_flag);
      if (!bar_and(1, 128, ok)) break;
      tc_fence_after();
      {
        const int cb = warp >> 1, r = tid & 63;
        float wv[64];
        tmem_ld64(tmem + TM_DW + lanes + 64 * cb, wv);
#pragma unroll
        for (int c = 0; c < 64; ++c) wv[c] = -wv[c];
        store_row_bf16(st + ST_W + cb * ST_CB, r, wv);
      }
      tc_fence_before();
      fence_proxy_async();
      mbar_arrive(&bars[B_PREPD0 + s]);
    }
  } else {
    // ================= chain warpgroup =================
    // warps 4-5: output rows (lanes 0-63), warps 6-7: U rows (lanes 64-127),
    // all four: state rows (lane = d_k index)
    const int ct = tid - 128, cw = warp - 4;
    const uint32_t lanes = (uint32_t)(32 * cw) << 16;
    uint8_t* s_tile = sm + OFF_S;
    float S[64];
    if (scale_rows) {
      const int a0 = row0 - dv;
#pragma unroll
      for (int c = 0; c < 64; ++c) S[c] = (ct == a0 + c) ? 1.f : 0.f;
    } else if (split_tail) {
#pragma unroll
      for (int c = 0; c < 64; ++c) S[c] = 0.f;
    } else if (part > 0) {
      const float* src = p.ws_start + ((nh * p.parts + part) * dv + row0) * DK + ct;
#pragma unroll
      for (int c = 0; c < 64; ++c) S[c] = src[(size_t)c * DK];
    } else if (p.h0) {
      const float4* src =
          reinterpret_cast<const float4*>(p.h0 + (nh * DK + ct) * dv + row0);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float4 v4 = src[c];
        S[4 * c] = v4.x; S[4 * c + 1] = v4.y; S[4 * c + 2] = v4.z; S[4 * c + 3] = v4.w;
      }
    } else {
#pragma unroll
      for (int c = 0; c < 64; ++c) S[c] = 0.f;
    }
    store_row_bf16(s_tile, ct, S);
    bool ok = true;
    // per-chunk scalars read while the chunk's stage is certainly resident:
    // gamma (all), e^{G_r} of the output row (warps 4-5)
    float gam = 1.f, eg = 1.f;
    if (nloc > 0) {
      ok = mbar_wait(&bars[B_FULL0], 0, abort_flag);
      const float* vec = reinterpret_cast<const float*>(sm + OFF_VEC);
      gam = vec[VEC_GAMMA];
      eg = vec[VEC_EG + (ct & 63)];
    }
    fence_proxy_async();
    mbar_arrive(&bars[B_SREADY]);
    for (int i = 0; i < nloc; ++i) {
      const int b = i & 1, s = i & 1;
      const long long t0 = bos + (long long)(c_begin + i) * C;
      const int len = (int)min((long long)C, eos - t0);
      if (cw >= 2) {
        // U = U0 - W S^T (rows 64-127 of the accumulator)
        const int r = ct - 64;
        bool ok1 = ok && mbar_wait(&bars[B_D1FULL0 + b], (i >> 1) & 1, abort_flag);
        ok1 = bar_and(3, 64, ok1);
        if (ok1) {
          tc_fence_after();
          const float dec = reinterpret_cast<const float*>(sm + OFF_VEC)[
              s * VEC_FLOATS + VEC_DEC + r];
          float u[64];
          tmem_ld64(tmem + TM_D1 + 64 * b + lanes, u);
          store_row_bf16(sm + OFF_U, r, u);
#pragma unroll
          for (int c = 0; c < 64; ++c) u[c] *= dec;
          store_row_bf16(sm + OFF_UD, r, u);
          fence_proxy_async();
          tc_fence_before();
          mbar_arrive(&bars[B_UREADY]);
        }
        ok = ok1;
      }
      bool ok3 = ok && mbar_wait(&bars[B_D2FULL], i & 1, abort_flag);
      if (!bar_and(2, 128, ok3)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        float dl[64];
        tmem_ld64(tmem + TM_D2 + lanes, dl);
#pragma unroll
        for (int c = 0; c < 64; ++c) S[c] = fmaf(gam, S[c], dl[c]);
      }
      store_row_bf16(s_tile, ct, S);
      const float eg_now = eg;
      if (i + 1 < nloc) {
        ok = mbar_wait(&bars[B_FULL0 + (b ^ 1)], ((i + 1) >> 1) & 1, abort_flag);
        const float* vec =
            reinterpret_cast<const float*>(sm + OFF_VEC) + (b ^ 1) * VEC_FLOATS;
        gam = vec[VEC_GAMMA];
        eg = vec[VEC_EG + (ct & 63)];
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&bars[B_SREADY]);
      if (cw < 2) {
        // O = e^{G_r} H + P U
        const int r = ct;
        bool ok4 = ok && mbar_wait(&bars[B_D3FULL0 + b], (i >> 1) & 1, abort_flag);
        ok4 = bar_and(4, 64, ok4);
        if (ok4) {
          tc_fence_after();
          const bool store = emit && r < len;
          uint4* dst = reinterpret_cast<uint4*>(
              static_cast<__nv_bfloat16*>(p.out) +
              ((size_t)(t0 + (store ? r : 0)) * H + h) * dv + row0);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float o[32], pu[32];
            tmem_ld32(tmem + TM_D1 + 64 * b + lanes + 32 * half, o);
            tmem_ld32(tmem + TM_D3 + 64 * b + lanes + 32 * half, pu);
            tmem_ld_wait();
            if (store) {
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                uint4 wq;
                wq.x = pack_bf16x2(fmaf(eg_now, o[8 * c + 0], pu[8 * c + 0]),
                                   fmaf(eg_now, o[8 * c + 1], pu[8 * c + 1]));
                wq.y = pack_bf16x2(fmaf(eg_now, o[8 * c + 2], pu[8 * c + 2]),
                                   fmaf(eg_now, o[8 * c + 3], pu[8 * c + 3]));
                wq.z = pack_bf16x2(fmaf(eg_now, o[8 * c + 4], pu[8 * c + 4]),
                                   fmaf(eg_now, o[8 * c + 5], pu[8 * c + 5]));
                wq.w = pack_bf16x2(fmaf(eg_now, o[8 * c + 6], pu[8 * c + 6]),
                                   fmaf(eg_now, o[8 * c + 7], pu[8 * c + 7]));
                dst[4 * half + c] = wq;
              }
            }
          }
          tc_fence_before();
          mbar_arrive(&bars[B_D1FREE0 + b]);
        }
        ok = ok && ok4;
      }
      if (!bar_and(2, 128, ok)) {
        ok = false;
        break;
      }
    }
    if (ok && !*abort_flag) {
      if (p.mode == kModeSplit) {
        if (part == 0) {
          if (p.parts > 1) {
            float* dst = p.ws_start + ((nh * p.parts + 1) * dv + row0) * DK + ct;
#pragma unroll
            for (int c = 0; c < 64; ++c) dst[(size_t)c * DK] = S[c];
          }
        } else {
          float* dst =
              p.ws_end + ((nh * p.parts + part) * (dv + DK) + row0) * DK + ct;
#pragma unroll
          for (int c = 0; c < 64; ++c) dst[(size_t)c * DK] = S[c];
        }
      } else if (p.hT && part == p.parts - 1) {
        float4* dst = reinterpret_cast<float4*>(p.hT + (nh * DK + ct) * dv + row0);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          dst[c] = make_float4(S[4 * c], S[4 * c + 1], S[4 * c + 2], S[4 * c + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
  if (tid == 0 && *abort_flag) record_status(p.status, GDN_ERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// Self-test: D = A * B (x2 when twice) with the layouts above, one CTA.
// N = 64 or 128 (an N-major B of 128 columns is two 64-column blocks).
__global__ void __launch_bounds__(128)
    selftest_mma_kernel(const __nv_bfloat16* A, const __nv_bfloat16* B,
                        float* D, int K, int N, int a_mn, int b_mn,
                        int b_stacked, int twice, int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 65536);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + 65544);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + 65548);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tmem_alloc(slot, 128);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < 65536 / 16; i += 128)
    reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  for (int idx = tid; idx < 128 * K; idx += 128) {
    const int m = idx / K, k = idx % K;
    const uint32_t off =
        a_mn ? (uint32_t)((m >> 6) * (K * 128)) + sw128(k, (m & 63) >> 3) + (m & 7) * 2
             : (uint32_t)((k >> 6) * 16384) + sw128(m, (k & 63) >> 3) + (k & 7) * 2;
    *reinterpret_cast<__nv_bfloat16*>(sm + off) = A[idx];
  }
  const uint32_t bstride = b_stacked ? 16384u : (uint32_t)N * 128u;
  for (int idx = tid; idx < K * N; idx += 128) {
    const int k = idx / N, nn = idx % N;
    const uint32_t off =
        b_mn ? (uint32_t)((nn >> 6) * (K * 128)) + sw128(k, (nn & 63) >> 3) + (nn & 7) * 2
             : (uint32_t)(k >> 6) * bstride + sw128(nn, (k & 63) >> 3) + (k & 7) * 2;
    *reinterpret_cast<__nv_bfloat16*>(sm + 32768 + off) = B[idx];
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  if (tid == 0) {
    const uint32_t id = idesc_bf16(128, N, a_mn != 0, b_mn != 0);
    for (int pass = 0; pass <= (twice ? 1 : 0); ++pass)
      for (int s = 0; s < K / 16; ++s) {
        const uint64_t a =
            a_mn ? sdesc(base + s * 2048, K * 128, 1024)
                 : sdesc(base + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024);
        const uint64_t b =
            b_mn ? sdesc(base + 32768 + s * 2048, K * 128, 1024)
                 : sdesc(base + 32768 + (s >> 2) * bstride + (s & 3) * 32, 16, 1024);
        mma_bf16(tmem, a, b, id, (pass > 0 || s > 0) ? 1u : 0u);
      }
    mma_commit(bar);
  }
  const bool ok = __syncthreads_and(mbar_wait(bar, 0, abort_flag)) != 0;
  tc_fence_after();
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 64) {
      float d[64];
      tmem_ld64(tmem + ((uint32_t)(32 * warp) << 16) + c0, d);
#pragma unroll
      for (int c = 0; c < 64; ++c) D[tid * N + c0 + c] = d[c];
    }
  } else if (tid == 0) {
    record_status(status, GDN_ERR_TIMEOUT);
  }
  if (!ok) wait_ignoring_abort(bar, 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// ---------------------------------------------------------------------------
// Host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// 3-D map over a [tokens, H, d] bf16 tensor, box = 64 features x 1 head x
// 64 tokens, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* ptr, int d, int H,
              long long tokens) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr),
             dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int VARIANT>
cudaError_t launch_variant(const ChunkParams& p, const CUtensorMap& mq,
                           const CUtensorMap& mk, const CUtensorMap& mv,
                           cudaStream_t stream) {
  auto kern = chunk_tc_kernel<VARIANT>;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int rows = p.mode == kModeSplit ? p.dv + DK : p.dv;
  dim3 grid(rows / DVT, p.H, p.N * p.part_count);
  kern<<<grid, kThreads, SMEM_BYTES, stream>>>(p, mq, mk, mv);
  return cudaGetLastError();
}

}  // namespace

bool chunk_tc_supported(int dk, int dv, long long tokens) {
  return dk == DK && (dv == 64 || dv == 128) && tokens > 0 &&
         tokens < (1ll << 31) - 64;
}

cudaError_t launch_chunk_tc(const ChunkParams& p, cudaStream_t stream) {
  const long long tokens =
      p.cu_seqlens ? (long long)p.T : (long long)p.N * p.T;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, p.q, p.dk, p.H, tokens) ||
      !make_map(&mk, p.k, p.dk, p.H, tokens) ||
      !make_map(&mv, p.v, p.dv, p.H, tokens))
    return cudaErrorInvalidValue;
  return p.variant == GDN_GATE_AFTER_PREDICT
             ? launch_variant<GDN_GATE_AFTER_PREDICT>(p, mq, mk, mv, stream)
             : launch_variant<GDN_GATE_BEFORE_PREDICT>(p, mq, mk, mv, stream);
}

}  // namespace gdn

extern "C" int gdn_selftest_mma(const void* A, const void* B, float* D, int K,
                                int N, int a_mn, int b_mn, int b_stacked,
                                int twice, gdn_stream_t stream) {
  using namespace gdn;
  if (!A || !B || !D || (K != 64 && K != 128) || (N != 64 && N != 128))
    return GDN_ERR_INVALID_ARG;
  if (b_stacked && N != 64) return GDN_ERR_INVALID_ARG;
  if (b_stacked && b_mn) return GDN_ERR_INVALID_ARG;
  int* status = nullptr;
  int rc = device_status_ptr(&status);
  if (rc != GDN_OK) return rc;
  const int bytes = 65536 + 64 + 1024;
  if (cudaFuncSetAttribute(selftest_mma_kernel,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           bytes) != cudaSuccess)
    return GDN_ERR_CUDA;
  selftest_mma_kernel<<<1, 128, bytes, stream>>>(
      static_cast<const __nv_bfloat16*>(A),
      static_cast<const __nv_bfloat16*>(B), D, K, N, a_mn, b_mn, b_stacked,
      twice, status);
  if (count_launches(cudaGetLastError(), 1) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return GDN_ERR_CUDA;
  return gdn_device_status(stream);
}
