// Chunkwise Gated DeltaNet forward pass on the sm_103a tensor cores.
//
// One CTA owns (sequence, head, a 64-row tile of the state's d_v rows) and
// walks the sequence's chunks (C = 64, d_k = 128) in order. The state is kept
// transposed, S^T (d_k x 64), in fp32 registers of the "chain" warpgroup (one
// d_k row per thread) and mirrored as bf16 in shared memory for the MMAs.
// Per chunk (illustrated DeltaNet walk-through: UT transform, chunkwise state
// passing and output; scalar gate prefixes of its GLA section):
//
//   MMA0  [K;Q] K^T           -> K K^T (rows 0-63), Q K^T (rows 64-127)
//   prep  A = strict_lower(diag(beta) K K^T (.) D'),  T = (I + A)^{-1}
//         P = (Q K^T) (.) D (.) M_incl,  Q^ = diag(e^G) Q,  Kbar = diag(e^{G_L-G}) K
//   MMA1  [K;Q^] S^T          -> K S^T, Q^ S^T  (history read)
//   chain R = diag(beta) (V - diag(e^{G'}) K S^T)
//   MMA2  [T;0] R             -> U = T R  (= U0 - W S^T of the WY form)
//   MMA3  Kbar^T U            -> Delta;  S^T <- gamma S^T + Delta
//   MMA4  [0;P] U  (accumulated onto the history read) -> O = Q^ S^T + P U
//
// Folding W into U = T diag(beta)(V - diag(e^{G'}) K S^T) is the same algebra
// as U = U0 - W S^T with U0 = T diag(beta) V, W = T diag(beta e^{G'}) K; it
// removes the W product and its store. D_rj = exp(G_r - G_j) with G the
// chunk-local cumulative log gate, D' and G' take G_{r-1} for
// GDN_GATE_AFTER_PREDICT. Decays are formed as running products of alpha, so
// no exponent is ever positive.
//
// Warp roles (320 threads): warps 0-3 prep, 4-7 chain, 8 TMA producer, 9 MMA
// issuer. Operand tiles are bf16 with the 128-byte swizzle; K/Q/V arrive by
// TMA in a two-stage ring. Every wait is bounded; a CTA that gives up records
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
constexpr int kThreads = 320;

// Stage: [K;Q] stacked K-major tile (two 16 KB column blocks of 64 columns;
// rows 0-63 K, rows 64-127 Q) followed by the V tile (64 x 64).
constexpr uint32_t ST_K = 0;
constexpr uint32_t ST_Q = 8192;
constexpr uint32_t ST_CB = 16384;
constexpr uint32_t ST_V = 32768;
constexpr uint32_t STAGE_BYTES = 40960;
// T | 0 | P buffer: [T;0] and [0;P] are both 128-row K-major tiles.
constexpr uint32_t TP_T = 0, TP_Z = 8192, TP_P = 16384, TP_BYTES = 24576;

constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_TP = 2 * STAGE_BYTES;
constexpr uint32_t OFF_KBAR = OFF_TP + 2 * TP_BYTES;
constexpr uint32_t OFF_S = OFF_KBAR + 16384;
constexpr uint32_t OFF_R = OFF_S + 16384;
constexpr uint32_t OFF_U = OFF_R + 8192;
constexpr int AP = 68;  // fp32 row pitch of the solve buffers
constexpr uint32_t OFF_AT = OFF_U + 8192;
constexpr uint32_t OFF_TF = OFF_AT + 64 * AP * 4;
constexpr int VEC_G = 0, VEC_ALPHA = 64, VEC_EG = 128, VEC_EGP = 192,
              VEC_BETA = 256, VEC_DEC = 320, VEC_GAMMA = 384, VEC_FLOATS = 388;
constexpr uint32_t OFF_VEC = OFF_TF + 64 * AP * 4;
constexpr uint32_t OFF_GB = OFF_VEC + 2 * VEC_FLOATS * 4;
constexpr uint32_t OFF_BAR = OFF_GB + 2 * 128 * 4;

enum {
  B_FULL0, B_FULL1, B_EMPTY0, B_EMPTY1, B_MMA0, B_D0FREE, B_PREP, B_SREADY,
  B_D1FULL0, B_D1FULL1, B_RREADY, B_UFULL, B_UREADY, B_D2FULL, B_D3FULL0,
  B_D3FULL1, B_D1FREE0, B_D1FREE1, B_TPFREE0, B_TPFREE1, B_KBFREE, B_DRAIN,
  NBARS
};
constexpr uint32_t OFF_MISC = OFF_BAR + NBARS * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// TMEM columns (fp32 accumulators, 128 lanes each).
constexpr uint32_t TM_D0 = 0, TM_D1 = 64, TM_DTR = 192, TM_D2 = 256;
constexpr uint32_t TMEM_COLS = 512;

constexpr uint32_t ID_KK = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_KMN = idesc_bf16(128, 64, false, true);
constexpr uint32_t ID_MNMN = idesc_bf16(128, 64, true, true);

__device__ __forceinline__ uint32_t bar_count(int b) {
  switch (b) {
    case B_FULL0: case B_FULL1: return 2;
    case B_D0FREE: case B_PREP: case B_SREADY: return 128;
    case B_RREADY: case B_UREADY: case B_D1FREE0: case B_D1FREE1: return 64;
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

// Scale the 64 bf16 values of row r / column block cb of a swizzled tile.
__device__ __forceinline__ void scale_row_half(const uint8_t* src, uint8_t* dst,
                                               int r, float s) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint4 u = *reinterpret_cast<const uint4*>(src + sw128(r, c));
    float f[8];
    unpack_bf16x8(u, f);
    uint4 w;
    w.x = pack_bf16x2(f[0] * s, f[1] * s);
    w.y = pack_bf16x2(f[2] * s, f[3] * s);
    w.z = pack_bf16x2(f[4] * s, f[5] * s);
    w.w = pack_bf16x2(f[6] * s, f[7] * s);
    *reinterpret_cast<uint4*>(dst + sw128(r, c)) = w;
  }
}

// ---------------------------------------------------------------------------
// (I + A)^{-1} for the strictly lower 64 x 64 A, stored transposed in At
// (At[j][r] = A_rj, zero for r <= j). Result in Tf (lower triangle, unit
// diagonal; entries above the diagonal are not meaningful except inside the
// 32 x 32 diagonal blocks, whose upper parts stay zero). Blocked: the 16 x 16
// diagonal blocks by forward substitution, then T_10 = -T_11 A_10 T_00 at
// 16 and at 32. Products use the zero part of At (r < j) as scratch.
// All 128 prep threads take part.
__device__ __forceinline__ void solve_unit_lower(float* At, float* Tf,
                                                 int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  // 1. diagonal 16 x 16 blocks, one per warp, one column per lane
  if (lane < 16) {
    const int b = 16 * warp;
    float xs[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) xs[m] = (m == lane) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float xj = xs[j];
      const float* arow = At + (b + j) * AP + b;  // A_{b+m, b+j}
#pragma unroll
      for (int m = j + 1; m < 16; ++m) xs[m] = fmaf(-arow[m], xj, xs[m]);
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) Tf[(b + m) * AP + b + lane] = xs[m];
  }
  named_bar(1, 128);
  // 2. merge pairs of 16-blocks: (0,1) by warps 0-1, (2,3) by warps 2-3
  {
    const int pair = warp >> 1;
    const int kb = 32 * pair, rb = kb + 16;
    const int pp = tid & 63, c = pp & 15, rg = pp >> 4;
    float tcol[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) tcol[k] = Tf[(kb + k) * AP + kb + c];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = rg * 4 + q;
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k)
        acc = fmaf(At[(kb + k) * AP + rb + r], tcol[k], acc);
      At[(kb + 16 + r) * AP + kb + c] = acc;  // X = A_10 T_00 (scratch)
    }
    named_bar(5 + pair, 64);
    float xcol[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) xcol[k] = At[(kb + 16 + k) * AP + kb + c];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = rg * 4 + q;
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k)
        acc = fmaf(Tf[(rb + r) * AP + rb + k], xcol[k], acc);
      Tf[(rb + r) * AP + kb + c] = -acc;
    }
  }
  named_bar(1, 128);
  // 3. merge the two 32-blocks
  {
    const int c = tid & 31, rg = tid >> 5;
    float tcol[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) tcol[k] = Tf[k * AP + c];
    float xv[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int r = rg * 8 + q;
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k)
        acc = fmaf(At[k * AP + 32 + r], tcol[k], acc);
      xv[q] = acc;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) At[(32 + rg * 8 + q) * AP + c] = xv[q];
    named_bar(1, 128);
    float xcol[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) xcol[k] = At[(32 + k) * AP + c];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int r = rg * 8 + q;
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k)
        acc = fmaf(Tf[(32 + r) * AP + 32 + k], xcol[k], acc);
      Tf[(32 + r) * AP + c] = -acc;
    }
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
    // zero blocks of both T|0|P buffers and the whole fp32 T buffer
    uint4 z = make_uint4(0, 0, 0, 0);
    for (int i = tid; i < 2 * 512; i += 128) {
      const int b = i >> 9, e = i & 511;
      *reinterpret_cast<uint4*>(sm + OFF_TP + b * TP_BYTES + TP_Z + e * 16) = z;
    }
    for (int i = tid; i < 64 * AP / 4; i += 128)
      reinterpret_cast<uint4*>(sm + OFF_TF)[i] = z;
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

  if (warp == 8) {
    // ================= TMA producer =================
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
        mbar_arrive_expect_tx(full, STAGE_BYTES);
        const int tok = (int)t0;
        tma_load_3d(st + ST_K, &tmk, full, 0, h, tok);
        tma_load_3d(st + ST_K + ST_CB, &tmk, full, 64, h, tok);
        tma_load_3d(st + ST_Q, &tmq, full, 0, h, tok);
        tma_load_3d(st + ST_Q + ST_CB, &tmq, full, 64, h, tok);
        tma_load_3d(st + ST_V, &tmv, full, value_rows ? row0 : 0, h, tok);
      }
      float* gb = reinterpret_cast<float*>(sm + OFF_GB) + s * 128;
      for (int r = lane; r < C; r += 32) {
        float gg = 0.f, bb = 0.f;
        if (r < len) {
          const size_t row = (size_t)(t0 + r) * H + h;
          gg = p.g[row];
          bb = p.beta[row];
        }
        gb[r] = gg;
        gb[64 + r] = bb;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(full);
      issued = i + 1;
    }
    // never leave with a TMA copy still landing in shared memory
    if (lane == 0)
      for (int i = max(0, issued - 2); i < issued; ++i)
        wait_ignoring_abort(&bars[B_FULL0 + (i & 1)], (i >> 1) & 1);
  } else if (warp == 9) {
    // ================= MMA issuer =================
    if (lane == 0 && nloc > 0) {
      auto stage = [&](int i) { return base + OFF_STAGE + (i & 1) * STAGE_BYTES; };
      auto mma0 = [&](int i) {
        const uint32_t st = stage(i);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t a = sdesc(st + (k >> 2) * ST_CB + (k & 3) * 32, 16, 1024);
          mma_bf16(tmem + TM_D0, a, a, ID_KK, k > 0);
        }
      };
      bool ok = mbar_wait(&bars[B_FULL0], 0, abort_flag);
      if (ok) {
        tc_fence_after();
        mma0(0);
        mma_commit(&bars[B_MMA0]);
      }
      for (int i = 0; ok && i < nloc; ++i) {
        const int b = i & 1;
        if (i + 1 < nloc) {
          ok = mbar_wait(&bars[B_FULL0 + ((i + 1) & 1)], ((i + 1) >> 1) & 1,
                         abort_flag) &&
               mbar_wait(&bars[B_D0FREE], i & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          mma0(i + 1);
          mma_commit(&bars[B_MMA0]);
        }
        ok = mbar_wait(&bars[B_SREADY], i & 1, abort_flag) &&
             mbar_wait(&bars[B_PREP], i & 1, abort_flag) &&
             (i < 2 || mbar_wait(&bars[B_D1FREE0 + b], ((i >> 1) - 1) & 1,
                                 abort_flag));
        if (!ok) break;
        tc_fence_after();
        const uint32_t st = stage(i);
        const uint32_t d1 = tmem + TM_D1 + 64 * b;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_bf16(d1, sdesc(st + (k >> 2) * ST_CB + (k & 3) * 32, 16, 1024),
                   sdesc(base + OFF_S + k * 2048, 8192, 1024), ID_KMN, k > 0);
        mma_commit(&bars[B_D1FULL0 + b]);

        ok = mbar_wait(&bars[B_RREADY], i & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tp = base + OFF_TP + b * TP_BYTES;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem + TM_DTR, sdesc(tp + TP_T + k * 32, 16, 1024),
                   sdesc(base + OFF_R + k * 2048, 8192, 1024), ID_KMN, k > 0);
        mma_commit(&bars[B_UFULL]);
        mma_commit(&bars[B_EMPTY0 + b]);

        ok = mbar_wait(&bars[B_UREADY], i & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem + TM_D2, sdesc(base + OFF_KBAR + k * 2048, 8192, 1024),
                   sdesc(base + OFF_U + k * 2048, 8192, 1024), ID_MNMN, k > 0);
        mma_commit(&bars[B_D2FULL]);
        mma_commit(&bars[B_KBFREE]);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(d1, sdesc(tp + TP_Z + k * 32, 16, 1024),
                   sdesc(base + OFF_U + k * 2048, 8192, 1024), ID_KMN, 1);
        mma_commit(&bars[B_D3FULL0 + b]);
        mma_commit(&bars[B_TPFREE0 + b]);
      }
      // every MMA issued must finish before TMEM is released
      mma_commit(&bars[B_DRAIN]);
      wait_ignoring_abort(&bars[B_DRAIN], 0);
    }
  } else if (warp < 4) {
    // ================= prep warpgroup =================
    float* At = reinterpret_cast<float*>(sm + OFF_AT);
    float* Tf = reinterpret_cast<float*>(sm + OFF_TF);
    const uint32_t lanes = (uint32_t)(32 * warp) << 16;
    for (int j = 0; j < nloc; ++j) {
      const int s = j & 1;
      float* vec = reinterpret_cast<float*>(sm + OFF_VEC) + s * VEC_FLOATS;
      const float* gb = reinterpret_cast<const float*>(sm + OFF_GB) + s * 128;
      uint8_t* st = sm + OFF_STAGE + s * STAGE_BYTES;
      uint8_t* tp = sm + OFF_TP + s * TP_BYTES;
      // the stage's TMA data and gates (full) and the K K^T / Q K^T product
      bool ok = mbar_wait(&bars[B_FULL0 + s], (j >> 1) & 1, abort_flag) &&
                mbar_wait(&bars[B_MMA0], j & 1, abort_flag);
      if (!bar_and(1, 128, ok)) break;
      tc_fence_after();
      if (warp == 0) {
        // chunk-local gate prefixes (inclusive scan of g over 64 tokens)
        const unsigned full = 0xffffffffu;
        const float g0 = gb[lane], g1 = gb[lane + 32];
        float s0 = g0, s1 = g1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float t0 = __shfl_up_sync(full, s0, o);
          const float t1 = __shfl_up_sync(full, s1, o);
          if (lane >= o) {
            s0 += t0;
            s1 += t1;
          }
        }
        s1 += __shfl_sync(full, s0, 31);
        const float Gl = __shfl_sync(full, s1, 31);
        vec[VEC_G + lane] = s0;
        vec[VEC_G + 32 + lane] = s1;
        vec[VEC_ALPHA + lane] = expf(g0);
        vec[VEC_ALPHA + 32 + lane] = expf(g1);
        vec[VEC_EG + lane] = expf(s0);
        vec[VEC_EG + 32 + lane] = expf(s1);
        const float p0 = VARIANT == GDN_GATE_BEFORE_PREDICT ? s0 : s0 - g0;
        const float p1 = VARIANT == GDN_GATE_BEFORE_PREDICT ? s1 : s1 - g1;
        vec[VEC_EGP + lane] = expf(p0);
        vec[VEC_EGP + 32 + lane] = expf(p1);
        vec[VEC_BETA + lane] = gb[64 + lane];
        vec[VEC_BETA + 32 + lane] = gb[96 + lane];
        vec[VEC_DEC + lane] = expf(Gl - s0);
        vec[VEC_DEC + 32 + lane] = expf(Gl - s1);
        if (lane == 0) vec[VEC_GAMMA] = expf(Gl);
      }
      float x[64];
      tmem_ld64(tmem + TM_D0 + lanes, x);
      tc_fence_before();
      mbar_arrive(&bars[B_D0FREE]);
      ok = j < 2 || mbar_wait(&bars[B_TPFREE0 + s], ((j >> 1) - 1) & 1,
                              abort_flag);
      if (!bar_and(1, 128, ok)) break;  // also publishes vec
      const float* alpha = vec + VEC_ALPHA;
      if (tid < 64) {
        // row r of A: beta_r exp(G'_r - G_j) k_r.k_j for j < r
        const int r = tid;
        const float br = vec[VEC_BETA + r];
        float d = 1.f;
#pragma unroll
        for (int jj = 63; jj >= 0; --jj) {
          float a = 0.f;
          if (jj < r) {
            if (VARIANT == GDN_GATE_BEFORE_PREDICT) {
              d *= alpha[jj + 1];
              a = br * d * x[jj];
            } else {
              a = br * d * x[jj];
              d *= alpha[jj];
            }
          }
          At[jj * AP + r] = a;
        }
      } else {
        // row r of P: exp(G_r - G_j) q_r.k_j for j <= r
        const int r = tid - 64;
        float d = 1.f;
#pragma unroll
        for (int jj = 63; jj >= 0; --jj) {
          float pv = 0.f;
          if (jj <= r) {
            pv = d * x[jj];
            d *= alpha[jj];
          }
          x[jj] = pv;
        }
        store_row_bf16(tp + TP_P, r, x);
      }
      {
        // Q^ = diag(e^G) Q in place (MMA0 is done with Q)
        const int r = tid >> 1, cb = tid & 1;
        uint8_t* q = st + ST_Q + cb * ST_CB;
        scale_row_half(q, q, r, vec[VEC_EG + r]);
      }
      named_bar(1, 128);
      solve_unit_lower(At, Tf, tid);
      {
        // T -> bf16 rows 0-63 of [T;0]
        const int r = tid >> 1, hh = tid & 1;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int cc = hh * 4 + q4;
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int col = cc * 8 + e;
            f[e] = col < r ? Tf[r * AP + col] : (col == r ? 1.f : 0.f);
          }
          uint4 w;
          w.x = pack_bf16x2(f[0], f[1]);
          w.y = pack_bf16x2(f[2], f[3]);
          w.z = pack_bf16x2(f[4], f[5]);
          w.w = pack_bf16x2(f[6], f[7]);
          *reinterpret_cast<uint4*>(tp + TP_T + sw128(r, cc)) = w;
        }
      }
      ok = j == 0 || mbar_wait(&bars[B_KBFREE], (j - 1) & 1, abort_flag);
      if (!bar_and(1, 128, ok)) break;
      {
        // Kbar = diag(e^{G_L - G}) K
        const int r = tid >> 1, cb = tid & 1;
        scale_row_half(st + ST_K + cb * ST_CB, sm + OFF_KBAR + cb * 8192, r,
                       vec[VEC_DEC + r]);
      }
      fence_proxy_async();
      mbar_arrive(&bars[B_PREP]);
    }
  } else {
    // ================= chain warpgroup =================
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
    fence_proxy_async();
    mbar_arrive(&bars[B_SREADY]);
    bool ok = true;
    for (int i = 0; i < nloc; ++i) {
      const int s = i & 1, b = i & 1;
      ok = ok && mbar_wait(&bars[B_PREP], i & 1, abort_flag);
      if (!bar_and(2, 128, ok)) {
        ok = false;
        break;
      }
      const float* vec = reinterpret_cast<const float*>(sm + OFF_VEC) + s * VEC_FLOATS;
      const float gam = vec[VEC_GAMMA];
      const long long t0 = bos + (long long)(c_begin + i) * C;
      const int len = (int)min((long long)C, eos - t0);
      if (cw < 2) {
        const int r = ct;
        bool ok1 = mbar_wait(&bars[B_FULL0 + s], (i >> 1) & 1, abort_flag) &&
                   mbar_wait(&bars[B_D1FULL0 + b], (i >> 1) & 1, abort_flag);
        ok1 = bar_and(3, 64, ok1);
        if (ok1) {
          tc_fence_after();
          float ks[64];
          tmem_ld64(tmem + TM_D1 + 64 * b + lanes, ks);
          const float e = vec[VEC_EGP + r], be = vec[VEC_BETA + r];
          const uint8_t* vt = sm + OFF_STAGE + s * STAGE_BYTES + ST_V;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float f[8];
            if (scale_rows) {
#pragma unroll
              for (int e8 = 0; e8 < 8; ++e8) f[e8] = 0.f;
            } else {
              unpack_bf16x8(*reinterpret_cast<const uint4*>(vt + sw128(r, c)), f);
            }
#pragma unroll
            for (int e8 = 0; e8 < 8; ++e8)
              ks[8 * c + e8] = be * fmaf(-e, ks[8 * c + e8], f[e8]);
          }
          store_row_bf16(sm + OFF_R, r, ks);
          fence_proxy_async();
          tc_fence_before();
          mbar_arrive(&bars[B_RREADY]);
          bool ok2 = mbar_wait(&bars[B_UFULL], i & 1, abort_flag);
          ok2 = bar_and(3, 64, ok2);
          if (ok2) {
            tc_fence_after();
            float u[64];
            tmem_ld64(tmem + TM_DTR + lanes, u);
            store_row_bf16(sm + OFF_U, r, u);
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(&bars[B_UREADY]);
          }
          ok = ok2;
        } else {
          ok = false;
        }
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
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&bars[B_SREADY]);
      if (cw >= 2) {
        const int r = ct - 64;
        bool ok4 = mbar_wait(&bars[B_D3FULL0 + b], (i >> 1) & 1, abort_flag);
        ok4 = bar_and(4, 64, ok4);
        if (ok4) {
          tc_fence_after();
          float o[64];
          tmem_ld64(tmem + TM_D1 + 64 * b + lanes, o);
          if (emit && r < len) {
            uint4* dst = reinterpret_cast<uint4*>(
                static_cast<__nv_bfloat16*>(p.out) +
                ((size_t)(t0 + r) * H + h) * dv + row0);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint4 w;
              w.x = pack_bf16x2(o[8 * c + 0], o[8 * c + 1]);
              w.y = pack_bf16x2(o[8 * c + 2], o[8 * c + 3]);
              w.z = pack_bf16x2(o[8 * c + 4], o[8 * c + 5]);
              w.w = pack_bf16x2(o[8 * c + 6], o[8 * c + 7]);
              dst[c] = w;
            }
          }
          tc_fence_before();
          mbar_arrive(&bars[B_D1FREE0 + b]);
        } else {
          ok = false;
        }
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
__global__ void __launch_bounds__(128)
    selftest_mma_kernel(const __nv_bfloat16* A, const __nv_bfloat16* B,
                        float* D, int K, int a_mn, int b_mn, int b_stacked,
                        int twice, int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 65536);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + 65544);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + 65548);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tmem_alloc(slot, 64);
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
  const uint32_t bstride = b_stacked ? 16384u : 8192u;
  for (int idx = tid; idx < K * 64; idx += 128) {
    const int k = idx / 64, nn = idx % 64;
    const uint32_t off =
        b_mn ? sw128(k, nn >> 3) + (nn & 7) * 2
             : (uint32_t)(k >> 6) * bstride + sw128(nn, (k & 63) >> 3) + (k & 7) * 2;
    *reinterpret_cast<__nv_bfloat16*>(sm + 32768 + off) = B[idx];
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  if (tid == 0) {
    const uint32_t id = idesc_bf16(128, 64, a_mn != 0, b_mn != 0);
    for (int pass = 0; pass <= (twice ? 1 : 0); ++pass)
      for (int s = 0; s < K / 16; ++s) {
        const uint64_t a =
            a_mn ? sdesc(base + s * 2048, K * 128, 1024)
                 : sdesc(base + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024);
        const uint64_t b =
            b_mn ? sdesc(base + 32768 + s * 2048, 8192, 1024)
                 : sdesc(base + 32768 + (s >> 2) * bstride + (s & 3) * 32, 16, 1024);
        mma_bf16(tmem, a, b, id, (pass > 0 || s > 0) ? 1u : 0u);
      }
    mma_commit(bar);
  }
  const bool ok = __syncthreads_and(mbar_wait(bar, 0, abort_flag)) != 0;
  tc_fence_after();
  if (ok) {
    float d[64];
    tmem_ld64(tmem + ((uint32_t)(32 * warp) << 16), d);
#pragma unroll
    for (int c = 0; c < 64; ++c) D[tid * 64 + c] = d[c];
  } else if (tid == 0) {
    record_status(status, GDN_ERR_TIMEOUT);
  }
  if (!ok) wait_ignoring_abort(bar, 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
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
                                int a_mn, int b_mn, int b_stacked, int twice,
                                gdn_stream_t stream) {
  using namespace gdn;
  if (!A || !B || !D || (K != 64 && K != 128)) return GDN_ERR_INVALID_ARG;
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
      static_cast<const __nv_bfloat16*>(B), D, K, a_mn, b_mn, b_stacked, twice,
      status);
  if (count_launches(cudaGetLastError(), 1) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return GDN_ERR_CUDA;
  return gdn_device_status(stream);
}
