// Chunked KDA (per-channel decay) for the tensor-core chain: the preparation
// of every (chunk, head).
//
// Illustrated DeltaNet walk-through: the KDA paragraphs of its
// hybrid-architecture section give the recurrence
//   S_t = S_{t-1} diag(e^{g_t}) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
//   o_t = S_t q_t,
// its UT transform and WY sections the chunk form, and its GLA section the
// per-channel cumulative gates with the rescaling over 16-token sub-chunks.
// With Gamma_t = sum_{s <= t} g_s the chunk-local cumulative log-decay (a
// vector over the key channels; the decay of token t acts before its
// prediction) one chunk of C = 64 tokens from the state S_0 is
//   A_rs = beta_r sum_c k_rc k_sc e^{Gamma_rc - Gamma_sc}      (s < r)
//   P_rs = sum_c q_rc k_sc e^{Gamma_rc - Gamma_sc}             (s <= r)
//   T = (I + A)^{-1},  T_U = T diag(beta),  W = T_U (K (.) e^Gamma)
//   U = T_U V - W S_0^T,   O = (Q (.) e^Gamma) S_0^T + P U
//   S_C = S_0 diag(e^{Gamma_L}) + U^T (K (.) e^{Gamma_L - Gamma})
// (Gamma_L: the chunk's last token). That is the scalar-gate chunk form with
// Q_g = Q (.) e^Gamma, K_d = K (.) e^{Gamma_L - Gamma} and a decay vector
// gamma = e^{Gamma_L}, so the whole-state chain kernel runs it unchanged but
// for the column-wise decay of the state; this kernel writes -W, P, T_U, Q_g
// and K_d as bf16 tile images and e^{Gamma_L} as the chunk's decay record.
//
// A and P need e^{Gamma_r - Gamma_s} channel by channel. With ref(t) the
// cumulative decay before the first token of t's 16-token block the kernel
// factors it as
//   e^{Gamma_r - ref(r)}  x  e^{ref(r) - ref(s)}  x  e^{ref(s) - Gamma_s}
// (left table K_E = K (.) e^{Gamma - ref}, Q_E likewise, right table
// K_B = K (.) e^{ref - Gamma}, one vector per pair of blocks), so every block
// of A and P is one bf16 tensor-core product over d_k. All factors but
// the right table's lie in (0, 1] for decays (g <= 0); the right table grows
// by at most the decay across one block. A chunk in which some channel decays
// by more than 2^120 across one block (or grows by that much between two)
// takes the exact pairwise sum instead (one exp per term; slow, but only for
// such chunks).
//
// One CTA of 256 threads per (chunk, head) at a time, two CTAs per SM,
// persistent. The g and k rows of the CTA's next item arrive by two
// tensor-map copies into the operand tables' space once the A and P products
// have read them (per-thread loads of those rows were held to about 2.5 TB/s
// by the requests an SM keeps in flight); q rows by per-thread loads.
// Tensor-core products with mma.sync m16n8k16 (bf16 in, fp32 accumulate)
// from ldmatrix fragments, the inverse by the blocked substitution shared
// with the scalar-gate preparation; images out by a bulk copy (P) or plain
// stores (T_U, -W, Q_g, K_d: a proxy fence while the next rows land would
// wait for them).
#include "chunk_tiles.cuh"

namespace gdn {
namespace {
using namespace tc;

constexpr int kKpThreads = 256;
constexpr int kKpCtas = 2;
// bf16 operand tables, 64 rows of 136 values (the 16-byte pad makes the
// eight rows of an ldmatrix tile hit distinct banks)
constexpr int KP_PITCH = 272;
constexpr uint32_t KP_TAB = 64 * KP_PITCH;
constexpr uint32_t KP_KE = 0, KP_QE = KP_TAB, KP_KB = 2 * KP_TAB,
                   KP_KG = 3 * KP_TAB;
// exact fallback: Gamma in fp32 over K_E / Q_E, raw K in the K_B table
constexpr int GP = 132;
constexpr uint32_t KP_GAM = 0;
constexpr uint32_t KP_AT = 4 * KP_TAB;             // fp32 A, then T (pitch AP)
// -W image after T_U is built, over the solve buffer
constexpr uint32_t KP_W = KP_AT;
// The next item's g rows (fp32 [64][d_k]) and k rows (bf16 [64][d_k]) arrive
// by tensor-map copies over K_E / Q_E and K_B once the A and P products are
// done
constexpr uint32_t KP_SG = 0, KP_SK = KP_KB;
constexpr uint32_t KP_P = KP_AT + 64 * AP * 4;     // P image
constexpr uint32_t KP_TU = KP_P + TILE_BYTES;      // T_U image
constexpr uint32_t KP_V = KP_TU + TILE_BYTES;      // 6 pair vectors x 128
constexpr uint32_t KP_QT = KP_V + 6 * DK * 4;      // per-block decay totals
constexpr uint32_t KP_BETA = KP_QT + 4 * DK * 4;    // beta (0 past the end)
constexpr uint32_t KP_BAR = KP_BETA + 64 * 4;       // stage mbarrier, abort flag
constexpr uint32_t KP_SMEM = KP_BAR + 16 + 1024;
static_assert(64 * GP * 4 <= KP_KB, "Gamma table overlaps the raw K table");
static_assert(WS_W_BYTES <= 64 * AP * 4, "-W image fits the solve buffer");
static_assert(64 * DK * 4 <= KP_KB && KP_SK + 64 * DK * 2 <= KP_KG,
              "row stage fits the operand tables");
static_assert(KP_BAR % 8 == 0, "mbarrier alignment");
static_assert(KP_P % 1024 == 0 && KP_TU % 1024 == 0, "image alignment");
static_assert(kKpCtas * (KP_SMEM + 1024) <= 233472, "two CTAs per SM");
// largest |log2 factor| a table entry may carry
constexpr float kSpanLimit = 120.f;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr)
      : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr)
      : "memory");
}
// c += a b (m16n8k16, bf16 inputs, fp32 accumulators)
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t u, float2 s) {
  const float lo = __uint_as_float(u << 16), hi = __uint_as_float(u & 0xffff0000u);
  return pack_bf16x2(lo * s.x, hi * s.y);
}
// 2^x on the special-function unit (flushes results below 2^-126 to 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float bf16_bits(uint32_t b) {
  return __uint_as_float(b << 16);
}

__global__ void __launch_bounds__(kKpThreads, kKpCtas)
    kda_prep_kernel(const ChunkParams p,
                    const __grid_constant__ CUtensorMap tmg,
                    const __grid_constant__ CUtensorMap tmk, int nch_dense,
                    int total_chunks_bound) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H;
  // an invalid packing (already recorded as GDN_ERR_INVALID_ARG) can count
  // more chunks than the workspace holds: never write past it
  const int total_chunks =
      p.chunk_off ? min(p.chunk_off[p.N], total_chunks_bound) : total_chunks_bound;
  const int items = total_chunks * H;
  // the chain kernel behind this one may be scheduled from here on; it waits
  // for this grid to complete before it reads the images
  griddep_launch_dependents();

  float* AT = reinterpret_cast<float*>(sm + KP_AT);
  float* vpair = reinterpret_cast<float*>(sm + KP_V);
  float* bet = reinterpret_cast<float*>(sm + KP_BETA);
  const uint16_t* qin = static_cast<const uint16_t*>(p.q);

  auto chunk_of = [&](int it, int& h, long long& t0, int& len) {
    const int cidx = it / H;
    h = it - cidx * H;
    int n, lc;
    locate_chunk(p, cidx, nch_dense, n, lc);
    long long bos, eos;
    if (!sequence_range(p, n, bos, eos)) bos = eos = 0;
    t0 = bos + (long long)lc * C;
    len = (int)max(0ll, min((long long)C, eos - t0));
  };
  uint64_t* sbar = reinterpret_cast<uint64_t*>(sm + KP_BAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + KP_BAR + 8);
  if (tid == 0) {
    mbar_init(sbar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Item it_'s g and k rows (64 tokens of one head: tiles of d_k x 64,
  // rows past the tensor's end zero-filled, rows past the sequence's end
  // unused) into the stage by two tensor-map copies that complete on the
  // stage barrier; one thread. q is loaded per thread: the tables leave no
  // room for its rows.
  auto issue_stage = [&](int it_) {
    int h_, len_;
    long long t0_;
    chunk_of(it_, h_, t0_, len_);
    mbar_arrive_expect_tx(sbar, 64 * DK * 4 + 64 * DK * 2);
    tma_load_3d(sm + KP_SG, &tmg, sbar, 0, h_, (int)t0_);
    tma_load_3d(sm + KP_SK, &tmk, sbar, 0, h_, (int)t0_);
  };
  int staged = 0, li = 0;  // stages issued, stages consumed (same in every thread)
  if (blockIdx.x < items) {
    if (tid == 0) {
      prefetch_tmap(&tmg);
      prefetch_tmap(&tmk);
      issue_stage(blockIdx.x);
    }
    ++staged;
  }

  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    int h, len;
    long long t0;
    chunk_of(it, h, t0, len);
    // the CTA's next item's q rows (256 bytes each) into L2 while this one
    // is processed (its g and k rows come by the stage)
    if (warp == 7 && it + (int)gridDim.x < items) {
      int h2, len2;
      long long t2;
      chunk_of(it + gridDim.x, h2, t2, len2);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int t = lane + 32 * hf;
        if (t < len2) {
          const size_t e = ((size_t)(t2 + t) * H + h2) * DK;
          prefetch_l2(qin + e, DK * 2);
        }
      }
    }
    // ---- 1. cumulative log2-decay over the chunk --------------------------
    // thread (block R1 = tid >> 6, channel pair cp = tid & 63): tokens
    // 16 R1 .. 16 R1 + 15 of key channels 2 cp and 2 cp + 1. Each block is
    // referred to the cumulative decay before its first token, ref_R1.
    const int R1 = tid >> 6, cp = tid & 63, c0 = 2 * cp;
    float2 x[16];           // Gamma_t - ref_R1 (log2 units)
    uint32_t kk2[16], qq2[16];  // raw k and q, two channels each
    {
      // the q rows first, so that they travel while the stage is awaited
      const size_t e0 = ((size_t)(t0 + 16 * R1) * H + h) * DK + c0;
      const size_t rs = (size_t)H * DK;  // token stride in elements
#pragma unroll
      for (int j = 0; j < 16; ++j)
        qq2[j] = 16 * R1 + j < len
                     ? __ldg(reinterpret_cast<const uint32_t*>(qin + e0 + (size_t)j * rs))
                     : 0u;
    }
    // the previous item's bulk copies have read their images; this item's
    // g and k rows have landed
    if (tid == 0) bulk_wait_read();
    const bool landed = mbar_wait(sbar, li & 1, abort_flag);
    if (!bar_and(2, kKpThreads, landed)) break;
    ++li;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float2 gv = make_float2(0.f, 0.f);
      uint32_t kb = 0;
      const int t = 16 * R1 + j;
      if (t < len) {
        gv = *reinterpret_cast<const float2*>(sm + KP_SG + t * (DK * 4) + c0 * 4);
        kb = *reinterpret_cast<const uint32_t*>(sm + KP_SK + t * (DK * 2) + c0 * 2);
      }
      x[j] = make_float2(gv.x * kLog2e, gv.y * kLog2e);
      kk2[j] = kb;
    }
#pragma unroll
    for (int j = 1; j < 16; ++j) {
      x[j].x += x[j - 1].x;
      x[j].y += x[j - 1].y;
    }
    float2* qtot = reinterpret_cast<float2*>(sm + KP_QT);  // [4 blocks][64 pairs]
    qtot[R1 * 64 + cp] = x[15];
    if (tid < 64) bet[tid] = tid < len ? __ldg(p.beta + ((size_t)(t0 + tid) * H + h)) : 0.f;
    __syncthreads();
    float2 own = make_float2(0.f, 0.f), xl = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 v = qtot[q * 64 + cp];
      if (q < R1) {
        own.x += v.x;
        own.y += v.y;
      }
      xl.x += v.x;
      xl.y += v.y;
    }
    bool bad = false;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      bad |= fabsf(x[j].x) > kSpanLimit || fabsf(x[j].y) > kSpanLimit;
    {
      // 2^{ref_R1 - ref_S} for the blocks S < R1: the pair vectors
      float2 acc = make_float2(0.f, 0.f);
      for (int S = R1 - 1; S >= 0; --S) {
        const float2 v = qtot[S * 64 + cp];
        acc.x += v.x;
        acc.y += v.y;
        bad |= acc.x > kSpanLimit || acc.y > kSpanLimit;
        *reinterpret_cast<float2*>(vpair + (R1 * (R1 - 1) / 2 + S) * DK + c0) =
            make_float2(ex2(acc.x), ex2(acc.y));
      }
    }
    const bool exact = __syncthreads_or(bad) != 0;

    // ---- 2. operand tables, the Q_g / K_d images, the decay record -------
    {
      float* cv = p.cv + (size_t)it * KCV_FLOATS;
      // e^G = 1 for the chain's read-out (the decay is inside Q_g)
      if (R1 == 1) *reinterpret_cast<float2*>(cv + c0) = make_float2(1.f, 1.f);
      if (R1 == 0)
        *reinterpret_cast<float2*>(cv + CV_GAMMA + c0) = make_float2(ex2(xl.x), ex2(xl.y));
      uint8_t* qimg = static_cast<uint8_t*>(p.qg) + (size_t)it * WS_QG_BYTES +
                      (c0 >> 6) * TILE_BYTES + (c0 & 7) * 2;
      uint8_t* kimg = static_cast<uint8_t*>(p.kd) + (size_t)it * WS_KD_BYTES +
                      (c0 >> 6) * TILE_BYTES + (c0 & 7) * 2;
      const int cchunk = (c0 & 63) >> 3;
      const float2 eown = make_float2(ex2(own.x), ex2(own.y));
      float2* gam = reinterpret_cast<float2*>(sm + KP_GAM);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = 16 * R1 + j;
        const float k0 = bf16_bits(kk2[j] & 0xffffu), k1 = bf16_bits(kk2[j] >> 16);
        const float q0 = bf16_bits(qq2[j] & 0xffffu), q1 = bf16_bits(qq2[j] >> 16);
        const float E0 = ex2(x[j].x), E1 = ex2(x[j].y);
        const float g0 = E0 * eown.x, g1 = E1 * eown.y;  // e^{Gamma_t}
        const float d0 = ex2(xl.x - own.x - x[j].x), d1 = ex2(xl.y - own.y - x[j].y);
        const uint32_t off = sw128(t, cchunk);
        *reinterpret_cast<uint32_t*>(qimg + off) = pack_bf16x2(q0 * g0, q1 * g1);
        *reinterpret_cast<uint32_t*>(kimg + off) = pack_bf16x2(k0 * d0, k1 * d1);
        const uint32_t row = t * KP_PITCH + c0 * 2;
        *reinterpret_cast<uint32_t*>(sm + KP_KG + row) = pack_bf16x2(k0 * g0, k1 * g1);
        if (!exact) {
          const float I0 = ex2(-x[j].x), I1 = ex2(-x[j].y);
          *reinterpret_cast<uint32_t*>(sm + KP_KE + row) = pack_bf16x2(k0 * E0, k1 * E1);
          *reinterpret_cast<uint32_t*>(sm + KP_QE + row) = pack_bf16x2(q0 * E0, q1 * E1);
          *reinterpret_cast<uint32_t*>(sm + KP_KB + row) = pack_bf16x2(k0 * I0, k1 * I1);
        } else {
          gam[(t * GP + c0) >> 1] = make_float2(x[j].x + own.x, x[j].y + own.y);
          *reinterpret_cast<uint32_t*>(sm + KP_KB + row) = kk2[j];
        }
      }
    }
    __syncthreads();

    // ---- 3. A and P in 16 x 16 blocks, spread over the warps --------------
    // 20 blocks on or below the diagonal (12 off it first: those carry the
    // pair vectors), then the 12 zero blocks above it; warp w takes jobs
    // w, w + 8, ..
    {
      const int g = lane >> 2, t4 = lane & 3;
      uint8_t* pimg = sm + KP_P;
      float acc[2][4];
      // block (mat, R, S) out of the accumulators: A (times beta_r, s < r)
      // into the solve buffer, P (s <= r) into its bf16 image
      auto put_block = [&](int mat, int R, int S) {
        const int r0 = 16 * R + g, r1 = r0 + 8;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          const int s = 16 * S + 8 * n + 2 * t4;
          if (mat == 0) {
            const float b0 = bet[r0], b1 = bet[r1];
            *reinterpret_cast<float2*>(AT + r0 * AP + s) =
                make_float2(s < r0 ? b0 * acc[n][0] : 0.f,
                            s + 1 < r0 ? b0 * acc[n][1] : 0.f);
            *reinterpret_cast<float2*>(AT + r1 * AP + s) =
                make_float2(s < r1 ? b1 * acc[n][2] : 0.f,
                            s + 1 < r1 ? b1 * acc[n][3] : 0.f);
          } else {
            *reinterpret_cast<uint32_t*>(pimg + sw128(r0, s >> 3) + (s & 7) * 2) =
                pack_bf16x2(s <= r0 ? acc[n][0] : 0.f, s + 1 <= r0 ? acc[n][1] : 0.f);
            *reinterpret_cast<uint32_t*>(pimg + sw128(r1, s >> 3) + (s & 7) * 2) =
                pack_bf16x2(s <= r1 ? acc[n][2] : 0.f, s + 1 <= r1 ? acc[n][3] : 0.f);
          }
        }
      };
      // pair index pr (0..5) -> (R, S), S < R: (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
      auto pair_rs = [](int pr, int& R, int& S) {
        R = pr < 1 ? 1 : (pr < 3 ? 2 : 3);
        S = pr - R * (R - 1) / 2;
      };
      for (int job = warp; job < 32; job += 8) {
        int mat, R, S;
        if (job < 12) {
          mat = job / 6;
          pair_rs(job % 6, R, S);
        } else if (job < 20) {
          mat = (job - 12) >> 2;
          R = S = (job - 12) & 3;
        } else {
          mat = (job - 20) / 6;
          pair_rs((job - 20) % 6, S, R);  // mirrored: above the diagonal
        }
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
        if (job < 20 && !exact) {
          // left rows 16 R.. (K_E or Q_E), right rows 16 S.. of K_B (two
          // 8-row n tiles, times the pair vector off the diagonal)
          const uint32_t tab = base + (mat ? KP_QE : KP_KE);
          const int ar = 16 * R + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int br = 16 * S + (lane & 7) + (lane >> 4) * 8;
          const int ac = (lane >> 4) * 8, bc = ((lane >> 3) & 1) * 8;
          const float* vp = vpair + (R * (R - 1) / 2 + S) * DK + 2 * t4;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            uint32_t a[4], b[4];
            ldsm_x4(tab + ar * KP_PITCH + (16 * kk + ac) * 2, a);
            ldsm_x4(base + KP_KB + br * KP_PITCH + (16 * kk + bc) * 2, b);
            if (S < R) {
              const float2 v0 = *reinterpret_cast<const float2*>(vp + 16 * kk);
              const float2 v1 = *reinterpret_cast<const float2*>(vp + 16 * kk + 8);
              b[0] = scale_bf16x2(b[0], v0);
              b[1] = scale_bf16x2(b[1], v1);
              b[2] = scale_bf16x2(b[2], v0);
              b[3] = scale_bf16x2(b[3], v1);
            }
            mma16816(acc[0], a, b[0], b[1]);
            mma16816(acc[1], a, b[2], b[3]);
          }
        } else if (job < 20) {
          // exact sum: each lane's 8 entries of the block, channel by channel
          const float* gam = reinterpret_cast<const float*>(sm + KP_GAM);
          const uint16_t* kraw = reinterpret_cast<const uint16_t*>(sm + KP_KB);
          const int kp = KP_PITCH / 2;
          const int r0 = 16 * R + g, r1 = r0 + 8;
          for (int ch = 0; ch < DK; ++ch) {
            const float gr0 = gam[r0 * GP + ch], gr1 = gam[r1 * GP + ch];
            float x0, x1;
            if (mat == 0) {
              x0 = bf16_bits(kraw[r0 * kp + ch]);
              x1 = bf16_bits(kraw[r1 * kp + ch]);
            } else {
              x0 = r0 < len ? bf16_bits(__ldg(qin + ((size_t)(t0 + r0) * H + h) * DK + ch)) : 0.f;
              x1 = r1 < len ? bf16_bits(__ldg(qin + ((size_t)(t0 + r1) * H + h) * DK + ch)) : 0.f;
            }
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int s = 16 * S + 8 * n + 2 * t4 + e;
                const float ks = bf16_bits(kraw[s * kp + ch]), gs = gam[s * GP + ch];
                acc[n][e] = fmaf(x0 * ks, exp2f(gr0 - gs), acc[n][e]);
                acc[n][2 + e] = fmaf(x1 * ks, exp2f(gr1 - gs), acc[n][2 + e]);
              }
          }
        }
        put_block(mat, R, S);
      }
      fence_proxy_async();
    }
    __syncthreads();
    if (tid == 0) {
      bulk_store(static_cast<uint8_t*>(p.pm) + (size_t)it * WS_P_BYTES, sm + KP_P,
                 TILE_BYTES);
      bulk_commit();
    }
    // the operand tables are read: the next item's rows may land over them
    // while the inverse and W run (warp 7 does not take part in the solve)
    if (it + (int)gridDim.x < items) {
      if (tid == 7 * 32) {
        fence_proxy_async();
        issue_stage(it + gridDim.x);
      }
      ++staged;
    }

    // ---- 4. T = (I + A)^{-1}; T_U = T diag(beta) -------------------------
    if (warp < 4) solve_unit_lower(AT, tid);
    __syncthreads();
    {
      const int r = tid >> 2, q4 = tid & 3;  // row r, columns 16 q4 ..
      float tv[16];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const float4 v = *reinterpret_cast<const float4*>(AT + r * AP + 16 * q4 + 4 * c4);
        tv[4 * c4] = v.x; tv[4 * c4 + 1] = v.y; tv[4 * c4 + 2] = v.z; tv[4 * c4 + 3] = v.w;
      }
      // to shared memory (the W product's operand) and straight to the
      // workspace: plain stores, since a proxy fence here would wait for the
      // next item's rows still landing
      uint8_t* tu = sm + KP_TU;
      uint8_t* tug = static_cast<uint8_t*>(p.tu) + (size_t)it * WS_TU_BYTES;
#pragma unroll
      for (int h8 = 0; h8 < 2; ++h8) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int col = 16 * q4 + 8 * h8 + e;
          const float t = col < r ? tv[8 * h8 + e] : (col == r ? 1.f : 0.f);
          y[e] = t * bet[col];
        }
        uint4 w;
        w.x = pack_bf16x2(y[0], y[1]);
        w.y = pack_bf16x2(y[2], y[3]);
        w.z = pack_bf16x2(y[4], y[5]);
        w.w = pack_bf16x2(y[6], y[7]);
        *reinterpret_cast<uint4*>(tu + sw128(r, 2 * q4 + h8)) = w;
        *reinterpret_cast<uint4*>(tug + sw128(r, 2 * q4 + h8)) = w;
      }
    }
    __syncthreads();

    // ---- 5. W = T_U K_G; -W image ----------------------------------------
    {
      const int R = warp & 3, nh = warp >> 2;  // rows 16 R.., columns 64 nh..
      const int g = lane >> 2, t4 = lane & 3;
      uint32_t a[4][4];
      const int ar = 16 * R + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        ldsm_x4(base + KP_TU + sw128(ar, 2 * kk + (lane >> 4)), a[kk]);
      float acc[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
      const int br = (lane & 7) + ((lane >> 3) & 1) * 8, bc = (lane >> 4) * 8;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t b[4];
          ldsm_x4_t(base + KP_KG + (16 * kk + br) * KP_PITCH +
                        (64 * nh + 16 * np + bc) * 2,
                    b);
          mma16816(acc[2 * np], a[kk], b[0], b[1]);
          mma16816(acc[2 * np + 1], a[kk], b[2], b[3]);
        }
      }
      uint8_t* wimg = sm + KP_W + nh * TILE_BYTES;
      const int r0 = 16 * R + g, r1 = r0 + 8;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int cc = 8 * n + 2 * t4;
        *reinterpret_cast<uint32_t*>(wimg + sw128(r0, cc >> 3) + (cc & 7) * 2) =
            pack_bf16x2(-acc[n][0], -acc[n][1]);
        *reinterpret_cast<uint32_t*>(wimg + sw128(r1, cc >> 3) + (cc & 7) * 2) =
            pack_bf16x2(-acc[n][2], -acc[n][3]);
      }
    }
    __syncthreads();
    {
      // the image out with 16-byte stores (no proxy fence, as for T_U)
      const uint4* src = reinterpret_cast<const uint4*>(sm + KP_W);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.wneg) +
                                            (size_t)it * WS_W_BYTES);
#pragma unroll
      for (int i = 0; i < (int)(WS_W_BYTES / 16 / kKpThreads); ++i)
        dst[tid + i * kKpThreads] = src[tid + i * kKpThreads];
    }
  }
  if (tid == 0) {
    // never leave with a row copy still landing (an item cut short by a
    // timeout), nor with an image copy still reading
    if (staged > li) wait_ignoring_abort(sbar, li & 1);
    bulk_wait_all();
    if (*abort_flag) record_status(p.status, GDN_ERR_TIMEOUT);
  }
}

int sm_count_kp() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) ==
          cudaSuccess &&
      v > 0)
    return v;
  return 148;
}

}  // namespace

cudaError_t launch_kda_prep(const ChunkParams& p, cudaStream_t stream,
                            int* launches) {
  cudaError_t e = launch_chunk_offsets(p, stream, launches);
  if (e != cudaSuccess) return e;
  const long long bound = chunk_tc_chunks_bound(p);
  const long long items = bound * p.H;
  if (items <= 0) return cudaSuccess;
  const int grid =
      (int)std::min<long long>(items, (long long)kKpCtas * sm_count_kp());
  const long long tokens = p.cu_seqlens ? (long long)p.T : (long long)p.N * p.T;
  CUtensorMap mg, mk;
  if (!make_rows_map(&mg, p.g, true, DK, p.H, tokens, DK, C) ||
      !make_rows_map(&mk, p.k, false, DK, p.H, tokens, DK, C))
    return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(kda_prep_kernel,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)KP_SMEM);
  if (e != cudaSuccess) return e;
  const int t = timing_start(GDN_KERNEL_KDA_PREP, stream);
  kda_prep_kernel<<<grid, kKpThreads, KP_SMEM, stream>>>(
      p, mg, mk, chunk_tc_nch_dense(p), (int)bound);
  e = cudaGetLastError();
  timing_stop(t, stream, e);
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace gdn
