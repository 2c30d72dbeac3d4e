// Chunkwise Gated DeltaNet forward pass on the sm_103a tensor cores.
//
// Two kernels, in stream order (illustrated DeltaNet walk-through: UT
// transform, WY representation, chunkwise state passing and output; scalar
// gate prefixes of its GLA section). D_rj = exp(G_r - G_j) with G the
// chunk-local cumulative log gate, G' = G (decay first) or G_{r-1} (decay
// after the prediction); every gate factor lies in (0, 1] and is folded into
// an operand that is written anyway.
//
// ut_prep_kernel — everything that does not depend on the running state,
// fully parallel over (chunk, head), four CTAs per SM:
//     [K;Q] K^T on tcgen05  ->  A = strict_lower(diag(beta) K K^T (.) D')
//                               P = (Q K^T) (.) D (.) M_incl
//     T = (I + A)^{-1} (blocked substitution + m16n8k8 tf32 merges)
//     T_W = T diag(beta e^{G'}),  T_U = T diag(beta)
//     W = T_W K on tcgen05
//   and writes -W, P, T_U (bf16) and the chunk's decay vectors (fp32) for
//   the chain kernel.
//
// chunk_tc_kernel — one CTA per (sequence, head, 64 state rows) walking the
// chunks in order; the state S^T (d_k x 64) lives in fp32 registers of the
// chain warps and as bf16 in shared memory for the MMAs. Per chunk:
//   side   [0;T_U] V -> U0 starts the chunk's accumulator (rows 64-127)
//   chain  += [Q;-W] S^T -> H = Q S^T (rows 0-63), U = U0 - W S^T (64-127)
//          K^T diag(e^{G_L - G}) U -> Delta;   S^T <- gamma S^T + Delta
//          [P;.] U -> P U;   O = diag(e^G) H + P U at read-out
// The serial chain per chunk is two MMA round trips and two short register
// phases; everything else arrives by TMA.
//
// Warp roles of chunk_tc_kernel (kChainWarps + 3 warps; with 8 chain warps
// 352 threads): the chain warps hold the state rows (those with lane quarter
// 2-3 also U rows, 0-1 output rows; each takes 32 of the 64 columns), then
// the TMA producer, the P U warp and the U0 / [Q;-W] S^T / Delta warp.
// Only warps 4k and 4k + 1 reach TMEM lanes 0-63 (the output rows), so the
// U-row warps take the elementwise work of the fused output gate (each
// chunk's gate logits turned into sigmoids in shared memory while the U rows
// wait for the Delta product) to keep the output-row warps within a chunk's
// period. The MMA warp is woken by barriers: the state in shared memory for
// [Q;-W] S^T, diag(e^{G_L-G}) U for the Delta product. Operand tiles are
// bf16 with the 128-byte swizzle and arrive in a two-stage ring, each stage
// in two parts (the first two chunks' q, k, v requested before the wait for
// the preparation kernel); whole output tiles leave by TMA store. Every wait
// is bounded; a CTA that gives up records GDN_ERR_TIMEOUT, drains its MMAs,
// frees its TMEM and exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_internal.cuh"
#include "gdn_selftest.h"
#include "tc_ptx.cuh"
#include "chunk_tiles.cuh"

namespace gdn {
namespace {
using namespace tc;

// log alpha = -softplus(a) and beta = sigmoid(b) from the logits.
__device__ __forceinline__ float neg_softplus(float a) {
  return -(fmaxf(a, 0.f) + log1pf(expf(-fabsf(a))));
}
__device__ __forceinline__ float sigmoid_f(float b) {
  return 1.f / (1.f + expf(-b));
}

// Gate vectors of the chunk whose first token row (token * H + head) is
// rbase; tokens at or past len get g = 0 and beta = 0. One whole warp, lane
// l taking tokens l and l + 32. With `logits` the inputs are a and b of
// log alpha = -softplus(a), beta = sigmoid(b). Computed into registers
// (gate_lanes) and written out separately (put), so that a caller can form
// them before the buffer is free.
struct GateLanes {
  float G[2], alpha[2], egpb[2], beta[2], eg[2], dec[2], ieg[2];
  float gam, safe;
};

template <int VARIANT>
__device__ __forceinline__ GateLanes gate_lanes(const float* g,
                                                const float* beta,
                                                size_t rbase, int H, int len,
                                                bool logits, int lane) {
  const unsigned fm = 0xffffffffu;
  float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
  if (lane < len) {
    g0 = g[rbase + (size_t)lane * H];
    b0 = beta[rbase + (size_t)lane * H];
    if (logits) {
      g0 = neg_softplus(g0);
      b0 = sigmoid_f(b0);
    }
  }
  if (lane + 32 < len) {
    g1 = g[rbase + (size_t)(lane + 32) * H];
    b1 = beta[rbase + (size_t)(lane + 32) * H];
    if (logits) {
      g1 = neg_softplus(g1);
      b1 = sigmoid_f(b1);
    }
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
  const bool in_range =
      __all_sync(fm, s0 >= -87.f && s0 <= 87.f && s1 >= -87.f && s1 <= 87.f);
  GateLanes v;
  v.G[0] = s0; v.G[1] = s1;
  v.alpha[0] = expf(g0); v.alpha[1] = expf(g1);
  v.egpb[0] = expf(p0) * b0; v.egpb[1] = expf(p1) * b1;
  v.beta[0] = b0; v.beta[1] = b1;
  v.eg[0] = expf(s0); v.eg[1] = expf(s1);
  v.dec[0] = expf(Gl - s0); v.dec[1] = expf(Gl - s1);
  v.ieg[0] = expf(-s0); v.ieg[1] = expf(-s1);
  v.gam = expf(Gl);
  v.safe = in_range ? 1.f : 0.f;
  return v;
}

__device__ __forceinline__ void put_gate_lanes(const GateLanes& v, float* vec,
                                               int lane) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    vec[VEC_G + 32 * k + lane] = v.G[k];
    vec[VEC_ALPHA + 32 * k + lane] = v.alpha[k];
    vec[VEC_EGPB + 32 * k + lane] = v.egpb[k];
    vec[VEC_BETA + 32 * k + lane] = v.beta[k];
    vec[VEC_EG + 32 * k + lane] = v.eg[k];
    vec[VEC_DEC + 32 * k + lane] = v.dec[k];
    vec[VEC_IEG + 32 * k + lane] = v.ieg[k];
  }
  if (lane == 0) {
    vec[VEC_GAMMA] = v.gam;
    vec[VEC_SAFE] = v.safe;
  }
}

template <int VARIANT>
__device__ __forceinline__ void gate_vectors(const float* g, const float* beta,
                                             size_t rbase, int H, int len,
                                             float* vec, bool logits,
                                             int lane) {
  put_gate_lanes(gate_lanes<VARIANT>(g, beta, rbase, H, len, logits, lane),
                 vec, lane);
}


// ---------------------------------------------------------------------------
// ut_prep_kernel: the state-independent part of every (chunk, head).
// 160 threads: warps 0-3 compute, warp 4 loads the K and Q tiles by TMA and
// writes the gate vectors. kPrepStages stages, kPrepCtas CTAs per SM.
constexpr int kPrepThreads = 160;
constexpr int kPrepStages = 1;
constexpr int kPrepCtas = 4;
constexpr int kPrepVecs = kPrepStages + 1;  // gate-vector buffers
// Stage: K0 | Q0 | K1 | Q1 (8 KB each, 64-column blocks of d_k): [K_c;Q_c]
// is a 128-row K-major tile and K (two blocks, 16 KB apart) the N-major B
// operand of W = T_W K. Once Q's last reader is done its blocks hold output
// images on their way to the workspace: P in Q0, T_U in Q1; -W goes out of
// the solve buffer, so the stage is released right after the W product.
constexpr uint32_t PR_STAGE = 32768;
// fp32 A / T (row pitch AP); after T is read out the same bytes hold the
// 128-row bf16 tile [T_W; T_W], and after the W product the -W images.
constexpr uint32_t PR_OFF_AT = kPrepStages * PR_STAGE;
constexpr uint32_t PR_OFF_VEC = PR_OFF_AT + 64 * AP * 4;
constexpr uint32_t PR_OFF_BAR = PR_OFF_VEC + kPrepVecs * VEC_FLOATS * 4;
enum {
  PB_FULL = 0, PB_EMPTY = PB_FULL + kPrepStages,
  PB_MMA = PB_EMPTY + kPrepStages, PB_MMAW, PB_DRAIN, PB_N
};
constexpr uint32_t PR_OFF_MISC = PR_OFF_BAR + PB_N * 8;
constexpr uint32_t PR_SMEM_BYTES = PR_OFF_MISC + 16 + 1024;
constexpr uint32_t PR_TMEM_COLS = 128;
// Largest workspace (-W, P, T_U images) written with an evict-last L2 hint.
constexpr long long kKeepWsBytes = 96ll << 20;
constexpr uint32_t ID_PREP = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_PREP_W = idesc_bf16(128, 128, false, true);
static_assert(64 * AP * 4 >= 16384, "[T_W; T_W] must fit the solve buffer");
static_assert(PR_OFF_BAR % 8 == 0, "mbarrier alignment");

template <int VARIANT>
__global__ void __launch_bounds__(kPrepThreads, kPrepCtas)
    ut_prep_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmq, int nch_dense,
                   int total_chunks_bound, int keep_ws) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + PR_OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + PR_OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + PR_OFF_MISC + 4);
  float* vecs = reinterpret_cast<float*>(sm + PR_OFF_VEC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H;
  // an invalid packing (already recorded as GDN_ERR_INVALID_ARG) can count
  // more chunks than the workspace holds: never write past it
  const int total_chunks =
      p.chunk_off ? min(p.chunk_off[p.N], total_chunks_bound) : total_chunks_bound;
  const int items = total_chunks * H;
  // the chain kernel behind this one may be scheduled once every CTA of this
  // grid has passed here (so all of them hold their SMs already and none can
  // be starved by it); it takes SMs as they free up and waits for this grid
  // to complete before touching its output
  griddep_launch_dependents();

  if (tid == 0) {
    for (int st = 0; st < kPrepStages; ++st) {
      mbar_init(&bars[PB_FULL + st], 1);
      mbar_init(&bars[PB_EMPTY + st], 1);
    }
    mbar_init(&bars[PB_MMA], 1);
    mbar_init(&bars[PB_MMAW], 1);
    mbar_init(&bars[PB_DRAIN], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, PR_TMEM_COLS);
    tmem_relinquish();
    if (lane == 0) {
      prefetch_tmap(&tmk);
      prefetch_tmap(&tmq);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ================= TMA producer + gate vectors =================
    // The gate vectors of item li go to buffer li % kPrepVecs (its previous
    // user finished before the stage wait of the previous iteration) ahead of
    // the wait for the stage, so they overlap the items in flight.
    int li = 0;
    for (int it = blockIdx.x; it < items; it += gridDim.x, ++li) {
      const int c = it / H, h = it - (it / H) * H;
      int n, lc;
      locate_chunk(p, c, nch_dense, n, lc);
      long long bos, eos;
      if (!sequence_range(p, n, bos, eos)) bos = eos = 0;
      const long long t0 = bos + (long long)lc * C;
      const int len = (int)max(0ll, min((long long)C, eos - t0));
      gate_vectors<VARIANT>(p.g, p.beta, (size_t)t0 * H + h, H, len,
                            vecs + (li % kPrepVecs) * VEC_FLOATS,
                            p.prologue != 0, lane);
      __syncwarp();
      const int s = li % kPrepStages;
      if (li >= kPrepStages &&
          !mbar_wait(&bars[PB_EMPTY + s], (li / kPrepStages - 1) & 1, abort_flag))
        break;
      if (lane == 0) {
        uint64_t* full = &bars[PB_FULL + s];
        uint8_t* st = sm + s * PR_STAGE;
        mbar_arrive_expect_tx(full, PR_STAGE);
        tma_load_3d(st, &tmk, full, 0, h, (int)t0);
        tma_load_3d(st + 8192, &tmq, full, 0, h, (int)t0);
        tma_load_3d(st + 16384, &tmk, full, 64, h, (int)t0);
        tma_load_3d(st + 24576, &tmq, full, 64, h, (int)t0);
        // the CTA's next item into L2 while this one is processed
        const int nx = it + gridDim.x;
        if (nx < items) {
          const int c2 = nx / H, h2 = nx - (nx / H) * H;
          int n2, lc2;
          locate_chunk(p, c2, nch_dense, n2, lc2);
          long long b2, e2;
          if (sequence_range(p, n2, b2, e2)) {
            const int tok2 = (int)(b2 + (long long)lc2 * C);
            prefetch_l2_3d(&tmk, 0, h2, tok2);
            prefetch_l2_3d(&tmk, 64, h2, tok2);
            prefetch_l2_3d(&tmq, 0, h2, tok2);
            prefetch_l2_3d(&tmq, 64, h2, tok2);
          }
        }
      }
    }
    // never leave with a TMA copy still landing in shared memory
    if (lane == 0)
      for (int j = max(0, li - kPrepStages); j < li; ++j)
        wait_ignoring_abort(&bars[PB_FULL + j % kPrepStages],
                            (j / kPrepStages) & 1);
  } else {
    // ================= compute warps =================
    float* AT = reinterpret_cast<float*>(sm + PR_OFF_AT);
    int li = 0;
    for (int it = blockIdx.x; it < items; it += gridDim.x, ++li) {
      const int s = li % kPrepStages;
      uint8_t* st = sm + s * PR_STAGE;            // this item's stage
      const uint32_t stb = base + s * PR_STAGE;   // (shared-window address)
      bool ok = mbar_wait(&bars[PB_FULL + s], (li / kPrepStages) & 1, abort_flag);
      if (!bar_and(1, 128, ok)) break;
      float* vec = vecs + (li % kPrepVecs) * VEC_FLOATS;
      if (tid == 0) {
        // [K;Q] K^T: rows 0-63 K K^T, rows 64-127 Q K^T
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t a = sdesc(stb + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
          mma_bf16(tmem, a, a, ID_PREP, k > 0);
        }
        mma_commit(&bars[PB_MMA]);
      }
      {
        // Inverse lengths of the raw k and q rows (when the prologue is on):
        // thread t < 64 takes row t of K, t >= 64 row t - 64 of Q, both
        // 64-column blocks of the swizzled tile. They are folded into the
        // factors the rows and columns are scaled with anyway: 1/|k| into
        // beta e^{G'} (rows of A, columns of T_W), e^{-G} (columns of A and
        // P) and e^{G_L - G} (the chain's diag(e^{G_L-G}) U); 1/|q| into e^G
        // (rows of P and of the chain's output).
        const int r = tid & 63;
        float inv = 1.f;
        if (p.prologue) {
          const uint8_t* tl = st + (tid < 64 ? 0 : 8192);
          float ss = 0.f;
#pragma unroll
          for (int cb = 0; cb < 2; ++cb) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              float f[8];
              unpack_bf16x8(*reinterpret_cast<const uint4*>(tl + cb * 16384 + sw128(r, c)), f);
#pragma unroll
              for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
            }
          }
          inv = ss > 0.f ? rsqrtf(ss) : 0.f;
        }
        vec[(tid < 64 ? VEC_SK : VEC_SQ) + r] = inv;
        if (p.prologue) {
          if (tid < 64) {
            vec[VEC_EGPB + r] *= inv;
            vec[VEC_IEG + r] *= inv;
            vec[VEC_DEC + r] *= inv;
          } else {
            vec[VEC_EG + r] *= inv;
          }
        }
        named_bar(1, 128);
        // the chain kernel's decay vectors (after the fold)
        float* cv = p.cv + (size_t)it * CV_FLOATS;
        if (tid < 64) {
          cv[CV_EG + tid] = vec[VEC_EG + tid];
          cv[CV_DEC + tid] = vec[VEC_DEC + tid];
        } else if (tid < 68) {
          cv[CV_GAMMA + tid - 64] = tid == 64 ? vec[VEC_GAMMA] : 0.f;
        }
      }
      ok = mbar_wait(&bars[PB_MMA], li & 1, abort_flag);
      if (tid == 0) bulk_wait_read();  // previous -W copy out of the buffer
      if (!bar_and(1, 128, ok)) break;
      tc_fence_after();
      const size_t tile = (size_t)it;  // it = chunk * H + head
      if (warp < 2) {
        // row r of A: beta_r exp(G'_r - G_j) k_r.k_j for j < r, in two
        // 32-column halves (high half first so the fallback's running decay
        // product runs from the diagonal down)
        const int r = tid;
        const bool safe = vec[VEC_SAFE] != 0.f;
        const float er = vec[VEC_EGPB + r];
        const float br = vec[VEC_BETA + r] * vec[VEC_SK + r];
        const float* alpha = vec + VEC_ALPHA;
        const float* sk = vec + VEC_SK;
        float d = 1.f;
#pragma unroll
        for (int hf = 1; hf >= 0; --hf) {
          float x[32];
          tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * hf, x);
          tmem_ld_wait();
          if (safe) {
            const float4* w4 = reinterpret_cast<const float4*>(vec + VEC_IEG + 32 * hf);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 w = w4[c4];
              const int j = 32 * hf + 4 * c4;
              x[4 * c4] = j < r ? er * w.x * x[4 * c4] : 0.f;
              x[4 * c4 + 1] = j + 1 < r ? er * w.y * x[4 * c4 + 1] : 0.f;
              x[4 * c4 + 2] = j + 2 < r ? er * w.z * x[4 * c4 + 2] : 0.f;
              x[4 * c4 + 3] = j + 3 < r ? er * w.w * x[4 * c4 + 3] : 0.f;
            }
          } else {
            // D'_rj = prod of alpha over (j, r] (decay first) or [j, r)
#pragma unroll
            for (int e = 31; e >= 0; --e) {
              const int jj = 32 * hf + e;
              float a = 0.f;
              if (jj < r) {
                if (VARIANT == GDN_GATE_BEFORE_PREDICT) {
                  d *= alpha[jj + 1];
                  a = br * d * sk[jj] * x[e];
                } else {
                  a = br * d * sk[jj] * x[e];
                  d *= alpha[jj];
                }
              }
              x[e] = a;
            }
          }
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4)
            *reinterpret_cast<float4*>(AT + r * AP + 32 * hf + 4 * c4) =
                make_float4(x[4 * c4], x[4 * c4 + 1], x[4 * c4 + 2], x[4 * c4 + 3]);
        }
      } else {
        // row r of P: exp(G_r - G_j) q_r.k_j for j <= r (lanes 64-127), to
        // the workspace as bf16
        const int r = tid - 64;
        const bool safe = vec[VEC_SAFE] != 0.f;
        const float er = vec[VEC_EG + r];
        const float* alpha = vec + VEC_ALPHA;
        uint8_t* ptile = st + 8192;  // Q0: read by the K K^T MMA only
        float d = 1.f;
#pragma unroll
        for (int hf = 1; hf >= 0; --hf) {
          float x[32];
          tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * hf, x);
          tmem_ld_wait();
          if (safe) {
            const float4* w4 = reinterpret_cast<const float4*>(vec + VEC_IEG + 32 * hf);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 w = w4[c4];
              const int j = 32 * hf + 4 * c4;
              x[4 * c4] = j <= r ? w.x * x[4 * c4] : 0.f;
              x[4 * c4 + 1] = j + 1 <= r ? w.y * x[4 * c4 + 1] : 0.f;
              x[4 * c4 + 2] = j + 2 <= r ? w.z * x[4 * c4 + 2] : 0.f;
              x[4 * c4 + 3] = j + 3 <= r ? w.w * x[4 * c4 + 3] : 0.f;
            }
            store_half_bf16_scaled(ptile, r, hf, x, er);
          } else {
            // D_rj = prod of alpha over (j, r]
            const float* sk = vec + VEC_SK;
#pragma unroll
            for (int e = 31; e >= 0; --e) {
              const int jj = 32 * hf + e;
              float pv = 0.f;
              if (jj <= r) {
                pv = d * sk[jj] * x[e];
                d *= alpha[jj];
              }
              x[e] = pv;
            }
            store_half_bf16_scaled(ptile, r, hf, x, vec[VEC_SQ + r]);
          }
        }
      }
      fence_proxy_async();
      tc_fence_before();
      named_bar(1, 128);
      solve_unit_lower(AT, tid);
      {
        // T_W rows into the [T_W; T_W] operand tile (over the solve buffer,
        // so every thread reads its part of T first), T_U rows into Q1.
        // Thread (r, hh) handles columns 32 hh .. 32 hh + 31.
        const int r = tid & 63, hh = tid >> 6;
        float t[32];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 v = *reinterpret_cast<const float4*>(AT + r * AP + 32 * hh + 4 * c4);
          t[4 * c4] = v.x; t[4 * c4 + 1] = v.y; t[4 * c4 + 2] = v.z; t[4 * c4 + 3] = v.w;
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = 32 * hh + e;
          t[e] = col < r ? t[e] : (col == r ? 1.f : 0.f);
        }
        named_bar(1, 128);  // T fully read before the tile overwrites it
        float tw[32], tu[32];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 w4 = *reinterpret_cast<const float4*>(vec + VEC_EGPB + 32 * hh + 4 * c4);
          const float4 u4 = *reinterpret_cast<const float4*>(vec + VEC_BETA + 32 * hh + 4 * c4);
          tw[4 * c4] = t[4 * c4] * w4.x; tw[4 * c4 + 1] = t[4 * c4 + 1] * w4.y;
          tw[4 * c4 + 2] = t[4 * c4 + 2] * w4.z; tw[4 * c4 + 3] = t[4 * c4 + 3] * w4.w;
          tu[4 * c4] = t[4 * c4] * u4.x; tu[4 * c4 + 1] = t[4 * c4 + 1] * u4.y;
          tu[4 * c4 + 2] = t[4 * c4 + 2] * u4.z; tu[4 * c4 + 3] = t[4 * c4 + 3] * u4.w;
        }
        uint8_t* tile_tw = sm + PR_OFF_AT;
        store_half_bf16(tile_tw, r, hh, tw);
        store_half_bf16(tile_tw, 64 + r, hh, tw);
        store_half_bf16(st + 24576, r, hh, tu);
        fence_proxy_async();
      }
      named_bar(1, 128);
      if (tid == 0) {
        if (keep_ws) {
          const uint64_t pol = l2_policy_evict_last();
          bulk_store_hint(static_cast<uint8_t*>(p.pm) + tile * WS_P_BYTES,
                          st + 8192, TILE_BYTES, pol);
          bulk_store_hint(static_cast<uint8_t*>(p.tu) + tile * WS_TU_BYTES,
                          st + 24576, TILE_BYTES, pol);
        } else {
          bulk_store(static_cast<uint8_t*>(p.pm) + tile * WS_P_BYTES, st + 8192,
                     TILE_BYTES);
          bulk_store(static_cast<uint8_t*>(p.tu) + tile * WS_TU_BYTES,
                     st + 24576, TILE_BYTES);
        }
        bulk_commit();
        // [T_W; T_W] K: both halves of the accumulator hold W
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem, sdesc(base + PR_OFF_AT + k * 32, 16, 1024),
                   sdesc(stb + k * 2048, 16384, 1024), ID_PREP_W, k > 0);
        mma_commit(&bars[PB_MMAW]);
      }
      ok = mbar_wait(&bars[PB_MMAW], li & 1, abort_flag);
      if (!bar_and(1, 128, ok)) break;
      if (tid == 0) {
        // the W product has read K and the P / T_U copies have read Q: the
        // stage is free for the next item while -W is read out
        bulk_wait_read();
        mbar_arrive(&bars[PB_EMPTY + s]);
      }
      tc_fence_after();
      {
        // -W images into the solve buffer, whose [T_W; T_W] tile the W
        // product has read: warps 0-1 columns 0-63 (lanes 0-63), warps 2-3
        // columns 64-127 (lanes 64-127, the copy)
        const int r = tid & 63, cb = warp >> 1;
        uint8_t* wtile = sm + PR_OFF_AT + cb * TILE_BYTES;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          float x[32];
          tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 64 * cb + 32 * hf, x);
          tmem_ld_wait();
          store_half_bf16_scaled(wtile, r, hf, x, -1.f);
        }
        fence_proxy_async();
      }
      tc_fence_before();
      named_bar(1, 128);  // vec and TMEM free again; -W complete
      if (tid == 0) {
        if (keep_ws)
          bulk_store_hint(static_cast<uint8_t*>(p.wneg) + tile * WS_W_BYTES,
                          sm + PR_OFF_AT, WS_W_BYTES, l2_policy_evict_last());
        else
          bulk_store(static_cast<uint8_t*>(p.wneg) + tile * WS_W_BYTES,
                     sm + PR_OFF_AT, WS_W_BYTES);
        bulk_commit();
      }
    }
    if (tid == 0) {
      mma_commit(&bars[PB_DRAIN]);
      wait_ignoring_abort(&bars[PB_DRAIN], 0);
      bulk_wait_all();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, PR_TMEM_COLS);
  }
  if (tid == 0 && *abort_flag) record_status(p.status, GDN_ERR_TIMEOUT);
}

// Exclusive prefix of per-sequence block counts: chunk_off[n] = sum_{m<n}
// ceil(len_m / L) (L = C for chunks), chunk_off[N] = total. One CTA.
__global__ void __launch_bounds__(1024)
    chunk_offsets_kernel(const int32_t* cu_seqlens, int N, int T, int L,
                         int32_t* chunk_off, int* status) {
  __shared__ int carry;
  __shared__ int warp_sums[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < N; base += blockDim.x) {
    const int n = base + tid;
    int v = 0;
    if (n < N) {
      const int b = cu_seqlens[n], e = cu_seqlens[n + 1];
      if (b < 0 || e < b || e > T) {
        record_status(status, GDN_ERR_INVALID_ARG);
      } else {
        v = (e - b + L - 1) / L;
      }
    }
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int incl = x + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (n < N) chunk_off[n] = carry + incl - v;
    __syncthreads();
    if (tid == (int)blockDim.x - 1) carry += incl;
    __syncthreads();
  }
  if (tid == 0) chunk_off[N] = carry;
}



// ---------------------------------------------------------------------------
// chunk_tc_kernel: the serial chain (see the top of this file).
// Chain warps: lane quarter warp & 3, column group warp >> 2 of the CTA's 64
// state columns (kCW columns each); then the producer, the P U warp and the
// U0 / [Q;-W] S^T warp.
constexpr int kChainWarps = 8;
constexpr int kChainThreads = 32 * kChainWarps;
constexpr int kCW = 64 / (kChainWarps / 4);
constexpr int kWarpProducer = kChainWarps, kWarpPU = kChainWarps + 1,
              kWarpMMA = kChainWarps + 2;
constexpr int kThreads = 32 * (kChainWarps + 3);
// Stage: per 64-column block of d_k, three 64-row groups K | Q | -W: [Q;-W]
// is a 128-row K-major tile and K alone the M-major operand of the Delta
// product. Then V, a zero block and T_U ([0;T_U] is a 128-row tile), P
// ([P;...] feeds only discarded rows beyond 64) and the decay vectors.
constexpr uint32_t ST_K = 0, ST_Q = 8192, ST_W = 16384, ST_CB = 24576;
constexpr uint32_t ST_V = 49152, ST_Z = 57344, ST_TU = 65536, ST_P = 73728,
                   ST_CV = 81920;
constexpr uint32_t ST_G = 82944;  // output gate tile (fused epilogue only)
constexpr uint32_t STAGE_BYTES = 91136;
// A stage arrives in two parts: what U0 and the chain warps' scalars need
// (V, T_U, decay vectors) first, then Q, -W, K and P.
constexpr uint32_t STAGE_A_BYTES = 16384 + CV_BYTES;  // V, T_U, cv
constexpr uint32_t STAGE_B_BYTES = 57344;             // Q, -W, K, P

constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_S = 2 * STAGE_BYTES;   // S^T, bf16 (N-major B)
constexpr uint32_t OFF_U = OFF_S + 16384;     // U, bf16
constexpr uint32_t OFF_UD = OFF_U + 8192;     // diag(e^{G_L-G}) U, bf16
constexpr uint32_t OFF_O = OFF_UD + 8192;     // output tile on its way out
// fused epilogue: norm weights of the CTA's 64 columns, per-row partial sums
// of squares of the column groups, and the partner CTA's row sums (two
// chunk-parity slots written by the partner)
constexpr uint32_t OFF_EPW = OFF_O + 8192;
constexpr uint32_t OFF_EPRED = OFF_EPW + 64 * 4;
constexpr uint32_t OFF_EPX = OFF_EPRED + (kChainWarps / 4) * 64 * 4;
constexpr uint32_t OFF_BAR = OFF_EPX + 2 * 64 * 4;
static_assert(ST_CV + CV_BYTES <= STAGE_BYTES && STAGE_BYTES % 1024 == 0,
              "stage layout");

enum {
  B_FULLA0, B_FULLA1, B_FULLB0, B_FULLB1, B_EMPTY0, B_EMPTY1, B_SREADY,
  B_D1FULL0, B_D1FULL1,
  B_UREADY, B_D2FULL, B_D3FULL0, B_D3FULL1, B_D3FREE0, B_D3FREE1, B_DRAIN_C,
  B_DRAIN_S, B_XS0, B_XS1, B_UDREADY, B_GREADY0, B_GREADY1, NBARS
};
constexpr uint32_t OFF_MISC = OFF_BAR + NBARS * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// TMEM columns (fp32 accumulators, 128 lanes each).
constexpr uint32_t TM_D1 = 0, TM_D3 = 128, TM_D2 = 256;  // D1, D3 two buffers
constexpr uint32_t TMEM_COLS = 512;

constexpr uint32_t ID_KMN = idesc_bf16(128, 64, false, true);
constexpr uint32_t ID_MNMN = idesc_bf16(128, 64, true, true);

__device__ __forceinline__ uint32_t bar_count(int b) {
  switch (b) {
    // the MMA warp's commit after the Delta product and the P U warp's
    // commit, one per chain warp (each chain warp arrives once, after its
    // lanes' reads)
    case B_EMPTY0: case B_EMPTY1: return 2 + kChainThreads / 32;
    case B_SREADY: return kChainThreads / 32;
    // the U-row warps (UREADY, UDREADY, GREADY) or the output-row warps
    case B_UREADY: case B_D3FREE0: case B_D3FREE1: case B_UDREADY:
    case B_GREADY0: case B_GREADY1:
      return kChainThreads / 64;
    // the partner's 64 row sums, counted in bytes (armed once per use)
    default: return 1;
  }
}

// How many chunks ahead of the one being loaded the chain kernels'
// producers prefetch into L2. Chain kernel time per call with d_k = d_v =
// 128 for 4 x 16 sequence-heads of 2,048 tokens / 16 heads of 65,536 tokens
// (split) / 32 packed sequences of 256-8,192 tokens: 1 ahead 0.0499 / 0.482
// / 0.562 ms, 2 ahead 0.0505 / 0.494 / 0.568, 4 ahead 0.0520 / 0.543 /
// 0.666 (lines held longer in L2 evict ones still to be read), none 0.0549
// / 0.488 / 0.571.
constexpr int kChainPrefetch = 1;

// EPI: the fused sublayer's epilogue (RMS normalisation over d_v, output
// gate) compiled in; the plain forward pass is instantiated without it.
template <int VARIANT, bool EPI>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_tc_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap tmq,
                    const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv,
                    const __grid_constant__ CUtensorMap tmo,
                    const __grid_constant__ CUtensorMap tmg, int nch_dense,
                    int tiles) {
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
  // d_k = 64 runs on the d_k = 128 layout: the second 64-column block of
  // K and Q loads as zeros (its tensor-map box lies outside the tensor), so
  // the state's rows d_k..127 stay zero; only rows < d_k are read and
  // written
  const int dkr = p.dk;
  if (!value_rows && !(split_tail && row0 < dv + dkr)) return;
  const bool scale_rows = !value_rows;
  const bool emit = (p.mode == kModeOutput) || part == 0;
  // fused epilogue on this CTA's outputs; for the RMS normalisation with
  // d_v = 128 the two CTAs of a (sequence, head, part) form a cluster and
  // exchange the per-row sums of squares of their halves of each output row
  const bool epi = EPI && p.epilogue && emit;
  const bool clustered = EPI && p.epilogue && p.norm_w && dv == 128;
  const bool has_gate = epi && p.gate_z != nullptr;
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
  if (tid < kChainThreads) {
    // zero blocks of both stages; V tiles too for rows of the scaling matrix
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int i = tid; i < 1024; i += kChainThreads) {
      const uint32_t st = (i >> 9) * STAGE_BYTES;
      *reinterpret_cast<uint4*>(sm + st + ST_Z + (i & 511) * 16) = z;
      if (scale_rows) *reinterpret_cast<uint4*>(sm + st + ST_V + (i & 511) * 16) = z;
    }
  }
  if (warp == kWarpPU) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == kWarpProducer && lane == 0) {
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
    prefetch_tmap(&tmo);
    if (has_gate) prefetch_tmap(&tmg);
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto stage = [&](int i) { return base + OFF_STAGE + (i & 1) * STAGE_BYTES; };
  // The inputs of the first two chunks (q, k, v and the output gate, which
  // the preceding kernel does not write) are requested before waiting for
  // it: their stage barriers expect these bytes without an arrival, and the
  // workspace part of the stage arrives after the wait.
  const int npre = min(nloc, 2);
  if (warp == kWarpProducer && lane == 0) {
    for (int i = 0; i < npre; ++i) {
      const int tok = (int)(bos + (long long)(c_begin + i) * C);
      uint8_t* st = sm + OFF_STAGE + (i & 1) * STAGE_BYTES;
      uint64_t* fa = &bars[B_FULLA0 + (i & 1)];
      uint64_t* fb = &bars[B_FULLB0 + (i & 1)];
      if (!scale_rows) {
        mbar_expect_tx(fa, 8192u);
        tma_load_3d(st + ST_V, &tmv, fa, row0, h, tok);
      }
      mbar_expect_tx(fb, 32768u + (has_gate ? 8192u : 0u));
      if (has_gate) tma_load_3d(st + ST_G, &tmg, fb, row0, h, tok);
      tma_load_3d(st + ST_Q, &tmq, fb, 0, h, tok);
      tma_load_3d(st + ST_Q + ST_CB, &tmq, fb, 64, h, tok);
      tma_load_3d(st + ST_K, &tmk, fb, 0, h, tok);
      tma_load_3d(st + ST_K + ST_CB, &tmk, fb, 64, h, tok);
    }
  }
  // set-up above overlaps the tail of the preceding kernel; nothing it
  // writes (workspace, chunk offsets, split states, outputs) is touched
  // before this point
  griddep_wait();
  const int cbase = nloc > 0 ? chunk_base(p, n, nch_dense) + c_begin : 0;
  if (epi && tid < 64) {
    reinterpret_cast<float*>(sm + OFF_EPW)[tid] =
        p.norm_w ? p.norm_w[row0 + tid] : 1.f;
  }
  // slots of the first two chunks armed for the partner's 64 row sums, and
  // the partner's barriers initialised, before anything is sent
  if (clustered && tid == 0) {
    mbar_arrive_expect_tx(&bars[B_XS0], 64 * 4);
    mbar_arrive_expect_tx(&bars[B_XS1], 64 * 4);
  }
  if (clustered) cluster_sync();

  if (warp == kWarpProducer) {
    // ================= TMA producer =================
    // K, Q, V by tensor map; -W, P, T_U and the decay vectors are images in
    // the workspace (plain bulk copies; the tile index is clamped because
    // those copies have no bounds check and an invalid packing, already
    // recorded, could otherwise send them past the workspace). Chunk
    // i + kChainPrefetch is prefetched into L2 when chunk i is loaded.
    if (lane == 0) {
      const uint8_t* wimg = static_cast<const uint8_t*>(p.wneg);
      const uint8_t* pimg = static_cast<const uint8_t*>(p.pm);
      const uint8_t* uimg = static_cast<const uint8_t*>(p.tu);
      auto prefetch = [&](int i) {
        const int tok = (int)(bos + (long long)(c_begin + i) * C);
        const size_t tz = (size_t)min((cbase + i) * H + h, tiles - 1);
        prefetch_l2_3d(&tmk, 0, h, tok);
        prefetch_l2_3d(&tmk, 64, h, tok);
        prefetch_l2_3d(&tmq, 0, h, tok);
        prefetch_l2_3d(&tmq, 64, h, tok);
        if (!scale_rows) prefetch_l2_3d(&tmv, row0, h, tok);
        prefetch_l2(wimg + tz * WS_W_BYTES, WS_W_BYTES);
        prefetch_l2(pimg + tz * WS_P_BYTES, WS_P_BYTES);
        prefetch_l2(uimg + tz * WS_TU_BYTES, WS_TU_BYTES);
        prefetch_l2(p.cv + tz * CV_FLOATS, CV_BYTES);
      };
      for (int i = 0; i < min(nloc, kChainPrefetch); ++i) prefetch(i);
      int issued = 0;
      for (int i = 0; i < nloc; ++i) {
        const int s = i & 1;
        if (i >= 2 && !mbar_wait(&bars[B_EMPTY0 + s], ((i >> 1) - 1) & 1,
                                 abort_flag))
          break;
        const int tok = (int)(bos + (long long)(c_begin + i) * C);
        const size_t tz = (size_t)min((cbase + i) * H + h, tiles - 1);
        uint8_t* st = sm + OFF_STAGE + s * STAGE_BYTES;
        uint64_t* fa = &bars[B_FULLA0 + s];
        uint64_t* fb = &bars[B_FULLB0 + s];
        // the input part's bytes are expected first (before the wait for
        // the first two chunks), then the workspace part's with the arrival
        const bool pre = i < npre;
        if (!pre && !scale_rows) mbar_expect_tx(fa, 8192u);
        mbar_arrive_expect_tx(fa, STAGE_A_BYTES - 8192u);  // T_U, decay vectors
        if (!pre && !scale_rows) tma_load_3d(st + ST_V, &tmv, fa, row0, h, tok);
        bulk_load(st + ST_TU, uimg + tz * WS_TU_BYTES, TILE_BYTES, fa);
        bulk_load(st + ST_CV, p.cv + tz * CV_FLOATS, CV_BYTES, fa);
        if (!pre) mbar_expect_tx(fb, 32768u + (has_gate ? 8192u : 0u));
        mbar_arrive_expect_tx(fb, STAGE_B_BYTES - 32768u);  // -W, P
        if (!pre) {
          if (has_gate) tma_load_3d(st + ST_G, &tmg, fb, row0, h, tok);
          tma_load_3d(st + ST_Q, &tmq, fb, 0, h, tok);
          tma_load_3d(st + ST_Q + ST_CB, &tmq, fb, 64, h, tok);
          tma_load_3d(st + ST_K, &tmk, fb, 0, h, tok);
          tma_load_3d(st + ST_K + ST_CB, &tmk, fb, 64, h, tok);
        }
        bulk_load(st + ST_W, wimg + tz * WS_W_BYTES, TILE_BYTES, fb);
        bulk_load(st + ST_W + ST_CB, wimg + tz * WS_W_BYTES + TILE_BYTES,
                  TILE_BYTES, fb);
        bulk_load(st + ST_P, pimg + tz * WS_P_BYTES, TILE_BYTES, fb);
        if (i + kChainPrefetch < nloc) prefetch(i + kChainPrefetch);
        issued = i + 1;
      }
      // never leave with a TMA copy still landing in shared memory
      for (int i = max(0, issued - 2); i < issued; ++i) {
        wait_ignoring_abort(&bars[B_FULLA0 + (i & 1)], (i >> 1) & 1);
        wait_ignoring_abort(&bars[B_FULLB0 + (i & 1)], (i >> 1) & 1);
      }
    }
  } else if (warp == kWarpMMA) {
    // ================= U0 and [Q;-W] S^T =================
    if (lane == 0 && nloc > 0) {
      // All from one thread so that they execute in issue order: U0 =
      // [0;T_U] V starts a chunk's accumulator, [Q;-W] S^T is added once
      // the state is in shared memory and the Delta product K^T diag(e^{G_L-
      // G}) U goes in once the U rows have written its operand. The next
      // chunk's U0 goes in right behind this chunk's [Q;-W] S^T if its
      // operands have landed (it then runs while U is read out), else behind
      // the Delta product. The accumulator of chunk i + 1 was last read (H
      // and U of chunk i - 1) before the chain warps signalled the state of
      // chunk i, which this thread has waited for. Barriers on the chain are
      // polled rather than waited with suspension.
      auto issue_u0 = [&](int j) {
        const int s = j & 1;
        if (!mbar_wait(&bars[B_FULLA0 + s], (j >> 1) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t st = stage(j);
        mma_bf16_run<4>(tmem + TM_D1 + 64 * s, sdesc(st + ST_Z, 16, 1024), 32,
                        sdesc(st + ST_V, 8192, 1024), 2048, ID_KMN, false);
        return true;
      };
      bool ok = issue_u0(0);
      for (int i = 0; ok && i < nloc; ++i) {
        const int b = i & 1;
        // the stage (landed long before) first, then the state barrier
        if (!mbar_wait(&bars[B_FULLB0 + b], (i >> 1) & 1, abort_flag) ||
            !mbar_spin(&bars[B_SREADY], i & 1, abort_flag))
          break;
        tc_fence_after();
        const uint32_t st = stage(i);
        const uint64_t sb = sdesc(base + OFF_S, 8192, 1024);
        mma_bf16_run<4>(tmem + TM_D1 + 64 * b, sdesc(st + ST_Q, 16, 1024), 32, sb,
                        2048, ID_KMN, true);
        mma_bf16_run<4>(tmem + TM_D1 + 64 * b, sdesc(st + ST_Q + ST_CB, 16, 1024),
                        32, sb + (8192 >> 4), 2048, ID_KMN, true);
        mma_commit(&bars[B_D1FULL0 + b]);
        const bool u0_now =
            i + 1 < nloc &&
            mbar_test(&bars[B_FULLA0 + (b ^ 1)], ((i + 1) >> 1) & 1);
        if (u0_now && !issue_u0(i + 1)) break;
        if (!mbar_spin(&bars[B_UDREADY], i & 1, abort_flag)) break;
        tc_fence_after();
        mma_bf16_run<4>(tmem + TM_D2, sdesc(st + ST_K, ST_CB, 1024), 2048,
                        sdesc(base + OFF_UD, 8192, 1024), 2048, ID_MNMN, false);
        mma_commit(&bars[B_D2FULL]);
        mma_commit(&bars[B_EMPTY0 + b]);
        if (i + 1 < nloc && !u0_now) ok = issue_u0(i + 1);
      }
      mma_commit(&bars[B_DRAIN_C]);
      wait_ignoring_abort(&bars[B_DRAIN_C], 0);
    }
  } else if (warp == kWarpPU) {
    // ================= P U, off the chain =================
    if (lane == 0 && nloc > 0) {
      // P U of chunk j goes in once the chunk's Delta product has
      // completed, so that the two never share the tensor pipe (the Delta
      // product is on the chain). No phase of D2FULL can pass unseen: the
      // Delta product of chunk j + 1 waits for the U rows of chunk j + 1,
      // and they wait for this P U first.
      for (int j = 0; j < nloc; ++j) {
        const int b = j & 1;
        if (!mbar_wait(&bars[B_UREADY], j & 1, abort_flag) ||
            !mbar_wait(&bars[B_D2FULL], j & 1, abort_flag) ||
            !mbar_wait(&bars[B_FULLB0 + b], (j >> 1) & 1, abort_flag))
          break;
        // P U of chunk j - 2 has been read out of this accumulator
        if (j >= 2 &&
            !mbar_wait(&bars[B_D3FREE0 + b], ((j >> 1) - 1) & 1, abort_flag))
          break;
        tc_fence_after();
        const uint32_t st = stage(j);
        mma_bf16_run<4>(tmem + TM_D3 + 64 * b, sdesc(st + ST_P, 16, 1024), 32,
                        sdesc(base + OFF_U, 8192, 1024), 2048, ID_KMN, false);
        mma_commit(&bars[B_D3FULL0 + b]);
        mma_commit(&bars[B_EMPTY0 + b]);
      }
      mma_commit(&bars[B_DRAIN_S]);
      wait_ignoring_abort(&bars[B_DRAIN_S], 0);
    }
  } else {
    // ================= chain warps =================
    // lane quarter qw = warp & 3 (TMEM lanes 32 qw ..), column group cg:
    // state rows ct = 32 qw + lane (d_k index), columns cols .. cols + kCW - 1;
    // qw >= 2 also U rows ct - 64, qw < 2 output rows ct.
    const int qw = warp & 3, cg = warp >> 2;
    const int ct = 32 * qw + lane;
    const uint32_t lanes = (uint32_t)(32 * qw) << 16;
    const uint32_t cols = kCW * cg;
    const int chunk0 = cols / 8;  // first 16-byte chunk of the columns
    const bool u_rows = qw >= 2;
    uint8_t* s_tile = sm + OFF_S;
    float S[kCW];
    if (scale_rows) {
      const int a0 = row0 - dv + (int)cols;
#pragma unroll
      for (int c = 0; c < kCW; ++c) S[c] = (ct == a0 + c) ? 1.f : 0.f;
    } else if (split_tail) {
#pragma unroll
      for (int c = 0; c < kCW; ++c) S[c] = 0.f;
    } else if (ct >= dkr) {
#pragma unroll
      for (int c = 0; c < kCW; ++c) S[c] = 0.f;
    } else if (part > 0) {
      const float* src =
          p.ws_start + ((nh * p.parts + part) * dv + row0 + cols) * dkr + ct;
#pragma unroll
      for (int c = 0; c < kCW; ++c) S[c] = src[(size_t)c * dkr];
    } else if (p.h0) {
      const float4* src = reinterpret_cast<const float4*>(
          p.h0 + (nh * dkr + ct) * dv + row0 + cols);
#pragma unroll
      for (int c = 0; c < kCW / 4; ++c) {
        const float4 v4 = src[c];
        S[4 * c] = v4.x; S[4 * c + 1] = v4.y; S[4 * c + 2] = v4.z; S[4 * c + 3] = v4.w;
      }
    } else {
#pragma unroll
      for (int c = 0; c < kCW; ++c) S[c] = 0.f;
    }
    store_cols_bf16<kCW>(s_tile, ct, chunk0, S);
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B_SREADY]);
    // Output gate: a U-row thread turns the gate logits of chunk j (row
    // ct - 64 of its stage tile, the thread's kCW columns, the same slice its
    // output-row twin reads) into sigmoid(z) in place and its warp arrives on
    // GREADY of the stage. It does so in chunk j itself, between storing U
    // and the state update, when the stage has landed (the chunk's MMAs have
    // read it): waiting for a later stage there would hold up the U rows.
    // The tile of chunk j + 2 reuses the stage only after the output rows
    // have read chunk j's and released the stage, so one barrier per stage
    // sees its phases in order.
    auto gate_to_sigmoid = [&](int j, bool okj) {
      const int sj = j & 1;
      okj = okj && mbar_wait(&bars[B_FULLB0 + sj], (j >> 1) & 1, abort_flag);
      if (okj) {
        uint8_t* gt = sm + OFF_STAGE + sj * STAGE_BYTES + ST_G;
#pragma unroll
        for (int c = 0; c < kCW / 8; ++c) {
          uint4* q = reinterpret_cast<uint4*>(gt + sw128(ct - 64, chunk0 + c));
          uint4 w = *q;
          w.x = sigmoid2_bf16(w.x);
          w.y = sigmoid2_bf16(w.y);
          w.z = sigmoid2_bf16(w.z);
          w.w = sigmoid2_bf16(w.w);
          *q = w;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_GREADY0 + sj]);
    };
    // [Q;-W] S^T accumulated onto U0: H = Q S^T (rows 0-63), U (64-127)
    // Fused epilogue on one chunk's output rows (o: this thread's kCW
    // columns of row r; gzv: sigmoid of the gate logits, bf16): o <- o /
    // sqrt(mean(o^2) + eps) * w, then * sigmoid(gate). Returns false, the
    // same on every output thread, when a wait for the partner CTA gave up.
    const float* ep_w = reinterpret_cast<const float*>(sm + OFF_EPW);
    float* ep_red = reinterpret_cast<float*>(sm + OFF_EPRED);
    float* ep_x = reinterpret_cast<float*>(sm + OFF_EPX);
    const uint32_t partner = clustered ? (cluster_ctarank() ^ 1u) : 0u;
    auto epilogue_rows = [&](float (&o)[kCW], const uint4 (&gzv)[kCW / 8],
                             int r, int cgi, int i, int b) {
      bool okp = true;
      if (p.norm_w) {
        float ss = 0.f;
#pragma unroll
        for (int c = 0; c < kCW; ++c) ss = fmaf(o[c], o[c], ss);
        ep_red[cgi * 64 + r] = ss;
        named_bar(4, kChainThreads / 2);
        float tot = 0.f;
#pragma unroll
        for (int g = 0; g < kChainWarps / 4; ++g) tot += ep_red[g * 64 + r];
        if (clustered) {
          // Send this half-row sum to the partner (its slot b counts the
          // bytes), then take the partner's from ours. Slot b is not
          // rewritten before it is read here: the partner sends chunk i + 2
          // only after it has received this CTA's chunk i + 1, sent after
          // this read.
          if (cgi == 0)
            st_async_f32(map_to_cta(ep_x + b * 64 + r, partner), tot,
                         map_to_cta(&bars[B_XS0 + b], partner));
          okp = mbar_wait_cluster(&bars[B_XS0 + b], (i >> 1) & 1, abort_flag);
          if (okp) tot += ep_x[b * 64 + r];
          okp = bar_and(4, kChainThreads / 2, okp);  // every row read its slot
          // arm slot b for chunk i + 2
          if (okp && tid == 0 && i + 2 < nloc)
            mbar_arrive_expect_tx(&bars[B_XS0 + b], 64 * 4);
        }
        const float sc = rsqrtf(tot * (1.f / (float)dv) + p.eps);
#pragma unroll
        for (int c = 0; c < kCW; ++c) o[c] *= sc * ep_w[cols + c];
      }
      if (has_gate) {
#pragma unroll
        for (int c8 = 0; c8 < kCW / 8; ++c8) {
          float f[8];
          unpack_bf16x8(gzv[c8], f);
#pragma unroll
          for (int e = 0; e < 8; ++e) o[8 * c8 + e] *= f[e];
        }
      }
      return okp;
    };
    // The loop has no early exit: a failed wait only clears `ok` (made
    // warp-uniform before every warp-collective TMEM read), so every warp
    // passes every named barrier of every chunk and no group can be left
    // waiting at one; the work of a failed chunk is skipped.
    bool ok = true;
    for (int i = 0; i < nloc; ++i) {
      const int b = i & 1;
      const long long t0 = bos + (long long)(c_begin + i) * C;
      const int len = (int)min((long long)C, eos - t0);
      // this chunk's scalars; the stage is recycled only after every chain
      // warp has said it is done with them (and the chunk's MMAs completed)
      ok = ok && mbar_wait(&bars[B_FULLA0 + b], (i >> 1) & 1, abort_flag);
      const float* cv =
          reinterpret_cast<const float*>(sm + OFF_STAGE + b * STAGE_BYTES + ST_CV);
      const float gam = cv[CV_GAMMA];
      const float rowf = cv[(u_rows ? CV_DEC : CV_EG) + (ct & 63)];
      // with an output gate the output rows read its logits at read-out and
      // release the stage only then (nothing is held in registers across
      // the chunk)
      __syncwarp();
      if (lane == 0 && !(has_gate && !u_rows)) mbar_arrive(&bars[B_EMPTY0 + b]);
      float hq[kCW];  // H = Q S^T of this chunk (output rows)
      if (!u_rows) {
        // read H as soon as it is complete: the accumulator is reused by the
        // U0 product of the chunk after next, issued after this chunk's state
        // barrier
        ok = __all_sync(0xffffffffu,
                        ok && mbar_wait(&bars[B_D1FULL0 + b], (i >> 1) & 1,
                                        abort_flag));
        if (ok) {
          tc_fence_after();
          tmem_ldn<kCW>(tmem + TM_D1 + 64 * b + lanes + cols, hq);
          tmem_ld_wait();
          tc_fence_before();
        }
      }
      if (u_rows) {
        // U = U0 - W S^T (rows 64-127 of the accumulator)
        const int r = ct - 64;
        // the U tile is free once the previous chunk's P U has completed
        // (long before U itself: waited first, off the chain)
        bool ok1 = ok && (i == 0 || mbar_wait(&bars[B_D3FULL0 + (b ^ 1)],
                                              ((i - 1) >> 1) & 1, abort_flag));
        ok1 = ok1 && mbar_wait(&bars[B_D1FULL0 + b], (i >> 1) & 1, abort_flag);
        ok1 = __all_sync(0xffffffffu, ok1);
        float u[kCW];
        if (ok1) {
          tc_fence_after();
          float ud[kCW];
          tmem_ldn<kCW>(tmem + TM_D1 + 64 * b + lanes + cols, u);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < kCW; ++c) ud[c] = u[c] * rowf;
          store_cols_bf16<kCW>(sm + OFF_UD, r, chunk0, ud);
          fence_proxy_async();
        }
        // diag(e^{G_L-G}) U complete in this warp: the MMA warp issues the
        // Delta product once all U-row warps have arrived
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_UDREADY]);
        if (ok1) {
          // U itself only feeds P U, off the chain
          store_cols_bf16<kCW>(sm + OFF_U, r, chunk0, u);
          fence_proxy_async();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[B_UREADY]);
        }
        if (has_gate) gate_to_sigmoid(i, ok1);
        ok = ok1;
      }
      const bool ok3 = __all_sync(
          0xffffffffu, ok && mbar_wait(&bars[B_D2FULL], i & 1, abort_flag));
      ok = ok3;
      if (ok3) {
        tc_fence_after();
        float dl[kCW];
        tmem_ldn<kCW>(tmem + TM_D2 + lanes + cols, dl);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < kCW; ++c) S[c] = fmaf(gam, S[c], dl[c]);
        store_cols_bf16<kCW>(s_tile, ct, chunk0, S);
        fence_proxy_async();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_SREADY]);
      if (!u_rows) {
        // O = e^{G_r} H + P U, through a shared-memory tile and a TMA store
        // for a whole chunk, direct stores for a partial one
        const int r = ct;
        uint4 gz[kCW / 8];  // sigmoid of the output row's gate logits
        if (has_gate) {
          ok = ok && mbar_wait(&bars[B_GREADY0 + b], (i >> 1) & 1, abort_flag);
          const uint8_t* gt = sm + OFF_STAGE + b * STAGE_BYTES + ST_G;
#pragma unroll
          for (int c = 0; c < kCW / 8; ++c)
            gz[c] = ok ? *reinterpret_cast<const uint4*>(gt + sw128(ct, chunk0 + c))
                       : make_uint4(0, 0, 0, 0);
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[B_EMPTY0 + b]);
        }
        bool ok4 = ok && mbar_wait(&bars[B_D3FULL0 + b], (i >> 1) & 1, abort_flag);
        if (tid == 0) bulk_wait_read();  // previous output tile read out
        ok4 = bar_and(4, kChainThreads / 2, ok4);
        if (ok4) {
          tc_fence_after();
          float o[kCW];
          tmem_ldn<kCW>(tmem + TM_D3 + 64 * b + lanes + cols, o);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < kCW; ++c) o[c] = fmaf(rowf, hq[c], o[c]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[B_D3FREE0 + b]);
          if (epi) ok4 = epilogue_rows(o, gz, r, cg, i, b);
          if (emit && len == C) {
            store_cols_bf16<kCW>(sm + OFF_O, r, chunk0, o);
            fence_proxy_async();
          } else if (emit && r < len) {
            uint4* dst = reinterpret_cast<uint4*>(
                static_cast<__nv_bfloat16*>(p.out) +
                ((size_t)(t0 + r) * H + h) * dv + row0 + cols);
#pragma unroll
            for (int c = 0; c < kCW / 8; ++c) {
              uint4 wq;
              wq.x = pack_bf16x2(o[8 * c + 0], o[8 * c + 1]);
              wq.y = pack_bf16x2(o[8 * c + 2], o[8 * c + 3]);
              wq.z = pack_bf16x2(o[8 * c + 4], o[8 * c + 5]);
              wq.w = pack_bf16x2(o[8 * c + 6], o[8 * c + 7]);
              dst[c] = wq;
            }
          }
        }
        if (emit && len == C) {
          named_bar(4, kChainThreads / 2);
          if (tid == 0 && ok4) {
            tma_store_3d(&tmo, sm + OFF_O, row0, h, (int)t0);
            bulk_commit();
          }
        }
        ok = ok && ok4;
      }
    }
    ok = bar_and(2, kChainThreads, ok);
    if (tid == 0) bulk_wait_all();
    if (ok && !*abort_flag && ct < dkr) {
      if (p.mode == kModeSplit) {
        if (part == 0) {
          if (p.parts > 1) {
            float* dst =
                p.ws_start + ((nh * p.parts + 1) * dv + row0 + cols) * dkr + ct;
#pragma unroll
            for (int c = 0; c < kCW; ++c) dst[(size_t)c * dkr] = S[c];
          }
        } else {
          float* dst = p.ws_end +
                       ((nh * p.parts + part) * (dv + dkr) + row0 + cols) * dkr + ct;
#pragma unroll
          for (int c = 0; c < kCW; ++c) dst[(size_t)c * dkr] = S[c];
        }
      } else if (p.hT && part == p.parts - 1) {
        float4* dst = reinterpret_cast<float4*>(p.hT + (nh * dkr + ct) * dv + row0 + cols);
#pragma unroll
        for (int c = 0; c < kCW / 4; ++c)
          dst[c] = make_float4(S[4 * c], S[4 * c + 1], S[4 * c + 2], S[4 * c + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // no CTA leaves while its partner may still write into its shared memory
  if (clustered) cluster_sync();
  if (warp == kWarpPU) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
  if (tid == 0 && *abort_flag) record_status(p.status, GDN_ERR_TIMEOUT);
}


// ---------------------------------------------------------------------------
// chain_tx_kernel: the serial chain with the state rows in TMEM lanes, one
// CTA per (sequence, head, part) and 128 state rows (the d_v value rows,
// padded with zero rows when d_v = 64; in a split pass a second CTA takes
// the 128 rows of the scaling matrix). With S (rows x d_k) and U^T (rows x tokens) in TMEM lanes both
// are A operands straight from TMEM, so the chain has no shared-memory
// round trip:
//   side   V^T T_U^T -> U0^T starts the chunk's accumulator (cols 0-63; the
//          output warps zeroed cols 64-127 when they read the accumulator
//          out)
//   chain  += S [-W;Q]^T -> U^T = U0^T - S W^T (cols 0-63),
//                           H^T = S Q^T (cols 64-127)
//          U^T -> bf16 pairs in TMEM;  U^T K_d -> Delta^T;
//          S <- gamma S + Delta^T -> bf16 pairs in TMEM
//   side   U^T P^T -> cols 0-63 (U^T has been converted)
//   out    O^T = H^T diag(e^G) + U^T P^T
// with K_d = diag(e^{G_L-G}) K scaled in place in shared memory by the chain
// warps while the [-W;Q] product runs.
//
// Warps: 0-7 chain (lane quarter warp & 3, d_k half warp >> 2: 64 fp32 state
// columns each), 8-11 output (one row of O^T per thread), 12 TMA producer,
// 13 issuer of the chain's products ([-W;Q_g], Delta^T), 14 issuer of the
// side products (U0^T, P), which it slots into the tensor pipe's idle spells
// of the chain (the conversion of U^T, the state update).
constexpr int kTxChainThreads = 256;
constexpr int kTxOutThreads = 128;
constexpr int kTxWarpProducer = 12, kTxWarpMMA = 13, kTxWarpSide = 14;
constexpr int kTxThreads = 15 * 32;
constexpr int TXR = 128;  // state rows per CTA
// Stage: per 64-column block of d_k a 128-row K-major tile [-W; Q]; K
// (N-major B of the Delta^T product; two 64-column blocks); V (M-major A of
// U0^T; two 64-column blocks); T_U (K-major B); P; the decay vectors.
constexpr uint32_t TX_W = 0, TX_Q = 8192, TX_WQ_CB = 16384;
constexpr uint32_t TX_K = 32768, TX_V = 49152, TX_TU = 65536, TX_P = 73728,
                   TX_CV = 81920;
constexpr uint32_t TX_STAGE = 82944;
// A stage arrives and is released in three groups, each as soon as its last
// reader is done: V, T_U (U0^T); -W, Q ([-W;Q] product); K, P and the decay
// vectors (Delta^T and P products, chain and output warps).
constexpr uint32_t TX_A_BYTES = 16384 + TILE_BYTES;             // V, T_U
constexpr uint32_t TX_B_BYTES = 2 * 16384;                      // -W, Q
constexpr uint32_t TX_C_BYTES = 16384 + TILE_BYTES + CV_BYTES;  // K, P, cv
// After the two stages: two output tiles (64 tokens x 128 values, two
// 64-column blocks each; the fused gate is loaded into them), the output
// warps' partial sums of squares and per-token scales.
constexpr uint32_t TXO_OUT = 2 * TX_STAGE;
constexpr uint32_t TXO_RED = TXO_OUT + 2 * 16384;
constexpr uint32_t TXO_RS = TXO_RED + 4 * 64 * 4;
// KDA: each chain warp's 64 values of gamma (per key channel), copied out
// of the stage before it is released
constexpr uint32_t TXO_GAM = TXO_RS + 64 * 4;
constexpr uint32_t TXO_BAR = TXO_GAM + 8 * 64 * 4;
enum {
  TB_FULLA0, TB_FULLA1, TB_FULLB0, TB_FULLB1, TB_FULLC0, TB_FULLC1,
  TB_EMPTYA0, TB_EMPTYA1, TB_EMPTYB0, TB_EMPTYB1, TB_EMPTYC0, TB_EMPTYC1,
  TB_SREADY, TB_D1FULL0, TB_D1FULL1, TB_UREADY,
  TB_D2FULL, TB_OFULL0, TB_OFULL1, TB_D1FREE0, TB_D1FREE1, TB_GATE0,
  TB_GATE1, TB_U0DONE0, TB_U0DONE1, TB_DRAIN, TB_DRAIN2, TB_COUNT
};
constexpr uint32_t TXO_MISC = TXO_BAR + TB_COUNT * 8;
constexpr uint32_t TX_SMEM = TXO_MISC + 16 + 1024;
// The fused kernel's chain CTA keeps P and the decay vectors in a ring of
// three slots of their own (P tile | decay vectors), so that the
// preparation CTA can deliver them a chunk earlier than the two-deep stage
// allows; then full / empty barriers of the ring.
constexpr uint32_t TXO_PC = ((TXO_MISC + 16 + 1023) / 1024) * 1024;
constexpr uint32_t PC_SLOT = 9216, PC_CV = 8192;
constexpr uint32_t TXO_PCBAR = TXO_PC + 3 * PC_SLOT;
// READY barriers of the hand-off ring's four slots (the preparation CTA
// arrives once a slot holds the chunk)
constexpr uint32_t TXO_RDYBAR = TXO_PCBAR + 6 * 8;
constexpr uint32_t TX_FUSED_SMEM = TXO_RDYBAR + 4 * 8 + 1024;
static_assert(TX_FUSED_SMEM <= 232448, "shared memory budget");
static_assert(TX_CV + KCV_BYTES <= TX_STAGE && TX_STAGE % 1024 == 0,
              "transposed stage layout");
static_assert(TX_SMEM <= 232448, "shared memory budget");
// TMEM columns: two accumulators [U^T -> U^T P^T | H^T] (128 each),
// Delta^T (128), S and U^T as bf16 pairs (64, 32).
constexpr uint32_t TX_D1 = 0, TX_D2 = 256, TX_SB = 384, TX_UB = 448;
constexpr uint32_t ID_TX_U0 = idesc_bf16(128, 64, true, false);
constexpr uint32_t ID_TX_N128 = idesc_bf16(128, 128, false, false);
constexpr uint32_t ID_TX_D = idesc_bf16(128, 128, false, true);
constexpr uint32_t ID_TX_N64 = idesc_bf16(128, 64, false, false);

__device__ __forceinline__ uint32_t tx_bar_count(int b, bool fused) {
  switch (b) {
    case TB_D1FREE0: case TB_D1FREE1: return kTxOutThreads / 32;
    // both issuers' commits (Delta^T reads K_d, P U reads P), one per chain
    // warp (gamma, K_d) and one per output warp (e^G); in the fused kernel
    // P and e^G live in a ring of their own, so K alone: the Delta^T
    // issuer's commit and the chain warps
    case TB_EMPTYC0: case TB_EMPTYC1:
      return fused ? 1 + kTxChainThreads / 32
                   : 2 + (kTxChainThreads + kTxOutThreads) / 32;
    case TB_SREADY: case TB_UREADY: return kTxChainThreads / 32;
    default: return 1;
  }
}

// Byte offset of element (token t, column c) of a 64-token x 128-column
// bf16 tile stored as two 64-column blocks with the 128-byte swizzle.
__device__ __forceinline__ uint32_t tx_tile_off(int t, int c) {
  return (uint32_t)((c >> 6) * 8192) + sw128(t, (c & 63) >> 3) + (c & 7) * 2;
}

// Scale the 64 rows of a bf16 tile pair (two 8 KB 64-column blocks `blk`
// bytes apart) by f[row], in place; the 256 chain threads, thread c of them.
// All loads go out before the first store (the stores could alias them).
__device__ __forceinline__ void tx_scale_rows(uint8_t* tile, uint32_t blk,
                                              const float* f, int c) {
  uint4 x[4];
  float s[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = c + k * kTxChainThreads, t = (e >> 3) & 63;
    x[k] = *reinterpret_cast<const uint4*>(tile + (e >> 9) * blk + t * 128 +
                                           (e & 7) * 16);
    s[k] = f[t];
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = c + k * kTxChainThreads, t = (e >> 3) & 63;
    float v[8];
    unpack_bf16x8(x[k], v);
    uint4 w;
    w.x = pack_bf16x2(v[0] * s[k], v[1] * s[k]);
    w.y = pack_bf16x2(v[2] * s[k], v[3] * s[k]);
    w.z = pack_bf16x2(v[4] * s[k], v[5] * s[k]);
    w.w = pack_bf16x2(v[6] * s[k], v[7] * s[k]);
    *reinterpret_cast<uint4*>(tile + (e >> 9) * blk + t * 128 + (e & 7) * 16) = w;
  }
}

// ---------------------------------------------------------------------------
// The preparation CTA of the fused kernel (fused_chunk_kernel below): the
// state-independent part of every chunk of one (sequence, head), handed to
// the chain CTA of its cluster through distributed shared memory instead of
// a workspace in global memory. Three groups of four compute warps take the
// chunks in turn (chunk i: group i % 3), each with a loader warp (gate
// vectors, K and Q by TMA into the group's one stage). P is built over Q's
// first 64-column block and T_U over the second once the [K;Q] K^T product
// has read them. When a chunk is done its results (-W, P, T_U, the chain's
// decay vectors) are gathered into outbox i % 2, so that the stage is free
// for the group's next chunk at once; a copier warp stores the outboxes in
// chunk order, by one bulk copy each, into slot i % 4 of the (sequence,
// head)'s hand-off ring in global memory (small enough to stay in L2; a
// copy between the two CTAs' shared memories measured at about 8 bytes per
// cycle, too slow for 33 KB a chunk), then tells the chain CTA (READY
// barrier i % 4 there), whose producer loads the slot into its stage with
// the chunk's own tiles. A ring slot is refilled once the chain CTA reports
// that the chunk four before has landed (LANDED barrier i % 4 here; the
// chain warps arrive on it when they start on the chunk).
constexpr int kFpGroups = 3;
constexpr uint32_t FP_KQ = 0;        // K0 | Q0 | K1 | Q1 (8 KB each)
constexpr uint32_t FP_AT = 32768;    // fp32 solve buffer, then [T_W; T_W]
constexpr uint32_t FP_VEC = FP_AT + 64 * AP * 4;      // gate vectors
constexpr uint32_t FP_CVS = FP_VEC + VEC_FLOATS * 4;  // the chain's decay
                                                      // vectors, staged
constexpr uint32_t FP_GROUP = 53248;                  // bytes per group
// outboxes, each the image of a ring slot: -W (two 64-column blocks) | P |
// T_U | decay vectors
constexpr uint32_t FP_OB = kFpGroups * FP_GROUP;
constexpr uint32_t OB_W = 0, OB_P = 16384, OB_TU = 24576, OB_CV = 32768;
constexpr uint32_t FP_OB_BYTES = 33792;
constexpr uint32_t RING_COPY = OB_CV + CV_BYTES;  // bytes stored per chunk
constexpr int kRingSlots = 4;
constexpr uint32_t FP_BAR = FP_OB + 2 * FP_OB_BYTES;
enum {
  FB_FULL = 0, FB_MMA = FB_FULL + kFpGroups, FB_MMAW = FB_MMA + kFpGroups,
  FB_DRAIN = FB_MMAW + kFpGroups, FB_SFREE = FB_DRAIN + kFpGroups,
  FB_OBREADY = FB_SFREE + kFpGroups, FB_STORED = FB_OBREADY + 2,
  FB_LANDED = FB_STORED + 6, FB_N = FB_LANDED + kRingSlots
};
constexpr uint32_t FP_MISC = FP_BAR + FB_N * 8;
constexpr uint32_t FP_SMEM = FP_MISC + 16 + 1024;
static_assert(FP_CVS + CV_BYTES <= FP_GROUP && FP_AT % 1024 == 0 &&
                  FP_GROUP % 1024 == 0 && FP_OB_BYTES % 1024 == 0 &&
                  OB_CV + CV_BYTES <= FP_OB_BYTES,
              "preparation CTA layout");
static_assert(FP_SMEM <= 232448, "shared memory budget");
static_assert(kFpGroups * 5 * 32 + 32 == 16 * 32,
              "three groups of four compute warps and a loader, one copier");
// the fused kernel's shared memory serves both roles
constexpr uint32_t FUSED_SMEM =
    FP_SMEM > TX_FUSED_SMEM ? FP_SMEM : TX_FUSED_SMEM;

template <int VARIANT>
__device__ __forceinline__ void prep_role(const ChunkParams& p,
                                          const CUtensorMap& tmk,
                                          const CUtensorMap& tmq, int n,
                                          int h, uint32_t chain) {
  const long long u_index = (long long)n * p.H + h;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + FP_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + FP_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + FP_MISC + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // warps 0-11: compute (group warp / 4); 12-14: the groups' loaders; 15:
  // the outbox copier
  constexpr int kWarpCopier = 4 * kFpGroups + kFpGroups;
  const bool loader = warp >= 4 * kFpGroups && warp < kWarpCopier;
  const int grp = warp < 4 * kFpGroups ? warp >> 2
                                       : (loader ? warp - 4 * kFpGroups : 0);
  const int H = p.H;
  long long bos = 0, eos = 0;
  if (!sequence_range(p, n, bos, eos)) bos = eos = 0;
  const int nch = (int)((eos - bos + C - 1) / C);

  if (tid == 0) {
    for (int b = 0; b < FB_N; ++b) mbar_init(&bars[b], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (loader && lane == 0) {
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmq);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // both CTAs' barriers are initialised before either side uses the other's
  cluster_sync();
  const uint32_t tmem = *tmem_slot + 128u * grp;
  uint8_t* gs = sm + grp * FP_GROUP;
  const uint32_t gsb = base + grp * FP_GROUP;
  float* vec = reinterpret_cast<float*>(gs + FP_VEC);
  uint64_t* full = &bars[FB_FULL + grp];
  const int bid = 1 + grp;  // the group's named barrier

  if (warp == kWarpCopier) {
    // ============ copier: outbox i % 2 into ring slot i % 4 ============
    if (lane == 0) {
      uint8_t* ring = static_cast<uint8_t*>(p.ring) +
                      (size_t)u_index * kRingSlots * FP_OB_BYTES;
      for (int i = 0; i < nch; ++i) {
        const int s = i & 1;
        // the outbox is filled; the slot's previous chunk (i - 4) has
        // landed in the chain CTA
        if (!mbar_wait(&bars[FB_OBREADY + s], (i >> 1) & 1, abort_flag) ||
            (i >= kRingSlots &&
             !mbar_spin_remote(&bars[FB_LANDED + i % kRingSlots],
                               ((i / kRingSlots) - 1) & 1, abort_flag)))
          break;
        bulk_store(ring + (size_t)(i % kRingSlots) * FP_OB_BYTES,
                   sm + FP_OB + s * FP_OB_BYTES, RING_COPY);
        bulk_commit();
        bulk_wait_read();
        // outbox s may take chunk i + 2 (STORED barrier i % 6: its waiter,
        // the group of chunk i + 2, waits every phase of it in order)
        mbar_arrive(&bars[FB_STORED + i % 6]);
        bulk_wait_all();
        // the slot's bytes are in global memory: tell the chain CTA
        asm volatile("fence.proxy.async.global;" ::: "memory");
        mbar_arrive_cluster(
            map_to_cta(sm + TXO_RDYBAR + 8 * (i % kRingSlots), chain));
      }
    }
  } else if (loader) {
    // ============ loader: gate vectors, K and Q by TMA ============
    int li = 0;
    bool ok = true;
    for (int i = grp; i < nch; i += kFpGroups, ++li) {
      const long long t0 = bos + (long long)i * C;
      const int len = (int)min((long long)C, eos - t0);
      // the gate vectors are formed while the group still works on its
      // previous chunk; they and the stage are written once the compute
      // warps have finished it
      const GateLanes gl = gate_lanes<VARIANT>(p.g, p.beta, (size_t)t0 * H + h,
                                               H, len, p.prologue != 0, lane);
      if (lane == 0 && li >= 1)
        ok = mbar_wait(&bars[FB_SFREE + grp], (li - 1) & 1, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      put_gate_lanes(gl, vec, lane);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(full, 32768);
        tma_load_3d(gs + FP_KQ, &tmk, full, 0, h, (int)t0);
        tma_load_3d(gs + FP_KQ + 8192, &tmq, full, 0, h, (int)t0);
        tma_load_3d(gs + FP_KQ + 16384, &tmk, full, 64, h, (int)t0);
        tma_load_3d(gs + FP_KQ + 24576, &tmq, full, 64, h, (int)t0);
        if (i + kFpGroups < nch) {
          const int t2 = (int)(t0 + kFpGroups * C);
          prefetch_l2_3d(&tmk, 0, h, t2);
          prefetch_l2_3d(&tmk, 64, h, t2);
          prefetch_l2_3d(&tmq, 0, h, t2);
          prefetch_l2_3d(&tmq, 64, h, t2);
        }
      }
    }
    // never leave with a TMA copy still landing in shared memory
    if (lane == 0 && li > 0) wait_ignoring_abort(full, (li - 1) & 1);
  } else if (warp < 4 * kFpGroups) {
    // ================= compute warps of the group =================
    // A warp reaches the TMEM lanes of its quarter warp % 4 only; the four
    // compute warps of a group cover the four quarters: thread ct owns row
    // ct of the group's 128-lane accumulator.
    const int q = warp & 3;
    const int ct = 32 * q + lane;  // 0..127
    float* AT = reinterpret_cast<float*>(gs + FP_AT);
    uint8_t* st = gs + FP_KQ;
    const uint32_t stb = gsb + FP_KQ;
    int li = 0;
    for (int i = grp; i < nch; i += kFpGroups, ++li) {
      bool ok = mbar_wait(full, li & 1, abort_flag);
      if (!bar_and(bid, 128, ok)) break;
      if (ct == 0) {
        // [K;Q] K^T: rows 0-63 K K^T, rows 64-127 Q K^T
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t a = sdesc(stb + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
          mma_bf16(tmem, a, a, ID_PREP, k > 0);
        }
        mma_commit(&bars[FB_MMA + grp]);
      }
      {
        // inverse lengths of raw k / q rows (prologue), folded into the
        // factors the rows and columns are scaled with (as in
        // ut_prep_kernel)
        const int r = ct & 63;
        float inv = 1.f;
        if (p.prologue) {
          const uint8_t* tl = st + (ct < 64 ? 0 : 8192);
          float ss = 0.f;
#pragma unroll
          for (int cb = 0; cb < 2; ++cb) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              float f[8];
              unpack_bf16x8(*reinterpret_cast<const uint4*>(tl + cb * 16384 + sw128(r, c)), f);
#pragma unroll
              for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
            }
          }
          inv = ss > 0.f ? rsqrtf(ss) : 0.f;
        }
        vec[(ct < 64 ? VEC_SK : VEC_SQ) + r] = inv;
        if (p.prologue) {
          if (ct < 64) {
            vec[VEC_EGPB + r] *= inv;
            vec[VEC_IEG + r] *= inv;
            vec[VEC_DEC + r] *= inv;
          } else {
            vec[VEC_EG + r] *= inv;
          }
        }
        named_bar(bid, 128);
        // the chain's decay vectors (after the fold), staged for the outbox
        float* cv = reinterpret_cast<float*>(gs + FP_CVS);
        if (ct < 64) {
          cv[CV_EG + ct] = vec[VEC_EG + ct];
          cv[CV_DEC + ct] = vec[VEC_DEC + ct];
        } else if (ct < 68) {
          cv[CV_GAMMA + ct - 64] = ct == 64 ? vec[VEC_GAMMA] : 0.f;
        }
      }
      ok = mbar_wait(&bars[FB_MMA + grp], li & 1, abort_flag);
      if (!bar_and(bid, 128, ok)) break;
      tc_fence_after();
      const uint32_t lanes = (uint32_t)(32 * q) << 16;
      if (ct < 64) {
        // row r of A (as in ut_prep_kernel)
        const int r = ct;
        const bool safe = vec[VEC_SAFE] != 0.f;
        const float er = vec[VEC_EGPB + r];
        const float br = vec[VEC_BETA + r] * vec[VEC_SK + r];
        const float* alpha = vec + VEC_ALPHA;
        const float* sk = vec + VEC_SK;
        float d = 1.f;
#pragma unroll
        for (int hf = 1; hf >= 0; --hf) {
          float x[32];
          tmem_ld32(tmem + lanes + 32 * hf, x);
          tmem_ld_wait();
          if (safe) {
            const float4* w4 = reinterpret_cast<const float4*>(vec + VEC_IEG + 32 * hf);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 w = w4[c4];
              const int j = 32 * hf + 4 * c4;
              x[4 * c4] = j < r ? er * w.x * x[4 * c4] : 0.f;
              x[4 * c4 + 1] = j + 1 < r ? er * w.y * x[4 * c4 + 1] : 0.f;
              x[4 * c4 + 2] = j + 2 < r ? er * w.z * x[4 * c4 + 2] : 0.f;
              x[4 * c4 + 3] = j + 3 < r ? er * w.w * x[4 * c4 + 3] : 0.f;
            }
          } else {
#pragma unroll
            for (int e = 31; e >= 0; --e) {
              const int jj = 32 * hf + e;
              float a = 0.f;
              if (jj < r) {
                if (VARIANT == GDN_GATE_BEFORE_PREDICT) {
                  d *= alpha[jj + 1];
                  a = br * d * sk[jj] * x[e];
                } else {
                  a = br * d * sk[jj] * x[e];
                  d *= alpha[jj];
                }
              }
              x[e] = a;
            }
          }
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4)
            *reinterpret_cast<float4*>(AT + r * AP + 32 * hf + 4 * c4) =
                make_float4(x[4 * c4], x[4 * c4 + 1], x[4 * c4 + 2], x[4 * c4 + 3]);
        }
      } else {
        // row r of P, over Q's first block (read by the K K^T product only)
        const int r = ct - 64;
        const bool safe = vec[VEC_SAFE] != 0.f;
        const float er = vec[VEC_EG + r];
        const float* alpha = vec + VEC_ALPHA;
        uint8_t* ptile = st + 8192;
        float d = 1.f;
#pragma unroll
        for (int hf = 1; hf >= 0; --hf) {
          float x[32];
          tmem_ld32(tmem + lanes + 32 * hf, x);
          tmem_ld_wait();
          if (safe) {
            const float4* w4 = reinterpret_cast<const float4*>(vec + VEC_IEG + 32 * hf);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 w = w4[c4];
              const int j = 32 * hf + 4 * c4;
              x[4 * c4] = j <= r ? w.x * x[4 * c4] : 0.f;
              x[4 * c4 + 1] = j + 1 <= r ? w.y * x[4 * c4 + 1] : 0.f;
              x[4 * c4 + 2] = j + 2 <= r ? w.z * x[4 * c4 + 2] : 0.f;
              x[4 * c4 + 3] = j + 3 <= r ? w.w * x[4 * c4 + 3] : 0.f;
            }
            store_half_bf16_scaled(ptile, r, hf, x, er);
          } else {
            const float* sk = vec + VEC_SK;
#pragma unroll
            for (int e = 31; e >= 0; --e) {
              const int jj = 32 * hf + e;
              float pv = 0.f;
              if (jj <= r) {
                pv = d * sk[jj] * x[e];
                d *= alpha[jj];
              }
              x[e] = pv;
            }
            store_half_bf16_scaled(ptile, r, hf, x, vec[VEC_SQ + r]);
          }
        }
      }
      tc_fence_before();
      named_bar(bid, 128);
      solve_unit_lower(AT, ct, bid);
      {
        // T_W rows into [T_W; T_W] over the solve buffer, T_U rows over Q's
        // second block (thread (r, hh): columns 32 hh .. 32 hh + 31)
        const int r = ct & 63, hh = ct >> 6;
        float t[32];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 v = *reinterpret_cast<const float4*>(AT + r * AP + 32 * hh + 4 * c4);
          t[4 * c4] = v.x; t[4 * c4 + 1] = v.y; t[4 * c4 + 2] = v.z; t[4 * c4 + 3] = v.w;
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = 32 * hh + e;
          t[e] = col < r ? t[e] : (col == r ? 1.f : 0.f);
        }
        named_bar(bid, 128);  // T fully read before the tile overwrites it
        float tw[32], tu[32];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 w4 = *reinterpret_cast<const float4*>(vec + VEC_EGPB + 32 * hh + 4 * c4);
          const float4 u4 = *reinterpret_cast<const float4*>(vec + VEC_BETA + 32 * hh + 4 * c4);
          tw[4 * c4] = t[4 * c4] * w4.x; tw[4 * c4 + 1] = t[4 * c4 + 1] * w4.y;
          tw[4 * c4 + 2] = t[4 * c4 + 2] * w4.z; tw[4 * c4 + 3] = t[4 * c4 + 3] * w4.w;
          tu[4 * c4] = t[4 * c4] * u4.x; tu[4 * c4 + 1] = t[4 * c4 + 1] * u4.y;
          tu[4 * c4 + 2] = t[4 * c4 + 2] * u4.z; tu[4 * c4 + 3] = t[4 * c4 + 3] * u4.w;
        }
        uint8_t* tile_tw = gs + FP_AT;
        store_half_bf16(tile_tw, r, hh, tw);
        store_half_bf16(tile_tw, 64 + r, hh, tw);
        store_half_bf16(st + 24576, r, hh, tu);
        fence_proxy_async();
      }
      named_bar(bid, 128);
      if (ct == 0) {
        // [T_W; T_W] K: both halves of the accumulator hold W
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem, sdesc(gsb + FP_AT + k * 32, 16, 1024),
                   sdesc(stb + k * 2048, 16384, 1024), ID_PREP_W, k > 0);
        mma_commit(&bars[FB_MMAW + grp]);
      }
      // Outbox i % 2 is free once the copier has stored chunk i - 2 from it
      // (STORED barrier (i - 2) % 6, whose phases this group alone waits, in
      // order; a barrier per outbox would be waited by the groups in turn,
      // and a group running ahead could take a phase two back for its own).
      ok = mbar_wait(&bars[FB_MMAW + grp], li & 1, abort_flag) &&
           (ct != 0 || i < 2 ||
            mbar_wait(&bars[FB_STORED + (i - 2) % 6], ((i - 2) / 6) & 1,
                      abort_flag));
      if (!bar_and(bid, 128, ok)) break;
      tc_fence_after();
      {
        uint8_t* ob = sm + FP_OB + (i & 1) * FP_OB_BYTES;
        // -W: warps of lane quarters 0-1 columns 0-63, 2-3 columns 64-127
        // (the copy of W in lanes 64-127)
        const int r = ct & 63, cb = q >> 1;
        uint8_t* wtile = ob + OB_W + cb * TILE_BYTES;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          float x[32];
          tmem_ld32(tmem + lanes + 64 * cb + 32 * hf, x);
          tmem_ld_wait();
          store_half_bf16_scaled(wtile, r, hf, x, -1.f);
        }
        // P, T_U and the decay vectors: byte images, 16 bytes a piece
        uint4 pv[4], uv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pv[e] = reinterpret_cast<const uint4*>(st + 8192)[ct + 128 * e];
          uv[e] = reinterpret_cast<const uint4*>(st + 24576)[ct + 128 * e];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          reinterpret_cast<uint4*>(ob + OB_P)[ct + 128 * e] = pv[e];
          reinterpret_cast<uint4*>(ob + OB_TU)[ct + 128 * e] = uv[e];
        }
        if (ct < (int)(CV_BYTES / 16))
          reinterpret_cast<uint4*>(ob + OB_CV)[ct] =
              reinterpret_cast<const uint4*>(gs + FP_CVS)[ct];
        fence_proxy_async();  // the bulk copies read the outbox
      }
      tc_fence_before();
      named_bar(bid, 128);
      if (ct == 0) {
        mbar_arrive(&bars[FB_SFREE + grp]);        // the stage may load again
        mbar_arrive(&bars[FB_OBREADY + (i & 1)]);  // the outbox may be copied
      }
    }
    if (ct == 0) {
      mma_commit(&bars[FB_DRAIN + grp]);
      wait_ignoring_abort(&bars[FB_DRAIN + grp], 0);
    }
  }
  // Neither CTA leaves while the other may still write into it: every copy
  // from this CTA into the chain CTA has landed once the chain CTA arrives
  // here (it consumed every chunk, or gave up after its bounded waits), and
  // the chain CTA's remote arrivals were issued before it arrives.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(*tmem_slot, 512);
  }
  if (tid == 0 && *abort_flag) record_status(p.status, GDN_ERR_TIMEOUT);
}

// The whole-state chain. KDA: per-channel decays (the Q_g / K_d images from
// the workspace, the state decayed column by column); otherwise the scalar
// gate. FUSED: the chain CTA of fused_chunk_kernel, fed by the preparation
// CTA of its cluster (rank 0) instead of the workspace; `xblock` is the
// 128-row block (blockIdx.x of chain_tx_kernel, 0 in the fused kernel).
template <bool KDA, bool FUSED>
__device__ __forceinline__ void chain_tx_body(
    const ChunkParams& p, const CUtensorMap& tmq, const CUtensorMap& tmk,
    const CUtensorMap& tmv, const CUtensorMap& tmo, const CUtensorMap& tmg,
    int nch_dense, int tiles, int xblock, int h, int zblock, uint32_t prep) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + TXO_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + TXO_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + TXO_MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H, dv = p.dv;
  const int n = zblock / p.part_count;
  const int part = p.part_begin + zblock % p.part_count;
  const int row0 = xblock * TXR;
  const bool value_rows = row0 < dv;
  const bool split_tail = (p.mode == kModeSplit) && part > 0;
  // d_k = 64 runs on the d_k = 128 layout (K and Q's second 64-column block
  // loads as zeros): the state's columns (and the scaling matrix's rows)
  // d_k..127 stay zero; only those < d_k are read and written
  const int dkr = p.dk;
  if (!value_rows && !(split_tail && row0 < dv + dkr)) return;
  const bool scale_rows = !value_rows;
  const bool emit = value_rows && ((p.mode == kModeOutput) || part == 0);
  const bool epi = p.epilogue && emit;
  const bool has_gate = epi && p.gate_z != nullptr;
  long long bos = 0, eos = 0;
  // (the fused kernel's chain CTA carries on with no chunks: it meets its
  // preparation CTA at the cluster barriers)
  if (!sequence_range(p, n, bos, eos) && !FUSED) return;
  const int nch = (int)((eos - bos + C - 1) / C);
  int c_begin, c_end;
  part_range(nch, p.parts, part, c_begin, c_end);
  const int nloc = c_end - c_begin;
  const size_t nh = (size_t)n * H + h;

  // ---- set-up ----
  // fused: P and decay-vector ring (full: the producer's arm; empty: the
  // side issuer's P U commit, the chain warps and the output warps)
  uint64_t* pcbars = reinterpret_cast<uint64_t*>(sm + TXO_PCBAR);
  if (tid == 0) {
    for (int b = 0; b < TB_COUNT; ++b)
      mbar_init(&bars[b], tx_bar_count(b, FUSED));
    if (FUSED) {
      for (int r = 0; r < 3; ++r) {
        mbar_init(&pcbars[r], 1);
        mbar_init(&pcbars[3 + r], 1 + (kTxChainThreads + kTxOutThreads) / 32);
      }
      for (int r = 0; r < 4; ++r) mbar_init(&pcbars[6 + r], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < kTxChainThreads) {
    // V of both stages for rows of the scaling matrix (the second 64-column
    // block only when d_v = 64)
    const uint4 z = make_uint4(0, 0, 0, 0);
    const int v0 = scale_rows ? 0 : dv * 8;
    for (int i = tid; i < 2048; i += kTxChainThreads)
      if ((i & 1023) >= v0)
        *reinterpret_cast<uint4*>(sm + (i >> 10) * TX_STAGE + TX_V + (i & 1023) * 16) = z;
  }
  if (warp == kTxWarpMMA) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == kTxWarpProducer && lane == 0) {
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
    prefetch_tmap(&tmo);
    if (has_gate) prefetch_tmap(&tmg);
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // fused: both CTAs' barriers initialised before either side uses the
  // other's
  if (FUSED) cluster_sync();
  const uint32_t tmem = *tmem_slot;
  auto stage = [&](int i) { return base + (i & 1) * TX_STAGE; };
  // set-up above overlaps the tail of the preceding kernel
  griddep_wait();
  const int cbase = (nloc > 0 && !FUSED) ? chunk_base(p, n, nch_dense) + c_begin : 0;

  if (FUSED && warp == kTxWarpProducer) {
    // ================= producer of the fused kernel =================
    // Q, K, V by tensor map; -W, P, T_U and the decay vectors are stored
    // into the stage by the preparation CTA (rank `prep`). Each group's
    // barrier is armed for all of its bytes, then the preparation CTA is
    // told (SLOT barrier i % 6) that stage i % 2 may take chunk i.
    if (lane == 0) {
      auto prefetch_v = [&](int i) {
        const int tok = (int)(bos + (long long)(c_begin + i) * C);
        prefetch_l2_3d(&tmv, 0, h, tok);
        if (dv > 64) prefetch_l2_3d(&tmv, 64, h, tok);
      };
      if (nloc > 0) prefetch_v(0);
      if (nloc > 1) prefetch_v(1);
      int armed = 0;  // chunks whose places are all armed
      const uint8_t* ring = static_cast<const uint8_t*>(p.ring) +
                            ((size_t)n * H + h) * kRingSlots * FP_OB_BYTES;
      uint64_t* ready = pcbars + 6;
      for (int i = 0; i < nloc; ++i) {
        const int s = i & 1, r = i % 3;
        const uint32_t ph = ((i >> 1) - 1) & 1;  // release of chunk i - 2
        const int tok = (int)(bos + (long long)(c_begin + i) * C);
        uint8_t* st = sm + s * TX_STAGE;
        const uint8_t* slot = ring + (size_t)(i % kRingSlots) * FP_OB_BYTES;
        // the preparation CTA has stored chunk i in its ring slot
        if (!mbar_wait(&ready[i % kRingSlots], (i / kRingSlots) & 1, abort_flag))
          break;
        asm volatile("fence.acq_rel.cluster;\n\tfence.proxy.async.global;" :::
                         "memory");
        // ring slot r (released by chunk i - 3): P and the decay vectors
        if (i >= 3 && !mbar_wait(&pcbars[3 + r], ((i / 3) - 1) & 1, abort_flag))
          break;
        mbar_arrive_expect_tx(&pcbars[r], TILE_BYTES + CV_BYTES);
        bulk_load(sm + TXO_PC + r * PC_SLOT, slot + OB_P, TILE_BYTES, &pcbars[r]);
        bulk_load(sm + TXO_PC + r * PC_SLOT + PC_CV, slot + OB_CV, CV_BYTES,
                  &pcbars[r]);
        // group A: V and T_U
        if (i >= 2 && !mbar_wait(&bars[TB_EMPTYA0 + s], ph, abort_flag)) break;
        uint64_t* fa = &bars[TB_FULLA0 + s];
        mbar_arrive_expect_tx(fa, TX_A_BYTES - 128u * (128 - dv));
        tma_load_3d(st + TX_V, &tmv, fa, 0, h, tok);
        if (dv > 64) tma_load_3d(st + TX_V + 8192, &tmv, fa, 64, h, tok);
        bulk_load(st + TX_TU, slot + OB_TU, TILE_BYTES, fa);
        // group B: Q and -W
        if (i >= 2 && !mbar_wait(&bars[TB_EMPTYB0 + s], ph, abort_flag)) break;
        uint64_t* fb = &bars[TB_FULLB0 + s];
        mbar_arrive_expect_tx(fb, TX_B_BYTES);
        tma_load_3d(st + TX_Q, &tmq, fb, 0, h, tok);
        tma_load_3d(st + TX_Q + TX_WQ_CB, &tmq, fb, 64, h, tok);
        bulk_load(st + TX_W, slot + OB_W, TILE_BYTES, fb);
        bulk_load(st + TX_W + TX_WQ_CB, slot + OB_W + TILE_BYTES, TILE_BYTES, fb);
        // group C: K alone
        if (i >= 2 && !mbar_wait(&bars[TB_EMPTYC0 + s], ph, abort_flag)) break;
        uint64_t* fc = &bars[TB_FULLC0 + s];
        mbar_arrive_expect_tx(fc, 16384);
        tma_load_3d(st + TX_K, &tmk, fc, 0, h, tok);
        tma_load_3d(st + TX_K + 8192, &tmk, fc, 64, h, tok);
        armed = i + 1;
        if (i + 2 < nloc) prefetch_v(i + 2);
      }
      // never leave with a copy still landing in shared memory: the latest
      // use of every place (a chunk cut short by an abort may have some of
      // its places armed but never filled: those waits give up after the
      // bounded wait)
      const int last = min(armed + 1, nloc);  // chunks that may be in flight
      for (int i = max(0, last - 3); i < last; ++i)
        wait_ignoring_abort(&pcbars[i % 3], (i / 3) & 1);
      for (int i = max(0, last - 2); i < last; ++i) {
        const uint32_t pf = (i >> 1) & 1;
        wait_ignoring_abort(&bars[TB_FULLA0 + (i & 1)], pf);
        wait_ignoring_abort(&bars[TB_FULLB0 + (i & 1)], pf);
        wait_ignoring_abort(&bars[TB_FULLC0 + (i & 1)], pf);
      }
    }
  } else if (warp == kTxWarpProducer) {
    // ================= TMA producer =================
    // Q, K, V by tensor map; -W, P, T_U and the decay vectors are images in
    // the workspace (bulk copies; the tile index is clamped because those
    // copies have no bounds check). Chunk i + kChainPrefetch is prefetched
    // into L2 when chunk i is loaded.
    if (lane == 0) {
      const uint8_t* wimg = static_cast<const uint8_t*>(p.wneg);
      const uint8_t* pimg = static_cast<const uint8_t*>(p.pm);
      const uint8_t* uimg = static_cast<const uint8_t*>(p.tu);
      const uint8_t* qimg = static_cast<const uint8_t*>(p.qg);
      const uint8_t* kimg = static_cast<const uint8_t*>(p.kd);
      const bool kda = KDA;
      const int cvf = kda ? KCV_FLOATS : CV_FLOATS;
      const uint32_t cvb = kda ? KCV_BYTES : CV_BYTES;
      auto prefetch = [&](int i) {
        const int tok = (int)(bos + (long long)(c_begin + i) * C);
        const size_t tz = (size_t)min((cbase + i) * H + h, tiles - 1);
        if (kda) {
          prefetch_l2(kimg + tz * WS_KD_BYTES, WS_KD_BYTES);
          if (emit) prefetch_l2(qimg + tz * WS_QG_BYTES, WS_QG_BYTES);
        } else {
          prefetch_l2_3d(&tmk, 0, h, tok);
          prefetch_l2_3d(&tmk, 64, h, tok);
          if (emit) {
            prefetch_l2_3d(&tmq, 0, h, tok);
            prefetch_l2_3d(&tmq, 64, h, tok);
          }
        }
        if (!scale_rows) prefetch_l2_3d(&tmv, 0, h, tok);
        if (!scale_rows && dv > 64) prefetch_l2_3d(&tmv, 64, h, tok);
        prefetch_l2(wimg + tz * WS_W_BYTES, WS_W_BYTES);
        prefetch_l2(pimg + tz * WS_P_BYTES, WS_P_BYTES);
        prefetch_l2(uimg + tz * WS_TU_BYTES, WS_TU_BYTES);
        prefetch_l2(p.cv + tz * cvf, cvb);
      };
      for (int i = 0; i < min(nloc, kChainPrefetch); ++i) prefetch(i);
      int issued = 0, part_groups = 0;  // chunks fully issued; groups of the next
      for (int i = 0; i < nloc; ++i) {
        const int s = i & 1;
        const uint32_t ph = ((i >> 1) - 1) & 1;  // release of chunk i - 2
        const int tok = (int)(bos + (long long)(c_begin + i) * C);
        const size_t tz = (size_t)min((cbase + i) * H + h, tiles - 1);
        uint8_t* st = sm + s * TX_STAGE;
        if (i >= 2 && !mbar_wait(&bars[TB_EMPTYA0 + s], ph, abort_flag)) break;
        uint64_t* fa = &bars[TB_FULLA0 + s];
        mbar_arrive_expect_tx(fa, TX_A_BYTES - (scale_rows ? 16384u : 128u * (128 - dv)));
        if (!scale_rows) tma_load_3d(st + TX_V, &tmv, fa, 0, h, tok);
        if (!scale_rows && dv > 64) tma_load_3d(st + TX_V + 8192, &tmv, fa, 64, h, tok);
        bulk_load(st + TX_TU, uimg + tz * WS_TU_BYTES, TILE_BYTES, fa);
        if (i >= 2 && !mbar_wait(&bars[TB_EMPTYB0 + s], ph, abort_flag)) {
          part_groups = 1;  // group A of chunk i is in flight
          break;
        }
        uint64_t* fb = &bars[TB_FULLB0 + s];
        mbar_arrive_expect_tx(fb, TX_B_BYTES);
        bulk_load(st + TX_W, wimg + tz * WS_W_BYTES, TILE_BYTES, fb);
        bulk_load(st + TX_W + TX_WQ_CB, wimg + tz * WS_W_BYTES + TILE_BYTES,
                  TILE_BYTES, fb);
        if (kda) {
          bulk_load(st + TX_Q, qimg + tz * WS_QG_BYTES, TILE_BYTES, fb);
          bulk_load(st + TX_Q + TX_WQ_CB, qimg + tz * WS_QG_BYTES + TILE_BYTES,
                    TILE_BYTES, fb);
        } else {
          tma_load_3d(st + TX_Q, &tmq, fb, 0, h, tok);
          tma_load_3d(st + TX_Q + TX_WQ_CB, &tmq, fb, 64, h, tok);
        }
        if (i >= 2 && !mbar_wait(&bars[TB_EMPTYC0 + s], ph, abort_flag)) {
          part_groups = 2;  // groups A and B of chunk i are in flight
          break;
        }
        uint64_t* fc = &bars[TB_FULLC0 + s];
        mbar_arrive_expect_tx(fc, TX_C_BYTES - CV_BYTES + cvb);
        if (kda) {
          bulk_load(st + TX_K, kimg + tz * WS_KD_BYTES, WS_KD_BYTES, fc);
        } else {
          tma_load_3d(st + TX_K, &tmk, fc, 0, h, tok);
          tma_load_3d(st + TX_K + 8192, &tmk, fc, 64, h, tok);
        }
        bulk_load(st + TX_P, pimg + tz * WS_P_BYTES, TILE_BYTES, fc);
        bulk_load(st + TX_CV, p.cv + tz * cvf, cvb, fc);
        if (i + kChainPrefetch < nloc) prefetch(i + kChainPrefetch);
        issued = i + 1;
      }
      // never leave with a copy still landing in shared memory: the groups
      // of the last two chunks issued (a chunk cut short by an abort has
      // only its first groups in flight)
      const int full = issued;
      for (int i = max(0, full - 2); i < full; ++i) {
        wait_ignoring_abort(&bars[TB_FULLA0 + (i & 1)], (i >> 1) & 1);
        wait_ignoring_abort(&bars[TB_FULLB0 + (i & 1)], (i >> 1) & 1);
        wait_ignoring_abort(&bars[TB_FULLC0 + (i & 1)], (i >> 1) & 1);
      }
      if (part_groups >= 1)
        wait_ignoring_abort(&bars[TB_FULLA0 + (full & 1)], (full >> 1) & 1);
      if (part_groups >= 2)
        wait_ignoring_abort(&bars[TB_FULLB0 + (full & 1)], (full >> 1) & 1);
    }
  } else if (warp == kTxWarpMMA) {
    // ================= chain products =================
    // [-W;Q] of chunk i once the state is in TMEM (and U0^T of chunk i has
    // completed), Delta^T once U^T and K_d are; polled, so that each goes
    // in the moment its barrier completes.
    if (lane == 0 && nloc > 0) {
      for (int i = 0; i < nloc; ++i) {
        const int b = i & 1;
        if (!mbar_spin(&bars[TB_SREADY], i & 1, abort_flag) ||
            !mbar_spin(&bars[TB_FULLB0 + b], (i >> 1) & 1, abort_flag) ||
            !mbar_spin(&bars[TB_U0DONE0 + b], (i >> 1) & 1, abort_flag))
          break;
        tc_fence_after();
        const uint32_t st = stage(i);
        const uint32_t d1 = tmem + TX_D1 + 128 * b;
        // += S [-W; Q]^T, one 64-column block of d_k at a time
        mma_bf16_ta_run<4>(d1, tmem + TX_SB, sdesc(st + TX_W, 16, 1024), 32,
                           ID_TX_N128, true);
        mma_bf16_ta_run<4>(d1, tmem + TX_SB + 32,
                           sdesc(st + TX_W + TX_WQ_CB, 16, 1024), 32,
                           ID_TX_N128, true);
        mma_commit(&bars[TB_D1FULL0 + b]);
        mma_commit(&bars[TB_EMPTYB0 + b]);
        if (!mbar_spin(&bars[TB_UREADY], i & 1, abort_flag) ||
            !mbar_spin(&bars[TB_FULLC0 + b], (i >> 1) & 1, abort_flag))
          break;
        tc_fence_after();
        // Delta^T = U^T K_d
        mma_bf16_ta_run<4>(tmem + TX_D2, tmem + TX_UB,
                           sdesc(st + TX_K, 8192, 1024), 2048, ID_TX_D, false);
        mma_commit(&bars[TB_D2FULL]);
        mma_commit(&bars[TB_EMPTYC0 + b]);
      }
      mma_commit(&bars[TB_DRAIN]);
      wait_ignoring_abort(&bars[TB_DRAIN], 0);
    }
  } else if (warp == kTxWarpSide) {
    // ================= side products =================
    // U0^T of chunk i + 1 into the other accumulator once chunk i's [-W;Q]
    // product has completed (it then runs while U^T is converted) and the
    // output warps have read chunk i - 1 out of it (and zeroed its H^T); U^T P^T of chunk i over
    // the converted U^T once chunk i's Delta^T has completed (it runs during
    // the state update). A commit covers only this thread's products, so
    // the chain warps check P U (chunk i - 1) before they overwrite U^T.
    if (lane == 0 && nloc > 0) {
      auto u0 = [&](int j) {
        const int s = j & 1;
        if (!mbar_wait(&bars[TB_FULLA0 + s], (j >> 1) & 1, abort_flag))
          return false;
        // (the output warps free each accumulator once before chunk 0)
        if (emit && !mbar_wait(&bars[TB_D1FREE0 + s], (j >> 1) & 1, abort_flag))
          return false;
        tc_fence_after();
        const uint32_t st = stage(j);
        mma_bf16_run<4>(tmem + TX_D1 + 128 * s, sdesc(st + TX_V, 8192, 1024),
                        2048, sdesc(st + TX_TU, 16, 1024), 32, ID_TX_U0, false);
        mma_commit(&bars[TB_U0DONE0 + s]);
        mma_commit(&bars[TB_EMPTYA0 + s]);
        return true;
      };
      bool ok = u0(0);
      if (FUSED) {
        // The preparation CTA's T_U of chunk i + 1 may land after chunk i's
        // Delta^T: issue U0^T of chunk i + 1 and U^T P^T of chunk i in
        // whichever order their operands arrive.
        for (int i = 0; ok && i < nloc; ++i) {
          const int b = i & 1, nb = b ^ 1;
          bool need_u0 = i + 1 < nloc, need_pu = true;
          const uint64_t t0 = globaltimer_ns();
          for (uint32_t it = 0; need_u0 || need_pu; ++it) {
            if (need_u0 && mbar_test(&bars[TB_D1FULL0 + b], (i >> 1) & 1) &&
                mbar_test(&bars[TB_FULLA0 + nb], ((i + 1) >> 1) & 1) &&
                mbar_test(&bars[TB_D1FREE0 + nb], ((i + 1) >> 1) & 1)) {
              tc_fence_after();
              const uint32_t st = stage(i + 1);
              mma_bf16_run<4>(tmem + TX_D1 + 128 * nb, sdesc(st + TX_V, 8192, 1024),
                              2048, sdesc(st + TX_TU, 16, 1024), 32, ID_TX_U0,
                              false);
              mma_commit(&bars[TB_U0DONE0 + nb]);
              mma_commit(&bars[TB_EMPTYA0 + nb]);
              need_u0 = false;
            }
            if (need_pu && mbar_test(&bars[TB_D2FULL], i & 1) &&
                mbar_test(&pcbars[i % 3], (i / 3) & 1)) {
              tc_fence_after();
              // U^T P^T over U^T (P in ring slot i % 3)
              mma_bf16_ta_run<4>(tmem + TX_D1 + 128 * b, tmem + TX_UB,
                                 sdesc(base + TXO_PC + (i % 3) * PC_SLOT, 16, 1024),
                                 32, ID_TX_N64, false);
              mma_commit(&bars[TB_OFULL0 + b]);
              mma_commit(&pcbars[3 + i % 3]);
              need_pu = false;
            }
            if ((it & 255) == 255) {
              if (*abort_flag) { ok = false; break; }
              if (globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                ok = false;
                break;
              }
            }
          }
        }
      }
      for (int i = 0; !FUSED && ok && i < nloc; ++i) {
        const int b = i & 1;
        if (i + 1 < nloc) {
          ok = mbar_wait(&bars[TB_D1FULL0 + b], (i >> 1) & 1, abort_flag) &&
               u0(i + 1);
          if (!ok) break;
        }
        if (emit) {
          if (!mbar_wait(&bars[TB_D2FULL], i & 1, abort_flag) ||
              !mbar_wait(&bars[TB_FULLC0 + b], (i >> 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // U^T P^T over U^T
          mma_bf16_ta_run<4>(tmem + TX_D1 + 128 * b, tmem + TX_UB,
                             sdesc(stage(i) + TX_P, 16, 1024), 32, ID_TX_N64,
                             false);
          mma_commit(&bars[TB_OFULL0 + b]);
        }
        mma_commit(&bars[TB_EMPTYC0 + b]);
      }
      mma_commit(&bars[TB_DRAIN2]);
      wait_ignoring_abort(&bars[TB_DRAIN2], 0);
    }
  } else if (warp < kTxChainThreads / 32) {
    // ================= chain warps =================
    // row r = 32 (warp & 3) + lane of S (TMEM lane r), d_k columns
    // 64 ch .. 64 ch + 63 with ch = warp >> 2 (fp32, in registers)
    const int ch = warp >> 2;
    const int r = 32 * (warp & 3) + lane;
    const uint32_t lanes = (uint32_t)(32 * (warp & 3)) << 16;
    float S[64];
    // value rows r >= d_v (d_v = 64) and scaling-matrix rows r >= d_k stay
    // zero: no input, no output; so do the columns 64 ch >= d_k
    const bool live = scale_rows ? r < dkr : r < dv;
    const bool live_cols = 64 * ch < dkr;
    if (scale_rows) {
#pragma unroll
      for (int c = 0; c < 64; ++c) S[c] = (live && r == 64 * ch + c) ? 1.f : 0.f;
    } else if (split_tail || !live || !live_cols) {
#pragma unroll
      for (int c = 0; c < 64; ++c) S[c] = 0.f;
    } else if (part > 0) {
      const float4* src = reinterpret_cast<const float4*>(
          p.ws_start + ((nh * p.parts + part) * dv + r) * dkr + 64 * ch);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float4 v4 = src[c];
        S[4 * c] = v4.x; S[4 * c + 1] = v4.y; S[4 * c + 2] = v4.z; S[4 * c + 3] = v4.w;
      }
    } else if (p.h0) {
      const float* src = p.h0 + (nh * dkr + 64 * ch) * dv + r;
#pragma unroll
      for (int c = 0; c < 64; ++c) S[c] = src[(size_t)c * dv];
    } else {
#pragma unroll
      for (int c = 0; c < 64; ++c) S[c] = 0.f;
    }
    // S as bf16 pairs: the A operand of the next [-W;Q_g] product
    auto put_s = [&]() {
      uint32_t w[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) w[c] = pack_bf16x2(S[2 * c], S[2 * c + 1]);
      tmem_st32(tmem + TX_SB + lanes + 32 * ch, w);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[TB_SREADY]);
    };
    bool ok = true;
    const bool kda = KDA;
    float* gv = reinterpret_cast<float*>(sm + TXO_GAM) + 64 * warp;
    put_s();
    for (int i = 0; ok && i < nloc; ++i) {
      const int b = i & 1;
      // (fused: the decay vectors in ring slot i % 3)
      const float* cvs = reinterpret_cast<const float*>(
          FUSED ? sm + TXO_PC + (i % 3) * PC_SLOT + PC_CV
                : sm + b * TX_STAGE + TX_CV);
      ok = __all_sync(0xffffffffu,
                      ok && mbar_wait(&bars[TB_FULLC0 + b], (i >> 1) & 1, abort_flag) &&
                          (!FUSED || mbar_wait(&pcbars[i % 3], (i / 3) & 1, abort_flag)));
      if (!ok) break;


      if (kda) {
        // this warp's half of gamma (per key channel) out of the stage
        // before it is released; read back in the state update below
        gv[lane] = cvs[CV_GAMMA + 64 * ch + lane];
        gv[lane + 32] = cvs[CV_GAMMA + 64 * ch + 32 + lane];
        __syncwarp();
      }
      const float gam = cvs[CV_GAMMA];
      // K -> K_d in place while the [-W;Q] product runs (the stage is
      // released only after the products that read K_d have completed);
      // KDA's K_d arrives as an image
      if (!kda) tx_scale_rows(sm + b * TX_STAGE + TX_K, 8192, cvs + CV_DEC, tid);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[TB_EMPTYC0 + b]);
        if (FUSED) mbar_arrive(&pcbars[3 + i % 3]);
      }
      // U^T (fp32, accumulator columns 32 ch ..: tokens) -> bf16 pairs, over
      // chunk i - 1's, which P U has read
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&bars[TB_D1FULL0 + b], (i >> 1) & 1, abort_flag) &&
                          (!emit || i == 0 ||
                           mbar_wait(&bars[TB_OFULL0 + (b ^ 1)], ((i - 1) >> 1) & 1,
                                     abort_flag)));
      if (!ok) break;
      // Fused: the [-W;Q] product of chunk i has completed, so every part of
      // the chunk has landed (T_U and -W included): the preparation CTA may
      // refill its ring slot (LANDED barrier i % 4). (Waiting on the
      // chunk's own full barriers here instead could see them two phases
      // on.)
      if (FUSED && tid == 0)
        mbar_arrive_cluster(map_to_cta(
            sm + FP_BAR + 8 * (FB_LANDED + (c_begin + i) % kRingSlots), prep));
      tc_fence_after();
      {
        float u[32];
        tmem_ldn<32>(tmem + TX_D1 + 128 * b + lanes + 32 * ch, u);
        tmem_ld_wait();
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) w[c] = pack_bf16x2(u[2 * c], u[2 * c + 1]);
        tmem_st16(tmem + TX_UB + lanes + 16 * ch, w);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[TB_UREADY]);

      // S <- gamma S + Delta^T
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[TB_D2FULL], i & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      {
        float d[32];
        tmem_ldn<32>(tmem + TX_D2 + lanes + 64 * ch, d);
        tmem_ld_wait();
        if (kda) {
#pragma unroll
          for (int c = 0; c < 32; ++c) S[c] = fmaf(gv[c], S[c], d[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) S[c] = fmaf(gam, S[c], d[c]);
        }
        tmem_ldn<32>(tmem + TX_D2 + lanes + 64 * ch + 32, d);
        tmem_ld_wait();
        if (kda) {
#pragma unroll
          for (int c = 0; c < 32; ++c) S[32 + c] = fmaf(gv[32 + c], S[32 + c], d[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) S[32 + c] = fmaf(gam, S[32 + c], d[c]);
        }
      }
      put_s();
    }
    if (ok && live && live_cols && !*abort_flag) {
      if (p.mode == kModeSplit) {
        float* dst = nullptr;
        if (part == 0) {
          if (p.parts > 1) dst = p.ws_start + ((nh * p.parts + 1) * dv + r) * dkr;
        } else {
          dst = p.ws_end +
                ((nh * p.parts + part) * (dv + dkr) + (scale_rows ? dv : 0) + r) * dkr;
        }
        if (dst) {
          float4* d4 = reinterpret_cast<float4*>(dst + 64 * ch);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            d4[c] = make_float4(S[4 * c], S[4 * c + 1], S[4 * c + 2], S[4 * c + 3]);
        }
      } else if (p.hT && part == p.parts - 1) {
        float* dst = p.hT + (nh * dkr + 64 * ch) * dv + r;
#pragma unroll
        for (int c = 0; c < 64; ++c) dst[(size_t)c * dv] = S[c];
      }
    }
  } else if (warp < kTxThreads / 32) {
    // ================= output =================
    // Thread o of 128 (warp 8 + (warp & 3), TMEM lane quarter warp & 3) owns
    // row r of O^T, i.e. output column r of the chunk's 64 tokens.
    const int o = tid - kTxChainThreads;
    const int r = 32 * (warp & 3) + lane;
    const uint32_t lanes = (uint32_t)(32 * (warp & 3)) << 16;
    const float wr = (epi && p.norm_w && r < dv) ? p.norm_w[r] : 1.f;
    float* red = reinterpret_cast<float*>(sm + TXO_RED);
    float* rs = reinterpret_cast<float*>(sm + TXO_RS);
    auto gate_load = [&](int j) {  // gate tile of chunk j into output tile j & 1
      const int tok = (int)(bos + (long long)(c_begin + j) * C);
      uint8_t* ob = sm + TXO_OUT + (j & 1) * 16384;
      uint64_t* gb = &bars[TB_GATE0 + (j & 1)];
      mbar_arrive_expect_tx(gb, 128u * dv);
      tma_load_3d(ob, &tmg, gb, 0, h, tok);
      if (dv > 64) tma_load_3d(ob + 8192, &tmg, gb, 64, h, tok);
    };
    bool ok = true;
    if (emit) {
      // H^T columns of both accumulators start at zero ([-W;Q] accumulates
      // onto them); each is then free for its first U0^T
      uint32_t z[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) z[c] = 0u;
#pragma unroll
      for (int bb = 0; bb < 2; ++bb) {
        tmem_st32(tmem + TX_D1 + 128 * bb + 64 + lanes, z);
        tmem_st32(tmem + TX_D1 + 128 * bb + 96 + lanes, z);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[TB_D1FREE0]);
        mbar_arrive(&bars[TB_D1FREE1]);
      }
    }
    if (has_gate && o == 0 && nloc > 0) gate_load(0);
    for (int i = 0; ok && i < nloc; ++i) {
      const int b = i & 1;
      if (!emit) {
        // nothing to read out: only release the chunk's last stage group
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&bars[TB_FULLC0 + b], (i >> 1) & 1, abort_flag));
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[TB_EMPTYC0 + b]);
        continue;
      }
      const long long t0 = bos + (long long)(c_begin + i) * C;
      const int len = (int)min((long long)C, eos - t0);
      // (all output threads decide alike: they meet at named barriers)
      ok = bar_and(5, kTxOutThreads,
                   (FUSED ? mbar_wait(&pcbars[i % 3], (i / 3) & 1, abort_flag)
                          : mbar_wait(&bars[TB_FULLC0 + b], (i >> 1) & 1, abort_flag)) &&
                       mbar_wait(&bars[TB_OFULL0 + b], (i >> 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      // O^T = H^T diag(e^G) + U^T P^T, 32 tokens at a time (fused: the
      // decay vectors in ring slot i % 3)
      const float* eg = reinterpret_cast<const float*>(
                            FUSED ? sm + TXO_PC + (i % 3) * PC_SLOT + PC_CV
                                  : sm + b * TX_STAGE + TX_CV) + CV_EG;
      float y[64];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float hv[32];
        tmem_ldn<32>(tmem + TX_D1 + 128 * b + 64 + 32 * hh + lanes, hv);
        tmem_ldn<32>(tmem + TX_D1 + 128 * b + 32 * hh + lanes,
                     *reinterpret_cast<float(*)[32]>(&y[32 * hh]));
        tmem_ld_wait();
#pragma unroll
        for (int t4 = 0; t4 < 8; ++t4) {
          const float4 e4 = reinterpret_cast<const float4*>(eg + 32 * hh)[t4];
          float* yy = y + 32 * hh + 4 * t4;
          yy[0] = fmaf(e4.x, hv[4 * t4], yy[0]);
          yy[1] = fmaf(e4.y, hv[4 * t4 + 1], yy[1]);
          yy[2] = fmaf(e4.z, hv[4 * t4 + 2], yy[2]);
          yy[3] = fmaf(e4.w, hv[4 * t4 + 3], yy[3]);
        }
      }
      {
        // H^T back to zero for the accumulator's next chunk
        uint32_t z[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) z[c] = 0u;
        tmem_st32(tmem + TX_D1 + 128 * b + 64 + lanes, z);
        tmem_st32(tmem + TX_D1 + 128 * b + 96 + lanes, z);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[TB_D1FREE0 + b]);
        // e^G has been read (fused: from ring slot i % 3)
        mbar_arrive(FUSED ? &pcbars[3 + i % 3] : &bars[TB_EMPTYC0 + b]);
      }
      if (epi && p.norm_w) {
        // sum over the 128 rows of O^T (a token's d_v values) of y^2: a
        // transposing butterfly leaves lane l the warp's sums of tokens
        // tb(l) and tb(l) + 1, then the four warps add up in shared memory
        float x[64];
#pragma unroll
        for (int t = 0; t < 64; ++t) x[t] = y[t] * y[t];
#pragma unroll
        for (int w = 32, m = 16; m >= 1; w >>= 1, m >>= 1) {
          const bool up = (lane & m) != 0;
#pragma unroll
          for (int j = 0; j < w; ++j) {
            const float give = up ? x[j] : x[j + w];
            const float keep = up ? x[j + w] : x[j];
            x[j] = keep + __shfl_xor_sync(0xffffffffu, give, m);
          }
        }
        const int tb = ((lane & 16) ? 32 : 0) + ((lane & 8) ? 16 : 0) +
                       ((lane & 4) ? 8 : 0) + ((lane & 2) ? 4 : 0) +
                       ((lane & 1) ? 2 : 0);
        red[(warp & 3) * 64 + tb] = x[0];
        red[(warp & 3) * 64 + tb + 1] = x[1];
        named_bar(5, kTxOutThreads);
        if (o < 64)
          rs[o] = rsqrtf((red[o] + red[64 + o] + red[128 + o] + red[192 + o]) *
                             (1.f / (float)dv) + p.eps);
        named_bar(5, kTxOutThreads);
#pragma unroll
        for (int t = 0; t < 64; ++t) y[t] *= rs[t] * wr;
      }
      uint8_t* ob = sm + TXO_OUT + b * 16384;
      if (has_gate) {
        ok = bar_and(5, kTxOutThreads,
                     mbar_wait(&bars[TB_GATE0 + b], (i >> 1) & 1, abort_flag));
        if (!ok) break;
#pragma unroll
        for (int t = 0; t < 64; ++t)
          y[t] *= sigmoid_approx(__bfloat162float(
              *reinterpret_cast<const __nv_bfloat16*>(ob + tx_tile_off(t, r))));
      }
      // (the tile's previous store, chunk i - 2, was read out before the
      // barrier at the top of this iteration)
      if (len == C) {
        // through the tile (column r of its rows) and one TMA store
#pragma unroll
        for (int t = 0; t < 64; ++t)
          *reinterpret_cast<__nv_bfloat16*>(ob + tx_tile_off(t, r)) =
              __float2bfloat16_rn(y[t]);
        fence_proxy_async();
        named_bar(5, kTxOutThreads);
        if (o == 0) {
          tma_store_3d(&tmo, ob, 0, h, (int)t0);
          if (dv > 64) tma_store_3d(&tmo, ob + 8192, 64, h, (int)t0);
          bulk_commit();
        }
      } else if (r < dv) {
        // a partial chunk (the end of a sequence): directly, column r
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) +
                             ((size_t)t0 * H + h) * dv + r;
#pragma unroll
        for (int t = 0; t < 64; ++t)
          if (t < len) dst[(size_t)t * H * dv] = __float2bfloat16_rn(y[t]);
      }
      // the other tile's store (chunk i - 1) read out before the next
      // iteration writes into it; then the gate of chunk i + 1 into it
      if (o == 0) bulk_wait_read_1();
      if (has_gate && o == 0 && i + 1 < nloc) gate_load(i + 1);
    }
    if (o == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  // fused: the preparation CTA's pushes into this CTA have all landed (or
  // this CTA gave up on them), and neither CTA leaves before the other's
  // last remote write
  if (FUSED) cluster_sync();
  if (warp == kTxWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
  if (tid == 0 && *abort_flag) record_status(p.status, GDN_ERR_TIMEOUT);
}

template <bool KDA>
__global__ void __launch_bounds__(kTxThreads, 1)
    chain_tx_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap tmq,
                    const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv,
                    const __grid_constant__ CUtensorMap tmo,
                    const __grid_constant__ CUtensorMap tmg, int nch_dense,
                    int tiles) {
  chain_tx_body<KDA, false>(p, tmq, tmk, tmv, tmo, tmg, nch_dense, tiles,
                            blockIdx.x, blockIdx.y, blockIdx.z, 0);
}

// The fused kernel's block: the chain CTA's fifteen warps and one more,
// idle there; in the preparation CTA twelve compute warps (three groups of
// four), a loader warp per group and one warp that copies the outboxes.
constexpr int kFusedThreads = 16 * 32;

// fused_chunk_kernel: the whole forward pass with no workspace. A cluster
// of four CTAs serves two (sequence, head) pairs u = 2c and 2c + 1: ranks 0
// and 1 prepare every chunk of pair 2c + rank (prep_role) and push -W, P,
// T_U and the decay vectors into the stages of ranks 2 and 3, which run the
// whole-state chains and write the outputs (chain_tx_body). The two
// preparation CTAs share a TPC and so do the two chains: a chain whose TPC
// neighbour runs a preparation measured about twice as slow per chunk (and
// the preparation too) as one beside another chain. Grid (4 ceil(N H / 2)),
// cluster (4, 1, 1); one sub-sequence (no split). A rank with no pair (odd
// N H) only meets the others at the cluster barriers.
template <int VARIANT>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_chunk_kernel(const ChunkParams p,
                       const __grid_constant__ CUtensorMap tmq,
                       const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv,
                       const __grid_constant__ CUtensorMap tmo,
                       const __grid_constant__ CUtensorMap tmg) {
  const uint32_t rank = cluster_ctarank();
  const long long u = 2ll * (blockIdx.x >> 2) + (rank & 1);
  if (u >= (long long)p.N * p.H) {
    cluster_sync();
    cluster_sync();
    return;
  }
  const int n = (int)(u / p.H), h = (int)(u - (long long)n * p.H);
  if (rank < 2)
    prep_role<VARIANT>(p, tmk, tmq, n, h, rank + 2);
  else
    chain_tx_body<false, true>(p, tmq, tmk, tmv, tmo, tmg, 1, 1, 0, h, n,
                               rank - 2);
}


// ---------------------------------------------------------------------------
// Self-test: D = A * B (x2 when twice) with the layouts above, one CTA.
// N = 64 or 128 (an N-major B of 128 columns is two 64-column blocks).
// a_mn: 0 A K-major in shared memory, 1 M-major, 2 A in TMEM (bf16 pairs in
// columns 128 .. 128 + K / 2, written with tcgen05.st).
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
    tmem_alloc(slot, 256);
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
  for (int idx = tid; a_mn != 2 && idx < 128 * K; idx += 128) {
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
  if (a_mn == 2) {
    // row tid of A into this thread's lane (warp w owns lanes 32 w ..)
    for (int c0 = 0; c0 < K / 2; c0 += 32) {
      uint32_t u[32];
#pragma unroll
      for (int j = 0; j < 32; ++j)
        u[j] = pack_bf16x2(__bfloat162float(A[tid * K + 2 * (c0 + j)]),
                           __bfloat162float(A[tid * K + 2 * (c0 + j) + 1]));
      tmem_st32(tmem + ((uint32_t)(32 * warp) << 16) + 128 + c0, u);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (tid == 0) {
    const uint32_t id = idesc_bf16(128, N, a_mn == 1, b_mn != 0);
    for (int pass = 0; pass <= (twice ? 1 : 0); ++pass)
      for (int s = 0; s < K / 16; ++s) {
        const uint64_t a =
            a_mn ? sdesc(base + s * 2048, K * 128, 1024)
                 : sdesc(base + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024);
        const uint64_t b =
            b_mn ? sdesc(base + 32768 + s * 2048, K * 128, 1024)
                 : sdesc(base + 32768 + (s >> 2) * bstride + (s & 3) * 32, 16, 1024);
        if (a_mn == 2)
          mma_bf16_ta(tmem, tmem + 128 + 8 * s, b, id, (pass > 0 || s > 0) ? 1u : 0u);
        else
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
    tmem_dealloc(tmem, 256);
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

// 3-D bf16 map, dims (d0, d1, d2) with d0 contiguous, box (64, b1, b2),
// 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* ptr, long long d0, long long d1,
              long long d2, uint32_t b1, uint32_t b2) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  cuuint64_t strides[2] = {(cuuint64_t)d0 * 2, (cuuint64_t)d0 * d1 * 2};
  cuuint32_t box[3] = {64, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr),
             dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

long long call_tokens(const ChunkParams& p) {
  return p.cu_seqlens ? (long long)p.T : (long long)p.N * p.T;
}

int sm_count() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) ==
          cudaSuccess &&
      v > 0)
    return v;
  return 148;
}

}  // namespace

bool make_rows_map(CUtensorMap* map, const void* ptr, bool fp32, long long d0,
                   long long d1, long long d2, uint32_t b0, uint32_t b2) {
  auto enc = encode_fn();
  if (!enc) return false;
  const long long es = fp32 ? 4 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  cuuint64_t strides[2] = {(cuuint64_t)(d0 * es), (cuuint64_t)(d0 * d1 * es)};
  cuuint32_t box[3] = {b0, 1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map,
             fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
             3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool chunk_tc_supported(int dk, int dv, long long tokens, int N, int H) {
  // chunk-tile indices (chunk * H + head) and token rows stay in int
  // d_k = 64: the d_k = 128 kernels with K and Q zero-filled to 128
  return (dk == DK || dk == 64) && (dv == 64 || dv == 128) && tokens > 0 &&
         tokens < (1ll << 31) - 64 &&
         (tokens / C + N + 1) * (long long)H < (1ll << 31);
}

int chunk_tc_nch_dense(const ChunkParams& p) { return (p.T + C - 1) / C; }

long long chunk_tc_chunks_bound(const ChunkParams& p) {
  // packed: sum of ceil(len / C) <= T / C + N
  return p.cu_seqlens ? (long long)(p.T + C - 1) / C + p.N
                      : (long long)p.N * chunk_tc_nch_dense(p);
}

size_t chunk_tc_workspace_bytes(const ChunkParams& p) {
  const size_t tiles = (size_t)chunk_tc_chunks_bound(p) * p.H;
  size_t bytes = tiles * (WS_W_BYTES + WS_P_BYTES + WS_TU_BYTES +
                          (p.kda ? KCV_BYTES + WS_QG_BYTES + WS_KD_BYTES
                                 : CV_BYTES));
  if (p.cu_seqlens) bytes += ((size_t)p.N + 1) * sizeof(int32_t) + 256;
  return bytes;
}

void chunk_tc_bind_workspace(ChunkParams& p, void* ws) {
  const size_t tiles = (size_t)chunk_tc_chunks_bound(p) * p.H;
  char* c = static_cast<char*>(ws);
  p.wneg = c;
  c += tiles * WS_W_BYTES;
  p.pm = c;
  c += tiles * WS_P_BYTES;
  p.tu = c;
  c += tiles * WS_TU_BYTES;
  p.cv = reinterpret_cast<float*>(c);
  c += tiles * (p.kda ? KCV_BYTES : CV_BYTES);
  if (p.kda) {
    p.qg = c;
    c += tiles * WS_QG_BYTES;
    p.kd = c;
    c += tiles * WS_KD_BYTES;
  }
  p.chunk_off = p.cu_seqlens ? reinterpret_cast<int32_t*>(c) : nullptr;
}

// Chunk offsets of packed calls (nothing for dense ones).
cudaError_t launch_chunk_offsets(const ChunkParams& p, cudaStream_t stream,
                                 int* launches) {
  *launches = 0;
  if (!p.cu_seqlens) return cudaSuccess;
  const int t = timing_start(GDN_KERNEL_CHUNK_OFFSETS, stream);
  chunk_offsets_kernel<<<1, 1024, 0, stream>>>(
      p.cu_seqlens, p.N, p.T, C, const_cast<int32_t*>(p.chunk_off), p.status);
  cudaError_t e = cudaGetLastError();
  timing_stop(t, stream, e);
  if (e == cudaSuccess) ++*launches;
  return e;
}

// Prefix of ceil(len / L) over the packed sequences (one CTA).
cudaError_t launch_block_offsets(const int32_t* cu_seqlens, int N, int T,
                                 int L, int32_t* out, int* status,
                                 cudaStream_t stream) {
  const int t = timing_start(GDN_KERNEL_CHUNK_OFFSETS, stream);
  chunk_offsets_kernel<<<1, 1024, 0, stream>>>(cu_seqlens, N, T, L, out, status);
  cudaError_t e = cudaGetLastError();
  timing_stop(t, stream, e);
  return e;
}

// Chunk offsets (packed calls) and the preparation of every chunk.
cudaError_t launch_ut_prep(const ChunkParams& p, cudaStream_t stream,
                           int* launches) {
  cudaError_t e0 = launch_chunk_offsets(p, stream, launches);
  if (e0 != cudaSuccess) return e0;
  CUtensorMap mk, mq;
  if (!make_map(&mk, p.k, p.dk, p.H, call_tokens(p), 1, 64) ||
      !make_map(&mq, p.q, p.dk, p.H, call_tokens(p), 1, 64))
    return cudaErrorInvalidValue;
  const long long bound = chunk_tc_chunks_bound(p);
  const long long items = bound * p.H;
  const int grid = (int)std::min<long long>(items, (long long)kPrepCtas * sm_count());
  const int nchd = chunk_tc_nch_dense(p);
  // A workspace that fits the L2 well is written with an evict-last hint,
  // so that the chain kernel right behind finds its first chunks' -W, P and
  // T_U there rather than in HBM (on a larger one the hint would only push
  // out lines still to be read).
  const int keep_ws =
      items * (long long)(WS_W_BYTES + WS_P_BYTES + WS_TU_BYTES) <= kKeepWsBytes;
  auto launch = [&](auto kern) {
    cudaError_t e = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PR_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int t = timing_start(GDN_KERNEL_CHUNK_PREP, stream);
    kern<<<grid, kPrepThreads, PR_SMEM_BYTES, stream>>>(p, mk, mq, nchd,
                                                         (int)bound, keep_ws);
    e = cudaGetLastError();
    timing_stop(t, stream, e);
    return e;
  };
  cudaError_t e = p.variant == GDN_GATE_AFTER_PREDICT
                      ? launch(ut_prep_kernel<GDN_GATE_AFTER_PREDICT>)
                      : launch(ut_prep_kernel<GDN_GATE_BEFORE_PREDICT>);
  if (e == cudaSuccess) ++*launches;
  return e;
}

size_t fused_ring_bytes(const ChunkParams& p) {
  return (size_t)p.N * p.H * kRingSlots * FP_OB_BYTES;
}

// The fused single-kernel path: per two (sequence, head) pairs a cluster of
// two preparation and two chain CTAs, handing chunks over through a ring in
// global memory (p.ring, fused_ring_bytes; one sub-sequence; dense or
// packed).
cudaError_t launch_chunk_fused(const ChunkParams& p, cudaStream_t stream) {
  const long long tokens = call_tokens(p);
  CUtensorMap mq, mk, mv, mo, mg;
  if (!make_map(&mq, p.q, p.dk, p.H, tokens, 1, 64) ||
      !make_map(&mk, p.k, p.dk, p.H, tokens, 1, 64) ||
      !make_map(&mv, p.v, p.dv, p.H, tokens, 1, 64) ||
      !make_map(&mo, p.out, p.dv, p.H, tokens, 1, 64) ||
      !make_map(&mg, p.gate_z ? p.gate_z : p.out, p.dv, p.H, tokens, 1, 64))
    return cudaErrorInvalidValue;
  auto launch = [&](auto kern) {
    cudaError_t e = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)FUSED_SMEM);
    if (e != cudaSuccess) return e;
    const int t = timing_start(GDN_KERNEL_CHUNK_FUSED, stream);
    cudaLaunchConfig_t cfg{};
    const long long pairs = ((long long)p.N * p.H + 1) / 2;
    cfg.gridDim = dim3((unsigned)(4 * pairs), 1, 1);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = FUSED_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 4;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p, mq, mk, mv, mo, mg);
    if (e == cudaSuccess) e = cudaGetLastError();
    timing_stop(t, stream, e);
    return e;
  };
  return p.variant == GDN_GATE_AFTER_PREDICT
             ? launch(fused_chunk_kernel<GDN_GATE_AFTER_PREDICT>)
             : launch(fused_chunk_kernel<GDN_GATE_BEFORE_PREDICT>);
}

// One pass of the chain kernel (after launch_ut_prep on the same stream).
cudaError_t launch_chunk_tc(const ChunkParams& p, cudaStream_t stream) {
  const long long tokens = call_tokens(p);
  const long long tiles = chunk_tc_chunks_bound(p) * p.H;
  CUtensorMap mq, mk, mv, mo, mg;
  if (!make_map(&mq, p.q, p.dk, p.H, tokens, 1, 64) ||
      !make_map(&mk, p.k, p.dk, p.H, tokens, 1, 64) ||
      !make_map(&mv, p.v, p.dv, p.H, tokens, 1, 64) ||
      !make_map(&mo, p.out, p.dv, p.H, tokens, 1, 64) ||
      !make_map(&mg, p.gate_z ? p.gate_z : p.out, p.dv, p.H, tokens, 1, 64))
    return cudaErrorInvalidValue;
  const int nchd = chunk_tc_nch_dense(p);
  if (p.chain_rows == TXR) {
    // one CTA per 128 state rows: the value rows, and in a split pass the
    // rows of the scaling matrix
    auto kern = p.kda ? chain_tx_kernel<true> : chain_tx_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TX_SMEM);
    if (e != cudaSuccess) return e;
    const int blocks = p.mode == kModeSplit ? 2 : 1;
    const int t = timing_start(GDN_KERNEL_CHUNK_CHAIN_WHOLE, stream);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(blocks, p.H, p.N * p.part_count);
    cfg.blockDim = dim3(kTxThreads);
    cfg.dynamicSmemBytes = TX_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p, mq, mk, mv, mo, mg, nchd,
                           (int)tiles);
    if (e == cudaSuccess) e = cudaGetLastError();
    timing_stop(t, stream, e);
    return e;
  }
  // the fused epilogue's RMS normalisation pairs the two CTAs of each
  // (sequence, head, part) when d_v = 128 (grid.x is then 2 or 4); the
  // output gate alone needs no partner
  const bool clustered = p.epilogue && p.norm_w && p.dv == 128;
  auto launch = [&](auto kern) {
    cudaError_t e = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int rows = p.mode == kModeSplit ? p.dv + p.dk : p.dv;
    dim3 grid(rows / DVT, p.H, p.N * p.part_count);
    const int t = timing_start(GDN_KERNEL_CHUNK_CHAIN, stream);
    // programmatic stream serialisation: the launch may begin while the
    // preceding kernel drains; the kernel waits for it in griddep_wait
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = clustered ? 2 : 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = clustered ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, p, mq, mk, mv, mo, mg, nchd, (int)tiles);
    if (e == cudaSuccess) e = cudaGetLastError();
    timing_stop(t, stream, e);
    return e;
  };
  return p.variant == GDN_GATE_AFTER_PREDICT
             ? (p.epilogue ? launch(chunk_tc_kernel<GDN_GATE_AFTER_PREDICT, true>)
                           : launch(chunk_tc_kernel<GDN_GATE_AFTER_PREDICT, false>))
             : (p.epilogue ? launch(chunk_tc_kernel<GDN_GATE_BEFORE_PREDICT, true>)
                           : launch(chunk_tc_kernel<GDN_GATE_BEFORE_PREDICT, false>));
}

}  // namespace gdn

extern "C" int gdn_selftest_mma(const void* A, const void* B, float* D, int K,
                                int N, int a_mn, int b_mn, int b_stacked,
                                int twice, gdn_stream_t stream) {
  using namespace gdn;
  if (!A || !B || !D || (K != 64 && K != 128) || (N != 64 && N != 128))
    return GDN_ERR_INVALID_ARG;
  if (b_stacked && N != 64) return GDN_ERR_INVALID_ARG;
  if (a_mn < 0 || a_mn > 2) return GDN_ERR_INVALID_ARG;
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

