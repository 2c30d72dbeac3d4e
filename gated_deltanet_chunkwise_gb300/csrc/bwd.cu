// Backward pass of the delta rule with a decay before the prediction (the
// scalar gate of Gated DeltaNet, or KDA's per-channel decay), token by token
// with recomputation from checkpointed states.
//
// Illustrated DeltaNet walk-through (cost table and memory paragraphs: a
// chunked model stores only the state at chunk boundaries and recomputes
// the rest for the gradient) and the lqnn.cn page (block recompute in the
// section on the chunk form). One token of the forward map,
//   S_bar = S diag(a_t), a_t = e^{g_t};  e = v_t - S_bar k_t;  u = beta_t e;
//   S_t = S_bar + u k_t^T;  o_t = S_t q_t,
// has, for the gradient dS arriving at S_t and do_t, the adjoint
//   dq_t = S_t^T do_t;  dS += do_t q_t^T;  du = dS k_t;
//   dk_t = dS^T u - beta_t S_bar^T du;  dbeta_t = du . e;  dv_t = beta_t du;
//   dS_bar = dS - beta_t du k_t^T;  dg_t = colsum(dS_bar (.) S_bar);
//   dS_{t-1} = dS_bar diag(a_t).
//
// Rows of the state (value coordinates) never mix in either direction, so
// the work spreads over (32-row blocks, heads, sequences) exactly as in the
// token-serial forward kernel: 8 warps of 4 rows, each lane d_k / 32 key
// channels of its 4 rows. Pass 1 runs the forward map and stores the state
// at the start of every 16-token block (the checkpoints). Pass 2 walks the
// blocks backwards: it recomputes the block from its checkpoint, keeping
// S_bar of each token in a per-CTA window (global memory, 256 KB per CTA,
// meant to stay in L2) and e in shared memory, then runs the adjoint over
// the block's tokens in reverse. The sums over rows (dq, dk, dg, dbeta) meet
// in shared memory once per token (each warp's partial in its own slot, then
// a fixed-order sum, so the result does not depend on warp timing) and leave
// as one partial per row block; a second kernel adds the row blocks' partials
// (and, for the scalar gate, the channels of dg).
//
// With the other gate placement (predict with the undecayed state S, then
// decay: S_t = S diag(a_t) + u k_t^T) the window keeps S instead of S_bar and
// the adjoint's last steps become dk_t = dS^T u - beta_t S^T du, dg_t =
// colsum(dS (.) S diag(a_t)), dS_{t-1} = dS diag(a_t) - beta_t du k_t^T.
#include <functional>
#include <type_traits>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kBwRpw = 4;                  // state rows per warp (per thread)
constexpr int kBwRows = 8 * kBwRpw;        // state rows per CTA
constexpr int kBwThreads = 256;
constexpr int kBwTok = 16;                 // tokens per block (checkpoint spacing)

struct BwdArgs {
  const void* q;          // bf16 or fp32 (the kernel's input type), as k, v, dout
  const void* k;
  const void* v;
  const float* g;         // [tokens, H, dk] (per channel) or [tokens, H]
  const float* beta;      // [tokens, H]
  const float* h0;        // [N, H, dk, dv] or null
  const void* dout;       // [tokens, H, dv]
  const float* dhT;       // [N, H, dk, dv] or null
  float* dv_out;          // [tokens, H, dv]
  float* dh0;             // [N, H, dk, dv] or null
  float* part;            // [3][RB][tokens * H][dk]: dq, dk, dg per row block
  float* part_b;          // [RB][tokens * H]: dbeta per row block
  float* ckpt;            // [blocks of 16 tokens][H][RB][256 threads x 4 * CPT]
  float* win;             // [N][H][RB][16 tokens][256 threads x 4 * CPT]
  const int32_t* cu_seqlens;
  const int32_t* blk_off;  // [N + 1] first 16-token block of each sequence
  int N, H, T, dv, g_chan;  // g_chan: dk (per channel) or 1 (scalar gate)
  int decay_first;          // 1: decay, then predict; 0: predict, then decay
  long long rows;           // tokens * H
  int* status;
  int passes;               // 1: forward sweep, 2: reverse sweep, 3: both
  float* o_out;             // [tokens, H, dv] fp32: o_t from the forward sweep, or null
};

__device__ __forceinline__ void unpack8(uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <int N>
__device__ __forceinline__ void ld_slice(const float* p, float (&x)[N]) {
  if constexpr (N == 4) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else {
    const float2 v = *reinterpret_cast<const float2*>(p);
    x[0] = v.x; x[1] = v.y;
  }
}

// The warp's sums of x[r] over its lanes for its 4 rows: lane l ends with
// row l / 8's sum (transposing butterfly: two halving exchanges, then three
// adds within groups of 8 lanes).
__device__ __forceinline__ float rowsum4(float (&x)[kBwRpw], int lane) {
#pragma unroll
  for (int nv = kBwRpw, off = 16; nv > 1; nv >>= 1, off >>= 1) {
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
  for (int off = 4; off >= 1; off >>= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
  return y;
}

// Shared-memory layout (floats) of the backward kernel for a given d_k.
template <int DK>
struct BwSmem {
  static constexpr int SK = 0, SQ = SK + kBwTok * DK, SA = SQ + kBwTok * DK,
                       SV = SA + kBwTok * DK, SDO = SV + kBwTok * kBwRows,
                       SE = SDO + kBwTok * kBwRows, SDV = SE + kBwTok * kBwRows,
                       SB = SDV + kBwTok * kBwRows;
  // one warp's partial: dq, dk, dg, dbeta (padded to 16-byte rows)
  static constexpr int RW = 3 * DK + 4;
  static constexpr int SLOT = SB + kBwTok, ACC = SLOT + 2 * 8 * RW,
                       TOTAL = ACC + kBwTok * RW;
};

// TI: the type of q, k, v and dout (bf16, or fp32 for gdn_chunk_bwd_f32;
// fp32 rows are staged straight from global memory, bf16 rows one block
// ahead through registers)
template <int DK, typename TI>
__global__ void __launch_bounds__(kBwThreads, 2) bwd_kernel(const BwdArgs a) {
  constexpr bool kF32 = std::is_same<TI, float>::value;
  const TI* gq = static_cast<const TI*>(a.q);
  const TI* gk = static_cast<const TI*>(a.k);
  const TI* gv = static_cast<const TI*>(a.v);
  const TI* gdo = static_cast<const TI*>(a.dout);
  constexpr int CPT = DK / 32;            // channels per lane
  constexpr int NS = kBwRpw * CPT;        // state floats per thread
  using L = BwSmem<DK>;
  static_assert(L::SLOT % 4 == 0 && L::RW % 4 == 0 && L::SDO % 4 == 0 &&
                    L::SE % 4 == 0 && L::SA % 4 == 0,
                "16-byte shared-memory accesses");
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int rb = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int RB = gridDim.x, H = a.H, dv = a.dv;
  const int row0 = rb * kBwRows, a0 = row0 + kBwRpw * w;
  const int rr = lane >> 3;  // the row whose sums this lane ends up with
  long long bos, eos;
  if (a.cu_seqlens) {
    bos = a.cu_seqlens[n];
    eos = a.cu_seqlens[n + 1];
    if (bos < 0 || eos < bos || eos > a.T) {
      if (tid == 0) record_status(a.status, GDN_ERR_INVALID_ARG);
      return;
    }
  } else {
    bos = (long long)n * a.T;
    eos = bos + a.T;
  }
  const size_t nh = (size_t)n * H + h;
  const int nblk = (int)((eos - bos + kBwTok - 1) / kBwTok);
  const long long blk0 = a.blk_off ? a.blk_off[n] : (long long)n * ((a.T + kBwTok - 1) / kBwTok);
  // this CTA's checkpoint of block b and window slot of token tt (each
  // thread's NS floats contiguous)
  auto ckpt = [&](int b) {
    return a.ckpt + (((size_t)(blk0 + b) * H + h) * RB + rb) * (kBwThreads * NS) + tid * NS;
  };
  float* win = a.win + ((nh * RB + rb) * kBwTok) * (size_t)(kBwThreads * NS) + tid * NS;

  // ---- staging of a 16-token block --------------------------------------
  constexpr int KTOT = kBwTok * DK / 8, KCH = (KTOT + kBwThreads - 1) / kBwThreads;
  constexpr int GTOT = kBwTok * DK / 4, GCH = (GTOT + kBwThreads - 1) / kBwThreads;
  uint4 rk[KCH], rq[KCH], rv, rdo;
  float4 rg[GCH];
  float rbeta = 0.f;
  auto fetch = [&](long long t0, bool with_q, bool back) {
    const int nt = (int)max(0ll, min((long long)kBwTok, eos - t0));
#pragma unroll
    for (int j = 0; j < KCH; ++j) {
      const int e = tid + j * kBwThreads, tt = e / (DK / 8), c8 = e % (DK / 8);
      rk[j] = rq[j] = make_uint4(0, 0, 0, 0);
      if (!kF32 && e < KTOT && tt < nt) {
        const size_t r = ((size_t)(t0 + tt) * H + h) * DK + 8 * c8;
        rk[j] = *reinterpret_cast<const uint4*>(gk + r);
        if (with_q) rq[j] = *reinterpret_cast<const uint4*>(gq + r);
      }
    }
#pragma unroll
    for (int j = 0; j < GCH; ++j) {
      const int e = tid + j * kBwThreads, tt = e / (DK / 4), c4 = e % (DK / 4);
      rg[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < GTOT && tt < nt) {
        if (a.g_chan == 1) {
          const float x = a.g[(size_t)(t0 + tt) * H + h];
          rg[j] = make_float4(x, x, x, x);
        } else {
          rg[j] = *reinterpret_cast<const float4*>(a.g + ((size_t)(t0 + tt) * H + h) * DK + 4 * c4);
        }
      }
    }
    rv = rdo = make_uint4(0, 0, 0, 0);
    if (!kF32 && tid < kBwTok * kBwRows / 8) {
      const int tt = tid / (kBwRows / 8), r8 = tid % (kBwRows / 8);
      if (tt < nt) {
        const size_t r = ((size_t)(t0 + tt) * H + h) * dv + row0 + 8 * r8;
        rv = *reinterpret_cast<const uint4*>(gv + r);
        if (back) rdo = *reinterpret_cast<const uint4*>(gdo + r);
      }
    }
    if (tid < kBwTok) rbeta = tid < nt ? a.beta[(size_t)(t0 + tid) * H + h] : 0.f;
  };
  // 8 consecutive fp32 values (zeros past the block's end)
  auto ld8f = [&](const TI* src, bool live, float (&f)[8]) {
    if constexpr (kF32) {
      float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
      if (live) {
        x0 = *reinterpret_cast<const float4*>(src);
        x1 = *reinterpret_cast<const float4*>(src + 4);
      }
      f[0] = x0.x; f[1] = x0.y; f[2] = x0.z; f[3] = x0.w;
      f[4] = x1.x; f[5] = x1.y; f[6] = x1.z; f[7] = x1.w;
    }
  };
  auto stage = [&](long long t0, bool with_q, bool back) {
    const int nt = (int)max(0ll, min((long long)kBwTok, eos - t0));
#pragma unroll
    for (int j = 0; j < KCH; ++j) {
      const int e = tid + j * kBwThreads, tt = e / (DK / 8), c8 = e % (DK / 8);
      if (e >= KTOT) continue;
      float f[8];
      if constexpr (kF32) {
        const size_t r = ((size_t)(t0 + tt) * H + h) * DK + 8 * c8;
        ld8f(gk + r, tt < nt, f);
      } else {
        unpack8(rk[j], f);
      }
#pragma unroll
      for (int x = 0; x < 8; ++x) sm[L::SK + tt * DK + 8 * c8 + x] = f[x];
      if constexpr (kF32) {
        const size_t r = ((size_t)(t0 + tt) * H + h) * DK + 8 * c8;
        ld8f(gq + r, with_q && tt < nt, f);
      } else {
        unpack8(rq[j], f);
      }
#pragma unroll
      for (int x = 0; x < 8; ++x) sm[L::SQ + tt * DK + 8 * c8 + x] = f[x];
    }
#pragma unroll
    for (int j = 0; j < GCH; ++j) {
      const int e = tid + j * kBwThreads, tt = e / (DK / 4), c4 = e % (DK / 4);
      if (e >= GTOT) continue;
      *reinterpret_cast<float4*>(&sm[L::SA + tt * DK + 4 * c4]) =
          make_float4(expf(rg[j].x), expf(rg[j].y), expf(rg[j].z), expf(rg[j].w));
    }
    if (tid < kBwTok * kBwRows / 8) {
      const int tt = tid / (kBwRows / 8), r8 = tid % (kBwRows / 8);
      const size_t r = ((size_t)(t0 + tt) * H + h) * dv + row0 + 8 * r8;
      float f[8];
      if constexpr (kF32) ld8f(gv + r, tt < nt, f); else unpack8(rv, f);
#pragma unroll
      for (int x = 0; x < 8; ++x) sm[L::SV + tt * kBwRows + 8 * r8 + x] = f[x];
      if constexpr (kF32) ld8f(gdo + r, back && tt < nt, f); else unpack8(rdo, f);
#pragma unroll
      for (int x = 0; x < 8; ++x) sm[L::SDO + tt * kBwRows + 8 * r8 + x] = f[x];
    }
    if (tid < kBwTok) sm[L::SB + tid] = rbeta;
  };

  // ---- pass 1: the forward map, checkpointing every block ---------------
  float S[kBwRpw][CPT];
#pragma unroll
  for (int r = 0; r < kBwRpw; ++r)
#pragma unroll
    for (int j = 0; j < CPT; ++j)
      S[r][j] = a.h0 ? a.h0[(nh * DK + CPT * lane + j) * dv + a0 + r] : 0.f;
  auto put = [&](float* dst) {
#pragma unroll
    for (int r = 0; r < kBwRpw; ++r)
      if constexpr (CPT == 4)
        *reinterpret_cast<float4*>(dst + 4 * r) = make_float4(S[r][0], S[r][1], S[r][2], S[r][3]);
      else
        *reinterpret_cast<float2*>(dst + 2 * r) = make_float2(S[r][0], S[r][1]);
  };
  auto get = [&](const float* src, float (&X)[kBwRpw][CPT]) {
#pragma unroll
    for (int r = 0; r < kBwRpw; ++r) ld_slice<CPT>(src + CPT * r, X[r]);
  };
  const bool dfirst = a.decay_first != 0;
  // one forward token on S (registers); `save` receives the state the
  // prediction reads; returns e for row rr
  auto forward_token = [&](int tt, float* save) {
    float av[CPT], kv[CPT];
    ld_slice<CPT>(&sm[L::SA + tt * DK + CPT * lane], av);
    ld_slice<CPT>(&sm[L::SK + tt * DK + CPT * lane], kv);
    float p[kBwRpw];
#pragma unroll
    for (int r = 0; r < kBwRpw; ++r) {
      p[r] = 0.f;
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
        if (dfirst) S[r][j] *= av[j];
        p[r] = fmaf(S[r][j], kv[j], p[r]);
      }
    }
    if (save) put(save);
    const float pred = rowsum4(p, lane);
    const float e = sm[L::SV + tt * kBwRows + kBwRpw * w + rr] - pred;
    const float ur = sm[L::SB + tt] * e;
#pragma unroll
    for (int r = 0; r < kBwRpw; ++r) {
      const float u = __shfl_sync(0xffffffffu, ur, 8 * r);
#pragma unroll
      for (int j = 0; j < CPT; ++j)
        S[r][j] = fmaf(u, kv[j], dfirst ? S[r][j] : S[r][j] * av[j]);
    }
    return e;
  };
  const bool want_o = a.o_out != nullptr;
  if (a.passes & 1) {
    fetch(bos, want_o, false);
    for (int b = 0; b < nblk; ++b) {
      const long long t0 = bos + (long long)b * kBwTok;
      const int nt = (int)min((long long)kBwTok, eos - t0);
      __syncthreads();
      stage(t0, want_o, false);
      __syncthreads();
      if (b + 1 < nblk) fetch(t0 + kBwTok, want_o, false);
      put(ckpt(b));
      for (int tt = 0; tt < nt; ++tt) {
        forward_token(tt, nullptr);
        if (want_o) {
          // o_t = S_t q_t, this warp's rows
          float qv[CPT], p[kBwRpw];
          ld_slice<CPT>(&sm[L::SQ + tt * DK + CPT * lane], qv);
#pragma unroll
          for (int r = 0; r < kBwRpw; ++r) {
            p[r] = 0.f;
#pragma unroll
            for (int j = 0; j < CPT; ++j) p[r] = fmaf(S[r][j], qv[j], p[r]);
          }
          const float orow = rowsum4(p, lane);
          if ((lane & 7) == 0) sm[L::SDV + tt * kBwRows + kBwRpw * w + rr] = orow;
        }
      }
      if (want_o) {
        __syncthreads();
        for (int idx = tid; idx < nt * kBwRows; idx += kBwThreads) {
          const int tt = idx / kBwRows, r = idx - tt * kBwRows;
          a.o_out[((size_t)(t0 + tt) * H + h) * dv + row0 + r] =
              sm[L::SDV + tt * kBwRows + r];
        }
      }
    }
  }
  if (!(a.passes & 2)) return;

  // ---- pass 2: the blocks in reverse ------------------------------------
  float dS[kBwRpw][CPT];
#pragma unroll
  for (int r = 0; r < kBwRpw; ++r)
#pragma unroll
    for (int j = 0; j < CPT; ++j)
      dS[r][j] = a.dhT ? a.dhT[(nh * DK + CPT * lane + j) * dv + a0 + r] : 0.f;
  if (nblk > 0) fetch(bos + (long long)(nblk - 1) * kBwTok, true, true);
  for (int b = nblk - 1; b >= 0; --b) {
    const long long t0 = bos + (long long)b * kBwTok;
    const int nt = (int)min((long long)kBwTok, eos - t0);
    __syncthreads();  // the previous block's shared data has been written out
    stage(t0, true, true);
    __syncthreads();
    if (b > 0) fetch(t0 - kBwTok, true, true);
    // recompute the block: S_bar of each token into the window, e of each
    // row into shared memory
    get(ckpt(b), S);
    for (int tt = 0; tt < nt; ++tt) {
      const float e = forward_token(tt, win + (size_t)tt * (kBwThreads * NS));
      if ((lane & 7) == 0) sm[L::SE + tt * kBwRows + kBwRpw * w + rr] = e;
    }
    __syncwarp();
    // the adjoint, tokens in reverse
    for (int tt = nt - 1; tt >= 0; --tt) {
      float Sb[kBwRpw][CPT];
      get(win + (size_t)tt * (kBwThreads * NS), Sb);
      float av[CPT], kv[CPT], qv[CPT];
      ld_slice<CPT>(&sm[L::SA + tt * DK + CPT * lane], av);
      ld_slice<CPT>(&sm[L::SK + tt * DK + CPT * lane], kv);
      ld_slice<CPT>(&sm[L::SQ + tt * DK + CPT * lane], qv);
      const float bt = sm[L::SB + tt];
      float dor[kBwRpw], er[kBwRpw];
      ld_slice<kBwRpw>(&sm[L::SDO + tt * kBwRows + kBwRpw * w], dor);
      ld_slice<kBwRpw>(&sm[L::SE + tt * kBwRows + kBwRpw * w], er);
      float dq[CPT], dkk[CPT], dg[CPT], pdu[kBwRpw];
#pragma unroll
      for (int j = 0; j < CPT; ++j) dq[j] = dkk[j] = dg[j] = 0.f;
#pragma unroll
      for (int r = 0; r < kBwRpw; ++r) {
        const float u = bt * er[r];
        pdu[r] = 0.f;
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          const float st = fmaf(u, kv[j], dfirst ? Sb[r][j] : Sb[r][j] * av[j]);
          dq[j] = fmaf(st, dor[r], dq[j]);  // S_t^T do
          dS[r][j] = fmaf(dor[r], qv[j], dS[r][j]);
          pdu[r] = fmaf(dS[r][j], kv[j], pdu[r]);
        }
      }
      const float du_rr = rowsum4(pdu, lane);
      float dbeta = 0.f;
#pragma unroll
      for (int r = 0; r < kBwRpw; ++r) {
        const float du = __shfl_sync(0xffffffffu, du_rr, 8 * r);
        const float u = bt * er[r], bdu = bt * du;
        dbeta = fmaf(du, er[r], dbeta);
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          dkk[j] = fmaf(dS[r][j], u, dkk[j]);
          dkk[j] = fmaf(-bdu, Sb[r][j], dkk[j]);
          if (dfirst) {
            const float dsb = fmaf(-bdu, kv[j], dS[r][j]);
            dg[j] = fmaf(dsb, Sb[r][j], dg[j]);
            dS[r][j] = dsb * av[j];
          } else {
            const float ds = dS[r][j] * av[j];
            dg[j] = fmaf(ds, Sb[r][j], dg[j]);
            dS[r][j] = fmaf(-bdu, kv[j], ds);
          }
        }
      }
      if ((lane & 7) == 0) sm[L::SDV + tt * kBwRows + kBwRpw * w + rr] = bt * du_rr;
      // this warp's partial into its slot, then a fixed-order sum over the
      // eight warps (slots alternate between tokens: one barrier each)
      float* slot = sm + L::SLOT + (tt & 1) * 8 * L::RW + w * L::RW;
      auto st_slice = [&](float* dst, const float (&x)[CPT]) {
        if constexpr (CPT == 4)
          *reinterpret_cast<float4*>(dst) = make_float4(x[0], x[1], x[2], x[3]);
        else
          *reinterpret_cast<float2*>(dst) = make_float2(x[0], x[1]);
      };
      st_slice(slot + CPT * lane, dq);
      st_slice(slot + DK + CPT * lane, dkk);
      st_slice(slot + 2 * DK + CPT * lane, dg);
      if (lane == 0) slot[3 * DK] = dbeta;
      __syncthreads();
      const float* s0 = sm + L::SLOT + (tt & 1) * 8 * L::RW;
      for (int idx = tid; idx < 3 * DK + 1; idx += kBwThreads) {
        float acc = 0.f;
#pragma unroll
        for (int ww = 0; ww < 8; ++ww) acc += s0[ww * L::RW + idx];
        sm[L::ACC + tt * L::RW + idx] = acc;
      }
    }
    __syncthreads();
    // the block's row-block partials and its dv rows
    for (int idx = tid; idx < nt * 3 * DK; idx += kBwThreads) {
      const int tt = idx / (3 * DK), rem = idx - tt * (3 * DK), which = rem / DK,
                c = rem - which * DK;
      const size_t row = (size_t)(t0 + tt) * H + h;
      a.part[(((size_t)which * RB + rb) * a.rows + row) * DK + c] =
          sm[L::ACC + tt * L::RW + rem];
    }
    if (tid < nt)
      a.part_b[(size_t)rb * a.rows + (size_t)(t0 + tid) * H + h] =
          sm[L::ACC + tid * L::RW + 3 * DK];
    for (int idx = tid; idx < nt * kBwRows; idx += kBwThreads) {
      const int tt = idx / kBwRows, r = idx - tt * kBwRows;
      a.dv_out[((size_t)(t0 + tt) * H + h) * dv + row0 + r] = sm[L::SDV + tt * kBwRows + r];
    }
  }
  if (a.dh0) {
#pragma unroll
    for (int r = 0; r < kBwRpw; ++r)
#pragma unroll
      for (int j = 0; j < CPT; ++j)
        a.dh0[(nh * DK + CPT * lane + j) * dv + a0 + r] = dS[r][j];
  }
}

// dq, dk, dg (per channel, or summed over channels for the scalar gate) and
// dbeta: the sums of the row blocks' partials in row-block order, one warp
// per (token, head) row (each lane DK / 32 consecutive channels, loaded as
// one vector: all 3 x RB loads of a row in flight at once).
constexpr int kFinThreads = 256;
template <int DK>
__global__ void __launch_bounds__(kFinThreads)
    bwd_finalize_kernel(const float* __restrict__ part,
                        const float* __restrict__ part_b, int RB,
                        long long rows, float* dq, float* dk, float* dg,
                        float* dbeta, int g_chan) {
  constexpr int CPL = DK / 32;
  using V = typename std::conditional<CPL == 4, float4, float2>::type;
  const int lane = threadIdx.x & 31;
  const long long w0 = ((long long)blockIdx.x * kFinThreads + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * kFinThreads) >> 5;
  auto add = [](float (&acc)[CPL], const V& x) {
    const float* f = reinterpret_cast<const float*>(&x);
#pragma unroll
    for (int j = 0; j < CPL; ++j) acc[j] += f[j];
  };
  auto put = [](float* dst, const float (&x)[CPL]) {
    V v;
    float* f = reinterpret_cast<float*>(&v);
#pragma unroll
    for (int j = 0; j < CPL; ++j) f[j] = x[j];
    *reinterpret_cast<V*>(dst) = v;
  };
  for (long long row = w0; row < rows; row += nw) {
    float sq[CPL], sk[CPL], sg[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) sq[j] = sk[j] = sg[j] = 0.f;
    const size_t c0 = (size_t)row * DK + CPL * lane;
    for (int rb = 0; rb < RB; ++rb) {
      const V xq = *reinterpret_cast<const V*>(part + ((size_t)0 * RB + rb) * rows * DK + c0);
      const V xk = *reinterpret_cast<const V*>(part + ((size_t)1 * RB + rb) * rows * DK + c0);
      const V xg = *reinterpret_cast<const V*>(part + ((size_t)2 * RB + rb) * rows * DK + c0);
      add(sq, xq);
      add(sk, xk);
      add(sg, xg);
    }
    put(dq + c0, sq);
    put(dk + c0, sk);
    if (g_chan != 1) {
      put(dg + c0, sg);
    } else {
      float t = 0.f;
#pragma unroll
      for (int j = 0; j < CPL; ++j) t += sg[j];
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
      if (lane == 0) dg[row] = t;
    }
    if (lane == 0) {
      float sb = 0.f;
      for (int rb = 0; rb < RB; ++rb) sb += part_b[(size_t)rb * rows + row];
      dbeta[row] = sb;
    }
  }
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Both entry points: g_chan = dk (KDA) or 1 (scalar gate).
int run_bwd(const void* q, const void* k, const void* v, const float* g,
            const float* beta, const float* h0, const void* dout,
            const float* dhT, float* dq, float* dk, float* dvo, float* dg,
            float* dbeta, float* dh0, const int32_t* cu_seqlens, int B, int H,
            int T, int dk_, int dv, bool per_channel, int variant, bool f32,
            cudaStream_t stream, float* o_out,
            const std::function<cudaError_t()>* between) {
  if (B < 0 || H <= 0 || T < 0) return GDN_ERR_INVALID_ARG;
  if (variant != GDN_GATE_BEFORE_PREDICT && variant != GDN_GATE_AFTER_PREDICT)
    return GDN_ERR_INVALID_ARG;
  if (cu_seqlens && B == 0) return GDN_ERR_INVALID_ARG;
  if ((dk_ != 64 && dk_ != 128) || (dv != 64 && dv != 128))
    return GDN_ERR_UNSUPPORTED;
  const long long tokens = cu_seqlens ? (long long)T : (long long)B * T;
  if (B == 0) return GDN_OK;
  if (tokens > 0 && (!q || !k || !v || !g || !beta || !dout || !dq || !dk ||
                     !dvo || !dg || !dbeta))
    return GDN_ERR_INVALID_ARG;
  if (B > 65535 || tokens * H > (1ll << 40) || (long long)B * H > 0x7fffffffll)
    return GDN_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k, v, g, beta, h0, dout, dhT, dq, dk, dvo, dg, dbeta, dh0,
                        cu_seqlens};
  for (const void* p : ptrs)
    if (p && !al16(p)) return GDN_ERR_MISALIGNED;
  const void* outs[] = {dq, dk, dvo, dg, dbeta};
  for (const void* o : outs)
    if (o && (o == q || o == k || o == v || o == g || o == beta || o == dout))
      return GDN_ERR_INVALID_ARG;
  int* status = nullptr;
  int rc = device_status_ptr(&status);
  if (rc != GDN_OK) return rc;

  const int RB = dv / kBwRows, NS = kBwRpw * (dk_ / 32);
  const long long nblk = cu_seqlens ? tokens / kBwTok + B
                                    : (long long)B * ((T + kBwTok - 1) / kBwTok);
  const size_t rows = (size_t)tokens * H;
  const size_t per_cta = (size_t)kBwThreads * NS * sizeof(float);
  const size_t off_b = cu_seqlens ? (((size_t)B + 1) * sizeof(int32_t) + 255) & ~(size_t)255 : 0;
  const size_t ck_b = (size_t)nblk * H * RB * per_cta;
  const size_t win_b = (size_t)B * H * RB * kBwTok * per_cta;
  const size_t part_b = 3ull * RB * rows * dk_ * sizeof(float);
  const size_t pb_b = (size_t)RB * rows * sizeof(float);
  char* ws = nullptr;
  const size_t total = off_b + ck_b + win_b + part_b + pb_b;
  if (cudaMallocAsync(reinterpret_cast<void**>(&ws), total, stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  BwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g; a.beta = beta; a.h0 = h0;
  a.dout = dout;
  a.dhT = dhT; a.dv_out = dvo; a.dh0 = dh0;
  a.blk_off = cu_seqlens ? reinterpret_cast<const int32_t*>(ws) : nullptr;
  a.ckpt = reinterpret_cast<float*>(ws + off_b);
  a.win = reinterpret_cast<float*>(ws + off_b + ck_b);
  a.part = reinterpret_cast<float*>(ws + off_b + ck_b + win_b);
  a.part_b = reinterpret_cast<float*>(ws + off_b + ck_b + win_b + part_b);
  a.cu_seqlens = cu_seqlens;
  a.N = B; a.H = H; a.T = T; a.dv = dv;
  a.g_chan = per_channel ? dk_ : 1;
  a.decay_first = variant == GDN_GATE_BEFORE_PREDICT ? 1 : 0;
  a.rows = (long long)rows;
  a.status = status;
  cudaError_t e = cudaSuccess;
  int launches = 0;
  if (cu_seqlens) {
    e = launch_block_offsets(cu_seqlens, B, T, kBwTok, const_cast<int32_t*>(a.blk_off),
                             status, stream);
    if (e == cudaSuccess) ++launches;
  }
  auto go = [&](auto kern, auto fin, int DKv) {
    const int smem = (DKv == 64 ? BwSmem<64>::TOTAL : BwSmem<128>::TOTAL) * (int)sizeof(float);
    cudaError_t x = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (x != cudaSuccess) return x;
    // both sweeps in one launch, or (with work to do between them: the
    // gradient of the output from o) the forward sweep, that work, and the
    // reverse sweep
    BwdArgs a1 = a;
    a1.passes = between ? 1 : 3;
    a1.o_out = o_out;
    int t = timing_start(GDN_KERNEL_BWD, stream);
    kern<<<dim3(RB, H, B), kBwThreads, smem, stream>>>(a1);
    x = cudaGetLastError();
    timing_stop(t, stream, x);
    if (x != cudaSuccess) return x;
    ++launches;
    if (between) {
      x = (*between)();
      if (x != cudaSuccess) return x;
      BwdArgs a2 = a;
      a2.passes = 2;
      a2.o_out = nullptr;
      t = timing_start(GDN_KERNEL_BWD, stream);
      kern<<<dim3(RB, H, B), kBwThreads, smem, stream>>>(a2);
      x = cudaGetLastError();
      timing_stop(t, stream, x);
      if (x != cudaSuccess) return x;
      ++launches;
    }
    if (rows == 0) return cudaSuccess;
    const long long grid = std::min<long long>(((long long)rows + 7) / 8, 152ll * 8);
    t = timing_start(GDN_KERNEL_BWD_FINALIZE, stream);
    fin<<<(int)grid, kFinThreads, 0, stream>>>(a.part, a.part_b, RB, (long long)rows, dq,
                                               dk, dg, dbeta, a.g_chan);
    x = cudaGetLastError();
    timing_stop(t, stream, x);
    if (x == cudaSuccess) ++launches;
    return x;
  };
  if (e == cudaSuccess) {
    if (f32)
      e = dk_ == 64 ? go(bwd_kernel<64, float>, bwd_finalize_kernel<64>, 64)
                    : go(bwd_kernel<128, float>, bwd_finalize_kernel<128>, 128);
    else
      e = dk_ == 64 ? go(bwd_kernel<64, __nv_bfloat16>, bwd_finalize_kernel<64>, 64)
                    : go(bwd_kernel<128, __nv_bfloat16>, bwd_finalize_kernel<128>, 128);
  }
  count_launches(e, launches);
  const cudaError_t f = cudaFreeAsync(ws, stream);
  return (e == cudaSuccess && f == cudaSuccess) ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn

extern "C" int gdn_kda_bwd(const void* q, const void* k, const void* v,
                           const float* g, const float* beta, const float* h0,
                           const void* dout, const float* dhT, float* dq,
                           float* dk, float* dv, float* dg, float* dbeta,
                           float* dh0, const int32_t* cu_seqlens, int B, int H,
                           int T, int dk_, int dv_, gdn_stream_t stream) {
  return gdn::run_bwd(q, k, v, g, beta, h0, dout, dhT, dq, dk, dv, dg, dbeta, dh0,
                      cu_seqlens, B, H, T, dk_, dv_, true,
                      GDN_GATE_BEFORE_PREDICT, false,
                      static_cast<cudaStream_t>(stream), nullptr, nullptr);
}

extern "C" int gdn_chunk_bwd(const void* q, const void* k, const void* v,
                             const float* g, const float* beta, const float* h0,
                             const void* dout, const float* dhT, float* dq,
                             float* dk, float* dv, float* dg, float* dbeta,
                             float* dh0, const int32_t* cu_seqlens, int B,
                             int H, int T, int dk_, int dv_, int variant,
                             gdn_stream_t stream) {
  return gdn::run_bwd(q, k, v, g, beta, h0, dout, dhT, dq, dk, dv, dg, dbeta, dh0,
                      cu_seqlens, B, H, T, dk_, dv_, false, variant, false,
                      static_cast<cudaStream_t>(stream), nullptr, nullptr);
}

extern "C" int gdn_chunk_bwd_f32(const float* q, const float* k, const float* v,
                                 const float* g, const float* beta,
                                 const float* h0, const float* dout,
                                 const float* dhT, float* dq, float* dk,
                                 float* dv, float* dg, float* dbeta, float* dh0,
                                 const int32_t* cu_seqlens, int B, int H, int T,
                                 int dk_, int dv_, int variant,
                                 gdn_stream_t stream) {
  return gdn::run_bwd(q, k, v, g, beta, h0, dout, dhT, dq, dk, dv, dg, dbeta, dh0,
                      cu_seqlens, B, H, T, dk_, dv_, false, variant, true,
                      static_cast<cudaStream_t>(stream), nullptr, nullptr);
}
