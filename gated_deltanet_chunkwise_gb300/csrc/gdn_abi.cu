// C-ABI entry points: host-side argument checks, workspace, kernel choice.
// Every check runs before anything is enqueued; a failing check returns a
// negative gdn_status_t and leaves the stream untouched.
#include <atomic>
#include <mutex>
#include <vector>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

// Status word written by kernels (first error wins), one per device.
__device__ int g_device_status;

std::atomic<unsigned long long> g_launches{0};

cudaError_t counted(cudaError_t e, int launches) {
  if (e == cudaSuccess) g_launches.fetch_add(launches);
  return e;
}

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices];
std::mutex g_status_mutex;

int current_status_ptr(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_status_mutex);
  if (!g_status_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess)
      return GDN_ERR_CUDA;
    g_status_ptr[dev] = static_cast<int*>(ptr);
  }
  *out = g_status_ptr[dev];
  return GDN_OK;
}

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

bool head_dim_ok(int d) { return d == 64 || d == 128; }

int check_chunk_args(const void* q, const void* k, const void* v,
                     const float* g, const float* beta, const float* h0,
                     const void* out, const float* hT,
                     const int32_t* cu_seqlens, int B, int H, int T, int dk,
                     int dv, int C, int dtype, int variant, int path,
                     int sp_parts) {
  if (B < 0 || H <= 0 || T < 0) return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_DTYPE_BF16 && dtype != GDN_DTYPE_F32)
    return GDN_ERR_INVALID_ARG;
  if (variant != GDN_GATE_BEFORE_PREDICT && variant != GDN_GATE_AFTER_PREDICT)
    return GDN_ERR_INVALID_ARG;
  if (path < GDN_PATH_AUTO || path > GDN_PATH_TCGEN05_FUSED)
    return GDN_ERR_INVALID_ARG;
  if (sp_parts < 0 || sp_parts > 4096) return GDN_ERR_INVALID_ARG;
  // the fused single-kernel path has no sequence-parallel split
  if (path == GDN_PATH_TCGEN05_FUSED && sp_parts > 1) return GDN_ERR_UNSUPPORTED;
  if (cu_seqlens && B == 0) return GDN_ERR_INVALID_ARG;
  const long long tokens = cu_seqlens ? (long long)T : (long long)B * T;
  if (tokens > 0 || (cu_seqlens && B > 0)) {
    if (!q || !k || !v || !g || !beta || !out) return GDN_ERR_INVALID_ARG;
  }
  if (!head_dim_ok(dk) || !head_dim_ok(dv) || C != 64)
    return GDN_ERR_UNSUPPORTED;
  if (path >= GDN_PATH_TCGEN05 && dtype != GDN_DTYPE_BF16)
    return GDN_ERR_UNSUPPORTED;
  // Size limits: token-head rows index with 64-bit math, but grid.z holds
  // sequences x parts and the tensor maps hold 32-bit extents.
  if ((long long)tokens * H > (1ll << 40)) return GDN_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k, v, g, beta, h0, out, hT, cu_seqlens};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
  // out must not alias an input.
  if (out && (out == q || out == k || out == v)) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

int choose_parts(int requested, int N, int H, int T, int dv, int C,
                 bool packed) {
  if (requested > 0) return requested;
  if (packed) return 1;
  // Automatic split: only long sequences, and only until the state-row CTAs
  // cover the SMs about twice.
  const int nch = (T + C - 1) / C;
  int sms = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) ==
            cudaSuccess && v > 0)
      sms = v;
  }
  const long long ctas = (long long)N * H * (dv / 32);
  if (nch < 64 || ctas >= 2ll * sms) return 1;
  int parts = (int)((2ll * sms + ctas - 1) / ctas);
  parts = parts < 2 ? 2 : parts;
  const int max_parts = nch / 16;  // keep >= 16 chunks per sub-sequence
  if (parts > max_parts) parts = max_parts;
  return parts < 1 ? 1 : parts;
}

// Chain kernel and sequence-parallel split for the tensor-core path. One
// chain CTA per SM, so a pass costs (waves of resident CTAs) x (chunks per
// sub-sequence); `rows` state rows per CTA (64: the split chain kernel, 128:
// the whole-state one), so a (sequence, head) takes ceil(dv / rows) CTAs and
// a split pass ceil(dk / rows) more for the scaling matrix. Picks the split
// count P that minimises split pass + corrected output pass and returns
// that cost.
long long parts_cost_tc(int requested, int N, int H, int T, int dk, int dv,
                        int C, bool packed, int rows, int sms,
                        int* parts_out) {
  const long long nch = (T + C - 1) / C;
  const long long nh = (long long)N * H, tv = (dv + rows - 1) / rows,
                  tk = (dk + rows - 1) / rows;
  auto waves = [&](long long ctas) { return (ctas + sms - 1) / sms; };
  // packed calls: passes over the longest possible sequence
  const long long len = packed ? (long long)T / C + 1 : nch;
  auto cost_at = [&](int P) {
    if (P <= 1) return waves(nh * tv) * len;
    const long long per = (len + P - 1) / P;
    const long long split = nh * (tv + (long long)(P - 2) * (tv + tk));
    const long long outp = nh * (P - 1) * tv;
    return (waves(split) + waves(outp)) * per;
  };
  if (requested > 0 || packed) {
    *parts_out = requested > 0 ? requested : 1;
    return cost_at(*parts_out);
  }
  long long best = cost_at(1);
  int best_p = 1;
  for (int P = 2; P <= 64 && P <= nch; ++P) {
    const long long cost = cost_at(P);
    if (cost < best) {
      best = cost;
      best_p = P;
    }
  }
  *parts_out = best_p;
  return best;
}

// rows per chain CTA and the split for the tensor-core path (`path` may fix
// the chain kernel)
// `path` may fix the chain kernel; GDN_PATH_TCGEN05_FUSED asks for the
// single-launch form (`*fused`, one sub-sequence). The automatic choice
// keeps the two-kernel form: measured on GB300, the single launch moves
// far fewer DRAM bytes (the hand-off stays in L2) but is not faster (W1
// 0.095 vs 0.086 ms, the packed workload 1.41 vs 1.08 ms).
void choose_chain_tc(int path, int requested, int N, int H, int T, int dk,
                     int dv, int C, bool packed, int* rows, int* parts,
                     bool* fused) {
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) ==
            cudaSuccess && v > 0)
      sms = v;
  }
  int p64 = 1, p128 = 1;
  const long long c64 = parts_cost_tc(requested, N, H, T, dk, dv, C, packed,
                                      64, sms, &p64);
  const long long c128 = parts_cost_tc(requested, N, H, T, dk, dv, C, packed,
                                       128, sms, &p128);
  const bool whole = path == GDN_PATH_TCGEN05_WHOLE ||
                     (path != GDN_PATH_TCGEN05_SPLIT && c128 < c64);
  *rows = whole ? 128 : 64;
  *parts = whole ? p128 : p64;
  *fused = path == GDN_PATH_TCGEN05_FUSED;
  if (*fused) {
    *rows = 128;
    *parts = 1;
  }
}

// The steps either side of the recurrence (gdn_chunk_fwd_fused).
struct Sublayer {
  bool on = false;
  const float* norm_w = nullptr;
  const void* gate = nullptr;
  float eps = 0.f;
};

int run_chunk(const void* q, const void* k, const void* v, const float* g,
              const float* beta, const float* h0, void* out, float* hT,
              const int32_t* cu_seqlens, int B, int H, int T, int dk, int dv,
              int C, int dtype, int variant, int path, int sp_parts,
              cudaStream_t stream, const Sublayer& sub = Sublayer{},
              bool kda = false) {
  // combination of sub-sequences (flags above the path)
  const int sp_mode = path & (GDN_SP_CHAIN | GDN_SP_SCAN);
  if ((path & ~0xFF & ~(GDN_SP_CHAIN | GDN_SP_SCAN)) != 0 ||
      sp_mode == (GDN_SP_CHAIN | GDN_SP_SCAN))
    return GDN_ERR_INVALID_ARG;
  path &= 0xFF;
  int rc = check_chunk_args(q, k, v, g, beta, h0, out, hT, cu_seqlens, B, H,
                            T, dk, dv, C, dtype, variant, path, sp_parts);
  if (rc != GDN_OK) return rc;
  if (sub.on) {
    if (!(sub.eps >= 0.f) || sub.eps > 3.0e38f) return GDN_ERR_INVALID_ARG;
    // the tensor-core path's shapes only
    if (dtype != GDN_DTYPE_BF16 || dk != 128 || (dv != 64 && dv != 128))
      return GDN_ERR_UNSUPPORTED;
    if ((sub.norm_w && !aligned16(sub.norm_w)) ||
        (sub.gate && !aligned16(sub.gate)))
      return GDN_ERR_MISALIGNED;
    if (sub.gate && sub.gate == out) return GDN_ERR_INVALID_ARG;
  }
  if (B == 0 || H == 0) return GDN_OK;
  const bool bf16 = dtype == GDN_DTYPE_BF16;
  const long long tokens = cu_seqlens ? (long long)T : (long long)B * T;
  const bool tc_ok = bf16 && chunk_tc_supported(dk, dv, tokens, B, H);
  if ((path >= GDN_PATH_TCGEN05 || sub.on || kda) && !tc_ok)
    return GDN_ERR_UNSUPPORTED;
  // KDA runs on the whole-state chain only (its column-wise state decay),
  // with its own preparation kernel for d_k = 128
  if (kda && (path == GDN_PATH_SIMT || path == GDN_PATH_TCGEN05_SPLIT ||
              dk != 128))
    return GDN_ERR_UNSUPPORTED;
  int* status = nullptr;
  if ((rc = current_status_ptr(&status)) != GDN_OK) return rc;

  ChunkParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.h0 = h0;
  p.out = out; p.hT = hT; p.cu_seqlens = cu_seqlens;
  p.N = B; p.H = H; p.T = T; p.dk = dk; p.dv = dv; p.C = C;
  p.variant = variant;
  p.status = status;
  const bool use_tc = tc_ok && path != GDN_PATH_SIMT;
  p.kda = kda ? 1 : 0;
  if (sub.on) {
    p.prologue = 1;
    p.epilogue = (sub.norm_w || sub.gate) ? 1 : 0;
    p.norm_w = sub.norm_w;
    p.gate_z = sub.gate;
    p.eps = sub.eps;
  }
  auto launch = [&](const ChunkParams& q) {
    return use_tc ? launch_chunk_tc(q, stream)
                  : launch_chunk_simt(q, bf16, stream);
  };
  int parts = 1;
  bool fused = false;
  if (use_tc)
    choose_chain_tc(kda ? GDN_PATH_TCGEN05_WHOLE : path, sp_parts, B, H, T,
                    dk, dv, C, cu_seqlens != nullptr, &p.chain_rows, &parts,
                    &fused);
  else
    parts = choose_parts(sp_parts, B, H, T, dv, C, cu_seqlens != nullptr);
  p.parts = parts;
  if (fused) {
    // one launch; the hand-off ring (a few slots per (sequence, head))
    p.part_begin = 0; p.part_count = 1; p.mode = kModeOutput;
    void* ring = nullptr;
    if (cudaMallocAsync(&ring, fused_ring_bytes(p), stream) != cudaSuccess)
      return GDN_ERR_CUDA;
    p.ring = ring;
    const cudaError_t e = counted(launch_chunk_fused(p, stream), 1);
    const cudaError_t f = cudaFreeAsync(ring, stream);
    return (e == cudaSuccess && f == cudaSuccess) ? GDN_OK : GDN_ERR_CUDA;
  }
  // Combination of the sub-sequences: the scan when forced, or when its
  // rounds of parallel work (64-row CTAs, two per SM, each worth four of the
  // chain's 16-row steps) take less time than the chain's P - 2 dependent
  // steps.
  bool use_scan = false;
  if (parts > 2 && sp_mode != GDN_SP_CHAIN) {
    if (sp_mode == GDN_SP_SCAN) {
      use_scan = true;
    } else {
      int sms = 148, dev = 0, v = 0;
      if (cudaGetDevice(&dev) == cudaSuccess &&
          cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) ==
              cudaSuccess && v > 0)
        sms = v;
      const long long L = parts - 2, slots = 2ll * sms;
      const long long nh = (long long)B * H;
      long long scan = 4 * ((nh * L * (dv / 64) + slots - 1) / slots);  // apply
      for (long long d = 1; d < L; d *= 2)
        scan += 4 * ((nh * L * ((dv + dk) / 64) + slots - 1) / slots);
      use_scan = scan < L;
    }
  }

  // Workspace: UT factors (tensor-core path) and sequence-parallel states
  // (and the scan's second buffer of sub-sequence maps).
  const size_t nhp = (size_t)B * H * parts;
  const size_t end_bytes =
      parts > 1 ? nhp * (size_t)(dv + dk) * dk * sizeof(float) : 0;
  const size_t start_bytes =
      parts > 1 ? nhp * (size_t)dv * dk * sizeof(float) : 0;
  const size_t tc_bytes = use_tc ? chunk_tc_workspace_bytes(p) : 0;
  const size_t scan_off = (end_bytes + start_bytes + tc_bytes + 255) & ~(size_t)255;
  const size_t total =
      use_scan ? scan_off + end_bytes : end_bytes + start_bytes + tc_bytes;
  void* ws = nullptr;
  if (total > 0 && cudaMallocAsync(&ws, total, stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  char* wsc = static_cast<char*>(ws);
  if (parts > 1) {
    p.ws_end = reinterpret_cast<float*>(wsc);
    p.ws_start = reinterpret_cast<float*>(wsc + end_bytes);
  }
  if (use_tc) chunk_tc_bind_workspace(p, wsc + end_bytes + start_bytes);
  float* scan_buf =
      use_scan ? reinterpret_cast<float*>(wsc + scan_off) : nullptr;

  cudaError_t e = cudaSuccess;
  if (use_tc) {
    int n_prep = 0;
    e = kda ? launch_kda_prep(p, stream, &n_prep)
            : launch_ut_prep(p, stream, &n_prep);
    counted(e, n_prep);
  }
  if (e == cudaSuccess) {
    if (parts == 1) {
      p.part_begin = 0; p.part_count = 1; p.mode = kModeOutput;
      e = counted(launch(p), 1);
    } else {
      // split pass, correction chain, corrected output pass
      p.mode = kModeSplit; p.part_begin = 0; p.part_count = parts - 1;
      e = counted(launch(p), 1);
      if (e == cudaSuccess && parts > 2) {
        if (use_scan) {
          int n_scan = 0;
          e = launch_sp_scan(p, scan_buf, stream, &n_scan);
          counted(e, n_scan);
        } else {
          e = counted(launch_sp_chain(p, stream), 1);
        }
      }
      if (e == cudaSuccess) {
        p.mode = kModeOutput; p.part_begin = 1; p.part_count = parts - 1;
        e = counted(launch(p), 1);
      }
    }
  }
  cudaError_t f = ws ? cudaFreeAsync(ws, stream) : cudaSuccess;
  return (e == cudaSuccess && f == cudaSuccess) ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

int validate_chunk_args(const void* q, const void* k, const void* v,
                        const float* g, const float* beta, const float* h0,
                        const void* out, const float* hT,
                        const int32_t* cu_seqlens, int B, int H, int T,
                        int dk, int dv, int C, int dtype, int variant,
                        int path, int sp_parts) {
  return check_chunk_args(q, k, v, g, beta, h0, out, hT, cu_seqlens, B, H, T,
                          dk, dv, C, dtype, variant, path, sp_parts);
}

int device_status_ptr(int** out) { return current_status_ptr(out); }

cudaError_t count_launches(cudaError_t e, int launches) {
  return counted(e, launches);
}

// ---- per-kernel timing ------------------------------------------------------
namespace {
struct TimingRecord {
  int kernel;
  int device;
  cudaEvent_t start, stop;
  bool closed;
};
std::mutex g_timing_mutex;
bool g_timing_on = false;
std::vector<TimingRecord> g_timing_pending;
std::vector<cudaEvent_t> g_event_pool[kMaxDevices];
unsigned g_timing_generation = 0;  // bumped whenever pending is cleared
double g_timing_ms[GDN_KERNEL_COUNT];
unsigned long long g_timing_launches[GDN_KERNEL_COUNT];

// Caller holds g_timing_mutex.
cudaEvent_t take_event(int dev) {
  std::vector<cudaEvent_t>& pool = g_event_pool[dev];
  if (!pool.empty()) {
    cudaEvent_t e = pool.back();
    pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

void give_back(const TimingRecord& r) {
  g_event_pool[r.device].push_back(r.start);
  g_event_pool[r.device].push_back(r.stop);
}
}  // namespace

int timing_start(int kernel, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_timing_mutex);
  if (!g_timing_on) return -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return -1;
  TimingRecord r{kernel, dev, take_event(dev), take_event(dev), false};
  if (!r.start || !r.stop || cudaEventRecord(r.start, stream) != cudaSuccess) {
    if (r.start) g_event_pool[dev].push_back(r.start);
    if (r.stop) g_event_pool[dev].push_back(r.stop);
    return -1;
  }
  g_timing_pending.push_back(r);
  return (int)((g_timing_generation & 0x7f) << 24) |
         ((int)g_timing_pending.size() - 1);
}

void timing_stop(int token, cudaStream_t stream, cudaError_t launch_result) {
  if (token < 0) return;
  std::lock_guard<std::mutex> lock(g_timing_mutex);
  const int index = token & 0xffffff;
  if ((unsigned)(token >> 24) != (g_timing_generation & 0x7f) ||
      index >= (int)g_timing_pending.size())
    return;  // discarded meanwhile
  TimingRecord& r = g_timing_pending[index];
  if (launch_result == cudaSuccess &&
      cudaEventRecord(r.stop, stream) == cudaSuccess)
    r.closed = true;
}

}  // namespace gdn

extern "C" {

int gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                  const float* beta, const float* h0, void* out, float* hT,
                  const int32_t* cu_seqlens, int B, int H, int T, int dk,
                  int dv, int C, gdn_stream_t stream) {
  return gdn::run_chunk(q, k, v, g, beta, h0, out, hT, cu_seqlens, B, H, T,
                        dk, dv, C, GDN_DTYPE_BF16, GDN_GATE_BEFORE_PREDICT,
                        GDN_PATH_AUTO, 0, stream);
}

int gdn_chunk_fwd_f32(const float* q, const float* k, const float* v,
                      const float* g, const float* beta, const float* h0,
                      float* out, float* hT, const int32_t* cu_seqlens, int B,
                      int H, int T, int dk, int dv, int C,
                      gdn_stream_t stream) {
  return gdn::run_chunk(q, k, v, g, beta, h0, out, hT, cu_seqlens, B, H, T,
                        dk, dv, C, GDN_DTYPE_F32, GDN_GATE_BEFORE_PREDICT,
                        GDN_PATH_AUTO, 0, stream);
}

int gdn_chunk_fwd_ex(const void* q, const void* k, const void* v,
                     const float* g, const float* beta, const float* h0,
                     void* out, float* hT, const int32_t* cu_seqlens, int B,
                     int H, int T, int dk, int dv, int C, int dtype,
                     int variant, int path, int sp_parts,
                     gdn_stream_t stream) {
  return gdn::run_chunk(q, k, v, g, beta, h0, out, hT, cu_seqlens, B, H, T,
                        dk, dv, C, dtype, variant, path, sp_parts, stream);
}

int gdn_chunk_fwd_fused(const void* q, const void* k, const void* v,
                        const float* a, const float* b, const float* h0,
                        void* out, float* hT, const int32_t* cu_seqlens,
                        const float* norm_weight, const void* gate, float eps,
                        int B, int H, int T, int dk, int dv, int C, int path,
                        gdn_stream_t stream) {
  if (path < GDN_PATH_AUTO || path > GDN_PATH_TCGEN05_FUSED)
    return GDN_ERR_INVALID_ARG;
  if (path == GDN_PATH_SIMT) return GDN_ERR_UNSUPPORTED;
  gdn::Sublayer sub;
  sub.on = true;
  sub.norm_w = norm_weight;
  sub.gate = gate;
  sub.eps = eps;
  return gdn::run_chunk(q, k, v, a, b, h0, out, hT, cu_seqlens, B, H, T, dk,
                        dv, C, GDN_DTYPE_BF16, GDN_GATE_BEFORE_PREDICT,
                        path == GDN_PATH_AUTO ? GDN_PATH_TCGEN05 : path, 0,
                        stream, sub);
}

int gdn_chunk_bwd_fused(const void* q, const void* k, const void* v,
                        const float* a, const float* b, const float* h0,
                        const int32_t* cu_seqlens, const float* norm_weight,
                        const void* gate, float eps, const void* dout,
                        const float* dhT, float* dq, float* dk, float* dv,
                        float* da, float* db, float* dh0, float* dweight,
                        float* dgate, int B, int H, int T, int dk_dim,
                        int dv_dim, gdn_stream_t stream) {
  using namespace gdn;
  if (B < 0 || H <= 0 || T < 0) return GDN_ERR_INVALID_ARG;
  if (cu_seqlens && B == 0) return GDN_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || eps > 3.0e38f) return GDN_ERR_INVALID_ARG;
  if (!head_dim_ok(dk_dim) || !head_dim_ok(dv_dim)) return GDN_ERR_UNSUPPORTED;
  const long long tokens = cu_seqlens ? (long long)T : (long long)B * T;
  if (tokens > 0 && (!q || !k || !v || !a || !b || !dout || !dq || !dk || !dv ||
                     !da || !db))
    return GDN_ERR_INVALID_ARG;
  if ((dweight && !norm_weight) || (dgate && !gate)) return GDN_ERR_INVALID_ARG;
  if (B > 65535 || tokens * H > (1ll << 40) || (long long)B * H > 0x7fffffffll)
    return GDN_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k, v, a, b, h0, cu_seqlens, norm_weight, gate, dout,
                        dhT, dq, dk, dv, da, db, dh0, dweight, dgate};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
  const void* ins[] = {q, k, v, a, b, h0, norm_weight, gate, dout};
  const void* outs[] = {dq, dk, dv, da, db, dweight, dgate};
  for (const void* o : outs)
    for (const void* in : ins)
      if (o && o == in) return GDN_ERR_INVALID_ARG;
  if (B == 0) return GDN_OK;
  int* status = nullptr;
  int rc = current_status_ptr(&status);
  if (rc != GDN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long rows = tokens * H;
  FusedBwdBufs f{};
  const size_t bytes = fused_bwd_bind(f, nullptr, rows, dk_dim, dv_dim);
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, bytes, st) != cudaSuccess) return GDN_ERR_CUDA;
  fused_bwd_bind(f, ws, rows, dk_dim, dv_dim);
  // the steps before the recurrence, the recurrence's output in fp32, the
  // adjoints of the steps after it, the recurrence's backward, the adjoints
  // of the steps before it
  cudaError_t e = counted(launch_sub_prologue(f, q, k, v, a, b, rows, dk_dim,
                                              dv_dim, st), rows > 0 ? 1 : 0);
  if (e == cudaSuccess) {
    // the recurrence's backward, whose forward sweep also yields o: the
    // epilogue's adjoint runs between its two sweeps and produces the
    // output gradient the reverse sweep reads
    const std::function<cudaError_t()> between = [&]() {
      return counted(launch_sub_epilogue_bwd(f, dout, norm_weight, gate, eps,
                                             rows, dv_dim, dgate, dweight, st),
                     rows > 0 ? (dweight ? 2 : 1) : 0);
    };
    rc = run_bwd(f.qh, f.kh, f.vf, f.g, f.beta, h0, f.dO, dhT, f.dqh, f.dkh, dv,
                 f.dg, f.dbeta, dh0, cu_seqlens, B, H, T, dk_dim, dv_dim, false,
                 GDN_GATE_BEFORE_PREDICT, true, st, f.o, &between);
    if (rc != GDN_OK) e = cudaErrorUnknown;
  }
  if (e == cudaSuccess)
    e = counted(launch_sub_prologue_bwd(f, a, rows, dk_dim, dq, dk, da, db, st),
                rows > 0 ? 1 : 0);
  const cudaError_t fr = cudaFreeAsync(ws, st);
  if (rc != GDN_OK) return rc;
  return (e == cudaSuccess && fr == cudaSuccess) ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_recurrent_step(const void* q, const void* k, const void* v,
                       const float* g, const float* beta, float* state,
                       void* out, int N, int H, int dk, int dv,
                       gdn_stream_t stream) {
  if (N < 0 || H <= 0) return GDN_ERR_INVALID_ARG;
  if (!gdn::head_dim_ok(dk) || !gdn::head_dim_ok(dv))
    return GDN_ERR_UNSUPPORTED;
  if (N == 0) return GDN_OK;
  if (!q || !k || !v || !g || !beta || !state || !out)
    return GDN_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, g, beta, state, out};
  for (const void* p : ptrs)
    if (!gdn::aligned16(p)) return GDN_ERR_MISALIGNED;
  if ((long long)N * H > 0x7fffffffll) return GDN_ERR_UNSUPPORTED;
  if (out == q || out == k || out == v) return GDN_ERR_INVALID_ARG;
  gdn::DecodeParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.state = state;
  p.out = out; p.N = N; p.H = H; p.dk = dk; p.dv = dv;
  p.variant = GDN_GATE_BEFORE_PREDICT;
  return gdn::counted(gdn::launch_decode(p, stream), 1) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

int gdn_kda_fwd(const void* q, const void* k, const void* v, const float* g,
                const float* beta, const float* h0, void* out, float* hT,
                const int32_t* cu_seqlens, int B, int H, int T, int dk, int dv,
                gdn_stream_t stream) {
  if (B < 0 || H <= 0 || T < 0) return GDN_ERR_INVALID_ARG;
  if (cu_seqlens && B == 0) return GDN_ERR_INVALID_ARG;
  if (!gdn::head_dim_ok(dk) || !gdn::head_dim_ok(dv)) return GDN_ERR_UNSUPPORTED;
  const long long tokens = cu_seqlens ? (long long)T : (long long)B * T;
  if (B == 0) return GDN_OK;
  if (tokens > 0 && (!q || !k || !v || !g || !beta || !out))
    return GDN_ERR_INVALID_ARG;
  if ((long long)tokens * H > (1ll << 40) || (long long)B * H > 0x7fffffffll)
    return GDN_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k, v, g, beta, h0, out, hT, cu_seqlens};
  for (const void* p : ptrs)
    if (p && !gdn::aligned16(p)) return GDN_ERR_MISALIGNED;
  if (out && (out == q || out == k || out == v)) return GDN_ERR_INVALID_ARG;
  int* status = nullptr;
  int rc = gdn::current_status_ptr(&status);
  if (rc != GDN_OK) return rc;
  gdn::KdaParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.h0 = h0;
  p.out = out; p.hT = hT; p.cu_seqlens = cu_seqlens;
  p.N = B; p.H = H; p.T = T; p.dk = dk; p.dv = dv; p.status = status;
  return gdn::counted(gdn::launch_kda(p, stream), 1) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

int gdn_kda_fwd_ex(const void* q, const void* k, const void* v,
                   const float* g, const float* beta, const float* h0,
                   void* out, float* hT, const int32_t* cu_seqlens, int B,
                   int H, int T, int dk, int dv, int path, int sp_parts,
                   gdn_stream_t stream) {
  const int sp_mode = path & (GDN_SP_CHAIN | GDN_SP_SCAN);
  const int kernels = path & ~(GDN_SP_CHAIN | GDN_SP_SCAN);
  if (kernels < GDN_PATH_AUTO || kernels > GDN_PATH_TCGEN05_FUSED)
    return GDN_ERR_INVALID_ARG;
  // the chunk form of KDA runs on the whole-state chain with its own
  // preparation kernel only
  if (kernels == GDN_PATH_TCGEN05_SPLIT || kernels == GDN_PATH_TCGEN05_FUSED)
    return GDN_ERR_UNSUPPORTED;
  const long long tokens = cu_seqlens ? (long long)T : (long long)B * T;
  // nothing to compute but the state copy: the token-by-token kernel
  if (kernels == GDN_PATH_SIMT || B <= 0 || H <= 0 || T <= 0 || tokens <= 0 ||
      (kernels == GDN_PATH_AUTO &&
       (dk != 128 || !gdn::chunk_tc_supported(dk, dv, tokens, B, H))))
    return gdn_kda_fwd(q, k, v, g, beta, h0, out, hT, cu_seqlens, B, H, T, dk,
                       dv, stream);
  return gdn::run_chunk(q, k, v, g, beta, h0, out, hT, cu_seqlens, B, H, T, dk,
                        dv, 64, GDN_DTYPE_BF16, GDN_GATE_BEFORE_PREDICT,
                        (kernels == GDN_PATH_AUTO ? GDN_PATH_TCGEN05 : kernels) |
                            sp_mode,
                        sp_parts, stream, gdn::Sublayer{}, true);
}

int gdn_device_status(gdn_stream_t stream) {
  int* status = nullptr;
  int rc = gdn::current_status_ptr(&status);
  if (rc != GDN_OK) return rc;
  int value = 0;
  if (cudaMemcpyAsync(&value, status, sizeof(int), cudaMemcpyDeviceToHost,
                      stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaMemsetAsync(status, 0, sizeof(int), stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return GDN_ERR_CUDA;
  return value;
}

const char* gdn_status_string(int status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_MISALIGNED: return "GDN_ERR_MISALIGNED";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
    default: return "GDN_UNKNOWN_STATUS";
  }
}

int gdn_version(void) { return 100; }

unsigned long long gdn_kernel_launches(void) { return gdn::g_launches.load(); }

int gdn_timing_enable(int on) {
  using namespace gdn;
  std::lock_guard<std::mutex> lock(g_timing_mutex);
  int rc = GDN_OK;
  for (const TimingRecord& r : g_timing_pending) {
    if (r.closed && cudaEventSynchronize(r.stop) != cudaSuccess) rc = GDN_ERR_CUDA;
    give_back(r);
  }
  g_timing_pending.clear();
  ++g_timing_generation;
  for (int k = 0; k < GDN_KERNEL_COUNT; ++k) {
    g_timing_ms[k] = 0.0;
    g_timing_launches[k] = 0;
  }
  g_timing_on = on != 0;
  return rc;
}

int gdn_timing_read(int kernel, unsigned long long* launches,
                    double* total_ms) {
  using namespace gdn;
  if (kernel < 0 || kernel >= GDN_KERNEL_COUNT) return GDN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_timing_mutex);
  int rc = GDN_OK;
  for (const TimingRecord& r : g_timing_pending) {
    float ms = 0.f;
    if (r.closed) {
      if (cudaEventSynchronize(r.stop) == cudaSuccess &&
          cudaEventElapsedTime(&ms, r.start, r.stop) == cudaSuccess) {
        g_timing_ms[r.kernel] += ms;
        g_timing_launches[r.kernel] += 1;
      } else {
        rc = GDN_ERR_CUDA;
      }
    }
    give_back(r);
  }
  g_timing_pending.clear();
  ++g_timing_generation;
  if (launches) *launches = g_timing_launches[kernel];
  if (total_ms) *total_ms = g_timing_ms[kernel];
  return rc;
}

}  // extern "C"
