// Sequence-parallel chunked forward pass without any device allocation.
//
// Some callers cannot allocate device memory at the moment they enqueue work:
// an inference engine's plugin whose memory plan is fixed before the first
// request, a serving loop that runs inside a fixed memory budget, or any host
// code that is not allowed to call cudaMalloc / cudaMallocAsync (or a caching
// allocator) on its hot path. gdn_chunk_fwd_ex takes the sequence-parallel
// workspace with cudaMallocAsync; this entry point runs the same kernels with
// the workspace taken from a fixed array in device memory that the library
// owns instead.
//
// The array is a file-scope __device__ variable of GDN_NOALLOC_SCRATCH_BYTES:
// every device that loads this library holds it until the process exits. All
// calls on a device share it and it keeps the previous call's contents; every
// entry a call reads is written earlier in the same call, so nothing needs
// clearing. Calls whose work overlaps on the GPU (two streams, or two host
// threads) race on the array: the caller must order them.
#include <cuda.h>

#include <mutex>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

static __device__ __align__(256) unsigned char
    g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
// Per device: the array's address and the driver context it belongs to.
void* g_scratch_addr[kMaxDevices];
unsigned long long g_scratch_ctx[kMaxDevices];
std::mutex g_scratch_mutex;

// Unique id of the calling thread's current driver context (0 when there is
// none yet), through driver entry points so that the library needs no link
// against the driver library. A device reset, or another context made
// current on the same device, gives a different id: the module holding the
// array has been loaded again there and its address must be looked up anew.
typedef CUresult (*ctx_current_fn)(CUcontext*);
typedef CUresult (*ctx_id_fn)(CUcontext, unsigned long long*);
ctx_current_fn g_ctx_current;
ctx_id_fn g_ctx_id;
std::once_flag g_ctx_once;

bool current_context_id(unsigned long long* id) {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<ctx_current_fn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<ctx_id_fn>(fn);
  });
  if (!g_ctx_current || !g_ctx_id) return false;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return false;
  *id = 0;
  return ctx == nullptr || g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the array in the current device's current context. In
// host code the symbol itself is only a host-side stand-in, so the address
// is looked up with the device current (the first call on a device, and the
// first call after its context changed) and cached.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  unsigned long long ctx = 0;
  if (!current_context_id(&ctx)) return GDN_ERR_CUDA;
  if (!g_scratch_addr[dev] || ctx == 0 || g_scratch_ctx[dev] != ctx) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess ||
        ptr == nullptr)
      return GDN_ERR_CUDA;
    // the lookup made the runtime's context current if none was
    if (!current_context_id(&ctx) || ctx == 0) return GDN_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_addr[dev];
  return GDN_OK;
}

}  // namespace
}  // namespace gdn

extern "C" unsigned long long gdn_noalloc_scratch_bytes(int B, int H, int dk,
                                                        int dv,
                                                        int sp_parts) {
  // only the head dimensions the entry point serves (64, 128); all
  // products in 64 bits
  const bool dims_ok = (dk == 64 || dk == 128) && (dv == 64 || dv == 128);
  if (B <= 0 || H <= 0 || !dims_ok || sp_parts < 2) return 0;
  const unsigned long long nhp = (unsigned long long)B *
                                 (unsigned long long)H *
                                 (unsigned long long)sp_parts;
  return nhp * (2ull * (unsigned long long)dv + (unsigned long long)dk) *
         (unsigned long long)dk * sizeof(float);
}

extern "C" int gdn_chunk_fwd_sp_noalloc(
    const void* q, const void* k, const void* v, const float* g,
    const float* beta, const float* h0, void* out, float* hT,
    const int32_t* cu_seqlens, int B, int H, int T, int dk, int dv, int C,
    int dtype, int variant, int sp_parts, gdn_stream_t stream) {
  using namespace gdn;
  if (sp_parts < 2) return GDN_ERR_INVALID_ARG;
  int rc = validate_chunk_args(q, k, v, g, beta, h0, out, hT, cu_seqlens, B,
                               H, T, dk, dv, C, dtype, variant,
                               GDN_PATH_SIMT, sp_parts);
  if (rc != GDN_OK) return rc;
  if (B == 0) return GDN_OK;
  const unsigned long long need =
      gdn_noalloc_scratch_bytes(B, H, dk, dv, sp_parts);
  if (need > GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_UNSUPPORTED;

  void* ws = nullptr;
  if ((rc = scratch_address(&ws)) != GDN_OK) return rc;
  int* status = nullptr;
  if ((rc = device_status_ptr(&status)) != GDN_OK) return rc;

  ChunkParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.h0 = h0;
  p.out = out; p.hT = hT; p.cu_seqlens = cu_seqlens;
  p.N = B; p.H = H; p.T = T; p.dk = dk; p.dv = dv; p.C = C;
  p.variant = variant;
  p.status = status;
  p.parts = sp_parts;
  const size_t nhp = (size_t)B * H * sp_parts;
  p.ws_end = static_cast<float*>(ws);
  p.ws_start = p.ws_end + nhp * (size_t)(dv + dk) * dk;
  const bool bf16 = dtype == GDN_DTYPE_BF16;

  p.mode = kModeSplit; p.part_begin = 0; p.part_count = sp_parts - 1;
  cudaError_t e = count_launches(launch_chunk_simt(p, bf16, stream), 1);
  if (e == cudaSuccess && sp_parts > 2)
    e = count_launches(launch_sp_chain(p, stream), 1);
  if (e == cudaSuccess) {
    p.mode = kModeOutput; p.part_begin = 1; p.part_count = sp_parts - 1;
    e = count_launches(launch_chunk_simt(p, bf16, stream), 1);
  }
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
