// attn_bwd_noalloc: the attention backward for callers that cannot allocate
// device memory themselves.
//
// attn_bwd needs a caller-provided workspace (D = sum_j P dP per row and head,
// per-tile minimum seg, a status header). Some callers have no way to obtain
// one: a plugin that is handed only its input and output buffers by a host
// engine, code that runs where the process's memory manager forbids raw
// cudaMalloc after start-up, or a thin language binding with no device
// allocator. For them this entry point keeps its scratch in a fixed array
// compiled into the library, so a call needs only the inputs and outputs.
//
// Costs and limits, stated for the user:
//  - the array is kNoAllocScratchBytes (4 MiB) of device memory, held on every
//    GPU that loads this library until the process exits;
//  - the workspace layout must fit in it: seq_len * n_heads <= ~1M (e.g.
//    16384 x 32 uses 2.1 MB); larger shapes return GQA_ERR_UNSUPPORTED;
//  - every call shares the one array: calls whose GPU work overlaps (two
//    streams, two host threads) race on it and give wrong results;
//  - the first call on a device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current) and caches it together
//    with the id of the device's current CUDA context; make that first call
//    before any stream capture on the device. A later call that finds another
//    context current (after cudaDeviceReset or a primary-context teardown the
//    library's device code is loaded again and the array may move) looks the
//    address up again instead of using the stale one.
// The kernels are the CUDA-core backward (the same ones attn_bwd_simt runs).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>
#include <utility>

#include "common.cuh"

namespace gqa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

// In host code this name is only a stand-in for the device array: its device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};   // context id the address belongs to

// Unique id of the calling thread's current CUDA context (driver entry
// points looked up once through the runtime, as for the tensor maps).
gqa_status current_context_id(unsigned long long* id) {
  static const auto fns = [] {
    std::pair<PFN_cuCtxGetCurrent_v4000, PFN_cuCtxGetId_v12000> f{nullptr, nullptr};
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.first = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.second = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    return f;
  }();
  if (fns.first == nullptr || fns.second == nullptr)
    return set_error(GQA_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId unavailable");
  CUcontext ctx = nullptr;
  if (fns.first(&ctx) != CUDA_SUCCESS || ctx == nullptr)
    return set_error(GQA_ERR_CUDA, "no current CUDA context");
  if (fns.second(ctx, id) != CUDA_SUCCESS)
    return set_error(GQA_ERR_CUDA, "cuCtxGetId failed");
  return GQA_OK;
}

gqa_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return set_error(GQA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(GQA_ERR_UNSUPPORTED, "device ordinal %d is beyond %d", dev, kMaxDevices);
  // cudaSetDevice initialises the device's primary context and makes it
  // current (a no-op when it already is), so that the context id below is the
  // one the launches will use; it allocates nothing
  if ((e = cudaSetDevice(dev)) != cudaSuccess)
    return set_error(GQA_ERR_CUDA, "cudaSetDevice(%d): %s", dev, cudaGetErrorString(e));
  unsigned long long ctx = 0;
  gqa_status r = current_context_id(&ctx);
  if (r != GQA_OK) return r;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return set_error(GQA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_addr[dev];
  return GQA_OK;
}

}  // namespace
}  // namespace gqa

using namespace gqa;

extern "C" gqa_status attn_bwd_noalloc(const float* Q, const float* K, const float* V,
                                       const float* dO, const float* LSE, const uint32_t* seg,
                                       float* dQ, float* dK, float* dV, int seq_len, int n_heads,
                                       int n_kv_heads, int head_dim, float scale, void* stream) {
  gqa_status r = check_attn_args(seq_len, n_heads, n_kv_heads, head_dim, scale, 128);
  if (r != GQA_OK || seq_len == 0) return r;
  const void* p[] = {Q, K, V, dO, LSE, seg, dQ, dK, dV};
  const char* nm[] = {"Q", "K", "V", "dO", "LSE", "seg", "dQ", "dK", "dV"};
  for (int i = 0; i < 9; ++i) {
    if (p[i] == nullptr) return set_error(GQA_ERR_INVALID_ARG, "%s is NULL", nm[i]);
    if (!aligned16(p[i])) return set_error(GQA_ERR_INVALID_ARG, "%s is not 16-byte aligned", nm[i]);
  }
  const size_t need = ws_layout(seq_len, n_heads).total;
  if (need > kNoAllocScratchBytes)
    return set_error(GQA_ERR_UNSUPPORTED,
                     "attn_bwd_noalloc: seq_len %d x n_heads %d needs %zu bytes of scratch, "
                     "more than its fixed %zu; use attn_bwd with a workspace",
                     seq_len, n_heads, need, kNoAllocScratchBytes);
  void* ws = nullptr;
  if ((r = scratch_address(&ws)) != GQA_OK) return r;
  cudaStream_t st = (cudaStream_t)stream;
  // The array keeps the previous call's contents: the status header must start
  // at zero; D and the per-tile minima are fully rewritten before they are read.
  if (cudaMemsetAsync(ws, 0, kWsHeader, st) != cudaSuccess)
    return check_launch("attn_bwd_noalloc scratch header reset");
  if ((r = debug_check_seg(seg, seq_len, ws, st)) != GQA_OK) return r;
  Shape sh{seq_len, n_heads, n_kv_heads, head_dim, n_heads / n_kv_heads, scale};
  return simt_bwd(Q, K, V, dO, LSE, seg, dQ, dK, dV, sh, (char*)ws, st, no_rope());
}
