// Entry points of libgqa_attn.so (declared in include/gqa_attn.h): argument
// checks on the host, workspace layout, and the choice of kernel.
#include <cuda_runtime.h>
#include <math.h>

#include <atomic>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "common.cuh"

namespace gqa {

static thread_local char g_last_error[512] = "";
static thread_local ProfileHook g_hook;

static std::atomic<unsigned long long> g_launches{0};
static std::atomic<int> g_short_path{1};

ProfileHook& profile_hook() { return g_hook; }
void note_launch(int n) { g_launches.fetch_add((unsigned long long)n); }

gqa_status set_error(gqa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

gqa_status check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(GQA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return GQA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gqa_status check_attn_args(int S, int H, int Hk, int d, float scale, int max_d) {
  if (S < 0) return set_error(GQA_ERR_INVALID_ARG, "seq_len must be >= 0 (got %d)", S);
  if (H <= 0 || Hk <= 0)
    return set_error(GQA_ERR_INVALID_ARG, "n_heads and n_kv_heads must be > 0 (got %d, %d)", H, Hk);
  if (H % Hk != 0)
    return set_error(GQA_ERR_INVALID_ARG, "n_heads (%d) must be a multiple of n_kv_heads (%d)", H, Hk);
  if (d <= 0 || d % 4 != 0)
    return set_error(GQA_ERR_INVALID_ARG, "head_dim must be a positive multiple of 4 (got %d)", d);
  if (d > max_d)
    return set_error(GQA_ERR_UNSUPPORTED, "head_dim %d > %d has no kernel", d, max_d);
  if (!isfinite(scale)) return set_error(GQA_ERR_INVALID_ARG, "scale must be finite");
  const long long widest = (long long)S * (long long)(H > Hk ? H : Hk) * d;
  if (widest >= (1LL << 31))
    return set_error(GQA_ERR_UNSUPPORTED, "seq_len*heads*head_dim = %lld must be < 2^31", widest);
  return GQA_OK;
}

static gqa_status check_ptrs(const void* const* ptrs, const char* const* names, int n) {
  for (int i = 0; i < n; ++i) {
    if (ptrs[i] == nullptr) return set_error(GQA_ERR_INVALID_ARG, "%s is NULL", names[i]);
    if (!aligned16(ptrs[i]))
      return set_error(GQA_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
  }
  return GQA_OK;
}

static gqa_status check_bwd(const float* Q, const float* K, const float* V, const float* dO,
                            const float* LSE, const uint32_t* seg, float* dQ, float* dK,
                            float* dV, int S, int H, int Hk, int d, float scale, void* ws,
                            size_t ws_bytes) {
  gqa_status r = check_attn_args(S, H, Hk, d, scale, 128);
  if (r != GQA_OK || S == 0) return r;
  const void* p[] = {Q, K, V, dO, LSE, seg, dQ, dK, dV, ws};
  const char* nm[] = {"Q", "K", "V", "dO", "LSE", "seg", "dQ", "dK", "dV", "workspace"};
  r = check_ptrs(p, nm, 10);
  if (r != GQA_OK) return r;
  const size_t need = ws_layout(S, H).total;
  if (ws_bytes < need)
    return set_error(GQA_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  return GQA_OK;
}

}  // namespace gqa

using namespace gqa;

extern "C" {

const char* gqa_status_str(gqa_status s) {
  switch (s) {
    case GQA_OK: return "GQA_OK";
    case GQA_ERR_INVALID_ARG: return "GQA_ERR_INVALID_ARG";
    case GQA_ERR_UNSUPPORTED: return "GQA_ERR_UNSUPPORTED";
    case GQA_ERR_CUDA: return "GQA_ERR_CUDA";
    case GQA_ERR_DEVICE_TIMEOUT: return "GQA_ERR_DEVICE_TIMEOUT";
    case GQA_ERR_DEVICE_CHECK: return "GQA_ERR_DEVICE_CHECK";
  }
  return "GQA_ERR_UNKNOWN";
}

const char* gqa_last_error(void) { return g_last_error; }

void gqa_profile_events(void* before, void* after) {
  if (before && after) {
    g_hook.before = (cudaEvent_t)before;
    g_hook.after = (cudaEvent_t)after;
  } else {
    g_hook.before = g_hook.after = nullptr;
  }
}

const char* gqa_profile_stage_name(void) { return g_hook.stage; }

unsigned long long gqa_launch_count(void) { return g_launches.load(); }

size_t attn_bwd_workspace_bytes(int seq_len, int n_heads, int n_kv_heads, int head_dim) {
  if (seq_len <= 0 || n_heads <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads) return kWsHeader;
  const Shape sh{seq_len, n_heads, n_kv_heads, head_dim, n_heads / n_kv_heads, 1.f};
  size_t need = tc_supported(sh) ? tc_ws_layout(seq_len, n_heads, n_kv_heads, head_dim).total
                                 : ws_layout(seq_len, n_heads).total;
  if (head_dim > 0 && head_dim <= 128 && short_supported(sh)) {
    const size_t s = short_ws_bytes(seq_len, n_heads, head_dim);
    if (s > need) need = s;
  }
  return need;
}

int gqa_set_short_path(int enable) { return g_short_path.exchange(enable != 0 ? 1 : 0); }

gqa_status attn_fwd_lse(const float* Q, const float* K, const float* V, const uint32_t* seg,
                        float* O, float* LSE, int seq_len, int n_heads, int n_kv_heads,
                        int head_dim, float scale, void* stream) {
  gqa_status r = check_attn_args(seq_len, n_heads, n_kv_heads, head_dim, scale, 128);
  if (r != GQA_OK || seq_len == 0) return r;
  const void* p[] = {Q, K, V, seg, O, LSE};
  const char* nm[] = {"Q", "K", "V", "seg", "O", "LSE"};
  if ((r = check_ptrs(p, nm, 6)) != GQA_OK) return r;
  Shape sh{seq_len, n_heads, n_kv_heads, head_dim, n_heads / n_kv_heads, scale};
  return simt_fwd_lse(Q, K, V, seg, O, LSE, sh, (cudaStream_t)stream);
}

size_t attn_fwd_workspace_bytes(int seq_len, int n_heads, int n_kv_heads, int head_dim) {
  if (seq_len <= 0 || n_heads <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads) return kWsHeader;
  const Shape sh{seq_len, n_heads, n_kv_heads, head_dim, n_heads / n_kv_heads, 1.f};
  if (tc_fwd_supported(sh)) return tc_fwd_ws_bytes(seq_len, n_kv_heads, head_dim);
  return kWsHeader;
}

gqa_status attn_fwd(const float* Q, const float* K, const float* V, const uint32_t* seg, float* O,
                    float* LSE, int seq_len, int n_heads, int n_kv_heads, int head_dim, float scale,
                    void* workspace, size_t workspace_bytes, void* stream) {
  gqa_status r = check_attn_args(seq_len, n_heads, n_kv_heads, head_dim, scale, 128);
  if (r != GQA_OK || seq_len == 0) return r;
  const void* p[] = {Q, K, V, seg, O, LSE, workspace};
  const char* nm[] = {"Q", "K", "V", "seg", "O", "LSE", "workspace"};
  if ((r = check_ptrs(p, nm, 7)) != GQA_OK) return r;
  const size_t need = attn_fwd_workspace_bytes(seq_len, n_heads, n_kv_heads, head_dim);
  if (workspace_bytes < need)
    return set_error(GQA_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  const Shape sh{seq_len, n_heads, n_kv_heads, head_dim, n_heads / n_kv_heads, scale};
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(workspace, 0, kWsHeader, st) != cudaSuccess)
    return check_launch("workspace header reset");
  if ((r = debug_check_seg(seg, seq_len, workspace, st)) != GQA_OK) return r;
  if (!tc_fwd_supported(sh)) return simt_fwd_lse(Q, K, V, seg, O, LSE, sh, st);
  return tc_fwd(Q, K, V, seg, O, LSE, sh, (char*)workspace, st);
}

size_t attn_decode_bwd_workspace_bytes(int history_len, int n_heads, int n_kv_heads, int head_dim) {
  if (history_len <= 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0) return kWsHeader;
  return decode_ws_bytes(history_len, n_heads, head_dim);
}

gqa_status attn_decode_bwd(const float* q, const float* k_hist, const float* v_hist,
                           const float* probs, const float* d_out, float* d_scores, float* d_q,
                           float* d_k_hist, float* d_v_hist, int history_len, int n_heads,
                           int n_kv_heads, int head_dim, float scale, void* workspace,
                           size_t workspace_bytes, void* stream) {
  gqa_status r = check_attn_args(history_len, n_heads, n_kv_heads, head_dim, scale, 128);
  if (r != GQA_OK) return r;
  if (head_dim % 32 != 0)
    return set_error(GQA_ERR_UNSUPPORTED, "decode backward: head_dim %d not in {32, 64, 96, 128}", head_dim);
  if (n_kv_heads > 65535)
    return set_error(GQA_ERR_UNSUPPORTED, "decode backward: n_kv_heads %d > 65535", n_kv_heads);
  if (history_len == 0) return GQA_OK;
  const void* p[] = {q, k_hist, v_hist, probs, d_out, d_scores, d_q, d_k_hist, d_v_hist, workspace};
  const char* nm[] = {"q", "k_hist", "v_hist", "probs", "d_out", "d_scores", "d_q", "d_k_hist",
                      "d_v_hist", "workspace"};
  if ((r = check_ptrs(p, nm, 10)) != GQA_OK) return r;
  const size_t need = attn_decode_bwd_workspace_bytes(history_len, n_heads, n_kv_heads, head_dim);
  if (workspace_bytes < need)
    return set_error(GQA_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  return decode_bwd(q, k_hist, v_hist, probs, d_out, d_scores, d_q, d_k_hist, d_v_hist, history_len,
                    n_heads, n_kv_heads, head_dim, scale, (char*)workspace, (cudaStream_t)stream);
}

gqa_status attn_bwd_simt(const float* Q, const float* K, const float* V, const float* dO,
                         const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                         int seq_len, int n_heads, int n_kv_heads, int head_dim, float scale,
                         void* workspace, size_t workspace_bytes, void* stream) {
  gqa_status r = check_bwd(Q, K, V, dO, LSE, seg, dQ, dK, dV, seq_len, n_heads, n_kv_heads,
                           head_dim, scale, workspace, workspace_bytes);
  if (r != GQA_OK || seq_len == 0) return r;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(workspace, 0, kWsHeader, st) != cudaSuccess)
    return check_launch("workspace header reset");
  if ((r = debug_check_seg(seg, seq_len, workspace, st)) != GQA_OK) return r;
  Shape sh{seq_len, n_heads, n_kv_heads, head_dim, n_heads / n_kv_heads, scale};
  return simt_bwd(Q, K, V, dO, LSE, seg, dQ, dK, dV, sh, (char*)workspace, st, no_rope());
}

}  // extern "C"

namespace gqa {
// attn_bwd and attn_bwd_rope: tensor-core kernels where the shape allows.
static gqa_status bwd_dispatch(const float* Q, const float* K, const float* V, const float* dO,
                               const float* LSE, const uint32_t* seg, float* dQ, float* dK,
                               float* dV, int seq_len, int n_heads, int n_kv_heads, int head_dim,
                               float scale, void* workspace, size_t workspace_bytes, void* stream,
                               const RopeParams& rope, const float* O = nullptr) {
  gqa_status r = check_bwd(Q, K, V, dO, LSE, seg, dQ, dK, dV, seq_len, n_heads, n_kv_heads,
                           head_dim, scale, workspace, workspace_bytes);
  if (r != GQA_OK || seq_len == 0) return r;
  const Shape sh{seq_len, n_heads, n_kv_heads, head_dim, n_heads / n_kv_heads, scale};
  cudaStream_t st = (cudaStream_t)stream;
  if (g_short_path.load() != 0 && short_supported(sh)) {
    const size_t need = short_ws_bytes(seq_len, n_heads, head_dim);
    if (workspace_bytes < need)
      return set_error(GQA_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
    if (cudaMemsetAsync(workspace, 0, kWsHeader, st) != cudaSuccess)
      return check_launch("workspace header reset");
    if ((r = debug_check_seg(seg, seq_len, workspace, st)) != GQA_OK) return r;
    return short_bwd(Q, K, V, dO, LSE, seg, dQ, dK, dV, sh, (char*)workspace, st, rope);
  }
  if (!tc_supported(sh)) {
    if (cudaMemsetAsync(workspace, 0, kWsHeader, st) != cudaSuccess)
      return check_launch("workspace header reset");
    if ((r = debug_check_seg(seg, seq_len, workspace, st)) != GQA_OK) return r;
    return simt_bwd(Q, K, V, dO, LSE, seg, dQ, dK, dV, sh, (char*)workspace, st, rope);
  }
  const size_t need = tc_ws_layout(seq_len, n_heads, n_kv_heads, head_dim).total;
  if (workspace_bytes < need)
    return set_error(GQA_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  if (cudaMemsetAsync(workspace, 0, kWsHeader, st) != cudaSuccess)
    return check_launch("workspace header reset");
  if ((r = debug_check_seg(seg, seq_len, workspace, st)) != GQA_OK) return r;
  return tc_bwd(Q, K, V, dO, LSE, seg, dQ, dK, dV, sh, (char*)workspace, st, rope, O);
}

static gqa_status check_rope(int seq_len, int head_dim, int pos_offset, float base) {
  if (pos_offset < 0) return set_error(GQA_ERR_INVALID_ARG, "pos_offset must be >= 0");
  if (!(base > 0.f) || !isfinite(base)) return set_error(GQA_ERR_INVALID_ARG, "base must be > 0");
  if ((long long)seq_len + pos_offset >= (1LL << 31))
    return set_error(GQA_ERR_INVALID_ARG, "seq_len + pos_offset must be < 2^31");
  (void)head_dim;
  return GQA_OK;
}
}  // namespace gqa

extern "C" {

gqa_status attn_bwd(const float* Q, const float* K, const float* V, const float* dO,
                    const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                    int seq_len, int n_heads, int n_kv_heads, int head_dim, float scale,
                    void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_dispatch(Q, K, V, dO, LSE, seg, dQ, dK, dV, seq_len, n_heads, n_kv_heads, head_dim,
                      scale, workspace, workspace_bytes, stream, no_rope());
}

gqa_status attn_bwd_short(const float* Q, const float* K, const float* V, const float* dO,
                          const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                          int seq_len, int n_heads, int n_kv_heads, int head_dim, float scale,
                          void* workspace, size_t workspace_bytes, void* stream) {
  gqa_status r = check_attn_args(seq_len, n_heads, n_kv_heads, head_dim, scale, 128);
  if (r != GQA_OK || seq_len == 0) return r;
  const Shape sh{seq_len, n_heads, n_kv_heads, head_dim, n_heads / n_kv_heads, scale};
  if (!short_supported(sh))
    return set_error(GQA_ERR_UNSUPPORTED,
                     "short path: seq_len %d, n_heads %d, head_dim %d exceed its limits "
                     "(seq_len <= 2048, tile work <= 2^27)", seq_len, n_heads, head_dim);
  const void* p[] = {Q, K, V, dO, LSE, seg, dQ, dK, dV, workspace};
  const char* nm[] = {"Q", "K", "V", "dO", "LSE", "seg", "dQ", "dK", "dV", "workspace"};
  if ((r = check_ptrs(p, nm, 10)) != GQA_OK) return r;
  const size_t need = short_ws_bytes(seq_len, n_heads, head_dim);
  if (workspace_bytes < need)
    return set_error(GQA_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(workspace, 0, kWsHeader, st) != cudaSuccess)
    return check_launch("workspace header reset");
  if ((r = debug_check_seg(seg, seq_len, workspace, st)) != GQA_OK) return r;
  return short_bwd(Q, K, V, dO, LSE, seg, dQ, dK, dV, sh, (char*)workspace, st, no_rope());
}

gqa_status attn_bwd_o(const float* Q, const float* K, const float* V, const float* dO,
                      const float* O, const float* LSE, const uint32_t* seg, float* dQ, float* dK,
                      float* dV, int seq_len, int n_heads, int n_kv_heads, int head_dim,
                      float scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (seq_len > 0) {
    if (O == nullptr) return set_error(GQA_ERR_INVALID_ARG, "O is NULL");
    if (!aligned16(O)) return set_error(GQA_ERR_INVALID_ARG, "O is not 16-byte aligned");
  }
  return bwd_dispatch(Q, K, V, dO, LSE, seg, dQ, dK, dV, seq_len, n_heads, n_kv_heads, head_dim,
                      scale, workspace, workspace_bytes, stream, no_rope(), O);
}

gqa_status attn_bwd_rope(const float* Q, const float* K, const float* V, const float* dO,
                         const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                         int seq_len, int n_heads, int n_kv_heads, int head_dim, float scale,
                         int pos_offset, float base, void* workspace, size_t workspace_bytes,
                         void* stream) {
  const gqa_status r = check_rope(seq_len, head_dim, pos_offset, base);
  if (r != GQA_OK) return r;
  return bwd_dispatch(Q, K, V, dO, LSE, seg, dQ, dK, dV, seq_len, n_heads, n_kv_heads, head_dim,
                      scale, workspace, workspace_bytes, stream,
                      make_rope(head_dim, pos_offset, base));
}

gqa_status rope_bwd_inplace(float* dX, int seq_len, int n_heads, int head_dim, int pos_offset,
                            float base, void* stream) {
  if (seq_len < 0) return set_error(GQA_ERR_INVALID_ARG, "seq_len must be >= 0");
  if (n_heads <= 0) return set_error(GQA_ERR_INVALID_ARG, "n_heads must be > 0");
  if (head_dim <= 0 || head_dim % 4 != 0)
    return set_error(GQA_ERR_INVALID_ARG, "head_dim must be a positive multiple of 4");
  if (head_dim > 128) return set_error(GQA_ERR_UNSUPPORTED, "head_dim > 128 has no kernel");
  if (pos_offset < 0) return set_error(GQA_ERR_INVALID_ARG, "pos_offset must be >= 0");
  if (!(base > 0.f) || !isfinite(base)) return set_error(GQA_ERR_INVALID_ARG, "base must be > 0");
  if ((long long)seq_len * n_heads * head_dim >= (1LL << 31))
    return set_error(GQA_ERR_UNSUPPORTED, "buffer too large (>= 2^31 elements)");
  if (seq_len == 0) return GQA_OK;
  if (dX == nullptr) return set_error(GQA_ERR_INVALID_ARG, "dX is NULL");
  if (!aligned16(dX)) return set_error(GQA_ERR_INVALID_ARG, "dX is not 16-byte aligned");
  return rope_bwd_launch(dX, seq_len, n_heads, head_dim, pos_offset, base, (cudaStream_t)stream);
}

gqa_status gqa_wait_selftest(void* workspace, size_t workspace_bytes, long long limit_cycles,
                             void* stream) {
  if (workspace == nullptr || !aligned16(workspace))
    return set_error(GQA_ERR_INVALID_ARG, "workspace is NULL or not 16-byte aligned");
  if (workspace_bytes < kWsHeader)
    return set_error(GQA_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes,
                     kWsHeader);
  if (limit_cycles <= 0 || limit_cycles > 100000000LL)
    return set_error(GQA_ERR_INVALID_ARG, "limit_cycles must be in (0, 1e8]");
  return wait_selftest(workspace, limit_cycles, (cudaStream_t)stream);
}

gqa_status gqa_grid_barrier_selftest(void* workspace, size_t workspace_bytes,
                                     long long limit_cycles, void* stream) {
  if (workspace == nullptr || !aligned16(workspace))
    return set_error(GQA_ERR_INVALID_ARG, "workspace is NULL or not 16-byte aligned");
  if (workspace_bytes < kWsHeader)
    return set_error(GQA_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes,
                     kWsHeader);
  if (limit_cycles <= 0 || limit_cycles > 100000000LL)
    return set_error(GQA_ERR_INVALID_ARG, "limit_cycles must be in (0, 1e8]");
  return grid_barrier_selftest(workspace, limit_cycles, (cudaStream_t)stream);
}

gqa_status attn_read_device_status(const void* workspace, void* stream) {
  if (workspace == nullptr) return set_error(GQA_ERR_INVALID_ARG, "workspace is NULL");
  uint32_t word = 0;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return check_launch("status read");
  if (cudaStreamSynchronize(st) != cudaSuccess) return check_launch("status read sync");
  if (word & kStatusTimeout)
    return set_error(GQA_ERR_DEVICE_TIMEOUT, "device status word 0x%08x: a bounded wait gave up", word);
  if (word & kStatusCheck)
    return set_error(GQA_ERR_DEVICE_CHECK,
                     "device status word 0x%08x: a device-side check of the debug build failed "
                     "(0x1 seg[s] > s, 0x2/0x4 query-major store/load, 0x8/0x10 key-major "
                     "store/load, 0x20 short path, 0x40 CUDA-core path, 0x80 forward)", word);
  if (word != 0)
    return set_error(GQA_ERR_DEVICE_TIMEOUT, "device status word 0x%08x", word);
  return GQA_OK;
}

}  // extern "C"
