// Internal definitions shared by the translation units of libgqa_attn.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

#include "gqa_attn.h"   // include/ is on the include path (build.py)
#include "rope_common.cuh"

namespace gqa {

// ---------------------------------------------------------------------------
// Workspace layout (caller-allocated, 256-byte aligned pieces)
//   [0, 256)                       header: status word (uint32) at byte 0
//   [kWsD, kWsD + S*H*4)           D[i, h] = sum_j P_ij dP_ij   (fp32, [S, H])
//   [kWsD + align256(S*H*4), ...)  per query tile: smallest seg in the tile
//                                  (uint32, one per 64-row tile and one per
//                                  128-row tile)
// ---------------------------------------------------------------------------
constexpr size_t kWsHeader = 256;

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t d_off;       // D
  size_t minseg64;    // min seg per 64-row query tile
  size_t minseg128;   // min seg per 128-row query tile
  size_t total;
};

inline WsLayout ws_layout(int S, int H) {
  WsLayout w;
  w.d_off = kWsHeader;
  size_t off = w.d_off + align256(size_t(S) * size_t(H) * sizeof(float));
  w.minseg64 = off;
  off += align256(size_t((S + 63) / 64) * sizeof(uint32_t));
  w.minseg128 = off;
  off += align256(size_t((S + 127) / 128) * sizeof(uint32_t));
  w.total = off;
  return w;
}

// The tensor-core path needs more: K^T per kv head, [Hk*d rows][ld_kt],
// ld_kt = S rounded up to 32 (so TMA row strides stay 128-byte multiples).
// Q^T and dO^T per kv group, [Hk*d rows][ld_qt] with column q*G + h'
// (ld_qt = S*G rounded up to 32), and the minimum seg per key-major block of
// (128 or 64)/G queries.
struct TcWsLayout {
  long long ld_kt, ld_qt;
  long long rows_kp;   // rows of K' (S rounded up to 64; 0 when there is no K')
  long long ld_meta;   // key-major column records per kv head (S*G rounded up to 64)
  size_t kt_off, qt_off, dot_off, blk_off, blkmax_off, kp_off, meta_off, part_off;
  size_t total;
};
TcWsLayout tc_ws_layout(int S, int H, int Hk, int d);

// ---------------------------------------------------------------------------
// Device status word (workspace byte 0, cleared by each call). A bounded wait
// that gives up ORs kStatusTimeout | its site. In the debug build
// (-DGQA_CHECKS, built as libgqa_attn_checks.so) a failed device-side check
// ORs kStatusCheck | its site and the checked access is skipped (no trap, no
// fault). attn_read_device_status reports GQA_ERR_DEVICE_TIMEOUT, else
// GQA_ERR_DEVICE_CHECK. In the release build the checks compile to nothing.
// ---------------------------------------------------------------------------
constexpr uint32_t kStatusTimeout = 0x80000000u, kStatusCheck = 0x40000000u;
enum : uint32_t {
  kChkSeg = 1u << 0,        // seg[s] > s somewhere (the documented precondition)
  kChkTcQmStore = 1u << 1,  // query-major kernel: dQ / D / Q^T / dO^T store index
  kChkTcQmLoad = 1u << 2,   // query-major kernel: Q / dO row or TMA coordinate
  kChkTcKmStore = 1u << 3,  // key-major kernel: dK / dV / part-sum store index
  kChkTcKmLoad = 1u << 4,   // key-major kernel: K row, column metadata or TMA coordinate
  kChkShort = 1u << 5,      // short path: partial or final store index
  kChkSimt = 1u << 6,       // CUDA-core path: dQ / dK / dV / D store index
  kChkFwd = 1u << 7,        // tensor-core forward: O / LSE store index or TMA coordinate
};
#ifdef GQA_CHECKS
__device__ __forceinline__ bool dcheck(uint32_t* status, bool ok, uint32_t site) {
  if (!ok) atomicOr(status, kStatusCheck | site);
  return ok;
}
#define GQA_DCHECK(status, cond, site) ::gqa::dcheck((status), (cond), (site))
#else
#define GQA_DCHECK(status, cond, site) true
#endif
// Debug build: one pass over seg that flags seg[s] > s (kChkSeg) in the
// status word at `ws`; the release build launches nothing.
gqa_status debug_check_seg(const uint32_t* seg, int S, void* ws, cudaStream_t st);

// Problem description passed by value to kernels.
struct Shape {
  int S, H, Hk, d, G;   // seq_len, n_heads, n_kv_heads, head_dim, H / Hk
  float scale;
};

// Measurement hook (gqa_profile_events): one-shot events around the dominant
// stage of the next backward call on this host thread.
struct ProfileHook {
  cudaEvent_t before = nullptr, after = nullptr;
  const char* stage = "";
};
ProfileHook& profile_hook();
inline void profile_before(cudaStream_t st, const char* stage) {
  ProfileHook& h = profile_hook();
  h.stage = stage;
  if (h.before) cudaEventRecord(h.before, st);
}
inline void profile_after(cudaStream_t st) {
  ProfileHook& h = profile_hook();
  if (h.after) cudaEventRecord(h.after, st);
  h.before = h.after = nullptr;
}

// Count of kernels this library has launched (gqa_launch_count).
void note_launch(int n = 1);

// Host-side error reporting (thread-local one-line reason).
gqa_status set_error(gqa_status st, const char* fmt, ...);
gqa_status check_launch(const char* what);

// Argument checks shared by the attention entry points; returns GQA_OK or an
// error with gqa_last_error() set.
gqa_status check_attn_args(int S, int H, int Hk, int d, float scale, int max_d);
bool aligned16(const void* p);

// SIMT (CUDA-core) kernels, simt_attn.cu
gqa_status simt_fwd_lse(const float* Q, const float* K, const float* V, const uint32_t* seg,
                        float* O, float* LSE, const Shape& sh, cudaStream_t st);
// With rope.on, the RoPE backward is applied to the attention gradients of Q
// and K before they are added to dQ / dK (attn_bwd_rope).
gqa_status simt_bwd(const float* Q, const float* K, const float* V, const float* dO,
                    const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                    const Shape& sh, char* ws, cudaStream_t st, const RopeParams& rope);

gqa_status tile_minseg(const uint32_t* seg, int S, int tile, uint32_t* out, cudaStream_t st,
                       uint32_t* out_max = nullptr);

// Tensor-core backward, tc_bwd.cu: true if this shape has a tensor-core path.
bool tc_supported(const Shape& sh);
// With O != nullptr, D = rowsum(dO * O) is formed by a row-dot pass instead
// of the query-major kernel's first pass (attn_bwd_o).
gqa_status tc_bwd(const float* Q, const float* K, const float* V, const float* dO,
                  const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                  const Shape& sh, char* ws, cudaStream_t st, const RopeParams& rope,
                  const float* O = nullptr);

gqa_status wait_selftest(void* workspace, long long limit_cycles, cudaStream_t st);

// Single-launch backward for short sequences, short_bwd.cu: one cooperative
// launch (three phases split by bounded grid barriers). Supported for
// seq_len <= 2048 with at most kShortMaxWork multiply-adds per contraction,
// counted over whole 32 x 32 (query, key) tiles:
//   nt (nt + 1) / 2 * 32 * 32 * n_heads * padded head_dim <= kShortMaxWork,
// nt = ceil(seq_len / 32). Above that the tensor-core kernels are faster.
constexpr long long kShortMaxWork = 1LL << 27;
bool short_supported(const Shape& sh);
size_t short_ws_bytes(int S, int H, int d);
// Test helper: the short path's bounded grid barrier, made to run out.
gqa_status grid_barrier_selftest(void* workspace, long long limit_cycles, cudaStream_t st);
gqa_status short_bwd(const float* Q, const float* K, const float* V, const float* dO,
                     const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                     const Shape& sh, char* ws, cudaStream_t st, const RopeParams& rope);

// Tensor-core host helpers (tc_bwd.cu): the 128-byte-swizzled panel view of a
// row-major matrix (dims 32 floats x rows x panels; one box fills box_panels
// panels of box_rows x 128 B) and the group transpose Xt [Hk*d][ld] of
// X [S][Hk*Gx][d].
gqa_status tc_map_panels(CUtensorMap* m, const float* base, long long ld, long long rows,
                         long long n_panels, int box_rows, int box_panels);
gqa_status tc_transpose(const float* X, float* Xt, int S, int Hk, int Gx, int d, long long ld,
                        cudaStream_t st);

// Tensor-core forward, tc_fwd.cu: O and LSE (d in {32, 64, 128}); the
// workspace holds the status header and V^T.
bool tc_fwd_supported(const Shape& sh);
size_t tc_fwd_ws_bytes(int S, int Hk, int d);
gqa_status tc_fwd(const float* Q, const float* K, const float* V, const uint32_t* seg, float* O,
                  float* LSE, const Shape& sh, char* ws, cudaStream_t st);

// RoPE backward, rope_bwd.cu
size_t decode_ws_bytes(int L, int H, int d);
gqa_status decode_bwd(const float* q, const float* k_hist, const float* v_hist, const float* probs,
                      const float* d_out, float* d_scores, float* d_q, float* d_k, float* d_v,
                      int L, int H, int Hk, int d, float scale, char* ws, cudaStream_t st);

gqa_status rope_bwd_launch(float* X, int S, int H, int d, int pos_offset, float base,
                           cudaStream_t st);

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace gqa
