/*
 * gqa_attn.h — C ABI of libgqa_attn.so: causal grouped-query attention on one
 * GB300 (sm_103a). Forward producing O and the log-sum-exp, the backward pass
 * from a saved log-sum-exp, and the interleaved RoPE backward.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller. The library
 *    never allocates, frees or keeps them, and never synchronises the stream
 *    (attn_read_device_status is the one exception, and says so).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Every launch is asynchronous on it.
 *  - Layouts are row-major fp32 (backward_attention.wgsl, bindings of kernel
 *    attention_backward): Q, dO, dQ, O are [seq_len, n_heads * head_dim], head
 *    h in columns [h*head_dim, (h+1)*head_dim); K, V, dK, dV are
 *    [seq_len, n_kv_heads * head_dim]; LSE is [seq_len, n_heads]; seg is
 *    [seq_len] uint32.
 *  - GQA grouping is blocked: query head h reads kv head h / (n_heads /
 *    n_kv_heads) (backward_attention.wgsl, attention_backward: kv_h =
 *    h / q_per_group; tang llm.rs, causal_attention_fused).
 *  - Masking: key j is visible to query i iff seg[i] <= j <= i, where seg[i]
 *    is the first position of the document holding i (backward_attention.wgsl,
 *    attention_backward: doc_start / causal_len). seg[i] <= i is a
 *    precondition; seg need not be monotone. seg all zero = pure causal.
 *  - Arguments are checked on the host before any launch. A bad argument
 *    returns GQA_ERR_INVALID_ARG (or GQA_ERR_UNSUPPORTED for a valid shape the
 *    library has no kernel for) and launches nothing; gqa_last_error() then
 *    holds a one-line reason. seq_len == 0 is a no-op that returns GQA_OK.
 *  - Pointers must be 16-byte aligned and n_heads*head_dim, n_kv_heads*head_dim
 *    multiples of 4 (row starts on 16-byte boundaries, as TMA requires).
 *  - Sizes: seq_len * max(n_heads, n_kv_heads) * head_dim must stay below 2^31.
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARG = 1,    /* bad pointer, size, alignment or workspace        */
  GQA_ERR_UNSUPPORTED = 2,    /* valid shape with no kernel (e.g. head_dim > 128) */
  GQA_ERR_CUDA = 3,           /* a CUDA launch or copy failed                     */
  GQA_ERR_DEVICE_TIMEOUT = 4, /* a bounded device-side wait gave up (see below)   */
  GQA_ERR_DEVICE_CHECK = 5    /* debug build only: a device-side check failed     */
} gqa_status;

/*
 * attn_fwd_lse — forward attention with the log-sum-exp.
 * tang llm.rs, causal_attention_fused (row max, sum of exponentials, weighted
 * V) with the document mask of backward_attention.wgsl; the LSE is the one the
 * backward consumes (backward_attention.wgsl header: P = exp(scale*Q.K - LSE)).
 *   O[i, h]   = sum_j exp(scale*q_i.k_j - LSE[i,h]) v_j   over visible j
 *   LSE[i, h] = ln sum_j exp(scale*q_i.k_j)               (natural log, scale in)
 * In:  Q, K, V, seg. Out (overwritten): O, LSE. head_dim: 4..128, multiple of 4.
 * fp32 on CUDA cores; needs no workspace (attn_fwd is the tensor-core form).
 */
gqa_status attn_fwd_lse(const float* Q, const float* K, const float* V, const uint32_t* seg,
                        float* O, float* LSE, int seq_len, int n_heads, int n_kv_heads,
                        int head_dim, float scale, void* stream);

/*
 * attn_fwd_workspace_bytes / attn_fwd — the same forward as attn_fwd_lse (O
 * and LSE overwritten, same definitions and arguments), on tensor cores for
 * head_dim 32, 64, 128 (tcgen05 kind::tf32: S = scale Q.K^T with TF32
 * operands, fp32 accumulation; one pass over the visible keys with an online
 * softmax: a running row max m and sum l, P = exp(s - m) (a TF32 operand of
 * O += P V), the accumulator rescaled when m rises; at the end O = O / l and
 * LSE = m + ln l), else on CUDA cores.
 * workspace: >= attn_fwd_workspace_bytes(...) device bytes, caller-owned (a
 * status header and a transposed copy of V). Bounded device waits report
 * through attn_read_device_status(workspace) as for attn_bwd.
 */
size_t attn_fwd_workspace_bytes(int seq_len, int n_heads, int n_kv_heads, int head_dim);
gqa_status attn_fwd(const float* Q, const float* K, const float* V, const uint32_t* seg, float* O,
                    float* LSE, int seq_len, int n_heads, int n_kv_heads, int head_dim, float scale,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_bwd_workspace_bytes / attn_decode_bwd — decode-style attention
 * backward from saved probabilities: one query per head against history_len
 * cached keys (rullama training.rs, attention_backward_dq_chained: d_q and the
 * staged d_scores from k_hist, v_hist, probs, d_out; attention_backward_dkv_chained:
 * d_k_hist, d_v_hist from q, probs, d_out, d_scores). The page gives the
 * bindings and launch shapes only; the arithmetic is the softmax backward of
 * probs = softmax_j(scale * q_h . k_j), kv head g(h) = h / (n_heads / n_kv_heads):
 *   dP[h, j]       = d_out_h . v_j,   D_h = sum_j probs[h, j] dP[h, j]
 *   d_scores[h, j] = probs[h, j] (dP[h, j] - D_h)      (gradient of the scores)
 *   d_q_h      += scale * sum_j d_scores[h, j] k_j
 *   d_k_hist_j += scale * sum_{h in g} d_scores[h, j] q_h
 *   d_v_hist_j += sum_{h in g} probs[h, j] d_out_h
 * Layouts (row-major fp32, device memory, caller-owned): q, d_out, d_q
 * [n_heads * head_dim]; k_hist, v_hist, d_k_hist, d_v_hist
 * [history_len, n_kv_heads * head_dim]; probs, d_scores [n_heads, history_len].
 * d_q, d_k_hist, d_v_hist accumulate (+=); d_scores is overwritten (it also
 * stages dP between the passes). probs is used as given (its rows need not
 * sum to one). head_dim in {32, 64, 96, 128} (else GQA_ERR_UNSUPPORTED);
 * n_kv_heads <= 65535; every pointer non-NULL and 16-byte aligned;
 * workspace >= attn_decode_bwd_workspace_bytes(...) bytes, any contents.
 * history_len == 0 is a no-op. Deterministic (no atomics); CUDA cores,
 * bound by HBM bandwidth. Errors are returned before any launch.
 */
size_t attn_decode_bwd_workspace_bytes(int history_len, int n_heads, int n_kv_heads, int head_dim);
gqa_status attn_decode_bwd(const float* q, const float* k_hist, const float* v_hist,
                           const float* probs, const float* d_out, float* d_scores, float* d_q,
                           float* d_k_hist, float* d_v_hist, int history_len, int n_heads,
                           int n_kv_heads, int head_dim, float scale, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * attn_bwd_workspace_bytes — bytes of device workspace attn_bwd (and
 * attn_bwd_o, attn_bwd_rope, attn_bwd_short, attn_bwd_simt) needs for this
 * shape (a multiple of 256). It depends on the shape alone, not on the device
 * (the part it reserves for a split key-tile walk is sized for devices with
 * up to 192 SMs; a device with more SMs splits no further than that). The
 * caller allocates it (any contents) and may reuse it across calls that do
 * not overlap on the GPU.
 */
size_t attn_bwd_workspace_bytes(int seq_len, int n_heads, int n_kv_heads, int head_dim);

/*
 * attn_bwd — backward pass of causal GQA attention from a saved LSE.
 * backward_attention.wgsl, header and kernel attention_backward (P recomputed
 * from the saved LSE, dP = dO.V, D = sum_j P*dP, dS = scale*P*(dP - D)); the
 * explicit-matrix form is tang llm.rs, GpuCausalAttention::backward.
 *   dQ[i,h] += sum_j dS_ij k_j,  dK[j,g] += sum_{h in g, i} dS_ij q_i,
 *   dV[j,g] += sum_{h in g, i} P_ij dO_i
 * In:  Q, K, V, dO, LSE, seg, scale. In/out: dQ, dK, dV are ACCUMULATED (+=),
 * as in the streaming kernel: zero them before the first call of a step.
 * workspace: >= attn_bwd_workspace_bytes(...) device bytes, caller-owned.
 * Path: short problems (those attn_bwd_short accepts) run its single
 * cooperative launch on CUDA cores, unless gqa_set_short_path(0) turned that
 * off; otherwise head_dim 32, 64 or 128 runs the tensor-core path where it is
 * built, and other multiples of 4 up to 128 the CUDA-core path
 * (attn_bwd_simt). The result stays within fp32/TF32 rounding of the exact
 * value; which path ran decides the rounding. (At head_dim 128 the
 * tensor-core path forms dQ in one pass over the keys as
 * scale * (sum_j P_ij dP_ij k_j - D_i sum_j P_ij k_j), equal to sum_j dS_ij k_j
 * in exact arithmetic.)
 */
gqa_status attn_bwd(const float* Q, const float* K, const float* V, const float* dO,
                    const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                    int seq_len, int n_heads, int n_kv_heads, int head_dim, float scale,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_bwd_short — attn_bwd for short sequences in ONE kernel launch (the
 * analogue of backward_attention.wgsl's attention_backward_short /
 * attention_backward_short_dKdV, which serve short sequences with one
 * dispatch each and keep P and dS for every (query, key, head) in an
 * O(seq_len^2 * n_heads) scratch buffer; none of that is kept here). Work is
 * cut into cells of 32 query rows x 32 keys x one query head; a cooperative
 * launch runs three phases split by grid-wide barriers: (A) per cell, the
 * partial row sums of P * dP; (B) per cell, D_i = the row's partials summed,
 * dS = scale * P * (dP - D) and the cell's partial dQ = dS K, dK = dS^T Q,
 * dV = P^T dO; (C) per output tile, the partials summed in a fixed order
 * (dK, dV over the GQA group's query heads and the query tiles) and added
 * once to dQ, dK, dV. fp32 FFMA on CUDA cores, deterministic.
 * Limits: seq_len <= 2048 and nt*(nt+1)/2 * 1024 * n_heads * hp <= 2^27, where
 * nt = ceil(seq_len / 32) and hp = head_dim rounded up to 32, 64 or 128;
 * beyond them GQA_ERR_UNSUPPORTED (attn_bwd then runs its other paths).
 * Same arguments, semantics (+=), workspace query (attn_bwd_workspace_bytes
 * covers it) and errors as attn_bwd. Every grid-barrier wait is bounded
 * (~1 s); one that gives up sets the status word that
 * attn_read_device_status reports as GQA_ERR_DEVICE_TIMEOUT.
 */
gqa_status attn_bwd_short(const float* Q, const float* K, const float* V, const float* dO,
                          const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                          int seq_len, int n_heads, int n_kv_heads, int head_dim, float scale,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * gqa_set_short_path — process-wide switch: whether attn_bwd, attn_bwd_o and
 * attn_bwd_rope send the shapes attn_bwd_short accepts to it (1, the
 * default) or to their tensor-core / CUDA-core kernels (0). Returns the
 * previous setting. Not tied to a stream: change it only between calls.
 */
int gqa_set_short_path(int enable);

/*
 * attn_bwd_o — attn_bwd for callers that kept the forward output O [seq_len,
 * n_heads * head_dim] (e.g. from attn_fwd_lse): D_i = sum_j P_ij dP_ij is
 * formed as the row dot product dO_i . O_i (equal when O and LSE come from
 * the same forward: O_i = sum_j P_ij v_j; cf. backward_attention.wgsl, where
 * D is the Pass A row sum), which replaces the query-major kernel's first
 * pass and its two contractions (S and dP). The pages have no separate
 * entry point for this; it is this library's addition. Same arguments,
 * workspace, semantics (+=) and errors as attn_bwd, plus O (non-NULL, 16-byte
 * aligned). Where the short path (attn_bwd_short) or the CUDA-core path
 * (head_dim not 32/64/128) runs, O is not read and D is formed as in attn_bwd.
 */
gqa_status attn_bwd_o(const float* Q, const float* K, const float* V, const float* dO,
                      const float* O, const float* LSE, const uint32_t* seg, float* dQ, float* dK,
                      float* dV, int seq_len, int n_heads, int n_kv_heads, int head_dim,
                      float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_bwd_rope — attn_bwd followed by the interleaved RoPE backward on the
 * attention gradients of Q and K (the step of a RoPE model: the pages apply
 * rope_q_backward / rope_k_backward of backward_attention.wgsl, and tang
 * llm.rs interleaved_rope_backward, to dQ and dK after the attention
 * backward). The rotation is fused into the kernels' final writes:
 *   dQ[i,h] += R_i^T (attention dQ[i,h]),  dK[j,g] += R_j^T (attention dK[j,g]),
 *   dV[j,g] += attention dV[j,g]
 * where R_t rotates pair p of a head by t*base^(-2p/head_dim), t = pos_offset
 * + row (the same rotation as rope_bwd_inplace). With dQ, dK zeroed first
 * this equals attn_bwd then rope_bwd_inplace on dQ and dK; with non-zero
 * dQ / dK only the new contribution is rotated. Same arguments, workspace,
 * paths and errors as attn_bwd, plus pos_offset >= 0 and base > 0
 * (GQA_ERR_INVALID_ARG otherwise).
 */
gqa_status attn_bwd_rope(const float* Q, const float* K, const float* V, const float* dO,
                         const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                         int seq_len, int n_heads, int n_kv_heads, int head_dim, float scale,
                         int pos_offset, float base, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * attn_bwd_simt — the same operation and contract as attn_bwd, computed with
 * fp32 FFMA on CUDA cores only (no tensor cores): exact fp32 products, any
 * head_dim that is a multiple of 4 up to 128. Deterministic.
 */
gqa_status attn_bwd_simt(const float* Q, const float* K, const float* V, const float* dO,
                         const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                         int seq_len, int n_heads, int n_kv_heads, int head_dim, float scale,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_bwd_noalloc — attn_bwd for callers that cannot allocate device memory
 * (no counterpart on the pages: an addition of this library). Some callers
 * are handed only their input and output buffers — a plugin inside a host
 * engine, code where the process's memory manager forbids raw cudaMalloc after
 * start-up, a binding with no device allocator — and so cannot provide the
 * workspace attn_bwd needs. This entry point takes the same arguments minus
 * the workspace and uses a fixed 4 MiB device array inside the library
 * instead; it calls no allocator. Limits: seq_len * n_heads must fit that
 * array (about 1M, e.g. 16384 x 32); larger shapes return
 * GQA_ERR_UNSUPPORTED before any launch. Every GPU that loads the library
 * holds the array until exit. All calls share it: calls whose GPU work
 * overlaps (other streams or host threads) race and give wrong results. The
 * first call on a device looks up the array's address with that device
 * current; make that first call before any stream capture. The address is
 * kept with the id of the device's current CUDA context and looked up again
 * when another context is current (after cudaDeviceReset the array may have
 * moved). It runs the CUDA-core kernels (same results as attn_bwd_simt); dQ, dK, dV are
 * accumulated (+=) as in attn_bwd.
 */
gqa_status attn_bwd_noalloc(const float* Q, const float* K, const float* V, const float* dO,
                            const float* LSE, const uint32_t* seg, float* dQ, float* dK,
                            float* dV, int seq_len, int n_heads, int n_kv_heads, int head_dim,
                            float scale, void* stream);

/*
 * rope_bwd_inplace — interleaved RoPE backward, in place on dX
 * [seq_len, n_heads * head_dim] (backward_attention.wgsl, rope_q_backward /
 * rope_k_backward; tang llm.rs, interleaved_rope_backward). For pair p <
 * head_dim/2 of every head at row s, with t = pos_offset + s and
 * theta = t * base^(-2p/head_dim):
 *   (x0, x1) <- (x0*cos theta + x1*sin theta, -x0*sin theta + x1*cos theta)
 * on columns (2p, 2p+1). The per-pair frequencies base^(-2p/head_dim) are
 * formed in fp64 on the host; the angle is reduced modulo 2*pi before fp32
 * sin/cos, so large positions keep fp32 accuracy (an fp32 product alone is
 * ~1e-3 rad off at t = 16k): for t < 2^15 in fp32 (the frequency split into
 * two floats, t * f_hi carried exactly with its FMA error term, 2*pi split
 * into three constants: Cody & Waite's reduction), for larger t in fp64.
 * head_dim a multiple of 4 (at most 128), base > 0, pos_offset >= 0.
 */
gqa_status rope_bwd_inplace(float* dX, int seq_len, int n_heads, int head_dim,
                            int pos_offset, float base, void* stream);

/*
 * attn_read_device_status — test/debug helper: SYNCHRONISES `stream`, then
 * reads the device-side status word that the last attn_bwd on this workspace
 * left (GQA_OK, or GQA_ERR_DEVICE_TIMEOUT if a bounded wait inside a kernel
 * gave up and the kernel returned early instead of hanging).
 *
 * Debug build. libgqa_attn_checks.so is the same library compiled with
 * -DGQA_CHECKS (stand-ins for a memory checker, after the defensive clamps
 * and guards of backward_attention.wgsl's attention_backward_short and
 * attention_backward): every call taking a workspace first checks the
 * precondition seg[s] <= s on the device, and the kernels check the indices
 * of their global stores and loads (and the coordinates of their TMA boxes)
 * against the tensors' extents. A failed check sets a bit in the status word
 * (0x40000000 | site: 0x1 seg, 0x2/0x4 query-major store/load, 0x8/0x10
 * key-major store/load, 0x20 short path, 0x40 CUDA-core path, 0x80 forward)
 * and skips the access; it never traps. attn_read_device_status then
 * returns GQA_ERR_DEVICE_CHECK (GQA_ERR_DEVICE_TIMEOUT takes precedence).
 * In the release library the checks are compiled out.
 */
gqa_status attn_read_device_status(const void* workspace, void* stream);

/*
 * gqa_profile_events — measurement hook (no counterpart on the pages). When
 * both are non-NULL cudaEvent_t handles, the next backward (attn_bwd and its
 * variants) or tensor-core forward (attn_fwd) call on this host thread
 * records `before` on its stream immediately before
 * its dominant kernel stage and `after` immediately after it, then clears the
 * hook. The events are owned by the caller. Stage: the whole two-kernel
 * backward on the CUDA-core path; both tensor-core kernels (query-major and
 * key-major) on the tensor-core path; the one cooperative launch on the short
 * path; the tensor-core kernel of attn_fwd. gqa_profile_stage_name() names it.
 */
void gqa_profile_events(void* before, void* after);
const char* gqa_profile_stage_name(void);

/* Number of kernels this library has launched in this process (all threads). */
unsigned long long gqa_launch_count(void);

/*
 * gqa_wait_selftest — test helper for the device-side failure path (no
 * counterpart on the pages). Launches one thread that waits, through the same
 * bounded mbarrier wait the tensor-core kernels use, on a barrier that nothing
 * arrives on, with a limit of limit_cycles SM cycles (at most 1e8, i.e. well
 * under a second). The wait gives up, sets the status word in `workspace`
 * (>= 256 bytes, its header is cleared first) and the kernel returns; a
 * following attn_read_device_status() then reports GQA_ERR_DEVICE_TIMEOUT and
 * the CUDA context stays usable. Nothing hangs and nothing faults.
 */
gqa_status gqa_wait_selftest(void* workspace, size_t workspace_bytes, long long limit_cycles,
                             void* stream);

/*
 * gqa_grid_barrier_selftest — the same check for attn_bwd_short's grid-wide
 * barrier (no counterpart on the pages): a cooperative launch of two CTAs
 * waits, through that bounded barrier, for one arrival more than the grid
 * makes, with a limit of limit_cycles SM cycles (at most 1e8). The wait gives
 * up, sets the status word in `workspace` (>= 256 bytes, header cleared
 * first; bit 0x400 marks this site), both CTAs return, and
 * attn_read_device_status() reports GQA_ERR_DEVICE_TIMEOUT. Nothing hangs or
 * faults, and the context stays usable.
 */
gqa_status gqa_grid_barrier_selftest(void* workspace, size_t workspace_bytes,
                                     long long limit_cycles, void* stream);

/* Static string naming a status code. */
const char* gqa_status_str(gqa_status status);

/* One-line reason for the last non-OK status returned on this host thread. */
const char* gqa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
