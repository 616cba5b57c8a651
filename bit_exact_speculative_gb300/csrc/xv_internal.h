// Host-side internals shared by the translation units of libxv.so.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/xv.h"

namespace xv {

// Records the message for xv_last_error() and returns `code`.
xv_status fail(xv_status code, const char* fmt, ...);
// Checks a CUDA runtime result; on failure records it and returns XV_ERR_CUDA.
xv_status cuda_check(cudaError_t e, const char* what);
// Kernel kinds of the launch trace.
enum Kind : int { K_GEMM = 0, K_GDN, K_ATTN_SPLIT, K_ATTN_COMBINE, K_KV_APPEND, K_EMBED, K_RMSNORM, K_SWIGLU,
                  K_GATES, K_ARGMAX, K_ACCEPT, K_COMMIT, K_ZERO, K_CONV, K_GNORM, K_GEMM_COMBINE, K_TILE, K_COUNT };
// Call right before a launch on stream s (records the opening trace event when tracing).
void trace_pre(cudaStream_t s);
// Checks the launch just made on the calling thread, counts it and closes its trace record.
xv_status launched(const char* what, cudaStream_t s, int kind, long long bytes);
// Programmatic dependent launch between the library's kernels (on by default).
bool overlap_enabled();
// Launches `kern` on stream s with the programmatic-serialization attribute when
// overlap is enabled: the kernel may start before its predecessor ends, and it
// calls griddep_wait() before touching memory that earlier kernels produce or read.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = overlap_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
// Same, as clusters of `cluster` CTAs (cluster dimensions given as a dim3).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                    dim3 cluster, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = overlap_enabled() ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster.x;
    attr[1].val.clusterDim.y = cluster.y;
    attr[1].val.clusterDim.z = cluster.z;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
// Device address of the library's device-side error word for the current device.
unsigned* device_error_word();
// Raises fn's dynamic shared-memory limit to at least `bytes` (and, with max_carveout, asks for the
// largest shared-memory carveout) on the current device, once per device and kernel; thread-safe.
xv_status kernel_smem_once(const void* fn, int bytes, bool max_carveout, const char* what);
// Number of SMs of the current device (looked up once per device; thread-safe).
xv_status device_sm_count(int* out);

// cuTensorMapEncodeTiled through the runtime's driver entry point.
xv_status encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swizzle);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// ---- GEMM (gemm.cu)
constexpr int GEMM_BN = 128;   // weight rows per CTA (MMA M)
constexpr int GEMM_BK = 64;    // K elements per pipeline stage (one 128-byte swizzle row)
constexpr int GEMM_TOK = 64;   // token columns of every MMA (MMA N), whatever M is
int gemm_splits(int N, int K);
size_t gemm_workspace_size(int M, int N, int K);
// Bytes at the start of a GEMM workspace that hold the tile arrival counters (zero between calls).
constexpr size_t GEMM_COUNTER_BYTES = 1024;
// Whether a GEMM of this shape combines its split-K partials through the workspace's tile counters.
bool gemm_uses_counters(int M, int N, int K);
// defer_part: when the GEMM splits K into more segments than a cluster combines, it writes its
// partials [S][M][N] and returns them and S instead of combining them (for any M; else
// *defer_part = nullptr): the caller adds them in segment order.
// Weight layouts: row-major [N, K]; tiled (gemm_tile_weights_launch); gated tiled, a gate/up
// weight [2F, K] whose tiles pair 64 gate rows with the 64 up rows of the same features, read by
// the GEMM with the SwiGLU fused (N = 2F weight rows in, F bf16 activations per row out, never
// split).
enum WLayout : int { W_ROWS = 0, W_TILED = 1, W_GATED = 2 };
// amax (fp32 out, unsplit shapes only): also writes, for every row m and weight tile t, the tile's
// maximum and its lowest index as amax[m * ceil(N/128) + t] = (value, index bits); Y may then be
// null (no outputs written).
xv_status gemm_launch(const uint16_t* X, int ldx, const uint16_t* W, WLayout wl, void* Y, int ldy, bool f32out, int M,
                      int N, int K, void* ws, size_t ws_bytes, cudaStream_t s, float** defer_part = nullptr,
                      int* defer_S = nullptr, float2* amax = nullptr);
// The tiled weight layout: [ceil(N/128)][ceil(K/64)][128][64] bf16, zero past N and K.
size_t gemm_tiled_bytes(int N, int K);
xv_status gemm_tile_weights_launch(const uint16_t* W, int N, int K, bool gated, uint16_t* Wt, cudaStream_t s);

// ---- GDN (gdn.cu)
// Steps one GDN call stages: up to XV_KMAX replayed ones and XV_KMAX speculative ones.
constexpr int XV_GDN_MAX_STAGED = 2 * XV_KMAX;
// Dynamic shared memory a GDN launch may take per CTA, and the shared memory of an SM.
constexpr int XV_GDN_SMEM_MAX = 227 * 1024;
constexpr int XV_GDN_SMEM_SM = 228 * 1024;
struct GdnStepsDev {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const uint16_t* beta;
    const uint16_t* gate;
    long long qkv_stride;
    long long gate_stride;
    int rows_per_seq;
    // 0: beta and gate hold bf16 beta = sigmoid(b) and gate = exp(-softplus(a));
    // 1: they point at the raw b and a projection columns and the kernel applies those maps
    int raw_gates;
};
// Replays n_commit[b] (or n_fixed when n_commit is null) pending steps into
// the state, writing o for them when emit_replay; then k speculative steps of
// `draft` writing o rows b*k + t.
xv_status gdn_launch(float* state, const GdnStepsDev& pending, const int32_t* n_commit, int n_fixed, int max_commit,
                     bool emit_replay, const GdnStepsDev& draft, int k, uint16_t* o, long long o_stride, int B, int H,
                     int Hk,
                     int dk, int dv, int qk_l2norm, cudaStream_t s);

// ---- complete GDN layer parts (gdn_layer.cu)
// Shifts the n_commit[b] pending rows into the state [B, Kc-1, C], then convolves the k rows of x
// (row b*x_rows + t) into y (row b*k + t): y = bf16(silu(taps . window)).
xv_status conv_launch(uint16_t* state, const uint16_t* pend, long long pend_stride, int pend_rows,
                      const int32_t* n_commit, int max_commit, const uint16_t* x, long long x_stride, int x_rows, int k,
                      const uint16_t* w, int C, int Kc, int B, uint16_t* y, long long y_stride, cudaStream_t s);
// y = bf16(o / sqrt(mean(o^2) + eps) * (1 + w) * silu(z)) per (row, head) of dv values; y may be o.
xv_status gated_norm_launch(const uint16_t* o, long long o_stride, const uint16_t* z, long long z_stride,
                            const uint16_t* w, int M, int H, int dv, float eps, uint16_t* y, long long y_stride,
                            cudaStream_t s);

// ---- attention (attn.cu)
// Splits at fixed absolute boundaries: ATTN_SPLIT positions each below ATTN_SPLIT_SWITCH,
// ATTN_SPLIT_LONG beyond.  Measured on GB300 (verify step, context 131072): splits of 2048 past
// 4096 instead of 512 throughout cut the persistent CTAs' item boundaries (about 3 us each) from
// ~7 to ~2 per CTA at batch 1 and from ~54 to ~15 at batch 8: 900 -> 872 us and 1738 -> 1636 us
// per step; 1024 past 4096 or 2048: -9 / -95 us; 4096 past 16384: +370 us at batch 8 (too few,
// too coarse items to balance); shorter contexts are unchanged.
constexpr int ATTN_SPLIT = 512, ATTN_SPLIT_SWITCH = 4096, ATTN_SPLIT_LONG = 2048;
// First position of split s; split s covers [attn_split_begin(s), attn_split_begin(s + 1)).
__host__ __device__ inline int attn_split_begin(int s) {
    constexpr int NS = ATTN_SPLIT_SWITCH / ATTN_SPLIT;
    return s < NS ? s * ATTN_SPLIT : ATTN_SPLIT_SWITCH + (s - NS) * ATTN_SPLIT_LONG;
}
// Splits a row of `len` visible positions spans.
__host__ __device__ inline int attn_split_count(int len) {
    constexpr int NS = ATTN_SPLIT_SWITCH / ATTN_SPLIT;
    return len <= ATTN_SPLIT_SWITCH ? (len + ATTN_SPLIT - 1) / ATTN_SPLIT
                                    : NS + (len - ATTN_SPLIT_SWITCH + ATTN_SPLIT_LONG - 1) / ATTN_SPLIT_LONG;
}
constexpr int ATTN_TILE = 64;     // positions per tile inside a split
size_t attn_workspace_size(int B, int R, int Hq, int hd, int max_len);
// Where position p of sequence b lives in a K or V cache of Hkv heads: page
// table[b * max_pages + p / page], row p % page, in a pool [n_pages, Hkv, page, hd].
// A contiguous cache [B, Hkv, Lmax, hd] is one page of Lmax positions per sequence
// (table == nullptr, page = Lmax, max_pages = 1, n_pages = B).  Positions run to
// page * max_pages.
struct KvPages {
    const int32_t* table;
    int page, max_pages, n_pages;
};
inline KvPages kv_contiguous(int B, int Lmax) { return KvPages{nullptr, Lmax, 1, B}; }
// Row r of sequence b sees ctx_len[b] + len_bias + r positions; max_len bounds every such length.
xv_status attn_launch(const uint16_t* q, long long q_stride, const uint16_t* kc, const uint16_t* vc, const KvPages& kv,
                      const int32_t* ctx_len, int len_bias, int R, int B, int Hq, int Hkv, int hd, int max_len,
                      float scale, const uint16_t* gate, long long gate_stride, uint16_t* out, long long out_stride,
                      void* ws, size_t ws_bytes, cudaStream_t s);
// Row (b, r) of src goes to position ctx_len[b] + pos_bias + r.
xv_status kv_append_launch(const uint16_t* src, long long src_stride, const int32_t* ctx_len, int pos_bias, int R,
                           int B, int Hkv, int hd, const KvPages& kv, uint16_t* kc, uint16_t* vc, cudaStream_t s);

// ---- glue (glue.cu)
xv_status rmsnorm_launch(const uint16_t* x, const uint16_t* w, int M, int H, float eps, uint16_t* y, cudaStream_t s);
// x[m] <- E[tokens[m]]; xn[m] = rmsnorm(x[m], w) (one kernel)
xv_status embed_rmsnorm_launch(const int32_t* tokens, int M, const uint16_t* E, int V, int H, const uint16_t* w,
                               float eps, uint16_t* x, uint16_t* xn, cudaStream_t s);
// x <- bf16(x + y); xn <- rmsnorm(x, w)
// the same with y = bf16(sum of a GEMM's S split-K partials [S][M][H] in segment order)
xv_status residual_rmsnorm_part_launch(uint16_t* x, const float* part, int S, const uint16_t* w, int M, int H, float eps,
                                       uint16_t* xn, cudaStream_t s);
xv_status residual_rmsnorm_launch(uint16_t* x, const uint16_t* y, const uint16_t* w, int M, int H, float eps,
                                  uint16_t* xn, cudaStream_t s);
// act[m][i] = bf16(silu(gu[m][i]) * gu[m][F + i])
xv_status swiglu_launch(const uint16_t* gu, int M, int F, uint16_t* act, cudaStream_t s);
size_t argmax_workspace_size(int M, int V);
// idx[b*k + j] = argmax of logits row b*k + j (lowest index among equal maxima);
// n_accept[b] = leading drafts tokens[b][j+1] (j + 1 < k_b) equal to idx[b*k + j], where
// k_b = k_seq[b] (k when k_seq is null) (two kernels)
// With ctx_len != null the acceptance kernel also commits n_accept[b] + 1 positions of every
// sequence (ctx_len[b] += n, n_commit[b] = n), as the commit kernel would.
xv_status argmax_accept_launch(const float* logits, int B, int k, int V, int32_t* idx, void* ws,
                               const int32_t* tokens, const int32_t* k_seq, int32_t* n_accept, cudaStream_t s,
                               int32_t* ctx_len = nullptr, int32_t* n_commit = nullptr);
// The same from per-chunk (max, index) partials part[row * nchunk + c] already formed (the LM
// head GEMM's amax output): the second kernel only.
xv_status accept_from_parts_launch(const float2* part, int nchunk, int B, int k, int32_t* idx, const int32_t* tokens,
                                   const int32_t* k_seq, int32_t* n_accept, cudaStream_t s, int32_t* ctx_len = nullptr,
                                   int32_t* n_commit = nullptr);
// ctx_len[b] += keep[b] + keep_bias; n_commit[b] = keep[b] + keep_bias (checked to lie in [1, k_b],
// k_b = k_seq[b] or k)
xv_status commit_launch(const int32_t* keep, int keep_bias, int B, int k, const int32_t* k_seq, int32_t* ctx_len,
                        int32_t* n_commit, cudaStream_t s);
xv_status zero_i32_launch(int32_t* p, int n, cudaStream_t s);

}  // namespace xv
