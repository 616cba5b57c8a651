/*
 * xv — exact speculative verify for hybrid gated-delta-net / attention decoders
 * on one GB300 (sm_103a).  C ABI of libxv.so.
 *
 * The operations follow a recipe described on these pages:
 *   [post]  "Follow-up to my earlier post on Qwen3.8-27B decode speed"
 *           (r/LocalLLaMA post, feedman.me copy)
 *   [card]  "Qwen3.8-27B Bit-Exact Spec-Decode 1x RTX PRO 6000 SGLang"
 *           (localairecipes recipe card), summary and install notes
 *   [digest] "Bit-exact speculative decoding hits 106 t/s on Qwen3.8-27B with
 *           one RTX PRO 6000" (agihunt digest), Key findings
 * Their claim, which this library is built to: checking k draft tokens in one
 * verify pass gives exactly the bits (token ids and logprobs) of decoding the
 * same tokens one at a time.  Three parts make that so ([post]): the small-M
 * projection GEMMs reduce in an order that does not depend on the row count;
 * verify steps the GDN recurrence with the decode step's own code, tiling and
 * rounding (beta and gate in the decode dtype, bf16); verify attention runs
 * each draft position as its own decode row.
 *
 * Conventions (all entry points):
 *   - bf16 tensors are passed as uint16_t* bit patterns; fp32 as float*.
 *   - Every pointer argument is DEVICE memory owned by the caller unless it is
 *     documented as host memory.  The library allocates nothing, frees
 *     nothing and never synchronises the stream; work is enqueued on the
 *     caller's stream `s` (0 = legacy default stream).
 *   - Scratch space comes from a caller workspace `ws` of `ws_bytes` bytes,
 *     sized by the matching *_workspace_size() query.  A workspace must be
 *     zero-filled once before its first use (e.g. cudaMemsetAsync); every call
 *     leaves its internal counters at zero again.  Calls that run at the same
 *     time must use distinct workspaces.
 *   - Arguments are validated on the host before anything is enqueued; on an
 *     error nothing is launched and the return code says why.  Kernel waits
 *     are bounded; a wait that runs out records a device-side error that
 *     xv_device_check() reports.
 *   - Layout of the row dimension: a batch of B sequences with R rows each is
 *     stored row (b, r) at index b*R + r.
 */
#ifndef XV_H_
#define XV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* xv_stream;   /* same type as cudaStream_t */
typedef int xv_status;

#define XV_OK               0
#define XV_ERR_ARG         -1   /* null pointer, bad shape or inconsistent sizes */
#define XV_ERR_UNSUPPORTED -2   /* size or alignment outside what the kernels handle */
#define XV_ERR_WORKSPACE   -3   /* workspace missing or too small */
#define XV_ERR_CUDA        -4   /* a CUDA runtime call or launch failed */
#define XV_ERR_DEVICE_CHECK -5  /* a kernel recorded a device-side error (see xv_device_check) */

#define XV_ABI_VERSION 5
#define XV_GEMM_M_MAX 64        /* rows per small-M GEMM call */
#define XV_KMAX 64              /* tokens per sequence per verify (or prefill chunk) call */
#define XV_CONV_MAX 8           /* widest causal convolution of a complete GDN layer */

/* Version of this header's ABI (XV_ABI_VERSION). */
int xv_abi_version(void);

/* Message for the last error returned on the calling host thread ("" if none).
 * The string is owned by the library and valid until the next call on the thread. */
const char* xv_last_error(void);

/* Synchronises `s`, then reads and clears the device-side error word of the
 * current device.  Returns XV_OK, or XV_ERR_DEVICE_CHECK with *code set to the
 * recorded bits (code may be NULL): 1 a bounded wait gave up, 2 a token id
 * outside [0, vocab), 4 a context length outside what the launch was sized
 * for, 8 a commit count or per-sequence k outside its range, 16 a KV page
 * table entry outside the pool.  The only call in the library that
 * synchronises. */
xv_status xv_device_check(xv_stream s, unsigned* code);

/* Number of kernels this library has launched in this process (host counter). */
unsigned long long xv_launch_count(void);

/* Programmatic dependent launch between consecutive kernels of this library
 * (default on): a kernel may start its independent prologue (barrier set-up,
 * TMEM allocation, prefetch of weights) while its predecessor in the stream
 * finishes, and waits for the predecessor before touching activations.
 * Weights are requested before that wait, so they must be complete when the
 * GEMM is enqueued: written by a kernel that has finished, a copy, or
 * xv_gemm_tile_weights / xv_gemm_tile_gate_up (which end with a kernel that
 * lets its successor start only after the tiling is complete in memory).
 * Results are identical either way; 0 turns it off (for timing comparisons). */
xv_status xv_set_overlap(int enable);

/* Launch trace, a profiling hook outside the verify method.  While enabled,
 * every kernel the library launches is bracketed by two CUDA events recorded
 * on its stream, and the launch's kind and algorithmic bytes (inputs read
 * plus outputs written, as the op defines them; 0 where the host cannot know
 * them) are noted.  xv_trace_enable creates 2*capacity events on the current
 * device the first time (or when capacity grows) and restarts the record;
 * launches beyond capacity are not traced.  xv_trace_read synchronises the
 * recorded events and fills, for the first n launches, the elapsed
 * milliseconds, the kind (see xv_trace_kind_name) and the bytes (all host
 * arrays, any may be NULL).  Not thread-safe; for benchmarks. */
xv_status xv_trace_enable(int capacity);
xv_status xv_trace_disable(void);
int xv_trace_count(void);
xv_status xv_trace_read(float* ms, int* kind, long long* bytes, int n);
const char* xv_trace_kind_name(int kind);

/* ------------------------------------------------------------------ GEMM
 * Small-M bf16 GEMM  Y[M,N] = X[M,K] . W[N,K]^T  with fp32 accumulation.
 * [post] and [card] summary: at small batch the projection GEMMs of decode
 * and verify go to a tile that yields the same bits whatever the row count,
 * and it must stream the weights near DRAM speed ([post]: the previous kernel
 * read them at about a third of it).
 *
 * Contract: row i of Y is bit-identical for every M in 1..XV_GEMM_M_MAX and
 * for every position of that row inside X, and identical from run to run.
 * The reduction order over K is a function of (N, K) only.
 *
 *   X   [M, ldx] bf16, row-major, 16-byte aligned, ldx % 8 == 0, ldx >= K
 *   W   [N, K]  bf16, row-major (the weight layout), 16-byte aligned, K % 8 == 0
 *   Y   [M, ldy] bf16 (xv_gemm_small_m) or fp32 (xv_gemm_small_m_f32out), ldy >= N
 *   1 <= M <= XV_GEMM_M_MAX, N >= 1, K >= 8
 * Errors: XV_ERR_ARG (null pointer, M/N/K/ld out of range), XV_ERR_UNSUPPORTED
 * (alignment, M > XV_GEMM_M_MAX), XV_ERR_WORKSPACE (ws_bytes below
 * xv_gemm_workspace_size(M, N, K)), XV_ERR_CUDA. */
size_t xv_gemm_workspace_size(int M, int N, int K);
xv_status xv_gemm_small_m(const uint16_t* X, int ldx, const uint16_t* W, uint16_t* Y, int ldy,
                          int M, int N, int K, void* ws, size_t ws_bytes, xv_stream s);
xv_status xv_gemm_small_m_f32out(const uint16_t* X, int ldx, const uint16_t* W, float* Y, int ldy,
                                 int M, int N, int K, void* ws, size_t ws_bytes, xv_stream s);
/* Number of K-segments the GEMM uses for (N, K) (a pure function of N and K). */
int xv_gemm_splits(int N, int K);

/* Tiled weight layout (a layout of this library; the pages have none).  The
 * GEMM streams each 128-row x 64-column weight tile (one ring stage) as one
 * copy; row-major, such a tile is 128 pieces of 128 bytes, K * 2 bytes apart.
 * The tiled layout stores it as one contiguous 16 KiB block, and the K-blocks
 * of a tile row one after another:
 *     Wt[t][kb][r][c] = W[128 t + r][64 kb + c],
 * t < ceil(N/128), kb < ceil(K/64), zero past N or K.  The GEMM places the
 * same values in the same shared-memory slots from either layout, so Y is
 * bit-identical to the row-major call's.  Measured on GB300 the tiled weights
 * stream faster (the 151936 x 5120 LM head at M = 8: 254 -> 242 us alone).
 *
 * xv_gemm_tiled_bytes: bytes of the tiled copy of an N x K weight (0 for
 *   N < 1 or K < 1).
 * xv_gemm_tile_weights: writes Wt (device, xv_gemm_tiled_bytes(N, K) bytes,
 *   caller-owned) from W [N, K] row-major on stream s (the tiling kernel,
 *   then an empty kernel that lets the next one start only once the tiles
 *   are complete, so a GEMM may follow on the same stream at once).  W and
 *   Wt 16-byte aligned and not overlapping, K % 8 == 0.  Errors: XV_ERR_ARG
 *   (null pointer, N < 1, K < 8), XV_ERR_UNSUPPORTED (K % 8 != 0,
 *   alignment), XV_ERR_CUDA.
 * xv_gemm_small_m_tiled(_f32out): xv_gemm_small_m(_f32out) reading the
 *   weights from a tiled copy Wt (16-byte aligned); arguments, errors and
 *   the bits of Y as there. */
size_t xv_gemm_tiled_bytes(int N, int K);
xv_status xv_gemm_tile_weights(const uint16_t* W, int N, int K, uint16_t* Wt, xv_stream s);

/* Gate/up projection with the SwiGLU fused.  xv_gemm_tile_gate_up tiles a
 * gate/up weight W [2F, K] (F gate rows, then F up rows) so that tile t holds
 * gate rows 64t..64t+63 followed by up rows F+64t..F+64t+63 (Wt of
 * xv_gemm_tiled_bytes(2F, K) bytes; F % 64 == 0, K % 8 == 0, 16-byte
 * aligned; enqueued as xv_gemm_tile_weights is, fence kernel included).
 * xv_gemm_swiglu_tiled then computes, for each row m of X and
 * feature f < F,
 *     act[m, f] = bf16(silu(g) u),  g = bf16((X W^T)[m, f]),
 *                                   u = bf16((X W^T)[m, F + f]),
 * silu(g) u = (g / (1 + exp(-g))) u in fp32: the bits of xv_gemm_small_m into
 * a [M, 2F] buffer followed by the SwiGLU of the verify block, in one kernel
 * and without the [M, 2F] buffer.  The GEMM is never split over K (no
 * workspace).  act [M, ldact] bf16, ldact >= F.  Errors: XV_ERR_ARG (null
 * pointer, sizes out of range, ldact < F), XV_ERR_UNSUPPORTED (F % 64,
 * K % 8, alignment, M > XV_GEMM_M_MAX), XV_ERR_CUDA. */
xv_status xv_gemm_tile_gate_up(const uint16_t* W, int F, int K, uint16_t* Wt, xv_stream s);
xv_status xv_gemm_swiglu_tiled(const uint16_t* X, int ldx, const uint16_t* Wt, uint16_t* act, int ldact,
                               int M, int F, int K, xv_stream s);
xv_status xv_gemm_small_m_tiled(const uint16_t* X, int ldx, const uint16_t* Wt, uint16_t* Y, int ldy,
                                int M, int N, int K, void* ws, size_t ws_bytes, xv_stream s);
xv_status xv_gemm_small_m_tiled_f32out(const uint16_t* X, int ldx, const uint16_t* Wt, float* Y, int ldy,
                                       int M, int N, int K, void* ws, size_t ws_bytes, xv_stream s);

/* The same GEMM (bf16 out) for callers that cannot allocate device memory or
 * pass a workspace: code running under another framework's memory pool,
 * plugins inside a host process that owns every device allocation, loops
 * where an allocation is not allowed.  The method itself needs no such entry point; this is
 * a convenience of this library.  Its scratch (split-K partial sums and tile
 * counters) is a fixed array of XV_GEMM_NOALLOC_SCRATCH_BYTES that every GPU
 * loading the library holds until the process exits.  The first call on a
 * device looks up that array's device address, so make the first call on each
 * device before any stream capture.  A call whose shape combines its split-K
 * partials through the tile counters (M <= 8 and more than 4 K-segments) first
 * clears them on the stream (a 1 KiB memset), so a call that follows one whose
 * bounded wait gave up still starts from zero.  Shapes whose
 * scratch need (xv_gemm_workspace_size) exceeds the array are rejected with
 * XV_ERR_UNSUPPORTED; with this size every shape with M <= XV_GEMM_M_MAX fits.
 * All calls share the array: calls that overlap on the GPU race, so callers
 * serialise them (one stream, or events).  Allocates nothing.  Arguments and
 * bits of Y are as for xv_gemm_small_m. */
#define XV_GEMM_NOALLOC_SCRATCH_BYTES (10u * 1024u * 1024u)
xv_status xv_gemm_small_m_noalloc(const uint16_t* X, int ldx, const uint16_t* W, uint16_t* Y, int ldy,
                                  int M, int N, int K, xv_stream s);

/* ------------------------------------------------------------------- GDN
 * Gated delta rule, per sequence b and head h, state S [dv][dk] in fp32:
 *     S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T ,   o_t = S_t q_t
 * [post]: verify runs the recurrence through the decode kernel (the faulty
 * verify tiled the state differently and kept beta in fp32).  Here decode and
 * verify are the same kernel and the same step function; a step computes, in
 * fp32 with every operation rounded once:  S <- a S;  r = S k;
 * u = beta (v - r);  S <- S + u k^T;  o = S q  (o rounded to bf16).
 *
 * Step inputs for a set of steps, row (b, t) at index b*rows_per_seq + t:
 *   q, k  [rows, H, dk] bf16 and v [rows, H, dv] bf16, consecutive rows
 *         qkv_stride elements apart (heads contiguous inside a row); q, k
 *         and v 16-byte aligned and qkv_stride a multiple of 8;
 *   beta, gate [rows, H] bf16 (beta = sigmoid(.), gate = exp(-softplus(.))
 *         already rounded to bf16), rows gate_stride elements apart.
 * With qk_l2norm != 0 the kernel normalises q and k per head in fp32
 * (x / sqrt(sum x^2 + 1e-6)); with 0 they are used as given. */
typedef struct {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const uint16_t* beta;
    const uint16_t* gate;
    long long qkv_stride;
    long long gate_stride;
    int rows_per_seq;
} xv_gdn_steps;

/* One decode step for B sequences: state [B, H, dv, dk] fp32 is updated in
 * place, o [B, H, dv] bf16 (row b at b*o_stride) receives o_t.
 * dk in {64, 128}; dv a multiple of 32; 1 <= B, 1 <= H.
 * Errors (for this and the two verify calls below): XV_ERR_ARG (null state,
 * o or step pointers, B or H < 1, rows_per_seq < 1 or fewer rows than the
 * steps used, gate_stride < H, o_stride < H*dv, n_commit missing with
 * max_commit > 0, H not a multiple of Hk); XV_ERR_UNSUPPORTED (dk, dv, B or H
 * above 65535, q/k/v not 16-byte aligned or qkv_stride not a multiple of 8,
 * k or max_commit outside [0, XV_KMAX]); XV_ERR_CUDA (launch).  A count
 * n_commit[b] outside [0, max_commit] is clamped on the device and reported
 * by xv_device_check. */
xv_status xv_gdn_decode_step(float* state, const xv_gdn_steps* step, uint16_t* o, long long o_stride,
                             int B, int H, int dk, int dv, int qk_l2norm, xv_stream s);

/* Verify with deferred commit.  For each sequence b:
 *   1. replay n_commit[b] steps of `pending` (rows b*pending.rows_per_seq + 0..)
 *      into `state` and write the state back (nothing written if 0);
 *   2. run k speculative steps of `draft` from that state, writing only
 *      o [B, k, H, dv] bf16 (row (b,t) at (b*k + t)*o_stride).
 * k = 0 is a pure commit.  After the call the caller keeps `draft` alive: it
 * becomes the next call's `pending`, with n_commit = the number of positions
 * kept.  Bit-exactness: o of step t equals the o of decode step t from the
 * same committed state, and the state after replaying j steps equals j
 * decode steps.  n_commit is device memory [B] with 0 <= n_commit[b] <= max_commit;
 * 0 <= k <= XV_KMAX, max_commit <= XV_KMAX. */
xv_status xv_gdn_verify(float* state, const xv_gdn_steps* pending, const int32_t* n_commit, int max_commit,
                        const xv_gdn_steps* draft, int k, uint16_t* o, long long o_stride,
                        int B, int H, int dk, int dv, int qk_l2norm, xv_stream s);

/* xv_gdn_verify with grouped heads: H v heads (state, v, beta, gate, o per v
 * head) over Hk q/k heads, H a multiple of Hk; v head h reads q and k of head
 * h / (H / Hk) (q and k rows hold Hk*dk values). */
xv_status xv_gdn_verify_grouped(float* state, const xv_gdn_steps* pending, const int32_t* n_commit, int max_commit,
                                const xv_gdn_steps* draft, int k, uint16_t* o, long long o_stride,
                                int B, int H, int Hk, int dk, int dv, int qk_l2norm, xv_stream s);

/* ------------------------------------------ complete GDN layer parts
 * Not on the pages (which measure GDN layers without them); the complete
 * layer of gated-delta-net decoders adds a depthwise causal convolution over
 * the q|k|v projection channels and a per-head output RMSNorm gated by
 * silu(z).  Both are computed per output from its own inputs in a fixed
 * order, so verify rows get the bits of decode steps.
 *
 * Convolution of width Kc (2..XV_CONV_MAX) over C channels for B sequences.
 * state [B, Kc-1, C] bf16 holds each sequence's Kc-1 previous inputs, oldest
 * first.  The call first shifts the n_commit[b] (device, 0..max_commit)
 * pending rows pend[b*pend_rows + t] into the state and writes it back, then
 * convolves the k rows x[b*x_rows + t]:
 *     y[b*k + t][c] = bf16( silu( sum_j w[c][j] * window[j] ) ),
 * the window being the Kc-1 prior inputs then x (tap Kc-1 meets the newest).
 * The k rows do not enter the state: the caller passes them as the next
 * call's pending rows (deferred commit, as for the recurrence).  Strides are
 * in elements; w is [C, Kc] bf16.  k = 0 with max_commit > 0 is a pure commit.
 * Errors: XV_ERR_ARG (null state or taps, B outside [1, 65535], C < 1, pending
 * rows or x rows fewer than max_commit or k, strides below C),
 * XV_ERR_UNSUPPORTED (Kc outside [2, XV_CONV_MAX], k or max_commit outside
 * [0, XV_KMAX]), XV_ERR_CUDA (launch).  A count n_commit[b] out of range is
 * clamped on the device and reported by xv_device_check. */
xv_status xv_gdn_conv(uint16_t* state, const uint16_t* pend, long long pend_stride, int pend_rows,
                      const int32_t* n_commit, int max_commit, const uint16_t* x, long long x_stride, int x_rows,
                      int k, const uint16_t* w, int C, int Kc, int B, uint16_t* y, long long y_stride, xv_stream s);

/* Gated output norm over M rows of H heads of dv values (dv a multiple of 32
 * up to 256): y = bf16( o / sqrt(mean(o^2) + eps) * (1 + w) * silu(z) ), w
 * [dv]; y may be o.  Rows are o_stride / z_stride / y_stride elements apart.
 * Errors: XV_ERR_ARG (null pointer, M or H < 1, a stride below H*dv),
 * XV_ERR_UNSUPPORTED (dv, or M*H above 2^30), XV_ERR_CUDA (launch). */
xv_status xv_gated_norm(const uint16_t* o, long long o_stride, const uint16_t* z, long long z_stride,
                        const uint16_t* w, int M, int H, int dv, float eps, uint16_t* y, long long y_stride,
                        xv_stream s);

/* ------------------------------------------------------------- attention
 * Decode-row attention over a bf16 KV cache.  [post]: verify attention runs
 * as decode rows, one per draft position.  Row r of sequence b is the query
 * at position ctx_len[b] - 1 + r and attends to positions [0, ctx_len[b] + r):
 *   out = softmax(q . K^T * scale) V      per query head h, kv head h / (Hq/Hkv).
 * The positions are cut into splits at fixed absolute boundaries (split s
 * covers [xv_attn_split_begin(s), xv_attn_split_begin(s + 1)): 512 positions
 * each below 4096, 2048 beyond), each split is reduced with an fp32 online
 * softmax over fixed 64-position tiles, and the splits are combined in split
 * order; a row therefore gets the same bits as an R = 1 call with
 * ctx_len[b] + r.
 *
 *   q     [B*R rows, Hq*hd] bf16, row stride q_stride elements (16-byte aligned rows)
 *   kc,vc [B, Hkv, Lmax, hd] bf16 (16-byte aligned)
 *   ctx_len [B] int32 device: visible length of row 0 (includes its own token),
 *         1 <= ctx_len[b] and ctx_len[b] + R - 1 <= max_ctx <= Lmax
 *   max_ctx host int: upper bound used to size the grid (a larger value only
 *         launches blocks that exit at once)
 *   out   [B*R rows, Hq*hd] bf16, row stride out_stride
 *   gate  optional [B*R rows, Hq*hd] bf16 with row stride gate_stride, or NULL:
 *         when given, out = bf16( bf16(attn) * sigmoid(gate) ) (the gated
 *         attention layer's output gate), else out = bf16(attn)
 *   hd = 256 or 64 (hd % 64 == 0), Hq % Hkv == 0, 1 <= R <= XV_KMAX (the R*(Hq/Hkv) rows of a
 *         kv head go in tiles of 64 rows, one CTA each per split)
 * Workspace: xv_attn_workspace_size(B, R, Hq, hd, max_ctx) bytes, 16-byte aligned (0 is returned
 * for sizes below 1).
 * Errors: XV_ERR_ARG (null pointer, sizes < 1, Hq not a multiple of Hkv,
 * max_ctx outside [R, Lmax], row strides below Hq*hd), XV_ERR_UNSUPPORTED (hd,
 * R > XV_KMAX, B or Hkv above 65535, B*Hkv*Lmax above 2^31, unaligned q rows,
 * caches or workspace), XV_ERR_WORKSPACE (missing or small workspace),
 * XV_ERR_CUDA (launch).  A sequence whose ctx_len[b] + R - 1 falls outside
 * [1, max_ctx] is skipped on the device and reported by xv_device_check. */
int xv_attn_split_begin(int s);   /* -1 for s < 0 */
size_t xv_attn_workspace_size(int B, int R, int Hq, int hd, int max_ctx);
xv_status xv_attn_decode_rows(const uint16_t* q, long long q_stride, const uint16_t* kc, const uint16_t* vc,
                              const int32_t* ctx_len, int R, int B, int Hq, int Hkv, int hd, int Lmax,
                              int max_ctx, float scale, const uint16_t* gate, long long gate_stride,
                              uint16_t* out, long long out_stride, void* ws, size_t ws_bytes, xv_stream s);

/* Writes the K and V rows of a verify block into the caches: row (b, r) of
 * kv_src (k at column offset 0, v at column offset Hkv*hd, row stride
 * src_stride) goes to position ctx_len[b] - 1 + r of sequence b.
 * Errors: XV_ERR_ARG (null pointer, sizes < 1, hd not a multiple of 8,
 * src_stride < 2*Hkv*hd), XV_ERR_UNSUPPORTED (kv_src, kc, vc not 16-byte
 * aligned or src_stride not a multiple of 8), XV_ERR_CUDA (launch).  A
 * position outside [0, Lmax) is skipped on the device and reported by
 * xv_device_check. */
xv_status xv_kv_append(const uint16_t* kv_src, long long src_stride, const int32_t* ctx_len, int R, int B,
                       int Hkv, int hd, int Lmax, uint16_t* kc, uint16_t* vc, xv_stream s);

/* Paged KV cache.  The K and V pools are [n_pages, Hkv, page_size, hd] bf16
 * (16-byte aligned); position p of sequence b is row p % page_size of page
 * page_table[b * max_pages + p / page_size], so a sequence holds up to
 * page_size * max_pages positions and pages are handed out by the caller
 * (pages of one pool may be shared out among the sequences in any order).
 * page_size is a positive multiple of 64: a page holds whole 64-position
 * tiles, so the split/tile schedule, and with it every bit of the result, is
 * the one of a contiguous cache holding the same values.  Every table entry
 * that a call reads (positions below ctx_len[b] + R - 1) must name a page in
 * [0, n_pages); an entry outside it is recorded as device error bit 16 and
 * replaced by page 0 (attention) or skipped (append). */
typedef struct {
    const int32_t* page_table;   /* [B, max_pages] int32 device */
    int page_size;               /* positions per page, a multiple of 64 */
    int max_pages;               /* table entries per sequence */
    int n_pages;                 /* pages in each pool */
} xv_kv_pages;

/* xv_attn_decode_rows over paged pools; R <= max_ctx <= page_size * max_pages. */
xv_status xv_attn_decode_rows_paged(const uint16_t* q, long long q_stride, const uint16_t* kpool, const uint16_t* vpool,
                                    const xv_kv_pages* pages, const int32_t* ctx_len, int R, int B, int Hq, int Hkv,
                                    int hd, int max_ctx, float scale, const uint16_t* gate, long long gate_stride,
                                    uint16_t* out, long long out_stride, void* ws, size_t ws_bytes, xv_stream s);

/* xv_kv_append into paged pools. */
xv_status xv_kv_append_paged(const uint16_t* kv_src, long long src_stride, const int32_t* ctx_len, int R, int B,
                             int Hkv, int hd, const xv_kv_pages* pages, uint16_t* kpool, uint16_t* vpool, xv_stream s);

/* ------------------------------------------------------------ the block
 * A stack of decoder layers (each: x + mixer(rmsnorm(x)), then
 * h + SwiGLU-MLP(rmsnorm(h))), mixers being GDN or gated attention layers,
 * under an embedding and an LM head with a final RMSNorm.  Verify takes k
 * token ids per sequence (the last committed token, then k-1 drafts) and
 * returns the fp32 logits of the k positions, their argmax (lowest index on
 * ties) and the greedy acceptance count ([post]: temperature 0, every draft
 * compared with the target's argmax).  Decode is k = 1 through the same path.
 *
 * Column layouts of the input projections (rows of w_in):
 *   GDN:       [ q (Hk*dk) | k (Hk*dk) | v (H*dv) | z (H*dv, with the gated
 *                output norm only) | b (H) | a (H) ]   (H = gdn_heads v heads,
 *                Hk = gdn_qk_heads q/k heads, Hk = H unless set)
 *   attention: [ q (Hq*hd) | gate (Hq*hd) | k (Hkv*hd) | v (Hkv*hd) ]
 * A complete GDN layer (gdn_conv > 0 and/or gdn_out_norm) runs the q|k|v
 * columns through the causal convolution (xv_gdn_conv) before the
 * recurrence and its output through the gated norm (xv_gated_norm).
 * RMSNorm: y = bf16( x / sqrt(mean(x^2) + eps) * (1 + w) ). */
typedef struct {
    int hidden;               /* H */
    int vocab;                /* V */
    int mlp;                  /* F */
    int n_layers;
    const int32_t* layer_kind;/* HOST array [n_layers]: 0 = GDN, 1 = attention */
    int gdn_heads, gdn_dk, gdn_dv;
    int attn_hq, attn_hkv, attn_hd;
    float rms_eps;
    int gdn_qk_heads;         /* q/k heads of a GDN layer (0: gdn_heads); divides gdn_heads */
    int gdn_conv;             /* causal convolution width over q|k|v (0: none, else 2..XV_CONV_MAX) */
    int gdn_out_norm;         /* 1: z columns after v and the gated output norm */
} xv_block_config;

typedef struct {
    const uint16_t* norm1;    /* [H] */
    const uint16_t* w_in;     /* [in_dim, H] */
    const uint16_t* w_out;    /* [H, inner] (inner = gdn_heads*gdn_dv or attn_hq*attn_hd) */
    const uint16_t* norm2;    /* [H] */
    const uint16_t* w_gate_up;/* [2F, H]: F gate rows, then F up rows */
    const uint16_t* w_down;   /* [H, F] */
    const uint16_t* conv_w;   /* GDN layer with a convolution: [C, Kc], C = xv_gdn_conv_dim(cfg) */
    const uint16_t* out_norm; /* GDN layer with the gated output norm: [dv] */
} xv_layer_weights;

typedef struct {
    const uint16_t* embed;            /* [V, H] */
    const xv_layer_weights* layers;   /* HOST array [n_layers] of device pointers */
    const uint16_t* final_norm;       /* [H] */
    const uint16_t* lm_head;          /* [V, H] */
    int tiled;                        /* 1: w_in, w_out, w_down and lm_head are tiled copies
                                         (xv_gemm_tile_weights), w_gate_up a gated tiled copy
                                         (xv_gemm_tile_gate_up; the SwiGLU is then fused into its
                                         GEMM; mlp % 64 == 0); embed stays [V, H].  0: every weight
                                         row-major.  The bits do not depend on it. */
} xv_block_weights;

typedef struct {
    float* gdn_state;         /* GDN layer: [B, heads, dv, dk] fp32 */
    uint16_t* gdn_hist[2];    /* GDN layer: two [B*kmax, xv_gdn_hist_stride(cfg)] bf16 projection buffers */
    uint16_t* gdn_conv_state; /* GDN layer with a convolution: [B, Kc-1, C] bf16, prior inputs, oldest first */
    uint16_t* gdn_conv_out[2];/* GDN layer with a convolution: two [B*kmax, xv_gdn_conv_stride(cfg)] bf16
                                 buffers of convolution outputs (this call's and the pending ones) */
    uint16_t* k_cache;        /* attention layer: [B, Hkv, Lmax, hd] bf16, or a pool
                                 [kv_pages.n_pages, Hkv, page_size, hd] when the state is paged */
    uint16_t* v_cache;
} xv_layer_state;

typedef struct {
    int B, kmax, Lmax;
    int32_t* ctx_len;         /* [B] device: tokens committed to the KV cache */
    int32_t* n_commit;        /* [B] device: pending GDN steps (set by commit) */
    int parity;               /* host: which history buffer the next verify writes */
    int pending_rows;         /* host: rows per sequence of the pending history (k of the last verify) */
    int max_ctx;              /* host: upper bound of every ctx_len[b] (grid sizing and the Lmax
                                 check); a commit raises it by the verify's k, as the accepted
                                 counts stay on the device; a caller that has read the lengths
                                 back may lower it to their maximum (never below it) */
    int last_k;               /* host: k of the last verify not yet committed (0 = none) */
    xv_layer_state* layers;   /* HOST array [n_layers] */
    xv_kv_pages kv_pages;     /* page_table NULL: contiguous caches; else every attention layer's
                                 caches are pools addressed by this one table, and
                                 Lmax <= page_size * max_pages */
    const int32_t* last_k_seq;/* host: the k_seq of the last verify not yet committed (NULL = k) */
} xv_block_state;

int xv_gdn_in_dim(const xv_block_config* cfg);
/* Row stride (elements) of the GDN step-history buffers: xv_gdn_in_dim rounded up to 8. */
int xv_gdn_hist_stride(const xv_block_config* cfg);
int xv_attn_in_dim(const xv_block_config* cfg);
/* Channels of a GDN layer's convolution (q|k|v: 2*Hk*dk + H*dv) and the row stride of its output
 * buffers (rounded up to 8). */
int xv_gdn_conv_dim(const xv_block_config* cfg);
int xv_gdn_conv_stride(const xv_block_config* cfg);

/* Workspace for xv_verify_block with B sequences of up to kmax tokens (0 for an invalid
 * configuration or sizes below 1). */
size_t xv_block_workspace_size(const xv_block_config* cfg, int B, int kmax, int Lmax);

/* tokens [B, k] int32 device; logits [B*k, V] fp32 device or NULL (then no
 * logits are written: the LM head leaves only per-tile argmax partials); argmax
 * [B*k] int32; n_accept [B] int32 = leading drafts equal to the argmax of the
 * position before them (0..k-1).  Requires 1 <= k <= st->kmax, B == st->B,
 * B*k <= XV_GEMM_M_MAX, st->max_ctx + k <= Lmax.  Appends the k rows to the KV
 * caches (uncommitted), replays the pending GDN steps into the states and
 * records this call's GDN inputs as the next pending steps.  Once the call's
 * work has run on the stream, the workspace begins (offset 0) with the
 * residual stream after the last layer, i.e. the hidden state before the final
 * RMSNorm: bf16 [B*k][H], row b*k + j for position j of sequence b; it stays
 * there until the workspace is used again.
 * Errors: XV_ERR_ARG (invalid configuration, incomplete weights or state, null
 * tokens/argmax/n_accept, k outside [1, kmax], the previous verify not yet
 * committed, st->max_ctx + k > Lmax, pending_rows out of range),
 * XV_ERR_UNSUPPORTED (B*k > XV_GEMM_M_MAX, unaligned buffers, shapes the
 * kernels do not take), XV_ERR_WORKSPACE, XV_ERR_CUDA.  Nothing is enqueued
 * when a host check fails; token ids or lengths found out of range on the
 * device are clamped and reported by xv_device_check. */
xv_status xv_verify_block(const xv_block_config* cfg, const xv_block_weights* w, xv_block_state* st,
                          const int32_t* tokens, int k, float* logits, int32_t* argmax, int32_t* n_accept,
                          void* ws, size_t ws_bytes, xv_stream s);

/* xv_verify_block followed by xv_block_commit_accepted, the step of a greedy
 * speculative loop, with one launch fewer: the acceptance kernel commits each
 * sequence's accepted drafts + 1 itself (ctx_len += n_accept[b] + 1,
 * n_commit = n_accept[b] + 1) and the host-side state advances as the commit
 * would advance it.  Arguments, errors and every bit of the outputs and of
 * the state as with the two calls. */
xv_status xv_verify_block_commit_accepted(const xv_block_config* cfg, const xv_block_weights* w, xv_block_state* st,
                                          const int32_t* tokens, int k, float* logits, int32_t* argmax,
                                          int32_t* n_accept, void* ws, size_t ws_bytes, xv_stream s);

/* One step of a host-driven greedy speculative loop, all enqueued on the stream by one call:
 * the drafts host_tokens [B, k] int32 (pinned host memory) are copied into dev_tokens (device,
 * [B, k]), xv_verify_block_commit_accepted runs (no logits), and the results are copied back:
 * dev_results (device, [B*kmax + B] int32: an argmax region of B*kmax entries, of which row
 * b*k + j holds position j of sequence b and entries from B*k on are left as they were, then
 * n_accept [B]) into host_results (pinned host memory, the same layout).  The caller synchronises the stream before
 * reading host_results.  Errors as for xv_verify_block, and XV_ERR_ARG for a null buffer. */
xv_status xv_block_step_host(const xv_block_config* cfg, const xv_block_weights* w, xv_block_state* st,
                             const int32_t* host_tokens, int32_t* dev_tokens, int k, int32_t* dev_results,
                             int32_t* host_results, void* ws, size_t ws_bytes, xv_stream s);

/* Verify with a number of tokens per sequence: sequence b verifies k_b =
 * k_seq[b] tokens (device [B] int32, 1 <= k_b <= k), laid out as the first
 * k_b of its k rows in tokens [B, k]; rows k_b..k-1 are padding (any valid
 * token ids).  Rows below k_b get the bits a call with k = k_b (or k_b
 * decode steps) gives them; the outputs of padding rows are unspecified.
 * n_accept[b] counts drafts among the k_b - 1 of sequence b.  k_seq must
 * stay unchanged until the commit, which keeps 1..k_b positions of sequence
 * b (a count outside is recorded as device error bit 8 and clamped).
 * k_seq = NULL is xv_verify_block. */
xv_status xv_verify_block_ragged(const xv_block_config* cfg, const xv_block_weights* w, xv_block_state* st,
                                 const int32_t* tokens, int k, const int32_t* k_seq, float* logits, int32_t* argmax,
                                 int32_t* n_accept, void* ws, size_t ws_bytes, xv_stream s);

/* Commit n_keep[b] (device, 1..k) positions of the last verify: ctx_len += n_keep,
 * n_commit = n_keep; flips the history parity and advances max_ctx by the k of
 * that verify.  [post]: the result must also be exact with every draft forced
 * to reject (n_keep = 1).  Errors: XV_ERR_ARG (null state or counts, no
 * uncommitted verify), XV_ERR_CUDA; a count outside 1..k is clamped on the
 * device and reported by xv_device_check. */
xv_status xv_block_commit(xv_block_state* st, const int32_t* n_keep, xv_stream s);

/* Standard commit: n_keep = n_accept + 1 (device arrays). */
xv_status xv_block_commit_accepted(xv_block_state* st, const int32_t* n_accept, xv_stream s);

/* Replays the pending GDN steps of every GDN layer into its state (k = 0
 * verify per layer) and zeroes n_commit, so the states hold the committed
 * position.  Needs the same cfg as the verify calls.  Errors: XV_ERR_ARG
 * (invalid configuration or state, an uncommitted verify), XV_ERR_CUDA. */
xv_status xv_block_flush(const xv_block_config* cfg, xv_block_state* st, xv_stream s);

/* Exact chunked prefill.  Feeds tokens [B, T] (int32 device, row b = the
 * next T tokens of sequence b) through the verify pass in chunks of `chunk`
 * tokens (the last one shorter if T % chunk != 0) and commits every
 * position, all enqueued on `s` without a host synchronisation.  Because a
 * verify gives the bits of decoding its tokens one at a time and a commit
 * of all k positions is the same state as k decode steps, the KV caches,
 * GDN (and convolution) states and lengths afterwards are bit-identical to T
 * decode steps, for every chunk size: batch-invariant by construction.
 * last_logits [B, V] fp32 and last_argmax [B] int32 (device, each may be
 * NULL) receive the logits and greedy token after each sequence's last
 * prompt token; only the last chunk runs the LM head.  1 <= chunk <= st->kmax,
 * B*chunk <= XV_GEMM_M_MAX (so a prefill of one sequence takes chunks of up to 64
 * tokens); the last verify must have been committed; st->max_ctx + T <= Lmax.
 * Workspace: xv_block_prefill_workspace_size(cfg, B, kmax, Lmax) (0 for an
 * invalid configuration).  Errors: XV_ERR_ARG (null tokens, T < 1, chunk
 * outside [1, kmax], an uncommitted verify, st->max_ctx + T > Lmax, and every
 * error of xv_verify_block), XV_ERR_UNSUPPORTED (B*chunk > XV_GEMM_M_MAX),
 * XV_ERR_WORKSPACE, XV_ERR_CUDA.  The limits are checked before anything is
 * enqueued; a failure inside a later chunk leaves the chunks before it
 * committed. */
size_t xv_block_prefill_workspace_size(const xv_block_config* cfg, int B, int kmax, int Lmax);
xv_status xv_block_prefill(const xv_block_config* cfg, const xv_block_weights* w, xv_block_state* st,
                           const int32_t* tokens, int T, int chunk, float* last_logits, int32_t* last_argmax,
                           void* ws, size_t ws_bytes, xv_stream s);

#ifdef __cplusplus
}
#endif
#endif /* XV_H_ */
