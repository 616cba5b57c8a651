// C-ABI entry points of libxv.so (except the block, in block.cu): argument
// validation, error reporting, the device error word and tensor-map encoding.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "xv_internal.h"

namespace xv {

namespace {
thread_local char g_msg[512] = "";
std::atomic<unsigned long long> g_launches{0};
std::atomic<bool> g_overlap{true};

// One error word per device; kernels OR error bits into it.
__device__ unsigned g_dev_err;
constexpr int MAX_DEVICES = 64;
unsigned* g_err_ptr[MAX_DEVICES] = {};
std::mutex g_err_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// Kernels whose dynamic shared-memory size has been raised, per device (function
// attributes belong to the device that was current when they were set).
struct AttrSet {
    int dev;
    const void* fn;
    int bytes;
};
std::vector<AttrSet> g_attr_set;
int g_sm_count[MAX_DEVICES] = {};
std::mutex g_attr_mu;

EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

bool overlap_enabled() { return g_overlap.load(std::memory_order_relaxed); }

xv_status fail(xv_status code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return code;
}

xv_status cuda_check(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return XV_OK;
    return fail(XV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

namespace {
struct Trace {
    bool on = false;
    int capacity = 0, count = 0;
    std::vector<cudaEvent_t> ev;
    std::vector<int> kind;
    std::vector<long long> bytes;
} g_trace;
const char* const KIND_NAMES[K_COUNT] = {"gemm_small_m", "gdn", "attn_split", "attn_combine", "kv_append", "embed",
                                         "rmsnorm", "swiglu", "gdn_gates", "argmax", "accept", "commit", "zero",
                                         "conv", "gated_norm", "gemm_combine", "tile_weights"};
}  // namespace

void trace_pre(cudaStream_t s) {
    if (g_trace.on && g_trace.count < g_trace.capacity) cudaEventRecord(g_trace.ev[2 * g_trace.count], s);
}

xv_status launched(const char* what, cudaStream_t s, int kind, long long bytes) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    xv_status st = cuda_check(cudaGetLastError(), what);
    if (g_trace.on && g_trace.count < g_trace.capacity) {
        cudaEventRecord(g_trace.ev[2 * g_trace.count + 1], s);
        g_trace.kind[g_trace.count] = kind;
        g_trace.bytes[g_trace.count] = bytes;
        ++g_trace.count;
    }
    return st;
}

xv_status kernel_smem_once(const void* fn, int bytes, bool max_carveout, const char* what) {
    int dev = 0;
    if (xv_status st = cuda_check(cudaGetDevice(&dev), what)) return st;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    for (const AttrSet& a : g_attr_set)
        if (a.dev == dev && a.fn == fn && a.bytes >= bytes) return XV_OK;
    if (max_carveout)
        if (xv_status st = cuda_check(cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100), what))
            return st;
    if (xv_status st = cuda_check(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes), what))
        return st;
    for (AttrSet& a : g_attr_set)
        if (a.dev == dev && a.fn == fn) {
            a.bytes = bytes;
            return XV_OK;
        }
    g_attr_set.push_back(AttrSet{dev, fn, bytes});
    return XV_OK;
}

xv_status device_sm_count(int* out) {
    int dev = 0;
    if (xv_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return st;
    if (dev < 0 || dev >= MAX_DEVICES) return fail(XV_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (!g_sm_count[dev])
        if (xv_status st = cuda_check(cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev),
                                      "SM count"))
            return st;
    *out = g_sm_count[dev];
    return XV_OK;
}

unsigned* device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
    std::lock_guard<std::mutex> lk(g_err_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dev_err) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<unsigned*>(p);
    }
    return g_err_ptr[dev];
}

xv_status encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    if (!g_encode) return fail(XV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides_bytes[i];
    }
    CUresult r = g_encode(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, st, b, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(XV_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return XV_OK;
}

}  // namespace xv

using namespace xv;

extern "C" {

int xv_abi_version(void) { return XV_ABI_VERSION; }

const char* xv_last_error(void) { return g_msg; }

unsigned long long xv_launch_count(void) { return g_launches.load(); }

xv_status xv_set_overlap(int enable) {
    g_overlap.store(enable != 0);
    return XV_OK;
}

xv_status xv_trace_enable(int capacity) {
    if (capacity < 1) return fail(XV_ERR_ARG, "trace: capacity must be >= 1");
    if (capacity > g_trace.capacity) {
        for (cudaEvent_t e : g_trace.ev) cudaEventDestroy(e);
        g_trace.ev.assign(2 * capacity, nullptr);
        for (auto& e : g_trace.ev)
            if (xv_status st = cuda_check(cudaEventCreate(&e), "trace: cudaEventCreate")) return st;
        g_trace.kind.assign(capacity, 0);
        g_trace.bytes.assign(capacity, 0);
        g_trace.capacity = capacity;
    }
    g_trace.count = 0;
    g_trace.on = true;
    return XV_OK;
}

xv_status xv_trace_disable(void) {
    g_trace.on = false;
    return XV_OK;
}

int xv_trace_count(void) { return g_trace.count; }

xv_status xv_trace_read(float* ms, int* kind, long long* bytes, int n) {
    if (n < 0 || n > g_trace.count) return fail(XV_ERR_ARG, "trace: %d records requested, %d recorded", n, g_trace.count);
    for (int i = 0; i < n; ++i) {
        if (ms) {
            if (xv_status st = cuda_check(cudaEventSynchronize(g_trace.ev[2 * i + 1]), "trace: cudaEventSynchronize"))
                return st;
            if (xv_status st = cuda_check(cudaEventElapsedTime(&ms[i], g_trace.ev[2 * i], g_trace.ev[2 * i + 1]),
                                          "trace: cudaEventElapsedTime"))
                return st;
        }
        if (kind) kind[i] = g_trace.kind[i];
        if (bytes) bytes[i] = g_trace.bytes[i];
    }
    return XV_OK;
}

const char* xv_trace_kind_name(int kind) { return (kind >= 0 && kind < K_COUNT) ? KIND_NAMES[kind] : "?"; }

xv_status xv_device_check(xv_stream s, unsigned* code) {
    unsigned* w = device_error_word();
    if (!w) return fail(XV_ERR_CUDA, "cannot resolve the device error word");
    xv_status st = cuda_check(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    if (st) return st;
    unsigned v = 0;
    if ((st = cuda_check(cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost), "read device error word"))) return st;
    if (v) {
        unsigned zero = 0;
        if ((st = cuda_check(cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice), "clear device error word")))
            return st;
    }
    if (code) *code = v;
    if (v) return fail(XV_ERR_DEVICE_CHECK, "device-side error bits 0x%x", v);
    return XV_OK;
}

// ------------------------------------------------------------------ GEMM

int xv_gemm_splits(int N, int K) { return (N > 0 && K > 0) ? gemm_splits(N, K) : 0; }

size_t xv_gemm_workspace_size(int M, int N, int K) {
    if (M < 1 || N < 1 || K < 1) return 0;
    return gemm_workspace_size(M, N, K);
}

static xv_status gemm_checks(const uint16_t* X, int ldx, const uint16_t* W, const void* Y, int ldy, int M, int N, int K,
                             const void* ws, size_t ws_bytes, bool split = true) {
    if (!X || !W || !Y) return fail(XV_ERR_ARG, "gemm: null X, W or Y");
    if (M < 1 || N < 1 || K < 8) return fail(XV_ERR_ARG, "gemm: need M >= 1, N >= 1, K >= 8 (got %d, %d, %d)", M, N, K);
    if (M > XV_GEMM_M_MAX) return fail(XV_ERR_UNSUPPORTED, "gemm: M = %d exceeds %d", M, XV_GEMM_M_MAX);
    if (ldx < K || ldy < N) return fail(XV_ERR_ARG, "gemm: ldx < K or ldy < N");
    if (K % 8 || ldx % 8) return fail(XV_ERR_UNSUPPORTED, "gemm: K and ldx must be multiples of 8");
    if (!aligned16(X) || !aligned16(W)) return fail(XV_ERR_UNSUPPORTED, "gemm: X and W must be 16-byte aligned");
    size_t need = split ? gemm_workspace_size(M, N, K) : 0;
    if (need && (!ws || ws_bytes < need))
        return fail(XV_ERR_WORKSPACE, "gemm: workspace of %zu bytes needed, %zu given", need, ws ? ws_bytes : 0);
    return XV_OK;
}

xv_status xv_gemm_small_m(const uint16_t* X, int ldx, const uint16_t* W, uint16_t* Y, int ldy, int M, int N, int K,
                          void* ws, size_t ws_bytes, xv_stream s) {
    if (xv_status st = gemm_checks(X, ldx, W, Y, ldy, M, N, K, ws, ws_bytes)) return st;
    return gemm_launch(X, ldx, W, W_ROWS, Y, ldy, false, M, N, K, ws, ws_bytes, reinterpret_cast<cudaStream_t>(s));
}

xv_status xv_gemm_small_m_f32out(const uint16_t* X, int ldx, const uint16_t* W, float* Y, int ldy, int M, int N, int K,
                                 void* ws, size_t ws_bytes, xv_stream s) {
    if (xv_status st = gemm_checks(X, ldx, W, Y, ldy, M, N, K, ws, ws_bytes)) return st;
    return gemm_launch(X, ldx, W, W_ROWS, Y, ldy, true, M, N, K, ws, ws_bytes, reinterpret_cast<cudaStream_t>(s));
}

size_t xv_gemm_tiled_bytes(int N, int K) { return (N < 1 || K < 1) ? 0 : gemm_tiled_bytes(N, K); }

xv_status xv_gemm_tile_weights(const uint16_t* W, int N, int K, uint16_t* Wt, xv_stream s) {
    if (!W || !Wt) return fail(XV_ERR_ARG, "tile weights: null W or Wt");
    if (N < 1 || K < 8) return fail(XV_ERR_ARG, "tile weights: need N >= 1, K >= 8 (got %d, %d)", N, K);
    if (K % 8) return fail(XV_ERR_UNSUPPORTED, "tile weights: K must be a multiple of 8");
    if (!aligned16(W) || !aligned16(Wt)) return fail(XV_ERR_UNSUPPORTED, "tile weights: W and Wt must be 16-byte aligned");
    return gemm_tile_weights_launch(W, N, K, false, Wt, reinterpret_cast<cudaStream_t>(s));
}

xv_status xv_gemm_tile_gate_up(const uint16_t* W, int F, int K, uint16_t* Wt, xv_stream s) {
    if (!W || !Wt) return fail(XV_ERR_ARG, "tile gate/up: null W or Wt");
    if (F < 1 || K < 8) return fail(XV_ERR_ARG, "tile gate/up: need F >= 1, K >= 8 (got %d, %d)", F, K);
    if (F % 64 || K % 8) return fail(XV_ERR_UNSUPPORTED, "tile gate/up: F must be a multiple of 64 and K of 8");
    if (!aligned16(W) || !aligned16(Wt)) return fail(XV_ERR_UNSUPPORTED, "tile gate/up: W and Wt must be 16-byte aligned");
    return gemm_tile_weights_launch(W, 2 * F, K, true, Wt, reinterpret_cast<cudaStream_t>(s));
}

xv_status xv_gemm_swiglu_tiled(const uint16_t* X, int ldx, const uint16_t* Wt, uint16_t* act, int ldact, int M, int F,
                               int K, xv_stream s) {
    if (!act) return fail(XV_ERR_ARG, "gemm swiglu: null act");
    if (F < 1 || F % 64) return fail(XV_ERR_UNSUPPORTED, "gemm swiglu: F must be a positive multiple of 64");
    if (ldact < F) return fail(XV_ERR_ARG, "gemm swiglu: ldact < F");
    if (xv_status st = gemm_checks(X, ldx, Wt, act, 2 * F, M, 2 * F, K, nullptr, 0, false)) return st;
    return gemm_launch(X, ldx, Wt, W_GATED, act, ldact, false, M, 2 * F, K, nullptr, 0, reinterpret_cast<cudaStream_t>(s));
}

xv_status xv_gemm_small_m_tiled(const uint16_t* X, int ldx, const uint16_t* Wt, uint16_t* Y, int ldy, int M, int N,
                                int K, void* ws, size_t ws_bytes, xv_stream s) {
    if (xv_status st = gemm_checks(X, ldx, Wt, Y, ldy, M, N, K, ws, ws_bytes)) return st;
    return gemm_launch(X, ldx, Wt, W_TILED, Y, ldy, false, M, N, K, ws, ws_bytes, reinterpret_cast<cudaStream_t>(s));
}

xv_status xv_gemm_small_m_tiled_f32out(const uint16_t* X, int ldx, const uint16_t* Wt, float* Y, int ldy, int M,
                                       int N, int K, void* ws, size_t ws_bytes, xv_stream s) {
    if (xv_status st = gemm_checks(X, ldx, Wt, Y, ldy, M, N, K, ws, ws_bytes)) return st;
    return gemm_launch(X, ldx, Wt, W_TILED, Y, ldy, true, M, N, K, ws, ws_bytes, reinterpret_cast<cudaStream_t>(s));
}

// ------------------------------------------------------------------- GDN

static xv_status gdn_dims(int B, int H, int dk, int dv) {
    if (B < 1 || H < 1) return fail(XV_ERR_ARG, "gdn: need B >= 1 and H >= 1");
    if (dk != 64 && dk != 128) return fail(XV_ERR_UNSUPPORTED, "gdn: dk must be 64 or 128 (got %d)", dk);
    if (dv < 32 || dv % 32) return fail(XV_ERR_UNSUPPORTED, "gdn: dv must be a positive multiple of 32 (got %d)", dv);
    if (B > 65535 || H > 65535) return fail(XV_ERR_UNSUPPORTED, "gdn: B and H must be below 65536");
    return XV_OK;
}

static xv_status gdn_steps_ok(const xv_gdn_steps* st, const char* which, int dk, int H) {
    if (!st) return fail(XV_ERR_ARG, "gdn: %s steps missing", which);
    if (!st->q || !st->k || !st->v || !st->beta || !st->gate) return fail(XV_ERR_ARG, "gdn: null pointer in %s", which);
    if (st->rows_per_seq < 1) return fail(XV_ERR_ARG, "gdn: %s.rows_per_seq must be >= 1", which);
    if (st->qkv_stride < 0 || st->gate_stride < H) return fail(XV_ERR_ARG, "gdn: bad strides in %s", which);
    if (!aligned16(st->q) || !aligned16(st->k) || !aligned16(st->v) || (st->qkv_stride % 8))
        return fail(XV_ERR_UNSUPPORTED, "gdn: q, k and v of %s must be 16-byte aligned with qkv_stride %% 8 == 0", which);
    (void)dk;
    return XV_OK;
}

static GdnStepsDev to_dev(const xv_gdn_steps& s) {
    return GdnStepsDev{s.q, s.k, s.v, s.beta, s.gate, s.qkv_stride, s.gate_stride, s.rows_per_seq};
}

xv_status xv_gdn_decode_step(float* state, const xv_gdn_steps* step, uint16_t* o, long long o_stride, int B, int H,
                             int dk, int dv, int qk_l2norm, xv_stream s) {
    if (xv_status st = gdn_dims(B, H, dk, dv)) return st;
    if (!state || !o) return fail(XV_ERR_ARG, "gdn: null state or o");
    if (xv_status st = gdn_steps_ok(step, "step", dk, H)) return st;
    if (o_stride < (long long)H * dv) return fail(XV_ERR_ARG, "gdn: o_stride below H*dv");
    GdnStepsDev p = to_dev(*step), none{};
    return gdn_launch(state, p, nullptr, 1, 1, true, none, 0, o, o_stride, B, H, H, dk, dv, qk_l2norm,
                      reinterpret_cast<cudaStream_t>(s));
}

xv_status xv_gdn_verify(float* state, const xv_gdn_steps* pending, const int32_t* n_commit, int max_commit,
                        const xv_gdn_steps* draft, int k, uint16_t* o, long long o_stride, int B, int H, int dk, int dv,
                        int qk_l2norm, xv_stream s) {
    return xv_gdn_verify_grouped(state, pending, n_commit, max_commit, draft, k, o, o_stride, B, H, H, dk, dv, qk_l2norm,
                                 s);
}

xv_status xv_gdn_verify_grouped(float* state, const xv_gdn_steps* pending, const int32_t* n_commit, int max_commit,
                                const xv_gdn_steps* draft, int k, uint16_t* o, long long o_stride, int B, int H, int Hk,
                                int dk, int dv, int qk_l2norm, xv_stream s) {
    if (xv_status st = gdn_dims(B, H, dk, dv)) return st;
    if (Hk < 1 || H % Hk) return fail(XV_ERR_ARG, "gdn: H = %d is not a multiple of Hk = %d", H, Hk);
    if (!state) return fail(XV_ERR_ARG, "gdn: null state");
    if (k < 0 || k > XV_KMAX) return fail(XV_ERR_UNSUPPORTED, "gdn: k = %d outside [0, %d]", k, XV_KMAX);
    if (max_commit < 0 || max_commit > XV_KMAX)
        return fail(XV_ERR_UNSUPPORTED, "gdn: max_commit = %d outside [0, %d]", max_commit, XV_KMAX);
    if (max_commit > 0) {
        if (!n_commit) return fail(XV_ERR_ARG, "gdn: n_commit missing");
        if (xv_status st = gdn_steps_ok(pending, "pending", dk, H)) return st;
        if (pending->rows_per_seq < max_commit) return fail(XV_ERR_ARG, "gdn: pending.rows_per_seq < max_commit");
    }
    if (k > 0) {
        if (xv_status st = gdn_steps_ok(draft, "draft", dk, H)) return st;
        if (draft->rows_per_seq < k) return fail(XV_ERR_ARG, "gdn: draft.rows_per_seq < k");
        if (!o) return fail(XV_ERR_ARG, "gdn: null o");
        if (o_stride < (long long)H * dv) return fail(XV_ERR_ARG, "gdn: o_stride below H*dv");
    }
    if (k == 0 && max_commit == 0) return XV_OK;
    GdnStepsDev p = max_commit > 0 ? to_dev(*pending) : GdnStepsDev{};
    GdnStepsDev d = k > 0 ? to_dev(*draft) : GdnStepsDev{};
    return gdn_launch(state, p, max_commit > 0 ? n_commit : nullptr, 0, max_commit, false, d, k, o, o_stride, B, H, Hk,
                      dk, dv, qk_l2norm, reinterpret_cast<cudaStream_t>(s));
}

// ------------------------------------------------ complete GDN layer parts

xv_status xv_gdn_conv(uint16_t* state, const uint16_t* pend, long long pend_stride, int pend_rows,
                      const int32_t* n_commit, int max_commit, const uint16_t* x, long long x_stride, int x_rows, int k,
                      const uint16_t* w, int C, int Kc, int B, uint16_t* y, long long y_stride, xv_stream s) {
    if (!state || (k > 0 && !w)) return fail(XV_ERR_ARG, "conv: null state or taps");
    if (B < 1 || B > 65535 || C < 1) return fail(XV_ERR_ARG, "conv: need 1 <= B <= 65535 and C >= 1");
    if (Kc < 2 || Kc > XV_CONV_MAX) return fail(XV_ERR_UNSUPPORTED, "conv: width %d outside [2, %d]", Kc, XV_CONV_MAX);
    if (k < 0 || k > XV_KMAX || max_commit < 0 || max_commit > XV_KMAX)
        return fail(XV_ERR_UNSUPPORTED, "conv: k and max_commit must lie in [0, %d]", XV_KMAX);
    if (max_commit > 0 && (!pend || !n_commit || pend_rows < max_commit || pend_stride < C))
        return fail(XV_ERR_ARG, "conv: pending rows need pend, n_commit, pend_rows >= max_commit, pend_stride >= C");
    if (k > 0 && (!x || !y || x_rows < k || x_stride < C || y_stride < C))
        return fail(XV_ERR_ARG, "conv: the k rows need x, y, x_rows >= k and strides >= C");
    if (k == 0 && max_commit == 0) return XV_OK;
    return conv_launch(state, pend, pend_stride, pend_rows, n_commit, max_commit, x, x_stride, x_rows, k, w, C, Kc, B, y,
                       y_stride, reinterpret_cast<cudaStream_t>(s));
}

xv_status xv_gated_norm(const uint16_t* o, long long o_stride, const uint16_t* z, long long z_stride, const uint16_t* w,
                        int M, int H, int dv, float eps, uint16_t* y, long long y_stride, xv_stream s) {
    if (!o || !z || !w || !y) return fail(XV_ERR_ARG, "gated norm: null pointer");
    if (M < 1 || H < 1) return fail(XV_ERR_ARG, "gated norm: need M >= 1 and H >= 1");
    if (dv < 32 || dv % 32 || dv > 256) return fail(XV_ERR_UNSUPPORTED, "gated norm: dv must be a multiple of 32 up to 256");
    const long long row = static_cast<long long>(H) * dv;
    if (o_stride < row || z_stride < row || y_stride < row) return fail(XV_ERR_ARG, "gated norm: row strides below H*dv");
    if (static_cast<long long>(M) * H > (1ll << 30)) return fail(XV_ERR_UNSUPPORTED, "gated norm: too many rows");
    return gated_norm_launch(o, o_stride, z, z_stride, w, M, H, dv, eps, y, y_stride, reinterpret_cast<cudaStream_t>(s));
}

// ------------------------------------------------------------- attention

int xv_attn_split_begin(int s) { return s < 0 ? -1 : attn_split_begin(s); }

size_t xv_attn_workspace_size(int B, int R, int Hq, int hd, int max_ctx) {
    if (B < 1 || R < 1 || Hq < 1 || hd < 1 || max_ctx < 1) return 0;
    return attn_workspace_size(B, R, Hq, hd, max_ctx);
}

static xv_status attn_checks(const uint16_t* q, long long q_stride, const uint16_t* kc, const uint16_t* vc,
                             const int32_t* ctx_len, int R, int B, int Hq, int Hkv, int hd, int Lmax, int max_len,
                             const uint16_t* gate, long long gate_stride, const uint16_t* out, long long out_stride) {
    if (!q || !kc || !vc || !ctx_len || !out) return fail(XV_ERR_ARG, "attn: null pointer");
    if (B < 1 || R < 1 || Hq < 1 || Hkv < 1 || Lmax < 1) return fail(XV_ERR_ARG, "attn: sizes must be positive");
    if (R > XV_KMAX) return fail(XV_ERR_UNSUPPORTED, "attn: R = %d exceeds %d", R, XV_KMAX);
    if (Hq % Hkv) return fail(XV_ERR_ARG, "attn: Hq must be a multiple of Hkv");
    if (hd != 64 && hd != 256) return fail(XV_ERR_UNSUPPORTED, "attn: hd must be 64 or 256 (got %d)", hd);
    if (max_len < R || max_len > Lmax) return fail(XV_ERR_ARG, "attn: need R <= max_ctx <= Lmax");
    if (B > 65535 || Hkv > 65535) return fail(XV_ERR_UNSUPPORTED, "attn: B and Hkv must be below 65536");
    if ((long long)B * Hkv * Lmax > (1ll << 31)) return fail(XV_ERR_UNSUPPORTED, "attn: cache too large");
    if (q_stride < (long long)Hq * hd || out_stride < (long long)Hq * hd) return fail(XV_ERR_ARG, "attn: row stride below Hq*hd");
    if (gate && gate_stride < (long long)Hq * hd) return fail(XV_ERR_ARG, "attn: gate_stride below Hq*hd");
    if (!aligned16(q) || (q_stride % 8) || !aligned16(kc) || !aligned16(vc))
        return fail(XV_ERR_UNSUPPORTED, "attn: q rows and caches must be 16-byte aligned");
    return XV_OK;
}

xv_status xv_attn_decode_rows(const uint16_t* q, long long q_stride, const uint16_t* kc, const uint16_t* vc,
                              const int32_t* ctx_len, int R, int B, int Hq, int Hkv, int hd, int Lmax, int max_ctx,
                              float scale, const uint16_t* gate, long long gate_stride, uint16_t* out,
                              long long out_stride, void* ws, size_t ws_bytes, xv_stream s) {
    if (xv_status st = attn_checks(q, q_stride, kc, vc, ctx_len, R, B, Hq, Hkv, hd, Lmax, max_ctx, gate, gate_stride,
                                   out, out_stride))
        return st;
    size_t need = attn_workspace_size(B, R, Hq, hd, max_ctx);
    if (!ws || ws_bytes < need) return fail(XV_ERR_WORKSPACE, "attn: workspace of %zu bytes needed", need);
    if (!aligned16(ws)) return fail(XV_ERR_UNSUPPORTED, "attn: workspace must be 16-byte aligned");
    return attn_launch(q, q_stride, kc, vc, kv_contiguous(B, Lmax), ctx_len, 0, R, B, Hq, Hkv, hd, max_ctx, scale, gate,
                       gate_stride, out, out_stride, ws, ws_bytes, reinterpret_cast<cudaStream_t>(s));
}

// A page table and its sizes as the kernels take them; Lmax = the positions a sequence can hold.
static xv_status kv_pages_check(const xv_kv_pages* pages, int Hkv, int hd, KvPages* kv, int* Lmax) {
    if (!pages || !pages->page_table) return fail(XV_ERR_ARG, "paged KV: null page table");
    if (pages->page_size < 64 || pages->page_size % 64)
        return fail(XV_ERR_UNSUPPORTED, "paged KV: page_size must be a positive multiple of 64 (got %d)", pages->page_size);
    if (pages->max_pages < 1 || pages->n_pages < 1) return fail(XV_ERR_ARG, "paged KV: max_pages and n_pages must be positive");
    if (static_cast<long long>(pages->page_size) * pages->max_pages > (1ll << 30))
        return fail(XV_ERR_UNSUPPORTED, "paged KV: page_size * max_pages exceeds 2^30 positions");
    if (static_cast<long long>(pages->n_pages) * Hkv * pages->page_size * hd > (1ll << 40))
        return fail(XV_ERR_UNSUPPORTED, "paged KV: pool too large");
    if (static_cast<long long>(pages->n_pages) * Hkv > (1ll << 31)) return fail(XV_ERR_UNSUPPORTED, "paged KV: too many pages");
    *kv = KvPages{pages->page_table, pages->page_size, pages->max_pages, pages->n_pages};
    *Lmax = pages->page_size * pages->max_pages;
    return XV_OK;
}

xv_status xv_attn_decode_rows_paged(const uint16_t* q, long long q_stride, const uint16_t* kpool, const uint16_t* vpool,
                                    const xv_kv_pages* pages, const int32_t* ctx_len, int R, int B, int Hq, int Hkv,
                                    int hd, int max_ctx, float scale, const uint16_t* gate, long long gate_stride,
                                    uint16_t* out, long long out_stride, void* ws, size_t ws_bytes, xv_stream s) {
    KvPages kv{};
    int Lmax = 0;
    if (xv_status st = kv_pages_check(pages, Hkv, hd, &kv, &Lmax)) return st;
    // the pool is addressed as one cache of n_pages sequences of page_size positions
    if (xv_status st = attn_checks(q, q_stride, kpool, vpool, ctx_len, R, 1, Hq, Hkv, hd, kv.page, R, gate, gate_stride,
                                   out, out_stride))
        return st;
    if (B < 1 || B > 65535) return fail(XV_ERR_ARG, "attn: B must lie in [1, 65535]");
    if (max_ctx < R || max_ctx > Lmax) return fail(XV_ERR_ARG, "attn: need R <= max_ctx <= page_size * max_pages");
    size_t need = attn_workspace_size(B, R, Hq, hd, max_ctx);
    if (!ws || ws_bytes < need) return fail(XV_ERR_WORKSPACE, "attn: workspace of %zu bytes needed", need);
    if (!aligned16(ws)) return fail(XV_ERR_UNSUPPORTED, "attn: workspace must be 16-byte aligned");
    return attn_launch(q, q_stride, kpool, vpool, kv, ctx_len, 0, R, B, Hq, Hkv, hd, max_ctx, scale, gate, gate_stride,
                       out, out_stride, ws, ws_bytes, reinterpret_cast<cudaStream_t>(s));
}

xv_status xv_kv_append(const uint16_t* kv_src, long long src_stride, const int32_t* ctx_len, int R, int B, int Hkv,
                       int hd, int Lmax, uint16_t* kc, uint16_t* vc, xv_stream s) {
    if (!kv_src || !ctx_len || !kc || !vc) return fail(XV_ERR_ARG, "kv_append: null pointer");
    if (R < 1 || B < 1 || Hkv < 1 || hd < 8 || Lmax < 1 || hd % 8) return fail(XV_ERR_ARG, "kv_append: bad sizes");
    if (src_stride < 2ll * Hkv * hd) return fail(XV_ERR_ARG, "kv_append: src_stride below 2*Hkv*hd");
    if (!aligned16(kv_src) || (src_stride % 8) || !aligned16(kc) || !aligned16(vc))
        return fail(XV_ERR_UNSUPPORTED, "kv_append: 16-byte alignment required");
    return kv_append_launch(kv_src, src_stride, ctx_len, -1, R, B, Hkv, hd, kv_contiguous(B, Lmax), kc, vc,
                            reinterpret_cast<cudaStream_t>(s));
}

xv_status xv_kv_append_paged(const uint16_t* kv_src, long long src_stride, const int32_t* ctx_len, int R, int B, int Hkv,
                             int hd, const xv_kv_pages* pages, uint16_t* kpool, uint16_t* vpool, xv_stream s) {
    if (!kv_src || !ctx_len || !kpool || !vpool) return fail(XV_ERR_ARG, "kv_append: null pointer");
    if (R < 1 || B < 1 || Hkv < 1 || hd < 8 || hd % 8) return fail(XV_ERR_ARG, "kv_append: bad sizes");
    KvPages kv{};
    int Lmax = 0;
    if (xv_status st = kv_pages_check(pages, Hkv, hd, &kv, &Lmax)) return st;
    if (src_stride < 2ll * Hkv * hd) return fail(XV_ERR_ARG, "kv_append: src_stride below 2*Hkv*hd");
    if (!aligned16(kv_src) || (src_stride % 8) || !aligned16(kpool) || !aligned16(vpool))
        return fail(XV_ERR_UNSUPPORTED, "kv_append: 16-byte alignment required");
    return kv_append_launch(kv_src, src_stride, ctx_len, -1, R, B, Hkv, hd, kv, kpool, vpool,
                            reinterpret_cast<cudaStream_t>(s));
}

}  // extern "C"
