// xv_gemm_small_m_noalloc: the small-M GEMM for callers that cannot allocate.
//
// Some callers of this library cannot call cudaMalloc or hand over a
// workspace: code that runs inside another framework's memory pool and may
// not touch the allocator, plugins loaded into a host process that owns all
// device memory, or real-time loops where an allocation (and the
// synchronisation it can imply) is not allowed.  For them this entry point
// runs the same GEMM kernel as xv_gemm_small_m with its scratch — the split-K
// partial sums and the per-tile arrival counters — in a fixed array that
// lives in this library's own device memory.  The caller still provides X, W
// and Y.
//
// The array is a file-scope __device__ object of XV_GEMM_NOALLOC_SCRATCH_BYTES
// per GPU that loads the library, held until the process exits.  Host code
// cannot use its name as a device address, so the first call on each device
// looks the address up with cudaGetSymbolAddress (with that device current)
// and caches it; that first call should therefore come before any stream
// capture.  The per-tile arrival counters at the start of the array must be
// zero when a split GEMM starts; a GEMM that completes leaves them zero, but
// one whose bounded wait gave up (xv_device_check reports bit 0) may not, so
// every call whose shape uses them first clears them on the caller's stream.
// All calls share the one array: calls whose kernels overlap on the GPU (other
// streams, other host threads) race and must be serialised by the caller.
#include <mutex>

#include "xv_internal.h"

namespace xv {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[XV_GEMM_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
void* g_scratch_ptr[MAX_DEVICES] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set-up on first use).
xv_status scratch_address(void** out) {
    int dev = 0;
    if (xv_status st = cuda_check(cudaGetDevice(&dev), "gemm_noalloc: cudaGetDevice")) return st;
    if (dev < 0 || dev >= MAX_DEVICES) return fail(XV_ERR_CUDA, "gemm_noalloc: device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (xv_status st = cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch), "gemm_noalloc: cudaGetSymbolAddress"))
            return st;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return XV_OK;
}

}  // namespace
}  // namespace xv

using namespace xv;

extern "C" xv_status xv_gemm_small_m_noalloc(const uint16_t* X, int ldx, const uint16_t* W, uint16_t* Y, int ldy, int M,
                                             int N, int K, xv_stream stream) {
    if (!X || !W || !Y) return fail(XV_ERR_ARG, "gemm_noalloc: null X, W or Y");
    if (M < 1 || N < 1 || K < 8) return fail(XV_ERR_ARG, "gemm_noalloc: need M >= 1, N >= 1, K >= 8");
    if (M > XV_GEMM_M_MAX) return fail(XV_ERR_UNSUPPORTED, "gemm_noalloc: M = %d exceeds %d", M, XV_GEMM_M_MAX);
    if (ldx < K || ldy < N) return fail(XV_ERR_ARG, "gemm_noalloc: ldx < K or ldy < N");
    if (K % 8 || ldx % 8) return fail(XV_ERR_UNSUPPORTED, "gemm_noalloc: K and ldx must be multiples of 8");
    if (!aligned16(X) || !aligned16(W)) return fail(XV_ERR_UNSUPPORTED, "gemm_noalloc: X and W must be 16-byte aligned");
    const size_t need = gemm_workspace_size(M, N, K);
    if (need > XV_GEMM_NOALLOC_SCRATCH_BYTES)
        return fail(XV_ERR_UNSUPPORTED,
                    "gemm_noalloc: M=%d N=%d K=%d needs %zu bytes of scratch, more than the fixed %zu bytes; "
                    "use xv_gemm_small_m with a workspace",
                    M, N, K, need, static_cast<size_t>(XV_GEMM_NOALLOC_SCRATCH_BYTES));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void* scratch = nullptr;
    if (xv_status st = scratch_address(&scratch)) return st;
    if (gemm_uses_counters(M, N, K))
        if (xv_status st = cuda_check(cudaMemsetAsync(scratch, 0, GEMM_COUNTER_BYTES, s), "gemm_noalloc: clear counters"))
            return st;
    return gemm_launch(X, ldx, W, W_ROWS, Y, ldy, false, M, N, K, scratch, XV_GEMM_NOALLOC_SCRATCH_BYTES, s);
}
