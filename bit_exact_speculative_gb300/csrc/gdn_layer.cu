// The parts of the complete GDN layer around the recurrence: the depthwise
// causal convolution over the q|k|v channels, whose state of prior inputs is
// committed like the recurrence state (deferred: a call first shifts in the
// kept rows of the previous call), and the per-head output RMSNorm gated by
// silu(z).
//
// Neither is printed on the pages; the layer follows gated-delta-net
// decoders:
//   u_t[c] = silu( sum_{j < Kc} w[c][j] x_{t-Kc+1+j}[c] )     x: projection outputs
//   y_h    = o_h / sqrt(mean(o_h^2) + eps) * (1 + w_n) * silu(z_h)   per v head h
// Every output is a function of its own inputs in a fixed order (taps in
// order, one rounding per multiply-add; the norm's sum in a fixed tree), so a
// verify row gets the bits of the decode step at its position, which is what
// "Follow-up to my earlier post on Qwen3.8-27B decode speed" (r/LocalLLaMA
// post) asks of every part of the verify pass.
#include "xv_internal.h"
#include "xv_ptx.cuh"

namespace xv {
namespace {

constexpr int CONV_THREADS = 128;

__device__ __forceinline__ float bfv(uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); }
__device__ __forceinline__ float silu_f(float x) { return __fmul_rn(x, __frcp_rn(__fadd_rn(1.f, expf(-x)))); }

struct ConvArgs {
    uint16_t* state;            // [B, Kc-1, C]
    const uint16_t* pend;       // pending rows (previous call's inputs), row b*pend_rows + t
    long long pend_stride;
    int pend_rows;
    const int32_t* n_commit;    // [B] or null (nothing to commit)
    int max_commit;
    const uint16_t* x;          // this call's rows, row b*x_rows + t
    long long x_stride;
    int x_rows, k;
    const uint16_t* w;          // [C, Kc]
    int C;
    uint16_t* y;                // row b*k + t
    long long y_stride;
    unsigned* err;
};

// One thread per (channel, sequence).  The new window is the last Kc-1 entries
// of (state ++ pending[0, n)); the k input rows come in predicated bursts of
// XC rows (the first burst is issued with the window's loads); the window
// slides over them in registers.
template <int KC>
__global__ void __launch_bounds__(CONV_THREADS) conv_kernel(ConvArgs A) {
    griddep_launch();
    griddep_wait();
    constexpr int W = KC - 1;
    const int c = blockIdx.x * CONV_THREADS + threadIdx.x;
    const int b = blockIdx.y;
    if (c >= A.C) return;
    uint16_t* st = A.state + static_cast<long long>(b) * W * A.C + c;
    constexpr int XC = 16;
    uint16_t old[W], win[W], xs[XC];
#pragma unroll
    for (int j = 0; j < W; ++j) old[j] = st[static_cast<long long>(j) * A.C];
    int nc = A.n_commit ? A.n_commit[b] : 0;
    if (nc < 0 || nc > A.max_commit) {
        if (c == 0) atomicOr(A.err, ERR_BAD_COUNT);
        nc = nc < 0 ? 0 : A.max_commit;
    }
    const long long prow = static_cast<long long>(b) * A.pend_rows;
#pragma unroll
    for (int j = 0; j < W; ++j) {
        const int i = nc + j;   // index in (state ++ pending)
        if (i >= W) {
            win[j] = A.pend[(prow + i - W) * A.pend_stride + c];
        } else {
            uint16_t v = 0;
#pragma unroll
            for (int q = 0; q < W; ++q)
                if (q == i) v = old[q];
            win[j] = v;
        }
    }
    const long long xrow = static_cast<long long>(b) * A.x_rows;
    auto burst = [&](int t0) {
#pragma unroll
        for (int t = 0; t < XC; ++t) xs[t] = t0 + t < A.k ? A.x[(xrow + t0 + t) * A.x_stride + c] : uint16_t(0);
    };
    burst(0);
    if (nc > 0) {
#pragma unroll
        for (int j = 0; j < W; ++j) st[static_cast<long long>(j) * A.C] = win[j];
    }
    if (A.k == 0) return;
    float w[KC];
#pragma unroll
    for (int j = 0; j < KC; ++j) w[j] = bfv(A.w[static_cast<long long>(c) * KC + j]);
    for (int t0 = 0; t0 < A.k; t0 += XC) {
        if (t0 > 0) burst(t0);
#pragma unroll
        for (int t = 0; t < XC; ++t) {
            if (t0 + t < A.k) {
                float acc = __fmul_rn(w[0], bfv(win[0]));
#pragma unroll
                for (int j = 1; j < W; ++j) acc = __fmaf_rn(w[j], bfv(win[j]), acc);
                acc = __fmaf_rn(w[W], bfv(xs[t]), acc);
                A.y[(static_cast<long long>(b) * A.k + t0 + t) * A.y_stride + c] = f32_to_bf16(silu_f(acc));
#pragma unroll
                for (int j = 0; j + 1 < W; ++j) win[j] = win[j + 1];
                win[W - 1] = xs[t];
            }
        }
    }
}

struct NormArgs {
    const uint16_t* o;
    long long o_stride;
    const uint16_t* z;
    long long z_stride;
    const uint16_t* w;
    int M, H, dv;
    float eps;
    uint16_t* y;
    long long y_stride;
};

constexpr int NORM_WARPS = 4;

// One warp per (row, head): lane l holds elements l, l + 32, ...; its squares
// are summed in that order, then across the warp by an xor tree (16, 8, 4, 2, 1).
__global__ void __launch_bounds__(32 * NORM_WARPS) gated_norm_kernel(NormArgs A) {
    griddep_launch();
    griddep_wait();
    const long long unit = static_cast<long long>(blockIdx.x) * NORM_WARPS + (threadIdx.x >> 5);
    if (unit >= static_cast<long long>(A.M) * A.H) return;
    const int lane = threadIdx.x & 31;
    const long long m = unit / A.H;
    const int h = static_cast<int>(unit % A.H);
    const uint16_t* orow = A.o + m * A.o_stride + static_cast<long long>(h) * A.dv;
    const uint16_t* zrow = A.z + m * A.z_stride + static_cast<long long>(h) * A.dv;
    constexpr int EMAX = 8;   // dv <= 256
    float v[EMAX];
    const int E = A.dv / 32;
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        if (e < E) {
            v[e] = bfv(orow[lane + 32 * e]);
            ss = e == 0 ? __fmul_rn(v[e], v[e]) : __fmaf_rn(v[e], v[e], ss);
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(A.dv)), A.eps)));
    uint16_t* yrow = A.y + m * A.y_stride + static_cast<long long>(h) * A.dv;
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        if (e < E) {
            const int i = lane + 32 * e;
            const float g = __fmul_rn(__fmul_rn(v[e], inv), __fadd_rn(1.f, bfv(A.w[i])));
            yrow[i] = f32_to_bf16(__fmul_rn(g, silu_f(bfv(zrow[i]))));
        }
    }
}

template <int KC>
void launch_conv(const ConvArgs& a, int B, cudaStream_t s) {
    launch_k(conv_kernel<KC>, dim3(ceil_div(a.C, CONV_THREADS), B), dim3(CONV_THREADS), 0, s, a);
}

}  // namespace

xv_status conv_launch(uint16_t* state, const uint16_t* pend, long long pend_stride, int pend_rows,
                      const int32_t* n_commit, int max_commit, const uint16_t* x, long long x_stride, int x_rows, int k,
                      const uint16_t* w, int C, int Kc, int B, uint16_t* y, long long y_stride, cudaStream_t s) {
    unsigned* err = device_error_word();
    if (!err) return fail(XV_ERR_CUDA, "conv: device error word unavailable");
    if (Kc < 2 || Kc > XV_CONV_MAX) return fail(XV_ERR_UNSUPPORTED, "conv: width %d outside [2, %d]", Kc, XV_CONV_MAX);
    if (k < 0 || k > XV_KMAX || max_commit < 0 || max_commit > XV_KMAX)
        return fail(XV_ERR_UNSUPPORTED, "conv: k and max_commit must lie in [0, %d]", XV_KMAX);
    ConvArgs a{state, pend, pend_stride, pend_rows, max_commit > 0 ? n_commit : nullptr, max_commit, x, x_stride, x_rows,
               k, w, C, y, y_stride, err};
    trace_pre(s);
    switch (Kc) {
        case 2: launch_conv<2>(a, B, s); break;
        case 3: launch_conv<3>(a, B, s); break;
        case 4: launch_conv<4>(a, B, s); break;
        case 5: launch_conv<5>(a, B, s); break;
        case 6: launch_conv<6>(a, B, s); break;
        case 7: launch_conv<7>(a, B, s); break;
        default: launch_conv<8>(a, B, s); break;
    }
    const long long bytes = 2ll * B * C * (2 * (Kc - 1) + max_commit + 2 * k) + 2ll * C * Kc;
    return launched("conv_kernel", s, K_CONV, bytes);
}

xv_status gated_norm_launch(const uint16_t* o, long long o_stride, const uint16_t* z, long long z_stride,
                            const uint16_t* w, int M, int H, int dv, float eps, uint16_t* y, long long y_stride,
                            cudaStream_t s) {
    if (dv < 32 || dv % 32 || dv > 256) return fail(XV_ERR_UNSUPPORTED, "gated norm: dv must be a multiple of 32 up to 256");
    NormArgs a{o, o_stride, z, z_stride, w, M, H, dv, eps, y, y_stride};
    trace_pre(s);
    launch_k(gated_norm_kernel, dim3(ceil_div(static_cast<long long>(M) * H, NORM_WARPS)), dim3(32 * NORM_WARPS), 0, s, a);
    return launched("gated_norm_kernel", s, K_GNORM, 6ll * M * H * dv + 2ll * dv);
}

}  // namespace xv
