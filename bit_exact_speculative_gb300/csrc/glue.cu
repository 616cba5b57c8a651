// Row-wise glue of the verify block: embedding gather, RMSNorm (fused with the
// residual add), SwiGLU, GDN gates, argmax, greedy acceptance and commit.
//
// Every kernel here computes each row from that row alone, with a reduction
// tree fixed by the row length, so a row's bits do not depend on how many
// rows are in the call (the batch invariance that deterministic inference
// asks for: "Follow-up to my earlier post on Qwen3.8-27B decode speed",
// r/LocalLLaMA post — deterministic mode is necessary, but not sufficient).
#include <cmath>

#include "xv_internal.h"
#include "xv_ptx.cuh"

namespace xv {

namespace {
constexpr int NORM_THREADS = 256;

// Sum of v over the block in a fixed tree: xor-shuffle inside each warp, then
// warp partials added in warp order by warp 0.
__device__ __forceinline__ float block_sum_fixed(float v, float* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float t = lane < nw ? red[lane] : 0.f;
        float acc = __shfl_sync(0xffffffffu, t, 0);
        for (int w = 1; w < nw; ++w) acc = __fadd_rn(acc, __shfl_sync(0xffffffffu, t, w));
        if (lane == 0) red[32] = acc;
    }
    __syncthreads();
    const float r = red[32];
    __syncthreads();
    return r;
}

__global__ void embed_kernel(const int32_t* __restrict__ tokens, const uint16_t* __restrict__ E, int V, int H,
                             uint16_t* __restrict__ x, unsigned* err) {
    const int m = blockIdx.x;
    int t = tokens[m];
    if (t < 0 || t >= V) {
        if (threadIdx.x == 0) atomicOr(err, ERR_BAD_TOKEN);
        t = 0;
    }
    const uint4* src = reinterpret_cast<const uint4*>(E + static_cast<long long>(t) * H);
    uint4* dst = reinterpret_cast<uint4*>(x + static_cast<long long>(m) * H);
    for (int i = threadIdx.x; i < H / 8; i += blockDim.x) dst[i] = src[i];
}

// y = bf16( x / sqrt(mean(x^2) + eps) * (1 + w) ); with y_res != null first x <- bf16(x + y_res).
__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_kernel(uint16_t* __restrict__ x, const uint16_t* __restrict__ y_res,
                                                               const uint16_t* __restrict__ w, int H, float eps,
                                                               uint16_t* __restrict__ out) {
    __shared__ float red[33];
    const long long row = blockIdx.x;
    uint16_t* xr = x + row * H;
    float ss = 0.f;
    bool first = true;
    for (int i = threadIdx.x; i < H; i += blockDim.x) {
        float v = bf16_to_f32(xr[i]);
        if (y_res) {
            v = bf16_to_f32(f32_to_bf16(__fadd_rn(v, bf16_to_f32(y_res[row * H + i]))));
            xr[i] = f32_to_bf16(v);
        }
        ss = first ? __fmul_rn(v, v) : __fmaf_rn(v, v, ss);
        first = false;
    }
    ss = block_sum_fixed(ss, red);
    const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(H)), eps)));
    for (int i = threadIdx.x; i < H; i += blockDim.x) {
        const float v = bf16_to_f32(xr[i]);
        out[row * H + i] = f32_to_bf16(__fmul_rn(__fmul_rn(v, inv), __fadd_rn(1.f, bf16_to_f32(w[i]))));
    }
}

__device__ __forceinline__ float sigmoid_f(float x) { return __frcp_rn(__fadd_rn(1.f, expf(-x))); }

__global__ void swiglu_kernel(const uint16_t* __restrict__ gu, int F, uint16_t* __restrict__ act) {
    const long long row = blockIdx.y;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < F; i += gridDim.x * blockDim.x) {
        const float g = bf16_to_f32(gu[row * 2 * F + i]);
        const float u = bf16_to_f32(gu[row * 2 * F + F + i]);
        act[row * F + i] = f32_to_bf16(__fmul_rn(__fmul_rn(g, sigmoid_f(g)), u));
    }
}

// beta = bf16(sigmoid(b)), gate = bf16(exp(-softplus(a))), softplus(x) = x for x > 20
__global__ void gdn_gates_kernel(const uint16_t* __restrict__ proj, long long stride, int b_col, int H,
                                 uint16_t* __restrict__ gates) {
    const long long m = blockIdx.x;
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        const float bb = bf16_to_f32(proj[m * stride + b_col + h]);
        const float aa = bf16_to_f32(proj[m * stride + b_col + H + h]);
        const float sp = aa > 20.f ? aa : log1pf(expf(aa));
        gates[m * 2 * H + h] = f32_to_bf16(sigmoid_f(bb));
        gates[m * 2 * H + H + h] = f32_to_bf16(expf(-sp));
    }
}

// Lowest index among the maxima of each row (fixed-order tree; ties and NaN-free).
__global__ void argmax_kernel(const float* __restrict__ logits, int V, int32_t* __restrict__ idx) {
    __shared__ float sv[32];
    __shared__ int si[32];
    const long long row = blockIdx.x;
    const float* x = logits + row * V;
    float best = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = threadIdx.x; i < V; i += blockDim.x) {
        const float v = x[i];
        if (v > best) { best = v; bi = i; }   // i increases, so ties keep the lower index
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) { sv[warp] = best; si[warp] = bi; }
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        best = lane < nw ? sv[lane] : -INFINITY;
        bi = lane < nw ? si[lane] : 0x7fffffff;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, best, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
        }
        if (lane == 0) idx[row] = bi == 0x7fffffff ? 0 : bi;
    }
}

// n_accept[b] = number of leading drafts tokens[b][j+1] equal to pred[b][j]
__global__ void accept_kernel(const int32_t* __restrict__ tokens, const int32_t* __restrict__ pred, int B, int k,
                              int32_t* __restrict__ n_accept) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int n = 0;
    while (n < k - 1 && pred[b * k + n] == tokens[b * k + n + 1]) ++n;
    n_accept[b] = n;
}

__global__ void commit_kernel(const int32_t* __restrict__ keep, int keep_bias, int B, int k, int32_t* __restrict__ ctx_len,
                              int32_t* __restrict__ n_commit, unsigned* err) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int n = keep[b] + keep_bias;
    if (n < 1 || n > k) {
        atomicOr(err, ERR_BAD_COUNT);
        n = n < 1 ? 1 : k;
    }
    ctx_len[b] += n;
    n_commit[b] = n;
}

__global__ void zero_i32_kernel(int32_t* p, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) p[i] = 0;
}

}  // namespace

xv_status embed_launch(const int32_t* tokens, int M, const uint16_t* E, int V, int H, uint16_t* x, cudaStream_t s) {
    unsigned* err = device_error_word();
    if (!err) return fail(XV_ERR_CUDA, "embed: device error word unavailable");
    trace_pre(s);
    embed_kernel<<<M, 128, 0, s>>>(tokens, E, V, H, x, err);
    return launched("embed_kernel", s, K_EMBED, 4ll * M * H + 4ll * M);
}

xv_status rmsnorm_launch(const uint16_t* x, const uint16_t* w, int M, int H, float eps, uint16_t* y, cudaStream_t s) {
    trace_pre(s);
    rmsnorm_kernel<<<M, NORM_THREADS, 0, s>>>(const_cast<uint16_t*>(x), nullptr, w, H, eps, y);
    return launched("rmsnorm_kernel", s, K_RMSNORM, 4ll * M * H + 2ll * H);
}

xv_status residual_rmsnorm_launch(uint16_t* x, const uint16_t* y, const uint16_t* w, int M, int H, float eps, uint16_t* xn,
                                  cudaStream_t s) {
    trace_pre(s);
    rmsnorm_kernel<<<M, NORM_THREADS, 0, s>>>(x, y, w, H, eps, xn);
    return launched("rmsnorm_kernel(residual)", s, K_RMSNORM, 8ll * M * H + 2ll * H);
}

xv_status swiglu_launch(const uint16_t* gu, int M, int F, uint16_t* act, cudaStream_t s) {
    dim3 grid(ceil_div(F, 256 * 4), M);
    trace_pre(s);
    swiglu_kernel<<<grid, 256, 0, s>>>(gu, F, act);
    return launched("swiglu_kernel", s, K_SWIGLU, 6ll * M * F);
}

xv_status gdn_gates_launch(const uint16_t* proj, long long proj_stride, int b_col, int M, int H, uint16_t* gates,
                           cudaStream_t s) {
    trace_pre(s);
    gdn_gates_kernel<<<M, 64, 0, s>>>(proj, proj_stride, b_col, H, gates);
    return launched("gdn_gates_kernel", s, K_GATES, 8ll * M * H);
}

xv_status argmax_launch(const float* logits, int M, int V, int32_t* idx, cudaStream_t s) {
    trace_pre(s);
    argmax_kernel<<<M, 1024, 0, s>>>(logits, V, idx);
    return launched("argmax_kernel", s, K_ARGMAX, 4ll * M * V + 4ll * M);
}

xv_status accept_launch(const int32_t* tokens, const int32_t* pred, int B, int k, int32_t* n_accept, cudaStream_t s) {
    trace_pre(s);
    accept_kernel<<<ceil_div(B, 128), 128, 0, s>>>(tokens, pred, B, k, n_accept);
    return launched("accept_kernel", s, K_ACCEPT, 8ll * B * k + 4ll * B);
}

xv_status commit_launch(const int32_t* keep, int keep_bias, int B, int k, int32_t* ctx_len, int32_t* n_commit,
                        cudaStream_t s) {
    unsigned* err = device_error_word();
    if (!err) return fail(XV_ERR_CUDA, "commit: device error word unavailable");
    trace_pre(s);
    commit_kernel<<<ceil_div(B, 128), 128, 0, s>>>(keep, keep_bias, B, k, ctx_len, n_commit, err);
    return launched("commit_kernel", s, K_COMMIT, 16ll * B);
}

xv_status zero_i32_launch(int32_t* p, int n, cudaStream_t s) {
    trace_pre(s);
    zero_i32_kernel<<<ceil_div(n, 256), 256, 0, s>>>(p, n);
    return launched("zero_i32_kernel", s, K_ZERO, 4ll * n);
}

}  // namespace xv
