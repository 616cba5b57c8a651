// Row-wise glue of the verify block: embedding gather, RMSNorm (fused with the
// residual add), SwiGLU, argmax, greedy acceptance and commit.
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

// y = bf16( x / sqrt(mean(x^2) + eps) * (1 + w) ); with y_res != null first x <- bf16(x + y_res);
// with tokens != null the row is first gathered from the embedding, x <- E[tokens[row]].
// A thread-block cluster of NORM_CL CTAs per row: CTA q owns the 8-element chunks
// [q cpc, (q + 1) cpc) of the row (cpc = ceil(H / 8 / NORM_CL)) and its thread t the chunks
// q cpc + t, + nt, ... (at most NORM_MAXC).  The sum of squares runs per thread in chunk and
// element order, through a fixed shuffle tree per warp, over the warps in order per CTA, and
// over the CTAs in rank order (every CTA reads all the CTA sums over distributed shared memory
// and adds them the same way), so its order is fixed by H alone.
//
// With part != null, y_res is instead bf16(part_0 + ... + part_{S-1}), a GEMM's split-K partials
// [S][M][H] added in segment order (the bits of the GEMM's own combine), formed by the chunk's
// owner.  Spreading a row over a cluster (rather than one CTA per row) spreads those partial
// loads over NORM_CL SMs: measured at 8 rows, a row of 7 partials is 140 KB.
constexpr int NORM_MAXC = 4;
constexpr int NORM_CL = 8;

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ uint4 pack8(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = static_cast<uint32_t>(f32_to_bf16(f[2 * i])) | (static_cast<uint32_t>(f32_to_bf16(f[2 * i + 1])) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Sum of the S partials of the 8 elements of chunk c of `row`, in segment order, as bf16.
__device__ __forceinline__ uint4 partial_sum8(const float* __restrict__ part, int S, int M, int H, long long row, int c) {
    constexpr int G = 8;   // segments whose loads are in flight together (7 per projection: one round trip)
    float r[8];
    for (int q0 = 0; q0 < S; q0 += G) {
        float4 p[G][2];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float4* pp = reinterpret_cast<const float4*>(part + (static_cast<long long>(q0 + g) * M + row) * H) + 2 * c;
            p[g][0] = q0 + g < S ? __ldcg(pp) : make_float4(0.f, 0.f, 0.f, 0.f);
            p[g][1] = q0 + g < S ? __ldcg(pp + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float a[8] = {p[g][0].x, p[g][0].y, p[g][0].z, p[g][0].w, p[g][1].x, p[g][1].y, p[g][1].z, p[g][1].w};
            if (q0 + g == 0) {
#pragma unroll
                for (int e = 0; e < 8; ++e) r[e] = a[e];
            } else if (q0 + g < S) {
#pragma unroll
                for (int e = 0; e < 8; ++e) r[e] = __fadd_rn(r[e], a[e]);
            }
        }
    }
    return pack8(r);
}

constexpr int NORM_THREADS_MAX = 256;   // a row of up to NORM_CL * NORM_THREADS_MAX * NORM_MAXC chunks

template <bool PART>
__global__ void __launch_bounds__(NORM_THREADS_MAX) rmsnorm_kernel(uint16_t* __restrict__ x, const uint16_t* __restrict__ y_res,
                                                       const uint16_t* __restrict__ w, int H, float eps,
                                                       uint16_t* __restrict__ out, const int32_t* __restrict__ tokens,
                                                       const uint16_t* __restrict__ E, int V, unsigned* err,
                                                       const float* __restrict__ part, int S, int M, int cpc) {
    griddep_launch();
    griddep_wait();
    __shared__ float red[33];
    __shared__ float cta_ss;
    const int q = static_cast<int>(cluster_ctarank());
    const long long row = blockIdx.y;
    const int nch = H / 8, nt = blockDim.x;
    const int c0 = q * cpc, c1 = min(c0 + cpc, nch);
    uint4* xr = reinterpret_cast<uint4*>(x + row * H);
    const uint4* src = xr;
    if (tokens) {
        int t = tokens[row];
        if (t < 0 || t >= V) {
            if (q == 0 && threadIdx.x == 0) atomicOr(err, ERR_BAD_TOKEN);
            t = 0;
        }
        src = reinterpret_cast<const uint4*>(E + static_cast<long long>(t) * H);
    }
    const uint4* yr = y_res ? reinterpret_cast<const uint4*>(y_res + row * H) : nullptr;
    float v[NORM_MAXC][8];
    float ss = 0.f;
    bool first = true;
#pragma unroll
    for (int j = 0; j < NORM_MAXC; ++j) {
        const int c = c0 + threadIdx.x + j * nt;
        if (c < c1) {
            const uint4 raw = src[c];
            if (tokens) xr[c] = raw;
            unpack8(raw, v[j]);
            if (PART || yr) {
                float t[8];
                unpack8(PART ? partial_sum8(part, S, M, H, row, c) : yr[c], t);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[j][e] = bf16_to_f32(f32_to_bf16(__fadd_rn(v[j][e], t[e])));
                xr[c] = pack8(v[j]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                ss = first ? __fmul_rn(v[j][e], v[j][e]) : __fmaf_rn(v[j][e], v[j][e], ss);
                first = false;
            }
        }
    }
    ss = block_sum_fixed(ss, red);
    if (threadIdx.x == 0) cta_ss = ss;
    cluster_sync();
    const uint32_t a = smem_u32(&cta_ss);
    ss = ld_dsmem(mapa_shared(a, 0));
    for (int r = 1; r < NORM_CL; ++r) ss = __fadd_rn(ss, ld_dsmem(mapa_shared(a, r)));
    cluster_sync();   // no CTA leaves while a peer may still read its sum
    const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(H)), eps)));
    const uint4* wr = reinterpret_cast<const uint4*>(w);
    uint4* orow = reinterpret_cast<uint4*>(out + row * H);
#pragma unroll
    for (int j = 0; j < NORM_MAXC; ++j) {
        const int c = c0 + threadIdx.x + j * nt;
        if (c < c1) {
            float wf[8], o[8];
            unpack8(wr[c], wf);
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = __fmul_rn(__fmul_rn(v[j][e], inv), __fadd_rn(1.f, wf[e]));
            orow[c] = pack8(o);
        }
    }
}


// act = bf16(silu(g) * u), 8 elements per thread
__global__ void swiglu_kernel(const uint16_t* __restrict__ gu, int F, uint16_t* __restrict__ act) {
    griddep_launch();
    griddep_wait();
    const long long row = blockIdx.y;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= F / 8) return;
    float g[8], u[8], o[8];
    unpack8(reinterpret_cast<const uint4*>(gu + row * 2 * F)[c], g);
    unpack8(reinterpret_cast<const uint4*>(gu + row * 2 * F + F)[c], u);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = swiglu_f(g[e], u[e]);
    reinterpret_cast<uint4*>(act + row * F)[c] = pack8(o);
}

// Argmax, lowest index among the maxima.  Pass 1: CTA (chunk, row) takes ARGMAX_CHUNK
// consecutive logits (thread t: elements t*4 .. t*4+3 of every 1024-element stripe, in
// increasing order) and writes its (max, index); pass 2 reduces a row's chunk results.
// (value, -index) is a total order, so the result does not depend on the reduction order.
constexpr int ARGMAX_THREADS = 256;
constexpr int ARGMAX_CHUNK = 8192;

__device__ __forceinline__ void better(float& bv, int& bi, float v, int i) {
    if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
}
__device__ __forceinline__ void warp_best(float& bv, int& bi) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        better(bv, bi, ov, oi);
    }
}

__global__ void __launch_bounds__(ARGMAX_THREADS) argmax_chunk_kernel(const float* __restrict__ logits, int V,
                                                                       float2* __restrict__ part, int nchunk) {
    griddep_launch();
    griddep_wait();
    __shared__ float sv[ARGMAX_THREADS / 32];
    __shared__ int si[ARGMAX_THREADS / 32];
    const long long row = blockIdx.y;
    const int base = blockIdx.x * ARGMAX_CHUNK;
    const float* x = logits + row * V;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    const bool vec = (V % 4) == 0;
#pragma unroll
    for (int j = 0; j < ARGMAX_CHUNK / (ARGMAX_THREADS * 4); ++j) {
        const int i0 = base + j * ARGMAX_THREADS * 4 + threadIdx.x * 4;
        if (vec && i0 + 3 < V) {
            const float4 f = __ldg(reinterpret_cast<const float4*>(x + i0));
            better(bv, bi, f.x, i0);
            better(bv, bi, f.y, i0 + 1);
            better(bv, bi, f.z, i0 + 2);
            better(bv, bi, f.w, i0 + 3);
        } else {
            for (int e = 0; e < 4; ++e)
                if (i0 + e < V) better(bv, bi, x[i0 + e], i0 + e);
        }
    }
    warp_best(bv, bi);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
    __syncthreads();
    if (warp == 0) {
        bv = lane < ARGMAX_THREADS / 32 ? sv[lane] : -INFINITY;
        bi = lane < ARGMAX_THREADS / 32 ? si[lane] : 0x7fffffff;
        warp_best(bv, bi);
        if (lane == 0) part[row * nchunk + blockIdx.x] = make_float2(bv, __int_as_float(bi));
    }
}

// Pass 2 and the greedy acceptance of one sequence per CTA: warp j reduces the chunk results of
// row b*k + j into idx[b*k + j]; then n_accept[b] = the number of leading drafts tokens[b][j+1]
// equal to idx[b*k + j], over the sequence's own k_b <= k rows.  With ctx_len != null the CTA
// then commits those positions itself, as the commit kernel would with n_accept[b] + 1:
// ctx_len[b] += n_accept[b] + 1, n_commit[b] = n_accept[b] + 1 (always within [1, k_b]).
__global__ void argmax_accept_kernel(const float2* __restrict__ part, int nchunk, int k, int32_t* __restrict__ idx,
                                     const int32_t* __restrict__ tokens, const int32_t* __restrict__ k_seq,
                                     int32_t* __restrict__ n_accept, unsigned* err, int32_t* __restrict__ ctx_len,
                                     int32_t* __restrict__ n_commit) {
    griddep_launch();
    griddep_wait();
    __shared__ int pred[XV_KMAX];
    const int b = blockIdx.x, lane = threadIdx.x & 31;
    for (int j = threadIdx.x >> 5; j < k; j += blockDim.x >> 5) {   // warp per row
        const long long row = static_cast<long long>(b) * k + j;
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        // 16 partials per lane in flight before their compares (a row has one per LM-head tile,
        // 1187 at a vocabulary of 151936); (value, -index) is a total order, so the batching
        // leaves the result as it is
        constexpr int U = 16;
        for (int c0 = lane; c0 < nchunk; c0 += 32 * U) {
            float2 p[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * 32;
                p[u] = c < nchunk ? part[row * nchunk + c] : make_float2(-INFINITY, __int_as_float(0x7fffffff));
            }
#pragma unroll
            for (int u = 0; u < U; ++u) better(bv, bi, p[u].x, __float_as_int(p[u].y));
        }
        warp_best(bv, bi);
        if (lane == 0) {
            const int id = bi == 0x7fffffff ? 0 : bi;
            idx[row] = id;
            pred[j] = id;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int kb = k;
        if (k_seq) {
            kb = k_seq[b];
            if (kb < 1 || kb > k) {
                atomicOr(err, ERR_BAD_COUNT);
                kb = kb < 1 ? 1 : k;
            }
        }
        int n = 0;
        while (n < kb - 1 && pred[n] == tokens[static_cast<long long>(b) * k + n + 1]) ++n;
        n_accept[b] = n;
        if (ctx_len) {
            ctx_len[b] += n + 1;
            n_commit[b] = n + 1;
        }
    }
}

__global__ void commit_kernel(const int32_t* __restrict__ keep, int keep_bias, int B, int k,
                              const int32_t* __restrict__ k_seq, int32_t* __restrict__ ctx_len,
                              int32_t* __restrict__ n_commit, unsigned* err) {
    griddep_launch();
    griddep_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int kb = k;
    if (k_seq) {
        kb = k_seq[b];
        if (kb < 1 || kb > k) {
            atomicOr(err, ERR_BAD_COUNT);
            kb = kb < 1 ? 1 : k;
        }
    }
    int n = keep[b] + keep_bias;
    if (n < 1 || n > kb) {
        atomicOr(err, ERR_BAD_COUNT);
        n = n < 1 ? 1 : kb;
    }
    ctx_len[b] += n;
    n_commit[b] = n;
}

__global__ void zero_i32_kernel(int32_t* p, int n) {
    griddep_launch();
    griddep_wait();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) p[i] = 0;
}

}  // namespace


// Chunks per CTA of a row's cluster, and threads per CTA (one chunk each when that fits).
static int norm_cpc(int H) { return (H / 8 + NORM_CL - 1) / NORM_CL; }
static int norm_threads(int H) {
    const int cpc = norm_cpc(H);
    int t = ((cpc + NORM_MAXC - 1) / NORM_MAXC + 31) / 32 * 32;
    const int want = (cpc + 31) / 32 * 32;       // one chunk per thread when it fits
    if (want <= NORM_THREADS_MAX) t = want;
    return t < 32 ? 32 : t;
}
static xv_status norm_width(int H) {
    if (H < 8 || H % 8 || norm_threads(H) > NORM_THREADS_MAX)
        return fail(XV_ERR_UNSUPPORTED, "rmsnorm: width %d (a multiple of 8 up to %d)", H,
                    NORM_CL * NORM_THREADS_MAX * NORM_MAXC * 8);
    return XV_OK;
}

template <bool PART, typename... Args>
static void launch_norm(int M, int H, cudaStream_t s, Args&&... args) {
    launch_k_cluster(rmsnorm_kernel<PART>, dim3(NORM_CL, M), dim3(norm_threads(H)), 0, s, dim3(NORM_CL, 1, 1),
                     static_cast<Args&&>(args)..., norm_cpc(H));
}

xv_status rmsnorm_launch(const uint16_t* x, const uint16_t* w, int M, int H, float eps, uint16_t* y, cudaStream_t s) {
    if (xv_status st = norm_width(H)) return st;
    trace_pre(s);
    launch_norm<false>(M, H, s, const_cast<uint16_t*>(x), nullptr, w, H, eps, y, nullptr, nullptr, 0, nullptr, nullptr,
                       0, 0);
    return launched("rmsnorm_kernel", s, K_RMSNORM, 4ll * M * H + 2ll * H);
}

xv_status embed_rmsnorm_launch(const int32_t* tokens, int M, const uint16_t* E, int V, int H, const uint16_t* w,
                               float eps, uint16_t* x, uint16_t* xn, cudaStream_t s) {
    unsigned* err = device_error_word();
    if (!err) return fail(XV_ERR_CUDA, "embed: device error word unavailable");
    if (xv_status st = norm_width(H)) return st;
    trace_pre(s);
    launch_norm<false>(M, H, s, x, nullptr, w, H, eps, xn, tokens, E, V, err, nullptr, 0, 0);
    return launched("rmsnorm_kernel(embed)", s, K_EMBED, 6ll * M * H + 2ll * H + 4ll * M);
}

xv_status residual_rmsnorm_launch(uint16_t* x, const uint16_t* y, const uint16_t* w, int M, int H, float eps, uint16_t* xn,
                                  cudaStream_t s) {
    if (xv_status st = norm_width(H)) return st;
    trace_pre(s);
    launch_norm<false>(M, H, s, x, y, w, H, eps, xn, nullptr, nullptr, 0, nullptr, nullptr, 0, 0);
    return launched("rmsnorm_kernel(residual)", s, K_RMSNORM, 8ll * M * H + 2ll * H);
}

xv_status residual_rmsnorm_part_launch(uint16_t* x, const float* part, int S, const uint16_t* w, int M, int H, float eps,
                                       uint16_t* xn, cudaStream_t s) {
    if (S < 1 || S > 16) return fail(XV_ERR_ARG, "rmsnorm: %d partials outside [1, 16]", S);
    if (xv_status st = norm_width(H)) return st;
    trace_pre(s);
    launch_norm<true>(M, H, s, x, nullptr, w, H, eps, xn, nullptr, nullptr, 0, nullptr, part, S, M);
    return launched("rmsnorm_kernel(residual, partials)", s, K_RMSNORM, 4ll * S * M * H + 6ll * M * H + 2ll * H);
}

xv_status swiglu_launch(const uint16_t* gu, int M, int F, uint16_t* act, cudaStream_t s) {
    dim3 grid(ceil_div(F / 8, 256), M);
    trace_pre(s);
    launch_k(swiglu_kernel, grid, dim3(256), 0, s, gu, F, act);
    return launched("swiglu_kernel", s, K_SWIGLU, 6ll * M * F);
}

size_t argmax_workspace_size(int M, int V) { return static_cast<size_t>(M) * ceil_div(V, ARGMAX_CHUNK) * sizeof(float2); }

xv_status argmax_accept_launch(const float* logits, int B, int k, int V, int32_t* idx, void* ws,
                               const int32_t* tokens, const int32_t* k_seq, int32_t* n_accept, cudaStream_t s,
                               int32_t* ctx_len, int32_t* n_commit) {
    unsigned* err = device_error_word();
    if (!err) return fail(XV_ERR_CUDA, "argmax: device error word unavailable");
    if (k < 1 || k > XV_KMAX) return fail(XV_ERR_ARG, "argmax: k = %d outside [1, %d]", k, XV_KMAX);
    const int M = B * k;
    const int nchunk = ceil_div(V, ARGMAX_CHUNK);
    float2* part = static_cast<float2*>(ws);
    trace_pre(s);
    launch_k(argmax_chunk_kernel, dim3(nchunk, M), dim3(ARGMAX_THREADS), 0, s, logits, V, part, nchunk);
    if (xv_status st = launched("argmax_chunk_kernel", s, K_ARGMAX, 4ll * M * V)) return st;
    trace_pre(s);
    launch_k(argmax_accept_kernel, dim3(B), dim3(32 * (k < 32 ? k : 32)), 0, s, part, nchunk, k, idx, tokens, k_seq,
             n_accept, err, ctx_len, n_commit);
    return launched("argmax_accept_kernel", s, K_ACCEPT, 8ll * M * nchunk + 8ll * M + 4ll * B);
}

xv_status accept_from_parts_launch(const float2* part, int nchunk, int B, int k, int32_t* idx, const int32_t* tokens,
                                   const int32_t* k_seq, int32_t* n_accept, cudaStream_t s, int32_t* ctx_len,
                                   int32_t* n_commit) {
    unsigned* err = device_error_word();
    if (!err) return fail(XV_ERR_CUDA, "argmax: device error word unavailable");
    if (k < 1 || k > XV_KMAX) return fail(XV_ERR_ARG, "argmax: k = %d outside [1, %d]", k, XV_KMAX);
    const int M = B * k;
    trace_pre(s);
    launch_k(argmax_accept_kernel, dim3(B), dim3(32 * (k < 32 ? k : 32)), 0, s, part, nchunk, k, idx, tokens, k_seq,
             n_accept, err, ctx_len, n_commit);
    return launched("argmax_accept_kernel", s, K_ACCEPT, 8ll * M * nchunk + 8ll * M + 4ll * B);
}

xv_status commit_launch(const int32_t* keep, int keep_bias, int B, int k, const int32_t* k_seq, int32_t* ctx_len,
                        int32_t* n_commit,
                        cudaStream_t s) {
    unsigned* err = device_error_word();
    if (!err) return fail(XV_ERR_CUDA, "commit: device error word unavailable");
    trace_pre(s);
    launch_k(commit_kernel, dim3(ceil_div(B, 128)), dim3(128), 0, s, keep, keep_bias, B, k, k_seq, ctx_len, n_commit, err);
    return launched("commit_kernel", s, K_COMMIT, 16ll * B);
}

xv_status zero_i32_launch(int32_t* p, int n, cudaStream_t s) {
    trace_pre(s);
    launch_k(zero_i32_kernel, dim3(ceil_div(n, 256)), dim3(256), 0, s, p, n);
    return launched("zero_i32_kernel", s, K_ZERO, 4ll * n);
}

}  // namespace xv
