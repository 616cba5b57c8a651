// Gated delta rule: decode step and verify with deferred commit, ONE kernel.
//
// "Follow-up to my earlier post on Qwen3.8-27B decode speed" (r/LocalLLaMA
// post): verify must run the GDN recurrence through the decode kernel; the
// faulty verify kernel tiled the state in another order and kept beta in
// fp32.  Here there is only one kernel and one step function: decode is the
// kernel replaying one step with output, verify replays the pending steps and
// then runs k speculative steps.  Tiling, thread-to-element mapping,
// reduction trees and rounding are therefore identical by construction.
//
// Recurrence per head (S is [dv][dk] fp32, rows independent):
//     S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T ,  o_t = S_t q_t
// computed in the algebraically equal error-correcting order, every op
// rounded once (explicit _rn intrinsics, so no contraction can differ):
//     S <- a S;  r = S k;  u = b (v - r);  S <- S + u k^T;  o = S q.
//
// Tiling: a CTA owns (sequence b, head h, 16 state rows); each row is split
// over 8 consecutive lanes, lane g holding float4 chunks g, g+8, g+16, ... of
// the row (coalesced 128-byte segments per 8 lanes).  Row dot products are a
// fixed two-chain sum over the lane's elements, then an xor-shuffle tree over
// the 8 lanes (offsets 1, 2, 4): every lane ends with the same bits.  The
// state lives in registers across all replay and speculative steps; it is
// read once and (after a replay) written once.
#include "xv_internal.h"
#include "xv_ptx.cuh"

namespace xv {

namespace {
constexpr int ROWS_PER_CTA = 16;
constexpr int THREADS = 128;        // 4 warps x 4 rows x 8 lanes

struct GdnArgs {
    float* state;
    GdnStepsDev pend;
    const int32_t* n_commit;
    int n_fixed;
    int max_commit;
    int emit_replay;
    GdnStepsDev draft;
    int k;
    uint16_t* o;
    long long o_stride;
    int H, dv, l2;
    unsigned* err;
};

// Per-step inputs staged in shared memory: normalised q and k (fp32), this
// CTA's 16 v entries, beta and gate.
template <int DK>
struct StepSmem {
    float q[DK];
    float k[DK];
    float v[ROWS_PER_CTA];
    float beta, gate;
    float pad[2];
};

// Loads one step's inputs for (row index `row`, head h) and normalises q, k
// with a fixed reduction (one warp per step: lane j sums elements j, j+32,
// ... in order, then an xor tree over 32 lanes).
template <int DK>
__device__ __forceinline__ void stage_step(StepSmem<DK>& dst, const GdnStepsDev& src, long long row, int h, int dv,
                                           int row0, int l2, int lane) {
    const uint16_t* q = src.q + row * src.qkv_stride + static_cast<long long>(h) * DK;
    const uint16_t* k = src.k + row * src.qkv_stride + static_cast<long long>(h) * DK;
    const uint16_t* v = src.v + row * src.qkv_stride + static_cast<long long>(h) * dv + row0;
    constexpr int PER = DK / 32;
    float qv[PER], kv[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        qv[e] = bf16_to_f32(q[lane + 32 * e]);
        kv[e] = bf16_to_f32(k[lane + 32 * e]);
    }
    if (l2) {
        float sq = __fmul_rn(qv[0], qv[0]), sk = __fmul_rn(kv[0], kv[0]);
#pragma unroll
        for (int e = 1; e < PER; ++e) {
            sq = __fmaf_rn(qv[e], qv[e], sq);
            sk = __fmaf_rn(kv[e], kv[e], sk);
        }
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, off));
            sk = __fadd_rn(sk, __shfl_xor_sync(0xffffffffu, sk, off));
        }
        const float iq = __frcp_rn(__fsqrt_rn(__fadd_rn(sq, 1e-6f)));
        const float ik = __frcp_rn(__fsqrt_rn(__fadd_rn(sk, 1e-6f)));
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            qv[e] = __fmul_rn(qv[e], iq);
            kv[e] = __fmul_rn(kv[e], ik);
        }
    }
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        dst.q[lane + 32 * e] = qv[e];
        dst.k[lane + 32 * e] = kv[e];
    }
    if (lane < ROWS_PER_CTA) dst.v[lane] = bf16_to_f32(v[lane]);
    if (lane == 0) {
        dst.beta = bf16_to_f32(src.beta[row * src.gate_stride + h]);
        dst.gate = bf16_to_f32(src.gate[row * src.gate_stride + h]);
    }
}

// The step function shared by decode, replay and verify.  s[] holds this
// lane's EPL state entries of row `r`; kk/qq point at the staged step.
template <int DK>
__device__ __forceinline__ float gdn_step(float (&s)[DK / 8], const StepSmem<DK>& in, int g, int r, bool want_o) {
    constexpr int EPL = DK / 8;
    float kk[EPL];
#pragma unroll
    for (int u = 0; u < EPL / 4; ++u) {
        const float4 t = *reinterpret_cast<const float4*>(&in.k[4 * (g + 8 * u)]);
        kk[4 * u] = t.x; kk[4 * u + 1] = t.y; kk[4 * u + 2] = t.z; kk[4 * u + 3] = t.w;
    }
    const float a = in.gate, b = in.beta;
#pragma unroll
    for (int e = 0; e < EPL; ++e) s[e] = __fmul_rn(a, s[e]);
    float r0 = __fmul_rn(s[0], kk[0]), r1 = __fmul_rn(s[1], kk[1]);
#pragma unroll
    for (int e = 2; e < EPL; e += 2) {
        r0 = __fmaf_rn(s[e], kk[e], r0);
        r1 = __fmaf_rn(s[e + 1], kk[e + 1], r1);
    }
    float rr = __fadd_rn(r0, r1);
    rr = __fadd_rn(rr, __shfl_xor_sync(0xffffffffu, rr, 1));
    rr = __fadd_rn(rr, __shfl_xor_sync(0xffffffffu, rr, 2));
    rr = __fadd_rn(rr, __shfl_xor_sync(0xffffffffu, rr, 4));
    const float uu = __fmul_rn(b, __fsub_rn(in.v[r], rr));
#pragma unroll
    for (int e = 0; e < EPL; ++e) s[e] = __fmaf_rn(uu, kk[e], s[e]);
    if (!want_o) return 0.f;
    float qq[EPL];
#pragma unroll
    for (int u = 0; u < EPL / 4; ++u) {
        const float4 t = *reinterpret_cast<const float4*>(&in.q[4 * (g + 8 * u)]);
        qq[4 * u] = t.x; qq[4 * u + 1] = t.y; qq[4 * u + 2] = t.z; qq[4 * u + 3] = t.w;
    }
    float o0 = __fmul_rn(s[0], qq[0]), o1 = __fmul_rn(s[1], qq[1]);
#pragma unroll
    for (int e = 2; e < EPL; e += 2) {
        o0 = __fmaf_rn(s[e], qq[e], o0);
        o1 = __fmaf_rn(s[e + 1], qq[e + 1], o1);
    }
    float oo = __fadd_rn(o0, o1);
    oo = __fadd_rn(oo, __shfl_xor_sync(0xffffffffu, oo, 1));
    oo = __fadd_rn(oo, __shfl_xor_sync(0xffffffffu, oo, 2));
    oo = __fadd_rn(oo, __shfl_xor_sync(0xffffffffu, oo, 4));
    return oo;
}

template <int DK>
__global__ void __launch_bounds__(THREADS) gdn_kernel(GdnArgs A) {
    griddep_launch();
    griddep_wait();
    constexpr int EPL = DK / 8;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    StepSmem<DK>* steps = reinterpret_cast<StepSmem<DK>*>(smem_raw);

    const int slab = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = warp * 4 + (lane >> 3);        // row within the slab
    const int g = lane & 7;                      // lane within the row group
    const int row0 = slab * ROWS_PER_CTA;
    const int i = row0 + r;                      // state row (v index)

    int nc = A.n_commit ? A.n_commit[b] : A.n_fixed;
    if (nc < 0 || nc > A.max_commit) {
        if (threadIdx.x == 0) atomicOr(A.err, ERR_BAD_COUNT);
        nc = nc < 0 ? 0 : A.max_commit;
    }
    const int total = nc + A.k;

    // stage every step's inputs (warp w takes steps w, w+4, ...)
    for (int t = warp; t < total; t += THREADS / 32) {
        if (t < nc) stage_step<DK>(steps[t], A.pend, static_cast<long long>(b) * A.pend.rows_per_seq + t, h, A.dv, row0, A.l2, lane);
        else stage_step<DK>(steps[t], A.draft, static_cast<long long>(b) * A.draft.rows_per_seq + (t - nc), h, A.dv, row0, A.l2, lane);
    }
    __syncthreads();

    float* srow = A.state + ((static_cast<size_t>(b) * A.H + h) * A.dv + i) * DK;
    float s[EPL];
#pragma unroll
    for (int u = 0; u < EPL / 4; ++u) {
        const float4 t = *reinterpret_cast<const float4*>(srow + 4 * (g + 8 * u));
        s[4 * u] = t.x; s[4 * u + 1] = t.y; s[4 * u + 2] = t.z; s[4 * u + 3] = t.w;
    }

    // replay the committed steps (these change the stored state)
    for (int t = 0; t < nc; ++t) {
        const float o = gdn_step<DK>(s, steps[t], g, r, A.emit_replay != 0);
        if (A.emit_replay && g == 0)
            A.o[(static_cast<long long>(b) * nc + t) * A.o_stride + static_cast<long long>(h) * A.dv + i] = f32_to_bf16(o);
    }
    if (nc > 0) {
#pragma unroll
        for (int u = 0; u < EPL / 4; ++u)
            *reinterpret_cast<float4*>(srow + 4 * (g + 8 * u)) = make_float4(s[4 * u], s[4 * u + 1], s[4 * u + 2], s[4 * u + 3]);
    }
    // speculative steps: outputs only, the state in memory stays committed
    for (int t = 0; t < A.k; ++t) {
        const float o = gdn_step<DK>(s, steps[nc + t], g, r, true);
        if (g == 0)
            A.o[(static_cast<long long>(b) * A.k + t) * A.o_stride + static_cast<long long>(h) * A.dv + i] = f32_to_bf16(o);
    }
}

}  // namespace

xv_status gdn_launch(float* state, const GdnStepsDev& pending, const int32_t* n_commit, int n_fixed, int max_commit,
                     bool emit_replay, const GdnStepsDev& draft, int k, uint16_t* o, long long o_stride, int B, int H,
                     int dk, int dv, int qk_l2norm, cudaStream_t s) {
    unsigned* err = device_error_word();
    if (!err) return fail(XV_ERR_CUDA, "gdn: device error word unavailable");
    GdnArgs a{state, pending, n_commit, n_fixed, max_commit, emit_replay ? 1 : 0, draft, k, o, o_stride, H, dv,
              qk_l2norm ? 1 : 0, err};
    const int max_steps = max_commit + k;
    dim3 grid(dv / ROWS_PER_CTA, H, B);
    trace_pre(s);
    if (dk == 128) {
        const size_t sm = sizeof(StepSmem<128>) * (max_steps > 0 ? max_steps : 1);
        launch_k(gdn_kernel<128>, dim3(grid), dim3(THREADS), sm, s, a);
    } else {
        const size_t sm = sizeof(StepSmem<64>) * (max_steps > 0 ? max_steps : 1);
        launch_k(gdn_kernel<64>, dim3(grid), dim3(THREADS), sm, s, a);
    }
    // algorithmic bytes with every sequence replaying max_commit steps: the state
    // read (and written back after a replay), the step inputs, the outputs
    const long long state_bytes = 4ll * B * H * dv * dk;
    const long long per_step = 2ll * B * H * (2 * dk + dv + 2);
    const long long outs = 2ll * B * H * dv * (k + (emit_replay ? max_commit : 0));
    const long long bytes = state_bytes * (max_commit > 0 ? 2 : 1) + per_step * (max_commit + k) + outs;
    return launched("gdn_kernel", s, K_GDN, bytes);
}

}  // namespace xv
