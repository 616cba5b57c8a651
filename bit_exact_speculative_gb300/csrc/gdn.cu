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
// Tiling: a CTA owns (sequence b, head h, 32 state rows) with 64 threads; a
// row is split over 4 consecutive lanes (lane g holds float4 chunks g, g+4,
// g+8, ... of the row) and each thread carries 2 rows, so the staged k and q
// slices are loaded once for both and the two rows' dependency chains run
// side by side.  Row dot products: two packed f32x2 accumulators (even and
// odd pairs), a fixed sum of their four lanes, then an xor-shuffle tree over
// the row's 4 lanes (offsets 1, 2): every lane ends with the same bits.  The
// state lives in registers across all replay and speculative steps; it is read
// once (its loads issued before the step inputs are staged) and, after a
// replay, written once.  All step inputs are staged in one round of
// independent loads, then normalised from shared memory.
#include "xv_internal.h"
#include "xv_ptx.cuh"

namespace xv {

namespace {
constexpr int LPR = 4;                          // lanes per state row
constexpr int RPT = 2;                          // state rows per thread
constexpr int WARPS = 2;
constexpr int ROWS_PER_WARP = 32 / LPR * RPT;   // 16
constexpr int ROWS_PER_CTA = ROWS_PER_WARP * WARPS;
constexpr int THREADS = 32 * WARPS;

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

// Per-step inputs staged in shared memory: q and k (fp32, normalised in place), this
// CTA's v entries, beta and gate.
template <int DK>
struct StepSmem {
    float q[DK];
    float k[DK];
    float v[ROWS_PER_CTA];
    float beta, gate;
    float pad[2];
};

// Source of staged slot t for sequence b: slots [0, max_commit) hold pending rows 0.., slots
// [max_commit, max_commit + k) the draft rows.  All are staged whatever n_commit[b] is, so
// staging never waits for it; only the first n_commit[b] pending slots are replayed.
__device__ __forceinline__ const GdnStepsDev& step_src(const GdnArgs& A, int b, int t, long long* row) {
    if (t < A.max_commit) {
        *row = static_cast<long long>(b) * A.pend.rows_per_seq + t;
        return A.pend;
    }
    *row = static_cast<long long>(b) * A.draft.rows_per_seq + (t - A.max_commit);
    return A.draft;
}

__device__ __forceinline__ void store8(float* dst, const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float4 a = make_float4(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u),
                           __uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xFFFF0000u));
    float4 b = make_float4(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xFFFF0000u),
                           __uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xFFFF0000u));
    *reinterpret_cast<float4*>(dst) = a;
    *reinterpret_cast<float4*>(dst + 4) = b;
}

// Every step's raw inputs, converted to fp32 in shared memory.  q, k and this CTA's v slab
// go as 16-byte chunks, STAGE_BATCH per thread issued back to back before any is used (one
// round trip to memory for a verify's worth of steps); beta and gate are scalars.
constexpr int STAGE_BATCH = 10;

template <int DK>
__device__ __forceinline__ const uint16_t* chunk_addr(const GdnArgs& A, int b, int h, int row0, int idx) {
    constexpr int CH = DK / 8, VCH = ROWS_PER_CTA / 8, PER = 2 * CH + VCH;
    const int t = idx / PER, j = idx - t * PER;
    long long row;
    const GdnStepsDev& src = step_src(A, b, t, &row);
    const long long base = row * src.qkv_stride;
    if (j < CH) return src.q + base + static_cast<long long>(h) * DK + 8 * j;
    if (j < 2 * CH) return src.k + base + static_cast<long long>(h) * DK + 8 * (j - CH);
    return src.v + base + static_cast<long long>(h) * A.dv + row0 + 8 * (j - 2 * CH);
}

// Shared-memory destination of chunk idx (q, k and v of a slot are contiguous floats).
template <int DK>
__device__ __forceinline__ float* chunk_dst(StepSmem<DK>* steps, int idx) {
    constexpr int PER = 2 * (DK / 8) + ROWS_PER_CTA / 8;
    const int t = idx / PER, j = idx - t * PER;
    return reinterpret_cast<float*>(&steps[t]) + 8 * j;
}

// One round of staging for thread slot `base`: issue() starts the loads (a beta/gate scalar
// and up to STAGE_BATCH chunks) into registers, commit() converts and stores them.
template <int DK>
struct StageRound {
    uint4 v[STAGE_BATCH];
    uint16_t bg;
    int base;

    __device__ __forceinline__ void issue(StepSmem<DK>* steps, const GdnArgs& A, int b, int h, int row0, int total,
                                          int base_) {
        constexpr int PER = 2 * (DK / 8) + ROWS_PER_CTA / 8;
        base = base_;
        const int n = total * PER;
        if (base < 2 * total) {
            long long row;
            const GdnStepsDev& src = step_src(A, b, base >> 1, &row);
            bg = (base & 1) ? src.gate[row * src.gate_stride + h] : src.beta[row * src.gate_stride + h];
        }
#pragma unroll
        for (int u = 0; u < STAGE_BATCH; ++u) {
            const int idx = base + u * THREADS;
            if (idx < n) v[u] = *reinterpret_cast<const uint4*>(chunk_addr<DK>(A, b, h, row0, idx));
        }
    }
    __device__ __forceinline__ void commit(StepSmem<DK>* steps, int total) {
        constexpr int PER = 2 * (DK / 8) + ROWS_PER_CTA / 8;
        const int n = total * PER;
#pragma unroll
        for (int u = 0; u < STAGE_BATCH; ++u)
            if (base + u * THREADS < n) store8(chunk_dst<DK>(steps, base + u * THREADS), v[u]);
        if (base < 2 * total) {
            if (base & 1) steps[base >> 1].gate = bf16_to_f32(bg);
            else steps[base >> 1].beta = bf16_to_f32(bg);
        }
    }
};

// Per-head L2 normalisation of q and k in shared memory: x / sqrt(sum x^2 + 1e-6).
// Vector w (slot w/2, q for even w, k for odd) belongs to the thread pair (2w', 2w'+1) with
// w' = w mod (THREADS/2); thread p of the pair sums elements p*DK/2 .. (p+1)*DK/2 - 1 in four
// interleaved chains (e mod 4), adds them as (c0 + c1) + (c2 + c3), the pair adds its two
// halves (one shuffle), and each thread scales its half.
template <int DK>
__device__ __forceinline__ void normalise_all(StepSmem<DK>* steps, int total) {
    constexpr int HALF = DK / 2;
    const int p = threadIdx.x & 1;
    for (int w0 = 0; w0 < 2 * total; w0 += THREADS / 2) {   // same trip count for every thread
        const int w = w0 + (threadIdx.x >> 1);
        const bool act = w < 2 * total;
        float* x = (w & 1) ? steps[act ? w >> 1 : 0].k : steps[act ? w >> 1 : 0].q;
        float* h = x + p * HALF;
        float c[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) c[q4] = __fmul_rn(h[q4], h[q4]);
#pragma unroll
        for (int e = 4; e < HALF; e += 4) {
            const float4 v = *reinterpret_cast<const float4*>(h + e);
            c[0] = __fmaf_rn(v.x, v.x, c[0]);
            c[1] = __fmaf_rn(v.y, v.y, c[1]);
            c[2] = __fmaf_rn(v.z, v.z, c[2]);
            c[3] = __fmaf_rn(v.w, v.w, c[3]);
        }
        float ss = __fadd_rn(__fadd_rn(c[0], c[1]), __fadd_rn(c[2], c[3]));
        ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 1));
        const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(ss, 1e-6f)));
        if (!act) continue;
#pragma unroll
        for (int e = 0; e < HALF; e += 4) {
            float4 v = *reinterpret_cast<const float4*>(h + e);
            v.x = __fmul_rn(v.x, inv);
            v.y = __fmul_rn(v.y, inv);
            v.z = __fmul_rn(v.z, inv);
            v.w = __fmul_rn(v.w, inv);
            *reinterpret_cast<float4*>(h + e) = v;
        }
    }
}

// Sum over the LPR lanes of a row (xor 1, 2): every lane gets the same bits.
__device__ __forceinline__ float row_sum(float v) {
    v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1));
    v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 2));
    return v;
}

// Dot product of a lane's row slice with a staged vector: packed pair j = elements
// (2j, 2j+1) of the slice; two packed accumulators over even and odd pairs, then
// (A.x + A.y) + (B.x + B.y), then the lanes of the row.
template <int NP>
__device__ __forceinline__ float slice_dot(const float2 (&s)[NP], const float2 (&v)[NP]) {
    float2 a = __fmul2_rn(s[0], v[0]);
    float2 c = __fmul2_rn(s[1], v[1]);
#pragma unroll
    for (int j = 2; j < NP; j += 2) {
        a = __ffma2_rn(s[j], v[j], a);
        c = __ffma2_rn(s[j + 1], v[j + 1], c);
    }
    return row_sum(__fadd_rn(__fadd_rn(a.x, a.y), __fadd_rn(c.x, c.y)));
}

// Lane g of a row holds the 16-byte chunks g, g + LPR, g + 2 LPR, ... of the row.
template <int DK>
__device__ __forceinline__ void load_slice(float2 (&d)[DK / (2 * LPR)], const float* src, int g) {
#pragma unroll
    for (int u = 0; u < DK / (4 * LPR); ++u) {
        const float4 t = *reinterpret_cast<const float4*>(src + 4 * (g + LPR * u));
        d[2 * u] = make_float2(t.x, t.y);
        d[2 * u + 1] = make_float2(t.z, t.w);
    }
}

// The step function shared by decode, replay and verify, for this thread's RPT rows:
//   S <- a S;  r = S k;  u = beta (v - r);  S <- S + u k^T;  o = S q
// each operation rounded once (packed f32x2 lanes are independent IEEE fp32 ops).
template <int DK>
__device__ __forceinline__ void gdn_step(float2 (&s)[RPT][DK / (2 * LPR)], const StepSmem<DK>& in, int g,
                                         const int (&r)[RPT], bool want_o, float (&o)[RPT]) {
    constexpr int NP = DK / (2 * LPR);
    float2 kk[NP];
    load_slice<DK>(kk, in.k, g);
    const float2 a2 = make_float2(in.gate, in.gate);
#pragma unroll
    for (int x = 0; x < RPT; ++x) {
#pragma unroll
        for (int j = 0; j < NP; ++j) s[x][j] = __fmul2_rn(a2, s[x][j]);
    }
    float rr[RPT];
#pragma unroll
    for (int x = 0; x < RPT; ++x) rr[x] = slice_dot<NP>(s[x], kk);
#pragma unroll
    for (int x = 0; x < RPT; ++x) {
        const float uu = __fmul_rn(in.beta, __fsub_rn(in.v[r[x]], rr[x]));
        const float2 u2 = make_float2(uu, uu);
#pragma unroll
        for (int j = 0; j < NP; ++j) s[x][j] = __ffma2_rn(u2, kk[j], s[x][j]);
    }
    if (!want_o) return;
    float2 qq[NP];
    load_slice<DK>(qq, in.q, g);
#pragma unroll
    for (int x = 0; x < RPT; ++x) o[x] = slice_dot<NP>(s[x], qq);
}

template <int DK>
__global__ void __launch_bounds__(THREADS, 8) gdn_kernel(GdnArgs A) {
    griddep_launch();
    griddep_wait();
    constexpr int NP = DK / (2 * LPR);
    extern __shared__ __align__(16) uint8_t smem_raw[];
    StepSmem<DK>* steps = reinterpret_cast<StepSmem<DK>*>(smem_raw);

    const int slab = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane % LPR;
    int r[RPT];                                           // rows within the slab
#pragma unroll
    for (int x = 0; x < RPT; ++x) r[x] = warp * ROWS_PER_WARP + x * (32 / LPR) + lane / LPR;
    const int row0 = slab * ROWS_PER_CTA;

    // Loads in flight together: the first staging round (the step inputs gate the start of
    // the recurrence), then the state rows, which arrive while the inputs are normalised.
    const int total = A.max_commit + A.k;
    constexpr int PER = 2 * (DK / 8) + ROWS_PER_CTA / 8;
    const int n_items = total * PER > 2 * total ? total * PER : 2 * total;
    StageRound<DK> first;
    first.issue(steps, A, b, h, row0, total, threadIdx.x);
    float2 s[RPT][NP];
#pragma unroll
    for (int x = 0; x < RPT; ++x)
        load_slice<DK>(s[x], A.state + ((static_cast<size_t>(b) * A.H + h) * A.dv + row0 + r[x]) * DK, g);
    first.commit(steps, total);
    for (int base = threadIdx.x + THREADS * STAGE_BATCH; base < n_items; base += THREADS * STAGE_BATCH) {
        StageRound<DK> more;   // long verify blocks only: further rounds
        more.issue(steps, A, b, h, row0, total, base);
        more.commit(steps, total);
    }
    int nc = A.n_commit ? A.n_commit[b] : A.n_fixed;
    if (nc < 0 || nc > A.max_commit) {
        if (threadIdx.x == 0) atomicOr(A.err, ERR_BAD_COUNT);
        nc = nc < 0 ? 0 : A.max_commit;
    }
    __syncthreads();
    if (A.l2) normalise_all<DK>(steps, total);
    __syncthreads();

    float o[RPT];
    // replay the committed steps (these change the stored state)
    for (int t = 0; t < nc; ++t) {
        gdn_step<DK>(s, steps[t], g, r, A.emit_replay != 0, o);
        if (A.emit_replay && g == 0) {
#pragma unroll
            for (int x = 0; x < RPT; ++x)
                A.o[(static_cast<long long>(b) * nc + t) * A.o_stride + static_cast<long long>(h) * A.dv + row0 + r[x]] =
                    f32_to_bf16(o[x]);
        }
    }
    if (nc > 0) {
#pragma unroll
        for (int x = 0; x < RPT; ++x) {
            float* srow = A.state + ((static_cast<size_t>(b) * A.H + h) * A.dv + row0 + r[x]) * DK;
#pragma unroll
            for (int u = 0; u < NP / 2; ++u)
                *reinterpret_cast<float4*>(srow + 4 * (g + LPR * u)) =
                    make_float4(s[x][2 * u].x, s[x][2 * u].y, s[x][2 * u + 1].x, s[x][2 * u + 1].y);
        }
    }
    // speculative steps: outputs only, the state in memory stays committed
    for (int t = 0; t < A.k; ++t) {
        gdn_step<DK>(s, steps[A.max_commit + t], g, r, true, o);
        if (g == 0) {
#pragma unroll
            for (int x = 0; x < RPT; ++x)
                A.o[(static_cast<long long>(b) * A.k + t) * A.o_stride + static_cast<long long>(h) * A.dv + row0 + r[x]] =
                    f32_to_bf16(o[x]);
        }
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
    dim3 grid(dv / ROWS_PER_CTA, H, B);   // dv is a multiple of ROWS_PER_CTA (checked)
    trace_pre(s);
    static bool carve[2] = {false, false};
    if (!carve[dk == 128]) {
        // as much shared memory as possible for the carveout: 8 CTAs per SM need ~150 KB
        if (dk == 128) cudaFuncSetAttribute(gdn_kernel<128>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        else cudaFuncSetAttribute(gdn_kernel<64>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        carve[dk == 128] = true;
    }
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
