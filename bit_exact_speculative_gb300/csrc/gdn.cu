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
// Grouped heads: with fewer q/k heads than v heads, v head h reads q/k head
// h / qk_group (the state and v, beta, gate are per v head).
//
// Arithmetic of a row (fixed): a row is split over 4 consecutive lanes (lane g
// holds float4 chunks g, g+4, g+8, ... of the row).  Row dot products: two
// packed f32x2 accumulators (even and odd pairs), a fixed sum of their four
// lanes, then an xor-shuffle tree over the row's 4 lanes (offsets 1, 2): every
// lane ends with the same bits.  Nothing a row computes depends on which
// thread, warp or CTA holds it.
//
// Tiling (free, chosen per launch): a thread holds RPT rows (rows lane/4,
// lane/4 + 8, ... of its warp's 8 * RPT), a CTA WARPS warps.  Every step reads
// the whole k and q vectors from shared memory into each row's lanes; with
// one row per thread that read (1 KB per row per step) is the bound, so wide
// launches hold 4 rows per thread and read each slice once for the four.  The
// state lives in registers across all replay and speculative steps; it is
// read once (plain loads issued first) and, after a replay, written once.
// The step inputs (per step: q and k of the head, this CTA's slice of v, beta
// and gate) are staged by 16-byte asynchronous copies spread over the CTA's
// threads and issued together with the state loads, so the whole verify's
// inputs arrive in a single round trip without holding registers; q and k are
// then L2-normalised by 4 threads per vector into fp32.
#include "xv_internal.h"
#include "xv_ptx.cuh"

namespace xv {

namespace {
constexpr int LPR = 4;                          // lanes per state row
constexpr int NORM_LANES = 4;                   // threads per q or k vector in the normalisation

// A launch shape: RPT state rows per thread, WARPS warps per CTA, at least MIN_BLOCKS CTAs per SM.
template <int RPT_, int WARPS_, int MIN_BLOCKS_>
struct Tiling {
    static constexpr int RPT = RPT_;
    static constexpr int WARPS = WARPS_;
    static constexpr int MIN_BLOCKS = MIN_BLOCKS_;
    static constexpr int ROWS_PER_WARP = 32 / LPR * RPT;
    static constexpr int ROWS = ROWS_PER_WARP * WARPS;   // state rows per CTA
    static constexpr int THREADS = 32 * WARPS;
};
using NarrowTiling = Tiling<1, 4, 4>;   // 32 rows, 128 threads: few CTAs (latency-bound launches)
using WideTiling = Tiling<4, 1, 8>;     // 32 rows, 32 threads: many CTAs (shared-memory reads amortised)
static_assert(NarrowTiling::ROWS == WideTiling::ROWS, "both tilings cut a head into the same slabs");
constexpr int SLAB = NarrowTiling::ROWS;

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
    int H, dv, l2, qk_group;
    unsigned* err;
};

// Per-step inputs staged in shared memory: q and k (fp32, normalised), this CTA's v entries,
// beta and gate; and the raw bf16 q, k, v the asynchronous copies land in.
template <int DK>
struct StepSmem {
    float q[DK];
    float k[DK];
    float v[SLAB];
    float beta, gate;
    float pad[2];
};
template <int DK>
struct RawStep {
    uint16_t q[DK];
    uint16_t k[DK];
    uint16_t v[SLAB];
};
template <int DK>
constexpr size_t step_smem_bytes() { return sizeof(StepSmem<DK>) + sizeof(RawStep<DK>); }

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

__device__ __forceinline__ float bf16f(uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); }

// Issues the asynchronous copies of every staged step's raw q, k (of q/k head hk) and this
// CTA's v slice (rows row0.., of v head h): 16-byte pieces spread over the CTA's threads.
template <int DK, int THREADS>
__device__ __forceinline__ void stage_raw(RawStep<DK>* raw, const GdnArgs& A, int b, int h, int hk, int row0,
                                          int total) {
    constexpr int QC = DK / 8, VC = SLAB / 8, PER_STEP = 2 * QC + VC;
    for (int idx = threadIdx.x; idx < total * PER_STEP; idx += THREADS) {
        const int t = idx / PER_STEP, c = idx % PER_STEP;
        long long row;
        const GdnStepsDev& src = step_src(A, b, t, &row);
        const uint16_t* g;
        uint16_t* d;
        if (c < QC) {
            g = src.q + row * src.qkv_stride + static_cast<long long>(hk) * DK + 8 * c;
            d = raw[t].q + 8 * c;
        } else if (c < 2 * QC) {
            g = src.k + row * src.qkv_stride + static_cast<long long>(hk) * DK + 8 * (c - QC);
            d = raw[t].k + 8 * (c - QC);
        } else {
            g = src.v + row * src.qkv_stride + static_cast<long long>(h) * A.dv + row0 + 8 * (c - 2 * QC);
            d = raw[t].v + 8 * (c - 2 * QC);
        }
        cp_async16(d, g);
    }
}

// Vector w of the staged steps (step w / 2; q for even w, k for odd) from its raw bf16 copy to
// fp32, L2-normalised when l2 (x / sqrt(sum x^2 + 1e-6)): thread j of the vector's group of
// NORM_LANES takes elements [j DK/4, (j+1) DK/4), sums their squares in four interleaved chains
// (e mod 4) added as (c0 + c1) + (c2 + c3), the group adds its partials by an xor tree (1, 2),
// and every thread scales its own elements.
template <int DK, int THREADS>
__device__ __forceinline__ void normalise_all(StepSmem<DK>* steps, const RawStep<DK>* raw, int total, bool l2) {
    constexpr int PART = DK / NORM_LANES;
    const int jl = threadIdx.x % NORM_LANES;
    for (int w0 = 0; w0 < 2 * total; w0 += THREADS / NORM_LANES) {   // same trip count for every thread
        const int w = w0 + static_cast<int>(threadIdx.x) / NORM_LANES;
        const bool act = w < 2 * total;
        const int t = act ? w >> 1 : 0;
        const uint16_t* x = ((w & 1) ? raw[t].k : raw[t].q) + jl * PART;
        float* y = ((w & 1) ? steps[t].k : steps[t].q) + jl * PART;
        float f[PART];
#pragma unroll
        for (int c = 0; c < PART / 8; ++c) {
            const uint4 u = *reinterpret_cast<const uint4*>(x + 8 * c);
            const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                f[8 * c + 2 * e] = __uint_as_float(wd[e] << 16);
                f[8 * c + 2 * e + 1] = __uint_as_float(wd[e] & 0xFFFF0000u);
            }
        }
        float inv = 1.f;
        if (l2) {
            float c[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) c[q4] = __fmul_rn(f[q4], f[q4]);
#pragma unroll
            for (int e = 4; e < PART; e += 4) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) c[q4] = __fmaf_rn(f[e + q4], f[e + q4], c[q4]);
            }
            float ss = __fadd_rn(__fadd_rn(c[0], c[1]), __fadd_rn(c[2], c[3]));
            ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 1));
            ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 2));
            inv = __frcp_rn(__fsqrt_rn(__fadd_rn(ss, 1e-6f)));
        }
        if (!act) continue;
#pragma unroll
        for (int e = 0; e < PART; e += 4)
            *reinterpret_cast<float4*>(y + e) =
                l2 ? make_float4(__fmul_rn(f[e], inv), __fmul_rn(f[e + 1], inv), __fmul_rn(f[e + 2], inv),
                                 __fmul_rn(f[e + 3], inv))
                   : make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
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

// The step function shared by decode, replay and verify, for this thread's RPT rows (each
// row's operations are the same whatever RPT is):
//   S <- a S;  r = S k;  u = beta (v - r);  S <- S + u k^T;  o = S q
// each operation rounded once (packed f32x2 lanes are independent IEEE fp32 ops).
template <int DK, int RPT>
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

template <int DK, class T>
__global__ void __launch_bounds__(T::THREADS, T::MIN_BLOCKS) gdn_kernel(GdnArgs A) {
    griddep_launch();
    constexpr int NP = DK / (2 * LPR);
    constexpr int RPT = T::RPT, THREADS = T::THREADS;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int total = A.max_commit + A.k;
    StepSmem<DK>* steps = reinterpret_cast<StepSmem<DK>*>(smem_raw);
    RawStep<DK>* raw = reinterpret_cast<RawStep<DK>*>(smem_raw + sizeof(StepSmem<DK>) * (total > 0 ? total : 1));

    const int slab = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane % LPR;
    int r[RPT];                                           // rows within the slab
#pragma unroll
    for (int x = 0; x < RPT; ++x) r[x] = warp * T::ROWS_PER_WARP + x * (32 / LPR) + lane / LPR;
    const int row0 = slab * SLAB;
    float* srow0 = A.state + ((static_cast<size_t>(b) * A.H + h) * A.dv + row0) * DK;
    if (threadIdx.x == 0) l2_prefetch(srow0, SLAB * DK * 4);   // a hint only: the loads come after the wait
    griddep_wait();

    // Every load of the CTA in flight at once: each thread's state rows (the longest trip, into
    // registers), the asynchronous copies of the steps' q, k, v, the commit count and the beta
    // and gate scalars.
    float2 s[RPT][NP];
#pragma unroll
    for (int x = 0; x < RPT; ++x) load_slice<DK>(s[x], srow0 + static_cast<size_t>(r[x]) * DK, g);
    stage_raw<DK, THREADS>(raw, A, b, h, h / A.qk_group, row0, total);
    int nc = A.n_commit ? A.n_commit[b] : A.n_fixed;
    for (int idx = threadIdx.x; idx < 2 * total; idx += THREADS) {
        long long row;
        const GdnStepsDev& src = step_src(A, b, idx >> 1, &row);
        float x = bf16f((idx & 1) ? src.gate[row * src.gate_stride + h] : src.beta[row * src.gate_stride + h]);
        if (src.raw_gates) {
            // beta = bf16(sigmoid(b)), gate = bf16(exp(-softplus(a))), softplus(x) = x for x > 20
            if (idx & 1) x = bf16f(f32_to_bf16(expf(-(x > 20.f ? x : log1pf(expf(x))))));
            else x = bf16f(f32_to_bf16(__frcp_rn(__fadd_rn(1.f, expf(-x)))));
        }
        if (idx & 1) steps[idx >> 1].gate = x;
        else steps[idx >> 1].beta = x;
    }
    if (nc < 0 || nc > A.max_commit) {
        if (threadIdx.x == 0) atomicOr(A.err, ERR_BAD_COUNT);
        nc = nc < 0 ? 0 : A.max_commit;
    }
    cp_async_wait_all();
    __syncthreads();
    normalise_all<DK, THREADS>(steps, raw, total, A.l2 != 0);
    for (int idx = threadIdx.x; idx < total * SLAB; idx += THREADS)
        steps[idx / SLAB].v[idx % SLAB] = bf16f(raw[idx / SLAB].v[idx % SLAB]);
    __syncthreads();

    float o[RPT];
    // replay the committed steps (these change the stored state)
    for (int t = 0; t < nc; ++t) {
        gdn_step<DK, RPT>(s, steps[t], g, r, A.emit_replay != 0, o);
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
    // speculative steps: outputs only, the state in memory stays committed (with one row per
    // thread unrolled by 2 so that one step's output product can overlap the next step's decay
    // and key product; with several rows per thread those give the overlap)
#pragma unroll(RPT == 1 ? 2 : 1)
    for (int t = 0; t < A.k; ++t) {
        gdn_step<DK, RPT>(s, steps[A.max_commit + t], g, r, true, o);
        if (g == 0) {
#pragma unroll
            for (int x = 0; x < RPT; ++x)
                A.o[(static_cast<long long>(b) * A.k + t) * A.o_stride + static_cast<long long>(h) * A.dv + row0 + r[x]] =
                    f32_to_bf16(o[x]);
        }
    }
}

template <int DK, class T>
xv_status launch_tiled(const GdnArgs& a, int B, int H, int dv, int total, cudaStream_t s) {
    const size_t per_step = step_smem_bytes<DK>();
    const int max_bytes = static_cast<int>(per_step * XV_GDN_MAX_STAGED);
    if (xv_status st = kernel_smem_once(reinterpret_cast<const void*>(gdn_kernel<DK, T>), max_bytes, true,
                                        "gdn: set shared memory size"))
        return st;
    const dim3 grid(dv / SLAB, H, B);   // dv is a multiple of SLAB (checked)
    launch_k(gdn_kernel<DK, T>, grid, dim3(T::THREADS), per_step * (total > 0 ? total : 1), s, a);
    return XV_OK;
}

}  // namespace

xv_status gdn_launch(float* state, const GdnStepsDev& pending, const int32_t* n_commit, int n_fixed, int max_commit,
                     bool emit_replay, const GdnStepsDev& draft, int k, uint16_t* o, long long o_stride, int B, int H,
                     int Hk, int dk, int dv, int qk_l2norm, cudaStream_t s) {
    unsigned* err = device_error_word();
    if (!err) return fail(XV_ERR_CUDA, "gdn: device error word unavailable");
    if (Hk < 1 || H % Hk) return fail(XV_ERR_ARG, "gdn: %d v heads are not a multiple of %d q/k heads", H, Hk);
    GdnArgs a{state, pending, n_commit, n_fixed, max_commit, emit_replay ? 1 : 0, draft, k, o, o_stride, H, dv,
              qk_l2norm ? 1 : 0, H / Hk, err};
    const int max_steps = max_commit + k;
    if (max_steps > XV_GDN_MAX_STAGED)
        return fail(XV_ERR_UNSUPPORTED, "gdn: %d steps in one call exceed %d", max_steps, XV_GDN_MAX_STAGED);
    // Slabs of 32 rows: with at least two per SM the wide tiling (4 rows per thread, one warp per
    // slab) reads each k and q slice once for four rows; below that the narrow one (one row per
    // thread, four warps per slab) keeps more warps per SM on the latency-bound chain.  Every row's
    // arithmetic is the same in both.
    int sms = 0;
    if (xv_status st = device_sm_count(&sms)) return st;
    const long long slabs = static_cast<long long>(B) * H * (dv / SLAB);
    const bool wide = slabs >= 2ll * sms;
    trace_pre(s);
    xv_status st;
    if (dk == 128)
        st = wide ? launch_tiled<128, WideTiling>(a, B, H, dv, max_steps, s)
                  : launch_tiled<128, NarrowTiling>(a, B, H, dv, max_steps, s);
    else
        st = wide ? launch_tiled<64, WideTiling>(a, B, H, dv, max_steps, s)
                  : launch_tiled<64, NarrowTiling>(a, B, H, dv, max_steps, s);
    if (st) return st;
    // algorithmic bytes with every sequence replaying max_commit steps: the state
    // read (and written back after a replay), the step inputs, the outputs
    const long long state_bytes = 4ll * B * H * dv * dk;
    const long long per_step = 2ll * B * (2 * Hk * dk + H * (dv + 2));
    const long long outs = 2ll * B * H * dv * (k + (emit_replay ? max_commit : 0));
    const long long bytes = state_bytes * (max_commit > 0 ? 2 : 1) + per_step * (max_commit + k) + outs;
    return launched("gdn_kernel", s, K_GDN, bytes);
}

}  // namespace xv
