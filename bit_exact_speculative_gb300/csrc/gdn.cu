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
// lane/4 + 8, ... of its warp's 8 * RPT) of a slab of 32 state rows.  Every
// step reads the whole k and q vectors from shared memory into each row's
// lanes; with one row per thread that read (1 KB per row per step) is the
// bound, so wide calls hold 4 rows per thread (a warp per slab) and read each
// slice once for the four.
//  - Narrow calls (fewer heads than SMs: latency-bound) give each slab a CTA
//    of 4 warps with one row per thread.
//  - Wide calls give each (sequence, head) a CTA with a warp per slab; the
//    head's staged steps (q, k normalised once, v, beta, gate) are shared by
//    its warps, which keeps the shared memory of a head small enough for two
//    heads per SM, so a whole batch of 8 is one wave.
//
// Data movement: everything a CTA reads arrives by asynchronous bulk copies
// on mbarriers, issued right after the dependency wait: the state (16 KB per
// slab, contiguous rows) and the steps' raw q, k and v.  (Plain per-thread
// loads of the state, one 16-byte piece at a time, queued behind each other in
// the load/store unit and held the shared-memory traffic of the steps behind
// them.)  In wide calls the steps come by tensor copies (one per source and
// vector) and the slabs are requested one after another, each on its own
// barrier, so the first warps start on their slab while the later slabs are
// still arriving.  The state then lives in registers across all replay and
// speculative steps; after a replay it goes back through shared memory and a
// bulk store, and the outputs of every step are gathered in shared memory and
// written in 16-byte pieces at the end.
#include "xv_internal.h"
#include "xv_ptx.cuh"

namespace xv {

namespace {
constexpr int LPR = 4;                          // lanes per state row
constexpr int NORM_LANES = 4;                   // threads per q or k vector in the normalisation
constexpr int SLAB = 32;                        // state rows per team

// A launch shape: RPT state rows per thread, TEAM threads per slab.
template <int RPT_>
struct Tiling {
    static constexpr int RPT = RPT_;
    static constexpr int TEAM = SLAB * LPR / RPT;        // threads sharing one slab
    static constexpr int ROWS_PER_WARP = 32 / LPR * RPT;
};
using NarrowTiling = Tiling<1>;   // 128 threads per slab, one CTA each: few heads (latency-bound calls)
using WideTiling = Tiling<4>;     // one warp per slab, a CTA per head: shared-memory reads amortised
static_assert(WideTiling::TEAM == 32 && WideTiling::ROWS_PER_WARP == SLAB, "a wide team is one warp holding a slab");
constexpr int MAX_SLABS_PER_HEAD = 8;   // dv <= 256

// Tensor maps of the wide kernel: its step inputs (pending q, k, v, then draft q, k, v: 2-D views
// [rows, columns] of the step sources, a box one head's vector over the staged rows), then the
// state viewed as [B H dv rows, dk columns] fp32 in boxes of 32 rows x 32 columns (128 bytes, with
// the 128-byte swizzle: in shared memory the 16-byte chunk j of row r sits at chunk j ^ (r % 8),
// so the lanes of two rows never meet in a bank).
struct GdnMaps {
    CUtensorMap m[7];
};
constexpr int SW_COLS = 32;                     // fp32 columns of one swizzled state box (128 bytes)

// Address of fp32 element 4 c of row r in a swizzled slab: column block c / 8, chunk c % 8 of the
// row's 128 bytes there, moved to c % 8 ^ (r % 8).
__device__ __forceinline__ float* swz(float* slab, int r, int c) {
    return slab + (c >> 3) * (SLAB * SW_COLS) + r * SW_COLS + 4 * ((c & 7) ^ (r & 7));
}

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
    int o_vec;     // o and o_stride allow 16-byte stores
    int n_slabs;   // B * H * dv / SLAB
};

// Per-step inputs staged in shared memory: q and k (fp32, normalised; their raw bf16 copies land in
// the upper halves), beta and gate.
template <int DK>
struct StepSmem {
    float q[DK];
    float k[DK];
    float beta, gate;
    float pad[2];
};
static_assert(sizeof(StepSmem<128>) % 16 == 0 && sizeof(StepSmem<64>) % 16 == 0, "16-byte aligned steps");

// Shared-memory plan of one team: the state slab, the staged steps, the raw v slices, the outputs
// of every step (replayed ones first when they are emitted), the mbarrier.
template <int DK>
struct GdnSmem {
    size_t steps, rawv, obuf, bar, total;
    __host__ __device__ GdnSmem(int n_steps, int n_out) {
        steps = static_cast<size_t>(SLAB) * DK * 4;
        rawv = steps + sizeof(StepSmem<DK>) * n_steps;
        obuf = rawv + static_cast<size_t>(SLAB) * 2 * n_steps;
        bar = (obuf + static_cast<size_t>(SLAB) * 2 * n_out + 15) & ~static_cast<size_t>(15);
        total = (bar + 16 + 127) & ~static_cast<size_t>(127);
    }
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

__device__ __forceinline__ float bf16f(uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); }

// Synchronises the threads of a team: a wide team is one warp, a narrow one the whole CTA.
template <int TEAM>
__device__ __forceinline__ void team_sync() {
    if constexpr (TEAM == 32) __syncwarp();
    else __syncthreads();
}

// Vector w of the staged steps (step w / 2; q for even w, k for odd) from its raw bf16 copy to fp32,
// L2-normalised when l2 (x / sqrt(sum x^2 + 1e-6)).  The raw copy is row t of rq / rk, or, when rq
// is null, the upper half of the fp32 array itself (converted in place).  Thread j of the vector's
// group of NORM_LANES takes the 16-byte raw pieces j, j + 4, j + 8, ... (8 elements each, so the
// group's reads and writes fall in distinct banks), sums their squares in four interleaved chains
// (element index mod 4) added as (c0 + c1) + (c2 + c3), the group adds its partials by an xor
// tree (1, 2), and every thread scales its own elements.  nthreads threads (whole warps) take part.
template <int DK>
__device__ __forceinline__ void normalise_all(StepSmem<DK>* steps, const uint16_t* rq, const uint16_t* rk, int total,
                                              bool l2, int tid, int nthreads) {
    constexpr int PIECES = DK / 8 / NORM_LANES;   // raw 16-byte pieces per thread
    const int jl = tid % NORM_LANES;
    for (int w0 = 0; w0 < 2 * total; w0 += nthreads / NORM_LANES) {   // same trip count for every thread
        const int w = w0 + tid / NORM_LANES;
        const bool act = w < 2 * total;
        const int t = act ? w >> 1 : 0;
        float* y = (w & 1) ? steps[t].k : steps[t].q;
        const uint16_t* x = rq ? ((w & 1) ? rk : rq) + static_cast<size_t>(t) * DK
                               : reinterpret_cast<const uint16_t*>(y + DK / 2);
        float f[8 * PIECES];
#pragma unroll
        for (int i = 0; i < PIECES; ++i) {
            const uint4 u = *reinterpret_cast<const uint4*>(x + 8 * (jl + NORM_LANES * i));
            const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                f[8 * i + 2 * e] = __uint_as_float(wd[e] << 16);
                f[8 * i + 2 * e + 1] = __uint_as_float(wd[e] & 0xFFFF0000u);
            }
        }
        float inv = 1.f;
        if (l2) {
            float c[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) c[q4] = __fmul_rn(f[q4], f[q4]);
#pragma unroll
            for (int e = 4; e < 8 * PIECES; e += 4) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) c[q4] = __fmaf_rn(f[e + q4], f[e + q4], c[q4]);
            }
            float ss = __fadd_rn(__fadd_rn(c[0], c[1]), __fadd_rn(c[2], c[3]));
            ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 1));
            ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 2));
            inv = __frcp_rn(__fsqrt_rn(__fadd_rn(ss, 1e-6f)));
        }
        __syncwarp();   // an in-place group's raw halves are read before any fp32 element overwrites them
        if (!act) continue;
#pragma unroll
        for (int i = 0; i < PIECES; ++i) {
            float* d = y + 8 * (jl + NORM_LANES * i);
            const float* v = f + 8 * i;
            if (l2) {
                *reinterpret_cast<float4*>(d) =
                    make_float4(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv), __fmul_rn(v[2], inv), __fmul_rn(v[3], inv));
                *reinterpret_cast<float4*>(d + 4) =
                    make_float4(__fmul_rn(v[4], inv), __fmul_rn(v[5], inv), __fmul_rn(v[6], inv), __fmul_rn(v[7], inv));
            } else {
                *reinterpret_cast<float4*>(d) = make_float4(v[0], v[1], v[2], v[3]);
                *reinterpret_cast<float4*>(d + 4) = make_float4(v[4], v[5], v[6], v[7]);
            }
        }
    }
}

// beta = bf16(sigmoid(b)) (is_gate: gate = bf16(exp(-softplus(a))), softplus(x) = x for x > 20)
// from the raw projection column when the source holds raw values, else the bf16 value itself.
__device__ __forceinline__ float gate_value(uint16_t raw, bool is_gate, bool raw_gates) {
    float x = bf16f(raw);
    if (raw_gates) {
        if (is_gate) x = bf16f(f32_to_bf16(expf(-(x > 20.f ? x : log1pf(expf(x))))));
        else x = bf16f(f32_to_bf16(__frcp_rn(__fadd_rn(1.f, expf(-x)))));
    }
    return x;
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
__device__ __forceinline__ void gdn_step(float2 (&s)[RPT][DK / (2 * LPR)], const StepSmem<DK>& in,
                                         const uint16_t* v, int g, const int (&r)[RPT], bool want_o, float (&o)[RPT]) {
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
        const float uu = __fmul_rn(in.beta, __fsub_rn(bf16f(v[r[x]]), rr[x]));
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
__global__ void __launch_bounds__(T::TEAM, 2) gdn_kernel(GdnArgs A) {
    griddep_launch();
    constexpr int NP = DK / (2 * LPR);
    constexpr int RPT = T::RPT, TEAM = T::TEAM;
    extern __shared__ __align__(128) uint8_t smem_all[];
    const int total = A.max_commit + A.k;
    const int n_out = A.k + (A.emit_replay ? A.max_commit : 0);
    const GdnSmem<DK> L(total, n_out);
    const int tid = static_cast<int>(threadIdx.x);
    const int slab_id = blockIdx.x;
    uint8_t* smem_raw = smem_all;
    float* sstate = reinterpret_cast<float*>(smem_raw);
    StepSmem<DK>* steps = reinterpret_cast<StepSmem<DK>*>(smem_raw + L.steps);
    uint16_t* rawv = reinterpret_cast<uint16_t*>(smem_raw + L.rawv);
    uint16_t* obuf = reinterpret_cast<uint16_t*>(smem_raw + L.obuf);
    const uint32_t bar = smem_u32(smem_raw + L.bar);

    const int slabs_per_head = A.dv / SLAB;
    const int slab = slab_id % slabs_per_head, h = (slab_id / slabs_per_head) % A.H;
    const int b = slab_id / (slabs_per_head * A.H), hk = h / A.qk_group;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane % LPR;
    int r[RPT];                                           // rows within the slab
#pragma unroll
    for (int x = 0; x < RPT; ++x) r[x] = warp * T::ROWS_PER_WARP + x * (32 / LPR) + lane / LPR;
    const int row0 = slab * SLAB;
    float* gslab = A.state + ((static_cast<size_t>(b) * A.H + h) * A.dv + row0) * DK;
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        l2_prefetch(gslab, SLAB * DK * 4);   // a hint only: the copies come after the wait
    }
    team_sync<TEAM>();
    griddep_wait();

    // Every copy of the team in flight at once, spread over its threads: the state slab, then per
    // staged step its raw q and k (into the upper halves of the fp32 arrays) and its v slice.
    // The beta and gate scalars and the commit count are plain loads issued alongside.
    constexpr uint32_t QK_BYTES = DK * 2, V_BYTES = SLAB * 2;
    if (tid == 0) mbar_arrive_expect_tx(bar, SLAB * DK * 4 + total * (2 * QK_BYTES + V_BYTES));
    for (int c = tid; c < 1 + 3 * total; c += TEAM) {
        if (c == 0) {
            bulk_load(smem_u32(sstate), gslab, SLAB * DK * 4, bar);
            continue;
        }
        const int t = (c - 1) / 3, which = (c - 1) % 3;
        long long row;
        const GdnStepsDev& src = step_src(A, b, t, &row);
        const long long base = row * src.qkv_stride;
        if (which == 0)
            bulk_load(smem_u32(steps[t].q + DK / 2), src.q + base + static_cast<long long>(hk) * DK, QK_BYTES, bar);
        else if (which == 1)
            bulk_load(smem_u32(steps[t].k + DK / 2), src.k + base + static_cast<long long>(hk) * DK, QK_BYTES, bar);
        else
            bulk_load(smem_u32(rawv + t * SLAB), src.v + base + static_cast<long long>(h) * A.dv + row0, V_BYTES, bar);
    }
    uint16_t bg[2] = {0, 0};   // entries tid and tid + TEAM of (beta, gate) x step
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int idx = tid + q * TEAM;
        if (idx < 2 * total) {
            long long row;
            const GdnStepsDev& src = step_src(A, b, idx >> 1, &row);
            bg[q] = (idx & 1) ? src.gate[row * src.gate_stride + h] : src.beta[row * src.gate_stride + h];
        }
    }
    int nc = A.n_commit ? A.n_commit[b] : A.n_fixed;
    if (nc < 0 || nc > A.max_commit) {
        if (tid == 0) atomicOr(A.err, ERR_BAD_COUNT);
        nc = nc < 0 ? 0 : A.max_commit;
    }
    mbar_wait(bar, 0, A.err);

    normalise_all<DK>(steps, nullptr, nullptr, total, A.l2 != 0, tid, TEAM);
    for (int idx = tid; idx < 2 * total; idx += TEAM) {
        long long row;
        const GdnStepsDev& src = step_src(A, b, idx >> 1, &row);
        const uint16_t raw = idx < 2 * TEAM ? (idx >= TEAM ? bg[1] : bg[0])
                                            : ((idx & 1) ? src.gate[row * src.gate_stride + h]
                                                         : src.beta[row * src.gate_stride + h]);
        const float x = gate_value(raw, idx & 1, src.raw_gates != 0);
        if (idx & 1) steps[idx >> 1].gate = x;
        else steps[idx >> 1].beta = x;
    }
    float2 s[RPT][NP];
#pragma unroll
    for (int x = 0; x < RPT; ++x) load_slice<DK>(s[x], sstate + r[x] * DK, g);
    team_sync<TEAM>();

    float o[RPT];
    // replay the committed steps (these change the stored state)
    const int orow_spec = A.emit_replay ? nc : 0;
    for (int t = 0; t < nc; ++t) {
        gdn_step<DK, RPT>(s, steps[t], rawv + t * SLAB, g, r, A.emit_replay != 0, o);
        if (A.emit_replay && g == 0) {
#pragma unroll
            for (int x = 0; x < RPT; ++x) obuf[t * SLAB + r[x]] = f32_to_bf16(o[x]);
        }
    }
    if (nc > 0) {
        // the committed state goes back through shared memory and one bulk store
#pragma unroll
        for (int x = 0; x < RPT; ++x) {
#pragma unroll
            for (int u = 0; u < NP / 2; ++u)
                *reinterpret_cast<float4*>(sstate + r[x] * DK + 4 * (g + LPR * u)) =
                    make_float4(s[x][2 * u].x, s[x][2 * u].y, s[x][2 * u + 1].x, s[x][2 * u + 1].y);
        }
        fence_proxy_async_smem();
        team_sync<TEAM>();
        if (tid == 0) {
            bulk_store(gslab, smem_u32(sstate), SLAB * DK * 4);
            bulk_commit();
        }
    }
    // speculative steps: outputs only, the state in memory stays committed (with one row per
    // thread unrolled by 2 so that one step's output product can overlap the next step's decay
    // and key product; with several rows per thread those give the overlap)
#pragma unroll(RPT == 1 ? 2 : 1)
    for (int t = 0; t < A.k; ++t) {
        gdn_step<DK, RPT>(s, steps[A.max_commit + t], rawv + (A.max_commit + t) * SLAB, g, r, true, o);
        if (g == 0) {
#pragma unroll
            for (int x = 0; x < RPT; ++x) obuf[(orow_spec + t) * SLAB + r[x]] = f32_to_bf16(o[x]);
        }
    }
    team_sync<TEAM>();
    // outputs: row t of the buffer is the slab's 32 values of output row (b, t) (replayed rows
    // first when emitted, then the speculative ones), 16 bytes per thread
    const int rows_out = orow_spec + A.k;
    constexpr int CH = SLAB / 8;
    for (int idx = tid; idx < rows_out * CH; idx += TEAM) {
        const int t = idx / CH, c = idx % CH;
        const long long orow = t < orow_spec ? static_cast<long long>(b) * nc + t
                                             : static_cast<long long>(b) * A.k + (t - orow_spec);
        uint16_t* dst = A.o + orow * A.o_stride + static_cast<long long>(h) * A.dv + row0 + 8 * c;
        const uint4 v = *reinterpret_cast<const uint4*>(obuf + t * SLAB + 8 * c);
        if (A.o_vec) {
            *reinterpret_cast<uint4*>(dst) = v;
        } else {
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dst[2 * i] = static_cast<uint16_t>(w[i] & 0xFFFFu);
                dst[2 * i + 1] = static_cast<uint16_t>(w[i] >> 16);
            }
        }
    }
    if (nc > 0 && tid == 0) bulk_wait_read();   // the state slab stays in shared memory until read
}

// Shared-memory plan of a wide (per-head) CTA: the staged steps (fp32 q, k, beta, gate), the raw
// q, k and v rows the tensor copies land in, each warp's state slab and outputs, the barriers (the
// step inputs', then one per slab).
template <int DK>
struct HeadSmem {
    size_t rawq, rawk, rawv, state, obuf, bars, total;
    __host__ __device__ HeadSmem(int n_steps, int n_out, int dv) {
        const size_t nsl = dv / SLAB;
        auto r128 = [](size_t x) { return (x + 127) & ~static_cast<size_t>(127); };
        rawq = r128(sizeof(StepSmem<DK>) * n_steps);
        rawk = r128(rawq + static_cast<size_t>(n_steps) * DK * 2);
        rawv = r128(rawk + static_cast<size_t>(n_steps) * DK * 2);
        state = (rawv + static_cast<size_t>(n_steps) * dv * 2 + 1023) & ~static_cast<size_t>(1023);
        obuf = state + nsl * SLAB * DK * 4;
        bars = r128(obuf + nsl * n_out * SLAB * 2);
        total = bars + 8 * (1 + nsl);
    }
};

// One (sequence, head) per CTA, a warp per 32-row slab with 4 rows per thread.  Thread 0 requests
// the step inputs (six tensor copies: pending and draft q, k, v over the staged rows), then the
// slabs one after another, each on its own barrier; all threads normalise the head's q and k once;
// each warp then waits only for its own slab.
template <int DK>
__global__ void __launch_bounds__(32 * MAX_SLABS_PER_HEAD, 1)
    gdn_head_kernel(const __grid_constant__ GdnMaps M, GdnArgs A) {
    griddep_launch();
    constexpr int NP = DK / (2 * LPR), RPT = WideTiling::RPT;
    extern __shared__ __align__(128) uint8_t smem[];
    const int total = A.max_commit + A.k;
    const int n_out = A.k + (A.emit_replay ? A.max_commit : 0);
    const int nsl = A.dv / SLAB, nthreads = 32 * nsl;
    const HeadSmem<DK> L(total, n_out, A.dv);
    StepSmem<DK>* steps = reinterpret_cast<StepSmem<DK>*>(smem);
    uint16_t* rawq = reinterpret_cast<uint16_t*>(smem + L.rawq);
    uint16_t* rawk = reinterpret_cast<uint16_t*>(smem + L.rawk);
    uint16_t* rawv = reinterpret_cast<uint16_t*>(smem + L.rawv);
    const int h = blockIdx.x % A.H, b = blockIdx.x / A.H, hk = h / A.qk_group;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane % LPR;
    float* sstate = reinterpret_cast<float*>(smem + L.state) + warp * SLAB * DK;
    uint16_t* obuf = reinterpret_cast<uint16_t*>(smem + L.obuf) + warp * n_out * SLAB;
    const uint32_t bar_in = smem_u32(smem + L.bars), bar_slab = bar_in + 8 * (1 + warp);
    const int row0 = warp * SLAB;
    int r[RPT];                                           // rows within the slab
#pragma unroll
    for (int x = 0; x < RPT; ++x) r[x] = x * (32 / LPR) + lane / LPR;
    if (tid == 0) {
        for (int i = 0; i <= nsl; ++i) mbar_init(bar_in + 8 * i, 1);
        fence_mbar_init();
        for (int i = 0; i < 7; ++i) tma_prefetch_desc(&M.m[i]);
    }
    __syncthreads();
    griddep_wait();
    // The beta and gate scalars first (plain loads by warps 1.., so they are queued ahead of the
    // copies and warp 0 is free to issue those), then thread 0 requests the step inputs and the
    // slabs in order.
    const int gtid = tid - 32, gthreads = nthreads - 32;   // the gate threads (all warps but 0)
    uint16_t bg[2] = {0, 0};   // entries gtid and gtid + gthreads of (beta, gate) x step
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int idx = gtid + q * gthreads;
        if (gtid >= 0 && idx < 2 * total) {
            long long row;
            const GdnStepsDev& src = step_src(A, b, idx >> 1, &row);
            bg[q] = (idx & 1) ? src.gate[row * src.gate_stride + h] : src.beta[row * src.gate_stride + h];
        }
    }
    if (tid == 0) {
        mbar_arrive_expect_tx(bar_in, static_cast<uint32_t>(total) * (4 * DK + 2 * A.dv));
        if (A.max_commit > 0) {
            const int y = b * A.pend.rows_per_seq;
            tma_load_2d(smem_u32(rawq), &M.m[0], hk * DK, y, bar_in);
            tma_load_2d(smem_u32(rawk), &M.m[1], hk * DK, y, bar_in);
            tma_load_2d(smem_u32(rawv), &M.m[2], h * A.dv, y, bar_in);
        }
        if (A.k > 0) {
            const int y = b * A.draft.rows_per_seq;
            tma_load_2d(smem_u32(rawq + A.max_commit * DK), &M.m[3], hk * DK, y, bar_in);
            tma_load_2d(smem_u32(rawk + A.max_commit * DK), &M.m[4], hk * DK, y, bar_in);
            tma_load_2d(smem_u32(rawv + A.max_commit * A.dv), &M.m[5], h * A.dv, y, bar_in);
        }
        const int grow = (b * A.H + h) * A.dv;   // first state row of the head
        for (int w = 0; w < nsl; ++w) {
            const uint32_t bw = bar_in + 8 * (1 + w);
            float* slab = reinterpret_cast<float*>(smem + L.state) + w * SLAB * DK;
            mbar_arrive_expect_tx(bw, SLAB * DK * 4);
#pragma unroll
            for (int cb = 0; cb < DK / SW_COLS; ++cb)
                tma_load_2d(smem_u32(slab + cb * SLAB * SW_COLS), &M.m[6], cb * SW_COLS, grow + w * SLAB, bw);
        }
    }
    int nc = A.n_commit ? A.n_commit[b] : A.n_fixed;
    if (nc < 0 || nc > A.max_commit) {
        if (tid == 0) atomicOr(A.err, ERR_BAD_COUNT);
        nc = nc < 0 ? 0 : A.max_commit;
    }
    mbar_wait(bar_in, 0, A.err);
    normalise_all<DK>(steps, rawq, rawk, total, A.l2 != 0, tid, nthreads);
    for (int idx = gtid; gtid >= 0 && idx < 2 * total; idx += gthreads) {
        long long row;
        const GdnStepsDev& src = step_src(A, b, idx >> 1, &row);
        const uint16_t raw = idx < 2 * gthreads ? (idx >= gthreads ? bg[1] : bg[0])
                                                : ((idx & 1) ? src.gate[row * src.gate_stride + h]
                                                             : src.beta[row * src.gate_stride + h]);
        const float x = gate_value(raw, idx & 1, src.raw_gates != 0);
        if (idx & 1) steps[idx >> 1].gate = x;
        else steps[idx >> 1].beta = x;
    }
    __syncthreads();
    mbar_wait(bar_slab, 0, A.err);
    float2 s[RPT][NP];
#pragma unroll
    for (int x = 0; x < RPT; ++x) {
#pragma unroll
        for (int u = 0; u < NP / 2; ++u) {
            const float4 t = *reinterpret_cast<const float4*>(swz(sstate, r[x], g + LPR * u));
            s[x][2 * u] = make_float2(t.x, t.y);
            s[x][2 * u + 1] = make_float2(t.z, t.w);
        }
    }
    __syncwarp();

    float o[RPT];
    const int orow_spec = A.emit_replay ? nc : 0;
    for (int t = 0; t < nc; ++t) {
        gdn_step<DK, RPT>(s, steps[t], rawv + t * A.dv + row0, g, r, A.emit_replay != 0, o);
        if (A.emit_replay && g == 0) {
#pragma unroll
            for (int x = 0; x < RPT; ++x) obuf[t * SLAB + r[x]] = f32_to_bf16(o[x]);
        }
    }
    if (nc > 0) {
#pragma unroll
        for (int x = 0; x < RPT; ++x) {
#pragma unroll
            for (int u = 0; u < NP / 2; ++u)
                *reinterpret_cast<float4*>(swz(sstate, r[x], g + LPR * u)) =
                    make_float4(s[x][2 * u].x, s[x][2 * u].y, s[x][2 * u + 1].x, s[x][2 * u + 1].y);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            const int grow = (b * A.H + h) * A.dv + row0;
#pragma unroll
            for (int cb = 0; cb < DK / SW_COLS; ++cb)
                tma_store_2d(&M.m[6], cb * SW_COLS, grow, smem_u32(sstate + cb * SLAB * SW_COLS));
            bulk_commit();
        }
    }
    for (int t = 0; t < A.k; ++t) {
        gdn_step<DK, RPT>(s, steps[A.max_commit + t], rawv + (A.max_commit + t) * A.dv + row0, g, r, true, o);
        if (g == 0) {
#pragma unroll
            for (int x = 0; x < RPT; ++x) obuf[(orow_spec + t) * SLAB + r[x]] = f32_to_bf16(o[x]);
        }
    }
    __syncwarp();
    const int rows_out = orow_spec + A.k;
    constexpr int CH = SLAB / 8;
    for (int idx = lane; idx < rows_out * CH; idx += 32) {
        const int t = idx / CH, c = idx % CH;
        const long long orow = t < orow_spec ? static_cast<long long>(b) * nc + t
                                             : static_cast<long long>(b) * A.k + (t - orow_spec);
        uint16_t* dst = A.o + orow * A.o_stride + static_cast<long long>(h) * A.dv + row0 + 8 * c;
        const uint4 v = *reinterpret_cast<const uint4*>(obuf + t * SLAB + 8 * c);
        if (A.o_vec) {
            *reinterpret_cast<uint4*>(dst) = v;
        } else {
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dst[2 * i] = static_cast<uint16_t>(w4[i] & 0xFFFFu);
                dst[2 * i + 1] = static_cast<uint16_t>(w4[i] >> 16);
            }
        }
    }
    if (nc > 0 && lane == 0) bulk_wait_read();   // the slab stays in shared memory until read
}

template <int DK>
xv_status launch_narrow(const GdnArgs& a, int total, int n_out, cudaStream_t s) {
    using T = NarrowTiling;
    if (xv_status st = kernel_smem_once(reinterpret_cast<const void*>(gdn_kernel<DK, T>), XV_GDN_SMEM_MAX, true,
                                        "gdn: set shared memory size"))
        return st;
    launch_k(gdn_kernel<DK, T>, dim3(a.n_slabs), dim3(T::TEAM), GdnSmem<DK>(total, n_out).total, s, a);
    return XV_OK;
}

// 2-D view [rows, cols] of a step source's columns starting at `base`, boxes of `box_cols` x
// `box_rows` (bf16, no swizzle).
inline xv_status step_map(CUtensorMap* m, const uint16_t* base, long long cols, long long rows, long long stride,
                          int box_cols, int box_rows) {
    const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
    const uint64_t strides[1] = {static_cast<uint64_t>(stride) * 2};
    const uint32_t box[2] = {static_cast<uint32_t>(box_cols), static_cast<uint32_t>(box_rows)};
    return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int DK>
xv_status launch_head(const GdnArgs& a, int B, int Hk, int total, int n_out, size_t smem, cudaStream_t s) {
    GdnMaps M{};
    const GdnStepsDev* src[2] = {&a.pend, &a.draft};
    const int rows[2] = {a.max_commit, a.k};
    for (int i = 0; i < 2; ++i) {
        if (rows[i] == 0) continue;
        const GdnStepsDev& d = *src[i];
        const long long nrows = static_cast<long long>(B) * d.rows_per_seq;
        xv_status st;
        if ((st = step_map(&M.m[3 * i], d.q, static_cast<long long>(Hk) * DK, nrows, d.qkv_stride, DK, rows[i])))
            return st;
        if ((st = step_map(&M.m[3 * i + 1], d.k, static_cast<long long>(Hk) * DK, nrows, d.qkv_stride, DK, rows[i])))
            return st;
        if ((st = step_map(&M.m[3 * i + 2], d.v, static_cast<long long>(a.H) * a.dv, nrows, d.qkv_stride, a.dv, rows[i])))
            return st;
    }
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(DK), static_cast<uint64_t>(B) * a.H * a.dv};
        const uint64_t strides[1] = {static_cast<uint64_t>(DK) * 4};
        const uint32_t box[2] = {SW_COLS, SLAB};
        if (xv_status st = encode_tiled(&M.m[6], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.state, dims, strides, box,
                                        CU_TENSOR_MAP_SWIZZLE_128B))
            return st;
    }
    if (xv_status st = kernel_smem_once(reinterpret_cast<const void*>(gdn_head_kernel<DK>), XV_GDN_SMEM_MAX, true,
                                        "gdn: set shared memory size"))
        return st;
    (void)total;
    (void)n_out;
    launch_k(gdn_head_kernel<DK>, dim3(B * a.H), dim3(32 * (a.dv / SLAB)), smem, s, M, a);
    return XV_OK;
}

}  // namespace

xv_status gdn_launch(float* state, const GdnStepsDev& pending, const int32_t* n_commit, int n_fixed, int max_commit,
                     bool emit_replay, const GdnStepsDev& draft, int k, uint16_t* o, long long o_stride, int B, int H,
                     int Hk, int dk, int dv, int qk_l2norm, cudaStream_t s) {
    unsigned* err = device_error_word();
    if (!err) return fail(XV_ERR_CUDA, "gdn: device error word unavailable");
    if (Hk < 1 || H % Hk) return fail(XV_ERR_ARG, "gdn: %d v heads are not a multiple of %d q/k heads", H, Hk);
    if (!aligned16(state)) return fail(XV_ERR_UNSUPPORTED, "gdn: the state must be 16-byte aligned");
    const long long slabs = static_cast<long long>(B) * H * (dv / SLAB);   // dv is a multiple of SLAB (checked)
    if (slabs > (1ll << 30)) return fail(XV_ERR_UNSUPPORTED, "gdn: %lld slabs", slabs);
    GdnArgs a{state, pending, n_commit, n_fixed, max_commit, emit_replay ? 1 : 0, draft, k, o, o_stride, H, dv,
              qk_l2norm ? 1 : 0, H / Hk, err, (aligned16(o) && o_stride % 8 == 0) ? 1 : 0, static_cast<int>(slabs)};
    const int max_steps = max_commit + k;
    if (max_steps > XV_GDN_MAX_STAGED)
        return fail(XV_ERR_UNSUPPORTED, "gdn: %d steps in one call exceed %d", max_steps, XV_GDN_MAX_STAGED);
    const int n_out = k + (emit_replay ? max_commit : 0);
    // With at least one head per SM the wide kernel (a CTA per head, a warp per slab, 4 rows per
    // thread) reads each k and q slice once for four rows and shares the head's staged steps among
    // its slabs, as long as two such CTAs fit an SM (else the batch would take two waves); below
    // that, or with more staged steps (prefill chunks), the narrow one (a CTA per slab, a row per
    // thread) keeps more warps on each slab's latency-bound chain.  Every row's arithmetic is the
    // same in both.
    int sms = 0;
    if (xv_status st = device_sm_count(&sms)) return st;
    const size_t head_smem = dk == 128 ? HeadSmem<128>(max_steps, n_out, dv).total : HeadSmem<64>(max_steps, n_out, dv).total;
    const bool wide = static_cast<long long>(B) * H >= sms && dv / SLAB >= 2 && dv / SLAB <= MAX_SLABS_PER_HEAD &&
                      2 * (head_smem + 1024) <= static_cast<size_t>(XV_GDN_SMEM_SM) && B * H < (1 << 30);
    trace_pre(s);
    xv_status st;
    if (wide)
        st = dk == 128 ? launch_head<128>(a, B, Hk, max_steps, n_out, head_smem, s)
                       : launch_head<64>(a, B, Hk, max_steps, n_out, head_smem, s);
    else
        st = dk == 128 ? launch_narrow<128>(a, max_steps, n_out, s) : launch_narrow<64>(a, max_steps, n_out, s);
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
