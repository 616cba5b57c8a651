// Small-M bf16 weight-streaming GEMM on the 5th-generation tensor cores.
//
//   Y[M, N] = X[M, K] . W[N, K]^T, fp32 accumulate, bf16 (or fp32) out.
//
// Why it exists ("Follow-up to my earlier post on Qwen3.8-27B decode speed",
// r/LocalLLaMA post, and the recipe card's summary): at decode and verify
// batch sizes the projection GEMMs must (1) give the same bits for a row
// whatever the number of rows, so that verifying k tokens at once equals
// decoding them one by one, and (2) stream the weights near DRAM speed
// (the post measured the previous small-batch kernel at about a third).
//
// Design (GB300, sm_103a):
//   - Swap-AB: a CTA owns 128 weight rows (the MMA's M side); the tokens are
//     the MMA's N side, ALWAYS padded to 64 columns whatever M is, so every
//     call issues the identical tcgen05.mma sequence.  Each output element is
//     the dot product of one weight row with one token row: no element reads
//     another row's data, which makes row i independent of M and of its
//     position (the padding rows are TMA zero fill).
//   - Weights and tokens arrive by TMA (cp.async.bulk.tensor, 128-byte
//     swizzle) into a 4-stage shared-memory ring, 64 K-elements per stage;
//     one thread issues TMA, one thread issues tcgen05.mma, the accumulator
//     (128 x 64 fp32) lives in TMEM and is read back with tcgen05.ld.
//   - Split-K over S segments with S a function of (N, K) only; a segment
//     covers K-blocks [s*nkb/S, (s+1)*nkb/S).  Segment partials go to the
//     workspace; the last-arriving CTA of a tile (atomic counter after a
//     __threadfence) adds them in segment order 0..S-1 — the same order
//     whichever CTA is last — rounds once and resets the counter.
//   - Every mbarrier wait is bounded; a timeout records an error bit and
//     the CTA drains its copies in flight, frees TMEM and returns.
//   - Gate/up with the SwiGLU fused: in the gated tiled layout a tile holds
//     64 gate rows and the 64 up rows of the same features, so one CTA has
//     both halves of each of its 64 features; the epilogue rounds g and u to
//     bf16 as a stored gate/up row would be, forms bf16(silu(g) u) with the
//     SwiGLU kernel's own arithmetic and writes only the activations.  Such a
//     GEMM is never split (each output is one whole-K sum, as for the
//     34816-wide gate/up anyway), so its bits are those of GEMM + SwiGLU.
//   - Weights come in one of two layouts: row-major [N, K], or tiled, each
//     128 x 64 tile (one ring stage) a contiguous 16 KiB and a tile row's
//     K-blocks one after another.  A row-major stage is 128 pieces of 128
//     bytes, K * 2 bytes apart; a tiled stage is one contiguous run, and a
//     CTA's whole segment one longer run.  The TMA delivers the same values
//     to the same shared-memory places from either layout, so the bits
//     agree; measured on GB300 the tiled layout streams faster (the 151936 x
//     5120 LM head 254 -> 242 us, the verify step 894 -> 865 us).
//   - The unsplit fp32 GEMM (the LM head) can also leave, for every token row
//     and weight tile, the tile's maximum and its lowest index, from which the
//     argmax follows without a pass over the logits (which it then need not
//     write).
//   - A split GEMM can hand its segment partials [S][M][N] to the caller
//     instead of combining them; the residual RMSNorm adds them in the same
//     segment order, so the bits are those of the combine.
#include "xv_internal.h"
#include "xv_ptx.cuh"

namespace xv {

namespace {
constexpr int STAGES = 4;
constexpr int A_BYTES = GEMM_BN * GEMM_BK * 2;   // 16 KB of weights per stage
constexpr int B_BYTES = GEMM_TOK * GEMM_BK * 2;  //  8 KB: 64 token rows of one K-block
// Token rows have a ring of their own.  For M > 8 it holds STAGES slots of 64 rows (8 KB) and
// advances with the weights.  For M <= 8 a slot is the 8 rows of one K-block (one 1 KB swizzle
// atom) and the ring has X_RING slots, so the tokens are requested up to X_RING - STAGES
// K-blocks ahead of the weights: every CTA re-reads them from L2 on every stage, and measured
// on GB300 that read stalls the 4-stage weight ring whenever the activation buffer sits at an
// unlucky place in memory (up to +14% per GEMM).  The MMA still sees 64 token rows: its 8-row
// groups all read the one atom (group stride 0), so columns 8..63 repeat columns 0..7.
constexpr int X_RING = 16;
constexpr int X_SMALL_M = 8;
constexpr int N_BARS = 2 * STAGES + 2 * X_RING + 1;   // full, empty, xfull, xempty, done
constexpr int TMEM_COLS = 64;
constexpr int smem_bytes(int xb, int xr) { return 1024 + STAGES * A_BYTES + xr * xb + 8 * N_BARS + 16; }
constexpr int SMEM_MAX = smem_bytes(B_BYTES, STAGES) > smem_bytes(1024, X_RING) ? smem_bytes(B_BYTES, STAGES)
                                                                                   : smem_bytes(1024, X_RING);
constexpr uint32_t IDESC = idesc_bf16_f32(GEMM_BN, GEMM_TOK);
constexpr int SM_COUNT_TARGET = 152;   // GB300
// Splits of 2..CLUSTER_MAX segments are combined inside a thread-block cluster through
// distributed shared memory (no workspace); larger ones, used only by narrow shapes with
// too few tiles to fill the GPU otherwise, go through the workspace.
constexpr int CLUSTER_MAX = 4;
constexpr int RESIDENT_PER_SM = 2;
constexpr int MIN_SEGMENT_KB = 8;    // K-blocks a split-K segment streams at least

template <bool F32OUT, bool GATED>
__global__ void __launch_bounds__(128, RESIDENT_PER_SM)
    gemm_small_m_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                        void* __restrict__ Y, int ldy, int M, int N, int nkb, int S, float* __restrict__ part,
                        unsigned* __restrict__ cnt, unsigned* __restrict__ err, int cluster_combine, int xb,
                        int xr, int wtiled, float2* __restrict__ amax) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_last;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const uint32_t sA = base;
    const uint32_t sX = base + STAGES * A_BYTES;            // token ring: xr slots of xb bytes
    const uint32_t bar0 = sX + xr * xb;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto xfull = [&](int j) { return bar0 + 8u * (2 * STAGES + j); };
    auto xempty = [&](int j) { return bar0 + 8u * (2 * STAGES + X_RING + j); };
    const uint32_t done = bar0 + 8u * (2 * STAGES + 2 * X_RING);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + (bar0 - base) + 8 * N_BARS);
    const uint32_t xgroup = xb == B_BYTES ? 1024u : 0u;   // 8-row group stride of the token operand

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x, seg = blockIdx.y;
    const int kb0 = static_cast<int>(static_cast<long long>(seg) * nkb / S);
    const int kb1 = static_cast<int>(static_cast<long long>(seg + 1) * nkb / S);
    const int nk = kb1 - kb0;

    griddep_launch();
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int j = 0; j < xr; ++j) {
            mbar_init(xfull(j), 1);
            mbar_init(xempty(j), 1);
        }
        mbar_init(done, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    bool ok = true;
    if (warp == 0 && lane == 0) {
        // ---- producer: TMA into the ring.  The weights of the first stages are requested
        // before waiting for the previous kernel (they do not depend on it); the token rows
        // only after.
        const uint64_t stream_policy = l2_policy_evict_first();   // each weight is read once
        // the weight tile (tile, K-block kb): row-major at (kb * BK, tile * BN); tiled, the
        // (tile * nkb + kb)-th 128-row block of a [tiles * nkb * 128, 64] array
        auto wx = [&](int kb) { return wtiled ? 0 : kb * GEMM_BK; };
        auto wy = [&](int kb) { return wtiled ? (tile * nkb + kb) * GEMM_BN : tile * GEMM_BN; };
        const int pre = nk < STAGES ? nk : STAGES;
        for (int i = 0; i < pre; ++i) {
            mbar_arrive_expect_tx(full(i), A_BYTES);
            tma_load_2d_hint(sA + i * A_BYTES, &tmW, wx(kb0 + i), wy(kb0 + i), full(i), stream_policy);
        }
        griddep_wait();
        // token K-blocks up to (but not including) `lim`; slot reuse waits for the MMAs of the
        // K-block xr earlier, never stricter than the weight ring's own wait
        int xi = 0;
        auto issue_x = [&](int lim) -> bool {
            for (; xi < lim; ++xi) {
                const int js = xi % xr;
                if (xi >= xr && !mbar_wait(xempty(js), ((xi / xr) & 1u) ^ 1u, err)) return false;
                mbar_arrive_expect_tx(xfull(js), xb);
                tma_load_2d(sX + js * xb, &tmX, (kb0 + xi) * GEMM_BK, 0, xfull(js));
            }
            return true;
        };
        ok = issue_x(min(nk, xr));
        int issued = pre;
        for (int i = pre; ok && i < nk; ++i) {
            const int st = i % STAGES;
            const uint32_t ph = (i / STAGES) & 1u;
            if (i >= STAGES && !mbar_wait(empty(st), ph ^ 1u, err)) { ok = false; break; }
            mbar_arrive_expect_tx(full(st), A_BYTES);
            tma_load_2d_hint(sA + st * A_BYTES, &tmW, wx(kb0 + i), wy(kb0 + i), full(st), stream_policy);
            issued = i + 1;
            ok = issue_x(min(nk, i + 1 + xr - STAGES));
        }
        if (!ok) {  // drain: every issued copy must land before the CTA may exit
            for (int j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j)
                mbar_wait(full(j % STAGES), (j / STAGES) & 1u, err);
            for (int j = xi > xr ? xi - xr : 0; j < xi; ++j) mbar_wait(xfull(j % xr), (j / xr) & 1u, err);
        }
    } else {
        // An L2 prefetch of this CTA's K-blocks beyond the ring, issued here before the wait, was
        // measured to slow the verify step down (897 -> 908 us with 8 blocks, 962 with 24): the
        // ring's own early weight loads are the useful prefetch.
        griddep_wait();   // before any read or write of activations, partials or counters
    }
    if (warp == 1 && lane == 0) {
        // ---- MMA issuer: 4 MMAs of K = 16 per stage, accumulate in TMEM
        for (int i = 0; i < nk; ++i) {
            const int st = i % STAGES, js = i % xr;
            if (!mbar_wait(full(st), (i / STAGES) & 1u, err)) { ok = false; break; }
            if (!mbar_wait(xfull(js), (i / xr) & 1u, err)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < GEMM_BK / 16; ++kk) {
                const uint64_t ad = sw128_kmajor_desc(sA + st * A_BYTES + kk * 32);
                const uint64_t bd = sw128_kmajor_desc(sX + js * xb + kk * 32, xgroup);
                tc_mma_bf16(tmem, ad, bd, IDESC, (i > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(empty(st));   // the stage and the token slot are free once these MMAs have read them
            tc_commit(xempty(js));
        }
        tc_commit(done);            // all MMAs issued by this thread are complete
    }
    __syncwarp();

    // ---- epilogue: TMEM -> registers; warp w owns weight rows 32w..32w+31
    if (!mbar_wait(done, 0, err)) ok = false;
    __syncwarp();   // tcgen05.ld is warp-collective: reconverge after the wait loop
    tc_fence_after();
    float acc[GEMM_TOK];
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll
    for (int c = 0; c < GEMM_TOK / 16; ++c)
        if (c * 16 < M) tmem_ld16(trow + c * 16, acc + c * 16);
    tmem_ld_wait();

    const int n = tile * GEMM_BN + warp * 32 + lane;
    const bool live = n < N;
    if (cluster_combine) {
        // The S segments of this tile form one cluster.  Each CTA parks its partial in its own
        // shared memory (the drained stage ring) as [m][row]; after a cluster barrier, CTA q
        // finishes the contiguous rows [q*128/S, (q+1)*128/S) by reading every segment's partial
        // over DSMEM and adding them in segment order 0..S-1 — the same sum, in the same order,
        // as the workspace path below, so the bits do not depend on the path.  Consecutive
        // threads take consecutive rows: conflict-free DSMEM reads, coalesced stores.
        float* pbuf = reinterpret_cast<float*>(smem);
        const int r_local = warp * 32 + lane;
#pragma unroll
        for (int m = 0; m < GEMM_TOK; ++m)
            if (m < M) pbuf[m * GEMM_BN + r_local] = acc[m];
        __syncwarp();
        cluster_sync();
        const uint32_t q = cluster_ctarank();
        const int r0 = static_cast<int>(q) * GEMM_BN / S, r1 = (static_cast<int>(q) + 1) * GEMM_BN / S;
        const int nr = r1 - r0;
        const int total = nr * M;
        const uint32_t pbase = smem_u32(pbuf);
        // 8 elements per thread per batch, all their DSMEM loads in flight together
        for (int e0 = threadIdx.x; e0 < total; e0 += 8 * blockDim.x) {
            float v[8][CLUSTER_MAX];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = e0 + j * blockDim.x;
                const int r = r0 + e % nr, m = e / nr;
                const uint32_t off = static_cast<uint32_t>((m * GEMM_BN + r) * 4);
#pragma unroll
                for (int s2 = 0; s2 < CLUSTER_MAX; ++s2)
                    v[j][s2] = (e < total && s2 < S) ? ld_dsmem(mapa_shared(pbase + off, s2)) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = e0 + j * blockDim.x;
                if (e >= total) continue;
                const int r = r0 + e % nr, m = e / nr;
                float sum = v[j][0];
#pragma unroll
                for (int s2 = 1; s2 < CLUSTER_MAX; ++s2)
                    if (s2 < S) sum = __fadd_rn(sum, v[j][s2]);
                const int row = tile * GEMM_BN + r;
                if (row < N) {
                    const size_t o = static_cast<size_t>(m) * ldy + row;
                    if (F32OUT) static_cast<float*>(Y)[o] = sum;
                    else static_cast<uint16_t*>(Y)[o] = f32_to_bf16(sum);
                }
            }
        }
        __syncwarp();
        cluster_sync();   // no CTA leaves while a peer may still read its shared memory
    } else if (GATED) {
        // rows 0..63 of the tile are the gate rows of features 64 tile + 0..63, rows 64..127 the
        // up rows of the same features: every warp parks its rows rounded to bf16 (as a stored
        // gate/up row would be) in shared memory (the drained stage ring), then the CTA forms the
        // M x 64 activations, consecutive threads on consecutive features.  The loop is kept
        // short (unrolled by 4): fully unrolled over the 64 token rows, each with an exp, it was
        // measured 3-6 us slower per launch, its code streaming through the instruction cache.
        uint16_t* gbuf = reinterpret_cast<uint16_t*>(smem);   // [m][128]: gate rows, then up rows
        const int r_local = warp * 32 + lane;
#pragma unroll
        for (int m = 0; m < GEMM_TOK; ++m)
            if (m < M) gbuf[m * GEMM_BN + r_local] = f32_to_bf16(acc[m]);
        __syncthreads();
        const int F = N >> 1;
#pragma unroll 4
        for (int e = threadIdx.x; e < M * 64; e += blockDim.x) {
            const int m = e >> 6, fl = e & 63, f = tile * 64 + fl;
            if (f < F) {
                const float g = bf16_to_f32(gbuf[m * GEMM_BN + fl]);
                const float u = bf16_to_f32(gbuf[m * GEMM_BN + 64 + fl]);
                static_cast<uint16_t*>(Y)[static_cast<size_t>(m) * ldy + f] = f32_to_bf16(swiglu_f(g, u));
            }
        }
    } else if (S == 1) {
        if (live && Y) {
#pragma unroll
            for (int m = 0; m < GEMM_TOK; ++m) {
                if (m < M) {
                    if (F32OUT) static_cast<float*>(Y)[static_cast<size_t>(m) * ldy + n] = acc[m];
                    else static_cast<uint16_t*>(Y)[static_cast<size_t>(m) * ldy + n] = f32_to_bf16(acc[m]);
                }
            }
        }
        if (F32OUT && amax) {
            // the tile's (max, lowest index) of every token row, for the argmax: rows parked in
            // shared memory (the drained stage ring), then warp w reduces token rows w, w + 4, ...
            // (value, -index) is a total order (a NaN never wins), so the final argmax over the
            // tiles equals that of the whole row whatever the grouping
            float* vbuf = reinterpret_cast<float*>(smem);   // [m][128]
#pragma unroll
            for (int m = 0; m < GEMM_TOK; ++m)
                if (m < M) vbuf[m * GEMM_BN + warp * 32 + lane] = acc[m];
            __syncthreads();
#pragma unroll 1
            for (int m = warp; m < M; m += 4) {
                float bv = -INFINITY;
                int bi = 0x7fffffff;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int r = q * 32 + lane, row = tile * GEMM_BN + r;
                    const float v = vbuf[m * GEMM_BN + r];
                    if (row < N && (v > bv || (v == bv && row < bi))) { bv = v; bi = row; }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                    if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
                }
                if (lane == 0) amax[static_cast<size_t>(m) * gridDim.x + tile] = make_float2(bv, __int_as_float(bi));
            }
        }
    } else if (!cnt) {
        // the partials are combined by gemm_combine_kernel, launched next on the stream
        if (live) {
#pragma unroll
            for (int m = 0; m < GEMM_TOK; ++m)
                if (m < M) part[(static_cast<size_t>(seg) * M + m) * N + n] = acc[m];
        }
    } else {
        if (live) {
#pragma unroll
            for (int m = 0; m < GEMM_TOK; ++m)
                if (m < M) part[(static_cast<size_t>(seg) * M + m) * N + n] = acc[m];
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) s_last = (atomicAdd(&cnt[tile], 1u) == static_cast<unsigned>(S - 1));
        __syncthreads();
        if (s_last) {
            __threadfence();
            if (live) {
                // r = p_0 + p_1 + ... + p_{S-1} in segment order (this CTA's own partial is read
                // back too, so every load is unconditional).  Rows go in batches of 8 and the
                // loads of up to 8 segments are issued together before any add, so a batch
                // costs one round trip to L2 per 8 segments.
                for (int mc = 0; mc < M; mc += 8) {
                    float r[8];
                    for (int sg = 0; sg < S; sg += 8) {
                        float v[8][8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float* ps = part + (static_cast<size_t>(sg + q) * M + mc) * N + n;
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                v[q][j] = (sg + q < S && mc + j < M) ? __ldcg(ps + static_cast<size_t>(j) * N) : 0.f;
                        }
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            if (sg + q < S) {
#pragma unroll
                                for (int j = 0; j < 8; ++j) r[j] = (sg + q == 0) ? v[q][j] : __fadd_rn(r[j], v[q][j]);
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (mc + j < M) {
                            const size_t o = static_cast<size_t>(mc + j) * ldy + n;
                            if (F32OUT) static_cast<float*>(Y)[o] = r[j];
                            else static_cast<uint16_t*>(Y)[o] = f32_to_bf16(r[j]);
                        }
                    }
                }
            }
            if (threadIdx.x == 0) cnt[tile] = 0u;   // every segment has arrived: ready for the next call
        }
    }
    (void)ok;

    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// Y[m][n] = p_0 + p_1 + ... + p_{S-1} (segment order, the sum of the in-kernel combines) of the
// partials part[(seg*M + m)*N + n]; one thread per output, every segment's load in flight at once.
constexpr int COMBINE_THREADS = 256;
template <bool F32OUT>
__global__ void __launch_bounds__(COMBINE_THREADS)
    gemm_combine_kernel(const float* __restrict__ part, void* __restrict__ Y, int ldy, int M, int N, int S) {
    griddep_launch();
    griddep_wait();
    const long long idx = static_cast<long long>(blockIdx.x) * COMBINE_THREADS + threadIdx.x;
    if (idx >= static_cast<long long>(M) * N) return;
    const int m = static_cast<int>(idx / N), n = static_cast<int>(idx % N);
    float v[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) v[q] = q < S ? __ldcg(part + (static_cast<size_t>(q) * M + m) * N + n) : 0.f;
    float r = v[0];
#pragma unroll
    for (int q = 1; q < 16; ++q)
        if (q < S) r = __fadd_rn(r, v[q]);
    const size_t o = static_cast<size_t>(m) * ldy + n;
    if (F32OUT) static_cast<float*>(Y)[o] = r;
    else static_cast<uint16_t*>(Y)[o] = f32_to_bf16(r);
}

inline int num_tiles(int N) { return ceil_div(N, GEMM_BN); }
inline size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

// Shapes with more tiles than SMs stay whole; shapes of one to two SMs' worth split K in two;
// narrow shapes split K to fill one wave of 2 CTAs per SM, with at least 8 K-blocks per segment.
// Measured on GB300 with tiled weights, the verify step (B = 1 / B = 8, context 2183): the
// 34816-wide gate/up and the LM head whole instead of in two halves 865 -> 819 / 1006 -> 918 us
// (a CTA streams one contiguous run of its whole tile row, and no combine); the GDN output
// projection (N = 5120, K = 4096) in 7 segments (9 K-blocks each) instead of 4 and the attention
// output projection (K = 6144) in 7 instead of 6, now that their partials go to the residual
// RMSNorm: -3.5 / -2 us (in 4 segments, while the last CTA of a tile still combined them, the
// GDN output projection had been 5 us faster than in 7); the input
// projections (97 and 112 tiles) whole +18 us, in 3 segments +9..+24 us; the down projection in
// 6 or 7 segments the same, in 8 (a second wave) +67 us.  (With row-major weights the two-way
// splits of the wide shapes had been the faster choice.)
int gemm_splits(int N, int K) {
    const int tiles = num_tiles(N);
    const int nkb = ceil_div(K, GEMM_BK);
    int s;
    if (tiles > SM_COUNT_TARGET) {
        s = 1;
    } else if (2 * tiles > SM_COUNT_TARGET) {
        s = 2;
    } else {
        s = (SM_COUNT_TARGET * RESIDENT_PER_SM) / tiles;
        if (s > 16) s = 16;
    }
    while (s > 1 && nkb / s < MIN_SEGMENT_KB) --s;
    return s;
}

// Workspace layout: [tile counters, COUNTER_BYTES at offset 0][segment partials].
// The counters sit at the same place for every shape, so one zeroed workspace
// can serve GEMMs of different shapes in turn (each call leaves them zero).
// A split GEMM has at most SM_COUNT_TARGET * RESIDENT_PER_SM / 2 tiles.
constexpr size_t COUNTER_BYTES = GEMM_COUNTER_BYTES;
static_assert(COUNTER_BYTES / sizeof(unsigned) >= SM_COUNT_TARGET * RESIDENT_PER_SM / 2, "counter region too small");
// The largest scratch need: a split shape has S * tiles <= SM_COUNT_TARGET * RESIDENT_PER_SM and
// N <= tiles * GEMM_BN, so its partials take at most M_MAX * 4 bytes * that many tiles' columns;
// the allocation-free entry point's fixed array must hold it for every M <= XV_GEMM_M_MAX.
static_assert(COUNTER_BYTES + 256 + static_cast<size_t>(XV_GEMM_M_MAX) * sizeof(float) * SM_COUNT_TARGET *
                                          RESIDENT_PER_SM * GEMM_BN <=
                  XV_GEMM_NOALLOC_SCRATCH_BYTES,
              "the allocation-free scratch array is smaller than the largest split-K need");

bool gemm_uses_counters(int M, int N, int K) { return gemm_splits(N, K) > CLUSTER_MAX && M <= X_SMALL_M; }

size_t gemm_workspace_size(int M, int N, int K) {
    const int S = gemm_splits(N, K);
    if (S <= CLUSTER_MAX) return 0;
    return COUNTER_BYTES + round256(static_cast<size_t>(S) * M * N * sizeof(float));
}

xv_status gemm_launch(const uint16_t* X, int ldx, const uint16_t* W, WLayout wl, void* Y, int ldy, bool f32out, int M,
                      int N, int K, void* ws, size_t ws_bytes, cudaStream_t s, float** defer_part, int* defer_S,
                      float2* amax) {
    (void)ws_bytes;
    const bool wtiled = wl != W_ROWS, gated = wl == W_GATED;
    if (gated && (f32out || N % 128))
        return fail(XV_ERR_UNSUPPORTED, "gemm: the fused SwiGLU needs bf16 out and a multiple of 64 features");
    if (amax && (!f32out || gemm_splits(N, K) != 1))
        return fail(XV_ERR_UNSUPPORTED, "gemm: argmax partials need fp32 out and an unsplit shape");
    if (!Y && !amax) return fail(XV_ERR_ARG, "gemm: null Y");
    if (defer_part) *defer_part = nullptr;
    unsigned* err = device_error_word();
    if (!err) return fail(XV_ERR_CUDA, "gemm: device error word unavailable");
    CUtensorMap tmW, tmX;
    {
        // tiled: a [tiles * nkb * 128, 64] array of 128-byte rows; row-major: [N, K]
        const uint64_t rows = static_cast<uint64_t>(num_tiles(N)) * ceil_div(K, GEMM_BK) * GEMM_BN;
        const uint64_t dims[2] = {wtiled ? static_cast<uint64_t>(GEMM_BK) : static_cast<uint64_t>(K),
                                  wtiled ? rows : static_cast<uint64_t>(N)};
        const uint64_t strides[1] = {wtiled ? static_cast<uint64_t>(GEMM_BK) * 2 : static_cast<uint64_t>(K) * 2};
        const uint32_t box[2] = {GEMM_BK, GEMM_BN};
        if (xv_status st = encode_tiled(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, dims, strides, box,
                                        CU_TENSOR_MAP_SWIZZLE_128B))
            return st;
    }
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
        const uint64_t strides[1] = {static_cast<uint64_t>(ldx) * 2};
        const uint32_t box[2] = {GEMM_BK, static_cast<uint32_t>(M <= X_SMALL_M ? X_SMALL_M : GEMM_TOK)};
        if (xv_status st = encode_tiled(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, dims, strides, box,
                                        CU_TENSOR_MAP_SWIZZLE_128B))
            return st;
    }
    const int tiles = num_tiles(N), S = gated ? 1 : gemm_splits(N, K), nkb = ceil_div(K, GEMM_BK);
    float* part = nullptr;
    unsigned* cnt = nullptr;
    // Past 8 token rows the last-arriving CTA's combine is a long serial tail (one round trip per
    // 8 rows); a separate kernel with a thread per output combines them in one round trip.  A
    // caller that can take the partials itself (the residual RMSNorm after the output and down
    // projections) always does: measured in the verify step at 8 rows, the last-arriving CTA's
    // combine (fence, counter, then its partial loads queued behind the next GEMM's early weight
    // loads) took 5-7 us after the last MMAs, and handing the partials on took the step from
    // 805 to 795 us.
    const bool sep_combine = S > CLUSTER_MAX && (M > X_SMALL_M || defer_part != nullptr);
    if (S > CLUSTER_MAX) {
        cnt = sep_combine ? nullptr : static_cast<unsigned*>(ws);
        part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + COUNTER_BYTES);
    }
    auto kern = gated ? gemm_small_m_kernel<false, true>
                      : (f32out ? gemm_small_m_kernel<true, false> : gemm_small_m_kernel<false, false>);
    if (xv_status st = kernel_smem_once(reinterpret_cast<const void*>(kern), SMEM_MAX, false, "gemm: set shared memory size"))
        return st;
    const int xb = M <= X_SMALL_M ? 1024 : B_BYTES, xr = M <= X_SMALL_M ? X_RING : STAGES;
    const int smem = smem_bytes(xb, xr);
    dim3 grid(tiles, S);
    const int cluster = (S > 1 && S <= CLUSTER_MAX) ? 1 : 0;
    trace_pre(s);
    if (cluster)
        launch_k_cluster(kern, grid, dim3(128), smem, s, dim3(1, S, 1), tmW, tmX, Y, ldy, M, N, nkb, S, part, cnt,
                         err, cluster, xb, xr, wtiled ? 1 : 0, amax);
    else
        launch_k(kern, grid, dim3(128), smem, s, tmW, tmX, Y, ldy, M, N, nkb, S, part, cnt, err, cluster, xb, xr,
                 wtiled ? 1 : 0, amax);
    const long long bytes = 2ll * N * K + 2ll * M * K +
                            (Y ? static_cast<long long>(M) * (gated ? N / 2 : N) * (f32out ? 4 : 2) : 0) +
                            (amax ? 8ll * M * tiles : 0);
    if (xv_status st = launched("gemm_small_m_kernel", s, K_GEMM, bytes)) return st;
    if (sep_combine && defer_part) {
        *defer_part = part;
        if (defer_S) *defer_S = S;
        return XV_OK;
    }
    if (sep_combine) {
        trace_pre(s);
        const long long outs = static_cast<long long>(M) * N;
        auto ck = f32out ? gemm_combine_kernel<true> : gemm_combine_kernel<false>;
        launch_k(ck, dim3(ceil_div(outs, COMBINE_THREADS)), dim3(COMBINE_THREADS), 0, s, part, Y, ldy, M, N, S);
        return launched("gemm_combine_kernel", s, K_GEMM_COMBINE, 4ll * S * outs + outs * (f32out ? 4 : 2));
    }
    return XV_OK;
}

namespace {
// One thread per 16 bytes of the tiled array (8 elements of a tile row): element c of row r of
// tile (t, kb) is W[128 t + r][64 kb + c], zero past N or K (K % 8 == 0, so a 16-byte piece lies
// wholly inside or wholly outside W).  Consecutive threads write consecutive pieces; 8 of them
// read one 128-byte piece of a weight row.
__global__ void tile_weights_kernel(const uint4* __restrict__ W, int N, int K, int nkb, long long pieces, int gate_f,
                                    uint4* __restrict__ Wt) {
    griddep_launch();
    griddep_wait();
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= pieces) return;
    const int c8 = static_cast<int>(i & 7);
    const int r = static_cast<int>((i >> 3) & (GEMM_BN - 1));
    const long long blk = i >> 10;   // (t, kb) block: 128 rows x 8 pieces
    const int kb = static_cast<int>(blk % nkb);
    const long long t = blk / nkb;
    // gated (gate_f = F features): rows 0..63 of tile t are gate rows 64 t + r, rows 64..127 the
    // up rows F + 64 t + r - 64
    const long long row = gate_f ? (r < 64 ? t * 64 + r : gate_f + t * 64 + r - 64) : t * GEMM_BN + r;
    const int col = kb * GEMM_BK + c8 * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < N && col < K) v = W[(row * K + col) / 8];
    Wt[i] = v;
}

// Enqueued right after a tiling with a plain launch (no programmatic serialisation): it starts
// only once the tiled weights are complete in memory, and it lets its successor start only when
// it has exited.  Every GEMM requests its first weight tiles before its dependency wait (weights
// are not written by the kernel before it), so this is what keeps a GEMM launched straight after
// a tiling from reading tiles still being written.
__global__ void tile_fence_kernel() {}
}  // namespace

size_t gemm_tiled_bytes(int N, int K) {
    return static_cast<size_t>(num_tiles(N)) * ceil_div(K, GEMM_BK) * GEMM_BN * GEMM_BK * 2;
}

xv_status gemm_tile_weights_launch(const uint16_t* W, int N, int K, bool gated, uint16_t* Wt, cudaStream_t s) {
    const long long pieces = static_cast<long long>(gemm_tiled_bytes(N, K) / 16);
    constexpr int T = 256;
    trace_pre(s);
    launch_k(tile_weights_kernel, dim3(static_cast<unsigned>((pieces + T - 1) / T)), dim3(T), 0, s,
             reinterpret_cast<const uint4*>(W), N, K, ceil_div(K, GEMM_BK), pieces, gated ? N / 2 : 0,
             reinterpret_cast<uint4*>(Wt));
    if (xv_status e = launched("tile_weights_kernel", s, K_TILE, 2 * static_cast<long long>(gemm_tiled_bytes(N, K))))
        return e;
    trace_pre(s);
    tile_fence_kernel<<<1, 32, 0, s>>>();
    return launched("tile_fence_kernel", s, K_TILE, 0);
}

}  // namespace xv
