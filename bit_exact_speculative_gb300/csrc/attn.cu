// Decode-row attention over a bf16 KV cache, and the KV append of a verify block.
//
// "Follow-up to my earlier post on Qwen3.8-27B decode speed" (r/LocalLLaMA
// post): verify attention must run as decode rows, one per draft position.
// Here every row — a decode token or draft position r of a verify block — is
// computed by exactly the same sequence of operations, determined by its own
// length alone:
//   - positions are cut into splits of ATTN_SPLIT tokens at fixed absolute
//     boundaries, and each split into tiles of 64 positions;
//   - inside a split, an fp32 online softmax (log2 domain) runs over the
//     split's tiles in order; a tile or position past the row's length is
//     masked to -inf, contributes p = 0, and leaves the running max, sum and
//     output bit-for-bit unchanged (correction factor exp2(0) = 1);
//   - the splits 0..ceil(len/ATTN_SPLIT)-1 are combined in split order by a
//     second kernel.
// The rows of a verify block share the K/V tiles (loaded once per CTA, for
// all q heads of a kv head and all R rows), but no arithmetic of one row
// touches another row's data: each output element of a tensor-core product
// is the dot product of its own row and column.
//
// Kernel 1 (attn_split_kernel), one CTA per (split, kv head, sequence):
// K and V tiles arrive by TMA (3-D tensor map over [pages*Hkv, page, hd], 128-byte
// swizzle; a contiguous cache is one page of Lmax positions per sequence, a
// paged one pages of a multiple of 64 positions, so a tile never straddles two
// pages and the page a tile comes from changes nothing in its arithmetic)
// into a 3-stage shared-memory ring; QK^T and PV run on mma.sync
// m16n8k16 bf16 -> fp32 with P rounded to bf16; one warp owns 16 query rows.
// Kernel 2 (attn_combine_kernel), one CTA per (row, q head): fixed-order
// split combine, normalisation, optional output gate, bf16 store.
#include <cmath>

#include "xv_internal.h"
#include "xv_ptx.cuh"

namespace xv {

namespace {
constexpr int T = ATTN_TILE;
constexpr float NEG_INF = -INFINITY;

// Page of position p of sequence b (row *row inside it); an entry outside the pool is
// recorded and replaced by page 0, so no copy leaves the pool.  p < page * max_pages.
__device__ __forceinline__ int kv_page(const KvPages& kv, int b, int p, int* row, unsigned* err) {
    if (!kv.table) {
        *row = p;
        return b;
    }
    const int j = p / kv.page;
    *row = p - j * kv.page;
    int pg = kv.table[static_cast<long long>(b) * kv.max_pages + j];
    if (pg < 0 || pg >= kv.n_pages) {
        atomicOr(err, ERR_BAD_PAGE);
        pg = 0;
    }
    return pg;
}

template <int HD>
struct AttnShape {
    static constexpr int CB = HD / 64;                   // 128-byte column blocks per row
    static constexpr int TILE_BYTES = T * HD * 2;        // one K or V tile
    static constexpr int STAGES = HD == 256 ? 3 : 4;
    static constexpr int RING_BYTES = STAGES * 2 * TILE_BYTES;
    static int smem_bytes(int rows_pad) { return 1024 + RING_BYTES + rows_pad * HD * 2 + 8 * STAGES + 64; }
};

struct AttnArgs {
    const uint16_t* q;
    long long q_stride;
    KvPages kv;
    const int32_t* ctx_len;
    int len_bias;
    int R, G, Hq, Hkv, nsplit, max_len;
    float sl2;          // scale * log2(e)
    float* opart;       // [B*R*Hq][nsplit][HD]
    float2* ml;         // [B*R*Hq][nsplit] (running max in log2 units, sum)
    unsigned* err;
};

template <int HD>
__global__ void __launch_bounds__(128, 1)
    attn_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnArgs A) {
    griddep_launch();
    griddep_wait();
    using S = AttnShape<HD>;
    constexpr int CB = S::CB, STAGES = S::STAGES, TILE_BYTES = S::TILE_BYTES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const int nw = blockDim.x >> 5;
    const int rows_pad = nw * 16;
    const uint32_t sQ = base + S::RING_BYTES;
    const uint32_t bar0 = sQ + rows_pad * HD * 2;
    auto sK = [&](int st) { return base + st * 2 * TILE_BYTES; };
    auto sV = [&](int st) { return base + st * 2 * TILE_BYTES + TILE_BYTES; };
    auto full = [&](int st) { return bar0 + 8u * st; };

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rows = A.R * A.G;
    const int L0 = A.ctx_len[b] + A.len_bias;     // visible length of row 0
    const int maxlen = L0 + A.R - 1;
    if (L0 < 1 || maxlen > A.max_len) {
        if (tid == 0 && split == 0 && g == 0) atomicOr(A.err, ERR_BAD_LENGTH);
        return;
    }
    const int p_begin = split * ATTN_SPLIT;
    if (p_begin >= maxlen) return;
    const int p_end = min(p_begin + ATTN_SPLIT, maxlen);
    const int ntiles = (p_end - p_begin + T - 1) / T;

    // page and row of every tile of the split, looked up once by thread 0 (all loads in flight together)
    __shared__ int tile_z[ATTN_SPLIT / T], tile_row[ATTN_SPLIT / T];
    auto issue = [&](int i) {
        const int st = i % STAGES;
        mbar_arrive_expect_tx(full(st), 2 * TILE_BYTES);
        const int z = tile_z[i], row = tile_row[i];
#pragma unroll
        for (int cb = 0; cb < CB; ++cb) {
            tma_load_3d(sK(st) + cb * T * 128, &tmK, cb * 64, row, z, full(st));
            tma_load_3d(sV(st) + cb * T * 128, &tmV, cb * 64, row, z, full(st));
        }
    };
    int issued = 0;   // tiles whose copies thread 0 has started
    if (tid == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
#pragma unroll
        for (int i = 0; i < ATTN_SPLIT / T; ++i) {
            if (i < ntiles) {
                int row;
                tile_z[i] = kv_page(A.kv, b, p_begin + i * T, &row, A.err) * A.Hkv + g;
                tile_row[i] = row;
            }
        }
        for (int st = 0; st < STAGES; ++st) mbar_init(full(st), 1);
        fence_mbar_init();
        for (; issued < STAGES && issued < ntiles; ++issued) issue(issued);
    }
    // Q rows (r, gh) -> tile row r*G + gh, 16-byte chunks XOR-swizzled by row
    for (int idx = tid; idx < rows_pad * (HD / 8); idx += blockDim.x) {
        const int row = idx / (HD / 8), ch = idx % (HD / 8);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < rows) {
            const int r = row / A.G, h = g * A.G + row % A.G;
            v = *reinterpret_cast<const uint4*>(A.q + (static_cast<long long>(b) * A.R + r) * A.q_stride +
                                                static_cast<long long>(h) * HD + ch * 8);
        }
        *reinterpret_cast<uint4*>(smem + (sQ - base) + row * HD * 2 + ((ch ^ (row & 7)) * 16)) = v;
    }
    __syncthreads();

    const int rho0 = warp * 16 + (lane >> 2), rho1 = rho0 + 8;
    const int len0 = rho0 < rows ? L0 + rho0 / A.G : 0;
    const int len1 = rho1 < rows ? L0 + rho1 / A.G : 0;
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
    float O[HD / 8][4];
#pragma unroll
    for (int j = 0; j < HD / 8; ++j) O[j][0] = O[j][1] = O[j][2] = O[j][3] = 0.f;

    bool ok = true;
    for (int i = 0; i < ntiles; ++i) {
        const int st = i % STAGES;
        if (!mbar_wait(full(st), (i / STAGES) & 1u, A.err)) { ok = false; }
        if (!__syncthreads_and(ok)) { ok = false; break; }
        const int p0 = p_begin + i * T;
        if (p0 + T > maxlen) {
            // positions past every row's length: zero V so that p = 0 never meets a non-finite value
            const int first = maxlen - p0;
            for (int idx = tid; idx < (T - first) * CB * 8; idx += blockDim.x) {
                const int prow = first + idx / (CB * 8), rem = idx % (CB * 8);
                *reinterpret_cast<uint4*>(smem + (sV(st) - base) + (rem >> 3) * T * 128 + prow * 128 + (rem & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
            }
            __syncthreads();
        }

        // ---- S = Q K^T for this warp's 16 rows and the tile's 64 positions
        float sacc[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll 4
        for (int ks = 0; ks < HD / 16; ++ks) {
            uint32_t a0, a1, a2, a3;
            {
                const int qr = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int qc = ks * 2 + (lane >> 4);
                ldsm_x4(sQ + qr * HD * 2 + ((qc ^ (qr & 7)) * 16), a0, a1, a2, a3);
            }
            const int chunk = ks * 2 + ((lane >> 3) & 1);
            const int cb = chunk >> 3, cic = chunk & 7;
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                const int pos = np * 16 + (lane & 7) + ((lane >> 4) << 3);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sK(st) + cb * T * 128 + pos * 128 + ((cic ^ (pos & 7)) * 16), b0, b1, b2, b3);
                mma_16816(sacc[2 * np], a0, a1, a2, a3, b0, b1);
                mma_16816(sacc[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }

        // ---- online softmax (row stats held by the 4 lanes of a quad)
        float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int pos = p0 + nt * 8 + 2 * (lane & 3) + j;
                const float v0 = pos < len0 ? __fmul_rn(sacc[nt][j], A.sl2) : NEG_INF;
                const float v1 = pos < len1 ? __fmul_rn(sacc[nt][2 + j], A.sl2) : NEG_INF;
                sacc[nt][j] = v0;
                sacc[nt][2 + j] = v1;
                mx0 = fmaxf(mx0, v0);
                mx1 = fmaxf(mx1, v1);
            }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const bool dead0 = mn0 == NEG_INF, dead1 = mn1 == NEG_INF;
        const float al0 = dead0 ? 1.f : exp2f(__fsub_rn(m0, mn0));
        const float al1 = dead1 ? 1.f : exp2f(__fsub_rn(m1, mn1));
        float ts0 = 0.f, ts1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float p0v = dead0 ? 0.f : exp2f(__fsub_rn(sacc[nt][j], mn0));
                const float p1v = dead1 ? 0.f : exp2f(__fsub_rn(sacc[nt][2 + j], mn1));
                sacc[nt][j] = p0v;
                sacc[nt][2 + j] = p1v;
                ts0 = __fadd_rn(ts0, p0v);
                ts1 = __fadd_rn(ts1, p1v);
            }
        }
        l0 = __fadd_rn(__fmul_rn(l0, al0), ts0);
        l1 = __fadd_rn(__fmul_rn(l1, al1), ts1);
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int j = 0; j < HD / 8; ++j) {
            O[j][0] = __fmul_rn(O[j][0], al0);
            O[j][1] = __fmul_rn(O[j][1], al0);
            O[j][2] = __fmul_rn(O[j][2], al1);
            O[j][3] = __fmul_rn(O[j][3], al1);
        }

        // ---- O += P V  (P rounded to bf16)
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
            const uint32_t a0 = pack_bf16x2(sacc[2 * kp][0], sacc[2 * kp][1]);
            const uint32_t a1 = pack_bf16x2(sacc[2 * kp][2], sacc[2 * kp][3]);
            const uint32_t a2 = pack_bf16x2(sacc[2 * kp + 1][0], sacc[2 * kp + 1][1]);
            const uint32_t a3 = pack_bf16x2(sacc[2 * kp + 1][2], sacc[2 * kp + 1][3]);
            const int pos = kp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int dp = 0; dp < HD / 16; ++dp) {
                const int chunk = dp * 2 + (lane >> 4);
                const int cb = chunk >> 3, cic = chunk & 7;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(sV(st) + cb * T * 128 + pos * 128 + ((cic ^ (pos & 7)) * 16), b0, b1, b2, b3);
                mma_16816(O[2 * dp], a0, a1, a2, a3, b0, b1);
                mma_16816(O[2 * dp + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncthreads();   // every warp is done with stage st
        if (tid == 0 && i + STAGES < ntiles) {
            fence_proxy_async_smem();
            issue(i + STAGES);
            ++issued;
        }
    }
    if (!ok) {
        // drain copies still in flight before the CTA leaves
        if (tid == 0)
            for (int j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j)
                mbar_wait(full(j % STAGES), (j / STAGES) & 1u, A.err);
        return;
    }

    l0 = __fadd_rn(l0, __shfl_xor_sync(0xffffffffu, l0, 1));
    l0 = __fadd_rn(l0, __shfl_xor_sync(0xffffffffu, l0, 2));
    l1 = __fadd_rn(l1, __shfl_xor_sync(0xffffffffu, l1, 1));
    l1 = __fadd_rn(l1, __shfl_xor_sync(0xffffffffu, l1, 2));

#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int rho = half ? rho1 : rho0;
        const int len = half ? len1 : len0;
        if (rho >= rows || len <= p_begin) continue;
        const int r = rho / A.G, h = g * A.G + rho % A.G;
        const long long idx = ((static_cast<long long>(b) * A.R + r) * A.Hq + h) * A.nsplit + split;
        float* op = A.opart + idx * HD;
#pragma unroll
        for (int j = 0; j < HD / 8; ++j)
            *reinterpret_cast<float2*>(op + j * 8 + 2 * (lane & 3)) =
                half ? make_float2(O[j][2], O[j][3]) : make_float2(O[j][0], O[j][1]);
        if ((lane & 3) == 0) A.ml[idx] = half ? make_float2(m1, l1) : make_float2(m0, l0);
    }
}

struct CombineArgs {
    const int32_t* ctx_len;
    int len_bias, R, Hq, nsplit, max_len, hd;
    const float* opart;
    const float2* ml;
    const uint16_t* gate;
    long long gate_stride;
    uint16_t* out;
    long long out_stride;
    unsigned* err;
};

// One CTA per (row, q head); thread t owns output elements 2t and 2t+1.
__global__ void attn_combine_kernel(CombineArgs C) {
    griddep_launch();
    griddep_wait();
    const int hq = blockIdx.x % C.Hq;
    const long long br = blockIdx.x / C.Hq;
    const int b = static_cast<int>(br / C.R), r = static_cast<int>(br % C.R);
    const int len = C.ctx_len[b] + C.len_bias + r;
    if (len < 1 || len - r + C.R - 1 > C.max_len) return;   // reported by the split kernel
    const int ns = (len + ATTN_SPLIT - 1) / ATTN_SPLIT;
    const long long idx0 = (br * C.Hq + hq) * C.nsplit;
    float M = NEG_INF;
#pragma unroll 8
    for (int s = 0; s < ns; ++s) M = fmaxf(M, C.ml[idx0 + s].x);
    const int d = 2 * threadIdx.x;
    float L = 0.f, acc0 = 0.f, acc1 = 0.f;
    // chunks of CH splits: every load of a chunk is issued before its adds, which stay in split order
    constexpr int CH = 16;
    for (int s0 = 0; s0 < ns; s0 += CH) {
        float2 ml[CH], o[CH];
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const int s = s0 + j < ns ? s0 + j : ns - 1;
            ml[j] = C.ml[idx0 + s];
            o[j] = *reinterpret_cast<const float2*>(C.opart + (idx0 + s) * C.hd + d);
        }
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            if (s0 + j < ns) {
                const float w = exp2f(__fsub_rn(ml[j].x, M));
                L = __fadd_rn(L, __fmul_rn(w, ml[j].y));
                acc0 = __fadd_rn(acc0, __fmul_rn(w, o[j].x));
                acc1 = __fadd_rn(acc1, __fmul_rn(w, o[j].y));
            }
        }
    }
    float y0 = __fdiv_rn(acc0, L), y1 = __fdiv_rn(acc1, L);
    if (C.gate) {
        const uint16_t* gp = C.gate + br * C.gate_stride + static_cast<long long>(hq) * C.hd + d;
        const float g0 = bf16_to_f32(gp[0]), g1 = bf16_to_f32(gp[1]);
        const float s0 = __frcp_rn(__fadd_rn(1.f, expf(-g0)));
        const float s1 = __frcp_rn(__fadd_rn(1.f, expf(-g1)));
        y0 = __fmul_rn(bf16_to_f32(f32_to_bf16(y0)), s0);
        y1 = __fmul_rn(bf16_to_f32(f32_to_bf16(y1)), s1);
    }
    uint16_t* op = C.out + br * C.out_stride + static_cast<long long>(hq) * C.hd + d;
    op[0] = f32_to_bf16(y0);
    op[1] = f32_to_bf16(y1);
}

__global__ void kv_append_kernel(const uint16_t* __restrict__ src, long long src_stride, const int32_t* __restrict__ ctx_len,
                                 int pos_bias, int R, int Hkv, int hd, KvPages kv, uint16_t* __restrict__ kc,
                                 uint16_t* __restrict__ vc, unsigned* err) {
    griddep_launch();
    griddep_wait();
    const int row = blockIdx.x, b = row / R, r = row % R;
    const int pos = ctx_len[b] + pos_bias + r;
    if (pos < 0 || pos >= kv.page * kv.max_pages) {
        if (threadIdx.x == 0) atomicOr(err, ERR_BAD_LENGTH);
        return;
    }
    int prow = pos;
    int pg = b;
    if (kv.table) {
        const int j = pos / kv.page;
        prow = pos - j * kv.page;
        pg = kv.table[static_cast<long long>(b) * kv.max_pages + j];
        if (pg < 0 || pg >= kv.n_pages) {
            if (threadIdx.x == 0) atomicOr(err, ERR_BAD_PAGE);
            return;
        }
    }
    const int chunks = Hkv * hd / 8;
    for (int c = threadIdx.x; c < 2 * chunks; c += blockDim.x) {
        const bool is_v = c >= chunks;
        const int cc = is_v ? c - chunks : c;
        const int h = cc / (hd / 8), d = (cc % (hd / 8)) * 8;
        const uint4 v = *reinterpret_cast<const uint4*>(src + row * src_stride + (is_v ? Hkv * hd : 0) + h * hd + d);
        uint16_t* dst = (is_v ? vc : kc) + ((static_cast<long long>(pg) * Hkv + h) * kv.page + prow) * hd + d;
        *reinterpret_cast<uint4*>(dst) = v;
    }
}

inline size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline int nsplit_for(int max_len) { return (max_len + ATTN_SPLIT - 1) / ATTN_SPLIT; }

template <int HD>
xv_status launch_split(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnArgs& a, int B, cudaStream_t s) {
    using S = AttnShape<HD>;
    const int rows = a.R * a.G;
    const int nw = (rows + 15) / 16;
    const int smem = S::smem_bytes(nw * 16);
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return fail(XV_ERR_CUDA, "attn: device ordinal out of range");
    if (!attr_done[dev]) {
        const int maxsm = S::smem_bytes(64);
        if (xv_status st = cuda_check(cudaFuncSetAttribute(attn_split_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, maxsm),
                                      "attn: set shared memory size"))
            return st;
        attr_done[dev] = true;
    }
    dim3 grid(a.nsplit, a.Hkv, B);
    trace_pre(s);
    launch_k(attn_split_kernel<HD>, dim3(grid), dim3(nw * 32), smem, s, tmK, tmV, a);
    // bound: every sequence at the longest length the launch is sized for
    const long long bytes = 4ll * B * a.Hkv * a.max_len * HD + 2ll * B * a.R * a.Hq * HD +
                            4ll * B * a.R * a.Hq * a.nsplit * (HD + 2);
    return launched("attn_split_kernel", s, K_ATTN_SPLIT, bytes);
}

}  // namespace

size_t attn_workspace_size(int B, int R, int Hq, int hd, int max_len) {
    const size_t rows = static_cast<size_t>(B) * R * Hq * nsplit_for(max_len);
    return round256(rows * hd * sizeof(float)) + round256(rows * sizeof(float2));
}

xv_status attn_launch(const uint16_t* q, long long q_stride, const uint16_t* kc, const uint16_t* vc, const KvPages& kv,
                      const int32_t* ctx_len, int len_bias, int R, int B, int Hq, int Hkv, int hd, int max_len,
                      float scale, const uint16_t* gate, long long gate_stride, uint16_t* out, long long out_stride,
                      void* ws, size_t ws_bytes, cudaStream_t s) {
    (void)ws_bytes;
    unsigned* err = device_error_word();
    if (!err) return fail(XV_ERR_CUDA, "attn: device error word unavailable");
    CUtensorMap tmK, tmV;
    const uint64_t dims[3] = {static_cast<uint64_t>(hd), static_cast<uint64_t>(kv.page),
                              static_cast<uint64_t>(kv.n_pages) * Hkv};
    const uint64_t strides[2] = {static_cast<uint64_t>(hd) * 2, static_cast<uint64_t>(kv.page) * hd * 2};
    const uint32_t box[3] = {64, static_cast<uint32_t>(T), 1};
    if (xv_status st = encode_tiled(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kc, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return st;
    if (xv_status st = encode_tiled(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, vc, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return st;
    const int nsplit = nsplit_for(max_len);
    const size_t rows = static_cast<size_t>(B) * R * Hq * nsplit;
    float* opart = static_cast<float*>(ws);
    float2* ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) + round256(rows * hd * sizeof(float)));
    AttnArgs a{q, q_stride, kv, ctx_len, len_bias, R, Hq / Hkv, Hq, Hkv, nsplit, max_len,
               scale * 1.4426950408889634f, opart, ml, err};
    xv_status st = hd == 256 ? launch_split<256>(tmK, tmV, a, B, s) : launch_split<64>(tmK, tmV, a, B, s);
    if (st) return st;
    CombineArgs c{ctx_len, len_bias, R, Hq, nsplit, max_len, hd, opart, ml, gate, gate_stride, out, out_stride, err};
    trace_pre(s);
    launch_k(attn_combine_kernel, dim3(B * R * Hq), dim3(hd / 2), 0, s, c);
    return launched("attn_combine_kernel", s, K_ATTN_COMBINE,
                    4ll * B * R * Hq * nsplit * (hd + 2) + 2ll * B * R * Hq * hd * (gate ? 2 : 1));
}

xv_status kv_append_launch(const uint16_t* src, long long src_stride, const int32_t* ctx_len, int pos_bias, int R, int B,
                           int Hkv, int hd, const KvPages& kv, uint16_t* kc, uint16_t* vc, cudaStream_t s) {
    unsigned* err = device_error_word();
    if (!err) return fail(XV_ERR_CUDA, "kv_append: device error word unavailable");
    trace_pre(s);
    launch_k(kv_append_kernel, dim3(B * R), dim3(128), 0, s, src, src_stride, ctx_len, pos_bias, R, Hkv, hd, kv, kc, vc, err);
    return launched("kv_append_kernel", s, K_KV_APPEND, 8ll * B * R * Hkv * hd);
}

}  // namespace xv
