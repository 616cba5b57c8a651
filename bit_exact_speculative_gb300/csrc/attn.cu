// Decode-row attention over a bf16 KV cache, and the KV append of a verify block.
//
// "Follow-up to my earlier post on Qwen3.8-27B decode speed" (r/LocalLLaMA
// post): verify attention must run as decode rows, one per draft position.
// Here every row — a decode token or draft position r of a verify block — is
// computed by exactly the same sequence of operations, determined by its own
// length alone:
//   - positions are cut into splits at fixed absolute boundaries (512
//     positions each below 4096, 2048 beyond: attn_split_begin), and each
//     split into tiles of 64 positions;
//   - inside a split, an fp32 online softmax (log2 domain) runs over the
//     split's tiles in order; a tile or position past the row's length is
//     masked to -inf, contributes p = 0, and leaves the reference max, sum and
//     output bit-for-bit unchanged;
//   - the splits 0..attn_split_count(len)-1 are combined in split order by a
//     second kernel.
// The rows of a verify block share the K/V tiles (loaded once per CTA, for
// up to 64 rows (r, q head) of a kv head; more rows take more CTAs, which
// read the same tiles through L2), but no arithmetic of one row
// touches another row's data: each output element of a tensor-core product
// is the dot product of its own row and column.
//
// Kernel 1 (attn_split_kernel), work items (split, 64-row tile, kv head, sequence):
// one CTA per item up to two waves of them, else one persistent CTA per SM
// walking a contiguous range of items.  K and V tiles arrive by TMA (3-D tensor map over [pages*Hkv, page, hd], 128-byte
// swizzle; a contiguous cache is one page of Lmax positions per sequence, a
// paged one pages of a multiple of 64 positions, so a tile never straddles two
// pages and the page a tile comes from changes nothing in its arithmetic)
// into a shared-memory ring; QK^T and PV run on tcgen05 (fp32 accumulators in
// tensor memory, bf16 operands in shared memory, P rounded to bf16); the
// softmax is one thread per query row, reading its S row from tensor memory;
// two epilogue warps read O out.
// Kernel 2 (attn_combine_kernel), one CTA per (row, q head): fixed-order
// split combine (the split partials streamed through shared memory),
// normalisation, optional output gate, bf16 store.
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

// Shared-memory plan of the split kernel (offsets from a 1024-byte aligned base):
//   Q      CB blocks of [64 rows][64 dims], 128-byte swizzle: the A operand of Q K^T.  The MMA
//          reads 128 rows: rows 64..127 of a block are the 8 KB that follow it (the next block,
//          then P), and land in TMEM lanes nobody reads
//   P[2]   [64 rows][64 positions] bf16, the A operand of P V, double-buffered (rows 64..127
//          of P[0] read P[1], of P[1] the K ring)
//   K ring SK stages of a K tile: CB blocks of [64 positions][64 dims] (B of Q K^T, K-major)
//   V ring SV stages of a V tile, same layout, read as the MN-major B operand of P V
//   barriers
template <int HD>
struct AttnShape {
    static constexpr int CB = HD / 64;                   // 128-byte column blocks per row
    static constexpr int BLK = T * 128;                  // one [64][64] bf16 block: 8 KB
    static constexpr int TILE_BYTES = CB * BLK;          // one K or V tile
    static constexpr int SK = HD == 256 ? 3 : 4;
    static constexpr int SV = HD == 256 ? 2 : 4;
    static constexpr int Q_OFF = 0;
    static constexpr int P_OFF = Q_OFF + CB * BLK;
    static constexpr int K_OFF = P_OFF + 2 * BLK;
    static constexpr int V_OFF = K_OFF + SK * TILE_BYTES;
    static constexpr int BAR_OFF = V_OFF + SV * TILE_BYTES;
    // fullK, emptyK, fullV, emptyV, vfix, sbar[2], sfree[2], pready[2], pfree[2], done, ofree, qfull,
    // mlready
    static constexpr int N_BARS = 2 * SK + 3 * SV + 12;
    static constexpr int SMEM = 1024 + BAR_OFF + 8 * N_BARS;
    static constexpr uint32_t TMEM_COLS = HD == 256 ? 512 : 256;   // S[2] (64 columns each) + O (HD)
};

struct AttnArgs {
    const uint16_t* q;
    long long q_stride;
    KvPages kv;
    const int32_t* ctx_len;
    int len_bias;
    int R, G, Hq, Hkv, nsplit, max_len, B;
    float sl2;          // scale * log2(e)
    float* opart;       // [B*R*Hq][nsplit][HD]
    float2* ml;         // [B*R*Hq][nsplit] (reference max in log2 units, sum)
    unsigned* err;
};

// warps 0-1 softmax, 2 K loads, 3 V loads, 4-5 epilogue (tensor-memory lanes 0-63, as 0-1), 6 MMA
constexpr int ATTN_THREADS = 224;
constexpr float RESCALE_SLACK = 2.f;

// A unit of work: (split, 64-row tile, kv head, sequence), numbered with the split fastest so
// that a CTA's consecutive items mostly share their Q tile.  Dead items (the split starts at or
// past every row's length, or the sequence's length is out of range) are skipped by every warp.
struct AttnItem {
    int b, g, row_base, split, L0, maxlen, p_begin, ntiles;
    bool live, bad;
};

__device__ __forceinline__ AttnItem attn_item(const AttnArgs& A, int it, int nrt) {
    AttnItem I;
    I.split = it % A.nsplit;
    int rest = it / A.nsplit;
    I.row_base = (rest % nrt) * 64;
    rest /= nrt;
    I.g = rest % A.Hkv;
    I.b = rest / A.Hkv;
    const int rows = A.R * A.G;
    I.L0 = __ldg(A.ctx_len + I.b) + A.len_bias;     // visible length of row 0
    I.bad = I.L0 < 1 || I.L0 + A.R - 1 > A.max_len;
    // the longest visible length among the item's rows; positions past a row's own length are
    // masked (p = 0), so how far the item runs does not change any row's bits
    I.maxlen = I.L0 + (min(rows, I.row_base + 64) - 1) / A.G;
    I.p_begin = attn_split_begin(I.split);
    I.live = !I.bad && I.p_begin < I.maxlen;
    I.ntiles = I.live ? (min(attn_split_begin(I.split + 1), I.maxlen) - I.p_begin + T - 1) / T : 0;
    return I;
}

// Q rows (r, gh) of an item -> block row r*G + gh, tile row r*G + gh - row_base, 16-byte chunks
// XOR-swizzled by row; rows past the block's R*G rows zero.  NT threads from t0, every load of a
// thread issued before its stores.
template <int HD, int BLK, int NT>
__device__ __forceinline__ void load_q_tile(uint8_t* sq, const AttnArgs& A, const AttnItem& I, int t0) {
    constexpr int N = 64 * (HD / 8), PER = (N + NT - 1) / NT;
    const int rows = A.R * A.G;
    uint4 v[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int idx = t0 + j * NT;
        const int row = idx / (HD / 8), ch = idx % (HD / 8);
        v[j] = make_uint4(0, 0, 0, 0);
        if (idx < N && I.row_base + row < rows) {
            const int r = (I.row_base + row) / A.G, h = I.g * A.G + (I.row_base + row) % A.G;
            v[j] = *reinterpret_cast<const uint4*>(A.q + (static_cast<long long>(I.b) * A.R + r) * A.q_stride +
                                                   static_cast<long long>(h) * HD + ch * 8);
        }
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int idx = t0 + j * NT;
        const int row = idx / (HD / 8), ch = idx % (HD / 8);
        if (idx < N) *reinterpret_cast<uint4*>(sq + (ch >> 3) * BLK + row * 128 + (((ch & 7) ^ (row & 7)) * 16)) = v[j];
    }
}

// Persistent CTAs (at most one per SM), each walking a contiguous range of items.  Per 64-position
// tile of an item:
//   MMA warp   S[t%2] = Q K_t^T on tcgen05 (M = 128 rows, N = 64 positions, fp32 in TMEM), issued
//              one tile ahead
//   softmax    thread = query row: its S row from TMEM, mask, scale; the reference max m moves
//              to the tile's max when that exceeds it by more than RESCALE_SLACK (log2 units) or
//              at the row's first live tile, and then O (TMEM) and the sum l are rescaled by
//              exp2(m_old - m_new); P = bf16(exp2(s - m)) into shared memory, l += its fp32
//              values in position order (exp2 by the hardware approximation)
//   MMA warp   O += P V_t (N = HD; V straight from its TMA stage as an MN-major operand)
//   epilogue   two warps on the softmax warps' tensor-memory lanes: once the item's last P V has
//              completed and the softmax warps have left the item's m and l in shared memory
//              (mlready), O is read out and written as the item's partials; meanwhile the softmax
//              warps are already on the next item's first S
// t counts the CTA's tiles across its items, so the K/V rings, the two S buffers and the two P
// buffers keep cycling from one item to the next; an item's first P V overwrites O once the
// epilogue warps have read the previous item's O out (ofree), and Q is reloaded (qfull) only when
// the item's (sequence, kv head, row tile) changes.  A row's operations depend on its own length
// and the absolute tile positions only, so a verify row gets the bits of the decode row at its
// position, whichever CTA and whichever neighbours it has.  MULTI = false is the launch with one
// item per CTA (CTA i takes item i), with the cross-item hand-offs compiled out.
template <int HD, bool MULTI>
__global__ void __launch_bounds__(ATTN_THREADS, 1)
    attn_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnArgs A) {
    griddep_launch();
    using S = AttnShape<HD>;
    constexpr int CB = S::CB, SK = S::SK, SV = S::SV, TILE_BYTES = S::TILE_BYTES, BLK = S::BLK;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int s_abort;
    __shared__ float2 ml_sm[64];   // (m, l) of each row of the item being written out
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const uint32_t sQ = base + S::Q_OFF, sP = base + S::P_OFF;
    auto sK = [&](int st) { return base + S::K_OFF + st * TILE_BYTES; };
    auto sV = [&](int st) { return base + S::V_OFF + st * TILE_BYTES; };
    const uint32_t bar0 = base + S::BAR_OFF;
    auto fullK = [&](int st) { return bar0 + 8u * st; };
    auto emptyK = [&](int st) { return bar0 + 8u * (SK + st); };
    auto fullV = [&](int st) { return bar0 + 8u * (2 * SK + st); };
    auto emptyV = [&](int st) { return bar0 + 8u * (2 * SK + SV + st); };
    // vfix[st]: the V rows of an item's last tile past every row's length have been zeroed in
    // stage st (one barrier per stage: two fixes of one stage are a ring turn apart, so a wait is
    // never two phases behind)
    auto vfix = [&](int st) { return bar0 + 8u * (2 * SK + 2 * SV + st); };
    const uint32_t bx = bar0 + 8u * (2 * SK + 3 * SV);
    auto sbar = [&](int j) { return bx + 8u * j; };
    auto sfree = [&](int j) { return bx + 8u * (2 + j); };
    auto pready = [&](int j) { return bx + 8u * (4 + j); };
    // pfree[j]: P V of tile k (k % 2 == j) has completed (so have all MMAs before it); a wait for
    // P V of tile k only ever happens once that of tile k - 2 is known complete, so the barrier is
    // never two phases away from the one waited for
    auto pfree = [&](int j) { return bx + 8u * (6 + j); };
    const uint32_t done = bx + 8u * 8, ofree = bx + 8u * 9, qfull = bx + 8u * 10, mlready = bx + 8u * 11;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rows = A.R * A.G, nrt = (rows + 63) / 64;
    const int n_items = A.nsplit * nrt * A.Hkv * A.B;
    // One CTA per item: blocks take the items split-slowest, so the rows' last splits (often a
    // few tiles only) come last and fill a second wave that a full split would drag out; a
    // persistent CTA walks a contiguous range numbered split-fastest (consecutive items share Q).
    const int per_split = n_items / A.nsplit;
    const int it0 = MULTI ? static_cast<int>(static_cast<long long>(blockIdx.x) * n_items / gridDim.x)
                          : (static_cast<int>(blockIdx.x) % per_split) * A.nsplit + static_cast<int>(blockIdx.x) / per_split;
    const int it1 = MULTI ? static_cast<int>(static_cast<long long>(blockIdx.x + 1) * n_items / gridDim.x) : it0 + 1;
    griddep_wait();
    int first = it0;
    while (first < it1 && !attn_item(A, first, nrt).live) ++first;
    if (tid == 0)
        for (int it = it0; it < it1; ++it) {
            const AttnItem I = attn_item(A, it, nrt);
            if (I.bad && I.split == 0 && I.row_base == 0 && I.g == 0) atomicOr(A.err, ERR_BAD_LENGTH);
        }
    if (first == it1) return;   // nothing live here: no barrier or tensor memory was set up

    if (tid == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        for (int st = 0; st < SK; ++st) {
            mbar_init(fullK(st), 1);
            mbar_init(emptyK(st), 1);
        }
        for (int st = 0; st < SV; ++st) {
            mbar_init(fullV(st), 1);
            mbar_init(emptyV(st), 1);
            mbar_init(vfix(st), 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(sbar(j), 1);
            mbar_init(sfree(j), 64);
            mbar_init(pready(j), 64);
            mbar_init(pfree(j), 1);
        }
        mbar_init(done, 1);
        mbar_init(ofree, 64);
        mbar_init(qfull, 64);
        mbar_init(mlready, 64);
        fence_mbar_init();
        s_abort = 0;
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_slot), S::TMEM_COLS);
        tmem_relinquish();
    }
    // All threads load the first item's Q; the softmax warps reload it when an item's Q differs
    // from the previous one's.  (Starting the K/V copies before this, in parallel with it, was
    // measured slower.)
    load_q_tile<HD, BLK, ATTN_THREADS>(smem + S::Q_OFF, A, attn_item(A, first, nrt), tid);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    // bounded waits, sleeping between tests (a waiting warp leaves the issue slots to the softmax
    // warps that share its scheduler); after the first one that gives up, every later wait
    // returns at once
    auto W = [&](uint32_t bar, uint32_t par) -> bool {
        if (s_abort) return false;
        if (!mbar_wait_sleep(bar, par, A.err)) {
            s_abort = 1;
            return false;
        }
        return true;
    };
    // the same verdict for every lane of a warp that goes on to warp-collective instructions
    auto WW = [&](uint32_t bar, uint32_t par) -> bool { return __all_sync(0xffffffffu, W(bar, par)); };
    auto same_q = [](const AttnItem& x, int b, int g, int rb) { return x.b == b && x.g == g && x.row_base == rb; };

    const uint32_t tS = tmem, tO = tmem + 128;   // columns: S[0] 0..63, S[1] 64..127, O 128..128+HD-1

    if (warp == 2 || warp == 3) {
        // ---- TMA producers: warp 2 the K tiles, warp 3 the V tiles (and the V fix of an item's
        // last tile: once its copy has landed, rows past every row's length are zeroed so that
        // p = 0 never meets a non-finite value there)
        const bool isK = warp == 2;
        const int NS = isK ? SK : SV;
        const CUtensorMap* map = isK ? &tmK : &tmV;
        int t = 0;   // tiles issued so far
        bool ok = true;
        for (int it = first; ok && it < it1; ++it) {
            const AttnItem I = attn_item(A, it, nrt);
            if (!I.live) continue;
            if (lane == 0) {
                for (int i = 0; i < I.ntiles; ++i) {
                    const int st = t % NS;
                    if (t >= NS && !W(isK ? emptyK(st) : emptyV(st), ((t / NS) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = isK ? fullK(st) : fullV(st);
                    const uint32_t dst = isK ? sK(st) : sV(st);
                    mbar_arrive_expect_tx(fb, TILE_BYTES);
                    int row;
                    const int z = kv_page(A.kv, I.b, I.p_begin + i * T, &row, A.err) * A.Hkv + I.g;
#pragma unroll
                    for (int cb = 0; cb < CB; ++cb) tma_load_3d(dst + cb * BLK, map, cb * 64, row, z, fb);
                    ++t;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            t = __shfl_sync(0xffffffffu, t, 0);
            if (!isK && ok && I.p_begin + I.ntiles * T > I.maxlen) {
                const int tl = t - 1, st = tl % SV;
                const int first_row = I.maxlen - (I.p_begin + (I.ntiles - 1) * T);
                if (WW(fullV(st), (tl / SV) & 1u)) {
                    for (int idx = first_row * 8 + lane; idx < T * 8; idx += 32)
#pragma unroll
                        for (int cb = 0; cb < CB; ++cb)
                            *reinterpret_cast<uint4*>(smem + (sV(st) - base) + cb * BLK + idx * 16) = make_uint4(0, 0, 0, 0);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(vfix(st));
                } else {
                    ok = false;
                }
            }
        }
        // every issued copy lands before the CTA may leave
        if (lane == 0)
            for (int j = t > NS ? t - NS : 0; j < t; ++j) mbar_wait(isK ? fullK(j % NS) : fullV(j % NS), (j / NS) & 1u, A.err);
    } else if (warp == 6) {
        // ---- MMA issuer: Q K^T of tile t+1 goes out before P V of tile t (within an item)
        if (lane == 0) {
            constexpr uint32_t IDS = idesc_bf16_f32(128, T), IDO = idesc_bf16_f32(128, HD, true);
            // the next 64 dims of V sit one block further; with a single block the field is never
            // used and holds the group stride, which keeps every address of the operand inside
            // its stage under either reading of the two fields
            constexpr uint32_t VBLK = CB > 1 ? BLK : 1024;
            auto qk = [&](int tt) -> bool {
                const int st = tt % SK;
                if (!W(fullK(st), (tt / SK) & 1u)) return false;
                if (tt >= 2 && !W(sfree(tt & 1), ((tt - 2) >> 1) & 1u)) return false;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < HD / 16; ++ks) {
                    const uint64_t ad = sw128_kmajor_desc(sQ + (ks >> 2) * BLK + (ks & 3) * 32);
                    const uint64_t bd = sw128_kmajor_desc(sK(st) + (ks >> 2) * BLK + (ks & 3) * 32);
                    tc_mma_bf16(tS + (tt & 1) * T, ad, bd, IDS, ks > 0 ? 1u : 0u);
                }
                tc_commit(sbar(tt & 1));
                tc_commit(emptyK(st));
                return true;
            };
            int t = 0, jl = 0, nq = 0;
            uint32_t fixpar = 0;   // bit st: parity of the next vfix phase of V stage st
            int qb = -1, qg = -1, qrb = -1;
            bool ok = true, pre = false;   // pre: this item's first Q K^T went out with the last item
            for (int it = first; ok && it < it1; ++it) {
                const AttnItem I = attn_item(A, it, nrt);
                if (!I.live) continue;
                if (MULTI && jl > 0 && !same_q(I, qb, qg, qrb)) {
                    if (!W(qfull, nq & 1u)) break;
                    ++nq;
                }
                qb = I.b, qg = I.g, qrb = I.row_base;
                if (!pre && !qk(t)) break;
                pre = false;
                // the next live item: with the same Q its first Q K^T goes out before this item's
                // last P V, so its S is ready when the softmax warps come to it
                bool next_same = false;
                if (MULTI) {
                    int nx = it + 1;
                    while (nx < it1 && !attn_item(A, nx, nrt).live) ++nx;
                    next_same = nx < it1 && same_q(attn_item(A, nx, nrt), I.b, I.g, I.row_base);
                }
                for (int i = 0; i < I.ntiles; ++i) {
                    const int tt = t + i, sv = tt % SV;
                    if ((i + 1 < I.ntiles || next_same) && !qk(tt + 1)) { ok = false; break; }
                    if (i + 1 == I.ntiles && next_same) pre = true;
                    const bool fix = i == I.ntiles - 1 && I.p_begin + I.ntiles * T > I.maxlen;
                    if (MULTI && i == 0 && jl > 0 && !W(ofree, (jl - 1) & 1u)) { ok = false; break; }
                    if (!W(pready(tt & 1), (tt >> 1) & 1u) ||
                        !W(fix ? vfix(sv) : fullV(sv), fix ? (fixpar >> sv) & 1u : (tt / SV) & 1u)) {
                        ok = false;
                        break;
                    }
                    if (fix) fixpar ^= 1u << sv;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < T / 16; ++kk)   // 16 positions = two 8-row groups of the V tile
                        tc_mma_bf16(tO, sw128_kmajor_desc(sP + (tt & 1) * BLK + kk * 32),
                                    sw128_mnmajor_desc(sV(sv) + kk * 2048, VBLK, 1024), IDO, (i > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(pfree(tt & 1));
                    tc_commit(emptyV(sv));
                }
                t += I.ntiles;
                ++jl;
            }
            tc_commit(done);   // every MMA issued is complete before the CTA may leave
            mbar_wait(done, 0u, A.err);
        }
    } else if (warp >= 4) {
        // ---- epilogue: thread = tile row rho (TMEM lane rho, the lanes of warps 0-1)
        const int rho = tid - 128;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        int t = 0, jl = 0;
        for (int it = first; it < it1; ++it) {
            const AttnItem I = attn_item(A, it, nrt);
            if (!I.live) continue;
            const int tl = t + I.ntiles - 1;
            // m and l of the item (the softmax warps are done with it), then its last P V
            if (!WW(mlready, jl & 1u) || !WW(pfree(tl & 1), (tl >> 1) & 1u)) break;
            tc_fence_after();
            const int grow = I.row_base + rho;
            const int len = grow < rows ? I.L0 + grow / A.G : 0;
            // tcgen05.ld is warp-collective: every lane loads, the live rows store
            const bool live = grow < rows && len > I.p_begin;
            const int r = grow / A.G, h = I.g * A.G + grow % A.G;
            const long long idx = ((static_cast<long long>(I.b) * A.R + r) * A.Hq + h) * A.nsplit + I.split;
            float* op = A.opart + idx * HD;
            const float2 ml = ml_sm[rho];
#pragma unroll 1
            for (int c = 0; c < HD / 64; ++c) {
                float o[64];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) tmem_ld16(tO + lane_off + c * 64 + q4 * 16, o + q4 * 16);
                tmem_ld_wait();
                if (live) {
#pragma unroll
                    for (int e = 0; e < 64; e += 4)
                        *reinterpret_cast<float4*>(op + c * 64 + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
                }
            }
            if (live) A.ml[idx] = ml;
            tc_fence_before();
            mbar_arrive(ofree);   // O (and ml_sm) may be overwritten by the next item
            t += I.ntiles;
            ++jl;
        }
    } else {
        // ---- softmax: thread = tile row rho (TMEM lane rho)
        const int rho = tid;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        int t = 0, jl = 0;
        int qb = -1, qg = -1, qrb = -1;
        for (int it = first; it < it1; ++it) {
            const AttnItem I = attn_item(A, it, nrt);
            if (!I.live) continue;
            if constexpr (MULTI) {
                if (jl > 0 && !same_q(I, qb, qg, qrb)) {
                    // every Q K^T that read the old Q has completed (this warp has seen the S of
                    // the previous item's last tile; P V does not read Q), and the MMA warp issues
                    // nothing for this item until qfull
                    load_q_tile<HD, BLK, 64>(smem + S::Q_OFF, A, I, rho);
                    fence_proxy_async_smem();
                    mbar_arrive(qfull);
                }
            }
            qb = I.b, qg = I.g, qrb = I.row_base;
            const int grow = I.row_base + rho;   // row of the verify block
            const int len = grow < rows ? I.L0 + grow / A.G : 0;
            float m = NEG_INF, l = 0.f;
            bool ok = true;
            for (int i = 0; i < I.ntiles; ++i) {
                const int tt = t + i;
                if (!WW(sbar(tt & 1), (tt >> 1) & 1u)) { ok = false; break; }
                tc_fence_after();
                float s[T];
#pragma unroll
                for (int c = 0; c < T / 16; ++c) tmem_ld16(tS + lane_off + (tt & 1) * T + c * 16, s + c * 16);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(sfree(tt & 1));
                const int p0 = I.p_begin + i * T;
                float mx = NEG_INF;
#pragma unroll
                for (int j = 0; j < T; ++j) {
                    s[j] = p0 + j < len ? __fmul_rn(s[j], A.sl2) : NEG_INF;
                    mx = fmaxf(mx, s[j]);
                }
                const float mn = (m == NEG_INF || mx > __fadd_rn(m, RESCALE_SLACK)) ? mx : m;
                const bool dead = mn == NEG_INF;
                const float al = (dead || mn == m) ? 1.f : ex2_approx(__fsub_rn(m, mn));
                float ts = 0.f;
                uint32_t pk[T / 2];
#pragma unroll
                for (int j = 0; j < T; j += 2) {
                    const float a0 = dead ? 0.f : ex2_approx(__fsub_rn(s[j], mn));
                    const float a1 = dead ? 0.f : ex2_approx(__fsub_rn(s[j + 1], mn));
                    ts = __fadd_rn(__fadd_rn(ts, a0), a1);
                    pk[j / 2] = pack_bf16x2(a0, a1);
                }
                l = __fadd_rn(__fmul_rn(l, al), ts);
                m = mn;
                // O is rescaled once P V of tile tt-1 has completed (tcgen05.ld/st are warp-collective)
                if (i >= 1 && __any_sync(0xffffffffu, al != 1.f)) {
                    if (!WW(pfree((tt - 1) & 1), ((tt - 1) >> 1) & 1u)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < HD / 64; ++c) {
                        float o[64];
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) tmem_ld16(tO + lane_off + c * 64 + q4 * 16, o + q4 * 16);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 64; ++e) o[e] = __fmul_rn(o[e], al);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) tmem_st16(tO + lane_off + c * 64 + q4 * 16, o + q4 * 16);
                    }
                    tmem_st_wait();
                }
                // P buffer tt%2 was last read by P V of tile tt-2
                if (tt >= 2 && !WW(pfree(tt & 1), ((tt - 2) >> 1) & 1u)) { ok = false; break; }
#pragma unroll
                for (int c = 0; c < T / 8; ++c)
                    *reinterpret_cast<uint4*>(smem + S::P_OFF + (tt & 1) * BLK + rho * 128 + ((c ^ (rho & 7)) * 16)) =
                        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(pready(tt & 1));
            }
            if (!ok) break;
            // hand m and l to the epilogue warps (once they are done with the previous item's)
            if (MULTI && jl > 0 && !WW(ofree, (jl - 1) & 1u)) break;
            ml_sm[rho] = make_float2(m, l);
            mbar_arrive(mlready);
            t += I.ntiles;
            ++jl;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, S::TMEM_COLS);
    }
}

struct CombineArgs {
    const int32_t* ctx_len;
    int len_bias, R, Hq, nsplit, max_len, hd;
    int ch, nb;   // splits per staged chunk and chunk buffers (combine_shape)
    const float* opart;
    const float2* ml;
    const uint16_t* gate;
    long long gate_stride;
    uint16_t* out;
    long long out_stride;
    unsigned* err;
};

// One CTA per (row, q head); thread t owns output elements 2t and 2t+1.  Per thread, in split
// order s = 0..ns-1:  w_s = exp2(m_s - M), L += w_s l_s, acc += w_s o_s;  out = acc / L, where M
// is the largest m_s (a maximum is exact in any order, so the CTA takes it as a tree).  The
// split partials o_s of a (row, head) are contiguous: they stream through shared memory in
// chunks of up to COMB_CH splits by bulk copies, up to COMB_NB chunks in flight.  The staging is
// sized by the number of splits (a short context needs a few KB, not 96): measured at batch 8 /
// context 2183 (2048 CTAs), the full 96 KB let 2 CTAs share an SM and the combine ran in ~7
// waves, 13 us of the step.
constexpr int COMB_CH = 32, COMB_NB = 3;

inline void combine_shape(int nsplit, int* ch, int* nb) {
    *ch = nsplit < COMB_CH ? nsplit : COMB_CH;
    const int chunks = (nsplit + *ch - 1) / *ch;
    *nb = chunks < COMB_NB ? chunks : COMB_NB;
}

inline size_t combine_smem(int hd, int nsplit) {
    int ch, nb;
    combine_shape(nsplit, &ch, &nb);
    return static_cast<size_t>(nb) * ch * hd * 4 + static_cast<size_t>(nsplit) * 8;
}

__global__ void __launch_bounds__(128) attn_combine_kernel(CombineArgs C) {
    griddep_launch();
    griddep_wait();
    extern __shared__ __align__(128) uint8_t csm[];
    __shared__ __align__(8) uint64_t cbar[COMB_NB];
    const int CH = C.ch, NB = C.nb;
    __shared__ float wmax[4];
    __shared__ volatile int s_abort;
    const int hq = blockIdx.x % C.Hq;
    const long long br = blockIdx.x / C.Hq;
    const int b = static_cast<int>(br / C.R), r = static_cast<int>(br % C.R);
    const int len = C.ctx_len[b] + C.len_bias + r;
    if (len < 1 || len - r + C.R - 1 > C.max_len) return;   // reported by the split kernel
    const int ns = attn_split_count(len);
    const long long idx0 = (br * C.Hq + hq) * C.nsplit;
    const int tid = threadIdx.x, nt = blockDim.x;
    float* obuf = reinterpret_cast<float*>(csm);               // NB chunks of [CH][hd]
    float* wv = obuf + NB * CH * C.hd;                         // w_s
    float* lv = wv + C.nsplit;                                 // l_s
    const int nchunk = (ns + CH - 1) / CH;
    const float* src = C.opart + idx0 * C.hd;
    auto bar = [&](int i) { return smem_u32(&cbar[i]); };
    auto issue = [&](int c) {
        const int n = min(CH, ns - c * CH);
        const uint32_t bytes = static_cast<uint32_t>(n) * C.hd * 4;
        mbar_arrive_expect_tx(bar(c % NB), bytes);
        bulk_load(smem_u32(obuf + (c % NB) * CH * C.hd), src + static_cast<long long>(c) * CH * C.hd, bytes,
                  bar(c % NB));
    };
    int issued = 0;   // thread 0: chunks whose copies have been issued
    if (tid == 0) {
        for (int i = 0; i < NB; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
        s_abort = 0;
        for (; issued < nchunk && issued < NB; ++issued) issue(issued);
    }
    float mx = NEG_INF;
    for (int s = tid; s < ns; s += nt) {
        const float2 v = C.ml[idx0 + s];
        wv[s] = v.x;
        lv[s] = v.y;
        mx = fmaxf(mx, v.x);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((tid & 31) == 0) wmax[tid >> 5] = mx;
    __syncthreads();
    float M = wmax[0];
    for (int w = 1; w < (nt >> 5); ++w) M = fmaxf(M, wmax[w]);
    for (int s = tid; s < ns; s += nt) wv[s] = exp2f(__fsub_rn(wv[s], M));
    __syncthreads();
    const int d = 2 * tid;
    float L = 0.f, acc0 = 0.f, acc1 = 0.f;
    for (int c = 0; c < nchunk; ++c) {
        const int st = c % NB;
        if (!s_abort && !mbar_wait(bar(st), (c / NB) & 1u, C.err)) s_abort = 1;
        if (!s_abort) {
            const float* ob = obuf + st * CH * C.hd + d;
            const int s0 = c * CH, n = min(CH, ns - s0);
            for (int j = 0; j < n; ++j) {
                const float w = wv[s0 + j];
                const float2 o = *reinterpret_cast<const float2*>(ob + j * C.hd);
                L = __fadd_rn(L, __fmul_rn(w, lv[s0 + j]));
                acc0 = __fadd_rn(acc0, __fmul_rn(w, o.x));
                acc1 = __fadd_rn(acc1, __fmul_rn(w, o.y));
            }
        }
        __syncthreads();   // every thread is done with chunk c's buffer
        if (tid == 0 && c + NB < nchunk && !s_abort) {
            fence_proxy_async_smem();
            issue(c + NB);
            ++issued;
        }
    }
    if (s_abort) {
        // copies still in flight land before the CTA leaves: wait for the last one of each buffer
        if (tid == 0)
            for (int c = issued - 1; c >= 0 && c >= issued - NB; --c) mbar_wait(bar(c % NB), (c / NB) & 1u, C.err);
        return;
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
inline int nsplit_for(int max_len) { return attn_split_count(max_len); }

template <int HD>
xv_status launch_split(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnArgs& a, int B, cudaStream_t s) {
    using S = AttnShape<HD>;
    int sms = 0;
    if (xv_status st = kernel_smem_once(reinterpret_cast<const void*>(attn_split_kernel<HD, true>), S::SMEM, false,
                                        "attn: set shared memory size"))
        return st;
    if (xv_status st = kernel_smem_once(reinterpret_cast<const void*>(attn_split_kernel<HD, false>), S::SMEM, false,
                                        "attn: set shared memory size"))
        return st;
    if (xv_status st = device_sm_count(&sms)) return st;
    // past two waves of items, one persistent CTA per SM (the shared-memory plan admits one);
    // otherwise one CTA per item (measured in the verify step: with 160 items the persistent
    // launch was 4 us slower, with 1028 and 8224 items 15 and 218 us faster)
    const long long n_items = static_cast<long long>(a.nsplit) * ((a.R * a.G + 63) / 64) * a.Hkv * B;
    if (n_items > (1ll << 30)) return fail(XV_ERR_UNSUPPORTED, "attn: %lld work items", n_items);
    const bool multi = n_items > 2ll * sms;
    dim3 grid(static_cast<unsigned>(multi ? sms : n_items));
    trace_pre(s);
    if (multi) launch_k(attn_split_kernel<HD, true>, dim3(grid), dim3(ATTN_THREADS), S::SMEM, s, tmK, tmV, a);
    else launch_k(attn_split_kernel<HD, false>, dim3(grid), dim3(ATTN_THREADS), S::SMEM, s, tmK, tmV, a);
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
    AttnArgs a{q, q_stride, kv, ctx_len, len_bias, R, Hq / Hkv, Hq, Hkv, nsplit, max_len, B,
               scale * 1.4426950408889634f, opart, ml, err};
    xv_status st = hd == 256 ? launch_split<256>(tmK, tmV, a, B, s) : launch_split<64>(tmK, tmV, a, B, s);
    if (st) return st;
    int cch, cnb;
    combine_shape(nsplit, &cch, &cnb);
    CombineArgs c{ctx_len, len_bias, R, Hq, nsplit, max_len, hd, cch, cnb, opart, ml, gate, gate_stride, out, out_stride,
                  err};
    const size_t csm = combine_smem(hd, nsplit);
    if (xv_status e = kernel_smem_once(reinterpret_cast<const void*>(attn_combine_kernel), static_cast<int>(csm), false,
                                       "attn: set combine shared memory size"))
        return e;
    trace_pre(s);
    launch_k(attn_combine_kernel, dim3(B * R * Hq), dim3(hd / 2), csm, s, c);
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
