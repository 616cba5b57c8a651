// The verify block: a stack of hybrid decoder layers under an embedding and
// an LM head, run for B sequences x k tokens in one stream-ordered pass.
//
// Decode is the same pass with k = 1; nothing in it depends on k except the
// row count, and every kernel it calls gives a row the same bits whatever the
// row count ("Follow-up to my earlier post on Qwen3.8-27B decode speed",
// r/LocalLLaMA post: with the verify fixes, every token id and every logprob
// matched decoding without speculation, also with every draft forced to
// reject and with 8 requests in flight).
//
// GDN layers use deferred commit: a verify call first replays the pending
// steps (the inputs of the previous verify's kept positions) into the
// committed state, then speculates over this call's k tokens without
// writing the state; its own inputs become the next pending steps.  State
// traffic is one read and one write per call instead of k writes.
#include <algorithm>
#include <vector>

#include "xv_internal.h"

namespace xv {
namespace {

struct Dims {
    int H, V, F, L;
    int gh, dk, dv, gin, ginner, gstride;
    int hk, kc, onorm, cdim, cstride, bcol;   // q/k heads, conv width, gated norm, conv channels, b column
    int hq, hkv, hd, ain, ainner;
};

xv_status check_cfg(const xv_block_config* c, Dims* d) {
    if (!c) return fail(XV_ERR_ARG, "block: null config");
    if (c->hidden < 64 || c->hidden % 64 || c->vocab < 1 || c->mlp < 64 || c->mlp % 64 || c->n_layers < 1 || !c->layer_kind)
        return fail(XV_ERR_ARG, "block: hidden and mlp must be positive multiples of 64, vocab and n_layers >= 1");
    bool has_gdn = false, has_attn = false;
    for (int l = 0; l < c->n_layers; ++l) {
        if (c->layer_kind[l] == 0) has_gdn = true;
        else if (c->layer_kind[l] == 1) has_attn = true;
        else return fail(XV_ERR_ARG, "block: layer_kind[%d] must be 0 (GDN) or 1 (attention)", l);
    }
    d->H = c->hidden; d->V = c->vocab; d->F = c->mlp; d->L = c->n_layers;
    d->gh = c->gdn_heads; d->dk = c->gdn_dk; d->dv = c->gdn_dv;
    d->hq = c->attn_hq; d->hkv = c->attn_hkv; d->hd = c->attn_hd;
    d->hk = c->gdn_qk_heads > 0 ? c->gdn_qk_heads : c->gdn_heads;
    d->kc = c->gdn_conv;
    d->onorm = c->gdn_out_norm ? 1 : 0;
    d->ginner = d->gh * d->dv;
    d->cdim = 2 * d->hk * d->dk + d->ginner;
    d->cstride = (d->cdim + 7) / 8 * 8;
    d->bcol = d->cdim + (d->onorm ? d->ginner : 0);
    d->gin = d->bcol + 2 * d->gh;
    d->gstride = (d->gin + 7) / 8 * 8;
    d->ain = 2 * d->hq * d->hd + 2 * d->hkv * d->hd;
    d->ainner = d->hq * d->hd;
    if (has_gdn) {
        if ((d->dk != 64 && d->dk != 128) || d->dv < 32 || d->dv % 32 || d->gh < 1)
            return fail(XV_ERR_UNSUPPORTED, "block: GDN needs dk in {64,128}, dv a multiple of 32");
        if (d->ginner % 8) return fail(XV_ERR_UNSUPPORTED, "block: GDN heads*dv must be a multiple of 8");
        if (d->hk < 1 || d->gh % d->hk) return fail(XV_ERR_ARG, "block: gdn_qk_heads must divide gdn_heads");
        if (d->kc != 0 && (d->kc < 2 || d->kc > XV_CONV_MAX))
            return fail(XV_ERR_UNSUPPORTED, "block: gdn_conv must be 0 or lie in [2, %d]", XV_CONV_MAX);
        if (c->gdn_out_norm != 0 && c->gdn_out_norm != 1) return fail(XV_ERR_ARG, "block: gdn_out_norm must be 0 or 1");
        if (d->onorm && d->dv > 256) return fail(XV_ERR_UNSUPPORTED, "block: the gated output norm needs dv <= 256");
    } else {
        d->gin = d->ginner = d->cdim = 0;
        d->kc = d->onorm = 0;
    }
    if (has_attn) {
        if ((d->hd != 64 && d->hd != 256) || d->hkv < 1 || d->hq % d->hkv)
            return fail(XV_ERR_UNSUPPORTED, "block: attention needs hd in {64,256} and Hq a multiple of Hkv");
    } else {
        d->ain = d->ainner = 0;
    }
    return XV_OK;
}

inline size_t r256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Carves the block workspace; returns the total size when base is null.
struct Carve {
    uint16_t *x, *xn, *proj, *obuf, *y, *gu, *act;
    float* logits;
    void* argmax_ws;
    void* gemm_ws;
    size_t gemm_ws_bytes;
    void* attn_ws;
    size_t attn_ws_bytes;
    size_t total;
};

Carve carve(const Dims& d, int B, int kmax, int Lmax, uint8_t* base) {
    Carve c{};
    const int M = B * kmax;
    size_t off = 0;
    auto take = [&](size_t bytes) { uint8_t* p = base ? base + off : nullptr; off += r256(bytes); return p; };
    // the residual stream comes first: the header promises the final hidden state at offset 0
    c.x = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(M) * d.H * 2));
    c.xn = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(M) * d.H * 2));
    c.proj = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(M) * (d.ain > 0 ? d.ain : 8) * 2));
    const int inner = d.ginner > d.ainner ? d.ginner : d.ainner;
    c.obuf = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(M) * inner * 2));
    c.y = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(M) * d.H * 2));
    c.gu = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(M) * 2 * d.F * 2));
    c.act = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(M) * d.F * 2));
    c.logits = reinterpret_cast<float*>(take(static_cast<size_t>(M) * d.V * 4));
    // argmax partials: per 8192-logit chunk, or per LM-head tile when the LM head forms them
    const size_t amax_tiles = static_cast<size_t>(M) * ceil_div(d.V, GEMM_BN) * sizeof(float2);
    c.argmax_ws = take(std::max(argmax_workspace_size(M, d.V), amax_tiles));
    size_t g = 0;
    auto gm = [&](int N, int K) { size_t s = gemm_workspace_size(M, N, K); if (s > g) g = s; };
    if (d.gin) { gm(d.gin, d.H); gm(d.H, d.ginner); }
    if (d.ain) { gm(d.ain, d.H); gm(d.H, d.ainner); }
    gm(2 * d.F, d.H); gm(d.H, d.F); gm(d.V, d.H);
    c.gemm_ws_bytes = g;
    c.gemm_ws = take(g > 0 ? g : 256);
    c.attn_ws_bytes = d.ain ? attn_workspace_size(B, kmax, d.hq, d.hd, Lmax) : 0;
    c.attn_ws = take(c.attn_ws_bytes > 0 ? c.attn_ws_bytes : 256);
    c.total = off;
    return c;
}

}  // namespace
}  // namespace xv

using namespace xv;

extern "C" {

int xv_gdn_in_dim(const xv_block_config* cfg) {
    Dims d{};
    return check_cfg(cfg, &d) ? -1 : d.gin;
}

int xv_gdn_hist_stride(const xv_block_config* cfg) {
    Dims d{};
    return check_cfg(cfg, &d) ? -1 : d.gstride;
}

int xv_attn_in_dim(const xv_block_config* cfg) {
    Dims d{};
    return check_cfg(cfg, &d) ? -1 : d.ain;
}

int xv_gdn_conv_dim(const xv_block_config* cfg) {
    Dims d{};
    return check_cfg(cfg, &d) ? -1 : d.cdim;
}

int xv_gdn_conv_stride(const xv_block_config* cfg) {
    Dims d{};
    return check_cfg(cfg, &d) ? -1 : d.cstride;
}

size_t xv_block_workspace_size(const xv_block_config* cfg, int B, int kmax, int Lmax) {
    Dims d{};
    if (check_cfg(cfg, &d) || B < 1 || kmax < 1 || Lmax < 1) return 0;
    return carve(d, B, kmax, Lmax, nullptr).total;
}

static xv_status check_state(const Dims& d, const xv_block_config* cfg, const xv_block_state* st) {
    if (!st || !st->ctx_len || !st->n_commit || !st->layers) return fail(XV_ERR_ARG, "block: incomplete state");
    if (st->B < 1 || st->kmax < 1 || st->kmax > XV_KMAX || st->Lmax < 1)
        return fail(XV_ERR_ARG, "block: state needs B >= 1, 1 <= kmax <= %d, Lmax >= 1", XV_KMAX);
    const xv_kv_pages& pg = st->kv_pages;
    if (pg.page_table) {
        if (pg.page_size < 64 || pg.page_size % 64 || pg.max_pages < 1 || pg.n_pages < 1)
            return fail(XV_ERR_ARG, "block: paged KV needs page_size a positive multiple of 64, max_pages, n_pages >= 1");
        if (static_cast<long long>(pg.page_size) * pg.max_pages < st->Lmax)
            return fail(XV_ERR_ARG, "block: Lmax exceeds page_size * max_pages");
        if (static_cast<long long>(pg.n_pages) * d.hkv > (1ll << 31))
            return fail(XV_ERR_UNSUPPORTED, "block: too many KV pages");
    }
    for (int l = 0; l < d.L; ++l) {
        const xv_layer_state& ls = st->layers[l];
        if (cfg->layer_kind[l] == 0) {
            if (!ls.gdn_state || !ls.gdn_hist[0] || !ls.gdn_hist[1])
                return fail(XV_ERR_ARG, "block: GDN layer %d state incomplete", l);
            if (!aligned16(ls.gdn_hist[0]) || !aligned16(ls.gdn_hist[1]))
                return fail(XV_ERR_UNSUPPORTED, "block: GDN history buffers must be 16-byte aligned");
            if (d.kc) {
                if (!ls.gdn_conv_state || !ls.gdn_conv_out[0] || !ls.gdn_conv_out[1])
                    return fail(XV_ERR_ARG, "block: GDN layer %d convolution state or outputs missing", l);
                if (!aligned16(ls.gdn_conv_out[0]) || !aligned16(ls.gdn_conv_out[1]))
                    return fail(XV_ERR_UNSUPPORTED, "block: GDN convolution output buffers must be 16-byte aligned");
            }
        } else {
            if (!ls.k_cache || !ls.v_cache) return fail(XV_ERR_ARG, "block: attention layer %d cache missing", l);
            if (!aligned16(ls.k_cache) || !aligned16(ls.v_cache))
                return fail(XV_ERR_UNSUPPORTED, "block: caches must be 16-byte aligned");
        }
    }
    return XV_OK;
}

static KvPages state_pages(const xv_block_state* st) {
    const xv_kv_pages& pg = st->kv_pages;
    return pg.page_table ? KvPages{pg.page_table, pg.page_size, pg.max_pages, pg.n_pages} : kv_contiguous(st->B, st->Lmax);
}

// The verify pass; with head = false it stops after the final RMSNorm (no LM head, argmax or
// acceptance: a prefill chunk whose logits nobody reads).
// With commit, the acceptance kernel also commits the accepted drafts + 1 of every sequence and
// the host-side state advances as xv_block_commit_accepted would advance it.
static xv_status verify_impl(const xv_block_config* cfg, const xv_block_weights* w, xv_block_state* st,
                             const int32_t* tokens, int k, const int32_t* k_seq, float* logits, int32_t* argmax,
                             int32_t* n_accept, void* ws, size_t ws_bytes, xv_stream stream, bool head,
                             bool commit = false) {
    Dims d{};
    if (xv_status e = check_cfg(cfg, &d)) return e;
    if (xv_status e = check_state(d, cfg, st)) return e;
    if (!w || !w->embed || !w->layers || !w->final_norm || !w->lm_head) return fail(XV_ERR_ARG, "block: incomplete weights");
    for (int l = 0; l < d.L; ++l) {
        const xv_layer_weights& lw = w->layers[l];
        if (!lw.norm1 || !lw.w_in || !lw.w_out || !lw.norm2 || !lw.w_gate_up || !lw.w_down)
            return fail(XV_ERR_ARG, "block: layer %d weights incomplete", l);
        if (cfg->layer_kind[l] == 0 && ((d.kc && !lw.conv_w) || (d.onorm && !lw.out_norm)))
            return fail(XV_ERR_ARG, "block: GDN layer %d convolution taps or output norm weights missing", l);
    }
    if (!tokens || (head && (!argmax || !n_accept))) return fail(XV_ERR_ARG, "block: null tokens, argmax or n_accept");
    if (w->tiled && d.F % 64) return fail(XV_ERR_UNSUPPORTED, "block: tiled weights need mlp a multiple of 64");
    if (st->last_k != 0) return fail(XV_ERR_ARG, "block: the previous verify has not been committed");
    const int B = st->B;
    if (k < 1 || k > st->kmax) return fail(XV_ERR_ARG, "block: k = %d outside [1, kmax = %d]", k, st->kmax);
    const int M = B * k;
    if (M > XV_GEMM_M_MAX) return fail(XV_ERR_UNSUPPORTED, "block: B*k = %d exceeds %d", M, XV_GEMM_M_MAX);
    if (st->max_ctx < 0 || st->max_ctx + k > st->Lmax)
        return fail(XV_ERR_ARG, "block: max_ctx + k (%d) exceeds Lmax (%d)", st->max_ctx + k, st->Lmax);
    if (st->pending_rows < 1 || st->pending_rows > st->kmax) return fail(XV_ERR_ARG, "block: pending_rows out of range");
    const Carve need = carve(d, B, st->kmax, st->Lmax, nullptr);
    if (!ws || ws_bytes < need.total) return fail(XV_ERR_WORKSPACE, "block: workspace of %zu bytes needed", need.total);
    const Carve c = carve(d, B, st->kmax, st->Lmax, static_cast<uint8_t*>(ws));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    float* lg = logits ? logits : c.logits;
    const float eps = cfg->rms_eps;
    const int par = st->parity & 1;
    const int attn_len = st->max_ctx + k;   // bound on ctx_len + 1 + (k - 1)
    const KvPages kv = state_pages(st);
    const WLayout wt = w->tiled ? W_TILED : W_ROWS;

#define XV_TRY(expr) do { if (xv_status e_ = (expr)) return e_; } while (0)
    XV_TRY(embed_rmsnorm_launch(tokens, M, w->embed, d.V, d.H, w->layers[0].norm1, eps, c.x, c.xn, s));
    // a projection into the residual stream, then x <- bf16(x + y), xn <- rmsnorm(x, gain); where
    // the GEMM would combine its split-K partials in a kernel of its own, the norm kernel sums
    // them itself (the same sums in the same order: the same bits)
    auto residual_gemm = [&](const uint16_t* A, int K, const uint16_t* Wt, const uint16_t* gain) -> xv_status {
        float* part = nullptr;
        int S = 0;
        XV_TRY(gemm_launch(A, K, Wt, wt, c.y, d.H, false, M, d.H, K, c.gemm_ws, c.gemm_ws_bytes, s, &part, &S));
        if (part) return residual_rmsnorm_part_launch(c.x, part, S, gain, M, d.H, eps, c.xn, s);
        return residual_rmsnorm_launch(c.x, c.y, gain, M, d.H, eps, c.xn, s);
    };
    for (int l = 0; l < d.L; ++l) {
        const xv_layer_weights& lw = w->layers[l];
        xv_layer_state& ls = st->layers[l];
        if (cfg->layer_kind[l] == 0) {
            uint16_t* hist = ls.gdn_hist[par];
            XV_TRY(gemm_launch(c.xn, d.H, lw.w_in, wt, hist, d.gstride, false, M, d.gin, d.H, c.gemm_ws, c.gemm_ws_bytes, s));
            // the recurrence kernel reads q, k, v (the convolution's outputs, or the history rows
            // themselves) and the raw b, a columns of the history rows
            const uint16_t* ph = ls.gdn_hist[par ^ 1];
            const uint16_t* qkv_pend = ph;
            const uint16_t* qkv_cur = hist;
            long long qstride = d.gstride;
            if (d.kc) {
                XV_TRY(conv_launch(ls.gdn_conv_state, ph, d.gstride, st->pending_rows, st->n_commit, st->pending_rows,
                                   hist, d.gstride, k, k, lw.conv_w, d.cdim, d.kc, B, ls.gdn_conv_out[par], d.cstride, s));
                qkv_pend = ls.gdn_conv_out[par ^ 1];
                qkv_cur = ls.gdn_conv_out[par];
                qstride = d.cstride;
            }
            const int qk = d.hk * d.dk;
            GdnStepsDev pend{qkv_pend, qkv_pend + qk, qkv_pend + 2 * qk, ph + d.bcol, ph + d.bcol + d.gh, qstride,
                             d.gstride, st->pending_rows, 1};
            GdnStepsDev draft{qkv_cur, qkv_cur + qk, qkv_cur + 2 * qk, hist + d.bcol, hist + d.bcol + d.gh, qstride,
                              d.gstride, k, 1};
            XV_TRY(gdn_launch(ls.gdn_state, pend, st->n_commit, 0, st->pending_rows, false, draft, k, c.obuf, d.ginner, B,
                              d.gh, d.hk, d.dk, d.dv, 1, s));
            if (d.onorm)
                XV_TRY(gated_norm_launch(c.obuf, d.ginner, hist + d.cdim, d.gstride, lw.out_norm, M, d.gh, d.dv, eps,
                                         c.obuf, d.ginner, s));
            XV_TRY(residual_gemm(c.obuf, d.ginner, lw.w_out, lw.norm2));
        } else {
            XV_TRY(gemm_launch(c.xn, d.H, lw.w_in, wt, c.proj, d.ain, false, M, d.ain, d.H, c.gemm_ws, c.gemm_ws_bytes, s));
            XV_TRY(kv_append_launch(c.proj + 2 * d.ainner, d.ain, st->ctx_len, 0, k, B, d.hkv, d.hd, kv, ls.k_cache,
                                    ls.v_cache, s));
            XV_TRY(attn_launch(c.proj, d.ain, ls.k_cache, ls.v_cache, kv, st->ctx_len, 1, k, B, d.hq, d.hkv, d.hd,
                               attn_len, 1.0f / sqrtf(static_cast<float>(d.hd)), c.proj + d.ainner, d.ain, c.obuf,
                               d.ainner, c.attn_ws, c.attn_ws_bytes, s));
            XV_TRY(residual_gemm(c.obuf, d.ainner, lw.w_out, lw.norm2));
        }
        if (wt == W_TILED) {
            // gate/up in the gated tiled layout: the GEMM writes the SwiGLU activations itself
            XV_TRY(gemm_launch(c.xn, d.H, lw.w_gate_up, W_GATED, c.act, d.F, false, M, 2 * d.F, d.H, nullptr, 0, s));
        } else {
            XV_TRY(gemm_launch(c.xn, d.H, lw.w_gate_up, wt, c.gu, 2 * d.F, false, M, 2 * d.F, d.H, c.gemm_ws,
                               c.gemm_ws_bytes, s));
            XV_TRY(swiglu_launch(c.gu, M, d.F, c.act, s));
        }
        const uint16_t* next_norm = (l + 1 < d.L) ? w->layers[l + 1].norm1 : w->final_norm;
        XV_TRY(residual_gemm(c.act, d.F, lw.w_down, next_norm));
    }
    if (head) {
        if (gemm_splits(d.V, d.H) == 1) {
            // the LM head leaves each tile's (max, lowest index) per row and writes logits only
            // when the caller wants them; the acceptance kernel finishes the argmax
            float2* amax = static_cast<float2*>(c.argmax_ws);
            XV_TRY(gemm_launch(c.xn, d.H, w->lm_head, wt, logits, d.V, true, M, d.V, d.H, c.gemm_ws, c.gemm_ws_bytes, s,
                               nullptr, nullptr, amax));
            XV_TRY(accept_from_parts_launch(amax, ceil_div(d.V, GEMM_BN), B, k, argmax, tokens, k_seq, n_accept, s,
                                            commit ? st->ctx_len : nullptr, commit ? st->n_commit : nullptr));
        } else {
            XV_TRY(gemm_launch(c.xn, d.H, w->lm_head, wt, lg, d.V, true, M, d.V, d.H, c.gemm_ws, c.gemm_ws_bytes, s));
            XV_TRY(argmax_accept_launch(lg, B, k, d.V, argmax, c.argmax_ws, tokens, k_seq, n_accept, s,
                                        commit ? st->ctx_len : nullptr, commit ? st->n_commit : nullptr));
        }
    }
#undef XV_TRY
    if (commit && head) {
        st->parity ^= 1;
        st->pending_rows = k;
        st->max_ctx += k;
        st->last_k = 0;
        st->last_k_seq = nullptr;
        return XV_OK;
    }
    st->last_k = k;
    st->last_k_seq = k_seq;
    return XV_OK;
}

xv_status xv_verify_block_commit_accepted(const xv_block_config* cfg, const xv_block_weights* w, xv_block_state* st,
                                          const int32_t* tokens, int k, float* logits, int32_t* argmax,
                                          int32_t* n_accept, void* ws, size_t ws_bytes, xv_stream stream) {
    return verify_impl(cfg, w, st, tokens, k, nullptr, logits, argmax, n_accept, ws, ws_bytes, stream, true, true);
}

xv_status xv_block_step_host(const xv_block_config* cfg, const xv_block_weights* w, xv_block_state* st,
                             const int32_t* host_tokens, int32_t* dev_tokens, int k, int32_t* dev_results,
                             int32_t* host_results, void* ws, size_t ws_bytes, xv_stream stream) {
    if (!st || !host_tokens || !dev_tokens || !dev_results || !host_results)
        return fail(XV_ERR_ARG, "step: null buffer");
    if (k < 1 || k > st->kmax) return fail(XV_ERR_ARG, "step: k = %d outside [1, kmax = %d]", k, st->kmax);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t B = static_cast<size_t>(st->B);
    if (xv_status e = cuda_check(cudaMemcpyAsync(dev_tokens, host_tokens, 4 * B * k, cudaMemcpyHostToDevice, s),
                                 "step: copy the drafts in"))
        return e;
    int32_t* argmax = dev_results;
    int32_t* n_accept = dev_results + B * st->kmax;
    if (xv_status e = verify_impl(cfg, w, st, dev_tokens, k, nullptr, nullptr, argmax, n_accept, ws, ws_bytes, stream,
                                  true, true))
        return e;
    return cuda_check(cudaMemcpyAsync(host_results, dev_results, 4 * (B * st->kmax + B), cudaMemcpyDeviceToHost, s),
                      "step: copy the results out");
}

xv_status xv_verify_block_ragged(const xv_block_config* cfg, const xv_block_weights* w, xv_block_state* st,
                                 const int32_t* tokens, int k, const int32_t* k_seq, float* logits, int32_t* argmax,
                                 int32_t* n_accept, void* ws, size_t ws_bytes, xv_stream stream) {
    return verify_impl(cfg, w, st, tokens, k, k_seq, logits, argmax, n_accept, ws, ws_bytes, stream, true);
}

xv_status xv_verify_block(const xv_block_config* cfg, const xv_block_weights* w, xv_block_state* st,
                          const int32_t* tokens, int k, float* logits, int32_t* argmax, int32_t* n_accept, void* ws,
                          size_t ws_bytes, xv_stream stream) {
    return xv_verify_block_ragged(cfg, w, st, tokens, k, nullptr, logits, argmax, n_accept, ws, ws_bytes, stream);
}

xv_status xv_block_commit(xv_block_state* st, const int32_t* n_keep, xv_stream stream) {
    if (!st || !st->ctx_len || !st->n_commit || !n_keep) return fail(XV_ERR_ARG, "commit: null argument");
    if (st->last_k < 1) return fail(XV_ERR_ARG, "commit: no verify to commit");
    xv_status e = commit_launch(n_keep, 0, st->B, st->last_k, st->last_k_seq, st->ctx_len, st->n_commit,
                                reinterpret_cast<cudaStream_t>(stream));
    if (e) return e;
    st->parity ^= 1;
    st->pending_rows = st->last_k;
    st->max_ctx += st->last_k;
    st->last_k = 0;
    st->last_k_seq = nullptr;
    return XV_OK;
}

xv_status xv_block_commit_accepted(xv_block_state* st, const int32_t* n_accept, xv_stream stream) {
    if (!st || !st->ctx_len || !st->n_commit || !n_accept) return fail(XV_ERR_ARG, "commit: null argument");
    if (st->last_k < 1) return fail(XV_ERR_ARG, "commit: no verify to commit");
    xv_status e = commit_launch(n_accept, 1, st->B, st->last_k, st->last_k_seq, st->ctx_len, st->n_commit,
                                reinterpret_cast<cudaStream_t>(stream));
    if (e) return e;
    st->parity ^= 1;
    st->pending_rows = st->last_k;
    st->max_ctx += st->last_k;
    st->last_k = 0;
    st->last_k_seq = nullptr;
    return XV_OK;
}

// Prefill scratch after the verify workspace: the chunk's tokens [B, kmax], argmax [B, kmax],
// n_accept [B] and a zero array [B] (the commit keeps 0 + k positions).
static size_t prefill_extra(int B, int kmax) { return r256(8ull * B * kmax) + 2 * r256(4ull * B); }

size_t xv_block_prefill_workspace_size(const xv_block_config* cfg, int B, int kmax, int Lmax) {
    const size_t v = xv_block_workspace_size(cfg, B, kmax, Lmax);
    return v ? r256(v) + prefill_extra(B, kmax) : 0;
}

xv_status xv_block_prefill(const xv_block_config* cfg, const xv_block_weights* w, xv_block_state* st,
                           const int32_t* tokens, int T, int chunk, float* last_logits, int32_t* last_argmax, void* ws,
                           size_t ws_bytes, xv_stream stream) {
    Dims d{};
    if (xv_status e = check_cfg(cfg, &d)) return e;
    if (xv_status e = check_state(d, cfg, st)) return e;
    if (!tokens || T < 1) return fail(XV_ERR_ARG, "prefill: need tokens and T >= 1");
    if (chunk < 1 || chunk > st->kmax) return fail(XV_ERR_ARG, "prefill: chunk = %d outside [1, kmax = %d]", chunk, st->kmax);
    if (static_cast<long long>(st->B) * chunk > XV_GEMM_M_MAX)
        return fail(XV_ERR_UNSUPPORTED, "prefill: B*chunk = %lld exceeds %d", static_cast<long long>(st->B) * chunk,
                    XV_GEMM_M_MAX);
    if (st->last_k != 0) return fail(XV_ERR_ARG, "prefill: the previous verify has not been committed");
    if (st->max_ctx < 0 || static_cast<long long>(st->max_ctx) + T > st->Lmax)
        return fail(XV_ERR_ARG, "prefill: max_ctx + T exceeds Lmax (%d)", st->Lmax);
    const int B = st->B;
    const size_t vbytes = r256(carve(d, B, st->kmax, st->Lmax, nullptr).total);
    if (!ws || ws_bytes < vbytes + prefill_extra(B, st->kmax))
        return fail(XV_ERR_WORKSPACE, "prefill: workspace of %zu bytes needed", vbytes + prefill_extra(B, st->kmax));
    uint8_t* extra = static_cast<uint8_t*>(ws) + vbytes;
    int32_t* tok = reinterpret_cast<int32_t*>(extra);
    int32_t* am = tok + static_cast<size_t>(B) * st->kmax;
    int32_t* na = reinterpret_cast<int32_t*>(extra + r256(8ull * B * st->kmax));
    int32_t* zeros = reinterpret_cast<int32_t*>(extra + r256(8ull * B * st->kmax) + r256(4ull * B));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (xv_status e = zero_i32_launch(zeros, B, s)) return e;
    const Carve c = carve(d, B, st->kmax, st->Lmax, static_cast<uint8_t*>(ws));
    xv_status e_check = XV_OK;
    for (int t0 = 0; t0 < T; t0 += chunk) {
        const int k = T - t0 < chunk ? T - t0 : chunk;
        const bool last = t0 + k == T;
        // the chunk of every sequence, [B, k]
        if (xv_status e = cuda_check(cudaMemcpy2DAsync(tok, 4ull * k, tokens + t0, 4ull * T, 4ull * k, B,
                                                       cudaMemcpyDeviceToDevice, s),
                                     "prefill: gather the chunk"))
            return e;
        // only the last chunk's logits are read: the others stop before the LM head, and the
        // last one writes its logits (into the workspace) only when the caller asks for them
        float* lg = (last && last_logits) ? c.logits : nullptr;
        if (xv_status e = verify_impl(cfg, w, st, tok, k, nullptr, lg, am, na, ws, vbytes, stream, last)) return e;
        if (last) {
            // the last position of each sequence: row b*k + k - 1
            if (last_logits &&
                (e_check = cuda_check(cudaMemcpy2DAsync(last_logits, 4ull * d.V, c.logits + static_cast<size_t>(k - 1) * d.V,
                                                        4ull * k * d.V, 4ull * d.V, B, cudaMemcpyDeviceToDevice, s),
                                      "prefill: last logits")))
                return e_check;
            if (last_argmax &&
                (e_check = cuda_check(cudaMemcpy2DAsync(last_argmax, 4, am + (k - 1), 4ull * k, 4, B,
                                                        cudaMemcpyDeviceToDevice, s),
                                      "prefill: last argmax")))
                return e_check;
        }
        if (xv_status e = commit_launch(zeros, k, B, k, nullptr, st->ctx_len, st->n_commit, s)) return e;
        st->parity ^= 1;
        st->pending_rows = k;
        st->max_ctx += k;
        st->last_k = 0;
        st->last_k_seq = nullptr;
    }
    return XV_OK;
}

xv_status xv_block_flush(const xv_block_config* cfg, xv_block_state* st, xv_stream stream) {
    Dims d{};
    if (xv_status e = check_cfg(cfg, &d)) return e;
    if (xv_status e = check_state(d, cfg, st)) return e;
    if (st->last_k != 0) return fail(XV_ERR_ARG, "flush: the last verify has not been committed");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int par = st->parity & 1;
    for (int l = 0; l < d.L; ++l) {
        if (cfg->layer_kind[l] != 0) continue;
        xv_layer_state& ls = st->layers[l];
        const uint16_t* ph = ls.gdn_hist[par ^ 1];
        const uint16_t* qkv_pend = ph;
        long long qstride = d.gstride;
        if (d.kc) {
            // the state takes the kept rows; no taps are needed without rows to convolve
            if (xv_status e = conv_launch(ls.gdn_conv_state, ph, d.gstride, st->pending_rows, st->n_commit,
                                          st->pending_rows, nullptr, 0, 0, 0, nullptr, d.cdim, d.kc, st->B, nullptr, 0, s))
                return e;
            qkv_pend = ls.gdn_conv_out[par ^ 1];
            qstride = d.cstride;
        }
        const int qk = d.hk * d.dk;
        GdnStepsDev pend{qkv_pend, qkv_pend + qk, qkv_pend + 2 * qk, ph + d.bcol, ph + d.bcol + d.gh, qstride, d.gstride,
                         st->pending_rows, 1};
        GdnStepsDev none{};
        if (xv_status e = gdn_launch(ls.gdn_state, pend, st->n_commit, 0, st->pending_rows, false, none, 0, nullptr, 0,
                                     st->B, d.gh, d.hk, d.dk, d.dv, 1, s))
            return e;
    }
    return zero_i32_launch(st->n_commit, st->B, s);
}

}  // extern "C"
