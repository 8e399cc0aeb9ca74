// The execution engine behind the C ABI (include/orca.h).
//
// One engine = one model on one GPU.  It borrows the caller's weights, owns
// the K/V pool (allocated once at creation: "論文解説: Orca", implementation
// notes, item 1), the activation buffers sized for max_tokens rows, and the
// scratch of the split-K GEMM and split-K decode attention.  Each call runs
// exactly one iteration (garden.houmin.site Orca notes, 3.1.1): the scheduler
// decides which requests run; the engine only executes.
//
// An iteration is described to the device by a "plan": the batch descriptor
// plus derived tables (prefix-sum row offsets, per-row position and K/V slot,
// decode split-K work items, prefill row tiles), packed into int32 words by
// the host and copied to the device in one transfer.  The plan is what
// replaces explicit split/merge copies: kernels find a request's rows through
// the offsets (selective batching, 3.1.2 of the same notes).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>
#include <type_traits>
#include <unordered_set>
#include <vector>

#include <cstdlib>

#include <nvtx3/nvToolsExt.h>  // header-only; inert unless a profiler attaches

#include "../../include/orca.h"
#include "kernels.cuh"
#include "kvpool.h"

using namespace orca;

namespace {

constexpr int32_t kPlanMagic = 0x4F524341;
constexpr int kHdr = 32;
enum : int {
    P_MAGIC = 0,
    P_NREQ,
    P_NROWS,
    P_NDEC,
    P_NPRE,
    P_NDECWORK,
    P_NPRETILES,
    P_CHUNK,
    P_REQOFF,
    P_REQCTX,
    P_REQKV,
    P_TOKENS,
    P_ROWPOS,
    P_ROWSLOT,
    P_DECWB,
    P_DECNCH,
    P_DECWORK,
    P_PRETILES,
    P_LASTROW,
    P_TOTAL,
    P_PREVN,
    P_DECKEYS,      // sum over decode requests of their keys (ctx + 1)
    P_PREKEYS,      // sum over prefill requests of their keys (ctx + n)
    P_PREPAIRS_HI,  // sum over prefill rows of (pos + 1), split in two words
    P_PREPAIRS_LO,
    P_DECORDER,  // decode work items, longest first
    P_DECITEM,   // their 8-word records (AttnPlan::dec_items)
    P_REQKEYS,   // keys each decode request's work items cover (AttnPlan::req_keys)
    P_PADDED,    // 1: every request padded to the batch's longest input (a conventional batch)
    P_FIELDS
};

// NVTX ranges around every iteration and every kernel launch, named by kind,
// when ORCA_NVTX=1 (read once): a timeline tool then shows the iteration's
// structure.  Off by default.
bool nvtx_on() {
    static const bool on = [] {
        const char *v = getenv("ORCA_NVTX");
        return v && v[0] == '1';
    }();
    return on;
}
const char *kind_name(int kind) {
    static const char *names[] = {"embed",     "layernorm", "gemm_qkv",  "kv_append", "attn_decode", "attn_prefill",
                                  "gemm_o",    "gemm_ffn1", "gemm_ffn2", "lm_head",   "argmax",      "final_ln"};
    return kind >= 0 && kind < (int)(sizeof(names) / sizeof(names[0])) ? names[kind] : "kernel";
}

struct KRec {
    int32_t kind, layer;
    int ev_a, ev_b;
    double bytes, flops;
};

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }
int64_t align4(int64_t w) { return (w + 3) & ~int64_t(3); }

}  // namespace

struct orca_engine {
    orca_model_config cfg{};
    int H = 0, nh = 0, d = 0, F = 0, V = 0, L = 0;
    bool bf = false;
    size_t es = 4;
    cudaStream_t st = nullptr;
    int num_sms = 148;
    bool has_weights = false;
    const void *tok_emb = nullptr, *pos_emb = nullptr;
    const float *lnf_g = nullptr, *lnf_b = nullptr;
    std::vector<orca_layer_weights> layers;
    bool packed = false;  // layers[].w_* and lm_head point into `packed_buf`
    void *packed_buf = nullptr;
    const void *lm_head = nullptr;

    orca::KVPool pool{0};
    void *kv = nullptr;
    float *x = nullptr, *y32 = nullptr, *logits = nullptr;
    void *h = nullptr, *qkv = nullptr, *attn = nullptr, *f = nullptr, *y = nullptr;
    int32_t *next = nullptr;
    int32_t *h_next = nullptr;
    int32_t *h_plan = nullptr, *d_plan = nullptr;
    int64_t plan_cap = 0;
    // GEMM launch contexts: `gs` without a stream-K workspace (the one-tile
    // kernel, and the whole-tile walk for layers of more than one wave of
    // tiles), `gs_op` with one (stream-K allowed: stand-alone orca_op_linear
    // calls and FFN1).  Inside an iteration stream-K proper, which fills every
    // SM, is mostly slower end to end: the one-tile kernel's idle SMs let the
    // next launch start early under programmatic launch.
    GemmScratch gs, gs_op;
    float *part = nullptr;  // split-K partial slabs of the residual projections
    size_t part_cap = 0;
    float *attn_part = nullptr;
    int *attn_cnt = nullptr;
    float *sk_part = nullptr;  // stream-K GEMM: partial tiles of cut tiles
    int *sk_cnt = nullptr;     // stream-K GEMM: per-tile arrival counters
    int64_t attn_part_work = 0;
    unsigned *d_err = nullptr, *h_err = nullptr;

    int built_prev_n = 0;  // n_req of the last plan built (feedback validation)
    int run_prev_n = 0;    // n_req of the last iteration run
    int last_n = 0;
    int64_t iterations = 0, launches = 0;

    bool timing = false;
    std::vector<cudaEvent_t> events;
    size_t ev_next = 0;
    std::vector<KRec> recs;

    ~orca_engine() {
        for (cudaEvent_t e : events) cudaEventDestroy(e);
        void *dev[] = {kv, x, y32, logits, h, qkv, attn, f, y, next, d_plan, part, attn_part, attn_cnt, sk_part, sk_cnt, d_err,
                       packed_buf};
        for (void *p : dev)
            if (p) cudaFree(p);
        if (h_plan) cudaFreeHost(h_plan);
        if (h_next) cudaFreeHost(h_next);
        if (h_err) cudaFreeHost(h_err);
    }

    // Issue one kernel launch (fn), counting it and, when timing is on and the
    // layer is the sampled one, bracketing it with events.
    template <typename Fn>
    int launch(int kind, int layer, double bytes, double flops, Fn fn) {
        const bool rec = timing && (layer < 0 || layer == (int)(iterations % L)) && ev_next + 2 <= events.size();
        int a = 0;
        if (rec) {
            a = (int)ev_next;
            cudaEventRecord(events[ev_next++], st);
        }
        const bool nvtx = nvtx_on();
        if (nvtx) nvtxRangePushA(kind_name(kind));
        cudaError_t e = fn();
        if (nvtx) nvtxRangePop();
        ++launches;
        if (rec) {
            cudaEventRecord(events[ev_next++], st);
            recs.push_back({kind, layer, a, a + 1, bytes, flops});
        }
        return e == cudaSuccess ? ORCA_OK : ORCA_ERR_CUDA;
    }
};

namespace {

// Sizes of one plan; the same function drives both orca_plan_words and the build.
//
// A padded plan runs the batch the conventional way ([houmin] 3.1.2 "问题";
// [arcsin2] 3.2): one [B, Lq] block of rows, every request padded with token 0
// after its own rows to the batch's longest input Lq, and the single-row
// (increment) requests attending over the batch's longest key range with the
// keys past their own context masked.  Pad rows sit at the positions after the
// request's real rows and append their K/V there (inside its reservation,
// overwritten by its next real row); the next token comes from each request's
// last real row, so the results equal the selective batch's.
struct Layout {
    int B, R, n_dec, n_pre, n_dec_work, n_pre_tiles, chunk;
    int padded, lq, lk;  // padded: rows per request and keys per increment request
    int64_t off[P_FIELDS];
};

// Rows request i takes, and the keys its decode items cover.
int rows_of(const Layout &lay, const orca_batch *b, int i) { return lay.padded ? lay.lq : b->n_input[i]; }
int keys_of(const Layout &lay, const orca_batch *b, int i) { return lay.padded ? lay.lk : b->ctx_len[i] + 1; }

// ORCA_DECODE_CHUNK: the largest decode chunk in keys (64 .. 512, a power of
// two; tuning); unset = 512.
int max_decode_chunk() {
    static const int v = [] {
        const char *e = getenv("ORCA_DECODE_CHUNK");
        const int c = e && *e ? atoi(e) : 512;
        return c == 64 || c == 128 || c == 256 ? c : 512;
    }();
    return v;
}

int decode_chunk(const orca_engine *E, const orca_batch *b, const Layout &lay) {
    int chunk = max_decode_chunk();
    // shrink the chunk until the decode grid has a few CTAs per SM
    while (chunk > 64) {
        int64_t items = 0;
        for (int i = 0; i < b->n_req; ++i)
            if (rows_of(lay, b, i) == 1) items += ceil_div(keys_of(lay, b, i), chunk);
        if (items * E->nh >= 4LL * E->num_sms) break;
        chunk /= 2;
    }
    return chunk;
}

int layout(const orca_engine *E, const orca_batch *b, Layout *lay, bool padded) {
    if (!b || b->n_req < 1 || b->n_req > E->cfg.max_batch) return ORCA_ERR_INVALID;
    if (!b->request_id || !b->phase || !b->n_input || !b->ctx_len || !b->kv_offset || !b->tokens)
        return ORCA_ERR_INVALID;
    lay->B = b->n_req;
    lay->padded = padded;
    lay->lq = lay->lk = 0;
    int64_t R = 0;
    for (int i = 0; i < b->n_req; ++i) {
        if (b->n_input[i] < 1 || b->ctx_len[i] < 0) return ORCA_ERR_INVALID;
        R += b->n_input[i];
        lay->lq = std::max(lay->lq, b->n_input[i]);
        lay->lk = std::max(lay->lk, b->ctx_len[i] + 1);
    }
    if (padded) R = (int64_t)lay->lq * b->n_req;
    if (R > E->cfg.max_tokens) return ORCA_ERR_INVALID;
    lay->R = (int)R;
    lay->chunk = decode_chunk(E, b, *lay);
    int nd = 0, np = 0, work = 0, tiles = 0;
    for (int i = 0; i < b->n_req; ++i) {
        const int n = rows_of(*lay, b, i);
        if (n == 1) {
            ++nd;
            work += ceil_div(keys_of(*lay, b, i), lay->chunk);
        } else {
            ++np;
            tiles += ceil_div(n, kPrefillRowsPerTile);
        }
    }
    lay->n_dec = nd, lay->n_pre = np, lay->n_dec_work = work, lay->n_pre_tiles = tiles;
    const int B = lay->B;
    int64_t w = kHdr;
    auto put = [&](int field, int64_t words) {
        lay->off[field] = w;
        w = align4(w + words);
    };
    put(P_REQOFF, B + 1);
    put(P_REQCTX, B);
    put(P_REQKV, B);
    put(P_TOKENS, R);
    put(P_ROWPOS, R);
    put(P_ROWSLOT, R);
    put(P_DECWB, B);
    put(P_DECNCH, B);
    put(P_DECWORK, 2 * (int64_t)work);
    put(P_DECORDER, work);
    put(P_DECITEM, 8 * (int64_t)work);
    put(P_PRETILES, 2 * (int64_t)tiles);
    put(P_LASTROW, B);
    put(P_REQKEYS, B);
    lay->off[P_TOTAL] = w;
    return ORCA_OK;
}

int build(orca_engine *E, const orca_batch *b, int32_t *buf, int64_t cap, bool padded) {
    Layout lay;
    int rc = layout(E, b, &lay, padded);
    if (rc != ORCA_OK) return rc;
    if (!buf || cap < lay.off[P_TOTAL]) return ORCA_ERR_INVALID;
    const int B = lay.B;
    // validation against the model limits and the K/V reservations (a
    // padded request's pad rows must fit them too)
    std::unordered_set<int64_t> seen;
    int64_t tok_i = 0;
    for (int i = 0; i < B; ++i) {
        const int64_t id = b->request_id[i];
        if (!seen.insert(id).second) return ORCA_ERR_INVALID;
        const int n = b->n_input[i], ctx = b->ctx_len[i], rows = rows_of(lay, b, i);
        if (b->phase[i] != (ctx > 0 ? 1 : 0)) return ORCA_ERR_INVALID;
        if ((int64_t)ctx + rows > E->cfg.max_pos) return ORCA_ERR_INVALID;
        int64_t off = 0, len = 0;
        if (!E->pool.lookup(id, &off, &len)) return ORCA_ERR_INVALID;
        if (b->kv_offset[i] != off || (int64_t)ctx + rows > len) return ORCA_ERR_INVALID;
        for (int j = 0; j < n; ++j, ++tok_i) {
            const int32_t t = b->tokens[tok_i];
            if (t >= E->V || (t < 0 && -1 - (int64_t)t >= E->built_prev_n)) return ORCA_ERR_INVALID;
        }
    }
    std::memset(buf, 0, sizeof(int32_t) * kHdr);
    int32_t *req_off = buf + lay.off[P_REQOFF], *req_ctx = buf + lay.off[P_REQCTX], *req_kv = buf + lay.off[P_REQKV];
    int32_t *tokens = buf + lay.off[P_TOKENS], *row_pos = buf + lay.off[P_ROWPOS], *row_slot = buf + lay.off[P_ROWSLOT];
    int32_t *dec_wb = buf + lay.off[P_DECWB], *dec_nch = buf + lay.off[P_DECNCH];
    int32_t *dec_work = buf + lay.off[P_DECWORK], *pre_tiles = buf + lay.off[P_PRETILES];
    int32_t *last_row = buf + lay.off[P_LASTROW], *req_keys = buf + lay.off[P_REQKEYS];
    int r = 0, work = 0, tiles = 0;
    int64_t dec_keys = 0, pre_keys = 0, pre_pairs = 0, src = 0;
    for (int i = 0; i < B; ++i) {
        const int n = rows_of(lay, b, i), real = b->n_input[i], ctx = b->ctx_len[i];
        req_off[i] = r;
        req_ctx[i] = ctx;
        req_kv[i] = (int32_t)b->kv_offset[i];
        req_keys[i] = keys_of(lay, b, i);
        for (int j = 0; j < n; ++j, ++r) {
            tokens[r] = j < real ? b->tokens[src + j] : 0;  // pad rows: token 0
            row_pos[r] = ctx + j;
            row_slot[r] = (int32_t)(b->kv_offset[i] + ctx + j);
        }
        src += real;
        last_row[i] = req_off[i] + real - 1;
        if (n == 1) {
            const int nch = ceil_div(req_keys[i], lay.chunk);
            dec_wb[i] = work;
            dec_nch[i] = nch;
            for (int c = 0; c < nch; ++c, ++work) dec_work[2 * work] = i, dec_work[2 * work + 1] = c;
            dec_keys += req_keys[i];
        } else {
            dec_wb[i] = -1;
            dec_nch[i] = 0;
            for (int q = 0; q < n; q += kPrefillRowsPerTile, ++tiles) pre_tiles[2 * tiles] = i, pre_tiles[2 * tiles + 1] = q;
            pre_keys += ctx + n;
            pre_pairs += (int64_t)n * ctx + (int64_t)n * (n + 1) / 2;
        }
    }
    req_off[B] = r;
    prefill_order(pre_tiles, tiles, req_off, req_ctx);
    decode_order(dec_work, lay.n_dec_work, req_keys, lay.chunk, buf + lay.off[P_DECORDER]);
    decode_items(buf + lay.off[P_DECORDER], dec_work, lay.n_dec_work, req_off, req_keys, req_kv, dec_wb, dec_nch,
                 lay.chunk, buf + lay.off[P_DECITEM]);
    buf[P_MAGIC] = kPlanMagic;
    buf[P_NREQ] = B;
    buf[P_NROWS] = lay.R;
    buf[P_NDEC] = lay.n_dec;
    buf[P_NPRE] = lay.n_pre;
    buf[P_NDECWORK] = lay.n_dec_work;
    buf[P_NPRETILES] = lay.n_pre_tiles;
    buf[P_CHUNK] = lay.chunk;
    for (int f = P_REQOFF; f <= P_TOTAL; ++f) buf[f] = (int32_t)lay.off[f];
    buf[P_PREVN] = E->built_prev_n;
    buf[P_DECKEYS] = (int32_t)std::min<int64_t>(dec_keys, INT32_MAX);
    buf[P_PREKEYS] = (int32_t)std::min<int64_t>(pre_keys, INT32_MAX);
    buf[P_PREPAIRS_HI] = (int32_t)(pre_pairs >> 31);
    buf[P_PREPAIRS_LO] = (int32_t)(pre_pairs & 0x7FFFFFFF);
    buf[P_DECORDER] = (int32_t)lay.off[P_DECORDER];
    buf[P_DECITEM] = (int32_t)lay.off[P_DECITEM];
    buf[P_REQKEYS] = (int32_t)lay.off[P_REQKEYS];
    buf[P_PADDED] = lay.padded;
    E->built_prev_n = B;
    return ORCA_OK;
}

// stream_k: the layer may take the stream-K kernel (E->gs_op carries its
// workspace).  Only FFN1 does inside an iteration: its 160 output tiles at
// the 13B shape quantise worst on 152 SMs, and on the same GPU and trace it
// made prompt-carrying iterations 1 % faster (15.55 -> 15.38 ms, decode-only
// unchanged), where stream-K for QKV as well had cost 2 %.
template <typename T>
cudaError_t linear(orca_engine *E, const void *x, int x_cap, const void *w, int m, int n, int k, const Epilogue &e,
                   int *n_partials = nullptr, bool stream_k = false) {
    if (n_partials) *n_partials = 0;
    if constexpr (std::is_same<T, bf16>::value)
        return gemm_tc_bf16((const bf16 *)x, x_cap, (const bf16 *)w, E->packed, m, n, k, e,
                            stream_k ? E->gs_op : E->gs, E->st, n_partials);
    else
        return gemm_simt_f32((const float *)x, (const float *)w, m, n, k, e, E->st);
}

template <typename T>
int run_plan(orca_engine *E, const int32_t *hp, const int32_t *dp, int32_t *dev_out) {
    const int B = hp[P_NREQ], R = hp[P_NROWS];
    const int H = E->H, F = E->F, V = E->V, nh = E->nh;
    const double es = (double)E->es;
    cudaStream_t st = E->st;
    const int cap = E->cfg.max_tokens;
    AttnPlan ap;
    ap.req_off = dp + hp[P_REQOFF];
    ap.req_ctx = dp + hp[P_REQCTX];
    ap.req_kvoff = dp + hp[P_REQKV];
    ap.dec_work = dp + hp[P_DECWORK];
    ap.dec_wbegin = dp + hp[P_DECWB];
    ap.dec_nch = dp + hp[P_DECNCH];
    ap.dec_order = dp + hp[P_DECORDER];
    ap.dec_items = dp + hp[P_DECITEM];
    ap.pre_tiles = dp + hp[P_PRETILES];
    ap.req_keys = dp + hp[P_REQKEYS];
    ap.n_dec_work = hp[P_NDECWORK];
    ap.n_pre_tiles = hp[P_NPRETILES];
    ap.chunk = hp[P_CHUNK];
    ap.n_rows = hp[P_NROWS];
    ap.claim = decode_claim_enabled() ? E->attn_cnt + (size_t)E->cfg.max_batch * E->cfg.n_heads : nullptr;
    const int32_t *tokens = dp + hp[P_TOKENS], *row_pos = dp + hp[P_ROWPOS], *row_slot = dp + hp[P_ROWSLOT];
    const int32_t *last_row = dp + hp[P_LASTROW];
    const double dec_keys = hp[P_DECKEYS], pre_keys = hp[P_PREKEYS];
    const double pre_pairs = (double)(((int64_t)hp[P_PREPAIRS_HI] << 31) | (int64_t)hp[P_PREPAIRS_LO]);
    const int prev_n = E->run_prev_n;
    T *h = (T *)E->h, *qkv = (T *)E->qkv, *attn = (T *)E->attn, *f = (T *)E->f, *y = (T *)E->y;
    const int64_t layer_elems = 2LL * nh * E->cfg.kv_slots * E->d;
    int rc;

#define ORCA_TRY(expr)               \
    do {                             \
        rc = (expr);                 \
        if (rc != ORCA_OK) return rc; \
    } while (0)

    ORCA_TRY(E->launch(ORCA_K_EMBED, -1, R * H * (2 * es + 4), 0, [&] {
        return embed<T>(tokens, row_pos, E->next, prev_n, (const T *)E->tok_emb, (const T *)E->pos_emb, E->x, R, H,
                        V, E->cfg.max_pos, E->d_err, st);
    }));
    // split-K partial slabs of the last residual projection, completed by the next LayerNorm
    int pend_n = 0;
    const float *pend_bias = nullptr;
    const bool bf = std::is_same<T, bf16>::value;
    for (int l = 0; l < E->L; ++l) {
        const orca_layer_weights &W = E->layers[l];
        T *pool_l = (T *)E->kv + (size_t)l * layer_elems;
        ORCA_TRY(E->launch(ORCA_K_LN, l, R * H * (4 + es) + 4.0 * R * H * (pend_n ? pend_n + 1 : 0), 0, [&] {
            return layernorm<T>(E->x, nullptr, W.ln1_g, W.ln1_b, h, nullptr, R, H, st, E->part, pend_n, R, pend_bias);
        }));
        {
            Epilogue e;
            e.bias = W.b_qkv;
            if (bf) {
                e.out_bf16 = (bf16 *)qkv;
                // k and v rows go straight to the pool at each row's slot (the K/V append)
                e.kv_pool = (bf16 *)pool_l;
                e.row_slot = row_slot;
                e.kv_slots = E->cfg.kv_slots;
                e.kv_h = H, e.kv_hd = E->d, e.kv_nh = nh;
            } else {
                e.out_f32 = (float *)qkv;
            }
            e.ld_out = 3 * H;
            ORCA_TRY(E->launch(ORCA_K_GEMM_QKV, l, es * (3.0 * H * H + (double)R * H + 3.0 * R * H),
                               2.0 * R * 3 * H * H, [&] { return linear<T>(E, h, cap, W.w_qkv, R, 3 * H, H, e); }));
        }
        if (!bf)
            ORCA_TRY(E->launch(ORCA_K_KV_APPEND, l, 4.0 * R * H * es, 0, [&] {
                return kv_append<T>(qkv, row_slot, pool_l, E->cfg.kv_slots, R, H, nh, st);
            }));
        if (ap.n_dec_work > 0)
            ORCA_TRY(E->launch(ORCA_K_ATTN_DECODE, l, es * (2.0 * dec_keys * H + 2.0 * hp[P_NDEC] * H),
                               4.0 * dec_keys * H, [&] {
                                   return attention<T>(qkv, pool_l, E->cfg.kv_slots, attn, ap, H, nh, E->attn_part,
                                                       E->attn_cnt, E->d_err, st, true, false);
                               }));
        if (ap.n_pre_tiles > 0)
            ORCA_TRY(E->launch(ORCA_K_ATTN_PREFILL, l, es * (2.0 * pre_keys * H + 2.0 * (R - hp[P_NDEC]) * H),
                               4.0 * pre_pairs * H, [&] {
                                   return attention<T>(qkv, pool_l, E->cfg.kv_slots, attn, ap, H, nh, E->attn_part,
                                                       E->attn_cnt, E->d_err, st, false, true);
                               }));
        int np_o = 0;
        {
            Epilogue e;
            e.bias = W.b_o;
            e.resid = E->x;
            e.out_f32 = E->x;
            e.ld_out = H;
            e.part = E->part;
            e.part_cap = E->part_cap;
            ORCA_TRY(E->launch(ORCA_K_GEMM_O, l, es * ((double)H * H + (double)R * H) + 8.0 * R * H,
                               2.0 * R * H * H, [&] { return linear<T>(E, attn, cap, W.w_o, R, H, H, e, &np_o); }));
        }
        ORCA_TRY(E->launch(ORCA_K_LN, l, R * H * (4 + es) + 4.0 * R * H * (np_o ? np_o + 1 : 0), 0, [&] {
            return layernorm<T>(E->x, nullptr, W.ln2_g, W.ln2_b, h, nullptr, R, H, st, E->part, np_o, R, W.b_o);
        }));
        {
            Epilogue e;
            e.bias = W.b_1;
            e.gelu = 1;
            if (std::is_same<T, bf16>::value) e.out_bf16 = (bf16 *)f; else e.out_f32 = (float *)f;
            e.ld_out = F;
            ORCA_TRY(E->launch(ORCA_K_GEMM_FFN1, l, es * ((double)F * H + (double)R * H + (double)R * F),
                               2.0 * R * F * H, [&] { return linear<T>(E, h, cap, W.w_1, R, F, H, e, nullptr, true); }));
        }
        {
            Epilogue e;
            e.bias = W.b_2;
            e.resid = E->x;
            e.out_f32 = E->x;
            e.ld_out = H;
            e.part = E->part;
            e.part_cap = E->part_cap;
            ORCA_TRY(E->launch(ORCA_K_GEMM_FFN2, l, es * ((double)H * F + (double)R * F) + 8.0 * R * H,
                               2.0 * R * H * F, [&] { return linear<T>(E, f, cap, W.w_2, R, H, F, e, &pend_n); }));
            pend_bias = W.b_2;
        }
    }
    ORCA_TRY(E->launch(ORCA_K_FINAL_LN, -1, B * H * (8 + es) + 4.0 * B * H * (pend_n ? pend_n + 1 : 0), 0, [&] {
        return layernorm<T>(E->x, last_row, E->lnf_g, E->lnf_b, y, E->y32, B, H, st, E->part, pend_n, R, pend_bias);
    }));
    {
        Epilogue e;
        e.out_f32 = E->logits;
        e.ld_out = V;
        ORCA_TRY(E->launch(ORCA_K_LM_HEAD, -1, es * ((double)V * H + (double)B * H) + 4.0 * B * V,
                           2.0 * B * V * H, [&] { return linear<T>(E, y, E->cfg.max_batch, E->lm_head, B, V, H, e); }));
    }
    ORCA_TRY(E->launch(ORCA_K_ARGMAX, -1, 4.0 * B * V, 0,
                       [&] { return argmax_rows(E->logits, B, V, E->next, dev_out, st); }));
#undef ORCA_TRY
    E->run_prev_n = B;
    E->last_n = B;
    E->iterations++;
    return ORCA_OK;
}

int run_planned_impl(orca_engine *E, const int32_t *hp, const int32_t *dp, int32_t *dev_out) {
    if (!E->has_weights || !hp || !dp || hp[P_MAGIC] != kPlanMagic) return ORCA_ERR_INVALID;
    if (hp[P_PREVN] != E->run_prev_n) return ORCA_ERR_INVALID;  // plans must run in build order
    const bool nvtx = nvtx_on();
    if (nvtx) nvtxRangePushA("iteration");
    const int rc = E->bf ? run_plan<bf16>(E, hp, dp, dev_out) : run_plan<float>(E, hp, dp, dev_out);
    if (nvtx) nvtxRangePop();
    return rc;
}

int check_flag(orca_engine *E) {
    if (*E->h_err == 0) return ORCA_OK;
    *E->h_err = 0;
    cudaMemsetAsync(E->d_err, 0, sizeof(unsigned), E->st);
    // a kernel that gave up may have left split-request arrival counters or the
    // decode work-claim counters part-way
    cudaMemsetAsync(E->attn_cnt, 0, ((size_t)E->cfg.max_batch * E->cfg.n_heads + 2) * 4, E->st);
    if (E->sk_cnt) cudaMemsetAsync(E->sk_cnt, 0, (size_t)E->gs_op.sk_cnt_n * 4, E->st);
    cudaStreamSynchronize(E->st);
    return ORCA_ERR_DEVICE_FLAG;
}

template <typename P>
int dev_alloc(P **p, size_t bytes) {
    if (cudaMalloc((void **)p, std::max<size_t>(bytes, 16)) != cudaSuccess) {
        *p = nullptr;
        cudaGetLastError();
        return ORCA_ERR_OOM;
    }
    return ORCA_OK;
}

}  // namespace

extern "C" {

const char *orca_strerror(int code) {
    switch (code) {
        case ORCA_OK: return "ok";
        case ORCA_ERR_INVALID: return "invalid argument or batch descriptor";
        case ORCA_ERR_KV_FULL: return "K/V pool has no free range of that size";
        case ORCA_ERR_CUDA: return "CUDA call failed";
        case ORCA_ERR_DEVICE_FLAG: return "a kernel recorded an error";
        case ORCA_ERR_NOT_FOUND: return "unknown request id";
        case ORCA_ERR_OOM: return "allocation failed";
        case ORCA_ERR_LIMIT: return "sizes exceed the fixed scratch of the allocation-free entry point";
        default: return "unknown status";
    }
}

int orca_engine_create(const orca_model_config *cfg, const orca_weights *w, void *stream, orca_engine **out) {
    if (!cfg || !out) return ORCA_ERR_INVALID;
    *out = nullptr;
    const orca_model_config &c = *cfg;
    if (c.n_layers < 1 || c.hidden < 8 || c.n_heads < 1 || c.hidden % c.n_heads || c.ffn < 1 || c.vocab < 1 ||
        c.max_pos < 1 || c.max_tokens < 1 || c.max_batch < 1 || c.kv_slots < 1 || c.kv_slots > INT32_MAX)
        return ORCA_ERR_INVALID;
    const int d = c.hidden / c.n_heads;
    if ((d != 16 && d != 32 && d != 64 && d != 128) || c.hidden % 8 || c.hidden > 8192) return ORCA_ERR_INVALID;
    if (c.dtype != ORCA_DTYPE_FP32 && c.dtype != ORCA_DTYPE_BF16) return ORCA_ERR_INVALID;
    if (c.dtype == ORCA_DTYPE_BF16 && (c.hidden % 64 || c.ffn % 64)) return ORCA_ERR_INVALID;
    orca_engine *E = new (std::nothrow) orca_engine();
    if (!E) return ORCA_ERR_OOM;
    E->cfg = c;
    E->H = c.hidden, E->nh = c.n_heads, E->d = d, E->F = c.ffn, E->V = c.vocab, E->L = c.n_layers;
    E->bf = c.dtype == ORCA_DTYPE_BF16;
    E->es = E->bf ? 2 : 4;
    E->st = (cudaStream_t)stream;
    E->pool = orca::KVPool(c.kv_slots);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&E->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        delete E;
        return ORCA_ERR_CUDA;
    }
    if (w) {
        if (!w->tok_emb || !w->pos_emb || !w->lnf_g || !w->lnf_b || !w->layers) {
            delete E;
            return ORCA_ERR_INVALID;
        }
        E->has_weights = true;
        E->tok_emb = w->tok_emb, E->pos_emb = w->pos_emb, E->lnf_g = w->lnf_g, E->lnf_b = w->lnf_b;
        E->layers.assign(w->layers, w->layers + c.n_layers);
        E->lm_head = w->tok_emb;
    }
    const size_t R = c.max_tokens, B = c.max_batch, H = c.hidden, F = c.ffn, es = E->es;
    // decode split-K work items: at most one per 64 keys of every request
    E->attn_part_work = (int64_t)B * ceil_div(c.max_pos, 64);
    E->plan_cap = kHdr + 64 + 8 * (int64_t)B + 3 * (int64_t)R + 11 * E->attn_part_work + 2 * ((int64_t)R / 16 + B);
    E->gs.num_sms = E->num_sms;
    // up to 8 partial slabs of up to 512 rows (split-K is only chosen when the rows are few)
    E->part_cap = E->bf ? (size_t)8 * std::min<size_t>(R, 512) * H : 0;
    int rc = ORCA_OK;
    const size_t kv_bytes = (size_t)c.n_layers * 2 * H * (size_t)c.kv_slots * es;
    if (rc == ORCA_OK) rc = dev_alloc(&E->kv, kv_bytes);
    if (rc == ORCA_OK) rc = dev_alloc(&E->x, R * H * 4);
    if (rc == ORCA_OK) rc = dev_alloc(&E->h, R * H * es);
    if (rc == ORCA_OK) rc = dev_alloc(&E->qkv, R * 3 * H * es);
    if (rc == ORCA_OK) rc = dev_alloc(&E->attn, R * H * es);
    if (rc == ORCA_OK) rc = dev_alloc(&E->f, R * F * es);
    if (rc == ORCA_OK) rc = dev_alloc(&E->y, B * H * es);
    if (rc == ORCA_OK) rc = dev_alloc(&E->y32, B * H * 4);
    if (rc == ORCA_OK) rc = dev_alloc(&E->logits, B * (size_t)c.vocab * 4);
    if (rc == ORCA_OK) rc = dev_alloc(&E->next, B * 4);
    if (rc == ORCA_OK) rc = dev_alloc(&E->d_plan, (size_t)E->plan_cap * 4);
    if (rc == ORCA_OK && E->part_cap) rc = dev_alloc(&E->part, E->part_cap * 4);
    if (rc == ORCA_OK) rc = dev_alloc(&E->attn_part, (size_t)E->attn_part_work * c.n_heads * (d + 2) * 4);
    // per-(request, head) arrival counters, then the decode kernel's two work-claim counters
    if (rc == ORCA_OK) rc = dev_alloc(&E->attn_cnt, (B * c.n_heads + 2) * 4);
    if (rc == ORCA_OK && E->bf) {
        // stream-K GEMM workspace (token rows of any linear layer, the LM head's included)
        E->gs_op.sk_part_floats = gemm_sk_part_floats(E->num_sms);
        E->gs_op.sk_cnt_n = gemm_sk_counters((int)R, std::max({3 * c.hidden, c.ffn, c.vocab}));
        rc = dev_alloc(&E->sk_part, E->gs_op.sk_part_floats * 4);
        if (rc == ORCA_OK) rc = dev_alloc(&E->sk_cnt, (size_t)E->gs_op.sk_cnt_n * 4);
        if (rc == ORCA_OK && cudaMemset(E->sk_cnt, 0, (size_t)E->gs_op.sk_cnt_n * 4) != cudaSuccess)
            rc = ORCA_ERR_CUDA;
        E->gs_op.sk_part = E->sk_part;
        E->gs_op.sk_cnt = E->sk_cnt;
    }
    if (rc == ORCA_OK) rc = dev_alloc(&E->d_err, 4);
    if (rc == ORCA_OK && (cudaMallocHost((void **)&E->h_plan, (size_t)E->plan_cap * 4) != cudaSuccess ||
                          cudaMallocHost((void **)&E->h_next, B * 4) != cudaSuccess ||
                          cudaMallocHost((void **)&E->h_err, 4) != cudaSuccess))
        rc = ORCA_ERR_OOM;
    if (rc == ORCA_OK) {
        *E->h_err = 0;
        E->gs.err = E->d_err;
        E->gs_op.err = E->d_err;
        E->gs_op.num_sms = E->num_sms;
        if (cudaMemset(E->attn_cnt, 0, (B * c.n_heads + 2) * 4) != cudaSuccess || cudaMemset(E->d_err, 0, 4) != cudaSuccess ||
            cudaMemset(E->next, 0, B * 4) != cudaSuccess)
            rc = ORCA_ERR_CUDA;
    }
    if (rc == ORCA_OK && E->has_weights && E->bf && c.pack_weights) {
        // one engine-owned buffer with every matrix repacked tile-contiguous
        const int Hh = c.hidden, Ff = c.ffn;
        const size_t per_layer = packed_weight_elems(3 * Hh, Hh) + packed_weight_elems(Hh, Hh) +
                                 packed_weight_elems(Ff, Hh) + packed_weight_elems(Hh, Ff);
        const size_t total = per_layer * c.n_layers + packed_weight_elems(c.vocab, Hh);
        rc = dev_alloc(&E->packed_buf, total * 2);
        bf16 *p = (bf16 *)E->packed_buf;
        auto pack = [&](const void *src, int n, int k) -> const void * {
            if (rc != ORCA_OK) return src;
            if (pack_weight_bf16((const bf16 *)src, n, k, p, E->st) != cudaSuccess) rc = ORCA_ERR_CUDA;
            const void *dst = p;
            p += packed_weight_elems(n, k);
            return dst;
        };
        for (int l = 0; l < c.n_layers && rc == ORCA_OK; ++l) {
            orca_layer_weights &L = E->layers[l];
            L.w_qkv = pack(L.w_qkv, 3 * Hh, Hh);
            L.w_o = pack(L.w_o, Hh, Hh);
            L.w_1 = pack(L.w_1, Ff, Hh);
            L.w_2 = pack(L.w_2, Hh, Ff);
        }
        E->lm_head = pack(E->tok_emb, c.vocab, Hh);
        if (rc == ORCA_OK && cudaStreamSynchronize(E->st) != cudaSuccess) rc = ORCA_ERR_CUDA;
        E->packed = rc == ORCA_OK;
    }
    if (rc != ORCA_OK) {
        cudaGetLastError();
        delete E;
        return rc;
    }
    *out = E;
    return ORCA_OK;
}

int64_t orca_packed_weight_elems(int32_t n_out, int32_t k) {
    if (n_out < 1 || k < 64 || k % 64) return ORCA_ERR_INVALID;
    return (int64_t)packed_weight_elems(n_out, k);
}

int orca_pack_weight(orca_engine *E, const void *w, int32_t n_out, int32_t k, void *out) {
    if (!E || !w || !out || n_out < 1 || k < 64 || k % 64) return ORCA_ERR_INVALID;
    if (pack_weight_bf16((const bf16 *)w, n_out, k, (bf16 *)out, E->st) != cudaSuccess) {
        cudaGetLastError();
        return ORCA_ERR_CUDA;
    }
    E->launches++;
    return ORCA_OK;
}

int orca_engine_destroy(orca_engine *E) {
    if (!E) return ORCA_ERR_INVALID;
    cudaStreamSynchronize(E->st);
    delete E;
    return ORCA_OK;
}

int orca_kv_alloc(orca_engine *E, int64_t id, int32_t n, int64_t *out_offset) {
    if (!E || !out_offset) return ORCA_ERR_INVALID;
    const int64_t off = E->pool.alloc(id, n);
    if (off == -1) return ORCA_ERR_KV_FULL;
    if (off < 0) return ORCA_ERR_INVALID;
    *out_offset = off;
    return ORCA_OK;
}

int orca_kv_free(orca_engine *E, int64_t id) {
    if (!E) return ORCA_ERR_INVALID;
    return E->pool.release(id) ? ORCA_OK : ORCA_ERR_NOT_FOUND;
}

int orca_kv_layout_get(orca_engine *E, orca_kv_layout *out) {
    if (!E || !out) return ORCA_ERR_INVALID;
    out->base = E->kv;
    out->kv_slots = E->cfg.kv_slots;
    out->n_layers = E->L;
    out->n_heads = E->nh;
    out->head_dim = E->d;
    out->elem_bytes = (int32_t)E->es;
    return ORCA_OK;
}

int64_t orca_plan_words(const orca_engine *E, const orca_batch *b) {
    if (!E) return ORCA_ERR_INVALID;
    Layout lay;
    const int rc = layout(E, b, &lay, false);
    return rc == ORCA_OK ? lay.off[P_TOTAL] : rc;
}

int orca_plan_build(orca_engine *E, const orca_batch *b, int32_t *host_buf, int64_t cap_words) {
    if (!E) return ORCA_ERR_INVALID;
    return build(E, b, host_buf, cap_words, false);
}

int64_t orca_plan_words_padded(const orca_engine *E, const orca_batch *b) {
    if (!E) return ORCA_ERR_INVALID;
    Layout lay;
    const int rc = layout(E, b, &lay, true);
    return rc == ORCA_OK ? lay.off[P_TOTAL] : rc;
}

int orca_plan_build_padded(orca_engine *E, const orca_batch *b, int32_t *host_buf, int64_t cap_words) {
    if (!E) return ORCA_ERR_INVALID;
    return build(E, b, host_buf, cap_words, true);
}

int orca_run_planned(orca_engine *E, const int32_t *host_plan, const int32_t *dev_plan, int32_t *dev_out_next) {
    if (!E) return ORCA_ERR_INVALID;
    return run_planned_impl(E, host_plan, dev_plan, dev_out_next);
}

int orca_engine_sync(orca_engine *E) {
    if (!E) return ORCA_ERR_INVALID;
    if (cudaMemcpyAsync(E->h_err, E->d_err, 4, cudaMemcpyDeviceToHost, E->st) != cudaSuccess ||
        cudaStreamSynchronize(E->st) != cudaSuccess) {
        cudaGetLastError();
        return ORCA_ERR_CUDA;
    }
    return check_flag(E);
}

namespace {
int run_iteration_impl(orca_engine *E, const orca_batch *b, int32_t *out_next, bool padded) {
    if (!E || !out_next || !E->has_weights) return ORCA_ERR_INVALID;
    const int saved_prev = E->built_prev_n;
    E->built_prev_n = E->run_prev_n;  // feedback refers to the last iteration actually run
    int rc = build(E, b, E->h_plan, E->plan_cap, padded);
    if (rc != ORCA_OK) {
        E->built_prev_n = saved_prev;
        return rc;
    }
    const int B = b->n_req;
    if (cudaMemcpyAsync(E->d_plan, E->h_plan, (size_t)E->h_plan[P_TOTAL] * 4, cudaMemcpyHostToDevice, E->st) !=
        cudaSuccess) {
        cudaGetLastError();
        return ORCA_ERR_CUDA;
    }
    rc = run_planned_impl(E, E->h_plan, E->d_plan, nullptr);
    if (rc != ORCA_OK) return rc;
    if (cudaMemcpyAsync(E->h_next, E->next, (size_t)B * 4, cudaMemcpyDeviceToHost, E->st) != cudaSuccess ||
        cudaMemcpyAsync(E->h_err, E->d_err, 4, cudaMemcpyDeviceToHost, E->st) != cudaSuccess ||
        cudaStreamSynchronize(E->st) != cudaSuccess) {
        cudaGetLastError();
        return ORCA_ERR_CUDA;
    }
    rc = check_flag(E);
    if (rc != ORCA_OK) return rc;
    std::memcpy(out_next, E->h_next, (size_t)B * 4);
    return ORCA_OK;
}
}  // namespace

int orca_run_iteration(orca_engine *E, const orca_batch *b, int32_t *out_next) {
    return run_iteration_impl(E, b, out_next, false);
}

int orca_run_iteration_padded(orca_engine *E, const orca_batch *b, int32_t *out_next) {
    return run_iteration_impl(E, b, out_next, true);
}

int orca_get_last_hidden(orca_engine *E, float *host_out, int64_t n) {
    if (!E || !host_out) return ORCA_ERR_INVALID;
    const int64_t need = (int64_t)E->last_n * E->H;
    if (n < need) return ORCA_ERR_INVALID;
    if (cudaMemcpyAsync(host_out, E->y32, need * 4, cudaMemcpyDeviceToHost, E->st) != cudaSuccess ||
        cudaStreamSynchronize(E->st) != cudaSuccess) {
        cudaGetLastError();
        return ORCA_ERR_CUDA;
    }
    return ORCA_OK;
}

int orca_get_last_logits(orca_engine *E, float *host_out, int64_t n) {
    if (!E || !host_out) return ORCA_ERR_INVALID;
    const int64_t need = (int64_t)E->last_n * E->V;
    if (n < need) return ORCA_ERR_INVALID;
    if (cudaMemcpyAsync(host_out, E->logits, need * 4, cudaMemcpyDeviceToHost, E->st) != cudaSuccess ||
        cudaStreamSynchronize(E->st) != cudaSuccess) {
        cudaGetLastError();
        return ORCA_ERR_CUDA;
    }
    return ORCA_OK;
}

int orca_engine_stats_get(orca_engine *E, orca_engine_stats *out) {
    if (!E || !out) return ORCA_ERR_INVALID;
    out->launches = E->launches;
    out->iterations = E->iterations;
    return ORCA_OK;
}

int orca_engine_timing(orca_engine *E, int32_t enable) {
    if (!E) return ORCA_ERR_INVALID;
    if (enable && E->events.empty()) {
        E->events.resize(16384);
        for (auto &e : E->events)
            if (cudaEventCreate(&e) != cudaSuccess) {
                cudaGetLastError();
                return ORCA_ERR_CUDA;
            }
    }
    E->timing = enable != 0;
    return ORCA_OK;
}

int orca_engine_timing_read(orca_engine *E, orca_kernel_time *out, int32_t cap, int32_t *n_out) {
    if (!E || !n_out || (cap > 0 && !out)) return ORCA_ERR_INVALID;
    if (cudaStreamSynchronize(E->st) != cudaSuccess) {
        cudaGetLastError();
        return ORCA_ERR_CUDA;
    }
    int32_t n = 0;
    for (const KRec &r : E->recs) {
        if (n >= cap) break;
        float ms = 0.f;
        cudaEventElapsedTime(&ms, E->events[r.ev_a], E->events[r.ev_b]);
        out[n++] = {r.kind, r.layer, ms, r.bytes, r.flops};
    }
    *n_out = n;
    E->recs.clear();
    E->ev_next = 0;
    return ORCA_OK;
}

int orca_debug_expire_wait(orca_engine *E, int64_t limit_ns) {
    if (!E || limit_ns < 1 || limit_ns > 10000000000LL) return ORCA_ERR_INVALID;
    if (expire_wait((unsigned long long)limit_ns, E->d_err, E->st) != cudaSuccess) {
        cudaGetLastError();
        return ORCA_ERR_CUDA;
    }
    E->launches++;
    return ORCA_OK;
}

int orca_op_attention(orca_engine *E, int32_t dtype, const void *qkv, const void *kv_layer, int64_t kv_slots,
                      int32_t n_heads, int32_t head_dim, int32_t n_req, const int32_t *n_input,
                      const int32_t *ctx_len, const int64_t *kv_offset, void *out) {
    if (!E || !qkv || !kv_layer || !out || !n_input || !ctx_len || !kv_offset) return ORCA_ERR_INVALID;
    if (n_req < 1 || n_req > E->cfg.max_batch || n_heads < 1 || kv_slots < 1 || kv_slots > INT32_MAX)
        return ORCA_ERR_INVALID;
    if (head_dim != 16 && head_dim != 32 && head_dim != 64 && head_dim != 128) return ORCA_ERR_INVALID;
    if (dtype != ORCA_DTYPE_FP32 && dtype != ORCA_DTYPE_BF16) return ORCA_ERR_INVALID;
    if (n_heads > E->nh) return ORCA_ERR_INVALID;  // split-K counters are sized for the engine's heads
    // describe the batch through the iteration's layout rules (ids and tokens are not read)
    std::vector<int64_t> ids(n_req);
    std::vector<int32_t> phase(n_req);
    int64_t rows = 0;
    for (int i = 0; i < n_req; ++i) {
        if (n_input[i] < 1 || ctx_len[i] < 0 || kv_offset[i] < 0 ||
            kv_offset[i] + (int64_t)ctx_len[i] + n_input[i] > kv_slots)
            return ORCA_ERR_INVALID;
        ids[i] = i;
        phase[i] = ctx_len[i] > 0;
        rows += n_input[i];
    }
    std::vector<int32_t> toks((size_t)rows, 0);
    orca_batch b{n_req, ids.data(), phase.data(), n_input, ctx_len, kv_offset, toks.data()};
    Layout lay;
    int rc = layout(E, &b, &lay, false);
    if (rc != ORCA_OK) return rc;
    if (lay.off[P_TOTAL] > E->plan_cap ||
        (int64_t)lay.n_dec_work * n_heads * (head_dim + 2) > E->attn_part_work * E->nh * (E->d + 2))
        return ORCA_ERR_INVALID;
    // the engine's plan buffers are reused: wait for any iteration still reading them
    if (cudaStreamSynchronize(E->st) != cudaSuccess) {
        cudaGetLastError();
        return ORCA_ERR_CUDA;
    }
    int32_t *buf = E->h_plan;
    int32_t *req_off = buf + lay.off[P_REQOFF], *req_ctx = buf + lay.off[P_REQCTX], *req_kv = buf + lay.off[P_REQKV];
    int32_t *dec_wb = buf + lay.off[P_DECWB], *dec_nch = buf + lay.off[P_DECNCH];
    int32_t *dec_work = buf + lay.off[P_DECWORK], *pre_tiles = buf + lay.off[P_PRETILES];
    int32_t *req_keys = buf + lay.off[P_REQKEYS];
    int r = 0, work = 0, tiles = 0;
    for (int i = 0; i < n_req; ++i) {
        req_off[i] = r;
        req_ctx[i] = ctx_len[i];
        req_kv[i] = (int32_t)kv_offset[i];
        req_keys[i] = ctx_len[i] + 1;
        if (n_input[i] == 1) {
            const int nch = ceil_div((int64_t)ctx_len[i] + 1, lay.chunk);
            dec_wb[i] = work;
            dec_nch[i] = nch;
            for (int c = 0; c < nch; ++c, ++work) dec_work[2 * work] = i, dec_work[2 * work + 1] = c;
        } else {
            dec_wb[i] = -1;
            dec_nch[i] = 0;
            for (int q = 0; q < n_input[i]; q += kPrefillRowsPerTile, ++tiles)
                pre_tiles[2 * tiles] = i, pre_tiles[2 * tiles + 1] = q;
        }
        r += n_input[i];
    }
    req_off[n_req] = r;
    prefill_order(pre_tiles, tiles, req_off, req_ctx);
    decode_order(dec_work, lay.n_dec_work, req_keys, lay.chunk, buf + lay.off[P_DECORDER]);
    decode_items(buf + lay.off[P_DECORDER], dec_work, lay.n_dec_work, req_off, req_keys, req_kv, dec_wb, dec_nch,
                 lay.chunk, buf + lay.off[P_DECITEM]);
    if (cudaMemcpyAsync(E->d_plan, E->h_plan, (size_t)lay.off[P_TOTAL] * 4, cudaMemcpyHostToDevice, E->st) !=
        cudaSuccess) {
        cudaGetLastError();
        return ORCA_ERR_CUDA;
    }
    const int32_t *dp = E->d_plan;
    AttnPlan ap;
    ap.req_off = dp + lay.off[P_REQOFF];
    ap.req_ctx = dp + lay.off[P_REQCTX];
    ap.req_kvoff = dp + lay.off[P_REQKV];
    ap.dec_work = dp + lay.off[P_DECWORK];
    ap.dec_wbegin = dp + lay.off[P_DECWB];
    ap.dec_nch = dp + lay.off[P_DECNCH];
    ap.dec_order = dp + lay.off[P_DECORDER];
    ap.dec_items = dp + lay.off[P_DECITEM];
    ap.pre_tiles = dp + lay.off[P_PRETILES];
    ap.req_keys = dp + lay.off[P_REQKEYS];
    ap.n_dec_work = lay.n_dec_work;
    ap.n_pre_tiles = lay.n_pre_tiles;
    ap.chunk = lay.chunk;
    ap.n_rows = (int)rows;
    ap.claim = decode_claim_enabled() ? E->attn_cnt + (size_t)E->cfg.max_batch * E->cfg.n_heads : nullptr;
    const int H = n_heads * head_dim;
    cudaError_t ce;
    if (dtype == ORCA_DTYPE_BF16)
        ce = attention<bf16>((const bf16 *)qkv, (const bf16 *)kv_layer, kv_slots, (bf16 *)out, ap, H, n_heads,
                             E->attn_part, E->attn_cnt, E->d_err, E->st, true, true);
    else
        ce = attention<float>((const float *)qkv, (const float *)kv_layer, kv_slots, (float *)out, ap, H, n_heads,
                              E->attn_part, E->attn_cnt, E->d_err, E->st, true, true);
    E->launches += (ap.n_dec_work > 0) + (ap.n_pre_tiles > 0);
    if (ce != cudaSuccess) {
        cudaGetLastError();
        return ORCA_ERR_CUDA;
    }
    return ORCA_OK;
}

int orca_op_linear(orca_engine *E, int32_t dtype, const void *x, const void *w, int32_t w_packed, int32_t m,
                   int32_t n, int32_t k, const float *bias, int32_t gelu, const float *resid, float *out_f32,
                   void *out_bf16, int32_t ld_out) {
    if (!E || !x || !w || m < 0 || n < 1 || k < 1 || ld_out < n) return ORCA_ERR_INVALID;
    if ((out_f32 != nullptr) == (out_bf16 != nullptr) || (resid && !out_f32)) return ORCA_ERR_INVALID;
    Epilogue e;
    e.bias = bias;
    e.gelu = gelu;
    e.resid = resid;
    e.out_f32 = out_f32;
    e.out_bf16 = (bf16 *)out_bf16;
    e.ld_out = ld_out;
    cudaError_t ce;
    if (dtype == ORCA_DTYPE_BF16) {
        if (k % 64) return ORCA_ERR_INVALID;
        ce = gemm_tc_bf16((const bf16 *)x, m, (const bf16 *)w, w_packed != 0, m, n, k, e, E->gs_op, E->st);
    } else if (dtype == ORCA_DTYPE_FP32) {
        if (out_bf16 || w_packed) return ORCA_ERR_INVALID;
        ce = gemm_simt_f32((const float *)x, (const float *)w, m, n, k, e, E->st);
    } else {
        return ORCA_ERR_INVALID;
    }
    E->launches++;
    if (ce != cudaSuccess) {
        cudaGetLastError();
        return ORCA_ERR_CUDA;
    }
    return ORCA_OK;
}

}  // extern "C"
