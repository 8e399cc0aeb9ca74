// Attention of one layer, split per request and merged back by indexing.
//
// Selective batching ("論文解説: Orca", Selective Batching; garden.houmin.site
// Orca notes, 3.1.2 "方案"): the [sum L, 3H] projection is split by request,
// attention runs per request over that request's own K/V, and the outputs are
// merged back into [sum L, H].  Here the split and the merge are the prefix-sum
// row offsets: each CTA reads its request's q rows straight out of the qkv
// matrix and writes its output rows straight into the attention matrix, so no
// copy is made.  The page notes that attention has no weights to share across
// requests, so not batching it costs little; what it costs is the K/V read,
// which is what these kernels stream.
//
// K/V pool layout per layer: [K|V][head][slot][head_dim], so the keys of one
// head of one request are contiguous (head_dim * elem bytes per token).
//
// decode  : requests with one input row (increment phase).  Work item =
//           (request, chunk of `chunk` keys) x head, its K/V rows streamed into
//           shared memory by a producer warp; a request whose keys span
//           several chunks is merged by the last CTA to finish (per-(request,
//           head) arrival counter; no CTA ever waits on another).  bf16 with
//           head_dim 64/128: TMA-loaded stages scored and accumulated on the
//           tensor cores (below); otherwise bulk copies and SIMT dot products.
// prefill : requests with several input rows (initiation phase, or any
//           multi-row request).  Work item = (request, 128 query rows) x head.
//           bf16 with head_dim 64/128: flash-attention tiles on the tcgen05
//           tensor cores, S and O in tensor memory (below; an mma.sync
//           version is kept for comparisons).  Otherwise each warp owns one
//           query row at a time and attends causally over keys 0..pos of its
//           request.
// Scores use exp2 with log2(e)/sqrt(head_dim) folded into q; the softmax is
// the online (running max / running sum) form, exact up to rounding.
#include <algorithm>
#include <cstdlib>
#include <type_traits>

#include "common.cuh"
#include "kernels.cuh"

namespace orca {

namespace {

constexpr int kAttnThreads = 128;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr float kNegBig = -1e30f;

// ORCA_ATTN_PREFILL_TC=-1: bf16 prefill on the mma.sync kernel instead of the
// tcgen05 one (read once; comparisons).
int override_prefill_tc() {
    static const int v = [] {
        const char *e = getenv("ORCA_ATTN_PREFILL_TC");
        return e && *e ? atoi(e) : 0;
    }();
    return v;
}
}  // namespace

// ORCA_ATTN_DECODE_CLAIM=-1: the tensor-core decode kernel deals every CTA a
// fixed share of the work items instead of claiming them at run time (read
// once; comparisons).
bool decode_claim_enabled() {
    static const bool on = [] {
        const char *e = getenv("ORCA_ATTN_DECODE_CLAIM");
        return !(e && *e && atoi(e) < 0);
    }();
    return on;
}

namespace {

// ORCA_ATTN_DECODE_EARLY=-1: the decode kernel's producer waits for the
// previous kernel before its first load (read once; comparisons).
int override_decode_early() {
    static const int v = [] {
        const char *e = getenv("ORCA_ATTN_DECODE_EARLY");
        return e && *e ? atoi(e) : 0;
    }();
    return v;
}

template <typename T>
struct AttnArgs {
    const T *qkv;
    const T *kpool;  // layer's K block: [head][slot][D]
    const T *vpool;
    int64_t kv_slots;
    T *out;
    int H, n_heads;
    float scale_log2;
    AttnPlan p;
    float *part;
    int *counters;
    unsigned *err;
    int early;  // the decode producer may load keys before the context end ahead of the grid wait
};

// One warp attends its query (q, already scaled, VEC values of its lane's
// slice) to keys t in [t_begin, t_end) of one head, the lane group g of the
// warp taking tokens t_begin + g + j*step for j = 0, 1, ...  Updates the lane's
// running (m, l, o).  The loop trip count is uniform across the warp.
template <typename T, int D, int U>
__device__ __forceinline__ void attend_range(const float *q, const T *kb, const T *vb, int t_begin, int t_end,
                                             int step, float &m, float &l, float *o) {
    constexpr int VEC = Elem<T>::kPer16;
    constexpr int LPT = D / VEC;
    const int g = (threadIdx.x & 31) / LPT;
    for (int base = t_begin; base < t_end; base += step * U) {
        float kk[U][VEC], vv[U][VEC];
        bool valid[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = base + g + u * step;
            valid[u] = t < t_end;
            if (valid[u]) {
                load16_stream(kb + (size_t)t * D, kk[u]);
                load16_stream(vb + (size_t)t * D, vv[u]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) kk[u][e] = 0.f, vv[u][e] = 0.f;
            }
        }
        float s[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc = fmaf(q[e], kk[u][e], acc);
#pragma unroll
            for (int off = LPT / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            s[u] = valid[u] ? acc : kNegBig;
        }
        float mx = m;
#pragma unroll
        for (int u = 0; u < U; ++u) mx = fmaxf(mx, s[u]);
        const float corr = exp2f(m - mx);
        l *= corr;
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] *= corr;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float pr = valid[u] ? exp2f(s[u] - mx) : 0.f;
            l += pr;
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[e] = fmaf(pr, vv[u][e], o[e]);
        }
        m = mx;
    }
}

// Merge the running states of the lane groups of a warp (lanes with the same
// slice of head_dim); afterwards every lane holds the warp's total for its slice.
template <int LPT, int VEC>
__device__ __forceinline__ void merge_groups(float &m, float &l, float *o) {
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
        const float mx = fmaxf(m, m2);
        const float c1 = exp2f(m - mx), c2 = exp2f(m2 - mx);
        l = l * c1 + l2 * c2;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const float o2 = __shfl_xor_sync(0xffffffffu, o[e], off);
            o[e] = o[e] * c1 + o2 * c2;
        }
        m = mx;
    }
}

// Decode: the K and V rows of one (request, head, chunk) are contiguous in the
// pool, so a producer warp streams them into a ring of shared-memory stages
// with bulk asynchronous copies (kTok tokens of K and of V per stage,
// completing on an mbarrier); four consumer warps score and accumulate from
// shared memory and release each stage through a second mbarrier.
// Persistent: a grid of a few CTAs per SM walks the (work item, head) list --
// work items sorted by length, longest first -- CTA b taking entries b,
// b + grid, ...  The producer runs ahead across item boundaries, so the ring
// never drains between items, and the consumers prefetch the next item's q.
constexpr int kDecStages = 4;
constexpr int kDecConsumers = 4;
constexpr int kDecThreads = 32 * (kDecConsumers + 1);
constexpr int kDecCtasPerSm = 3;

// Tokens per stage: at least 32, and at least one warp-wide step per consumer.
template <typename T, int D>
constexpr int dec_tok() {
    return 32 > kDecConsumers * (32 / (D / Elem<T>::kPer16)) ? 32 : kDecConsumers * (32 / (D / Elem<T>::kPer16));
}

template <typename T, int D>
struct DecodeSmem {
    static constexpr int kTok = dec_tok<T, D>();
    T kv[kDecStages][2][kTok][D];
    uint64_t full[kDecStages], empty[kDecStages];
    float m[kDecConsumers], l[kDecConsumers];
    float o[kDecConsumers][D];
    int last, abort;
};

// Barrier over the 128 consumer threads only (the producer warp never joins).
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool consumers_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

template <typename T, int D>
__global__ void __launch_bounds__(kDecThreads) attn_decode_kernel(const AttnArgs<T> a) {
    constexpr int VEC = Elem<T>::kPer16;
    constexpr int LPT = D / VEC;
    constexpr int TPW = 32 / LPT;                      // tokens per warp-wide step
    constexpr int kDecTok = DecodeSmem<T, D>::kTok;
    constexpr int PER_WARP = kDecTok / kDecConsumers;  // tokens of a stage per consumer warp
    constexpr int STEPS = PER_WARP / TPW;
    static_assert(PER_WARP % TPW == 0, "stage split");
    extern __shared__ __align__(128) uint8_t dyn_smem[];
    DecodeSmem<T, D> &sm = *reinterpret_cast<DecodeSmem<T, D> *>(dyn_smem);
    pdl_trigger();
    pdl_wait();

    const int total = a.p.n_dec_work * a.n_heads;
    const int G = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // entry q of the list -> (request i, chunk c, head h)
    auto item = [&](int q, int &i, int &c, int &h) {
        const int w = a.p.dec_order[q / a.n_heads];
        h = q % a.n_heads;
        i = a.p.dec_work[2 * w];
        c = a.p.dec_work[2 * w + 1];
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kDecStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kDecConsumers);
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kDecConsumers) {
        // ------------------------------ producer ------------------------------
        if (elect_one()) {
            const uint64_t pol = l2_policy_evict_first();  // every cached row is read once per iteration
            uint32_t g = 0, issued = 0;
            bool ok = true;
            for (int q = blockIdx.x; q < total && ok; q += G) {
                int i, c, h;
                item(q, i, c, h);
                const int n_keys = a.p.req_keys ? a.p.req_keys[i] : a.p.req_ctx[i] + 1;
                const int t0 = c * a.p.chunk, t1 = min(n_keys, t0 + a.p.chunk);
                const size_t head_base = ((size_t)h * a.kv_slots + a.p.req_kvoff[i]) * D;
                for (int t = t0; t < t1; t += kDecTok, ++g) {
                    const int s = g % kDecStages;
                    const uint32_t ph = (g / kDecStages) & 1u;
                    if (!mbar_wait_bounded(&sm.empty[s], ph ^ 1u, a.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bytes = (uint32_t)(min(kDecTok, t1 - t) * D * sizeof(T));
                    mbar_arrive_expect_tx(&sm.full[s], 2 * bytes);
                    bulk_load(&sm.kv[s][0][0][0], a.kpool + head_base + (size_t)t * D, bytes, &sm.full[s], pol);
                    bulk_load(&sm.kv[s][1][0][0], a.vpool + head_base + (size_t)t * D, bytes, &sm.full[s], pol);
                    ++issued;
                }
            }
            if (!ok) {  // let the copies in flight land before the CTA exits
                sm.abort = 1;
                for (uint32_t j = issued > kDecStages ? issued - kDecStages : 0; j < issued; ++j)
                    mbar_wait_bounded(&sm.full[j % kDecStages], (j / kDecStages) & 1u, a.err);
            }
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    const int g_lane = lane / LPT, sub = lane % LPT;
    uint32_t g = 0;
    float qn[VEC];
    if (blockIdx.x < total) {
        int i, c, h;
        item(blockIdx.x, i, c, h);
        load16(a.qkv + (size_t)a.p.req_off[i] * 3 * a.H + h * D + sub * VEC, qn);
    }
    for (int q = blockIdx.x; q < total; q += G) {
        int i, c, h;
        item(q, i, c, h);
        const int row = a.p.req_off[i];
        const int n_keys = a.p.req_keys ? a.p.req_keys[i] : a.p.req_ctx[i] + 1;
        const int n_valid = a.p.req_ctx[i] + 1;  // keys past the context (a padded batch's) are masked
        const int t0 = c * a.p.chunk, t1 = min(n_keys, t0 + a.p.chunk);
        float qv[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) qv[e] = qn[e] * a.scale_log2;
        if (q + G < total) {  // the next item's q, in flight during this item
            int i2, c2, h2;
            item(q + G, i2, c2, h2);
            load16(a.qkv + (size_t)a.p.req_off[i2] * 3 * a.H + h2 * D + sub * VEC, qn);
        }
        float m = kNegBig, l = 0.f, o[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = 0.f;
        bool ok = true;
        for (int t = t0; t < t1; t += kDecTok, ++g) {
            const int s = g % kDecStages;
            const uint32_t ph = (g / kDecStages) & 1u;
            if (!mbar_wait_bounded(&sm.full[s], ph, a.err)) {
                ok = false;
                break;
            }
            const int ntok = min(kDecTok, min(t1, n_valid) - t);  // (<= 0: a stage of masked keys only)
            float sc[STEPS], vv[STEPS][VEC];
#pragma unroll
            for (int st = 0; st < STEPS; ++st) {
                const int j = warp * PER_WARP + st * TPW + g_lane;
                const bool valid = j < ntok;
                float kk[VEC];
                if (valid) {
                    load16(&sm.kv[s][0][j][sub * VEC], kk);
                    load16(&sm.kv[s][1][j][sub * VEC], vv[st]);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) kk[e] = 0.f, vv[st][e] = 0.f;
                }
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc = fmaf(qv[e], kk[e], acc);
#pragma unroll
                for (int off = LPT / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                sc[st] = valid ? acc : kNegBig;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);  // this warp's rows of stage s are in registers
            float mx = m;
#pragma unroll
            for (int st = 0; st < STEPS; ++st) mx = fmaxf(mx, sc[st]);
            const float corr = exp2f(m - mx);
            l *= corr;
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[e] *= corr;
#pragma unroll
            for (int st = 0; st < STEPS; ++st) {
                const float pr = sc[st] > kNegBig ? exp2f(sc[st] - mx) : 0.f;
                l += pr;
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = fmaf(pr, vv[st][e], o[e]);
            }
            m = mx;
        }
        if (!consumers_all(ok && sm.abort == 0)) return;  // every consumer warp leaves together
        merge_groups<LPT, VEC>(m, l, o);
        if (lane < LPT) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) sm.o[warp][sub * VEC + e] = o[e];
        }
        if (lane == 0) sm.m[warp] = m, sm.l[warp] = l;
        consumers_sync();

        const int nch = a.p.dec_nch[i];
        float M = kNegBig, L = 0.f, O = 0.f;
        const int d = threadIdx.x;
        if (d < D) {
#pragma unroll
            for (int w = 0; w < kDecConsumers; ++w) M = fmaxf(M, sm.m[w]);
#pragma unroll
            for (int w = 0; w < kDecConsumers; ++w) {
                const float cw = exp2f(sm.m[w] - M);
                L += sm.l[w] * cw;
                O += sm.o[w][d] * cw;
            }
        }
        T *dst = a.out + (size_t)row * a.H + h * D;
        if (nch == 1) {
            if (d < D) dst[d] = Elem<T>::from_f(O / L);
        } else {
            // several chunks: publish the partial, the last CTA of (request, head) merges
            const int w_idx = a.p.dec_wbegin[i] + c;
            float *mine = a.part + ((size_t)w_idx * a.n_heads + h) * (D + 2);
            if (d < D) mine[d] = O;
            if (d == 0) mine[D] = M, mine[D + 1] = L;
            __threadfence();
            consumers_sync();
            if (threadIdx.x == 0) {
                const int old = atomicAdd(&a.counters[i * a.n_heads + h], 1);
                sm.last = (old == nch - 1);
            }
            consumers_sync();
            if (sm.last) {
                __threadfence();
                if (d < D) {
                    const int wb = a.p.dec_wbegin[i];
                    float Mt = kNegBig;
                    for (int j = 0; j < nch; ++j)
                        Mt = fmaxf(Mt, __ldcg(a.part + ((size_t)(wb + j) * a.n_heads + h) * (D + 2) + D));
                    float Lt = 0.f, Ot = 0.f;
                    for (int j = 0; j < nch; ++j) {
                        const float *pj = a.part + ((size_t)(wb + j) * a.n_heads + h) * (D + 2);
                        const float cw = exp2f(__ldcg(pj + D) - Mt);
                        Lt += __ldcg(pj + D + 1) * cw;
                        Ot += __ldcg(pj + d) * cw;
                    }
                    dst[d] = Elem<T>::from_f(Ot / Lt);
                }
                if (threadIdx.x == 0) a.counters[i * a.n_heads + h] = 0;
            }
        }
        consumers_sync();  // the merge buffers are reused by the next item
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kAttnThreads) attn_prefill_kernel(const AttnArgs<T> a) {
    constexpr int VEC = Elem<T>::kPer16;
    constexpr int LPT = D / VEC;
    constexpr int TPW = 32 / LPT;
    constexpr int U = 4;
    pdl_trigger();
    pdl_wait();
    const int tile = blockIdx.x, h = blockIdx.y;
    const int i = a.p.pre_tiles[2 * tile], r0 = a.p.pre_tiles[2 * tile + 1];  // r0: first row within the request
    const int off = a.p.req_off[i];
    const int n = a.p.req_off[i + 1] - off;
    const int ctx = a.p.req_ctx[i];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane % LPT;
    const size_t head_base = ((size_t)h * a.kv_slots + a.p.req_kvoff[i]) * D + sub * VEC;
    const int r_end = min(n, r0 + kPrefillRowsPerTile);
    for (int r = r0 + warp; r < r_end; r += kAttnWarps) {
        const int row = off + r;
        const int pos = ctx + r;
        float q[VEC];
        load16(a.qkv + (size_t)row * 3 * a.H + h * D + sub * VEC, q);
#pragma unroll
        for (int e = 0; e < VEC; ++e) q[e] *= a.scale_log2;
        float m = kNegBig, l = 0.f, o[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = 0.f;
        attend_range<T, D, U>(q, a.kpool + head_base, a.vpool + head_base, 0, pos + 1, TPW, m, l, o);
        merge_groups<LPT, VEC>(m, l, o);
        if (lane < LPT) {
            float res[VEC];
            const float inv = 1.f / l;
#pragma unroll
            for (int e = 0; e < VEC; ++e) res[e] = o[e] * inv;
            store16(a.out + (size_t)row * a.H + h * D + sub * VEC, res);
        }
    }
}

// ---------------------------------------------------------------------------
// Prefill on tensor cores (bf16, head_dim 64 or 128): flash-attention tiling.
// CTA = (request, 64 query rows, head), 4 warps x 16 rows; blockIdx.z picks
// the half of the plan's 128-row tile.  K/V tiles of 64
// keys are double-buffered in shared memory (cp.async, 16-byte chunks stored
// XOR-swizzled by row so ldmatrix reads are conflict-free); S = Q K^T and
// O += P V run on mma.sync m16n8k16 with fp32 accumulators; the softmax is the
// online form, rows held in registers.  Causal: row r of the request sits at
// position ctx + r and sees keys 0 .. ctx + r.
// ---------------------------------------------------------------------------
constexpr int kPreRows = 64;  // query rows per CTA (half of kPrefillRowsPerTile)
constexpr int kPreKeys = 64;  // keys per tile

template <int D>
struct PrefillSmem {
    bf16 q[kPreRows * D];
    bf16 k[2][kPreKeys * D];
    bf16 v[2][kPreKeys * D];
};

// byte offset of 16-byte chunk `ch` of row `row` in a swizzled [rows][D] bf16 tile
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int ch) {
    return (uint32_t)(row * D * 2 + ((ch ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float *c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <int D>
__global__ void __launch_bounds__(128) attn_prefill_mma_kernel(const AttnArgs<bf16> a) {
    constexpr int CH = D / 8;   // 16-byte chunks per row
    constexpr int NT = D / 8;   // n-tiles of the output (8 columns each)
    constexpr int KS = D / 16;  // k-steps of S = Q K^T
    extern __shared__ __align__(128) uint8_t dyn_smem[];
    PrefillSmem<D> &sm = *reinterpret_cast<PrefillSmem<D> *>(dyn_smem);
    const uint32_t sq = smem_u32(sm.q), sk0 = smem_u32(sm.k[0]), sv0 = smem_u32(sm.v[0]);
    constexpr uint32_t kTileBytes = kPreKeys * D * 2;
    pdl_trigger();
    pdl_wait();

    const int tile = blockIdx.x, h = blockIdx.y;
    const int i = a.p.pre_tiles[2 * tile], q0 = a.p.pre_tiles[2 * tile + 1] + kPreRows * (int)blockIdx.z;
    const int off = a.p.req_off[i];
    const int n = a.p.req_off[i + 1] - off;
    if (q0 >= n) return;  // the tile's second half is past the request
    const int ctx = a.p.req_ctx[i];
    const int rows = min(kPreRows, n - q0);
    const int n_keys = ctx + q0 + rows;  // keys any row of this tile may see
    const int n_kt = (n_keys + kPreKeys - 1) / kPreKeys;
    const bf16 *gk = a.kpool + ((size_t)h * a.kv_slots + a.p.req_kvoff[i]) * D;
    const bf16 *gv = a.vpool + ((size_t)h * a.kv_slots + a.p.req_kvoff[i]) * D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // Q tile (rows beyond the request are zero-filled)
    for (int c = tid; c < kPreRows * CH; c += 128) {
        const int r = c / CH, ch = c % CH;
        const bool ok = r < rows;
        const bf16 *src = a.qkv + (size_t)(off + q0 + (ok ? r : 0)) * 3 * a.H + h * D + ch * 8;
        cp_async16(sq + swz<D>(r, ch), src, ok);
    }
    auto load_kv = [&](int kt, int buf) {
        for (int c = tid; c < kPreKeys * CH; c += 128) {
            const int r = c / CH, ch = c % CH;
            const int t = kt * kPreKeys + r;
            const bool ok = t < n_keys;
            const size_t so = (size_t)(ok ? t : 0) * D + ch * 8;
            cp_async16(sk0 + buf * kTileBytes + swz<D>(r, ch), gk + so, ok);
            cp_async16(sv0 + buf * kTileBytes + swz<D>(r, ch), gv + so, ok);
        }
    };
    load_kv(0, 0);
    cp_async_commit();

    const int g = lane >> 2, tg = lane & 3;
    const int row_lo = warp * 16 + g, row_hi = row_lo + 8;  // this thread's two rows within the tile
    const int pos_lo = ctx + q0 + row_lo, pos_hi = ctx + q0 + row_hi;
    uint32_t qa[KS][4];
    float o[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m_lo = kNegBig, m_hi = kNegBig, l_lo = 0.f, l_hi = 0.f;

    for (int kt = 0; kt < n_kt; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < n_kt) {
            load_kv(kt + 1, buf ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (kt == 0) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int r = warp * 16 + (lane & 15);
                const int ch = ks * 2 + (lane >> 4);
                ldsm_x4(sq + swz<D>(r, ch), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
            }
        }
        const uint32_t skb = sk0 + buf * kTileBytes, svb = sv0 + buf * kTileBytes;
        // S = Q K^T for this warp's 16 rows x 64 keys
        float sc[kPreKeys / 8][4];
#pragma unroll
        for (int j = 0; j < kPreKeys / 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
            for (int jn = 0; jn < kPreKeys / 16; ++jn) {  // two 8-key n-tiles per ldmatrix.x4
                const int key = jn * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int ch = ks * 2 + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(skb + swz<D>(key, ch), b0, b1, b2, b3);
                mma_bf16(sc[2 * jn], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                mma_bf16(sc[2 * jn + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
            }
        }
        // scale, causal mask, online softmax
        float mx_lo = m_lo, mx_hi = m_hi;
#pragma unroll
        for (int j = 0; j < kPreKeys / 8; ++j) {
            const int key = kt * kPreKeys + j * 8 + 2 * tg;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                sc[j][e] = (key + e <= pos_lo) ? sc[j][e] * a.scale_log2 : kNegBig;
                sc[j][2 + e] = (key + e <= pos_hi) ? sc[j][2 + e] * a.scale_log2 : kNegBig;
                mx_lo = fmaxf(mx_lo, sc[j][e]);
                mx_hi = fmaxf(mx_hi, sc[j][2 + e]);
            }
        }
#pragma unroll
        for (int sh = 1; sh < 4; sh <<= 1) {
            mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, sh));
            mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, sh));
        }
        const float c_lo = exp2f(m_lo - mx_lo), c_hi = exp2f(m_hi - mx_hi);
        m_lo = mx_lo, m_hi = mx_hi;
        float s_lo = 0.f, s_hi = 0.f;
#pragma unroll
        for (int j = 0; j < kPreKeys / 8; ++j) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                sc[j][e] = sc[j][e] > kNegBig ? exp2f(sc[j][e] - mx_lo) : 0.f;
                sc[j][2 + e] = sc[j][2 + e] > kNegBig ? exp2f(sc[j][2 + e] - mx_hi) : 0.f;
                s_lo += sc[j][e];
                s_hi += sc[j][2 + e];
            }
        }
        l_lo = l_lo * c_lo + s_lo;  // per-thread partial sums; reduced across the quad at the end
        l_hi = l_hi * c_hi + s_hi;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            o[j][0] *= c_lo, o[j][1] *= c_lo;
            o[j][2] *= c_hi, o[j][3] *= c_hi;
        }
        // O += P V
#pragma unroll
        for (int kk = 0; kk < kPreKeys / 16; ++kk) {
            const uint32_t p0 = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
            const uint32_t p1 = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
            const uint32_t p2 = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
            const uint32_t p3 = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
            for (int jn = 0; jn < NT / 2; ++jn) {  // two 8-column output tiles per ldmatrix.x4.trans
                const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int ch = jn * 2 + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(svb + swz<D>(key, ch), b0, b1, b2, b3);
                mma_bf16(o[2 * jn], p0, p1, p2, p3, b0, b1);
                mma_bf16(o[2 * jn + 1], p0, p1, p2, p3, b2, b3);
            }
        }
        __syncthreads();  // every warp is done with `buf` before it is refilled
    }
#pragma unroll
    for (int sh = 1; sh < 4; sh <<= 1) {
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, sh);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, sh);
    }
    const float inv_lo = 1.f / l_lo, inv_hi = 1.f / l_hi;
    bf16 *out_lo = a.out + (size_t)(off + q0 + row_lo) * a.H + h * D + 2 * tg;
    bf16 *out_hi = a.out + (size_t)(off + q0 + row_hi) * a.H + h * D + 2 * tg;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        if (row_lo < rows) *reinterpret_cast<uint32_t *>(out_lo + j * 8) = pack_bf16(o[j][0] * inv_lo, o[j][1] * inv_lo);
        if (row_hi < rows) *reinterpret_cast<uint32_t *>(out_hi + j * 8) = pack_bf16(o[j][2] * inv_hi, o[j][3] * inv_hi);
    }
}

// ---------------------------------------------------------------------------
// Prefill on the fifth-generation tensor cores (bf16, head_dim 64 or 128).
// Persistent: one CTA per SM walks items (head, 128 query rows of a request),
// TMEM and barriers set up once; the next item's Q and first keys load and
// its first S runs while this item finishes, and O has two TMEM buffers so
// that an item's P V can start while the last item's O is written out.
// Both contractions are tcgen05 MMAs with M = 128 query rows, one TMEM lane
// per row, fp32 accumulators in tensor memory:
//   S  = Q K^T   A = Q (K-major), B = a tile of 128 keys of K (K-major)
//   O += P V     A = P (K-major, written by the softmax warps), B = the V tile
//                read MN-major straight from its [key][dim] TMA image
// Warp 0 streams Q and 128-key tiles of K and of V by TMA (two stages each,
// on separate barriers, so S can start before V has landed).  Warp 1 issues
// S_{j+1} while the softmax warps work on S_j, then O += P_j V_j.  Warps 2-9
// hold half a query row per thread (two warps per TMEM lane quarter, 64 keys
// of each tile and half of O's columns; a row's two halves meet in shared
// memory for its max and its sum): the scale, the causal mask (row r at
// position ctx + q0 + r sees keys 0 .. ctx + q0 + r, masked by index where a
// tile reaches past some row's last key), the running max m and sum l in
// fp32, and P_j = exp2(S_j - m) rounded to bf16 for the MMA.  O is rescaled
// in TMEM (read, scaled, written back) only when a row's max has grown by
// more than 2^8 since m was last set: every P is formed against the m that
// O and l carry, so the result is the same up to rounding, and P stays below
// 2^8.  The last tile may reach past the tile's keys into slots of other
// requests or slots never written: those scores are masked by index and
// those V rows zeroed in shared memory before P V reads them.
// ---------------------------------------------------------------------------
constexpr int kPtRows = 128;         // query rows per item (== kPrefillRowsPerTile)
constexpr int kPtKeys = 128;         // keys per tile
constexpr int kPtThreads = 320;      // TMA warp, MMA warp, eight softmax warps (two per TMEM lane quarter)
constexpr uint32_t kPtAtom = 16384;  // 128 rows x 128 bytes: one 128-byte-swizzled block
constexpr float kPtRescale = 8.f;    // log2 growth of a row's max that triggers a rescale of O
constexpr uint32_t kPtTmemCols = 512;
constexpr uint32_t kPtTmemO = 256;   // O's two buffers; S_0 and S_1 take columns 0 .. 255
constexpr uint32_t kPtOCols = 128;   // columns per O buffer (head_dim <= 128)
// Device error bit: a kernel's dynamic shared memory did not start 1024-byte
// aligned (its swizzled tiles need it); the kernel did nothing.
constexpr unsigned kErrSmemAlign = 8u;

template <int D>
struct PtLayout {  // byte offsets from the 1024-aligned base of dynamic shared memory
    static constexpr int kAtoms = D / 64;  // 64-dim blocks of a row of Q, K, V
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + kAtoms * kPtAtom;      // 2 stages
    static constexpr uint32_t kV = kK + 2 * kAtoms * kPtAtom;  // 2 stages
    static constexpr uint32_t kP = kV + 2 * kAtoms * kPtAtom;  // 2 buffers of 2 blocks (keys 0-63, 64-127)
    static constexpr uint32_t kBars = kP + 4 * kPtAtom;
    static constexpr uint32_t kRed = kBars + 256;              // [2 tiles][2 halves][128 rows] floats
    static constexpr uint32_t kBytes = kRed + 2048;            // (the base must be 1024-aligned: checked)
};

struct PtBars {
    uint64_t q_full, q_empty, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2], pv_done[2];
    uint64_t o_free[2], drain;
    uint64_t pair[4];  // the two softmax warps of each TMEM lane quarter
    uint32_t tmem;
    int abort;
};

// Shared-memory matrix descriptor for an MN-major operand written by TMA with
// 128-byte swizzling as blocks of [K rows][64 MN elements]: rows 128 B apart,
// 8-row groups 1024 B apart (stride byte offset), 64-element MN blocks
// `mn_block` bytes apart (leading byte offset); version 1, swizzle mode 2.
__device__ __forceinline__ uint64_t smem_desc_mn128(uint32_t saddr, uint32_t mn_block) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((mn_block >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
                   "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}
// Waits for this thread's TMEM loads; the registers are operands, so no use
// of them is placed before the wait.
__device__ __forceinline__ void tmem_wait_ld32(uint32_t *r) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
                   "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
                 "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
                 :
                 : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                   "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
                   "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
                   "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 2^x by the SFU's approximation (flush-to-zero; 2^-inf = +0)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kPtThreads, 1)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmkv,
                           const AttnArgs<bf16> a) {
    using L = PtLayout<D>;
    extern __shared__ __align__(1024) uint8_t pt_smem_raw[];
    if (smem_u32(pt_smem_raw) & 1023u) {  // uniform: every thread leaves before any barrier
        if (threadIdx.x == 0) raise_err(a.err, kErrSmemAlign);
        return;
    }
    uint8_t *sm = pt_smem_raw;
    PtBars &bar = *reinterpret_cast<PtBars *>(sm + L::kBars);
    volatile int *abort = &bar.abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr unsigned kFull = 0xffffffffu;

    pdl_trigger();
    if (threadIdx.x == 0) {
        mbar_init(&bar.q_full, 1);
        mbar_init(&bar.q_empty, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bar.k_full[b], 1);
            mbar_init(&bar.k_empty[b], 1);
            mbar_init(&bar.v_full[b], 1);
            mbar_init(&bar.v_empty[b], 1);
            mbar_init(&bar.s_full[b], 1);
            mbar_init(&bar.p_full[b], 8);  // one arrival per softmax warp
            mbar_init(&bar.pv_done[b], 1);
            mbar_init(&bar.o_free[b], 8);
        }
        mbar_init(&bar.drain, 1);
        for (int q = 0; q < 4; ++q) mbar_init(&bar.pair[q], 2);
        *abort = 0;
        fence_mbar_init();
        prefetch_tmap(&tmq);
        prefetch_tmap(&tmkv);
    }
    if (warp == 1) {
        tmem_alloc(&bar.tmem, kPtTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem;
    pdl_wait();  // q and this iteration's K/V rows come from the kernels before

    // This CTA's items: b, b + G, ... of (head, tile) with the tiles of a head
    // innermost (the query tiles of one request, which read the same keys,
    // run at about the same time), each head's tiles in the plan's order
    // (longest first).
    const int n_items = a.p.n_pre_tiles * a.n_heads;
    struct Item {
        int h, off, q0, ctx, kv0, rows, n_keys, n_kt;
    };
    auto item_at = [&](int k) {
        Item it;
        const int idx = (int)blockIdx.x + k * (int)gridDim.x;
        it.h = idx / a.p.n_pre_tiles;
        const int t = idx - it.h * a.p.n_pre_tiles;
        const int i = a.p.pre_tiles[2 * t];
        it.q0 = a.p.pre_tiles[2 * t + 1];
        it.off = a.p.req_off[i];
        it.ctx = a.p.req_ctx[i];
        it.kv0 = a.p.req_kvoff[i];
        it.rows = min(kPtRows, a.p.req_off[i + 1] - it.off - it.q0);
        it.n_keys = it.ctx + it.q0 + it.rows;  // keys any row of the tile may see
        it.n_kt = (it.n_keys + kPtKeys - 1) / kPtKeys;
        return it;
    };
    const int n_mine = n_items > (int)blockIdx.x ? (n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    // Phases: key tiles are numbered g = 0, 1, .. across this CTA's items (K/V
    // stage, S buffer, P buffer: g & 1; the barrier's use: g >> 1), items k =
    // 0, 1, .. (Q: k; O buffer k & 1, its use k >> 1).

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        const bool leader = elect_one();
        const uint64_t pol = l2_policy_evict_normal();  // every query tile of the request reads them
        int g = 0, q_issued = 0, k_issued = 0, v_issued = 0;
        bool ok = true;
        for (int k = 0; k < n_mine && ok; ++k) {
            const Item it = item_at(k);
            // Q of item k - 1 has been read by its last S
            if (k >= 1 && !__all_sync(kFull, !*abort && mbar_wait_bounded(&bar.q_empty, (uint32_t)(k - 1) & 1u, a.err))) {
                ok = false;
                break;
            }
            if (leader) {
                mbar_arrive_expect_tx(&bar.q_full, L::kAtoms * kPtAtom);
                for (int c = 0; c < L::kAtoms; ++c)
                    tma_load_2d(sm + L::kQ + c * kPtAtom, &tmq, &bar.q_full, it.h * D + 64 * c, it.off + it.q0);
            }
            __syncwarp();
            q_issued = k + 1;
            for (int j = 0; j < it.n_kt; ++j, ++g) {
                const int b = g & 1;
                const uint32_t ep = (uint32_t)((g - 2) >> 1) & 1u;  // the release of tile g - 2
                if (g >= 2 && !__all_sync(kFull, !*abort && mbar_wait_bounded(&bar.k_empty[b], ep, a.err))) {
                    ok = false;
                    break;
                }
                if (leader) {
                    mbar_arrive_expect_tx(&bar.k_full[b], L::kAtoms * kPtAtom);
                    for (int c = 0; c < L::kAtoms; ++c)
                        tma_load_3d_hint(sm + L::kK + (b * L::kAtoms + c) * kPtAtom, &tmkv, &bar.k_full[b], 64 * c,
                                         it.kv0 + j * kPtKeys, it.h, pol);
                }
                __syncwarp();
                k_issued = g + 1;
                if (g >= 2 && !__all_sync(kFull, !*abort && mbar_wait_bounded(&bar.v_empty[b], ep, a.err))) {
                    ok = false;
                    break;
                }
                if (leader) {
                    mbar_arrive_expect_tx(&bar.v_full[b], L::kAtoms * kPtAtom);
                    for (int c = 0; c < L::kAtoms; ++c)
                        tma_load_3d_hint(sm + L::kV + (b * L::kAtoms + c) * kPtAtom, &tmkv, &bar.v_full[b], 64 * c,
                                         it.kv0 + j * kPtKeys, a.n_heads + it.h, pol);
                }
                __syncwarp();
                v_issued = g + 1;
            }
        }
        if (!ok) {
            *abort = 1;
            // let the copies in flight (each barrier's latest use at most) land before the CTA exits
            if (leader) {
                if (q_issued > 0) mbar_wait_bounded(&bar.q_full, (uint32_t)(q_issued - 1) & 1u, a.err);
                for (int x = max(0, k_issued - 2); x < k_issued; ++x)
                    mbar_wait_bounded(&bar.k_full[x & 1], (uint32_t)(x >> 1) & 1u, a.err);
                for (int x = max(0, v_issued - 2); x < v_issued; ++x)
                    mbar_wait_bounded(&bar.v_full[x & 1], (uint32_t)(x >> 1) & 1u, a.err);
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        const bool leader = elect_one();
        const uint32_t idesc_s = idesc_bf16_f32(kPtRows, kPtKeys);
        const uint32_t idesc_pv = idesc_bf16_f32(kPtRows, D) | (1u << 16);  // B (V) MN-major
        const uint32_t q_s = smem_u32(sm + L::kQ);
        // S of key tile g (the item's j-th): Q K_g^T into S buffer g & 1; the item's
        // last S also releases Q
        auto issue_s = [&](int g, bool last) {
            const int b = g & 1;
            if (!__all_sync(kFull, !*abort && mbar_wait_bounded(&bar.k_full[b], (uint32_t)(g >> 1) & 1u, a.err)))
                return false;
            tc_fence_after();
            const uint32_t k_s = smem_u32(sm + L::kK + b * L::kAtoms * kPtAtom);
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {  // 16 dims per MMA: 32 B within a 64-dim block
                    const uint32_t o = (uint32_t)(ks >> 2) * kPtAtom + (uint32_t)(ks & 3) * 32u;
                    tc_mma_f16(tmem + (uint32_t)(b * kPtKeys), smem_desc_k128(q_s + o), smem_desc_k128(k_s + o),
                               idesc_s, (uint32_t)(ks != 0));
                }
                tc_commit(&bar.k_empty[b]);
                tc_commit(&bar.s_full[b]);
                if (last) tc_commit(&bar.q_empty);
            }
            __syncwarp();
            return true;
        };
        // O (buffer ob) += P_g V_g; the item's first overwrites O
        auto issue_pv = [&](int g, int ob, bool first) {
            const int b = g & 1;
            const uint32_t ph = (uint32_t)(g >> 1) & 1u;
            if (!__all_sync(kFull, !*abort && mbar_wait_bounded(&bar.p_full[b], ph, a.err) &&
                                       mbar_wait_bounded(&bar.v_full[b], ph, a.err)))
                return false;
            tc_fence_after();
            const uint32_t p_s = smem_u32(sm + L::kP + b * 2 * kPtAtom);
            const uint32_t v_s = smem_u32(sm + L::kV + b * L::kAtoms * kPtAtom);
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < kPtKeys / 16; ++ks)  // 16 keys per MMA: two 8-row groups of V
                    tc_mma_f16(tmem + kPtTmemO + (uint32_t)(ob * kPtOCols),
                               smem_desc_k128(p_s + (uint32_t)(ks >> 2) * kPtAtom + (uint32_t)(ks & 3) * 32u),
                               smem_desc_mn128(v_s + (uint32_t)ks * 2048u, kPtAtom), idesc_pv,
                               (uint32_t)(!first || ks != 0));
                tc_commit(&bar.v_empty[b]);
                tc_commit(&bar.pv_done[b]);
            }
            __syncwarp();
            return true;
        };
        // S runs one key tile ahead of P V across item boundaries, so the next
        // item's first S is done while the softmax warps finish this item
        int k_next = 0, j_next = 0, g_next = 0;  // the next S: item k_next, its tile j_next
        int nkt_next = n_mine > 0 ? item_at(0).n_kt : 0;
        auto issue_next_s = [&]() {
            if (j_next == 0 &&
                !__all_sync(kFull, !*abort && mbar_wait_bounded(&bar.q_full, (uint32_t)k_next & 1u, a.err)))
                return false;
            if (!issue_s(g_next, j_next + 1 == nkt_next)) return false;
            ++g_next;
            if (++j_next == nkt_next) {
                j_next = 0;
                if (++k_next < n_mine) nkt_next = item_at(k_next).n_kt;
            }
            return true;
        };
        bool ok = n_mine == 0 || issue_next_s();
        int g = 0;
        for (int k = 0; ok && k < n_mine; ++k) {
            const int n_kt = item_at(k).n_kt, ob = k & 1;
            for (int j = 0; ok && j < n_kt; ++j, ++g) {
                if (k_next < n_mine) ok = issue_next_s();
                // O buffer ob was read out by the softmax warps at the end of item k - 2
                if (ok && j == 0 && k >= 2)
                    ok = __all_sync(kFull, !*abort && mbar_wait_bounded(&bar.o_free[ob],
                                                                        (uint32_t)((k - 2) >> 1) & 1u, a.err));
                if (ok) ok = issue_pv(g, ob, j == 0);
            }
        }
        if (!ok) *abort = 1;
        // every MMA issued has completed before the stages and TMEM are released
        if (leader) tc_commit(&bar.drain);
        __syncwarp();
        mbar_wait_bounded(&bar.drain, 0u, a.err);
    } else {
        // ------------------------------ softmax ------------------------------
        // Two warps per TMEM lane quarter: warps 2-5 take keys 0-63 of their
        // rows, warps 6-9 keys 64-127 (and the matching halves of O's
        // columns); the two halves of a row meet in shared memory for its max
        // and, at the end of an item, its sum.
        const int quarter = warp & 3;      // TMEM lanes 32 * (warp % 4) ..
        const int half = (warp - 2) >> 2;  // which 64 keys of a tile, which half of O's columns
        const int r = quarter * 32 + lane;
        const uint32_t lane_t = tmem + ((uint32_t)(quarter * 32) << 16);
        float *red = reinterpret_cast<float *>(sm + L::kRed);  // [meeting parity][half][row]
        // the two warps of a quarter meet on its mbarrier (one arrival each, a bounded wait);
        // meeting z exchanges through the slots of parity z & 1, which are written
        // again at meeting z + 2, after the partner has read them (it reads before
        // arriving at meeting z + 1)
        int n_pair = 0;
        auto exchange = [&](float v, bool &met) {
            float *slot = red + ((n_pair & 1) * 2 + half) * kPtRows + r;
            *slot = v;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.pair[quarter]);
            met = __all_sync(kFull, mbar_wait_bounded(&bar.pair[quarter], (uint32_t)(n_pair & 1), a.err));
            const float other = slot[(1 - 2 * half) * kPtRows];  // the same row's other half
            ++n_pair;
            return other;
        };
        constexpr int kOc = D / 2;  // O columns of this half
        // An item's output is read out of O after the next item's first P has
        // been written (O has two buffers), so the tensor pipe has that
        // item's P V and S to work on meanwhile.
        struct Done {  // a finished item whose output is still in O
            int k, g_last, row, h, rows;
            float l;
        };
        auto write_out = [&](const Done &e) {
            bool met;
            const float lt = e.l + exchange(e.l, met);  // the row's sum over both halves
            if (!met || !__all_sync(kFull, !*abort && mbar_wait_bounded(&bar.pv_done[e.g_last & 1],
                                                                       (uint32_t)(e.g_last >> 1) & 1u, a.err)))
                return false;
            tc_fence_after();
            const uint32_t ot = lane_t + kPtTmemO + (uint32_t)((e.k & 1) * kPtOCols + kOc * half);
            const float inv = 1.f / lt;
            bf16 *dst = a.out + (size_t)(e.row + r) * a.H + e.h * D + kOc * half;
#pragma unroll
            for (int c = 0; c < kOc / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(ot + 32 * c, o);
                tmem_wait_ld32(o);
                if (r < e.rows) {
                    uint32_t w[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(o[2 * x]) * inv,
                                                                       __uint_as_float(o[2 * x + 1]) * inv);
                        w[x] = *reinterpret_cast<const uint32_t *>(&v);
                    }
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * c);
#pragma unroll
                    for (int x = 0; x < 4; ++x) d4[x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
                }
            }
            // O buffer k & 1 may take item k + 2
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.o_free[e.k & 1]);
            return true;
        };
        Done late{};
        bool has_late = false;
        bool ok = true;
        int g = 0;
        for (int k = 0; k < n_mine && ok; ++k) {
            const Item it = item_at(k);
            const int ob = k & 1;
            const uint32_t o_t = lane_t + kPtTmemO + (uint32_t)(ob * kPtOCols + kOc * half);  // this half of O
            const int row_keys = min(it.ctx + it.q0 + r + 1, it.n_keys);  // keys 0 .. row_keys - 1 are this row's
            const int first_keys = min(it.ctx + it.q0 + 1, it.n_keys);    // the fewest any row of the tile sees
            float m = kNegBig, l = 0.f;
            for (int j = 0; j < it.n_kt; ++j, ++g) {
                const int b = g & 1, kbase = j * kPtKeys;
                if (!__all_sync(kFull, !*abort && mbar_wait_bounded(&bar.s_full[b], (uint32_t)(g >> 1) & 1u, a.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t s[64];
                tmem_ld32(lane_t + (uint32_t)(b * kPtKeys + 64 * half), s);
                tmem_ld32(lane_t + (uint32_t)(b * kPtKeys + 64 * half + 32), s + 32);
                tmem_wait_ld32(s);
                tmem_wait_ld32(s + 32);
                // every row sees all of this tile's keys, or a prefix of them (masked by index)
                const bool whole = kbase + kPtKeys <= first_keys;
                if (!whole) {
                    const int valid = min(max(row_keys - kbase - 64 * half, 0), 64);
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (c >= valid) s[c] = __float_as_uint(kNegBig);
                }
                float mx = kNegBig;
#pragma unroll
                for (int c = 0; c < 64; ++c) mx = fmaxf(mx, __uint_as_float(s[c]));
                bool met;
                mx = fmaxf(mx, exchange(mx, met)) * a.scale_log2;  // (scale > 0)
                if (!met) {
                    ok = false;
                    break;
                }
                float alpha = 1.f;
                if (j == 0) {
                    m = mx;
                } else if (mx > m + kPtRescale) {
                    alpha = ex2_approx(m - mx);
                    m = mx;
                    l *= alpha;
                }
                // P buffer b was read by the P V of key tile g - 2
                if (g >= 2 &&
                    !__all_sync(kFull, mbar_wait_bounded(&bar.pv_done[b], (uint32_t)((g - 2) >> 1) & 1u, a.err))) {
                    ok = false;
                    break;
                }
                if (__any_sync(kFull, alpha != 1.f)) {
                    // O = the item's P V so far: once the last of them (tile g - 1) is done, scale this half
                    if (!__all_sync(kFull, mbar_wait_bounded(&bar.pv_done[(g - 1) & 1], (uint32_t)((g - 1) >> 1) & 1u,
                                                             a.err))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < kOc / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(o_t + 32 * c, o);
                        tmem_wait_ld32(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(o_t + 32 * c, o);
                    }
                    tmem_wait_st();
                }
                // P_g, this half: row r of 64-key block `half`, 16-byte chunk c at position c ^ (r % 8);
                // masked keys hold kNegBig, whose exp2 is 0
                const uint32_t p_row = smem_u32(sm + L::kP + (b * 2 + half) * kPtAtom) + (uint32_t)r * 128u;
                const float neg_m = -m;
                float ls = 0.f;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float p0 = ex2_approx(fmaf(__uint_as_float(s[8 * c8 + 2 * e]), a.scale_log2, neg_m));
                        const float p1 = ex2_approx(fmaf(__uint_as_float(s[8 * c8 + 2 * e + 1]), a.scale_log2, neg_m));
                        ls += p0 + p1;
                        const __nv_bfloat162 pv = __floats2bfloat162_rn(p0, p1);
                        w[e] = *reinterpret_cast<const uint32_t *>(&pv);
                    }
                    st_shared_v4(p_row + ((uint32_t)(c8 ^ (r & 7)) << 4), w[0], w[1], w[2], w[3]);
                }
                l += ls;
                // the tile's V rows past its keys: zeroed (once they have landed) before P V reads them
                const int tile_keys = min(it.n_keys - kbase, kPtKeys);
                if (tile_keys < kPtKeys) {
                    if (!__all_sync(kFull, mbar_wait_bounded(&bar.v_full[b], (uint32_t)(g >> 1) & 1u, a.err))) {
                        ok = false;
                        break;
                    }
                    if (half < L::kAtoms && r >= tile_keys)
#pragma unroll
                        for (int x = 0; x < 8; ++x)
                            st_shared_v4(smem_u32(sm + L::kV + (b * L::kAtoms + half) * kPtAtom) + (uint32_t)r * 128u +
                                             16u * x,
                                         0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();  // P (and the zeroed rows) before the tensor core reads them
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.p_full[b]);
                if (j == 0 && has_late) {  // the item before: its output, now that this item's first P is out
                    if (!write_out(late)) {
                        ok = false;
                        break;
                    }
                    has_late = false;
                }
            }
            if (!ok) break;
            late = Done{k, g - 1, it.off + it.q0, it.h, it.rows, l};
            has_late = true;
        }
        if (ok && has_late) ok = write_out(late);
        if (!ok) *abort = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kPtTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Decode on tensor cores (bf16, head_dim 64 or 128).  Same persistent layout
// as the kernel above -- a producer warp streams stages of kMdTok tokens of
// one (request chunk, head) into a ring, consumer warps drain it, the producer
// runs ahead across item boundaries -- but the stages arrive by 3-D TMA boxes
// of 64 dims x kMdTok tokens with 128-byte swizzling (so ldmatrix reads them
// without bank conflicts), and each of the four consumer warps scores and
// accumulates its 16 tokens of a stage on mma.sync m16n8k16.  With one query
// per (request, head) the keys take the M dimension:
//   S^T = K q^T    A = the warp's 16-token x 16-dim K tile (ldmatrix), B = q
//   O^T += V^T p   A = a 16-dim x 16-token V^T tile (ldmatrix.trans), B = p
// Every column of B holds the same vector, so every column of each 16 x 8
// result holds the answer.  p enters the MMA rounded to bf16 and l sums those
// rounded weights.  An item's last stage is loaded in boxes of 16 tokens (a
// second tensor map), so at most 15 keys past its end are read; rows past the
// end are masked out of the scores and zeroed in V (they may belong to
// another request, or be stale).
// ---------------------------------------------------------------------------
constexpr int kMdTok = 64;
constexpr int kMdConsumers = kMdTok / 16;
constexpr int kMdMergers = 2;  // merge warps, taking the items in turn
constexpr int kMdProducerWarp = kMdConsumers, kMdMergerWarp = kMdConsumers + 1;
constexpr int kMdThreads = 32 * (kMdConsumers + 1 + kMdMergers);
constexpr int kMdCtasPerSm = 2;
constexpr int kMdMerge = 4;  // item results queued for the merge warp
constexpr int kMdIds = 8;    // ring of the CTA's item ids, producer -> consumers

template <int D>
__host__ __device__ constexpr uint32_t md_stage_bytes() {
    return 2u * D * kMdTok * 2u;  // K and V
}
template <int D>
__host__ __device__ constexpr int md_stages() {
    return (int)(98304u / md_stage_bytes<D>());  // 96 KiB of ring
}
template <int D>
struct MdTail {  // after the ring
    uint64_t full[md_stages<D>()], empty[md_stages<D>()];
    uint64_t mfull[kMdMerge], mempty[kMdMerge];
    uint64_t id_full[kMdIds];
    int ids[kMdIds];    // the CTA's j-th item (j >= 1) at [(j - 1) % kMdIds] (>= total: no more)
    int mq[kMdMerge];   // the item of each merge entry (-1: no more)
    float o[kMdMerge][kMdConsumers][D];  // each consumer warp's unnormalised output of an item
    float m[kMdMerge][kMdConsumers], l[kMdMerge][kMdConsumers];
    volatile int abort;
};
template <int D>
__host__ __device__ constexpr size_t md_smem_bytes() {
    return 1024 + md_stages<D>() * md_stage_bytes<D>() + sizeof(MdTail<D>);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kMdThreads) attn_decode_mma_kernel(const __grid_constant__ CUtensorMap tm,
                                                                     const __grid_constant__ CUtensorMap tm16,
                                                                     const AttnArgs<bf16> a) {
    constexpr int NB = D / 64;  // 64-dim boxes per row
    constexpr int KS = D / 16;  // k-steps of the scores
    constexpr int MT = D / 16;  // 16-dim tiles of the output
    constexpr int S = md_stages<D>();
    constexpr uint32_t kBox = kMdTok * 128;
    constexpr uint32_t kStage = md_stage_bytes<D>();
    static_assert(D % 64 == 0 && S >= 2, "tile shape");
    extern __shared__ uint8_t dyn_smem[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    MdTail<D> &sm = *reinterpret_cast<MdTail<D> *>(ring + S * kStage);
    pdl_trigger();

    const int total = a.p.n_dec_work * a.n_heads;
    const int G = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // entry q = (sorted work item q / n_heads, head q % n_heads): {kv slot of the first key,
    // keys, first row, request} and {chunk, the request's chunks, its first work item, first key}
    auto rec = [&](int q, int4 &r0, int4 &r1) {
        const int4 *r = reinterpret_cast<const int4 *>(a.p.dec_items) + 2 * (q / a.n_heads);
        r0 = r[0], r1 = r[1];
    };
    // This CTA's k-th entry of the (longest-first) list: rounds of G entries,
    // dealt forwards and backwards in turn so that every CTA's share of the
    // large and the small items evens out.  Past the list once >= total.
    auto nth = [&](int k) { return k * G + ((k & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x); };
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kMdConsumers);
        }
        for (int e = 0; e < kMdMerge; ++e) {
            mbar_init(&sm.mfull[e], kMdConsumers);
            mbar_init(&sm.mempty[e], 1);
        }
        for (int j = 0; j < kMdIds; ++j) mbar_init(&sm.id_full[j], 1);
        sm.abort = 0;
        fence_mbar_init();
        prefetch_tmap(&tm);
        prefetch_tmap(&tm16);
    }
    __syncthreads();

    // Every wait is bounded; a role whose wait gives up raises the abort flag
    // and leaves, and the others leave at their next wait or item.
    if (warp == kMdProducerWarp) {
        // ------------------------------ producer ------------------------------
        // This iteration's K/V rows (key ctx of every request, ctx its context
        // before the iteration) are appended by the previous kernel; the keys
        // before them were written by earlier iterations.  So the ring's first
        // stages, while they hold only such keys, are loaded before waiting for
        // the previous kernel: the stream starts during its tail.
        //
        // The CTA's items: the first is dealt (entry blockIdx.x, so it can
        // stream before the wait); the others are claimed at run time from the
        // plan's counter, in list order (longest first), so that SMs that
        // stream faster take more -- after the wait, so that a following
        // launch never claims before this one has ended.  Each is claimed two
        // items ahead (the atomic's round trip overlaps an item) and its id
        // handed to the consumer warps before the item before it starts.
        // Without a counter the k-th item is the dealt entry nth(k).
        if (elect_one()) {
            const uint64_t pol = l2_policy_evict_first();  // every cached row is read once per iteration
            uint32_t g = 0, issued = 0;
            bool ok = true, waited = false, claiming = a.p.claim != nullptr;
            int nxt = total, nxt2 = total;  // items k + 1 and k + 2, once known
            auto take = [&](int j) {  // the CTA's j-th item, j >= 1
                if (!a.p.claim) return nth(j);
                const int v = G + atomicAdd(a.p.claim, 1);
                if (v >= total) {  // this CTA's last claim: the last CTA to finish claiming resets the counters
                    claiming = false;
                    if (atomicAdd(a.p.claim + 1, 1) == G - 1) a.p.claim[0] = 0, a.p.claim[1] = 0;
                }
                return v;
            };
            auto publish = [&](int j, int v) {  // item j's id (j >= 1) for the consumers (the arrive releases it)
                sm.ids[(j - 1) % kMdIds] = v;
                mbar_arrive(&sm.id_full[(j - 1) % kMdIds]);
            };
            int4 r0, r1, n0, n1;
            auto grid_wait = [&]() {  // then items 1 and 2 are claimed, item 1 handed over
                pdl_wait();
                waited = true;
                nxt = take(1);
                publish(1, nxt);
                nxt2 = nxt < total ? take(2) : total;
                if (nxt < total) rec(nxt, n0, n1);  // the next record, in flight meanwhile
            };
            rec((int)blockIdx.x, n0, n1);  // (the grid has at most `total` CTAs)
            for (int k = 0, q = (int)blockIdx.x; q < total && ok; ++k, q = nxt) {
                r0 = n0, r1 = n1;
                if (k >= 1) {
                    nxt = nxt2;
                    publish(k + 1, nxt);
                    nxt2 = nxt < total ? take(k + 2) : total;
                    if (nxt < total) rec(nxt, n0, n1);
                }
                const int h = q % a.n_heads, y0 = r0.x, nk = r0.y;
                // keys [0, old) of the item precede the request's context end
                const int old = waited || !a.early ? 0 : a.p.req_ctx[r0.w] - r1.w;
                for (int t = 0; t < nk; t += kMdTok, ++g) {
                    if (!waited && (issued >= (uint32_t)S || t + min(kMdTok, nk - t) > old)) grid_wait();
                    const int s = g % S;
                    if (sm.abort || !mbar_wait_bounded(&sm.empty[s], ((g / S) & 1u) ^ 1u, a.err)) {
                        ok = false;
                        break;
                    }
                    uint8_t *dst = ring + s * kStage;
                    const int ntok = min(kMdTok, nk - t);
                    if (ntok == kMdTok) {
                        mbar_arrive_expect_tx(&sm.full[s], kStage);
#pragma unroll
                        for (int b = 0; b < NB; ++b) {
                            tma_load_3d_hint(dst + b * kBox, &tm, &sm.full[s], 64 * b, y0 + t, h, pol);
                            tma_load_3d_hint(dst + (NB + b) * kBox, &tm, &sm.full[s], 64 * b, y0 + t, a.n_heads + h,
                                             pol);
                        }
                    } else {  // 16-token boxes at 2 KiB (16-row) offsets keep the 128-byte swizzle phase
                        const int nq = (ntok + 15) / 16;
                        mbar_arrive_expect_tx(&sm.full[s], (uint32_t)nq * (kStage / (kMdTok / 16)));
                        for (int j = 0; j < nq; ++j)
#pragma unroll
                            for (int b = 0; b < NB; ++b) {
                                tma_load_3d_hint(dst + b * kBox + j * 2048, &tm16, &sm.full[s], 64 * b, y0 + t + 16 * j,
                                                 h, pol);
                                tma_load_3d_hint(dst + (NB + b) * kBox + j * 2048, &tm16, &sm.full[s], 64 * b,
                                                 y0 + t + 16 * j, a.n_heads + h, pol);
                            }
                    }
                    ++issued;
                }
                if (ok && !waited) grid_wait();  // the first item held only earlier keys, in fewer than S stages
            }
            if (!ok) {  // let the copies in flight land before the CTA exits
                sm.abort = 1;
                for (uint32_t j = issued > (uint32_t)S ? issued - S : 0; j < issued; ++j)
                    mbar_wait_bounded(&sm.full[j % S], (j / S) & 1u, a.err);
            }
        }
        return;
    }

    pdl_wait();  // q and this iteration's K/V rows come from the previous kernel
    if (warp >= kMdMergerWarp) {
        // ---------------- merge: the consumer warps' states of each item ----------------
        const int mw = warp - kMdMergerWarp;  // items k = mw, mw + kMdMergers, ...
        for (int k = mw;; k += kMdMergers) {
            const int e = k % kMdMerge;
            if (!__all_sync(0xffffffffu, !sm.abort && mbar_wait_bounded(&sm.mfull[e], (k / kMdMerge) & 1u, a.err))) {
                sm.abort = 1;
                return;
            }
            const int q = *reinterpret_cast<volatile int *>(&sm.mq[e]);  // the item, or -1: no more
            if (q < 0) return;
            int4 r0, r1;
            rec(q, r0, r1);
            const int h = q % a.n_heads, i = r0.w, c = r1.x;
            float M = kNegBig;
#pragma unroll
            for (int w = 0; w < kMdConsumers; ++w) M = fmaxf(M, sm.m[e][w]);
            float cw[kMdConsumers], L = 0.f;
#pragma unroll
            for (int w = 0; w < kMdConsumers; ++w) cw[w] = exp2f(sm.m[e][w] - M), L += sm.l[e][w] * cw[w];
            float O[D / 32];
#pragma unroll
            for (int u = 0; u < D / 32; ++u) {
                O[u] = 0.f;
#pragma unroll
                for (int w = 0; w < kMdConsumers; ++w) O[u] += sm.o[e][w][lane + 32 * u] * cw[w];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.mempty[e]);  // the entry is free again
            const int nch = r1.y;
            bf16 *dst = a.out + (size_t)r0.z * a.H + h * D;
            if (nch == 1) {
                const float inv = 1.f / L;
#pragma unroll
                for (int u = 0; u < D / 32; ++u) dst[lane + 32 * u] = __float2bfloat16_rn(O[u] * inv);
                continue;
            }
            // several chunks: publish the partial; the last to arrive merges them in chunk order
            const int wb = r1.z;
            float *mine = a.part + ((size_t)(wb + c) * a.n_heads + h) * (D + 2);
#pragma unroll
            for (int u = 0; u < D / 32; ++u) mine[lane + 32 * u] = O[u];
            if (lane == 0) mine[D] = M, mine[D + 1] = L;
            __syncwarp();  // the warp's stores, then lane 0's release
            int last = 0;
            if (lane == 0) {
                int *cnt = a.counters + i * a.n_heads + h;
                last = atom_add_acq_rel(cnt, 1) == nch - 1;
                if (last) *cnt = 0;
            }
            if (__shfl_sync(0xffffffffu, last, 0)) {
                // chunks in order, up to 4 at a time with every load in flight before the first use
                float Mt = kNegBig, Lt = 0.f, Ot[D / 32];
#pragma unroll
                for (int u = 0; u < D / 32; ++u) Ot[u] = 0.f;
                for (int j0 = 0; j0 < nch; j0 += 4) {
                    float pm[4], pl[4], po[4][D / 32];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        if (j0 + jj < nch) {
                            const float *pj = a.part + ((size_t)(wb + j0 + jj) * a.n_heads + h) * (D + 2);
                            pm[jj] = __ldcg(pj + D), pl[jj] = __ldcg(pj + D + 1);
#pragma unroll
                            for (int u = 0; u < D / 32; ++u) po[jj][u] = __ldcg(pj + lane + 32 * u);
                        }
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        if (j0 + jj < nch) {  // online merge: rescale the running sums to the new maximum
                            const float mn = fmaxf(Mt, pm[jj]);
                            const float c_old = exp2f(Mt - mn), c_new = exp2f(pm[jj] - mn);
                            Lt = Lt * c_old + pl[jj] * c_new;
#pragma unroll
                            for (int u = 0; u < D / 32; ++u) Ot[u] = Ot[u] * c_old + po[jj][u] * c_new;
                            Mt = mn;
                        }
                }
#pragma unroll
                for (int u = 0; u < D / 32; ++u) dst[lane + 32 * u] = __float2bfloat16_rn(Ot[u] / Lt);
            }
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    const int g8 = lane >> 2, t4 = lane & 3;
    const int j0 = 16 * warp;  // this warp's 16 tokens of every stage
    // q as the B operand (any column): b0 = dims 16ks + 2t4, +1; b1 = dims 16ks + 8 + 2t4, +1
    auto load_q = [&](int q, uint32_t (*qb)[2]) {
        int4 r0, r1;
        rec(q, r0, r1);
        const uint32_t *qp =
            reinterpret_cast<const uint32_t *>(a.qkv + (size_t)r0.z * 3 * a.H + (q % a.n_heads) * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) qb[ks][0] = qp[8 * ks + t4], qb[ks][1] = qp[8 * ks + 4 + t4];
    };
    uint32_t qn[KS][2];
    load_q((int)blockIdx.x, qn);  // (the grid has at most `total` CTAs)
    uint32_t g = 0;
    int k = 0;
    for (int q = (int)blockIdx.x, q_nx; q < total; ++k, q = q_nx) {
        // the CTA's next item (handed over before this one's first stage, or after the grid wait)
        // (item j >= 1 at entry (j - 1) % kMdIds, its (j - 1) / kMdIds-th use)
        if (!__all_sync(0xffffffffu, !sm.abort && mbar_wait_bounded(&sm.id_full[k % kMdIds],
                                                                    (uint32_t)(k / kMdIds) & 1u, a.err))) {
            sm.abort = 1;
            return;
        }
        q_nx = *reinterpret_cast<volatile int *>(&sm.ids[k % kMdIds]);
        int4 r0, r1;
        rec(q, r0, r1);
        const int t0 = 0, t1 = r0.y;  // keys of this item, from its first
        // keys of the item within the request's context (fewer than t1 in a
        // padded batch: the rest are loaded but masked; <= 0 for an item of
        // padding only)
        const int t_valid = a.p.req_ctx[r0.w] + 1 - r1.w;
        uint32_t qb[KS][2];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) qb[ks][0] = qn[ks][0], qb[ks][1] = qn[ks][1];
        if (q_nx < total) load_q(q_nx, qn);  // the next item's q, in flight during this one
        float m = kNegBig, l = 0.f, o[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        for (int t = t0; t < t1; t += kMdTok, ++g) {
            const int s = g % S;
            if (!__all_sync(0xffffffffu, !sm.abort && mbar_wait_bounded(&sm.full[s], (g / S) & 1u, a.err))) {
                sm.abort = 1;  // (uniform: ldmatrix and mma below are warp-wide)
                return;
            }
            const uint32_t kb = smem_u32(ring + s * kStage), vb = kb + NB * kBox;
            const int ntok = min(kMdTok, min(t1, t_valid) - t);  // rows to use (past them: masked, V zeroed)
            if (j0 < ntok) {
                // S^T = K q^T for tokens j0 .. j0 + 15: lane (g8, t4) gets tokens j0 + g8 and j0 + g8 + 8
                float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
                {
                    const int r = j0 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const int d = 16 * ks + (lane >> 4) * 8;
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(kb + (d >> 6) * kBox + r * 128 + ((((d & 63) >> 3) ^ (r & 7)) << 4), a0, a1, a2, a3);
                        mma_bf16((ks & 1) ? c1 : c0, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
                    }
                }
                const float s_lo = j0 + g8 < ntok ? (c0[0] + c1[0]) * a.scale_log2 : kNegBig;
                const float s_hi = j0 + g8 + 8 < ntok ? (c0[2] + c1[2]) * a.scale_log2 : kNegBig;
                float mx = fmaxf(s_lo, s_hi);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                if (mx > m) {  // warp-uniform
                    const float corr = exp2f(m - mx);
                    m = mx;
                    l *= corr;
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
                        o[mt][0] *= corr, o[mt][1] *= corr, o[mt][2] *= corr, o[mt][3] *= corr;
                }
                const uint32_t pw = pack_bf16(exp2f(s_lo - m), exp2f(s_hi - m));  // {p(j0 + g8), p(j0 + g8 + 8)}
                {
                    const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162 *>(&pw);
                    l += __low2float(pr) + __high2float(pr);
                }
                if (ntok < j0 + 16) {  // rows past the item may hold anything: zero this warp's in V
                    for (int idx = lane; idx < (j0 + 16 - ntok) * NB * 8; idx += 32) {
                        const int rr = ntok + idx / (NB * 8), b = (idx / 8) % NB, ch = idx % 8;
                        st_shared_zero16(vb + b * kBox + rr * 128 + ch * 16);
                    }
                    fence_proxy_async_smem();  // before the slot's next TMA write
                    __syncwarp();
                }
                // O^T += V^T p; B = p as a column: b0 = p(2t4), p(2t4 + 1); b1 = p(2t4 + 8), p(2t4 + 9)
                const uint32_t x0 = __shfl_sync(0xffffffffu, pw, 8 * t4);
                const uint32_t x1 = __shfl_sync(0xffffffffu, pw, 8 * t4 + 4);
                const uint32_t b0 = prmt(x0, x1, 0x5410), b1 = prmt(x0, x1, 0x7632);
                const int r = j0 + (lane >> 4) * 8 + (lane & 7);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const int d = 16 * mt + ((lane >> 3) & 1) * 8;
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(vb + (d >> 6) * kBox + r * 128 + ((((d & 63) >> 3) ^ (r & 7)) << 4), a0, a1, a2, a3);
                    mma_bf16(o[mt], a0, a1, a2, a3, b0, b1);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);  // this warp is done with slot s
        }
        // hand the item's state to the merge warp: l over the 8 token groups; lane (g8, t4) holds
        // o[mt][0] = dim 16mt + g8 and o[mt][2] = dim 16mt + g8 + 8
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        const int e = k % kMdMerge;
        if (k >= kMdMerge &&
            !__all_sync(0xffffffffu, !sm.abort && mbar_wait_bounded(&sm.mempty[e], ((k / kMdMerge) - 1) & 1u, a.err))) {
            sm.abort = 1;
            return;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            if ((mt & 3) == t4) sm.o[e][warp][16 * mt + g8] = o[mt][0], sm.o[e][warp][16 * mt + g8 + 8] = o[mt][2];
        if (lane == 0) sm.m[e][warp] = m, sm.l[e][warp] = l;
        if (lane == 0 && warp == 0) sm.mq[e] = q;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.mfull[e]);
    }
    // no more items: the merge warps' next entries (k and k + 1, one for each) say so
    for (int kk = k; kk < k + kMdMergers; ++kk) {
        const int e = kk % kMdMerge;
        if (kk >= kMdMerge &&
            !__all_sync(0xffffffffu, !sm.abort && mbar_wait_bounded(&sm.mempty[e], ((kk / kMdMerge) - 1) & 1u, a.err))) {
            sm.abort = 1;
            return;
        }
        if (lane == 0 && warp == 0) sm.mq[e] = -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.mfull[e]);
    }
}

template <typename T, int D>
cudaError_t launch_attn(const AttnArgs<T> &a, bool decode, bool prefill, cudaStream_t st) {
    if constexpr (std::is_same<T, bf16>::value && D % 64 == 0)
        if (decode && a.p.n_dec_work > 0) {
            {
                cudaError_t e = max_smem_once((const void *)attn_decode_mma_kernel<D>, (int)md_smem_bytes<D>());
                if (e != cudaSuccess) return e;
            }
            // the layer's pool as [K|V][head] planes of [slot][D]
            CUtensorMap tm, tm16;
            const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.kv_slots, (uint64_t)2 * a.n_heads};
            const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)a.kv_slots * D * 2};
            const uint32_t box[3] = {64, kMdTok, 1}, box16[3] = {64, 16, 1};
            if (a.kv_slots > INT32_MAX || (reinterpret_cast<uintptr_t>(a.kpool) & 15) ||
                !encode_tensor_map(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.kpool, dims, strides, box,
                                   CU_TENSOR_MAP_SWIZZLE_128B) ||
                !encode_tensor_map(&tm16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.kpool, dims, strides, box16,
                                   CU_TENSOR_MAP_SWIZZLE_128B))
                return cudaErrorInvalidValue;
            int sms = 0, dev = 0;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            const int total = a.p.n_dec_work * a.n_heads;
            const int grid = std::max(1, std::min(total, kMdCtasPerSm * sms));
            cudaError_t e = launch_pdl(attn_decode_mma_kernel<D>, dim3(grid), dim3(kMdThreads), md_smem_bytes<D>(), st,
                                       tm, tm16, a);
            if (e != cudaSuccess) return e;
            decode = false;
        }
    if (decode && a.p.n_dec_work > 0) {
        {
            cudaError_t e = max_smem_once((const void *)attn_decode_kernel<T, D>, (int)sizeof(DecodeSmem<T, D>));
            if (e != cudaSuccess) return e;
        }
        int sms = 0, dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int total = a.p.n_dec_work * a.n_heads;
        const int grid = std::max(1, std::min(total, kDecCtasPerSm * sms));
        cudaError_t e = launch_pdl(attn_decode_kernel<T, D>, dim3(grid), dim3(kDecThreads), sizeof(DecodeSmem<T, D>),
                                   st, a);
        if (e != cudaSuccess) return e;
    }
    if (prefill && a.p.n_pre_tiles > 0) {
        if constexpr (std::is_same<T, bf16>::value && (D == 64 || D == 128)) {
            {
                cudaError_t e = max_smem_once((const void *)attn_prefill_mma_kernel<D>, (int)sizeof(PrefillSmem<D>));
                if (e != cudaSuccess) return e;
            }
            cudaError_t e = cudaSuccess;
            if (a.p.n_rows > 0 && override_prefill_tc() >= 0) {
                // q as [rows][3H] (boxes of 64 dims x 128 rows), the pool as [K|V][head] planes of [slot][D]
                CUtensorMap tmq, tmkv;
                const uint64_t qdims[2] = {(uint64_t)3 * a.H, (uint64_t)a.p.n_rows};
                const uint64_t qstrides[1] = {(uint64_t)3 * a.H * 2};
                const uint32_t qbox[2] = {64, kPtRows};
                const uint64_t kdims[3] = {(uint64_t)D, (uint64_t)a.kv_slots, (uint64_t)2 * a.n_heads};
                const uint64_t kstrides[2] = {(uint64_t)D * 2, (uint64_t)a.kv_slots * D * 2};
                const uint32_t kbox[3] = {64, kPtKeys, 1};
                if (!encode_tensor_map(&tmq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.qkv, qdims, qstrides, qbox,
                                       CU_TENSOR_MAP_SWIZZLE_128B) ||
                    !encode_tensor_map(&tmkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.kpool, kdims, kstrides, kbox,
                                       CU_TENSOR_MAP_SWIZZLE_128B))
                    return cudaErrorInvalidValue;
                e = max_smem_once((const void *)attn_prefill_tc_kernel<D>, (int)PtLayout<D>::kBytes);
                if (e != cudaSuccess) return e;
                // persistent: one CTA per SM walks the (head, tile) items
                int sms = 0, dev = 0;
                cudaGetDevice(&dev);
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
                const int grid = std::max(1, std::min(a.p.n_pre_tiles * a.n_heads, sms));
                e = launch_pdl(attn_prefill_tc_kernel<D>, dim3(grid), dim3(kPtThreads), PtLayout<D>::kBytes, st, tmq,
                               tmkv, a);
            } else {
                e = launch_pdl(attn_prefill_mma_kernel<D>, dim3(a.p.n_pre_tiles, a.n_heads, 2), dim3(128),
                               sizeof(PrefillSmem<D>), st, a);
            }
            if (e != cudaSuccess) return e;
        } else {
            cudaError_t e = launch_pdl(attn_prefill_kernel<T, D>, dim3(a.p.n_pre_tiles, a.n_heads),
                                       dim3(kAttnThreads), 0, st, a);
            if (e != cudaSuccess) return e;
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

void decode_order(const int32_t *dec_work, int n_work, const int32_t *req_keys, int chunk, int32_t *order) {
    if (chunk < 1 || chunk > 512) {  // (the engine's chunks are 64 .. 512) keep the given order
        for (int w = 0; w < n_work; ++w) order[w] = w;
        return;
    }
    // counting sort of the work items by keys in the chunk (1 .. chunk <= 512), longest first
    int start[513 + 1] = {0};
    auto keys = [&](int w) {
        const int i = dec_work[2 * w], c = dec_work[2 * w + 1];
        return std::min(chunk, req_keys[i] - c * chunk);
    };
    for (int w = 0; w < n_work; ++w) ++start[chunk - keys(w) + 1];
    for (int b = 1; b <= chunk; ++b) start[b] += start[b - 1];
    for (int w = 0; w < n_work; ++w) order[start[chunk - keys(w)]++] = w;
}

void prefill_order(int32_t *pre_tiles, int n_tiles, const int32_t *req_off, const int32_t *req_ctx) {
    struct Tile {
        int32_t i, q0;
    };
    static_assert(sizeof(Tile) == 2 * sizeof(int32_t), "tiles are (request, first row) pairs");
    Tile *t = reinterpret_cast<Tile *>(pre_tiles);
    auto keys = [&](const Tile &x) {
        return req_ctx[x.i] + x.q0 + std::min(kPrefillRowsPerTile, req_off[x.i + 1] - req_off[x.i] - x.q0);
    };
    std::stable_sort(t, t + n_tiles, [&](const Tile &x, const Tile &y) { return keys(x) > keys(y); });
}

void decode_items(const int32_t *order, const int32_t *dec_work, int n_work, const int32_t *req_off,
                  const int32_t *req_keys, const int32_t *req_kvoff, const int32_t *dec_wbegin, const int32_t *dec_nch,
                  int chunk, int32_t *items) {
    for (int k = 0; k < n_work; ++k) {
        const int w = order[k], i = dec_work[2 * w], c = dec_work[2 * w + 1];
        const int t0 = c * chunk, t1 = std::min(req_keys[i], t0 + chunk);
        int32_t *r = items + 8 * (size_t)k;
        r[0] = req_kvoff[i] + t0, r[1] = t1 - t0, r[2] = req_off[i], r[3] = i;
        r[4] = c, r[5] = dec_nch[i], r[6] = dec_wbegin[i], r[7] = t0;
    }
}

template <typename T>
cudaError_t attention(const T *qkv, const T *pool_layer, int64_t kv_slots, T *out, const AttnPlan &p, int H,
                      int n_heads, float *part, int *counters, unsigned *err, cudaStream_t st, bool decode,
                      bool prefill) {
    const int D = H / n_heads;
    AttnArgs<T> a;
    a.qkv = qkv;
    a.kpool = pool_layer;
    a.vpool = pool_layer + (size_t)n_heads * kv_slots * D;
    a.kv_slots = kv_slots;
    a.out = out;
    a.H = H;
    a.n_heads = n_heads;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    a.p = p;
    a.part = part;
    a.counters = counters;
    a.err = err;
    a.early = override_decode_early() >= 0;
    switch (D) {
        case 16: return launch_attn<T, 16>(a, decode, prefill, st);
        case 32: return launch_attn<T, 32>(a, decode, prefill, st);
        case 64: return launch_attn<T, 64>(a, decode, prefill, st);
        case 128: return launch_attn<T, 128>(a, decode, prefill, st);
        default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------------------
// Allocation-free decode attention (orca_attention_decode_noalloc in orca.h).
// The split-K decode kernel above, with its scratch -- plan tables, arrival
// counters and partials -- carved out of one file-scope device array instead
// of engine-allocated buffers.  Host code must not use the array's name as a
// pointer (that is a host-side stand-in): its device address is looked up
// once per device with cudaGetSymbolAddress.
// ---------------------------------------------------------------------------
namespace {

constexpr int kNaMaxReq = 256;
constexpr int kNaMaxHeads = 128;
constexpr size_t kNaPartFloats = size_t(1) << 22;                    // 16 MiB of partials
constexpr size_t kNaCounterWords = size_t(kNaMaxReq) * kNaMaxHeads;  // 128 KiB
constexpr size_t kNaPlanWords = 8 * kNaMaxReq + 11 * 8192 + 16;      // tables + up to 8192 work items
constexpr size_t kNaScratchBytes = 4 * (kNaPartFloats + kNaCounterWords + kNaPlanWords);
constexpr int kNaMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaScratchBytes];

struct NaDevice {
    bool ready = false;
    unsigned char *scratch = nullptr;  // device address of g_noalloc_scratch
    int num_sms = 0;
};
NaDevice g_na_dev[kNaMaxDevices];
int32_t g_na_plan[kNaPlanWords];  // host staging of the tables (pageable)

}  // namespace

}  // namespace orca

extern "C" int orca_attention_decode_noalloc(int32_t dtype, const void *qkv, const void *kv_layer, int64_t kv_slots,
                                             int32_t n_heads, int32_t head_dim, int32_t n_req,
                                             const int32_t *ctx_len, const int64_t *kv_offset, void *out,
                                             void *stream) {
    using namespace orca;
    constexpr int kOk = 0, kInvalid = -1, kCuda = -3, kLimit = -7;  // ORCA_OK / _ERR_INVALID / _CUDA / _LIMIT
    if (!qkv || !kv_layer || !out || !ctx_len || !kv_offset || n_req < 1 || n_heads < 1 || kv_slots < 1 ||
        kv_slots > INT32_MAX)
        return kInvalid;
    if (dtype != 0 && dtype != 1) return kInvalid;
    if (head_dim != 16 && head_dim != 32 && head_dim != 64 && head_dim != 128) return kInvalid;
    for (int i = 0; i < n_req; ++i)
        if (ctx_len[i] < 0 || kv_offset[i] < 0 || kv_offset[i] + (int64_t)ctx_len[i] + 1 > kv_slots) return kInvalid;
    if (n_req > kNaMaxReq || n_heads > kNaMaxHeads) return kLimit;

    // once per device, with that device current: the array's device address
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices) {
        cudaGetLastError();
        return kCuda;
    }
    NaDevice &nd = g_na_dev[dev];
    if (!nd.ready) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p ||
            cudaDeviceGetAttribute(&nd.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return kCuda;
        }
        nd.scratch = static_cast<unsigned char *>(p);
        nd.ready = true;
    }

    // split-K chunking as in the engine: shrink chunks until there are a few CTAs per SM
    int chunk = 512;
    while (chunk > 64) {
        int64_t items = 0;
        for (int i = 0; i < n_req; ++i) items += ((int64_t)ctx_len[i] + chunk) / chunk;
        if (items * n_heads >= 4LL * nd.num_sms) break;
        chunk /= 2;
    }
    int64_t n_work = 0;
    for (int i = 0; i < n_req; ++i) n_work += ((int64_t)ctx_len[i] + chunk) / chunk;
    const size_t items_at = (7 * (size_t)n_req + 1 + 3 * (size_t)n_work + 3) & ~size_t(3);  // 16-byte aligned
    const size_t words = items_at + 8 * (size_t)n_work;
    if (words > kNaPlanWords || (size_t)n_work * n_heads * (head_dim + 2) > kNaPartFloats) return kLimit;

    // tables: req_off, req_ctx, req_kvoff, dec_wbegin, dec_nch, dec_work
    int32_t *req_off = g_na_plan, *req_ctx = req_off + n_req + 1, *req_kv = req_ctx + n_req;
    int32_t *dec_wb = req_kv + n_req, *dec_nch = dec_wb + n_req, *req_keys = dec_nch + n_req;
    int32_t *dec_work = req_keys + n_req;
    int32_t *dec_ord = dec_work + 2 * n_work;
    int w = 0;
    for (int i = 0; i < n_req; ++i) {
        const int nch = (int)(((int64_t)ctx_len[i] + chunk) / chunk);
        req_off[i] = i;
        req_ctx[i] = ctx_len[i];
        req_kv[i] = (int32_t)kv_offset[i];
        req_keys[i] = ctx_len[i] + 1;
        dec_wb[i] = w;
        dec_nch[i] = nch;
        for (int c = 0; c < nch; ++c, ++w) dec_work[2 * w] = i, dec_work[2 * w + 1] = c;
    }
    req_off[n_req] = n_req;
    decode_order(dec_work, (int)n_work, req_keys, chunk, dec_ord);
    decode_items(dec_ord, dec_work, (int)n_work, req_off, req_keys, req_kv, dec_wb, dec_nch, chunk, g_na_plan + items_at);

    float *part = reinterpret_cast<float *>(nd.scratch);
    int32_t *counters = reinterpret_cast<int32_t *>(part + kNaPartFloats);
    int32_t *plan = counters + kNaCounterWords;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(counters, 0, sizeof(int32_t) * (size_t)n_req * n_heads, st) != cudaSuccess ||
        cudaMemcpyAsync(plan, g_na_plan, sizeof(int32_t) * words, cudaMemcpyHostToDevice, st) != cudaSuccess) {
        cudaGetLastError();
        return kCuda;
    }
    AttnPlan ap;
    ap.req_off = plan;
    ap.req_ctx = plan + (req_ctx - g_na_plan);
    ap.req_kvoff = plan + (req_kv - g_na_plan);
    ap.dec_wbegin = plan + (dec_wb - g_na_plan);
    ap.dec_nch = plan + (dec_nch - g_na_plan);
    ap.dec_work = plan + (dec_work - g_na_plan);
    ap.dec_order = plan + (dec_ord - g_na_plan);
    ap.dec_items = plan + items_at;
    ap.req_keys = plan + (req_keys - g_na_plan);
    ap.pre_tiles = nullptr;
    ap.n_dec_work = (int)n_work;
    ap.n_pre_tiles = 0;
    ap.chunk = chunk;
    ap.n_rows = 0;
    ap.claim = nullptr;  // a fixed share per CTA: no counter to keep between calls
    const int H = n_heads * head_dim;
    cudaError_t ce =
        dtype == 1 ? attention<bf16>((const bf16 *)qkv, (const bf16 *)kv_layer, kv_slots, (bf16 *)out, ap, H, n_heads,
                                     part, counters, nullptr, st, true, false)
                   : attention<float>((const float *)qkv, (const float *)kv_layer, kv_slots, (float *)out, ap, H,
                                      n_heads, part, counters, nullptr, st, true, false);
    if (ce != cudaSuccess) {
        cudaGetLastError();
        return kCuda;
    }
    return kOk;
}

namespace orca {

template cudaError_t attention<float>(const float *, const float *, int64_t, float *, const AttnPlan &, int, int,
                                      float *, int *, unsigned *, cudaStream_t, bool, bool);
template cudaError_t attention<bf16>(const bf16 *, const bf16 *, int64_t, bf16 *, const AttnPlan &, int, int,
                                     float *, int *, unsigned *, cudaStream_t, bool, bool);

}  // namespace orca
