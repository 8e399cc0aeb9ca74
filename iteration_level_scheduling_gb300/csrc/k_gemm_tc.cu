// Flattened linear layers on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Selective batching applies every non-attention operation to all requests'
// rows at once, as one [sum L, H] matrix ("論文解説: Orca", Selective Batching;
// garden.houmin.site Orca notes, 3.1.2): the weights are read once per
// iteration for the whole batch.  The notes also observe that increment-phase
// rows make these projections GEMV-like and initiation rows GEMM-like, so one
// kernel has to serve sum L from 1 to tens of thousands.
//
// Orientation ("swap AB"): the weight is the MMA's A operand (M = 128 output
// features per CTA), the token rows are the B operand (N = BN tokens, a
// multiple of 16 up to 256; or one wide tile of 257..448 rows, taken as two
// MMAs per K step into 512 TMEM columns, in its own kernel instantiation, when
// a launch model of measured per-stage times prefers it and its CTAs fit one
// round).  Both are K-major in memory (w[f, k], x[t, k]), so
// TMA loads 64-wide K slices with 128-byte swizzling straight into the layout
// tcgen05.mma reads.  The fp32 accumulator tile (128 lanes x BN columns) lives
// in tensor memory; lane = output feature, column = token.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM owner and
// single-thread MMA issuer, warps 2-5 = epilogue (each reads its 32-lane
// quarter of TMEM).  A ring of `stages` shared-memory stages with full/empty
// mbarriers decouples loads from MMAs; tcgen05.commit releases a stage when the
// MMAs reading it are done.
//
// Small sum L (decode) gives few output tiles.  When the caller can complete
// a split-K sum itself (the residual projections: the next LayerNorm reads the
// row anyway), K is split over up to 8 CTAs per tile, each writing its fp32
// partial tile to a slab; no CTA waits on another.  Otherwise one CTA per tile
// with a deep stage ring, one CTA per SM when the tiles fit in one wave.
//
// With 129+ token rows two more launch shapes run on the stream-K kernel
// further below.  When the one-tile launch would need more than one wave of
// tiles (two waves where a stream-K workspace is given), the whole-tile walk
// (gemm_uses_whole): one persistent CTA per SM takes whole tiles in this
// kernel's raster order, its ring and a double-buffered accumulator carried
// across tiles.  Below that, with at least one output tile per SM and a
// stream-K workspace in the caller's launch context, stream-K proper
// (gemm_uses_sk).  The engine gives the workspace to stand-alone linear calls
// and to FFN1 only: elsewhere in an iteration the one-tile kernel is faster
// end to end, because its idle SMs let the next launch start early.
//
// Weights can be pre-packed (pack_weight_bf16) so each 128 x 64 stage tile is
// one contiguous, already swizzled 16 KiB block read by a single bulk copy:
// sequential DRAM streaming instead of 128 rows of 128 bytes each.
//
// Epilogue: the accumulator is staged in the idle ring (at most 256 token
// columns at a time), then + bias, exact GeLU, + residual (fp32), store fp32
// or bf16 rows [token, feature] with 16-byte (fp32) or 8-byte (bf16) stores
// along the feature dimension, four rows per warp in flight.
//
// The producer and MMA loops keep the ring slot and phase as running
// counters: they are single-thread critical paths, and a division per stage
// there (the ring depth is a run-time value) cost up to 20 %.
//
// Every mbarrier wait is bounded (see common.cuh); on expiry the CTA records
// an error bit, skips its remaining work and still frees its tensor memory.
#include <cuda.h>

#include <algorithm>
#include <cstdlib>

#include "common.cuh"
#include "kernels.cuh"

namespace orca {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 192;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxStages = 9;
constexpr int kMaxSplits = 8;  // split-K ways (partial slabs)
constexpr int kStageA = BM * BK * 2;  // 16 KiB
constexpr int kGroup = 16;            // feature tiles per raster group
constexpr int kRows = 4;              // epilogue rows per warp in flight
constexpr size_t kSmemPerSm = 228 * 1024;
constexpr size_t kSmemMaxCta = 227 * 1024;
constexpr size_t kSmemReserve = 1024;  // per CTA, kept by the driver
constexpr size_t kSmemExtra = 1024 + 256;  // alignment slack + barriers

struct TcArgs {
    int m_tok, n_out, num_kb, kb_per_split, splits, bn, stages;
    int n_feat_tiles, n_tok_tiles;
    // a token tile of more than 256 rows is two MMAs per K step: columns
    // [0, 256) with idesc, [256, bn) with idesc1 (TMEM columns likewise)
    uint32_t idesc, idesc1, tmem_cols;
    Epilogue e;
    int vec_out;  // output / residual rows allow 16-byte (fp32) or 8-byte (bf16) vector access
    int mode;     // kDirect, or kPartial (split-K slabs to e.part)
    int w_policy; // L2 policy of the weight loads: 0 evict-first (read once), 1 normal, 2 evict-last (reused)
    const bf16 *w_packed;  // weights in the tile-contiguous layout of pack_weight_bf16, or null (tensor map)
    unsigned *err;
};
enum { kDirect = 0, kPartial = 2 };

__device__ __forceinline__ void tile_coords(int lin, const TcArgs &a, int &ft, int &tt) {
    const int per_group = kGroup * a.n_tok_tiles;
    const int g = lin / per_group;
    const int first = g * kGroup;
    const int gsize = min(a.n_feat_tiles - first, kGroup);
    const int r = lin - g * per_group;
    ft = first + r % gsize;
    tt = r / gsize;
}

// AND of `v` over the 128 epilogue threads (named barrier 1).
__device__ __forceinline__ bool epilogue_all(bool v) {
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

// kWide: token tiles of more than 256 rows, two activation boxes and two MMAs
// per K step (a separate instantiation: the single MMA-issuing lane is on the
// critical path of the ordinary kernel, and a run-time branch beside every MMA
// cost it up to 20 % at decode sizes).
template <bool kWide>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx,
                   const __grid_constant__ CUtensorMap tmx1, const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stage_b = a.bn * BK * 2;
    const int stage_bytes = kStageA + stage_b;
    float *stage_c = reinterpret_cast<float *>(smem);  // accumulator tile [bn][128] after the mainloop
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.stages * stage_bytes);
    uint64_t *empty = full + kMaxStages;
    uint64_t *done = empty + kMaxStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *flags = reinterpret_cast<volatile int *>(tmem_slot + 1);  // [0] abort

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.splits;
    const int split = (int)(blockIdx.x % S);
    int ft, tt;
    tile_coords(blockIdx.x / S, a, ft, tt);
    const int kb0 = split * a.kb_per_split;
    const int nkb = min(a.num_kb, kb0 + a.kb_per_split) - kb0;
    const int t_base = tt * a.bn;
    const int t_lim = min(a.bn, a.m_tok - t_base);  // valid token columns of this tile
    const int bn0 = kWide ? 256 : a.bn;  // rows of the first activation box (the second: a.bn - 256)

    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        flags[0] = 0;
        fence_mbar_init();
        prefetch_tmap(&tmw);
        prefetch_tmap(&tmx);
        if (kWide) prefetch_tmap(&tmx1);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // The whole warp runs the loop (so addresses and coordinates stay warp-
        // uniform) and one elected lane issues the copies.
        const bool leader = elect_one();
        // with one token tile the weights are read exactly once: stream them past
        // L2; with several, the CTAs of a raster group reuse them from L2
        const bool stream_w = a.n_tok_tiles == 1;
        const uint64_t pol_w = a.w_policy == 0   ? l2_policy_evict_first()
                               : a.w_policy == 1 ? l2_policy_evict_normal()
                                                 : l2_policy_evict_last();
        // packed weights: tile (ft, kb) is one contiguous 16 KiB block, already in
        // the swizzled shared-memory image, so one bulk copy moves it
        const bf16 *wp = a.w_packed ? a.w_packed + (size_t)ft * a.num_kb * (BM * BK) : nullptr;
        auto load_w = [&](int i, int s) {
            uint8_t *sa = smem + (size_t)s * stage_bytes;
            if (wp)
                bulk_load(sa, wp + (size_t)(kb0 + i) * (BM * BK), kStageA, &full[s], pol_w);
            else if (stream_w || a.w_policy != 1)
                tma_load_2d_hint(sa, &tmw, &full[s], (kb0 + i) * BK, ft * BM, pol_w);
            else
                tma_load_2d(sa, &tmw, &full[s], (kb0 + i) * BK, ft * BM);
        };
        // The weights do not depend on earlier kernels: fill the first stages
        // with weight slices before waiting for the previous kernel, then add
        // the activation slices.
        const int pre = min(nkb, a.stages);
        if (leader)
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(&full[i], (uint32_t)stage_bytes);
                load_w(i, i);
            }
        pdl_wait();
        auto load_x = [&](int i, int s) {
            uint8_t *sb = smem + (size_t)s * stage_bytes + kStageA;
            tma_load_2d(sb, &tmx, &full[s], (kb0 + i) * BK, t_base);
            if constexpr (kWide) tma_load_2d(sb + bn0 * (BK * 2), &tmx1, &full[s], (kb0 + i) * BK, t_base + bn0);
        };
        if (leader)
            for (int i = 0; i < pre; ++i) load_x(i, i);
        __syncwarp();
        int issued = pre;
        bool ok = true;
        // ring slot and phase kept as running counters (no division per stage:
        // this loop is on the critical path)
        int s = pre == a.stages ? 0 : pre;
        uint32_t ph = pre == a.stages ? 1u : 0u;
        for (int i = pre; i < nkb; ++i) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[s], ph ^ 1u, a.err))) {
                ok = false;
                break;
            }
            if (leader) {
                mbar_arrive_expect_tx(&full[s], (uint32_t)stage_bytes);
                load_w(i, s);
                load_x(i, s);
            }
            ++issued;
            if (++s == a.stages) s = 0, ph ^= 1u;
        }
        if (!ok && leader) {
            flags[0] = 1;
            // let the copies already in flight land before the CTA exits
            for (int j = max(0, issued - a.stages); j < issued; ++j)
                mbar_wait_bounded(&full[j % a.stages], (uint32_t)(j / a.stages) & 1u, a.err);
        }
    } else if (warp == 1) {
        // whole warp in the loop, one elected lane issues the MMAs and commits
        pdl_wait();
        const bool leader = elect_one();
        bool ok = true;
        int s = 0;
        uint32_t ph = 0u;
        for (int i = 0; i < nkb; ++i) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[s], ph, a.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + (size_t)s * stage_bytes);
            const uint64_t ad = smem_desc_k128(sa), bd = smem_desc_k128(sa + kStageA);
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)  // 16 bf16 = 32 B per MMA: +2 in the >>4 address field
                    tc_mma_f16(tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), a.idesc,
                               (uint32_t)((i | kk) != 0));
                if constexpr (kWide) {  // token columns 256.. into TMEM columns 256..
                    const uint64_t bd1 = smem_desc_k128(sa + kStageA + (uint32_t)(bn0 * BK * 2));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc_mma_f16(tmem + 256u, ad + (uint64_t)(2 * kk), bd1 + (uint64_t)(2 * kk), a.idesc1,
                                   (uint32_t)((i | kk) != 0));
                }
                tc_commit(&empty[s]);
            }
            if (++s == a.stages) s = 0, ph ^= 1u;
        }
        if (leader) {
            if (ok) {
                tc_commit(done);
            } else {
                flags[0] = 1;
                mbar_arrive(done);
            }
        }
    } else {
        // the accumulator is complete once `done` fires (every MMA, hence every
        // load of the ring, has finished): the ring may then hold the staged tile
        pdl_wait();
        bool ok = mbar_wait_bounded(done, 0, a.err);
        tc_fence_after();
        ok = epilogue_all(ok && flags[0] == 0);  // the four epilogue warps take the same branch
        if (!ok && threadIdx.x == 64) flags[0] = 1;
    }
    tc_fence_before();
    __syncwarp();
    __syncthreads();

    // The epilogue in halves of at most 256 token columns (the staged fp32 half
    // tile, 128 KiB at most, fits in the ring).
    for (int cb = 0; cb < t_lim; cb += 256) {
        const int r1 = min(256, t_lim - cb);  // token rows of this half
        const int tb = t_base + cb;          // their first token
        if (cb > 0) __syncthreads();         // the previous half is stored
        // --------- phase 1: TMEM -> shared memory tile [token][feature] ---------
        if (warp >= 2 && flags[0] == 0) {
            const int quarter = warp & 3;
            const int row = quarter * 32 + lane;  // output feature within the tile
            __syncwarp();                         // tcgen05.ld is .sync.aligned
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
            for (int c0 = 0; c0 < r1; c0 += 16) {
                float v[16];
                tmem_ld16(taddr + (uint32_t)(cb + c0), v);
#pragma unroll
                for (int j = 0; j < 16; ++j) stage_c[(c0 + j) * BM + row] = v[j];
            }
        }
        tc_fence_before();
        __syncwarp();
        __syncthreads();

        // --------- phase 2: split partials, or bias / GeLU / residual, stored ---------
        if (flags[0] == 0 && a.mode == kPartial) {
            // this split's partial tile, as is, to slab `split` of the workspace
            const int f0 = ft * BM + 4 * lane;
            if (f0 < a.n_out) {
                float *slab = a.e.part + (size_t)split * a.m_tok * a.n_out;
                for (int t = warp; t < r1; t += kWarps)
                    *reinterpret_cast<float4 *>(slab + (size_t)(tb + t) * a.n_out + f0) =
                        *reinterpret_cast<const float4 *>(stage_c + t * BM + 4 * lane);
            }
        } else if (flags[0] == 0) {
            const Epilogue &e = a.e;
            const int f0 = ft * BM + 4 * lane;
            const bool full4 = a.vec_out && f0 + 3 < a.n_out;
            float4 bias = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e.bias) {
                if (f0 + 0 < a.n_out) bias.x = e.bias[f0 + 0];
                if (f0 + 1 < a.n_out) bias.y = e.bias[f0 + 1];
                if (f0 + 2 < a.n_out) bias.z = e.bias[f0 + 2];
                if (f0 + 3 < a.n_out) bias.w = e.bias[f0 + 3];
            }
            // K/V append: output features >= kv_h go to the pool at the row's slot
            bf16 *kv_dst = nullptr;
            if (e.kv_pool && f0 >= e.kv_h && f0 < a.n_out) {
                int c = f0 - e.kv_h;
                const int which = c >= e.kv_h;
                c -= which * e.kv_h;
                const int head = c / e.kv_hd;
                kv_dst = e.kv_pool + ((size_t)(which * e.kv_nh + head) * e.kv_slots) * e.kv_hd + (c - head * e.kv_hd);
            }
            for (int t0 = warp * kRows; t0 < r1; t0 += kWarps * kRows) {
                float4 acc[kRows];
                float4 res[kRows];
    #pragma unroll
                for (int u = 0; u < kRows; ++u) {
                    const int t = t0 + u;
                    acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    res[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (t < r1) {
                        acc[u] = *reinterpret_cast<const float4 *>(stage_c + t * BM + 4 * lane);
                        if (e.resid && full4)
                            res[u] = *reinterpret_cast<const float4 *>(e.resid + (size_t)(tb + t) * e.ld_out + f0);
                    }
                }
    #pragma unroll
                for (int u = 0; u < kRows; ++u) {
                    const int t = t0 + u;
                    if (t >= r1) break;
                    float y[4] = {acc[u].x + bias.x, acc[u].y + bias.y, acc[u].z + bias.z, acc[u].w + bias.w};
                    if (e.gelu) {
    #pragma unroll
                        for (int q = 0; q < 4; ++q) y[q] = gelu_erf(y[q]);
                    }
                    const size_t o = (size_t)(tb + t) * e.ld_out + f0;
                    if (full4) {
                        if (e.resid) {
                            *reinterpret_cast<float4 *>(e.out_f32 + o) =
                                make_float4(res[u].x + y[0], res[u].y + y[1], res[u].z + y[2], res[u].w + y[3]);
                        } else if (e.out_f32) {
                            *reinterpret_cast<float4 *>(e.out_f32 + o) = make_float4(y[0], y[1], y[2], y[3]);
                        } else {
                            __nv_bfloat162 lo = __floats2bfloat162_rn(y[0], y[1]), hi = __floats2bfloat162_rn(y[2], y[3]);
                            uint2 pk;
                            pk.x = *reinterpret_cast<uint32_t *>(&lo);
                            pk.y = *reinterpret_cast<uint32_t *>(&hi);
                            if (kv_dst)
                                *reinterpret_cast<uint2 *>(kv_dst + (size_t)e.row_slot[tb + t] * e.kv_hd) = pk;
                            else
                                *reinterpret_cast<uint2 *>(e.out_bf16 + o) = pk;
                        }
                    } else {
    #pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if (f0 + q >= a.n_out) break;
                            if (e.resid)
                                e.out_f32[o + q] = e.resid[o + q] + y[q];
                            else if (e.out_f32)
                                e.out_f32[o + q] = y[q];
                            else
                                e.out_bf16[o + q] = __float2bfloat16_rn(y[q]);
                        }
                    }
                }
            }
        }
    }
    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

// ---------------------------------------------------------------------------
// Stream-K variant (many token rows).
//
// With a few hundred token rows the layer is compute-bound, yet the one-tile-
// per-CTA kernel leaves SMs idle: 80 tiles on 152 SMs for the 5120-wide
// outputs, 2.1 waves of 320 tiles for the 20480-wide one, each tile paying its
// own pipeline fill and an epilogue the MMAs do not overlap.  Here the
// iteration space "tiles x 64-wide K blocks" (K block innermost) is cut into
// equal contiguous ranges, one persistent CTA per SM, so every SM does the
// same share of MMAs and streams the same share of weight bytes whatever the
// tile count.  A CTA walks its range tile piece by tile piece; the producer
// runs ahead across piece boundaries, and the accumulator is double-buffered
// in TMEM (2 x bn <= 512 columns) so the epilogue of one piece overlaps the
// MMAs of the next.  A tile cut between CTAs is completed by whichever of them
// finishes last (an arrival counter per tile; no CTA ever waits on another):
// each other piece is stored as an fp32 partial tile and the finisher sums the
// pieces in CTA order -- a fixed order, so results do not depend on timing --
// before the epilogue.
//
// Warp roles (320 threads): warp 0 = producer, warp 1 = TMEM owner and MMA
// issuer, warps 2-9 = epilogue, two per TMEM lane quarter (warp % 4), taking
// alternate 16-column chunks.  The epilogue runs straight from TMEM: thread =
// output feature, 16 token columns per tcgen05.ld, so a warp's 32 features
// make each store one contiguous run.
// ---------------------------------------------------------------------------
constexpr int kSkThreads = 320;
constexpr int kSkEpiThreads = 256;
constexpr int kSkEpiWarps = kSkEpiThreads / 32;
constexpr int kSkMaxStages = 12;
constexpr int kSkMaxBn = 256;
// after the ring: full[12], empty[12], acc_full[2], acc_empty[2] (224 B), the
// TMEM base address, flags[2]; the tile's K/V slots from byte 256
constexpr int kSkTail = 256 + kSkMaxBn * 4;
constexpr size_t kSkSmemExtra = 1024 + kSkTail;

struct SkArgs {
    int m_tok, n_out, num_kb, bn, stages;
    int n_tok_tiles, n_feat_tiles, n_units, chunk;
    // tile order: kSkFeatMajor (tile = ft * ntt + tt), kSkTokMajor (tt * nft + ft),
    // or kSkWhole: CTA b takes whole tiles b, b + G, b + 2G, ... of the one-tile
    // kernel's raster order (no tile is cut; n_units and chunk are unused)
    int order;
    uint32_t idesc, tmem_cols;
    Epilogue e;
    const bf16 *w_packed;  // tile-contiguous weights (pack_weight_bf16), or null (tensor map)
    // piece of a cut tile held by CTA b: slot 2b if it is b's first tile, else
    // 2b + 1 (a cut tile is the first or the last tile of every CTA holding a
    // piece of it); slot layout [feature 128][bn tokens]
    float *part;
    int *cnt;  // per-tile arrival counters, zero between launches
    unsigned *err;
};

enum { kSkFeatMajor = 0, kSkTokMajor = 1, kSkWhole = 2 };

__device__ __forceinline__ int sk_unit_begin(int b, const SkArgs &a) { return min(b * a.chunk, a.n_units); }
// Raster order of the whole-tile walk: groups of kGroup feature tiles, the
// token tiles inside a group, a group's feature tiles innermost.  The tiles
// that all CTAs hold at one time (consecutive in this order) then span a few
// token tiles of one group: its weights and those activations stay in L2.
__device__ __forceinline__ void sk_raster(int lin, int nft, int ntt, int &ft, int &tt) {
    const int per_group = kGroup * ntt;
    const int g = lin / per_group;
    const int first = g * kGroup;
    const int gsize = min(nft - first, kGroup);
    const int r = lin - g * per_group;
    ft = first + r % gsize;
    tt = r / gsize;
}
__device__ __forceinline__ int sk_part_slot(int b, int tile, const SkArgs &a) {
    return 2 * b + (sk_unit_begin(b, a) / a.num_kb == tile ? 0 : 1);
}
// barrier / AND over the 256 epilogue threads (named barrier 1)
__device__ __forceinline__ void sk_epi_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool sk_epi_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, 256, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(kSkThreads, 1)
    gemm_sk_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx, const SkArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stage_bytes = kStageA + a.bn * BK * 2;
    uint8_t *tail = smem + (size_t)a.stages * stage_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(tail);
    uint64_t *empty = full + kSkMaxStages;
    uint64_t *acc_full = empty + kSkMaxStages;  // [2] accumulator buffer ready for the epilogue
    uint64_t *acc_empty = acc_full + 2;         // [2] accumulator buffer drained
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 2);
    volatile int *flags = reinterpret_cast<volatile int *>(tmem_slot + 1);  // [0] abort, [1] finisher
    int *tile_slot = reinterpret_cast<int *>(tail + 256);                  // [bn] K/V pool slot of each token

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Tile order.  Feature-tile major, a CTA takes a feature tile's token
    // tiles one after the other, re-reading its weights.  Token-tile major
    // (chosen with four or more token tiles), the CTAs holding the token tiles
    // of one feature tile are nft * nkb units apart: they walk the same weight
    // blocks at about the same time and share them in L2.  Whole tiles: this
    // CTA's units are numbered 0.. over its own tiles (tile index j of the
    // walk = raster tile blockIdx.x + j * gridDim.x), so no unit range cuts a tile.
    const int nkb = a.num_kb, ntt = a.n_tok_tiles, nft = a.n_feat_tiles;
    const bool whole = a.order == kSkWhole;
    const int n_whole = whole ? max(0, (nft * ntt - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x) : 0;
    const int u_begin = whole ? 0 : sk_unit_begin(blockIdx.x, a);
    const int u_end = whole ? n_whole * nkb : sk_unit_begin(blockIdx.x + 1, a);
    auto coords = [&](int tile, int &ft, int &tt) {
        if (whole) {
            sk_raster((int)blockIdx.x + tile * (int)gridDim.x, nft, ntt, ft, tt);
        } else {
            ft = a.order == kSkTokMajor ? tile % nft : tile / ntt;
            tt = a.order == kSkTokMajor ? tile / nft : tile % ntt;
        }
    };

    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kSkEpiWarps);  // one arrival per epilogue warp
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
        prefetch_tmap(&tmw);
        prefetch_tmap(&tmx);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        // Stage i of the ring holds unit u_begin + i; the whole warp runs the
        // loop (warp-uniform control) and one elected lane issues the copies.
        const bool leader = elect_one();
        // weights are streamed past L2 unless token tiles share them there
        const uint64_t pol_w = a.order != kSkFeatMajor ? l2_policy_evict_normal() : l2_policy_evict_first();
        // A unit's tile and K block are tracked as running counters, and the
        // ring slot and phase too: no division per stage on this path.
        struct Cursor {
            int tile, kb, ft, tt;
        };
        auto cursor_at = [&](int u) {
            Cursor c;
            c.tile = u / nkb;
            c.kb = u - c.tile * nkb;
            coords(c.tile, c.ft, c.tt);
            return c;
        };
        auto step = [&](Cursor &c) {
            if (++c.kb == nkb) {
                c.kb = 0;
                ++c.tile;
                coords(c.tile, c.ft, c.tt);
            }
        };
        auto load_w = [&](const Cursor &c, int s) {
            uint8_t *sa = smem + (size_t)s * stage_bytes;
            if (a.w_packed)  // tile (ft, kb) is one contiguous 16 KiB block, already in the swizzled image
                bulk_load(sa, a.w_packed + ((size_t)c.ft * nkb + c.kb) * (BM * BK), kStageA, &full[s], pol_w);
            else
                tma_load_2d(sa, &tmw, &full[s], c.kb * BK, c.ft * BM);
        };
        auto load_x = [&](const Cursor &c, int s) {
            tma_load_2d(smem + (size_t)s * stage_bytes + kStageA, &tmx, &full[s], c.kb * BK, c.tt * a.bn);
        };
        const int n_mine = u_end - u_begin;
        // the weights do not depend on earlier kernels: fill the first stages
        // with weight slices before waiting for the previous kernel
        const int pre = min(n_mine, a.stages);
        Cursor cw = cursor_at(u_begin);
        if (leader)
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(&full[i], (uint32_t)stage_bytes);
                load_w(cw, i);
                step(cw);
            }
        pdl_wait();
        Cursor cx = cursor_at(u_begin);
        if (leader)
            for (int i = 0; i < pre; ++i) {
                load_x(cx, i);
                step(cx);
            }
        __syncwarp();
        // the copies of units u_begin + pre .. follow (cw and cx are only
        // advanced by the leader: recompute them warp-wide)
        Cursor c = cursor_at(u_begin + pre);
        int issued = pre;
        bool ok = true;
        int s = pre == a.stages ? 0 : pre;
        uint32_t ph = pre == a.stages ? 1u : 0u;
        for (int i = pre; i < n_mine; ++i) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[s], ph ^ 1u, a.err))) {
                ok = false;
                break;
            }
            if (leader) {
                mbar_arrive_expect_tx(&full[s], (uint32_t)stage_bytes);
                load_w(c, s);
                load_x(c, s);
            }
            __syncwarp();
            ++issued;
            step(c);
            if (++s == a.stages) s = 0, ph ^= 1u;
        }
        if (!ok && leader) {
            flags[0] = 1;
            // let the copies already in flight land before the CTA exits
            for (int j = max(0, issued - a.stages); j < issued; ++j)
                mbar_wait_bounded(&full[j % a.stages], (uint32_t)(j / a.stages) & 1u, a.err);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        const bool leader = elect_one();
        bool ok = true;
        int i = 0, p = 0;
        int s = 0;  // ring slot and phase of unit u_begin + i
        uint32_t ph = 0u;
        for (int u = u_begin; u < u_end; ++p) {
            const int tile = u / nkb, k0 = u - tile * nkb, k1 = min(nkb, k0 + (u_end - u));
            const int buf = p & 1;
            if (p >= 2) {  // the epilogue has drained this buffer's previous piece
                if (!__all_sync(0xffffffffu,
                                mbar_wait_bounded(&acc_empty[buf], (uint32_t)((p - 2) >> 1) & 1u, a.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            const uint32_t d_tmem = tmem + (uint32_t)(buf * a.bn);
            for (int kb = k0; kb < k1; ++kb, ++i) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[s], ph, a.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + (size_t)s * stage_bytes);
                const uint64_t ad = smem_desc_k128(sa), bd = smem_desc_k128(sa + kStageA);
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)  // 16 bf16 = 32 B per MMA: +2 in the >>4 address field
                        tc_mma_f16(d_tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), a.idesc,
                                   (uint32_t)(kb != k0 || kk != 0));
                    tc_commit(&empty[s]);
                }
                __syncwarp();
                if (++s == a.stages) s = 0, ph ^= 1u;
            }
            if (!ok) break;
            if (leader) tc_commit(&acc_full[buf]);
            __syncwarp();
            u += k1 - k0;
        }
        if (!ok && leader) {
            flags[0] = 1;
            tc_commit(&acc_full[p & 1]);  // arrives once every MMA issued so far has completed
        }
    } else {
        // ------------------------------ epilogue ------------------------------
        pdl_wait();
        const Epilogue &e = a.e;
        const int quarter = warp & 3;        // TMEM lanes 32 * (warp % 4) ..
        const int half = (warp - 2) >> 2;    // this warp's 16-column chunks: c0 = 16 * half + 32 j
        const int row = quarter * 32 + lane;  // output feature within the tile
        const int et = threadIdx.x - 64;     // 0 .. 255
        const uint32_t lane_taddr = tmem + ((uint32_t)(quarter * 32) << 16);
        int p = 0;
        for (int u = u_begin; u < u_end; ++p) {
            const int tile = u / nkb, k0 = u - tile * nkb, k1 = min(nkb, k0 + (u_end - u));
            u += k1 - k0;
            const int buf = p & 1;
            int ft, tt;
            coords(tile, ft, tt);
            const int t_base = tt * a.bn, t_lim = min(a.bn, a.m_tok - t_base);
            const int f = ft * BM + row;
            const bool f_ok = f < a.n_out;
            // everything the epilogue reads is fetched while the MMAs run
            const float bias = (e.bias && f_ok) ? e.bias[f] : 0.f;
            // K/V append: output features >= kv_h go to the pool at the row's slot
            bf16 *kv_dst = nullptr;
            if (e.kv_pool && f_ok && f >= e.kv_h) {
                int c = f - e.kv_h;
                const int which = c >= e.kv_h;
                c -= which * e.kv_h;
                const int head = c / e.kv_hd;
                kv_dst = e.kv_pool + ((size_t)(which * e.kv_nh + head) * e.kv_slots) * e.kv_hd + (c - head * e.kv_hd);
            }
            if (e.kv_pool) {
                sk_epi_sync();  // the previous piece's slots are no longer read
                for (int t = et; t < t_lim; t += kSkEpiThreads) tile_slot[t] = e.row_slot[t_base + t];
                sk_epi_sync();
            }
            // A cut tile: its pieces are summed in CTA order b_first .. b_last by
            // the finisher -- the piece that finds every other piece stored
            // (its own part straight from TMEM), else the last to arrive.
            const bool cut = !(k0 == 0 && k1 == nkb);
            const int b_first = cut ? (tile * nkb) / a.chunk : 0;
            const int b_last = cut ? (tile * nkb + nkb - 1) / a.chunk : 0;
            auto piece = [&](int b) { return a.part + (size_t)sk_part_slot(b, tile, a) * a.bn * BM + (size_t)row * a.bn; };
            auto others_stored = [&]() {  // uniform over the epilogue threads
                if (et == 0) flags[1] = ld_acquire(&a.cnt[tile]) == b_last - b_first;
                sk_epi_sync();
                const bool r = flags[1];
                sk_epi_sync();
                return r;
            };
            bool fast = cut && others_stored();
            const bool ok = mbar_wait_bounded(&acc_full[buf], (uint32_t)(p >> 1) & 1u, a.err);
            tc_fence_after();
            if (!sk_epi_all(ok && flags[0] == 0)) {  // the epilogue warps leave together
                if (et == 0) flags[0] = 1;
                break;
            }
            __syncwarp();  // tcgen05.ld is .sync.aligned
            // bias / GeLU / residual / store of 16 token columns from c0 (v is overwritten)
            auto finish = [&](float *v, int c0) {
                if (!f_ok) return;
                const int n = min(16, t_lim - c0);
                const size_t ld = (size_t)e.ld_out;
                const size_t o0 = (size_t)(t_base + c0) * ld + f;
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += bias;
                if (e.gelu) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = gelu_erf(v[j]);
                }
                if (e.resid) {
                    float r[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) r[j] = j < n ? e.resid[o0 + j * ld] : 0.f;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (j < n) e.out_f32[o0 + j * ld] = v[j] + r[j];
                } else if (e.out_f32) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (j < n) e.out_f32[o0 + j * ld] = v[j];
                } else if (kv_dst) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (j < n) kv_dst[(size_t)tile_slot[c0 + j] * e.kv_hd] = __float2bfloat16_rn(v[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (j < n) e.out_bf16[o0 + j * ld] = __float2bfloat16_rn(v[j]);
                }
            };
            auto release = [&]() {  // this accumulator buffer may take the next piece
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[buf]);
            };
            // v = sum of the pieces in CTA order over 16 tokens from c0, this
            // CTA's own values in its place; two pieces in flight at a time
            auto sum_pieces = [&](float *v, const float *own, int c0) {
                float acc[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] = 0.f;
                for (int b = b_first; b <= b_last; b += 2) {
                    float4 q[2][4];
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        if (b + i <= b_last && b + i != (int)blockIdx.x) {
                            const float4 *src = reinterpret_cast<const float4 *>(piece(b + i) + c0);
#pragma unroll
                            for (int h = 0; h < 4; ++h) q[i][h] = __ldcg(src + h);
                        }
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        if (b + i > b_last) break;
                        if (b + i == (int)blockIdx.x) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) acc[j] += own[j];
                        } else {
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                acc[4 * h] += q[i][h].x, acc[4 * h + 1] += q[i][h].y;
                                acc[4 * h + 2] += q[i][h].z, acc[4 * h + 3] += q[i][h].w;
                            }
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = acc[j];
            };
            const uint32_t taddr = lane_taddr + (uint32_t)(buf * a.bn);
            auto finish_tile = [&]() {  // the finisher: own piece from TMEM, the others from their slots
                for (int c0 = 16 * half; c0 < t_lim; c0 += 32) {
                    float own[16], v[16];
                    tmem_ld16(taddr + c0, own);
                    sum_pieces(v, own, c0);
                    finish(v, c0);
                }
            };
            if (!cut) {
                // the whole tile is in this CTA's accumulator
                for (int c0 = 16 * half; c0 < t_lim; c0 += 32) {
                    float v[16];
                    tmem_ld16(taddr + c0, v);
                    finish(v, c0);
                }
            } else {
                if (!fast) fast = others_stored();  // second look, now that this piece is done
                if (fast) {
                    finish_tile();
                    if (et == 0) a.cnt[tile] = 0;  // every other piece has arrived: ready for the next launch
                } else {
                    // store this piece and arrive; the last to arrive completes the tile
                    float *mine = piece(blockIdx.x);
                    for (int c0 = 16 * half; c0 < t_lim; c0 += 32) {
                        float v[16];
                        tmem_ld16(taddr + c0, v);
#pragma unroll
                        for (int h = 0; h < 4; ++h)
                            *reinterpret_cast<float4 *>(mine + c0 + 4 * h) =
                                make_float4(v[4 * h], v[4 * h + 1], v[4 * h + 2], v[4 * h + 3]);
                    }
                    sk_epi_sync();  // every thread's stores precede the one release below
                    if (et == 0) {
                        __threadfence();
                        const int old = atom_add_acq_rel(&a.cnt[tile], 1);
                        const int last = old == b_last - b_first;
                        if (last) a.cnt[tile] = 0;
                        flags[1] = last;
                    }
                    sk_epi_sync();
                    const bool last = flags[1];
                    sk_epi_sync();  // flags[1] is read by all before it is rewritten
                    if (last) finish_tile();
                }
            }
            release();
        }
    }
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

// Pack w [n_out, k] into tiles of 128 rows x 64 columns, tile (ft, kb) at
// element offset (ft * (k / 64) + kb) * 8192, each tile laid out exactly as
// the 128-byte-swizzled K-major shared-memory image (row r at r * 128 bytes,
// 16-byte chunk c at position c ^ (r % 8)); rows past n_out are zero.
__global__ void __launch_bounds__(256) pack_weight_kernel(const bf16 *w, int n_out, int k, bf16 *out) {
    pdl_trigger();
    pdl_wait();
    const int num_kb = k / BK;
    const int ft = blockIdx.x / num_kb, kb = blockIdx.x % num_kb;
    uint4 *dst = reinterpret_cast<uint4 *>(out + (size_t)blockIdx.x * (BM * BK));
    for (int idx = threadIdx.x; idx < BM * 8; idx += 256) {
        const int r = idx >> 3, c = idx & 7;
        const int row = ft * BM + r;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < n_out) v = *reinterpret_cast<const uint4 *>(w + (size_t)row * k + kb * BK + c * 8);
        dst[r * 8 + (c ^ (r & 7))] = v;
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D bf16 map over a row-major [rows, k] matrix, box = 64 (k) x box_rows, 128B swizzle.
bool make_map(CUtensorMap *m, const void *ptr, int rows, int k, int box_rows) {
    const uint64_t dims[2] = {(uint64_t)k, (uint64_t)rows};
    const uint64_t strides[1] = {(uint64_t)k * 2};
    const uint32_t box[2] = {(uint32_t)BK, (uint32_t)box_rows};
    return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Optional tuning overrides (ORCA_GEMM_SPLITS, ORCA_GEMM_STAGES, ORCA_GEMM_SK), read once.
int env_int(const char *name) {
    const char *v = getenv(name);
    return v ? atoi(v) : 0;
}
int override_splits() {
    static int v = env_int("ORCA_GEMM_SPLITS");
    return v;
}
int override_stages() {
    static int v = env_int("ORCA_GEMM_STAGES");
    return v;
}
// ORCA_GEMM_WPOL: L2 policy of the weights, 1 normal, 2 evict-last, 3
// evict-first; unset = by token tiles (tuning).
int override_wpol() {
    static int v = env_int("ORCA_GEMM_WPOL");
    return v;
}

// ORCA_GEMM_SK: 1 = stream-K whenever the workspace allows, -1 = never,
// unset / 0 = by token rows (kSkMinRows).
int override_sk() {
    static int v = env_int("ORCA_GEMM_SK");
    return v;
}
constexpr int kSkMinRows = 129;
// Above this many rows the one-tile kernel is used: its raster groups keep 16
// feature tiles' weights in L2 while every token tile streams past them, where
// the stream-K order (token tiles outermost from four of them) re-streams the
// whole weight once per token tile.  Measured on the 13B FFN1 at 25777 rows:
// stream-K 7.99 ms with 55 GB of DRAM reads, one-tile about 1.4x faster.
constexpr int kSkMaxRows = 1024;
// ORCA_GEMM_WHOLE: 1 = the whole-tile persistent walk whenever the one-tile
// launch needs two waves or more (more than one without a stream-K
// workspace), 2 = more than one wave in any case, -1 = never; unset = the
// same as 1 from kWholeMinRows rows (tuning, tests).
// Measured on the 13B shapes (stand-alone): QKV at 572 rows 98.5 -> 82.6 us,
// FFN1 at 1024 rows 229 -> 161 us, at 25777 rows 4621 -> 3101 us; inside the
// 13B trace's window 6656 -> 6713 tok/s; at 64 rows the LM head (393 tiles)
// is 2.4 us slower, hence the row floor.
int override_whole() {
    static int v = env_int("ORCA_GEMM_WHOLE");
    return v;
}
constexpr int kWholeMinRows = 129;

}  // namespace

bool encode_tensor_map(CUtensorMap *m, CUtensorMapDataType dt, uint32_t rank, const void *base, const uint64_t *dims,
                       const uint64_t *strides, const uint32_t *box, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], estr[5];
    for (uint32_t r = 0; r < rank; ++r) {
        d[r] = dims[r];
        bx[r] = box[r];
        estr[r] = 1;
        if (r + 1 < rank) st[r] = strides[r];
    }
    return fn(m, dt, rank, const_cast<void *>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// Widest token tile: two MMAs per K step (256 + up to 192 columns of TMEM) and
// a ring of three 72 KiB stages.
constexpr int kMaxBn = 448;

// Launch shape with `ntt` token tiles.
TcShape tc_shape_tiles(int m_tok, int n_out, int k, const GemmScratch &s, bool allow_partial, size_t part_cap,
                       int ntt) {
    TcShape t{};
    const int m = std::max(m_tok, 1);
    t.n_tok_tiles = ntt;
    t.bn = std::min(kMaxBn, std::max(16, ceil_div(ceil_div(m, ntt), 16) * 16));
    t.n_feat_tiles = ceil_div(n_out, BM);
    t.tmem_cols = 32;
    while ((int)t.tmem_cols < t.bn) t.tmem_cols *= 2;
    const int num_kb = k / BK;
    const int tiles = t.n_tok_tiles * t.n_feat_tiles;
    // split-K only into partial slabs the caller completes, and only up to one CTA per SM
    int splits = 1;
    if (allow_partial && n_out % 4 == 0 && 2 * tiles <= s.num_sms) {
        splits = std::max(1, std::min({kMaxSplits, s.num_sms / tiles, num_kb / 4}));
        if (override_splits() > 0) splits = std::min({override_splits(), kMaxSplits, num_kb});
        while (splits > 1 && (size_t)splits * m_tok * n_out > part_cap) --splits;
    }
    t.kb_per_split = ceil_div(num_kb, splits);
    t.splits = ceil_div(num_kb, t.kb_per_split);
    // one CTA per SM with a deep ring when everything runs in one wave, else two
    const int ctas_per_sm = (tiles * t.splits > s.num_sms && t.bn <= 128) ? 2 : 1;
    const size_t budget = std::min(kSmemMaxCta, kSmemPerSm / ctas_per_sm - kSmemReserve) - kSmemExtra;
    const int stage_bytes = kStageA + t.bn * BK * 2;
    const size_t max_stages_1cta = (kSmemMaxCta - kSmemExtra) / stage_bytes;
    t.stages = std::min<int>(kMaxStages, (int)(budget / stage_bytes));
    if (override_stages() > 0) t.stages = std::min<int>(std::min(override_stages(), kMaxStages), (int)max_stages_1cta);
    // the ring must also hold a staged fp32 half tile (min(bn, 256) x 512 B) after the mainloop
    while ((size_t)t.stages * stage_bytes < (size_t)std::min(t.bn, 256) * BM * 4 && t.stages < (int)max_stages_1cta)
        ++t.stages;
    t.smem = (size_t)t.stages * stage_bytes + kSmemExtra;
    return t;
}

// Modelled time of a shape (microseconds): rounds of CTAs, each taking its K
// blocks at the time one ring stage of a token tile of bn rows was measured to
// take on a GB300 (one CTA per SM, 13B layer shapes, stand-alone launches:
// 0.46 us at 64 rows, where streaming the 16 KiB weight block bounds it, 0.47
// at 176, 0.58 at 192, 0.835 at 304, 0.86 at 336, 0.94 at 448; linear in
// between), plus a fixed cost per round for the pipeline fill and epilogue.
double tc_stage_us(int bn) {
    static const double pts[][2] = {{64, 0.46}, {176, 0.47}, {192, 0.58}, {304, 0.835}, {336, 0.86}, {448, 0.94}};
    const int n = (int)(sizeof(pts) / sizeof(pts[0]));
    if (bn <= pts[0][0]) return pts[0][1];
    for (int i = 1; i < n; ++i)
        if (bn <= pts[i][0])
            return pts[i - 1][1] + (bn - pts[i - 1][0]) * (pts[i][1] - pts[i - 1][1]) / (pts[i][0] - pts[i - 1][0]);
    return pts[n - 1][1];
}
double tc_model_us(const TcShape &t, int num_sms) {
    const int ctas = t.n_tok_tiles * t.n_feat_tiles * t.splits;
    const int per_round = std::max(1, num_sms) * ((ctas > num_sms && t.bn <= 128) ? 2 : 1);
    const int rounds = ceil_div(ctas, per_round);
    return rounds * (t.kb_per_split * tc_stage_us(t.bn) + 4.0);
}

}  // namespace

// Token tiles of at most 256 rows; with 257..448 rows one wide token tile when
// all its CTAs run in one round and the model prefers it (its weights are then
// streamed once instead of once per token tile, and fewer tiles leave room for
// split-K).  Measured on the 13B shapes: QKV at 335 rows 74.8 -> 68.8 us; FFN1,
// whose 160 wide tiles need two rounds, 115 -> 146 us, hence the round rule.
TcShape gemm_tc_shape(int m_tok, int n_out, int k, const GemmScratch &s, bool allow_partial, size_t part_cap) {
    const int m = std::max(m_tok, 1);
    TcShape best = tc_shape_tiles(m_tok, n_out, k, s, allow_partial, part_cap, ceil_div(m, 256));
    if (m > 256 && m <= kMaxBn) {
        const TcShape one = tc_shape_tiles(m_tok, n_out, k, s, allow_partial, part_cap, 1);
        if (one.n_feat_tiles * one.splits <= s.num_sms && tc_model_us(one, s.num_sms) < tc_model_us(best, s.num_sms))
            best = one;
    }
    return best;
}

size_t packed_weight_elems(int n_out, int k) { return (size_t)ceil_div(n_out, BM) * BM * (size_t)k; }

SkShape gemm_sk_shape(int m_tok, int n_out, int k, int num_sms) {
    SkShape t{};
    const int m = std::max(m_tok, 1);
    t.n_tok_tiles = ceil_div(m, kSkMaxBn);
    t.bn = std::min(kSkMaxBn, std::max(16, ceil_div(ceil_div(m, t.n_tok_tiles), 16) * 16));
    t.n_feat_tiles = ceil_div(n_out, BM);
    t.tiles = t.n_tok_tiles * t.n_feat_tiles;
    t.num_kb = k / BK;
    t.units = t.tiles * t.num_kb;
    const int g0 = std::max(1, std::min(num_sms, t.units));
    t.chunk = ceil_div(t.units, g0);
    t.grid = ceil_div(t.units, t.chunk);
    t.tmem_cols = 32;  // two accumulator buffers of bn columns
    while (t.tmem_cols < 2 * t.bn) t.tmem_cols *= 2;
    const int stage_bytes = kStageA + t.bn * BK * 2;
    t.stages = std::min<int>(kSkMaxStages, (int)((kSmemMaxCta - kSkSmemExtra) / stage_bytes));
    if (override_stages() > 0) t.stages = std::min(t.stages, override_stages());
    t.smem = (size_t)t.stages * stage_bytes + kSkSmemExtra;
    t.part_floats = (size_t)2 * t.grid * t.bn * BM;
    return t;
}

size_t gemm_sk_part_floats(int num_sms) { return (size_t)2 * std::max(num_sms, 1) * kSkMaxBn * BM; }
int gemm_sk_counters(int max_rows, int max_n) {
    // at least 64 Ki tiles, so stand-alone linear calls of other shapes qualify too
    return std::max(1 << 16, ceil_div(std::max(max_rows, 1), kSkMaxBn) * ceil_div(std::max(max_n, 1), BM));
}

// The whole-tile persistent walk (SkArgs::order == kSkWhole) for layers whose
// one-tile launch needs several waves: one CTA per SM keeps its ring streaming
// across tiles and drains each accumulator while the next tile's MMAs run,
// where every one-tile CTA pays its own pipeline fill and an epilogue nothing
// overlaps.  It cuts no tile, so it needs no workspace.
bool gemm_uses_whole(int m_tok, int n_out, int k, const GemmScratch &s) {
    if (m_tok <= 0 || k % BK != 0 || k <= 0 || n_out <= 0 || override_whole() < 0) return false;
    const SkShape t = gemm_sk_shape(m_tok, n_out, k, s.num_sms);
    // from two waves of tiles; from more than one where the caller gives no
    // stream-K workspace (stream-K balances one to two waves better, where
    // it may run: FFN1 at 200 rows 67 us against 81 us on the walk)
    const bool one_wave = override_whole() == 2 || !s.sk_part;
    if (t.stages < 2 || t.tiles < (one_wave ? s.num_sms + 1 : 2 * s.num_sms)) return false;
    return override_whole() > 0 || m_tok >= kWholeMinRows;
}

bool gemm_uses_sk(int m_tok, int n_out, int k, const GemmScratch &s) {
    if (!s.sk_part || !s.sk_cnt || m_tok <= 0 || k % BK != 0 || k <= 0 || n_out <= 0) return false;
    if (override_sk() < 0) return false;
    const SkShape t = gemm_sk_shape(m_tok, n_out, k, s.num_sms);
    // by default only with many rows and at least one tile per CTA, so a tile
    // is cut at most once (a two-piece finish)
    if (override_sk() == 0 && (m_tok < kSkMinRows || m_tok > kSkMaxRows || t.tiles < t.grid)) return false;
    return t.tiles <= s.sk_cnt_n && t.part_floats <= s.sk_part_floats && t.stages >= 2 &&
           !(reinterpret_cast<uintptr_t>(s.sk_part) & 15);
}

namespace {
cudaError_t launch_sk(const bf16 *x, int x_rows_cap, const bf16 *w, bool w_packed, int m_tok, int n_out, int k,
                      const Epilogue &e, const GemmScratch &s, cudaStream_t st, bool whole) {
    SkShape t = gemm_sk_shape(m_tok, n_out, k, s.num_sms);
    if (whole) t.grid = std::min(t.tiles, s.num_sms);
    {
        cudaError_t ae = max_smem_once((const void *)gemm_sk_kernel, (int)kSmemMaxCta);
        if (ae != cudaSuccess) return ae;
    }
    CUtensorMap mw, mx;
    if (!make_map(&mw, w, w_packed ? BM : n_out, k, BM) || !make_map(&mx, x, x_rows_cap, k, t.bn))
        return cudaErrorInvalidValue;  // (the weight map is unused when the weights are packed)
    SkArgs a;
    a.m_tok = m_tok;
    a.n_out = n_out;
    a.num_kb = t.num_kb;
    a.bn = t.bn;
    a.stages = t.stages;
    a.n_tok_tiles = t.n_tok_tiles;
    a.n_feat_tiles = t.n_feat_tiles;
    a.order = whole ? kSkWhole : t.n_tok_tiles >= 4 ? kSkTokMajor : kSkFeatMajor;
    a.n_units = t.units;
    a.chunk = t.chunk;
    a.idesc = idesc_bf16_f32(BM, t.bn);
    a.tmem_cols = (uint32_t)t.tmem_cols;
    a.e = e;
    a.w_packed = w_packed ? w : nullptr;
    a.part = whole ? nullptr : s.sk_part;
    a.cnt = whole ? nullptr : s.sk_cnt;
    a.err = s.err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(t.grid);
    cfg.blockDim = dim3(kSkThreads);
    cfg.dynamicSmemBytes = t.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_sk_kernel, mw, mx, a);
}
}  // namespace

cudaError_t gemm_tc_bf16(const bf16 *x, int x_rows_cap, const bf16 *w, bool w_packed, int m_tok, int n_out, int k,
                         const Epilogue &e, const GemmScratch &s, cudaStream_t st, int *n_partials) {
    if (n_partials) *n_partials = 0;
    if (m_tok <= 0) return cudaSuccess;
    if (k % BK != 0 || k <= 0 || n_out <= 0 || x_rows_cap < m_tok) return cudaErrorInvalidValue;
    if (e.kv_pool && (e.kv_hd % 4 != 0 || !e.row_slot || !e.out_bf16)) return cudaErrorInvalidValue;
    if (w_packed && (reinterpret_cast<uintptr_t>(w) & 15)) return cudaErrorInvalidValue;
    if (gemm_uses_whole(m_tok, n_out, k, s)) return launch_sk(x, x_rows_cap, w, w_packed, m_tok, n_out, k, e, s, st, true);
    if (gemm_uses_sk(m_tok, n_out, k, s)) return launch_sk(x, x_rows_cap, w, w_packed, m_tok, n_out, k, e, s, st, false);
    const bool allow_partial = e.part != nullptr && !(reinterpret_cast<uintptr_t>(e.part) & 15);
    const TcShape t = gemm_tc_shape(m_tok, n_out, k, s, allow_partial, e.part_cap);
    if (t.stages < 2 || (size_t)t.stages * (kStageA + t.bn * BK * 2) < (size_t)std::min(t.bn, 256) * BM * 4)
        return cudaErrorInvalidValue;
    {
        cudaError_t ae = max_smem_once((const void *)gemm_tc_kernel<false>, (int)kSmemMaxCta);
        if (ae == cudaSuccess) ae = max_smem_once((const void *)gemm_tc_kernel<true>, (int)kSmemMaxCta);
        if (ae != cudaSuccess) return ae;
    }
    CUtensorMap mw, mx, mx1;
    const int bn0 = std::min(t.bn, 256), bn1 = t.bn - bn0;
    if (!make_map(&mw, w, w_packed ? BM : n_out, k, BM) || !make_map(&mx, x, x_rows_cap, k, bn0) ||
        !make_map(&mx1, x, x_rows_cap, k, bn1 ? bn1 : bn0))
        return cudaErrorInvalidValue;  // (the weight map is unused when the weights are packed)
    TcArgs a;
    a.m_tok = m_tok;
    a.n_out = n_out;
    a.num_kb = k / BK;
    a.kb_per_split = t.kb_per_split;
    a.splits = t.splits;
    a.bn = t.bn;
    a.stages = t.stages;
    a.n_feat_tiles = t.n_feat_tiles;
    a.n_tok_tiles = t.n_tok_tiles;
    a.idesc = idesc_bf16_f32(BM, bn0);
    a.idesc1 = idesc_bf16_f32(BM, bn1 ? bn1 : 16);
    a.tmem_cols = (uint32_t)t.tmem_cols;
    a.e = e;
    const uintptr_t align_mask = e.out_bf16 ? 7 : 15;
    a.vec_out = (e.ld_out % 4 == 0) &&
                !(reinterpret_cast<uintptr_t>(e.out_f32 ? (const void *)e.out_f32 : (const void *)e.out_bf16) & align_mask) &&
                !(reinterpret_cast<uintptr_t>(e.resid) & 15);
    if (e.kv_pool && !a.vec_out) return cudaErrorInvalidValue;
    a.mode = t.splits == 1 ? kDirect : kPartial;
    // Weights stream past L2 (evict-first) unless many token tiles reuse them
    // long after their first read: up to 8 token tiles the tiles that share a
    // weight block run at about the same time and hit it in L2 anyway, and
    // evict-first leaves L2 to the activations (13B QKV at 572 rows 866 ->
    // 927 TFLOP/s); with 101 token tiles (25777 rows) evict-first made every
    // token tile re-read the weights from DRAM (13.1 GB read, against 2.3 GB
    // with the normal policy; 1210 -> 1354 TFLOP/s).
    a.w_policy = override_wpol() == 1 ? 1 : override_wpol() == 2 ? 2 : override_wpol() == 3 ? 0
                 : t.n_tok_tiles > 8 ? 1 : 0;
    a.w_packed = w_packed ? w : nullptr;
    a.err = s.err;
    if (a.mode == kPartial && n_partials) *n_partials = t.splits;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(t.n_feat_tiles * t.n_tok_tiles * t.splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = t.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return bn1 ? cudaLaunchKernelEx(&cfg, gemm_tc_kernel<true>, mw, mx, mx1, a)
               : cudaLaunchKernelEx(&cfg, gemm_tc_kernel<false>, mw, mx, mx1, a);
}

cudaError_t pack_weight_bf16(const bf16 *w, int n_out, int k, bf16 *out, cudaStream_t st) {
    if (k % BK != 0 || k <= 0 || n_out <= 0) return cudaErrorInvalidValue;
    return launch_pdl(pack_weight_kernel, dim3(ceil_div(n_out, BM) * (k / BK)), dim3(256), 0, st, w, n_out, k, out);
}

}  // namespace orca
