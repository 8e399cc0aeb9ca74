// Host-side launchers of the device kernels (internal to liborca).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace orca {

using bf16 = __nv_bfloat16;

// Epilogue of a linear layer y[t, f] = sum_k x[t, k] w[f, k]:
//   y += bias[f]; y = GeLU(y) if gelu;
//   resid ? out_f32[t, f] = resid[t, f] + y : (out_f32 ? out_f32 : out_bf16)[t, f] = y.
struct Epilogue {
    const float *bias = nullptr;
    int gelu = 0;
    const float *resid = nullptr;
    float *out_f32 = nullptr;
    bf16 *out_bf16 = nullptr;
    int ld_out = 0;
    // Optional split-K partial output: when set and K is split, each split
    // writes its fp32 partial product (no bias / GeLU / residual) to slab s of
    // part ([s][m_tok][n_out]) and the caller reduces them.
    float *part = nullptr;
    size_t part_cap = 0;  // floats available at part
    // Optional K/V append (bf16 QKV projection): output features >= kv_h are
    // k (then v) rows, written to the pool layer at the row's slot instead of
    // to out_bf16.  Pool layout [K|V][head][slot][kv_hd].
    bf16 *kv_pool = nullptr;
    const int32_t *row_slot = nullptr;
    int64_t kv_slots = 0;
    int kv_h = 0, kv_hd = 0, kv_nh = 0;
};

// Launch context of the tensor-core GEMM: the device error word, the SM
// count and the stream-K workspace (partial tiles of cut tiles and one
// arrival counter per tile, zero between launches).  Without a workspace the
// stream-K kernel is never chosen.
struct GemmScratch {
    unsigned *err = nullptr;
    int num_sms = 148;
    float *sk_part = nullptr;
    size_t sk_part_floats = 0;
    int *sk_cnt = nullptr;
    int sk_cnt_n = 0;
};

// tcgen05 GEMM, bf16 operands, fp32 accumulation in tensor memory.
// x: [x_rows_cap, k] row-major (rows >= m_tok are never stored), w: [n_out, k].
// Returns in *n_partials the number of partial slabs written (0: the full
// epilogue was applied).
// w_packed: w is in the layout written by pack_weight_bf16.
cudaError_t gemm_tc_bf16(const bf16 *x, int x_rows_cap, const bf16 *w, bool w_packed, int m_tok, int n_out, int k,
                         const Epilogue &e, const GemmScratch &s, cudaStream_t st, int *n_partials = nullptr);
// Tile-contiguous, pre-swizzled copy of a [n_out, k] bf16 weight (k % 64 == 0).
size_t packed_weight_elems(int n_out, int k);
cudaError_t pack_weight_bf16(const bf16 *w, int n_out, int k, bf16 *out, cudaStream_t st);
// Shape the tcgen05 GEMM would use (for scratch sizing and accounting).
struct TcShape {
    int bn, n_tok_tiles, n_feat_tiles, splits, kb_per_split, stages, tmem_cols;
    size_t smem;
};
TcShape gemm_tc_shape(int m_tok, int n_out, int k, const GemmScratch &s, bool allow_partial = false,
                      size_t part_cap = 0);
// Stream-K launch shape: token tiles of bn <= 256 rows, the units
// (tile, 64-wide K block) cut into `grid` ranges of `chunk` units.
struct SkShape {
    int bn, n_tok_tiles, n_feat_tiles, tiles, num_kb, units, chunk, grid, stages, tmem_cols;
    size_t smem, part_floats;
};
SkShape gemm_sk_shape(int m_tok, int n_out, int k, int num_sms);
// Whether gemm_tc_bf16 takes the stream-K kernel for this shape.
bool gemm_uses_sk(int m_tok, int n_out, int k, const GemmScratch &s);
// Workspace the stream-K kernel needs at most for up to max_rows token rows
// and outputs of up to max_n features.
size_t gemm_sk_part_floats(int num_sms);
int gemm_sk_counters(int max_rows, int max_n);


// cuTensorMapEncodeTiled, reached through the runtime's driver entry point;
// dims/strides/box innermost first (strides in bytes, rank - 1 of them).
bool encode_tensor_map(CUtensorMap *m, CUtensorMapDataType dt, uint32_t rank, const void *base, const uint64_t *dims,
                       const uint64_t *strides, const uint32_t *box, CUtensorMapSwizzle swizzle);

// SIMT FFMA GEMM, fp32 operands.
cudaError_t gemm_simt_f32(const float *x, const float *w, int m_tok, int n_out, int k, const Epilogue &e,
                          cudaStream_t st);

// x[r] = tok_emb[tok(r)] + pos_emb[row_pos[r]] (fp32 out).  tok(r) = tokens[r]
// if >= 0, else prev_next[-1 - tokens[r]].
template <typename T>
cudaError_t embed(const int32_t *tokens, const int32_t *row_pos, const int32_t *prev_next, int prev_n,
                  const T *tok_emb, const T *pos_emb, float *x, int n_rows, int H, int V, int max_pos,
                  unsigned *err, cudaStream_t st);

// y[r] = LN(x[src(r)]) with src(r) = row_map ? row_map[r] : r; optional fp32 copy.
// With n_part > 0 the row is first completed from the split-K partials of the
// preceding projection: x[src] += add_bias + sum_s part[s][src] (written back
// to x), part slabs having part_rows rows of H floats.
template <typename T>
cudaError_t layernorm(float *x, const int32_t *row_map, const float *g, const float *b, T *y, float *y32, int n_rows,
                      int H, cudaStream_t st, const float *part = nullptr, int n_part = 0, int part_rows = 0,
                      const float *add_bias = nullptr);

// Copy this iteration's k, v rows (columns H..3H of qkv) into the pool layer.
template <typename T>
cudaError_t kv_append(const T *qkv, const int32_t *row_slot, T *pool_layer, int64_t kv_slots, int n_rows, int H,
                      int n_heads, cudaStream_t st);

struct AttnPlan {
    const int32_t *req_off, *req_ctx, *req_kvoff;
    // keys each decode request's work items cover: ctx + 1, or in a padded
    // batch the batch's longest (keys past ctx + 1 are loaded and masked); null = ctx + 1
    const int32_t *req_keys;
    const int32_t *dec_work, *dec_wbegin, *dec_nch;  // decode split-K work items
    const int32_t *dec_order;                        // work items, longest first
    // per entry of dec_order, 8 words (16-byte aligned): kv_offset + first key,
    // keys, first row, request, chunk, the request's chunks, its first work item, first key
    const int32_t *dec_items;
    const int32_t *pre_tiles;                        // prefill (request, first row) tiles
    int n_dec_work, n_pre_tiles, chunk;
    int n_rows;  // rows of the qkv matrix (bounds the tcgen05 prefill's q loads; 0: that kernel is not used)
    // two ints, zero between launches: the tensor-core decode kernel claims work
    // items from [0] at run time, counting finished CTAs in [1] (null: every
    // CTA takes a fixed share)
    int *claim;
};

// Attention for one layer.  Decode: requests with one input row, split-K over
// their cached keys.  Prefill: requests with several rows, causal.
template <typename T>
cudaError_t attention(const T *qkv, const T *pool_layer, int64_t kv_slots, T *out, const AttnPlan &p, int H,
                      int n_heads, float *part, int *counters, unsigned *err, cudaStream_t st, bool decode,
                      bool prefill);

// Order of the decode work items (request, chunk) by number of keys, longest
// first (stable), for the persistent decode kernel's load balance.
// req_keys[i]: the keys request i's items cover (AttnPlan::req_keys).
void decode_order(const int32_t *dec_work, int n_work, const int32_t *req_keys, int chunk, int32_t *order);
// Whether the engine gives the decode kernel its work-claim counters
// (AttnPlan::claim); ORCA_ATTN_DECODE_CLAIM=-1 turns that off.
bool decode_claim_enabled();
// Order the prefill tiles ((request, first row) pairs, kPrefillRowsPerTile
// rows each) by the keys their rows see, most first (stable): the persistent
// prefill kernel walks them in this order, longest first.
void prefill_order(int32_t *pre_tiles, int n_tiles, const int32_t *req_off, const int32_t *req_ctx);
// The 8-word records of AttnPlan::dec_items, in the order of `order`.
void decode_items(const int32_t *order, const int32_t *dec_work, int n_work, const int32_t *req_off,
                  const int32_t *req_keys, const int32_t *req_kvoff, const int32_t *dec_wbegin, const int32_t *dec_nch,
                  int chunk, int32_t *items);

// next[b] = argmax_j logits[b, j] (lowest j on ties); also to out2 if non-null.
cudaError_t argmax_rows(const float *logits, int n_rows, int V, int32_t *next, int32_t *out2, cudaStream_t st);

constexpr int kPrefillRowsPerTile = 128;  // query rows per prefill tile (the tcgen05 kernel's M)

// A bounded wait that nothing satisfies, given up after limit_ns (failure-
// detection tests of the device error word).
cudaError_t expire_wait(unsigned long long limit_ns, unsigned *err, cudaStream_t st);

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device.  The attribute belongs to the device that was current when it was
// set, so it is set once per (device, kernel): an engine or an
// allocation-free call on another GPU sets its own.
cudaError_t max_smem_once(const void *kernel, int bytes);

// Launch with programmatic stream serialization (the kernel calls pdl_wait()).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace orca
