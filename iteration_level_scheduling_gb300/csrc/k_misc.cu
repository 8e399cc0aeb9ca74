// Row-wise kernels of one iteration: embedding, LayerNorm, K/V append, argmax.
//
// All act on the flattened [sum L, H] rows of selective batching
// (garden.houmin.site Orca notes, 3.1.2: the token-wise operations do not care
// which request a row belongs to).  Each is HBM-bound: one CTA per row, 16-byte
// vector accesses along the row.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "kernels.cuh"

namespace orca {

namespace {

constexpr int kRowThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kRowThreads) embed_kernel(const int32_t *tokens, const int32_t *row_pos,
                                                            const int32_t *prev_next, int prev_n, const T *tok_emb,
                                                            const T *pos_emb, float *x, int H, int V, int max_pos,
                                                            unsigned *err) {
    constexpr int VEC = Elem<T>::kPer16;
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x;
    int t = tokens[r];
    if (t < 0) {
        int j = -1 - t;
        if (j >= prev_n) {
            if (threadIdx.x == 0) raise_err(err, ERR_BAD_TOKEN);
            t = 0;
        } else {
            t = prev_next[j];
        }
    }
    if (t < 0 || t >= V) {
        if (threadIdx.x == 0) raise_err(err, ERR_BAD_TOKEN);
        t = 0;
    }
    int p = row_pos[r];
    if (p < 0 || p >= max_pos) {
        if (threadIdx.x == 0) raise_err(err, ERR_BAD_POS);
        p = 0;
    }
    const T *te = tok_emb + (size_t)t * H;
    const T *pe = pos_emb + (size_t)p * H;
    float *xr = x + (size_t)r * H;
    for (int e = threadIdx.x * VEC; e < H; e += kRowThreads * VEC) {
        float a[VEC], b[VEC];
        load16(te + e, a);
        load16(pe + e, b);
#pragma unroll
        for (int i = 0; i < VEC; i += 4) {
            float s[4] = {a[i] + b[i], a[i + 1] + b[i + 1], a[i + 2] + b[i + 2], a[i + 3] + b[i + 3]};
            store16(xr + e + i, s);
        }
    }
}

template <typename T>
__device__ __forceinline__ void store_vec4(T *p, const float *v);
template <>
__device__ __forceinline__ void store_vec4<float>(float *p, const float *v) {
    store16(p, v);
}
template <>
__device__ __forceinline__ void store_vec4<bf16>(bf16 *p, const float *v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}

// LayerNorm with biased variance, eps 1e-5, statistics in fp32 from registers.
// One CTA of 4 warps per row; every load of the row (and, when completing a
// split-K projection, of its partial rows) is issued before the first use,
// and each reduction is warp shuffles plus one block barrier.
constexpr int kLnThreads = 128;
constexpr int kLnMaxH = 8192;
constexpr int kLnChunks = kLnMaxH / (4 * kLnThreads);  // float4 per thread

__device__ __forceinline__ float ln_block_sum(float v, float *red, int slot) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[slot * 4 + (threadIdx.x >> 5)] = v;
    __syncthreads();
    return red[slot * 4 + 0] + red[slot * 4 + 1] + red[slot * 4 + 2] + red[slot * 4 + 3];  // fixed order
}

template <typename T>
__global__ void __launch_bounds__(kLnThreads) layernorm_kernel(float *x, const int32_t *row_map, const float *g,
                                                               const float *b, T *y, float *y32, int H,
                                                               const float *part, int n_part, int part_rows,
                                                               const float *add_bias) {
    __shared__ float red[8];
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x;
    const int src = row_map ? row_map[r] : r;
    float *xr = x + (size_t)src * H;
    const int nc = H / 4;  // float4 chunks of the row; thread t handles chunks t, t + 128, ...
    float4 v[kLnChunks];
#pragma unroll
    for (int i = 0; i < kLnChunks; ++i)
        if (i * kLnThreads + (int)threadIdx.x < nc)
            v[i] = *reinterpret_cast<const float4 *>(xr + (i * kLnThreads + threadIdx.x) * 4);
    if (n_part > 0) {
        // complete the residual row: x + (bias + the split-K partials, in split order)
#pragma unroll
        for (int i = 0; i < kLnChunks; ++i) {
            const int c = i * kLnThreads + threadIdx.x;
            if (c >= nc) break;
            float4 acc = add_bias ? *reinterpret_cast<const float4 *>(add_bias + 4 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
            float4 pv[8];
#pragma unroll
            for (int sp = 0; sp < 8; ++sp)
                if (sp < n_part) pv[sp] = *reinterpret_cast<const float4 *>(part + ((size_t)sp * part_rows + src) * H + 4 * c);
#pragma unroll
            for (int sp = 0; sp < 8; ++sp)
                if (sp < n_part) acc.x += pv[sp].x, acc.y += pv[sp].y, acc.z += pv[sp].z, acc.w += pv[sp].w;
            v[i].x += acc.x, v[i].y += acc.y, v[i].z += acc.z, v[i].w += acc.w;
            *reinterpret_cast<float4 *>(xr + 4 * c) = v[i];
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kLnChunks; ++i)
        if (i * kLnThreads + (int)threadIdx.x < nc) s += v[i].x + v[i].y + v[i].z + v[i].w;
    const float mean = ln_block_sum(s, red, 0) / (float)H;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kLnChunks; ++i)
        if (i * kLnThreads + (int)threadIdx.x < nc) {
            const float a0 = v[i].x - mean, a1 = v[i].y - mean, a2 = v[i].z - mean, a3 = v[i].w - mean;
            ss += a0 * a0 + a1 * a1 + a2 * a2 + a3 * a3;
        }
    const float rstd = rsqrtf(ln_block_sum(ss, red, 1) / (float)H + 1e-5f);
#pragma unroll
    for (int i = 0; i < kLnChunks; ++i) {
        const int c = i * kLnThreads + threadIdx.x;
        if (c >= nc) break;
        const float4 gg = *reinterpret_cast<const float4 *>(g + 4 * c);
        const float4 bb = *reinterpret_cast<const float4 *>(b + 4 * c);
        float o[4] = {(v[i].x - mean) * rstd * gg.x + bb.x, (v[i].y - mean) * rstd * gg.y + bb.y,
                      (v[i].z - mean) * rstd * gg.z + bb.z, (v[i].w - mean) * rstd * gg.w + bb.w};
        store_vec4<T>(y + (size_t)r * H + 4 * c, o);
        if (y32) store16(y32 + (size_t)r * H + 4 * c, o);
    }
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads) kv_append_kernel(const T *qkv, const int32_t *row_slot,
                                                                T *pool_layer, int64_t kv_slots, int H, int d,
                                                                int n_heads) {
    constexpr int VEC = Elem<T>::kPer16;
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x;
    const int64_t slot = row_slot[r];
    const T *src = qkv + (size_t)r * 3 * H + H;  // k then v, 2H contiguous values
    for (int e = threadIdx.x * VEC; e < 2 * H; e += kRowThreads * VEC) {
        const int which = e >= H;
        const int c = e - which * H;
        const int h = c / d, dd = c - h * d;
        T *dst = pool_layer + (((int64_t)(which * n_heads + h) * kv_slots + slot) * d + dd);
        *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src + e);
    }
}

constexpr int kArgmaxThreads = 512;

__global__ void __launch_bounds__(kArgmaxThreads) argmax_kernel(const float *logits, int V, int32_t *next,
                                                                int32_t *out2) {
    __shared__ float sv[kArgmaxThreads / 32];
    __shared__ int si[kArgmaxThreads / 32];
    pdl_trigger();
    pdl_wait();
    const float *lr = logits + (size_t)blockIdx.x * V;
    float best = -FLT_MAX;
    int idx = INT_MAX;
    for (int j = threadIdx.x; j < V; j += kArgmaxThreads) {
        float v = lr[j];
        if (v > best || idx == INT_MAX) best = v, idx = j;  // ascending j: first occurrence wins
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, best, o);
        int oi = __shfl_xor_sync(0xffffffffu, idx, o);
        if (ov > best || (ov == best && oi < idx)) best = ov, idx = oi;
    }
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) sv[w] = best, si[w] = idx;
    __syncthreads();
    if (w == 0) {
        best = l < kArgmaxThreads / 32 ? sv[l] : -FLT_MAX;
        idx = l < kArgmaxThreads / 32 ? si[l] : INT_MAX;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, best, o);
            int oi = __shfl_xor_sync(0xffffffffu, idx, o);
            if (ov > best || (ov == best && oi < idx)) best = ov, idx = oi;
        }
        if (l == 0) {
            next[blockIdx.x] = idx;
            if (out2) out2[blockIdx.x] = idx;
        }
    }
}

}  // namespace

template <typename T>
cudaError_t embed(const int32_t *tokens, const int32_t *row_pos, const int32_t *prev_next, int prev_n,
                  const T *tok_emb, const T *pos_emb, float *x, int n_rows, int H, int V, int max_pos,
                  unsigned *err, cudaStream_t st) {
    if (n_rows <= 0) return cudaSuccess;
    return launch_pdl(embed_kernel<T>, dim3(n_rows), dim3(kRowThreads), 0, st, tokens, row_pos, prev_next, prev_n,
                      tok_emb, pos_emb, x, H, V, max_pos, err);
}

template <typename T>
cudaError_t layernorm(float *x, const int32_t *row_map, const float *g, const float *b, T *y, float *y32, int n_rows,
                      int H, cudaStream_t st, const float *part, int n_part, int part_rows, const float *add_bias) {
    if (n_rows <= 0) return cudaSuccess;
    if (H % 4 != 0 || H > kLnMaxH || n_part > 8) return cudaErrorInvalidValue;
    return launch_pdl(layernorm_kernel<T>, dim3(n_rows), dim3(kLnThreads), 0, st, x, row_map, g, b, y, y32, H, part,
                      n_part, part_rows, add_bias);
}

template <typename T>
cudaError_t kv_append(const T *qkv, const int32_t *row_slot, T *pool_layer, int64_t kv_slots, int n_rows, int H,
                      int n_heads, cudaStream_t st) {
    if (n_rows <= 0) return cudaSuccess;
    return launch_pdl(kv_append_kernel<T>, dim3(n_rows), dim3(kRowThreads), 0, st, qkv, row_slot, pool_layer, kv_slots,
                      H, H / n_heads, n_heads);
}

cudaError_t argmax_rows(const float *logits, int n_rows, int V, int32_t *next, int32_t *out2, cudaStream_t st) {
    if (n_rows <= 0) return cudaSuccess;
    return launch_pdl(argmax_kernel, dim3(n_rows), dim3(kArgmaxThreads), 0, st, logits, V, next, out2);
}

template cudaError_t embed<float>(const int32_t *, const int32_t *, const int32_t *, int, const float *,
                                  const float *, float *, int, int, int, int, unsigned *, cudaStream_t);
template cudaError_t embed<bf16>(const int32_t *, const int32_t *, const int32_t *, int, const bf16 *, const bf16 *,
                                 float *, int, int, int, int, unsigned *, cudaStream_t);
template cudaError_t layernorm<float>(float *, const int32_t *, const float *, const float *, float *, float *, int,
                                      int, cudaStream_t, const float *, int, int, const float *);
template cudaError_t layernorm<bf16>(float *, const int32_t *, const float *, const float *, bf16 *, float *, int, int,
                                     cudaStream_t, const float *, int, int, const float *);
template cudaError_t kv_append<float>(const float *, const int32_t *, float *, int64_t, int, int, int, cudaStream_t);
template cudaError_t kv_append<bf16>(const bf16 *, const int32_t *, bf16 *, int64_t, int, int, int, cudaStream_t);

}  // namespace orca
