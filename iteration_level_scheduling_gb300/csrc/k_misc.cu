// Row-wise kernels of one iteration: embedding, LayerNorm, K/V append, argmax.
//
// All act on the flattened [sum L, H] rows of selective batching
// (garden.houmin.site Orca notes, 3.1.2: the token-wise operations do not care
// which request a row belongs to).  Each is HBM-bound: one CTA per row, 16-byte
// vector accesses along the row.
#include <cfloat>
#include <climits>
#include <mutex>
#include <set>
#include <utility>

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

constexpr int kLnThreads = 512;
constexpr int kLnMaxVec = 4;  // H <= kLnThreads * 4 * kLnMaxVec = 8192
// the many-rows shape (layernorm_rows_kernel): 256 threads, three CTAs per SM
constexpr int kLnRowsThreads = 256, kLnRowsVec = 8, kLnRowsCtas = 3;
constexpr int kLnRowsFrom = 256;  // rows from which it runs

__device__ __forceinline__ float block_sum(float v, float *red) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    if (w == 0) {
        t = (l < (int)(blockDim.x >> 5)) ? red[l] : 0.f;
        t = warp_sum(t);
        if (l == 0) red[32] = t;
    }
    __syncthreads();
    t = red[32];
    __syncthreads();
    return t;
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

// LayerNorm with biased variance, eps 1e-5, statistics in fp32 from registers
// (two passes over the row held in registers).
template <typename T>
__global__ void __launch_bounds__(kLnThreads) layernorm_kernel(float *x, const int32_t *row_map, const float *g,
                                                               const float *b, T *y, float *y32, int H,
                                                               const float *part, int n_part, int part_rows,
                                                               const float *add_bias) {
    __shared__ float red[33];
    pdl_trigger();
    // gamma, beta and the completed projection's bias are weights: pulled into
    // L1 before waiting for the previous kernel, so their loads after the
    // reductions do not add a memory round trip
#pragma unroll
    for (int i = 0; i < kLnMaxVec; ++i) {
        const int e = (threadIdx.x + i * kLnThreads) * 4;
        if (e < H) {
            prefetch_l1(g + e);
            prefetch_l1(b + e);
            if (n_part > 0 && add_bias) prefetch_l1(add_bias + e);
        }
    }
    pdl_wait();
    const int r = blockIdx.x;
    const int src = row_map ? row_map[r] : r;
    float *xr = x + (size_t)src * H;
    // every load of the row (and of its split-K partials and bias) is issued
    // before the first use
    constexpr int kInline = 3;  // partial slabs loaded up front (13B shapes split K at most 3 ways; more: second pass)
    float4 q[kLnMaxVec], bias[kLnMaxVec], pv[kLnMaxVec][kInline];
#pragma unroll
    for (int i = 0; i < kLnMaxVec; ++i) {
        const int e = (threadIdx.x + i * kLnThreads) * 4;
        if (e < H) {
            q[i] = *reinterpret_cast<const float4 *>(xr + e);
            if (n_part > 0) {
                bias[i] = add_bias ? *reinterpret_cast<const float4 *>(add_bias + e) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int sp = 0; sp < kInline; ++sp)
                    if (sp < n_part)
                        pv[i][sp] = *reinterpret_cast<const float4 *>(part + ((size_t)sp * part_rows + src) * H + e);
            }
        }
    }
    float v[kLnMaxVec][4];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kLnMaxVec; ++i) {
        const int e = (threadIdx.x + i * kLnThreads) * 4;
        if (e < H) {
            if (n_part > 0) {
                // complete the residual row: x + (bias + the split-K partials, in split order)
                float4 acc = bias[i];
#pragma unroll
                for (int sp = 0; sp < kInline; ++sp)
                    if (sp < n_part) acc.x += pv[i][sp].x, acc.y += pv[i][sp].y, acc.z += pv[i][sp].z, acc.w += pv[i][sp].w;
                for (int sp = kInline; sp < n_part; ++sp) {
                    const float4 p = *reinterpret_cast<const float4 *>(part + ((size_t)sp * part_rows + src) * H + e);
                    acc.x += p.x, acc.y += p.y, acc.z += p.z, acc.w += p.w;
                }
                q[i].x += acc.x, q[i].y += acc.y, q[i].z += acc.z, q[i].w += acc.w;
                *reinterpret_cast<float4 *>(xr + e) = q[i];
            }
            v[i][0] = q[i].x, v[i][1] = q[i].y, v[i][2] = q[i].z, v[i][3] = q[i].w;
            s += q[i].x + q[i].y + q[i].z + q[i].w;
        }
    }
    const float mean = block_sum(s, red) / (float)H;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kLnMaxVec; ++i) {
        int e = (threadIdx.x + i * kLnThreads) * 4;
        if (e < H) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float d = v[i][j] - mean;
                ss += d * d;
            }
        }
    }
    const float var = block_sum(ss, red) / (float)H;
    const float rstd = rsqrtf(var + 1e-5f);
#pragma unroll
    for (int i = 0; i < kLnMaxVec; ++i) {
        int e = (threadIdx.x + i * kLnThreads) * 4;
        if (e < H) {
            float4 gg = *reinterpret_cast<const float4 *>(g + e);
            float4 bb = *reinterpret_cast<const float4 *>(b + e);
            float o[4] = {(v[i][0] - mean) * rstd * gg.x + bb.x, (v[i][1] - mean) * rstd * gg.y + bb.y,
                          (v[i][2] - mean) * rstd * gg.z + bb.z, (v[i][3] - mean) * rstd * gg.w + bb.w};
            store_vec4<T>(y + (size_t)r * H + e, o);
            if (y32) store16(y32 + (size_t)r * H + e, o);
        }
    }
}

// The same LayerNorm (and split-K completion, the partials summed in the same
// order; the row statistics sum in a different fixed order) for launches of
// hundreds of rows and more: the
// 512-thread kernel above fills an SM's registers with one row, so only one
// row per SM is in flight (13B, 25777 rows: 382 us per launch, 0.3 of HBM).
// Here 256 threads take a row and hold only the completed row (8 float4 at
// most), so three CTAs share an SM.
template <typename T>
__global__ void __launch_bounds__(kLnRowsThreads, kLnRowsCtas)
    layernorm_rows_kernel(float *x, const int32_t *row_map, const float *g, const float *b, T *y, float *y32, int H,
                          const float *part, int n_part, int part_rows, const float *add_bias) {
    __shared__ float red[33];
    pdl_trigger();
#pragma unroll
    for (int i = 0; i < kLnRowsVec; ++i) {
        const int e = (threadIdx.x + i * kLnRowsThreads) * 4;
        if (e < H) {
            prefetch_l1(g + e);
            prefetch_l1(b + e);
        }
    }
    pdl_wait();
    const int r = blockIdx.x;
    const int src = row_map ? row_map[r] : r;
    float *xr = x + (size_t)src * H;
    float4 q[kLnRowsVec];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kLnRowsVec; ++i) {
        const int e = (threadIdx.x + i * kLnRowsThreads) * 4;
        q[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < H) {
            q[i] = *reinterpret_cast<const float4 *>(xr + e);
            if (n_part > 0) {
                // complete the residual row: x + (bias + the split-K partials, in split order)
                float4 acc = add_bias ? *reinterpret_cast<const float4 *>(add_bias + e) : make_float4(0.f, 0.f, 0.f, 0.f);
                for (int sp = 0; sp < n_part; ++sp) {
                    const float4 p = *reinterpret_cast<const float4 *>(part + ((size_t)sp * part_rows + src) * H + e);
                    acc.x += p.x, acc.y += p.y, acc.z += p.z, acc.w += p.w;
                }
                q[i].x += acc.x, q[i].y += acc.y, q[i].z += acc.z, q[i].w += acc.w;
                *reinterpret_cast<float4 *>(xr + e) = q[i];
            }
            s += q[i].x + q[i].y + q[i].z + q[i].w;
        }
    }
    const float mean = block_sum(s, red) / (float)H;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kLnRowsVec; ++i) {
        const int e = (threadIdx.x + i * kLnRowsThreads) * 4;
        if (e < H) {
            const float d0 = q[i].x - mean, d1 = q[i].y - mean, d2 = q[i].z - mean, d3 = q[i].w - mean;
            ss += d0 * d0 + d1 * d1 + d2 * d2 + d3 * d3;
        }
    }
    const float var = block_sum(ss, red) / (float)H;
    const float rstd = rsqrtf(var + 1e-5f);
#pragma unroll
    for (int i = 0; i < kLnRowsVec; ++i) {
        const int e = (threadIdx.x + i * kLnRowsThreads) * 4;
        if (e < H) {
            const float4 gg = *reinterpret_cast<const float4 *>(g + e);
            const float4 bb = *reinterpret_cast<const float4 *>(b + e);
            float o[4] = {(q[i].x - mean) * rstd * gg.x + bb.x, (q[i].y - mean) * rstd * gg.y + bb.y,
                          (q[i].z - mean) * rstd * gg.z + bb.z, (q[i].w - mean) * rstd * gg.w + bb.w};
            store_vec4<T>(y + (size_t)r * H + e, o);
            if (y32) store16(y32 + (size_t)r * H + e, o);
        }
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
    if (H % 4 != 0 || H > kLnThreads * 4 * kLnMaxVec || n_part > 8) return cudaErrorInvalidValue;
    static_assert(kLnRowsThreads * 4 * kLnRowsVec >= kLnThreads * 4 * kLnMaxVec, "same H limit for both shapes");
    if (n_rows >= kLnRowsFrom)
        return launch_pdl(layernorm_rows_kernel<T>, dim3(n_rows), dim3(kLnRowsThreads), 0, st, x, row_map, g, b, y, y32,
                          H, part, n_part, part_rows, add_bias);
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

namespace {
// One thread waits, bounded, on an mbarrier nothing arrives on: the wait runs
// out after limit_ns and records ERR_WAIT_TIMEOUT, as an expired wait in any
// kernel would.
__global__ void expire_wait_kernel(unsigned long long limit_ns, unsigned *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0u, err, limit_ns);
}
}  // namespace

cudaError_t expire_wait(unsigned long long limit_ns, unsigned *err, cudaStream_t st) {
    expire_wait_kernel<<<1, 32, 0, st>>>(limit_ns, err);
    return cudaGetLastError();
}

cudaError_t max_smem_once(const void *kernel, int bytes) {
    static std::mutex mu;
    static std::set<std::pair<int, const void *>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({dev, kernel})) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.insert({dev, kernel});
    return e;
}

}  // namespace orca
