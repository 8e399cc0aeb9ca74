// Flattened linear layers in fp32 on the CUDA cores (FFMA, no TF32), for the
// fp32 model.  Same contract as the tensor-core kernel: y[t, f] =
// sum_k x[t, k] w[f, k] over the [sum L, H] rows of the batch, followed by the
// fused epilogue (bias, exact GeLU, residual).  64 x 64 output tile per CTA,
// 16 x 16 threads with a 4 x 4 register block each, K staged through shared
// memory 16 at a time.
#include "common.cuh"
#include "kernels.cuh"

namespace orca {

namespace {

constexpr int TB = 64, TK = 16;

__global__ void __launch_bounds__(256) gemm_simt_f32_kernel(const float *x, const float *w, int M, int N, int K,
                                                            Epilogue e) {
    __shared__ float xs[TK][TB + 1];
    __shared__ float ws[TK][TB + 1];
    pdl_trigger();
    pdl_wait();
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int t0 = blockIdx.y * TB, f0 = blockIdx.x * TB;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += TK) {
        for (int idx = threadIdx.x; idx < TB * TK; idx += 256) {
            const int r = idx / TK, c = idx % TK;
            const int t = t0 + r, f = f0 + r, k = k0 + c;
            xs[c][r] = (t < M && k < K) ? x[(size_t)t * K + k] : 0.f;
            ws[c][r] = (f < N && k < K) ? w[(size_t)f * K + k] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int c = 0; c < TK; ++c) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = xs[c][ty * 4 + i], b[i] = ws[c][tx * 4 + i];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty * 4 + i;
        if (t >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int f = f0 + tx * 4 + j;
            if (f >= N) continue;
            float y = acc[i][j];
            if (e.bias) y += e.bias[f];
            if (e.gelu) y = gelu_erf(y);
            const size_t o = (size_t)t * e.ld_out + f;
            if (e.resid)
                e.out_f32[o] = e.resid[o] + y;
            else
                e.out_f32[o] = y;
        }
    }
}

}  // namespace

cudaError_t gemm_simt_f32(const float *x, const float *w, int m_tok, int n_out, int k, const Epilogue &e,
                          cudaStream_t st) {
    if (m_tok <= 0) return cudaSuccess;
    if (!e.out_f32) return cudaErrorInvalidValue;
    dim3 grid((n_out + TB - 1) / TB, (m_tok + TB - 1) / TB);
    return launch_pdl(gemm_simt_f32_kernel, grid, dim3(256), 0, st, x, w, m_tok, n_out, k, e);
}

}  // namespace orca
