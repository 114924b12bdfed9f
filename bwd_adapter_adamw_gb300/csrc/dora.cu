// DoRA row norm and magnitude gradient ("8. LoRA Fundamentals", How it works: canonical DoRA
// y = (magnitude / ||W + Delta||) * (W x + Delta x) with the row norm detached from gradients).
#include "lora_kernels.h"

namespace lora {

namespace {

// n_o = || W_o + s (B A)_o ||_2. One CTA per 4 output rows; B's rows sit in shared memory and
// every thread walks a strided set of input columns, forming the merged weight on the fly.
// Squares are summed in fp32 per thread and combined across threads in double.
template <typename T>
__global__ void __launch_bounds__(256) k_dora_norm(const T* __restrict__ W, const float* __restrict__ A,
                                                   const float* __restrict__ B, float s,
                                                   int64_t out_dim, int64_t in_dim, int32_t rank,
                                                   float* __restrict__ norm_out) {
  constexpr int R = 4;
  __shared__ float sb[R][LORA_MAX_RANK];
  __shared__ double red[R][8];
  const int64_t o0 = (int64_t)blockIdx.x * R;
  for (int e = threadIdx.x; e < R * rank; e += blockDim.x) {
    const int r = e / rank, j = e % rank;
    sb[r][j] = (o0 + r < out_dim) ? B[(o0 + r) * rank + j] : 0.f;
  }
  __syncthreads();
  float acc[R] = {0.f, 0.f, 0.f, 0.f};
  for (int64_t i = threadIdx.x; i < in_dim; i += blockDim.x) {
    float d[R] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < rank; ++j) {
      const float a = __ldg(A + (int64_t)j * in_dim + i);
#pragma unroll
      for (int r = 0; r < R; ++r) d[r] = fmaf(sb[r][j], a, d[r]);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (o0 + r < out_dim) {
        const float w = to_f(W[(o0 + r) * in_dim + i]);
        const float merged = fmaf(s, d[r], w);
        acc[r] = fmaf(merged, merged, acc[r]);
      }
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    double v = (double)acc[r];
    for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(0xffffffffu, v, off);
    if (lane == 0) red[r][warp] = v;
  }
  __syncthreads();
  if (threadIdx.x < R) {
    const int r = threadIdx.x;
    double v = 0.0;
    for (int w = 0; w < 8; ++w) v += red[r][w];
    if (o0 + r < out_dim) norm_out[o0 + r] = (float)sqrt(v);
  }
}

// dm_o += (sum_t dY[t, o] * Y[t, o]) / m_o  (= sum_t dY * Z / n with Y = (m / n) Z).
template <typename T>
__global__ void k_dora_dm(const T* __restrict__ dY, const T* __restrict__ Y,
                          const float* __restrict__ mag, int64_t Tn, int64_t out_dim,
                          float* __restrict__ dm) {
  const int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (o >= out_dim) return;
  float acc = 0.f;
  for (int64_t t = 0; t < Tn; ++t) acc = fmaf(to_f(dY[t * out_dim + o]), to_f(Y[t * out_dim + o]), acc);
  dm[o] += acc / mag[o];
}

}  // namespace

cudaError_t launch_dora_norm(int dtype, const void* W, const float* A, const float* B, float s,
                             int64_t out_dim, int64_t in_dim, int32_t rank, float* norm_out,
                             cudaStream_t st) {
  const unsigned blocks = (unsigned)((out_dim + 3) / 4);
  if (dtype == LORA_F32)
    { prof_begin(0, st); k_dora_norm<float><<<blocks, 256, 0, st>>>((const float*)W, A, B, s, out_dim, in_dim, rank, norm_out); }
  else
    { prof_begin(0, st); k_dora_norm<__nv_bfloat16><<<blocks, 256, 0, st>>>((const __nv_bfloat16*)W, A, B, s, out_dim,
                                                       in_dim, rank, norm_out); }
  return cudaGetLastError();
}

cudaError_t launch_dora_dm(int dtype, const void* dY, const void* Y, const float* mag, int64_t T,
                           int64_t out_dim, float* dm, cudaStream_t st) {
  const unsigned blocks = (unsigned)((out_dim + 127) / 128);
  if (dtype == LORA_F32)
    { prof_begin(0, st); k_dora_dm<float><<<blocks, 128, 0, st>>>((const float*)dY, (const float*)Y, mag, T, out_dim, dm); }
  else
    { prof_begin(0, st); k_dora_dm<__nv_bfloat16><<<blocks, 128, 0, st>>>((const __nv_bfloat16*)dY,
                                                     (const __nv_bfloat16*)Y, mag, T, out_dim, dm); }
  return cudaGetLastError();
}

}  // namespace lora
