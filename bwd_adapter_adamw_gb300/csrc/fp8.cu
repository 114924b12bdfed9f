// FP8 (E4M3) frozen base: per-row scaled quantisation of the frozen product's operands and the
// per-row rescaling of the LoRA operands that share its accumulator ("LoRA Training and
// Serving", Quantized rollout: an FP8 base under a bf16-trained adapter; "Backward Bug Hunts and
// Vulkan Tiled GEMM": quantized frozen weights under the LoRA backward).
//
// Quantisation of a row x (all fp32): amax = max |x|, r = 448 / amax, codes = e4m3(x * r)
// rounded to nearest even with saturation to +-448, dequantisation scale s = amax / 448;
// r = s = 1 when amax is 0 or 448 / amax is not finite.
#include <cuda_fp8.h>

#include "lora_kernels.h"

namespace lora {

namespace {

constexpr int kQThreads = 256;
constexpr int kQVec = 8;   // bf16 per 16-byte load

__device__ __forceinline__ void row_scales(float amax, float& rcp, float& scale) {
  rcp = __fdiv_rn(448.f, amax);
  if (amax > 0.f && isfinite(rcp)) {
    scale = __fdiv_rn(amax, 448.f);
  } else {
    rcp = 1.f;
    scale = 1.f;
  }
}

__device__ __forceinline__ uint8_t e4m3(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float block_max(float v, float* sh) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  float m = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, sh[w]);
  return m;
}

// One CTA per row of src [rows, K] bf16 (K % 8 == 0, K <= kQThreads * kQVec * VPT): the row stays
// in registers between the absmax and the encode.
template <int VPT>
__global__ void __launch_bounds__(kQThreads) k_quant_rows(const __nv_bfloat16* __restrict__ src,
                                                          int64_t rows, int64_t K,
                                                          uint8_t* __restrict__ dst,
                                                          float* __restrict__ scale) {
  grid_dep_sync();
  __shared__ float sh[kQThreads / 32];
  const int64_t r = blockIdx.x;
  if (r >= rows) return;
  const __nv_bfloat16* x = src + r * K;
  uint4 v[VPT];
  float amax = 0.f;
#pragma unroll
  for (int u = 0; u < VPT; ++u) {
    const int64_t i = ((int64_t)threadIdx.x + (int64_t)u * kQThreads) * kQVec;
    v[u] = i < K ? *reinterpret_cast<const uint4*>(x + i) : make_uint4(0, 0, 0, 0);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[u]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  amax = block_max(amax, sh);
  float rcp, sc;
  row_scales(amax, rcp, sc);
  if (threadIdx.x == 0) scale[r] = sc;
#pragma unroll
  for (int u = 0; u < VPT; ++u) {
    const int64_t i = ((int64_t)threadIdx.x + (int64_t)u * kQThreads) * kQVec;
    if (i >= K) continue;
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[u]);
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      const uint32_t lo = e4m3(__fmul_rn(f.x, rcp)), hi = e4m3(__fmul_rn(f.y, rcp));
      w[e >> 1] |= (lo | (hi << 8)) << ((e & 1) * 16);
    }
    *reinterpret_cast<uint2*>(dst + r * K + i) = make_uint2(w[0], w[1]);
  }
}

// Columns of W [rows, cols] bf16 quantised as the rows of W^T: dst [cols, rows] codes, one scale
// per column. CTA = 32 columns; pass 1 takes each column's absmax, pass 2 encodes 32 x 32 tiles
// and writes them transposed through shared memory.
__global__ void __launch_bounds__(256) k_quant_cols(const __nv_bfloat16* __restrict__ W,
                                                    int64_t rows, int64_t cols,
                                                    uint8_t* __restrict__ dst,
                                                    float* __restrict__ scale) {
  grid_dep_sync();
  __shared__ float smax[8][33];
  __shared__ float srcp[32];
  __shared__ uint8_t tile[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t c0 = (int64_t)blockIdx.x * 32;
  const int64_t c = c0 + tx;
  float amax = 0.f;
  if (c < cols)
    for (int64_t r = ty; r < rows; r += 8) amax = fmaxf(amax, fabsf(__bfloat162float(W[r * cols + c])));
  smax[ty][tx] = amax;
  __syncthreads();
  if (ty == 0) {
    float m = 0.f;
    for (int k = 0; k < 8; ++k) m = fmaxf(m, smax[k][tx]);
    float rcp, sc;
    row_scales(m, rcp, sc);
    srcp[tx] = rcp;
    if (c < cols) scale[c] = sc;
  }
  __syncthreads();
  for (int64_t r0 = 0; r0 < rows; r0 += 32) {
    for (int k = ty; k < 32; k += 8) {
      const int64_t r = r0 + k;
      tile[k][tx] = (r < rows && c < cols) ? e4m3(__fmul_rn(__bfloat162float(W[r * cols + c]), srcp[tx]))
                                           : (uint8_t)0;
    }
    __syncthreads();
    for (int k = ty; k < 32; k += 8) {
      const int64_t cc = c0 + k, r = r0 + tx;
      if (cc < cols && r < rows) dst[cc * rows + r] = tile[tx][k];
    }
    __syncthreads();
  }
}

// dst[r, :] = src[r, :] / scale[r] for an fp32 [rows, cols] matrix (row strides lds, ldd).
// Two row divisions in one launch (the LoRA operands of an E4M3 product: Hs or Gs by the token
// scales, B or A^T by the weight's scales); the grid-stride index runs over job 0's elements,
// then job 1's.
__global__ void k_div_rows(const DivRowsJob j0, const DivRowsJob j1) {
  grid_dep_sync();
  const int64_t n0 = j0.rows * j0.cols, n = n0 + j1.rows * j1.cols;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const bool second = e >= n0;
    const int64_t ee = second ? e - n0 : e;
    const int64_t cols = second ? j1.cols : j0.cols;
    const int64_t r = ee / cols, c = ee - r * cols;
    const float* src = second ? j1.src : j0.src;
    const float* scale = second ? j1.scale : j0.scale;
    float* dst = second ? j1.dst : j0.dst;
    const int64_t lds = second ? j1.lds : j0.lds, ldd = second ? j1.ldd : j0.ldd;
    dst[r * ldd + c] = __fdiv_rn(src[r * lds + c], scale[r]);
  }
}

}  // namespace

cudaError_t launch_quant_rows_e4m3(const void* src, int64_t rows, int64_t K, uint8_t* dst,
                                   float* scale, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (K % kQVec) return cudaErrorInvalidValue;
  const int64_t vpt = (K / kQVec + kQThreads - 1) / kQThreads;
  prof_begin(0, st);
  const __nv_bfloat16* s = static_cast<const __nv_bfloat16*>(src);
  const unsigned g = (unsigned)rows;
  if (vpt <= 2) launch_kernel(k_quant_rows<2>, g, kQThreads, 0, st, s, rows, K, dst, scale);
  else if (vpt <= 4) launch_kernel(k_quant_rows<4>, g, kQThreads, 0, st, s, rows, K, dst, scale);
  else if (vpt <= 8) launch_kernel(k_quant_rows<8>, g, kQThreads, 0, st, s, rows, K, dst, scale);
  else return cudaErrorInvalidValue;   // K > 16384
  return cudaGetLastError();
}

cudaError_t launch_quant_cols_e4m3(const void* W, int64_t rows, int64_t cols, uint8_t* dst,
                                   float* scale, cudaStream_t st) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  prof_begin(0, st);
  launch_kernel(k_quant_cols, (unsigned)((cols + 31) / 32), 256, 0, st,
                static_cast<const __nv_bfloat16*>(W), rows, cols, dst, scale);
  return cudaGetLastError();
}

cudaError_t launch_div_rows2(const DivRowsJob& a, const DivRowsJob& b, cudaStream_t st) {
  const int64_t n = (a.rows > 0 && a.cols > 0 ? a.rows * a.cols : 0) +
                    (b.rows > 0 && b.cols > 0 ? b.rows * b.cols : 0);
  if (n <= 0) return cudaSuccess;
  DivRowsJob j0 = a, j1 = b;
  if (j0.rows <= 0 || j0.cols <= 0) { j0.rows = 0; j0.cols = 1; }
  if (j1.rows <= 0 || j1.cols <= 0) { j1.rows = 0; j1.cols = 1; }
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  prof_begin(0, st);
  launch_kernel(k_div_rows, (unsigned)blocks, 256, 0, st, j0, j1);
  return cudaGetLastError();
}

}  // namespace lora
