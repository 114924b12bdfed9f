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
  grid_dep_sync();
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

// ---------------------------------------------------------------------------------------------
// Row norm from the expanded identity (bf16 W): with H = W A^T [out, r] (tensor cores, the
// shrink kernel applied to W's rows) and the Gram matrix C = A A^T [r, r],
//   ||W_o + s (B A)_o||^2 = ||W_o||^2 + 2 s sum_j H[o, j] B[o, j] + s^2 B_o C B_o^T.
// ---------------------------------------------------------------------------------------------

// C[j, k] for k in [8 blockIdx.y, 8 blockIdx.y + 8): 256 threads stride over the input columns.
__global__ void __launch_bounds__(256) k_dora_gram(const float* __restrict__ A, int64_t in_dim,
                                                   int32_t rank, float* __restrict__ C) {
  grid_dep_sync();
  __shared__ float red[8][8];
  const int j = blockIdx.x, k0 = blockIdx.y * 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  // four strides of the input columns per pass, every load issued before the FMAs
  for (int64_t i0 = threadIdx.x; i0 < in_dim; i0 += 4 * 256) {
    float a[4], b[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + (int64_t)u * 256;
      const bool ok = i < in_dim;
      a[u] = ok ? __ldg(A + (int64_t)j * in_dim + i) : 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        b[u][kk] = (ok && k0 + kk < rank) ? __ldg(A + (int64_t)(k0 + kk) * in_dim + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (i0 + (int64_t)u * 256 >= in_dim) continue;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        if (k0 + kk < rank) acc[kk] = fmaf(a[u], b[u][kk], acc[kk]);
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    float v = acc[kk];
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) red[warp][kk] = v;
  }
  __syncthreads();
  if (threadIdx.x < 8 && k0 + threadIdx.x < rank) {
    float v = 0.f;
    for (int w = 0; w < 8; ++w) v += red[w][threadIdx.x];
    C[j * rank + k0 + threadIdx.x] = v;
  }
}

// One warp per output row: ||W_o||^2 from 16-byte loads of the row (four per lane in flight), the
// H.B and B C B^T terms with C in shared memory (lane j of the warp takes ranks j and j + 32).
// C = A A^T is symmetric bit for bit (k_dora_gram forms C[j, k] and C[k, j] with the same
// products in the same order), so lane j reads C[k, j]: consecutive lanes, distinct banks.
__global__ void __launch_bounds__(256) k_dora_combine(const __nv_bfloat16* __restrict__ W,
                                                      const float* __restrict__ H,
                                                      const float* __restrict__ B,
                                                      const float* __restrict__ C, float s,
                                                      int64_t out_dim, int64_t in_dim, int32_t rank,
                                                      float* __restrict__ norm_out) {
  grid_dep_sync();
  __shared__ float sC[LORA_MAX_RANK * LORA_MAX_RANK];
  for (int e = threadIdx.x; e < rank * rank; e += 256) sC[e] = C[e];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t o = (int64_t)blockIdx.x * 8 + warp;
  if (o >= out_dim) return;
  const __nv_bfloat16* w = W + o * in_dim;
  float wsq = 0.f;
  for (int64_t i0 = (int64_t)lane * 8; i0 < in_dim; i0 += 4 * 256) {
    uint4 raw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + (int64_t)u * 256;
      raw[u] = i < in_dim ? __ldg(reinterpret_cast<const uint4*>(w + i)) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (i0 + (int64_t)u * 256 >= in_dim) continue;
      const uint32_t q[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(q[e] << 16), hi = __uint_as_float(q[e] & 0xFFFF0000u);
        wsq = fmaf(lo, lo, wsq);
        wsq = fmaf(hi, hi, wsq);
      }
    }
  }
  float hb = 0.f, bcb = 0.f;
  for (int j = lane; j < rank; j += 32) {
    const float bj = B[o * rank + j];
    hb = fmaf(H[o * rank + j], bj, hb);
    float cb = 0.f;
    for (int k = 0; k < rank; ++k) cb = fmaf(sC[k * rank + j], B[o * rank + k], cb);
    bcb = fmaf(bj, cb, bcb);
  }
  for (int off = 16; off > 0; off >>= 1) {
    wsq += __shfl_xor_sync(0xffffffffu, wsq, off);
    hb += __shfl_xor_sync(0xffffffffu, hb, off);
    bcb += __shfl_xor_sync(0xffffffffu, bcb, off);
  }
  if (lane == 0) {
    const double n2 = (double)wsq + 2.0 * (double)s * hb + (double)s * (double)s * bcb;
    norm_out[o] = (float)sqrt(n2 > 0.0 ? n2 : 0.0);
  }
}

__device__ __forceinline__ void dm_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float dm_ld_peer(const float* local, uint32_t rank) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(local), remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

constexpr int kDmGroups = 8;   // token groups = CTAs of one cluster (16 for narrow outputs)
constexpr int kDmU = 8;        // tokens per warp in flight

// dm_o += (sum_t dY[t, o] * Y[t, o]) / m_o  (= sum_t dY * Z / n with Y = (m / n) Z).
// A cluster of kDmGroups CTAs covers a block of 32 * VEC columns (VEC = 16 bytes of elements per
// lane); CTA g sums its token group (8 warps taking every 8th token, kDmU loads in flight per
// warp), reduces its warps in warp order, and then each CTA adds, for its share of the block's
// columns, the groups' sums in group order (from the peers' shared memory) into dm.
// the V elements of a raw 16-byte chunk as floats
__device__ __forceinline__ void unpack16(const uint4& v, float (&out)[4]) {
  out[0] = __uint_as_float(v.x); out[1] = __uint_as_float(v.y);
  out[2] = __uint_as_float(v.z); out[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack16(const uint4& v, float (&out)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    out[2 * j] = __uint_as_float(w[j] << 16);
    out[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

template <typename T>
__global__ void __launch_bounds__(256, 3) k_dora_dm(const T* __restrict__ dY, const T* __restrict__ Y,
                                                 const float* __restrict__ mag, int64_t Tn,
                                                 int64_t out_dim, float* __restrict__ dm) {
  grid_dep_sync();
  constexpr int V = Vec<T>::N;
  constexpr int kCols = 32 * V;
  __shared__ float red[8][kCols];
  __shared__ float mine[kCols];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nb = (int64_t)blockIdx.x * kCols;
  const int64_t n0 = nb + (int64_t)lane * V;
  const bool nok = n0 < out_dim;   // out_dim is a multiple of 8, so a lane's columns are all in
  const int g = blockIdx.y;
  const int groups = gridDim.y;   // == the cluster size
  const int64_t tg = (Tn + groups - 1) / groups;
  const int64_t t_begin = (int64_t)g * tg;
  const int64_t t_end = min(Tn, t_begin + tg);
  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  if (nok) {
    for (int64_t t = t_begin + warp; t < t_end; t += 8 * kDmU) {
      // the loads stay raw (4 registers per chunk) until they are used
      uint4 a[kDmU], b[kDmU];
#pragma unroll
      for (int u = 0; u < kDmU; ++u) {
        const int64_t tt = t + 8 * u;
        if (tt < t_end) {
          a[u] = __ldg(reinterpret_cast<const uint4*>(dY + tt * out_dim + n0));
          b[u] = __ldg(reinterpret_cast<const uint4*>(Y + tt * out_dim + n0));
        } else {
          a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int u = 0; u < kDmU; ++u) {
        float x[V], y[V];
        unpack16(a[u], x);
        unpack16(b[u], y);
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = fmaf(x[e], y[e], acc[e]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < V; ++e) red[warp][lane * V + e] = acc[e];
  __syncthreads();
  for (int c = threadIdx.x; c < kCols; c += 256) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += red[w][c];
    mine[c] = sum;
  }
  dm_cluster_sync();
  const int share = kCols / groups;
  for (int cc = threadIdx.x; cc < share; cc += 256) {
    const int c = g * share + cc;
    const int64_t o = nb + c;
    if (o < out_dim) {
      float sum = 0.f;
      for (int gg = 0; gg < groups; ++gg) sum += dm_ld_peer(&mine[c], (uint32_t)gg);
      dm[o] += sum / mag[o];
    }
  }
  dm_cluster_sync();   // peers' shared memory stays alive until every CTA has read it
}

}  // namespace

cudaError_t launch_dora_norm(int dtype, const void* W, const float* A, const float* B, float s,
                             int64_t out_dim, int64_t in_dim, int32_t rank, float* norm_out,
                             cudaStream_t st) {
  const unsigned blocks = (unsigned)((out_dim + 3) / 4);
  if (dtype == LORA_F32)
    { prof_begin(0, st); launch_kernel(k_dora_norm<float>, blocks, 256, 0, st, (const float*)W, A, B, s, out_dim, in_dim, rank, norm_out); }
  else
    { prof_begin(0, st); launch_kernel(k_dora_norm<__nv_bfloat16>, blocks, 256, 0, st, (const __nv_bfloat16*)W, A, B, s, out_dim,
                                                       in_dim, rank, norm_out); }
  return cudaGetLastError();
}

cudaError_t launch_dora_gram_combine(const void* W, const float* H, const float* A, const float* B,
                                     float s, int64_t out_dim, int64_t in_dim, int32_t rank,
                                     float* C, float* norm_out, cudaStream_t st) {
  prof_begin(0, st);
  launch_kernel(k_dora_gram, dim3((unsigned)rank, (unsigned)((rank + 7) / 8)), 256, 0, st, A, in_dim, rank, C);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prof_begin(0, st);
  launch_kernel(k_dora_combine, (unsigned)((out_dim + 7) / 8), 256, 0, st, 
      (const __nv_bfloat16*)W, H, B, C, s, out_dim, in_dim, rank, norm_out);
  return cudaGetLastError();
}

cudaError_t launch_dora_dm(int dtype, const void* dY, const void* Y, const float* mag, int64_t T,
                           int64_t out_dim, float* dm, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int cols = dtype == LORA_F32 ? 32 * Vec<float>::N : 32 * Vec<__nv_bfloat16>::N;
  const int64_t blocks = (out_dim + cols - 1) / cols;
  // 16 token groups when 8 would leave most SMs idle (narrow outputs), if the device hosts such
  // clusters (the size above 8 needs the non-portable attribute)
  static int wide_ok[2] = {-1, -1};
  const int ti = dtype == LORA_F32 ? 0 : 1;
  if (wide_ok[ti] < 0) {
    cudaError_t ea = dtype == LORA_F32
        ? cudaFuncSetAttribute(k_dora_dm<float>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)
        : cudaFuncSetAttribute(k_dora_dm<__nv_bfloat16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    int n = 0;
    if (ea == cudaSuccess) {
      cudaLaunchConfig_t q{};
      q.gridDim = dim3(1, 16, 1);
      q.blockDim = dim3(256);
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = 1;
      qa[0].val.clusterDim.y = 16;
      qa[0].val.clusterDim.z = 1;
      q.attrs = qa;
      q.numAttrs = 1;
      if ((dtype == LORA_F32 ? cudaOccupancyMaxActiveClusters(&n, k_dora_dm<float>, &q)
                             : cudaOccupancyMaxActiveClusters(&n, k_dora_dm<__nv_bfloat16>, &q)) !=
          cudaSuccess)
        n = 0;
    }
    cudaGetLastError();
    wide_ok[ti] = n > 0 ? 1 : 0;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 152;
  const int groups = (wide_ok[ti] == 1 && blocks * kDmGroups < sms) ? 16 : kDmGroups;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)blocks, (unsigned)groups);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)groups;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = add_pdl_attr(attr, 1);
  prof_begin(0, st);
  cudaError_t e = dtype == LORA_F32
                      ? cudaLaunchKernelEx(&cfg, k_dora_dm<float>, (const float*)dY, (const float*)Y,
                                           mag, T, out_dim, dm)
                      : cudaLaunchKernelEx(&cfg, k_dora_dm<__nv_bfloat16>,
                                           (const __nv_bfloat16*)dY, (const __nv_bfloat16*)Y, mag, T,
                                           out_dim, dm);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace lora
