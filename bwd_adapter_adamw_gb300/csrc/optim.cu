// Two-pass global-norm clip and the fused clip + A-only decoupled AdamW update over flat fp32
// arenas ("4.3. Training Guide", Gradient clipping: pass 1 accumulates the squared norm in double
// and rejects non-finite values before any mutation, pass 2 applies one combined normalisation x
// clipping factor; Optimizer: decay on A only from the pre-update value with the scheduled lr,
// LoRA+ ratio on B's lr, moments see the gradient without decay).
#include <mutex>

#include "lora_kernels.h"

namespace lora {

namespace {

// a^2 added exactly into the float-float pair (hi, lo): the square is split error-free with an
// FMA (TwoProduct) and added with Knuth's TwoSum. The *_rn intrinsics keep the compiler from
// fusing or reassociating these steps.
__device__ __forceinline__ void ff_add_square(float a, float& hi, float& lo) {
  const float p = __fmul_rn(a, a);
  const float e = fmaf(a, a, -p);
  const float s = __fadd_rn(hi, p);
  const float bp = __fsub_rn(s, hi);
  const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(p, bp));
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(err, e));
}

// One element of pass 1. |a| > 2^60 (and +-Inf) goes to a double accumulator so that no finite
// square overflows; NaN propagates through hi. The block sum is non-finite iff an element is.
__device__ __forceinline__ void sq_accum(float a, float& hi, float& lo, double& big) {
  if (fabsf(a) > 0x1p60f) {
    const double d = (double)a;
    big = fma(d, d, big);
  } else {
    ff_add_square(a, hi, lo);
  }
}

__device__ __forceinline__ double block_sum_double(double v, double* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(0xffffffffu, v, off);
  __syncthreads();
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  double r = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r += sh[w];
  return r;  // valid in thread 0
}

__device__ __forceinline__ int find_group(const GroupTab& g, int b) {
  int lo = 0, hi = g.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (g.block_begin[mid] <= b) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kPrepThreads, 4) k_grad_prepare(const float* __restrict__ grads,
                                                               const GroupTab gt,
                                                               double* __restrict__ scale_norm,
                                                               int32_t* __restrict__ status,
                                                               double* part, uint32_t* counter,
                                                               int64_t per_block) {
  grid_dep_sync();
  __shared__ double sh[kPrepThreads / 32];
  __shared__ bool am_last;
  const int b = blockIdx.x;
  const int g = find_group(gt, b);
  const int64_t begin = (int64_t)(b - gt.block_begin[g]) * per_block;
  const int64_t n = min(per_block, gt.count[g] - begin);
  const float* p = grads + gt.offset[g] + begin;
  // Two independent float-float accumulators per thread (x, y and z, w of each float4) halve the
  // dependent chain, and each batch issues kPrepBatch independent 16-byte loads before any add,
  // so that enough bytes are in flight to stream at the memory's rate.
  constexpr int kPrepBatch = 8;
  float hi0 = 0.f, lo0 = 0.f, hi1 = 0.f, lo1 = 0.f;
  double big = 0.0;
  const int64_t nv = n >> 2;
  const float4* p4 = reinterpret_cast<const float4*>(p);
  int64_t v = threadIdx.x;
  for (; v + (kPrepBatch - 1) * kPrepThreads < nv; v += kPrepBatch * kPrepThreads) {
    float4 x[kPrepBatch];
#pragma unroll
    for (int u = 0; u < kPrepBatch; ++u) x[u] = __ldcs(p4 + v + u * kPrepThreads);
#pragma unroll
    for (int u = 0; u < kPrepBatch; ++u) {
      sq_accum(x[u].x, hi0, lo0, big);
      sq_accum(x[u].y, hi0, lo0, big);
      sq_accum(x[u].z, hi1, lo1, big);
      sq_accum(x[u].w, hi1, lo1, big);
    }
  }
  for (; v < nv; v += kPrepThreads) {
    const float4 x = __ldcs(p4 + v);
    sq_accum(x.x, hi0, lo0, big);
    sq_accum(x.y, hi0, lo0, big);
    sq_accum(x.z, hi1, lo1, big);
    sq_accum(x.w, hi1, lo1, big);
  }
  for (int64_t e = (nv << 2) + threadIdx.x; e < n; e += kPrepThreads) sq_accum(p[e], hi0, lo0, big);
  const double mine = (((double)hi0 + (double)lo0) + ((double)hi1 + (double)lo1)) + big;
  const double tot = block_sum_double(mine, sh);
  if (threadIdx.x == 0) {
    part[b] = tot;
    __threadfence();
    const uint32_t done = atomicAdd(counter, 1u);
    am_last = (done == gridDim.x - 1);
  }
  __syncthreads();
  if (!am_last) return;
  __threadfence();
  // last block: per group, fixed-order reduction of that group's block partials
  for (int gg = 0; gg < gt.n; ++gg) {
    const int b0 = gt.block_begin[gg], b1 = gt.block_begin[gg + 1];
    double acc = 0.0;
#pragma unroll 4
    for (int k = b0 + threadIdx.x; k < b1; k += kPrepThreads) acc += __ldcg(part + k);
    const double S = block_sum_double(acc, sh);
    if (threadIdx.x == 0) {
      if (!isfinite(S)) {
        status[gg] = LORA_ERR_NONFINITE;
        scale_norm[2 * gg] = 0.0;
        scale_norm[2 * gg + 1] = S;
      } else {
        const double gamma = gt.gamma[gg];
        const double norm = sqrt(S) * gamma;
        const double mx = (double)gt.max_norm[gg];
        const double c = (mx > 0.0 && norm > mx) ? gamma * (mx / norm) : gamma;
        status[gg] = LORA_OK;
        scale_norm[2 * gg] = c;
        scale_norm[2 * gg + 1] = norm;
      }
    }
  }
}

__device__ __forceinline__ void adam_elem(float& p, float g, float& m, float& v, int kind,
                                          float c, float lr, const AdamK& k, float inv_bc1,
                                          float inv_bc2) {
  const float gh = g * c;
  m = fmaf(k.b1, m, k.omb1 * gh);
  v = fmaf(k.b2, v, k.omb2 * gh * gh);
  const float u = (m * inv_bc1) / (sqrtf(v * inv_bc2) + k.eps);
  if (kind == 0)
    p = p - lr * u - lr * k.wd * p;
  else if (kind == 1)
    p = p - (lr * k.rho) * u;
  else
    p = p - lr * u;
}

__global__ void __launch_bounds__(kAdamThreads) k_adamw(float* __restrict__ P, float* __restrict__ G,
                                                        float* __restrict__ Mo, float* __restrict__ V,
                                                        const GroupTab gt, const AdamK hp,
                                                        const double* __restrict__ scale_norm,
                                                        const int32_t* __restrict__ status,
                                                        int zero_grads) {
  grid_dep_sync();
  const int b = blockIdx.x;
  const int g = find_group(gt, b);
  if (status[g] != LORA_OK) return;
  const float c = (float)scale_norm[2 * g];
  const float lr = gt.lr[g];
  const float inv_bc1 = 1.f / gt.bc1[g], inv_bc2 = 1.f / gt.bc2[g];
  const int64_t begin = (int64_t)(b - gt.block_begin[g]) * kAdamElemsPerBlock;
  const int64_t n = min((int64_t)kAdamElemsPerBlock, gt.count[g] - begin);
  const int64_t base = gt.offset[g] + begin;
  const int64_t na = gt.n_a[g], nab = gt.n_a[g] + gt.n_b[g];
  const int64_t nv = n >> 2;
  for (int64_t q = threadIdx.x; q < nv; q += kAdamThreads) {
    const int64_t e = base + (q << 2);
    float4 p = *reinterpret_cast<float4*>(P + e);
    float4 gr = *reinterpret_cast<float4*>(G + e);
    float4 m = *reinterpret_cast<float4*>(Mo + e);
    float4 v = *reinterpret_cast<float4*>(V + e);
    float* pp = &p.x; float* gg = &gr.x; float* mm = &m.x; float* vv = &v.x;
    const int64_t li = begin + (q << 2);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t l = li + j;
      const int kind = (l < na) ? 0 : ((l < nab) ? 1 : 2);
      adam_elem(pp[j], gg[j], mm[j], vv[j], kind, c, lr, hp, inv_bc1, inv_bc2);
    }
    *reinterpret_cast<float4*>(P + e) = p;
    *reinterpret_cast<float4*>(Mo + e) = m;
    *reinterpret_cast<float4*>(V + e) = v;
    if (zero_grads) *reinterpret_cast<float4*>(G + e) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int64_t l = begin + (nv << 2) + threadIdx.x; l < begin + n; l += kAdamThreads) {
    const int64_t e = gt.offset[g] + l;
    const int kind = (l < na) ? 0 : ((l < nab) ? 1 : 2);
    float p = P[e], gr = G[e], m = Mo[e], v = V[e];
    adam_elem(p, gr, m, v, kind, c, lr, hp, inv_bc1, inv_bc2);
    P[e] = p; Mo[e] = m; V[e] = v;
    if (zero_grads) G[e] = 0.f;
  }
}

// Adapter-state maintenance over the groups' ranges (snapshot, restore with optimizer reset,
// slot retirement): dst = src when kMaintCopy, dst = 0 when kMaintZeroDst, G = 0 when kMaintZeroG,
// M = V = 0 when kMaintZeroMV. One CTA per kAdamElemsPerBlock elements of a group.
__global__ void __launch_bounds__(kAdamThreads) k_group_maint(float* __restrict__ dst,
                                                              const float* __restrict__ src,
                                                              float* __restrict__ G,
                                                              float* __restrict__ M,
                                                              float* __restrict__ V,
                                                              const GroupTab gt, int flags) {
  grid_dep_sync();
  const int b = blockIdx.x;
  const int g = find_group(gt, b);
  const int64_t begin = (int64_t)(b - gt.block_begin[g]) * kAdamElemsPerBlock;
  const int64_t n = min((int64_t)kAdamElemsPerBlock, gt.count[g] - begin);
  const int64_t base = gt.offset[g] + begin;
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  const int64_t nv = n >> 2;
  for (int64_t q = threadIdx.x; q < nv; q += kAdamThreads) {
    const int64_t e = base + (q << 2);
    if (flags & kMaintCopy)
      *reinterpret_cast<float4*>(dst + e) = *reinterpret_cast<const float4*>(src + e);
    else if (flags & kMaintZeroDst)
      *reinterpret_cast<float4*>(dst + e) = z4;
    if (flags & kMaintZeroG) *reinterpret_cast<float4*>(G + e) = z4;
    if (flags & kMaintZeroMV) {
      *reinterpret_cast<float4*>(M + e) = z4;
      *reinterpret_cast<float4*>(V + e) = z4;
    }
  }
  for (int64_t e = base + (nv << 2) + threadIdx.x; e < base + n; e += kAdamThreads) {
    if (flags & kMaintCopy) dst[e] = src[e];
    else if (flags & kMaintZeroDst) dst[e] = 0.f;
    if (flags & kMaintZeroG) G[e] = 0.f;
    if (flags & kMaintZeroMV) { M[e] = 0.f; V[e] = 0.f; }
  }
}

int set_blocks(GroupTab& g, int64_t per_block) {
  int total = 0;
  for (int i = 0; i < g.n; ++i) {
    g.block_begin[i] = total;
    total += (int)((g.count[i] + per_block - 1) / per_block);
  }
  g.block_begin[g.n] = total;
  return total;
}

}  // namespace

int prepare_blocks(const GroupTab& g, int64_t per_block) {
  GroupTab t = g;
  return set_blocks(t, per_block);
}

cudaError_t launch_grad_prepare(const float* grads, const GroupTab& g_in, double* d_scale_norm,
                                int32_t* d_status, double* part, uint32_t* counter, cudaStream_t st,
                                int64_t per_block) {
  GroupTab g = g_in;
  int blocks = set_blocks(g, per_block);
  cudaError_t e = cudaMemsetAsync(counter, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  if (blocks == 0) {
    // every group is empty: one block writes the zero-norm results
    blocks = 1;
    g.block_begin[g.n] = 1;
    for (int i = 0; i < g.n; ++i) g.block_begin[i] = 0;
  }
  prof_begin(LORA_PROF_PREPARE, st);
  launch_kernel(k_grad_prepare, blocks, kPrepThreads, 0, st, grads, g, d_scale_norm, d_status, part, counter,
                                                  per_block);
  prof_end(LORA_PROF_PREPARE, st);
  return cudaGetLastError();
}

cudaError_t launch_group_maint(float* dst, const float* src, float* g, float* m, float* v,
                               const GroupTab& gt_in, int flags, cudaStream_t st) {
  GroupTab gt = gt_in;
  const int blocks = set_blocks(gt, kAdamElemsPerBlock);
  if (blocks == 0) return cudaSuccess;
  prof_begin(0, st);
  launch_kernel(k_group_maint, blocks, kAdamThreads, 0, st, dst, src, g, m, v, gt, flags);
  return cudaGetLastError();
}

cudaError_t launch_adamw(float* p, float* g, float* m, float* v, const GroupTab& gt_in,
                         const AdamK& hp, const double* d_scale_norm, const int32_t* d_status,
                         int zero_grads, cudaStream_t st) {
  GroupTab gt = gt_in;
  const int blocks = set_blocks(gt, kAdamElemsPerBlock);
  if (blocks == 0) return cudaSuccess;
  prof_begin(LORA_PROF_ADAMW, st);
  launch_kernel(k_adamw, blocks, kAdamThreads, 0, st, p, g, m, v, gt, hp, d_scale_norm, d_status, zero_grads);
  prof_end(LORA_PROF_ADAMW, st);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Allocation-free variant of the prepare launch: its scratch (the per-block double partials and
// the last-block counter) lives in this file-scope device array instead of a caller workspace.
// Every GPU that loads the library holds the array until exit; all calls share it, so calls
// that overlap on the GPU race, and the counter is cleared by every call.
// ------------------------------------------------------------------------------------------
namespace {
constexpr size_t kNoallocCounterOffset = sizeof(double) * kNoallocMaxPartials;
constexpr size_t kNoallocBytes = kNoallocCounterOffset + 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

std::mutex g_noalloc_mu;
constexpr int kMaxDevices = 64;
void* g_noalloc_ptr[kMaxDevices] = {};

// Host code cannot use &g_noalloc_scratch as a device address (it names a host-side stand-in);
// the device address is looked up once per device, with that device current.
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_grad_prepare_noalloc(const float* grads, const GroupTab& g,
                                        double* d_scale_norm, int32_t* d_status,
                                        cudaStream_t st) {
  void* base = nullptr;
  cudaError_t e = noalloc_scratch(&base);
  if (e != cudaSuccess) return e;
  double* part = reinterpret_cast<double*>(base);
  uint32_t* counter = reinterpret_cast<uint32_t*>(static_cast<char*>(base) + kNoallocCounterOffset);
  return launch_grad_prepare(grads, g, d_scale_norm, d_status, part, counter, st,
                             kPrepElemsPerBlock);
}

}  // namespace lora
