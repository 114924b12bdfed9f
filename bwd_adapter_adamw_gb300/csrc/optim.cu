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

// (ah, al) += (bh, bl) for float-float pairs: TwoSum of the high parts, the low parts and that
// rounding error added, then renormalised with Fast2Sum.
__device__ __forceinline__ void ff_add(float& ah, float& al, float bh, float bl) {
  const float s = __fadd_rn(ah, bh);
  const float bp = __fsub_rn(s, ah);
  const float err = __fadd_rn(__fsub_rn(ah, __fsub_rn(s, bp)), __fsub_rn(bh, bp));
  const float t = __fadd_rn(__fadd_rn(al, bl), err);
  const float h = __fadd_rn(s, t);
  al = __fsub_rn(t, __fsub_rn(h, s));
  ah = h;
}

// One element of pass 1. |a| > 2^40 (and +-Inf) goes to a double accumulator: a square below
// 2^80 keeps a CTA's float-float sum (at most 2^24 elements) far inside the float range, so no
// finite gradient overflows; NaN propagates through hi. The block sum is non-finite iff an
// element is.
__device__ __forceinline__ void sq_accum(float a, float& hi, float& lo, double& big) {
  if (fabsf(a) > 0x1p40f) {
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
  __shared__ float2 shf[kPrepThreads / 32];
  __shared__ bool am_last;
  const int b = blockIdx.x;
  const int g = find_group(gt, b);
  const int64_t begin = (int64_t)(b - gt.block_begin[g]) * per_block;
  const int64_t n = min(per_block, gt.count[g] - begin);
  const float* p = grads + gt.offset[g] + begin;
  // Two independent float-float accumulators per thread (x, y and z, w of each float4) halve the
  // dependent chain, and every batch issues its kPrepBatch 16-byte loads before any add (the
  // last batch predicated, zeros past the end), so that a thread's whole run is in flight in one
  // or two round trips. A zero adds nothing to the pair, so each thread still sums its own
  // elements in increasing order.
  constexpr int kPrepBatch = 8;
  float hi0 = 0.f, lo0 = 0.f, hi1 = 0.f, lo1 = 0.f;
  double big = 0.0;
  const int64_t nv = n >> 2;
  const float4* p4 = reinterpret_cast<const float4*>(p);
  for (int64_t v0 = 0; v0 < nv; v0 += kPrepBatch * kPrepThreads) {
    float4 x[kPrepBatch];
#pragma unroll
    for (int u = 0; u < kPrepBatch; ++u) {
      const int64_t v = v0 + threadIdx.x + u * kPrepThreads;
      x[u] = v < nv ? __ldcs(p4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // One warp-uniform test per batch keeps the per-element path in FP32: only a batch of a warp
    // that holds a value above 2^40 or an infinity takes the per-element test with its double
    // accumulator (fmaxf passes over NaN, which the float-float pair propagates by itself).
    float mx = 0.f;
#pragma unroll
    for (int u = 0; u < kPrepBatch; ++u)
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x[u].x), fabsf(x[u].y)), fmaxf(fabsf(x[u].z), fabsf(x[u].w))));
    if (__any_sync(0xffffffffu, mx > 0x1p40f)) {
#pragma unroll
      for (int u = 0; u < kPrepBatch; ++u) {
        sq_accum(x[u].x, hi0, lo0, big);
        sq_accum(x[u].y, hi0, lo0, big);
        sq_accum(x[u].z, hi1, lo1, big);
        sq_accum(x[u].w, hi1, lo1, big);
      }
    } else {
#pragma unroll
      for (int u = 0; u < kPrepBatch; ++u) {
        ff_add_square(x[u].x, hi0, lo0);
        ff_add_square(x[u].y, hi0, lo0);
        ff_add_square(x[u].z, hi1, lo1);
        ff_add_square(x[u].w, hi1, lo1);
      }
    }
  }
  for (int64_t e = (nv << 2) + threadIdx.x; e < n; e += kPrepThreads) sq_accum(p[e], hi0, lo0, big);
  // The CTA's pairs are summed in float-float in a fixed tree (lanes by shuffles, then the warps
  // in order by thread 0): FP64 runs at a small fraction of the FP32 rate on this part, so
  // double arithmetic is kept to one conversion per CTA (and the rare large-element sum).
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  ff_add(hi0, lo0, hi1, lo1);
  for (int off = 16; off > 0; off >>= 1) {
    const float oh = __shfl_down_sync(0xffffffffu, hi0, off);
    const float ol = __shfl_down_sync(0xffffffffu, lo0, off);
    ff_add(hi0, lo0, oh, ol);
  }
  if (lane == 0) shf[warp] = make_float2(hi0, lo0);
  const bool any_big = __syncthreads_or(big != 0.0);
  const double big_sum = any_big ? block_sum_double(big, sh) : 0.0;
  if (threadIdx.x == 0) {
    float th = shf[0].x, tl = shf[0].y;
    for (int w = 1; w < kPrepThreads / 32; ++w) ff_add(th, tl, shf[w].x, shf[w].y);
    part[b] = ((double)th + (double)tl) + big_sum;
    __threadfence();
    const uint32_t done = atomicAdd(counter, 1u);
    am_last = (done == gridDim.x - 1);
  }
  __syncthreads();
  if (!am_last) return;
  __threadfence();
  // last block: one warp per group, each reducing that group's block partials in a fixed order
  // (lane l sums partials l, l + 32, ... in turn, then a fixed shuffle tree), all groups at once
  for (int gg = warp; gg < gt.n; gg += kPrepThreads / 32) {
    const int b0 = gt.block_begin[gg], b1 = gt.block_begin[gg + 1];
    double S = 0.0;
#pragma unroll 8
    for (int k = b0 + lane; k < b1; k += 32) S += __ldcg(part + k);
    for (int off = 16; off > 0; off >>= 1) S += __shfl_down_sync(0xffffffffu, S, off);
    if (lane == 0) {
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
                                                        int zero_grads, int64_t per_block) {
  grid_dep_sync();
  const int b = blockIdx.x;
  const int g = find_group(gt, b);
  // the group's verdict and factor are read alongside the first batch, not ahead of it
  const int32_t verdict = status[g];
  const double factor = scale_norm[2 * g];
  const float lr = gt.lr[g];
  const float inv_bc1 = 1.f / gt.bc1[g], inv_bc2 = 1.f / gt.bc2[g];
  const int64_t begin = (int64_t)(b - gt.block_begin[g]) * per_block;
  const int64_t n = min(per_block, gt.count[g] - begin);
  const int64_t base = gt.offset[g] + begin;
  const int64_t na = gt.n_a[g], nab = gt.n_a[g] + gt.n_b[g];
  const int64_t nv = n >> 2;
  // kAdamBatch float4 of each of p, g, m, v per thread in flight before any update
  constexpr int kAdamBatch = 2;
  for (int64_t q0 = 0; q0 < nv; q0 += kAdamBatch * kAdamThreads) {
    float4 p[kAdamBatch], gr[kAdamBatch], m[kAdamBatch], v[kAdamBatch];
#pragma unroll
    for (int u = 0; u < kAdamBatch; ++u) {
      const int64_t q = q0 + threadIdx.x + u * kAdamThreads;
      if (q < nv) {
        const int64_t e = base + (q << 2);
        p[u] = *reinterpret_cast<const float4*>(P + e);
        gr[u] = *reinterpret_cast<const float4*>(G + e);
        m[u] = *reinterpret_cast<const float4*>(Mo + e);
        v[u] = *reinterpret_cast<const float4*>(V + e);
      }
    }
    if (verdict != LORA_OK) return;
    const float c = (float)factor;
#pragma unroll
    for (int u = 0; u < kAdamBatch; ++u) {
      const int64_t q = q0 + threadIdx.x + u * kAdamThreads;
      if (q >= nv) continue;
      const int64_t e = base + (q << 2);
      float* pp = &p[u].x; float* gg = &gr[u].x; float* mm = &m[u].x; float* vv = &v[u].x;
      const int64_t li = begin + (q << 2);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t l = li + j;
        const int kind = (l < na) ? 0 : ((l < nab) ? 1 : 2);
        adam_elem(pp[j], gg[j], mm[j], vv[j], kind, c, lr, hp, inv_bc1, inv_bc2);
      }
      *reinterpret_cast<float4*>(P + e) = p[u];
      *reinterpret_cast<float4*>(Mo + e) = m[u];
      *reinterpret_cast<float4*>(V + e) = v[u];
      if (zero_grads) *reinterpret_cast<float4*>(G + e) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (verdict != LORA_OK) return;
  const float c = (float)factor;
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
  // elements per CTA: about eight CTAs per SM over the whole arena, each thread holding one or
  // more batches, so that a small arena still has all its loads in flight at once
  int64_t total = 0;
  for (int i = 0; i < gt.n; ++i) total += gt.count[i];
  const int64_t unit = 2 * 4 * kAdamThreads;   // one batch of the kernel
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 152;
  const int64_t target = (int64_t)8 * sms;
  int64_t per = (total / target + unit - 1) / unit * unit;
  per = per < unit ? unit : (per > 4 * unit ? 4 * unit : per);
  const int blocks = set_blocks(gt, per);
  if (blocks == 0) return cudaSuccess;
  prof_begin(LORA_PROF_ADAMW, st);
  launch_kernel(k_adamw, blocks, kAdamThreads, 0, st, p, g, m, v, gt, hp, d_scale_norm, d_status,
                zero_grads, per);
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
