// Streaming CUDA-core low-rank products for fp32 activations (and small ranks): at rank r the
// products do ~r/2 flops per streamed byte of X or dY, so for the ranks of fp32 workloads they
// are bound by HBM, not by the FMA units, and run at exact rank width here.
//
//  k_rowdot:  out[t, j] = alpha_slot * sum_k A'[t, k] S_slot[j, k]   (shrink with S = A,
//             G with S = B^T); one warp per token, lanes stride over K with 16-byte loads, the
//             slot's S staged in shared memory one K-chunk at a time, warp-shuffle reduction.
//             Since it reads every A'[t, k] anyway, it also writes the bf16 hi / lo split of A'
//             that the split fp32 frozen product consumes (X in the forward, dY' in the backward).
//  k_colred:  part[item][n][j] = sum_{t in item} P[t, j] B'[t, n]   (dB with P = Hs, B' = dY';
//             dA^T with P = Gs, B' = Xd); every thread owns CPT adjacent columns, the item's P
//             rows are staged in shared memory, one partial per work item, reduced in order.
// ("Backward Bug Hunts and Vulkan Tiled GEMM", The fix: a 16x16 shared-memory tiled GEMM --
// operand reuse through shared memory; here the reused operand is the small adapter side.)
#include "lora_kernels.h"

namespace lora {

namespace {

// bf16 hi / lo of A'[t, k .. k + 3] for the tokens t = t0 + u < t1 (the split frozen product's
// operands)
template <int U>
__device__ __forceinline__ void write_split(const RowDotArgs& a, const float (&x)[U][4], int64_t t0,
                                            int64_t t1, int64_t k) {
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (t0 + u >= t1) continue;
    const int64_t o = (t0 + u) * a.K + k;
    uint2 h, l;
    bf16_split4(x[u], h, l);
    *reinterpret_cast<uint2*>(a.split_hi + o) = h;
    *reinterpret_cast<uint2*>(a.split_lo + o) = l;
  }
}

constexpr int kRowWarps = 8;
constexpr int kRowSmemFloats = 12288;              // 48 KB of S per K-chunk

// tokens per warp: 4 for small ranks (amortises the shared S reads), 1 for large ranks
template <int R> struct RowTpw { static constexpr int v = R <= 16 ? 4 : 1; };

template <typename TA, int R>
__global__ void __launch_bounds__(256) k_rowdot(const RowDotArgs a) {
  grid_dep_sync();
  constexpr int kTokPerWarp = RowTpw<R>::v;
  constexpr int kRowTok = kRowWarps * kTokPerWarp;   // tokens per CTA (within one work item)
  __shared__ __align__(16) float sS[kRowSmemFloats];
  const int item = blockIdx.x;
  TokenItem it;
  if (!get_item(a.items, a.n_items, item, a.T, it)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tbase = (int64_t)it.t0 + (int64_t)blockIdx.y * kRowTok + warp * kTokPerWarp;
  if ((int64_t)it.t0 + (int64_t)blockIdx.y * kRowTok >= it.t1) return;
  const int slot = it.slot;
  const int32_t r = slot >= 0 ? a.rank[slot] : 0;
  const float* S = slot >= 0 ? a.s[slot] : nullptr;
  const int64_t K = a.K;
  // chunk width: columns of S held in shared memory (a multiple of 128 = 32 lanes x 4)
  int64_t chunk = (kRowSmemFloats / R) / 128 * 128;
  if (chunk > K) chunk = (K + 127) / 128 * 128;
  float acc[kTokPerWarp][R];
#pragma unroll
  for (int u = 0; u < kTokPerWarp; ++u)
#pragma unroll
    for (int j = 0; j < R; ++j) acc[u][j] = 0.f;
  const bool split = Vec<TA>::N == 4 && a.split_hi != nullptr;
  for (int64_t k0 = 0; k0 < K && (r > 0 || split); k0 += chunk) {
    const int64_t kn = min(chunk, K - k0);
    __syncthreads();
    for (int64_t e = threadIdx.x; e < (int64_t)R * chunk; e += 256) {
      const int j = (int)(e / chunk);
      const int64_t k = e - (int64_t)j * chunk;
      sS[e] = (j < r && k < kn) ? __ldg(S + (a.s_rows_k ? (k0 + k) * a.lds + j : (int64_t)j * a.lds + k0 + k))
                                : 0.f;
    }
    __syncthreads();
    for (int64_t k = lane * 4; k < kn; k += 128) {
      float s4[R][4];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const float4 v = *reinterpret_cast<const float4*>(&sS[(int64_t)j * chunk + k]);
        s4[j][0] = v.x; s4[j][1] = v.y; s4[j][2] = v.z; s4[j][3] = v.w;
      }
#pragma unroll
      for (int u = 0; u < kTokPerWarp; ++u) {
        const int64_t t = tbase + u;
        if (t >= it.t1) continue;
        float x[8];
        const TA* src = reinterpret_cast<const TA*>(a.a) + t * a.lda + k0 + k;
        if (Vec<TA>::N == 4) {
          load16(reinterpret_cast<const float*>(src), x);
        } else {
          // bf16: 4 elements = 8 bytes
          const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
          x[0] = __uint_as_float(w.x << 16); x[1] = __uint_as_float(w.x & 0xFFFF0000u);
          x[2] = __uint_as_float(w.y << 16); x[3] = __uint_as_float(w.y & 0xFFFF0000u);
        }
        if (a.colscale) {
#pragma unroll
          for (int e = 0; e < 4; ++e) x[e] *= __ldg(a.colscale + k0 + k + e);
        }
        if (split) {
          const float xs[1][4] = {{x[0], x[1], x[2], x[3]}};
          write_split<1>(a, xs, t, it.t1, k0 + k);
        }
        if (a.mask) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (!drop_keep(a.drop, t, k0 + k + e)) x[e] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < R; ++j)
          acc[u][j] = fmaf(x[0], s4[j][0], fmaf(x[1], s4[j][1], fmaf(x[2], s4[j][2], fmaf(x[3], s4[j][3], acc[u][j]))));
      }
    }
  }
  const float alpha = slot >= 0 ? a.alpha[slot] : 0.f;
#pragma unroll
  for (int u = 0; u < kTokPerWarp; ++u) {
#pragma unroll
    for (int j = 0; j < R; ++j) {
      float v = acc[u][j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      acc[u][j] = v;
    }
    const int64_t t = tbase + u;
    if (t < it.t1) {
      // lane j writes column j (columns r..ldo-1 are zero)
      for (int j = lane; j < a.ldo; j += 32) {
        float v = 0.f;
#pragma unroll
        for (int jj = 0; jj < R; ++jj)
          if (jj == j) v = acc[u][jj];
        a.out[t * a.ldo + j] = (j < r) ? v * alpha : 0.f;
      }
    }
  }
}

constexpr int kColThreads = 256;
constexpr int kColTokChunk = 64;

template <typename TB, int R, int CPT>
__global__ void __launch_bounds__(kColThreads) k_colred(const ColRedArgs a) {
  grid_dep_sync();
  __shared__ __align__(16) float sP[kColTokChunk * R];
  const int item = blockIdx.y;
  TokenItem it;
  if (!get_item(a.items, a.n_items, item, a.T, it)) return;
  if (it.slot < 0) return;
  const int32_t r = a.rank[it.slot];
  const int64_t n0 = ((int64_t)blockIdx.x * kColThreads + threadIdx.x) * CPT;
  float acc[CPT][R];
#pragma unroll
  for (int c = 0; c < CPT; ++c)
#pragma unroll
    for (int j = 0; j < R; ++j) acc[c][j] = 0.f;
  for (int64_t t0 = it.t0; t0 < it.t1; t0 += kColTokChunk) {
    const int nt = (int)min((int64_t)kColTokChunk, (int64_t)it.t1 - t0);
    __syncthreads();
    for (int e = threadIdx.x; e < kColTokChunk * R; e += kColThreads) {
      const int tt = e / R, j = e - tt * R;
      sP[e] = (tt < nt && j < r) ? a.p[(t0 + tt) * a.ldp + j] : 0.f;
    }
    __syncthreads();
    if (n0 < a.N) {
      for (int tt = 0; tt < nt; ++tt) {
        const int64_t t = t0 + tt;
        float b[CPT];
        const TB* src = reinterpret_cast<const TB*>(a.b) + t * a.ldb + n0;
        if (CPT == 4 && Vec<TB>::N == 4) {
          load16(reinterpret_cast<const float*>(src), b);
        } else {
#pragma unroll
          for (int c = 0; c < CPT; ++c) b[c] = to_f(src[c]);
        }
        if (a.colscale) {
#pragma unroll
          for (int c = 0; c < CPT; ++c) b[c] *= __ldg(a.colscale + n0 + c);
        }
        if (a.mask) {
#pragma unroll
          for (int c = 0; c < CPT; ++c)
            if (!drop_keep(a.drop, t, n0 + c)) b[c] = 0.f;
        }
        float pv[R];
#pragma unroll
        for (int j = 0; j < R; j += 4) {
          const float4 v = *reinterpret_cast<const float4*>(&sP[tt * R + j]);
          pv[j] = v.x; pv[j + 1] = v.y; pv[j + 2] = v.z; pv[j + 3] = v.w;
        }
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
          for (int j = 0; j < R; ++j) acc[c][j] = fmaf(pv[j], b[c], acc[c][j]);
      }
    }
  }
  if (n0 >= a.N) return;
  float* part = a.part + (int64_t)item * a.N * a.ldpart;
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    float* dst = part + (n0 + c) * a.ldpart;
#pragma unroll
    for (int j = 0; j < R; ++j)
      if (j < a.ldpart) dst[j] = acc[c][j];
  }
}

template <typename TA, int R>
void rowdot_launch(const RowDotArgs& a, int max_items, cudaStream_t st) {
  constexpr int tok = kRowWarps * RowTpw<R>::v;
  dim3 grid((unsigned)max_items, (unsigned)((kGemmTileT + tok - 1) / tok));
  launch_kernel(k_rowdot<TA, R>, grid, 256, 0, st, a);
}

// ---------------------------------------------------------------------------------------------
// Wide variants for ranks <= 16: many small CTAs and all loads of a thread in flight at once.
// ---------------------------------------------------------------------------------------------
constexpr int kRdTok = 8;       // tokens per CTA
constexpr int kRdCols = 1024;   // K columns per CTA (256 threads x 4)

// Sum each of V values over the 32 lanes by recursive halving: afterwards lane L holds the totals
// of the original indices [L * V / 32, (L + 1) * V / 32) in v[0 .. V / 32).
template <int V>
__device__ __forceinline__ void warp_halving_sum(float (&v)[V], const int lane) {
#pragma unroll
  for (int off = 16, n = V; off >= 1; off >>= 1, n >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
}

// part[kc][t][j] = sum over the CTA's K-chunk kc of A'[t, k] S_slot[j, k]
template <typename TA, int R>
__global__ void __launch_bounds__(256) k_rowdot_wide(const RowDotArgs a, float* __restrict__ part) {
  grid_dep_sync();
  constexpr int V = kRdTok * R;
  __shared__ float red[8][V];
  const int item = blockIdx.x / (kGemmTileT / kRdTok);
  const int grp = blockIdx.x % (kGemmTileT / kRdTok);
  TokenItem it;
  if (!get_item(a.items, a.n_items, item, a.T, it)) return;
  const int64_t tg = (int64_t)it.t0 + (int64_t)grp * kRdTok;
  if (tg >= it.t1) return;
  const int kc = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = it.slot;
  const int32_t r = slot >= 0 ? a.rank[slot] : 0;
  const int64_t k = (int64_t)kc * kRdCols + threadIdx.x * 4;
  const bool kin = k < a.K;
  const bool kok = kin && r > 0;
  float sv[R][4];
#pragma unroll
  for (int j = 0; j < R; ++j) {
    if (kok && j < r) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(a.s[slot] + (int64_t)j * a.lds + k));
      sv[j][0] = q.x; sv[j][1] = q.y; sv[j][2] = q.z; sv[j][3] = q.w;
    } else {
      sv[j][0] = sv[j][1] = sv[j][2] = sv[j][3] = 0.f;
    }
  }
  float x[kRdTok][4];
#pragma unroll
  for (int u = 0; u < kRdTok; ++u) {
    const int64_t t = tg + u;
    if (kin && t < it.t1) {
      const TA* src = reinterpret_cast<const TA*>(a.a) + t * a.lda + k;
      if (Vec<TA>::N == 4) {
        load16(reinterpret_cast<const float*>(src), x[u]);
      } else {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
        x[u][0] = __uint_as_float(w.x << 16); x[u][1] = __uint_as_float(w.x & 0xFFFF0000u);
        x[u][2] = __uint_as_float(w.y << 16); x[u][3] = __uint_as_float(w.y & 0xFFFF0000u);
      }
    } else {
      x[u][0] = x[u][1] = x[u][2] = x[u][3] = 0.f;
    }
  }
  if (kin && a.colscale) {
    const float4 c4 = __ldg(reinterpret_cast<const float4*>(a.colscale + k));
#pragma unroll
    for (int u = 0; u < kRdTok; ++u) { x[u][0] *= c4.x; x[u][1] *= c4.y; x[u][2] *= c4.z; x[u][3] *= c4.w; }
  }
  if (Vec<TA>::N == 4 && kin && a.split_hi) write_split(a, x, tg, it.t1, k);
  if (kok && a.mask) {
#pragma unroll
    for (int u = 0; u < kRdTok; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (tg + u < it.t1 && !drop_keep(a.drop, tg + u, k + e)) x[u][e] = 0.f;
  }
  float v[V];
#pragma unroll
  for (int u = 0; u < kRdTok; ++u)
#pragma unroll
    for (int j = 0; j < R; ++j)
      v[u * R + j] = fmaf(x[u][0], sv[j][0], fmaf(x[u][1], sv[j][1], fmaf(x[u][2], sv[j][2], x[u][3] * sv[j][3])));
  warp_halving_sum<V>(v, lane);
#pragma unroll
  for (int i = 0; i < V / 32; ++i) red[warp][lane * (V / 32) + i] = v[i];
  __syncthreads();
  for (int idx = threadIdx.x; idx < V; idx += 256) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) acc += red[w][idx];
    const int u = idx / R, j = idx - u * R;
    const int64_t t = tg + u;
    if (t < it.t1) part[((int64_t)kc * a.T + t) * R + j] = acc;
  }
}

// out[t, j] = alpha_slot * sum_kc part[kc][t][j] for j < r_slot, 0 for r_slot <= j < ldo
template <int R>
__global__ void k_rowdot_finish(const RowDotArgs a, const float* __restrict__ part, int nkc) {
  grid_dep_sync();
  const int item = blockIdx.x;
  TokenItem it;
  if (!get_item(a.items, a.n_items, item, a.T, it)) return;
  const int32_t r = it.slot >= 0 ? a.rank[it.slot] : 0;
  const float alpha = it.slot >= 0 ? a.alpha[it.slot] : 0.f;
  const int64_t n = (int64_t)(it.t1 - it.t0) * a.ldo;
  for (int64_t e = threadIdx.x; e < n; e += blockDim.x) {
    const int64_t t = it.t0 + e / a.ldo;
    const int j = (int)(e % a.ldo);
    float v = 0.f;
    if (j < r)
      for (int kc = 0; kc < nkc; ++kc) v += part[((int64_t)kc * a.T + t) * R + j];
    a.out[t * a.ldo + j] = (j < r) ? v * alpha : 0.f;
  }
}

constexpr int kCrTok = 32;      // tokens per CTA
constexpr int kCrCols = 512;    // columns per CTA (256 threads x 2)

// part[g][n][j] = sum over the 32 tokens of token group g (within one work item) of P[t, j] B'[t, n]
template <typename TB, int R>
__global__ void __launch_bounds__(256) k_colred_wide(const ColRedArgs a) {
  grid_dep_sync();
  __shared__ __align__(16) float sP[kCrTok * R];
  const int item = blockIdx.y / (kRedTileT / kCrTok);
  const int sub = blockIdx.y % (kRedTileT / kCrTok);
  TokenItem it;
  if (!get_item(a.items, a.n_items, item, a.T, it)) return;
  const int64_t t0 = (int64_t)it.t0 + (int64_t)sub * kCrTok;
  const int64_t n0 = (int64_t)blockIdx.x * kCrCols + threadIdx.x * 2;
  float* dst = a.part + (int64_t)blockIdx.y * a.N * a.ldpart;
  if (it.slot < 0) return;
  const int32_t r = a.rank[it.slot];
  const int nt = (int)max((int64_t)0, min((int64_t)kCrTok, (int64_t)it.t1 - t0));
  for (int e = threadIdx.x; e < kCrTok * R; e += 256) {
    const int tt = e / R, j = e - tt * R;
    sP[e] = (tt < nt && j < r) ? a.p[(t0 + tt) * a.ldp + j] : 0.f;
  }
  __syncthreads();
  if (n0 >= a.N) return;
  float acc[2][R];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int j = 0; j < R; ++j) acc[c][j] = 0.f;
  float cs0 = 1.f, cs1 = 1.f;
  if (a.colscale) { cs0 = __ldg(a.colscale + n0); cs1 = __ldg(a.colscale + n0 + 1); }
#pragma unroll 1
  for (int tb = 0; tb < kCrTok; tb += 8) {
    float b[8][2];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int tt = tb + u;
      if (tt < nt) {
        const TB* src = reinterpret_cast<const TB*>(a.b) + (t0 + tt) * a.ldb + n0;
        b[u][0] = to_f(src[0]);
        b[u][1] = to_f(src[1]);
      } else {
        b[u][0] = b[u][1] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int tt = tb + u;
      float b0 = b[u][0] * cs0, b1 = b[u][1] * cs1;
      if (a.mask && tt < nt) {
        if (!drop_keep(a.drop, t0 + tt, n0)) b0 = 0.f;
        if (!drop_keep(a.drop, t0 + tt, n0 + 1)) b1 = 0.f;
      }
#pragma unroll
      for (int j = 0; j < R; j += 4) {
        const float4 pv = *reinterpret_cast<const float4*>(&sP[tt * R + j]);
        acc[0][j] = fmaf(pv.x, b0, acc[0][j]); acc[1][j] = fmaf(pv.x, b1, acc[1][j]);
        acc[0][j + 1] = fmaf(pv.y, b0, acc[0][j + 1]); acc[1][j + 1] = fmaf(pv.y, b1, acc[1][j + 1]);
        acc[0][j + 2] = fmaf(pv.z, b0, acc[0][j + 2]); acc[1][j + 2] = fmaf(pv.z, b1, acc[1][j + 2]);
        acc[0][j + 3] = fmaf(pv.w, b0, acc[0][j + 3]); acc[1][j + 3] = fmaf(pv.w, b1, acc[1][j + 3]);
      }
    }
  }
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    float* d = dst + (n0 + c) * a.ldpart;
#pragma unroll
    for (int j = 0; j < R; ++j)
      if (j < a.ldpart) d[j] = acc[c][j];
  }
}

// ---------------------------------------------------------------------------------------------
// Single-pass forms for single-adapter calls (ranks <= 16): no partial buffers, no second launch.
// ---------------------------------------------------------------------------------------------

// two consecutive elements (8- or 4-byte aligned) as floats
__device__ __forceinline__ void load2(const float* p, float* out) {
  const float2 v = __ldg(reinterpret_cast<const float2*>(p));
  out[0] = v.x; out[1] = v.y;
}
__device__ __forceinline__ void load2(const __nv_bfloat16* p, float* out) {
  const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(p));
  out[0] = __uint_as_float(w << 16); out[1] = __uint_as_float(w & 0xFFFF0000u);
}

// Side tasks of a row-dot launch, spread over all its threads (see RowDotArgs).
__device__ __forceinline__ void rowdot_side_tasks(const RowDotArgs& a) {
  const int64_t gt = ((int64_t)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t gs = (int64_t)gridDim.x * gridDim.y * blockDim.x;
  if (a.t_src) {
    const int64_t n = a.t_rows * a.t_cols;
    for (int64_t e = gt; e < n; e += gs) {
      const int64_t r = e / a.t_cols, c = e - r * a.t_cols;
      a.t_dst[c * a.t_rows + r] = __ldg(a.t_src + e);
    }
  }
}

// S[j, k .. k + 3] (zero for j >= r) and A'[t, k .. k + 3] for the TOK tokens from tg (zero past t1)
template <typename TA, int R, int TOK>
__device__ __forceinline__ void rowdot_load(const RowDotArgs& a, const float* S, int32_t r, int64_t tg,
                                            int64_t t1, int64_t k, float (&sv)[R][4], float (&x)[TOK][4]) {
  if (a.s_rows_k) {
    // S[j, k + e] = S_store[(k + e) lds + j]: rank-contiguous rows of B
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
      for (int j4 = 0; j4 < R / 4; ++j4) {
        float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
        if (4 * j4 < r) q = __ldg(reinterpret_cast<const float4*>(S + (k + e) * a.lds + 4 * j4));
        sv[4 * j4][e] = q.x; sv[4 * j4 + 1][e] = q.y; sv[4 * j4 + 2][e] = q.z; sv[4 * j4 + 3][e] = q.w;
      }
  } else {
#pragma unroll
    for (int j = 0; j < R; ++j) {
      float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < r) q = __ldg(reinterpret_cast<const float4*>(S + (int64_t)j * a.lds + k));
      sv[j][0] = q.x; sv[j][1] = q.y; sv[j][2] = q.z; sv[j][3] = q.w;
    }
  }
#pragma unroll
  for (int u = 0; u < TOK; ++u) {
    const int64_t t = tg + u;
    if (t < t1) {
      const TA* src = reinterpret_cast<const TA*>(a.a) + t * a.lda + k;
      if (Vec<TA>::N == 4) {
        load16(reinterpret_cast<const float*>(src), x[u]);
      } else {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
        x[u][0] = __uint_as_float(w.x << 16); x[u][1] = __uint_as_float(w.x & 0xFFFF0000u);
        x[u][2] = __uint_as_float(w.y << 16); x[u][3] = __uint_as_float(w.y & 0xFFFF0000u);
      }
    } else {
      x[u][0] = x[u][1] = x[u][2] = x[u][3] = 0.f;
    }
  }
}

// out[t, j] = alpha * sum_k A'[t, k] S[j, k] for TOK tokens per CTA over the whole K (256 threads
// x 4 columns per pass, per-thread sums kept across passes), then one warp / CTA reduction. Two
// CTAs per SM (at most 128 registers): with TOK tokens per CTA the grid is several CTAs per SM,
// and one resident CTA would leave each SM waiting on a single CTA's load latency.
template <typename TA, int R, int TOK>
__global__ void __launch_bounds__(256, 2) k_rowdot_full(const RowDotArgs a) {
  grid_dep_sync();
  constexpr int V = TOK * R;
  static_assert(V % 32 == 0, "per-thread values must fill the warp reduction");
  __shared__ float red[8][V];
  rowdot_side_tasks(a);
  const int item = blockIdx.x / (kGemmTileT / TOK);
  const int grp = blockIdx.x % (kGemmTileT / TOK);
  TokenItem it;
  if (!get_item(a.items, a.n_items, item, a.T, it)) return;
  const int64_t tg = (int64_t)it.t0 + (int64_t)grp * TOK;
  if (tg >= it.t1) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = it.slot;
  const int32_t r = slot >= 0 ? a.rank[slot] : 0;
  const float* S = slot >= 0 ? a.s[slot] : nullptr;
  float v[V];
#pragma unroll
  for (int i = 0; i < V; ++i) v[i] = 0.f;
  for (int64_t k = (int64_t)threadIdx.x * 4; k < a.K; k += 1024) {
    float sv[R][4], x[TOK][4];
    rowdot_load<TA, R, TOK>(a, S, r, tg, it.t1, k, sv, x);
    if (a.colscale) {
      const float4 c4 = __ldg(reinterpret_cast<const float4*>(a.colscale + k));
#pragma unroll
      for (int u = 0; u < TOK; ++u) { x[u][0] *= c4.x; x[u][1] *= c4.y; x[u][2] *= c4.z; x[u][3] *= c4.w; }
    }
    if (Vec<TA>::N == 4 && a.split_hi) write_split(a, x, tg, it.t1, k);
    if (a.mask) {
#pragma unroll
      for (int u = 0; u < TOK; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (tg + u < it.t1 && !drop_keep(a.drop, tg + u, k + e)) x[u][e] = 0.f;
    }
#pragma unroll
    for (int u = 0; u < TOK; ++u)
#pragma unroll
      for (int j = 0; j < R; ++j)
        v[u * R + j] = fmaf(x[u][0], sv[j][0], fmaf(x[u][1], sv[j][1],
                            fmaf(x[u][2], sv[j][2], fmaf(x[u][3], sv[j][3], v[u * R + j]))));
  }
  warp_halving_sum<V>(v, lane);
#pragma unroll
  for (int i = 0; i < V / 32; ++i) red[warp][lane * (V / 32) + i] = v[i];
  __syncthreads();
  const float alpha = slot >= 0 ? a.alpha[slot] : 0.f;
  for (int idx = threadIdx.x; idx < V; idx += 256) {
    const int u = idx / R, j = idx - u * R;
    const int64_t t = tg + u;
    if (t >= it.t1 || j >= a.ldo) continue;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) acc += red[w][idx];
    a.out[t * a.ldo + j] = j < r ? acc * alpha : 0.f;
  }
}

// Thread-block cluster helpers (distributed shared memory).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// value of float `local` (a shared-memory address in this CTA's layout) in cluster CTA `rank`
__device__ __forceinline__ float ld_peer(const float* local, uint32_t rank) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(local), remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// Fused token reduction of a single-adapter call (ColRedArgs, fused form). The kColGroups CTAs of
// one 64-column block form a cluster; CTA g sums P[t, j] B'[t, n] over token group g (2 columns
// per lane; the 8 warps take every 8th token of a 128-token chunk, P rows staged in shared
// memory) and reduces its warps in warp order. Then every CTA of the cluster adds, for 8 of the
// block's columns, the groups' sums in group order (read from the peers' shared memory) into
// out, so reruns are bitwise equal and no partials leave the chip. Two reductions over the same
// tokens (dB and dA of a linear) can share a launch: grid x runs over job 0's column blocks, then
// job 1's.
struct ColRedJobs {
  ColRedArgs job[2];
  int32_t n_jobs;
  int32_t blocks0;   // job 0's 64-column blocks
};

template <typename TB, int R>
__global__ void __launch_bounds__(256) k_colred_fused(const __grid_constant__ ColRedJobs jobs) {
  grid_dep_sync();
  const int jb = (jobs.n_jobs > 1 && (int)blockIdx.x >= jobs.blocks0) ? 1 : 0;
  const ColRedArgs& a = jobs.job[jb];
  const int bx = (int)blockIdx.x - (jb ? jobs.blocks0 : 0);
  constexpr int kChunk = 128;   // tokens staged per pass (16 per warp, all loads in flight)
  constexpr int U = kChunk / 8;
  __shared__ __align__(16) float sP[kChunk * R];
  __shared__ float red[8][kColBlock * R];
  __shared__ float mine[kColBlock * R];   // this group's sums, [col][j]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t N = a.N;
  const int64_t nb = (int64_t)bx * kColBlock;
  const int64_t n0 = nb + 2 * lane;
  const bool nok = n0 < N;
  const int g = blockIdx.y;   // == rank in the cluster (cluster dims 1 x kColGroups)
  const int64_t tg = (a.T + kColGroups - 1) / kColGroups;
  const int64_t t_begin = (int64_t)g * tg;
  const int64_t t_end = min(a.T, t_begin + tg);
  const int32_t r = a.rank[0];
  float cs0 = 1.f, cs1 = 1.f;
  if (a.colscale && nok) { cs0 = __ldg(a.colscale + n0); cs1 = __ldg(a.colscale + n0 + 1); }
  float acc[2][R];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int j = 0; j < R; ++j) acc[c][j] = 0.f;
  for (int64_t c0 = t_begin; c0 < t_end; c0 += kChunk) {
    const int nt = (int)min((int64_t)kChunk, t_end - c0);
    // B' loads first, so that they are in flight while P is staged
    float b[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int tt = warp + 8 * u;
      b[u][0] = b[u][1] = 0.f;
      if (nok && tt < nt) load2(reinterpret_cast<const TB*>(a.b) + (c0 + tt) * a.ldb + n0, b[u]);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kChunk * R; e += 256) {
      const int tt = e / R, j = e - tt * R;
      sP[e] = (tt < nt && j < r) ? __ldg(a.p + (c0 + tt) * a.ldp + j) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int tt = warp + 8 * u;
      b[u][0] *= cs0;
      b[u][1] *= cs1;
      if (a.mask && nok && tt < nt) {
        if (!drop_keep(a.drop, c0 + tt, n0)) b[u][0] = 0.f;
        if (!drop_keep(a.drop, c0 + tt, n0 + 1)) b[u][1] = 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float* pr = sP + (warp + 8 * u) * R;   // zero rows past the chunk's tokens
#pragma unroll
      for (int j = 0; j < R; j += 4) {
        const float4 pv = *reinterpret_cast<const float4*>(pr + j);
        acc[0][j] = fmaf(pv.x, b[u][0], acc[0][j]); acc[1][j] = fmaf(pv.x, b[u][1], acc[1][j]);
        acc[0][j + 1] = fmaf(pv.y, b[u][0], acc[0][j + 1]); acc[1][j + 1] = fmaf(pv.y, b[u][1], acc[1][j + 1]);
        acc[0][j + 2] = fmaf(pv.z, b[u][0], acc[0][j + 2]); acc[1][j + 2] = fmaf(pv.z, b[u][1], acc[1][j + 2]);
        acc[0][j + 3] = fmaf(pv.w, b[u][0], acc[0][j + 3]); acc[1][j + 3] = fmaf(pv.w, b[u][1], acc[1][j + 3]);
      }
    }
  }
  // reduce the 8 warps in warp order: red[w][j][col] (column-minor, conflict-free)
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int j = 0; j < R; ++j) red[warp][j * kColBlock + 2 * lane + c] = acc[c][j];
  __syncthreads();
  for (int e = threadIdx.x; e < kColBlock * R; e += 256) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += red[w][e];
    mine[e] = sum;
  }
  cluster_sync();
  // this CTA's share of the block: columns [g * 8, g * 8 + 8), all j; groups summed in order
  constexpr int kShare = kColBlock / kColGroups;
  for (int e = threadIdx.x; e < kShare * R; e += 256) {
    const int jj = e / kShare, cc = e - jj * kShare;
    const int col = g * kShare + cc;
    const int64_t n = nb + col;
    if (n < N && jj < r) {
      float sum = 0.f;
      for (int gg = 0; gg < kColGroups; ++gg) sum += ld_peer(&mine[jj * kColBlock + col], (uint32_t)gg);
      float* o = a.out_transposed ? a.out + (int64_t)jj * N + n : a.out + n * a.ldpart + jj;
      *o += sum;
    }
  }
  cluster_sync();   // peers' shared memory stays alive until every CTA has read it
}

template <typename TA>
cudaError_t rowdot_for_rank(const RowDotArgs& a, int max_items, cudaStream_t st) {
  const int rm = a.max_rank;
  if (rm <= 4) rowdot_launch<TA, 4>(a, max_items, st);
  else if (rm <= 8) rowdot_launch<TA, 8>(a, max_items, st);
  else if (rm <= 16) rowdot_launch<TA, 16>(a, max_items, st);
  else if (rm <= 32) rowdot_launch<TA, 32>(a, max_items, st);
  else rowdot_launch<TA, 64>(a, max_items, st);
  return cudaGetLastError();
}

template <typename TB>
cudaError_t colred_for_rank(const ColRedArgs& a, int max_items, cudaStream_t st) {
  const int rm = a.max_rank;
  auto grid = [&](int cpt) {
    return dim3((unsigned)((a.N + (int64_t)kColThreads * cpt - 1) / ((int64_t)kColThreads * cpt)),
                (unsigned)max_items);
  };
  if (rm <= 4) launch_kernel(k_colred<TB, 4, 1>, grid(1), kColThreads, 0, st, a);
  else if (rm <= 8) launch_kernel(k_colred<TB, 8, 1>, grid(1), kColThreads, 0, st, a);
  else if (rm <= 16) launch_kernel(k_colred<TB, 16, 1>, grid(1), kColThreads, 0, st, a);
  else if (rm <= 32) launch_kernel(k_colred<TB, 32, 1>, grid(1), kColThreads, 0, st, a);
  else launch_kernel(k_colred<TB, 64, 1>, grid(1), kColThreads, 0, st, a);
  return cudaGetLastError();
}

}  // namespace

template <typename TA, int R>
cudaError_t rowdot_wide(const RowDotArgs& a, int max_items, cudaStream_t st, int prof_kind) {
  const int nkc = (int)((a.K + kRdCols - 1) / kRdCols);
  dim3 grid((unsigned)(max_items * (kGemmTileT / kRdTok)), (unsigned)nkc);
  prof_begin(prof_kind, st);
  launch_kernel(k_rowdot_wide<TA, R>, grid, 256, 0, st, a, a.part);
  prof_end(prof_kind, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prof_begin(0, st);
  launch_kernel(k_rowdot_finish<R>, (unsigned)max_items, 256, 0, st, a, a.part, nkc);
  return cudaGetLastError();
}

template <typename TA, int R, int TOK>
cudaError_t rowdot_full(const RowDotArgs& a, int max_items, cudaStream_t st, int prof_kind) {
  prof_begin(prof_kind, st);
  launch_kernel(k_rowdot_full<TA, R, TOK>, (unsigned)(max_items * (kGemmTileT / TOK)), 256, 0, st, a);
  prof_end(prof_kind, st);
  return cudaGetLastError();
}

cudaError_t launch_rowdot(int dtype, const RowDotArgs& a, int max_items, cudaStream_t st,
                          int prof_kind) {
  if (max_items <= 0) return cudaSuccess;
  const bool side = a.t_src != nullptr;
  if (a.single_pass && a.max_rank <= 16) {
    const bool f = dtype == LORA_F32;
    if (a.max_rank <= 4)
      return f ? rowdot_full<float, 4, 8>(a, max_items, st, prof_kind)
               : rowdot_full<__nv_bfloat16, 4, 8>(a, max_items, st, prof_kind);
    if (a.max_rank <= 8)
      return f ? rowdot_full<float, 8, 4>(a, max_items, st, prof_kind)
               : rowdot_full<__nv_bfloat16, 8, 4>(a, max_items, st, prof_kind);
    return f ? rowdot_full<float, 16, 2>(a, max_items, st, prof_kind)
             : rowdot_full<__nv_bfloat16, 16, 2>(a, max_items, st, prof_kind);
  }
  if (side || a.s_rows_k) return cudaErrorInvalidValue;   // only the single-pass form has these
  if (a.part && a.max_rank <= 16 && (a.K % 4) == 0) {
    const bool f = dtype == LORA_F32;
    if (a.max_rank <= 4)
      return f ? rowdot_wide<float, 4>(a, max_items, st, prof_kind)
               : rowdot_wide<__nv_bfloat16, 4>(a, max_items, st, prof_kind);
    if (a.max_rank <= 8)
      return f ? rowdot_wide<float, 8>(a, max_items, st, prof_kind)
               : rowdot_wide<__nv_bfloat16, 8>(a, max_items, st, prof_kind);
    return f ? rowdot_wide<float, 16>(a, max_items, st, prof_kind)
             : rowdot_wide<__nv_bfloat16, 16>(a, max_items, st, prof_kind);
  }
  prof_begin(prof_kind, st);
  cudaError_t e = dtype == LORA_F32 ? rowdot_for_rank<float>(a, max_items, st)
                                    : rowdot_for_rank<__nv_bfloat16>(a, max_items, st);
  prof_end(prof_kind, st);
  return e;
}

namespace {
// the fused single-adapter form of one or two jobs (ranks <= 16, same rank, T and dtype)
cudaError_t colred_fused(int dtype, const ColRedArgs* js, int n_jobs, cudaStream_t st,
                         int prof_kind) {
  const ColRedArgs& a = js[0];
  if (a.T <= 0) return cudaSuccess;
  if (a.max_rank > 16) return cudaErrorInvalidValue;
  ColRedJobs jobs{};
  unsigned blocks = 0;
  for (int q = 0; q < n_jobs; ++q) {
    jobs.job[q] = js[q];
    blocks += (unsigned)((js[q].N + kColBlock - 1) / kColBlock);
  }
  jobs.n_jobs = n_jobs;
  jobs.blocks0 = (int32_t)((a.N + kColBlock - 1) / kColBlock);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(blocks, (unsigned)kColGroups);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = kColGroups;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = add_pdl_attr(attr, 1);
  cudaError_t e;
  prof_begin(prof_kind, st);
  if (dtype == LORA_F32) {
    if (a.max_rank <= 4) e = cudaLaunchKernelEx(&cfg, k_colred_fused<float, 4>, jobs);
    else if (a.max_rank <= 8) e = cudaLaunchKernelEx(&cfg, k_colred_fused<float, 8>, jobs);
    else e = cudaLaunchKernelEx(&cfg, k_colred_fused<float, 16>, jobs);
  } else {
    if (a.max_rank <= 4) e = cudaLaunchKernelEx(&cfg, k_colred_fused<__nv_bfloat16, 4>, jobs);
    else if (a.max_rank <= 8) e = cudaLaunchKernelEx(&cfg, k_colred_fused<__nv_bfloat16, 8>, jobs);
    else e = cudaLaunchKernelEx(&cfg, k_colred_fused<__nv_bfloat16, 16>, jobs);
  }
  prof_end(prof_kind, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}
}  // namespace

cudaError_t launch_colred2(int dtype, const ColRedArgs& a, const ColRedArgs& b, cudaStream_t st,
                           int prof_kind) {
  if (!a.out || !b.out || a.T != b.T || a.max_rank != b.max_rank) return cudaErrorInvalidValue;
  const ColRedArgs js[2] = {a, b};
  return colred_fused(dtype, js, 2, st, prof_kind);
}

cudaError_t launch_colred(int dtype, const ColRedArgs& a, int max_items, cudaStream_t st,
                          int prof_kind) {
  if (a.out) return colred_fused(dtype, &a, 1, st, prof_kind);
  if (max_items <= 0) return cudaSuccess;
  // the partial layout must match what the caller reduces: kRedTileT / kCrTok partials per item
  // from the wide kernel (ranks <= 16), one per item otherwise
  if (a.sub_groups != (a.max_rank <= 16 ? kRedTileT / kCrTok : 1)) return cudaErrorInvalidValue;
  if (a.max_rank <= 16) {
    dim3 grid((unsigned)((a.N + kCrCols - 1) / kCrCols), (unsigned)(max_items * a.sub_groups));
    prof_begin(prof_kind, st);
    if (dtype == LORA_F32) {
      if (a.max_rank <= 4) launch_kernel(k_colred_wide<float, 4>, grid, 256, 0, st, a);
      else if (a.max_rank <= 8) launch_kernel(k_colred_wide<float, 8>, grid, 256, 0, st, a);
      else launch_kernel(k_colred_wide<float, 16>, grid, 256, 0, st, a);
    } else {
      if (a.max_rank <= 4) launch_kernel(k_colred_wide<__nv_bfloat16, 4>, grid, 256, 0, st, a);
      else if (a.max_rank <= 8) launch_kernel(k_colred_wide<__nv_bfloat16, 8>, grid, 256, 0, st, a);
      else launch_kernel(k_colred_wide<__nv_bfloat16, 16>, grid, 256, 0, st, a);
    }
    prof_end(prof_kind, st);
    return cudaGetLastError();
  }
  prof_begin(prof_kind, st);
  cudaError_t e = dtype == LORA_F32 ? colred_for_rank<float>(a, max_items, st)
                                    : colred_for_rank<__nv_bfloat16>(a, max_items, st);
  prof_end(prof_kind, st);
  return e;
}

}  // namespace lora
