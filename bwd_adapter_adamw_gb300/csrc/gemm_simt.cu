// SIMT (CUDA-core) tiled products of the LoRA-linear step.
//
// tok_gemm:  out[t, n] = alpha * ( [mask(t,n)] * sum_j P[t,j] Q_slot[n,j]  +  sum_k A[t,k] B[n,k] ) * cs[n]
//            for the tokens of one work item (<= 128 tokens of one adapter slot). Both operands are
//            K-contiguous. Used for the frozen forward (X W^T with the up-projection Hs B^T as
//            extra K-steps), the frozen dX (dY' W via W^T, with the masked Gs A term), the shrink
//            (Xd A^T) and G (dY' B via B^T).
// red_gemm:  part[item][m, j] = sum_{t in item} A[t, m] * Bv[t, j]: the token reductions of dB
//            (dY'^T Hs) and dA^T (Xd^T Gs), one partial per work item, reduced in item order
//            afterwards so that every rerun is bitwise identical.
//
// ("Backward Bug Hunts and Vulkan Tiled GEMM", The fix: a 16x16 shared-memory tiled GEMM -- the
// pages stage 16x16 tiles of both operands in shared memory per K chunk. Here each 256-thread CTA
// stages 128 x 16 tiles, double-buffered, and every thread accumulates an 8 x 8 register block.)
#include "lora_kernels.h"

namespace lora {

namespace {

constexpr int BM = 128;
constexpr int BK = 16;
constexpr int PAD = 4;

template <int BN>
struct Smem {
  float a[2][BK][BM + PAD];
  float b[2][BK][BN + PAD];
};

// Operand description resolved per CTA.
struct OpRef {
  const void* p;        // stored tensor base
  int64_t ld;           // elements between stored rows
  int64_t row_begin;    // K-major: first M/N row; M-major: first token (K)
  int64_t row_end;      // exclusive
  int64_t col_end;      // K-major: K extent; M-major: M/N extent
  const float* colscale;  // multiply by colscale[stored column]
  int mask;               // dropout keep(token, input column)
  int token_is_row;       // for the mask: stored rows are tokens (both layouts use tokens as rows)
};

// K-major tile loader: ROWS operand rows x BK columns of K, converted to float.
template <typename T, int ROWS>
struct KLoad {
  static constexpr int VEC = Vec<T>::N;
  static constexpr int VPR = BK / VEC;
  static constexpr int NV = ROWS * VPR;
  static constexpr int PT = (NV + 255) / 256;
  float v[PT][VEC];

  __device__ __forceinline__ void load(const OpRef& o, int64_t row0, int64_t k0, const DropParams& dp) {
#pragma unroll
    for (int j = 0; j < PT; ++j) {
      const int idx = threadIdx.x + j * 256;
      const int r = idx / VPR;
      const int kv = (idx % VPR) * VEC;
      const int64_t row = row0 + r;
      const int64_t k = k0 + kv;
      if (idx < NV && row < o.row_end && k < o.col_end) {
        load16(reinterpret_cast<const T*>(o.p) + row * o.ld + k, v[j]);
        if (o.colscale) {
#pragma unroll
          for (int e = 0; e < VEC; ++e) v[j][e] *= __ldg(o.colscale + k + e);
        }
        if (o.mask) {
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            if (!drop_keep(dp, row, k + e)) v[j][e] = 0.f;
        }
      } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) v[j][e] = 0.f;
      }
    }
  }
  template <int LD>
  __device__ __forceinline__ void store(float (*s)[LD]) const {
#pragma unroll
    for (int j = 0; j < PT; ++j) {
      const int idx = threadIdx.x + j * 256;
      if (idx < NV) {
        const int r = idx / VPR;
        const int kv = (idx % VPR) * VEC;
#pragma unroll
        for (int e = 0; e < VEC; ++e) s[kv + e][r] = v[j][e];
      }
    }
  }
};

// M-major tile loader: BK stored rows (tokens) x ROWS contiguous columns.
template <typename T, int ROWS>
struct MLoad {
  static constexpr int VEC = Vec<T>::N;
  static constexpr int VPR = ROWS / VEC;
  static constexpr int NV = BK * VPR;
  static constexpr int PT = (NV + 255) / 256;
  float v[PT][VEC];

  __device__ __forceinline__ void load(const OpRef& o, int64_t col0, int64_t t0, const DropParams& dp) {
#pragma unroll
    for (int j = 0; j < PT; ++j) {
      const int idx = threadIdx.x + j * 256;
      const int kr = idx / VPR;
      const int cv = (idx % VPR) * VEC;
      const int64_t t = t0 + kr;
      const int64_t c = col0 + cv;
      if (idx < NV && t < o.row_end && c < o.col_end) {
        load16(reinterpret_cast<const T*>(o.p) + t * o.ld + c, v[j]);
        if (o.colscale) {
#pragma unroll
          for (int e = 0; e < VEC; ++e) v[j][e] *= __ldg(o.colscale + c + e);
        }
        if (o.mask) {
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            if (!drop_keep(dp, t, c + e)) v[j][e] = 0.f;
        }
      } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) v[j][e] = 0.f;
      }
    }
  }
  template <int LD>
  __device__ __forceinline__ void store(float (*s)[LD]) const {
#pragma unroll
    for (int j = 0; j < PT; ++j) {
      const int idx = threadIdx.x + j * 256;
      if (idx < NV) {
        const int kr = idx / VPR;
        const int cv = (idx % VPR) * VEC;
#pragma unroll
        for (int e = 0; e < VEC; ++e) s[kr][cv + e] = v[j][e];
      }
    }
  }
};

// Accumulator of one thread's 8 x TN outputs. COMP: every 16-wide K-tile is summed into fresh
// registers and the tile sums are added with Knuth's TwoSum, carrying the rounding error in
// `comp`, so that the long reductions of the skinny products (K = in, out or a token range)
// lose no more than one tile's worth of fp32 rounding.
template <int TN, bool COMP>
struct Acc {
  float v[8][TN];
  float c[8][TN];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) v[i][j] = 0.f, c[i][j] = 0.f;
  }
  __device__ __forceinline__ float get(int i, int j) const { return COMP ? v[i][j] + c[i][j] : v[i][j]; }
  __device__ __forceinline__ void scale(int i, int j, float s) { v[i][j] *= s; c[i][j] *= s; }
};

template <int BN, bool COMP>
__device__ __forceinline__ void mma_tile(Acc<BN / 16, COMP>& acc, const float (*sa)[BM + PAD],
                                         const float (*sb)[BN + PAD]) {
  constexpr int TN = BN / 16;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float t[8][TN];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) t[i][j] = COMP ? 0.f : acc.v[i][j];
#pragma unroll
  for (int kk = 0; kk < BK; ++kk) {
    float a[8], b[TN];
    *reinterpret_cast<float4*>(&a[0]) = *reinterpret_cast<const float4*>(&sa[kk][ty * 4]);
    *reinterpret_cast<float4*>(&a[4]) = *reinterpret_cast<const float4*>(&sa[kk][64 + ty * 4]);
    *reinterpret_cast<float4*>(&b[0]) = *reinterpret_cast<const float4*>(&sb[kk][tx * 4]);
    if (TN == 8)
      *reinterpret_cast<float4*>(&b[4]) = *reinterpret_cast<const float4*>(&sb[kk][64 + tx * 4]);
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) t[i][j] = fmaf(a[i], b[j], t[i][j]);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      if (COMP) {
        const float s = __fadd_rn(acc.v[i][j], t[i][j]);
        const float bp = __fsub_rn(s, acc.v[i][j]);
        const float err = __fadd_rn(__fsub_rn(acc.v[i][j], __fsub_rn(s, bp)), __fsub_rn(t[i][j], bp));
        acc.v[i][j] = s;
        acc.c[i][j] = __fadd_rn(acc.c[i][j], err);
      } else {
        acc.v[i][j] = t[i][j];
      }
    }
}

// Double-buffered main loop over K-major operands (rows along M for A, along N for B).
template <typename TA, typename TB, int BN, bool COMP>
__device__ void loop_kk(Acc<BN / 16, COMP>& acc, Smem<BN>& sm, const OpRef& a, int64_t m0,
                        const OpRef& b, int64_t n0, int64_t K, const DropParams& dp) {
  const int ntiles = (int)((K + BK - 1) / BK);
  if (ntiles <= 0) return;
  KLoad<TA, BM> la;
  KLoad<TB, BN> lb;
  la.load(a, m0, 0, dp);
  lb.load(b, n0, 0, dp);
  la.store(sm.a[0]);
  lb.store(sm.b[0]);
  __syncthreads();
  for (int t = 0; t < ntiles; ++t) {
    const int cur = t & 1;
    if (t + 1 < ntiles) {
      la.load(a, m0, (int64_t)(t + 1) * BK, dp);
      lb.load(b, n0, (int64_t)(t + 1) * BK, dp);
    }
    mma_tile<BN, COMP>(acc, sm.a[cur], sm.b[cur]);
    if (t + 1 < ntiles) {
      la.store(sm.a[cur ^ 1]);
      lb.store(sm.b[cur ^ 1]);
    }
    __syncthreads();
  }
}

// Double-buffered main loop over M-major operands: K = tokens [t0, t1).
template <typename TA, typename TB, int BN, bool COMP>
__device__ void loop_mm(Acc<BN / 16, COMP>& acc, Smem<BN>& sm, const OpRef& a, int64_t m0,
                        const OpRef& b, int64_t n0, int64_t t0, int64_t t1, const DropParams& dp) {
  const int ntiles = (int)((t1 - t0 + BK - 1) / BK);
  if (ntiles <= 0) return;
  MLoad<TA, BM> la;
  MLoad<TB, BN> lb;
  la.load(a, m0, t0, dp);
  lb.load(b, n0, t0, dp);
  la.store(sm.a[0]);
  lb.store(sm.b[0]);
  __syncthreads();
  for (int t = 0; t < ntiles; ++t) {
    const int cur = t & 1;
    if (t + 1 < ntiles) {
      la.load(a, m0, t0 + (int64_t)(t + 1) * BK, dp);
      lb.load(b, n0, t0 + (int64_t)(t + 1) * BK, dp);
    }
    mma_tile<BN, COMP>(acc, sm.a[cur], sm.b[cur]);
    if (t + 1 < ntiles) {
      la.store(sm.a[cur ^ 1]);
      lb.store(sm.b[cur ^ 1]);
    }
    __syncthreads();
  }
}

__device__ __forceinline__ int row_of(int i) { return (i < 4) ? ((threadIdx.x >> 4) * 4 + i) : (64 + (threadIdx.x >> 4) * 4 + i - 4); }

template <typename TA, typename TB, typename TOUT, int BN>
__global__ void __launch_bounds__(256) k_tok_gemm(const TokGemmArgs args) {
  __shared__ __align__(16) Smem<BN> sm;
  const int item = blockIdx.y;
  if (item >= *args.n_items) return;
  const TokenItem it = args.items[item];
  const int slot = it.slot;
  const int64_t m0 = it.t0;
  const int64_t n0 = (int64_t)blockIdx.x * BN;
  constexpr int TN = BN / 16;
  constexpr bool COMP = (BN == 64);
  Acc<TN, COMP> acc;
  acc.zero();

  // LoRA phase: sum_j P[t, j] Q_slot[n, j] over the slot's rank (the up-projection as extra K-steps)
  if (args.lora_phase && slot >= 0) {
    OpRef p{args.lp, args.ldlp, m0, it.t1, args.lq.rank[slot], nullptr, 0, 1};
    OpRef q{args.lq.p[slot], args.lq.ld[slot], 0, args.n_rows, args.lq.rank[slot], nullptr, 0, 0};
    loop_kk<float, float, BN, COMP>(acc, sm, p, m0, q, n0, args.lq.rank[slot], args.drop);
    if (args.mask_after_lora) {
      const int tx = threadIdx.x & 15;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t m = m0 + row_of(i);
#pragma unroll
        for (int j = 0; j < TN; ++j) {
          const int64_t n = n0 + ((j < 4) ? (tx * 4 + j) : (64 + tx * 4 + j - 4));
          if (m < it.t1 && n < args.n_rows && !drop_keep(args.drop, m, n)) acc.scale(i, j, 0.f);
        }
      }
    }
  }

  // main phase: sum_k A[t, k] B[n, k]
  {
    OpRef a{args.a, args.lda, m0, it.t1, args.K, args.a_colscale, args.a_mask, 1};
    OpRef b;
    if (args.b_per_slot) {
      const int32_t rows = (slot >= 0) ? args.bslot.rank[slot] : 0;
      b = OpRef{slot >= 0 ? args.bslot.p[slot] : args.a, slot >= 0 ? args.bslot.ld[slot] : 0, 0,
                rows, args.K, nullptr, 0, 0};
    } else {
      b = OpRef{args.b, args.ldb, 0, args.n_rows, args.K, nullptr, 0, 0};
    }
    if (!(args.b_per_slot && slot < 0)) loop_kk<TA, TB, BN, COMP>(acc, sm, a, m0, b, n0, args.K, args.drop);
  }

  // epilogue
  float alpha = args.alpha;
  if (args.alpha_per_slot) alpha = (slot >= 0) ? args.bslot.alpha[slot] : 0.f;
  TOUT* out = reinterpret_cast<TOUT*>(args.out);
  const int tx = threadIdx.x & 15;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t m = m0 + row_of(i);
    if (m >= it.t1) continue;
#pragma unroll
    for (int g = 0; g < TN / 4; ++g) {
      const int64_t n = n0 + g * 64 + tx * 4;
      if (n >= args.n_out) continue;
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[e] = acc.get(i, g * 4 + e) * alpha;
        if (args.n_colscale) v[e] *= __ldg(args.n_colscale + n + e);
      }
      store4(out + m * args.ldo + n, v);
    }
  }
}

template <typename TA>
__global__ void __launch_bounds__(256) k_red_gemm(const RedGemmArgs args) {
  constexpr int BN = 64;
  __shared__ __align__(16) Smem<BN> sm;
  const int item = blockIdx.z;
  if (item >= *args.n_items) return;
  const TokenItem it = args.items[item];
  if (it.slot < 0) return;
  const int64_t m0 = (int64_t)blockIdx.y * BM;
  const int64_t n0 = (int64_t)blockIdx.x * BN;
  const int32_t nrank = args.rank[it.slot];
  Acc<4, true> acc;
  acc.zero();
  OpRef a{args.a, args.lda, it.t0, it.t1, args.M, args.a_colscale, args.a_mask, 1};
  OpRef b{args.b, args.ldb, it.t0, it.t1, nrank, nullptr, 0, 1};
  loop_mm<TA, float, BN, true>(acc, sm, a, m0, b, n0, it.t0, it.t1, args.drop);
  float* part = args.part + (int64_t)item * args.M * args.ldp;
  const int tx = threadIdx.x & 15;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t m = m0 + row_of(i);
    const int64_t n = n0 + tx * 4;
    if (m >= args.M || n >= args.ldp) continue;
    float v[4] = {acc.get(i, 0), acc.get(i, 1), acc.get(i, 2), acc.get(i, 3)};
    store4(part + m * args.ldp + n, v);
  }
}

}  // namespace

cudaError_t launch_tok_gemm(int dtype_a, int dtype_b, int dtype_out, int bn, const TokGemmArgs& a,
                            int max_items, cudaStream_t st, int prof_kind) {
  const int ntile = (int)((a.n_out + bn - 1) / bn);
  dim3 grid(ntile, max_items);
  if (max_items <= 0 || ntile <= 0) return cudaSuccess;
  if (bn == 128) {
    if (dtype_a == LORA_F32 && dtype_b == LORA_F32 && dtype_out == LORA_F32)
      { prof_begin(prof_kind, st); k_tok_gemm<float, float, float, 128><<<grid, 256, 0, st>>>(a); prof_end(prof_kind, st); }
    else if (dtype_a == LORA_BF16 && dtype_b == LORA_BF16 && dtype_out == LORA_BF16)
      { prof_begin(prof_kind, st); k_tok_gemm<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16, 128><<<grid, 256, 0, st>>>(a); prof_end(prof_kind, st); }
    else
      return cudaErrorInvalidValue;
  } else if (bn == 64) {
    if (dtype_a == LORA_F32 && dtype_b == LORA_F32 && dtype_out == LORA_F32)
      { prof_begin(prof_kind, st); k_tok_gemm<float, float, float, 64><<<grid, 256, 0, st>>>(a); prof_end(prof_kind, st); }
    else if (dtype_a == LORA_BF16 && dtype_b == LORA_F32 && dtype_out == LORA_F32)
      { prof_begin(prof_kind, st); k_tok_gemm<__nv_bfloat16, float, float, 64><<<grid, 256, 0, st>>>(a); prof_end(prof_kind, st); }
    else
      return cudaErrorInvalidValue;
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_red_gemm(int dtype_a, const RedGemmArgs& a, int max_items, cudaStream_t st,
                            int prof_kind) {
  dim3 grid((unsigned)((a.ldp + 63) / 64), (unsigned)((a.M + BM - 1) / BM), (unsigned)max_items);
  if (max_items <= 0) return cudaSuccess;
  if (dtype_a == LORA_F32)
    { prof_begin(prof_kind, st); k_red_gemm<float><<<grid, 256, 0, st>>>(a); prof_end(prof_kind, st); }
  else
    { prof_begin(prof_kind, st); k_red_gemm<__nv_bfloat16><<<grid, 256, 0, st>>>(a); prof_end(prof_kind, st); }
  return cudaGetLastError();
}

}  // namespace lora
