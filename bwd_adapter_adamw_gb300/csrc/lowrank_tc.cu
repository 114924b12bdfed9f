// Tensor-core low-rank products for bf16 activations (sm_103a): the shrink Hs = s' Xd A^T, the
// G = s' dY' B product and the token reductions dA += Gs^T Xd, dB += dY'^T Hs
// ("8. LoRA Fundamentals", How it works; "Backward Bug Hunts and Vulkan Tiled GEMM", Bug #1 and
// Bug #2: the adapter gradients as out_prod-style token reductions).
//
// The fp32 operand of each product (A, B^T, Hs or Gs) is split into bf16 hi + lo parts
// (x = hi + lo + O(2^-16 |x|)); both parts are multiplied against the exact bf16 activations, so
// the products keep fp32-level accuracy while running on kind::f16 tensor cores.
//
//  k_tc_rows: part[z][t][j] = sum_{k in split z} A[t, k] (S_slot[j, k] + S_slot[r + j, k])
//             (shrink, G). M = 128 tokens of one work item, N = NP >= 2 r (hi rows then lo
//             rows), K-major; the epilogue adds the hi and lo columns.
//  k_tc_red:  part[item][j][n] = sum_{t in item} (ST_slot[j, t] + ST_slot[r + j, t]) Bmn[t, n]
//             (dA, dB^T). M = 128 (2 r rows of the slot's transposed split), N = 256 columns of
//             dY or X (MN-major tiles), K = the item's tokens in 64-token blocks; the epilogue adds
//             the hi and lo rows.
// Both run two CTAs per SM so that one CTA's prologue and epilogue overlap the other's stream.
// Partials are combined in a fixed order by the finish kernels, so reruns are bitwise equal.
#include <cstring>
#include <mutex>

#include "tc_ptx.cuh"

namespace lora {

namespace {
using namespace tc;

constexpr int kThreads = 192;
constexpr int kBM = 128;

__device__ __forceinline__ uint16_t bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
}
__device__ __forceinline__ float bf16_val(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// ---------------------------------------------------------------------------------------------
// k_tc_rows
// ---------------------------------------------------------------------------------------------
struct RowsParams {
  CUtensorMap ta;                    // A [T, K] bf16, box {64, 128}
  CUtensorMap ts[LORA_MAX_SLOTS];    // S_slot [2 r, K] bf16, box {64, NP}
  const TokenItem* items;
  const int32_t* n_items;
  uint32_t* err;
  int32_t rank[LORA_MAX_SLOTS];
  int32_t nk;                        // K blocks in total
  int32_t nk_per_split;
  int32_t ldp;                       // partial row stride (largest rank)
  float* part;                       // [splits][T][ldp]
  int64_t T;
};

template <int NP>
struct RowsCfg {
  static constexpr int kBBytes = NP * 128;
  static constexpr int kStageBytes = 16384 + kBBytes;
  // about 100 KB of stages, so that two CTAs fit one SM
  static constexpr int kStages = (100 * 1024 / kStageBytes) < 8 ? (100 * 1024 / kStageBytes) : 8;
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 1024;
  static constexpr int kLdb = NP + 4;   // staging row stride of the epilogue (floats)
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(kBM * kLdb * 4 <= kStages * kStageBytes, "epilogue staging fits the stages");
  static constexpr uint32_t kCols = NP < 32 ? 32u : (uint32_t)NP;
  static constexpr uint32_t kIdesc = idesc(kFmtBF16, kBM, NP);
};

template <int NP>
__global__ void __launch_bounds__(kThreads, 2) k_tc_rows(const __grid_constant__ RowsParams p) {
  grid_dep_sync();
  using C = RowsCfg<NP>;
  extern __shared__ uint8_t smem_raw[];
  TokenItem it;
  if (!get_item(p.items, p.n_items, blockIdx.x, p.T, it)) return;
  const int z = blockIdx.y;
  const int kb0 = z * p.nk_per_split;
  const int kb1 = min(p.nk, kb0 + p.nk_per_split);
  float* part = p.part + (int64_t)z * p.T * p.ldp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (it.slot < 0 || kb0 >= kb1) {
    // no adapter for these tokens (or an empty split): the partial rows are zero
    float4* dst = reinterpret_cast<float4*>(part + (int64_t)it.t0 * p.ldp);
    const int n4 = (it.t1 - it.t0) * (p.ldp / 4);
    for (int e = threadIdx.x; e < n4; e += kThreads) dst[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int nk = kb1 - kb0;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(base + C::kStages * C::kStageBytes);
  uint64_t* empty_bar = full_bar + C::kStages;
  uint64_t* acc_bar = empty_bar + C::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(acc_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kCols);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % C::kStages;
        const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
        if (i >= C::kStages && !mbar_wait(&empty_bar[s], ph ^ 1u, 1u, p.err)) break;
        uint8_t* sa = base + s * C::kStageBytes;
        mbar_expect_tx(&full_bar[s], C::kStageBytes);
        tma_load_2d(sa, &p.ta, &full_bar[s], (kb0 + i) * 64, it.t0);
        tma_load_2d(sa + 16384, &p.ts[it.slot], &full_bar[s], (kb0 + i) * 64, 0);
        issued = i + 1;
      }
      for (int i = (issued > C::kStages ? issued - C::kStages : 0); i < issued; ++i)
        if (!mbar_wait(&full_bar[i % C::kStages], (uint32_t)(i / C::kStages) & 1u, 1u, p.err)) break;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < nk; ++i) {
        const int s = i % C::kStages;
        if (!mbar_wait(&full_bar[s], (uint32_t)(i / C::kStages) & 1u, 2u, p.err)) break;
        fence_after();
        const uint32_t sa = smem_u32(base + s * C::kStageBytes);
        const uint64_t da = smem_desc_sw128(sa), db = smem_desc_sw128(sa + 16384);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_f16(tmem, da + 2 * k, db + 2 * k, C::kIdesc, (i > 0 || k > 0) ? 1u : 0u);
        umma_commit(&empty_bar[s]);
      }
      umma_commit(acc_bar);
    }
  } else {
    // epilogue: the accumulator rows go through shared memory (the stages are idle once acc_bar
    // has fired), then hi + lo columns are added and the item's [n, ldp] partial block, which is
    // contiguous in memory, is written with coalesced float4 stores
    const int q = warp & 3;
    const int row = q * 32 + lane;
    float* buf = reinterpret_cast<float*>(base);
    const bool ready = __all_sync(0xffffffffu, mbar_wait(acc_bar, 0u, 4u, p.err));
    if (ready) {
      fence_after();
#pragma unroll
      for (int c = 0; c < NP / 16; ++c) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 16), v);
        float4* dst = reinterpret_cast<float4*>(buf + row * C::kLdb + c * 16);
#pragma unroll
        for (int g = 0; g < 4; ++g) dst[g] = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
      }
    }
    fence_before();
    asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
    if (ready) {
      const int r = p.rank[it.slot];
      const int r4 = r / 4, l4 = p.ldp / 4;
      const int n4 = (it.t1 - it.t0) * l4;
      float4* dst = reinterpret_cast<float4*>(part + (int64_t)it.t0 * p.ldp);
      for (int e = threadIdx.x - 64; e < n4; e += 128) {
        const int i = e / l4, c = e - i * l4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < r4) {
          const float4 h = *reinterpret_cast<const float4*>(buf + i * C::kLdb + 4 * c);
          const float4 l = *reinterpret_cast<const float4*>(buf + i * C::kLdb + r + 4 * c);
          v = make_float4(h.x + l.x, h.y + l.y, h.z + l.z, h.w + l.w);
        }
        dst[e] = v;
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, C::kCols);
  }
}

// out[t, j] = alpha_slot * sum_z part[z][t][j] for j < r, 0 for r <= j < ncols (alpha_slot = 1
// when use_alpha is 0; out may be null); ldp and ld_out are the row strides of part and out. With outT, also the transposed bf16 split that the token
// reductions take as their K-major operand:
// outT[region_slot + j][t] = hi(out[t, j]), outT[region_slot + r + j][t] = lo(out[t, j]).
// CTA (item, blockIdx.y) covers kFinishTok tokens of the item; every thread issues all of its
// loads (kFinishVec float4 groups x the splits) before the first add.
constexpr int kFinishTok = 32;
constexpr int kFinishThreads = 256;
constexpr int kFinishVec = kFinishTok * LORA_MAX_RANK / 4 / kFinishThreads;
constexpr int kMaxSplitsRows = 8;   // K splits of the rows kernel (the launcher rejects more)
__global__ void __launch_bounds__(kFinishThreads) k_rows_finish(
    const float* __restrict__ part, int32_t splits, int64_t T, int64_t ldp, int32_t ncols,
    int use_alpha,
    const TokenItem* __restrict__ items, const int32_t* __restrict__ n_items, const SlotInfo si,
    float* __restrict__ out, int64_t ld_out, float* __restrict__ out2, int64_t ld2,
    uint16_t* __restrict__ outT, int64_t ldt) {
  grid_dep_sync();
  __shared__ float tile[kFinishTok][LORA_MAX_RANK + 1];
  TokenItem it;
  if (!get_item(items, n_items, blockIdx.x, T, it)) return;
  const int64_t tb = (int64_t)it.t0 + (int64_t)blockIdx.y * kFinishTok;
  if (tb >= it.t1) return;
  const int32_t r = it.slot >= 0 ? si.rank[it.slot] : 0;
  const float alpha = !use_alpha ? 1.f : it.slot >= 0 ? si.alpha[it.slot] : 0.f;
  const int nt = (int)min((int64_t)kFinishTok, (int64_t)it.t1 - tb);
  const int c4n = ncols / 4;   // float4 groups per token: columns 0 .. ncols - 1
  const int n4 = nt * c4n;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 pz[kFinishVec][kMaxSplitsRows];
#pragma unroll
  for (int u = 0; u < kFinishVec; ++u) {
    const int q = threadIdx.x + u * kFinishThreads;
    const int i = q / c4n, c = q - i * c4n;
    const bool live = q < n4 && 4 * c < r;
    const float4* src = reinterpret_cast<const float4*>(part + (tb + i) * ldp) + c;
#pragma unroll
    for (int z = 0; z < kMaxSplitsRows; ++z)
      pz[u][z] = (live && z < splits) ? src[(int64_t)z * T * c4n] : zero;
  }
#pragma unroll
  for (int u = 0; u < kFinishVec; ++u) {
    const int q = threadIdx.x + u * kFinishThreads;
    if (q >= n4) continue;
    const int i = q / c4n, c = q - i * c4n;
    float4 v = zero;
    if (4 * c < r) {
#pragma unroll
      for (int z = 0; z < kMaxSplitsRows; ++z)
        if (z < splits) {
          v.x += pz[u][z].x;
          v.y += pz[u][z].y;
          v.z += pz[u][z].z;
          v.w += pz[u][z].w;
        }
      v = make_float4(v.x * alpha, v.y * alpha, v.z * alpha, v.w * alpha);
      tile[i][4 * c] = v.x;
      tile[i][4 * c + 1] = v.y;
      tile[i][4 * c + 2] = v.z;
      tile[i][4 * c + 3] = v.w;
    }
    if (out) reinterpret_cast<float4*>(out + (tb + i) * ld_out)[c] = v;
    if (out2 && 4 * c < r)   // the slot-expanded copy: the slot's own column block
      reinterpret_cast<float4*>(out2 + (tb + i) * ld2 + si.pcol[it.slot])[c] = v;
  }
  if (!outT || it.slot < 0) return;   // uniform over the CTA
  __syncthreads();
  uint16_t* d = outT + (int64_t)si.region[it.slot] * ldt + tb;
  for (int e = threadIdx.x; e < nt * r; e += kFinishThreads) {
    const int j = e / nt, i = e - j * nt;
    const float x = tile[i][j];
    const uint16_t hb = bf16_bits(x);
    d[(int64_t)j * ldt + i] = hb;
    d[(int64_t)(r + j) * ldt + i] = bf16_bits(x - bf16_val(hb));
  }
}

// ---------------------------------------------------------------------------------------------
// k_tc_red
// ---------------------------------------------------------------------------------------------
struct RedParams {
  CUtensorMap tst[LORA_MAX_SLOTS];   // ST_slot [2 r, T] bf16 (tokens contiguous), box {64, 128}
  CUtensorMap tb;                    // B [T, N] bf16, box {64 (n), 64 (t)}
  const TokenItem* items;
  const int32_t* n_items;
  uint32_t* err;
  int32_t rank[LORA_MAX_SLOTS];
  int32_t rstride;                   // partial rows per item (largest rank)
  float* part;                       // [items][rstride][N]
  int64_t N;
  int64_t T;
  int64_t span;                      // tokens per uniform item (null item table)
};

constexpr int kRedBN = 256;
constexpr int kRedStageBytes = 16384 + 32768;
constexpr int kRedStages = 2;       // about 100 KB of stages, so that two CTAs fit one SM
constexpr int kRedSmem = kRedStages * kRedStageBytes + 1024 + 1024;
constexpr int kRedHalf = kRedBN / 2;   // epilogue columns staged per pass
constexpr int kRedLdb = kRedHalf + 4;
static_assert(kBM * kRedLdb * 4 <= kRedStages * kRedStageBytes, "epilogue staging fits the stages");
constexpr uint32_t kRedIdesc = idesc(kFmtBF16, kBM, kRedBN, false, true);

__global__ void __launch_bounds__(kThreads, 2) k_tc_red(const __grid_constant__ RedParams p) {
  grid_dep_sync();
  extern __shared__ uint8_t smem_raw[];
  const int item = blockIdx.y;
  TokenItem it;
  if (!get_span_item(p.items, p.n_items, item, p.T, p.span, it)) return;
  if (it.slot < 0) return;
  const int32_t n0 = blockIdx.x * kRedBN;
  const int32_t tb0 = it.t0 & ~63;                  // 64-token blocks covering [t0, t1)
  const int nk = (it.t1 - tb0 + 63) / 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(base + kRedStages * kRedStageBytes);
  uint64_t* empty_bar = full_bar + kRedStages;
  uint64_t* acc_bar = empty_bar + kRedStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRedStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(acc_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, 256u);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % kRedStages;
        const uint32_t ph = (uint32_t)(i / kRedStages) & 1u;
        if (i >= kRedStages && !mbar_wait(&empty_bar[s], ph ^ 1u, 1u, p.err)) break;
        uint8_t* sa = base + s * kRedStageBytes;
        mbar_expect_tx(&full_bar[s], kRedStageBytes);
        const int32_t t = tb0 + i * 64;
        tma_load_2d(sa, &p.tst[it.slot], &full_bar[s], t, 0);
#pragma unroll
        for (int b = 0; b < 4; ++b) tma_load_2d(sa + 16384 + b * 8192, &p.tb, &full_bar[s], n0 + 64 * b, t);
        issued = i + 1;
      }
      for (int i = (issued > kRedStages ? issued - kRedStages : 0); i < issued; ++i)
        if (!mbar_wait(&full_bar[i % kRedStages], (uint32_t)(i / kRedStages) & 1u, 1u, p.err)) break;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < nk; ++i) {
        const int s = i % kRedStages;
        if (!mbar_wait(&full_bar[s], (uint32_t)(i / kRedStages) & 1u, 2u, p.err)) break;
        fence_after();
        const uint32_t sa = smem_u32(base + s * kRedStageBytes);
        const uint64_t da = smem_desc_sw128(sa);
        const uint64_t db = smem_desc_sw128_mn(sa + 16384, 8192);
        // K step of 16 tokens: +32 bytes in the K-major A rows, +2 KB (two 8-row atoms) in B
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_f16(tmem, da + 2 * k, db + 128 * k, kRedIdesc, (i > 0 || k > 0) ? 1u : 0u);
        umma_commit(&empty_bar[s]);
      }
      umma_commit(acc_bar);
    }
  } else {
    // epilogue, in two passes of 128 columns: the accumulator rows go through shared memory (the
    // stages are idle once acc_bar has fired), then row j (hi) and row r + j (lo) are added and
    // written along n with coalesced float4 stores
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int r = p.rank[it.slot];
    float* buf = reinterpret_cast<float*>(base);
    float* part = p.part + (int64_t)item * p.rstride * p.N;
    const bool ready = __all_sync(0xffffffffu, mbar_wait(acc_bar, 0u, 4u, p.err));
    if (ready) fence_after();
    for (int h = 0; h < kRedBN / kRedHalf; ++h) {
      if (ready) {
#pragma unroll
        for (int c = 0; c < kRedHalf / 32; ++c) {
          float v[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * kRedHalf + c * 32), v);
          float4* dst = reinterpret_cast<float4*>(buf + row * kRedLdb + c * 32);
#pragma unroll
          for (int g = 0; g < 8; ++g) dst[g] = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (ready) {
        constexpr int kC4 = kRedHalf / 4;
        for (int e = threadIdx.x - 64; e < r * kC4; e += 128) {
          const int j = e / kC4, c = e - j * kC4;
          const int64_t nb = (int64_t)n0 + h * kRedHalf + 4 * c;
          if (nb + 4 <= p.N) {
            const float4 hi = *reinterpret_cast<const float4*>(buf + j * kRedLdb + 4 * c);
            const float4 lo = *reinterpret_cast<const float4*>(buf + (r + j) * kRedLdb + 4 * c);
            *reinterpret_cast<float4*>(part + (int64_t)j * p.N + nb) =
                make_float4(hi.x + lo.x, hi.y + lo.y, hi.z + lo.z, hi.w + lo.w);
          }
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");   // the staging rows are reused next pass
    }
    fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, 256u);
  }
}

// dst_slot += sum over the slot's items (in item order) of their partial rows:
// transposed == 0: dst[j * N + n] (dA [r, N]); transposed == 1: dst[n * r + j] (dB [N, r]).
// The slot's items are contiguous in the table, from counts[1 + slot] to counts[2 + slot] (a null
// table is the uniform runs of a single-adapter call, all of slot 0). CTA (blockIdx.x, slot)
// covers kRedFinCols columns; each thread holds kRedFinVec float4 groups and loads four items'
// partials before adding them.
constexpr int kRedFinCols = 32;
constexpr int kRedFinC4 = kRedFinCols / 4;
constexpr int kRedFinVec = LORA_MAX_RANK * kRedFinC4 / kFinishThreads;
__global__ void __launch_bounds__(kFinishThreads) k_red_finish(
    const float* __restrict__ part, const TokenItem* __restrict__ items,
    const int32_t* __restrict__ counts, int64_t N, int32_t rstride, int transposed,
    const ReduceTab tab, int64_t T, int64_t span) {
  grid_dep_sync();
  __shared__ float tile[kRedFinCols][LORA_MAX_RANK + 1];
  const int slot = blockIdx.y;
  const int32_t r = tab.rank[slot];
  float* dst = tab.out[slot];
  int32_t i0 = 0, i1 = 0;
  if (items) {
    i0 = counts[1 + slot];
    i1 = counts[2 + slot];
  } else if (slot == 0) {
    i1 = (int32_t)((T + span - 1) / span);
  }
  if (i1 <= i0) return;
  const int64_t n0 = (int64_t)blockIdx.x * kRedFinCols;
  const int nc = (int)min((int64_t)kRedFinCols, N - n0);
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 acc[kRedFinVec];
  int64_t off[kRedFinVec];
  bool live[kRedFinVec];
#pragma unroll
  for (int u = 0; u < kRedFinVec; ++u) {
    const int q = threadIdx.x + u * kFinishThreads;
    const int j = q / kRedFinC4, c = q - j * kRedFinC4;
    live[u] = j < r && 4 * c < nc;
    off[u] = (int64_t)j * N + n0 + 4 * c;
    acc[u] = zero;
  }
  const int64_t istride = (int64_t)rstride * N;
  for (int32_t i = i0; i < i1; i += 4) {
    float4 v[4][kRedFinVec];
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int u = 0; u < kRedFinVec; ++u)
        v[k][u] = (live[u] && i + k < i1)
                      ? *reinterpret_cast<const float4*>(part + (int64_t)(i + k) * istride + off[u])
                      : zero;
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int u = 0; u < kRedFinVec; ++u)
        if (i + k < i1) {
          acc[u].x += v[k][u].x;
          acc[u].y += v[k][u].y;
          acc[u].z += v[k][u].z;
          acc[u].w += v[k][u].w;
        }
  }
  if (!transposed) {
#pragma unroll
    for (int u = 0; u < kRedFinVec; ++u) {
      if (!live[u]) continue;
      float4* p = reinterpret_cast<float4*>(dst + off[u]);
      float4 d = *p;
      d.x += acc[u].x;
      d.y += acc[u].y;
      d.z += acc[u].z;
      d.w += acc[u].w;
      *p = d;
    }
    return;
  }
  // dB [N, r]: through shared memory so that the row-major writes are coalesced
#pragma unroll
  for (int u = 0; u < kRedFinVec; ++u) {
    if (!live[u]) continue;
    const int q = threadIdx.x + u * kFinishThreads;
    const int j = q / kRedFinC4, c = q - j * kRedFinC4;
    tile[4 * c][j] = acc[u].x;
    tile[4 * c + 1][j] = acc[u].y;
    tile[4 * c + 2][j] = acc[u].z;
    tile[4 * c + 3][j] = acc[u].w;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < nc * r; e += kFinishThreads) {
    const int n = e / r, j = e - n * r;
    dst[(n0 + n) * r + j] += tile[n][j];
  }
}

// ---------------------------------------------------------------------------------------------
// split helpers
// ---------------------------------------------------------------------------------------------
// dst [2 r, K] bf16: rows j < r = hi(src[j, :]), rows r + j = lo(src[j, :]); src [r, K] fp32.
// transposed: src is [K, r] and row j of dst takes column j of src.
__global__ void k_split(const SplitTab tab) {
  grid_dep_sync();
  const int z = blockIdx.z;
  const int32_t r = tab.rank[z];
  const int64_t K = tab.K;
  const float* src = tab.src[z];
  uint16_t* dst = tab.dst[z];
  const int64_t n = (int64_t)r * K;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    int64_t j, k;
    if (tab.transposed) {   // walk src row-major for coalesced reads
      k = e / r;
      j = e - k * r;
    } else {
      j = e / K;
      k = e - j * K;
    }
    const float x = tab.transposed ? src[k * r + j] : src[j * K + k];
    const uint16_t hb = bf16_bits(x);
    dst[j * K + k] = hb;
    dst[(r + j) * K + k] = bf16_bits(x - bf16_val(hb));
  }
}

// Reduction work items: for every slot, the absolute 64-token blocks that hold any of its tokens
// (segment walk as in the token items), merged into runs and cut into spans of at most
// span_blocks blocks. A block shared by two slots is listed for both; each slot's transposed
// operand is zero at the other slot's tokens, so every token counts exactly once.
__global__ void k_make_red_items_tc(int64_t T, int32_t n_seg, const int32_t* __restrict__ seg_start,
                                    const int32_t* __restrict__ seg_slot, int32_t n_slots,
                                    int32_t span_blocks, TokenItem* items, int32_t* count,
                                    int32_t max_items) {
  grid_dep_sync();
  // The segment table is staged in shared memory; thread s walks it for slot s (counting its
  // items, then writing them after the lower slots' items), so the table is the same as a walk
  // slot by slot.
  __shared__ int32_t s_start[kSegSmem + 1], s_slot[kSegSmem];
  __shared__ int32_t s_count[LORA_MAX_SLOTS + 1];
  const SegView sv = stage_segments(n_seg, seg_start, seg_slot, s_start, s_slot);
  const int32_t nsegs = seg_start ? n_seg : (n_seg < 0 ? 1 : 0);
  const int s = threadIdx.x;
  auto walk = [&](bool write, int32_t base) {
    int32_t n = 0;
    auto emit_run = [&](int64_t b0, int64_t b1) {
      for (int64_t b = b0; b < b1; b += span_blocks) {
        if (write && base + n < max_items)
          items[base + n] = TokenItem{(int32_t)(b * 64), (int32_t)(min(b1, b + span_blocks) * 64), s, 0};
        ++n;
      }
    };
    int64_t cursor = 0, rb = -1, re = -1;
    for (int32_t k = 0; k < nsegs; ++k) {
      int64_t a = seg_start ? (int64_t)sv.start[k] : 0;
      int64_t b = seg_start ? (int64_t)sv.start[k + 1] : T;
      int32_t slot = seg_slot ? sv.slot[k] : 0;
      if (slot < 0 || slot >= n_slots) slot = -1;
      a = max((int64_t)0, min(a, T));
      b = max((int64_t)0, min(b, T));
      if (a < cursor) a = cursor;
      if (b <= a) continue;
      cursor = b;
      if (slot != s) continue;
      const int64_t ba = a / 64, bb = (b + 63) / 64;
      if (re >= 0 && ba <= re) {
        re = max(re, bb);
      } else {
        if (re >= 0) emit_run(rb, re);
        rb = ba;
        re = bb;
      }
    }
    if (re >= 0) emit_run(rb, re);
    return n;
  };
  if (s < n_slots) s_count[s + 1] = walk(false, 0);
  __syncthreads();
  if (s == 0) {
    s_count[0] = 0;
    for (int k = 1; k <= n_slots; ++k) s_count[k] += s_count[k - 1];
    *count = min(s_count[n_slots], max_items);
    for (int k = 0; k <= n_slots; ++k) count[1 + k] = min(s_count[k], max_items);   // slot ranges
  }
  __syncthreads();
  if (s < n_slots) walk(true, s_count[s]);
}

// Xd = bf16(M * X): the masked operand of the shrink and of dA when dropout is on. Rows run over
// blockIdx.y (grid-stride); a thread masks 8 consecutive columns (one 16-byte load and store).
__global__ void __launch_bounds__(256) k_mask_bf16(const __nv_bfloat16* __restrict__ X, int64_t T,
                                                   int64_t in_dim, const DropParams dp,
                                                   __nv_bfloat16* __restrict__ Xd) {
  grid_dep_sync();
  const int64_t i0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i0 >= in_dim) return;
  for (int64_t t = blockIdx.y; t < T; t += gridDim.y) {
    const DropRow dr = drop_row(dp, t);
    uint4 v = *reinterpret_cast<const uint4*>(X + t * in_dim + i0);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (!drop_keep_at(dr, dp.tau, i0 + e)) w[e / 2] &= (e & 1) ? 0x0000FFFFu : 0xFFFF0000u;
    *reinterpret_cast<uint4*>(Xd + t * in_dim + i0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

// ---------------------------------------------------------------------------------------------
cudaError_t launch_tc_rows(const TcRowsArgs& a, cudaStream_t st, int prof_kind) {
  static RowsParams prm;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  std::memset(&prm, 0, sizeof(prm));
  const int NP = a.NP;
  if (!tc::make_map_2d(&prm.ta, a.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.K, a.T,
                       a.lda > 0 ? a.lda : a.K, 64, kBM))
    return cudaErrorInvalidValue;
  for (int k = 0; k < a.n_slots; ++k)
    if (!tc::make_map_2d(&prm.ts[k], a.s[k], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.K,
                         2 * (uint64_t)a.rank[k], a.K, 64, (uint32_t)NP))
      return cudaErrorInvalidValue;
  for (int k = 0; k < a.n_slots; ++k) {
    if (2 * a.rank[k] > NP || a.rank[k] > a.ldo || a.rank[k] % 4) return cudaErrorInvalidValue;
    prm.rank[k] = a.rank[k];
  }
  if (a.splits < 1 || a.splits > kMaxSplitsRows || a.ldo % 4 || a.ldo > LORA_MAX_RANK)
    return cudaErrorInvalidValue;
  prm.items = a.items;
  prm.n_items = a.n_items;
  prm.err = tc::error_word();
  if (!prm.err) return cudaErrorInvalidDevice;
  prm.nk = (int32_t)((a.K + 63) / 64);
  prm.nk_per_split = (prm.nk + a.splits - 1) / a.splits;
  prm.ldp = (int32_t)a.ldo;
  prm.part = a.part;
  prm.T = a.T;
  dim3 grid((unsigned)a.max_items, (unsigned)a.splits);
  cudaError_t e = cudaSuccess;
  prof_begin(prof_kind, st);
  switch (NP) {
#define LORA_ROWS_CASE(NPV)                                                        \
  case NPV: {                                                                      \
    static bool attr = false;                                                      \
    if (!attr) {                                                                   \
      e = set_smem(k_tc_rows<NPV>, RowsCfg<NPV>::kSmem);                           \
      if (e != cudaSuccess) return e;                                              \
      attr = true;                                                                 \
    }                                                                              \
    launch_kernel(k_tc_rows<NPV>, grid, kThreads, RowsCfg<NPV>::kSmem, st, prm);              \
    break;                                                                         \
  }
    LORA_ROWS_CASE(16)
    LORA_ROWS_CASE(32)
    LORA_ROWS_CASE(64)
    LORA_ROWS_CASE(128)
#undef LORA_ROWS_CASE
    default:
      return cudaErrorInvalidValue;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.outT && a.items) {   // tokens of other slots read as zero in each slot's rows
    e = cudaMemsetAsync(a.outT, 0, a.outT_bytes, st);
    if (e != cudaSuccess) return e;
  }
  prof_begin(0, st);
  launch_kernel(k_rows_finish, dim3((unsigned)a.max_items, (unsigned)(kBM / kFinishTok)), kFinishThreads, 0, st, 
      a.part, a.splits, a.T, a.ldo, (int32_t)a.ldo, 1, a.items, a.n_items, a.si, a.out,
      a.ld_out > 0 ? a.ld_out : a.ldo, a.out2, a.ld2, a.outT, a.ldt);
  prof_end(prof_kind, st);   // the class's time spans the product and its split-K finish
  return cudaGetLastError();
}

cudaError_t launch_tc_red(const TcRedArgs& a, cudaStream_t st, int prof_kind) {
  static RedParams prm;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  std::memset(&prm, 0, sizeof(prm));
  for (int k = 0; k < a.n_slots; ++k) {
    if (!tc::make_map_2d(&prm.tst[k], a.st[k], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T,
                         2 * (uint64_t)a.rank[k], a.ldt, 64, kBM))
      return cudaErrorInvalidValue;
    prm.rank[k] = a.rank[k];
  }
  if (!tc::make_map_2d(&prm.tb, a.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.N, a.T,
                       a.ldb > 0 ? a.ldb : a.N, 64, 64))
    return cudaErrorInvalidValue;
  prm.items = a.items;
  prm.n_items = a.n_items;
  prm.err = tc::error_word();
  if (!prm.err) return cudaErrorInvalidDevice;
  prm.part = a.part;
  prm.N = a.N;
  prm.T = a.T;
  prm.span = a.span_tokens;
  prm.rstride = a.max_rank;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_smem(k_tc_red, kRedSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid((unsigned)((a.N + kRedBN - 1) / kRedBN), (unsigned)a.max_items);
  prof_begin(prof_kind, st);
  launch_kernel(k_tc_red, grid, kThreads, kRedSmem, st, prm);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t blocks = (a.N + kRedFinCols - 1) / kRedFinCols;
  prof_begin(0, st);
  launch_kernel(k_red_finish, dim3((unsigned)blocks, (unsigned)a.n_slots), kFinishThreads, 0, st, 
      a.part, a.items, a.n_items, a.N, a.max_rank, a.transposed, a.tab, a.T, a.span_tokens);
  prof_end(prof_kind, st);   // the class's time spans the product and its item reduction
  return cudaGetLastError();
}

cudaError_t launch_split(const SplitTab& t, int n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  int64_t most = 0;
  for (int k = 0; k < n; ++k) most = (int64_t)t.rank[k] * t.K > most ? (int64_t)t.rank[k] * t.K : most;
  int64_t blocks = (most + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  prof_begin(0, st);
  launch_kernel(k_split, dim3((unsigned)blocks, 1, (unsigned)n), 256, 0, st, t);
  return cudaGetLastError();
}

cudaError_t launch_split_rows_t(const float* src, int64_t lds, int64_t ncols, int64_t ldt,
                                const TokenItem* items,
                                const int32_t* n_items, int max_items, const SlotInfo& si,
                                uint16_t* dst, size_t dst_bytes, int64_t T, cudaStream_t st) {
  if (max_items <= 0) return cudaSuccess;
  // With an item table, tokens of other slots must read as zero in each slot's rows. A null table
  // (single adapter) writes every token of the one slot, and the tensor maps stop at T.
  if (items) {
    cudaError_t e = cudaMemsetAsync(dst, 0, dst_bytes, st);
    if (e != cudaSuccess) return e;
  }
  if (lds % 4 || ncols % 4 || ncols > LORA_MAX_RANK || ncols > lds) return cudaErrorInvalidValue;
  prof_begin(0, st);
  launch_kernel(k_rows_finish, dim3((unsigned)max_items, (unsigned)(kBM / kFinishTok)), kFinishThreads, 0, st, 
      src, 1, T, lds, (int32_t)ncols, 0, items, n_items, si, nullptr, (int64_t)0, nullptr,
      (int64_t)0, dst, ldt);
  return cudaGetLastError();
}

cudaError_t launch_make_red_items_tc(int64_t T, int32_t n_seg, const int32_t* seg_start,
                                     const int32_t* seg_slot, int32_t n_slots, int32_t span_blocks,
                                     TokenItem* items, int32_t* count, int32_t max_items,
                                     cudaStream_t st) {
  prof_begin(0, st);
  launch_kernel(k_make_red_items_tc, 1, 128, 0, st, T, n_seg, seg_start, seg_slot, n_slots, span_blocks,
                                         items, count, max_items);
  return cudaGetLastError();
}

cudaError_t launch_mask_bf16(const void* X, int64_t T, int64_t in_dim, const DropParams& dp,
                             void* Xd, cudaStream_t st) {
  if (T <= 0 || in_dim <= 0) return cudaSuccess;
  if (in_dim % 8) return cudaErrorInvalidValue;
  const unsigned gx = (unsigned)((in_dim / 8 + 255) / 256);
  const unsigned gy = (unsigned)(T < 8192 ? T : 8192);
  prof_begin(0, st);
  launch_kernel(k_mask_bf16, dim3(gx, gy), 256, 0, st, (const __nv_bfloat16*)X, T, in_dim, dp,
                (__nv_bfloat16*)Xd);
  return cudaGetLastError();
}

}  // namespace lora
