// Tensor-core low-rank products for bf16 activations (sm_103a): the shrink Hs = s' Xd A^T, the
// G = s' dY' B product and the token reductions dA += Gs^T Xd, dB += dY'^T Hs
// ("8. LoRA Fundamentals", How it works; "Backward Bug Hunts and Vulkan Tiled GEMM", Bug #1 and
// Bug #2: the adapter gradients as out_prod-style token reductions).
//
// The fp32 operand of each product (A, B^T, Hs or Gs) is split into bf16 hi + lo parts
// (x = hi + lo + O(2^-16 |x|)); both parts are multiplied against the exact bf16 activations, so
// the products keep fp32-level accuracy while running on kind::f16 tensor cores.
//
//  k_tc_rows: out[t, j] = alpha * sum_k A[t, k] (S[j, k] + S[r + j, k]) (shrink, G). M = 128
//             tokens of one work item, N = NP >= 2 r (hi rows then lo rows; or several adapters'
//             splits side by side), K split over a thread-block cluster of 1-8 CTAs.
//  k_tc_red:  dst += sum_t (ST[j, t] + ST[r + j, t]) Bmn[t, n] (dA, dB^T). M = 128 (2 r rows of
//             the slot's transposed split), N = 256 or 128 columns of dY' or Xd (MN-major
//             tiles), K = tokens in 64-token blocks split over a cluster of 1 to 16 CTAs. Up to
//             four reductions over the same tokens (dB and dA of a linear, the dB of every
//             projection of a fused group) share one launch as a job table along grid x.
//  k_tc_red_multi: dA of two to four adapters that read one Xd, each Xd tile streamed once.
// One CTA per SM with about 192 KB of stages in flight. The split partials stay in shared memory
// and the cluster adds them in split order through distributed shared memory, so no partial
// reaches global memory and reruns are bitwise equal.
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
  SlotInfo si;
  int32_t nk;                        // K blocks in total
  int32_t nk_per_split;
  int32_t ncols;                     // columns of out written per token (zeros past the rank)
  float* out;                        // [T, ld_out] (nullable)
  int64_t ld_out;
  float* out2;                       // slot-expanded copy [T, ld2] (nullable)
  int64_t ld2;
  uint16_t* outT;                    // per slot [2 r, ldt] transposed bf16 split (nullable)
  int64_t ldt;
  // side task: the transposed bf16 split of another [T, ldh] fp32 operand of the same tokens
  // into side_outT (per slot [2 r, ldt]), e.g. the saved Hs next to the G product
  const float* side_h;
  int64_t side_ldh;
  uint16_t* side_outT;
  int32_t pair_r;                    // wide tiles: hi / lo block width of each adapter
  int64_t T;
};

// NP <= 128: one adapter, N = NP >= 2 r (hi rows then lo rows), the raw tile staged and its hi
// and lo columns added in place. NP 256-512: several adapters side by side (the bf16 split of
// each in turn, hi rows then lo rows of pair_r each), two MMAs of N = NP / 2 per K-step above
// N 256, hi and lo added while the accumulator is read, so only the NP / 2 result columns are
// staged.
template <int NP>
struct RowsCfg {
  static constexpr bool kWide = NP > 128;
  static constexpr int kBBytes = NP * 128;
  static constexpr int kStageBytes = 16384 + kBBytes;
  // one CTA per SM with about 192 KB of stages in flight
  static constexpr int kStages = (192 * 1024 / kStageBytes) < 10 ? (192 * 1024 / kStageBytes) : 10;
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 1024;
  static constexpr int kLdb = (kWide ? NP / 2 : NP) + 4;   // staging row stride (floats)
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(kBM * kLdb * 4 <= kStages * kStageBytes, "partial tile fits the stages");
  static_assert(NP <= 512, "TMEM columns");
  // TMEM is allocated in powers of two columns (32 .. 512)
  static constexpr uint32_t kCols = NP <= 32 ? 32u : NP <= 64 ? 64u : NP <= 128 ? 128u
                                    : NP <= 256 ? 256u : 512u;
  static constexpr int kMmaN = NP > 256 ? NP / 2 : NP;   // one or two MMAs per K-step
  static constexpr uint32_t kIdesc = idesc(kFmtBF16, kBM, kMmaN);
  static constexpr int kBoxRows = NP > 256 ? NP / 2 : NP;   // TMA boxes hold at most 256 rows
};

// One work item (<= 128 tokens, one slot) per cluster of `splits` CTAs along y; CTA z multiplies
// the item's rows by its share of the K-blocks into TMEM and leaves the partial tile (hi and lo
// columns added) in its shared memory. The cluster then adds the partials in split order through
// distributed shared memory (reruns are bitwise equal): CTA z finishes token rows
// [z R, z R + R), R = 128 / splits, scales them by the slot's alpha and writes out, the
// slot-expanded copy and the transposed bf16 split (no partials reach global memory).
template <int NP>
__global__ void __launch_bounds__(kThreads, 1) k_tc_rows(const __grid_constant__ RowsParams p) {
  grid_dep_sync();
  using C = RowsCfg<NP>;
  extern __shared__ uint8_t smem_raw[];
  TokenItem it;
  if (!get_item(p.items, p.n_items, blockIdx.x, p.T, it)) return;   // the same for the cluster
  const int z = blockIdx.y;   // == rank in the cluster (cluster dims 1 x splits)
  const int splits = gridDim.y;
  const int R = kBM / splits;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (it.slot < 0) {
    // no adapter for these tokens: their rows of out are zero (the same for the whole cluster)
    if (p.out) {
      const int c4n = p.ncols / 4;
      for (int e = threadIdx.x; e < R * c4n; e += kThreads) {
        const int64_t t = (int64_t)it.t0 + z * R + e / c4n;
        if (t < it.t1)
          reinterpret_cast<float4*>(p.out + t * p.ld_out)[e % c4n] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    return;
  }
  const int r = p.si.rank[it.slot];
  const int kb0 = z * p.nk_per_split;
  const int kb1 = min(p.nk, kb0 + p.nk_per_split);
  const int nk = kb1 > kb0 ? kb1 - kb0 : 0;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(base + C::kStages * C::kStageBytes);
  uint64_t* empty_bar = full_bar + C::kStages;
  uint64_t* acc_bar = empty_bar + C::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
  float* buf = reinterpret_cast<float*>(base);   // partial tile [128][kLdb], over the idle stages
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

  bool ready = true;
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
#pragma unroll
        for (int h = 0; h < NP / C::kBoxRows; ++h)
          tma_load_2d(sa + 16384 + h * C::kBoxRows * 128, &p.ts[it.slot], &full_bar[s],
                      (kb0 + i) * 64, h * C::kBoxRows);
        issued = i + 1;
      }
      // every issued load has landed before the stages are reused as the partial tile
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
        for (int k = 0; k < 4; ++k) {
          umma_f16(tmem, da + 2 * k, db + 2 * k, C::kIdesc, (i > 0 || k > 0) ? 1u : 0u);
          if constexpr (NP > 256)   // the second half of the rows: 1024-byte atoms, so +NP/2 * 8
            umma_f16(tmem + (uint32_t)(NP / 2), da + 2 * k, db + (uint64_t)(NP / 2) * 8 + 2 * k,
                     C::kIdesc, (i > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&empty_bar[s]);
      }
      if (nk > 0) umma_commit(acc_bar);   // with no K-blocks the epilogue does not wait
    }
  } else {
    // epilogue: this thread's accumulator row (one token) -> its staging row, then hi + lo
    const int q = warp & 3;
    const int row = q * 32 + lane;
    if (p.side_h) {
      // side task while the K-blocks stream: the transposed split of the side operand's rows
      // [z R, z R + R) of this item, straight from global memory (a thread per token and half
      // of the columns; a warp's stores of one row are 32 consecutive tokens)
      const int64_t sb0 = (int64_t)it.t0 + z * R;
      const int e0 = threadIdx.x - 64;   // 0 .. 127
      const int halves = 128 / R;        // threads per token
      const int i = e0 % R, hpart = e0 / R;
      const int64_t t = sb0 + i;
      if (t < it.t1) {
        const int per = (r + halves - 1) / halves;
        const int j0 = hpart * per, j1 = min(r, j0 + per);
        const float* src = p.side_h + t * p.side_ldh;
        uint16_t* d = p.side_outT + (int64_t)p.si.region[it.slot] * p.ldt + t;
        for (int j = j0; j < j1; ++j) {
          const float x = __ldg(src + j);
          const uint16_t hb = bf16_bits(x);
          d[(int64_t)j * p.ldt] = hb;
          d[(int64_t)(r + j) * p.ldt] = bf16_bits(x - bf16_val(hb));
        }
      }
    }
    ready = nk == 0 || __all_sync(0xffffffffu, mbar_wait(acc_bar, 0u, 4u, p.err));
    if (ready) fence_after();
    float* br = buf + row * C::kLdb;
    if constexpr (C::kWide) {
      // output column o: adapter o / pair_r, hi column 2 pair_r (o / pair_r) + o % pair_r, its lo
      // column pair_r further on; 16 columns at a time
      const int pr = p.pair_r;
      for (int o = 0; o < NP / 2; o += 16) {
        float h[16], l[16];
        if (ready && nk > 0) {
          const int hc = 2 * pr * (o / pr) + (o % pr);
          tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)hc, h);
          tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(hc + pr), l);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) h[e] = l[e] = 0.f;
        }
        float4* dst = reinterpret_cast<float4*>(br + o);
#pragma unroll
        for (int g = 0; g < 4; ++g)
          dst[g] = make_float4(h[4 * g] + l[4 * g], h[4 * g + 1] + l[4 * g + 1],
                               h[4 * g + 2] + l[4 * g + 2], h[4 * g + 3] + l[4 * g + 3]);
      }
    } else if (ready && nk > 0) {
#pragma unroll
      for (int c = 0; c < NP / 16; ++c) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 16), v);
        float4* dst = reinterpret_cast<float4*>(br + c * 16);
#pragma unroll
        for (int g = 0; g < 4; ++g) dst[g] = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
      }
      for (int j = 0; j < r; j += 4) {
        const float4 h = *reinterpret_cast<const float4*>(br + j);
        const float4 l = *reinterpret_cast<const float4*>(br + r + j);
        *reinterpret_cast<float4*>(br + j) = make_float4(h.x + l.x, h.y + l.y, h.z + l.z, h.w + l.w);
      }
    } else {
      for (int j = 0; j < r; j += 4) *reinterpret_cast<float4*>(br + j) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    fence_before();
  }
  __syncthreads();
  cluster_sync_all();   // every CTA's partial tile is in its shared memory
  // CTA z: token rows [z R, z R + R) summed over the splits in split order
  const float alpha = p.si.alpha[it.slot];
  const int r4 = r / 4, c4n = p.ncols / 4;
  for (int e = threadIdx.x; e < R * c4n; e += kThreads) {
    const int i = z * R + e / c4n, c = e - (e / c4n) * c4n;
    const int64_t t = (int64_t)it.t0 + i;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < r4) {
      float4 pz[8];
#pragma unroll
      for (int zz = 0; zz < 8; ++zz)
        if (zz < splits) pz[zz] = dsmem_ld4(buf + i * C::kLdb + 4 * c, (uint32_t)zz);
#pragma unroll
      for (int zz = 0; zz < 8; ++zz)
        if (zz < splits) {
          v.x += pz[zz].x; v.y += pz[zz].y; v.z += pz[zz].z; v.w += pz[zz].w;
        }
      v = make_float4(v.x * alpha, v.y * alpha, v.z * alpha, v.w * alpha);
    }
    if (t < it.t1) {
      if (p.out) reinterpret_cast<float4*>(p.out + t * p.ld_out)[c] = v;
      if (p.out2 && c < r4) reinterpret_cast<float4*>(p.out2 + t * p.ld2 + p.si.pcol[it.slot])[c] = v;
    }
    // the finished values, for the transposed split below: only this CTA reads rows
    // [z R, z R + R) of its own tile, and each element is rewritten by the thread that read it
    if (c < r4) *reinterpret_cast<float4*>(buf + i * C::kLdb + 4 * c) = v;
  }
  const int64_t tb = (int64_t)it.t0 + z * R;
  const int nt = (int)max((int64_t)0, min((int64_t)R, (int64_t)it.t1 - tb));
  // transposed split of rows [z R, z R + nt) of this CTA's tile into d (per slot [2 r, ldt])
  auto write_split_t = [&](uint16_t* d) {
    for (int e = threadIdx.x; e < nt * r; e += kThreads) {
      const int j = e / nt, i = e - j * nt;
      const float x = buf[(z * R + i) * C::kLdb + j];
      const uint16_t hb = bf16_bits(x);
      d[(int64_t)j * p.ldt + i] = hb;
      d[(int64_t)(r + j) * p.ldt + i] = bf16_bits(x - bf16_val(hb));
    }
  };
  if (p.outT) {
    __syncthreads();
    write_split_t(p.outT + (int64_t)p.si.region[it.slot] * p.ldt + tb);
  }

  cluster_sync_all();   // peers' shared memory stays alive until every CTA has read it
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, C::kCols);
  }
}

constexpr int kMaxSplitsRows = 8;   // K splits of the rows kernel (the launcher rejects more)

// ---------------------------------------------------------------------------------------------
// k_tc_red
// ---------------------------------------------------------------------------------------------
struct RedJob {
  CUtensorMap tst[LORA_MAX_SLOTS];   // ST_slot [2 r, T] bf16 (tokens contiguous), box {64, 128}
  CUtensorMap tb;                    // B [T, N] bf16, box {64 (n), 64 (t)}
  int32_t rank[LORA_MAX_SLOTS];
  float* dst[LORA_MAX_SLOTS];        // dB_slot [N, r] (transposed) or dA_slot [r, N]
  int32_t transposed;
  int32_t tiles;                     // BN-column tiles of B: the job's share of the grid's x
  int64_t N;
};

// Up to kRedMaxJobs reductions over the same tokens, slots and run table (dB and dA of a linear,
// or the dB of every projection of a fused group) in one launch: grid x runs over job 0's tiles,
// then job 1's, and so on.
constexpr int kRedMaxJobs = 4;
struct RedParams {
  RedJob job[kRedMaxJobs];
  int32_t n_jobs;
  const TokenItem* items;            // 64-token aligned runs grouped by slot (null: the uniform
                                     // runs of kRedSpanBlocks blocks over [0, T), slot 0)
  const int32_t* counts;             // counts[1 + slot] .. counts[2 + slot]: the slot's items
  uint32_t* err;
  int64_t T;
};
static_assert(sizeof(RedParams) <= 32764, "kernel parameter block");

// Tile: M = 128 split rows (2 r used), N = BN columns of B (256 or 128), K = 64 tokens per stage;
// one CTA per SM with about 192 KB of stages in flight.
template <int BN>
struct RedCfg {
  static constexpr int kStageBytes = 16384 + BN * 128;
  static constexpr int kStages = (192 * 1024) / kStageBytes;
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 1024;
  static constexpr int kLdA = BN + 4;                 // staging [r][kLdA] (dA)
  static constexpr int kLdB = LORA_MAX_RANK + 4;      // staging [BN][kLdB] (dB, transposed)
  static_assert(LORA_MAX_RANK * kLdA * 4 <= kStages * kStageBytes, "dA staging fits");
  static_assert(BN * kLdB * 4 <= kStages * kStageBytes, "dB staging fits");
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kIdesc = idesc(kFmtBF16, kBM, BN, false, true);
};
constexpr int kRedMaxSplits = 16;

// dst_slot += (ST_hi + ST_lo) Bmn over the slot's tokens, for one BN-column tile of B.
// A cluster of `splits` CTAs along y shares the tile; CTA z accumulates its share of the slot's
// 64-token blocks in TMEM (M = 2 r split rows, N = BN columns, K = tokens) and leaves its partial
// (hi and lo rows added) in shared memory; the cluster then adds the partials in split order
// through distributed shared memory (reruns are bitwise equal) and CTA z adds columns
// [z W, z W + W), W = BN / splits, into dst. No partials reach global memory.
template <int BN>
__global__ void __launch_bounds__(kThreads, 1) k_tc_red(const __grid_constant__ RedParams p) {
  grid_dep_sync();
  using C = RedCfg<BN>;
  constexpr int kRedStages = C::kStages;
  constexpr int kRedStageBytes = C::kStageBytes;
  constexpr int kRedLdA = C::kLdA;
  constexpr int kRedLdB = C::kLdB;
  constexpr int kRedBN = BN;
  extern __shared__ uint8_t smem_raw[];
  const int slot = blockIdx.z;
  const int z = blockIdx.y;   // == rank in the cluster (cluster dims 1 x splits)
  const int splits = gridDim.y;
  int jb = 0, bx = (int)blockIdx.x;
  while (jb + 1 < p.n_jobs && bx >= p.job[jb].tiles) bx -= p.job[jb++].tiles;
  const RedJob& J = p.job[jb];
  const int32_t n0 = bx * BN;
  const int r = J.rank[slot];
  // this CTA's work: items [w0, w1) of the slot's items, split evenly over the cluster (the
  // uniform runs of a single-adapter call are the items of one segment covering [0, T))
  const int32_t nb_all = (int32_t)((p.T + 63) / 64);
  int32_t ia = 0, ib = (nb_all + kRedSpanBlocks - 1) / kRedSpanBlocks;
  if (p.items) {
    ia = p.counts[1 + slot];
    ib = p.counts[2 + slot];
  }
  const int32_t w0 = ia + (int32_t)((int64_t)(ib - ia) * z / splits);
  const int32_t w1 = ia + (int32_t)((int64_t)(ib - ia) * (z + 1) / splits);
  auto blocks_of = [&](int32_t w, int32_t& tb0, int32_t& nblk) {
    if (p.items) {
      const TokenItem it = p.items[w];
      tb0 = it.t0 & ~63;
      nblk = (it.t1 - tb0 + 63) / 64;
    } else {
      tb0 = w * kRedSpanBlocks * 64;
      nblk = min(kRedSpanBlocks, nb_all - w * kRedSpanBlocks);
    }
  };
  int nk = 0;
  for (int32_t w = w0; w < w1; ++w) {
    int32_t tb0, nb;
    blocks_of(w, tb0, nb);
    nk += nb;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(base + kRedStages * kRedStageBytes);
  uint64_t* empty_bar = full_bar + kRedStages;
  uint64_t* acc_bar = empty_bar + kRedStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
  float* buf = reinterpret_cast<float*>(base);   // staging over the idle stages
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRedStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(acc_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, (uint32_t)BN);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int i = 0;
      bool ok = true;
      for (int32_t w = w0; w < w1 && ok; ++w) {
        int32_t tb0, nb;
        blocks_of(w, tb0, nb);
        for (int b = 0; b < nb; ++b, ++i) {
          const int s = i % kRedStages;
          const uint32_t ph = (uint32_t)(i / kRedStages) & 1u;
          if (i >= kRedStages && !mbar_wait(&empty_bar[s], ph ^ 1u, 1u, p.err)) { ok = false; break; }
          uint8_t* sa = base + s * kRedStageBytes;
          mbar_expect_tx(&full_bar[s], kRedStageBytes);
          const int32_t t = tb0 + b * 64;
          tma_load_2d(sa, &J.tst[slot], &full_bar[s], t, 0);
#pragma unroll
          for (int q = 0; q < BN / 64; ++q)
            tma_load_2d(sa + 16384 + q * 8192, &J.tb, &full_bar[s], n0 + 64 * q, t);
        }
      }
      // every issued load has landed before the stages are reused as the staging tile
      for (int k = (i > kRedStages ? i - kRedStages : 0); k < i; ++k)
        if (!mbar_wait(&full_bar[k % kRedStages], (uint32_t)(k / kRedStages) & 1u, 1u, p.err)) break;
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
          umma_f16(tmem, da + 2 * k, db + 128 * k, C::kIdesc, (i > 0 || k > 0) ? 1u : 0u);
        umma_commit(&empty_bar[s]);
      }
      if (nk > 0) umma_commit(acc_bar);   // with no K-blocks the epilogue does not wait
    }
  } else {
    // epilogue: accumulator row `row` is split row j = row (hi, row < r) or j = row - r (lo,
    // r <= row < 2 r); hi rows are staged first, then lo rows are added onto them.
    // dA stages [j][n] (rows along dst's rows), dB stages [n][j] (dst is [N, r]).
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const bool ready = nk == 0 || __all_sync(0xffffffffu, mbar_wait(acc_bar, 0u, 4u, p.err));
    if (ready) fence_after();
    const bool live = ready && nk > 0;
    for (int phase = 0; phase < 2; ++phase) {
      const bool mine = phase == 0 ? row < r : (row >= r && row < 2 * r);
      const int j = phase == 0 ? row : row - r;
#pragma unroll 1
      for (int c = 0; c < kRedBN / 32; ++c) {
        float v[32];
        if (live) {
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), v);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = 0.f;
        }
        if (!mine) continue;
        if (!J.transposed) {
          float* d = buf + j * kRedLdA + c * 32;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            float4 x = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
            if (phase == 1) {
              const float4 h = reinterpret_cast<const float4*>(d)[g];
              x = make_float4(h.x + x.x, h.y + x.y, h.z + x.z, h.w + x.w);
            }
            reinterpret_cast<float4*>(d)[g] = x;
          }
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            float* d = buf + (c * 32 + k) * kRedLdB + j;
            *d = phase == 0 ? v[k] : *d + v[k];
          }
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
    }
    fence_before();
  }
  __syncthreads();
  cluster_sync_all();   // every CTA's partial tile is in its shared memory
  // CTA z adds columns [cz0, cz1) of the tile: W (a multiple of 4) each, the last CTAs of a
  // cluster whose size does not divide BN fewer or none
  const int W = ((kRedBN + splits - 1) / splits + 3) / 4 * 4;
  const int cz0 = z * W, cz1 = min(kRedBN, cz0 + W);
  const int Wz = cz1 > cz0 ? cz1 - cz0 : 0;
  float* dst = J.dst[slot];
  if (!J.transposed) {
    // dA [r, N]: rows j, columns n0 + cz0 ..
    const int w4 = Wz / 4;
    for (int e = threadIdx.x; e < r * w4; e += kThreads) {
      const int j = e / w4, c = cz0 + 4 * (e - (e / w4) * w4);
      const int64_t n = (int64_t)n0 + c;
      if (n >= J.N) continue;
      float4 pz[kRedMaxSplits];
#pragma unroll
      for (int zz = 0; zz < kRedMaxSplits; ++zz)
        if (zz < splits) pz[zz] = dsmem_ld4(buf + j * kRedLdA + c, (uint32_t)zz);
      float4* o = reinterpret_cast<float4*>(dst + (int64_t)j * J.N + n);
      float4 acc = *o;
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int zz = 0; zz < kRedMaxSplits; ++zz)
        if (zz < splits) {
          sum.x += pz[zz].x; sum.y += pz[zz].y; sum.z += pz[zz].z; sum.w += pz[zz].w;
        }
      acc.x += sum.x; acc.y += sum.y; acc.z += sum.z; acc.w += sum.w;
      *o = acc;
    }
  } else {
    // dB [N, r]: rows n0 + cz0 .., columns j
    const int r4 = r / 4;
    for (int e = threadIdx.x; e < Wz * r4; e += kThreads) {
      const int c = cz0 + e / r4, j = 4 * (e - (e / r4) * r4);
      const int64_t n = (int64_t)n0 + c;
      if (n >= J.N) continue;
      float4 pz[kRedMaxSplits];
#pragma unroll
      for (int zz = 0; zz < kRedMaxSplits; ++zz)
        if (zz < splits) pz[zz] = dsmem_ld4(buf + c * kRedLdB + j, (uint32_t)zz);
      float4* o = reinterpret_cast<float4*>(dst + n * r + j);
      float4 acc = *o;
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int zz = 0; zz < kRedMaxSplits; ++zz)
        if (zz < splits) {
          sum.x += pz[zz].x; sum.y += pz[zz].y; sum.z += pz[zz].z; sum.w += pz[zz].w;
        }
      acc.x += sum.x; acc.y += sum.y; acc.z += sum.z; acc.w += sum.w;
      *o = acc;
    }
  }
  cluster_sync_all();   // peers' shared memory stays alive until every CTA has read it
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, (uint32_t)BN);
  }
}

// ---------------------------------------------------------------------------------------------
// k_tc_red_multi: dA of several adapters that read one input (fused projections)
// ---------------------------------------------------------------------------------------------
// dA_m [r, N] += (ST_m[hi] + ST_m[lo])^T-rows x Xd over all tokens, for NA adapters of rank r
// (2 r <= 128) at once: per 64-token block the stage holds each adapter's [2 r, 64] transposed
// split (an M = 128 tile each) and one [64, 128] tile of Xd, so Xd is read once for the group;
// NA MMAs per K-step into TMEM columns m * 128 .. . The token split and its cluster reduction
// are those of k_tc_red.
constexpr int kRedMultiBN = 128;
template <int NA>
struct RedMultiCfg {
  static constexpr int kStageBytes = NA * 16384 + kRedMultiBN * 128;
  static constexpr int kStages = (192 * 1024) / kStageBytes;
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 1024;
  static constexpr int kLd = kRedMultiBN + 4;                   // staging [m][r][kLd]
  static constexpr int kStagingFloats = NA * LORA_MAX_RANK * kLd;
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(kStagingFloats * 4 <= kStages * kStageBytes, "staging fits the stages");
  static_assert(NA * kRedMultiBN <= 512, "TMEM columns");
  static constexpr uint32_t kCols = NA * kRedMultiBN <= 256 ? 256u : 512u;
  static constexpr uint32_t kIdesc = idesc(kFmtBF16, kBM, kRedMultiBN, false, true);
};

struct RedMultiParams {
  CUtensorMap tst[LORA_MAX_SLOTS];   // ST_m [2 r, T] bf16, box {64, 128}
  CUtensorMap tb;                    // Xd [T, N] bf16, box {64 (n), 64 (t)}
  uint32_t* err;
  float* dst[LORA_MAX_SLOTS];        // dA_m [r, N]
  int32_t r;
  int64_t N;
  int64_t T;
};

template <int NA>
__global__ void __launch_bounds__(kThreads, 1) k_tc_red_multi(const __grid_constant__ RedMultiParams p) {
  grid_dep_sync();
  using C = RedMultiCfg<NA>;
  extern __shared__ uint8_t smem_raw[];
  const int z = blockIdx.y;   // == rank in the cluster (cluster dims 1 x splits)
  const int splits = gridDim.y;
  const int32_t n0 = blockIdx.x * kRedMultiBN;
  const int r = p.r;
  // this CTA's 64-token blocks: the same runs of kRedSpanBlocks blocks as the single-adapter form
  const int32_t nb_all = (int32_t)((p.T + 63) / 64);
  const int32_t n_runs = (nb_all + kRedSpanBlocks - 1) / kRedSpanBlocks;
  const int32_t w0 = (int32_t)((int64_t)n_runs * z / splits);
  const int32_t w1 = (int32_t)((int64_t)n_runs * (z + 1) / splits);
  const int32_t blk0 = w0 * kRedSpanBlocks, blk1 = min(nb_all, w1 * kRedSpanBlocks);
  const int nk = blk1 > blk0 ? blk1 - blk0 : 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(base + C::kStages * C::kStageBytes);
  uint64_t* empty_bar = full_bar + C::kStages;
  uint64_t* acc_bar = empty_bar + C::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
  float* buf = reinterpret_cast<float*>(base);   // staging over the idle stages
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
      int i = 0;
      for (; i < nk; ++i) {
        const int s = i % C::kStages;
        const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
        if (i >= C::kStages && !mbar_wait(&empty_bar[s], ph ^ 1u, 1u, p.err)) break;
        uint8_t* sa = base + s * C::kStageBytes;
        mbar_expect_tx(&full_bar[s], C::kStageBytes);
        const int32_t t = (blk0 + i) * 64;
#pragma unroll
        for (int m = 0; m < NA; ++m) tma_load_2d(sa + m * 16384, &p.tst[m], &full_bar[s], t, 0);
#pragma unroll
        for (int q = 0; q < kRedMultiBN / 64; ++q)
          tma_load_2d(sa + NA * 16384 + q * 8192, &p.tb, &full_bar[s], n0 + 64 * q, t);
      }
      // every issued load has landed before the stages are reused as the staging tile
      for (int k = (i > C::kStages ? i - C::kStages : 0); k < i; ++k)
        if (!mbar_wait(&full_bar[k % C::kStages], (uint32_t)(k / C::kStages) & 1u, 1u, p.err)) break;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < nk; ++i) {
        const int s = i % C::kStages;
        if (!mbar_wait(&full_bar[s], (uint32_t)(i / C::kStages) & 1u, 2u, p.err)) break;
        fence_after();
        const uint32_t sa = smem_u32(base + s * C::kStageBytes);
        const uint64_t db = smem_desc_sw128_mn(sa + NA * 16384, 8192);
#pragma unroll
        for (int m = 0; m < NA; ++m) {
          const uint64_t da = smem_desc_sw128(sa + m * 16384);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_f16(tmem + (uint32_t)(m * kRedMultiBN), da + 2 * k, db + 128 * k, C::kIdesc,
                     (i > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&empty_bar[s]);
      }
      if (nk > 0) umma_commit(acc_bar);   // with no K-blocks the epilogue does not wait
    }
  } else {
    // epilogue: per adapter, hi rows staged first, then lo rows added onto them
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const bool ready = nk == 0 || __all_sync(0xffffffffu, mbar_wait(acc_bar, 0u, 4u, p.err));
    if (ready) fence_after();
    const bool live = ready && nk > 0;
    for (int phase = 0; phase < 2; ++phase) {
      const bool mine = phase == 0 ? row < r : (row >= r && row < 2 * r);
      const int j = phase == 0 ? row : row - r;
      for (int m = 0; m < NA; ++m) {
#pragma unroll 1
        for (int c = 0; c < kRedMultiBN / 32; ++c) {
          float v[32];
          if (live) {
            tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(m * kRedMultiBN + c * 32), v);
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = 0.f;
          }
          if (!mine) continue;
          float* d = buf + ((size_t)m * LORA_MAX_RANK + j) * C::kLd + c * 32;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            float4 x = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
            if (phase == 1) {
              const float4 h = reinterpret_cast<const float4*>(d)[g];
              x = make_float4(h.x + x.x, h.y + x.y, h.z + x.z, h.w + x.w);
            }
            reinterpret_cast<float4*>(d)[g] = x;
          }
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
    }
    fence_before();
  }
  __syncthreads();
  cluster_sync_all();   // every CTA's partial tiles are in its shared memory
  // columns [z W, z W + W) of every adapter's rows, summed over the cluster in split order
  const int W = kRedMultiBN / splits;
  const int w4 = W / 4;
  for (int e = threadIdx.x; e < NA * r * w4; e += kThreads) {
    const int m = e / (r * w4), rem = e - m * (r * w4);
    const int j = rem / w4, c = z * W + 4 * (rem - (rem / w4) * w4);
    const int64_t n = (int64_t)n0 + c;
    if (n >= p.N) continue;
    float4 pz[kRedMaxSplits];
#pragma unroll
    for (int zz = 0; zz < kRedMaxSplits; ++zz)
      if (zz < splits) pz[zz] = dsmem_ld4(buf + ((size_t)m * LORA_MAX_RANK + j) * C::kLd + c, (uint32_t)zz);
    float4* o = reinterpret_cast<float4*>(p.dst[m] + (int64_t)j * p.N + n);
    float4 acc = *o;
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int zz = 0; zz < kRedMaxSplits; ++zz)
      if (zz < splits) {
        sum.x += pz[zz].x; sum.y += pz[zz].y; sum.z += pz[zz].z; sum.w += pz[zz].w;
      }
    acc.x += sum.x; acc.y += sum.y; acc.z += sum.z; acc.w += sum.w;
    *o = acc;
  }
  cluster_sync_all();   // peers' shared memory stays alive until every CTA has read it
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, C::kCols);
  }
}

// ---------------------------------------------------------------------------------------------
// split helpers
// ---------------------------------------------------------------------------------------------
// The backward's adapter operands in one launch of 32 x 32 shared-memory tiles: A_slot^T (fp32,
// the dX product's LoRA operand) and the bf16 hi / lo split of B_slot^T (the G product's operand),
// both read and written along rows. Flat tile index: the tiles of every (task, slot) in turn.
__global__ void __launch_bounds__(256) k_adapter_prep(const TransposeTab ta, const SplitTab sb,
                                                      const AdapterPrepTiles pt) {
  grid_dep_sync();
  __shared__ float tile[32][33];
  int u = 0;
  while (u + 1 < pt.n && (int)blockIdx.x >= pt.first[u + 1]) ++u;
  const bool split = u >= pt.n_t;                 // tasks: transposes first, then splits
  const int k = split ? u - pt.n_t : u;           // slot
  const int local = (int)blockIdx.x - pt.first[u];
  const int64_t rows = split ? (pt.split_k[k] > 0 ? pt.split_k[k] : sb.K) : ta.rows[k];   // src rows (B: out, A: r)
  const int64_t cols = split ? sb.rank[k] : ta.cols[k];    // src cols (B: r, A: in)
  const int64_t ncb = (cols + 31) / 32;
  const int64_t r0 = (int64_t)(local / ncb) * 32, c0 = (int64_t)(local % ncb) * 32;
  const float* src = split ? sb.src[k] : ta.src[k];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int i = ty; i < 32; i += 8) {
    const int64_t r = r0 + i, c = c0 + tx;
    tile[i][tx] = (r < rows && c < cols) ? src[r * cols + c] : 0.f;
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int64_t c = c0 + i, r = r0 + tx;   // dst row c (a src column), dst column r
    if (r >= rows || c >= cols) continue;
    const float x = tile[tx][i];
    if (!split) {
      const int64_t ldd = ta.ld_dst[k] > 0 ? ta.ld_dst[k] : rows;
      ta.dst[k][c * ldd + r] = x;
    } else {
      const uint16_t hb = bf16_bits(x);
      sb.dst[k][c * rows + r] = hb;
      sb.dst[k][(cols + c) * rows + r] = bf16_bits(x - bf16_val(hb));
    }
  }
}

// dst [2 r, K] bf16: rows j < r = hi(src[j, :]), rows r + j = lo(src[j, :]); src [r, K] fp32.
// transposed: src is [K, r] and row j of dst takes column j of src.
__global__ void k_split(const SplitTab tab) {
  grid_dep_sync();
  const int z = blockIdx.z;
  const int32_t r = tab.rank[z];
  const int64_t K = tab.K;
  const float* src = tab.src[z];
  uint16_t* dst = tab.dst[z];
  if (!tab.transposed && K % 4 == 0) {
    // rows along y, four adjacent columns per thread: one 16-byte load, two 8-byte stores
    for (int64_t j = blockIdx.y; j < r; j += gridDim.y)
      for (int64_t k = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; k < K;
           k += (int64_t)gridDim.x * blockDim.x * 4) {
        const float4 x = *reinterpret_cast<const float4*>(src + j * K + k);
        const float v[4] = {x.x, x.y, x.z, x.w};
        uint16_t hb[4], lb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          hb[u] = bf16_bits(v[u]);
          lb[u] = bf16_bits(v[u] - bf16_val(hb[u]));
        }
        *reinterpret_cast<uint2*>(dst + j * K + k) =
            make_uint2((uint32_t)hb[0] | ((uint32_t)hb[1] << 16), (uint32_t)hb[2] | ((uint32_t)hb[3] << 16));
        *reinterpret_cast<uint2*>(dst + (r + j) * K + k) =
            make_uint2((uint32_t)lb[0] | ((uint32_t)lb[1] << 16), (uint32_t)lb[2] | ((uint32_t)lb[3] << 16));
      }
    return;
  }
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
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster_y(void (*kernel)(KArgs...), dim3 grid, int cluster_y, int smem,
                             cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)cluster_y;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = add_pdl_attr(attr, 1);
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

cudaError_t launch_tc_rows(const TcRowsArgs& a, cudaStream_t st, int prof_kind) {
  static RowsParams prm;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  std::memset(&prm, 0, sizeof(prm));
  const int NP = a.NP;
  if (!tc::make_map_2d(&prm.ta, a.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.K, a.T,
                       a.lda > 0 ? a.lda : a.K, 64, kBM))
    return cudaErrorInvalidValue;
  const bool wide = NP > 128;
  const uint32_t box_rows = NP > 256 ? (uint32_t)NP / 2 : (uint32_t)NP;
  for (int k = 0; k < a.n_slots; ++k)
    if (!tc::make_map_2d(&prm.ts[k], a.s[k], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.K,
                         2 * (uint64_t)a.rank[k], a.K, 64, box_rows))
      return cudaErrorInvalidValue;
  for (int k = 0; k < a.n_slots; ++k)
    if (2 * a.rank[k] > NP || a.rank[k] > a.ldo || a.rank[k] % 4 || a.si.rank[k] != a.rank[k])
      return cudaErrorInvalidValue;
  // the cluster splits the 128 token rows evenly: 1, 2, 4 or 8 CTAs
  if (a.splits < 1 || a.splits > kMaxSplitsRows || (a.splits & (a.splits - 1)) || a.ldo % 4 ||
      a.ldo > (wide ? NP / 2 : LORA_MAX_RANK))
    return cudaErrorInvalidValue;
  // wide tiles: one item table slot whose rank is the adapters' total, NP = twice it, adapters of
  // pair_r columns (a multiple of 16 dividing the total); no transposed outputs
  if (wide && (a.n_slots != 1 || 2 * a.rank[0] != NP || a.pair_r < 16 || a.pair_r % 16 ||
               a.rank[0] % a.pair_r || a.outT || a.side_h || a.items))
    return cudaErrorInvalidValue;
  prm.pair_r = wide ? a.pair_r : a.rank[0];
  prm.items = a.items;
  prm.n_items = a.n_items;
  prm.err = tc::error_word();
  if (!prm.err) return cudaErrorInvalidDevice;
  prm.si = a.si;
  prm.nk = (int32_t)((a.K + 63) / 64);
  prm.nk_per_split = (prm.nk + a.splits - 1) / a.splits;
  prm.ncols = (int32_t)a.ldo;
  prm.out = a.out;
  prm.ld_out = a.ld_out > 0 ? a.ld_out : a.ldo;
  prm.out2 = a.out2;
  prm.ld2 = a.ld2;
  prm.outT = a.outT;
  prm.ldt = a.ldt;
  prm.side_h = a.side_h;
  prm.side_ldh = a.side_ldh;
  prm.side_outT = a.side_outT;
  prm.T = a.T;
  if (a.side_h && (!a.side_outT || a.side_ldh % 4 || a.side_ldh < a.ldo || a.ldt <= 0))
    return cudaErrorInvalidValue;
  if (a.max_items <= 0) return cudaSuccess;
  if (a.items) {   // tokens of other slots read as zero in each slot's rows
    if (a.outT) {
      cudaError_t e = cudaMemsetAsync(a.outT, 0, a.outT_bytes, st);
      if (e != cudaSuccess) return e;
    }
    if (a.side_outT) {
      cudaError_t e = cudaMemsetAsync(a.side_outT, 0, a.outT_bytes, st);
      if (e != cudaSuccess) return e;
    }
  }
  dim3 grid((unsigned)a.max_items, (unsigned)a.splits);
  cudaError_t e = cudaSuccess;
  prof_begin(prof_kind, st);
  switch (NP) {
#define LORA_ROWS_CASE(NPV)                                                             \
  case NPV: {                                                                           \
    static bool attr = false;                                                           \
    if (!attr) {                                                                        \
      e = set_smem(k_tc_rows<NPV>, RowsCfg<NPV>::kSmem);                                \
      if (e != cudaSuccess) return e;                                                   \
      attr = true;                                                                      \
    }                                                                                   \
    e = launch_cluster_y(k_tc_rows<NPV>, grid, a.splits, RowsCfg<NPV>::kSmem, st, prm); \
    break;                                                                              \
  }
    LORA_ROWS_CASE(16)
    LORA_ROWS_CASE(32)
    LORA_ROWS_CASE(64)
    LORA_ROWS_CASE(128)
    LORA_ROWS_CASE(256)
    LORA_ROWS_CASE(384)
    LORA_ROWS_CASE(512)
#undef LORA_ROWS_CASE
    default:
      return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  prof_end(prof_kind, st);
  return cudaGetLastError();
}

// Clusters of `size` CTAs of a kernel that can be resident at once (0 when the size cannot be
// hosted). Sizes above 8 need the non-portable cluster attribute.
template <typename K>
int resident_clusters(K kernel, int smem, int size) {
  int n = 0;
  bool ok = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
            cudaSuccess;
  if (ok && size > 8)
    ok = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
         cudaSuccess;
  if (ok) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1, (unsigned)size, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)size;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  return n;
}

// resident clusters of k_tc_red<BN> per cluster size 1 .. kRedMaxSplits (cached per device)
template <int BN>
int red_resident(int size) {
  static int cache[64][kRedMaxSplits];
  static bool done[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (size < 1 || size > kRedMaxSplits) return 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!done[dev]) {
    for (int i = 0; i < kRedMaxSplits; ++i)
      cache[dev][i] = resident_clusters(k_tc_red<BN>, RedCfg<BN>::kSmem, i + 1);
    done[dev] = true;
  }
  return cache[dev][size - 1];
}

template <int BN>
cudaError_t launch_red_bn(dim3 grid, int splits, cudaStream_t st, const RedParams& prm) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_smem(k_tc_red<BN>, RedCfg<BN>::kSmem);
    if (e != cudaSuccess) return e;
    if (cudaFuncSetAttribute(k_tc_red<BN>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess)
      cudaGetLastError();
    attr = true;
  }
  return launch_cluster_y(k_tc_red<BN>, grid, splits, RedCfg<BN>::kSmem, st, prm);
}

namespace {
bool fill_red_job(RedJob& j, const TcRedArgs& a, int bn) {
  for (int k = 0; k < a.n_slots; ++k) {
    if (!tc::make_map_2d(&j.tst[k], a.st[k], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T,
                         2 * (uint64_t)a.rank[k], a.ldt, 64, kBM))
      return false;
    if (a.rank[k] % 4 || a.rank[k] > LORA_MAX_RANK) return false;
    j.rank[k] = a.rank[k];
    j.dst[k] = a.tab.out[k];
  }
  if (!tc::make_map_2d(&j.tb, a.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.N, a.T,
                       a.ldb > 0 ? a.ldb : a.N, 64, 64))
    return false;
  if (a.N % 4) return false;
  j.transposed = a.transposed;
  j.N = a.N;
  j.tiles = (int32_t)((a.N + bn - 1) / bn);
  return true;
}

cudaError_t launch_tc_red_jobs(const TcRedArgs* jobs, int n_jobs, cudaStream_t st, int prof_kind) {
  if (n_jobs < 1 || n_jobs > kRedMaxJobs) return cudaErrorInvalidValue;
  static RedParams prm;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  std::memset(&prm, 0, sizeof(prm));
  const TcRedArgs& a = jobs[0];
  if (a.T <= 0 || a.n_slots <= 0) return cudaSuccess;
  // Tile width and token splits (CTAs of one cluster, any size up to kRedMaxSplits): the most
  // CTAs, one per SM at most, whose clusters are all resident at once, with at least two 64-token
  // blocks of T per split; the wider tile and the smaller cluster on ties (the wider tile
  // re-reads the split operand less).
  const int sms = tc::sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  int best_bn = 256, best_splits = 1;
  int64_t best_ctas = -1;
  for (int bn : {256, 128}) {
    int64_t tiles = 0;
    for (int q = 0; q < n_jobs; ++q) tiles += (jobs[q].N + bn - 1) / bn;
    for (int c = 1; c <= kRedMaxSplits; ++c) {
      const int64_t clusters = tiles * a.n_slots;
      if (clusters * c > sms || (c > 1 && (a.T + 63) / 64 < 2 * (int64_t)c)) break;
      const int res = bn == 256 ? red_resident<256>(c) : red_resident<128>(c);
      if (clusters > res) continue;
      if (clusters * c > best_ctas) {
        best_ctas = clusters * c;
        best_bn = bn;
        best_splits = c;
      }
    }
  }
  const int bn = best_bn, splits = best_splits;
  int64_t tiles = 0;
  for (int q = 0; q < n_jobs; ++q) {
    if (!fill_red_job(prm.job[q], jobs[q], bn)) return cudaErrorInvalidValue;
    tiles += prm.job[q].tiles;
  }
  prm.n_jobs = n_jobs;
  prm.items = a.items;
  prm.counts = a.n_items;
  prm.err = tc::error_word();
  if (!prm.err) return cudaErrorInvalidDevice;
  prm.T = a.T;
  dim3 grid((unsigned)tiles, (unsigned)splits, (unsigned)a.n_slots);
  prof_begin(prof_kind, st);
  cudaError_t e = bn == 256 ? launch_red_bn<256>(grid, splits, st, prm)
                            : launch_red_bn<128>(grid, splits, st, prm);
  if (e != cudaSuccess) return e;
  prof_end(prof_kind, st);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_tc_red(const TcRedArgs& a, cudaStream_t st, int prof_kind) {
  return launch_tc_red_jobs(&a, 1, st, prof_kind);
}

cudaError_t launch_tc_red_n(const TcRedArgs* jobs, int n, cudaStream_t st, int prof_kind) {
  // in launches of at most kRedMaxJobs jobs
  for (int q0 = 0; q0 < n; q0 += kRedMaxJobs) {
    const int m = n - q0 < kRedMaxJobs ? n - q0 : kRedMaxJobs;
    const TcRedArgs& a = jobs[q0];
    for (int q = q0 + 1; q < q0 + m; ++q) {
      const TcRedArgs& b = jobs[q];
      if (a.T != b.T || a.n_slots != b.n_slots || a.items != b.items || a.n_items != b.n_items)
        return cudaErrorInvalidValue;
      for (int k = 0; k < a.n_slots; ++k)
        if (a.rank[k] != b.rank[k]) return cudaErrorInvalidValue;
    }
    cudaError_t e = launch_tc_red_jobs(jobs + q0, m, st, prof_kind);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_tc_red2(const TcRedArgs& a, const TcRedArgs& b, cudaStream_t st, int prof_kind) {
  const TcRedArgs jobs[2] = {a, b};
  return launch_tc_red_n(jobs, 2, st, prof_kind);
}

cudaError_t launch_adapter_prep(const TransposeTab& ta, const SplitTab& sb, int n,
                                cudaStream_t st, const int64_t* split_k) {
  if (n <= 0) return cudaSuccess;
  if (!sb.transposed || n > LORA_MAX_SLOTS) return cudaErrorInvalidValue;
  AdapterPrepTiles pt{};
  pt.n_t = n;
  pt.n = 2 * n;
  for (int k = 0; k < n; ++k) pt.split_k[k] = split_k ? split_k[k] : 0;
  int total = 0;
  for (int u = 0; u < 2 * n; ++u) {
    const bool split = u >= n;
    const int k = split ? u - n : u;
    const int64_t rows = split ? (pt.split_k[k] > 0 ? pt.split_k[k] : sb.K) : ta.rows[k];
    const int64_t cols = split ? sb.rank[k] : ta.cols[k];
    pt.first[u] = total;
    total += (int)(((rows + 31) / 32) * ((cols + 31) / 32));
  }
  if (total <= 0) return cudaSuccess;
  prof_begin(0, st);
  launch_kernel(k_adapter_prep, dim3((unsigned)total), dim3(256), 0, st, ta, sb, pt);
  return cudaGetLastError();
}

template <int NA>
int red_multi_resident(int size) {
  static int cache[64][5];
  static bool done[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!done[dev]) {
    for (int i = 0; i < 5; ++i)
      cache[dev][i] = resident_clusters(k_tc_red_multi<NA>, RedMultiCfg<NA>::kSmem, 1 << i);
    done[dev] = true;
  }
  int i = 0;
  while (i < 4 && (1 << i) < size) ++i;
  return (1 << i) == size ? cache[dev][i] : 0;
}

template <int NA>
cudaError_t launch_red_multi_na(const TcRedMultiArgs& a, cudaStream_t st, int prof_kind) {
  static RedMultiParams prm;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  std::memset(&prm, 0, sizeof(prm));
  const int sms = tc::sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int64_t tiles = (a.N + kRedMultiBN - 1) / kRedMultiBN;
  int splits = 1;
  for (int c = 2; c <= kRedMaxSplits; c *= 2) {
    if (tiles * c > sms || (a.T + 63) / 64 < 2 * (int64_t)c) break;
    if (tiles <= red_multi_resident<NA>(c)) splits = c;
  }
  for (int m = 0; m < NA; ++m) {
    if (!tc::make_map_2d(&prm.tst[m], a.st[m], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T,
                         2 * (uint64_t)a.r, a.ldt, 64, kBM))
      return cudaErrorInvalidValue;
    prm.dst[m] = a.dst[m];
  }
  if (!tc::make_map_2d(&prm.tb, a.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.N, a.T,
                       a.ldb > 0 ? a.ldb : a.N, 64, 64))
    return cudaErrorInvalidValue;
  prm.err = tc::error_word();
  if (!prm.err) return cudaErrorInvalidDevice;
  prm.r = a.r;
  prm.N = a.N;
  prm.T = a.T;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_smem(k_tc_red_multi<NA>, RedMultiCfg<NA>::kSmem);
    if (e != cudaSuccess) return e;
    if (cudaFuncSetAttribute(k_tc_red_multi<NA>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess)
      cudaGetLastError();
    attr = true;
  }
  dim3 grid((unsigned)tiles, (unsigned)splits, 1);
  prof_begin(prof_kind, st);
  cudaError_t e = launch_cluster_y(k_tc_red_multi<NA>, grid, splits, RedMultiCfg<NA>::kSmem, st, prm);
  if (e != cudaSuccess) return e;
  prof_end(prof_kind, st);
  return cudaGetLastError();
}

cudaError_t launch_tc_red_multi(const TcRedMultiArgs& a, cudaStream_t st, int prof_kind) {
  if (a.T <= 0) return cudaSuccess;
  if (a.r < 4 || a.r % 4 || 2 * a.r > kBM || a.r > LORA_MAX_RANK || a.N % 8) return cudaErrorInvalidValue;
  switch (a.n) {
    case 2: return launch_red_multi_na<2>(a, st, prof_kind);
    case 3: return launch_red_multi_na<3>(a, st, prof_kind);
    case 4: return launch_red_multi_na<4>(a, st, prof_kind);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_split(const SplitTab& t, int n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  int64_t most = 0;
  int32_t rmax = 0;
  for (int k = 0; k < n; ++k) {
    most = (int64_t)t.rank[k] * t.K > most ? (int64_t)t.rank[k] * t.K : most;
    rmax = t.rank[k] > rmax ? t.rank[k] : rmax;
  }
  if (most <= 0) return cudaSuccess;
  dim3 grid;
  if (!t.transposed && t.K % 4 == 0) {   // the kernel's row-wise form
    int64_t bx = (t.K / 4 + 255) / 256;
    grid = dim3((unsigned)(bx > 64 ? 64 : bx), (unsigned)rmax, (unsigned)n);
  } else {
    int64_t blocks = (most + 255) / 256;
    grid = dim3((unsigned)(blocks > 4096 ? 4096 : blocks), 1, (unsigned)n);
  }
  prof_begin(0, st);
  launch_kernel(k_split, grid, 256, 0, st, t);
  return cudaGetLastError();
}

cudaError_t launch_make_red_items_tc(int64_t T, int32_t n_seg, const int32_t* seg_start,
                                     const int32_t* seg_slot, int32_t n_slots, int32_t span_blocks,
                                     TokenItem* items, int32_t* count, int32_t max_items,
                                     cudaStream_t st) {
  if (seg_start && seg_slot && n_seg >= 1 && n_seg <= 2048 && T <= INT32_MAX - 64)
    return launch_make_red_items_par(T, n_seg, seg_start, seg_slot, n_slots, span_blocks, items,
                                     count, max_items, st);
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
