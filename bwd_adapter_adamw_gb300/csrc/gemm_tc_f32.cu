// Tensor-core frozen products for fp32 activations (sm_103a), as bf16 products of split operands:
//
//   out[t, n] = ( sum_k A[t, k] B[n, k] + [mask(t, n)] * sum_j P[t, j] Q_slot[n, j] ) * colscale[n]
//
// with every fp32 operand x of the main product split into x_hi = bf16(x) and x_lo =
// bf16(x - x_hi), and the product formed as A_hi B_hi + A_hi B_lo + A_lo B_hi + A_lo B_lo with
// tcgen05.mma kind::f16 (bf16 operands, fp32 accumulation). The split keeps 16 significant bits
// of every operand (|x - x_hi - x_lo| <= 2^-16 |x|). The fourth product costs one N = 128 MMA
// more per K-step and keeps heavy-tailed operands over long K inside the fp32 paths' 1e-5
// relative bound (with three products a Student-t upstream gradient over K = 1024 measured
// 1.4e-5).
// The short LoRA K-blocks (P = Hs or Gs, Q = B or A^T, at most two 32-wide blocks) land raw and
// are split in shared memory by two converter warps into tf32 hi / lo (three kind::tf32 products,
// about 2^-21 relative). (Same roles as the bf16 kernel: frozen forward X W^T + Hs B^T, frozen
// dX dY' W + (Gs A) * M; "8. LoRA Fundamentals", How it works; "Backward Bug Hunts and Vulkan
// Tiled GEMM", Bug #1.)
//
// The frozen operands arrive already split in HBM: B (W or W^T) by the weight preparation, once,
// and A (X or dY') by the streaming shrink / G kernel, which reads A anyway. So the main K-loop
// is a plain TMA -> MMA pipeline of four bf16 tiles per stage (A_hi, A_lo, B_hi, B_lo), 64
// elements of K each.
//
// Per K-step two N = 256 MMAs (the stage holds B_hi and B_lo back to back): A_hi x [B_hi; B_lo],
// whose first 128 columns take A_hi B_hi and last 128 A_hi B_lo, then A_lo x [B_hi; B_lo] into
// the same columns (A_lo B_hi, A_lo B_lo); the epilogue adds the two halves. N = 256 MMAs run
// about 1.3x faster per flop than N = 128 ones.
//
// The tensor core's fp32 accumulation loses a little at every MMA, so no accumulation chain is
// allowed to grow with K: two 256-column TMEM regions take turns, each holding the partial sum of
// 256 elements of K (a period: 4 main K-blocks), and while one fills, the epilogue warps drain
// the other into fp32 registers with ordinary round-to-nearest adds. The LoRA K-blocks form a
// period of their own, masked element-wise when the LoRA term is dropout-masked.
//
// CTA (384 threads): warp 0 TMA, warp 1 TMEM + MMA issue, warps 2..9 epilogue, warps 10..11 LoRA
// split. Tile 128 x 128; every K-block is one 128-byte swizzled row (64 bf16 of the main
// product, 32 fp32 of the LoRA term); three stages of four tiles.
#include <cstring>
#include <mutex>

#include "tc_ptx.cuh"

namespace lora {

namespace {
using namespace tc;

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBK = 32;                        // LoRA K-block: 32 fp32, one 128-byte swizzled row
constexpr int kBKm = 64;                       // main K-block: 64 bf16, one 128-byte swizzled row
constexpr int kStages = 3;
constexpr int kTile = 128 * kBK * 4;           // 128 rows x 128 bytes
constexpr int kStageBytes = 4 * kTile;         // A_hi, A_lo, B_hi, B_lo
constexpr int kEpiWarps = 8;     // two per TMEM lane quarter, 64 columns each
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kConvThreads = 64;
// TMA, MMA, epilogue, LoRA split: 12 warps, 3 per SM sub-partition, so up to 168 registers each
constexpr int kThreads = 64 + kEpiThreads + kConvThreads;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 1024;
constexpr int kMaxLoraKb = (LORA_MAX_RANK + kBK - 1) / kBK;   // LoRA K-blocks per tile
static_assert(kSmemBytes <= 232448, "dynamic shared memory per CTA");

__device__ __forceinline__ uint64_t kdesc(uint32_t saddr) {
  return kBK == 32 ? smem_desc_sw128(saddr) : smem_desc_sw64(saddr);
}
constexpr uint32_t kIdesc = idesc(kFmtTF32, kBM, kBN);            // LoRA: lo x Q_hi into the big half
constexpr uint32_t kIdesc2 = idesc(kFmtTF32, kBM, 2 * kBN);       // LoRA: hi x [Q_hi; Q_lo]
constexpr uint32_t kIdescB2 = idesc(kFmtBF16, kBM, 2 * kBN);      // main: hi or lo x [B_hi; B_lo]
constexpr int kPeriod = 4;   // main K-blocks (256 elements) accumulated in one TMEM region
constexpr int kPartLd = kBN + 4;   // row stride (floats) of a split-K partial tile in shared memory
constexpr int kMaxSplits = 8;      // portable cluster size
static_assert(kBM * kPartLd * 4 <= kStages * kStageBytes, "partial tile fits the stage buffers");

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// float4 at `local` (this CTA's shared-memory layout) in cluster CTA `rank`
__device__ __forceinline__ float4 ld_peer4(const float* local, uint32_t rank) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(local), remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote) : "memory");
  return v;
}

struct F32Params {
  CUtensorMap tah, tal;               // A hi / lo [T, K] bf16, box {64, 128}
  CUtensorMap tbh, tbl;               // B hi / lo [N, K] bf16, box {64, 128}
  CUtensorMap tp;                     // P [T, ldp] fp32, box {32, 128}
  CUtensorMap tq[LORA_MAX_SLOTS];     // Q_slot [N, r] fp32, box {32, 128}
  CUtensorMap to;                     // out [T, ldo] fp32, box {32, 32} (the epilogue's stores)
  const TokenItem* items;             // null: uniform 128-token tiles, slot 0
  const int32_t* n_items;
  int64_t T;
  uint32_t* err;
  int32_t nk_main;
  int32_t splits;                     // CTAs of one cluster splitting the main K-blocks (1..8)
  int32_t kb_per_split;
  int32_t has_lora;
  int32_t lora_separate;
  int32_t q_rank[LORA_MAX_SLOTS];
  const float* n_colscale;
  float* out;
  int64_t ldo;
  int64_t n_out;
  DropParams drop;
};

// Split the raw fp32 tile at t in place into its tf32 part, and write the remainder one tile on.
__device__ __forceinline__ void split_tile(uint8_t* t, int ct) {
#pragma unroll 4
  for (int i = ct; i < kTile / 16; i += kConvThreads) {
    float4* hi = reinterpret_cast<float4*>(t + i * 16);
    float4* lo = reinterpret_cast<float4*>(t + kTile + i * 16);
    const float4 v = *hi;
    const float4 h = make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z), tf32_hi(v.w));
    *hi = h;
    *lo = make_float4(v.x - h.x, v.y - h.y, v.z - h.z, v.w - h.w);
  }
}

__global__ void __launch_bounds__(kThreads, 1) k_tc_gemm_f32(const __grid_constant__ F32Params p) {
  grid_dep_sync();
  extern __shared__ uint8_t smem_raw[];
  TokenItem it;
  if (!get_item(p.items, p.n_items, blockIdx.y, p.T, it)) return;
  const int slot = it.slot;
  const int32_t m0 = it.t0;
  const int32_t n0 = blockIdx.x * kBN;
  // this CTA's main K-blocks (split z of the cluster) and, for split 0, the LoRA K-blocks; local
  // index i runs over [0, nml) main blocks then [nml, nk) LoRA blocks
  const int z = blockIdx.z;
  const int kb_lo = z * p.kb_per_split;
  const int nml = max(0, min(p.nk_main, kb_lo + p.kb_per_split) - kb_lo);
  const int nk_lora = (p.has_lora && slot >= 0 && z == 0) ? (p.q_rank[slot] + kBK - 1) / kBK : 0;
  const int nk = nml + nk_lora;
  const bool sep = p.lora_separate && nk_lora > 0;
  const uint32_t ncols = 512u;   // two regions of 256 columns: [hi x B_hi (+ lo x B_hi) | hi x B_lo]
  // accumulation periods: kPeriod main K-blocks each, then the LoRA K-blocks as a period of their
  // own (masked element-wise in the epilogue when the LoRA term is dropout-masked)
  const int n_main_periods = (nml + kPeriod - 1) / kPeriod;
  const int n_periods = n_main_periods + (nk_lora > 0 ? 1 : 0);

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // full_bar / empty_bar: the stage ring of the main K-blocks. The LoRA K-blocks use the same
  // stages (after empty_bar) but single-use barriers of their own, lora_full (TMA landed) and
  // lora_conv (split done), so that no wait ever targets a phase more than one ahead.
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(base + kStages * kStageBytes);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* lora_full = empty_bar + kStages;
  uint64_t* lora_conv = lora_full + kMaxLoraKb;
  uint64_t* acc_full = lora_conv + kMaxLoraKb;   // [2]: a region's period is complete
  uint64_t* acc_empty = acc_full + 2;           // [2]: the epilogue has drained the region
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int j = 0; j < kMaxLoraKb; ++j) {
      mbar_init(&lora_full[j], 1);
      mbar_init(&lora_conv[j], kConvThreads);
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(&acc_full[r], 1);
      mbar_init(&acc_empty[r], kEpiThreads);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, ncols);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kStages;
        const uint32_t ph = (uint32_t)(kb / kStages) & 1u;
        if (kb >= kStages && !mbar_wait(&empty_bar[s], ph ^ 1u, 1u, p.err)) break;
        uint8_t* st = base + s * kStageBytes;
        if (kb < nml) {
          const int x = (kb_lo + kb) * kBKm;
          mbar_expect_tx(&full_bar[s], 4 * kTile);
          tma_load_2d(st, &p.tah, &full_bar[s], x, m0);
          tma_load_2d(st + kTile, &p.tal, &full_bar[s], x, m0);
          tma_load_2d(st + 2 * kTile, &p.tbh, &full_bar[s], x, n0);
          tma_load_2d(st + 3 * kTile, &p.tbl, &full_bar[s], x, n0);
        } else {
          const int j = kb - nml;
          mbar_expect_tx(&lora_full[j], 2 * kTile);
          tma_load_2d(st, &p.tp, &lora_full[j], j * kBK, m0);
          tma_load_2d(st + 2 * kTile, &p.tq[slot], &lora_full[j], j * kBK, n0);
        }
        issued = kb + 1;
      }
      // copies still in flight complete before the CTA can exit
      for (int kb = (issued > kStages ? issued - kStages : 0); kb < issued; ++kb) {
        const bool ok = kb < nml
                            ? mbar_wait(&full_bar[kb % kStages], (uint32_t)(kb / kStages) & 1u, 1u, p.err)
                            : mbar_wait(&lora_full[kb - nml], 0u, 1u, p.err);
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // Per K-step: hi x [B_hi; B_lo] and lo x [B_hi; B_lo] as N = 256 MMAs (first half: x B_hi,
      // second half: x B_lo); the LoRA K-blocks take hi x [Q_hi; Q_lo] and lo x Q_hi (tf32).
      // Regions alternate per period; a region is reused only after the epilogue has drained it.
      int per = -1;
      uint32_t d = tmem;
      bool ok = true;
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % kStages;
        const bool lora = kb >= nml;
        const bool start = lora ? kb == nml : (kb % kPeriod) == 0;
        if (start) {
          if (per >= 0) umma_commit(&acc_full[per & 1]);
          ++per;
          const int use = per >> 1;
          if (use >= 1 && !mbar_wait(&acc_empty[per & 1], (uint32_t)(use - 1) & 1u, 2u, p.err)) break;
          fence_after();
          d = tmem + 256u * (uint32_t)(per & 1);
        }
        // main K-blocks are consumed as landed; LoRA K-blocks once the converter has split them
        ok = lora ? mbar_wait(&lora_conv[kb - nml], 0u, 2u, p.err)
                  : mbar_wait(&full_bar[s], (uint32_t)(kb / kStages) & 1u, 2u, p.err);
        if (!ok) break;
        fence_after();
        const uint32_t sa = smem_u32(base + s * kStageBytes);
        const uint64_t ah = kdesc(sa), al = kdesc(sa + kTile), bh = kdesc(sa + 2 * kTile);
        // four 32-byte K-steps per 128-byte row: K 16 of bf16 (main) or K 8 of tf32 (LoRA)
        if (lora) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            umma_tf32(d, ah + 2 * k, bh + 2 * k, kIdesc2, (start && k == 0) ? 0u : 1u);
            umma_tf32(d, al + 2 * k, bh + 2 * k, kIdesc, 1u);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            umma_f16(d, ah + 2 * k, bh + 2 * k, kIdescB2, (start && k == 0) ? 0u : 1u);
            umma_f16(d, al + 2 * k, bh + 2 * k, kIdescB2, 1u);
          }
        }
        umma_commit(&empty_bar[s]);
      }
      if (per >= 0) umma_commit(&acc_full[per & 1]);
    }
  } else if (warp >= 2 + kEpiWarps) {
    // LoRA K-blocks: split the landed P and Q tiles (x -> tf32(x) in place, x - tf32(x) one tile on)
    const int ct = threadIdx.x - (64 + kEpiThreads);
    for (int kb = nml; kb < nk; ++kb) {
      const int s = kb % kStages;
      if (!mbar_wait(&lora_full[kb - nml], 0u, 8u, p.err)) break;
      uint8_t* st = base + s * kStageBytes;
      split_tile(st, ct);
      split_tile(st + 2 * kTile, ct);
      // generic-proxy writes must be visible to the tensor core's async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&lora_conv[kb - nml])) : "memory");
    }
  } else {
    // epilogue warps 2..9: TMEM lanes 32 * (warp % 4), columns [64 half, 64 half + 64); each
    // thread keeps its row's 64 sums in registers and adds every drained period into them
    // (round-to-nearest fp32 adds)
    constexpr int kCols = kBN / 2;
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const int64_t m = (int64_t)m0 + row;
    const bool row_ok = m < it.t1;
    const int c0 = half * kCols;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0;
    float run[kCols];
#pragma unroll
    for (int j = 0; j < kCols; ++j) run[j] = 0.f;
    bool ready = true;
    for (int per = 0; per < n_periods && ready; ++per) {
      const int r = per & 1;
      ready = __all_sync(0xffffffffu, mbar_wait(&acc_full[r], (uint32_t)(per >> 1) & 1u, 4u, p.err));
      if (!ready) break;
      fence_after();
      const bool masked = sep && per == n_periods - 1;
      const DropRow drow = masked ? drop_row(p.drop, m) : DropRow{0, 0};
      const uint32_t reg = lane_base + 256u * (uint32_t)r;
#pragma unroll
      for (int h = 0; h < kCols / 16; ++h) {
        uint32_t big[16], small[16];
        tmem_ld16_nw(reg + (uint32_t)(h * 16), big);
        tmem_ld16_nw(reg + 128u + (uint32_t)(h * 16), small);
        tmem_wait_ld();
        if (masked) {
          // dropout-masked LoRA term: keep bits first (a rolled loop: the hash is register-heavy)
          uint32_t keep = 0u;
#pragma unroll 1
          for (int j = 0; j < 16; ++j) {
            const int64_t n = (int64_t)n0 + c0 + h * 16 + j;
            if (row_ok && n < p.n_out && drop_keep_at(drow, p.drop.tau, n)) keep |= 1u << j;
          }
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (!((keep >> j) & 1u)) big[j] = small[j] = 0u;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) run[h * 16 + j] += __uint_as_float(big[j]) + __uint_as_float(small[j]);
      }
      fence_before();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&acc_empty[r])) : "memory");
    }
    if (ready && p.splits > 1) {
      // split K: this CTA's partial tile goes to shared memory (row stride kPartLd floats, so
      // that the float4 row writes of a quarter warp hit distinct banks); the cluster sums the
      // splits below
      float* part = reinterpret_cast<float*>(base) + (size_t)row * kPartLd + c0;
#pragma unroll
      for (int g = 0; g < kCols / 4; ++g)
        *reinterpret_cast<float4*>(part + 4 * g) =
            make_float4(run[4 * g], run[4 * g + 1], run[4 * g + 2], run[4 * g + 3]);
    } else if (ready) {
      // Whole tiles (and the last tile of the call, which the tensor bounds clip) leave through
      // bulk tensor stores of 32 x 32 boxes staged in the now idle stage buffers, 128-byte
      // swizzled so that the row-per-thread writes hit distinct banks. A partial item of a
      // multi-adapter call stores row by row: the rows past it belong to other CTAs.
      const bool tile_store = (it.t1 - it.t0 == kBM) || ((int64_t)it.t1 == p.T);
      uint8_t* box0 = base + (size_t)(warp - 2) * (kCols / 32) * 4096;
#pragma unroll
      for (int c = 0; c < kCols / 32; ++c) {
        const int64_t nb = (int64_t)n0 + c0 + c * 32;
        float* v = run + c * 32;
        if (p.n_colscale) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= (nb + j < p.n_out) ? __ldg(p.n_colscale + nb + j) : 0.f;
        }
        if (tile_store) {
          uint8_t* box = box0 + c * 4096 + lane * 128;
#pragma unroll
          for (int g = 0; g < 8; ++g)
            *reinterpret_cast<float4*>(box + ((g ^ (lane & 7)) << 4)) =
                make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
        } else if (row_ok) {
#pragma unroll
          for (int g = 0; g < 8; ++g)
            if (nb + 4 * g + 4 <= p.n_out)
              *reinterpret_cast<float4*>(p.out + m * p.ldo + nb + 4 * g) =
                  make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
        }
      }
      if (tile_store) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int c = 0; c < kCols / 32; ++c)
            tma_store_2d(&p.to, box0 + c * 4096, n0 + c0 + c * 32, m0 + q * 32);
          tma_store_commit_and_wait_read();
        }
        __syncwarp();
      }
    }
    fence_before();
  }
  __syncthreads();
  if (p.splits > 1) {
    // CTA z of the cluster adds rows [z R, z R + R) of the tile over all splits, in split order
    // (reruns are bitwise equal), from the peers' shared memory, and stores them coalesced
    cluster_sync();
    const int rows = kBM / p.splits;
    const float* part = reinterpret_cast<const float*>(base);
    for (int e = threadIdx.x; e < rows * (kBN / 4); e += kThreads) {
      const int rr = z * rows + e / (kBN / 4);
      const int cc = 4 * (e % (kBN / 4));
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int zz = 0; zz < p.splits; ++zz) {
        const float4 v = ld_peer4(part + (size_t)rr * kPartLd + cc, (uint32_t)zz);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      const int64_t m = (int64_t)m0 + rr;
      const int64_t n = (int64_t)n0 + cc;
      if (m < it.t1 && n < p.n_out) {
        if (p.n_colscale) {
          acc.x *= __ldg(p.n_colscale + n); acc.y *= __ldg(p.n_colscale + n + 1);
          acc.z *= __ldg(p.n_colscale + n + 2); acc.w *= __ldg(p.n_colscale + n + 3);
        }
        *reinterpret_cast<float4*>(p.out + m * p.ldo + n) = acc;
      }
    }
    cluster_sync();   // peers' shared memory stays alive until every CTA has read it
  }
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

}  // namespace

cudaError_t launch_tc_gemm_f32(const TcGemmArgs& a, cudaStream_t st, int prof_kind) {
  static F32Params prm;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  std::memset(&prm, 0, sizeof(prm));
  const auto F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const auto BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!a.a_lo || !a.b_lo) return cudaErrorInvalidValue;
  if (!tc::make_map_2d(&prm.tah, a.a, BF16, 2, a.K, a.T, a.K, kBKm, kBM) ||
      !tc::make_map_2d(&prm.tal, a.a_lo, BF16, 2, a.K, a.T, a.K, kBKm, kBM) ||
      !tc::make_map_2d(&prm.tbh, a.b, BF16, 2, a.K, a.n_rows, a.K, kBKm, kBN) ||
      !tc::make_map_2d(&prm.tbl, a.b_lo, BF16, 2, a.K, a.n_rows, a.K, kBKm, kBN))
    return cudaErrorInvalidValue;
  prm.has_lora = a.p != nullptr;
  if (a.p) {
    if (!tc::make_map_2d(&prm.tp, a.p, F32, 4, a.ldp, a.T, a.ldp, kBK, kBM)) return cudaErrorInvalidValue;
    for (int k = 0; k < a.n_slots; ++k) {
      if (a.q_rank[k] > kMaxLoraKb * kBK) return cudaErrorInvalidValue;
      prm.q_rank[k] = a.q_rank[k];
      if (!tc::make_map_2d(&prm.tq[k], a.q[k], F32, 4, a.q_rank[k], a.n_rows, a.q_rank[k], kBK, kBN))
        return cudaErrorInvalidValue;
    }
  }
  prm.items = a.items;
  prm.n_items = a.n_items;
  prm.T = a.T;
  if (!tc::make_map_2d(&prm.to, a.out, F32, 4, a.n_rows, a.T, a.ldo, 32, 32))
    return cudaErrorInvalidValue;
  prm.err = tc::error_word();
  if (!prm.err) return cudaErrorInvalidDevice;
  prm.nk_main = (int32_t)((a.K + kBKm - 1) / kBKm);
  // Split the K-blocks over a cluster when the tile grid alone would leave most SMs idle (few
  // output tiles, long K): up to 8 splits, at least 4 K-blocks each, and at most ~80 CTAs in
  // all. (Measured at T 1024, K 2048, N 256: 35 us unsplit, 14 us as 4 splits over 64 CTAs,
  // 21 us as 8 splits over 128 CTAs, whose 8-SM clusters no longer fit the GPCs in one wave.)
  const int64_t tiles = ((a.n_rows + kBN - 1) / kBN) * (int64_t)(a.max_items > 0 ? a.max_items : 1);
  int splits = 1;
  while (splits < kMaxSplits && tiles * splits * 2 <= 80 && prm.nk_main >= 4 * splits * 2) splits *= 2;
  prm.kb_per_split = (prm.nk_main + splits - 1) / splits;
  prm.splits = (prm.nk_main + prm.kb_per_split - 1) / prm.kb_per_split;
  prm.lora_separate = a.lora_separate;
  prm.n_colscale = a.n_colscale;
  prm.out = reinterpret_cast<float*>(a.out);
  prm.ldo = a.ldo;
  prm.n_out = a.n_rows;
  prm.drop = a.drop;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_tc_gemm_f32, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  if (a.max_items <= 0) return cudaSuccess;
  dim3 grid((unsigned)((a.n_rows + kBN - 1) / kBN), (unsigned)a.max_items, (unsigned)prm.splits);
  prof_begin(prof_kind, st);
  cudaError_t e = cudaSuccess;
  if (prm.splits > 1) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)prm.splits;
    cfg.attrs = attr;
    cfg.numAttrs = add_pdl_attr(attr, 1);
    e = cudaLaunchKernelEx(&cfg, k_tc_gemm_f32, prm);
  } else {
    launch_kernel(k_tc_gemm_f32, grid, kThreads, kSmemBytes, st, prm);
  }
  prof_end(prof_kind, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace lora
