// Tensor-core frozen products for bf16 activations on sm_103a: TMA -> shared-memory ring ->
// tcgen05.mma -> TMEM -> epilogue.
//
//   out[t, n] = ( sum_k A[t, k] B[n, k]                      (kind::f16, bf16 operands)
//               + [mask(t, n)] * sum_j P[t, j] Q_slot[n, j] ) (kind::tf32, the fp32 LoRA term)
//               * colscale[n]
//
// for the tokens of one work item (<= 128 tokens, one adapter slot). The frozen forward uses
// A = X, B = W, P = Hs, Q = B_slot (the up-projection as extra K-steps into the same TMEM
// accumulator); the frozen dX uses A = dY', B = W^T, P = Gs, Q = A_slot^T, and when dropout is
// on the LoRA term goes to its own TMEM columns so that the epilogue can mask it
// ("8. LoRA Fundamentals", How it works: W_eff = W + s B A; "Backward Bug Hunts and Vulkan
// Tiled GEMM", Bug #1: the activation gradient through the frozen weight).
//
// CTA layout (192 threads): warp 0 issues TMA loads, warp 1 allocates TMEM and issues the MMAs
// (one thread), warps 2..5 drain the accumulator (one TMEM lane = one output row per thread)
// and store it through shared-memory boxes with bulk tensor stores. Tile 128 x BN (BN 256, 224
// or 192), K-block 64 bf16 / 128 E4M3 (32 fp32 for the LoRA blocks) = one 128-byte swizzled
// row. Persistent CTAs, one per SM. Every mbarrier wait is bounded; on timeout the kernel records
// an error bit and unwinds.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "tc_ptx.cuh"

namespace lora {
namespace tc {
namespace {
__device__ uint32_t g_tc_error = 0;
std::mutex g_err_mu;
uint32_t* g_err_ptr[64] = {};
}  // namespace

uint32_t* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tc_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<uint32_t*>(p);
  }
  return g_err_ptr[dev];
}
}  // namespace tc

namespace {
using namespace tc;

constexpr int kBM = 128;
constexpr int kABytes = kBM * 128;   // 16 KB: 128 rows x 128 bytes
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
// Epilogue store boxes: each epilogue warp stages 32 rows x 32 bf16 columns (64-byte rows,
// 64-byte swizzle) and writes them with one bulk tensor store, alternating between two boxes so
// that one store can still be reading while the next box fills. At BN 224 the boxes would cost
// the fifth pipeline stage, which is worth more: that width stores row by row.
constexpr int kEpiBox = 32 * 64;
template <int BN>
constexpr int epi_bytes() { return BN == 224 ? 0 : 4 * 2 * kEpiBox; }
// Items per tile group (rasterization for L2 reuse): 32 when W spans more than 16 N tiles; with
// fewer, the N tile runs fastest (group of 1), so that the CTAs of one wave read all of W
// together. Measured at T 8192 (us): N 4096 / K 4096: 152 (N fastest), 152 (8), 162 (16);
// N 14336 / K 4096: 688, 585, 550 (16); N 4096 / K 14336: 542, 566, 557. Later, cold in one
// capture, N 14336 / K 4096 (and the dX of K 14336 back to N 14336): 577 us and 555 MB of DRAM
// reads with groups of 16, 566 / 436 MB with 24, 564 / 330 MB with 32, 603 / 1399 MB with 64
// (the band of W no longer fits L2). (A threshold of 32 tiles left c3, T 4096 / N 4096 at 19
// tiles of 224, unchanged.)
constexpr int kGroupWide = 32;
constexpr int kGroupMinTiles = 16;

// Tile 128 x BN. BN = 256 is the fastest MMA shape per flop; 224 and 192 (the same kernel with
// narrower B tiles and accumulators) let the host trade a little MMA rate for fewer idle SMs in
// the last round of tiles.
template <int BN>
struct GemmCfg {
  static_assert(BN % 32 == 0 && BN >= 128 && BN <= 256, "tile width");
  static constexpr int kBBytes = BN * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kEpiBytes = epi_bytes<BN>();
  // as many stages as fit beside the epilogue's store boxes (4 at BN 256, 5 at 224 and 192)
  static constexpr int kStageRoom = 227 * 1024 - kEpiBytes - 2048;
  static constexpr int kStages = (kStageRoom / kStageBytes) < 6 ? (kStageRoom / kStageBytes) : 6;
  static constexpr int kSmemBytes =
      kStages * kStageBytes + kEpiBytes + 1024 /*barriers*/ + 1024 /*alignment*/;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kIdescBF16 = tc::idesc(tc::kFmtBF16, kBM, BN);
  static constexpr uint32_t kIdescE4M3 = tc::idesc(tc::kFmtE4M3, kBM, BN);
  static constexpr uint32_t kIdescTF32 = tc::idesc(tc::kFmtTF32, kBM, BN);
  static_assert(kStageBytes % 1024 == 0, "stage alignment of the 128-byte swizzle");
};

struct TcParams {
  CUtensorMap ta;                       // A [rows, K] bf16, box {64, 128}
  CUtensorMap tb;                       // B [N, K] bf16, box {64, BN}
  CUtensorMap tp;                       // P [T, ldp] fp32, box {32, 128}
  CUtensorMap tq[LORA_MAX_SLOTS];       // Q_slot [N, r] fp32, box {32, BN}
  CUtensorMap to;                       // out [T, N] bf16, box {32, 32} (the epilogue's stores)
  const TokenItem* items;               // null: uniform 128-token tiles, slot 0
  const int32_t* n_items;
  int64_t T;
  int32_t n_tiles;                      // N tiles per item
  int32_t max_items;                    // item slots
  int32_t group_m;                      // items per tile group
  int32_t total_tiles;                  // n_tiles x item slots
  uint32_t* err;
  unsigned long long wait_limit;        // bound of the pipeline waits (cycles); drains keep kWaitCycles
  int32_t nk_main;
  int32_t has_lora;
  int32_t lora_separate;
  int32_t q_rank[LORA_MAX_SLOTS];
  const uint32_t* tile_mask;            // routed uniform tiles: slots present per 128-token tile
  int32_t slot_pcol[LORA_MAX_SLOTS];
  int32_t slot_qx[LORA_MAX_SLOTS];
  int32_t slot_qmap[LORA_MAX_SLOTS];
  int32_t n_col_groups;                 // > 0: the adapter is chosen by output column, not token
  int32_t col_end[LORA_MAX_SLOTS];      // group k covers columns [col_end[k-1], col_end[k])
  int32_t p_col[LORA_MAX_SLOTS];        // group k's LoRA operand starts at column p_col[k] of P
  const float* n_colscale;
  const float* m_rowscale;
  void* out;
  int64_t ldo;
  int64_t n_out;
  DropParams drop;
};

// ---- the kernel ---------------------------------------------------------------------------
// Persistent: CTA b takes tiles b, b + gridDim.x, ... Tiles are ordered in groups of group_m items:
// within a group the item index runs fastest, then the N tile, so that for a wide W one wave of
// CTAs touches group_m items of A and about 152 / group_m N-tiles of W, which both stay in L2
// (with the N tile fastest, every few items would stream all of a wide W from HBM again). The
// stage ring runs on across tiles, and two
// 256-column TMEM accumulators alternate between tiles, so that the epilogue of one tile drains
// and stores while the MMAs of the next run. With a dropout-masked LoRA term the second 256
// columns hold that term instead, and tiles take turns on one accumulator.
// The adapter of a tile, the column of P where its LoRA operand starts and the first output
// column of its Q: the item's slot, or, for fused projections, the column group that holds the
// tile's first output column (whose Q rows count from the group's first column).
__device__ __forceinline__ int tile_slot(const TcParams& p, const TokenItem& it, int32_t n0,
                                         int& pcol, int& qcol0) {
  pcol = 0;
  qcol0 = 0;
  if (p.n_col_groups <= 0) return it.slot;
  int k = 0;
  while (k + 1 < p.n_col_groups && n0 >= p.col_end[k]) ++k;
  pcol = p.p_col[k];
  qcol0 = k > 0 ? p.col_end[k - 1] : 0;
  return k;
}

// LoRA K-blocks of a tile: from the item's slot (token-routed items), the column group holding
// the tile (fused projections), or every slot present in a uniform tile of a routed call
// (tile_mask: each slot's operand occupies its own column block of P, zero at the other slots'
// tokens, so the slots' terms add up in one accumulator).
struct LoraTile {
  uint32_t mask;
  int slot;
  int pcol;
  int qrow0;
};

__device__ __forceinline__ int lora_tile(const TcParams& p, const TokenItem& it, int32_t n0,
                                         LoraTile& lt) {
  lt.mask = 0;
  lt.slot = -1;
  lt.pcol = 0;
  lt.qrow0 = 0;
  if (!p.has_lora) return 0;
  if (p.tile_mask) {
    lt.mask = p.tile_mask[it.t0 / kBM];
    int nb = 0;
    for (uint32_t m = lt.mask; m; m &= m - 1) nb += (p.q_rank[__ffs(m) - 1] + 31) / 32;
    return nb;
  }
  lt.slot = tile_slot(p, it, n0, lt.pcol, lt.qrow0);
  return lt.slot >= 0 ? (p.q_rank[lt.slot] + 31) / 32 : 0;
}

// Tensor map and coordinates of LoRA K-block jj of a tile.
__device__ __forceinline__ void lora_block(const TcParams& p, const LoraTile& lt, int jj,
                                           int& qmap, int& px, int& qx, int& qrow0) {
  if (!lt.mask) {
    qmap = lt.slot;
    px = lt.pcol + 32 * jj;
    qx = 32 * jj;
    qrow0 = lt.qrow0;
    return;
  }
  uint32_t m = lt.mask;
  int sl = __ffs(m) - 1;
  for (;;) {
    const int nb = (p.q_rank[sl] + 31) / 32;
    if (jj < nb) break;
    jj -= nb;
    m &= m - 1;
    sl = __ffs(m) - 1;
  }
  qmap = p.slot_qmap[sl];
  px = p.slot_pcol[sl] + 32 * jj;
  qx = p.slot_qx[sl] + 32 * jj;
  qrow0 = 0;
}

// Tile t of the persistent schedule: its work item and first output column.
template <int BN>
__device__ __forceinline__ bool decode_tile(const TcParams& p, int t, TokenItem& it, int32_t& n0) {
  const int per_group = p.group_m * p.n_tiles;
  const int group = t / per_group;
  const int first = group * p.group_m;
  const int gsize = min(p.group_m, p.max_items - first);
  const int idx = t - group * per_group;
  n0 = (idx / gsize) * BN;
  return get_item(p.items, p.n_items, first + idx % gsize, p.T, it);
}

// F8: the main K-blocks are E4M3 codes (128 per 128-byte row, kind::f8f6f4); the accumulator is
// then in code units and the epilogue multiplies by the row and column scales. The LoRA K-blocks
// arrive pre-divided by the same scales, so that they share the accumulator.
template <int BN, bool F8>
__global__ void __launch_bounds__(kThreads, 1) k_tc_gemm(const __grid_constant__ TcParams p) {
  // The set-up below (barriers, TMEM, tensor-map prefetch) touches nothing that an earlier kernel
  // writes, so it runs before grid_dep_sync() and overlaps the previous kernel's tail.
  using C = GemmCfg<BN>;
  const int t_first = (int)blockIdx.x;
  const int t_step = (int)gridDim.x;
  constexpr int kStages = C::kStages;
  constexpr int kStageBytes = C::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = base;
  uint8_t* epi_boxes = base + kStages * kStageBytes;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(epi_boxes + C::kEpiBytes);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* acc_full = empty_bar + kStages;   // [2]: a tile's accumulation is complete
  uint64_t* acc_empty = acc_full + 2;         // [2]: the epilogue has drained the accumulator
  uint64_t* mma_done = acc_empty + 2;         // every MMA this CTA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t ncols = 512u;
  const int nbuf = p.lora_separate ? 1 : 2;

  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.ta)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tb)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.to)) : "memory");
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiThreads);
    }
    mbar_init(mma_done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, ncols);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_sync();   // from here on, the earlier kernels' outputs are visible

  if (warp == 0) {
    if (lane == 0) {
      int g = 0;   // stage uses so far (across tiles)
      bool ok = true;
      for (int t = t_first; t < p.total_tiles && ok; t += t_step) {
        TokenItem it;
        int32_t n0;
        if (!decode_tile<BN>(p, t, it, n0)) continue;
        LoraTile lt;
        const int nk = p.nk_main + lora_tile(p, it, n0, lt);
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = g % kStages;
          const uint32_t ph = (uint32_t)(g / kStages) & 1u;
          if (g >= kStages && !mbar_wait_for(&empty_bar[s], ph ^ 1u, 1u, p.err, p.wait_limit)) {
            ok = false;
            break;
          }
          uint8_t* sa = tiles + s * kStageBytes;
          uint8_t* sb = sa + kABytes;
          mbar_expect_tx(&full_bar[s], kStageBytes);
          if (kb < p.nk_main) {
            constexpr int kKBlock = F8 ? 128 : 64;   // elements in one 128-byte row
            tma_load_2d(sa, &p.ta, &full_bar[s], kb * kKBlock, it.t0);
            tma_load_2d(sb, &p.tb, &full_bar[s], kb * kKBlock, n0);
          } else {
            int qmap, px, qx, qrow0;
            lora_block(p, lt, kb - p.nk_main, qmap, px, qx, qrow0);
            tma_load_2d(sa, &p.tp, &full_bar[s], px, it.t0);
            tma_load_2d(sb, &p.tq[qmap], &full_bar[s], qx, n0 - qrow0);
          }
        }
      }
      // drain: every issued load must have landed before the CTA may exit
      for (int gg = (g > kStages ? g - kStages : 0); gg < g; ++gg) {
        const uint32_t par = (uint32_t)(gg / kStages) & 1u;
        if (!mbar_wait(&full_bar[gg % kStages], par, 1u, p.err)) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int g = 0, j = 0;
      bool ok = true;
      for (int t = t_first; t < p.total_tiles && ok; t += t_step) {
        TokenItem it;
        int32_t n0;
        if (!decode_tile<BN>(p, t, it, n0)) continue;
        LoraTile lt;
        const int nk_lora = lora_tile(p, it, n0, lt);
        const int nk = p.nk_main + nk_lora;
        const bool sep = p.lora_separate && nk_lora > 0;
        const int b = j % nbuf, use = j / nbuf;
        if (use >= 1 && !mbar_wait_for(&acc_empty[b], (uint32_t)(use - 1) & 1u, 2u, p.err, p.wait_limit))
          break;
        fence_after();
        const uint32_t dm = tmem + 256u * (uint32_t)b;
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = g % kStages;
          const uint32_t ph = (uint32_t)(g / kStages) & 1u;
          if (!mbar_wait_for(&full_bar[s], ph, 2u, p.err, p.wait_limit)) { ok = false; break; }
          fence_after();
          const uint32_t sa = smem_u32(tiles + s * kStageBytes);
          const uint32_t sb = sa + kABytes;
          const uint64_t da = smem_desc_sw128(sa), db = smem_desc_sw128(sb);
          if (kb < p.nk_main) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if constexpr (F8)
                umma_f8(dm, da + 2 * k, db + 2 * k, C::kIdescE4M3, (kb > 0 || k > 0) ? 1u : 0u);
              else
                umma_f16(dm, da + 2 * k, db + 2 * k, C::kIdescBF16, (kb > 0 || k > 0) ? 1u : 0u);
          } else {
            const uint32_t d = sep ? tmem + 256u : dm;
            const bool first = sep && kb == p.nk_main;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_tf32(d, da + 2 * k, db + 2 * k, C::kIdescTF32, (first && k == 0) ? 0u : 1u);
          }
          umma_commit(&empty_bar[s]);
        }
        if (!ok) break;
        umma_commit(&acc_full[b]);
        ++j;
      }
      // every MMA issued above has completed before the tensor memory is freed (after an early
      // exit nothing else waits for them)
      umma_commit(mma_done);
      mbar_wait(mma_done, 0u, 2u, p.err);
    }
  } else {
    // epilogue: warp w drains TMEM lanes 32*(w % 4) .. +31 (one output row per thread)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
    uint8_t* boxes = epi_boxes + (warp - 2) * 2 * kEpiBox;
    int nbox = 0;   // boxes filled so far by this warp
    int j = 0;
    for (int t = t_first; t < p.total_tiles; t += t_step) {
      TokenItem it;
      int32_t n0;
      if (!decode_tile<BN>(p, t, it, n0)) continue;
      LoraTile lt;
      const bool sep = p.lora_separate && lora_tile(p, it, n0, lt) > 0;
      const int b = j % nbuf, use = j / nbuf;
      const int64_t m = (int64_t)it.t0 + row;
      const bool row_ok = m < it.t1;
      // dropout keep bits of this row's BN columns, evaluated while the tile's MMAs still run
      uint32_t keep[BN / 32];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) keep[c] = 0u;
      if (sep && row_ok) {
        const DropRow drow = drop_row(p.drop, m);
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
#pragma unroll 4
          for (int jj = 0; jj < 32; ++jj) {
            const int64_t n = (int64_t)n0 + c * 32 + jj;
            if (n < p.n_out && drop_keep_at(drow, p.drop.tau, n)) keep[c] |= 1u << jj;
          }
        }
      }
      // warp-uniform decision: the TMEM loads below are .sync.aligned
      const bool ready =
          __all_sync(0xffffffffu, mbar_wait_for(&acc_full[b], (uint32_t)use & 1u, 4u, p.err, p.wait_limit));
      if (!ready) break;
      fence_after();
      const uint32_t acc = tmem + ((uint32_t)(q * 32) << 16) + 256u * (uint32_t)b;
      // This warp's 32 rows leave through bulk tensor stores when they all lie in the item, or
      // when the end of the tensor clips them; a partial item of a routed call stores row by
      // row (the rows past it belong to other CTAs).
      const int64_t wrow0 = (int64_t)it.t0 + q * 32;
      const bool box_store = C::kEpiBytes > 0 && wrow0 < it.t1 &&
                             (wrow0 + 32 <= it.t1 || (int64_t)it.t1 == p.T);
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tmem_ld32(acc + (uint32_t)(c * 32), v);
        if (sep) {
          float w[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + 256u + (uint32_t)(c * 32), w);
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            if ((keep[c] >> jj) & 1u) v[jj] += w[jj];
        }
        const int64_t nb = (int64_t)n0 + c * 32;
        if (p.m_rowscale && row_ok) {
          const float rs = __ldg(p.m_rowscale + m);
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) v[jj] *= rs;
        }
        if (p.n_colscale) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            v[jj] *= (nb + jj < p.n_out) ? __ldg(p.n_colscale + nb + jj) : 0.f;
        }
        if (box_store) {
          // the store issued from this box two boxes ago has read it
          uint8_t* box = boxes + (nbox & 1) * kEpiBox;
          ++nbox;
          if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          __syncwarp();
          uint8_t* rowp = box + lane * 64;
#pragma unroll
          for (int gq = 0; gq < 4; ++gq)
            store8(reinterpret_cast<__nv_bfloat16*>(rowp + ((gq ^ ((lane >> 1) & 3)) << 4)), v + gq * 8);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&p.to, box, (int32_t)nb, (int32_t)wrow0);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
        } else if (row_ok) {
#pragma unroll
          for (int gq = 0; gq < 4; ++gq)
            if (nb + gq * 8 + 8 <= p.n_out) store8(out + m * p.ldo + nb + gq * 8, v + gq * 8);
        }
      }
      fence_before();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&acc_empty[b])) : "memory");
      ++j;
    }
    // the bulk stores have written their rows before the kernel completes
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
    fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// ---- host side ----------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace

namespace tc {
int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

bool make_map_2d(CUtensorMap* map, const void* ptr, CUtensorMapDataType dt, int elem, uint64_t inner,
              uint64_t outer, uint64_t row_elems, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_elems * (uint64_t)elem};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  // the box row decides the swizzle: 128-byte rows -> 128B, 64-byte rows -> 64B
  const uint32_t row_bytes = box_inner * (uint32_t)elem;
  if (row_bytes != 128 && row_bytes != 64) return false;
  const CUtensorMapSwizzle swz = row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return fn(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

namespace {
template <int BN, bool F8>
cudaError_t launch_gemm_bn(unsigned grid, cudaStream_t st, const TcParams& prm) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_tc_gemm<BN, F8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         GemmCfg<BN>::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_kernel(k_tc_gemm<BN, F8>, grid, kThreads, GemmCfg<BN>::kSmemBytes, st, prm);
}

// Tile width: the fewest tile-columns of MMA work per SM, rounds x BN x (relative cost of a
// column at that width), over the persistent CTAs' rounds of tiles.
int pick_tile_n(int64_t n_rows, int64_t items, int sms) {
  static const int kWidths[] = {256, 224, 192};
  static const double kColumnCost[] = {1.0, 1.10, 1.17};   // measured per-column MMA time
  int best = 256;
  double best_cost = 1e300;
  for (int i = 0; i < 3; ++i) {
    const int64_t tiles = items * ((n_rows + kWidths[i] - 1) / kWidths[i]);
    const int64_t rounds = (tiles + sms - 1) / sms;
    const double cost = (double)rounds * kWidths[i] * kColumnCost[i];
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best = kWidths[i];
    }
  }
  return best;
}

std::atomic<unsigned long long> g_wait_limit{0};   // pipeline-wait bound in cycles; 0: the default
}  // namespace

void set_tc_wait_limit(unsigned long long cycles) { g_wait_limit.store(cycles); }

cudaError_t launch_tc_gemm(const TcGemmArgs& a, cudaStream_t st, int prof_kind) {
  static TcParams prm;   // large: filled per call on the host, copied into the launch
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  std::memset(&prm, 0, sizeof(prm));
  const int sms = tc::sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  // column groups must start on tile boundaries: fused projections use 256-wide tiles
  const int bn = a.n_col_groups > 0 ? 256 : pick_tile_n(a.n_rows, a.max_items, sms);
  if (a.n_col_groups > 0) {
    if (a.n_col_groups > LORA_MAX_SLOTS || a.n_col_groups != a.n_slots) return cudaErrorInvalidValue;
    for (int k = 0; k < a.n_col_groups; ++k)
      if (a.col_end[k] % 256 || (k > 0 && a.col_end[k] <= a.col_end[k - 1]) || a.p_col[k] % 4)
        return cudaErrorInvalidValue;
    if (a.col_end[a.n_col_groups - 1] != a.n_rows) return cudaErrorInvalidValue;
  }
  // one 128-byte row per K-block: 64 bf16 or 128 E4M3 codes
  const CUtensorMapDataType adt = a.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int esz = a.fp8 ? 1 : 2, kblk = a.fp8 ? 128 : 64;
  const uint32_t b_rows = (uint32_t)bn;
  if (!tc::make_map_2d(&prm.ta, a.a, adt, esz, a.K, a.T, a.K, kblk, kBM) ||
      !tc::make_map_2d(&prm.tb, a.b, adt, esz, a.K, a.n_rows, a.K, kblk, b_rows))
    return cudaErrorInvalidValue;
  prm.has_lora = a.p != nullptr;
  if (a.p) {
    if (!tc::make_map_2d(&prm.tp, a.p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.ldp, a.T, a.ldp, 32, kBM))
      return cudaErrorInvalidValue;
    for (int k = 0; k < a.n_slots; ++k) prm.q_rank[k] = a.q_rank[k];
    const int n_maps = a.n_q_maps > 0 ? a.n_q_maps : a.n_slots;
    for (int k = 0; k < n_maps; ++k) {
      const int64_t q_in = a.q_inner[k] > 0 ? a.q_inner[k] : a.q_rank[k];
      // Q_k has the output rows of its column group (fused projections) or all of them
      const int64_t q_rows = a.n_col_groups > 0
                                 ? a.col_end[k] - (k > 0 ? a.col_end[k - 1] : 0)
                                 : a.n_rows;
      if (!tc::make_map_2d(&prm.tq[k], a.q[k], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, q_in, q_rows,
                    q_in, 32, b_rows))
        return cudaErrorInvalidValue;
    }
  }
  prm.items = a.items;
  prm.n_items = a.n_items;
  prm.T = a.T;
  if (!tc::make_map_2d(&prm.to, a.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.n_rows, a.T, a.ldo, 32,
                       32))
    return cudaErrorInvalidValue;
  prm.err = tc::error_word();
  if (!prm.err) return cudaErrorInvalidDevice;
  const unsigned long long lim = g_wait_limit.load();
  prm.wait_limit = lim ? lim : tc::kWaitCycles;
  prm.nk_main = (int32_t)((a.K + kblk - 1) / kblk);
  prm.lora_separate = a.lora_separate;
  prm.n_colscale = a.n_colscale;
  prm.m_rowscale = a.m_rowscale;
  prm.tile_mask = a.tile_mask;
  if (a.tile_mask) {
    if (a.items) return cudaErrorInvalidValue;   // slot sets need uniform tiles
    for (int k = 0; k < a.n_slots; ++k) {
      prm.slot_pcol[k] = a.slot_pcol[k];
      prm.slot_qx[k] = a.slot_qx[k];
      prm.slot_qmap[k] = a.slot_qmap[k];
      if (a.slot_pcol[k] % 4 || a.slot_qx[k] % 4 || a.slot_qmap[k] < 0 ||
          a.slot_qmap[k] >= (a.n_q_maps > 0 ? a.n_q_maps : a.n_slots))
        return cudaErrorInvalidValue;
    }
  }
  prm.n_col_groups = a.n_col_groups;
  for (int k = 0; k < a.n_col_groups; ++k) {
    prm.col_end[k] = (int32_t)a.col_end[k];
    prm.p_col[k] = a.p_col[k];
  }
  prm.out = a.out;
  prm.ldo = a.ldo;
  prm.n_out = a.n_rows;
  prm.drop = a.drop;
  if (a.max_items <= 0) return cudaSuccess;
  prm.n_tiles = (int32_t)((a.n_rows + bn - 1) / bn);
  prm.max_items = a.max_items;
  // tile groups for L2 reuse, counted in items
  prm.group_m = prm.n_tiles > kGroupMinTiles ? kGroupWide : 1;
  const int64_t total = (int64_t)prm.n_tiles * a.max_items;
  if (total > INT32_MAX) return cudaErrorInvalidValue;
  prm.total_tiles = (int32_t)total;
  // one persistent CTA per SM
  const unsigned grid = (unsigned)(total < sms ? total : sms);
  prof_begin(prof_kind, st);
  cudaError_t e = cudaErrorInvalidValue;
  switch (bn * 2 + (a.fp8 ? 1 : 0)) {
    case 512: e = launch_gemm_bn<256, false>(grid, st, prm); break;
    case 448: e = launch_gemm_bn<224, false>(grid, st, prm); break;
    case 384: e = launch_gemm_bn<192, false>(grid, st, prm); break;
    case 513: e = launch_gemm_bn<256, true>(grid, st, prm); break;
    case 449: e = launch_gemm_bn<224, true>(grid, st, prm); break;
    case 385: e = launch_gemm_bn<192, true>(grid, st, prm); break;
  }
  if (e != cudaSuccess) return e;
  prof_end(prof_kind, st);
  return cudaGetLastError();
}

cudaError_t read_tc_error(uint32_t* out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, tc::g_tc_error, sizeof(uint32_t));
  if (e != cudaSuccess || !reset) return e;
  const uint32_t zero = 0;
  return cudaMemcpyToSymbol(tc::g_tc_error, &zero, sizeof(uint32_t));
}

}  // namespace lora
