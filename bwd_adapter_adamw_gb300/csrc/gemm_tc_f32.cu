// Tensor-core frozen products for fp32 activations (sm_103a), 3xTF32:
//
//   out[t, n] = ( sum_k A[t, k] B[n, k] + [mask(t, n)] * sum_j P[t, j] Q_slot[n, j] ) * colscale[n]
//
// with every fp32 operand x split into x_hi = tf32(x) (round to nearest) and x_lo = x - x_hi, and
// each product formed as A_hi B_hi + A_hi B_lo + A_lo B_hi with tcgen05.mma kind::tf32 into fp32
// TMEM accumulators. The dropped A_lo B_lo term and the tf32 reading of x_lo are both O(2^-22)
// relative, so the result stays at fp32-level accuracy. (Same roles as the bf16 kernel: frozen
// forward X W^T + Hs B^T, frozen dX dY' W + (Gs A) * M; "8. LoRA Fundamentals", How it works;
// "Backward Bug Hunts and Vulkan Tiled GEMM", Bug #1.)
//
// The frozen operands arrive already split in HBM: B (W or W^T) by the weight preparation, once,
// and A (X or dY') by the streaming shrink / G kernel, which reads A anyway. So the main K-loop
// is a plain TMA -> MMA pipeline of four tiles per stage (A_hi, A_lo, B_hi, B_lo). Only the
// short LoRA K-blocks (P = Hs or Gs, Q = B or A^T, at most two 32-wide blocks) land raw and are
// split in shared memory by four converter warps.
//
// The tensor core's fp32 accumulation loses a little at every MMA, so the K-blocks are spread
// round-robin over up to four TMEM accumulators (three when the masked LoRA term needs its own)
// and summed in the epilogue with ordinary round-to-nearest fp32 adds.
//
// CTA (320 threads): warp 0 TMA, warp 1 TMEM + MMA issue, warps 2..5 epilogue, warps 6..9 LoRA
// split. Tile 128 x 128; K-block 32 fp32 = one 128-byte swizzled row; three stages of four tiles.
// (Seven stages of 16-wide K-blocks in the 64-byte swizzle measured slower: the TMA engine moves
// 64-byte rows at a lower byte rate than 128-byte rows.)
#include <cstring>
#include <mutex>

#include "tc_ptx.cuh"

namespace lora {

namespace {
using namespace tc;

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBK = 32;                        // fp32 K per K-block: one 128-byte swizzled row
constexpr int kStages = 3;
constexpr int kTile = 128 * kBK * 4;           // 128 rows x 128 bytes
constexpr int kStageBytes = 4 * kTile;         // A, A_lo, B, B_lo
constexpr int kThreads = 320;
constexpr int kConvThreads = 128;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 1024;
constexpr int kMaxLoraKb = (LORA_MAX_RANK + kBK - 1) / kBK;   // LoRA K-blocks per tile
static_assert(kSmemBytes <= 232448, "dynamic shared memory per CTA");

__device__ __forceinline__ uint64_t kdesc(uint32_t saddr) {
  return kBK == 32 ? smem_desc_sw128(saddr) : smem_desc_sw64(saddr);
}
constexpr uint32_t kIdesc = idesc(kFmtTF32, kBM, kBN);

struct F32Params {
  CUtensorMap tah, tal;               // A hi / lo [T, K] fp32, box {32, 128}
  CUtensorMap tbh, tbl;               // B hi / lo [N, K] fp32, box {32, 128}
  CUtensorMap tp;                     // P [T, ldp] fp32, box {32, 128}
  CUtensorMap tq[LORA_MAX_SLOTS];     // Q_slot [N, r] fp32, box {32, 128}
  const TokenItem* items;             // null: uniform 128-token tiles, slot 0
  const int32_t* n_items;
  int64_t T;
  uint32_t* err;
  int32_t nk_main;
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
  extern __shared__ uint8_t smem_raw[];
  TokenItem it;
  if (!get_item(p.items, p.n_items, blockIdx.y, p.T, it)) return;
  const int slot = it.slot;
  const int32_t m0 = it.t0;
  const int32_t n0 = blockIdx.x * kBN;
  const int nk_lora = (p.has_lora && slot >= 0) ? (p.q_rank[slot] + kBK - 1) / kBK : 0;
  const int nk = p.nk_main + nk_lora;
  const bool sep = p.lora_separate && nk_lora > 0;
  const uint32_t ncols = 512u;
  const int nacc = p.lora_separate ? 3 : 4;                  // main-product accumulators
  const int nused = p.nk_main < nacc ? p.nk_main : nacc;     // accumulators actually written
  const uint32_t lora_col = 384u;                            // separate LoRA accumulator

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // full_bar / empty_bar: the stage ring of the main K-blocks. The LoRA K-blocks use the same
  // stages (after empty_bar) but single-use barriers of their own, lora_full (TMA landed) and
  // lora_conv (split done), so that no wait ever targets a phase more than one ahead.
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(base + kStages * kStageBytes);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* lora_full = empty_bar + kStages;
  uint64_t* lora_conv = lora_full + kMaxLoraKb;
  uint64_t* acc_bar = lora_conv + kMaxLoraKb;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
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
    mbar_init(acc_bar, 1);
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
        if (kb < p.nk_main) {
          mbar_expect_tx(&full_bar[s], 4 * kTile);
          tma_load_2d(st, &p.tah, &full_bar[s], kb * kBK, m0);
          tma_load_2d(st + kTile, &p.tal, &full_bar[s], kb * kBK, m0);
          tma_load_2d(st + 2 * kTile, &p.tbh, &full_bar[s], kb * kBK, n0);
          tma_load_2d(st + 3 * kTile, &p.tbl, &full_bar[s], kb * kBK, n0);
        } else {
          const int j = kb - p.nk_main;
          mbar_expect_tx(&lora_full[j], 2 * kTile);
          tma_load_2d(st, &p.tp, &lora_full[j], j * kBK, m0);
          tma_load_2d(st + 2 * kTile, &p.tq[slot], &lora_full[j], j * kBK, n0);
        }
        issued = kb + 1;
      }
      // copies still in flight complete before the CTA can exit
      for (int kb = (issued > kStages ? issued - kStages : 0); kb < issued; ++kb) {
        const bool ok = kb < p.nk_main
                            ? mbar_wait(&full_bar[kb % kStages], (uint32_t)(kb / kStages) & 1u, 1u, p.err)
                            : mbar_wait(&lora_full[kb - p.nk_main], 0u, 1u, p.err);
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kStages;
        const bool lora = kb >= p.nk_main;
        // main K-blocks are consumed as landed; LoRA K-blocks once the converter has split them
        const bool ok = lora ? mbar_wait(&lora_conv[kb - p.nk_main], 0u, 2u, p.err)
                             : mbar_wait(&full_bar[s], (uint32_t)(kb / kStages) & 1u, 2u, p.err);
        if (!ok) break;
        fence_after();
        const uint32_t sa = smem_u32(base + s * kStageBytes);
        const uint64_t ah = kdesc(sa), al = kdesc(sa + kTile);
        const uint64_t bh = kdesc(sa + 2 * kTile), bl = kdesc(sa + 3 * kTile);
        const uint32_t d = lora ? (sep ? tmem + lora_col : tmem) : tmem + 128u * (uint32_t)(kb % nacc);
        const bool first = lora ? (sep && kb == p.nk_main) : (kb < nacc);
#pragma unroll
        for (int k = 0; k < kBK / 8; ++k) {
          umma_tf32(d, al + 2 * k, bh + 2 * k, kIdesc, (first && k == 0) ? 0u : 1u);
          umma_tf32(d, ah + 2 * k, bl + 2 * k, kIdesc, 1u);
          umma_tf32(d, ah + 2 * k, bh + 2 * k, kIdesc, 1u);
        }
        umma_commit(&empty_bar[s]);
      }
      umma_commit(acc_bar);
    }
  } else if (warp >= 6) {
    // LoRA K-blocks: split the landed P and Q tiles (x -> tf32(x) in place, x - tf32(x) one tile on)
    const int ct = threadIdx.x - 192;
    for (int kb = p.nk_main; kb < nk; ++kb) {
      const int s = kb % kStages;
      if (!mbar_wait(&lora_full[kb - p.nk_main], 0u, 8u, p.err)) break;
      uint8_t* st = base + s * kStageBytes;
      split_tile(st, ct);
      split_tile(st + 2 * kTile, ct);
      // generic-proxy writes must be visible to the tensor core's async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&lora_conv[kb - p.nk_main])) : "memory");
    }
  } else {
    // epilogue warps 2..5: TMEM lanes 32 * (warp % 4)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int64_t m = (int64_t)m0 + row;
    const bool row_ok = m < it.t1;
    const bool ready = __all_sync(0xffffffffu, mbar_wait(acc_bar, 0u, 4u, p.err));
    if (ready) {
      fence_after();
      for (int c = 0; c < kBN / 32; ++c) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), v);
        for (int a = 1; a < nused; ++a) {
          float u[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + 128u * (uint32_t)a + (uint32_t)(c * 32), u);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] += u[j];
        }
        if (sep) {
          float w[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + lora_col + (uint32_t)(c * 32), w);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int64_t n = (int64_t)n0 + c * 32 + j;
            if (row_ok && n < p.n_out && drop_keep(p.drop, m, n)) v[j] += w[j];
          }
        }
        const int64_t nb = (int64_t)n0 + c * 32;
        if (p.n_colscale) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= (nb + j < p.n_out) ? __ldg(p.n_colscale + nb + j) : 0.f;
        }
        if (row_ok) {
#pragma unroll
          for (int g = 0; g < 8; ++g)
            if (nb + 4 * g + 4 <= p.n_out)
              *reinterpret_cast<float4*>(p.out + m * p.ldo + nb + 4 * g) =
                  make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
        }
      }
    }
    fence_before();
  }
  __syncthreads();
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
  if (!a.a_lo || !a.b_lo) return cudaErrorInvalidValue;
  if (!tc::make_map_2d(&prm.tah, a.a, F32, 4, a.K, a.T, a.K, kBK, kBM) ||
      !tc::make_map_2d(&prm.tal, a.a_lo, F32, 4, a.K, a.T, a.K, kBK, kBM) ||
      !tc::make_map_2d(&prm.tbh, a.b, F32, 4, a.K, a.n_rows, a.K, kBK, kBN) ||
      !tc::make_map_2d(&prm.tbl, a.b_lo, F32, 4, a.K, a.n_rows, a.K, kBK, kBN))
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
  prm.err = tc::error_word();
  if (!prm.err) return cudaErrorInvalidDevice;
  prm.nk_main = (int32_t)((a.K + kBK - 1) / kBK);
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
  dim3 grid((unsigned)((a.n_rows + kBN - 1) / kBN), (unsigned)a.max_items);
  prof_begin(prof_kind, st);
  k_tc_gemm_f32<<<grid, kThreads, kSmemBytes, st>>>(prm);
  prof_end(prof_kind, st);
  return cudaGetLastError();
}

}  // namespace lora
