// Tensor-core frozen products for fp32 activations (sm_103a), 3xTF32:
//
//   out[t, n] = ( sum_k A'[t, k] B[n, k] + [mask(t, n)] * sum_j P[t, j] Q_slot[n, j] ) * colscale[n]
//
// with every fp32 operand x split in shared memory into x_hi = tf32(x) (round to nearest) and
// x_lo = x - x_hi, and each product formed as A_hi B_hi + A_hi B_lo + A_lo B_hi with
// tcgen05.mma kind::tf32 into one fp32 TMEM accumulator. The dropped A_lo B_lo term and the
// tf32 reading of x_lo are both O(2^-22) relative, so the result stays at fp32-level accuracy.
// (Same roles as the bf16 kernel: frozen forward X W^T + Hs B^T, frozen dX dY' W + (Gs A) * M;
// "8. LoRA Fundamentals", How it works; "Backward Bug Hunts and Vulkan Tiled GEMM", Bug #1.)
//
// The tensor core's fp32 accumulation loses a little at every MMA, so the K-blocks are spread
// round-robin over up to four TMEM accumulators (three when the masked LoRA term needs its own)
// and summed in the epilogue with ordinary round-to-nearest fp32 adds.
//
// CTA (320 threads): warp 0 TMA, warp 1 TMEM + MMA issue, warps 2..5 epilogue, warps 6..9 split
// each landed stage into hi (in place) and lo (a second buffer), applying A's column scale
// (DoRA dY') on the way. Tile 128 x 128, K-block 32 fp32 = one 128-byte swizzled row.
#include <cstring>
#include <mutex>

#include "tc_ptx.cuh"

namespace lora {

namespace {
using namespace tc;

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kStages = 3;
constexpr int kTile = 16384;                   // 128 rows x 128 bytes
constexpr int kStageBytes = 4 * kTile;         // A, A_lo, B, B_lo
constexpr int kThreads = 320;
constexpr int kConvThreads = 128;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 1024;
constexpr uint32_t kIdesc = idesc(kFmtTF32, kBM, kBN);

struct F32Params {
  CUtensorMap ta;                     // A [T, K] fp32, box {32, 128}
  CUtensorMap tb;                     // B [N, K] fp32, box {32, 128}
  CUtensorMap tp;                     // P [T, ldp] fp32, box {32, 128}
  CUtensorMap tq[LORA_MAX_SLOTS];     // Q_slot [N, r] fp32, box {32, 128}
  const TokenItem* items;
  const int32_t* n_items;
  uint32_t* err;
  int32_t nk_main;
  int32_t has_lora;
  int32_t lora_separate;
  int32_t q_rank[LORA_MAX_SLOTS];
  const float* a_colscale;
  const float* n_colscale;
  float* out;
  int64_t ldo;
  int64_t n_out;
  int64_t K;
  DropParams drop;
};

__device__ __forceinline__ float tf32_rn(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// Column (K index within the 32-wide block) of the float at byte offset o of a 128B-swizzled
// 128 x 128-byte tile: 16-byte chunk c' in a row holds logical chunk c' ^ (row % 8).
__device__ __forceinline__ int swz_col(int o) {
  const int row = o >> 7;
  const int chunk = ((o >> 4) & 7) ^ (row & 7);
  return chunk * 4 + ((o >> 2) & 3);
}

__global__ void __launch_bounds__(kThreads, 1) k_tc_gemm_f32(const __grid_constant__ F32Params p) {
  extern __shared__ uint8_t smem_raw[];
  const int item = blockIdx.y;
  if (item >= *p.n_items) return;
  const TokenItem it = p.items[item];
  const int slot = it.slot;
  const int32_t m0 = it.t0;
  const int32_t n0 = blockIdx.x * kBN;
  const int nk_lora = (p.has_lora && slot >= 0) ? (p.q_rank[slot] + 31) / 32 : 0;
  const int nk = p.nk_main + nk_lora;
  const bool sep = p.lora_separate && nk_lora > 0;
  const uint32_t ncols = 512u;
  const int nacc = p.lora_separate ? 3 : 4;                  // main-product accumulators
  const int nused = p.nk_main < nacc ? p.nk_main : nacc;     // accumulators actually written
  const uint32_t lora_col = 384u;                            // separate LoRA accumulator

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(base + kStages * kStageBytes);
  uint64_t* conv_bar = full_bar + kStages;
  uint64_t* empty_bar = conv_bar + kStages;
  uint64_t* acc_bar = empty_bar + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&conv_bar[s], kConvThreads);
      mbar_init(&empty_bar[s], 1);
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
        mbar_expect_tx(&full_bar[s], 2 * kTile);
        if (kb < p.nk_main) {
          tma_load_2d(st, &p.ta, &full_bar[s], kb * 32, m0);
          tma_load_2d(st + 2 * kTile, &p.tb, &full_bar[s], kb * 32, n0);
        } else {
          const int j = kb - p.nk_main;
          tma_load_2d(st, &p.tp, &full_bar[s], j * 32, m0);
          tma_load_2d(st + 2 * kTile, &p.tq[slot], &full_bar[s], j * 32, n0);
        }
        issued = kb + 1;
      }
      for (int kb = (issued > kStages ? issued - kStages : 0); kb < issued; ++kb)
        if (!mbar_wait(&full_bar[kb % kStages], (uint32_t)(kb / kStages) & 1u, 1u, p.err)) break;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kStages;
        if (!mbar_wait(&conv_bar[s], (uint32_t)(kb / kStages) & 1u, 2u, p.err)) break;
        fence_after();
        const uint32_t sa = smem_u32(base + s * kStageBytes);
        const uint64_t ah = smem_desc_sw128(sa), al = smem_desc_sw128(sa + kTile);
        const uint64_t bh = smem_desc_sw128(sa + 2 * kTile), bl = smem_desc_sw128(sa + 3 * kTile);
        const bool lora = kb >= p.nk_main;
        const uint32_t d = lora ? (sep ? tmem + lora_col : tmem) : tmem + 128u * (uint32_t)(kb % nacc);
        const bool first = lora ? (sep && kb == p.nk_main) : (kb < nacc);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          umma_tf32(d, al + 2 * k, bh + 2 * k, kIdesc, (first && k == 0) ? 0u : 1u);
          umma_tf32(d, ah + 2 * k, bl + 2 * k, kIdesc, 1u);
          umma_tf32(d, ah + 2 * k, bh + 2 * k, kIdesc, 1u);
        }
        umma_commit(&empty_bar[s]);
      }
      umma_commit(acc_bar);
    }
  } else if (warp >= 6) {
    // split landed stages: x -> (tf32(x) in place, x - tf32(x) one tile further)
    const int ct = threadIdx.x - 192;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kStages;
      if (!mbar_wait(&full_bar[s], (uint32_t)(kb / kStages) & 1u, 8u, p.err)) break;
      uint8_t* st = base + s * kStageBytes;
      const bool scale = p.a_colscale && kb < p.nk_main;
#pragma unroll 4
      for (int i = ct; i < 2 * kTile / 16; i += kConvThreads) {
        const int tile = i >= kTile / 16 ? 2 : 0;            // A or B
        const int o = (i % (kTile / 16)) * 16;
        float4* hi = reinterpret_cast<float4*>(st + tile * kTile + o);
        float4* lo = reinterpret_cast<float4*>(st + (tile + 1) * kTile + o);
        float4 v = *hi;
        if (scale && tile == 0) {
          const int64_t k = (int64_t)kb * 32 + swz_col(o);
          v.x *= (k < p.K) ? __ldg(p.a_colscale + k) : 0.f;
          v.y *= (k + 1 < p.K) ? __ldg(p.a_colscale + k + 1) : 0.f;
          v.z *= (k + 2 < p.K) ? __ldg(p.a_colscale + k + 2) : 0.f;
          v.w *= (k + 3 < p.K) ? __ldg(p.a_colscale + k + 3) : 0.f;
        }
        const float4 h = make_float4(tf32_rn(v.x), tf32_rn(v.y), tf32_rn(v.z), tf32_rn(v.w));
        *hi = h;
        *lo = make_float4(v.x - h.x, v.y - h.y, v.z - h.z, v.w - h.w);
      }
      // generic-proxy writes must be visible to the tensor core's async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&conv_bar[s])) : "memory");
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
  if (!tc::make_map_2d(&prm.ta, a.a, F32, 4, a.K, a.T, a.K, 32, kBM) ||
      !tc::make_map_2d(&prm.tb, a.b, F32, 4, a.K, a.n_rows, a.K, 32, kBN))
    return cudaErrorInvalidValue;
  prm.has_lora = a.p != nullptr;
  if (a.p) {
    if (!tc::make_map_2d(&prm.tp, a.p, F32, 4, a.ldp, a.T, a.ldp, 32, kBM)) return cudaErrorInvalidValue;
    for (int k = 0; k < a.n_slots; ++k) {
      prm.q_rank[k] = a.q_rank[k];
      if (!tc::make_map_2d(&prm.tq[k], a.q[k], F32, 4, a.q_rank[k], a.n_rows, a.q_rank[k], 32, kBN))
        return cudaErrorInvalidValue;
    }
  }
  prm.items = a.items;
  prm.n_items = a.n_items;
  prm.err = tc::error_word();
  if (!prm.err) return cudaErrorInvalidDevice;
  prm.nk_main = (int32_t)((a.K + 31) / 32);
  prm.lora_separate = a.lora_separate;
  prm.a_colscale = a.a_colscale;
  prm.n_colscale = a.n_colscale;
  prm.out = reinterpret_cast<float*>(a.out);
  prm.ldo = a.ldo;
  prm.n_out = a.n_rows;
  prm.K = a.K;
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
