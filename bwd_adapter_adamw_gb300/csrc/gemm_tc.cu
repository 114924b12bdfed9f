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
// (one thread), warps 2..5 drain the accumulator (one TMEM lane = one output row per thread).
// Tile 128 x 256, K-block 64 bf16 (32 fp32 for the LoRA blocks) = one 128-byte swizzled row.
// Every mbarrier wait is bounded; on timeout the kernel records an error bit and unwinds.
#include <cudaTypedefs.h>

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
constexpr int kBN = 256;
constexpr int kStages = 4;
constexpr int kABytes = kBM * 128;   // 16 KB: 128 rows x 128 bytes
constexpr int kBBytes = kBN * 128;   // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*barriers*/ + 1024 /*alignment*/;
constexpr uint32_t kIdescBF16 = tc::idesc(tc::kFmtBF16, kBM, kBN);
constexpr uint32_t kIdescTF32 = tc::idesc(tc::kFmtTF32, kBM, kBN);

struct TcParams {
  CUtensorMap ta;                       // A [rows, K] bf16, box {64, 128}
  CUtensorMap tb;                       // B [N, K] bf16, box {64, 256}
  CUtensorMap tp;                       // P [T, ldp] fp32, box {32, 128}
  CUtensorMap tq[LORA_MAX_SLOTS];       // Q_slot [N, r] fp32, box {32, 256}
  const TokenItem* items;               // null: uniform 128-token tiles, slot 0
  const int32_t* n_items;
  int64_t T;
  uint32_t* err;
  int32_t nk_main;
  int32_t has_lora;
  int32_t lora_separate;
  int32_t q_rank[LORA_MAX_SLOTS];
  const float* n_colscale;
  void* out;
  int64_t ldo;
  int64_t n_out;
  DropParams drop;
};

// ---- the kernel ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) k_tc_gemm(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  TokenItem it;
  if (!get_item(p.items, p.n_items, blockIdx.y, p.T, it)) return;
  const int slot = it.slot;
  const int32_t m0 = it.t0;
  const int32_t n0 = blockIdx.x * kBN;
  const int nk_lora = (p.has_lora && slot >= 0) ? (p.q_rank[slot] + 31) / 32 : 0;
  const int nk = p.nk_main + nk_lora;
  const bool sep = p.lora_separate && nk_lora > 0;

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = base;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(base + kStages * kStageBytes);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* acc_bar = empty_bar + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t ncols = p.lora_separate ? 512u : 256u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
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
        uint8_t* sa = tiles + s * kStageBytes;
        uint8_t* sb = sa + kABytes;
        mbar_expect_tx(&full_bar[s], kStageBytes);
        if (kb < p.nk_main) {
          tma_load_2d(sa, &p.ta, &full_bar[s], kb * 64, m0);
          tma_load_2d(sb, &p.tb, &full_bar[s], kb * 64, n0);
        } else {
          const int j = kb - p.nk_main;
          tma_load_2d(sa, &p.tp, &full_bar[s], j * 32, m0);
          tma_load_2d(sb, &p.tq[slot], &full_bar[s], j * 32, n0);
        }
        issued = kb + 1;
      }
      // drain: every issued load must have landed before the CTA may exit
      for (int kb = (issued > kStages ? issued - kStages : 0); kb < issued; ++kb)
        if (!mbar_wait(&full_bar[kb % kStages], (uint32_t)(kb / kStages) & 1u, 1u, p.err)) break;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = true;
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % kStages;
        const uint32_t ph = (uint32_t)(kb / kStages) & 1u;
        if (!mbar_wait(&full_bar[s], ph, 2u, p.err)) { ok = false; break; }
        fence_after();
        const uint32_t sa = smem_u32(tiles + s * kStageBytes);
        const uint32_t sb = sa + kABytes;
        const uint64_t da = smem_desc_sw128(sa), db = smem_desc_sw128(sb);
        if (kb < p.nk_main) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_f16(tmem, da + 2 * k, db + 2 * k, kIdescBF16, (kb > 0 || k > 0) ? 1u : 0u);
        } else {
          const uint32_t d = sep ? tmem + 256u : tmem;
          const bool first = sep && kb == p.nk_main;
#pragma unroll
          for (int k = 0; k < 4; ++k) umma_tf32(d, da + 2 * k, db + 2 * k, kIdescTF32, (first && k == 0) ? 0u : 1u);
        }
        umma_commit(&empty_bar[s]);
      }
      umma_commit(acc_bar);
    }
  } else {
    // epilogue: warp w drains TMEM lanes 32*(w % 4) .. +31 (one output row per thread)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int64_t m = (int64_t)m0 + row;
    const bool row_ok = m < it.t1;
    // warp-uniform decision: the TMEM loads below are .sync.aligned
    const bool ready = __all_sync(0xffffffffu, mbar_wait(acc_bar, 0u, 4u, p.err));
    if (ready) {
      fence_after();
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
      for (int c = 0; c < kBN / 32; ++c) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), v);
        if (sep) {
          float w[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + 256u + (uint32_t)(c * 32), w);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int64_t n = (int64_t)n0 + c * 32 + j;
            if (row_ok && n < p.n_out && drop_keep(p.drop, m, n)) v[j] += w[j];
          }
        }
        const int64_t nb = (int64_t)n0 + c * 32;
        if (p.n_colscale) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            v[j] *= (nb + j < p.n_out) ? __ldg(p.n_colscale + nb + j) : 0.f;
        }
        if (row_ok) {
#pragma unroll
          for (int g = 0; g < 4; ++g)
            if (nb + g * 8 + 8 <= p.n_out) store8(out + m * p.ldo + nb + g * 8, v + g * 8);
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

cudaError_t launch_tc_gemm(const TcGemmArgs& a, cudaStream_t st, int prof_kind) {
  static TcParams prm;   // large: filled per call on the host, copied into the launch
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  std::memset(&prm, 0, sizeof(prm));
  if (!tc::make_map_2d(&prm.ta, a.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.K, a.T, a.K, 64, kBM) ||
      !tc::make_map_2d(&prm.tb, a.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.K, a.n_rows, a.K, 64, kBN))
    return cudaErrorInvalidValue;
  prm.has_lora = a.p != nullptr;
  if (a.p) {
    if (!tc::make_map_2d(&prm.tp, a.p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.ldp, a.T, a.ldp, 32, kBM))
      return cudaErrorInvalidValue;
    for (int k = 0; k < a.n_slots; ++k) {
      prm.q_rank[k] = a.q_rank[k];
      if (!tc::make_map_2d(&prm.tq[k], a.q[k], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.q_rank[k], a.n_rows,
                    a.q_rank[k], 32, kBN))
        return cudaErrorInvalidValue;
    }
  }
  prm.items = a.items;
  prm.n_items = a.n_items;
  prm.T = a.T;
  prm.err = tc::error_word();
  if (!prm.err) return cudaErrorInvalidDevice;
  prm.nk_main = (int32_t)((a.K + 63) / 64);
  prm.lora_separate = a.lora_separate;
  prm.n_colscale = a.n_colscale;
  prm.out = a.out;
  prm.ldo = a.ldo;
  prm.n_out = a.n_rows;
  prm.drop = a.drop;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_tc_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid((unsigned)((a.n_rows + kBN - 1) / kBN), (unsigned)a.max_items);
  if (a.max_items <= 0) return cudaSuccess;
  prof_begin(prof_kind, st);
  k_tc_gemm<<<grid, kThreads, kSmemBytes, st>>>(prm);
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
