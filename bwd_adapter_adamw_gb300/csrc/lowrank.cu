// Token work items, adapter transposes, ordered split reductions and the test hooks.
#include <algorithm>
#include <climits>

#include "lora_kernels.h"

namespace lora {

namespace {

// Token work items from the segment table ("Multi-LoRA Training Example (fully-async)", Design:
// a batch holds contiguous per-adapter sample groups; here a segment is a contiguous token range
// with one slot). Segments are taken in order; each covers [max(start, end of coverage so far),
// end), clamped to [0, T). Uncovered tokens form items with slot -1 (frozen output only).
// Items never cross a segment boundary, so every CTA works for exactly one slot.
__global__ void k_make_items(int64_t T, int32_t n_seg, const int32_t* __restrict__ seg_start,
                             const int32_t* __restrict__ seg_slot, int32_t n_slots,
                             TokenItem* gitems, int32_t* gcount, int32_t gmax, TokenItem* ritems,
                             int32_t* rcount, int32_t rmax) {
  grid_dep_sync();
  __shared__ int32_t s_start[kSegSmem + 1], s_slot[kSegSmem];
  const SegView sv = stage_segments(n_seg, seg_start, seg_slot, s_start, s_slot);
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  int32_t ng = 0, nr = 0;
  int64_t cursor = 0;
  auto emit = [&](int64_t a, int64_t b, int32_t slot) {
    for (int64_t t = a; t < b; t += kGemmTileT)
      if (ng < gmax) gitems[ng++] = TokenItem{(int32_t)t, (int32_t)min(b, t + kGemmTileT), slot, 0};
    if (slot >= 0 && ritems)
      for (int64_t t = a; t < b; t += kRedTileT)
        if (nr < rmax) ritems[nr++] = TokenItem{(int32_t)t, (int32_t)min(b, t + kRedTileT), slot, 0};
  };
  // n_seg < 0: one implicit segment [0, T) with slot 0 (single-adapter calls)
  const int32_t nsegs = seg_start ? n_seg : (n_seg < 0 ? 1 : 0);
  for (int32_t k = 0; k < nsegs; ++k) {
    int64_t a = seg_start ? (int64_t)sv.start[k] : 0;
    int64_t b = seg_start ? (int64_t)sv.start[k + 1] : T;
    int32_t slot = seg_slot ? sv.slot[k] : 0;
    if (slot < 0 || slot >= n_slots) slot = -1;
    a = max((int64_t)0, min(a, T));
    b = max((int64_t)0, min(b, T));
    if (a < cursor) a = cursor;
    if (b <= a) continue;
    if (a > cursor) emit(cursor, a, -1);
    emit(a, b, slot);
    cursor = b;
  }
  if (cursor < T) emit(cursor, T, -1);
  *gcount = ng;
  if (rcount) *rcount = nr;
}

// 32 x 32 shared-memory tile transpose of fp32 matrices, one matrix per blockIdx.z.
__global__ void k_transpose_slots(const TransposeTab tab) {
  grid_dep_sync();
  __shared__ float tile[32][33];
  const int z = blockIdx.z;
  const int64_t rows = tab.rows[z], cols = tab.cols[z];
  const int64_t c0 = (int64_t)blockIdx.x * 32, r0 = (int64_t)blockIdx.y * 32;
  if (r0 >= rows || c0 >= cols) return;
  const float* src = tab.src[z];
  float* dst = tab.dst[z];
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[i][threadIdx.x] = src[r * cols + c];
  }
  __syncthreads();
  const int64_t ldd = tab.ld_dst[z] > 0 ? tab.ld_dst[z] : rows;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) dst[c * ldd + r] = tile[threadIdx.x][i];
  }
}

template <typename T>
__global__ void k_transpose_w(const T* __restrict__ src, T* __restrict__ dst, int64_t rows,
                              int64_t cols) {
  grid_dep_sync();
  __shared__ T tile[32][33];
  const int64_t c0 = (int64_t)blockIdx.x * 32, r0 = (int64_t)blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[i][threadIdx.x] = src[r * cols + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) dst[c * rows + r] = tile[threadIdx.x][i];
  }
}

// fp32 prepared weight: W [rows, cols] -> bf16 [W_hi | W_lo | W^T_hi | W^T_lo] (the bf16 split
// of every element: hi = bf16(x), lo = bf16(x - hi))
__device__ __forceinline__ void split_one(float x, uint16_t* hi, uint16_t* lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  *hi = __bfloat16_as_ushort(h);
  *lo = __bfloat16_as_ushort(__float2bfloat16_rn(x - __bfloat162float(h)));
}

__global__ void k_prepare_w_f32(const float* __restrict__ src, uint16_t* __restrict__ dst,
                                int64_t rows, int64_t cols) {
  grid_dep_sync();
  __shared__ float tile[32][33];
  const int64_t n = rows * cols;
  const int64_t c0 = (int64_t)blockIdx.x * 32, r0 = (int64_t)blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) {
      const float x = src[r * cols + c];
      split_one(x, dst + r * cols + c, dst + n + r * cols + c);
      tile[i][threadIdx.x] = x;
    }
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) split_one(tile[threadIdx.x][i], dst + 2 * n + c * rows + r, dst + 3 * n + c * rows + r);
  }
}

// A_cat and the block-diagonal B_cat of an fp32 fused group (CatTab), one element per thread;
// with `zero`, the gradient scratch dA_cat, dB_cat (same sizes, after them) is cleared too
__global__ void k_pack_cat(const CatTab t, float* __restrict__ Acat, float* __restrict__ Bcat,
                           float* __restrict__ dAcat, float* __restrict__ dBcat, int zero) {
  grid_dep_sync();
  const int64_t nr = (int64_t)t.n * t.r;
  const int64_t na = nr * t.in, nb = t.off[t.n] * nr;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t total = zero ? 2 * (na + nb) : na + nb;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
    if (e >= na + nb) {
      const int64_t z = e - (na + nb);
      if (z < na) dAcat[z] = 0.f;
      else dBcat[z - na] = 0.f;
    } else if (e < na) {
      const int64_t row = e / t.in, i = e - row * t.in;
      const int k = (int)(row / t.r);
      Acat[e] = t.A[k][(row - (int64_t)k * t.r) * t.in + i];
    } else {
      const int64_t f = e - na, o = f / nr, c = f - o * nr;
      int k = 0;
      while (k + 1 < t.n && o >= t.off[k + 1]) ++k;
      const int kc = (int)(c / t.r);
      Bcat[f] = kc == k ? t.B[k][(o - t.off[k]) * t.r + (c - (int64_t)kc * t.r)] : 0.f;
    }
  }
}

__global__ void k_add_cat_grads(const CatTab t, const float* __restrict__ dAcat,
                                const float* __restrict__ dBcat) {
  grid_dep_sync();
  const int64_t nr = (int64_t)t.n * t.r;
  const int64_t na = nr * t.in, nb = t.off[t.n] * t.r;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < na + nb; e += stride) {
    if (e < na) {
      const int64_t row = e / t.in, i = e - row * t.in;
      const int k = (int)(row / t.r);
      t.dA[k][(row - (int64_t)k * t.r) * t.in + i] += dAcat[e];
    } else {
      const int64_t f = e - na, o = f / t.r, j = f - o * t.r;
      int k = 0;
      while (k + 1 < t.n && o >= t.off[k + 1]) ++k;
      t.dB[k][(o - t.off[k]) * t.r + j] += dBcat[o * nr + (int64_t)k * t.r + j];
    }
  }
}

// out_slot += sum over the slot's items, in item order, of the per-item partials.
// part[item * sub + g] is [M][ldp] (sub partials per item); element (m, j), j < rank_slot, goes to
// out_slot[m * rank + j]
// (transposed == 0, dB layout [out, r]) or out_slot[j * M + m] (transposed == 1, dA [r, in]).
__global__ void k_reduce_parts(const float* __restrict__ part, const TokenItem* __restrict__ items,
                               const int32_t* __restrict__ n_items, int32_t sub, int64_t M,
                               int64_t ldp, int transposed, const ReduceTab tab) {
  grid_dep_sync();
  const int slot = blockIdx.y;
  const int32_t r = tab.rank[slot];
  float* out = tab.out[slot];
  const int64_t total = M * ldp;
  const int32_t ni = *n_items;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = e / ldp;
    const int32_t j = (int32_t)(e - m * ldp);
    if (j >= r) continue;
    float acc = 0.f;
    bool any = false;
    for (int32_t it = 0; it < ni; ++it) {
      if (items[it].slot != slot) continue;
      for (int32_t g = 0; g < sub; ++g) acc += part[((int64_t)it * sub + g) * total + e];
      any = true;
    }
    if (!any) continue;
    const int64_t o = transposed ? ((int64_t)j * M + m) : (m * r + j);
    out[o] += acc;
  }
}

__global__ void k_dropout_mask(const DropParams dp, int64_t T, int64_t in_dim, uint8_t* mask) {
  grid_dep_sync();
  const int64_t n = T * in_dim;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = e / in_dim, i = e - t * in_dim;
    mask[e] = (!dp.enabled || drop_keep(dp, t, i)) ? 1 : 0;
  }
}

// dst[t, o] = bf16(src[t, o] * scale[o]): the DoRA dY' operand of the tensor-core dX product,
// whose column scale runs along K and so cannot be applied in the epilogue. A thread owns 8
// adjacent columns (their scales loaded once) and walks a band of `band` rows (32, more when the
// grid's y extent would exceed its limit) with four 16-byte loads in flight; consecutive threads
// take consecutive 16-byte chunks of a row.
constexpr int kColscaleThreads = 128;
constexpr int kColscaleRows = 32;
__global__ void __launch_bounds__(kColscaleThreads) k_colscale_bf16(
    const __nv_bfloat16* __restrict__ src, const float* __restrict__ scale, int64_t rows,
    int64_t cols, int64_t band, __nv_bfloat16* __restrict__ dst) {
  grid_dep_sync();
  const int64_t c = ((int64_t)blockIdx.x * kColscaleThreads + threadIdx.x) * 8;
  if (c >= cols) return;
  const float4 s0 = __ldg(reinterpret_cast<const float4*>(scale + c));
  const float4 s1 = __ldg(reinterpret_cast<const float4*>(scale + c + 4));
  const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  const int64_t r0 = (int64_t)blockIdx.y * band;
  const int64_t r1 = min(rows, r0 + band);
  for (int64_t r = r0; r < r1; r += 4) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (r + u < r1) v[u] = __ldg(reinterpret_cast<const uint4*>(src + (r + u) * cols + c));
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (r + u >= r1) continue;
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint4 o;
      uint32_t* ow = &o.x;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float x0 = __uint_as_float(w[j] << 16) * sc[2 * j];
        const float x1 = __uint_as_float(w[j] & 0xFFFF0000u) * sc[2 * j + 1];
        __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
        ow[j] = *reinterpret_cast<uint32_t*>(&h);
      }
      *reinterpret_cast<uint4*>(dst + (r + u) * cols + c) = o;
    }
  }
}

__global__ void k_ratio(const float* __restrict__ num, const float* __restrict__ den, int64_t n,
                        float* __restrict__ out) {
  grid_dep_sync();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = num[i] / den[i];
}

// Slot of every token by the same segment walk as k_make_items: one CTA, segments in order,
// the CTA's threads fill each covered range.
__global__ void k_token_slots(int64_t T, int32_t n_seg, const int32_t* __restrict__ seg_start,
                              const int32_t* __restrict__ seg_slot, int32_t n_slots,
                              int32_t* __restrict__ token_slot) {
  grid_dep_sync();
  int64_t cursor = 0;
  for (int32_t k = 0; k < n_seg; ++k) {
    int64_t a = max((int64_t)0, min((int64_t)seg_start[k], T));
    int64_t b = max((int64_t)0, min((int64_t)seg_start[k + 1], T));
    int32_t slot = seg_slot[k];
    if (slot < 0 || slot >= n_slots) slot = -1;
    if (a < cursor) a = cursor;
    if (b <= a) continue;
    for (int64_t t = cursor + threadIdx.x; t < a; t += blockDim.x) token_slot[t] = -1;
    for (int64_t t = a + threadIdx.x; t < b; t += blockDim.x) token_slot[t] = slot;
    cursor = b;
  }
  for (int64_t t = cursor + threadIdx.x; t < T; t += blockDim.x) token_slot[t] = -1;
}

// The same items, built in parallel by one CTA of kItemThreads threads for tables of up to
// 2 * kItemThreads segments (the serial walk costs about 15 us at 30 segments). Segment k's
// coverage starts at max(its start, the largest end of the non-empty segments before it) (an
// exclusive prefix maximum), which is exactly the cursor of the serial walk; its items (a gap
// item run first when it leaves uncovered tokens behind) are placed by exclusive prefix sums of
// the per-segment item counts, so the table is the serial walk's, item for item.
constexpr int kItemThreads = 1024;
constexpr int kItemSegs = 2 * kItemThreads;

__device__ __forceinline__ void block_scan2(int32_t* v, int n, bool is_max) {
  // inclusive Hillis-Steele scan of v[0, n) (n <= kItemSegs), two elements per thread
  for (int off = 1; off < n; off <<= 1) {
    int32_t x[2];
    for (int u = 0; u < 2; ++u) {
      const int i = threadIdx.x + u * kItemThreads;
      x[u] = (i < n && i >= off) ? v[i - off] : (is_max ? INT32_MIN : 0);
    }
    __syncthreads();
    for (int u = 0; u < 2; ++u) {
      const int i = threadIdx.x + u * kItemThreads;
      if (i < n) v[i] = is_max ? max(v[i], x[u]) : v[i] + x[u];
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kItemThreads) k_make_items_par(
    int64_t T, int32_t n_seg, const int32_t* __restrict__ seg_start,
    const int32_t* __restrict__ seg_slot, int32_t n_slots, TokenItem* gitems, int32_t* gcount,
    int32_t gmax, TokenItem* ritems, int32_t* rcount, int32_t rmax) {
  grid_dep_sync();
  __shared__ int32_t s_a[kItemSegs], s_b[kItemSegs];
  __shared__ int8_t s_slot[kItemSegs];   // -1 .. LORA_MAX_SLOTS - 1
  __shared__ int32_t s_cur[kItemSegs], s_g[kItemSegs], s_r[kItemSegs];
  const int n = n_seg;   // 1 .. kItemSegs (the launcher checks)
  const int64_t TT = T;
  for (int u = 0; u < 2; ++u) {
    const int k = threadIdx.x + u * kItemThreads;
    if (k >= n) continue;
    int64_t a = seg_start[k], b = seg_start[k + 1];
    int32_t slot = seg_slot[k];
    if (slot < 0 || slot >= n_slots) slot = -1;
    a = max((int64_t)0, min(a, TT));
    b = max((int64_t)0, min(b, TT));
    s_a[k] = (int32_t)a;
    s_b[k] = (int32_t)b;
    s_slot[k] = (int8_t)slot;
    s_cur[k] = b > a ? (int32_t)b : 0;   // contributes to the coverage of later segments
  }
  __syncthreads();
  block_scan2(s_cur, n, true);   // inclusive max: coverage after segment k
  // exclusive: coverage before segment k; then this segment's item counts
  int32_t cur[2], ea[2];
  for (int u = 0; u < 2; ++u) {
    const int k = threadIdx.x + u * kItemThreads;
    cur[u] = ea[u] = 0;
    if (k >= n) continue;
    cur[u] = k > 0 ? max(0, s_cur[k - 1]) : 0;
    ea[u] = max(s_a[k], cur[u]);
  }
  __syncthreads();
  for (int u = 0; u < 2; ++u) {
    const int k = threadIdx.x + u * kItemThreads;
    if (k >= n) continue;
    const int32_t b = s_b[k];
    const bool acc = b > ea[u];
    const int32_t gap = acc ? ea[u] - cur[u] : 0;
    const int32_t seg = acc ? b - ea[u] : 0;
    s_g[k] = (gap + kGemmTileT - 1) / kGemmTileT + (seg + kGemmTileT - 1) / kGemmTileT;
    s_r[k] = s_slot[k] >= 0 ? (seg + kRedTileT - 1) / kRedTileT : 0;
    s_cur[k] = cur[u];   // keep the coverage before k (the scan is no longer needed)
    s_a[k] = acc ? ea[u] : -1;
  }
  __syncthreads();
  // coverage after the last segment (for the tail gap): the largest end of a non-empty segment
  __shared__ int32_t s_end;
  if (threadIdx.x == 0) s_end = 0;
  __syncthreads();
  for (int u = 0; u < 2; ++u) {
    const int k = threadIdx.x + u * kItemThreads;
    if (k < n && s_b[k] > s_a[k] && s_a[k] >= 0) atomicMax(&s_end, s_b[k]);
  }
  block_scan2(s_g, n, false);
  block_scan2(s_r, n, false);
  for (int u = 0; u < 2; ++u) {
    const int k = threadIdx.x + u * kItemThreads;
    if (k >= n || s_a[k] < 0) continue;
    int32_t og = k > 0 ? s_g[k - 1] : 0, orr = k > 0 ? s_r[k - 1] : 0;
    const int32_t c = s_cur[k], a = s_a[k], b = s_b[k], slot = s_slot[k];
    for (int32_t t = c; t < a; t += kGemmTileT, ++og)
      if (og < gmax) gitems[og] = TokenItem{t, min(a, t + kGemmTileT), -1, 0};
    for (int32_t t = a; t < b; t += kGemmTileT, ++og)
      if (og < gmax) gitems[og] = TokenItem{t, min(b, t + kGemmTileT), slot, 0};
    if (slot >= 0 && ritems)
      for (int32_t t = a; t < b; t += kRedTileT, ++orr)
        if (orr < rmax) ritems[orr] = TokenItem{t, min(b, t + kRedTileT), slot, 0};
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t og = s_g[n - 1];
    for (int32_t t = s_end; t < TT; t += kGemmTileT, ++og)
      if (og < gmax) gitems[og] = TokenItem{t, (int32_t)min(TT, (int64_t)t + kGemmTileT), -1, 0};
    *gcount = min(og, gmax);
    if (rcount) *rcount = min(s_r[n - 1], rmax);
  }
}

// Reduction work items of the tensor-core dA / dB products (the serial walk is
// k_make_red_items_tc in lowrank_tc.cu): per slot, the 64-token blocks of its segments merged
// into runs and cut into spans of span_blocks blocks, the slots' items one after the other. The
// segments' coverage is computed in parallel (as in k_make_items_par), so that each slot's walker
// thread only tests a staged slot id per segment and merges its own segments' block ranges.
__global__ void __launch_bounds__(kItemThreads) k_make_red_items_par(
    int64_t T, int32_t n_seg, const int32_t* __restrict__ seg_start,
    const int32_t* __restrict__ seg_slot, int32_t n_slots, int32_t span_blocks, TokenItem* items,
    int32_t* count, int32_t max_items) {
  grid_dep_sync();
  __shared__ int32_t s_ba[kItemSegs], s_bb[kItemSegs], s_cur[kItemSegs];
  __shared__ int8_t s_sl[kItemSegs];
  __shared__ int32_t s_count[LORA_MAX_SLOTS + 1];
  const int n = n_seg;   // 1 .. kItemSegs (the launcher checks)
  const int64_t TT = T;
  int32_t a_[2], b_[2], sl_[2];
  for (int u = 0; u < 2; ++u) {
    const int k = threadIdx.x + u * kItemThreads;
    a_[u] = b_[u] = 0;
    sl_[u] = -1;
    if (k >= n) continue;
    int64_t a = seg_start[k], b = seg_start[k + 1];
    int32_t slot = seg_slot[k];
    if (slot < 0 || slot >= n_slots) slot = -1;
    a = max((int64_t)0, min(a, TT));
    b = max((int64_t)0, min(b, TT));
    a_[u] = (int32_t)a;
    b_[u] = (int32_t)b;
    sl_[u] = slot;
    s_cur[k] = b > a ? (int32_t)b : 0;
  }
  __syncthreads();
  block_scan2(s_cur, n, true);
  for (int u = 0; u < 2; ++u) {
    const int k = threadIdx.x + u * kItemThreads;
    if (k >= n) continue;
    const int32_t cur = k > 0 ? max(0, s_cur[k - 1]) : 0;
    const int32_t ea = max(a_[u], cur);
    const bool acc = b_[u] > ea;
    s_ba[k] = (acc && sl_[u] >= 0) ? ea / 64 : -1;
    s_bb[k] = (b_[u] + 63) / 64;
    s_sl[k] = (int8_t)sl_[u];
  }
  __syncthreads();
  const int s = threadIdx.x;
  auto walk = [&](bool write, int32_t base) {
    int32_t cnt = 0;
    auto emit_run = [&](int32_t b0, int32_t b1) {
      for (int32_t b = b0; b < b1; b += span_blocks) {
        if (write && base + cnt < max_items)
          items[base + cnt] = TokenItem{b * 64, min(b1, b + span_blocks) * 64, s, 0};
        ++cnt;
      }
    };
    int32_t rb = -1, re = -1;
    for (int k = 0; k < n; ++k) {
      if (s_sl[k] != s) continue;
      const int32_t ba = s_ba[k];
      if (ba < 0) continue;
      const int32_t bb = s_bb[k];
      if (re >= 0 && ba <= re) {
        re = max(re, bb);
      } else {
        if (re >= 0) emit_run(rb, re);
        rb = ba;
        re = bb;
      }
    }
    if (re >= 0) emit_run(rb, re);
    return cnt;
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

}  // namespace

cudaError_t launch_make_red_items_par(int64_t T, int32_t n_seg, const int32_t* seg_start,
                                      const int32_t* seg_slot, int32_t n_slots,
                                      int32_t span_blocks, TokenItem* items, int32_t* count,
                                      int32_t max_items, cudaStream_t st) {
  if (!seg_start || !seg_slot || n_seg < 1 || n_seg > kItemSegs || T > INT32_MAX - 64 ||
      span_blocks < 1 || n_slots > LORA_MAX_SLOTS)
    return cudaErrorInvalidValue;
  prof_begin(0, st);
  launch_kernel(k_make_red_items_par, 1, kItemThreads, 0, st, T, n_seg, seg_start, seg_slot,
                n_slots, span_blocks, items, count, max_items);
  return cudaGetLastError();
}

cudaError_t launch_make_items(int64_t T, int32_t n_seg, const int32_t* seg_start,
                              const int32_t* seg_slot, int32_t n_slots, TokenItem* gitems,
                              int32_t* gcount, int32_t gmax, TokenItem* ritems, int32_t* rcount,
                              int32_t rmax, cudaStream_t st) {
  prof_begin(0, st);
  if (seg_start && seg_slot && n_seg >= 1 && n_seg <= kItemSegs && T <= INT32_MAX - kGemmTileT)
    launch_kernel(k_make_items_par, 1, kItemThreads, 0, st, T, n_seg, seg_start, seg_slot, n_slots,
                  gitems, gcount, gmax, ritems, rcount, rmax);
  else
    launch_kernel(k_make_items, 1, 128, 0, st, T, n_seg, seg_start, seg_slot, n_slots, gitems,
                  gcount, gmax, ritems, rcount, rmax);
  return cudaGetLastError();
}

// Slot bitmask of every 128-token tile: bit s is set when a token of the tile is routed to slot s
// (segments taken in order, each covering [max(start, coverage so far), end) clamped to [0, T),
// exactly as for the token items). One thread per tile scans the staged segment table.
__global__ void __launch_bounds__(256) k_tile_slot_masks(int64_t T, int32_t n_seg,
                                                         const int32_t* __restrict__ seg_start,
                                                         const int32_t* __restrict__ seg_slot,
                                                         int32_t n_slots, uint32_t* masks,
                                                         int64_t n_tiles) {
  grid_dep_sync();
  __shared__ int32_t s_start[kSegSmem + 1], s_slot[kSegSmem];
  const SegView sv = stage_segments(n_seg, seg_start, seg_slot, s_start, s_slot);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_tiles;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t lo = i * kGemmTileT, hi = min(T, lo + kGemmTileT);
    uint32_t m = 0;
    int64_t cursor = 0;
    for (int32_t k = 0; k < sv.n; ++k) {
      int64_t a = sv.start[k], b = sv.start[k + 1];
      a = max((int64_t)0, min(a, T));
      b = max((int64_t)0, min(b, T));
      if (a < cursor) a = cursor;
      if (b <= a) continue;
      cursor = b;
      if (a >= hi) break;   // this and every later segment start after the tile
      const int32_t slot = sv.slot[k];
      if (slot >= 0 && slot < n_slots && b > lo) m |= 1u << slot;
    }
    masks[i] = m;
  }
}

cudaError_t launch_tile_slot_masks(int64_t T, int32_t n_seg, const int32_t* seg_start,
                                   const int32_t* seg_slot, int32_t n_slots, uint32_t* masks,
                                   cudaStream_t st) {
  const int64_t n_tiles = (T + kGemmTileT - 1) / kGemmTileT;
  if (n_tiles <= 0) return cudaSuccess;
  int64_t blocks = (n_tiles + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  prof_begin(0, st);
  launch_kernel(k_tile_slot_masks, (unsigned)blocks, 256, 0, st, T, n_seg, seg_start, seg_slot,
                n_slots, masks, n_tiles);
  return cudaGetLastError();
}

cudaError_t launch_transpose_slots(const TransposeTab& t, int n, int64_t max_rows, int64_t max_cols,
                                   cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  dim3 grid((unsigned)((max_cols + 31) / 32), (unsigned)((max_rows + 31) / 32), (unsigned)n);
  { prof_begin(0, st); launch_kernel(k_transpose_slots, grid, dim3(32, 8), 0, st, t); }
  return cudaGetLastError();
}

static unsigned elementwise_blocks(int64_t n) {
  return (unsigned)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, 152 * 8));
}

cudaError_t launch_pack_cat(const CatTab& t, float* Acat, float* Bcat, float* dAcat, float* dBcat,
                            cudaStream_t st) {
  const int64_t nr = (int64_t)t.n * t.r;
  const int zero = dAcat != nullptr && dBcat != nullptr;
  const int64_t n = (nr * t.in + t.off[t.n] * nr) * (zero ? 2 : 1);
  prof_begin(0, st);
  launch_kernel(k_pack_cat, elementwise_blocks(n), 256, 0, st, t, Acat, Bcat, dAcat, dBcat, zero);
  return cudaGetLastError();
}

cudaError_t launch_add_cat_grads(const CatTab& t, const float* dAcat, const float* dBcat,
                                 cudaStream_t st) {
  const int64_t nr = (int64_t)t.n * t.r;
  prof_begin(0, st);
  launch_kernel(k_add_cat_grads, elementwise_blocks(nr * t.in + t.off[t.n] * t.r), 256, 0, st, t,
                dAcat, dBcat);
  return cudaGetLastError();
}

cudaError_t launch_prepare_weight(int dtype, const void* W, void* Wt, int64_t rows, int64_t cols,
                                  cudaStream_t st) {
  dim3 grid((unsigned)((cols + 31) / 32), (unsigned)((rows + 31) / 32));
  if (dtype == LORA_F32)
    { prof_begin(0, st); launch_kernel(k_prepare_w_f32, grid, dim3(32, 8), 0, st, (const float*)W, (uint16_t*)Wt, rows, cols); }
  else
    { prof_begin(0, st); launch_kernel(k_transpose_w<__nv_bfloat16>, grid, dim3(32, 8), 0, st, (const __nv_bfloat16*)W,
                                                                (__nv_bfloat16*)Wt, rows, cols); }
  return cudaGetLastError();
}

cudaError_t launch_reduce_parts(const float* part, const TokenItem* items, const int32_t* n_items,
                                int max_items, int32_t sub, int64_t M, int64_t ldp, int transposed,
                                const ReduceTab& tab, int n_slots, cudaStream_t st) {
  (void)max_items;
  const int64_t total = M * ldp;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  dim3 grid((unsigned)blocks, (unsigned)n_slots);
  { prof_begin(0, st); launch_kernel(k_reduce_parts, grid, threads, 0, st, part, items, n_items, sub, M, ldp, transposed, tab); }
  return cudaGetLastError();
}

cudaError_t launch_dropout_mask(const DropParams& dp, int64_t T, int64_t in_dim, uint8_t* mask,
                                cudaStream_t st) {
  const int64_t n = T * in_dim;
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 8192) blocks = 8192;
  { prof_begin(0, st); launch_kernel(k_dropout_mask, (unsigned)blocks, 256, 0, st, dp, T, in_dim, mask); }
  return cudaGetLastError();
}

cudaError_t launch_colscale_bf16(const void* src, const float* scale, int64_t rows, int64_t cols,
                                 void* dst, cudaStream_t st) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  if (cols % 8) return cudaErrorInvalidValue;
  int64_t band = kColscaleRows;
  while ((rows + band - 1) / band > 65535) band *= 2;
  const dim3 grid((unsigned)((cols / 8 + kColscaleThreads - 1) / kColscaleThreads),
                  (unsigned)((rows + band - 1) / band));
  prof_begin(0, st);
  launch_kernel(k_colscale_bf16, grid, kColscaleThreads, 0, st, (const __nv_bfloat16*)src, scale,
                rows, cols, band, (__nv_bfloat16*)dst);
  return cudaGetLastError();
}

cudaError_t launch_ratio(const float* num, const float* den, int64_t n, float* out, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  { prof_begin(0, st); launch_kernel(k_ratio, (unsigned)((n + 255) / 256), 256, 0, st, num, den, n, out); }
  return cudaGetLastError();
}

cudaError_t launch_token_slots(int64_t T, int32_t n_seg, const int32_t* seg_start,
                               const int32_t* seg_slot, int32_t n_slots, int32_t* token_slot,
                               cudaStream_t st) {
  { prof_begin(0, st); launch_kernel(k_token_slots, 1, 256, 0, st, T, n_seg, seg_start, seg_slot, n_slots, token_slot); }
  return cudaGetLastError();
}

}  // namespace lora
