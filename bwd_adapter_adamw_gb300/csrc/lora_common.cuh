// Shared device helpers for the LoRA-linear kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lora_gb300.h"

namespace lora {

// Programmatic dependent launch. Every kernel of the library starts with grid_dep_sync(): it waits
// until the kernels before it in the stream have completed and their writes are visible
// (griddepcontrol.wait), then lets the next kernel in the stream begin its launch
// (griddepcontrol.launch_dependents). Launched with the programmatic stream serialization
// attribute (launch_kernel), a kernel's launch and CTA dispatch overlap the tail of the kernel
// before it; launched without it, the wait returns at once.
__device__ __forceinline__ void grid_dep_sync() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

constexpr int kGemmTileT = 128;   // token rows per forward/dX/shrink/G work item
constexpr int kRedTileT = 128;    // tokens per split of the CUDA-core token reductions (dA, dB)
constexpr int kRedSub = 4;        // token groups (separate partials) per reduction item
constexpr int kRowPartCols = 16;  // partial row width of the CUDA-core shrink / G (ranks <= 16)
constexpr int kRowChunk = 1024;   // K columns per partial of the CUDA-core shrink / G

// ------------------------------------------------------------------------------------------
// Stateless dropout hash ("4.3. Training Guide", Dropout: masks come from a stateless index
// hash of seed, optimizer step, accumulation ordinal, token position, layer and projection).
// Mixer: the SplitMix64 output finaliser (Steele, Lea & Flood 2014, Stafford variant 13).
// key(chunk) = mix(mix(mix(seed ^ gamma) ^ step) ^ (ordinal << 48 | layer << 16 | proj)),
// element (position t, column i): h = mix(key ^ (t * in + i)); kept iff (h >> 32) >= tau,
// tau = floor(p * 2^32). The per-chunk keys are computed on the host.
// ------------------------------------------------------------------------------------------
__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

struct DropParams {
  int32_t enabled;        // 0: every element kept, no hash evaluated
  uint32_t tau;
  int64_t chunk_tokens;   // tokens per accumulation chunk within the call (> 0)
  int64_t in_dim;
  uint64_t keys[LORA_MAX_CHUNKS_PER_CALL];
};

// Keep decision for token t (index within the call) and input column i.
__device__ __forceinline__ bool drop_keep(const DropParams& d, int64_t t, int64_t i) {
  const int64_t c = t / d.chunk_tokens;
  const int64_t pos = t - c * d.chunk_tokens;
  const uint64_t h = mix64(d.keys[c] ^ (uint64_t)(pos * d.in_dim + i));
  return (uint32_t)(h >> 32) >= d.tau;
}

// The per-token part of the keep decision (the chunk's key and the token's element index base), for
// loops over the columns of one token: drop_keep_at(drop_row(d, t), d.tau, i) == drop_keep(d, t, i).
struct DropRow {
  uint64_t key;
  uint64_t base;
};
__device__ __forceinline__ DropRow drop_row(const DropParams& d, int64_t t) {
  const int64_t c = t / d.chunk_tokens;
  const int64_t pos = t - c * d.chunk_tokens;
  return DropRow{d.keys[c], (uint64_t)(pos * d.in_dim)};
}
__device__ __forceinline__ bool drop_keep_at(const DropRow& r, uint32_t tau, int64_t i) {
  return (uint32_t)(mix64(r.key ^ (r.base + (uint64_t)i)) >> 32) >= tau;
}

// ------------------------------------------------------------------------------------------
// element loads
// ------------------------------------------------------------------------------------------
template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<__nv_bfloat16> { static constexpr int N = 8; };

// Load VEC consecutive elements (16 bytes) as floats.
__device__ __forceinline__ void load16(const float* p, float* out) {
  const float4 v = __ldg(reinterpret_cast<const float4*>(p));
  out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
}
__device__ __forceinline__ void load16(const __nv_bfloat16* p, float* out) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    out[2 * j] = __uint_as_float(w[j] << 16);
    out[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Store 4 consecutive outputs.
__device__ __forceinline__ void store4(float* p, const float* v) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, const float* v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// tf32 split for the LoRA K-blocks of the fp32 products (three tf32 products): hi = x rounded to
// tf32 (nearest, ties away from zero), lo = x - hi (exact in fp32). The tensor core reads lo as
// tf32 too, so a product formed as hi*hi' + hi*lo' + lo*hi' is within about 2^-21 of the fp32
// product, relative.
__device__ __forceinline__ float tf32_hi(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// bf16 split for the fp32 frozen products: hi = x rounded to bf16 (nearest even) and lo = the
// remainder x - hi (exact in fp32) rounded to bf16. Each rounding keeps 8 significant bits, so
// |x - hi - lo| <= 2^-16 |x|, and a product formed on bf16 tensor cores as
// hi*hi' + hi*lo' + lo*hi' (the dropped lo*lo' is below 2^-16 too) stays within a few 2^-16 of
// the fp32 product, relative, for every term; over a dot product the errors partly cancel.
__device__ __forceinline__ void bf16_split4(const float (&x)[4], uint2& hi, uint2& lo) {
  const __nv_bfloat162 h01 = __floats2bfloat162_rn(x[0], x[1]);
  const __nv_bfloat162 h23 = __floats2bfloat162_rn(x[2], x[3]);
  const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
  const __nv_bfloat162 l01 = __floats2bfloat162_rn(x[0] - f01.x, x[1] - f01.y);
  const __nv_bfloat162 l23 = __floats2bfloat162_rn(x[2] - f23.x, x[3] - f23.y);
  hi.x = *reinterpret_cast<const uint32_t*>(&h01);
  hi.y = *reinterpret_cast<const uint32_t*>(&h23);
  lo.x = *reinterpret_cast<const uint32_t*>(&l01);
  lo.y = *reinterpret_cast<const uint32_t*>(&l23);
}

// A token range handled by one CTA, with the adapter slot of those tokens (-1: none).
struct TokenItem {
  int32_t t0, t1, slot, pad;
};

// Work item idx of a call: from the item table, or, when the table is null (a single-adapter
// call), the uniform kGemmTileT-token tiles of [0, T) with slot 0. False past the last item.
__device__ __forceinline__ bool get_item(const TokenItem* items, const int32_t* n_items, int idx,
                                         int64_t T, TokenItem& it) {
  if (items) {
    if (idx >= *n_items) return false;
    it = items[idx];
    return true;
  }
  const int64_t t0 = (int64_t)idx * kGemmTileT;
  if (t0 >= T) return false;
  it.t0 = (int32_t)t0;
  it.t1 = (int32_t)(T < t0 + kGemmTileT ? T : t0 + kGemmTileT);
  it.slot = 0;
  it.pad = 0;
  return true;
}

// Segment table staged in shared memory by a block (at most kSegSmem segments; larger tables are
// read from global memory): start[k], end[k] = start[k + 1], slot[k].
constexpr int kSegSmem = 2048;
struct SegView {
  const int32_t* start;   // [n + 1]
  const int32_t* slot;    // [n]
  int32_t n;
};
__device__ __forceinline__ SegView stage_segments(int32_t n_seg, const int32_t* seg_start,
                                                  const int32_t* seg_slot, int32_t* s_start,
                                                  int32_t* s_slot) {
  if (!seg_start || n_seg > kSegSmem) return SegView{seg_start, seg_slot, seg_start ? n_seg : 0};
  for (int k = threadIdx.x; k <= n_seg; k += blockDim.x) {
    s_start[k] = seg_start[k];
    if (k < n_seg) s_slot[k] = seg_slot[k];
  }
  __syncthreads();
  return SegView{s_start, s_slot, n_seg};
}

// Token-reduction work item idx: from the table, or (null table, single-adapter call) the uniform
// runs of span tokens covering [0, T), slot 0.
__device__ __forceinline__ bool get_span_item(const TokenItem* items, const int32_t* n_items, int idx,
                                              int64_t T, int64_t span, TokenItem& it) {
  if (items) {
    if (idx >= *n_items) return false;
    it = items[idx];
    return true;
  }
  const int64_t t0 = (int64_t)idx * span;
  if (t0 >= T) return false;
  it.t0 = (int32_t)t0;
  it.t1 = (int32_t)(T < t0 + span ? T : t0 + span);
  it.slot = 0;
  it.pad = 0;
  return true;
}

}  // namespace lora
