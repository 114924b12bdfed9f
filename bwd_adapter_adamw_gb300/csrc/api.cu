// C-ABI entry points: argument validation on the host, workspace carving, kernel orchestration.
// Every entry point validates everything before enqueueing anything, so a nonzero status means
// nothing was launched (except LORA_ERR_CUDA, which reports a failed launch).
#include <cmath>
#include <cstring>

#include "lora_kernels.h"

using namespace lora;

namespace {

constexpr size_t kWsAlign = 256;

struct Carve {
  char* base;
  size_t off = 0;
  explicit Carve(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t count) {
    off = (off + kWsAlign - 1) / kWsAlign * kWsAlign;
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

thread_local cudaError_t t_last_error = cudaSuccess;

// Errors left behind by other code in this thread (cudaGetLastError reports the most recent
// error of any runtime call) are cleared before our launches, so that a LORA_ERR_CUDA is ours.
inline void clear_stale() { (void)cudaGetLastError(); }

inline int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return LORA_OK;
  t_last_error = e;
  return LORA_ERR_CUDA;
}

#define LORA_TRY(expr)                                 \
  do {                                                 \
    cudaError_t _e = (expr);                           \
    if (_e != cudaSuccess) return cuda_status(_e);     \
  } while (0)

int64_t max_gemm_items(int64_t T, int32_t n_seg) {
  if (n_seg < 1) n_seg = 1;
  return (T + kGemmTileT - 1) / kGemmTileT + 2 * (int64_t)n_seg + 2;
}
int64_t max_red_items(int64_t T, int32_t n_seg) {
  if (n_seg < 1) n_seg = 1;
  return (T + kRedTileT - 1) / kRedTileT + (int64_t)n_seg + 1;
}

// Shape/dtype checks shared by every per-linear call.
int check_desc(const lora_desc* d, int64_t T, bool multi) {
  if (!d || T < 0) return LORA_ERR_INVALID;
  if (d->in_dim <= 0 || d->out_dim <= 0) return LORA_ERR_INVALID;
  if (d->dtype != LORA_F32 && d->dtype != LORA_BF16 && d->dtype != LORA_BF16_FP8)
    return LORA_ERR_INVALID;
  if (d->rank <= 0) return LORA_ERR_INVALID;
  if (d->rank > LORA_MAX_RANK || (d->rank % 4) != 0) return LORA_ERR_UNSUPPORTED;
  if ((d->in_dim % 8) != 0 || (d->out_dim % 8) != 0) return LORA_ERR_ALIGN;
  if (!(d->dropout_p >= 0.f && d->dropout_p < 1.f)) return LORA_ERR_INVALID;
  if (d->proj_id > 0xFFFFu) return LORA_ERR_INVALID;
  if (d->dora != 0 && d->dora != 1) return LORA_ERR_INVALID;
  if (multi && d->dora) return LORA_ERR_UNSUPPORTED;
  if (d->dtype == LORA_BF16_FP8) {
    // E4M3 rows are K bytes (16-byte TMA strides); a row is quantised from registers
    if ((d->in_dim % 16) != 0 || (d->out_dim % 16) != 0) return LORA_ERR_ALIGN;
    if (multi || d->dora || d->in_dim > 16384 || d->out_dim > 16384) return LORA_ERR_UNSUPPORTED;
  }
  if (!multi && !std::isfinite(d->scale)) return LORA_ERR_INVALID;
  if (T >= (int64_t(1) << 31) - kRedTileT) return LORA_ERR_UNSUPPORTED;
  return LORA_OK;
}

// Host side of the dropout hash: per-chunk keys of this call ("4.3. Training Guide", Dropout).
int build_drop(const lora_desc* d, const lora_ctx* c, int64_t T, DropParams& dp) {
  std::memset(&dp, 0, sizeof(dp));
  const lora_ctx zero{0, 0, 0};
  if (!c) c = &zero;
  if (c->chunk_tokens < 0) return LORA_ERR_INVALID;
  dp.in_dim = d->in_dim;
  dp.chunk_tokens = c->chunk_tokens > 0 ? c->chunk_tokens : (T > 0 ? T : 1);
  const int64_t n_chunks = T > 0 ? (T + dp.chunk_tokens - 1) / dp.chunk_tokens : 0;
  if (n_chunks > LORA_MAX_CHUNKS_PER_CALL) return LORA_ERR_UNSUPPORTED;
  if ((int64_t)c->accum_ordinal + n_chunks > 65536) return LORA_ERR_INVALID;
  if (d->dropout_p <= 0.f) {
    dp.enabled = 0;
    dp.tau = 0;
    return LORA_OK;
  }
  dp.enabled = 1;
  const double t = std::floor((double)d->dropout_p * 4294967296.0);
  dp.tau = t >= 4294967295.0 ? 0xFFFFFFFFu : (uint32_t)t;
  const uint64_t k1 = mix64(mix64(d->seed ^ 0x9E3779B97F4A7C15ull) ^ c->opt_step);
  for (int64_t i = 0; i < n_chunks; ++i) {
    const uint64_t ord = (uint64_t)(c->accum_ordinal + i) & 0xFFFFull;
    const uint64_t packed = (ord << 48) | ((uint64_t)d->layer_id << 16) | (uint64_t)d->proj_id;
    dp.keys[i] = mix64(k1 ^ packed);
  }
  return LORA_OK;
}

float dropout_q(const lora_desc* d) {
  return d->dropout_p > 0.f ? (float)(1.0 / (1.0 - (double)d->dropout_p)) : 1.f;
}

// Slot view shared by single-adapter and multi-adapter calls.
struct Slots {
  int n = 0;
  const float* A[LORA_MAX_SLOTS];
  const float* B[LORA_MAX_SLOTS];
  float* dA[LORA_MAX_SLOTS];
  float* dB[LORA_MAX_SLOTS];
  int32_t rank[LORA_MAX_SLOTS];
  float scale[LORA_MAX_SLOTS];
  int64_t rank_sum = 0;
};

int slots_from_table(const lora_desc* d, int32_t n_slots, const lora_slot* tab, bool need_grads,
                     Slots& s) {
  if (!tab || n_slots < 1) return LORA_ERR_INVALID;
  if (n_slots > LORA_MAX_SLOTS) return LORA_ERR_UNSUPPORTED;
  s.n = n_slots;
  s.rank_sum = 0;
  for (int k = 0; k < n_slots; ++k) {
    const lora_slot& e = tab[k];
    if (!e.A || !e.B) return LORA_ERR_INVALID;
    if (need_grads && (!e.dA || !e.dB)) return LORA_ERR_INVALID;
    if (e.rank <= 0 || e.rank > d->rank) return LORA_ERR_INVALID;
    if (e.rank % 4) return LORA_ERR_UNSUPPORTED;
    if (!std::isfinite(e.scale)) return LORA_ERR_INVALID;
    if (!al16(e.A) || !al16(e.B) || (need_grads && (!al16(e.dA) || !al16(e.dB))))
      return LORA_ERR_ALIGN;
    s.A[k] = e.A; s.B[k] = e.B; s.dA[k] = e.dA; s.dB[k] = e.dB;
    s.rank[k] = e.rank; s.scale[k] = e.scale;
    s.rank_sum += e.rank;
  }
  return LORA_OK;
}

void single_slot(const lora_desc* d, const float* A, const float* B, float* dA, float* dB, Slots& s) {
  s.n = 1;
  s.A[0] = A; s.B[0] = B; s.dA[0] = dA; s.dB[0] = dB;
  s.rank[0] = d->rank; s.scale[0] = d->scale;
  s.rank_sum = d->rank;
}

// ---- tensor-core path shape choices (bf16 activations) ---------------------------------------
constexpr int kMaxRowSplits = 8;

int np_for(int rmax) {           // MMA N covering hi + lo rows of the largest slot
  const int n = 2 * rmax;
  return n <= 16 ? 16 : n <= 32 ? 32 : n <= 64 ? 64 : 128;
}

// Resident CTAs of the skinny tensor-core products: one per SM on the 152-SM part (each holds
// about 192 KB of stages). A shape choice only (any count is correct).
constexpr int64_t kLowRankSlots = 152;

// K splits of the skinny token-row products (the CTAs of one cluster, a power of two that divides
// the 128-token tile): as many as keep every CTA resident in one wave.
int row_splits(int64_t T, int32_t n_seg, int64_t K) {
  const int64_t items = max_gemm_items(T, n_seg);
  int64_t s = kLowRankSlots / items;
  const int64_t nk = (K + 63) / 64;
  if (s > nk / 2) s = nk / 2;
  if (s > kMaxRowSplits) s = kMaxRowSplits;
  int p2 = 1;
  while (2 * p2 <= s) p2 *= 2;
  return p2;
}

// 64-token blocks per reduction work item: short runs, so that the CTAs of a reduction cluster,
// which split a slot's items evenly, get nearly equal token counts. The single-adapter form walks
// the same runs over [0, T), so that one slot routed every token gives the same sums bit for bit.
int red_span_blocks(int64_t, int64_t) { return kRedSpanBlocks; }

int64_t red_items_bound(int64_t T, int32_t n_seg, int n_slots, int span) {
  const int64_t ns = n_seg < 1 ? 1 : n_seg;
  const int64_t nb = (T + 63) / 64;
  return ns + 1 + n_slots + (nb + ns + span - 1) / span;
}

struct Layout {
  TokenItem* gitems; int32_t* gcount;
  TokenItem* ritems; int32_t* rcount;   // SIMT token reductions (fp32 path)
  int64_t gmax, rmax;
  float* ratio;        // [out] DoRA m / n
  float* Gs;           // [T, rmax]
  float* At;           // per slot [in, r_s]
  float* Bt;           // per slot [r_s, out] (fp32 path)
  float* partB;        // [rmax_items][out][rank] (fp32 path)
  float* partA;        // [rmax_items][in][rank] (fp32 path)
  uint16_t* dYs;       // [T, out] bf16 dY * (m / n) for the DoRA tensor-core products
  float* rd_part;      // [K chunks][T][16] partials of the CUDA-core shrink / G (fp32 path)
  uint16_t* Ah;        // [T, K] bf16 split of X (forward) or dY' (backward): hi ... (fp32 path)
  uint16_t* Al;        // ... and lo

  // tensor-core path
  uint16_t* Xd;        // [T, in] bf16 masked input (dropout)
  uint16_t* Sa;        // per slot [2 r, in] bf16 split of A
  uint16_t* Sb;        // per slot [2 r, out] bf16 split of B^T
  int64_t ldt;         // padded token stride of the transposed splits
  uint16_t* HsT;       // per slot [2 r, ldt] bf16
  uint16_t* GsT;       // per slot [2 r, ldt] bf16
  TokenItem* items_db; int32_t* count_db; int64_t max_db; int span_db;
  TokenItem* items_da; int32_t* count_da; int64_t max_da; int span_da;
  // FP8 frozen base
  uint8_t* Aq;         // [T, max(in, out)] E4M3 codes of X (forward) or dY' (backward)
  float* sq;           // [T] their row scales
  float* Pq;           // [T, rank] Hs or Gs divided by sq
  float* Qq;           // [max(in, out), rank] B divided by the W row scales, or A^T by W^T's
  // routed calls (bf16): frozen products on uniform 128-token tiles with per-tile slot sets
  uint32_t* tmask;     // [ceil(T / 128)] slots present in each tile
  float* Px;           // [T, ldx] Hs or Gs expanded: token t's values in its slot's column block
  float* Atx;          // [in, ldx] every slot's A^T side by side, blocks 32-column aligned
  int64_t ldx;         // upper bound of the padded column blocks' total
  size_t bytes;
};

// first column of each slot's 32-aligned block in the expanded operands, and their total
int32_t expanded_cols(const Slots& s, int32_t* pcol) {
  int32_t c = 0;
  for (int k = 0; k < s.n; ++k) {
    pcol[k] = c;
    c += (s.rank[k] + 31) / 32 * 32;
  }
  return c;
}

// E4M3 prepared weight: [W8 (out x in) | sw (out) | WT8 (in x out) | swT (in)], 16-byte sections
struct Fp8Prep {
  const uint8_t* W8;
  const float* sw;
  const uint8_t* WT8;
  const float* swT;
};
size_t al16_up(size_t b) { return (b + 15) / 16 * 16; }
size_t fp8_prep_bytes(int64_t out, int64_t in) {
  return al16_up((size_t)out * in) + al16_up((size_t)out * 4) + al16_up((size_t)in * out) +
         al16_up((size_t)in * 4);
}
Fp8Prep fp8_prep(const void* Wp, int64_t out, int64_t in) {
  const uint8_t* b = static_cast<const uint8_t*>(Wp);
  Fp8Prep f;
  f.W8 = b;
  b += al16_up((size_t)out * in);
  f.sw = reinterpret_cast<const float*>(b);
  b += al16_up((size_t)out * 4);
  f.WT8 = b;
  b += al16_up((size_t)in * out);
  f.swT = reinterpret_cast<const float*>(b);
  return f;
}

Layout carve(const lora_desc* d, int64_t T, int32_t n_seg, int n_slots, int64_t rank_sum,
             bool backward, void* ws) {
  Layout L{};
  Carve c(ws);
  const bool tc = d->dtype != LORA_F32;
  L.gmax = max_gemm_items(T, n_seg);
  L.rmax = max_red_items(T, n_seg);
  L.gitems = c.take<TokenItem>((size_t)L.gmax);
  L.gcount = c.take<int32_t>(4);
  L.ratio = c.take<float>((size_t)d->out_dim);
  if (tc) {
    if (d->dropout_p > 0.f) L.Xd = c.take<uint16_t>((size_t)T * d->in_dim);
    L.Sa = c.take<uint16_t>((size_t)2 * rank_sum * d->in_dim);
  }
  if (backward) {
    L.Gs = c.take<float>((size_t)T * d->rank);
    L.At = c.take<float>((size_t)rank_sum * d->in_dim);
    if (d->dora && tc) L.dYs = c.take<uint16_t>((size_t)T * d->out_dim);
    if (tc) {
      L.Sb = c.take<uint16_t>((size_t)2 * rank_sum * d->out_dim);
      L.ldt = (T + 7) / 8 * 8;
      L.HsT = c.take<uint16_t>((size_t)2 * rank_sum * L.ldt);
      L.GsT = c.take<uint16_t>((size_t)2 * rank_sum * L.ldt);
      L.span_db = red_span_blocks(T, d->out_dim);
      L.span_da = red_span_blocks(T, d->in_dim);
      L.max_db = red_items_bound(T, n_seg, n_slots, L.span_db);
      L.max_da = red_items_bound(T, n_seg, n_slots, L.span_da);
      L.items_db = c.take<TokenItem>((size_t)L.max_db);
      L.count_db = c.take<int32_t>(LORA_MAX_SLOTS + 8);   // total, then per-slot item ranges
      L.items_da = c.take<TokenItem>((size_t)L.max_da);
      L.count_da = c.take<int32_t>(LORA_MAX_SLOTS + 8);
    } else {
      L.ritems = c.take<TokenItem>((size_t)L.rmax);
      L.rcount = c.take<int32_t>(4);
      L.Bt = c.take<float>((size_t)rank_sum * d->out_dim);
      L.partB = c.take<float>((size_t)L.rmax * kRedSub * d->out_dim * d->rank);
      L.partA = c.take<float>((size_t)L.rmax * kRedSub * d->in_dim * d->rank);
    }
  } else if (!tc) {
    L.ritems = c.take<TokenItem>((size_t)L.rmax);
    L.rcount = c.take<int32_t>(4);
  }
  if (tc && n_seg >= 0) {
    // 32-aligned column blocks: each rank (a multiple of 4) pads by at most 28 columns
    L.ldx = rank_sum + 28 * (int64_t)n_slots;
    L.tmask = c.take<uint32_t>((size_t)((T + kGemmTileT - 1) / kGemmTileT));
    L.Px = c.take<float>((size_t)T * L.ldx);
    if (backward) L.Atx = c.take<float>((size_t)d->in_dim * L.ldx);
  }
  if (d->dtype == LORA_BF16_FP8) {
    const int64_t kmax = d->in_dim > d->out_dim ? d->in_dim : d->out_dim;
    L.Aq = c.take<uint8_t>((size_t)T * kmax);
    L.sq = c.take<float>((size_t)T);
    L.Pq = c.take<float>((size_t)T * d->rank);
    L.Qq = c.take<float>((size_t)kmax * d->rank);
  }
  if (!tc) {
    const int64_t kmax = d->in_dim > d->out_dim ? d->in_dim : d->out_dim;
    L.rd_part = c.take<float>((size_t)((kmax + kRowChunk - 1) / kRowChunk) * T * kRowPartCols);
    L.Ah = c.take<uint16_t>((size_t)T * kmax);
    L.Al = c.take<uint16_t>((size_t)T * kmax);
  }
  L.bytes = c.off + kWsAlign;
  return L;
}

size_t ws_size(const lora_desc* d, int64_t T, int32_t n_seg, int n_slots, int64_t rank_sum) {
  return carve(d, T, n_seg, n_slots, rank_sum, true, nullptr).bytes;
}

// Routing plan: the token work tables of routed calls over one batch (T, segments, slots), built
// once and read by every planned call: the row products' items, the fp32 reductions' items, the
// tensor-core reductions' runs and the slot mask of every 128-token tile. Its layout is a function
// of (T, n_seg, n_slots) alone.
struct RoutePlan {
  TokenItem* gitems; int32_t* gcount; int64_t gmax;
  TokenItem* ritems; int32_t* rcount; int64_t rmax;
  TokenItem* items_red; int32_t* count_red; int64_t max_red;
  uint32_t* tmask;
  size_t bytes;
};

RoutePlan plan_carve(int64_t T, int32_t n_seg, int32_t n_slots, void* buf) {
  RoutePlan P{};
  Carve c(buf);
  P.gmax = max_gemm_items(T, n_seg);
  P.rmax = max_red_items(T, n_seg);
  P.max_red = red_items_bound(T, n_seg, n_slots, kRedSpanBlocks);
  P.gitems = c.take<TokenItem>((size_t)P.gmax);
  P.gcount = c.take<int32_t>(4);
  P.ritems = c.take<TokenItem>((size_t)P.rmax);
  P.rcount = c.take<int32_t>(4);
  P.items_red = c.take<TokenItem>((size_t)P.max_red);
  P.count_red = c.take<int32_t>(LORA_MAX_SLOTS + 8);
  P.tmask = c.take<uint32_t>((size_t)((T + kGemmTileT - 1) / kGemmTileT));
  P.bytes = c.off + kWsAlign;
  return P;
}

// The call's tables become the plan's (the workspace copies go unused).
void apply_plan(Layout& L, const RoutePlan& P) {
  L.gitems = P.gitems; L.gcount = P.gcount;
  if (L.ritems) { L.ritems = P.ritems; L.rcount = P.rcount; }
  if (L.items_db) {
    L.items_db = L.items_da = P.items_red;
    L.count_db = L.count_da = P.count_red;
    L.max_db = L.max_da = P.max_red;
  }
  if (L.tmask) L.tmask = P.tmask;
}

SlotInfo slot_info(const Slots& s, float q) {
  SlotInfo si{};
  int32_t region = 0;
  for (int k = 0; k < s.n; ++k) {
    si.rank[k] = s.rank[k];
    si.alpha[k] = s.scale[k] * q;
    si.region[k] = region;
    region += 2 * s.rank[k];
  }
  expanded_cols(s, si.pcol);
  return si;
}

// A single-adapter call (no segments) runs on uniform work items that the kernels compute from
// the index: 128-token tiles and span-token reduction runs, all of slot 0. No item tables.
void use_uniform_items(Layout& L, int64_t T) {
  L.gitems = nullptr; L.gcount = nullptr;
  L.gmax = (T + kGemmTileT - 1) / kGemmTileT;
  L.items_db = nullptr; L.count_db = nullptr;
  L.max_db = (T + (int64_t)L.span_db * 64 - 1) / ((int64_t)L.span_db * 64);
  L.items_da = nullptr; L.count_da = nullptr;
  L.max_da = (T + (int64_t)L.span_da * 64 - 1) / ((int64_t)L.span_da * 64);
}

// shrink on tensor cores: Hs[t, j] = s_k q (Xd[t, :] . A_k[j, :]) via the hi/lo split of A_k
int tc_shrink(const lora_desc* d, const DropParams& dp, int64_t T, const void* X, int32_t n_seg,
              const Slots& s, const Layout& L, float* H, float* Hx, cudaStream_t st) {
  const float q = dropout_q(d);
  const void* Xin = X;
  if (dp.enabled) {
    LORA_TRY(launch_mask_bf16(X, T, d->in_dim, dp, L.Xd, st));
    Xin = L.Xd;
  }
  SplitTab sp{};
  sp.K = d->in_dim;
  TcRowsArgs r{};
  int64_t off = 0;
  for (int k = 0; k < s.n; ++k) {
    sp.src[k] = s.A[k];
    sp.dst[k] = L.Sa + off;
    sp.rank[k] = s.rank[k];
    r.s[k] = L.Sa + off;
    r.rank[k] = s.rank[k];
    off += 2 * (int64_t)s.rank[k] * d->in_dim;
  }
  LORA_TRY(launch_split(sp, s.n, st));
  r.a = Xin; r.T = T; r.K = d->in_dim; r.n_slots = s.n;
  r.NP = np_for(d->rank);
  r.splits = row_splits(T, n_seg, d->in_dim);
  r.si = slot_info(s, q);
  r.out = H; r.ldo = d->rank;
  r.out2 = Hx; r.ld2 = L.ldx;   // routed calls: the slot-expanded copy for the frozen product
  r.items = L.gitems; r.n_items = L.gcount; r.max_items = (int)L.gmax;
  LORA_TRY(launch_tc_rows(r, st, LORA_PROF_SHRINK));
  return LORA_OK;
}

// Routed call: the frozen products run on uniform 128-token tiles, each tile adding the LoRA
// terms of the slots present in it from the slot-expanded operand (zeroed first: a token's row is
// zero outside its slot's column block).
int routed_tiles(int64_t T, int32_t n_seg, const int32_t* seg_start, const int32_t* seg_slot,
                 const Slots& s, const Layout& L, bool masks_ready, cudaStream_t st) {
  if (!masks_ready)
    LORA_TRY(launch_tile_slot_masks(T, n_seg, seg_start, seg_slot, s.n, L.tmask, st));
  LORA_TRY(cudaMemsetAsync(L.Px, 0, (size_t)T * L.ldx * sizeof(float), st));
  return LORA_OK;
}

void set_routed_gemm(TcGemmArgs& t, const Slots& s, const Layout& L, int64_t T, bool dx) {
  int32_t pcol[LORA_MAX_SLOTS];
  expanded_cols(s, pcol);
  t.items = nullptr;
  t.n_items = nullptr;
  t.max_items = (int)((T + kGemmTileT - 1) / kGemmTileT);
  t.tile_mask = L.tmask;
  t.p = L.Px;
  t.ldp = L.ldx;
  for (int k = 0; k < s.n; ++k) {
    t.slot_pcol[k] = pcol[k];
    t.slot_qx[k] = dx ? pcol[k] : 0;     // dX: one A^T map, the slot's block of columns
    t.slot_qmap[k] = dx ? 0 : k;         // forward: slot k's own B map
  }
  if (dx) {
    t.q[0] = L.Atx;
    t.q_inner[0] = L.ldx;
    t.n_q_maps = 1;
  }
}

// forward, bf16 activations: shrink and frozen product on tensor cores
int run_forward_tc(const lora_desc* d, const DropParams& dp, int64_t T, const void* X,
                   const void* W, const void* Wprep, int32_t n_seg, const int32_t* seg_start,
                   const int32_t* seg_slot, const Slots& s, const float* ratio_src_m,
                   const float* ratio_src_n, void* Y, float* H, void* ws, cudaStream_t st,
                   const RoutePlan* plan = nullptr) {
  Layout L = carve(d, T, n_seg, s.n, s.rank_sum, false, ws);
  clear_stale();
  if (n_seg < 0)
    use_uniform_items(L, T);
  else if (plan)
    apply_plan(L, *plan);
  else
    LORA_TRY(launch_make_items(T, n_seg, seg_start, seg_slot, s.n, L.gitems, L.gcount,
                               (int32_t)L.gmax, nullptr, nullptr, 0, st));
  const float* ratio = nullptr;
  if (ratio_src_m) {
    LORA_TRY(launch_ratio(ratio_src_m, ratio_src_n, d->out_dim, L.ratio, st));
    ratio = L.ratio;
  }
  const bool fp8 = d->dtype == LORA_BF16_FP8;
  if (fp8)   // E4M3 codes and per-token scales of X for the frozen product
    LORA_TRY(launch_quant_rows_e4m3(X, T, d->in_dim, L.Aq, L.sq, st));
  const bool routed = n_seg >= 0;
  if (routed) {
    int rr = routed_tiles(T, n_seg, seg_start, seg_slot, s, L, plan != nullptr, st);
    if (rr) return rr;
  }
  int rc = tc_shrink(d, dp, T, X, n_seg, s, L, H, routed ? L.Px : nullptr, st);
  if (rc) return rc;
  TcGemmArgs t{};
  t.a = X; t.T = T; t.b = W; t.n_rows = d->out_dim; t.K = d->in_dim;
  t.p = H; t.ldp = d->rank; t.n_slots = s.n;
  for (int k = 0; k < s.n; ++k) { t.q[k] = s.B[k]; t.q_rank[k] = s.rank[k]; }
  t.n_colscale = ratio; t.out = Y; t.ldo = d->out_dim;
  if (fp8) {
    // Y = sx sw (X8 W8^T) + Hs B^T = sx sw (X8 W8^T + (Hs / sx)(B / sw)^T): one accumulator
    const Fp8Prep f = fp8_prep(Wprep, d->out_dim, d->in_dim);
    LORA_TRY(launch_div_rows2(DivRowsJob{H, d->rank, L.sq, T, d->rank, L.Pq, d->rank},
                              DivRowsJob{s.B[0], d->rank, f.sw, d->out_dim, d->rank, L.Qq, d->rank},
                              st));
    t.a = L.Aq; t.b = f.W8; t.fp8 = 1;
    t.p = L.Pq; t.q[0] = L.Qq;
    t.m_rowscale = L.sq; t.n_colscale = f.sw;
  }
  t.items = L.gitems; t.n_items = L.gcount; t.max_items = (int)L.gmax; t.drop = dp;
  if (routed) set_routed_gemm(t, s, L, T, false);
  LORA_TRY(launch_tc_gemm(t, st, LORA_PROF_FROZEN_FWD));
  return LORA_OK;
}

// backward, bf16 activations: G, dX, dB and dA on tensor cores
int run_backward_tc(const lora_desc* d, const DropParams& dp, int64_t T, const void* X,
                    const void* Wt, int32_t n_seg, const int32_t* seg_start,
                    const int32_t* seg_slot, const Slots& s, const void* dY, const float* H,
                    const float* dora_m, const float* dora_n, const void* Y_save, void* dX,
                    float* dm, void* ws, cudaStream_t st, const RoutePlan* plan = nullptr) {
  Layout L = carve(d, T, n_seg, s.n, s.rank_sum, true, ws);
  clear_stale();
  if (n_seg < 0) {
    use_uniform_items(L, T);
  } else if (plan) {
    if (L.span_db != kRedSpanBlocks || L.span_da != kRedSpanBlocks) return LORA_ERR_INVALID;
    apply_plan(L, *plan);
    int rr = routed_tiles(T, n_seg, seg_start, seg_slot, s, L, true, st);
    if (rr) return rr;
  } else {
    LORA_TRY(launch_make_items(T, n_seg, seg_start, seg_slot, s.n, L.gitems, L.gcount,
                               (int32_t)L.gmax, nullptr, nullptr, 0, st));
    LORA_TRY(launch_make_red_items_tc(T, n_seg, seg_start, seg_slot, s.n, L.span_db, L.items_db,
                                      L.count_db, (int32_t)L.max_db, st));
    if (L.span_da == L.span_db) {   // the same runs serve both reductions
      L.items_da = L.items_db;
      L.count_da = L.count_db;
      L.max_da = L.max_db;
    } else {
      LORA_TRY(launch_make_red_items_tc(T, n_seg, seg_start, seg_slot, s.n, L.span_da, L.items_da,
                                        L.count_da, (int32_t)L.max_da, st));
    }
    int rr = routed_tiles(T, n_seg, seg_start, seg_slot, s, L, false, st);
    if (rr) return rr;
  }
  const bool routed = n_seg >= 0;
  const float q = dropout_q(d);
  const SlotInfo si = slot_info(s, q);
  // A^T (fp32) for the LoRA K-steps of dX; hi/lo split of B^T for G
  float* At[LORA_MAX_SLOTS];
  {
    TransposeTab ta{};
    SplitTab sp{};
    sp.K = d->out_dim;
    sp.transposed = 1;
    int64_t oa = 0, ob = 0;
    for (int k = 0; k < s.n; ++k) {
      At[k] = L.At + oa; oa += (int64_t)s.rank[k] * d->in_dim;
      ta.src[k] = s.A[k]; ta.dst[k] = At[k]; ta.rows[k] = s.rank[k]; ta.cols[k] = d->in_dim;
      sp.src[k] = s.B[k]; sp.dst[k] = L.Sb + ob; sp.rank[k] = s.rank[k];
      ob += 2 * (int64_t)s.rank[k] * d->out_dim;
    }
    if (routed) {   // every slot's A^T side by side in one operand, 32-aligned blocks
      LORA_TRY(cudaMemsetAsync(L.Atx, 0, (size_t)d->in_dim * L.ldx * sizeof(float), st));
      for (int k = 0; k < s.n; ++k) {
        ta.dst[k] = L.Atx + si.pcol[k];
        ta.ld_dst[k] = L.ldx;
      }
    }
    LORA_TRY(launch_adapter_prep(ta, sp, s.n, st));
  }
  const void* dYp = dY;
  if (dora_m) {   // DoRA: dY' = dY * (m / n), materialised once in bf16 for every product
    LORA_TRY(launch_ratio(dora_m, dora_n, d->out_dim, L.ratio, st));
    LORA_TRY(launch_colscale_bf16(dY, L.ratio, T, d->out_dim, L.dYs, st));
    dYp = L.dYs;
  }
  const void* Xin = X;
  if (dp.enabled) {
    LORA_TRY(launch_mask_bf16(X, T, d->in_dim, dp, L.Xd, st));
    Xin = L.Xd;
  }
  // Gs[t, j] = s_k q (dY'[t, :] . B_k[:, j])
  {
    TcRowsArgs r{};
    int64_t ob = 0;
    for (int k = 0; k < s.n; ++k) {
      r.s[k] = L.Sb + ob;
      r.rank[k] = s.rank[k];
      ob += 2 * (int64_t)s.rank[k] * d->out_dim;
    }
    r.a = dYp; r.T = T; r.K = d->out_dim; r.n_slots = s.n;
    r.NP = np_for(d->rank);
    r.splits = row_splits(T, n_seg, d->out_dim);
    r.si = si;
    r.out = L.Gs; r.ldo = d->rank;
    r.outT = L.GsT; r.ldt = L.ldt; r.outT_bytes = (size_t)2 * s.rank_sum * L.ldt * sizeof(uint16_t);
    r.side_h = H; r.side_ldh = d->rank; r.side_outT = L.HsT;   // the saved Hs for dB
    if (routed) {   // the slot-expanded Gs for the dX product's uniform tiles
      r.out2 = L.Px;
      r.ld2 = L.ldx;
    }
    r.items = L.gitems; r.n_items = L.gcount; r.max_items = (int)L.gmax;
    LORA_TRY(launch_tc_rows(r, st, LORA_PROF_G));
  }
  // dX = dY' W + (Gs A_k) * M
  if (dX) {
    TcGemmArgs t{};
    t.a = dYp; t.T = T; t.b = Wt; t.n_rows = d->in_dim; t.K = d->out_dim;
    t.p = L.Gs; t.ldp = d->rank; t.n_slots = s.n;
    for (int k = 0; k < s.n; ++k) { t.q[k] = At[k]; t.q_rank[k] = s.rank[k]; }
    t.lora_separate = dp.enabled; t.out = dX; t.ldo = d->in_dim;
    t.items = L.gitems; t.n_items = L.gcount; t.max_items = (int)L.gmax; t.drop = dp;
    if (routed) set_routed_gemm(t, s, L, T, true);
    if (d->dtype == LORA_BF16_FP8) {
      // dX = sd swT (dY8 WT8^T) + Gs A: the LoRA operands divided by the same scales
      const Fp8Prep f = fp8_prep(Wt, d->out_dim, d->in_dim);
      LORA_TRY(launch_quant_rows_e4m3(dYp, T, d->out_dim, L.Aq, L.sq, st));
      LORA_TRY(launch_div_rows2(DivRowsJob{L.Gs, d->rank, L.sq, T, d->rank, L.Pq, d->rank},
                                DivRowsJob{At[0], d->rank, f.swT, d->in_dim, d->rank, L.Qq, d->rank},
                                st));
      t.a = L.Aq; t.b = f.WT8; t.fp8 = 1;
      t.p = L.Pq; t.q[0] = L.Qq;
      t.m_rowscale = L.sq; t.n_colscale = f.swT;
    }
    LORA_TRY(launch_tc_gemm(t, st, LORA_PROF_FROZEN_DX));
  }
  // dB_k += dY'^T Hs over the slot's tokens (as dB^T rows of the transposed Hs split, written by
  // the G product's CTAs) and dA_k += Gs^T Xd (GsT, written by the G product): one launch when
  // both walk the same run table
  TcRedArgs rb{}, ra{};
  for (int k = 0; k < s.n; ++k) {
    rb.st[k] = L.HsT + (int64_t)si.region[k] * L.ldt;
    ra.st[k] = L.GsT + (int64_t)si.region[k] * L.ldt;
    rb.rank[k] = ra.rank[k] = s.rank[k];
    rb.tab.rank[k] = ra.tab.rank[k] = s.rank[k];
    rb.tab.out[k] = s.dB[k];
    ra.tab.out[k] = s.dA[k];
  }
  rb.n_slots = ra.n_slots = s.n;
  rb.max_rank = ra.max_rank = d->rank;
  rb.T = ra.T = T;
  rb.ldt = ra.ldt = L.ldt;
  rb.b = dYp; rb.N = d->out_dim; rb.transposed = 1;
  ra.b = Xin; ra.N = d->in_dim; ra.transposed = 0;
  rb.items = L.items_db; rb.n_items = L.count_db;
  ra.items = L.items_da; ra.n_items = L.count_da;
  if (rb.items == ra.items && rb.n_items == ra.n_items) {
    LORA_TRY(launch_tc_red2(rb, ra, st, LORA_PROF_RED));
  } else {
    LORA_TRY(launch_tc_red(rb, st, LORA_PROF_RED_DB));
    LORA_TRY(launch_tc_red(ra, st, LORA_PROF_RED_DA));
  }
  if (dm) LORA_TRY(launch_dora_dm(d->dtype, dY, Y_save, dora_m, T, d->out_dim, dm, st));
  return LORA_OK;
}

// forward: shrink then the frozen product with the up-projection as extra K-steps
int run_forward(const lora_desc* d, const DropParams& dp, int64_t T, const void* X, const void* W,
                const void* Wprep, int32_t n_seg, const int32_t* seg_start, const int32_t* seg_slot, const Slots& s,
                const float* ratio_src_m, const float* ratio_src_n, void* Y, float* H, void* ws,
                cudaStream_t st, const RoutePlan* plan = nullptr) {
  if (d->dtype != LORA_F32)
    return run_forward_tc(d, dp, T, X, W, Wprep, n_seg, seg_start, seg_slot, s, ratio_src_m,
                          ratio_src_n, Y, H, ws, st, plan);
  Layout L = carve(d, T, n_seg, s.n, s.rank_sum, false, ws);
  clear_stale();
  if (plan && n_seg >= 0) apply_plan(L, *plan);
  // single adapter, rank <= 16: uniform token tiles computed in the kernels, single-pass shrink
  const bool fused = n_seg < 0 && d->rank <= 16;
  const TokenItem* items = fused ? nullptr : L.gitems;
  const int32_t* n_items = fused ? nullptr : L.gcount;
  const int max_items = fused ? (int)((T + kGemmTileT - 1) / kGemmTileT) : (int)L.gmax;
  if (!fused && !(plan && n_seg >= 0))
    LORA_TRY(launch_make_items(T, n_seg, seg_start, seg_slot, s.n, L.gitems, L.gcount,
                               (int32_t)L.gmax, L.ritems, L.rcount, (int32_t)L.rmax, st));
  const float q = dropout_q(d);
  const float* ratio = nullptr;
  if (ratio_src_m) {
    LORA_TRY(launch_ratio(ratio_src_m, ratio_src_n, d->out_dim, L.ratio, st));
    ratio = L.ratio;
  }
  // shrink: Hs[t, j] = s_k q sum_i M[t,i] X[t,i] A_k[j,i]   (columns j >= r_k written as 0)
  {
    RowDotArgs a{};
    a.a = X; a.lda = d->in_dim; a.K = d->in_dim; a.lds = d->in_dim;
    for (int k = 0; k < s.n; ++k) {
      a.s[k] = s.A[k]; a.rank[k] = s.rank[k]; a.alpha[k] = s.scale[k] * q;
    }
    a.max_rank = d->rank; a.mask = dp.enabled; a.drop = dp;
    a.out = H; a.ldo = d->rank;
    a.items = items; a.n_items = n_items; a.single_pass = fused;
    a.T = T; a.part = L.rd_part;
    a.split_hi = L.Ah; a.split_lo = L.Al;
    LORA_TRY(launch_rowdot(d->dtype, a, max_items, st, LORA_PROF_SHRINK));
  }
  // frozen product + Hs B_k^T, times m/n per column in DoRA mode (three bf16 products of the
  // split operands); the prepared weight holds bf16 [W_hi | W_lo | W^T_hi | W^T_lo]
  {
    const int64_t n = d->out_dim * d->in_dim;
    TcGemmArgs t{};
    t.a = L.Ah; t.a_lo = L.Al; t.T = T;
    t.b = Wprep; t.b_lo = static_cast<const uint16_t*>(Wprep) + n;
    t.n_rows = d->out_dim; t.K = d->in_dim;
    t.p = H; t.ldp = d->rank; t.n_slots = s.n;
    for (int k = 0; k < s.n; ++k) { t.q[k] = s.B[k]; t.q_rank[k] = s.rank[k]; }
    t.n_colscale = ratio; t.out = Y; t.ldo = d->out_dim;
    t.items = items; t.n_items = n_items; t.max_items = max_items; t.drop = dp;
    LORA_TRY(launch_tc_gemm_f32(t, st, LORA_PROF_FROZEN_FWD));
  }
  return LORA_OK;
}

int run_backward(const lora_desc* d, const DropParams& dp, int64_t T, const void* X, const void* Wt,
                 int32_t n_seg, const int32_t* seg_start, const int32_t* seg_slot, const Slots& s,
                 const void* dY, const float* H, const float* dora_m, const float* dora_n,
                 const void* Y_save, void* dX, float* dm, void* ws, cudaStream_t st,
                 const RoutePlan* plan = nullptr) {
  if (d->dtype != LORA_F32)
    return run_backward_tc(d, dp, T, X, Wt, n_seg, seg_start, seg_slot, s, dY, H, dora_m, dora_n,
                           Y_save, dX, dm, ws, st, plan);
  Layout L = carve(d, T, n_seg, s.n, s.rank_sum, true, ws);
  clear_stale();
  if (plan && n_seg >= 0) apply_plan(L, *plan);
  // single adapter, rank <= 16: uniform token tiles, single-pass G that also writes A^T, and
  // token reductions that finish inside their thread-block clusters (4 launches)
  const bool fused = n_seg < 0 && d->rank <= 16;
  const TokenItem* items = fused ? nullptr : L.gitems;
  const int32_t* n_items = fused ? nullptr : L.gcount;
  const int max_items = fused ? (int)((T + kGemmTileT - 1) / kGemmTileT) : (int)L.gmax;
  if (!fused && !(plan && n_seg >= 0))
    LORA_TRY(launch_make_items(T, n_seg, seg_start, seg_slot, s.n, L.gitems, L.gcount,
                               (int32_t)L.gmax, L.ritems, L.rcount, (int32_t)L.rmax, st));
  const float q = dropout_q(d);
  // transposed adapters: At_k = A_k^T [in, r_k], Bt_k = B_k^T [r_k, out]
  float* At[LORA_MAX_SLOTS];
  float* Bt[LORA_MAX_SLOTS];
  if (fused) {
    At[0] = L.At;                  // written by the G pass below
    Bt[0] = nullptr;               // G reads B in place
  } else {
    TransposeTab ta{}, tb{};
    int64_t oa = 0, ob = 0;
    for (int k = 0; k < s.n; ++k) {
      At[k] = L.At + oa; oa += (int64_t)s.rank[k] * d->in_dim;
      Bt[k] = L.Bt + ob; ob += (int64_t)s.rank[k] * d->out_dim;
      ta.src[k] = s.A[k]; ta.dst[k] = At[k]; ta.rows[k] = s.rank[k]; ta.cols[k] = d->in_dim;
      tb.src[k] = s.B[k]; tb.dst[k] = Bt[k]; tb.rows[k] = d->out_dim; tb.cols[k] = s.rank[k];
    }
    LORA_TRY(launch_transpose_slots(ta, s.n, d->rank, d->in_dim, st));
    LORA_TRY(launch_transpose_slots(tb, s.n, d->out_dim, d->rank, st));
  }
  const float* ratio = nullptr;
  if (dora_m) {
    LORA_TRY(launch_ratio(dora_m, dora_n, d->out_dim, L.ratio, st));
    ratio = L.ratio;
  }
  // Gs[t, j] = s_k q sum_o dY'[t, o] B_k[o, j]
  {
    RowDotArgs a{};
    a.a = dY; a.lda = d->out_dim; a.K = d->out_dim; a.lds = d->out_dim;
    for (int k = 0; k < s.n; ++k) {
      a.s[k] = Bt[k]; a.rank[k] = s.rank[k]; a.alpha[k] = s.scale[k] * q;
    }
    a.max_rank = d->rank; a.colscale = ratio; a.drop = dp;
    a.out = L.Gs; a.ldo = d->rank;
    a.items = items; a.n_items = n_items;
    a.T = T; a.part = L.rd_part;
    if (dX) { a.split_hi = L.Ah; a.split_lo = L.Al; }
    if (fused) {
      a.single_pass = 1;
      a.s[0] = s.B[0]; a.lds = d->rank; a.s_rows_k = 1;
      a.t_src = s.A[0]; a.t_dst = At[0]; a.t_rows = d->rank; a.t_cols = d->in_dim;
    }
    LORA_TRY(launch_rowdot(d->dtype, a, max_items, st, LORA_PROF_G));
  }
  // dX = dY' W + (Gs A_k) * M, from the split of dY' and of W^T
  if (dX) {
    const int64_t n = d->out_dim * d->in_dim;
    TcGemmArgs t{};
    t.a = L.Ah; t.a_lo = L.Al; t.T = T;
    t.b = static_cast<const uint16_t*>(Wt) + 2 * n; t.b_lo = static_cast<const uint16_t*>(Wt) + 3 * n;
    t.n_rows = d->in_dim; t.K = d->out_dim;
    t.p = L.Gs; t.ldp = d->rank; t.n_slots = s.n;
    for (int k = 0; k < s.n; ++k) { t.q[k] = At[k]; t.q_rank[k] = s.rank[k]; }
    t.lora_separate = dp.enabled; t.out = dX; t.ldo = d->in_dim;
    t.items = items; t.n_items = n_items; t.max_items = max_items; t.drop = dp;
    LORA_TRY(launch_tc_gemm_f32(t, st, LORA_PROF_FROZEN_DX));
  }
  ReduceTab rt{};
  for (int k = 0; k < s.n; ++k) rt.rank[k] = s.rank[k];
  // item-based reductions: ranks <= 16 stream 4 token groups per item (4 partials per item), larger
  // ranks one partial per item
  const int32_t sub = d->rank <= 16 ? kRedSub : 1;
  // dB_k += sum_t dY'[t, o] Hs[t, j]
  ColRedArgs rb{};
  rb.p = H; rb.ldp = d->rank;
  rb.b = dY; rb.ldb = d->out_dim; rb.N = d->out_dim; rb.colscale = ratio;
  for (int k = 0; k < s.n; ++k) rb.rank[k] = s.rank[k];
  rb.max_rank = d->rank; rb.drop = dp;
  rb.part = L.partB; rb.ldpart = d->rank; rb.sub_groups = sub;
  rb.items = L.ritems; rb.n_items = L.rcount;
  // dA_k += sum_t Gs[t, j] M[t, i] X[t, i]   (computed as dA^T partials)
  ColRedArgs ra{};
  ra.p = L.Gs; ra.ldp = d->rank;
  ra.b = X; ra.ldb = d->in_dim; ra.N = d->in_dim; ra.mask = dp.enabled;
  for (int k = 0; k < s.n; ++k) ra.rank[k] = s.rank[k];
  ra.max_rank = d->rank; ra.drop = dp;
  ra.part = L.partA; ra.ldpart = d->rank; ra.sub_groups = sub;
  ra.items = L.ritems; ra.n_items = L.rcount;
  if (fused) {   // both in one launch, each cluster adding its fixed-order sum into dB / dA^T
    rb.T = T; rb.out = s.dB[0]; rb.out_transposed = 0;
    ra.T = T; ra.out = s.dA[0]; ra.out_transposed = 1;
    LORA_TRY(launch_colred2(d->dtype, rb, ra, st, LORA_PROF_RED));
  } else {
    LORA_TRY(launch_colred(d->dtype, rb, (int)L.rmax, st, LORA_PROF_RED_DB));
    for (int k = 0; k < s.n; ++k) rt.out[k] = s.dB[k];
    LORA_TRY(launch_reduce_parts(L.partB, L.ritems, L.rcount, (int)L.rmax, sub, d->out_dim,
                                 d->rank, 0, rt, s.n, st));
    LORA_TRY(launch_colred(d->dtype, ra, (int)L.rmax, st, LORA_PROF_RED_DA));
    for (int k = 0; k < s.n; ++k) rt.out[k] = s.dA[k];
    LORA_TRY(launch_reduce_parts(L.partA, L.ritems, L.rcount, (int)L.rmax, sub, d->in_dim,
                                 d->rank, 1, rt, s.n, st));
  }
  if (dm) LORA_TRY(launch_dora_dm(d->dtype, dY, Y_save, dora_m, T, d->out_dim, dm, st));
  return LORA_OK;
}

// DoRA row norm for bf16 W on tensor cores: H = W A^T by the shrink kernel over W's rows (the hi /
// lo bf16 split of A), then ||W_o||^2 + 2 s H_o . B_o + s^2 B_o (A A^T) B_o^T per row.
struct NormLayout {
  uint16_t* Sa;        // [2 r, in] bf16 split of A
  float* H;            // [out, r]
  float* C;            // [r, r]
  size_t bytes;
};

NormLayout dora_norm_carve(const lora_desc* d, void* ws) {
  NormLayout L{};
  Carve c(ws);
  if (d->dtype == LORA_BF16) {
    L.Sa = c.take<uint16_t>((size_t)2 * d->rank * d->in_dim);
    L.H = c.take<float>((size_t)d->out_dim * d->rank);
    L.C = c.take<float>((size_t)d->rank * d->rank);
  }
  L.bytes = c.off + kWsAlign;
  return L;
}

cudaError_t run_dora_norm_tc(const lora_desc* d, const void* W, const float* A, const float* B,
                             float* norm_out, void* ws, cudaStream_t st) {
  NormLayout L = dora_norm_carve(d, ws);
  SplitTab sp{};
  sp.K = d->in_dim;
  sp.src[0] = A;
  sp.dst[0] = L.Sa;
  sp.rank[0] = d->rank;
  cudaError_t e = launch_split(sp, 1, st);
  if (e != cudaSuccess) return e;
  TcRowsArgs r{};
  r.a = W; r.T = d->out_dim; r.K = d->in_dim; r.n_slots = 1;
  r.s[0] = L.Sa; r.rank[0] = d->rank;
  r.NP = np_for(d->rank);
  r.splits = row_splits(d->out_dim, -1, d->in_dim);
  r.si.rank[0] = d->rank; r.si.alpha[0] = 1.f; r.si.region[0] = 0;
  r.out = L.H; r.ldo = d->rank;
  r.items = nullptr; r.n_items = nullptr;   // uniform 128-row tiles of W
  r.max_items = (int)((d->out_dim + kGemmTileT - 1) / kGemmTileT);
  e = launch_tc_rows(r, st, 0);
  if (e != cudaSuccess) return e;
  return launch_dora_gram_combine(W, L.H, A, B, d->scale, d->out_dim, d->in_dim, d->rank, L.C,
                                  norm_out, st);
}

// ---- fused projections: one frozen product over stacked weights, one adapter per projection --
// ("LoRA Training and Serving", --lora-type: fused projections versus one adapter per q/k/v and
// gate/up projection). Projection k owns output columns [off_k, off_k + out_k) of the fused
// linear; its LoRA operands sit in columns k r .. k r + r - 1 of H (Hs) and G.
struct FusedProjs {
  int n = 0;
  const float* A[LORA_MAX_SLOTS];
  const float* B[LORA_MAX_SLOTS];
  float* dA[LORA_MAX_SLOTS];
  float* dB[LORA_MAX_SLOTS];
  int64_t out[LORA_MAX_SLOTS];
  int64_t off[LORA_MAX_SLOTS];
  int64_t out_max = 0;
};

int fused_from_table(const lora_desc* d, int32_t n_proj, const lora_proj* tab, bool need_grads,
                     FusedProjs& f) {
  if (!tab || n_proj < 1 || n_proj > LORA_MAX_SLOTS) return LORA_ERR_INVALID;
  if ((d->dtype != LORA_BF16 && d->dtype != LORA_F32) || d->dora) return LORA_ERR_UNSUPPORTED;
  // fp32: the group runs as one adapter of rank n_proj * rank
  if (d->dtype == LORA_F32 && (int64_t)n_proj * d->rank > LORA_MAX_RANK) return LORA_ERR_UNSUPPORTED;
  int64_t sum = 0;
  for (int k = 0; k < n_proj; ++k) {
    const lora_proj& e = tab[k];
    if (!e.A || !e.B || e.out_dim <= 0) return LORA_ERR_INVALID;
    if (need_grads && (!e.dA || !e.dB)) return LORA_ERR_INVALID;
    // bf16: column groups start on 256-wide tiles
    if (d->dtype == LORA_BF16 && e.out_dim % 256) return LORA_ERR_UNSUPPORTED;
    if (!al16(e.A) || !al16(e.B) || (need_grads && (!al16(e.dA) || !al16(e.dB))))
      return LORA_ERR_ALIGN;
    f.A[k] = e.A;
    f.B[k] = e.B;
    f.dA[k] = e.dA;
    f.dB[k] = e.dB;
    f.out[k] = e.out_dim;
    f.off[k] = sum;
    sum += e.out_dim;
    if (e.out_dim > f.out_max) f.out_max = e.out_dim;
  }
  if (sum != d->out_dim) return LORA_ERR_INVALID;
  f.n = n_proj;
  return LORA_OK;
}

// The per-projection low-rank products run one projection after the other in stream order and
// reuse one projection's scratch, sized for the widest projection; G and A^T of all the
// projections sit side by side after it.
struct FusedLayout {
  Layout L;
  float* Gcat;     // [T, n r]
  float* Atcat;    // [in, n r]
  uint16_t* Sbk;   // per projection [2 r, out_k] bf16 split of B_k^T, one after the other
  uint16_t* Sacat; // per projection [2 r, in] bf16 split of A_k, one after the other
  uint16_t* GsTk;  // per projection [2 r, ldt] transposed split of Gs_k, one after the other
  uint16_t* HsTk;  // per projection [2 r, ldt] transposed split of the saved Hs_k
  size_t bytes;
};

FusedLayout fused_carve(const lora_desc* d, int64_t T, const FusedProjs& f, void* ws) {
  lora_desc sd = *d;
  sd.out_dim = f.out_max;
  FusedLayout F;
  F.L = carve(&sd, T, -1, 1, d->rank, true, ws);
  Carve c(ws);
  c.off = F.L.bytes;
  F.Gcat = c.take<float>((size_t)T * f.n * d->rank);
  F.Atcat = c.take<float>((size_t)d->in_dim * f.n * d->rank);
  F.Sbk = c.take<uint16_t>((size_t)2 * d->rank * d->out_dim);   // sum of out_k = out_dim
  F.Sacat = c.take<uint16_t>((size_t)2 * d->rank * f.n * d->in_dim);
  F.GsTk = c.take<uint16_t>((size_t)2 * d->rank * f.n * F.L.ldt);
  F.HsTk = c.take<uint16_t>((size_t)2 * d->rank * f.n * F.L.ldt);
  F.bytes = c.off + kWsAlign;
  return F;
}

SlotInfo fused_slot_info(const lora_desc* d) {
  Slots one;
  one.n = 1;
  one.rank[0] = d->rank;
  one.scale[0] = d->scale;
  return slot_info(one, dropout_q(d));
}

// fp32 fused projections: the group runs as one single-adapter linear of rank n r whose adapter
// is A_cat = [A_0; ...; A_{n-1}] and the block-diagonal B_cat (CatTab). Then
// Y = X W_cat^T + s' (Xd A_cat^T) B_cat^T is every projection's forward at once, with
// Hs_cat = s' Xd A_cat^T holding Hs_k in columns k r ..; G_cat = s' dY' B_cat holds G_k in its
// columns k r .., so that the dX product's LoRA term is sum_k G_k A_k and dA_cat = G_cat^T Xd
// holds dA_k in its rows k r ..; dB_cat = dY'^T Hs_cat holds dB_k in its diagonal blocks. The
// shrink reads X once and the G pass dY once for the whole group, and the frozen products run
// once over the stacked weight.
struct FusedF32Layout {
  float* Acat;    // [n r, in]
  float* Bcat;    // [sum out_k, n r]
  float* dAcat;   // [n r, in]
  float* dBcat;   // [sum out_k, n r]
  void* inner;    // workspace of the rank-n r linear
  size_t bytes;
};

lora_desc cat_desc(const lora_desc* d, const FusedProjs& f) {
  lora_desc c = *d;
  c.rank = f.n * d->rank;
  return c;
}

FusedF32Layout fused_f32_carve(const lora_desc* d, int64_t T, const FusedProjs& f, void* ws) {
  const lora_desc cd = cat_desc(d, f);
  const size_t nr = (size_t)cd.rank;
  FusedF32Layout F;
  Carve c(ws);
  F.Acat = c.take<float>(nr * d->in_dim);
  F.Bcat = c.take<float>((size_t)d->out_dim * nr);
  F.dAcat = c.take<float>(nr * d->in_dim);
  F.dBcat = c.take<float>((size_t)d->out_dim * nr);
  F.inner = c.take<uint8_t>(ws_size(&cd, T, -1, 1, cd.rank));
  F.bytes = c.off + kWsAlign;
  return F;
}

size_t fused_ws_bytes(const lora_desc* d, int64_t T, const FusedProjs& f) {
  return d->dtype == LORA_F32 ? fused_f32_carve(d, T, f, nullptr).bytes
                              : fused_carve(d, T, f, nullptr).bytes;
}

CatTab cat_tab(const lora_desc* d, const FusedProjs& f) {
  CatTab t{};
  t.n = f.n;
  t.r = d->rank;
  t.in = d->in_dim;
  for (int k = 0; k < f.n; ++k) {
    t.A[k] = f.A[k];
    t.B[k] = f.B[k];
    t.dA[k] = f.dA[k];
    t.dB[k] = f.dB[k];
    t.off[k] = f.off[k];
  }
  t.off[f.n] = d->out_dim;
  return t;
}

int run_fused_forward_f32(const lora_desc* d, const DropParams& dp, int64_t T, const void* X,
                          const void* W, const void* Wprep, const FusedProjs& f, void* Y, float* H,
                          void* ws, cudaStream_t st) {
  const FusedF32Layout F = fused_f32_carve(d, T, f, ws);
  const lora_desc cd = cat_desc(d, f);
  LORA_TRY(launch_pack_cat(cat_tab(d, f), F.Acat, F.Bcat, nullptr, nullptr, st));
  Slots s;
  single_slot(&cd, F.Acat, F.Bcat, nullptr, nullptr, s);
  return run_forward(&cd, dp, T, X, W, Wprep, -1, nullptr, nullptr, s, nullptr, nullptr, Y, H,
                     F.inner, st);
}

int run_fused_backward_f32(const lora_desc* d, const DropParams& dp, int64_t T, const void* X,
                           const void* Wt, const FusedProjs& f, const void* dY, const float* H,
                           void* dX, void* ws, cudaStream_t st) {
  const FusedF32Layout F = fused_f32_carve(d, T, f, ws);
  const lora_desc cd = cat_desc(d, f);
  const CatTab tab = cat_tab(d, f);
  LORA_TRY(launch_pack_cat(tab, F.Acat, F.Bcat, F.dAcat, F.dBcat, st));
  Slots s;
  single_slot(&cd, F.Acat, F.Bcat, F.dAcat, F.dBcat, s);
  const int rc = run_backward(&cd, dp, T, X, Wt, -1, nullptr, nullptr, s, dY, H, nullptr, nullptr,
                              nullptr, dX, nullptr, F.inner, st);
  if (rc) return rc;
  LORA_TRY(launch_add_cat_grads(tab, F.dAcat, F.dBcat, st));
  return LORA_OK;
}

int run_fused_forward(const lora_desc* d, const DropParams& dp, int64_t T, const void* X,
                      const void* W, const FusedProjs& f, void* Y, float* H, void* ws,
                      cudaStream_t st) {
  FusedLayout F = fused_carve(d, T, f, ws);
  Layout& L = F.L;
  clear_stale();
  use_uniform_items(L, T);
  const int64_t r = d->rank, ldh = (int64_t)f.n * r;
  const SlotInfo si = fused_slot_info(d);
  const void* Xin = X;
  if (dp.enabled) {   // one mask for the projections: they read the same input
    LORA_TRY(launch_mask_bf16(X, T, d->in_dim, dp, L.Xd, st));
    Xin = L.Xd;
  }
  const int64_t np = 2 * ldh;
  if ((np == 256 || np == 384 || np == 512) && r % 16 == 0) {
    // one shrink for the group: X read once against every A_k (their splits side by side), Hs_k
    // into columns k r .. of H
    SplitTab sp{};
    sp.K = d->in_dim;
    for (int k = 0; k < f.n; ++k) {
      sp.src[k] = f.A[k];
      sp.dst[k] = F.Sacat + (int64_t)k * 2 * r * d->in_dim;
      sp.rank[k] = (int32_t)r;
    }
    LORA_TRY(launch_split(sp, f.n, st));
    TcRowsArgs a{};
    a.a = Xin; a.T = T; a.K = d->in_dim; a.n_slots = 1;
    a.s[0] = F.Sacat; a.rank[0] = (int32_t)ldh;
    a.NP = (int32_t)np; a.pair_r = (int32_t)r;
    a.splits = row_splits(T, -1, d->in_dim);
    a.si = si; a.si.rank[0] = (int32_t)ldh;
    a.out = H; a.ldo = ldh; a.ld_out = ldh;
    a.items = nullptr; a.n_items = nullptr; a.max_items = (int)L.gmax;
    LORA_TRY(launch_tc_rows(a, st, LORA_PROF_SHRINK));
  } else {
    for (int k = 0; k < f.n; ++k) {   // Hs_k = s' Xd A_k^T into columns k r .. of H
      SplitTab sp{};
      sp.K = d->in_dim;
      sp.src[0] = f.A[k];
      sp.dst[0] = L.Sa;
      sp.rank[0] = (int32_t)r;
      LORA_TRY(launch_split(sp, 1, st));
      TcRowsArgs a{};
      a.a = Xin; a.T = T; a.K = d->in_dim; a.n_slots = 1;
      a.s[0] = L.Sa; a.rank[0] = (int32_t)r;
      a.NP = np_for((int)r);
      a.splits = row_splits(T, -1, d->in_dim);
      a.si = si;
      a.out = H + k * r; a.ldo = r; a.ld_out = ldh;
      a.items = nullptr; a.n_items = nullptr; a.max_items = (int)L.gmax;
      LORA_TRY(launch_tc_rows(a, st, LORA_PROF_SHRINK));
    }
  }
  TcGemmArgs t{};
  t.a = X; t.T = T; t.b = W; t.n_rows = d->out_dim; t.K = d->in_dim;
  t.p = H; t.ldp = ldh; t.n_slots = f.n; t.n_col_groups = f.n;
  for (int k = 0; k < f.n; ++k) {
    t.q[k] = f.B[k];
    t.q_rank[k] = (int32_t)r;
    t.col_end[k] = f.off[k] + f.out[k];
    t.p_col[k] = (int32_t)(k * r);
  }
  t.out = Y; t.ldo = d->out_dim;
  t.items = nullptr; t.n_items = nullptr; t.max_items = (int)L.gmax; t.drop = dp;
  LORA_TRY(launch_tc_gemm(t, st, LORA_PROF_FROZEN_FWD));
  return LORA_OK;
}

int run_fused_backward(const lora_desc* d, const DropParams& dp, int64_t T, const void* X,
                       const void* Wt, const FusedProjs& f, const void* dY, const float* H,
                       void* dX, void* ws, cudaStream_t st) {
  FusedLayout F = fused_carve(d, T, f, ws);
  Layout& L = F.L;
  clear_stale();
  use_uniform_items(L, T);
  const int64_t r = d->rank, ldh = (int64_t)f.n * r;
  const SlotInfo si = fused_slot_info(d);
  // one launch: A_k^T into columns k r .. of A^T_cat [in, n r] for the dX product's LoRA term,
  // and the bf16 split of every B_k^T for its G product
  uint16_t* sbk[LORA_MAX_SLOTS];
  {
    TransposeTab ta{};
    SplitTab sp{};
    sp.transposed = 1;
    sp.K = f.out[0];
    int64_t kk[LORA_MAX_SLOTS];
    int64_t ob = 0;
    for (int k = 0; k < f.n; ++k) {
      ta.src[k] = f.A[k];
      ta.dst[k] = F.Atcat + k * r;
      ta.rows[k] = r;
      ta.cols[k] = d->in_dim;
      ta.ld_dst[k] = ldh;
      sbk[k] = F.Sbk + ob;
      sp.src[k] = f.B[k];
      sp.dst[k] = sbk[k];
      sp.rank[k] = (int32_t)r;
      kk[k] = f.out[k];
      ob += 2 * r * f.out[k];
    }
    LORA_TRY(launch_adapter_prep(ta, sp, f.n, st, kk));
  }
  const void* Xin = X;
  if (dp.enabled) {
    LORA_TRY(launch_mask_bf16(X, T, d->in_dim, dp, L.Xd, st));
    Xin = L.Xd;
  }
  const size_t split_bytes = (size_t)2 * r * L.ldt * sizeof(uint16_t);
  const uint16_t* dYb = static_cast<const uint16_t*>(dY);
  // dA of the whole group in one reduction that reads Xd once, after every G_k
  const bool group_da = f.n >= 2 && f.n <= 4 && 2 * r <= 128 && d->in_dim % 8 == 0;
  for (int k = 0; k < f.n; ++k) {
    // G_k = s' dY_k B_k (projection k's columns of dY) into columns k r .. of G, with its
    // transposed split for dA_k and, as a side task, the transposed split of the saved Hs_k,
    // each in the projection's own region
    TcRowsArgs g{};
    g.a = dYb + f.off[k]; g.lda = d->out_dim; g.T = T; g.K = f.out[k]; g.n_slots = 1;
    g.s[0] = sbk[k]; g.rank[0] = (int32_t)r;
    g.NP = np_for((int)r);
    g.splits = row_splits(T, -1, f.out[k]);
    g.si = si;
    g.out = F.Gcat + k * r; g.ldo = r; g.ld_out = ldh;
    g.outT = F.GsTk + (int64_t)k * 2 * r * L.ldt; g.ldt = L.ldt; g.outT_bytes = split_bytes;
    g.side_h = H + k * r; g.side_ldh = ldh; g.side_outT = F.HsTk + (int64_t)k * 2 * r * L.ldt;
    g.items = nullptr; g.n_items = nullptr; g.max_items = (int)L.gmax;
    LORA_TRY(launch_tc_rows(g, st, LORA_PROF_G));
  }
  // dB_k += dY_k^T Hs_k for every k and, without the group dA, dA_k += Gs_k^T Xd: jobs of shared
  // reduction launches
  TcRedArgs jobs[2 * LORA_MAX_SLOTS];
  int nj = 0;
  for (int k = 0; k < f.n; ++k) {
    TcRedArgs& b = jobs[nj++];
    b = TcRedArgs{};
    b.st[0] = F.HsTk + (int64_t)k * 2 * r * L.ldt;
    b.rank[0] = (int32_t)r; b.n_slots = 1; b.max_rank = (int32_t)r;
    b.T = T; b.ldt = L.ldt; b.b = dYb + f.off[k]; b.ldb = d->out_dim; b.N = f.out[k];
    b.tab.rank[0] = (int32_t)r; b.tab.out[0] = f.dB[k]; b.transposed = 1;
    if (!group_da) {
      TcRedArgs& a = jobs[nj++];
      a = TcRedArgs{};
      a.st[0] = F.GsTk + (int64_t)k * 2 * r * L.ldt;
      a.rank[0] = (int32_t)r; a.n_slots = 1; a.max_rank = (int32_t)r;
      a.T = T; a.ldt = L.ldt; a.b = Xin; a.N = d->in_dim;
      a.tab.rank[0] = (int32_t)r; a.tab.out[0] = f.dA[k]; a.transposed = 0;
    }
  }
  LORA_TRY(launch_tc_red_n(jobs, nj, st, group_da ? LORA_PROF_RED_DB : LORA_PROF_RED));
  if (group_da) {   // dA_k += Gs_k^T Xd for every k, Xd streamed once
    TcRedMultiArgs a{};
    for (int k = 0; k < f.n; ++k) {
      a.st[k] = F.GsTk + (int64_t)k * 2 * r * L.ldt;
      a.dst[k] = f.dA[k];
    }
    a.n = f.n; a.r = (int32_t)r; a.T = T; a.ldt = L.ldt; a.b = Xin; a.N = d->in_dim;
    LORA_TRY(launch_tc_red_multi(a, st, LORA_PROF_RED_DA));
  }
  // dX = dY_cat W_cat + (G_cat A_cat) * M: the projections' input gradients summed in one product
  if (dX) {
    TcGemmArgs t{};
    t.a = dY; t.T = T; t.b = Wt; t.n_rows = d->in_dim; t.K = d->out_dim;
    t.p = F.Gcat; t.ldp = ldh; t.n_slots = 1;
    t.q[0] = F.Atcat; t.q_rank[0] = (int32_t)ldh;
    t.lora_separate = dp.enabled; t.out = dX; t.ldo = d->in_dim;
    t.items = nullptr; t.n_items = nullptr; t.max_items = (int)L.gmax; t.drop = dp;
    LORA_TRY(launch_tc_gemm(t, st, LORA_PROF_FROZEN_DX));
  }
  return LORA_OK;
}

}  // namespace

extern "C" {

const char* lora_last_cuda_error(void) { return cudaGetErrorString(t_last_error); }

int lora_device_error(uint32_t* flags, int32_t reset) {
  if (!flags) return LORA_ERR_INVALID;
  return cuda_status(read_tc_error(flags, reset != 0));
}

int lora_device_check(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e);
  uint32_t flags = 0;
  e = read_tc_error(&flags, false);
  if (e != cudaSuccess) return cuda_status(e);
  return flags ? LORA_ERR_TIMEOUT : LORA_OK;
}

int lora_set_wait_limit(uint64_t cycles) {
  set_tc_wait_limit((unsigned long long)cycles);
  return LORA_OK;
}

const char* lora_status_string(int status) {
  switch (status) {
    case LORA_OK: return "ok";
    case LORA_ERR_INVALID: return "invalid argument";
    case LORA_ERR_ALIGN: return "pointer or row stride not 16-byte aligned";
    case LORA_ERR_UNSUPPORTED: return "unsupported dtype, rank or size";
    case LORA_ERR_WORKSPACE: return "workspace too small";
    case LORA_ERR_CUDA: return "CUDA launch or runtime error";
    case LORA_ERR_NONFINITE: return "non-finite gradient: update rejected";
    case LORA_ERR_TIMEOUT: return "a device pipeline wait ran out of its bound: outputs invalid";
    default: return "unknown status";
  }
}

float lora_scale(float alpha, int32_t rank, int32_t rslora) {
  if (rank <= 0) return 0.f;
  return rslora ? (float)((double)alpha / std::sqrt((double)rank)) : (float)((double)alpha / rank);
}

double lora_lr_at(int32_t kind, double base, uint64_t step, uint64_t warmup, uint64_t total,
                  double min_lr) {
  if (kind == LORA_SCHED_CONSTANT) return base;
  if (kind != LORA_SCHED_WARMUP_COSINE) return std::nan("");
  if (step < warmup) return base * (double)(step + 1) / (double)warmup;
  if (total <= warmup) return min_lr;
  double progress = (double)(step - warmup) / (double)(total - warmup);
  if (progress > 1.0) progress = 1.0;
  return min_lr + 0.5 * (base - min_lr) * (1.0 + std::cos(M_PI * progress));
}

size_t lora_workspace_size(const lora_desc* d, int64_t T) {
  if (check_desc(d, T, false) != LORA_OK) return 0;
  return ws_size(d, T, -1, 1, d->rank);
}

size_t multi_lora_workspace_size(const lora_desc* d, int64_t T, int32_t n_seg, int32_t n_slots,
                                 const lora_slot* slots) {
  if (check_desc(d, T, true) != LORA_OK || n_seg < 0) return 0;
  Slots s;
  if (slots_from_table(d, n_slots, slots, false, s) != LORA_OK) return 0;
  return ws_size(d, T, n_seg, s.n, s.rank_sum);
}

size_t lora_prepared_weight_size(const lora_desc* d) {
  if (check_desc(d, 0, false) != LORA_OK) return 0;
  const size_t n = (size_t)d->out_dim * (size_t)d->in_dim;
  if (d->dtype == LORA_BF16_FP8) return fp8_prep_bytes(d->out_dim, d->in_dim);
  return d->dtype == LORA_F32 ? 8 * n : 2 * n;
}

int lora_prepare_weight(const lora_desc* d, const void* W, void* W_prep, void* stream) {
  int rc = check_desc(d, 0, false);
  if (rc) return rc;
  if (!W || !W_prep) return LORA_ERR_INVALID;
  if (!al16(W) || !al16(W_prep)) return LORA_ERR_ALIGN;
  clear_stale();
  if (d->dtype == LORA_BF16_FP8) {
    // W8: W's rows (forward: K = in), WT8: W's columns as rows (dX: K = out)
    const Fp8Prep f = fp8_prep(W_prep, d->out_dim, d->in_dim);
    cudaError_t e = launch_quant_rows_e4m3(W, d->out_dim, d->in_dim, const_cast<uint8_t*>(f.W8),
                                           const_cast<float*>(f.sw), (cudaStream_t)stream);
    if (e == cudaSuccess)
      e = launch_quant_cols_e4m3(W, d->out_dim, d->in_dim, const_cast<uint8_t*>(f.WT8),
                                 const_cast<float*>(f.swT), (cudaStream_t)stream);
    return cuda_status(e);
  }
  return cuda_status(launch_prepare_weight(d->dtype, W, W_prep, d->out_dim, d->in_dim,
                                           (cudaStream_t)stream));
}

size_t lora_dora_norm_workspace_size(const lora_desc* d) {
  if (check_desc(d, 0, false) != LORA_OK) return 0;
  return dora_norm_carve(d, nullptr).bytes;
}

int lora_dora_norm(const lora_desc* d, const void* W, const float* A, const float* B,
                   float* norm_out, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_desc(d, 0, false);
  if (rc) return rc;
  if (!W || !A || !B || !norm_out || !ws) return LORA_ERR_INVALID;
  if (!al16(W) || !al16(A) || !al16(B) || !al16(norm_out) || !al16(ws)) return LORA_ERR_ALIGN;
  if (ws_bytes < dora_norm_carve(d, nullptr).bytes) return LORA_ERR_WORKSPACE;
  clear_stale();
  cudaStream_t st = (cudaStream_t)stream;
  if (d->dtype == LORA_F32)
    return cuda_status(launch_dora_norm(d->dtype, W, A, B, d->scale, d->out_dim, d->in_dim,
                                        d->rank, norm_out, st));
  return cuda_status(run_dora_norm_tc(d, W, A, B, norm_out, ws, st));
}

int lora_forward(const lora_desc* d, const lora_ctx* c, int64_t T, const void* X, const void* W,
                 const void* W_prep, const float* A, const float* B, const float* dora_m,
                 const float* dora_n, void* Y, float* H_save, void* ws, size_t ws_bytes,
                 void* stream) {
  int rc = check_desc(d, T, false);
  if (rc) return rc;
  DropParams dp;
  if ((rc = build_drop(d, c, T, dp))) return rc;
  if (!X || !W || !W_prep || !A || !B || !Y || !H_save || !ws) return LORA_ERR_INVALID;
  if (d->dora && (!dora_m || !dora_n)) return LORA_ERR_INVALID;
  if (!al16(X) || !al16(W) || !al16(W_prep) || !al16(A) || !al16(B) || !al16(Y) ||
      !al16(H_save) || !al16(ws))
    return LORA_ERR_ALIGN;
  if (d->dora && (!al16(dora_m) || !al16(dora_n))) return LORA_ERR_ALIGN;
  if (ws_bytes < ws_size(d, T, -1, 1, d->rank)) return LORA_ERR_WORKSPACE;
  if (T == 0) return LORA_OK;
  Slots s;
  single_slot(d, A, B, nullptr, nullptr, s);
  return run_forward(d, dp, T, X, W, W_prep, -1, nullptr, nullptr, s, d->dora ? dora_m : nullptr,
                     d->dora ? dora_n : nullptr, Y, H_save, ws, (cudaStream_t)stream);
}

int lora_backward(const lora_desc* d, const lora_ctx* c, int64_t T, const void* X,
                  const void* W_prep, const float* A, const float* B, const void* dY,
                  const float* H_save, const float* dora_m, const float* dora_n,
                  const void* Y_save, void* dX, float* dA, float* dB, float* dm, void* ws,
                  size_t ws_bytes, void* stream) {
  int rc = check_desc(d, T, false);
  if (rc) return rc;
  DropParams dp;
  if ((rc = build_drop(d, c, T, dp))) return rc;
  if (!X || !W_prep || !A || !B || !dY || !H_save || !dA || !dB || !ws) return LORA_ERR_INVALID;
  if (d->dora && (!dora_m || !dora_n || !Y_save || !dm)) return LORA_ERR_INVALID;
  if (!al16(X) || !al16(W_prep) || !al16(A) || !al16(B) || !al16(dY) || !al16(H_save) || !al16(dA) ||
      !al16(dB) || !al16(ws) || (dX && !al16(dX)))
    return LORA_ERR_ALIGN;
  if (d->dora && (!al16(dora_m) || !al16(dora_n) || !al16(Y_save) || !al16(dm)))
    return LORA_ERR_ALIGN;
  if (ws_bytes < ws_size(d, T, -1, 1, d->rank)) return LORA_ERR_WORKSPACE;
  if (T == 0) return LORA_OK;
  Slots s;
  single_slot(d, A, B, dA, dB, s);
  return run_backward(d, dp, T, X, W_prep, -1, nullptr, nullptr, s, dY, H_save,
                      d->dora ? dora_m : nullptr, d->dora ? dora_n : nullptr, Y_save, dX,
                      d->dora ? dm : nullptr, ws, (cudaStream_t)stream);
}

}  // extern "C"

namespace {
int multi_forward(const lora_desc* d, const lora_ctx* c, int64_t T, const void* X, const void* W,
                  const void* W_prep, int32_t n_seg, const int32_t* d_seg_start,
                  const int32_t* d_seg_slot, const RoutePlan* plan, int32_t n_slots,
                  const lora_slot* slots, void* Y, float* H_save, void* ws, size_t ws_bytes,
                  void* stream) {
  int rc = check_desc(d, T, true);
  if (rc) return rc;
  DropParams dp;
  if ((rc = build_drop(d, c, T, dp))) return rc;
  Slots s;
  if ((rc = slots_from_table(d, n_slots, slots, false, s))) return rc;
  if (n_seg < 0 || (n_seg > 0 && !plan && (!d_seg_start || !d_seg_slot))) return LORA_ERR_INVALID;
  if (!X || !W || !W_prep || !Y || !H_save || !ws) return LORA_ERR_INVALID;
  if (!al16(X) || !al16(W) || !al16(W_prep) || !al16(Y) || !al16(H_save) || !al16(ws))
    return LORA_ERR_ALIGN;
  if (ws_bytes < ws_size(d, T, n_seg, s.n, s.rank_sum)) return LORA_ERR_WORKSPACE;
  if (T == 0) return LORA_OK;
  return run_forward(d, dp, T, X, W, W_prep, n_seg, n_seg ? d_seg_start : nullptr,
                     n_seg ? d_seg_slot : nullptr, s, nullptr, nullptr, Y, H_save, ws,
                     (cudaStream_t)stream, plan);
}

int multi_backward(const lora_desc* d, const lora_ctx* c, int64_t T, const void* X,
                   const void* W_prep, int32_t n_seg, const int32_t* d_seg_start,
                   const int32_t* d_seg_slot, const RoutePlan* plan, int32_t n_slots,
                   const lora_slot* slots, const void* dY, const float* H_save, void* dX, void* ws,
                   size_t ws_bytes, void* stream) {
  int rc = check_desc(d, T, true);
  if (rc) return rc;
  DropParams dp;
  if ((rc = build_drop(d, c, T, dp))) return rc;
  Slots s;
  if ((rc = slots_from_table(d, n_slots, slots, true, s))) return rc;
  if (n_seg < 0 || (n_seg > 0 && !plan && (!d_seg_start || !d_seg_slot))) return LORA_ERR_INVALID;
  if (!X || !W_prep || !dY || !H_save || !ws) return LORA_ERR_INVALID;
  if (!al16(X) || !al16(W_prep) || !al16(dY) || !al16(H_save) || !al16(ws) || (dX && !al16(dX)))
    return LORA_ERR_ALIGN;
  if (ws_bytes < ws_size(d, T, n_seg, s.n, s.rank_sum)) return LORA_ERR_WORKSPACE;
  if (T == 0) return LORA_OK;
  return run_backward(d, dp, T, X, W_prep, n_seg, n_seg ? d_seg_start : nullptr,
                      n_seg ? d_seg_slot : nullptr, s, dY, H_save, nullptr, nullptr, nullptr, dX,
                      nullptr, ws, (cudaStream_t)stream, plan);
}

// a plan's tables for (T, n_seg, n_slots), or LORA_ERR_* on bad arguments
int plan_of(int64_t T, int32_t n_seg, int32_t n_slots, const void* plan, RoutePlan& P) {
  if (!plan || T < 0 || n_seg < 1 || n_slots < 1 || n_slots > LORA_MAX_SLOTS)
    return LORA_ERR_INVALID;
  if (!al16(plan)) return LORA_ERR_ALIGN;
  P = plan_carve(T, n_seg, n_slots, const_cast<void*>(plan));
  return LORA_OK;
}
}  // namespace

extern "C" {

int multi_lora_forward(const lora_desc* d, const lora_ctx* c, int64_t T, const void* X,
                       const void* W, const void* W_prep, int32_t n_seg,
                       const int32_t* d_seg_start, const int32_t* d_seg_slot, int32_t n_slots,
                       const lora_slot* slots, void* Y, float* H_save, void* ws, size_t ws_bytes, void* stream) {
  return multi_forward(d, c, T, X, W, W_prep, n_seg, d_seg_start, d_seg_slot, nullptr, n_slots,
                       slots, Y, H_save, ws, ws_bytes, stream);
}

int multi_lora_backward(const lora_desc* d, const lora_ctx* c, int64_t T, const void* X,
                        const void* W_prep, int32_t n_seg, const int32_t* d_seg_start,
                        const int32_t* d_seg_slot, int32_t n_slots, const lora_slot* slots,
                        const void* dY, const float* H_save, void* dX, void* ws,
                        size_t ws_bytes, void* stream) {
  return multi_backward(d, c, T, X, W_prep, n_seg, d_seg_start, d_seg_slot, nullptr, n_slots,
                        slots, dY, H_save, dX, ws, ws_bytes, stream);
}

size_t multi_lora_plan_size(int64_t T, int32_t n_seg, int32_t n_slots) {
  if (T < 0 || n_seg < 1 || n_slots < 1 || n_slots > LORA_MAX_SLOTS) return 0;
  return plan_carve(T, n_seg, n_slots, nullptr).bytes;
}

int multi_lora_plan_build(int64_t T, int32_t n_seg, const int32_t* d_seg_start,
                          const int32_t* d_seg_slot, int32_t n_slots, void* plan, size_t plan_bytes,
                          void* stream) {
  RoutePlan P;
  int rc = plan_of(T, n_seg, n_slots, plan, P);
  if (rc) return rc;
  if (!d_seg_start || !d_seg_slot) return LORA_ERR_INVALID;
  if (T > INT32_MAX - 256) return LORA_ERR_UNSUPPORTED;
  if (plan_bytes < P.bytes) return LORA_ERR_WORKSPACE;
  if (T == 0) return LORA_OK;   // planned calls over no tokens return before reading the plan
  clear_stale();
  const cudaStream_t st = (cudaStream_t)stream;
  LORA_TRY(launch_make_items(T, n_seg, d_seg_start, d_seg_slot, n_slots, P.gitems, P.gcount,
                             (int32_t)P.gmax, P.ritems, P.rcount, (int32_t)P.rmax, st));
  LORA_TRY(launch_make_red_items_tc(T, n_seg, d_seg_start, d_seg_slot, n_slots, kRedSpanBlocks,
                                    P.items_red, P.count_red, (int32_t)P.max_red, st));
  LORA_TRY(launch_tile_slot_masks(T, n_seg, d_seg_start, d_seg_slot, n_slots, P.tmask, st));
  return LORA_OK;
}

int multi_lora_forward_planned(const lora_desc* d, const lora_ctx* c, int64_t T, int32_t n_seg,
                               const void* plan, const void* X, const void* W, const void* W_prep,
                               int32_t n_slots, const lora_slot* slots, void* Y, float* H_save,
                               void* ws, size_t ws_bytes, void* stream) {
  RoutePlan P;
  int rc = plan_of(T, n_seg, n_slots, plan, P);
  if (rc) return rc;
  return multi_forward(d, c, T, X, W, W_prep, n_seg, nullptr, nullptr, &P, n_slots, slots, Y,
                       H_save, ws, ws_bytes, stream);
}

int multi_lora_backward_planned(const lora_desc* d, const lora_ctx* c, int64_t T, int32_t n_seg,
                                const void* plan, const void* X, const void* W_prep,
                                int32_t n_slots, const lora_slot* slots, const void* dY,
                                const float* H_save, void* dX, void* ws, size_t ws_bytes,
                                void* stream) {
  RoutePlan P;
  int rc = plan_of(T, n_seg, n_slots, plan, P);
  if (rc) return rc;
  return multi_backward(d, c, T, X, W_prep, n_seg, nullptr, nullptr, &P, n_slots, slots, dY,
                        H_save, dX, ws, ws_bytes, stream);
}

size_t lora_grad_prepare_workspace_size(int32_t n_groups, const lora_group* groups) {
  if (!groups || n_groups < 1 || n_groups > LORA_MAX_GROUPS) return 0;
  GroupTab g{};
  g.n = n_groups;
  for (int i = 0; i < n_groups; ++i) g.count[i] = groups[i].n_a + groups[i].n_b + groups[i].n_mag;
  const int blocks = prepare_blocks(g);
  Carve c(nullptr);
  c.take<double>((size_t)(blocks > 0 ? blocks : 1));
  c.take<uint32_t>(4);
  return c.off + kWsAlign;
}

}  // extern "C"

namespace {
int build_groups(int32_t n_groups, const lora_group* groups, GroupTab& g, const lora_adamw_hp* hp) {
  if (!groups || n_groups < 1) return LORA_ERR_INVALID;
  if (n_groups > LORA_MAX_GROUPS) return LORA_ERR_UNSUPPORTED;
  std::memset(&g, 0, sizeof(g));
  g.n = n_groups;
  for (int i = 0; i < n_groups; ++i) {
    const lora_group& e = groups[i];
    if (e.offset < 0 || e.n_a < 0 || e.n_b < 0 || e.n_mag < 0 || e.step < 0) return LORA_ERR_INVALID;
    if (!(e.max_norm >= 0.f) || !std::isfinite(e.grad_scale) || !std::isfinite(e.lr))
      return LORA_ERR_INVALID;
    if (e.offset % 4) return LORA_ERR_ALIGN;
    g.offset[i] = e.offset;
    g.count[i] = e.n_a + e.n_b + e.n_mag;
    g.n_a[i] = e.n_a;
    g.n_b[i] = e.n_b;
    g.gamma[i] = e.grad_scale;
    g.max_norm[i] = e.max_norm;
    g.lr[i] = e.lr;
    if (hp) {
      const double k = (double)e.step + 1.0;
      g.bc1[i] = (float)(1.0 - std::pow((double)hp->beta1, k));
      g.bc2[i] = (float)(1.0 - std::pow((double)hp->beta2, k));
      if (!(g.bc1[i] > 0.f) || !(g.bc2[i] > 0.f)) return LORA_ERR_INVALID;
    }
  }
  for (int i = 0; i < n_groups; ++i)
    for (int j = i + 1; j < n_groups; ++j) {
      const int64_t a0 = g.offset[i], a1 = a0 + g.count[i], b0 = g.offset[j], b1 = b0 + g.count[j];
      if (a0 < b1 && b0 < a1 && g.count[i] > 0 && g.count[j] > 0) return LORA_ERR_INVALID;
    }
  return LORA_OK;
}
}  // namespace

extern "C" {

int lora_grad_prepare(const float* grads, int32_t n_groups, const lora_group* groups,
                      double* d_scale_norm, int32_t* d_status, void* ws, size_t ws_bytes,
                      void* stream) {
  GroupTab g;
  int rc = build_groups(n_groups, groups, g, nullptr);
  if (rc) return rc;
  if (!grads || !d_scale_norm || !d_status || !ws) return LORA_ERR_INVALID;
  if (!al16(grads) || !al16(ws) || (reinterpret_cast<uintptr_t>(d_scale_norm) & 7u) ||
      (reinterpret_cast<uintptr_t>(d_status) & 3u))
    return LORA_ERR_ALIGN;
  if (ws_bytes < lora_grad_prepare_workspace_size(n_groups, groups)) return LORA_ERR_WORKSPACE;
  const int blocks = prepare_blocks(g);   // the workspace holds this many partials (the most)
  Carve c(ws);
  double* part = c.take<double>((size_t)(blocks > 0 ? blocks : 1));
  uint32_t* counter = c.take<uint32_t>(4);
  // elements per CTA: enough CTAs for about eight per SM over the whole arena, each streaming a
  // long run (a multiple of the workspace form's run, so the partials still fit)
  int64_t total = 0;
  for (int i = 0; i < g.n; ++i) total += g.count[i];
  int64_t per = (total / kPrepTargetBlocks + kPrepElemsWs - 1) / kPrepElemsWs * kPrepElemsWs;
  if (per < kPrepElemsWs) per = kPrepElemsWs;
  clear_stale();
  return cuda_status(launch_grad_prepare(grads, g, d_scale_norm, d_status, part, counter,
                                         (cudaStream_t)stream, per));
}

int lora_grad_prepare_noalloc(const float* grads, int32_t n_groups, const lora_group* groups,
                              double* d_scale_norm, int32_t* d_status, void* stream) {
  GroupTab g;
  int rc = build_groups(n_groups, groups, g, nullptr);
  if (rc) return rc;
  if (!grads || !d_scale_norm || !d_status) return LORA_ERR_INVALID;
  if (!al16(grads) || (reinterpret_cast<uintptr_t>(d_scale_norm) & 7u) ||
      (reinterpret_cast<uintptr_t>(d_status) & 3u))
    return LORA_ERR_ALIGN;
  if (prepare_blocks(g, kPrepElemsPerBlock) > kNoallocMaxPartials) return LORA_ERR_UNSUPPORTED;
  clear_stale();
  return cuda_status(launch_grad_prepare_noalloc(grads, g, d_scale_norm, d_status,
                                                 (cudaStream_t)stream));
}

int lora_adamw_step(float* params, float* grads, float* m, float* v, int32_t n_groups,
                    const lora_group* groups, const lora_adamw_hp* hp, const double* d_scale_norm,
                    const int32_t* d_status, int32_t zero_grads, void* stream) {
  if (!hp) return LORA_ERR_INVALID;
  if (!(hp->beta1 >= 0.0 && hp->beta1 < 1.0 && hp->beta2 >= 0.0 && hp->beta2 < 1.0 &&
        hp->eps > 0.0 && std::isfinite(hp->weight_decay) && std::isfinite(hp->plus_ratio)))
    return LORA_ERR_INVALID;
  GroupTab g;
  int rc = build_groups(n_groups, groups, g, hp);
  if (rc) return rc;
  if (!params || !grads || !m || !v || !d_scale_norm || !d_status) return LORA_ERR_INVALID;
  if (!al16(params) || !al16(grads) || !al16(m) || !al16(v)) return LORA_ERR_ALIGN;
  AdamK k;
  k.b1 = (float)hp->beta1;
  k.omb1 = (float)(1.0 - hp->beta1);
  k.b2 = (float)hp->beta2;
  k.omb2 = (float)(1.0 - hp->beta2);
  k.eps = (float)hp->eps;
  k.wd = (float)hp->weight_decay;
  k.rho = (float)hp->plus_ratio;
  clear_stale();
  return cuda_status(launch_adamw(params, grads, m, v, g, k, d_scale_norm, d_status, zero_grads,
                                  (cudaStream_t)stream));
}

int lora_snapshot(const float* params, float* snap, int32_t n_groups, const lora_group* groups,
                  void* stream) {
  GroupTab g;
  int rc = build_groups(n_groups, groups, g, nullptr);
  if (rc) return rc;
  if (!params || !snap) return LORA_ERR_INVALID;
  if (!al16(params) || !al16(snap)) return LORA_ERR_ALIGN;
  clear_stale();
  return cuda_status(launch_group_maint(snap, params, nullptr, nullptr, nullptr, g, kMaintCopy,
                                        (cudaStream_t)stream));
}

int lora_restore(float* params, const float* snap, float* grads, float* m, float* v,
                 int32_t n_groups, const lora_group* groups, int32_t zero_grads, void* stream) {
  GroupTab g;
  int rc = build_groups(n_groups, groups, g, nullptr);
  if (rc) return rc;
  if (!params || !snap || !m || !v || (zero_grads && !grads)) return LORA_ERR_INVALID;
  if (!al16(params) || !al16(snap) || !al16(m) || !al16(v) || (zero_grads && !al16(grads)))
    return LORA_ERR_ALIGN;
  clear_stale();
  const int flags = kMaintCopy | kMaintZeroMV | (zero_grads ? kMaintZeroG : 0);
  return cuda_status(launch_group_maint(params, snap, grads, m, v, g, flags,
                                        (cudaStream_t)stream));
}

int lora_retire(float* params, float* grads, float* m, float* v, int32_t n_groups,
                const lora_group* groups, int32_t clear_params, void* stream) {
  GroupTab g;
  int rc = build_groups(n_groups, groups, g, nullptr);
  if (rc) return rc;
  if (!grads || !m || !v || (clear_params && !params)) return LORA_ERR_INVALID;
  if (!al16(grads) || !al16(m) || !al16(v) || (clear_params && !al16(params)))
    return LORA_ERR_ALIGN;
  clear_stale();
  const int flags = kMaintZeroG | kMaintZeroMV | (clear_params ? kMaintZeroDst : 0);
  return cuda_status(launch_group_maint(params, nullptr, grads, m, v, g, flags,
                                        (cudaStream_t)stream));
}

size_t lora_fused_workspace_size(const lora_desc* d, int64_t T, int32_t n_proj,
                                 const lora_proj* projs) {
  if (check_desc(d, T, false) != LORA_OK) return 0;
  FusedProjs f;
  if (fused_from_table(d, n_proj, projs, false, f) != LORA_OK) return 0;
  return fused_ws_bytes(d, T, f);
}

int lora_fused_forward(const lora_desc* d, const lora_ctx* c, int64_t T, const void* X,
                       const void* W, const void* W_prep, int32_t n_proj, const lora_proj* projs,
                       void* Y, float* H_save, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_desc(d, T, false);
  if (rc) return rc;
  FusedProjs f;
  if ((rc = fused_from_table(d, n_proj, projs, false, f))) return rc;
  DropParams dp;
  if ((rc = build_drop(d, c, T, dp))) return rc;
  if (!X || !W || !W_prep || !Y || !H_save || !ws) return LORA_ERR_INVALID;
  if (!al16(X) || !al16(W) || !al16(W_prep) || !al16(Y) || !al16(H_save) || !al16(ws))
    return LORA_ERR_ALIGN;
  if (ws_bytes < fused_ws_bytes(d, T, f)) return LORA_ERR_WORKSPACE;
  if (T == 0) return LORA_OK;
  if (d->dtype == LORA_F32)
    return run_fused_forward_f32(d, dp, T, X, W, W_prep, f, Y, H_save, ws, (cudaStream_t)stream);
  return run_fused_forward(d, dp, T, X, W, f, Y, H_save, ws, (cudaStream_t)stream);
}

int lora_fused_backward(const lora_desc* d, const lora_ctx* c, int64_t T, const void* X,
                        const void* W_prep, int32_t n_proj, const lora_proj* projs,
                        const void* dY, const float* H_save, void* dX, void* ws, size_t ws_bytes,
                        void* stream) {
  int rc = check_desc(d, T, false);
  if (rc) return rc;
  FusedProjs f;
  if ((rc = fused_from_table(d, n_proj, projs, true, f))) return rc;
  DropParams dp;
  if ((rc = build_drop(d, c, T, dp))) return rc;
  if (!X || !W_prep || !dY || !H_save || !ws) return LORA_ERR_INVALID;
  if (!al16(X) || !al16(W_prep) || !al16(dY) || !al16(H_save) || !al16(ws) ||
      (dX && !al16(dX)))
    return LORA_ERR_ALIGN;
  if (ws_bytes < fused_ws_bytes(d, T, f)) return LORA_ERR_WORKSPACE;
  if (T == 0) return LORA_OK;
  if (d->dtype == LORA_F32)
    return run_fused_backward_f32(d, dp, T, X, W_prep, f, dY, H_save, dX, ws, (cudaStream_t)stream);
  return run_fused_backward(d, dp, T, X, W_prep, f, dY, H_save, dX, ws, (cudaStream_t)stream);
}

int lora_quantize_e4m3(const void* src, int64_t rows, int64_t K, uint8_t* codes, float* scales,
                       void* stream) {
  if (rows < 0 || K <= 0 || !src || !codes || !scales) return LORA_ERR_INVALID;
  if (K % 16) return LORA_ERR_ALIGN;
  if (K > 16384) return LORA_ERR_UNSUPPORTED;
  if (!al16(src) || !al16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u)) return LORA_ERR_ALIGN;
  clear_stale();
  return cuda_status(launch_quant_rows_e4m3(src, rows, K, codes, scales, (cudaStream_t)stream));
}

int lora_dropout_mask(const lora_desc* d, const lora_ctx* c, int64_t T, uint8_t* d_mask,
                      void* stream) {
  int rc = check_desc(d, T, false);
  if (rc) return rc;
  DropParams dp;
  if ((rc = build_drop(d, c, T, dp))) return rc;
  if (!d_mask) return LORA_ERR_INVALID;
  clear_stale();
  return cuda_status(launch_dropout_mask(dp, T, d->in_dim, d_mask, (cudaStream_t)stream));
}

int multi_lora_token_slots(int64_t T, int32_t n_seg, const int32_t* d_seg_start,
                           const int32_t* d_seg_slot, int32_t n_slots, int32_t* d_token_slot,
                           void* stream) {
  if (T < 0 || n_seg < 0 || n_slots < 1 || !d_token_slot) return LORA_ERR_INVALID;
  if (n_seg > 0 && (!d_seg_start || !d_seg_slot)) return LORA_ERR_INVALID;
  if (n_slots > LORA_MAX_SLOTS) return LORA_ERR_UNSUPPORTED;
  if (T >= (int64_t(1) << 31) - kRedTileT) return LORA_ERR_UNSUPPORTED;
  if (T == 0) return LORA_OK;
  clear_stale();
  return cuda_status(launch_token_slots(T, n_seg, d_seg_start, d_seg_slot, n_slots, d_token_slot,
                                        (cudaStream_t)stream));
}

}  // extern "C"
