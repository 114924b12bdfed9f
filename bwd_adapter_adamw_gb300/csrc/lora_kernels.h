// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include "lora_common.cuh"

namespace lora {

// profile.cu: programmatic dependent launch switch (on unless LORA_PDL=0 is in the environment).
bool pdl_enabled();

// Appends the programmatic stream serialization attribute to attr[0 .. n) when it is enabled and
// returns the new count. Every kernel begins with grid_dep_sync(), which makes this safe.
inline unsigned add_pdl_attr(cudaLaunchAttribute* attr, unsigned n) {
  if (!pdl_enabled()) return n;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  return n + 1;
}

// Kernel launch on a stream with programmatic dependent launch. Errors are also left for
// cudaGetLastError, like a <<<>>> launch.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = add_pdl_attr(attr, 0);
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// profile.cu: launch counter and optional event brackets per kernel class (LORA_PROF_*).
void prof_begin(int kind, cudaStream_t st);
void prof_end(int kind, cudaStream_t st);

// ---- gemm_tc.cu: tcgen05 frozen products (bf16 activations) ----
struct TcGemmArgs {
  const void* a;             // [T, K] K-contiguous: bf16, or the bf16 hi part (fp32 kernel)
  const void* a_lo;          // fp32 kernel: [T, K] bf16 remainders bf16(a - hi)
  int64_t T;
  const void* b;             // [n_rows, K] K-contiguous: bf16, or the bf16 hi part (fp32 kernel)
  const void* b_lo;          // fp32 kernel: [n_rows, K] bf16 remainders
  int64_t n_rows;
  int64_t K;
  const float* p;            // LoRA term P [T, ldp] fp32 (nullptr: no LoRA term)
  int64_t ldp;
  const float* q[LORA_MAX_SLOTS];   // Q_slot [n_rows, q_rank] fp32
  int32_t q_rank[LORA_MAX_SLOTS];
  int32_t n_slots;
  int32_t lora_separate;     // LoRA term in its own accumulator, masked by dropout at (t, n)
  DropParams drop;
  const float* n_colscale;   // per output column scale (DoRA m / n, or the FP8 W scales), nullable
  const float* m_rowscale;   // per token-row scale (the FP8 activation scales), nullable
  const uint32_t* tile_mask; // routed calls on uniform 128-token tiles: the slots of each tile;
  int32_t slot_pcol[LORA_MAX_SLOTS];   //   slot s's LoRA operand: P columns slot_pcol[s] ..,
  int32_t slot_qx[LORA_MAX_SLOTS];     //   Q map slot_qmap[s] from column slot_qx[s]
  int32_t slot_qmap[LORA_MAX_SLOTS];
  int32_t n_q_maps;          // Q tensor maps to build (0: n_slots)
  int64_t q_inner[LORA_MAX_SLOTS];     // Q_k row length (0: q_rank[k])
  int32_t n_col_groups;      // > 0: fused projections, adapter k covers output columns
  int64_t col_end[LORA_MAX_SLOTS];   //   [col_end[k-1], col_end[k]) (multiples of 256), its
  int32_t p_col[LORA_MAX_SLOTS];     //   LoRA operand in columns p_col[k].. of P
  int32_t fp8;               // 1: A and B are E4M3 codes (kind::f8f6f4), 0: bf16
  void* out;                 // [T, ldo] in the activation dtype
  int64_t ldo;
  const TokenItem* items;     // null: uniform 128-token tiles of a single-adapter call
  const int32_t* n_items;
  int max_items;
};
cudaError_t launch_tc_gemm(const TcGemmArgs& a, cudaStream_t st, int prof_kind);
// gemm_tc_f32.cu: the same products for fp32 activations, as three bf16 products of operands
// split beforehand (bf16 hi / lo)
cudaError_t launch_tc_gemm_f32(const TcGemmArgs& a, cudaStream_t st, int prof_kind);
cudaError_t read_tc_error(uint32_t* out, bool reset);
// Bound (cycles) of the frozen products' pipeline waits for the launches that follow; 0 restores
// the default. Their drain waits (copies in flight, MMAs before the tensor memory is freed) keep
// the default bound.
void set_tc_wait_limit(unsigned long long cycles);

// out_slot[j, i] (+)= sum over items of `slot` of part[item][...]; see lowrank.cu
struct ReduceTab {
  float* out[LORA_MAX_SLOTS];
  int32_t rank[LORA_MAX_SLOTS];
};

// ---- lowrank_tc.cu: tensor-core low-rank products (bf16 activations) ----
struct SlotInfo {
  int32_t rank[LORA_MAX_SLOTS];
  float alpha[LORA_MAX_SLOTS];
  int32_t region[LORA_MAX_SLOTS];   // first row of the slot in a per-slot [sum 2 r, ldt] buffer
  int32_t pcol[LORA_MAX_SLOTS];     // first column of the slot in a slot-expanded [T, ld2] copy
};
struct TcRowsArgs {                 // out[t, j] = alpha * (A[t, :] . (S_hi[j] + S_lo[j]))
  const void* a;                    // [T, K] bf16
  int64_t T;
  int64_t K;
  const uint16_t* s[LORA_MAX_SLOTS];   // per slot [2 r, K] bf16 split (hi rows, lo rows)
  int32_t rank[LORA_MAX_SLOTS];
  int32_t n_slots;
  int32_t NP;                       // MMA N: 16, 32, 64 or 128 (>= 2 * max rank), or 256, 384,
                                    //   512 for adapters side by side (one slot, rank = their
                                    //   total, NP = 2 rank, the split of each in turn)
  int32_t pair_r;                   // NP > 128: rank of each side-by-side adapter
  int32_t splits;                   // K splits: CTAs of one cluster (1, 2, 4 or 8)
  SlotInfo si;
  float* out;                       // [T, ld_out] fp32 (columns < ldo written)
  int64_t ldo;                      // partial row stride (largest rank)
  int64_t ld_out;                   // out row stride (0: ldo)
  int64_t lda;                      // A row stride in elements (0: K)
  float* out2;                      // optional slot-expanded copy [T, ld2]: token t's values in
  int64_t ld2;                      //   columns si.pcol[slot(t)] .. + r (other columns untouched)
  uint16_t* outT;                   // optional per slot [2 r, ldt] bf16 transposed split of out
  int64_t ldt;
  size_t outT_bytes;                // zeroed first when an item table routes several slots
  const float* side_h;              // optional [T, side_ldh] fp32: its transposed bf16 split
  int64_t side_ldh;                 //   goes to side_outT (per slot [2 r, ldt], same layout and
  uint16_t* side_outT;              //   size as outT), written by the same CTAs
  const TokenItem* items;
  const int32_t* n_items;
  int max_items;
};
constexpr int kRedSpanBlocks = 2;   // 64-token blocks per reduction work item
struct TcRedArgs {                  // dst_slot += (ST_hi + ST_lo)[., t] x B[t, .] over the slot's tokens
  const uint16_t* st[LORA_MAX_SLOTS];  // per slot [2 r, ldt] bf16 transposed split
  int32_t rank[LORA_MAX_SLOTS];
  int32_t n_slots;
  int32_t max_rank;
  int64_t T;
  int64_t ldt;
  const void* b;                    // [T, N] bf16 (dY' or Xd), row stride ldb
  int64_t N;
  int64_t ldb;                      // 0: N
  ReduceTab tab;
  int32_t transposed;               // 1: dst is [N, r] (dB); 0: dst is [r, N] (dA)
  const TokenItem* items;           // 64-token aligned runs grouped by slot
  const int32_t* n_items;           //   (launch_make_red_items_tc); null: slot 0 over all T
};
struct SplitTab {
  const float* src[LORA_MAX_SLOTS];
  uint16_t* dst[LORA_MAX_SLOTS];
  int32_t rank[LORA_MAX_SLOTS];
  int64_t K;
  int32_t transposed;               // src is [K, r] instead of [r, K]
};
// dA of n (2 .. 4) adapters of rank r that read one input, the input streamed once:
// dst[m] [r, N] += sum_t (ST_m[j, t] + ST_m[r + j, t]) B[t, n] over all T tokens
struct TcRedMultiArgs {
  const uint16_t* st[LORA_MAX_SLOTS];  // per adapter [2 r, ldt] bf16 transposed split
  float* dst[LORA_MAX_SLOTS];
  int32_t n, r;
  int64_t T, ldt;
  const void* b;                        // [T, N] bf16, row stride ldb
  int64_t N, ldb;
};
cudaError_t launch_tc_red_multi(const TcRedMultiArgs& a, cudaStream_t st, int prof_kind);
cudaError_t launch_tc_rows(const TcRowsArgs& a, cudaStream_t st, int prof_kind);
cudaError_t launch_tc_red(const TcRedArgs& a, cudaStream_t st, int prof_kind);
// Reductions over the same tokens, slots, ranks and run table (dB and dA of a linear, the dB of
// every projection of a fused group) sharing launches, up to four jobs per launch;
// cudaErrorInvalidValue when they differ in any of these.
cudaError_t launch_tc_red_n(const TcRedArgs* jobs, int n, cudaStream_t st, int prof_kind);
cudaError_t launch_tc_red2(const TcRedArgs& a, const TcRedArgs& b, cudaStream_t st, int prof_kind);
cudaError_t launch_split(const SplitTab& t, int n, cudaStream_t st);
// count[0] = the number of items; count[1 + k] (k = 0 .. n_slots) = the first item of slot k, the
// items being grouped by slot in slot order (count needs n_slots + 2 entries).
cudaError_t launch_make_red_items_tc(int64_t T, int32_t n_seg, const int32_t* seg_start,
                                     const int32_t* seg_slot, int32_t n_slots, int32_t span_blocks,
                                     TokenItem* items, int32_t* count, int32_t max_items,
                                     cudaStream_t st);
// the same table built by a parallel coverage pass (lowrank.cu), for 1 .. 2048 segments
cudaError_t launch_make_red_items_par(int64_t T, int32_t n_seg, const int32_t* seg_start,
                                      const int32_t* seg_slot, int32_t n_slots,
                                      int32_t span_blocks, TokenItem* items, int32_t* count,
                                      int32_t max_items, cudaStream_t st);
cudaError_t launch_mask_bf16(const void* X, int64_t T, int64_t in_dim, const DropParams& dp,
                             void* Xd, cudaStream_t st);

// ---- fp8.cu: E4M3 frozen base ----
// rows of src [rows, K] bf16 -> dst [rows, K] E4M3 codes, scale[r] = amax_r / 448 (K % 8 == 0,
// K <= 16384)
cudaError_t launch_quant_rows_e4m3(const void* src, int64_t rows, int64_t K, uint8_t* dst,
                                   float* scale, cudaStream_t st);
// columns of W [rows, cols] bf16 -> dst [cols, rows] E4M3 codes (the rows of W^T), scale[c]
cudaError_t launch_quant_cols_e4m3(const void* W, int64_t rows, int64_t cols, uint8_t* dst,
                                   float* scale, cudaStream_t st);
// dst[r, :] = src[r, :] / scale[r] (fp32), two such divisions in one launch (a job with no
// rows is skipped)
struct DivRowsJob {
  const float* src;
  int64_t lds;
  const float* scale;
  int64_t rows, cols;
  float* dst;
  int64_t ldd;
};
cudaError_t launch_div_rows2(const DivRowsJob& a, const DivRowsJob& b, cudaStream_t st);

// ---- lowrank_simt.cu: streaming CUDA-core low-rank products (fp32 activations) ----
struct RowDotArgs {                 // out[t, j] = alpha_slot * sum_k A'[t, k] S_slot[j, k]
  const void* a;                    // [T, lda]
  int64_t lda;
  int64_t K;
  const float* s[LORA_MAX_SLOTS];   // per slot [rank, lds] fp32
  int64_t lds;
  int32_t rank[LORA_MAX_SLOTS];
  float alpha[LORA_MAX_SLOTS];
  int32_t max_rank;
  const float* colscale;            // A'[t, k] = A[t, k] * colscale[k] (nullable)
  int32_t mask;                     // A'[t, k] = 0 where the dropout mask drops (t, k)
  DropParams drop;
  float* out;                       // [T, ldo]
  int32_t ldo;
  const TokenItem* items;           // <= 128-token items (null: uniform tiles, slot 0)
  const int32_t* n_items;
  int64_t T;
  float* part;                      // K-chunk partials [ceil(K / 1024)][T][16] (ranks <= 16)
  int32_t single_pass;              // ranks <= 16: whole K per CTA, no partials
  int32_t s_rows_k;                 // S_slot stored as [K, lds] (element (j, k) at k lds + j)
  // side task done by the kernel's CTAs before the product (saves a launch): write the transpose
  // t_dst [t_cols, t_rows] of t_src [t_rows, t_cols]
  const float* t_src;
  float* t_dst;
  int64_t t_rows, t_cols;
  uint16_t* split_hi;               // bf16, nullable: A' (colscaled, unmasked) rounded to bf16 ...
  uint16_t* split_lo;               // ... and bf16(A' - hi), both [T, K]: the split product's operands
};
struct ColRedArgs {                 // part[item][n][j] = sum_{t in item} P[t, j] B'[t, n]
  const float* p;                   // [T, ldp] fp32
  int64_t ldp;
  const void* b;                    // [T, ldb]
  int64_t ldb;
  int64_t N;
  int32_t rank[LORA_MAX_SLOTS];
  int32_t max_rank;
  const float* colscale;            // B'[t, n] = B[t, n] * colscale[n] (nullable)
  int32_t mask;                     // B'[t, n] = 0 where the dropout mask drops (t, n)
  DropParams drop;
  float* part;                      // [items * sub_groups][N][ldpart]
  int32_t ldpart;
  int32_t sub_groups;               // token groups per item (partials per item)
  const TokenItem* items;
  const int32_t* n_items;
  // single-adapter fused form (out != null, ranks <= 16): kColGroups token groups of all T tokens,
  // one cluster per 64-column block, whose fixed-order sum is added into out ([N, ldpart], or
  // [ldpart, N] when out_transposed)
  int64_t T;
  float* out;
  int32_t out_transposed;
};
constexpr int kColGroups = 8;
constexpr int kColBlock = 64;
cudaError_t launch_rowdot(int dtype, const RowDotArgs& a, int max_items, cudaStream_t st,
                          int prof_kind);
cudaError_t launch_colred(int dtype, const ColRedArgs& a, int max_items, cudaStream_t st,
                          int prof_kind);
// Two fused single-adapter reductions (out set) over the same T and rank in one launch.
cudaError_t launch_colred2(int dtype, const ColRedArgs& a, const ColRedArgs& b, cudaStream_t st,
                           int prof_kind);

// ---- lowrank.cu ----
cudaError_t launch_colscale_bf16(const void* src, const float* scale, int64_t rows, int64_t cols,
                                 void* dst, cudaStream_t st);
// masks[i] = bitmask of the slots routed any token of 128-token tile i (i < ceil(T / 128))
cudaError_t launch_tile_slot_masks(int64_t T, int32_t n_seg, const int32_t* seg_start,
                                   const int32_t* seg_slot, int32_t n_slots, uint32_t* masks,
                                   cudaStream_t st);
cudaError_t launch_make_items(int64_t T, int32_t n_seg, const int32_t* seg_start,
                              const int32_t* seg_slot, int32_t n_slots, TokenItem* gitems,
                              int32_t* gcount, int32_t gmax, TokenItem* ritems, int32_t* rcount,
                              int32_t rmax, cudaStream_t st);

struct TransposeTab {
  const float* src[LORA_MAX_SLOTS];
  float* dst[LORA_MAX_SLOTS];
  int64_t rows[LORA_MAX_SLOTS];   // src rows
  int64_t cols[LORA_MAX_SLOTS];   // src cols
  int64_t ld_dst[LORA_MAX_SLOTS]; // dst row stride (0: rows)
};
cudaError_t launch_transpose_slots(const TransposeTab& t, int n, int64_t max_rows, int64_t max_cols,
                                   cudaStream_t st);
// bf16 backward: A_slot^T (TransposeTab, n slots) and the split of B_slot^T (SplitTab with
// transposed = 1) in one launch
struct AdapterPrepTiles {
  int32_t n, n_t;                       // (task, slot) units; the first n_t are transposes
  int32_t first[2 * LORA_MAX_SLOTS];    // first tile of each unit
  int64_t split_k[LORA_MAX_SLOTS];      // rows of B_slot (its K) for the splits; 0: SplitTab.K
};
cudaError_t launch_adapter_prep(const TransposeTab& ta, const SplitTab& sb, int n,
                                cudaStream_t st, const int64_t* split_k = nullptr);
// fp32 fused projections as one adapter of rank n r: A_cat = [A_0; ...; A_{n-1}] ([n r, in]) and
// the block-diagonal B_cat ([off[n], n r]: B_k in rows off[k].., columns k r..; zeros elsewhere)
struct CatTab {
  const float* A[LORA_MAX_SLOTS];
  const float* B[LORA_MAX_SLOTS];
  float* dA[LORA_MAX_SLOTS];
  float* dB[LORA_MAX_SLOTS];
  int64_t off[LORA_MAX_SLOTS + 1];   // projection k's first output row; off[n] = sum out_k
  int32_t n, r;
  int64_t in;
};
// (dA_cat and dB_cat, when given, are cleared in the same launch)
cudaError_t launch_pack_cat(const CatTab& t, float* Acat, float* Bcat, float* dAcat, float* dBcat,
                            cudaStream_t st);
// dA_k += rows k r .. of dA_cat; dB_k += the diagonal block k of dB_cat (the off-diagonal blocks
// are cross terms of one projection's dY with another's Hs, not gradients)
cudaError_t launch_add_cat_grads(const CatTab& t, const float* dAcat, const float* dBcat,
                                 cudaStream_t st);

// prepared copy of a frozen W [rows, cols]: bf16 W^T, or fp32 bf16-split [W_hi | W_lo | W^T_hi | W^T_lo]
cudaError_t launch_prepare_weight(int dtype, const void* W, void* Wt, int64_t rows, int64_t cols,
                                  cudaStream_t st);

cudaError_t launch_reduce_parts(const float* part, const TokenItem* items, const int32_t* n_items,
                                int max_items, int32_t sub, int64_t M, int64_t ldp, int transposed,
                                const ReduceTab& tab, int n_slots, cudaStream_t st);

cudaError_t launch_dropout_mask(const DropParams& dp, int64_t T, int64_t in_dim, uint8_t* mask,
                                cudaStream_t st);
cudaError_t launch_ratio(const float* num, const float* den, int64_t n, float* out, cudaStream_t st);
cudaError_t launch_token_slots(int64_t T, int32_t n_seg, const int32_t* seg_start,
                               const int32_t* seg_slot, int32_t n_slots, int32_t* token_slot,
                               cudaStream_t st);

// ---- dora.cu ----
cudaError_t launch_dora_norm(int dtype, const void* W, const float* A, const float* B, float s,
                             int64_t out_dim, int64_t in_dim, int32_t rank, float* norm_out,
                             cudaStream_t st);
// bf16 W: the Gram matrix C = A A^T [r, r] and the row norms from H = W A^T [out, r]
cudaError_t launch_dora_gram_combine(const void* W, const float* H, const float* A, const float* B,
                                     float s, int64_t out_dim, int64_t in_dim, int32_t rank,
                                     float* C, float* norm_out, cudaStream_t st);
cudaError_t launch_dora_dm(int dtype, const void* dY, const void* Y, const float* mag, int64_t T,
                           int64_t out_dim, float* dm, cudaStream_t st);

// ---- optim.cu ----
struct GroupTab {
  int32_t n;
  int64_t offset[LORA_MAX_GROUPS];
  int64_t count[LORA_MAX_GROUPS];
  int64_t n_a[LORA_MAX_GROUPS];
  int64_t n_b[LORA_MAX_GROUPS];
  int32_t block_begin[LORA_MAX_GROUPS + 1];
  double gamma[LORA_MAX_GROUPS];
  float max_norm[LORA_MAX_GROUPS];
  float lr[LORA_MAX_GROUPS];
  float bc1[LORA_MAX_GROUPS];   // 1 - beta1^k
  float bc2[LORA_MAX_GROUPS];   // 1 - beta2^k
};
constexpr int kPrepThreads = 256;
constexpr int kPrepElemsWs = kPrepThreads * 16;         // per CTA, workspace form (more CTAs)
constexpr int kPrepElemsPerBlock = kPrepThreads * 64;   // per CTA, allocation-free form
constexpr int64_t kPrepTargetBlocks = 4 * 152;          // CTAs of the workspace form, large arenas (one wave)
// adapter-state maintenance (launch_group_maint flags)
constexpr int kMaintCopy = 1;     // dst = src
constexpr int kMaintZeroDst = 2;  // dst = 0
constexpr int kMaintZeroG = 4;    // grads = 0
constexpr int kMaintZeroMV = 8;   // Adam moments = 0
cudaError_t launch_group_maint(float* dst, const float* src, float* g, float* m, float* v,
                               const GroupTab& gt, int flags, cudaStream_t st);
constexpr int kAdamThreads = 256;
constexpr int kAdamElemsPerBlock = kAdamThreads * 16;

// workspace: [blocks] double partials, [blocks] int flags, 1 int counter
// CTAs (and double partials) of one prepare launch
int prepare_blocks(const GroupTab& g, int64_t per_block = kPrepElemsWs);
cudaError_t launch_grad_prepare(const float* grads, const GroupTab& g, double* d_scale_norm,
                                int32_t* d_status, double* part, uint32_t* counter, cudaStream_t st,
                                int64_t per_block = kPrepElemsWs);
struct AdamK {
  float b1, omb1, b2, omb2, eps, wd, rho;   // 1 - beta formed in double on the host
};
// Allocation-free prepare: at most kNoallocMaxPartials CTAs (partials) in total.
constexpr int kNoallocMaxPartials = 16384;
cudaError_t launch_grad_prepare_noalloc(const float* grads, const GroupTab& g,
                                        double* d_scale_norm, int32_t* d_status, cudaStream_t st);
cudaError_t launch_adamw(float* p, float* g, float* m, float* v, const GroupTab& gt,
                         const AdamK& hp, const double* d_scale_norm, const int32_t* d_status,
                         int zero_grads, cudaStream_t st);

}  // namespace lora
