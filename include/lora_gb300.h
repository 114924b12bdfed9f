/*
 * lora_gb300.h -- C ABI for one training step of a LoRA-adapted linear layer on GB300 (sm_103a).
 *
 * The step (for each adapted linear with frozen W [out, in], adapter A [r, in], B [out, r]):
 *   forward   Y  = X W^T + s' (Xd A^T) B^T,  Xd = M * X, s' = s / (1 - p)
 *             ("8. LoRA Fundamentals", How it works: W_eff = W + s B A, s = alpha/r or alpha/sqrt(r))
 *   DoRA      Y  = (m / n) * (X W^T + s' (Xd A^T) B^T),  n_o = ||W_o + s (B A)_o||, n detached
 *             ("8. LoRA Fundamentals", How it works: canonical DoRA)
 *   backward  dY' = dY (or dY * m/n), G = dY' B, dX = dY' W + s' (G A) * M,
 *             dA += s' G^T Xd, dB += s' dY'^T (Xd A^T), dm += sum_t dY * Y / m
 *             ("Backward Bug Hunts and Vulkan Tiled GEMM", Bug #1 and Bug #2: the activation
 *             gradient through the frozen weight and the out_prod LoRA-B gradient)
 *   prepare   S = sum g^2 (double); non-finite -> reject; c = gamma * min(1, max_norm / norm)
 *             ("4.3. Training Guide", Gradient accumulation and Gradient clipping)
 *   AdamW     A-only decoupled decay from the pre-update value with the scheduled lr; LoRA+ ratio
 *             on B's lr ("4.3. Training Guide", Optimizer and Schedules)
 *   multi     token segments routed to per-slot adapters, per-slot scale/clip/Adam
 *             ("Multi-LoRA Training Example (fully-async)", Design)
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller, row-major, densely packed.
 *     Descriptor structs, group tables and slot tables are HOST pointers read during the call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Every call only
 *     enqueues work on that stream and returns; nothing synchronises unless documented.
 *   - Argument errors are found on the host before any launch and return a nonzero status with
 *     nothing enqueued. A launch error returns LORA_ERR_CUDA.
 *   - The library allocates no device memory. Scratch comes from a caller workspace whose size
 *     the matching *_workspace_size call gives; a smaller workspace returns LORA_ERR_WORKSPACE.
 *   - Calls are not thread-safe on one workspace; two calls in flight need two workspaces.
 *   - Activations X, dY, Y, dX and the frozen W share one dtype (LORA_F32 or LORA_BF16;
 *     LORA_BF16_FP8 is bf16 with an E4M3 frozen product, see its definition).
 *     A, B, their gradients, the Adam moments, H and the DoRA vectors are always fp32.
 *   - Shapes: 1 <= rank <= LORA_MAX_RANK and rank % 4 == 0; in and out multiples of 8;
 *     all pointers 16-byte aligned (LORA_ERR_ALIGN otherwise).
 */
#ifndef LORA_GB300_H
#define LORA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------------------------------*/
#define LORA_OK 0
#define LORA_ERR_INVALID 1      /* null pointer, negative size, bad rank, bad enum */
#define LORA_ERR_ALIGN 2        /* pointer or row stride not 16-byte aligned */
#define LORA_ERR_UNSUPPORTED 3  /* valid request this build does not serve (dtype, rank, sizes) */
#define LORA_ERR_WORKSPACE 4    /* workspace too small */
#define LORA_ERR_CUDA 5         /* a CUDA launch or runtime call failed */
#define LORA_ERR_NONFINITE 6    /* device status: a gradient element is NaN or +-Inf */
#define LORA_ERR_TIMEOUT 7      /* device status: a tensor-core pipeline wait ran out of its bound */

/* ---- enums ----------------------------------------------------------------------------------*/
/* fp32 activations and frozen W. The frozen products (forward and dX) run on bf16 tensor cores as
 * four products of a two-term bf16 split of each operand (hi = bf16(x), lo = bf16(x - hi);
 * hi*hi' + hi*lo' + lo*hi' + lo*lo'), accumulated in fp32 in periods of 256 K-elements; the
 * adapter terms and the low-rank products run in fp32. Each output of the split products is
 * within 2^-17 of sum_k |a_k w_k| of the exact product. Against a float64 reference the
 * per-tensor max relative error is shown below 1e-5 for N(0, 1)-scaled operands with
 * K <= 14336 and for heavy-tailed ones (Student-t, 3 degrees of freedom) up to K = 8192 on the
 * GPU and K = 14336 in the split arithmetic alone. */
#define LORA_F32 0
#define LORA_BF16 1
/* bf16 activations and frozen W whose frozen products (forward and dX) run on E4M3 tensor
 * cores: W quantised once by lora_prepare_weight (per output row for the forward, per input
 * column for dX), X and dY' per token inside each call, every row scaled so that its largest
 * magnitude maps to 448 (r = 448 / amax, codes = e4m3(x * r) rounded to nearest even and
 * saturated, scale = amax / 448, all in fp32; r = scale = 1 for an all-zero row). The adapter
 * branch (shrink, G, dA, dB) reads the bf16 tensors unchanged ("LoRA Training and Serving",
 * Quantized rollout: an FP8 base under a bf16-trained adapter). Single-adapter calls without
 * DoRA; in_dim and out_dim multiples of 16 and at most 16384 (LORA_ERR_UNSUPPORTED otherwise). */
#define LORA_BF16_FP8 2

#define LORA_SCHED_CONSTANT 0
#define LORA_SCHED_WARMUP_COSINE 1

#define LORA_MAX_RANK 64
#define LORA_MAX_SLOTS 32
#define LORA_MAX_GROUPS 64
#define LORA_MAX_CHUNKS_PER_CALL 64

/* One adapted linear. W is [out_dim, in_dim] (nn.Linear layout). */
typedef struct lora_desc {
  int64_t in_dim;
  int64_t out_dim;
  int32_t rank;        /* r; for multi-LoRA calls: the largest slot rank (H row stride) */
  float scale;         /* s = lora_scale(alpha, rank, rslora); ignored by multi-LoRA calls */
  int32_t dtype;       /* LORA_F32 | LORA_BF16 | LORA_BF16_FP8 for X, W, dY, Y, dX */
  float dropout_p;     /* 0 <= p < 1; applies to the adapter branch input only */
  uint64_t seed;       /* dropout seed */
  uint32_t layer_id;   /* dropout key fields */
  uint32_t proj_id;    /* < 65536 */
  int32_t dora;        /* 1: DoRA row-magnitude mode (single-adapter calls only) */
} lora_desc;

/* Where the call's tokens sit in the optimizer step (dropout key fields). Token t of a call
 * belongs to accumulation chunk accum_ordinal + t / chunk_tokens at position t % chunk_tokens;
 * chunk_tokens == 0 means all T tokens are one chunk. At most LORA_MAX_CHUNKS_PER_CALL chunks
 * per call, and accum_ordinal + chunks <= 65536. */
typedef struct lora_ctx {
  uint64_t opt_step;
  uint32_t accum_ordinal;
  int64_t chunk_tokens;
} lora_ctx;

/* One slot of the multi-LoRA page table ("Multi-LoRA Training Example", Design: slot-keyed
 * adapter page table with per-slot rank/alpha). All pointers device, fp32. */
typedef struct lora_slot {
  const float* A;   /* [rank, in_dim] */
  const float* B;   /* [out_dim, rank] */
  float* dA;        /* [rank, in_dim], accumulated (+=) by multi_lora_backward */
  float* dB;        /* [out_dim, rank], accumulated (+=) */
  int32_t rank;     /* 1..desc.rank, multiple of 4 */
  float scale;      /* s_k = lora_scale(alpha_k, rank_k, rslora) */
} lora_slot;

/* A group of adapter parameters stored contiguously in the flat fp32 arenas (params, grads,
 * m, v share one layout): [n_a elements of kind A | n_b of kind B | n_mag DoRA magnitudes]
 * starting at `offset`. One group = one clip norm and one Adam clock: the whole model for a
 * single adapter set (global clip), or one slot for multi-LoRA. */
typedef struct lora_group {
  int64_t offset;
  int64_t n_a;
  int64_t n_b;
  int64_t n_mag;
  double grad_scale;   /* gamma: 1 / prediction tokens, or 1 / adapter_global_batch_size */
  float max_norm;      /* 0 disables clipping (normalisation by gamma still applies) */
  float lr;            /* scheduled learning rate of this update (lora_lr_at) */
  int64_t step;        /* completed updates of this group before this one (bias correction) */
} lora_group;

/* Doubles so that 1 - beta is formed on the host before rounding (0.999f would shift 1 - beta2
 * by 1.3e-5 relative). The kernels compute in fp32. */
typedef struct lora_adamw_hp {
  double beta1;         /* 0.9 */
  double beta2;         /* 0.999 */
  double eps;           /* 1e-8, added outside the square root */
  double weight_decay;  /* applied to kind A only */
  double plus_ratio;    /* LoRA+: B's lr = lr * plus_ratio */
} lora_adamw_hp;

/* ---- host helpers ---------------------------------------------------------------------------*/
/* Static string for a status code. */
const char* lora_status_string(int status);

/* s = alpha / rank, or alpha / sqrt(rank) when rslora != 0 ("8. LoRA Fundamentals", How it
 * works). Returns 0 for rank <= 0. */
float lora_scale(float alpha, int32_t rank, int32_t rslora);

/* Learning rate at optimizer-update index `step` ("4.3. Training Guide", Schedules): constant,
 * or linear warmup base*(step+1)/warmup then cosine from base to min_lr over total - warmup
 * updates (progress clamped to 1). Returns NaN for an unknown kind. */
double lora_lr_at(int32_t kind, double base, uint64_t step, uint64_t warmup, uint64_t total,
                  double min_lr);

/* Workspace bytes for lora_forward / lora_backward on T tokens. */
size_t lora_workspace_size(const lora_desc* d, int64_t T);

/* ---- frozen-weight preparation (once per frozen W, not per step) ----------------------------*/
/* Bytes of the prepared copy of W that lora_prepare_weight writes (W is frozen, so this is made
 * once and kept resident beside W):
 *   bf16: W^T [in_dim, out_dim] bf16, the K-contiguous operand of the dX product
 *         (2 * in_dim * out_dim bytes);
 *   fp32: the bf16 split of W and of W^T for the split tensor-core products, four bf16 arrays
 *         [W_hi | W_lo | W^T_hi | W^T_lo], each element x stored as x_hi = x rounded to bf16
 *         (nearest even) and x_lo = (x - x_hi) rounded to bf16 (8 * in_dim * out_dim bytes);
 *   bf16 with the E4M3 frozen product: [W8 (out x in codes) | sw (out fp32 row scales) |
 *         WT8 (in x out codes of W's columns) | swT (in fp32)], each section starting on a
 *         16-byte boundary (about 2 * in_dim * out_dim bytes).
 * Returns 0 for an invalid descriptor. */
size_t lora_prepared_weight_size(const lora_desc* d);

/* Writes the prepared copy (above) of W [out_dim, in_dim] into W_prep (16-byte aligned, at least
 * lora_prepared_weight_size bytes). */
int lora_prepare_weight(const lora_desc* d, const void* W, void* W_prep, void* stream);

/* DoRA row norm n_o = || W_o + s (B A)_o ||_2 for the current A, B (fp32 [out_dim]); call once
 * per optimizer step before the first forward ("8. LoRA Fundamentals", How it works, and its
 * norm-refresh event). For bf16 W it is evaluated on tensor cores from the expanded form
 * ||W_o||^2 + 2 s (W A^T)_o . B_o + s^2 B_o (A A^T) B_o^T (the same quantity); scratch comes from
 * ws (at least lora_dora_norm_workspace_size bytes, 16-byte aligned). */
size_t lora_dora_norm_workspace_size(const lora_desc* d);
int lora_dora_norm(const lora_desc* d, const void* W, const float* A, const float* B,
                   float* norm_out, void* ws, size_t ws_bytes, void* stream);

/* ---- forward / backward (one adapted linear, T tokens) --------------------------------------*/
/* Y [T, out] = X W^T + Hs B^T, then * (dora_m / dora_n) per column in DoRA mode.
 * W is the frozen weight and W_prep its prepared copy (lora_prepare_weight); both are required
 * (the bf16 product reads W, the fp32 product reads W_prep).
 * H_save [T, rank] fp32 receives Hs = s' (Xd A^T) (the scaled shrink), which lora_backward
 * reads. dora_m, dora_n: [out] fp32, required iff desc.dora. */
int lora_forward(const lora_desc* d, const lora_ctx* c, int64_t T, const void* X, const void* W,
                 const void* W_prep, const float* A, const float* B, const float* dora_m,
                 const float* dora_n, void* Y, float* H_save, void* ws, size_t ws_bytes,
                 void* stream);

/* dX [T, in] = dY' W + (Gs A) * M with Gs = s' dY' B (written, may be NULL to skip dX);
 * dA [r, in] += Gs^T Xd; dB [out, r] += dY'^T H_save; dm [out] += sum_t dY * Y_save / m (DoRA).
 * W_prep from lora_prepare_weight. Y_save (the forward's Y) and dm are required iff desc.dora.
 * Accumulation over chunks is the caller's sequence of calls (or one call with chunk_tokens);
 * the token sums inside one call are reduced in a fixed order, so reruns are bitwise equal. */
int lora_backward(const lora_desc* d, const lora_ctx* c, int64_t T, const void* X,
                  const void* W_prep, const float* A, const float* B, const void* dY,
                  const float* H_save, const float* dora_m, const float* dora_n,
                  const void* Y_save, void* dX, float* dA, float* dB, float* dm, void* ws,
                  size_t ws_bytes, void* stream);

/* ---- grad prepare and AdamW over flat fp32 arenas -------------------------------------------*/
/* Workspace bytes for lora_grad_prepare over these groups. */
size_t lora_grad_prepare_workspace_size(int32_t n_groups, const lora_group* groups);

/* Pass 1 of the two-pass clip for each group: S_g = sum of squares of grads[offset, offset+n)
 * accumulated beyond float precision (exact float-float per-thread partials, summed in
 * float-float within a CTA and in double across CTAs; elements above 2^40 in magnitude go to a
 * double accumulator, so no finite gradient overflows), then
 *   status[g] = LORA_ERR_NONFINITE if any element is NaN or +-Inf, else LORA_OK;
 *   scale_norm[2g]   = c = gamma * max_norm / norm if max_norm > 0 and norm > max_norm, else gamma
 *   scale_norm[2g+1] = norm = gamma * sqrt(S_g)
 * d_scale_norm [2 * n_groups] double and d_status [n_groups] int32 are device outputs.
 * 1 <= n_groups <= LORA_MAX_GROUPS. Groups must not overlap. */
int lora_grad_prepare(const float* grads, int32_t n_groups, const lora_group* groups,
                      double* d_scale_norm, int32_t* d_status, void* ws, size_t ws_bytes,
                      void* stream);

/* Allocation-free lora_grad_prepare (the paper has no counterpart; this is a deployment aid).
 * For callers that cannot allocate device memory and so cannot supply a workspace: code that
 * runs under another framework's allocator which owns the whole device pool, code that must not
 * allocate after initialisation (allocation can stall or fail mid-training), and code that
 * enqueues work while some other component is capturing a CUDA graph, where a cudaMalloc would
 * break or poison the capture. Same arguments and results as lora_grad_prepare, minus the
 * workspace: the scratch is a fixed file-scope device array of LORA_NOALLOC_PREPARE_PARTIALS
 * doubles plus a counter (about 128 KB), which every GPU that loads the library holds until
 * process exit. The call allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 *   - Size limit: sum over groups of ceil(elements / 16384) must be at most
 *     LORA_NOALLOC_PREPARE_PARTIALS (one group: at most 268,435,456 elements); larger requests
 *     return LORA_ERR_UNSUPPORTED with nothing enqueued.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 *     that device current; make that first call before any stream capture on that device.
 *   - All calls share the one array: calls that overlap on the GPU (other streams, other host
 *     threads) race and give wrong results; order them on one stream. The array keeps the last
 *     call's contents; each call clears the counter it needs before use. */
#define LORA_NOALLOC_PREPARE_PARTIALS 16384
int lora_grad_prepare_noalloc(const float* grads, int32_t n_groups, const lora_group* groups,
                              double* d_scale_norm, int32_t* d_status, void* stream);

/* Pass 2 fused with the AdamW update, for every group whose device status is LORA_OK (groups
 * with another status are left untouched: params, moments and grads):
 *   g_hat = c g; m = b1 m + (1-b1) g_hat; v = b2 v + (1-b2) g_hat^2; k = step + 1;
 *   u = (m / (1 - b1^k)) / (sqrt(v / (1 - b2^k)) + eps)
 *   A:   p -= lr u + lr wd p      B: p -= lr plus_ratio u      MAG: p -= lr u
 * zero_grads != 0 also clears the group's gradients after reading them. The caller advances
 * each group's step (and re-evaluates lr) only for groups whose status was LORA_OK. */
int lora_adamw_step(float* params, float* grads, float* m, float* v, int32_t n_groups,
                    const lora_group* groups, const lora_adamw_hp* hp, const double* d_scale_norm,
                    const int32_t* d_status, int32_t zero_grads, void* stream);

/* ---- fused projections ----------------------------------------------------------------------*/
/* Projections that read one input (q/k/v, gate/up) run as one fused linear: one frozen product
 * over the stacked weight W_cat = [W_0; W_1; ...] ([sum out_k, in]) and one output
 * Y_cat [T, sum out_k] whose columns [off_k, off_k + out_k) (off_k = out_0 + ... + out_{k-1})
 * are projection k's, while every projection keeps its own adapter ("LoRA Training and Serving",
 * --lora-type: fused projections, and canonical adapters per q/k/v and gate/up projection):
 *   Y_k = X W_k^T + s' (Xd A_k^T) B_k^T,   dX = sum_k (dY_k W_k + s' (G_k A_k) * M),
 *   dA_k += s' G_k^T Xd,  dB_k += s' dY_k^T (Xd A_k^T),  G_k = dY_k B_k.
 * desc: in_dim, out_dim = sum out_k, the shared rank and scale, dtype LORA_BF16 or LORA_F32, no
 * DoRA; one dropout mask (desc.layer_id / proj_id) for all the projections;
 * 1 <= n_proj <= LORA_MAX_SLOTS. LORA_BF16: every out_k is a multiple of 256. LORA_F32:
 * n_proj * rank <= LORA_MAX_RANK (the group runs as one adapter of that rank whose up-projection
 * is block-diagonal). LORA_ERR_UNSUPPORTED otherwise. W_prep is lora_prepare_weight of W_cat
 * (desc above); the forward reads W (bf16) or W_prep (fp32), as lora_forward does.
 * H_save [T, n_proj * rank] fp32 holds Hs_k = s' Xd A_k^T in columns k rank .. k rank + rank - 1.
 * dX may be NULL. */
typedef struct lora_proj {
  const float* A;   /* [rank, in_dim] */
  const float* B;   /* [out_dim, rank] */
  float* dA;        /* [rank, in_dim], accumulated (+=) by lora_fused_backward */
  float* dB;        /* [out_dim, rank], accumulated (+=) */
  int64_t out_dim;  /* out_k */
} lora_proj;
size_t lora_fused_workspace_size(const lora_desc* d, int64_t T, int32_t n_proj,
                                 const lora_proj* projs);
int lora_fused_forward(const lora_desc* d, const lora_ctx* c, int64_t T, const void* X,
                       const void* W, const void* W_prep, int32_t n_proj, const lora_proj* projs,
                       void* Y, float* H_save, void* ws, size_t ws_bytes, void* stream);
int lora_fused_backward(const lora_desc* d, const lora_ctx* c, int64_t T, const void* X,
                        const void* W_prep, int32_t n_proj, const lora_proj* projs,
                        const void* dY, const float* H_save, void* dX, void* ws, size_t ws_bytes,
                        void* stream);

/* ---- adapter-state maintenance --------------------------------------------------------------*/
/* Snapshot, restore and retirement of adapter state over the groups' ranges
 * [offset, offset + n_a + n_b + n_mag) of the flat fp32 arenas ("4.3. Training Guide",
 * Validation early stopping: the best A/B are snapshotted, restored on exit, and the optimizer
 * is reset after the restore; "Multi-LoRA Training Example", a finished adapter is retired:
 * its slot cleared, its optimizer state and retained gradients zeroed, its partially
 * accumulated gradients discarded). All arrays are device fp32 with the arenas' layout and
 * 16-byte aligned; only the groups' ranges are read or written. Asynchronous on `stream`;
 * groups are checked as for lora_grad_prepare (LORA_ERR_INVALID / LORA_ERR_ALIGN before any
 * launch), a launch failure gives LORA_ERR_CUDA.
 *
 * lora_snapshot: snap = params.
 * lora_restore:  params = snap, m = v = 0, and grads = 0 when zero_grads != 0. The caller
 *                restarts each group's update count (lora_group.step = 0 on its next
 *                lora_adamw_step), which completes the optimizer reset.
 * lora_retire:   grads = m = v = 0, and params = 0 when clear_params != 0. The caller resets
 *                the slots' accumulated sample counts and update counts on the host. */
int lora_snapshot(const float* params, float* snap, int32_t n_groups, const lora_group* groups,
                  void* stream);
int lora_restore(float* params, const float* snap, float* grads, float* m, float* v,
                 int32_t n_groups, const lora_group* groups, int32_t zero_grads, void* stream);
int lora_retire(float* params, float* grads, float* m, float* v, int32_t n_groups,
                const lora_group* groups, int32_t clear_params, void* stream);

/* ---- slot-keyed multi-LoRA ------------------------------------------------------------------*/
/* Segments: segment k covers tokens [seg_start[k], seg_start[k+1]) (device int32 [n_seg + 1],
 * non-decreasing, within [0, T]) and uses slot seg_slot[k] (device int32 [n_seg]). Tokens in no
 * segment, or in a segment whose slot id is outside [0, n_slots), get no adapter (frozen output
 * only). `slots` is a host array of n_slots entries (1 <= n_slots <= LORA_MAX_SLOTS); desc.rank
 * is the largest slot rank and the row stride of H_save. desc.dora must be 0. */
size_t multi_lora_workspace_size(const lora_desc* d, int64_t T, int32_t n_seg, int32_t n_slots,
                                 const lora_slot* slots);

int multi_lora_forward(const lora_desc* d, const lora_ctx* c, int64_t T, const void* X,
                       const void* W, const void* W_prep, int32_t n_seg,
                       const int32_t* d_seg_start, const int32_t* d_seg_slot, int32_t n_slots,
                       const lora_slot* slots, void* Y, float* H_save, void* ws, size_t ws_bytes, void* stream);

/* dX may be NULL. Each slot's dA/dB accumulate that slot's tokens with weight 1; per-slot
 * 1/adapter_global_batch_size, clip and Adam are lora_grad_prepare / lora_adamw_step with one
 * group per ready slot. */
int multi_lora_backward(const lora_desc* d, const lora_ctx* c, int64_t T, const void* X,
                        const void* W_prep, int32_t n_seg, const int32_t* d_seg_start,
                        const int32_t* d_seg_slot, int32_t n_slots, const lora_slot* slots,
                        const void* dY, const float* H_save, void* dX, void* ws,
                        size_t ws_bytes, void* stream);

/* Routing plan. Every routed call over the same batch (T, segments, slots: the same token
 * routing for every projection and layer, "Multi-LoRA Training Example", Design: slot-keyed
 * page table, one routing per batch) needs the same token work tables: the row products' token
 * items, the token reductions' runs and the slot set of every 128-token tile. A plan holds them
 * in a caller-owned device buffer of multi_lora_plan_size(T, n_seg, n_slots) bytes (0 for bad
 * arguments), 16-byte aligned. multi_lora_plan_build fills it from the segment table (the same
 * rules as multi_lora_forward; three launches on `stream`); the *_planned calls take
 * (T, n_seg, plan) in place of the segment table, read the plan on their own stream and build
 * nothing, so any number of calls, on any streams ordered after the build, may share one plan.
 * A plan stays valid until the caller rewrites its buffer; its contents depend on
 * (T, n_seg, n_slots) and the segment table only, so a planned call passes the same T, n_seg and
 * n_slots as the build. Results are bit-identical to the unplanned calls. Errors: LORA_ERR_INVALID
 * (null pointers, n_seg < 1, n_slots outside 1..LORA_MAX_SLOTS), LORA_ERR_ALIGN,
 * LORA_ERR_WORKSPACE (plan_bytes too small), LORA_ERR_UNSUPPORTED (T above 2^31 - 257), then
 * the checks of multi_lora_forward / multi_lora_backward. */
size_t multi_lora_plan_size(int64_t T, int32_t n_seg, int32_t n_slots);
int multi_lora_plan_build(int64_t T, int32_t n_seg, const int32_t* d_seg_start,
                          const int32_t* d_seg_slot, int32_t n_slots, void* plan, size_t plan_bytes,
                          void* stream);
int multi_lora_forward_planned(const lora_desc* d, const lora_ctx* c, int64_t T, int32_t n_seg,
                               const void* plan, const void* X, const void* W, const void* W_prep,
                               int32_t n_slots, const lora_slot* slots, void* Y, float* H_save,
                               void* ws, size_t ws_bytes, void* stream);
int multi_lora_backward_planned(const lora_desc* d, const lora_ctx* c, int64_t T, int32_t n_seg,
                                const void* plan, const void* X, const void* W_prep,
                                int32_t n_slots, const lora_slot* slots, const void* dY,
                                const float* H_save, void* dX, void* ws, size_t ws_bytes,
                                void* stream);

/* ---- test hooks (not part of the timed path) ------------------------------------------------*/
/* Keep mask M [T, in_dim] as uint8 (1 = kept), exactly as the kernels regenerate it. */
/* Test hook: the per-row E4M3 quantisation of LORA_BF16_FP8 (see its definition) applied to a bf16
 * [rows, K] matrix: codes [rows, K] uint8 and scales [rows] fp32. K % 16 == 0, K <= 16384. */
int lora_quantize_e4m3(const void* src, int64_t rows, int64_t K, uint8_t* codes, float* scales,
                       void* stream);
int lora_dropout_mask(const lora_desc* d, const lora_ctx* c, int64_t T, uint8_t* d_mask,
                      void* stream);

/* Slot of every token (int32 [T], -1 = no adapter) under the segment rules above. */
int multi_lora_token_slots(int64_t T, int32_t n_seg, const int32_t* d_seg_start,
                           const int32_t* d_seg_slot, int32_t n_slots, int32_t* d_token_slot,
                           void* stream);

/* ---- instrumentation (benchmark and tests; not part of the method) -------------------------*/
/* Kernel classes for lora_profile_arm. */
#define LORA_PROF_NONE 0
#define LORA_PROF_FROZEN_FWD 1   /* frozen forward product with the fused up-projection */
#define LORA_PROF_FROZEN_DX 2    /* frozen dX product with the fused LoRA dX term */
#define LORA_PROF_SHRINK 3       /* Hs = s' Xd A^T */
#define LORA_PROF_G 4            /* Gs = s' dY' B */
#define LORA_PROF_RED_DB 5       /* dB token reduction */
#define LORA_PROF_RED_DA 6       /* dA token reduction */
#define LORA_PROF_PREPARE 7      /* grad-prepare pass 1 */
#define LORA_PROF_ADAMW 8        /* fused clip + AdamW */
#define LORA_PROF_RED 9          /* dB and dA token reductions in one launch */

/* Arm event brackets: the next n launches of `kernel_class` record start_events[i] before and
 * stop_events[i] after launch i on the launching stream (cudaEvent_t handles, caller-owned).
 * Re-arming replaces the previous set; n == 0 disarms. Under stream capture the records become
 * graph nodes and fire on every replay. Not thread-safe with concurrent arming. */
int lora_profile_arm(int32_t kernel_class, void* const* start_events, void* const* stop_events,
                     int32_t n);
/* How many armed brackets have been used so far. */
int32_t lora_profile_used(void);
/* Kernel launches enqueued by this library since it was loaded (all classes). */
uint64_t lora_launch_counter(void);
/* Text of the last CUDA error an entry point of this library reported as LORA_ERR_CUDA in the
 * calling thread ("no error" if none). */
const char* lora_last_cuda_error(void);
/* Error bits raised on the device by the tensor-core products when a pipeline wait ran out of
 * its bound (bit 0 loads, bit 1 MMA, bit 2 epilogue): the kernel then skipped its remaining
 * work, released its tensor memory and returned, so the output is invalid. Synchronous (reads
 * a device word of the current device); reset != 0 clears it. */
int lora_device_error(uint32_t* flags, int32_t reset);
/* Synchronises `stream`, then reports the device error word: LORA_ERR_TIMEOUT if any bit is set
 * (left set for lora_device_error), LORA_ERR_CUDA if the stream holds a CUDA error, else LORA_OK.
 * This is how a caller learns, after the fact, that an asynchronous call's outputs are invalid
 * because one of its kernels gave up waiting and returned early (no hang, the context stays
 * usable). The bound of each wait guards against a pipeline that can no longer make progress
 * ("4.3. Training Guide", Gradient clipping: a bad step is detected and rejected before any
 * state changes; here the same rule for a stalled kernel). */
int lora_device_check(void* stream);
/* Test hook: bound, in SM clock cycles, of the pipeline waits of the frozen-product kernels
 * (bf16 and E4M3) launched after this call; 0 restores the default (2^33 cycles, seconds).
 * Process-wide, not thread-safe with concurrent launches. A small bound makes a correct launch
 * give up: its error bits are set and its outputs are invalid. Waits that drain work already
 * issued (copies in flight, MMAs before the tensor memory is freed) keep the default bound, so
 * a kernel that gives up still leaves nothing running behind it. */
int lora_set_wait_limit(uint64_t cycles);

#ifdef __cplusplus
}
#endif

#endif /* LORA_GB300_H */
