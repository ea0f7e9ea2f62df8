/*
 * prism.h -- C ABI of the B300 (sm_103a) Prism block-sparse attention path.
 *
 * Prism: Dynamic Sparse Attention for Native 2K Joint Video-Audio Generation
 * Model Training (arXiv 2610.05416).  The pages state the method in the
 * Abstract and the Fig. 2 caption: the latent token grid is cut into
 * spatiotemporal macro-zones; each zone gets a block shape from the
 * directional variance of the video features and the norms of the
 * audio-to-video cross-attention output; tokens are regrouped so that every
 * block is contiguous; block-level (pooled) features give block scores; a
 * hybrid Top-k / Top-p rule picks key blocks per query block; block-sparse
 * attention runs over the picked blocks, forward and backward.
 *
 * Conventions shared by every entry point
 *   - All device pointers are owned by the caller.  The library never
 *     allocates device memory; it allocates only the host-side plan.
 *   - Every call is asynchronous on the caller's stream `stream`
 *     (a cudaStream_t passed as void*; NULL = legacy default stream) and
 *     returns once the work is enqueued.  Argument errors are detected on
 *     the host before anything is enqueued.
 *   - Token layout of model-side tensors (Q, K, V, dO, O, dQ, dK, dV):
 *     [B, N, H, d] row-major bf16, token n = (t * Hg + y) * W + x over the
 *     real grid (T, Hg, W).  a2v: [B, N, Ca] bf16.
 *   - Permuted ("block order") tensors Xp: [B, H, Np, d] row-major; slot
 *     s of head h belongs to block s / S.  Padding slots hold zeros.
 *   - bf16 values are passed as uint16_t bit patterns.
 *   - Device pointers must be 16-byte aligned; d must be a multiple of 8.
 *   - Return value: PRISM_OK (0) or a negative PRISM_ERR_* code.  Errors
 *     raised inside a kernel (a bounded wait that ran out, an index out of
 *     range) are recorded in the status word of the workspace and read
 *     with prism_device_status().
 */
#ifndef PRISM_H_
#define PRISM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PRISM_MAX_SHAPES 32
#define PRISM_MAX_CLASSES 3

enum {
  PRISM_OK = 0,
  PRISM_ERR_ARG = -1,            /* null pointer, bad size or inconsistent configuration */
  PRISM_ERR_ALIGN = -2,          /* a device pointer is not 16-byte aligned */
  PRISM_ERR_UNSUPPORTED = -3,    /* d, block size or menu outside what the kernels handle */
  PRISM_ERR_NO_ADMISSIBLE_SHAPE = -4, /* no menu shape tiles the macro-zone */
  PRISM_ERR_CUDA = -5,           /* a CUDA runtime call failed (launch, copy, attribute) */
  PRISM_ERR_DEVICE_TIMEOUT = -6, /* a device-side wait exceeded its bound; results are invalid */
  PRISM_ERR_DEVICE_BOUNDS = -7   /* a device-side index check failed; results are invalid */
};

/* Problem statement (Prism Abstract; Fig. 2 caption; Tables 7, 9, 10, 12). */
typedef struct prism_config {
  int B, H, d;            /* batch, heads, head dim (multiple of 8, <= 128)          */
  int T, Hg, W;           /* real latent grid (frames, height, width) in tokens     */
  int zT, zH, zW;         /* macro-zone extents; the grid is zero-padded up to      */
                          /* multiples of them                                      */
  int block_tokens;       /* S: tokens per block; every menu shape has bT*bH*bW==S  */
  int n_shapes;           /* menu size, 1..PRISM_MAX_SHAPES                         */
  int shapes[PRISM_MAX_SHAPES][3]; /* menu of (bT, bH, bW) block shapes            */
  int Ca;                 /* channels of the audio-to-video cross-attention output  */
  double alpha;           /* Eq. 7 exponent: b*_d proportional to g_d^-alpha        */
  double eps;             /* floor added to the guidance g_d                        */
  int per_head;           /* 1: shapes per head; 0: one shape per zone for all heads */
  int use_video;          /* 1: video variance guidance on (Table 12 ablates it)    */
  int use_audio;          /* 1: audio guidance on (Table 12 ablates it)             */
  int topk_floor;         /* Top-k: minimum number of key blocks per query block    */
  float topp;             /* Top-p: cumulative block weight that must be exceeded   */
  unsigned long long timeout_cycles; /* bound on any device wait; 0 = default (~2 s) */
  int attn_kernel;        /* 0: tensor-core (tcgen05) attention where supported
                             (S = 128, d = 128), CUDA-core kernels otherwise;
                             1: CUDA-core kernels always                         */
  int fault_inject;       /* 0 in normal use.  PRISM_FAULT_STARVE_LOADS (tests of
                             failure detection only): the producer warps of the
                             tensor-core attention kernels issue no loads, so the
                             first bounded wait of their consumers runs out; the
                             kernels free their tensor memory and return, and the
                             status word reads PRISM_ERR_DEVICE_TIMEOUT.  No copy
                             is in flight when they return.                       */
  int key_chunk_blocks;   /* key blocks per range of the tensor-core forward / dQ
                             kernels (prism_sizes_t.key_chunks): 0 = automatic
                             (ceil(nb / 900) equal ranges once a head has more
                             than 1024 key blocks, else one range); > 0 = ranges
                             of this many blocks (at most 64 ranges)              */
  double class_tau[PRISM_MAX_CLASSES - 1];
                          /* block-size classes (Table 10 caption: thresholds
                             tau_128 / tau_256; Table 11: classes C_64, C_128,
                             C_256).  The menu's distinct token counts are the
                             classes, ascending; each must be block_tokens / 2
                             (tensor-core plans only: two such blocks share one
                             tile), block_tokens, 2 block_tokens or
                             4 block_tokens (a block then spans 1, 2 or 4
                             consecutive tiles of block_tokens slots).
                             A zone of complexity c = V_z / mean V + a_bar
                             (V_z: its summed directional video variance, a_bar
                             its audio gate; each term only when that guidance is
                             on) takes class k = number of thresholds c is below;
                             thresholds descending, the first n_classes - 1 used.
                             A zone with padding takes no class smaller than a
                             tile. */
} prism_config_t;

#define PRISM_FAULT_STARVE_LOADS 1

/* Derived sizes of a plan. */
typedef struct prism_sizes {
  int Tp, Hp, Wp;         /* padded grid */
  int nzT, nzH, nzW;      /* zones per axis */
  int Z;                  /* zones = nzT * nzH * nzW */
  int nb;                 /* tiles per (b, h) = Np / S (S = block_tokens); one block
                             per tile for a single class of S tokens */
  int blocks_per_zone;    /* tiles per zone */
  long long N, Np;        /* real and padded tokens */
  int n_admissible;       /* menu shapes that tile the zone */
  int admissible[PRISM_MAX_SHAPES];
  long long max_pairs;    /* capacity needed for col_idx / row_idx: B*H*nb*nb */
  size_t ws_bytes;        /* workspace bytes needed by prism_block_select,
                             prism_sparse_attn_fwd and prism_sparse_attn_bwd */
  int tensor_core_fwd;    /* 1 when the forward attention runs on tcgen05 kernels */
  int tensor_core_bwd;    /* 1 when the backward attention runs on tcgen05 kernels */
  int key_chunks;         /* the tensor-core attention kernels split each head's
                             blocks into this many ranges of chunk_blocks and walk
                             them range by range (the forward and dQ kernels: key
                             blocks, for all query blocks of a head one range at a
                             time; the dK / dV kernel: query blocks, likewise), so
                             that the tiles in use fit in L2; partial results are
                             combined per block afterwards (their room is part of
                             ws_bytes).  1 = no split. */
  int chunk_blocks;       /* blocks per range (nb when key_chunks == 1) */
  int n_classes;          /* block-size classes of the menu */
  int class_tokens[PRISM_MAX_CLASSES]; /* their token counts, ascending */
  int multi_tile;         /* 1 when some block spans several tiles or shares one:
                             n_valid and the block lists then count tiles, and
                             the block means sit at a block's first slot */
  int slot_tokens;        /* granularity of the block table: block_tokens, or half
                             of it when the menu has a class of half a tile (two
                             such blocks share one tile; tensor-core plans only) */
  int nslots;             /* slots per (b, h) = Np / slot_tokens: the length of the
                             Qbar / Kbar / sel_tie rows (nb unless half_tile) */
  int half_tile;          /* 1 when the menu has a class of half a tile */
  size_t ws_csr_mask;     /* half_tile: workspace offset of the uint8 sub-tile masks
                             of the CSR entries (one per col_idx entry), written by
                             prism_block_select and read by the attention calls:
                             bit 2 qh + kh set = the query tile's half qh does NOT
                             attend the key tile's half kh (0: the whole pair) */
  size_t ws_csc_mask;     /* half_tile: likewise for the CSC entries (row_idx) */
  size_t ws_scores;       /* workspace offset of the block scores that
                             prism_block_select writes: the unscaled dots
                             Qbar_i . Kbar_j as double-float, fp32 hi
                             [B, H, nslots, nslots] followed by fp32 lo of the
                             same shape (read-only for callers; tests) */
} prism_sizes_t;

typedef struct prism_plan prism_plan_t;

/* Validate `cfg` and build a host plan.  Errors: PRISM_ERR_ARG (sizes,
 * thresholds not descending), PRISM_ERR_UNSUPPORTED (a menu token count that
 * is not 1, 2 or 4 times block_tokens, d, S), PRISM_ERR_NO_ADMISSIBLE_SHAPE
 * (a class with no menu shape that divides the zone, or a menu whose only
 * class is half a tile on a grid with padded zones: a padded zone needs a
 * class of at least a tile). */
int prism_plan_create(const prism_config_t* cfg, prism_plan_t** out);
void prism_plan_destroy(prism_plan_t* plan);
int prism_plan_query(const prism_plan_t* plan, prism_sizes_t* out);

/* Clear the device status word at the start of the workspace (async). */
int prism_ws_init(const prism_plan_t* plan, void* ws, void* stream);
/* Wait for `stream`, read the status word; returns PRISM_OK or the first
 * device error (PRISM_ERR_DEVICE_TIMEOUT / PRISM_ERR_DEVICE_BOUNDS). */
int prism_device_status(const prism_plan_t* plan, const void* ws, void* stream);
const char* prism_strerror(int code);

/* Kernel timing hooks.  The paper has no counterpart: this lets a caller
 * time each kernel of the path on its own with CUDA events, without a
 * profiler.  Slots:
 *   PRISM_TRACE_ATTN_FWD      the forward attention kernel
 *   PRISM_TRACE_BWD_PRE       rowsum(dO * O) (and -LSE log2 e) before the backward
 *   PRISM_TRACE_ATTN_DKDV     the dK/dV kernel (tensor cores) or the CUDA-core backward
 *   PRISM_TRACE_ATTN_DQ       the dQ kernel (tensor cores) or the dQ conversion
 *   PRISM_TRACE_ZONE_STATS    the zone-statistics kernel (prism_zone_stats,
 *                             prism_zone_stats_norms)
 *   PRISM_TRACE_PERMUTE_POOL  the permutation + pooling kernel
 *                             (prism_assign_and_permute, prism_permute_shapes)
 *   PRISM_TRACE_SCORE         the block-score kernel inside prism_block_select
 *   PRISM_TRACE_SELECT        every kernel of prism_block_select
 * events: NULL (clears every slot) or an array of 2 * PRISM_TRACE_SLOTS
 * cudaEvent_t handles, begin then end for each slot; a NULL handle leaves
 * that mark out.  The handles are copied into the plan and stay owned by the
 * caller, who must keep them alive while the plan records into them.  While
 * set, the calls above record the begin event on the call's stream just
 * before the slot's kernels are enqueued and the end event just after.  Not
 * synchronised with other threads using the same plan.
 * Errors: PRISM_ERR_ARG (plan NULL). */
#define PRISM_TRACE_SLOTS 8
enum {
  PRISM_TRACE_ATTN_FWD = 0,
  PRISM_TRACE_BWD_PRE = 1,
  PRISM_TRACE_ATTN_DKDV = 2,
  PRISM_TRACE_ATTN_DQ = 3,
  PRISM_TRACE_ZONE_STATS = 4,
  PRISM_TRACE_PERMUTE_POOL = 5,
  PRISM_TRACE_SCORE = 6,
  PRISM_TRACE_SELECT = 7
};
int prism_plan_set_trace_events(prism_plan_t* plan, void* const* events);

/* Step 1 -- zone statistics (Prism Abstract: video feature variance along
 * each axis and A2V feature norms; Table 9 caption: per-channel variance of
 * the value features r_{v,d}, audio coupling gate a_bar, audio directional
 * variance v_hat_{a,d}).
 *   V      [B, N, H, d] bf16     value features (post-projection)
 *   a2v    [B, N, Ca]  bf16      audio-to-video cross-attention output
 *   stats  [B, H, Z, 8] fp32 out (var_v_T, var_v_H, var_v_W,
 *                                 var_n_T, var_n_H, var_n_W, nbar, n_valid)
 * var_*_d: mean over the zone's lines along d (lines with >= 2 real tokens)
 * and over channels of the population variance on the line; n = ||a2v||_2. */
int prism_zone_stats(const prism_plan_t* plan, const uint16_t* V, const uint16_t* a2v,
                     float* stats, void* stream);

/* Step 1a -- the per-token norms of the audio-to-video (A2V) cross-attention
 * output, computed on the device (Prism Abstract: the zone signals use
 * "feature norms from the audio-to-video cross-attention").  Reading: one
 * attention head, softmax over the audio tokens, scale 1/sqrt(Ca):
 *   n_i = || softmax(Qa_i Ka^T / sqrt(Ca)) Va ||_2
 *   Qa  [B, N, Ca] bf16  the video tokens' cross-attention queries
 *   Ka  [B, Na, Ca] bf16 the audio tokens' keys
 *   Va  [B, Na, Ca] bf16 the audio tokens' values (may alias Ka); |Va| < 65504
 *   Na  audio tokens per batch entry, 1..256
 *   n   [B, N] fp32 out
 *   ws  workspace (status word: bounded waits, a value out of range)
 * Tensor cores (tcgen05) for Qa Ka^T and for P Va, with P split into two
 * fp16 terms; n carries a relative error of about 1e-6 (fp32 logits).
 * Errors: PRISM_ERR_UNSUPPORTED unless Ca is 64 or 128 and Na <= 256. */
int prism_a2v_norms(const prism_plan_t* plan, const uint16_t* Qa, const uint16_t* Ka,
                    const uint16_t* Va, int Na, float* n, void* ws, void* stream);

/* Step 1 with the A2V norms given (as prism_a2v_norms writes them) instead of
 * the A2V output: the same statistics as prism_zone_stats, with n [B, N] fp32
 * in place of ||a2v||. */
int prism_zone_stats_norms(const prism_plan_t* plan, const uint16_t* V, const float* n,
                           float* stats, void* stream);

/* Step 2 -- block shape per zone (Eq. 7 quantisation, Table 10 caption) and
 * the token permutation into zone / block order, fused with block pooling.
 *   stats      [B, H, Z, 8] fp32 in
 *   Q, K, V    [B, N, H, d] bf16 in
 *   shape_id   [B, H, Z] uint8 out: menu index of the zone's shape
 *   shape_tie  [B, H, Z] uint8 out: 1 when the best two costs differ < 1e-4
 *   perm       [B, H, Np] int32 out: slot -> token, -1 for a padding slot
 *   inv        [B, H, N]  int32 out: token -> slot
 *   Qp, Kp, Vp [B, H, Np, d] bf16 out
 *   Qbar, Qbar_lo, Kbar, Kbar_lo [B, H, nslots, d] fp32 out: mean over the
 *              block's real tokens as a double-float pair: Qbar is the fp32
 *              rounding of the mean and Qbar_lo the fp32 rounding of the rest
 *              (Qbar + Qbar_lo carries about 46 significant bits); 0 for a
 *              block without real tokens; a block that spans several tiles
 *              has its mean at its first slot and 0 at the slots that continue it
 *   n_valid    [B, H, nb] int32 out: real tokens in each tile (a block's real
 *              tokens come first in it, so they fill its first tiles) */
int prism_assign_and_permute(const prism_plan_t* plan, const float* stats,
                             const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                             uint8_t* shape_id, uint8_t* shape_tie, int32_t* perm,
                             int32_t* inv, uint16_t* Qp, uint16_t* Kp, uint16_t* Vp,
                             float* Qbar, float* Qbar_lo, float* Kbar, float* Kbar_lo,
                             int32_t* n_valid, void* stream);

/* Step 2 with the block shapes given by the caller instead of Eq. 7: the
 * fixed-shape and random-shape baselines of the block-shape ablation (Prism,
 * Table 9: "Random Shape", "Fixed 4^3", ...) run through the same
 * permutation, pooling, selection and attention kernels.
 *   shape_id   [B, H, Z] uint8 in: menu index of each zone's shape; it must
 *              be admissible for the zone (prism_sizes_t.admissible)
 *   ws         workspace (for the status word)
 *   other arguments as for prism_assign_and_permute.
 * A shape id that is not admissible is recorded as PRISM_ERR_DEVICE_BOUNDS
 * in the status word (read it with prism_device_status) and that zone uses
 * the first admissible shape instead, so every access stays in bounds. */
int prism_permute_shapes(const prism_plan_t* plan, const uint8_t* shape_id, const uint16_t* Q,
                         const uint16_t* K, const uint16_t* V, int32_t* perm, int32_t* inv,
                         uint16_t* Qp, uint16_t* Kp, uint16_t* Vp, float* Qbar, float* Qbar_lo,
                         float* Kbar, float* Kbar_lo, int32_t* n_valid, void* ws, void* stream);

/* Step 3+4 -- block scores Qbar Kbar^T / sqrt(d) and hybrid Top-k / Top-p
 * selection (Table 7 caption; Abstract: per-query sparsity), then the
 * block lists in both directions.
 *   shape_id    [B, H, Z] uint8 in: the zones' shapes (as step 2 wrote or was
 *               given them); with blocks that span several tiles
 *               (prism_sizes_t.multi_tile) the selection runs over blocks and
 *               every list below is over tiles: each tile of a query block
 *               lists every tile of every key block its block selected
 *   Qbar, Qbar_lo, Kbar, Kbar_lo [B, H, nslots, d] fp32 in (as written above)
 *   n_valid     [B, H, nb] int32 in
 *   row_ptr     [B*H*nb + 1] int32 out: CSR offsets over all (b, h, i)
 *   col_idx     [max_pairs] int32 out: key blocks of each query block, ascending
 *   col_ptr     [B*H*nb + 1] int32 out: CSC offsets over all (b, h, j)
 *   row_idx     [max_pairs] int32 out: query blocks of each key block, ascending
 *   sel_tie     [B, H, nslots] uint8 out: 1 where the decision sat within 1e-6
 *               of a boundary (score gap or cumulative mass), at a block's
 *               first slot
 *   ws          workspace of ws_bytes
 * Query blocks with no real token select nothing; candidates are the key
 * blocks with at least one real token. */
int prism_block_select(const prism_plan_t* plan, const uint8_t* shape_id, const float* Qbar,
                       const float* Qbar_lo, const float* Kbar, const float* Kbar_lo,
                       const int32_t* n_valid, int32_t* row_ptr, int32_t* col_idx,
                       int32_t* col_ptr, int32_t* row_idx, uint8_t* sel_tie, void* ws,
                       void* stream);

/* Step 5a -- block-sparse attention forward (Fig. 2 caption).
 * For every query block i and every key block j in its list, exact softmax
 * over the real tokens of the listed key blocks, scale `scale`.  With
 * prism_sizes_t.key_chunks > 1 the key blocks are walked in ranges and the
 * per-range partial results, kept in `ws`, are combined before the call's
 * last kernel writes Op and lse; prism_sparse_attn_bwd does the same for dQ,
 * dK and dV.  The results do not depend on the split beyond rounding.  With
 * blocks of half a tile (prism_sizes_t.half_tile) both calls read the
 * sub-tile masks that prism_block_select left in `ws` for these lists.
 *   Qp, Kp, Vp [B, H, Np, d] bf16 in; n_valid, row_ptr, col_idx as above
 *   Op  [B, H, Np, d] bf16 out (padding rows 0)
 *   lse [B, H, Np] fp32 out: natural-log log-sum-exp per row (padding 0) */
int prism_sparse_attn_fwd(const prism_plan_t* plan, const uint16_t* Qp, const uint16_t* Kp,
                          const uint16_t* Vp, const int32_t* n_valid, const int32_t* row_ptr,
                          const int32_t* col_idx, float scale, uint16_t* Op, float* lse,
                          void* ws, void* stream);

/* Gather a model-side tensor into block order: Xp[b,h,s] = X[b,perm[s],h]
 * (zeros where perm[s] < 0).  X [B, N, H, d] bf16 -> Xp [B, H, Np, d] bf16. */
int prism_permute(const prism_plan_t* plan, const int32_t* perm, const uint16_t* X,
                  uint16_t* Xp, void* stream);

/* Step 5b -- backward of step 5a (Prism trains through this attention; it
 * replaces video self-attention during training, Table 2 caption).  The
 * selection and the permutation are constants.
 *   dOp [B, H, Np, d] bf16 in (padding rows must be 0, as prism_permute writes)
 *   dQp, dKp, dVp [B, H, Np, d] bf16 out (padding rows 0) */
int prism_sparse_attn_bwd(const prism_plan_t* plan, const uint16_t* Qp, const uint16_t* Kp,
                          const uint16_t* Vp, const uint16_t* Op, const uint16_t* dOp,
                          const float* lse, const int32_t* n_valid, const int32_t* row_ptr,
                          const int32_t* col_idx, const int32_t* col_ptr,
                          const int32_t* row_idx, float scale, uint16_t* dQp, uint16_t* dKp,
                          uint16_t* dVp, void* ws, void* stream);

/* Backward without a workspace, for callers that cannot allocate device
 * memory when they run it (for example code confined to a memory pool it does
 * not own, or a runtime that forbids cudaMalloc / cudaFree after start-up).
 * The paper has no counterpart: this is a library convenience.  Arguments and
 * results are those of prism_sparse_attn_bwd minus ws.  The scratch lives in a
 * 32 MiB array inside the library, held on every GPU that loads the library
 * until the process exits.  With R = B*H*Np, the call needs
 *   256 + round_up(4*R, 256) + 4*R*X  <=  32 MiB   (33554432 bytes),
 * X = 1 on the tensor-core path (rowsum D, then LSE * log2 e) and X = d on the
 * CUDA-core path (D, then the fp32 dQ accumulator); larger problems return
 * PRISM_ERR_UNSUPPORTED before anything is enqueued.  The first call on a
 * device looks the array's address up and keeps it: make that first call
 * before any stream capture, and do not use the entry point across a
 * cudaDeviceReset of that device (the kept address belongs to the context
 * that was current at the first call).  All calls share the array: calls
 * whose kernels overlap on the GPU race and give wrong results.  Device-side
 * wait timeouts go to the array's status word, cleared at the start of each
 * call; read it with prism_noalloc_device_status.  Plans with blocks of half a
 * tile (prism_sizes_t.half_tile) return PRISM_ERR_UNSUPPORTED: their sub-tile
 * masks live in the workspace. */
int prism_sparse_attn_bwd_noalloc(const prism_plan_t* plan, const uint16_t* Qp,
                                  const uint16_t* Kp, const uint16_t* Vp, const uint16_t* Op,
                                  const uint16_t* dOp, const float* lse, const int32_t* n_valid,
                                  const int32_t* row_ptr, const int32_t* col_idx,
                                  const int32_t* col_ptr, const int32_t* row_idx, float scale,
                                  uint16_t* dQp, uint16_t* dKp, uint16_t* dVp, void* stream);

/* Status word of the workspace-free backward's scratch on the current device:
 * waits for `stream`, then returns PRISM_OK or the first device error of the
 * last prism_sparse_attn_bwd_noalloc call on this device
 * (PRISM_ERR_DEVICE_TIMEOUT / PRISM_ERR_DEVICE_BOUNDS).  The paper has no
 * counterpart.  Allocates nothing. */
int prism_noalloc_device_status(void* stream);

/* Inverse permutation: X[b,n,h] = Xp[b,h,inv[n]].  Xp [B, H, Np, d] bf16 ->
 * X [B, N, H, d] bf16. */
int prism_unpermute(const prism_plan_t* plan, const int32_t* inv, const uint16_t* Xp,
                    uint16_t* X, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PRISM_H_ */
