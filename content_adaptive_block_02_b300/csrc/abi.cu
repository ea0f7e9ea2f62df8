// The C ABI of libprism: plan validation, workspace layout and the entry
// points declared in include/prism.h.  Every entry point checks its
// arguments on the host, then enqueues kernels on the caller's stream.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "prism_internal.cuh"

using prism::Plan;

struct prism_plan {
  Plan p;
  cudaEvent_t trace[2 * PRISM_TRACE_SLOTS];  // optional timing marks, caller-owned
};

namespace prism {
cudaError_t launch_bwd_pre(const Plan& p, const uint16_t* Op, const uint16_t* dOp,
                           const float* lse, float* D, float* nlse2, float* dQacc,
                           cudaStream_t st);
cudaError_t launch_attn_fwd_simt(const Plan& p, const uint16_t* Qp, const uint16_t* Kp,
                                 const uint16_t* Vp, const int32_t* n_valid,
                                 const int32_t* row_ptr, const int32_t* col_idx, float scale,
                                 uint16_t* Op, float* lse, cudaStream_t st);
cudaError_t launch_attn_bwd_simt(const Plan& p, const uint16_t* Qp, const uint16_t* Kp,
                                 const uint16_t* Vp, const uint16_t* dOp, const float* lse,
                                 const float* D, const int32_t* n_valid,
                                 const int32_t* col_ptr, const int32_t* row_idx, float scale,
                                 float* dQacc, uint16_t* dKp, uint16_t* dVp, cudaStream_t st);
cudaError_t launch_attn_fwd_tc(const Plan& p, const uint16_t* Qp, const uint16_t* Kp,
                               const uint16_t* Vp, const int32_t* n_valid, const int32_t* row_ptr,
                               const int32_t* col_idx, float scale, uint16_t* Op, float* lse,
                               uint8_t* ws, cudaStream_t st);
cudaError_t launch_attn_dkdv_tc(const Plan& p, const uint16_t* Qp, const uint16_t* Kp,
                                const uint16_t* Vp, const uint16_t* dOp, const float* nlse2,
                                const float* D, const int32_t* n_valid, const int32_t* col_ptr,
                                const int32_t* row_idx, float scale, uint16_t* dKp, uint16_t* dVp,
                                uint8_t* ws, uint16_t* dkvpart, cudaStream_t st);
cudaError_t launch_fwd_combine(const Plan& p, const int32_t* row_ptr, const int32_t* col_idx,
                               const int32_t* n_valid, const uint8_t* ws, uint16_t* Op, float* lse,
                               cudaStream_t st);
cudaError_t launch_sum_combine(const Plan& p, const int32_t* ptr, const int32_t* idx,
                               const uint16_t* part, uint16_t* out, cudaStream_t st);
cudaError_t launch_attn_dq_tc(const Plan& p, const uint16_t* Qp, const uint16_t* Kp,
                              const uint16_t* Vp, const uint16_t* dOp, const float* lse,
                              const float* D, const int32_t* n_valid, const int32_t* row_ptr,
                              const int32_t* col_idx, float scale, uint16_t* dQp, uint8_t* ws,
                              uint16_t* dqpart, cudaStream_t st);
}  // namespace prism

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

inline int ilog2_exact(int v) {
  int r = 0;
  while ((1 << r) < v) ++r;
  return (1 << r) == v ? r : -1;
}

#define PRISM_CHECK_PTR(p)                 \
  do {                                     \
    if ((p) == nullptr) return PRISM_ERR_ARG; \
    if (!aligned16(p)) return PRISM_ERR_ALIGN; \
  } while (0)

#define PRISM_CUDA(call)                      \
  do {                                        \
    if ((call) != cudaSuccess) return PRISM_ERR_CUDA; \
  } while (0)

// Record the begin (end = 0) or end (end = 1) mark of a trace slot, if set.
inline cudaError_t trace_mark(const prism_plan* plan, int slot, int end, cudaStream_t st) {
  cudaEvent_t e = plan->trace[2 * slot + end];
  return e == nullptr ? cudaSuccess : cudaEventRecord(e, st);
}

#define PRISM_TRACED(slot, call)                            \
  do {                                                      \
    PRISM_CUDA(trace_mark(plan, (slot), 0, st));            \
    PRISM_CUDA(call);                                       \
    PRISM_CUDA(trace_mark(plan, (slot), 1, st));            \
  } while (0)

}  // namespace

extern "C" {

const char* prism_strerror(int code) {
  switch (code) {
    case PRISM_OK: return "ok";
    case PRISM_ERR_ARG: return "invalid argument";
    case PRISM_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case PRISM_ERR_UNSUPPORTED: return "configuration not supported by the kernels";
    case PRISM_ERR_NO_ADMISSIBLE_SHAPE: return "no menu shape tiles the macro-zone";
    case PRISM_ERR_CUDA: return "CUDA runtime error";
    case PRISM_ERR_DEVICE_TIMEOUT: return "a device-side wait exceeded its bound";
    case PRISM_ERR_DEVICE_BOUNDS: return "a device-side index check failed";
    default: return "unknown error";
  }
}

int prism_plan_create(const prism_config_t* cfg, prism_plan_t** out) {
  if (cfg == nullptr || out == nullptr) return PRISM_ERR_ARG;
  *out = nullptr;
  const prism_config_t& c = *cfg;
  if (c.B < 1 || c.H < 1 || c.d < 1 || c.T < 1 || c.Hg < 1 || c.W < 1 || c.zT < 1 ||
      c.zH < 1 || c.zW < 1 || c.block_tokens < 1 || c.Ca < 1 || c.topk_floor < 0 ||
      !(c.topp >= 0.f) || c.n_shapes < 1 || c.n_shapes > PRISM_MAX_SHAPES ||
      !(c.alpha == c.alpha) || !(c.eps >= 0.0) ||
      (c.fault_inject != 0 && c.fault_inject != PRISM_FAULT_STARVE_LOADS) ||
      c.key_chunk_blocks < 0)
    return PRISM_ERR_ARG;
  if (c.d % 32 != 0 || c.d > 128) return PRISM_ERR_UNSUPPORTED;
  const int lS = ilog2_exact(c.block_tokens);
  if (lS < 2 || c.block_tokens > 128) return PRISM_ERR_UNSUPPORTED;
  if (c.d * c.block_tokens > 16384) return PRISM_ERR_UNSUPPORTED;
  // block-size classes: the menu's token counts, each 1, 2 or 4 tiles
  int classes[PRISM_MAX_CLASSES + 1];
  int n_classes = 0;
  for (int k = 0; k < c.n_shapes; ++k) {
    const int* s = c.shapes[k];
    if (s[0] < 1 || s[1] < 1 || s[2] < 1) return PRISM_ERR_ARG;
    const int t = s[0] * s[1] * s[2];
    if (2 * t != c.block_tokens && t != c.block_tokens && t != 2 * c.block_tokens &&
        t != 4 * c.block_tokens)
      return PRISM_ERR_UNSUPPORTED;
    bool seen = false;
    for (int q = 0; q < n_classes; ++q) seen |= classes[q] == t;
    if (!seen) {
      if (n_classes == PRISM_MAX_CLASSES) return PRISM_ERR_UNSUPPORTED;
      classes[n_classes++] = t;
    }
  }
  for (int a = 1; a < n_classes; ++a)  // ascending
    for (int q = a; q > 0 && classes[q - 1] > classes[q]; --q) {
      const int tmp = classes[q];
      classes[q] = classes[q - 1];
      classes[q - 1] = tmp;
    }
  for (int q = 1; q + 1 < n_classes; ++q)
    if (!(c.class_tau[q - 1] > c.class_tau[q])) return PRISM_ERR_ARG;  // descending
  for (int q = 0; q + 1 < n_classes; ++q)
    if (!(c.class_tau[q] == c.class_tau[q])) return PRISM_ERR_ARG;
  const long long vol = static_cast<long long>(c.zT) * c.zH * c.zW;
  if (vol > 3072) return PRISM_ERR_UNSUPPORTED;
  Plan p;
  memset(&p, 0, sizeof(p));
  p.cfg = c;
  prism_sizes_t& z = p.sz;
  z.nzT = (c.T + c.zT - 1) / c.zT;
  z.nzH = (c.Hg + c.zH - 1) / c.zH;
  z.nzW = (c.W + c.zW - 1) / c.zW;
  z.Tp = z.nzT * c.zT;
  z.Hp = z.nzH * c.zH;
  z.Wp = z.nzW * c.zW;
  z.Z = z.nzT * z.nzH * z.nzW;
  z.N = static_cast<long long>(c.T) * c.Hg * c.W;
  z.Np = static_cast<long long>(z.Tp) * z.Hp * z.Wp;
  for (int k = 0; k < c.n_shapes; ++k) {
    const int* s = c.shapes[k];
    if (c.zT % s[0] == 0 && c.zH % s[1] == 0 && c.zW % s[2] == 0)
      z.admissible[z.n_admissible++] = k;
  }
  if (z.n_admissible == 0) return PRISM_ERR_NO_ADMISSIBLE_SHAPE;
  z.n_classes = n_classes;
  for (int q = 0; q < n_classes; ++q) {
    z.class_tokens[q] = classes[q];
    bool any = false;
    for (int a = 0; a < z.n_admissible; ++a) {
      const int* s = c.shapes[z.admissible[a]];
      any |= s[0] * s[1] * s[2] == classes[q];
    }
    if (!any) return PRISM_ERR_NO_ADMISSIBLE_SHAPE;
  }
  z.half_tile = 2 * classes[0] == c.block_tokens ? 1 : 0;
  // a zone with padding cannot take the half-tile class (both halves of a
  // shared tile must be real): it needs a class of at least a tile
  if (z.half_tile && n_classes == 1 && (z.Tp != c.T || z.Hp != c.Hg || z.Wp != c.W))
    return PRISM_ERR_NO_ADMISSIBLE_SHAPE;
  z.multi_tile = (classes[n_classes - 1] > c.block_tokens || z.half_tile) ? 1 : 0;
  z.slot_tokens = z.half_tile ? c.block_tokens / 2 : c.block_tokens;
  z.blocks_per_zone = static_cast<int>(vol / c.block_tokens);
  const long long nb = z.Np / c.block_tokens;
  if (nb > 8192 || z.Np >= (1LL << 31) || z.N >= (1LL << 31)) return PRISM_ERR_UNSUPPORTED;
  z.nb = static_cast<int>(nb);
  z.nslots = static_cast<int>(z.Np / z.slot_tokens);
  const long long rows = static_cast<long long>(c.B) * c.H * nb;
  const long long srows = static_cast<long long>(c.B) * c.H * z.nslots;  // selection rows
  z.max_pairs = rows * nb;
  if (z.max_pairs >= (1LL << 31) || srows * z.nslots >= (1LL << 31)) return PRISM_ERR_UNSUPPORTED;
  {
    const bool tc_shape = c.block_tokens == 128 && c.d == 128 && c.attn_kernel == 0;
    z.tensor_core_fwd = tc_shape ? 1 : 0;
    z.tensor_core_bwd = tc_shape ? 1 : 0;
  }
  if (z.half_tile && !z.tensor_core_fwd) return PRISM_ERR_UNSUPPORTED;
  if (c.attn_kernel < 0 || c.attn_kernel > 1) return PRISM_ERR_ARG;
  for (int k = 0; k < PRISM_MAX_SHAPES; ++k)
    for (int a = 0; a < 3; ++a) {
      const int e = k < c.n_shapes ? c.shapes[k][a] : 1;
      const int l = ilog2_exact(e);
      p.log2_ext[k][a] = l >= 0 ? static_cast<double>(l) : log2(static_cast<double>(e));
    }
  p.log2_S = static_cast<double>(lS);
  // workspace layout (the selection runs over slots: tiles, or half tiles)
  const int nwords = (z.nb + 31) / 32;
  const int swords = (z.nslots + 31) / 32;
  size_t off = 256;
  p.off_rowcnt = off; off = align256(off + srows * 4);
  p.off_colcnt = off; off = align256(off + srows * 4);
  p.off_amb = off; off = align256(off + srows * 4);
  p.off_bitmask = off; off = align256(off + srows * swords * 4);
  p.off_scores = off; off = align256(off + 2 * srows * z.nslots * 4);
  p.off_D = off; off = align256(off + static_cast<size_t>(c.B) * c.H * z.Np * 4);
  p.off_lse2 = off; off = align256(off + static_cast<size_t>(c.B) * c.H * z.Np * 4);
  p.off_dq = off;
  if (!z.tensor_core_bwd) off = align256(off + static_cast<size_t>(c.B) * c.H * z.Np * c.d * 4);
  // multi-tile blocks: real tokens per block at its first tile, first tile of
  // every tile's block, and the tile-level selection bitmask
  p.off_nsel = p.off_bstart = p.off_tbitmask = off;
  z.ws_csr_mask = z.ws_csc_mask = 0;
  if (z.multi_tile) {
    p.off_nsel = off; off = align256(off + srows * 4);
    p.off_bstart = off; off = align256(off + srows * 4);
    p.off_tbitmask = off; off = align256(off + rows * nwords * 4);
  }
  if (z.half_tile) {
    // sub-tile masks of the tile lists (one byte per CSR / CSC entry)
    z.ws_csr_mask = off; off = align256(off + static_cast<size_t>(z.max_pairs));
    z.ws_csc_mask = off; off = align256(off + static_cast<size_t>(z.max_pairs));
  }
  // once a head has more than 1024 key blocks, equal key ranges of at most
  // 900 blocks (56 MB of K and V per head: a range of the head stays in L2);
  // the partial results are capped at 32 GB
  z.key_chunks = 1;
  const int kcb = c.key_chunk_blocks > 0
                      ? c.key_chunk_blocks
                      : (z.nb > 1024 ? (z.nb + (z.nb + 899) / 900 - 1) / ((z.nb + 899) / 900) : z.nb);
  if (z.tensor_core_fwd && kcb < z.nb) {
    long long C = (z.nb + kcb - 1) / kcb;
    if (C > 64) C = 64;
    const long long per = static_cast<long long>(rows) * (2 * c.block_tokens * c.d * 2 +
                                                          c.block_tokens * 8);
    const long long cap = (32LL << 30) / per;
    if (C > cap) C = cap < 1 ? 1 : cap;
    z.key_chunks = static_cast<int>(C);
  }
  z.chunk_blocks = (z.nb + z.key_chunks - 1) / z.key_chunks;
  p.off_part = off;
  p.off_ml = off;
  if (z.key_chunks > 1) {
    // two bf16 tiles per (block, range): dK and dV partials (O and dQ use the first)
    off = align256(off + 2 * static_cast<size_t>(rows) * z.key_chunks * c.block_tokens * c.d * 2);
    p.off_ml = off;
    off = align256(off + static_cast<size_t>(rows) * z.key_chunks * c.block_tokens * 8);
  }
  // digits and exponents of the block means for the tensor-core scores
  p.off_digits = off;
  off = align256(off + score_digit_bytes(p));
  z.ws_scores = p.off_scores;
  z.ws_bytes = off;
  prism_plan* h = static_cast<prism_plan*>(malloc(sizeof(prism_plan)));
  if (h == nullptr) return PRISM_ERR_ARG;
  h->p = p;
  for (int i = 0; i < 2 * PRISM_TRACE_SLOTS; ++i) h->trace[i] = nullptr;
  *out = h;
  return PRISM_OK;
}

void prism_plan_destroy(prism_plan_t* plan) { free(plan); }

int prism_plan_query(const prism_plan_t* plan, prism_sizes_t* out) {
  if (plan == nullptr || out == nullptr) return PRISM_ERR_ARG;
  *out = plan->p.sz;
  return PRISM_OK;
}

int prism_ws_init(const prism_plan_t* plan, void* ws, void* stream) {
  if (plan == nullptr) return PRISM_ERR_ARG;
  PRISM_CHECK_PTR(ws);
  PRISM_CUDA(cudaMemsetAsync(ws, 0, 256, static_cast<cudaStream_t>(stream)));
  return PRISM_OK;
}

int prism_device_status(const prism_plan_t* plan, const void* ws, void* stream) {
  if (plan == nullptr) return PRISM_ERR_ARG;
  PRISM_CHECK_PTR(ws);
  uint32_t word = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PRISM_CUDA(cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, st));
  PRISM_CUDA(cudaStreamSynchronize(st));
  if (word == prism::DEV_ERR_TIMEOUT) return PRISM_ERR_DEVICE_TIMEOUT;
  if (word != 0) return PRISM_ERR_DEVICE_BOUNDS;
  return PRISM_OK;
}

int prism_zone_stats(const prism_plan_t* plan, const uint16_t* V, const uint16_t* a2v,
                     float* stats, void* stream) {
  if (plan == nullptr) return PRISM_ERR_ARG;
  PRISM_CHECK_PTR(V);
  PRISM_CHECK_PTR(a2v);
  PRISM_CHECK_PTR(stats);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PRISM_TRACED(PRISM_TRACE_ZONE_STATS,
               prism::launch_zone_stats(plan->p, V, a2v, nullptr, stats, st));
  return PRISM_OK;
}

int prism_a2v_norms(const prism_plan_t* plan, const uint16_t* Qa, const uint16_t* Ka,
                    const uint16_t* Va, int Na, float* n, void* ws, void* stream) {
  if (plan == nullptr || Na < 1) return PRISM_ERR_ARG;
  PRISM_CHECK_PTR(Qa); PRISM_CHECK_PTR(Ka); PRISM_CHECK_PTR(Va);
  PRISM_CHECK_PTR(n); PRISM_CHECK_PTR(ws);
  const prism_config_t& c = plan->p.cfg;
  if (c.Ca % 64 != 0 || c.Ca > 128 || Na > 256) return PRISM_ERR_UNSUPPORTED;
  PRISM_CUDA(prism::launch_a2v_norms(plan->p, Qa, Ka, Va, Na, n, static_cast<uint8_t*>(ws),
                                     static_cast<cudaStream_t>(stream)));
  return PRISM_OK;
}

int prism_zone_stats_norms(const prism_plan_t* plan, const uint16_t* V, const float* n,
                           float* stats, void* stream) {
  if (plan == nullptr) return PRISM_ERR_ARG;
  PRISM_CHECK_PTR(V);
  PRISM_CHECK_PTR(n);
  PRISM_CHECK_PTR(stats);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PRISM_TRACED(PRISM_TRACE_ZONE_STATS,
               prism::launch_zone_stats(plan->p, V, nullptr, n, stats, st));
  return PRISM_OK;
}

int prism_assign_and_permute(const prism_plan_t* plan, const float* stats, const uint16_t* Q,
                             const uint16_t* K, const uint16_t* V, uint8_t* shape_id,
                             uint8_t* shape_tie, int32_t* perm, int32_t* inv, uint16_t* Qp,
                             uint16_t* Kp, uint16_t* Vp, float* Qbar, float* Qbar_lo,
                             float* Kbar, float* Kbar_lo, int32_t* n_valid, void* stream) {
  if (plan == nullptr) return PRISM_ERR_ARG;
  PRISM_CHECK_PTR(stats);
  PRISM_CHECK_PTR(Q); PRISM_CHECK_PTR(K); PRISM_CHECK_PTR(V);
  PRISM_CHECK_PTR(shape_id); PRISM_CHECK_PTR(shape_tie);
  PRISM_CHECK_PTR(perm); PRISM_CHECK_PTR(inv);
  PRISM_CHECK_PTR(Qp); PRISM_CHECK_PTR(Kp); PRISM_CHECK_PTR(Vp);
  PRISM_CHECK_PTR(Qbar); PRISM_CHECK_PTR(Qbar_lo);
  PRISM_CHECK_PTR(Kbar); PRISM_CHECK_PTR(Kbar_lo);
  PRISM_CHECK_PTR(n_valid);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PRISM_CUDA(prism::launch_assign(plan->p, stats, shape_id, shape_tie, st));
  PRISM_TRACED(PRISM_TRACE_PERMUTE_POOL,
               prism::launch_permute_pool(plan->p, shape_id, Q, K, V, perm, inv, Qp, Kp, Vp,
                                          Qbar, Qbar_lo, Kbar, Kbar_lo, n_valid, nullptr, st));
  return PRISM_OK;
}

int prism_permute_shapes(const prism_plan_t* plan, const uint8_t* shape_id, const uint16_t* Q,
                         const uint16_t* K, const uint16_t* V, int32_t* perm, int32_t* inv,
                         uint16_t* Qp, uint16_t* Kp, uint16_t* Vp, float* Qbar, float* Qbar_lo,
                         float* Kbar, float* Kbar_lo, int32_t* n_valid, void* ws, void* stream) {
  if (plan == nullptr) return PRISM_ERR_ARG;
  PRISM_CHECK_PTR(Q); PRISM_CHECK_PTR(K); PRISM_CHECK_PTR(V);
  PRISM_CHECK_PTR(shape_id);
  PRISM_CHECK_PTR(perm); PRISM_CHECK_PTR(inv);
  PRISM_CHECK_PTR(Qp); PRISM_CHECK_PTR(Kp); PRISM_CHECK_PTR(Vp);
  PRISM_CHECK_PTR(Qbar); PRISM_CHECK_PTR(Qbar_lo);
  PRISM_CHECK_PTR(Kbar); PRISM_CHECK_PTR(Kbar_lo);
  PRISM_CHECK_PTR(n_valid); PRISM_CHECK_PTR(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PRISM_TRACED(PRISM_TRACE_PERMUTE_POOL,
               prism::launch_permute_pool(plan->p, shape_id, Q, K, V, perm, inv, Qp, Kp, Vp,
                                          Qbar, Qbar_lo, Kbar, Kbar_lo, n_valid,
                                          static_cast<uint32_t*>(ws), st));
  return PRISM_OK;
}

int prism_block_select(const prism_plan_t* plan, const uint8_t* shape_id, const float* Qbar,
                       const float* Qbar_lo, const float* Kbar, const float* Kbar_lo,
                       const int32_t* n_valid, int32_t* row_ptr, int32_t* col_idx,
                       int32_t* col_ptr, int32_t* row_idx, uint8_t* sel_tie, void* ws,
                       void* stream) {
  if (plan == nullptr) return PRISM_ERR_ARG;
  PRISM_CHECK_PTR(shape_id);
  PRISM_CHECK_PTR(Qbar); PRISM_CHECK_PTR(Qbar_lo);
  PRISM_CHECK_PTR(Kbar); PRISM_CHECK_PTR(Kbar_lo);
  PRISM_CHECK_PTR(n_valid);
  PRISM_CHECK_PTR(row_ptr); PRISM_CHECK_PTR(col_idx);
  PRISM_CHECK_PTR(col_ptr); PRISM_CHECK_PTR(row_idx);
  PRISM_CHECK_PTR(sel_tie); PRISM_CHECK_PTR(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PRISM_TRACED(PRISM_TRACE_SELECT,
               prism::launch_select(plan->p, shape_id, Qbar, Qbar_lo, Kbar, Kbar_lo, n_valid,
                                    sel_tie, row_ptr, col_idx, col_ptr, row_idx,
                                    static_cast<uint8_t*>(ws), st,
                                    plan->trace[2 * PRISM_TRACE_SCORE],
                                    plan->trace[2 * PRISM_TRACE_SCORE + 1]));
  return PRISM_OK;
}

int prism_sparse_attn_fwd(const prism_plan_t* plan, const uint16_t* Qp, const uint16_t* Kp,
                          const uint16_t* Vp, const int32_t* n_valid, const int32_t* row_ptr,
                          const int32_t* col_idx, float scale, uint16_t* Op, float* lse,
                          void* ws, void* stream) {
  if (plan == nullptr || !(scale > 0.f)) return PRISM_ERR_ARG;
  PRISM_CHECK_PTR(Qp); PRISM_CHECK_PTR(Kp); PRISM_CHECK_PTR(Vp);
  PRISM_CHECK_PTR(n_valid); PRISM_CHECK_PTR(row_ptr); PRISM_CHECK_PTR(col_idx);
  PRISM_CHECK_PTR(Op); PRISM_CHECK_PTR(lse); PRISM_CHECK_PTR(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Plan& p = plan->p;
  if (p.sz.tensor_core_fwd) {
    PRISM_TRACED(PRISM_TRACE_ATTN_FWD,
                 prism::launch_attn_fwd_tc(p, Qp, Kp, Vp, n_valid, row_ptr, col_idx, scale, Op,
                                           lse, static_cast<uint8_t*>(ws), st));
    if (p.sz.key_chunks > 1)
      PRISM_CUDA(prism::launch_fwd_combine(p, row_ptr, col_idx, n_valid,
                                           static_cast<const uint8_t*>(ws), Op, lse, st));
  } else {
    PRISM_TRACED(PRISM_TRACE_ATTN_FWD,
                 prism::launch_attn_fwd_simt(p, Qp, Kp, Vp, n_valid, row_ptr, col_idx, scale, Op,
                                             lse, st));
  }
  return PRISM_OK;
}

int prism_permute(const prism_plan_t* plan, const int32_t* perm, const uint16_t* X, uint16_t* Xp,
                  void* stream) {
  if (plan == nullptr) return PRISM_ERR_ARG;
  PRISM_CHECK_PTR(perm); PRISM_CHECK_PTR(X); PRISM_CHECK_PTR(Xp);
  PRISM_CUDA(prism::launch_permute(plan->p, perm, X, Xp, static_cast<cudaStream_t>(stream)));
  return PRISM_OK;
}

int prism_sparse_attn_bwd(const prism_plan_t* plan, const uint16_t* Qp, const uint16_t* Kp,
                          const uint16_t* Vp, const uint16_t* Op, const uint16_t* dOp,
                          const float* lse, const int32_t* n_valid, const int32_t* row_ptr,
                          const int32_t* col_idx, const int32_t* col_ptr, const int32_t* row_idx,
                          float scale, uint16_t* dQp, uint16_t* dKp, uint16_t* dVp, void* ws,
                          void* stream) {
  if (plan == nullptr || !(scale > 0.f)) return PRISM_ERR_ARG;
  PRISM_CHECK_PTR(Qp); PRISM_CHECK_PTR(Kp); PRISM_CHECK_PTR(Vp);
  PRISM_CHECK_PTR(Op); PRISM_CHECK_PTR(dOp); PRISM_CHECK_PTR(lse);
  PRISM_CHECK_PTR(n_valid); PRISM_CHECK_PTR(row_ptr); PRISM_CHECK_PTR(col_idx);
  PRISM_CHECK_PTR(col_ptr); PRISM_CHECK_PTR(row_idx);
  PRISM_CHECK_PTR(dQp); PRISM_CHECK_PTR(dKp); PRISM_CHECK_PTR(dVp); PRISM_CHECK_PTR(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Plan& p = plan->p;
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* D = reinterpret_cast<float*>(w + p.off_D);
  if (p.sz.tensor_core_bwd) {
    // dK, dV over the key blocks' lists; dQ over the query blocks' lists
    float* lse2 = reinterpret_cast<float*>(w + p.off_lse2);
    PRISM_TRACED(PRISM_TRACE_BWD_PRE,
                 prism::launch_bwd_pre(p, Op, dOp, lse, D, lse2, nullptr, st));
    const bool ranges = p.sz.key_chunks > 1;
    uint16_t* part = reinterpret_cast<uint16_t*>(w + p.off_part);
    PRISM_TRACED(PRISM_TRACE_ATTN_DKDV,
                 prism::launch_attn_dkdv_tc(p, Qp, Kp, Vp, dOp, lse2, D, n_valid, col_ptr,
                                            row_idx, scale, dKp, dVp, w, ranges ? part : nullptr,
                                            st));
    if (ranges) {
      // dK partials first, then dV partials (one tile per key block and range)
      const size_t tiles = static_cast<size_t>(p.cfg.B) * p.cfg.H * p.sz.nb * p.sz.key_chunks;
      PRISM_CUDA(prism::launch_sum_combine(p, col_ptr, row_idx, part, dKp, st));
      PRISM_CUDA(prism::launch_sum_combine(p, col_ptr, row_idx, part + tiles * 128 * 128, dVp,
                                           st));
    }
    PRISM_TRACED(PRISM_TRACE_ATTN_DQ,
                 prism::launch_attn_dq_tc(
                     p, Qp, Kp, Vp, dOp, lse, D, n_valid, row_ptr, col_idx, scale, dQp, w,
                     ranges ? part : nullptr, st));
    if (ranges) PRISM_CUDA(prism::launch_sum_combine(p, row_ptr, col_idx, part, dQp, st));
  } else {
    float* dq = reinterpret_cast<float*>(w + p.off_dq);
    PRISM_TRACED(PRISM_TRACE_BWD_PRE,
                 prism::launch_bwd_pre(p, Op, dOp, lse, D, nullptr, dq, st));
    PRISM_TRACED(PRISM_TRACE_ATTN_DKDV,
                 prism::launch_attn_bwd_simt(p, Qp, Kp, Vp, dOp, lse, D, n_valid, col_ptr,
                                             row_idx, scale, dq, dKp, dVp, st));
    // dQ in block order, bf16, scaled
    PRISM_TRACED(PRISM_TRACE_ATTN_DQ, prism::launch_dq_convert(p, dq, scale, dQp, st));
  }
  return PRISM_OK;
}

int prism_plan_set_trace_events(prism_plan_t* plan, void* const* events) {
  if (plan == nullptr) return PRISM_ERR_ARG;
  for (int i = 0; i < 2 * PRISM_TRACE_SLOTS; ++i)
    plan->trace[i] = events == nullptr ? nullptr : static_cast<cudaEvent_t>(events[i]);
  return PRISM_OK;
}

int prism_unpermute(const prism_plan_t* plan, const int32_t* inv, const uint16_t* Xp, uint16_t* X,
                    void* stream) {
  if (plan == nullptr) return PRISM_ERR_ARG;
  PRISM_CHECK_PTR(inv); PRISM_CHECK_PTR(Xp); PRISM_CHECK_PTR(X);
  PRISM_CUDA(prism::launch_unpermute(plan->p, inv, Xp, X, static_cast<cudaStream_t>(stream)));
  return PRISM_OK;
}

}  // extern "C"
