// Internal declarations shared by the Prism CUDA translation units:
// the host plan, the workspace layout, the device status word and the
// kernel launchers.  Nothing here is part of the public C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "prism.h"

namespace prism {

// ---------------------------------------------------------------- plan ----

struct Plan {
  prism_config_t cfg;
  prism_sizes_t sz;
  double log2_ext[PRISM_MAX_SHAPES][3];  // log2 of every menu extent
  double log2_S;
  // workspace offsets (bytes), each region 256-aligned
  size_t off_rowcnt, off_colcnt, off_amb, off_bitmask, off_scores, off_D, off_lse2, off_dq;
  size_t off_part, off_ml;  // key-range partial results (key_chunks > 1)
  size_t off_nsel, off_bstart, off_tbitmask;  // multi-tile blocks (sz.multi_tile)
  size_t off_digits;  // score digits and exponents of the block means
};

// Workspace layout (bytes from the start of ws, each region 256-aligned):
//   [0, 256)        status word (uint32 at 0) and small counters
//   off_rowcnt      int32 [B*H*nb]       selected key blocks per query block
//   off_colcnt      int32 [B*H*nb]       query blocks that selected each key block
//   off_amb         int32 [B*H*nb]       rows whose fp32 decision was ambiguous
//   off_bitmask     u32   [B*H*nb*nw]    selection bitmask, nw = ceil(nb/32)
//   off_scores      fp32  [2*B*H*nb*nb]  block scores (unscaled dots), hi then lo
//   off_D           fp32  [B*H*Np]       rowsum(dO * O) for the backward
//   off_lse2        fp32  [B*H*Np]       -LSE * log2(e) for the backward
//   off_dq          fp32  [B*H*Np*d]     dQ accumulator of the CUDA-core backward
//                                        (empty for a tensor-core plan)
//   off_nsel        int32 [B*H*nb]       (multi-tile blocks) real tokens of the block
//                                        starting at each tile, 0 on continuations
//   off_bstart      int32 [B*H*nb]       (multi-tile blocks) first tile of each tile's block
//   off_tbitmask    u32   [B*H*nb*nw]    (multi-tile blocks) tile-level selection bitmask
//   off_part        bf16  2 x [B*H*nb, C, S, d] per key / query range: the forward's
//                                        normalised partial O, later the dK and dV
//                                        kernel's partial dK and dV, then the dQ
//                                        kernel's partial dQ (first half)
//   off_ml          fp32  [B*H*nb, C, S, 2] per key range: running max (log2 units)
//                                        and row sum of the forward
//   off_digits      bf16  2 x [7, B*H*nslots, dpad] 7-bit digits of the query and
//                                        key block means (score_tc.cu), then int32
//                                        2 x [B*H*nslots] their exponents
enum : int {
  WS_STATUS = 0,      // uint32: first device error code (0 = none)
  WS_AMB_COUNT = 1,   // uint32: number of ambiguous rows appended by the select kernel
  WS_FWD_QUEUE = 2,   // uint32: next work item of the persistent forward
  WS_BWD_QUEUE = 3,   // uint32: next work item of the persistent backward
  WS_ERR_INFO = 4,    // uint32 x4: where a device error was raised
  WS_DQ_QUEUE = 8,    // uint32: next work item of the persistent dQ kernel
};

enum : uint32_t { DEV_ERR_TIMEOUT = 1, DEV_ERR_BOUNDS = 2 };

// --------------------------------------------------------- launchers ------
// Each returns cudaGetLastError() after enqueueing.

// nrm: when not null, the A2V norms [B, N] (fp32) are read instead of a2v
cudaError_t launch_zone_stats(const Plan& p, const uint16_t* V, const uint16_t* a2v,
                              const float* nrm, float* stats, cudaStream_t st);
cudaError_t launch_a2v_norms(const Plan& p, const uint16_t* Qa, const uint16_t* Ka,
                             const uint16_t* Va, int Na, float* n, uint8_t* ws, cudaStream_t st);
size_t a2v_smem_bytes(int Ca, int Na);
cudaError_t launch_assign(const Plan& p, const float* stats, uint8_t* shape_id,
                          uint8_t* shape_tie, cudaStream_t st);
// status: when not null, a shape id that is not admissible is recorded there
// (DEV_ERR_BOUNDS); such a zone always falls back to the first admissible shape.
cudaError_t launch_permute_pool(const Plan& p, const uint8_t* shape_id, const uint16_t* Q,
                                const uint16_t* K, const uint16_t* V, int32_t* perm,
                                int32_t* inv, uint16_t* Qp, uint16_t* Kp, uint16_t* Vp,
                                float* Qh, float* Ql, float* Kh, float* Kl, int32_t* n_valid,
                                uint32_t* status, cudaStream_t st);
cudaError_t launch_permute(const Plan& p, const int32_t* perm, const uint16_t* X, uint16_t* Xp,
                           cudaStream_t st);
cudaError_t launch_unpermute(const Plan& p, const int32_t* inv, const uint16_t* Xp, uint16_t* X,
                             cudaStream_t st);
cudaError_t launch_dq_convert(const Plan& p, const float* dq, float scale, uint16_t* dQp,
                              cudaStream_t st);
cudaError_t launch_select(const Plan& p, const uint8_t* shape_id, const float* Qh,
                          const float* Ql, const float* Kh, const float* Kl,
                          const int32_t* n_valid, uint8_t* sel_tie,
                          int32_t* row_ptr, int32_t* col_idx, int32_t* col_ptr,
                          int32_t* row_idx, uint8_t* ws, cudaStream_t st,
                          cudaEvent_t score_begin = nullptr, cudaEvent_t score_end = nullptr);

// Block scores on the tensor cores (exact digit products): Shi / Slo
// [B*H, nslots, nslots] from the double-float block means.
cudaError_t launch_score_tc(const Plan& p, const float* Qh, const float* Ql, const float* Kh,
                            const float* Kl, float* Shi, float* Slo, uint8_t* ws,
                            cudaStream_t st);
size_t score_digit_bytes(const Plan& p);  // workspace bytes at off_digits

// ----------------------------------------------------- device helpers -----

__device__ __forceinline__ void dev_error(uint32_t* status, uint32_t code, uint32_t a = 0,
                                          uint32_t b = 0) {
  if (atomicCAS(status + WS_STATUS, 0u, code) == 0u) {
    status[WS_ERR_INFO + 0] = a;
    status[WS_ERR_INFO + 1] = b;
    status[WS_ERR_INFO + 2] = blockIdx.x;
    status[WS_ERR_INFO + 3] = threadIdx.x;
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f(uint16_t u) {
  return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

// Round-to-nearest-even float -> bf16 bits (NaN kept quiet).
__device__ __forceinline__ uint16_t f_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// First position in col[lo, hi) holding a value >= key (col ascending).
__device__ __forceinline__ int lower_bound_i32(const int32_t* col, int lo, int hi, int key) {
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (col[mid] < key)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ------------------------------------------------------ double-float -----
// A value carried as an unevaluated sum hi + lo of two fp32 numbers
// (|lo| <= ulp(hi)/2).  Every operation below uses explicitly rounded
// intrinsics so that the compiler cannot contract them into FMAs.
// Packed pairs of fp32 for the fp32x2 fma / add / sub / mul of sm_100-class
// SMs: one instruction for two lanes, each rounded exactly as the scalar
// operation would be.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

struct df {
  float hi, lo;
};
__device__ __forceinline__ df two_sum(float a, float b) {  // Knuth
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, err};
}
__device__ __forceinline__ df fast_two_sum(float a, float b) {  // Dekker, |a| >= |b|
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ df df_add(df x, df y) {
  df s = two_sum(x.hi, y.hi);
  s.lo = __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo));
  return fast_two_sum(s.hi, s.lo);
}
__device__ __forceinline__ df df_neg(df x) { return {-x.hi, -x.lo}; }
__device__ __forceinline__ df df_mul(df x, df y) {
  const float p = __fmul_rn(x.hi, y.hi);
  float e = fmaf(x.hi, y.hi, -p);
  e = fmaf(x.hi, y.lo, e);
  e = fmaf(x.lo, y.hi, e);
  return fast_two_sum(p, e);
}
// x / n for a positive integer n < 2^24: the remainder of a correctly
// rounded fp32 quotient is exact, so two fp32 divisions give ~46 bits.
__device__ __forceinline__ df df_div_int(df x, int n) {
  const float fn = static_cast<float>(n);
  const float q1 = __fdiv_rn(x.hi, fn);
  float r = fmaf(-q1, fn, x.hi);
  r = __fadd_rn(r, x.lo);
  const float q2 = __fdiv_rn(r, fn);
  return fast_two_sum(q1, q2);
}

}  // namespace prism
