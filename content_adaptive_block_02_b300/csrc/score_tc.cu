// Block scores S_ij = Qbar_i . Kbar_j (unscaled) on the 5th-generation tensor
// cores, for every (query block, key block) pair of a head, exact enough that
// the Top-k / Top-p selection can certify its decisions.
//
// Prism (arXiv 2610.05416), Fig. 2 caption: block-level (pooled) features give
// a query-block x key-block score.  The selection must not depend on rounding,
// so the scores are needed to far better than fp32 accuracy, while the tensor
// cores accumulate in fp32.  The product is therefore made error-free by
// splitting (Ozaki, Ogita, Oishi and Rump, "Error-free transformations of
// matrix multiplication by using fast routines of matrix multiplication and
// its applications", Numer. Algorithms 59, 2012), with integer digits:
//
//   * each row v of the double-float block means (hi + lo, d channels) is
//     scaled by 2^-e, e the exponent of its largest |hi| (so |v 2^-e| < 1), and
//     written as kSlices digits of 7 bits:
//         v 2^-e = sum_s d_s 2^(-7(s+1)) + rho,   |rho| <= 2^(-7 kSlices - 1)(1 + 2^-20),
//     |d_0| <= 128, |d_s| <= 64 (s >= 1): integers that bf16 holds exactly;
//   * digit slices multiply on the tensor cores (kind::f16, bf16 in, fp32
//     accumulation).  All products d_s(q) d_t(k) of one level u = s + t carry
//     the same weight 2^(-7(u+2)), so each level has its own accumulator
//         P_u = sum_{s+t=u} sum_c d_s,c(q) d_t,c(k),
//     an integer of magnitude below (2 * 128 * 64 + 5 * 64 * 64) * 128 < 2^23
//     (d <= 128): every partial sum is an integer below 2^24, exact in fp32,
//     in whatever order the hardware adds;
//   * levels u <= kSlices - 1 are kept; S = 2^(eq+ek) sum_u P_u 2^(-7(u+2)),
//     summed in double-float (TwoSum) from the smallest level.
// Error of S (unscaled, with d channels): the dropped levels u >= kSlices and
// the digit remainders give |S - S_exact| <= 2^(eq+ek) d 1.3 * 2^(-7 kSlices)
// (4.5e-15 2^(eq+ek) d with kSlices = 7), i.e. about 2.3e-12 max|q| max|k| for
// d = 128 -- the size of the double-float block means' own error, and far
// below the 1e-6 margin the selection certifies its decisions against.
//
// Layout.  Digits: bf16 [kSlices, R, dpad] per operand (R = B*H*nslots rows,
// dpad = d rounded up to 64, zero channels past d), exponents int32 [R].
// Kernel: one CTA per (128 key blocks, 64 query blocks, head); the key digits
// are the A operand (M = 128: tensor-memory lane = key block, so that the
// epilogue's stores along a score row are coalesced), the query digits the B
// operand (N = 64).  All kSlices query slices stay in shared memory; key
// slices stream through two stages.  Accumulator u takes tensor-memory
// columns [64u, 64u + 64).  Two threads issue the MMAs (levels split between
// them, so no accumulator is written by both): one tcgen05.mma issue every
// ~100 cycles per thread is the bound, not the tensor pipe.
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace prism {

bool make_bf16_map(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
using namespace tc;

constexpr int kSlices = 7;
constexpr int kTJ = 128;                 // key blocks per tile (M)
constexpr int kTI = 64;                  // query blocks per tile (N)
constexpr int kThreads = 128;
constexpr int kBoxK = kTJ * 128;         // bytes of one 64-channel box of a key slice
constexpr int kBoxQ = kTI * 128;         // bytes of one 64-channel box of a query slice

// 2^k for an integer k in [-126, 127] (a normal float, exact).
__device__ __forceinline__ float pow2i(int k) {
  return __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
}

// ------------------------------------------------------------ digits ------
// One warp per row of the double-float means (hi, lo) [R, d]: the row's
// exponent e and its kSlices 7-bit digits, written as bf16 to
// D[s][row][0..dpad) (channels past d are zero).  blockIdx.y selects the
// operand (0: query means, 1: key means).
struct DigitArgs {
  const float* hi[2];
  const float* lo[2];
  uint16_t* D[2];
  int32_t* ex[2];
  long long R;
  int d, dpad;
};

__global__ void __launch_bounds__(256) score_digits_kernel(DigitArgs a) {
  const int op = blockIdx.y;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.R) return;
  // operands picked by selects, not by a dynamic index into the parameters
  const float* h = (op ? a.hi[1] : a.hi[0]) + row * a.d;
  const float* l = (op ? a.lo[1] : a.lo[0]) + row * a.d;
  float vh[4], vl[4];
  float m = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int c = lane + 32 * q;
    vh[q] = c < a.d ? h[c] : 0.f;
    vl[q] = c < a.d ? l[c] : 0.f;
    m = fmaxf(m, fabsf(vh[q]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  // e with max|hi| < 2^e (and >= 2^(e-1) for a normal maximum); 0 for a zero
  // row; at most 127, so that 2^(eq + ek) splits into two normal factors
  const uint32_t bx = (__float_as_uint(m) >> 23) & 0xffu;
  int e = m == 0.f ? 0 : (bx == 0 ? -126 : static_cast<int>(bx) - 126);
  e = e > 127 ? 127 : e;
  const int e1 = e >> 1, e2 = e - e1;
  const float s1 = pow2i(-e1), s2 = pow2i(-e2);
  uint16_t* D = op ? a.D[1] : a.D[0];
  const long long slice = a.R * a.dpad;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int c = lane + 32 * q;
    if (c >= a.dpad) break;
    // the remainder as an unevaluated pair (x, y), kept normalised by TwoSum
    float x = vh[q] * s1 * s2, y = vl[q] * s1 * s2;
#pragma unroll
    for (int s = 0; s < kSlices; ++s) {
      const float z = x * 128.f;
      const float dg = rintf(z);
      const df t = two_sum(z - dg, y * 128.f);  // z - dg: exact fractional part
      x = t.hi;
      y = t.lo;
      // |dg| <= 128 is an integer: its bf16 pattern is the float's upper half
      D[s * slice + row * a.dpad + c] = static_cast<uint16_t>(__float_as_uint(dg) >> 16);
    }
  }
  if (lane == 0) (op ? a.ex[1] : a.ex[0])[row] = e;
}

// ------------------------------------------------------- digit GEMM --------
struct ScoreParams {
  const int32_t* eq;   // [R] query-row exponents
  const int32_t* ek;   // [R] key-row exponents
  float* Shi;          // [B*H, nb, nb]
  float* Slo;
  uint32_t* status;
  long long R;         // rows of one digit slice
  int nb;              // blocks (slots) per head
  int nbox;            // 64-channel boxes per row (dpad / 64)
  unsigned long long limit;
};

// Which of the two issuing threads owns level u (pairs per level: u + 1;
// 15 of the 28 pairs for thread 0, 13 for thread 1).
__host__ __device__ constexpr int level_owner(int u) {
  return (u == 6 || u == 4 || u == 1 || u == 0) ? 0 : 1;
}

__global__ void __launch_bounds__(kThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tmKd,
                    const __grid_constant__ CUtensorMap tmQd, ScoreParams P) {
  extern __shared__ uint8_t dsm_raw[];
  __shared__ uint64_t q_full, k_full[2], k_empty[2], done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ int s_eq[kTI];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const int nbox = P.nbox;
  uint8_t* sK = dsm;                                // 2 stages x nbox boxes of kBoxK
  uint8_t* sQ = dsm + 2 * nbox * kBoxK;             // kSlices x nbox boxes of kBoxQ
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.z;
  const int j0 = blockIdx.x * kTJ, i0 = blockIdx.y * kTI;
  const long long rowK = static_cast<long long>(bh) * P.nb + j0;
  const long long rowQ = static_cast<long long>(bh) * P.nb + i0;

  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 2);  // both issuers commit once per key slice
    }
    mbar_init(&done, 2);          // both issuers commit once after their last MMA
    abort_flag = 0;
    mbar_init_fence();
  }
  if (threadIdx.x < kTI)
    s_eq[threadIdx.x] = i0 + static_cast<int>(threadIdx.x) < P.nb ? P.eq[rowQ + threadIdx.x] : 0;
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base;
  const Waiter W{&abort_flag, P.status, P.limit};

  int k_issued[2] = {0, 0}, k_waited[2] = {0, 0};  // thread 0: loads per stage, to drain
  bool q_waited = false;
  auto load_k = [&](int s) {  // thread 0: key slice s into stage s & 1
    const int st = s & 1;
    ++k_issued[st];
    mbar_expect_tx(&k_full[st], nbox * kBoxK);
    for (int k = 0; k < nbox; ++k)
      tma_load_2d(sK + (st * nbox + k) * kBoxK, &tmKd, &k_full[st], 64 * k,
                  static_cast<int>(s * P.R + rowK));
  };
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmKd);
    tma_prefetch_desc(&tmQd);
    mbar_expect_tx(&q_full, kSlices * nbox * kBoxQ);
    for (int s = 0; s < kSlices; ++s)
      for (int k = 0; k < nbox; ++k)
        tma_load_2d(sQ + (s * nbox + k) * kBoxQ, &tmQd, &q_full, 64 * k,
                    static_cast<int>(s * P.R + rowQ));
    load_k(0);
    load_k(1);
  }

  bool ok = true;
  if (threadIdx.x == 0 || threadIdx.x == 32) {
    const int me = threadIdx.x == 0 ? 0 : 1;
    const uint32_t idesc = idesc_bf16(kTJ, kTI, 0, 0);  // A = key digits, B = query digits
    ok = W.wait(&q_full, 0, 401);
    if (me == 0) q_waited = ok;
    for (int s = 0; s < kSlices && ok; ++s) {
      const int st = s & 1;
      ok = W.wait(&k_full[st], (s >> 1) & 1, 402);
      if (!ok) break;
      if (me == 0) ++k_waited[st];
      fence_after();
      const uint64_t a0 = sdesc_sw128(smem_u32(sK + st * nbox * kBoxK), 16, 1024);
      for (int t = 0; s + t < kSlices; ++t) {
        const int u = s + t;
        if (level_owner(u) != me) continue;
        const uint64_t b0 = sdesc_sw128(smem_u32(sQ + t * nbox * kBoxQ), 16, 1024);
        for (int kk = 0; kk < 4 * nbox; ++kk) {
          const uint64_t ao = static_cast<uint64_t>(((kk >> 2) * kBoxK + (kk & 3) * 32) >> 4);
          const uint64_t bo = static_cast<uint64_t>(((kk >> 2) * kBoxQ + (kk & 3) * 32) >> 4);
          // level u's first product (s = 0, kk = 0) initialises its accumulator
          mma_ss(tmem + 64u * u, a0 + ao, b0 + bo, idesc, (s > 0 || kk > 0) ? 1u : 0u);
        }
      }
      commit(&k_empty[st]);
      // key slice s + 1 goes where slice s - 1 was, once both issuers' MMAs on
      // slice s - 1 have completed
      if (me == 0 && s + 1 < kSlices && s >= 1) {
        ok = W.wait(&k_empty[(s + 1) & 1], ((s - 1) >> 1) & 1, 403);
        if (ok) load_k(s + 1);
      }
    }
    commit(&done);  // also on an abort: the teardown waits for the MMAs issued
  }
  __syncwarp();
  // ---- epilogue: thread = key block j (tensor-memory lane), 64 query columns
  ok = W.wait(&done, 0, 404) && ok;
  ok = __syncthreads_and(ok);
  if (ok) {
    fence_after();
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int j = j0 + warp * 32 + lane;
    const bool jv = j < P.nb;
    const int ekj = jv ? P.ek[rowK + warp * 32 + lane] : 0;
    float* shi = P.Shi + static_cast<long long>(bh) * P.nb * P.nb + j;
    float* slo = P.Slo + static_cast<long long>(bh) * P.nb * P.nb + j;
    for (int c0 = 0; c0 < kTI; c0 += 16) {
      if (i0 + c0 >= P.nb) break;  // uniform over the CTA
      uint32_t acc[kSlices][16];
#pragma unroll
      for (int u = 0; u < kSlices; ++u) tmem_ld16(tmem + lane_base + 64u * u + c0, acc[u]);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int i = i0 + c0 + e;
        // levels from the smallest: each term P_u 2^(-7(u+2)) is exact
        float s = __uint_as_float(acc[kSlices - 1][e]) * pow2i(-7 * (kSlices + 1));
        float cc = 0.f;
#pragma unroll
        for (int u = kSlices - 2; u >= 0; --u) {
          const df t = two_sum(s, __uint_as_float(acc[u][e]) * pow2i(-7 * (u + 2)));
          s = t.hi;
          cc = __fadd_rn(cc, t.lo);
        }
        const df r = fast_two_sum(s, cc);
        const int f = s_eq[c0 + e] + ekj, f1 = f >> 1, f2 = f - f1;
        const float g1 = pow2i(f1), g2 = pow2i(f2);
        if (jv && i < P.nb) {
          const long long o = static_cast<long long>(i) * P.nb;
          shi[o] = r.hi * g1 * g2;
          slo[o] = r.lo * g1 * g2;
        }
      }
    }
  }

  // ---------------------------------------------------------- teardown ----
  fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    // no copy may still be landing in shared memory when the CTA leaves
    if (!q_waited && !wait_raw(&q_full, 0, P.limit)) dev_error(P.status, DEV_ERR_TIMEOUT, 497, 0);
    for (int st = 0; st < 2; ++st)
      if (k_issued[st] > k_waited[st] &&
          !wait_raw(&k_full[st], (k_issued[st] - 1) & 1, P.limit))
        dev_error(P.status, DEV_ERR_TIMEOUT, 498, st);
  }
  if (warp == 0) {
    // every MMA of both issuers has completed before the columns are freed
    if (!wait_raw(&done, 0, P.limit) && lane == 0) dev_error(P.status, DEV_ERR_TIMEOUT, 499, 0);
    fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t score_digit_bytes(const Plan& p) {
  const long long R = static_cast<long long>(p.cfg.B) * p.cfg.H * p.sz.nslots;
  const int dpad = (p.cfg.d + 63) / 64 * 64;
  return 2 * (static_cast<size_t>(kSlices) * R * dpad * 2 + 256) + 2 * static_cast<size_t>(R) * 4;
}

cudaError_t launch_score_tc(const Plan& p, const float* Qh, const float* Ql, const float* Kh,
                            const float* Kl, float* Shi, float* Slo, uint8_t* ws,
                            cudaStream_t st) {
  const prism_config_t& c = p.cfg;
  const int nb = p.sz.nslots;
  const long long R = static_cast<long long>(c.B) * c.H * nb;
  const int dpad = (c.d + 63) / 64 * 64;
  const size_t slice_bytes = static_cast<size_t>(kSlices) * R * dpad * 2;
  uint8_t* base = ws + p.off_digits;
  uint16_t* DQ = reinterpret_cast<uint16_t*>(base);
  uint16_t* DK = reinterpret_cast<uint16_t*>(base + slice_bytes + 256);
  int32_t* eQ = reinterpret_cast<int32_t*>(base + 2 * (slice_bytes + 256));
  int32_t* eK = eQ + R;
  if (R * kSlices >= (1LL << 31)) return cudaErrorInvalidValue;
  DigitArgs da;
  da.hi[0] = Qh; da.lo[0] = Ql; da.D[0] = DQ; da.ex[0] = eQ;
  da.hi[1] = Kh; da.lo[1] = Kl; da.D[1] = DK; da.ex[1] = eK;
  da.R = R;
  da.d = c.d;
  da.dpad = dpad;
  score_digits_kernel<<<dim3(static_cast<unsigned>((R + 7) / 8), 2), 256, 0, st>>>(da);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap tmKd, tmQd;
  if (!make_bf16_map(&tmKd, DK, kSlices * R, dpad, kTJ) ||
      !make_bf16_map(&tmQd, DQ, kSlices * R, dpad, kTI))
    return cudaErrorInvalidValue;
  ScoreParams a;
  a.eq = eQ;
  a.ek = eK;
  a.Shi = Shi;
  a.Slo = Slo;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.R = R;
  a.nb = nb;
  a.nbox = dpad / 64;
  a.limit = c.timeout_cycles ? c.timeout_cycles : 4000000000ull;
  const size_t smem = static_cast<size_t>(a.nbox) * (2 * kBoxK + kSlices * kBoxQ) + 1024;
  e = cudaFuncSetAttribute(score_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 g(static_cast<unsigned>((nb + kTJ - 1) / kTJ), static_cast<unsigned>((nb + kTI - 1) / kTI),
               static_cast<unsigned>(c.B * c.H));
  score_tc_kernel<<<g, kThreads, smem, st>>>(tmKd, tmQd, a);
  return cudaGetLastError();
}

}  // namespace prism
