// Combination of the per-range partial results of the tensor-core attention
// kernels (plans with key_chunks > 1).
//
// Prism (arXiv 2610.05416), Fig. 2 caption: a query block attends to the
// union of its selected key blocks.  The kernels walk each head's key blocks
// range by range; a query block's selected blocks in range c give a partial
// softmax state (normalised O_c, running max m_c in log2 units, row sum l_c)
// and a partial dQ_c; the dK / dV kernel walks the query blocks that
// selected a key block range by range in the same way (partial dK_c, dV_c).
// Exact combination:
//   M = max_c m_c,  w_c = l_c 2^(m_c - M),  O = sum_c w_c O_c / sum_c w_c,
//   LSE = (M + log2 sum_c w_c) ln 2,   dQ = sum_c dQ_c,  dK = sum_c dK_c, ...
// over the ranges that hold at least one entry of the block's list.
//
// One CTA per block (256 threads; a query block for O and dQ, a key block
// for dK and dV): the ranges that hold entries are found by binary search in
// the block's ascending list (CSR or CSC); half-warps then take one token row
// each, 16 lanes x 16 bytes = one 256-byte row.
#include "prism_internal.cuh"

namespace prism {
namespace {

constexpr int kCombThreads = 256;
constexpr int kMaxChunks = 64;

// Ranges c in [0, C) with at least one entry of the block's list.
__device__ __forceinline__ void range_flags(const int32_t* row_ptr, const int32_t* col_idx,
                                            long long row, int C, int kc, int* flag) {
  __shared__ int bound[kMaxChunks + 1];
  const int beg = row_ptr[row], end = row_ptr[row + 1];
  if (threadIdx.x <= C)
    bound[threadIdx.x] = threadIdx.x == C ? end : lower_bound_i32(col_idx, beg, end, threadIdx.x * kc);
  __syncthreads();
  if (threadIdx.x < C) flag[threadIdx.x] = bound[threadIdx.x + 1] > bound[threadIdx.x] ? 1 : 0;
  __syncthreads();
}

__global__ void __launch_bounds__(kCombThreads) fwd_combine_kernel(
    int nb, long long Np, int C, int kc, const int32_t* __restrict__ row_ptr,
    const int32_t* __restrict__ col_idx, const int32_t* __restrict__ n_valid,
    const uint16_t* __restrict__ Opart, const float2* __restrict__ ml, uint16_t* __restrict__ Op,
    float* __restrict__ lse) {
  __shared__ int flag[kMaxChunks];
  const long long row = blockIdx.x;
  range_flags(row_ptr, col_idx, row, C, kc, flag);
  const int nvq = n_valid[row];
  bool any = false;
  for (int c = 0; c < C; ++c) any = any || flag[c] != 0;
  const long long bh = row / nb;
  const int i = static_cast<int>(row % nb);
  const int q = threadIdx.x & 15;  // 16-byte piece of the row
  for (int r = threadIdx.x >> 4; r < 128; r += kCombThreads / 16) {
    const long long grow = bh * Np + static_cast<long long>(i) * 128 + r;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float out_lse = 0.f;
    if (any && r < nvq) {
      float M = -INFINITY;
      for (int c = 0; c < C; ++c)
        if (flag[c]) M = fmaxf(M, ml[(row * C + c) * 128 + r].x);
      float L = 0.f;
      for (int c = 0; c < C; ++c)
        if (flag[c]) {
          const float2 v = ml[(row * C + c) * 128 + r];
          L += v.y * exp2f(v.x - M);
        }
      const float invL = 1.f / L;
      for (int c = 0; c < C; ++c) {
        if (!flag[c]) continue;
        const float2 v = ml[(row * C + c) * 128 + r];
        const float wgt = v.y * exp2f(v.x - M) * invL;
        const uint4 u = ldg_nc_v4(Opart + ((row * C + c) * 128 + r) * 128 + q * 8);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[2 * e] = fmaf(wgt, bf16_lo(w4[e]), acc[2 * e]);
          acc[2 * e + 1] = fmaf(wgt, bf16_hi(w4[e]), acc[2 * e + 1]);
        }
      }
      out_lse = (M + log2f(L)) * 0.69314718055994531f;
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(Op + grow * 128 + q * 8) = o;
    if (q == 0) lse[grow] = out_lse;
  }
}

// out tile = sum over the ranges holding entries of the block's list
// (CSR for dQ, CSC for dK and dV) of the bf16 partial tiles.
__global__ void __launch_bounds__(kCombThreads) sum_combine_kernel(
    int nb, long long Np, int C, int kc, const int32_t* __restrict__ ptr,
    const int32_t* __restrict__ idx, const uint16_t* __restrict__ part,
    uint16_t* __restrict__ out) {
  __shared__ int flag[kMaxChunks];
  const long long row = blockIdx.x;
  range_flags(ptr, idx, row, C, kc, flag);
  const long long bh = row / nb;
  const int i = static_cast<int>(row % nb);
  const int q = threadIdx.x & 15;
  for (int r = threadIdx.x >> 4; r < 128; r += kCombThreads / 16) {
    const long long grow = bh * Np + static_cast<long long>(i) * 128 + r;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int c = 0; c < C; ++c) {
      if (!flag[c]) continue;
      const uint4 u = ldg_nc_v4(part + ((row * C + c) * 128 + r) * 128 + q * 8);
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[2 * e] += bf16_lo(w4[e]);
        acc[2 * e + 1] += bf16_hi(w4[e]);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(out + grow * 128 + q * 8) = o;
  }
}

}  // namespace

cudaError_t launch_fwd_combine(const Plan& p, const int32_t* row_ptr, const int32_t* col_idx,
                               const int32_t* n_valid, const uint8_t* ws, uint16_t* Op, float* lse,
                               cudaStream_t st) {
  const long long rows = static_cast<long long>(p.cfg.B) * p.cfg.H * p.sz.nb;
  if (p.sz.key_chunks > kMaxChunks || p.cfg.block_tokens != 128 || p.cfg.d != 128)
    return cudaErrorInvalidValue;
  fwd_combine_kernel<<<static_cast<unsigned>(rows), kCombThreads, 0, st>>>(
      p.sz.nb, p.sz.Np, p.sz.key_chunks, p.sz.chunk_blocks, row_ptr, col_idx, n_valid,
      reinterpret_cast<const uint16_t*>(ws + p.off_part),
      reinterpret_cast<const float2*>(ws + p.off_ml), Op, lse);
  return cudaGetLastError();
}

cudaError_t launch_sum_combine(const Plan& p, const int32_t* ptr, const int32_t* idx,
                               const uint16_t* part, uint16_t* out, cudaStream_t st) {
  const long long rows = static_cast<long long>(p.cfg.B) * p.cfg.H * p.sz.nb;
  if (p.sz.key_chunks > kMaxChunks || p.cfg.block_tokens != 128 || p.cfg.d != 128)
    return cudaErrorInvalidValue;
  sum_combine_kernel<<<static_cast<unsigned>(rows), kCombThreads, 0, st>>>(
      p.sz.nb, p.sz.Np, p.sz.key_chunks, p.sz.chunk_blocks, ptr, idx, part, out);
  return cudaGetLastError();
}

}  // namespace prism
