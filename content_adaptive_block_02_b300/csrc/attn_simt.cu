// Block-sparse attention on CUDA cores, for any block size S <= 128 and
// head dim d <= 128 (multiples of 8).  The tensor-core kernels cover S = 128,
// d = 128; this path serves the small configurations (e.g. 16-token blocks).
//
// Prism (arXiv 2610.05416), Fig. 2 caption: attention runs only between a
// query block and the key blocks selected for it.  Reading used here: exact
// softmax over the real tokens of the selected key blocks (padding slots are
// masked), scale `scale`, no causal mask, natural-log LSE.  Backward: the
// standard softmax-attention VJP with the selection held fixed (Prism trains
// through this attention, Table 2 caption).
#include <float.h>

#include "prism_internal.cuh"

namespace prism {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxCh = 64;  // channels per thread (d / (256 / S) <= 64)

__device__ __forceinline__ void load_tile(uint16_t* dst, const uint16_t* src, int rows, int d) {
  const int P = d / 8;
  for (int e = threadIdx.x; e < rows * P; e += blockDim.x)
    reinterpret_cast<uint4*>(dst)[e] = ldg_nc_v4(src + static_cast<long long>(e) * 8);
}

__device__ __forceinline__ float dot_bf16(const uint16_t* a, const uint16_t* b, int d) {
  float s = 0.f;
  const uint32_t* a2 = reinterpret_cast<const uint32_t*>(a);
  const uint32_t* b2 = reinterpret_cast<const uint32_t*>(b);
  for (int c = 0; c < d / 2; ++c) {
    const uint32_t x = a2[c], y = b2[c];
    s = fmaf(bf16_lo(x), bf16_lo(y), s);
    s = fmaf(bf16_hi(x), bf16_hi(y), s);
  }
  return s;
}

struct FwdArgs {
  int S, d, nb;
  long long Np, rows;
  float scale_log2;  // scale * log2(e)
  const uint16_t *Qp, *Kp, *Vp;
  const int32_t *n_valid, *row_ptr, *col_idx;
  uint16_t* Op;
  float* lse;
};

// One CTA per (b, h, query block).  Thread t owns query row r = t % S and
// channel group cg = t / S (d / (256/S) channels).
__global__ void __launch_bounds__(kThreads) simt_fwd_kernel(FwdArgs a) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int S = a.S, d = a.d;
  uint16_t* Qs = reinterpret_cast<uint16_t*>(sm);
  uint16_t* Ks = Qs + S * d;
  uint16_t* Vs = Ks + S * d;
  float* Ps = reinterpret_cast<float*>(Vs + S * d);  // [S][S + 1]
  const long long row = blockIdx.x;                 // (b*H + h)*nb + i
  const long long bh = row / a.nb;
  const int i = static_cast<int>(row % a.nb);
  const int CG = kThreads / S, cpt = d / CG;
  const int r = threadIdx.x % S, cg = threadIdx.x / S;
  const int nvi = a.n_valid[row];
  const int beg = a.row_ptr[row], end = a.row_ptr[row + 1];
  const long long base = (bh * a.Np + static_cast<long long>(i) * S);
  if (nvi == 0 || beg == end) {
    for (int e = threadIdx.x; e < S * d / 8; e += blockDim.x)
      reinterpret_cast<uint4*>(a.Op + base * d)[e] = make_uint4(0, 0, 0, 0);
    for (int e = threadIdx.x; e < S; e += blockDim.x) a.lse[base + e] = 0.f;
    return;
  }
  load_tile(Qs, a.Qp + base * d, S, d);
  float acc[kMaxCh];
#pragma unroll
  for (int k = 0; k < kMaxCh; ++k) acc[k] = 0.f;
  float m = -FLT_MAX, l = 0.f;
  for (int t = beg; t < end; ++t) {
    const int j = a.col_idx[t];
    const int nvj = a.n_valid[bh * a.nb + j];
    __syncthreads();
    load_tile(Ks, a.Kp + (bh * a.Np + static_cast<long long>(j) * S) * d, S, d);
    load_tile(Vs, a.Vp + (bh * a.Np + static_cast<long long>(j) * S) * d, S, d);
    __syncthreads();
    for (int e = threadIdx.x; e < S * S; e += blockDim.x) {
      const int rr = e / S, cc = e % S;
      Ps[rr * (S + 1) + cc] =
          cc < nvj ? dot_bf16(Qs + rr * d, Ks + cc * d, d) * a.scale_log2 : -FLT_MAX;
    }
    __syncthreads();
    float mx = m;
    for (int cc = 0; cc < nvj; ++cc) mx = fmaxf(mx, Ps[r * (S + 1) + cc]);
    const float corr = exp2f(m - mx);
    l *= corr;
#pragma unroll
    for (int k = 0; k < kMaxCh; ++k) acc[k] *= corr;
    for (int cc = 0; cc < nvj; ++cc) {
      const float p = exp2f(Ps[r * (S + 1) + cc] - mx);
      l += p;
      const uint16_t* v = Vs + cc * d + cg * cpt;
#pragma unroll
      for (int k = 0; k < kMaxCh; ++k)
        if (k < cpt) acc[k] = fmaf(p, bf16_to_f(v[k]), acc[k]);
    }
    m = mx;
  }
  uint16_t* o = a.Op + (base + r) * d + cg * cpt;
  const float inv = r < nvi ? 1.f / l : 0.f;
#pragma unroll
  for (int k = 0; k < kMaxCh; ++k)
    if (k < cpt) o[k] = f_to_bf16(acc[k] * inv);
  if (cg == 0) a.lse[base + r] = r < nvi ? (m + log2f(l)) * 0.69314718055994531f : 0.f;
}

struct BwdArgs {
  int S, d, nb;
  long long Np;
  float scale, scale_log2;
  const uint16_t *Qp, *Kp, *Vp, *dOp;
  const float *lse, *D;
  const int32_t *n_valid, *col_ptr, *row_idx;
  float* dQacc;
  uint16_t *dKp, *dVp;
};

// One CTA per (b, h, key block j) looping over the query blocks that
// selected j (ascending).  Thread t owns key row c = t % S and a channel
// group for dK / dV, and query row r = t % S for the dQ partial, which is
// added to the fp32 accumulator with atomics.
__global__ void __launch_bounds__(kThreads) simt_bwd_kernel(BwdArgs a) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int S = a.S, d = a.d;
  uint16_t* Qs = reinterpret_cast<uint16_t*>(sm);
  uint16_t* dOs = Qs + S * d;
  uint16_t* Ks = dOs + S * d;
  uint16_t* Vs = Ks + S * d;
  float* Ps = reinterpret_cast<float*>(Vs + S * d);  // [S][S + 1]
  float* Ls = Ps + S * (S + 1);                     // lse (log2 units) [S]
  float* Ds = Ls + S;                               // D [S]
  const long long col = blockIdx.x;                 // (b*H + h)*nb + j
  const long long bh = col / a.nb;
  const int j = static_cast<int>(col % a.nb);
  const int CG = kThreads / S, cpt = d / CG;
  const int c = threadIdx.x % S, cg = threadIdx.x / S;
  const int nvj = a.n_valid[col];
  const int beg = a.col_ptr[col], end = a.col_ptr[col + 1];
  const long long kbase = bh * a.Np + static_cast<long long>(j) * S;
  load_tile(Ks, a.Kp + kbase * d, S, d);
  load_tile(Vs, a.Vp + kbase * d, S, d);
  float dk[kMaxCh], dv[kMaxCh];
#pragma unroll
  for (int k = 0; k < kMaxCh; ++k) dk[k] = dv[k] = 0.f;
  for (int t = beg; t < end; ++t) {
    const int i = a.row_idx[t];
    const int nvi = a.n_valid[bh * a.nb + i];
    const long long qbase = bh * a.Np + static_cast<long long>(i) * S;
    __syncthreads();
    load_tile(Qs, a.Qp + qbase * d, S, d);
    load_tile(dOs, a.dOp + qbase * d, S, d);
    for (int e = threadIdx.x; e < S; e += blockDim.x) {
      Ls[e] = a.lse[qbase + e] * 1.4426950408889634f;
      Ds[e] = a.D[qbase + e];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < S * S; e += blockDim.x) {
      const int rr = e / S, cc = e % S;
      float p = 0.f;
      if (rr < nvi && cc < nvj)
        p = exp2f(dot_bf16(Qs + rr * d, Ks + cc * d, d) * a.scale_log2 - Ls[rr]);
      Ps[rr * (S + 1) + cc] = p;
    }
    __syncthreads();
    for (int rr = 0; rr < S; ++rr) {
      const float p = Ps[rr * (S + 1) + c];
      const uint16_t* g = dOs + rr * d + cg * cpt;
#pragma unroll
      for (int k = 0; k < kMaxCh; ++k)
        if (k < cpt) dv[k] = fmaf(p, bf16_to_f(g[k]), dv[k]);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < S * S; e += blockDim.x) {
      const int rr = e / S, cc = e % S;
      const float p = Ps[rr * (S + 1) + cc];
      if (p != 0.f) Ps[rr * (S + 1) + cc] = p * (dot_bf16(dOs + rr * d, Vs + cc * d, d) - Ds[rr]);
    }
    __syncthreads();
    for (int rr = 0; rr < S; ++rr) {
      const float ds = Ps[rr * (S + 1) + c];
      const uint16_t* q = Qs + rr * d + cg * cpt;
#pragma unroll
      for (int k = 0; k < kMaxCh; ++k)
        if (k < cpt) dk[k] = fmaf(ds, bf16_to_f(q[k]), dk[k]);
    }
    {
      const int r = c;  // query row for the dQ partial
      float dq[kMaxCh];
#pragma unroll
      for (int k = 0; k < kMaxCh; ++k) dq[k] = 0.f;
      for (int cc = 0; cc < nvj; ++cc) {
        const float ds = Ps[r * (S + 1) + cc];
        const uint16_t* kk = Ks + cc * d + cg * cpt;
#pragma unroll
        for (int k = 0; k < kMaxCh; ++k)
          if (k < cpt) dq[k] = fmaf(ds, bf16_to_f(kk[k]), dq[k]);
      }
      if (r < nvi) {
        float* dst = a.dQacc + (qbase + r) * d + cg * cpt;
#pragma unroll
        for (int k = 0; k < kMaxCh; ++k)
          if (k < cpt) atomicAdd(dst + k, dq[k]);
      }
    }
  }
  uint16_t* ok = a.dKp + (kbase + c) * d + cg * cpt;
  uint16_t* ov = a.dVp + (kbase + c) * d + cg * cpt;
  const bool real = c < nvj;
#pragma unroll
  for (int k = 0; k < kMaxCh; ++k)
    if (k < cpt) {
      ok[k] = f_to_bf16(real ? dk[k] * a.scale : 0.f);
      ov[k] = f_to_bf16(real ? dv[k] : 0.f);
    }
}

}  // namespace

// D[b,h,s] = sum_c dOp * Op (fp32); when nlse2 is given, also
// nlse2 = -lse * log2(e); when dQacc is given, that row of the accumulator is
// cleared.  Four lanes per row of d channels (d <= 128: at most four 16-byte
// pieces of O and of dO per lane, all loads issued before the first use).
__global__ void bwd_pre_kernel(long long rows, int d, const uint16_t* __restrict__ Op,
                               const uint16_t* __restrict__ dOp, const float* __restrict__ lse,
                               float* __restrict__ D, float* __restrict__ nlse2,
                               float* __restrict__ dQacc) {
  const long long tid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  const long long row = tid >> 2;
  const int sub = static_cast<int>(tid & 3);
  const bool live = row < rows;  // no early return: the row's lanes shuffle below
  const int P = d / 8;           // 16-byte pieces per row
  float s = 0.f;
  if (live) {
    const uint16_t* orow = Op + row * d;
    const uint16_t* grow = dOp + row * d;
    uint4 ov[4], gv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int q = sub + 4 * k;
      if (q < P) {
        ov[k] = ldg_nc_v4(orow + q * 8);
        gv[k] = ldg_nc_v4(grow + q * 8);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int q = sub + 4 * k;
      if (q < P) {
        const uint32_t ow[4] = {ov[k].x, ov[k].y, ov[k].z, ov[k].w};
        const uint32_t gw[4] = {gv[k].x, gv[k].y, gv[k].z, gv[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          s = fmaf(bf16_lo(ow[e]), bf16_lo(gw[e]), s);
          s = fmaf(bf16_hi(ow[e]), bf16_hi(gw[e]), s);
        }
        if (dQacc != nullptr) {
          float4* dq = reinterpret_cast<float4*>(dQacc + row * d + q * 8);
          dq[0] = make_float4(0.f, 0.f, 0.f, 0.f);
          dq[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  if (live && sub == 0) {
    D[row] = s;
    if (nlse2 != nullptr) nlse2[row] = -lse[row] * 1.4426950408889634f;
  }
}

cudaError_t launch_bwd_pre(const Plan& p, const uint16_t* Op, const uint16_t* dOp,
                           const float* lse, float* D, float* nlse2, float* dQacc,
                           cudaStream_t st) {
  const long long rows = static_cast<long long>(p.cfg.B) * p.cfg.H * p.sz.Np;
  bwd_pre_kernel<<<static_cast<unsigned>((rows * 4 + 255) / 256), 256, 0, st>>>(
      rows, p.cfg.d, Op, dOp, lse, D, nlse2, dQacc);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd_simt(const Plan& p, const uint16_t* Qp, const uint16_t* Kp,
                                 const uint16_t* Vp, const int32_t* n_valid,
                                 const int32_t* row_ptr, const int32_t* col_idx, float scale,
                                 uint16_t* Op, float* lse, cudaStream_t st) {
  const prism_config_t& c = p.cfg;
  FwdArgs a;
  a.S = c.block_tokens;
  a.d = c.d;
  a.nb = p.sz.nb;
  a.Np = p.sz.Np;
  a.rows = static_cast<long long>(c.B) * c.H * p.sz.nb;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.Qp = Qp; a.Kp = Kp; a.Vp = Vp;
  a.n_valid = n_valid; a.row_ptr = row_ptr; a.col_idx = col_idx;
  a.Op = Op; a.lse = lse;
  const size_t smem = 3ull * a.S * a.d * 2 + static_cast<size_t>(a.S) * (a.S + 1) * 4;
  cudaError_t e = cudaFuncSetAttribute(simt_fwd_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  simt_fwd_kernel<<<static_cast<unsigned>(a.rows), kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_simt(const Plan& p, const uint16_t* Qp, const uint16_t* Kp,
                                 const uint16_t* Vp, const uint16_t* dOp, const float* lse,
                                 const float* D, const int32_t* n_valid,
                                 const int32_t* col_ptr, const int32_t* row_idx, float scale,
                                 float* dQacc, uint16_t* dKp, uint16_t* dVp, cudaStream_t st) {
  const prism_config_t& c = p.cfg;
  BwdArgs a;
  a.S = c.block_tokens;
  a.d = c.d;
  a.nb = p.sz.nb;
  a.Np = p.sz.Np;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.Qp = Qp; a.Kp = Kp; a.Vp = Vp; a.dOp = dOp;
  a.lse = lse; a.D = D;
  a.n_valid = n_valid; a.col_ptr = col_ptr; a.row_idx = row_idx;
  a.dQacc = dQacc; a.dKp = dKp; a.dVp = dVp;
  const size_t smem = 4ull * a.S * a.d * 2 + static_cast<size_t>(a.S) * (a.S + 1) * 4 +
                      2ull * a.S * 4;
  cudaError_t e = cudaFuncSetAttribute(simt_bwd_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long cols = static_cast<long long>(c.B) * c.H * p.sz.nb;
  simt_bwd_kernel<<<static_cast<unsigned>(cols), kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace prism
