// Block scores and hybrid Top-k / Top-p block selection, then the block
// lists in both directions (CSR: query block -> key blocks, CSC: key block
// -> query blocks).
//
// Prism (arXiv 2610.05416): block-level (pooled) features give a query-block x
// key-block score (Fig. 2 caption); Top-p(y) keeps the smallest set of key
// blocks whose cumulative attention weight exceeds y and Top-k keeps a fixed
// number (Table 7 caption); the hybrid rule sets the sparsity per query block
// (Abstract).  Reading used here: weights = softmax over the candidate key
// blocks (those with a real token) of s_ij = Qbar_i . Kbar_j / sqrt(d), ranked
// by (score desc, block index asc); keep m = max(min(k, n_cand), m_p) blocks,
// where m_p is the smallest prefix whose weight is strictly above p (all
// candidates when none is, or when p >= 1).
//
// Precision.  The block lists must not depend on rounding.  Scores are
// computed for every pair as double-float (hi + lo fp32 pairs) from the
// double-float block means by an error-free splitting of the product into
// exact integer digit products on the tensor cores (score_tc.cu), with an
// error near 2e-12 max|q| max|k|, below the block means' own.  The selection then runs on those scores with fp32 weights exp(s - max)
// (CUDA expf, 2 ulp) and compensated sums, so every cumulative weight carries
// an error below 4e-7.  A query block whose decision lies within 1e-6 of a
// boundary (cumulative weight near p, or a score gap at the cut) is decided
// again by an exact pass: full sort of the double-float scores and fp64
// weights and running sums.
#include <float.h>

#include "prism_internal.cuh"

namespace prism {
namespace {

// Order-preserving map of a float to uint32 (larger float -> larger key);
// every finite value maps to a key >= 1 so that 0 marks "no candidate".
__device__ __forceinline__ uint32_t fkey(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float fkey_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// ------------------------------------------------- fast selection ----------
constexpr int kEPL = 40;  // score elements held per lane

struct SelParams {
  int nb, nwords, topk;
  long long rows;  // B*H*nb
  float topp;
  df inv_sqrt_d;
  const float* Shi;
  const float* Slo;
  const int32_t* n_valid;
  uint32_t* bitmask;
  int32_t* rowcnt;
  uint8_t* tie;
  int32_t* amb;
  uint32_t* status;
};

// Reductions over the R warps that share one row.  Each call uses its own
// slot of a small ring so one named barrier per reduction suffices.
template <int R>
struct Group {
  int grp, wig, lane;
  float* scratch;  // 4 slots of R 32-bit words (a double-float uses two slots)
  int slot;
  __device__ __forceinline__ void sync() const {
    if (R > 1) asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(R * 32) : "memory");
  }
  template <class T, class Op>
  __device__ __forceinline__ T reduce(T v, Op op) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (R == 1) return v;
    T* s = reinterpret_cast<T*>(scratch) + slot * R;
    if (lane == 0) s[wig] = v;
    sync();
    T r = s[0];
#pragma unroll
    for (int w = 1; w < R; ++w) r = op(r, s[w]);
    slot = (slot + 1) & 3;
    return r;
  }
  __device__ __forceinline__ df reduce_df(df v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      df w;
      w.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
      w.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
      v = (lane & o) ? df_add(w, v) : df_add(v, w);  // lower lane first: deterministic
    }
    if (R == 1) return v;
    float* s = scratch + slot * R;  // slots slot and slot+1
    if (lane == 0) {
      s[2 * wig] = v.hi;
      s[2 * wig + 1] = v.lo;
    }
    sync();
    df r = {s[0], s[1]};
#pragma unroll
    for (int w = 1; w < R; ++w) r = df_add(r, df{s[2 * w], s[2 * w + 1]});
    slot = (slot + 2) & 3;
    return r;
  }
};

constexpr float kBand = 1e-6f;    // decision margin on cumulative weights
constexpr float kGapAbs = 1e-7f;  // decision margin on the score gap at the cut

// One row group (R warps) per query block.  Lane l of warp w holds the
// candidates j = w*32 + l + k*R*32, k < kEPL.
template <int R>
__global__ void __launch_bounds__(256) select_fast_kernel(SelParams P) {
  __shared__ float scratch_all[8][4 * 8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_per_cta = (blockDim.x >> 5) / R;
  Group<R> G;
  G.grp = warp / R;
  G.wig = warp % R;
  G.lane = lane;
  G.scratch = scratch_all[G.grp];
  G.slot = 0;
  const long long row = static_cast<long long>(blockIdx.x) * rows_per_cta + G.grp;
  if (row >= P.rows) return;  // the whole group leaves together
  const long long bh = row / P.nb;
  const int nb = P.nb;
  uint32_t* bm = P.bitmask + row * P.nwords;
  if (P.n_valid[row] == 0) {
    for (int w = G.wig * 32 + lane; w < P.nwords; w += R * 32) bm[w] = 0u;
    if (G.wig == 0 && lane == 0) {
      P.rowcnt[row] = 0;
      P.tie[row] = 0;
    }
    return;
  }
  // ---- the row: key of the hi part (0 = not a candidate), scaled scores ----
  const float* shr = P.Shi + row * nb;
  const float* slr = P.Slo + row * nb;
  const int32_t* nvk = P.n_valid + bh * nb;
  uint32_t key[kEPL];
  float sl[kEPL];  // lo part of the scaled score, later the weight
  float mx = -FLT_MAX;
  int ncand = 0;
#pragma unroll
  for (int k = 0; k < kEPL; ++k) {
    const int j = G.wig * 32 + lane + k * R * 32;
    key[k] = 0u;
    sl[k] = 0.f;
    if (j < nb && nvk[j] > 0) {
      const df s = df_mul(df{shr[j], slr[j]}, P.inv_sqrt_d);
      key[k] = fkey(s.hi);
      sl[k] = s.lo;
      mx = fmaxf(mx, s.hi);
      ++ncand;
    }
  }
  mx = G.reduce(mx, [](float a, float b) { return fmaxf(a, b); });
  ncand = G.reduce(ncand, [](int a, int b) { return a + b; });
  // weights e = exp(s - mx), s = hi + lo, error <= 2 ulp (expf) + O(u)
  df zl = {0.f, 0.f};
#pragma unroll
  for (int k = 0; k < kEPL; ++k) {
    if (key[k]) {
      const df x = two_sum(fkey_inv(key[k]), -mx);
      const float ex = expf(x.hi);
      sl[k] = fmaf(ex, __fadd_rn(x.lo, sl[k]), ex);
      zl = df_add(zl, df{sl[k], 0.f});
    } else {
      sl[k] = 0.f;
    }
  }
  float* e = sl;
  const df Z = G.reduce_df(zl);
  const float Zf = __fadd_rn(Z.hi, Z.lo);
  const int kf = min(P.topk, ncand);
  int m = ncand;
  uint32_t tau = 1u;  // select every candidate with key >= tau
  bool ambiguous = false;
  bool flag = false;
  if (!(P.topp >= 1.f) && kf < ncand) {
    const float target = P.topp * Zf;
    auto mass_ge = [&](uint32_t t) {
      float a = 0.f;
#pragma unroll
      for (int k = 0; k < kEPL; ++k) a += key[k] >= t ? e[k] : 0.f;
      return G.reduce(a, [](float x, float y) { return x + y; });
    };
    auto count_ge = [&](uint32_t t) {
      int a = 0;
#pragma unroll
      for (int k = 0; k < kEPL; ++k) a += (key[k] >= t && key[k]) ? 1 : 0;
      return G.reduce(a, [](int x, int y) { return x + y; });
    };
    uint32_t kmin = 0xffffffffu, kmx = 0u;
#pragma unroll
    for (int k = 0; k < kEPL; ++k)
      if (key[k]) {
        kmin = min(kmin, key[k]);
        kmx = max(kmx, key[k]);
      }
    kmin = G.reduce(kmin, [](uint32_t a, uint32_t b) { return min(a, b); });
    kmx = G.reduce(kmx, [](uint32_t a, uint32_t b) { return max(a, b); });
    // largest key tp with weight(key >= tp) > p * Z
    uint64_t lo = kmin, hi = static_cast<uint64_t>(kmx) + 1;
    while (hi - lo > 1) {
      const uint64_t mid = lo + ((hi - lo) >> 1);
      if (mass_ge(static_cast<uint32_t>(mid)) > target) lo = mid; else hi = mid;
    }
    uint32_t tsel = static_cast<uint32_t>(lo);
    int mp;
    float cum_prev, cum_at;
    {
      df egt_l = {0.f, 0.f};
      int cgt = 0, ceq = 0;
      float eeq = 0.f;
#pragma unroll
      for (int k = 0; k < kEPL; ++k) {
        if (!key[k]) continue;
        if (key[k] > tsel) {
          egt_l = df_add(egt_l, df{e[k], 0.f});
          ++cgt;
        } else if (key[k] == tsel) {
          ++ceq;
          eeq = e[k];
        }
      }
      const df Egt = G.reduce_df(egt_l);
      cgt = G.reduce(cgt, [](int a, int b) { return a + b; });
      ceq = G.reduce(ceq, [](int a, int b) { return a + b; });
      eeq = G.reduce(eeq, [](float a, float b) { return fmaxf(a, b); });
      if (ceq != 1) ambiguous = true;  // equal hi parts: order decided by lo / index
      mp = cgt + 1;
      const df at = df_add(Egt, df{eeq, 0.f});
      cum_prev = __fdiv_rn(__fadd_rn(Egt.hi, Egt.lo), Zf);
      cum_at = __fdiv_rn(__fadd_rn(at.hi, at.lo), Zf);
      if (!(cum_prev < P.topp - kBand)) ambiguous = true;
      if (mp < ncand && !(cum_at > P.topp + kBand)) ambiguous = true;
      flag = fabsf(cum_at - P.topp) <= 1e-6f || (mp >= 2 && fabsf(cum_prev - P.topp) <= 1e-6f);
    }
    if (mp < kf) {
      // the Top-k floor decides: largest key tk with count(key >= tk) >= kf
      uint64_t l2 = kmin, h2 = static_cast<uint64_t>(kmx) + 1;
      while (h2 - l2 > 1) {
        const uint64_t mid = l2 + ((h2 - l2) >> 1);
        if (count_ge(static_cast<uint32_t>(mid)) >= kf) l2 = mid; else h2 = mid;
      }
      tsel = static_cast<uint32_t>(l2);
      m = kf;
      // the Top-p count must stay below the floor: weight of the kf best > p
      df ek_l = {0.f, 0.f};
#pragma unroll
      for (int k = 0; k < kEPL; ++k)
        if (key[k] && key[k] >= tsel) ek_l = df_add(ek_l, df{e[k], 0.f});
      const df Ek = G.reduce_df(ek_l);
      if (!(__fdiv_rn(__fadd_rn(Ek.hi, Ek.lo), Zf) > P.topp + kBand)) ambiguous = true;
    } else {
      m = mp;
    }
    if (m < ncand) {
      // the cut: exactly m keys >= tsel, and a clear gap to the next score
      int cge = 0;
      uint32_t below = 0u;
      float lo_at = 0.f, lo_below = 0.f;
#pragma unroll
      for (int k = 0; k < kEPL; ++k) {
        if (!key[k]) continue;
        if (key[k] >= tsel) ++cge; else below = max(below, key[k]);
      }
      cge = G.reduce(cge, [](int a, int b) { return a + b; });
      below = G.reduce(below, [](uint32_t a, uint32_t b) { return max(a, b); });
      if (cge != m) ambiguous = true;
      const float s_at = fkey_inv(tsel), s_below = fkey_inv(below);
      (void)lo_at;
      (void)lo_below;
      const float gap = s_at - s_below;  // hi parts; lo parts are below 1e-7 of them
      if (!(gap > kGapAbs * fmaxf(1.f, fabsf(s_at)) + 2e-7f * fabsf(s_at))) ambiguous = true;
      flag |= gap <= 1e-6f * fmaxf(1.f, fabsf(s_at));
    }
    tau = tsel;
  }
  if (ambiguous) {
    if (G.wig == 0 && lane == 0) {
      const uint32_t slot = atomicAdd(P.status + WS_AMB_COUNT, 1u);
      P.amb[slot] = static_cast<int32_t>(row);
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < kEPL; ++k) {
    const int w = G.wig + k * R;
    const uint32_t bits = __ballot_sync(0xffffffffu, key[k] != 0u && key[k] >= tau);
    if (w < P.nwords && lane == 0) bm[w] = bits;
  }
  if (G.wig == 0 && lane == 0) {
    P.rowcnt[row] = m;
    P.tie[row] = flag ? 1 : 0;
  }
}

// ---------------------------------------------- exact fallback -------------
struct FbParams {
  int nb, nwords, topk, P2;
  float topp;
  df inv_sqrt_d;
  const float* Shi;
  const float* Slo;
  const int32_t* n_valid;
  uint32_t* bitmask;
  int32_t* rowcnt;
  uint8_t* tie;
  const int32_t* amb;
  uint32_t* status;
};

__device__ __forceinline__ uint64_t df_key(df s) {
  return (static_cast<uint64_t>(fkey(s.hi)) << 32) | fkey(s.lo);
}
__device__ __forceinline__ df df_key_inv(uint64_t k) {
  return {fkey_inv(static_cast<uint32_t>(k >> 32)), fkey_inv(static_cast<uint32_t>(k))};
}
__device__ __forceinline__ double df_to_d(df x) {
  return static_cast<double>(x.hi) + static_cast<double>(x.lo);
}

// One CTA per ambiguous row (grid-stride over the list): sort the candidates
// by (double-float score desc, index asc), fp64 weights exp(s - max) and
// their running sum in sorted order, the hybrid count, the bitmask.
// Smem: keys[P2] (u64), cum[P2] (fp64), idx[P2] (u32).
__global__ void __launch_bounds__(256) select_fallback_kernel(FbParams P) {
  extern __shared__ __align__(16) uint8_t sm[];
  uint64_t* keys = reinterpret_cast<uint64_t*>(sm);
  double* cum = reinterpret_cast<double*>(sm + 8ull * P.P2);
  uint32_t* idx = reinterpret_cast<uint32_t*>(sm + 16ull * P.P2);
  __shared__ double red[32];
  __shared__ int sh_nc, sh_mp;
  const uint32_t count = *reinterpret_cast<volatile uint32_t*>(P.status + WS_AMB_COUNT);
  const int nb = P.nb;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (uint32_t a = blockIdx.x; a < count; a += gridDim.x) {
    const long long row = P.amb[a];
    const long long bh = row / nb;
    const int32_t* nvk = P.n_valid + bh * nb;
    if (threadIdx.x == 0) sh_nc = 0;
    __syncthreads();
    int nc = 0;
    for (int j = threadIdx.x; j < P.P2; j += blockDim.x) {
      uint64_t kk = 0;  // not a candidate: sorts last
      if (j < nb && nvk[j] > 0) {
        const df s = df_mul(df{P.Shi[row * nb + j], P.Slo[row * nb + j]}, P.inv_sqrt_d);
        kk = df_key(s);
        ++nc;
      }
      keys[j] = kk;
      idx[j] = static_cast<uint32_t>(j);
    }
    for (int o = 16; o > 0; o >>= 1) nc += __shfl_xor_sync(0xffffffffu, nc, o);
    if (lane == 0) atomicAdd(&sh_nc, nc);
    __syncthreads();
    // bitonic sort: key descending, index ascending
    for (int k = 2; k <= P.P2; k <<= 1) {
      for (int jj = k >> 1; jj > 0; jj >>= 1) {
        for (int t = threadIdx.x; t < P.P2; t += blockDim.x) {
          const int o = t ^ jj;
          if (o > t) {
            const bool desc = (t & k) == 0;
            const uint64_t ka = keys[t], kb = keys[o];
            const uint32_t ia = idx[t], ib = idx[o];
            const bool a_first = ka > kb || (ka == kb && ia < ib);
            if (a_first != desc) {
              keys[t] = kb;
              keys[o] = ka;
              idx[t] = ib;
              idx[o] = ia;
            }
          }
        }
        __syncthreads();
      }
    }
    const int ncand = sh_nc;
    const double smax = df_to_d(df_key_inv(keys[0]));
    for (int j = threadIdx.x; j < P.P2; j += blockDim.x)
      cum[j] = j < ncand ? exp(df_to_d(df_key_inv(keys[j])) - smax) : 0.0;
    __syncthreads();
    {
      // running sum in sorted order: per-thread runs, then a scan of the runs
      const int per = P.P2 / blockDim.x;
      const int b0 = threadIdx.x * per;
      double run = 0.0;
      for (int q = 0; q < per; ++q) {
        run += cum[b0 + q];
        cum[b0 + q] = run;
      }
      double incl = run;
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) red[warp] = incl;
      __syncthreads();
      if (threadIdx.x == 0) {
        double acc = 0.0;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
          const double t = red[w];
          red[w] = acc;
          acc += t;
        }
      }
      __syncthreads();
      const double off = red[warp] + (incl - run);
      for (int q = 0; q < per; ++q) cum[b0 + q] += off;
    }
    if (threadIdx.x == 0) sh_mp = ncand;
    __syncthreads();
    const double Zt = cum[ncand - 1];
    const double p = P.topp;
    if (!(P.topp >= 1.f)) {
      // smallest m with cum_m / Z > p (1-based)
      for (int j = threadIdx.x; j < ncand; j += blockDim.x) {
        const bool over = cum[j] / Zt > p;
        const bool prev_over = j > 0 && cum[j - 1] / Zt > p;
        if (over && !prev_over) atomicMin(&sh_mp, j + 1);
      }
    }
    __syncthreads();
    const int mp = sh_mp;
    const int m = max(min(P.topk, ncand), mp);
    uint32_t* bm = P.bitmask + row * P.nwords;
    for (int w = threadIdx.x; w < P.nwords; w += blockDim.x) bm[w] = 0u;
    __syncthreads();
    for (int j = threadIdx.x; j < m; j += blockDim.x) atomicOr(bm + (idx[j] >> 5), 1u << (idx[j] & 31));
    if (threadIdx.x == 0) {
      P.rowcnt[row] = m;
      bool flag = false;
      if (m < ncand) {
        const double sa = df_to_d(df_key_inv(keys[m - 1])), sb = df_to_d(df_key_inv(keys[m]));
        flag |= fabs(sa - sb) <= 1e-6 * fmax(1.0, fabs(sa));
      }
      flag |= fabs(cum[mp - 1] / Zt - p) <= 1e-6;
      if (mp >= 2) flag |= fabs(cum[mp - 2] / Zt - p) <= 1e-6;
      P.tie[row] = flag ? 1 : 0;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------- list building --------
// Exclusive scan of cnt[0..n) into ptr[0..n]; one CTA of 1024 threads.
__global__ void __launch_bounds__(1024) scan_kernel(long long n, const int32_t* __restrict__ cnt,
                                                    int32_t* __restrict__ ptr) {
  __shared__ int32_t part[1024];
  const long long per = (n + blockDim.x - 1) / blockDim.x;
  const long long b0 = threadIdx.x * per;
  int32_t s = 0;
  for (long long q = 0; q < per && b0 + q < n; ++q) s += cnt[b0 + q];
  part[threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t acc = 0;
    for (int t = 0; t < static_cast<int>(blockDim.x); ++t) {
      const int32_t v = part[t];
      part[t] = acc;
      acc += v;
    }
    ptr[n] = acc;
  }
  __syncthreads();
  int32_t acc = part[threadIdx.x];
  for (long long q = 0; q < per && b0 + q < n; ++q) {
    ptr[b0 + q] = acc;
    acc += cnt[b0 + q];
  }
}

// CSR: one warp per query block, expanding its bitmask in ascending order.
__global__ void csr_fill_kernel(long long rows, int nwords, const uint32_t* __restrict__ bitmask,
                                const int32_t* __restrict__ row_ptr, int32_t* __restrict__ col_idx) {
  const int lane = threadIdx.x & 31;
  const long long row = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  if (row >= rows) return;
  const uint32_t* bm = bitmask + row * nwords;
  int base = row_ptr[row];
  for (int w0 = 0; w0 < nwords; w0 += 32) {
    const int w = w0 + lane;
    const uint32_t bits = w < nwords ? bm[w] : 0u;
    const int c = __popc(bits);
    int incl = c;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int pos = base + incl - c;
    uint32_t b = bits;
    while (b) {
      const int bit = __ffs(b) - 1;
      col_idx[pos++] = w * 32 + bit;
      b &= b - 1;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// CSC counts / fill: one warp per (b, h, 32-column word), lanes = columns,
// rows visited in ascending order.
__global__ void csc_count_kernel(int nb, int nwords, long long units,
                                 const uint32_t* __restrict__ bitmask, int32_t* __restrict__ cnt) {
  const int lane = threadIdx.x & 31;
  const long long u = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  if (u >= units) return;
  const long long bh = u / nwords;
  const int w = static_cast<int>(u % nwords);
  const uint32_t* bm = bitmask + bh * nb * static_cast<long long>(nwords) + w;
  int c = 0;
  for (int i = 0; i < nb; ++i) c += (bm[static_cast<long long>(i) * nwords] >> lane) & 1u;
  const int j = w * 32 + lane;
  if (j < nb) cnt[bh * nb + j] = c;
}

__global__ void csc_fill_kernel(int nb, int nwords, long long units,
                                const uint32_t* __restrict__ bitmask,
                                const int32_t* __restrict__ col_ptr, int32_t* __restrict__ row_idx) {
  const int lane = threadIdx.x & 31;
  const long long u = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  if (u >= units) return;
  const long long bh = u / nwords;
  const int w = static_cast<int>(u % nwords);
  const int j = w * 32 + lane;
  const uint32_t* bm = bitmask + bh * nb * static_cast<long long>(nwords) + w;
  int pos = j < nb ? col_ptr[bh * nb + j] : 0;
  for (int i = 0; i < nb; ++i) {
    const uint32_t word = bm[static_cast<long long>(i) * nwords];
    if (j < nb && ((word >> lane) & 1u)) row_idx[pos++] = i;
  }
}

// ------------------------------------------------- multi-tile blocks -----
// Block table from the zones' shapes: for every tile, the first tile of its
// block, and at a block's first tile the block's real-token count (the sum
// of its tiles' counts; 0 on the tiles that continue a block).
struct ShapeTokens {
  int32_t t[PRISM_MAX_SHAPES];  // token count of every menu shape
};

__global__ void block_table_kernel(long long rows, int nu, int upz, int Z, int U, int T,
                                   ShapeTokens ext_tokens,
                                   const uint8_t* __restrict__ shape_id,
                                   const int32_t* __restrict__ n_valid,
                                   int32_t* __restrict__ n_sel, int32_t* __restrict__ bstart) {
  // units of U slots (a tile, or half a tile); rows = B*H*nu
  const long long r = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (r >= rows) return;
  const long long bh = r / nu;
  const int u = static_cast<int>(r % nu);
  const int z = u / upz, lu = u % upz;
  const int sid = shape_id[bh * Z + z];
  const int SB = sid < PRISM_MAX_SHAPES ? ext_tokens.t[sid] : T;
  const int upb = max(1, SB / U);
  const int first = u - lu % upb;
  bstart[r] = first;
  int nv = 0;
  if (first == u) {
    const int nt = nu / (T / U);                      // tiles per (b, h)
    const long long t0 = bh * nt + static_cast<long long>(u) * U / T;
    if (SB >= T) {
      for (int q = 0; q < SB / T; ++q) nv += n_valid[t0 + q];
    } else {  // half a tile: this block's part of its tile's real tokens
      const int hb = (u * U) % T / SB;
      nv = min(SB, max(0, n_valid[t0] - hb * SB));
    }
  }
  n_sel[r] = nv;
}

// Tile-level selection: tile u is selected for tile t when some block of t
// (one, or two of half a tile each) selected some block of u.  One thread
// per (tile row, 32-tile word); also the row's count.  per = table units per
// tile (1 or 2); bm_unit is the selection bitmask over units (uwords words
// per row), bstart the first unit of every unit's block.
__device__ __forceinline__ uint32_t pair_bits(const uint32_t* __restrict__ bm_unit, int uwords,
                                              const int32_t* __restrict__ bs, long long bh, int nu,
                                              int per, int qt, int kt) {
  uint32_t bits = 0u;
  for (int qh = 0; qh < per; ++qh) {
    const long long row = bh * nu + bs[qt * per + qh];
    const uint32_t* src = bm_unit + row * uwords;
    for (int kh = 0; kh < per; ++kh) {
      const int j = bs[kt * per + kh];
      bits |= ((src[j >> 5] >> (j & 31)) & 1u) << (qh * per + kh);
    }
  }
  return bits;
}

__global__ void expand_bitmask_kernel(long long rows, int nb, int nwords, int nu, int uwords,
                                      int per, const uint32_t* __restrict__ bm_unit,
                                      const int32_t* __restrict__ bstart,
                                      uint32_t* __restrict__ bm_tile,
                                      int32_t* __restrict__ rowcnt) {
  const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  const long long r = i / 32;
  const int lane = static_cast<int>(i % 32);
  if (r >= rows) return;
  const long long bh = r / nb;
  const int t = static_cast<int>(r % nb);
  const int32_t* bs = bstart + bh * nu;
  int cnt = 0;
  for (int w = lane; w < nwords; w += 32) {
    uint32_t out = 0u;
    for (int k = 0; k < 32; ++k) {
      const int u = w * 32 + k;
      if (u >= nb) break;
      out |= (pair_bits(bm_unit, uwords, bs, bh, nu, per, t, u) != 0u ? 1u : 0u) << k;
    }
    bm_tile[r * nwords + w] = out;
    cnt += __popc(out);
  }
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if (lane == 0) rowcnt[r] = cnt;
}

// Sub-tile masks of the tile lists (blocks of half a tile): for every entry
// of the CSR (rows = query tiles) or CSC (rows = key tiles) lists, bit
// 2 qh + kh set when the query tile's half qh does not attend the key tile's
// half kh.  One warp per row, lanes over its entries.
__global__ void list_mask_kernel(long long rows, int nb, int nu, int uwords, int per, int csc,
                                 const int32_t* __restrict__ ptr, const int32_t* __restrict__ idx,
                                 const uint32_t* __restrict__ bm_unit,
                                 const int32_t* __restrict__ bstart, uint8_t* __restrict__ mask) {
  const long long r = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const long long bh = r / nb;
  const int me = static_cast<int>(r % nb);
  const int32_t* bs = bstart + bh * nu;
  const uint32_t full = (1u << (per * per)) - 1u;
  for (int e = ptr[r] + lane; e < ptr[r + 1]; e += 32) {
    const int other = idx[e];
    const uint32_t bits = csc ? pair_bits(bm_unit, uwords, bs, bh, nu, per, other, me)
                              : pair_bits(bm_unit, uwords, bs, bh, nu, per, me, other);
    mask[e] = static_cast<uint8_t>(~bits & full);
  }
}

}  // namespace

cudaError_t launch_select(const Plan& p, const uint8_t* shape_id, const float* Qh,
                          const float* Ql, const float* Kh, const float* Kl,
                          const int32_t* n_valid, uint8_t* sel_tie,
                          int32_t* row_ptr, int32_t* col_idx, int32_t* col_ptr,
                          int32_t* row_idx, uint8_t* ws, cudaStream_t st,
                          cudaEvent_t score_begin, cudaEvent_t score_end) {
  const prism_config_t& c = p.cfg;
  // the selection runs over the block table's units (tiles, or half tiles);
  // the lists handed on are over tiles
  const int nt = p.sz.nb;
  const long long trows = static_cast<long long>(c.B) * c.H * nt;
  const int twords = (nt + 31) / 32;
  const int nb = p.sz.nslots;
  const long long rows = static_cast<long long>(c.B) * c.H * nb;
  const int nwords = (nb + 31) / 32;
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float* Shi = reinterpret_cast<float*>(ws + p.off_scores);
  float* Slo = Shi + rows * nb;
  uint32_t* bitmask = reinterpret_cast<uint32_t*>(ws + p.off_bitmask);
  int32_t* rowcnt = reinterpret_cast<int32_t*>(ws + p.off_rowcnt);
  int32_t* colcnt = reinterpret_cast<int32_t*>(ws + p.off_colcnt);
  int32_t* amb = reinterpret_cast<int32_t*>(ws + p.off_amb);
  const double isd = 1.0 / sqrt(static_cast<double>(c.d));
  df isd_df;
  isd_df.hi = static_cast<float>(isd);
  isd_df.lo = static_cast<float>(isd - static_cast<double>(isd_df.hi));
  cudaError_t e = cudaMemsetAsync(status + WS_AMB_COUNT, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  int32_t* bstart = reinterpret_cast<int32_t*>(ws + p.off_bstart);
  const int per = c.block_tokens / p.sz.slot_tokens;  // table units per tile
  if (p.sz.multi_tile) {
    // blocks span several tiles or share one: select over blocks (their first
    // units), with each block's real-token count in place of the tile counts
    ShapeTokens ext;
    for (int k = 0; k < PRISM_MAX_SHAPES; ++k)
      ext.t[k] = k < c.n_shapes ? c.shapes[k][0] * c.shapes[k][1] * c.shapes[k][2] : c.block_tokens;
    int32_t* n_sel = reinterpret_cast<int32_t*>(ws + p.off_nsel);
    block_table_kernel<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, st>>>(
        rows, nb, c.zT * c.zH * c.zW / p.sz.slot_tokens, p.sz.Z, p.sz.slot_tokens,
        c.block_tokens, ext, shape_id, n_valid, n_sel, bstart);
    n_valid = n_sel;
  }
  // optional timing marks around the score kernels alone
  if (score_begin != nullptr && (e = cudaEventRecord(score_begin, st)) != cudaSuccess) return e;
  if ((e = launch_score_tc(p, Qh, Ql, Kh, Kl, Shi, Slo, ws, st)) != cudaSuccess) return e;
  if (score_end != nullptr && (e = cudaEventRecord(score_end, st)) != cudaSuccess) return e;
  SelParams sp;
  sp.nb = nb;
  sp.nwords = nwords;
  sp.topk = c.topk_floor;
  sp.rows = rows;
  sp.topp = c.topp;
  sp.inv_sqrt_d = isd_df;
  sp.Shi = Shi;
  sp.Slo = Slo;
  sp.n_valid = n_valid;
  sp.bitmask = bitmask;
  sp.rowcnt = rowcnt;
  sp.tie = sel_tie;
  sp.amb = amb;
  sp.status = status;
  const int R = (nb + 32 * kEPL - 1) / (32 * kEPL);
  const int rpc = 8 / (R <= 1 ? 1 : R <= 2 ? 2 : R <= 4 ? 4 : 8);
  const unsigned gsel = static_cast<unsigned>((rows + rpc - 1) / rpc);
  if (R <= 1) select_fast_kernel<1><<<gsel, 256, 0, st>>>(sp);
  else if (R <= 2) select_fast_kernel<2><<<gsel, 256, 0, st>>>(sp);
  else if (R <= 4) select_fast_kernel<4><<<gsel, 256, 0, st>>>(sp);
  else select_fast_kernel<8><<<gsel, 256, 0, st>>>(sp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  FbParams fp;
  fp.nb = nb;
  fp.nwords = nwords;
  fp.topk = c.topk_floor;
  int P2 = 256;
  while (P2 < nb) P2 <<= 1;
  fp.P2 = P2;
  fp.topp = c.topp;
  fp.inv_sqrt_d = isd_df;
  fp.Shi = Shi;
  fp.Slo = Slo;
  fp.n_valid = n_valid;
  fp.bitmask = bitmask;
  fp.rowcnt = rowcnt;
  fp.tie = sel_tie;
  fp.amb = amb;
  fp.status = status;
  const size_t fsm = 20ull * P2;
  e = cudaFuncSetAttribute(select_fallback_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(fsm));
  if (e != cudaSuccess) return e;
  select_fallback_kernel<<<296, 256, fsm, st>>>(fp);
  uint32_t* bm_unit = bitmask;
  if (p.sz.multi_tile) {
    // block lists -> tile lists: every tile of a query block gets every tile
    // of every key block its block selected
    uint32_t* tbm = reinterpret_cast<uint32_t*>(ws + p.off_tbitmask);
    expand_bitmask_kernel<<<static_cast<unsigned>((trows * 32 + 255) / 256), 256, 0, st>>>(
        trows, nt, twords, nb, nwords, per, bitmask, bstart, tbm, rowcnt);
    bitmask = tbm;
  }
  scan_kernel<<<1, 1024, 0, st>>>(trows, rowcnt, row_ptr);
  csr_fill_kernel<<<static_cast<unsigned>((trows * 32 + 255) / 256), 256, 0, st>>>(
      trows, twords, bitmask, row_ptr, col_idx);
  const long long units = static_cast<long long>(c.B) * c.H * twords;
  csc_count_kernel<<<static_cast<unsigned>((units * 32 + 255) / 256), 256, 0, st>>>(
      nt, twords, units, bitmask, colcnt);
  scan_kernel<<<1, 1024, 0, st>>>(trows, colcnt, col_ptr);
  csc_fill_kernel<<<static_cast<unsigned>((units * 32 + 255) / 256), 256, 0, st>>>(
      nt, twords, units, bitmask, col_ptr, row_idx);
  if (p.sz.half_tile) {
    uint8_t* mcsr = ws + p.sz.ws_csr_mask;
    uint8_t* mcsc = ws + p.sz.ws_csc_mask;
    const unsigned gm = static_cast<unsigned>((trows * 32 + 255) / 256);
    list_mask_kernel<<<gm, 256, 0, st>>>(trows, nt, nb, nwords, per, 0, row_ptr, col_idx, bm_unit,
                                         bstart, mcsr);
    list_mask_kernel<<<gm, 256, 0, st>>>(trows, nt, nb, nwords, per, 1, col_ptr, row_idx, bm_unit,
                                         bstart, mcsc);
  }
  return cudaGetLastError();
}

}  // namespace prism
