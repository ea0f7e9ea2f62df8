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
// Precision.  The block lists must not depend on rounding, so the decision is
// certified: the fast path computes fp32 scores (tiled SGEMM) and runs the
// selection on them, together with a rigorous bound delta on the score error
// ((d + 5) u ||q|| ||k_max|| / sqrt(d), u = 2^-24).  A row whose decision sits
// within that bound of a boundary (score gap at the cut, or cumulative mass
// near p) is re-done from the double-float block means (hi + lo fp32 pairs)
// with compensated (Dot2, Ogita-Rump-Oishi 2005) scores accurate to ~1e-13, a
// full sort and an fp64 cumulative sum -- the same decision as an fp64 reading.
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

// ------------------------------------------------------------- norms -------
__global__ void norms_kernel(long long rows, int d, const float* __restrict__ Qb,
                             const float* __restrict__ Kb, float* __restrict__ qn,
                             float* __restrict__ kn) {
  const int lane = threadIdx.x & 31;
  const long long w = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  if (w >= 2 * rows) return;
  const float* src = w < rows ? Qb + w * d : Kb + (w - rows) * d;
  float s = 0.f;
  for (int c = lane; c < d; c += 32) s = fmaf(src[c], src[c], s);
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) {
    // round the norm up a little so that it bounds the exact norm
    const float r = sqrtf(s) * (1.f + 1e-6f);
    if (w < rows) qn[w] = r; else kn[w - rows] = r;
  }
}

// ---------------------------------------------------- score SGEMM ----------
// S[bh][i][j] = sum_c Q[bh][i][c] * K[bh][j][c] in fp32 (ragged edges zero
// filled).  128 x 128 tile per CTA, 256 threads with an 8 x 8 register tile
// each, K-dimension staged 16 channels at a time (transposed in smem).
constexpr int kTile = 128, kBK = 16;

__global__ void __launch_bounds__(256) score_gemm_kernel(int nb, int d,
                                                         const float* __restrict__ Qb,
                                                         const float* __restrict__ Kb,
                                                         float* __restrict__ S) {
  __shared__ __align__(16) float As[kBK][kTile + 4];
  __shared__ __align__(16) float Bs[kBK][kTile + 4];
  const int bh = blockIdx.z;
  const int i0 = blockIdx.y * kTile, j0 = blockIdx.x * kTile;
  const float* A = Qb + static_cast<long long>(bh) * nb * d;
  const float* B = Kb + static_cast<long long>(bh) * nb * d;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[8][8];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
  for (int c0 = 0; c0 < d; c0 += kBK) {
    // 128 rows x 16 channels per operand = 2048 floats, 8 per thread
    for (int e = threadIdx.x; e < kTile * kBK; e += 256) {
      const int r = e / kBK, cc = e % kBK;
      const int gi = i0 + r, gj = j0 + r, c = c0 + cc;
      As[cc][r] = (gi < nb && c < d) ? A[static_cast<long long>(gi) * d + c] : 0.f;
      Bs[cc][r] = (gj < nb && c < d) ? B[static_cast<long long>(gj) * d + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int cc = 0; cc < kBK; ++cc) {
      float a[8], b[8];
      const float4 a0 = *reinterpret_cast<const float4*>(&As[cc][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[cc][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[cc][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[cc][64 + tx * 4]);
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
      a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
      b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int x = 0; x < 8; ++x)
#pragma unroll
        for (int y = 0; y < 8; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
    }
    __syncthreads();
  }
  float* out = S + static_cast<long long>(bh) * nb * nb;
#pragma unroll
  for (int x = 0; x < 8; ++x) {
    const int gi = i0 + (x < 4 ? ty * 4 + x : 64 + ty * 4 + x - 4);
    if (gi >= nb) continue;
#pragma unroll
    for (int y = 0; y < 8; ++y) {
      const int gj = j0 + (y < 4 ? tx * 4 + y : 64 + tx * 4 + y - 4);
      if (gj < nb) out[static_cast<long long>(gi) * nb + gj] = acc[x][y];
    }
  }
}

// ------------------------------------------------- fast selection ----------
constexpr int kEPL = 40;  // score elements held per lane

struct SelParams {
  int nb, nwords, d, topk;
  long long rows;  // B*H*nb
  float topp, inv_sqrt_d, u_scale;
  const float* S;
  const int32_t* n_valid;
  const float* qn;
  const float* kn;
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
  float* scratch;  // [R * 4] floats (viewed as any 32-bit type)
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
      // combine in a fixed lane-independent order: lower lane first
      v = (lane & o) ? df_add(w, v) : df_add(v, w);
    }
    if (R == 1) return v;
    float* s = scratch + slot * R * 2;  // uses two slots
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

template <int R>
__global__ void __launch_bounds__(256) select_fast_kernel(SelParams P) {
  __shared__ float scratch_all[8][4 * 8 * 2];
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
  const int nv_i = P.n_valid[row];
  if (nv_i == 0) {
    for (int w = G.wig * 32 + lane; w < P.nwords; w += R * 32) bm[w] = 0u;
    if (G.wig == 0 && lane == 0) {
      P.rowcnt[row] = 0;
      P.tie[row] = 0;
    }
    return;
  }
  // ---- load the row: key (0 = not a candidate), value, weight ----
  const float* srow = P.S + row * nb;
  const int32_t* nvk = P.n_valid + bh * nb;
  const float* knr = P.kn + bh * nb;
  uint32_t key[kEPL];
  float e[kEPL];
  float mx = -FLT_MAX, kmax = 0.f;
  int ncand = 0;
#pragma unroll
  for (int k = 0; k < kEPL; ++k) {
    const int j = G.wig * 32 + lane + k * R * 32;
    key[k] = 0u;
    e[k] = 0.f;
    if (j < nb && nvk[j] > 0) {
      const float s = __fmul_rn(srow[j], P.inv_sqrt_d);
      key[k] = fkey(s);
      e[k] = s;
      mx = fmaxf(mx, s);
      kmax = fmaxf(kmax, knr[j]);
      ++ncand;
    }
  }
  mx = G.reduce(mx, [](float a, float b) { return fmaxf(a, b); });
  kmax = G.reduce(kmax, [](float a, float b) { return fmaxf(a, b); });
  ncand = G.reduce(ncand, [](int a, int b) { return a + b; });
  df zl = {0.f, 0.f};
#pragma unroll
  for (int k = 0; k < kEPL; ++k) {
    if (key[k]) {
      e[k] = expf(e[k] - mx);
      zl = df_add(zl, df{e[k], 0.f});
    }
  }
  const df Z = G.reduce_df(zl);
  const float Zf = Z.hi + Z.lo;
  const int kf = min(P.topk, ncand);
  int m = ncand;
  uint32_t tau = 1u;  // select every candidate key >= tau
  bool ambiguous = false;
  bool flag = false;
  if (!(P.topp >= 1.f) && kf < ncand) {
    // certified error of an fp32 score and of a cumulative weight
    const float delta = P.u_scale * P.qn[row] * kmax;
    const float band = 2.1f * delta + 16.f * 5.9604645e-8f;
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
    // largest key tp with mass(key >= tp) > target
    uint64_t lo = kmin, hi = static_cast<uint64_t>(kmx) + 1;
    while (hi - lo > 1) {
      const uint64_t mid = lo + ((hi - lo) >> 1);
      if (mass_ge(static_cast<uint32_t>(mid)) > target) lo = mid; else hi = mid;
    }
    const uint32_t tp = static_cast<uint32_t>(lo);
    // exact pieces around tp: compensated mass above, tie count, neighbours
    df egt_l = {0.f, 0.f};
    int cgt = 0, ceq = 0;
    uint32_t above = 0xffffffffu, below = 0u;
#pragma unroll
    for (int k = 0; k < kEPL; ++k) {
      if (!key[k]) continue;
      if (key[k] > tp) {
        egt_l = df_add(egt_l, df{e[k], 0.f});
        ++cgt;
        above = min(above, key[k]);
      } else if (key[k] == tp) {
        ++ceq;
      } else {
        below = max(below, key[k]);
      }
    }
    const df Egt = G.reduce_df(egt_l);
    cgt = G.reduce(cgt, [](int a, int b) { return a + b; });
    ceq = G.reduce(ceq, [](int a, int b) { return a + b; });
    above = G.reduce(above, [](uint32_t a, uint32_t b) { return min(a, b); });
    below = G.reduce(below, [](uint32_t a, uint32_t b) { return max(a, b); });
    const float stp = fkey_inv(tp);
    const float etp = expf(stp - mx);
    const float egt = Egt.hi + Egt.lo;
    int t = 1;
    while (t < ceq && egt + t * etp <= target) ++t;
    const int mp = cgt + t;
    const float cum_prev = (egt + (t - 1) * etp) / Zf;
    const float cum_at = (egt + t * etp) / Zf;
    const float s_above = above != 0xffffffffu ? fkey_inv(above) : 0.f;
    const float s_below = below ? fkey_inv(below) : 0.f;
    if (mp >= kf) {
      m = mp;
      tau = tp;
      // the cut must not split ties, and must clear the error bound on
      // both sides of the Top-p count and on the mass
      if (t < ceq) ambiguous = true;
      if (mp < ncand && !(stp - s_below > 2.f * delta)) ambiguous = true;
      if (mp >= 2 && (t >= 2 || !(s_above - stp > 2.f * delta))) ambiguous = true;
      if (!(cum_prev < P.topp - band)) ambiguous = true;
      if (mp < ncand && !(cum_at > P.topp + band)) ambiguous = true;
      flag = (mp < ncand && stp - s_below <= 1e-6f * fmaxf(1.f, fabsf(stp))) ||
             fabsf(cum_at - P.topp) <= 1e-6f || (mp >= 2 && fabsf(cum_prev - P.topp) <= 1e-6f);
    } else {
      // the Top-k floor decides: largest key tk with count(key >= tk) >= kf
      uint64_t l2 = kmin, h2 = static_cast<uint64_t>(kmx) + 1;
      while (h2 - l2 > 1) {
        const uint64_t mid = l2 + ((h2 - l2) >> 1);
        if (count_ge(static_cast<uint32_t>(mid)) >= kf) l2 = mid; else h2 = mid;
      }
      const uint32_t tk = static_cast<uint32_t>(l2);
      df ek_l = {0.f, 0.f};
      int cge = 0;
      uint32_t bel = 0u;
#pragma unroll
      for (int k = 0; k < kEPL; ++k) {
        if (!key[k]) continue;
        if (key[k] >= tk) {
          ek_l = df_add(ek_l, df{e[k], 0.f});
          ++cge;
        } else {
          bel = max(bel, key[k]);
        }
      }
      const df Ek = G.reduce_df(ek_l);
      cge = G.reduce(cge, [](int a, int b) { return a + b; });
      bel = G.reduce(bel, [](uint32_t a, uint32_t b) { return max(a, b); });
      m = kf;
      tau = tk;
      const float stk = fkey_inv(tk);
      const float sbel = bel ? fkey_inv(bel) : 0.f;
      const float cumk = (Ek.hi + Ek.lo) / Zf;
      if (cge != kf) ambiguous = true;  // ties straddle the cut
      if (!(stk - sbel > 2.f * delta)) ambiguous = true;
      if (!(cumk > P.topp + band)) ambiguous = true;
      flag = (stk - sbel <= 1e-6f * fmaxf(1.f, fabsf(stk))) ||
             fabsf(cum_at - P.topp) <= 1e-6f || (mp >= 2 && fabsf(cum_prev - P.topp) <= 1e-6f);
    }
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
  int nb, nwords, d, topk, P2;
  float topp;
  df inv_sqrt_d;
  const float* Qh;
  const float* Ql;
  const float* Kh;
  const float* Kl;
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

// One CTA per ambiguous row (grid-stride over the list).  Smem: keys[P2]
// (u64, descending order wanted), idx[P2] (u32), cum[P2] (fp64 weights, then
// their running sum), the query's double-float mean.
__global__ void __launch_bounds__(256) select_fallback_kernel(FbParams P) {
  extern __shared__ __align__(16) uint8_t sm[];
  uint64_t* keys = reinterpret_cast<uint64_t*>(sm);
  double* cum = reinterpret_cast<double*>(sm + 8ull * P.P2);
  uint32_t* idx = reinterpret_cast<uint32_t*>(sm + 16ull * P.P2);
  float* qh = reinterpret_cast<float*>(sm + 20ull * P.P2);
  float* ql = qh + P.d;
  __shared__ double red[32];
  __shared__ int sh_m, sh_mp;
  const uint32_t count = *reinterpret_cast<volatile uint32_t*>(P.status + WS_AMB_COUNT);
  const int nb = P.nb;
  for (uint32_t a = blockIdx.x; a < count; a += gridDim.x) {
    const long long row = P.amb[a];
    const long long bh = row / nb;
    for (int c = threadIdx.x; c < P.d; c += blockDim.x) {
      qh[c] = P.Qh[row * P.d + c];
      ql[c] = P.Ql[row * P.d + c];
    }
    __syncthreads();
    const int32_t* nvk = P.n_valid + bh * nb;
    // Dot2 scores of all candidates, as sortable keys
    for (int j = threadIdx.x; j < P.P2; j += blockDim.x) {
      uint64_t kk = 0;  // not a candidate: sorts last
      if (j < nb && nvk[j] > 0) {
        const float* kh = P.Kh + (bh * nb + j) * P.d;
        const float* kl = P.Kl + (bh * nb + j) * P.d;
        float s = 0.f, c = 0.f;
        for (int q = 0; q < P.d; ++q) {
          const float p = __fmul_rn(qh[q], kh[q]);
          const float pe = fmaf(qh[q], kh[q], -p);
          const float cross = fmaf(qh[q], kl[q], __fmul_rn(ql[q], kh[q]));
          const df t = two_sum(s, p);
          s = t.hi;
          c = __fadd_rn(c, __fadd_rn(t.lo, __fadd_rn(pe, cross)));
        }
        const df dot = fast_two_sum(s, c);
        kk = df_key(df_mul(dot, P.inv_sqrt_d));
      }
      keys[j] = kk;
      idx[j] = static_cast<uint32_t>(j);
    }
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
              keys[t] = kb; keys[o] = ka;
              idx[t] = ib; idx[o] = ia;
            }
          }
        }
        __syncthreads();
      }
    }
    // weights exp(s - max) in fp64, then the running sum in sorted order
    const df smax = df_key_inv(keys[0]);
    for (int j = threadIdx.x; j < P.P2; j += blockDim.x) {
      double w = 0.0;
      if (keys[j]) {
        const df x = df_add(df_key_inv(keys[j]), df_neg(smax));
        float ex = expf(x.hi);
        ex = fmaf(ex, x.lo, ex);
        w = static_cast<double>(ex);
      }
      cum[j] = w;
    }
    __syncthreads();
    {
      const int per = P.P2 / blockDim.x;  // P2 is a multiple of blockDim
      const int b0 = threadIdx.x * per;
      double run = 0.0;
      for (int q = 0; q < per; ++q) {
        run += cum[b0 + q];
        cum[b0 + q] = run;
      }
      // exclusive scan of the per-thread totals (warp shuffles + smem)
      double incl = run;
      const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
    __syncthreads();
    int ncand = 0;
    for (int j = threadIdx.x; j < nb; j += blockDim.x) ncand += nvk[j] > 0 ? 1 : 0;
    for (int o = 16; o > 0; o >>= 1) ncand += __shfl_xor_sync(0xffffffffu, ncand, o);
    if (threadIdx.x == 0) sh_mp = ncand;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) atomicAdd(&sh_m, 0);  // keep sh_m live
    __shared__ int ncand_s;
    if (threadIdx.x == 0) ncand_s = 0;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) atomicAdd(&ncand_s, ncand);
    __syncthreads();
    const int nc = ncand_s;
    const double Zt = cum[nc - 1];
    if (threadIdx.x == 0) sh_mp = nc;
    __syncthreads();
    if (!(P.topp >= 1.f)) {
      // smallest m with cum_m / Z > p (1-based)
      for (int j = threadIdx.x; j < nc; j += blockDim.x) {
        const bool over = cum[j] / Zt > static_cast<double>(P.topp);
        const bool prev_over = j > 0 && cum[j - 1] / Zt > static_cast<double>(P.topp);
        if (over && !prev_over) atomicMin(&sh_mp, j + 1);
      }
    }
    __syncthreads();
    const int mp = sh_mp;
    const int m = max(min(P.topk, nc), mp);
    uint32_t* bm = P.bitmask + row * P.nwords;
    for (int w = threadIdx.x; w < P.nwords; w += blockDim.x) bm[w] = 0u;
    __syncthreads();
    for (int j = threadIdx.x; j < m; j += blockDim.x) atomicOr(bm + (idx[j] >> 5), 1u << (idx[j] & 31));
    if (threadIdx.x == 0) {
      P.rowcnt[row] = m;
      bool flag = false;
      if (m < nc) {
        const df a = df_key_inv(keys[m - 1]), b = df_key_inv(keys[m]);
        const double sa = static_cast<double>(a.hi) + a.lo, sb = static_cast<double>(b.hi) + b.lo;
        flag |= fabs(sa - sb) <= 1e-6 * fmax(1.0, fabs(sa));
      }
      const double p = P.topp;
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

}  // namespace

cudaError_t launch_select(const Plan& p, const float* Qh, const float* Ql, const float* Kh,
                          const float* Kl, const int32_t* n_valid, uint8_t* sel_tie,
                          int32_t* row_ptr, int32_t* col_idx, int32_t* col_ptr,
                          int32_t* row_idx, uint8_t* ws, cudaStream_t st) {
  const prism_config_t& c = p.cfg;
  const int nb = p.sz.nb;
  const long long rows = static_cast<long long>(c.B) * c.H * nb;
  const int nwords = (nb + 31) / 32;
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float* S = reinterpret_cast<float*>(ws + p.off_scores);
  uint32_t* bitmask = reinterpret_cast<uint32_t*>(ws + p.off_bitmask);
  int32_t* rowcnt = reinterpret_cast<int32_t*>(ws + p.off_rowcnt);
  int32_t* colcnt = reinterpret_cast<int32_t*>(ws + p.off_colcnt);
  int32_t* amb = reinterpret_cast<int32_t*>(ws + p.off_amb);
  float* qn = reinterpret_cast<float*>(ws + p.off_qn);
  float* kn = qn + rows;
  cudaError_t e;
  e = cudaMemsetAsync(status + WS_AMB_COUNT, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  norms_kernel<<<static_cast<unsigned>((2 * rows * 32 + 255) / 256), 256, 0, st>>>(rows, c.d, Qh,
                                                                                   Kh, qn, kn);
  dim3 g((nb + kTile - 1) / kTile, (nb + kTile - 1) / kTile, c.B * c.H);
  score_gemm_kernel<<<g, 256, 0, st>>>(nb, c.d, Qh, Kh, S);
  SelParams sp;
  sp.nb = nb;
  sp.nwords = nwords;
  sp.d = c.d;
  sp.topk = c.topk_floor;
  sp.rows = rows;
  sp.topp = c.topp;
  sp.inv_sqrt_d = static_cast<float>(1.0 / sqrt(static_cast<double>(c.d)));
  sp.u_scale = static_cast<float>(1.01 * (c.d + 5) * 5.9604644775390625e-8 /
                                  sqrt(static_cast<double>(c.d)));
  sp.S = S;
  sp.n_valid = n_valid;
  sp.qn = qn;
  sp.kn = kn;
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
  fp.d = c.d;
  fp.topk = c.topk_floor;
  int P2 = 256;
  while (P2 < nb) P2 <<= 1;
  fp.P2 = P2;
  fp.topp = c.topp;
  {
    const double isd = 1.0 / sqrt(static_cast<double>(c.d));
    fp.inv_sqrt_d.hi = static_cast<float>(isd);
    fp.inv_sqrt_d.lo = static_cast<float>(isd - static_cast<double>(fp.inv_sqrt_d.hi));
  }
  fp.Qh = Qh;
  fp.Ql = Ql;
  fp.Kh = Kh;
  fp.Kl = Kl;
  fp.n_valid = n_valid;
  fp.bitmask = bitmask;
  fp.rowcnt = rowcnt;
  fp.tie = sel_tie;
  fp.amb = amb;
  fp.status = status;
  const size_t fsm = 20ull * P2 + 8ull * c.d;
  e = cudaFuncSetAttribute(select_fallback_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(fsm));
  if (e != cudaSuccess) return e;
  select_fallback_kernel<<<296, 256, fsm, st>>>(fp);
  scan_kernel<<<1, 1024, 0, st>>>(rows, rowcnt, row_ptr);
  csr_fill_kernel<<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, st>>>(
      rows, nwords, bitmask, row_ptr, col_idx);
  const long long units = static_cast<long long>(c.B) * c.H * nwords;
  csc_count_kernel<<<static_cast<unsigned>((units * 32 + 255) / 256), 256, 0, st>>>(
      nb, nwords, units, bitmask, colcnt);
  scan_kernel<<<1, 1024, 0, st>>>(rows, colcnt, col_ptr);
  csc_fill_kernel<<<static_cast<unsigned>((units * 32 + 255) / 256), 256, 0, st>>>(
      nb, nwords, units, bitmask, col_ptr, row_idx);
  return cudaGetLastError();
}

}  // namespace prism
