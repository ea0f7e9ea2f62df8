// Zone statistics and block-shape assignment.
//
// Prism (arXiv 2610.05416), Abstract: each spatiotemporal macro-zone is
// described by the variance of the video features along each axis and by
// the norms of the audio-to-video (A2V) cross-attention output; Table 9
// caption names the three signals (per-channel variance of the value
// features r_{v,d}, audio coupling gate a_bar, audio directional variance
// v_hat_{a,d}); Table 10 caption gives the Eq. 7 quantisation
// b*_d ~ g_d^-alpha with alpha = 1 the best setting.
//
// zone_stats (zones wider than 4 x 16 x 16): one CTA per (zone, head) for
// the value variance and one CTA per zone for the A2V norm statistics.  The zone's real tokens are staged in
// shared memory 32 channels at a time (cp.async, 16-byte rows pieces, two
// stages so the next chunk loads while this one is reduced), then every line
// along every axis is reduced exactly with a two-pass mean / variance.
#include <cooperative_groups.h>
#include <string.h>

#include "prism_internal.cuh"

namespace prism {
namespace {

constexpr int kStatsThreads = 256;
constexpr int kChunk = 32;  // channels per smem stage (64 bytes of bf16)

struct ZoneGeom {
  int t0, y0, x0;  // zone origin on the padded grid
  int vt, vy, vx;  // real extents inside the zone (>= 1 each)
};

__device__ __forceinline__ ZoneGeom zone_geom(const prism_config_t& c, int nzH, int nzW, int z) {
  ZoneGeom g;
  int zt = z / (nzH * nzW), zh = (z / nzW) % nzH, zw = z % nzW;
  g.t0 = zt * c.zT;
  g.y0 = zh * c.zH;
  g.x0 = zw * c.zW;
  g.vt = min(c.zT, c.T - g.t0);
  g.vy = min(c.zH, c.Hg - g.y0);
  g.vx = min(c.zW, c.W - g.x0);
  return g;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N));
}

// Sum over the CTA, fixed order (deterministic).
template <int NV>
__device__ __forceinline__ void block_sum(float (&v)[NV], float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
  }
  __syncthreads();
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < NV; ++k) red[warp * NV + k] = v[k];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int nw = blockDim.x >> 5;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      float s = 0.f;
      for (int w = 0; w < nw; ++w) s += red[w * NV + k];
      v[k] = s;
    }
  }
}

// Accumulate, over the lines along one axis, the population variance of
// every channel pair held in a [vt][vy][vx][kChunk] bf16 smem tile.
// `len` tokens per line with stride `step` (in tokens); lines are indexed by
// (a, b) over extents (na, nb) with strides (sa, sb).
__device__ __forceinline__ float lines_variance(const uint32_t* tile, int na, int nb, int sa,
                                                int sb, int len, int step) {
  float acc = 0.f;
  if (len < 2) return 0.f;
  const int pairs = kChunk / 2;
  const int items = na * nb * pairs;
  const float inv = 1.f / static_cast<float>(len);
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    const int cp = it % pairs;
    const int ln = it / pairs;
    const int base = (ln / nb) * sa + (ln % nb) * sb;
    float m0 = 0.f, m1 = 0.f;
    for (int k = 0; k < len; ++k) {
      uint32_t u = tile[(base + k * step) * pairs + cp];
      m0 += bf16_lo(u);
      m1 += bf16_hi(u);
    }
    m0 *= inv;
    m1 *= inv;
    float s0 = 0.f, s1 = 0.f;
    for (int k = 0; k < len; ++k) {
      uint32_t u = tile[(base + k * step) * pairs + cp];
      float a = bf16_lo(u) - m0, b = bf16_hi(u) - m1;
      s0 = fmaf(a, a, s0);
      s1 = fmaf(b, b, s1);
    }
    acc += (s0 + s1) * inv;
  }
  return acc;
}

// A2V norm map of one zone: n_i = ||a2v_i||_2 and its directional
// statistics.  The audio directional variance is a ratio of variances that
// can be tiny (a norm map that is nearly constant over the zone), so the
// norms are accurate to ~1e-11 and the line statistics run in fp64: 768
// norms and ~350 lines per zone.  Written to slots 3..7 of every head's
// record.
__device__ void audio_zone_stats(const prism_config_t& c, const ZoneGeom& g, int b, int z, int Z,
                                 const uint16_t* __restrict__ a2v, const float* __restrict__ nrm,
                                 float* __restrict__ stats, uint8_t* smem) {
  const int vol = g.vt * g.vy * g.vx;
  const long long N = static_cast<long long>(c.T) * c.Hg * c.W;
  double* nmap = reinterpret_cast<double*>(smem);
  __shared__ double dred[32 * 4];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  // one token per thread: the squares of bf16 values are exact in fp32 and
  // are summed as a double-float (TwoSum), so n^2 carries ~1e-11 relative
  // error before the fp64 square root -- far below the 1e-10 nbar^2 floor on
  // the directional variance, at FP32 rather than FP64 throughput
  const bool vec = (c.Ca % 8) == 0;
  for (int li = threadIdx.x; li < vol; li += blockDim.x) {
    const int x = li % g.vx, y = (li / g.vx) % g.vy, t = li / (g.vx * g.vy);
    const long long n =
        (static_cast<long long>(g.t0 + t) * c.Hg + (g.y0 + y)) * c.W + (g.x0 + x);
    if (nrm != nullptr) {  // norms given (computed by the A2V kernel)
      nmap[li] = static_cast<double>(nrm[static_cast<long long>(b) * N + n]);
      continue;
    }
    const uint16_t* row = a2v + (static_cast<long long>(b) * N + n) * c.Ca;
    float hi = 0.f, lo = 0.f;
    auto add = [&](float v) {
      const float p = v * v;
      const float s2 = hi + p, bb = s2 - hi;
      lo += (hi - (s2 - bb)) + (p - bb);
      hi = s2;
    };
    if (vec) {
      const uint4* r4 = reinterpret_cast<const uint4*>(row);
      for (int k = 0; k < c.Ca / 8; ++k) {
        const uint4 q = __ldg(r4 + k);
        const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          add(bf16_lo(u[e]));
          add(bf16_hi(u[e]));
        }
      }
    } else {
      for (int k = 0; k < c.Ca; ++k) add(bf16_to_f(row[k]));
    }
    nmap[li] = sqrt(static_cast<double>(hi) + static_cast<double>(lo));
  }
  __syncthreads();
  // line variances of the scalar map, thread per line
  double acc[4] = {0.0, 0.0, 0.0, 0.0};
  const int nlT = g.vy * g.vx, nlH = g.vt * g.vx, nlW = g.vt * g.vy;
  for (int ln = threadIdx.x; ln < nlT + nlH + nlW; ln += blockDim.x) {
    int base, len, step, axis;
    if (ln < nlT) {
      axis = 0; base = ln; len = g.vt; step = g.vy * g.vx;
    } else if (ln < nlT + nlH) {
      const int l = ln - nlT;
      axis = 1; base = (l / g.vx) * g.vy * g.vx + (l % g.vx); len = g.vy; step = g.vx;
    } else {
      const int l = ln - nlT - nlH;
      axis = 2; base = l * g.vx; len = g.vx; step = 1;
    }
    if (len < 2) continue;
    double m = 0.0;
    for (int k = 0; k < len; ++k) m += nmap[base + k * step];
    m /= static_cast<double>(len);
    double s = 0.0;
    for (int k = 0; k < len; ++k) {
      const double e = nmap[base + k * step] - m;
      s = fma(e, e, s);
    }
    acc[axis] += s / static_cast<double>(len);
  }
  for (int li = threadIdx.x; li < vol; li += blockDim.x) acc[3] += nmap[li];
  // fixed-order reduction (deterministic)
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
  __syncthreads();
  if (lane == 0)
    for (int k = 0; k < 4; ++k) dred[warp * 4 + k] = acc[k];
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 0; k < 4; ++k) {
      double s = 0.0;
      for (int q = 0; q < nw; ++q) s += dred[q * 4 + k];
      acc[k] = s;
    }
    const double nl[3] = {static_cast<double>(nlT), static_cast<double>(nlH),
                          static_cast<double>(nlW)};
    const int len[3] = {g.vt, g.vy, g.vx};
    float out[5];
    for (int a = 0; a < 3; ++a) out[a] = len[a] >= 2 ? static_cast<float>(acc[a] / nl[a]) : 0.f;
    out[3] = static_cast<float>(acc[3] / static_cast<double>(vol));
    out[4] = static_cast<float>(vol);
    for (int hh = 0; hh < c.H; ++hh) {
      float* o = stats + ((static_cast<long long>(b) * c.H + hh) * Z + z) * 8;
      for (int k = 0; k < 5; ++k) o[3 + k] = out[k];
    }
  }
}

__global__ void __launch_bounds__(kStatsThreads) zone_stats_kernel(
    prism_config_t c, int nzH, int nzW, int Z, const uint16_t* __restrict__ V,
    const uint16_t* __restrict__ a2v, const float* __restrict__ nrm, float* __restrict__ stats) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float red[32 * 4];
  const int z = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const ZoneGeom g = zone_geom(c, nzH, nzW, z);
  const int vol = g.vt * g.vy * g.vx;
  const long long N = static_cast<long long>(c.T) * c.Hg * c.W;

  if (h < c.H) {
    // ---- directional variance of the value features of head h ----
    const int nchunk = c.d / kChunk;
    const size_t stage_bytes = static_cast<size_t>(vol) * kChunk * 2;
    auto load_chunk = [&](int ch, int stage) {
      uint8_t* dst = smem + stage * stage_bytes;
      const int pieces = vol * (kChunk / 8);
      for (int i = threadIdx.x; i < pieces; i += blockDim.x) {
        const int li = i >> 2, q = i & 3;
        const int x = li % g.vx, y = (li / g.vx) % g.vy, t = li / (g.vx * g.vy);
        const long long n =
            (static_cast<long long>(g.t0 + t) * c.Hg + (g.y0 + y)) * c.W + (g.x0 + x);
        const uint16_t* src = V + ((static_cast<long long>(b) * N + n) * c.H + h) * c.d +
                              ch * kChunk + q * 8;
        cp_async16(dst + static_cast<size_t>(li) * kChunk * 2 + q * 16, src);
      }
      cp_async_commit();
    };
    float acc[3] = {0.f, 0.f, 0.f};
    load_chunk(0, 0);
    for (int ch = 0; ch < nchunk; ++ch) {
      if (ch + 1 < nchunk) {
        load_chunk(ch + 1, (ch + 1) & 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      const uint32_t* tile = reinterpret_cast<const uint32_t*>(smem + (ch & 1) * stage_bytes);
      // token index li = (t*vy + y)*vx + x
      acc[0] += lines_variance(tile, g.vy, g.vx, g.vx, 1, g.vt, g.vy * g.vx);  // along T
      acc[1] += lines_variance(tile, g.vt, g.vx, g.vy * g.vx, 1, g.vy, g.vx);  // along H
      acc[2] += lines_variance(tile, g.vt, g.vy, g.vy * g.vx, g.vx, g.vx, 1);  // along W
      __syncthreads();
    }
    block_sum<3>(acc, red);
    if (threadIdx.x == 0) {
      const float nl[3] = {static_cast<float>(g.vy * g.vx), static_cast<float>(g.vt * g.vx),
                           static_cast<float>(g.vt * g.vy)};
      const int len[3] = {g.vt, g.vy, g.vx};
      float* o = stats + ((static_cast<long long>(b) * c.H + h) * Z + z) * 8;
      for (int a = 0; a < 3; ++a)
        o[a] = len[a] >= 2 ? acc[a] / (nl[a] * static_cast<float>(c.d)) : 0.f;
    }
  } else {
    audio_zone_stats(c, g, b, z, Z, a2v, nrm, stats, smem);
  }
}

// Zones of at most kPT x kPH x kPW tokens (the 3 x 16 x 16 zones of the
// latent grids, and smaller ones) take the cluster kernel below; each token
// row (t, y) of a staged 32-channel slice is padded by 64 bytes so that the
// register passes are free of bank conflicts.  Thread (cp, j): cp = channel
// pair of the slice (16), j = y or x (16).  Every line is reduced with a
// two-pass mean / variance in fp32.
constexpr int kPT = 4, kPH = 16, kPW = 16;

// Packed pairs of fp32 (the two channels of a bf16x2 word) for the fp32x2
// arithmetic of sm_100-class SMs (add2 / sub2 / mul2 / fma2, shared helpers).
__device__ __forceinline__ f32x2 unpack2(uint32_t u) {  // bf16x2 -> (lo, hi) fp32
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(u << 16), "r"(u & 0xffff0000u));
  return r;
}
__device__ __forceinline__ f32x2 splat2(float a) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(a));
  return r;
}
__device__ __forceinline__ float hsum2(f32x2 a) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a));
  return lo + hi;
}

// Sum over both channels of the squared deviations from the line mean of
// v[0..n) (two-pass); with n a compile-time constant (full zones) every
// predicate folds away.
template <int M>
__device__ __forceinline__ float line_ss(const f32x2 (&v)[M], int n) {
  f32x2 m = 0ull;
#pragma unroll
  for (int k = 0; k < M; ++k)
    if (k < n) m = add2(m, v[k]);
  m = mul2(m, splat2(1.f / static_cast<float>(n)));
  f32x2 s = 0ull;
#pragma unroll
  for (int k = 0; k < M; ++k)
    if (k < n) {
      const f32x2 e = sub2(v[k], m);
      s = fma2(e, e, s);
    }
  return hsum2(s);
}

// The lines of one staged 32-channel slice, one line set at a time so that
// a thread holds at most one line (16 words) in registers: along W the
// (t, y = j) rows, along T the (y = j, x) columns, along H the (t, x = j)
// columns.  Each staged element is read three times from shared memory.
template <int MT, int MH, int MW, bool EXACT>
__device__ __forceinline__ void lines_chunk(const uint32_t* __restrict__ tile, int rs, int vt_,
                                            int vy_, int vx_, int cp, int j, float (&acc)[3]) {
  const int vt = EXACT ? MT : vt_, vy = EXACT ? MH : vy_, vx = EXACT ? MW : vx_;
  constexpr int P = kChunk / 2;  // words per token in a stage
  if (j < vy) {
    if (vx >= 2) {
      const float inv = 1.f / static_cast<float>(vx);
#pragma unroll 1
      for (int t = 0; t < vt; ++t) {
        f32x2 v[MW];
#pragma unroll
        for (int x = 0; x < MW; ++x)
          v[x] = unpack2(x < vx ? tile[(t * vy + j) * rs + x * P + cp] : 0u);
        acc[2] += line_ss(v, vx) * inv;
      }
    }
    if (vt >= 2) {
      const float inv = 1.f / static_cast<float>(vt);
#pragma unroll 1
      for (int x = 0; x < vx; ++x) {
        f32x2 v[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t)
          v[t] = unpack2(t < vt ? tile[(t * vy + j) * rs + x * P + cp] : 0u);
        acc[0] += line_ss(v, vt) * inv;
      }
    }
  }
  if (j < vx && vy >= 2) {
    const float inv = 1.f / static_cast<float>(vy);
#pragma unroll 1
    for (int t = 0; t < vt; ++t) {
      f32x2 v[MH];
#pragma unroll
      for (int y = 0; y < MH; ++y)
        v[y] = unpack2(y < vy ? tile[(t * vy + y) * rs + j * P + cp] : 0u);
      acc[1] += line_ss(v, vy) * inv;
    }
  }
}

// Same statistics with the channels split over a thread-block cluster: the
// d / 32 CTAs of a cluster take one 32-channel slice each of the same
// (zone, head), stage it in shared memory in one go (all loads issued at
// once, no chunk loop), reduce their lines as above, and the cluster's
// first CTA sums the slices' partial sums in fixed order through distributed
// shared memory (deterministic).  Up to four clusters' CTAs share an SM, so
// many more loads are in flight than with one CTA walking the channel
// chunks of a (zone, head) in turn.  The audio statistics take the first CTA
// of the cluster of the extra head slot h == H.
__global__ void __launch_bounds__(kStatsThreads, 4) zone_stats_cluster_kernel(
    prism_config_t c, int nzH, int nzW, int Z, const uint16_t* __restrict__ V,
    const uint16_t* __restrict__ a2v, const float* __restrict__ nrm, float* __restrict__ stats) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float red[32 * 4];
  __shared__ float part[3];
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int ncl = static_cast<int>(cluster.num_blocks());       // channel slices
  const int slice = static_cast<int>(cluster.block_rank());
  const int h = blockIdx.x / ncl, z = blockIdx.y, b = blockIdx.z;
  const ZoneGeom g = zone_geom(c, nzH, nzW, z);
  if (h == c.H) {  // uniform over the cluster: no cluster barrier on this path
    if (slice == 0) audio_zone_stats(c, g, b, z, Z, a2v, nrm, stats, smem);
    return;
  }
  const long long N = static_cast<long long>(c.T) * c.Hg * c.W;
  const int vol = g.vt * g.vy * g.vx;
  const int rs = g.vx * (kChunk / 2) + 16;  // words per padded token row (t, y)
  uint32_t* tile = reinterpret_cast<uint32_t*>(smem);
  {
    // one 16-byte piece per thread and pass: piece i = (token, quarter);
    // full 16 x 16 frames take their token coordinates by shifts
    const uint16_t* vb = V + (static_cast<long long>(b) * N * c.H + h) * c.d + slice * kChunk;
    const long long tok_stride = static_cast<long long>(c.H) * c.d;  // elements per token
    const int pieces = vol * (kChunk / 8);
    if (g.vy == 16 && g.vx == 16) {
#pragma unroll 4
      for (int i = threadIdx.x; i < pieces; i += blockDim.x) {
        const int li = i >> 2, q = i & 3;
        const int x = li & 15, y = (li >> 4) & 15, t = li >> 8;
        const long long n = (static_cast<long long>(g.t0 + t) * c.Hg + (g.y0 + y)) * c.W + (g.x0 + x);
        cp_async16(tile + (t * 16 + y) * rs + x * (kChunk / 2) + q * 4, vb + n * tok_stride + q * 8);
      }
    } else {
      for (int i = threadIdx.x; i < pieces; i += blockDim.x) {
        const int li = i >> 2, q = i & 3;
        const int x = li % g.vx, y = (li / g.vx) % g.vy, t = li / (g.vx * g.vy);
        const long long n =
            (static_cast<long long>(g.t0 + t) * c.Hg + (g.y0 + y)) * c.W + (g.x0 + x);
        cp_async16(tile + (t * g.vy + y) * rs + x * (kChunk / 2) + q * 4, vb + n * tok_stride + q * 8);
      }
    }
    cp_async_commit();
    cp_async_wait<0>();
  }
  __syncthreads();
  const int cp = threadIdx.x & 15, j = threadIdx.x >> 4;
  float acc[3] = {0.f, 0.f, 0.f};
  if (g.vt == 3 && g.vy == 16 && g.vx == 16)
    lines_chunk<3, 16, 16, true>(tile, rs, 3, 16, 16, cp, j, acc);
  else if (g.vt == 4 && g.vy == 16 && g.vx == 16)
    lines_chunk<4, 16, 16, true>(tile, rs, 4, 16, 16, cp, j, acc);
  else
    lines_chunk<kPT, kPH, kPW, false>(tile, rs, g.vt, g.vy, g.vx, cp, j, acc);
  block_sum<3>(acc, red);
  if (threadIdx.x == 0)
    for (int a = 0; a < 3; ++a) part[a] = acc[a];
  cluster.sync();
  if (slice == 0 && threadIdx.x == 0) {
    float tot[3] = {0.f, 0.f, 0.f};
    for (int r = 0; r < ncl; ++r) {
      const float* pr = cluster.map_shared_rank(part, r);
      for (int a = 0; a < 3; ++a) tot[a] += pr[a];
    }
    const float nl[3] = {static_cast<float>(g.vy * g.vx), static_cast<float>(g.vt * g.vx),
                         static_cast<float>(g.vt * g.vy)};
    const int len[3] = {g.vt, g.vy, g.vx};
    float* o = stats + ((static_cast<long long>(b) * c.H + h) * Z + z) * 8;
    for (int a = 0; a < 3; ++a)
      o[a] = len[a] >= 2 ? tot[a] / (nl[a] * static_cast<float>(c.d)) : 0.f;
  }
  cluster.sync();  // the partial sums stay readable until the first CTA has them
}

// ------------------------------------------------------------ assign ------

struct MenuConst {
  double log2_ext[PRISM_MAX_SHAPES][3];
  int adm[PRISM_MAX_CLASSES][PRISM_MAX_SHAPES];  // admissible menu shapes per class
  int n_adm[PRISM_MAX_CLASSES];
  double log2_S[PRISM_MAX_CLASSES];             // log2 of each class's token count
  double tau[PRISM_MAX_CLASSES - 1];            // class thresholds, descending
  int n_classes;
  int half_tile;                                // class 0 is half a tile
  int zone_volume;
};

// Eq. 7 (Table 10 caption) in log space: with bT*bH*bW = S fixed, the
// continuous optimum of b_d ~ g_d^-alpha is
//   log2 b*_d = log2(S)/3 + alpha * (mean_d log2 g_d - log2 g_d)
// and each admissible menu shape is scored by sum_d (log2 b_d - log2 b*_d)^2.
// Guidance g_d = u_v r_{v,d} + u_a a_bar v_hat_{a,d} + eps, with
// r_{v,d} = var_v_d / sum var_v, v_hat_{a,d} = var_n_d / sum var_n (1/3 each
// when the sum is 0) and a_bar = nbar / max over the zones of nbar.
// With several block-size classes (Table 10 caption: thresholds
// tau_128 / tau_256), S is the zone's class: the number of thresholds its
// complexity c = u_v V_z / mean_z V + u_a a_bar is below, V_z = sum_d var_v_d.
__global__ void __launch_bounds__(256) assign_kernel(prism_config_t c, int Z, MenuConst menu,
                                                     const float* __restrict__ stats,
                                                     uint8_t* __restrict__ shape_id,
                                                     uint8_t* __restrict__ shape_tie) {
  __shared__ double red[32], red2[32];
  const int h = blockIdx.x, b = blockIdx.y;
  const float* sb = stats + static_cast<long long>(b) * c.H * Z * 8;
  const float* sh = sb + static_cast<long long>(h) * Z * 8;
  // the zone's video statistics (this head's, or the mean over heads)
  auto video = [&](int z, double (&sv)[3]) {
    if (c.per_head) {
      for (int a = 0; a < 3; ++a) sv[a] = sh[z * 8 + a];
    } else {
      for (int a = 0; a < 3; ++a) {
        double s = 0.0;
        for (int hh = 0; hh < c.H; ++hh)
          s += static_cast<double>(sb[(static_cast<long long>(hh) * Z + z) * 8 + a]);
        sv[a] = s / c.H;
      }
    }
  };
  // max over zones of nbar (the audio statistics are the same for every head)
  // and, for the class rule, the sum over zones of V_z (fixed order)
  double mx = 0.0, vs = 0.0;
  for (int z = threadIdx.x; z < Z; z += blockDim.x) {
    mx = fmax(mx, static_cast<double>(sh[z * 8 + 6]));
    if (menu.n_classes > 1) {
      double sv[3];
      video(z, sv);
      vs += sv[0] + sv[1] + sv[2];
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    vs += __shfl_xor_sync(0xffffffffu, vs, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5] = mx;
    red2[threadIdx.x >> 5] = vs;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double m = 0.0, v = 0.0;
    for (int w = 0; w < (blockDim.x >> 5); ++w) {
      m = fmax(m, red[w]);
      v += red2[w];
    }
    red[0] = m;
    red2[0] = v / Z;
  }
  __syncthreads();
  const double nmax = red[0], vmean = red2[0];
  const double uv = c.use_video ? 1.0 : 0.0, ua = c.use_audio ? 1.0 : 0.0;
  for (int z = threadIdx.x; z < Z; z += blockDim.x) {
    double sv[3], sn[3], nbar;
    video(z, sv);
    for (int a = 0; a < 3; ++a) sn[a] = sh[z * 8 + 3 + a];
    nbar = sh[z * 8 + 6];
    const double ssv = sv[0] + sv[1] + sv[2];
    const double ssn = sn[0] + sn[1] + sn[2];
    // no audio direction when the norm map's variance is round-off (a
    // constant map, or one whose spread is below what fp32 norms resolve):
    // at most 1e-10 nbar^2
    const bool no_var = !(ssn > 1e-10 * nbar * nbar);
    const double abar = nmax > 0.0 ? nbar / nmax : 0.0;
    // block-size class
    int cls = 0;
    bool class_tie = false;
    if (menu.n_classes > 1) {
      const double cz = uv * (vmean > 0.0 ? ssv / vmean : 0.0) + ua * abar;
      for (int q = 0; q + 1 < menu.n_classes; ++q) {
        cls += cz < menu.tau[q] ? 1 : 0;
        class_tie |= fabs(cz - menu.tau[q]) <= 1e-5 * fmax(1.0, fabs(menu.tau[q]));
      }
      // a zone with padding takes no class smaller than a tile
      if (menu.half_tile && cls == 0 && sh[z * 8 + 7] < static_cast<float>(menu.zone_volume))
        cls = 1;
    }
    double lg[3];
    for (int a = 0; a < 3; ++a) {
      const double r = ssv > 0.0 ? sv[a] / ssv : 1.0 / 3.0;
      const double vh = no_var ? 1.0 / 3.0 : sn[a] / ssn;
      const double gd = uv * r + ua * abar * vh + c.eps;
      lg[a] = log2(gd);
    }
    const double mean = (lg[0] + lg[1] + lg[2]) / 3.0;
    double lstar[3];
    for (int a = 0; a < 3; ++a) lstar[a] = menu.log2_S[cls] / 3.0 + c.alpha * (mean - lg[a]);
    double best = 1e300, second = 1e300;
    int bk = menu.adm[cls][0];
    for (int q = 0; q < menu.n_adm[cls]; ++q) {
      const int k = menu.adm[cls][q];
      double cost = 0.0;
      for (int a = 0; a < 3; ++a) {
        const double e = menu.log2_ext[k][a] - lstar[a];
        cost += e * e;
      }
      if (cost < best) {
        second = best;
        best = cost;
        bk = k;
      } else if (cost < second) {
        second = cost;
      }
    }
    const long long o = (static_cast<long long>(b) * c.H + h) * Z + z;
    shape_id[o] = static_cast<uint8_t>(bk);
    shape_tie[o] = ((menu.n_adm[cls] > 1 && (second - best) < 1e-4) || class_tie) ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_zone_stats(const Plan& p, const uint16_t* V, const uint16_t* a2v,
                              const float* nrm, float* stats, cudaStream_t st) {
  const prism_config_t& c = p.cfg;
  const int vol = c.zT * c.zH * c.zW;
  const size_t smem_video = 2ull * vol * kChunk * 2;
  const size_t smem_audio = static_cast<size_t>(vol) * sizeof(double);
  const size_t smem = smem_video > smem_audio ? smem_video : smem_audio;
  if (c.zT <= kPT && c.zH <= kPH && c.zW <= kPW && p.sz.Z <= 65535) {
    const int ncl = c.d / kChunk;  // channel slices = CTAs per cluster (d <= 128: <= 4)
    const size_t sv = static_cast<size_t>(c.zT) * c.zH * (c.zW * (kChunk / 2) + 16) * 4;
    const size_t sm = sv > smem_audio ? sv : smem_audio;
    cudaError_t e = cudaFuncSetAttribute(zone_stats_cluster_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sm));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((c.H + 1) * ncl, p.sz.Z, c.B);
    cfg.blockDim = dim3(kStatsThreads, 1, 1);
    cfg.dynamicSmemBytes = sm;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ncl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, zone_stats_cluster_kernel, c, p.sz.nzH, p.sz.nzW, p.sz.Z, V,
                           a2v, nrm, stats);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  cudaError_t e = cudaFuncSetAttribute(zone_stats_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(p.sz.Z, c.H + 1, c.B);
  zone_stats_kernel<<<grid, kStatsThreads, smem, st>>>(c, p.sz.nzH, p.sz.nzW, p.sz.Z, V, a2v,
                                                      nrm, stats);
  return cudaGetLastError();
}

cudaError_t launch_assign(const Plan& p, const float* stats, uint8_t* shape_id,
                          uint8_t* shape_tie, cudaStream_t st) {
  MenuConst m;
  memset(&m, 0, sizeof(m));
  const prism_config_t& c = p.cfg;
  for (int k = 0; k < PRISM_MAX_SHAPES; ++k)
    for (int a = 0; a < 3; ++a) m.log2_ext[k][a] = p.log2_ext[k][a];
  m.n_classes = p.sz.n_classes;
  m.half_tile = p.sz.half_tile;
  m.zone_volume = c.zT * c.zH * c.zW;
  for (int q = 0; q < p.sz.n_classes; ++q) {
    m.log2_S[q] = log2(static_cast<double>(p.sz.class_tokens[q]));
    for (int a = 0; a < p.sz.n_admissible; ++a) {
      const int k = p.sz.admissible[a];
      if (c.shapes[k][0] * c.shapes[k][1] * c.shapes[k][2] == p.sz.class_tokens[q])
        m.adm[q][m.n_adm[q]++] = k;
    }
    if (q + 1 < p.sz.n_classes) m.tau[q] = c.class_tau[q];
  }
  assign_kernel<<<dim3(p.cfg.H, p.cfg.B), 256, 0, st>>>(p.cfg, p.sz.Z, m, stats, shape_id,
                                                        shape_tie);
  return cudaGetLastError();
}

}  // namespace prism
