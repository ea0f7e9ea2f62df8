// Token permutation into zone / block order, block pooling, and the inverse.
//
// Prism (arXiv 2610.05416), Abstract: every zone is cut into blocks of its
// assigned shape and the tokens inside a block are kept together, so that a
// block-level (pooled) feature summarises coherent content.  Order used here:
// zones in raster (zt, zh, zw) order, the zone's blocks in raster order of its
// shape, and inside a block its real tokens first in (t, h, w) raster order,
// then its padding slots.  Because padding sits at the high end of every
// axis, the real tokens of a block form a box [0,et)x[0,ey)x[0,ex) at the
// block origin, so slot k < et*ey*ex maps to a token in closed form.
//
// All kernels move 16-byte pieces: a token row of one head (d bf16) is d/8
// pieces read by d/8 consecutive lanes, so every access is a full-sector,
// aligned 16-byte vector.
#include "prism_internal.cuh"

namespace prism {
namespace {

struct Menu {
  int ext[PRISM_MAX_SHAPES][3];
  uint32_t adm_mask;  // bit k: menu shape k tiles the zone
  int first_adm;      // lowest admissible menu index
};

struct BlockGeom {
  int t0, y0, x0, et, ey, ex;
};

// Geometry of block `local` (raster order of the zone's shape) of zone z.
__device__ __forceinline__ BlockGeom block_geom(const prism_config_t& c, int nzH, int nzW,
                                                const Menu& menu, int sid, int z, int local) {
  const int zt = z / (nzH * nzW), zh = (z / nzW) % nzH, zw = z % nzW;
  const int bT = menu.ext[sid][0], bH = menu.ext[sid][1], bW = menu.ext[sid][2];
  const int nbh = c.zH / bH, nbw = c.zW / bW;
  const int it = local / (nbh * nbw), ih = (local / nbw) % nbh, iw = local % nbw;
  BlockGeom g;
  g.t0 = zt * c.zT + it * bT;
  g.y0 = zh * c.zH + ih * bH;
  g.x0 = zw * c.zW + iw * bW;
  g.et = max(0, min(bT, c.T - g.t0));
  g.ey = max(0, min(bH, c.Hg - g.y0));
  g.ex = max(0, min(bW, c.W - g.x0));
  return g;
}

__device__ __forceinline__ long long slot_token(const prism_config_t& c, const BlockGeom& g,
                                                int k) {
  const int exy = g.ey * g.ex;
  const int t = g.t0 + k / exy, y = g.y0 + (k / g.ex) % g.ey, x = g.x0 + k % g.ex;
  return (static_cast<long long>(t) * c.Hg + y) * c.W + x;
}

constexpr int kPermThreads = 256;

// One CTA per (tile, head, batch).  A tile that starts a block gathers the
// Q, K, V rows of the whole block (1, 2 or 4 tiles of S slots: its class's
// token count) into contiguous block order, writes perm / inv, the real-token
// count of each of its tiles, and the block means of Q and K at its first
// tile (zeros at the tiles that continue it); a continuation tile's CTA
// returns at once.  The means are carried in double-float (hi + lo
// fp32): per-thread compensated sums (two_sum) over the thread's tokens, a
// fixed-order double-float reduction over the token groups, and a
// double-float division by the real-token count -- about 46 significant
// bits, without fp64 arithmetic.
// Three CTAs per SM (80 registers) with two tokens in flight per thread
// move more bytes at once than two CTAs with four (128 registers).
__global__ void __launch_bounds__(kPermThreads, 3) permute_pool_kernel(
    prism_config_t c, int nzH, int nzW, int bpz, int Z, int nb, int nslots, int U, long long Np,
    Menu menu, const uint8_t* __restrict__ shape_id, const uint16_t* __restrict__ Q,
    const uint16_t* __restrict__ K, const uint16_t* __restrict__ V, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv, uint16_t* __restrict__ Qp, uint16_t* __restrict__ Kp,
    uint16_t* __restrict__ Vp, float* __restrict__ Qh, float* __restrict__ Ql,
    float* __restrict__ Kh, float* __restrict__ Kl, int32_t* __restrict__ n_valid,
    uint32_t* __restrict__ status) {
  extern __shared__ __align__(16) float2 red2[];
  const int h = blockIdx.x, blk = blockIdx.y, b = blockIdx.z;  // heads fastest: the heads
                                                                 // of a block share token rows
  const int S = c.block_tokens, d = c.d, P = d / 8;  // S: tile slots; U: table unit slots
  const int G = kPermThreads / P;  // tokens handled per pass
  const int q = threadIdx.x % P, grp = threadIdx.x / P;
  const long long N = static_cast<long long>(c.T) * c.Hg * c.W;
  const long long bh = static_cast<long long>(b) * c.H + h;
  const int z = blk / bpz, lu = blk % bpz;  // bpz: units per zone
  int sid = shape_id[bh * Z + z];
  if (sid >= PRISM_MAX_SHAPES || !((menu.adm_mask >> sid) & 1u)) {
    // a caller-given shape that does not tile the zone: report, fall back
    if (status != nullptr && threadIdx.x == 0 && lu == 0)
      dev_error(status, DEV_ERR_BOUNDS, 0x5A1, static_cast<uint32_t>(sid));
    sid = menu.first_adm;
  }
  const int SB = menu.ext[sid][0] * menu.ext[sid][1] * menu.ext[sid][2];  // block tokens
  const int upb = SB / U;                                                   // units per block
  if (lu % upb != 0) return;  // written by the CTA of the block's first unit
  const BlockGeom g = block_geom(c, nzH, nzW, menu, sid, z, lu / upb);
  const int nv = g.et * g.ey * g.ex;
  if (SB < S && nv < SB && status != nullptr && threadIdx.x == 0)
    // a block of half a tile must be full (its tile's halves are both real)
    dev_error(status, DEV_ERR_BOUNDS, 0x5A2, static_cast<uint32_t>(sid));
  df sq[8], sk[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) sq[k] = sk[k] = df{0.f, 0.f};
  const long long slot0 = static_cast<long long>(blk) * U;
  constexpr int IF = 2;  // tokens per thread in flight
  for (int k0 = grp; k0 < SB; k0 += IF * G) {
    uint4 vq[IF], vk[IF], vv[IF];
    long long nn[IF];
#pragma unroll
    for (int u = 0; u < IF; ++u) {
      const int k = k0 + u * G;
      vq[u] = vk[u] = vv[u] = make_uint4(0, 0, 0, 0);
      nn[u] = -1;
      if (k < nv) {  // nv <= SB
        nn[u] = slot_token(c, g, k);
        const long long src = ((static_cast<long long>(b) * N + nn[u]) * c.H + h) * d + q * 8;
        vq[u] = ldg_nc_v4(Q + src);
        vk[u] = ldg_nc_v4(K + src);
        vv[u] = ldg_nc_v4(V + src);
      }
    }
#pragma unroll
    for (int u = 0; u < IF; ++u) {
      const int k = k0 + u * G;
      if (k >= SB) break;
      const long long dst = (bh * Np + slot0 + k) * d + q * 8;
      if (nn[u] >= 0) {
        const uint32_t wq[4] = {vq[u].x, vq[u].y, vq[u].z, vq[u].w};
        const uint32_t wk[4] = {vk[u].x, vk[u].y, vk[u].z, vk[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          sq[2 * j] = df_add(sq[2 * j], df{bf16_lo(wq[j]), 0.f});
          sq[2 * j + 1] = df_add(sq[2 * j + 1], df{bf16_hi(wq[j]), 0.f});
          sk[2 * j] = df_add(sk[2 * j], df{bf16_lo(wk[j]), 0.f});
          sk[2 * j + 1] = df_add(sk[2 * j + 1], df{bf16_hi(wk[j]), 0.f});
        }
        if (q == 0) {
          perm[bh * Np + slot0 + k] = static_cast<int32_t>(nn[u]);
          inv[bh * N + nn[u]] = static_cast<int32_t>(slot0 + k);
        }
      } else if (q == 0) {
        perm[bh * Np + slot0 + k] = -1;
      }
      *reinterpret_cast<uint4*>(Qp + dst) = vq[u];
      *reinterpret_cast<uint4*>(Kp + dst) = vk[u];
      *reinterpret_cast<uint4*>(Vp + dst) = vv[u];
    }
  }
  // cross-group reduction of the channel sums, fixed order
  float2* rq = red2;
  float2* rk = red2 + G * d;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    rq[grp * d + q * 8 + k] = make_float2(sq[k].hi, sq[k].lo);
    rk[grp * d + q * 8 + k] = make_float2(sk[k].hi, sk[k].lo);
  }
  __syncthreads();
  for (int ch = threadIdx.x; ch < 2 * d; ch += blockDim.x) {
    const float2* r = ch < d ? rq : rk;
    const int cc = ch < d ? ch : ch - d;
    df s = {0.f, 0.f};
    for (int j = 0; j < G; ++j) s = df_add(s, df{r[j * d + cc].x, r[j * d + cc].y});
    const df mean = nv > 0 ? df_div_int(s, nv) : df{0.f, 0.f};
    for (int t = 0; t < upb; ++t) {
      const long long o = (bh * nslots + blk + t) * d + cc;
      const df v = t == 0 ? mean : df{0.f, 0.f};
      if (ch < d) {
        Qh[o] = v.hi;
        Ql[o] = v.lo;
      } else {
        Kh[o] = v.hi;
        Kl[o] = v.lo;
      }
    }
  }
  // real tokens per tile: a block of one or more tiles fills its first tiles;
  // two blocks of half a tile share one (both full), written by the first
  const long long t0 = slot0 / S;
  if (SB >= S) {
    if (threadIdx.x < SB / S)
      n_valid[bh * nb + t0 + threadIdx.x] = min(S, max(0, nv - static_cast<int>(threadIdx.x) * S));
  } else if (threadIdx.x == 0 && slot0 % S == 0) {
    n_valid[bh * nb + t0] = S;
  }
}

// Xp[b,h,s,:] = X[b,perm[s],h,:] (zeros on padding slots).  One thread per
// 16-byte piece of the output.
__global__ void __launch_bounds__(256) permute_kernel(int H, int d, long long N, long long Np,
                                                      const int32_t* __restrict__ perm,
                                                      const uint16_t* __restrict__ X,
                                                      uint16_t* __restrict__ Xp) {
  const int P = d / 8;
  const long long total = Np * P;
  const int h = blockIdx.y, b = blockIdx.z;
  const long long bh = static_cast<long long>(b) * H + h;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long s = i / P;
    const int q = static_cast<int>(i % P);
    const int n = perm[bh * Np + s];
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n >= 0) v = ldg_nc_v4(X + ((static_cast<long long>(b) * N + n) * H + h) * d + q * 8);
    *reinterpret_cast<uint4*>(Xp + (bh * Np + s) * d + q * 8) = v;
  }
}

// X[b,n,h,:] = Xp[b,h,inv[n],:].  One thread per 16-byte piece of the
// output, which is written in its natural [B, N, H, d] order.
__global__ void __launch_bounds__(256) unpermute_kernel(int H, int d, long long N, long long Np,
                                                        const int32_t* __restrict__ inv,
                                                        const uint16_t* __restrict__ Xp,
                                                        uint16_t* __restrict__ X) {
  const int P = d / 8;
  const long long per_b = N * H * P;
  const int b = blockIdx.y;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < per_b;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long n = i / (H * P);
    const int r = static_cast<int>(i % (H * P));
    const int h = r / P, q = r % P;
    const long long bh = static_cast<long long>(b) * H + h;
    const int s = inv[bh * N + n];
    const uint4 v = ldg_nc_v4(Xp + (bh * Np + s) * d + q * 8);
    *reinterpret_cast<uint4*>(X + ((static_cast<long long>(b) * N + n) * H + h) * d + q * 8) = v;
  }
}

// fp32 dQ accumulator -> bf16, times `scale`, in block order.  One thread
// per 8 channels.
__global__ void __launch_bounds__(256) dq_convert_kernel(long long pieces,
                                                         const float* __restrict__ dq,
                                                         float scale, uint16_t* __restrict__ out) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < pieces;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float* src = dq + i * 8;
    const uint4 a = ldg_nc_v4(src), c4 = ldg_nc_v4(src + 4);
    uint4 o;
    o.x = pack_bf16x2(__uint_as_float(a.x) * scale, __uint_as_float(a.y) * scale);
    o.y = pack_bf16x2(__uint_as_float(a.z) * scale, __uint_as_float(a.w) * scale);
    o.z = pack_bf16x2(__uint_as_float(c4.x) * scale, __uint_as_float(c4.y) * scale);
    o.w = pack_bf16x2(__uint_as_float(c4.z) * scale, __uint_as_float(c4.w) * scale);
    *reinterpret_cast<uint4*>(out + i * 8) = o;
  }
}

int grid_for(long long pieces) {
  long long g = (pieces + 255) / 256;
  const long long cap = 148LL * 16;  // a few waves over the 148 SMs; loops cover the rest
  return static_cast<int>(g < cap ? (g < 1 ? 1 : g) : cap);
}

}  // namespace

cudaError_t launch_permute_pool(const Plan& p, const uint8_t* shape_id, const uint16_t* Q,
                                const uint16_t* K, const uint16_t* V, int32_t* perm,
                                int32_t* inv, uint16_t* Qp, uint16_t* Kp, uint16_t* Vp,
                                float* Qh, float* Ql, float* Kh, float* Kl, int32_t* n_valid,
                                uint32_t* status, cudaStream_t st) {
  const prism_config_t& c = p.cfg;
  Menu m;
  for (int k = 0; k < PRISM_MAX_SHAPES; ++k)
    for (int a = 0; a < 3; ++a) m.ext[k][a] = k < c.n_shapes ? c.shapes[k][a] : 1;
  m.adm_mask = 0;
  for (int q = 0; q < p.sz.n_admissible; ++q) m.adm_mask |= 1u << p.sz.admissible[q];
  m.first_adm = p.sz.admissible[0];
  const int G = kPermThreads / (c.d / 8);
  const size_t smem = 2ull * G * c.d * sizeof(float2);
  cudaError_t e = cudaFuncSetAttribute(permute_pool_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (p.sz.nb > 65535) return cudaErrorInvalidValue;
  if (p.sz.nslots > 65535) return cudaErrorInvalidValue;
  const int U = p.sz.slot_tokens;
  const int upz = c.zT * c.zH * c.zW / U;  // table units per zone
  dim3 grid(c.H, p.sz.nslots, c.B);
  permute_pool_kernel<<<grid, kPermThreads, smem, st>>>(
      c, p.sz.nzH, p.sz.nzW, upz, p.sz.Z, p.sz.nb, p.sz.nslots, U, p.sz.Np, m, shape_id, Q, K,
      V, perm, inv, Qp, Kp, Vp, Qh, Ql, Kh, Kl, n_valid, status);
  return cudaGetLastError();
}

cudaError_t launch_permute(const Plan& p, const int32_t* perm, const uint16_t* X, uint16_t* Xp,
                           cudaStream_t st) {
  const prism_config_t& c = p.cfg;
  const long long pieces = p.sz.Np * (c.d / 8);
  int gx = grid_for(pieces * c.H * c.B) / (c.H * c.B);
  if (gx < 1) gx = 1;
  permute_kernel<<<dim3(gx, c.H, c.B), 256, 0, st>>>(c.H, c.d, p.sz.N, p.sz.Np, perm, X, Xp);
  return cudaGetLastError();
}

cudaError_t launch_unpermute(const Plan& p, const int32_t* inv, const uint16_t* Xp, uint16_t* X,
                             cudaStream_t st) {
  const prism_config_t& c = p.cfg;
  const long long pieces = p.sz.N * c.H * (c.d / 8);
  int gx = grid_for(pieces * c.B) / c.B;
  if (gx < 1) gx = 1;
  unpermute_kernel<<<dim3(gx, c.B), 256, 0, st>>>(c.H, c.d, p.sz.N, p.sz.Np, inv, Xp, X);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const Plan& p, const float* dq, float scale, uint16_t* dQp,
                              cudaStream_t st) {
  const long long pieces = static_cast<long long>(p.cfg.B) * p.cfg.H * p.sz.Np * (p.cfg.d / 8);
  dq_convert_kernel<<<grid_for(pieces), 256, 0, st>>>(pieces, dq, scale, dQp);
  return cudaGetLastError();
}

}  // namespace prism
