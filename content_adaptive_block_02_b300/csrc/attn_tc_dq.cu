// dQ of the block-sparse attention on the tcgen05 tensor cores, 128-token
// blocks, head dim 128.
//
// Prism (arXiv 2610.05416) trains through its sparse attention (Table 2
// caption).  dQ_i = scale * sum over the key blocks j selected by query
// block i of dS_ij K_j, with P_ij = exp(Q_i K_j^T * scale - LSE_i) and
// dS_ij = P_ij * (dO_i V_j^T - D_i).  The key-block side (dK, dV) runs in a
// separate kernel, so dQ needs no atomics: it is summed in tensor memory over
// the key blocks of a range and written once per range, in bf16 (once in all
// when the plan does not split the keys), deterministically.
//
// Work item = one query block (b, h, i) with its ascending list of key
// blocks (CSR), restricted to one range of key blocks when the plan walks
// them in ranges (partial dQ per range, summed in combine.cu).  Per key block
// j, three 128x128x128 products:
//   S  = Q_i K_j^T     A = Q_i (smem),  B = K_j (smem)        -> TMEM S
//   dP = dO_i V_j^T    A = dO_i (smem), B = V_j (smem)        -> TMEM dP
//   dQ += dS K_j       A = dS (TMEM, bf16), B = K_j (MN-major) -> TMEM dQ
// Roles (384 threads, one persistent CTA per SM):
//   warps 0-7  compute: thread = query row; warps w and w+4 split the key
//              columns in halves.  P = exp2(S*c - LSE*log2 e), dS = P (dP - D)
//              -> bf16 pairs in TMEM (two buffers); epilogue dQ * scale -> bf16.
//              No exchange between the halves is needed: LSE and D are known.
//   warp 8     producer: work counter, TMA loads of Q_i and dO_i (once per
//              item) and of K_j (3-stage ring) and V_j (2-stage ring).  V_j
//              is free as soon as dP_j is done, K_j only after dQ += dS K_j,
//              so the two rings are separate and K is fetched further ahead.
//   warp 9     S issuer: S_j, as soon as the compute warps have read the
//              previous S tile.
//   warp 11    dP issuer: dP_j, as soon as they have read the previous dP.
//   warp 10    dQ issuer: dQ += dS_j K_j.
//   One thread issues a tcgen05.mma only every ~120 cycles, about twice the
//   time the tensor pipe needs for a 128 x 128 x 16 product, so each of the
//   three products has its own issuing thread (on its own SM sub-partition)
//   and the three streams overlap on the pipe.
// Tensor memory: S [0,128), dP [128,256), dQ [256,384), dS0 [384,448),
// dS1 [448,512).
#include "tc_common.cuh"

namespace prism {
namespace {
using namespace tc;

constexpr int kS = 128, kD = 128;
constexpr int kTile = kS * kD * 2;  // 32 KB
constexpr int kKStages = 3, kVStages = 2;
constexpr int kThreads = 384;
constexpr int kCompute = 256;
constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DQ = 256, TM_DS0 = 384, TM_DS1 = 448;
constexpr int kOffQ = 0, kOffDO = kTile, kOffK = 2 * kTile, kOffV = kOffK + kKStages * kTile;
constexpr int kOffBar = kOffV + kVStages * kTile;

struct DqBars {
  uint64_t qd_full, qd_empty, k_full[kKStages], k_empty[kKStages], v_full[kVStages],
      v_empty[kVStages];
  uint64_t s_full, dp_full, s_free, dp_free, ds_ready[2], ds_empty[2];
  uint64_t dq_done, dq_free, final_bar;
  uint64_t work_full[2], work_empty[2];
  int work_row[2], work_beg[2], work_end[2], work_nvq[2], work_chunk[2];
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kSmemBytes = kOffBar + sizeof(DqBars);
static_assert(kSmemBytes <= 232448, "dynamic shared memory above the per-CTA limit");

struct DqParams {
  const float* lse;
  const float* D;
  const int32_t* n_valid;
  const int32_t* row_ptr;
  const int32_t* col_idx;
  uint16_t* dQp;
  uint16_t* dqpart;  // chunks > 1: partial dQ (scaled, bf16) per (row, key range)
  uint32_t* status;
  long long rows;    // B*H*nb query blocks
  long long items;   // rows * chunks work items
  long long Np;
  int nb;
  int chunks;        // key ranges per head (1: no split)
  int chunk_blocks;  // key blocks per range
  float scale, scale_log2;
  unsigned long long limit;
  int starve;  // fault injection (test only): the producer issues no loads
  const uint8_t* mask;  // blocks of half a tile: sub-tile mask per CSR entry (else null)
};

__global__ void __launch_bounds__(kThreads, 1)
    attn_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmdO, DqParams P) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  DqBars& sm = *reinterpret_cast<DqBars*>(dsm + kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((smem_u32(dsm) & 1023u) != 0) {  // swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) dev_error(P.status, DEV_ERR_BOUNDS, 0xA12, smem_u32(dsm));
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&sm.qd_full, 1);
    mbar_init(&sm.qd_empty, 2);  // the S and the dP issuer
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 2);  // K is read by both issuers
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.dp_full, 1);
    mbar_init(&sm.s_free, kCompute);
    mbar_init(&sm.dp_free, kCompute);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.ds_ready[b], kCompute);
      mbar_init(&sm.ds_empty[b], 1);
      mbar_init(&sm.work_full[b], 1);
      mbar_init(&sm.work_empty[b], 3 + kCompute);
    }
    mbar_init(&sm.dq_done, 1);
    mbar_init(&sm.dq_free, kCompute);
    mbar_init(&sm.final_bar, 3);
    sm.abort = 0;
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(&sm.tmem_base, 512);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = sm.tmem_base;
  const Waiter W{&sm.abort, P.status, P.limit};
  uint8_t* kbuf = dsm + kOffK;  // K stage s at s * kTile
  uint8_t* vbuf = dsm + kOffV;  // V stage s at s * kTile

  if (warp == 8) {
    // ------------------------------------------------------ producer ----
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      uint32_t use = 0, items = 0;
      bool ok = true;
      for (uint32_t it = 0; ok; ++it) {
        const int ws = it & 1;
        if (!W.wait(&sm.work_empty[ws], ((it >> 1) & 1) ^ 1, 61)) break;
        const long long item = atomicAdd(P.status + WS_DQ_QUEUE, 1u);
        if (item >= P.items) {
          sm.work_row[ws] = -1;
          mbar_arrive(&sm.work_full[ws]);
          break;
        }
        // item -> (b, h), key range c, query block i (ranges outermost within
        // a head, so the K / V tiles in use stay in L2)
        const long long per_bh = static_cast<long long>(P.chunks) * P.nb;
        const long long bhi = item / per_bh;
        const int rem = static_cast<int>(item - bhi * per_bh);
        const int c = rem / P.nb;
        const long long row = bhi * P.nb + (rem - c * P.nb);
        int beg = P.row_ptr[row], end = P.row_ptr[row + 1];
        if (P.chunks > 1) {
          const int lo = c * P.chunk_blocks;
          beg = lower_bound_i32(P.col_idx, beg, end, lo);
          end = lower_bound_i32(P.col_idx, beg, end, lo + P.chunk_blocks);
        }
        const int nvq = P.n_valid[row];
        sm.work_row[ws] = static_cast<int>(row);
        sm.work_chunk[ws] = c;
        sm.work_beg[ws] = beg;
        sm.work_end[ws] = nvq > 0 ? end : beg;
        sm.work_nvq[ws] = nvq;
        mbar_arrive(&sm.work_full[ws]);
        if (nvq == 0 || end == beg) continue;
        const long long bh = row / P.nb;
        const int i = static_cast<int>(row % P.nb);
        const int yq = static_cast<int>(bh * P.Np + static_cast<long long>(i) * kS);
        // Q_i, dO_i once the previous item's S / dP products are done
        if (!W.wait(&sm.qd_empty, (items & 1) ^ 1, 62)) break;
        ++items;
        if (!P.starve) {  // fault injection: no loads, consumers time out
          mbar_expect_tx(&sm.qd_full, 2 * kTile);
          tma_load_2d(dsm + kOffQ, &tmQ, &sm.qd_full, 0, yq);
          tma_load_2d(dsm + kOffQ + kTile / 2, &tmQ, &sm.qd_full, 64, yq);
          tma_load_2d(dsm + kOffDO, &tmdO, &sm.qd_full, 0, yq);
          tma_load_2d(dsm + kOffDO + kTile / 2, &tmdO, &sm.qd_full, 64, yq);
        }
        for (int t = beg; t < end; ++t) {
          const int j = P.col_idx[t];
          const int y = static_cast<int>(bh * P.Np + static_cast<long long>(j) * kS);
          const int ks = use % kKStages, vs = use % kVStages;
          if (!W.wait(&sm.k_empty[ks], ((use / kKStages) & 1) ^ 1, 63)) { ok = false; break; }
          uint8_t* kb = kbuf + ks * kTile;
          if (!P.starve) {  // fault injection: no loads, consumers time out
            mbar_expect_tx(&sm.k_full[ks], kTile);
            tma_load_2d(kb, &tmK, &sm.k_full[ks], 0, y);
            tma_load_2d(kb + kTile / 2, &tmK, &sm.k_full[ks], 64, y);
          }
          if (!W.wait(&sm.v_empty[vs], ((use / kVStages) & 1) ^ 1, 60)) { ok = false; break; }
          uint8_t* vb = vbuf + vs * kTile;
          if (!P.starve) {
            mbar_expect_tx(&sm.v_full[vs], kTile);
            tma_load_2d(vb, &tmV, &sm.v_full[vs], 0, y);
            tma_load_2d(vb + kTile / 2, &tmV, &sm.v_full[vs], 64, y);
          }
          ++use;
        }
      }
    }
    __syncwarp();
  } else if (warp == 9 || warp == 11) {
    // ------------------------------------------------ S issuer, dP issuer ----
    if (lane == 0) {
      const bool is_s = warp == 9;
      constexpr uint32_t id_kk = idesc_bf16(128, 128, 0, 0);
      // S = Q K^T reads Q and K; dP = dO V^T reads dO and V
      const uint64_t ad = sdesc_sw128(smem_u32(dsm + (is_s ? kOffQ : kOffDO)), 16, 1024);
      uint8_t* bbuf = is_s ? kbuf : vbuf;
      const int nst = is_s ? kKStages : kVStages;
      uint64_t* full = is_s ? sm.k_full : sm.v_full;
      uint64_t* empty = is_s ? sm.k_empty : sm.v_empty;
      uint64_t* done = is_s ? &sm.s_full : &sm.dp_full;
      uint64_t* freed = is_s ? &sm.s_free : &sm.dp_free;
      const uint32_t dt = tmem + (is_s ? TM_S : TM_DP);
      const uint32_t wbase = is_s ? 64 : 90;  // wait-site codes
      auto koff = [](int kk) {
        return static_cast<uint64_t>(((kk >> 2) * (kTile / 2) + (kk & 3) * 32) >> 4);
      };
      uint32_t use = 0, items = 0, idx = 0;
      bool ok = true;
      for (uint32_t it = 0; ok; ++it) {
        const int ws = it & 1;
        if (!W.wait(&sm.work_full[ws], (it >> 1) & 1, wbase)) break;
        if (sm.work_row[ws] < 0) break;
        const int n = sm.work_end[ws] - sm.work_beg[ws];
        if (n > 0) {
          if (!W.wait(&sm.qd_full, items & 1, wbase + 1)) break;
          ++items;
          for (int jj = 0; jj < n; ++jj) {
            const int st = use % nst;
            if (!W.wait(&full[st], (use / nst) & 1, wbase + 2)) { ok = false; break; }
            // the compute warps have read this product's previous tile
            if (idx > 0 && !W.wait(freed, (idx - 1) & 1, wbase + 3)) { ok = false; break; }
            fence_after();
            const uint64_t bd = sdesc_sw128(smem_u32(bbuf + st * kTile), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_ss(dt, ad + koff(kk), bd + koff(kk), id_kk, kk > 0 ? 1u : 0u);
            commit(done);
            commit(&empty[st]);
            ++use;
            ++idx;
          }
          if (ok) commit(&sm.qd_empty);
        }
        if (ok) mbar_arrive(&sm.work_empty[ws]);
      }
      commit(&sm.final_bar);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ------------------------------------------------------ issuer B: dQ ----
    if (lane == 0) {
      constexpr uint32_t id_kn = idesc_bf16(128, 128, 0, 1);  // A = dS (TMEM), B = K MN-major
      uint32_t use = 0, gidx = 0, items = 0;
      bool ok = true;
      for (uint32_t it = 0; ok; ++it) {
        const int ws = it & 1;
        if (!W.wait(&sm.work_full[ws], (it >> 1) & 1, 71)) break;
        if (sm.work_row[ws] < 0) break;
        const int n = sm.work_end[ws] - sm.work_beg[ws];
        if (n > 0) {
          // the previous item's dQ has been read out before it is overwritten
          if (items > 0 && !W.wait(&sm.dq_free, (items - 1) & 1, 72)) break;
          ++items;
          for (int jj = 0; jj < n; ++jj) {
            const uint32_t b = gidx & 1;
            if (!W.wait(&sm.ds_ready[b], (gidx >> 1) & 1, 73)) { ok = false; break; }
            const int ks = use % kKStages;
            if (!W.wait(&sm.k_full[ks], (use / kKStages) & 1, 74)) { ok = false; break; }
            fence_after();
            const uint64_t kd = sdesc_sw128(smem_u32(kbuf + ks * kTile), kTile / 2, 1024);
            const uint32_t a = tmem + (b ? TM_DS1 : TM_DS0);
#pragma unroll
            for (int kk = 0; kk < kS / 16; ++kk)
              mma_ts(tmem + TM_DQ, a + kk * 8, kd + static_cast<uint64_t>((kk * 2048) >> 4), id_kn,
                     (jj > 0 || kk > 0) ? 1u : 0u);
            commit(&sm.ds_empty[b]);
            commit(&sm.k_empty[ks]);
            ++use;
            ++gidx;
          }
          if (ok) commit(&sm.dq_done);
        }
        if (ok) mbar_arrive(&sm.work_empty[ws]);
      }
      commit(&sm.final_bar);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------ compute ----
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;  // query row == TMEM lane
    const uint32_t lb = static_cast<uint32_t>(quarter * 32) << 16;
    const int c0 = half * 64;  // first key column (and dQ channel) of this half
    uint32_t sidx = 0, gidx = 0, items = 0;
    for (uint32_t it = 0;; ++it) {
      const int ws = it & 1;
      if (!W.wait(&sm.work_full[ws], (it >> 1) & 1, 81)) break;
      const int row = sm.work_row[ws];
      if (row < 0) break;
      const int beg = sm.work_beg[ws], n = sm.work_end[ws] - beg, nvq = sm.work_nvq[ws];
      const long long bh = row / P.nb;
      const int i = row % P.nb;
      const long long grow = bh * P.Np + static_cast<long long>(i) * kS + r;
      // output row: the final dQ, or this key range's partial dQ
      const long long prow =
          (static_cast<long long>(row) * P.chunks + sm.work_chunk[ws]) * kS + r;
      uint4* drow =
          reinterpret_cast<uint4*>(P.chunks > 1 ? P.dqpart + prow * kD : P.dQp + grow * kD) +
          half * 8;
      if (n == 0) {
        // (with key ranges, the combining kernel handles empty ranges)
        if (P.chunks == 1) {
#pragma unroll
          for (int q = 0; q < 8; ++q) drow[q] = make_uint4(0, 0, 0, 0);
        }
        mbar_arrive(&sm.work_empty[ws]);
        continue;
      }
      const bool real = r < nvq;
      const float lse2 = P.lse[grow] * 1.4426950408889634f;
      const float Dr = P.D[grow];
      // real-token counts of the listed key blocks, fetched ahead of use:
      // the block index two key blocks ahead, its count one block ahead
      const int32_t* nvb = P.n_valid + bh * P.nb;
      const int32_t* cols = P.col_idx + beg;
      int nvk_next = nvb[cols[0]];
      int j_next2 = n > 1 ? cols[1] : 0;
      // blocks of half a tile: bit 2 qh + kh of an entry's mask set = this
      // row half (qh) does not attend that key half (kh = this column half)
      const int mbit = (quarter >> 1) * 2 + half;
      bool ok = true;
      for (int jj = 0; jj < n; ++jj) {
        const int nvk = nvk_next;
        if (jj + 1 < n) nvk_next = nvb[j_next2];
        if (jj + 2 < n) j_next2 = cols[jj + 2];
        const bool act = P.mask == nullptr || !((P.mask[beg + jj] >> mbit) & 1);
        const int lim = (real && act) ? nvk - c0 : 0;  // real key columns of this half
        // wait results are made warp-uniform: TMEM loads and stores are
        // warp-collective
        if (!__all_sync(0xffffffffu, W.wait(&sm.s_full, sidx & 1, 82))) { ok = false; break; }
        fence_after();
        uint32_t sv[2][32], dp[2][32];
        tmem_ld32(tmem + lb + TM_S + c0, sv[0]);
        tmem_ld32(tmem + lb + TM_S + c0 + 32, sv[1]);
        tmem_ld_wait();
        fence_before();
        mbar_arrive(&sm.s_free);
        if (!__all_sync(0xffffffffu, W.wait(&sm.dp_full, sidx & 1, 83))) { ok = false; break; }
        fence_after();
        tmem_ld32(tmem + lb + TM_DP + c0, dp[0]);
        tmem_ld32(tmem + lb + TM_DP + c0 + 32, dp[1]);
        tmem_ld_wait();
        fence_before();
        mbar_arrive(&sm.dp_free);
        ++sidx;
        uint32_t pk[32];
        if (lim >= 64) {
          // two keys per fp32x2 instruction: x = s * c - LSE log2 e, dS = P (dP - D)
          const f32x2 c2 = pack2(P.scale_log2, P.scale_log2), nl2 = pack2(-lse2, -lse2);
          const f32x2 D2 = pack2(Dr, Dr);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int k0 = 2 * e, k1 = k0 + 1;
            const f32x2 x2 = fma2(pack2(__uint_as_float(sv[k0 >> 5][k0 & 31]),
                                        __uint_as_float(sv[k1 >> 5][k1 & 31])),
                                  c2, nl2);
            float x0, x1;
            unpack2(x2, x0, x1);
            const f32x2 ds2 = mul2(pack2(ex2(x0), ex2(x1)),
                                   sub2(pack2(__uint_as_float(dp[k0 >> 5][k0 & 31]),
                                              __uint_as_float(dp[k1 >> 5][k1 & 31])),
                                        D2));
            float d0, d1;
            unpack2(ds2, d0, d1);
            pk[e] = pack_bf16x2(d0, d1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int k0 = 2 * e, k1 = k0 + 1;
            const float p0 = k0 < lim ? ex2(fmaf(__uint_as_float(sv[k0 >> 5][k0 & 31]), P.scale_log2, -lse2)) : 0.f;
            const float p1 = k1 < lim ? ex2(fmaf(__uint_as_float(sv[k1 >> 5][k1 & 31]), P.scale_log2, -lse2)) : 0.f;
            pk[e] = pack_bf16x2(p0 * (__uint_as_float(dp[k0 >> 5][k0 & 31]) - Dr),
                                p1 * (__uint_as_float(dp[k1 >> 5][k1 & 31]) - Dr));
          }
        }
        // the dQ product that read this dS buffer two key blocks ago is done
        const uint32_t b = gidx & 1;
        if (!__all_sync(0xffffffffu, gidx < 2 || W.wait(&sm.ds_empty[b], ((gidx >> 1) - 1) & 1, 84))) {
          ok = false;
          break;
        }
        fence_after();
        tmem_st32(tmem + lb + (b ? TM_DS1 : TM_DS0) + half * 32, pk);
        tmem_st_wait();
        fence_before();
        mbar_arrive(&sm.ds_ready[b]);
        ++gidx;
      }
      if (!ok) break;
      // epilogue: dQ * scale -> bf16, this half of the channels
      if (!__all_sync(0xffffffffu, W.wait(&sm.dq_done, items & 1, 85))) break;
      ++items;
      fence_after();
      const float mul = real ? P.scale : 0.f;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lb + TM_DQ + c0 + c * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * mul, __uint_as_float(o[8 * q + 1]) * mul);
          v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * mul, __uint_as_float(o[8 * q + 3]) * mul);
          v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * mul, __uint_as_float(o[8 * q + 5]) * mul);
          v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * mul, __uint_as_float(o[8 * q + 7]) * mul);
          drow[c * 4 + q] = v;
        }
      }
      fence_before();
      mbar_arrive(&sm.dq_free);
      mbar_arrive(&sm.work_empty[ws]);
    }
  }

  // ---------------------------------------------------------- teardown ----
  __syncthreads();
  if (warp == 0) {
    if (!wait_raw(&sm.final_bar, 0, P.limit) && lane == 0)
      dev_error(P.status, DEV_ERR_TIMEOUT, 299, 0);
    fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_attn_dq_tc(const Plan& p, const uint16_t* Qp, const uint16_t* Kp,
                              const uint16_t* Vp, const uint16_t* dOp, const float* lse,
                              const float* D, const int32_t* n_valid, const int32_t* row_ptr,
                              const int32_t* col_idx, float scale, uint16_t* dQp, uint8_t* ws,
                              uint16_t* dqpart, cudaStream_t st) {
  const prism_config_t& c = p.cfg;
  const long long rows_total = static_cast<long long>(c.B) * c.H * p.sz.Np;
  CUtensorMap tmQ, tmK, tmV, tmdO;
  if (!make_tile_map(&tmQ, Qp, rows_total) || !make_tile_map(&tmK, Kp, rows_total) ||
      !make_tile_map(&tmV, Vp, rows_total) || !make_tile_map(&tmdO, dOp, rows_total))
    return cudaErrorInvalidValue;
  DqParams a;
  a.lse = lse;
  a.D = D;
  a.n_valid = n_valid;
  a.row_ptr = row_ptr;
  a.col_idx = col_idx;
  a.dQp = dQp;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.rows = static_cast<long long>(c.B) * c.H * p.sz.nb;
  a.dqpart = dqpart;
  a.chunks = dqpart != nullptr ? p.sz.key_chunks : 1;
  a.chunk_blocks = a.chunks > 1 ? p.sz.chunk_blocks : p.sz.nb;
  a.items = a.rows * a.chunks;
  a.Np = p.sz.Np;
  a.nb = p.sz.nb;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.limit = c.timeout_cycles ? c.timeout_cycles : 4000000000ull;
  a.starve = c.fault_inject == PRISM_FAULT_STARVE_LOADS ? 1 : 0;
  a.mask = (p.sz.half_tile && ws != nullptr) ? ws + p.sz.ws_csr_mask : nullptr;
  cudaError_t e = cudaMemsetAsync(a.status + WS_DQ_QUEUE, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const long long g = a.items < sm_count() ? a.items : sm_count();
  attn_dq_tc_kernel<<<static_cast<unsigned>(g), kThreads, kSmemBytes, st>>>(tmQ, tmK, tmV, tmdO,
                                                                             a);
  return cudaGetLastError();
}

}  // namespace prism
