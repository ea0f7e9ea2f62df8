// Block-sparse attention forward on the 5th-generation tensor cores
// (tcgen05 + tensor memory), 128-token blocks, head dim 128, bf16 in, fp32
// accumulation.
//
// Prism (arXiv 2610.05416), Fig. 2 caption: each query block attends only to
// the key blocks selected for it.  Reading used here: exact softmax over the
// real tokens of the selected key blocks, scale `scale`, natural-log LSE.
//
// Design (one persistent CTA per SM, 352 threads, warp-specialised):
//   warp 8  producer: takes the next work item -- a query block and one
//           range of the head's key blocks (the whole range unless the plan
//           splits it; see combine.cu) -- from a global work counter,
//           publishes it in a 2-slot work ring, and streams the K and V tiles
//           of its selected key blocks in that range into two 3-stage rings
//           with TMA (128-byte swizzle, 2 boxes of 64 x 128 per tile).  A K
//           tile is free once its score tile is done, long before the V tile
//           of the same key block, so the rings are separate.
//   warp 9  S issuer (one thread): S = Q K^T with Q held in tensor memory
//           (A from TMEM, B = K tile from smem), as soon as the softmax warps
//           have read the previous S tile, so the next score tile is on the
//           tensor pipe while they work on this one.  (Two 128 x 64 score
//           tiles, one per column half, would let the halves drift apart, but
//           N = 64 products issue at about the same cost as N = 128 ones.)
//   warp 10 PV issuer (one thread): O_h += P_h V_h for each column half h
//           (keys 64h..64h+63; A = P from TMEM, B = V rows from smem,
//           MN-major), as soon as that half's P is in.  Two issuing threads
//           keep the tensor pipe fed: a tcgen05.mma issue blocks while the
//           pipe's queue is full, and each issuer's waits overlap the other's
//           MMAs.
//   warps 0-7  softmax, two independent halves: warps w and w+4 share the
//           query rows of TMEM lane quarter w%4 (thread = query row) and split
//           the 128 key columns.  Each half keeps its own running max m_h,
//           row sum l_h and output accumulator O_h = sum_j P_h V_h (all 128
//           channels), so the halves never wait for each other inside a query
//           block and the exp work of one overlaps the loads, maxima and
//           waits of the other.  Online softmax in the log2 domain with lazy
//           rescaling: O_h is rescaled only when m_h grows by more than
//           kRescaleLog2 (P stays below 2^kRescaleLog2, far inside the bf16
//           and fp32 ranges).
//           At the end of the query block the halves meet once and combine:
//           O = (O_0 2^(m_0-M) + O_1 2^(m_1-M)) / (l_0 2^(m_0-M) + l_1 2^(m_1-M)),
//           M = max(m_0, m_1); each half writes 64 of the output channels.
// Tensor memory (512 columns): S [0,128), O_0 [128,256), O_1 [256,384),
// Q [384,448), P [448,512) (half h: [448+32h, 480+32h)).
// Every wait is bounded: on expiry the CTA raises a flag, records the error in
// the workspace status word, and every role stops issuing and leaves.
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace prism {
namespace {
using namespace tc;

constexpr int kS = 128;
constexpr int kD = 128;
constexpr int kTile = kS * kD * 2;  // 32 KB
constexpr int kKStages = 3, kVStages = 3;
constexpr int kFwdThreads = 352;
constexpr float kRescaleLog2 = 16.f;
constexpr int kSoftmaxThreads = 256;
constexpr uint32_t TM_S = 0, TM_O0 = 128, TM_O1 = 256, TM_Q = 384, TM_P = 448;

struct FwdShared {
  uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
  uint64_t s_full, s_free, p_full[2], p_empty[2], q_ready, final_bar;  // p_*: per column half
  uint64_t work_full[2], work_empty[2];
  int work_row[2], work_beg[2], work_end[2], work_nvq[2], work_chunk[2];
  float xm[2][128];       // [column half][row]: running max at the end of a query block
  float xl[2][128];       // [column half][row]: row sum at the end of a query block
  int xok[2][2][4];       // [exchange parity][column half][lane quarter]: still on track
  uint32_t tmem_base;
  int abort;
};

struct FwdParams {
  const uint16_t* Qp;
  const int32_t* n_valid;
  const int32_t* row_ptr;
  const int32_t* col_idx;
  uint16_t* Op;
  float* lse;
  uint32_t* status;
  long long rows;
  long long items;    // rows * chunks
  long long Np;
  int nb;
  int chunks;         // key ranges per head (1: no split)
  int chunk_blocks;   // key blocks per range
  uint16_t* Opart;    // chunks > 1: normalised partial O per (row, range)
  float* ml;          // chunks > 1: (max in log2 units, row sum) per (row, range, query row)
  float scale_log2;
  unsigned long long limit;
  int starve;  // fault injection (test only): the producer issues no loads
  const uint8_t* mask;  // blocks of half a tile: sub-tile mask per CSR entry (else null)
};

__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, FwdParams P) {
  extern __shared__ uint8_t dsm_raw[];
  __shared__ FwdShared sm;
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  uint8_t* kbuf = dsm;                     // K stage s at s * kTile
  uint8_t* vbuf = dsm + kKStages * kTile;  // V stage s at s * kTile
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);  // released by the S issuer
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);  // released by the PV issuer
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.s_free, kSoftmaxThreads);
    mbar_init(&sm.p_full[0], kSoftmaxThreads / 2);
    mbar_init(&sm.p_full[1], kSoftmaxThreads / 2);
    mbar_init(&sm.p_empty[0], 1);
    mbar_init(&sm.p_empty[1], 1);
    mbar_init(&sm.q_ready, kSoftmaxThreads);
    mbar_init(&sm.final_bar, 2);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.work_full[s], 1);
      mbar_init(&sm.work_empty[s], 2 + kSoftmaxThreads);
    }
    sm.abort = 0;
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(&sm.tmem_base, 512);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = sm.tmem_base;
  const Waiter W{&sm.abort, P.status, P.limit};
  uint32_t* queue = P.status + WS_FWD_QUEUE;

  if (warp == 8) {
    // ------------------------------------------------------ producer ----
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint32_t use = 0;
      for (uint32_t it = 0;; ++it) {
        const int ws = it & 1;
        if (!W.wait(&sm.work_empty[ws], ((it >> 1) & 1) ^ 1, 1)) break;
        const long long item = atomicAdd(queue, 1u);
        if (item >= P.items) {
          sm.work_row[ws] = -1;
          mbar_arrive(&sm.work_full[ws]);
          break;
        }
        // item -> (b, h), key range c, query block i: within a head all query
        // blocks take range 0, then range 1, ... so the K / V tiles in use
        // stay in L2
        const long long per_bh = static_cast<long long>(P.chunks) * P.nb;
        const long long bh = item / per_bh;
        const int rem = static_cast<int>(item - bh * per_bh);
        const int c = rem / P.nb;
        const long long row = bh * P.nb + (rem - c * P.nb);
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
        if (nvq == 0) continue;
        bool ok = true;
        for (int t = beg; t < end; ++t) {
          const int j = P.col_idx[t];
          const int y = static_cast<int>(bh * P.Np + static_cast<long long>(j) * kS);
          const int ks = use % kKStages, vs = use % kVStages;
          if (!W.wait(&sm.k_empty[ks], ((use / kKStages) & 1) ^ 1, 2)) { ok = false; break; }
          uint8_t* kb = kbuf + ks * kTile;
          if (!P.starve) {  // fault injection: no loads, consumers time out
            mbar_expect_tx(&sm.k_full[ks], kTile);
            tma_load_2d(kb, &tmK, &sm.k_full[ks], 0, y);
            tma_load_2d(kb + kTile / 2, &tmK, &sm.k_full[ks], 64, y);
          }
          if (!W.wait(&sm.v_empty[vs], ((use / kVStages) & 1) ^ 1, 3)) { ok = false; break; }
          uint8_t* vb = vbuf + vs * kTile;
          if (!P.starve) {
            mbar_expect_tx(&sm.v_full[vs], kTile);
            tma_load_2d(vb, &tmV, &sm.v_full[vs], 0, y);
            tma_load_2d(vb + kTile / 2, &tmV, &sm.v_full[vs], 64, y);
          }
          ++use;
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------ S issuer ----
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, 128, 0, 0);  // A = Q (TMEM), B = K, K-major
      uint32_t use = 0, sidx = 0, qcnt = 0;
      bool ok = true;
      for (uint32_t it = 0; ok; ++it) {
        const int ws = it & 1;
        if (!W.wait(&sm.work_full[ws], (it >> 1) & 1, 4)) break;
        if (sm.work_row[ws] < 0) break;
        const int n = sm.work_end[ws] - sm.work_beg[ws];
        if (n > 0) {
          if (!W.wait(&sm.q_ready, qcnt & 1, 5)) break;
          ++qcnt;
          for (int jj = 0; jj < n; ++jj) {
            if (jj > 0 && !W.wait(&sm.s_free, (sidx - 1) & 1, 6)) { ok = false; break; }
            const int ks = use % kKStages;
            if (!W.wait(&sm.k_full[ks], (use / kKStages) & 1, 9)) { ok = false; break; }
            fence_after();
            const uint64_t kd = sdesc_sw128(smem_u32(kbuf + ks * kTile), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_ts(tmem + TM_S, tmem + TM_Q + kk * 8,
                     kd + static_cast<uint64_t>(((kk >> 2) * (kTile / 2) + (kk & 3) * 32) >> 4), idS,
                     kk > 0 ? 1u : 0u);
            commit(&sm.s_full);
            commit(&sm.k_empty[ks]);
            ++use;
            ++sidx;
          }
        }
        if (ok) mbar_arrive(&sm.work_empty[ws]);
      }
      commit(&sm.final_bar);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ------------------------------------------------------ PV issuer ----
    if (lane == 0) {
      constexpr uint32_t idPV = idesc_bf16(128, 128, 0, 1);  // A = P (TMEM), B = V, MN-major
      uint32_t use = 0, pidx = 0, qcnt = 0;
      bool ok = true;
      for (uint32_t it = 0; ok; ++it) {
        const int ws = it & 1;
        if (!W.wait(&sm.work_full[ws], (it >> 1) & 1, 14)) break;
        if (sm.work_row[ws] < 0) break;
        const int n = sm.work_end[ws] - sm.work_beg[ws];
        if (n > 0) {
          // the first PV overwrites O_h: the previous block's epilogue has read it
          if (!W.wait(&sm.q_ready, qcnt & 1, 15)) break;
          ++qcnt;
          for (int jj = 0; jj < n; ++jj) {
            const int vs = use % kVStages;
            const uint64_t vd = sdesc_sw128(smem_u32(vbuf + vs * kTile), kTile / 2, 1024);
            for (int h = 0; h < 2; ++h) {
              if (!W.wait(&sm.p_full[h], pidx & 1, 7)) { ok = false; break; }
              if (h == 0 && !W.wait(&sm.v_full[vs], (use / kVStages) & 1, 8)) { ok = false; break; }
              fence_after();
              const uint32_t o = tmem + (h ? TM_O1 : TM_O0);
#pragma unroll
              for (int k4 = 0; k4 < kS / 32; ++k4) {
                const int kk = h * (kS / 32) + k4;  // 16-key step: keys 16kk .. 16kk+15
                mma_ts(o, tmem + TM_P + kk * 8, vd + static_cast<uint64_t>((kk * 2048) >> 4), idPV,
                       (jj > 0 || k4 > 0) ? 1u : 0u);
              }
              commit(&sm.p_empty[h]);
            }
            if (!ok) break;
            commit(&sm.v_empty[vs]);
            ++use;
            ++pidx;
          }
        }
        if (ok) mbar_arrive(&sm.work_empty[ws]);
      }
      commit(&sm.final_bar);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ softmax ----
    // Warps w and w+4 meet at a named barrier (64 threads) three times per
    // query block: at its start, before the epilogue and after it.  A named
    // barrier has no time limit, so the two never leave a loop on their own:
    // every bounded wait only clears `ok`, the flags are exchanged at each
    // meeting, and both warps leave together at the first meeting after
    // either of them failed.  (A half that stops inside the key-block loop
    // stops arriving at s_free; the S issuer's bounded wait then runs out and
    // the other half's next wait sees the abort flag.)
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;  // query row of the block == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + TM_S + half * 64;
    const uint32_t tO = tmem + lane_base + (half ? TM_O1 : TM_O0);  // this half's accumulator
    const uint32_t tP = tmem + lane_base + TM_P + half * 32;
    const int c0 = half * 64;  // first key column (and output channel) of this half
    uint32_t xpar = 0;         // parity of the flag slots of the next meeting
    auto meet = [&](bool mine) -> bool {  // pair barrier, returns both flags ANDed
      mine = __all_sync(0xffffffffu, mine);  // one flag per warp
      const int slot = xpar & 1;
      ++xpar;
      if (lane == 0) sm.xok[slot][half][quarter] = mine ? 1 : 0;
      asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
      return mine && sm.xok[slot][half ^ 1][quarter] != 0;
    };
    // wait until column half h's PV of key block g (CTA-local count) is done
    auto pv_done = [&](int h, uint32_t g, uint32_t where) {
      return W.wait(&sm.p_empty[h], g & 1, where);
    };
    uint32_t sidx = 0, pidx = 0;
    bool ok = true;
    bool s_ready = false;  // early look at the next S tile, taken after the last P store
    for (uint32_t it = 0;; ++it) {
      const int ws = it & 1;
      ok = meet(ok && W.wait(&sm.work_full[ws], (it >> 1) & 1, 10));
      if (!ok) break;
      const int row = sm.work_row[ws];
      if (row < 0) break;
      const int beg = sm.work_beg[ws], n = sm.work_end[ws] - beg, nvq = sm.work_nvq[ws];
      const int chunk = sm.work_chunk[ws];
      const long long bh = row / P.nb;
      const int i = row % P.nb;
      const long long grow = bh * P.Np + static_cast<long long>(i) * kS + r;
      // output row: the final O, or this key range's normalised partial O
      const long long prow = (static_cast<long long>(row) * P.chunks + chunk) * kS + r;
      uint4* orow = reinterpret_cast<uint4*>(P.chunks > 1 ? P.Opart + prow * kD : P.Op + grow * kD) +
                    half * 8;
      if (n == 0) {
        // (with key ranges, the combining kernel handles empty ranges)
        if (P.chunks == 1) {
#pragma unroll
          for (int q = 0; q < 8; ++q) orow[q] = make_uint4(0, 0, 0, 0);
          if (half == 0) P.lse[grow] = 0.f;
        }
        mbar_arrive(&sm.work_empty[ws]);
        continue;
      }
      {
        // this half of the row of Q -> tensor memory (bf16 pairs, 32 columns)
        const uint4* qrow = reinterpret_cast<const uint4*>(P.Qp + grow * kD) + half * 8;
        uint32_t a[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 v = ldg_nc_v4(qrow + q);
          a[4 * q] = v.x; a[4 * q + 1] = v.y; a[4 * q + 2] = v.z; a[4 * q + 3] = v.w;
        }
        tmem_st32(tmem + lane_base + TM_Q + half * 32, a);
        tmem_st_wait();
        fence_before();
        mbar_arrive(&sm.q_ready);
      }
      float m = -INFINITY, l = 0.f;  // this half's running max (log2 units) and row sum
      // real-token counts of the listed key blocks, fetched ahead of use:
      // the block index two key blocks ahead, its count one block ahead
      const int32_t* nvb = P.n_valid + bh * P.nb;
      const int32_t* cols = P.col_idx + beg;
      int nvk_next = nvb[cols[0]];
      int j_next2 = n > 1 ? cols[1] : 0;
      // blocks of half a tile: bit 2 qh + kh of an entry's mask set = this
      // row half (qh) does not attend that key half (kh = this column half)
      const int mbit = (quarter >> 1) * 2 + half;
      for (int jj = 0; jj < n; ++jj) {
        const int nvk = nvk_next;
        if (jj + 1 < n) nvk_next = nvb[j_next2];
        if (jj + 2 < n) j_next2 = cols[jj + 2];
        const bool act = P.mask == nullptr || !((P.mask[beg + jj] >> mbit) & 1);
        const int lim = act ? nvk - c0 : 0;  // columns of this half that hold real keys
        // wait results are made warp-uniform: the TMEM loads and stores
        // below are warp-collective
        ok = __all_sync(0xffffffffu, ok && (s_ready || W.wait(&sm.s_full, sidx & 1, 11)));
        ++sidx;
        if (!ok) break;
        uint32_t s[2][32];
        float mx = -INFINITY;
        fence_after();
        tmem_ld32(tS, s[0]);
        tmem_ld32(tS + 32, s[1]);
        tmem_ld_wait();
        fence_before();
        mbar_arrive(&sm.s_free);
        if (lim >= 64) {
          // four independent chains of three-input maxima (depth 8, not 64)
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float& a = m4[c * 2 + ((e >> 4) & 1)];
              a = fmax3(a, __uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1]));
            }
          mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
        } else {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c * 32 + e < lim) mx = fmaxf(mx, __uint_as_float(s[c][e]));
        }
        mx *= P.scale_log2;
        const bool resc = mx > m + kRescaleLog2;
        const float m_new = resc ? mx : m;
        const float corr = resc ? ex2(m - m_new) : 1.f;
        // this half's P buffer and O_h are free once its previous PV is done
        bool pv_prev = pidx == 0 || mbar_test(&sm.p_empty[half], (pidx - 1) & 1);
        if (jj > 0 && __any_sync(0xffffffffu, resc)) {
          if (!pv_prev) ok = ok && pv_done(half, pidx - 1, 12);
          ok = __all_sync(0xffffffffu, ok);
          pv_prev = true;
          if (ok) {
            fence_after();
#pragma unroll
            for (int c = 0; c < kD / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
              tmem_st32(tO + c * 32, o);
            }
            tmem_st_wait();
          }
        }
        l *= corr;
        m = m_new;
        float lsum = 0.f;
        uint32_t pk[32];
        if (lim >= 64) {
          // two keys per fp32x2 instruction: x = s * c - m, partial row sums
          const f32x2 c2 = pack2(P.scale_log2, P.scale_log2), nm2 = pack2(-m, -m);
          f32x2 ls2[2] = {pack2(0.f, 0.f), pack2(0.f, 0.f)};
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int k0 = 2 * e;
            const f32x2 x2 = fma2(pack2(__uint_as_float(s[k0 >> 5][k0 & 31]),
                                        __uint_as_float(s[(k0 + 1) >> 5][(k0 + 1) & 31])),
                                  c2, nm2);
            float x0, x1;
            unpack2(x2, x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            ls2[e & 1] = add2(ls2[e & 1], pack2(p0, p1));
            pk[e] = pack_bf16x2(p0, p1);
          }
          float a0, a1, b0, b1;
          unpack2(ls2[0], a0, a1);
          unpack2(ls2[1], b0, b1);
          lsum = (a0 + b0) + (a1 + b1);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int k0 = 2 * e;
            const float p0 = k0 < lim ? ex2(fmaf(__uint_as_float(s[k0 >> 5][k0 & 31]), P.scale_log2, -m)) : 0.f;
            const float p1 = k0 + 1 < lim ? ex2(fmaf(__uint_as_float(s[(k0 + 1) >> 5][(k0 + 1) & 31]), P.scale_log2, -m)) : 0.f;
            lsum += p0 + p1;
            pk[e] = pack_bf16x2(p0, p1);
          }
        }
        l += lsum;
        if (!pv_prev) ok = ok && pv_done(half, pidx - 1, 16);
        ok = __all_sync(0xffffffffu, ok);
        ++pidx;
        if (!ok) break;
        fence_after();
        tmem_st32(tP, pk);
        tmem_st_wait();
        fence_before();
        mbar_arrive(&sm.p_full[half]);
        s_ready = mbar_test(&sm.s_full, sidx & 1);  // the next S tile, most often done
      }
      // epilogue: both halves' last PV done, then combine the two halves
      sm.xm[half][r] = m;
      sm.xl[half][r] = l;
      ok = meet(ok);
      if (!ok) break;
      ok = __all_sync(0xffffffffu, ok && pv_done(0, pidx - 1, 13) && pv_done(1, pidx - 1, 17));
      if (ok) {
        fence_after();
        const float m0 = sm.xm[0][r], m1 = sm.xm[1][r];
        const float M = fmaxf(m0, m1);
        // no key at all for this row in this item (possible only with
        // sub-tile masks, within one key range): O = 0, weight 0
        const bool none = !(M > -INFINITY);
        const float a0 = none ? 0.f : ex2(m0 - M), a1 = none ? 0.f : ex2(m1 - M);
        const float lt = sm.xl[0][r] * a0 + sm.xl[1][r] * a1;
        const bool real = r < nvq;
        const float inv = (real && !none) ? 1.f / lt : 0.f;
        const float w0 = a0 * inv, w1 = a1 * inv;
        const uint32_t tO0 = tmem + lane_base + TM_O0 + c0, tO1 = tmem + lane_base + TM_O1 + c0;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t o0[32], o1[32];
          tmem_ld32(tO0 + c * 32, o0);
          tmem_ld32(tO1 + c * 32, o1);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              v[e] = fmaf(__uint_as_float(o0[8 * q + e]), w0, __uint_as_float(o1[8 * q + e]) * w1);
            uint4 u;
            u.x = pack_bf16x2(v[0], v[1]);
            u.y = pack_bf16x2(v[2], v[3]);
            u.z = pack_bf16x2(v[4], v[5]);
            u.w = pack_bf16x2(v[6], v[7]);
            orow[c * 4 + q] = u;
          }
        }
        if (half == 0) {
          if (P.chunks == 1)
            P.lse[grow] = (real && !none) ? (M + log2f(lt)) * 0.69314718055994531f : 0.f;
          else
            reinterpret_cast<float2*>(P.ml)[prow] = make_float2(M, none ? 0.f : lt);
        }
      }
      // both halves have read O_0, O_1, xm and xl before either moves on
      ok = meet(ok);
      if (!ok) break;
      fence_before();
      mbar_arrive(&sm.work_empty[ws]);
    }
  }

  // ---------------------------------------------------------- teardown ----
  __syncthreads();
  if (warp == 0) {
    // every MMA this CTA issued has completed before the columns are freed
    if (!wait_raw(&sm.final_bar, 0, P.limit) && lane == 0)
      dev_error(P.status, DEV_ERR_TIMEOUT, 99, 0);
    fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D map over a [rows, 128] bf16 matrix, box 64 x 128 (128-byte rows),
// 128-byte swizzle: one box is one half (64 channels) of a 128-row tile.
bool make_tile_map(CUtensorMap* m, const void* base, long long rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kS)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

cudaError_t launch_attn_fwd_tc(const Plan& p, const uint16_t* Qp, const uint16_t* Kp,
                               const uint16_t* Vp, const int32_t* n_valid, const int32_t* row_ptr,
                               const int32_t* col_idx, float scale, uint16_t* Op, float* lse,
                               uint8_t* ws, cudaStream_t st) {
  const prism_config_t& c = p.cfg;
  const long long rows_total = static_cast<long long>(c.B) * c.H * p.sz.Np;
  CUtensorMap tmK, tmV;
  if (!make_tile_map(&tmK, Kp, rows_total) || !make_tile_map(&tmV, Vp, rows_total))
    return cudaErrorInvalidValue;
  FwdParams a;
  a.Qp = Qp;
  a.n_valid = n_valid;
  a.row_ptr = row_ptr;
  a.col_idx = col_idx;
  a.Op = Op;
  a.lse = lse;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.rows = static_cast<long long>(c.B) * c.H * p.sz.nb;
  a.items = a.rows * p.sz.key_chunks;
  a.Np = p.sz.Np;
  a.nb = p.sz.nb;
  a.chunks = p.sz.key_chunks;
  a.chunk_blocks = p.sz.chunk_blocks;
  a.Opart = reinterpret_cast<uint16_t*>(ws + p.off_part);
  a.ml = reinterpret_cast<float*>(ws + p.off_ml);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.limit = c.timeout_cycles ? c.timeout_cycles : 4000000000ull;
  a.starve = c.fault_inject == PRISM_FAULT_STARVE_LOADS ? 1 : 0;
  a.mask = p.sz.half_tile ? ws + p.sz.ws_csr_mask : nullptr;
  cudaError_t e = cudaMemsetAsync(a.status + WS_FWD_QUEUE, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  const size_t smem = static_cast<size_t>(kKStages + kVStages) * kTile + 1024;  // K, V rings
  e = cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long g = a.items < sm_count() ? a.items : sm_count();
  attn_fwd_tc_kernel<<<static_cast<unsigned>(g), kFwdThreads, smem, st>>>(tmK, tmV, a);
  return cudaGetLastError();
}

}  // namespace prism
