// Block-sparse attention forward on the 5th-generation tensor cores
// (tcgen05 + tensor memory), 128-token blocks, head dim 128, bf16 in, fp32
// accumulation.
//
// Prism (arXiv 2610.05416), Fig. 2 caption: each query block attends only to
// the key blocks selected for it.  Reading used here: exact softmax over the
// real tokens of the selected key blocks, scale `scale`, natural-log LSE.
//
// Design (one persistent CTA per SM, 352 threads, warp-specialised):
//   warp 8  producer: takes the next query block from a global work counter,
//           publishes it in a 2-slot work ring, and streams the K and V tiles
//           of its selected key blocks into a 3-stage shared-memory ring (one
//           K + V pair per stage) with TMA (128-byte swizzle, 2 boxes of
//           64 x 128 per tile).
//   warp 9  S issuer (one thread): S = Q K^T with Q held in tensor memory
//           (A from TMEM, B = K tile from smem), as soon as the softmax warps
//           have read the previous S tile, so the next score tile is on the
//           tensor pipe while they work on this one.
//   warp 10 PV issuer (one thread): O += P V with P in tensor memory (A from
//           TMEM, B = V tile, MN-major).  Two issuing threads keep the tensor
//           pipe fed: a tcgen05.mma issue blocks while the pipe's queue is full,
//           and each issuer's barrier waits overlap the other's MMAs.
//   warps 0-7  softmax, two warpgroups: warps w and w+4 share the query rows
//           of TMEM lane quarter w%4 (thread = query row) and split the 128
//           key columns (and the 128 O columns) in halves.  Per key block: the
//           half row of S from TMEM to registers, the half maxima exchanged
//           through shared memory (one 64-thread named barrier per lane
//           quarter), online softmax in the log2 domain with lazy rescaling
//           (O in TMEM is rescaled only when the running max grows by more
//           than 2^8), P (bf16) -> TMEM; at the end O / l -> bf16, LSE.
// Tensor memory (512 columns): S [0,128), O [128,256), Q [256,320),
// P0 [320,384), P1 [384,448).
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
constexpr int kStages = 3;
constexpr int kFwdThreads = 352;
constexpr int kSoftmaxThreads = 256;
constexpr uint32_t TM_S = 0, TM_O = 128, TM_Q = 256, TM_P0 = 320, TM_P1 = 384;

struct FwdShared {
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full, s_free, p_full[2], p_empty[2], q_ready, final_bar;
  uint64_t work_full[2], work_empty[2];
  int work_row[2], work_beg[2], work_end[2], work_nvq[2];
  float xmax[2][2][128];  // [tile parity][column half][row]: half-row maxima
  float xsum[2][128];     // [column half][row]: half-row sums at the end
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
  long long Np;
  int nb;
  float scale_log2;
  unsigned long long limit;
  int starve;  // fault injection (test only): the producer issues no loads
};

__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, FwdParams P) {
  extern __shared__ uint8_t dsm_raw[];
  __shared__ FwdShared sm;
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  uint8_t* kvbuf = dsm;  // stage s: K at s * 2 * kTile, V right after
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 2);  // released by the S and the PV issuer
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.s_free, kSoftmaxThreads);
    mbar_init(&sm.p_full[0], kSoftmaxThreads);
    mbar_init(&sm.p_full[1], kSoftmaxThreads);
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
        const long long row = atomicAdd(queue, 1u);
        if (row >= P.rows) {
          sm.work_row[ws] = -1;
          mbar_arrive(&sm.work_full[ws]);
          break;
        }
        const int beg = P.row_ptr[row], end = P.row_ptr[row + 1];
        const int nvq = P.n_valid[row];
        sm.work_row[ws] = static_cast<int>(row);
        sm.work_beg[ws] = beg;
        sm.work_end[ws] = nvq > 0 ? end : beg;
        sm.work_nvq[ws] = nvq;
        mbar_arrive(&sm.work_full[ws]);
        if (nvq == 0) continue;
        const long long bh = row / P.nb;
        bool ok = true;
        for (int t = beg; t < end; ++t) {
          const int j = P.col_idx[t];
          const int y = static_cast<int>(bh * P.Np + static_cast<long long>(j) * kS);
          const int st = use % kStages;
          if (!W.wait(&sm.kv_empty[st], ((use / kStages) & 1) ^ 1, 2)) { ok = false; break; }
          uint8_t* kb = kvbuf + st * 2 * kTile;
          if (!P.starve) {  // fault injection: no loads, consumers time out
            mbar_expect_tx(&sm.kv_full[st], 2 * kTile);
            tma_load_2d(kb, &tmK, &sm.kv_full[st], 0, y);
            tma_load_2d(kb + kTile / 2, &tmK, &sm.kv_full[st], 64, y);
            tma_load_2d(kb + kTile, &tmV, &sm.kv_full[st], 0, y);
            tma_load_2d(kb + kTile + kTile / 2, &tmV, &sm.kv_full[st], 64, y);
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
            const int st = use % kStages;
            if (!W.wait(&sm.kv_full[st], (use / kStages) & 1, 9)) { ok = false; break; }
            fence_after();
            const uint64_t kd = sdesc_sw128(smem_u32(kvbuf + st * 2 * kTile), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_ts(tmem + TM_S, tmem + TM_Q + kk * 8,
                     kd + static_cast<uint64_t>(((kk >> 2) * (kTile / 2) + (kk & 3) * 32) >> 4), idS,
                     kk > 0 ? 1u : 0u);
            commit(&sm.s_full);
            commit(&sm.kv_empty[st]);
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
          // the first PV overwrites O: the previous block's epilogue has read it
          if (!W.wait(&sm.q_ready, qcnt & 1, 15)) break;
          ++qcnt;
          for (int jj = 0; jj < n; ++jj) {
            const uint32_t pb = pidx & 1;
            if (!W.wait(&sm.p_full[pb], (pidx >> 1) & 1, 7)) { ok = false; break; }
            const int st = use % kStages;
            if (!W.wait(&sm.kv_full[st], (use / kStages) & 1, 8)) { ok = false; break; }
            fence_after();
            const uint64_t vd =
                sdesc_sw128(smem_u32(kvbuf + st * 2 * kTile + kTile), kTile / 2, 1024);
            const uint32_t pa = tmem + (pb ? TM_P1 : TM_P0);
#pragma unroll
            for (int kk = 0; kk < kS / 16; ++kk)
              mma_ts(tmem + TM_O, pa + kk * 8, vd + static_cast<uint64_t>((kk * 2048) >> 4), idPV,
                     (jj > 0 || kk > 0) ? 1u : 0u);
            commit(&sm.p_empty[pb]);
            commit(&sm.kv_empty[st]);
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
    // Warps w and w+4 meet at a named barrier (64 threads) once per key block
    // and twice per query block.  A named barrier has no time limit, so the
    // two never leave a loop on their own: every bounded wait only clears
    // `ok`, the flags are exchanged at each meeting, and both warps leave
    // together at the first meeting after either of them failed.
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;  // query row of the block == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + TM_S + half * 64;
    const uint32_t tO = tmem + lane_base + TM_O + half * 64;
    const int c0 = half * 64;  // first key column (and O column) of this half
    uint32_t xpar = 0;         // parity of the flag slots of the next meeting
    auto meet = [&](bool mine) -> bool {  // pair barrier, returns both flags ANDed
      const int slot = xpar & 1;
      ++xpar;
      if (lane == 0) sm.xok[slot][half][quarter] = mine ? 1 : 0;
      asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
      return mine && sm.xok[slot][half ^ 1][quarter] != 0;
    };
    // wait until the PV that used P buffer (g & 1) for key block g is done
    auto pv_done = [&](uint32_t g, uint32_t where) {
      return W.wait(&sm.p_empty[g & 1], (g >> 1) & 1, where);
    };
    uint32_t sidx = 0, pidx = 0, tile = 0;
    bool ok = true;
    for (uint32_t it = 0;; ++it) {
      const int ws = it & 1;
      ok = meet(ok && W.wait(&sm.work_full[ws], (it >> 1) & 1, 10));
      if (!ok) break;
      const int row = sm.work_row[ws];
      if (row < 0) break;
      const int beg = sm.work_beg[ws], n = sm.work_end[ws] - beg, nvq = sm.work_nvq[ws];
      const long long bh = row / P.nb;
      const int i = row % P.nb;
      const long long grow = bh * P.Np + static_cast<long long>(i) * kS + r;
      uint4* orow = reinterpret_cast<uint4*>(P.Op + grow * kD) + half * 8;
      if (n == 0) {
#pragma unroll
        for (int q = 0; q < 8; ++q) orow[q] = make_uint4(0, 0, 0, 0);
        if (half == 0) P.lse[grow] = 0.f;
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
      float m = -INFINITY, l = 0.f;
      const int32_t* nvb = P.n_valid + bh * P.nb;
      int nvk_next = nvb[P.col_idx[beg]];
      for (int jj = 0; jj < n; ++jj) {
        const int nvk = nvk_next;
        if (jj + 1 < n) nvk_next = nvb[P.col_idx[beg + jj + 1]];  // ahead of its use
        const int lim = nvk - c0;  // columns of this half that hold real keys
        ok = ok && W.wait(&sm.s_full, sidx & 1, 11);
        uint32_t s[2][32];
        float mx = -INFINITY;
        if (ok) {
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
        }
        ++sidx;
        const int par = tile & 1;
        ++tile;
        sm.xmax[par][half][r] = mx;
        ok = meet(ok);
        if (!ok) break;
        mx = fmaxf(mx, sm.xmax[par][half ^ 1][r]) * P.scale_log2;
        const bool resc = mx > m + 8.f;
        const float m_new = resc ? mx : m;
        const float corr = resc ? ex2(m - m_new) : 1.f;
        if (jj > 0 && __any_sync(0xffffffffu, resc)) {
          ok = ok && pv_done(pidx - 1, 12);  // the previous key block's PV
          if (ok) {
            fence_after();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
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
        // early, non-blocking look at the release of the P buffer this key
        // block will write (its PV two blocks back); consumed at the store
        const bool p_free_early =
            pidx < 2 || mbar_test(&sm.p_empty[pidx & 1], ((pidx - 2) >> 1) & 1);
        float lsum = 0.f;
        uint32_t pk[32];
        if (lim >= 64) {
          float ls4[4] = {0.f, 0.f, 0.f, 0.f};  // independent partial sums
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int k0 = 2 * e;
            const float p0 = ex2(fmaf(__uint_as_float(s[k0 >> 5][k0 & 31]), P.scale_log2, -m));
            const float p1 = ex2(fmaf(__uint_as_float(s[(k0 + 1) >> 5][(k0 + 1) & 31]), P.scale_log2, -m));
            ls4[e & 3] += p0 + p1;
            pk[e] = pack_bf16x2(p0, p1);
          }
          lsum = (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
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
        // the PV issued two key blocks ago has finished reading this P buffer
        if (!p_free_early) ok = ok && pv_done(pidx - 2, 16);
        if (ok) {
          fence_after();
          tmem_st32(tmem + lane_base + ((pidx & 1) ? TM_P1 : TM_P0) + half * 32, pk);
          tmem_st_wait();
          fence_before();
          mbar_arrive(&sm.p_full[pidx & 1]);
        }
        ++pidx;
      }
      // epilogue: row sum over both halves, wait for the last PV, write the row
      sm.xsum[half][r] = l;
      ok = meet(ok);
      if (!ok) break;
      const float lt = sm.xsum[0][r] + sm.xsum[1][r];
      ok = ok && pv_done(pidx - 1, 13);
      if (ok) {
        fence_after();
        const bool real = r < nvq;
        const float inv = real ? 1.f / lt : 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
            orow[c * 4 + q] = v;
          }
        }
        if (half == 0) P.lse[grow] = real ? (m + log2f(lt)) * 0.69314718055994531f : 0.f;
      }
      // both halves have read xsum before either writes it for the next block
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
  a.Np = p.sz.Np;
  a.nb = p.sz.nb;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.limit = c.timeout_cycles ? c.timeout_cycles : 4000000000ull;
  a.starve = c.fault_inject == PRISM_FAULT_STARVE_LOADS ? 1 : 0;
  cudaError_t e = cudaMemsetAsync(a.status + WS_FWD_QUEUE, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  const size_t smem = 2ull * kStages * kTile + 1024;  // K + V per stage
  e = cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long g = a.rows < sm_count() ? a.rows : sm_count();
  attn_fwd_tc_kernel<<<static_cast<unsigned>(g), kFwdThreads, smem, st>>>(tmK, tmV, a);
  return cudaGetLastError();
}

}  // namespace prism
