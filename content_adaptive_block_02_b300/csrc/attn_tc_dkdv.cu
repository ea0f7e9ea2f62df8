// dK and dV of the block-sparse attention on the tcgen05 tensor cores,
// 128-token blocks, head dim 128.
//
// Prism (arXiv 2610.05416) trains through its sparse attention (Table 2
// caption: trainable methods replace video self-attention during training).
// The backward is the softmax-attention VJP restricted to the selected
// (query block, key block) pairs; the selection itself is a constant.  dQ
// runs in its own kernel (attn_tc_dq.cu), so that no gradient needs atomics.
//
// Work item = one key block j of one (b, h) with the ascending list of query
// blocks i that selected it (CSC), restricted to one range of query blocks
// when the plan walks them in ranges (partial dK / dV per range, summed in
// combine.cu).  For each i, four 128x128x128 products:
//   (1) S^T  = K_j Q_i^T           A = K_j (smem),  B = Q_i (smem)   -> TMEM
//   (2) dP^T = V_j dO_i^T          A = V_j (smem),  B = dO_i (smem)  -> TMEM
//       P^T = exp(S^T * scale - LSE_i)     (row = key, column = query)
//       dS^T = P^T * (dP^T - D_i)
//   (3) dV  += P^T dO_i            A = P^T (TMEM, written over S^T), B = dO_i (MN-major)
//   (4) dK  += dS^T Q_i            A = dS^T (smem, K-major), B = Q_i (MN-major)
// S^T and dP^T of a query block take the two 128-column regions of tensor
// memory in turn: block g's S^T (then its P^T) goes in region g % 2, its
// dP^T in the other.  So the next S^T goes where this block's dP^T was, as
// soon as the compute warps have read it, without waiting for (3) to read
// this block's P^T; the next dP^T goes where this block's P^T was, after (3).
//
// Roles (384 threads, one persistent CTA per SM):
//   warps 0-7  compute, two warpgroups: warps w and w+4 own the key rows of
//              TMEM lane quarter w%4 (thread = key row) and split the 128
//              query columns in halves; P^T, dS^T, epilogue dK * scale, dV
//              -> bf16 (the halves split the 128 channels there).
//   warp 8     producer: work counter, TMA loads of K_j, V_j (once per item)
//              and of Q_i, dO_i, -LSE_i * log2 e, D_i (2-stage ring) plus the
//              stage's query-block real-token count.  A stage's dO part is
//              free after (3), its Q part (with -LSE log2 e and D) only after
//              (4), and each is reloaded as soon as it is free: the Q part's
//              reload is on the loop that bounds the kernel (the next S^T
//              needs it), so it carries half the bytes.
//   warp 9     issuer of (1).
//   warp 10    issuer of (3) and (2), in the order 2_0 3_0 2_1 3_1 2_2 ...:
//              (2) of the next block overwrites the P^T that (3) of this
//              block reads, and MMAs of one thread run in issue order.
//   warp 11    issuer of (4).
//   One thread issues a tcgen05.mma only every ~120 cycles, about twice the
//   time the tensor pipe needs for a 128 x 128 x 16 product; three issuing
//   threads on three SM sub-partitions keep the pipe fed.
// Tensor memory: regions [0,128) and [128,256) (S^T / P^T of one block, dP^T
// of the other; P^T of query half h as bf16 pairs in the region's columns
// [64h, 64h + 32)), dV [256,384), dK [384,512).
#include "tc_common.cuh"

namespace prism {
namespace {
using namespace tc;

constexpr int kS = 128, kD = 128;
constexpr int kTile = kS * kD * 2;           // 32 KB
constexpr int kStage = 2 * kTile + 1024;     // Q, dO, LSE (512 B), D (512 B)
constexpr int kThreads = 384;
constexpr int kCompute = 256;
// S^T / P^T of query block g in region tm_r(g & 1), its dP^T in the other
__device__ __forceinline__ uint32_t tm_r(uint32_t parity) { return parity ? 128u : 0u; }
constexpr uint32_t TM_DV = 256, TM_DK = 384;
constexpr int kOffV = kTile, kOffStage = 2 * kTile, kOffDS = 2 * kTile + 2 * kStage;
constexpr int kOffBar = kOffDS + kTile;

struct BwdBars {
  uint64_t kv_full, kv_empty;
  // a stage's Q, -LSE log2 e and D (read until (4)) and its dO (read until
  // (3)) have their own barriers, so each part is reloaded as soon as it is free
  uint64_t q_full[2], q_empty[2], do_full[2], do_empty[2];
  uint64_t s_full, dp_free, ds_ready, ds_empty;
  // one barrier per block parity: with the regions alternating, the compute
  // warps can be one block ahead of the dV issuer, never two
  uint64_t dp_full[2], p_ready[2];
  uint64_t kv_done, kv_free, final_bar;
  uint64_t work_full[2], work_empty[2];
  int work_col[2], work_beg[2], work_end[2], work_nvk[2], work_chunk[2];
  int stage_i[2], stage_nvq[2];  // query block of each Q / dO stage and its real rows
  int xok[2][2][4];  // [meeting parity][column half][lane quarter]: still on track
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kSmemBytes = kOffBar + sizeof(BwdBars);

struct BwdParams {
  const float* nlse2;  // -LSE * log2(e)
  const float* D;
  const int32_t* n_valid;
  const int32_t* col_ptr;
  const int32_t* row_idx;
  uint16_t* dKp;
  uint16_t* dVp;
  uint16_t* dkpart;  // chunks > 1: partial dK (scaled) / dV per (key block, query range)
  uint16_t* dvpart;
  uint32_t* status;
  long long cols;    // B*H*nb key blocks
  long long items;   // cols * chunks work items
  long long Np;
  int nb;
  int chunks;        // query ranges per head (1: no split)
  int chunk_blocks;  // query blocks per range
  float scale, scale_log2;
  unsigned long long limit;
  int starve;  // fault injection (test only): the producer issues no loads
  const uint8_t* mask;  // blocks of half a tile: sub-tile mask per CSC entry (else null)
};

// 14 warps: 3-4 per SM sub-partition, so at most 128 registers per thread.
__global__ void __launch_bounds__(kThreads, 1)
    attn_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmdO, BwdParams P) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  BwdBars& sm = *reinterpret_cast<BwdBars*>(dsm + kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((smem_u32(dsm) & 1023u) != 0) {  // swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) dev_error(P.status, DEV_ERR_BOUNDS, 0xA11, smem_u32(dsm));
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 2);  // the S^T issuer (K) and the dP^T issuer (V)
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);   // the dK issuer
      mbar_init(&sm.do_full[s], 1);
      mbar_init(&sm.do_empty[s], 1);  // the dV issuer
      mbar_init(&sm.work_full[s], 1);
      mbar_init(&sm.work_empty[s], 3 + kCompute);
    }
    mbar_init(&sm.s_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.dp_full[b], 1);
      mbar_init(&sm.p_ready[b], kCompute);
    }
    mbar_init(&sm.dp_free, kCompute);
    mbar_init(&sm.ds_ready, kCompute);
    mbar_init(&sm.ds_empty, 1);
    mbar_init(&sm.kv_done, 2);  // the dV and the dK issuer
    mbar_init(&sm.kv_free, kCompute);
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
  uint8_t* kbuf = dsm;
  uint8_t* vbuf = dsm + kOffV;
  uint8_t* dsbuf = dsm + kOffDS;
  auto stage = [&](int s) { return dsm + kOffStage + s * kStage; };

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
        if (!W.wait(&sm.work_empty[ws], ((it >> 1) & 1) ^ 1, 21)) break;
        const long long item = atomicAdd(P.status + WS_BWD_QUEUE, 1u);
        if (item >= P.items) {
          sm.work_col[ws] = -1;
          mbar_arrive(&sm.work_full[ws]);
          break;
        }
        // item -> (b, h), query range c, key block j (ranges outermost within
        // a head, so the Q / dO tiles in use stay in L2)
        const long long per_bh = static_cast<long long>(P.chunks) * P.nb;
        const long long bhi = item / per_bh;
        const int rem = static_cast<int>(item - bhi * per_bh);
        const int c = rem / P.nb;
        const long long col = bhi * P.nb + (rem - c * P.nb);
        int beg = P.col_ptr[col], end = P.col_ptr[col + 1];
        if (P.chunks > 1) {
          const int lo = c * P.chunk_blocks;
          beg = lower_bound_i32(P.row_idx, beg, end, lo);
          end = lower_bound_i32(P.row_idx, beg, end, lo + P.chunk_blocks);
        }
        sm.work_col[ws] = static_cast<int>(col);
        sm.work_chunk[ws] = c;
        sm.work_beg[ws] = beg;
        sm.work_end[ws] = end;
        sm.work_nvk[ws] = P.n_valid[col];
        mbar_arrive(&sm.work_full[ws]);
        if (end == beg) continue;
        const long long bh = col / P.nb;
        const int j = static_cast<int>(col % P.nb);
        const int yk = static_cast<int>(bh * P.Np + static_cast<long long>(j) * kS);
        if (!W.wait(&sm.kv_empty, (items & 1) ^ 1, 22)) break;
        ++items;
        if (!P.starve) {  // fault injection: no loads, consumers time out
          mbar_expect_tx(&sm.kv_full, 2 * kTile);
          tma_load_2d(kbuf, &tmK, &sm.kv_full, 0, yk);
          tma_load_2d(kbuf + kTile / 2, &tmK, &sm.kv_full, 64, yk);
          tma_load_2d(vbuf, &tmV, &sm.kv_full, 0, yk);
          tma_load_2d(vbuf + kTile / 2, &tmV, &sm.kv_full, 64, yk);
        }
        for (int t = beg; t < end; ++t) {
          const int i = P.row_idx[t];
          const long long yq = bh * P.Np + static_cast<long long>(i) * kS;
          const int s = use & 1;
          const int nvq = P.n_valid[bh * P.nb + i];
          uint8_t* st = stage(s);
          // dO: free once (3) of the block two back is done
          if (!W.wait(&sm.do_empty[s], ((use >> 1) & 1) ^ 1, 24)) { ok = false; break; }
          if (!P.starve) {  // fault injection: no loads, consumers time out
            mbar_expect_tx(&sm.do_full[s], kTile);
            tma_load_2d(st + kTile, &tmdO, &sm.do_full[s], 0, static_cast<int>(yq));
            tma_load_2d(st + kTile + kTile / 2, &tmdO, &sm.do_full[s], 64, static_cast<int>(yq));
          }
          // Q, -LSE log2 e, D: free once (4) of the block two back is done
          if (!W.wait(&sm.q_empty[s], ((use >> 1) & 1) ^ 1, 23)) { ok = false; break; }
          sm.stage_i[s] = i;
          sm.stage_nvq[s] = nvq;
          if (!P.starve) {
            mbar_expect_tx(&sm.q_full[s], kTile + 1024);
            tma_load_2d(st, &tmQ, &sm.q_full[s], 0, static_cast<int>(yq));
            tma_load_2d(st + kTile / 2, &tmQ, &sm.q_full[s], 64, static_cast<int>(yq));
            bulk_load(st + 2 * kTile, P.nlse2 + yq, 512, &sm.q_full[s]);
            bulk_load(st + 2 * kTile + 512, P.D + yq, 512, &sm.q_full[s]);
          }
          ++use;
        }
      }
    }
    __syncwarp();
  } else if (warp >= 9 && warp <= 11) {
    // ------------------------------------------------------ MMA issuers ----
    if (lane == 0) {
      const int role = warp - 9;  // 0: (1) S^T, 1: (3) dV then (2) dP^T, 2: (4) dK
      constexpr uint32_t id_kk = idesc_bf16(128, 128, 0, 0);  // A K-major, B K-major
      constexpr uint32_t id_kn = idesc_bf16(128, 128, 0, 1);  // A K-major, B MN-major
      const uint64_t kd_k = sdesc_sw128(smem_u32(kbuf), 16, 1024);          // K, K-major
      const uint64_t vd_k = sdesc_sw128(smem_u32(vbuf), 16, 1024);          // V, K-major
      const uint64_t dsd_k = sdesc_sw128(smem_u32(dsbuf), 16, 1024);        // dS^T, K-major
      auto koff = [](int kk) {  // K-major 16-element step inside two 64-column panels
        return static_cast<uint64_t>(((kk >> 2) * (kTile / 2) + (kk & 3) * 32) >> 4);
      };
      auto noff = [](int kk) {  // MN-major 16-row step
        return static_cast<uint64_t>((kk * 2048) >> 4);
      };
      // (2) dP^T of query block g (CTA-wide count) into its region; the
      // region held P^T of block g - 1, read by (3) of g - 1, which this same
      // thread issued before
      auto issue_dp = [&](uint32_t g) -> bool {
        const int sq = g & 1;
        if (!W.wait(&sm.do_full[sq], (g >> 1) & 1, 35)) return false;
        fence_after();
        const uint64_t dd = sdesc_sw128(smem_u32(stage(sq) + kTile), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss(tmem + tm_r((g & 1) ^ 1), vd_k + koff(kk), dd + koff(kk), id_kk, kk > 0 ? 1u : 0u);
        commit(&sm.dp_full[g & 1]);
        return true;
      };
      uint32_t use = 0, items = 0, kvcnt = 0;
      bool ok = true;
      for (uint32_t it = 0; ok; ++it) {
        const int ws = it & 1;
        if (!W.wait(&sm.work_full[ws], (it >> 1) & 1, 31)) break;
        if (sm.work_col[ws] < 0) break;
        const int n = sm.work_end[ws] - sm.work_beg[ws];
        if (n > 0) {
          if (role != 2 && !W.wait(&sm.kv_full, items & 1, 32)) break;
          ++items;
          fence_after();
          if (role == 0) {
            for (int k = 0; k < n; ++k) {
              const uint32_t g = use + k;
              const int st = g & 1;
              if (!W.wait(&sm.q_full[st], (g >> 1) & 1, 34)) { ok = false; break; }
              // S^T of block g goes where dP^T of block g - 1 was: the compute
              // warps have read it
              if (g > 0 && !W.wait(&sm.dp_free, (g - 1) & 1, 38)) { ok = false; break; }
              fence_after();
              const uint64_t qd_k = sdesc_sw128(smem_u32(stage(st)), 16, 1024);
              // (1) S^T = K Q^T
#pragma unroll
              for (int kk = 0; kk < kD / 16; ++kk)
                mma_ss(tmem + tm_r(g & 1), kd_k + koff(kk), qd_k + koff(kk), id_kk,
                       kk > 0 ? 1u : 0u);
              commit(&sm.s_full);
            }
            if (!ok) break;
            commit(&sm.kv_empty);
          } else if (role == 1) {
            if (!issue_dp(use)) break;
            // the previous item's dK / dV have been read out
            if (kvcnt > 0 && !W.wait(&sm.kv_free, (kvcnt - 1) & 1, 33)) break;
            for (int k = 0; k < n; ++k) {
              const uint32_t g = use + k;
              const int st = g & 1;
              // (3) dV += P^T dO, once P^T has replaced S^T in block g's region
              if (!W.wait(&sm.p_ready[g & 1], (g >> 1) & 1, 36)) { ok = false; break; }
              fence_after();
              const uint64_t dod_n = sdesc_sw128(smem_u32(stage(st) + kTile), kTile / 2, 1024);
#pragma unroll
              for (int kk = 0; kk < kS / 16; ++kk)
                mma_ts(tmem + TM_DV, tmem + tm_r(g & 1) + (kk >> 2) * 64 + (kk & 3) * 8,
                       dod_n + noff(kk), id_kn, (k > 0 || kk > 0) ? 1u : 0u);
              commit(&sm.do_empty[st]);
              if (k + 1 < n && !issue_dp(g + 1)) { ok = false; break; }
            }
            if (!ok) break;
            commit(&sm.kv_done);
            commit(&sm.kv_empty);
          } else {
            if (kvcnt > 0 && !W.wait(&sm.kv_free, (kvcnt - 1) & 1, 39)) break;
            for (int k = 0; k < n; ++k) {
              const uint32_t g = use + k;
              const int st = g & 1;
              // (4) dK += dS^T Q
              if (!W.wait(&sm.ds_ready, g & 1, 37)) { ok = false; break; }
              if (!W.wait(&sm.q_full[st], (g >> 1) & 1, 30)) { ok = false; break; }
              fence_after();
              const uint64_t qd_n = sdesc_sw128(smem_u32(stage(st)), kTile / 2, 1024);
#pragma unroll
              for (int kk = 0; kk < kS / 16; ++kk)
                mma_ss(tmem + TM_DK, dsd_k + koff(kk), qd_n + noff(kk), id_kn,
                       (k > 0 || kk > 0) ? 1u : 0u);
              commit(&sm.ds_empty);
              commit(&sm.q_empty[st]);
            }
            if (!ok) break;
            commit(&sm.kv_done);
          }
          use += n;
          ++kvcnt;
        }
        mbar_arrive(&sm.work_empty[ws]);
      }
      commit(&sm.final_bar);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------ compute ----
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;  // key row == TMEM lane
    const uint32_t lb = static_cast<uint32_t>(quarter * 32) << 16;
    const int q0 = half * 64;  // first query column (and first channel) of this half
    // Warps w and w+4 meet at a named barrier (64 threads) once per work
    // item.  A named barrier has no time limit, so the two never leave the
    // item loop on their own: a failed bounded wait clears `ok` and ends the
    // query-block loop (every later wait of the other warp then fails at
    // once on the abort flag), the flags are exchanged at each meeting, and
    // both warps leave together at the first meeting after either failed.
    uint32_t xpar = 0;
    auto meet = [&](bool mine) -> bool {
      mine = __all_sync(0xffffffffu, mine);  // one flag per warp
      const int slot = xpar & 1;
      ++xpar;
      if (lane == 0) sm.xok[slot][half][quarter] = mine ? 1 : 0;
      asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
      return mine && sm.xok[slot][half ^ 1][quarter] != 0;
    };
    uint32_t use = 0, scnt = 0, dpcnt = 0, dsidx = 0, kvcnt = 0;
    bool ok = true;
    for (uint32_t it = 0;; ++it) {
      const int ws = it & 1;
      ok = meet(ok && W.wait(&sm.work_full[ws], (it >> 1) & 1, 41));
      if (!ok) break;
      const int col = sm.work_col[ws];
      if (col < 0) break;
      const int beg = sm.work_beg[ws], n = sm.work_end[ws] - beg, nvk = sm.work_nvk[ws];
      const long long bh = col / P.nb;
      const int j = static_cast<int>(col % P.nb);
      const long long krow = bh * P.Np + static_cast<long long>(j) * kS + r;
      // output rows: the final dK / dV, or this query range's partial ones
      const long long prow =
          (static_cast<long long>(col) * P.chunks + sm.work_chunk[ws]) * kS + r;
      uint4* dkrow =
          reinterpret_cast<uint4*>(P.chunks > 1 ? P.dkpart + prow * kD : P.dKp + krow * kD) +
          half * 8;
      uint4* dvrow =
          reinterpret_cast<uint4*>(P.chunks > 1 ? P.dvpart + prow * kD : P.dVp + krow * kD) +
          half * 8;
      if (n == 0) {
        // (with query ranges, the combining kernel handles empty ranges)
        if (P.chunks == 1) {
#pragma unroll
          for (int q = 0; q < 8; ++q) dkrow[q] = dvrow[q] = make_uint4(0, 0, 0, 0);
        }
        mbar_arrive(&sm.work_empty[ws]);
        continue;
      }
      for (int k = 0; k < n; ++k) {
        const int s_ = (use + k) & 1;
        // -LSE_i log2 e and D_i arrive with Q_i on the stage's Q barrier
        ok = ok && W.wait(&sm.q_full[s_], ((use + k) >> 1) & 1, 40);
        // blocks of half a tile: bit 2 qh + kh of an entry's mask set = the
        // query half qh (this column half) does not attend the key half kh
        // (this row's half)
        const bool act =
            P.mask == nullptr || !((P.mask[beg + k] >> (half * 2 + (quarter >> 1))) & 1);
        const int lim = (r < nvk && act) ? sm.stage_nvq[s_] - q0 : 0;  // real query columns here
        const float4* lse4 = reinterpret_cast<const float4*>(stage(s_) + 2 * kTile) + half * 16;
        const float4* D4 = lse4 + 32;
        // ---- P^T = exp(S^T * scale - LSE) on this half of the queries ----
        ok = __all_sync(0xffffffffu, ok && W.wait(&sm.s_full, scnt & 1, 42));
        ++scnt;
        if (!ok) break;
        float p[64];
        {
          fence_after();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t sv[32];
            tmem_ld32(tmem + lb + tm_r((use + k) & 1) + q0 + c * 32, sv);
            tmem_ld_wait();
            // two queries per fp32x2 instruction: x = s * c - LSE log2 e
            const f32x2 c2 = pack2(P.scale_log2, P.scale_log2);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              const float4 L = lse4[c * 8 + g];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int q = c * 32 + g * 4 + 2 * e;
                const f32x2 x2 = fma2(pack2(__uint_as_float(sv[g * 4 + 2 * e]),
                                            __uint_as_float(sv[g * 4 + 2 * e + 1])),
                                      c2, e ? pack2(L.z, L.w) : pack2(L.x, L.y));
                float x0, x1;
                unpack2(x2, x0, x1);
                p[q] = q < lim ? ex2(x0) : 0.f;
                p[q + 1] = q + 1 < lim ? ex2(x1) : 0.f;
              }
            }
          }
        }
        // P^T (bf16 pairs) over the first 32 of this half's own 64 S^T
        // columns, which only this thread's row has read: no wait for the
        // other half
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(p[h * 32 + 2 * e], p[h * 32 + 2 * e + 1]);
          tmem_st16(tmem + lb + tm_r((use + k) & 1) + q0 + h * 16, pk);
        }
        tmem_st_wait();
        fence_before();
        mbar_arrive(&sm.p_ready[(use + k) & 1]);
        // ---- dS^T = P^T * (dP^T - D) -> smem panel `half` (128-byte swizzle) ----
        ok = ok && W.wait(&sm.dp_full[dpcnt & 1], (dpcnt >> 1) & 1, 43);
        ++dpcnt;
        if (dsidx > 0) ok = ok && W.wait(&sm.ds_empty, (dsidx - 1) & 1, 44);
        ok = __all_sync(0xffffffffu, ok);
        ++dsidx;
        if (ok) {
          fence_after();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t dp[32];
            tmem_ld32(tmem + lb + tm_r(((use + k) & 1) ^ 1) + q0 + c * 32, dp);
            tmem_ld_wait();
            if (c == 1) {
              fence_before();
              mbar_arrive(&sm.dp_free);  // the next S^T may be written here
            }
#pragma unroll
            for (int g = 0; g < 4; ++g) {  // 8 queries = one 16-byte chunk
              const int ql = c * 32 + g * 8;  // local query index in this half
              const float4 da = D4[ql / 4], db4 = D4[ql / 4 + 1];
              const f32x2 dv2[4] = {pack2(da.x, da.y), pack2(da.z, da.w), pack2(db4.x, db4.y),
                                    pack2(db4.z, db4.w)};
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {  // two queries per fp32x2 instruction
                const f32x2 ds2 = mul2(pack2(p[ql + 2 * e], p[ql + 2 * e + 1]),
                                       sub2(pack2(__uint_as_float(dp[g * 8 + 2 * e]),
                                                  __uint_as_float(dp[g * 8 + 2 * e + 1])),
                                            dv2[e]));
                float x0, x1;
                unpack2(ds2, x0, x1);
                w4[e] = pack_bf16x2(x0, x1);
              }
              const int chunk = ql >> 3;
              const uint32_t off = half * (kTile / 2) + r * 128 + ((chunk ^ (r & 7)) << 4);
              *reinterpret_cast<uint4*>(dsbuf + off) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
          fence_proxy_async();
          fence_before();
          mbar_arrive(&sm.ds_ready);
        }
      }
      // a failure in the last query block is caught at the next meeting
      use += n;
      // ---- epilogue: dV, dK * scale -> bf16, this half of the channels ----
      ok = __all_sync(0xffffffffu, ok && W.wait(&sm.kv_done, kvcnt & 1, 45));
      ++kvcnt;
      if (!ok) continue;  // both halves leave at the next meeting
      fence_after();
      const bool real = r < nvk;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        uint4* dst = which ? dkrow : dvrow;
        const float mul = real ? (which ? P.scale : 1.f) : 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lb + (which ? TM_DK : TM_DV) + q0 + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * mul, __uint_as_float(o[8 * q + 1]) * mul);
            v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * mul, __uint_as_float(o[8 * q + 3]) * mul);
            v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * mul, __uint_as_float(o[8 * q + 5]) * mul);
            v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * mul, __uint_as_float(o[8 * q + 7]) * mul);
            dst[c * 4 + q] = v;
          }
        }
      }
      fence_before();
      mbar_arrive(&sm.kv_free);
      mbar_arrive(&sm.work_empty[ws]);
    }
  }

  // ---------------------------------------------------------- teardown ----
  __syncthreads();
  if (warp == 0) {
    if (!wait_raw(&sm.final_bar, 0, P.limit) && lane == 0)
      dev_error(P.status, DEV_ERR_TIMEOUT, 199, 0);
    fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_attn_dkdv_tc(const Plan& p, const uint16_t* Qp, const uint16_t* Kp,
                                const uint16_t* Vp, const uint16_t* dOp, const float* nlse2,
                                const float* D, const int32_t* n_valid, const int32_t* col_ptr,
                                const int32_t* row_idx, float scale, uint16_t* dKp, uint16_t* dVp,
                                uint8_t* ws, uint16_t* dkvpart, cudaStream_t st) {
  const prism_config_t& c = p.cfg;
  const long long rows_total = static_cast<long long>(c.B) * c.H * p.sz.Np;
  CUtensorMap tmQ, tmK, tmV, tmdO;
  if (!make_tile_map(&tmQ, Qp, rows_total) || !make_tile_map(&tmK, Kp, rows_total) ||
      !make_tile_map(&tmV, Vp, rows_total) || !make_tile_map(&tmdO, dOp, rows_total))
    return cudaErrorInvalidValue;
  BwdParams a;
  a.nlse2 = nlse2;
  a.D = D;
  a.n_valid = n_valid;
  a.col_ptr = col_ptr;
  a.row_idx = row_idx;
  a.dKp = dKp;
  a.dVp = dVp;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.cols = static_cast<long long>(c.B) * c.H * p.sz.nb;
  a.chunks = dkvpart != nullptr ? p.sz.key_chunks : 1;
  a.chunk_blocks = a.chunks > 1 ? p.sz.chunk_blocks : p.sz.nb;
  a.items = a.cols * a.chunks;
  // dK partials, then dV partials
  a.dkpart = dkvpart;
  a.dvpart = dkvpart != nullptr ? dkvpart + a.items * kS * kD : nullptr;
  a.Np = p.sz.Np;
  a.nb = p.sz.nb;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.limit = c.timeout_cycles ? c.timeout_cycles : 4000000000ull;
  a.starve = c.fault_inject == PRISM_FAULT_STARVE_LOADS ? 1 : 0;
  a.mask = (p.sz.half_tile && ws != nullptr) ? ws + p.sz.ws_csc_mask : nullptr;
  cudaError_t e = cudaMemsetAsync(a.status + WS_BWD_QUEUE, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_dkdv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const long long g = a.items < sm_count() ? a.items : sm_count();
  attn_dkdv_tc_kernel<<<static_cast<unsigned>(g), kThreads, kSmemBytes, st>>>(tmQ, tmK, tmV, tmdO,
                                                                            a);
  return cudaGetLastError();
}

}  // namespace prism
