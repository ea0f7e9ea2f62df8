// Audio-to-video (A2V) cross-attention norms on the 5th-generation tensor
// cores: n_i = || softmax(Qa_i Ka^T / sqrt(Ca)) Va ||_2 for every video token.
//
// Prism (arXiv 2610.05416), Abstract: the zone signals use the feature norms
// of the audio-to-video cross-attention output.  Reading used here: one
// attention head; the video tokens' cross-attention queries Qa [B, N, Ca]
// attend to the audio tokens' keys Ka and values Va [B, Na, Ca] with scale
// 1/sqrt(Ca); only the norm of each output row leaves the kernel (the output
// itself is never written).
//
// Design (persistent CTAs, 128 threads = one query row per thread, thread 0
// also issues the TMA loads and the MMAs):
//   * Ka and Va of the batch entry are loaded once per CTA (TMA, 128-byte
//     swizzle); Va is converted in shared memory from bf16 to fp16 (exact for
//     |v| < 65504, checked) so that the P V product can take P in fp16.
//   * per tile of 128 video tokens: S = Qa Ka^T (tcgen05 kind::f16, bf16,
//     fp32 accumulation in tensor memory, N = Na rounded up to 16);
//     softmax of each row in the log2 domain; the weights, scaled by 2^8,
//     are split into two fp16 terms p_hi + p_lo (22 significant bits, so the
//     products carry about fp32 precision, not bf16's); O = (p_hi + p_lo) Va
//     as two accumulating TS-form MMAs (A from tensor memory); the epilogue
//     reads its row of O and writes ||O|| / (2^8 l).
//   * the next tile's Qa is loaded while this tile's softmax, P V product and
//     epilogue run.
// Tensor memory (512 columns): O [0, 128), S [128, 384) (p_hi is written
// over the S columns already read), p_lo [384, 512).
// Every wait is bounded; on expiry the CTA records PRISM_ERR_DEVICE_TIMEOUT
// in the status word, every thread leaves the tile loop together, and tensor
// memory is freed once the CTA's MMAs have completed.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace prism {
namespace {
using namespace tc;

constexpr int kRows = 128;            // video tokens per tile
constexpr int kThreads = 128;
constexpr uint32_t TM_O = 0, TM_S = 128, TM_PLO = 384;
constexpr float kPScale = 256.f;      // weights scaled by 2^8 before the fp16 split

struct A2VParams {
  float* n;                 // [B, N] out
  uint32_t* status;
  long long N;              // video tokens per batch entry
  int B, Na, Na_pad, Ca;
  int tiles_per_b;
  float scale_log2;         // log2(e) / sqrt(Ca)
  unsigned long long limit;
};

// Instruction descriptor, kind::f16 with fp16 A and B, fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(kThreads, 1)
    a2v_norm_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, A2VParams P) {
  extern __shared__ uint8_t dsm_raw[];
  __shared__ uint64_t q_full, kv_full, s_full, o_full, final_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const int nbox = P.Ca / 64;                        // 64-channel boxes per row
  const uint32_t qbox = kRows * 128;                 // bytes of one Qa box
  const uint32_t abox = static_cast<uint32_t>(P.Na_pad) * 128;  // bytes of one Ka / Va box
  uint8_t* sQ = dsm;
  uint8_t* sK = sQ + nbox * qbox;
  uint8_t* sV = sK + nbox * abox;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = P.B * P.tiles_per_b;

  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    mbar_init(&kv_full, 1);
    mbar_init(&s_full, 1);
    mbar_init(&o_full, 1);
    mbar_init(&final_bar, 1);
    abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base;
  const Waiter W{&abort_flag, P.status, P.limit};
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const int r = warp * 32 + lane;  // row of the tile == TMEM lane

  uint32_t q_issued = 0, kv_issued = 0;  // loads issued (thread 0), to drain on an abort
  auto load_q = [&](int tile) {  // thread 0
    ++q_issued;
    const int b = tile / P.tiles_per_b;
    const int y = static_cast<int>(b * P.N + static_cast<long long>(tile % P.tiles_per_b) * kRows);
    mbar_expect_tx(&q_full, nbox * qbox);
    for (int k = 0; k < nbox; ++k) tma_load_2d(sQ + k * qbox, &tmQ, &q_full, 64 * k, y);
  };
  if (threadIdx.x == 0 && static_cast<int>(blockIdx.x) < ntiles) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    load_q(blockIdx.x);
  }

  const uint32_t idS = idesc_bf16(kRows, P.Na_pad, 0, 0);   // A = Qa, B = Ka, both K-major
  const uint32_t idPV = idesc_f16(kRows, P.Ca, 0, 1);       // A = P (TMEM), B = Va MN-major
  int cur_b = -1;
  uint32_t qph = 0, kvph = 0, tph = 0;
  bool ok = true;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tph) {
    const int b = tile / P.tiles_per_b;
    const long long t0 = static_cast<long long>(tile % P.tiles_per_b) * kRows;
    if (b != cur_b) {
      // this batch entry's audio keys and values (the previous tile's MMAs,
      // which read them, completed before its epilogue)
      if (threadIdx.x == 0) {
        ++kv_issued;
        mbar_expect_tx(&kv_full, 2 * nbox * abox);
        for (int k = 0; k < nbox; ++k) {
          tma_load_2d(sK + k * abox, &tmK, &kv_full, 64 * k, b * P.Na);
          tma_load_2d(sV + k * abox, &tmV, &kv_full, 64 * k, b * P.Na);
        }
      }
      ok = W.wait(&kv_full, kvph & 1, 201);
      ++kvph;
      if (!__syncthreads_and(ok)) break;
      // bf16 -> fp16 in place (the swizzle moves whole 16-byte pieces, so
      // each element keeps its slot)
      uint32_t* v32 = reinterpret_cast<uint32_t*>(sV);
      bool range_ok = true;
      for (int i = threadIdx.x; i < nbox * static_cast<int>(abox) / 4; i += kThreads) {
        const uint32_t u = v32[i];
        const float lo = bf16_lo(u), hi = bf16_hi(u);
        range_ok &= fabsf(lo) < 65504.f && fabsf(hi) < 65504.f;
        v32[i] = pack_f16x2(lo, hi);
      }
      if (!range_ok) dev_error(P.status, DEV_ERR_BOUNDS, 210, b);
      fence_proxy_async();
      __syncthreads();
      cur_b = b;
    }
    // ---- S = Qa Ka^T ----
    if (threadIdx.x == 0) {
      ok = W.wait(&q_full, qph & 1, 202);
      ++qph;
      if (ok) {
        fence_after();
        const uint64_t qd = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t kd = sdesc_sw128(smem_u32(sK), 16, 1024);
        for (int kk = 0; kk < P.Ca / 16; ++kk) {
          const uint64_t qo = static_cast<uint64_t>(((kk >> 2) * qbox + (kk & 3) * 32) >> 4);
          const uint64_t ko = static_cast<uint64_t>(((kk >> 2) * abox + (kk & 3) * 32) >> 4);
          mma_ss(tmem + TM_S, qd + qo, kd + ko, idS, kk > 0 ? 1u : 0u);
        }
        commit(&s_full);
      }
    }
    ok = ok && W.wait(&s_full, tph & 1, 203);
    if (!__syncthreads_and(ok)) break;
    fence_after();
    // the S product has read this tile's Qa: fetch the next tile's
    if (threadIdx.x == 0 && tile + static_cast<int>(gridDim.x) < ntiles)
      load_q(tile + gridDim.x);
    // ---- softmax of this thread's row over the Na real audio tokens ----
    const int nch = (P.Na + 31) / 32;
    float mx = -INFINITY;
    for (int c = 0; c < nch; ++c) {
      uint32_t s[32];
      tmem_ld32(tmem + lane_base + TM_S + 32 * c, s);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (32 * c + e < P.Na) mx = fmaxf(mx, __uint_as_float(s[e]));
    }
    const float mxl = mx * P.scale_log2;
    float l = 0.f;
    for (int c = 0; c < P.Na_pad / 32 + ((P.Na_pad & 31) ? 1 : 0); ++c) {
      uint32_t s[32], hi[16], lo[16];
      tmem_ld32(tmem + lane_base + TM_S + 32 * c, s);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int k0 = 32 * c + 2 * e;
        const float p0 = k0 < P.Na ? ex2(fmaf(__uint_as_float(s[2 * e]), P.scale_log2, -mxl)) : 0.f;
        const float p1 =
            k0 + 1 < P.Na ? ex2(fmaf(__uint_as_float(s[2 * e + 1]), P.scale_log2, -mxl)) : 0.f;
        l += p0 + p1;
        const float q0 = p0 * kPScale, q1 = p1 * kPScale;
        const uint32_t h = pack_f16x2(q0, q1);
        const float h0 = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xffffu)));
        const float h1 = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
        hi[e] = h;
        lo[e] = pack_f16x2(q0 - h0, q1 - h1);
      }
      // p_hi over S columns this thread has already read; p_lo apart
      tmem_st16(tmem + lane_base + TM_S + 16 * c, hi);
      tmem_st16(tmem + lane_base + TM_PLO + 16 * c, lo);
    }
    tmem_st_wait();
    fence_before();
    __syncthreads();
    // ---- O = (p_hi + p_lo) Va ----
    if (threadIdx.x == 0) {
      fence_after();
      const uint64_t vd = sdesc_sw128(smem_u32(sV), abox, 1024);
      for (int kk = 0; kk < P.Na_pad / 16; ++kk)
        mma_ts(tmem + TM_O, tmem + TM_S + kk * 8, vd + static_cast<uint64_t>((kk * 2048) >> 4),
               idPV, kk > 0 ? 1u : 0u);
      for (int kk = 0; kk < P.Na_pad / 16; ++kk)
        mma_ts(tmem + TM_O, tmem + TM_PLO + kk * 8, vd + static_cast<uint64_t>((kk * 2048) >> 4),
               idPV, 1u);
      commit(&o_full);
    }
    ok = W.wait(&o_full, tph & 1, 204);
    if (!__syncthreads_and(ok)) break;
    fence_after();
    // ---- epilogue: ||O_r|| / (2^8 l) ----
    float ss = 0.f;
    for (int c = 0; c < P.Ca / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(tmem + lane_base + TM_O + 32 * c, o);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) ss = fmaf(__uint_as_float(o[e]), __uint_as_float(o[e]), ss);
    }
    const long long tok = t0 + r;
    if (tok < P.N) P.n[static_cast<long long>(b) * P.N + tok] = sqrtf(ss) / (kPScale * l);
    // every thread has read O and S before the next tile's MMAs overwrite them
    fence_before();
    __syncthreads();
  }

  // ---------------------------------------------------------- teardown ----
  __syncthreads();
  if (threadIdx.x == 0) {
    // no copy may still be landing in shared memory when the CTA leaves
    if (q_issued > qph && !wait_raw(&q_full, qph & 1, P.limit)) dev_error(P.status, DEV_ERR_TIMEOUT, 297, 0);
    if (kv_issued > kvph && !wait_raw(&kv_full, kvph & 1, P.limit)) dev_error(P.status, DEV_ERR_TIMEOUT, 298, 0);
  }
  if (warp == 0) {
    if (lane == 0) commit(&final_bar);
    __syncwarp();
    // every MMA this CTA issued has completed before the columns are freed
    if (!wait_raw(&final_bar, 0, P.limit) && lane == 0) dev_error(P.status, DEV_ERR_TIMEOUT, 299, 0);
    fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t a2v_smem_bytes(int Ca, int Na) {
  const int na_pad = (Na + 15) / 16 * 16;
  return static_cast<size_t>(Ca / 64) * (kRows * 128 + 2ull * na_pad * 128) + 1024;
}

cudaError_t launch_a2v_norms(const Plan& p, const uint16_t* Qa, const uint16_t* Ka,
                             const uint16_t* Va, int Na, float* n, uint8_t* ws, cudaStream_t st) {
  const prism_config_t& c = p.cfg;
  A2VParams a;
  a.n = n;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.N = p.sz.N;
  a.B = c.B;
  a.Na = Na;
  a.Na_pad = (Na + 15) / 16 * 16;
  a.Ca = c.Ca;
  a.tiles_per_b = static_cast<int>((p.sz.N + kRows - 1) / kRows);
  a.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(c.Ca)));
  a.limit = c.timeout_cycles ? c.timeout_cycles : 4000000000ull;
  CUtensorMap tmQ, tmK, tmV;
  if (!make_bf16_map(&tmQ, Qa, static_cast<long long>(c.B) * p.sz.N, c.Ca, kRows) ||
      !make_bf16_map(&tmK, Ka, static_cast<long long>(c.B) * Na, c.Ca, a.Na_pad) ||
      !make_bf16_map(&tmV, Va, static_cast<long long>(c.B) * Na, c.Ca, a.Na_pad))
    return cudaErrorInvalidValue;
  const size_t smem = a2v_smem_bytes(c.Ca, Na);
  cudaError_t e = cudaFuncSetAttribute(a2v_norm_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long tiles = static_cast<long long>(c.B) * a.tiles_per_b;
  const long long g = tiles < sm_count() ? tiles : sm_count();
  a2v_norm_tc_kernel<<<static_cast<unsigned>(g), kThreads, smem, st>>>(tmQ, tmK, tmV, a);
  return cudaGetLastError();
}

}  // namespace prism
