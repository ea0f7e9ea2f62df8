// Backward entry point that allocates nothing and takes no workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// backward: code that runs inside a memory-pool arena it does not own, or
// inside a runtime that forbids cudaMalloc / cudaFree after start-up.  For
// them the backward's scratch -- the per-row rowsum D, the fp32 dQ
// accumulator and the small status / work-counter words -- lives in one
// fixed-size array that is part of this library (below), instead of in a
// caller-provided workspace.
//
// The array is kNoAllocScratchBytes (32 MiB) on every GPU that loads the
// library and is held until the process exits.  All calls share it and it
// keeps the last call's contents; everything that must start at zero is
// cleared at the start of each call.  Two calls whose kernels overlap on the
// GPU (different streams, or different threads without ordering) race on the
// array and give wrong results.  Device-side wait timeouts of this variant are
// recorded in the array's own status word, which prism_noalloc_device_status
// reads back.
#include <mutex>

#include "prism_internal.cuh"

namespace prism {
cudaError_t launch_bwd_pre(const Plan& p, const uint16_t* Op, const uint16_t* dOp,
                           const float* lse, float* D, float* nlse2, float* dQacc,
                           cudaStream_t st);
cudaError_t launch_attn_bwd_simt(const Plan& p, const uint16_t* Qp, const uint16_t* Kp,
                                 const uint16_t* Vp, const uint16_t* dOp, const float* lse,
                                 const float* D, const int32_t* n_valid,
                                 const int32_t* col_ptr, const int32_t* row_idx, float scale,
                                 float* dQacc, uint16_t* dKp, uint16_t* dVp, cudaStream_t st);
cudaError_t launch_attn_dkdv_tc(const Plan& p, const uint16_t* Qp, const uint16_t* Kp,
                                const uint16_t* Vp, const uint16_t* dOp, const float* nlse2,
                                const float* D, const int32_t* n_valid, const int32_t* col_ptr,
                                const int32_t* row_idx, float scale, uint16_t* dKp, uint16_t* dVp,
                                uint8_t* ws, uint16_t* dkvpart, cudaStream_t st);
cudaError_t launch_attn_dq_tc(const Plan& p, const uint16_t* Qp, const uint16_t* Kp,
                              const uint16_t* Vp, const uint16_t* dOp, const float* lse,
                              const float* D, const int32_t* n_valid, const int32_t* row_ptr,
                              const int32_t* col_idx, float scale, uint16_t* dQp, uint8_t* ws,
                              uint16_t* dqpart, cudaStream_t st);
}  // namespace prism

struct prism_plan {
  prism::Plan p;
};

namespace {

constexpr size_t kNoAllocScratchBytes = 32ull << 20;

// The scratch itself.  In host code `g_noalloc_scratch` names a host-side
// stand-in, not device memory: its device address comes from
// cudaGetSymbolAddress, taken once per device below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch on the current device (set up on the first
// call on that device).  The cached address belongs to the device's primary
// context as it was then: after cudaDeviceReset (or with another context
// current on that device) it is no longer valid.
cudaError_t scratch_address(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = static_cast<uint8_t*>(g_addr[dev]);
  return cudaSuccess;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int prism_sparse_attn_bwd_noalloc(
    const prism_plan_t* plan, const uint16_t* Qp, const uint16_t* Kp, const uint16_t* Vp,
    const uint16_t* Op, const uint16_t* dOp, const float* lse, const int32_t* n_valid,
    const int32_t* row_ptr, const int32_t* col_idx, const int32_t* col_ptr,
    const int32_t* row_idx, float scale, uint16_t* dQp, uint16_t* dKp, uint16_t* dVp,
    void* stream) {
  if (plan == nullptr || !(scale > 0.f)) return PRISM_ERR_ARG;
  const void* ptrs[] = {Qp,      Kp,      Vp,      Op,  dOp, lse, n_valid, row_ptr,
                        col_idx, col_ptr, row_idx, dQp, dKp, dVp};
  for (const void* q : ptrs) {
    if (q == nullptr) return PRISM_ERR_ARG;
    if (!al16(q)) return PRISM_ERR_ALIGN;
  }
  const prism::Plan& p = plan->p;
  // blocks of half a tile: the sub-tile masks live in the plan's workspace
  if (p.sz.half_tile) return PRISM_ERR_UNSUPPORTED;
  // layout inside the scratch: status words, D, then LSE * log2(e) for the
  // tensor-core kernels or the fp32 dQ accumulator for the CUDA-core ones
  const size_t rows = static_cast<size_t>(p.cfg.B) * p.cfg.H * p.sz.Np;
  const size_t off_D = 256;
  const size_t off_x = off_D + ((rows * 4 + 255) & ~static_cast<size_t>(255));
  const size_t need = off_x + rows * 4 * (p.sz.tensor_core_bwd ? 1 : p.cfg.d);
  if (need > kNoAllocScratchBytes) return PRISM_ERR_UNSUPPORTED;  // problem too large for it
  uint8_t* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return PRISM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* D = reinterpret_cast<float*>(base + off_D);
  float* x = reinterpret_cast<float*>(base + off_x);
  if (cudaMemsetAsync(base, 0, 256, st) != cudaSuccess) return PRISM_ERR_CUDA;
  if (p.sz.tensor_core_bwd) {
    if (prism::launch_bwd_pre(p, Op, dOp, lse, D, x, nullptr, st) != cudaSuccess)
      return PRISM_ERR_CUDA;
    if (prism::launch_attn_dkdv_tc(p, Qp, Kp, Vp, dOp, x, D, n_valid, col_ptr, row_idx, scale,
                                   dKp, dVp, base, nullptr, st) != cudaSuccess)
      return PRISM_ERR_CUDA;
    // the whole key range in one pass (no partial-result scratch here)
    if (prism::launch_attn_dq_tc(p, Qp, Kp, Vp, dOp, lse, D, n_valid, row_ptr, col_idx, scale,
                                 dQp, base, nullptr, st) != cudaSuccess)
      return PRISM_ERR_CUDA;
  } else {
    if (prism::launch_bwd_pre(p, Op, dOp, lse, D, nullptr, x, st) != cudaSuccess)
      return PRISM_ERR_CUDA;
    if (prism::launch_attn_bwd_simt(p, Qp, Kp, Vp, dOp, lse, D, n_valid, col_ptr, row_idx, scale,
                                    x, dKp, dVp, st) != cudaSuccess)
      return PRISM_ERR_CUDA;
    if (prism::launch_dq_convert(p, x, scale, dQp, st) != cudaSuccess) return PRISM_ERR_CUDA;
  }
  return PRISM_OK;
}

extern "C" int prism_noalloc_device_status(void* stream) {
  uint8_t* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return PRISM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, base, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return PRISM_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PRISM_ERR_CUDA;
  if (word == prism::DEV_ERR_TIMEOUT) return PRISM_ERR_DEVICE_TIMEOUT;
  if (word != 0) return PRISM_ERR_DEVICE_BOUNDS;
  return PRISM_OK;
}
