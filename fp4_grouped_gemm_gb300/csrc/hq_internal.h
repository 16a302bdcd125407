// hq_internal.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/hq.h"

namespace hq {

// The CUDA context current on the calling thread (driver handle), or nullptr.
void* current_context();

// Device address of the status word on the current device (resolved with
// cudaGetSymbolAddress once per device and context); nullptr on failure.
uint32_t* status_word_ptr();

// Current limit for bounded pipeline waits, in nanoseconds.
uint64_t wait_limit_ns();

// Number of SMs of the current device (cached per device); 0 on failure.
int num_sms();

// Stage whose "full" arrival the pair GEMM's first producer withholds (-1:
// none; set by hq_set_fault_injection for the abort-path test).
int64_t fault_injection_stage();

// Forced GEMM tile width (0 = automatic).
int forced_tile_n();

// Whether GEMMs may use the 2-SM (cluster pair) kernel.
bool use_2sm();

// Forced pair tile width (256 or 384), or 0 to choose automatically.
int pair_width();

// cuTensorMapEncodeTiled through the runtime's driver entry point.
// Returns HQ_OK or HQ_ERR_CUDA.
int encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle);

// dbias[i] = bf16(float(dbias[i]) + ws[i]) for i < count, on stream st (the
// final pass of the dGLU GEMMs' dbias reduction).  Returns HQ_OK or HQ_ERR_CUDA.
// dbias[i] = bf16(dbias[i] + ws[i]); pdl: launched as a programmatic
// dependent of the preceding kernel, whose completion it waits for first.
int dbias_finalize(uint16_t* dbias, const float* ws, int64_t count, cudaStream_t st, bool pdl = false);
// Zeroes a[0..na) and b[0..nb) (either may be empty); lets the next kernel,
// if launched as a programmatic dependent, start at once (that kernel waits
// for the zeroes before it adds into them).
int zero_floats(float* a, int64_t na, float* b, int64_t nb, cudaStream_t st);

// Discrete weights: the leading part of the caller's workspace holds one
// 128-byte tensor map per expert, then one int32 flag per expert (1: the
// expert's pointers passed the device checks), rounded up to 256 bytes.
inline size_t discrete_maps_bytes(int L) {
  return (static_cast<size_t>(L) * (sizeof(CUtensorMap) + sizeof(int32_t)) + 255) / 256 * 256;
}

// N-major discrete BF16 weights: bytes of one expert's K-major copy (256-byte
// multiple), and the pass that writes every expert's copy and pointer.
size_t nmajor_copy_bytes(int64_t n, int64_t k);
int nmajor_to_kmajor(const int64_t* b_ptrs, uint16_t* copies, int64_t* ptrs, int L, int64_t n, int64_t k,
                     cudaStream_t st);

// Launches the kernel that turns b_ptrs (and the checks of sfb_ptrs, which
// may be null) into per-expert tensor maps built from tmpl.  Returns HQ_OK or
// HQ_ERR_CUDA.
int build_weight_maps(const CUtensorMap& tmpl, const int64_t* b_ptrs, const int64_t* sfb_ptrs,
                      CUtensorMap* maps, int32_t* ok, int L, cudaStream_t st);

// Raises the dynamic shared-memory limit of kernel Kern to `bytes` once per
// device (the attribute persists, and setting it on every launch costs host
// time on the small problems).  Returns HQ_OK or HQ_ERR_CUDA.
template <auto Kern>
int set_smem_once(int bytes) {
  static std::atomic<uint64_t> done{0};  // one bit per device 0..63
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return HQ_ERR_CUDA;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return HQ_OK;
  if (cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return HQ_ERR_CUDA;
  done.fetch_or(bit, std::memory_order_release);
  return HQ_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch with optional programmatic-dependent-launch attribute.
template <typename... KArgs, typename... Args>
inline cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace hq
