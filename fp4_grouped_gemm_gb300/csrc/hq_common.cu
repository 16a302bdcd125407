// hq_common.cu -- library-wide state and small entry points: the device status
// word, capability constants, status strings, scale-buffer sizing, the
// bounded-wait self-test, tensor-map encoding and per-device caches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "hq_internal.h"
#include "hq_ptx.cuh"

namespace hq {

// One 32-bit status word per device that loads the library.  Kernels receive
// its device address as an argument (resolved per device below).
__device__ uint32_t g_status_word;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t* g_status_ptr[kMaxDevices] = {};
void* g_status_ctx[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::atomic<uint64_t> g_wait_limit_ns{1000000000ull};
std::atomic<int> g_tile_n{0};
std::atomic<int> g_use_2sm{1};
std::atomic<int64_t> g_inject_skip{-1};
using EncodeFn = decltype(&cuTensorMapEncodeTiled);
EncodeFn g_encode = nullptr;

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}
}  // namespace

void* current_context() {
  using CtxFn = CUresult (*)(CUcontext*);
  static CtxFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<CtxFn>(nullptr);
    return reinterpret_cast<CtxFn>(f);
  }();
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

uint32_t* status_word_ptr() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  void* ctx = current_context();
  std::lock_guard<std::mutex> lk(g_mu);
  // the cached address belongs to the context it was resolved in: resolve it
  // again when another context is current on this device
  if (!g_status_ptr[dev] || g_status_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<uint32_t*>(p);
    g_status_ctx[dev] = ctx;
  }
  return g_status_ptr[dev];
}

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(); }

int forced_tile_n() { return g_tile_n.load(); }

int64_t fault_injection_stage() { return g_inject_skip.load(); }

bool use_2sm() { return g_use_2sm.load() != 0; }

int pair_width() {
  const int v = g_use_2sm.load();
  return v == 256 || v == 384 ? v : 0;
}

int num_sms() {
  const int dev = current_device();
  if (dev < 0) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

// A tensor map depends only on its encoding arguments (not on the memory's
// contents), so recently encoded maps are kept and reused when every argument
// matches: encoding through the driver costs host time on every small call.
namespace {
struct MapKey {
  int dtype, rank, swizzle, dev;
  void* base;
  uint64_t dims[5], strides[4];
  uint32_t box[5];
};
constexpr int kMapCache = 32;
MapKey g_map_keys[kMapCache];
CUtensorMap g_maps[kMapCache];
int g_map_used = 0, g_map_next = 0;
std::mutex g_map_mu;
}  // namespace

int encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle) {
  if (rank < 1 || rank > 5) return HQ_ERR_INVALID;
  MapKey key;
  memset(&key, 0, sizeof(key));
  key.dtype = static_cast<int>(dtype);
  key.rank = rank;
  key.swizzle = static_cast<int>(swizzle);
  key.dev = current_device();
  key.base = base;
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
    if (i > 0) key.strides[i - 1] = strides_bytes[i - 1];
  }
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (int i = 0; i < g_map_used; ++i)
      if (memcmp(&g_map_keys[i], &key, sizeof(key)) == 0) {
        *map = g_maps[i];
        return HQ_OK;
      }
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return HQ_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeFn>(fn);
    }
  }
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bdim[5];
  cuuint32_t estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i > 0) gstride[i - 1] = strides_bytes[i - 1];
  }
  CUresult r = g_encode(map, dtype, rank, base, gdim, gstride, bdim, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return HQ_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    g_map_keys[g_map_next] = key;
    g_maps[g_map_next] = *map;
    g_map_next = (g_map_next + 1) % kMapCache;
    if (g_map_used < kMapCache) ++g_map_used;
  }
  return HQ_OK;
}

// Streaming floor probe: every 32-byte group of src is read (16-byte loads,
// four groups per thread in flight) and one 8-byte word, the XOR of its two
// halves, is written to dst (the quantiser's NVFP4 byte ratio).  bytes == 0
// launches the same grid with no work: the fixed cost of one launch.
__global__ void __launch_bounds__(256) stream_probe_kernel(const uint4* __restrict__ src, size_t groups,
                                                           uint2* __restrict__ dst) {
  const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t nt = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t base = tid; base < groups; base += 4 * nt) {
    uint4 v[4][2];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const size_t g = base + u * nt;
      const bool ok = g < groups;
      v[u][0] = ok ? __ldcs(src + 2 * g) : make_uint4(0, 0, 0, 0);
      v[u][1] = ok ? __ldcs(src + 2 * g + 1) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const size_t g = base + u * nt;
      if (g < groups)
        dst[g] = make_uint2(v[u][0].x ^ v[u][0].z ^ v[u][1].x ^ v[u][1].z,
                            v[u][0].y ^ v[u][0].w ^ v[u][1].y ^ v[u][1].w);
    }
  }
}

// Debug builds: one thread checks index 4 against the 4-element buffer below;
// the check fails, so the write is skipped and HQ_STATUS_BOUNDS is set.  The
// release build compiles the body away (and the host never launches it).
__device__ int g_debug_sink[4];
__global__ void debug_selftest_kernel(uint32_t* status) {
#if HQ_DEBUG
  const int n = 4;
  const int idx = n;
  if (in_bounds(idx < n, status)) g_debug_sink[idx & 3] = 1;
#else
  (void)status;
#endif
}

// Waits on an mbarrier that nothing arrives on; the bounded wait expires.
__global__ void selftest_wait_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    WaitCtx w{status, &abort_flag, limit_ns};
    wait_bounded(smem_u32(&bar), 0, w);
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Discrete weights (cuDNN frontend "Grouped GEMM + dGLU (SM100)", discrete
// mode: b_ptrs / sfb_ptrs hold one device pointer per expert).  One warp per
// expert copies the host-encoded template tensor map (the stacked layout of one
// expert) into shared memory, replaces its global address with b_ptrs[g] and
// publishes the result to maps[g] with the release fence of the tensor-map
// proxy; a kernel that loads through maps[g] issues the matching acquire
// before its first copy.  ok[g] = 1 when the expert's pointers are non-null
// and 16-byte aligned; otherwise ok[g] = 0, maps[g] keeps the template's
// address, HQ_STATUS_BAD_POINTER is set, and the GEMMs skip that expert.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) weight_maps_kernel(const __grid_constant__ CUtensorMap tmpl,
                                                          const int64_t* b_ptrs, const int64_t* sfb_ptrs,
                                                          CUtensorMap* maps, int32_t* ok, int L,
                                                          uint32_t* status) {
  __shared__ alignas(128) CUtensorMap sm[4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x * 4 + warp;
  if (g >= L) return;  // warp-uniform
  const uint64_t b = static_cast<uint64_t>(__ldg(b_ptrs + g));
  const uint64_t sf = sfb_ptrs ? static_cast<uint64_t>(__ldg(sfb_ptrs + g)) : 16u;
  const bool good = b != 0 && (b & 15u) == 0 && sf != 0 && (sf & 15u) == 0;
  reinterpret_cast<uint32_t*>(&sm[warp])[lane] = reinterpret_cast<const uint32_t*>(&tmpl)[lane];
  __syncwarp();
  const uint32_t sa = smem_u32(&sm[warp]);
  if (lane == 0 && good)
    asm volatile("tensormap.replace.tile.global_address.shared::cta.b1024.b64 [%0], %1;" ::"r"(sa),
                 "l"(b)
                 : "memory");
  __syncwarp();
  asm volatile(
      "tensormap.cp_fenceproxy.global.shared::cta.tensormap::generic.release.gpu.sync.aligned"
      " [%0], [%1], 128;" ::"l"(reinterpret_cast<uint64_t>(maps + g)),
      "r"(sa)
      : "memory");
  if (lane == 0) {
    ok[g] = good ? 1 : 0;
    if (!good) atomicOr(status, HQ_STATUS_BAD_POINTER);
  }
}

int build_weight_maps(const CUtensorMap& tmpl, const int64_t* b_ptrs, const int64_t* sfb_ptrs,
                      CUtensorMap* maps, int32_t* ok, int L, cudaStream_t st) {
  uint32_t* status = status_word_ptr();
  if (!status) return HQ_ERR_CUDA;
  weight_maps_kernel<<<(L + 3) / 4, 128, 0, st>>>(tmpl, b_ptrs, sfb_ptrs, maps, ok, L, status);
  return cudaGetLastError() == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Tensor-core issue-rate probe: one thread per CTA (per cluster pair) issues
// MMAs back to back on operands resident in shared memory; clock64 and the
// global timer bracket the timed MMAs, which complete on an mbarrier through
// tcgen05.commit.  Waits are bounded (2 s); a CTA whose wait expired reports
// zero cycles.
// ---------------------------------------------------------------------------
namespace {
constexpr int kProbeThreads = 128;

template <int KIND>
__host__ __device__ constexpr uint32_t probe_idesc(int m, int n) {
  return (KIND == 0 ? ((1u << 4) | (1u << 7) | (1u << 10))          // f32 <- bf16 x bf16
          : KIND == 1 ? ((0u << 7) | (0u << 10) | (1u << 23))        // E4M3, UE8M0
          : KIND == 3 ? ((1u << 7) | (1u << 10) | (1u << 23))        // E2M1, UE8M0
                      : ((1u << 7) | (1u << 10) | (0u << 23))) |     // E2M1, UE4M3
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

template <int KIND, int PAIR>
__global__ void __launch_bounds__(kProbeThreads, 1) mma_rate_kernel(int n, int iters, uint64_t* out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int b_rows = PAIR ? n / 2 : n;
  const int bytes = 16384 + b_rows * 128;  // A: 128 rows x 128 B, B: b_rows x 128 B
  const int warp = threadIdx.x >> 5;
  // operand bytes: small E4M3 / E2M1 / BF16 values, never NaN
  for (int i = threadIdx.x * 4; i < bytes; i += kProbeThreads * 4) {
    uint32_t h = static_cast<uint32_t>(i) * 2654435761u ^ blockIdx.x * 97u;
    h ^= h >> 13;
    h *= 0x5bd1e995u;
    h ^= h >> 15;
    *reinterpret_cast<uint32_t*>(smem + i) = h & 0x3F3F3F3Fu;
  }
  const uint32_t bar = sbase + bytes;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + bytes + 16);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    if (PAIR) { tmem_alloc_2sm(smem_u32(slot), 512); tmem_relinquish_2sm(); }
    else { tmem_alloc(smem_u32(slot), 512); tmem_relinquish(); }
  }
  __syncthreads();
  if (PAIR) cluster_sync();
  tc_fence_after();
  const uint32_t tb = *slot;
  {
    // scale columns [256, 288) of every lane: 1.0 (UE8M0 127, UE4M3 0x38)
    uint32_t v[16];
    const uint32_t one = KIND == 2 ? 0x38383838u : 0x7F7F7F7Fu;
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = one;
    const uint32_t lq = static_cast<uint32_t>((warp & 3) * 32) << 16;
    tmem_st_32x32b<16>(lq + tb + 256, v);
    tmem_st_32x32b<16>(lq + tb + 272, v);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();
  tc_fence_after();
  const bool issuer = threadIdx.x == 0 && (!PAIR || cluster_ctarank() == 0);
  if (issuer) {
    const uint64_t ad = smem_desc_sw128(sbase), bd = smem_desc_sw128(sbase + 16384);
    const uint32_t id = probe_idesc<KIND>(PAIR ? 256 : 128, n);
    const uint32_t sfa = tb + 256, sfb = tb + 272;
    auto run = [&](int count) {
      for (int it = 0; it < count; ++it) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t acc = (it | j) ? 1u : 0u;
          if (PAIR) {
            if (KIND == 0) mma_bf16_2sm(tb, ad + 2 * j, bd + 2 * j, id, acc);
            else if (KIND == 1) mma_mxf8_2sm(tb, ad + 2 * j, bd + 2 * j, id, sfa, sfb, acc);
            else if (KIND == 2) mma_nvf4_2sm(tb, ad + 2 * j, bd + 2 * j, id, sfa, sfb, acc);
            else mma_mxf4_2sm(tb, ad + 2 * j, bd + 2 * j, id, sfa, sfb, acc);
          } else {
            if (KIND == 0) mma_bf16(tb, ad + 2 * j, bd + 2 * j, id, acc);
            else if (KIND == 1) mma_mxf8(tb, ad + 2 * j, bd + 2 * j, id, sfa, sfb, acc);
            else if (KIND == 2) mma_nvf4(tb, ad + 2 * j, bd + 2 * j, id, sfa, sfb, acc);
            else mma_mxf4(tb, ad + 2 * j, bd + 2 * j, id, sfa, sfb, acc);
          }
        }
      }
      if (PAIR) tc_commit_2sm_mc(bar, 0x1);
      else tc_commit(bar);
    };
    run(16);  // warm-up
    bool ok = wait_drain(bar, 0, 2000000000ull);
    const uint64_t c0 = clock64(), g0 = globaltimer_ns();
    run(iters);
    ok = wait_drain(bar, 1, 2000000000ull) && ok;
    const uint64_t c1 = clock64(), g1 = globaltimer_ns();
    const int slot_i = PAIR ? blockIdx.x >> 1 : blockIdx.x;
    out[2 * slot_i] = ok ? c1 - c0 : 0;
    out[2 * slot_i + 1] = ok ? g1 - g0 : 0;
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();
  if (warp == 0) {
    tc_fence_after();
    if (PAIR) tmem_dealloc_2sm(tb, 512);
    else tmem_dealloc(tb, 512);
  }
}

template <int KIND, int PAIR>
int launch_mma_rate(int n, int iters, uint64_t* out, cudaStream_t st) {
  auto kern = mma_rate_kernel<KIND, PAIR>;
  // at least 120 KB of shared memory: one CTA per SM
  constexpr int kSmem = 120 * 1024;
  if (set_smem_once<mma_rate_kernel<KIND, PAIR>>(kSmem) != HQ_OK) return HQ_ERR_CUDA;
  const int sms = num_sms();
  if (sms < 2) return HQ_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(PAIR ? sms / 2 * 2 : sms));
  cfg.blockDim = dim3(kProbeThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, n, iters, out) == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
}

template <int KIND>
int launch_mma_rate_kind(int pair, int n, int iters, uint64_t* out, cudaStream_t st) {
  return pair ? launch_mma_rate<KIND, 1>(n, iters, out, st) : launch_mma_rate<KIND, 0>(n, iters, out, st);
}
}  // namespace

}  // namespace hq

extern "C" {

size_t hq_gemm_discrete_workspace_size(int L, int64_t dbias_n) {
  if (L < 1 || dbias_n < 0) return 0;
  size_t bytes = hq::discrete_maps_bytes(L);
  if (dbias_n > 0) bytes += (static_cast<size_t>(L) * 2 * dbias_n * sizeof(float) + 255) / 256 * 256;
  return bytes;
}


int hq_capabilities(hq_capabilities_t* out) {
  if (!out) return HQ_ERR_INVALID;
  out->abi_version = 2;
  out->sfatom_rows = 128;
  out->sfatom_cols = 4;
  out->sfatom_bytes = 512;
  out->group_mxfp8 = 32;
  out->group_nvfp4 = 16;
  out->contig_row_align = 256;
  out->tile_m = 128;
  out->ptr_align_bytes = 16;
  out->max_groups = 1024;
  out->glu_block = 32;
  out->group_mxfp4 = 32;
  return HQ_OK;
}

const char* hq_status_string(int status) {
  switch (status) {
    case HQ_OK: return "HQ_OK";
    case HQ_ERR_INVALID: return "HQ_ERR_INVALID: invalid argument (pointer, shape, stride or alignment)";
    case HQ_ERR_UNSUPPORTED: return "HQ_ERR_UNSUPPORTED: valid request not supported by this library";
    case HQ_ERR_CUDA: return "HQ_ERR_CUDA: a CUDA call failed";
    case HQ_ERR_TIMEOUT: return "HQ_ERR_TIMEOUT: a bounded pipeline wait expired on the device";
    default: return "unknown hq status";
  }
}

size_t hq_sf_bytes(int64_t rows, int64_t k, hq_mode mode) {
  int64_t gs = (mode == HQ_MXFP8 || mode == HQ_MXFP4 || mode == HQ_MXFP8_E5M2) ? 32
              : (mode == HQ_NVFP4 ? 16 : 0);
  if (gs == 0 || rows < 0 || k <= 0 || k % (4 * gs) != 0) return 0;
  return static_cast<size_t>((rows + 127) / 128 * 128) * static_cast<size_t>(k / gs);
}

int hq_get_device_status(uint32_t* out, int clear, hq_stream_t s) {
  if (!out) return HQ_ERR_INVALID;
  uint32_t* p = hq::status_word_ptr();
  if (!p) return HQ_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, p, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return HQ_ERR_CUDA;
  if (clear && cudaMemsetAsync(p, 0, sizeof(uint32_t), st) != cudaSuccess) return HQ_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return HQ_ERR_CUDA;
  *out = v;
  return (v & HQ_STATUS_WAIT_TIMEOUT) ? HQ_ERR_TIMEOUT : HQ_OK;
}

int hq_set_wait_limit_ns(uint64_t ns) {
  if (ns == 0) return HQ_ERR_INVALID;
  hq::g_wait_limit_ns.store(ns);
  return HQ_OK;
}

int hq_set_gemm_tile_n(int tile_n) {
  if (tile_n != 0 && tile_n != 128 && tile_n != 256) return HQ_ERR_INVALID;
  hq::g_tile_n.store(tile_n);
  return HQ_OK;
}

int hq_set_gemm_2sm(int enable) {
  if (enable != 0 && enable != 1 && enable != 256 && enable != 384) return HQ_ERR_INVALID;
  hq::g_use_2sm.store(enable);
  return HQ_OK;
}

int hq_set_fault_injection(int64_t skip_stage) {
  if (skip_stage < -1) return HQ_ERR_INVALID;
  hq::g_inject_skip.store(skip_stage);
  return HQ_OK;
}

int hq_selftest_wait_expiry(uint64_t limit_ns, hq_stream_t s) {
  if (limit_ns == 0 || limit_ns > 10000000000ull) return HQ_ERR_INVALID;
  uint32_t* status = hq::status_word_ptr();
  if (!status) return HQ_ERR_CUDA;
  hq::selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(s)>>>(status, limit_ns);
  return cudaGetLastError() == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
}

int hq_probe_stream(const void* src, size_t bytes, void* dst, hq_stream_t s) {
  if (bytes % 32 != 0) return HQ_ERR_INVALID;
  if (bytes > 0 && (!src || !dst)) return HQ_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) return HQ_ERR_INVALID;
  const int sms = hq::num_sms();
  if (sms <= 0) return HQ_ERR_CUDA;
  hq::stream_probe_kernel<<<static_cast<unsigned>(4 * sms), 256, 0, reinterpret_cast<cudaStream_t>(s)>>>(
      static_cast<const uint4*>(src), bytes / 32, static_cast<uint2*>(dst));
  return cudaGetLastError() == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
}

int hq_debug_build(void) { return HQ_DEBUG ? 1 : 0; }

int hq_debug_selftest(hq_stream_t s) {
  if (!HQ_DEBUG) return HQ_ERR_UNSUPPORTED;
  uint32_t* status = hq::status_word_ptr();
  if (!status) return HQ_ERR_CUDA;
  hq::debug_selftest_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(s)>>>(status);
  return cudaGetLastError() == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
}

int hq_probe_mma_rate(int kind, int pair, int n, int iters, uint64_t* out, hq_stream_t s) {
  if (kind < 0 || kind > 3 || (n != 128 && n != 256) || iters < 1 || iters > (1 << 20)) return HQ_ERR_INVALID;
  if (!out || (reinterpret_cast<uintptr_t>(out) & 7u)) return HQ_ERR_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  switch (kind) {
    case 0: return hq::launch_mma_rate_kind<0>(pair, n, iters, out, st);
    case 1: return hq::launch_mma_rate_kind<1>(pair, n, iters, out, st);
    case 2: return hq::launch_mma_rate_kind<2>(pair, n, iters, out, st);
    default: return hq::launch_mma_rate_kind<3>(pair, n, iters, out, st);
  }
}

}  // extern "C"
