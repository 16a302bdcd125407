// hq_quant.cu -- the group-wise quantiser (hq_quant) and the fused SwiGLU +
// requantisation pass (hq_swiglu_quant).
//
// Both are HBM-bound streaming passes.  A warp handles a 256-element segment of
// one row per step: every lane loads 16 bytes (8 BF16 values; the SwiGLU pass
// loads 8 gate and 8 up values), the lanes of one scale group (4 lanes for a
// 32-element MXFP8 group, 2 for a 16-element NVFP4 group) reduce |x| with
// shuffles, derive the scale byte, encode their 8 elements and store them with
// one 8-byte (E4M3) or 4-byte (packed E2M1) store, so each warp writes a
// contiguous 256- or 128-byte run.  The first lane of a group writes its
// scale byte at the SfAtom (or row-major) position.
//
// Scale rule (cuDNN frontend "Grouped GEMM + dGLU (SM100)", Step 3, with the
// HALOps group_wise_quant encodings), evaluated in IEEE float32:
//   s = (g * amax) * rcp_max,   rcp_max = 1/448 (E4M3) or 1/6 (E2M1)
//   MXFP8: UE8M0 = clamp(ceil(log2 s) + 127, 0, 254) (0 if s == 0),
//          q = E4M3(x * 2^(127 - UE8M0))
//   NVFP4: UE4M3 = E4M3(s), q = E2M1(x * (g / value(UE4M3))) (0 if value 0)
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "hq_internal.h"
#include "hq_ptx.cuh"

namespace hq {
namespace {

constexpr int kThreads = 256;
constexpr int kSegElems = 256;  // elements per warp step (32 lanes x 8)

struct QuantParams {
  const uint16_t* in;        // BF16 rows (quant: [rows, k]; swiglu: [rows, 2k])
  int64_t rows;
  int64_t k;                 // output elements per row (swiglu: H)
  int64_t in_stride;         // input row stride in elements
  int64_t S;                 // scale columns of the output layout
  int64_t S_real;            // scale columns holding real scales (k / group)
  int64_t rows_pad;          // ceil(rows / 128) * 128
  int swizzle;               // 1: SfAtom, 0: row-major
  const float* global_scale; // NVFP4 norm_const, may be null (= 1)
  uint8_t* q;
  uint8_t* sf;
  const int32_t* token_nums; // swiglu only, may be null
  int64_t rows_per_expert;
  int E;
  int zero_pad_rows;         // write 0 to the scale bytes of padding rows
  uint32_t* status;
};

__device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t s, int64_t S, int swizzle) {
  if (!swizzle) return r * S + s;
  return ((r >> 7) * (S >> 2) + (s >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (s & 3);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&x)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// ceil(log2 s) + 127 clamped to [0, 254] for s >= 0 (0 for s == 0), from the
// float32 bit pattern.
__device__ __forceinline__ uint32_t ue8m0_ceil(float s) {
  const uint32_t bits = __float_as_uint(s);
  if (bits == 0) return 0;
  const uint32_t e = bits >> 23, man = bits & 0x7FFFFFu;
  if (e == 0) {  // subnormal: s = man * 2^-149
    const int b = (32 - __clz(static_cast<int>(man - 1))) - 22;
    return b > 0 ? static_cast<uint32_t>(b) : 0u;
  }
  const uint32_t b = e + (man != 0 ? 1u : 0u);
  return b > 254u ? 254u : b;
}

__device__ __forceinline__ float pow2_neg_unbiased(uint32_t byte) {  // 2^(127 - byte)
  return byte <= 253u ? __uint_as_float((254u - byte) << 23) : __uint_as_float(0x00400000u);
}

template <int MODE>
__device__ __forceinline__ void encode_group_lane(const float (&x)[8], float amax, float g,
                                                  uint32_t& scale_byte, uint2& packed) {
  if (MODE == HQ_MXFP8) {
    const float s = __fmul_rn(__fmul_rn(g, amax), 1.0f / 448.0f);
    scale_byte = ue8m0_ceil(s);
    const float mult = pow2_neg_unbiased(scale_byte);
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      c[i] = cvt_e4m3x2(__fmul_rn(x[2 * i + 1], mult), __fmul_rn(x[2 * i], mult));
    packed.x = c[0] | (c[1] << 16);
    packed.y = c[2] | (c[3] << 16);
  } else {
    const float s = __fmul_rn(__fmul_rn(g, amax), 1.0f / 6.0f);
    scale_byte = cvt_e4m3x2(0.0f, s) & 0xFFu;
    const float sd = ue4m3_value(scale_byte);
    const float r = sd == 0.0f ? 0.0f : __fdiv_rn(g, sd);
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w |= cvt_e2m1x2(__fmul_rn(x[2 * i + 1], r), __fmul_rn(x[2 * i], r)) << (8 * i);
    packed.x = w;
    packed.y = 0;
  }
}

template <int MODE, bool SWIGLU>
__global__ void __launch_bounds__(kThreads) quant_kernel(const QuantParams p) {
  pdl_wait();
  constexpr int GS = MODE == HQ_MXFP8 ? 32 : 16;
  constexpr int LPG = GS / 8;  // lanes per scale group
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  const int64_t segs = (p.k + kSegElems - 1) / kSegElems;
  const int64_t items = p.rows * segs;
  const float g = (MODE == HQ_NVFP4 && p.global_scale) ? __ldg(p.global_scale) : 1.0f;

  for (int64_t item = warp; item < items; item += nwarps) {
    const int64_t row = item / segs;
    const int64_t col = (item - row * segs) * kSegElems + lane * 8;
    if (SWIGLU && p.token_nums) {
      const int64_t e = row / p.rows_per_expert;
      const int64_t local = row - e * p.rows_per_expert;
      int tn = __ldg(p.token_nums + e);
      if (tn < 0 || tn > p.rows_per_expert) {
        if (lane == 0 && local == 0) atomicOr(p.status, HQ_STATUS_TOKENS_CLAMPED);
        tn = tn < 0 ? 0 : static_cast<int>(p.rows_per_expert);
      }
      if (local >= tn) continue;  // warp-uniform: the whole row is skipped
    }
    const bool in_range = col < p.k;
    float x[8];
    if (in_range) {
      const uint16_t* src = p.in + row * p.in_stride + col;
      if (SWIGLU) {
        float gt[8], up[8];
        bf16x8_to_f32(__ldcs(reinterpret_cast<const uint4*>(src)), gt);
        bf16x8_to_f32(__ldcs(reinterpret_cast<const uint4*>(src + p.k)), up);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float e = expf(-gt[i]);
          const float t = __fdiv_rn(gt[i], __fadd_rn(1.0f, e));
          x[i] = __fmul_rn(up[i], t);
        }
      } else {
        bf16x8_to_f32(__ldcs(reinterpret_cast<const uint4*>(src)), x);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = 0.0f;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 1; o < LPG; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (!in_range) continue;
    uint32_t sbyte;
    uint2 packed;
    encode_group_lane<MODE>(x, amax, g, sbyte, packed);
    if (MODE == HQ_MXFP8) {
      *reinterpret_cast<uint2*>(p.q + row * p.k + col) = packed;
    } else {
      *reinterpret_cast<uint32_t*>(p.q + (row * p.k + col) / 2) = packed.x;
    }
    if ((lane % LPG) == 0) p.sf[sf_offset(row, col / GS, p.S, p.swizzle)] = static_cast<uint8_t>(sbyte);
  }

  // Scale bytes that hold 0: padding rows, and (swiglu, MXFP8) the columns
  // past k / 32 of written rows.
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * kThreads;
  if (p.zero_pad_rows) {
    const int64_t n = (p.rows_pad - p.rows) * p.S;
    for (int64_t i = tid; i < n; i += nthreads) {
      const int64_t r = p.rows + i / p.S, s = i % p.S;
      p.sf[sf_offset(r, s, p.S, p.swizzle)] = 0;
    }
  }
  if (p.S > p.S_real) {
    const int64_t extra = p.S - p.S_real;
    const int64_t n = p.rows * extra;
    for (int64_t i = tid; i < n; i += nthreads) {
      const int64_t r = i / extra, s = p.S_real + i % extra;
      if (SWIGLU && p.token_nums) {
        const int64_t e = r / p.rows_per_expert;
        int64_t tn = __ldg(p.token_nums + e);
        tn = tn < 0 ? 0 : (tn > p.rows_per_expert ? p.rows_per_expert : tn);
        if (r - e * p.rows_per_expert >= tn) continue;
      }
      p.sf[sf_offset(r, s, p.S, p.swizzle)] = 0;
    }
  }
  pdl_launch_dependents();
}

template <int MODE, bool SWIGLU>
int launch_quant(const QuantParams& p, cudaStream_t st, bool pdl) {
  const int sms = num_sms();
  if (sms <= 0) return HQ_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quant_kernel<MODE, SWIGLU>, kThreads,
                                                    0) != cudaSuccess)
    return HQ_ERR_CUDA;
  if (per_sm < 1) per_sm = 1;
  const int64_t segs = (p.k + kSegElems - 1) / kSegElems;
  const int64_t warps_needed = p.rows * segs + 1;
  int64_t blocks = (warps_needed + (kThreads / 32) - 1) / (kThreads / 32);
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaError_t e = launch(quant_kernel<MODE, SWIGLU>, dim3(static_cast<unsigned>(blocks)),
                         dim3(kThreads), 0, st, pdl, p);
  return e == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
}

int dispatch(hq_mode mode, bool swiglu, const QuantParams& p, cudaStream_t st, bool pdl) {
  if (mode == HQ_MXFP8)
    return swiglu ? launch_quant<HQ_MXFP8, true>(p, st, pdl) : launch_quant<HQ_MXFP8, false>(p, st, pdl);
  return swiglu ? launch_quant<HQ_NVFP4, true>(p, st, pdl) : launch_quant<HQ_NVFP4, false>(p, st, pdl);
}

}  // namespace
}  // namespace hq

extern "C" {

int hq_quant(const hq_bf16* x, int64_t m, int64_t k, hq_mode mode, int use_swizzle,
             const float* global_scale, void* q_out, uint8_t* sf_out, int use_pdl,
             hq_stream_t s) {
  if (mode != HQ_MXFP8 && mode != HQ_NVFP4) return HQ_ERR_INVALID;
  const int64_t gs = mode == HQ_MXFP8 ? 32 : 16;
  if (m < 0 || k <= 0 || k % (4 * gs) != 0) return HQ_ERR_INVALID;
  if (mode == HQ_MXFP8 && global_scale) return HQ_ERR_UNSUPPORTED;
  if (m == 0) return HQ_OK;
  if (!x || !q_out || !sf_out) return HQ_ERR_INVALID;
  if (!hq::aligned16(x) || !hq::aligned16(q_out) || !hq::aligned16(sf_out)) return HQ_ERR_INVALID;
  if (global_scale && (reinterpret_cast<uintptr_t>(global_scale) & 3u)) return HQ_ERR_INVALID;
  hq::QuantParams p{};
  p.in = x;
  p.rows = m;
  p.k = k;
  p.in_stride = k;
  p.S = k / gs;
  p.S_real = k / gs;
  p.rows_pad = (m + 127) / 128 * 128;
  p.swizzle = use_swizzle ? 1 : 0;
  p.global_scale = global_scale;
  p.q = static_cast<uint8_t*>(q_out);
  p.sf = sf_out;
  p.zero_pad_rows = 1;
  p.status = hq::status_word_ptr();
  if (!p.status) return HQ_ERR_CUDA;
  return hq::dispatch(mode, false, p, reinterpret_cast<cudaStream_t>(s), use_pdl != 0);
}

int hq_swiglu_quant(const hq_bf16* in, int64_t rows, int64_t H, const int32_t* token_nums, int E,
                    int64_t rows_per_expert, hq_mode mode, const float* global_scale,
                    void* q_out, uint8_t* sf_out, hq_stream_t s) {
  if (mode != HQ_MXFP8 && mode != HQ_NVFP4) return HQ_ERR_INVALID;
  if (rows < 0 || H <= 0) return HQ_ERR_INVALID;
  if (mode == HQ_MXFP8 && H % 128 != 0) return HQ_ERR_INVALID;
  if (mode == HQ_NVFP4 && H % 64 != 0) return HQ_ERR_INVALID;
  if (mode == HQ_MXFP8 && global_scale) return HQ_ERR_UNSUPPORTED;
  if (token_nums) {
    if (E <= 0 || rows_per_expert <= 0 || static_cast<int64_t>(E) * rows_per_expert != rows)
      return HQ_ERR_INVALID;
  }
  if (rows == 0) return HQ_OK;
  if (!in || !q_out || !sf_out) return HQ_ERR_INVALID;
  if (!hq::aligned16(in) || !hq::aligned16(q_out) || !hq::aligned16(sf_out)) return HQ_ERR_INVALID;
  const int64_t gs = mode == HQ_MXFP8 ? 32 : 16;
  hq::QuantParams p{};
  p.in = in;
  p.rows = rows;
  p.k = H;
  p.in_stride = 2 * H;
  p.S = mode == HQ_MXFP8 ? (H + 511) / 512 * 16 : H / 16;
  p.S_real = H / gs;
  p.rows_pad = (rows + 127) / 128 * 128;
  p.swizzle = 1;
  p.global_scale = global_scale;
  p.q = static_cast<uint8_t*>(q_out);
  p.sf = sf_out;
  p.token_nums = token_nums;
  p.rows_per_expert = token_nums ? rows_per_expert : rows;
  p.E = token_nums ? E : 1;
  p.zero_pad_rows = token_nums ? 0 : 1;
  p.status = hq::status_word_ptr();
  if (!p.status) return HQ_ERR_CUDA;
  return hq::dispatch(mode, true, p, reinterpret_cast<cudaStream_t>(s), false);
}

}  // extern "C"
