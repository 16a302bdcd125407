// hq_quant.cu -- the group-wise quantiser (hq_quant) and the fused SwiGLU +
// requantisation pass (hq_swiglu_quant).
//
// Both are HBM-bound streaming passes.  Each lane owns whole scale groups
// (32 values for MXFP8, 16 for NVFP4): it loads the group with 16-byte loads
// (the SwiGLU pass also loads the matching up values), takes |x|max locally,
// derives the scale byte, encodes the group and stores it with 16-byte (E4M3)
// or 8-byte (packed E2M1) stores; a warp step covers 32 consecutive groups of
// one row.  Four consecutive groups share one 32-bit word of the SfAtom (and
// row-major) scale layout; their bytes are gathered by shuffles and written
// with one 4-byte store.  NVFP4's per-group multiplier g / value(UE4M3) comes
// from a 128-entry table each CTA builds once with IEEE division.
//
// Scale rule (cuDNN frontend "Grouped GEMM + dGLU (SM100)", Step 3, with the
// HALOps group_wise_quant encodings), evaluated in IEEE float32:
//   s = (g * amax) * rcp_max,   rcp_max = 1/448 (E4M3), 1/57344 (E5M2) or 1/6 (E2M1)
//   MXFP8: UE8M0 = clamp(ceil(log2 s) + 127, 0, 254) (0 if s == 0),
//          q = E4M3(x * 2^(127 - UE8M0))
//   NVFP4: UE4M3 = E4M3(s), q = E2M1(x * (g / value(UE4M3))) (0 if value 0)
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "hq_internal.h"
#include "hq_ptx.cuh"

namespace hq {
namespace {

constexpr int kThreads = 256;
// experts a token-count array may hold (their valid-row prefix is kept in
// shared memory)
constexpr int kMaxCountExperts = 8192;

// Lanes that share one scale group: the MXFP8 SwiGLU pass splits each
// 32-value group over a lane pair (two groups in flight per lane pair: fewer
// registers per lane and more warps resident per SM than one whole group per
// lane, which the other passes keep).
__host__ __device__ constexpr int lanes_per_group(int mode, bool swiglu) {
  return swiglu && mode == HQ_MXFP8 ? 2 : 1;
}
// Groups a lane (or lane pair) holds in flight.
__host__ __device__ constexpr int groups_per_lane(int mode, bool swiglu) {
  return mode == HQ_NVFP4 ? (swiglu ? 2 : 4) : (swiglu ? 2 : 1);
}
// Scale groups of one row a warp takes per item.
__host__ __device__ constexpr int groups_per_item(int mode, bool swiglu) {
  return 32 / lanes_per_group(mode, swiglu) * groups_per_lane(mode, swiglu);
}

struct QuantParams {
  const uint16_t* in;        // BF16 (or FP16) rows (quant: [rows, k]; swiglu: [rows, 2k])
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
  const int32_t* token_nums; // valid rows per block of rows_per_expert rows, or null (all valid)
  int64_t rows_per_expert;
  int E;
  int zero_pad_rows;         // write 0 to the scale bytes of padding rows
  uint32_t* status;
};

__device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t s, int64_t S, int swizzle) {
  if (!swizzle) return r * S + s;
  return ((r >> 7) * (S >> 2) + (s >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (s & 3);
}

// exp(-a) for two values without a library call: with t = -a log2(e) split
// as t_hi = fl(-a * L) (L = log2(e) rounded to float) plus r, where the FMA
// residual fma(-a, L, -t_hi) recovers the product's rounding error exactly
// (the error-free product transformation of Ogita, Rump and Oishi, "Accurate
// sum and dot product", 2005) and -a * L_lo adds log2(e) - L, exp(-a) =
// 2^t_hi * 2^r with 2^t_hi from the hardware base-2 exponential and
// 2^r = 1 + r ln 2 to within r^2 (|r| < 2^-16 wherever 2^t_hi is finite and
// normal).  The error is that of ex2.approx plus about 2^-23, independent of
// |a|: a product fl(-a * L) alone would add |a| 2^-24.  2^t_hi = inf (a <
// -88.7) stays inf and 0 stays 0: the correction factor is positive.
__device__ __forceinline__ void exp_neg_x2(float a0, float a1, float& e0, float& e1) {
  constexpr float kL2E = 1.44269502162933349609375f;  // log2(e) rounded to float
  constexpr float kL2ELo = 1.925963033500011e-08f;    // log2(e) - kL2E
  constexpr float kLn2 = 0.693147182464599609375f;
  float t0, t1, r0, r1;
  mul_f32x2(t0, t1, a0, a1, -kL2E);
  fma_f32x2(r0, r1, a0, a1, -kL2E, -kL2E, -t0, -t1);       // exact residual
  fma_f32x2(r0, r1, a0, a1, -kL2ELo, -kL2ELo, r0, r1);     // + (-a) (log2 e - L)
  fma_f32x2(r0, r1, r0, r1, kLn2, kLn2, 1.0f, 1.0f);       // 1 + r ln 2
  mul2_f32x2(e0, e1, ex2_approx_ftz(t0), ex2_approx_ftz(t1), r0, r1);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&x)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// eight FP16 values (exact conversion to float32)
__device__ __forceinline__ void f16x8_to_f32(const uint4& v, float (&x)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}


// Eight floats -> one word of eight E2M1 codes (element 2 j in the low nibble
// of byte j): four paired conversions packed with one vector move.
__device__ __forceinline__ uint32_t cvt_e2m1x8(float x0, float x1, float x2, float x3, float x4,
                                               float x5, float x6, float x7) {
  uint32_t w;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(w)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3), "f"(x4), "f"(x5), "f"(x6), "f"(x7));
  return w;
}

// Four floats -> one word of four E4M3 codes (element j in byte j).
__device__ __forceinline__ uint32_t cvt_e4m3x4(float x0, float x1, float x2, float x3) {
  uint32_t w;
  asm("{\n\t.reg .b16 l, h;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 l, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h, %4, %3;\n\t"
      "mov.b32 %0, {l, h};\n\t}"
      : "=r"(w)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return w;
}

// Four floats -> one word of four E5M2 codes (element j in byte j).
__device__ __forceinline__ uint32_t cvt_e5m2x4(float x0, float x1, float x2, float x3) {
  uint32_t w;
  asm("{\n\t.reg .b16 l, h;\n\t"
      "cvt.rn.satfinite.e5m2x2.f32 l, %2, %1;\n\t"
      "cvt.rn.satfinite.e5m2x2.f32 h, %4, %3;\n\t"
      "mov.b32 %0, {l, h};\n\t}"
      : "=r"(w)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return w;
}

// LPG lanes quantise one scale group; each holds GL = group / LPG of its
// values x[0..GL) (a lane pair: the even lane the first half).  MXFP8 writes
// GL E4M3 bytes to qw[0..GL/4); NVFP4 and MXFP4 write GL/2 packed bytes to
// qw[0..GL/8).  All 32 lanes must call it (the pair's amax is a shuffle).
template <int MODE, int GL, int LPG = 1>
__device__ __forceinline__ uint32_t encode_group(const float (&x)[GL], float g,
                                                 const float* r_table, uint32_t (&qw)[GL / 4]) {
  constexpr int GS = GL;  // values this lane encodes
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < GS; ++i) amax = fmaxf(amax, fabsf(x[i]));
  if (LPG == 2) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  if (MODE == HQ_MXFP8 || MODE == HQ_MXFP8_E5M2) {
    // s = (g amax) / max element (448 for E4M3, 57344 for E5M2), rounded up
    // to a power of two; the products x * 2^(127 - byte) are exact
    constexpr float kRcpMax = MODE == HQ_MXFP8 ? 1.0f / 448.0f : 1.0f / 57344.0f;
    const float s = __fmul_rn(__fmul_rn(g, amax), kRcpMax);
    const uint32_t byte = ue8m0_ceil(s);
    const float mult = pow2_neg_unbiased(byte);
#pragma unroll
    for (int i = 0; i < GS / 4; ++i) {
      float y[4];
      mul_f32x2(y[0], y[1], x[4 * i], x[4 * i + 1], mult);
      mul_f32x2(y[2], y[3], x[4 * i + 2], x[4 * i + 3], mult);
      qw[i] = MODE == HQ_MXFP8 ? cvt_e4m3x4(y[0], y[1], y[2], y[3]) : cvt_e5m2x4(y[0], y[1], y[2], y[3]);
    }
    return byte;
  } else if (MODE == HQ_MXFP4) {
    // UE8M0 as for MXFP8, with the E2M1 range: s = amax * fp32(1/6), rounded up
    // to a power of two; the products x * 2^(127 - byte) are exact
    const float s = __fmul_rn(amax, 1.0f / 6.0f);
    const uint32_t byte = ue8m0_ceil(s);
    const float mult = pow2_neg_unbiased(byte);
#pragma unroll
    for (int i = 0; i < GS / 8; ++i) {
      float y[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) mul_f32x2(y[2 * j], y[2 * j + 1], x[8 * i + 2 * j], x[8 * i + 2 * j + 1], mult);
      qw[i] = cvt_e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
    }
    return byte;
  } else {
    const float s = __fmul_rn(__fmul_rn(g, amax), 1.0f / 6.0f);
    const uint32_t byte = cvt_e4m3x2(0.0f, s) & 0x7Fu;
    const float r = r_table[byte];  // g / value(byte), 0 for a zero scale
#pragma unroll
    for (int i = 0; i < GS / 8; ++i) {
      float y[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) mul_f32x2(y[2 * j], y[2 * j + 1], x[8 * i + 2 * j], x[8 * i + 2 * j + 1], r);
      qw[i] = cvt_e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
    }
    return byte;
  }
}

// F16IN: the input rows hold IEEE binary16 values instead of BF16.
// COUNTS: p.token_nums is set (only each expert's first token_nums[e] rows).
template <int MODE, bool SWIGLU, bool F16IN = false, bool COUNTS = false>
__global__ void __launch_bounds__(kThreads) quant_kernel(const QuantParams p) {
  constexpr int GS = MODE == HQ_NVFP4 ? 16 : 32;
  constexpr int LPG = lanes_per_group(MODE, SWIGLU);
  constexpr int GL = GS / LPG;        // values per lane and group
  constexpr int NV = GL / 8;          // 16-byte loads per operand, group and lane
  constexpr int U = groups_per_lane(MODE, SWIGLU);  // groups a lane holds in flight
  constexpr int GPI = groups_per_item(MODE, SWIGLU);
  constexpr int GPU_ = GPI / U;       // groups per warp and u
  __shared__ float r_table[128];
  pdl_wait();  // the global scale and the input may come from the preceding kernel
  const float g = (MODE == HQ_NVFP4 && p.global_scale) ? __ldg(p.global_scale) : 1.0f;
  if (MODE == HQ_NVFP4) {
    // g / value(UE4M3 code) for every positive code, IEEE division
    if (threadIdx.x < 128) {
      const float sd = ue4m3_value(threadIdx.x);
      r_table[threadIdx.x] = sd == 0.0f ? 0.0f : __fdiv_rn(g, sd);
    }
    __syncthreads();
  }
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  // token_nums: only the first token_nums[e] rows of each expert's
  // rows_per_expert are processed.  One warp turns the (clamped, flagged)
  // counts into an exclusive prefix of valid rows in shared memory, so the
  // items below run over valid rows only.
  extern __shared__ int32_t s_valid_prefix[];  // [E + 1] with token_nums
  if (COUNTS) {
    if (threadIdx.x < 32) {
      int32_t carry = 0;
      bool clamped = false;
      for (int base = 0; base < p.E; base += 32) {
        const int e = base + lane;
        int32_t c = 0;
        if (e < p.E) {
          c = __ldg(p.token_nums + e);
          if (c < 0 || c > p.rows_per_expert) {
            clamped = true;
            c = c < 0 ? 0 : static_cast<int32_t>(p.rows_per_expert);
          }
        }
        int32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += u;
        }
        if (e < p.E) s_valid_prefix[e] = carry + incl - c;
        carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      if (lane == 0) s_valid_prefix[p.E] = carry;
      if (__any_sync(0xFFFFFFFFu, clamped) && lane == 0 && blockIdx.x == 0)
        atomicOr(p.status, HQ_STATUS_TOKENS_CLAMPED);
    }
    __syncthreads();
  }
  // an item is GPI consecutive groups of one (valid) row; lane l works on
  // groups l / LPG, l / LPG + GPI / U, ... (part l % LPG of each)
  const int64_t groups_row = p.S_real;
  const int64_t chunks = (groups_row + GPI - 1) / GPI;
  const int64_t valid_rows = COUNTS ? s_valid_prefix[p.E] : p.rows;
  const int64_t items = valid_rows * chunks;
  const bool small = items < (1ll << 31);

  // Software pipeline: the loads of a warp's next item are issued before the
  // current item is encoded, so load latency overlaps the arithmetic.
  // item -> (row, first group): valid row vr = item / chunks, which with
  // token_nums lies in the last expert e whose prefix is <= vr; a warp's
  // items increase, so its expert index only moves forward
  // cur_e's first valid row and the next expert's, kept in registers
  int cur_e = 0;
  int64_t cur_base = 0, next_bound = 0;
  auto set_expert = [&](int e) {
    cur_e = e;
    cur_base = s_valid_prefix[e];
    next_bound = e + 1 < p.E ? s_valid_prefix[e + 1] : INT64_MAX;
  };
  auto item_pos = [&](int64_t item, int64_t& row, int64_t& s0) {
    const int64_t vr = small ? static_cast<int64_t>(static_cast<uint32_t>(item) / static_cast<uint32_t>(chunks))
                             : item / chunks;
    s0 = (item - vr * chunks) * GPI;
    if (!COUNTS) {
      row = vr;
      return;
    }
    while (vr >= next_bound) set_expert(cur_e + 1);
    row = static_cast<int64_t>(cur_e) * p.rows_per_expert + (vr - cur_base);
  };
  uint4 v0[U][NV], v1[U][NV];
  int64_t next_row = 0, next_s0 = 0;  // position of the item whose loads are in v0 / v1
  auto load_item = [&](int64_t item) {
    int64_t row, s0;
    item_pos(item, row, s0);
    next_row = row;
    next_s0 = s0;
    const uint16_t* src_row = p.in + row * p.in_stride;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t s = s0 + u * GPU_ + lane / LPG;
      const bool ok = s < groups_row;
      const uint4* src = reinterpret_cast<const uint4*>(src_row + s * GS + (lane % LPG) * GL);
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        v0[u][i] = ok ? __ldcs(src + i) : make_uint4(0, 0, 0, 0);
        if (SWIGLU) v1[u][i] = ok ? __ldcs(src + i + p.k / 8) : make_uint4(0, 0, 0, 0);
      }
    }
  };
  if (COUNTS && warp < items) {
    // the warp's first expert by binary search; later ones by stepping
    const int64_t vr = warp / chunks;
    int lo = 0, hi = p.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_valid_prefix[mid] <= vr) lo = mid; else hi = mid - 1;
    }
    set_expert(lo);
  }
  if (warp < items) load_item(warp);
  for (int64_t item = warp; item < items; item += nwarps) {
    uint4 c0[U][NV], c1[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        c0[u][i] = v0[u][i];
        if (SWIGLU) c1[u][i] = v1[u][i];
      }
    const int64_t row = next_row, s0 = next_s0;  // this item's position (set when its loads were issued)
    if (item + nwarps < items) load_item(item + nwarps);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t s = s0 + u * GPU_ + lane / LPG;
      if (s0 + u * GPU_ >= groups_row) break;  // warp-uniform
      float x[GL];
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        float a[8];
        if (F16IN) f16x8_to_f32(c0[u][i], a);
        else bf16x8_to_f32(c0[u][i], a);
        if (SWIGLU) {
          float b[8];
          bf16x8_to_f32(c1[u][i], b);
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            // silu(gate) = gate / (1 + exp(-gate)), in pairs; the reciprocal
            // is the hardware approximation (within 1 ulp)
            float e0, e1, d0, d1, t0, t1;
            exp_neg_x2(a[j], a[j + 1], e0, e1);
            add_f32x2(d0, d1, e0, e1, 1.0f, 1.0f);
            mul2_f32x2(t0, t1, a[j], a[j + 1], rcp_approx(d0), rcp_approx(d1));
            mul2_f32x2(x[8 * i + j], x[8 * i + j + 1], b[j], b[j + 1], t0, t1);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) x[8 * i + j] = a[j];
        }
      }
      uint32_t qw[GL / 4];
      const uint32_t byte = encode_group<MODE, GL, LPG>(x, g, r_table, qw);
      // four consecutive groups (lane groups 4j..4j+3) share one 32-bit scale word
      const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, byte, LPG);
      const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, byte, 2 * LPG);
      const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, byte, 3 * LPG);
      if (s >= groups_row) continue;
      const int64_t e0 = row * p.k + s * GS + (lane % LPG) * GL;  // first element of this lane
      // debug builds: the codes lie inside q (the scale word: below)
      if (!in_bounds(row < p.rows && s * GS + (lane % LPG) * GL + GL <= p.k, p.status)) continue;
      if (MODE == HQ_MXFP8 || MODE == HQ_MXFP8_E5M2) {
        uint4* dst = reinterpret_cast<uint4*>(p.q + e0);
#pragma unroll
        for (int i = 0; i < GL / 16; ++i) dst[i] = make_uint4(qw[4 * i], qw[4 * i + 1], qw[4 * i + 2], qw[4 * i + 3]);
      } else if (MODE == HQ_MXFP4) {
        *reinterpret_cast<uint4*>(p.q + e0 / 2) = make_uint4(qw[0], qw[1], qw[2], qw[3]);
      } else if (GL == 16) {
        *reinterpret_cast<uint2*>(p.q + e0 / 2) = make_uint2(qw[0], qw[1]);
      } else {
        *reinterpret_cast<uint32_t*>(p.q + e0 / 2) = qw[0];
      }
      // the lane of the first of four groups (s % 4 == 0) writes their word
      if ((lane & (4 * LPG - 1)) == 0 &&
          in_bounds(sf_offset(row, s, p.S, p.swizzle) + 4 <= p.rows_pad * p.S, p.status)) {
        const uint32_t word = byte | (b1 << 8) | (b2 << 16) | (b3 << 24);
        *reinterpret_cast<uint32_t*>(p.sf + sf_offset(row, s, p.S, p.swizzle)) = word;
      }
    }
  }

  // Scale bytes that hold 0: padding rows, and (swiglu, MXFP8) the columns
  // past k / 32 of written rows.
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * kThreads;
  if (p.zero_pad_rows) {
    const int64_t n = (p.rows_pad - p.rows) * p.S;
    for (int64_t i = tid; i < n; i += nthreads) {
      const int64_t r = p.rows + i / p.S, s = i % p.S;
      if (in_bounds(sf_offset(r, s, p.S, p.swizzle) < p.rows_pad * p.S, p.status))
        p.sf[sf_offset(r, s, p.S, p.swizzle)] = 0;
    }
  }
  if (p.S > p.S_real) {
    const int64_t extra = p.S - p.S_real;
    const int64_t n = p.rows * extra;
    for (int64_t i = tid; i < n; i += nthreads) {
      const int64_t r = i / extra, s = p.S_real + i % extra;
      if (COUNTS) {
        const int64_t e = r / p.rows_per_expert;
        int64_t tn = __ldg(p.token_nums + e);
        tn = tn < 0 ? 0 : (tn > p.rows_per_expert ? p.rows_per_expert : tn);
        if (r - e * p.rows_per_expert >= tn) continue;
      }
      if (in_bounds(sf_offset(r, s, p.S, p.swizzle) < p.rows_pad * p.S, p.status))
        p.sf[sf_offset(r, s, p.S, p.swizzle)] = 0;
    }
  }
  pdl_launch_dependents();
}

template <int MODE, bool SWIGLU, bool F16IN = false, bool COUNTS = false>
int launch_quant(const QuantParams& p, cudaStream_t st, bool pdl) {
  const int sms = num_sms();
  if (sms <= 0) return HQ_ERR_CUDA;
  // the valid-row prefix (token counts only) lives in dynamic shared memory
  const size_t smem = COUNTS ? static_cast<size_t>(p.E + 1) * sizeof(int32_t) : 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quant_kernel<MODE, SWIGLU, F16IN, COUNTS>,
                                                    kThreads, smem) != cudaSuccess)
    return HQ_ERR_CUDA;
  if (per_sm < 1) per_sm = 1;
  constexpr int64_t kItem = groups_per_item(MODE, SWIGLU);
  const int64_t warps_needed = p.rows * ((p.S_real + kItem - 1) / kItem);
  int64_t blocks = (warps_needed + (kThreads / 32) - 1) / (kThreads / 32);
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaError_t e = launch(quant_kernel<MODE, SWIGLU, F16IN, COUNTS>, dim3(static_cast<unsigned>(blocks)),
                         dim3(kThreads), smem, st, pdl, p);
  return e == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
}

int dispatch_f16(hq_mode mode, const QuantParams& p, cudaStream_t st, bool pdl) {
  if (mode == HQ_MXFP8) return launch_quant<HQ_MXFP8, false, true>(p, st, pdl);
  if (mode == HQ_MXFP8_E5M2) return launch_quant<HQ_MXFP8_E5M2, false, true>(p, st, pdl);
  if (mode == HQ_MXFP4) return launch_quant<HQ_MXFP4, false, true>(p, st, pdl);
  return launch_quant<HQ_NVFP4, false, true>(p, st, pdl);
}

// With per-expert counts (token_nums) only the valid rows are mapped to work.
template <bool COUNTS>
int dispatch_bf16(hq_mode mode, bool swiglu, const QuantParams& p, cudaStream_t st, bool pdl) {
  if (mode == HQ_MXFP8)
    return swiglu ? launch_quant<HQ_MXFP8, true, false, COUNTS>(p, st, pdl)
                  : launch_quant<HQ_MXFP8, false, false, COUNTS>(p, st, pdl);
  if (mode == HQ_MXFP4) return swiglu ? HQ_ERR_INVALID : launch_quant<HQ_MXFP4, false, false, COUNTS>(p, st, pdl);
  if (mode == HQ_MXFP8_E5M2)
    return swiglu ? HQ_ERR_INVALID : launch_quant<HQ_MXFP8_E5M2, false, false, COUNTS>(p, st, pdl);
  return swiglu ? launch_quant<HQ_NVFP4, true, false, COUNTS>(p, st, pdl)
                : launch_quant<HQ_NVFP4, false, false, COUNTS>(p, st, pdl);
}

int dispatch(hq_mode mode, bool swiglu, const QuantParams& p, cudaStream_t st, bool pdl) {
  return p.token_nums ? dispatch_bf16<true>(mode, swiglu, p, st, pdl)
                      : dispatch_bf16<false>(mode, swiglu, p, st, pdl);
}

// Shared host side of hq_quant / hq_quant_f16: validation, then the launch.
int quant_entry(const uint16_t* x, bool f16, int64_t m, int64_t k, hq_mode mode, int use_swizzle,
                const float* global_scale, void* q_out, uint8_t* sf_out, int use_pdl,
                hq_stream_t s, const int32_t* token_nums = nullptr, int E = 0,
                int64_t rows_per_expert = 0) {
  if (mode != HQ_MXFP8 && mode != HQ_MXFP4 && mode != HQ_NVFP4 && mode != HQ_MXFP8_E5M2)
    return HQ_ERR_INVALID;
  const int64_t gs = mode == HQ_NVFP4 ? 16 : 32;
  if (m < 0 || k <= 0 || k % (4 * gs) != 0) return HQ_ERR_INVALID;
  if (mode != HQ_NVFP4 && global_scale) return HQ_ERR_UNSUPPORTED;
  if (m == 0) return HQ_OK;
  if (!x || !q_out || !sf_out) return HQ_ERR_INVALID;
  if (!aligned16(x) || !aligned16(q_out) || !aligned16(sf_out)) return HQ_ERR_INVALID;
  if (global_scale && (reinterpret_cast<uintptr_t>(global_scale) & 3u)) return HQ_ERR_INVALID;
  QuantParams p{};
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
  if (token_nums) {
    p.token_nums = token_nums;
    p.rows_per_expert = rows_per_expert;
    p.E = E;
  } else {
    p.rows_per_expert = m;
    p.E = 1;
  }
  p.status = status_word_ptr();
  if (!p.status) return HQ_ERR_CUDA;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  return f16 ? dispatch_f16(mode, p, st, use_pdl != 0) : dispatch(mode, false, p, st, use_pdl != 0);
}

}  // namespace
}  // namespace hq

extern "C" {

int hq_quant(const hq_bf16* x, int64_t m, int64_t k, hq_mode mode, int use_swizzle,
             const float* global_scale, void* q_out, uint8_t* sf_out, int use_pdl,
             hq_stream_t s) {
  return hq::quant_entry(x, false, m, k, mode, use_swizzle, global_scale, q_out, sf_out, use_pdl, s);
}

int hq_quant_f16(const uint16_t* x, int64_t m, int64_t k, hq_mode mode, int use_swizzle,
                 const float* global_scale, void* q_out, uint8_t* sf_out, int use_pdl,
                 hq_stream_t s) {
  return hq::quant_entry(x, true, m, k, mode, use_swizzle, global_scale, q_out, sf_out, use_pdl, s);
}

int hq_quant_masked(const hq_bf16* x, int E, int64_t max_m, const int32_t* masked_m, int64_t k,
                    hq_mode mode, int use_swizzle, const float* global_scale, void* q_out,
                    uint8_t* sf_out, int use_pdl, hq_stream_t s) {
  if (E <= 0 || E > hq::kMaxCountExperts || max_m <= 0 || max_m % 128 != 0) return HQ_ERR_INVALID;
  if (!masked_m || (reinterpret_cast<uintptr_t>(masked_m) & 3u)) return HQ_ERR_INVALID;
  if (max_m > (1ll << 31) / E) return HQ_ERR_INVALID;
  return hq::quant_entry(x, false, static_cast<int64_t>(E) * max_m, k, mode, use_swizzle, global_scale, q_out,
                         sf_out, use_pdl, s, masked_m, E, max_m);
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
    if (E <= 0 || E > hq::kMaxCountExperts || rows_per_expert <= 0 ||
        static_cast<int64_t>(E) * rows_per_expert != rows)
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
