// hq_gemm_bs.cu -- block-scaled GEMMs (MXFP8, MXFP4, NVFP4) on 5th-generation
// tensor cores: out = alpha_g * (A . B_g^T) + bias_g, BF16 output, and the
// epilogues built on the same main loop.
//
// Two persistent kernels serve the dense, grouped-contiguous (padded_offsets),
// per-row expert-id and grouped-masked problems (HALOps "GEMM" API
// dense_gemm / group_contiguous_gemm / group_masked_gemm; cuDNN frontend
// "Grouped GEMM + dGLU (SM100)" Step 1):
//   bs_gemm_kernel      one CTA per SM, tiles of 128 rows x BN (128 or 256)
//                       columns, one or two TMEM accumulators; also carries
//                       the dSwiGLU / dGeGLU epilogues (block-scaled dGLU
//                       backward) and the fused up-proj SwiGLU + requant
//                       epilogue, and discrete (per-expert pointer) weights;
//   bs_gemm_2sm_kernel  two-CTA clusters, cta_group::2 MMAs of M = 256 over
//                       tiles of 256 x 256 (or 256 x 384) columns, for the
//                       dense, contiguous, masked and fused up-proj problems.
// Warp roles in both (448 threads):
//   warp 0       TMA producer: A and B tiles (128-byte swizzled, K-major) and
//                bulk copies of the 512-byte SfAtom scale atoms into a ring of
//                shared-memory stages, completion tracked by mbarriers;
//   warp 1       MMA issuer (the even CTA's in a pair); owns TMEM;
//   warps 2..9   epilogue: TMEM -> registers (tcgen05.ld), alpha / bias,
//                BF16 round-to-nearest-even (or the fused epilogue's math),
//                coalesced stores; rows outside the valid range never written;
//   warps 10..13 scale staging: the stage's scale atoms shared -> TMEM
//                (tcgen05.st into each TMEM lane quarter), then an arrival
//                on the barrier the MMA issuer waits on for that stage.
// Every role decodes the same tile sequence (n fastest inside each row block)
// from device-resident group information (padded_offsets, masked_m or the
// per-row segment list), validated on the device; every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "hq_internal.h"
#include "hq_ptx.cuh"
#include "hq_sched.cuh"

namespace hq {
namespace {

// How scale atoms reach TMEM (the SFP parameter of the single-SM kernel):
//   0  the MMA thread issues tcgen05.cp (32x128b.warpx4) before its MMAs:
//      no scale warps, so the CTA's ten warps may hold 168 registers each
//      (the tensor pipe spends time on the copies);
//   1  a dedicated warp issues the tcgen05.cp and signals the MMA thread;
//   2  four scale warps (one per TMEM lane quarter) read the atoms from shared
//      memory and write them with tcgen05.st, replicated into every quarter
//      exactly as the warpx4 copy would, then signal the MMA thread (the
//      default; the 2-SM kernel always stages this way).
constexpr int kSfPath = 2;
constexpr int sf_warps(int path) { return path == 1 ? 1 : (path == 2 ? 4 : 0); }
constexpr int kEpiWarps = 8;             // warps 2..9: two per TMEM lane quarter
constexpr int kSfWarp0 = 2 + kEpiWarps;  // first scale-staging warp
constexpr int threads_for(int path) { return 32 * (kSfWarp0 + sf_warps(path)); }
constexpr int kThreads = threads_for(kSfPath);
constexpr int kBKBytes = 128;   // bytes of K per stage and row (one 128B swizzle span)
constexpr int kMmaKBytes = 32;  // bytes of K consumed by one MMA
constexpr int kSmemLimit = 232448;

struct GemmParams {
  const uint8_t* sfa;
  const uint8_t* sfb;
  const float* alpha;        // [groups] or null
  const uint16_t* bias;      // [groups, n] or null
  uint16_t* out;             // [a_rows, n]
  GroupSched gs;             // group layout (rows, offsets or masks, status word)
  int64_t n, k;
  int64_t S;                 // scale columns = k / group
  int64_t sfb_group_bytes;   // ceil(n/128)*128*S
  uint64_t wait_limit_ns;
  // bits ORed into every MMA instruction descriptor: the E5M2 operand type of
  // kind::mxf8f6f4 (A and B format fields), 0 for the other modes
  uint32_t idesc_ab;
  // D_row / D_col element type of the dGLU epilogues (kDBf16 .. kDE5M2)
  int d_type;
  // dGLU epilogues: D_row leaves through the warp's buffer and a TMA store
  // (1: BF16 D_row, 2: FP8 D_row with SFD_row), 0: straight from registers
  int d_tma;
  // test aid (hq_set_fault_injection): cluster 0's producer withholds the
  // arrival on the "full" barrier of this stage (count of stages it issued);
  // -1 = never
  int64_t inject_skip;
  // dGLU epilogues only (cuDNN "Grouped GEMM + dGLU (SM100)", block-scaled
  // contract): out is not used; D_row = dGLU(alpha_g^2 acc, C) instead
  const uint16_t* c;         // [a_rows, 2n] BF16 forward intermediate
  const float* beta;         // [groups] (dSwiGLU)
  const float* prob;         // [a_rows]
  float* dprob;              // [a_rows], accumulated
  float* dbias_ws;           // [groups, 2n] float32 partial sums, or null
  uint8_t* d_row;            // [a_rows, 2n]: BF16, or E4M3 when sfd_row is set
  uint8_t* sfd_row;          // SfAtom UE8M0 scales of D_row, [ceil(a_rows/128)*128, 2n/32], or null
  const float* norm_const;   // FP8 D_row norm_const (device [1]) or null (= 1)
  uint8_t* d_col;            // [a_rows, 2n] E4M3 column-quantised D, or null
  uint8_t* sfd_col;          // SfAtom UE8M0 of [2n rows, ceil(a_rows/128)*4 cols], or null
  int64_t sfd_col_s;         // scale columns of sfd_col (ceil(a_rows / 128) * 4)
  float* amax;               // [groups, 2]: max |D| over gate / input columns, or null
  // fused up-proj epilogue only: n is H, B holds 2H rows per group (gate rows
  // [0, H), up rows [H, 2H)); out is not used, y = up * silu(gate) is
  // quantised instead
  uint8_t* q;                // [a_rows, H] E4M3 (MXFP8) or [a_rows, H / 2] packed E2M1 (NVFP4)
  uint8_t* sfq;              // SfAtom scales of q, sfq_cols columns
  int64_t sfq_cols;          // MXFP8: ceil(H / 512) * 16; NVFP4: H / 16
  int q_mode;                // HQ_MXFP8 or HQ_NVFP4
  const float* q_gscale;     // NVFP4 global scale (device [1]) or null (= 1)
  // discrete weights (one pointer per expert): B of group g is loaded through
  // b_maps[g], built on the device from b_ptrs[g] before the GEMM; its scales
  // start at sfb_ptrs[g]; w_ok[g] == 0 marks an expert whose pointers failed
  // the device checks (its tiles load nothing from B and write nothing)
  const int64_t* b_ptrs;     // [groups], or null: B stacked as [groups, n, k]
  const int64_t* sfb_ptrs;   // [groups]
  CUtensorMap* b_maps;       // [groups] in the caller's workspace
  int32_t* w_ok;             // [groups] in the caller's workspace
};

enum Epi : int { kEpiGemm = 0, kEpiDSwiGLU = 1, kEpiDGeGLU = 2, kEpiSwiGLUQ = 3 };
enum DType : int { kDBf16 = HQ_D_BF16, kDF32 = HQ_D_F32, kDE4M3 = HQ_D_E4M3, kDE5M2 = HQ_D_E5M2 };

// The kernel instantiation a mode runs on: E5M2 operands take the MXFP8
// kernels (same bytes per element, scales and MMA kind; the operand type is
// in the instruction descriptor bits that base_params sets).
inline hq_mode kernel_mode(hq_mode mode) { return mode == HQ_MXFP8_E5M2 ? HQ_MXFP8 : mode; }
inline bool valid_mode(hq_mode mode) {
  return mode == HQ_MXFP8 || mode == HQ_MXFP4 || mode == HQ_NVFP4 || mode == HQ_MXFP8_E5M2;
}

// TABLE: entries of the per-CTA group table (0 for the dense GEMM, which
// needs none and spends the shared memory on a deeper pipeline instead).
template <int MODE, int BN, int STAGES, int ACC, int TABLE, int OUTB = 1024>
struct Cfg {
  static constexpr int GS = MODE == HQ_NVFP4 ? 16 : 32;
  static constexpr int EPB = MODE == HQ_MXFP8 ? 1 : 2;            // elements per byte
  static constexpr int BK = kBKBytes * EPB;                       // elements per stage
  static constexpr int ATOMS = BK / GS / 4;                       // k-atoms per stage
  static constexpr int RB = BN / 128;                             // 128-row blocks of B
  static constexpr int A_BYTES = kBM * kBKBytes;
  static constexpr int B_BYTES = BN * kBKBytes;
  static constexpr int SFA_BYTES = ATOMS * 512;
  static constexpr int SFB_BYTES = RB * ATOMS * 512;
  static constexpr int SFA_COLS = (ATOMS * 4 + 7) / 8 * 8;         // padded to 8 columns
  static constexpr int SFB_COLS = RB * ATOMS * 4;
  static constexpr int SF_STAGE_COLS = (SFA_COLS + SFB_COLS + 15) / 16 * 16;
  static constexpr int SF_BASE_COL = ACC * BN;
  static constexpr int TMEM_USED = ACC * BN + STAGES * SF_STAGE_COLS;
  static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64
                                 : TMEM_USED <= 128 ? 128 : TMEM_USED <= 256 ? 256 : 512;
  static_assert(TMEM_USED <= 512, "TMEM budget");
  // shared-memory layout (offsets from a 1024-aligned base)
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  // OUTB bytes per epilogue warp: 1 KB of output staging, 4 KB for the dGLU's
  // C / D_row segments (1024-aligned for the TMA swizzle)
  static constexpr int OFF_STAGE_OUT = (OFF_SFB + STAGES * SFB_BYTES + 1023) / 1024 * 1024;
  static constexpr int OFF_TABLE = OFF_STAGE_OUT + kEpiWarps * OUTB;  // 2 x TABLE int32
  static constexpr int OFF_BAR = OFF_TABLE + 2 * TABLE * 4 + 8;
  static constexpr int NUM_BARS = 3 * STAGES + 2 * ACC + 2 + kEpiWarps;  // + one C barrier per epilogue warp
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= kSmemLimit, "shared memory budget");
  static_assert(OFF_BAR % 8 == 0, "barrier alignment");
  // instruction descriptor (block-scaled kinds): A/B K-major, M=128, N=BN
  static constexpr uint32_t IDESC_BASE =
      (MODE == HQ_MXFP8 ? ((0u << 7) | (0u << 10) | (1u << 23))   // E4M3 x E4M3, UE8M0
       : MODE == HQ_MXFP4 ? ((1u << 7) | (1u << 10) | (1u << 23))  // E2M1 x E2M1, UE8M0
                          : ((1u << 7) | (1u << 10) | (0u << 23)))  // E2M1 x E2M1, UE4M3
      | (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(kBM >> 4) << 24);
};

// ---------------------------------------------------------------------------
// Epilogue of one accumulator tile for one warp: TMEM lane quarter q holds
// rows row0 + 32 q + lane; the warp owns tile columns [cw, cw + BN / 2).
//   out[row, n0 + j] = bf16_rne(alpha * acc[row, j] + bias[n0 + j])
// DRAIN: the warp first moves its whole share out of TMEM (as BF16 pairs in
// registers) and calls release() before any global store, so the MMAs of the
// next tile can start while the stores drain; otherwise release() follows the
// stores.  Stores go through the warp's 1 KB staging buffer, 16 columns at a
// time, so that two lanes write each row's 32 contiguous bytes.
// ---------------------------------------------------------------------------
struct EpiArgs {
  uint32_t acc_t;        // TMEM address of (lane quarter, tile column 0)
  int cw;                // first tile column of this warp
  int64_t n0, n;         // tile's first output column, output width
  float alpha;
  const uint16_t* bias;  // bias row of the group (column 0) or null
  uint16_t* out;         // output row of lane 0 of this quarter (column 0)
  int rows_here;         // valid rows of this quarter (may be <= 0 or > 32) ...
  int rows_lo;           // ... from this row of the quarter on (may be <= 0)
  uint32_t stage_s;      // this warp's staging buffer (shared address)
  int lane;
  int64_t row_abs;       // absolute row of lane 0 of this quarter (debug bounds checks)
  int64_t rows_total;    // rows of out
  uint32_t* status;
};

__device__ __forceinline__ void epi_convert16(const EpiArgs& e, int64_t col0, const uint32_t (&r)[16],
                                              uint32_t* packed) {
  if (e.bias) {
    const uint4* bp = reinterpret_cast<const uint4*>(e.bias + col0);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4 v = __ldg(bp + i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float v0, v1;
        mul_f32x2(v0, v1, __uint_as_float(r[8 * i + 2 * j]), __uint_as_float(r[8 * i + 2 * j + 1]),
                  e.alpha);
        add_f32x2(v0, v1, v0, v1, __uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u));
        __nv_bfloat162 b2 = __floats2bfloat162_rn(v0, v1);
        packed[4 * i + j] = *reinterpret_cast<uint32_t*>(&b2);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float v0, v1;
      mul_f32x2(v0, v1, __uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), e.alpha);
      __nv_bfloat162 b2 = __floats2bfloat162_rn(v0, v1);
      packed[i] = *reinterpret_cast<uint32_t*>(&b2);
    }
  }
}

__device__ __forceinline__ void epi_store16(const EpiArgs& e, int64_t col0, const uint32_t* packed) {
  const int lane = e.lane;
  // stage: row = lane, two 16-byte units, unit index xor-swizzled by row bit 2
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const uint32_t off = lane * 32 + ((u ^ ((lane >> 2) & 1)) * 16);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(e.stage_s + off),
                 "r"(packed[4 * u]), "r"(packed[4 * u + 1]), "r"(packed[4 * u + 2]),
                 "r"(packed[4 * u + 3])
                 : "memory");
  }
  __syncwarp();
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int rr = it * 16 + (lane >> 1);
    const int u = lane & 1;
    const uint32_t off = rr * 32 + ((u ^ ((rr >> 2) & 1)) * 16);
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(e.stage_s + off)
                 : "memory");
    if (rr >= e.rows_lo && rr < e.rows_here &&
        in_bounds(e.row_abs + rr < e.rows_total && col0 + u * 8 + 8 <= e.n, e.status))
      *reinterpret_cast<uint4*>(e.out + rr * e.n + col0 + u * 8) = v;
  }
  __syncwarp();
}

template <int BN, bool DRAIN, typename Release>
__device__ __forceinline__ void epilogue_tile(const EpiArgs& e, Release release) {
  constexpr int kPieces = BN / 2 / 16;  // 16-column pieces per warp
  if (DRAIN) {
    // piece s + 1 is read from TMEM while piece s is converted
    uint32_t packed[kPieces * 8];
    uint32_t r[2][16];
    tmem_ld_32x32b_x16(e.acc_t + e.cw, r[0]);
    tmem_ld_wait(r[0]);
#pragma unroll
    for (int s = 0; s < kPieces; ++s) {
      if (s + 1 < kPieces) tmem_ld_32x32b_x16(e.acc_t + e.cw + (s + 1) * 16, r[(s + 1) & 1]);
      const int64_t col0 = e.n0 + e.cw + s * 16;
      if (col0 < e.n) epi_convert16(e, col0, r[s & 1], packed + 8 * s);
      if (s + 1 < kPieces) tmem_ld_wait(r[(s + 1) & 1]);
    }
    tc_fence_before();
    __syncwarp();
    release();
#pragma unroll
    for (int s = 0; s < kPieces; ++s) {
      const int64_t col0 = e.n0 + e.cw + s * 16;
      if (col0 < e.n) epi_store16(e, col0, packed + 8 * s);
    }
  } else {
    for (int s = 0; s < kPieces; ++s) {
      uint32_t r[16], packed[8];
      tmem_ld_32x32b_x16(e.acc_t + e.cw + s * 16, r);
      tmem_ld_wait(r);
      const int64_t col0 = e.n0 + e.cw + s * 16;
      if (col0 >= e.n) continue;
      epi_convert16(e, col0, r, packed);
      epi_store16(e, col0, packed);
    }
    tc_fence_before();
    __syncwarp();
    release();
  }
}

// Wide pair tile (384 columns): the warp drains tile columns [cw, cw + 128)
// of the first 256 and its 64 columns [256 + cw2, 256 + cw2 + 64) of the
// last 128 into registers (converted to BF16 while the next piece is read),
// releases the accumulator, then stores both parts.
template <typename Release>
__device__ __forceinline__ void epilogue_tile_wide(const EpiArgs& e, int cw2, Release release) {
  constexpr int kPieces = 12;  // 8 of the first 256 columns, 4 of the last 128
  auto piece_col = [&](int s) { return s < 8 ? e.cw + s * 16 : 256 + cw2 + (s - 8) * 16; };
  uint32_t packed[kPieces * 8];
#pragma unroll
  for (int s = 0; s < kPieces; ++s) {
    uint32_t r[16];
    tmem_ld_32x32b_x16(e.acc_t + piece_col(s), r);
    tmem_ld_wait(r);
    const int64_t col0 = e.n0 + piece_col(s);
    if (col0 < e.n) epi_convert16(e, col0, r, packed + 8 * s);
  }
  tc_fence_before();
  __syncwarp();
  release();
#pragma unroll
  for (int s = 0; s < kPieces; ++s) {
    const int64_t col0 = e.n0 + piece_col(s);
    if (col0 < e.n) epi_store16(e, col0, packed + 8 * s);
  }
}

// ---------------------------------------------------------------------------
// dGLU epilogue of one 32-column chunk (compact columns [j0, j0 + 32)) for the
// calling thread's row: R = a2 * acc, C's 32 gate and 32 input values of the
// row, D_row written at the same 64 columns (BF16, or E4M3 with two UE8M0
// scale bytes), the row's dprob partial added, and, when requested, the
// warp's column sums of D added to the dbias workspace.
//   dSwiGLU: X = beta C, s = sigmoid(gate)
//     dgate = R prob input s (1 + gate (1 - s)),  dinput = R prob gate s,
//     dprob += R gate s input
//   dGeGLU:  gate_c = min(gate, 7), up_c = clamp(up, -7, 7), s = sigmoid(1.702 gate_c)
//     dgate = R prob (up_c + 1) s (1 + 1.702 gate_c (1 - s)) [gate <= 7]
//     dup   = R prob gate_c s [-7 <= up <= 7],  dprob += R gate_c s (up_c + 1)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float dglu_bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float dglu_bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int EPI>
__device__ __forceinline__ void dglu_math(const uint32_t (&r)[32], const uint4 (&cv)[8], float a2, float beta,
                                          float prob, float (&dg)[32], float (&di)[32], float& dprob) {
  float dp0 = 0.0f, dp1 = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t gw = reinterpret_cast<const uint32_t*>(cv)[i];
    const uint32_t iw = reinterpret_cast<const uint32_t*>(cv)[16 + i];
    float R0, R1, rp0, rp1;
    mul_f32x2(R0, R1, __uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), a2);
    mul_f32x2(rp0, rp1, R0, R1, prob);
    if (EPI == kEpiDSwiGLU) {
      float g0, g1, x0, x1;
      mul_f32x2(g0, g1, dglu_bf16_lo(gw), dglu_bf16_hi(gw), beta);
      mul_f32x2(x0, x1, dglu_bf16_lo(iw), dglu_bf16_hi(iw), beta);
      float s0, s1;
      sigmoid_x2(g0, g1, s0, s1);  // sigmoid(gate)
      float om0, om1, t0, t1, gs0, gs1, u0, u1, q0, q1;
      fma_f32x2(om0, om1, s0, s1, -1.0f, -1.0f, 1.0f, 1.0f);
      fma_f32x2(t0, t1, g0, g1, om0, om1, 1.0f, 1.0f);
      mul2_f32x2(gs0, gs1, g0, g1, s0, s1);
      mul2_f32x2(u0, u1, rp0, rp1, x0, x1);
      mul2_f32x2(u0, u1, u0, u1, s0, s1);
      mul2_f32x2(dg[2 * i], dg[2 * i + 1], u0, u1, t0, t1);
      mul2_f32x2(di[2 * i], di[2 * i + 1], rp0, rp1, gs0, gs1);
      mul2_f32x2(q0, q1, R0, R1, gs0, gs1);
      fma_f32x2(dp0, dp1, q0, q1, x0, x1, dp0, dp1);
    } else {
      const float g0 = dglu_bf16_lo(gw), g1 = dglu_bf16_hi(gw);
      const float x0 = dglu_bf16_lo(iw), x1 = dglu_bf16_hi(iw);
      const float gc0 = fminf(g0, 7.0f), gc1 = fminf(g1, 7.0f);
      const float uc0 = fminf(fmaxf(x0, -7.0f), 7.0f), uc1 = fminf(fmaxf(x1, -7.0f), 7.0f);
      float kg0, kg1;
      mul_f32x2(kg0, kg1, gc0, gc1, 1.702f);
      float s0, s1;
      sigmoid_x2(kg0, kg1, s0, s1);
      float om0, om1, t0, t1, up0, up1, gs0, gs1, w0, w1, a0, a1, b0, b1, q0, q1;
      fma_f32x2(om0, om1, s0, s1, -1.0f, -1.0f, 1.0f, 1.0f);
      fma_f32x2(t0, t1, kg0, kg1, om0, om1, 1.0f, 1.0f);
      add_f32x2(up0, up1, uc0, uc1, 1.0f, 1.0f);
      mul2_f32x2(gs0, gs1, gc0, gc1, s0, s1);
      mul2_f32x2(w0, w1, rp0, rp1, up0, up1);
      mul2_f32x2(w0, w1, w0, w1, s0, s1);
      mul2_f32x2(a0, a1, w0, w1, t0, t1);
      mul2_f32x2(b0, b1, rp0, rp1, gs0, gs1);
      dg[2 * i] = g0 <= 7.0f ? a0 : 0.0f;
      dg[2 * i + 1] = g1 <= 7.0f ? a1 : 0.0f;
      di[2 * i] = (x0 >= -7.0f && x0 <= 7.0f) ? b0 : 0.0f;
      di[2 * i + 1] = (x1 >= -7.0f && x1 <= 7.0f) ? b1 : 0.0f;
      mul2_f32x2(q0, q1, R0, R1, gs0, gs1);
      fma_f32x2(dp0, dp1, q0, q1, up0, up1, dp0, dp1);
    }
  }
  dprob = dp0 + dp1;
}

// The row's D_row segment (and SFD_row bytes) and its dprob partial.  D_row
// goes to the warp's buffer at dbuf (sent by the caller with one TMA store:
// BF16 in the 128-byte swizzle, FP8 as plain 64-byte rows) when dbuf != 0,
// else straight to global memory.
__device__ __forceinline__ void dglu_write_row(const GemmParams& p, const float (&dg)[32],
                                               const float (&di)[32], bool row_ok, int64_t row,
                                               int64_t j0, float norm, float dprob, uint32_t dbuf,
                                               int lane) {
  const int64_t two_n = 2 * p.n;
  // FP8 D (Step 3): E4M3 or E5M2 codes, the scale rule's range to match
  const bool e5 = p.d_type == kDE5M2;
  const float rcp_max = e5 ? 1.0f / 57344.0f : 1.0f / 448.0f;
  auto cvt8x2 = [&](float hi, float lo) -> uint32_t { return e5 ? cvt_e5m2x2(hi, lo) : cvt_e4m3x2(hi, lo); };
  if (row_ok) {
    if (p.d_type == kDF32) {
      float4* dst = reinterpret_cast<float4*>(p.d_row + (row * two_n + 2 * j0) * 4);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float* v = u < 8 ? dg + 4 * u : di + 4 * (u - 8);
        dst[u] = make_float4(v[0], v[1], v[2], v[3]);
      }
    } else if (!p.sfd_row) {
      uint4* dst = reinterpret_cast<uint4*>(p.d_row + (row * two_n + 2 * j0) * 2);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float* v = u < 4 ? dg + 8 * u : di + 8 * (u - 4);
        __nv_bfloat162 b0 = __floats2bfloat162_rn(v[0], v[1]), b1 = __floats2bfloat162_rn(v[2], v[3]),
                       b2 = __floats2bfloat162_rn(v[4], v[5]), b3 = __floats2bfloat162_rn(v[6], v[7]);
        const uint4 w4 = make_uint4(*reinterpret_cast<uint32_t*>(&b0), *reinterpret_cast<uint32_t*>(&b1),
                                    *reinterpret_cast<uint32_t*>(&b2), *reinterpret_cast<uint32_t*>(&b3));
        if (dbuf) {
          // 16-byte unit u of row `lane` at unit u ^ (lane & 7): the TMA 128-byte swizzle
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                           dbuf + static_cast<uint32_t>(lane) * 128u + ((static_cast<uint32_t>(u) ^ (lane & 7)) << 4)),
                       "r"(w4.x), "r"(w4.y), "r"(w4.z), "r"(w4.w)
                       : "memory");
        } else {
          dst[u] = w4;
        }
      }
    } else {
      // Step 3: per 32 D_row values, s = (norm * amax) / 448 (E5M2: 57344)
      // rounded up to a power of two, codes E4M3 / E5M2 ((D * norm) * 2^(127 - byte))
      uint32_t bytes2 = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float* v = h == 0 ? dg : di;
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
        const uint32_t byte = ue8m0_ceil(__fmul_rn(__fmul_rn(norm, amax), rcp_max));
        const float mult = pow2_neg_unbiased(byte);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          // (D * norm) * mult, each product rounded, two values per instruction
          float y[4];
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            mul_f32x2(y[u], y[u + 1], v[4 * i + u], v[4 * i + u + 1], norm);
            mul_f32x2(y[u], y[u + 1], y[u], y[u + 1], mult);
          }
          w[i] = cvt8x2(y[1], y[0]) | (cvt8x2(y[3], y[2]) << 16);
        }
        if (dbuf) {
          // plain 64-byte rows: this half's 32 codes are units 2 h and 2 h + 1 of row `lane`
          const uint32_t a0 = dbuf + static_cast<uint32_t>(lane) * 64u + 32u * h;
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a0), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                       "r"(w[3])
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a0 + 16u), "r"(w[4]), "r"(w[5]),
                       "r"(w[6]), "r"(w[7])
                       : "memory");
        } else {
          uint4* dst = reinterpret_cast<uint4*>(p.d_row + row * two_n + 2 * j0 + 32 * h);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
        bytes2 |= byte << (8 * h);
      }
      // the chunk's two scale columns s, s + 1 (s even) are adjacent in the atom row
      const int64_t S = two_n / 32, s = 2 * j0 / 32;
      const int64_t off = ((row >> 7) * (S >> 2) + (s >> 2)) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (s & 3);
      *reinterpret_cast<uint16_t*>(p.sfd_row + off) = static_cast<uint16_t>(bytes2);
    }
    atomicAdd(p.dprob + row, dprob);
  }
}

// The chunk's warp-collective parts: the per-group amax, D_col with its
// column scales, and the dbias column sums.
__device__ __forceinline__ void dglu_tail(const GemmParams& p, float (&dg)[32], float (&di)[32], bool row_ok,
                                          int64_t row, int64_t j0, int g, float norm, int lane) {
  const int64_t two_n = 2 * p.n;
  const bool e5 = p.d_type == kDE5M2;
  const float rcp_max = e5 ? 1.0f / 57344.0f : 1.0f / 448.0f;
  auto cvt8x2 = [&](float hi, float lo) -> uint32_t { return e5 ? cvt_e5m2x2(hi, lo) : cvt_e4m3x2(hi, lo); };
  if (p.amax) {
    // per-group max |D| over the gate and the input columns: a max all-reduce
    // over the warp, then one integer atomic max per value (|D| >= 0, so the
    // float order is the order of the bit patterns)
    float mg = 0.0f, mi = 0.0f;
    if (row_ok) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        mg = fmaxf(mg, fabsf(dg[i]));
        mi = fmaxf(mi, fabsf(di[i]));
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      mg = fmaxf(mg, __shfl_xor_sync(0xFFFFFFFFu, mg, o));
      mi = fmaxf(mi, __shfl_xor_sync(0xFFFFFFFFu, mi, o));
    }
    if (lane == 0) {
      atomicMax(reinterpret_cast<int*>(p.amax + 2 * g), __float_as_int(mg));
      atomicMax(reinterpret_cast<int*>(p.amax + 2 * g + 1), __float_as_int(mi));
    }
  }
  if (p.d_col) {
    // Step 3 along M: each D column's scale over the warp's 32 rows (one
    // 32-row block), from a max all-reduce across the lanes; lane l keeps the
    // bytes of gate column l and input column l
    const int64_t blk = (row - lane) >> 5;
    uint32_t my_byte[2] = {0u, 0u};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float* v = h == 0 ? dg : di;
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float y[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float x = row_ok ? v[2 * i + u] : 0.0f;
          float mx = fabsf(x);
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
          const uint32_t byte = ue8m0_ceil(__fmul_rn(__fmul_rn(norm, mx), rcp_max));
          if (lane == 2 * i + u) my_byte[h] = byte;
          y[u] = __fmul_rn(__fmul_rn(x, norm), pow2_neg_unbiased(byte));
        }
        const uint32_t pair = cvt8x2(y[1], y[0]);
        if ((i & 1) == 0) w[i >> 1] = pair;
        else w[i >> 1] |= pair << 16;
      }
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(p.d_col + row * two_n + 2 * j0 + 32 * h);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    }
    const int64_t S = p.sfd_col_s;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t col = 2 * j0 + 32 * h + lane;
      const int64_t off = ((col >> 7) * (S >> 2) + (blk >> 2)) * 512 + (col & 31) * 16 +
                          ((col >> 5) & 3) * 4 + (blk & 3);
      p.sfd_col[off] = static_cast<uint8_t>(my_byte[h]);
    }
  }
  if (p.dbias_ws) {
    // column sums over the warp's 32 rows (butterfly reduce-scatter): lane l
    // ends with the sums of gate column l and input column l
    if (!row_ok) {
#pragma unroll
      for (int i = 0; i < 32; ++i) { dg[i] = 0.0f; di[i] = 0.0f; }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < o; ++i) {
        const float sg = upper ? dg[i] : dg[i + o];
        const float si = upper ? di[i] : di[i + o];
        const float kg = upper ? dg[i + o] : dg[i];
        const float ki = upper ? di[i + o] : di[i];
        dg[i] = kg + __shfl_xor_sync(0xFFFFFFFFu, sg, o);
        di[i] = ki + __shfl_xor_sync(0xFFFFFFFFu, si, o);
      }
    }
    float* ws = p.dbias_ws + static_cast<int64_t>(g) * two_n + 2 * j0;
    atomicAdd(ws + lane, dg[0]);
    atomicAdd(ws + 32 + lane, di[0]);
  }
}

// ---------------------------------------------------------------------------
// Fused up-proj epilogue: SwiGLU of the GEMM's float32 result followed by the
// group-wise requantisation (cuDNN frontend "Grouped GEMM + dGLU (SM100)",
// forward SwiGLU and Step 3; HALOps group_wise_quant encodings).  The tile's
// accumulator holds 128 gate columns (TMEM columns [0, 128)) and the matching
// 128 up columns ([128, 256)) of one expert; the calling warp owns compact
// columns [cw, cw + 64) of its lane quarter, one row per thread:
//   gate = alpha acc_g, up = alpha acc_u, y = up * (gate / (1 + exp(-gate)))
// swiglu_drain forms y while reading TMEM; swiglu_store (after TMEM is
// released) encodes each scale group of y and writes the codes and the scale
// bytes:
//   MXFP8  per 32: UE8M0 = ceil(log2(amax / 448)) + 127, q = E4M3(y 2^(127 - UE8M0))
//   NVFP4  per 16: UE4M3 = E4M3((g amax) / 6), q = E2M1(y (g / value(UE4M3)))
// ---------------------------------------------------------------------------
__device__ __forceinline__ void swiglu_drain(uint32_t tcol, float alpha, float (&y)[64]) {
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    uint32_t rg[16], ru[16];
    tmem_ld_32x32b_x16(tcol + 16 * s, rg);
    tmem_ld_32x32b_x16(tcol + 128 + 16 * s, ru);
    tmem_ld_wait(rg);
    tmem_ld_wait(ru);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      float g0, g1, u0, u1;
      mul_f32x2(g0, g1, __uint_as_float(rg[i]), __uint_as_float(rg[i + 1]), alpha);
      mul_f32x2(u0, u1, __uint_as_float(ru[i]), __uint_as_float(ru[i + 1]), alpha);
      const float t0 = __fmul_rn(g0, rcp_approx(__fadd_rn(1.0f, __expf(-g0))));
      const float t1 = __fmul_rn(g1, rcp_approx(__fadd_rn(1.0f, __expf(-g1))));
      mul2_f32x2(y[16 * s + i], y[16 * s + i + 1], u0, u1, t0, t1);
    }
  }
}

__device__ __forceinline__ int64_t sfatom_offset(int64_t r, int64_t s, int64_t S) {
  return ((r >> 7) * (S >> 2) + (s >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (s & 3);
}

__device__ __forceinline__ void swiglu_store(const GemmParams& p, const float (&y)[64], int64_t row,
                                             int64_t j0, float gq) {
  const int64_t H = p.n;
  if (!in_bounds(row < p.gs.a_rows && j0 + 64 <= H, p.gs.status)) return;
  if (p.q_mode == HQ_MXFP8) {
    uint32_t bytes2 = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float* v = y + 32 * h;
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
      const uint32_t byte = ue8m0_ceil(__fmul_rn(amax, 1.0f / 448.0f));
      const float mult = pow2_neg_unbiased(byte);
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t lo = cvt_e4m3x2(__fmul_rn(v[4 * i + 1], mult), __fmul_rn(v[4 * i], mult));
        const uint32_t hi = cvt_e4m3x2(__fmul_rn(v[4 * i + 3], mult), __fmul_rn(v[4 * i + 2], mult));
        w[i] = lo | (hi << 16);
      }
      uint4* dst = reinterpret_cast<uint4*>(p.q + row * H + j0 + 32 * h);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      bytes2 |= byte << (8 * h);
    }
    // scale columns j0 / 32 (even) and the next one are adjacent in the atom row
    *reinterpret_cast<uint16_t*>(p.sfq + sfatom_offset(row, j0 / 32, p.sfq_cols)) =
        static_cast<uint16_t>(bytes2);
  } else {
    uint32_t bytes4 = 0;
    uint32_t w[8];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float* v = y + 16 * h;
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
      const uint32_t byte = cvt_e4m3x2(0.0f, __fmul_rn(__fmul_rn(gq, amax), 1.0f / 6.0f)) & 0x7Fu;
      const float sd = ue4m3_value(byte);
      const float r = sd == 0.0f ? 0.0f : __fdiv_rn(gq, sd);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        uint32_t x = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          x |= cvt_e2m1x2(__fmul_rn(v[8 * i + 2 * j + 1], r), __fmul_rn(v[8 * i + 2 * j], r)) << (8 * j);
        w[2 * h + i] = x;
      }
      bytes4 |= byte << (8 * h);
    }
    uint4* dst = reinterpret_cast<uint4*>(p.q + (row * H + j0) / 2);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    // scale columns j0 / 16 .. + 3 form one 32-bit word of the atom row
    *reinterpret_cast<uint32_t*>(p.sfq + sfatom_offset(row, j0 / 16, p.sfq_cols)) = bytes4;
  }
}

// tmC / tmD: the dGLU epilogues' C and D_row segment maps (other epilogues
// get unused placeholders)
template <int MODE, int BN, int STAGES, int ACC, int TABLE, int EPI = kEpiGemm, int SFP = kSfPath>
__global__ void __launch_bounds__(threads_for(SFP), 1)
    bs_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                   const GemmParams p) {
  constexpr bool kDglu = EPI == kEpiDSwiGLU || EPI == kEpiDGeGLU;
  using C = Cfg<MODE, BN, STAGES, ACC, TABLE, kDglu ? 4096 : 1024>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int32_t* tab0 = reinterpret_cast<int32_t*>(smem + C::OFF_TABLE);
  int32_t* tab1 = tab0 + TABLE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + ACC + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * ACC);
  const uint32_t drain_sf_bar = drain_bar + 8u;
  auto sfready_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 2 * ACC + 2 + s); };
  const uint32_t cbar0 = bar0 + 8u * (3 * STAGES + 2 * ACC + 2);  // dGLU: one per epilogue warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  int64_t* total_mtiles_s = reinterpret_cast<int64_t*>(smem + C::OFF_MISC + 8);

  if (warp == 0 && lane == 0) {
    *abort_flag = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    mbar_init(drain_sf_bar, 1);
    for (int s = 0; s < STAGES; ++s) mbar_init(sfready_bar(s), SFP == 2 ? 4 : 1);
    for (int w = 0; w < kEpiWarps; ++w) mbar_init(cbar0 + 8u * w, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (kDglu) {
      tma_prefetch_desc(&tmC);
      if (p.d_tma) tma_prefetch_desc(&tmD);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  pdl_wait();  // inputs of a preceding kernel are visible after this point
  if (warp == 2) build_table(p.gs, tab0, tab1, lane, total_mtiles_s);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // the fused up-proj tile covers 128 compact columns: its 256 B rows are
  // gate rows [n0, n0 + 128) and up rows [H + n0, H + n0 + 128)
  constexpr bool kUpProj = EPI == kEpiSwiGLUQ;
  constexpr int TW = kUpProj ? BN / 2 : BN;
  static_assert(!kUpProj || (BN == 256 && ACC == 1), "fused up-proj tiles are 128 + 128 wide");
  auto rb_of = [&](const TileInfo& ti) -> int {
    if (kUpProj) return C::RB;
    const int v = static_cast<int>((p.n - ti.n0 + 127) / 128);
    return v < C::RB ? v : C::RB;
  };
  // discrete weights: an expert whose pointers failed the checks writes nothing
  auto tile_ok = [&](const TileInfo& ti) -> bool { return !p.w_ok || __ldg(p.w_ok + ti.g) != 0; };
  Schedule sch;
  sch.n_tiles = static_cast<int>((p.n + TW - 1) / TW);
  sch.total_tiles = *total_mtiles_s * sch.n_tiles;
  sch.tab0 = tab0;
  sch.tab1 = tab1;
  const int num_kb = static_cast<int>((p.k + C::BK - 1) / C::BK);
  const int atoms_total = static_cast<int>(p.S / 4);
  const WaitCtx wctx{p.gs.status, abort_flag, p.wait_limit_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t filled_mask = 0, last_parity = 0;
      bool ok = true;
      int map_g = -1;  // group whose discrete tensor map was last acquired
      for (int64_t t = blockIdx.x; ok && t < sch.total_tiles; t += gridDim.x) {
        const TileInfo ti = decode_tile(p.gs, sch, t, TW);
        const uint8_t* sfa_rows = p.sfa + (ti.row0 / kBM) * atoms_total * 512;
        // stacked B: one map over all groups (z = group); discrete B: the
        // group's own map (z = 0) and scale pointer
        const CUtensorMap* mapB = &tmB;
        int32_t zb = ti.g;
        bool w_ok = true;
        const uint8_t* sfb_grp;
        if (p.b_maps) {
          mapB = p.b_maps + ti.g;
          zb = 0;
          w_ok = __ldg(p.w_ok + ti.g) != 0;
          sfb_grp = reinterpret_cast<const uint8_t*>(__ldg(p.sfb_ptrs + ti.g));
          if (ti.g != map_g) {
            tensormap_acquire(mapB);
            map_g = ti.g;
          }
        } else {
          sfb_grp = p.sfb + static_cast<int64_t>(ti.g) * p.sfb_group_bytes;
        }
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, wctx)) { ok = false; break; }
          int atoms = atoms_total - kb * C::ATOMS;
          atoms = atoms < C::ATOMS ? atoms : C::ATOMS;
          // a skipped expert's stage holds stale B data: its MMAs run, its
          // results are never stored
          const int rb_valid = w_ok ? rb_of(ti) : 0;
          const uint32_t bytes =
              C::A_BYTES + (w_ok ? C::B_BYTES : 0u) + atoms * 512u * (1 + rb_valid);
          mbar_arrive_expect_tx(full_bar(stage), bytes);
          tma_load_2d(sbase + C::OFF_A + stage * C::A_BYTES, &tmA, full_bar(stage),
                      kb * kBKBytes, static_cast<int32_t>(ti.row0));
          if (!w_ok) {
          } else if (kUpProj) {
            // two 128-row boxes; with the 128-byte swizzle repeating every 8
            // rows the pair lands exactly as one 256-row box would
            tma_load_3d(sbase + C::OFF_B + stage * C::B_BYTES, mapB, full_bar(stage),
                        kb * kBKBytes, ti.n0, zb);
            tma_load_3d(sbase + C::OFF_B + stage * C::B_BYTES + 128 * kBKBytes, mapB, full_bar(stage),
                        kb * kBKBytes, static_cast<int32_t>(p.n + ti.n0), zb);
          } else {
            tma_load_3d(sbase + C::OFF_B + stage * C::B_BYTES, mapB, full_bar(stage),
                        kb * kBKBytes, ti.n0, zb);
          }
          bulk_load(sbase + C::OFF_SFA + stage * C::SFA_BYTES, sfa_rows + kb * C::ATOMS * 512,
                    atoms * 512u, full_bar(stage));
          for (int rb = 0; rb < rb_valid; ++rb) {
            // 128-row block of B holding tile rows [128 rb, 128 rb + 128)
            const int64_t blk = kUpProj ? (rb * p.n + ti.n0) / 128 : ti.n0 / 128 + rb;
            const uint8_t* src = sfb_grp + (blk * atoms_total + kb * C::ATOMS) * 512;
            bulk_load(sbase + C::OFF_SFB + stage * C::SFB_BYTES + rb * C::ATOMS * 512, src,
                      atoms * 512u, full_bar(stage));
          }
          filled_mask |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // every copy this thread issued has landed before the CTA may exit
      for (int s = 0; s < STAGES; ++s)
        if (filled_mask & (1u << s)) wait_drain(full_bar(s), (last_parity >> s) & 1u, p.wait_limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      // The tensor pipe keeps only about one MMA queued behind the executing
      // one, so every instruction this thread runs between MMAs can leave it
      // idle: descriptors are formed once and advanced by constants, and a
      // whole k-block's MMAs are issued unrolled.
      const uint64_t adesc0 = smem_desc_sw128(sbase + C::OFF_A);
      const uint64_t bdesc0 = smem_desc_sw128(sbase + C::OFF_B);
      constexpr int kFullMma = MODE == HQ_NVFP4 ? C::ATOMS : kBKBytes / kMmaKBytes;
      for (int64_t t = blockIdx.x; ok && t < sch.total_tiles; t += gridDim.x) {
        const TileInfo ti = decode_tile(p.gs, sch, t, TW);
        const int rb_valid = rb_of(ti);
        if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, wctx)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          // SFP 0: this thread stages the scales; otherwise the scale
          // warp(s) signal sfready after the stage's scales are in TMEM
          const uint32_t ready = SFP == 0 ? full_bar(stage) : sfready_bar(stage);
          if (!wait_bounded(ready, phase, wctx)) { ok = false; break; }
          tc_fence_after();
          int atoms = atoms_total - kb * C::ATOMS;
          atoms = atoms < C::ATOMS ? atoms : C::ATOMS;
          const uint32_t sfa_t = tmem_base + C::SF_BASE_COL + stage * C::SF_STAGE_COLS;
          const uint32_t sfb_t = sfa_t + C::SFA_COLS;
          if (SFP == 0) {
            const uint32_t sfa_s = sbase + C::OFF_SFA + stage * C::SFA_BYTES;
            const uint32_t sfb_s = sbase + C::OFF_SFB + stage * C::SFB_BYTES;
            for (int a = 0; a < atoms; ++a) {
              tc_cp_32x128b_warpx4(sfa_t + a * 4, smem_desc_sfatom(sfa_s + a * 512));
              for (int rb = 0; rb < rb_valid; ++rb)
                tc_cp_32x128b_warpx4(sfb_t + (a * C::RB + rb) * 4,
                                     smem_desc_sfatom(sfb_s + (rb * C::ATOMS + a) * 512));
            }
          }
          // descriptor start addresses are in 16-byte units; one MMA consumes
          // 32 bytes of K
          const uint64_t ad = adesc0 + static_cast<uint64_t>((stage * C::A_BYTES) >> 4);
          const uint64_t bd = bdesc0 + static_cast<uint64_t>((stage * C::B_BYTES) >> 4);
          const uint32_t acc0 = kb > 0 ? 1u : 0u;
          auto issue = [&](int j, uint32_t acc_flag) {
            if (MODE == HQ_MXFP8) {
              // one scale per row per MMA: byte j of the atom's 32-bit columns
              const uint32_t idesc = C::IDESC_BASE | p.idesc_ab | (static_cast<uint32_t>(j) << 4) |
                                     (static_cast<uint32_t>(j) << 29);
              mma_mxf8(d_tmem, ad + 2 * j, bd + 2 * j, idesc,
                       sfa_t | (static_cast<uint32_t>(j) << 30),
                       sfb_t | (static_cast<uint32_t>(j) << 30), acc_flag);
            } else if (MODE == HQ_MXFP4) {
              // two scales per row per MMA: bytes 2 (j % 2), +1 of atom j / 2
              const uint32_t sf = static_cast<uint32_t>(j & 1) * 2u;
              const uint32_t idesc = C::IDESC_BASE | (sf << 4) | (sf << 29);
              mma_mxf4(d_tmem, ad + 2 * j, bd + 2 * j, idesc, (sfa_t + (j >> 1) * 4) | (sf << 30),
                       (sfb_t + (j >> 1) * C::RB * 4) | (sf << 30), acc_flag);
            } else {
              // four scales per row per MMA: one whole atom column group
              mma_nvf4(d_tmem, ad + 2 * j, bd + 2 * j, C::IDESC_BASE, sfa_t + j * 4,
                       sfb_t + j * C::RB * 4, acc_flag);
            }
          };
          if (MODE == HQ_MXFP8 || atoms == C::ATOMS) {
#pragma unroll
            for (int j = 0; j < kFullMma; ++j) issue(j, j > 0 ? 1u : acc0);
          } else {
            // a partial last k-block: one MMA per atom (NVFP4), two (MXFP4)
            const int n_mma = MODE == HQ_MXFP4 ? 2 * atoms : atoms;
            for (int j = 0; j < n_mma; ++j) issue(j, j > 0 ? 1u : acc0);
          }
          tc_commit(empty_bar(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));
        if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
      }
      // all tcgen05 work issued by this thread is complete before TMEM is freed
      tc_commit(drain_bar);
      wait_drain(drain_bar, 0, p.wait_limit_ns);
    }
  } else if (warp >= kSfWarp0) {
    // ------------------------------------------------------------ scale staging
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; ok && t < sch.total_tiles; t += gridDim.x) {
      const TileInfo ti = decode_tile(p.gs, sch, t, TW);
      const int rb_valid = rb_of(ti);
      for (int kb = 0; kb < num_kb; ++kb) {
        int atoms = atoms_total - kb * C::ATOMS;
        atoms = atoms < C::ATOMS ? atoms : C::ATOMS;
        const uint32_t sfa_t = tmem_base + C::SF_BASE_COL + stage * C::SF_STAGE_COLS;
        const uint32_t sfb_t = sfa_t + C::SFA_COLS;
        const uint32_t sfa_s = sbase + C::OFF_SFA + stage * C::SFA_BYTES;
        const uint32_t sfb_s = sbase + C::OFF_SFB + stage * C::SFB_BYTES;
        if (SFP == 1) {
          if (lane == 0) {
            ok = wait_bounded(full_bar(stage), phase, wctx);
            if (ok) {
              tc_fence_after();
              for (int a = 0; a < atoms; ++a) {
                tc_cp_32x128b_warpx4(sfa_t + a * 4, smem_desc_sfatom(sfa_s + a * 512));
                for (int rb = 0; rb < rb_valid; ++rb)
                  tc_cp_32x128b_warpx4(sfb_t + (a * C::RB + rb) * 4,
                                       smem_desc_sfatom(sfb_s + (rb * C::ATOMS + a) * 512));
              }
              tc_commit(sfready_bar(stage));
            }
          }
          ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        } else {
          const bool w = wait_bounded(full_bar(stage), phase, wctx);
          ok = __all_sync(0xFFFFFFFFu, w);
          if (!ok) break;
          // lane i carries row i of each 512-byte atom: 16 bytes = 4 columns
          const uint32_t lq = static_cast<uint32_t>(q * 32) << 16;
          if (atoms == C::ATOMS && rb_valid == C::RB) {
            // whole k-block: all loads first, then one wide store per operand
            constexpr int NA = 4 * C::ATOMS;
            constexpr int NB = 4 * C::ATOMS * C::RB;
            uint32_t va[NA], vb[NB];
#pragma unroll
            for (int a = 0; a < C::ATOMS; ++a) {
              lds128(sfa_s + a * 512 + lane * 16, va + 4 * a);
#pragma unroll
              for (int rb = 0; rb < C::RB; ++rb)
                lds128(sfb_s + (rb * C::ATOMS + a) * 512 + lane * 16, vb + 4 * (a * C::RB + rb));
            }
            tmem_st_32x32b<NA>(lq + sfa_t, va);
            tmem_st_32x32b<NB>(lq + sfb_t, vb);
          } else {
          for (int a = 0; a < atoms; ++a) {
            uint32_t v0, v1, v2, v3;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                         : "r"(sfa_s + a * 512 + lane * 16));
            tmem_st_32x32b_x4(lq + sfa_t + a * 4, v0, v1, v2, v3);
            for (int rb = 0; rb < rb_valid; ++rb) {
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                           : "r"(sfb_s + (rb * C::ATOMS + a) * 512 + lane * 16));
              tmem_st_32x32b_x4(lq + sfb_t + (a * C::RB + rb) * 4, v0, v1, v2, v3);
            }
          }
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sfready_bar(stage));
        }
        if (!ok) break;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (SFP == 1 && lane == 0) {
      tc_commit(drain_sf_bar);
      wait_drain(drain_sf_bar, 0, p.wait_limit_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int ew = warp - 2;
    int acc = 0;
    uint32_t acc_phase = 0;
    if (kUpProj) {
      // fused up-proj: the warp owns compact columns [64 h, 64 h + 64) of
      // the tile; y is formed while TMEM is drained, TMEM is released, then
      // y is quantised and stored (one row per thread)
      const float gq = p.q_gscale ? __ldg(p.q_gscale) : 1.0f;
      const int h = ew >> 2;
      for (int64_t t = blockIdx.x; t < sch.total_tiles; t += gridDim.x) {
        const TileInfo ti = decode_tile(p.gs, sch, t, TW);
        const float alpha = p.alpha ? __ldg(p.alpha + ti.g) : 1.0f;  // loaded before the wait
        const bool okw = wait_bounded(tfull_bar(acc), acc_phase, wctx);
        if (!__all_sync(0xFFFFFFFFu, okw)) break;
        tc_fence_after();
        float y[64];
        swiglu_drain(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + 64 * h, alpha, y);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(acc));
        const int r_local = q * 32 + lane;
        if (r_local >= ti.row_lo && r_local < ti.rows_valid && tile_ok(ti)) {
          const int64_t row = ti.row0 + r_local;
          swiglu_store(p, y, row, ti.n0 + 64 * h, gq);
          // MXFP8 scale columns past H / 32 (the layout pads them to a
          // multiple of 16) hold 0; the last tile of the row writes them
          if (p.q_mode == HQ_MXFP8 && h == 1 && ti.n0 + TW == p.n)
            for (int64_t sc = p.n / 32; sc < p.sfq_cols; sc += 4)
              *reinterpret_cast<uint32_t*>(p.sfq + sfatom_offset(row, sc, p.sfq_cols)) = 0u;
        }
        if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
      }
    }
    if (EPI == kEpiDSwiGLU || EPI == kEpiDGeGLU) {
      // dGLU: the warp owns two 32-column chunks of its lane quarter.  A
      // chunk's C segment [32 rows x 64 values] arrives by TMA in the warp's
      // 4 KB buffer (128-byte swizzle); each lane reads its row, and when
      // d_tma is set writes its D_row segment back into the buffer for one
      // TMA store.  The next chunk's C load is issued once that store has
      // read the buffer, so it overlaps the chunk's amax / D_col / dbias
      // work and the next accumulator wait.  Contiguous-schedule tiles are
      // whole 128-row blocks (group ends are multiples of 128).
      static_assert(EPI == kEpiGemm || kUpProj || (BN == 128 && ACC == 2), "dGLU tiles are 128 wide");
      const float norm = p.norm_const ? __ldg(p.norm_const) : 1.0f;
      const uint32_t eb = sbase + C::OFF_STAGE_OUT + ew * 4096;
      const uint32_t cbar = cbar0 + 8u * ew;
      uint32_t c_phase = 0;
      bool c_pending = false;
      auto chunk_live = [&](const TileInfo& ti, int c) -> bool {
        return ti.n0 + c * 32 < p.n && ti.rows_valid > q * 32 && tile_ok(ti);
      };
      auto load_c = [&](const TileInfo& ti, int c) {
        if (lane == 0) {
          bulk_wait_group_read0();  // the previous D_row store has read the buffer
          mbar_arrive_expect_tx(cbar, 4096);
          tma_load_2d(eb, &tmC, cbar, static_cast<int32_t>(2 * (ti.n0 + c * 32)),
                      static_cast<int32_t>(ti.row0 + q * 32));
        }
        c_pending = true;
      };
      const int cw0 = (ew >> 2) * 2;  // the warp's first chunk
      int64_t t = blockIdx.x;
      if (t < sch.total_tiles) {
        const TileInfo t0i = decode_tile(p.gs, sch, t, TW);
        if (chunk_live(t0i, cw0)) load_c(t0i, cw0);
      }
      bool ok = true;
      for (; ok && t < sch.total_tiles; t += gridDim.x) {
        const TileInfo ti = decode_tile(p.gs, sch, t, TW);
        const int r_local = q * 32 + lane;
        const bool row_ok = r_local < ti.rows_valid;
        const int64_t row = ti.row0 + r_local;
        const float alpha = __ldg(p.alpha + ti.g);
        const float a2 = __fmul_rn(alpha, alpha);
        const float beta = EPI == kEpiDSwiGLU ? __ldg(p.beta + ti.g) : 1.0f;
        const float prob = row_ok ? __ldg(p.prob + row) : 0.0f;
        for (int cc = 0; cc < 2; ++cc) {
          const int c = cw0 + cc;
          const int64_t j0 = ti.n0 + c * 32;
          const bool live = chunk_live(ti, c);
          if (cc == 0) {
            const bool w = wait_bounded(tfull_bar(acc), acc_phase, wctx);
            if (!__all_sync(0xFFFFFFFFu, w)) { ok = false; break; }
            tc_fence_after();
          }
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + c * 32, r);
          tmem_ld_wait();
          if (cc == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
          }
          float dg[32], di[32];
          bool row_w = false;
          if (live) {
            const bool w = wait_bounded(cbar, c_phase, wctx);
            if (!__all_sync(0xFFFFFFFFu, w)) { ok = false; break; }
            c_pending = false;
            c_phase ^= 1u;
            uint4 cv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint32_t v[4];
              lds128(eb + static_cast<uint32_t>(lane) * 128u + ((static_cast<uint32_t>(i) ^ (lane & 7)) << 4), v);
              cv[i] = make_uint4(v[0], v[1], v[2], v[3]);
            }
            float dprob = 0.0f;
            dglu_math<EPI>(r, cv, a2, beta, prob, dg, di, dprob);
            // debug builds: this row and chunk lie inside D_row (and D_col)
            row_w = row_ok && in_bounds(row < p.gs.a_rows && j0 + 32 <= p.n && ti.g < p.gs.groups,
                                        p.gs.status);
            const uint32_t dbuf = (p.d_tma && __all_sync(0xFFFFFFFFu, row_w)) ? eb : 0u;
            dglu_write_row(p, dg, di, row_w, row, j0, norm, dprob, dbuf, lane);
            if (dbuf) {
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmD, eb, static_cast<int32_t>(2 * j0), static_cast<int32_t>(ti.row0 + q * 32));
                bulk_commit_group();
              }
            }
          }
          // the next C segment: this tile's second chunk, or the next tile's first
          if (cc == 0) {
            if (chunk_live(ti, c + 1)) load_c(ti, c + 1);
          } else if (t + gridDim.x < sch.total_tiles) {
            const TileInfo tn = decode_tile(p.gs, sch, t + gridDim.x, TW);
            if (chunk_live(tn, cw0)) load_c(tn, cw0);
          }
          if (live) dglu_tail(p, dg, di, row_w, row, j0, ti.g, norm, lane);
        }
        if (!ok) break;
        if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
      }
      // abort: a C load still in flight lands before the CTA exits; every TMA
      // store has completed before the CTA exits
      if (c_pending) wait_drain(cbar, c_phase, p.wait_limit_ns);
      if (lane == 0) bulk_wait_group0();
    }
    for (int64_t t = blockIdx.x; EPI == kEpiGemm && t < sch.total_tiles; t += gridDim.x) {
      const TileInfo ti = decode_tile(p.gs, sch, t, TW);
      const float alpha = p.alpha ? __ldg(p.alpha + ti.g) : 1.0f;  // loaded before the wait
      // every lane waits; the warp proceeds only if all lanes saw completion
      const bool ok = wait_bounded(tfull_bar(acc), acc_phase, wctx);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      tc_fence_after();
      EpiArgs e;
      e.acc_t = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      e.cw = (ew >> 2) * (BN / 2);
      e.n0 = ti.n0;
      e.n = p.n;
      e.alpha = alpha;
      e.bias = p.bias ? p.bias + static_cast<int64_t>(ti.g) * p.n : nullptr;
      e.out = p.out + (ti.row0 + q * 32) * p.n;
      e.rows_here = tile_ok(ti) ? ti.rows_valid - q * 32 : 0;
      e.rows_lo = ti.row_lo - q * 32;
      e.stage_s = sbase + C::OFF_STAGE_OUT + ew * 1024;
      e.lane = lane;
      e.row_abs = ti.row0 + q * 32;
      e.rows_total = p.gs.a_rows;
      e.status = p.gs.status;
      const uint32_t tempty = tempty_bar(acc);
      // with one accumulator the next tile's MMAs wait for this epilogue:
      // release TMEM before storing
      epilogue_tile<BN, ACC == 1>(e, [&] { if (lane == 0) mbar_arrive(tempty); });
      if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
    }
  }

  __syncthreads();
  pdl_launch_dependents();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}


// ---------------------------------------------------------------------------
// 2-SM variant of the dense GEMM (cta_group::2): a cluster of two CTAs on two
// SMs computes a 256 x 256 tile.  CTA r loads rows [128 r, 128 r + 128) of the
// A tile and rows [128 r, 128 r + 128) of the B tile into its own shared
// memory; the even CTA issues MMAs of M = 256, N = 256 that
// read both CTAs' operands and write each CTA's 128 x 256 accumulator half in
// its own TMEM.  Per SM this halves the B operand bytes fetched for the same
// work compared with the 128 x 256 single-SM tile.
//
// Both CTAs' A / B copies complete on the even CTA's "full" barrier (the
// cta_group::2 form of the TMA load), which expects the bytes of the pair; the
// scale copies complete on each CTA's own barrier.  Each CTA's scale warps
// stage its scales into its TMEM and arrive on that same "full" barrier of
// the even CTA (nine arrivals: the producer's expect-tx and four scale warps
// per CTA), so the MMA issuer waits on one barrier per stage and whichever
// of the copies and the scale writes completes last releases it directly.
// The even CTA's commits are multicast to both CTAs' "empty" and "accumulator
// full" barriers; all epilogue warps arrive on the even CTA's "accumulator
// empty" barrier.  Those cross-CTA arrivals are relaxed: what they order is
// tcgen05 work already completed with tcgen05.wait, and a
// release would first wait for the warp's earlier global stores.  Scale factors: each CTA holds the A scales of
// its own 128 rows and the B scales of all 256 tile columns in its TMEM, in
// the same layout as the single-SM N = 256 tile.
// ---------------------------------------------------------------------------
// BN_ = 256: one M = 256, N = 256 MMA per K step.  BN_ = 384 (the wide
// tile): an N = 256 MMA into accumulator columns [0, 256) and an N = 128 MMA
// into [256, 384); each CTA holds 192 B rows (128 for the first MMA, then 64
// for the second), the B scales of all 384 tile rows, and TMEM has room for
// only SF_SLOTS stages of scales, reused once the MMAs of an older stage are
// done.
template <int MODE, int STAGES, int BN_ = 256>
struct Cfg2 {
  static constexpr int GS = MODE == HQ_NVFP4 ? 16 : 32;
  static constexpr int EPB = MODE == HQ_MXFP8 ? 1 : 2;
  static constexpr int BK = kBKBytes * EPB;
  static constexpr int ATOMS = BK / GS / 4;
  static constexpr int BN = BN_;                       // tile columns (both CTAs)
  static constexpr int RB = BN / 128;                  // 128-row blocks of the tile's B scales
  static constexpr int A_BYTES = kBM * kBKBytes;       // this CTA's 128 rows of A
  static constexpr int B_BYTES = (BN / 2) * kBKBytes;  // this CTA's BN / 2 rows of B
  static constexpr int SFA_BYTES = ATOMS * 512;        // this CTA's 128 A rows
  static constexpr int SFB_BYTES = RB * ATOMS * 512;   // all BN B rows of the tile
  static constexpr int SFA_COLS = (ATOMS * 4 + 7) / 8 * 8;
  static constexpr int SFB_COLS = RB * ATOMS * 4;      // first MMA: 8 per atom; second: 4
  static constexpr int SF_STAGE_COLS = (SFA_COLS + SFB_COLS + 15) / 16 * 16;
  static constexpr int SF_BASE_COL = BN;
  static constexpr int SF_FIT = (512 - BN) / SF_STAGE_COLS;
  static constexpr int SF_SLOTS = SF_FIT < STAGES ? SF_FIT : STAGES;
  static_assert(SF_SLOTS >= 1 && STAGES % SF_SLOTS == 0, "scale slots");
  static constexpr int TMEM_USED = BN + SF_SLOTS * SF_STAGE_COLS;
  static constexpr int TMEM_COLS = 512;
  static_assert(TMEM_USED <= 512, "TMEM budget");
  static_assert(BN == 256 || BN == 384, "pair tiles of 256 or 384 columns");
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_STAGE_OUT = OFF_SFB + STAGES * SFB_BYTES;
  static constexpr int OFF_TABLE = OFF_STAGE_OUT + kEpiWarps * 1024;  // masked: 2 x (kMaxGroups + 1) int32
  static constexpr int OFF_BAR = OFF_TABLE + 2 * (kMaxGroups + 1) * 4 + 8;
  static constexpr int NUM_BARS = 3 * STAGES + 3;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static_assert(SMEM_BYTES <= kSmemLimit, "shared memory budget");
  // M = 256 across the pair; N = 256 (IDESC_BASE) and, for the wide tile's
  // second MMA, N = 128 (IDESC_N128)
  static constexpr uint32_t IDESC_KIND =
      (MODE == HQ_MXFP8 ? ((0u << 7) | (0u << 10) | (1u << 23))
       : MODE == HQ_MXFP4 ? ((1u << 7) | (1u << 10) | (1u << 23))
                          : ((1u << 7) | (1u << 10) | (0u << 23)))
      | (static_cast<uint32_t>(256 >> 4) << 24);
  static constexpr uint32_t IDESC_BASE = IDESC_KIND | (static_cast<uint32_t>(256 >> 3) << 17);
  static constexpr uint32_t IDESC_N128 = IDESC_KIND | (static_cast<uint32_t>(128 >> 3) << 17);
};

// EPI = kEpiSwiGLUQ: the fused up-proj (p.n = H): the tile's 256 B rows are
// gate rows [n0, n0 + 128) (even CTA) and up rows [H + n0, H + n0 + 128) (odd
// CTA), so each CTA's accumulator half holds gate in columns [0, 128) and up
// in [128, 256), as in the single-SM fused tile; tiles step 128 compact columns.
template <int MODE, int STAGES, int EPI = kEpiGemm, int BN = 256>
__global__ void __launch_bounds__(kThreads, 1)
    bs_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmB64, const __grid_constant__ CUtensorMap tmSFB,
                       const GemmParams p) {
  using C = Cfg2<MODE, STAGES, BN>;
  constexpr bool kUpProj = EPI == kEpiSwiGLUQ;
  constexpr bool kWide = BN == 384;
  static_assert(EPI == kEpiGemm || kUpProj, "2-SM epilogues: plain GEMM or fused up-proj");
  static_assert(!(kWide && kUpProj), "the fused up-proj uses 256-column pair tiles");
  constexpr int TW = kUpProj ? C::BN / 2 : C::BN;  // output columns per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  const bool leader = rank == 0;

  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };  // the pair's A, B and scales in TMEM (leader)
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };     // leader's commit
  auto sffull_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); }; // this CTA's scales
  const uint32_t tfull_bar = bar0 + 8u * (3 * STAGES);
  const uint32_t tempty_bar = tfull_bar + 8u;  // used in the leader
  const uint32_t drain_bar = tfull_bar + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  int64_t* total_pairs_s = reinterpret_cast<int64_t*>(smem + C::OFF_MISC + 8);
  int32_t* tab0 = reinterpret_cast<int32_t*>(smem + C::OFF_TABLE);
  int32_t* tab1 = tab0 + (kMaxGroups + 1);
  const bool masked = p.gs.sched == kMasked;
  const bool contig = p.gs.sched == kContig;

  if (warp == 0 && lane == 0) {
    *abort_flag = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 9);  // the producer's expect-tx + 4 scale warps in each CTA
      mbar_init(empty_bar(s), 1);
      mbar_init(sffull_bar(s), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, 2 * kEpiWarps);  // every epilogue warp of both CTAs
    mbar_init(drain_bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (kWide) tma_prefetch_desc(&tmB64);
    if (!kUpProj) tma_prefetch_desc(&tmSFB);
  }
  if (warp == 1) {  // one warp in each CTA allocates, collectively for the pair
    tmem_alloc_2sm(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish_2sm();
  }
  pdl_wait();
  // masked layout: per expert the number of 256-row pairs holding valid rows
  // and their exclusive prefix (both CTAs build the same table).
  // contiguous layout: tab0 = the sanitised group ends, tab1 = the exclusive
  // prefix of each group's 256-row pairs (a group's pairs start at its first
  // row, so a pair never mixes two groups)
  if (warp == 2 && masked) build_table(p.gs, tab0, tab1, lane, total_pairs_s, 256);
  if (warp == 2 && contig) {
    build_table(p.gs, tab0, tab1, lane, total_pairs_s);
    __syncwarp();
    int32_t carry = 0;
    for (int base = 0; base < p.gs.groups; base += 32) {
      const int g = base + lane;
      int32_t pairs = 0;
      if (g < p.gs.groups) {
        const int32_t start = g > 0 ? tab0[g - 1] : 0;
        pairs = (tab0[g] - start + 255) / 256;
      }
      int32_t incl = pairs;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
      }
      if (g < p.gs.groups) tab1[g] = carry + incl - pairs;
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) *total_pairs_s = carry;
  }
  __syncthreads();
  cluster_sync();  // both CTAs' barriers and TMEM exist before any cross-CTA use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int n_tiles = static_cast<int>((p.n + TW - 1) / TW);
  const int64_t m_pairs = (masked || contig) ? *total_pairs_s : (p.gs.a_rows + 255) / 256;
  const int64_t total = m_pairs * n_tiles;
  const int64_t cluster_id = blockIdx.x >> 1;
  const int64_t num_clusters = gridDim.x >> 1;
  const int64_t rows_pad = (p.gs.a_rows + kBM - 1) / kBM * kBM;  // rows the scale buffer holds
  const int num_kb = static_cast<int>((p.k + C::BK - 1) / C::BK);
  const int atoms_total = static_cast<int>(p.S / 4);
  const WaitCtx wctx{p.gs.status, abort_flag, p.wait_limit_ns};
  // Tile t of the pair: 256 rows from `base` (dense: all rows; masked: one
  // expert's rows, from e * max_m), columns [n0, n0 + 256).  CTA r owns rows
  // [base + 128 r, base + 128 r + 128), of which valid0 / valid1 (0..128) hold data.
  struct PairTile {
    int64_t row0;  // this CTA's first row
    int n0;
    int g;
    int valid0, valid1;  // valid rows of the even / odd CTA
    int mine;            // valid rows of this CTA
  };
  auto pair_tile = [&](int64_t t) {
    PairTile pt;
    const int64_t mt = t / n_tiles;
    pt.n0 = static_cast<int>(t - mt * n_tiles) * TW;
    int64_t base, cnt;
    if (masked || contig) {
      const int32_t* prefix = masked ? tab0 : tab1;
      int lo = 0, hi = p.gs.groups - 1;  // last group with prefix[g] <= mt
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= mt) lo = mid; else hi = mid - 1;
      }
      const int64_t local = mt - prefix[lo];
      pt.g = lo;
      if (masked) {
        base = static_cast<int64_t>(lo) * p.gs.max_m + local * 256;
        cnt = static_cast<int64_t>(tab1[lo]) - local * 256;
      } else {
        const int64_t start = lo > 0 ? tab0[lo - 1] : 0;
        base = start + local * 256;
        cnt = static_cast<int64_t>(tab0[lo]) - base;
      }
    } else {
      pt.g = 0;
      base = mt * 256;
      cnt = p.gs.a_rows - base;
    }
    pt.valid0 = cnt <= 0 ? 0 : (cnt >= 128 ? 128 : static_cast<int>(cnt));
    pt.valid1 = cnt <= 128 ? 0 : (cnt >= 256 ? 128 : static_cast<int>(cnt - 128));
    pt.mine = rank ? pt.valid1 : pt.valid0;
    pt.row0 = base + rank * kBM;
    return pt;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, filled_a = 0, filled_s = 0, par_a = 0, par_s = 0;
      int64_t issued = 0;  // stages issued by this producer
      bool ok = true;
      for (int64_t t = cluster_id; ok && t < total; t += num_clusters) {
        const PairTile pt = pair_tile(t);
        const int64_t row0 = pt.row0;
        // this CTA's first 128 B rows, and the 128-row blocks of the tile's B
        const int nh0 = kUpProj ? (rank ? static_cast<int>(p.n) + pt.n0 : pt.n0)
                                : pt.n0 + static_cast<int>(rank) * 128;
        auto sfb_blk = [&](int rb) -> int64_t {
          return kUpProj && rb == 1 ? (p.n + pt.n0) / 128 : pt.n0 / 128 + rb;
        };
        // a CTA whose 128 rows hold no valid row loads no A and no A scales
        // (its accumulator half is never stored)
        const bool has_a = pt.mine > 0;
        // B scale blocks inside n (a 384-wide tile may end past n: its last
        // block's scales do not exist; those columns are never stored)
        const int64_t rb_in = (p.n - pt.n0 + 127) / 128;
        const uint32_t rb_valid = static_cast<uint32_t>(kUpProj || rb_in >= C::RB ? C::RB : rb_in);
        const bool has_sfa = has_a && row0 < rows_pad;
        const uint32_t pair_bytes = (pt.valid0 > 0 ? C::A_BYTES : 0u) +
                                    (pt.valid1 > 0 ? C::A_BYTES : 0u) + 2u * C::B_BYTES;
        const uint8_t* sfa_rows = p.sfa + (row0 / kBM) * atoms_total * 512;
        const uint8_t* sfb_grp = p.sfb + static_cast<int64_t>(pt.g) * p.sfb_group_bytes;
        const int64_t sfb_blk0 = static_cast<int64_t>(pt.g) * (p.sfb_group_bytes / (128 * p.S));
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, wctx)) { ok = false; break; }
          int atoms = atoms_total - kb * C::ATOMS;
          atoms = atoms < C::ATOMS ? atoms : C::ATOMS;
          // the scale copies go first: they are small, and the scale warps'
          // staging into TMEM then overlaps the A / B copies still landing
          // (1% faster than issuing them last)
          // B scales: one box of the tile's RB consecutive 128-row blocks
          // (atoms past K and blocks past the tensor read as zeros and count
          // in full; blocks past n are never used); the fused up-proj's two
          // blocks are apart, one bulk copy each
          const uint32_t sfb_bytes = kUpProj ? atoms * 512u * rb_valid : static_cast<uint32_t>(C::SFB_BYTES);
          mbar_arrive_expect_tx(sffull_bar(stage), (has_sfa ? atoms * 512u : 0u) + sfb_bytes);
          if (has_sfa)
            bulk_load(sbase + C::OFF_SFA + stage * C::SFA_BYTES, sfa_rows + kb * C::ATOMS * 512,
                      atoms * 512u, sffull_bar(stage));
          if (kUpProj) {
            for (int rb = 0; rb < rb_valid; ++rb)
              bulk_load(sbase + C::OFF_SFB + stage * C::SFB_BYTES + rb * C::ATOMS * 512,
                        sfb_grp + (sfb_blk(rb) * atoms_total + kb * C::ATOMS) * 512,
                        atoms * 512u, sffull_bar(stage));
          } else {
            tma_load_3d(sbase + C::OFF_SFB + stage * C::SFB_BYTES, &tmSFB, sffull_bar(stage), 0, kb * C::ATOMS,
                        static_cast<int32_t>(sfb_blk0 + pt.n0 / 128));
          }
          // both CTAs' A / B tiles complete on the even CTA's full barrier,
          // which expects the bytes of the pair (a fault-injection test
          // withholds this arrival once: the stage never completes and the
          // MMA issuer's bounded wait expires)
          if (leader && !(cluster_id == 0 && issued == p.inject_skip))
            mbar_arrive_expect_tx(full_bar(stage), pair_bytes);
          ++issued;
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          if (has_a)
            tma_load_2d_pair(sbase + C::OFF_A + stage * C::A_BYTES, &tmA, fb, kb * kBKBytes,
                             static_cast<int32_t>(row0));
          const uint32_t b_s = sbase + C::OFF_B + stage * C::B_BYTES;
          // B rows [n0 + 128 r, + 128) for the N = 256 MMA and, for the wide
          // tile, [n0 + 256 + 64 r, + 64) for the N = 128 MMA
          tma_load_3d_pair(b_s, &tmB, fb, kb * kBKBytes, nh0, pt.g);
          if (kWide)
            tma_load_3d_pair(b_s + 128 * kBKBytes, &tmB64, fb, kb * kBKBytes,
                             pt.n0 + 256 + static_cast<int>(rank) * 64, pt.g);
          filled_a |= 1u << stage;
          filled_s |= 1u << stage;
          par_a = (par_a & ~(1u << stage)) | (phase << stage);
          par_s = par_a;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // the even CTA's full barriers count both CTAs' A / B bytes, so its
      // drain covers the odd CTA's copies too (the odd CTA stays resident
      // until the final cluster barrier); after an abort a phase may also
      // lack scale-warp arrivals, and the bounded drain then ends at its limit
      for (int s = 0; s < STAGES; ++s) {
        if (leader && (filled_a & (1u << s)))
          wait_drain(full_bar(s), (par_a >> s) & 1u, p.wait_limit_ns);
        if (filled_s & (1u << s)) wait_drain(sffull_bar(s), (par_s >> s) & 1u, p.wait_limit_ns);
      }
    }
  } else if (warp == 1 && !leader) {
    // odd CTA: no MMA issuer
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      // as in the single-SM kernel: constant descriptor advances, unrolled
      // MMAs, one wait per stage
      const uint64_t adesc0 = smem_desc_sw128(sbase + C::OFF_A);
      const uint64_t bdesc0 = smem_desc_sw128(sbase + C::OFF_B);
      constexpr int kFullMma = MODE == HQ_NVFP4 ? C::ATOMS : kBKBytes / kMmaKBytes;
      for (int64_t t = cluster_id; ok && t < total; t += num_clusters) {
        if (!wait_bounded(tempty_bar, acc_phase ^ 1u, wctx)) break;
        tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb) {
          // "full" completes once the pair's A / B tiles landed and both
          // CTAs' scales for the stage are in TMEM: one wait per stage (two
          // waits, on the tiles and on the scales apart, cost 4% more time)
          if (!wait_bounded(full_bar(stage), phase, wctx)) { ok = false; break; }
          tc_fence_after();
          int atoms = atoms_total - kb * C::ATOMS;
          atoms = atoms < C::ATOMS ? atoms : C::ATOMS;
          const int slot = stage % C::SF_SLOTS;
          const uint32_t sfa_t = tmem_base + C::SF_BASE_COL + slot * C::SF_STAGE_COLS;
          const uint32_t sfb_t = sfa_t + C::SFA_COLS;
          const uint32_t sfb2_t = sfb_t + C::ATOMS * 8;  // wide tile: the N = 128 MMA's scales
          const uint64_t ad = adesc0 + static_cast<uint64_t>((stage * C::A_BYTES) >> 4);
          const uint64_t bd = bdesc0 + static_cast<uint64_t>((stage * C::B_BYTES) >> 4);
          const uint64_t bd2 = bd + static_cast<uint64_t>((128 * kBKBytes) >> 4);
          const uint32_t acc0 = kb > 0 ? 1u : 0u;
          auto issue = [&](int j, uint32_t acc_flag) {
            if (MODE == HQ_MXFP8) {
              const uint32_t sel = (static_cast<uint32_t>(j) << 4) | (static_cast<uint32_t>(j) << 29);
              const uint32_t sfs = static_cast<uint32_t>(j) << 30;
              mma_mxf8_2sm(tmem_base, ad + 2 * j, bd + 2 * j, C::IDESC_BASE | p.idesc_ab | sel, sfa_t | sfs,
                           sfb_t | sfs, acc_flag);
              if (kWide)
                mma_mxf8_2sm(tmem_base + 256, ad + 2 * j, bd2 + 2 * j, C::IDESC_N128 | p.idesc_ab | sel, sfa_t | sfs,
                             sfb2_t | sfs, acc_flag);
            } else if (MODE == HQ_MXFP4) {
              const uint32_t sf = static_cast<uint32_t>(j & 1) * 2u;
              const uint32_t sel = (sf << 4) | (sf << 29);
              mma_mxf4_2sm(tmem_base, ad + 2 * j, bd + 2 * j, C::IDESC_BASE | sel,
                           (sfa_t + (j >> 1) * 4) | (sf << 30), (sfb_t + (j >> 1) * 8) | (sf << 30),
                           acc_flag);
              if (kWide)
                mma_mxf4_2sm(tmem_base + 256, ad + 2 * j, bd2 + 2 * j, C::IDESC_N128 | sel,
                             (sfa_t + (j >> 1) * 4) | (sf << 30), (sfb2_t + (j >> 1) * 4) | (sf << 30),
                             acc_flag);
            } else {
              mma_nvf4_2sm(tmem_base, ad + 2 * j, bd + 2 * j, C::IDESC_BASE, sfa_t + j * 4,
                           sfb_t + j * 8, acc_flag);
              if (kWide)
                mma_nvf4_2sm(tmem_base + 256, ad + 2 * j, bd2 + 2 * j, C::IDESC_N128, sfa_t + j * 4,
                             sfb2_t + j * 4, acc_flag);
            }
          };
          if (MODE == HQ_MXFP8 || atoms == C::ATOMS) {
#pragma unroll
            for (int j = 0; j < kFullMma; ++j) issue(j, j > 0 ? 1u : acc0);
          } else {
            const int n_mma = MODE == HQ_MXFP4 ? 2 * atoms : atoms;
            for (int j = 0; j < n_mma; ++j) issue(j, j > 0 ? 1u : acc0);
          }
          tc_commit_2sm_mc(empty_bar(stage), 0x3);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit_2sm_mc(tfull_bar, 0x3);
        acc_phase ^= 1u;
      }
      tc_commit_2sm_mc(drain_bar, 0x1);
      wait_drain(drain_bar, 0, p.wait_limit_ns);
    }
  } else if (warp >= kSfWarp0) {
    // ------------------------------------------------------------ scale staging (both CTAs)
    const int q = warp & 3;
    const uint32_t lq = static_cast<uint32_t>(q * 32) << 16;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int64_t kbi = 0;  // k-blocks this warp has staged
    for (int64_t t = cluster_id; ok && t < total; t += num_clusters) {
      for (int kb = 0; kb < num_kb; ++kb) {
        int atoms = atoms_total - kb * C::ATOMS;
        atoms = atoms < C::ATOMS ? atoms : C::ATOMS;
        const bool w = wait_bounded(sffull_bar(stage), phase, wctx);
        ok = __all_sync(0xFFFFFFFFu, w);
        if (!ok) break;
        const int slot = stage % C::SF_SLOTS;
        const uint32_t sfa_t = tmem_base + C::SF_BASE_COL + slot * C::SF_STAGE_COLS;
        const uint32_t sfb_t = sfa_t + C::SFA_COLS;
        const uint32_t sfb2_t = sfb_t + C::ATOMS * 8;
        const uint32_t sfa_s = sbase + C::OFF_SFA + stage * C::SFA_BYTES;
        const uint32_t sfb_s = sbase + C::OFF_SFB + stage * C::SFB_BYTES;
        // the TMEM scale slot is shared with k-block kbi - SF_SLOTS: its MMAs
        // (committed to that stage's empty barrier) must be done before the
        // slot is written; the stage's atoms are read from shared memory
        // first, so only the TMEM writes wait
        auto wait_slot = [&]() -> bool {
          if (C::SF_SLOTS < STAGES && kbi >= C::SF_SLOTS) {
            const int64_t j = kbi - C::SF_SLOTS;
            const bool we = wait_bounded(empty_bar(static_cast<int>(j % STAGES)),
                                         static_cast<uint32_t>(j / STAGES) & 1u, wctx);
            if (!__all_sync(0xFFFFFFFFu, we)) return false;
            tc_fence_after();
          }
          return true;
        };
        // B scales at columns sfb_t + (a * 2 + rb) * 4 (k-atom a, 128-row
        // block rb = 0, 1) and, for the wide tile, sfb2_t + a * 4 (block 2)
        if (atoms == C::ATOMS) {
          constexpr int NA = 4 * C::ATOMS;
          uint32_t va[NA], vb[2 * NA], vb2[NA];
#pragma unroll
          for (int a = 0; a < C::ATOMS; ++a) {
            lds128(sfa_s + a * 512 + lane * 16, va + 4 * a);
#pragma unroll
            for (int rb = 0; rb < 2; ++rb)
              lds128(sfb_s + (rb * C::ATOMS + a) * 512 + lane * 16, vb + 4 * (a * 2 + rb));
            if (kWide) lds128(sfb_s + (2 * C::ATOMS + a) * 512 + lane * 16, vb2 + 4 * a);
          }
          if (!wait_slot()) { ok = false; break; }
          tmem_st_32x32b<NA>(lq + sfa_t, va);
          tmem_st_32x32b<2 * NA>(lq + sfb_t, vb);
          if (kWide) tmem_st_32x32b<NA>(lq + sfb2_t, vb2);
        } else {
          if (!wait_slot()) { ok = false; break; }
          for (int a = 0; a < atoms; ++a) {
            uint32_t v[4];
            lds128(sfa_s + a * 512 + lane * 16, v);
            tmem_st_32x32b<4>(lq + sfa_t + a * 4, v);
            for (int rb = 0; rb < 2; ++rb) {
              lds128(sfb_s + (rb * C::ATOMS + a) * 512 + lane * 16, v);
              tmem_st_32x32b<4>(lq + sfb_t + (a * 2 + rb) * 4, v);
            }
            if (kWide) {
              lds128(sfb_s + (2 * C::ATOMS + a) * 512 + lane * 16, v);
              tmem_st_32x32b<4>(lq + sfb2_t + a * 4, v);
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(full_bar(stage), 0));
        ++kbi;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int ew = warp - 2;
    const uint32_t tempty_leader = mapa_shared(tempty_bar, 0);
    uint32_t acc_phase = 0;
    if (kUpProj) {
      // as the single-SM fused epilogue: y formed while draining, TMEM
      // released, then quantised and stored (one row per thread)
      const float gq = p.q_gscale ? __ldg(p.q_gscale) : 1.0f;
      const int h = ew >> 2;
      for (int64_t t = cluster_id; t < total; t += num_clusters) {
        const PairTile pt = pair_tile(t);
        const float alpha = p.alpha ? __ldg(p.alpha + pt.g) : 1.0f;
        const bool okw = wait_bounded(tfull_bar, acc_phase, wctx);
        if (!__all_sync(0xFFFFFFFFu, okw)) break;
        tc_fence_after();
        float y[64];
        swiglu_drain(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + 64 * h, alpha, y);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader);
        const int r_local = q * 32 + lane;
        if (r_local < pt.mine) {
          const int64_t row = pt.row0 + r_local;
          swiglu_store(p, y, row, pt.n0 + 64 * h, gq);
          if (p.q_mode == HQ_MXFP8 && h == 1 && pt.n0 + TW == p.n)
            for (int64_t sc = p.n / 32; sc < p.sfq_cols; sc += 4)
              *reinterpret_cast<uint32_t*>(p.sfq + sfatom_offset(row, sc, p.sfq_cols)) = 0u;
        }
        acc_phase ^= 1u;
      }
    }
    for (int64_t t = cluster_id; !kUpProj && t < total; t += num_clusters) {
      const PairTile pt = pair_tile(t);
      const float alpha = p.alpha ? __ldg(p.alpha + pt.g) : 1.0f;  // loaded before the wait
      const bool okw = wait_bounded(tfull_bar, acc_phase, wctx);
      if (!__all_sync(0xFFFFFFFFu, okw)) break;
      tc_fence_after();
      EpiArgs e;
      e.acc_t = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      e.cw = (ew >> 2) * 128;  // the first 256 columns (the wide tile's rest: epilogue_tile_wide)
      e.n0 = pt.n0;
      e.n = p.n;
      e.alpha = alpha;
      e.bias = p.bias ? p.bias + static_cast<int64_t>(pt.g) * p.n : nullptr;
      e.out = p.out + (pt.row0 + q * 32) * p.n;
      e.rows_here = pt.mine - q * 32;
      e.rows_lo = 0;
      e.stage_s = sbase + C::OFF_STAGE_OUT + ew * 1024;
      e.lane = lane;
      e.row_abs = pt.row0 + q * 32;
      e.rows_total = p.gs.a_rows;
      e.status = p.gs.status;
      auto release = [&] { if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader); };
      if (kWide) epilogue_tile_wide(e, (ew >> 2) * 64, release);
      else epilogue_tile<C::BN, true>(e, release);
      acc_phase ^= 1u;
    }
  }

  __syncthreads();
  pdl_launch_dependents();
  cluster_sync();  // the peer may still read this CTA's shared memory and TMEM until here
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_2sm(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <int MODE, int BN, int STAGES, int ACC, int TABLE, int EPI = kEpiGemm, int SFP = kSfPath>
int run_bs(const void* a, const void* b, const GemmParams& p0, int sm_count, bool pdl,
           cudaStream_t st) {
  constexpr bool kDglu = EPI == kEpiDSwiGLU || EPI == kEpiDGeGLU;
  using C = Cfg<MODE, BN, STAGES, ACC, TABLE, kDglu ? 4096 : 1024>;
  GemmParams p = p0;
  const uint64_t kbytes = static_cast<uint64_t>(p.k) / C::EPB;
  CUtensorMap tmA, tmB;
  {
    const uint64_t dims[2] = {kbytes, static_cast<uint64_t>(p.gs.a_rows)};
    const uint64_t strides[1] = {kbytes};
    const uint32_t box[2] = {kBKBytes, kBM};
    int rc = encode_tensor_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a), dims,
                               strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != HQ_OK) return rc;
  }
  // the fused up-proj B holds 2 n rows per group, loaded as two 128-row boxes
  constexpr bool kUpProj = EPI == kEpiSwiGLUQ;
  const uint64_t b_rows = static_cast<uint64_t>(kUpProj ? 2 * p.n : p.n);
  {
    // discrete weights: a one-group map whose address the device replaces per
    // expert; it is encoded over the workspace (a valid address) and is never
    // loaded through as it stands
    const bool discrete = p.b_ptrs != nullptr;
    const uint64_t groups = discrete ? 1 : static_cast<uint64_t>(p.gs.groups);
    const uint64_t dims[3] = {kbytes, b_rows, groups};
    const uint64_t strides[2] = {kbytes, kbytes * b_rows};
    const uint32_t box[3] = {kBKBytes, static_cast<uint32_t>(kUpProj ? 128 : BN), 1};
    void* base = discrete ? static_cast<void*>(p.b_maps) : const_cast<void*>(b);
    int rc = encode_tensor_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != HQ_OK) return rc;
    if (discrete) {
      rc = build_weight_maps(tmB, p.b_ptrs, p.sfb_ptrs, p.b_maps, p.w_ok, p.gs.groups, st);
      if (rc != HQ_OK) return rc;
    }
  }
  // dGLU: C and D_row [a_rows, 2n] in 32-row x 64-value segments; D_row by
  // TMA for BF16 (128-byte swizzle, like C) and for FP8 with SFD_row (plain
  // 64-byte rows); other D types are stored from registers
  CUtensorMap tmC = tmA, tmD = tmA;
  p.d_tma = 0;
  if (kDglu) {
    const uint64_t dims[2] = {static_cast<uint64_t>(2 * p.n), static_cast<uint64_t>(p.gs.a_rows)};
    const uint32_t box[2] = {64, 32};
    const uint64_t sc[1] = {static_cast<uint64_t>(2 * p.n) * 2};
    int rc = encode_tensor_map(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(p.c), dims,
                               sc, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != HQ_OK) return rc;
    if (p.d_type == kDBf16 && !p.sfd_row) {
      rc = encode_tensor_map(&tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.d_row, dims, sc, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
      if (rc != HQ_OK) return rc;
      p.d_tma = 1;
    } else if ((p.d_type == kDE4M3 || p.d_type == kDE5M2) && p.sfd_row) {
      const uint64_t s8[1] = {static_cast<uint64_t>(2 * p.n)};
      rc = encode_tensor_map(&tmD, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, p.d_row, dims, s8, box,
                             CU_TENSOR_MAP_SWIZZLE_NONE);
      if (rc != HQ_OK) return rc;
      p.d_tma = 2;
    }
  }
  auto kern = bs_gemm_kernel<MODE, BN, STAGES, ACC, TABLE, EPI, SFP>;
  if (set_smem_once<bs_gemm_kernel<MODE, BN, STAGES, ACC, TABLE, EPI, SFP>>(C::SMEM_BYTES) != HQ_OK)
    return HQ_ERR_CUDA;
  const int sms = num_sms();
  if (sms <= 0) return HQ_ERR_CUDA;
  int64_t mtiles_bound;
  if (p.gs.sched == kMasked)
    mtiles_bound = static_cast<int64_t>(p.gs.groups) * ((p.gs.max_m + kBM - 1) / kBM);
  else
    mtiles_bound = (p.gs.a_rows + kBM - 1) / kBM;
  const int64_t tw = kUpProj ? BN / 2 : BN;
  const int64_t tiles_bound = mtiles_bound * ((p.n + tw - 1) / tw);
  int64_t grid = sm_count > 0 ? sm_count : sms;
  if (grid > sms) grid = sms;
  if (grid > tiles_bound) grid = tiles_bound;
  if (grid < 1) grid = 1;
  cudaError_t e = launch(kern, dim3(static_cast<unsigned>(grid)), dim3(threads_for(SFP)), C::SMEM_BYTES, st,
                         pdl, tmA, tmB, tmC, tmD, p);
  return e == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
}

template <int MODE, int STAGES, int EPI = kEpiGemm, int BN = 256>
int run_bs_2sm(const void* a, const void* b, const GemmParams& p, int sm_count, bool pdl,
               cudaStream_t st) {
  using C = Cfg2<MODE, STAGES, BN>;
  constexpr bool kUpProj = EPI == kEpiSwiGLUQ;
  const uint64_t b_rows = static_cast<uint64_t>(kUpProj ? 2 * p.n : p.n);
  const uint64_t kbytes = static_cast<uint64_t>(p.k) / C::EPB;
  CUtensorMap tmA, tmB;
  {
    const uint64_t dims[2] = {kbytes, static_cast<uint64_t>(p.gs.a_rows)};
    const uint64_t strides[1] = {kbytes};
    const uint32_t box[2] = {kBKBytes, kBM};
    int rc = encode_tensor_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a), dims,
                               strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != HQ_OK) return rc;
  }
  CUtensorMap tmB64, tmSFB;
  {
    const uint64_t dims[3] = {kbytes, b_rows, static_cast<uint64_t>(p.gs.groups)};
    const uint64_t strides[2] = {kbytes, kbytes * b_rows};
    const uint32_t box[3] = {kBKBytes, 128u, 1};
    int rc = encode_tensor_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(b), dims,
                               strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != HQ_OK) return rc;
    tmB64 = tmB;
    if (BN == 384) {  // the wide tile's last 128 rows: 64 per CTA
      const uint32_t box64[3] = {kBKBytes, 64u, 1};
      rc = encode_tensor_map(&tmB64, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(b), dims, strides,
                             box64, CU_TENSOR_MAP_SWIZZLE_128B);
      if (rc != HQ_OK) return rc;
    }
  }
  // B scale atoms as [blocks of 128 rows][k-atoms][128 words of 32 bits]; a
  // box is a tile's RB blocks of one k-block
  tmSFB = tmB;
  if (!kUpProj) {
    const uint64_t atoms_total = static_cast<uint64_t>(p.S / 4);
    const uint64_t blocks = static_cast<uint64_t>(p.sfb_group_bytes / (128 * p.S)) *
                            static_cast<uint64_t>(p.gs.groups);
    const uint64_t dims[3] = {128, atoms_total, blocks};
    const uint64_t strides[2] = {512, atoms_total * 512};
    const uint32_t box[3] = {128, static_cast<uint32_t>(C::ATOMS), static_cast<uint32_t>(C::RB)};
    int rc = encode_tensor_map(&tmSFB, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t*>(p.sfb), dims,
                               strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != HQ_OK) return rc;
  }
  auto kern = bs_gemm_2sm_kernel<MODE, STAGES, EPI, BN>;
  if (set_smem_once<bs_gemm_2sm_kernel<MODE, STAGES, EPI, BN>>(C::SMEM_BYTES) != HQ_OK)
    return HQ_ERR_CUDA;
  const int sms = num_sms();
  if (sms < 2) return HQ_ERR_CUDA;
  // an upper bound of the pairs (contiguous: each group adds at most one
  // partial pair)
  const int64_t m_pairs = p.gs.sched == kMasked
                             ? static_cast<int64_t>(p.gs.groups) * ((p.gs.max_m + 255) / 256)
                             : (p.gs.a_rows + 255) / 256 + (p.gs.sched == kContig ? p.gs.groups : 0);
  const int64_t tw = kUpProj ? 128 : BN;
  const int64_t pairs_needed = m_pairs * ((p.n + tw - 1) / tw);
  int64_t pairs = (sm_count > 0 ? sm_count : sms) / 2;
  if (pairs > sms / 2) pairs = sms / 2;
  if (pairs > pairs_needed) pairs = pairs_needed;
  if (pairs < 1) pairs = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmB64, tmSFB, p);
  return e == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
}

int run_gemm(hq_mode mode, const void* a, const void* b, const GemmParams& p, int sm_count,
             bool pdl, cudaStream_t st) {
  mode = kernel_mode(mode);
  int bn = forced_tile_n();
  // dense, contiguous and masked problems with whole 256-column tiles
  // (masked: experts padded to a multiple of 256 rows) use the 2-SM kernel
  // unless a single-SM tile width is forced
  // (384-column pair tiles: n a multiple of 384; chosen automatically for
  // dense problems)
  const bool pairable = !p.b_maps && (p.gs.sched == kDense || p.gs.sched == kContig ||
                                      (p.gs.sched == kMasked && p.gs.max_m % 256 == 0));
  const int pw = pair_width();
  // a dense problem with fewer pair tiles than clusters keeps more SMs busy
  // with single-SM 128 x 128 tiles (unless a pair width is forced)
  if (bn == 0 && pw == 0 && p.gs.sched == kDense &&
      ((p.gs.a_rows + 255) / 256) * ((p.n + 255) / 256) < num_sms() / 2)
    bn = 128;
  // 384-wide pair tiles: automatically for dense problems with n a multiple
  // of 384; forced (pair width 384) for any n of at least 384 (the last tile
  // may end past n)
  const bool wide = (p.n % 384 == 0 && pw == 0 && p.gs.sched == kDense) || (pw == 384 && p.n >= 384);
  if (bn == 0 && pairable && use_2sm() && wide) {
    if (mode == HQ_MXFP8) return run_bs_2sm<HQ_MXFP8, 4, kEpiGemm, 384>(a, b, p, sm_count, pdl, st);
    if (mode == HQ_MXFP4) return run_bs_2sm<HQ_MXFP4, 4, kEpiGemm, 384>(a, b, p, sm_count, pdl, st);
    return run_bs_2sm<HQ_NVFP4, 4, kEpiGemm, 384>(a, b, p, sm_count, pdl, st);
  }
  if (bn == 0 && pairable && p.n % 256 == 0 && use_2sm()) {
    if (mode == HQ_MXFP8) return run_bs_2sm<HQ_MXFP8, 6>(a, b, p, sm_count, pdl, st);
    if (mode == HQ_MXFP4) return run_bs_2sm<HQ_MXFP4, 5>(a, b, p, sm_count, pdl, st);
    return run_bs_2sm<HQ_NVFP4, 5>(a, b, p, sm_count, pdl, st);
  }
  if (bn == 0) bn = (p.n % 256 == 0) ? 256 : 128;
  if (bn == 256 && p.n % 256 != 0 && p.n < 256) bn = 128;
  constexpr int T = kMaxGroups + 1;
  const bool dense = p.gs.sched == kDense;
  if (mode == HQ_MXFP8) {
    if (bn == 256) return dense ? run_bs<HQ_MXFP8, 256, 4, 1, 0>(a, b, p, sm_count, pdl, st)
                                : run_bs<HQ_MXFP8, 256, 4, 1, T>(a, b, p, sm_count, pdl, st);
    return dense ? run_bs<HQ_MXFP8, 128, 6, 2, 0>(a, b, p, sm_count, pdl, st)
                 : run_bs<HQ_MXFP8, 128, 6, 2, T>(a, b, p, sm_count, pdl, st);
  }
  if (mode == HQ_MXFP4) {
    if (bn == 256) return dense ? run_bs<HQ_MXFP4, 256, 4, 1, 0>(a, b, p, sm_count, pdl, st)
                                : run_bs<HQ_MXFP4, 256, 3, 1, T>(a, b, p, sm_count, pdl, st);
    return dense ? run_bs<HQ_MXFP4, 128, 5, 2, 0>(a, b, p, sm_count, pdl, st)
                 : run_bs<HQ_MXFP4, 128, 5, 2, T>(a, b, p, sm_count, pdl, st);
  }
  if (bn == 256) return dense ? run_bs<HQ_NVFP4, 256, 4, 1, 0>(a, b, p, sm_count, pdl, st)
                              : run_bs<HQ_NVFP4, 256, 3, 1, T>(a, b, p, sm_count, pdl, st);
  return dense ? run_bs<HQ_NVFP4, 128, 5, 2, 0>(a, b, p, sm_count, pdl, st)
               : run_bs<HQ_NVFP4, 128, 5, 2, T>(a, b, p, sm_count, pdl, st);
}

// Host-side checks shared by the three entry points.
// With discrete weights b and sfb are the device arrays of per-expert
// pointers (8-byte aligned); the pointers themselves are checked on the device.
int check_common(const void* a, const uint8_t* sfa, const void* b, const void* sfb,
                 const float* alpha, const hq_bf16* bias, const void* out, int64_t n, int64_t k,
                 hq_mode mode, bool discrete = false) {
  if (!valid_mode(mode)) return HQ_ERR_INVALID;
  const int64_t gs = mode == HQ_NVFP4 ? 16 : 32;
  if (n <= 0 || k <= 0 || k % (4 * gs) != 0 || n % 128 != 0) return HQ_ERR_INVALID;
  if (n > (1ll << 30) || k > (1ll << 30)) return HQ_ERR_INVALID;
  if (!a || !sfa || !b || !sfb || !out) return HQ_ERR_INVALID;
  if (!aligned16(a) || !aligned16(sfa) || !aligned16(out)) return HQ_ERR_INVALID;
  if (discrete ? ((reinterpret_cast<uintptr_t>(b) | reinterpret_cast<uintptr_t>(sfb)) & 7u) != 0
               : (!aligned16(b) || !aligned16(sfb)))
    return HQ_ERR_INVALID;
  if (bias && !aligned16(bias)) return HQ_ERR_INVALID;
  if (alpha && (reinterpret_cast<uintptr_t>(alpha) & 3u)) return HQ_ERR_INVALID;
  // HALOps "GEMM" API: alpha required for w4a4-nvfp4, not accepted for
  // w4a4-mxfp4; bias only in w8a8-mxfp8 mode
  if (mode == HQ_NVFP4 && !alpha) return HQ_ERR_UNSUPPORTED;
  if (mode == HQ_MXFP4 && alpha) return HQ_ERR_UNSUPPORTED;
  if (mode != HQ_MXFP8 && mode != HQ_MXFP8_E5M2 && bias) return HQ_ERR_UNSUPPORTED;
  return HQ_OK;
}

// ---------------------------------------------------------------------------
// Segment list for the per-row expert-id form of the contiguous GEMM (HALOps
// group_contiguous_gemm).  Row r is valid if 0 <= id[r] < L and (r == 0 or
// id[r] >= id[r - 1]); a segment is a maximal run of valid rows with one id
// inside one 128-row block.  One warp per block: lane l holds rows l + 32 j
// (j = 0..3); boundaries and starts come from ballots over the block's 128
// rows.  Pass 0 counts a block's segments, pass 1 writes them at the block's
// exclusive prefix (computed in between by seg_scan).
// Workspace: int32 [0] = segment count, [1..3] unused, then int4
// {row0, expert, first row - row0, end row - row0} per segment, then the
// per-block counts and prefixes.
// ---------------------------------------------------------------------------
struct SegParams {
  const int32_t* ids;
  int64_t M;
  int L;
  int64_t nblocks;
  int64_t cap;          // segment capacity of the list
  int32_t* ws;          // header + list
  int32_t* blk_count;   // [nblocks]
  int32_t* blk_base;    // [nblocks]
  uint32_t* status;
};

template <int PASS>
__global__ void __launch_bounds__(256) seg_build(const SegParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (b >= p.nblocks) return;
  const int64_t r0 = b * kBM;
  uint32_t valid_m[4], start_m[4];
  int id_of[4], prev_of[4];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int64_t r = r0 + lane + 32 * j;
    const bool in = r < p.M;
    const int id = in ? __ldg(p.ids + r) : -1;
    const int prev = (in && r > 0) ? __ldg(p.ids + r - 1) : -1;
    const bool v = in && id >= 0 && id < p.L && (r == 0 || id >= prev);
    if (in && !v) bad = true;
    valid_m[j] = __ballot_sync(0xFFFFFFFFu, v);
    id_of[j] = id;
    prev_of[j] = prev;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // a valid row starts a segment unless the row before it, in this block,
    // is valid with the same id
    const bool v = (valid_m[j] >> lane) & 1u;
    const bool prev_valid = lane > 0 ? ((valid_m[j] >> (lane - 1)) & 1u)
                                     : (j > 0 ? ((valid_m[j - 1] >> 31) & 1u) : false);
    const bool st = v && (!prev_valid || prev_of[j] != id_of[j]);
    start_m[j] = __ballot_sync(0xFFFFFFFFu, st);
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && PASS == 0) atomicOr(p.status, HQ_STATUS_BAD_OFFSETS);
  const int count = __popc(start_m[0]) + __popc(start_m[1]) + __popc(start_m[2]) + __popc(start_m[3]);
  if (PASS == 0) {
    if (lane == 0) p.blk_count[b] = count;
    return;
  }
  // boundary = a start or an invalid row: a segment ends at the next boundary
  uint32_t bnd[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) bnd[j] = start_m[j] | ~valid_m[j];
  int k = p.blk_base[b];
  int4* list = reinterpret_cast<int4*>(p.ws) + 1;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const bool st = (start_m[j] >> lane) & 1u;
    // rank of this start within the block
    int rank = __popc(start_m[j] & ((1u << lane) - 1u));
    for (int jj = 0; jj < j; ++jj) rank += __popc(start_m[jj]);
    if (st) {
      const int s = lane + 32 * j;
      int e = kBM;  // first boundary row after s
      for (int w = s + 1; w < kBM; ++w)
        if ((bnd[w >> 5] >> (w & 31)) & 1u) { e = w; break; }
      const int64_t slot = static_cast<int64_t>(k) + rank;
      if (slot < p.cap)
        list[slot] = make_int4(static_cast<int>(r0), id_of[j], s, e);
    }
  }
}

__global__ void __launch_bounds__(1024) seg_scan(const SegParams p) {
  // single CTA: exclusive prefix of the per-block counts, in chunks of 1024
  __shared__ int32_t part[32];
  int64_t carry = 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t base = 0; base < p.nblocks; base += 1024) {
    const int64_t b = base + threadIdx.x;
    const int32_t c = b < p.nblocks ? p.blk_count[b] : 0;
    int32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) part[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int32_t v = part[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t u = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o) v += u;
      }
      part[lane] = v;  // inclusive prefix of warp totals
    }
    __syncthreads();
    const int32_t warp_off = warp > 0 ? part[warp - 1] : 0;
    if (b < p.nblocks) p.blk_base[b] = static_cast<int32_t>(carry + warp_off + incl - c);
    carry += part[31];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    int64_t total = carry;
    if (total > p.cap) {
      atomicOr(p.status, HQ_STATUS_BAD_OFFSETS);
      total = p.cap;
    }
    p.ws[0] = static_cast<int32_t>(total);
  }
}

GemmParams base_params(const uint8_t* sfa, const uint8_t* sfb, const float* alpha,
                       const hq_bf16* bias, hq_bf16* out, int64_t n, int64_t k, hq_mode mode) {
  GemmParams p{};
  const int64_t gs = mode == HQ_NVFP4 ? 16 : 32;
  p.sfa = sfa;
  p.sfb = sfb;
  p.alpha = alpha;
  p.bias = bias;
  p.out = out;
  p.n = n;
  p.k = k;
  p.S = k / gs;
  p.sfb_group_bytes = (n + 127) / 128 * 128 * (k / gs);
  p.gs.status = status_word_ptr();
  p.wait_limit_ns = wait_limit_ns();
  p.inject_skip = fault_injection_stage();
  p.idesc_ab = mode == HQ_MXFP8_E5M2 ? ((1u << 7) | (1u << 10)) : 0u;
  p.d_type = kDBf16;
  return p;
}

// Points p at per-expert weights: the tensor maps and flags go to the start
// of the caller's workspace (checked by the caller to hold
// discrete_maps_bytes(L) bytes, 256-byte aligned).
void set_discrete(GemmParams& p, const int64_t* b_ptrs, const int64_t* sfb_ptrs, void* workspace,
                  int L) {
  p.b_ptrs = b_ptrs;
  p.sfb_ptrs = sfb_ptrs;
  p.b_maps = static_cast<CUtensorMap*>(workspace);
  p.w_ok = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) +
                                      static_cast<size_t>(L) * sizeof(CUtensorMap));
}

bool workspace_ok(const void* ws, size_t ws_bytes, size_t need) {
  return ws && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0 && ws_bytes >= need;
}

// Block-scaled grouped GEMM + dGLU backward, stacked (b, sfb) or discrete
// (b_ptrs, sfb_ptrs) weights.
int dglu_bs_impl(const void* a, const uint8_t* sfa, const void* b, const uint8_t* sfb,
                 const int64_t* b_ptrs, const int64_t* sfb_ptrs, const hq_bf16* c, const int32_t* padded_offsets, int L, const float* alpha,
                    const float* beta, const float* prob, int act, void* d_row, uint8_t* sfd_row,
                    void* d_col, uint8_t* sfd_col, const float* norm_const, float* dprob,
                    hq_bf16* dbias, float* amax, int64_t m, int64_t n, int64_t k, hq_mode mode,
                    int d_type, void* workspace, size_t ws_bytes, int sm_count, hq_stream_t s) {
  if (act != 0 && act != 1) return HQ_ERR_INVALID;
  if (!valid_mode(mode)) return HQ_ERR_INVALID;
  if (d_type != kDBf16 && d_type != kDF32 && d_type != kDE4M3 && d_type != kDE5M2) return HQ_ERR_INVALID;
  // FP8 D_row carries its SFD_row scales; BF16 and float32 D_row carry none
  const bool fp8_d = d_type == kDE4M3 || d_type == kDE5M2;
  if (fp8_d != (sfd_row != nullptr)) return HQ_ERR_INVALID;
  // cuDNN "Grouped GEMM + dGLU (SM100)", Additional Type Constraints: FP4
  // operands with 16-value scale groups and float32 D need the dbias path
  if (d_type == kDF32 && mode == HQ_NVFP4 && !dbias) return HQ_ERR_UNSUPPORTED;
  const int64_t gs = mode == HQ_NVFP4 ? 16 : 32;
  if (n <= 0 || k <= 0 || k % (4 * gs) != 0 || n % 128 != 0) return HQ_ERR_INVALID;
  if (n > (1ll << 28) || k > (1ll << 30)) return HQ_ERR_INVALID;
  if (m < 0 || m > (1ll << 31) - 256) return HQ_ERR_INVALID;
  if (L < 1 || L > kMaxGroups) return HQ_ERR_INVALID;
  const bool discrete = b_ptrs != nullptr;
  if (discrete ? (!sfb_ptrs || ((reinterpret_cast<uintptr_t>(b_ptrs) |
                                 reinterpret_cast<uintptr_t>(sfb_ptrs)) & 7u))
               : (!b || !sfb))
    return HQ_ERR_INVALID;
  if (!a || !sfa || !c || !padded_offsets || !alpha || !prob || !d_row || !dprob)
    return HQ_ERR_INVALID;
  if (act == 0 && !beta) return HQ_ERR_INVALID;
  if (!aligned16(a) || !aligned16(sfa) || (!discrete && (!aligned16(b) || !aligned16(sfb))) ||
      !aligned16(c) || !aligned16(d_row) || (sfd_row && !aligned16(sfd_row)))
    return HQ_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(padded_offsets) | reinterpret_cast<uintptr_t>(alpha) |
       reinterpret_cast<uintptr_t>(beta ? beta : alpha) | reinterpret_cast<uintptr_t>(prob) |
       reinterpret_cast<uintptr_t>(dprob) |
       reinterpret_cast<uintptr_t>(norm_const ? norm_const : alpha)) & 3u)
    return HQ_ERR_INVALID;
  if (norm_const && !sfd_row) return HQ_ERR_INVALID;  // norm_const belongs to the FP8 output
  if ((d_col != nullptr) != (sfd_col != nullptr) || (d_col && !sfd_row)) return HQ_ERR_INVALID;
  if (d_col && (!aligned16(d_col) || !aligned16(sfd_col))) return HQ_ERR_INVALID;
  if (amax && (reinterpret_cast<uintptr_t>(amax) & 3u)) return HQ_ERR_INVALID;
  // workspace: [per-expert tensor maps and flags (discrete weights)] [dbias sums]
  const size_t maps_bytes = discrete ? discrete_maps_bytes(L) : 0;
  if (dbias && (reinterpret_cast<uintptr_t>(dbias) & 1u)) return HQ_ERR_INVALID;
  if ((dbias || discrete) &&
      !workspace_ok(workspace, ws_bytes, maps_bytes + (dbias ? hq_gemm_dswiglu_workspace_size(L, n) : 0)))
    return HQ_ERR_INVALID;
  if (m == 0) return HQ_OK;
  GemmParams p = base_params(sfa, sfb, alpha, nullptr, nullptr, n, k, mode);
  if (discrete) set_discrete(p, b_ptrs, sfb_ptrs, workspace, L);
  void* dbias_ws = dbias ? static_cast<uint8_t*>(workspace) + maps_bytes : nullptr;
  if (!p.gs.status) return HQ_ERR_CUDA;
  p.gs.a_rows = m;
  p.gs.groups = L;
  p.gs.group_info = padded_offsets;
  p.gs.sched = kContig;
  p.c = c;
  p.beta = beta;
  p.prob = prob;
  p.dprob = dprob;
  p.dbias_ws = static_cast<float*>(dbias_ws);
  p.d_row = static_cast<uint8_t*>(d_row);
  p.sfd_row = sfd_row;
  p.norm_const = norm_const;
  p.d_col = static_cast<uint8_t*>(d_col);
  p.sfd_col = sfd_col;
  p.sfd_col_s = (m + 127) / 128 * 4;
  p.amax = amax;
  p.d_type = d_type;
  mode = kernel_mode(mode);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  // (zeroing the sums and the final dbias pass as programmatic dependents
  // of this kernel measured 5 us slower here than plain stream order)
  if (amax && cudaMemsetAsync(amax, 0, static_cast<size_t>(L) * 2 * sizeof(float), st) != cudaSuccess)
    return HQ_ERR_CUDA;
  const int64_t ws_count = static_cast<int64_t>(L) * 2 * n;
  if (dbias && cudaMemsetAsync(dbias_ws, 0, ws_count * sizeof(float), st) != cudaSuccess)
    return HQ_ERR_CUDA;
  const bool pdl = false;
  constexpr int T = kMaxGroups + 1;
  int rc;
  if (mode == HQ_MXFP8)
    // MXFP8 with dbias: the MMA thread copies the scales (two atoms per
    // k-block), so the epilogue's column sums get 168 registers instead of 128
    if (dbias)
      rc = act == 0 ? run_bs<HQ_MXFP8, 128, 5, 2, T, kEpiDSwiGLU, 0>(a, b, p, sm_count, pdl, st)
                    : run_bs<HQ_MXFP8, 128, 5, 2, T, kEpiDGeGLU, 0>(a, b, p, sm_count, pdl, st);
    else
      rc = act == 0 ? run_bs<HQ_MXFP8, 128, 5, 2, T, kEpiDSwiGLU>(a, b, p, sm_count, pdl, st)
                    : run_bs<HQ_MXFP8, 128, 5, 2, T, kEpiDGeGLU>(a, b, p, sm_count, pdl, st);
  else if (mode == HQ_MXFP4)
    rc = act == 0 ? run_bs<HQ_MXFP4, 128, 5, 2, T, kEpiDSwiGLU>(a, b, p, sm_count, pdl, st)
                  : run_bs<HQ_MXFP4, 128, 5, 2, T, kEpiDGeGLU>(a, b, p, sm_count, pdl, st);
  else
    rc = act == 0 ? run_bs<HQ_NVFP4, 128, 5, 2, T, kEpiDSwiGLU>(a, b, p, sm_count, pdl, st)
                  : run_bs<HQ_NVFP4, 128, 5, 2, T, kEpiDGeGLU>(a, b, p, sm_count, pdl, st);
  if (rc != HQ_OK) return rc;
  if (dbias)
    return dbias_finalize(reinterpret_cast<uint16_t*>(dbias), static_cast<const float*>(dbias_ws),
                          ws_count, st);
  return HQ_OK;
}

}  // namespace
}  // namespace hq

extern "C" {

int hq_gemm_dense(const void* a, const uint8_t* sfa, const void* b, const uint8_t* sfb,
                  const float* alpha, const hq_bf16* bias, hq_bf16* out, int64_t m, int64_t n,
                  int64_t k, hq_mode mode, int sm_count, int use_pdl, hq_stream_t s) {
  int rc = hq::check_common(a, sfa, b, sfb, alpha, bias, out, n, k, mode);
  if (rc != HQ_OK) return rc;
  if (m < 0 || m > (1ll << 31) - 256) return HQ_ERR_INVALID;
  if (m == 0) return HQ_OK;
  hq::GemmParams p = hq::base_params(sfa, sfb, alpha, bias, out, n, k, mode);
  if (!p.gs.status) return HQ_ERR_CUDA;
  p.gs.a_rows = m;
  p.gs.groups = 1;
  p.gs.sched = hq::kDense;
  return hq::run_gemm(mode, a, b, p, sm_count, use_pdl != 0, reinterpret_cast<cudaStream_t>(s));
}

int hq_gemm_grouped_contig(const void* a, const uint8_t* sfa, const void* b, const uint8_t* sfb,
                           const int32_t* padded_offsets, int L, const float* alpha,
                           const hq_bf16* bias, hq_bf16* out, int64_t m_rows, int64_t n,
                           int64_t k, hq_mode mode, int sm_count, hq_stream_t s) {
  int rc = hq::check_common(a, sfa, b, sfb, alpha, bias, out, n, k, mode);
  if (rc != HQ_OK) return rc;
  if (!padded_offsets || L < 1 || L > hq::kMaxGroups) return HQ_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(padded_offsets) & 3u) return HQ_ERR_INVALID;
  if (m_rows < 0 || m_rows > (1ll << 31) - 256) return HQ_ERR_INVALID;
  if (m_rows == 0) return HQ_OK;
  hq::GemmParams p = hq::base_params(sfa, sfb, alpha, bias, out, n, k, mode);
  if (!p.gs.status) return HQ_ERR_CUDA;
  p.gs.a_rows = m_rows;
  p.gs.groups = L;
  p.gs.group_info = padded_offsets;
  p.gs.sched = hq::kContig;
  return hq::run_gemm(mode, a, b, p, sm_count, false, reinterpret_cast<cudaStream_t>(s));
}

int hq_gemm_grouped_contig_discrete(const void* a, const uint8_t* sfa, const int64_t* b_ptrs,
                                    const int64_t* sfb_ptrs, const int32_t* padded_offsets, int L,
                                    const float* alpha, const hq_bf16* bias, hq_bf16* out,
                                    int64_t m_rows, int64_t n, int64_t k, hq_mode mode,
                                    void* workspace, size_t ws_bytes, int sm_count, hq_stream_t s) {
  int rc = hq::check_common(a, sfa, b_ptrs, sfb_ptrs, alpha, bias, out, n, k, mode, true);
  if (rc != HQ_OK) return rc;
  if (!padded_offsets || L < 1 || L > hq::kMaxGroups) return HQ_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(padded_offsets) & 3u) return HQ_ERR_INVALID;
  if (m_rows < 0 || m_rows > (1ll << 31) - 256) return HQ_ERR_INVALID;
  if (!hq::workspace_ok(workspace, ws_bytes, hq::discrete_maps_bytes(L))) return HQ_ERR_INVALID;
  if (m_rows == 0) return HQ_OK;
  hq::GemmParams p = hq::base_params(sfa, nullptr, alpha, bias, out, n, k, mode);
  if (!p.gs.status) return HQ_ERR_CUDA;
  p.gs.a_rows = m_rows;
  p.gs.groups = L;
  p.gs.group_info = padded_offsets;
  p.gs.sched = hq::kContig;
  hq::set_discrete(p, b_ptrs, sfb_ptrs, workspace, L);
  return hq::run_gemm(mode, a, nullptr, p, sm_count, false, reinterpret_cast<cudaStream_t>(s));
}

int hq_gemm_grouped_contig_swiglu_quant(const void* a, const uint8_t* sfa, const void* b,
                                        const uint8_t* sfb, const int32_t* padded_offsets, int L,
                                        const float* alpha, int64_t m_rows, int64_t H, int64_t k,
                                        hq_mode mode, hq_mode out_mode, const float* global_scale,
                                        void* q_out, uint8_t* sf_out, int sm_count, hq_stream_t s) {
  if (H <= 0 || H % 128 != 0 || H > (1ll << 28)) return HQ_ERR_INVALID;
  int rc = hq::check_common(a, sfa, b, sfb, alpha, nullptr, static_cast<const hq_bf16*>(q_out), 2 * H,
                            k, mode);
  if (rc != HQ_OK) return rc;
  if (out_mode != HQ_MXFP8 && out_mode != HQ_NVFP4) return HQ_ERR_INVALID;
  if (out_mode == HQ_MXFP8 && global_scale) return HQ_ERR_UNSUPPORTED;
  if (!sf_out || !hq::aligned16(sf_out)) return HQ_ERR_INVALID;
  if (global_scale && (reinterpret_cast<uintptr_t>(global_scale) & 3u)) return HQ_ERR_INVALID;
  if (!padded_offsets || L < 1 || L > hq::kMaxGroups) return HQ_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(padded_offsets) & 3u) return HQ_ERR_INVALID;
  if (m_rows < 0 || m_rows > (1ll << 31) - 256) return HQ_ERR_INVALID;
  if (m_rows == 0) return HQ_OK;
  hq::GemmParams p = hq::base_params(sfa, sfb, alpha, nullptr, nullptr, 2 * H, k, mode);
  if (!p.gs.status) return HQ_ERR_CUDA;
  mode = hq::kernel_mode(mode);
  p.n = H;  // compact columns; the B scale blocks stay those of 2H rows
  p.gs.a_rows = m_rows;
  p.gs.groups = L;
  p.gs.group_info = padded_offsets;
  p.gs.sched = hq::kContig;
  p.q = static_cast<uint8_t*>(q_out);
  p.sfq = sf_out;
  p.sfq_cols = out_mode == HQ_MXFP8 ? (H + 511) / 512 * 16 : H / 16;
  p.q_mode = out_mode;
  p.q_gscale = global_scale;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  constexpr int T = hq::kMaxGroups + 1;
  constexpr int E = hq::kEpiSwiGLUQ;
  if (hq::use_2sm() && hq::forced_tile_n() == 0) {
    // two-CTA pairs: the even CTA holds the gate rows, the odd CTA the up rows
    if (mode == HQ_MXFP8) return hq::run_bs_2sm<HQ_MXFP8, 6, E>(a, b, p, sm_count, false, st);
    if (mode == HQ_MXFP4) return hq::run_bs_2sm<HQ_MXFP4, 5, E>(a, b, p, sm_count, false, st);
    return hq::run_bs_2sm<HQ_NVFP4, 5, E>(a, b, p, sm_count, false, st);
  }
  if (mode == HQ_MXFP8) return hq::run_bs<HQ_MXFP8, 256, 4, 1, T, E>(a, b, p, sm_count, false, st);
  if (mode == HQ_MXFP4) return hq::run_bs<HQ_MXFP4, 256, 3, 1, T, E>(a, b, p, sm_count, false, st);
  return hq::run_bs<HQ_NVFP4, 256, 3, 1, T, E>(a, b, p, sm_count, false, st);
}

int hq_gemm_dglu_bs(const void* a, const uint8_t* sfa, const void* b, const uint8_t* sfb,
                    const hq_bf16* c, const int32_t* padded_offsets, int L, const float* alpha,
                    const float* beta, const float* prob, int act, void* d_row, uint8_t* sfd_row,
                    void* d_col, uint8_t* sfd_col, const float* norm_const, float* dprob,
                    hq_bf16* dbias, float* amax, int64_t m, int64_t n, int64_t k, hq_mode mode,
                    void* workspace, size_t ws_bytes, int sm_count, hq_stream_t s) {
  return hq::dglu_bs_impl(a, sfa, b, sfb, nullptr, nullptr, c, padded_offsets, L, alpha, beta, prob,
                          act, d_row, sfd_row, d_col, sfd_col, norm_const, dprob, dbias, amax, m, n,
                          k, mode, sfd_row ? hq::kDE4M3 : hq::kDBf16, workspace, ws_bytes, sm_count, s);
}

int hq_gemm_dglu_bs_typed(const void* a, const uint8_t* sfa, const void* b, const uint8_t* sfb,
                          const hq_bf16* c, const int32_t* padded_offsets, int L, const float* alpha,
                          const float* beta, const float* prob, int act, void* d_row, uint8_t* sfd_row,
                          void* d_col, uint8_t* sfd_col, const float* norm_const, float* dprob,
                          hq_bf16* dbias, float* amax, int64_t m, int64_t n, int64_t k, hq_mode mode,
                          hq_dtype d_type, void* workspace, size_t ws_bytes, int sm_count, hq_stream_t s) {
  return hq::dglu_bs_impl(a, sfa, b, sfb, nullptr, nullptr, c, padded_offsets, L, alpha, beta, prob,
                          act, d_row, sfd_row, d_col, sfd_col, norm_const, dprob, dbias, amax, m, n,
                          k, mode, static_cast<int>(d_type), workspace, ws_bytes, sm_count, s);
}

int hq_gemm_dglu_bs_discrete(const void* a, const uint8_t* sfa, const int64_t* b_ptrs,
                             const int64_t* sfb_ptrs, const hq_bf16* c,
                             const int32_t* padded_offsets, int L, const float* alpha,
                             const float* beta, const float* prob, int act, void* d_row,
                             uint8_t* sfd_row, void* d_col, uint8_t* sfd_col,
                             const float* norm_const, float* dprob, hq_bf16* dbias, float* amax,
                             int64_t m, int64_t n, int64_t k, hq_mode mode, void* workspace,
                             size_t ws_bytes, int sm_count, hq_stream_t s) {
  if (!b_ptrs) return HQ_ERR_INVALID;
  return hq::dglu_bs_impl(a, sfa, nullptr, nullptr, b_ptrs, sfb_ptrs, c, padded_offsets, L, alpha,
                          beta, prob, act, d_row, sfd_row, d_col, sfd_col, norm_const, dprob, dbias,
                          amax, m, n, k, mode, sfd_row ? hq::kDE4M3 : hq::kDBf16, workspace, ws_bytes,
                          sm_count, s);
}

size_t hq_gemm_grouped_rows_workspace_size(int64_t m_rows, int L) {
  if (m_rows < 0 || L < 1) return 0;
  const size_t nblocks = static_cast<size_t>((m_rows + hq::kBM - 1) / hq::kBM);
  const size_t cap = 2 * nblocks + static_cast<size_t>(L);
  const size_t bytes = 16 + 16 * cap + 8 * nblocks;
  return (bytes + 255) / 256 * 256;
}

int hq_gemm_grouped_rows(const void* a, const uint8_t* sfa, const void* b, const uint8_t* sfb,
                         const int32_t* expert_ids, int L, const float* alpha, const hq_bf16* bias,
                         hq_bf16* out, int64_t m_rows, int64_t n, int64_t k, hq_mode mode,
                         void* workspace, size_t ws_bytes, int sm_count, hq_stream_t s) {
  int rc = hq::check_common(a, sfa, b, sfb, alpha, bias, out, n, k, mode);
  if (rc != HQ_OK) return rc;
  if (!expert_ids || L < 1 || L > hq::kMaxGroups) return HQ_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(expert_ids) & 3u) return HQ_ERR_INVALID;
  if (m_rows < 0 || m_rows > (1ll << 31) - 256) return HQ_ERR_INVALID;
  if (m_rows == 0) return HQ_OK;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      ws_bytes < hq_gemm_grouped_rows_workspace_size(m_rows, L))
    return HQ_ERR_INVALID;
  hq::GemmParams p = hq::base_params(sfa, sfb, alpha, bias, out, n, k, mode);
  if (!p.gs.status) return HQ_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  hq::SegParams sp{};
  sp.ids = expert_ids;
  sp.M = m_rows;
  sp.L = L;
  sp.nblocks = (m_rows + hq::kBM - 1) / hq::kBM;
  sp.cap = 2 * sp.nblocks + L;
  sp.ws = static_cast<int32_t*>(workspace);
  sp.blk_count = sp.ws + 4 + 4 * sp.cap;
  sp.blk_base = sp.blk_count + sp.nblocks;
  sp.status = p.gs.status;
  const unsigned grid = static_cast<unsigned>((sp.nblocks * 32 + 255) / 256);
  hq::seg_build<0><<<grid, 256, 0, st>>>(sp);
  hq::seg_scan<<<1, 1024, 0, st>>>(sp);
  hq::seg_build<1><<<grid, 256, 0, st>>>(sp);
  if (cudaGetLastError() != cudaSuccess) return HQ_ERR_CUDA;
  p.gs.a_rows = m_rows;
  p.gs.groups = L;
  p.gs.group_info = sp.ws;
  p.gs.sched = hq::kSegments;
  return hq::run_gemm(mode, a, b, p, sm_count, false, st);
}

int hq_gemm_grouped_masked(const void* a, const uint8_t* sfa, const void* b, const uint8_t* sfb,
                           const int32_t* masked_m, int E, int64_t max_m, const float* alpha,
                           const hq_bf16* bias, hq_bf16* out, int64_t n, int64_t k, hq_mode mode,
                           int sm_count, hq_stream_t s) {
  int rc = hq::check_common(a, sfa, b, sfb, alpha, bias, out, n, k, mode);
  if (rc != HQ_OK) return rc;
  if (!masked_m || E < 1 || E > hq::kMaxGroups) return HQ_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(masked_m) & 3u) return HQ_ERR_INVALID;
  if (max_m <= 0 || max_m % 128 != 0) return HQ_ERR_INVALID;
  if (static_cast<int64_t>(E) * max_m > (1ll << 31) - 256) return HQ_ERR_INVALID;
  hq::GemmParams p = hq::base_params(sfa, sfb, alpha, bias, out, n, k, mode);
  if (!p.gs.status) return HQ_ERR_CUDA;
  p.gs.a_rows = static_cast<int64_t>(E) * max_m;
  p.gs.groups = E;
  p.gs.group_info = masked_m;
  p.gs.max_m = max_m;
  p.gs.sched = hq::kMasked;
  return hq::run_gemm(mode, a, b, p, sm_count, false, reinterpret_cast<cudaStream_t>(s));
}

}  // extern "C"
