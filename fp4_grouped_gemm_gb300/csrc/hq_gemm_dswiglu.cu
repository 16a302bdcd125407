// hq_gemm_dswiglu.cu -- BF16 grouped GEMM fused with the dSwiGLU or clamped
// dGeGLU backward epilogue (cuDNN frontend "Grouped GEMM + dGLU (SM100)", BF16
// contract, act_func = "dswiglu" / "dgeglu"; B stacked [L, n, k] or one
// pointer per expert).  Shown for dSwiGLU:
//
//   R_g = alpha_g^2 A_g B_g^T  (tcgen05.mma kind::f16, BF16 x BF16 -> FP32 in TMEM)
//   X_g = beta_g C_g, split into alternating 32-column gate / input blocks
//   D_row[gate col]  = R prob input s (1 + gate (1 - s)),  s = sigmoid(gate)
//   D_row[input col] = R prob gate s
//   dprob[m]        += sum_j R gate s input
//   dbias[g, c]     += sum_{m in g} D_row[m, c]
//
// Persistent warp-specialised kernel: warp 0 streams A / B tiles with TMA into
// a ring of shared-memory stages, warp 1 issues the MMAs into one of two TMEM
// accumulators (so the epilogue of tile i overlaps the main loop of tile i+1),
// warps 2..9 run the epilogue (two per TMEM lane quarter, each owning two of
// the tile's four 32-column chunks).  A compact tile of 128 columns j maps to the
// 256 C / D_row columns [2 j0, 2 j0 + 256).  Each epilogue thread owns one
// row: it reads that row's C segment, writes its D_row segment, adds its
// dprob partial with one float atomic, and, when dbias is requested, the warp
// reduces its fp32 D values over its 32 rows with a butterfly of shuffles and
// adds the column sums to a float32 workspace with one atomic per column.  A final pass adds the workspace
// into the caller's BF16 dbias.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "hq_internal.h"
#include "hq_ptx.cuh"
#include "hq_sched.cuh"

namespace hq {
namespace {

constexpr int kEpiWarps = 8;      // two per TMEM lane quarter
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kBKElems = 64;      // BF16 elements of K per k-block (128 bytes)
constexpr int kAcc = 2;
constexpr int kABytes = kBM * kBKElems * 2;  // one k-block of A (16 KB)

constexpr int kEpiBytes = 32 * 128;          // one epilogue warp's C / D_row buffer
constexpr int kSmemMax = 232448;

// Tile and shared-memory plan: BN compact columns per 128-row tile (the
// accumulator is 128 x BN float32 in TMEM, two of them), KPS k-blocks per
// pipeline stage.  Operand bytes per FLOP fall with BN, and the copy engine's
// cost is per copy more than per byte: 128 x 256 tiles load a 16 KB A box
// and a 32 KB B box per stage, four deep; 128 x 128 tiles, when K is a whole
// number of k-blocks, two k-blocks of A and of B as one 32 KB box per operand
// (a view of the [rows, K] matrix with the k-block as its outer dimension),
// three deep; otherwise one 16 KB box each, four deep.  The group table
// (2 x (L + 1) int32) closes the block and is sized at launch.
template <int KPS, int BN>
struct DsCfg {
  static_assert(BN == 128 || (BN == 256 && KPS == 1), "tile plans");
  static constexpr int kBBytes = BN * kBKElems * 2;   // one k-block of B
  static constexpr int kTmemCols = kAcc * BN;
  // kind::f16 instruction descriptor: D f32, A/B bf16, K-major, M = 128, N = BN
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                     (static_cast<uint32_t>(BN >> 3) << 17) |
                                     (static_cast<uint32_t>(kBM >> 4) << 24);
  static constexpr int kStages = KPS == 1 ? 4 : 3;
  static constexpr int kAStage = KPS * kABytes;
  static constexpr int kBStage = KPS * kBBytes;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kAStage;
  static constexpr int kOffEpi = kOffB + kStages * kBStage;  // 1024-aligned (TMA swizzle)
  static constexpr int kOffBar = kOffEpi + kEpiWarps * kEpiBytes;
  static constexpr int kNumBars = 2 * kStages + 2 * kAcc + 1 + kEpiWarps;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffTable = kOffMisc + 16;
  // bytes for L groups (+1024: the dynamic block is aligned up to 1024 in the kernel)
  static constexpr int64_t smem_bytes(int L) { return kOffTable + 8 * (static_cast<int64_t>(L) + 1) + 1024; }
  static_assert(kOffEpi % 1024 == 0, "epilogue buffers 1024-aligned");
};
static_assert(DsCfg<1, 128>::smem_bytes(kMaxGroups) <= kSmemMax, "shared memory budget");

struct DsParams {
  GroupSched gs;
  const uint16_t* c;      // [m, 2n]
  const float* alpha;     // [L]
  const float* beta;      // [L]
  const float* prob;      // [m]
  uint16_t* d_row;        // [m, 2n]
  float* dprob;           // [m]
  float* dbias_ws;        // [L, 2n] float32 partial sums, or null
  int64_t n, k;
  uint64_t wait_limit_ns;
  // discrete weights: B of group g through b_maps[g] (built on the device
  // from per-expert pointers); w_ok[g] == 0: the expert is skipped
  CUtensorMap* b_maps;    // [L] or null (B stacked as [L, n, k])
  int32_t* w_ok;          // [L]
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

enum Act : int { kSwiGLU = 0, kGeGLU = 1 };

// dGLU of one 32-column chunk (compact columns [j0, j0 + 32)) for the calling
// thread's row: r holds the alpha_g^2-unscaled accumulator values (R = a2 r),
// cv the row's 32 gate then 32 input C values; produces the row's 32 gate and
// 32 input D values (float32) and its dprob partial.
template <int ACT>
__device__ __forceinline__ void dglu_row_math(const uint32_t (&r)[32], const uint4 (&cv)[8], float a2,
                                              float beta, float prob, float (&dg)[32], float (&di)[32],
                                              float& dprob_part) {
  // per element pair (2i, 2i+1), in packed f32x2 arithmetic; dprob is
  // accumulated pairwise and the two halves added at the end
  float dp0 = 0.0f, dp1 = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    // gate words cv[0..15], input words cv[16..31] (as 32-bit words)
    const uint32_t gw = reinterpret_cast<const uint32_t*>(cv)[i];
    const uint32_t iw = reinterpret_cast<const uint32_t*>(cv)[16 + i];
    float R0, R1, rp0, rp1;
    mul_f32x2(R0, R1, __uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), a2);
    mul_f32x2(rp0, rp1, R0, R1, prob);
    if (ACT == kSwiGLU) {
      float g0, g1, x0, x1;
      mul_f32x2(g0, g1, bf16_lo(gw), bf16_hi(gw), beta);
      mul_f32x2(x0, x1, bf16_lo(iw), bf16_hi(iw), beta);
      float s0, s1;
      sigmoid_x2(g0, g1, s0, s1);  // sigmoid(gate)
      float om0, om1, t0, t1, gs0, gs1, u0, u1;
      fma_f32x2(om0, om1, s0, s1, -1.0f, -1.0f, 1.0f, 1.0f);      // 1 - s
      fma_f32x2(t0, t1, g0, g1, om0, om1, 1.0f, 1.0f);            // 1 + gate (1 - s)
      mul2_f32x2(gs0, gs1, g0, g1, s0, s1);                       // gate s
      mul2_f32x2(u0, u1, rp0, rp1, x0, x1);                       // R prob input
      mul2_f32x2(u0, u1, u0, u1, s0, s1);
      mul2_f32x2(dg[2 * i], dg[2 * i + 1], u0, u1, t0, t1);
      mul2_f32x2(di[2 * i], di[2 * i + 1], rp0, rp1, gs0, gs1);
      float q0, q1;
      mul2_f32x2(q0, q1, R0, R1, gs0, gs1);
      fma_f32x2(dp0, dp1, q0, q1, x0, x1, dp0, dp1);             // += R gate s input
    } else {
      // clamped GeGLU: gate <= 7, up in [-7, 7], s = sigmoid(1.702 gate_c),
      // gradients kept at equality with the bounds, linear offset 1
      const float g0 = bf16_lo(gw), g1 = bf16_hi(gw);
      const float x0 = bf16_lo(iw), x1 = bf16_hi(iw);
      const float gc0 = fminf(g0, 7.0f), gc1 = fminf(g1, 7.0f);
      const float uc0 = fminf(fmaxf(x0, -7.0f), 7.0f), uc1 = fminf(fmaxf(x1, -7.0f), 7.0f);
      float kg0, kg1;
      mul_f32x2(kg0, kg1, gc0, gc1, 1.702f);
      float s0, s1;
      sigmoid_x2(kg0, kg1, s0, s1);
      float om0, om1, t0, t1, up0, up1, gs0, gs1, w0, w1, a0, a1, b0, b1;
      fma_f32x2(om0, om1, s0, s1, -1.0f, -1.0f, 1.0f, 1.0f);      // 1 - s
      fma_f32x2(t0, t1, kg0, kg1, om0, om1, 1.0f, 1.0f);          // 1 + 1.702 gate_c (1 - s)
      add_f32x2(up0, up1, uc0, uc1, 1.0f, 1.0f);                  // up_c + 1
      mul2_f32x2(gs0, gs1, gc0, gc1, s0, s1);                     // gate_c s
      mul2_f32x2(w0, w1, rp0, rp1, up0, up1);
      mul2_f32x2(w0, w1, w0, w1, s0, s1);
      mul2_f32x2(a0, a1, w0, w1, t0, t1);
      mul2_f32x2(b0, b1, rp0, rp1, gs0, gs1);
      dg[2 * i] = g0 <= 7.0f ? a0 : 0.0f;
      dg[2 * i + 1] = g1 <= 7.0f ? a1 : 0.0f;
      di[2 * i] = (x0 >= -7.0f && x0 <= 7.0f) ? b0 : 0.0f;
      di[2 * i + 1] = (x1 >= -7.0f && x1 <= 7.0f) ? b1 : 0.0f;
      float q0, q1;
      mul2_f32x2(q0, q1, R0, R1, gs0, gs1);
      fma_f32x2(dp0, dp1, q0, q1, up0, up1, dp0, dp1);           // += R gate_c s (up_c + 1)
    }
  }
  dprob_part = dp0 + dp1;
}

// Column sums of the warp's 32 rows by a butterfly reduce-scatter (afterwards
// lane l holds the sums of gate column l and input column l), added to the
// float32 dbias workspace with one atomic per column.
__device__ __forceinline__ void dbias_reduce(const DsParams& p, float (&dg)[32], float (&di)[32], int g,
                                             int64_t j0, int lane) {
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
  float* ws = p.dbias_ws + static_cast<int64_t>(g) * (2 * p.n) + 2 * j0;
  atomicAdd(ws + lane, dg[0]);
  atomicAdd(ws + 32 + lane, di[0]);
}

// A warp's 4 KB epilogue buffer holds 32 rows x 128 bytes (one chunk's C or
// D_row segment: 32 gate then 32 input BF16 values per row) in the TMA
// 128-byte swizzle: 16-byte unit u of row r sits at unit u ^ (r & 7), so the
// eight lanes of a 16-byte access phase, one row each, hit distinct banks.
__device__ __forceinline__ uint32_t epi_unit(uint32_t buf, int row, int u) {
  return buf + static_cast<uint32_t>(row) * 128u + (static_cast<uint32_t>(u ^ (row & 7)) << 4);
}

// One tile of the epilogue as this CTA sees it: its first row, the tile's
// first compact column, the group, and whether its rows are to be written
// (a pair's odd half past its group's end is not).
struct EpiTile {
  int64_t row0;
  int n0;
  int g;
  bool rows;
};

// The epilogue role of one warp (ew = warp - 2): it owns one TMEM lane
// quarter q and 32 rows of every tile, and BN / 64 of the quarter's BN / 32
// chunks of 32 compact columns.  Per chunk: the C segment [32 rows x 64
// values] arrives by TMA in the warp's buffer, each lane reads its row,
// computes its D_row segment and writes it back in place, and one TMA store
// writes the segment to D_row.  The next chunk's C load is issued once that
// store has read the buffer, so it overlaps the dbias reduction and the next
// accumulator wait.  Contiguous-schedule tiles are whole 128-row blocks
// (group ends are multiples of 128), so a warp writes all 32 rows or none.
// Tiles t0, t0 + stride, ... < total; decode(t) describes tile t; the
// accumulator of the i-th tile is a = i % 2 (TMEM columns a * BN), its
// "full" barrier tfull0 + 8 a, and release(a) hands it back.
template <int ACT, int BN, typename Decode, typename Release>
__device__ __forceinline__ void dglu_epilogue(const DsParams& p, const CUtensorMap* tmC,
                                              const CUtensorMap* tmD, int64_t t0, int64_t stride,
                                              int64_t total, Decode decode, uint32_t tfull0,
                                              Release release, uint32_t tmem_base, uint32_t eb,
                                              uint32_t cbar, const WaitCtx& wctx, int warp, int lane) {
  constexpr int kChunksPerWarp = BN / 64;
  const int q = warp & 3;                // TMEM lane quarter this warp may access
  const int cg = ((warp - 2) >> 2);      // the warp's chunks: cg * kChunksPerWarp + 0, 1, ...
  uint32_t c_phase = 0;
  bool c_pending = false;
  // launched as a programmatic dependent of the workspace zeroing: its
  // zeroes are visible before this warp's first dbias / dprob add
  pdl_wait();
  auto chunk_live = [&](const EpiTile& et, int c) -> bool {
    return et.rows && et.n0 + c * 32 < p.n && (!p.w_ok || __ldg(p.w_ok + et.g) != 0) &&
           // debug builds: the segment's rows, columns and group lie inside D_row / dbias
           in_bounds(et.row0 + q * 32 + 32 <= p.gs.a_rows && et.n0 + c * 32 + 32 <= p.n &&
                         et.g < p.gs.groups,
                     p.gs.status);
  };
  auto load_c = [&](const EpiTile& et, int c) {
    if (lane == 0) {
      bulk_wait_group_read0();  // the previous D store has read the buffer
      mbar_arrive_expect_tx(cbar, kEpiBytes);
      tma_load_2d(eb, tmC, cbar, static_cast<int32_t>(2 * (et.n0 + c * 32)),
                  static_cast<int32_t>(et.row0 + q * 32));
    }
    c_pending = true;
  };
  int acc = 0;
  uint32_t acc_phase = 0;
  int64_t t = t0;
  // a tile's per-row / per-group factors are loaded while the previous tile
  // is still being processed
  EpiTile et{0, 0, 0, false};
  float alpha = 0.0f, beta = 1.0f, prob = 0.0f;
  auto factors = [&](const EpiTile& e, float& al, float& be, float& pr) {
    al = __ldg(p.alpha + e.g);
    be = ACT == kSwiGLU ? __ldg(p.beta + e.g) : 1.0f;
    pr = e.rows ? __ldg(p.prob + e.row0 + q * 32 + lane) : 0.0f;
  };
  if (t < total) {
    et = decode(t);
    if (chunk_live(et, cg * kChunksPerWarp)) load_c(et, cg * kChunksPerWarp);
    factors(et, alpha, beta, prob);
  }
  bool ok = true;
  for (; ok && t < total; t += stride) {
    const int64_t row = et.row0 + q * 32 + lane;
    const float a2 = __fmul_rn(alpha, alpha);
    EpiTile en = et;
    float alpha_n = alpha, beta_n = beta, prob_n = prob;
#pragma unroll 1
    for (int cc = 0; cc < kChunksPerWarp; ++cc) {
      const int c = cg * kChunksPerWarp + cc;
      const int64_t j0 = et.n0 + c * 32;
      const bool live = chunk_live(et, c);
      if (cc == 0) {
        const bool w = wait_bounded(tfull0 + 8u * acc, acc_phase, wctx);
        if (!__all_sync(0xFFFFFFFFu, w)) { ok = false; break; }
        tc_fence_after();
      }
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + c * 32, r);
      tmem_ld_wait();
      if (cc == kChunksPerWarp - 1) {
        // the warp's last chunk is in registers: release the accumulator
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release(acc);
      }
      float dg[32], di[32], dprob_part = 0.0f;
      if (live) {
        const bool w = wait_bounded(cbar, c_phase, wctx);
        if (!__all_sync(0xFFFFFFFFu, w)) { ok = false; break; }
        c_pending = false;
        c_phase ^= 1u;
        uint4 cv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t v[4];
          lds128(epi_unit(eb, lane, i), v);
          cv[i] = make_uint4(v[0], v[1], v[2], v[3]);
        }
        dglu_row_math<ACT>(r, cv, a2, beta, prob, dg, di, dprob_part);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t w4[4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // units 0..3: gate values 8i.., units 4..7: input values
            const float* src = i < 4 ? dg : di;
            const int e = (i & 3) * 8 + 4 * h;
            __nv_bfloat162 b0 = __floats2bfloat162_rn(src[e], src[e + 1]);
            __nv_bfloat162 b1 = __floats2bfloat162_rn(src[e + 2], src[e + 3]);
            w4[2 * h] = *reinterpret_cast<uint32_t*>(&b0);
            w4[2 * h + 1] = *reinterpret_cast<uint32_t*>(&b1);
          }
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(epi_unit(eb, lane, i)),
                       "r"(w4[0]), "r"(w4[1]), "r"(w4[2]), "r"(w4[3])
                       : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(tmD, eb, static_cast<int32_t>(2 * j0), static_cast<int32_t>(et.row0 + q * 32));
          bulk_commit_group();
        }
      }
      // the next C segment this warp reads: its next chunk of this tile, or
      // its first chunk of its next tile
      if (cc + 1 < kChunksPerWarp) {
        if (chunk_live(et, c + 1)) load_c(et, c + 1);
      } else if (t + stride < total) {
        en = decode(t + stride);
        if (chunk_live(en, cg * kChunksPerWarp)) load_c(en, cg * kChunksPerWarp);
        factors(en, alpha_n, beta_n, prob_n);
      }
      if (live) {
        atomicAdd(p.dprob + row, dprob_part);
        if (p.dbias_ws) dbias_reduce(p, dg, di, et.g, j0, lane);
      }
    }
    if (!ok) break;
    if (++acc == kAcc) { acc = 0; acc_phase ^= 1u; }
    et = en;
    alpha = alpha_n;
    beta = beta_n;
    prob = prob_n;
  }
  // abort: a C load still in flight lands before the CTA exits; every TMA
  // store has completed before the CTA exits
  if (c_pending) wait_drain(cbar, c_phase, wctx.limit_ns);
  if (lane == 0) bulk_wait_group0();
}

template <int ACT, int KPS, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    dglu_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                const DsParams p) {
  using C = DsCfg<KPS, BN>;
  constexpr int kStages = C::kStages;
  constexpr int kBN = BN;
  constexpr int kBBytes = C::kBBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int32_t* tab0 = reinterpret_cast<int32_t*>(smem + C::kOffTable);
  int32_t* tab1 = tab0 + (p.gs.groups + 1);
  const uint32_t bar0 = sbase + C::kOffBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + kAcc + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 2 * kAcc);
  const uint32_t cbar0 = bar0 + 8u * (2 * kStages + 2 * kAcc + 1);  // one per epilogue warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  int64_t* total_mtiles_s = reinterpret_cast<int64_t*>(smem + C::kOffMisc + 8);

  if (warp == 0 && lane == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < kAcc; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    for (int w = 0; w < kEpiWarps; ++w) mbar_init(cbar0 + 8u * w, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmD);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 2) build_table(p.gs, tab0, tab1, lane, total_mtiles_s);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  Schedule sch;
  sch.n_tiles = static_cast<int>((p.n + kBN - 1) / kBN);
  sch.total_tiles = *total_mtiles_s * sch.n_tiles;
  sch.tab0 = tab0;
  sch.tab1 = tab1;
  const int num_kb = static_cast<int>((p.k + kBKElems - 1) / kBKElems);
  const int num_st = (num_kb + KPS - 1) / KPS;  // stages per tile (an odd tail k-block loads zeros)
  const WaitCtx wctx{p.gs.status, abort_flag, p.wait_limit_ns};

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, filled_mask = 0, last_parity = 0;
      bool ok = true;
      int map_g = -1;  // group whose discrete tensor map was last acquired
      for (int64_t t = blockIdx.x; ok && t < sch.total_tiles; t += gridDim.x) {
        const TileInfo ti = decode_tile(p.gs, sch, t, kBN);
        const CUtensorMap* mapB = &tmB;
        int32_t zb = ti.g;
        bool w_ok = true;
        if (p.b_maps) {
          mapB = p.b_maps + ti.g;
          zb = 0;
          w_ok = __ldg(p.w_ok + ti.g) != 0;
          if (ti.g != map_g) {
            tensormap_acquire(mapB);
            map_g = ti.g;
          }
        }
        for (int si = 0; si < num_st; ++si) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, wctx)) { ok = false; break; }
          // a skipped expert's stage holds stale B data; its results are never stored
          mbar_arrive_expect_tx(full_bar(stage), C::kAStage + (w_ok ? C::kBStage : 0u));
          const uint32_t dA = sbase + C::kOffA + stage * C::kAStage;
          const uint32_t dB = sbase + C::kOffB + stage * C::kBStage;
          if (KPS == 1) {
            tma_load_2d(dA, &tmA, full_bar(stage), si * kBKElems, static_cast<int32_t>(ti.row0));
            if (w_ok) tma_load_3d(dB, mapB, full_bar(stage), si * kBKElems, ti.n0, zb);
          } else {
            tma_load_3d(dA, &tmA, full_bar(stage), 0, static_cast<int32_t>(ti.row0), si * KPS);
            if (w_ok) tma_load_4d(dB, mapB, full_bar(stage), 0, ti.n0, si * KPS, zb);
          }
          filled_mask |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      for (int s = 0; s < kStages; ++s)
        if (filled_mask & (1u << s)) wait_drain(full_bar(s), (last_parity >> s) & 1u, p.wait_limit_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      // the tensor pipe keeps only about one MMA queued behind the executing
      // one: descriptors advance by constants and the MMAs are unrolled
      const uint64_t adesc0 = smem_desc_sw128(sbase + C::kOffA);
      const uint64_t bdesc0 = smem_desc_sw128(sbase + C::kOffB);
      for (int64_t t = blockIdx.x; ok && t < sch.total_tiles; t += gridDim.x) {
        if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, wctx)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kBN;
        for (int si = 0; si < num_st; ++si) {
          if (!wait_bounded(full_bar(stage), phase, wctx)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = adesc0 + static_cast<uint64_t>((stage * C::kAStage) >> 4);
          const uint64_t bd = bdesc0 + static_cast<uint64_t>((stage * C::kBStage) >> 4);
          const uint32_t acc0 = si > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < KPS; ++kk)  // k-block kk of the stage: 16 KB further on
#pragma unroll
            for (int j = 0; j < 4; ++j)  // 4 x K=16 per 128-byte swizzle row (32 bytes each)
              mma_bf16(d_tmem, ad + static_cast<uint64_t>((kk * kABytes) >> 4) + 2 * j,
                       bd + static_cast<uint64_t>((kk * kBBytes) >> 4) + 2 * j, C::kIdesc,
                       (kk > 0 || j > 0) ? 1u : acc0);
          tc_commit(empty_bar(stage));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));
        if (++acc == kAcc) { acc = 0; acc_phase ^= 1u; }
      }
      tc_commit(drain_bar);
      wait_drain(drain_bar, 0, p.wait_limit_ns);
    }
  } else {
    const int ew = warp - 2;
    auto decode = [&](int64_t t) -> EpiTile {
      const TileInfo ti = decode_tile(p.gs, sch, t, kBN);
      return EpiTile{ti.row0, ti.n0, ti.g, true};
    };
    auto release = [&](int a) { mbar_arrive(tempty_bar(a)); };
    dglu_epilogue<ACT, BN>(p, &tmC, &tmD, blockIdx.x, gridDim.x, sch.total_tiles, decode, tfull_bar(0),
                           release, tmem_base, sbase + C::kOffEpi + ew * kEpiBytes, cbar0 + 8u * ew, wctx,
                           warp, lane);
  }

  __syncthreads();
  pdl_launch_dependents();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Two-CTA pairs (tcgen05 cta_group::2): a cluster of two CTAs computes a
// 256 x 256 tile of one group.  Each CTA loads its 128 rows of A and its 128
// of the tile's 256 B rows per k-block (two k-blocks per stage, the
// shared-memory plan of the 128 x 128 two-k-block tiles), the even CTA issues
// M = 256, N = 256 MMAs over both CTAs' stages, and each CTA's TMEM receives
// its 128 rows x 256 columns, which its own epilogue warps drain.  Per SM
// this moves two thirds of the operand bytes of the 128 x 256 single-SM tile
// for the same FLOPs.  A group's pairs start at its first row; when a group
// holds an odd number of 128-row blocks its last pair's odd CTA has no rows:
// it loads no A and writes nothing.
// ---------------------------------------------------------------------------
constexpr uint32_t kPairIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(256 >> 3) << 17) |
                                (static_cast<uint32_t>(256 >> 4) << 24);

template <int ACT>
__global__ void __launch_bounds__(kThreads, 1)
    dglu_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                     const DsParams p) {
  using C = DsCfg<2, 128>;  // per CTA: 128 A rows and 128 B rows per k-block
  constexpr int kStages = C::kStages;
  constexpr int kTN = 256;  // tile columns
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  const bool leader = rank == 0;

  int32_t* tab0 = reinterpret_cast<int32_t*>(smem + C::kOffTable);
  int32_t* tab1 = tab0 + (p.gs.groups + 1);
  const uint32_t bar0 = sbase + C::kOffBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };                      // the pair's A, B (leader)
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };         // the leader's commit
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };     // the leader's commit
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + kAcc + a); };  // used in the leader
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 2 * kAcc);
  const uint32_t cbar0 = bar0 + 8u * (2 * kStages + 2 * kAcc + 1);  // one per epilogue warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  int64_t* total_pairs_s = reinterpret_cast<int64_t*>(smem + C::kOffMisc + 8);

  if (warp == 0 && lane == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < kAcc; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * kEpiWarps);  // every epilogue warp of both CTAs
    }
    mbar_init(drain_bar, 1);
    for (int w = 0; w < kEpiWarps; ++w) mbar_init(cbar0 + 8u * w, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmD);
  }
  if (warp == 1) {  // one warp in each CTA allocates, collectively for the pair
    tmem_alloc_2sm(smem_u32(tmem_slot), 512);
    tmem_relinquish_2sm();
  }
  if (warp == 2) {
    // tab0 = the sanitised group ends, tab1 = the exclusive prefix of each
    // group's 256-row pairs (both CTAs build the same table)
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

  const int n_tiles = static_cast<int>((p.n + kTN - 1) / kTN);
  const int64_t total = *total_pairs_s * n_tiles;
  const int64_t cluster_id = blockIdx.x >> 1;
  const int64_t num_clusters = gridDim.x >> 1;
  const int num_kb = static_cast<int>(p.k / kBKElems);  // K is a whole number of k-blocks
  const int num_st = (num_kb + 1) / 2;                  // an odd tail k-block loads zeros
  const WaitCtx wctx{p.gs.status, abort_flag, p.wait_limit_ns};
  struct PairTile {
    int64_t row0;  // this CTA's first row
    int n0;
    int g;
    bool valid0, valid1;  // the even / odd CTA's 128 rows belong to the group
  };
  auto pair_tile = [&](int64_t t) {
    PairTile pt;
    const int64_t mt = t / n_tiles;
    pt.n0 = static_cast<int>(t - mt * n_tiles) * kTN;
    int lo = 0, hi = p.gs.groups - 1;  // last group with prefix <= mt
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tab1[mid] <= mt) lo = mid; else hi = mid - 1;
    }
    pt.g = lo;
    const int64_t start = lo > 0 ? tab0[lo - 1] : 0;
    const int64_t base = start + (mt - tab1[lo]) * 256;
    const int64_t cnt = static_cast<int64_t>(tab0[lo]) - base;  // a multiple of 128, >= 128
    pt.valid0 = cnt > 0;
    pt.valid1 = cnt > 128;
    pt.row0 = base + rank * kBM;
    return pt;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, filled_mask = 0, last_parity = 0;
      bool ok = true;
      int map_g = -1;
      for (int64_t t = cluster_id; ok && t < total; t += num_clusters) {
        const PairTile pt = pair_tile(t);
        const CUtensorMap* mapB = &tmB;
        int32_t zb = pt.g;
        bool w_ok = true;
        if (p.b_maps) {
          mapB = p.b_maps + pt.g;
          zb = 0;
          w_ok = __ldg(p.w_ok + pt.g) != 0;
          if (pt.g != map_g) {
            tensormap_acquire(mapB);
            map_g = pt.g;
          }
        }
        const bool has_a = rank ? pt.valid1 : pt.valid0;
        // the even CTA's full barrier expects the bytes of both CTAs' copies
        const uint32_t pair_bytes = (pt.valid0 ? C::kAStage : 0u) + (pt.valid1 ? C::kAStage : 0u) +
                                    (w_ok ? 2u * C::kBStage : 0u);
        for (int si = 0; si < num_st; ++si) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, wctx)) { ok = false; break; }
          if (leader) mbar_arrive_expect_tx(full_bar(stage), pair_bytes);
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          if (has_a)
            tma_load_3d_pair(sbase + C::kOffA + stage * C::kAStage, &tmA, fb, 0,
                             static_cast<int32_t>(pt.row0), 2 * si);
          if (w_ok)
            tma_load_4d_pair(sbase + C::kOffB + stage * C::kBStage, mapB, fb, 0,
                             pt.n0 + static_cast<int>(rank) * 128, 2 * si, zb);
          filled_mask |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // the even CTA's full barriers count both CTAs' bytes, so its drain
      // covers the odd CTA's copies too (the odd CTA stays resident until the
      // final cluster barrier)
      if (leader)
        for (int s = 0; s < kStages; ++s)
          if (filled_mask & (1u << s)) wait_drain(full_bar(s), (last_parity >> s) & 1u, p.wait_limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      const uint64_t adesc0 = smem_desc_sw128(sbase + C::kOffA);
      const uint64_t bdesc0 = smem_desc_sw128(sbase + C::kOffB);
      for (int64_t t = cluster_id; ok && t < total; t += num_clusters) {
        if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, wctx)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kTN;
        for (int si = 0; si < num_st; ++si) {
          if (!wait_bounded(full_bar(stage), phase, wctx)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = adesc0 + static_cast<uint64_t>((stage * C::kAStage) >> 4);
          const uint64_t bd = bdesc0 + static_cast<uint64_t>((stage * C::kBStage) >> 4);
          const uint32_t acc0 = si > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)  // k-block kk of the stage: 16 KB further on
#pragma unroll
            for (int j = 0; j < 4; ++j)   // 4 x K=16 per 128-byte swizzle row
              mma_bf16_2sm(d_tmem, ad + static_cast<uint64_t>((kk * kABytes) >> 4) + 2 * j,
                           bd + static_cast<uint64_t>((kk * kABytes) >> 4) + 2 * j, kPairIdesc,
                           (kk > 0 || j > 0) ? 1u : acc0);
          tc_commit_2sm_mc(empty_bar(stage), 0x3);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit_2sm_mc(tfull_bar(acc), 0x3);
        if (++acc == kAcc) { acc = 0; acc_phase ^= 1u; }
      }
      tc_commit_2sm_mc(drain_bar, 0x1);
      wait_drain(drain_bar, 0, p.wait_limit_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int ew = warp - 2;
    auto decode = [&](int64_t t) -> EpiTile {
      const PairTile pt = pair_tile(t);
      return EpiTile{pt.row0, pt.n0, pt.g, rank ? pt.valid1 : pt.valid0};
    };
    auto release = [&](int a) { mbar_arrive_cluster_relaxed(mapa_shared(tempty_bar(a), 0)); };
    dglu_epilogue<ACT, kTN>(p, &tmC, &tmD, cluster_id, num_clusters, total, decode, tfull_bar(0), release,
                            tmem_base, sbase + C::kOffEpi + ew * kEpiBytes, cbar0 + 8u * ew, wctx, warp,
                            lane);
  }

  __syncthreads();
  pdl_launch_dependents();
  cluster_sync();  // the peer may still read this CTA's shared memory and TMEM until here
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_2sm(tmem_base, 512);
  }
}

// dbias[i] = bf16(float(dbias[i]) + ws[i])
__global__ void dbias_finalize_kernel(uint16_t* dbias, const float* ws, int64_t count) {
  pdl_wait();  // the dGLU kernel's sums are complete and visible
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float v = __fadd_rn(__uint_as_float(static_cast<uint32_t>(dbias[i]) << 16), ws[i]);
    __nv_bfloat16 b = __float2bfloat16_rn(v);
    dbias[i] = *reinterpret_cast<uint16_t*>(&b);
  }
}

__global__ void zero_floats_kernel(float* a, int64_t na, float* b, int64_t nb) {
  pdl_launch_dependents();  // the dGLU kernel may start; it waits for these zeroes before adding
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nt = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = tid; i < na; i += nt) a[i] = 0.0f;
  for (int64_t i = tid; i < nb; i += nt) b[i] = 0.0f;
}

}  // namespace

int dbias_finalize(uint16_t* dbias, const float* ws, int64_t count, cudaStream_t st, bool pdl) {
  const int sms = num_sms();
  if (sms <= 0) return HQ_ERR_CUDA;
  int64_t blocks = (count + 255) / 256;
  if (blocks > 4 * sms) blocks = 4 * sms;
  if (blocks < 1) blocks = 1;
  return launch(dbias_finalize_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, pdl, dbias, ws,
                count) == cudaSuccess
             ? HQ_OK
             : HQ_ERR_CUDA;
}

int zero_floats(float* a, int64_t na, float* b, int64_t nb, cudaStream_t st) {
  const int sms = num_sms();
  if (sms <= 0) return HQ_ERR_CUDA;
  const int64_t n = na > nb ? na : nb;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 2 * sms) blocks = 2 * sms;
  if (blocks < 1) blocks = 1;
  zero_floats_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(a, na, b, nb);
  return cudaGetLastError() == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
}

}  // namespace hq

extern "C" {

size_t hq_gemm_dswiglu_workspace_size(int L, int64_t n) {
  if (L < 1 || n <= 0) return 0;
  const size_t bytes = static_cast<size_t>(L) * static_cast<size_t>(2 * n) * sizeof(float);
  return (bytes + 255) / 256 * 256;
}

}  // extern "C"

namespace hq {

// ---------------------------------------------------------------------------
// N-major discrete BF16 weights (cuDNN frontend "Grouped GEMM + dGLU (SM100)",
// BF16 contract, discrete b_ptrs with b_major = "n"): expert g's B is stored
// [k, n] (n contiguous).  A transpose pass writes a K-major copy of each
// expert into the caller's workspace (coalesced reads along n and writes
// along k through a shared-memory tile) and the expert's pointer list, which
// the K-major discrete path then consumes.  An expert whose pointer is null
// or not 16-byte aligned gets pointer 0 (skipped downstream, flagged).
// ---------------------------------------------------------------------------
size_t nmajor_copy_bytes(int64_t n, int64_t k) {
  return (static_cast<size_t>(n) * static_cast<size_t>(k) * 2 + 255) / 256 * 256;
}

namespace {
constexpr int kTr = 64;  // transpose tile (elements per side)

__global__ void __launch_bounds__(256) nmajor_transpose_kernel(const int64_t* b_ptrs, uint16_t* copies,
                                                              int64_t* ptrs, int64_t n, int64_t k,
                                                              size_t copy_elems, uint32_t* status) {
  __shared__ uint16_t tile[kTr][kTr + 2];
  const int g = blockIdx.z;
  const uint64_t src_addr = static_cast<uint64_t>(__ldg(b_ptrs + g));
  const bool good = src_addr != 0 && (src_addr & 15u) == 0;
  uint16_t* dst = copies + static_cast<size_t>(g) * copy_elems;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    ptrs[g] = good ? static_cast<int64_t>(reinterpret_cast<uintptr_t>(dst)) : 0;
    if (!good) atomicOr(status, HQ_STATUS_BAD_POINTER);
  }
  if (!good) return;  // block-uniform
  const uint16_t* src = reinterpret_cast<const uint16_t*>(src_addr);
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kTr;  // source columns (n)
  const int64_t k0 = static_cast<int64_t>(blockIdx.y) * kTr;  // source rows (k)
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;     // 64 x 4 threads
  for (int r = ty; r < kTr; r += 4) {
    const int64_t kk = k0 + r, nn = n0 + tx;
    tile[r][tx] = (kk < k && nn < n) ? src[kk * n + nn] : 0;
  }
  __syncthreads();
  for (int r = ty; r < kTr; r += 4) {
    const int64_t nn = n0 + r, kk = k0 + tx;
    if (nn < n && kk < k) dst[nn * k + kk] = tile[tx][r];
  }
}
}  // namespace

int nmajor_to_kmajor(const int64_t* b_ptrs, uint16_t* copies, int64_t* ptrs, int L, int64_t n, int64_t k,
                     cudaStream_t st) {
  uint32_t* status = status_word_ptr();
  if (!status) return HQ_ERR_CUDA;
  const dim3 grid(static_cast<unsigned>((n + kTr - 1) / kTr), static_cast<unsigned>((k + kTr - 1) / kTr),
                  static_cast<unsigned>(L));
  if (grid.y > 65535u) return HQ_ERR_INVALID;
  nmajor_transpose_kernel<<<grid, 256, 0, st>>>(b_ptrs, copies, ptrs, n, k, nmajor_copy_bytes(n, k) / 2, status);
  return cudaGetLastError() == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
}

namespace {

// b: stacked weights [L, n, k]; or b == null and b_ptrs: one device pointer
// per expert (discrete weights), tensor maps built in the workspace's head.
template <int ACT>
int run_dglu(const hq_bf16* a, const hq_bf16* b, const int64_t* b_ptrs, const hq_bf16* c,
             const int32_t* padded_offsets, int L, const float* alpha, const float* beta,
             const float* prob, hq_bf16* d_row, float* dprob, hq_bf16* dbias, int64_t m, int64_t n,
             int64_t k, void* workspace, size_t ws_bytes, int sm_count, hq_stream_t s) {
  if (L < 1 || L > kMaxGroups) return HQ_ERR_INVALID;
  if (m < 0 || n <= 0 || k <= 0 || n % 32 != 0 || k % 8 != 0) return HQ_ERR_INVALID;
  if (m > (1ll << 31) - 256 || n > (1ll << 28) || k > (1ll << 30)) return HQ_ERR_INVALID;
  const bool discrete = b_ptrs != nullptr;
  if (!a || !(b || discrete) || !c || !padded_offsets || !alpha || !prob || !d_row || !dprob)
    return HQ_ERR_INVALID;
  if (ACT == kSwiGLU && !beta) return HQ_ERR_INVALID;
  if (!aligned16(a) || (!discrete && !aligned16(b)) || !aligned16(c) || !aligned16(d_row))
    return HQ_ERR_INVALID;
  if (discrete && (reinterpret_cast<uintptr_t>(b_ptrs) & 7u)) return HQ_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(padded_offsets) | reinterpret_cast<uintptr_t>(alpha) |
       reinterpret_cast<uintptr_t>(beta ? beta : alpha) | reinterpret_cast<uintptr_t>(prob) |
       reinterpret_cast<uintptr_t>(dprob)) & 3u)
    return HQ_ERR_INVALID;
  // workspace: [per-expert tensor maps and flags (discrete weights)] [dbias sums]
  const size_t maps_bytes = discrete ? discrete_maps_bytes(L) : 0;
  if (dbias && (reinterpret_cast<uintptr_t>(dbias) & 1u)) return HQ_ERR_INVALID;
  if (dbias || discrete) {
    const size_t need = maps_bytes + (dbias ? hq_gemm_dswiglu_workspace_size(L, n) : 0);
    if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
      return HQ_ERR_INVALID;
  }
  if (m == 0) return HQ_OK;
  void* dbias_ws = dbias ? static_cast<uint8_t*>(workspace) + maps_bytes : nullptr;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  DsParams p{};
  p.gs.group_info = padded_offsets;
  p.gs.a_rows = m;
  p.gs.groups = L;
  p.gs.sched = kContig;
  p.gs.status = status_word_ptr();
  if (!p.gs.status) return HQ_ERR_CUDA;
  p.c = c;
  p.alpha = alpha;
  p.beta = beta;
  p.prob = prob;
  p.d_row = d_row;
  p.dprob = dprob;
  p.dbias_ws = static_cast<float*>(dbias_ws);
  if (discrete) {
    p.b_maps = static_cast<CUtensorMap*>(workspace);
    p.w_ok = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) +
                                        static_cast<size_t>(L) * sizeof(CUtensorMap));
  }
  p.n = n;
  p.k = k;
  p.wait_limit_ns = wait_limit_ns();

  // Tile plan.  128 x 256 tiles move a quarter fewer operand bytes per FLOP
  // than 128 x 128 ones (measured 14% faster at n = 1408 although 9% of
  // their columns are padding), so they run unless they pad more than a
  // quarter beyond the 128-wide tiling or the group table does not fit.
  // Otherwise two k-blocks per stage when K is a whole number of at least
  // two k-blocks (the k-block view must not run past a row's end).
  // 256 x 256 tiles on CTA pairs halve the B bytes per SM again; they take
  // the two-k-block stages and run when the problem has at least a wave of
  // pairs (counting 256-row blocks of all m rows).
  const int64_t pad128 = (n + 127) / 128 * 128, pad256 = (n + 255) / 256 * 256;
  const int sms = num_sms();
  if (sms <= 0) return HQ_ERR_CUDA;
  int64_t cap = sm_count > 0 ? sm_count : sms;
  if (cap > sms) cap = sms;
  const bool kwhole = k % kBKElems == 0 && k >= 2 * kBKElems;
  const bool wide = 4 * pad256 <= 5 * pad128;
  const bool pair = wide && kwhole && cap >= 2 && DsCfg<2, 128>::smem_bytes(L) <= kSmemMax &&
                    ((m + 255) / 256) * (pad256 / 256) >= cap / 2;
  const bool wide1 = wide && !pair && DsCfg<1, 256>::smem_bytes(L) <= kSmemMax;
  const bool kb2 = (pair || !wide1) && kwhole && DsCfg<2, 128>::smem_bytes(L) <= kSmemMax;
  const int bn = wide1 ? 256 : 128;  // B box rows (a pair CTA loads 128 of its tile's 256)
  const uint64_t nkb = static_cast<uint64_t>(k / kBKElems);
  CUtensorMap tmA, tmB;
  {
    int rc;
    if (kb2) {
      // [rows, K] viewed as [k-block][row][64 elements]
      const uint64_t dims[3] = {kBKElems, static_cast<uint64_t>(m), nkb};
      const uint64_t strides[2] = {static_cast<uint64_t>(k) * 2, kBKElems * 2};
      const uint32_t box[3] = {kBKElems, kBM, 2};
      rc = encode_tensor_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<hq_bf16*>(a), dims,
                             strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    } else {
      const uint64_t dims[2] = {static_cast<uint64_t>(k), static_cast<uint64_t>(m)};
      const uint64_t strides[1] = {static_cast<uint64_t>(k) * 2};
      const uint32_t box[2] = {kBKElems, kBM};
      rc = encode_tensor_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<hq_bf16*>(a), dims,
                             strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (rc != HQ_OK) return rc;
  }
  {
    // discrete weights: a one-expert map encoded over the workspace (a valid
    // address, never loaded through as it stands) whose address the device
    // replaces per expert
    const uint64_t groups = static_cast<uint64_t>(discrete ? 1 : L);
    void* base = discrete ? workspace : const_cast<hq_bf16*>(b);
    int rc;
    if (kb2) {
      const uint64_t dims[4] = {kBKElems, static_cast<uint64_t>(n), nkb, groups};
      const uint64_t strides[3] = {static_cast<uint64_t>(k) * 2, kBKElems * 2,
                                   static_cast<uint64_t>(k) * 2 * n};
      const uint32_t box[4] = {kBKElems, 128, 2, 1};
      rc = encode_tensor_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    } else {
      const uint64_t dims[3] = {static_cast<uint64_t>(k), static_cast<uint64_t>(n), groups};
      const uint64_t strides[2] = {static_cast<uint64_t>(k) * 2, static_cast<uint64_t>(k) * 2 * n};
      const uint32_t box[3] = {kBKElems, static_cast<uint32_t>(bn), 1};
      rc = encode_tensor_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (rc != HQ_OK) return rc;
    if (discrete) {
      rc = build_weight_maps(tmB, b_ptrs, nullptr, p.b_maps, p.w_ok, L, st);
      if (rc != HQ_OK) return rc;
    }
  }
  // C and D_row [m, 2n]: the epilogue's 32-row x 64-value segments
  CUtensorMap tmC, tmD;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(2 * n), static_cast<uint64_t>(m)};
    const uint64_t strides[1] = {static_cast<uint64_t>(2 * n) * 2};
    const uint32_t box[2] = {64, 32};
    int rc = encode_tensor_map(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<hq_bf16*>(c), dims,
                               strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != HQ_OK) return rc;
    rc = encode_tensor_map(&tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d_row, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != HQ_OK) return rc;
  }
  // with dbias: zero the sums, then the dGLU kernel and the final pass as
  // programmatic dependents (each waits for its predecessor's results where
  // it needs them; the launches overlap)
  if (dbias) {
    const int rc = zero_floats(static_cast<float*>(dbias_ws), static_cast<int64_t>(L) * 2 * n, nullptr, 0, st);
    if (rc != HQ_OK) return rc;
  }
  const bool pdl = dbias != nullptr;
  if (set_smem_once<dglu_kernel<ACT, 1, 128>>(kSmemMax) != HQ_OK ||
      set_smem_once<dglu_kernel<ACT, 2, 128>>(kSmemMax) != HQ_OK ||
      set_smem_once<dglu_kernel<ACT, 1, 256>>(kSmemMax) != HQ_OK ||
      set_smem_once<dglu_pair_kernel<ACT>>(kSmemMax) != HQ_OK)
    return HQ_ERR_CUDA;
  if (pair) {
    int64_t pairs = cap / 2;
    const int64_t pairs_bound = ((m + 255) / 256) * (pad256 / 256);
    if (pairs > pairs_bound) pairs = pairs_bound;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(DsCfg<2, 128>::smem_bytes(L));
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
    if (cudaLaunchKernelEx(&cfg, dglu_pair_kernel<ACT>, tmA, tmB, tmC, tmD, p) != cudaSuccess)
      return HQ_ERR_CUDA;
  }
  const int64_t tiles_bound = ((m + kBM - 1) / kBM) * ((n + bn - 1) / bn);
  int64_t grid = cap;
  if (grid > tiles_bound) grid = tiles_bound;
  if (grid < 1) grid = 1;
  const dim3 g1(static_cast<unsigned>(grid));
  const cudaError_t le =
      pair ? cudaSuccess
      : wide1 ? launch(dglu_kernel<ACT, 1, 256>, g1, dim3(kThreads),
                    static_cast<int>(DsCfg<1, 256>::smem_bytes(L)), st, pdl, tmA, tmB, tmC, tmD, p)
      : kb2 ? launch(dglu_kernel<ACT, 2, 128>, g1, dim3(kThreads),
                     static_cast<int>(DsCfg<2, 128>::smem_bytes(L)), st, pdl, tmA, tmB, tmC, tmD, p)
            : launch(dglu_kernel<ACT, 1, 128>, g1, dim3(kThreads),
                     static_cast<int>(DsCfg<1, 128>::smem_bytes(L)), st, pdl, tmA, tmB, tmC, tmD, p);
  if (le != cudaSuccess) return HQ_ERR_CUDA;
  if (dbias) {
    const int rc = dbias_finalize(reinterpret_cast<uint16_t*>(dbias),
                                  static_cast<const float*>(dbias_ws),
                                  static_cast<int64_t>(L) * 2 * n, st, true);
    if (rc != HQ_OK) return rc;
  }
  return HQ_OK;
}

}  // namespace
}  // namespace hq

extern "C" {

int hq_gemm_dswiglu(const hq_bf16* a, const hq_bf16* b, const hq_bf16* c,
                    const int32_t* padded_offsets, int L, const float* alpha, const float* beta,
                    const float* prob, hq_bf16* d_row, float* dprob, hq_bf16* dbias, int64_t m,
                    int64_t n, int64_t k, void* workspace, size_t ws_bytes, int sm_count,
                    hq_stream_t s) {
  return hq::run_dglu<hq::kSwiGLU>(a, b, nullptr, c, padded_offsets, L, alpha, beta, prob, d_row, dprob,
                                   dbias, m, n, k, workspace, ws_bytes, sm_count, s);
}

int hq_gemm_dgeglu(const hq_bf16* a, const hq_bf16* b, const hq_bf16* c,
                   const int32_t* padded_offsets, int L, const float* alpha, const float* prob,
                   hq_bf16* d_row, float* dprob, hq_bf16* dbias, int64_t m, int64_t n, int64_t k,
                   void* workspace, size_t ws_bytes, int sm_count, hq_stream_t s) {
  return hq::run_dglu<hq::kGeGLU>(a, b, nullptr, c, padded_offsets, L, alpha, nullptr, prob, d_row, dprob,
                                  dbias, m, n, k, workspace, ws_bytes, sm_count, s);
}

size_t hq_gemm_dglu_discrete_nmajor_workspace_size(int L, int64_t n, int64_t k, int with_dbias) {
  if (L < 1 || n <= 0 || k <= 0) return 0;
  return static_cast<size_t>(L) * hq::nmajor_copy_bytes(n, k) + (static_cast<size_t>(L) * 8 + 255) / 256 * 256 +
         hq_gemm_discrete_workspace_size(L, with_dbias ? n : 0);
}

int hq_gemm_dglu_discrete_nmajor(const hq_bf16* a, const int64_t* b_ptrs, const hq_bf16* c,
                                 const int32_t* padded_offsets, int L, const float* alpha,
                                 const float* beta, const float* prob, int act, hq_bf16* d_row,
                                 float* dprob, hq_bf16* dbias, int64_t m, int64_t n, int64_t k,
                                 void* workspace, size_t ws_bytes, int sm_count, hq_stream_t s) {
  if (!b_ptrs || (reinterpret_cast<uintptr_t>(b_ptrs) & 7u)) return HQ_ERR_INVALID;
  if (act != 0 && act != 1) return HQ_ERR_INVALID;
  if (L < 1 || L > hq::kMaxGroups || n <= 0 || k <= 0 || n % 32 != 0 || k % 8 != 0) return HQ_ERR_INVALID;
  if (n > (1ll << 28) || k > (1ll << 30) || m < 0) return HQ_ERR_INVALID;
  const size_t need = hq_gemm_dglu_discrete_nmajor_workspace_size(L, n, k, dbias != nullptr);
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return HQ_ERR_INVALID;
  if (m == 0) return HQ_OK;
  // workspace: [K-major copies of the experts' weights] [their pointers]
  //            [the discrete path's tensor maps, flags and dbias sums]
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t copies = static_cast<size_t>(L) * hq::nmajor_copy_bytes(n, k);
  int64_t* ptrs = reinterpret_cast<int64_t*>(ws + copies);
  uint8_t* rest = ws + copies + (static_cast<size_t>(L) * 8 + 255) / 256 * 256;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  int rc = hq::nmajor_to_kmajor(b_ptrs, reinterpret_cast<uint16_t*>(ws), ptrs, L, n, k, st);
  if (rc != HQ_OK) return rc;
  return hq_gemm_dglu_discrete(a, ptrs, c, padded_offsets, L, alpha, beta, prob, act, d_row, dprob, dbias,
                               m, n, k, rest, ws_bytes - static_cast<size_t>(rest - ws), sm_count, s);
}

int hq_gemm_dglu_discrete(const hq_bf16* a, const int64_t* b_ptrs, const hq_bf16* c,
                          const int32_t* padded_offsets, int L, const float* alpha,
                          const float* beta, const float* prob, int act, hq_bf16* d_row,
                          float* dprob, hq_bf16* dbias, int64_t m, int64_t n, int64_t k,
                          void* workspace, size_t ws_bytes, int sm_count, hq_stream_t s) {
  if (!b_ptrs) return HQ_ERR_INVALID;
  if (act == 0)
    return hq::run_dglu<hq::kSwiGLU>(a, nullptr, b_ptrs, c, padded_offsets, L, alpha, beta, prob,
                                     d_row, dprob, dbias, m, n, k, workspace, ws_bytes, sm_count, s);
  if (act == 1)
    return hq::run_dglu<hq::kGeGLU>(a, nullptr, b_ptrs, c, padded_offsets, L, alpha, nullptr, prob,
                                    d_row, dprob, dbias, m, n, k, workspace, ws_bytes, sm_count, s);
  return HQ_ERR_INVALID;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant of hq_gemm_dswiglu.
//
// The dbias partial sums need float32 scratch.  hq_gemm_dswiglu takes it from
// the caller; this variant instead uses one fixed array in device global
// memory that belongs to the library, so a caller that cannot allocate device
// memory can still get dbias.  Every GPU that loads the library holds this
// array (1 MiB) until the process exits.
// ---------------------------------------------------------------------------
namespace hq {
namespace {

constexpr size_t kNoAllocScratchFloats = 262144;  // 1 MiB: L * 2n <= 262144

static __device__ __align__(256) float g_dswiglu_scratch[kNoAllocScratchFloats];

constexpr int kMaxDev = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDev] = {};
void* g_scratch_ctx[kMaxDev] = {};

// Device address of g_dswiglu_scratch on the current device.  Host code must
// not use the symbol itself (on the host it names a stand-in, not device
// memory); the address is resolved once per device, with that device current,
// and again if another context has become current on the device since.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  void* ctx = current_context();
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_dswiglu_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_addr[dev] = ptr;
    g_scratch_ctx[dev] = ctx;
  }
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace hq

extern "C" int hq_gemm_dswiglu_noalloc(const hq_bf16* a, const hq_bf16* b, const hq_bf16* c,
                                       const int32_t* padded_offsets, int L, const float* alpha,
                                       const float* beta, const float* prob, hq_bf16* d_row,
                                       float* dprob, hq_bf16* dbias, int64_t m, int64_t n,
                                       int64_t k, int sm_count, hq_stream_t s) {
  if (L < 1 || n <= 0) return HQ_ERR_INVALID;
  // L * 2n in unsigned arithmetic: no signed overflow for any n > 0
  if (dbias && static_cast<uint64_t>(L) * 2u * static_cast<uint64_t>(n) > hq::kNoAllocScratchFloats)
    return HQ_ERR_UNSUPPORTED;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  if (dbias) {
    ws = hq::scratch_address();
    if (!ws) return HQ_ERR_CUDA;
    ws_bytes = sizeof(float) * hq::kNoAllocScratchFloats;
  }
  // hq_gemm_dswiglu validates the rest and clears the used part of the
  // scratch on the stream before the GEMM accumulates into it.
  return hq_gemm_dswiglu(a, b, c, padded_offsets, L, alpha, beta, prob, d_row, dprob, dbias, m, n, k,
                         ws, ws_bytes, sm_count, s);
}
