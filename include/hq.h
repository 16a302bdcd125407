/*
 * hq.h -- C ABI of the block-scaled low-precision MoE GEMM library (libhq.so).
 *
 * One GB300 (sm_103a) hot path: a group-wise quantiser (BF16 -> MXFP8 / NVFP4
 * with scales in the 128x4 SfAtom layout), dense / grouped-contiguous /
 * grouped-masked block-scaled GEMMs with BF16 output, a fused SwiGLU +
 * requantisation pass, and a BF16 grouped GEMM fused with the dSwiGLU
 * backward (per-row dprob, per-expert dbias).
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - Every tensor argument is a DEVICE pointer into memory the caller owns and
 *    has allocated (outputs are pre-allocated and written in place, as the
 *    HALOps "GEMM" API does for every op: "Written in-place").  The library
 *    allocates no memory; where a call needs scratch space the caller passes
 *    it (sized by a *_workspace_size query), so it can be allocated before a
 *    CUDA-graph capture (FlashRT fp4-gemm notes, large-M tier workspace).
 *    Host memory is not a supported argument, pinned (cudaHostAlloc,
 *    cudaHostRegister) or pageable, even on a platform whose GPU can address
 *    it (coherent host links): the GEMMs read their operands through TMA
 *    tensor maps and the other kernels assume device-memory bandwidth and
 *    alignment.  The host does not check where a pointer points (that would
 *    cost a driver query per pointer and call); passing host memory is a
 *    precondition violation.  Move host data with cudaMemcpyAsync first.
 *  - Every call is asynchronous on the given stream (NULL = legacy default
 *    stream).  The library keeps no pointer after it returns, but every
 *    buffer must stay alive and unchanged until the stream reaches the work.
 *  - Every call validates its arguments on the host and returns a status
 *    BEFORE launching anything ("Unsupported calls raise before launch" --
 *    FlashRT fp4-gemm notes; "rejected before allocation or compilation" --
 *    cuDNN "Grouped GEMM + dGLU (SM100)", Backend dispatch).  On a non-zero
 *    status nothing was launched and no output was touched.
 *  - Values the host cannot see (device-resident offsets, masks, counts) are
 *    checked on the device: a violation is clamped to a safe value, the
 *    affected rows are skipped, and a bit is set in the device status word
 *    (read with hq_get_device_status).  A pipeline wait that exceeds the
 *    wait limit sets HQ_STATUS_WAIT_TIMEOUT and the kernel returns early
 *    instead of hanging.
 *  - Matrices are row-major.  A and B are K-major (the contiguous dimension is
 *    K); outputs are N-major.  FP8 data is one byte per element
 *    (float8_e4m3fn); FP4 data is packed E2M1, two elements per byte with the
 *    even element index in the low nibble, so an [r, k] FP4 matrix occupies
 *    r * k / 2 bytes.  BF16 values are passed as raw 16-bit patterns.
 *  - Scale factors: one byte per group of 32 (MXFP8, UE8M0 = power-of-two
 *    biased exponent) or 16 (NVFP4, UE4M3 = float8_e4m3fn bit pattern with a
 *    clear sign bit) consecutive K elements.  The swizzled layout is the
 *    "SfAtom 128x4" of the HALOps API (cuDNN shape (32, 4, ceil(R/128), 4,
 *    ceil(S/4), L)): for R rows and S = K / group scale columns the byte of
 *    (row r, column s) is at
 *        ((r / 128) * (S / 4) + s / 4) * 512
 *          + (r % 32) * 16 + ((r % 128) / 32) * 4 + (s % 4),
 *    the buffer holds ceil(R / 128) * 128 * S bytes, and expert-stacked weight
 *    scales place expert e at e * ceil(N / 128) * 128 * S.
 */
#ifndef HQ_H_
#define HQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle type as cudaStream_t / CUstream (NULL = legacy default stream). */
typedef struct CUstream_st *hq_stream_t;

/* A BF16 value as its raw bit pattern. */
typedef uint16_t hq_bf16;

/* Quantisation recipe ("mode" string of the HALOps API). */
typedef enum {
  HQ_MXFP8 = 0, /* "w8a8-mxfp8": E4M3 elements, UE8M0 scale per 32          */
  HQ_MXFP4 = 1, /* "w4a4-mxfp4": packed E2M1, UE8M0 scale per 32, no alpha  */
  HQ_NVFP4 = 2, /* "w4a4-nvfp4": packed E2M1, UE4M3 scale per 16, FP32 alpha */
  HQ_MXFP8_E5M2 = 3 /* MXFP8 with float8_e5m2 elements, UE8M0 scale per 32
                       (cuDNN "Grouped GEMM + dGLU (SM100)", Data Types) */
} hq_mode;

/* Return codes. */
enum {
  HQ_OK = 0,
  HQ_ERR_INVALID = 1,     /* null pointer, bad shape, stride or alignment      */
  HQ_ERR_UNSUPPORTED = 2, /* valid request this library does not implement    */
  HQ_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed                 */
  HQ_ERR_TIMEOUT = 4      /* device status reports an expired pipeline wait    */
};

/* Bits of the device status word. */
#define HQ_STATUS_WAIT_TIMEOUT 0x1u   /* a bounded mbarrier wait expired           */
#define HQ_STATUS_MASK_CLAMPED 0x2u   /* masked_m[e] outside [0, max_m]: clamped    */
#define HQ_STATUS_BAD_OFFSETS 0x4u    /* padded_offsets not monotone / 128-aligned /
                                         beyond the row count: rows skipped      */
#define HQ_STATUS_TOKENS_CLAMPED 0x8u /* token_nums[e] outside [0, rows/expert]    */
#define HQ_STATUS_ROUTING_DROPPED 0x10u /* permute: a bad expert id or a full expert */
#define HQ_STATUS_BAD_POINTER 0x20u   /* discrete weights: a null or unaligned
                                         per-expert pointer; that expert skipped */
#define HQ_STATUS_BOUNDS 0x40u        /* debug build only: a device bounds check on
                                         a global write failed; that write skipped */

/* Layout and alignment constants, so integrations need not copy them
 * (FlashRT fp4-gemm notes: "Read capabilities() instead of duplicating
 * scale-factor layout or alignment constants"). */
typedef struct {
  int abi_version;       /* 2                                               */
  int sfatom_rows;       /* 128 rows per atom                               */
  int sfatom_cols;       /* 4 scale columns per atom                        */
  int sfatom_bytes;      /* 512                                             */
  int group_mxfp8;       /* 32                                              */
  int group_nvfp4;       /* 16                                              */
  int contig_row_align;  /* 256: padded_offsets alignment the pages fix     */
  int tile_m;            /* 128: rows per GEMM tile (offsets must be multiples) */
  int ptr_align_bytes;   /* 16: every tensor base pointer                   */
  int max_groups;        /* 1024 experts at most                            */
  int glu_block;         /* 32: dGLU gate/input interleave width            */
  int group_mxfp4;       /* 32                                              */
} hq_capabilities_t;

/* Fills *out.  Returns HQ_ERR_INVALID if out is NULL. */
int hq_capabilities(hq_capabilities_t *out);

/* Human-readable name of a return code (static string, never NULL). */
const char *hq_status_string(int status);

/* Bytes of a scale buffer for `rows` rows of K = k elements in `mode`:
 * ceil(rows / 128) * 128 * (k / group).  Returns 0 if k is not a multiple of
 * 4 * group or mode is unknown. */
size_t hq_sf_bytes(int64_t rows, int64_t k, hq_mode mode);

/* Reads the device status word of the current device (after the work queued
 * on `s` completes: this call synchronises `s`) into *out; if clear != 0 the
 * word is reset to 0.  Returns HQ_ERR_TIMEOUT if HQ_STATUS_WAIT_TIMEOUT is
 * set, HQ_ERR_CUDA on a CUDA failure, else HQ_OK. */
int hq_get_device_status(uint32_t *out, int clear, hq_stream_t s);

/* Limit of every bounded pipeline wait inside the kernels, in nanoseconds
 * (default 1e9).  Applies to launches made after the call.  After a wait
 * expires the kernel still waits for its copies in flight, each such drain
 * wait bounded by the same limit, so an aborted launch can take several times
 * the limit before it returns. */
int hq_set_wait_limit_ns(uint64_t ns);

/* Self-test of the bounded wait: launches one CTA that waits on a pipeline
 * barrier nothing ever arrives on, with the given limit.  The wait expires,
 * HQ_STATUS_WAIT_TIMEOUT is set in the device status word and the kernel
 * returns; the context stays usable.  No GPU fault is involved. */
int hq_selftest_wait_expiry(uint64_t limit_ns, hq_stream_t s);

/* Test aid for the GEMMs' abort path (no counterpart on the pages): from
 * the next launch on, the two-CTA pair GEMM kernel's first cluster withholds
 * the arrival that completes its skip_stage-th operand stage (counted from 0
 * over the stages its producer issues), so the MMA issuer's bounded wait
 * expires: the kernel sets HQ_STATUS_WAIT_TIMEOUT, stops every role, drains
 * its copies and MMAs with bounded waits, frees TMEM and returns.  Tiles the
 * aborted cluster had not finished are not written; nothing outside the
 * output's valid rows is written.  -1 (the default) turns it off.  Nothing
 * faults or hangs: the failure is a barrier that nothing completes.
 * Returns HQ_ERR_INVALID for skip_stage < -1. */
int hq_set_fault_injection(int64_t skip_stage);

/* Debug build (libhq_debug.so: the same sources compiled with HQ_DEBUG=1;
 * a device-side check for the sanitizer the pool does not offer).  Its
 * kernels check the data-dependent indices of their global writes (output
 * rows and columns, scale-atom offsets, the dGLU dprob / dbias rows and the
 * TMA store coordinates, the permute's destination rows); a failed check sets
 * HQ_STATUS_BOUNDS in the device status word and skips that write instead of
 * trapping.  In the release library the checks compile to nothing.
 * hq_debug_build returns 1 in the debug library, 0 otherwise (no GPU needed).
 * hq_debug_selftest (debug library only) launches one thread that checks
 * index n against an n-element buffer: the check fails, the write is skipped
 * and HQ_STATUS_BOUNDS is set; read it with hq_get_device_status.  Returns
 * HQ_ERR_UNSUPPORTED in the release library, where it launches nothing. */
int hq_debug_build(void);
int hq_debug_selftest(hq_stream_t s);

/* Measurement aid for the HBM-bound passes (no counterpart on the pages): a
 * plain streaming kernel with the quantiser's byte ratio.  It reads `bytes`
 * from src (device memory, 16-byte aligned, bytes a multiple of 32) with
 * 16-byte loads, four 32-byte groups per thread in flight over 4 CTAs per SM,
 * and writes bytes / 4 to dst: per 32-byte group one 8-byte word, the XOR of
 * the group's two 16-byte halves (words 0^2 of each half, words 1^3).
 * bytes == 0 launches the same grid with no work.  Timed like a quantiser
 * launch it gives the floor that launch size allows: the quantiser's time
 * over it is the part the encoding adds.  Returns HQ_ERR_INVALID for a size
 * or alignment outside that contract. */
int hq_probe_stream(const void* src, size_t bytes, void* dst, hq_stream_t s);

/* Tensor-core issue-rate probe (a measurement aid, no counterpart on the
 * pages): every CTA of one wave (one per SM, or one two-CTA cluster per SM
 * pair when pair != 0) issues `iters` x 4 back-to-back tcgen05.mma of the
 * given kind from one thread into one TMEM accumulator, with the operands
 * resident in shared memory (M = 128 per SM, N = n, K = 16 for BF16, 32 for
 * MXFP8, 64 for NVFP4 / MXFP4; scales constant), and records per issuing CTA
 * the SM clock cycles and the nanoseconds of the timed MMAs.
 *   kind   0 kind::f16 (BF16), 1 kind::mxf8f6f4 (MXFP8),
 *          2 kind::mxf4nvf4 scale_vec::4X (NVFP4), 3 kind::mxf4 scale_vec::2X
 *   n      128 or 256
 *   out    device uint64 [2 * ctas]: out[2 i] = cycles, out[2 i + 1] = ns of
 *          issuing CTA i (ctas = the number of SMs, halved when pair != 0)
 * Cycles per MMA = cycles / (4 iters).  Returns HQ_ERR_INVALID for a bad
 * kind, n, iters outside [1, 1 << 20] or a null / unaligned out. */
int hq_probe_mma_rate(int kind, int pair, int n, int iters, uint64_t *out, hq_stream_t s);

/* Tuning knob: GEMM tile width in N for the block-scaled GEMMs (0 = choose
 * automatically, 128 or 256 = force a single-SM tile).  Applies to later
 * calls. */
int hq_set_gemm_tile_n(int tile_n);

/* Tuning knob for the pair tiles.  1 (default, the faster choice on GB300)
 * runs the dense, contiguous-grouped (padded_offsets), masked (max_m a
 * multiple of 256) and fused up-proj block-scaled GEMMs on pairs of SMs: a
 * two-CTA cluster computing 256-row tiles with cta_group::2 MMAs, which cuts
 * the operand bytes each SM loads per FLOP.  Tiles are 256 columns wide, or
 * 384 (an N = 256 and an N = 128 MMA per K step) for dense GEMMs whose n is a
 * multiple of 384.  256 or 384 forces that width where n allows it; 0 keeps
 * every GEMM on single-SM tiles.  Other values: HQ_ERR_INVALID.  Applies to
 * later calls. */
int hq_set_gemm_2sm(int enable);

/* ------------------------------------------------------------------------- *
 * Group-wise quantiser
 *
 * HALOps "GEMM" API, group_wise_quant: quantises a 2-D BF16 tensor per group
 * along K and returns the data and the block scales (SfAtom layout when
 * use_swizzle, plain row-major otherwise).  Scale rule (cuDNN "Grouped GEMM +
 * dGLU (SM100)", Step 3): SF = norm_const * amax(group) * rcp_max,
 * q = x * norm_const / SF, with norm_const = *global_scale (NVFP4; 1 when
 * NULL) or 1 (MXFP8, MXFP4), rcp_max = 1/448 (E4M3), 1/57344 (E5M2) or 1/6
 * (E2M1), evaluated in IEEE float32 in that order.  MXFP8 (either element
 * type) and MXFP4 round SF up to a power of two (UE8M0 = clamp(ceil(log2 SF)
 * + 127, 0, 254), 0 for an all-zero group) and store E4M3, E5M2 or E2M1 of
 * x * 2^(127 - UE8M0); NVFP4 stores
 * UE4M3 = E4M3(SF) and E2M1(x * (g / SF_decoded)).  Element encodes round to
 * nearest even and saturate; E2M1 codes are packed two per byte, the even
 * element in the low nibble.
 *
 *   x            [m, k] BF16, 16-byte aligned
 *   mode         HQ_MXFP8, HQ_MXFP8_E5M2, HQ_MXFP4 or HQ_NVFP4
 *   use_swizzle  1: SfAtom layout; 0: row-major [ceil(m/128)*128, k/group]
 *   global_scale NVFP4 only: device float [1] or NULL (=1); must be NULL for
 *                MXFP8 and MXFP4 (HQ_ERR_UNSUPPORTED otherwise)
 *   q_out        MXFP8 (E4M3 or E5M2) [m, k] bytes; MXFP4 / NVFP4 [m, k/2] bytes; 16-byte
 *                aligned
 *   sf_out       hq_sf_bytes(m, k, mode) bytes; padding rows written as 0
 *   use_pdl      1: launch with programmatic dependent launch
 * Requires k % (4 * group) == 0 (HQ_ERR_INVALID otherwise).  m == 0 is a
 * no-op. */
int hq_quant(const hq_bf16 *x, int64_t m, int64_t k, hq_mode mode, int use_swizzle,
             const float *global_scale, void *q_out, uint8_t *sf_out, int use_pdl,
             hq_stream_t s);

/* HALOps group_wise_quant with a float16 input (the page accepts BF16 or
 * FP16): identical to hq_quant except that x holds IEEE binary16 bit
 * patterns, each converted exactly to float32 before the scale rule. */
int hq_quant_f16(const uint16_t *x, int64_t m, int64_t k, hq_mode mode, int use_swizzle,
                 const float *global_scale, void *q_out, uint8_t *sf_out, int use_pdl,
                 hq_stream_t s);

/* hq_quant over the grouped-masked layout (HALOps group_masked_gemm: E
 * experts of max_m rows each, masked_m[e] valid rows from row e * max_m):
 * quantises only the valid rows of x [E * max_m, k], as the masked GEMM
 * reads no other row's result.  Rows past masked_m[e] keep their codes and
 * scale bytes untouched; masked_m[e] outside [0, max_m] is clamped and sets
 * HQ_STATUS_TOKENS_CLAMPED.  Only valid rows are visited (their prefix is
 * kept in shared memory: E <= 8192).  max_m % 128 == 0 (HQ_ERR_INVALID otherwise), so
 * sf_out holds hq_sf_bytes(E * max_m, k, mode) bytes and no padding rows.
 * masked_m: device int32 [E], 4-byte aligned.  The other arguments are
 * hq_quant's. */
int hq_quant_masked(const hq_bf16 *x, int E, int64_t max_m, const int32_t *masked_m, int64_t k,
                    hq_mode mode, int use_swizzle, const float *global_scale, void *q_out,
                    uint8_t *sf_out, int use_pdl, hq_stream_t s);

/* ------------------------------------------------------------------------- *
 * Block-scaled GEMMs: out = alpha * (A . B^T) + bias, BF16 output (RNE).
 *
 * Common arguments:
 *   a, sfa   quantised A and its SfAtom scales (as hq_quant writes them)
 *   b, sfb   quantised B (one [n, k] matrix per group, stacked) and its
 *            SfAtom scales (per group ceil(n/128)*128*(k/group) bytes)
 *   mode     HQ_MXFP8, HQ_MXFP8_E5M2 (A and B both float8_e5m2), HQ_MXFP4
 *            or HQ_NVFP4
 *   alpha    device float per group, or NULL (= 1).  Required for HQ_NVFP4
 *            (HQ_ERR_UNSUPPORTED if NULL), optional for the MXFP8 modes, not
 *            accepted for HQ_MXFP4 (HQ_ERR_UNSUPPORTED if given)
 *   bias     device BF16 [groups, n] or NULL.  MXFP8 modes only
 *            (HQ_ERR_UNSUPPORTED with the FP4 modes), as the HALOps API states
 *   sm_count number of persistent CTAs (<= 0: all SMs)
 * Shape rules: k % (4 * group) == 0; n % 128 == 0; all pointers 16-byte
 * aligned.  Each tile is 128 rows by 128 or 256 columns.
 * ------------------------------------------------------------------------- */

/* HALOps "GEMM" API, dense_gemm: out[m, n] = alpha * a[m, k] . b[n, k]^T + bias.
 * sfa holds ceil(m/128)*128 rows.  A batched GEMM (batch_gemm) is
 * hq_gemm_grouped_masked with masked_m[e] = max_m, or hq_gemm_grouped_contig
 * with padded_offsets[e] = (e + 1) * M. */
int hq_gemm_dense(const void *a, const uint8_t *sfa, const void *b, const uint8_t *sfb,
                  const float *alpha, const hq_bf16 *bias, hq_bf16 *out, int64_t m, int64_t n,
                  int64_t k, hq_mode mode, int sm_count, int use_pdl, hq_stream_t s);

/* cuDNN "Grouped GEMM + dGLU (SM100)", Step 1 with groups "contiguous in the M
 * dimension and described by padded_offsets (cumulative aligned end
 * offsets)"; HALOps group_contiguous_gemm with per-expert weights.
 *   a [m_rows, k], out [m_rows, n]; b [L, n, k]; sfb per expert as above
 *   padded_offsets  device int32 [L], non-decreasing group ends, each a
 *                   multiple of 128 (the pages use 256), last <= m_rows
 *   L               1..1024
 * Rows in [off[g-1], off[g]) use expert g; rows >= off[L-1] are not written.
 * Offset violations set HQ_STATUS_BAD_OFFSETS and the affected rows are
 * skipped. */
int hq_gemm_grouped_contig(const void *a, const uint8_t *sfa, const void *b, const uint8_t *sfb,
                           const int32_t *padded_offsets, int L, const float *alpha,
                           const hq_bf16 *bias, hq_bf16 *out, int64_t m_rows, int64_t n,
                           int64_t k, hq_mode mode, int sm_count, hq_stream_t s);

/* HALOps "GEMM" API, group_contiguous_gemm in its own form: rows of all
 * experts packed contiguously without per-expert padding, expert_ids[m]
 * (device int32 [m_rows], non-decreasing) naming the expert of row m.  A
 * 128-row tile that holds rows of several experts is computed once per
 * expert, each pass writing only that expert's rows.  A row whose id is
 * outside [0, L), or below the id of the row before it, is not written and
 * sets HQ_STATUS_BAD_OFFSETS.  workspace: caller-owned device memory of
 * hq_gemm_grouped_rows_workspace_size(m_rows, L) bytes, 256-byte aligned (it
 * holds the list of (tile, expert, row range) segments a preparatory kernel
 * builds; at most 2 * ceil(m_rows / 128) + L segments, beyond which - only
 * with ids that break the order on many rows - later rows are not written).
 * Other arguments as hq_gemm_grouped_contig. */
int hq_gemm_grouped_rows(const void *a, const uint8_t *sfa, const void *b, const uint8_t *sfb,
                         const int32_t *expert_ids, int L, const float *alpha, const hq_bf16 *bias,
                         hq_bf16 *out, int64_t m_rows, int64_t n, int64_t k, hq_mode mode,
                         void *workspace, size_t ws_bytes, int sm_count, hq_stream_t s);
size_t hq_gemm_grouped_rows_workspace_size(int64_t m_rows, int L);

/* HALOps "GEMM" API, group_masked_gemm: a [E * max_m, k] with expert e's rows
 * at e * max_m; masked_m (device int32 [E]) valid rows per expert; only rows
 * e * max_m + i, i < masked_m[e], are computed and written -- every other
 * output row is left untouched.  max_m > 0 and max_m % 128 == 0;
 * masked_m[e] outside [0, max_m] is clamped (HQ_STATUS_MASK_CLAMPED). */
int hq_gemm_grouped_masked(const void *a, const uint8_t *sfa, const void *b, const uint8_t *sfb,
                           const int32_t *masked_m, int E, int64_t max_m, const float *alpha,
                           const hq_bf16 *bias, hq_bf16 *out, int64_t n, int64_t k, hq_mode mode,
                           int sm_count, hq_stream_t s);

/* ------------------------------------------------------------------------- *
 * HALOps "GEMM" API, fused_swiglu_quant: y = up * silu(gate) over input =
 * [gate | up] (gate = columns [0, H), up = [H, 2H)), then y (float32) is
 * quantised exactly as hq_quant does (MXFP8: group 32, UE8M0; NVFP4: group
 * 16, UE4M3, norm_const = *global_scale or 1).
 *   in          [rows, 2H] BF16
 *   token_nums  device int32 [E] valid rows per expert, or NULL (all rows).
 *               With token_nums, row r belongs to expert r / rows_per_expert
 *               and is written only if r % rows_per_expert < token_nums[e]
 *               (nothing of an invalid row is written, not even its scales).
 *   q_out       MXFP8 [rows, H] bytes; NVFP4 [rows, H/2] bytes
 *   sf_out      SfAtom scales of kb_dim columns over ceil(rows/128)*128 rows:
 *               MXFP8 kb_dim = ceil(H / 512) * 16, NVFP4 kb_dim = H / 16;
 *               MXFP8 columns [H/32, kb_dim) of written rows hold 0; with
 *               token_nums == NULL the padding rows hold 0.
 * Requires H % 128 == 0 (MXFP8) or H % 64 == 0 (NVFP4), rows_per_expert > 0
 * and E * rows_per_expert == rows when token_nums is given, with E <= 8192
 * (the valid-row prefix is kept in shared memory); only valid rows are
 * visited, so the time follows the valid rows, not all of them. */
int hq_swiglu_quant(const hq_bf16 *in, int64_t rows, int64_t H, const int32_t *token_nums, int E,
                    int64_t rows_per_expert, hq_mode mode, const float *global_scale,
                    void *q_out, uint8_t *sf_out, hq_stream_t s);

/* The grouped up-proj GEMM with the SwiGLU + requantisation above fused into
 * its epilogue (HALOps fused_swiglu_quant applied to the output of
 * group_contiguous_gemm; cuDNN "Grouped GEMM + dGLU (SM100)" forward
 * SwiGLU): per group g and row m of the group
 *     gate_up = alpha_g * (a[m] . b[g]^T)      (float32, never rounded to BF16)
 *     y       = up * gate / (1 + exp(-gate)),  gate = gate_up[0, H), up = [H, 2H)
 * and y is quantised in out_mode as hq_swiglu_quant quantises its float32 y.
 *   a, sfa          [m_rows, k] quantised in `mode` (as hq_gemm_grouped_contig)
 *   b, sfb          [L, 2H, k] quantised in `mode`: rows [0, H) of expert g
 *                   are its gate weights, rows [H, 2H) its up weights
 *   padded_offsets  as hq_gemm_grouped_contig; alpha as there (per group)
 *   out_mode        HQ_MXFP8 or HQ_NVFP4 (the format of y)
 *   global_scale    NVFP4 output norm_const (device float [1]) or NULL (= 1);
 *                   not accepted with HQ_MXFP8 output (HQ_ERR_UNSUPPORTED)
 *   q_out, sf_out   as hq_swiglu_quant: MXFP8 [m_rows, H] codes, NVFP4
 *                   [m_rows, H/2]; SfAtom scales of kb_dim columns (MXFP8
 *                   ceil(H / 512) * 16 with columns [H/32, kb_dim) written 0;
 *                   NVFP4 H / 16) over ceil(m_rows/128)*128 rows.
 * Rows >= padded_offsets[L-1] (codes and scales) are not written.  No bias.
 * Requires H % 128 == 0, k % (4 * group) == 0; pointers 16-byte aligned.
 * Differs from the unfused path (GEMM to BF16, then hq_swiglu_quant) only in
 * that gate_up keeps its float32 value: codes and scale bytes may differ by
 * one rounding step where the BF16 rounding of gate_up would decide them. */
int hq_gemm_grouped_contig_swiglu_quant(const void *a, const uint8_t *sfa, const void *b,
                                        const uint8_t *sfb, const int32_t *padded_offsets, int L,
                                        const float *alpha, int64_t m_rows, int64_t H, int64_t k,
                                        hq_mode mode, hq_mode out_mode, const float *global_scale,
                                        void *q_out, uint8_t *sf_out, int sm_count, hq_stream_t s);

/* ------------------------------------------------------------------------- *
 * cuDNN "Grouped GEMM + dGLU (SM100)", BF16 contract, act_func = "dswiglu",
 * dense B:  R_g = alpha_g^2 A_g B_g^T,  X_g = beta_g C_g; X is split into
 * alternating 32-column gate / input blocks (within each 64 columns: 32 gate
 * then 32 input); with s = sigmoid(gate):
 *     D_row[gate col]  = dgate  = R prob input s (1 + gate (1 - s))
 *     D_row[input col] = dinput = R prob gate s
 *     dprob[m]        += sum_j R gate s input           (no prob factor)
 *     dbias[g, c]     += sum over rows m of group g of D_row[m, c]
 *   a        [m, k] BF16                  b  [L, n, k] BF16 (K-major)
 *   c        [m, 2n] BF16 (saved forward) d_row [m, 2n] BF16 output
 *   padded_offsets device int32 [L] (rules as hq_gemm_grouped_contig)
 *   alpha, beta    device float [L];  prob device float [m]
 *   dprob    device float [m], caller-zeroed, accumulated (+=)
 *   dbias    device BF16 [L, 2n] or NULL; caller-zeroed, accumulated (+=) from
 *            float32 partial sums of the unrounded D values
 *   workspace      device scratch of hq_gemm_dswiglu_workspace_size(L, n)
 *                  bytes (may be NULL when dbias is NULL); contents need not
 *                  be initialised; 256-byte aligned
 * Rows >= padded_offsets[L-1] are not written.  Requires n % 32 == 0,
 * k % 8 == 0, 1 <= L <= 1024. */
int hq_gemm_dswiglu(const hq_bf16 *a, const hq_bf16 *b, const hq_bf16 *c,
                    const int32_t *padded_offsets, int L, const float *alpha, const float *beta,
                    const float *prob, hq_bf16 *d_row, float *dprob, hq_bf16 *dbias, int64_t m,
                    int64_t n, int64_t k, void *workspace, size_t ws_bytes, int sm_count,
                    hq_stream_t s);

/* Bytes of scratch hq_gemm_dswiglu needs for dbias: L * 2n float32, rounded
 * up to 256 bytes. */
size_t hq_gemm_dswiglu_workspace_size(int L, int64_t n);

/* ------------------------------------------------------------------------- *
 * cuDNN "Grouped GEMM + dGLU (SM100)", BF16 contract, act_func = "dgeglu":
 * the same grouped GEMM R_g = alpha_g^2 A_g B_g^T, and a clamped-GeGLU
 * backward over the saved C used as stored (no beta), with the BF16
 * backend's fixed constants geglu_alpha = 1.702, glu_clamp_max = 7,
 * glu_clamp_min = -7, linear_offset = 1.  Within every 64 columns of C the
 * first 32 are gate and the next 32 are up:
 *     gate_c = min(gate, 7),  up_c = clamp(up, -7, 7),  s = sigmoid(1.702 gate_c)
 *     D_row[gate col] = R prob (up_c + 1) s (1 + 1.702 gate_c (1 - s))  if gate <= 7, else 0
 *     D_row[up col]   = R prob gate_c s                                 if -7 <= up <= 7, else 0
 *     dprob[m]       += sum_j R gate_c s (up_c + 1)
 *     dbias[g, c]    += sum over rows m of group g of D_row[m, c]
 * Arguments, layouts, accumulation, workspace and errors as hq_gemm_dswiglu
 * (there is no beta). */
int hq_gemm_dgeglu(const hq_bf16 *a, const hq_bf16 *b, const hq_bf16 *c,
                   const int32_t *padded_offsets, int L, const float *alpha, const float *prob,
                   hq_bf16 *d_row, float *dprob, hq_bf16 *dbias, int64_t m, int64_t n, int64_t k,
                   void *workspace, size_t ws_bytes, int sm_count, hq_stream_t s);

/* cuDNN frontend "Grouped GEMM + dGLU (SM100)", block-scaled contract:
 * Step 1 R = alpha_g^2 * (dequantised A . dequantised B_g^T) with A, B and
 * their SfAtom scales as hq_quant writes them (mode HQ_MXFP8, HQ_MXFP8_E5M2,
 * HQ_MXFP4 or HQ_NVFP4), groups contiguous in M by padded_offsets (as
 * hq_gemm_grouped_contig); Step 2 the dGLU epilogue of hq_gemm_dswiglu
 * (act 0) or hq_gemm_dgeglu (act 1) on the BF16 C [m, 2n]; Step 3 optional
 * FP8 output.
 *   d_row      sfd_row == NULL: BF16 [m, 2n].  Otherwise E4M3 [m, 2n] bytes
 *              with sfd_row the UE8M0 scales of every 32 consecutive D_row
 *              values of a row (SfAtom layout, ceil(m/128)*128 rows, 2n/32
 *              columns): SF = norm_const * amax * (1/448) rounded up to a
 *              power of two, D_q = E4M3(D * norm_const / SF)
 *   d_col      NULL, or (with sfd_row) E4M3 [m, 2n]: D quantised along M,
 *              one UE8M0 scale per column and 32 consecutive rows in sfd_col
 *              (SfAtom layout of a [2n, ceil(m/128)*4] matrix:
 *              ceil(2n/128)*128 * ceil(m/128)*4 bytes), same rule
 *   norm_const device float [1] or NULL (= 1); only with sfd_row
 *   amax       NULL, or device float [L, 2], overwritten: max |D| over each
 *              group's rows and its gate columns ([g, 0]) / input columns
 *              ([g, 1]) (0 for an empty group; m == 0 leaves it untouched)
 *   alpha, beta, prob, dprob, dbias, workspace as hq_gemm_dswiglu (beta
 *              ignored and may be NULL for act 1)
 * Requires n % 128 == 0 and k % (4 * group) == 0. */
int hq_gemm_dglu_bs(const void *a, const uint8_t *sfa, const void *b, const uint8_t *sfb,
                    const hq_bf16 *c, const int32_t *padded_offsets, int L, const float *alpha,
                    const float *beta, const float *prob, int act, void *d_row, uint8_t *sfd_row,
                    void *d_col, uint8_t *sfd_col, const float *norm_const, float *dprob,
                    hq_bf16 *dbias, float *amax, int64_t m, int64_t n, int64_t k, hq_mode mode,
                    void *workspace, size_t ws_bytes, int sm_count, hq_stream_t s);

/* D_row / D_col element type of hq_gemm_dglu_bs_typed (the cuDNN page's
 * d_dtype values). */
typedef enum {
  HQ_D_BF16 = 0, /* bfloat16                                              */
  HQ_D_F32 = 1,  /* float32 (4 bytes per element)                         */
  HQ_D_E4M3 = 2, /* float8_e4m3fn with UE8M0 SFD scales (Step 3)          */
  HQ_D_E5M2 = 3  /* float8_e5m2 with UE8M0 SFD scales (Step 3)            */
} hq_dtype;

/* hq_gemm_dglu_bs with the D element type given explicitly (cuDNN
 * "Grouped GEMM + dGLU (SM100)", Data Types table: d_dtype bfloat16 /
 * float32 for FP4 operands, float8_e4m3fn / float8_e5m2 for FP8 operands;
 * the other pairings run as well).
 *   d_type  HQ_D_BF16 or HQ_D_F32: sfd_row, d_col, sfd_col, norm_const NULL;
 *           d_row is [m, 2n] of bfloat16 or float32.
 *           HQ_D_E4M3 or HQ_D_E5M2: sfd_row required, D_row (and D_col) as
 *           hq_gemm_dglu_bs's FP8 output with rcp_max = 1/448 (E4M3) or
 *           1/57344 (E5M2) and codes of that type.
 * HQ_ERR_INVALID for another d_type or a mismatched sfd_row;
 * HQ_ERR_UNSUPPORTED for HQ_D_F32 with HQ_NVFP4 operands and dbias == NULL
 * (the page's "non-dbias paths" constraint).  Everything else as
 * hq_gemm_dglu_bs. */
int hq_gemm_dglu_bs_typed(const void *a, const uint8_t *sfa, const void *b, const uint8_t *sfb,
                          const hq_bf16 *c, const int32_t *padded_offsets, int L,
                          const float *alpha, const float *beta, const float *prob, int act,
                          void *d_row, uint8_t *sfd_row, void *d_col, uint8_t *sfd_col,
                          const float *norm_const, float *dprob, hq_bf16 *dbias, float *amax,
                          int64_t m, int64_t n, int64_t k, hq_mode mode, hq_dtype d_type,
                          void *workspace, size_t ws_bytes, int sm_count, hq_stream_t s);

/* ------------------------------------------------------------------------- *
 * Discrete weights (cuDNN frontend "Grouped GEMM + dGLU (SM100)", weight
 * layout modes: "Discrete mode: Per-expert weight pointers (no weight
 * stacking required)"; b_ptrs / sfb_ptrs are device int64 arrays of shape
 * (num_experts,)).  Instead of one stacked B [L, n, k] (and its stacked
 * scales), expert g's K-major B [n, k] starts at b_ptrs[g] and, for the
 * block-scaled modes, its SfAtom scales (ceil(n/128)*128 * k/group bytes) at
 * sfb_ptrs[g].  Both arrays are device memory, 8-byte aligned.
 *
 * Before the GEMM a small kernel builds one TMA tensor map per expert in the
 * head of the caller's workspace (from a host-encoded template whose global
 * address it replaces with b_ptrs[g]).  An expert whose b_ptrs[g] or
 * sfb_ptrs[g] is 0 or not 16-byte aligned is skipped: nothing is loaded
 * through its pointers, none of its rows is written (dprob, dbias and amax
 * get nothing from it), and HQ_STATUS_BAD_POINTER is set.  Any other pointer
 * value must address a whole [n, k] matrix (and its scales), as for every
 * device pointer of this API.
 *
 * Workspace: hq_gemm_discrete_workspace_size(L, dbias_n) bytes, 256-byte
 * aligned, where dbias_n is the dGLU call's n when it produces dbias, else 0
 * (the head holds L tensor maps of 128 bytes and L int32 flags, the rest the
 * dbias partial sums). */
size_t hq_gemm_discrete_workspace_size(int L, int64_t dbias_n);

/* hq_gemm_grouped_contig with discrete weights. */
int hq_gemm_grouped_contig_discrete(const void *a, const uint8_t *sfa, const int64_t *b_ptrs,
                                    const int64_t *sfb_ptrs, const int32_t *padded_offsets, int L,
                                    const float *alpha, const hq_bf16 *bias, hq_bf16 *out,
                                    int64_t m_rows, int64_t n, int64_t k, hq_mode mode,
                                    void *workspace, size_t ws_bytes, int sm_count, hq_stream_t s);

/* hq_gemm_dglu_bs with discrete weights (the block-scaled contract). */
int hq_gemm_dglu_bs_discrete(const void *a, const uint8_t *sfa, const int64_t *b_ptrs,
                             const int64_t *sfb_ptrs, const hq_bf16 *c,
                             const int32_t *padded_offsets, int L, const float *alpha,
                             const float *beta, const float *prob, int act, void *d_row,
                             uint8_t *sfd_row, void *d_col, uint8_t *sfd_col,
                             const float *norm_const, float *dprob, hq_bf16 *dbias, float *amax,
                             int64_t m, int64_t n, int64_t k, hq_mode mode, void *workspace,
                             size_t ws_bytes, int sm_count, hq_stream_t s);

/* hq_gemm_dswiglu (act 0) / hq_gemm_dgeglu (act 1) with discrete BF16
 * weights: b_ptrs[g] -> K-major BF16 [n, k] (the BF16 contract's
 * b_major = "k"; N-major per-expert weights: hq_gemm_dglu_discrete_nmajor).  beta as
 * hq_gemm_dswiglu (ignored, may be NULL, for act 1). */
int hq_gemm_dglu_discrete(const hq_bf16 *a, const int64_t *b_ptrs, const hq_bf16 *c,
                          const int32_t *padded_offsets, int L, const float *alpha,
                          const float *beta, const float *prob, int act, hq_bf16 *d_row,
                          float *dprob, hq_bf16 *dbias, int64_t m, int64_t n, int64_t k,
                          void *workspace, size_t ws_bytes, int sm_count, hq_stream_t s);

/* hq_gemm_dglu_discrete with N-major per-expert BF16 weights (the BF16
 * contract's discrete b_major = "n"): b_ptrs[g] -> BF16 [k, n], n
 * contiguous, 16-byte aligned.  A transpose pass first writes a K-major copy
 * of every expert into the workspace, then the K-major discrete path runs on
 * the copies; an expert whose pointer is null or unaligned is skipped and
 * flagged (HQ_STATUS_BAD_POINTER) as there.
 *   workspace  hq_gemm_dglu_discrete_nmajor_workspace_size(L, n, k,
 *              dbias != NULL) bytes, 256-byte aligned, caller-owned
 * Arguments, results and errors otherwise as hq_gemm_dglu_discrete. */
size_t hq_gemm_dglu_discrete_nmajor_workspace_size(int L, int64_t n, int64_t k, int with_dbias);
int hq_gemm_dglu_discrete_nmajor(const hq_bf16 *a, const int64_t *b_ptrs, const hq_bf16 *c,
                                 const int32_t *padded_offsets, int L, const float *alpha,
                                 const float *beta, const float *prob, int act, hq_bf16 *d_row,
                                 float *dprob, hq_bf16 *dbias, int64_t m, int64_t n, int64_t k,
                                 void *workspace, size_t ws_bytes, int sm_count, hq_stream_t s);

/* ------------------------------------------------------------------------- *
 * hq_gemm_dswiglu without caller-provided scratch.  The paper has no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory -- for example a plugin or custom op loaded into a
 * host framework that owns every device allocation and hands it only its
 * inputs and outputs, or code that must not call cudaMalloc because that can
 * synchronise the device and stall other work already running on it.
 *
 * Same arguments and results as hq_gemm_dswiglu, minus workspace/ws_bytes.
 * The dbias partial sums go to a fixed scratch array inside the library:
 * 1 MiB of device memory (262144 floats) that every GPU which loads
 * libhq.so holds until the process exits.  dbias therefore needs
 * L * 2n <= 262144; larger requests return HQ_ERR_UNSUPPORTED before
 * anything is launched (dbias == NULL has no limit).  The call allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * The first call on a device resolves the scratch array's device address
 * (once per device and CUDA context, with that device current); make that
 * first call before any stream capture.  Calling cudaDeviceReset while the
 * library is loaded is not supported: the library keeps per-device state
 * (resolved addresses, kernel attributes) that a reset discards.  Every call clears the part of the scratch it uses
 * before accumulating into it, because the array keeps the previous call's
 * contents.  All calls share the one array, so two calls whose work overlaps
 * on the GPU (different streams, no ordering between them) race on it and
 * their dbias results are undefined; order such calls on one stream or with
 * events. */
int hq_gemm_dswiglu_noalloc(const hq_bf16 *a, const hq_bf16 *b, const hq_bf16 *c,
                            const int32_t *padded_offsets, int L, const float *alpha,
                            const float *beta, const float *prob, hq_bf16 *d_row, float *dprob,
                            hq_bf16 *dbias, int64_t m, int64_t n, int64_t k, int sm_count,
                            hq_stream_t s);

/* ------------------------------------------------------------------------- *
 * HALOps "GEMM" API, prefill_permute_to_masked_gemm: rearranges tokens into
 * the padded expert layout [E * max_token_num, hidden] of
 * hq_gemm_grouped_masked and converts their scale factors into the SfAtom
 * layout of [E * max_token_num, hidden / 32] bytes.
 *   x            [num_tokens, hidden] elements of elem_bytes bytes (1: E4M3,
 *                2: BF16); 16-byte aligned
 *   scale        scale_mode 0 ("broadcast"): int32 [num_tokens, hidden / 512],
 *                byte b of word i is the scale of elements [128 (4i + b),
 *                +128) and is repeated for its four 32-element groups;
 *                scale_mode 1 ("direct"): uint8 [num_tokens, hidden / 32];
 *                4-byte aligned
 *   topk_ids     int64 [num_tokens, topk] expert per (token, slot); -1 means
 *                unassigned
 *   permute_x    [E * max_token_num, hidden] output (same element type)
 *   out_scale    SfAtom output, E * max_token_num * hidden / 32 bytes
 *   indice_map   int32 [num_tokens, topk]: the expert-local row of each
 *                (token, slot), -1 if unassigned or dropped
 *   token_nums   int32 [E]: rows written per expert (the masked_m of the
 *                following hq_gemm_grouped_masked)
 *   workspace    hq_prefill_permute_workspace_size(num_tokens, E) bytes,
 *                256-byte aligned, caller-owned
 * Each expert's rows are filled in increasing (token, slot) order.  An id
 * outside [0, E) other than -1, or an entry whose expert already holds
 * max_token_num rows, is dropped (map -1) and sets HQ_STATUS_ROUTING_DROPPED;
 * nothing is written out of bounds.  Rows past token_nums[e] and their scale
 * bytes are not written.  Requires 1 <= topk <= 32, 1 <= E <= 1024,
 * max_token_num a positive multiple of 128, hidden a multiple of 512
 * (broadcast) or 128 (direct). */
int hq_prefill_permute(const void *x, int elem_bytes, const void *scale, int scale_mode,
                       const int64_t *topk_ids, int64_t num_tokens, int64_t hidden, int topk,
                       int num_experts, int64_t max_token_num, void *permute_x, uint8_t *out_scale,
                       int32_t *indice_map, int32_t *token_nums, void *workspace, size_t ws_bytes,
                       hq_stream_t s);
size_t hq_prefill_permute_workspace_size(int64_t num_tokens, int num_experts);

#ifdef __cplusplus
}
#endif

#endif /* HQ_H_ */
