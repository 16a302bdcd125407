// hq_permute.cu -- routing permute of tokens and their scale factors into the
// padded expert layout of the masked GEMM (HALOps "GEMM" API,
// prefill_permute_to_masked_gemm).
//
// Three passes over blocks of kTok tokens, all deterministic:
//   count    per block, a shared-memory histogram of its valid expert ids
//            -> counts[e][block] (workspace);
//   scan     one warp per expert: the exclusive prefix of its block counts,
//            32 blocks at a time with a warp scan -> base[e][block]
//            (workspace), and token_nums[e] = min(total, max_token_num);
//   scatter  per block, warp 0 ranks the block's (token, slot) entries in
//            order -- 32 at a time with __match_any_sync, plus a running
//            per-expert count in shared memory -- so every expert's rows are
//            filled in increasing (token, slot) order; then each warp takes
//            whole tokens: it reads a token's row once with 16-byte loads and
//            stores it to every destination row of the token's slots, and
//            writes the scale bytes into SfAtom positions the same way, one
//            4-byte store per four scale columns (the four columns of an
//            atom row are contiguous).
// An id outside [0, E) other than -1, or an entry that finds its expert full,
// is dropped: its map entry is -1 and HQ_STATUS_ROUTING_DROPPED is set.  Rows
// past token_nums[e] (data and scales) are not written.
#include <cuda.h>
#include <cuda_runtime.h>

#include "hq_internal.h"
#include "hq_ptx.cuh"

namespace hq {
namespace {

constexpr int kTok = 16;             // tokens per block (small blocks: many CTAs copy in parallel)
constexpr int kThreads = 32 * kTok;  // the scatter copies one token per warp
constexpr int kMaxTopk = 32;
constexpr int kMaxExperts = 1024;

struct PermuteParams {
  const uint8_t* x;          // [T, hidden] elements of elem_bytes
  const uint8_t* scale;      // broadcast: int32 [T, hidden / 512]; direct: uint8 [T, hidden / 32]
  const int64_t* ids;        // [T, topk]
  int64_t T, hidden;
  int topk, E, elem_bytes, broadcast;
  int64_t cap;               // max_token_num
  uint8_t* out_x;            // [E * cap, hidden]
  uint8_t* out_sf;           // SfAtom bytes of [E * cap, hidden / 32]
  int32_t* imap;             // [T, topk]
  int32_t* token_nums;       // [E]
  int32_t* counts;           // [E, nblk] workspace
  int32_t* base;             // [E, nblk] workspace
  int nblk;
  uint32_t* status;
};

// The scan and the scatter are launched as programmatic dependents of the
// pass before them: each lets its dependent start launching at once and the
// dependent waits (griddepcontrol.wait) for its results before reading them.
__global__ void __launch_bounds__(kThreads) permute_count(const PermuteParams p) {
  pdl_launch_dependents();
  __shared__ int32_t hist[kMaxExperts];
  for (int i = threadIdx.x; i < p.E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTok;
  const int64_t ntok = p.T - t0 < kTok ? p.T - t0 : kTok;
  const int entries = static_cast<int>(ntok) * p.topk;
  const int64_t* ids = p.ids + t0 * p.topk;
  for (int j = threadIdx.x; j < entries; j += blockDim.x) {
    const int64_t e = __ldg(ids + j);
    if (e >= 0 && e < p.E) atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < p.E; i += blockDim.x)
    p.counts[static_cast<int64_t>(i) * p.nblk + blockIdx.x] = hist[i];
}

// One warp per expert (32 experts per CTA of 1024 threads).
__global__ void __launch_bounds__(1024) permute_scan(const PermuteParams p) {
  pdl_launch_dependents();
  pdl_wait();  // the block counts
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + (threadIdx.x >> 5);
  if (e >= p.E) return;
  const int32_t* cnt = p.counts + static_cast<int64_t>(e) * p.nblk;
  int32_t* base = p.base + static_cast<int64_t>(e) * p.nblk;
  int64_t run = 0;
  constexpr int kBatch = 8;  // 32-block chunks whose counts are loaded before any is scanned
  for (int c0 = 0; c0 < p.nblk; c0 += 32 * kBatch) {
    int32_t cs[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int b = c0 + 32 * i + lane;
      cs[i] = b < p.nblk ? cnt[b] : 0;
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int b = c0 + 32 * i + lane;
      const int32_t c = cs[i];
      int32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
      }
      const int64_t excl = run + incl - c;
      if (b < p.nblk) base[b] = static_cast<int32_t>(excl < p.cap ? excl : p.cap);
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
  if (lane == 0) {
    p.token_nums[e] = static_cast<int32_t>(run < p.cap ? run : p.cap);
    if (run > p.cap) atomicOr(p.status, HQ_STATUS_ROUTING_DROPPED);
  }
}

__global__ void __launch_bounds__(kThreads) permute_scatter(const PermuteParams p) {
  __shared__ int32_t running[kMaxExperts];
  __shared__ int32_t dest[kTok * kMaxTopk];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTok;
  const int64_t ntok = p.T - t0 < kTok ? p.T - t0 : kTok;
  const int entries = static_cast<int>(ntok) * p.topk;
  pdl_wait();  // the block bases
  for (int i = threadIdx.x; i < p.E; i += blockDim.x)
    running[i] = p.base[static_cast<int64_t>(i) * p.nblk + blockIdx.x];
  __syncthreads();
  if (warp == 0) {
    // rank the entries in (token, slot) order, 32 at a time
    const uint32_t lt = (1u << lane) - 1u;
    bool dropped = false;
    for (int c = 0; c < entries; c += 32) {
      const int j = c + lane;
      const int64_t e = j < entries ? __ldg(p.ids + t0 * p.topk + j) : -1;
      const bool valid = e >= 0 && e < p.E;
      if (j < entries && !valid && e != -1) dropped = true;
      // lanes with the same valid expert share a key; every other lane is alone
      const int key = valid ? static_cast<int>(e) : -1 - lane;
      const uint32_t same = __match_any_sync(0xFFFFFFFFu, key);
      const int rank = __popc(same & lt);
      const int before = valid ? running[e] : 0;
      __syncwarp();
      if (valid && rank == 0) running[e] = before + __popc(same);
      __syncwarp();
      const int64_t pos = static_cast<int64_t>(before) + rank;
      int32_t d = -1;
      if (valid) {
        if (pos < p.cap) d = static_cast<int32_t>(e * p.cap + pos);
        else dropped = true;
      }
      if (j < entries) {
        dest[j] = d;
        p.imap[t0 * p.topk + j] = d >= 0 ? static_cast<int32_t>(pos) : -1;
      }
    }
    if (__any_sync(0xFFFFFFFFu, dropped) && lane == 0) atomicOr(p.status, HQ_STATUS_ROUTING_DROPPED);
  }
  __syncthreads();
  // copy rows: one warp per token, its row read once and stored to each of
  // its destination rows
  const int64_t row_bytes = p.hidden * p.elem_bytes;
  const int nvec = static_cast<int>(row_bytes / 16);
  const int64_t S = p.hidden / 32;       // scale columns
  const int words = static_cast<int>(S / 4);
  const int nwarps = blockDim.x >> 5;
  const int64_t rows_out = static_cast<int64_t>(p.E) * p.cap;
  for (int tt = warp; tt < ntok; tt += nwarps) {
    const int32_t* dt = dest + tt * p.topk;
    const int64_t t = t0 + tt;
    const uint4* src = reinterpret_cast<const uint4*>(p.x + t * row_bytes);
    // debug builds: every destination row lies inside the [E * cap] output
    auto dst_ok = [&](int32_t d) { return d >= 0 && in_bounds(d < rows_out, p.status); };
    int v = lane;
    for (; v + 96 < nvec; v += 128) {  // four 16-byte loads in flight per lane
      const uint4 a = __ldg(src + v), b = __ldg(src + v + 32), c = __ldg(src + v + 64),
                  e = __ldg(src + v + 96);
      for (int k = 0; k < p.topk; ++k) {
        const int32_t d = dt[k];
        if (!dst_ok(d)) continue;
        uint4* dst = reinterpret_cast<uint4*>(p.out_x + static_cast<int64_t>(d) * row_bytes);
        dst[v] = a;
        dst[v + 32] = b;
        dst[v + 64] = c;
        dst[v + 96] = e;
      }
    }
    for (; v < nvec; v += 32) {
      const uint4 a = __ldg(src + v);
      for (int k = 0; k < p.topk; ++k) {
        const int32_t d = dt[k];
        if (!dst_ok(d)) continue;
        reinterpret_cast<uint4*>(p.out_x + static_cast<int64_t>(d) * row_bytes)[v] = a;
      }
    }
    for (int w = lane; w < words; w += 32) {
      uint32_t word;
      if (p.broadcast) {
        // word w holds the four 32-groups of 128-group w: its byte, repeated
        const uint32_t packed = __ldg(reinterpret_cast<const uint32_t*>(p.scale) + t * (S / 16) + w / 4);
        word = ((packed >> (8 * (w & 3))) & 0xFFu) * 0x01010101u;
      } else {
        word = __ldg(reinterpret_cast<const uint32_t*>(p.scale + t * S) + w);
      }
      for (int k = 0; k < p.topk; ++k) {
        const int32_t d = dt[k];
        if (!dst_ok(d)) continue;
        const int64_t r = d;
        const int64_t off = ((r >> 7) * (S >> 2) + w) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
        *reinterpret_cast<uint32_t*>(p.out_sf + off) = word;
      }
    }
  }
}

}  // namespace
}  // namespace hq

extern "C" {

size_t hq_prefill_permute_workspace_size(int64_t num_tokens, int num_experts) {
  if (num_tokens < 0 || num_experts < 1) return 0;
  const size_t nblk = static_cast<size_t>((num_tokens + hq::kTok - 1) / hq::kTok);
  const size_t bytes = 2 * nblk * static_cast<size_t>(num_experts) * sizeof(int32_t);
  return (bytes + 255) / 256 * 256;
}

int hq_prefill_permute(const void* x, int elem_bytes, const void* scale, int scale_mode,
                       const int64_t* topk_ids, int64_t num_tokens, int64_t hidden, int topk,
                       int num_experts, int64_t max_token_num, void* permute_x, uint8_t* out_scale,
                       int32_t* indice_map, int32_t* token_nums, void* workspace, size_t ws_bytes,
                       hq_stream_t s) {
  if (elem_bytes != 1 && elem_bytes != 2) return HQ_ERR_INVALID;
  if (scale_mode != 0 && scale_mode != 1) return HQ_ERR_INVALID;
  if (num_tokens < 0 || num_tokens > (1ll << 31) / hq::kMaxTopk) return HQ_ERR_INVALID;
  if (hidden <= 0 || hidden % (scale_mode == 0 ? 512 : 128) != 0 || hidden > (1ll << 24))
    return HQ_ERR_INVALID;
  if (topk < 1 || topk > hq::kMaxTopk) return HQ_ERR_INVALID;
  if (num_experts < 1 || num_experts > hq::kMaxExperts) return HQ_ERR_INVALID;
  if (max_token_num < 128 || max_token_num % 128 != 0) return HQ_ERR_INVALID;
  if (static_cast<int64_t>(num_experts) * max_token_num > (1ll << 31) - 1) return HQ_ERR_INVALID;
  if (!token_nums || (reinterpret_cast<uintptr_t>(token_nums) & 3u)) return HQ_ERR_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  if (num_tokens > 0) {
    if (!x || !scale || !topk_ids || !permute_x || !out_scale || !indice_map || !workspace)
      return HQ_ERR_INVALID;
    if (!hq::aligned16(x) || !hq::aligned16(permute_x) || !hq::aligned16(out_scale) ||
        (reinterpret_cast<uintptr_t>(scale) & 3u) || (reinterpret_cast<uintptr_t>(topk_ids) & 7u) ||
        (reinterpret_cast<uintptr_t>(indice_map) & 3u) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
      return HQ_ERR_INVALID;
    if (ws_bytes < hq_prefill_permute_workspace_size(num_tokens, num_experts)) return HQ_ERR_INVALID;
  }
  hq::PermuteParams p{};
  p.x = static_cast<const uint8_t*>(x);
  p.scale = static_cast<const uint8_t*>(scale);
  p.ids = topk_ids;
  p.T = num_tokens;
  p.hidden = hidden;
  p.topk = topk;
  p.E = num_experts;
  p.elem_bytes = elem_bytes;
  p.broadcast = scale_mode == 0 ? 1 : 0;
  p.cap = max_token_num;
  p.out_x = static_cast<uint8_t*>(permute_x);
  p.out_sf = out_scale;
  p.imap = indice_map;
  p.token_nums = token_nums;
  p.nblk = static_cast<int>((num_tokens + hq::kTok - 1) / hq::kTok);
  p.counts = static_cast<int32_t*>(workspace);
  p.base = p.counts + static_cast<int64_t>(p.nblk) * num_experts;
  p.status = hq::status_word_ptr();
  if (!p.status) return HQ_ERR_CUDA;
  if (p.nblk > 0) {
    hq::permute_count<<<p.nblk, hq::kThreads, 0, st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return HQ_ERR_CUDA;
  }
  if (hq::launch(hq::permute_scan, dim3((num_experts + 31) / 32), dim3(1024), 0, st, p.nblk > 0, p) != cudaSuccess)
    return HQ_ERR_CUDA;
  if (p.nblk > 0 &&
      hq::launch(hq::permute_scatter, dim3(p.nblk), dim3(hq::kThreads), 0, st, true, p) != cudaSuccess)
    return HQ_ERR_CUDA;
  return HQ_OK;
}

}  // extern "C"
