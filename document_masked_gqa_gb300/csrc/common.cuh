// Plan object and launch parameters shared by the library's translation
// units (host + device).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/dma.h"

namespace dma {

constexpr int kTileM = 128;  // query rows per tile (positions x heads of a group)
constexpr int kTileN = 128;  // key positions per tile
constexpr uint32_t kPartialBit = 0x80000000u;
constexpr uint32_t kIndexMask = 0x7FFFFFFFu;

// dK/dV work items are (key tile, K/V head).  When a shape has fewer than
// kKvSplitItems of them (a short sequence with one K/V head, say), most SMs
// would idle, so each key tile's list of query tiles is cut into segments,
// up to kKvMaxSegs, each its own work item writing an fp32 partial of dK, dV;
// a reduction sums the partials in segment order.
constexpr int kKvSplitItems = 256;
constexpr int kKvMaxSegs = 8;
__host__ __device__ inline int kv_segments(int batch, int seq_len, int n_kv_heads) {
  const long long items = static_cast<long long>(batch) * (seq_len / kTileN) * n_kv_heads;
  if (items <= 0 || items >= kKvSplitItems) return 1;
  const long long s = (kKvSplitItems + items - 1) / items;
  return static_cast<int>(s < kKvMaxSegs ? s : kKvMaxSegs);
}

constexpr int kSchedFwd = 0, kSchedDkdv = 2;
// bytes at the start of the workspace: status words [0, 16), work counters [32, 48)
constexpr int kStatusBytes = 64, kSchedOffset = 32;

// Device-visible shape and workspace pointers of one rank's plan.
struct PlanDev {
  int batch, seq_len, cp_size, cp_rank, n_heads, n_kv_heads, head_dim;
  int chunk, local_len, group, tile_pos, n_qtiles, n_ktiles;
  float scale;       // softmax scale
  float scale_log2;  // scale * log2(e)
  uint64_t timeout_ns;
  uint32_t* status;   // [0] error word (kernels do nothing once set), [1] warning bits
  int32_t* sched;     // work counters of the persistent kernels, two per kernel
                      // (next item, CTAs exited): forward at kSchedFwd, dK/dV at
                      // kSchedDkdv; zeroed with the status words by the plan
  int32_t* qpos;      // [Lq]
  int32_t* doc_lo;    // [B][Lq]
  int32_t* doc_hi;    // [B][S] end (exclusive) of each key position's document
  int32_t* chunk_order;
  uint8_t* tile_class;  // [B][nQt][nKt]
  int32_t* row_cnt;   // [B*nQt]
  int32_t* row_ptr;   // [B*nQt + 1]
  int32_t* row_idx;   // [B*nQt*nKt]
  int32_t* col_cnt;   // [B*nKt]
  int32_t* col_ptr;   // [B*nKt + 1]
  int32_t* col_idx;   // [B*nQt*nKt]
  int32_t* fwd_order; // [B*nQt]
  int32_t* bwd_order; // [B*nKt]
  float* delta;       // [B][Hq][Lq]
  uint16_t* v16;      // [B][S][Hkv][D] fp16 copy of V for the forward's P V
  int kv_segs;        // segments per key tile's query list (kv_segments)
  float* kv_part;     // kv_segs > 1: [2][kv_segs][B][S][Hkv][D] partial dK, then dV
};

struct WorkspaceLayout {
  size_t status, qpos, doc_lo, doc_hi, chunk_order, tile_class, row_cnt, row_ptr, row_idx, col_cnt,
      col_ptr, col_idx, fwd_order, bwd_order, delta, v16, kv_part, total;
};

}  // namespace dma

struct dma_plan_s {
  dma::PlanDev d;
  int device;
  int num_sms;
  const int32_t* cu;  // only read while the plan kernels run
  int n_docs;
};

namespace dma {
// Launchers implemented in the .cu files (host side).
#ifdef __CUDACC__
// Work item of round k for this CTA of the dQ kernel (a static order; the
// forward and dK/dV kernels take theirs from the plan's work counters):
// rounds alternate direction over the CTAs, so that a longest-first item
// order spreads its work evenly (CTA c takes c, 2G-1-c, 2G+c, ...).
__device__ __forceinline__ int snake_item(int k) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}
#endif

cudaError_t launch_plan_kernels(const dma_plan_s& p, cudaStream_t s);
cudaError_t launch_cp_copy(const dma_plan_s& p, const void* src, void* dst, size_t row_bytes,
                           bool gather, cudaStream_t s);
cudaError_t launch_v_to_f16(const dma_plan_s& p, const dma_bf16* v, cudaStream_t s);
cudaError_t launch_fwd(const dma_plan_s& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv16, const CUtensorMap& to, float* o, float* lse,
                       cudaStream_t s);
cudaError_t launch_delta(const dma_plan_s& p, const float* o, const dma_bf16* dout,
                         cudaStream_t s);
cudaError_t launch_dkdv(const dma_plan_s& p, const float* lse, const CUtensorMap& tq,
                        const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                        const CUtensorMap& tdk, const CUtensorMap& tdv, cudaStream_t s);
// to != nullptr: the dQ kernel also computes Delta from O (map `to`, fp32)
// and stores it in the plan's workspace
cudaError_t launch_dq(const dma_plan_s& p, const float* lse, const CUtensorMap& tq,
                      const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                      const CUtensorMap& tdq, const CUtensorMap* to, const float* o,
                      const dma_bf16* dout, dma_bf16* dq, cudaStream_t s);
cudaError_t launch_kv_reduce(const dma_plan_s& p, float* dk, float* dv, cudaStream_t s);
cudaError_t launch_wait_probe(uint64_t timeout_ns, uint32_t* status, cudaStream_t s);
cudaError_t launch_status_out(const uint32_t* status, uint32_t* out, cudaStream_t s);
cudaError_t launch_cp_chunk_copy(const void* src, void* dst, int batch, int seq_len, int cp_size,
                                 size_t row_bytes, bool to_natural, cudaStream_t s);
}  // namespace dma
