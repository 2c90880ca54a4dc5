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

// dK/dV work: a key tile's list of query tiles is one work unit per K/V
// head; a list much longer than the mean work per SM would hold one SM long
// after the others are done, so the planner may cut the lists longer than a
// length L into ceil(n / L) contiguous segments (never shorter than
// kSegMin tiles).  Segment 0 writes dK, dV; the others write fp32 partials
// into a pool of slots, summed in segment order into dK, dV at the end of the
// dK/dV kernel.  The planner splits only when its bound on the greedy
// makespan of the longest-first order exceeds kSplitOn = 23/20 times the
// mean work per SM, and then picks the longest L whose bound is within
// kSplitTarget = 11/10 times the mean (see plan.cu).
constexpr int kSegMin = 16;
// the final sum of a cut list runs as kSumChunks items of 128 / kSumChunks key rows
constexpr int kSumChunks = 8;
constexpr int kSplitOnNum = 23, kSplitOnDen = 20, kSplitTargetNum = 11, kSplitTargetDen = 10;
// Pool slots (one slot: 128 key rows x all K/V heads x D, for dK and for dV)
// the workspace holds: as many as there are (sample, key tile) units, at
// least 512 / Hkv where the lists are long enough to be cut at all.
__host__ __device__ inline int kv_pool_slots(int batch, int seq_len, int n_kv_heads,
                                             int n_qtiles) {
  const long long units = static_cast<long long>(batch) * (seq_len / kTileN);
  const long long max_extra = units * ((n_qtiles + kSegMin - 1) / kSegMin - 1);
  long long floor_slots = (512 + n_kv_heads - 1) / n_kv_heads;
  if (floor_slots > max_extra) floor_slots = max_extra;
  const long long s = units > floor_slots ? units : floor_slots;
  return static_cast<int>(s < 0 ? 0 : s);
}

// int32 words at kSchedOffset: the forward's work counters (next item, CTAs
// exited), the dK/dV kernel's, the number of dK/dV list slices and of split
// units (written by the planner), and the dK/dV kernel's counter of the
// (split unit, row chunk) sums taken
constexpr int kSchedFwd = 0, kSchedDkdv = 2, kSchedSlices = 4, kSchedSplits = 5, kSchedTail = 6;
// bytes at the start of the workspace: status words [0, 16), the words above [32, 64)
constexpr int kStatusBytes = 64, kSchedOffset = 32;

// Device-visible shape and workspace pointers of one rank's plan.
struct PlanDev {
  int batch, seq_len, cp_size, cp_rank, n_heads, n_kv_heads, head_dim;
  int chunk, local_len, group, tile_pos, n_qtiles, n_ktiles;
  int n_sms;         // SMs of the device (the dK/dV split rule balances over them)
  float scale;       // softmax scale
  float scale_log2;  // scale * log2(e)
  uint64_t timeout_ns;
  uint32_t* status;   // [0] error word (kernels do nothing once set), [1] warning bits
  int32_t* sched;     // work counters and dK/dV list counts (kSched*); zeroed
                      // with the status words by the plan
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
  // dK/dV work list, in launch order: per slice (a unit's list or one
  // segment of it) 8 int32: unit b*n_ktiles + kt, first entry in col_idx,
  // length, segment, split-unit index (-1: not split), pool slot (-1:
  // segment 0 or not split, which write dK, dV), 0, 0
  int32_t* kv_slice;  // [units + kv_cap][8]
  // per split unit: unit, first pool slot (of segment 1), segments, 0
  int32_t* kv_split;  // [units][4]
  int32_t* kv_done;   // [2][units] per split unit: epilogue warps done with its
                      // segments, then sum chunks done
  int kv_cap;         // pool slots (kv_pool_slots)
  float* kv_pool;     // [2][kv_cap][128][Hkv][D] partial dK, then dV
};

struct WorkspaceLayout {
  size_t status, qpos, doc_lo, doc_hi, chunk_order, tile_class, row_cnt, row_ptr, row_idx, col_cnt,
      col_ptr, col_idx, fwd_order, bwd_order, delta, v16, kv_slice, kv_split, kv_done,
      fwd_total, kv_pool, total;
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
// tpk, tpv: the plan's pool of partial dK, dV (segments 1.. of split lists)
cudaError_t launch_dkdv(const dma_plan_s& p, const float* lse, const CUtensorMap& tq,
                        const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                        const CUtensorMap& tdk, const CUtensorMap& tdv, const CUtensorMap& tpk,
                        const CUtensorMap& tpv, float* dk, float* dv, cudaStream_t s);
// to != nullptr: the dQ kernel also computes Delta from O (map `to`, fp32)
// and stores it in the plan's workspace
cudaError_t launch_dq(const dma_plan_s& p, const float* lse, const CUtensorMap& tq,
                      const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                      const CUtensorMap& tdq, const CUtensorMap* to, const float* o,
                      const dma_bf16* dout, dma_bf16* dq, cudaStream_t s);
cudaError_t launch_wait_probe(uint64_t timeout_ns, uint32_t* status, cudaStream_t s);
cudaError_t launch_status_out(const uint32_t* status, uint32_t* out, cudaStream_t s);
cudaError_t launch_cp_chunk_copy(const void* src, void* dst, int batch, int seq_len, int cp_size,
                                 size_t row_bytes, bool to_natural, cudaStream_t s);
}  // namespace dma
