// Context-parallel shard planner and block-mask builder.
//
// Planner: the query-position map of a rank holding chunks i and 2*CP-1-i
// ("The Llama 3 Herd of Models - part 3/16", 3.3.2, "Context parallelism for
// long sequences"), the document start of each local query from the whole
// sequence's document boundaries (review of "Scaling Llama 3 Training with
// Efficient Parallelism Strategies", CP integration: every rank sees the
// full sequence's document information), and validation of cu_doc_lens.
//
// Block-mask builder: for each (query tile, key tile) the class skip / full /
// partial under the causal + document mask.  A query tile covers P = 128/g
// consecutive local positions (never straddling the rank's two chunks, so
// positions are consecutive), whose allowed key ranges are [lo(p), p] with
// both ends non-decreasing in p.  The tile pair is
//   skip    iff no row's range meets [k0, k1],
//   full    iff every row's range contains [k0, k1],
//   partial otherwise,
// then row lists (per query tile, ascending key tiles), column lists (per key
// tile, ascending query tiles) and longest-first launch orders.
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dma {

namespace {

__global__ void plan_positions_kernel(PlanDev p, const int32_t* __restrict__ cu, int n_docs) {
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  const int nthreads = gridDim.x * blockDim.x;
  const int C = p.chunk, Lq = p.local_len, S = p.seq_len;
  const long long total = static_cast<long long>(p.batch) * S;

  // --- validation of the document table
  for (int i = tid; i < n_docs; i += nthreads) {
    if (cu[i + 1] <= cu[i]) atomicCAS(p.status, 0u, static_cast<uint32_t>(DMA_ERR_BAD_DOCS));
  }
  if (tid == 0) {
    if (cu[0] != 0 || static_cast<long long>(cu[n_docs]) != total)
      atomicCAS(p.status, 0u, static_cast<uint32_t>(DMA_ERR_BAD_DOCS));
  }
  for (int b = tid + 1; b < p.batch; b += nthreads) {
    // every sample boundary b*S must be a document boundary
    const long long want = static_cast<long long>(b) * S;
    int lo = 0, hi = n_docs;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu[mid] <= want) lo = mid; else hi = mid - 1;
    }
    if (cu[lo] != want) atomicCAS(p.status, 0u, static_cast<uint32_t>(DMA_ERR_BAD_DOCS));
  }

  // --- column counts start at zero (the block-mask builder adds to them), and
  // so do the dK/dV kernel's per-unit counters of finished segments
  for (int i = tid; i < p.batch * p.n_ktiles; i += nthreads) {
    p.col_cnt[i] = 0;
    p.kv_done[i] = 0;
    p.kv_done[p.batch * p.n_ktiles + i] = 0;
  }

  // --- chunk order (rank-major) and position map
  for (int j = tid; j < 2 * p.cp_size; j += nthreads)
    p.chunk_order[j] = (j & 1) ? (2 * p.cp_size - 1 - (j >> 1)) : (j >> 1);
  const int ca = p.cp_rank, cb = 2 * p.cp_size - 1 - p.cp_rank;
  for (int l = tid; l < Lq; l += nthreads) p.qpos[l] = (l < C) ? (ca * C + l) : (cb * C + (l - C));

  // --- document start of every local query of every sample
  const long long n = static_cast<long long>(p.batch) * Lq;
  for (long long i = tid; i < n; i += nthreads) {
    const int b = static_cast<int>(i / Lq);
    const int l = static_cast<int>(i % Lq);
    const int pos = (l < C) ? (ca * C + l) : (cb * C + (l - C));
    const long long g = static_cast<long long>(b) * S + pos;
    int lo = 0, hi = n_docs - 1;  // last d with cu[d] <= g
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu[mid] <= g) lo = mid; else hi = mid - 1;
    }
    long long start = static_cast<long long>(cu[lo]) - static_cast<long long>(b) * S;
    // keep indices in range even for a malformed table (the status is set)
    if (start < 0) start = 0;
    if (start > pos) start = pos;
    p.doc_lo[i] = static_cast<int32_t>(start);
  }

  // --- end (exclusive) of the document of every key position of every sample
  const long long nk = static_cast<long long>(p.batch) * S;
  for (long long i = tid; i < nk; i += nthreads) {
    const int b = static_cast<int>(i / S);
    const int pos = static_cast<int>(i % S);
    int lo = 0, hi = n_docs - 1;  // last d with cu[d] <= i
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu[mid] <= i) lo = mid; else hi = mid - 1;
    }
    long long end = static_cast<long long>(cu[lo + 1]) - static_cast<long long>(b) * S;
    if (end <= pos) end = pos + 1;  // malformed table: keep the range sane
    if (end > S) end = S;
    p.doc_hi[i] = static_cast<int32_t>(end);
  }
}

// grid (n_qtiles, batch), block 128
__global__ void mask_classify_kernel(PlanDev p) {
  __shared__ int s_q[kTileM], s_lo[kTileM];
  __shared__ int s_cnt;
  const int t = blockIdx.x, b = blockIdx.y;
  const int P = p.tile_pos;
  const int l0 = t * P;
  if (threadIdx.x == 0) s_cnt = 0;
  for (int r = threadIdx.x; r < P; r += blockDim.x) {
    s_q[r] = p.qpos[l0 + r];
    s_lo[r] = p.doc_lo[static_cast<long long>(b) * p.local_len + l0 + r];
  }
  __syncthreads();
  const int q_min = s_q[0], lo_max = s_lo[P - 1];
  int cnt = 0;
  uint8_t* cls_row = p.tile_class + (static_cast<long long>(b) * p.n_qtiles + t) * p.n_ktiles;
  for (int kt = threadIdx.x; kt < p.n_ktiles; kt += blockDim.x) {
    const int k0 = kt * kTileN, k1 = k0 + kTileN - 1;
    // the tile's positions are consecutive (q_min + r) and their document
    // starts non-decreasing: the rows at or after key k0 start at r0, and the
    // smallest document start among them is row r0's
    const int r0 = k0 - q_min < 0 ? 0 : k0 - q_min;
    const bool any = r0 < P && s_lo[r0] <= k1;
    uint8_t c = DMA_TILE_SKIP;
    if (any) c = (lo_max <= k0 && k1 <= q_min) ? DMA_TILE_FULL : DMA_TILE_PARTIAL;
    cls_row[kt] = c;
    if (c != DMA_TILE_SKIP) {
      ++cnt;
      atomicAdd(&p.col_cnt[b * p.n_ktiles + kt], 1);
    }
  }
  atomicAdd(&s_cnt, cnt);
  __syncthreads();
  if (threadIdx.x == 0) p.row_cnt[b * p.n_qtiles + t] = s_cnt;
}

// Block-wide exclusive scan helper (blockDim.x a multiple of 32, at most 1024).
template <typename T>
__device__ T block_exclusive_scan(T v, T* s_tmp, T* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_tmp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    T w = (lane < static_cast<int>(blockDim.x >> 5)) ? s_tmp[lane] : T(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_tmp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const T warp_prefix = (wid > 0) ? s_tmp[wid - 1] : T(0);
  const T incl = x + warp_prefix;
  *total = s_tmp[(blockDim.x >> 5) - 1];
  __syncthreads();
  return incl - v;
}

constexpr int kSortMax = 2048;  // units the one-block sort of the launch orders takes

// Block-wide maximum (blockDim.x a multiple of 32).
template <typename T>
__device__ T block_max(T v, T* s_tmp) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const T y = __shfl_xor_sync(0xffffffffu, v, o);
    v = y > v ? y : v;
  }
  if (lane == 0) s_tmp[wid] = v;
  __syncthreads();
  T r = s_tmp[0];
  for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) r = s_tmp[i] > r ? s_tmp[i] : r;
  __syncthreads();
  return r;
}

// Block-wide sums of K ints per thread: s_red [32 K] scratch, out [K];
// every thread may read out[] on return.
template <int K>
__device__ void block_sum(const int (&v)[K], int* s_red, int* out) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int q = 0; q < K; ++q) {
    int x = v[q];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) s_red[wid * K + q] = x;
  }
  __syncthreads();
  if (threadIdx.x < K) {
    int t = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += s_red[w * K + threadIdx.x];
    out[threadIdx.x] = t;
  }
  __syncthreads();
}

// Sorts s_key[0, npow) ascending (npow a power of two) with a bitonic
// network; the whole block takes part.  The steps with a partner distance of
// 32 or more exchange through shared memory, one barrier each; the
// distances below 32 stay within a warp's 32 consecutive keys and run in
// registers with shuffles (a warp's keys all lie below npow or all above it,
// npow >= 32 and blockDim.x a multiple of 32).
__device__ void bitonic_sort(unsigned long long* s_key, int npow) {
  for (int k = 2; k <= npow; k <<= 1) {
    int j = k >> 1;
    for (; j > 0 && (j >= 32 || npow < 32); j >>= 1) {
      for (int i = threadIdx.x; i < npow; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = s_key[i], b = s_key[ixj];
          if ((a > b) == ((i & k) == 0)) {
            s_key[i] = b;
            s_key[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
    if (j == 0) continue;
    for (int i = threadIdx.x; i < npow; i += blockDim.x) {
      unsigned long long v = s_key[i];
      const bool asc = (i & k) == 0;
      for (int jj = j; jj > 0; jj >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, jj);
        // the lower index of a pair keeps the smaller key when ascending
        const bool keep_min = ((i & jj) == 0) == asc;
        v = keep_min ? (o < v ? o : v) : (o > v ? o : v);
      }
      s_key[i] = v;
    }
    __syncthreads();
  }
}

__device__ __forceinline__ int key_count(unsigned long long k) {
  return 0x7FFFFFFF - static_cast<int>(k >> 32);
}

__device__ __forceinline__ void put_slice(const PlanDev& p, int at, int unit, int first, int n,
                                          int seg, int split, int slot) {
  int4* e = reinterpret_cast<int4*>(p.kv_slice + 8 * static_cast<long long>(at));
  e[0] = make_int4(unit, first, n, seg);
  e[1] = make_int4(split, slot, 0, 0);
}

// The dK/dV work list, from the units (sample, key tile) sorted longest list
// first in s_key (keys as the launch orders' sort leaves them), for n <=
// kSortMax units; block of 1024 threads, two units per thread.
//
// Greedy list scheduling takes each work item, in order, on the SM that
// frees first, so item j starts no later than the work before it divided by
// the SMs, and ends no later than that plus its own length.  With the units'
// K/V heads side by side, unit o (list length c_o, lists before it summing to
// pre_o) thus ends by E_o = (Hkv pre_o + (Hkv - 1) c_o) / P + c_o, against a
// mean of m = Hkv sum(c) / P per SM.  Cutting every list longer than L into
// ceil(c / L) segments leaves the bounds of the units at or after the first
// one not longer than L as they were and caps those before at about their
// end plus L.  So: no cut when every E_o <= kSplitOn m; else L = the length
// at the first position from which every E_o <= kSplitTarget m (at least
// kSegMin), lengthened while the pool cannot hold the segments.  The cut
// units' segments are then ordered by their length among the other units.
// The comparisons run exactly in integers: P E_o against the ratios' numerators
// and denominators times P m = Hkv sum(c).
__device__ void plan_dkdv_slices(const PlanDev& p, unsigned long long* s_key, int n, int npow,
                                 int* s_tmp, long long* s_ll, int* s_red) {
  const long long Hkv = p.n_kv_heads, P = p.n_sms > 0 ? p.n_sms : 1;
  // thread t holds launch positions 2t and 2t + 1
  const int o0 = 2 * static_cast<int>(threadIdx.x);
  int c[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) c[j] = o0 + j < n ? key_count(s_key[o0 + j]) : 0;
  int carry;
  const int pre0 = block_exclusive_scan(c[0] + c[1], s_tmp, &carry);
  const long long hw = Hkv * carry;  // P m
  long long pe[2];                   // P E_o
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int pre = pre0 + (j ? c[0] : 0);
    pe[j] = o0 + j < n ? Hkv * pre + (Hkv - 1) * c[j] + P * c[j] : 0;
  }
  const long long pe_max = block_max(pe[0] > pe[1] ? pe[0] : pe[1], s_ll);
  int L = 0x7FFFFFFF;  // no cut
  if (carry > 0 && kSplitOnDen * pe_max > kSplitOnNum * hw) {
    long long last = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (o0 + j < n && kSplitTargetDen * pe[j] > kSplitTargetNum * hw) last = o0 + j + 1;
    const int last_over = static_cast<int>(block_max(last, s_ll)) - 1;
    const int o_star = last_over + 1 < n ? last_over + 1 : n - 1;
    const int c_first = key_count(s_key[0]);
    L = key_count(s_key[o_star]);
    if (L < kSegMin) L = kSegMin;
    // L grows by at least an eighth per step (a few hundred steps reach any
    // list length) until the pool holds the segments, else no cut; each
    // round of the search tries the next kCand lengths of that sequence
    constexpr int kCand = 8;
    bool fits = false;
    for (int round = 0; round < 512 && !fits && L < c_first; ++round) {
      int cand[kCand], need[kCand];
      int x = L;
#pragma unroll
      for (int q = 0; q < kCand; ++q) {
        cand[q] = x;
        need[q] = 0;
#pragma unroll
        for (int j = 0; j < 2; ++j)
          if (c[j] > x) need[q] += (c[j] + x - 1) / x - 1;
        x += x / 8 > 1 ? x / 8 : 1;
      }
      block_sum<kCand>(need, s_red, s_red + 32 * kCand);
      const int* total = s_red + 32 * kCand;
      // stop at the first candidate that reaches the longest list (no cut)
      // or whose segments the pool holds
      int next = x;
      bool stop = false;
#pragma unroll
      for (int q = 0; q < kCand; ++q) {
        if (stop) continue;
        if (cand[q] >= c_first) {
          stop = true;
          next = cand[q];
        } else if (total[q] <= p.kv_cap) {
          stop = true;
          fits = true;
          next = cand[q];
        }
      }
      __syncthreads();  // every thread has read the totals before the next round
      L = next;
    }
    if (!fits) L = 0x7FFFFFFF;
  }
  if (L == 0x7FFFFFFF) {  // uniform: the launch order, uncut
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (o0 + j < n) {
        const int unit = static_cast<int>(s_key[o0 + j] & 0xFFFFFFFFull);
        put_slice(p, o0 + j, unit, p.col_ptr[unit], c[j], 0, -1, -1);
      }
    }
    if (threadIdx.x == 0) {
      p.sched[kSchedSlices] = n;
      p.sched[kSchedSplits] = 0;
    }
    return;
  }
  __syncthreads();  // every read of the first order is done
  // order the units by their segments' length, longest first
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    if (o0 + j < n) {
      const unsigned int unit = static_cast<unsigned int>(s_key[o0 + j] & 0xFFFFFFFFull);
      const int segs = c[j] > L ? (c[j] + L - 1) / L : 1;
      const int len = (c[j] + segs - 1) / segs;
      s_key[o0 + j] = (static_cast<unsigned long long>(0x7FFFFFFF - len) << 32) | unit;
    }
  }
  __syncthreads();
  bitonic_sort(s_key, npow);
  // slices, split units and pool slots in launch order, from one scan of
  // (slices, split units, pool slots) packed 21 bits apiece (n <= 2048 units
  // and at most as many pool slots as units or 512: each sum < 2^21)
  int unit[2], cnt[2], segs[2];
  long long pk[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    unit[j] = 0;
    cnt[j] = 0;
    segs[j] = 0;
    if (o0 + j < n) {
      unit[j] = static_cast<int>(s_key[o0 + j] & 0xFFFFFFFFull);
      cnt[j] = p.col_cnt[unit[j]];
      segs[j] = cnt[j] > L ? (cnt[j] + L - 1) / L : 1;
    }
    pk[j] = static_cast<long long>(segs[j]) | (static_cast<long long>(segs[j] > 1) << 21) |
            (static_cast<long long>(segs[j] > 1 ? segs[j] - 1 : 0) << 42);
  }
  long long tot;
  const long long base = block_exclusive_scan(pk[0] + pk[1], s_ll, &tot);
  constexpr long long kField = (1ll << 21) - 1;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    if (o0 + j >= n) continue;
    const long long at = base + (j ? pk[0] : 0);
    const int my_at = static_cast<int>(at & kField);
    const int my_split = static_cast<int>((at >> 21) & kField);
    const int my_slot = static_cast<int>((at >> 42) & kField);
    const int first = p.col_ptr[unit[j]];
    if (segs[j] == 1) {
      put_slice(p, my_at, unit[j], first, cnt[j], 0, -1, -1);
    } else {
      // segment sg: q + 1 query tiles for sg < r, else q (q, r = cnt / segs, cnt % segs)
      const int q = cnt[j] / segs[j], r = cnt[j] - q * segs[j];
      int lo = 0;
      for (int sg = 0; sg < segs[j]; ++sg) {
        const int len = q + (sg < r ? 1 : 0);
        put_slice(p, my_at + sg, unit[j], first + lo, len, sg, my_split,
                  sg > 0 ? my_slot + sg - 1 : -1);
        lo += len;
      }
      reinterpret_cast<int4*>(p.kv_split)[my_split] = make_int4(unit[j], my_slot, segs[j], 0);
    }
  }
  if (threadIdx.x == 0) {
    p.sched[kSchedSlices] = static_cast<int>(tot & kField);
    p.sched[kSchedSplits] = static_cast<int>((tot >> 21) & kField);
  }
}

// two blocks of 1024, block 0 for the rows and block 1 for the columns:
// exclusive scan of the counts, then the longest-first launch order when
// there are at most kSortMax units (order_kernel takes larger ones).  The order sorts the keys
// (INT_MAX - count, index) ascending with a bitonic network in shared
// memory: longer lists first, ties by ascending index.  Block 1 then lays
// out the dK/dV work list (plan_dkdv_slices).
__global__ void scan_order_kernel(PlanDev p) {
  __shared__ int s_tmp[32];
  __shared__ long long s_ll[32];
  __shared__ int s_red[33 * 8];
  __shared__ unsigned long long s_key[kSortMax];
  {
    const int which = blockIdx.x;
    const int n = which == 0 ? p.batch * p.n_qtiles : p.batch * p.n_ktiles;
    const int32_t* cnt = which == 0 ? p.row_cnt : p.col_cnt;
    int32_t* ptr = which == 0 ? p.row_ptr : p.col_ptr;
    int carry = 0;
    for (int base = 0; base < n; base += blockDim.x) {
      const int i = base + threadIdx.x;
      const int v = (i < n) ? cnt[i] : 0;
      int tot;
      const int ex = block_exclusive_scan(v, s_tmp, &tot);
      if (i < n) ptr[i] = carry + ex;
      carry += tot;
    }
    if (threadIdx.x == 0) ptr[n] = carry;
    __syncthreads();
    if (n > kSortMax) {  // uniform across the block
      // the dK/dV work list is the launch order itself (kv_slices_kernel)
      if (which == 1 && threadIdx.x == 0) {
        p.sched[kSchedSlices] = n;
        p.sched[kSchedSplits] = 0;
      }
      return;
    }
    int32_t* order = which == 0 ? p.fwd_order : p.bwd_order;
    int npow = 1;
    while (npow < n) npow <<= 1;
    for (int i = threadIdx.x; i < npow; i += blockDim.x)
      s_key[i] = (i < n) ? ((static_cast<unsigned long long>(0x7FFFFFFF - cnt[i]) << 32) |
                            static_cast<unsigned int>(i))
                         : ~0ull;
    __syncthreads();
    bitonic_sort(s_key, npow);
    for (int i = threadIdx.x; i < n; i += blockDim.x)
      order[i] = static_cast<int32_t>(s_key[i] & 0xFFFFFFFFull);
    __syncthreads();
    if (which == 1) plan_dkdv_slices(p, s_key, n, npow, s_tmp, s_ll, s_red);
  }
}

// The dK/dV work list of more than kSortMax units: the launch order, uncut.
__global__ void kv_slices_kernel(PlanDev p) {
  const int o = blockIdx.x * blockDim.x + threadIdx.x;
  if (o >= p.batch * p.n_ktiles) return;
  const int unit = p.bwd_order[o];
  put_slice(p, o, unit, p.col_ptr[unit], p.col_cnt[unit], 0, -1, -1);
}

// grid (n_qtiles + n_ktiles, batch): row lists, then column lists; block 256
__global__ void fill_lists_kernel(PlanDev p) {
  __shared__ int s_tmp[32];
  const int columns = blockIdx.x >= p.n_qtiles;
  const int line = columns ? blockIdx.x - p.n_qtiles : blockIdx.x, b = blockIdx.y;
  const int n = columns ? p.n_qtiles : p.n_ktiles;
  const long long stride = columns ? p.n_ktiles : 1;
  const uint8_t* base =
      columns ? p.tile_class + static_cast<long long>(b) * p.n_qtiles * p.n_ktiles + line
              : p.tile_class + (static_cast<long long>(b) * p.n_qtiles + line) * p.n_ktiles;
  const int list = columns ? b * p.n_ktiles + line : b * p.n_qtiles + line;
  int32_t* out = columns ? p.col_idx + p.col_ptr[list] : p.row_idx + p.row_ptr[list];
  int carry = 0;
  for (int s0 = 0; s0 < n; s0 += blockDim.x) {
    const int i = s0 + threadIdx.x;
    const uint8_t c = (i < n) ? base[i * stride] : static_cast<uint8_t>(DMA_TILE_SKIP);
    const int flag = c != DMA_TILE_SKIP;
    int tot;
    const int ex = block_exclusive_scan(flag, s_tmp, &tot);
    if (flag)
      out[carry + ex] = static_cast<int32_t>(static_cast<uint32_t>(i) |
                                             (c == DMA_TILE_PARTIAL ? kPartialBit : 0u));
    carry += tot;
  }
}

// Longest-first order: position of unit u = #units with larger count +
// #units with equal count and smaller index.
__global__ void order_kernel(const int32_t* __restrict__ cnt, int n, int32_t* __restrict__ order) {
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= n) return;
  const int c = cnt[u];
  int pos = 0;
  for (int j = 0; j < n; ++j) {
    const int cj = cnt[j];
    pos += (cj > c) || (cj == c && j < u);
  }
  order[pos] = u;
}

// Row copy between full-sequence and local layouts.  One block per row.
__global__ void cp_copy_kernel(PlanDev p, const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                               size_t row_bytes, int gather) {
  const long long row = blockIdx.x;  // b*Lq + l
  const int b = static_cast<int>(row / p.local_len);
  const int l = static_cast<int>(row % p.local_len);
  const long long full_row = static_cast<long long>(b) * p.seq_len + p.qpos[l];
  const uint8_t* s = src + (gather ? full_row : row) * row_bytes;
  uint8_t* d = dst + (gather ? row : full_row) * row_bytes;
  if ((row_bytes & 15) == 0 && ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0) {
    const uint4* s4 = reinterpret_cast<const uint4*>(s);
    uint4* d4 = reinterpret_cast<uint4*>(d);
    for (size_t i = threadIdx.x; i < row_bytes / 16; i += blockDim.x) d4[i] = s4[i];
  } else {
    for (size_t i = threadIdx.x; i < row_bytes; i += blockDim.x) d[i] = s[i];
  }
}

// Chunk-order copies between the rank-major layout of an all-gather over the
// CP ranks, [cp_size][batch][2 C][row] (rank r's block holds its chunks r
// and 2 CP - 1 - r), and natural sequence order, [batch][seq_len][row].
// One block per (rank, sample, local row); `to_natural` selects the
// direction.
__global__ void cp_chunk_copy_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                     int batch, int seq_len, int cp_size, size_t row_bytes,
                                     int to_natural) {
  const long long i = blockIdx.x;  // ((rank * batch) + b) * 2C + l
  const int C = seq_len / (2 * cp_size), Lq = 2 * C;
  const int l = static_cast<int>(i % Lq);
  const long long rb = i / Lq;
  const int b = static_cast<int>(rb % batch), r = static_cast<int>(rb / batch);
  const int pos = (l < C) ? (r * C + l) : ((2 * cp_size - 1 - r) * C + (l - C));
  const long long nat = static_cast<long long>(b) * seq_len + pos;
  const uint8_t* s = src + (to_natural ? i : nat) * row_bytes;
  uint8_t* d = dst + (to_natural ? nat : i) * row_bytes;
  if ((row_bytes & 15) == 0 && ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0) {
    const uint4* s4 = reinterpret_cast<const uint4*>(s);
    uint4* d4 = reinterpret_cast<uint4*>(d);
    for (size_t k = threadIdx.x; k < row_bytes / 16; k += blockDim.x) d4[k] = s4[k];
  } else {
    for (size_t k = threadIdx.x; k < row_bytes; k += blockDim.x) d[k] = s[k];
  }
}

// The status a caller sees for a plan: the error word if set, else
// DMA_WARN_V_SATURATED if the warning word says V was saturated, else OK.
__global__ void status_out_kernel(const uint32_t* __restrict__ st, uint32_t* __restrict__ out) {
  const uint32_t e = st[0];
  *out = e != 0u ? e : ((st[1] & 1u) ? static_cast<uint32_t>(DMA_WARN_V_SATURATED) : 0u);
}

__global__ void wait_probe_kernel(uint64_t timeout_ns, uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  WaitCtl ctl{&abort_flag, status, timeout_ns};
  // Phase 0 of this barrier never completes: nothing arrives on it.  The
  // bounded wait gives up after timeout_ns and records DMA_ERR_TIMEOUT.
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0u, ctl);
  __syncthreads();
}

}  // namespace

cudaError_t launch_plan_kernels(const dma_plan_s& pl, cudaStream_t s) {
  const PlanDev& p = pl.d;
  cudaError_t e = cudaMemsetAsync(p.status, 0, kStatusBytes, s);  // status words, work counters
  if (e != cudaSuccess) return e;
  if (p.batch == 0) return cudaSuccess;
  const long long n = static_cast<long long>(p.batch) * p.seq_len;
  int blocks = static_cast<int>((n + 255) / 256);
  if (blocks > 4 * pl.num_sms) blocks = 4 * pl.num_sms;
  if (blocks < 1) blocks = 1;
  plan_positions_kernel<<<blocks, 256, 0, s>>>(p, pl.cu, pl.n_docs);
  mask_classify_kernel<<<dim3(p.n_qtiles, p.batch), 128, 0, s>>>(p);
  scan_order_kernel<<<2, 1024, 0, s>>>(p);
  const int nq = p.batch * p.n_qtiles, nk = p.batch * p.n_ktiles;
  if (nq > kSortMax) order_kernel<<<(nq + 255) / 256, 256, 0, s>>>(p.row_cnt, nq, p.fwd_order);
  if (nk > kSortMax) {
    order_kernel<<<(nk + 255) / 256, 256, 0, s>>>(p.col_cnt, nk, p.bwd_order);
    kv_slices_kernel<<<(nk + 255) / 256, 256, 0, s>>>(p);
  }
  fill_lists_kernel<<<dim3(p.n_qtiles + p.n_ktiles, p.batch), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_cp_copy(const dma_plan_s& pl, const void* src, void* dst, size_t row_bytes,
                           bool gather, cudaStream_t s) {
  const PlanDev& p = pl.d;
  const long long rows = static_cast<long long>(p.batch) * p.local_len;
  if (rows == 0) return cudaSuccess;
  cp_copy_kernel<<<static_cast<unsigned>(rows), 128, 0, s>>>(
      p, static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), row_bytes, gather ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_cp_chunk_copy(const void* src, void* dst, int batch, int seq_len, int cp_size,
                                 size_t row_bytes, bool to_natural, cudaStream_t s) {
  const long long rows = static_cast<long long>(batch) * seq_len;
  if (rows == 0) return cudaSuccess;
  cp_chunk_copy_kernel<<<static_cast<unsigned>(rows), 128, 0, s>>>(
      static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), batch, seq_len, cp_size,
      row_bytes, to_natural ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_status_out(const uint32_t* status, uint32_t* out, cudaStream_t s) {
  status_out_kernel<<<1, 1, 0, s>>>(status, out);
  return cudaGetLastError();
}

cudaError_t launch_wait_probe(uint64_t timeout_ns, uint32_t* status, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(timeout_ns, status);
  return cudaGetLastError();
}

}  // namespace dma
