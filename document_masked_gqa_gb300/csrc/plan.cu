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

  // --- column counts start at zero (the block-mask builder adds to them)
  for (int i = tid; i < p.batch * p.n_ktiles; i += nthreads) p.col_cnt[i] = 0;

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
__device__ int block_exclusive_scan(int v, int* s_tmp, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_tmp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = (lane < (blockDim.x >> 5)) ? s_tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_tmp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int warp_prefix = (wid > 0) ? s_tmp[wid - 1] : 0;
  const int incl = x + warp_prefix;
  *total = s_tmp[(blockDim.x >> 5) - 1];
  __syncthreads();
  return incl - v;
}

constexpr int kSortMax = 2048;  // units the one-block sort of the launch orders takes

// two blocks of 1024, block 0 for the rows and block 1 for the columns:
// exclusive scan of the counts, then the longest-first launch order when
// there are at most kSortMax units (order_kernel takes larger ones).  The order sorts the keys
// (INT_MAX - count, index) ascending with a bitonic network in shared
// memory: longer lists first, ties by ascending index.
__global__ void scan_order_kernel(PlanDev p) {
  __shared__ int s_tmp[32];
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
    if (n > kSortMax) return;  // uniform across the block
    int32_t* order = which == 0 ? p.fwd_order : p.bwd_order;
    int npow = 1;
    while (npow < n) npow <<= 1;
    for (int i = threadIdx.x; i < npow; i += blockDim.x)
      s_key[i] = (i < n) ? ((static_cast<unsigned long long>(0x7FFFFFFF - cnt[i]) << 32) |
                            static_cast<unsigned int>(i))
                         : ~0ull;
    __syncthreads();
    for (int k = 2; k <= npow; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
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
    }
    for (int i = threadIdx.x; i < n; i += blockDim.x)
      order[i] = static_cast<int32_t>(s_key[i] & 0xFFFFFFFFull);
    __syncthreads();
  }
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
  if (nk > kSortMax) order_kernel<<<(nk + 255) / 256, 256, 0, s>>>(p.col_cnt, nk, p.bwd_order);
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
