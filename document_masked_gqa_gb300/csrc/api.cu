// Host implementation of the C ABI declared in include/dma.h: argument
// checks, workspace layout, TMA tensor maps, launches and status handling.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "common.cuh"

namespace {

using dma::WorkspaceLayout;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shape rules; returns DMA_OK or the status to report.
dma_status check_shape(int batch, int seq_len, int cp_size, int cp_rank, int n_heads,
                       int n_kv_heads, int head_dim) {
  if (batch < 0 || seq_len <= 0 || cp_size < 1 || cp_rank < 0 || cp_rank >= cp_size ||
      n_heads <= 0 || n_kv_heads <= 0)
    return DMA_ERR_INVALID_ARG;
  if (seq_len % (2 * cp_size) != 0) return DMA_ERR_INVALID_ARG;
  if (n_heads % n_kv_heads != 0) return DMA_ERR_INVALID_ARG;
  const int g = n_heads / n_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16) return DMA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return DMA_ERR_UNSUPPORTED;
  const int C = seq_len / (2 * cp_size);
  if (C % 64 != 0 || C % (dma::kTileM / g) != 0) return DMA_ERR_UNSUPPORTED;
  // index arithmetic is 32-bit for positions and tiles
  if (static_cast<long long>(batch) * seq_len >= (1ll << 31)) return DMA_ERR_UNSUPPORTED;
  if (static_cast<long long>(batch) * seq_len * n_heads >= (1ll << 31)) return DMA_ERR_UNSUPPORTED;
  return DMA_OK;
}

WorkspaceLayout layout_for(int batch, int seq_len, int cp_size, int n_heads, int n_kv_heads,
                           int head_dim) {
  const int g = n_heads / n_kv_heads;
  const size_t Lq = static_cast<size_t>(seq_len / cp_size);
  const size_t nqt = Lq / (dma::kTileM / g), nkt = static_cast<size_t>(seq_len) / dma::kTileN;
  const size_t B = static_cast<size_t>(batch);
  WorkspaceLayout w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  w.status = take(dma::kStatusBytes);
  w.qpos = take(4 * Lq);
  w.doc_lo = take(4 * B * Lq);
  w.doc_hi = take(4 * B * static_cast<size_t>(seq_len));
  w.chunk_order = take(4 * 2 * static_cast<size_t>(cp_size));
  w.tile_class = take(B * nqt * nkt);
  w.row_cnt = take(4 * B * nqt);
  w.row_ptr = take(4 * (B * nqt + 1));
  w.row_idx = take(4 * B * nqt * nkt);
  w.col_cnt = take(4 * B * nkt);
  w.col_ptr = take(4 * (B * nkt + 1));
  w.col_idx = take(4 * B * nqt * nkt);
  w.fwd_order = take(4 * B * nqt);
  w.bwd_order = take(4 * B * nkt);
  w.delta = take(4 * B * static_cast<size_t>(n_heads) * Lq);
  w.v16 = take(2 * B * static_cast<size_t>(seq_len) * n_kv_heads * head_dim);
  const size_t units = B * nkt;
  const size_t cap = static_cast<size_t>(
      dma::kv_pool_slots(batch, seq_len, n_kv_heads, static_cast<int>(nqt)));
  w.kv_slice = take(32 * (units + cap));
  w.kv_split = take(16 * units);
  w.kv_done = take(2 * 4 * units);
  // the pool of partial dK, dV comes last: only the backward uses it
  w.fwd_total = off;
  w.kv_pool = take(2 * cap * dma::kTileN * n_kv_heads * head_dim * 4);
  w.total = off;
  return w;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dma_status encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
                  const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                  CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return DMA_ERR_CUDA;
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DMA_OK : DMA_ERR_CUDA;
}

// [rows][heads][D] bf16 viewed 3-D; box = 64 columns x g heads x P positions.
dma_status map_rows_heads(CUtensorMap* m, const void* base, const dma::PlanDev& p, int heads,
                          int rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p.head_dim), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(p.head_dim) * 2,
                                 static_cast<cuuint64_t>(heads) * p.head_dim * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(p.group),
                             static_cast<cuuint32_t>(p.tile_pos)};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_128B);
}

// K / V: [B*S][Hkv*D] bf16; box = 64 columns x 128 positions.
dma_status map_kv(CUtensorMap* m, const void* base, const dma::PlanDev& p,
                  CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.n_kv_heads) * p.head_dim,
                              static_cast<cuuint64_t>(p.batch) * p.seq_len};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.n_kv_heads) * p.head_dim * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(dma::kTileN)};
  return encode(m, dt, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// dK / dV (fp32 [rows][Hkv*D]: rows = B*S, or 128 per slot of the plan's
// pool of partials) as TMA store targets: box = 32 columns x 32 key rows,
// 128-byte swizzled (one warp's block of the epilogue).
dma_status map_kv_out_f32(CUtensorMap* m, void* base, const dma::PlanDev& p, long long rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.n_kv_heads) * p.head_dim,
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.n_kv_heads) * p.head_dim * 4};
  const cuuint32_t box[2] = {32, 32};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_128B);
}

// O (fp32 [rows][heads][D]) as a TMA store target: box = 32 columns x g heads
// x 32/g positions (one epilogue warp's 32 rows), 128-byte swizzled.
dma_status map_o_f32(CUtensorMap* m, void* base, const dma::PlanDev& p, int rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p.head_dim),
                              static_cast<cuuint64_t>(p.n_heads), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(p.head_dim) * 4,
                                 static_cast<cuuint64_t>(p.n_heads) * p.head_dim * 4};
  const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(p.group),
                             static_cast<cuuint32_t>(32 / p.group)};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_128B);
}

// Fills a plan's shape, scale, wait limit and device pointers into the
// scratch at `ws` (laid out as `w`), and its device and SM count.  Shared by
// dma_plan (caller's workspace) and dma_attn_fwd_noalloc (the library's
// static scratch), so that the two cannot drift apart.
dma_status init_plan(dma_plan_s& pl, const int32_t* cu_doc_lens, int n_docs, int batch,
                     int seq_len, int cp_size, int cp_rank, int n_heads, int n_kv_heads,
                     int head_dim, float softmax_scale, uint8_t* ws, const WorkspaceLayout& w) {
  dma::PlanDev& p = pl.d;
  p.batch = batch;
  p.seq_len = seq_len;
  p.cp_size = cp_size;
  p.cp_rank = cp_rank;
  p.n_heads = n_heads;
  p.n_kv_heads = n_kv_heads;
  p.head_dim = head_dim;
  p.chunk = seq_len / (2 * cp_size);
  p.local_len = 2 * p.chunk;
  p.group = n_heads / n_kv_heads;
  p.tile_pos = dma::kTileM / p.group;
  p.n_qtiles = p.local_len / p.tile_pos;
  p.n_ktiles = seq_len / dma::kTileN;
  p.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
  p.scale_log2 = p.scale * 1.4426950408889634f;
  p.timeout_ns = 2000000000ull;
  if (const char* env = std::getenv("DMA_WAIT_TIMEOUT_NS")) {
    const unsigned long long t = std::strtoull(env, nullptr, 10);
    if (t > 0) p.timeout_ns = t;
  }
  p.status = reinterpret_cast<uint32_t*>(ws + w.status);
  p.sched = reinterpret_cast<int32_t*>(ws + w.status + dma::kSchedOffset);
  p.qpos = reinterpret_cast<int32_t*>(ws + w.qpos);
  p.doc_lo = reinterpret_cast<int32_t*>(ws + w.doc_lo);
  p.doc_hi = reinterpret_cast<int32_t*>(ws + w.doc_hi);
  p.chunk_order = reinterpret_cast<int32_t*>(ws + w.chunk_order);
  p.tile_class = ws + w.tile_class;
  p.row_cnt = reinterpret_cast<int32_t*>(ws + w.row_cnt);
  p.row_ptr = reinterpret_cast<int32_t*>(ws + w.row_ptr);
  p.row_idx = reinterpret_cast<int32_t*>(ws + w.row_idx);
  p.col_cnt = reinterpret_cast<int32_t*>(ws + w.col_cnt);
  p.col_ptr = reinterpret_cast<int32_t*>(ws + w.col_ptr);
  p.col_idx = reinterpret_cast<int32_t*>(ws + w.col_idx);
  p.fwd_order = reinterpret_cast<int32_t*>(ws + w.fwd_order);
  p.bwd_order = reinterpret_cast<int32_t*>(ws + w.bwd_order);
  p.delta = reinterpret_cast<float*>(ws + w.delta);
  p.v16 = reinterpret_cast<uint16_t*>(ws + w.v16);
  p.kv_slice = reinterpret_cast<int32_t*>(ws + w.kv_slice);
  p.kv_split = reinterpret_cast<int32_t*>(ws + w.kv_split);
  p.kv_done = reinterpret_cast<int32_t*>(ws + w.kv_done);
  p.kv_cap = dma::kv_pool_slots(batch, seq_len, n_kv_heads, p.n_qtiles);
  p.kv_pool = reinterpret_cast<float*>(ws + w.kv_pool);
  pl.cu = cu_doc_lens;
  pl.n_docs = n_docs;
  if (cudaGetDevice(&pl.device) != cudaSuccess ||
      cudaDeviceGetAttribute(&pl.num_sms, cudaDevAttrMultiProcessorCount, pl.device) !=
          cudaSuccess)
    return DMA_ERR_CUDA;
  p.n_sms = pl.num_sms;
  return DMA_OK;
}

// O (fp32 [rows][heads][D]) as a TMA load source: box = 32 columns x g
// heads x P positions (one 128-row query tile, 16 KB), 128-byte swizzled.
dma_status map_o_load(CUtensorMap* m, const void* base, const dma::PlanDev& p, int rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p.head_dim),
                              static_cast<cuuint64_t>(p.n_heads), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(p.head_dim) * 4,
                                 static_cast<cuuint64_t>(p.n_heads) * p.head_dim * 4};
  const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(p.group),
                             static_cast<cuuint32_t>(p.tile_pos)};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_128B);
}

dma_status check_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DMA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return DMA_ERR_CUDA;
  if (major != 10 || minor != 3) return DMA_ERR_UNSUPPORTED;
  return DMA_OK;
}

}  // namespace

extern "C" {

size_t dma_plan_workspace_bytes(int batch, int seq_len, int cp_size, int n_heads, int n_kv_heads,
                                int head_dim, int max_docs) {
  (void)max_docs;
  if (check_shape(batch, seq_len, cp_size, 0, n_heads, n_kv_heads, head_dim) != DMA_OK) return 0;
  return layout_for(batch, seq_len, cp_size, n_heads, n_kv_heads, head_dim).total;
}

dma_status dma_plan(const int32_t* cu_doc_lens, int n_docs, int batch, int seq_len, int cp_size,
                    int cp_rank, int n_heads, int n_kv_heads, int head_dim, float softmax_scale,
                    void* workspace, size_t workspace_bytes, void* stream, dma_plan_t* out) {
  if (!out) return DMA_ERR_INVALID_ARG;
  *out = nullptr;
  const dma_status sh = check_shape(batch, seq_len, cp_size, cp_rank, n_heads, n_kv_heads, head_dim);
  if (sh != DMA_OK) return sh;
  if (!workspace) return DMA_ERR_INVALID_ARG;
  if (batch > 0 && (!cu_doc_lens || n_docs < 1)) return DMA_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return DMA_ERR_INVALID_ARG;
  const WorkspaceLayout w = layout_for(batch, seq_len, cp_size, n_heads, n_kv_heads, head_dim);
  if (workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return DMA_ERR_WORKSPACE;
  const dma_status dv = check_device();
  if (dv != DMA_OK) return dv;

  dma_plan_s* pl = new (std::nothrow) dma_plan_s();
  if (!pl) return DMA_ERR_CUDA;
  if (init_plan(*pl, cu_doc_lens, n_docs, batch, seq_len, cp_size, cp_rank, n_heads, n_kv_heads,
                head_dim, softmax_scale, static_cast<uint8_t*>(workspace), w) != DMA_OK) {
    delete pl;
    return DMA_ERR_CUDA;
  }
  if (dma::launch_plan_kernels(*pl, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    delete pl;
    return DMA_ERR_CUDA;
  }
  *out = pl;
  return DMA_OK;
}

dma_status dma_attn_fwd(dma_plan_t plan, const dma_bf16* q, const dma_bf16* k, const dma_bf16* v,
                        float* o, float* lse, void* stream) {
  if (!plan) return DMA_ERR_INVALID_ARG;
  const dma::PlanDev& p = plan->d;
  if (p.batch == 0) return DMA_OK;
  if (!q || !k || !v || !o || !lse) return DMA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return DMA_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv16, to;
  dma_status st;
  if ((st = map_rows_heads(&tq, q, p, p.n_heads, p.batch * p.local_len)) != DMA_OK) return st;
  if ((st = map_o_f32(&to, o, p, p.batch * p.local_len)) != DMA_OK) return st;
  if ((st = map_kv(&tk, k, p)) != DMA_OK) return st;
  if ((st = map_kv(&tv16, p.v16, p, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != DMA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dma::launch_v_to_f16(*plan, v, s) != cudaSuccess) return DMA_ERR_CUDA;
  return dma::launch_fwd(*plan, tq, tk, tv16, to, o, lse, s) == cudaSuccess ? DMA_OK : DMA_ERR_CUDA;
}

dma_status dma_attn_bwd_delta(dma_plan_t plan, const float* o, const dma_bf16* dout,
                              void* stream) {
  if (!plan) return DMA_ERR_INVALID_ARG;
  if (plan->d.batch == 0) return DMA_OK;
  if (!o || !dout || !aligned16(o) || !aligned16(dout)) return DMA_ERR_INVALID_ARG;
  return dma::launch_delta(*plan, o, dout, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DMA_OK
             : DMA_ERR_CUDA;
}

dma_status dma_attn_bwd_dkdv(dma_plan_t plan, const dma_bf16* q, const dma_bf16* k,
                             const dma_bf16* v, const float* lse, const dma_bf16* dout, float* dk,
                             float* dv, void* stream) {
  if (!plan) return DMA_ERR_INVALID_ARG;
  const dma::PlanDev& p = plan->d;
  if (p.batch == 0) return DMA_OK;
  if (!q || !k || !v || !lse || !dout || !dk || !dv) return DMA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dk) || !aligned16(dv))
    return DMA_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv, tdo;
  dma_status st;
  const int rows = p.batch * p.local_len;
  if ((st = map_rows_heads(&tq, q, p, p.n_heads, rows)) != DMA_OK) return st;
  if ((st = map_rows_heads(&tdo, dout, p, p.n_heads, rows)) != DMA_OK) return st;
  if ((st = map_kv(&tk, k, p)) != DMA_OK) return st;
  if ((st = map_kv(&tv, v, p)) != DMA_OK) return st;
  CUtensorMap tdk, tdv, tpk, tpv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long kv_rows = static_cast<long long>(p.batch) * p.seq_len;
  if ((st = map_kv_out_f32(&tdk, dk, p, kv_rows)) != DMA_OK) return st;
  if ((st = map_kv_out_f32(&tdv, dv, p, kv_rows)) != DMA_OK) return st;
  // the pool of partials (segments 1.. of split lists): dK slots, then dV
  const long long prow = static_cast<long long>(p.kv_cap > 0 ? p.kv_cap : 1) * dma::kTileN;
  if ((st = map_kv_out_f32(&tpk, p.kv_pool, p, prow)) != DMA_OK) return st;
  if ((st = map_kv_out_f32(&tpv, p.kv_pool + static_cast<size_t>(p.kv_cap) * dma::kTileN *
                                                 p.n_kv_heads * p.head_dim,
                           p, prow)) != DMA_OK)
    return st;
  return dma::launch_dkdv(*plan, lse, tq, tk, tv, tdo, tdk, tdv, tpk, tpv, dk, dv, s) ==
                 cudaSuccess
             ? DMA_OK
             : DMA_ERR_CUDA;
}

namespace {
// dQ, and with o != nullptr also Delta (into the plan's workspace), in one
// launch of the dQ kernel
dma_status bwd_dq(dma_plan_t plan, const dma_bf16* q, const dma_bf16* k, const dma_bf16* v,
                  const float* o, const float* lse, const dma_bf16* dout, dma_bf16* dq,
                  void* stream) {
  if (!plan) return DMA_ERR_INVALID_ARG;
  const dma::PlanDev& p = plan->d;
  if (p.batch == 0) return DMA_OK;
  if (!q || !k || !v || !lse || !dout || !dq) return DMA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || (o && !aligned16(o)))
    return DMA_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv, tdo, tdq, to;
  dma_status st;
  const int rows = p.batch * p.local_len;
  if ((st = map_rows_heads(&tq, q, p, p.n_heads, rows)) != DMA_OK) return st;
  if ((st = map_rows_heads(&tdo, dout, p, p.n_heads, rows)) != DMA_OK) return st;
  if ((st = map_rows_heads(&tdq, dq, p, p.n_heads, rows)) != DMA_OK) return st;
  if ((st = map_kv(&tk, k, p)) != DMA_OK) return st;
  if ((st = map_kv(&tv, v, p)) != DMA_OK) return st;
  if (o && (st = map_o_load(&to, o, p, rows)) != DMA_OK) return st;
  return dma::launch_dq(*plan, lse, tq, tk, tv, tdo, tdq, o ? &to : nullptr, o, dout, dq,
                        static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DMA_OK
             : DMA_ERR_CUDA;
}
}  // namespace

dma_status dma_attn_bwd_dq(dma_plan_t plan, const dma_bf16* q, const dma_bf16* k,
                           const dma_bf16* v, const float* lse, const dma_bf16* dout,
                           dma_bf16* dq, void* stream) {
  return bwd_dq(plan, q, k, v, nullptr, lse, dout, dq, stream);
}

dma_status dma_attn_bwd_dq_delta(dma_plan_t plan, const dma_bf16* q, const dma_bf16* k,
                                 const dma_bf16* v, const float* o, const float* lse,
                                 const dma_bf16* dout, dma_bf16* dq, void* stream) {
  if (!o) return DMA_ERR_INVALID_ARG;
  return bwd_dq(plan, q, k, v, o, lse, dout, dq, stream);
}

dma_status dma_attn_bwd(dma_plan_t plan, const dma_bf16* q, const dma_bf16* k, const dma_bf16* v,
                        const float* o, const float* lse, const dma_bf16* dout, dma_bf16* dq,
                        float* dk, float* dv, void* stream) {
  if (!plan) return DMA_ERR_INVALID_ARG;
  if (plan->d.batch == 0) return DMA_OK;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return DMA_ERR_INVALID_ARG;
  // dQ first: its kernel also produces Delta, which dK/dV reads
  dma_status st = dma_attn_bwd_dq_delta(plan, q, k, v, o, lse, dout, dq, stream);
  if (st != DMA_OK) return st;
  return dma_attn_bwd_dkdv(plan, q, k, v, lse, dout, dk, dv, stream);
}

dma_status dma_plan_check(dma_plan_t plan, void* stream) {
  if (!plan) return DMA_ERR_INVALID_ARG;
  uint32_t st[2] = {0u, 0u};  // error word, warning word
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(st, plan->d.status, sizeof(st), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DMA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DMA_ERR_CUDA;
  if (st[0] != 0u) return static_cast<dma_status>(st[0]);
  if (st[1] & 1u) return DMA_WARN_V_SATURATED;
  return DMA_OK;
}

dma_status dma_plan_destroy(dma_plan_t plan) {
  delete plan;
  return DMA_OK;
}

const char* dma_status_str(dma_status s) {
  switch (s) {
    case DMA_OK: return "ok";
    case DMA_ERR_INVALID_ARG: return "invalid argument";
    case DMA_ERR_BAD_DOCS: return "cu_doc_lens violates its contract";
    case DMA_ERR_UNSUPPORTED: return "unsupported shape or device";
    case DMA_ERR_CUDA: return "CUDA call failed";
    case DMA_ERR_TIMEOUT: return "bounded device wait expired";
    case DMA_ERR_WORKSPACE: return "workspace too small or misaligned";
    case DMA_WARN_V_SATURATED:
      return "finite v values beyond +-65504 were saturated in the fp16 copy";
  }
  return "unknown status";
}

dma_status dma_cp_gather(dma_plan_t plan, const void* full, void* local, size_t row_bytes,
                         void* stream) {
  if (!plan || row_bytes == 0) return DMA_ERR_INVALID_ARG;
  if (plan->d.batch == 0) return DMA_OK;
  if (!full || !local) return DMA_ERR_INVALID_ARG;
  return dma::launch_cp_copy(*plan, full, local, row_bytes, true,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DMA_OK
             : DMA_ERR_CUDA;
}

dma_status dma_cp_scatter(dma_plan_t plan, const void* local, void* full, size_t row_bytes,
                          void* stream) {
  if (!plan || row_bytes == 0) return DMA_ERR_INVALID_ARG;
  if (plan->d.batch == 0) return DMA_OK;
  if (!full || !local) return DMA_ERR_INVALID_ARG;
  return dma::launch_cp_copy(*plan, local, full, row_bytes, false,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DMA_OK
             : DMA_ERR_CUDA;
}

namespace {
dma_status cp_chunk_copy(const void* src, void* dst, int batch, int seq_len, int cp_size,
                         size_t row_bytes, bool to_natural, void* stream) {
  if (batch < 0 || seq_len <= 0 || cp_size < 1 || row_bytes == 0 ||
      seq_len % (2 * cp_size) != 0)
    return DMA_ERR_INVALID_ARG;
  if (batch == 0) return DMA_OK;
  if (!src || !dst) return DMA_ERR_INVALID_ARG;
  if (static_cast<long long>(batch) * seq_len >= (1ll << 31)) return DMA_ERR_UNSUPPORTED;
  return dma::launch_cp_chunk_copy(src, dst, batch, seq_len, cp_size, row_bytes, to_natural,
                                   static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DMA_OK
             : DMA_ERR_CUDA;
}
}  // namespace

dma_status dma_cp_unpermute(const void* gathered, void* full, int batch, int seq_len,
                            int cp_size, size_t row_bytes, void* stream) {
  return cp_chunk_copy(gathered, full, batch, seq_len, cp_size, row_bytes, true, stream);
}

dma_status dma_cp_permute(const void* full, void* gathered, int batch, int seq_len,
                          int cp_size, size_t row_bytes, void* stream) {
  return cp_chunk_copy(full, gathered, batch, seq_len, cp_size, row_bytes, false, stream);
}

dma_status dma_plan_get_view(dma_plan_t plan, dma_plan_view* out) {
  if (!plan || !out) return DMA_ERR_INVALID_ARG;
  const dma::PlanDev& p = plan->d;
  out->batch = p.batch;
  out->seq_len = p.seq_len;
  out->cp_size = p.cp_size;
  out->cp_rank = p.cp_rank;
  out->n_heads = p.n_heads;
  out->n_kv_heads = p.n_kv_heads;
  out->head_dim = p.head_dim;
  out->chunk = p.chunk;
  out->local_len = p.local_len;
  out->group = p.group;
  out->q_tile_positions = p.tile_pos;
  out->n_qtiles = p.n_qtiles;
  out->n_ktiles = p.n_ktiles;
  out->softmax_scale = p.scale;
  out->qpos = p.qpos;
  out->doc_lo = p.doc_lo;
  out->chunk_order = p.chunk_order;
  out->tile_class = p.tile_class;
  out->row_ptr = p.row_ptr;
  out->row_idx = p.row_idx;
  out->col_ptr = p.col_ptr;
  out->col_idx = p.col_idx;
  out->fwd_order = p.fwd_order;
  out->bwd_order = p.bwd_order;
  out->status = p.status;
  out->kv_slices = p.kv_slice;
  out->kv_splits = p.kv_split;
  out->counts = p.sched + dma::kSchedSlices;
  out->n_sms = p.n_sms;
  out->kv_pool_slots = p.kv_cap;
  return DMA_OK;
}

dma_status dma_plan_set_wait_timeout(dma_plan_t plan, uint64_t timeout_ns) {
  if (!plan || timeout_ns == 0) return DMA_ERR_INVALID_ARG;
  plan->d.timeout_ns = timeout_ns;
  return DMA_OK;
}

dma_status dma_debug_wait_probe(uint64_t timeout_ns, uint32_t* status_dev, void* stream) {
  if (!status_dev || timeout_ns == 0) return DMA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(status_dev, 0, sizeof(uint32_t), s) != cudaSuccess) return DMA_ERR_CUDA;
  if (dma::launch_wait_probe(timeout_ns, status_dev, s) != cudaSuccess) return DMA_ERR_CUDA;
  uint32_t st = 0;
  if (cudaMemcpyAsync(&st, status_dev, sizeof(st), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DMA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DMA_ERR_CUDA;
  return static_cast<dma_status>(st);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free forward.
//
// For callers that cannot allocate device memory at all: code running where
// the allocator is off limits (inside a framework's memory pool that it must
// not grow, a plugin host that forbids cudaMalloc, or a process that has to
// keep its footprint fixed).  Every other entry point needs a caller-owned
// plan workspace; this one builds the plan and the fp16 copy of V in a fixed
// scratch array compiled into the library instead.
namespace {

// 64 MiB of scratch per device, held by every GPU that loads the library
// until the process exits.  It fits the plan plus the fp16 V copy of, e.g.,
// an 8K-token batch of 2 with 8 K/V heads of 128 (about 34 MiB), or one
// 128K-token sample with one K/V head of 128 at CP = 16 (about 42 MiB); at
// CP = 1 the same sample needs about 186 MiB, mostly its tile lists.
// dma_plan_workspace_bytes gives the exact need of a shape.
constexpr size_t kNoAllocScratchBytes = 64ull << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// In host code `g_noalloc_scratch` is only a stand-in for the symbol, not a
// device address: its device address is looked up per device, with that
// device current.  Only a successful lookup is kept; a failed one (made under
// stream capture, say) is retried by the next call.
constexpr int kNoAllocMaxDevices = 64;
void* g_noalloc_ptr[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

void* noalloc_scratch(int dev) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess) {
      (void)cudaGetLastError();  // clear the (non-sticky) error for the caller
      return nullptr;
    }
    g_noalloc_ptr[dev] = a;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" dma_status dma_attn_fwd_noalloc(const int32_t* cu_doc_lens, int n_docs, int batch,
                                           int seq_len, int cp_size, int cp_rank, int n_heads,
                                           int n_kv_heads, int head_dim, float softmax_scale,
                                           const dma_bf16* q, const dma_bf16* k,
                                           const dma_bf16* v, float* o, float* lse,
                                           uint32_t* status_dev, void* stream) {
  const dma_status sh = check_shape(batch, seq_len, cp_size, cp_rank, n_heads, n_kv_heads, head_dim);
  if (sh != DMA_OK) return sh;
  if (batch == 0) return DMA_OK;
  if (!cu_doc_lens || n_docs < 1 || !q || !k || !v || !o || !lse) return DMA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return DMA_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return DMA_ERR_INVALID_ARG;
  const WorkspaceLayout w = layout_for(batch, seq_len, cp_size, n_heads, n_kv_heads, head_dim);
  // the forward needs the workspace up to the backward's pool of partials
  if (w.fwd_total > kNoAllocScratchBytes) return DMA_ERR_WORKSPACE;  // shape needs > 64 MiB
  const dma_status dv = check_device();
  if (dv != DMA_OK) return dv;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DMA_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return DMA_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(noalloc_scratch(dev));
  if (!ws) return DMA_ERR_CUDA;

  // the plan lives on this stack frame and in the scratch array
  dma_plan_s pl{};
  if (init_plan(pl, cu_doc_lens, n_docs, batch, seq_len, cp_size, cp_rank, n_heads, n_kv_heads,
                head_dim, softmax_scale, ws, w) != DMA_OK)
    return DMA_ERR_CUDA;
  pl.d.kv_pool = nullptr;  // past the scratch; only the backward would use it
  const dma::PlanDev& p = pl.d;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the plan kernels clear what must start at zero (status word, column
  // counts) and write every other array before it is read
  if (dma::launch_plan_kernels(pl, s) != cudaSuccess) return DMA_ERR_CUDA;
  CUtensorMap tq, tk, tv16, to;
  dma_status st;
  if ((st = map_rows_heads(&tq, q, p, p.n_heads, p.batch * p.local_len)) != DMA_OK) return st;
  if ((st = map_o_f32(&to, o, p, p.batch * p.local_len)) != DMA_OK) return st;
  if ((st = map_kv(&tk, k, p)) != DMA_OK) return st;
  if ((st = map_kv(&tv16, p.v16, p, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != DMA_OK) return st;
  if (dma::launch_v_to_f16(pl, v, s) != cudaSuccess) return DMA_ERR_CUDA;
  if (dma::launch_fwd(pl, tq, tk, tv16, to, o, lse, s) != cudaSuccess) return DMA_ERR_CUDA;
  if (status_dev && dma::launch_status_out(p.status, status_dev, s) != cudaSuccess)
    return DMA_ERR_CUDA;
  return DMA_OK;
}
