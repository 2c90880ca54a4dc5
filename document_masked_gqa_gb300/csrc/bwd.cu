// Backward kernels: causal + document-masked GQA attention for one CP rank.
//
// The backward recomputes the scores from Q, K and the forward's row
// log-sum-exp instead of storing them ("Training Infrastructure and
// Systems", "FlashAttention: never write the score matrix", "Tiling": the
// backward recomputes the scores).  With P = exp(scale*S - LSE):
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - Delta),  Delta = rowsum(dO*O),
//   dQ = scale * dS K,  dK = scale * dS^T Q.
// dK and dV are this rank's partial sums (its own query rows only), kept in
// fp32 ("The Llama 3 Herd of Models - part 3/16", 3.3.2 "Numerical
// stability": gradients accumulated and reduce-scattered in FP32).
//
// Kernels (the default backward launches dq_kernel<D, true> and then
// dkdv_kernel):
//   dq_kernel     work item = (query tile, K/V head): Q and dO are copied into
//                 TMEM (tcgen05.cp by the S and dP issuers); the item walks
//                 the row list of key tiles; S, dP and the dQ accumulator in
//                 TMEM; four row warpgroups split each tile's key columns.
//                 With kDelta it also computes Delta at each item's start and
//                 stores it for the dK/dV pass.
//   dkdv_kernel   work item = (key tile or a segment of its list, K/V
//                 head): K and V stay in shared memory; the item walks the
//                 column list of query tiles (all g heads of the group
//                 packed in each 128-row tile, so the GQA reduction over the
//                 group happens inside the accumulation), a whole 128-row
//                 query tile per step shared by two element-wise
//                 warpgroups; dV, dK accumulate in TMEM.  Segments 1.. of a
//                 cut list leave fp32 partials, which the element-wise warps
//                 add into dK, dV in segment order once all items are taken.
//   delta_kernel  Delta[b, h, l] = sum_d dO * O as a pass of its own
//                 (HBM-bound), for the split entry points.
// Both attention kernels are persistent (one CTA per SM) with one TMA
// producer thread, one tcgen05-issuing thread per product on its own warp,
// element-wise warpgroups and an epilogue that overlaps the next item;
// bounded waits everywhere.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dma {
namespace {

constexpr int kMaxSmem = 232448;  // 227 KB opt-in per block on sm_103
// dK/dV register split of the 512 threads launched at 128 registers each: the
// producer-issuer warpgroup (warps 0-3) and the epilogue warpgroup give
// registers to the element-wise warps.  Each warpgroup sets its share at one
// call site at the top of its branch, the same count for its four warps.
constexpr uint32_t kDkdvCtlRegs = 64, kDkdvEwRegs = 184, kDkdvEpiRegs = 80;
static_assert(4 * kDkdvCtlRegs + 8 * kDkdvEwRegs + 4 * kDkdvEpiRegs <= 16 * 128,
              "dK/dV register split exceeds the launch's 512 x 128 registers");
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// Bits t in [lo, hi) of a 32-column chunk (clamped to the chunk).
__device__ __forceinline__ uint32_t range_bits(int lo, int hi) {
  lo = max(lo, 0);
  hi = min(hi, 32);
  if (hi <= lo) return 0u;
  const uint32_t upto_hi = (hi >= 32) ? 0xFFFFFFFFu : ((1u << hi) - 1u);
  const uint32_t below_lo = (1u << lo) - 1u;
  return upto_hi & ~below_lo;
}

// Warp-uniform bounded wait (every lane waits; all agree on the outcome).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& c) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, c));
}

// ---------------------------------------------------------------- Delta

// Delta[(b*Hq + h)*Lq + l] = sum_d dO[b,l,h,d] * O[b,l,h,d] (O fp32, dO bf16);
// D/8 threads per row, 8 elements each.
template <int D>
__global__ void delta_kernel(const float* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                             float* __restrict__ delta, int rows, int n_heads, int local_len) {
  constexpr int TPR = D / 8;
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / TPR;
  const int sub = threadIdx.x % TPR;
  float acc = 0.f;
  if (row < rows) {
    const float4 a0 = reinterpret_cast<const float4*>(o + row * D)[2 * sub];
    const float4 a1 = reinterpret_cast<const float4*>(o + row * D)[2 * sub + 1];
    const uint4 b = reinterpret_cast<const uint4*>(dout + row * D)[sub];
    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(av[2 * i], __uint_as_float(bw[i] << 16), acc);
      acc = fmaf(av[2 * i + 1], __uint_as_float(bw[i] & 0xFFFF0000u), acc);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && sub == 0) {
    const long long bl = row / n_heads;  // b*Lq + l
    const int h = static_cast<int>(row % n_heads);
    const long long b = bl / local_len, l = bl % local_len;
    delta[(b * n_heads + h) * local_len + l] = acc;
  }
}

// ---------------------------------------------------------------- dK / dV

// 32 columns of one key row, first phase: P = exp2(S * scale*log2e -
// LSE*log2e) (zero where the mask bit is clear when kMasked), packed as bf16
// pairs: the A operand of dV += P^T dO, and kept for dS = P (dP - Delta).
// nlse_c holds -LSE*log2e per column.
template <bool kMasked>
__device__ __forceinline__ void p_chunk32(const uint32_t* su, const float4* nlse_c,
                                          uint32_t allow, float sl2, uint32_t* pb) {
  const uint64_t sl2x2 = f2(sl2, sl2);
#pragma unroll
  for (int q = 0; q < 32; q += 4) {
    const float4 l4 = nlse_c[q >> 2];
    float x0, x1, x2, x3;
    f2_split(f2_fma(f2(__uint_as_float(su[q]), __uint_as_float(su[q + 1])), sl2x2, f2(l4.x, l4.y)),
             x0, x1);
    f2_split(f2_fma(f2(__uint_as_float(su[q + 2]), __uint_as_float(su[q + 3])), sl2x2,
                    f2(l4.z, l4.w)),
             x2, x3);
    float pv[4] = {ex2(x0), ex2(x1), ex2(x2), ex2(x3)};
    if (kMasked) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (!((allow >> (q + u)) & 1u)) pv[u] = 0.f;
    }
    pb[q >> 1] = pack_bf16(pv[0], pv[1]);
    pb[(q >> 1) + 1] = pack_bf16(pv[2], pv[3]);
  }
}

// Second phase: dS = P (dP - Delta) for the same 32 columns, packed bf16
// (the A operand of dK += dS^T Q).  P comes back from its bf16 pairs (a bf16
// widens to fp32 by a 16-bit shift), the values dV was computed with.
__device__ __forceinline__ void ds_chunk32(const uint32_t* du, const uint32_t* pb,
                                           const float4* del_c, uint32_t* pd) {
#pragma unroll
  for (int q = 0; q < 32; q += 4) {
    const float4 d4 = del_c[q >> 2];
    const uint32_t w0 = pb[q >> 1], w1 = pb[(q >> 1) + 1];
    float d0, d1, d2, d3;
    f2_split(f2_mul(f2(__uint_as_float(w0 << 16), __uint_as_float(w0 & 0xFFFF0000u)),
                    f2_sub(f2(__uint_as_float(du[q]), __uint_as_float(du[q + 1])), f2(d4.x, d4.y))),
             d0, d1);
    f2_split(f2_mul(f2(__uint_as_float(w1 << 16), __uint_as_float(w1 & 0xFFFF0000u)),
                    f2_sub(f2(__uint_as_float(du[q + 2]), __uint_as_float(du[q + 3])),
                           f2(d4.z, d4.w))),
             d2, d3);
    pd[q >> 1] = pack_bf16(d0, d1);
    pd[(q >> 1) + 1] = pack_bf16(d2, d3);
  }
}

//
// dK/dV works a whole query tile at a time.  Query tiles alternate between
// two 128-column TMEM buffers: tile t uses buffer t % 2 for S^T = K Q^T,
// then for dP^T = V dO^T, then for P^T and dS^T.  The element-wise
// warpgroups (thread = key, warpgroup w = query columns [64w, 64w + 64))
// load S^T into registers, which lets dP^T be computed into the same
// columns while they turn S^T into P^T (bf16 pairs, kept in registers).
// Then they load dP^T, write P^T over the first 32 of the columns they read
// (dV += P^T dO starts) and dS^T = P^T (dP^T - Delta) over the other 32 (dK
// += dS^T Q starts, in two halves).  The buffer takes tile t + 2's S^T once
// dV(t) and dK(t) are done.  With two tiles in flight the next tile's S^T is
// always ready when the element-wise warps finish a tile, and its dP^T is
// computed while they exponentiate.
template <int D>
struct DkdvCfg {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kRegion = 16384;
  static constexpr int kChunks = D / 64;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;         // 2 stages
  static constexpr int kDO = kQ + 2 * kTile;    // 2 stages
  // dK / dV staging of the epilogue warps: per warp one 4 KB block of
  // 32 rows x 32 fp32 in the 128-byte swizzled layout of a TMA store
  static constexpr int kStage = kDO + 2 * kTile;
  // per element-wise warp: [2 stages][64 -LSE*log2e, 64 Delta]
  static constexpr int kCOL = kStage + 4 * 4096;
  static constexpr int kBar = kCOL + 8 * 2 * 128 * 4;
  // work items published by the producer to the other roles (ItemRing)
  static constexpr int kRing = 8;
  static constexpr int kNumBars = 26 + 2 * kRing;
  static constexpr int kMisc = kBar + kNumBars * 8;
  // kMisc: TMEM address, abort flag, then the ring's slots, then the split
  // unit the element-wise warps sum (two words, by round parity)
  static constexpr int kUnit = 16 + 4 * kRing;
  static constexpr int kNeed = kMisc + kUnit + 8;
  static constexpr int kAlloc = (kNeed + 1024 <= kMaxSmem) ? kNeed + 1024 : kMaxSmem;
  // TMEM: dV [0,128), dK [128,256), tile buffers [256,384) and [384,512);
  // once dP^T has been read, warpgroup w's P^T sits in columns
  // [64w, 64w + 32) of the tile's buffer and its dS^T in the next 32
  static constexpr uint32_t kTmemDV = 0, kTmemDK = 128, kTmemBuf = 256;
  static_assert(kNeed <= kMaxSmem, "dK/dV shared-memory layout exceeds 227 KB");
};

// Work item `item` of the dK/dV pass: slice item / Hkv of the plan's work
// list (a key tile's list of query tiles, or one segment of a list the
// planner cut) times K/V head item % Hkv (the heads of one slice side by
// side).  `split` >= 0: the unit's segments are summed at the end of the
// kernel; `slot` >= 0: this segment writes its partial into that pool slot
// (segment 0 writes dK, dV).
struct DkdvItem {
  int b, kvh, kt, n, seg, split, slot;
  const int32_t* list;
};
__device__ __forceinline__ DkdvItem dkdv_item(const PlanDev& p, int item) {
  DkdvItem it;
  const int s = item / p.n_kv_heads;
  it.kvh = item - s * p.n_kv_heads;
  const int4* e = reinterpret_cast<const int4*>(p.kv_slice) + 2 * s;
  const int4 a = e[0], c = e[1];
  it.b = a.x / p.n_ktiles;
  it.kt = a.x - it.b * p.n_ktiles;
  it.list = p.col_idx + a.y;
  it.n = a.z;
  it.seg = a.w;
  it.split = c.x;
  it.slot = c.y;
  return it;
}

// Rows [rows0, rows0 + 128 / kSumChunks) of split unit u's dK, dV (all K/V
// heads) = segment 0's values, already there, plus the pool partials of
// segments 1, 2, ... added in that order (the same on every run).  Threads
// t of nt, two float4 positions and four segments' loads in flight each;
// every load and store bypasses L1 (the partials were written by other SMs
// during this launch).
template <int D>
__device__ __forceinline__ void kv_sum_chunk(const PlanDev& p, int u, int chunk, float* dk,
                                             float* dv, int t, int nt) {
  const int4 e = reinterpret_cast<const int4*>(p.kv_split)[u];
  const int unit = e.x, slot0 = e.y, segs = e.z;
  const long long row_f = static_cast<long long>(p.n_kv_heads) * D;  // floats per key row
  const long long tile = kTileN * row_f;
  constexpr int kRows = kTileN / kSumChunks;
  const int b = unit / p.n_ktiles, kt = unit - b * p.n_ktiles;
  const long long row0 = static_cast<long long>(b) * p.seq_len +
                         static_cast<long long>(kt) * kTileN + chunk * kRows;
  const int n4 = static_cast<int>(kRows * row_f / 4);
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    float4* out = reinterpret_cast<float4*>((which ? dv : dk) + row0 * row_f);
    const float4* part = reinterpret_cast<const float4*>(
        p.kv_pool + (static_cast<long long>(which) * p.kv_cap + slot0) * tile +
        chunk * kRows * row_f);
    const long long seg_stride = tile / 4;  // float4 per pool slot
#pragma unroll 1
    for (int i0 = t; i0 < n4; i0 += 2 * nt) {
      const int i1 = i0 + nt;
      const bool has1 = i1 < n4;
      float4 a0 = __ldcg(out + i0);
      float4 a1 = has1 ? __ldcg(out + i1) : make_float4(0.f, 0.f, 0.f, 0.f);
      int sg = 1;
#pragma unroll 1
      for (; sg + 3 < segs; sg += 4) {
        float4 x[4], y[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4* src = part + (sg + k - 1) * seg_stride;
          x[k] = __ldcg(src + i0);
          if (has1) y[k] = __ldcg(src + i1);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // in segment order
          a0.x += x[k].x; a0.y += x[k].y; a0.z += x[k].z; a0.w += x[k].w;
          if (has1) { a1.x += y[k].x; a1.y += y[k].y; a1.z += y[k].z; a1.w += y[k].w; }
        }
      }
      for (; sg < segs; ++sg) {
        const float4* src = part + (sg - 1) * seg_stride;
        const float4 x = __ldcg(src + i0);
        a0.x += x.x; a0.y += x.y; a0.z += x.z; a0.w += x.w;
        if (has1) {
          const float4 y = __ldcg(src + i1);
          a1.x += y.x; a1.y += y.y; a1.z += y.z; a1.w += y.w;
        }
      }
      __stcg(out + i0, a0);
      if (has1) __stcg(out + i1, a1);
    }
  }
}

// Persistent: the producer thread takes work items from the plan's counter
// one at a time and publishes them to every other role (ItemRing).  Every
// role keeps the same counters across non-empty items: query tiles so far
// (tbase: the Q / dO stage and the parity of every per-tile barrier) and
// items so far (ibase: parity of kv_full, kv_empty, acc_done, acc_free).
template <int D>
__global__ void __launch_bounds__(512, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv,
                const __grid_constant__ CUtensorMap tpk, const __grid_constant__ CUtensorMap tpv,
                const PlanDev p, const float* __restrict__ lse, float* dk, float* dv) {
  using Cfg = DkdvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  int32_t* const ctr = p.sched + kSchedDkdv;
  int32_t* const tail = p.sched + kSchedTail;
  if (__syncthreads_or(threadIdx.x == 0 &&
                       *reinterpret_cast<volatile uint32_t*>(p.status) != 0u)) {
    if (threadIdx.x == 0) items_exit(ctr, tail);
    return;
  }
  if (pad + Cfg::kNeed > static_cast<uint32_t>(Cfg::kAlloc)) {  // cannot lay out the tiles
    if (threadIdx.x == 0) {
      atomicCAS(p.status, 0u, static_cast<uint32_t>(DMA_ERR_UNSUPPORTED));
      items_exit(ctr, tail);
    }
    return;
  }
  uint8_t* smem = smem_raw + pad;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.group, P = p.tile_pos, Lq = p.local_len;

  uint8_t* sK = smem + Cfg::kK;
  uint8_t* sV = smem + Cfg::kV;
  uint8_t* sQ = smem + Cfg::kQ;
  uint8_t* sDO = smem + Cfg::kDO;
  float* sCOL = reinterpret_cast<float*>(smem + Cfg::kCOL);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBar);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;     // [2] per query-tile stage (tile t: stage t % 2)
  uint64_t* q_empty = bars + 3;    // [2]
  uint64_t* do_full = bars + 5;    // [2]
  uint64_t* do_empty = bars + 7;   // [2]
  // per TMEM tile buffer (tile t: buffer t % 2, phase t / 2)
  uint64_t* s_full = bars + 9;     // [2] S^T computed
  uint64_t* s_read = bars + 11;    // [2] the element-wise warps hold S^T in registers
  uint64_t* dp_full = bars + 13;   // [2] dP^T computed
  uint64_t* p_full = bars + 15;    // [2] P^T written into the buffer
  uint64_t* ds_full = bars + 17;   // [2 buffers][2 halves] dS^T written: query columns
                                   // [0, 32) and [64, 96) of the tile, then the rest
  uint64_t* buf_free = bars + 21;  // [2] dV and dK of the buffer's tile done
  uint64_t* acc_done = bars + 23;  // an item's dV, dK complete
  uint64_t* kv_empty = bars + 24;  // an item's last S^T and dP^T done (two commits)
  uint64_t* acc_free = bars + 25;  // the epilogue warps have read an item's dV, dK
  uint64_t* item_full = bars + 26;  // [kRing]
  uint64_t* item_empty = item_full + Cfg::kRing;
  const ItemRing<Cfg::kRing> ring{reinterpret_cast<volatile int*>(smem + Cfg::kMisc + 16), item_full,
                                  item_empty};
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + Cfg::kMisc + 4);

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&do_full[i], 1);
      mbar_init(&do_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&dp_full[i], 1);
      mbar_init(&buf_free[i], 1);
      mbar_init(&s_read[i], 8);     // one arrival per element-wise warp
      mbar_init(&p_full[i], 8);
      mbar_init(&ds_full[2 * i], 8);
      mbar_init(&ds_full[2 * i + 1], 8);
    }
    mbar_init(acc_done, 1);
    mbar_init(kv_empty, 2);
    mbar_init(acc_free, 4);
    // readers of the item ring: three issuers, eight element-wise warps, four
    // epilogue warps
    for (int i = 0; i < Cfg::kRing; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], 15);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  if (warp < 4) {
    // warpgroup 0: producer (warp 0), issuers (warps 1-3)
    reg_dealloc<kDkdvCtlRegs>();
    if (warp == 0) {
      if (lane == 0) {
        // --------------------------------------- producer: K, V, then Q, dO
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tdo);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        int last_t = -1, ibase = 0, tbase = 0;
        bool kv_pending = false, ok = true;
        // the next index is taken as an item's last query tile loads: late, so
        // that no SM holds an item it cannot start for long (a long item would
        // otherwise pin a second one behind it), yet early enough to hide the
        // atomic's latency.  Every index is published, empty items too (the
        // epilogue writes their zero rows).
        const int n_items = p.sched[kSchedSlices] * p.n_kv_heads;
        int next_idx = take_item(ctr);
        for (int rk = 0; ok; ++rk) {
          const int item = next_idx < n_items ? next_idx : -1;
          if (!ring.put(rk, item, ctl)) { ok = false; break; }
          if (item < 0) break;
          const DkdvItem it = dkdv_item(p, item);
          if (it.n == 0) {
            next_idx = take_item(ctr);
            continue;
          }
          const int krow0 = it.b * p.seq_len + it.kt * kTileN;
          kv_pending = false;
          // K and V of the previous item are read until its last S^T / dP^T
          if (ibase > 0 && !mbar_wait(kv_empty, (ibase - 1) & 1, ctl)) { ok = false; break; }
          mbar_arrive_expect_tx(kv_full, 2 * Cfg::kTile);
#pragma unroll
          for (int c = 0; c < Cfg::kChunks; ++c) {
            tma_load_2d(sK + c * Cfg::kRegion, &tk, kv_full, it.kvh * D + c * 64, krow0);
            tma_load_2d(sV + c * Cfg::kRegion, &tv, kv_full, it.kvh * D + c * 64, krow0);
          }
          kv_pending = true;
          for (int i = 0; i < it.n; ++i) {
            const int ig = tbase + i, st = ig & 1;
            const uint32_t ph = (ig >> 1) & 1;
            const int qt = static_cast<int>(static_cast<uint32_t>(it.list[i]) & kIndexMask);
            if (!mbar_wait(&q_empty[st], ph ^ 1u, ctl)) { ok = false; break; }
            mbar_arrive_expect_tx(&q_full[st], Cfg::kTile);
#pragma unroll
            for (int c = 0; c < Cfg::kChunks; ++c)
              tma_load_3d(sQ + st * Cfg::kTile + c * Cfg::kRegion, &tq, &q_full[st], c * 64,
                          it.kvh * g, it.b * Lq + qt * P);
            if (!mbar_wait(&do_empty[st], ph ^ 1u, ctl)) { ok = false; break; }
            mbar_arrive_expect_tx(&do_full[st], Cfg::kTile);
#pragma unroll
            for (int c = 0; c < Cfg::kChunks; ++c)
              tma_load_3d(sDO + st * Cfg::kTile + c * Cfg::kRegion, &tdo, &do_full[st], c * 64,
                          it.kvh * g, it.b * Lq + qt * P);
            last_t = ig;
            if (i == it.n - 1) next_idx = take_item(ctr);
          }
          tbase += it.n;
          ++ibase;
        }
        if (!ok) {  // drain this CTA's copies still in flight
          if (kv_pending) drain_wait(kv_full, ibase & 1, 100000000ull);
          for (int ii = max(0, last_t - 1); ii <= last_t; ++ii) {
            drain_wait(&q_full[ii & 1], (ii >> 1) & 1, 100000000ull);
            drain_wait(&do_full[ii & 1], (ii >> 1) & 1, 100000000ull);
          }
        }
      }
    } else if (warp == 1 || warp == 2) {
      if (lane == 0) {
        // --------------------------------------- MMA issuers: S^T and dP^T
        // warp 1: S^T(t) = K Q^T into buffer t % 2 once dV(t-2) and dK(t-2),
        // which read P^T and dS^T there, are done.  warp 2: dP^T(t) = V dO^T
        // into the same buffer once the element-wise warps hold S^T(t) in
        // registers.
        const bool is_s = warp == 1;
        constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
        const uint32_t a_addr = smem_u32(is_s ? sK : sV);
        uint8_t* const b_tiles = is_s ? sQ : sDO;
        uint64_t* const b_full = is_s ? q_full : do_full;
        uint64_t* const done_bar = is_s ? s_full : dp_full;
        uint64_t* last_commit = nullptr;
        uint32_t last_parity = 0;
        bool ok = true;
        int tbase = 0, ibase = 0;
        for (int rk = 0; ok; ++rk) {
          int item;
          if (!ring.get(rk, item, ctl)) { ok = false; break; }
          if (item < 0) break;
          const DkdvItem it = dkdv_item(p, item);
          if (it.n == 0) continue;
          if (!mbar_wait(kv_full, ibase & 1, ctl)) { ok = false; break; }
          for (int i = 0; i < it.n; ++i) {
            const int ig = tbase + i, x = ig & 1;
            const uint32_t use = (ig >> 1) & 1;  // parity of this use of buffer x
            if (is_s) {
              if (ig >= 2 && !mbar_wait(&buf_free[x], use ^ 1u, ctl)) { ok = false; break; }
            } else {
              if (!mbar_wait(&s_read[x], use, ctl)) { ok = false; break; }
            }
            if (!mbar_wait(&b_full[x], use, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t b_addr = smem_u32(b_tiles + x * Cfg::kTile);
            const uint32_t d_tmem = tmem + Cfg::kTmemBuf + 128 * x;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * Cfg::kRegion + (kk & 3) * 32;
              mma_bf16_ss(d_tmem, sdesc_sw128(a_addr + off, 16, 1024),
                          sdesc_sw128(b_addr + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
            }
            mma_commit(&done_bar[x]);
            last_commit = &done_bar[x];
            last_parity = use;
          }
          if (!ok) break;
          mma_commit(kv_empty);  // this item's K (V) reads are done once these complete
          tbase += it.n;
          ++ibase;
        }
        if (!ok && last_commit) drain_wait(last_commit, last_parity, 100000000ull);
      }
    } else if (warp == 3) {
      if (lane == 0) {
        // ------------------------------------------- MMA issuer: dV, then dK
        // once P^T is in the tile's buffer: dV += P^T dO; then dK += dS^T Q,
        // each half of dS^T as soon as it is written (A operands from TMEM:
        // warpgroup w's query columns [64w, 64w + 64) sit in 32 columns of the
        // buffer, 8 per 16-deep step).  The commit after dK covers dV too.
        constexpr uint32_t idesc_g = idesc_bf16_f32(128, D, 0, 1);
        uint64_t* last_commit = nullptr;
        uint32_t last_parity = 0;
        bool ok = true;
        int tbase = 0, ibase = 0;
        for (int rk = 0; ok; ++rk) {
          int item;
          if (!ring.get(rk, item, ctl)) { ok = false; break; }
          if (item < 0) break;
          const DkdvItem it = dkdv_item(p, item);
          if (it.n == 0) continue;
          for (int i = 0; i < it.n; ++i) {
            const int ig = tbase + i, x = ig & 1;
            const uint32_t use = (ig >> 1) & 1;
            const uint32_t buf = tmem + Cfg::kTmemBuf + 128 * x;
            // the item's first products overwrite dV, dK: the previous item's
            // must have been read out by the epilogue warps
            if (i == 0 && ibase > 0 && !mbar_wait(acc_free, (ibase - 1) & 1, ctl)) { ok = false; break; }
            if (!mbar_wait(&do_full[x], use, ctl)) { ok = false; break; }
            if (!mbar_wait(&q_full[x], use, ctl)) { ok = false; break; }
            if (!mbar_wait(&p_full[x], use, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t do_addr = smem_u32(sDO + x * Cfg::kTile);
            const uint32_t q_addr = smem_u32(sQ + x * Cfg::kTile);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_f16_ts(tmem + Cfg::kTmemDV, buf + 64 * (kk >> 2) + 8 * (kk & 3),
                         sdesc_sw128(do_addr + kk * 2048, Cfg::kRegion, 1024), idesc_g,
                         (i > 0 || kk > 0) ? 1u : 0u);
            // each half of dS^T as soon as it is written: steps kk = 4w + 2h + {0, 1}
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (!mbar_wait(&ds_full[2 * x + h], use, ctl)) { ok = false; break; }
              tc_fence_after();
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int kk = 4 * (e >> 1) + 2 * h + (e & 1);
                mma_f16_ts(tmem + Cfg::kTmemDK, buf + 32 + 64 * (kk >> 2) + 8 * (kk & 3),
                           sdesc_sw128(q_addr + kk * 2048, Cfg::kRegion, 1024), idesc_g,
                           (i > 0 || kk > 0) ? 1u : 0u);
              }
            }
            if (!ok) break;
            mma_commit(&buf_free[x]);
            // S^T and dP^T of this tile completed before P^T / dS^T existed:
            // its Q and dO are free once dV and dK are
            mma_commit(&do_empty[x]);
            mma_commit(&q_empty[x]);
            last_commit = &buf_free[x];
            last_parity = use;
            if (i == it.n - 1) {
              mma_commit(acc_done);
              last_commit = acc_done;
              last_parity = ibase & 1;
            }
          }
          if (!ok) break;
          tbase += it.n;
          ++ibase;
        }
        if (!ok && last_commit) drain_wait(last_commit, last_parity, 100000000ull);
      }
    }
  } else if (warp < 12) {
    reg_alloc<kDkdvEwRegs>();
    // ----------------------------------------------------------- key rows
    // thread r of warpgroup w owns key r and query columns [64w, 64w + 64)
    // of every query tile
    const int t = threadIdx.x - 128;
    const int r = t & 127, w = t >> 7;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int lg = 31 - __clz(g);
    const float sl2 = p.scale_log2;
    const int C = p.chunk, ca = p.cp_rank, cb = 2 * p.cp_size - 1 - p.cp_rank;
    // statistics of this warpgroup's 64 columns, staged by each warp for
    // itself, so that no warp waits for another: lane l holds -LSE*log2e
    // and Delta of columns 64w + l and 64w + 32 + l
    const int qcol = 64 * w + lane;
    float* col = sCOL + (warp - 4) * 256;  // [2 stages][64 -LSE*log2e, 64 Delta]
    // this warpgroup's 64 columns of TMEM tile buffer 0; buffer 1 is 128 further
    const uint32_t buf_cols = tmem + lane_base + Cfg::kTmemBuf + 64 * w;
    bool ok = true;
    int tbase = 0;
    for (int rk = 0; ok; ++rk) {
      int item;
      if (!ring.get_warp(rk, item, ctl)) { ok = false; break; }
      if (item < 0) break;
      const DkdvItem it = dkdv_item(p, item);
      if (it.n == 0) continue;
      const int key = it.kt * kTileN + r;  // position within the sample
      // queries that may attend this key: positions [key, doc_end)
      const int doc_end = p.doc_hi[static_cast<long long>(it.b) * p.seq_len + key];
      // (B Hq Lq < 2^31: the plan rejects larger shapes)
      const int stat_base = (it.b * p.n_heads + it.kvh * g + (qcol & (g - 1))) * Lq + (qcol >> lg);
      const int s32 = 32 >> lg;  // column + 32: 32 / g positions further
      // list entries of this tile (e) and the next two (e1, e2): they run two
      // tiles ahead and the statistics one tile ahead, so that no load waits
      // on the one before it
      uint32_t e = static_cast<uint32_t>(it.list[0]);
      uint32_t e1 = it.n > 1 ? static_cast<uint32_t>(it.list[1]) : 0u;
      uint32_t e2 = it.n > 2 ? static_cast<uint32_t>(it.list[2]) : 0u;
      int so = stat_base + static_cast<int>(e & kIndexMask) * P;
      float nl0 = lse[so], nl1 = lse[so + s32], nd0 = p.delta[so], nd1 = p.delta[so + s32];
      for (int i = 0; i < it.n; ++i) {
        const int ig = tbase + i;
        if (i > 0) {
          e = e1;
          e1 = e2;
          if (i + 2 < it.n) e2 = static_cast<uint32_t>(it.list[i + 2]);
        }
        {
          // stage this tile's statistics, fetch the next tile's
          float* cs = col + (ig & 1) * 128;
          cs[lane] = nl0 * -kLog2e;
          cs[lane + 32] = nl1 * -kLog2e;
          cs[lane + 64] = nd0;
          cs[lane + 96] = nd1;
          if (i + 1 < it.n) {
            so = stat_base + static_cast<int>(e1 & kIndexMask) * P;
            nl0 = lse[so];
            nl1 = lse[so + s32];
            nd0 = p.delta[so];
            nd1 = p.delta[so + s32];
          }
          __syncwarp();
        }
        // allowed query positions of this key in the tile: [key, doc_end);
        // in tile columns: [lo_c, hi_c)
        int lo_c = 0, hi_c = 128;
        if (e & kPartialBit) {
          const int l0 = static_cast<int>(e & kIndexMask) * P;
          const int q0 = (l0 < C) ? (ca * C + l0) : (cb * C + (l0 - C));
          lo_c = max(0, key - q0) << lg;
          hi_c = min(P, max(0, doc_end - q0)) << lg;
        }
        const bool masked = (e & kPartialBit) != 0;
        const float4* nlse_c = reinterpret_cast<const float4*>(col + (ig & 1) * 128);
        const float4* del_c = reinterpret_cast<const float4*>(col + (ig & 1) * 128 + 64);
        const int x = ig & 1;
        const uint32_t use = (ig >> 1) & 1;
        const uint32_t cols = buf_cols + 128 * x;
        // phase 1: P^T from S^T.  All 64 columns come in with one wait (a
        // TMEM load takes hundreds of cycles while the tensor pipe is busy);
        // once they are in registers dP^T can be computed over them.
        if (!warp_wait(&s_full[x], use, ctl)) { ok = false; break; }
        tc_fence_after();
        uint32_t pb[32];  // P of the 64 columns as bf16 pairs
        {
          uint32_t su[64];
          tmem_ld32_nowait(cols, su);
          tmem_ld32_nowait(cols + 32, su + 32);
          tmem_wait_ld();
          reg_fence32(su);
          reg_fence32(su + 32);
          warp_arrive(&s_read[x]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (masked)
              p_chunk32<true>(su + 32 * h, nlse_c + 8 * h,
                              range_bits(lo_c - 64 * w - 32 * h, hi_c - 64 * w - 32 * h), sl2,
                              pb + 16 * h);
            else
              p_chunk32<false>(su + 32 * h, nlse_c + 8 * h, 0u, sl2, pb + 16 * h);
          }
        }
        // phase 2: load dP^T, write P^T over its first 32 columns (dV starts),
        // then dS^T over the other 32, in two halves (dK starts on each)
        if (!warp_wait(&dp_full[x], use, ctl)) { ok = false; break; }
        tc_fence_after();
        {
          uint32_t du[64];
          tmem_ld32_nowait(cols, du);
          tmem_ld32_nowait(cols + 32, du + 32);
          tmem_wait_ld();
          reg_fence32(du);
          reg_fence32(du + 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) tmem_st8_nowait(cols + 8 * q4, pb + 8 * q4);
          tmem_wait_st();
          warp_arrive(&p_full[x]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pd[16];
            ds_chunk32(du + 32 * h, pb + 16 * h, del_c + 8 * h, pd);
            tmem_st8_nowait(cols + 32 + 16 * h, pd);
            tmem_st8_nowait(cols + 32 + 16 * h + 8, pd + 8);
            tmem_wait_st();
            warp_arrive(&ds_full[2 * x + h]);
          }
        }
      }
      tbase += it.n;
    }
    // ----------------------------------------------- sums of split lists
    // Once every item is taken, the element-wise warps of each CTA take the
    // (split unit, row chunk) sums one at a time and, when the epilogue warps
    // of all the unit's segments have counted them done, add the partials
    // into dK, dV.  Every segment waited for is held by a running CTA, so the
    // waits end.  The last chunk of a unit puts its two counters back to
    // zero for the next launch.
    const int n_split = p.sched[kSchedSplits];
    if (n_split > 0) {
      const int n_sum = n_split * kSumChunks;
      int32_t* const chunks_done = p.kv_done + p.batch * p.n_ktiles;
      volatile int* s_unit = reinterpret_cast<volatile int*>(smem + Cfg::kMisc + Cfg::kUnit);
#pragma unroll 1
      for (int round = 0;; ++round) {
        if (t == 0) {
          int x = n_sum;
          if (!*abort_flag && *reinterpret_cast<volatile uint32_t*>(p.status) == 0u) {
            x = atomicAdd(tail, 1);
            if (x < n_sum) {
              const int u = x / kSumChunks;
              const int segs = p.kv_split[4 * u + 2];
              if (!wait_count(p.kv_done + u, 4 * p.n_kv_heads * segs, ctl)) x = n_sum;
            }
          }
          s_unit[round & 1] = x;
        }
        named_bar_sync(1, 256);
        const int x = s_unit[round & 1];
        if (x >= n_sum) break;
        const int u = x / kSumChunks;
        kv_sum_chunk<D>(p, u, x - u * kSumChunks, dk, dv, t, 256);
        named_bar_sync(1, 256);  // every thread's stores issued before the count
        if (t == 0) {
          __threadfence();
          if (atomicAdd(chunks_done + u, 1) == kSumChunks - 1) {
            p.kv_done[u] = 0;  // every chunk has waited on it: nothing reads it now
            chunks_done[u] = 0;
          }
        }
      }
    }
  } else {
    reg_dealloc<kDkdvEpiRegs>();
    // --------------------------------------------------------------- epilogue
    // warp w - 12 owns key rows 32 (w - 12) .. + 31 of each item: once its dV
    // and dK are complete it reads them out of TMEM 32 columns at a time,
    // stages each block (scaled, fp32, 128-byte swizzled rows) and writes it
    // with its own TMA store; the accumulators are handed back after the
    // last read.  Items without queries get zero rows the same way.
    const int wq = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t stg = smem_u32(smem + Cfg::kStage) + wq * 4096;
    bool ok = true;
    int ibase = 0;
    for (int rk = 0; ok; ++rk) {
      int item;
      if (!ring.get_warp(rk, item, ctl)) { ok = false; break; }
      if (item < 0) break;
      const DkdvItem it = dkdv_item(p, item);
      // segments 1.. of a split list go to their pool slot, the rest to dK, dV
      const bool to_pool = it.slot >= 0;
      const int row0 = to_pool ? it.slot * kTileN + 32 * wq
                               : it.b * p.seq_len + it.kt * kTileN + 32 * wq;
      const CUtensorMap* map_k = to_pool ? &tpk : &tdk;
      const CUtensorMap* map_v = to_pool ? &tpv : &tdv;
      const bool empty = it.n == 0;
      if (!empty) {
        if (!warp_wait(acc_done, ibase & 1, ctl)) { ok = false; break; }
        tc_fence_after();
      }
#pragma unroll 1
      for (int blk = 0; blk < 2 * (D / 32); ++blk) {
        const bool is_dk = blk >= D / 32;
        const int c0 = (blk % (D / 32)) * 32;
        uint32_t u[32];
        if (!empty) {
          tmem_ld32_nowait(tmem + lane_base + (is_dk ? Cfg::kTmemDK : Cfg::kTmemDV) + c0, u);
          tmem_wait_ld();
          reg_fence32(u);
          if (blk == 2 * (D / 32) - 1) warp_arrive(acc_free);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) u[c] = 0u;
        }
        const float sc = is_dk ? p.scale : 1.f;
        // the previous block's store must have read the staging buffer
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          st_shared_v4(stg + lane * 128 + ((ch ^ (lane & 7)) << 4),
                       __float_as_uint(__uint_as_float(u[4 * ch]) * sc),
                       __float_as_uint(__uint_as_float(u[4 * ch + 1]) * sc),
                       __float_as_uint(__uint_as_float(u[4 * ch + 2]) * sc),
                       __float_as_uint(__uint_as_float(u[4 * ch + 3]) * sc));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          asm volatile(
              "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                  reinterpret_cast<uint64_t>(is_dk ? map_k : map_v)),
              "r"(stg), "r"(it.kvh * D + c0), "r"(row0)
              : "memory");
          bulk_commit();
        }
      }
      if (!empty) ++ibase;
      if (it.split >= 0) {
        // this warp's rows of the segment count once its stores are complete
        // (4 warps x Hkv heads x segments complete a split unit)
        if (lane == 0) {
          bulk_wait_all();
          fence_proxy_async_global();
          __threadfence();
          atomicAdd(p.kv_done + it.split, 1);
        }
        __syncwarp();
      }
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) items_exit(ctr, tail);
}

// ------------------------------------------------------------------- dQ

template <int D>
struct DqCfg {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kRegion = 16384;
  static constexpr int kChunks = D / 64;
  // one ring of tile-sized slots carries every load in stream order: per
  // work item Q, dO, (when the kernel also computes Delta) O in two slots,
  // then K_j, V_j for each key tile j of its row list
  static constexpr int kSlots = (D == 128) ? 6 : 8;
  static constexpr int kDS = kSlots * kTile;     // dS (128 x 128 bf16)
  // item descriptors published by the producer, two entries of 8 ints
  static constexpr int kDesc = kDS + 128 * 128 * 2;
  static constexpr int kBar = kDesc + 2 * 8 * 4;
  static constexpr int kNumBars = 2 * kSlots + 16;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kNeed = kMisc + 16;
  static constexpr int kAlloc = (kNeed + 1024 <= kMaxSmem) ? kNeed + 1024 : kMaxSmem;
  // S, dP, dQ accumulators (fp32), then Q and dO as bf16 pairs (A operands)
  static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemDQ = 256;
  static constexpr uint32_t kTmemQ = 384, kTmemDO = 384 + D / 2;
  static_assert(kTmemDO + D / 2 <= 512, "dQ TMEM layout exceeds 512 columns");
  static_assert(kNeed + 1024 <= kMaxSmem, "dQ shared-memory layout exceeds 227 KB");
};

// Work item `item` of the dQ pass: (sample, query tile) in longest-list-first
// order times K/V head.
struct DqItem {
  int b, kvh, l0, n;
  const int32_t* list;
};
__device__ __forceinline__ DqItem dq_item(const PlanDev& p, int item) {
  DqItem it;
  const int ord = item / p.n_kv_heads;
  it.kvh = item % p.n_kv_heads;
  const int bq = p.fwd_order[ord];
  it.b = bq / p.n_qtiles;
  it.l0 = (bq % p.n_qtiles) * p.tile_pos;
  const int rp0 = p.row_ptr[bq];
  it.n = p.row_ptr[bq + 1] - rp0;
  it.list = p.row_idx + rp0;
  return it;
}

// Persistent: CTA c takes work items in snake order.  Counters that
// every role keeps identically across items: the stream index of the next
// slot load (sidx), the number of key tiles processed so far (tbase, which
// fixes the parity of every per-tile barrier) and the number of non-empty
// items so far (ibase, the parity of epi_full and epi_free).
//
// kDelta: the kernel also computes Delta = rowsum(dO * O) of each query row
// (the backward preprocess) from the item's dO (already in TMEM) and O
// (loaded through the ring), uses it, and stores it for the dK/dV pass: the
// rows' O is read while the tensor cores work, instead of in a pass of its
// own.  Otherwise Delta is read from the plan's workspace.
template <int D, bool kDelta>
__global__ void __launch_bounds__(640, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
              const __grid_constant__ CUtensorMap tdq, const __grid_constant__ CUtensorMap to,
              const PlanDev p, const float* __restrict__ lse, const float* __restrict__ o,
              const __nv_bfloat16* __restrict__ dout, __nv_bfloat16* __restrict__ dq,
              int n_items) {
  using Cfg = DqCfg<D>;
  constexpr int NS = Cfg::kSlots;
  constexpr int NO = kDelta ? 2 : 0;  // ring slots of an item's O (fp32, D / 64 boxes each)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (__syncthreads_or(threadIdx.x == 0 &&
                       *reinterpret_cast<volatile uint32_t*>(p.status) != 0u))
    return;
  if (pad + Cfg::kNeed > static_cast<uint32_t>(Cfg::kAlloc)) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, static_cast<uint32_t>(DMA_ERR_UNSUPPORTED));
    return;
  }
  uint8_t* smem = smem_raw + pad;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.group, Lq = p.local_len;

  uint8_t* sDS = smem + Cfg::kDS;
  int* sDesc = reinterpret_cast<int*>(smem + Cfg::kDesc);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBar);
  uint64_t* slot_full = bars;           // [NS]
  uint64_t* slot_empty = bars + NS;     // [NS]
  uint64_t* s_full = bars + 2 * NS;     // S of a key tile computed
  uint64_t* s_free = s_full + 1;        // the row warps have read S
  uint64_t* dp_full = s_full + 2;       // dP computed
  uint64_t* dp_free = s_full + 3;       // the row warps have read dP (and, first tile of
                                        // an item, its dO columns from TMEM)
  uint64_t* ds_full = s_full + 4;       // dS written to shared memory
  uint64_t* ds_done = s_full + 5;       // dQ += dS K done reading dS
  uint64_t* epi_full = s_full + 6;      // an item's dQ tile staged in the dS buffer
  uint64_t* epi_free = s_full + 7;      // its store has read the dS buffer
  uint64_t* desc_full = s_full + 8;     // [2] an item descriptor published
  uint64_t* desc_empty = s_full + 10;   // [2] ... and read by every row warp
  uint64_t* xch_full = s_full + 12;     // every row warp posted its Delta parts
  uint64_t* xch_free = s_full + 13;     // ... and read the sums (the dS buffer is free)
  uint64_t* do_ready = s_full + 14;     // an item's dO copied into TMEM
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + Cfg::kMisc + 4);
  auto slot_ptr = [&](int idx) { return smem + (idx % NS) * Cfg::kTile; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&slot_full[i], 1);
      mbar_init(&slot_empty[i], 1);
    }
    // the row warps arrive once per warp
    mbar_init(s_full, 1);
    mbar_init(s_free, 16);
    mbar_init(dp_full, 1);
    mbar_init(dp_free, 16);
    mbar_init(ds_full, 16);
    mbar_init(ds_done, 1);
    mbar_init(epi_full, 16);
    mbar_init(epi_free, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&desc_full[i], 1);
      mbar_init(&desc_empty[i], 16);
    }
    mbar_init(xch_full, 16);
    mbar_init(xch_free, 16);
    mbar_init(do_ready, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ producer: the stream
      // It publishes the descriptors of the CTA's items for the row warps, one
      // item ahead (all items, empty ones too, then an end marker), and per
      // non-empty item loads Q, dO, (O), and K_j, V_j for every key tile of
      // the item's list.
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tdo);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      if (kDelta) tma_prefetch_desc(&to);
      int sidx = 0, nd = 0;
      bool ok = true;
      auto acquire = [&](int idx) -> bool {
        if (!mbar_wait(&slot_empty[idx % NS], ((idx / NS) & 1) ^ 1u, ctl)) return false;
        mbar_arrive_expect_tx(&slot_full[idx % NS], Cfg::kTile);
        return true;
      };
      // descriptor entry nd % 2: b, kvh, l0, n (-1: no more items), list offset,
      // first list entry
      auto publish = [&](const DqItem* it) -> bool {
        const int e = nd & 1;
        if (nd >= 2 && !mbar_wait(&desc_empty[e], ((nd >> 1) - 1) & 1, ctl)) return false;
        int* d = sDesc + 8 * e;
        if (it) {
          d[0] = it->b;
          d[1] = it->kvh;
          d[2] = it->l0;
          d[3] = it->n;
          d[4] = static_cast<int>(it->list - p.row_idx);
          d[5] = it->n > 0 ? it->list[0] : 0;
        } else {
          d[3] = -1;
        }
        mbar_arrive(&desc_full[e]);
        ++nd;
        return true;
      };
      // the CTA's items in order; each item's successor is published as the
      // item's loads begin, so that the row warps find it well before they
      // finish the item
      int kn = -1;
      auto next_item = [&](DqItem& out) -> bool {
        for (++kn; kn * static_cast<int>(gridDim.x) < n_items; ++kn) {
          const int cand = snake_item(kn);
          if (cand >= n_items) continue;
          out = dq_item(p, cand);
          return true;
        }
        return false;
      };
      DqItem nx{};
      bool have_nx = next_item(nx);
      if (!publish(have_nx ? &nx : nullptr)) ok = false;
      while (ok && have_nx) {
        const DqItem it = nx;
        have_nx = next_item(nx);
        if (!publish(have_nx ? &nx : nullptr)) { ok = false; break; }
        if (it.n == 0) continue;
        const int qrow = it.b * Lq + it.l0;
        if (!acquire(sidx)) { ok = false; break; }
#pragma unroll
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_3d(slot_ptr(sidx) + c * Cfg::kRegion, &tq, &slot_full[sidx % NS], c * 64,
                      it.kvh * g, qrow);
        ++sidx;
        if (!acquire(sidx)) { ok = false; break; }
#pragma unroll
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_3d(slot_ptr(sidx) + c * Cfg::kRegion, &tdo, &slot_full[sidx % NS], c * 64,
                      it.kvh * g, qrow);
        ++sidx;
        if (kDelta) {
          // O (fp32): boxes of 32 columns x 128 rows (16 KB), D / 64 per slot
#pragma unroll
          for (int s2 = 0; s2 < NO; ++s2) {
            if (!acquire(sidx)) { ok = false; break; }
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(slot_ptr(sidx) + c * 16384, &to, &slot_full[sidx % NS],
                          32 * (s2 * (D / 64) + c), it.kvh * g, qrow);
            ++sidx;
          }
          if (!ok) break;
        }
        for (int j = 0; j < it.n; ++j) {
          const int kt = static_cast<int>(static_cast<uint32_t>(it.list[j]) & kIndexMask);
          const int krow = it.b * p.seq_len + kt * kTileN;
          if (!acquire(sidx)) { ok = false; break; }
#pragma unroll
          for (int c = 0; c < Cfg::kChunks; ++c)
            tma_load_2d(slot_ptr(sidx) + c * Cfg::kRegion, &tk, &slot_full[sidx % NS],
                        it.kvh * D + c * 64, krow);
          ++sidx;
          if (!acquire(sidx)) { ok = false; break; }
#pragma unroll
          for (int c = 0; c < Cfg::kChunks; ++c)
            tma_load_2d(slot_ptr(sidx) + c * Cfg::kRegion, &tv, &slot_full[sidx % NS],
                        it.kvh * D + c * 64, krow);
          ++sidx;
        }
      }
      if (!ok) {  // drain this CTA's copies still in flight
        for (int idx = max(0, sidx - NS); idx < sidx; ++idx)
          drain_wait(&slot_full[idx % NS], (idx / NS) & 1, 100000000ull);
      }
    }
  } else if (warp <= 3) {
    if (lane == 0) {
      // ------------------------------------------------------ MMA issuers
      // per key tile: S = Q K_j^T (warp 1) and dP = dO V_j^T (warp 2) into
      // TMEM with Q and dO as TMEM A operands; once the row warps have
      // written dS: dQ += dS K_j (warp 3).  S and dP have separate buffers,
      // each reissued as soon as the row warps have read it.  One issuing
      // thread per product on its own warp scheduler keeps the tensor pipe
      // fed while the row warps keep the schedulers busy.
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t idesc_g = idesc_bf16_f32(128, D, 0, 1);
      uint64_t* last_commit = nullptr;
      uint32_t last_parity = 0;
      bool ok = true;
      int sidx = 0, tbase = 0, ibase = 0;
      for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_items; ++k) {
      const int item = snake_item(k);
      if (item >= n_items) continue;
        const DqItem it = dq_item(p, item);
        if (it.n == 0) continue;
        if (warp == 1 || warp == 2) {
          // the item's Q (warp 1) or dO (warp 2) into TMEM by tcgen05.cp,
          // once the previous item is done with the old one (its last S has
          // completed; the row warps have read its last dP, and with it the
          // dO columns they read for Delta); the copy is ordered before this
          // thread's next MMAs, and the slot goes back to the producer when
          // it completes
          const int cidx = sidx + (warp == 1 ? 0 : 1);
          if (tbase > 0 && !mbar_wait(warp == 1 ? s_full : (kDelta ? dp_free : dp_full),
                                      (tbase - 1) & 1, ctl)) {
            ok = false;
            break;
          }
          if (!mbar_wait(&slot_full[cidx % NS], (cidx / NS) & 1, ctl)) { ok = false; break; }
          tc_fence_after();
          const uint32_t src = smem_u32(slot_ptr(cidx));
          const uint32_t dst_t = tmem + (warp == 1 ? Cfg::kTmemQ : Cfg::kTmemDO);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tmem_cp_128x256b(dst_t + 8 * kk,
                             sdesc_sw128(src + (kk >> 2) * Cfg::kRegion + (kk & 3) * 32, 16, 1024));
          mma_commit(&slot_empty[cidx % NS]);
          if (kDelta && warp == 2) mma_commit(do_ready);  // the row warps read it for Delta
        }
        for (int j = 0; j < it.n; ++j) {
          const int t = tbase + j;
          const int kidx = sidx + 2 + NO + 2 * j, vidx = kidx + 1;
          if (warp == 1) {
            if (!mbar_wait(&slot_full[kidx % NS], (kidx / NS) & 1, ctl)) { ok = false; break; }
            if (t > 0 && !mbar_wait(s_free, (t - 1) & 1, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t k_addr = smem_u32(slot_ptr(kidx));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {  // S = Q K^T
              const uint32_t off = (kk >> 2) * Cfg::kRegion + (kk & 3) * 32;
              mma_f16_ts(tmem + Cfg::kTmemS, tmem + Cfg::kTmemQ + 8 * kk,
                         sdesc_sw128(k_addr + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
            }
            mma_commit(s_full);
            last_commit = s_full;
            last_parity = t & 1;
          } else if (warp == 2) {
            if (!mbar_wait(&slot_full[vidx % NS], (vidx / NS) & 1, ctl)) { ok = false; break; }
            if (t > 0 && !mbar_wait(dp_free, (t - 1) & 1, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t v_addr = smem_u32(slot_ptr(vidx));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {  // dP = dO V^T
              const uint32_t off = (kk >> 2) * Cfg::kRegion + (kk & 3) * 32;
              mma_f16_ts(tmem + Cfg::kTmemDP, tmem + Cfg::kTmemDO + 8 * kk,
                         sdesc_sw128(v_addr + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
            }
            mma_commit(dp_full);
            mma_commit(&slot_empty[vidx % NS]);
            last_commit = dp_full;
            last_parity = t & 1;
          } else {
            // S_j has completed before dS_j exists, so K_j's slot is free
            // once this product is done
            if (!mbar_wait(ds_full, t & 1, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t ds_addr = smem_u32(sDS);
            const uint32_t k_addr = smem_u32(slot_ptr(kidx));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // dQ += dS K
              const uint64_t a =
                  sdesc_sw128(ds_addr + (kk >> 2) * Cfg::kRegion + (kk & 3) * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(k_addr + kk * 2048, Cfg::kRegion, 1024);
              mma_bf16_ss(tmem + Cfg::kTmemDQ, a, bd, idesc_g, (j > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(ds_done);
            mma_commit(&slot_empty[kidx % NS]);
            last_commit = ds_done;
            last_parity = t & 1;
          }
        }
        if (ok && warp == 3) {
          // the row warps staged this item's dQ tile (bf16, the layout a
          // Q tile load produces) in the dS buffer: store it, and hand the
          // buffer back once the store has read it
          if (!mbar_wait(epi_full, ibase & 1, ctl)) { ok = false; break; }
#pragma unroll
          for (int c = 0; c < Cfg::kChunks; ++c)
            tma_store_3d(&tdq, sDS + c * Cfg::kRegion, c * 64, it.kvh * g, it.b * Lq + it.l0);
          bulk_commit();
          bulk_wait_read_all();
          mbar_arrive(epi_free);
        }
        sidx += 2 + NO + 2 * it.n;
        tbase += it.n;
        ++ibase;
      }
      if (warp == 3) bulk_wait_all();
      if (!ok && last_commit) drain_wait(last_commit, last_parity, 100000000ull);
    }
  } else {
    // ----------------------------------------------------------- query rows
    // four warpgroups: thread (r, q) owns query row r and key columns
    // [32q, 32q + 32) of each key tile, and head_dim columns
    // [q D/4, (q + 1) D/4) of the row for Delta and the dQ epilogue
    const int r = (threadIdx.x - 128) & 127;
    const int q = (threadIdx.x - 128) >> 7;
    const int cbase = 32 * q;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int lg = 31 - __clz(g);
    const int pos = r >> lg, h = r & (g - 1);
    const int C = p.chunk;
    const float sl2 = p.scale_log2;
    // this thread's 64 bytes of dS row r: one half of a 64-column region
    const uint32_t ds_row = smem_u32(sDS) + (q >> 1) * Cfg::kRegion + r * 128;
    const int ch0 = (q & 1) * 4;
    constexpr int DQ = D / 4;  // head_dim columns of dQ this warpgroup writes
    float* xch = reinterpret_cast<float*>(sDS);  // [4][128] Delta partials, at item start
    bool ok = true;
    int tbase = 0, ibase = 0, nd = 0, sidx = 0;
    // this row's data of the next item, loaded during the current one
    int pf_lo = 0;
    float pf_lse = 0.f, pf_del = 0.f;
    bool pf = false;
    for (;;) {
      // the next item's descriptor, published by the producer
      const int de = nd & 1;
      if (!warp_wait(&desc_full[de], (nd >> 1) & 1, ctl)) { ok = false; break; }
      DqItem it;
      const int* dsc = sDesc + 8 * de;
      it.b = dsc[0];
      it.kvh = dsc[1];
      it.l0 = dsc[2];
      it.n = dsc[3];
      it.list = p.row_idx + dsc[4];
      uint32_t e_next = static_cast<uint32_t>(dsc[5]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&desc_empty[de]);
      ++nd;
      if (it.n < 0) break;
      const int l = it.l0 + pos;
      const int hq = it.kvh * g + h;
      const long long stat =
          (static_cast<long long>(it.b) * p.n_heads + it.kvh * g + h) * Lq + it.l0 + pos;
      const long long orow = (static_cast<long long>(it.b) * Lq + l) * p.n_heads + hq;
      if (it.n == 0) {
        // (every row attends at least its own key, so an item has at least
        // one key tile; kept for completeness) dQ = 0, Delta from memory
        uint4* dst = reinterpret_cast<uint4*>(dq + orow * D + q * DQ);
#pragma unroll
        for (int c = 0; c < DQ / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
        if (kDelta && q == 0) {
          float acc = 0.f;
          for (int d = 0; d < D; ++d)
            acc = fmaf(o[orow * D + d], __bfloat162float(dout[orow * D + d]), acc);
          p.delta[stat] = acc;
        }
        pf = false;
        continue;
      }
      const int qabs =
          (l < C) ? (p.cp_rank * C + l) : ((2 * p.cp_size - 1 - p.cp_rank) * C + l - C);
      const int lo_r = pf ? pf_lo : p.doc_lo[static_cast<long long>(it.b) * Lq + l];
      const float lse2 = (pf ? pf_lse : lse[stat]) * kLog2e;
      float del = (!kDelta && pf) ? pf_del : (kDelta ? 0.f : p.delta[stat]);
      if (kDelta) {
        // once the item's dO is in TMEM (copied there for dP)
        if (!warp_wait(do_ready, ibase & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        // Delta of this row: its dO (bf16 pairs in TMEM, copied there for
        // dP) times its O (fp32, from the ring), this warpgroup's D/4
        // columns, then the four warpgroups' parts added in order
        uint32_t od[DQ / 2];
        if constexpr (DQ == 32) {
          tmem_ld16_nowait(tmem + lane_base + Cfg::kTmemDO + q * (DQ / 2), od);
          tmem_wait_ld();
          reg_fence16(od);
        } else {
          tmem_ld8_nowait(tmem + lane_base + Cfg::kTmemDO + q * (DQ / 2), od);
          tmem_wait_ld();
          reg_fence8(od);
        }
        // the O box holding these columns: box (q D/4) / 32, D / 64 boxes a slot
        const int box = (q * DQ) / 32;
        const int oidx = sidx + 2 + box / (D / 64);
        if (!warp_wait(&slot_full[oidx % NS], (oidx / NS) & 1, ctl)) { ok = false; break; }
        // row r of the box: 128 bytes, 16-byte chunks swizzled by r & 7
        const uint32_t orow_s =
            smem_u32(slot_ptr(oidx)) + (box % (D / 64)) * 16384 + r * 128;
        const int cb0 = ((q * DQ) % 32) / 4;
        float part = 0.f;
#pragma unroll
        for (int c = 0; c < DQ / 4; ++c) {
          float4 ov;
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(ov.x), "=f"(ov.y), "=f"(ov.z), "=f"(ov.w)
                       : "r"(orow_s + (((cb0 + c) ^ (r & 7)) << 4)));
          const uint32_t w0 = od[2 * c], w1 = od[2 * c + 1];
          part = fmaf(ov.x, __uint_as_float(w0 << 16), part);
          part = fmaf(ov.y, __uint_as_float(w0 & 0xFFFF0000u), part);
          part = fmaf(ov.z, __uint_as_float(w1 << 16), part);
          part = fmaf(ov.w, __uint_as_float(w1 & 0xFFFF0000u), part);
        }
        // the parts go through the dS buffer: the previous item's dQ
        // store must have read it
        if (ibase > 0 && !warp_wait(epi_free, (ibase - 1) & 1, ctl)) { ok = false; break; }
        xch[q * 128 + r] = part;
        __syncwarp();
        if (lane == 0) mbar_arrive(xch_full);
        if (!warp_wait(xch_full, ibase & 1, ctl)) { ok = false; break; }
        del = (xch[r] + xch[128 + r]) + (xch[256 + r] + xch[384 + r]);
        if (threadIdx.x == 128) {
          // every row warp has read O: its slots go back to the producer
#pragma unroll
          for (int s2 = 0; s2 < NO; ++s2) mbar_arrive(&slot_empty[(sidx + 2 + s2) % NS]);
        }
        if (q == 0) p.delta[stat] = del;
        // dS overwrites the parts only once every warp has read them
        __syncwarp();
        if (lane == 0) mbar_arrive(xch_free);
        if (!warp_wait(xch_free, ibase & 1, ctl)) { ok = false; break; }
      }
      for (int j = 0; j < it.n; ++j) {
        const int t = tbase + j;
        const uint32_t e = e_next;  // list entries run one tile ahead
        if (j + 1 < it.n) e_next = static_cast<uint32_t>(it.list[j + 1]);
        uint32_t allow = 0xFFFFFFFFu;
        if (e & kPartialBit) {
          const int k0 = static_cast<int>(e & kIndexMask) * kTileN + cbase;
          allow = range_bits(lo_r - k0, qabs - k0 + 1);
        }
        // P = exp2(S * scale*log2e - LSE*log2e) for this thread's 32 columns
        if (!warp_wait(s_full, t & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        float pv[32];
        {
          uint32_t su[32];
          tmem_ld32_nowait(tmem + lane_base + Cfg::kTmemS + cbase, su);
          tmem_wait_ld();
          reg_fence32(su);
          warp_arrive(s_free);  // S is in registers: the buffer can take the next S
          const uint64_t sl2x2 = f2(sl2, sl2), nlse2x2 = f2(-lse2, -lse2);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const uint64_t x = f2_fma(f2(__uint_as_float(su[c]), __uint_as_float(su[c + 1])),
                                      sl2x2, nlse2x2);
            float x0, x1;
            f2_split(x, x0, x1);
            pv[c] = ex2(x0);
            pv[c + 1] = ex2(x1);
          }
          if (allow != 0xFFFFFFFFu) {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (!((allow >> c) & 1u)) pv[c] = 0.f;
          }
        }
        // dS = P (dP - Delta)
        if (!warp_wait(dp_full, t & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        uint32_t pk[16];
        {
          uint32_t du[32];
          tmem_ld32_nowait(tmem + lane_base + Cfg::kTmemDP + cbase, du);
          tmem_wait_ld();
          reg_fence32(du);
          // dP (and, first tile of an item, the item's dO) read: the buffer
          // can take the next dP
          warp_arrive(dp_free);
          const uint64_t delx2 = f2(del, del);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const uint64_t d = f2_mul(f2(pv[c], pv[c + 1]),
                                      f2_sub(f2(__uint_as_float(du[c]), __uint_as_float(du[c + 1])),
                                             delx2));
            float d0, d1;
            f2_split(d, d0, d1);
            pk[c >> 1] = pack_bf16(d0, d1);
          }
        }
        if (t > 0 && !warp_wait(ds_done, (t - 1) & 1, ctl)) { ok = false; break; }
        // the dS buffer may still be read by the store of the previous dQ tile
        if (!kDelta && j == 0 && ibase > 0 && !warp_wait(epi_free, (ibase - 1) & 1, ctl)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
          st_shared_v4(ds_row + (((ch0 + c) ^ (r & 7)) << 4), pk[4 * c], pk[4 * c + 1],
                       pk[4 * c + 2], pk[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(ds_full);
      }
      if (!ok) break;
      // the next item's row data: its descriptor is published (the producer
      // publishes it before loading that item), so the loads are issued now
      // and land during this item's epilogue
      pf = false;
      {
        const int de2 = nd & 1;
        if (!warp_wait(&desc_full[de2], (nd >> 1) & 1, ctl)) { ok = false; break; }
        const int* d2 = sDesc + 8 * de2;
        const int nb = d2[0], nkvh = d2[1], nl0 = d2[2], nn = d2[3];
        if (nn > 0) {
          const long long nstat =
              (static_cast<long long>(nb) * p.n_heads + nkvh * g + h) * Lq + nl0 + pos;
          pf_lo = p.doc_lo[static_cast<long long>(nb) * Lq + nl0 + pos];
          pf_lse = lse[nstat];
          if (!kDelta) pf_del = p.delta[nstat];
          pf = true;
        }
      }
      // epilogue: dQ (scaled, bf16) staged in the dS buffer in the layout of
      // a Q tile load (64-column regions, row r = 128 bytes, 16-byte chunks
      // swizzled by r & 7); the dQ issuer stores it with one TMA store per
      // region.  Warpgroup q stages head_dim columns [q*D/4, (q+1)*D/4).
      const int t_last = tbase + it.n - 1;
      if (!warp_wait(ds_done, t_last & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      {
        const float sc = p.scale;
        const uint32_t row = smem_u32(sDS) + ((q * DQ) / 64) * Cfg::kRegion + r * 128;
        const int chb = ((q * DQ) % 64) / 8;
#pragma unroll
        for (int c0 = 0; c0 < DQ; c0 += 16) {
          uint32_t u[16];
          tmem_ld16_nowait(tmem + lane_base + Cfg::kTmemDQ + q * DQ + c0, u);
          tmem_wait_ld();
          reg_fence16(u);
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            const int ch = chb + c0 / 8 + q2;
            st_shared_v4(row + ((ch ^ (r & 7)) << 4),
                         pack_bf16(__uint_as_float(u[8 * q2 + 0]) * sc, __uint_as_float(u[8 * q2 + 1]) * sc),
                         pack_bf16(__uint_as_float(u[8 * q2 + 2]) * sc, __uint_as_float(u[8 * q2 + 3]) * sc),
                         pack_bf16(__uint_as_float(u[8 * q2 + 4]) * sc, __uint_as_float(u[8 * q2 + 5]) * sc),
                         pack_bf16(__uint_as_float(u[8 * q2 + 6]) * sc, __uint_as_float(u[8 * q2 + 7]) * sc));
          }
        }
      }
      fence_proxy_async_smem();
      // the next item's first dQ product overwrites the accumulator only
      // after every warp has arrived on ds_full for it, i.e. after this read
      warp_arrive(epi_full);
      sidx += 2 + NO + 2 * it.n;
      tbase += it.n;
      ++ibase;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_delta_d(const dma_plan_s& pl, const float* o, const dma_bf16* dout,
                           cudaStream_t s) {
  const PlanDev& p = pl.d;
  const int rows = p.batch * p.local_len * p.n_heads;
  if (rows == 0) return cudaSuccess;
  constexpr int TPR = D / 8;
  const int blocks = (rows * TPR + 255) / 256;
  delta_kernel<D><<<blocks, 256, 0, s>>>(o, reinterpret_cast<const __nv_bfloat16*>(dout), p.delta,
                                         rows, p.n_heads, p.local_len);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dkdv_d(const dma_plan_s& pl, const float* lse, const CUtensorMap& tq,
                          const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                          const CUtensorMap& tdk, const CUtensorMap& tdv, const CUtensorMap& tpk,
                          const CUtensorMap& tpv, float* dk, float* dv, cudaStream_t s) {
  const PlanDev& p = pl.d;
  // the planner writes the work list on the device; at most one slice per
  // unit plus one per pool slot
  const long long items_max =
      (static_cast<long long>(p.batch) * p.n_ktiles + p.kv_cap) * p.n_kv_heads;
  if (items_max == 0) return cudaSuccess;
  // persistent: one CTA per SM (TMEM and shared memory allow no more)
  const int grid = items_max < pl.num_sms ? static_cast<int>(items_max) : pl.num_sms;
  cudaError_t e = cudaFuncSetAttribute(dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       DkdvCfg<D>::kAlloc);
  if (e != cudaSuccess) return e;
  dkdv_kernel<D><<<grid, 512, DkdvCfg<D>::kAlloc, s>>>(tq, tk, tv, tdo, tdk, tdv, tpk, tpv, p, lse,
                                                       dk, dv);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dq_d(const dma_plan_s& pl, const float* lse, const CUtensorMap& tq,
                        const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                        const CUtensorMap& tdq, const CUtensorMap* to, const float* o,
                        const dma_bf16* dout, dma_bf16* dq, cudaStream_t s) {
  const PlanDev& p = pl.d;
  const int items = p.batch * p.n_qtiles * p.n_kv_heads;
  if (items == 0) return cudaSuccess;
  // persistent: one CTA per SM (TMEM and shared memory allow no more)
  const int grid = items < pl.num_sms ? items : pl.num_sms;
  const auto* pdo = reinterpret_cast<const __nv_bfloat16*>(dout);
  auto* pdq = reinterpret_cast<__nv_bfloat16*>(dq);
  if (to) {  // Delta computed here
    cudaError_t e = cudaFuncSetAttribute(dq_kernel<D, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DqCfg<D>::kAlloc);
    if (e != cudaSuccess) return e;
    dq_kernel<D, true><<<grid, 640, DqCfg<D>::kAlloc, s>>>(tq, tk, tv, tdo, tdq, *to, p, lse, o,
                                                          pdo, pdq, items);
  } else {
    cudaError_t e = cudaFuncSetAttribute(dq_kernel<D, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DqCfg<D>::kAlloc);
    if (e != cudaSuccess) return e;
    dq_kernel<D, false><<<grid, 640, DqCfg<D>::kAlloc, s>>>(tq, tk, tv, tdo, tdq, tq, p, lse, o,
                                                           pdo, pdq, items);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_delta(const dma_plan_s& pl, const float* o, const dma_bf16* dout,
                         cudaStream_t s) {
  return pl.d.head_dim == 128 ? launch_delta_d<128>(pl, o, dout, s)
                              : launch_delta_d<64>(pl, o, dout, s);
}

cudaError_t launch_dkdv(const dma_plan_s& pl, const float* lse, const CUtensorMap& tq,
                        const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                        const CUtensorMap& tdk, const CUtensorMap& tdv, const CUtensorMap& tpk,
                        const CUtensorMap& tpv, float* dk, float* dv, cudaStream_t s) {
  return pl.d.head_dim == 128
             ? launch_dkdv_d<128>(pl, lse, tq, tk, tv, tdo, tdk, tdv, tpk, tpv, dk, dv, s)
             : launch_dkdv_d<64>(pl, lse, tq, tk, tv, tdo, tdk, tdv, tpk, tpv, dk, dv, s);
}

cudaError_t launch_dq(const dma_plan_s& pl, const float* lse, const CUtensorMap& tq,
                      const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                      const CUtensorMap& tdq, const CUtensorMap* to, const float* o,
                      const dma_bf16* dout, dma_bf16* dq, cudaStream_t s) {
  return pl.d.head_dim == 128 ? launch_dq_d<128>(pl, lse, tq, tk, tv, tdo, tdq, to, o, dout, dq, s)
                              : launch_dq_d<64>(pl, lse, tq, tk, tv, tdo, tdq, to, o, dout, dq, s);
}

}  // namespace dma
