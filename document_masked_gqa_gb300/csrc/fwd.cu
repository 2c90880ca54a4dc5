// Forward kernel: causal + document-masked GQA attention for one CP rank.
//
// Work item = (query tile, K/V head).  A query tile is 128 rows: P = 128/g
// consecutive local positions x the g query heads sharing K/V head `kvh`
// (GQA, "The Llama 3 Herd of Models - part 3/16", 3.3.2, and "Paper notes:
// The Llama 3 Herd of Models", 8 key-value heads), so one K/V tile feeds g
// heads at once.  An item walks the tile's list of non-skipped key tiles
// (built by the block-mask builder) and keeps the online-softmax running max
// and sum per row, rescaling the partial output, then divides by the sum
// ("Training Infrastructure and Systems", "FlashAttention: never write the
// score matrix", sections "Online softmax" and "Tiling").
//
// GB300 mapping (sm_103a), one persistent CTA per SM, 16 warps:
//   warp 0      TMA producer: per item Q, then K_j and V_j (fp16 copy) for
//               each key tile, through one ring of tile-sized slots
//   warp 1      tcgen05 issuer for S = Q K^T into one of two TMEM buffers (Q
//               copied once per item into TMEM as the A operand); owns the
//               TMEM allocation
//   warp 3      tcgen05 issuer for O += P V with P taken from TMEM
//   warps 4-11  softmax: two warpgroups split each tile's 128 key columns,
//               thread r of each owns row r (TMEM lane r); they exchange row
//               maxima, exponentiate in base 2, write their half of P (fp16
//               pairs) back over the S columns each has read, and rescale
//               their half of O in TMEM when the reference max moves
//   warps 12-15 epilogue: O (fp32) and LSE of an item while the softmax
//               warps start the next one
// Separate issuing threads keep the tensor pipe fed while the softmax warps
// keep the warp schedulers busy.
// Keeping Q and P in TMEM leaves the tensor core only K and V to read from
// shared memory, which halves the shared-memory traffic per tile.
// P V runs in fp16 against an fp16 copy of V made once per call
// (v_to_f16_kernel): fp16's 11-bit significand keeps the rounding of the
// probabilities 8x below bf16's, so O meets a 1e-2 absolute bound even on
// rows that see only a few keys.
// The reference max only moves when a row's max grows by more than 2^8, so
// most tiles need no rescale of O; the final O / l is exact either way.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dma {
namespace {

template <int D>
struct FwdCfg {
  static constexpr int kRegion = 128 * 128;       // one 64-column SW128 region of a 128-row tile
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = 128 * D * 2;  // Q, K or V tile (16-bit)
  // a ring of tile-sized slots carries K_j, V_j for each key tile j of each
  // work item's row list; Q has a buffer of its own (the next item's Q is
  // loaded as soon as the current one has been copied into TMEM)
  static constexpr int kSlots = (D == 128) ? 5 : 10;
  static constexpr int kQbuf = kSlots * kTileBytes;
  // O epilogue staging: per epilogue warp one 4 KB block of 32 rows x 32
  // fp32 in the 128-byte swizzled layout of a TMA store
  static constexpr int kStage = kQbuf + kTileBytes;
  // row maxima [2 tiles][2 warpgroups][128], then per item parity: row sums
  // [2][2 warpgroups][128] and reference maxima [2][128]
  static constexpr int kXchg = kStage + 4 * 4096;
  // per item parity, staged by the epilogue warps ahead of the item: n, list
  // offset, first list entry, then per row the query position and its
  // document's first position
  static constexpr int kMeta = kXchg + (2 * 2 * 128 + 2 * 2 * 128 + 2 * 128) * 4;
  static constexpr int kMetaInts = 4 + 2 * 128;
  static constexpr int kBar = kMeta + 2 * kMetaInts * 4;
  static constexpr int kNumBars = 2 * kSlots + 2 + 2 + 2 + 2 + 1 + 2 + 1 + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kEnd = kMisc + 16;
  static constexpr int kSmemBytes = kEnd + 1024;
  static constexpr uint32_t kTmemCols = 512;
  // TMEM: S buffers (128 columns each; P overwrites part of them as fp16
  // pairs), the O accumulator, and two Q buffers as bf16 pairs (the A
  // operand of Q K^T; item i uses buffer i % 2)
  static constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemO = 256, kTmemQ = 384;
  static_assert(kTmemQ + D <= 512, "forward TMEM layout exceeds 512 columns");
  static_assert(kSmemBytes <= 232448, "forward shared-memory layout exceeds 227 KB");
};

// Wait for a phase ignoring the abort flag, bounded by limit_ns (used only to
// drain this CTA's own copies before it exits after an abort).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// Work item `item`: (sample, query tile) in longest-list-first order times
// K/V head.
struct FwdItem {
  int b, kvh, l0, n;
  const int32_t* list;
};
__device__ __forceinline__ FwdItem fwd_item(const PlanDev& p, int item) {
  FwdItem it;
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

// Persistent: CTA c takes work items c, c + gridDim.x, ...  Every role keeps
// the same counters across items: the stream index of the next slot load
// (sidx), the key tiles processed so far (tbase: S buffer t & 1 and every
// per-tile barrier parity follow from the global tile index t) and the
// items so far (ibase: parity of q_tmem and l_ready).
template <int D>
__global__ void __launch_bounds__(512, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
               const PlanDev p, float* __restrict__ o, float* __restrict__ lse, int n_items) {
  using Cfg = FwdCfg<D>;
  constexpr int NS = Cfg::kSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  // a failed plan or an earlier expired wait: do nothing (CTA-uniform)
  if (__syncthreads_or(threadIdx.x == 0 &&
                       *reinterpret_cast<volatile uint32_t*>(p.status) != 0u))
    return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.group, Lq = p.local_len;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBar);
  uint64_t* slot_full = bars;          // [NS]
  uint64_t* slot_empty = bars + NS;    // [NS]
  uint64_t* s_full = bars + 2 * NS;    // [2] S computed in buffer t & 1
  // per S buffer (tile parity), so that no waiter can fall two phases behind
  // while the S and P V issuers run independently
  uint64_t* p_full = s_full + 2;       // [2] P written over S
  uint64_t* o_done = p_full + 2;       // [2] P V of a tile done (its S buffer is free)
  uint64_t* mx_ready = o_done + 2;     // [2] both softmax warpgroups posted a tile's row maxima
  uint64_t* l_ready = mx_ready + 2;    // both posted an item's partial row sums
  uint64_t* q_tmem = l_ready + 1;      // [2] an item's Q copied into TMEM Q buffer item % 2
  uint64_t* o_free = q_tmem + 2;       // the epilogue warps have read an item's O
  uint64_t* q_full = o_free + 1;       // an item's Q in the Q buffer
  uint64_t* q_empty = q_full + 1;      // ... copied into TMEM (buffer free)
  uint8_t* sQ = smem + Cfg::kQbuf;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + Cfg::kMisc + 4);
  auto slot_ptr = [&](int idx) { return smem + (idx % NS) * Cfg::kTileBytes; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&slot_full[i], 1);
      mbar_init(&slot_empty[i], 1);
    }
    // the softmax and epilogue warps arrive once per warp
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 8);
      mbar_init(&o_done[i], 1);
      mbar_init(&mx_ready[i], 8);
    }
    mbar_init(l_ready, 8);
    mbar_init(&q_tmem[0], 4);
    mbar_init(&q_tmem[1], 4);
    mbar_init(o_free, 4);
    mbar_init(q_full, 1);
    mbar_init(q_empty, 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, Cfg::kTmemCols);
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
      // K_j, V_j of every item through the slot ring; each item's Q into the
      // Q buffer, the next one as soon as the current one is in TMEM
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      int sidx = 0, qn = 0;  // slot loads issued, Q loads issued
      bool ok = true;
      auto acquire = [&](int idx) -> bool {
        if (!mbar_wait(&slot_empty[idx % NS], ((idx / NS) & 1) ^ 1u, ctl)) return false;
        mbar_arrive_expect_tx(&slot_full[idx % NS], Cfg::kTileBytes);
        return true;
      };
      auto load_q = [&](const FwdItem& qi) -> bool {
        if (qn > 0 && !mbar_wait(q_empty, (qn - 1) & 1, ctl)) return false;
        mbar_arrive_expect_tx(q_full, Cfg::kTileBytes);
#pragma unroll
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_3d(sQ + c * Cfg::kRegion, &tq, q_full, c * 64, qi.kvh * g, qi.b * Lq + qi.l0);
        ++qn;
        return true;
      };
      bool first = true;
      for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_items; ++k) {
        const int item = snake_item(k);
        if (item >= n_items) continue;
        const FwdItem it = fwd_item(p, item);
        if (it.n == 0) continue;
        if (first) {
          if (!load_q(it)) { ok = false; break; }
          first = false;
        }
        // the next item's Q: the buffer frees once this item's Q is in TMEM;
        // issued between K / V loads as soon as that has happened
        FwdItem nx{};
        bool q_next = false;
        for (int kx = k + 1; kx * static_cast<int>(gridDim.x) < n_items; ++kx) {
          const int cand = snake_item(kx);
          if (cand >= n_items) continue;
          nx = fwd_item(p, cand);
          if (nx.n == 0) continue;
          q_next = true;
          break;
        }
        for (int j = 0; j < it.n; ++j) {
          if (q_next && mbar_try_wait(q_empty, (qn - 1) & 1)) {
            if (!load_q(nx)) { ok = false; break; }
            q_next = false;
          }
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
        if (ok && q_next && !load_q(nx)) ok = false;
      }
      if (!ok) {  // drain this CTA's copies still in flight
        for (int idx = max(0, sidx - NS); idx < sidx; ++idx)
          drain_wait(&slot_full[idx % NS], (idx / NS) & 1, 100000000ull);
        if (qn > 0) drain_wait(q_full, (qn - 1) & 1, 100000000ull);
      }
    }
  } else if (warp == 1 || warp == 3) {
    if (lane == 0) {
      // ------------------------------------------------------ MMA issuers
      // warp 1: S_t = Q K_t^T into TMEM buffer t & 1 (A = Q from TMEM); the
      // buffer is reused for S_{t+2} once P_t V_t (which reads P_t from it)
      // has completed.  warp 3: once the softmax has written P_t over S_t:
      // O += P_t V_t with A = P_t from TMEM.  Two issuing threads keep the
      // tensor pipe fed while the softmax warps keep the schedulers busy.
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t idesc_o = idesc_f16_f32(128, D, 0, 1);
      uint64_t* last_commit = nullptr;
      uint32_t last_parity = 0;
      bool ok = true;
      int sidx = 0, tbase = 0, ibase = 0;
      for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_items; ++k) {
      const int item = snake_item(k);
      if (item >= n_items) continue;
        const FwdItem it = fwd_item(p, item);
        if (it.n == 0) continue;
        if (warp == 1 && !mbar_wait(&q_tmem[ibase & 1], (ibase >> 1) & 1, ctl)) { ok = false; break; }
        for (int j = 0; j < it.n; ++j) {
          const int t = tbase + j, sb = t & 1;
          const int kidx = sidx + 2 * j, vidx = kidx + 1;
          if (warp == 1) {
            if (!mbar_wait(&slot_full[kidx % NS], (kidx / NS) & 1, ctl)) { ok = false; break; }
            if (t >= 2 && !mbar_wait(&o_done[sb], ((t - 2) >> 1) & 1, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t k_addr = smem_u32(slot_ptr(kidx));
            const uint32_t d_s = tmem + (sb ? Cfg::kTmemS1 : Cfg::kTmemS0);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_f16_ts(d_s, tmem + Cfg::kTmemQ + (ibase & 1) * (D / 2) + 8 * kk,
                         sdesc_sw128(k_addr + (kk >> 2) * Cfg::kRegion + (kk & 3) * 32, 16, 1024),
                         idesc_s, kk > 0 ? 1u : 0u);
            mma_commit(&s_full[sb]);
            mma_commit(&slot_empty[kidx % NS]);
            last_commit = &s_full[sb];
            last_parity = (t >> 1) & 1;
          } else {
            // the item's first P V overwrites O: the previous item's O must
            // have been read out by the epilogue warps
            if (j == 0 && ibase > 0 && !mbar_wait(o_free, (ibase - 1) & 1, ctl)) { ok = false; break; }
            if (!mbar_wait(&p_full[sb], (t >> 1) & 1, ctl)) { ok = false; break; }
            if (!mbar_wait(&slot_full[vidx % NS], (vidx / NS) & 1, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t v_addr = smem_u32(slot_ptr(vidx));
            const uint32_t pb = tmem + (sb ? Cfg::kTmemS1 : Cfg::kTmemS0);
#pragma unroll
            for (int kk = 0; kk < kTileN / 16; ++kk)  // P of keys 64w.. sits at columns 64w..
              mma_f16_ts(tmem + Cfg::kTmemO, pb + 8 * kk + (kk >= 4 ? 32 : 0),
                         sdesc_sw128(v_addr + kk * 2048, Cfg::kRegion, 1024), idesc_o,
                         (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&o_done[sb]);
            mma_commit(&slot_empty[vidx % NS]);
            last_commit = &o_done[sb];
            last_parity = (t >> 1) & 1;
          }
        }
        sidx += 2 * it.n;
        tbase += it.n;
        ++ibase;
      }
      if (!ok && last_commit) drain_wait(last_commit, last_parity, 100000000ull);
    }
  } else if (warp >= 4 && warp < 12) {
    // ---------------------------------------------------------------- softmax
    // two warpgroups; thread (r, w) owns row r and key columns [64w, 64w+64)
    // of every tile.  Per tile the two post their partial row maxima and
    // take the same reference max; each keeps its own partial row sum and
    // writes its half of P (fp16 pairs) over the first 32 columns of the S
    // columns it read, so neither overwrites what the other still reads.
    const int r = (threadIdx.x - 128) & 127;
    const int w = (threadIdx.x - 128) >> 7;
    const int cw = 64 * w;
    const int wq = warp & 3;  // TMEM lane quarter: rows 32*wq .. 32*wq + 31
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const int lg = 31 - __clz(g);
    const float sl2 = p.scale_log2;
    float* xmax = reinterpret_cast<float*>(smem + Cfg::kXchg);  // [2 tiles][2 warpgroups][128]
    float* xsum = xmax + 2 * 2 * 128;                           // [2 items][2 warpgroups][128]
    float* xm = xsum + 2 * 2 * 128;                             // [2 items][128]
    bool ok = true;
    int tbase = 0, ibase = 0;
    // items in order, as staged by the epilogue warps (n == 0 ends the list)
    for (;;) {
      if (!__all_sync(0xffffffffu, mbar_wait(&q_tmem[ibase & 1], (ibase >> 1) & 1, ctl))) {
        ok = false;
        break;
      }
      const int* meta = reinterpret_cast<const int*>(smem + Cfg::kMeta) + (ibase & 1) * Cfg::kMetaInts;
      FwdItem it;
      it.n = meta[0];
      if (it.n == 0) break;
      it.list = p.row_idx + meta[1];
      const int qabs = meta[4 + r];
      const int lo_r = meta[4 + 128 + r];
      float m_run = -INFINITY, l_run = 0.f;
      uint32_t e_next = static_cast<uint32_t>(meta[2]);
      for (int j = 0; j < it.n; ++j) {
        const int t = tbase + j, sb = t & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&s_full[sb], (t >> 1) & 1, ctl))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sc = tmem + lane_base + (sb ? Cfg::kTmemS1 : Cfg::kTmemS0) + cw;
        float s[64];
        {
          uint32_t u[64];
          tmem_ld32_nowait(sc, u);
          tmem_ld32_nowait(sc + 32, u + 32);
          tmem_wait_ld();
          reg_fence32(u);
          reg_fence32(u + 32);
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(u[c]);
        }
        const uint32_t e = e_next;  // list entries run one tile ahead
        if (j + 1 < it.n) e_next = static_cast<uint32_t>(it.list[j + 1]);
        if (e & kPartialBit) {
          const int k0 = static_cast<int>(e & kIndexMask) * kTileN + cw;
          const int lo_c = lo_r - k0, hi_c = qabs - k0;
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < lo_c || c > hi_c) s[c] = -INFINITY;
        }
        float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
        for (int c = 4; c < 64; c += 4) {
          mx0 = fmaxf(mx0, s[c]);
          mx1 = fmaxf(mx1, s[c + 1]);
          mx2 = fmaxf(mx2, s[c + 2]);
          mx3 = fmaxf(mx3, s[c + 3]);
        }
        float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
        xmax[(sb * 2 + w) * 128 + r] = mx;
        __syncwarp();
        if (lane == 0) mbar_arrive(&mx_ready[sb]);
        if (!__all_sync(0xffffffffu, mbar_wait(&mx_ready[sb], (t >> 1) & 1, ctl))) {
          ok = false;
          break;
        }
        mx = fmaxf(mx, xmax[(sb * 2 + (w ^ 1)) * 128 + r]);
        const float mxl2 = mx * sl2;
        const float m_new = (mxl2 > m_run + 8.f) ? mxl2 : m_run;
        const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2(m_run - m_ref);
        // P enters the P V product in fp16 (11-bit significand) against an
        // fp16 copy of V; its values lie in [0, 2^8] thanks to the lazy max.
        // exponent arguments and row sums in packed fp32 pairs
        const uint64_t sl2x2 = f2(sl2, sl2), nm2 = f2(-m_ref, -m_ref);
        uint64_t acc0 = f2(0.f, 0.f), acc1 = f2(0.f, 0.f);
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float x0, x1;
          f2_split(f2_fma(f2(s[c], s[c + 1]), sl2x2, nm2), x0, x1);
          const float e0 = ex2(x0), e1 = ex2(x1);
          if (c & 2) acc1 = f2_add(acc1, f2(e0, e1));
          else acc0 = f2_add(acc0, f2(e0, e1));
          pk[c >> 1] = pack_f16(e0, e1);
        }
        float sa, sb2, sc2, sd;
        f2_split(acc0, sa, sb2);
        f2_split(acc1, sc2, sd);
        l_run = l_run * alpha + ((sa + sb2) + (sc2 + sd));
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_st8_nowait(sc + 8 * q, pk + 8 * q);
        if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // the reference max moved: rescale this warpgroup's half of O
          // once P_{t-1} V_{t-1} is in
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, ctl))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < D / 2; c0 += 32) {
            float tt[32];
            const uint32_t oc = tmem + lane_base + Cfg::kTmemO + w * (D / 2) + c0;
            tmem_ld32(oc, tt);
#pragma unroll
            for (int i = 0; i < 32; ++i) tt[i] *= alpha;
            tmem_st32(oc, tt);
          }
        }
        tmem_wait_st();
        warp_arrive(&p_full[sb]);
        m_run = m_new;
      }
      if (!ok) break;
      // post this item's row statistics for the epilogue warps: each
      // warpgroup's partial row sum, and the reference max (the same in
      // both).  Only once the epilogue has taken the previous item (its O
      // released): l_ready then never runs two phases ahead of the epilogue,
      // and the buffers of this parity (last read for item ibase - 2) are free.
      if (ibase >= 1 && !__all_sync(0xffffffffu, mbar_wait(o_free, (ibase - 1) & 1, ctl))) {
        ok = false;
        break;
      }
      xsum[((ibase & 1) * 2 + w) * 128 + r] = l_run;
      if (w == 0) xm[(ibase & 1) * 128 + r] = m_run;
      __syncwarp();
      if (lane == 0) mbar_arrive(l_ready);
      tbase += it.n;
      ++ibase;
    }
  } else if (warp >= 12) {
    // --------------------------------------------------------------- epilogue
    // per item: once its last P V is done and the softmax warps have posted
    // the row statistics, read O out of TMEM (row r = lane of warp w - 12),
    // hand the accumulator back, then write O / l (per warp, TMA stores of
    // 32 x 32 fp32 blocks) and the LSE; this overlaps the next item's tiles.
    // Ahead of that, the warps copy the next item's Q into the other TMEM Q
    // buffer and stage its metadata for the softmax warps.
    const int wq = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const int lg = 31 - __clz(g);
    const int r = 32 * wq + lane;
    const float* xsum = reinterpret_cast<const float*>(smem + Cfg::kXchg) + 2 * 2 * 128;
    const float* xm = xsum + 2 * 2 * 128;
    const uint32_t stage = smem_u32(smem + Cfg::kStage) + wq * 4096;
    bool ok = true;
    int tbase = 0, ibase = 0;
    // row r of an item's Q (slot q_idx) into TMEM Q buffer qb.  Buffer qb was
    // last used by the item two back, whose products completed before its
    // epilogue, which these warps have done.
    int qn = 0;  // Q tiles copied so far (the q_full / q_empty phase)
    // stage item `mi`'s metadata for the softmax warps into buffer qb (the
    // softmax warps read buffer qb at the top of the item two back, which
    // they have finished); n = 0 marks the end of this CTA's items
    auto stage_meta = [&](int qb, const FwdItem* mi) {
      int* meta = reinterpret_cast<int*>(smem + Cfg::kMeta) + qb * Cfg::kMetaInts;
      if (mi == nullptr) {
        if (r == 0) meta[0] = 0;
        return;
      }
      const int rpos = mi->l0 + (r >> lg);
      meta[4 + r] = p.qpos[rpos];
      meta[4 + 128 + r] = p.doc_lo[static_cast<long long>(mi->b) * Lq + rpos];
      if (r == 0) {
        meta[0] = mi->n;
        meta[1] = static_cast<int>(mi->list - p.row_idx);
        meta[2] = mi->list[0];
      }
    };
    auto copy_q = [&](int qb, const FwdItem& mi) -> bool {
      stage_meta(qb, &mi);
      if (!__all_sync(0xffffffffu, mbar_wait(q_full, qn & 1, ctl))) return false;
      sw128_row_to_tmem<D>(smem_u32(sQ), r, tmem + lane_base + Cfg::kTmemQ + qb * (D / 2));
      tmem_wait_st();
      warp_arrive(&q_tmem[qb]);
      warp_arrive(q_empty);
      ++qn;
      return true;
    };
    bool first = true;
    for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_items; ++k) {
      const int item = snake_item(k);
      if (item >= n_items) continue;
      const FwdItem it = fwd_item(p, item);
      if (it.n == 0) continue;
      if (first) {
        if (!copy_q(ibase & 1, it)) { ok = false; break; }
        first = false;
      }
      // the next item's Q into the other buffer as soon as it has landed, so
      // that the S products run on into the next item without a gap
      {
        bool more = false;
        for (int kx = k + 1; kx * static_cast<int>(gridDim.x) < n_items; ++kx) {
          const int cand = snake_item(kx);
          if (cand >= n_items) continue;
          const FwdItem nx = fwd_item(p, cand);
          if (nx.n == 0) continue;
          if (!copy_q((ibase + 1) & 1, nx)) ok = false;
          more = true;
          break;
        }
        if (!ok) break;
        if (!more) {  // end of this CTA's items
          stage_meta((ibase + 1) & 1, nullptr);
          warp_arrive(&q_tmem[(ibase + 1) & 1]);
        }
      }
      const int t_last = tbase + it.n - 1;
      if (!__all_sync(0xffffffffu, mbar_wait(l_ready, ibase & 1, ctl)) ||
          !__all_sync(0xffffffffu,
                      mbar_wait(&o_done[t_last & 1], (t_last >> 1) & 1, ctl))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float l_tot = xsum[((ibase & 1) * 2) * 128 + r] + xsum[((ibase & 1) * 2 + 1) * 128 + r];
      const float m_ref = xm[(ibase & 1) * 128 + r];
      const float inv = 1.f / l_tot;
      uint32_t u[D];
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32)
        tmem_ld32_nowait(tmem + lane_base + Cfg::kTmemO + c0, u + c0);
      tmem_wait_ld();
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) reg_fence32(u + c0);
      warp_arrive(o_free);
      // O / l in blocks of 32 columns x this warp's 32 rows, each written
      // with one TMA store (rows = 32/g positions x the g heads)
      const int zrow = it.b * Lq + it.l0 + ((32 * wq) >> lg);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        // the previous block's store must have read the staging buffer
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          st_shared_v4(stage + lane * 128 + ((ch ^ (lane & 7)) << 4),
                       __float_as_uint(__uint_as_float(u[c0 + 4 * ch]) * inv),
                       __float_as_uint(__uint_as_float(u[c0 + 4 * ch + 1]) * inv),
                       __float_as_uint(__uint_as_float(u[c0 + 4 * ch + 2]) * inv),
                       __float_as_uint(__uint_as_float(u[c0 + 4 * ch + 3]) * inv));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&to, smem + Cfg::kStage + wq * 4096, c0, it.kvh * g, zrow);
          bulk_commit();
        }
      }
      lse[(static_cast<long long>(it.b) * p.n_heads + it.kvh * g + (r & (g - 1))) * Lq + it.l0 +
          (r >> lg)] = (m_ref + lg2(l_tot)) * 0.6931471805599453f;
      tbase += it.n;
      ++ibase;
    }
    if (ok && first) {  // no items at all: release the softmax warps
      stage_meta(0, nullptr);
      warp_arrive(&q_tmem[0]);
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

// V (bf16) -> fp16 copy for the P V product; values beyond the fp16 range
// saturate at +-65504.  8 elements per thread.
__global__ void v_to_f16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                long long n8) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 a = src[i];
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    uint32_t o4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = fminf(fmaxf(__uint_as_float(w[e] << 16), -65504.f), 65504.f);
      const float hi = fminf(fmaxf(__uint_as_float(w[e] & 0xFFFF0000u), -65504.f), 65504.f);
      o4[e] = pack_f16(lo, hi);
    }
    dst[i] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
  }
}

template <int D>
cudaError_t launch_fwd_d(const dma_plan_s& pl, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv16, const CUtensorMap& to, float* o, float* lse,
                         cudaStream_t s) {
  const PlanDev& p = pl.d;
  const int items = p.batch * p.n_qtiles * p.n_kv_heads;
  if (items == 0) return cudaSuccess;
  // persistent: one CTA per SM (TMEM and shared memory allow no more)
  const int grid = items < pl.num_sms ? items : pl.num_sms;
  const int smem = FwdCfg<D>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  fwd_kernel<D><<<grid, 512, smem, s>>>(tq, tk, tv16, to, p, o, lse, items);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_v_to_f16(const dma_plan_s& pl, const dma_bf16* v, cudaStream_t s) {
  const PlanDev& p = pl.d;
  const long long n8 = static_cast<long long>(p.batch) * p.seq_len * p.n_kv_heads * p.head_dim / 8;
  if (n8 == 0) return cudaSuccess;
  long long blocks = (n8 + 255) / 256;
  if (blocks > 8LL * pl.num_sms) blocks = 8LL * pl.num_sms;
  v_to_f16_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(reinterpret_cast<const uint4*>(v),
                                                        reinterpret_cast<uint4*>(p.v16), n8);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const dma_plan_s& pl, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv16, const CUtensorMap& to, float* o, float* lse,
                       cudaStream_t s) {
  if (pl.d.head_dim == 128) return launch_fwd_d<128>(pl, tq, tk, tv16, to, o, lse, s);
  return launch_fwd_d<64>(pl, tq, tk, tv16, to, o, lse, s);
}

}  // namespace dma
