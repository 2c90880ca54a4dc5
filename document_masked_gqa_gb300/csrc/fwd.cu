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
//   warp 0      TMA producer: per item Q (two buffers), then K_j and V_j
//               (fp16 copy) for each key tile through two rings of
//               tile-sized slots, K one tile ahead of V
//   warp 1      tcgen05 issuer for S = Q K^T into one of three TMEM buffers
//               (Q and K from shared memory); owns the TMEM allocation
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
// Three S buffers let S_{t+1} and S_{t+2} be computed while tile t's
// softmax and P V run: S_{t+3} waits only for P_t V_t, which reads P_t from
// S_t's buffer, so the softmax warps rarely wait for a score tile.
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
  // K_j and V_j of each work item's row list go through two rings of
  // tile-sized slots, K loaded a tile ahead of V; Q has two buffers of its
  // own (item i uses buffer i % 2, so the next item's Q loads while the
  // current one is still in use)
  static constexpr int kKVSlots = (D == 128) ? 2 : 4;  // per ring
  static constexpr int kKring = 0;
  static constexpr int kVring = kKring + kKVSlots * kTileBytes;
  static constexpr int kQbuf = kVring + kKVSlots * kTileBytes;  // 2 buffers
  // O epilogue staging: per epilogue warp one 4 KB block of 32 rows x 32
  // fp32 in the 128-byte swizzled layout of a TMA store
  static constexpr int kStage = kQbuf + 2 * kTileBytes;
  // row maxima [2 tiles][2 warpgroups][128], then per item parity: row sums
  // [2][2 warpgroups][128] and reference maxima [2][128]
  static constexpr int kXchg = kStage + 4 * 4096;
  // per item parity, staged by the epilogue warps ahead of the item: n, list
  // offset, first list entry, then per row the query position and its
  // document's first position
  static constexpr int kMeta = kXchg + (2 * 2 * 128 + 2 * 2 * 128 + 2 * 128) * 4;
  static constexpr int kMetaInts = 4 + 2 * 128;
  static constexpr int kBar = kMeta + 2 * kMetaInts * 4;
  // work items published by the producer to the other roles (ItemRing)
  static constexpr int kRing = 8;
  static constexpr int kNumBars = 4 * kKVSlots + 3 * 3 + 2 + 1 + 2 + 1 + 2 + 2 + 2 * kRing;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kEnd = kMisc + 16 + 4 * kRing;
  static constexpr int kSmemBytes = kEnd + 1024;
  static constexpr uint32_t kTmemCols = 512;
  // TMEM: three S buffers (128 columns each; P overwrites part of one as
  // fp16 pairs; tile t uses buffer t % 3) and the O accumulator
  static constexpr uint32_t kTmemO = 384;
  static_assert(kTmemO + D <= 512, "forward TMEM layout exceeds 512 columns");
  static_assert(kSmemBytes <= 232448, "forward shared-memory layout exceeds 227 KB");
};

// Register split of the 512 threads launched at 128 registers each: the
// producer / issuer warpgroup (warps 0-3) and the epilogue warpgroup give
// registers to the softmax warps (measured: the softmax runs faster with the
// room).  Each warpgroup sets its share at one call site at the top of its
// branch, the same count for its four warps.
constexpr uint32_t kFwdCtlRegs = 88, kFwdSmRegs = 168, kFwdEpiRegs = 88;
static_assert(4 * kFwdCtlRegs + 8 * kFwdSmRegs + 4 * kFwdEpiRegs <= 16 * 128,
              "forward register split exceeds the launch's 512 x 128 registers");

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

// Persistent: the producer thread takes work items from the plan's counter
// one at a time and publishes them to the S and P V issuers and the epilogue
// warps (ItemRing); the softmax warps get theirs from the epilogue warps'
// metadata.  Every role keeps the same counters across non-empty items: the key tiles processed so far
// (tbase: K / V slot t % kKVSlots, S buffer t % 3 and every per-tile barrier
// parity follow from the global tile index t) and the items so far (ibase:
// Q buffer and metadata buffer ibase % 2, parity of l_ready and o_free).
template <int D>
__global__ void __launch_bounds__(512, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
               const PlanDev p, float* __restrict__ o, float* __restrict__ lse, int n_items) {
  using Cfg = FwdCfg<D>;
  constexpr int NS = Cfg::kKVSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  int32_t* const ctr = p.sched + kSchedFwd;

  // a failed plan or an earlier expired wait: do nothing (CTA-uniform)
  if (__syncthreads_or(threadIdx.x == 0 &&
                       *reinterpret_cast<volatile uint32_t*>(p.status) != 0u)) {
    if (threadIdx.x == 0) items_exit(ctr);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.group, Lq = p.local_len;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBar);
  uint64_t* k_full = bars;              // [NS] K ring
  uint64_t* k_empty = bars + NS;        // [NS]
  uint64_t* v_full = bars + 2 * NS;     // [NS] V ring
  uint64_t* v_empty = bars + 3 * NS;    // [NS]
  // per S buffer (tile t uses buffer t % 3), so that no waiter can fall two
  // phases behind while the S and P V issuers run independently
  uint64_t* s_full = bars + 4 * NS;    // [3] S computed
  uint64_t* p_full = s_full + 3;       // [3] P written over S
  uint64_t* o_done = p_full + 3;       // [3] P V of a tile done (its S buffer is free)
  uint64_t* mx_ready = o_done + 3;     // [2] both softmax warpgroups posted a tile's row maxima
  uint64_t* l_ready = mx_ready + 2;    // both posted an item's partial row sums
  uint64_t* meta_ready = l_ready + 1;  // [2] an item's metadata staged in buffer item % 2
  uint64_t* o_free = meta_ready + 2;   // the epilogue warps have read an item's O
  uint64_t* q_full = o_free + 1;       // [2] an item's Q in Q buffer item % 2
  uint64_t* q_empty = q_full + 2;      // [2] ... and all its S products done
  uint64_t* item_full = q_empty + 2;   // [kRing]
  uint64_t* item_empty = item_full + Cfg::kRing;
  const ItemRing<Cfg::kRing> ring{reinterpret_cast<volatile int*>(smem + Cfg::kMisc + 16), item_full,
                                  item_empty};
  uint8_t* sQ = smem + Cfg::kQbuf;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + Cfg::kMisc + 4);
  auto k_slot = [&](int t) { return smem + Cfg::kKring + (t % NS) * Cfg::kTileBytes; };
  auto v_slot = [&](int t) { return smem + Cfg::kVring + (t % NS) * Cfg::kTileBytes; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    // the softmax and epilogue warps arrive once per warp
    for (int i = 0; i < 3; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 8);
      mbar_init(&o_done[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&mx_ready[i], 8);
      mbar_init(&meta_ready[i], 4);
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    mbar_init(l_ready, 8);
    mbar_init(o_free, 4);
    // readers of the item ring: the producer's V cursor, the two issuers, the
    // four epilogue warps
    for (int i = 0; i < Cfg::kRing; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], 7);
    }
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

  if (warp < 4) {
    // warpgroup 0: producer (warp 0), issuers (warps 1, 3); warp 2 has no role
    reg_dealloc<kFwdCtlRegs>();
    if (warp == 0) {
      if (lane == 0) {
        // ------------------------------------------------ producer: the stream
        // Two cursors walk this CTA's key tiles in order: the K cursor (which
        // also loads an item's Q when it enters the item) runs one tile ahead
        // of the V cursor, so that the S products never wait for a V slot to
        // free.  Tile t's K goes to K slot t % NS once S_{t-NS} is done, its V
        // to V slot t % NS once P_{t-NS} V_{t-NS} is done.
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        struct Cursor {
          int r;     // ring entries read (the K cursor: published)
          int j;     // tile within the current item
          int t;     // global tile index
          int item;  // non-empty items entered so far - 1
          FwdItem it;
          bool done;
        };
        // move a cursor to the first tile of the next non-empty item: the K
        // cursor takes the next index from the counter (one item ahead, so
        // that the atomic's latency is hidden) and publishes it unless its
        // list is empty; the V cursor reads what the K cursor published
        int next_idx = take_item(ctr);
        auto next_item = [&](Cursor& c, bool is_k) -> bool {
          for (;;) {
            int item;
            if (is_k) {
              item = next_idx < n_items ? next_idx : -1;
              if (item >= 0) {
                next_idx = take_item(ctr);
                if (fwd_item(p, item).n == 0) continue;
              }
              if (!ring.put(c.r++, item, ctl)) return false;
            } else if (!ring.get(c.r++, item, ctl)) {
              return false;
            }
            if (item < 0) {
              c.done = true;
              return true;
            }
            c.it = fwd_item(p, item);
            c.j = 0;
            ++c.item;
            return true;
          }
        };
        Cursor kc{0, 0, 0, -1, FwdItem{}, false}, vc = kc;
        bool ok = next_item(kc, true) && next_item(vc, false);
        int q_issued = 0;  // Q loads issued (item index of the next one)
        while (ok && !vc.done) {
          const bool do_k = !kc.done && kc.t <= vc.t + 1;
          Cursor& c = do_k ? kc : vc;
          if (do_k && c.j == 0 && q_issued == c.item) {
            // entering an item: its Q into buffer item % 2 once the S products
            // of the item two back are done
            const int qb = c.item & 1;
            if (!mbar_wait(&q_empty[qb], ((c.item >> 1) & 1) ^ 1u, ctl)) { ok = false; break; }
            mbar_arrive_expect_tx(&q_full[qb], Cfg::kTileBytes);
#pragma unroll
            for (int ch = 0; ch < Cfg::kChunks; ++ch)
              tma_load_3d(sQ + qb * Cfg::kTileBytes + ch * Cfg::kRegion, &tq, &q_full[qb], ch * 64,
                          c.it.kvh * g, c.it.b * Lq + c.it.l0);
            ++q_issued;
          }
          const int kt = static_cast<int>(static_cast<uint32_t>(c.it.list[c.j]) & kIndexMask);
          const int krow = c.it.b * p.seq_len + kt * kTileN;
          const int sl = c.t % NS;
          const uint32_t ph = ((c.t / NS) & 1) ^ 1u;
          uint64_t* full = do_k ? &k_full[sl] : &v_full[sl];
          if (!mbar_wait(do_k ? &k_empty[sl] : &v_empty[sl], ph, ctl)) { ok = false; break; }
          mbar_arrive_expect_tx(full, Cfg::kTileBytes);
          uint8_t* dst = do_k ? k_slot(c.t) : v_slot(c.t);
#pragma unroll
          for (int ch = 0; ch < Cfg::kChunks; ++ch)
            tma_load_2d(dst + ch * Cfg::kRegion, do_k ? &tk : &tv, full, c.it.kvh * D + ch * 64, krow);
          ++c.t;
          if (++c.j == c.it.n && !next_item(c, do_k)) ok = false;
        }
        if (!ok) {  // drain this CTA's copies still in flight
          for (int t = max(0, kc.t - NS); t < kc.t; ++t)
            drain_wait(&k_full[t % NS], (t / NS) & 1, 100000000ull);
          for (int t = max(0, vc.t - NS); t < vc.t; ++t)
            drain_wait(&v_full[t % NS], (t / NS) & 1, 100000000ull);
          for (int i = max(0, q_issued - 2); i < q_issued; ++i)
            drain_wait(&q_full[i & 1], (i >> 1) & 1, 100000000ull);
        }
      }
    } else if (warp == 1 || warp == 3) {
      if (lane == 0) {
        // ------------------------------------------------------ MMA issuers
        // warp 1: S_t = Q K_t^T into TMEM buffer t % 3 (Q and K from shared
        // memory); the buffer is reused for S_{t+3} once P_t V_t (which reads
        // P_t from it) has completed.  warp 3: once the softmax has written P_t
        // over S_t: O += P_t V_t with A = P_t from TMEM.  Two issuing threads
        // keep the tensor pipe fed while the softmax warps keep the schedulers
        // busy.
        constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
        constexpr uint32_t idesc_o = idesc_f16_f32(128, D, 0, 1);
        uint64_t* last_commit = nullptr;
        uint32_t last_parity = 0;
        bool ok = true;
        int tbase = 0, ibase = 0;
        for (int rk = 0; ok; ++rk) {
          int item;
          if (!ring.get(rk, item, ctl)) { ok = false; break; }
          if (item < 0) break;
          const FwdItem it = fwd_item(p, item);
          if (it.n == 0) continue;
          const int qb = ibase & 1;
          if (warp == 1 && !mbar_wait(&q_full[qb], (ibase >> 1) & 1, ctl)) { ok = false; break; }
          const uint32_t q_addr = smem_u32(sQ + qb * Cfg::kTileBytes);
          for (int j = 0; j < it.n; ++j) {
            const int t = tbase + j, sb = t % 3;
            const uint32_t use = (t / 3) & 1;  // parity of this use of buffer sb
            const uint32_t kv_ph = (t / NS) & 1;
            if (warp == 1) {
              if (!mbar_wait(&k_full[t % NS], kv_ph, ctl)) { ok = false; break; }
              if (t >= 3 && !mbar_wait(&o_done[sb], use ^ 1u, ctl)) { ok = false; break; }
              tc_fence_after();
              const uint32_t k_addr = smem_u32(k_slot(t));
              const uint32_t d_s = tmem + 128 * sb;
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * Cfg::kRegion + (kk & 3) * 32;
                mma_bf16_ss(d_s, sdesc_sw128(q_addr + off, 16, 1024),
                            sdesc_sw128(k_addr + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
              }
              mma_commit(&s_full[sb]);
              mma_commit(&k_empty[t % NS]);
              last_commit = &s_full[sb];
              last_parity = use;
            } else {
              // the item's first P V overwrites O: the previous item's O must
              // have been read out by the epilogue warps
              if (j == 0 && ibase > 0 && !mbar_wait(o_free, (ibase - 1) & 1, ctl)) { ok = false; break; }
              if (!mbar_wait(&p_full[sb], use, ctl)) { ok = false; break; }
              if (!mbar_wait(&v_full[t % NS], kv_ph, ctl)) { ok = false; break; }
              tc_fence_after();
              const uint32_t v_addr = smem_u32(v_slot(t));
              const uint32_t pb = tmem + 128 * sb;
#pragma unroll
              for (int kk = 0; kk < kTileN / 16; ++kk)  // P of keys 64w.. sits at columns 64w..
                mma_f16_ts(tmem + Cfg::kTmemO, pb + 8 * kk + (kk >= 4 ? 32 : 0),
                           sdesc_sw128(v_addr + kk * 2048, Cfg::kRegion, 1024), idesc_o,
                           (j > 0 || kk > 0) ? 1u : 0u);
              mma_commit(&o_done[sb]);
              mma_commit(&v_empty[t % NS]);
              last_commit = &o_done[sb];
              last_parity = use;
            }
          }
          if (!ok) break;
          if (warp == 1) mma_commit(&q_empty[qb]);  // the item's Q reads are done once these complete
          tbase += it.n;
          ++ibase;
        }
        if (!ok && last_commit) drain_wait(last_commit, last_parity, 100000000ull);
      }
    }
  } else if (warp < 12) {
    reg_alloc<kFwdSmRegs>();
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
      if (!__all_sync(0xffffffffu, mbar_wait(&meta_ready[ibase & 1], (ibase >> 1) & 1, ctl))) {
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
        const int t = tbase + j, sb = t % 3, xb = t & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&s_full[sb], (t / 3) & 1, ctl))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sc = tmem + lane_base + 128 * sb + cw;
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
        // row max of this half: three-input maxima, four chains
        float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
        for (int c = 4; c < 60; c += 8) {
          mx0 = max3f(mx0, s[c], s[c + 1]);
          mx1 = max3f(mx1, s[c + 2], s[c + 3]);
          mx2 = max3f(mx2, s[c + 4], s[c + 5]);
          mx3 = max3f(mx3, s[c + 6], s[c + 7]);
        }
        mx0 = max3f(mx0, s[60], s[61]);
        mx1 = max3f(mx1, s[62], s[63]);
        float mx = max3f(mx0, mx1, fmaxf(mx2, mx3));
        xmax[(xb * 2 + w) * 128 + r] = mx;
        __syncwarp();
        if (lane == 0) mbar_arrive(&mx_ready[xb]);
        if (!__all_sync(0xffffffffu, mbar_wait(&mx_ready[xb], (t >> 1) & 1, ctl))) {
          ok = false;
          break;
        }
        mx = fmaxf(mx, xmax[(xb * 2 + (w ^ 1)) * 128 + r]);
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
                          mbar_wait(&o_done[(t - 1) % 3], ((t - 1) / 3) & 1, ctl))) {
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
    tmem_wait_ld();  // (after an abort a score load may still be in flight)
  } else {
    reg_dealloc<kFwdEpiRegs>();
    // --------------------------------------------------------------- epilogue
    // per item: once its last P V is done and the softmax warps have posted
    // the row statistics, read O out of TMEM (row r = lane of warp w - 12),
    // hand the accumulator back, then write O / l (per warp, TMA stores of
    // 32 x 32 fp32 blocks) and the LSE; this overlaps the next item's tiles.
    // Ahead of that, the warps stage the next item's metadata for the
    // softmax warps.
    const int wq = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const int lg = 31 - __clz(g);
    const int r = 32 * wq + lane;
    const float* xsum = reinterpret_cast<const float*>(smem + Cfg::kXchg) + 2 * 2 * 128;
    const float* xm = xsum + 2 * 2 * 128;
    const uint32_t stage = smem_u32(smem + Cfg::kStage) + wq * 4096;
    bool ok = true;
    int tbase = 0, ibase = 0;
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
    auto post_meta = [&](int qb, const FwdItem* mi) {
      stage_meta(qb, mi);
      warp_arrive(&meta_ready[qb]);
    };
    // the next non-empty item from the ring (found = false at the end)
    int rk = 0;
    auto read_item = [&](FwdItem& out, bool& found) -> bool {
      for (;;) {
        int item;
        if (!ring.get_warp(rk++, item, ctl)) return false;
        if (item < 0) {
          found = false;
          return true;
        }
        out = fwd_item(p, item);
        if (out.n > 0) {
          found = true;
          return true;
        }
      }
    };
    FwdItem nx{};
    bool have = false;
    ok = read_item(nx, have);
    if (ok) post_meta(0, have ? &nx : nullptr);  // nothing at all: releases the softmax warps
    while (ok && have) {
      const FwdItem it = nx;
      // the next item's metadata into the other buffer, so that the softmax
      // warps run on into the next item without a gap (n = 0: the end)
      if (!read_item(nx, have)) {
        ok = false;
        break;
      }
      post_meta((ibase + 1) & 1, have ? &nx : nullptr);
      const int t_last = tbase + it.n - 1;
      if (!__all_sync(0xffffffffu, mbar_wait(l_ready, ibase & 1, ctl)) ||
          !__all_sync(0xffffffffu,
                      mbar_wait(&o_done[t_last % 3], (t_last / 3) & 1, ctl))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float l_tot = xsum[((ibase & 1) * 2) * 128 + r] + xsum[((ibase & 1) * 2 + 1) * 128 + r];
      const float m_ref = xm[(ibase & 1) * 128 + r];
      const float inv = 1.f / l_tot;
      // O / l in blocks of 32 columns x this warp's 32 rows, each written
      // with one TMA store (rows = 32/g positions x the g heads); O is read
      // out of TMEM 64 columns at a time and handed back after the last read
      const int zrow = it.b * Lq + it.l0 + ((32 * wq) >> lg);
#pragma unroll
      for (int h0 = 0; h0 < D; h0 += 64) {
        uint32_t u[64];
        tmem_ld32_nowait(tmem + lane_base + Cfg::kTmemO + h0, u);
        tmem_ld32_nowait(tmem + lane_base + Cfg::kTmemO + h0 + 32, u + 32);
        tmem_wait_ld();
        reg_fence32(u);
        reg_fence32(u + 32);
        if (h0 + 64 >= D) warp_arrive(o_free);
#pragma unroll
        for (int c1 = 0; c1 < 64; c1 += 32) {
          // the previous block's store must have read the staging buffer
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            st_shared_v4(stage + lane * 128 + ((ch ^ (lane & 7)) << 4),
                         __float_as_uint(__uint_as_float(u[c1 + 4 * ch]) * inv),
                         __float_as_uint(__uint_as_float(u[c1 + 4 * ch + 1]) * inv),
                         __float_as_uint(__uint_as_float(u[c1 + 4 * ch + 2]) * inv),
                         __float_as_uint(__uint_as_float(u[c1 + 4 * ch + 3]) * inv));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&to, smem + Cfg::kStage + wq * 4096, h0 + c1, it.kvh * g, zrow);
            bulk_commit();
          }
        }
      }
      lse[(static_cast<long long>(it.b) * p.n_heads + it.kvh * g + (r & (g - 1))) * Lq + it.l0 +
          (r >> lg)] = (m_ref + lg2(l_tot)) * 0.6931471805599453f;
      tbase += it.n;
      ++ibase;
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
  if (threadIdx.x == 0) items_exit(ctr);
}

// V (bf16) -> fp16 copy for the P V product, 8 elements per thread.  NaN and
// +-Inf pass through unchanged (a NaN in V reaches O as it would in bf16
// arithmetic).  Finite values beyond the fp16 range (|v| > 65504) saturate at
// +-65504, and the kernel then sets bit 0 of warn (the plan's warning word),
// which dma_plan_check reports as DMA_WARN_V_SATURATED.
__device__ __forceinline__ float sat_f16_range(float x, bool& clamped) {
  const bool over = fabsf(x) > 65504.f && fabsf(x) <= 3.402823466e38f;  // finite only
  clamped |= over;
  return over ? copysignf(65504.f, x) : x;
}
__global__ void v_to_f16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                long long n8, uint32_t* __restrict__ warn) {
  bool clamped = false;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 a = src[i];
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    uint32_t o4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = sat_f16_range(__uint_as_float(w[e] << 16), clamped);
      const float hi = sat_f16_range(__uint_as_float(w[e] & 0xFFFF0000u), clamped);
      o4[e] = pack_f16(lo, hi);
    }
    dst[i] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
  }
  if (__any_sync(0xffffffffu, clamped) && (threadIdx.x & 31) == 0) atomicOr(warn, 1u);
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
  v_to_f16_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(v), reinterpret_cast<uint4*>(p.v16), n8, p.status + 1);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const dma_plan_s& pl, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv16, const CUtensorMap& to, float* o, float* lse,
                       cudaStream_t s) {
  if (pl.d.head_dim == 128) return launch_fwd_d<128>(pl, tq, tk, tv16, to, o, lse, s);
  return launch_fwd_d<64>(pl, tq, tk, tv16, to, o, lse, s);
}

}  // namespace dma
