// Forward kernel: causal + document-masked GQA attention for one CP rank.
//
// One CTA per (query tile, K/V head).  A query tile is 128 rows: P = 128/g
// consecutive local positions x the g query heads sharing K/V head `kvh`
// (GQA, "The Llama 3 Herd of Models - part 3/16", 3.3.2, and "Paper notes:
// The Llama 3 Herd of Models", 8 key-value heads), so one K/V tile feeds g
// heads at once.  The CTA walks the tile's list of non-skipped key tiles
// (built by the block-mask builder) and keeps the online-softmax running max
// and sum per row, rescaling the partial output, then divides by the sum
// ("Training Infrastructure and Systems", "FlashAttention: never write the
// score matrix", sections "Online softmax" and "Tiling").
//
// GB300 mapping (sm_103a):
//   warp 0      TMA producer: Q once, then K tiles into a 3-stage ring
//   warp 2      TMA producer: V tiles into a 2-stage ring (decoupled from K,
//               so a K load never queues behind the release of a V slot)
//   warp 1      tcgen05 issuer: S = Q K^T into one of two TMEM buffers (Q
//               copied once into TMEM as the A operand), O += P V into a
//               TMEM accumulator with P taken from TMEM; owns the allocation
//   warps 2-3   load the tile's positions / document starts first
//   warps 4-7   softmax: thread r owns row r (TMEM lane r): masks partial
//               tiles, exponentiates in base 2, writes P (fp16 pairs) back
//               over the S columns it has read, rescales O in TMEM when its
//               reference max moves, and writes O (fp32) and LSE.
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
  static constexpr int kStagesK = 3;
  static constexpr int kStagesV = 3;
  static constexpr int kRegion = 128 * 128;       // one 64-column SW128 region of a 128-row tile
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = 128 * D * 2;  // Q, K or V tile (16-bit)
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kStagesK * kTileBytes;
  static constexpr int kBar = kV + kStagesV * kTileBytes;
  static constexpr int kNumBars = 2 + 2 * kStagesK + 2 * kStagesV + 2 + 2 + 2 + 3;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kEnd = kMisc + 16 + 2 * 128 * 4;
  static constexpr int kSmemBytes = kEnd + 1024;
  static constexpr uint32_t kTmemCols = 512;
  // TMEM: S buffers (128 columns each; P overwrites their first 64 as fp16
  // pairs), the O accumulator, and Q as bf16 pairs (the A operand of Q K^T)
  static constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemO = 256, kTmemQ = 384;
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

template <int D>
__global__ void __launch_bounds__(384, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const PlanDev p,
               float* __restrict__ o, float* __restrict__ lse) {
  using Cfg = FwdCfg<D>;
  constexpr int SK = Cfg::kStagesK, SV = Cfg::kStagesV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  // a failed plan or an earlier expired wait: do nothing (CTA-uniform)
  if (__syncthreads_or(threadIdx.x == 0 &&
                       *reinterpret_cast<volatile uint32_t*>(p.status) != 0u))
    return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = p.n_kv_heads, g = p.group, P = p.tile_pos, Lq = p.local_len;
  const int ord = blockIdx.x / Hkv, kvh = blockIdx.x % Hkv;
  const int bq = p.fwd_order[ord];
  const int b = bq / p.n_qtiles, qt = bq % p.n_qtiles;
  const int l0 = qt * P;
  const int rp0 = p.row_ptr[bq];
  const int n = p.row_ptr[bq + 1] - rp0;
  const int32_t* list = p.row_idx + rp0;

  uint8_t* sQ = smem + Cfg::kQ;
  uint8_t* sK = smem + Cfg::kK;
  uint8_t* sV = smem + Cfg::kV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBar);
  uint64_t* q_full = bars;          // Q in shared memory
  uint64_t* q_tmem = bars + 1;      // Q copied into TMEM
  uint64_t* k_full = bars + 2;
  uint64_t* k_empty = k_full + SK;
  uint64_t* v_full = k_empty + SK;
  uint64_t* v_empty = v_full + SV;
  uint64_t* s_full = v_empty + SV;  // [2]
  // per S buffer (tile parity), so that no waiter can fall two phases behind
  // while the S and P V issuers run independently
  uint64_t* p_full = s_full + 2;    // [2] P written over S
  uint64_t* o_done = p_full + 2;    // [2] P V of a tile done (its S buffer is free)
  uint64_t* mx_ready = o_done + 2;  // [2] both softmax warpgroups posted a tile's row maxima
  uint64_t* l_ready = mx_ready + 2; // both posted their partial row sums
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + Cfg::kMisc + 4);
  int* s_qpos = reinterpret_cast<int*>(smem + Cfg::kMisc + 16);
  int* s_lo = s_qpos + 128;

  if (threadIdx.x == 0) {
    // the softmax warps arrive once per warp (8 warps; 4 of them copy Q)
    mbar_init(q_full, 1);
    mbar_init(q_tmem, 4);
    for (int i = 0; i < SK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < SV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&s_full[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 8);
      mbar_init(&o_done[i], 1);
      mbar_init(&mx_ready[i], 8);
    }
    mbar_init(l_ready, 8);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, Cfg::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 2 || warp == 3) {
    for (int r = threadIdx.x - 64; r < P; r += 64) {
      s_qpos[r] = p.qpos[l0 + r];
      s_lo[r] = p.doc_lo[static_cast<long long>(b) * Lq + l0 + r];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------- producer: Q, then K
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      int last_k[SK];
#pragma unroll
      for (int i = 0; i < SK; ++i) last_k[i] = -1;
      mbar_arrive_expect_tx(q_full, Cfg::kTileBytes);
#pragma unroll
      for (int c = 0; c < Cfg::kChunks; ++c)
        tma_load_3d(sQ + c * Cfg::kRegion, &tq, q_full, c * 64, kvh * g, b * Lq + l0);
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        const int st = j % SK;
        const uint32_t ph = (j / SK) & 1;
        const int kt = static_cast<int>(static_cast<uint32_t>(list[j]) & kIndexMask);
        if (!mbar_wait(&k_empty[st], ph ^ 1u, ctl)) { ok = false; break; }
        mbar_arrive_expect_tx(&k_full[st], Cfg::kTileBytes);
#pragma unroll
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_2d(sK + st * Cfg::kTileBytes + c * Cfg::kRegion, &tk, &k_full[st],
                      kvh * D + c * 64, b * p.seq_len + kt * kTileN);
#pragma unroll
        for (int i = 0; i < SK; ++i)
          if (i == st) last_k[i] = static_cast<int>(ph);
      }
      if (!ok) {  // drain our own copies before the CTA exits
        drain_wait(q_full, 0, 100000000ull);
#pragma unroll
        for (int i = 0; i < SK; ++i)
          if (last_k[i] >= 0) drain_wait(&k_full[i], last_k[i], 100000000ull);
      }
    }
  } else if (warp == 2) {
    if (lane == 0) {
      // ------------------------------------------------------ producer: V
      tma_prefetch_desc(&tv);
      int last_v[SV];
#pragma unroll
      for (int i = 0; i < SV; ++i) last_v[i] = -1;
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        const int st = j % SV;
        const uint32_t ph = (j / SV) & 1;
        const int kt = static_cast<int>(static_cast<uint32_t>(list[j]) & kIndexMask);
        if (!mbar_wait(&v_empty[st], ph ^ 1u, ctl)) { ok = false; break; }
        mbar_arrive_expect_tx(&v_full[st], Cfg::kTileBytes);
#pragma unroll
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_2d(sV + st * Cfg::kTileBytes + c * Cfg::kRegion, &tv, &v_full[st],
                      kvh * D + c * 64, b * p.seq_len + kt * kTileN);
#pragma unroll
        for (int i = 0; i < SV; ++i)
          if (i == st) last_v[i] = static_cast<int>(ph);
      }
      if (!ok) {
#pragma unroll
        for (int i = 0; i < SV; ++i)
          if (last_v[i] >= 0) drain_wait(&v_full[i], last_v[i], 100000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && n > 0) {
      // ------------------------------------------------------ MMA issuer: S
      // S_j = Q K_j^T into TMEM buffer j%2 (A = Q from TMEM); the buffer is
      // reused for S_{j+2} once P_j V_j (which reads P_j from it) has
      // completed.
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
      uint64_t* last_commit = nullptr;
      uint32_t last_parity = 0;
      bool ok = mbar_wait(q_tmem, 0, ctl);
      for (int j = 0; ok && j < n; ++j) {
        const int st = j % SK;
        const uint32_t ph = (j / SK) & 1;
        const int sb = j & 1;
        if (!mbar_wait(&k_full[st], ph, ctl)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(&o_done[sb], ((j - 2) >> 1) & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        const uint32_t k_addr = smem_u32(sK + st * Cfg::kTileBytes);
        const uint32_t d_s = tmem + (sb ? Cfg::kTmemS1 : Cfg::kTmemS0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_f16_ts(d_s, tmem + Cfg::kTmemQ + 8 * kk,
                     sdesc_sw128(k_addr + (kk >> 2) * Cfg::kRegion + (kk & 3) * 32, 16, 1024),
                     idesc_s, kk > 0 ? 1u : 0u);
        mma_commit(&s_full[sb]);
        mma_commit(&k_empty[st]);
        last_commit = &s_full[sb];
        last_parity = (j >> 1) & 1;
      }
      if (!ok && last_commit) drain_wait(last_commit, last_parity, 100000000ull);
    }
  } else if (warp == 3) {
    if (lane == 0 && n > 0) {
      // ----------------------------------------------------- MMA issuer: P V
      // once the softmax has written P_j (fp16) over S_j: O += P_j V_j with
      // A = P_j from TMEM.  A second issuing thread keeps this product queued
      // while the S issuer waits.
      constexpr uint32_t idesc_o = idesc_f16_f32(128, D, 0, 1);
      uint64_t* last_commit = nullptr;
      uint32_t last_parity = 0;
      bool ok = true;
      for (int i = 0; ok && i < n; ++i) {
        const int st = i % SV;
        const uint32_t ph = (i / SV) & 1;
        if (!mbar_wait(&p_full[i & 1], (i >> 1) & 1, ctl)) { ok = false; break; }
        if (!mbar_wait(&v_full[st], ph, ctl)) { ok = false; break; }
        tc_fence_after();
        const uint32_t v_addr = smem_u32(sV + st * Cfg::kTileBytes);
        const uint32_t pb = tmem + ((i & 1) ? Cfg::kTmemS1 : Cfg::kTmemS0);
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk)  // P of keys 64w.. sits at columns 64w..
          mma_f16_ts(tmem + Cfg::kTmemO, pb + 8 * kk + (kk >= 4 ? 32 : 0),
                     sdesc_sw128(v_addr + kk * 2048, Cfg::kRegion, 1024), idesc_o,
                     (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&o_done[i & 1]);
        mma_commit(&v_empty[st]);
        last_commit = &o_done[i & 1];
        last_parity = (i >> 1) & 1;
      }
      if (!ok && last_commit) drain_wait(last_commit, last_parity, 100000000ull);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax
    // two warpgroups; thread (r, w) owns row r and key columns [64w, 64w+64)
    // of every tile.  Per tile the two post their partial row maxima and
    // take the same reference max; each keeps its own partial row sum and
    // writes its half of P (fp16 pairs) over the first 32 columns of the S
    // columns it read, so neither overwrites what the other still reads.
    const int r = (threadIdx.x - 128) & 127;
    const int w = (threadIdx.x - 128) >> 7;
    const int cw = 64 * w;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int lg = 31 - __clz(g);
    const int pos = r >> lg, h = r & (g - 1);
    const int qabs = s_qpos[pos], lo_r = s_lo[pos];
    const float sl2 = p.scale_log2;
    // row maxima / sums exchange in the Q buffer, free once Q is in TMEM
    float* xmax = reinterpret_cast<float*>(sQ);        // [2 tiles][2 warpgroups][128]
    float* xsum = xmax + 2 * 2 * 128;                  // [2 warpgroups][128]
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t e_next = n > 0 ? static_cast<uint32_t>(list[0]) : 0u;
    bool ok = true;
    if (n > 0 && w == 0) {  // row r of Q into TMEM (bf16 pairs), the A operand of Q K^T
      if (!__all_sync(0xffffffffu, mbar_wait(q_full, 0, ctl))) {
        ok = false;
      } else {
        sw128_row_to_tmem<D>(smem_u32(sQ), r, tmem + lane_base + Cfg::kTmemQ);
        tmem_wait_st();
        warp_arrive(q_tmem);
      }
    }
    for (int j = 0; ok && j < n; ++j) {
      const int sb = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[sb], (j >> 1) & 1, ctl))) {
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
      if (j + 1 < n) e_next = static_cast<uint32_t>(list[j + 1]);
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
      if (!__all_sync(0xffffffffu, mbar_wait(&mx_ready[sb], (j >> 1) & 1, ctl))) {
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
      float sum0 = 0.f, sum1 = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float e0 = ex2(fmaf(s[c], sl2, -m_ref));
        const float e1 = ex2(fmaf(s[c + 1], sl2, -m_ref));
        sum0 += e0;
        sum1 += e1;
        pk[c >> 1] = pack_f16(e0, e1);
      }
      l_run = l_run * alpha + (sum0 + sum1);
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_st8_nowait(sc + 8 * q, pk + 8 * q);
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // the reference max moved: rescale this warpgroup's half of O once
        // P_{j-1} V_{j-1} is in
        if (!__all_sync(0xffffffffu, mbar_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, ctl))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
          float t[32];
          const uint32_t oc = tmem + lane_base + Cfg::kTmemO + w * (D / 2) + c0;
          tmem_ld32(oc, t);
#pragma unroll
          for (int i = 0; i < 32; ++i) t[i] *= alpha;
          tmem_st32(oc, t);
        }
      }
      tmem_wait_st();
      warp_arrive(&p_full[sb]);
      m_run = m_new;
    }
    if (ok && n > 0) {
      xsum[w * 128 + r] = l_run;
      __syncwarp();
      if (lane == 0) mbar_arrive(l_ready);
      ok = __all_sync(0xffffffffu, mbar_wait(l_ready, 0, ctl));
    }
    if (ok && n > 0 && __all_sync(0xffffffffu, mbar_wait(&o_done[(n - 1) & 1], ((n - 1) >> 1) & 1, ctl))) {
      tc_fence_after();
      const float l_tot = xsum[r] + xsum[128 + r];
      const float inv = 1.f / l_tot;
      const int hq = kvh * g + h;
      const long long row = static_cast<long long>(b) * Lq + l0 + pos;
      float4* dst = reinterpret_cast<float4*>(o + (row * p.n_heads + hq) * D + w * (D / 2));
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        float t[32];
        tmem_ld32(tmem + lane_base + Cfg::kTmemO + w * (D / 2) + c0, t);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          dst[c0 / 4 + q4] = make_float4(t[4 * q4] * inv, t[4 * q4 + 1] * inv,
                                         t[4 * q4 + 2] * inv, t[4 * q4 + 3] * inv);
      }
      if (w == 0)
        lse[(static_cast<long long>(b) * p.n_heads + hq) * Lq + l0 + pos] =
            (m_run + lg2(l_tot)) * 0.6931471805599453f;
    }
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
                         const CUtensorMap& tv16, float* o, float* lse, cudaStream_t s) {
  const PlanDev& p = pl.d;
  const int grid = p.batch * p.n_qtiles * p.n_kv_heads;
  if (grid == 0) return cudaSuccess;
  const int smem = FwdCfg<D>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  fwd_kernel<D><<<grid, 384, smem, s>>>(tq, tk, tv16, p, o, lse);
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
                       const CUtensorMap& tv16, float* o, float* lse, cudaStream_t s) {
  if (pl.d.head_dim == 128) return launch_fwd_d<128>(pl, tq, tk, tv16, o, lse, s);
  return launch_fwd_d<64>(pl, tq, tk, tv16, o, lse, s);
}

}  // namespace dma
