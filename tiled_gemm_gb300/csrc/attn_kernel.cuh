// attn_kernel.cuh -- FlashAttention forward pass on the GEMM's sm_103a primitives.
//
// O = softmax(Q K^T / sqrt(D)) V for every (batch, head), Q, K, V and O laid out
// [B, S, H, D] with fp16/bf16 elements, optionally causal (query i sees keys j <= i).
// The pages give this as their second workload on the same tile primitives
// ("TileLang: a tile language one level below Triton", section "FlashAttention:
// online softmax as tile code"): each block owns a tile of queries, walks the keys
// in tiles, keeps a running row maximum and row sum, rescales the output
// accumulator whenever the maximum grows, works with exp2 on scores pre-multiplied
// by log2(e), and divides by the row sum once at the end; the causal form skips key
// tiles wholly above the diagonal and masks the diagonal tile.
//
// Work unit: one 128-query tile of one (batch, head).  The grid is persistent (at most
// one CTA per SM, 256 threads), and every CTA walks its own fixed list of units, so the
// loads and first products of a unit overlap the end of the one before:
//   * CTA c takes work items c, c + G, c + 2G, ... (G CTAs).  An item is one unit, the
//     query tiles of a head in turn (consecutive items share K and V, which the CTAs
//     running side by side then read from L2), longest causal tile first;
//   * causal with more units than SMs: an item is the pair of query tiles (n-1-k, k)
//     of one head, n + 1 key tiles in all for every item, so the static split is even.
// Roles:
//   warps 0, 2 (one thread each)  TMA producers: warp 0 loads each unit's Q tile (two
//                        Q buffers, so the next unit's is in flight early) and the K
//                        tiles (128 keys) through a 2-stage ring, warp 2 the V tiles
//                        through their own 2-stage ring; the rings run on across units.
//                        K_i is released as soon as S_i has read it, V_i only after
//                        PV_i, so the K loads run well ahead.  A 4-D tensor map over
//                        [B, S, H, D] zero-fills keys and queries past the sequence end.
//   warp 1 (one thread)  MMA issuer: S_i = Q K_i^T into Tensor Memory (two S buffers,
//                        so S_{i+1} is computed while the softmax works on S_i), then
//                        O += P_i V_i into the Tensor Memory accumulator O.  The next
//                        unit's S_0 goes in before the last PV of the current one.  Warp
//                        1 also owns the Tensor Memory allocation.
//   warps 4-7            softmax: thread r owns query row r (its Tensor Memory lane).
//                        It loads S_i's row, masks, updates the running max m and sum
//                        l, rescales its row of O in Tensor Memory when m grew (after
//                        PV_{i-1} has landed), writes P_i = exp2(S_i - m) as 16-bit
//                        pairs back over its row of S_i in Tensor Memory, where the PV
//                        MMA takes it as its A operand, and hands it to the MMA thread.
//                        At the end of a unit it divides O by l and stores the row; the
//                        next unit's first PV, which overwrites O, waits for its P_0,
//                        which these warps write only after that.
//   warp 3               idle.
//
// Every wait is bounded as in the GEMM kernel; on a timeout the status word records
// the site and every role unwinds.
#pragma once

#include "gemm_kernel.cuh"

namespace tl {

constexpr int kAttnBM = 128;        // queries per CTA (Tensor Memory lanes)
constexpr int kAttnBN = 128;        // keys per tile
constexpr int kAttnThreads = 256;

enum AttnWaitSite : uint32_t {
  kSiteAttnKvEmpty = 21,
  kSiteAttnQFull = 22,
  kSiteAttnKvFull = 23,
  kSiteAttnQEmpty = 24,
  kSiteAttnPFull = 25,
  kSiteAttnSFull = 26,
  kSiteAttnPvDone = 27,
  kSiteAttnDrain = 28,
};

struct AttnParams {
  int32_t B, S, H;
  int32_t causal;
  int32_t n_q_tiles;            // ceil(S / 128)
  int32_t items_per_head;       // n_q_tiles, or ceil(n_q_tiles / 2) with pairing
  int32_t n_items;              // B * H * items_per_head
  int32_t pair;                 // an item is the query tiles (n-1-k, k) of a head
  float scale_log2;             // log2(e) / sqrt(D)
  void* O;
  uint32_t idesc_s;             // S = Q K^T: M 128, N 128, both K-major
  uint32_t idesc_o;             // O += P V: M 128, N D, P K-major, V N-major
  uint32_t* status;
  uint64_t timeout_ns;
};

template <int D>
__host__ __device__ constexpr uint32_t attn_tile_bytes() {      // 128 rows x D, 2 bytes
  return 128u * D * 2u;
}

// Tensor Memory: three S buffers of 128 columns (the MMA thread issues S_g before PV_{g-2},
// so S_g must not land on P_{g-2}), then the O accumulator at column 384.
constexpr int kAttnSBufs = 3;
constexpr uint32_t kAttnOCol = 128u * kAttnSBufs;

// Barriers: K full and V full per stage (2), q_full and q_empty per Q buffer (2),
// s_full, p_full and pv_done per S buffer (3), done.  Then the Tensor Memory slot, the
// abort flag and the laps of the last load into each K, V and Q buffer.
__host__ __device__ constexpr uint32_t attn_barrier_bytes() {
  return 8u * (4u + 4u + 3u * kAttnSBufs + 1u) + 4u * 8u;
}

template <int D>
__host__ __device__ constexpr uint32_t attn_smem_bytes() {
  // +1024 alignment slack; 2 Q buffers; 2 stages of K and of V; the O staging tile;
  // barriers
  return 1024u + attn_tile_bytes<D>() * 7u + attn_barrier_bytes();
}

// 2^x by the special-function unit's approximation (relative error ~2^-22, enough
// for probabilities that are rounded to 16 bits); 2^-inf = +0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The running maximum is only moved (and O rescaled) when a row's new maximum exceeds
// it by more than this many doublings: probabilities computed against a stale
// maximum then stay below 2^8, exact enough in fp32 and well inside the 16-bit range
// of P, and the final division by the row sum cancels the common factor.
constexpr float kRescaleThreshold = 8.0f;

template <bool kBf16>
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  if constexpr (kBf16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  } else {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
}

// The softmax is bound by instruction issue (one warp per scheduler), so its
// arithmetic uses packed fp32 pairs (one f32x2 instruction does two scores' worth)
// and a three-input maximum (two new scores per step).
__device__ __forceinline__ uint64_t pair_bits(float2 a) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
  return r;
}
__device__ __forceinline__ float2 pair_of(uint64_t r) {
  float2 a;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
  return a;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pair_bits(a)), "l"(pair_bits(b)), "l"(pair_bits(c)));
  return pair_of(d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pair_bits(a)), "l"(pair_bits(b)));
  return pair_of(d);
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <int D, bool kBf16>
__global__ void __launch_bounds__(kAttnThreads, 1)
    tl_attention_kernel(const __grid_constant__ CUtensorMap tmap_q,
                        const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __grid_constant__ CUtensorMap tmap_o, const AttnParams p) {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  constexpr int kChunks = D / 64;                 // 128-byte chunks of a row
  constexpr uint32_t kTile = attn_tile_bytes<D>();
  constexpr uint32_t kChunkBytes = 128u * 128u;   // one 64-element chunk of 128 rows
  constexpr uint32_t kTmemCols = 512;             // S[3] at 0, 128, 256; O at 384
  static_assert(kAttnOCol + D <= kTmemCols, "S buffers and O fit in Tensor Memory");

  grid_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t sQ = base;                       // Q buffer t at sQ + t * kTile
  const uint32_t sK = sQ + 2 * kTile;             // K of stage s at sK + s * kTile
  const uint32_t sV = sK + 2 * kTile;             // V of stage s at sV + s * kTile
  const uint32_t sStage = sV + 2 * kTile;         // O of 128 rows on its way out
  const uint32_t sBar = sStage + kTile;
  // Key tile g (counted over all of this CTA's units) uses K and V stage g & 1 and S
  // buffer g % 3.  The stages are released by the barriers that mark the products
  // reading them: K_g by s_full (S_g done), V_g by pv_done (PV_g done).  A producer
  // reusing a stage for tile g waits for tile g - 2's completion there; the next
  // completion on that S buffer's barrier is tile g + 1's, which needs a load the
  // producer has not issued yet, so its parity wait cannot see a later phase.
  auto k_full = [&](int s) { return sBar + 8u * s; };
  auto v_full = [&](int s) { return sBar + 8u * (2 + s); };
  auto q_full = [&](int t) { return sBar + 8u * (4 + t); };
  auto q_empty = [&](int t) { return sBar + 8u * (6 + t); };
  auto s_full = [&](int b) { return sBar + 8u * (8 + b); };                   // S_g computed
  auto p_full = [&](int b) { return sBar + 8u * (8 + kAttnSBufs + b); };      // P_g over S_g
  auto pv_done = [&](int b) { return sBar + 8u * (8 + 2 * kAttnSBufs + b); }; // PV_g done
  const uint32_t done_bar = sBar + 8u * (8 + 3 * kAttnSBufs);
  const uint32_t slot = done_bar + 8u;
  volatile uint32_t* const tmem_slot_ptr =
      reinterpret_cast<volatile uint32_t*>(base_ptr + (slot - base));
  volatile uint32_t* const abort_flag = tmem_slot_ptr + 1;
  // laps of the last load issued into each K, V and Q buffer (-1: none), for the drain
  volatile int32_t* const lap_k = reinterpret_cast<volatile int32_t*>(tmem_slot_ptr + 2);  // [2]
  volatile int32_t* const lap_v = lap_k + 2;                                                 // [2]
  volatile int32_t* const lap_q = lap_v + 2;                                                 // [2]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // This CTA's units in order: f(q-tile, head, batch) returns false to stop early.
  auto for_each_unit = [&](auto&& f) {
    for (int w = static_cast<int>(blockIdx.x); w < p.n_items; w += static_cast<int>(gridDim.x)) {
      const int hb = w / p.items_per_head;
      const int k = w - hb * p.items_per_head;
      const int h = hb % p.H, b = hb / p.H;
      const int hi = p.n_q_tiles - 1 - k;
      if (!f(hi, h, b)) return;
      if (p.pair && k != hi && !f(k, h, b)) return;
    }
  };
  auto kv_tiles = [&](int qt) {
    const int kv_end = p.causal ? min(p.S, (qt + 1) * kAttnBM) : p.S;
    return (kv_end + kAttnBN - 1) / kAttnBN;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(v_full(s), 1);
      lap_k[s] = lap_v[s] = -1;
      mbar_init(q_full(s), 1);
      mbar_init(q_empty(s), 1);
    }
    for (int b = 0; b < kAttnSBufs; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(p_full(b), 4);
      mbar_init(pv_done(b), 1);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0u;
    lap_q[0] = lap_q[1] = -1;
    fence_barrier_init();
  }
  if (threadIdx.x == 64) {
    tma_prefetch_map(&tmap_q);
    tma_prefetch_map(&tmap_k);
    tma_prefetch_map(&tmap_v);
    tma_prefetch_map(&tmap_o);
  }
  if (warp == 1) {
    tmem_alloc(slot, kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot_ptr;

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ producers --
    if (lane == 0) {
      grid_dependency_wait();
      const bool is_k = warp == 0;
      int g = 0;                                  // key tiles loaded so far (all units)
      int u = 0;                                  // units so far
      for_each_unit([&](int qt, int h, int b) -> bool {
        if (is_k) {
          const int qb = u & 1;
          if (!wait_bounded<false>(q_empty(qb), (static_cast<uint32_t>(u >> 1) & 1u) ^ 1u,
                                   abort_flag, p.timeout_ns)) {
            record_timeout(p.status, abort_flag, kSiteAttnQEmpty);
            return false;
          }
          mbar_arrive_expect_tx(q_full(qb), kTile);
          for (int c = 0; c < kChunks; ++c)
            tma_load_4d(sQ + qb * kTile + c * kChunkBytes, &tmap_q, q_full(qb), 64 * c, h,
                        qt * kAttnBM, b);
          lap_q[qb] = u >> 1;
        }
        ++u;
        const int n_kv = kv_tiles(qt);
        for (int i = 0; i < n_kv; ++i, ++g) {
          const int st = g & 1;
          const int lap = g >> 1;
          if (g >= 2) {
            // stage st last held tile g - 2: wait for the product that read it
            const int b = (g - 2) % kAttnSBufs;
            const uint32_t ph = static_cast<uint32_t>((g - 2) / kAttnSBufs) & 1u;
            if (!wait_bounded<false>(is_k ? s_full(b) : pv_done(b), ph, abort_flag,
                                     p.timeout_ns)) {
              record_timeout(p.status, abort_flag, kSiteAttnKvEmpty);
              return false;
            }
          }
          const uint32_t full = is_k ? k_full(st) : v_full(st);
          mbar_arrive_expect_tx(full, kTile);
          const uint32_t dst = (is_k ? sK : sV) + st * kTile;
          for (int c = 0; c < kChunks; ++c)
            tma_load_4d(dst + c * kChunkBytes, is_k ? &tmap_k : &tmap_v, full, 64 * c, h,
                        i * kAttnBN, b);
          (is_k ? lap_k : lap_v)[st] = lap;
        }
        return true;
      });
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer --
    grid_dependency_wait();
    if (lane == 0) {
      // K-major step k (16 elements): chunk k/4, then 32 B along the swizzled row
      auto kmaj = [](int k) -> uint64_t {
        return (static_cast<uint64_t>(k / 4) * kChunkBytes + (k % 4) * 32u) >> 4;
      };
      // Descriptors of buffer 0; buffer t is kTile further on (the start address field
      // holds address / 16 in 14 bits, and every buffer lies below 256 KB, so adding
      // t * kTile / 16 cannot carry out of it).  V is the N-major B operand: 64-column
      // chunks of 128 key rows (LBO = chunk stride), K step = 16 key rows of 128 B.
      const uint64_t q_desc0 = smem_desc_sw128(sQ, 16u, 1024u);
      const uint64_t k_desc0 = smem_desc_sw128(sK, 16u, 1024u);
      const uint64_t v_desc0 = smem_desc_sw128(sV, kChunkBytes, 1024u);
      // This thread's waits sit between batches of MMAs, where every cycle it spends
      // leaves the tensor pipe idle: one non-blocking test first, the bounded wait only
      // when the phase is still open.
      auto wait_fast = [&](uint32_t bar, uint32_t parity, uint32_t site) -> bool {
        if (mbar_test_wait(bar, parity)) return true;
        if (wait_bounded<false>(bar, parity, abort_flag, p.timeout_ns)) return true;
        record_timeout(p.status, abort_flag, site);
        return false;
      };
      // O += P_j V_j for a key tile j (all units' tiles counted together) in S buffer b
      // (phase ph there); `first`: the unit's first tile, whose product overwrites O
      struct Pending {
        int j, b;
        uint32_t ph;
        bool first;
      };
      auto pv_wait = [&](const Pending& t) -> bool {
        return wait_fast(p_full(t.b), t.ph, kSiteAttnPFull) &&
               wait_fast(v_full(t.j & 1), static_cast<uint32_t>(t.j >> 1) & 1u, kSiteAttnKvFull);
      };
      auto pv_issue = [&](const Pending& t) {
        const int vs = t.j & 1;                     // V stage of tile j
        const uint64_t v_desc = v_desc0 + static_cast<uint64_t>(vs) * (kTile >> 4);
        // P_j is the A operand in Tensor Memory, over S_j: 16 keys = 8 columns per step
#pragma unroll
        for (int k = 0; k < kAttnBN / 16; ++k) {
          mma_f16_ts(tmem_base + kAttnOCol, tmem_base + t.b * 128u + 8u * k,
                     v_desc + ((static_cast<uint64_t>(k) * 16u * 128u) >> 4), p.idesc_o,
                     (!t.first || k > 0) ? 1u : 0u);
        }
        mma_commit(pv_done(t.b));         // also releases V stage vs
      };
      // One batch per key tile: S_g, then PV_{g-2}.  With PV two tiles behind, P_{g-2} is
      // normally ready by the time K_g is, and the softmax, busy with tile g - 1, needs
      // S_g only a softmax later.  The batch's barriers are tested together and waited
      // on only if one is still open: every cycle this thread spends between batches
      // leaves the tensor pipe idle.
      int g = 0, u = 0;
      int sb = 0;                                  // S buffer of tile g
      uint32_t sph = 0;                            // its phase
      Pending pend0{}, pend1{};                    // PVs still to issue, oldest first
      int n_pend = 0;
      bool ok = true;
      for_each_unit([&](int qt, int, int) -> bool {
        const int qb = u & 1;
        if (!wait_fast(q_full(qb), static_cast<uint32_t>(u >> 1) & 1u, kSiteAttnQFull))
          return ok = false;
        const uint64_t q_desc = q_desc0 + static_cast<uint64_t>(qb) * (kTile >> 4);
        const int n_kv = kv_tiles(qt);
        for (int i = 0; i < n_kv; ++i, ++g) {
          const int st = g & 1;                     // K stage
          const uint32_t kph = static_cast<uint32_t>(g >> 1) & 1u;
          const bool with_pv = n_pend == 2;
          bool ready = mbar_test_wait(k_full(st), kph);
          if (with_pv)
            ready = mbar_test_wait(p_full(pend0.b), pend0.ph) &&
                    mbar_test_wait(v_full(pend0.j & 1), static_cast<uint32_t>(pend0.j >> 1) & 1u) &&
                    ready;
          if (!ready) {
            if (!wait_fast(k_full(st), kph, kSiteAttnKvFull)) return ok = false;
            if (with_pv && !pv_wait(pend0)) return ok = false;
          }
          // S buffer sb last held P_{g-3}; PV_{g-3}, issued before this point by this
          // thread, reads it before these MMAs overwrite it (tcgen05 operations of one
          // thread execute in order), so no wait is needed
          tc_fence_after_sync();
          const uint64_t k_desc = k_desc0 + static_cast<uint64_t>(st) * (kTile >> 4);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            mma_f16_ss(tmem_base + sb * 128u, q_desc + kmaj(k), k_desc + kmaj(k), p.idesc_s,
                       k > 0 ? 1u : 0u);
          }
          mma_commit(s_full(sb));           // also releases K stage st
          if (i == n_kv - 1) mma_commit(q_empty(qb));
          const Pending cur{g, sb, sph, i == 0};
          if (with_pv) {
            pv_issue(pend0);
            pend0 = pend1;
            pend1 = cur;
          } else if (n_pend == 1) {
            pend1 = cur;
            n_pend = 2;
          } else {
            pend0 = cur;
            n_pend = 1;
          }
          if (++sb == kAttnSBufs) {
            sb = 0;
            sph ^= 1u;
          }
        }
        ++u;
        return true;
      });
      if (ok && n_pend >= 1 && (ok = pv_wait(pend0))) {
        tc_fence_after_sync();
        pv_issue(pend0);
      }
      if (ok && n_pend == 2 && (ok = pv_wait(pend1))) {
        tc_fence_after_sync();
        pv_issue(pend1);
      }
      mma_commit(done_bar);
      if (!wait_bounded<false>(done_bar, 0, nullptr, p.timeout_ns))
        record_timeout(p.status, abort_flag, kSiteAttnDrain);
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- softmax --
    grid_dependency_wait();
    const int qd = warp & 3;                        // Tensor Memory lane quadrant
    const int row = qd * 32 + lane;                 // this thread's query row in the tile
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(qd * 32) << 16);
    // This warp's 32 rows of the O staging tile: 64-column chunks of 32 rows x 128 B, the
    // 16-byte units of a row XOR-swizzled by the row (the TMA store's 128-byte swizzle;
    // the tile is 1024-byte aligned)
    const uint32_t stage_w = sStage + static_cast<uint32_t>(qd) * (kTile / 4u);
    auto wait_warp = [&](uint32_t bar, uint32_t parity, uint32_t site) -> bool {
      bool r = true;
      if (lane == 0) r = wait_bounded<false>(bar, parity, abort_flag, p.timeout_ns);
      __syncwarp();
      r = __shfl_sync(0xFFFFFFFFu, r ? 1 : 0, 0) != 0;
      if (!r && lane == 0 && !*abort_flag) record_timeout(p.status, abort_flag, site);
      return r;
    };
    bool in_flight = false;                         // a TMA store may still read the staging
    // O / l of a finished unit, whose last PV is the one from S buffer ob (phase oph),
    // into this warp's staging rows
    auto stage_o = [&](int ob, uint32_t oph, float lsum) -> bool {
      if (!wait_warp(pv_done(ob), oph, kSiteAttnPvDone)) return false;
      tc_fence_after_sync();
      if (in_flight) {
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
      }
      const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_load_32cols(lane_base + kAttnOCol + 32u * c, ov);
        tmem_load_wait();
        uint32_t o2[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          o2[j] = pack_half2<kBf16>(__uint_as_float(ov[2 * j]) * inv,
                                    __uint_as_float(ov[2 * j + 1]) * inv);
        const uint32_t chunk = stage_w + static_cast<uint32_t>(c >> 1) * 4096u + lane * 128u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t unit = static_cast<uint32_t>((c & 1) * 4 + j) ^ (lane & 7u);
          st_shared_v4(chunk + unit * 16u, o2[4 * j], o2[4 * j + 1], o2[4 * j + 2], o2[4 * j + 3]);
        }
      }
      return true;
    };
    // the staged rows to O: rows past the sequence end are clipped by the tensor map
    auto store_o = [&](int qt, int h, int b) {
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        for (int c = 0; c < kChunks; ++c)
          tma_store_4d(&tmap_o, stage_w + static_cast<uint32_t>(c) * 4096u, 64 * c, h,
                       qt * kAttnBM + qd * 32, b);
        bulk_commit_group();
      }
      in_flight = true;
    };
    int sb = 0;                                     // S buffer of the current key tile
    uint32_t sph = 0;                               // its phase
    int pb = 0;                                     // S buffer of the previous key tile
    uint32_t pph = 0;                               // its phase
    // the previous unit, whose O goes out once this unit's first P is ready (its first
    // PV overwrites O, so that P is handed over only after O has been read)
    bool have_prev = false;
    float l_prev = 0.0f;
    int qt_prev = 0, h_prev = 0, b_prev = 0;
    const bool all_ok = [&] {
      bool done = true;
      for_each_unit([&](int qt, int h, int b) -> bool {
        const int qi = qt * kAttnBM + row;          // this thread's query in the sequence
        const int n_kv = kv_tiles(qt);
        float m = -INFINITY, l = 0.0f;
        for (int i = 0; i < n_kv; ++i) {
          const int st = sb;
          if (!wait_warp(s_full(st), sph, kSiteAttnSFull)) return done = false;
          tc_fence_after_sync();
          uint32_t sv[128];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tmem_load_32cols(lane_base + st * 128u + 32u * c,
                             *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c]));
          tmem_load_wait();
          // keys past the end (and, causal, past qi) are masked
          const int kv0 = i * kAttnBN;
          const int lim = p.causal ? min(p.S - kv0, qi - kv0 + 1) : p.S - kv0;
          // Row maximum with four independent partial maxima, two new scores per step (a
          // single running maximum would be a long dependency chain); masking only on
          // the tiles that need it.
          if (lim < 128) {
#pragma unroll
            for (int j = 0; j < 128; ++j)
              if (j >= lim) sv[j] = __float_as_uint(-INFINITY);
          }
          float mxp[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) mxp[t] = -INFINITY;
#pragma unroll
          for (int j = 0; j < 64; ++j)
            mxp[j & 3] = max3(mxp[j & 3], __uint_as_float(sv[2 * j]), __uint_as_float(sv[2 * j + 1]));
          float mx = fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3]));
          mx *= p.scale_log2;
          // keep the stale maximum unless the row's maximum grew by more than the
          // threshold (a row that has seen no key yet, m = -inf, takes the new one)
          const float m_use = (mx > m + kRescaleThreshold) ? mx : m;
          const float corr = (m_use == m) ? 1.0f : fast_exp2(m - m_use);
          float2 rsp[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) rsp[t] = make_float2(0.0f, 0.0f);
          uint32_t pk[64];
          if (m_use == -INFINITY) {
#pragma unroll
            for (int j = 0; j < 64; ++j) pk[j] = 0u;
          } else {
            const float2 sc = make_float2(p.scale_log2, p.scale_log2);
            const float2 nm = make_float2(-m_use, -m_use);
#pragma unroll
            for (int j = 0; j < 64; ++j) {
              const float2 y = fma2(make_float2(__uint_as_float(sv[2 * j]), __uint_as_float(sv[2 * j + 1])),
                                    sc, nm);
              const float2 e = make_float2(fast_exp2(y.x), fast_exp2(y.y));
              rsp[j & 3] = add2(rsp[j & 3], e);
              pk[j] = pack_half2<kBf16>(e.x, e.y);
            }
          }
          // P (16-bit pairs, keys 2c and 2c+1 in column c) over this row's S in Tensor
          // Memory, where the PV MMA reads it as its A operand
          tmem_store_32cols(lane_base + st * 128u, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
          tmem_store_32cols(lane_base + st * 128u + 32u, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
          const float2 rs2 = add2(add2(rsp[0], rsp[1]), add2(rsp[2], rsp[3]));
          l = l * corr + (rs2.x + rs2.y);
          m = m_use;
          if (i > 0 && __any_sync(0xFFFFFFFFu, corr != 1.0f)) {
            // rescaling O needs the previous tile's PV to have landed in it (this tile's
            // PV, which reads this P, waits for the p_full arrival below)
            if (!wait_warp(pv_done(pb), pph, kSiteAttnPvDone)) return done = false;
            tc_fence_after_sync();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t ov[32];
              tmem_load_32cols(lane_base + kAttnOCol + 32u * c, ov);
              tmem_load_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * corr);
              tmem_store_32cols(lane_base + kAttnOCol + 32u * c, ov);
            }
          }
          tmem_store_wait();
          // the previous unit's O is read out of Tensor Memory before this P is handed
          // over (pb is still that unit's last tile)
          const bool flush = i == 0 && have_prev;
          if (flush && !stage_o(pb, pph, l_prev)) return done = false;
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_full(st));
          if (flush) store_o(qt_prev, h_prev, b_prev);
          pb = sb;
          pph = sph;
          if (++sb == kAttnSBufs) {
            sb = 0;
            sph ^= 1u;
          }
        }
        have_prev = true;
        l_prev = l;
        qt_prev = qt;
        h_prev = h;
        b_prev = b;
        return true;
      });
      return done;
    }();
    // the last unit's O
    if (all_ok && have_prev && stage_o(pb, pph, l_prev)) store_o(qt_prev, h_prev, b_prev);
    // the staging must stay valid until the bulk stores have read it; their global
    // writes complete before the grid is reported finished
    if (in_flight && lane == 0) bulk_wait_group_read<0>();
  }

  // ------------------------------------------------------------------ teardown --
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0) {
    // every load issued must have landed before the CTA exits
    auto drain = [&](uint32_t bar, int lap) {
      if (lap >= 0 && !wait_bounded<false>(bar, static_cast<uint32_t>(lap) & 1u, nullptr,
                                           p.timeout_ns)) {
        record_timeout(p.status, abort_flag, kSiteAttnDrain);
      }
    };
    for (int st = 0; st < 2; ++st) {
      drain(k_full(st), lap_k[st]);
      drain(v_full(st), lap_v[st]);
      drain(q_full(st), lap_q[st]);
    }
  }
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace tl
