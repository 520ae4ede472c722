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
// One CTA per 128-query tile of one (batch, head), 256 threads:
//   warps 0, 2 (one thread each)  TMA producers: warp 0 loads the Q tile once and then
//                        K tiles (128 keys) through a 2-stage ring, warp 2 the V tiles
//                        through their own 2-stage ring.  K_i is released as soon as
//                        S_i has read it, V_i only after PV_i, so the K loads run well
//                        ahead.  A 4-D tensor map over [B, S, H, D] zero-fills keys and
//                        queries past the sequence end.
//   warp 1 (one thread)  MMA issuer: S_i = Q K_i^T into Tensor Memory (two S buffers,
//                        so S_{i+1} is computed while the softmax works on S_i), then
//                        O += P_i V_i into the Tensor Memory accumulator O.  Warp 1
//                        also owns the Tensor Memory allocation.
//   warps 4-7            softmax: thread r owns query row r (its Tensor Memory lane).
//                        It loads S_i's row, masks, updates the running max m and sum
//                        l, rescales its row of O in Tensor Memory when m grew (after
//                        PV_{i-1} has landed), writes P_i = exp2(S_i - m) as 16-bit
//                        pairs back over its row of S_i in Tensor Memory, where the PV
//                        MMA takes it as its A operand, and hands it to the MMA thread.
//                        At the end it divides O by l and stores the row.
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
  kSiteAttnSEmpty = 24,
  kSiteAttnPFull = 25,
  kSiteAttnSFull = 26,
  kSiteAttnPvDone = 27,
  kSiteAttnDrain = 28,
};

struct AttnParams {
  int32_t B, S, H;
  int32_t causal;
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

__host__ __device__ constexpr uint32_t attn_barrier_bytes() { return 8u * 20u + 32u; }

template <int D>
__host__ __device__ constexpr uint32_t attn_smem_bytes() {
  // +1024 alignment slack; Q; 2 stages of K and of V; barriers
  return 1024u + attn_tile_bytes<D>() * 5u + attn_barrier_bytes();
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
                        const __grid_constant__ CUtensorMap tmap_v, const AttnParams p) {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  constexpr int kChunks = D / 64;                 // 128-byte chunks of a row
  constexpr uint32_t kTile = attn_tile_bytes<D>();
  constexpr uint32_t kChunkBytes = 128u * 128u;   // one 64-element chunk of 128 rows
  constexpr uint32_t kTmemCols = 512;             // S[2] at 0, 128; O at 256

  grid_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sK = sQ + kTile;                 // K of stage s at sK + s * kTile
  const uint32_t sV = sK + 2 * kTile;             // V of stage s at sV + s * kTile
  const uint32_t sBar = sQ + 5 * kTile;
  auto k_full = [&](int s) { return sBar + 8u * s; };
  auto k_empty = [&](int s) { return sBar + 8u * (2 + s); };
  auto v_full = [&](int s) { return sBar + 8u * (14 + s); };
  auto v_empty = [&](int s) { return sBar + 8u * (16 + s); };
  auto s_full = [&](int s) { return sBar + 8u * (4 + s); };
  const uint32_t q_full = sBar + 8u * 8;
  const uint32_t done_bar = sBar + 8u * 11;
  auto p_full = [&](int t) { return sBar + 8u * (12 + t); };    // P written in S buffer t
  auto pv_done = [&](int t) { return sBar + 8u * (18 + t); };   // PV from S buffer t done
  const uint32_t slot = sBar + 8u * 20;
  volatile uint32_t* const tmem_slot_ptr =
      reinterpret_cast<volatile uint32_t*>(base_ptr + (slot - base));
  volatile uint32_t* const abort_flag = tmem_slot_ptr + 1;
  volatile int32_t* const lap_k = reinterpret_cast<volatile int32_t*>(tmem_slot_ptr + 2);  // [2]
  volatile int32_t* const lap_v = lap_k + 2;                                                 // [2]
  volatile int32_t* const q_armed = lap_v + 2;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_q_tiles = static_cast<int>(gridDim.x);
  const int qt = n_q_tiles - 1 - static_cast<int>(blockIdx.x);   // longest causal tiles first
  const int h = static_cast<int>(blockIdx.y);
  const int b = static_cast<int>(blockIdx.z);
  const int q0 = qt * kAttnBM;
  const int kv_end = p.causal ? min(p.S, q0 + kAttnBM) : p.S;
  const int n_kv = (kv_end + kAttnBN - 1) / kAttnBN;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
      mbar_init(s_full(s), 1);
    }
    mbar_init(q_full, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(p_full(t), 4);
      mbar_init(pv_done(t), 1);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0u;
    lap_k[0] = lap_k[1] = lap_v[0] = lap_v[1] = -1;
    *q_armed = 0;
    fence_barrier_init();
  }
  if (threadIdx.x == 64) {
    tma_prefetch_map(&tmap_q);
    tma_prefetch_map(&tmap_k);
    tma_prefetch_map(&tmap_v);
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
      if (is_k) {
        mbar_arrive_expect_tx(q_full, kTile);
        for (int c = 0; c < kChunks; ++c)
          tma_load_4d(sQ + c * kChunkBytes, &tmap_q, q_full, 64 * c, h, q0, b);
        *q_armed = 1;
      }
      for (int i = 0; i < n_kv; ++i) {
        const int st = i & 1;
        const uint32_t ph = static_cast<uint32_t>(i >> 1) & 1u;
        const uint32_t empty = is_k ? k_empty(st) : v_empty(st);
        const uint32_t full = is_k ? k_full(st) : v_full(st);
        if (!wait_bounded<false>(empty, ph ^ 1u, abort_flag, p.timeout_ns)) {
          record_timeout(p.status, abort_flag, kSiteAttnKvEmpty);
          break;
        }
        mbar_arrive_expect_tx(full, kTile);
        const uint32_t dst = (is_k ? sK : sV) + st * kTile;
        for (int c = 0; c < kChunks; ++c)
          tma_load_4d(dst + c * kChunkBytes, is_k ? &tmap_k : &tmap_v, full, 64 * c, h,
                      i * kAttnBN, b);
        (is_k ? lap_k : lap_v)[st] = i >> 1;
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer --
    grid_dependency_wait();
    if (lane == 0) {
      const uint64_t q_desc = smem_desc_sw128(sQ, 16u, 1024u);
      // K-major step k (16 elements): chunk k/4, then 32 B along the swizzled row
      auto kmaj = [](int k) -> uint64_t {
        return (static_cast<uint64_t>(k / 4) * kChunkBytes + (k % 4) * 32u) >> 4;
      };
      bool ok = wait_bounded<false>(q_full, 0, abort_flag, p.timeout_ns);
      if (!ok) record_timeout(p.status, abort_flag, kSiteAttnQFull);
      for (int i = 0; ok && i <= n_kv; ++i) {
        if (i < n_kv) {
          const int st = i & 1;
          const uint32_t ph = static_cast<uint32_t>(i >> 1) & 1u;
          if (!wait_bounded<false>(k_full(st), ph, abort_flag, p.timeout_ns)) {
            record_timeout(p.status, abort_flag, kSiteAttnKvFull);
            break;
          }
          // S buffer st last held P_{i-2}; PV_{i-2}, issued before this point by this
          // thread, reads it before these MMAs overwrite it (tcgen05 operations of one
          // thread execute in order), so no wait is needed
          tc_fence_after_sync();
          const uint64_t k_desc = smem_desc_sw128(sK + st * kTile, 16u, 1024u);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            mma_f16_ss(tmem_base + st * 128u, q_desc + kmaj(k), k_desc + kmaj(k), p.idesc_s,
                       k > 0 ? 1u : 0u);
          }
          mma_commit(s_full(st));
          mma_commit(k_empty(st));        // K_i is read once S_i has completed
        }
        if (i >= 1) {
          const int j = i - 1;
          const int st = j & 1;                       // V stage and P buffer of tile j
          if (!wait_bounded<false>(p_full(st), static_cast<uint32_t>(j >> 1) & 1u, abort_flag,
                                   p.timeout_ns)) {
            record_timeout(p.status, abort_flag, kSiteAttnPFull);
            break;
          }
          if (!wait_bounded<false>(v_full(st), static_cast<uint32_t>(j >> 1) & 1u, abort_flag,
                                   p.timeout_ns)) {
            record_timeout(p.status, abort_flag, kSiteAttnKvFull);
            break;
          }
          tc_fence_after_sync();
          // V is the N-major B operand: 64-column chunks of 128 key rows (LBO = chunk
          // stride), K step = 16 key rows of 128 B
          const uint64_t v_desc = smem_desc_sw128(sV + st * kTile, kChunkBytes, 1024u);
          // P_j is the A operand in Tensor Memory, over S_j: 16 keys = 8 columns per step
#pragma unroll
          for (int k = 0; k < kAttnBN / 16; ++k) {
            mma_f16_ts(tmem_base + 256u, tmem_base + st * 128u + 8u * k,
                       v_desc + ((static_cast<uint64_t>(k) * 16u * 128u) >> 4), p.idesc_o,
                       (j > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(v_empty(st));
          mma_commit(pv_done(st));
        }
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
    const int qi = q0 + row;                        // its position in the sequence
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(qd * 32) << 16);
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    auto wait_warp = [&](uint32_t bar, uint32_t parity, uint32_t site) -> bool {
      bool r = true;
      if (lane == 0) r = wait_bounded<false>(bar, parity, abort_flag, p.timeout_ns);
      __syncwarp();
      r = __shfl_sync(0xFFFFFFFFu, r ? 1 : 0, 0) != 0;
      if (!r && lane == 0 && !*abort_flag) record_timeout(p.status, abort_flag, site);
      return r;
    };
    for (int i = 0; ok && i < n_kv; ++i) {
      const int st = i & 1;
      if (!(ok = wait_warp(s_full(st), static_cast<uint32_t>(i >> 1) & 1u, kSiteAttnSFull))) break;
      tc_fence_after_sync();
      uint32_t sv[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_load_32cols(lane_base + st * 128u + 32u * c, *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c]));
      tmem_load_wait();
      // keys past the end (and, causal, past qi) are masked
      const int kv0 = i * kAttnBN;
      const int lim = p.causal ? min(p.S - kv0, qi - kv0 + 1) : p.S - kv0;
      // Row maximum with four independent partial maxima, two new scores per step (a
      // single running maximum would be a long dependency chain); masking only on the
      // tiles that need it.
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
      // keep the stale maximum unless the row's maximum grew by more than the threshold
      // (a row that has seen no key yet, m = -inf, takes the new one)
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
      // P_i (16-bit pairs, keys 2c and 2c+1 in column c) over this row's S_i in Tensor
      // Memory, where the PV MMA reads it as its A operand
      tmem_store_32cols(lane_base + st * 128u, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_store_32cols(lane_base + st * 128u + 32u, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      const float2 rs2 = add2(add2(rsp[0], rsp[1]), add2(rsp[2], rsp[3]));
      const float rs = rs2.x + rs2.y;
      l = l * corr + rs;
      m = m_use;
      if (i > 0 && __any_sync(0xFFFFFFFFu, corr != 1.0f)) {
        // rescaling O needs PV_{i-1} to have landed in it (PV_i, which reads this P,
        // waits for the p_full arrival below)
        const int jp = i - 1;
        if (!(ok = wait_warp(pv_done(jp & 1), static_cast<uint32_t>(jp >> 1) & 1u,
                             kSiteAttnPvDone))) {
          break;
        }
        tc_fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_load_32cols(lane_base + 256u + 32u * c, ov);
          tmem_load_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * corr);
          tmem_store_32cols(lane_base + 256u + 32u * c, ov);
        }
        tmem_store_wait();
      }
      tmem_store_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(st));
    }
    if (ok && n_kv > 0 &&
        wait_warp(pv_done((n_kv - 1) & 1), static_cast<uint32_t>((n_kv - 1) >> 1) & 1u,
                  kSiteAttnPvDone)) {
      tc_fence_after_sync();
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      uint16_t* orow = reinterpret_cast<uint16_t*>(p.O) +
                       ((static_cast<int64_t>(b) * p.S + qi) * p.H + h) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_load_32cols(lane_base + 256u + 32u * c, ov);
        tmem_load_wait();
        if (qi < p.S) {
          uint32_t o2[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            o2[j] = pack_half2<kBf16>(__uint_as_float(ov[2 * j]) * inv,
                                      __uint_as_float(ov[2 * j + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = make_uint4(o2[4 * j], o2[4 * j + 1], o2[4 * j + 2], o2[4 * j + 3]);
        }
      }
    }
  }

  // ------------------------------------------------------------------ teardown --
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0) {
    // every load issued must have landed before the CTA exits
    if (*q_armed && !wait_bounded<false>(q_full, 0, nullptr, p.timeout_ns))
      record_timeout(p.status, abort_flag, kSiteAttnDrain);
    for (int st = 0; st < 2; ++st) {
      const int lk = lap_k[st], lv = lap_v[st];
      if (lk >= 0 && !wait_bounded<false>(k_full(st), static_cast<uint32_t>(lk) & 1u, nullptr,
                                          p.timeout_ns)) {
        record_timeout(p.status, abort_flag, kSiteAttnDrain);
      }
      if (lv >= 0 && !wait_bounded<false>(v_full(st), static_cast<uint32_t>(lv) & 1u, nullptr,
                                          p.timeout_ns)) {
        record_timeout(p.status, abort_flag, kSiteAttnDrain);
      }
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
