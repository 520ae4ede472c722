// mx_kernel.cuh -- block-scaled 8-bit GEMM (the MX formats) on tcgen05.
//
// C = epi( sum_k x_a(A[i,k]) 2^(SFA[i][k/32] - 127) * x_b(B[j,k]) 2^(SFB[j][k/32] - 127) )
// with A [M,K] and B [N,K] K-major E4M3/E5M2 codes and one E8M0 scale per 32 K elements
// of every row ("NVIDIA backend codegen" page, section 4.6.3: the Blackwell form of the
// block-scaled MMA, tcgen05 kind::mxf8f6f4.block_scale with the scale factors already
// in Tensor Memory).  fp32 accumulation in Tensor Memory; fp16 or bf16 out.
//
// Tiles of 128 x BN of C (BN = 128 or 256); a persistent grid of at most one CTA per SM,
// each CTA walking tiles blockIdx.x, + gridDim.x, ...; 256 threads:
//   warp 0 (one thread)  TMA producer: a stage is 128 K bytes of A (128 rows) and of B
//                        (128 rows), 128-byte swizzle, S stages in a ring; every
//                        kMxGroup stages also the tile's scale bytes for those stages
//                        (128 rows x 32 bytes of SFA and of SFB, unswizzled, two buffers).
//   warp 1 (one thread)  MMA issuer (and the Tensor Memory allocation): per stage four
//                        128 x BN x 32 block-scaled MMAs, one per 32-element block, the
//                        scale byte of block k selected by the descriptor's scale ids.
//   warps 4-7            scale loaders, then the epilogue.  Only the warp of a lane
//                        quadrant can write its Tensor Memory lanes, so these four warps
//                        copy each stage's scales there from shared memory (tcgen05.st)
//                        ahead of the MMA;
//                        after a tile's last stage they read the accumulator (freeing
//                        it for the next tile, whose loads are already in flight), apply
//                        ReLU, cast and store the tile.
//
// Scale layout in Tensor Memory for M = 128, N = 128 or 256 and one scale per 32
// elements (found with an exact probe: operands of ones, distinct power-of-two
// scales), each 32-bit word holding the scales of the stage's four blocks in its four
// bytes (byte k = the scale id of MMA k):
//   A: row i reads lane i, column sfa + i/32 (four columns);
//   B: column j of the product, for rows in lane quadrant q, reads lane 32q + j%32,
//      column sfb + j/32 (N/32 columns) -- so B's words go into every quadrant.
// The scale addresses stay on the boundaries the probe used (4 columns at N = 128,
// 16 at N = 256): an unaligned one is a misaligned address fault.
#pragma once

#include "gemm_kernel.cuh"

namespace tl {

constexpr int kMxBM = 128;
constexpr int kMxBK = 128;          // K bytes (= elements) per stage: four 32-element blocks
constexpr int kMxStages = 4;
constexpr int kMxGroup = 8;         // stages per TMA load of scale bytes (32 bytes a row)
constexpr int kMxThreads = 256;
constexpr uint32_t kMxEpiBytes = 4u * 32u * 64u;   // one 32 x 32 bf16/fp16 staging tile per epilogue warp

// The sizes of the 128 x BN tile.
template <int BN>
struct MxTile {
  static_assert(BN == 128 || BN == 256, "tile width 128 or 256");
  static constexpr uint32_t kStageBytes = (kMxBM + BN) * kMxBK;        // A + B of a stage
  static constexpr uint32_t kTmemCols = BN == 128 ? 256u : 512u;
  static constexpr uint32_t kSfCol = BN;                 // scales after the accumulator
  static constexpr uint32_t kSfStride = BN == 128 ? 8u : 32u;     // columns per stage
  static constexpr uint32_t kSfB = BN == 128 ? 4u : 16u;          // B's offset in a stage
  static constexpr uint32_t kScaleBytes = 4u * kMxGroup * (kMxBM + BN);   // one buffer
  static_assert(kSfCol + kMxStages * kSfStride <= kTmemCols, "scales fit in Tensor Memory");
};

enum MxWaitSite : uint32_t {
  kSiteMxEmpty = 31,
  kSiteMxFull = 32,
  kSiteMxScales = 33,
  kSiteMxAcc = 34,
  kSiteMxDrain = 35,
};

struct MxParams {
  int32_t M, N, K;
  int32_t k_blocks;           // ceil(K / 128)
  int32_t tiles_n;            // ceil(N / BN)
  int32_t num_tiles;          // ceil(M / 128) * tiles_n
  void* C;
  int64_t ldc;
  int32_t relu;
  int32_t c_vec;              // C and ldc allow 16-byte stores
  uint32_t idesc;             // formats, K-major both, N, M 128, E8M0 scales
  uint32_t* status;
  uint64_t timeout_ns;
};

template <int BN>
__host__ __device__ constexpr uint32_t mx_smem_bytes() {
  // +1024 alignment slack; operand stages; two scale buffers; barriers (full, empty,
  // sf_full per stage, sg_full and sg_empty per scale buffer, acc_full, acc_empty); Tensor Memory
  // slot, abort flag and the laps of the last loads (stages, then scale buffers)
  return 1024u + kMxStages * MxTile<BN>::kStageBytes + 2u * MxTile<BN>::kScaleBytes +
         kMxEpiBytes + 8u * (3 * kMxStages + 6) + 16u + 4u * (kMxStages + 2);
}

// Instruction descriptor of kind::mxf8f6f4 with block scales: B scale id (bits 4-5),
// A and B formats (7-9, 10-12: E4M3 = 0, E5M2 = 1), both K-major (15, 16 = 0), N >> 3
// (17-22), scale format E8M0 (bit 23), M >> 4 (24-28), A scale id (29-30).
__host__ __device__ constexpr uint32_t mma_idesc_mx(uint32_t a_fmt, uint32_t b_fmt, uint32_t m,
                                                    uint32_t n) {
  return (a_fmt << 7) | (b_fmt << 10) | ((n >> 3) << 17) | (1u << 23) | ((m >> 4) << 24);
}
__device__ __forceinline__ uint32_t mx_scale_ids(uint32_t idesc, uint32_t k) {
  return idesc | (k << 4) | (k << 29);
}

__device__ __forceinline__ void mma_mx_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_store_1col(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v)
               : "memory");
}
__device__ __forceinline__ void tmem_store_4cols(uint32_t taddr, uint32_t a, uint32_t b,
                                                 uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// The four scale bytes of stage kb of one row, from the row's 32 bytes of the current
// group in shared memory; rows past the matrix and blocks past K read as 2^0 (their
// operands are zero, and a NaN code there must not reach the sum).
__device__ __forceinline__ uint32_t mx_scale_word(const uint8_t* group_row, int row, int rows,
                                                  int kb, int n_blk) {
  if (row >= rows) return 0x7F7F7F7Fu;
  uint32_t w = *reinterpret_cast<const uint32_t*>(group_row + 4 * (kb % kMxGroup));
  const int valid = n_blk - 4 * kb;
  if (valid < 4) {
    const uint32_t keep = (1u << (8 * valid)) - 1u;
    w = (w & keep) | (0x7F7F7F7Fu & ~keep);
  }
  return w;
}

template <bool kBf16, int BN>
__global__ void __launch_bounds__(kMxThreads, 1)
    tl_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmap_a,
                      const __grid_constant__ CUtensorMap tmap_b,
                      const __grid_constant__ CUtensorMap tmap_sa,
                      const __grid_constant__ CUtensorMap tmap_sb, const MxParams p) {
  using T = MxTile<BN>;
  constexpr int S = kMxStages;
  constexpr uint32_t kA = kMxBM * kMxBK;           // bytes of A per stage
  grid_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t sScale = base + S * T::kStageBytes;     // scale buffer t at + t * T::kScaleBytes
  const uint32_t sEpi = sScale + 2u * T::kScaleBytes;     // epilogue warp q at + 2048 q
  const uint32_t sBar = sEpi + kMxEpiBytes;
  auto full = [&](int s) { return sBar + 8u * s; };
  auto empty = [&](int s) { return sBar + 8u * (S + s); };
  auto sf_full = [&](int s) { return sBar + 8u * (2 * S + s); };
  auto sg_full = [&](int t) { return sBar + 8u * (3 * S + t); };      // scale buffer loaded
  auto sg_empty = [&](int t) { return sBar + 8u * (3 * S + 2 + t); }; // scale buffer read
  const uint32_t acc_full = sBar + 8u * (3 * S + 4);
  const uint32_t acc_empty = sBar + 8u * (3 * S + 5);  // the epilogue has read the accumulator
  const uint32_t slot = acc_empty + 8u;
  volatile uint32_t* const tmem_slot_ptr =
      reinterpret_cast<volatile uint32_t*>(base_ptr + (slot - base));
  volatile uint32_t* const abort_flag = tmem_slot_ptr + 1;
  volatile int32_t* const lap_armed = reinterpret_cast<volatile int32_t*>(tmem_slot_ptr + 4);  // [S]
  volatile int32_t* const lap_sg = lap_armed + S;                                                // [2]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_blk = p.K / 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
      mbar_init(sf_full(s), 4);
      lap_armed[s] = -1;
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(sg_full(t), 1);
      mbar_init(sg_empty(t), 4);
      lap_sg[t] = -1;
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 4);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (threadIdx.x == 64) {
    tma_prefetch_map(&tmap_a);
    tma_prefetch_map(&tmap_b);
    tma_prefetch_map(&tmap_sa);
    tma_prefetch_map(&tmap_sb);
  }
  if (warp == 1) {
    tmem_alloc(slot, T::kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot_ptr;

  // The CTA's tiles: t = blockIdx.x, + gridDim.x, ...; tile t is rows 128 (t / tiles_n)
  // and columns BN (t % tiles_n).  Every role walks the same list; the stage ring and the
  // scale buffers run on across tiles (gs counts stages, gg groups of kMxGroup stages).
  const int first = static_cast<int>(blockIdx.x);
  const int step = static_cast<int>(gridDim.x);

  if (warp == 0) {
    // -------------------------------------------------------------- producer --
    if (lane == 0) {
      grid_dependency_wait();
      int gs = 0, gg = 0;
      bool ok = true;
      for (int tile = first; ok && tile < p.num_tiles; tile += step) {
        const int m0 = (tile / p.tiles_n) * kMxBM;
        const int n0 = (tile % p.tiles_n) * BN;
        for (int kb = 0; kb < p.k_blocks; ++kb, ++gs) {
          if (kb % kMxGroup == 0) {
            // the scale bytes of stages kb .. kb + kMxGroup - 1
            const int t = gg & 1;
            if (!wait_bounded<false>(sg_empty(t), (static_cast<uint32_t>(gg >> 1) & 1u) ^ 1u,
                                     abort_flag, p.timeout_ns)) {
              record_timeout(p.status, abort_flag, kSiteMxEmpty);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(sg_full(t), T::kScaleBytes);
            const uint32_t dst = sScale + t * T::kScaleBytes;
            tma_load_2d(dst, &tmap_sa, sg_full(t), 4 * kb, m0);
            tma_load_2d(dst + 4u * kMxGroup * kMxBM, &tmap_sb, sg_full(t), 4 * kb, n0);
            lap_sg[t] = gg >> 1;
            ++gg;
          }
          const int s = gs % S;
          const int lap = gs / S;
          if (!wait_bounded<false>(empty(s), (static_cast<uint32_t>(lap) & 1u) ^ 1u, abort_flag,
                                   p.timeout_ns)) {
            record_timeout(p.status, abort_flag, kSiteMxEmpty);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full(s), T::kStageBytes);
          const uint32_t dst = base + s * T::kStageBytes;
          tma_load_2d(dst, &tmap_a, full(s), kb * kMxBK, m0);
          tma_load_2d(dst + kA, &tmap_b, full(s), kb * kMxBK, n0);
          lap_armed[s] = lap;
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer --
    grid_dependency_wait();
    if (lane == 0) {
      const uint64_t a_desc0 = smem_desc_sw128(base, 16u, 1024u);
      const uint64_t b_desc0 = smem_desc_sw128(base + kA, 16u, 1024u);
      bool ok = true;
      int gs = 0, ti = 0;
      for (int tile = first; ok && tile < p.num_tiles; tile += step, ++ti) {
        // the accumulator is free once the epilogue has read the previous tile's
        if (!wait_bounded<false>(acc_empty, (static_cast<uint32_t>(ti) & 1u) ^ 1u, abort_flag,
                                 p.timeout_ns)) {
          record_timeout(p.status, abort_flag, kSiteMxAcc);
          ok = false;
          break;
        }
        for (int kb = 0; kb < p.k_blocks; ++kb, ++gs) {
          const int s = gs % S;
          const uint32_t ph = static_cast<uint32_t>(gs / S) & 1u;
          if (!wait_bounded<false>(full(s), ph, abort_flag, p.timeout_ns)) {
            record_timeout(p.status, abort_flag, kSiteMxFull);
            ok = false;
            break;
          }
          if (!wait_bounded<false>(sf_full(s), ph, abort_flag, p.timeout_ns)) {
            record_timeout(p.status, abort_flag, kSiteMxScales);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t stage = (static_cast<uint64_t>(s) * T::kStageBytes) >> 4;
          const uint32_t sfa = tmem_base + T::kSfCol + T::kSfStride * s;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // 32 K bytes per MMA: 32 B along the 128-byte swizzled row
            mma_mx_ss(tmem_base, a_desc0 + stage + 2u * k, b_desc0 + stage + 2u * k,
                      mx_scale_ids(p.idesc, static_cast<uint32_t>(k)), sfa, sfa + T::kSfB,
                      (kb > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(empty(s));           // frees the stage's operands and scales
        }
        if (ok) mma_commit(acc_full);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------- scales, then epilogue --
    grid_dependency_wait();
    const int q = warp & 3;                         // Tensor Memory lane quadrant
    const int row = q * 32 + lane;                  // this thread's row of the tile
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    auto wait_warp = [&](uint32_t bar, uint32_t parity, uint32_t site) -> bool {
      bool r = true;
      if (lane == 0) r = wait_bounded<false>(bar, parity, abort_flag, p.timeout_ns);
      __syncwarp();
      r = __shfl_sync(0xFFFFFFFFu, r ? 1 : 0, 0) != 0;
      if (!r && lane == 0 && !*abort_flag) record_timeout(p.status, abort_flag, site);
      return r;
    };
    // This warp's 32 x 32 staging tile: row r's 64 bytes at 64 r, its four 16-byte units
    // XOR-swizzled by (r/2) % 4.  Each thread writes its row of a chunk there, then every
    // store instruction writes 8 rows x 64 contiguous bytes instead of 32 rows x 16 (the
    // rows of C are ldc apart).
    uint8_t* const stg = base_ptr + (sEpi - base) + static_cast<uint32_t>(q) * 2048u;
    uint16_t* const c16 = reinterpret_cast<uint16_t*>(p.C);
    bool ok = true;
    int gs = 0, gg = 0, ti = 0;
    for (int tile = first; ok && tile < p.num_tiles; tile += step, ++ti) {
      const int m0 = (tile / p.tiles_n) * kMxBM;
      const int n0 = (tile % p.tiles_n) * BN;
      int t = 0;                                    // scale buffer of the current group
      for (int kb = 0; ok && kb < p.k_blocks; ++kb, ++gs) {
        if (kb % kMxGroup == 0) {
          t = gg & 1;
          if (!(ok = wait_warp(sg_full(t), static_cast<uint32_t>(gg >> 1) & 1u, kSiteMxScales)))
            break;
        }
        // this thread's words: A for row m0 + row, B for columns n0 + 32c + lane (every
        // quadrant writes all of B's, which each quadrant reads from its own lanes)
        const uint8_t* grp = base_ptr + (sScale - base) + t * T::kScaleBytes;
        const uint32_t wa = mx_scale_word(grp + row * 4 * kMxGroup, m0 + row, p.M, kb, n_blk);
        uint32_t wb[BN / 32];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
          wb[c] = mx_scale_word(grp + 4 * kMxGroup * (kMxBM + 32 * c + lane), n0 + 32 * c + lane,
                                p.N, kb, n_blk);
        if (kb % kMxGroup == kMxGroup - 1 || kb == p.k_blocks - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(sg_empty(t));     // this warp is done with the buffer
          ++gg;
        }
        const int s = gs % S;
        if (!(ok = wait_warp(empty(s), (static_cast<uint32_t>(gs / S) & 1u) ^ 1u, kSiteMxEmpty)))
          break;
        tc_fence_after_sync();
        const uint32_t col = T::kSfCol + T::kSfStride * s;
        tmem_store_1col(lane_base + col + static_cast<uint32_t>(q), wa);
#pragma unroll
        for (int c = 0; c < BN / 32; c += 4)
          tmem_store_4cols(lane_base + col + T::kSfB + c, wb[c], wb[c + 1], wb[c + 2], wb[c + 3]);
        tmem_store_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(sf_full(s));
      }
      if (!ok || !(ok = wait_warp(acc_full, static_cast<uint32_t>(ti) & 1u, kSiteMxAcc))) break;
      tc_fence_after_sync();
      const int gi = m0 + row;
      uint16_t* crow = c16 + static_cast<int64_t>(gi) * p.ldc;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_load_32cols(lane_base + 32u * c, v);
        tmem_load_wait();
        if (c == BN / 32 - 1) {
          // the whole accumulator is in registers or stored: the next tile may overwrite it
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty);
        }
        uint32_t o2[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float x0 = __uint_as_float(v[2 * j]), x1 = __uint_as_float(v[2 * j + 1]);
          if (p.relu) {
            x0 = x0 > 0.0f ? x0 : 0.0f;
            x1 = x1 > 0.0f ? x1 : 0.0f;
          }
          o2[j] = pack2<kBf16, false>(x0, x1);
        }
        const int gj = n0 + 32 * c;
        if (p.c_vec && gj + 32 <= p.N) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t u = static_cast<uint32_t>(j) ^ ((static_cast<uint32_t>(lane) >> 1) & 3u);
            *reinterpret_cast<uint4*>(stg + lane * 64 + u * 16) =
                make_uint4(o2[4 * j], o2[4 * j + 1], o2[4 * j + 2], o2[4 * j + 3]);
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = (lane >> 2) + 8 * i;        // row of this warp's 32
            const int j = lane & 3;                   // its 16-byte unit (8 columns)
            const uint32_t u = static_cast<uint32_t>(j) ^ ((static_cast<uint32_t>(r) >> 1) & 3u);
            const uint4 val = *reinterpret_cast<const uint4*>(stg + r * 64 + u * 16);
            const int grow = m0 + 32 * q + r;
            if (grow < p.M)
              *reinterpret_cast<uint4*>(c16 + static_cast<int64_t>(grow) * p.ldc + gj + 8 * j) = val;
          }
          __syncwarp();                               // the tile is read before it is reused
        } else if (gi < p.M) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (gj + j < p.N) crow[gj + j] = static_cast<uint16_t>(o2[j >> 1] >> (16 * (j & 1)));
          }
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
    for (int s = 0; s < S; ++s) {
      const int lap = lap_armed[s];
      if (lap >= 0 && !wait_bounded<false>(full(s), static_cast<uint32_t>(lap) & 1u, nullptr,
                                           p.timeout_ns)) {
        record_timeout(p.status, abort_flag, kSiteMxDrain);
      }
    }
    for (int t = 0; t < 2; ++t) {
      const int lap = lap_sg[t];
      if (lap >= 0 && !wait_bounded<false>(sg_full(t), static_cast<uint32_t>(lap) & 1u, nullptr,
                                           p.timeout_ns)) {
        record_timeout(p.status, abort_flag, kSiteMxDrain);
      }
    }
  }
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, T::kTmemCols);
  }
}

}  // namespace tl
