// gemm_kernel.cuh -- the persistent, warp-specialised tiled GEMM for sm_103a.
//
// C[M,N] = epi(op(A)[M,K] . op(B)[K,N]), fp16/bf16 operands, fp32 accumulation in
// Tensor Memory, epi in {identity, ReLU}, round-to-nearest-even on the way out.
//
// The pages' quickstart kernel tiles C into BM x BN blocks, copies A and B tiles
// global -> shared for each BK slice of K under a multi-stage software pipeline,
// multiplies them into an fp32 accumulator and copies the accumulator back
// ("TileLang: a tile language one level below Triton", section "first kernel:
// GEMM", and its generated-code excerpt: a producer that only issues TMA loads and
// a consumer that only issues MMAs, handing stages over through full/empty
// mbarrier pairs).  This kernel keeps that structure and maps it onto sm_103a:
//
//   warps 0, 6, 7        TMA producers (one thread each), taking turns by stage: for
//                        its (tile, k-block) iterations a producer waits for a free
//                        ring slot, arms the slot's "full" barrier with the stage's
//                        byte count and issues the A and B boxes.  Boxes that run
//                        past the matrix edge are zero-filled by the TMA unit, so
//                        partial tiles add exact zeros ("TileLang core primitives"
//                        page, section 4.2: out-of-range reads give the safe value 0).
//   warp 1 (one thread)  tcgen05 MMA issuer: waits for a full slot, issues BK/16
//                        MMAs of 128 x BN x 16 into a Tensor Memory accumulator
//                        (overwrite on the tile's first step: the pages' clear_accum
//                        = (k == 0)), and commits the slot back to the producer.
//                        After a tile's last k-block it commits the accumulator to
//                        the epilogue ("NVIDIA backend codegen" page, sections 3.4
//                        and 4.6.1).  Warp 1 also owns the Tensor Memory allocation.
//   warps 2-5            epilogue: Tensor Memory -> registers (tcgen05.ld), ReLU
//                        (max(x, 0), "TileLang core primitives" page, section 3.8),
//                        cast with round-to-nearest-even, swizzled shared staging,
//                        then TMA bulk stores that skip rows/columns outside C.
//                        (C^T plans: 16-byte stores after a transpose across lanes.
//                        CTA pairs: warps 0, 1, 6, 7 also finish half of the last tile.)
//
// The accumulator is double-buffered in Tensor Memory (2 x BN columns), so the
// epilogue of one tile overlaps the main loop of the next.  CTAs are persistent:
// CTA b handles tiles b, b + grid, b + 2*grid, ... of a grouped raster order
// (each tile exactly once, "TileLang: from tile dataflow to controllable AI
// kernels", section "concurrency correctness").
//
// Every wait is bounded: after p.timeout_ns a waiter records TL timeout status,
// raises a CTA-wide abort flag, and every role unwinds -- the producer waits for
// its issued loads, the MMA thread commits and waits for its issued MMAs, the
// epilogue waits for its bulk stores, and warp 1 frees Tensor Memory -- so a
// failure returns an error status instead of hanging the GPU.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace tl {

constexpr int kBM = 128;              // MMA M: one accumulator row per TMEM lane
// A pipeline stage holds, per matrix row, BK elements of K in 128-byte chunks (one
// swizzle row each): 64 elements of a 16-bit type or 128 of an 8-bit one.  One MMA
// consumes 32 bytes of K per row: K = 16 (kind::f16) or 32 (kind::f8f6f4).
constexpr int kChunkBytes = 128;
constexpr int kMmaKBytes = 32;
constexpr int kThreads = 256;         // 8 warps: producers 0, 6, 7; MMA 1; epilogue 2-5
constexpr int kProducers = 3;
constexpr int kEpiWarps = 4;
constexpr int kChunk = 64;            // epilogue columns per staging chunk (128 B)
constexpr uint32_t kStagingBytes = kEpiWarps * 2 * 32 * 128;  // 2 x (32 rows x 128 B) per warp

// Shared staging for the TMA store of C: 64-column chunks, so tiles narrower than 64
// columns (which write C with plain stores) need none.
template <int BN>
__host__ __device__ constexpr uint32_t staging_bytes() {
  return BN >= kChunk ? kStagingBytes : 0u;
}

// Status word layout (device global, first timeout wins):
//   bits 0-7  tl_status (8 = timeout), bits 8-15 wait site, bits 16-31 blockIdx.x
enum WaitSite : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaTmemEmpty = 2,
  kSiteMmaFull = 3,
  kSiteEpiTmemFull = 4,
  kSiteDrain = 5,
  kSiteStreamK = 6,
  kSiteInjected = 7,    // the test hook's wait that nothing ends (GemmParams::stall)
  kSiteClusterSplit = 8,  // cluster split-K hand-over of a partial accumulator
};

struct GemmParams {
  int32_t M, N, K;
  int32_t tiles_m, tiles_n, num_tiles, k_blocks;
  int32_t stages;
  int32_t raster_group;
  int32_t trans_a, trans_b;
  int32_t bf16;             // output type (and kind::f16 inputs) is bf16, else fp16
  int32_t relu;
  int32_t tma_store;        // 1: TMA bulk store of C; 0: predicated st.global
  int32_t c_trans;          // 1: the kernel computes C^T (operands swapped by the host):
                            // its element (i, j) goes to C[j * ldc + i], plain stores
  int32_t scale;            // 1: multiply the accumulator by alpha before the epilogue
  float alpha;
  int32_t c_vec;            // 1: C's base and pitch are 16-byte aligned: plain stores of
                            // a full chunk go out as 16-byte vectors
  int32_t l2_prefetch;      // k-blocks the producer prefetches into L2 ahead of the ring
  int32_t a3d, b3d;         // operand map is the 3-D view {64, rows, chunks} (one box
                            // per stage) instead of 2-D boxes of one 64-chunk each
  int32_t producers;        // producer threads taking turns by stage (1..3, <= stages)
  // Stream-K: tiles [0, dp_tiles) run whole, one per unit (CTA or CTA pair) in turn;
  // the k-block iterations of tiles [dp_tiles, num_tiles), sk_iters of them, are split
  // evenly over the units.  A unit that starts mid-tile stores that tile's partial sum
  // (fp32) in its slot of sk_partials and raises its flags (sk_token); the unit that
  // holds the tile's first k-block adds the partials in order and writes C.
  int32_t dp_tiles;
  int64_t sk_iters;
  // Cluster split-K (one-CTA tiles of a power-of-two width only): 1, or 2 CTAs of a
  // cluster on each tile, CTA r taking k-blocks [r kb / 2, (r + 1) kb / 2).  CTA r
  // finishes columns [r BN / 2, (r + 1) BN / 2) of the tile: each CTA sends the fp32
  // partial sums of the other half into its peer's shared memory (distributed shared
  // memory), adds the peer's to its own half and writes C.
  int32_t ksplit;
  int32_t serpentine;       // 1: odd-numbered whole tiles of each unit walk K backwards
  float* sk_partials;                 // [unit][cta][4 warps][BN/4 col groups][32 lanes][4]
  unsigned long long* sk_flags;       // [unit][cta][4 warps]
  unsigned long long sk_token;        // unique to this launch, never 0
  uint32_t idesc;
  void* C;                  // used when tma_store == 0
  int64_t ldc;
  uint32_t* status;         // device status word (never NULL)
  uint64_t timeout_ns;
  int32_t stall;            // test hook: 1 = the MMA thread first waits on a barrier that
                            // nothing arrives on, so the wait runs out and every role unwinds
};

// Shared memory of one stage in one CTA: A is 128 rows x BK, B is BN/CG columns x BK,
// elements of EB bytes.
template <int BK, int EB = 2>
__host__ __device__ constexpr uint32_t a_stage_bytes() {
  return static_cast<uint32_t>(kBM) * BK * EB;
}

template <int BN, int CG, int BK, int EB = 2>
__host__ __device__ constexpr uint32_t b_stage_bytes() {
  return static_cast<uint32_t>(BN / CG) * BK * EB;
}

// Barrier block: full[stages], empty[stages], tmem_full[2], tmem_empty[2], mma_done,
// red_full[4], red_empty[4] (cluster split-K, one per epilogue warp), then the 4-byte
// Tensor Memory base slot, the 4-byte abort flag, per stage the last lap at which a
// producer armed that stage (int32 x 8, -1 = never), and the peer CTA's abort flag as the
// peer wrote it at teardown (4 bytes, 8 reserved).
__host__ __device__ constexpr uint32_t barrier_bytes(int stages) {
  return static_cast<uint32_t>(8 * (2 * stages + 5 + 8) + 8 + 32 + 8);
}

// Cluster split-K receive buffer: the peer's partial sums of the BN / 2 columns this CTA
// finishes, per epilogue warp BN / 2 columns x 32 lanes, four columns per 16-byte entry,
// lane-major.
template <int BN>
__host__ __device__ constexpr uint32_t red_bytes(int ksplit) {
  return ksplit > 1 ? static_cast<uint32_t>(64 * BN * 4) : 0u;
}

// `staging`: the TMA-store staging of C; a kernel that computes C^T (plain stores) has none.
template <int BN, int CG, int BK, int EB = 2>
__host__ __device__ constexpr uint32_t smem_bytes_for(int stages, int ksplit = 1,
                                                      bool staging = true) {
  // +1024: the dynamic shared memory base is rounded up to 1024 B in the kernel
  return 1024u + stages * (a_stage_bytes<BK, EB>() + b_stage_bytes<BN, CG, BK, EB>()) +
         (staging ? staging_bytes<BN>() : 0u) + red_bytes<BN>(ksplit) + barrier_bytes(stages);
}

// Grouped raster order: walk `group` tile-rows top to bottom, then the next column.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group, int& mb,
                                            int& nb) {
  const int per_group = group * tiles_n;
  const int g = t / per_group;
  const int first_m = g * group;
  const int rows = min(tiles_m - first_m, group);
  const int r = t - g * per_group;
  mb = first_m + r % rows;
  nb = r / rows;
}

__device__ __forceinline__ void record_timeout(uint32_t* status, volatile uint32_t* abort_flag,
                                               uint32_t site) {
  *abort_flag = 1u;
  const uint32_t word = 8u | (site << 8) | (static_cast<uint32_t>(blockIdx.x & 0xFFFF) << 16);
  atomicCAS(status, 0u, word);
}

// One poll of a barrier phase; cluster scope when the arrivals may come from the
// peer CTA of a pair.
template <bool kCluster>
__device__ __forceinline__ bool poll(uint32_t bar, uint32_t parity) {
  return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
}

// Bounded wait for the phase with parity `parity` of barrier `bar`.  Returns false
// on timeout or, when `abort_flag` is not NULL, once another role of this CTA has
// raised it.  Drain waits (in-flight copies and MMAs at exit) pass NULL: they must
// see their operations land even while the CTA is unwinding.
//
// The limit is kept in SM cycles (%clock64 is cheap to read; a %globaltimer read in
// the poll loop delayed the wake-up of the pipeline threads by hundreds of cycles):
// 4 cycles per nanosecond of limit, so the wait lasts at least the limit for any SM
// clock up to 4 GHz.
template <bool kCluster>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile uint32_t* abort_flag, uint64_t timeout_ns) {
  if (poll<kCluster>(bar, parity)) return true;
  const uint64_t t0 = clock_cycles();
  const uint64_t limit = timeout_ns * 4u;
  uint32_t spins = 0;
  while (true) {
    if (poll<kCluster>(bar, parity)) return true;
    if ((++spins & 31u) == 0u) {
      if (abort_flag != nullptr && *abort_flag) return false;
      if (clock_cycles() - t0 > limit) return false;
    }
  }
}

// The work of one unit (CTA or CTA pair): whole tiles u, u + U, ... below dp_tiles,
// then its share [it, it_end) of the split iterations, cut at tile boundaries.  Every
// role of the unit walks the same sequence.
struct WorkItem {
  int tile, k0, k1;   // k-blocks [k0, k1) of tile `tile` (stream-K bookkeeping)
  int first, step, n; // the unit's walk: k-blocks first, first + step, ... (n of them)
  __device__ __forceinline__ int kb_at(int i) const { return first + step * i; }
};

__device__ __forceinline__ int64_t sk_begin(const GemmParams& p, int unit, int units) {
  return static_cast<int64_t>(unit) * p.sk_iters / units;
}

struct WorkIter {
  int next_dp, step, dp_end, kb, kr0, kr1, n_dp, serp;
  int64_t it, it_end;
  // krank: this CTA's share of each whole tile's k-blocks under the cluster split-K, the
  // contiguous range [krank kb / 2, (krank + 1) kb / 2).  (Every other k-block instead was
  // measured 3 % slower at M = 128 and 1 % faster at M = 16.)
  __device__ __forceinline__ WorkIter(const GemmParams& p, int unit, int units, int krank = 0)
      : next_dp(unit), step(units), dp_end(p.dp_tiles), kb(p.k_blocks),
        kr0(krank * p.k_blocks / max(1, p.ksplit)),
        kr1((krank + 1) * p.k_blocks / max(1, p.ksplit)), n_dp(0), serp(p.serpentine),
        it(sk_begin(p, unit, units)), it_end(sk_begin(p, unit + 1, units)) {}
  __device__ __forceinline__ bool next(WorkItem& w) {
    if (next_dp < dp_end) {
      // serpentine: every other whole tile walks K backwards, so that it starts on the
      // k-slices the previous wave of tiles (which shares its A or B panels) read last,
      // still in L2
      const bool rev = serp != 0 && (n_dp & 1) != 0;
      w = {next_dp, 0, kb, rev ? kr1 - 1 : kr0, rev ? -1 : 1, kr1 - kr0};
      next_dp += step;
      ++n_dp;
      return true;
    }
    if (it < it_end) {
      const int t = static_cast<int>(it / kb);
      const int k0 = static_cast<int>(it - static_cast<int64_t>(t) * kb);
      const int64_t left = it_end - it;
      const int k1 = left < static_cast<int64_t>(kb - k0) ? k0 + static_cast<int>(left) : kb;
      w = {dp_end + t, k0, k1, k0, 1, k1 - k0};
      it += k1 - k0;
      return true;
    }
    return false;
  }
};

// A compile-time integer passed as a value (the width of an epilogue step).
template <int V>
struct IntConst {
  static constexpr int value = V;
};

// W consecutive accumulator columns of the warp's 32 lanes into v (W = 8, 16 or a
// multiple of 32); tmem_load_wait() before use.
template <int W>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t* v) {
  if constexpr (W == 8) {
    tmem_load_8cols(taddr, *reinterpret_cast<uint32_t(*)[8]>(v));
  } else if constexpr (W == 16) {
    tmem_load_16cols(taddr, *reinterpret_cast<uint32_t(*)[16]>(v));
  } else {
    static_assert(W % 32 == 0, "accumulator loads of 8, 16 or 32k columns");
#pragma unroll
    for (int h = 0; h < W / 32; ++h)
      tmem_load_32cols(taddr + 32 * h, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * h));
  }
}

// Transpose of an 8 x 8 matrix of 16-bit elements held by 8 consecutive lanes: lane r
// (r = lane % 8) enters with row r as four words (word k = elements 2k, 2k + 1, the
// lower in the low half) and leaves with column r in the same form.  Three rounds of
// exchanges between lanes 4, 2 and 1 apart, each swapping the off-diagonal blocks of
// the next-smaller block size (4 x 4, 2 x 2, then single elements within a word).
// All 32 lanes of the warp take part.
__device__ __forceinline__ void transpose8x8_u16(uint32_t& w0, uint32_t& w1, uint32_t& w2,
                                                 uint32_t& w3, int r) {
  constexpr uint32_t kAll = 0xFFFFFFFFu;
  const bool h4 = (r & 4) != 0, h2 = (r & 2) != 0, h1 = (r & 1) != 0;
  uint32_t s0 = __shfl_xor_sync(kAll, h4 ? w0 : w2, 4);
  uint32_t s1 = __shfl_xor_sync(kAll, h4 ? w1 : w3, 4);
  if (h4) { w0 = s0; w1 = s1; } else { w2 = s0; w3 = s1; }
  s0 = __shfl_xor_sync(kAll, h2 ? w0 : w1, 2);
  s1 = __shfl_xor_sync(kAll, h2 ? w2 : w3, 2);
  if (h2) { w0 = s0; w2 = s1; } else { w1 = s0; w3 = s1; }
  auto swap_halves = [&](uint32_t& w) {
    const uint32_t got = __shfl_xor_sync(kAll, h1 ? (w & 0xFFFFu) : (w >> 16), 1);
    w = h1 ? ((w & 0xFFFF0000u) | got) : ((w & 0xFFFFu) | (got << 16));
  };
  swap_halves(w0);
  swap_halves(w1);
  swap_halves(w2);
  swap_halves(w3);
}

// One 32-row x 64-column chunk of C (a warp's rows, packed 16-bit pairs) through a
// staging buffer in the TMA store's 128-byte swizzle and one bulk store at (x, y) of C.
// Two buffers per warp alternate: before writing `buf`, the store issued two chunks ago
// (which read it) must have read it.  `store` false issues an empty group (the counts
// stay uniform across lanes and chunks).
__device__ __forceinline__ void stage_and_store_chunk(const CUtensorMap* map, uint32_t buf,
                                                      const uint32_t* packed, int lane, int x,
                                                      int y, bool store) {
  if (lane == 0) bulk_wait_group_read<1>();
  __syncwarp();
  // row `lane` of the 32 x 64 staging box: 16-byte chunk j lands at chunk j ^ (row % 8)
  const uint32_t row_addr = buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t dst = row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(packed[4 * j]),
                 "r"(packed[4 * j + 1]), "r"(packed[4 * j + 2]), "r"(packed[4 * j + 3])
                 : "memory");
  }
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0 && store) tma_store_2d(map, buf, x, y);   // clipped at M, N
  if (lane == 0) bulk_commit_group();
}

template <bool kBf16, bool kRelu>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kRelu) {
    lo = lo > 0.0f ? lo : 0.0f;   // max(x, 0); -0 and NaN give +0
    hi = hi > 0.0f ? hi : 0.0f;
  }
  if constexpr (kBf16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  } else {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
}

// Epilogue + cast of 2n fp32 values into n packed pairs.  The output type and the
// ReLU are template arguments so that the unrolled loop carries no branches (chosen
// once per chunk by pack_chunk; per-element branches on runtime flags cost the
// epilogue ~600 cycles per 64-column chunk in branch resolution).
template <int n, bool kBf16, bool kRelu>
__device__ __forceinline__ void pack_n(const uint32_t* v, uint32_t* packed) {
#pragma unroll
  for (int j = 0; j < n; ++j)
    packed[j] = pack2<kBf16, kRelu>(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
}

template <int n>
__device__ __forceinline__ void pack_chunk(const uint32_t* v, uint32_t* packed, int bf16, int relu) {
  if (bf16) {
    if (relu) pack_n<n, true, true>(v, packed);
    else pack_n<n, true, false>(v, packed);
  } else {
    if (relu) pack_n<n, false, true>(v, packed);
    else pack_n<n, false, false>(v, packed);
  }
}

// CG = 1: one CTA computes a 128 x BN tile.  CG = 2: a cluster of two CTAs on an SM
// pair computes a 256 x BN tile with cta_group::2 MMAs issued by the even CTA; CTA r
// holds rows [128 r, 128 r + 128) of A and columns [r BN/2, (r + 1) BN/2) of B, and
// receives accumulator rows [128 r, 128 r + 128) x all BN columns in its Tensor Memory.
// Each CTA's TMA copies complete on the even CTA's "full" barrier; the MMA commits are
// multicast to both CTAs' "empty", "tmem_full" and "done" barriers; both CTAs'
// epilogue warps release the accumulator on the even CTA's "tmem_empty" barrier.
//
// BK is the K depth of one pipeline stage: 1 or 2 chunks of 128 bytes per matrix row
// (each one swizzle row), i.e. 64 or 128 elements of fp16/bf16 (EB = 2) and 128 or 256
// of E4M3/E5M2 (EB = 1, kind::f8f6f4 MMAs).  Deeper stages halve the TMA instructions
// and barrier hand-offs per byte: on GB300 one TMA instruction costs the issuing
// thread a few hundred cycles whatever its box size.
template <int BN, int CG, int BK, int EB = 2>
__global__ void __launch_bounds__(kThreads, 1)
    tl_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b,
                   const __grid_constant__ CUtensorMap tmap_c, const GemmParams p) {
  static_assert(BN == 16 || BN == 32 || BN == 64 || BN == 128 || BN == 192 || BN == 224 ||
                    BN == 256,
                "BN must be 16, 32, 64, 128, 192, 224 or 256");
  static_assert(CG == 1 || (CG == 2 && BN >= 128), "pairs need BN/2 >= 64");
  constexpr bool kPair = CG == 2;
  static_assert(EB == 1 || EB == 2, "1- or 2-byte elements");
  static_assert(BK * EB == 128 || BK * EB == 256, "one or two 128-byte chunks per stage");
  static_assert(EB == 2 || BN >= 64, "8-bit operands: BN >= 64");
  constexpr int kChunkElems = kChunkBytes / EB;            // K (or MN) elements per chunk
  constexpr int kMmaK = kMmaKBytes / EB;                   // K elements of one MMA
  constexpr int kBnCta = BN / CG;                          // B columns this CTA loads
  constexpr int kKChunks = BK / kChunkElems;               // 128-byte K chunks per stage
  constexpr uint32_t kAStageBytes = a_stage_bytes<BK, EB>();
  constexpr uint32_t kBStage = b_stage_bytes<BN, CG, BK, EB>();
  constexpr uint32_t kMNChunkBytes = 128u * BK;            // one 128-byte(MN) x BK(K) chunk
  // Two accumulators, kAccStride columns apart.  Widths that are not a power of two
  // (192, 224: K-major B only) keep the second one at column 256, so that every Tensor
  // Memory address the kernel forms is a multiple of 32 columns; the allocation is a
  // power of two of at least 32 columns.
  constexpr uint32_t kAccStride = (BN == 192 || BN == 224) ? 256u : static_cast<uint32_t>(BN);
  constexpr uint32_t kTmemCols = 2 * kAccStride < 32 ? 32 : 2 * kAccStride;
  // Epilogue columns per step: one 128-byte staging row, or the whole tile when it is
  // narrower (then K-major B only: a 64-wide M/N-major box would not fit the tile).
  // A 224-wide tile ends with one 32-column step, written by plain stores.
  constexpr int kEC = BN < kChunk ? BN : kChunk;
  constexpr int kFull = BN / kEC;                          // full-width epilogue steps
  constexpr int kTail = BN - kFull * kEC;                  // 0, or 32 for BN 224
  // the cluster split-K halves the columns: power-of-two widths only
  constexpr bool kColumnSplit = CG == 1 && (BN & (BN - 1)) == 0;
  static_assert(kTail == 0 || kTail == 32, "epilogue tail of 32 columns");
  // A CTA pair's last whole tile (TMA stores of C) is finished by all eight warps: the
  // four epilogue warps take its first kHelpC 64-column steps, warps 0, 1, 6 and 7 (idle
  // by then; warp w reads the Tensor Memory lanes of quadrant w % 4) the rest.  (2048^3:
  // 18.0 -> 17.1 us.  Compiled into the one-CTA kernels, where the planner's tilings
  // leave it idle, the code alone cost the quickstart tiling 0.4 us per call.)
  constexpr bool kHelpable = kPair && kEC == kChunk && kFull >= 2;
  constexpr int kHelpC = kHelpable ? (kFull + 1) / 2 : kFull;

  // The next kernel in the stream may start its set-up now (it waits for this grid to
  // complete before it touches global memory, see grid_dependency_wait below).
  grid_launch_dependents();
  if (threadIdx.x == 64) {   // an epilogue warp, idle during set-up: fetch the maps early
    tma_prefetch_map(&tmap_a);
    tma_prefetch_map(&tmap_b);
    if (p.tma_store) tma_prefetch_map(&tmap_c);   // (else the map is left unencoded)
  }

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const int S = p.stages;

  const bool ksplit = !kPair && p.ksplit > 1;
  const uint32_t sA = base;
  const uint32_t sB = sA + S * kAStageBytes;
  const uint32_t sC = sB + S * kBStage;
  const uint32_t sRed = sC + (p.c_trans ? 0u : staging_bytes<BN>());   // C^T: no staging
  const uint32_t sBar = sRed + red_bytes<BN>(ksplit ? 2 : 1);
  auto full_bar = [&](int s) { return sBar + 8u * s; };
  auto empty_bar = [&](int s) { return sBar + 8u * (S + s); };
  auto tfull_bar = [&](int a) { return sBar + 8u * (2 * S + a); };
  auto tempty_bar = [&](int a) { return sBar + 8u * (2 * S + 2 + a); };
  const uint32_t done_bar = sBar + 8u * (2 * S + 4);
  auto red_full_bar = [&](int q) { return sBar + 8u * (2 * S + 5 + q); };
  auto red_empty_bar = [&](int q) { return sBar + 8u * (2 * S + 9 + q); };
  const uint32_t slot = sBar + 8u * (2 * S + 13);
  volatile uint32_t* const tmem_slot_ptr =
      reinterpret_cast<volatile uint32_t*>(base_ptr + (slot - base));
  volatile uint32_t* const abort_flag = tmem_slot_ptr + 1;
  volatile int32_t* const lap_armed = reinterpret_cast<volatile int32_t*>(tmem_slot_ptr + 2);
  volatile uint32_t* const peer_abort = tmem_slot_ptr + 10;   // written by the peer CTA
  const uint32_t peer_abort_addr = slot + 40u;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;   // position in the CTA pair
  const bool leader = rank == 0;
  // cluster split-K: krank 0 finishes each tile, krank 1 contributes its partial sum
  const int krank = ksplit ? static_cast<int>(cluster_ctarank()) : 0;
  const int cta_per_unit = CG * (ksplit ? 2 : 1);
  const int cluster_id = static_cast<int>(blockIdx.x) / cta_per_unit;
  const int n_clusters = static_cast<int>(gridDim.x) / cta_per_unit;

  // TMA boxes of one stage in this CTA (a chunk is kChunkElems = 128 bytes wide).
  // A: K-major, one 2-D box {chunk K, 128 M} per K chunk, or M-major, one 2-D box
  // {chunk M, BK K} per chunk of M; or, with a 3-D map, the whole stage in one box.
  // B likewise with BN/CG columns.
  const int n_a_boxes = p.a3d ? 1 : (p.trans_a ? kBM / kChunkElems : kKChunks);
  const int n_b_boxes = p.b3d ? 1 : (p.trans_b ? kKChunks : kBnCta / kChunkElems);
  const int n_boxes = n_a_boxes + n_b_boxes;
  // producers take turns by stage (see below); at most one per ring slot
  const int n_producers = min(kProducers, min(S, max(1, p.producers)));

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);   // the producer of that iteration arrives + TMA bytes
      mbar_init(empty_bar(s), 1);            // one tcgen05.commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);                 // one tcgen05.commit per tile
      mbar_init(tempty_bar(a), kEpiWarps * CG);   // every epilogue warp of the pair
    }
    mbar_init(done_bar, 1);
    for (int q = 0; q < 4; ++q) {
      mbar_init(red_full_bar(q), 32);    // the 32 lanes of the sending warp q
      mbar_init(red_empty_bar(q), 1);    // one lane of the finishing warp q
    }
    *abort_flag = 0u;
    *peer_abort = 0u;
    for (int s = 0; s < 8; ++s) lap_armed[s] = -1;
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(slot, kTmemCols);
      tmem_relinquish_alloc_permit_pair();
    } else {
      tmem_alloc(slot, kTmemCols);
      tmem_relinquish_alloc_permit();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (kPair || ksplit) cluster_sync_all();   // the peer's barriers exist before any use
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot_ptr;
  // Everything above touched only this CTA's shared and Tensor Memory.  The operands,
  // C and the split workspace may still be in use by the previous kernel of the
  // stream: every role passes grid_dependency_wait() before its first global access
  // and before its first bounded wait (so a long previous kernel cannot run down a
  // wait's limit).  The producers first work out their first box.

  if (warp == 0 || warp >= 6) {
    // ----------------------------------------------------------- producers --
    // One producer iteration (wait for a free slot, arm the stage's "full" barrier,
    // issue its boxes) occupies the issuing thread for ~600 cycles, mostly barrier
    // round trips, while further boxes in the same iteration cost ~100 each; several
    // producer threads in different warps multiply the rate.  So up to kProducers
    // threads take turns by stage: producer p issues every box of the iterations
    // g = p, p + P, p + 2P, ... of this CTA's (tile, k-block) sequence, g in stage
    // g mod S.  With P <= S the parity waits stay exact: before producer p reaches
    // iteration g the MMA has consumed everything up to g - P - S, so a slot's
    // barrier is never two phases behind its waiter.
    const int pi = warp == 0 ? 0 : warp - 5;           // producer index 0..2
    if (lane == 0 && pi < n_producers) {
      bool ok = true;
      // the j-th box of k-block kb: its shared-memory slot and coordinates
      auto issue_box = [&](int j, int kb, int m0, int nb0, uint32_t a_dst, uint32_t b_dst,
                           uint32_t fb, bool prefetch_only) {
        const int k0 = kb * BK;
        const CUtensorMap* map;
        uint32_t dst;
        int x, y, z = -1;                              // z >= 0: a 3-D box
        if (j < n_a_boxes) {
          map = &tmap_a;
          dst = a_dst;
          if (p.a3d) {
            if (!p.trans_a) { x = 0; y = m0; z = kb * kKChunks; }           // {chunk, 128, chunks}
            else { x = 0; y = k0; z = m0 / kChunkElems; }                     // {chunk, BK, 128/chunk}
          } else if (!p.trans_a) {
            dst += j * (kBM * 128u); x = k0 + kChunkElems * j; y = m0;        // {chunk K, 128 M}
          } else {
            dst += j * kMNChunkBytes; x = m0 + kChunkElems * j; y = k0;       // {chunk M, BK K}
          }
        } else {
          const int c = j - n_a_boxes;
          map = &tmap_b;
          dst = b_dst;
          if (p.b3d) {
            if (p.trans_b) { x = 0; y = nb0; z = kb * kKChunks; }           // {chunk, BN/CG, chunks}
            else { x = 0; y = k0; z = nb0 / kChunkElems; }                    // {chunk, BK, chunks}
          } else if (p.trans_b) {
            dst += c * (kBnCta * 128u); x = k0 + kChunkElems * c; y = nb0;    // {chunk K, BN/CG N}
          } else {
            dst += c * kMNChunkBytes; x = nb0 + kChunkElems * c; y = k0;      // {chunk N, BK K}
          }
        }
        if (z >= 0) {
          if (prefetch_only) tma_prefetch_l2_3d(map, x, y, z);
          else if (kPair) tma_load_3d_pair(dst, map, fb, x, y, z);
          else tma_load_3d(dst, map, fb, x, y, z);
        } else {
          if (prefetch_only) tma_prefetch_l2_2d(map, x, y);
          else if (kPair) tma_load_2d_pair(dst, map, fb, x, y);
          else tma_load_2d(dst, map, fb, x, y);
        }
      };
      // walk this unit's (tile, k-block) iterations g = 0, 1, ...; issue g = pi, pi + P, ...
      WorkIter work(p, cluster_id, n_clusters, krank);
      WorkItem w;
      int g = 0;
      while (ok && work.next(w)) {
        int mb, nb;
        tile_coords(w.tile, p.tiles_m, p.tiles_n, p.raster_group, mb, nb);
        const int m0 = mb * kBM * CG + static_cast<int>(rank) * kBM;    // this CTA's A rows
        const int nb0 = nb * BN + static_cast<int>(rank) * kBnCta;      // this CTA's B columns
        if (g == 0) grid_dependency_wait();
        for (int i = 0; i < w.n; ++i, ++g) {
          if (g % n_producers != pi) continue;
          const int kb = w.kb_at(i);
          const int stage = g % S;
          const uint32_t phase = static_cast<uint32_t>(g / S) & 1u;
          if (!wait_bounded<kPair>(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns)) {
            record_timeout(p.status, abort_flag, kSiteProducerEmpty);
            ok = false;
            break;
          }
          const uint32_t local_full = full_bar(stage);
          if (leader) mbar_arrive_expect_tx(local_full, (kAStageBytes + kBStage) * CG);
          const uint32_t fb = kPair ? mapa_shared(local_full, 0) : local_full;
          const uint32_t a_dst = sA + stage * kAStageBytes;
          const uint32_t b_dst = sB + stage * kBStage;
          for (int j = 0; j < n_boxes; ++j) issue_box(j, kb, m0, nb0, a_dst, b_dst, fb, false);
          if (leader) lap_armed[stage] = g / S;   // stage laps are armed in order
          // optional L2 prefetch of the k-block l2_prefetch iterations ahead (same item)
          if (p.l2_prefetch > 0 && i + p.l2_prefetch < w.n) {
            for (int j = 0; j < n_boxes; ++j)
              issue_box(j, w.kb_at(i + p.l2_prefetch), m0, nb0, 0, 0, 0, true);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer --
    grid_dependency_wait();
    if (lane == 0 && leader) {
      const uint32_t a_lbo = p.trans_a ? kMNChunkBytes : 16u;
      const uint32_t b_lbo = p.trans_b ? 16u : kMNChunkBytes;
      const uint64_t a_desc0 = smem_desc_sw128(sA, a_lbo, 1024u);
      const uint64_t b_desc0 = smem_desc_sw128(sB, b_lbo, 1024u);
      // Start-address offset of MMA k-step k (kMmaK elements = 32 bytes of K) within
      // a stage, in 16-byte descriptor units.  K-major: chunk k/4 of the stage, then
      // 32 B along the swizzled row; M/N-major: kMmaK rows of 128 B per step.
      auto k_off = [&](bool mn_major, uint32_t rows, int k) -> uint64_t {
        return mn_major ? (static_cast<uint64_t>(k) * kMmaK * 128u) >> 4
                        : (static_cast<uint64_t>(k / 4) * rows * 128u + (k % 4) * 32u) >> 4;
      };
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc = 0, acc_phase = 0;
      bool ok = true;
      if (p.stall) {
        // Nothing arrives on "done" before the MMA thread itself commits to it below, so
        // this wait can only run out: the timeout and unwind path under test.  It gets
        // half the limit, so that it runs out before the waits of the other roles, which
        // start at about the same time and wait for this thread's products.
        if (!wait_bounded<kPair>(done_bar, 0, abort_flag, p.timeout_ns / 2))
          record_timeout(p.status, abort_flag, kSiteInjected);
        ok = false;
      }
      WorkIter work(p, cluster_id, n_clusters, krank);
      WorkItem w;
      while (ok && work.next(w)) {
        if (!wait_bounded<kPair>(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
          record_timeout(p.status, abort_flag, kSiteMmaTmemEmpty);
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * kAccStride;
        for (int i = 0; i < w.n; ++i) {
          if (!wait_bounded<kPair>(full_bar(stage), phase, abort_flag, p.timeout_ns)) {
            record_timeout(p.status, abort_flag, kSiteMmaFull);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t a_desc = a_desc0 + ((stage * kAStageBytes) >> 4);
          const uint64_t b_desc = b_desc0 + ((stage * kBStage) >> 4);
#pragma unroll
          for (int k = 0; k < BK / kMmaK; ++k) {
            const uint32_t acc_in = (i != 0 || k != 0) ? 1u : 0u;   // the first overwrites
            const uint64_t ad = a_desc + k_off(p.trans_a, kBM, k);
            const uint64_t bd = b_desc + k_off(!p.trans_b, kBnCta, k);
            if constexpr (EB == 1) {
              if constexpr (kPair) mma_f8_ss_pair(d_tmem, ad, bd, p.idesc, acc_in);
              else mma_f8_ss(d_tmem, ad, bd, p.idesc, acc_in);
            } else {
              if constexpr (kPair) mma_f16_ss_pair(d_tmem, ad, bd, p.idesc, acc_in);
              else mma_f16_ss(d_tmem, ad, bd, p.idesc, acc_in);
            }
          }
          // frees the slot (in both CTAs) once these MMAs have read it
          if constexpr (kPair) mma_commit_pair(empty_bar(stage), 0x3);
          else mma_commit(empty_bar(stage));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // accumulator complete -> epilogue(s)
        if constexpr (kPair) mma_commit_pair(tfull_bar(acc), 0x3);
        else mma_commit(tfull_bar(acc));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // No MMA may still run when Tensor Memory is freed.
      if constexpr (kPair) mma_commit_pair(done_bar, 0x3);
      else mma_commit(done_bar);
      if (!wait_bounded<kPair>(done_bar, 0, nullptr, p.timeout_ns)) {
        record_timeout(p.status, abort_flag, kSiteDrain);
      }
    } else if (lane == 0 && kPair) {
      // odd CTA of a pair: its Tensor Memory is written by the even CTA's MMAs
      if (!wait_bounded<true>(done_bar, 0, nullptr, p.timeout_ns)) {
        record_timeout(p.status, abort_flag, kSiteDrain);
      }
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------- epilogue --
    grid_dependency_wait();
    const int q = warp & 3;                // Tensor Memory lane quadrant of this warp
    const int ew = warp - 2;               // staging-buffer owner index
    uint32_t acc = 0, acc_phase = 0;
    uint32_t sbuf = 0;
    uint32_t red_phase = 0;                // tiles exchanged so far, mod 2
    WorkIter work(p, cluster_id, n_clusters, krank);
    WorkItem w;
    while (work.next(w)) {
      int mb, nb;
      tile_coords(w.tile, p.tiles_m, p.tiles_n, p.raster_group, mb, nb);
      const int m0 = mb * kBM * CG + static_cast<int>(rank) * kBM;
      const int n0 = nb * BN;
      WorkIter peek = work;
      WorkItem w_next;
      const bool last_item = !peek.next(w_next);
      const bool helped = kHelpable && n_producers == kProducers && last_item && !ksplit &&
                          !p.c_trans && p.tma_store && w.k0 == 0 && w.k1 == p.k_blocks;
      // Stream-K roles: a partial item that starts mid-tile stores its sum for the
      // tile's finisher; an item that starts at k-block 0 but ends early is the
      // finisher and adds the partials of units cluster_id + 1 .. v_end - 1.
      const bool store_partial = !ksplit && w.k0 > 0;
      int v_end = cluster_id + 1;
      if (!ksplit && w.k0 == 0 && w.k1 < p.k_blocks) {
        const int64_t tile_end = static_cast<int64_t>(w.tile - p.dp_tiles + 1) * p.k_blocks;
        while (v_end < n_clusters && sk_begin(p, v_end, n_clusters) < tile_end) ++v_end;
      }
      const int slot_q = (static_cast<int>(rank) * 4 + q);     // this warp's slot in a unit
      // lane-major groups of four columns: one 16-byte access per lane per group, and
      // the warp's 32 lanes cover 512 contiguous bytes
      auto partial4_at = [&](int unit, int col4) -> float4* {
        return reinterpret_cast<float4*>(p.sk_partials) +
               ((static_cast<int64_t>(unit) * CG * 4 + slot_q) * (BN / 4) + col4) * 32 + lane;
      };
      auto flag_at = [&](int unit) -> unsigned long long* {
        return p.sk_flags + static_cast<int64_t>(unit) * CG * 4 + slot_q;
      };
      // units with an empty share of the split store nothing
      auto contributes = [&](int v) {
        return sk_begin(p, v, n_clusters) < sk_begin(p, v + 1, n_clusters);
      };
      // contributors' partials must be stored before they are read
      if (v_end > cluster_id + 1) {
        bool ok_sk = true;
        if (lane == 0) {
          for (int v = cluster_id + 1; v < v_end && ok_sk; ++v) {
            if (!contributes(v)) continue;
            const uint64_t t0 = clock_cycles();
            while (ld_acquire_gpu_u64(flag_at(v)) != p.sk_token) {
              if (clock_cycles() - t0 > p.timeout_ns * 4u || *abort_flag) { ok_sk = false; break; }
            }
          }
          if (!ok_sk && !*abort_flag) record_timeout(p.status, abort_flag, kSiteStreamK);
        }
        __syncwarp();
        // every lane acquires the flags it relies on before reading the partials
        for (int v = cluster_id + 1; v < v_end; ++v)
          if (contributes(v)) (void)ld_acquire_gpu_u64(flag_at(v));
      }
      // one lane waits, the warp follows its verdict.  (A try_wait with a suspend-time
      // hint was measured to wake microseconds after the phase completed: plain polls
      // by one lane per warp cost less.)
      bool ready = true;
      if (lane == 0)
        ready = wait_bounded<kPair>(tfull_bar(acc), acc_phase, abort_flag, p.timeout_ns);
      __syncwarp();
      if (!__shfl_sync(0xFFFFFFFFu, ready ? 1 : 0, 0)) {
        if (lane == 0 && !*abort_flag) record_timeout(p.status, abort_flag, kSiteEpiTmemFull);
        break;
      }
      tc_fence_after_sync();
      const uint32_t t_row =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccStride;
      // The whole accumulator is in registers: hand the buffer back to the MMA.  Lane 31
      // arrives: lane 0 issues the warp's bulk stores, and an arrive with release
      // semantics from it was measured to wait ~2,400 cycles behind them (CTA pairs).
      auto release_acc = [&]() {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 31) {
          if constexpr (kPair) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
          else mbar_arrive(tempty_bar(acc));
        }
      };
      // One epilogue step: W columns starting at column c_col of the tile, in v.
      auto finish_chunk = [&](auto width, uint32_t* v, int c_col) {
        constexpr int W = decltype(width)::value;
        if (store_partial) {
          // fp32 partial sum, four columns per 16-byte store
#pragma unroll
          for (int j = 0; j < W / 4; ++j)
            __stcg(partial4_at(cluster_id, c_col / 4 + j),
                   make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                               __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
          return;
        }
        // finisher: add the later k-blocks' partials, in unit order
        for (int u2 = cluster_id + 1; u2 < v_end; ++u2) {
          if (!contributes(u2)) continue;
#pragma unroll
          for (int j = 0; j < W / 4; ++j) {
            const float4 t = __ldcg(partial4_at(u2, c_col / 4 + j));
            v[4 * j] = __float_as_uint(__uint_as_float(v[4 * j]) + t.x);
            v[4 * j + 1] = __float_as_uint(__uint_as_float(v[4 * j + 1]) + t.y);
            v[4 * j + 2] = __float_as_uint(__uint_as_float(v[4 * j + 2]) + t.z);
            v[4 * j + 3] = __float_as_uint(__uint_as_float(v[4 * j + 3]) + t.w);
          }
        }
        if (p.scale) {
#pragma unroll
          for (int j = 0; j < W; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * p.alpha);
        }
        uint32_t packed[W / 2];
        pack_chunk<W / 2>(v, packed, p.bf16, p.relu);
        const int row = m0 + q * 32 + lane;      // this lane's row of the kernel's tile
        const int col0 = n0 + c_col;
        if (p.c_trans && p.c_vec) {
          // The kernel computed C^T: its row `row` is column `row` of C, and each of its
          // columns is a row of C.  Each 8 x 8 block (8 lanes x 8 columns) is transposed
          // across its lanes by shuffles, so that lane 8g + r then holds 8 consecutive
          // columns of C row col0 + 8b + r and writes them as one 16-byte store (one
          // 2-byte store per element was measured ~100 cycles per warp instruction).
          const int r = lane & 7;
          const int cn = m0 + q * 32 + 8 * (lane >> 3);       // first C column of the lane
#pragma unroll
          for (int b = 0; b < W / 8; ++b) {
            uint32_t w0 = packed[4 * b], w1 = packed[4 * b + 1];
            uint32_t w2 = packed[4 * b + 2], w3 = packed[4 * b + 3];
            transpose8x8_u16(w0, w1, w2, w3, r);
            const int cm = col0 + 8 * b + r;                    // C row
            if (cm < p.N && cn < p.M) {
              uint16_t* dst = reinterpret_cast<uint16_t*>(p.C) + static_cast<int64_t>(cm) * p.ldc + cn;
              if (cn + 8 <= p.M) {
                *reinterpret_cast<uint4*>(dst) = make_uint4(w0, w1, w2, w3);
              } else {
                const uint32_t wv[4] = {w0, w1, w2, w3};
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  if (cn + e < p.M) dst[e] = static_cast<uint16_t>(wv[e >> 1] >> (16 * (e & 1)));
              }
            }
          }
          return;
        }
        if (p.c_trans) {
          // The kernel computed C^T: its row `row` is column `row` of C, and each of
          // its columns is a row of C that the warp's 32 lanes write as 64 contiguous
          // bytes.
          if (row < p.M) {
            uint16_t* ccol = reinterpret_cast<uint16_t*>(p.C) + row;
#pragma unroll
            for (int j = 0; j < W / 2; ++j) {
              const int col = col0 + 2 * j;
              if (col < p.N) ccol[static_cast<int64_t>(col) * p.ldc] = static_cast<uint16_t>(packed[j] & 0xFFFFu);
              if (col + 1 < p.N) ccol[static_cast<int64_t>(col + 1) * p.ldc] = static_cast<uint16_t>(packed[j] >> 16);
            }
          }
          return;
        }
        if constexpr (W == kChunk) {
          if (p.tma_store) {
            stage_and_store_chunk(&tmap_c, sC + (ew * 2 + sbuf) * 4096u, packed, lane, col0,
                                  m0 + q * 32, m0 + q * 32 < p.M && col0 < p.N);
            sbuf ^= 1u;
            return;
          }
        }
        if (row < p.M) {
          uint16_t* crow = reinterpret_cast<uint16_t*>(p.C) + static_cast<int64_t>(row) * p.ldc;
          if (p.c_vec && col0 + W <= p.N) {
            // the lane's W values are 2 W contiguous bytes of its row of C
            uint4* dst = reinterpret_cast<uint4*>(crow + col0);
#pragma unroll
            for (int j = 0; j < W / 8; ++j)
              dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2],
                                  packed[4 * j + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < W / 2; ++j) {
              const int col = col0 + 2 * j;
              if (col < p.N) crow[col] = static_cast<uint16_t>(packed[j] & 0xFFFFu);
              if (col + 1 < p.N) crow[col + 1] = static_cast<uint16_t>(packed[j] >> 16);
            }
          }
        }
      };
      if constexpr (kColumnSplit) {
        if (ksplit) {
          // Cluster split-K: CTA r finishes columns [r H, (r + 1) H) of every row of the
          // tile (H = BN / 2).  Each warp first writes its rows' partial sums of the
          // peer's columns into the peer's receive buffer (once the peer has read the
          // previous tile's) and announces them; then it waits for the peer's partial
          // sums of its own columns, adds them to its own and finishes those columns.
          // All four warps of both CTAs share the work.  Every lane waits and arrives
          // itself where it orders its own accesses.
          constexpr int kHW = BN / 2;
          constexpr int kHC = kHW < kChunk ? kHW : kChunk;   // columns per step
          constexpr int kHN = kHW / kHC;
          const uint32_t peer = krank ^ 1u;
          // entry (column group j of the warp's half, lane): 16 bytes, lane-major, so a
          // warp's access covers 512 contiguous bytes
          const uint32_t my_entry = sRed + static_cast<uint32_t>(q * (kHW / 4) * 32 + lane) * 16u;
          const uint32_t peer_entry = mapa_shared(my_entry, peer);
          bool split_ok = wait_bounded<true>(red_empty_bar(q), red_phase ^ 1u, abort_flag, p.timeout_ns);
          if (__all_sync(0xFFFFFFFFu, split_ok)) {
#pragma unroll 1
            for (int h = 0; h < kHN; ++h) {
              uint32_t v[kHC];
              tmem_load_cols<kHC>(t_row + peer * kHW + h * kHC, v);
              tmem_load_wait();
#pragma unroll
              for (int j = 0; j < kHC / 4; ++j)
                st_cluster_v4(peer_entry + static_cast<uint32_t>(h * (kHC / 4) + j) * 512u,
                              v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            }
            // release: this lane's stores into the peer come first
            mbar_arrive_cluster(mapa_shared(red_full_bar(q), peer));
            split_ok = wait_bounded<true>(red_full_bar(q), red_phase, abort_flag, p.timeout_ns);
          }
          if (!__all_sync(0xFFFFFFFFu, split_ok)) {
            if (lane == 0 && !*abort_flag) record_timeout(p.status, abort_flag, kSiteClusterSplit);
            break;
          }
#pragma unroll 1
          for (int h = 0; h < kHN; ++h) {
            uint32_t v[kHC];
            tmem_load_cols<kHC>(t_row + krank * kHW + h * kHC, v);
            tmem_load_wait();
            if (h == kHN - 1) release_acc();
            // own partial + the peer's: one IEEE addition per element, so the sum does
            // not depend on which CTA finishes the column
#pragma unroll
            for (int j = 0; j < kHC / 4; ++j) {
              const float4 t = ld_shared_f4(my_entry + static_cast<uint32_t>(h * (kHC / 4) + j) * 512u);
              v[4 * j] = __float_as_uint(__uint_as_float(v[4 * j]) + t.x);
              v[4 * j + 1] = __float_as_uint(__uint_as_float(v[4 * j + 1]) + t.y);
              v[4 * j + 2] = __float_as_uint(__uint_as_float(v[4 * j + 2]) + t.z);
              v[4 * j + 3] = __float_as_uint(__uint_as_float(v[4 * j + 3]) + t.w);
            }
            finish_chunk(IntConst<kHC>{}, v, static_cast<int>(krank) * kHW + h * kHC);
          }
          // the buffer is read (every lane, then the warp barrier): the peer may write
          // the next tile's partial sums.  Lane 31 arrives, as for the accumulator.
          // After the pair's last tile nothing more is sent, and the hand-back (whose
          // release waits for this warp's stores of C) is left out: 1 % per call on
          // the skinny products.
          if (!last_item) {
            __syncwarp();
            if (lane == 31) mbar_arrive_cluster(mapa_shared(red_empty_bar(q), peer));
          }
          red_phase ^= 1u;
        }
      }
#pragma unroll 1
      for (int c = 0; c < (helped ? kHelpC : kFull) && !(kColumnSplit && ksplit); ++c) {
        uint32_t v[kEC];
        if constexpr (kEC == 16) {
          tmem_load_16cols(t_row + c * kEC, v);
        } else {
#pragma unroll
          for (int h = 0; h < kEC / 32; ++h)
            tmem_load_32cols(t_row + c * kEC + 32 * h,
                             *reinterpret_cast<uint32_t(*)[32]>(&v[32 * h]));
        }
        tmem_load_wait();
        if (kTail == 0 && c == kFull - 1) release_acc();
        finish_chunk(IntConst<kEC>{}, v, c * kEC);
      }
      if constexpr (kTail > 0) {
        if (!helped) {
          uint32_t v[32];
          tmem_load_32cols(t_row + kFull * kEC, v);
          tmem_load_wait();
          release_acc();
          finish_chunk(IntConst<32>{}, v, kFull * kEC);
        }
      }
      if (store_partial) {
        // the warp's partial stores happen before lane 0's fence (warp barrier); the
        // GPU-scope fence and release store make all of them visible before the flag
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          st_release_gpu_u64(flag_at(cluster_id), p.sk_token);
        }
      } else if (v_end > cluster_id + 1) {
        __syncwarp();                     // all lanes have read the partials: reset flags
        if (lane == 0)
          for (int u2 = cluster_id + 1; u2 < v_end; ++u2)
            if (contributes(u2)) *flag_at(u2) = 0ull;
      }
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    // the staging buffers must stay valid until the bulk stores have read them; the
    // global writes themselves complete before the grid is reported finished
    if (p.tma_store && lane == 0) bulk_wait_group_read<0>();
  }

  if constexpr (kHelpable) {
    // (only when warps 6 and 7 are producers too: then every helping warp reaches this
    // point within a few stages of the last MMA, and the wait below stays short)
    if ((warp <= 1 || warp >= 6) && n_producers == kProducers && !ksplit && !p.c_trans &&
        p.tma_store) {
      // ------------------------------------------- the last tile's other half --
      // The same walk as every role: the CTA's last item and its accumulator.  This warp
      // waits for the MMA thread's final commit ("done", one phase only: a parity wait
      // on the accumulator's own barrier could match an earlier tile's phase when the
      // warp gets here early).  Every MMA is then done, so the ring is idle and its first
      // 32 KB hold this warp's two staging buffers.
      WorkIter it(p, cluster_id, n_clusters, krank);
      WorkItem wl;
      int n_items = 0;
      while (it.next(wl)) ++n_items;
      if (n_items > 0 && wl.k0 == 0 && wl.k1 == p.k_blocks) {
        const uint32_t acc = static_cast<uint32_t>(n_items - 1) & 1u;
        bool ready = true;
        if (lane == 0)
          ready = wait_bounded<kPair>(done_bar, 0, abort_flag, p.timeout_ns) && !*abort_flag;
        __syncwarp();
        if (__shfl_sync(0xFFFFFFFFu, ready ? 1 : 0, 0)) {
          tc_fence_after_sync();
          int mb, nb;
          tile_coords(wl.tile, p.tiles_m, p.tiles_n, p.raster_group, mb, nb);
          const int q = warp & 3;
          const int m0 = mb * kBM * CG + static_cast<int>(rank) * kBM;
          const int n0 = nb * BN;
          const int hw = warp <= 1 ? warp : warp - 4;        // 0..3: staging owner
          const uint32_t t_row =
              tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccStride;
          uint32_t sbuf = 0;
#pragma unroll 1
          for (int c = kHelpC; c < kFull; ++c) {
            uint32_t v[kChunk];
#pragma unroll
            for (int h = 0; h < kChunk / 32; ++h)
              tmem_load_32cols(t_row + c * kChunk + 32 * h,
                               *reinterpret_cast<uint32_t(*)[32]>(&v[32 * h]));
            tmem_load_wait();
            if (p.scale) {
#pragma unroll
              for (int j = 0; j < kChunk; ++j)
                v[j] = __float_as_uint(__uint_as_float(v[j]) * p.alpha);
            }
            uint32_t packed[kChunk / 2];
            pack_chunk<kChunk / 2>(v, packed, p.bf16, p.relu);
            const int col0 = n0 + c * kChunk;
            stage_and_store_chunk(&tmap_c, sA + static_cast<uint32_t>(hw * 2 + sbuf) * 4096u,
                                  packed, lane, col0, m0 + q * 32,
                                  m0 + q * 32 < p.M && col0 < p.N);
            sbuf ^= 1u;
          }
          if constexpr (kTail > 0) {
            // the 32-column tail by plain stores, as in the epilogue warps
            uint32_t v[32];
            tmem_load_32cols(t_row + kFull * kChunk, v);
            tmem_load_wait();
            if (p.scale) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                v[j] = __float_as_uint(__uint_as_float(v[j]) * p.alpha);
            }
            uint32_t packed[16];
            pack_chunk<16>(v, packed, p.bf16, p.relu);
            const int row = m0 + q * 32 + lane;
            const int col0 = n0 + kFull * kChunk;
            if (row < p.M) {
              uint16_t* crow = reinterpret_cast<uint16_t*>(p.C) + static_cast<int64_t>(row) * p.ldc;
              if (p.c_vec && col0 + 32 <= p.N) {
                uint4* dst = reinterpret_cast<uint4*>(crow + col0);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2],
                                      packed[4 * j + 3]);
              } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  const int col = col0 + 2 * j;
                  if (col < p.N) crow[col] = static_cast<uint16_t>(packed[j] & 0xFFFFu);
                  if (col + 1 < p.N) crow[col + 1] = static_cast<uint16_t>(packed[j] >> 16);
                }
              }
            }
          }
          if (lane == 0) bulk_wait_group_read<0>();   // the staging is read before exit
        } else if (lane == 0 && !*abort_flag) {
          record_timeout(p.status, abort_flag, kSiteEpiTmemFull);
        }
      }
    }
  }

  // ------------------------------------------------------------------ teardown --
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  // Every load a producer issued must have landed before the CTA may exit.  All roles
  // are done, so the last armed lap of each stage is final and its phase parity is
  // unambiguous.  In a normal run the MMA thread consumed every stage and these waits
  // return at once.  (The even CTA's barriers also cover the odd CTA's loads.)
  if (threadIdx.x == 0 && leader) {
    for (int st = 0; st < S; ++st) {
      const int lap = lap_armed[st];
      if (lap >= 0 && !wait_bounded<kPair>(full_bar(st), static_cast<uint32_t>(lap) & 1u,
                                           nullptr, p.timeout_ns)) {
        record_timeout(p.status, abort_flag, kSiteDrain);
      }
    }
  }
  __syncthreads();
  if (kPair || ksplit) {
    // No CTA leaves while its peer may still touch it.  After a timeout in either CTA
    // (any role, or the drain above) copies still in flight may complete on the other
    // CTA's barriers or in its shared memory, and the odd CTA of a pair cannot see its
    // own loads land: each CTA tells the other whether it gave up, and if either did,
    // both wait out a grace period before they exit.  (The output is then undefined.)
    // (Both CTAs read the same "either gave up" after the barrier, so both or neither
    // take the pause and its second barrier.)
    if (threadIdx.x == 0)
      st_cluster_u32(mapa_shared(peer_abort_addr, cluster_ctarank() ^ 1u), *abort_flag);
    cluster_sync_all();
    if (*abort_flag != 0u || *peer_abort != 0u) {
      if (threadIdx.x == 0) {
        const uint64_t t0 = clock_cycles();
        while (clock_cycles() - t0 < 800000ull) __nanosleep(1000);   // >= 200 us
      }
      __syncthreads();
      cluster_sync_all();
    }
  }
  tc_fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    if constexpr (kPair) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

// C = epi(0) for K == 0 (no Tensor Memory involved).
__global__ void tl_fill_zero_kernel(uint16_t* C, int64_t M, int64_t N, int64_t ldc) {
  const int64_t total = M * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / N;
    const int64_t c = i - r * N;
    C[r * ldc + c] = 0;
  }
}

// Copy a rows x cols matrix of 1- or 2-byte elements from pitch `sp` to pitch `dp`
// (elements), used to give an operand a 16-byte-aligned pitch for the TMA unit.
template <typename T>
__global__ void tl_repack_kernel(const T* __restrict__ src, T* __restrict__ dst, int64_t rows,
                                 int64_t cols, int64_t sp, int64_t dp) {
  constexpr int64_t kPer = 8 / sizeof(T);           // elements per 8-byte unit
  const bool wide = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 7u) == 0 &&
                    (sp % kPer) == 0 && (dp % kPer) == 0 && (cols % kPer) == 0;
  if (wide) {
    const int64_t units = cols / kPer;               // 8-byte units per row
    const int64_t total = rows * units;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      const int64_t r = i / units;
      const int64_t u = i - r * units;
      const uint2 v = *reinterpret_cast<const uint2*>(src + r * sp + kPer * u);
      *reinterpret_cast<uint2*>(dst + r * dp + kPer * u) = v;
    }
  } else {
    const int64_t total = rows * cols;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      const int64_t r = i / cols;
      const int64_t c = i - r * cols;
      dst[r * dp + c] = src[r * sp + c];
    }
  }
}

}  // namespace tl
