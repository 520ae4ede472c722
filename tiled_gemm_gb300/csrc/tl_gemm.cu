// tl_gemm.cu -- host side of the C ABI declared in include/tl_gemm.h: argument
// checks, the tile planner, TMA descriptor encoding and the kernel launches.
//
// The call path mirrors the pages' host wrapper ("NVIDIA backend codegen" page,
// section 4.2.2: set the dynamic shared-memory attribute, encode one CUtensorMap
// per TMA operand with cuTensorMapEncodeTiled, launch with cudaLaunchKernelEx) and
// its generated host checks ("TileLang: from tile dataflow to controllable AI
// kernels", section "automatically generated host checks": null pointers, shapes,
// strides, device ids), but is written directly in C++ with no JIT in between.
// TMA eligibility follows the rule the pages give for bulk copies: the innermost
// stride is 1 and every other stride is a multiple of 16 bytes ("NVIDIA backend
// codegen" page, section 4.4.2).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdint>
#include <cstddef>
#include <cstring>
#include <mutex>
#include <random>
#include <unordered_map>

#include "attn_kernel.cuh"
#include "gemm_kernel.cuh"
#include "mx_kernel.cuh"
#include "tl_gemm.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxSmemPerCta = 232448;   // 227 KB opt-in per CTA on sm_100-class parts
constexpr int kDefaultSms = 152;         // GB300 (two dies of 76), when no device is asked

__device__ uint32_t g_status_word;           // bounded-wait outcome, see tl_device_status

std::atomic<uint64_t> g_timeout_ns{1000000000ull};
std::atomic<int> g_stall{0};                 // test hook, see tl_debug_set_stall

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  std::once_flag once;
  bool ok = false;
  bool sm103 = false;
  int sms = 0;
  int smem_optin = 0;                        // max dynamic shared memory per CTA
  uint32_t* status = nullptr;
  std::atomic<uint64_t> attr_done{0};        // bit i: smem attribute set for kernel i
  int max_units[64] = {};                    // resident CTAs (pairs) per kernel
  int max_clusters2[64] = {};                // resident clusters of two per kernel
  std::mutex mu;
};

DeviceState g_dev[kMaxDevices];
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  });
  return g_encode;
}

DeviceState* device_state(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceState& st = g_dev[dev];
  std::call_once(st.once, [&st, dev] {
    int major = 0, minor = 0, sms = 0, optin = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
      return;
    }
    st.sm103 = (major == 10 && minor == 3);
    st.sms = sms;
    st.smem_optin = std::min<int>(optin, static_cast<int>(kMaxSmemPerCta));
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return;
    st.status = static_cast<uint32_t*>(addr);
    st.ok = true;
  });
  if (dev_out) *dev_out = dev;
  return st.ok ? &st : nullptr;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool is_fp8(tl_dtype t) { return t == TL_E4M3 || t == TL_E5M2; }
int elem_bytes(tl_dtype t) { return is_fp8(t) ? 1 : 2; }

// The element types of one call: operands of `eb` bytes in formats a_fmt / b_fmt (the
// MMA's format codes), output `out` (fp16 or bf16), and the product scale alpha.
struct Types {
  int eb;
  tl_dtype a_type, b_type, out;
  float alpha;
  bool scale;
};

Types types_16(tl_dtype dtype) { return Types{2, dtype, dtype, dtype, 1.0f, false}; }

bool tma_ok(const void* p, int64_t ld, int eb = 2) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && ((ld * eb) & 15) == 0;
}

// Byte extent [lo, hi) touched by a rows x cols matrix with leading dimension ld.
void extent(const void* p, int64_t rows, int64_t cols, int64_t ld, uintptr_t* lo, uintptr_t* hi,
            int eb = 2) {
  *lo = reinterpret_cast<uintptr_t>(p);
  *hi = *lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * eb);
}

bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

tl_status check_device_pointer(const void* p, int dev) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_DEVICE;
  }
  if ((attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) ||
      attr.device != dev) {
    return TL_ERR_DEVICE;
  }
  return TL_OK;
}

// bm = 128: one CTA per 128 x bn tile.  bm = 256: a CTA pair (cluster of 2,
// cta_group::2 MMAs) per 256 x bn tile, each CTA holding half of B's columns.
// Narrow tiles (bn 16 or 32, for skinny products) come with 128-deep stages only.
// 8-bit operands (eb = 1): bk 128 or 256 (one or two 128-byte chunks), bn >= 64, no
// operand swap.
bool plan_supported(const tl_plan& pl, int eb = 2) {
  if (eb == 1) {
    const bool bn8 = (pl.bm == 128 && (pl.bn == 64 || pl.bn == 128 || pl.bn == 256)) ||
                     (pl.bm == 256 && (pl.bn == 128 || pl.bn == 256));
    return bn8 && (pl.bk == 128 || pl.bk == 256) && pl.stages >= 2 && pl.stages <= 8 &&
           pl.raster_group >= 1 && pl.grid >= 0 && pl.swap_ab == 0;
  }
  const bool narrow = pl.bm == 128 && (pl.bn == 16 || pl.bn == 32) && pl.bk == 128;
  // 192 and 224 columns (not a power of two): 128-deep stages, K-major B (narrow_ok)
  const bool odd = (pl.bm == 128 || pl.bm == 256) && (pl.bn == 192 || pl.bn == 224) &&
                   pl.bk == 128;
  const bool bn_ok = narrow || odd ||
                     (pl.bm == 128 && (pl.bn == 64 || pl.bn == 128 || pl.bn == 256)) ||
                     (pl.bm == 256 && (pl.bn == 128 || pl.bn == 256));
  return bn_ok && (pl.bk == 64 || pl.bk == 128) && pl.stages >= 2 && pl.stages <= 8 &&
         pl.raster_group >= 1 && pl.grid >= 0 && (pl.swap_ab == 0 || pl.swap_ab == 1);
}

// Narrow tiles read B in 64-element K chunks of bn rows: the kernel's B operand must
// be K-major.  With swap_ab the kernel's B is A, K-major when A is not transposed.
// 8-bit operands: an N-major B is read in boxes 128 elements wide, so each CTA's share
// of the tile's columns (bn / cg) must be a multiple of 128.
// Tiles of 192 or 224 columns also need a K-major B: an N-major B is loaded in boxes of
// 64 columns, which must tile each CTA's share of the tile.
bool narrow_ok(const tl_plan& pl, int trans_a, int trans_b, int eb = 2) {
  if (eb == 1) return trans_b == 1 || (pl.bn / (pl.bm / 128)) % 128 == 0;
  if (pl.bn >= 64 && pl.bn != 192 && pl.bn != 224) return true;
  return pl.swap_ab ? trans_a == 0 : trans_b == 1;
}

template <int BK, int EB>
uint32_t smem_for_bk(int bm, int bn, int stages, int ks, bool stg) {
  if constexpr (BK == 128 && EB == 2) {
    if (bn == 192) return bm == 256 ? tl::smem_bytes_for<192, 2, BK>(stages, 1, stg)
                                    : tl::smem_bytes_for<192, 1, BK>(stages, ks, stg);
    if (bn == 224) return bm == 256 ? tl::smem_bytes_for<224, 2, BK>(stages, 1, stg)
                                    : tl::smem_bytes_for<224, 1, BK>(stages, ks, stg);
  }
  if (bm == 256) {
    return bn == 128 ? tl::smem_bytes_for<128, 2, BK, EB>(stages, 1, stg)
                     : tl::smem_bytes_for<256, 2, BK, EB>(stages, 1, stg);
  }
  if constexpr (BK == 128 && EB == 2) {
    if (bn == 16) return tl::smem_bytes_for<16, 1, BK>(stages, ks, stg);
    if (bn == 32) return tl::smem_bytes_for<32, 1, BK>(stages, ks, stg);
  }
  switch (bn) {
    case 64: return tl::smem_bytes_for<64, 1, BK, EB>(stages, ks, stg);
    case 128: return tl::smem_bytes_for<128, 1, BK, EB>(stages, ks, stg);
    default: return tl::smem_bytes_for<256, 1, BK, EB>(stages, ks, stg);
  }
}

// Dynamic shared memory of one CTA; ks = 2 adds cluster split-K's receive buffer, and a
// plan that computes C^T (swap_ab, plain stores of C) has no TMA-store staging.
uint32_t smem_for(int bm, int bn, int bk, int stages, int eb = 2, int ks = 1, bool stg = true) {
  if (eb == 1) {
    return bk == 256 ? smem_for_bk<256, 1>(bm, bn, stages, ks, stg)
                     : smem_for_bk<128, 1>(bm, bn, stages, ks, stg);
  }
  return bk == 128 ? smem_for_bk<128, 2>(bm, bn, stages, ks, stg)
                   : smem_for_bk<64, 2>(bm, bn, stages, ks, stg);
}

tl_status validate_common(int64_t M, int64_t N, int64_t K, tl_dtype dtype, int trans_a,
                          int trans_b) {
  if (M < 0 || N < 0 || K < 0) return TL_ERR_INVALID_ARG;
  if (dtype != TL_F16 && dtype != TL_BF16 && !is_fp8(dtype)) return TL_ERR_INVALID_ARG;
  if ((trans_a != 0 && trans_a != 1) || (trans_b != 0 && trans_b != 1)) return TL_ERR_INVALID_ARG;
  // coordinates and tile counts are 32-bit inside the kernel
  if (M > (int64_t{1} << 31) - 256 || N > (int64_t{1} << 31) - 256 ||
      K > (int64_t{1} << 31) - 256) {
    return TL_ERR_UNSUPPORTED;
  }
  return TL_OK;
}

// Default L2 prefetch distance: off.  Measured on GB300 it did not shorten the
// latency-bound short-K shapes (their ring refills mostly hit L2 already) and it
// slowed the long ones; the plan field keeps it available for tuning.
int default_prefetch(const tl_plan& pl) {
  (void)pl;
  return 0;
}

// Work split over `units` persistent units.  Whole waves of tiles run data-parallel;
// when the tiles do not fill the last wave, the last full wave and the remainder are
// split by k-block evenly over all units (stream-K) if that shortens the critical
// path enough: data-parallel takes ceil(T/U) tile-lengths; the split takes (T_dp/U)
// tile-lengths plus ceil(iterations/U) k-blocks plus the fix-up.  Measured on GB300
// the fix-up (storing an fp32 partial tile, publishing it, the finisher reading it)
// costs ~6,000 SM cycles, i.e. fixup_kb k-blocks of about max(600, MMA cycles) each --
// so short tiles stay whole.  Under the power cap the split also raises the clock-
// limited work, hence the 0.87 margin.
//
// With cluster split-K (ksplit = 2) a unit is a cluster of two CTAs that share each of its
// whole tiles' k-blocks; nothing else is split.
void schedule(tl_plan* pl, int64_t units_avail, bool allow_split, int eb = 2) {
  const int cg = pl->bm / 128;
  const int ks = std::max(1, pl->ksplit);
  const int64_t units = std::max<int64_t>(1, units_avail);
  const int64_t T = pl->tiles, KI = pl->k_blocks;
  int64_t dp = T, iters = 0;
  if (ks == 1 && allow_split && pl->stream_k >= 0 && units > 1 && KI >= 2) {
    const int64_t full = T / units, rem = T % units;
    if (rem != 0 || pl->stream_k == 1) {
      const int64_t dp_try = full >= 1 ? (full - 1) * units : 0;
      const int64_t it = (T - dp_try) * KI;
      // per SM and k-block: 32 bytes of K per MMA step, bn/256 x 128 cycles each
      const double mma_cycles = static_cast<double>(pl->bn) * pl->bk * eb / 64.0;
      const double fixup_kb = 6000.0 / std::max(600.0, 1.1 * mma_cycles);
      const double t_dp = static_cast<double>(ceil_div(T, units) * KI);
      const double t_sk =
          static_cast<double>((dp_try / units) * KI + ceil_div(it, units)) + fixup_kb;
      if (pl->stream_k == 1 || t_sk < 0.87 * t_dp) {
        dp = dp_try;
        iters = it;
      }
    }
  }
  pl->dp_tiles = static_cast<int32_t>(dp);
  pl->sk_iters = iters;
  pl->grid = static_cast<int32_t>(cg * ks * (iters > 0 ? units : std::min<int64_t>(units, T)));
}

// Cluster split-K for one-CTA tiles: when at most half the SMs would hold a tile and the
// k-loop is long enough to halve, two CTAs of a cluster share each tile's k-blocks.  The
// quickstart 1024^3 tiling (64 tiles of 128 x 128, 16 k-blocks of 64) is bound by the
// latency of its 3-stage ring refills: split, each tile has two rings' loads in flight,
// and each CTA finishes half the tile's columns after a 32 KB exchange of partial sums
// with its peer through distributed shared memory.  The halves need a power-of-two
// tile width.
bool pow2_width(int bn) { return (bn & (bn - 1)) == 0; }

int auto_ksplit(const tl_plan& pl, int sms, int eb) {
  if (pl.bm != 128 || !pow2_width(pl.bn) || pl.stream_k == 1 || 2 * pl.tiles > sms ||
      pl.k_blocks < 4)
    return 1;
  // the receive buffer (128 x bn fp32) must fit beside the ring
  return smem_for(pl.bm, pl.bn, pl.bk, pl.stages, eb, 2, !pl.swap_ab) <= kMaxSmemPerCta ? 2 : 1;
}

// fp32 partial-sum slots (one 128 x bn tile per CTA) and ready flags (one per epilogue
// warp of each CTA) for a split over grid / cg units.
int64_t split_workspace_bytes(const tl_plan& pl) {
  if (pl.sk_iters == 0) return 0;
  return static_cast<int64_t>(pl.grid) * 128 * pl.bn * 4 + static_cast<int64_t>(pl.grid) * 4 * 8;
}

tl_status complete_plan(int64_t M, int64_t N, int64_t K, int trans_a, int trans_b, int num_sms,
                        tl_plan* pl, int eb = 2) {
  if (!plan_supported(*pl, eb) || !narrow_ok(*pl, trans_a, trans_b, eb)) return TL_ERR_INVALID_ARG;
  const int sms = num_sms > 0 ? num_sms : kDefaultSms;
  const int cg = pl->bm / 128;                       // CTAs per tile
  if (pl->swap_ab) std::swap(M, N);                  // the kernel computes C^T
  pl->tiles_m = ceil_div(M, pl->bm);
  pl->tiles_n = ceil_div(N, pl->bn);
  pl->tiles = pl->tiles_m * pl->tiles_n;
  pl->k_blocks = ceil_div(K, pl->bk);
  // per CTA: 128 rows of A and bn/cg columns of B per stage
  pl->ring_bytes =
      static_cast<int64_t>(pl->stages) * (128 * pl->bk + (pl->bn / cg) * pl->bk) * eb;
  // cluster split-K: 0 automatic, 1 off, 2 on (one-CTA tiles of a power-of-two width,
  // at least 2 k-blocks, and not with a forced stream-K split)
  if (pl->ksplit < 0 || pl->ksplit > 2) return TL_ERR_INVALID_ARG;
  if (pl->ksplit == 0) pl->ksplit = auto_ksplit(*pl, sms, eb);
  if (pl->ksplit == 2 &&
      (pl->bm != 128 || !pow2_width(pl->bn) || pl->k_blocks < 2 || pl->stream_k == 1))
    return TL_ERR_INVALID_ARG;
  pl->smem_bytes = smem_for(pl->bm, pl->bn, pl->bk, pl->stages, eb, pl->ksplit, !pl->swap_ab);
  if (pl->smem_bytes > kMaxSmemPerCta) return TL_ERR_INVALID_ARG;
  // two accumulators; 192- and 224-column tiles keep the second at column 256
  pl->tmem_cols = (pl->bn == 192 || pl->bn == 224) ? 512 : std::max(32, 2 * pl->bn);
  pl->tma_store = (!pl->swap_ab && pl->bn >= 64) ? 1 : 0;   // for a 16-byte aligned C
  pl->repack_a = pl->repack_b = 0;                            // ditto for A and B
  pl->tx_bytes = (128 + pl->bn / cg) * pl->bk * eb;
  if (pl->tiles > (int64_t{1} << 31) - 1) return TL_ERR_UNSUPPORTED;
  if (pl->stream_k < -1 || pl->stream_k > 1) return TL_ERR_INVALID_ARG;
  // grid in CTAs: a multiple of cg * ksplit; one persistent unit (CTA, pair or split
  // cluster) per SM or SM pair
  const int per_unit = cg * pl->ksplit;
  const int64_t want_units =
      pl->grid > 0 ? std::max<int64_t>(1, pl->grid / per_unit) : sms / per_unit;
  schedule(pl, want_units, true, eb);
  if (pl->l2_prefetch < 0) pl->l2_prefetch = default_prefetch(*pl);
  if (pl->l2_prefetch > 1024) return TL_ERR_INVALID_ARG;
  // producers take turns by stage: at most one per ring slot, at most three warps
  const int max_prod = std::min(3, pl->stages);
  pl->producers = pl->producers <= 0 ? max_prod : std::min(pl->producers, max_prod);
  pl->workspace_bytes = split_workspace_bytes(*pl);
  return TL_OK;
}

// Choose BN and the ring depth: fewest waves of tiles over the SMs, weighted by the
// per-tile cost of each width (narrower tiles re-read A more often and issue
// smaller MMAs).  Depth fills the shared memory left after the staging buffers.
void choose_tiling(int64_t M, int64_t N, int64_t K, int trans_a, int trans_b, int sms,
                   tl_plan* pl, int eb = 2) {
  pl->raster_group = 12;      // with serpentine K: the least DRAM traffic at 8192^3 (measured)
  pl->grid = 0;
  pl->l2_prefetch = -1;
  pl->swap_ab = 0;
  // Skinny products (M <= 128 rows against a long N and K) stream B from memory once and
  // are bound by that stream.  Computing C^T = op(B)^T op(A)^T puts N on the MMA's 128
  // rows and M on its narrow N side (16-, 32-, 64- or 128-column tiles), so each stage
  // carries 32 KB of B beside a small tile of A, instead of a mostly empty 128-row tile of
  // A (and A is read from L2 once per 128 rows of N, not once per 64 columns of C).  The
  // 128-row tiles of C^T (64 at N = 8192) then share each tile's k-blocks between the two
  // CTAs of a cluster (cluster split-K), so that 128 SMs stream B; C^T is written by plain
  // stores, so these plans carry no store staging and fit deeper rings.  Measured on GB300
  // at N = K = 8192 (us per call): M = 16: 33.8 with a stream-K split over all SMs, 27.1
  // with the cluster split; M = 64: 34.2 with direct 128 x 64 tiles, 29.3 swapped and split
  // with 4 stages; M = 128: 34.5 direct, 33.3 swapped and split with 3 stages.  Wider M,
  // or an N too long for the split at M > 64, keeps the direct form, and so does an
  // M-major A (trans_a), which cannot feed these boxes.
  const bool split_fits = 2 * ceil_div(N, 128) <= sms;
  if (eb == 2 && !trans_a && N >= 2048 && K >= 1024 && (M <= 64 || (M <= 128 && split_fits))) {
    pl->bm = 128;
    pl->bn = M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 64 ? 64 : 128));
    pl->bk = 128;
    pl->stages = pl->bn == 16 ? 6 : (pl->bn == 32 ? 5 : (pl->bn == 64 ? 4 : 3));
    pl->swap_ab = 1;
    return;
  }
  // One wave of narrow tiles.  When every 128 x 64 tile of C gets an SM of its own, the
  // call lasts one tile's k-loop plus its fill and epilogue.  Each k-block is paced by
  // the bytes the SM loads (A's 128 rows plus B's share; about 64 B per clock from L2),
  // which is the same 48 KB for a 128 x 64 tile as for one CTA of a 256 x 128 pair.  So
  // the narrow tile, which puts the most SMs to work and has the shortest epilogue,
  // finishes first.  Measured on GB300 (fp16, ReLU) it beats the pair tiles that the cost
  // model below would pick:
  //   1024^3              8.25 us vs  9.72 us
  //   768 x 768 x 2048   11.5 us  vs 13.0 us
  //   512 x 2048 x 4096  18.9 us  vs 25.4 us
  // Past about K = 6144, pair tiles split by k-block over all SMs catch up, and they
  // win by 1024 x 1024 x 16384 (44.5 us vs 60.9 us).
  if (eb == 2 && K >= 1024 && K <= 6144 &&
      ceil_div(M, 128) * ceil_div(N, 64) <= static_cast<int64_t>(sms)) {
    pl->bm = 128;
    pl->bn = 64;
    pl->bk = 128;
    pl->stages = 4;
    return;
  }
  // Relative time of one tile per unit of K.  Shared memory (~128 B/clk per SM)
  // carries both the TMA writes and the MMA operand reads, so a 1-CTA 128 x N tile
  // needs 128 (128 + N) / N bytes per MMA cycle: 192 for N = 256, 256 for N = 128;
  // a CTA pair sharing B halves that to 128 (128 + N/2) / N.  The figures below are
  // that model, calibrated on GB300 (a 1-CTA 128-wide tile runs at ~0.64 of the
  // per-SM rate of a 256-wide one).
  struct Cand { int bm, bn, bk, stages; double tile_cost; };
  // The 224- and 192-column pair tiles (K-major B only) fill whole waves where the
  // 256-column ones leave a short last wave, e.g. 4096^3: 16 x 19 = 304 tiles of
  // 256 x 224 are 4 waves of 76 SM pairs, against 3.4 waves of 256 x 256.
  const Cand cands[] = {{256, 256, 128, 3, 128.0}, {256, 256, 64, 6, 135.0},
                        {256, 224, 128, 3, 116.5}, {256, 192, 128, 3, 103.0},
                        {256, 128, 128, 4, 100.0}, {128, 256, 64, 4, 192.0},
                        {128, 128, 64, 6, 150.0},  {128, 64, 128, 4, 110.0},
                        {128, 64, 64, 8, 115.0}};
  constexpr int kCands = sizeof(cands) / sizeof(cands[0]);
  double best = 0.0;
  int pick = -1;
  // 8-bit operands: the same tiles with twice the K elements per stage (the same bytes).
  for (int i = 0; i < kCands; ++i) {
    const int bk = cands[i].bk * (eb == 1 ? 2 : 1);
    if (bk * eb == 256 && K < 1024 * (eb == 1 ? 2 : 1)) continue;   // deep stages: long K
    const int cg = cands[i].bm / 128;
    if (cg == 2 && M <= 128) continue;            // the odd CTA would hold no rows of A
    if (eb == 1 && !trans_b && (cands[i].bn / cg) % 128 != 0) continue;   // 128-wide N boxes
    if ((cands[i].bn == 192 || cands[i].bn == 224) && (eb != 2 || !trans_b)) continue;
    const int64_t tiles = ceil_div(M, cands[i].bm) * ceil_div(N, cands[i].bn);
    const int64_t waves = ceil_div(tiles, std::max(1, sms / cg));
    const double cost = static_cast<double>(waves) * cands[i].tile_cost;
    if (pick < 0 || cost < best - 1e-9) {
      best = cost;
      pick = i;
    }
  }
  pl->bm = cands[pick].bm;
  pl->bn = cands[pick].bn;
  pl->bk = cands[pick].bk * (eb == 1 ? 2 : 1);
  pl->stages = cands[pick].stages;
  // With at most 16 tile rows one raster group spans them all: 4096^3 (16 rows of pair
  // tiles) ran 1 % faster than with groups of 12 (measured, steady state).
  if (ceil_div(M, pl->bm) <= 16) pl->raster_group = 16;
}



// Launch attributes: a cluster of two for CTA pairs, and programmatic stream
// serialization, which lets the kernel start its set-up (barriers, Tensor Memory,
// descriptor prefetch) while the previous kernel of the stream finishes; the kernel
// waits for that kernel's completion (griddepcontrol.wait) before it reads or
// writes global memory.  attr must hold 2 entries.
template <int BN, int CG, int BK, int EB>
void launch_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, size_t smem,
                   cudaStream_t stream, int ks = 1) {
  *cfg = cudaLaunchConfig_t{};
  cfg->blockDim = dim3(tl::kThreads);
  cfg->dynamicSmemBytes = smem;
  cfg->stream = stream;
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (CG * ks > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(CG * ks);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg->attrs = attr;
  cfg->numAttrs = n;
}

// Once per device and kernel: allow the large dynamic shared memory, and find how many
// units (CTAs, CTA pairs, or with ks = 2 clusters of two one-CTA units) the device keeps
// resident at once -- the persistent grid must not exceed it (pairs sit on SM pairs
// within one GPC).  Returns that count, or -1 if the attribute could not be set.
template <int BN, int CG, int BK, int EB = 2>
int prepare_kernel(DeviceState* st, int ks = 1) {
  // slot of this kernel in the per-device caches: 0-11 the 16-bit tilings, 12-13 the
  // narrow ones, 16-27 the 8-bit ones (28-31: attention, 32-35: the block-scaled kernel),
  // 36-39 the 192- and 224-column ones
  constexpr int kIdx = (BN == 192 || BN == 224) ? 36 + (BN == 224) + 2 * (CG - 1)
                       : BN < 64 ? 12 + (BN == 32)
                                 : (BN == 64 ? 0 : (BN == 128 ? 1 : 2)) + 3 * (CG - 1) +
                                       6 * (BK * EB == 256) + 16 * (EB == 1);
  constexpr uint64_t bit = 1ull << kIdx;
  auto units_for = [&] { return ks == 2 ? st->max_clusters2[kIdx] : st->max_units[kIdx]; };
  if (st->attr_done.load(std::memory_order_acquire) & bit) return units_for();
  std::lock_guard<std::mutex> lock(st->mu);
  if (st->attr_done.load(std::memory_order_acquire) & bit) return units_for();
  auto kern = tl::tl_gemm_kernel<BN, CG, BK, EB>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           st->smem_optin) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  // resident clusters of two: the CTA pairs of CG = 2, or cluster split-K's pairs of
  // one-CTA units
  int pairs = st->sms / 2;
  {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    launch_config<BN, CG, BK, EB>(&cfg, attr, static_cast<size_t>(st->smem_optin), nullptr,
                                  CG == 2 ? 1 : 2);
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) {
      pairs = n;
    } else {
      (void)cudaGetLastError();
    }
  }
  st->max_units[kIdx] = CG == 2 ? pairs : st->sms;
  st->max_clusters2[kIdx] = pairs;
  st->attr_done.fetch_or(bit, std::memory_order_acq_rel);
  return units_for();
}

template <int BK, int EB>
int resident_units_bk(DeviceState* st, int bm, int bn, int ks) {
  if constexpr (BK == 128 && EB == 2) {
    if (bn == 192) return bm == 256 ? prepare_kernel<192, 2, BK>(st, ks) : prepare_kernel<192, 1, BK>(st, ks);
    if (bn == 224) return bm == 256 ? prepare_kernel<224, 2, BK>(st, ks) : prepare_kernel<224, 1, BK>(st, ks);
  }
  if (bm == 256) {
    return bn == 128 ? prepare_kernel<128, 2, BK, EB>(st, ks) : prepare_kernel<256, 2, BK, EB>(st, ks);
  }
  if constexpr (BK == 128 && EB == 2) {
    if (bn == 16) return prepare_kernel<16, 1, BK>(st, ks);
    if (bn == 32) return prepare_kernel<32, 1, BK>(st, ks);
  }
  switch (bn) {
    case 64: return prepare_kernel<64, 1, BK, EB>(st, ks);
    case 128: return prepare_kernel<128, 1, BK, EB>(st, ks);
    default: return prepare_kernel<256, 1, BK, EB>(st, ks);
  }
}

int resident_units(DeviceState* st, const tl_plan& pl, int eb) {
  if (eb == 1) {
    return pl.bk == 256 ? resident_units_bk<256, 1>(st, pl.bm, pl.bn, pl.ksplit)
                        : resident_units_bk<128, 1>(st, pl.bm, pl.bn, pl.ksplit);
  }
  return pl.bk == 128 ? resident_units_bk<128, 2>(st, pl.bm, pl.bn, pl.ksplit)
                      : resident_units_bk<64, 2>(st, pl.bm, pl.bn, pl.ksplit);
}

// Launch with exactly pl.grid CTAs: the work split in `prm` was computed for that grid.
template <int BN, int CG, int BK, int EB = 2>
tl_status launch_bn(DeviceState* st, const tl_plan& pl, const CUtensorMap& ta,
                    const CUtensorMap& tb, const CUtensorMap& tc, const tl::GemmParams& prm,
                    cudaStream_t stream) {
  if (prepare_kernel<BN, CG, BK, EB>(st) < 0) return TL_ERR_LAUNCH;
  auto kern = tl::tl_gemm_kernel<BN, CG, BK, EB>;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  launch_config<BN, CG, BK, EB>(&cfg, attr, static_cast<size_t>(pl.smem_bytes), stream,
                                std::max(1, pl.ksplit));
  cfg.gridDim = dim3(static_cast<unsigned>(pl.grid));
  if (cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, prm) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_LAUNCH;
  }
  return TL_OK;
}

template <int BK, int EB>
tl_status launch_tiling(DeviceState* st, const tl_plan& pl, const CUtensorMap& ta,
                        const CUtensorMap& tb, const CUtensorMap& tc, const tl::GemmParams& prm,
                        cudaStream_t stream) {
  if constexpr (BK == 128 && EB == 2) {
    if (pl.bn == 192)
      return pl.bm == 256 ? launch_bn<192, 2, BK>(st, pl, ta, tb, tc, prm, stream)
                          : launch_bn<192, 1, BK>(st, pl, ta, tb, tc, prm, stream);
    if (pl.bn == 224)
      return pl.bm == 256 ? launch_bn<224, 2, BK>(st, pl, ta, tb, tc, prm, stream)
                          : launch_bn<224, 1, BK>(st, pl, ta, tb, tc, prm, stream);
  }
  if (pl.bm == 256) {
    return pl.bn == 128 ? launch_bn<128, 2, BK, EB>(st, pl, ta, tb, tc, prm, stream)
                        : launch_bn<256, 2, BK, EB>(st, pl, ta, tb, tc, prm, stream);
  }
  if constexpr (BK == 128 && EB == 2) {
    if (pl.bn == 16) return launch_bn<16, 1, BK>(st, pl, ta, tb, tc, prm, stream);
    if (pl.bn == 32) return launch_bn<32, 1, BK>(st, pl, ta, tb, tc, prm, stream);
  }
  switch (pl.bn) {
    case 64: return launch_bn<64, 1, BK, EB>(st, pl, ta, tb, tc, prm, stream);
    case 128: return launch_bn<128, 1, BK, EB>(st, pl, ta, tb, tc, prm, stream);
    default: return launch_bn<256, 1, BK, EB>(st, pl, ta, tb, tc, prm, stream);
  }
}

tl_status launch_plan(DeviceState* st, const tl_plan& pl, int eb, const CUtensorMap& ta,
                      const CUtensorMap& tb, const CUtensorMap& tc, const tl::GemmParams& prm,
                      cudaStream_t stream) {
  if (eb == 1) {
    return pl.bk == 256 ? launch_tiling<256, 1>(st, pl, ta, tb, tc, prm, stream)
                        : launch_tiling<128, 1>(st, pl, ta, tb, tc, prm, stream);
  }
  return pl.bk == 128 ? launch_tiling<128, 2>(st, pl, ta, tb, tc, prm, stream)
                      : launch_tiling<64, 2>(st, pl, ta, tb, tc, prm, stream);
}

// ---- tensor-map descriptors --------------------------------------------------------
// A CUtensorMap is a pure function of (element type, rank, base address, extents,
// strides, box), so encoded maps are cached on that key: repeated calls on the same
// buffers skip cuTensorMapEncodeTiled.  The cache is bounded (cleared when full) and
// shared by all threads under a mutex.
struct MapKey {
  uint64_t base;
  uint64_t dims[4];
  uint64_t strides[3];
  uint32_t box[4];
  uint32_t dtype_rank;
  uint32_t swizzle;                          // 1: 128-byte swizzle, 0: none
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};

struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = 1469598103934665603ull;                     // FNV-1a over the key bytes
    const unsigned char* b = reinterpret_cast<const unsigned char*>(&k);
    for (size_t i = 0; i < sizeof(MapKey); ++i) h = (h ^ b[i]) * 1099511628211ull;
    return static_cast<size_t>(h);
  }
};

constexpr size_t kMapCacheMax = 4096;
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash>* g_maps = nullptr;

CUtensorMapDataType map_type(tl_dtype t) {
  if (t == TL_BF16) return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (t == TL_F16) return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return CU_TENSOR_MAP_DATA_TYPE_UINT8;           // E4M3 / E5M2 codes, moved as bytes
}

bool encode_cached(CUtensorMap* map, tl_dtype dtype, uint32_t rank, const void* base,
                   const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                   bool swizzle = true) {
  MapKey key;
  std::memset(&key, 0, sizeof(key));                        // padding bytes take part
  key.base = reinterpret_cast<uint64_t>(base);
  for (uint32_t i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
    if (i + 1 < rank) key.strides[i] = strides[i];
  }
  key.dtype_rank = static_cast<uint32_t>(dtype) * 8u + rank;
  key.swizzle = swizzle ? 1u : 0u;
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (g_maps != nullptr) {
      auto it = g_maps->find(key);
      if (it != g_maps->end()) {
        *map = it->second;
        return true;
      }
    }
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt = map_type(dtype);
  if (enc(map, dt, rank, const_cast<void*>(base), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE,
          swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
    return false;
  }
  std::lock_guard<std::mutex> lock(g_map_mu);
  if (g_maps == nullptr) g_maps = new std::unordered_map<MapKey, CUtensorMap, MapKeyHash>();
  if (g_maps->size() >= kMapCacheMax) g_maps->clear();
  (*g_maps)[key] = *map;
  return true;
}

bool encode_2d(CUtensorMap* map, tl_dtype dtype, const void* base, uint64_t inner, uint64_t outer,
               uint64_t ld_elems, uint32_t box_inner, uint32_t box_outer, bool swizzle = true) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld_elems * static_cast<uint64_t>(elem_bytes(dtype))};
  const cuuint32_t box[2] = {box_inner, box_outer};
  return encode_cached(map, dtype, 2, base, dims, strides, box, swizzle);
}

// A row-major [rows][ld] matrix whose contiguous extent `inner` is a multiple of the
// 128-byte chunk (c = 64 elements of 2 bytes, 128 of 1 byte), viewed as the 3-D tensor
// {c, rows, inner/c} (element (i, r, k) at r*ld + c*k + i) so that one box
// {c, box_rows, box_chunks} fetches several chunks of every row.  Exact (no reads
// past `inner`) because the chunks tile `inner` exactly.
bool encode_chunked_3d(CUtensorMap* map, tl_dtype dtype, const void* base, uint64_t inner,
                       uint64_t rows, uint64_t ld_elems, uint32_t box_rows,
                       uint32_t box_chunks) {
  const uint64_t eb = static_cast<uint64_t>(elem_bytes(dtype));
  const uint64_t chunk = 128 / eb;
  if (inner % chunk != 0) return false;
  const cuuint64_t dims[3] = {chunk, rows, inner / chunk};
  const cuuint64_t strides[2] = {ld_elems * eb, 128};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(chunk), box_rows, box_chunks};
  return encode_cached(map, dtype, 3, base, dims, strides, box);
}

int launch_blocks_for(int64_t elems) {
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ceil_div(elems, 256 * 4), 4096)));
}

// Flags of split tiles hold a value unique to the launch that set them (and are reset
// by their reader), so neither stale flags of earlier launches nor the replay of a
// captured launch can satisfy a wait early.  Random start, then a 64-bit count.
std::atomic<unsigned long long> g_split_token{0};
std::once_flag g_split_token_once;

unsigned long long next_split_token() {
  std::call_once(g_split_token_once, [] {
    std::random_device rd;
    const unsigned long long seed = (static_cast<unsigned long long>(rd()) << 32) ^ rd();
    g_split_token.store(seed | 1ull, std::memory_order_relaxed);
  });
  unsigned long long t = g_split_token.fetch_add(2, std::memory_order_relaxed);
  return t == 0 ? 1ull : t;
}

// ---- scratch for tl_gemm_noalloc -------------------------------------------------
// Callers that cannot allocate get the repack workspace from this fixed array instead
// of the stream-ordered allocator.  It exists on every device that loads the library,
// for the life of the process.  Host code must not use the array's name as a device
// address: its device address comes from cudaGetSymbolAddress, taken once per device
// with that device current.
constexpr int64_t kNoAllocScratchBytes = int64_t{32} << 20;   // 32 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocScratch {
  std::once_flag once;
  void* ptr = nullptr;
};
NoAllocScratch g_noalloc[kMaxDevices];

void* noalloc_scratch(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  NoAllocScratch& e = g_noalloc[dev];
  std::call_once(e.once, [&e] {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) == cudaSuccess) e.ptr = p;
    else (void)cudaGetLastError();
  });
  return e.ptr;
}

tl_status run(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
              int64_t lda, int64_t ldb, int64_t ldc, const Types& ty, int trans_a, int trans_b,
              tl_epilogue epilogue, const tl_plan* forced, cudaStream_t stream,
              bool no_alloc = false) {
  const tl_dtype dtype = ty.out;
  const int eb = ty.eb;
  tl_status s = validate_common(M, N, K, dtype, trans_a, trans_b);
  if (s != TL_OK) return s;
  if (epilogue != TL_EPI_NONE && epilogue != TL_EPI_RELU) return TL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return TL_OK;
  if (ldc < N) return TL_ERR_INVALID_ARG;
  if (C == nullptr) return TL_ERR_NULL_PTR;
  if (reinterpret_cast<uintptr_t>(C) & 1u) return TL_ERR_ALIGNMENT;
  const int64_t a_rows = trans_a ? K : M, a_cols = trans_a ? M : K;
  const int64_t b_rows = trans_b ? N : K, b_cols = trans_b ? K : N;
  if (K > 0) {
    if (lda < a_cols || ldb < b_cols) return TL_ERR_INVALID_ARG;
    if (A == nullptr || B == nullptr) return TL_ERR_NULL_PTR;
    if (eb == 2 && ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 1u))
      return TL_ERR_ALIGNMENT;
    uintptr_t c0, c1, a0, a1, b0, b1;
    extent(C, M, N, ldc, &c0, &c1);
    extent(A, a_rows, a_cols, lda, &a0, &a1, eb);
    extent(B, b_rows, b_cols, ldb, &b0, &b1, eb);
    if (overlaps(c0, c1, a0, a1) || overlaps(c0, c1, b0, b1)) return TL_ERR_ALIAS;
  }
  int dev = 0;
  DeviceState* st = device_state(&dev);
  if (st == nullptr) return TL_ERR_DEVICE;
  if (!st->sm103) return TL_ERR_UNSUPPORTED;
  // The allocation-free variant looks up its scratch array on every device's first call
  // (so the set-up never falls inside a later stream capture); only calls that need the
  // array fail if that lookup did.
  void* scratch = no_alloc ? noalloc_scratch(dev) : nullptr;
  if ((s = check_device_pointer(C, dev)) != TL_OK) return s;
  if (K > 0) {
    if ((s = check_device_pointer(A, dev)) != TL_OK) return s;
    if ((s = check_device_pointer(B, dev)) != TL_OK) return s;
  }
  uint16_t* c16 = static_cast<uint16_t*>(C);
  if (K == 0) {
    const int blocks = launch_blocks_for(M * N);
    tl::tl_fill_zero_kernel<<<blocks, 256, 0, stream>>>(c16, M, N, ldc);
    return cudaGetLastError() == cudaSuccess ? TL_OK : TL_ERR_LAUNCH;
  }

  tl_plan pl;
  std::memset(&pl, 0, sizeof(pl));
  if (forced) {
    pl.bm = forced->bm;
    pl.bn = forced->bn;
    pl.bk = forced->bk;
    pl.stages = forced->stages;
    pl.raster_group = forced->raster_group > 0 ? forced->raster_group : 16;
    pl.grid = forced->grid;
    pl.l2_prefetch = forced->l2_prefetch;
    pl.producers = forced->producers;
    pl.stream_k = forced->stream_k;
    pl.swap_ab = forced->swap_ab;
    pl.ksplit = forced->ksplit;
  } else {
    choose_tiling(M, N, K, trans_a, trans_b, st->sms, &pl, eb);
  }
  if ((s = complete_plan(M, N, K, trans_a, trans_b, st->sms, &pl, eb)) != TL_OK) return s;
  if (pl.smem_bytes > st->smem_optin) return TL_ERR_INVALID_ARG;
  // Re-split over the units this device really keeps resident (CTA pairs: the cluster
  // occupancy can be below SMs / 2).  Callers that cannot allocate get whole tiles only:
  // the split needs a workspace for partial sums.
  const int resident = resident_units(st, pl, eb);
  if (resident <= 0) return TL_ERR_LAUNCH;
  {
    const int per_unit = (pl.bm / 128) * pl.ksplit;
    const int64_t want_units = forced && forced->grid > 0
                                   ? std::max(1, forced->grid / per_unit)
                                   : st->sms / per_unit;
    schedule(&pl, std::min<int64_t>(want_units, resident), !no_alloc, eb);
  }
  const int64_t ws_split = split_workspace_bytes(pl);

  // Operands the TMA unit cannot address directly go through a padded copy (pitch
  // rounded up to 16 bytes).
  const int64_t pad = 16 / eb;
  const bool repack_a = !tma_ok(A, lda, eb);
  const bool repack_b = !tma_ok(B, ldb, eb);
  const int64_t lda_w = repack_a ? ceil_div(a_cols, pad) * pad : lda;
  const int64_t ldb_w = repack_b ? ceil_div(b_cols, pad) * pad : ldb;
  const int64_t ws_a = repack_a ? a_rows * lda_w * eb : 0;
  const int64_t ws_b = repack_b ? b_rows * ldb_w * eb : 0;
  void* ws = nullptr;
  const void* a_use = A;
  const void* b_use = B;
  float* sk_partials = nullptr;
  unsigned long long* sk_flags = nullptr;
  if (ws_a + ws_b + ws_split > 0) {
    const int64_t ws_a_rounded = ceil_div(ws_a, 256) * 256;
    const int64_t ws_b_rounded = ceil_div(ws_b, 256) * 256;
    uint8_t* w = nullptr;
    if (no_alloc) {
      if (ws_a_rounded + ws_b > kNoAllocScratchBytes) return TL_ERR_UNSUPPORTED;
      if (scratch == nullptr) return TL_ERR_DEVICE;
      w = static_cast<uint8_t*>(scratch);
    } else {
      if (cudaMallocAsync(&ws, static_cast<size_t>(ws_a_rounded + ws_b_rounded + ws_split),
                          stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return TL_ERR_LAUNCH;
      }
      w = static_cast<uint8_t*>(ws);
    }
    if (ws_split > 0) {
      uint8_t* split = w + ws_a_rounded + ws_b_rounded;
      sk_partials = reinterpret_cast<float*>(split);
      sk_flags = reinterpret_cast<unsigned long long*>(
          split + static_cast<int64_t>(pl.grid) * 128 * pl.bn * 4);
    }
    auto repack = [&](const void* src, void* dst, int64_t rows, int64_t cols, int64_t sp,
                      int64_t dp) {
      if (eb == 1) {
        tl::tl_repack_kernel<uint8_t><<<launch_blocks_for(rows * cols), 256, 0, stream>>>(
            static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), rows, cols, sp, dp);
      } else {
        tl::tl_repack_kernel<uint16_t><<<launch_blocks_for(rows * cols), 256, 0, stream>>>(
            static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst), rows, cols, sp, dp);
      }
    };
    if (repack_a) {
      repack(A, w, a_rows, a_cols, lda, lda_w);
      a_use = w;
    }
    if (repack_b) {
      uint8_t* wb = w + ws_a_rounded;
      repack(B, wb, b_rows, b_cols, ldb, ldb_w);
      b_use = wb;
    }
    if (cudaGetLastError() != cudaSuccess) {
      if (ws) (void)cudaFreeAsync(ws, stream);
      return TL_ERR_LAUNCH;
    }
  }
  // The kernel's operands: (A, B) as given, or (B, A) with their transposes flipped
  // when it computes C^T = op(B)^T op(A)^T.
  struct Operand {
    const void* ptr;
    int64_t ld;
    int trans;
    tl_dtype type;
  };
  const bool swap = pl.swap_ab != 0;
  const int64_t kM = swap ? N : M, kN = swap ? M : N;
  const Operand ka = swap ? Operand{b_use, ldb_w, !trans_b, ty.b_type}
                          : Operand{a_use, lda_w, trans_a, ty.a_type};
  const Operand kb = swap ? Operand{a_use, lda_w, !trans_a, ty.a_type}
                          : Operand{b_use, ldb_w, trans_b, ty.b_type};
  // C by TMA bulk stores from a swizzled staging buffer, or by plain stores from
  // registers (16-byte vectors when C is aligned).  A forced plan with tma_store = -1
  // asks for plain stores.
  const bool c_aligned = tma_ok(C, ldc);
  const bool tma_store = !swap && pl.bn >= 64 && c_aligned && !(forced && forced->tma_store < 0);

  // Operand maps.  One box per stage (a 3-D view) when the operand's contiguous extent
  // is a multiple of 64 and the stage spans several 64-element chunks; otherwise 2-D
  // boxes of one chunk each, whose out-of-range parts the TMA unit fills with zeros.
  CUtensorMap ta, tb, tc;
  std::memset(&tc, 0, sizeof(tc));
  const int cg = pl.bm / 128;
  const uint32_t bn_cta = static_cast<uint32_t>(pl.bn / cg);
  const uint32_t chunk = static_cast<uint32_t>(128 / eb);          // elements per 128 bytes
  const uint32_t kchunks = static_cast<uint32_t>(pl.bk * eb / 128);
  bool enc_ok = true;
  bool a3d = false, b3d = false;
  if (!ka.trans) {
    a3d = kchunks > 1 && encode_chunked_3d(&ta, ka.type, ka.ptr, K, kM, ka.ld, 128, kchunks);
    if (!a3d) enc_ok &= encode_2d(&ta, ka.type, ka.ptr, K, kM, ka.ld, chunk, 128);
  } else {
    a3d = encode_chunked_3d(&ta, ka.type, ka.ptr, kM, K, ka.ld, pl.bk, 128 / chunk);
    if (!a3d) enc_ok &= encode_2d(&ta, ka.type, ka.ptr, kM, K, ka.ld, chunk, pl.bk);
  }
  if (kb.trans) {
    b3d = kchunks > 1 && encode_chunked_3d(&tb, kb.type, kb.ptr, K, kN, kb.ld, bn_cta, kchunks);
    if (!b3d) enc_ok &= encode_2d(&tb, kb.type, kb.ptr, K, kN, kb.ld, chunk, bn_cta);
  } else {
    b3d = bn_cta > chunk &&
          encode_chunked_3d(&tb, kb.type, kb.ptr, kN, K, kb.ld, pl.bk, bn_cta / chunk);
    if (!b3d) enc_ok &= encode_2d(&tb, kb.type, kb.ptr, kN, K, kb.ld, chunk, pl.bk);
  }
  if (tma_store) enc_ok &= encode_2d(&tc, dtype, C, N, M, ldc, 64, 32);
  if (!enc_ok) {
    if (ws) (void)cudaFreeAsync(ws, stream);
    return TL_ERR_LAUNCH;
  }

  tl::GemmParams prm;
  std::memset(&prm, 0, sizeof(prm));
  prm.M = static_cast<int32_t>(kM);
  prm.N = static_cast<int32_t>(kN);
  prm.K = static_cast<int32_t>(K);
  prm.tiles_m = static_cast<int32_t>(pl.tiles_m);
  prm.tiles_n = static_cast<int32_t>(pl.tiles_n);
  prm.num_tiles = static_cast<int32_t>(pl.tiles);
  prm.k_blocks = static_cast<int32_t>(pl.k_blocks);
  prm.stages = pl.stages;
  prm.raster_group = pl.raster_group;
  prm.trans_a = ka.trans;
  prm.trans_b = kb.trans;
  prm.bf16 = dtype == TL_BF16 ? 1 : 0;
  prm.scale = ty.scale ? 1 : 0;
  prm.alpha = ty.alpha;
  prm.relu = epilogue == TL_EPI_RELU ? 1 : 0;
  prm.tma_store = tma_store ? 1 : 0;
  prm.c_trans = swap ? 1 : 0;
  prm.c_vec = c_aligned ? 1 : 0;
  prm.l2_prefetch = pl.l2_prefetch;
  prm.a3d = a3d ? 1 : 0;
  prm.b3d = b3d ? 1 : 0;
  prm.producers = pl.producers;
  prm.dp_tiles = pl.dp_tiles;
  prm.sk_iters = pl.sk_iters;
  prm.ksplit = pl.ksplit;
  prm.serpentine = 1;
  prm.sk_partials = sk_partials;
  prm.sk_flags = sk_flags;
  prm.sk_token = next_split_token();
  prm.idesc = eb == 1
                  ? tl::mma_idesc_f8(ka.type == TL_E5M2 ? 1u : 0u, kb.type == TL_E5M2 ? 1u : 0u,
                                     ka.trans ? 1u : 0u, kb.trans ? 0u : 1u,
                                     static_cast<uint32_t>(pl.bm), static_cast<uint32_t>(pl.bn))
                  : tl::mma_idesc_f16(prm.bf16, ka.trans ? 1u : 0u, kb.trans ? 0u : 1u,
                                      static_cast<uint32_t>(pl.bm), static_cast<uint32_t>(pl.bn));
  prm.C = C;
  prm.ldc = ldc;
  prm.status = st->status;
  prm.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  prm.stall = g_stall.load(std::memory_order_relaxed);

  s = launch_plan(st, pl, eb, ta, tb, tc, prm, stream);
  if (ws) {
    if (cudaFreeAsync(ws, stream) != cudaSuccess) {
      (void)cudaGetLastError();
      if (s == TL_OK) s = TL_ERR_LAUNCH;
    }
  }
  return s;
}

// ---- attention ---------------------------------------------------------------------
// Q, K, V, O are [B, S, H, D] row-major; the kernel reads 128-row tiles of one
// (batch, head) through a 4-D map {D, H, S, B} (box {64, 1, 128, 1}: a 64-element
// chunk of 128 sequence positions), which zero-fills rows past S.
bool encode_bshd(CUtensorMap* map, tl_dtype dtype, const void* base, int64_t B, int64_t S,
                 int64_t H, int64_t D, uint32_t box_rows) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D * 2), static_cast<cuuint64_t>(H * D * 2),
                                 static_cast<cuuint64_t>(S * H * D * 2)};
  const cuuint32_t box[4] = {64, 1, box_rows, 1};
  return encode_cached(map, dtype, 4, base, dims, strides, box);
}

template <int D, bool kBf16>
tl_status launch_attention(DeviceState* st, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& to,
                           const tl::AttnParams& prm, int64_t grid,
                           cudaStream_t stream) {
  // at least 120 KB, so that two CTAs never share an SM: each allocates all 512 Tensor
  // Memory columns, and a second allocation would wait for the first CTA to finish (the
  // grid has at most one CTA per SM, but another kernel's CTA could still be resident)
  constexpr uint32_t kSmem = tl::attn_smem_bytes<D>() > 122880u ? tl::attn_smem_bytes<D>() : 122880u;
  constexpr uint32_t bit = 1u << (28 + (D == 128) + 2 * kBf16);
  auto kern = tl::tl_attention_kernel<D, kBf16>;
  if (static_cast<int64_t>(kSmem) > st->smem_optin) return TL_ERR_UNSUPPORTED;
  if (!(st->attr_done.load(std::memory_order_acquire) & bit)) {
    std::lock_guard<std::mutex> lock(st->mu);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmem)) != cudaSuccess) {
      (void)cudaGetLastError();
      return TL_ERR_LAUNCH;
    }
    st->attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(tl::kAttnThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, to, prm) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_LAUNCH;
  }
  return TL_OK;
}

tl_status run_attention(const void* Q, const void* K, const void* V, void* O, int64_t B,
                        int64_t S, int64_t H, int64_t D, tl_dtype dtype, int causal,
                        cudaStream_t stream) {
  if (B < 0 || S < 0 || H < 0 || D <= 0) return TL_ERR_INVALID_ARG;
  if (dtype != TL_F16 && dtype != TL_BF16) return TL_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return TL_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return TL_ERR_UNSUPPORTED;
  if (B == 0 || S == 0 || H == 0) return TL_OK;
  if (S > (int64_t{1} << 31) - 256 || H > 65535 || B > 65535) return TL_ERR_UNSUPPORTED;
  if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr) return TL_ERR_NULL_PTR;
  if ((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
       reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(O)) & 15u) {
    return TL_ERR_ALIGNMENT;
  }
  const int64_t elems = B * S * H * D;
  const uintptr_t o0 = reinterpret_cast<uintptr_t>(O), o1 = o0 + static_cast<uintptr_t>(elems * 2);
  for (const void* x : {Q, K, V}) {
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(x);
    if (overlaps(o0, o1, x0, x0 + static_cast<uintptr_t>(elems * 2))) return TL_ERR_ALIAS;
  }
  int dev = 0;
  DeviceState* st = device_state(&dev);
  if (st == nullptr) return TL_ERR_DEVICE;
  if (!st->sm103) return TL_ERR_UNSUPPORTED;
  tl_status s;
  for (const void* x : {Q, K, V, static_cast<const void*>(O)}) {
    if ((s = check_device_pointer(x, dev)) != TL_OK) return s;
  }
  // Q, K, V in boxes of 128 rows; O is stored by each softmax warp in boxes of 32 rows
  CUtensorMap tq, tk, tv, to;
  if (!encode_bshd(&tq, dtype, Q, B, S, H, D, tl::kAttnBM) ||
      !encode_bshd(&tk, dtype, K, B, S, H, D, tl::kAttnBN) ||
      !encode_bshd(&tv, dtype, V, B, S, H, D, tl::kAttnBN) ||
      !encode_bshd(&to, dtype, O, B, S, H, D, 32)) {
    return TL_ERR_LAUNCH;
  }
  tl::AttnParams prm;
  std::memset(&prm, 0, sizeof(prm));
  prm.B = static_cast<int32_t>(B);
  prm.S = static_cast<int32_t>(S);
  prm.H = static_cast<int32_t>(H);
  prm.causal = causal;
  const uint32_t bf16 = dtype == TL_BF16 ? 1u : 0u;
  prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  prm.O = O;
  prm.idesc_s = tl::mma_idesc_f16(bf16, 0u, 0u, 128u, 128u);
  prm.idesc_o = tl::mma_idesc_f16(bf16, 0u, 1u, 128u, static_cast<uint32_t>(D));
  prm.status = st->status;
  prm.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  // Work items for the persistent grid: single query tiles, or (causal, more tiles than
  // SMs) pairs of tiles (n-1-k, k) of one head, n + 1 key tiles per pair.
  const int64_t q_tiles = ceil_div(S, tl::kAttnBM);
  const bool pair = causal && B * H * q_tiles > st->sms;
  const int64_t per_head = pair ? ceil_div(q_tiles, 2) : q_tiles;
  const int64_t items = B * H * per_head;
  if (items > INT32_MAX) return TL_ERR_UNSUPPORTED;
  prm.n_q_tiles = static_cast<int32_t>(q_tiles);
  prm.items_per_head = static_cast<int32_t>(per_head);
  prm.n_items = static_cast<int32_t>(items);
  prm.pair = pair ? 1 : 0;
  const int64_t grid = std::min<int64_t>(items, st->sms);
  if (dtype == TL_BF16)
    return D == 64 ? launch_attention<64, true>(st, tq, tk, tv, to, prm, grid, stream)
                   : launch_attention<128, true>(st, tq, tk, tv, to, prm, grid, stream);
  return D == 64 ? launch_attention<64, false>(st, tq, tk, tv, to, prm, grid, stream)
                 : launch_attention<128, false>(st, tq, tk, tv, to, prm, grid, stream);
}

// ---- the block-scaled (MX) 8-bit GEMM ---------------------------------------------
template <int BN, bool kBf16>
tl_status launch_mx(const void* A, const void* B, const void* SA, const void* SB, void* C,
                    int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                    int64_t sfa_ld, int64_t sfb_ld, tl_dtype a_type, tl_dtype b_type,
                    tl_epilogue epilogue, DeviceState* st, cudaStream_t stream) {
  const int64_t k_blocks = ceil_div(K, tl::kMxBK);
  // operands in 128-byte swizzled boxes; the scales in plain boxes of one group of
  // stages (kMxGroup stages x 4 bytes) of 128 rows
  CUtensorMap ta, tb, tsa, tsb;
  if (!encode_2d(&ta, a_type, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                 static_cast<uint64_t>(lda), tl::kMxBK, tl::kMxBM) ||
      !encode_2d(&tb, b_type, B, static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                 static_cast<uint64_t>(ldb), tl::kMxBK, BN) ||
      !encode_2d(&tsa, TL_E4M3, SA, static_cast<uint64_t>(sfa_ld), static_cast<uint64_t>(M),
                 static_cast<uint64_t>(sfa_ld), 4u * tl::kMxGroup, tl::kMxBM, false) ||
      !encode_2d(&tsb, TL_E4M3, SB, static_cast<uint64_t>(sfb_ld), static_cast<uint64_t>(N),
                 static_cast<uint64_t>(sfb_ld), 4u * tl::kMxGroup, BN, false)) {
    return TL_ERR_LAUNCH;
  }
  tl::MxParams prm;
  std::memset(&prm, 0, sizeof(prm));
  prm.M = static_cast<int32_t>(M);
  prm.N = static_cast<int32_t>(N);
  prm.K = static_cast<int32_t>(K);
  prm.k_blocks = static_cast<int32_t>(k_blocks);
  prm.tiles_n = static_cast<int32_t>(ceil_div(N, BN));
  prm.num_tiles = static_cast<int32_t>(ceil_div(M, tl::kMxBM) * prm.tiles_n);
  prm.C = C;
  prm.ldc = ldc;
  prm.relu = epilogue == TL_EPI_RELU ? 1 : 0;
  prm.c_vec = tma_ok(C, ldc) ? 1 : 0;
  prm.idesc = tl::mma_idesc_mx(a_type == TL_E5M2 ? 1u : 0u, b_type == TL_E5M2 ? 1u : 0u,
                               tl::kMxBM, BN);
  prm.status = st->status;
  prm.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  constexpr uint32_t kSmem = tl::mx_smem_bytes<BN>();
  if (static_cast<int64_t>(kSmem) > st->smem_optin) return TL_ERR_UNSUPPORTED;
  auto kern = tl::tl_gemm_mx_kernel<kBf16, BN>;
  constexpr uint64_t bit = 1ull << (32 + 2 * (BN == 256) + (kBf16 ? 1 : 0));   // slots 32-35
  if (!(st->attr_done.load(std::memory_order_acquire) & bit)) {
    std::lock_guard<std::mutex> lock(st->mu);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmem)) != cudaSuccess) {
      (void)cudaGetLastError();
      return TL_ERR_LAUNCH;
    }
    st->attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  // persistent: at most one CTA per SM (the shared memory allows no more)
  cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(prm.num_tiles, st->sms)));
  cfg.blockDim = dim3(tl::kMxThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, ta, tb, tsa, tsb, prm) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_LAUNCH;
  }
  return TL_OK;
}

tl_status run_mx(const void* A, const void* B, const void* SA, const void* SB, void* C,
                 int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                 int64_t sfa_ld, int64_t sfb_ld, tl_dtype a_type, tl_dtype b_type,
                 tl_dtype c_type, tl_epilogue epilogue, cudaStream_t stream) {
  if (M < 0 || N < 0 || K < 0 || K % 32 != 0) return TL_ERR_INVALID_ARG;
  if (!is_fp8(a_type) || !is_fp8(b_type)) return TL_ERR_INVALID_ARG;
  if (c_type != TL_F16 && c_type != TL_BF16) return TL_ERR_INVALID_ARG;
  if (epilogue != TL_EPI_NONE && epilogue != TL_EPI_RELU) return TL_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return TL_OK;
  if (M > INT32_MAX - tl::kMxBM || N > INT32_MAX - 256 || K > INT32_MAX - tl::kMxBK ||
      ceil_div(M, tl::kMxBM) * ceil_div(N, 128) > INT32_MAX)
    return TL_ERR_UNSUPPORTED;
  if (ldc < N) return TL_ERR_INVALID_ARG;
  if (C == nullptr) return TL_ERR_NULL_PTR;
  if (reinterpret_cast<uintptr_t>(C) & 1u) return TL_ERR_ALIGNMENT;
  const int64_t k_blocks = ceil_div(K, tl::kMxBK);
  if (K > 0) {
    if (lda < K || ldb < K || sfa_ld < 4 * k_blocks || sfb_ld < 4 * k_blocks)
      return TL_ERR_INVALID_ARG;
    if (A == nullptr || B == nullptr || SA == nullptr || SB == nullptr) return TL_ERR_NULL_PTR;
    // operands straight to the TMA unit; the scales as aligned 32-bit words
    if (!tma_ok(A, lda, 1) || !tma_ok(B, ldb, 1)) return TL_ERR_ALIGNMENT;
    if (!tma_ok(SA, sfa_ld, 1) || !tma_ok(SB, sfb_ld, 1)) return TL_ERR_ALIGNMENT;
    uintptr_t c0, c1, x0, x1;
    extent(C, M, N, ldc, &c0, &c1);
    const struct { const void* p; int64_t rows, cols, ld; } ins[4] = {
        {A, M, K, lda}, {B, N, K, ldb}, {SA, M, 4 * k_blocks, sfa_ld}, {SB, N, 4 * k_blocks, sfb_ld}};
    for (const auto& in : ins) {
      extent(in.p, in.rows, in.cols, in.ld, &x0, &x1, 1);
      if (overlaps(c0, c1, x0, x1)) return TL_ERR_ALIAS;
    }
  }
  int dev = 0;
  DeviceState* st = device_state(&dev);
  if (st == nullptr) return TL_ERR_DEVICE;
  if (!st->sm103) return TL_ERR_UNSUPPORTED;
  tl_status s;
  if ((s = check_device_pointer(C, dev)) != TL_OK) return s;
  if (K == 0) {
    tl::tl_fill_zero_kernel<<<launch_blocks_for(M * N), 256, 0, stream>>>(static_cast<uint16_t*>(C),
                                                                         M, N, ldc);
    return cudaGetLastError() == cudaSuccess ? TL_OK : TL_ERR_LAUNCH;
  }
  for (const void* x : {A, B, SA, SB}) {
    if ((s = check_device_pointer(x, dev)) != TL_OK) return s;
  }
  // 128 x 256 tiles (half the tiles and a quarter less operand traffic per flop) unless
  // N fits one 128-wide tile
  if (N > 128)
    return c_type == TL_BF16 ? launch_mx<256, true>(A, B, SA, SB, C, M, N, K, lda, ldb, ldc,
                                                   sfa_ld, sfb_ld, a_type, b_type, epilogue, st,
                                                   stream)
                             : launch_mx<256, false>(A, B, SA, SB, C, M, N, K, lda, ldb, ldc,
                                                    sfa_ld, sfb_ld, a_type, b_type, epilogue, st,
                                                    stream);
  return c_type == TL_BF16 ? launch_mx<128, true>(A, B, SA, SB, C, M, N, K, lda, ldb, ldc, sfa_ld,
                                                 sfb_ld, a_type, b_type, epilogue, st, stream)
                           : launch_mx<128, false>(A, B, SA, SB, C, M, N, K, lda, ldb, ldc,
                                                  sfa_ld, sfb_ld, a_type, b_type, epilogue, st,
                                                  stream);
}

}  // namespace

extern "C" {

tl_status tl_gemm(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                  int64_t lda, int64_t ldb, int64_t ldc, tl_dtype dtype, int trans_a,
                  int trans_b, tl_epilogue epilogue, tl_stream_t stream) {
  if (dtype != TL_F16 && dtype != TL_BF16) return TL_ERR_INVALID_ARG;
  return run(A, B, C, M, N, K, lda, ldb, ldc, types_16(dtype), trans_a, trans_b, epilogue,
             nullptr, reinterpret_cast<cudaStream_t>(stream));
}

tl_status tl_gemm_with_plan(const void* A, const void* B, void* C, int64_t M, int64_t N,
                            int64_t K, int64_t lda, int64_t ldb, int64_t ldc, tl_dtype dtype,
                            int trans_a, int trans_b, tl_epilogue epilogue, const tl_plan* plan,
                            tl_stream_t stream) {
  if (plan == nullptr) return TL_ERR_INVALID_ARG;
  if (dtype != TL_F16 && dtype != TL_BF16) return TL_ERR_INVALID_ARG;
  return run(A, B, C, M, N, K, lda, ldb, ldc, types_16(dtype), trans_a, trans_b, epilogue, plan,
             reinterpret_cast<cudaStream_t>(stream));
}

tl_status tl_gemm_mx(const void* A, const void* B, const void* SFA, const void* SFB, void* C,
                     int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                     int64_t sfa_ld, int64_t sfb_ld, tl_dtype a_type, tl_dtype b_type,
                     tl_dtype c_type, tl_epilogue epilogue, tl_stream_t stream) {
  return run_mx(A, B, SFA, SFB, C, M, N, K, lda, ldb, ldc, sfa_ld, sfb_ld, a_type, b_type, c_type,
                epilogue, reinterpret_cast<cudaStream_t>(stream));
}

tl_status tl_gemm_fp8(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int64_t ldc, tl_dtype a_type, tl_dtype b_type,
                      tl_dtype c_type, int trans_a, int trans_b, float alpha,
                      tl_epilogue epilogue, const tl_plan* plan, tl_stream_t stream) {
  if (!is_fp8(a_type) || !is_fp8(b_type)) return TL_ERR_INVALID_ARG;
  if (c_type != TL_F16 && c_type != TL_BF16) return TL_ERR_INVALID_ARG;
  if (!std::isfinite(alpha)) return TL_ERR_INVALID_ARG;
  const Types ty{1, a_type, b_type, c_type, alpha, alpha != 1.0f};
  return run(A, B, C, M, N, K, lda, ldb, ldc, ty, trans_a, trans_b, epilogue, plan,
             reinterpret_cast<cudaStream_t>(stream));
}

tl_status tl_gemm_plan(int64_t M, int64_t N, int64_t K, tl_dtype dtype, int trans_a, int trans_b,
                       int num_sms, tl_plan* plan) {
  if (plan == nullptr) return TL_ERR_NULL_PTR;
  const tl_status s = validate_common(M, N, K, dtype, trans_a, trans_b);
  if (s != TL_OK) return s;
  std::memset(plan, 0, sizeof(*plan));
  const int sms = num_sms > 0 ? num_sms : kDefaultSms;
  choose_tiling(M, N, K, trans_a, trans_b, sms, plan, elem_bytes(dtype));
  return complete_plan(M, N, K, trans_a, trans_b, sms, plan, elem_bytes(dtype));
}

tl_status tl_plan_complete(int64_t M, int64_t N, int64_t K, tl_dtype dtype, int trans_a,
                           int trans_b, int num_sms, tl_plan* plan) {
  if (plan == nullptr) return TL_ERR_NULL_PTR;
  const tl_status s = validate_common(M, N, K, dtype, trans_a, trans_b);
  if (s != TL_OK) return s;
  if (plan->raster_group <= 0) plan->raster_group = 16;
  const int32_t pf = plan->l2_prefetch;
  const int32_t prod = plan->producers;
  const int32_t sk = plan->stream_k;
  const int32_t swap = plan->swap_ab;
  const int32_t ks = plan->ksplit;
  std::memset(&plan->tiles_m, 0, sizeof(tl_plan) - offsetof(tl_plan, tiles_m));
  plan->l2_prefetch = pf;
  plan->producers = prod;
  plan->stream_k = sk;
  plan->swap_ab = swap;
  plan->ksplit = ks;
  return complete_plan(M, N, K, trans_a, trans_b, num_sms, plan, elem_bytes(dtype));
}

tl_status tl_gemm_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N,
                          int64_t K, int64_t lda, int64_t ldb, int64_t ldc, tl_dtype dtype,
                          int trans_a, int trans_b, tl_epilogue epilogue, tl_stream_t stream) {
  if (dtype != TL_F16 && dtype != TL_BF16) return TL_ERR_INVALID_ARG;
  return run(A, B, C, M, N, K, lda, ldb, ldc, types_16(dtype), trans_a, trans_b, epilogue,
             nullptr, reinterpret_cast<cudaStream_t>(stream), /*no_alloc=*/true);
}

int64_t tl_gemm_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

const char* tl_status_string(tl_status status) {
  switch (status) {
    case TL_OK: return "TL_OK";
    case TL_ERR_INVALID_ARG: return "TL_ERR_INVALID_ARG";
    case TL_ERR_NULL_PTR: return "TL_ERR_NULL_PTR";
    case TL_ERR_ALIGNMENT: return "TL_ERR_ALIGNMENT";
    case TL_ERR_UNSUPPORTED: return "TL_ERR_UNSUPPORTED";
    case TL_ERR_ALIAS: return "TL_ERR_ALIAS";
    case TL_ERR_DEVICE: return "TL_ERR_DEVICE";
    case TL_ERR_LAUNCH: return "TL_ERR_LAUNCH";
    case TL_ERR_TIMEOUT: return "TL_ERR_TIMEOUT";
  }
  return "TL_ERR_UNKNOWN";
}

tl_status tl_device_status(int reset, uint32_t* detail) {
  if (device_state(nullptr) == nullptr) return TL_ERR_DEVICE;
  if (cudaDeviceSynchronize() != cudaSuccess) return TL_ERR_DEVICE;
  uint32_t word = 0;
  if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)) != cudaSuccess) return TL_ERR_DEVICE;
  if (detail) *detail = word;
  if (reset) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return TL_ERR_DEVICE;
  }
  return word == 0 ? TL_OK : static_cast<tl_status>(word & 0xFFu);
}

tl_status tl_last_device_status(void) { return tl_device_status(0, nullptr); }

void tl_set_wait_timeout_ns(uint64_t ns) {
  ns = std::max<uint64_t>(100000ull, std::min<uint64_t>(ns, 60000000000ull));
  g_timeout_ns.store(ns, std::memory_order_relaxed);
}

tl_status tl_attention_fwd(const void* Q, const void* K, const void* V, void* O, int64_t B,
                           int64_t S, int64_t H, int64_t D, tl_dtype dtype, int causal,
                           tl_stream_t stream) {
  return run_attention(Q, K, V, O, B, S, H, D, dtype, causal,
                       reinterpret_cast<cudaStream_t>(stream));
}

void tl_debug_set_stall(int mode) { g_stall.store(mode == 1 ? 1 : 0, std::memory_order_relaxed); }

int tl_version(void) { return 100; }

}  // extern "C"
