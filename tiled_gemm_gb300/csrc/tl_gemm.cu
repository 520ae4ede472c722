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
#include <atomic>
#include <cstdint>
#include <cstddef>
#include <cstring>
#include <mutex>

#include "gemm_kernel.cuh"
#include "tl_gemm.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxSmemPerCta = 232448;   // 227 KB opt-in per CTA on sm_100-class parts
constexpr int kDefaultSms = 148;

__device__ uint32_t g_status_word;           // bounded-wait outcome, see tl_device_status

std::atomic<uint64_t> g_timeout_ns{2000000000ull};

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
  std::atomic<uint32_t> attr_done{0};        // bit i: smem attribute set for kernel i
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

bool tma_ok(const void* p, int64_t ld) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && ((ld * 2) & 15) == 0;
}

// Byte extent [lo, hi) touched by a rows x cols matrix with leading dimension ld.
void extent(const void* p, int64_t rows, int64_t cols, int64_t ld, uintptr_t* lo, uintptr_t* hi) {
  *lo = reinterpret_cast<uintptr_t>(p);
  *hi = *lo + static_cast<uintptr_t>(((rows - 1) * ld + cols) * 2);
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

bool plan_supported(const tl_plan& pl) {
  return pl.bm == 128 && (pl.bn == 64 || pl.bn == 128 || pl.bn == 256) && pl.bk == 64 &&
         pl.stages >= 2 && pl.stages <= 8 && pl.raster_group >= 1 && pl.grid >= 0;
}

uint32_t smem_for(int bn, int stages) {
  switch (bn) {
    case 64: return tl::smem_bytes_for<64>(stages);
    case 128: return tl::smem_bytes_for<128>(stages);
    default: return tl::smem_bytes_for<256>(stages);
  }
}

tl_status validate_common(int64_t M, int64_t N, int64_t K, tl_dtype dtype, int trans_a,
                          int trans_b) {
  if (M < 0 || N < 0 || K < 0) return TL_ERR_INVALID_ARG;
  if (dtype != TL_F16 && dtype != TL_BF16) return TL_ERR_INVALID_ARG;
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

tl_status complete_plan(int64_t M, int64_t N, int64_t K, int num_sms, tl_plan* pl) {
  if (!plan_supported(*pl)) return TL_ERR_INVALID_ARG;
  const int sms = num_sms > 0 ? num_sms : kDefaultSms;
  pl->tiles_m = ceil_div(M, pl->bm);
  pl->tiles_n = ceil_div(N, pl->bn);
  pl->tiles = pl->tiles_m * pl->tiles_n;
  pl->k_blocks = ceil_div(K, pl->bk);
  pl->ring_bytes = static_cast<int64_t>(pl->stages) * (pl->bm * pl->bk + pl->bn * pl->bk) * 2;
  pl->smem_bytes = smem_for(pl->bn, pl->stages);
  if (pl->smem_bytes > kMaxSmemPerCta) return TL_ERR_INVALID_ARG;
  pl->tmem_cols = 2 * pl->bn;
  pl->tx_bytes = (pl->bm + pl->bn) * pl->bk * 2;
  const int64_t want = pl->grid > 0 ? pl->grid : sms;
  pl->grid = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(want, pl->tiles)));
  if (pl->tiles > (int64_t{1} << 31) - 1) return TL_ERR_UNSUPPORTED;
  if (pl->l2_prefetch < 0) pl->l2_prefetch = default_prefetch(*pl);
  if (pl->l2_prefetch > 1024) return TL_ERR_INVALID_ARG;
  return TL_OK;
}

// Choose BN and the ring depth: fewest waves of tiles over the SMs, weighted by the
// per-tile cost of each width (narrower tiles re-read A more often and issue
// smaller MMAs).  Depth fills the shared memory left after the staging buffers.
void choose_tiling(int64_t M, int64_t N, int64_t K, int sms, tl_plan* pl) {
  (void)K;
  // Relative time of one tile per unit of K, measured on GB300: a 128-wide tile runs
  // at ~0.64 of the per-SM rate of a 256-wide one, a 64-wide one lower still.
  struct Cand { int bn, stages; double tile_cost; };
  const Cand cands[] = {{256, 4, 2.0}, {128, 6, 1.56}, {64, 8, 1.2}};
  double best = 0.0;
  int pick = 0;
  for (int i = 0; i < 3; ++i) {
    const int64_t tiles = ceil_div(M, 128) * ceil_div(N, cands[i].bn);
    const int64_t waves = ceil_div(tiles, sms);
    const double cost = static_cast<double>(waves) * cands[i].tile_cost;
    if (i == 0 || cost < best - 1e-9) {
      best = cost;
      pick = i;
    }
  }
  pl->bm = 128;
  pl->bn = cands[pick].bn;
  pl->bk = 64;
  pl->stages = cands[pick].stages;
  pl->raster_group = 16;
  pl->grid = 0;
  pl->l2_prefetch = -1;
}



template <int BN>
tl_status launch_bn(DeviceState* st, const tl_plan& pl, const CUtensorMap& ta,
                    const CUtensorMap& tb, const CUtensorMap& tc, const tl::GemmParams& prm,
                    cudaStream_t stream) {
  constexpr uint32_t bit = BN == 64 ? 1u : (BN == 128 ? 2u : 4u);
  auto kern = tl::tl_gemm_kernel<BN>;
  if (!(st->attr_done.load(std::memory_order_acquire) & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             st->smem_optin) != cudaSuccess) {
      (void)cudaGetLastError();
      return TL_ERR_LAUNCH;
    }
    st->attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.grid));
  cfg.blockDim = dim3(tl::kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(pl.smem_bytes);
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  if (cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, prm) != cudaSuccess) {
    (void)cudaGetLastError();
    return TL_ERR_LAUNCH;
  }
  return TL_OK;
}

bool encode_2d(CUtensorMap* map, tl_dtype dtype, const void* base, uint64_t inner, uint64_t outer,
               uint64_t ld_elems, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld_elems * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      dtype == TL_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch_blocks_for(int64_t elems) {
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ceil_div(elems, 256 * 4), 4096)));
}

tl_status run(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
              int64_t lda, int64_t ldb, int64_t ldc, tl_dtype dtype, int trans_a, int trans_b,
              tl_epilogue epilogue, const tl_plan* forced, cudaStream_t stream) {
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
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 1u)
      return TL_ERR_ALIGNMENT;
    uintptr_t c0, c1, a0, a1, b0, b1;
    extent(C, M, N, ldc, &c0, &c1);
    extent(A, a_rows, a_cols, lda, &a0, &a1);
    extent(B, b_rows, b_cols, ldb, &b0, &b1);
    if (overlaps(c0, c1, a0, a1) || overlaps(c0, c1, b0, b1)) return TL_ERR_ALIAS;
  }
  int dev = 0;
  DeviceState* st = device_state(&dev);
  if (st == nullptr) return TL_ERR_DEVICE;
  if (!st->sm103) return TL_ERR_UNSUPPORTED;
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
  } else {
    choose_tiling(M, N, K, st->sms, &pl);
  }
  if ((s = complete_plan(M, N, K, st->sms, &pl)) != TL_OK) return s;
  if (pl.smem_bytes > st->smem_optin) return TL_ERR_INVALID_ARG;

  // Operands the TMA unit cannot address directly go through a padded copy.
  const bool repack_a = !tma_ok(A, lda);
  const bool repack_b = !tma_ok(B, ldb);
  const int64_t lda_w = repack_a ? ceil_div(a_cols, 8) * 8 : lda;
  const int64_t ldb_w = repack_b ? ceil_div(b_cols, 8) * 8 : ldb;
  const int64_t ws_a = repack_a ? a_rows * lda_w * 2 : 0;
  const int64_t ws_b = repack_b ? b_rows * ldb_w * 2 : 0;
  void* ws = nullptr;
  const void* a_use = A;
  const void* b_use = B;
  if (ws_a + ws_b > 0) {
    const int64_t ws_a_rounded = ceil_div(ws_a, 256) * 256;
    if (cudaMallocAsync(&ws, static_cast<size_t>(ws_a_rounded + ws_b), stream) != cudaSuccess) {
      (void)cudaGetLastError();
      return TL_ERR_LAUNCH;
    }
    uint8_t* w = static_cast<uint8_t*>(ws);
    if (repack_a) {
      tl::tl_repack_kernel<<<launch_blocks_for(a_rows * a_cols), 256, 0, stream>>>(
          static_cast<const uint16_t*>(A), reinterpret_cast<uint16_t*>(w), a_rows, a_cols, lda,
          lda_w);
      a_use = w;
    }
    if (repack_b) {
      uint8_t* wb = w + ws_a_rounded;
      tl::tl_repack_kernel<<<launch_blocks_for(b_rows * b_cols), 256, 0, stream>>>(
          static_cast<const uint16_t*>(B), reinterpret_cast<uint16_t*>(wb), b_rows, b_cols, ldb,
          ldb_w);
      b_use = wb;
    }
    if (cudaGetLastError() != cudaSuccess) {
      (void)cudaFreeAsync(ws, stream);
      return TL_ERR_LAUNCH;
    }
  }
  const bool tma_store = tma_ok(C, ldc);

  CUtensorMap ta, tb, tc;
  std::memset(&tc, 0, sizeof(tc));
  bool enc_ok = true;
  if (!trans_a) enc_ok &= encode_2d(&ta, dtype, a_use, K, M, lda_w, 64, 128);
  else enc_ok &= encode_2d(&ta, dtype, a_use, M, K, lda_w, 64, 64);
  if (trans_b) enc_ok &= encode_2d(&tb, dtype, b_use, K, N, ldb_w, 64, pl.bn);
  else enc_ok &= encode_2d(&tb, dtype, b_use, N, K, ldb_w, 64, 64);
  if (tma_store) enc_ok &= encode_2d(&tc, dtype, C, N, M, ldc, 64, 32);
  if (!enc_ok) {
    if (ws) (void)cudaFreeAsync(ws, stream);
    return TL_ERR_LAUNCH;
  }

  tl::GemmParams prm;
  std::memset(&prm, 0, sizeof(prm));
  prm.M = static_cast<int32_t>(M);
  prm.N = static_cast<int32_t>(N);
  prm.K = static_cast<int32_t>(K);
  prm.tiles_m = static_cast<int32_t>(pl.tiles_m);
  prm.tiles_n = static_cast<int32_t>(pl.tiles_n);
  prm.num_tiles = static_cast<int32_t>(pl.tiles);
  prm.k_blocks = static_cast<int32_t>(pl.k_blocks);
  prm.stages = pl.stages;
  prm.raster_group = pl.raster_group;
  prm.trans_a = trans_a;
  prm.trans_b = trans_b;
  prm.bf16 = dtype == TL_BF16 ? 1 : 0;
  prm.relu = epilogue == TL_EPI_RELU ? 1 : 0;
  prm.tma_store = tma_store ? 1 : 0;
  prm.l2_prefetch = pl.l2_prefetch;
  prm.idesc = tl::mma_idesc_f16(prm.bf16, trans_a ? 1u : 0u, trans_b ? 0u : 1u, 128u,
                                static_cast<uint32_t>(pl.bn));
  prm.C = C;
  prm.ldc = ldc;
  prm.status = st->status;
  prm.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);

  switch (pl.bn) {
    case 64: s = launch_bn<64>(st, pl, ta, tb, tc, prm, stream); break;
    case 128: s = launch_bn<128>(st, pl, ta, tb, tc, prm, stream); break;
    default: s = launch_bn<256>(st, pl, ta, tb, tc, prm, stream); break;
  }
  if (ws) {
    if (cudaFreeAsync(ws, stream) != cudaSuccess) {
      (void)cudaGetLastError();
      if (s == TL_OK) s = TL_ERR_LAUNCH;
    }
  }
  return s;
}

}  // namespace

extern "C" {

tl_status tl_gemm(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                  int64_t lda, int64_t ldb, int64_t ldc, tl_dtype dtype, int trans_a,
                  int trans_b, tl_epilogue epilogue, tl_stream_t stream) {
  return run(A, B, C, M, N, K, lda, ldb, ldc, dtype, trans_a, trans_b, epilogue, nullptr,
             reinterpret_cast<cudaStream_t>(stream));
}

tl_status tl_gemm_with_plan(const void* A, const void* B, void* C, int64_t M, int64_t N,
                            int64_t K, int64_t lda, int64_t ldb, int64_t ldc, tl_dtype dtype,
                            int trans_a, int trans_b, tl_epilogue epilogue, const tl_plan* plan,
                            tl_stream_t stream) {
  if (plan == nullptr) return TL_ERR_INVALID_ARG;
  return run(A, B, C, M, N, K, lda, ldb, ldc, dtype, trans_a, trans_b, epilogue, plan,
             reinterpret_cast<cudaStream_t>(stream));
}

tl_status tl_gemm_plan(int64_t M, int64_t N, int64_t K, tl_dtype dtype, int trans_a, int trans_b,
                       int num_sms, tl_plan* plan) {
  if (plan == nullptr) return TL_ERR_NULL_PTR;
  const tl_status s = validate_common(M, N, K, dtype, trans_a, trans_b);
  if (s != TL_OK) return s;
  std::memset(plan, 0, sizeof(*plan));
  const int sms = num_sms > 0 ? num_sms : kDefaultSms;
  choose_tiling(M, N, K, sms, plan);
  return complete_plan(M, N, K, sms, plan);
}

tl_status tl_plan_complete(int64_t M, int64_t N, int64_t K, tl_dtype dtype, int trans_a,
                           int trans_b, int num_sms, tl_plan* plan) {
  if (plan == nullptr) return TL_ERR_NULL_PTR;
  const tl_status s = validate_common(M, N, K, dtype, trans_a, trans_b);
  if (s != TL_OK) return s;
  if (plan->raster_group <= 0) plan->raster_group = 16;
  const int32_t pf = plan->l2_prefetch;
  std::memset(&plan->tiles_m, 0, sizeof(tl_plan) - offsetof(tl_plan, tiles_m));
  plan->l2_prefetch = pf;
  return complete_plan(M, N, K, num_sms, plan);
}

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

void tl_set_wait_timeout_ns(uint64_t ns) {
  ns = std::max<uint64_t>(100000ull, std::min<uint64_t>(ns, 60000000000ull));
  g_timeout_ns.store(ns, std::memory_order_relaxed);
}

int tl_version(void) { return 100; }

}  // extern "C"
