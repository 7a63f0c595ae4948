// C ABI of the fp8 paged decode attention library (see include/pda.h):
// argument validation, the split-count heuristic, the per-stream workspace,
// and the launches of the split-KV decode and merge kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/pda.h"
#include "pda_kernels.cuh"

namespace {

using pda::kHeadDim;

std::atomic<int> g_split_override{0};
// Tail pieces of the persistent kernel (pda_set_tail_split); on by default.
std::atomic<int> g_tail_split{1};
// Four-row TMA gathers of scale rows and 16-token pages (pda_set_tma_gather);
// on by default.
std::atomic<int> g_tma_gather{1};
// pda_set_block_check: the pool size the decode kernels check block ids
// against (0 = no check), clamped to 2^31 (every int32 id below it).
std::atomic<uint32_t> g_block_limit{0u};
std::atomic<cudaEvent_t> g_prof_before{nullptr};
std::atomic<cudaEvent_t> g_prof_after{nullptr};

// Decode kernel instances the library launches.
enum KernelKind {
  kPlainWide = 0,
  kPlainDense,
  kSlotWide,
  kTokenWide,
  kTokenDense,
  kPersistWide,   // persistent, page-major pages
  kPersistToken,  // persistent, token-major pages through tensor maps
  kPersistSlot,   // persistent, page-major pages with per-slot scale tables
  kNumKinds
};
bool is_persistent(int k) { return k == kPersistWide || k == kPersistToken || k == kPersistSlot; }
// The per-unit instance that takes a persistent instance's calls when the
// persistent kernel cannot (past 2^31 units, or captured without a workspace).
KernelKind per_unit_of(KernelKind k) {
  return k == kPersistToken ? kTokenWide : (k == kPersistSlot ? kSlotWide : kPlainWide);
}

// Forgets pda_decode_noalloc's per-device set-up (defined with it below).
void noalloc_forget_devices();

struct DeviceInfo {
  int sm_count = 0;
  int cluster_launch = -1;                // cudaDevAttrClusterLaunch (-1: not read yet)
  int ctas_per_sm[kNumKinds][9] = {{0}};  // [instance][bs/16 (1..8)]
  bool smem_attr_set = false;
  // co-resident clusters of n split CTAs: [instance][bs/16][n] (-1: not asked yet)
  int max_clusters[kNumKinds][9][17];
  DeviceInfo() {
    for (auto& a : max_clusters)
      for (auto& b : a)
        for (int& c : b) c = -1;
  }
};
std::mutex g_dev_mu;
std::map<int, DeviceInfo> g_devices;

struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
  // Buffers this one replaced when it grew. A CUDA graph captured earlier
  // keeps their addresses in its kernel parameters, so they stay allocated
  // until pda_release.
  std::vector<void*> retired;
};
std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;
// Staging buffers of pda_decode_host, per (device, stream); under g_ws_mu.
std::map<std::pair<int, cudaStream_t>, Workspace> g_stage;

// Ring geometry for a block size: a stage holds max(16 * consumer warps, bs)
// tokens of K and V (whole pages); about kRingBytes of stages per CTA.
struct RingShape {
  int pages_per_stage;
  int num_stages;
  uint32_t stage_bytes;
  uint32_t scale_off;
  size_t smem_bytes;
};

RingShape ring_shape(int bs, bool slot_scales = false, int ring_bytes = pda::kRingBytes) {
  RingShape r;
  r.pages_per_stage = bs < pda::kStageTokensMin ? pda::kStageTokensMin / bs : 1;
  r.scale_off = 2u * (uint32_t)r.pages_per_stage * (uint32_t)(kHeadDim * bs);
  r.stage_bytes = r.scale_off + (slot_scales ? 2u * (uint32_t)r.pages_per_stage * (uint32_t)bs * 4u : 0u);
  r.num_stages = (int)((uint32_t)ring_bytes / r.scale_off);  // scale rows ride on top
  if (r.num_stages < 2) r.num_stages = 2;
  size_t ring = (size_t)r.num_stages * r.stage_bytes;
  // the CTA merge area, then the cluster merge's partial
  size_t merge = (size_t)pda::kClusterPartOff + pda::kClusterPartBytes;
  if (ring < merge) ring = merge;
  // + 1 KiB so the kernel can align the ring to 1024 bytes (128-byte swizzle).
  r.smem_bytes = ring + 2 * 8 * (size_t)r.num_stages + 16 + 1024;
  return r;
}

// Persistent-kernel ring: stages of K and V pages, each a multiple of 1 KiB
// (swizzled tensor-map pages need 1 KiB alignment) and at least the merge
// rows; then one side entry per stage (query rows, merge (m, l), header);
// then full and empty barriers per stage plus one consumer barrier.
// With per-slot scales the side entries are kAuxBytesSlot long and a
// stage's scale rows (2 x pages x bs floats) sit at the end of the entry's
// query-row area: scale_off is that offset within the entry.
RingShape persistent_ring_shape(int bs, bool slot_scales = false) {
  RingShape r = ring_shape(bs);
  const uint32_t kv = r.scale_off;
  uint32_t st = kv > pda::kPersistMergeBytes ? kv : pda::kPersistMergeBytes;
  st = (st + 1023u) & ~1023u;
  r.stage_bytes = st;
  r.num_stages = (int)((uint32_t)pda::kPersistRingBytes / st);
  if (r.num_stages < 2) r.num_stages = 2;
  const uint32_t aux = slot_scales ? pda::kAuxBytesSlot : pda::kAuxBytes;
  r.scale_off = slot_scales ? pda::kAuxMl - 2u * (uint32_t)r.pages_per_stage * (uint32_t)bs * 4u : 0u;
  r.smem_bytes = (size_t)r.num_stages * (st + aux) + 8 * (2 * (size_t)r.num_stages + 1) + 16 + 1024;
  return r;
}

// The persistent slot-scale instance fits a GQA group whose query rows
// (g x 256 bytes) leave room in the side entry for a stage's scale rows.
bool slot_persistent_fits(int gqa, int bs) {
  const RingShape r = persistent_ring_shape(bs, true);
  return (uint32_t)gqa * kHeadDim * 2u <= r.scale_off;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Cache writes of up to this many (token, kv head) items use the scattered
// writer (one warp per item).
#ifndef PDA_SCATTER_WRITE_MAX_ITEMS
#define PDA_SCATTER_WRITE_MAX_ITEMS 2048
#endif
constexpr long long kScatterWriteMaxItems = PDA_SCATTER_WRITE_MAX_ITEMS;

// Placeholder tensor maps for the page-major kernels (never dereferenced).
const CUtensorMap g_no_map = {};

// ---- token-major (strided) caches: tensor maps built on the host per call.

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once (no libcuda link).
EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

struct TokenMajorMaps {
  CUtensorMap k;
  CUtensorMap v;
  int dim_token, dim_head, dim_block;  // positions 1..3 in both maps
};

// One 4-D map over a cache whose row of 128 bytes for (block b, token t,
// kv head h) starts at base + b*sb + t*st + h*sh. Dimension 0 is the row's
// bytes; dimensions 1..3 are token, head and block sorted by stride, which
// must nest without overlap. The box is one page: all bs tokens of one
// (block, head), landing as [bs][128] with 128-byte swizzle.
pda_status make_token_major_map(const void* base, long long nb, int hk, int bs, long long sb, long long st,
                                long long sh, CUtensorMap* map, int* pos_token, int* pos_head, int* pos_block) {
  struct D {
    long long stride, extent;
    int what;  // 0 token, 1 head, 2 block
  } d[3] = {{st, bs, 0}, {sh, hk, 1}, {sb, nb, 2}};
  for (auto& x : d)
    if (x.stride <= 0 || (x.stride & 15) != 0 || x.extent <= 0 || x.extent > (1LL << 32) || x.stride >= (1LL << 40))
      return PDA_ERR_INVALID_ARG;
  // Sort by stride, dimensions of extent 1 (a single kv head or block,
  // whose stride is never used) last; those then get the stride that nests
  // exactly after the dimension before them.
  auto before = [](const D& a, const D& b) {
    if ((a.extent == 1) != (b.extent == 1)) return b.extent == 1;
    return a.extent != 1 && a.stride < b.stride;
  };
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (before(d[j], d[i])) std::swap(d[i], d[j]);
  for (int i = 1; i < 3; ++i)
    if (d[i].extent == 1) d[i].stride = d[i - 1].stride * d[i - 1].extent;
  if (d[0].stride < kHeadDim || d[1].stride < d[0].stride * d[0].extent || d[2].stride < d[1].stride * d[1].extent ||
      d[1].stride >= (1LL << 40) || d[2].stride >= (1LL << 40))
    return PDA_ERR_UNSUPPORTED;  // rows overlap: not a layout a tensor map can describe
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return PDA_ERR_CUDA;
  cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)d[0].extent, (cuuint64_t)d[1].extent,
                        (cuuint64_t)d[2].extent};
  cuuint64_t strides[3] = {(cuuint64_t)d[0].stride, (cuuint64_t)d[1].stride, (cuuint64_t)d[2].stride};
  cuuint32_t box[4] = {(cuuint32_t)kHeadDim, 1, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  for (int i = 0; i < 3; ++i) {
    if (d[i].what == 0) {
      box[1 + i] = (cuuint32_t)bs;
      *pos_token = 1 + i;
    } else if (d[i].what == 1) {
      *pos_head = 1 + i;
    } else {
      *pos_block = 1 + i;
    }
  }
  if (enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PDA_ERR_INVALID_ARG;
  return PDA_OK;
}

// Native V pages [NB][Hk][128][bs] of 32-, 64- or 128-token blocks through a
// tensor map with the TMA swizzle whose span is one page row (bs bytes): the
// box is one page (bs x 128 rows of one kv head of one block). The block
// extent is the int32 id range (the entry points are not told the pool
// size; reads stay where the table points, as with 1-D copies). Returns the
// kernel's swizzle mode, or kVSwizzleNone (then *map is unused) for other
// block sizes or when the driver entry point is missing.
int make_v_swizzle_map(const void* v_cache, int hk, int bs, CUtensorMap* map) {
  CUtensorMapSwizzle sw;
  int mode;
  switch (bs) {
    case 32: sw = CU_TENSOR_MAP_SWIZZLE_32B; mode = pda::kVSwizzle32; break;
    case 64: sw = CU_TENSOR_MAP_SWIZZLE_64B; mode = pda::kVSwizzle64; break;
    case 128: sw = CU_TENSOR_MAP_SWIZZLE_128B; mode = pda::kVSwizzle128; break;
    default: return pda::kVSwizzleNone;
  }
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return pda::kVSwizzleNone;
  const cuuint64_t dims[4] = {(cuuint64_t)bs, (cuuint64_t)kHeadDim, (cuuint64_t)hk, (cuuint64_t)INT32_MAX};
  const cuuint64_t strides[3] = {(cuuint64_t)bs, (cuuint64_t)kHeadDim * bs, (cuuint64_t)hk * kHeadDim * bs};
  const cuuint32_t box[4] = {(cuuint32_t)bs, (cuuint32_t)kHeadDim, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  if (enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(v_cache), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
      CUDA_SUCCESS)
    return pda::kVSwizzleNone;
  return mode;
}

// A per-slot scale table [NB][Hk][bs] (fp32) as a 2-D tensor map of rows
// b * Hk + h, bs floats each, for four-row gathers (box: one row). The row
// extent is the int32 range, as the entry points are not told the pool
// size; rows are read only where the block table points. False when the
// driver entry point is missing or refuses the map.
bool make_scale_row_map(const float* table, int bs, CUtensorMap* map) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)bs, (cuuint64_t)INT32_MAX};
  const cuuint64_t strides[1] = {(cuuint64_t)bs * sizeof(float)};
  const cuuint32_t box[2] = {(cuuint32_t)bs, 1};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(table), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A page-major cache of 16-token pages ([NB][Hk] pages of 2 KiB) as a 2-D
// tensor map of rows b * Hk + h, one page each (256 8-byte elements), for
// four-page gathers (box: one row). Row extent as in make_scale_row_map.
bool make_page_row_map(const void* cache, CUtensorMap* map) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)(kHeadDim * 16 / 8), (cuuint64_t)INT32_MAX};
  const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 16};
  const cuuint32_t box[2] = {(cuuint32_t)(kHeadDim * 16 / 8), 1};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(cache), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The checks of sizes and scalars every decode entry point makes.
pda_status validate_sizes(int num_seqs, int num_heads, int num_kv_heads, int head_size, int block_size,
                          int max_blocks, float scale, float k_scale, float v_scale) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 ||
      max_blocks < 0)
    return PDA_ERR_INVALID_ARG;
  if (num_heads % num_kv_heads != 0) return PDA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale)) return PDA_ERR_INVALID_ARG;
  if (head_size != kHeadDim) return PDA_ERR_UNSUPPORTED;
  if (block_size % 16 != 0 || block_size > 128) return PDA_ERR_UNSUPPORTED;
  const int g = num_heads / num_kv_heads;
  if (g > pda::kMaxGqa) return PDA_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PDA_ERR_UNSUPPORTED;
  if ((long long)max_blocks * block_size > (long long)INT32_MAX / 2) return PDA_ERR_UNSUPPORTED;
  return PDA_OK;
}

pda_status validate(const void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* seq_lens, int num_seqs, int num_heads,
                    int num_kv_heads, int head_size, int block_size, int max_blocks, float scale,
                    float k_scale, float v_scale) {
  const pda_status st =
      validate_sizes(num_seqs, num_heads, num_kv_heads, head_size, block_size, max_blocks, scale, k_scale, v_scale);
  if (st != PDA_OK || num_seqs == 0) return st;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PDA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return PDA_ERR_INVALID_ARG;
  return PDA_OK;
}

bool is_dense(KernelKind k) { return k == kPlainDense || k == kTokenDense; }
bool is_slot(KernelKind k) { return k == kSlotWide || k == kPersistSlot; }

RingShape ring_for(KernelKind k, int bs) {
  if (is_persistent(k)) return persistent_ring_shape(bs, k == kPersistSlot);
  return ring_shape(bs, is_slot(k), is_dense(k) ? pda::kDenseRingBytes : pda::kRingBytes);
}

// Kernel function types of the decode instances.
using SplitFn = void (*)(const pda::DecodeParams, const CUtensorMap, const CUtensorMap);
using PersistFn = void (*)(const pda::DecodeParams, unsigned*, int, const CUtensorMap, const CUtensorMap);

// Each decode instance comes in two builds: paired PV columns for GQA groups
// of at most 4 heads, a second PV MMA for wider groups (see TileWorker).
bool paired_for(int gqa) { return gqa <= pda::kMaxGqa / 2; }

template <bool kPaired>
SplitFn split_fn_of(KernelKind k) {
  switch (k) {
    case kPlainWide: return pda::pda_split_decode_kernel<false, false, pda::kWideCtasPerSm, kPaired, false>;
    case kPlainDense: return pda::pda_split_decode_kernel<false, false, pda::kDenseCtasPerSm, kPaired, false>;
    case kSlotWide: return pda::pda_split_decode_kernel<true, false, pda::kWideCtasPerSm, kPaired, false>;
    case kTokenWide: return pda::pda_split_decode_kernel<false, true, pda::kWideCtasPerSm, kPaired, false>;
    case kTokenDense: return pda::pda_split_decode_kernel<false, true, pda::kDenseCtasPerSm, kPaired, false>;
    default: return nullptr;
  }
}
// Cluster-merging builds of the instances that run one-wave split grids
// (none for the wide plain and token-major instances: those run only
// multi-wave grids).
template <bool kPaired>
SplitFn cluster_fn_of(KernelKind k) {
  switch (k) {
    case kPlainDense: return pda::pda_split_decode_kernel<false, false, pda::kDenseCtasPerSm, kPaired, true>;
    case kSlotWide: return pda::pda_split_decode_kernel<true, false, pda::kWideCtasPerSm, kPaired, true>;
    case kTokenDense: return pda::pda_split_decode_kernel<false, true, pda::kDenseCtasPerSm, kPaired, true>;
    default: return nullptr;
  }
}
SplitFn split_fn(KernelKind k, bool paired, bool cluster = false) {
  if (cluster) return paired ? cluster_fn_of<true>(k) : cluster_fn_of<false>(k);
  return paired ? split_fn_of<true>(k) : split_fn_of<false>(k);
}

PersistFn persist_fn(KernelKind k, bool paired) {
  if (k == kPersistToken)
    return paired ? pda::pda_persistent_decode_kernel<false, true, pda::kPersistCtasPerSm, true>
                  : pda::pda_persistent_decode_kernel<false, true, pda::kPersistCtasPerSm, false>;
  if (k == kPersistSlot)
    return paired ? pda::pda_persistent_decode_kernel<true, false, pda::kPersistCtasPerSm, true>
                  : pda::pda_persistent_decode_kernel<true, false, pda::kPersistCtasPerSm, false>;
  return paired ? pda::pda_persistent_decode_kernel<false, false, pda::kPersistCtasPerSm, true>
                : pda::pda_persistent_decode_kernel<false, false, pda::kPersistCtasPerSm, false>;
}

const void* kernel_fn(KernelKind k, bool paired) {
  if (is_persistent(k)) return (const void*)persist_fn(k, paired);
  return (const void*)split_fn(k, paired);
}

// SM count and resident CTAs per SM of instance `kind` for block size bs.
pda_status device_info(int dev, int bs, int* sm_count, int* ctas_per_sm, KernelKind kind = kPlainWide) {
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& di = g_devices[dev];
  if (di.sm_count == 0) {
    if (cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      di.sm_count = 0;
      return PDA_ERR_CUDA;
    }
  }
  if (di.cluster_launch < 0) {
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrClusterLaunch, dev) != cudaSuccess) return PDA_ERR_CUDA;
    di.cluster_launch = c ? 1 : 0;
  }
  if (!di.smem_attr_set) {
    // Opt every instance in to the largest ring any block size uses.
    size_t mx = 0;
    for (int b = 16; b <= 128; b += 16)
      for (int k = 0; k < kNumKinds; ++k) {
        const size_t sb = ring_for((KernelKind)k, b).smem_bytes;
        mx = sb > mx ? sb : mx;
      }
    for (int k = 0; k < kNumKinds; ++k)
      for (bool paired : {false, true}) {
        if (cudaFuncSetAttribute(kernel_fn((KernelKind)k, paired), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)mx) != cudaSuccess)
          return PDA_ERR_CUDA;
        const SplitFn cf = split_fn((KernelKind)k, paired, true);
        // clusters of up to 16 split CTAs (8 is the portable limit)
        if (cf && (cudaFuncSetAttribute(cf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mx) != cudaSuccess ||
                   cudaFuncSetAttribute(cf, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess))
          return PDA_ERR_CUDA;
      }
    di.smem_attr_set = true;
  }
  int& occ = di.ctas_per_sm[kind][bs / 16];
  if (occ == 0) {
    // the smaller residency of the two builds (the plan does not depend on g)
    int m = 0;
    for (bool paired : {false, true}) {
      int n = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel_fn(kind, paired), pda::kThreads,
                                                        ring_for(kind, bs).smem_bytes) != cudaSuccess)
        return PDA_ERR_CUDA;
      m = (m == 0 || n < m) ? n : m;
    }
    occ = m > 0 ? m : 1;
  }
  *sm_count = di.sm_count;
  *ctas_per_sm = occ;
  return PDA_OK;
}

int resolve_splits(int num_seqs, int num_kv_heads, int max_blocks, int bs, int sm_count, int ctas_per_sm,
                   int override_splits) {
  int n = override_splits;
  if (n <= 0) n = pda_choose_splits(num_seqs, num_kv_heads, max_blocks, bs, sm_count, ctas_per_sm);
  const int cap = max_blocks > 0 ? max_blocks : 1;
  if (n > cap) n = cap;
  if (n < 1) n = 1;
  return n;
}

// The wide instances of plain and token-major calls: the persistent kernel
// unless built out.
#ifdef PDA_DISABLE_PERSISTENT
constexpr KernelKind kWidePlain = kPlainWide;
constexpr KernelKind kWideToken = kTokenWide;
constexpr bool kPersistentSlot = false;
#else
constexpr KernelKind kWidePlain = kPersistWide;
constexpr KernelKind kWideToken = kPersistToken;
constexpr bool kPersistentSlot = true;
#endif

// The wide instance of per-slot-scale calls: the persistent kernel when the
// group's query rows leave room for the scale rows (g <= 6 at 16- to 64-token
// blocks), else the per-unit kernel. Its one-wave grids run the per-unit
// kernel (plan_from).
KernelKind slot_wide_kind(int gqa, int bs) {
  return (kPersistentSlot && slot_persistent_fits(gqa, bs)) ? kPersistSlot : kSlotWide;
}

// Split count and kernel instance for a call: the wide instance (3 CTAs per
// SM, 64 KiB ring) unless its planned grid fits one wave of the dense
// instance (4 CTAs per SM, 48 KiB ring), which then runs the whole batch at
// once (measured on GB300: 64 x 1K-token batch 27.6 us dense vs 37.3 us wide;
// large and ragged batches are faster wide).
struct Plan {
  KernelKind kind;
  int nsplit;
  unsigned grid = 0;         // persistent kernel: CTAs (resident slots, at most one per unit)
  long long ordered = 0;     // persistent kernel: units handed out longest first (0: ticket order)
  bool cluster = false;      // per-unit kernel: the splits merge inside their cluster (no merge kernel)
  // persistent kernel, tail pieces (0 units: none): the last tail_units
  // units handed out are cut into at most max_pieces pieces of at least
  // min_piece_pages pages
  int tail_units = 0;
  int max_pieces = 1;
  int min_piece_pages = 1;
};

// Smallest tail piece: 256 tokens.
int tail_min_piece_pages(int bs) { return (256 + bs - 1) / bs; }

// Largest batch (in work units) whose units the persistent kernel takes in
// longest-first order.
constexpr long long kMaxOrderedUnits = pda::kMaxOrderedUnits;


// The plan from sizes and residency alone (host only): split count with
// the wide instance's CTAs per SM; the dense instance when that grid fits
// one wave of it; the per-unit kernel instead of the persistent one past
// 2^31 units (32-bit tickets); the persistent grid and how many units it
// hands out in longest-first order.
Plan plan_from(int num_seqs, int num_kv_heads, int max_blocks, int bs, int sms, int occ, int occ_d, KernelKind wide,
               KernelKind dense, int override_splits) {
  Plan pl;
  const int MB = max_blocks > 0 ? max_blocks : 1;
  pl.kind = wide;
  pl.nsplit = resolve_splits(num_seqs, num_kv_heads, MB, bs, sms, occ, override_splits);
  if (dense != wide) {
    const long long ctas = (long long)num_seqs * num_kv_heads * pl.nsplit;
    // per-slot scales: the per-unit kernel for one wave (its splits can
    // merge in clusters), the persistent one past it
    const bool one_wave_slot = wide == kPersistSlot && ctas <= (long long)sms * occ;
    if ((occ_d > occ && ctas <= (long long)sms * occ_d) || one_wave_slot) {
      pl.kind = dense;
      pl.nsplit = resolve_splits(num_seqs, num_kv_heads, MB, bs, sms, occ_d, override_splits);
    }
  }
  if (is_persistent(pl.kind) && (long long)num_seqs * num_kv_heads * pl.nsplit > INT32_MAX) {
    // The persistent kernel counts units in 32-bit tickets; the per-unit
    // kernel's grid (splits, kv heads, sequences) has no such bound.
    pl.kind = per_unit_of(pl.kind);
  }
  if (is_persistent(pl.kind)) {
    const long long units = (long long)num_seqs * num_kv_heads * pl.nsplit;
    const long long slots = (long long)sms * occ;
    pl.grid = (unsigned)(units < slots ? units : slots);
    pl.ordered = (units > slots && units <= kMaxOrderedUnits) ? units - slots : 0;
    if (pl.ordered > 0) {
      // The units of the last, partial round of hand-outs are cut into
      // pieces that the CTAs done with their whole units share (GB300,
      // 256 x 4096 tokens: the last 224 units of 2048 over 456 CTAs left
      // half the CTAs idle for the call's last 50 us). A piece holds at
      // least 256 tokens, and units under 1024 tokens stay whole; the tail
      // merge kernel folds the pieces (into the split's partial with several
      // splits). A tail of a third of the CTAs or more is cut into pieces
      // that shrink toward the end (up to kMaxTailPieces), a smaller one
      // into equal pieces, about two per CTA (the order kernel's
      // tail_piece_count).
      const long long k = units % (long long)pl.grid;
      if (k > 0) {
        pl.tail_units = (int)(k < pda::kOrderThreads ? k : pda::kOrderThreads);
        pl.max_pieces = pda::tail_piece_cap(pl.tail_units, (int)pl.grid);
        pl.min_piece_pages = tail_min_piece_pages(bs);
      }
    }
  } else if (pl.nsplit >= 2 && pl.nsplit <= pda::kMaxClusterSplits) {
    // A one-wave grid of the per-unit kernel merges each unit's splits in
    // a cluster of nsplit CTAs, with no merge launch and no fp32 partials
    // (GB300, us per call against the merge kernel: 19 x 4 units of 4K
    // tokens in 8 splits 20.1 vs 21.3, 4 x 8 units of 4K in 16 splits 14.0
    // vs 14.9, 16 x 8 units of 1K in 4 splits 12.7 vs 12.7).
    const long long ctas = (long long)num_seqs * num_kv_heads * pl.nsplit;
    pl.cluster = ctas <= (long long)sms * (pl.kind == wide ? occ : occ_d);
  }
  return pl;
}

// Launch attributes of a cluster-merged per-unit grid: the nsplit CTAs of
// each unit (grid x) form one cluster. Under the default scheduling policy a
// full wave of clusters of 8 did not fit at once (a 608-CTA batch took
// 30.0 us instead of 21.4 us with the merge kernel); letting the hardware
// balance the clusters' CTAs over the SMs fits them (20.1 us, GB300).
int cluster_attrs(cudaLaunchAttribute* attr, int nsplit) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)nsplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
  attr[1].val.clusterSchedulingPolicyPreference = cudaClusterSchedulingPolicyLoadBalancing;
  return 2;
}

// Clusters of nsplit CTAs of instance kind that the device holds at once (0
// when it cannot launch them), cached per device.
pda_status max_active_clusters(int dev, KernelKind kind, int bs, int nsplit, int* out) {
  *out = 0;
  if (nsplit < 2 || nsplit > pda::kMaxClusterSplits || !split_fn(kind, false, true)) return PDA_OK;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& di = g_devices[dev];
  int& n = di.max_clusters[kind][bs / 16][nsplit];
  if (n < 0) {
    n = 0;
    if (di.cluster_launch == 1) {
      cudaLaunchConfig_t lc = {};
      lc.gridDim = dim3((unsigned)nsplit, 1, 1);
      lc.blockDim = dim3(pda::kThreads);
      lc.dynamicSmemBytes = ring_for(kind, bs).smem_bytes;
      cudaLaunchAttribute attr[2];
      lc.attrs = attr;
      lc.numAttrs = (unsigned)cluster_attrs(attr, nsplit);
      // the smaller count of the two builds
      for (bool paired : {false, true}) {
        int c = 0;
        if (cudaOccupancyMaxActiveClusters(&c, split_fn(kind, paired, true), &lc) != cudaSuccess) {
          (void)cudaGetLastError();  // not launchable this way: no clusters
          c = 0;
        }
        n = paired ? (c < n ? c : n) : c;
      }
    }
  }
  *out = n;
  return PDA_OK;
}

// Kernels one call launches under plan pl.
int plan_launches(const Plan& pl) {
  return 1 + (pl.ordered > 0 ? 1 : 0) + (pl.nsplit > 1 && !pl.cluster ? 1 : 0) + (pl.tail_units > 0 ? 1 : 0);
}

pda_status plan_call(int dev, int num_seqs, int num_kv_heads, int max_blocks, int bs, KernelKind wide,
                     KernelKind dense, Plan* out) {
  int sms = 0, occ = 0, occ_d = 0;
  pda_status st = device_info(dev, bs, &sms, &occ, wide);
  if (st != PDA_OK) return st;
  if (dense != wide) {
    st = device_info(dev, bs, &sms, &occ_d, dense);
    if (st != PDA_OK) return st;
  }
  *out = plan_from(num_seqs, num_kv_heads, max_blocks, bs, sms, occ, occ_d, wide, dense, g_split_override.load());
  if (!g_tail_split.load()) out->tail_units = 0;
  if (out->cluster) {
    // Only when the device runs every cluster of the grid at once.
    const long long ctas = (long long)num_seqs * num_kv_heads * out->nsplit;
    int n = 0;
    st = max_active_clusters(dev, out->kind, bs, out->nsplit, &n);
    if (st != PDA_OK) return st;
    out->cluster = n > 0 && (long long)n * out->nsplit >= ctas;
  }
  return PDA_OK;
}

// Profiling events: inside stream capture a plain record only expresses a
// dependency, so record them as external event nodes there.
cudaError_t record_profile_event(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    return cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  return cudaEventRecord(e, s);
}

// Workspace of one (device, stream): kQueueBytes of work-queue counters for
// the persistent kernel (zeroed when allocated; each launch leaves them at
// zero), the persistent kernel's unit order, then the split partials
// O [S][H][nsplit][D] and (m, l) [S][H][nsplit][2].
constexpr size_t kQueueBytes = 256;

// Bytes of the split partials (0 for one split).
size_t partial_bytes(int num_seqs, int num_heads, int nsplit) {
  if (nsplit <= 1) return 0;
  const size_t rows = (size_t)num_seqs * num_heads * nsplit;
  return rows * kHeadDim * sizeof(float) + rows * 2 * sizeof(float);
}

struct WsLayout {
  size_t order_off = 0;
  size_t piece_off = 0;  // tail pieces: piece table (int4 entries)
  size_t info_off = 0;   // tail pieces: {unit, first entry, pieces} per tail unit
  size_t rows_off = 0;   // tail pieces: (O, m, l) rows of each piece
  size_t part_off = 0;
  size_t bytes = 0;
};

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

WsLayout ws_layout(int num_seqs, int num_heads, const Plan& pl) {
  WsLayout w;
  const size_t part = pl.cluster ? 0 : partial_bytes(num_seqs, num_heads, pl.nsplit);
  if (!is_persistent(pl.kind) && part == 0) return w;
  const size_t pieces = (size_t)pl.tail_units * (size_t)pl.max_pieces;
  w.order_off = kQueueBytes;
  w.piece_off = w.order_off + align256((size_t)pl.ordered * sizeof(int));
  w.info_off = w.piece_off + align256(pieces * 4 * sizeof(int));
  w.rows_off = w.info_off + align256((size_t)pl.tail_units * 4 * sizeof(int));
  w.part_off = w.rows_off + align256(pieces * pda::kTailRowFloats * sizeof(float));
  w.bytes = w.part_off + part;
  return w;
}

// Returns the workspace pointer for (device, stream), growing it with
// stream-ordered allocation when not capturing.
pda_status get_workspace(int dev, cudaStream_t stream, size_t bytes, void** out) {
  *out = nullptr;
  if (bytes == 0) return PDA_OK;
  std::lock_guard<std::mutex> lk(g_ws_mu);
  Workspace& ws = g_ws[{dev, stream}];
  if (ws.bytes >= bytes) {
    *out = ws.ptr;
    return PDA_OK;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return PDA_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return PDA_ERR_WORKSPACE;
  size_t want = bytes + (bytes >> 3);
  want = (want + 255) & ~(size_t)255;
  void* p = nullptr;
  if (cudaMallocAsync(&p, want, stream) != cudaSuccess) return PDA_ERR_CUDA;
  if (cudaMemsetAsync(p, 0, kQueueBytes, stream) != cudaSuccess) {
    cudaFreeAsync(p, stream);
    return PDA_ERR_CUDA;
  }
  if (ws.ptr) ws.retired.push_back(ws.ptr);
  ws.ptr = p;
  ws.bytes = want;
  *out = p;
  return PDA_OK;
}

// Launch the merge kernel for partials of nsplit splits (one warp per row up
// to kMergeRowSplits splits, else one block per row), as the programmatic
// dependent of the kernel before it on `stream` when pdl is set.
cudaError_t launch_merge(const pda::MergeParams& mp, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t lc = {};
  if (mp.nsplit <= pda::kMergeRowSplits) {
    const long long rows = (long long)mp.num_seqs * mp.num_heads;
    lc.gridDim = dim3((unsigned)((rows + pda::kMergeRowsPerBlock - 1) / pda::kMergeRowsPerBlock));
  } else {
    lc.gridDim = dim3((unsigned)mp.num_heads, (unsigned)mp.num_seqs);
  }
  lc.blockDim = dim3(kHeadDim);
  lc.dynamicSmemBytes = 0;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
  }
  return mp.nsplit <= pda::kMergeRowSplits ? cudaLaunchKernelEx(&lc, pda::pda_merge_kernel, mp)
                                            : cudaLaunchKernelEx(&lc, pda::pda_merge_wide_kernel, mp);
}

}  // namespace

// Shared launch path of pda_decode (k_scales == v_scales == nullptr) and
// pda_decode_slot_scales (per-slot tables; k_scale, v_scale unused).
static pda_status launch_decode(bool slot, void* out, const void* q, const void* k_cache, const void* v_cache,
                                const float* k_scales, const float* v_scales, const int32_t* block_tables,
                                const int32_t* seq_lens, int num_seqs, int num_heads, int num_kv_heads,
                                int head_size, int block_size, int max_num_blocks_per_seq, float scale,
                                float k_scale, float v_scale, cudaStream_t stream, const float* sinks = nullptr,
                                int out_fp8 = 0, float out_scale = 1.f, int v_shuffled = 0,
                                const TokenMajorMaps* tm = nullptr) {
  pda_status st = validate(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads, num_kv_heads,
                           head_size, block_size, max_num_blocks_per_seq, scale, k_scale, v_scale);
  if (st != PDA_OK || num_seqs == 0) return st;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PDA_ERR_CUDA;
  const KernelKind wide = slot ? slot_wide_kind(num_heads / num_kv_heads, block_size) : (tm ? kWideToken : kWidePlain);
  const KernelKind dense = slot ? kSlotWide : (tm ? kTokenDense : kPlainDense);
  Plan pl;
  st = plan_call(dev, num_seqs, num_kv_heads, max_num_blocks_per_seq, block_size, wide, dense, &pl);
  if (st != PDA_OK) return st;
  const int nsplit = pl.nsplit;
  void* ws = nullptr;
  WsLayout wl = ws_layout(num_seqs, num_heads, pl);
  st = get_workspace(dev, stream, wl.bytes, &ws);
  if (st == PDA_ERR_WORKSPACE && is_persistent(pl.kind) && nsplit == 1) {
    // Captured without pda_reserve: the per-unit kernel needs no workspace.
    pl.kind = per_unit_of(pl.kind);
    wl = WsLayout();
    st = PDA_OK;
  }
  if (st != PDA_OK) return st;

  const RingShape rs = ring_for(pl.kind, block_size);
  pda::DecodeParams p;
  p.block_limit = g_block_limit.load();
  p.cluster_merge = pl.cluster ? 1 : 0;
  p.out = out;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  unsigned* queue = static_cast<unsigned*>(ws);
  const bool partials = nsplit > 1 && !pl.cluster;
  p.part_o = partials ? reinterpret_cast<float*>(static_cast<char*>(ws) + wl.part_off) : nullptr;
  p.part_ml = partials ? p.part_o + (size_t)num_seqs * num_heads * nsplit * kHeadDim : nullptr;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.gqa = num_heads / num_kv_heads;
  p.block_size = block_size;
  p.max_blocks = max_num_blocks_per_seq;
  p.nsplit = nsplit;
  p.pages_per_stage = rs.pages_per_stage;
  p.num_stages = rs.num_stages;
  p.stage_bytes = rs.stage_bytes;
  p.scale_off = rs.scale_off;
  p.k_scales = slot ? k_scales : nullptr;
  p.v_scales = slot ? v_scales : nullptr;
  p.logit_scale_log2 = (float)((double)scale * (slot ? 1.0 : (double)k_scale) * 1.4426950408889634);
  p.v_scale = v_scale;
  p.sinks = sinks;
  p.out_fp8 = out_fp8;
  p.out_scale = out_scale;
  p.v_shuffled = v_shuffled;
  if (tm) {
    p.tm_dim_token = tm->dim_token;
    p.tm_dim_head = tm->dim_head;
    p.tm_dim_block = tm->dim_block;
  }

  cudaEvent_t eb = g_prof_before.load(), ea = g_prof_after.load();
  if (eb && ea && record_profile_event(eb, stream) != cudaSuccess) return PDA_ERR_CUDA;
  dim3 grid((unsigned)nsplit, (unsigned)num_kv_heads, (unsigned)num_seqs);
  // Native V pages of 32-, 64- and 128-token blocks load through a swizzled
  // tensor map (no ldmatrix bank conflicts); the per-slot-scale instance's
  // stages carry scale rows and are not aligned for it.
  CUtensorMap vmap;
  if (!slot && !tm && !v_shuffled) p.v_swizzle = make_v_swizzle_map(v_cache, num_kv_heads, block_size, &vmap);
  // Per-slot scale rows: at 4 pages a stage each table's 4 rows in one
  // gather, else one bulk copy per row (rows of at least 128 bytes).
  CUtensorMap kscale_map, vscale_map;
  const bool gathers = g_tma_gather.load() != 0;
  if (slot) {
    if (gathers && rs.pages_per_stage != 4)
      p.scale_rows = pda::kScaleRowsBulk;
    else if (gathers && make_scale_row_map(k_scales, block_size, &kscale_map) &&
             make_scale_row_map(v_scales, block_size, &vscale_map))
      p.scale_rows = pda::kScaleRowsGather4;
    // the persistent kernel's stages take no cp.async pieces
    if (p.scale_rows == pda::kScaleRowsPieces && is_persistent(pl.kind)) p.scale_rows = pda::kScaleRowsBulk;
  }
  // Page-major 16-token pages: a stage's 4 pages of each cache in one
  // gather, on the persistent kernel and on per-unit grids whose splits do
  // not merge in clusters (GB300, 16 x 1024 tokens in clusters of 4: 12.77
  // against 12.65 us with gathers, so cluster grids keep bulk copies).
  CUtensorMap kpage_map, vpage_map;
  if (gathers && (is_persistent(pl.kind) || !pl.cluster) && !slot && !tm && rs.pages_per_stage == 4 &&
      block_size == 16 &&
      make_page_row_map(k_cache, &kpage_map) && make_page_row_map(v_cache, &vpage_map))
    p.page_gather = 1;
  const CUtensorMap* maps_k = &g_no_map;
  const CUtensorMap* maps_v = p.v_swizzle ? &vmap : &g_no_map;
  if (p.scale_rows == pda::kScaleRowsGather4) {
    maps_k = &kscale_map;
    maps_v = &vscale_map;
  } else if (p.page_gather) {
    maps_k = &kpage_map;
    maps_v = &vpage_map;
  }
  const CUtensorMap& mk = tm ? tm->k : *maps_k;
  const CUtensorMap& mv = tm ? tm->v : *maps_v;
  const bool paired = paired_for(p.gqa);
  if (is_persistent(pl.kind)) {
    const int units = num_seqs * num_kv_heads * nsplit;
    const PersistFn fn = persist_fn(pl.kind, paired);
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(pl.grid);
    lc.blockDim = dim3(pda::kThreads);
    lc.dynamicSmemBytes = rs.smem_bytes;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pl.ordered > 0) {
      // The order kernel, then the decode kernel as its programmatic
      // dependent: the decode CTAs start on their first units at once and
      // wait for the order only before taking a second one.
      pda::OrderParams op;
      op.seq_lens = seq_lens;
      op.order = reinterpret_cast<int*>(static_cast<char*>(ws) + wl.order_off);
      op.first = (int)pl.grid;
      op.num_units = units;
      op.num_kv_heads = num_kv_heads;
      op.nsplit = nsplit;
      op.block_size = block_size;
      op.max_blocks = max_num_blocks_per_seq;
      op.max_split_pages = (max_num_blocks_per_seq + nsplit - 1) / nsplit;
      if (pl.tail_units > 0) {
        op.tail_units = pl.tail_units;
        op.max_pieces = pl.max_pieces;
        op.min_piece_pages = pl.min_piece_pages;
        op.piece_table = reinterpret_cast<int4*>(static_cast<char*>(ws) + wl.piece_off);
        op.tail_info = reinterpret_cast<int4*>(static_cast<char*>(ws) + wl.info_off);
        op.num_tickets = reinterpret_cast<int*>(queue + 2);
        p.tail_first = (unsigned)(units - pl.tail_units);
        p.piece_table = op.piece_table;
        p.num_tickets = op.num_tickets;
        p.tail_rows = reinterpret_cast<float*>(static_cast<char*>(ws) + wl.rows_off);
      }
      pda::pda_order_units_kernel<<<1, pda::kOrderThreads, 0, stream>>>(op);
      if (cudaGetLastError() != cudaSuccess) return PDA_ERR_CUDA;
      p.unit_order = op.order;
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      lc.attrs = attr;
      lc.numAttrs = 1;
    }
    if (cudaLaunchKernelEx(&lc, fn, p, queue, units, mk, mv) != cudaSuccess) return PDA_ERR_CUDA;
    if (pl.tail_units > 0) {
      // the tail merge, as the decode kernel's programmatic dependent
      pda::TailMergeParams tp;
      tp.m.out = out;
      tp.m.num_heads = num_heads;
      tp.m.v_scale = slot ? 1.f : v_scale;  // slot scales: the pieces carry their V reference
      tp.m.sinks = sinks;
      tp.m.out_fp8 = out_fp8;
      tp.m.out_scale = out_scale;
      tp.m.nsplit = nsplit;
      tp.part_o = p.part_o;
      tp.part_ml = p.part_ml;
      tp.tail_info = reinterpret_cast<const int4*>(static_cast<char*>(ws) + wl.info_off);
      tp.tail_rows = p.tail_rows;
      tp.tail_units = pl.tail_units;
      tp.num_kv_heads = num_kv_heads;
      tp.gqa = p.gqa;
      cudaLaunchConfig_t tc = {};
      tc.gridDim = dim3((unsigned)((pl.tail_units * p.gqa + pda::kMergeRowsPerBlock - 1) / pda::kMergeRowsPerBlock));
      tc.blockDim = dim3(kHeadDim);
      tc.stream = stream;
      cudaLaunchAttribute ta[1];
      ta[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      ta[0].val.programmaticStreamSerializationAllowed = 1;
      tc.attrs = ta;
      tc.numAttrs = 1;
      if (cudaLaunchKernelEx(&tc, pda::pda_tail_merge_kernel, tp) != cudaSuccess) return PDA_ERR_CUDA;
    }
  } else {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = dim3(pda::kThreads);
    lc.dynamicSmemBytes = rs.smem_bytes;
    lc.stream = stream;
    cudaLaunchAttribute attr[2];
    if (pl.cluster) {
      lc.attrs = attr;
      lc.numAttrs = (unsigned)cluster_attrs(attr, nsplit);
    }
    if (cudaLaunchKernelEx(&lc, split_fn(pl.kind, paired, pl.cluster), p, mk, mv) != cudaSuccess)
      return PDA_ERR_CUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return PDA_ERR_CUDA;
  if (eb && ea && record_profile_event(ea, stream) != cudaSuccess) return PDA_ERR_CUDA;

  if (partials) {
    pda::MergeParams mp;
    mp.out = p.out;
    mp.part_o = p.part_o;
    mp.part_ml = p.part_ml;
    mp.seq_lens = seq_lens;
    mp.num_seqs = num_seqs;
    mp.num_heads = num_heads;
    mp.block_size = block_size;
    mp.max_blocks = max_num_blocks_per_seq;
    mp.nsplit = nsplit;
    mp.v_scale = slot ? 1.f : v_scale;
    mp.sinks = sinks;
    mp.out_fp8 = out_fp8;
    mp.out_scale = out_scale;
    // Programmatic dependent of the decode kernel: its launch overlaps the
    // decode kernel's last CTAs, and it waits for the partials on the device.
    if (launch_merge(mp, stream, true) != cudaSuccess) return PDA_ERR_CUDA;
  }
  return PDA_OK;
}


extern "C" {

const char* pda_status_string(int status) {
  switch (status) {
    case PDA_OK: return "ok";
    case PDA_ERR_INVALID_ARG: return "invalid argument";
    case PDA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PDA_ERR_WORKSPACE: return "workspace must grow during stream capture (call pda_reserve first)";
    case PDA_ERR_CUDA: return "CUDA runtime error";
    case PDA_ERR_DEVICE_TIMEOUT: return "a kernel gave up on a bounded wait";
    case PDA_ERR_NOALLOC_CAPACITY:
      return "the call needs more split scratch than pda_decode_noalloc's static buffer holds";
    default: return "unknown status";
  }
}

int pda_choose_splits(int num_seqs, int num_kv_heads, int max_num_blocks_per_seq, int block_size, int sm_count,
                      int ctas_per_sm) {
  if (num_seqs <= 0 || num_kv_heads <= 0 || max_num_blocks_per_seq <= 0 || block_size <= 0 || sm_count <= 0 ||
      ctas_per_sm <= 0)
    return 1;
  const long long units = (long long)num_seqs * num_kv_heads;
  const long long slots = (long long)sm_count * ctas_per_sm;
  // Two reasons to split a (sequence, kv head) unit, measured on GB300:
  //  * a unit's K/V bytes exceed kMaxSplitBytes: a few long CTAs leave most
  //    resident slots idle while the last wave drains;
  //  * the units fill less than one wave of resident CTAs: split up to one
  //    wave (more splits only add partial traffic and the merge launch).
  // Never below kMinSplitTokens tokens per split.
  const long long kMaxSplitBytes = 1LL << 20;
  const long long kMinSplitTokens = 256;
  const long long unit_bytes = (long long)max_num_blocks_per_seq * block_size * 128 * 2;
  long long want = (unit_bytes + kMaxSplitBytes - 1) / kMaxSplitBytes;
  if (units < slots) {
    const long long fill = slots / units;
    if (fill > want) want = fill;
  }
  const long long min_pages = (kMinSplitTokens + block_size - 1) / block_size;
  long long cap = max_num_blocks_per_seq / min_pages;
  if (cap < 1) cap = 1;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return (int)want;
}

int pda_choose_kernel(int num_seqs, int num_kv_heads, int max_num_blocks_per_seq, int block_size, int sm_count,
                      int ctas_per_sm, int ctas_per_sm_dense, int* num_splits, int* launches) {
  if (num_seqs <= 0 || num_kv_heads <= 0 || max_num_blocks_per_seq <= 0 || block_size <= 0 || sm_count <= 0 ||
      ctas_per_sm <= 0 || ctas_per_sm_dense <= 0)
    return -1;
  const Plan pl = plan_from(num_seqs, num_kv_heads, max_num_blocks_per_seq, block_size, sm_count, ctas_per_sm,
                            ctas_per_sm_dense, kWidePlain, kPlainDense, 0);
  if (num_splits) *num_splits = pl.nsplit;
  if (launches) *launches = plan_launches(pl);
  switch (pl.kind) {
    case kPlainDense: return PDA_KERNEL_PER_UNIT_DENSE;
    case kPersistWide: return PDA_KERNEL_PERSISTENT;
    default: return PDA_KERNEL_PER_UNIT;
  }
}

void pda_set_split_override(int num_splits) { g_split_override.store(num_splits > 0 ? num_splits : 0); }

void pda_set_tail_split(int enable) { g_tail_split.store(enable ? 1 : 0); }

void pda_set_tma_gather(int enable) { g_tma_gather.store(enable ? 1 : 0); }

void pda_set_block_check(long long num_blocks) {
  g_block_limit.store(num_blocks <= 0 ? 0u : (num_blocks >= (1LL << 31) ? (1u << 31) : (uint32_t)num_blocks));
}

int pda_plan_splits(int num_seqs, int num_heads, int num_kv_heads, int max_num_blocks_per_seq, int block_size) {
  (void)num_heads;
  if (block_size <= 0 || block_size % 16 != 0 || block_size > 128) return -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  Plan pl;
  if (plan_call(dev, num_seqs, num_kv_heads, max_num_blocks_per_seq, block_size, kWidePlain, kPlainDense, &pl) !=
      PDA_OK)
    return -1;
  return pl.nsplit;
}

int pda_plan_kernel(int num_seqs, int num_heads, int num_kv_heads, int max_num_blocks_per_seq, int block_size) {
  (void)num_heads;
  if (block_size <= 0 || block_size % 16 != 0 || block_size > 128) return -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  Plan pl;
  if (plan_call(dev, num_seqs, num_kv_heads, max_num_blocks_per_seq, block_size, kWidePlain, kPlainDense, &pl) !=
      PDA_OK)
    return -1;
  switch (pl.kind) {
    case kPlainDense: return PDA_KERNEL_PER_UNIT_DENSE;
    case kPersistWide: return PDA_KERNEL_PERSISTENT;
    default: return PDA_KERNEL_PER_UNIT;
  }
}

int pda_plan_launches(int num_seqs, int num_heads, int num_kv_heads, int max_num_blocks_per_seq, int block_size) {
  (void)num_heads;
  if (num_seqs == 0) return 0;
  if (block_size <= 0 || block_size % 16 != 0 || block_size > 128) return -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  Plan pl;
  if (plan_call(dev, num_seqs, num_kv_heads, max_num_blocks_per_seq, block_size, kWidePlain, kPlainDense, &pl) !=
      PDA_OK)
    return -1;
  return plan_launches(pl);
}

int pda_tail_pieces(int pages, int tail_units, int ctas, int block_size, int* sizes, int max_sizes) {
  if (pages < 0 || tail_units <= 0 || ctas <= 0 || tail_units >= ctas || block_size <= 0 || block_size % 16 != 0 ||
      block_size > 128 || max_sizes < 0 || (max_sizes > 0 && !sizes))
    return -1;
  const int m = tail_min_piece_pages(block_size);
  const int cap = pda::tail_piece_cap(tail_units, ctas);
  const int P = pda::tail_piece_count(pages, tail_units, ctas, m, cap);
  for (int r = 0; r < P && r < max_sizes; ++r) {
    int a = 0, b = pages;
    if (P > 1) pda::tail_piece_range(pages, tail_units, ctas, m, P, cap, r, a, b);
    sizes[r] = b - a;
  }
  return P;
}

int pda_plan_slot_scales(int num_seqs, int num_heads, int num_kv_heads, int max_num_blocks_per_seq, int block_size,
                         int* kernel, int* num_splits, int* launches) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 ||
      max_num_blocks_per_seq < 0 || block_size <= 0 || block_size % 16 != 0 || block_size > 128)
    return -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  Plan pl;
  if (plan_call(dev, num_seqs, num_kv_heads, max_num_blocks_per_seq, block_size,
                slot_wide_kind(num_heads / num_kv_heads, block_size), kSlotWide, &pl) != PDA_OK)
    return -1;
  if (kernel) *kernel = is_persistent(pl.kind) ? PDA_KERNEL_PERSISTENT : PDA_KERNEL_PER_UNIT;
  if (num_splits) *num_splits = pl.nsplit;
  if (launches) *launches = num_seqs == 0 ? 0 : plan_launches(pl);
  return 0;
}

void pda_set_profile_events(cudaEvent_t before, cudaEvent_t after) {
  if (before && after) {
    g_prof_before.store(before);
    g_prof_after.store(after);
  } else {
    g_prof_before.store(nullptr);
    g_prof_after.store(nullptr);
  }
}

pda_status pda_reserve(int num_seqs, int num_heads, int num_kv_heads, int max_num_blocks_per_seq, int block_size,
                       cudaStream_t stream) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || max_num_blocks_per_seq < 0 || block_size <= 0 ||
      block_size % 16 != 0 || block_size > 128)
    return PDA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PDA_ERR_CUDA;
  // Size for the largest plan any entry point makes for these sizes.
  size_t bytes = 0;
  const KernelKind pairs[3][2] = {{kWidePlain, kPlainDense},
                                  {slot_wide_kind(num_heads / num_kv_heads, block_size), kSlotWide},
                                  {kWideToken, kTokenDense}};
  for (const auto& pr : pairs) {
    Plan pl;
    pda_status st = plan_call(dev, num_seqs, num_kv_heads, max_num_blocks_per_seq, block_size, pr[0], pr[1], &pl);
    if (st != PDA_OK) return st;
    const size_t b = ws_layout(num_seqs, num_heads, pl).bytes;
    bytes = b > bytes ? b : bytes;
  }
  void* ws = nullptr;
  return get_workspace(dev, stream, bytes, &ws);
}

pda_status pda_release(void) {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  int prev = 0;
  cudaGetDevice(&prev);
  pda_status st = PDA_OK;
  for (auto* m : {&g_ws, &g_stage}) {
    for (auto& kv : *m) {
      if (!kv.second.ptr) continue;
      if (cudaSetDevice(kv.first.first) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        st = PDA_ERR_CUDA;
        continue;
      }
      kv.second.retired.push_back(kv.second.ptr);
      for (void* ptr : kv.second.retired)
        if (cudaFree(ptr) != cudaSuccess) st = PDA_ERR_CUDA;
    }
  }
  g_ws.clear();
  g_stage.clear();
  cudaSetDevice(prev);
  // Per-device set-up (SM counts, occupancy, shared-memory opt-ins, the
  // no-allocation scratch address) is taken again on the next call, so a
  // device reset between this call and the next does not leave it stale.
  {
    std::lock_guard<std::mutex> dk(g_dev_mu);
    g_devices.clear();
  }
  noalloc_forget_devices();
  return st;
}

pda_status pda_workspace_info(cudaStream_t stream, long long* bytes, int* retired) {
  if (!bytes || !retired) return PDA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PDA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_ws_mu);
  const auto it = g_ws.find({dev, stream});
  *bytes = it == g_ws.end() ? 0 : (long long)it->second.bytes;
  *retired = it == g_ws.end() ? 0 : (int)it->second.retired.size();
  return PDA_OK;
}

pda_status pda_query_device_status(cudaStream_t stream, int* code) {
  if (!code) return PDA_ERR_INVALID_ARG;
  *code = 0;
  unsigned int v = 0, zero = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PDA_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&v, pda::g_status, sizeof v) != cudaSuccess) return PDA_ERR_CUDA;
  if (cudaMemcpyToSymbol(pda::g_status, &zero, sizeof zero) != cudaSuccess) return PDA_ERR_CUDA;
  *code = (int)v;
  return v ? PDA_ERR_DEVICE_TIMEOUT : PDA_OK;
}

pda_status pda_test_bounded_wait(int timeout_us, cudaStream_t stream) {
  if (timeout_us < 1 || timeout_us > 2000000) return PDA_ERR_INVALID_ARG;
  pda::pda_bounded_wait_test_kernel<<<1, 32, 0, stream>>>((unsigned long long)timeout_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? PDA_OK : PDA_ERR_CUDA;
}

pda_status pda_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                                 const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_size,
                                 int block_size, long long num_blocks, float k_scale, float v_scale, int kv_layout,
                                 cudaStream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 || num_blocks < 0)
    return PDA_ERR_INVALID_ARG;
  if (kv_layout != PDA_KV_NATIVE && kv_layout != PDA_KV_SHUFFLED_V) return PDA_ERR_INVALID_ARG;
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale) || k_scale == 0.f || v_scale == 0.f)
    return PDA_ERR_INVALID_ARG;
  if (head_size != kHeadDim) return PDA_ERR_UNSUPPORTED;
  if (block_size % 16 != 0 || block_size > 128) return PDA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PDA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PDA_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PDA_ERR_INVALID_ARG;
  pda::CacheWriteParams p;
  p.key = static_cast<const __nv_bfloat16*>(key);
  p.value = static_cast<const __nv_bfloat16*>(value);
  p.k_cache = static_cast<uint8_t*>(k_cache);
  p.v_cache = static_cast<uint8_t*>(v_cache);
  p.slot_mapping = slot_mapping;
  p.num_tokens = num_tokens;
  p.num_kv_heads = num_kv_heads;
  p.block_size = block_size;
  p.num_slots = num_blocks * (long long)block_size;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.v_shuffled = kv_layout == PDA_KV_SHUFFLED_V ? 1 : 0;
  if (num_kv_heads > 65535) return PDA_ERR_UNSUPPORTED;
  // Small writes (a decode step's few hundred (token, kv head) items at
  // scattered slots) take one warp per item; larger ones one CTA per 16
  // tokens of a kv head, which stores a run of whole blocks as 16-byte V
  // rows and scattered slots a token at a time. Measured on GB300 (µs per
  // call, 8 kv heads, random slots / whole blocks): 256 tokens 4.1 / 4.8
  // one warp per item against 5.6 / 3.6 per 16 tokens; 4096 tokens 28.1 /
  // 31.4 against 33.8 / 7.4; 65,536 tokens 551 (earlier 16-token writer) /
  // 83.8 against 424 / 83.2.
  const long long items = (long long)num_tokens * num_kv_heads;
  if (items <= kScatterWriteMaxItems) {
    const long long blocks = (items + pda::kCacheWriteWarpsPerCta - 1) / pda::kCacheWriteWarpsPerCta;
    pda::pda_reshape_and_cache_scatter_kernel<<<(unsigned)blocks, pda::kCacheWriteWarpsPerCta * 32, 0, stream>>>(p);
  } else {
    const dim3 grid((unsigned)((num_tokens + pda::kCacheWriteTokens - 1) / pda::kCacheWriteTokens),
                    (unsigned)num_kv_heads);
    pda::pda_reshape_and_cache_kernel<<<grid, pda::kCacheWriteThreads, 0, stream>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? PDA_OK : PDA_ERR_CUDA;
}

pda_status pda_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* seq_lens, int num_seqs, int num_heads,
                      int num_kv_heads, int head_size, int block_size, int max_num_blocks_per_seq, float scale,
                      float k_scale, float v_scale, cudaStream_t stream) {
  return launch_decode(false, out, q, k_cache, v_cache, nullptr, nullptr, block_tables, seq_lens, num_seqs,
                       num_heads, num_kv_heads, head_size, block_size, max_num_blocks_per_seq, scale, k_scale,
                       v_scale, stream);
}

pda_status pda_decode_host(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int32_t* seq_lens, int num_seqs, int num_heads,
                           int num_kv_heads, int head_size, int block_size, int max_num_blocks_per_seq,
                           long long num_blocks, float scale, float k_scale, float v_scale, cudaStream_t stream) {
  // pda_decode's checks of sizes and scalars; host pointers need no
  // particular alignment.
  const pda_status vs = validate_sizes(num_seqs, num_heads, num_kv_heads, head_size, block_size,
                                       max_num_blocks_per_seq, scale, k_scale, v_scale);
  if (vs != PDA_OK || num_seqs == 0) return vs;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || num_blocks <= 0)
    return PDA_ERR_INVALID_ARG;
  // Every table entry and length the kernels will read.
  const long long max_len = (long long)max_num_blocks_per_seq * block_size;
  for (int s = 0; s < num_seqs; ++s) {
    const int L = seq_lens[s];
    if (L < 0 || L > max_len) return PDA_ERR_INVALID_ARG;
    const int32_t* row = block_tables + (size_t)s * max_num_blocks_per_seq;
    for (int i = 0, n = (L + block_size - 1) / block_size; i < n; ++i)
      if (row[i] < 0 || row[i] >= num_blocks) return PDA_ERR_INVALID_ARG;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PDA_ERR_CUDA;
  auto up = [](size_t b) { return (b + 255) & ~(size_t)255; };
  const size_t q_bytes = (size_t)num_seqs * num_heads * kHeadDim * 2;
  const size_t page_bytes = (size_t)num_blocks * num_kv_heads * kHeadDim * block_size;
  const size_t t_bytes = (size_t)num_seqs * max_num_blocks_per_seq * sizeof(int32_t);
  const size_t l_bytes = (size_t)num_seqs * sizeof(int32_t);
  const size_t off_k = up(q_bytes), off_v = off_k + up(page_bytes), off_t = off_v + up(page_bytes);
  const size_t off_l = off_t + up(t_bytes), off_o = off_l + up(l_bytes), total = off_o + up(q_bytes);
  char* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace& sb = g_stage[{dev, stream}];
    if (sb.bytes < total) {
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return PDA_ERR_CUDA;
      if (cs != cudaStreamCaptureStatusNone) return PDA_ERR_WORKSPACE;
      void* p = nullptr;
      if (cudaMallocAsync(&p, total, stream) != cudaSuccess) return PDA_ERR_CUDA;
      if (sb.ptr) sb.retired.push_back(sb.ptr);
      sb.ptr = p;
      sb.bytes = total;
    }
    base = static_cast<char*>(sb.ptr);
  }
  const struct {
    size_t off;
    const void* src;
    size_t bytes;
  } in[] = {{0, q, q_bytes}, {off_k, k_cache, page_bytes}, {off_v, v_cache, page_bytes},
            {off_t, block_tables, t_bytes}, {off_l, seq_lens, l_bytes}};
  for (const auto& c : in)
    if (c.bytes && cudaMemcpyAsync(base + c.off, c.src, c.bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
      return PDA_ERR_CUDA;
  pda_status st = launch_decode(false, base + off_o, base, base + off_k, base + off_v, nullptr, nullptr,
                                reinterpret_cast<const int32_t*>(base + off_t),
                                reinterpret_cast<const int32_t*>(base + off_l), num_seqs, num_heads, num_kv_heads,
                                head_size, block_size, max_num_blocks_per_seq, scale, k_scale, v_scale, stream);
  if (st != PDA_OK) return st;
  if (cudaMemcpyAsync(out, base + off_o, q_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return PDA_ERR_CUDA;
  return PDA_OK;
}

pda_status pda_decode_ex(void* out, const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, const int32_t* seq_lens, int num_seqs, int num_heads,
                         int num_kv_heads, int head_size, int block_size, int max_num_blocks_per_seq, float scale,
                         float k_scale, float v_scale, int kv_layout, const float* sinks, int out_dtype,
                         float output_scale, cudaStream_t stream) {
  if (kv_layout != PDA_KV_NATIVE && kv_layout != PDA_KV_SHUFFLED_V) return PDA_ERR_INVALID_ARG;
  if (out_dtype != PDA_OUT_BF16 && out_dtype != PDA_OUT_E4M3) return PDA_ERR_INVALID_ARG;
  if (out_dtype == PDA_OUT_E4M3 && !(std::isfinite(output_scale) && output_scale > 0.f)) return PDA_ERR_INVALID_ARG;
  if (sinks && (reinterpret_cast<uintptr_t>(sinks) & 3u)) return PDA_ERR_INVALID_ARG;
  return launch_decode(false, out, q, k_cache, v_cache, nullptr, nullptr, block_tables, seq_lens, num_seqs,
                       num_heads, num_kv_heads, head_size, block_size, max_num_blocks_per_seq, scale, k_scale,
                       v_scale, stream, sinks, out_dtype == PDA_OUT_E4M3 ? 1 : 0,
                       out_dtype == PDA_OUT_E4M3 ? output_scale : 1.f, kv_layout == PDA_KV_SHUFFLED_V ? 1 : 0);
}

pda_status pda_decode_strided(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, const int32_t* seq_lens, int num_seqs, int num_heads,
                              int num_kv_heads, int head_size, int block_size, int max_num_blocks_per_seq,
                              long long num_blocks, long long k_block_stride, long long k_token_stride,
                              long long k_head_stride, long long v_block_stride, long long v_token_stride,
                              long long v_head_stride, float scale, float k_scale, float v_scale,
                              cudaStream_t stream) {
  pda_status st = validate(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads, num_kv_heads,
                           head_size, block_size, max_num_blocks_per_seq, scale, k_scale, v_scale);
  if (st != PDA_OK || num_seqs == 0) return st;
  if (num_blocks <= 0) return PDA_ERR_INVALID_ARG;
  TokenMajorMaps tm;
  int vt = 0, vh = 0, vb = 0;
  st = make_token_major_map(k_cache, num_blocks, num_kv_heads, block_size, k_block_stride, k_token_stride,
                            k_head_stride, &tm.k, &tm.dim_token, &tm.dim_head, &tm.dim_block);
  if (st != PDA_OK) return st;
  st = make_token_major_map(v_cache, num_blocks, num_kv_heads, block_size, v_block_stride, v_token_stride,
                            v_head_stride, &tm.v, &vt, &vh, &vb);
  if (st != PDA_OK) return st;
  if (vt != tm.dim_token || vh != tm.dim_head || vb != tm.dim_block) return PDA_ERR_UNSUPPORTED;
  return launch_decode(false, out, q, k_cache, v_cache, nullptr, nullptr, block_tables, seq_lens, num_seqs,
                       num_heads, num_kv_heads, head_size, block_size, max_num_blocks_per_seq, scale, k_scale,
                       v_scale, stream, nullptr, 0, 1.f, 0, &tm);
}

pda_status pda_decode_slot_scales(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  const float* k_scales, const float* v_scales, const int32_t* block_tables,
                                  const int32_t* seq_lens, int num_seqs, int num_heads, int num_kv_heads,
                                  int head_size, int block_size, int max_num_blocks_per_seq, float scale,
                                  cudaStream_t stream) {
  if (num_seqs > 0 && (!k_scales || !v_scales || !aligned16(k_scales) || !aligned16(v_scales)))
    return PDA_ERR_INVALID_ARG;
  return launch_decode(true, out, q, k_cache, v_cache, k_scales, v_scales, block_tables, seq_lens, num_seqs,
                       num_heads, num_kv_heads, head_size, block_size, max_num_blocks_per_seq, scale, 1.f, 1.f,
                       stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// pda_decode_noalloc: the split-KV decode path with its split partials in a
// fixed device array that is part of the loaded library, for callers that
// must not allocate device memory (see include/pda.h). Nothing below touches
// the workspace, the host containers or any allocator.

namespace {

// Room for rows * 520 <= 16 MiB, i.e. num_seqs * num_heads * splits <= 32,263
// partial rows of 520 bytes (128 floats of O plus m and l).
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;  // 16 MiB per device

// The partials' storage. Host code may not use this name as an address (on
// the host it is only a stand-in); each device's address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
struct NoAllocDevice {
  bool ready;
  void* scratch;      // device address of g_noalloc_scratch on this device
  int sm_count;
  int occ[9];         // resident decode CTAs per SM, by block_size / 16
};
std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// One-time set-up for `dev` (which must be current): the scratch address,
// the SM count and the decode kernel's shared-memory opt-in. No allocation.
pda_status noalloc_setup(int dev, int bs, NoAllocDevice* out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return PDA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!d.ready) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return PDA_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PDA_ERR_CUDA;
    size_t mx = 0;
    for (int b = 16; b <= 128; b += 16) {
      const size_t sb = ring_shape(b).smem_bytes;
      mx = sb > mx ? sb : mx;
    }
    for (bool paired : {false, true})
      if (cudaFuncSetAttribute(split_fn(kPlainWide, paired), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mx) !=
          cudaSuccess)
        return PDA_ERR_CUDA;
    d.scratch = ptr;
    d.sm_count = sms;
    d.ready = true;
  }
  int& occ = d.occ[bs / 16];
  if (occ == 0) {
    int m = 0;
    for (bool paired : {false, true}) {
      int n = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, split_fn(kPlainWide, paired), pda::kThreads,
                                                        ring_shape(bs).smem_bytes) != cudaSuccess)
        return PDA_ERR_CUDA;
      m = (m == 0 || n < m) ? n : m;
    }
    occ = m > 0 ? m : 1;
  }
  *out = d;
  return PDA_OK;
}

void noalloc_forget_devices() {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  for (auto& d : g_noalloc_dev) d = NoAllocDevice{};
}

}  // namespace

extern "C" pda_status pda_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                                         int num_heads, int num_kv_heads, int head_size, int block_size,
                                         int max_num_blocks_per_seq, float scale, float k_scale, float v_scale,
                                         cudaStream_t stream) {
  pda_status st = validate(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads, num_kv_heads,
                           head_size, block_size, max_num_blocks_per_seq, scale, k_scale, v_scale);
  if (st != PDA_OK || num_seqs == 0) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PDA_ERR_CUDA;
  NoAllocDevice d;
  st = noalloc_setup(dev, block_size, &d);
  if (st != PDA_OK) return st;
  const int MB = max_num_blocks_per_seq > 0 ? max_num_blocks_per_seq : 1;
  const int nsplit =
      resolve_splits(num_seqs, num_kv_heads, MB, block_size, d.sm_count, d.occ[block_size / 16], g_split_override.load());
  if (partial_bytes(num_seqs, num_heads, nsplit) > kNoAllocScratchBytes) return PDA_ERR_NOALLOC_CAPACITY;

  const RingShape rs = ring_shape(block_size);
  float* scratch = static_cast<float*>(d.scratch);
  pda::DecodeParams p;
  p.block_limit = g_block_limit.load();
  p.out = out;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.part_o = scratch;
  p.part_ml = scratch + (size_t)num_seqs * num_heads * nsplit * kHeadDim;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.gqa = num_heads / num_kv_heads;
  p.block_size = block_size;
  p.max_blocks = max_num_blocks_per_seq;
  p.nsplit = nsplit;
  p.pages_per_stage = rs.pages_per_stage;
  p.num_stages = rs.num_stages;
  p.stage_bytes = rs.stage_bytes;
  p.scale_off = rs.scale_off;
  p.k_scales = nullptr;
  p.v_scales = nullptr;
  p.logit_scale_log2 = (float)((double)scale * (double)k_scale * 1.4426950408889634);
  p.v_scale = v_scale;
  dim3 grid((unsigned)nsplit, (unsigned)num_kv_heads, (unsigned)num_seqs);
  {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = dim3(pda::kThreads);
    lc.dynamicSmemBytes = rs.smem_bytes;
    lc.stream = stream;
    if (cudaLaunchKernelEx(&lc, split_fn(kPlainWide, paired_for(p.gqa)), p, g_no_map, g_no_map) != cudaSuccess)
      return PDA_ERR_CUDA;
  }
  if (nsplit > 1) {
    pda::MergeParams mp;
    mp.out = p.out;
    mp.part_o = p.part_o;
    mp.part_ml = p.part_ml;
    mp.seq_lens = seq_lens;
    mp.num_heads = num_heads;
    mp.block_size = block_size;
    mp.max_blocks = max_num_blocks_per_seq;
    mp.nsplit = nsplit;
    mp.v_scale = v_scale;
    mp.num_seqs = num_seqs;
    if (launch_merge(mp, stream, false) != cudaSuccess) return PDA_ERR_CUDA;
  }
  return PDA_OK;
}
