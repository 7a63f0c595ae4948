// The library's kernels (sm_103a):
//   pda_split_decode_kernel       one CTA per work unit (below)
//   pda_persistent_decode_kernel  one CTA per resident slot taking work units
//                                 from a queue, the same per-unit arithmetic
//   pda_order_units_kernel        longest-first order of the queued units,
//                                 and the pieces of the last partial round
//   pda_tail_merge_kernel         log-sum-exp fold of those pieces
//   pda_merge_kernel              log-sum-exp merge of split partials (one
//                                 warp per row; pda_merge_wide_kernel past
//                                 16 splits)
//   pda_reshape_and_cache_kernel  KV-cache write (and a scattered variant)
//
// Work unit: one (sequence, kv head, KV split). Per unit:
//   * warp kConsumerWarps (the producer) gathers the split's pages through
//     the block table and streams them with bulk (TMA) copies into a ring
//     of shared-memory stages, one mbarrier pair per stage (16-token pages
//     in the persistent kernel: four at a time by a TMA gather);
//   * warps 0..kConsumerWarps-1 (the consumers) each take 16-token tiles of
//     a stage and run, for all query heads of the GQA group at once,
//       S^T = K_tile (16 tok x 128) * Q^T (128 x 8 heads)     (warp MMA)
//       online softmax over tokens in fp32 (exp2 domain)
//       O^T += V_tile^T (128 x 16 tok) * P^T (16 tok x 8 heads)
//     with K and V dequantised exactly from e4m3 to f16 in registers, once
//     per tile for every head of the group, the query rows shifted by a
//     power of two into f16's range, and P carried as two f16 parts;
//   * the consumers merge their (m, l, O) through shared memory and either
//     write bf16 output (one split) or an fp32 partial (several splits) that
//     the merge kernel combines by log-sum-exp.
//
// The pages give the cache layout (K [blocks, kv_heads, head_size/16, bs, 16],
// V [blocks, kv_heads, head_size, bs]; vLLM pull request
// lishuoshuo-amd/vllm#3, "Details" -> "Layout") and what the call computes
// (vLLM API page vllm.v1.attention.backends.rocm_aiter_unified_attn,
// RocmAiterUnifiedAttentionImpl.forward). The kernel design is this
// library's own.
#pragma once

#include "pda_device.cuh"

namespace pda {

// Compile-time tuning: consumer warps per CTA and shared-memory ring bytes.
#ifndef PDA_CONSUMER_WARPS
#define PDA_CONSUMER_WARPS 4
#endif
#ifndef PDA_RING_BYTES
#define PDA_RING_BYTES 65536
#endif
// Two residency targets for the decode kernel, chosen per call: 3 CTAs per
// SM with the full ring for large batches, 4 CTAs per SM with a 48 KiB ring
// (registers capped by the launch bounds) when the whole grid fits one wave.
constexpr int kWideCtasPerSm = 3;
constexpr int kDenseCtasPerSm = 4;
constexpr int kDenseRingBytes = 49152;
#ifndef PDA_PERSIST_CTAS
#define PDA_PERSIST_CTAS 3
#endif
#ifndef PDA_PERSIST_RING_BYTES
#define PDA_PERSIST_RING_BYTES 65536
#endif
constexpr int kPersistCtasPerSm = PDA_PERSIST_CTAS;
constexpr int kPersistRingBytes = PDA_PERSIST_RING_BYTES;

constexpr int kHeadDim = 128;
constexpr int kChunks = kHeadDim / 16;       // 16-dim chunks of a K page
constexpr int kConsumerWarps = PDA_CONSUMER_WARPS;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;
constexpr int kStageTokensMin = 16 * kConsumerWarps;  // one 16-token tile per consumer warp per stage
constexpr int kRingBytes = PDA_RING_BYTES;
constexpr int kMaxPagesPerStage = kStageTokensMin / 16;  // 16-token pages; divides 32
static_assert(32 % kMaxPagesPerStage == 0, "stage pages must tile a 32-entry table chunk");
constexpr int kMaxGqa = 8;                   // MMA N dimension: query heads of a group
constexpr int kMergeStride = kHeadDim + 4;   // padded fp32 row of the CTA merge area
// Cluster merge (per-unit kernel, one wave, 2..kMaxClusterSplits splits):
// each CTA keeps its merged rows [kMaxGqa][kHeadDim] and (m, l) pairs
// [kMaxGqa][2] in shared memory right after the CTA merge area.
constexpr int kMaxClusterSplits = 16;
constexpr int kClusterPartOff = kConsumerWarps * kMaxGqa * (kMergeStride + 2) * 4;  // bytes
constexpr int kClusterPartBytes = (kMaxGqa * kHeadDim + kMaxGqa * 2) * 4;

// Swizzled native V pages ([128 dims][bs tokens], rows bs bytes apart): an
// ldmatrix reads the 8 rows of dims 8j..8j+7 at one 16-byte token chunk,
// which at 32-, 64- and 128-byte rows falls on 2, 2 and 1 bank groups
// (4- to 8-way conflicts). Loaded through a tensor map with the 32-, 64- or
// 128-byte TMA swizzle, chunk c of row d lands at chunk c ^ f(d):
//   32 B rows:  f(d) = (d >> 2) & 1      (address bit 4 ^= bit 7)
//   64 B rows:  f(d) = (d >> 1) & 3      (bits 4-5 ^= bits 7-8)
//   128 B rows: f(d) = d & 7             (bits 4-6 ^= bits 7-9)
// and the 8 rows of one ldmatrix fall on 8 distinct bank groups. Since the
// ldmatrix rows are dims 32mp + 8j + (lane & 7), f depends on the lane only.
enum : int { kVSwizzleNone = 0, kVSwizzle32 = 1, kVSwizzle64 = 2, kVSwizzle128 = 3 };
__device__ __forceinline__ uint32_t v_swizzle_xor(int mode, int lane) {
  switch (mode) {
    case kVSwizzle32: return (uint32_t)((lane >> 2) & 1);
    case kVSwizzle64: return (uint32_t)((lane >> 1) & 3);
    case kVSwizzle128: return (uint32_t)(lane & 7);
    default: return 0u;
  }
}

struct DecodeParams {
  void* out;                    // [S][H][D] bf16, or e4m3 bytes when out_fp8
  const __nv_bfloat16* q;       // [S][H][D]
  const uint8_t* k_cache;       // [NB][Hk][D/16][bs][16]
  const uint8_t* v_cache;       // [NB][Hk][D][bs]
  const int32_t* block_tables;  // [S][MB]
  const int32_t* seq_lens;      // [S]
  float* part_o;                // [S][H][nsplit][D]   (nsplit > 1)
  float* part_ml;               // [S][H][nsplit][2]   (nsplit > 1): m (log2 units), l
  int num_heads;
  int num_kv_heads;
  int gqa;
  int block_size;
  int max_blocks;               // block table row stride
  int nsplit;
  int pages_per_stage;
  int num_stages;
  uint32_t stage_bytes;
  uint32_t scale_off;           // per-slot scale rows inside a stage (slot-scale variant)
  const float* k_scales;        // [NB][Hk][bs] fp32 (slot-scale variant)
  const float* v_scales;        // [NB][Hk][bs] fp32 (slot-scale variant)
  // Slot-scale variant: how a stage's K and V scale rows arrive.
  // kScaleRowsGather4 (4 pages a stage): one four-row gather per table
  // through tm_k / tm_v (2-D maps over the tables as [NB * Hk][bs] rows);
  // kScaleRowsBulk: one bulk copy per row; kScaleRowsPieces: 16-byte
  // cp.async pieces spread over the producer warp.
  int scale_rows = 0;
  // Page-major 16-token pages (4 a stage), not per-slot scales nor cluster
  // merges: 1 = a stage's 4 K pages and 4 V pages arrive as one four-row
  // gather each through tm_k / tm_v (2-D maps over the caches as [NB * Hk]
  // rows of one 2 KiB page); 0 = one bulk copy per page.
  int page_gather = 0;
  float logit_scale_log2;       // scale * k_scale * log2(e)  (scale * log2(e) with slot scales)
  float v_scale;                // per-tensor V scale (unused with slot scales)
  int v_shuffled = 0;           // 1: V pages are [bs/16][D][16] (AITER shuffled), else [D][bs]
  // Native V pages of 32-, 64- or 128-token blocks arrive through a tensor
  // map (tm_v) with the TMA swizzle whose span is one page row (kVSwizzle*),
  // else (0) as one 1-D bulk copy.
  int v_swizzle = 0;
  // Token-major variant: position (1..3) of the token, kv-head and block
  // dimensions in the 4-D tensor maps (dimension 0 is the 128 bytes of a row).
  int tm_dim_token = 1;
  int tm_dim_head = 2;
  int tm_dim_block = 3;
  const float* sinks = nullptr; // [H] per-head sink logits (scale * q.k units), or none
  int out_fp8 = 0;              // 1: out holds E4M3(o / out_scale) bytes
  float out_scale = 1.f;
  // Persistent kernel: unit of ticket gridDim.x + i is unit_order[i]
  // (longest first, written by pda_order_units_kernel), or ticket order.
  const int* unit_order = nullptr;
  // Block check: nonzero = the pool size; a block id outside [0, block_limit)
  // is recorded in the status word and read as block 0.
  uint32_t block_limit = 0u;
  // 1 when the per-unit kernel's cluster build runs with clusters of nsplit
  // CTAs (read only by that build).
  int cluster_merge = 0;
  // Persistent kernel, tail pieces: tickets from tail_first on take the
  // entries {unit, first page, end page, slot} of piece_table (pages of the
  // unit's split; slot -1 for a whole unit), which the order kernel writes
  // each call along with the ticket count (*num_tickets). A piece stores
  // its (O, m, l) rows in tail_rows (kTailRowFloats per slot); the tail
  // merge kernel folds each unit's pieces.
  unsigned tail_first = 0xFFFFFFFFu;
  const int4* piece_table = nullptr;
  const int* num_tickets = nullptr;
  float* tail_rows = nullptr;
};
constexpr int kTailRowFloats = kMaxGqa * (kHeadDim + 2);
constexpr int kMaxTailPieces = 8;  // most pieces a tail unit is cut into
// A tail unit is cut only when it holds at least kMinCutPieces pieces of
// the minimum size: the tail merge kernel's fold costs about as much as a
// CTA spends on 1024 tokens alone (GB300, 256 sequences of 1 to 4000
// tokens: its shortest units in 2 pieces took 161.2 us per call, left
// whole 159.0 us).
constexpr int kMinCutPieces = 4;

// DecodeParams::scale_rows: how a stage's per-slot scale rows arrive.
constexpr int kScaleRowsPieces = 0;
constexpr int kScaleRowsGather4 = 1;
constexpr int kScaleRowsBulk = 2;

// The rows b * Hk + kvh of a stage's np (1..4) pages in a table or cache
// viewed as [NB * Hk] rows, for a four-row gather; rows past np repeat the
// first (the gather lands them in the stage's unused slots).
__device__ __forceinline__ int4 stage_rows(const int* blk, int np, int Hk, int kvh) {
  const int r0 = blk[0] * Hk + kvh;
  return make_int4(r0, np > 1 ? blk[1] * Hk + kvh : r0, np > 2 ? blk[2] * Hk + kvh : r0,
                   np > 3 ? blk[3] * Hk + kvh : r0);
}

// Splits of a sequence with `pages` pages that hold at least one page (the
// others are empty: they write no partial and take no part in the merge).
__device__ __forceinline__ int active_splits(int pages, int nsplit) {
  if (pages <= 0) return 0;
  const int per = (pages + nsplit - 1) / nsplit;
  return (pages + per - 1) / per;
}

// One log-sum-exp step: the running (M, den, acc) of 4 dims absorbs a split's
// (m, l, O). The products and sums are spelled out (no contraction choice
// left to the compiler), so every merge site gives the same bits.
__device__ __forceinline__ void lse_fold(float& M, float& den, float4& acc, float m, float l, const float4& o) {
  const float mn = fmaxf(M, m);
  const float a = fast_exp2(M - mn);  // 0 while M is -inf
  const float f = fast_exp2(m - mn);
  acc.x = __fmaf_rn(acc.x, a, __fmul_rn(f, o.x));
  acc.y = __fmaf_rn(acc.y, a, __fmul_rn(f, o.y));
  acc.z = __fmaf_rn(acc.z, a, __fmul_rn(f, o.z));
  acc.w = __fmaf_rn(acc.w, a, __fmul_rn(f, o.w));
  den = __fmaf_rn(den, a, __fmul_rn(f, l));
  M = mn;
}

// The partials of one (sequence, head) row folded in split order, dims
// 4 lane .. 4 lane + 3 (one warp per row). Row prow0 + i holds split i.
__device__ __forceinline__ void lse_fold_row(const float* part_o, const float* part_ml, size_t prow0, int active,
                                             int lane, float& M, float& den, float4& acc) {
  M = -INFINITY;
  den = 0.f;
  acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int i = 0; i < active; ++i) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(part_ml) + (prow0 + i));
    const float4 o = __ldcg(reinterpret_cast<const float4*>(part_o + (prow0 + i) * kHeadDim) + lane);
    lse_fold(M, den, acc, ml.x, ml.y, o);
  }
}

// A block id the producer is about to read, checked when the block check is on.
__device__ __forceinline__ int checked_block(int b, uint32_t limit) {
  if (limit != 0u && (uint32_t)b >= limit) {
    atomicOr(&g_status, kStatusBadBlock);
    return 0;
  }
  return b;
}

// Final normalisation shared by the decode kernel (one split) and the merge
// kernel: a sink logit zs (log2 units, -inf for none) joins the normaliser
// only; M is the running max of the numerator terms.
__device__ __forceinline__ float finish(float acc, float den, float M, float zs, float vfac) {
  if (zs != -INFINITY) {
    const float Mn = fmaxf(M, zs);
    const float f = (M == -INFINITY) ? 0.f : fast_exp2(M - Mn);
    acc *= f;
    den = den * f + fast_exp2(zs - Mn);
  }
  return den > 0.f ? acc * (vfac / den) : 0.f;
}

// Store one output element: bf16, or the e4m3 code of x / out_scale (IEEE
// binary32 quotient, round to nearest even, saturating at +-448).
__device__ __forceinline__ void store_out(void* out, size_t idx, float x, int out_fp8, float out_scale) {
  if (out_fp8) {
    static_cast<uint8_t*>(out)[idx] = (uint8_t)(f32x2_to_e4m3x2(__fdiv_rn(x, out_scale), 0.f) & 0xFFu);
  } else {
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(x);
  }
}

// Store lane's 4 dims of the merged row (s, h): zeros when no split held a
// page (any == false).
__device__ __forceinline__ void store_merged(void* out, const float* sinks, int out_fp8, float out_scale,
                                             float v_scale, int num_heads, int s, int h, int lane, bool any, float M,
                                             float den, const float4& acc) {
  const float zs = sinks ? __ldg(sinks + h) * 1.4426950408889634f : -INFINITY;
  const float r[4] = {acc.x, acc.y, acc.z, acc.w};
  const size_t o0 = ((size_t)s * num_heads + h) * kHeadDim + 4 * lane;
#pragma unroll
  for (int j = 0; j < 4; ++j) store_out(out, o0 + j, any ? finish(r[j], den, M, zs, v_scale) : 0.f, out_fp8, out_scale);
}

// Token order of the 16 MMA rows of a K tile. Row r of the QK accumulator
// holds token row_token(r); the order is chosen so that, after the P
// fragment is transposed with movmatrix, each lane holds the probabilities
// of exactly the 4 consecutive tokens whose V bytes ldmatrix hands it (as
// two pairs, in swapped order for lanes whose tig >= 2), and so that both
// 8-row K ldmatrix groups hit 8 distinct 16-byte bank groups.
// Rows 0..7 -> tokens 0,1,4,5,10,11,14,15; rows 8..15 -> 2,3,6,7,8,9,12,13.
__device__ __forceinline__ int row_token(int r) {
  const int hi = r >> 3;            // which 8-row half
  const int t = (r >> 1) & 3;       // lane quad index the row pair maps to
  const int e = r & 1;
  const int swap = (t >= 2) ? 1 : 0;
  return 4 * t + 2 * (hi ^ swap) + e;
}

// Pages [first, end) of split `split` for a sequence with `pages` pages.
__device__ __forceinline__ void split_range(int pages, int nsplit, int split, int& first, int& end) {
  const int per = (pages + nsplit - 1) / nsplit;
  first = split * per;
  end = min(pages, first + per);
}

__device__ __forceinline__ float warp_max_over_gid(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
  return v;
}
__device__ __forceinline__ float warp_sum_over_gid(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

// One consumer warp's share of a work unit: the GQA group's Q^T fragments
// and the running softmax state (m, l, O^T) of the unit, updated one
// 16-token tile at a time (the template flags are those of the kernels).
template <bool kSlotScales, bool kTokenMajor, bool kPaired, bool kLateRemainder = false>
struct TileWorker {
  int gid, tig;
  uint32_t k_lane_off;   // page-major K: ldmatrix row of this lane
  uint32_t tm_row, tm_xor, tm_hi;  // token-major tiles: row, swizzle and chunk half
  uint32_t v_row, v_lane_off;
  uint32_t v_xor;        // swizzled native V: this lane's chunk XOR (0 otherwise)
  bool low_quad;
  // Paired columns (kPaired, for GQA groups of at most 4 heads): MMA
  // columns 4..7 repeat heads 0..3, so the lanes that own them (tig >= 2)
  // compute the same scores, maxima and probabilities as their partners
  // (lane ^ 2) and feed the PV product the f16 remainder P - f16(P) instead
  // of f16(P); the two halves of O are added when the warp stores its merge
  // rows. Wider groups run a second PV MMA on the remainders. The choice is
  // a template parameter so that each kernel instance holds only its own
  // PV code (the other path's registers and branches cost the tile loop
  // time even when not taken).
  static constexpr bool paired = kPaired;
  bool hi_lane;          // tig < 2: this lane's P columns carry f16(P)
  int slot_tok_a, slot_tok_b;  // slot-scale instances: tokens of accumulator rows gid, gid + 8
  uint32_t qf[kChunks][2];
  float lsc0, lsc1;      // logit scale (log2 units) of columns 2tig, 2tig+1, with the query rows' shifts
  float m0, m1;          // running max (log2 units), heads 2tig, 2tig+1
  float l0, l1;          // running partial sums over this lane's tokens
  float o[kChunks][4];   // O^T: m-tile mt = dims 16mt.. ; cols heads 2tig, 2tig+1

  __device__ __forceinline__ void setup(int lane, int bs, int v_shuffled, int v_swizzle) {
    gid = lane >> 2;
    tig = lane & 3;
    // ldmatrix row assignment. K: lane l supplies token row_token(l & 15) of
    // chunk (2kk + (l >> 4)). V: lane l supplies dim (32mp + l).
    k_lane_off = (uint32_t)(row_token(lane & 15) * 16) + (uint32_t)((lane >> 4) * bs * 16);
    // Token-major tiles: lane l addresses token row (l & 15), chunk (2j + (l >> 4)),
    // swizzled by the row's low 3 bits.
    tm_row = (uint32_t)(lane & 15) * 128u;
    tm_xor = (uint32_t)(lane & 7);
    tm_hi = (uint32_t)(lane >> 4);
    // V: a 16-token tile is 128 rows of 16 bytes at stride v_row (bs for
    // [D][bs] pages; 16 for shuffled [bs/16][D][16] pages, whose tiles are
    // contiguous and so bank-conflict free for any block size).
    v_row = v_shuffled ? 16u : (uint32_t)bs;
    v_lane_off = (uint32_t)lane * v_row;
    v_xor = v_swizzle_xor(v_swizzle, lane);
    // The slot-scale instances read two scales per row every tile, so they
    // keep the rows' tokens in registers; the others compute them in tail
    // tiles only (tok_a / tok_b), where their registers are scarcer.
    slot_tok_a = tok_a();
    slot_tok_b = tok_b();
    low_quad = kTokenMajor ? true : tig < 2;
    hi_lane = tig < 2;
  }

  // Tokens of accumulator rows gid and gid + 8 (computed where needed, not
  // held in registers through the tile loop).
  __device__ __forceinline__ int tok_a() const { return kTokenMajor ? gid : row_token(gid); }
  __device__ __forceinline__ int tok_b() const { return kTokenMajor ? gid + 8 : row_token(gid + 8); }

  __device__ __forceinline__ void reset() {
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int i = 0; i < kChunks; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  }

  // The query head whose row MMA column `gid` holds: gid itself, or in
  // paired mode gid mod 4 (columns 4..7 repeat heads 0..3).
  __device__ __forceinline__ int q_head() const { return paired ? (gid & 3) : gid; }

  // Q^T fragments (B operand, 16 dims x 8 heads per chunk) in f16 from the
  // bf16 query row of head q_head() (zeros when that head is past the
  // group). Chunk c k-slots (2tig, 2tig+1) <- dims 16c+4tig+{0,1};
  // (2tig+8, 2tig+9) <- dims 16c+4tig+{2,3}; this matches how K bytes land
  // in the A fragments below.
  //
  // bf16 reaches 2^127 and f16 only 65504, so each row is first scaled by a
  // power of two 2^-e that puts its largest |q| in [2^14, 2^15): every bf16
  // value of the row down to 2^-24 of that maximum is then exact in f16
  // (smaller ones cannot move a logit by more than 2^-24 of the row's
  // largest term). The columns' logit scales are multiplied by 2^e, so the
  // logits are the unshifted ones (both factors are exact powers of two).
  // `lsc` is scale * k_scale * log2(e) (scale * log2(e) with slot scales).
  // ld(c) returns the 4 bf16 values of chunk c this lane holds; it is
  // called twice per chunk (max pass, convert pass), so that the raw row is
  // never held in registers at once.
  template <class Ld>
  __device__ __forceinline__ void set_q(const Ld& ld, float lsc) {
    uint32_t mx = 0u;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const uint2 v = ld(c);
      mx = __vmaxu2(mx, v.x & 0x7FFF7FFFu);
      mx = __vmaxu2(mx, v.y & 0x7FFF7FFFu);
    }
    mx = max(mx & 0xFFFFu, mx >> 16);  // |q| bits order like |q| (finite q)
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));  // over the row's four lanes
    const int e = mx == 0u ? 0 : min(max((int)(mx >> 7) - 127 - 14, -100), 113);
    const float down = exp2_int(-e);
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const uint2 v = ld(c);
      qf[c][0] = pack_f16x2(bf16lo_f32(v.x) * down, bf16hi_f32(v.x) * down);
      qf[c][1] = pack_f16x2(bf16lo_f32(v.y) * down, bf16hi_f32(v.y) * down);
    }
    // column 2tig's row sits in lanes 8tig..8tig+3, column 2tig+1's in 8tig+4..
    lsc0 = lsc * exp2_int(__shfl_sync(0xffffffffu, e, 8 * tig));
    lsc1 = lsc * exp2_int(__shfl_sync(0xffffffffu, e, 8 * tig + 4));
  }
  __device__ __forceinline__ void load_q_global(const __nv_bfloat16* qrow, bool live, float lsc) {
    const int t4 = 4 * tig;
    set_q([&](int c) { return live ? ld_nc_v2(qrow + 16 * c + t4) : make_uint2(0u, 0u); }, lsc);
  }
  __device__ __forceinline__ void load_q_shared(uint32_t qrow, bool live, float lsc) {
    const uint32_t t8 = (uint32_t)(8 * tig);
    set_q([&](int c) { return live ? ld_shared_v2(qrow + (uint32_t)(32 * c) + t8) : make_uint2(0u, 0u); }, lsc);
  }

  // One 16-token tile: K bytes at kbase, V bytes at vbase (shared), the first
  // n_valid (>= 1) tokens real. Slot scales: ks / vs point at the tile's 16
  // K and V scales, vinv is 1 / (the reference V scale).
  __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, int bs, int n_valid, const float* ks,
                                       const float* vs, float vinv) {
    // ---- S^T = K_tile * Q^T (two independent accumulator chains)
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    float sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < kChunks / 2; ++kk) {
      uint32_t r0, r1, r2, r3;
      if constexpr (kTokenMajor)
        ldsm_x4(kbase + tm_row + ((((uint32_t)(2 * kk) + tm_hi) ^ tm_xor) << 4), r0, r1, r2, r3);
      else
        ldsm_x4(kbase + k_lane_off + (uint32_t)(2 * kk * bs * 16), r0, r1, r2, r3);
      mma_f16(sc, e4m3x2_lo_to_f16x2(r0), e4m3x2_lo_to_f16x2(r1), e4m3x2_hi_to_f16x2(r0),
              e4m3x2_hi_to_f16x2(r1), qf[2 * kk][0], qf[2 * kk][1]);
      mma_f16(sd, e4m3x2_lo_to_f16x2(r2), e4m3x2_lo_to_f16x2(r3), e4m3x2_hi_to_f16x2(r2),
              e4m3x2_hi_to_f16x2(r3), qf[2 * kk + 1][0], qf[2 * kk + 1][1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) sc[i] += sd[i];

    // ---- online softmax (exp2 domain); tokens >= n_valid are masked
    float lA0 = lsc0, lA1 = lsc1, lB0 = lsc0, lB1 = lsc1, vsA = 1.f, vsB = 1.f;
    if constexpr (kSlotScales) {
      // Scales of slots past the length may hold anything (even NaN).
      const int tA = slot_tok_a, tB = slot_tok_b;
      const bool vA = tA < n_valid, vB = tB < n_valid;
      const float kA = vA ? ks[tA] : 0.f;
      const float kB = vB ? ks[tB] : 0.f;
      lA0 *= kA;
      lA1 *= kA;
      lB0 *= kB;
      lB1 *= kB;
      vsA = vA ? vs[tA] * vinv : 0.f;
      vsB = vB ? vs[tB] * vinv : 0.f;
    }
    float s0 = sc[0] * lA0;
    float s1 = sc[1] * lA1;
    float s2 = sc[2] * lB0;
    float s3 = sc[3] * lB1;
    if (n_valid < 16) {  // a tail tile (warp-uniform): its last slots are not tokens
      if (tok_a() >= n_valid) s0 = s1 = -INFINITY;
      if (tok_b() >= n_valid) s2 = s3 = -INFINITY;
    }
    const float mx0 = warp_max_over_gid(fmaxf(s0, s2));
    const float mx1 = warp_max_over_gid(fmaxf(s1, s3));
    const float mn0 = fmaxf(m0, mx0);
    const float mn1 = fmaxf(m1, mx1);
    const float c0 = fast_exp2(m0 - mn0);
    const float c1 = fast_exp2(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    const float p0 = fast_exp2(s0 - mn0);
    const float p1 = fast_exp2(s1 - mn1);
    const float p2 = fast_exp2(s2 - mn0);
    const float p3 = fast_exp2(s3 - mn1);
    l0 = l0 * c0 + (p0 + p2);
    l1 = l1 * c1 + (p1 + p3);
    if (__any_sync(0xffffffffu, (c0 != 1.f) | (c1 != 1.f))) {  // a running max moved
#pragma unroll
      for (int mt = 0; mt < kChunks; ++mt) {
        o[mt][0] *= c0;
        o[mt][1] *= c1;
        o[mt][2] *= c0;
        o[mt][3] *= c1;
      }
    }
    // P in two f16 parts, f16(P) and f16(P - f16(P)) (the difference is
    // exact in fp32): together they carry P to about 2^-22 relative (2^-25
    // absolute below 2^-3), where f16(P) alone would lose 2^-12.
    float a0 = p0, a1 = p1, a2 = p2, a3 = p3;
    if constexpr (kSlotScales) {
      a0 *= vsA;
      a1 *= vsA;
      a2 *= vsB;
      a3 *= vsB;
    }
    const uint32_t h0 = pack_f16x2(a0, a1);
    const uint32_t h1 = pack_f16x2(a2, a3);
    const uint32_t r0 = pack_f16x2(a0 - f16lo_f32(h0), a1 - f16hi_f32(h0));
    const uint32_t r1 = pack_f16x2(a2 - f16lo_f32(h1), a3 - f16hi_f32(h1));
    // P^T fragment: transpose (token rows x head cols) to (head rows x token
    // cols). Lane quads 2 and 3 hold their two token pairs in the other
    // order (row_token), so they swap the two halves of the B fragment. In
    // paired mode the remainder columns ride in the same fragment; otherwise
    // the remainders get a fragment of their own (pl0, pl1).
    const bool take_hi = !paired || hi_lane;
    const uint32_t t0 = movmatrix_trans(take_hi ? h0 : r0);
    const uint32_t t1 = movmatrix_trans(take_hi ? h1 : r1);
    const uint32_t pb0 = low_quad ? t0 : t1;
    const uint32_t pb1 = low_quad ? t1 : t0;

    // ---- O^T += V_tile^T * P^T
    // Page-major V: lane holds V bytes of tokens 4tig..4tig+3 of one dim.
    // Token-major V (ldmatrix.trans): a register holds tokens (2tig, 2tig+1)
    // x dims (2gid, 2gid+1) of a chunk; registers 0/2 tokens 0-7, 1/3 8-15.
    uint32_t vr[kChunks / 2][4];
#pragma unroll
    for (int mp = 0; mp < kChunks / 2; ++mp) {
      if constexpr (kTokenMajor)
        ldsm_x4_trans(vbase + tm_row + ((((uint32_t)(2 * mp) + tm_hi) ^ tm_xor) << 4), vr[mp][0], vr[mp][1],
                      vr[mp][2], vr[mp][3]);
      else
        ldsm_x4(vbase + v_lane_off + (uint32_t)(32 * mp) * v_row, vr[mp][0], vr[mp][1], vr[mp][2], vr[mp][3]);
    }
    if (n_valid < 16) {
      // Zero the V bytes of tokens >= n_valid: their e4m3 codes may be NaN
      // and 0 * NaN would poison the accumulator.
      if constexpr (kTokenMajor) {
        const uint32_t m_lo = (2 * tig < n_valid ? 0x0000FFFFu : 0u) | (2 * tig + 1 < n_valid ? 0xFFFF0000u : 0u);
        const uint32_t m_hi =
            (8 + 2 * tig < n_valid ? 0x0000FFFFu : 0u) | (9 + 2 * tig < n_valid ? 0xFFFF0000u : 0u);
#pragma unroll
        for (int mp = 0; mp < kChunks / 2; ++mp) {
          vr[mp][0] &= m_lo;
          vr[mp][1] &= m_hi;
          vr[mp][2] &= m_lo;
          vr[mp][3] &= m_hi;
        }
      } else {
        const int k = min(max(n_valid - 4 * tig, 0), 4);
        const uint32_t vmask = k >= 4 ? 0xFFFFFFFFu : ((1u << (8 * k)) - 1u);
#pragma unroll
        for (int mp = 0; mp < kChunks / 2; ++mp)
#pragma unroll
          for (int i = 0; i < 4; ++i) vr[mp][i] &= vmask;
      }
    }
    // Each instance has one straight block of conversions and MMAs, which the
    // compiler can interleave freely.
    if constexpr (kPaired) {
      pv_mma(vr, pb0, pb1, pb0, pb1, false);
    } else {
      const uint32_t u0 = movmatrix_trans(r0);
      const uint32_t u1 = movmatrix_trans(r1);
      pv_mma(vr, pb0, pb1, low_quad ? u0 : u1, low_quad ? u1 : u0, true);
    }
  }

  // V_tile^T A fragments of m-tile pair mp, half h (16 dims x 16 tokens, f16).
  __device__ __forceinline__ void v_frag(const uint32_t (&vr)[kChunks / 2][4], int mp, int h, uint32_t (&a)[4]) {
    if constexpr (kTokenMajor) {
      // bytes (t,d0) (t,d1) (t',d0) (t',d1) -> (t,d0) (t',d0) | (t,d1) (t',d1)
      const uint32_t ya = __byte_perm(vr[mp][2 * h], 0, 0x3120);
      const uint32_t yb = __byte_perm(vr[mp][2 * h + 1], 0, 0x3120);
      a[0] = e4m3x2_lo_to_f16x2(ya);
      a[1] = e4m3x2_hi_to_f16x2(ya);
      a[2] = e4m3x2_lo_to_f16x2(yb);
      a[3] = e4m3x2_hi_to_f16x2(yb);
    } else {
      a[0] = e4m3x2_lo_to_f16x2(vr[mp][2 * h]);
      a[1] = e4m3x2_lo_to_f16x2(vr[mp][2 * h + 1]);
      a[2] = e4m3x2_hi_to_f16x2(vr[mp][2 * h]);
      a[3] = e4m3x2_hi_to_f16x2(vr[mp][2 * h + 1]);
    }
  }

  // O^T += V_tile^T * P^T for the 8 m-tiles of 16 dims: B fragment (pb0,
  // pb1), and with `second` a second B fragment (pl0, pl1). With
  // kLateRemainder the second pass follows all first-pass MMAs (the V
  // fragments are converted again), so no MMA waits on its accumulator's
  // previous one; without it each second MMA reuses the converted
  // fragments right away (fewer registers, for the 4-CTA instances).
  __device__ __forceinline__ void pv_mma(const uint32_t (&vr)[kChunks / 2][4], uint32_t pb0, uint32_t pb1,
                                         uint32_t pl0, uint32_t pl1, bool second) {
#pragma unroll
    for (int mp = 0; mp < kChunks / 2; ++mp) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t a[4];
        v_frag(vr, mp, h, a);
        mma_f16(o[2 * mp + h], a[0], a[1], a[2], a[3], pb0, pb1);
        if (second && !kLateRemainder) mma_f16(o[2 * mp + h], a[0], a[1], a[2], a[3], pl0, pl1);
      }
    }
    if (second && kLateRemainder) {
#pragma unroll
      for (int mp = 0; mp < kChunks / 2; ++mp) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t a[4];
          v_frag(vr, mp, h, a);
          mma_f16(o[2 * mp + h], a[0], a[1], a[2], a[3], pl0, pl1);
        }
      }
    }
  }

  // Merge rows a warp stores: the group's heads. Paired instances keep only
  // heads 0..3 (columns 4..7 are their remainders, folded in below), so
  // their rows fit the padded stride even where the merge area is one ring
  // stage of 16 KiB.
  static constexpr int kMergeRows = kPaired ? kMaxGqa / 2 : kMaxGqa;

  // This warp's (m, l, O) into the CTA merge area: mo [w][kMergeRows][kStride],
  // mml [w][kMaxGqa][2].
  template <int kStride>
  __device__ __forceinline__ void store_merge(float* mo, float* mml, int warp) {
    l0 = warp_sum_over_gid(l0);
    l1 = warp_sum_over_gid(l1);
    if constexpr (kPaired) {
      // f16(P) . V (columns 0..3) + remainder . V (columns 4..7)
#pragma unroll
      for (int mt = 0; mt < kChunks; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[mt][i] += __shfl_xor_sync(0xffffffffu, o[mt][i], 2);
    }
    if (!kPaired || hi_lane) {
      float* mw = mo + warp * kMergeRows * kStride;
#pragma unroll
      for (int mt = 0; mt < kChunks; ++mt) {
        // accumulator rows gid / gid + 8 of m-tile mt hold these two dims
        const int d0 = kTokenMajor ? 16 * mt + 2 * gid : 16 * mt + gid;
        const int d1 = kTokenMajor ? d0 + 1 : d0 + 8;
        mw[(2 * tig) * kStride + d0] = o[mt][0];
        mw[(2 * tig + 1) * kStride + d0] = o[mt][1];
        mw[(2 * tig) * kStride + d1] = o[mt][2];
        mw[(2 * tig + 1) * kStride + d1] = o[mt][3];
      }
    }
    if (gid == 0) {
      float* ml = mml + warp * kMaxGqa * 2;
      ml[(2 * tig) * 2 + 0] = m0;
      ml[(2 * tig) * 2 + 1] = l0;
      ml[(2 * tig + 1) * 2 + 0] = m1;
      ml[(2 * tig + 1) * 2 + 1] = l1;
    }
  }
};

// Combine the consumer warps' (m, l, O) of unit (s, kvh, split) from the
// merge area and store the bf16 / e4m3 output (one split) or the fp32
// partial (several splits). Consumer thread `tid` of kConsumerThreads.
// vref: the slot-scale variant's reference V scale (1 otherwise). kStride:
// the fp32 row stride of mo.
// cpart: the cluster merge's shared-memory partial (rows, then (m, l)
// pairs), or nullptr for fp32 partials in global memory.
template <bool kSlotScales, int kStride, int kRows, bool kUnrollRows = false>
__device__ __forceinline__ void reduce_store(const DecodeParams& p, const float* mo, const float* mml, int tid, int s,
                                             int kvh, int split, float vref, float* cpart = nullptr) {
  if constexpr (kUnrollRows && kRows <= kMaxGqa / 2) {
    static_assert(kConsumerThreads == kHeadDim, "one consumer thread per dim");
    const int g = p.gqa;
    const int H = p.num_heads;
    const int d = tid;
    // Thread tid folds dim tid of head hh over the consumer warps and stores
    // it (live: hh is a head of the group).
    auto fold_store = [&](int hh, bool live) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mml[(w * kMaxGqa + hh) * 2]);
      float acc = 0.f, den = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float mw = mml[(w * kMaxGqa + hh) * 2];
          const float f = fast_exp2(mw - M);
          acc += f * mo[(w * kRows + hh) * kStride + d];
          den += f * mml[(w * kMaxGqa + hh) * 2 + 1];
        }
      }
      if (!live) return;
      const int h = kvh * g + hh;
      if (p.nsplit == 1) {
        const float zs = p.sinks ? __ldg(p.sinks + h) * 1.4426950408889634f : -INFINITY;
        const float r = finish(acc, den, M, zs, kSlotScales ? vref : p.v_scale);
        store_out(p.out, ((size_t)s * H + h) * kHeadDim + d, r, p.out_fp8, p.out_scale);
      } else if (cpart) {
        // The same values the global partial would hold, kept in this CTA.
        cpart[hh * kHeadDim + d] = kSlotScales ? acc * vref : acc;
        if (d == 0) {
          cpart[kMaxGqa * kHeadDim + hh * 2 + 0] = M;
          cpart[kMaxGqa * kHeadDim + hh * 2 + 1] = den;
        }
      } else {
        // Slot-scale partials carry their own V reference (the merge then uses 1).
        const size_t prow = ((size_t)s * H + h) * p.nsplit + split;
        p.part_o[prow * kHeadDim + d] = kSlotScales ? acc * vref : acc;
        if (d == 0) {
          p.part_ml[prow * 2 + 0] = M;
          p.part_ml[prow * 2 + 1] = den;
        }
      }
    };
    // Groups of at most 4 heads (paired builds) in the per-unit kernel: all
    // 4 rows unrolled and folded unconditionally (rows past the group are
    // merge-area memory too), so that the heads' independent load / exp2 /
    // divide chains overlap; only the stores are guarded. The CTA merge
    // took 0.6-1.0 us of a 16 x 1024 call (a timer trace); unrolled, GB300
    // runs 4 x 8 units of 4K tokens in 16 splits in 13.7 against 14.1 us
    // and 8 x 8 units of 2K in 9 splits in 12.9 against 13.2 us. Folding
    // all 8 rows of wider groups cost the g = 5 batches 1-1.5 %, and the
    // persistent kernel's per-unit merge lost 0.3 % on the 256 x 4096
    // batch, so those keep the loop over the group's heads.
#pragma unroll
    for (int hh = 0; hh < kRows; ++hh) fold_store(hh, hh < g);
    return;
  }
  const int g = p.gqa;
  const int H = p.num_heads;
  for (int i = tid; i < g * kHeadDim; i += kConsumerThreads) {
    const int hh = i / kHeadDim;
    const int d = i % kHeadDim;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mml[(w * kMaxGqa + hh) * 2]);
    float acc = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = mml[(w * kMaxGqa + hh) * 2];
        const float f = fast_exp2(mw - M);
        acc += f * mo[(w * kRows + hh) * kStride + d];
        den += f * mml[(w * kMaxGqa + hh) * 2 + 1];
      }
    }
    const int h = kvh * g + hh;
    if (p.nsplit == 1) {
      const float zs = p.sinks ? __ldg(p.sinks + h) * 1.4426950408889634f : -INFINITY;
      const float r = finish(acc, den, M, zs, kSlotScales ? vref : p.v_scale);
      store_out(p.out, ((size_t)s * H + h) * kHeadDim + d, r, p.out_fp8, p.out_scale);
    } else if (cpart) {
      // The same values the global partial would hold, kept in this CTA.
      cpart[hh * kHeadDim + d] = kSlotScales ? acc * vref : acc;
      if (d == 0) {
        cpart[kMaxGqa * kHeadDim + hh * 2 + 0] = M;
        cpart[kMaxGqa * kHeadDim + hh * 2 + 1] = den;
      }
    } else {
      // Slot-scale partials carry their own V reference (the merge then uses 1).
      const size_t prow = ((size_t)s * H + h) * p.nsplit + split;
      p.part_o[prow * kHeadDim + d] = kSlotScales ? acc * vref : acc;
      if (d == 0) {
        p.part_ml[prow * 2 + 0] = M;
        p.part_ml[prow * 2 + 1] = den;
      }
    }
  }
}

// Cluster merge of a one-wave split batch. The nsplit CTAs of one (sequence,
// kv head) unit form one thread-block cluster along x, so CTA rank = split.
// Each has left its merged (O, m, l) rows in its own shared memory at byte
// offset kClusterPartOff (reduce_store with cpart). After a cluster barrier,
// consumer warp w of CTA r folds head row r + nsplit * w (nsplit >= 2 and
// g <= 8: at most one row per warp) over the splits that hold pages, in
// split order, with lse_fold and the merge kernel's final step, reading the
// other CTAs' rows through distributed shared memory: the same operations on
// the same values as the merge kernel, so the same bits. The caller's second
// cluster barrier keeps every CTA's shared memory alive until all reads end.
template <bool kSlotScales>
__device__ __forceinline__ void cluster_merge_rows(const DecodeParams& p, uint32_t cpart, int s, int kvh, int split,
                                                   int L, int warp, int lane) {
  const int active = active_splits((L + p.block_size - 1) / p.block_size, p.nsplit);
  constexpr int kBatch = 4;  // splits whose remote loads are in flight together
  for (int hh = split + p.nsplit * warp; hh < p.gqa; hh += p.nsplit * kConsumerWarps) {
    float M = -INFINITY, den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = 0; i0 < active; i0 += kBatch) {
      float2 ml[kBatch];
      float4 o[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (i0 + j < active) {
          const uint32_t base = mapa_cluster(cpart, i0 + j);
          ml[j] = ld_cluster_f2(base + (uint32_t)((kMaxGqa * kHeadDim + hh * 2) * 4));
          o[j] = ld_cluster_f4(base + (uint32_t)((hh * kHeadDim + 4 * lane) * 4));
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (i0 + j < active) lse_fold(M, den, acc, ml[j].x, ml[j].y, o[j]);
    }
    store_merged(p.out, p.sinks, p.out_fp8, p.out_scale, kSlotScales ? 1.f : p.v_scale, p.num_heads, s,
                 kvh * p.gqa + hh, lane, active > 0, M, den, acc);
  }
}

// kSlotScales: K/V dequantise with per-slot fp32 tables [NB][Hk][bs] (the
// per-slot scale tables the pull request's "Scale tables" item describes)
// instead of the per-tensor scalars. The producer copies each page's two
// scale rows into the stage next to its K/V bytes; a token's K scale
// multiplies its logit, its V scale multiplies its probability before the PV
// product (relative to the V scale of the split's first slot, so P stays in
// f16's normal range), and the sum l uses the unscaled probabilities.
//
// kTokenMajor: K and V pages are token-major rows of 128 bytes reached
// through strided tensor maps (the flash / NHD family of layouts). Each page
// lands in shared memory as [bs][128] with 128-byte swizzle (16-byte chunk c
// of row t at c ^ (t & 7)); QK^T reads K rows with ldmatrix in natural token
// order, PV reads V with ldmatrix.trans, whose b16 transpose hands each lane
// 2 tokens x 2 dims per register, split into an even-dim and an odd-dim
// fragment row by one byte permute. Output row gid of m-tile mt is then dim
// 16mt + 2gid and row gid + 8 is dim 16mt + 2gid + 1.
//
// kCluster: the build launched with clusters of nsplit CTAs along x (the
// splits of one unit, 2..kMaxClusterSplits, p.cluster_merge = 1); the splits
// merge through distributed shared memory (cluster_merge_rows) instead of
// fp32 partials and the merge kernel. That build reads the flag at run time:
// with the branches folded at compile time it ran 1-3 % slower on GB300
// (608 CTAs in clusters of 8: 20.6 against 20.0 us). The other builds fold
// the flag to false and compile exactly as without clusters.
template <bool kSlotScales, bool kTokenMajor, int kMinCtasPerSm, bool kPaired, bool kCluster>
__global__ void __launch_bounds__(kThreads, kMinCtasPerSm)
    pda_split_decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(128) uint8_t smem[];
  // A merge kernel launched as this grid's programmatic dependent may start
  // its launch now; it waits for this grid's results before reading them.
  grid_dependents_launch();
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bs = p.block_size;
  const int H = p.num_heads;
  const int g = p.gqa;

  const bool cluster = kCluster && p.cluster_merge != 0;
  if (!kSlotScales && !kTokenMajor && p.page_gather && threadIdx.x == kConsumerWarps * 32) {
    // the producer's descriptors, fetched while the table loads below run
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }

  int L = __ldg(p.seq_lens + s);
  L = max(0, min(L, p.max_blocks * bs));
  const int pages = (L + bs - 1) / bs;
  int pg_first, pg_end;
  split_range(pages, p.nsplit, split, pg_first, pg_end);

  if (pg_first >= pg_end) {
    // No tokens for this split. With one split the row is all-zero output;
    // with several, the merge skips empty splits by the same rule. In a
    // cluster the CTA runs on with no pages: it still merges its share of
    // rows, and every thread takes part in both cluster barriers (its own
    // partial is never read).
    if (p.nsplit == 1) {
      for (int i = threadIdx.x; i < g * kHeadDim; i += blockDim.x) {
        const int h = kvh * g + i / kHeadDim;
        store_out(p.out, ((size_t)s * H + h) * kHeadDim + (i % kHeadDim), 0.f, p.out_fp8, p.out_scale);
      }
    }
    if (!cluster) return;
    pg_end = pg_first;
  }

  const int n_pages = pg_end - pg_first;
  // The producer's first 32 block-table entries: the load overlaps the
  // barrier setup below.
  const int32_t* row = p.block_tables + (size_t)s * p.max_blocks + pg_first;
  int my_block = (warp == kConsumerWarps && lane < n_pages) ? __ldg(row + lane) : 0;
  const int NS = p.num_stages;
  const int PPS = p.pages_per_stage;
  // Ring base aligned to 1024 bytes (the 128-byte swizzle repeats every 1 KiB).
  uint8_t* ring = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + (size_t)NS * p.stage_bytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * NS);
  const uint32_t ring_u32 = smem_u32(ring);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * NS;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      // slot scales by cp.async: one more arrival per producer lane (its
      // scale copies)
      mbar_init(full0 + 8u * i, (kSlotScales && p.scale_rows == kScaleRowsPieces) ? 33u : 1u);
      mbar_init(empty0 + 8u * i, kConsumerWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const int n_fills = (n_pages + PPS - 1) / PPS;
  const uint32_t page_bytes = (uint32_t)(kHeadDim * bs);

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const size_t head_stride = (size_t)page_bytes;
    const size_t block_stride = (size_t)p.num_kv_heads * page_bytes;
    int fill = 0;
    bool ok = true;
    for (int base = 0; base < n_pages && ok; base += 32) {
      // the next chunk's entries, loaded one chunk ahead of their use
      // this chunk's entries are checked now that they are needed
      my_block = checked_block(my_block, p.block_limit);
      const int next_block = base + 32 + lane < n_pages ? __ldg(row + base + 32 + lane) : 0;
      const int chunk_pages = min(32, n_pages - base);
      for (int j = 0; j < chunk_pages; j += PPS, ++fill) {
        const int stage = fill % NS;
        const uint32_t round = (uint32_t)(fill / NS);
        int blk[kMaxPagesPerStage];
#pragma unroll
        for (int t = 0; t < kMaxPagesPerStage; ++t) blk[t] = __shfl_sync(0xffffffffu, my_block, (j + t) & 31);
        const int np = min(PPS, chunk_pages - j);
        const bool got = mbar_wait_bounded(empty0 + 8u * stage, (round & 1u) ^ 1u, abort_flag, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) {
            atomicOr(&g_status, kStatusEmptyWaitTimeout);
            *abort_flag = 1;
          }
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t sbase = ring_u32 + (uint32_t)stage * p.stage_bytes;
          const uint32_t bar = full0 + 8u * stage;
          const uint32_t row_bytes = (uint32_t)bs * 4u;
          uint32_t scale_tx = 0u;
          if (kSlotScales && p.scale_rows == kScaleRowsGather4) scale_tx = 2u * 4u * row_bytes;
          if (kSlotScales && p.scale_rows == kScaleRowsBulk) scale_tx = 2u * (uint32_t)np * row_bytes;
          const bool gather = !kSlotScales && !kTokenMajor && p.page_gather;
          mbar_arrive_expect_tx(bar, 2u * page_bytes * (uint32_t)(gather ? 4 : np) + scale_tx);
          if constexpr (kSlotScales) {
            // K rows at scale_off, V rows PPS rows further; row of page t:
            // b * Hk + kvh of its table
            const int Hk = p.num_kv_heads;
            const uint32_t sc = sbase + p.scale_off;
            if (p.scale_rows == kScaleRowsGather4) {
              const int4 r = stage_rows(blk, np, Hk, kvh);
              tma_gather4_rows(sc, &tm_k, r.x, r.y, r.z, r.w, bar);
              tma_gather4_rows(sc + 4u * row_bytes, &tm_v, r.x, r.y, r.z, r.w, bar);
            } else if (p.scale_rows == kScaleRowsBulk) {
#pragma unroll
              for (int t = 0; t < kMaxPagesPerStage; ++t) {
                if (t < np) {
                  const size_t off = ((size_t)blk[t] * Hk + kvh) * (size_t)bs;
                  bulk_g2s(sc + (uint32_t)t * row_bytes, p.k_scales + off, row_bytes, bar);
                  bulk_g2s(sc + (uint32_t)(PPS + t) * row_bytes, p.v_scales + off, row_bytes, bar);
                }
              }
            }
          }
          if constexpr (kTokenMajor) {
#pragma unroll
            for (int t = 0; t < kMaxPagesPerStage; ++t) {
              if (t < np) {
                // coordinates: 0 for the row bytes and the token dim, kvh and
                // the block id in the head and block dims
                const int c1 = p.tm_dim_head == 1 ? kvh : (p.tm_dim_block == 1 ? blk[t] : 0);
                const int c2 = p.tm_dim_head == 2 ? kvh : (p.tm_dim_block == 2 ? blk[t] : 0);
                const int c3 = p.tm_dim_head == 3 ? kvh : (p.tm_dim_block == 3 ? blk[t] : 0);
                tma_load_4d(sbase + (uint32_t)t * page_bytes, &tm_k, 0, c1, c2, c3, bar);
                tma_load_4d(sbase + (uint32_t)(PPS + t) * page_bytes, &tm_v, 0, c1, c2, c3, bar);
              }
            }
          } else if (!kSlotScales && p.v_swizzle) {
            // Swizzled V (32- to 128-token blocks: at most 2 pages a stage).
            // One branch per stage, not per page: the slot-scale instance's
            // busy producer lost 2.5 % of a 2.15 GB batch to a per-page one
            // (that instance never swizzles: its stages carry scale rows).
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (t < np) {
                const size_t off = (size_t)blk[t] * block_stride + (size_t)kvh * head_stride;
                bulk_g2s(sbase + (uint32_t)t * page_bytes, p.k_cache + off, page_bytes, bar);
                // coordinates: row bytes, dim, kv head, block
                tma_load_4d(sbase + (uint32_t)(PPS + t) * page_bytes, &tm_v, 0, 0, kvh, blk[t], bar);
              }
            }
          } else if (gather) {
            // 16-token pages: two copies a stage instead of eight (GB300,
            // 64 x 1024 tokens in one wave: 27.38 against 27.76 us per call)
            const int4 r = stage_rows(blk, np, p.num_kv_heads, kvh);
            tma_gather4_rows(sbase, &tm_k, r.x, r.y, r.z, r.w, bar);
            tma_gather4_rows(sbase + (uint32_t)PPS * page_bytes, &tm_v, r.x, r.y, r.z, r.w, bar);
          } else {
#pragma unroll
            for (int t = 0; t < kMaxPagesPerStage; ++t) {
              if (t < np) {
                const size_t off = (size_t)blk[t] * block_stride + (size_t)kvh * head_stride;
                bulk_g2s(sbase + (uint32_t)t * page_bytes, p.k_cache + off, page_bytes, bar);
                bulk_g2s(sbase + (uint32_t)(PPS + t) * page_bytes, p.v_cache + off, page_bytes, bar);
              }
            }
          }
        }
        if (kSlotScales && p.scale_rows == kScaleRowsPieces) {
          // The stage's K and V scale rows (np pages x bs floats each) as
          // 16-byte cp.async pieces spread over the warp: tiny rows would
          // cost a bulk-copy operation each. Every lane then arrives once on
          // the full barrier when its pieces have landed.
          const int per_row = bs / 4;
          const int per_table = np * per_row;
          for (int c0 = 0; c0 < 2 * per_table; c0 += 32) {  // warp-uniform trip count
            const int c = min(c0 + lane, 2 * per_table - 1);
            const int table = c / per_table;
            const int t = (c % per_table) / per_row;
            const int piece = c % per_row;
            const int b = __shfl_sync(0xffffffffu, my_block, (j + t) & 31);
            if (c0 + lane < 2 * per_table) {
              const float* src =
                  (table ? p.v_scales : p.k_scales) + ((size_t)b * p.num_kv_heads + kvh) * (size_t)bs + 4 * piece;
              cp_async_16(ring_u32 + (uint32_t)stage * p.stage_bytes + p.scale_off +
                              (uint32_t)((table * PPS + t) * bs * 4 + piece * 16),
                          src);
            }
          }
          cp_async_arrive_noinc(full0 + 8u * stage);
        }
        __syncwarp();
      }
      my_block = next_block;
    }
    // Drain: never leave the CTA with copies still landing in its smem.
    const int issued = fill;
    for (int f = max(0, issued - NS); f < issued; ++f) {
      const int stage = f % NS;
      if (!mbar_wait_bounded(full0 + 8u * stage, (uint32_t)(f / NS) & 1u, nullptr, kWaitLimitNs)) {
        if (lane == 0) atomicOr(&g_status, kStatusDrainTimeout);
        break;
      }
    }
    if (cluster) {
      // the producer warp's arrivals at the consumers' two cluster barriers
      cluster_sync();
      cluster_sync();
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  TileWorker<kSlotScales, kTokenMajor, kPaired, (kMinCtasPerSm < 4)> w;
  w.setup(lane, bs, p.v_shuffled, p.v_swizzle);
  {
    const int qh = w.q_head();
    const bool live = qh < g;
    w.load_q_global(p.q + ((size_t)s * H + (size_t)kvh * g + (live ? qh : 0)) * kHeadDim, live,
                    p.logit_scale_log2);
  }
  w.reset();

  const int tiles_per_page = bs / 16;
  const uint32_t v_sub = p.v_shuffled ? (uint32_t)(kHeadDim * 16) : 16u;
  // Slot-scale variant: V scales enter P relative to vref (the split's first
  // slot), and vref multiplies the result back at the end.
  float vref = 1.f, vinv = 1.f;

  for (int fill = 0; fill < n_fills; ++fill) {
    const int stage = fill % NS;
    const uint32_t round = (uint32_t)(fill / NS);
    const bool got = mbar_wait_bounded(full0 + 8u * stage, round & 1u, abort_flag, kWaitLimitNs);
    if (!__all_sync(0xffffffffu, got)) {
      if (lane == 0) {
        atomicOr(&g_status, kStatusFullWaitTimeout);
        *abort_flag = 1;
      }
      break;
    }
    const int fill_first_page = pg_first + fill * PPS;
    const int np = min(PPS, pg_end - fill_first_page);
    const int n_tiles = np * tiles_per_page;
    const uint32_t sbase = ring_u32 + (uint32_t)stage * p.stage_bytes;
    // slot scales of the stage: K rows of its pages, then V rows
    const float* srow = reinterpret_cast<const float*>(ring + stage * p.stage_bytes + p.scale_off);
    if constexpr (kSlotScales) {
      if (fill == 0) {
        const float v0 = srow[PPS * bs];
        if (isfinite(v0) && v0 != 0.f) {
          vref = v0;
          vinv = 1.f / v0;
        }
      }
    }

    for (int tile = warp; tile < n_tiles; tile += kConsumerWarps) {
      const int pg = tile / tiles_per_page;
      const int sub = tile % tiles_per_page;
      const int tok0 = (fill_first_page + pg) * bs + sub * 16;
      if (tok0 >= L) continue;
      const uint32_t kbase = kTokenMajor ? sbase + (uint32_t)pg * page_bytes + (uint32_t)sub * 2048u
                                         : sbase + (uint32_t)pg * page_bytes + (uint32_t)(sub * 256);
      const uint32_t vbase = kTokenMajor ? sbase + (uint32_t)(PPS + pg) * page_bytes + (uint32_t)sub * 2048u
                                         : sbase + (uint32_t)(PPS + pg) * page_bytes + ((uint32_t)sub ^ w.v_xor) * v_sub;
      w.tile(kbase, vbase, bs, L - tok0, srow + pg * bs + sub * 16, srow + (PPS + pg) * bs + sub * 16, vinv);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8u * stage);
  }

  // ------------------------------------------------ merge the consumer warps
  // All consumer warps are past their last ring read once they pass this
  // barrier; the abort decision is the same for all of them.
  if (named_barrier_or(1, kConsumerThreads, *abort_flag)) {
    if (cluster) {
      // still at both cluster barriers (the merged rows are undefined then)
      cluster_sync();
      cluster_sync();
    }
    return;
  }

  using Worker = decltype(w);
  float* mo = reinterpret_cast<float*>(smem);                       // [w][row][kMergeStride]
  float* mml = mo + kConsumerWarps * kMaxGqa * kMergeStride;        // [w][head][2]
  w.template store_merge<kMergeStride>(mo, mml, warp);
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
  reduce_store<kSlotScales, kMergeStride, Worker::kMergeRows, true>(
      p, mo, mml, threadIdx.x, s, kvh, split, vref,
      cluster ? reinterpret_cast<float*>(smem + kClusterPartOff) : nullptr);
  if (cluster) {
    cluster_sync();
    cluster_merge_rows<kSlotScales>(p, smem_u32(smem + kClusterPartOff), s, kvh, split, L, warp, lane);
    cluster_sync();
  }
}

// --------------------------------------------------------------------------
// Persistent variant (per-tensor scales; page-major K and V in either V page
// order, or token-major pages through tensor maps): the grid is the resident
// CTA slots, and each CTA works through a
// queue of work units. Its producer warp takes the next unit from an atomic
// ticket counter as soon as the previous unit's pages are issued, so the
// ring keeps streaming across unit boundaries instead of filling and
// draining once per unit, and free CTAs pick up work dynamically. Each stage
// has a small side entry with a header naming its unit; for the unit's first
// stage it also holds the unit's query rows (copied with its pages). The
// consumer warps finish a unit on its last stage: they merge their O rows in
// that stage's page memory (and their (m, l) in its side entry) and only
// then release it to the producer.
//
// Shared memory: NS stages of stage_bytes (K pages, then V pages; a multiple
// of 1 KiB and at least the merge rows, so swizzled tensor-map pages stay
// aligned), then NS side entries of kAuxBytes, then the barriers.
//
// Unit u is (s, kvh, split) = (u / (Hk nsplit), (u / nsplit) % Hk, u % nsplit),
// the order of the per-unit grid. CTA b starts with unit b; its later
// tickets are gridDim.x + the counter's previous value, taken when the
// producer reaches the last stage of its current unit (so a CTA claims work
// only shortly before it can start it), and ticket gridDim.x + i is unit
// unit_order[i] when an order is given: longest units first, so that the
// last units to start are the short ones. That order comes from a kernel
// launched just before this one as its programmatic dependency; only the
// second ticket waits for it. queue[0] is the counter and queue[1] counts
// finished CTAs: the last CTA to finish zeroes both, so every launch finds
// them at zero (the workspace starts zeroed).
struct StageHeader {
  int s, kvh, split, L;
  int first_page;  // page index (in the sequence) of the stage's first page
  int np;          // pages in the stage (0: a zero-length sequence)
  int flags;       // kHdrFirst / kHdrLast / kHdrEnd
  int slot;        // tail piece: its tail_rows slot; -1 for a whole unit
};
constexpr int kHdrFirst = 1;
constexpr int kHdrLast = 2;
constexpr int kHdrEnd = 4;
constexpr uint32_t kAuxQ = 0;                                     // query rows, g x 256 B
constexpr uint32_t kAuxMl = kMaxGqa * kHeadDim * 2;              // merge (m, l) [w][head][2]
constexpr uint32_t kAuxHdr = kAuxMl + kConsumerWarps * kMaxGqa * 2 * 4;  // StageHeader
constexpr uint32_t kAuxBytes = kAuxHdr + sizeof(StageHeader);
// Side entries of the per-slot-scale instance: 128-byte multiples, so that
// the scale rows a TMA gather lands in the query-row area (at p.scale_off,
// past the group's query rows) start on a 128-byte boundary.
constexpr uint32_t kAuxBytesSlot = (kAuxBytes + 127u) & ~127u;
template <bool kSlotScales>
__host__ __device__ constexpr uint32_t aux_bytes() { return kSlotScales ? kAuxBytesSlot : kAuxBytes; }
// Merge rows in a persistent stage: 8 rows per warp at the unpadded stride
// fill 16 KiB exactly; paired instances store 4 rows per warp at the padded
// stride (bank-conflict free).
template <bool kPaired>
__host__ __device__ constexpr int persist_merge_stride() { return kPaired ? kMergeStride : kHeadDim; }
constexpr uint32_t kPersistMergeBytes = kConsumerWarps * kMaxGqa * kHeadDim * 4;
static_assert(kConsumerWarps * (kMaxGqa / 2) * kMergeStride * 4 <= kPersistMergeBytes, "paired rows fit the stage");
static_assert(kAuxBytes % 16 == 0, "side entries keep 16-byte alignment");

// Bounded barrier of the consumer warps on an mbarrier (count kConsumerWarps):
// false (with the status bit and the abort flag raised) after the wait
// limit, or when the CTA is aborting.
__device__ __forceinline__ bool consumer_sync(uint32_t bar, uint32_t& phase, int lane, volatile int* abort_flag) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar, phase & 1u, abort_flag, kWaitLimitNs));
  ++phase;
  if (!ok && lane == 0) {
    atomicOr(&g_status, kStatusMergeWaitTimeout);
    *abort_flag = 1;
  }
  return ok;
}

// Tail pieces (persistent kernel). tail_piece_rows: consumer thread tid
// folds dim tid of every head of the group over the consumer warps, as
// reduce_store does, and leaves the piece's (O, m, l) in its tail_rows slot:
// O rows [kMaxGqa][kHeadDim], then (m, l) pairs.
template <int kStride, int kRows>
__device__ __forceinline__ void tail_piece_rows(const DecodeParams& p, const float* mo, const float* mml, int tid,
                                                int slot, float vref) {
  float* rows = p.tail_rows + (size_t)slot * kTailRowFloats;
  const int d = tid;
  for (int hh = 0; hh < p.gqa; ++hh) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mml[(w * kMaxGqa + hh) * 2]);
    float acc = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = mml[(w * kMaxGqa + hh) * 2];
        const float f = fast_exp2(mw - M);
        acc += f * mo[(w * kRows + hh) * kStride + d];
        den += f * mml[(w * kMaxGqa + hh) * 2 + 1];
      }
    }
    // slot scales: the piece's own V reference goes into its O rows (the
    // tail merge then scales by 1)
    __stcg(rows + hh * kHeadDim + d, acc * vref);
    if (d == 0) {
      __stcg(rows + kMaxGqa * kHeadDim + hh * 2 + 0, M);
      __stcg(rows + kMaxGqa * kHeadDim + hh * 2 + 1, den);
    }
  }
}

// kSlotScales: per-slot scale tables (page-major pages only). Each stage's
// K and V scale rows land in its side entry at p.scale_off, by one TMA
// gather per table (p.scale_rows == kScaleRowsGather4) or one bulk copy per
// row; a unit's (or piece's) V reference is the first V scale of its first
// stage, as in the per-unit kernel.
template <bool kSlotScales, bool kTokenMajor, int kMinCtasPerSm, bool kPaired>
__global__ void __launch_bounds__(kThreads, kMinCtasPerSm)
    pda_persistent_decode_kernel(const DecodeParams p, unsigned* queue, int num_units,
                                 const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(128) uint8_t smem[];
  // A merge kernel launched as this grid's programmatic dependent may start
  // its launch now (with the order kernel: once this CTA has waited for
  // it, so that a dependent may read what the order kernel wrote); it waits
  // for this grid's results before reading them.
  if (p.unit_order == nullptr) grid_dependents_launch();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bs = p.block_size;
  const int g = p.gqa;
  const int NS = p.num_stages;
  const int PPS = p.pages_per_stage;

  static_assert(!(kSlotScales && kTokenMajor), "per-slot scales come with page-major pages");
  constexpr uint32_t kAux = aux_bytes<kSlotScales>();
  uint8_t* ring = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
  uint8_t* aux = ring + (size_t)NS * p.stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(aux + (size_t)NS * kAux);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * NS + 1);
  const uint32_t ring_u32 = smem_u32(ring);
  const uint32_t aux_u32 = smem_u32(aux);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * NS;
  const uint32_t cons_bar = full0 + 16u * NS;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + 8u * i, 1);
      mbar_init(empty0 + 8u * i, kConsumerWarps);
    }
    mbar_init(cons_bar, kConsumerWarps);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const uint32_t page_bytes = (uint32_t)(kHeadDim * bs);

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const size_t head_stride = (size_t)page_bytes;
    const size_t block_stride = (size_t)p.num_kv_heads * page_bytes;
    const int per_seq = p.num_kv_heads * p.nsplit;
    int fill = 0;
    bool ok = true;
    unsigned t = blockIdx.x;  // ticket
    unsigned unit = t;
    // Tickets past the whole units (tail pieces) exist once the order
    // kernel has counted them.
    unsigned n_tickets = (unsigned)num_units;
    int piece_a = 0, piece_b = 0, slot = -1;
    bool order_ready = false;
    while (ok && t < n_tickets) {
      const int s = (int)(unit / (unsigned)per_seq);
      const int kvh = (int)((unit / (unsigned)p.nsplit) % (unsigned)p.num_kv_heads);
      const int split = (int)(unit % (unsigned)p.nsplit);
      int L = __ldg(p.seq_lens + s);
      L = max(0, min(L, p.max_blocks * bs));
      const int pages = (L + bs - 1) / bs;
      int pg_first, pg_end;
      split_range(pages, p.nsplit, split, pg_first, pg_end);
      if (slot >= 0) {
        // a tail piece: pages [piece_a, piece_b) of the split (never empty)
        pg_end = pg_first + piece_b;
        pg_first += piece_a;
      }
      bool skip = false;
      if (pg_first >= pg_end) {
        // An empty split writes nothing (the merge kernel skips it); a
        // zero-length sequence gets one header-only stage so that the
        // consumers store its zero output.
        if (p.nsplit > 1) skip = true;
        pg_first = pg_end = 0;
      }
      unsigned t_next = 0;
      bool fetched = false;
      const int n_pages = pg_end - pg_first;
      const int n_st = skip ? 0 : (n_pages > 0 ? (n_pages + PPS - 1) / PPS : 1);
      const int32_t* row = p.block_tables + (size_t)s * p.max_blocks + pg_first;
      int my_block = 0, next_block = 0;
      for (int k = 0; k < n_st; ++k, ++fill) {
        const int j = k * PPS;  // page offset in the unit; stages never straddle a 32-page chunk
        if ((j & 31) == 0) {
          // this chunk's entries (loaded one chunk ahead, except the first)
          // and the next chunk's
          my_block = checked_block(j == 0 ? ((lane < n_pages) ? __ldg(row + lane) : 0) : next_block, p.block_limit);
          next_block = (j + 32 + lane < n_pages) ? __ldg(row + j + 32 + lane) : 0;
        }
        int blk[kMaxPagesPerStage];
#pragma unroll
        for (int u = 0; u < kMaxPagesPerStage; ++u) blk[u] = __shfl_sync(0xffffffffu, my_block, (j + u) & 31);
        const int np = max(0, min(PPS, n_pages - j));
        if (k == n_st - 1) {
          // next ticket: its latency overlaps the wait for this stage's slot
          if (lane == 0) t_next = gridDim.x + atomicAdd(queue, 1u);
          fetched = true;
        }
        const int stage = fill % NS;
        const uint32_t round = (uint32_t)(fill / NS);
        const bool got = mbar_wait_bounded(empty0 + 8u * stage, (round & 1u) ^ 1u, abort_flag, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) {
            atomicOr(&g_status, kStatusEmptyWaitTimeout);
            *abort_flag = 1;
          }
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t sbase = ring_u32 + (uint32_t)stage * p.stage_bytes;
          const uint32_t bar = full0 + 8u * stage;
          StageHeader* hd = reinterpret_cast<StageHeader*>(aux + (size_t)stage * kAux + kAuxHdr);
          hd->s = s;
          hd->kvh = kvh;
          hd->split = split;
          hd->L = L;
          hd->first_page = pg_first + j;
          hd->np = np;
          hd->flags = (k == 0 ? kHdrFirst : 0) | (k == n_st - 1 ? kHdrLast : 0);
          hd->slot = slot;
          const bool with_q = (k == 0) && (np > 0);
          const uint32_t q_bytes = with_q ? (uint32_t)g * kHeadDim * 2u : 0u;
          // a four-row gather always lands 4 pages (or scale rows) per table
          const uint32_t row_bytes = (uint32_t)bs * 4u;
          uint32_t scale_tx = 0u;
          if (kSlotScales && np > 0)
            scale_tx = 2u * row_bytes * (uint32_t)(p.scale_rows == kScaleRowsGather4 ? 4 : np);
          const uint32_t bytes =
              2u * page_bytes * (uint32_t)(p.page_gather && np > 0 ? 4 : np) + q_bytes + scale_tx;
          if (bytes == 0) {
            mbar_arrive(bar);  // release-orders the header for the consumers
          } else {
            mbar_arrive_expect_tx(bar, bytes);
            if (with_q)
              bulk_g2s(aux_u32 + (uint32_t)stage * kAux + kAuxQ,
                       p.q + ((size_t)s * p.num_heads + (size_t)kvh * g) * kHeadDim, q_bytes, bar);
            if constexpr (kSlotScales) {
              // the stage's K scale rows, then its V rows (PPS rows further)
              const uint32_t sc = aux_u32 + (uint32_t)stage * kAux + p.scale_off;
              if (p.scale_rows == kScaleRowsGather4) {
                if (np > 0) {
                  const int4 r = stage_rows(blk, np, p.num_kv_heads, kvh);
                  tma_gather4_rows(sc, &tm_k, r.x, r.y, r.z, r.w, bar);
                  tma_gather4_rows(sc + 4u * row_bytes, &tm_v, r.x, r.y, r.z, r.w, bar);
                }
              } else {
#pragma unroll
                for (int u = 0; u < kMaxPagesPerStage; ++u) {
                  if (u < np) {
                    const size_t off = ((size_t)blk[u] * p.num_kv_heads + kvh) * (size_t)bs;
                    bulk_g2s(sc + (uint32_t)u * row_bytes, p.k_scales + off, row_bytes, bar);
                    bulk_g2s(sc + (uint32_t)(PPS + u) * row_bytes, p.v_scales + off, row_bytes, bar);
                  }
                }
              }
            }
            if constexpr (kTokenMajor) {
#pragma unroll
              for (int u = 0; u < kMaxPagesPerStage; ++u) {
                if (u < np) {
                  // coordinates: 0 for the row bytes and the token dim, kvh
                  // and the block id in the head and block dims
                  const int c1 = p.tm_dim_head == 1 ? kvh : (p.tm_dim_block == 1 ? blk[u] : 0);
                  const int c2 = p.tm_dim_head == 2 ? kvh : (p.tm_dim_block == 2 ? blk[u] : 0);
                  const int c3 = p.tm_dim_head == 3 ? kvh : (p.tm_dim_block == 3 ? blk[u] : 0);
                  tma_load_4d(sbase + (uint32_t)u * page_bytes, &tm_k, 0, c1, c2, c3, bar);
                  tma_load_4d(sbase + (uint32_t)(PPS + u) * page_bytes, &tm_v, 0, c1, c2, c3, bar);
                }
              }
            } else if (p.v_swizzle) {
              // swizzled V (32- to 128-token blocks: at most 2 pages a stage);
              // one branch per stage, not per page
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                if (u < np) {
                  const size_t off = (size_t)blk[u] * block_stride + (size_t)kvh * head_stride;
                  bulk_g2s(sbase + (uint32_t)u * page_bytes, p.k_cache + off, page_bytes, bar);
                  // coordinates: row bytes, dim, kv head, block
                  tma_load_4d(sbase + (uint32_t)(PPS + u) * page_bytes, &tm_v, 0, 0, kvh, blk[u], bar);
                }
              }
            } else if (p.page_gather) {
              // 16-token pages: two copies a stage instead of eight (GB300,
              // us per call: 256 x 4096 tokens 309.1 against 311.4, 256 x
              // 1-4000 tokens 155.6 against 158.3)
              if (np > 0) {
                const int4 r = stage_rows(blk, np, p.num_kv_heads, kvh);
                tma_gather4_rows(sbase, &tm_k, r.x, r.y, r.z, r.w, bar);
                tma_gather4_rows(sbase + (uint32_t)PPS * page_bytes, &tm_v, r.x, r.y, r.z, r.w, bar);
              }
            } else {
#pragma unroll
              for (int u = 0; u < kMaxPagesPerStage; ++u) {
                if (u < np) {
                  const size_t off = (size_t)blk[u] * block_stride + (size_t)kvh * head_stride;
                  bulk_g2s(sbase + (uint32_t)u * page_bytes, p.k_cache + off, page_bytes, bar);
                  bulk_g2s(sbase + (uint32_t)(PPS + u) * page_bytes, p.v_cache + off, page_bytes, bar);
                }
              }
            }
          }
        }
        __syncwarp();
      }
      if (!ok) break;
      if (!fetched && lane == 0) t_next = gridDim.x + atomicAdd(queue, 1u);
      t = __shfl_sync(0xffffffffu, t_next, 0);
      unit = t;
      piece_a = piece_b = 0;
      slot = -1;
      if (p.unit_order != nullptr) {
        if (!order_ready) {
          grid_dependency_wait();  // the order kernel has finished and its writes are visible
          grid_dependents_launch();
          order_ready = true;
          if (p.num_tickets != nullptr) {
            unsigned n = 0;
            if (lane == 0) n = (unsigned)__ldcg(p.num_tickets);
            n_tickets = __shfl_sync(0xffffffffu, n, 0);
          }
        }
        if (t >= p.tail_first && t < n_tickets) {
          int4 e = make_int4(0, 0, 0, -1);
          if (lane == 0) e = __ldcg(p.piece_table + (t - p.tail_first));
          unit = (unsigned)__shfl_sync(0xffffffffu, e.x, 0);
          piece_a = __shfl_sync(0xffffffffu, e.y, 0);
          piece_b = __shfl_sync(0xffffffffu, e.z, 0);
          slot = __shfl_sync(0xffffffffu, e.w, 0);
        } else if (t < (unsigned)num_units) {
          unsigned u = 0;
          if (lane == 0) u = (unsigned)__ldcg(p.unit_order + (t - gridDim.x));
          unit = __shfl_sync(0xffffffffu, u, 0);
        }
      }
    }
    if (ok) {
      // End marker: a header-only stage that stops the consumers.
      const int stage = fill % NS;
      const uint32_t round = (uint32_t)(fill / NS);
      const bool got = mbar_wait_bounded(empty0 + 8u * stage, (round & 1u) ^ 1u, abort_flag, kWaitLimitNs);
      if (__all_sync(0xffffffffu, got)) {
        if (lane == 0) {
          StageHeader* hd = reinterpret_cast<StageHeader*>(aux + (size_t)stage * kAux + kAuxHdr);
          hd->flags = kHdrEnd;
          mbar_arrive(full0 + 8u * stage);
        }
        ++fill;
      } else if (lane == 0) {
        atomicOr(&g_status, kStatusEmptyWaitTimeout);
        *abort_flag = 1;
      }
      __syncwarp();
    }
    // Drain: never leave the CTA with copies still landing in its smem.
    for (int f = max(0, fill - NS); f < fill; ++f) {
      if (!mbar_wait_bounded(full0 + 8u * (f % NS), (uint32_t)(f / NS) & 1u, nullptr, kWaitLimitNs)) {
        if (lane == 0) atomicOr(&g_status, kStatusDrainTimeout);
        break;
      }
    }
    // Queue bookkeeping: this CTA takes no more tickets.
    if (lane == 0) {
      __threadfence();
      if (atomicAdd(queue + 1, 1u) == gridDim.x - 1) {
        atomicExch(queue, 0u);
        atomicExch(queue + 1, 0u);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  TileWorker<kSlotScales, kTokenMajor, kPaired, true> w;
  w.setup(lane, bs, p.v_shuffled, p.v_swizzle);
  w.reset();
  const int tiles_per_page = bs / 16;
  const uint32_t v_sub = p.v_shuffled ? (uint32_t)(kHeadDim * 16) : 16u;
  uint32_t cons_phase = 0;
  // Slot-scale variant: V scales enter P relative to vref (the first slot
  // of the unit or piece), and vref multiplies the result back at the end.
  float vref = 1.f, vinv = 1.f;

  for (int fill = 0;; ++fill) {
    const int stage = fill % NS;
    const uint32_t round = (uint32_t)(fill / NS);
    const bool got = mbar_wait_bounded(full0 + 8u * stage, round & 1u, abort_flag, kWaitLimitNs);
    if (!__all_sync(0xffffffffu, got)) {
      if (lane == 0) {
        atomicOr(&g_status, kStatusFullWaitTimeout);
        *abort_flag = 1;
      }
      break;
    }
    const StageHeader hd = *reinterpret_cast<const StageHeader*>(aux + (size_t)stage * kAux + kAuxHdr);
    if (hd.flags & kHdrEnd) break;
    const uint32_t sbase = ring_u32 + (uint32_t)stage * p.stage_bytes;
    // slot scales of the stage: K rows of its pages, then V rows
    const float* srow = kSlotScales ? reinterpret_cast<const float*>(aux + (size_t)stage * kAux + p.scale_off)
                                    : nullptr;
    if (hd.flags & kHdrFirst) {
      w.reset();
      if constexpr (kSlotScales) {
        vref = 1.f;
        vinv = 1.f;
        if (hd.np > 0) {
          const float v0 = srow[PPS * bs];
          if (isfinite(v0) && v0 != 0.f) {
            vref = v0;
            vinv = 1.f / v0;
          }
        }
      }
      if (hd.np > 0) {
        const int qh = w.q_head();
        const bool live = qh < g;
        w.load_q_shared(aux_u32 + (uint32_t)stage * kAux + kAuxQ + (uint32_t)(live ? qh : 0) * (kHeadDim * 2),
                        live, p.logit_scale_log2);
      }
    }
    const int n_tiles = hd.np * tiles_per_page;
    for (int tile = warp; tile < n_tiles; tile += kConsumerWarps) {
      const int pg = tile / tiles_per_page;
      const int sub = tile % tiles_per_page;
      const int tok0 = (hd.first_page + pg) * bs + sub * 16;
      if (tok0 >= hd.L) continue;
      const uint32_t kbase = kTokenMajor ? sbase + (uint32_t)pg * page_bytes + (uint32_t)sub * 2048u
                                         : sbase + (uint32_t)pg * page_bytes + (uint32_t)(sub * 256);
      const uint32_t vbase = kTokenMajor ? sbase + (uint32_t)(PPS + pg) * page_bytes + (uint32_t)sub * 2048u
                                         : sbase + (uint32_t)(PPS + pg) * page_bytes + ((uint32_t)sub ^ w.v_xor) * v_sub;
      if constexpr (kSlotScales)
        w.tile(kbase, vbase, bs, hd.L - tok0, srow + pg * bs + sub * 16, srow + (PPS + pg) * bs + sub * 16, vinv);
      else
        w.tile(kbase, vbase, bs, hd.L - tok0, nullptr, nullptr, 1.f);
    }
    if (hd.flags & kHdrLast) {
      // Every consumer warp is done with this stage's pages: its memory
      // becomes the merge area until the stage is released below.
      if (!consumer_sync(cons_bar, cons_phase, lane, abort_flag)) break;
      float* mo = reinterpret_cast<float*>(ring + (size_t)stage * p.stage_bytes);
      float* mml = reinterpret_cast<float*>(aux + (size_t)stage * kAux + kAuxMl);
      constexpr int kStride = persist_merge_stride<kPaired>();
      w.template store_merge<kStride>(mo, mml, warp);
      if (!consumer_sync(cons_bar, cons_phase, lane, abort_flag)) break;
      if (hd.slot < 0) {
        reduce_store<kSlotScales, kStride, decltype(w)::kMergeRows>(p, mo, mml, threadIdx.x, hd.s, hd.kvh, hd.split,
                                                                     vref);
      } else {
        // a tail piece: its (O, m, l) rows for the tail merge kernel
        tail_piece_rows<kStride, decltype(w)::kMergeRows>(p, mo, mml, threadIdx.x, hd.slot, kSlotScales ? vref : 1.f);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8u * stage);
  }
  // A consumer that leaves on a failed wait raises the abort flag; the
  // others then fail their next bounded wait and leave too.
}

// Longest-first order of the work units the persistent kernel hands out
// after each CTA's first one (units first .. num_units-1): a counting sort of
// the units by the number of pages of their split, in buckets of equal page
// count (of equal page-count ranges when a split can hold more than
// kOrderBuckets - 1 pages). Units in one bucket keep no particular order;
// the order only decides which CTA computes a unit and when, never the
// unit's result. One CTA; it lets the persistent kernel launch at once.
constexpr int kOrderThreads = 1024;
constexpr int kOrderBuckets = 4096;
// Largest batch (in work units) whose units the persistent kernel takes in
// longest-first order: the order kernel is one CTA, so its time grows with
// the units, and it must finish while the CTAs work on their first units.
constexpr int kMaxOrderedUnits = 16384;

struct OrderParams {
  const int32_t* seq_lens;
  int* order;           // [num_units - first]
  int first;            // units below this are taken by block index
  int num_units;
  int num_kv_heads;
  int nsplit;
  int block_size;
  int max_blocks;
  int max_split_pages;  // ceil(max_blocks / nsplit): largest page count of a split
  // Tail pieces: the last tail_units units of the order (at most
  // kOrderThreads) of at least kMinCutPieces * min_piece_pages pages are cut
  // into pieces of at least min_piece_pages pages, at most max_pieces each
  // (tail_piece_count); piece_table lists the tickets ({unit, first page,
  // end page, slot}, slot -1 for a whole unit), tail_info[j] = {unit, first
  // slot, pieces}, *num_tickets = units before the tail + the entries.
  int tail_units = 0;
  int max_pieces = 1;
  int min_piece_pages = 1;
  int4* piece_table = nullptr;
  int4* tail_info = nullptr;
  int* num_tickets = nullptr;
};

// Tail pieces of a split of n pages, with K tail units on C CTAs and
// pieces of at least m pages (at most cap; splits under kMinCutPieces * m
// pages stay whole). When the tail fills a third of the CTAs or more, piece
// r holds about K / C of what is left of the split and the last piece the
// rest, so the pieces get smaller toward the end of the hand-out (tickets go
// out piece index by piece index, over all tail units) and the CTAs finish
// close together: GB300, 256 x 4096 tokens (K = 224 on 456 CTAs, pieces of
// 126, 64, 32, 17 and 17 pages) took 307.9 us per call against 310.5 us
// with 5 equal pieces, its CTAs ending within 7 us instead of 15 us. A
// smaller tail is cut into equal pieces.
// (Host and device: the planner and a host-side check use the same rules.)
__host__ __device__ inline bool tail_geometric(int K, int C) { return 3 * K >= C; }

// Most pieces a tail unit is cut into: kMaxTailPieces for shrinking pieces,
// else about two equal pieces per CTA.
__host__ __device__ inline int tail_piece_cap(int K, int C) {
  if (tail_geometric(K, C)) return kMaxTailPieces;
  const long long per = (2LL * C + K - 1) / K;
  return per < kMaxTailPieces ? (int)per : kMaxTailPieces;
}

// The next shrinking piece cut from the rem pages left when `cut` pieces are
// already cut: about K / C of them, at least m. The cut that reaches the
// cap takes at least half, so that the last piece (the rest) is never the
// larger of the two.
__host__ __device__ inline int tail_piece_size(int rem, int K, int C, int m, int cut, int cap) {
  int sz = (int)(((long long)K * rem + C / 2) / C);
  if (sz < m) sz = m;
  if (cut == cap - 2 && sz < rem - rem / 2) sz = rem - rem / 2;
  return sz;
}

__host__ __device__ inline int tail_piece_count(int n, int K, int C, int m, int cap) {
  if (n < kMinCutPieces * m) return 1;
  if (!tail_geometric(K, C)) return n / m < cap ? n / m : cap;
  int rem = n, P = 1;
  while (P < cap) {
    const int sz = tail_piece_size(rem, K, C, m, P - 1, cap);
    if (rem - sz < m) break;
    rem -= sz;
    ++P;
  }
  return P;
}

// Pages [a, b) of piece r of the P that tail_piece_count gave. Equal
// pieces differ by at most a page and are never empty (n >= P): split_range's
// rounding would leave the last pieces empty when n / P is small (11 pages in
// 5 pieces: 3, 3, 3, 2 and none), and an empty piece stores no rows.
__host__ __device__ inline void tail_piece_range(int n, int K, int C, int m, int P, int cap, int r, int& a, int& b) {
  if (!tail_geometric(K, C)) {
    a = (int)((long long)r * n / P);
    b = (int)((long long)(r + 1) * n / P);
    return;
  }
  int rem = n, sz = 0;
  for (int i = 0; i <= r; ++i) {
    sz = i == P - 1 ? rem : tail_piece_size(rem, K, C, m, i, cap);
    if (i < r) rem -= sz;
  }
  a = n - rem;
  b = a + sz;
}

// Exclusive prefix sum of v over the order kernel's block (kOrderThreads
// threads, 32 warps); *total receives the block's sum. Uses wsum[32].
__device__ __forceinline__ int order_block_scan(int v, int* wsum, int* total) {
  static_assert(kOrderThreads == 32 * 32, "one warp's lanes cover the warp sums");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += x;
  }
  __syncthreads();  // wsum's previous readers are done
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += x;
    }
    wsum[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  *total = wsum[31];
  return (warp > 0 ? wsum[warp - 1] : 0) + incl - v;
}

__device__ __forceinline__ int order_key(const OrderParams& p, int u) {
  const int s = u / (p.num_kv_heads * p.nsplit);
  const int split = u % p.nsplit;
  int L = __ldg(p.seq_lens + s);
  L = max(0, min(L, p.max_blocks * p.block_size));
  int first, end;
  split_range((L + p.block_size - 1) / p.block_size, p.nsplit, split, first, end);
  const int n = max(0, end - first);
  const int k = p.max_split_pages < kOrderBuckets
                    ? n
                    : (int)((long long)n * (kOrderBuckets - 1) / (long long)p.max_split_pages);
  return kOrderBuckets - 1 - min(k, kOrderBuckets - 1);  // longest first
}

__global__ void __launch_bounds__(kOrderThreads) pda_order_units_kernel(const OrderParams p) {
  grid_dependents_launch();
  __shared__ unsigned count[kOrderBuckets];
  __shared__ unsigned warp_sum[kOrderThreads / 32];
  const int tid = threadIdx.x;
  for (int i = tid; i < kOrderBuckets; i += kOrderThreads) count[i] = 0u;
  __syncthreads();
  for (int u = p.first + tid; u < p.num_units; u += kOrderThreads) atomicAdd(&count[order_key(p, u)], 1u);
  __syncthreads();
  // exclusive prefix sum over the buckets: thread t owns buckets 4t .. 4t+3
  constexpr int kPer = kOrderBuckets / kOrderThreads;
  unsigned own[kPer];
  unsigned sum = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    own[j] = count[kPer * tid + j];
    sum += own[j];
  }
  const int lane = tid & 31, warp = tid >> 5;
  unsigned incl = sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    unsigned w = warp_sum[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const unsigned v = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += v;
    }
    warp_sum[lane] = w - warp_sum[lane];  // exclusive over warps
  }
  __syncthreads();
  const int n_order = p.num_units - p.first;
  const int K = p.tail_units;
  // Tail pieces: the tail is the last K positions of the order. The bucket
  // where it starts (tb) holds units of equal page count; which of them are
  // in the tail must not depend on the scatter's atomic order (a pieced
  // unit's result differs in the last bits from the whole unit's), so the
  // tail takes a fixed set of that bucket's units (below).
  __shared__ int s_tb, s_tb_start, s_tb_count, s_tb_tail;
  unsigned base = warp_sum[warp] + incl - sum;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    count[kPer * tid + j] = base;
    const unsigned t0 = (unsigned)(n_order - K);
    if (K > 0 && own[j] > 0 && base <= t0 && t0 < base + own[j]) {
      s_tb = kPer * tid + j;
      s_tb_start = (int)base;
      s_tb_count = (int)own[j];
      s_tb_tail = (int)(base + own[j] - t0);
    }
    base += own[j];
  }
  __syncthreads();
  // The tail's units of bucket tb are placed first, at fixed positions, and
  // marked; every other unit is then scattered in index order, so the kv
  // heads of a sequence stay next to each other within their bucket and run
  // side by side (token-major caches interleave their pages in one block:
  // GB300, 256 x 4096 tokens through [NB, bs, Hk, 128] caches took 378 us
  // per call with every bucket in scrambled order, against 330 us).
  __shared__ unsigned tail_bit[kMaxOrderedUnits / 32];
  const bool tail = K > 0 && n_order <= kMaxOrderedUnits;  // the host never orders more units
  if (tail) {
    for (int i = tid; i < kMaxOrderedUnits / 32; i += kOrderThreads) tail_bit[i] = 0u;
    // Units are visited in a fixed scrambled order v -> first + (v A mod n),
    // A coprime with n: the tail takes bucket tb's last units in that order,
    // a set spread over the sequences (tb's units in plain index order would
    // be whole sequences, whose kv heads then run side by side: 1 % slower).
    __shared__ int s_mult;
    if (tid == 0) {
      int a = n_order > 1 ? (int)(2654435761u % (unsigned)n_order) : 1;
      for (;; ++a) {
        if (a >= n_order) a = 1;
        int x = a, y = n_order;
        while (y != 0) {
          const int r = x % y;
          x = y;
          y = r;
        }
        if (x == 1) break;
      }
      s_mult = a;
    }
    __syncthreads();
    const int mult = s_mult;
    const int tb = s_tb, tb_start = s_tb_start, tb_keep = s_tb_count - s_tb_tail;
    int running = 0;  // units of bucket tb in earlier chunks (scrambled order)
    for (int base_v = 0; base_v < n_order; base_v += kOrderThreads) {
      const int v = base_v + tid;
      const int i = v < n_order ? (int)(((long long)v * mult) % n_order) : -1;
      const bool in_tb = i >= 0 && order_key(p, p.first + i) == tb;
      const unsigned m = __ballot_sync(0xffffffffu, in_tb);
      if (lane == 0) warp_sum[warp] = (unsigned)__popc(m);
      __syncthreads();
      if (warp == 0) {
        const unsigned c = warp_sum[lane];
        unsigned w = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const unsigned v = __shfl_up_sync(0xffffffffu, w, d);
          if (lane >= d) w += v;
        }
        warp_sum[lane] = w - c;  // exclusive over warps
        if (lane == 31) s_tb_count = (int)w;  // this chunk's units of tb (s_tb_count no longer needed)
      }
      __syncthreads();
      const int rank = running + (int)(warp_sum[warp] + __popc(m & ((1u << lane) - 1u)));
      running += s_tb_count;
      if (in_tb && rank >= tb_keep) {
        // tb's units past tb_keep (in scrambled order) take the tail's start
        p.order[tb_start + rank] = p.first + i;
        atomicOr(&tail_bit[i >> 5], 1u << (i & 31));
      }
      __syncthreads();  // warp_sum and s_tb_count are reused by the next chunk
    }
  }
  for (int u = p.first + tid; u < p.num_units; u += kOrderThreads) {
    const int i = u - p.first;
    if (tail && ((tail_bit[i >> 5] >> (i & 31)) & 1u)) continue;
    p.order[atomicAdd(&count[order_key(p, u)], 1u)] = u;
  }
  if (K <= 0) return;

  // ---- tail pieces: unit j of the last tail_units in the order is cut into
  // tail_piece_count pieces; their rows slots sit side by side (tail_info[j]
  // tells the tail merge kernel where), and their tickets go out piece index
  // by piece index over the tail units, so the last tickets are the last
  // (smallest) pieces.
  __syncthreads();  // the order entries written above are visible to the block
  const int C = p.first;  // the persistent grid: one CTA per unit of the first round
  const int m = p.min_piece_pages;
  int u = 0, n = 0, P = 0;
  if (tid < K) {
    u = p.order[n_order - K + tid];
    const int sq = u / (p.num_kv_heads * p.nsplit);
    int L = __ldg(p.seq_lens + sq);
    L = max(0, min(L, p.max_blocks * p.block_size));
    int first, end;
    split_range((L + p.block_size - 1) / p.block_size, p.nsplit, u % p.nsplit, first, end);
    n = max(0, end - first);
    P = tail_piece_count(n, K, C, m, p.max_pieces);
  }
  __shared__ int scan_buf[32];
  int total = 0;  // rows slots in all (sized by the host: at most K * max_pieces)
  const int slot0 = order_block_scan(P, scan_buf, &total);
  if (tid < K) p.tail_info[tid] = make_int4(u, slot0, P, 0);
  int issued = 0;  // tickets of the earlier piece indices
  for (int r = 0; r < p.max_pieces; ++r) {
    const int f = P > r ? 1 : 0;
    int cnt = 0;
    const int rank = order_block_scan(f, scan_buf, &cnt);
    if (f) {
      int4 e = make_int4(u, 0, 0, -1);
      if (P > 1) {
        tail_piece_range(n, K, C, m, P, p.max_pieces, r, e.y, e.z);
        e.w = slot0 + r;
      }
      p.piece_table[issued + rank] = e;
    }
    issued += cnt;
    if (cnt == 0) break;  // block-uniform
  }
  if (tid == 0) *p.num_tickets = p.num_units - K + issued;
}

// Log-sum-exp merge of the per-split partials:
//   M = max_i m_i,  out = v_scale * sum_i 2^(m_i - M) O_i / sum_i 2^(m_i - M) l_i
// with a sink logit, if any, added to the denominator (finish()).
// Splits with no pages were never written and are skipped by the same page
// rule the decode kernel uses; a zero-length sequence gets zeros.
//
// pda_merge_kernel: one warp per (sequence, head) row, 4 rows per 128-thread
// block; each lane folds the splits in order for 4 dims (lse_fold_row). Used
// up to kMergeRowSplits splits: a quarter of the blocks of one block per row
// (a batch of 128 x 64 rows at 2 splits went from 3.4 waves of short blocks
// to less than one).
// pda_merge_wide_kernel: one 128-thread block per row for more splits (a
// few very long sequences): warp w folds splits w, w + 4, ... and warp 0
// combines the four.
constexpr int kMergeRowSplits = 16;
constexpr int kMergeRowsPerBlock = kHeadDim / 32;

struct MergeParams {
  void* out;
  const float* part_o;
  const float* part_ml;
  const int32_t* seq_lens;
  int num_seqs;
  int num_heads;
  int block_size;
  int max_blocks;
  int nsplit;
  float v_scale;
  const float* sinks = nullptr;
  int out_fp8 = 0;
  float out_scale = 1.f;
};

// Store the merged row: lane's 4 dims of row (s, h).
__device__ __forceinline__ void merge_store(const MergeParams& p, int s, int h, int lane, bool any, float M, float den,
                                            const float4& acc) {
  store_merged(p.out, p.sinks, p.out_fp8, p.out_scale, p.v_scale, p.num_heads, s, h, lane, any, M, den, acc);
}

__global__ void __launch_bounds__(kHeadDim) pda_merge_kernel(const MergeParams p) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kMergeRowsPerBlock + (threadIdx.x >> 5);
  if (row >= (long long)p.num_seqs * p.num_heads) return;
  const int s = (int)(row / p.num_heads);
  const int h = (int)(row % p.num_heads);
  int L = __ldg(p.seq_lens + s);
  L = max(0, min(L, p.max_blocks * p.block_size));
  const int active = active_splits((L + p.block_size - 1) / p.block_size, p.nsplit);
  // Launched as the decode kernel's programmatic dependent: wait until it
  // has finished and its partials are visible (a no-op otherwise).
  grid_dependency_wait();
  float M, den;
  float4 acc;
  lse_fold_row(p.part_o, p.part_ml, (size_t)row * p.nsplit, active, lane, M, den, acc);
  merge_store(p, s, h, lane, active > 0, M, den, acc);
}

__global__ void __launch_bounds__(kHeadDim) pda_merge_wide_kernel(const MergeParams p) {
  constexpr int kWarps = kHeadDim / 32;
  const int h = blockIdx.x;
  const int s = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int L = __ldg(p.seq_lens + s);
  L = max(0, min(L, p.max_blocks * p.block_size));
  const int active = active_splits((L + p.block_size - 1) / p.block_size, p.nsplit);
  const size_t prow0 = ((size_t)s * p.num_heads + h) * p.nsplit;
  grid_dependency_wait();
  // Warp w folds splits w, w + kWarps, ... into a running (M, l, O) for dims
  // 4 lane .. 4 lane + 3, rescaling by 2^(M_old - M_new) as M grows.
  float M = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = warp; i < active; i += kWarps) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + (prow0 + i));
    const float4 o = __ldcg(reinterpret_cast<const float4*>(p.part_o + (prow0 + i) * kHeadDim) + lane);
    lse_fold(M, den, acc, ml.x, ml.y, o);
  }
  __shared__ float s_m[kWarps], s_l[kWarps];
  __shared__ float4 s_o[kWarps][32];
  if (lane == 0) {
    s_m[warp] = M;
    s_l[warp] = den;
  }
  s_o[warp][lane] = acc;
  __syncthreads();
  if (warp != 0) return;
  float Mt = -INFINITY;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) Mt = fmaxf(Mt, s_m[w]);
  float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
  float D = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (s_m[w] == -INFINITY) continue;  // a warp that merged no split
    const float f = fast_exp2(s_m[w] - Mt);
    const float4 o = s_o[w][lane];
    A.x = __fmaf_rn(f, o.x, A.x);
    A.y = __fmaf_rn(f, o.y, A.y);
    A.z = __fmaf_rn(f, o.z, A.z);
    A.w = __fmaf_rn(f, o.w, A.w);
    D = __fmaf_rn(f, s_l[w], D);
  }
  merge_store(p, s, h, lane, active > 0, Mt, D, A);
}

// Tail merge (persistent kernel with tail pieces): one warp per (tail unit,
// head) row, 4 rows per 128-thread block, launched as the decode kernel's
// programmatic dependent. Lane l folds dims 4l .. 4l+3 of the unit's pieces
// (tail_info[j] = {unit, first entry, pieces}) in piece order with
// lse_fold, then stores the row as the merge kernel does (one split per
// unit) or as the unit's split partial for the merge kernel, which is then
// launched as this grid's dependent. A unit of one piece was stored whole
// by the decode kernel. The decode kernel lets this grid launch only after
// its CTAs have waited for the order kernel, so tail_info can be read
// before waiting for the decode grid; with one split, rows with nothing to
// fold leave at once (with several, every row waits, so that this grid
// ends after the decode grid and the merge kernel after both).
struct TailMergeParams {
  MergeParams m;         // out, sinks, output format, v_scale, num_heads, nsplit
  float* part_o;         // several splits: the split partials the merge kernel folds
  float* part_ml;
  const int4* tail_info;
  const float* tail_rows;
  int tail_units;
  int num_kv_heads;
  int gqa;
};

__global__ void __launch_bounds__(kHeadDim) pda_tail_merge_kernel(const TailMergeParams p) {
  grid_dependents_launch();  // the merge kernel, if any, waits for this grid before reading
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kMergeRowsPerBlock + (threadIdx.x >> 5);
  const int nsplit = p.m.nsplit;
  if (row >= p.tail_units * p.gqa) {
    if (nsplit > 1) grid_dependency_wait();
    return;
  }
  const int j = row / p.gqa;
  const int hh = row % p.gqa;
  const int4 e = __ldcg(p.tail_info + j);
  if (e.z <= 1 && nsplit == 1) return;
  grid_dependency_wait();  // the decode kernel's pieces are stored and visible
  if (e.z <= 1) return;
  const int s = e.x / (p.num_kv_heads * nsplit);
  const int kvh = (e.x / nsplit) % p.num_kv_heads;
  const int split = e.x % nsplit;
  // every piece's values first, so the loads overlap, then the fold
  float2 ml[kMaxTailPieces];
  float4 o[kMaxTailPieces];
#pragma unroll
  for (int i = 0; i < kMaxTailPieces; ++i) {
    if (i < e.z) {
      const float* rows = p.tail_rows + (size_t)(e.y + i) * kTailRowFloats;
      ml[i] = __ldcg(reinterpret_cast<const float2*>(rows + kMaxGqa * kHeadDim) + hh);
      o[i] = __ldcg(reinterpret_cast<const float4*>(rows + hh * kHeadDim) + lane);
    }
  }
  float M = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < kMaxTailPieces; ++i)
    if (i < e.z) lse_fold(M, den, acc, ml[i].x, ml[i].y, o[i]);
  const int h = kvh * p.gqa + hh;
  if (nsplit == 1) {
    merge_store(p.m, s, h, lane, true, M, den, acc);
  } else {
    // the split's partial, as the decode kernel stores a whole split's
    const size_t prow = ((size_t)s * p.m.num_heads + h) * nsplit + split;
    reinterpret_cast<float4*>(p.part_o + prow * kHeadDim)[lane] = acc;
    if (lane == 0) reinterpret_cast<float2*>(p.part_ml)[prow] = make_float2(M, den);
  }
}

// One CTA waits on an mbarrier that nothing completes, with a short limit,
// then records kStatusTestWaitTimeout and returns. Exercises the bounded
// wait used by the decode kernel without faulting or hanging anything.
__global__ void pda_bounded_wait_test_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(b, 0u, nullptr, limit_ns)) atomicOr(&g_status, kStatusTestWaitTimeout);
  }
}

// KV-cache write: quantise new keys / values to e4m3 with the per-tensor
// scales and scatter them into the paged cache (vLLM API page
// vllm.v1.attention.backends.rocm_aiter_unified_attn, do_kv_cache_update ->
// reshape_and_cache), for slot = b * bs + o:
//   K bytes -> k_cache[b][k][d/16][o][d%16]
//   V bytes -> v_cache[b][k][d][o], or v_cache[b][k][o/16][d][o%16] (shuffled V)
// The code is decided on the IEEE binary32 quotient x / scale. Negative slots
// are padding; slots past the pool are skipped and flagged in the status word.
//
// One 128-thread CTA per (16 consecutive tokens, kv head). Thread (j, c)
// quantises token j's 16 dims of chunk c (two 32-byte loads per tensor, so
// many bytes are in flight) and stores its 16 K codes as one 16-byte K row.
// The V codes go through shared memory. V rows run over tokens: when the
// 16 slots form one aligned run of a block (a prefill writing whole
// groups), thread d stores dim d of the 16 tokens as one 16-byte row;
// otherwise (a decode step's slots, scattered over the pool) warp w stores
// tokens 4w..4w+3 one at a time, its 32 lanes writing 4 bytes each into that
// token's page, so every store instruction stays within one page.
struct CacheWriteParams {
  const __nv_bfloat16* key;      // [T][Hk][128]
  const __nv_bfloat16* value;    // [T][Hk][128]
  uint8_t* k_cache;
  uint8_t* v_cache;
  const int64_t* slot_mapping;   // [T]
  int num_tokens;
  int num_kv_heads;
  int block_size;
  long long num_slots;           // num_blocks * block_size
  float k_scale;
  float v_scale;
  int v_shuffled = 0;            // 1: V pages are [bs/16][D][16]
};

constexpr int kCacheWriteTokens = 16;   // one aligned run at most
constexpr int kCacheWriteThreads = 128;  // 16 tokens x 8 chunks of 16 dims
constexpr int kCacheWriteWarpsPerCta = 8;  // scattered writer: one warp per (token, kv head)

__device__ __forceinline__ uint4 quantize16(const __nv_bfloat16* src, float scale) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
  const uint4 b = __ldg(reinterpret_cast<const uint4*>(src) + 1);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(bf16lo_f32(w[2 * i]), scale), __fdiv_rn(bf16hi_f32(w[2 * i]), scale));
    const uint32_t hi =
        f32x2_to_e4m3x2(__fdiv_rn(bf16lo_f32(w[2 * i + 1]), scale), __fdiv_rn(bf16hi_f32(w[2 * i + 1]), scale));
    q[i] = lo | (hi << 16);
  }
  return make_uint4(q[0], q[1], q[2], q[3]);
}

__global__ void __launch_bounds__(kCacheWriteThreads) pda_reshape_and_cache_kernel(const CacheWriteParams p) {
  __shared__ __align__(16) uint8_t vt[kCacheWriteTokens][kHeadDim];  // V codes [token][dim]
  __shared__ long long slots[kCacheWriteTokens];                      // -1: nothing to write
  const int tid = threadIdx.x;
  const int j = tid >> 3;
  const int c = tid & 7;
  const int k = blockIdx.y;
  const int t = blockIdx.x * kCacheWriteTokens + j;
  const int bs = p.block_size;

  long long slot = -1;
  if (t < p.num_tokens) slot = __ldg(p.slot_mapping + t);
  const bool in_pool = slot < p.num_slots;
  if (slot >= 0 && !in_pool && c == 0) atomicOr(&g_status, kStatusBadSlot);
  const bool valid = slot >= 0 && in_pool;

  if (valid) {
    const size_t src = ((size_t)t * p.num_kv_heads + k) * kHeadDim + 16 * c;
    const uint4 kq = quantize16(p.key + src, p.k_scale);
    const uint4 vq = quantize16(p.value + src, p.v_scale);
    const long long b = slot / bs;
    const int o = (int)(slot % bs);
    const size_t page = ((size_t)b * p.num_kv_heads + k) * (size_t)kHeadDim * bs;
    *reinterpret_cast<uint4*>(p.k_cache + page + ((size_t)c * bs + o) * 16) = kq;
    *reinterpret_cast<uint4*>(&vt[j][16 * c]) = vq;
  }
  if (c == 0) slots[j] = valid ? slot : -1;
  __syncthreads();

  // One aligned run of 16 slots in one block? (uniform over the CTA)
  const long long first = slots[0];
  const bool run = valid && (first % kCacheWriteTokens == 0) && (slot == first + j);
  if (__syncthreads_and(run ? 1 : 0)) {
    // thread d gathers dim d of the 16 tokens: one V row of the run
    const int d = tid;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = (uint32_t)vt[4 * i][d] | ((uint32_t)vt[4 * i + 1][d] << 8) | ((uint32_t)vt[4 * i + 2][d] << 16) |
             ((uint32_t)vt[4 * i + 3][d] << 24);
    const long long b0 = first / bs;
    const int o0 = (int)(first % bs);
    const size_t page0 = ((size_t)b0 * p.num_kv_heads + k) * (size_t)kHeadDim * bs;
    const size_t off = p.v_shuffled ? ((size_t)(o0 / 16) * kHeadDim + d) * 16 : (size_t)d * bs + o0;
    *reinterpret_cast<uint4*>(p.v_cache + page0 + off) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    // warp w writes tokens 4w..4w+3 one after the other, lane l dims 4l..4l+3
    const int warp = tid >> 5;
    const int d0 = 4 * (tid & 31);
    const size_t vstride = p.v_shuffled ? 16 : (size_t)bs;
#pragma unroll
    for (int i = 0; i < kCacheWriteTokens / 4; ++i) {
      const int jj = 4 * warp + i;
      const long long sl = slots[jj];
      if (sl < 0) continue;
      const long long b = sl / bs;
      const int o = (int)(sl % bs);
      const uint32_t v = *reinterpret_cast<const uint32_t*>(&vt[jj][d0]);
      uint8_t* vrow = p.v_cache + ((size_t)b * p.num_kv_heads + k) * (size_t)kHeadDim * bs +
                      (p.v_shuffled ? ((size_t)(o / 16) * kHeadDim + d0) * 16 + (o % 16) : (size_t)d0 * bs + o);
#pragma unroll
      for (int q = 0; q < 4; ++q) vrow[(size_t)q * vstride] = (uint8_t)(v >> (8 * q));
    }
  }
}

// Scattered writer for small writes (a decode step: one token per sequence,
// at slots all over the pool): one warp per (token, kv head), 4 dims per
// lane, no shared memory or block barrier, so a small grid finishes soonest.
__global__ void __launch_bounds__(kCacheWriteWarpsPerCta * 32)
    pda_reshape_and_cache_scatter_kernel(const CacheWriteParams p) {
  const long long item = (long long)blockIdx.x * kCacheWriteWarpsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (item >= (long long)p.num_tokens * p.num_kv_heads) return;
  const int t = (int)(item / p.num_kv_heads);
  const int k = (int)(item % p.num_kv_heads);
  const long long slot = __ldg(p.slot_mapping + t);
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (lane == 0) atomicOr(&g_status, kStatusBadSlot);
    return;
  }
  const int bs = p.block_size;
  const long long b = slot / bs;
  const int o = (int)(slot % bs);
  const size_t src = ((size_t)t * p.num_kv_heads + k) * kHeadDim + 4 * lane;
  const uint2 kx = ld_nc_v2(p.key + src);
  const uint2 vx = ld_nc_v2(p.value + src);
  const float ks = p.k_scale, vs = p.v_scale;
  const uint32_t kq = f32x2_to_e4m3x2(__fdiv_rn(bf16lo_f32(kx.x), ks), __fdiv_rn(bf16hi_f32(kx.x), ks)) |
                      (f32x2_to_e4m3x2(__fdiv_rn(bf16lo_f32(kx.y), ks), __fdiv_rn(bf16hi_f32(kx.y), ks)) << 16);
  const uint32_t vq = f32x2_to_e4m3x2(__fdiv_rn(bf16lo_f32(vx.x), vs), __fdiv_rn(bf16hi_f32(vx.x), vs)) |
                      (f32x2_to_e4m3x2(__fdiv_rn(bf16lo_f32(vx.y), vs), __fdiv_rn(bf16hi_f32(vx.y), vs)) << 16);
  const size_t page = ((size_t)b * p.num_kv_heads + k) * (size_t)kHeadDim * bs;
  const int d0 = 4 * lane;
  *reinterpret_cast<uint32_t*>(p.k_cache + page + ((size_t)(d0 / 16) * bs + o) * 16 + (d0 % 16)) = kq;
  const size_t vstride = p.v_shuffled ? 16 : (size_t)bs;
  uint8_t* vrow =
      p.v_cache + page + (p.v_shuffled ? ((size_t)(o / 16) * kHeadDim + d0) * 16 + (o % 16) : (size_t)d0 * bs + o);
#pragma unroll
  for (int i = 0; i < 4; ++i) vrow[(size_t)i * vstride] = (uint8_t)(vq >> (8 * i));
}

}  // namespace pda
