// fp64 CPU oracle for fp8 paged decode attention.
//
// TEST INFRASTRUCTURE ONLY. This file is the parity reference for the CUDA
// decode path and shares no code, header, table or helper with it. Only the
// test suite, the smoke check and the benchmark's CPU-baseline leg may load it.
//
// What it computes (the plain definition, no splitting, no blocking):
//   for every sequence s and query head h, with kv = h / g (g = H / Hk) and
//   L = seq_lens[s]:
//     k_t[d] = E4M3(K byte of token t, dim d) * k_scale
//     v_t[d] = E4M3(V byte of token t, dim d) * v_scale
//     z_t    = scale * sum_d q[s][h][d] * k_t[d]                 (t < L)
//     out[s][h][d] = sum_t exp(z_t - max z) v_t[d] / sum_t exp(z_t - max z)
//   all in IEEE binary64. L = 0 gives a zero row.
//
// Sources for each part:
//  * single-query paged attention over seq_lens / block_table with a softmax
//    scale and K/V descale factors: vLLM API page
//    "vllm.v1.attention.backends.rocm_aiter_unified_attn",
//    RocmAiterUnifiedAttentionImpl.forward (the unified_attention call with
//    q, k, v, seqused_k, softmax_scale, block_table, k_descale, v_descale).
//  * page layout of an fp8 cache: vLLM pull request lishuoshuo-amd/vllm#3,
//    section "Details", item "Layout": K as [blocks, kv_heads, head_size/16,
//    16, 16] and V as [blocks, kv_heads, head_size, 16] for 16-token blocks.
//    The K intra-page order [dim/16][token][dim%16] follows the same API
//    page's _shuffle_kv_views (K viewed as (nb, nkv, hd//x, bs, x) with
//    x = 16 one-byte elements). For block sizes above 16 the V page is read
//    as [head_size][block_size], the direct generalisation of the item above.
//  * per-tensor scales broadcast to every slot: same pull request, section
//    "Details", item "Scale tables".
//  * fp8 flavour: OCP FP8 E4M3 ("e4m3fn": bias 7, no infinities, S.1111.111
//    is NaN, largest finite 448), the format the API page lists as fp8_e4m3.
//  * consecutive query heads share a kv head (h / g): the API page's forward
//    passes num_kv_heads K/V heads for num_heads query heads; the grouping
//    rule itself is not printed there, and h / g is the reading taken.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// OCP FP8 E4M3 decode from the format's definition: sign bit, 4-bit
// exponent with bias 7, 3-bit mantissa; exponent 0 is subnormal
// (2^-6 * m/8); exponent 15 with mantissa 7 is NaN (no infinities).
double e4m3_value(uint8_t code) {
  const int sign = (code >> 7) & 1;
  const int expo = (code >> 3) & 0xF;
  const int mant = code & 0x7;
  double mag;
  if (expo == 0xF && mant == 0x7) {
    return std::nan("");
  } else if (expo == 0) {
    mag = std::ldexp(static_cast<double>(mant) / 8.0, -6);
  } else {
    mag = std::ldexp(1.0 + static_cast<double>(mant) / 8.0, expo - 7);
  }
  return sign ? -mag : mag;
}

// bfloat16 is the upper half of an IEEE binary32: widen and reinterpret.
double bf16_value(uint16_t bits) {
  const uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// Nearest OCP E4M3 code to x by exhaustive search over the finite
// non-negative codes: ties go to the even code (even mantissa), magnitudes
// past 448 saturate to 448, the sign is kept (so -0 and tiny negatives give
// 0x80), NaN gives the NaN code with x's sign.
uint8_t e4m3_encode(double x) {
  if (std::isnan(x)) return std::signbit(x) ? 0xFF : 0x7F;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs(x);
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    const double d = std::fabs(a - e4m3_value(static_cast<uint8_t>(c)));
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return static_cast<uint8_t>(sign | best);
}

}  // namespace

extern "C" {

// Status codes returned by the oracle entry points.
enum {
  PDA_ORACLE_OK = 0,
  PDA_ORACLE_BAD_SHAPE = -1,      // non-positive sizes, H % Hk != 0, D % 16 != 0
  PDA_ORACLE_BAD_SEQ_LEN = -2,    // seq_lens[s] < 0 or > max_num_blocks_per_seq * block_size
  PDA_ORACLE_BAD_BLOCK_ID = -3,   // a block id a sequence uses is outside [0, num_blocks)
  PDA_ORACLE_BAD_SEQ_ID = -4,     // a requested sequence index is outside [0, num_seqs)
};

double pda_oracle_e4m3_value(uint8_t code) { return e4m3_value(code); }
double pda_oracle_bf16_value(uint16_t bits) { return bf16_value(bits); }

// Decode attention for the sequences listed in seq_ids (all of them when
// seq_ids is NULL). out is [n_out][num_heads][head_size] binary64 with
// n_out = n_ids (or num_seqs). Layouts (all row-major, unpadded):
//   q            [num_seqs][num_heads][head_size] bfloat16 bit patterns
//   k_cache      [num_blocks][num_kv_heads][head_size/16][block_size][16] e4m3 bytes
//   v_cache      [num_blocks][num_kv_heads][head_size][block_size] e4m3 bytes
//   block_tables [num_seqs][max_num_blocks_per_seq] int32 physical block ids
//   seq_lens     [num_seqs] int32
// Only the first ceil(seq_lens[s] / block_size) entries of a table row are
// read; only token slots t < seq_lens[s] are read from a page.
//
// V layout: v_shuffled == 0 reads V pages as [head_size][block_size];
// v_shuffled == 1 reads AITER's shuffled V, [block_size/16][head_size][16]
// per (block, kv head) (vLLM pull request lishuoshuo-amd/vllm#3, "Details",
// item "Layout"; the API page's _shuffle_kv_views, V viewed as
// (nb, nkv, bs//x, hd, x)). The two coincide at block_size 16.
//
// Attention sinks (the API page passes sinks= to unified_attention and its
// backend reports supports_sink; the arithmetic is not printed there): when
// sinks is non-NULL, sinks[h] is a logit of query head h, in the same units
// as scale * q . k, that joins the softmax normaliser but carries no value:
//   out = sum_t e^(z_t - M) v_t / (sum_t e^(z_t - M) + e^(sink_h - M)),
//   M = max(max_t z_t, sink_h); a zero-length sequence still gives zeros.
//
// Per-slot scale tables (vLLM pull request lishuoshuo-amd/vllm#3, "Details",
// item "Scale tables": the asm kernel reads per-slot [blocks, kv_heads,
// block_size] scales): when k_scales / v_scales are non-NULL they are fp32
// [num_blocks][num_kv_heads][block_size] and the token in slot o of block b,
// kv head k, dequantises with k_scales[b][k][o] (v_scales[b][k][o]) in place
// of the per-tensor k_scale (v_scale).
int pda_oracle_decode(double* out, const uint16_t* q, const uint8_t* k_cache,
                      const uint8_t* v_cache, const int32_t* block_tables,
                      const int32_t* seq_lens, int num_seqs, int num_heads,
                      int num_kv_heads, int head_size, int block_size,
                      int max_num_blocks_per_seq, long long num_blocks,
                      double scale, double k_scale, double v_scale,
                      const float* k_scales, const float* v_scales, const float* sinks,
                      int v_shuffled, const int32_t* seq_ids, int n_ids, int num_threads) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 ||
      block_size <= 0 || max_num_blocks_per_seq < 0 || num_blocks < 0 ||
      num_heads % num_kv_heads != 0 || head_size % 16 != 0) {
    return PDA_ORACLE_BAD_SHAPE;
  }
  const int n_out = seq_ids ? n_ids : num_seqs;
  const int g = num_heads / num_kv_heads;
  const int D = head_size;
  const long long bs = block_size;
  const long long MB = max_num_blocks_per_seq;

  // Validate every sequence the call will read before any work.
  for (int i = 0; i < n_out; ++i) {
    const int s = seq_ids ? seq_ids[i] : i;
    if (s < 0 || s >= num_seqs) return PDA_ORACLE_BAD_SEQ_ID;
    const long long L = seq_lens[s];
    if (L < 0 || L > MB * bs) return PDA_ORACLE_BAD_SEQ_LEN;
    const long long pages = (L + bs - 1) / bs;
    for (long long j = 0; j < pages; ++j) {
      const long long b = block_tables[s * MB + j];
      if (b < 0 || b >= num_blocks) return PDA_ORACLE_BAD_BLOCK_ID;
    }
  }

  // The 256 possible byte values, decoded once (same values as e4m3_value).
  double e4m3[256];
  for (int c = 0; c < 256; ++c) e4m3[c] = e4m3_value(static_cast<uint8_t>(c));

  const long long rows = static_cast<long long>(n_out) * num_heads;
#ifdef _OPENMP
  const int nt = num_threads > 0 ? num_threads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
#endif
  for (long long r = 0; r < rows; ++r) {
    const int i = static_cast<int>(r / num_heads);
    const int h = static_cast<int>(r % num_heads);
    const int s = seq_ids ? seq_ids[i] : i;
    const int kv = h / g;
    const long long L = seq_lens[s];
    double* o = out + r * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (L == 0) continue;

    std::vector<double> qd(D);
    for (int d = 0; d < D; ++d) qd[d] = bf16_value(q[(static_cast<long long>(s) * num_heads + h) * D + d]);

    // Logits z_t = scale * q . k_t.
    std::vector<double> z(L);
    for (long long t = 0; t < L; ++t) {
      const long long b = block_tables[s * MB + t / bs];
      const long long slot = t % bs;
      const uint8_t* kpage = k_cache + (b * num_kv_heads + kv) * static_cast<long long>(D) * bs;
      const double ks = k_scales ? static_cast<double>(k_scales[(b * num_kv_heads + kv) * bs + slot]) : k_scale;
      double acc = 0.0;
      for (int d = 0; d < D; ++d) {
        const uint8_t code = kpage[(static_cast<long long>(d / 16) * bs + slot) * 16 + (d % 16)];
        acc += qd[d] * (e4m3[code] * ks);
      }
      z[t] = scale * acc;
    }

    // softmax(z) . V (with the sink, if any, in the normaliser only)
    double zmax = z[0];
    for (long long t = 1; t < L; ++t) zmax = z[t] > zmax ? z[t] : zmax;
    const double zs = sinks ? static_cast<double>(sinks[h]) : -INFINITY;
    if (zs > zmax) zmax = zs;
    double denom = sinks ? std::exp(zs - zmax) : 0.0;
    std::vector<double> w(L);
    for (long long t = 0; t < L; ++t) {
      w[t] = std::exp(z[t] - zmax);
      denom += w[t];
    }
    for (long long t = 0; t < L; ++t) {
      const long long b = block_tables[s * MB + t / bs];
      const long long slot = t % bs;
      const uint8_t* vpage = v_cache + (b * num_kv_heads + kv) * static_cast<long long>(D) * bs;
      const double vs = v_scales ? static_cast<double>(v_scales[(b * num_kv_heads + kv) * bs + slot]) : v_scale;
      const double wt = w[t] / denom;
      for (int d = 0; d < D; ++d) {
        const long long vi = v_shuffled ? ((slot / 16) * D + d) * 16 + (slot % 16)
                                        : static_cast<long long>(d) * bs + slot;
        o[d] += wt * (e4m3[vpage[vi]] * vs);
      }
    }
  }
  return PDA_ORACLE_OK;
}

uint8_t pda_oracle_e4m3_encode(double x) { return e4m3_encode(x); }

// Static per-tensor fp8 output quantisation (the API page's fused output
// quantisation, kFp8StaticTensorSym: one scale, symmetric): code =
// E4M3(x / output_scale), nearest e4m3 value of the exact quotient, ties to
// even, saturating at +-448.
void pda_oracle_quantize_e4m3(const double* x, uint8_t* codes, long long n, double output_scale) {
  for (long long i = 0; i < n; ++i) codes[i] = e4m3_encode(x[i] / output_scale);
}

// KV-cache write: quantise new keys / values and scatter them into the
// paged cache (vLLM API page "vllm.v1.attention.backends.rocm_aiter_unified_attn",
// RocmAiterUnifiedAttentionImpl.do_kv_cache_update -> reshape_and_cache with
// key, value, key_cache, value_cache, slot_mapping, k_scale, v_scale).
// For token t with slot = slot_mapping[t] >= 0, block b = slot / block_size,
// offset o = slot % block_size, kv head k and dim d:
//   k_cache[b][k][d/16][o][d%16] = E4M3( float(key[t][k][d]) / k_scale )
//   v_cache[b][k][d][o]          = E4M3( float(value[t][k][d]) / v_scale )
// (v_shuffled = 1: v_cache[b][k][o/16][d][o%16], the shuffled V layout.)
// The quotient is the binary32 quotient (the cache stores what a binary32
// division produces before rounding to e4m3); E4M3 is e4m3_encode. Negative
// slots are skipped (padding). key / value are bf16 bit patterns
// [num_tokens][num_kv_heads][head_size]. Returns PDA_ORACLE_BAD_SHAPE or
// PDA_ORACLE_BAD_BLOCK_ID (a slot past the pool) without writing anything.
int pda_oracle_reshape_and_cache(uint8_t* k_cache, uint8_t* v_cache, const uint16_t* key,
                                 const uint16_t* value, const int64_t* slot_mapping, int num_tokens,
                                 int num_kv_heads, int head_size, int block_size, long long num_blocks,
                                 float k_scale, float v_scale, int v_shuffled) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || head_size % 16 != 0 ||
      block_size <= 0 || num_blocks < 0) {
    return PDA_ORACLE_BAD_SHAPE;
  }
  const long long bs = block_size;
  const long long D = head_size;
  for (int t = 0; t < num_tokens; ++t) {
    if (slot_mapping[t] >= num_blocks * bs) return PDA_ORACLE_BAD_BLOCK_ID;
  }
  for (int t = 0; t < num_tokens; ++t) {
    const long long slot = slot_mapping[t];
    if (slot < 0) continue;
    const long long b = slot / bs;
    const long long o = slot % bs;
    for (int k = 0; k < num_kv_heads; ++k) {
      for (long long d = 0; d < D; ++d) {
        const long long src = (static_cast<long long>(t) * num_kv_heads + k) * D + d;
        const float xk = static_cast<float>(bf16_value(key[src])) / k_scale;
        const float xv = static_cast<float>(bf16_value(value[src])) / v_scale;
        const long long page = (b * num_kv_heads + k) * D * bs;
        k_cache[page + ((d / 16) * bs + o) * 16 + (d % 16)] = e4m3_encode(xk);
        const long long vi = v_shuffled ? ((o / 16) * D + d) * 16 + (o % 16) : d * bs + o;
        v_cache[page + vi] = e4m3_encode(xv);
      }
    }
  }
  return PDA_ORACLE_OK;
}

int pda_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

}  // extern "C"
