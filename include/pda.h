/*
 * pda.h -- fp8 paged decode attention for NVIDIA GB300 (sm_103a), C ABI.
 *
 * One call computes single-query ("decode") attention for a batch of
 * sequences whose keys and values sit in a paged fp8 cache:
 *
 *   out[s][h][:] = softmax_t( scale * q[s][h] . k_t ) . v_t ,  t < seq_lens[s]
 *
 * with k_t, v_t the e4m3 cache bytes of token t times k_scale / v_scale,
 * gathered page by page through block_tables, and query head h reading kv
 * head h / (num_heads / num_kv_heads).
 *
 * Sources. What the call computes and its argument roles follow the vLLM API
 * page "vllm.v1.attention.backends.rocm_aiter_unified_attn"
 * (RocmAiterUnifiedAttentionImpl.forward: q, k, v, out, seqused_k,
 * softmax_scale, block_table, k_descale, v_descale). The cache layout follows
 * vLLM pull request lishuoshuo-amd/vllm#3 ("Details", item "Layout"): for an
 * fp8 cache, K as [blocks, kv_heads, head_size/16, 16, 16] and V as
 * [blocks, kv_heads, head_size, 16] with 16-token blocks, pages addressed by
 * a dense page stride. The K intra-page order (token-major inside each
 * 16-dimension chunk) is the one the API page's _shuffle_kv_views gives
 * (K viewed as (nb, nkv, hd//x, bs, x), x = 16 bytes). Per-tensor scales
 * follow the pull request's "Scale tables" item (a table filled with the
 * per-tensor scale); block sizes that are multiples of 16 follow the API
 * page's supports_block_size / customize_spec; GQA ratios up to 8 follow the
 * pull request's "Claims" and "Cut and precision" items.
 *
 * Threading and ordering. Every entry point is thread-safe. pda_decode is
 * stream-ordered: it validates on the host, enqueues its kernels on `stream`
 * and returns without synchronising the host, reading device memory from the
 * host, or allocating (once the workspace is large enough), so it can be
 * captured in a CUDA graph. Errors detected on the host return before any
 * launch; nothing is written to `out` then.
 */
#ifndef PDA_H_
#define PDA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same opaque handle types as the CUDA runtime's (identical typedefs). */
typedef struct CUstream_st* cudaStream_t;
typedef struct CUevent_st* cudaEvent_t;

typedef enum pda_status {
  PDA_OK = 0,
  PDA_ERR_INVALID_ARG = 1,     /* null / misaligned pointer, negative size, H % Hk != 0 */
  PDA_ERR_UNSUPPORTED = 2,     /* valid but outside the supported set (see pda_decode) */
  PDA_ERR_WORKSPACE = 3,       /* workspace must grow while the stream is being captured */
  PDA_ERR_CUDA = 4,            /* a CUDA runtime call or kernel launch failed */
  PDA_ERR_DEVICE_TIMEOUT = 5,  /* a kernel reported a device-side error (pda_query_device_status) */
  PDA_ERR_NOALLOC_CAPACITY = 6 /* pda_decode_noalloc: the call needs more scratch than its static buffer */
} pda_status;

/*
 * pda_decode -- decode attention over a paged fp8 KV cache.
 *
 * Device pointers (all on the device that is current for the calling thread
 * and that owns `stream`; each 16-byte aligned; row-major, unpadded):
 *   out           bf16  [num_seqs][num_heads][head_size]          written
 *   q             bf16  [num_seqs][num_heads][head_size]          read
 *   k_cache       e4m3  [num_blocks][num_kv_heads][head_size/16][block_size][16]  read
 *   v_cache       e4m3  [num_blocks][num_kv_heads][head_size][block_size]          read
 *   block_tables  int32 [num_seqs][max_num_blocks_per_seq]        read
 *   seq_lens      int32 [num_seqs]                                read
 * e4m3 is OCP FP8 E4M3 (torch.float8_e4m3fn). Sequence s reads the first
 * ceil(seq_lens[s] / block_size) entries of its table row and, in its last
 * page, only the slots below seq_lens[s]; other slots and entries may hold
 * anything. A sequence with seq_lens[s] == 0 gets a zero output row.
 *
 * Scalars: scale is the softmax scale (1/sqrt(head_size) for plain
 * attention); k_scale and v_scale multiply the e4m3 values on dequantisation
 * (value = e4m3 * scale), i.e. the k/v "descale" of the API page.
 *
 * Value range: q may hold any finite bf16 values (the whole bf16 range, not
 * only f16's): each query row is scaled by a power of two before it enters
 * the f16 tensor-core products and the logit scale by its inverse, which is
 * exact. The logits scale * k_scale * q . k_t must stay finite in binary32
 * (|logit| < 2^126 suffices), and they carry binary32's relative precision:
 * with logits of magnitude X, tokens whose logits differ by less than about
 * X * 2^-22 are weighted only that precisely (at X ~ 1e5, a few tenths of a
 * percent). NaN or infinite inputs give undefined output.
 * Arithmetic: e4m3 -> f16 is exact, and so is the shifted bf16 q -> f16 for
 * every value within 2^24 of its row's largest (smaller ones round to f16's
 * subnormal grid); scores, softmax and accumulation are fp32; the
 * probabilities enter the PV product as two f16 parts (f16(p) and
 * f16(p - f16(p))), about 2^-22 relative.
 *
 * max_num_blocks_per_seq is the row stride of block_tables. It is not in the
 * argument list the method states; it is required to index a [S, MB] table
 * and gives the host an upper bound on context length without reading
 * seq_lens back from the device (which would synchronise).
 *
 * Supported set: head_size == 128; block_size a multiple of 16, 16..128;
 * num_heads % num_kv_heads == 0 with a ratio of 1..8; num_seqs >= 0
 * (0 returns PDA_OK with no launch); seq_lens[s] <= max_num_blocks_per_seq *
 * block_size and every used block id in [0, num_blocks) are the caller's
 * contract (the kernel never reads past a table row and clamps lengths to
 * the row's capacity; it does not know num_blocks). pda_set_block_check
 * makes the kernels check block ids against a given pool size;
 * pda_decode_host checks the table on the host.
 *
 * Ownership: the caller owns every buffer. The library owns an internal
 * per-(device, stream) workspace: the persistent kernel's work-queue words
 * and unit order, and the split partials. It grows with cudaMallocAsync on
 * `stream` when a call needs more and the stream is not capturing. If it is
 * capturing, a call that needs split partials returns PDA_ERR_WORKSPACE
 * (size the workspace first with pda_reserve), and a one-split call runs the
 * per-unit kernel, which needs none. Calls on one stream run in stream order
 * and share its workspace; calls on different streams have their own.
 * A CUDA graph that captured a call keeps that call's workspace address: when
 * a later, larger call grows the workspace, the old buffer is kept allocated
 * (not reused) until pda_release, so replaying the graph stays valid.
 * pda_release frees every workspace, old ones included, and so invalidates
 * every graph that captured a pda_decode* call; re-capture after it. Two
 * replays of graphs that captured calls on one stream share that stream's
 * workspace and must not run at the same time.
 *
 * Determinism: for fixed inputs and a fixed split count the result is
 * bitwise reproducible. Which CTA computes a work unit, and when, changes
 * from call to call (the persistent kernel hands units out from a queue) but
 * never changes the unit's result. The split count depends on
 * num_seqs * num_kv_heads and max_num_blocks_per_seq, so a sequence's result
 * may change in the last bits with the batch it shares a call with.
 *
 * Returns PDA_OK, PDA_ERR_INVALID_ARG, PDA_ERR_UNSUPPORTED,
 * PDA_ERR_WORKSPACE or PDA_ERR_CUDA (launch failure).
 */
pda_status pda_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                      int num_heads, int num_kv_heads, int head_size, int block_size,
                      int max_num_blocks_per_seq, float scale, float k_scale, float v_scale,
                      cudaStream_t stream);

/*
 * KV cache layouts (pda_decode_ex, pda_reshape_and_cache). K is always
 * [num_blocks][num_kv_heads][head_size/16][block_size][16].
 *   PDA_KV_NATIVE      V [num_blocks][num_kv_heads][head_size][block_size]
 *   PDA_KV_SHUFFLED_V  V [num_blocks][num_kv_heads][block_size/16][head_size][16]
 * The shuffled V is AITER's layout; at block_size 16 the two are the same
 * bytes (vLLM pull request lishuoshuo-amd/vllm#3, "Details", item "Layout";
 * the API page's _shuffle_kv_views views V as (nb, nkv, bs//x, hd, x)).
 */
typedef enum pda_kv_layout {
  PDA_KV_NATIVE = 0,
  PDA_KV_SHUFFLED_V = 1
} pda_kv_layout;

/* Output element type of pda_decode_ex. */
typedef enum pda_out_dtype {
  PDA_OUT_BF16 = 0,  /* bf16 [num_seqs][num_heads][head_size] */
  PDA_OUT_E4M3 = 1   /* e4m3 bytes [num_seqs][num_heads][head_size]: E4M3(o / output_scale) */
} pda_out_dtype;

/*
 * pda_decode_ex -- pda_decode with attention sinks and fused fp8 output.
 *
 * Source: the vLLM API page "vllm.v1.attention.backends.rocm_aiter_unified_attn"
 * passes sinks= and output_scale= to the attention call (its backend reports
 * supports_sink, and fused output quantisation for kFp8StaticTensorSym, one
 * static symmetric per-tensor scale). The page does not print either
 * computation; this library takes the plain reading of each:
 *
 *   sinks        fp32 [num_heads] on the device, or NULL. sinks[h] is a
 *                logit of query head h in the units of scale * q . k that
 *                joins the softmax normaliser and carries no value:
 *                out = sum_t e^(z_t) v_t / (sum_t e^(z_t) + e^(sinks[h])).
 *                A zero-length sequence still gives zeros.
 *   out_dtype    PDA_OUT_BF16 (as pda_decode) or PDA_OUT_E4M3: out holds
 *                e4m3 bytes E4M3(o / output_scale), the binary32 quotient
 *                rounded to the nearest e4m3 value (ties to even),
 *                saturating at +-448.
 *   output_scale finite and > 0 when out_dtype is PDA_OUT_E4M3 (ignored
 *                otherwise).
 *
 *   kv_layout    PDA_KV_NATIVE (pda_decode's layout) or PDA_KV_SHUFFLED_V.
 *
 * Everything else is pda_decode's. Returns PDA_ERR_INVALID_ARG for an
 * unknown kv_layout or out_dtype, a bad output_scale or a misaligned sinks
 * pointer.
 */
pda_status pda_decode_ex(void* out, const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, const int32_t* seq_lens, int num_seqs, int num_heads,
                         int num_kv_heads, int head_size, int block_size, int max_num_blocks_per_seq, float scale,
                         float k_scale, float v_scale, int kv_layout, const float* sinks, int out_dtype,
                         float output_scale, cudaStream_t stream);

/*
 * pda_decode_strided -- pda_decode on token-major ("flash" / NHD family)
 * caches given by byte strides.
 *
 * Source: the vLLM API page "vllm.v1.attention.backends.rocm_aiter_unified_attn":
 * the backend's kv_cache is documented as [num_blocks, 2, block_size,
 * num_kv_heads, head_size], its _split_kv_cache turns a (blocks, heads,
 * tokens, 2*head_size) tensor into K and V views of shape (blocks, tokens,
 * heads, head_size) ("keep K and V packed in the content dim"), and it
 * supports the LBHNC and LHBNC layouts. In all of these the head_size bytes
 * of one (block, token, kv head) are contiguous and everything else is a
 * stride, so one entry point covers them:
 *
 *   K row of (block b, token t, kv head h) = k_cache + b*k_block_stride
 *                                           + t*k_token_stride + h*k_head_stride
 *   (V likewise with v_cache and the v_* strides), head_size = 128 bytes, e4m3.
 *
 * Examples (bytes; D = 128):
 *   [NB, bs, Hk, D] for K and for V:  block bs*Hk*D, token Hk*D, head D
 *   [NB, 2, bs, Hk, D]:               K = base, V = base + bs*Hk*D;
 *                                     block 2*bs*Hk*D, token Hk*D, head D
 *   [NB, Hk, bs, 2*D] (K|V packed):   K = base, V = base + D;
 *                                     block Hk*bs*2*D, token 2*D, head bs*2*D
 *
 * num_blocks bounds the block index (pages are read through TMA tensor maps
 * built from these strides; a block id outside [0, num_blocks) reads zeros).
 * Strides must be positive multiples of 16 that nest without overlap once
 * sorted (smallest >= 128), and K and V must sort in the same order; else
 * PDA_ERR_UNSUPPORTED. Everything else is pda_decode's.
 */
pda_status pda_decode_strided(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, const int32_t* seq_lens, int num_seqs, int num_heads,
                              int num_kv_heads, int head_size, int block_size, int max_num_blocks_per_seq,
                              long long num_blocks, long long k_block_stride, long long k_token_stride,
                              long long k_head_stride, long long v_block_stride, long long v_token_stride,
                              long long v_head_stride, float scale, float k_scale, float v_scale,
                              cudaStream_t stream);

/*
 * pda_decode_slot_scales -- pda_decode with per-slot dequantisation scales.
 *
 * Source: vLLM pull request lishuoshuo-amd/vllm#3, "Details", item "Scale
 * tables": the asm kernel reads per-slot [blocks, kv_heads, block_size]
 * scales (filled there with the per-tensor scale).
 *
 *   k_scales, v_scales  fp32 [num_blocks][num_kv_heads][block_size]  read,
 *                       16-byte aligned, on the current device
 *
 * The token in slot o of block b, kv head k, dequantises as e4m3 *
 * k_scales[b][k][o] (V: v_scales[b][k][o]). Every other argument, the
 * supported set and the error behaviour are pda_decode's; tables filled with
 * one value give pda_decode's result for that per-tensor scale (up to fp32
 * rounding order). Entries of slots past a sequence's length are never used
 * (they may hold anything). Within one KV split, the largest ratio between
 * two V scales must stay below 2^15 (each probability, times its slot's V
 * scale relative to the split's first one, enters the PV product in f16
 * parts, whose range ends at 65504); the tests cover ratios of 2^14.
 * Multi-wave calls of GQA groups of at most 6 heads (4 at 128-token blocks)
 * run on the persistent kernel, whose tail pieces each take their own first
 * slot as the reference (a subset of the split: the same bound holds);
 * pda_plan_slot_scales tells which kernel a call takes.
 */
pda_status pda_decode_slot_scales(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  const float* k_scales, const float* v_scales, const int32_t* block_tables,
                                  const int32_t* seq_lens, int num_seqs, int num_heads, int num_kv_heads,
                                  int head_size, int block_size, int max_num_blocks_per_seq, float scale,
                                  cudaStream_t stream);

/*
 * pda_reshape_and_cache -- KV-cache write: quantise new keys and values to
 * e4m3 with the per-tensor scales and scatter them into the paged cache.
 *
 * Source: vLLM API page "vllm.v1.attention.backends.rocm_aiter_unified_attn",
 * RocmAiterUnifiedAttentionImpl.do_kv_cache_update, which hands key, value,
 * key_cache, value_cache, slot_mapping, k_scale and v_scale to the cache
 * writer before attention runs; the page layout is pda_decode's.
 *
 *   key, value    bf16  [num_tokens][num_kv_heads][head_size]   read
 *   k_cache       e4m3  [num_blocks][num_kv_heads][head_size/16][block_size][16]  written
 *   v_cache       e4m3  as kv_layout says (PDA_KV_NATIVE: [num_blocks][num_kv_heads]
 *                 [head_size][block_size]; PDA_KV_SHUFFLED_V: [num_blocks]
 *                 [num_kv_heads][block_size/16][head_size][16])           written
 *   slot_mapping  int64 [num_tokens]: slot = block * block_size + offset;
 *                 negative = padding (skipped)
 *
 * Token t goes to block slot/block_size, offset slot%block_size; byte d of
 * kv head k is E4M3(float(x) / scale), the IEEE binary32 quotient rounded to
 * the nearest e4m3 value (ties to even), saturating at +-448 (infinities
 * included), NaN kept. Slots >= num_blocks * block_size are not written and
 * set a code in the device status word (see pda_query_device_status).
 * Slots must be distinct (two tokens writing one slot leave either value).
 * Pointers 16-byte aligned (slot_mapping 8-byte), all on the current device.
 * Supported: head_size 128, block_size a multiple of 16 up to 128. Scales
 * must be finite and nonzero. Stream-ordered, no host sync, capturable.
 */
pda_status pda_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                                 const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_size,
                                 int block_size, long long num_blocks, float k_scale, float v_scale, int kv_layout,
                                 cudaStream_t stream);

/*
 * pda_decode_noalloc -- pda_decode for callers that cannot allocate device
 * memory. No counterpart on the pages: this is an interface convenience of
 * this library.
 *
 * pda_decode keeps its split partials in a workspace it grows with
 * cudaMallocAsync. Some callers cannot allow that: a serving process that
 * reserved all device memory for its own pool at start-up, code that must
 * not add to the device's allocation (for example under a strict memory
 * budget or an allocator that must see every byte), or a caller whose first
 * use of a shape would otherwise trigger an allocation at a bad moment. This
 * entry point computes what pda_decode computes, with the same per-unit
 * arithmetic, but always on the per-unit decode kernel with 3 CTAs per SM
 * and the split count pda_choose_splits gives for that residency; its
 * partials live in a fixed 16 MiB array compiled into the library: every
 * GPU that loads the library holds that array until the process exits. It
 * calls no cudaMalloc, cudaFree or other allocating routine. Where
 * pda_decode plans the same split count (every batch that does not fit one
 * wave of 4 CTAs per SM) the results are bitwise equal; otherwise they
 * agree to rounding.
 *
 * Arguments, layouts, supported set and ordering are pda_decode's. Limit:
 * num_seqs * num_heads * splits * 520 bytes must fit in 16 MiB (splits is
 * the split count above; a call that needs one split uses no scratch at
 * all); larger calls return PDA_ERR_NOALLOC_CAPACITY before
 * launching anything. The first call on each device (and the first after
 * pda_release) also looks up the array's device address and the device's
 * properties (no allocation); make that call outside any stream capture. All calls on a device share
 * the one array: nothing in it needs to start at zero (each call writes the
 * partials it reads), but two calls whose kernels can run at the same time
 * on the GPU (on two streams with no ordering between them, from two host
 * threads, or from two libraries' copies in one process sharing a stream
 * order they do not control) race on it and give wrong results; order them
 * on one stream or with events. Profiling events
 * (pda_set_profile_events) are not recorded by this entry point.
 */
pda_status pda_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, const int32_t* seq_lens, int num_seqs, int num_heads,
                              int num_kv_heads, int head_size, int block_size, int max_num_blocks_per_seq,
                              float scale, float k_scale, float v_scale, cudaStream_t stream);

/*
 * pda_decode_host -- pda_decode on inputs and output in host memory. No
 * counterpart on the pages (whose decode call reads device tensors): an
 * interface convenience for callers whose batch lives on the host, and the
 * end-to-end path the benchmark times.
 *
 * Host pointers (layouts as pda_decode's; none needs 16-byte alignment):
 *   out           bf16  [num_seqs][num_heads][head_size]          written
 *   q             bf16  [num_seqs][num_heads][head_size]          read
 *   k_cache       e4m3  [num_blocks][num_kv_heads][head_size/16][block_size][16]  read
 *   v_cache       e4m3  [num_blocks][num_kv_heads][head_size][block_size]          read
 *   block_tables  int32 [num_seqs][max_num_blocks_per_seq]        read
 *   seq_lens      int32 [num_seqs]                                read
 * num_blocks is the number of blocks in the cache arrays (their extent,
 * which the call copies whole).
 *
 * Before anything is enqueued the host checks every table entry a sequence
 * reads (the first ceil(seq_lens[s] / block_size) of row s) against
 * [0, num_blocks) and every length against [0, max_num_blocks_per_seq *
 * block_size]; a bad entry or length returns PDA_ERR_INVALID_ARG and nothing
 * runs. Then, on `stream`: one cudaMemcpyAsync host -> device per input into
 * a staging buffer the library keeps per (device, stream), pda_decode on the
 * staged copies, and one cudaMemcpyAsync device -> host of the output. The
 * call returns without synchronising: the caller synchronises `stream`
 * before reading `out` and keeps every input unchanged and alive until then.
 * Pinned host memory (cudaHostAlloc / cudaHostRegister) makes the copies
 * asynchronous; with pageable memory they may block the calling thread.
 *
 * The staging buffer grows with cudaMallocAsync outside stream capture;
 * growing it during capture returns PDA_ERR_WORKSPACE (make one call of the
 * largest shape first). pda_release frees it. Other errors and the supported
 * set are pda_decode's.
 */
pda_status pda_decode_host(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int32_t* seq_lens, int num_seqs, int num_heads,
                           int num_kv_heads, int head_size, int block_size, int max_num_blocks_per_seq,
                           long long num_blocks, float scale, float k_scale, float v_scale, cudaStream_t stream);

/* Static text for a status code; never NULL. */
const char* pda_status_string(int status);

/*
 * pda_choose_splits -- the split-count heuristic (pure, host only).
 *
 * Returns how many KV splits each (sequence, kv head) work unit is cut into
 * for a batch of num_seqs * num_kv_heads units with at most
 * max_num_blocks_per_seq pages of block_size tokens, on a device with
 * sm_count SMs that hold ctas_per_sm decode CTAs each. Like the pull
 * request's dispatch rule ("Claims": work units compared with the
 * compute-unit count), it compares work units with the resident CTA slots:
 * a unit is split when its K/V bytes (at max_num_blocks_per_seq pages)
 * exceed 1 MiB, or when the units fill less than one wave of slots (then up
 * to one wave), never below 256 tokens per split. Result in
 * [1, max(1, max_num_blocks_per_seq)]. Invalid arguments return 1.
 */
int pda_choose_splits(int num_seqs, int num_kv_heads, int max_num_blocks_per_seq, int block_size,
                      int sm_count, int ctas_per_sm);

/*
 * pda_plan_splits -- the split count pda_decode would use on the current
 * device for these sizes (heuristic or override). Returns < 1 on error.
 */
int pda_plan_splits(int num_seqs, int num_heads, int num_kv_heads, int max_num_blocks_per_seq,
                    int block_size);

/* Decode kernel instances (pda_plan_kernel). */
typedef enum {
  PDA_KERNEL_PER_UNIT = 0,       /* one CTA per work unit, 3 CTAs per SM, 64 KiB page ring */
  PDA_KERNEL_PER_UNIT_DENSE = 1, /* one CTA per work unit, 4 CTAs per SM, 48 KiB page ring */
  PDA_KERNEL_PERSISTENT = 2      /* one CTA per resident slot working through a queue of units */
} pda_kernel;

/*
 * pda_plan_kernel -- the decode kernel instance pda_decode (and pda_decode_ex,
 * and pda_decode_strided with token-major pages) would launch on the current
 * device for these sizes: the dense per-unit
 * instance when the planned grid fits one wave of 4 CTAs per SM, else the
 * persistent kernel. A call captured into a CUDA graph without a prior
 * pda_reserve (so with no workspace for the persistent kernel's queue) runs
 * the 3-CTA per-unit instance instead. Diagnostic; returns < 0 on error.
 */
int pda_plan_kernel(int num_seqs, int num_heads, int num_kv_heads, int max_num_blocks_per_seq, int block_size);

/*
 * pda_choose_kernel -- the planner's choice for a pda_decode call (pure,
 * host only, no device needed): for a batch of num_seqs * num_kv_heads
 * units with at most max_num_blocks_per_seq pages of block_size tokens, on a
 * device with sm_count SMs holding ctas_per_sm per-unit / persistent CTAs
 * or ctas_per_sm_dense dense per-unit CTAs each. Returns the PDA_KERNEL_*
 * instance and, when the pointers are non-NULL, stores the split count and
 * the kernels launched per call. The dense per-unit instance is chosen when
 * its grid fits one wave, else the persistent kernel (the 3-CTA per-unit
 * kernel past 2^31 units). The split count follows pda_choose_splits with
 * the chosen residency; the split override is not applied. Invalid
 * arguments return -1. pda_plan_kernel / pda_plan_splits / pda_plan_launches
 * give the same answers for the current device.
 */
int pda_choose_kernel(int num_seqs, int num_kv_heads, int max_num_blocks_per_seq, int block_size, int sm_count,
                      int ctas_per_sm, int ctas_per_sm_dense, int* num_splits, int* launches);

/*
 * pda_plan_launches -- kernels one pda_decode call launches for these sizes
 * on the current device: the decode kernel, plus the unit-order kernel when
 * the persistent kernel has more units than resident CTAs (up to 16384
 * units), plus the tail merge kernel when those units leave a partial last
 * round (units modulo resident CTAs > 0; it runs even when no unit of that
 * round is long enough to cut), plus the merge kernel when the call splits
 * (with pda_set_tail_split(0): no tail merge kernel). A one-wave per-unit
 * call of 2 to 16 splits has no merge launch: the splits of each (sequence,
 * kv head) run as one thread-block cluster and combine their results
 * through distributed shared memory. 0 for num_seqs == 0;
 * < 0 on error. Diagnostic (counts graph nodes, profiler launches).
 */
int pda_plan_launches(int num_seqs, int num_heads, int num_kv_heads, int max_num_blocks_per_seq, int block_size);

/*
 * pda_tail_pieces -- the tail-piece cut the persistent kernel makes (host
 * only; no device is needed). A call whose units overrun the resident CTAs
 * (`ctas`) by a partial last round of `tail_units` units (0 < tail_units <
 * ctas) cuts each of those units of `pages` pages (of its split) into
 * pieces: at least 256 tokens each, units under 1024 tokens whole, pieces
 * that shrink toward the end of the hand-out when tail_units >= ctas / 3,
 * else equal ones. Writes the first min(pieces, max_sizes) piece sizes in
 * pages to `sizes` (in hand-out order within the unit) and returns the
 * piece count; -1 for invalid arguments. Diagnostic (tests, tuning); no
 * counterpart in the pages (a scheduling choice, not part of what the
 * operation computes).
 */
int pda_tail_pieces(int pages, int tail_units, int ctas, int block_size, int* sizes, int max_sizes);

/*
 * pda_plan_slot_scales -- the plan pda_decode_slot_scales makes for these
 * sizes on the current device. *kernel receives PDA_KERNEL_PERSISTENT when
 * the grid is past one wave of 3 CTAs per SM and the GQA group's query rows
 * leave room for a stage's scale rows in the persistent kernel's side
 * entries (g <= 6 at 16- to 64-token blocks, g <= 4 at 128), else
 * PDA_KERNEL_PER_UNIT; *num_splits the split count; *launches the kernels
 * one call launches (the unit-order, tail merge and merge kernels as for
 * pda_decode). Any out pointer may be NULL. Returns 0, or -1 for invalid
 * sizes or a CUDA error. Diagnostic.
 */
int pda_plan_slot_scales(int num_seqs, int num_heads, int num_kv_heads, int max_num_blocks_per_seq, int block_size,
                         int* kernel, int* num_splits, int* launches);

/*
 * pda_set_split_override -- force the split count of later pda_decode calls
 * (process-wide; 0 restores the heuristic). For tests and measurements.
 * Values above the table row length are clamped at call time.
 */
void pda_set_split_override(int num_splits);

/*
 * pda_set_tail_split -- tail pieces of the persistent kernel (process-wide;
 * on by default). When a multi-wave batch hands out its units in
 * longest-first order, the units of the last, partial round (units modulo
 * resident CTAs, at most 1024) that hold at least 1024 tokens are cut into
 * pieces of at least 256 tokens, at most 8 per unit, that the CTAs done with
 * their whole units share. A tail merge kernel, launched as the decode
 * kernel's programmatic dependent, folds the pieces' (O, m, l) in piece
 * order and stores the unit's result (or the split's partial, which the
 * merge kernel then folds), so the result of such a unit is not bitwise
 * the whole unit's (it is the same softmax, within rounding). 0 turns the
 * pieces off for later calls (tests that compare kernels bit for bit,
 * measurements).
 */
void pda_set_tail_split(int enable);

/*
 * pda_set_tma_gather -- four-row TMA gathers (process-wide; on by default).
 * With 16-token blocks the persistent decode kernel copies a stage's four
 * K pages and four V pages as one tile::gather4 copy per cache, and the
 * per-slot-scale entry point (pda_decode_slot_scales) a stage's four K and
 * four V scale rows as one gather per table (larger blocks: one bulk copy
 * per scale row). 0 copies pages one bulk copy each and scale rows as
 * 16-byte cp.async pieces, for later calls. The same bytes arrive either
 * way, so results are bitwise equal; for tests and measurements. No
 * counterpart in the pages (a copy strategy, not part of what the
 * operation computes).
 */
void pda_set_tma_gather(int enable);

/*
 * pda_set_block_check -- device-side check of block ids for later decode
 * calls (process-wide). pda_decode, pda_decode_ex, pda_decode_slot_scales
 * and pda_decode_noalloc are not given the pool size, so a table entry
 * outside the pool would make them read outside k_cache / v_cache (the
 * caller's error, see pda_decode). With num_blocks > 0 their kernels check
 * every block id they read against [0, num_blocks): an id outside it sets
 * bit 64 of the device status word (pda_query_device_status) and its page is
 * read from block 0 instead, so that call's output is wrong but no read
 * leaves the pool. 0 (the default) turns the check off. pda_decode_strided
 * and pda_decode_host, which are given the pool size, bound their reads
 * themselves. For debugging and for callers that cannot vouch for their
 * tables; the check adds a compare per block id in the producer warp.
 */
void pda_set_block_check(long long num_blocks);

/*
 * pda_reserve -- size the workspace of (current device, stream) for calls up
 * to these sizes (any entry point's plan: queue words, unit order, split
 * partials), so later calls (for example under stream capture) need no
 * allocation. Stream-ordered; returns PDA_OK or PDA_ERR_CUDA.
 */
pda_status pda_reserve(int num_seqs, int num_heads, int num_kv_heads, int max_num_blocks_per_seq,
                       int block_size, cudaStream_t stream);

/*
 * pda_release -- free every workspace and staging buffer the library holds,
 * the ones that growth retired included (synchronises each device used),
 * and forget the per-device set-up (SM counts, kernel attributes, the
 * pda_decode_noalloc array's address), which the next call takes again.
 * Graphs that captured a pda_decode* or pda_decode_host call refer to freed
 * memory afterwards and must not be replayed. A cudaDeviceReset destroys
 * everything the library set up on that device: call pda_release before
 * resetting a device the library has used.
 */
pda_status pda_release(void);

/*
 * pda_workspace_info -- the workspace of (current device, stream): *bytes
 * receives its current size (0 when it has none) and *retired the number of
 * smaller buffers it replaced that are still allocated for graphs that
 * captured them. Diagnostic; host only, no synchronisation.
 */
pda_status pda_workspace_info(cudaStream_t stream, long long* bytes, int* retired);

/*
 * pda_query_device_status -- synchronise `stream`, then read and clear the
 * device status word of the current device. *code receives 0 when every
 * kernel since the last query finished normally, or a nonzero code when a
 * kernel gave up on a bounded wait, or skipped or redirected an access
 * outside the pool (a cache-write slot past the pool: bit 16; with
 * pda_set_block_check, a block id outside the pool: bit 64); the output of
 * that call is then undefined. Returns PDA_ERR_DEVICE_TIMEOUT when
 * *code != 0. Test / debug call: it blocks.
 */
pda_status pda_query_device_status(cudaStream_t stream, int* code);

/*
 * pda_set_profile_events -- when both events are non-NULL, later pda_decode
 * calls record `before` immediately before and `after` immediately after the
 * split-KV decode kernel on their stream (capturable); with the persistent
 * kernel's unit-order kernel, `before` precedes that one too (the two run
 * overlapped), and with its tail merge kernel, `after` follows that one too
 * (a programmatic dependent of the decode kernel). The split merge kernel
 * stays outside. NULL, NULL turns it off. Process-wide; for measurement only.
 */
void pda_set_profile_events(cudaEvent_t before, cudaEvent_t after);

/*
 * pda_test_bounded_wait -- launch one CTA that waits on a barrier nothing
 * will complete, with a limit of timeout_us microseconds, on `stream`. The
 * kernel gives up, records PDA timeout code in the device status word and
 * returns (no trap, no fault); pda_query_device_status then reports it.
 * Exercises the bounded-wait error path of the decode kernel's barriers.
 * timeout_us must be in [1, 2000000].
 */
pda_status pda_test_bounded_wait(int timeout_us, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PDA_H_ */
