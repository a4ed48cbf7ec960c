/*
 * pagedkv.h — C ABI of the GB300 paged decode-attention library (libpagedkv.so).
 *
 * The library implements the decode-time hot path of a blocked ("paged") KV
 * cache as described by:
 *   - "AI大模型推理速度翻倍，Colossal-Inference开源发布", sections
 *     分块式KV缓存 (BlockedKeyValueCache), KV缓存量化 (KVCache Quant),
 *     投机采样 (Speculative decoding) and 分页注意力算法 (PagedAttention);
 *   - "AI 大模型推理优化技术详解", sections 2.1.2 Paged Attention (block size 16,
 *     logical-to-physical block table), 2.2.1 Flash Attention (softmax reduced
 *     without the whole row) and 2.2.2 GQA (query-head groups sharing one KV head);
 *   - "TACO-LLM 如何实现降本增效?", section 3 (TurboAttention: paged + flash
 *     attention for long generation) — the split-KV path serves that case.
 *
 * Conventions for every call
 *   - All pointers are DEVICE pointers unless stated otherwise. The caller owns
 *     every buffer; the library allocates no device memory and keeps no state
 *     besides a per-device cache of device properties and kernel attributes,
 *     filled on first use. cudaDeviceReset discards what that cache describes:
 *     do not call the library on a device after resetting it in the same process.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *     asynchronous: they enqueue kernels and return.
 *   - Return value: PKV_OK (0) or a negative pkv_status. Arguments are checked on
 *     the host before anything is launched; on error nothing is launched.
 *     Nothing throws across this boundary.
 *   - Problems only the device can see (an out-of-range block id or slot, a
 *     context length outside [q_per_seq, max_blocks_per_seq*16]) are reported by
 *     OR-ing PKV_DEV_* bits into `*device_status` when that pointer is not NULL.
 *     The library never clears it; the caller zeroes it when it wants a fresh
 *     reading. Such inputs never fault: a bad block reads as zeros, a bad slot is
 *     skipped.
 *
 * Cache layout (our own choice; the pages' [blocks, heads, head/x, block, x] key
 * layout is prior art, not used): K and V caches are separate arrays, each
 *     [num_blocks][num_kv_heads][block_size = 16][head_size]
 * row-major, elements fp16, bf16 or E5M2 (one byte). One (block, head) tile is
 * 16*head_size contiguous elements (4 KiB for fp16 at head_size 128), which the
 * decode kernel moves with one tensor-memory-accelerator copy. Token p of a
 * sequence lives in physical block block_tables[s][p / 16] at offset p % 16; its
 * slot number is block * 16 + offset.
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. The pages' FP8 cache is E5M2 (KVCache Quant section). */
typedef enum {
  PKV_FP16 = 0,
  PKV_BF16 = 1,
  PKV_FP8_E5M2 = 2,
  PKV_INT8 = 3      /* int8 codes with float32 row scales: see pkv_kv_cache_write_int8 */
} pkv_dtype;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARGUMENT = -1,   /* null pointer, non-positive size, misaligned pointer */
  PKV_ERR_UNSUPPORTED = -2,        /* shape or dtype combination this build does not handle */
  PKV_ERR_WORKSPACE_TOO_SMALL = -3,
  PKV_ERR_CUDA = -4,               /* a CUDA runtime call failed (launch, attribute, ...) */
  PKV_ERR_NO_DEVICE = -5,
  PKV_ERR_OUT_OF_BLOCKS = -6      /* block allocator: the pool cannot supply the blocks asked for */
} pkv_status;

/* Device-side status bits OR-ed into *device_status. */
#define PKV_DEV_BAD_SLOT   0x1  /* kv_cache_write: slot outside [-1, num_blocks*16) */
#define PKV_DEV_BAD_BLOCK  0x2  /* decode: block id outside [0, num_blocks); read as zeros */
#define PKV_DEV_BAD_CTX    0x4  /* decode: context_len < q_per_seq or > max_blocks_per_seq*16 */
#define PKV_DEV_TIMEOUT    0x8  /* decode: a pipeline wait gave up (never expected) */

/* Description of one K/V cache pair. block_size must be 16 (the pages' default,
 * 2.1.2 Paged Attention); head_size 64 or 128. */
typedef struct {
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_size;
} pkv_cache_desc;

/*
 * pkv_kv_cache_write — scatter new tokens into the cache ("kernel1" of the
 * KVCache Quant section: the writer casts fp16 to FP8 when the cache is E5M2).
 *
 *   key, value    [num_tokens][num_kv_heads][head_size], contiguous, src_dtype
 *                 (PKV_FP16 or PKV_BF16). 16-byte aligned.
 *   slot_mapping  [num_tokens] int32: physical slot (block*16 + offset) of each
 *                 token; -1 = skip the token. Other out-of-range values are
 *                 skipped and flagged PKV_DEV_BAD_SLOT.
 *   k_cache, v_cache  caches in the layout above, element type kv_dtype, 16-byte aligned.
 *   Allowed (src_dtype, kv_dtype): (FP16, FP16), (BF16, BF16), (FP16, FP8_E5M2).
 *   FP8 cast: round to nearest even; |x| > 57344 and +-inf saturate to +-57344;
 *   NaN -> 0x7E | sign. fp16/bf16 caches are plain copies.
 *   Two tokens mapped to the same slot race; the result is then unspecified.
 *   num_tokens == 0 is a no-op returning PKV_OK.
 */
int pkv_kv_cache_write(const void* key, const void* value, pkv_dtype src_dtype,
                       int32_t num_tokens, const int32_t* slot_mapping,
                       void* k_cache, void* v_cache, pkv_dtype kv_dtype,
                       const pkv_cache_desc* cache, int32_t* device_status, void* stream);

/*
 * pkv_decode_workspace_bytes — size of the scratch buffer paged attention needs
 * on the CURRENT device for this problem shape (split-KV partial results and a
 * per-(sequence, KV head) counter of finished pieces). It depends only on the arguments and the
 * device's multiprocessor count; any buffer at least this large works, and it
 * needs no initialisation. Returns 0 on invalid arguments.
 */
size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t q_per_seq,
                                  const pkv_cache_desc* cache);

/*
 * pkv_paged_attention_decode — decode attention over the blocked cache
 * ("kernel2" of the KVCache Quant section, the PagedAttention section's decode
 * kernel, with the GQA grouping of 2.2.2 and the multi-token verify of the
 * speculative-decoding section).
 *
 *   out, q        [num_seqs * q_per_seq][num_q_heads][head_size], contiguous.
 *                 Row s*q_per_seq + j is query token j of sequence s. Element
 *                 type: bf16 when kv_dtype is PKV_BF16, else fp16. 16-byte aligned.
 *   block_tables  [num_seqs][max_blocks_per_seq] int32 physical block ids.
 *   context_lens  [num_seqs] int32: cached tokens of each sequence INCLUDING its
 *                 q_per_seq query tokens, which are its last q_per_seq positions.
 *   scale         softmax scale (typically 1/sqrt(head_size)).
 *   workspace     device scratch of at least pkv_decode_workspace_bytes(...)
 *                 bytes, 16-byte aligned; contents need no initialisation. Two
 *                 calls in flight at the same time must not share a workspace.
 *                 A call may be captured in a CUDA graph and replayed: every
 *                 launch leaves the workspace's counters clear when it completes.
 *                 The counters are tagged with a per-call number (a scrambled
 *                 call count that does not repeat within 2^32 calls), so counters
 *                 left by an earlier call read as clear, and other data left in
 *                 the buffer matches a tag only by a 2^-32 chance per 8-byte word
 *                 (zero a buffer that held other data once if that matters). A
 *                 replayed graph reuses its call's number, so after a launch that
 *                 reported PKV_DEV_TIMEOUT (its counters may be left part-way)
 *                 zero the workspace (e.g. cudaMemsetAsync) before replaying it.
 *
 *   For each sequence s, query head hq (KV head h = hq / (num_q_heads/num_kv_heads))
 *   and query token j, with L = context_lens[s] - q_per_seq + j + 1:
 *       out[s,j,hq,:] = sum_{p<L} softmax_p(scale * q[s,j,hq,:] . K[s,p,h,:]) * V[s,p,h,:]
 *   accumulated in fp32 on tensor cores (P in the query dtype), rounded to the
 *   output dtype once. Requires num_q_heads % num_kv_heads == 0 and
 *   (num_q_heads/num_kv_heads) * q_per_seq <= 64.
 */
int pkv_paged_attention_decode(void* out, const void* q, int32_t num_seqs,
                               int32_t num_q_heads, int32_t q_per_seq,
                               const void* k_cache, const void* v_cache, pkv_dtype kv_dtype,
                               const pkv_cache_desc* cache, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* context_lens,
                               float scale, void* workspace, size_t workspace_bytes,
                               int32_t* device_status, void* stream);

/*
 * pkv_paged_attention_decode_varlen — the same attention for a batch whose
 * sequences carry different numbers of query tokens: plain decode (1 token),
 * speculative verify (several draft tokens) and short prefill chunks mixed in one
 * launch, with the tokens packed without padding ("nopadding" 1-D input of the
 * Continuous Batching section of the Colossal-Inference release page).
 *
 *   cu_q_lens     [num_seqs + 1] int32, device: sequence s owns query/output rows
 *                 cu_q_lens[s] .. cu_q_lens[s+1]-1 (cu_q_lens[0] = 0); its
 *                 n_s = cu_q_lens[s+1] - cu_q_lens[s] must be in [1, max_q_per_seq]
 *                 and its rows must lie in [0, num_q_rows). A sequence that breaks
 *                 either rule gets no output rows, reads none of q, and sets
 *                 PKV_DEV_BAD_CTX.
 *   num_q_rows    rows of q and out (normally cu_q_lens[num_seqs]); >= 1 when
 *                 num_seqs > 0.
 *   out, q        [num_q_rows][num_q_heads][head_size].
 *   max_q_per_seq sizes the per-unit row capacity: (num_q_heads/num_kv_heads) *
 *                 max_q_per_seq <= 64; pkv_decode_workspace_bytes(num_seqs,
 *                 num_q_heads, max_q_per_seq, cache) sizes the workspace.
 *   Query token j of sequence s sees positions p <= context_lens[s] - n_s + j.
 *   Everything else is as for pkv_paged_attention_decode.
 */
int pkv_paged_attention_decode_varlen(void* out, const void* q, const int32_t* cu_q_lens,
                                      int32_t num_q_rows, int32_t num_seqs, int32_t num_q_heads,
                                      int32_t max_q_per_seq,
                                      const void* k_cache, const void* v_cache, pkv_dtype kv_dtype,
                                      const pkv_cache_desc* cache, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* context_lens,
                                      float scale, void* workspace, size_t workspace_bytes,
                                      int32_t* device_status, void* stream);

/*
 * pkv_paged_attention_decode_tree — speculative verify of a token TREE: the n_s
 * query tokens of a sequence are candidate continuations organised as a tree
 * (the token-tree verification of FlexFlow Serve, nxhydt survey of inference
 * frameworks, section FlexFlow), and each query token may attend only to the
 * context before the drafts and to its own ancestors.
 *
 *   tree_masks    [num_q_rows] uint64, device, 8-byte aligned: bit i of the
 *                 mask of query token j of sequence s is set when j may attend to
 *                 draft token i, i.e. position context_lens[s] - n_s + i. A token
 *                 normally sees itself (bit j). A row that sees no position gets
 *                 output 0. The causal chain is mask (2 << j) - 1.
 *   cu_q_lens     may be NULL: then every sequence has max_q_per_seq tokens
 *                 (rows s*max_q_per_seq + j) and num_q_rows must be at least
 *                 num_seqs * max_q_per_seq; otherwise as for the _varlen call.
 *   num_q_rows    rows of q, out and tree_masks.
 *   max_q_per_seq <= 64 (one mask bit per draft token).
 *   Everything else is as for pkv_paged_attention_decode_varlen.
 */
int pkv_paged_attention_decode_tree(void* out, const void* q, const int32_t* cu_q_lens,
                                    const uint64_t* tree_masks, int32_t num_q_rows, int32_t num_seqs,
                                    int32_t num_q_heads, int32_t max_q_per_seq,
                                    const void* k_cache, const void* v_cache, pkv_dtype kv_dtype,
                                    const pkv_cache_desc* cache, const int32_t* block_tables,
                                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                                    float scale, void* workspace, size_t workspace_bytes,
                                    int32_t* device_status, void* stream);

/*
 * pkv_paged_attention_decode_noalloc — the same decode attention as
 * pkv_paged_attention_decode, for callers that cannot allocate device memory
 * when they run it (for example code running inside a custom allocator's
 * callbacks, or engines that hand the whole device to the KV pool up front and
 * forbid later cudaMalloc calls). The pages describe no such entry point; it
 * is a deployment convenience of this library.
 *
 *   Arguments, layouts and results are those of pkv_paged_attention_decode,
 *   without the workspace: the split-KV scratch comes from a buffer of
 *   PKV_NOALLOC_SCRATCH_BYTES built into the library. Inputs and outputs are
 *   still the caller's. The call itself allocates nothing.
 *   - Limit: a problem whose pkv_decode_workspace_bytes(...) exceeds
 *     PKV_NOALLOC_SCRATCH_BYTES is rejected with PKV_ERR_WORKSPACE_TOO_SMALL
 *     before anything is launched (use pkv_paged_attention_decode with your own
 *     workspace for it). Arguments the regular entry point refuses get the
 *     status it returns for them.
 *   - The buffer occupies PKV_NOALLOC_SCRATCH_BYTES of device memory on every
 *     device where the library's module holding it is loaded, until the process
 *     exits.
 *   - The first call on a device looks up the buffer's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call shares the one buffer and keeps the previous call's contents
 *     in it. Partial results are rewritten by each call; the split-KV counters
 *     start at zero when the module loads and are tagged with each call's
 *     number, so a counter an earlier call left behind (even one that reported
 *     PKV_DEV_TIMEOUT) reads as clear. Calls whose kernels overlap on the GPU
 *     (different streams, or concurrent host threads) race on it; serialise them.
 *   - The address is looked up once per device and kept (see cudaDeviceReset
 *     above).
 */
#define PKV_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

int pkv_paged_attention_decode_noalloc(void* out, const void* q, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t q_per_seq,
                                       const void* k_cache, const void* v_cache,
                                       pkv_dtype kv_dtype, const pkv_cache_desc* cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, float scale,
                                       int32_t* device_status, void* stream);

/* ==== INT8 KV cache ===========================================================
 *
 * The inference-framework survey lists "KV Cache INT8 量化" for LMDeploy
 * without a codec; this one is symmetric per (token, KV head) row:
 *   scale = max|x| / 127 rounded up to the nearest fp16 value,
 *   code = round-half-even(x / scale) clamped to [-127, 127],
 * both divisions in IEEE fp32; an all-zero row has scale 0 and codes 0; an
 * element's value is code * scale. (An fp16-valued scale folds exactly into the
 * fp16 weights of the attention's P V product.)
 *
 * Caches: one byte per element, [num_blocks][num_kv_heads][16][head_size],
 * each code stored in offset binary: byte = code + 128 (1..255; the decode
 * kernel widens it to fp16 with one byte permute); scales: one float32
 * array [num_blocks][num_kv_heads][2][16]: the 16 K row scales of a (block,
 * KV head) tile, then its 16 V row scales (so one 128-byte copy brings both),
 * all 16-byte aligned.
 * key/value: fp16 [num_tokens][num_kv_heads][head_size]. Slots as in
 * pkv_kv_cache_write (-1 skipped, other out-of-range slots skipped and flagged). */
int pkv_kv_cache_write_int8(const void* key, const void* value, int32_t num_tokens,
                            const int32_t* slot_mapping, void* k_cache, void* v_cache,
                            float* scales, const pkv_cache_desc* cache,
                            int32_t* device_status, void* stream);

/* pkv_paged_attention_decode over an INT8 cache (q and out fp16): each token's
 * score is scaled by its K row scale and its probability by its V row scale.
 * Workspace as for pkv_paged_attention_decode (pkv_decode_workspace_bytes). */
int pkv_paged_attention_decode_int8(void* out, const void* q, int32_t num_seqs, int32_t num_q_heads,
                                    int32_t q_per_seq, const void* k_cache, const void* v_cache,
                                    const float* scales,
                                    const pkv_cache_desc* cache, const int32_t* block_tables,
                                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                                    float scale, void* workspace, size_t workspace_bytes,
                                    int32_t* device_status, void* stream);

/* The mixed-batch and token-tree calls over an INT8 cache: arguments as for
 * pkv_paged_attention_decode_varlen and pkv_paged_attention_decode_tree (q and
 * out fp16), plus the cache's row scales as for pkv_paged_attention_decode_int8.
 * A batch that mixes plain decode rows and verify rows ("nopadding" packed
 * tokens, Continuous Batching section of the Colossal-Inference release page)
 * over the INT8 cache of the LMDeploy section of the inference-framework survey. */
int pkv_paged_attention_decode_int8_varlen(void* out, const void* q, const int32_t* cu_q_lens,
                                           int32_t num_q_rows, int32_t num_seqs, int32_t num_q_heads,
                                           int32_t max_q_per_seq, const void* k_cache, const void* v_cache,
                                           const float* scales, const pkv_cache_desc* cache,
                                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                                           const int32_t* context_lens, float scale, void* workspace,
                                           size_t workspace_bytes, int32_t* device_status, void* stream);
int pkv_paged_attention_decode_int8_tree(void* out, const void* q, const int32_t* cu_q_lens,
                                         const uint64_t* tree_masks, int32_t num_q_rows, int32_t num_seqs,
                                         int32_t num_q_heads, int32_t max_q_per_seq, const void* k_cache,
                                         const void* v_cache, const float* scales, const pkv_cache_desc* cache,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* context_lens, float scale, void* workspace,
                                         size_t workspace_bytes, int32_t* device_status, void* stream);

/*
 * pkv_paged_attention_decode_chunked — decode attention for a batch whose sequences
 * may carry ANY number of query tokens: prefill chunks beside decode and verify
 * tokens, packed without padding (the mixed batch of the Continuous Batching
 * section of the Colossal-Inference release page), with the per-sequence counts
 * and lengths given in HOST memory, as a scheduler holds them.
 *
 *   host_q_lens       [num_seqs] int32, host: n_s >= 1 query tokens of sequence s.
 *                     Its rows of q / out are cu_s .. cu_s + n_s - 1 with
 *                     cu_s = n_0 + ... + n_{s-1}.
 *   host_context_lens [num_seqs] int32, host: ctx_s >= n_s cached tokens including
 *                     the query tokens; query token j sees positions
 *                     p <= ctx_s - n_s + j (causal over the whole chunk).
 *   out, q            [n_0 + ... + n_{S-1}][num_q_heads][head_size], device.
 *   scales            an INT8 cache's row scales (as for
 *                     pkv_paged_attention_decode_int8), else NULL.
 *   workspace         device, 256-byte aligned, at least
 *                     pkv_decode_chunked_workspace_bytes(host_q_lens, num_seqs,
 *                     num_q_heads, max_blocks_per_seq, cache) bytes; owned by the
 *                     caller, reusable by the next call on the same stream.
 *   Everything else is as for pkv_paged_attention_decode_varlen.
 * A sequence's tokens run as row tiles of 64 / (num_q_heads / num_kv_heads) tokens
 * (the decode kernels' unit; fewer when no sequence has that many, so a batch of
 * plain decodes runs as it would through the _varlen call); each tile re-reads
 * the blocks its tokens see, so a
 * long chunk costs about (tiles) reads of its context: correct, not tuned for
 * prefill. The call reads the host arrays when it is made and passes the tiles'
 * lengths to a small setup kernel on `stream` as launch parameters (no host
 * synchronisation); the setup kernel writes them into the workspace and copies
 * each tile's block-table row there. The call may be captured in a CUDA graph,
 * which then replays the captured counts and lengths. Returns
 * PKV_ERR_INVALID_ARGUMENT for n_s < 1,
 * ctx_s < n_s or a missing array; other device-side problems are flagged in
 * device_status as for the _varlen call.
 */
size_t pkv_decode_chunked_workspace_bytes(const int32_t* host_q_lens, int32_t num_seqs, int32_t num_q_heads,
                                          int32_t max_blocks_per_seq, const pkv_cache_desc* cache);
int pkv_paged_attention_decode_chunked(void* out, const void* q, const int32_t* host_q_lens,
                                       const int32_t* host_context_lens, int32_t num_seqs, int32_t num_q_heads,
                                       const void* k_cache, const void* v_cache, const float* scales,
                                       pkv_dtype kv_dtype, const pkv_cache_desc* cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq, float scale,
                                       void* workspace, size_t workspace_bytes, int32_t* device_status,
                                       void* stream);

/*
 * pkv_selftest_bounded_wait — exercises, on the device, the bounded wait every
 * decode kernel puts on its pipeline barriers: one thread waits on an mbarrier
 * phase that nothing completes with a limit of limit_ns (1 .. 2e9 ns), gives up,
 * raises its CTA's abort flag and ORs PKV_DEV_TIMEOUT into *device_status; a
 * second thread, waiting with the decode kernels' own 2 s limit, leaves as soon
 * as it sees the flag. device_elapsed_ns[0..1] (device, 8-byte aligned) receive
 * the two waits' durations. Nothing faults or hangs; the context stays usable.
 * Returns PKV_ERR_INVALID_ARGUMENT for a missing or misaligned pointer or a limit
 * outside the range.
 */
int pkv_selftest_bounded_wait(int32_t* device_status, uint64_t limit_ns, unsigned long long* device_elapsed_ns,
                              void* stream);

/* ==== Block pool (host side) =================================================
 *
 * "AI 大模型推理优化技术详解", 2.1.2 Paged Attention: each sequence's KV cache is
 * a list of fixed-size blocks; a table maps its logical blocks to physical
 * blocks of a pool allocated up front; several logical blocks may map to one
 * physical block, whose reference count says how many do, and a block whose
 * count drops to 0 returns to the pool. "TACO-LLM 如何实现降本增效?",
 * 2、使用 Prefix Cache 技术降低 TTFT: the KV of earlier prompts is kept in a prefix
 * tree so a new prompt's matching prefix is looked up instead of recomputed.
 *
 * pkv_allocator manages the block ids of one pool of num_blocks blocks of 16
 * tokens (the caches themselves stay with the caller). It is plain host code,
 * not thread-safe (one owner thread), with deterministic choices:
 *   - a new block is the lowest-numbered free block;
 *   - sequences are identified by caller-chosen 64-bit ids;
 *   - fork gives the child the parent's block list (every block's count + 1);
 *   - appending to a sequence whose last block is shared (count > 1) first
 *     replaces that block by a fresh one and reports the pair (copy-on-write);
 *     the caller copies the block (pkv_copy_blocks) before writing new tokens;
 *   - the prefix cache is a tree of full blocks keyed by (parent block, the 16
 *     token ids); it holds one reference to each cached block; when the pool
 *     has no free block, the least recently used cached leaf that nothing else
 *     references is evicted and reused.
 * Every call either succeeds or leaves the allocator unchanged. */
typedef struct pkv_allocator pkv_allocator;

/* A new allocator over blocks 0 .. num_blocks-1, all free. NULL if num_blocks
 * is not in [1, 2^26] or memory runs out. */
pkv_allocator* pkv_allocator_create(int32_t num_blocks);
void pkv_allocator_destroy(pkv_allocator* a);

/* Blocks not referenced by anything. Cached blocks that only the prefix cache
 * references are not counted (pkv_allocator_evictable counts them). */
int32_t pkv_allocator_free_blocks(const pkv_allocator* a);
int32_t pkv_allocator_evictable(const pkv_allocator* a);
/* References to a block (sequences + the prefix cache); -1 if out of range. */
int32_t pkv_allocator_refcount(const pkv_allocator* a, int32_t block);

/* A new empty sequence. PKV_ERR_INVALID_ARGUMENT if the id exists. */
int pkv_seq_add(pkv_allocator* a, int64_t seq);
/* A new sequence sharing all of parent's blocks and its length. */
int pkv_seq_fork(pkv_allocator* a, int64_t parent, int64_t child);
/* Drops the sequence; its blocks lose one reference each. */
int pkv_seq_release(pkv_allocator* a, int64_t seq);
/* Tokens in the sequence, or -1 if unknown. */
int32_t pkv_seq_length(const pkv_allocator* a, int64_t seq);
/* Writes min(capacity, blocks) block ids of the sequence (its block-table row)
 * to out and returns the sequence's block count, or a negative status. */
int32_t pkv_seq_block_table(const pkv_allocator* a, int64_t seq, int32_t* out, int32_t capacity);

/* Reserves n new tokens at the end of the sequence and writes their slots
 * (block * 16 + offset, n of them) to slots. If the sequence's last block was
 * shared and receives tokens, it is replaced by a new block first: the pair is
 * written to copy_src[0] / copy_dst[0] and *num_copies = 1 (else 0); copy_src
 * and copy_dst must hold one entry. PKV_ERR_OUT_OF_BLOCKS if the pool (free and
 * evictable blocks) is too small, with nothing changed. */
int pkv_seq_append(pkv_allocator* a, int64_t seq, int32_t n, int32_t* slots, int32_t* copy_src,
                   int32_t* copy_dst, int32_t* num_copies);

/* Prefix cache. pkv_prefix_insert caches the sequence's full blocks holding its
 * first n tokens (token ids in tokens[0..n)), under the chain of their
 * contents; returns the number of blocks newly cached, or a negative status.
 * pkv_seq_add_cached creates a sequence whose first blocks are the cached
 * blocks matching the longest prefix of tokens[0..n) in whole blocks (each
 * gains a reference) and writes the number of tokens they hold to
 * *cached_tokens; the caller appends the rest. */
int32_t pkv_prefix_insert(pkv_allocator* a, int64_t seq, const int32_t* tokens, int32_t n);
int pkv_seq_add_cached(pkv_allocator* a, int64_t seq, const int32_t* tokens, int32_t n,
                       int32_t* cached_tokens);

/* ==== Block copy (device) ===================================================
 * For i < n: physical block dst[i] of both caches becomes a copy of block
 * src[i] (every head's 16 rows), and for an INT8 cache (kv_dtype PKV_INT8) so do
 * the block's row scales in `scales` ([num_blocks][num_kv_heads][2][16] floats,
 * 16-byte aligned; NULL for every other cache). src and dst are DEVICE int32
 * arrays; ids out of range are skipped and set PKV_DEV_BAD_BLOCK. The pairs
 * must not overlap in a way that reads a block after it was written in the same
 * call. Asynchronous on stream. */
int pkv_copy_blocks(void* k_cache, void* v_cache, float* scales, pkv_dtype kv_dtype,
                    const pkv_cache_desc* cache, const int32_t* src, const int32_t* dst, int32_t n,
                    int32_t* device_status, void* stream);

/* Static description of a status code. Never NULL. */
const char* pkv_error_string(int code);

/* Library version (major*10000 + minor*100 + patch). */
int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
