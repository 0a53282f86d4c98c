/*
 * pkv.h -- C ABI of libpkv: attention decode over a paged KV cache on
 * NVIDIA GB300 (sm_103a).
 *
 * A request's logically contiguous K/V history lives in fixed-size physical
 * blocks of `block_size` token rows scattered through one pool; a per-request
 * block table maps logical block j to a physical block id, and the last block
 * holds a valid-row tail ("M5.3 - KV Memory Layout and Exact Reuse", 0x03A,
 * 0x03C, 0x0A; "7. Memory Management and Local Model State", "Logical tokens,
 * physical blocks").
 *
 * CACHE LAYOUT.  One layer; K and V are separate device tensors with the
 * declared row-major axis order [num_blocks, block_size, num_kv_heads,
 * head_dim] (the token-major order of the checked address trace in M5.3
 * 0x03F, without its layer axis; strides follow 0x03E).  Element (b, o, h, c)
 * sits at ((b * block_size + o) * num_kv_heads + h) * head_dim + c.  All
 * offsets are computed in 64-bit integers ("Cache Concepts: Prefix Matching
 * vs. Storage": widen page ids to int64 before multiplying by pool strides).
 *
 * CONVENTIONS (every call).
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *     caller allocates and owns all device memory.  The library allocates
 *     no device memory at run time.  Its state between calls: one device
 *     error word per device (see pkv_get_device_error); the fixed scratch
 *     array that pkv_paged_attention_decode_static alone uses (a static
 *     device array, PKV_STATIC_SCRATCH_BYTES on every device that loads the
 *     library); and a host-side cache of up to 64 encoded TMA tensor maps,
 *     keyed by every argument of the encoding (base address, shape, strides,
 *     box, swizzle), so a hit returns the map a fresh encoding would give.
 *   - Every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *     default stream) and returns after enqueuing its kernels.
 *   - Arguments are validated on the host before any launch; a rejected call
 *     launches nothing and returns PKV_ERR_INVALID_ARG or PKV_ERR_UNSUPPORTED.
 *   - Device data the host cannot see (slot ids, block ids, lengths) is
 *     checked by the kernels: an out-of-range item sets a bit of the device
 *     error word and is skipped.  No kernel traps, asserts or waits without a
 *     time limit.
 *   - dtype is PKV_F32, PKV_BF16 or PKV_MXFP8.  With PKV_F32 or PKV_BF16,
 *     q, k, v, caches and out share it; with PKV_MXFP8 (quantized pools,
 *     below) the caches are MXFP8 and q, k, v and out are bf16.  Attention
 *     arithmetic is fp32 (accumulators, softmax state) whatever the storage
 *     type; bf16 results are rounded to nearest even.
 *   - MXFP8 POOLS.  "M5.3 - KV Memory Layout and Exact Reuse" (0x0BB) names
 *     quantized K/V a cache-ABI field, and TokenSpeed keeps MXFP8 KV scale
 *     planes beside the element planes; this library's schema: each K (or V)
 *     cache buffer holds the element plane, OCP FP8 E4M3 codes laid out
 *     [num_blocks, block_size, num_kv_heads, head_dim] as above, followed at
 *     byte offset num_blocks * block_size * num_kv_heads * head_dim by the
 *     scale plane [num_blocks, num_kv_heads, block_size, head_dim / 32] of
 *     E8M0 bytes s (the value 2^(s - 127)).  Scale byte (b, h, o, j) scales
 *     elements (b, o, h, 32 j .. 32 j + 31): element = code value * scale.
 *     kv_append quantizes: each 32-element group takes the smallest power of
 *     two X with max |x| / X <= 448 (no element saturates), and each element
 *     the E4M3 code nearest x / X (ties to even).  The scale plane is
 *     head-major within a block, so an MXFP8 pool cannot be read through
 *     tables expanded to smaller kernel blocks.  Supported by kv_append,
 *     kv_block_copy and the decode: on the CUDA cores for head_dim 64 or 128
 *     and Hq / Hkv <= 4, on the tensor cores (tiles widened to bf16 in shared
 *     memory) for head_dim 128 and Hq / Hkv = 8 with block_size 16, 32, 64,
 *     128 or 256; other group sizes return PKV_ERR_UNSUPPORTED.  The
 *     shared-prefix kernel and the chunk-first phase take bf16 only (a tree
 *     over MXFP8 pools runs sequence-first).
 *   - Pointers to the caches, q, k, v and out must be 16-byte aligned.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,  /* bad pointer, size, shape or workspace        */
  PKV_ERR_UNSUPPORTED = 2,  /* valid but not compiled (head_dim, group ...) */
  PKV_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed          */
  PKV_ERR_DEVICE = 4,       /* pkv_get_device_error found a device-side error */
  PKV_ERR_CAPACITY = 5      /* needs more than the fixed static scratch array */
} pkv_status;

typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_MXFP8 = 2 } pkv_dtype;

/* Bits of the device error word. */
#define PKV_DEVERR_SLOT 1u     /* a slot id >= num_blocks * block_size          */
#define PKV_DEVERR_BLOCK 2u    /* a block id outside [0, num_blocks)             */
#define PKV_DEVERR_LENGTH 4u   /* a length < 0 or beyond its block table row     */
#define PKV_DEVERR_TIMEOUT 8u  /* a bounded wait inside a kernel ran out         */

/* Shape of one paged K/V pool (host struct, passed by pointer). */
typedef struct {
  int64_t num_blocks;   /* physical blocks in the pool, >= 1                   */
  int32_t block_size;   /* token rows per block (P)                            */
  int32_t num_kv_heads; /* KV heads per token row (Hkv)                        */
  int32_t head_dim;     /* elements per head (D)                               */
  int32_t dtype;        /* pkv_dtype                                           */
} pkv_cache_desc;

/* Write new token rows into their slots (K/V append scatter).
 *   k, v:          [num_tokens, Hkv, D] rows to write.
 *   slot_mapping:  int64 [num_tokens]; row i goes to slot s = slot_mapping[i],
 *                  i.e. block s / P, offset s % P.  s < 0 skips the row (the
 *                  -1 skip sentinel of "Cache Concepts: Prefix Matching vs.
 *                  Storage"); s >= num_blocks * P sets PKV_DEVERR_SLOT and
 *                  skips it.  Slots must be distinct (one writer per slot).
 * The slot invariant table[req, pos // P] * P + pos % P and the append paths
 * follow M5.3 0x03D and 0x04E.  Any block_size >= 1; Hkv * D * elem must be a
 * multiple of 16 bytes.  Result is bit-exact (a byte copy). */
pkv_status pkv_kv_append(const pkv_cache_desc* cache, void* k_cache,
                         void* v_cache, const void* k, const void* v,
                         const int64_t* slot_mapping, int64_t num_tokens,
                         void* stream);

/* Copy-on-write block copy (M5.3 0x04C, 0x05A; the fused block-copy kernel of
 * PagedAttention): for each pair i, the whole block src = pairs[2i] of K and V
 * is copied to block dst = pairs[2i + 1].
 *   src_dst_pairs: int64 [num_pairs, 2].  Destinations must be pairwise
 *                  distinct and no destination may also be a source in the
 *                  same call (pairs run in parallel); ids outside the pool
 *                  set PKV_DEVERR_BLOCK and the pair is skipped.
 * Bit-exact. */
pkv_status pkv_kv_block_copy(const pkv_cache_desc* cache, void* k_cache,
                             void* v_cache, const int64_t* src_dst_pairs,
                             int64_t num_pairs, void* stream);

/* Split allocator blocks for the kernel (M5.3 0x0AC).  A pool whose
 * allocator blocks hold P_a = q * P_k token rows is, byte for byte, a pool of
 * q * num_blocks kernel blocks of P_k rows: [NB, P_a, Hkv, D] and
 * [q * NB, P_k, Hkv, D] are the same array, and allocator block a is kernel
 * blocks a q, a q + 1, ..., a q + q - 1.  This writes the kernel-visible
 * tables:
 *   out[r, c * q + j] = tables[r, c] * q + j     (j = 0 .. q - 1),
 * with a padding entry (< 0) becoming q entries of -1.  Slot ids are the same
 * in both views, so kv_append needs no change; decode the view with
 * cache->block_size = P_k and num_blocks = q * NB.
 *   tables: int32 [num_seqs, max_blocks] (device).
 *   out:    int32 [num_seqs, max_blocks * q] (device), caller-owned.
 *   alloc_block_size, kernel_block_size: P_a and P_k.  P_k must divide P_a:
 *     the reverse direction would need several separately allocated blocks to
 *     form one kernel block, so it is PKV_ERR_INVALID_ARG.
 * An id whose expansion passes INT32_MAX sets PKV_DEVERR_BLOCK and is written
 * as -1.  Bit-exact. */
pkv_status pkv_expand_block_tables(const int32_t* tables, int32_t num_seqs,
                                   int32_t max_blocks, int32_t alloc_block_size,
                                   int32_t kernel_block_size, int32_t* out,
                                   void* stream);

/* Bytes of device workspace pkv_paged_attention_decode needs for these sizes
 * and partition_size (see below); 0 for unsupported or invalid sizes.  It
 * depends on the device (its SM count), so query it with the device current. */
size_t pkv_decode_workspace_bytes(const pkv_cache_desc* cache, int32_t num_seqs,
                                  int32_t num_q_heads,
                                  int32_t max_blocks_per_seq,
                                  int32_t partition_size);

/* CTAs the decode's main kernel launches for these sizes and partition_size
 * (one wave of resident CTAs for partition_size 0); 0 for unsupported or
 * invalid sizes. */
int32_t pkv_decode_num_ctas(const pkv_cache_desc* cache, int32_t num_seqs,
                            int32_t num_q_heads, int32_t max_blocks_per_seq,
                            int32_t partition_size);

/* Paged attention decode (M5.3 0x0A, 0x0BA): one query row per sequence and
 * query head against the sequence's full logical history,
 *   out[r, h] = sum_t softmax_t(scale * q[r, h] . K_r[t]) V_r[t],
 *   lse[r, h] = log sum_t exp(scale * q[r, h] . K_r[t]),
 * where K_r[t], V_r[t] is token row t < seq_lens[r] of kv head
 * h / (Hq / Hkv), found in block block_tables[r, t / P] at offset t % P.  Rows
 * at offsets >= the request's tail are never read (M5.3 0x03G).
 *   out:           [num_seqs, Hq, D] (cache dtype).
 *   lse:           float [num_seqs, Hq] natural-log LSE, or NULL.  An empty
 *                  sequence gives out = 0 and lse = -inf.
 *   q:             [num_seqs, Hq, D].
 *   block_tables:  int32 [num_seqs, max_blocks_per_seq]; entries past
 *                  ceil(seq_lens[r] / P) are never read.
 *   seq_lens:      int32 [num_seqs].  The kernel may read it, and
 *                  block_tables, while the preceding kernel on `stream` still
 *                  runs, where that kernel allows its dependents to start
 *                  early (programmatic dependent launch; this library's
 *                  kv_append does): neither may be written by such a kernel.
 *                  Everything else is read only after the preceding work has
 *                  completed.
 *   partition_size: 0, or a multiple of block_size.  The work is split into
 *                  pieces (M5.3 0x0A: allocator block, kernel block and
 *                  reduction partition are three levels): the token rows of
 *                  every (sequence, kv head), in 32-row stages, are dealt out
 *                  in equal contiguous shares to persistent CTAs -- one wave of
 *                  them for 0 -- and a (sequence, kv head) cut between CTAs is
 *                  merged from its pieces' (output, LSE) states by log-sum-exp
 *                  in a second kernel.  A positive partition_size adds CTAs
 *                  until none streams more than max(stage, partition_size)
 *                  rows (a stage is 32 rows, or 128 on the tensor cores).
 *   workspace:     device scratch of at least pkv_decode_workspace_bytes
 *                  bytes, 256-byte aligned.  Nothing in it needs to be
 *                  initialised.
 * Supported: block_size 16 or a multiple of 32 up to 256; head_dim 64 or 128;
 * Hq / Hkv in {1, 2, 4, 8} (MXFP8 pools: see the top of this file);
 * num_seqs <= 65535.  Eight query heads per kv head with head_dim 128 and a
 * block size dividing 128 (or a multiple of it) run q.k and P.V on the
 * tcgen05 tensor cores (128-row stages; an MXFP8 pool's tiles are widened
 * to bf16 in shared memory first); everything else on the CUDA cores.  Same
 * results within the attention tolerance either way. */
pkv_status pkv_paged_attention_decode(
    const pkv_cache_desc* cache, void* out, float* lse, const void* q,
    const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
    int32_t num_q_heads, float scale, int32_t partition_size, void* workspace,
    size_t workspace_bytes, void* stream);

/* Bytes of device workspace pkv_shared_prefix_attention needs for these
 * sizes.  partition_size as for the suffix decode. */
size_t pkv_shared_prefix_workspace_bytes(const pkv_cache_desc* cache,
                                         int32_t num_seqs, int32_t num_q_heads,
                                         int32_t prefix_len,
                                         int32_t max_suffix_blocks,
                                         int32_t partition_size);

/* Shared-prefix attention (M5.3 0x0BC, Hydragen; merge of 0x0BA).  Request r's
 * logical history is the shared prefix -- prefix_len tokens in the blocks
 * prefix_block_ids[0 .. prefix_len / P) -- followed by its own suffix of
 * suffix_lens[r] tokens in blocks suffix_block_tables[r, 0 ..].  The result is
 * exactly pkv_paged_attention_decode over that concatenated history:
 *   - for each kv head, the prefix part is one dense contraction of all
 *     num_seqs * G query rows against the prefix keys on the tensor cores
 *     (bf16 in, fp32 accumulate), read once instead of once per request;
 *   - the suffixes run through the paged decode kernel;
 *   - the (output, LSE) states of both are merged by log-sum-exp.
 *   out, lse, q, scale, partition_size: as in pkv_paged_attention_decode.
 *   prefix_block_ids: int32 [prefix_len / P]; prefix_len a multiple of P (the
 *                  prefix is whole, shared blocks; a partly filled shared tail
 *                  is copied on write into each request's suffix first).
 *   suffix_block_tables: int32 [num_seqs, max_suffix_blocks]; suffix_lens:
 *                  int32 [num_seqs] (0 allowed).
 *   workspace:     at least pkv_shared_prefix_workspace_bytes, 256-byte
 *                  aligned.
 * Supported: bf16 only; head_dim 64 or 128; Hq / Hkv in {1, 2, 4, 8};
 * block_size 16, 32, 64, 128 or 256. */
pkv_status pkv_shared_prefix_attention(
    const pkv_cache_desc* cache, void* out, float* lse, const void* q,
    const void* k_cache, const void* v_cache, const int32_t* prefix_block_ids,
    int32_t prefix_len, const int32_t* suffix_block_tables,
    int32_t max_suffix_blocks, const int32_t* suffix_lens, int32_t num_seqs,
    int32_t num_q_heads, float scale, int32_t partition_size, void* workspace,
    size_t workspace_bytes, void* stream);

/* Keys per split the library uses for the prefix of these sizes (a multiple
 * of 128, chosen so that splits x query tiles x kv heads covers the SMs about
 * once); 0 for unsupported sizes. */
int32_t pkv_prefix_split_len(const pkv_cache_desc* cache, int32_t num_seqs,
                             int32_t num_q_heads, int32_t prefix_len);

/* Chunk-first phase of shared-prefix attention (M5.3 0x0BD, ChunkAttention:
 * batch the queries of every sequence against a shared chunk and materialise
 * partial softmax states; Hydragen's attention_with_lse over the shared part,
 * 0x0BC).  The prefix keys are cut into splits of split_len keys; for every
 * request r, query head h and split s it writes the state of attention of
 * q[r, h] over that split's keys alone:
 *   states_o[((r * Hq + h) * n + s) * D + c]  normalised output (fp32),
 *   states_lse[(r * Hq + h) * n + s]          natural-log LSE (fp32),
 * with n = ceil(prefix_len / split_len).  Merging a request's n states (and
 * any suffix state) by log-sum-exp gives attention over prefix ++ suffix.
 *   split_len: a positive multiple of 128 (pkv_prefix_split_len suggests one).
 * Other arguments and support as in pkv_shared_prefix_attention. */
pkv_status pkv_prefix_attention_states(const pkv_cache_desc* cache,
                                       float* states_o, float* states_lse,
                                       const void* q, const void* k_cache,
                                       const void* v_cache,
                                       const int32_t* prefix_block_ids,
                                       int32_t prefix_len, int32_t split_len,
                                       int32_t num_seqs, int32_t num_q_heads,
                                       float scale, void* stream);

/* ------------------------------------------------------------------------
 * Attention over a prefix tree (multi-level shared prefixes).
 *
 * A batch whose sequences share prefixes at several levels is described as a
 * tree snapshot ("M5.3 - KV Memory Layout and Exact Reuse", 0x0BB): an
 * ordered list of chunks, parents before children, each holding some K/V
 * rows in pool blocks and covering a half-open interval of sequence indices.
 * Sequence r's keys are the rows of every chunk whose interval holds r (its
 * root-to-leaf path); the result is exact attention of q[r] over them, as if
 * the path were one contiguous history (0x0BE's reference schedule).
 *
 * Execution follows ChunkAttention's two phases (0x0BD), and Hydragen's
 * batched attention per shared chunk (0x0BC):
 *   - chunk-first: a chunk covering more than `threshold` sequences is
 *     attended once for all of them, on the tensor cores (every covered
 *     sequence's G query heads against the chunk's keys, split in 128-key
 *     tiles); its partial softmax states are kept in the workspace;
 *   - sequence-first: every other (sequence, chunk) pair runs through the
 *     paged decode as one segment, leaving one state;
 *   - a merge kernel combines each sequence's states by log-sum-exp (0x0BA).
 * threshold = 0 attends every chunk chunk-first (hierarchical Hydragen);
 * a threshold >= the batch size attends everything sequence-first.  The
 * chunk-first phase needs bf16, head_dim 64 or 128, Hq / Hkv in {1, 2, 4,
 * 8} and 128 % P == 0 or P % 128 == 0; for other caches every chunk is
 * attended sequence-first.
 *
 * The snapshot is planned on the host into an opaque byte plan (the
 * metadata ChunkAttention builds on the host and transfers: chunk-first
 * work items and block ids, the decode's segment tables, each sequence's
 * state list).  The caller copies the plan verbatim to device memory and
 * passes both copies to pkv_chunk_tree_attention; a plan is valid for any
 * q, K/V contents and scale, as long as the tree, the pool shape and the
 * device it was planned on (SM count) stay the same. */

/* One chunk of a tree snapshot (host struct). */
typedef struct {
  int32_t first_id;  /* index in block_ids of the chunk's first block          */
  int32_t len;       /* K/V rows, >= 1: row t is in block                       */
                     /* block_ids[first_id + t / P] at offset t % P             */
  int32_t seq_begin; /* covered sequences: [seq_begin, seq_end), non-empty     */
  int32_t seq_end;
} pkv_chunk;

/* Plan a tree snapshot.
 *   chunks:        HOST [num_chunks], in tree order (parents first; any
 *                  order gives the same result up to rounding).
 *   block_ids:     HOST int32 [num_block_ids], every id in [0, num_blocks).
 *                  A chunk owns its blocks: a chunk whose len is not a
 *                  multiple of P leaves the rest of its last block unread.
 *   threshold:     chunks covering more than this many sequences go
 *                  chunk-first; < 0 picks 1 (every shared chunk).
 *   plan:          HOST buffer of plan_capacity bytes, or NULL to query the
 *                  sizes only.
 *   plan_bytes:    out (may be NULL): the plan's size.
 *   workspace_bytes: out (may be NULL): the device workspace
 *                  pkv_chunk_tree_attention needs.
 * Returns PKV_ERR_INVALID_ARG for a chunk with len < 1, an empty or
 * out-of-range interval, ids past num_block_ids or a block id outside the
 * pool; PKV_ERR_CAPACITY (sizes still reported) when plan_capacity is too
 * small.  Planning reads the device's SM count (the current device). */
pkv_status pkv_chunk_tree_plan(const pkv_cache_desc* cache, const pkv_chunk* chunks,
                               int32_t num_chunks, const int32_t* block_ids,
                               int64_t num_block_ids, int32_t num_seqs,
                               int32_t num_q_heads, int32_t threshold, void* plan,
                               size_t plan_capacity, size_t* plan_bytes,
                               size_t* workspace_bytes);

/* Attention over a planned tree snapshot.
 *   out:           [num_seqs, Hq, D] (cache dtype); a sequence no chunk
 *                  covers gets 0.
 *   lse:           fp32 [num_seqs, Hq] natural-log LSE (-inf for an empty
 *                  path), or NULL.
 *   q:             [num_seqs, Hq, D]; scale as in the decode.
 *   plan_host:     the plan as pkv_chunk_tree_plan wrote it (HOST).
 *   plan_device:   the same bytes in device memory, 256-byte aligned.
 *   workspace:     at least the planned workspace_bytes, 256-byte aligned.
 * Returns PKV_ERR_INVALID_ARG when the plan does not describe this cache,
 * num_seqs and num_q_heads (it checks the plan's header), or for a
 * workspace that is too small. */
pkv_status pkv_chunk_tree_attention(const pkv_cache_desc* cache, void* out, float* lse,
                                    const void* q, const void* k_cache, const void* v_cache,
                                    int32_t num_seqs, int32_t num_q_heads, float scale,
                                    const void* plan_host, const void* plan_device,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* Capacity in bytes of the library-owned scratch array used by
 * pkv_paged_attention_decode_static (16 MiB on every device that loads the
 * library, held until the process exits). */
#define PKV_STATIC_SCRATCH_BYTES (16u << 20)

/* Allocation-free variant of pkv_paged_attention_decode.  (The paper has no
 * counterpart: this is a deployment convenience of this library.)
 *
 * For callers that cannot allocate device memory themselves -- for example a
 * plugin whose host framework owns every device allocation, or a serving loop
 * that must never call cudaMalloc/cudaFree in its steady state (both can
 * synchronise the device or fail under memory pressure).  The decode's
 * workspace (its plan and piece states) is a fixed array of
 * PKV_STATIC_SCRATCH_BYTES bytes that the library
 * declares in device global memory, so the caller passes no workspace and the
 * call allocates nothing.  Arguments, results and errors are those of
 * pkv_paged_attention_decode, plus:
 *   - returns PKV_ERR_CAPACITY, launching nothing, when these sizes need more
 *     scratch than PKV_STATIC_SCRATCH_BYTES (pkv_decode_workspace_bytes tells
 *     how much they need); use pkv_paged_attention_decode with a caller-owned
 *     workspace then;
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture;
 *   - all calls on a device share the one array.  Calls that may run at the
 *     same time on the GPU (different streams without ordering between them)
 *     race on it and give wrong results: order them.  Nothing in the array
 *     needs to start at zero -- each call writes every value it reads -- so
 *     leftover contents from an earlier call do no harm. */
pkv_status pkv_paged_attention_decode_static(
    const pkv_cache_desc* cache, void* out, float* lse, const void* q,
    const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
    int32_t num_q_heads, float scale, int32_t partition_size, void* stream);

/* Read and clear the device error word of the current device.  Synchronises
 * `stream` first.  *code_out receives the PKV_DEVERR_* bits seen since the
 * last call.  Returns PKV_ERR_DEVICE if any bit was set, else PKV_OK. */
pkv_status pkv_get_device_error(int32_t* code_out, void* stream);

/* Static string for a status code. */
const char* pkv_status_string(pkv_status status);

#ifdef __cplusplus
}
#endif
#endif
