/*
 * pagedkv.h — C ABI of the GB300 (sm_103a) paged KV-cache decode path.
 *
 * The library implements the device side of PagedAttention-style KV-cache
 * management as the pages on the subject describe it:
 *
 *   "19.2 KV Cache 系统化管理" (book chapter 19.2): §19.2.2 block table and
 *      copy-on-write, §19.2.3 the block pool layout, write_slot /
 *      append_token and the block-wise online-softmax attention;
 *   "推理与 KV Cache 02:分页、共享与回收如何协作", section
 *      "从一个位置找到缓存块": logical block = floor(t/K), offset = t mod K,
 *      token slot = physical_block * K + offset;
 *   "KV Cache：长上下文为什么吃显存，PagedAttention 怎么救", §01 (the new
 *      token's query attends to K_{1:t}, V_{1:t}) and §02 (GQA ratio).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument except `code` in pkv_get_device_error is a DEVICE
 *   pointer to contiguous row-major memory owned by the caller.  The library
 *   allocates nothing and frees nothing.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Every compute call is asynchronous on that stream and returns once the
 *   work is enqueued.
 * - KV pool layout: k_cache and v_cache are [num_blocks, block_size,
 *   num_kv_heads, head_dim] (the pool of §19.2.3, its head axis holding the KV
 *   heads); seen as [num_blocks * block_size, num_kv_heads, head_dim] they are
 *   indexed by token slot.
 * - `dtype` is the storage type of q, k, v, the pools and out alike.
 * - Arguments are validated on the host before anything is launched; a bad
 *   argument returns PKV_ERR_INVALID_ARGUMENT or PKV_ERR_UNSUPPORTED and
 *   launches nothing.  A failed launch returns PKV_ERR_CUDA.
 * - Values that live on the device (block ids, slots, lengths, copy pairs)
 *   are checked by the kernels: an out-of-range value is never dereferenced;
 *   the offending element is skipped (attention treats an out-of-range block
 *   as zeros) and a code is recorded in a per-device error word that
 *   pkv_get_device_error reads.  No kernel traps.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(PKV_BUILD) && defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARGUMENT = 1,   /* null pointer, bad size, bad alignment  */
  PKV_ERR_UNSUPPORTED = 2,        /* shape/dtype this build does not handle */
  PKV_ERR_WORKSPACE_TOO_SMALL = 3,
  PKV_ERR_CUDA = 4,               /* a CUDA runtime call or launch failed   */
  PKV_ERR_DEVICE_CHECK = 5        /* returned by pkv_get_device_error only  */
} pkv_status;

typedef enum { PKV_F32 = 0, PKV_BF16 = 1 } pkv_dtype;

/* Codes recorded in the device error word (first one wins). */
enum {
  PKV_DEVERR_NONE = 0,
  PKV_DEVERR_BLOCK_ID = 1,     /* block-table entry outside [0, num_blocks)          */
  PKV_DEVERR_SLOT = 2,         /* slot outside [-1, num_blocks * block_size)          */
  PKV_DEVERR_COPY_PAIR = 3,    /* copy pair id outside [0, num_blocks)               */
  PKV_DEVERR_CONTEXT_LEN = 4,  /* context_lens[s] < 0, > max_context_len or beyond the
                                  table row (the length is clamped)                  */
  PKV_DEVERR_POSITION = 5,     /* position beyond the block-table row                */
  PKV_DEVERR_TIMEOUT = 6       /* a pipeline wait gave up after about a second       */
};

/* Human-readable name of a status.  Never NULL. */
PKV_API const char* pkv_status_string(pkv_status status);

/* Message of the last failure on the calling thread ("" if none). */
PKV_API const char* pkv_last_error_message(void);

/* ABI version: (major << 16) | minor. */
PKV_API int32_t pkv_version(void);

/*
 * a1 — slot mapping ("推理与 KV Cache 02", 从一个位置找到缓存块).
 *   slot_mapping[s] = block_tables[s][positions[s] / block_size] * block_size
 *                     + positions[s] % block_size
 * block_tables: int32 [num_seqs, max_blocks_per_seq]; positions: int32
 * [num_seqs]; slot_mapping: int64 [num_seqs] (output).  A negative position
 * gives slot -1 (padding).  A position past the table row or a block id
 * outside [0, num_blocks) gives -1 and records a device error.
 */
PKV_API pkv_status pkv_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* positions, int32_t num_seqs,
                            int32_t block_size, int64_t num_blocks,
                            int64_t* slot_mapping, void* stream);

/*
 * a2 — slot-mapped KV append ("19.2 KV Cache 系统化管理" §19.2.3, write_slot).
 *   k_cache.view(-1, H_kv, D)[slot_mapping[i]] = k[i]; same for v.
 * k, v: [num_tokens, num_kv_heads, head_dim]; slot_mapping: int64
 * [num_tokens].  Slot -1 skips the token.  Bit-exact copy of the rows.
 * Duplicate slots in one call: which token wins is unspecified.
 */
PKV_API pkv_status pkv_kv_write(const void* k, const void* v, const int64_t* slot_mapping,
                        int64_t num_tokens, void* k_cache, void* v_cache,
                        int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                        int32_t head_dim, pkv_dtype dtype, void* stream);

/*
 * a1 + a2 in one launch — slot mapping and KV append fused.
 *   For token i (block-table row i): slot = block_tables[i][positions[i] /
 *   block_size] * block_size + positions[i] % block_size, then
 *   k_cache.view(-1, H_kv, D)[slot] = k[i] and the same for v.
 * Same results as pkv_slot_mapping followed by pkv_kv_write; a negative
 * position skips the token; out-of-range positions / block ids skip it and
 * record a device error.  slot_mapping_out (int64 [num_tokens]) may be NULL;
 * when given it receives the slots (-1 for skipped tokens).
 */
PKV_API pkv_status pkv_kv_append(const void* k, const void* v, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* positions,
                                 int32_t num_tokens, void* k_cache, void* v_cache,
                                 int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                 int32_t head_dim, pkv_dtype dtype, int64_t* slot_mapping_out,
                                 void* stream);

/*
 * a5 — copy-on-write block copy ("19.2 KV Cache 系统化管理" §19.2.2, 写时复制:
 * allocate a new block and copy the shared block's contents into it).
 *   for each i: k_cache[pairs[i][1]] = k_cache[pairs[i][0]]; same for v_cache.
 * src_dst_pairs: int64 [num_pairs, 2].  Bit-exact.  A destination that is
 * also a source or another destination in the same call is unspecified.
 */
PKV_API pkv_status pkv_kv_block_copy(void* k_cache, void* v_cache, const int64_t* src_dst_pairs,
                             int64_t num_pairs, int64_t num_blocks, int32_t block_size,
                             int32_t num_kv_heads, int32_t head_dim, pkv_dtype dtype,
                             void* stream);

/* Optional tuning of pkv_attention_decode (pass NULL for the defaults). */
typedef struct {
  int32_t kernel;        /* 0 = automatic, 1 = TMA + tensor-core kernel
                            (bf16, block_size 8 or a multiple of 16, head_dim
                            64 or 128, G <= 8), 2 = CUDA-core kernel (any
                            supported shape) */
  int32_t num_splits;    /* kernel 1: CTAs sharing the token range of one KV-head
                            group (0 = SM count x CTAs per SM).  kernel 2:
                            tokens per partition (0 = automatic).              */
  int32_t share_prefix;  /* 0 = off.  1 = shared-prefix groups (decode with the
                            tensor-core kernel on bf16 pools; ignored by the
                            other plans): consecutive sequences are taken in
                            aligned groups of m = 16 / G (G = num_q_heads /
                            num_kv_heads, so G <= 8 gives m >= 2); the
                            leading tokens whose block-table entries are the
                            same physical blocks in every member's row
                            ("推理与 KV Cache 02", 前缀索引与 Block Table: whole
                            blocks shared through the table) are staged once
                            per group, one tile serving the query heads of
                            all members, and each member's remaining tokens
                            are read on their own; the partial states merge
                            in the split-K reduce.  Put the sequences that
                            share blocks (forks of one request, requests of
                            one prompt) next to each other.  Adds one small
                            launch that compares the table rows, and at most
                            1024 sequences go into one partition launch.   */
  int32_t reserved[5];   /* must be zero */
} pkv_attention_config;

/*
 * Workspace bytes pkv_attention_decode needs for these sizes (written to
 * *bytes).  Depends on the current device's SM count and on `config`.
 */
PKV_API pkv_status pkv_attention_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim,
                                         int32_t block_size, int32_t max_context_len,
                                         pkv_dtype dtype, const pkv_attention_config* config,
                                         size_t* bytes);

/*
 * Number of kernel launches pkv_attention_decode makes for these sizes
 * (written to *launches): one partition launch per batch of sequences, one
 * split-K reduce launch per batch when any sequence may be split, and with
 * share_prefix one table-comparison launch per batch.
 */
PKV_API pkv_status pkv_attention_launch_count(int32_t num_seqs, int32_t num_q_heads,
                                              int32_t num_kv_heads, int32_t head_dim,
                                              int32_t block_size, int32_t max_context_len,
                                              pkv_dtype dtype, const pkv_attention_config* config,
                                              int32_t* launches);

/*
 * a3 + a4 — decode attention over the paged cache with GQA and split-K
 * ("19.2 KV Cache 系统化管理" §19.2.3 paged_attention; "KV Cache：长上下文为什么
 * 吃显存" §01, §02).
 *   For each sequence s and query head h, with G = num_q_heads / num_kv_heads,
 *   j = h / G, L = context_lens[s] and token t in block
 *   block_tables[s][t / block_size] at offset t % block_size:
 *     out[s][h] = sum_t softmax_t(scale * q[s][h] . K_j[t]) * V_j[t]
 *   accumulated in fp32 with an online (running max / running sum) softmax.
 *   Long contexts are split across CTAs; partial (max, sum, output) states are
 *   merged by a second kernel with the same rescaling identity.
 * q: [num_seqs, num_q_heads, head_dim]; block_tables: int32 [num_seqs,
 * max_blocks_per_seq]; context_lens: int32 [num_seqs] (tokens read, including
 * the one appended this step); out: [num_seqs, num_q_heads, head_dim].
 * max_context_len: host-side upper bound of context_lens (sizes the split;
 * longer sequences are clamped to it and flagged).  A sequence of length 0
 * gets a zero output.  Entries of a table row past ceil(L / block_size) are
 * never read.  workspace: device scratch of at least
 * pkv_attention_workspace_bytes bytes, 256-byte aligned; no initial contents
 * are required; it must not be shared with a call that overlaps on the GPU.
 * Supported: num_q_heads % num_kv_heads == 0, G <= 16, head_dim in {32, 64,
 * 128, 256} (64 or 128 for the tensor-core kernel), 1 <= block_size <= 1024.
 */
PKV_API pkv_status pkv_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, int32_t max_context_len,
                                int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                float scale, void* out, void* workspace,
                                size_t workspace_bytes, pkv_dtype dtype,
                                const pkv_attention_config* config, void* stream);

/*
 * pkv_attention_decode without a caller-provided workspace.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory when they run attention.  Examples: an
 * inference engine that handed nearly all free HBM to its KV-cache pool at
 * start-up, so a cudaMalloc at decode time would fail; and code that must
 * not enter the CUDA allocator on the decode path at all, because cudaMalloc
 * and cudaFree can synchronise the device.  Here the split-K scratch lives in
 * a fixed array inside the library (PKV_NOALLOC_SCRATCH_BYTES, 64 MiB, held
 * on every GPU that loads the library until the process exits).  The call
 * allocates nothing.
 *
 * Arguments and results are those of pkv_attention_decode.  Sizes whose
 * scratch (pkv_attention_workspace_bytes) exceeds PKV_NOALLOC_SCRATCH_BYTES
 * are rejected with PKV_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 * The first call on a device looks up that device's copy of the array
 * (cudaGetSymbolAddress) with the device current; make that first call
 * before any stream capture.  The array is part of the library's device
 * module, which CUDA loads on a device at the library's first launch or
 * symbol lookup there: make the first call of any pkv_* compute function on
 * a device before the KV pool claims that device's free memory, or the
 * module (64 MiB of it this array) cannot be loaded.  A failed lookup
 * returns PKV_ERR_CUDA and is not remembered: the next call tries again.  All calls on a device share the one array:
 * calls that overlap on the GPU (different streams, no ordering between
 * them) race on it and give undefined results.  No initial contents are
 * needed; whatever a previous call left there is overwritten before use.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
PKV_API pkv_status pkv_attention_decode_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t max_context_len,
    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int64_t num_blocks, float scale, void* out, pkv_dtype dtype,
    const pkv_attention_config* config, void* stream);

/*
 * Self test of the failure path (the pages have no counterpart): launches one
 * CTA that waits on an mbarrier nothing ever arrives on, with the same
 * bounded wait the attention pipeline uses, limited to `limit_cycles`
 * (1 .. 2^31 SM cycles).  The wait gives up, records PKV_DEVERR_TIMEOUT and
 * the kernel exits; the context stays usable.  Read the code with
 * pkv_get_device_error.
 */
PKV_API pkv_status pkv_selftest_wait_timeout(int64_t limit_cycles, void* stream);

/*
 * Quantized KV cache (one byte per element).
 *
 * "学习大模型推理的显存优化", section KV Cache 量化: FP8 e4m3 (1 sign, 4
 * exponent, 3 mantissa bits, largest value 448); values are stored divided by
 * a scale and multiplied back when read; the default scale is 1.0.
 * "19.2 KV Cache 系统化管理" §19.2.4: INT8 with one scale per token,
 * k_int8 = round(k / scale), scale = max|k| / 127.
 *
 * PKV_KV_FP8_E4M3: pools hold e4m3 codes; one scale per tensor (k_scale for
 *   the K pool, v_scale for V); a value x is stored as e4m3(x / scale),
 *   rounded to nearest even and saturated to +-448.
 * PKV_KV_INT8_TOKEN: pools hold int8 codes; every token slot of a pool has
 *   its own float scale (k_token_scales / v_token_scales, device arrays of
 *   num_blocks * block_size floats) computed over the token's whole row (all
 *   KV heads x head_dim): scale = max|x| / 127 (float32), code =
 *   round_half_even(x / scale); an all-zero row gets scale 0 and codes 0.
 *   The tensor-core attention kernel forms each softmax weight times its
 *   token's V scale in f16: V scales must stay below 2048 (|v| below about
 *   260,000); larger ones may overflow to inf in the output.
 * PKV_KV_BF16K_FP8V: K kept more precise than V ("19.2 KV Cache 系统化管理"
 *   §19.2.4: K is the more sensitive of the two): the K pool holds bfloat16
 *   values (2 bytes per element; a float32 K row is rounded to nearest even),
 *   the V pool e4m3 codes of x / v_scale as in PKV_KV_FP8_E4M3 (k_scale is
 *   not used).  The tensor-core kernel needs a block size that is a multiple
 *   of 16; other shapes use the CUDA-core kernel.
 */
typedef enum {
  PKV_KV_PLAIN = 0,
  PKV_KV_FP8_E4M3 = 1,
  PKV_KV_INT8_TOKEN = 2,
  PKV_KV_BF16K_FP8V = 3
} pkv_kv_format;

typedef struct {
  int32_t format;          /* pkv_kv_format */
  float k_scale;           /* FP8: scale of the K pool (must be finite and > 0) */
  float v_scale;           /* FP8: scale of the V pool */
  float* k_token_scales;   /* INT8: [num_blocks * block_size] device floats */
  float* v_token_scales;   /* INT8: [num_blocks * block_size] device floats */
} pkv_kv_quant;

/*
 * a1 + a2 into a quantized pool: as pkv_kv_append, but the new rows k, v
 * (in_dtype: PKV_BF16 or PKV_F32) are quantized per `quant` before they are
 * stored; for INT8 the token's scales are stored at the same slot.
 */
PKV_API pkv_status pkv_kv_append_quant(const void* k, const void* v, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* positions,
                                       int32_t num_tokens, void* k_cache, void* v_cache,
                                       int64_t num_blocks, int32_t block_size,
                                       int32_t num_kv_heads, int32_t head_dim,
                                       pkv_dtype in_dtype, const pkv_kv_quant* quant,
                                       int64_t* slot_mapping_out, void* stream);

/*
 * a5 on a quantized pool: copies the byte blocks of K and V and, for INT8,
 * the blocks' per-token scales (so a copy is bit-exact in codes and scales).
 */
PKV_API pkv_status pkv_kv_block_copy_quant(void* k_cache, void* v_cache,
                                           const int64_t* src_dst_pairs, int64_t num_pairs,
                                           int64_t num_blocks, int32_t block_size,
                                           int32_t num_kv_heads, int32_t head_dim,
                                           const pkv_kv_quant* quant, void* stream);

/*
 * Block swap between two pools that may live in different memories
 * ("19.2 KV Cache 系统化管理" §19.2.6 调度与抢占, Swap: a preempted
 * request's KV blocks are parked in CPU memory and brought back when GPU
 * memory frees up; "企业官网建设流程全解析" §8.2: CPU memory as a second tier
 * of the block pool, oldest blocks out first, the block table hiding where
 * a block lives).
 *   for each i: dst_k[pairs[i][1]] = src_k[pairs[i][0]]; same for v.
 * One kernel moves every pair; the GPU reads and writes host memory directly
 * (NVLink-C2C / PCIe), so many small blocks cost one launch instead of one
 * copy call each.
 *   src_k, src_v: source pools, src_num_blocks blocks of block_bytes bytes.
 *   dst_k, dst_v: destination pools, dst_num_blocks blocks of block_bytes.
 *   block_bytes:  bytes of one block of one tensor: block_size * H_kv * D *
 *                 element bytes for a KV pool (any format), block_size * 4
 *                 for the float32 slot-scale arrays of an INT8 pool.
 *   pairs:        int64 [num_pairs, 2] (src block, dst block), in device
 *                 memory or in page-locked host memory.
 * src_v and dst_v may both be NULL (a single array per side).  Every pool
 * pointer must be device memory of the current device, or page-locked host
 * memory mapped into its address space (cudaHostAlloc, cudaHostRegister);
 * pageable host memory is refused with PKV_ERR_INVALID_ARGUMENT.  The source
 * is never written, so source and destination may be the same pool when no
 * destination block is also a source.  Ids outside their pool skip the pair
 * and record PKV_DEVERR_COPY_PAIR.  Bit-exact.  Asynchronous on `stream`:
 * the caller keeps host memory alive and unchanged until the stream reaches
 * the copy.
 */
PKV_API pkv_status pkv_kv_block_swap(const void* src_k, const void* src_v,
                                     int64_t src_num_blocks, void* dst_k, void* dst_v,
                                     int64_t dst_num_blocks, int64_t block_bytes,
                                     const int64_t* pairs, int64_t num_pairs, void* stream);

/* Workspace bytes of pkv_attention_decode_quant for these sizes. */
PKV_API pkv_status pkv_attention_quant_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                                       int32_t num_kv_heads, int32_t head_dim,
                                                       int32_t block_size,
                                                       int32_t max_context_len,
                                                       pkv_dtype q_dtype,
                                                       const pkv_kv_quant* quant,
                                                       const pkv_attention_config* config,
                                                       size_t* bytes);

/*
 * a3 + a4 over a quantized pool: the same attention as pkv_attention_decode
 * with every cached value read back as code * scale (per tensor for FP8, per
 * token slot for INT8).  q and out are q_dtype (PKV_BF16 or PKV_F32); the
 * accumulation is fp32.
 */
PKV_API pkv_status pkv_attention_decode_quant(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t max_context_len,
    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int64_t num_blocks, float scale, void* out, void* workspace,
    size_t workspace_bytes, pkv_dtype q_dtype, const pkv_kv_quant* quant,
    const pkv_attention_config* config, void* stream);

/*
 * Multi-query paged attention: several new tokens per sequence attend at
 * once over the paged cache — the chunks of a long prompt ("KV Cache：长上下文
 * 为什么吃显存，PagedAttention 怎么救" §06, Chunked Prefill), the suffix after a
 * prefix-cache hit ("推理与 KV Cache 02:分页、共享与回收如何协作", 前缀索引与
 * Block Table: the suffix still reads the prefix's KV), or speculative
 * candidate tokens ("企业官网建设流程全解析" §8.2).  Each new token is a query
 * of the new-token attention of "KV Cache：长上下文为什么吃显存" §01 at its own
 * position, causal among the new tokens:
 *   for sequence s with n = cu_seqlens[s+1] - cu_seqlens[s] new tokens and
 *   L = context_lens[s] (all tokens, the new ones included, already stored),
 *   new token i (packed row t = cu_seqlens[s] + i) at position p = L - n + i:
 *   out[t][h] = softmax_x(scale * q[t][h] . K[x][h/G]) V[x][h/G], x = 0 .. p.
 *   q, out:        [num_tokens, num_q_heads, head_dim] (dtype), packed by sequence.
 *   cu_seqlens:    int32 [num_seqs + 1], cu_seqlens[0] = 0, non-decreasing,
 *                  cu_seqlens[num_seqs] = num_tokens.
 *   context_lens:  int32 [num_seqs], each >= its new-token count.
 *   max_query_len: host bound on the new tokens of any sequence (sizes the
 *                  grid); max_context_len: host bound on context_lens.
 *   k_cache, v_cache, block_tables: as pkv_attention_decode.
 *   config:        NULL or kernel 0 = automatic, by the query rows of one
 *                  KV head (max_query_len x num_q_heads / num_kv_heads): up
 *                  to 8 -> the stream-K decode kernel; more -> tcgen05 tiles
 *                  of 128 rows (two per CTA sharing every K/V tile; one per
 *                  CTA when no KV head has more than 128 rows), except that
 *                  9 .. 64 rows with fewer (sequence, KV head) pairs than SMs,
 *                  or scale <= 0, take mma.sync tiles of 16 / 32 / 64 rows.
 *                  1 = tcgen05 (scale > 0, no split),
 *                  2 = mma.sync, 3 = stream-K decode kernel (at most 8 rows
 *                  per KV head, at most 2048 sequences, no split).
 *                  num_splits (mma.sync
 *                  kernel): 0 = automatic (key ranges of 512 tokens per CTA
 *                  when the grid would be small), n >= 1 = that many key
 *                  ranges.  Reserved fields must be 0.
 *   workspace:     device scratch of pkv_attention_prefill_workspace_bytes
 *                  bytes (256-byte aligned; may be NULL when that is 0),
 *                  holding the key-range partials merged by a second launch.
 * Supported: PKV_BF16, head_dim 64 or 128, block_size 8 or a multiple of 16
 * (else PKV_ERR_UNSUPPORTED).  n = 1 for every sequence is the decode step.
 * Inconsistent counts (n < 0, n > L, cu_seqlens past num_tokens) skip the
 * sequence and record PKV_DEVERR_CONTEXT_LEN.
 */
PKV_API pkv_status pkv_attention_prefill(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* cu_seqlens, const int32_t* context_lens,
                                         int32_t num_seqs, int32_t num_tokens,
                                         int32_t max_query_len, int32_t max_context_len,
                                         int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t block_size,
                                         int64_t num_blocks, float scale, void* out,
                                         void* workspace, size_t workspace_bytes,
                                         pkv_dtype dtype, const pkv_attention_config* config,
                                         void* stream);

/* Workspace bytes of pkv_attention_prefill for these sizes (0 when no key-
 * range split is used). */
PKV_API pkv_status pkv_attention_prefill_workspace_bytes(int32_t num_seqs, int32_t num_tokens,
                                                         int32_t max_query_len,
                                                         int32_t max_context_len,
                                                         int32_t num_q_heads,
                                                         int32_t num_kv_heads, int32_t head_dim,
                                                         int32_t block_size, float scale,
                                                         pkv_dtype dtype,
                                                         const pkv_attention_config* config,
                                                         size_t* bytes);

/*
 * a1 + a2 for the packed new tokens of pkv_attention_prefill: token t of
 * sequence s (cu_seqlens[s] <= t < cu_seqlens[s+1]) is stored at the slot of
 * position context_lens[s] - n_s + (t - cu_seqlens[s]) in s's block-table
 * row: k_cache.view(-1, H_kv, D)[slot] = k[t], same for v.  k, v:
 * [num_tokens, H_kv, D] (dtype).  slot_mapping_out (int64 [num_tokens]) may
 * be NULL; it receives the slots (-1 for skipped tokens).  Out-of-range
 * positions or block ids skip the token and record a device error.
 */
PKV_API pkv_status pkv_kv_append_varlen(const void* k, const void* v, const int32_t* cu_seqlens,
                                        const int32_t* context_lens, const int32_t* block_tables,
                                        int32_t max_blocks_per_seq, int32_t num_seqs,
                                        int32_t num_tokens, void* k_cache, void* v_cache,
                                        int64_t num_blocks, int32_t block_size,
                                        int32_t num_kv_heads, int32_t head_dim, pkv_dtype dtype,
                                        int64_t* slot_mapping_out, void* stream);

/*
 * Synchronises `stream`, copies the current device's error word into *code
 * (a PKV_DEVERR_* value) and clears it.  Returns PKV_ERR_DEVICE_CHECK when
 * the word was non-zero, PKV_OK when it was zero.
 */
PKV_API pkv_status pkv_get_device_error(int32_t* code, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
