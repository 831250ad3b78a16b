/*
 * dcp.h -- C ABI of libdcp: decode-time context parallelism (DCP) on one GPU.
 *
 * The method (Qiita write-up "vLLMの-dcpが長文脈のKVキャッシュ重複を消して3倍速くする",
 * section "トークンの区間でGPUに割り振る"; "Inference Systems Infrastructure
 * Notes (7): DCP", sections 2 and 3): the KV cache of every sequence is split
 * along the token axis into N contiguous ranges (shards). Each shard attends
 * the one-token decode query against its own slice only and emits a partial
 * output plus its log-sum-exp (LSE); the partials are then combined by
 * online-softmax reweighting into the exact full-context attention. Here the
 * N shards are virtual: N paged KV pools in the memory of one GPU, and the
 * cross-GPU gather/reduce-scatter becomes an on-device merge that reads one
 * caller-owned scratch buffer reused every step.
 *
 * Conventions for every entry point below:
 *  - Ownership: the caller allocates and frees every buffer. The library
 *    allocates no memory, keeps no per-call state and is re-entrant; the only
 *    global state is a per-device cache of launch limits (SM count, opt-in
 *    shared memory), filled on first use.
 *  - Pointers documented "device" must point to memory of the current CUDA
 *    device; "host" pointers to host memory. Arrays are dense, row-major,
 *    in the stated shape.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream). All work is enqueued on it; nothing synchronises.
 *  - Errors: arguments are validated on the host before any launch and a
 *    negative dcp_status is returned without touching the GPU. A failed launch
 *    returns DCP_ERR_CUDA. Inside kernels, a block-table entry outside
 *    [0, num_blocks), a logical block beyond max_blocks_per_seq or a position
 *    before shard 0 OR a DCP_DEVERR_* bit into *dev_err_flag (when the pointer
 *    is non-NULL) and skips that access; the caller reads the flag after the
 *    stream is synchronised and clears it itself.
 *  - Data types: queries are bf16 (raw 16-bit patterns); the KV cache and
 *    appended tokens are bf16, or optionally FP8 E4M3 codes with one scale
 *    for all keys and one for all values (dcp_attn_desc.kv_dtype);
 *    outputs and partials are fp32; LSE is the natural logarithm.
 */
#ifndef DCP_H_
#define DCP_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DCP_API __attribute__((visibility("default")))
#else
#define DCP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DCP_OK = 0,
  DCP_ERR_INVALID_ARG = -1, /* NULL where a pointer is required, bad count  */
  DCP_ERR_SHAPE = -2,       /* inconsistent sizes in the descriptor/shards   */
  DCP_ERR_UNSUPPORTED = -3, /* valid but not implemented (e.g. head_dim 96) */
  DCP_ERR_CUDA = -4,        /* a CUDA call or launch failed                  */
  DCP_ERR_WORKSPACE = -5,   /* workspace NULL, misaligned or too small       */
  DCP_ERR_SCRATCH_LIMIT = -6 /* problem needs more than the fixed scratch of
                                dcp_decode_partial_all_noalloc                */
} dcp_status;

/* Bits OR'ed into *dev_err_flag by kernels. */
#define DCP_DEVERR_BLOCK_RANGE 1 /* table entry < 0 or >= num_blocks            */
#define DCP_DEVERR_TABLE_RANGE 2 /* logical block >= max_blocks_per_seq        */
#define DCP_DEVERR_POSITION 4    /* position < 0 or before the first shard     */
#define DCP_DEVERR_TIMEOUT 8     /* a bounded on-device wait gave up            */

#define DCP_MAX_SHARDS 32

typedef enum { DCP_KIND_GQA = 0, DCP_KIND_MLA = 1 } dcp_kind;

/* Element type of the KV cache. P1 names KV cache quantization among the
 * techniques serving stacks pair with context parallelism, without a format;
 * the 8-bit option here is FP8 E4M3 (OCP "fn" variant: bias 7, no
 * infinities, 0x7F / 0xFF are NaN) with a per-tensor scale: a cached key is
 * k_scale * decode(code), a value v_scale * decode(code). */
typedef enum { DCP_KV_BF16 = 0, DCP_KV_FP8_E4M3 = 1 } dcp_kv_dtype;

/* Shape of one attention layer's decode step.
 *  GQA: query head h reads KV head h / (num_q_heads / num_kv_heads);
 *       head_dim_k == head_dim_v in {64, 128}; block_size a multiple of 16.
 *  MLA (absorbed): num_kv_heads == 1; the cached row is the latent of width
 *       head_dim_k (576); the key is the whole row and the value is its first
 *       head_dim_v (512) entries; block_size == 64. With the 8-bit cache the
 *       row is stored once as codes: key = k_scale * decode(row), value =
 *       v_scale * decode(row[:head_dim_v]).
 *  scale multiplies q.k before the softmax (e.g. 1/sqrt(head_dim_k)).
 *  kv_dtype DCP_KV_FP8_E4M3: k_scale and v_scale must be finite and > 0; the
 *  kernels widen the codes to fp16 exactly and convert q to fp16 (|q| must
 *  stay below 65504). For bf16 the scales are ignored. */
typedef struct {
  int kind;          /* dcp_kind */
  int num_q_heads;
  int num_kv_heads;
  int head_dim_k;
  int head_dim_v;
  int block_size;    /* tokens per paged block */
  float scale;
  int kv_dtype;      /* dcp_kv_dtype */
  float k_scale;     /* FP8 cache: key = k_scale * decode(code) */
  float v_scale;     /* FP8 cache: value = v_scale * decode(code) */
} dcp_attn_desc;

/* One shard's paged KV pool and block table (all device memory).
 *  GQA: k_pool [num_blocks, num_kv_heads, block_size, head_dim_k] bf16,
 *       v_pool [num_blocks, num_kv_heads, block_size, head_dim_v] bf16;
 *       FP8 cache: k_pool [num_blocks, num_kv_heads, block_size, head_dim_k]
 *       and v_pool [num_blocks, num_kv_heads, head_dim_v, block_size] E4M3
 *       codes (the values of a block stored transposed, dims by tokens).
 *  MLA: k_pool [num_blocks, block_size, head_dim_k] bf16 (or E4M3 codes),
 *       v_pool NULL.
 *  block_table: int32 [B, max_blocks_per_seq]; row b maps the shard-local
 *  logical block index (local position / block_size) of sequence b to a
 *  physical block of this pool. Pools must be 16-byte aligned. */
typedef struct {
  void* k_pool;
  void* v_pool;
  int64_t num_blocks;
  const int32_t* block_table;
  int32_t max_blocks_per_seq;
} dcp_shard;

/* Human-readable text for a dcp_status value (static storage). */
DCP_API const char* dcp_status_string(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
DCP_API int dcp_version(void);

/* Routing plan on the host (step 1 of the method: contiguous token ranges).
 * Passage: Qiita write-up "vLLMの-dcpが長文脈のKVキャッシュ重複を消して3倍速く
 * する", section "トークンの区間でGPUに割り振る" (a 200K-token request on 4 GPUs:
 * each GPU holds one contiguous interval of 50K tokens); "Inference Systems
 * Infrastructure Notes (7): DCP", section 2 (each GPU keeps only its
 * [start:end] slice of the sequence). Where the pages are silent (N does not
 * divide the length; where later tokens go) the reading is the one below.
 * For each sequence b with ctx_lens[b] tokens before decoding, the chunk is
 * C = max(1, ceil(ctx_lens[b] / N)); shard i starts at global position i*C;
 * shard i < N-1 owns [i*C, (i+1)*C) and the last shard is open-ended, so
 * appended decode tokens land there once the earlier shards are full.
 *   ctx_lens      host int32 [B], each >= 0
 *   shard_starts  host int32 [B, N] (out): i*C
 *   blocks_needed host int32 [B, N] (out, may be NULL): paged blocks shard i
 *                 needs to hold sequence b's tokens in [0, ctx_lens[b] +
 *                 reserve_tokens): ceil(tokens_in_shard / block_size).
 * Returns DCP_ERR_INVALID_ARG for N outside [1, DCP_MAX_SHARDS], B < 0,
 * block_size < 1, reserve_tokens < 0, a negative length, NULL outputs, or a
 * position that would not fit in int32. */
DCP_API int dcp_shard_plan(const int32_t* ctx_lens, int B, int N, int block_size, int reserve_tokens,
                   int32_t* shard_starts, int32_t* blocks_needed);

/* Write T tokens' K/V into the owning shards' paged pools (the per-step KV
 * append of decoding; with many tokens it also fills pools from a prefill).
 * Passage: "Inference Systems Infrastructure Notes (7): DCP", section 1
 * (decode is token by token: each step adds one token's KV to the cache) and
 * section 4 (decode shards the KV of every generated token; chunked and
 * cached prefill write and reuse KV slices); the Qiita write-up, section
 * "なぜテンソル並列だとKVキャッシュが二重に載るのか" (the cache holds the keys
 * and values of all past tokens; MLA keeps one latent row per token).
 * Token j belongs to sequence seq_ids[j] (or to sequence j when seq_ids is
 * NULL, which requires T == B) at global position positions[j]. Its owner is
 * the last shard i with shard_starts[b, i] <= position; the local position
 * p = position - shard_starts[b, i] selects logical block p / block_size and
 * slot p % block_size, and the block table gives the physical block.
 *   shards        host array of N dcp_shard (device pools/tables)
 *   shard_starts  device int32 [B, N] (from dcp_shard_plan)
 *   seq_ids       device int32 [T] or NULL;   positions device int32 [T]
 *   k_new         device bf16: GQA [T, num_kv_heads, head_dim_k]; MLA [T, head_dim_k]
 *   v_new         device bf16: GQA [T, num_kv_heads, head_dim_v]; MLA NULL
 *                 (FP8 cache: both E4M3 codes of the same shapes, already
 *                 quantised by the caller; v_new rows land transposed)
 * Bytes are copied as they are (bit-exact). T == 0 is a no-op. */
DCP_API int dcp_kv_append(const dcp_attn_desc* desc, const dcp_shard* shards, int N,
                  const int32_t* shard_starts, int B, const int32_t* seq_ids,
                  const int32_t* positions, const void* k_new, const void* v_new, int T,
                  int32_t* dev_err_flag, void* stream);

/* Bytes of workspace dcp_decode_partial / dcp_decode_partial_all need for up
 * to B sequences and N shards with this descriptor (0 on invalid input). The
 * workspace holds the work list and the split-KV temporaries; it is reused
 * by every call (no per-step allocation) and must be 256-byte aligned.
 * Passage: "Inference Systems Infrastructure Notes (7): DCP", section 3 (one
 * scratch buffer reused for the step's collectives instead of a temporary
 * allocation and copy per step). The size does not depend on the number of
 * cached tokens: the work list has one record per (shard, sequence) lane plus
 * one per work CTA, and the split-range temporaries are bounded by the CTA
 * count (a lane cut k ways needs k rows and holds k-1 CTA boundaries), so no
 * maximum token count enters. */
DCP_API size_t dcp_workspace_size(const dcp_attn_desc* desc, int B, int N);

/* Step 2 of the method for one shard: partial decode attention of every
 * sequence's one-token query against the tokens this shard holds.
 * Passage: Qiita write-up, section "トークンの区間でGPUに割り振る", second step
 * (each GPU runs attention of the gathered one-token query over its own KV
 * interval and keeps the partial output with its log-sum-exp); "Inference
 * Systems Infrastructure Notes (7): DCP", section 2 (slices processed in
 * parallel). The pages give no formula; the one below is plain softmax
 * attention restricted to the shard's tokens, which the merge of step 3
 * turns back into the exact full-context result.
 * For sequence b and query head h, over global positions t in
 * [shard_range[b,0], min(shard_range[b,1], seq_lens[b])):
 *   s_t = scale * <q[b,h], k_t>,  m = max s_t,  l = sum exp(s_t - m),
 *   o_part[b,h] = sum exp(s_t - m) v_t / l,  lse[b,h] = m + ln l.
 * A sequence with no token in range gets o_part = 0 and lse = -inf.
 *   q          device bf16 [B, num_q_heads, head_dim_k]
 *   shard      host pointer to one dcp_shard
 *   seq_lens   device int32 [B], global lengths including appended tokens
 *   shard_range device int32 [B, 2], global [start, end) of this shard
 *              (start is the shard's first position: local position 0)
 *   o_part     device fp32 [B, num_q_heads, head_dim_v] (out)
 *   lse        device fp32 [B, num_q_heads] (out)
 *   workspace  device, >= dcp_workspace_size(desc, B, 1) bytes            */
DCP_API int dcp_decode_partial(const dcp_attn_desc* desc, const void* q, const dcp_shard* shard,
                       const int32_t* seq_lens, const int32_t* shard_range, int B,
                       float* o_part, float* lse, void* workspace, size_t ws_bytes,
                       int32_t* dev_err_flag, void* stream);

/* Step 2 for all N shards in one pass of launches. Shard i of sequence b
 * covers [shard_starts[b,i], shard_starts[b,i+1]) (the last shard up to
 * seq_lens[b]), clipped to seq_lens[b].
 * Passage: as dcp_decode_partial (Qiita write-up, section "トークンの区間で
 * GPUに割り振る", second step); the N shards that run on N GPUs there run here
 * as one set of launches over N pools in one memory, with the same outputs.
 *   o_parts device fp32 [N, B, num_q_heads, head_dim_v] (out)
 *   lses    device fp32 [N, B, num_q_heads] (out)
 *   workspace >= dcp_workspace_size(desc, B, N) bytes                      */
DCP_API int dcp_decode_partial_all(const dcp_attn_desc* desc, const void* q, const dcp_shard* shards,
                           int N, const int32_t* seq_lens, const int32_t* shard_starts, int B,
                           float* o_parts, float* lses, void* workspace, size_t ws_bytes,
                           int32_t* dev_err_flag, void* stream);

/* Most query tokens per sequence that dcp_decode_partial_all_mtp accepts
 * (a speculative step's few tokens, or a whole prefill chunk). */
#define DCP_MAX_QUERY_TOKENS 8192

/* Bytes of workspace dcp_decode_partial_all_mtp needs for B sequences with
 * q_len query tokens each and N shards (0 on invalid input or q_len outside
 * [1, DCP_MAX_QUERY_TOKENS]); dcp_workspace_size(desc, B, N) is the q_len = 1
 * case. Same alignment and reuse rules as dcp_workspace_size, and the same
 * passage ("Inference Systems Infrastructure Notes (7): DCP", section 3: one
 * reused scratch buffer). */
DCP_API size_t dcp_workspace_size_mtp(const dcp_attn_desc* desc, int B, int q_len, int N);

/* Step 2 for all N shards when each sequence brings q_len new tokens at once
 * (a speculative-decoding or multi-token-prediction step). The pages name
 * speculative decoding and MTP as what DCP is combined with next (Qiita
 * write-up "vLLMの-dcpが長文脈のKVキャッシュ重複を消して3倍速くする", section
 * "実務でどう見るか"; "Inference Systems Infrastructure Notes (7): DCP",
 * section 5) without a formula; this call takes the reading that query token
 * j (0 <= j < q_len) of sequence b sits at global position
 * seq_lens[b] - q_len + j and attends every token at or before it -- causal
 * among the new tokens, as q_len consecutive one-token steps would. All q_len
 * tokens' K/V are appended first (dcp_kv_append with T = B * q_len).
 * The same call is one chunk of a chunked or cached prefill against the
 * sharded cache ("Inference Systems Infrastructure Notes (7): DCP", section
 * 4: long inputs prefilled in chunks; already computed KV slices reused):
 * the chunk's tokens are appended after the cached context and attend it and
 * each other causally; only q_len differs.
 * Each shard's range is clipped to the query token's causal limit
 * seq_lens[b] - q_len + j + 1; a query token before position 0, or with no
 * token in a shard's range, gets o = 0 and lse = -inf there.
 *   q        device bf16 [B, q_len, num_q_heads, head_dim_k]
 *   seq_lens device int32 [B], global lengths including the q_len new tokens
 *   o_parts  device fp32 [N, B, q_len, num_q_heads, head_dim_v] (out)
 *   lses     device fp32 [N, B, q_len, num_q_heads] (out)
 *   workspace >= dcp_workspace_size_mtp(desc, B, q_len, N) bytes
 * The merge of step 3 is dcp_merge with B * q_len rows of sequences. q_len
 * outside [1, DCP_MAX_QUERY_TOKENS] returns DCP_ERR_INVALID_ARG; q_len = 1 is
 * dcp_decode_partial_all. The block tables are indexed by sequence: every
 * query token of sequence b reads row b. */
DCP_API int dcp_decode_partial_all_mtp(const dcp_attn_desc* desc, const void* q, const dcp_shard* shards,
                                       int N, const int32_t* seq_lens, const int32_t* shard_starts, int B,
                                       int q_len, float* o_parts, float* lses, void* workspace,
                                       size_t ws_bytes, int32_t* dev_err_flag, void* stream);

/* Steps 2 and 3 in one call: the partial attention of every shard (as
 * dcp_decode_partial_all_mtp; q_len = 1 for a decode step) and the merge of
 * the shards by the LSE reweighting of dcp_merge. (The pages merge the
 * shards' partials after the per-shard attention -- Qiita write-up, section
 * "トークンの区間でGPUに割り振る", third step; this joins the two on one GPU,
 * keeping the intermediate results in reused buffers or on chip as
 * "Inference Systems Infrastructure Notes (7): DCP", section 3, does with its
 * scratch buffer.) Same result as dcp_decode_partial_all_mtp + dcp_merge
 * within the parity bar:
 *   GQA: after the attention kernel, one pass merges every output row's
 *        pieces -- the shard's partial row, or the pieces of a shard range the
 *        balanced split cut across several CTAs.
 *   MLA: the attention kernel merges the shards itself. A CTA pair carries one
 *        online softmax through consecutive shards of a query row (the shards
 *        meet inside the softmax's rescaling), rows cut by a CTA-run boundary
 *        leave pieces in the workspace, merged by the CTA completing their
 *        count (up to 4 pieces) or by a short finishing kernel; o_parts and
 *        lses are not touched. Results are deterministic for a given device,
 *        problem and workspace.
 *   o_parts, lses  device fp32 scratch [N, B, q_len, Hq, Dv] / [N, B, q_len, Hq]
 *                  (GQA: partial rows of shards whose range one CTA covered)
 *   o        device fp32 [B, q_len, num_q_heads, head_dim_v] (out)
 *   lse_out  device fp32 [B, q_len, num_q_heads] (out) or NULL
 *   workspace >= dcp_workspace_size_mtp(desc, B, q_len, N) bytes
 * head_dim_v must be a multiple of 4 and at most 512; o 16-byte aligned. */
DCP_API int dcp_attention_all(const dcp_attn_desc* desc, const void* q, const dcp_shard* shards, int N,
                              const int32_t* seq_lens, const int32_t* shard_starts, int B, int q_len,
                              float* o_parts, float* lses, float* o, float* lse_out, void* workspace,
                              size_t ws_bytes, int32_t* dev_err_flag, void* stream);

/* Same computation as dcp_decode_partial_all, for callers that cannot
 * allocate device memory at the point of the call: for example a plugin
 * running inside a serving engine that owns every byte of device memory
 * through its own pool and hands extensions no scratch buffer, or a
 * latency-critical decode loop that must not call cudaMalloc because it can
 * synchronise the device. (The pages describe no such entry point; it exists
 * only for these callers.)
 *
 * Instead of a caller-provided workspace it uses one fixed scratch array of
 * DCP_NOALLOC_SCRATCH_BYTES in device global memory, defined by the library
 * itself; every GPU that loads the library keeps that array until the process
 * exits. The call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it; make
 *    that first call before any stream capture. The cached address belongs
 *    to the device's context at that time: after cudaDeviceReset on that
 *    device it is stale, so do not call this entry point again in a process
 *    that has reset the device.
 *  - Problems whose workspace (dcp_workspace_size(desc, B, N)) exceeds
 *    DCP_NOALLOC_SCRATCH_BYTES are rejected with DCP_ERR_SCRATCH_LIMIT before
 *    any launch.
 *  - All calls on a device share the one array and leave their contents in
 *    it; nothing in it has to start at zero (each call writes everything it
 *    later reads). Calls whose work overlaps on the GPU -- concurrent streams,
 *    or several host threads -- race on the array: serialise them.
 * Arguments and outputs are those of dcp_decode_partial_all. */
#define DCP_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

DCP_API int dcp_decode_partial_all_noalloc(const dcp_attn_desc* desc, const void* q,
                                           const dcp_shard* shards, int N, const int32_t* seq_lens,
                                           const int32_t* shard_starts, int B, float* o_parts,
                                           float* lses, int32_t* dev_err_flag, void* stream);

/* Step 3 of the method: combine N partials by LSE reweighting
 * ("Inference Systems Infrastructure Notes (7): DCP", section 2; the Qiita
 * section "トークンの区間でGPUに割り振る", third step). For every row r:
 *   M = max_i lses[i,r],  w_i = exp(lses[i,r] - M),
 *   o[r] = sum_i w_i o_parts[i,r] / sum_i w_i,  lse_out[r] = M + ln sum_i w_i;
 * rows whose partials are all empty (LSE -inf) give o = 0, lse_out = -inf.
 *   o_parts device fp32 [N, B, Hq, Dv]; lses device fp32 [N, B, Hq]
 *   o       device fp32 [B, Hq, Dv] (out); lse_out device fp32 [B, Hq] or NULL
 * Dv must be a multiple of 4 and the pointers 16-byte aligned. */
DCP_API int dcp_merge(const float* o_parts, const float* lses, int N, int B, int Hq, int Dv, float* o,
              float* lse_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DCP_H_ */
