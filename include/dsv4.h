/*
 * dsv4.h - C ABI of the DeepSeek-V4 hybrid compressed-attention decode step on one GB300.
 *
 * One decode step of a CSA (compress ratio 4, top-k sparse) or HCA (ratio 128, dense) layer is
 *
 *   dsv4_kv_insert        the new tokens' latent rows -> paged sliding-window (SWA) cache
 *   dsv4_compress_update  fp32 compressor state store; every ratio-th token folds a group into
 *                         one compressed entry of the paged main cache
 *   dsv4_indexer_topk     Lightning-Indexer scores of every visible compressed entry and the
 *                         per-query top-k (CSA only)
 *   dsv4_sparse_mla_decode  one softmax per head over the SWA rows + the selected (or all)
 *                         compressed rows + an optional sink, shared-KV MQA
 *
 * Sources: "DeepSeek V4 Attention: Code Reading Map" (MAP), "DeepSeek-V4 Inference on Ascend:
 * The DSA Serving Stack in vllm-ascend" (ASCEND), "vllm.models.deepseek_v41.attention" (API).
 *
 * Conventions shared by every call
 *  - Every pointer in a params struct is a DEVICE pointer unless the field says otherwise; the
 *    caller owns all memory and the library allocates nothing.  Scratch memory is passed in as
 *    `workspace` and sized by the matching *_workspace_bytes() call (a pure host function).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream) and
 *    never synchronise the host, so a step can be captured into a CUDA graph.
 *  - Latent rows are DSV4_LATENT_DIM = 576 wide: dims 0..511 are the no-pe part (and the
 *    value), dims 512..575 the rope part.  Paged caches are [num_pages, page_size, row] with the
 *    row stored in the cache dtype; a logical row i of a sequence lives at page
 *    block_table[seq][i / page_size], offset i % page_size.
 *  - Token t belongs to sequence t / q_per_seq; a sequence's tokens are consecutive positions in
 *    increasing order (decode, or MTP-style multi-token decode).
 *  - A query at 0-based position p sees the window rows max(0, p - window + 1) .. p and
 *    n_c(p) = floor((p + 1) / ratio) compressed entries.
 *  - Structs start with `struct_size` (= sizeof the struct the caller was compiled with); a
 *    mismatch returns DSV4_ERR_INVALID.
 *  - Host-side validation (null pointers, misalignment, unsupported dtype/shape combinations,
 *    sizes over the limits) returns an error before anything is launched.  Device-side range
 *    checks (block-table pages, slots, top-k indices) skip the bad access and raise a flag that
 *    dsv4_read_device_flags() returns; no kernel traps or faults on bad indices.
 *  - Inside a kernel, warps hand work to each other through shared-memory barriers (TMA and tensor
 *    core completions, producer/consumer rings) and the CTAs of a cluster meet at cluster
 *    barriers.  Every such wait is bounded in time (about 0.25 s): a wait that runs out makes the
 *    kernel's roles drain and exit, leaves the affected outputs unspecified and raises the
 *    timeout flag (bit 2 of dsv4_read_device_flags()).  No kernel waits on another kernel or on
 *    the host.
 */
#ifndef DSV4_H
#define DSV4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSV4_ABI_VERSION 3
#define DSV4_LATENT_DIM 576
#define DSV4_VALUE_DIM 512
#define DSV4_ROPE_DIM 64
#define DSV4_FP8_DS_MLA_BYTES 656
#define DSV4_MAX_Q_PER_SEQ 4

typedef enum dsv4_status {
  DSV4_OK = 0,
  DSV4_ERR_INVALID = -1,      /* null / misaligned / out-of-range argument */
  DSV4_ERR_UNSUPPORTED = -2,  /* dtype or shape combination not implemented */
  DSV4_ERR_CUDA = -3,         /* a CUDA call failed; dsv4_last_cuda_error() has the code */
  DSV4_ERR_BOUNDS = -4,       /* returned by dsv4_read_device_flags() when a kernel skipped a bad index */
  DSV4_ERR_TIMEOUT = -5       /* returned by dsv4_read_device_flags() when a kernel gave up a bounded wait */
} dsv4_status;

/* Storage formats of rows and activations. */
typedef enum dsv4_dtype {
  DSV4_F32 = 0,          /* float32 elements */
  DSV4_BF16 = 1,         /* bfloat16 elements */
  /* 656-byte latent record: bytes [0,512) e4m3fn codes of dims 0..511, [512,640) bf16 of dims
   * 512..575, [640,648) one UE8M0 byte per 64-dim no-pe block (scale 2^(byte-127)), [648,656)
   * zero.  The UE8M0 exponent is the smallest e with 448 * 2^e >= the block's max |x| (MAP,
   * "How Does Compression Actually Work?" step 6; API, DeepseekV4Attention, fp8_ds_mla). */
  DSV4_FP8_DS_MLA = 2,
  /* indexer key record of head_dim + 4 bytes: head_dim int8 codes then the little-endian fp32
   * scale of the row; key = code * scale (API, _indexer_k_cache_head_dim: 128 + 4 = 132 B). */
  DSV4_I8_ROWSCALE = 3,
  /* MXFP4 indexer key record of head_dim / 2 + head_dim / 32 bytes (68 B for 128 dims; API,
   * _indexer_k_cache_head_dim): E2M1 codes, element 2i in the low nibble of byte i, then one UE8M0
   * byte per 32 elements; key = code * 2^(byte - 127).  The encoders here take the smallest block
   * exponent e with 6 * 2^e >= the block's max |x| and round to nearest even. */
  DSV4_MXFP4 = 4
} dsv4_dtype;

typedef void* dsv4_stream_t; /* cudaStream_t */

/* ---------------------------------------------------------------------------------------------
 * dsv4_kv_insert: write each new token's latent row into the paged SWA cache.
 * MAP "4. _fused_qnorm_rope_kv_insert() - Where SWA Happens"; API _fused_qnorm_rope_kv_insert
 * (the KV half: optional GPT-J RoPE of dims 512..575, encode, store at slot_mapping[t]).
 * ------------------------------------------------------------------------------------------- */
typedef struct dsv4_kv_insert_params {
  uint32_t struct_size;
  const void* kv_new;          /* [T, 576] in kv_dtype (DSV4_F32 or DSV4_BF16), rows contiguous */
  int32_t kv_dtype;
  const int64_t* slot_mapping; /* [T] slot = page * page_size + offset; -1 skips the token */
  void* cache;                 /* [num_pages, page_size, row] in cache_dtype (F32, BF16, FP8_DS_MLA) */
  int32_t cache_dtype;
  int32_t T;                   /* tokens, >= 0 (0 is a no-op) */
  int32_t page_size;           /* rows per page, > 0 */
  int64_t num_pages;           /* pages in `cache`; a slot past the end is skipped and flagged */
  const int32_t* positions;    /* [T] RoPE positions; only read when cos_sin != NULL */
  const float* cos_sin;        /* [max_pos, 64] (32 cos | 32 sin) or NULL = rows already rotated */
  int32_t max_pos;
  int32_t after_independent;   /* 0: the kernel waits for the kernel before it on `stream` before it
                                  starts its work (always safe), and lets the kernels after it start
                                  only once that wait is over.  1: the caller guarantees that the
                                  kernels before it on `stream`, back to and including the last one
                                  launched with 0 (or any other kernel), neither read nor write
                                  anything this call reads or writes (as the insert and the
                                  compressor of one step); the kernel then does its work at once
                                  and waits for the kernel before it only before it exits, so its
                                  completion still implies the earlier ones' */
} dsv4_kv_insert_params;

int dsv4_kv_insert(const dsv4_kv_insert_params* p, dsv4_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * dsv4_qnorm_rope_kv_insert: the query heads made ready for the attention and the new KV rows
 * stored, in one launch (MAP "Phase 2", default stream, item 2: per-head RMSNorm of every query
 * head, GPT-J RoPE of the last 64 dims of each query head and of kv, kv stored into the SWA cache;
 * API DeepseekV4Attention._fused_qnorm_rope_kv_insert: the query zero-padded to the padded head
 * count the attention backend allocates, see dsv4_padded_num_q_heads).
 * For token t at position p = positions[t] and head h < H:
 *   x = q[t][h];  if apply_q_norm: x = x / sqrt(mean(x^2) + eps) * q_norm_weight  (over 576 dims,
 *   fp32);  if apply_q_rope: dims 512..575 of x turned by GPT-J RoPE with cos_sin[p];
 *   q_out[t][h] = x in act_dtype (bf16: round to nearest even);  q_out[t][h] = 0 for H <= h < H_pad.
 * and kv_new[t] is stored at slot_mapping[t] exactly as dsv4_kv_insert does (RoPE at p when
 * apply_kv_rope).
 * ------------------------------------------------------------------------------------------- */
typedef struct dsv4_qnorm_rope_kv_insert_params {
  uint32_t struct_size;
  const void* q;               /* [T, H, 576] in act_dtype, 16-byte aligned */
  void* q_out;                 /* [T, H_pad, 576] in act_dtype, 16-byte aligned; may be q itself only
                                  when H_pad == H (in place), else must not overlap q */
  int32_t H, H_pad;            /* 1 <= H <= H_pad <= 1024 */
  const float* q_norm_weight;  /* [576] per-channel weight of the query RMSNorm, or NULL (= 1) */
  int32_t apply_q_norm, apply_q_rope;
  float eps;
  const void* kv_new;          /* [T, 576] in act_dtype */
  const int64_t* slot_mapping; /* [T] SWA slot = page * page_size + offset; -1 skips the token's kv */
  void* cache;                 /* [num_pages, page_size, row] in cache_dtype (F32, BF16, FP8_DS_MLA) */
  int32_t cache_dtype;
  int32_t page_size;
  int64_t num_pages;
  int32_t apply_kv_rope;
  int32_t act_dtype;           /* DSV4_F32 or DSV4_BF16: q, q_out and kv_new */
  int32_t T;                   /* tokens, >= 0 */
  const int32_t* positions;    /* [T] (read when some RoPE is applied; outside [0, max_pos) is flagged) */
  const float* cos_sin;        /* [max_pos, 64] (32 cos | 32 sin, GPT-J pairs); needed for any RoPE */
  int32_t max_pos;
  int32_t after_independent;   /* as in dsv4_kv_insert_params */
} dsv4_qnorm_rope_kv_insert_params;

int dsv4_qnorm_rope_kv_insert(const dsv4_qnorm_rope_kv_insert_params* p, dsv4_stream_t stream);

/* Query heads the attention's q and output buffers must hold for H real heads with caches of
 * cache_dtype (API get_padded_num_q_heads): the tensor-core attention of bf16 and fp8_ds_mla caches
 * takes heads in groups of 64, so H rounded up to 64; fp32 caches take H as it is.  A pure host
 * function; returns -1 for H < 1 or an unknown dtype. */
int dsv4_padded_num_q_heads(int H, int cache_dtype);

/* ---------------------------------------------------------------------------------------------
 * dsv4_compress_update: compressor state store and fold (MAP "What Are the Gate Scores?",
 * "How Does Compression Actually Work?", "Phase 2" compressor stream items 1-4).
 * For each sequence, for each of its new tokens in position order:
 *   state[b][p mod (coff*ratio)] = [kv half of kv_score[t] | score half + ape[p mod ratio]] (fp32)
 *   if (p + 1) % ratio == 0: entry j = p / ratio is the per-channel softmax-over-tokens weighted
 *   sum of kv over the group (ratio tokens via series A; with coff = 2 also the previous group's
 *   ratio tokens via series B, when j >= 1), RMSNorm * norm_weight, GPT-J RoPE of dims
 *   512..575 at position j * ratio, encoded into the main-cache row j of the sequence.
 * ------------------------------------------------------------------------------------------- */
typedef struct dsv4_compress_update_params {
  uint32_t struct_size;
  const float* kv_score;       /* [T, 2*coff*576]: kv series 0..coff-1, then score series 0..coff-1 */
  const int32_t* positions;    /* [T] */
  int32_t T, B, q_per_seq;     /* T = B * q_per_seq, q_per_seq in 1..DSV4_MAX_Q_PER_SEQ */
  int32_t ratio;               /* 4 or 128 */
  int32_t coff;                /* 2 (overlapping series, ratio 4) or 1 */
  float* state;                /* [B, coff*ratio, 2*coff*576] fp32 ring, read and written */
  const float* ape;            /* [ratio, coff*576] or NULL (no positional term) */
  const float* norm_weight;    /* [576] */
  float eps;
  const float* cos_sin;        /* [max_pos, 64]: row j*ratio rotates entry j */
  int32_t max_pos;
  void* main_cache;            /* [num_pages, page_size, row] in cache_dtype (F32, BF16, FP8_DS_MLA) */
  int32_t cache_dtype;
  int32_t page_size;
  int64_t num_pages;
  const int32_t* block_table;  /* [B, max_pages_per_seq] main-cache pages of each sequence */
  int32_t max_pages_per_seq;
  int32_t after_independent;   /* as in dsv4_kv_insert_params */
  /* Index-key store (optional; CSA layers whose indexer takes its keys from this compressor: API
   * DeepseekV4Indexer, "k = k_norm(wk(latent))"; _produce_k: at group-boundary tokens, RoPE'd at
   * the group position, quantised into the indexer K cache).  For every entry j folded by this call,
   * with latent_j = the entry after RMSNorm * norm_weight and before its RoPE:
   *   k = wk latent_j (fp32);  k = k / sqrt(mean(k^2) + ik_eps) * ik_norm_weight;  GPT-J RoPE of the
   *   last 64 dims of k at position j * ratio;  stored in ik_dtype into row j of the indexer cache
   *   (I8_ROWSCALE: scale = max|k| / 127 (1 when k = 0), code = round-half-even(k / scale) clamped
   *   to +-127, both in fp32). */
  const void* wk;              /* [ik_dim, 576] bf16, or NULL: no index keys */
  const float* ik_norm_weight; /* [ik_dim] */
  float ik_eps;
  int32_t ik_dim;              /* 64 or 128 */
  void* ik_cache;              /* [ik_num_pages, page_size, row] in ik_dtype (F32, BF16 or I8_ROWSCALE) */
  int32_t ik_dtype;
  int64_t ik_num_pages;
  const int32_t* ik_block_table; /* [B, ik_max_pages] indexer-cache pages of each sequence */
  int32_t ik_max_pages;
} dsv4_compress_update_params;

int dsv4_compress_update(const dsv4_compress_update_params* p, dsv4_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * dsv4_indexer_topk: Lightning-Indexer scoring and per-query top-k (MAP "Phase 2" indexer stream
 * item 4, "Concrete Trace" top-1024; API DeepseekV4Indexer.forward for the short-context fill).
 *   s[t][j] = sum_h weights[t][h] * max(0, q[t][h] . key_j), fp32, for j < n_c(positions[t]);
 *   topk_idx[t] = the min(topk, n_c) entries with the largest s (ties: lower j first), listed in
 *   increasing j, then -1 padding.  When n_c <= topk every entry is selected.
 * ------------------------------------------------------------------------------------------- */
typedef struct dsv4_indexer_topk_params {
  uint32_t struct_size;
  const void* q;               /* [T, n_heads, head_dim] in q_dtype (F32 or BF16) */
  int32_t q_dtype;
  const float* weights;        /* [T, n_heads] per-head weights (any scale factors folded in) */
  const void* k_cache;         /* [num_pages, page_size, row]: F32/BF16 rows of head_dim, or
                                  I8_ROWSCALE records of head_dim + 4 bytes */
  int32_t k_dtype;
  int64_t num_pages;
  const int32_t* block_table;  /* [B, max_pages_per_seq] indexer-cache pages of each sequence */
  int32_t max_pages_per_seq;
  const int32_t* positions;    /* [T] */
  int32_t T, B, q_per_seq, ratio, n_heads, head_dim, topk, page_size;
  int32_t max_context;         /* host bound on positions[t] + 1 (sizes the workspace and grid);
                                  max_context / ratio <= 2^20 compressed entries */
  int32_t* topk_idx;           /* [T, topk] output */
  float* topk_score;           /* [T, topk] output scores of topk_idx (-inf on padding) or NULL */
  void* workspace;             /* dsv4_indexer_topk_workspace_bytes() bytes, 256-byte aligned */
  size_t workspace_bytes;
  int32_t workspace_zeroed;    /* 0: the call first clears the histograms and counters it keeps in the
                                  workspace (one memset on `stream`).  1: the caller guarantees they are
                                  zero: the workspace was zero-filled once when allocated, and every
                                  call that completed without raising a flag left it so (each call
                                  clears what it used before it completes) */
  /* Two-level candidate filtering (API DeepseekV4Indexer: candidate_block_size,
     candidate_topk_blocks, candidate_write).  Off when cand_block_size is 0 (cand_blocks unused).
     Compressed entry j lies in candidate block j / cand_block_size.
     cand_write = 1 (the candidate source): scoring and top-k as above, and cand_blocks[t] receives
       the cand_topk blocks with the largest block score (the largest s[t][j] of the block's entries
       j < n_c; ties: lower block first), listed in increasing order, then -1 padding; every block
       when there are at most cand_topk.
     cand_write = 0 (a consumer): cand_blocks[t] names token t's blocks: its entries up to the first
       one that is negative or not larger than the entry before it.  When n_c > topk, only entries of
       named blocks take part: topk_idx[t] = the min(topk, their count) best of them (same order and
       padding as above); when n_c <= topk every entry is selected as without candidates.  With one
       query token a sequence (q_per_seq = 1) the blocks that are not named are never read or scored
       on the tensor-core path. */
  int32_t* cand_blocks;        /* [T, cand_topk] int32: read (consumer) or written (source) */
  int32_t cand_block_size;     /* 0 (off) or a power of two, 128 .. 65536 */
  int32_t cand_topk;           /* 1 .. 64 blocks per token */
  int32_t cand_write;          /* 0: consumer, 1: source */
} dsv4_indexer_topk_params;

size_t dsv4_indexer_topk_workspace_bytes(const dsv4_indexer_topk_params* p);
int dsv4_indexer_topk(const dsv4_indexer_topk_params* p, dsv4_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * dsv4_indexer_topk_noalloc: dsv4_indexer_topk for callers that cannot allocate device memory
 * (no cudaMalloc and no caching allocator: e.g. code embedded in a host runtime that owns all
 * device memory, or a plugin that may only touch the buffers it is handed).  The source pages
 * have no counterpart to this call; it exists for deployment only.
 * Same arguments, computation and outputs as dsv4_indexer_topk, except that `workspace` and
 * `workspace_bytes` are ignored: the scratch is a device array of DSV4_NOALLOC_SCRATCH_BYTES
 * built into the library, which every GPU that loads the library holds until the process exits.
 * The call allocates nothing.  Problems whose dsv4_indexer_topk_workspace_bytes() exceeds
 * DSV4_NOALLOC_SCRATCH_BYTES are rejected with DSV4_ERR_INVALID before any launch.
 * The first call on a device (made with that device current) looks up the array's device address
 * once and keeps it for the life of the process; make that first call outside any CUDA stream
 * capture, and do not use this call on a device after cudaDeviceReset() there (the address kept
 * belongs to the torn-down context).  Every call on a device shares the
 * one array and leaves its contents behind, so calls whose kernels overlap on the GPU (different
 * streams, or graph replays that run concurrently) race on it: order them on one stream.
 * ------------------------------------------------------------------------------------------- */
#define DSV4_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int dsv4_indexer_topk_noalloc(const dsv4_indexer_topk_params* p, dsv4_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * dsv4_sparse_mla_decode: shared-KV sparse MLA attention (MAP "Phase 3: forward_mqa()" items
 * 1-6 and "Layer-Type Summary"; API DeepseekV4Attention: sink init -inf = no effect).
 * For query token t at position p and head h, over the rows R = the window rows of the SWA
 * cache, then the compressed rows: topk_idx[t][i] for every i with 0 <= idx < n_c(p) (CSA), or
 * every j < n_c(p) when topk_idx is NULL (HCA), or none when ratio == 0 (SWA-only layer):
 *   z_i = softmax_scale * (q[t][h] . row_i) over all 576 dims
 *   out[t][h] = sum_i e^(z_i - m) row_i[0:512] / (sum_i e^(z_i - m) + e^(sink[h] - m))
 *   lse[t][h] = m + log(denominator),  m = max(max_i z_i, sink[h])
 * Rows are split across CTAs and the partial results merged (log-sum-exp weights).
 * ------------------------------------------------------------------------------------------- */
typedef struct dsv4_sparse_mla_decode_params {
  uint32_t struct_size;
  const void* q;               /* [T, H, 576] in q_dtype (F32 or BF16) */
  int32_t q_dtype;
  int32_t T, B, q_per_seq, H;  /* H <= 128 */
  const int32_t* positions;    /* [T] */
  const void* swa_cache;       /* [swa_num_pages, page_size, row] */
  const int32_t* swa_block_table; /* [B, swa_max_pages] over token positions */
  int32_t swa_max_pages;
  int64_t swa_num_pages;
  const void* main_cache;      /* [main_num_pages, page_size, row]; unused when ratio == 0 */
  const int32_t* main_block_table; /* [B, main_max_pages] over compressed indices */
  int32_t main_max_pages;
  int64_t main_num_pages;
  int32_t cache_dtype;         /* dtype of both caches: F32, BF16 or FP8_DS_MLA */
  int32_t page_size, ratio, window;
  const int32_t* topk_idx;     /* [T, topk] logical compressed indices (-1 = none) or NULL = dense */
  int32_t topk;
  const float* sink;           /* [H] per-head sink logit or NULL (= -inf) */
  float softmax_scale;
  void* out;                   /* [T, H, 512] in out_dtype (F32 or BF16) */
  int32_t out_dtype;
  float* lse;                  /* [T, H] or NULL */
  int32_t max_context;         /* host bound on positions[t] + 1 */
  void* workspace;             /* dsv4_sparse_mla_decode_workspace_bytes() bytes, 256-byte aligned */
  size_t workspace_bytes;
} dsv4_sparse_mla_decode_params;

size_t dsv4_sparse_mla_decode_workspace_bytes(const dsv4_sparse_mla_decode_params* p);
int dsv4_sparse_mla_decode(const dsv4_sparse_mla_decode_params* p, dsv4_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Utilities
 * ------------------------------------------------------------------------------------------- */
int dsv4_abi_version(void);
const char* dsv4_status_string(int status);
/* The cudaError_t of the last failed CUDA call made by this thread inside the library. */
int dsv4_last_cuda_error(void);
/* Kernels the library has enqueued since it was loaded, over all threads and devices.  A launch made
 * while the stream is being captured counts once, when it is recorded into the graph; replays of
 * that graph are not counted, so (count after - count before) around one capture is the kernels one
 * replay runs.  cudaMemsetAsync calls are not kernels of the library and are not counted. */
uint64_t dsv4_kernel_launches(void);
/* Synchronises the current device, returns the OR of the flags the kernels raised since the
 * previous call in *flags and clears them:
 *   bit 0 (1): a block-table page, slot or position out of range (the access was skipped),
 *   bit 1 (2): a top-k index out of range, or a top-k whose candidates did not fit,
 *   bit 2 (4): a bounded wait inside a kernel ran out (that call's outputs are unspecified).
 * Returns DSV4_ERR_TIMEOUT if bit 2 was set, else DSV4_ERR_BOUNDS if another bit was set, else
 * DSV4_OK (or DSV4_ERR_CUDA if the synchronisation failed). */
int dsv4_read_device_flags(uint32_t* flags);

#ifdef __cplusplus
}
#endif
#endif /* DSV4_H */
