/*
 * msa.h -- C ABI of libmsa: the MiniMax Sparse Attention (MSA) decode hot path
 * on one GB300 (sm_103a).
 *
 * What the path computes (vLLM blog "vLLM 实现 MiniMax-M3.1-Flash 的 Day-0 支持",
 * section "MSA 入门" and its Figure 1):
 *   1. a lightweight indexer scores every key of the paged context with one
 *      index query per GQA group against one shared 128-dim index-key head;
 *   2. the per-key scores are max-pooled to one score per 128-token block;
 *   3. per group the top-k blocks (k = 16 in the model) are kept, the most
 *      recent block always among them;
 *   4. exact softmax attention runs for every query head of the group over
 *      only the selected blocks (at most k x 128 keys).
 * The index scale and the softmax scale are both head_dim ** -0.5 in the model
 * (API page "vllm.models.minimax_m3.nvidia.model", MiniMaxM3SparseAttention:
 * the indexer is built with scale=self.scaling).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer inside the structs and every tensor argument is DEVICE
 *   memory of the current CUDA device unless stated otherwise.  The caller
 *   owns every buffer, the workspace included; the library allocates nothing
 *   and keeps no state beyond cached device attributes.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *   stream) and never synchronise the host, except msa_read_device_status.
 * - Host-checkable problems (null pointers, unsupported sizes or dtypes, a
 *   workspace that is too small) return an error before any launch.
 *   Launch failures return MSA_ERR_CUDA.  Data-dependent faults found on the
 *   device (a block-table entry outside [0, num_blocks), a sequence length
 *   outside [q_per_seq, max_blocks_per_seq * 128], a selected block id the
 *   query cannot see) set a sticky status word in the workspace; the kernels
 *   skip the offending work (outputs for it are left as documented below)
 *   and never trap.  msa_read_device_status reports and clears that word.
 * - Query token i (0-based) of the q_per_seq new tokens of sequence s sits at
 *   position seq_lens[s] - q_per_seq + i; its keys are already in the cache.
 *   Key t is visible to it iff t <= that position.
 * - Rows of per-query tensors are token-major: row = s * q_per_seq + i.
 *
 * Paged-cache layout (one physical block = 128 tokens; all dims = 128):
 *   K, V        BF16 / FP8: [num_blocks][num_kv_heads][128][head_dim] elements
 *               NVFP4: [num_blocks][num_kv_heads][128][head_dim/2] bytes, element
 *               2j in the low nibble of byte j; e4m3 scales k_sf / v_sf
 *               [num_blocks][num_kv_heads][128][head_dim/16] (one per 16
 *               consecutive elements), fp32 per-tensor k_global / v_global.
 *   FP8 scales  k_scale, v_scale: fp32 [num_blocks][num_kv_heads][128]
 *               (value = e4m3 * scale of its token and head).
 *   index keys  one shared head: [num_blocks][128][index_dim] (BF16 / FP8) or
 *               [num_blocks][128][index_dim/2] bytes + idx_sf
 *               [num_blocks][128][index_dim/16] (NVFP4); FP8 per-token fp32
 *               idx_scale [num_blocks][128]; NVFP4 per-tensor idx_global.
 *   The index cache is addressed with the same block table as K/V.
 *   Every base pointer must be 16-byte aligned.
 * Formats: FP8 = OCP E4M3 ("FN": bias 7, no inf); NVFP4 = e2m1 values, one
 * e4m3 scale per 16 elements, one fp32 per-tensor scale (Day-0 blog, section
 * "MiniMax-M3.1 架构中的新特性").  The fp32 value of an NVFP4 element is
 * fp32(e2m1 * e4m3_scale) * global (the inner product is exact in fp32).
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MSA_BLOCK_SIZE 128
#define MSA_HEAD_DIM 128

typedef struct CUstream_st* msa_stream_t; /* == cudaStream_t */

typedef enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARGUMENT = 1,   /* null pointer, bad size, misaligned base */
  MSA_ERR_UNSUPPORTED = 2,        /* valid but not implemented (dtype, topk, dims) */
  MSA_ERR_WORKSPACE_TOO_SMALL = 3,
  MSA_ERR_CUDA = 4,               /* a CUDA launch or copy failed */
  MSA_ERR_DEVICE_FAULT = 5,       /* a kernel found bad data (see status word) */
  MSA_ERR_TIMEOUT = 6             /* a bounded on-device wait gave up */
} msa_status_t;

typedef enum {
  MSA_DTYPE_BF16 = 0,
  MSA_DTYPE_FP8_E4M3 = 1,
  MSA_DTYPE_NVFP4 = 2
} msa_dtype_t;

/* How an NVFP4 element's two factors combine (vLLM Day-0 blog, "NVIDIA
 * Blackwell 优化的 MSA 内核": the Blackwell kernels dequantize NVFP4 to FP8 with
 * mul.e4m3x4.e2m1x4.e4m3x4, i.e. the product is rounded to E4M3).
 *   MSA_NVFP4_EXACT          e2m1 x e4m3 block scale exactly (it has at most six
 *                            significant bits), then x the fp32 per-tensor scale;
 *   MSA_NVFP4_E4M3_PRODUCT   the product rounded to E4M3 (nearest, ties to even,
 *                            saturating at +-448) first, as that dequant does. */
typedef enum {
  MSA_NVFP4_EXACT = 0,
  MSA_NVFP4_E4M3_PRODUCT = 1
} msa_nvfp4_mode_t;

/* The paged K/V cache and the index-key side cache of one attention layer.
 * K/V dtype and index dtype are independent (the model's
 * --kv-cache-dtype and indexer_kv_dtype settings).  Unused pointers (scales of
 * another format) may be NULL. */
typedef struct {
  msa_dtype_t kv_dtype;
  msa_dtype_t index_dtype;
  int32_t num_blocks;   /* physical blocks in the pool */
  int32_t block_size;   /* must be 128 */
  int32_t num_kv_heads; /* = number of GQA groups = number of index queries per token */
  int32_t head_dim;     /* must be 128 */
  int32_t index_dim;    /* must be 128 */
  const void* k;
  const void* v;
  const void* k_sf;     /* NVFP4 only */
  const void* v_sf;     /* NVFP4 only */
  const float* k_scale; /* FP8 only */
  const float* v_scale; /* FP8 only */
  const void* idx;
  const void* idx_sf;     /* NVFP4 only */
  const float* idx_scale; /* FP8 only */
  float k_global;       /* NVFP4 only */
  float v_global;
  float idx_global;
  int32_t nvfp4_mode;   /* msa_nvfp4_mode_t, for every NVFP4 tensor of the cache (0 = exact) */
} msa_cache_t;

/* The batch: num_seqs sequences with q_per_seq new query tokens each.
 * seq_lens[s] counts every token of sequence s, the new ones included.
 * block_table[s][b] is the physical block holding logical block b of s. */
typedef struct {
  int32_t num_seqs;
  int32_t q_per_seq;
  int32_t max_blocks_per_seq;   /* row stride of block_table */
  const int32_t* seq_lens;      /* device int32 [num_seqs] */
  const int32_t* block_table;   /* device int32 [num_seqs][max_blocks_per_seq] */
} msa_batch_t;

/* How the per-key index scores of a block pool into the block's score: the
 * indexer's score_type argument (API page "vllm.models.minimax_m3.nvidia.model",
 * MiniMaxM3SparseAttention.__init__: score_type=sparse_cfg.get(
 * "sparse_score_type", "max")).  The pages define only "max"; any other value
 * returns MSA_ERR_UNSUPPORTED. */
typedef enum {
  MSA_SCORE_MAX = 0
} msa_score_type_t;

/* Where msa_decode selects the blocks of a prefill chunk over FP8 caches (more
 * than 8 new tokens a sequence, the tcgen05 indexer).  The selection is the same
 * either way, bit for bit; the two differ in time and workspace. */
typedef enum {
  /* the indexer writes every pooled score, a top-k launch reads them back
     (default: the faster of the two on a 64K-token context) */
  MSA_PREFILL_SELECT_TOPK = 0,
  /* the indexer's epilogue keeps each row's 16 best free blocks as candidate
     lists and a merge launch picks from them: no pooled scores, so the
     workspace does not grow with the context length; topk <= 16 (otherwise,
     and in msa_decode_noalloc when the lists do not fit, the top-k launch) */
  MSA_PREFILL_SELECT_INDEXER = 1
} msa_prefill_select_t;

/* Method settings (the indexer's constructor arguments in the model). */
typedef struct {
  int32_t topk;         /* blocks kept per (query, group): 4, 8, 16 or 32 */
  int32_t init_blocks;  /* leading blocks always kept (model default 0) */
  int32_t local_blocks; /* blocks just before the query's own block always kept (default 0) */
  float index_scale;    /* multiplies the index scores; model: index_dim ** -0.5 */
  float sm_scale;       /* softmax scale; model: head_dim ** -0.5 */
  int32_t score_type;   /* msa_score_type_t; 0 (max) in a zero-initialised struct */
  int32_t prefill_select; /* msa_prefill_select_t; 0 (top-k launch) in a zero-initialised struct */
} msa_config_t;

/* A query tensor: BF16, or FP8 E4M3 codes times one fp32 per-tensor scale. */
typedef struct {
  const void* data;
  msa_dtype_t dtype; /* MSA_DTYPE_BF16 or MSA_DTYPE_FP8_E4M3 */
  float scale;       /* FP8 only */
} msa_query_t;

/* Bytes of workspace msa_decode (and each of the other entry points) needs
 * for this problem.  Host-only; returns 0 for an invalid description.  A
 * prefill chunk (more than 8 new tokens a sequence) over an FP8 cache also
 * holds one partial per (token, q head, selected block) -- o / l in fp16 (with
 * a power-of-two scale that keeps it in range), m, l and that scale in fp32:
 * 272 bytes x tokens x q heads x topk, and with a bf16 query its rows as two
 * e4m3 terms and a factor: 260 bytes x tokens x q heads (605 MB in all for
 * 8,192 tokens x 16 heads x 16). */
size_t msa_workspace_size(const msa_cache_t* cache, const msa_batch_t* batch,
                          const msa_config_t* cfg, int32_t num_q_heads);

/* Clear the device status word at the start of a (fresh) workspace.  Call once
 * after allocating a workspace; the word is sticky across calls until read. */
msa_status_t msa_workspace_init(void* workspace, size_t workspace_bytes, msa_stream_t stream);

/* Indexer score + block max-pool (steps 1-2 above).
 * index_q: [num_seqs * q_per_seq][num_kv_heads][index_dim].
 * pooled:  fp32 [num_seqs * q_per_seq][num_kv_heads][max_blocks_per_seq];
 *          pooled[row][g][b] = index_scale * max over the keys t of block b
 *          visible to that query of <index_q[row][g], index_key[t]>, and -inf
 *          for a block with no visible key (and for b >= the sequence's block
 *          count).  Rows of a sequence with a device fault are left -inf. */
msa_status_t msa_indexer_score(const msa_cache_t* cache, const msa_batch_t* batch,
                               const msa_config_t* cfg, const msa_query_t* index_q,
                               float* pooled, void* workspace, size_t workspace_bytes,
                               msa_stream_t stream);

/* Top-k block selection (step 3) from pooled scores laid out as above.
 * The output keeps the token-major layout of the model's shared top-k buffer
 * (API page "vllm.models.minimax_m3.nvidia.model", MiniMaxM3Model: the
 * indexer writes [tokens, index heads, topk] int32 block ids that the attend
 * reads back).
 * topk_idx:   int32 [num_seqs * q_per_seq][num_groups][topk], the query's own
 *             block ⌊pos/128⌋ always included (forced, together with the
 *             init/local blocks), the remaining slots filled with the highest
 *             pooled scores of the earlier blocks (equal scores: smaller block
 *             id first), ascending, padded with -1 when fewer blocks exist.
 * topk_score: optional fp32 [same shape], the pooled score of each entry
 *             (-inf for padding); may be NULL. */
msa_status_t msa_topk_blocks(const msa_batch_t* batch, const msa_config_t* cfg,
                             int32_t num_groups, const float* pooled, int32_t* topk_idx,
                             float* topk_score, void* workspace, size_t workspace_bytes,
                             msa_stream_t stream);

/* Sparse attend (step 4): for query head h of group g = h / (num_q_heads /
 * num_kv_heads), exact softmax attention over the visible keys of the blocks
 * topk_idx[row][g][*] (entries < 0 are skipped), logits scaled by sm_scale.
 * q:   [num_seqs * q_per_seq][num_q_heads][head_dim].
 * out: bf16 [num_seqs * q_per_seq][num_q_heads][head_dim] (caller-allocated).
 * lse: optional fp32 [num_seqs * q_per_seq][num_q_heads], natural-log
 *      log-sum-exp of the scaled logits; may be NULL.
 * A row whose selection holds no visible key gets out = 0, lse = -inf.
 * Entries naming a block the query cannot see, or repeating a block an
 * earlier entry of the same row names, are left out and raise the device
 * fault flag: the softmax runs over the selected key set, each key once. */
msa_status_t msa_sparse_attend(const msa_cache_t* cache, const msa_batch_t* batch,
                               const msa_config_t* cfg, const msa_query_t* q,
                               int32_t num_q_heads, const int32_t* topk_idx, void* out,
                               float* lse, void* workspace, size_t workspace_bytes,
                               msa_stream_t stream);

/* The whole path in one call on one stream (score -> pool -> top-k -> attend),
 * no host synchronisation.  topk_idx (output, layout as in msa_topk_blocks)
 * receives the selection; out / lse as in msa_sparse_attend. */
msa_status_t msa_decode(const msa_cache_t* cache, const msa_batch_t* batch,
                        const msa_config_t* cfg, const msa_query_t* index_q,
                        const msa_query_t* q, int32_t num_q_heads, int32_t* topk_idx,
                        void* out, float* lse, void* workspace, size_t workspace_bytes,
                        msa_stream_t stream);

/* Cache insert: write the K, V and index key of num_tokens new tokens into
 * the paged caches, quantized to the caches' formats -- the step just before
 * the path (Day-0 blog, section "QKV GEMM + norm + RoPE + KV 插入融合": K, V and
 * the index key are quantized and written straight into their caches; PR
 * "[M3] Enable FP8 sparse GQA", items 1 and 4: FP8 values stored through the
 * slot mapping).
 * slot_mapping: device int32 [num_tokens]; token t goes to physical block
 *   slot / 128, row slot % 128; negative entries are skipped (padding);
 *   entries at or beyond num_blocks * 128 raise the device fault flag
 *   (MSA_ERR_DEVICE_FAULT from msa_read_device_status) and are skipped.
 * k, v: device bf16 [num_tokens][num_kv_heads][head_dim]; index_k: device bf16
 *   [num_tokens][index_dim], or NULL to leave the index cache alone.  16-byte
 *   aligned.
 * Formats (per 128-element row, all arithmetic one fp32 operation each):
 *   BF16   the bits are copied;
 *   FP8    scale = amax / 448 (1 for an all-zero row) into k_scale / v_scale /
 *          idx_scale, codes = E4M3(x / scale), round to nearest even,
 *          saturating at +-448, the sign of a zero kept;
 *   NVFP4  with the cache's per-tensor k_global / v_global / idx_global g
 *          (the caller's calibrated scale), per 16 elements
 *          sf = E4M3(amax16 / (6 g)) into k_sf / v_sf / idx_sf and codes =
 *          E2M1(x / (sf * g)) (0 where sf * g = 0), round to nearest even,
 *          saturating at +-6, a value that rounds to zero stored as +0;
 *          element 2j in the low nibble of byte j.
 * The call writes through the cache struct's data and scale pointers (they are
 * declared const for the read-only entry points).  workspace: at least 256
 * bytes; only its status word is used.  Rows of one token may be written in
 * any order; two tokens mapped to one slot race. */
msa_status_t msa_cache_insert(const msa_cache_t* cache, int32_t num_tokens, const int32_t* slot_mapping,
                              const void* k, const void* v, const void* index_k, void* workspace,
                              size_t workspace_bytes, msa_stream_t stream);

/* Synchronise `stream`, read and clear the workspace's status word.
 * Returns MSA_OK, MSA_ERR_DEVICE_FAULT or MSA_ERR_TIMEOUT; *detail (optional,
 * host pointer) receives the raw flag bits. */
msa_status_t msa_read_device_status(void* workspace, msa_stream_t stream, int32_t* detail);

/* Static, human-readable name of a status code. */
const char* msa_status_string(msa_status_t status);

/* Test hook: the fp32 value of every element of the given physical blocks.
 * which: 0 = K, 1 = V (out fp32 [n][num_kv_heads][128][head_dim]),
 *        2 = index keys (out fp32 [n][128][index_dim]).
 * phys_blocks: device int32 [n].  Entries outside [0, num_blocks) produce NaN
 * rows.  The values are bit-identical to the definition in the format notes
 * above (one fp32 rounding for FP8 and NVFP4). */
msa_status_t msa_dequant_debug(const msa_cache_t* cache, int32_t which,
                               const int32_t* phys_blocks, int32_t n, float* out,
                               msa_stream_t stream);

/* Allocation-free variant of msa_decode (no counterpart in the paper; a
 * deployment convenience).  Some callers cannot allocate device memory for a
 * workspace: code running inside another framework's memory pool, a plugin
 * that must not call cudaMalloc (or a framework allocator) on its hot path, a
 * process whose device memory is reserved up front.  This entry point uses a
 * fixed scratch array inside the library instead of a caller workspace; it
 * allocates nothing and calls no allocating routine.
 *   - Limit: the problem's msa_workspace_size must be at most
 *     MSA_NOALLOC_SCRATCH_BYTES (8 MiB, held on every GPU that loads the
 *     library until the process exits); larger problems return
 *     MSA_ERR_WORKSPACE_TOO_SMALL before any launch.
 *   - The first call on each device looks up the scratch's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *     The address is kept for the life of the process: resetting the device
 *     (cudaDeviceReset) and calling again is not supported.
 *   - Every call shares the one scratch array, which keeps the last call's
 *     contents; each call clears what must start at zero.  Calls that overlap
 *     on the GPU (other streams, other host threads) race on it: serialise them.
 *   - status_out: optional device int32[2]; receives this call's device status
 *     flags (the same bits msa_read_device_status reports) at the end of the call.
 * Arguments, outputs and errors are otherwise those of msa_decode. */
#define MSA_NOALLOC_SCRATCH_BYTES (8u << 20)
msa_status_t msa_decode_noalloc(const msa_cache_t* cache, const msa_batch_t* batch,
                                const msa_config_t* cfg, const msa_query_t* index_q,
                                const msa_query_t* q, int32_t num_q_heads, int32_t* topk_idx,
                                void* out, float* lse, int32_t* status_out, msa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
