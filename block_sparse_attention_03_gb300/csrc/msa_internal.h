// Internal launch interface between the C ABI (msa_api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/msa.h"

namespace msa {

struct DeviceStatus;

// Element formats as the kernels see them.
enum Fmt : int { FMT_BF16 = 0, FMT_FP8 = 1, FMT_NVFP4 = 2 };

// The batch as the kernels see it.  A long chunk of new tokens (prefill) is
// split into `chunks` virtual sequences of Q tokens each: virtual sequence s
// is chunk s % chunks of real sequence s / chunks, sharing its block table,
// with its length ending at the chunk's last token.  Query rows keep the real
// token-major order (virtual row s*Q + i == real row).
struct BatchDev {
  const int32_t* seq_lens;
  const int32_t* block_table;
  int32_t S, Q, max_nb;  // virtual sequences and their query tokens
  int32_t chunks;        // virtual sequences per real sequence (1: none)
  int32_t q_real;        // new tokens per real sequence (= Q * chunks)

  // length of (virtual) sequence s; -1 if its real sequence is malformed
  __device__ __forceinline__ int seq_len(int s) const {
    if (chunks == 1) return __ldg(seq_lens + s);
    const int T = __ldg(seq_lens + s / chunks);
    if (T < q_real) return -1;
    return T - q_real + Q * (s % chunks + 1);
  }
  __device__ __forceinline__ const int32_t* row(int s) const {
    return block_table + (size_t)(chunks == 1 ? s : s / chunks) * max_nb;
  }
};

// Query-fragment geometry of one MMA operand set (see msa_qfrag.cuh).
//   cols: query columns (rows of the query matrix) per unit
//   sp:   number of split terms (2: bf16 -> e4m3 hi + lo; else 1)
//   nt:   8-column tiles = ceil(cols / 8)
//   ks:   k-steps over the 128 dims (4 for e4m3 k32, 8 for 16-bit k16)
struct FragGeom {
  int32_t cols, sp, nt, ks;
  __host__ __device__ int32_t words_per_unit() const { return sp * nt * ks * 2 * 32; }
};

struct IndexerParams {
  BatchDev batch;
  int32_t G;
  int32_t num_blocks;
  const uint8_t* idx;      // raw cache (NVFP4 path)
  const uint8_t* idx_sf;   // NVFP4 scales
  const float* idx_scale;  // FP8 per-token scales
  const void* index_q;     // [S*Q][G][128] bf16 or e4m3 codes
  int32_t iq_fp8;
  float iq_scale;          // per-tensor scale of e4m3 index queries
  float col_const;         // index_scale (x NVFP4 per-tensor scale)
  int32_t nv_round;        // NVFP4 keys: e2m1 x e4m3 rounded to E4M3 (MSA_NVFP4_E4M3_PRODUCT)
  FragGeom geom;
  float* pooled;           // [S*Q][G][max_nb]
  DeviceStatus* status;
};

struct TopkParams {
  BatchDev batch;
  int32_t G, topk, init_blocks, local_blocks;
  const float* pooled;
  int32_t* topk_idx;
  float* topk_score;
  int32_t* zero;            // attend work counters to clear (nullable)
  int32_t nzero;
  // attend query fragments for unit (s, g), written when frag != null
  const void* q;
  int32_t q_fp8;
  float q_scale, col_const;
  int32_t key_fmt, r, hq;
  FragGeom geom;
  uint32_t* frag;           // [S*G][geom.words_per_unit()]
  float* colf;              // [S*G][geom.nt*8]
  DeviceStatus* status;
};

struct UnionParams {
  BatchDev batch;
  int32_t G, topk;
  const int32_t* topk_idx;  // [S*Q][G][topk]
  int32_t cap;              // Q * topk
  int32_t* u_ids;           // [S][G][cap]
  uint32_t* u_mask;         // [S][G][cap]
  int32_t* u_count;         // [S][G]
  int32_t* zero;            // attend work counters to clear (nullable)
  int32_t nzero;
  // attend query fragments for unit (s, g), written when frag != null
  const void* q;
  int32_t q_fp8;
  float q_scale, col_const;
  int32_t key_fmt, r, hq;
  FragGeom geom;
  uint32_t* frag;           // [S*G][geom.words_per_unit()]
  float* colf;              // [S*G][geom.nt*8]
  DeviceStatus* status;
};

struct AttendParams {
  BatchDev batch;
  int32_t G, r;             // groups, q heads per group
  int32_t num_blocks;
  const uint8_t* k;         // raw caches (bulk paths)
  const uint8_t* v;
  const uint8_t* k_sf;
  const uint8_t* v_sf;
  const float* k_scale;
  const float* v_scale;
  float v_global;           // NVFP4 V per-tensor scale (K's is folded into col_const)
  int32_t nv_round;         // NVFP4 K / V: e2m1 x e4m3 rounded to E4M3 (MSA_NVFP4_E4M3_PRODUCT)
  const void* q;            // [S*Q][G*r][128] bf16 or e4m3 codes
  int32_t q_fp8;
  float q_scale;
  float col_const;          // sm_scale * log2(e) (x NVFP4 K per-tensor scale)
  FragGeom geom;
  int32_t direct;           // 1: single query token, read the selection rows directly
  const int32_t* topk_idx;  // direct mode: [S][G][topk]
  int32_t topk;
  const int32_t* u_ids;     // union mode
  const uint32_t* u_mask;
  const int32_t* u_count;
  int32_t cap;
  int32_t bps;              // selected blocks per split
  int32_t splits;
  const uint32_t* frag;     // [S*G][geom.words_per_unit()] query fragments (preceding kernel)
  const float* colf;        // [S*G][geom.nt*8] column factors
  int32_t* work_ctr;        // unused
  int32_t* sg_ctr;          // [S*G] splits finished per (sequence, group), zeroed by the preceding kernel
  float* part_o;            // [S*G][splits][cols][128]
  float* part_ml;           // [S*G][splits][cols][2]
  void* out;                // bf16 [S*Q][G*r][128]
  float* lse;               // [S*Q][G*r] or null
  DeviceStatus* status;
};


// Prefill indexer on tcgen05 (FP8 index cache with per-token scales): the
// real batch (no virtual sequences), pooled [S*Q][G][max_nb].
struct PrefillIndexerParams {
  BatchDev batch;
  int32_t G;               // 1, 2, 4 or 8: 128 / G query tokens per 128-row tile
  int32_t num_blocks;
  const float* idx_scale;  // per-token fp32 scales of the index keys
  const void* index_q;     // [S*Q][G][128] bf16 or e4m3 codes
  int32_t iq_fp8;
  float iq_scale;
  float col_const;         // index_scale
  float* pooled;           // [S*Q][G][max_nb] (lists == null)
  // Selection in the epilogue (lists != null, topk <= 16, max_nb <= 65536; no pooled scores):
  // each epilogue thread keeps the 16 best free blocks (top-k rule order) of
  // the blocks it scores for its row and writes them, per query tile it
  // touched, as one list of 64-bit keys (order key of the score above, ~block
  // id below; 0 = none) at slot (s * tiles + tile) + min(CTA index, the CTA's
  // first unit): lists[slot][128 tile rows][4 epilogue groups][16].
  uint64_t* lists;
  int32_t topk, init_blocks, local_blocks;
  DeviceStatus* status;
};

// The prefill selection from the indexer's candidate lists (one warp per
// (token, group) row): the row's free blocks with the kfree largest keys, plus
// the forced ones, ascending, as topk_kernel writes them.
struct PiSelectParams {
  BatchDev batch;            // the real batch
  int32_t G, topk, init_blocks, local_blocks;
  int32_t grid;              // CTAs of the indexer launch that wrote the lists
  const uint64_t* lists;
  int32_t* topk_idx;         // [S*Q][G][topk]
  DeviceStatus* status;
};

// Key-block-major attend of prefill chunks (the selections inverted into one
// list per (sequence, group, block) of the (token, slot) pairs that chose it).
struct K2qParams {
  BatchDev batch;            // the real batch: S sequences, Q new tokens each
  int32_t G, r, topk;
  int32_t num_blocks;
  const int32_t* topk_idx;   // [S*Q][G][topk]
  int32_t* cnt;              // [L = S*G*max_nb] pairs per list (zeroed before the count)
  int32_t* off;              // [L] first entry of each list
  int32_t* cur;              // [L] fill cursors
  int32_t* item_off;         // [L + 1] first attend item of each list; [L] = items in all
  int32_t* entries;          // [S*Q*G*topk] token * 32 + slot, list by list
  int32_t* item_list;        // [S*Q*G*topk] (at most one item per entry) the list of each attend item
  int32_t item_tokens;       // entries (tokens) per attend item: 128 / r, one MMA row per (token, head)
  const float* k_scale;      // FP8 per-token scales
  const float* v_scale;
  const void* q;             // [S*Q][G*r][128]
  int32_t q_fp8;
  float q_scale, col_const;
  uint8_t* qsplit;           // bf16 query: [S*Q*G*r][2][128] e4m3 hi, lo terms of q x 2^e (per row)
  float* qrowf;              // [S*Q*G*r] 2^-e x col_const
  uint16_t* part_o;          // [S*Q][topk][G*r][128] fp16 o / l x 2^-ev of each (token, slot, head);
                             // 16-byte chunk c of a row is stored at chunk c ^ (head % r)
  float* part_ml;            // [S*Q][topk][G*r][4]: m, l, 2^ev, unused
  void* out;                 // bf16 [S*Q][G*r][128]
  float* lse;
  DeviceStatus* status;
};

// Cache insert of new tokens (bf16 rows in, the caches' formats out).
struct InsertParams {
  int32_t num_tokens, H, num_blocks;
  int32_t kv_fmt, idx_fmt;
  const int32_t* slots;       // [num_tokens] physical block * 128 + offset, < 0: skip
  const __nv_bfloat16* k;     // [num_tokens][H][128]
  const __nv_bfloat16* v;
  const __nv_bfloat16* ik;    // [num_tokens][128] or null
  uint8_t *kc, *vc, *ic;      // cache data
  float *ks, *vs, *is;        // FP8 per-token scales
  uint8_t *ksf, *vsf, *isf;   // NVFP4 e4m3 scales
  float kg, vg, ig;           // NVFP4 per-tensor scales
  DeviceStatus* status;
};

// launchers (return cudaGetLastError())
cudaError_t launch_insert(const InsertParams& p, int num_sms, cudaStream_t st);
cudaError_t launch_k2q_build(const K2qParams& p, int num_sms, cudaStream_t st);    // count, scan, fill
cudaError_t launch_k2q_attend(const CUtensorMap* tk, const CUtensorMap* tv, const K2qParams& p, int num_sms,
                              cudaStream_t st);
cudaError_t launch_k2q_combine(const K2qParams& p, int num_sms, cudaStream_t st);
cudaError_t launch_prefill_indexer(const CUtensorMap* tmap, const PrefillIndexerParams& p, int num_sms,
                                   cudaStream_t st);
// the prefill indexer's grid (one CTA per SM)
int prefill_indexer_grid(int num_sms);
cudaError_t launch_prefill_select(const PiSelectParams& p, cudaStream_t st);
cudaError_t launch_indexer(int fmt, const CUtensorMap* tmap, const IndexerParams& p, int num_sms, cudaStream_t st,
                           bool pdl);
cudaError_t launch_topk(const TopkParams& p, cudaStream_t st, bool pdl);
// one warp per row (K <= 32; no scores, no fragment or counter job)
cudaError_t launch_topk_warp(const TopkParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_union(const UnionParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_attend(int fmt, const CUtensorMap* tmap_k, const CUtensorMap* tmap_v, const AttendParams& p,
                          int num_sms, cudaStream_t st, bool pdl);
// Blocks per split of the attend: the (sequence, group) units are cut into
// about as many splits as there are CTA slots on the GPU (slots / units
// splits each), so every CTA gets about one split; 2 to 16 blocks a split
// (a split of one block costs more in its partial and merge than it saves).
constexpr int kMaxBlocksPerSplit = 16;
inline int attend_blocks_per_split(int cap_blocks, long units, int cta_slots) {
  long want = units > 0 ? cta_slots / units : 1;
  if (want < 1) want = 1;
  int bps = (int)((cap_blocks + want - 1) / want);
  if (bps < 2) bps = 2;
  return bps > kMaxBlocksPerSplit ? kMaxBlocksPerSplit : bps;
}
cudaError_t launch_dequant(int fmt, int which, const msa_cache_t& c, const int32_t* phys, int32_t n, float* out,
                           cudaStream_t st);

// host-side limits shared with the API
constexpr int kMaxIndexerNT = 8;   // up to 64 (query x group) columns in the decode indexer
constexpr int kMaxAttendCols = 32; // up to 32 (query x head) columns per attend unit

}  // namespace msa
