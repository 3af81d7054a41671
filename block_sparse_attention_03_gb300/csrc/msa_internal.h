// Internal launch interface between the C ABI (msa_api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/msa.h"

namespace msa {

struct DeviceStatus;

// Element formats as the kernels see them.
enum Fmt : int { FMT_BF16 = 0, FMT_FP8 = 1, FMT_NVFP4 = 2 };

struct BatchDev {
  const int32_t* seq_lens;
  const int32_t* block_table;
  int32_t S, Q, max_nb;
};

// Query-fragment geometry of one MMA operand set (see msa_prep.cu).
//   cols: query columns (rows of the query matrix) per unit
//   sp:   number of split terms (2: bf16 -> e4m3 hi + lo; else 1)
//   nt:   8-column tiles = ceil(cols / 8)
//   ks:   k-steps over the 128 dims (4 for e4m3 k32, 8 for 16-bit k16)
struct FragGeom {
  int32_t cols, sp, nt, ks;
  __host__ __device__ int32_t words_per_unit() const { return sp * nt * ks * 2 * 32; }
};

struct PrepParams {
  const void* q;       // [units][cols][128] queries (bf16 or e4m3 codes)
  int32_t q_is_fp8;
  float q_scale;       // per-tensor scale of e4m3 queries
  float col_const;     // extra constant folded into every column factor
  int32_t key_fmt;     // operand format of the other side (Fmt)
  FragGeom geom;
  int32_t units;
  uint32_t* frag;      // [units][words_per_unit]
  float* colf;         // [units][nt * 8]
};

struct IndexerParams {
  BatchDev batch;
  int32_t G;
  int32_t num_blocks;
  const uint8_t* idx;      // raw cache (NVFP4 path)
  const uint8_t* idx_sf;   // NVFP4 scales
  const float* idx_scale;  // FP8 per-token scales
  const uint32_t* qfrag;   // [S][words]
  const float* colf;       // [S][nt*8]
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
  float v_global;           // NVFP4 V per-tensor scale (K's is folded into colf)
  const uint32_t* qfrag;    // [S*G][words]
  const float* colf;        // [S*G][nt*8]  (log2-domain logit factor per column)
  FragGeom geom;
  const int32_t* u_ids;
  const uint32_t* u_mask;
  const int32_t* u_count;
  int32_t cap;
  int32_t bps;              // union blocks per split
  int32_t splits;
  float* part_o;            // [S*G][splits][cols][128]
  float* part_ml;           // [S*G][splits][cols][2]
  DeviceStatus* status;
};

struct CombineParams {
  int32_t S, Q, G, r, splits, cols;
  const float* part_o;
  const float* part_ml;
  void* out;   // bf16 [S*Q][G*r][128]
  float* lse;  // [S*Q][G*r] or null
};

// launchers (return cudaGetLastError())
cudaError_t launch_prep_rows(const PrepParams& p, int a, int u2, int b, int c2, int c, cudaStream_t st);
int attend_max_stages(int fmt);
cudaError_t launch_indexer(int fmt, const CUtensorMap* tmap, const IndexerParams& p, int num_sms, cudaStream_t st,
                           bool pdl);
cudaError_t launch_topk(const TopkParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_union(const UnionParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_attend(int fmt, const CUtensorMap* tmap_k, const CUtensorMap* tmap_v, const AttendParams& p,
                          cudaStream_t st, bool pdl);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_dequant(int fmt, int which, const msa_cache_t& c, const int32_t* phys, int32_t n, float* out,
                           cudaStream_t st);

// host-side limits shared with the API
constexpr int kMaxIndexerNT = 8;   // up to 64 (query x group) columns in the decode indexer
constexpr int kMaxAttendCols = 32; // up to 32 (query x head) columns per attend unit

}  // namespace msa
