// C ABI of libmsa (declared in include/msa.h): argument checks, workspace
// carving, TMA descriptor encoding and the launch chains of each entry point.
#include <cmath>
#include <cstring>
#include <mutex>

#include "msa_device.cuh"
#include "msa_internal.h"

using namespace msa;

namespace {

// ---------------------------------------------------------------- device facts

int sm_count() {
  static int cache[64];
  static bool init[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!init[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
    init[dev] = true;
  }
  return cache[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D map over rows of 128 elements (FP8: 128 B, BF16: 256 B); one box is
// 128 rows x 128 bytes with the 128-byte swizzle.
bool encode_rows(CUtensorMap* m, const void* base, long rows, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {bf16 ? 256ull : 128ull};
  cuuint32_t box[2] = {bf16 ? 64u : 128u, 128u};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- checks

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int fmt_of(msa_dtype_t d) {
  switch (d) {
    case MSA_DTYPE_BF16: return FMT_BF16;
    case MSA_DTYPE_FP8_E4M3: return FMT_FP8;
    case MSA_DTYPE_NVFP4: return FMT_NVFP4;
    default: return -1;
  }
}

int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

msa_status_t check_batch(const msa_batch_t* b) {
  if (!b || !b->seq_lens || !b->block_table) return MSA_ERR_INVALID_ARGUMENT;
  if (b->num_seqs < 1 || b->q_per_seq < 1 || b->max_blocks_per_seq < 1) return MSA_ERR_INVALID_ARGUMENT;
  if ((long)b->max_blocks_per_seq * kBlock > (1l << 30)) return MSA_ERR_UNSUPPORTED;
  if ((long)b->q_per_seq > (long)b->max_blocks_per_seq * kBlock) return MSA_ERR_INVALID_ARGUMENT;
  return MSA_OK;
}

msa_status_t check_cfg(const msa_config_t* c) {
  if (!c) return MSA_ERR_INVALID_ARGUMENT;
  if (c->topk != 4 && c->topk != 8 && c->topk != 16 && c->topk != 32) return MSA_ERR_UNSUPPORTED;
  if (c->init_blocks < 0 || c->local_blocks < 0 || c->init_blocks + c->local_blocks > c->topk - 1)
    return MSA_ERR_INVALID_ARGUMENT;
  if (!(c->index_scale > 0.f) || !std::isfinite(c->index_scale)) return MSA_ERR_INVALID_ARGUMENT;
  if (!(c->sm_scale > 0.f) || !std::isfinite(c->sm_scale)) return MSA_ERR_INVALID_ARGUMENT;
  if (c->score_type != MSA_SCORE_MAX) return MSA_ERR_UNSUPPORTED;
  if (c->prefill_select != MSA_PREFILL_SELECT_TOPK && c->prefill_select != MSA_PREFILL_SELECT_INDEXER)
    return MSA_ERR_INVALID_ARGUMENT;
  return MSA_OK;
}

msa_status_t check_cache(const msa_cache_t* c, bool need_index, bool need_kv) {
  if (c && c->nvfp4_mode != MSA_NVFP4_EXACT && c->nvfp4_mode != MSA_NVFP4_E4M3_PRODUCT) return MSA_ERR_INVALID_ARGUMENT;
  if (!c) return MSA_ERR_INVALID_ARGUMENT;
  if (c->block_size != kBlock || c->head_dim != kDim || c->index_dim != kDim) return MSA_ERR_UNSUPPORTED;
  if (c->num_kv_heads < 1 || c->num_kv_heads > 8) return MSA_ERR_UNSUPPORTED;
  if (c->num_blocks < 1 || (long)c->num_blocks * c->num_kv_heads * kBlock >= (1l << 31)) return MSA_ERR_UNSUPPORTED;
  if (need_index) {
    const int f = fmt_of(c->index_dtype);
    if (f < 0) return MSA_ERR_UNSUPPORTED;
    if (!c->idx || !aligned16(c->idx)) return MSA_ERR_INVALID_ARGUMENT;
    if (f == FMT_FP8 && (!c->idx_scale || !aligned16(c->idx_scale))) return MSA_ERR_INVALID_ARGUMENT;
    if (f == FMT_NVFP4 && (!c->idx_sf || !aligned16(c->idx_sf) || !(c->idx_global > 0.f))) return MSA_ERR_INVALID_ARGUMENT;
  }
  if (need_kv) {
    const int f = fmt_of(c->kv_dtype);
    if (f < 0) return MSA_ERR_UNSUPPORTED;
    if (!c->k || !c->v || !aligned16(c->k) || !aligned16(c->v)) return MSA_ERR_INVALID_ARGUMENT;
    if (f == FMT_FP8 && (!c->k_scale || !c->v_scale || !aligned16(c->k_scale) || !aligned16(c->v_scale)))
      return MSA_ERR_INVALID_ARGUMENT;
    if (f == FMT_NVFP4 && (!c->k_sf || !c->v_sf || !aligned16(c->k_sf) || !aligned16(c->v_sf) ||
                           !(c->k_global > 0.f) || !(c->v_global > 0.f)))
      return MSA_ERR_INVALID_ARGUMENT;
  }
  return MSA_OK;
}

msa_status_t check_query(const msa_query_t* q) {
  if (!q || !q->data || !aligned16(q->data)) return MSA_ERR_INVALID_ARGUMENT;
  if (q->dtype != MSA_DTYPE_BF16 && q->dtype != MSA_DTYPE_FP8_E4M3) return MSA_ERR_UNSUPPORTED;
  if (q->dtype == MSA_DTYPE_FP8_E4M3 && !(q->scale > 0.f && std::isfinite(q->scale))) return MSA_ERR_INVALID_ARGUMENT;
  return MSA_OK;
}

// ---------------------------------------------------------------- workspace plan

FragGeom geom_for(int key_fmt, bool q_fp8, int cols) {
  FragGeom g;
  g.cols = cols;
  g.sp = (key_fmt == FMT_FP8 && !q_fp8) ? 2 : 1;
  g.ks = (key_fmt == FMT_FP8) ? 4 : 8;
  g.nt = next_pow2((cols + 7) / 8);
  return g;
}

struct Plan {
  int S = 0, Q = 0, chunks = 1;  // indexer: sequences / query tokens as it sees them (long chunks split)
  int Sa = 0, Qa = 0, chunks_a = 1;  // the same for the attend
  FragGeom gi, ga;          // indexer / attend query geometry
  int bps = 0, splits = 0, cap = 0, r = 0;
  bool direct = false;      // one query token: the attend reads the selection rows directly
  size_t off_status = 0, off_pooled = 0, off_uids = 0, off_umask = 0, off_ucount = 0, off_ctr = 0, off_qfa = 0,
         off_cfa = 0, off_po = 0, off_pml = 0, total = 0;
  int nctr = 0;             // attend counters: splits finished per (sequence, group)
  // prefill chunks over an FP8 cache: the key-block-major attend (selection lists,
  // one partial per (token, head, slot), a combine pass)
  bool k2q = false;
  // ... whose selection the tcgen05 indexer makes in its epilogue (candidate
  // lists and a merge launch instead of the pooled scores and a top-k launch)
  bool pisel = false;
  size_t off_plists = 0;
  size_t off_kcnt = 0, off_koff = 0, off_kcur = 0, off_kitem = 0, off_kent = 0, off_klist = 0, off_kpo = 0,
         off_kpml = 0, off_kq = 0, off_kqf = 0;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// A prefill chunk (more than 8 new tokens a sequence) over an FP8 index
// cache: the tcgen05 indexer, with the query tokens as the MMA's M side.
bool tc_indexer(const msa_cache_t* c, const msa_batch_t* b) {
  const int G = c->num_kv_heads;
  return fmt_of(c->index_dtype) == FMT_FP8 && b->q_per_seq > 8 && (G == 1 || G == 2 || G == 4 || G == 8);
}

// Plan for the given problem.  iq_fp8 / q_fp8: query dtypes (E4M3 or bf16).
msa_status_t make_plan(const msa_cache_t* c, const msa_batch_t* b, const msa_config_t* cfg, int hq, bool iq_fp8,
                       bool q_fp8, Plan& pl, bool allow_pisel = true) {
  // more than 8 new tokens per sequence (a prefill chunk): split into virtual
  // sequences of the largest of 8, 4, 2, 1 tokens dividing the count
  int QV = b->q_per_seq;
  if (QV > 8) {
    QV = 8;
    while (b->q_per_seq % QV) QV >>= 1;
  }
  pl.chunks = b->q_per_seq / QV;
  pl.S = b->num_seqs * pl.chunks;
  pl.Q = QV;
  // The attend runs every new token as its own one-token sequence (speculative
  // verify and prefill chunks alike): the tokens' selections overlap little, so
  // a union over 8 tokens streams each block for 32 query columns of which
  // about 4 chose it, four times the work per block for the few blocks saved.
  pl.Qa = 1;
  pl.chunks_a = b->q_per_seq / pl.Qa;
  pl.Sa = b->num_seqs * pl.chunks_a;
  const int Q = pl.Q, G = c->num_kv_heads;
  const int S = pl.Sa, Qa = pl.Qa;  // the attend's units size the buffers below
  if (hq < G || hq % G != 0) return MSA_ERR_INVALID_ARGUMENT;
  pl.r = hq / G;
  const int fi = fmt_of(c->index_dtype), fa = fmt_of(c->kv_dtype);
  pl.gi = geom_for(fi < 0 ? FMT_FP8 : fi, iq_fp8, Q * G);
  pl.ga = geom_for(fa < 0 ? FMT_FP8 : fa, q_fp8, Qa * pl.r);
  if (!tc_indexer(c, b) && (pl.gi.nt > kMaxIndexerNT || pl.gi.nt * pl.gi.sp > 8)) return MSA_ERR_UNSUPPORTED;
  if (pl.ga.cols > kMaxAttendCols || pl.ga.nt * pl.ga.sp > 8) return MSA_ERR_UNSUPPORTED;
  pl.cap = Qa * cfg->topk;
  pl.direct = (Qa == 1);
  // a union never holds more blocks than a sequence has
  const int cap_eff = pl.cap < b->max_blocks_per_seq ? pl.cap : b->max_blocks_per_seq;
  pl.bps = attend_blocks_per_split(cap_eff, (long)S * G, 2 * sm_count());
  pl.splits = (cap_eff + pl.bps - 1) / pl.bps;
  pl.nctr = S * G;  // splits finished per (sequence, group)
  size_t o = 0;
  pl.off_status = o; o = align256(o + 256);
  pl.k2q = fa == FMT_FP8 && b->q_per_seq > 8 && (pl.r == 1 || pl.r == 2 || pl.r == 4 || pl.r == 8);
  // (16 list entries a thread, 16-bit block ids)
  pl.pisel = allow_pisel && cfg->prefill_select == MSA_PREFILL_SELECT_INDEXER && pl.k2q && tc_indexer(c, b) &&
             cfg->topk <= 16 && b->max_blocks_per_seq <= 65536;
  pl.off_pooled = o;
  if (!pl.pisel) o = align256(o + (size_t)b->num_seqs * b->q_per_seq * G * b->max_blocks_per_seq * 4);
  pl.off_uids = o; o = align256(o + (size_t)S * G * pl.cap * 4);
  pl.off_umask = o; o = align256(o + (size_t)S * G * pl.cap * 4);
  pl.off_ucount = o; o = align256(o + (size_t)S * G * 4);
  pl.off_ctr = o; o = align256(o + (size_t)pl.nctr * 4);
  pl.off_qfa = o; o = align256(o + (size_t)S * G * pl.ga.words_per_unit() * 4);
  pl.off_cfa = o; o = align256(o + (size_t)S * G * pl.ga.nt * 8 * 4);
  pl.off_po = o; o = align256(o + (size_t)S * G * pl.splits * pl.ga.cols * 128 * 4);
  pl.off_pml = o; o = align256(o + (size_t)S * G * pl.splits * pl.ga.cols * 2 * 4);
  if (pl.pisel) {
    // a list slot per (CTA, query tile it touches): at most tiles + min(CTAs,
    // units) slots of 128 rows x 4 lists x 16 keys
    const size_t tiles = (size_t)b->num_seqs * ((b->q_per_seq + 128 / G - 1) / (128 / G));
    const size_t units = tiles * (size_t)((b->max_blocks_per_seq + 1) / 2);
    const size_t ctas = (size_t)prefill_indexer_grid(sm_count());
    pl.off_plists = o; o = align256(o + (tiles + (units < ctas ? units : ctas)) * 128 * 64 * 8);
  }
  if (pl.k2q) {
    const size_t L = (size_t)b->num_seqs * G * b->max_blocks_per_seq;
    const size_t E = (size_t)b->num_seqs * b->q_per_seq * G * cfg->topk;
    const size_t P = E * pl.r;
    if (P >= ((size_t)1 << 31)) return MSA_ERR_UNSUPPORTED;  // the list kernels count entries and partials in 32 bits
    pl.off_kcnt = o; o = align256(o + L * 4);
    pl.off_koff = o; o = align256(o + L * 4);
    pl.off_kcur = o; o = align256(o + L * 4);
    pl.off_kitem = o; o = align256(o + (L + 1) * 4);
    pl.off_kent = o; o = align256(o + E * 4 + 16);  // the attend copies entries from 16-byte boundaries
    pl.off_klist = o; o = align256(o + E * 4);
    pl.off_kpo = o; o = align256(o + P * 128 * 2);
    pl.off_kpml = o; o = align256(o + P * 4 * 4);
    const size_t R = (size_t)b->num_seqs * b->q_per_seq * hq;  // query rows (token, head)
    pl.off_kq = o; o = align256(o + (q_fp8 ? 0 : R * 256));
    pl.off_kqf = o; o = align256(o + (q_fp8 ? 0 : R * 4));
  }
  pl.total = o;
  return MSA_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

BatchDev batch_dev(const msa_batch_t* b, const Plan& pl) {
  BatchDev d;
  d.seq_lens = b->seq_lens;
  d.block_table = b->block_table;
  d.S = pl.S;
  d.Q = pl.Q;
  d.max_nb = b->max_blocks_per_seq;
  d.chunks = pl.chunks;
  d.q_real = b->q_per_seq;
  return d;
}

// the attend's view of the batch (its own virtual sequences)
BatchDev batch_dev_att(const msa_batch_t* b, const Plan& pl) {
  BatchDev d = batch_dev(b, pl);
  d.S = pl.Sa;
  d.Q = pl.Qa;
  d.chunks = pl.chunks_a;
  return d;
}

msa_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA; }

// ---------------------------------------------------------------- stages of the path

msa_status_t run_indexer(const msa_cache_t* c, const msa_batch_t* b, const msa_config_t* cfg, const msa_query_t* iq,
                         const Plan& pl, void* ws, float* pooled, cudaStream_t st, bool select = false) {
  const int G = c->num_kv_heads;
  const int fi = fmt_of(c->index_dtype);
  CUtensorMap tm;
  const CUtensorMap* tmp = nullptr;
  if (fi != FMT_NVFP4) {
    if (!encode_rows(&tm, c->idx, (long)c->num_blocks * kBlock, fi == FMT_BF16)) return MSA_ERR_CUDA;
    tmp = &tm;
  }
  if (tc_indexer(c, b)) {
    // a prefill chunk: the queries fill the tensor cores' M side (tcgen05)
    PrefillIndexerParams pp;
    Plan real;
    real.S = b->num_seqs;
    real.Q = b->q_per_seq;
    real.chunks = 1;
    pp.batch = batch_dev(b, real);
    pp.G = G;
    pp.num_blocks = c->num_blocks;
    pp.idx_scale = c->idx_scale;
    pp.index_q = iq->data;
    pp.iq_fp8 = iq->dtype == MSA_DTYPE_FP8_E4M3;
    pp.iq_scale = pp.iq_fp8 ? iq->scale : 1.f;
    pp.col_const = cfg->index_scale;
    pp.pooled = pooled;
    pp.lists = select ? at<uint64_t>(ws, pl.off_plists) : nullptr;
    pp.topk = cfg->topk;
    pp.init_blocks = cfg->init_blocks;
    pp.local_blocks = cfg->local_blocks;
    pp.status = at<DeviceStatus>(ws, pl.off_status);
    return cuda_status(launch_prefill_indexer(tmp, pp, sm_count(), st));
  }
  IndexerParams ip;
  ip.batch = batch_dev(b, pl);
  ip.G = G;
  ip.num_blocks = c->num_blocks;
  ip.idx = static_cast<const uint8_t*>(c->idx);
  ip.idx_sf = static_cast<const uint8_t*>(c->idx_sf);
  ip.idx_scale = c->idx_scale;
  ip.index_q = iq->data;
  ip.iq_fp8 = iq->dtype == MSA_DTYPE_FP8_E4M3;
  ip.iq_scale = ip.iq_fp8 ? iq->scale : 1.f;
  ip.col_const = cfg->index_scale * (fi == FMT_NVFP4 ? c->idx_global : 1.f);
  ip.nv_round = c->nvfp4_mode == MSA_NVFP4_E4M3_PRODUCT ? 1 : 0;
  ip.geom = pl.gi;
  ip.pooled = pooled;
  ip.status = at<DeviceStatus>(ws, pl.off_status);
  // first kernel of the call: plain stream order, so every earlier write to the
  // caches and queries is complete and visible before it reads them
  return cuda_status(launch_indexer(fi, tmp, ip, sm_count(), st, false));
}

// fill the attend query-fragment job of a top-k / union launch
template <typename P>
void set_frag_job(P& kp, const msa_cache_t* c, const msa_config_t* cfg, const msa_query_t* q, int hq, const Plan& pl,
                  void* ws) {
  const int fa = fmt_of(c->kv_dtype);
  kp.q = q->data;
  kp.q_fp8 = q->dtype == MSA_DTYPE_FP8_E4M3;
  kp.q_scale = kp.q_fp8 ? q->scale : 1.f;
  kp.col_const = cfg->sm_scale * 1.4426950408889634f * (fa == FMT_NVFP4 ? c->k_global : 1.f);
  kp.key_fmt = fa;
  kp.r = pl.r;
  kp.hq = hq;
  kp.geom = pl.ga;
  kp.frag = at<uint32_t>(ws, pl.off_qfa);
  kp.colf = at<float>(ws, pl.off_cfa);
}

struct FragJob {
  const msa_cache_t* c;
  const msa_query_t* q;
  int hq;
};

msa_status_t run_topk(const msa_batch_t* b, const msa_config_t* cfg, int G, const float* pooled, int32_t* topk_idx,
                      float* topk_score, void* ws, const Plan* pl, cudaStream_t st, bool pdl, bool clear_ctr,
                      const FragJob* frag_job = nullptr, bool warp_rows = false) {
  TopkParams tp;
  // positions T - Q + i are the same with or without virtual sequences: the real batch
  Plan real;
  real.S = b->num_seqs;
  real.Q = b->q_per_seq;
  real.chunks = 1;
  tp.batch = batch_dev(b, real);
  tp.G = G;
  tp.topk = cfg->topk;
  tp.init_blocks = cfg->init_blocks;
  tp.local_blocks = cfg->local_blocks;
  tp.pooled = pooled;
  tp.topk_idx = topk_idx;
  tp.topk_score = topk_score;
  tp.status = pl ? at<DeviceStatus>(ws, pl->off_status) : static_cast<DeviceStatus*>(ws);
  tp.zero = (clear_ctr && pl) ? at<int32_t>(ws, pl->off_ctr) : nullptr;  // for the attend that follows
  tp.nzero = (clear_ctr && pl) ? pl->nctr : 0;
  tp.frag = nullptr;
  tp.colf = nullptr;
  if (frag_job && pl) set_frag_job(tp, frag_job->c, cfg, frag_job->q, frag_job->hq, *pl, ws);
  // one warp per row: for many short rows with nothing else to do (no scores,
  // fragments or counters)
  if (warp_rows && !topk_score && !tp.frag && !tp.zero) return cuda_status(launch_topk_warp(tp, st, pdl));
  return cuda_status(launch_topk(tp, st, pdl));
}

// The prefill selection from the candidate lists the tcgen05 indexer left (Plan::pisel).
msa_status_t run_pisel(const msa_batch_t* b, const msa_config_t* cfg, int G, int32_t* topk_idx, const Plan& pl,
                       void* ws, cudaStream_t st) {
  Plan real;
  real.S = b->num_seqs;
  real.Q = b->q_per_seq;
  real.chunks = 1;
  PiSelectParams sp;
  sp.batch = batch_dev(b, real);
  sp.G = G;
  sp.topk = cfg->topk;
  sp.init_blocks = cfg->init_blocks;
  sp.local_blocks = cfg->local_blocks;
  sp.grid = prefill_indexer_grid(sm_count());
  sp.lists = at<uint64_t>(ws, pl.off_plists);
  sp.topk_idx = topk_idx;
  sp.status = at<DeviceStatus>(ws, pl.off_status);
  return cuda_status(launch_prefill_select(sp, st));
}

msa_status_t run_attend(const msa_cache_t* c, const msa_batch_t* b, const msa_config_t* cfg, const msa_query_t* q,
                        int hq, const int32_t* topk_idx, void* out, float* lse, const Plan& pl, void* ws,
                        cudaStream_t st, bool prepared) {
  // prepared: the preceding top-k launch (one query token) already cleared the
  // counters and wrote the query fragments; otherwise the union kernel does both
  const int G = c->num_kv_heads;
  const int fa = fmt_of(c->kv_dtype);
  DeviceStatus* status = at<DeviceStatus>(ws, pl.off_status);
  const bool direct = prepared && pl.direct;
  UnionParams up;
  up.batch = batch_dev_att(b, pl);
  up.G = G;
  up.topk = cfg->topk;
  up.topk_idx = topk_idx;
  up.cap = pl.cap;
  up.u_ids = at<int32_t>(ws, pl.off_uids);
  up.u_mask = at<uint32_t>(ws, pl.off_umask);
  up.u_count = at<int32_t>(ws, pl.off_ucount);
  up.zero = at<int32_t>(ws, pl.off_ctr);  // for the attend that follows
  up.nzero = pl.nctr;
  set_frag_job(up, c, cfg, q, hq, pl, ws);
  up.status = status;
  if (!direct) {
    if (launch_union(up, st, true) != cudaSuccess) return MSA_ERR_CUDA;
  }

  CUtensorMap tk, tv;
  const CUtensorMap *tkp = nullptr, *tvp = nullptr;
  if (fa != FMT_NVFP4) {
    const long rows = (long)c->num_blocks * G * kBlock;
    if (!encode_rows(&tk, c->k, rows, fa == FMT_BF16) || !encode_rows(&tv, c->v, rows, fa == FMT_BF16))
      return MSA_ERR_CUDA;
    tkp = &tk;
    tvp = &tv;
  }
  AttendParams ap;
  ap.batch = batch_dev_att(b, pl);
  ap.G = G;
  ap.r = pl.r;
  ap.num_blocks = c->num_blocks;
  ap.k = static_cast<const uint8_t*>(c->k);
  ap.v = static_cast<const uint8_t*>(c->v);
  ap.k_sf = static_cast<const uint8_t*>(c->k_sf);
  ap.v_sf = static_cast<const uint8_t*>(c->v_sf);
  ap.k_scale = c->k_scale;
  ap.v_scale = c->v_scale;
  ap.v_global = c->v_global;
  ap.nv_round = c->nvfp4_mode == MSA_NVFP4_E4M3_PRODUCT ? 1 : 0;
  ap.q = q->data;
  ap.q_fp8 = q->dtype == MSA_DTYPE_FP8_E4M3;
  ap.q_scale = ap.q_fp8 ? q->scale : 1.f;
  ap.col_const = cfg->sm_scale * 1.4426950408889634f * (fa == FMT_NVFP4 ? c->k_global : 1.f);
  ap.geom = pl.ga;
  ap.direct = direct ? 1 : 0;
  ap.frag = up.frag;
  ap.colf = up.colf;
  ap.topk_idx = topk_idx;
  ap.topk = cfg->topk;
  ap.u_ids = up.u_ids;
  ap.u_mask = up.u_mask;
  ap.u_count = up.u_count;
  ap.cap = pl.cap;
  ap.bps = pl.bps;
  ap.splits = pl.splits;
  ap.work_ctr = nullptr;
  ap.sg_ctr = at<int32_t>(ws, pl.off_ctr);
  ap.part_o = at<float>(ws, pl.off_po);
  ap.part_ml = at<float>(ws, pl.off_pml);
  ap.out = out;
  ap.lse = lse;
  ap.status = status;
  if (launch_attend(fa, tkp, tvp, ap, sm_count(), st, true) != cudaSuccess) return MSA_ERR_CUDA;
  return MSA_OK;
}

// The key-block-major attend of a prefill chunk from the selection topk_idx.
msa_status_t run_k2q(const msa_cache_t* c, const msa_batch_t* b, const msa_config_t* cfg, const msa_query_t* q,
                     int hq, const int32_t* topk_idx, void* out, float* lse, const Plan& pl, void* ws,
                     cudaStream_t st) {
  const int G = c->num_kv_heads;
  if (!aligned16(ws)) return MSA_ERR_INVALID_ARGUMENT;  // the attend's bulk copies read from it
  CUtensorMap tk, tv;
  const long rows = (long)c->num_blocks * G * kBlock;
  if (!encode_rows(&tk, c->k, rows, false) || !encode_rows(&tv, c->v, rows, false)) return MSA_ERR_CUDA;
  Plan real;
  real.S = b->num_seqs;
  real.Q = b->q_per_seq;
  real.chunks = 1;
  K2qParams kp;
  kp.batch = batch_dev(b, real);
  kp.G = G;
  kp.r = hq / G;
  kp.topk = cfg->topk;
  kp.num_blocks = c->num_blocks;
  kp.topk_idx = topk_idx;
  kp.cnt = at<int32_t>(ws, pl.off_kcnt);
  kp.off = at<int32_t>(ws, pl.off_koff);
  kp.cur = at<int32_t>(ws, pl.off_kcur);
  kp.item_off = at<int32_t>(ws, pl.off_kitem);
  kp.entries = at<int32_t>(ws, pl.off_kent);
  kp.item_list = at<int32_t>(ws, pl.off_klist);
  kp.item_tokens = kBlock / kp.r;
  kp.k_scale = c->k_scale;
  kp.v_scale = c->v_scale;
  kp.q = q->data;
  kp.q_fp8 = q->dtype == MSA_DTYPE_FP8_E4M3;
  kp.q_scale = kp.q_fp8 ? q->scale : 1.f;
  kp.col_const = cfg->sm_scale * 1.4426950408889634f;
  kp.qsplit = at<uint8_t>(ws, pl.off_kq);
  kp.qrowf = at<float>(ws, pl.off_kqf);
  kp.part_o = at<uint16_t>(ws, pl.off_kpo);
  kp.part_ml = at<float>(ws, pl.off_kpml);
  kp.out = out;
  kp.lse = lse;
  kp.status = at<DeviceStatus>(ws, pl.off_status);
  if (launch_k2q_build(kp, sm_count(), st) != cudaSuccess) return MSA_ERR_CUDA;
  if (launch_k2q_attend(&tk, &tv, kp, sm_count(), st) != cudaSuccess) return MSA_ERR_CUDA;
  if (launch_k2q_combine(kp, sm_count(), st) != cudaSuccess) return MSA_ERR_CUDA;
  return MSA_OK;
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

const char* msa_status_string(msa_status_t s) {
  switch (s) {
    case MSA_OK: return "MSA_OK";
    case MSA_ERR_INVALID_ARGUMENT: return "MSA_ERR_INVALID_ARGUMENT";
    case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED";
    case MSA_ERR_WORKSPACE_TOO_SMALL: return "MSA_ERR_WORKSPACE_TOO_SMALL";
    case MSA_ERR_CUDA: return "MSA_ERR_CUDA";
    case MSA_ERR_DEVICE_FAULT: return "MSA_ERR_DEVICE_FAULT";
    case MSA_ERR_TIMEOUT: return "MSA_ERR_TIMEOUT";
    default: return "MSA_ERR_UNKNOWN";
  }
}

size_t msa_workspace_size(const msa_cache_t* cache, const msa_batch_t* batch, const msa_config_t* cfg,
                          int32_t num_q_heads) {
  if (check_batch(batch) != MSA_OK || check_cfg(cfg) != MSA_OK || check_cache(cache, false, false) != MSA_OK)
    return 0;
  // the largest plan over query dtypes (a bf16 query against FP8 keys needs two terms)
  Plan pl;
  if (make_plan(cache, batch, cfg, num_q_heads, false, false, pl) != MSA_OK) {
    if (make_plan(cache, batch, cfg, num_q_heads, true, true, pl) != MSA_OK) return 0;
  }
  return pl.total;
}

msa_status_t msa_workspace_init(void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  if (!workspace || workspace_bytes < 256) return MSA_ERR_INVALID_ARGUMENT;
  return cuda_status(cudaMemsetAsync(workspace, 0, 256, (cudaStream_t)stream));
}

msa_status_t msa_indexer_score(const msa_cache_t* cache, const msa_batch_t* batch, const msa_config_t* cfg,
                               const msa_query_t* index_q, float* pooled, void* workspace, size_t workspace_bytes,
                               msa_stream_t stream) {
  msa_status_t s;
  if ((s = check_batch(batch)) != MSA_OK || (s = check_cfg(cfg)) != MSA_OK || (s = check_cache(cache, true, false)) != MSA_OK ||
      (s = check_query(index_q)) != MSA_OK)
    return s;
  if (!pooled || !workspace) return MSA_ERR_INVALID_ARGUMENT;
  Plan pl;
  if ((s = make_plan(cache, batch, cfg, cache->num_kv_heads, index_q->dtype == MSA_DTYPE_FP8_E4M3, false, pl)) != MSA_OK)
    return s;
  if (workspace_bytes < pl.off_pooled) return MSA_ERR_WORKSPACE_TOO_SMALL;
  return run_indexer(cache, batch, cfg, index_q, pl, workspace, pooled, (cudaStream_t)stream);
}

msa_status_t msa_topk_blocks(const msa_batch_t* batch, const msa_config_t* cfg, int32_t num_groups,
                             const float* pooled, int32_t* topk_idx, float* topk_score, void* workspace,
                             size_t workspace_bytes, msa_stream_t stream) {
  msa_status_t s;
  if ((s = check_batch(batch)) != MSA_OK || (s = check_cfg(cfg)) != MSA_OK) return s;
  if (num_groups < 1 || num_groups > 8 || !pooled || !topk_idx || !workspace) return MSA_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < 256) return MSA_ERR_WORKSPACE_TOO_SMALL;
  return run_topk(batch, cfg, num_groups, pooled, topk_idx, topk_score, workspace, nullptr, (cudaStream_t)stream, false,
                  false);
}

msa_status_t msa_sparse_attend(const msa_cache_t* cache, const msa_batch_t* batch, const msa_config_t* cfg,
                               const msa_query_t* q, int32_t num_q_heads, const int32_t* topk_idx, void* out,
                               float* lse, void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  msa_status_t s;
  if ((s = check_batch(batch)) != MSA_OK || (s = check_cfg(cfg)) != MSA_OK || (s = check_cache(cache, false, true)) != MSA_OK ||
      (s = check_query(q)) != MSA_OK)
    return s;
  if (!topk_idx || !out || !workspace || !aligned16(out)) return MSA_ERR_INVALID_ARGUMENT;
  Plan pl;
  if ((s = make_plan(cache, batch, cfg, num_q_heads, true, q->dtype == MSA_DTYPE_FP8_E4M3, pl)) != MSA_OK) return s;
  if (workspace_bytes < pl.total) return MSA_ERR_WORKSPACE_TOO_SMALL;
  if (pl.k2q) return run_k2q(cache, batch, cfg, q, num_q_heads, topk_idx, out, lse, pl, workspace, (cudaStream_t)stream);
  return run_attend(cache, batch, cfg, q, num_q_heads, topk_idx, out, lse, pl, workspace, (cudaStream_t)stream, false);
}

msa_status_t msa_decode(const msa_cache_t* cache, const msa_batch_t* batch, const msa_config_t* cfg,
                        const msa_query_t* index_q, const msa_query_t* q, int32_t num_q_heads, int32_t* topk_idx,
                        void* out, float* lse, void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  msa_status_t s;
  if ((s = check_batch(batch)) != MSA_OK || (s = check_cfg(cfg)) != MSA_OK || (s = check_cache(cache, true, true)) != MSA_OK ||
      (s = check_query(index_q)) != MSA_OK || (s = check_query(q)) != MSA_OK)
    return s;
  if (!topk_idx || !out || !workspace || !aligned16(out)) return MSA_ERR_INVALID_ARGUMENT;
  Plan pl;
  if ((s = make_plan(cache, batch, cfg, num_q_heads, index_q->dtype == MSA_DTYPE_FP8_E4M3,
                     q->dtype == MSA_DTYPE_FP8_E4M3, pl)) != MSA_OK)
    return s;
  if (workspace_bytes < pl.total) return MSA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = (cudaStream_t)stream;
  float* pooled = at<float>(workspace, pl.off_pooled);
  if ((s = run_indexer(cache, batch, cfg, index_q, pl, workspace, pooled, st, pl.pisel)) != MSA_OK) return s;
  if (pl.k2q) {
    if ((s = pl.pisel ? run_pisel(batch, cfg, cache->num_kv_heads, topk_idx, pl, workspace, st)
                      : run_topk(batch, cfg, cache->num_kv_heads, pooled, topk_idx, nullptr, workspace, &pl, st, true,
                                 false, nullptr, true)) != MSA_OK)
      return s;
    return run_k2q(cache, batch, cfg, q, num_q_heads, topk_idx, out, lse, pl, workspace, st);
  }
  const FragJob fj = {cache, q, num_q_heads};
  if ((s = run_topk(batch, cfg, cache->num_kv_heads, pooled, topk_idx, nullptr, workspace, &pl, st, true, true,
                    pl.direct ? &fj : nullptr)) != MSA_OK)
    return s;
  return run_attend(cache, batch, cfg, q, num_q_heads, topk_idx, out, lse, pl, workspace, st, true);
}

msa_status_t msa_cache_insert(const msa_cache_t* cache, int32_t num_tokens, const int32_t* slot_mapping,
                              const void* k, const void* v, const void* index_k, void* workspace,
                              size_t workspace_bytes, msa_stream_t stream) {
  msa_status_t s;
  if ((s = check_cache(cache, index_k != nullptr, true)) != MSA_OK) return s;
  if (num_tokens < 0 || !workspace) return MSA_ERR_INVALID_ARGUMENT;
  if (cache->num_kv_heads > 8) return MSA_ERR_UNSUPPORTED;
  if (workspace_bytes < 256) return MSA_ERR_WORKSPACE_TOO_SMALL;
  if (num_tokens == 0) return MSA_OK;
  if (!slot_mapping || !k || !v || !aligned16(k) || !aligned16(v) || (index_k && !aligned16(index_k)))
    return MSA_ERR_INVALID_ARGUMENT;
  InsertParams p;
  std::memset(&p, 0, sizeof(p));
  p.num_tokens = num_tokens;
  p.H = cache->num_kv_heads;
  p.num_blocks = cache->num_blocks;
  p.kv_fmt = fmt_of(cache->kv_dtype);
  p.idx_fmt = index_k ? fmt_of(cache->index_dtype) : FMT_BF16;
  p.slots = slot_mapping;
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.ik = static_cast<const __nv_bfloat16*>(index_k);
  // the insert writes through the cache's pointers
  p.kc = static_cast<uint8_t*>(const_cast<void*>(cache->k));
  p.vc = static_cast<uint8_t*>(const_cast<void*>(cache->v));
  p.ic = static_cast<uint8_t*>(const_cast<void*>(cache->idx));
  p.ks = const_cast<float*>(cache->k_scale);
  p.vs = const_cast<float*>(cache->v_scale);
  p.is = const_cast<float*>(cache->idx_scale);
  p.ksf = static_cast<uint8_t*>(const_cast<void*>(cache->k_sf));
  p.vsf = static_cast<uint8_t*>(const_cast<void*>(cache->v_sf));
  p.isf = static_cast<uint8_t*>(const_cast<void*>(cache->idx_sf));
  p.kg = cache->k_global;
  p.vg = cache->v_global;
  p.ig = cache->idx_global;
  p.status = static_cast<DeviceStatus*>(workspace);
  return cuda_status(launch_insert(p, sm_count(), (cudaStream_t)stream));
}

msa_status_t msa_read_device_status(void* workspace, msa_stream_t stream, int32_t* detail) {
  if (!workspace) return MSA_ERR_INVALID_ARGUMENT;
  DeviceStatus h = {0, 0};
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MSA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MSA_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(h), st) != cudaSuccess) return MSA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MSA_ERR_CUDA;
  if (detail) *detail = (int32_t)h.flags;
  if (h.flags & FLAG_TIMEOUT) return MSA_ERR_TIMEOUT;
  if (h.flags) return MSA_ERR_DEVICE_FAULT;
  return MSA_OK;
}

msa_status_t msa_dequant_debug(const msa_cache_t* cache, int32_t which, const int32_t* phys_blocks, int32_t n,
                               float* out, msa_stream_t stream) {
  if (which < 0 || which > 2 || n < 0 || (n > 0 && (!phys_blocks || !out))) return MSA_ERR_INVALID_ARGUMENT;
  msa_status_t s = check_cache(cache, which == 2, which != 2);
  if (s != MSA_OK) return s;
  const int f = fmt_of(which == 2 ? cache->index_dtype : cache->kv_dtype);
  return cuda_status(launch_dequant(f, which, *cache, phys_blocks, n, out, (cudaStream_t)stream));
}

}  // extern "C"

// ====================================================================== allocation-free decode
//
// Some callers cannot allocate device memory for a workspace: code that runs
// inside another framework's memory pool or allocator hooks, a plugin that
// must not call cudaMalloc (or torch's allocator) on its hot path, or a
// process whose device memory is fully reserved up front.  msa_decode_noalloc
// serves them with a fixed scratch area that lives in the library itself: the
// array below is part of the library's device image, so every GPU that loads
// libmsa holds these bytes until the process exits.

// MSA_NOALLOC_SCRATCH_BYTES (include/msa.h): the largest workspace it accepts.
static __device__ __align__(256) unsigned char msa_noalloc_scratch[MSA_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of msa_noalloc_scratch on the current device, looked up once
// per device (the host-side symbol is only a stand-in, never a device address).
// The cached address assumes the device's context lives as long as the
// process: a device reset (cudaDeviceReset) is not supported afterwards.
msa_status_t noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64];
  static bool have[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, msa_noalloc_scratch) != cudaSuccess || p == nullptr) return MSA_ERR_CUDA;
    addr[dev] = p;
    have[dev] = true;
  }
  *out = addr[dev];
  return MSA_OK;
}

}  // namespace

extern "C" msa_status_t msa_decode_noalloc(const msa_cache_t* cache, const msa_batch_t* batch,
                                           const msa_config_t* cfg, const msa_query_t* index_q,
                                           const msa_query_t* q, int32_t num_q_heads, int32_t* topk_idx,
                                           void* out, float* lse, int32_t* status_out, msa_stream_t stream) {
  msa_status_t s;
  if ((s = check_batch(batch)) != MSA_OK || (s = check_cfg(cfg)) != MSA_OK || (s = check_cache(cache, true, true)) != MSA_OK ||
      (s = check_query(index_q)) != MSA_OK || (s = check_query(q)) != MSA_OK)
    return s;
  if (!topk_idx || !out || !aligned16(out)) return MSA_ERR_INVALID_ARGUMENT;
  Plan pl;
  if ((s = make_plan(cache, batch, cfg, num_q_heads, index_q->dtype == MSA_DTYPE_FP8_E4M3,
                     q->dtype == MSA_DTYPE_FP8_E4M3, pl)) != MSA_OK)
    return s;
  if (pl.total > MSA_NOALLOC_SCRATCH_BYTES && pl.pisel &&
      (s = make_plan(cache, batch, cfg, num_q_heads, index_q->dtype == MSA_DTYPE_FP8_E4M3,
                     q->dtype == MSA_DTYPE_FP8_E4M3, pl, false)) != MSA_OK)  // pooled scores may still fit
    return s;
  if (pl.total > MSA_NOALLOC_SCRATCH_BYTES) return MSA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  if ((s = noalloc_scratch(&ws)) != MSA_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  // the status word must start at zero; every other region is written before it is read
  if (cudaMemsetAsync(ws, 0, 256, st) != cudaSuccess) return MSA_ERR_CUDA;
  float* pooled = at<float>(ws, pl.off_pooled);
  if ((s = run_indexer(cache, batch, cfg, index_q, pl, ws, pooled, st, pl.pisel)) != MSA_OK) return s;
  if (pl.k2q) {
    // a prefill chunk over an FP8 cache: the same chain as msa_decode's
    if ((s = pl.pisel ? run_pisel(batch, cfg, cache->num_kv_heads, topk_idx, pl, ws, st)
                      : run_topk(batch, cfg, cache->num_kv_heads, pooled, topk_idx, nullptr, ws, &pl, st, true, false,
                                 nullptr, true)) != MSA_OK)
      return s;
    if ((s = run_k2q(cache, batch, cfg, q, num_q_heads, topk_idx, out, lse, pl, ws, st)) != MSA_OK) return s;
  } else {
    const FragJob fj = {cache, q, num_q_heads};
    if ((s = run_topk(batch, cfg, cache->num_kv_heads, pooled, topk_idx, nullptr, ws, &pl, st, true, true,
                      pl.direct ? &fj : nullptr)) != MSA_OK)
      return s;
    if ((s = run_attend(cache, batch, cfg, q, num_q_heads, topk_idx, out, lse, pl, ws, st, true)) != MSA_OK)
      return s;
  }
  if (status_out &&
      cudaMemcpyAsync(status_out, ws, 2 * sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return MSA_ERR_CUDA;
  return MSA_OK;
}
