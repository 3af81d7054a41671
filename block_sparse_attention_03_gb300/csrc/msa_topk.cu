// Top-k block selection and the per-(sequence, group) union of selections.
//
// Selection (vLLM Day-0 blog, section "MSA 入门"): per (query, group) keep
// the top-k blocks by pooled indexer score, the most recent block always
// kept.  Readings the pages leave open: the query's own block counts as one of
// the k; the indexer constructor's init_blocks / local_blocks (model page,
// MiniMaxM3SparseAttention.__init__) force the first blocks and the blocks
// just before the query's block; equal scores keep the smaller block id; the
// output is ascending and padded with -1.
//
// Kernel: one CTA per (query row, group).  The free candidates form one
// contiguous id range [lo, hi) (everything between the forced init and local
// blocks), split into one contiguous id range per thread, keys in registers.
// Main path (threshold + rank test): the candidates are cut into 32 groups of
// consecutive threads; the kfree-th largest group maximum T is a lower bound
// with at least kfree candidates >= T, so the wanted kfree (by score, then id)
// are all among the candidates >= T -- typically a few dozen.  Those are
// compacted in id order into shared memory and each is kept iff fewer than
// kfree of them beat it.  Rows where that set is large (heavy ties) take a
// radix select over order-preserving 32-bit keys (4 passes of 8 bits,
// shared-memory histograms) with ties at the threshold resolved by id through
// a block-wide prefix count.  Either way the ids come out ascending without a
// sort because each thread owns a contiguous id range.
#include "msa_device.cuh"
#include "msa_internal.h"
#include "msa_qfrag.cuh"

namespace msa {

namespace {

constexpr int kTopkThreads = 256;
constexpr int kKeysPerThreadNarrow = 16;  // keys each thread holds in registers (256 threads)
constexpr int kKeysPerThreadWide = 8;     // (1024 threads)
constexpr int kCandMax = 1024;            // candidates >= T the rank test takes; more go to the radix select

// Histogram increment aggregated over the lanes of a warp that hit the same
// bin (the order keys of close scores share their top bits, so plain atomics
// would serialise on one bin).  Every lane of the warp must call it.
__device__ __forceinline__ void hist_add(int* hist, uint32_t bin, bool active) {
  const uint32_t act = __ballot_sync(0xffffffffu, active);
  if (!active) return;
  const uint32_t peers = __match_any_sync(act, bin);
  if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
}

constexpr int kMaxFragCols = 32;

// block-wide exclusive scan of one int per thread; returns the total
template <int THREADS>
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int& excl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  int wbase = 0, total = 0;
  for (int w = 0; w < THREADS / 32; ++w) {
    const int t = warp_tot[w];
    if (w < warp) wbase += t;
    total += t;
  }
  excl = wbase + x - v;
  __syncthreads();
  return total;
}

template <int THREADS>
__global__ void __launch_bounds__(THREADS) topk_kernel(const TopkParams p) {
  constexpr int kKeysPerThread = THREADS >= 1024 ? kKeysPerThreadWide : kKeysPerThreadNarrow;
  static_assert(THREADS % 32 == 0 && THREADS >= 32 && THREADS <= 1024, "thread count");
  __shared__ int hist[256];
  __shared__ int warp_tot[THREADS / 32];
  __shared__ uint32_t sh_prefix, sh_need;
  __shared__ uint32_t gmax[32];
  __shared__ uint32_t ck[kCandMax];
  __shared__ uint8_t csel[kCandMax];

  // the attend that follows may start its prologue now; it waits for this grid to finish
  pdl_launch_dependents();
  const BatchDev bt = p.batch;
  const int row = blockIdx.x;  // (s*Q + i) * G + g
  const bool real_row = row < bt.S * bt.Q * p.G;
  if (real_row && p.frag) {
    // one query token: this CTA's row is attend unit (s, g); build its query
    // fragments.  They come from the caller's q alone, so this overlaps the
    // indexer still running ahead of this kernel.
    __shared__ float qs[kMaxFragCols * (kDim + 1)];
    __shared__ float pscale[kMaxFragCols];
    const int s_ = row / p.G, g_ = row % p.G, r = p.r, hq = p.hq, cols = p.geom.cols;
    auto row_of = [&](int col) -> long { return col < cols ? ((long)s_ * hq + g_ * r + col) * kDim : -1l; };
    write_qfrag(p.q, p.q_fp8, row_of, p.q_scale, p.col_const, p.key_fmt, p.geom, qs, pscale,
                p.frag + (size_t)row * p.geom.words_per_unit(), p.colf + (size_t)row * p.geom.nt * 8);
  }
  // the row's facts come from the caller's sequence lengths: read before the wait
  const int sq = row / p.G;
  const int s = sq / bt.Q, i = sq % bt.Q;
  const int T = real_row ? bt.seq_len(s) : 0;
  pdl_wait();
  if (p.zero) {  // clear the attend's work counters for this call
    const int z = blockIdx.x * blockDim.x + threadIdx.x;
    if (z < p.nzero) p.zero[z] = 0;
  }
  if (!real_row) return;  // extra CTAs only clear counters
  const int K = p.topk;
  int32_t* out = p.topk_idx + (size_t)row * K;
  float* out_sc = p.topk_score ? p.topk_score + (size_t)row * K : nullptr;
  const float* pr = p.pooled + (size_t)row * bt.max_nb;

  if (T < bt.Q || T > bt.max_nb * kBlock) {
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
      out[k] = -1;
      if (out_sc) out_sc[k] = -INFINITY;
    }
    if (threadIdx.x == 0 && i == 0 && row % p.G == 0) raise_flag(p.status, FLAG_BAD_SEQLEN, s);
    pdl_launch_dependents();
    return;
  }
  const int pos = T - bt.Q + i;
  const int recent = pos / kBlock;
  const int n_init = min(p.init_blocks, recent);           // forced [0, n_init)
  const int n_local = min(p.local_blocks, recent - n_init); // forced [recent - n_local, recent)
  const int lo = n_init, hi = recent - n_local;            // free candidates [lo, hi)
  const int ncand = hi - lo;
  const int kfree = K - n_init - n_local - 1;

  // thread-owned contiguous candidate range
  const int per = (ncand + THREADS - 1) / THREADS;
  const int b0 = lo + threadIdx.x * per;
  const int b1 = min(hi, b0 + per);

  // this thread's candidate keys stay in registers across the passes (rows of
  // up to THREADS * kKeysPerThread candidates; longer rows re-read them)
  const int cnt = max(0, b1 - b0);
  const bool inreg = per <= kKeysPerThread;
  uint32_t keys[kKeysPerThread];
  // a full range on a 16-byte boundary (long rows) loads 16 bytes at a time: a
  // quarter of the L1 requests of the strided 4-byte loads (256 threads)
  const bool vec = THREADS < 1024 && inreg && cnt == kKeysPerThread &&
                   (reinterpret_cast<uintptr_t>(pr + b0) & 15u) == 0;
#pragma unroll
  for (int i = 0; i < kKeysPerThread; i += 4) {
    float f[4];
    bool ok[4];
    if (vec) {
      const float4 v = *reinterpret_cast<const float4*>(pr + b0 + i);
      f[0] = v.x;
      f[1] = v.y;
      f[2] = v.z;
      f[3] = v.w;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      ok[q] = inreg && i + q < cnt;
      if (!vec) f[q] = ok[q] ? pr[b0 + i + q] : 0.f;
      keys[i + q] = ok[q] ? float_order_key(f[q]) : 0u;
    }
  }
  auto key_at = [&](int i) -> uint32_t { return float_order_key(pr[b0 + i]); };

  uint32_t thr = 0;     // keys > thr are taken; keys == thr: the first `need_eq` by id
  int need_eq = 0;
  const bool take_all = ncand <= kfree;
  const bool take_none = !take_all && kfree <= 0;

  // ---------------- threshold + rank test
  if (!take_all && !take_none && inreg && kfree <= 32) {
    constexpr int L = THREADS / 32;  // threads per group (32 groups)
    const int lane = threadIdx.x & 31;
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < kKeysPerThread; ++i)
      if (i < cnt) m = max(m, keys[i]);
#pragma unroll
    for (int o = 1; o < L; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane % L == 0) gmax[threadIdx.x / L] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
      // rank of this group's maximum among the 32 (ties by group index)
      const uint32_t mine = gmax[lane];
      int rank = 0;
#pragma unroll 8
      for (int x = 0; x < 32; ++x) {
        const uint32_t o = gmax[x];
        rank += (o > mine) || (o == mine && x < lane);
      }
      if (rank == kfree - 1) sh_prefix = mine;
    }
    __syncthreads();
    const uint32_t tq = sh_prefix;
    int mine_c = 0;
#pragma unroll
    for (int i = 0; i < kKeysPerThread; ++i) mine_c += (i < cnt && keys[i] >= tq);
    int cbase = 0;
    const int C = block_exclusive_scan<THREADS>(mine_c, warp_tot, cbase);
    if (C <= kCandMax) {  // block-uniform
      uint32_t own_sel = 0;  // bit i: key i of this thread is a candidate
      {
        int c = cbase;
#pragma unroll
        for (int i = 0; i < kKeysPerThread; ++i)
          if (i < cnt && keys[i] >= tq) {
            ck[c++] = keys[i];
            own_sel |= 1u << i;
          }
      }
      __syncthreads();
      // candidate e is kept iff fewer than kfree candidates beat it (a higher
      // key, or the same key and a smaller id = a smaller index here)
      for (int e = threadIdx.x; e < C; e += THREADS) {
        const uint32_t ke = ck[e];
        int beat = 0;
        for (int x = 0; x < C; ++x) {
          const uint32_t kx = ck[x];
          beat += (kx > ke) || (kx == ke && x < e);
        }
        csel[e] = beat < kfree;
      }
      __syncthreads();
      // this thread's kept ids, in order, at n_init + (kept candidates before them)
      if (own_sel) {
        int o = n_init;
        for (int x = 0; x < cbase; ++x) o += csel[x];
        int e = cbase;
#pragma unroll
        for (int i = 0; i < kKeysPerThread; ++i)
          if (own_sel & (1u << i)) {
            if (csel[e]) {
              out[o] = b0 + i;
              if (out_sc) out_sc[o] = pr[b0 + i];
              ++o;
            }
            ++e;
          }
      }
      const int tail_r = n_init + kfree;
      for (int k = threadIdx.x; k < K; k += THREADS) {
        if (k < n_init) {
          out[k] = k;
          if (out_sc) out_sc[k] = pr[k];
        } else if (k >= tail_r) {
          const int b = hi + (k - tail_r);
          const bool real = b <= recent;
          out[k] = real ? b : -1;
          if (out_sc) out_sc[k] = real ? pr[b] : -INFINITY;
        }
      }
      pdl_launch_dependents();
      return;
    }
  }
  if (!take_all && !take_none) {
    uint32_t prefix = 0, pmask = 0;
    int remaining = kfree;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int k = threadIdx.x; k < 256; k += blockDim.x) hist[k] = 0;
      __syncthreads();
      if (inreg) {
#pragma unroll
        for (int i = 0; i < kKeysPerThread; ++i)
          hist_add(hist, (keys[i] >> shift) & 255, i < cnt && (keys[i] & pmask) == prefix);
      } else {
        for (int i = 0; i < cnt; ++i) {
          const uint32_t key = key_at(i);
          if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1);
        }
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        // lane l owns digits [8l, 8l+8); suffix sums from the top digit down
        const int lane = threadIdx.x;
        int own = 0;
        for (int k = 0; k < 8; ++k) own += hist[8 * lane + k];
        int suf = own;  // inclusive suffix over lanes >= lane
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_down_sync(0xffffffffu, suf, o);
          if (lane + o < 32) suf += y;
        }
        const int above = suf - own;  // count in lanes > lane
        if (above < remaining && suf >= remaining) {
          int acc = above;
          for (int k = 7; k >= 0; --k) {
            const int h = hist[8 * lane + k];
            if (acc + h >= remaining) {
              sh_prefix = prefix | ((uint32_t)(8 * lane + k) << shift);
              sh_need = (uint32_t)(remaining - acc);
              break;
            }
            acc += h;
          }
        }
      }
      __syncthreads();
      prefix = sh_prefix;
      remaining = (int)sh_need;
      pmask |= 255u << shift;
      __syncthreads();
    }
    thr = prefix;
    need_eq = remaining;
  }

  // count this thread's takes, in id order
  int n_gt = 0, n_eq = 0;
  if (!take_all && !take_none) {
    if (inreg) {
#pragma unroll
      for (int i = 0; i < kKeysPerThread; ++i)
        if (i < cnt) {
          n_gt += keys[i] > thr;
          n_eq += keys[i] == thr;
        }
    } else {
      for (int i = 0; i < cnt; ++i) {
        const uint32_t key = key_at(i);
        n_gt += key > thr;
        n_eq += key == thr;
      }
    }
  }
  int eq_before = 0;
  block_exclusive_scan<THREADS>(n_eq, warp_tot, eq_before);
  const int eq_take = (take_all || take_none) ? 0 : max(0, min(n_eq, need_eq - eq_before));
  const int my_take = take_all ? cnt : (take_none ? 0 : n_gt + eq_take);
  int base = 0;
  const int n_sel = block_exclusive_scan<THREADS>(my_take, warp_tot, base);

  // ascending output: [0, n_init) ++ selected ++ [hi, recent]
  int o = n_init + base;
  int eq_seen = 0;
  if (!take_none) {
    for (int i = 0; i < cnt; ++i) {
      const uint32_t key = inreg ? keys[0] : key_at(i);
      bool take = take_all;
      if (!take_all) {
        if (key > thr) take = true;
        else if (key == thr) take = (eq_seen++ < eq_take);
      }
      if (take) {
        out[o] = b0 + i;
        if (out_sc) out_sc[o] = pr[b0 + i];
        ++o;
      }
      if (inreg) {  // shift the register window (keeps the keys array in registers)
#pragma unroll
        for (int t = 0; t + 1 < kKeysPerThread; ++t) keys[t] = keys[t + 1];
      }
    }
  }
  const int tail0 = n_init + n_sel;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    if (k < n_init) {
      out[k] = k;
      if (out_sc) out_sc[k] = pr[k];
    } else if (k >= tail0) {
      const int b = hi + (k - tail0);
      const bool real = b <= recent;
      out[k] = real ? b : -1;
      if (out_sc) out_sc[k] = real ? pr[b] : -INFINITY;
    }
  }
  pdl_launch_dependents();
}

// The top-k blocks of one (query, group) row for the query at position pos,
// selected by one warp with the rule of the top-k kernel (vLLM Day-0 blog,
// "MSA 入门"): forced init / local / own blocks, then the highest pooled scores
// among the other visible blocks, ties to the smaller id, ascending.  Returns
// in lane k (k < the count) the k-th block id, -1 in the other lanes.
// Candidates are read interleaved (lane + 32 i: coalesced, and in id order
// when taken row by row).  Fast path: T = the kfree-th largest lane maximum
// bounds the wanted scores from below; the candidates >= T (at most 64) are
// ranked.  Otherwise an exact 4 x 8-bit radix select.
// scratch: sk[64], si[64], hist[256], out[32] in shared memory.
__device__ __noinline__ int warp_select_row(const float* __restrict__ pr, int pos, int K, int init_blocks,
                                            int local_blocks, uint32_t* sk, int* si, int* hist, int* out, int lane) {
  const unsigned FULL = 0xffffffffu;
  const unsigned lt = (1u << lane) - 1u;
  const int recent = pos / kBlock;
  const int n_init = min(init_blocks, recent);
  const int n_local = min(local_blocks, recent - n_init);
  const int lo = n_init, hi = recent - n_local;
  const int ncand = hi - lo;
  const int kfree = K - n_init - n_local - 1;
  const int per = (ncand + 31) / 32;
  int n_sel = 0;
  if (ncand <= kfree) {
    for (int c = lane; c < ncand; c += 32) out[n_init + c] = lo + c;
    n_sel = ncand;
  } else if (kfree > 0) {
    n_sel = kfree;
    // lane maxima, then the kfree-th largest of them (ties by lane)
    uint32_t m = 0;
#pragma unroll 4
    for (int i = 0; i < per; ++i) {
      const int c = lane + 32 * i;
      if (c < ncand) m = max(m, float_order_key(pr[lo + c]));
    }
    int rank = 0;
#pragma unroll 8
    for (int x = 0; x < 32; ++x) {
      const uint32_t o = __shfl_sync(FULL, m, x);
      rank += (o > m) || (o == m && x < lane);
    }
    const unsigned who = __ballot_sync(FULL, rank == kfree - 1);
    const uint32_t T = __shfl_sync(FULL, m, __ffs(who) - 1);
    // candidates >= T, compacted in id order
    int C = 0;
    for (int i = 0; i < per; ++i) {
      const int c = lane + 32 * i;
      const uint32_t key = (c < ncand) ? float_order_key(pr[lo + c]) : 0u;
      const bool in = c < ncand && key >= T;
      const unsigned bal = __ballot_sync(FULL, in);
      const int at = C + __popc(bal & lt);
      if (in && at < 64) {
        sk[at] = key;
        si[at] = lo + c;
      }
      C += __popc(bal);
    }
    __syncwarp();
    if (C <= 64) {
      // kept iff fewer than kfree of them beat it (higher key, or equal key and smaller id)
      bool sel[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = lane + 32 * h;
        sel[h] = false;
        if (e < C) {
          const uint32_t ke = sk[e];
          int beat = 0;
          for (int x = 0; x < C; ++x) {
            const uint32_t kx = sk[x];
            beat += (kx > ke) || (kx == ke && x < e);
          }
          sel[h] = beat < kfree;
        }
      }
      const unsigned b0 = __ballot_sync(FULL, sel[0]), b1 = __ballot_sync(FULL, sel[1]);
      if (sel[0]) out[n_init + __popc(b0 & lt)] = si[lane];
      if (sel[1]) out[n_init + __popc(b0) + __popc(b1 & lt)] = si[lane + 32];
    } else {
      // exact radix select of the kfree-th key (heavy ties), then one pass in id order
      uint32_t prefix = 0, pmask = 0;
      int remaining = kfree;
      for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int k = lane; k < 256; k += 32) hist[k] = 0;
        __syncwarp();
        for (int i = 0; i < per; ++i) {
          const int c = lane + 32 * i;
          if (c < ncand) {
            const uint32_t key = float_order_key(pr[lo + c]);
            if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1);
          }
        }
        __syncwarp();
        // lane l owns digits [8l, 8l+8); suffix sums from the top digit down
        int own = 0;
        for (int k = 0; k < 8; ++k) own += hist[8 * lane + k];
        int suf = own;
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_down_sync(FULL, suf, o);
          if (lane + o < 32) suf += y;
        }
        const int above = suf - own;
        int digit = -1, need = 0;
        if (above < remaining && suf >= remaining) {
          int acc = above;
          for (int k = 7; k >= 0; --k) {
            const int hk = hist[8 * lane + k];
            if (acc + hk >= remaining) {
              digit = 8 * lane + k;
              need = remaining - acc;
              break;
            }
            acc += hk;
          }
        }
        const unsigned src = __ballot_sync(FULL, digit >= 0);
        const int sl = __ffs(src) - 1;
        digit = __shfl_sync(FULL, digit, sl);
        remaining = __shfl_sync(FULL, need, sl);
        prefix |= (uint32_t)digit << shift;
        pmask |= 255u << shift;
        __syncwarp();
      }
      int base_eq = 0, base_sel = 0;
      for (int i = 0; i < per; ++i) {
        const int c = lane + 32 * i;
        const uint32_t key = (c < ncand) ? float_order_key(pr[lo + c]) : 0u;
        const bool eq = c < ncand && key == prefix;
        const unsigned beq = __ballot_sync(FULL, eq);
        const bool take = (c < ncand && key > prefix) || (eq && base_eq + __popc(beq & lt) < remaining);
        const unsigned btk = __ballot_sync(FULL, take);
        const int at = n_init + base_sel + __popc(btk & lt);
        if (take && at < K) out[at] = lo + c;
        base_eq += __popc(beq);
        base_sel += __popc(btk);
      }
    }
  }
  // forced blocks: [0, n_init) first, [hi, recent] last
  for (int k = lane; k < n_init; k += 32) out[k] = k;
  const int tail = n_init + n_sel;
  for (int k = tail + lane; k < K; k += 32) {
    const int b = hi + (k - tail);
    out[k] = (b <= recent) ? b : -1;
  }
  __syncwarp();
  const int id = (lane < K) ? out[lane] : -1;
  __syncwarp();
  return id;
}

// One warp per (token, group) row, 8 rows a CTA: for the many short rows of a
// prefill chunk, where a CTA per row spends its time in block-wide syncs.
// Same rule and output as topk_kernel (no scores, no fragment or counter job).
constexpr int kTopkWarpRows = 8;
__global__ void __launch_bounds__(32 * kTopkWarpRows) topk_warp_kernel(const TopkParams p) {
  __shared__ uint32_t sk[kTopkWarpRows][64];
  __shared__ int si[kTopkWarpRows][64];
  __shared__ int hist[kTopkWarpRows][256];
  __shared__ int outb[kTopkWarpRows][32];
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BatchDev bt = p.batch;
  const int rows = bt.S * bt.Q * p.G;  // below 2^31 (make_plan)
  const int row = blockIdx.x * kTopkWarpRows + warp;
  // the row's facts come from the caller's sequence lengths: read before the wait
  const int sq = row / p.G;
  const int s = sq / bt.Q, i = sq % bt.Q;
  const int T = row < rows ? bt.seq_len(s) : 0;
  pdl_wait();
  if (row >= rows) return;
  int id = -1;
  if (T < bt.Q || T > bt.max_nb * kBlock) {
    if (lane == 0 && i == 0 && row % p.G == 0) raise_flag(p.status, FLAG_BAD_SEQLEN, s);
  } else {
    id = warp_select_row(p.pooled + (size_t)row * bt.max_nb, T - bt.Q + i, p.topk, p.init_blocks, p.local_blocks,
                         sk[warp], si[warp], hist[warp], outb[warp], lane);
  }
  if (lane < p.topk) p.topk_idx[(size_t)row * p.topk + lane] = id;
}

// Union of the Q queries' selections of one (sequence, group), ascending, with
// a bit mask of the queries that chose each block.
__global__ void __launch_bounds__(256) union_kernel(const UnionParams p) {
  extern __shared__ int sh[];
  int* ids = sh;                                      // [cap]
  int* first = sh + p.cap;                            // [cap] 1 if first occurrence
  uint32_t* masks = reinterpret_cast<uint32_t*>(sh + 2 * p.cap);  // [cap]
  pdl_launch_dependents();  // the attend that follows may start its prologue; it waits for this grid
  pdl_wait();
  if (p.zero) {  // clear the attend's work counters for this call
    for (int z = blockIdx.x * blockDim.x + threadIdx.x; z < p.nzero; z += gridDim.x * blockDim.x) p.zero[z] = 0;
  }
  const BatchDev bt = p.batch;
  const int unit = blockIdx.x;  // s * G + g
  const int s = unit / p.G, g = unit % p.G;
  if (p.frag) {
    __shared__ float qs[kMaxFragCols * (kDim + 1)];
    __shared__ float pscale[kMaxFragCols];
    const int r = p.r, hq = p.hq, cols = p.geom.cols, Q = bt.Q;
    auto row_of = [&](int col) -> long {
      return col < cols ? ((long)(s * Q + col / r) * hq + g * r + col % r) * kDim : -1l;
    };
    write_qfrag(p.q, p.q_fp8, row_of, p.q_scale, p.col_const, p.key_fmt, p.geom, qs, pscale,
                p.frag + (size_t)unit * p.geom.words_per_unit(), p.colf + (size_t)unit * p.geom.nt * 8);
    __syncthreads();
  }
  const int T = bt.seq_len(s);
  const int n = bt.Q * p.topk;
  const bool seq_ok = !(T < bt.Q || T > bt.max_nb * kBlock);
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int i = e / p.topk, k = e % p.topk;
    int b = p.topk_idx[((size_t)(s * bt.Q + i) * p.G + g) * p.topk + k];
    if (b >= 0) {
      const int pos = T - bt.Q + i;
      if (!seq_ok || b > pos / kBlock) {
        if (seq_ok) raise_flag(p.status, FLAG_BAD_SELECT, b);
        b = -1;
      }
    }
    ids[e] = b;
    masks[e] = 0;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int b = ids[e];
    int f = b >= 0;
    for (int e2 = 0; e2 < e && f; ++e2) f = ids[e2] != b;
    first[e] = f;
    // the same block twice in one token's row: attended once, flagged
    if (b >= 0 && !f) {
      const int row0 = e - e % p.topk;
      bool twice = false;
      for (int e2 = row0; e2 < e && !twice; ++e2) twice = ids[e2] == b;
      if (twice) raise_flag(p.status, FLAG_BAD_SELECT, b);
    }
  }
  __syncthreads();
  // position of each unique block = number of unique blocks with a smaller id
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int b = ids[e];
    if (b < 0) continue;
    int rank = 0;
    for (int e2 = 0; e2 < n; ++e2) rank += first[e2] && ids[e2] >= 0 && ids[e2] < b;
    atomicOr(&masks[rank], 1u << (e / p.topk));
    if (first[e]) p.u_ids[(size_t)unit * p.cap + rank] = b;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int cnt = 0;
    for (int e = 0; e < n; ++e) cnt += first[e];
    p.u_count[unit] = cnt;
  }
  for (int e = threadIdx.x; e < n; e += blockDim.x) p.u_mask[(size_t)unit * p.cap + e] = masks[e];
  pdl_launch_dependents();
}

cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  const unsigned rows = (unsigned)(p.batch.S * p.batch.Q * p.G);
  // rows of more than 2,048 blocks: 1024 threads, 8 keys or fewer each (shorter
  // load and max chains per thread; at 4,096 blocks 1 us less than 256 threads)
  const bool wide = p.batch.max_nb > 2048;
  const unsigned threads = wide ? 1024u : (unsigned)kTopkThreads;
  const unsigned zrows = (unsigned)((p.nzero + threads - 1) / threads);
  cudaLaunchConfig_t cfg = make_cfg(dim3(rows > zrows ? rows : zrows), dim3(threads), 0, st, pdl, attr);
  if (wide) return cudaLaunchKernelEx(&cfg, topk_kernel<1024>, p);
  return cudaLaunchKernelEx(&cfg, topk_kernel<kTopkThreads>, p);
}

cudaError_t launch_topk_warp(const TopkParams& p, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  const long rows = (long)p.batch.S * p.batch.Q * p.G;
  const long grid = (rows + kTopkWarpRows - 1) / kTopkWarpRows;
  cudaLaunchConfig_t cfg = make_cfg(dim3((unsigned)(grid > 0 ? grid : 1)), dim3(32 * kTopkWarpRows), 0, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, topk_warp_kernel, p);
}

cudaError_t launch_union(const UnionParams& p, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  const size_t smem = (size_t)p.cap * 12;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = make_cfg(dim3((unsigned)(p.batch.S * p.G)), dim3(256), smem, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, union_kernel, p);
}

}  // namespace msa
