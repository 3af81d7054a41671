// Indexer score + block max-pool for prefill chunks on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// What it computes is the indexer of the decode path (vLLM Day-0 blog, section
// "MSA 入门"; section "NVIDIA Blackwell 优化的 MSA 内核" names an MSA indexer
// prefill kernel):
// for query token i of sequence s and group g,
//   P[s, i, g, b] = col_const * max over keys t of block b with t <= pos(i) of
//                   (index_q[s, i, g] . ik[t]) * kscale[t],
// -inf where block b holds no visible key.  With thousands of new tokens the
// contraction is dense, so the queries become the MMA's M side:
//   D[128 x 256] = A[128 rows = (token, group)] x B[256 keys of two blocks]^T
// with K = 128 index dims in four k32 steps of kind::f8f6f4 (e4m3 x e4m3);
// two key blocks per MMA halve the per-unit costs that do not scale with N
// (waits, commits, the accumulator hand-off to the epilogue).  A
// bf16 index query is scaled by a power of two per row (exact) and split into
// e4m3 hi + lo terms that accumulate into the same TMEM columns, carrying all 8
// significant bits of bf16; an e4m3 index query enters as is.
//
// One CTA (18 warps, persistent, one per SM) walks a contiguous run of units
// (query tile, two key blocks):
//   warp 0   copies key tiles (TMA, 128-byte swizzle) into a 5-stage ring of
//            two-tile stages (enough bytes in flight to cover L2 latency at the
//            MMA rate), freed by the MMAs' completion, and their per-token
//            scales into a 16-slot ring freed by the epilogue;
//   warp 1   owns the SM's 512 TMEM columns (two 256-column accumulators); one
//            thread issues the MMAs and commits them to mbarriers;
//   warps 2-17 four groups of four: groups 0 and 1 take the even units, 2 and
//            3 the odd ones, each pair one key block of the unit apiece (twice
//            the warps of one group per row, to hide the TMEM-load and
//            arithmetic latency); each thread owns one accumulator row
//            (tcgen05.ld 32x32b) of its block, multiplies by the key scales
//            (packed f32x2), masks the keys its token cannot see, takes the max
//            (three-input max) and writes P.  At each new query tile groups 0
//            and 2 build its operand (hi / lo e4m3 in the swizzled K-major
//            layout the MMA reads), group 0 the hi term, group 2 the lo term.
// Every mbarrier wait is bounded; a wait that gives up sets the timeout flag,
// the CTA stops issuing, drains what it issued and frees its TMEM.
//
// Selection in the epilogue (pindexer_kernel<true>, MSA_PREFILL_SELECT_INDEXER):
// instead of writing P, each epilogue thread keeps the 16 best free blocks
// (top-k rule order: score, then the smaller id) of the blocks it scores for its
// row in a shared-memory heap (worst entry at the root, so most blocks cost one
// compare), and at the end of each query tile it touched writes them as one
// list; the key ring drops to 4 stages to make room.  pi_select_kernel merges a
// row's lists (every block among the row's best is in its thread's list) and
// adds the forced blocks: the rows topk_kernel writes from P, bit for bit.
#include "msa_device.cuh"
#include "msa_internal.h"
#include "msa_tcgen05.cuh"

namespace msa {

namespace {

constexpr int kPiStages = 5;                   // units (two key tiles) in flight: L2 latency x the MMA rate
constexpr int kPiStagesSel = 4;                // with the selection lists in shared memory
constexpr int kPiSStages = 16;                 // key-scale slots (released by the epilogue, which lags)
constexpr int kPiAcc = 2;                      // accumulators of 256 columns (two key blocks)
constexpr int kPiCols = 256 * kPiAcc;          // TMEM columns (all 512 of the SM: one CTA per SM)
constexpr int kPiThreads = 576;                // producer, MMA, 4 x 4 epilogue warps
constexpr int kPiEpi = 512;                    // epilogue threads
constexpr int kPiList = 16;                    // entries of an epilogue thread's selection list
constexpr uint32_t kPiTile = 128 * 128;        // bytes of one e4m3 128 x 128 tile
constexpr uint32_t kPiStage = 2 * kPiTile;     // a unit's two key tiles, one 256-row operand
constexpr uint32_t kPiScales = 128 * 4;        // fp32 key scales of one block
constexpr uint32_t kPiSSlot = 2 * kPiScales;

template <int NST, bool SEL>
struct PiLayoutT {
  static constexpr uint32_t A = 0;                                  // [2 terms][16 KB]
  static constexpr uint32_t KT = 2 * kPiTile;                       // [stages][32 KB]
  static constexpr uint32_t KS = KT + NST * kPiStage;               // [scale slots][1 KB]
  // SEL: the epilogue threads' lists, [entry][thread] score keys then block ids
  static constexpr uint32_t LK = KS + kPiSStages * kPiSSlot;
  static constexpr uint32_t LI = LK + (SEL ? kPiList * kPiEpi * 4 : 0);
  static constexpr uint32_t BARS = LI + (SEL ? kPiList * kPiEpi * 2 : 0);  // mbarriers
  // kfull, kempty, sfull, sempty, tfull, tempty, afull, aempty, done
  static constexpr uint32_t NBARS = 2 * NST + 2 * kPiSStages + 2 * kPiAcc + 3;
  static constexpr uint32_t TSLOT = BARS + NBARS * 8;               // TMEM base from the allocator
  static constexpr uint32_t DEAD = TSLOT + 4;
  static constexpr uint32_t TOTAL = DEAD + 12;
  static constexpr uint32_t SMEM = TOTAL + 1024;                    // 1024-byte alignment slack
  static_assert(SMEM <= 232448, "shared memory of one CTA");
};

// Instruction descriptor: D fp32, A and B e4m3, both K-major, N = 256, M = 128.
constexpr uint32_t kIdescF8 = (1u << 4) | (0u << 7) | (0u << 10) | ((256u >> 3) << 17) | ((128u >> 4) << 24);

// ---------------------------------------------------------------- work walk

// The work units (sequence, query tile, key-block pair) in order:
// sequence-major, then tile, then pair.  Unit u of a tile covers key blocks 2u
// and 2u + 1 (the second absent when the sequence has an odd block count).  A
// sequence contributes tiles x ceil(blocks / 2) units; a malformed one (length
// outside [Q, max_blocks * 128]) none.
struct UnitCursor {
  int s, qt, b;  // b: the unit within the tile
  int nb;        // units of sequence s (kept so that walking reads no memory)
  int nblk;      // key blocks of sequence s
};

__device__ __forceinline__ int pi_seq_blocks(const BatchDev& bt, int s) {
  const int T = bt.seq_len(s);
  if (T < bt.Q || T > bt.max_nb * kBlock) return 0;
  return (T + kBlock - 1) / kBlock;
}

__device__ __forceinline__ void pi_locate(const BatchDev& bt, int tiles, long p, UnitCursor& c) {
  c.s = bt.S;
  c.qt = c.b = c.nb = c.nblk = 0;
  for (int s = 0; s < bt.S; ++s) {
    const int nblk = pi_seq_blocks(bt, s);
    const int nb = (nblk + 1) / 2;
    const long n = (long)tiles * nb;
    if (p < n) {
      c.s = s;
      c.nb = nb;
      c.nblk = nblk;
      c.qt = (int)(p / nb);
      c.b = (int)(p % nb);
      return;
    }
    p -= n;
  }
}

// k units further on (past the last unit: s = S)
__device__ __forceinline__ void pi_skip(const BatchDev& bt, int tiles, UnitCursor& c, int k) {
  c.b += k;
  while (c.s < bt.S && c.b >= c.nb) {
    c.b -= c.nb;
    if (++c.qt < tiles) continue;
    c.qt = 0;
    c.nb = c.nblk = 0;
    while (++c.s < bt.S) {
      c.nblk = pi_seq_blocks(bt, c.s);
      c.nb = (c.nblk + 1) / 2;
      if (c.nb > 0) break;
    }
  }
}

__device__ __forceinline__ void pi_advance(const BatchDev& bt, int tiles, UnitCursor& c) { pi_skip(bt, tiles, c, 1); }

__device__ __forceinline__ bool pi_wait(uint64_t* bar, uint32_t parity, int* dead, DeviceStatus* st, int where) {
  if (*reinterpret_cast<volatile int*>(dead)) return false;
  if (mbar_wait_sleep(bar, parity)) return true;
  *reinterpret_cast<volatile int*>(dead) = 1;
  raise_flag(st, FLAG_TIMEOUT, where);
  return false;
}

// ---------------------------------------------------------------- the kernel

template <bool SEL>
__global__ void __launch_bounds__(kPiThreads, 1) pindexer_kernel(const __grid_constant__ CUtensorMap tmap,
                                                               const PrefillIndexerParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int NSTG = SEL ? kPiStagesSel : kPiStages;
  using LY = PiLayoutT<NSTG, SEL>;
  uint64_t* kfull = reinterpret_cast<uint64_t*>(base + LY::BARS);
  uint64_t* kempty = kfull + NSTG;
  uint64_t* sfull = kempty + NSTG;
  uint64_t* sempty = sfull + kPiSStages;
  uint64_t* tfull = sempty + kPiSStages;
  uint64_t* tempty = tfull + kPiAcc;
  uint64_t* afull = tempty + kPiAcc;
  uint64_t* aempty = afull + 1;
  uint64_t* done = aempty + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(base + LY::TSLOT);
  int* dead = reinterpret_cast<int*>(base + LY::DEAD);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const BatchDev bt = p.batch;
  const int G = p.G, Q = bt.Q;
  const int tpt = 128 / G;                 // query tokens per tile
  const int tiles = (Q + tpt - 1) / tpt;
  const int terms = p.iq_fp8 ? 1 : 2;

  // this CTA's units [p0, p1)
  long P = 0;
  for (int s = 0; s < bt.S; ++s) P += (long)tiles * ((pi_seq_blocks(bt, s) + 1) / 2);
  const long p0 = (long)blockIdx.x * P / gridDim.x, p1 = (long)(blockIdx.x + 1) * P / gridDim.x;
  const int nunits = (int)(p1 - p0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSTG; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);  // the MMA commit
    }
    for (int i = 0; i < kPiSStages; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], 8);  // the unit's eight epilogue warps
    }
    for (int i = 0; i < kPiAcc; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 8);
    }
    mbar_init(afull, 8);
    mbar_init(aempty, 1);
    mbar_init(done, 1);
    *dead = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap);
  }
  if (warp == 1) tmem_alloc(smem_u32(tslot), kPiCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    // ---------------- key tiles and scales into the ring.  The block-table
    // entries of 32 units at a time are read by the 32 lanes together.
    UnitCursor c;
    pi_locate(bt, tiles, p0, c);
    int issued = 0;
    bool ok = true;
    for (int j0 = 0; j0 < nunits && ok; j0 += 32) {
      UnitCursor cl = c;
      pi_skip(bt, tiles, cl, lane);
      // physical blocks of this lane's unit (-2: no second block)
      const bool mine = j0 + lane < nunits;
      const int my_ph0 = mine ? bt.row(cl.s)[2 * cl.b] : -1;
      const int my_ph1 = (mine && 2 * cl.b + 1 < cl.nblk) ? bt.row(cl.s)[2 * cl.b + 1] : -2;
      const int my_qt = cl.qt;
      for (int t = 0; t < 32 && j0 + t < nunits; ++t) {
        const int ph0 = __shfl_sync(0xffffffffu, my_ph0, t);
        const int ph1 = __shfl_sync(0xffffffffu, my_ph1, t);
        const int qt = __shfl_sync(0xffffffffu, my_qt, t);
        const int j = j0 + t;
        if (lane == 0) {
          const int st = j % NSTG, ss = j % kPiSStages;
          if ((j >= NSTG && !pi_wait(&kempty[st], (uint32_t)(((j / NSTG) - 1) & 1), dead, p.status, 1)) ||
              (j >= kPiSStages && !pi_wait(&sempty[ss], (uint32_t)(((j / kPiSStages) - 1) & 1), dead, p.status, 8))) {
            ok = false;
          } else {
            uint8_t* kt = base + LY::KT + (size_t)st * kPiStage;
            uint8_t* ks = base + LY::KS + (size_t)ss * kPiSSlot;
            const bool v0 = ph0 >= 0 && ph0 < p.num_blocks;
            const bool v1 = ph1 >= 0 && ph1 < p.num_blocks;
            if (qt == 0 && !v0) raise_flag(p.status, FLAG_BAD_BLOCK, ph0);
            if (qt == 0 && ph1 != -2 && !v1) raise_flag(p.status, FLAG_BAD_BLOCK, ph1);
            // a block that is absent or rejected is not copied (its half of the
            // operand keeps stale bytes, its scores are not used); a unit with
            // nothing to copy completes its phases by plain arrivals
            if (v0 || v1) {
              fence_proxy_async();
              mbar_expect_tx(&kfull[st], (v0 ? kPiTile : 0u) + (v1 ? kPiTile : 0u));
              if (v0) tma_load_2d(kt, &tmap, 0, ph0 * kBlock, &kfull[st]);
              if (v1) tma_load_2d(kt + kPiTile, &tmap, 0, ph1 * kBlock, &kfull[st]);
              mbar_expect_tx(&sfull[ss], (v0 ? kPiScales : 0u) + (v1 ? kPiScales : 0u));
              if (v0) bulk_g2s(ks, p.idx_scale + (size_t)ph0 * kBlock, kPiScales, &sfull[ss]);
              if (v1) bulk_g2s(ks + kPiScales, p.idx_scale + (size_t)ph1 * kBlock, kPiScales, &sfull[ss]);
            } else {
              mbar_arrive(&kfull[st]);
              mbar_arrive(&sfull[ss]);
            }
            issued = j + 1;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      pi_skip(bt, tiles, c, 32);
    }
    // a CTA that gave up waits (bounded) for the copies it issued
    if (lane == 0) {
      for (int i = 0; i < NSTG && i < issued; ++i) {
        const int jj = issued - 1 - i;
        mbar_wait_sleep(&kfull[jj % NSTG], (uint32_t)((jj / NSTG) & 1), 2000);
      }
      for (int i = 0; i < kPiSStages && i < issued; ++i) {
        const int jj = issued - 1 - i;
        mbar_wait_sleep(&sfull[jj % kPiSStages], (uint32_t)((jj / kPiSStages) & 1), 2000);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issue (one thread)
    if (lane == 0) {
      UnitCursor c;
      pi_locate(bt, tiles, p0, c);
      int a_use = 0, cur_tile = -1, cur_s = -1;
      const uint32_t a0 = smem_u32(base + LY::A);
      for (int j = 0; j < nunits; ++j) {
        if (c.qt != cur_tile || c.s != cur_s) {
          if (!pi_wait(afull, (uint32_t)(a_use & 1), dead, p.status, 2)) break;
          ++a_use;
          cur_tile = c.qt;
          cur_s = c.s;
        }
        const int st = j % NSTG, ab = j % kPiAcc;
        if (!pi_wait(&kfull[st], (uint32_t)((j / NSTG) & 1), dead, p.status, 3)) break;
        if (j >= kPiAcc && !pi_wait(&tempty[ab], (uint32_t)(((j / kPiAcc) - 1) & 1), dead, p.status, 4)) break;
        tc_fence_after();
        const uint32_t bt0 = smem_u32(base + LY::KT + (size_t)st * kPiStage);
        const uint32_t d = tmem + (uint32_t)(ab * 256);
#pragma unroll 1
        for (int term = 0; term < terms; ++term)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f8(d, sw128_desc(a0 + term * kPiTile + 32 * k), sw128_desc(bt0 + 32 * k), kIdescF8,
                   (term | k) != 0);
        mma_commit(&tfull[ab]);
        mma_commit(&kempty[st]);
        pi_advance(bt, tiles, c);
        if (j + 1 == nunits || c.qt != cur_tile || c.s != cur_s) mma_commit(aempty);  // the query tile is free
      }
      mma_commit(done);
      mbar_wait_sleep(done, 0, 200000);
    }
  } else {
    // ---------------- query tiles + epilogue (thread = accumulator row)
    const int quarter = warp & 3;          // TMEM lanes 32 * quarter .. + 31
    const int egrp = (warp - 2) >> 2;      // 0..3
    const int group = egrp >> 1;           // takes the units j with j % 2 == group
    const int hb = egrp & 1;               // and key block hb of each
    const bool builder = hb == 0;          // groups 0 and 2 build the query operand (hi / lo)
    const int m = 32 * quarter + lane;     // row of the tile: token m / G, group m % G
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
    UnitCursor c;
    pi_locate(bt, tiles, p0, c);
    int a_use = 0, cur_tile = -1, cur_s = -1;
    int T = 0, pos = -1;
    bool row_ok = false;
    float rowf = 0.f;
    float* prow = nullptr;
    // SEL: the list slot of (this CTA, tile) is tile + the CTA's rank among the
    // CTAs with units (min(b, first unit): with more CTAs than units each holds
    // one or none), unique since later CTAs start at or after this one's tiles.
    const long cta_rank = blockIdx.x < p0 ? (long)blockIdx.x : p0;
    // SEL: this thread's 16 best free blocks of its row in the current tile,
    // in shared memory ([entry][thread]: conflict-free) as a binary heap whose
    // root is the worst entry (smallest score key, of those the largest block
    // id: the one the top-k rule gives up first); registers hold the count and
    // the root's key
    const int et = (int)threadIdx.x - 64;
    uint32_t* lks = reinterpret_cast<uint32_t*>(base + LY::LK) + et;
    uint16_t* lis = reinterpret_cast<uint16_t*>(base + LY::LI) + et;
    int lcnt = 0;
    uint32_t lwk = 0;
    int flo = 0, fhi = 0;  // the row's free candidate blocks [flo, fhi)
    // place (xk, xi) at heap position h, moving worse children up
    auto sift_down = [&](int h, uint32_t xk, int xi) {
#pragma unroll 1
      while (2 * h + 1 < kPiList) {
        int c = 2 * h + 1;
        uint32_t ck = lks[c * kPiEpi];
        int ci = lis[c * kPiEpi];
        if (c + 1 < kPiList) {
          const uint32_t dk = lks[(c + 1) * kPiEpi];
          const int di = lis[(c + 1) * kPiEpi];
          if (dk < ck || (dk == ck && di > ci)) {
            c = c + 1;
            ck = dk;
            ci = di;
          }
        }
        if (!(ck < xk || (ck == xk && ci > xi))) break;  // the child is not worse: x stays
        lks[h * kPiEpi] = ck;
        lis[h * kPiEpi] = (uint16_t)ci;
        h = c;
      }
      lks[h * kPiEpi] = xk;
      lis[h * kPiEpi] = (uint16_t)xi;
    };
    auto list_flush = [&]() {
      if constexpr (SEL) {
        if (cur_tile < 0 || !row_ok) return;
        const size_t slot = (size_t)cur_s * tiles + cur_tile + cta_rank;
        uint4* dst = reinterpret_cast<uint4*>(p.lists + ((slot * 128 + m) * 4 + egrp) * kPiList);
#pragma unroll 1
        for (int k = 0; k < kPiList; k += 2) {
          // 64-bit keys: score key above, ~block id below (0: no entry)
          const uint64_t e0 = k < lcnt ? ((uint64_t)lks[k * kPiEpi] << 32) | ~(uint32_t)lis[k * kPiEpi] : 0ull;
          const uint64_t e1 =
              k + 1 < lcnt ? ((uint64_t)lks[(k + 1) * kPiEpi] << 32) | ~(uint32_t)lis[(k + 1) * kPiEpi] : 0ull;
          dst[k / 2] = make_uint4((uint32_t)e0, (uint32_t)(e0 >> 32), (uint32_t)e1, (uint32_t)(e1 >> 32));
        }
      }
    };
    auto list_add = [&](int blk, float score) {
      if constexpr (SEL) {
        if (blk < flo || blk >= fhi) return;  // forced or not visible
        const uint32_t key = float_order_key(score);
        if (lcnt < kPiList) {
          lks[lcnt * kPiEpi] = key;
          lis[lcnt * kPiEpi] = (uint16_t)blk;
          if (++lcnt == kPiList) {  // full: heap order, bottom up
#pragma unroll 1
            for (int h = kPiList / 2 - 1; h >= 0; --h) sift_down(h, lks[h * kPiEpi], lis[h * kPiEpi]);
            lwk = lks[0];
          }
        } else if (key > lwk) {  // the thread's blocks come in increasing id order: an equal key loses
          sift_down(0, key, blk);
          lwk = lks[0];
        }
      }
    };
    for (int j = 0; j < nunits; ++j) {
      if (c.qt != cur_tile || c.s != cur_s) {
        list_flush();  // the tile this thread leaves
        // the MMAs of the previous tile must be done before its operand is overwritten
        if (a_use > 0 && !pi_wait(aempty, (uint32_t)((a_use - 1) & 1), dead, p.status, 5)) break;
        cur_tile = c.qt;
        cur_s = c.s;
        const int i = cur_tile * tpt + m / G, g = m % G;
        T = bt.seq_len(cur_s);
        row_ok = i < Q;
        pos = T - Q + i;
        prow = p.pooled + ((size_t)(cur_s * Q + i) * G + g) * bt.max_nb;
        if constexpr (SEL) {
          lcnt = 0;
          // the top-k rule's candidates: past the forced init blocks, before the
          // forced local blocks and the row's own block
          const int recent = max(pos, 0) / kBlock;
          const int n_init = min(p.init_blocks, recent);
          const int n_local = min(p.local_blocks, recent - n_init);
          flo = n_init;
          fhi = recent - n_local;
        }
        // this row of the operand: hi (and lo) e4m3, 16-byte chunks swizzled by row
        uint8_t* ahi = base + LY::A + (size_t)m * 128;
        uint8_t* alo = ahi + kPiTile;
        const size_t qoff = ((size_t)(cur_s * Q + i) * G + g) * kDim;
        if (p.iq_fp8) {
          const uint8_t* src = static_cast<const uint8_t*>(p.index_q) + qoff;
#pragma unroll
          for (int ch = 0; ch < 8 && builder && group == 0; ++ch) {
            const uint4 v = row_ok ? *reinterpret_cast<const uint4*>(src + 16 * ch) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(ahi + ((ch ^ (m & 7)) << 4)) = v;
          }
          rowf = p.iq_scale * p.col_const;
        } else {
          const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(p.index_q) + qoff;
          float amax = 0.f;
          for (int ch = 0; ch < 16; ++ch) {
            const uint4 v = row_ok ? *reinterpret_cast<const uint4*>(src + 8 * ch) : make_uint4(0, 0, 0, 0);
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(h[e]);
              amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          }
          const int ex = pow2_fit(amax, 448.f);
          const float ps = ldexpf(1.f, ex);
          rowf = ldexpf(1.f, -ex) * p.col_const;
          for (int ch = 0; ch < 8; ++ch) {  // 16 dims a chunk
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const uint4 v = row_ok ? *reinterpret_cast<const uint4*>(src + 16 * ch + 8 * half) : make_uint4(0, 0, 0, 0);
              const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
              for (int e = 0; e < 4; e += 2) {
                const float2 f0 = __bfloat1622float2(h[e]), f1 = __bfloat1622float2(h[e + 1]);
                float h0, l0, h1, l1, h2, l2, h3, l3;
                split_e4m3(f0.x * ps, h0, l0);
                split_e4m3(f0.y * ps, h1, l1);
                split_e4m3(f1.x * ps, h2, l2);
                split_e4m3(f1.y * ps, h3, l3);
                hw[2 * half + e / 2] = (uint32_t)pack_e4m3x2(h0, h1) | ((uint32_t)pack_e4m3x2(h2, h3) << 16);
                lw[2 * half + e / 2] = (uint32_t)pack_e4m3x2(l0, l1) | ((uint32_t)pack_e4m3x2(l2, l3) << 16);
              }
            }
            if (!builder) continue;
            if (group == 0) *reinterpret_cast<uint4*>(ahi + ((ch ^ (m & 7)) << 4)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            else *reinterpret_cast<uint4*>(alo + ((ch ^ (m & 7)) << 4)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
        if (builder) {
          fence_proxy_async();  // the MMA reads the operand through the async proxy
          __syncwarp();
          if (lane == 0) mbar_arrive(afull);
        }
        ++a_use;
      }
      if ((j & 1) != group) {  // the other group's unit
        pi_advance(bt, tiles, c);
        continue;
      }
      const int ab = j % kPiAcc;
      const int nblocks = (2 * c.b + 1 < c.nblk) ? 2 : 1;  // the unit's key blocks
      // physical blocks, used at the end: their latency hides behind the waits
      const int ph0 = hb == 0 ? bt.row(c.s)[2 * c.b] : -1;
      const int ph1 = (hb == 1 && nblocks == 2) ? bt.row(c.s)[2 * c.b + 1] : -1;
      if (!pi_wait(&tfull[ab], (uint32_t)((j / kPiAcc) & 1), dead, p.status, 6)) break;
      // the unit's key scales (their own ring: the slot is not reused before
      // this group releases it)
      const int ss = j % kPiSStages;
      if (!pi_wait(&sfull[ss], (uint32_t)((j / kPiSStages) & 1), dead, p.status, 7)) break;
      tc_fence_after();
      float mxs[2] = {-INFINITY, -INFINITY};
#pragma unroll 1
      for (int h = hb; h < nblocks && h == hb; ++h) {  // this group's block of the unit, if it has one
        const float* ks = reinterpret_cast<const float*>(base + LY::KS + (size_t)ss * kPiSSlot) + 128 * h;
        const int key0 = (2 * c.b + h) * kBlock;
        const bool full_vis = key0 + kBlock - 1 <= pos;
        float mx = -INFINITY;
#pragma unroll 1
        for (int half = 0; half < 4; ++half) {  // 32 columns a load (more warps hide the wait)
          float v[1][32];
          const uint32_t col = (uint32_t)(ab * 256 + 128 * h + 32 * half);
          tmem_ld32(lane_addr + col, v[0]);
          tmem_ld_wait();
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int q = 0; q < 1; ++q) {
            const int n0 = 32 * half;
            if (full_vis) {
              const float4* k4 = reinterpret_cast<const float4*>(ks + n0);
#pragma unroll
              for (int n = 0; n < 32; n += 8) {
                const float4 ka = k4[n >> 2], kb = k4[(n >> 2) + 1];
                const float2 p0 = mul2(v[q][n], v[q][n + 1], ka.x, ka.y);
                const float2 p1 = mul2(v[q][n + 2], v[q][n + 3], ka.z, ka.w);
                const float2 p2 = mul2(v[q][n + 4], v[q][n + 5], kb.x, kb.y);
                const float2 p3 = mul2(v[q][n + 6], v[q][n + 7], kb.z, kb.w);
                m4[0] = max3(m4[0], p0.x, p0.y);
                m4[1] = max3(m4[1], p1.x, p1.y);
                m4[2] = max3(m4[2], p2.x, p2.y);
                m4[3] = max3(m4[3], p3.x, p3.y);
              }
            } else {
#pragma unroll
              for (int n = 0; n < 32; ++n) {
                const float sc = (key0 + n0 + n <= pos) ? v[q][n] * ks[n0 + n] : -INFINITY;
                m4[n & 3] = fmaxf(m4[n & 3], sc);
              }
            }
          }
          mx = fmaxf(mx, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
        }
        mxs[h] = mx;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tempty[ab]);  // the accumulator may be overwritten
        mbar_arrive(&sempty[ss]);  // done with the scales
      }
      if constexpr (SEL) {
        if (row_ok && hb == 0) list_add(2 * c.b, (ph0 >= 0 && ph0 < p.num_blocks) ? mxs[0] * rowf : -INFINITY);
        if (row_ok && hb == 1 && nblocks == 2)
          list_add(2 * c.b + 1, (ph1 >= 0 && ph1 < p.num_blocks) ? mxs[1] * rowf : -INFINITY);
      } else {
        if (row_ok && hb == 0) prow[2 * c.b] = (ph0 >= 0 && ph0 < p.num_blocks) ? mxs[0] * rowf : -INFINITY;
        if (row_ok && hb == 1 && nblocks == 2)
          prow[2 * c.b + 1] = (ph1 >= 0 && ph1 < p.num_blocks) ? mxs[1] * rowf : -INFINITY;
      }
      pi_advance(bt, tiles, c);
    }
    list_flush();  // the last tile of the run
  }

  // blocks that hold no key of a sequence (past its length, or all of a
  // malformed sequence): -inf for every (token, group) row, a row per warp
  if constexpr (!SEL) {
    const long rows = (long)bt.S * Q * G;
    const long nw = (long)gridDim.x * (kPiThreads / 32);
    for (long row = (long)blockIdx.x * (kPiThreads / 32) + warp; row < rows; row += nw) {
      const int nb = pi_seq_blocks(bt, (int)(row / ((long)Q * G)));
      float* pr = p.pooled + row * bt.max_nb;
      for (int b = nb + lane; b < bt.max_nb; b += 32) pr[b] = -INFINITY;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    for (int s = 0; s < bt.S; ++s)
      if (pi_seq_blocks(bt, s) == 0) raise_flag(p.status, FLAG_BAD_SEQLEN, s);
  }
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kPiCols);
}

template <bool SEL>
cudaError_t launch_pi(const CUtensorMap* tmap, const PrefillIndexerParams& p, int num_sms, cudaStream_t st) {
  const size_t smem = PiLayoutT<SEL ? kPiStagesSel : kPiStages, SEL>::SMEM;
  auto kern = pindexer_kernel<SEL>;
  static bool ready = false;
  if (!ready) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kPiThreads, smem);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    ready = true;
  }
  kern<<<prefill_indexer_grid(num_sms), kPiThreads, smem, st>>>(*tmap, p);
  return cudaGetLastError();
}

}  // namespace

// all 512 TMEM columns: one CTA per SM
int prefill_indexer_grid(int num_sms) { return num_sms > 0 ? num_sms : 1; }

cudaError_t launch_prefill_indexer(const CUtensorMap* tmap, const PrefillIndexerParams& p, int num_sms,
                                   cudaStream_t st) {
  return p.lists ? launch_pi<true>(tmap, p, num_sms, st) : launch_pi<false>(tmap, p, num_sms, st);
}

namespace {

constexpr int kSelRows = 8;  // rows (warps) a CTA

__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
  const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)v, src);
  const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(v >> 32), src);
  return ((uint64_t)hi << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int o) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, o);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), o);
  return ((uint64_t)hi << 32) | lo;
}

// One warp per (token, group) row (vLLM Day-0 blog, "MSA 入门": the top-k
// blocks by pooled score, the most recent one always kept; forced init / local
// blocks as topk_kernel).  The row's tile was scored by the CTAs whose unit runs
// meet the tile's units (the indexer's static partition, unit u in CTA
// (((u + 1) * grid - 1) / P)); each left four lists of its epilogue groups'
// 16 best free blocks.  Every free block among the row's kfree best is in one of
// them, so kfree rounds of "largest key below the last one" over the lists
// give the selection; block ids come out ascending by their rank among the picks.
__global__ void __launch_bounds__(32 * kSelRows) pi_select_kernel(const PiSelectParams p) {
  __shared__ int outb[kSelRows][32];
  __shared__ uint64_t skey[kSelRows][64];
  pdl_launch_dependents();
  pdl_wait();  // the lists come from the indexer
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BatchDev bt = p.batch;
  const int G = p.G, Q = bt.Q, K = p.topk;
  const int rows = bt.S * Q * G;  // below 2^31 (make_plan)
  const int row = blockIdx.x * kSelRows + warp;
  if (row >= rows) return;
  const int sq = row / G, g = row - sq * G;
  const int s = sq / Q, i = sq - s * Q;
  const int T = bt.seq_len(s);
  int* out = outb[warp];
  int id = -1;
  if (T < Q || T > bt.max_nb * kBlock) {
    if (lane == 0 && i == 0 && g == 0) raise_flag(p.status, FLAG_BAD_SEQLEN, s);
  } else {
    const int pos = T - Q + i;
    const int recent = pos / kBlock;
    const int n_init = min(p.init_blocks, recent);
    const int n_local = min(p.local_blocks, recent - n_init);
    const int lo = n_init, hi = recent - n_local;
    const int ncand = hi - lo;
    const int kfree = K - n_init - n_local - 1;
    int n_sel = 0;
    if (ncand <= kfree) {
      for (int c = lane; c < ncand; c += 32) out[n_init + c] = lo + c;
      n_sel = ncand;
    } else if (kfree > 0) {
      n_sel = kfree;
      const int tpt = 128 / G, tiles = (Q + tpt - 1) / tpt;
      const int qt = i / tpt, m = (i - qt * tpt) * G + g;
      long P = 0, base = 0;
      int nb = 0;
      for (int s2 = 0; s2 < bt.S; ++s2) {
        const int n2 = (pi_seq_blocks(bt, s2) + 1) / 2;
        if (s2 < s) base += (long)tiles * n2;
        if (s2 == s) nb = n2;
        P += (long)tiles * n2;
      }
      const long gr = p.grid;
      // unit u is in CTA ((u + 1) * grid - 1) / P and CTA b starts at unit b * P / grid;
      // 32-bit divisions where the products fit
      const bool narrow = P * gr < (1l << 32);
      auto div_p = [&](long x) -> long { return narrow ? (long)((uint32_t)x / (uint32_t)P) : x / P; };
      auto div_g = [&](long x) -> long { return narrow ? (long)((uint32_t)x / (uint32_t)gr) : x / gr; };
      const long u0 = base + (long)qt * nb, u1 = u0 + nb - 1;  // the tile's units
      const int b0 = (int)div_p((u0 + 1) * gr - 1), b1 = (int)div_p((u1 + 1) * gr - 1);
      // (CTA b, this tile)'s slot: tile + min(b, b's first unit)
      const size_t tau = (size_t)s * tiles + qt;
      auto list_of = [&](int b, long first) {
        return reinterpret_cast<const unsigned long long*>(p.lists) + ((tau + (b < first ? b : first)) * 128 + m) * 64;
      };
      // up to four CTAs' lists held in registers, two keys a lane of each
      constexpr int kSegReg = 4;
      uint64_t kr[2 * kSegReg];
#pragma unroll
      for (int k = 0; k < 2 * kSegReg; ++k) kr[k] = 0;
      int nseg = 0;
      long first = div_g((long)b0 * P);
      for (int b = b0; b <= b1; ++b) {
        const long next = div_g((long)(b + 1) * P);
        if (first != next) {  // a CTA with units
          if (nseg < kSegReg) {
            const unsigned long long* L = list_of(b, first);
#pragma unroll
            for (int k = 0; k < kSegReg; ++k)
              if (k == nseg) {
                kr[2 * k] = __ldcg(L + lane);
                kr[2 * k + 1] = __ldcg(L + lane + 32);
              }
          }
          ++nseg;
        }
        first = next;
      }
      uint32_t mine = 0xffffffffu;  // selected lanes: ~id of a pick
      bool done = false;
      if (nseg <= kSegReg) {
        // T = the kfree-th largest lane maximum bounds the picks from below;
        // the keys >= T (at least kfree, usually a few dozen) are ranked
        uint64_t lm = 0;
#pragma unroll
        for (int k = 0; k < 2 * kSegReg; ++k) lm = kr[k] > lm ? kr[k] : lm;
        int rk = 0;
#pragma unroll 8
        for (int x = 0; x < 32; ++x) {
          const uint64_t o = shfl_u64(lm, x);
          rk += (o > lm) || (o == lm && x < lane);
        }
        const unsigned who = __ballot_sync(0xffffffffu, rk == kfree - 1);
        uint64_t T = shfl_u64(lm, __ffs(who) - 1);
        if (T == 0) T = 1;  // empty entries are 0
        uint64_t* sk = skey[warp];
        int C = 0;
#pragma unroll
        for (int k = 0; k < 2 * kSegReg; ++k) {
          const bool in = kr[k] >= T;
          const unsigned bal = __ballot_sync(0xffffffffu, in);
          const int at = C + __popc(bal & ((1u << lane) - 1u));
          if (in && at < 64) sk[at] = kr[k];
          C += __popc(bal);
        }
        __syncwarp();
        if (C <= 64) {
          // kept iff fewer than kfree keys beat it (keys are unique)
          bool keep[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int e = lane + 32 * h;
            keep[h] = false;
            if (e < C) {
              const uint64_t ke = sk[e];
              int beat = 0;
              for (int x = 0; x < C; ++x) beat += sk[x] > ke;
              keep[h] = beat < kfree;
            }
          }
          const unsigned k0 = __ballot_sync(0xffffffffu, keep[0]), k1 = __ballot_sync(0xffffffffu, keep[1]);
          // the picks to lanes 0..kfree-1
          const int n0 = __popc(k0);
          uint32_t v0 = keep[0] ? (uint32_t)sk[lane] : 0u, v1 = keep[1] ? (uint32_t)sk[lane + 32] : 0u;
          __syncwarp();
          if (keep[0]) reinterpret_cast<uint32_t*>(sk)[__popc(k0 & ((1u << lane) - 1u))] = v0;
          if (keep[1]) reinterpret_cast<uint32_t*>(sk)[n0 + __popc(k1 & ((1u << lane) - 1u))] = v1;
          __syncwarp();
          if (lane < kfree) mine = reinterpret_cast<uint32_t*>(sk)[lane];
          __syncwarp();
          done = true;
        }
      }
      if (!done) {
        // kfree rounds of "largest key below the last one"
        uint64_t prev = ~0ull;
        for (int r = 0; r < kfree; ++r) {
          uint64_t best = 0;
          if (nseg <= kSegReg) {
#pragma unroll
            for (int k = 0; k < 2 * kSegReg; ++k)
              if (kr[k] < prev && kr[k] > best) best = kr[k];
          } else {  // more CTAs than fit (short sequences): read the lists again
            long f = div_g((long)b0 * P);
            for (int b = b0; b <= b1; ++b) {
              const long next = div_g((long)(b + 1) * P);
              if (f != next) {
                const unsigned long long* L = list_of(b, f);
                const uint64_t k0 = __ldcg(L + lane), k1 = __ldcg(L + lane + 32);
                if (k0 < prev && k0 > best) best = k0;
                if (k1 < prev && k1 > best) best = k1;
              }
              f = next;
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const uint64_t y = shfl_xor_u64(best, o);
            if (y > best) best = y;
          }
          prev = best;
          if (lane == r) mine = (uint32_t)best;
        }
      }
      const uint32_t blk = ~mine;
      int rank = 0;
      for (int x = 0; x < kfree; ++x) rank += (~__shfl_sync(0xffffffffu, mine, x) < blk);
      if (lane < kfree) out[n_init + rank] = (int)blk;
    }
    for (int k = lane; k < n_init; k += 32) out[k] = k;
    const int tail = n_init + n_sel;
    for (int k = tail + lane; k < K; k += 32) {
      const int b = hi + (k - tail);
      out[k] = (b <= recent) ? b : -1;
    }
    __syncwarp();
    id = (lane < K) ? out[lane] : -1;
  }
  if (lane < K) p.topk_idx[(size_t)row * K + lane] = id;
}

}  // namespace

cudaError_t launch_prefill_select(const PiSelectParams& p, cudaStream_t st) {
  const long rows = (long)p.batch.S * p.batch.Q * p.G;
  const long grid = (rows + kSelRows - 1) / kSelRows;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(grid > 0 ? grid : 1));
  cfg.blockDim = dim3(32 * kSelRows);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pi_select_kernel, p);
}

}  // namespace msa
