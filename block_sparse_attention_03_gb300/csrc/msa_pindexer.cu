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
#include "msa_device.cuh"
#include "msa_internal.h"
#include "msa_tcgen05.cuh"

namespace msa {

namespace {

constexpr int kPiStages = 5;                   // units (two key tiles) in flight: L2 latency x the MMA rate
constexpr int kPiSStages = 16;                 // key-scale slots (released by the epilogue, which lags)
constexpr int kPiAcc = 2;                      // accumulators of 256 columns (two key blocks)
constexpr int kPiCols = 256 * kPiAcc;          // TMEM columns (all 512 of the SM: one CTA per SM)
constexpr int kPiThreads = 576;                // producer, MMA, 4 x 4 epilogue warps
constexpr uint32_t kPiTile = 128 * 128;        // bytes of one e4m3 128 x 128 tile
constexpr uint32_t kPiStage = 2 * kPiTile;     // a unit's two key tiles, one 256-row operand
constexpr uint32_t kPiScales = 128 * 4;        // fp32 key scales of one block
constexpr uint32_t kPiSSlot = 2 * kPiScales;

struct PiLayout {
  static constexpr uint32_t A = 0;                                  // [2 terms][16 KB]
  static constexpr uint32_t KT = 2 * kPiTile;                       // [stages][32 KB]
  static constexpr uint32_t KS = KT + kPiStages * kPiStage;         // [scale slots][1 KB]
  static constexpr uint32_t BARS = KS + kPiSStages * kPiSSlot;      // mbarriers
  // kfull, kempty, sfull, sempty, tfull, tempty, afull, aempty, done
  static constexpr uint32_t NBARS = 2 * kPiStages + 2 * kPiSStages + 2 * kPiAcc + 3;
  static constexpr uint32_t TSLOT = BARS + NBARS * 8;               // TMEM base from the allocator
  static constexpr uint32_t DEAD = TSLOT + 4;
  static constexpr uint32_t TOTAL = DEAD + 12;
  static constexpr uint32_t SMEM = TOTAL + 1024;                    // 1024-byte alignment slack
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
  if (mbar_wait(bar, parity)) return true;
  *reinterpret_cast<volatile int*>(dead) = 1;
  raise_flag(st, FLAG_TIMEOUT, where);
  return false;
}

// ---------------------------------------------------------------- the kernel

__global__ void __launch_bounds__(kPiThreads, 1) pindexer_kernel(const __grid_constant__ CUtensorMap tmap,
                                                               const PrefillIndexerParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using LY = PiLayout;
  uint64_t* kfull = reinterpret_cast<uint64_t*>(base + LY::BARS);
  uint64_t* kempty = kfull + kPiStages;
  uint64_t* sfull = kempty + kPiStages;
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
    for (int i = 0; i < kPiStages; ++i) {
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
          const int st = j % kPiStages, ss = j % kPiSStages;
          if ((j >= kPiStages && !pi_wait(&kempty[st], (uint32_t)(((j / kPiStages) - 1) & 1), dead, p.status, 1)) ||
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
      for (int i = 0; i < kPiStages && i < issued; ++i) {
        const int jj = issued - 1 - i;
        mbar_wait(&kfull[jj % kPiStages], (uint32_t)((jj / kPiStages) & 1), 2000);
      }
      for (int i = 0; i < kPiSStages && i < issued; ++i) {
        const int jj = issued - 1 - i;
        mbar_wait(&sfull[jj % kPiSStages], (uint32_t)((jj / kPiSStages) & 1), 2000);
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
        const int st = j % kPiStages, ab = j % kPiAcc;
        if (!pi_wait(&kfull[st], (uint32_t)((j / kPiStages) & 1), dead, p.status, 3)) break;
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
      mbar_wait(done, 0, 200000);
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
    for (int j = 0; j < nunits; ++j) {
      if (c.qt != cur_tile || c.s != cur_s) {
        // the MMAs of the previous tile must be done before its operand is overwritten
        if (a_use > 0 && !pi_wait(aempty, (uint32_t)((a_use - 1) & 1), dead, p.status, 5)) break;
        cur_tile = c.qt;
        cur_s = c.s;
        const int i = cur_tile * tpt + m / G, g = m % G;
        T = bt.seq_len(cur_s);
        row_ok = i < Q;
        pos = T - Q + i;
        prow = p.pooled + ((size_t)(cur_s * Q + i) * G + g) * bt.max_nb;
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
      if (row_ok && hb == 0) prow[2 * c.b] = (ph0 >= 0 && ph0 < p.num_blocks) ? mxs[0] * rowf : -INFINITY;
      if (row_ok && hb == 1 && nblocks == 2)
        prow[2 * c.b + 1] = (ph1 >= 0 && ph1 < p.num_blocks) ? mxs[1] * rowf : -INFINITY;
      pi_advance(bt, tiles, c);
    }
  }

  // blocks that hold no key of a sequence (past its length, or all of a
  // malformed sequence): -inf for every (token, group) row, a row per warp
  {
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

}  // namespace

cudaError_t launch_prefill_indexer(const CUtensorMap* tmap, const PrefillIndexerParams& p, int num_sms,
                                   cudaStream_t st) {
  const size_t smem = PiLayout::SMEM;
  static int per_sm = 0;
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(pindexer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(pindexer_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, pindexer_kernel, kPiThreads, smem);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    per_sm = 1;  // all 512 TMEM columns: one CTA per SM
  }
  const int grid = per_sm * (num_sms > 0 ? num_sms : 1);
  pindexer_kernel<<<grid, kPiThreads, smem, st>>>(*tmap, p);
  return cudaGetLastError();
}

}  // namespace msa
