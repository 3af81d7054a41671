// Indexer score + block max-pool over the paged index-key cache (decode and
// speculative verify: up to 64 (query x group) columns per sequence).
//
// Definition (vLLM Day-0 blog, section "MSA 入门"): every key t of the context
// is scored against one index query per GQA group through the single shared
// index-key head, s = scale * <index_q[g], key[t]>, and the scores are
// max-pooled to one value per 128-token block; keys a query cannot see
// (t > its position) do not take part.
//
// GB300 mapping.  The scan is HBM-bound (128 B/token for FP8 keys), but at
// 4 groups x 128 dims it needs 4 MACs per byte, more than the FP32 pipe can
// issue at HBM rate, so the dot products run on the tensor pipe:
//   S^T[key][col] = Keys[128 x 128] * Q^T[128 x cols]   (mma.sync, keys = rows)
// Each warp owns a private ring of NST shared-memory stages (several CTAs per
// SM, so 12 warps per SM hide the copy latency); lane 0 streams whole
// 128-token blocks into it (TMA tensor copy with the 128-byte swizzle
// for FP8/BF16, so ldmatrix reads are bank-conflict free; a 1-D bulk copy for
// NVFP4, whose 64-byte rows are read conflict-free as they are).  Keys are fed
// to the MMA without conversion (e4m3 / bf16) or dequantized exactly to f16 in
// registers (NVFP4: e2m1 -> f16, times the e4m3 block scale, an exact product).
// The per-token FP8 scale multiplies each row before the block max; the
// column factor (query scale, power-of-two prescale, index scale, NVFP4
// per-tensor scale: all positive) is applied after it.
//
// Work: unit = (sequence s, logical block b) over the blocks that hold keys,
// in sequence-major order, one contiguous run of units per warp; blocks past
// a sequence's end get -inf in a separate spread pass.
#include "msa_device.cuh"
#include "msa_internal.h"
#include "msa_qfrag.cuh"

namespace msa {

namespace {

template <int FMT>
struct IdxTraits;

template <>
struct IdxTraits<FMT_FP8> {
  static constexpr int KS = 4;               // k32 steps
  static constexpr int TILE = 128 * 128;     // bytes of one block of keys
  static constexpr int SCALES = 128 * 4;     // fp32 per-token scales
  static constexpr int WARPS = 4, NST = 1;   // 3 CTAs (12 warps) per SM
};
template <>
struct IdxTraits<FMT_BF16> {
  static constexpr int KS = 8;
  static constexpr int TILE = 128 * 256;     // two swizzled 128-byte halves
  static constexpr int SCALES = 0;
  static constexpr int WARPS = 4, NST = 1;
};
template <>
struct IdxTraits<FMT_NVFP4> {
  static constexpr int KS = 8;
  static constexpr int TILE = 128 * 64;      // packed e2m1
  static constexpr int SCALES = 128 * 8;     // e4m3 block scales
  static constexpr int WARPS = 4, NST = 2;   // 3 CTAs (12 warps) per SM
};

// Shared-memory layout of one CTA: per warp NST tiles, NST scale buffers,
// NST mbarriers and NST stage states; the tile region is 1024-byte aligned.
template <int FMT>
struct IdxLayout {
  using T = IdxTraits<FMT>;
  static constexpr int SC = T::SCALES > 16 ? T::SCALES : 16;
  static constexpr size_t SCAL = (size_t)T::WARPS * T::NST * T::TILE;
  static constexpr size_t BARS = SCAL + (size_t)T::WARPS * T::NST * SC;
  static constexpr size_t STATE = BARS + (size_t)T::WARPS * T::NST * 8;
  static constexpr size_t TOTAL = STATE + (size_t)T::WARPS * T::NST * 4;
  static constexpr size_t SMEM = TOTAL + 1024;  // alignment slack
};

enum : int { ST_SKIP = 0, ST_LOADED = 1, ST_BAD = 2 };

// Address of the 16-byte chunk `chunk` of row `row` in a 128-byte-row tile
// written by TMA with the 128-byte swizzle (1024-byte aligned base).
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int chunk) {
  return base + row * 128 + ((chunk ^ (row & 7)) << 4);
}

// m-tiles computed together: bounds the accumulator registers to 32 per lane
// while keeping enough independent MMA chains in flight.
template <int NT>
__host__ __device__ constexpr int m_group() {
  return NT >= 8 ? 1 : 8 / NT;
}

// Score one 128-key block held in shared memory: per lane, the running max
// over its rows of each of its columns (2 per 8-wide tile).
template <int FMT, int NT, int SP>
__device__ __forceinline__ void score_block(const uint8_t* tile, const uint8_t* scales,
                                            const uint32_t (&bq)[SP][NT][IdxTraits<FMT>::KS][2], int lane, int key0,
                                            const int (&lim)[NT][2], float (&cmax)[NT][2], bool nvr = false) {
  constexpr int KS = IdxTraits<FMT>::KS;
  constexpr int MG = m_group<NT>();
  const int g = lane >> 2, j = lane & 3;
  const uint32_t tb = smem_u32(tile);
#pragma unroll 1
  for (int m0 = 0; m0 < 8; m0 += MG) {
    float acc[MG][NT][4];
#pragma unroll
    for (int mi = 0; mi < MG; ++mi)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[mi][nt][0] = acc[mi][nt][1] = acc[mi][nt][2] = acc[mi][nt][3] = 0.f;
    if constexpr (FMT == FMT_FP8 || FMT == FMT_BF16) {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a[MG][4];
#pragma unroll
        for (int mi = 0; mi < MG; ++mi) {
          const int row = 16 * (m0 + mi) + (lane & 7) + ((lane >> 3) & 1) * 8;
          if constexpr (FMT == FMT_FP8)
            ldmatrix_x4(a[mi], swz(tb, row, 2 * ks + (lane >> 4)));
          else
            ldmatrix_x4(a[mi], swz(tb + (ks >> 2) * (128 * 128), row, 2 * (ks & 3) + (lane >> 4)));
        }
#pragma unroll
        for (int sp = 0; sp < SP; ++sp)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int mi = 0; mi < MG; ++mi) {
              if constexpr (FMT == FMT_FP8)
                mma_e4m3_k32(acc[mi][nt], a[mi], bq[sp][nt][ks][0], bq[sp][nt][ks][1]);
              else
                mma_bf16_k16(acc[mi][nt], a[mi], bq[0][nt][ks][0], bq[0][nt][ks][1]);
            }
      }
    } else {  // NVFP4: dequantize rows g and g+8 of each m-tile to f16 in registers
      uint32_t wa[MG][4], wb[MG][4], s0[MG][2], s1[MG][2];
#pragma unroll
      for (int mi = 0; mi < MG; ++mi) {
        const int r0 = 16 * (m0 + mi) + g, r1 = r0 + 8;
        const uint4 w0 = *reinterpret_cast<const uint4*>(tile + r0 * 64 + 16 * j);
        const uint4 w1 = *reinterpret_cast<const uint4*>(tile + r1 * 64 + 16 * j);
        wa[mi][0] = w0.x; wa[mi][1] = w0.y; wa[mi][2] = w0.z; wa[mi][3] = w0.w;
        wb[mi][0] = w1.x; wb[mi][1] = w1.y; wb[mi][2] = w1.z; wb[mi][3] = w1.w;
        const uint16_t sc0 = *reinterpret_cast<const uint16_t*>(scales + r0 * 8 + 2 * j);
        const uint16_t sc1 = *reinterpret_cast<const uint16_t*>(scales + r1 * 8 + 2 * j);
        uint32_t h;
        asm("{ .reg .b16 t; mov.b16 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h) : "h"(sc0));
        s0[mi][0] = (h & 0xffffu) | (h << 16);
        s0[mi][1] = (h >> 16) | (h & 0xffff0000u);
        asm("{ .reg .b16 t; mov.b16 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h) : "h"(sc1));
        s1[mi][0] = (h & 0xffffu) | (h << 16);
        s1[mi][1] = (h >> 16) | (h & 0xffff0000u);
      }
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        // bytes 2ks, 2ks+1 of the lane's 16 bytes hold dims 32j+4ks .. +3
        const int bi = 2 * ks;
        const int grp = bi >> 3;
#pragma unroll
        for (int mi = 0; mi < MG; ++mi) {
          uint32_t x0 = e2m1x2_to_f16x2((wa[mi][bi >> 2] >> (8 * (bi & 3))) & 0xffu);
          uint32_t x2 = e2m1x2_to_f16x2((wa[mi][bi >> 2] >> (8 * ((bi + 1) & 3))) & 0xffu);
          uint32_t x1 = e2m1x2_to_f16x2((wb[mi][bi >> 2] >> (8 * (bi & 3))) & 0xffu);
          uint32_t x3 = e2m1x2_to_f16x2((wb[mi][bi >> 2] >> (8 * ((bi + 1) & 3))) & 0xffu);
          uint32_t a[4];
          __half2 t;
          t = __hmul2(*reinterpret_cast<__half2*>(&x0), *reinterpret_cast<const __half2*>(&s0[mi][grp]));
          a[0] = *reinterpret_cast<uint32_t*>(&t);
          t = __hmul2(*reinterpret_cast<__half2*>(&x1), *reinterpret_cast<const __half2*>(&s1[mi][grp]));
          a[1] = *reinterpret_cast<uint32_t*>(&t);
          t = __hmul2(*reinterpret_cast<__half2*>(&x2), *reinterpret_cast<const __half2*>(&s0[mi][grp]));
          a[2] = *reinterpret_cast<uint32_t*>(&t);
          t = __hmul2(*reinterpret_cast<__half2*>(&x3), *reinterpret_cast<const __half2*>(&s1[mi][grp]));
          a[3] = *reinterpret_cast<uint32_t*>(&t);
          if (nvr) {  // the product rounded to E4M3, as the Blackwell NVFP4 -> FP8 dequant does
#pragma unroll
            for (int q = 0; q < 4; ++q) a[q] = e4m3_round_f16x2(a[q]);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_f16_k16(acc[mi][nt], a, bq[0][nt][ks][0], bq[0][nt][ks][1]);
        }
      }
    }
    // epilogue: rows r0 = 16m + g and r0 + 8 of each m-tile
#pragma unroll
    for (int mi = 0; mi < MG; ++mi) {
      const int r0 = 16 * (m0 + mi) + g, r1 = r0 + 8;
      float s0 = 1.f, s1 = 1.f;
      if constexpr (FMT == FMT_FP8) {
        s0 = reinterpret_cast<const float*>(scales)[r0];
        s1 = reinterpret_cast<const float*>(scales)[r1];
      }
      const int t0 = key0 + r0, t1 = key0 + r1;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const float v0 = (t0 <= lim[nt][c]) ? acc[mi][nt][c] * s0 : -INFINITY;
          const float v1 = (t1 <= lim[nt][c]) ? acc[mi][nt][2 + c] * s1 : -INFINITY;
          cmax[nt][c] = fmaxf(cmax[nt][c], fmaxf(v0, v1));
        }
    }
  }
}

// Blocks of sequence s that hold keys (0 for a sequence length outside
// [Q, max_blocks * 128], whose rows the kernel leaves at -inf).
__device__ __forceinline__ int seq_blocks(const BatchDev& bt, int s) {
  const int T = bt.seq_len(s);
  return (T < bt.Q || T > bt.max_nb * kBlock) ? 0 : (T + kBlock - 1) / kBlock;
}

// (s, b) of the unit `adv` units after (s, b) in the sequence-major order of
// all blocks that hold keys; s = S past the last one.
__device__ __forceinline__ void advance_unit(const BatchDev& bt, int& s, int& b, long adv) {
  long bb = b + adv;
  while (s < bt.S) {
    const int nb = seq_blocks(bt, s);
    if (bb < nb) break;
    bb -= nb;
    ++s;
  }
  b = (int)bb;
}

// (s, b) of unit v (v < total units), by the whole warp: 32 sequences a
// step, an inclusive scan of their block counts finds the one holding v.
__device__ __forceinline__ void locate_unit(const BatchDev& bt, long v, int lane, int& s_out, int& b_out) {
  long base = 0;
  s_out = bt.S;
  b_out = 0;
  for (int s0 = 0; s0 < bt.S; s0 += 32) {
    const int sl = s0 + lane;
    const int nb = (sl < bt.S) ? seq_blocks(bt, sl) : 0;
    long inc = nb;
    for (int o = 1; o < 32; o <<= 1) {
      const long y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const long total = __shfl_sync(0xffffffffu, inc, 31);
    if (v < base + total) {
      const unsigned hit = __ballot_sync(0xffffffffu, v < base + inc);
      const int l = __ffs(hit) - 1;
      const long before = __shfl_sync(0xffffffffu, inc - nb, l);
      s_out = s0 + l;
      b_out = (int)(v - base - before);
      return;
    }
    base += total;
  }
}

// Facts of one unit: (code, seq_len, s, b); code >= 0 physical block, -2 bad
// block-table entry (flag raised), -3 past the warp's last unit.
__device__ __forceinline__ int4 unit_facts(const IndexerParams& p, int s, int b, bool live) {
  const BatchDev& bt = p.batch;
  if (!live || s >= bt.S) return make_int4(-3, 0, 0, 0);
  const int T = bt.seq_len(s);
  const int phys = __ldg(bt.row(s) + b);
  if (phys < 0 || phys >= p.num_blocks) {
    raise_flag(p.status, FLAG_BAD_BLOCK, phys);
    return make_int4(-2, T, s, b);
  }
  return make_int4(phys, T, s, b);
}

template <int FMT, int NT, int SP>
__global__ void __launch_bounds__(IdxTraits<FMT>::WARPS * 32)
    indexer_kernel(const __grid_constant__ CUtensorMap tmap, const IndexerParams p) {
  using TR = IdxTraits<FMT>;
  using LY = IdxLayout<FMT>;
  constexpr int KS = TR::KS, NST = TR::NST, WARPS = TR::WARPS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* tiles = base + (size_t)warp * NST * TR::TILE;
  uint8_t* scal = base + LY::SCAL + (size_t)warp * NST * LY::SC;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + LY::BARS) + warp * NST;

  const BatchDev bt = p.batch;
  const int S = bt.S, Q = bt.Q, G = p.G;
  const long gw = (long)blockIdx.x * WARPS + warp;
  const long tw = (long)gridDim.x * WARPS;

  // Work: the blocks that hold keys, sequence-major, cut into one contiguous
  // run per warp of equal length (+-1) -- balanced whatever the sequence
  // lengths, and a warp's query fragments change only where its run crosses
  // into the next sequence.  Each warp counts the units itself.
  long V = 0;
  for (int s0 = 0; s0 < S; s0 += 32) {
    const int sl = s0 + lane;
    int nb = 0;
    if (sl < S) {
      nb = seq_blocks(bt, sl);
      if (nb == 0 && gw == 0) raise_flag(p.status, FLAG_BAD_SEQLEN, sl);
    }
    for (int o = 16; o > 0; o >>= 1) nb += __shfl_xor_sync(0xffffffffu, nb, o);
    V += nb;
  }
  const long v0 = gw * V / tw, v1 = (gw + 1) * V / tw;  // this warp's units [v0, v1)
  int ws, wb;  // (s, b) of unit v0 + it0 (the fact window's first unit)
  locate_unit(bt, v0, lane, ws, wb);

  if (lane == 0) {
    for (int st = 0; st < NST; ++st) mbar_init(&bars[st], 1);
    fence_mbar_init();
    if constexpr (FMT != FMT_NVFP4) prefetch_tmap(&tmap);
  }
  // unit facts for iterations [it0, it0 + 64): lane l holds it0 + l and it0 + 32 + l
  long it0 = 0;
  auto facts_at = [&](int s_, int b_, long first) -> int4 {
    int fs = s_, fb = b_;
    advance_unit(bt, fs, fb, lane);
    return unit_facts(p, fs, fb, v0 + first + lane < v1);
  };
  int4 inf0 = facts_at(ws, wb, 0);
  int ws1 = ws, wb1 = wb;
  advance_unit(bt, ws1, wb1, 32);
  int4 inf1 = facts_at(ws1, wb1, 32);
  __syncwarp();

  auto info_at = [&](long it) -> int4 {
    const int idx = (int)(it - it0);
    const int4 v = (idx < 32) ? inf0 : inf1;
    return make_int4(__shfl_sync(0xffffffffu, v.x, idx & 31), __shfl_sync(0xffffffffu, v.y, idx & 31),
                     __shfl_sync(0xffffffffu, v.z, idx & 31), __shfl_sync(0xffffffffu, v.w, idx & 31));
  };
  // copy the block of iteration `it` (facts `inf`) into stage st; lane 0 issues
  auto issue = [&](long it, int4 inf, int st) {
    if (lane == 0 && inf.x >= 0) {
      const int phys = inf.x;
      uint8_t* dst = tiles + (size_t)st * TR::TILE;
      fence_proxy_async();
      // the keys are read once: evict-first, so that they do not push the
      // block tables, scores and code of the kernels that follow out of L2
      const uint64_t pol = l2_policy_evict_first();
      if constexpr (FMT == FMT_FP8) {
        mbar_expect_tx(&bars[st], TR::TILE + TR::SCALES);
        tma_load_2d_hint(dst, &tmap, 0, phys * kBlock, &bars[st], pol);
        bulk_g2s_hint(scal + (size_t)st * LY::SC, p.idx_scale + (size_t)phys * kBlock, TR::SCALES, &bars[st], pol);
      } else if constexpr (FMT == FMT_BF16) {
        mbar_expect_tx(&bars[st], TR::TILE);
        tma_load_2d_hint(dst, &tmap, 0, phys * kBlock, &bars[st], pol);
        tma_load_2d_hint(dst + 128 * 128, &tmap, 64, phys * kBlock, &bars[st], pol);
      } else {
        mbar_expect_tx(&bars[st], TR::TILE + TR::SCALES);
        bulk_g2s_hint(dst, p.idx + (size_t)phys * TR::TILE, TR::TILE, &bars[st], pol);
        bulk_g2s_hint(scal + (size_t)st * LY::SC, p.idx_sf + (size_t)phys * TR::SCALES, TR::SCALES, &bars[st], pol);
      }
    }
  };

#pragma unroll
  for (int st = 0; st < NST; ++st) issue(st, info_at(st), st);

  uint32_t phase_bits = 0;
  int cur_s = -1;
  uint32_t bq[SP][NT][KS][2];
  float colf[NT][2];
  bool dead = false;

  for (long it = 0;; ++it) {
    if (it - it0 == 32) {  // slide the window of unit facts
      inf0 = inf1;
      it0 += 32;
      ws = ws1;
      wb = wb1;
      advance_unit(bt, ws1, wb1, 32);
      inf1 = facts_at(ws1, wb1, it0 + 32);
    }
    const int4 inf = info_at(it);
    if (inf.x == -3) break;
    const long u = v0 + it;
    // the kernels that follow may start their prologues once every warp is on
    // its last unit (they still wait for this grid to finish before reading P)
    if (u == v1 - 1) pdl_launch_dependents();
    const int st = (int)(it % NST);
    const int s = inf.z, b = inf.w;
    float* prow = p.pooled + (size_t)s * Q * G * bt.max_nb + b;
    if (inf.x >= 0 && !dead) {
      if (s != cur_s) {
        cur_s = s;
        // the query fragments come from the caller's index_q; a preceding kernel may still be writing it
        pdl_wait();
        long rows[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int col = nt * 8 + (lane >> 2);
          rows[nt] = (col < Q * G) ? ((long)s * Q * G + col) * kDim : -1;
        }
        build_qfrag<FMT, NT, SP, KS>(p.index_q, p.iq_fp8, rows, p.iq_scale, p.col_const, bq, colf, lane);
      }
      const int T = inf.y;
      int lim[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col = nt * 8 + 2 * (lane & 3) + c;
          lim[nt][c] = (col < Q * G) ? (T - Q + col / G) : -1;
        }
      const bool ok = mbar_wait_warp(&bars[st], (phase_bits >> st) & 1u);
      phase_bits ^= 1u << st;
      if (!ok) {
        if (lane == 0) raise_flag(p.status, FLAG_TIMEOUT, (int)u);
        dead = true;
      } else {
        float cmax[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) cmax[nt][0] = cmax[nt][1] = -INFINITY;
        score_block<FMT, NT, SP>(tiles + (size_t)st * TR::TILE, scal + (size_t)st * LY::SC, bq, lane, b * kBlock,
                                 lim, cmax, p.nv_round != 0);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float v = cmax[nt][c];
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
            const int col = nt * 8 + 2 * (lane & 3) + c;
            if (lane < 4 && col < Q * G) prow[(size_t)col * bt.max_nb] = v * colf[nt][c];
          }
      }
    }
    if (inf.x < 0 || dead) {
      for (int col = lane; col < Q * G; col += 32) prow[(size_t)col * bt.max_nb] = -INFINITY;
    }
    __syncwarp();
    if (!dead) issue(it + NST, info_at(it + NST), st);
  }
  // blocks that hold no key of a sequence (past its length, or all of a bad
  // sequence): -inf for every (query, group) row, spread over all threads
  {
    const long slots = (long)S * bt.max_nb;
    for (long e = gw * 32 + lane; e < slots; e += tw * 32) {
      const int s = (int)(e / bt.max_nb), b = (int)(e % bt.max_nb);
      if (b < seq_blocks(bt, s)) continue;
      float* prow = p.pooled + (size_t)s * Q * G * bt.max_nb + b;
      for (int col = 0; col < Q * G; ++col) prow[(size_t)col * bt.max_nb] = -INFINITY;
    }
  }
  pdl_launch_dependents();
  // a warp that gave up waits (bounded) for copies still in flight before exiting
  if (dead) {
    for (int st = 0; st < NST; ++st) mbar_wait(&bars[st], (phase_bits >> st) & 1u, 2000);
  }
}

template <int FMT, int NT, int SP>
cudaError_t launch_one(const CUtensorMap* tmap, const IndexerParams& p, int num_sms, cudaStream_t st, bool pdl) {
  using TR = IdxTraits<FMT>;
  const size_t smem = IdxLayout<FMT>::SMEM;
  auto kern = indexer_kernel<FMT, NT, SP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, TR::WARPS * 32, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const long units = (long)p.batch.S * p.batch.max_nb;
  long grid = (long)num_sms * per_sm;
  const long need = (units + TR::WARPS - 1) / TR::WARPS;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(TR::WARPS * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  CUtensorMap dummy = {};
  return cudaLaunchKernelEx(&cfg, kern, tmap ? *tmap : dummy, p);
}

template <int FMT>
cudaError_t launch_fmt(const CUtensorMap* tmap, const IndexerParams& p, int num_sms, cudaStream_t st, bool pdl) {
  const int nt = p.geom.nt, sp = p.geom.sp;
  if (sp == 2) {
    if constexpr (FMT == FMT_FP8) {
      switch (nt) {
        case 1: return launch_one<FMT, 1, 2>(tmap, p, num_sms, st, pdl);
        case 2: return launch_one<FMT, 2, 2>(tmap, p, num_sms, st, pdl);
        case 4: return launch_one<FMT, 4, 2>(tmap, p, num_sms, st, pdl);
        default: return cudaErrorInvalidValue;
      }
    }
    return cudaErrorInvalidValue;
  }
  switch (nt) {
    case 1: return launch_one<FMT, 1, 1>(tmap, p, num_sms, st, pdl);
    case 2: return launch_one<FMT, 2, 1>(tmap, p, num_sms, st, pdl);
    case 4: return launch_one<FMT, 4, 1>(tmap, p, num_sms, st, pdl);
    case 8: return launch_one<FMT, 8, 1>(tmap, p, num_sms, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_indexer(int fmt, const CUtensorMap* tmap, const IndexerParams& p, int num_sms, cudaStream_t st,
                           bool pdl) {
  switch (fmt) {
    case FMT_FP8: return launch_fmt<FMT_FP8>(tmap, p, num_sms, st, pdl);
    case FMT_BF16: return launch_fmt<FMT_BF16>(tmap, p, num_sms, st, pdl);
    case FMT_NVFP4: return launch_fmt<FMT_NVFP4>(tmap, p, num_sms, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace msa
