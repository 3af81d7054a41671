// Sparse attend over the selected blocks (split-K flash decoding) and the
// split combine.
//
// Definition (vLLM Day-0 blog, section "MSA 入门" and Figure 1): every query
// head of a GQA group attends, with exact softmax, to the keys of the blocks
// its group selected, at most k x 128 keys; logits are scaled by
// head_dim ** -0.5 (model page, MiniMaxM3SparseAttention: self.scaling).  With
// several new tokens per sequence (speculative verify, prefill chunks) each
// token has its own selection and causal limit.
//
// Work.  Item = (sequence, group, split): the group's selected blocks (for
// several query tokens: the union of their selections) cut into splits of
// `bps` blocks.  The kernel is persistent: a grid of as many CTAs as fit on
// the GPU walks the items with a static stride.  In each CTA one producer
// warp reads the items' facts (block ids, query masks, physical blocks; the
// counts of 32 items at once, so that empty splits cost nothing), publishes
// them in one of two item slots together with a bulk copy of the query
// fragments the preceding kernel prepared, and streams every block through a
// ring of shared-memory stages (TMA tensor copies with the 128-byte swizzle
// for FP8 / BF16, bulk copies for NVFP4), gated by per-stage full / empty
// mbarriers.  Four consumer warps own keys [32w, 32w+32) of every block, each
// with its own online softmax; at the end of an item they merge through a
// dedicated shared-memory area (named barriers among the consumers only), so
// the next item's copies keep streaming meanwhile.  A (sequence, group) that
// fits one split writes its bf16 output and LSE directly; otherwise each split
// writes a partial (o, m, l), and the CTA whose split finishes that
// (sequence, group) last (an acquire-release atomic count) merges all of its
// partials by log-sum-exp (merge_splits).  Every wait is bounded; a wait that
// gives up raises the timeout flag and the CTA winds down without further
// copies.
//
// Tensor-core mapping, keys as MMA rows (the query side is only Q x r <= 32
// columns wide):
//   logits^T[key][col] = K[key][:] . Q[col][:]        (A = K tile, B = query)
//   O^T[d][col]        = sum_key V[key][d] P[key][col] (A = V^T, B = P)
// FP8 tiles go to mma.sync e4m3 k32 unconverted.  V^T is built in registers
// with byte permutes from 16-byte shared-memory reads laid out so that the
// swizzled tile is read without bank conflicts.  A bf16 query or the fp32
// probabilities enter as two e4m3 terms (hi + lo) with a power-of-two scale,
// one MMA per term.  BF16 tiles use bf16 k16 MMAs with ldmatrix (.trans for
// V^T); NVFP4 tiles are dequantized exactly to f16 (K in registers, V through a
// per-warp swizzled shared-memory tile) for f16 k16 MMAs.
#include "msa_device.cuh"
#include "msa_internal.h"
#include "msa_qfrag.cuh"

namespace msa {

namespace {

constexpr int kWarps = 4;                 // consumer warps
constexpr int kThreads = 32 * (kWarps + 1);  // + the producer warp
constexpr int kConsumers = 32 * kWarps;
constexpr int kMaxBps = kMaxBlocksPerSplit;  // blocks per split at most
constexpr int kMergeRow = 132;  // padded row of the merge area (conflict-free stores)

// What the producer publishes for one item.
struct ItemFacts {
  int32_t sg, split, n, count;  // n = -1: no more items
  int32_t empty_sg, pad[3];
  int32_t sb[kMaxBps];          // block ids (-1: rejected)
  uint32_t smask[kMaxBps];      // query tokens that selected each block
  int32_t sok[kMaxBps];         // 1: the block was copied
};

template <int FMT>
struct AttTraits;
template <>
struct AttTraits<FMT_FP8> {
  static constexpr int KTILE = 128 * 128, VTILE = 128 * 128, KSC = 512, VSC = 512;
  static constexpr int QKS = 4;
};
template <>
struct AttTraits<FMT_BF16> {
  static constexpr int KTILE = 128 * 256, VTILE = 128 * 256, KSC = 0, VSC = 0;
  static constexpr int QKS = 8;
};
template <>
struct AttTraits<FMT_NVFP4> {
  static constexpr int KTILE = 128 * 64, VTILE = 128 * 64, KSC = 1024, VSC = 1024;
  static constexpr int QKS = 8;
};

__host__ __device__ constexpr size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <int FMT, int NT, int SP, int NSTAGES>
struct AttLayoutN {
  using T = AttTraits<FMT>;
  static constexpr int NC = NT * 8;
  static constexpr int NST = NSTAGES;
  static constexpr size_t TILES = (size_t)T::KTILE + T::VTILE + T::KSC + T::VSC;
  static constexpr size_t STAGE = round_up(TILES, 1024);
  static constexpr size_t FRAGW = (size_t)SP * NT * T::QKS * 64 * 4;  // query fragment words
  static constexpr size_t FRAG = FRAGW + NC * 4;                      // + column factors
  static constexpr size_t ISLOT = round_up(FRAG, 128);
  static constexpr size_t ITEM_OFF = STAGE * NST;                     // two item slots
  static constexpr size_t PSM = ITEM_OFF + 2 * ISLOT;                 // per-warp P tiles
  static constexpr size_t PSM_WARP = 64 * NC;
  static constexpr size_t VDQ = PSM + kWarps * PSM_WARP;              // NVFP4 V^T f16 tiles
  static constexpr size_t VDQ_WARP = (FMT == FMT_NVFP4) ? 32 * 256 : 0;  // x 4 warps: one 128-row f16 V tile
  static constexpr int KG = kWarps / NT;                              // warps sharing a column tile
  static constexpr size_t MERGE = round_up(VDQ + kWarps * VDQ_WARP, 16);  // KG > 1: the warps' o, m, l
  static constexpr size_t MERGE_BYTES = (KG > 1) ? (size_t)kWarps * 8 * (kMergeRow + 2) * 4 : 0;
  static constexpr size_t FACTS = round_up(MERGE + MERGE_BYTES + 16, 16);
  static constexpr size_t BARS = round_up(FACTS + 2 * sizeof(ItemFacts), 16);
  static constexpr size_t TOTAL = BARS + 8 * (2 * NST + 4) + 16;
  static constexpr size_t SMEM = TOTAL + 1024;
};

// Ring depth: three stages where two CTAs still fit on an SM (228 KB of
// shared memory, 1 KB of it reserved per CTA), else two.
template <int FMT, int NT, int SP>
constexpr int ring_stages() {
  return 2 * (AttLayoutN<FMT, NT, SP, 3>::SMEM + 1024) <= 228 * 1024 ? 3 : 2;
}
template <int FMT, int NT, int SP>
using AttLayout = AttLayoutN<FMT, NT, SP, ring_stages<FMT, NT, SP>()>;

__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int chunk) {
  return base + row * 128 + ((chunk ^ (row & 7)) << 4);
}

// 4x4 byte transpose: out[e] byte i = in[i] byte e.
__device__ __forceinline__ void transpose4x4(const uint32_t in[4], uint32_t out[4]) {
  const uint32_t t0 = __byte_perm(in[0], in[1], 0x5140);
  const uint32_t t1 = __byte_perm(in[0], in[1], 0x7362);
  const uint32_t t2 = __byte_perm(in[2], in[3], 0x5140);
  const uint32_t t3 = __byte_perm(in[2], in[3], 0x7362);
  out[0] = __byte_perm(t0, t2, 0x5410);
  out[1] = __byte_perm(t0, t2, 0x7632);
  out[2] = __byte_perm(t1, t3, 0x5410);
  out[3] = __byte_perm(t1, t3, 0x7632);
}

// 2^x by the hardware approximation (relative error about 2^-22; -inf -> 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// col / r for the small counts here (col < 4096, 1 <= r <= 64): the float
// quotient of col + 1/2 lies at least 1/(2r) from an integer, far beyond its
// rounding error, so the truncation is exact.
__device__ __forceinline__ int col_div(int col, int r) {
  return (int)(((float)col + 0.5f) * __frcp_rn((float)r));
}

// Phases of attend_block: 1 logits, 2 softmax, 4 P tile, 8 O^T += V^T P.
// A real block runs all of them; the dry run before the grid-dependency wait
// gives each consumer warp one phase, so the four warps fetch the four parts
// of the instruction path at the same time instead of one after the other.
constexpr unsigned kAllPhases = 15u;

// One block of keys for one consumer warp.  The four consumer warps split the
// work as NT column tiles x (4 / NT) key ranges: warp w takes column tile
// ct = w / (4 / NT) (8 query x head columns) and the KW = 32 * NT keys
// starting at kw.  Logits for its keys, masked online softmax, P into its
// shared tile, O^T += V^T P for its columns.
template <int FMT, int NT, int SP>
__device__ __forceinline__ void attend_block(const uint8_t* stg, uint8_t* psm, uint8_t* vdq,
                                             const uint32_t* __restrict__ fr, int ct, const float (&colf)[2],
                                             const int (&qlim)[2], const int (&qbit)[2], uint32_t qmask, int key0,
                                             int kw, int warp, int lane, float (&m_run)[2], float (&l_run)[2],
                                             float (&o)[8][4], int& e_prev, unsigned phases = kAllPhases,
                                             bool nvr = false) {
  using TR = AttTraits<FMT>;
  constexpr int MT = 2 * NT;  // m tiles of 16 keys
  constexpr int KW = 16 * MT; // keys of this warp
  const int g8 = lane >> 2, j = lane & 3;
  // query fragment word (term sp, k step ks, register rg) of this lane for column
  // tile ct, read from the item's shared copy where it is used
#define QF(sp, ks, rg) fr[((((sp) * NT + ct) * TR::QKS + (ks)) * 2 + (rg)) * 32 + lane]
  // ---------------- logits^T for this warp's keys
  float sacc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) sacc[mt][0] = sacc[mt][1] = sacc[mt][2] = sacc[mt][3] = 0.f;
  const uint32_t kt = smem_u32(stg);
  if (phases & 1u) {
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    if constexpr (FMT == FMT_FP8 || FMT == FMT_BF16) {
      const int row = kw + 16 * mt + (lane & 7) + ((lane >> 3) & 1) * 8;
      // two accumulators per m tile (the query's hi and lo terms, or alternate
      // k steps), summed at the end: MMA chains half as long
      float sacc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < TR::QKS; ++ks) {
        uint32_t a[4];
        if constexpr (FMT == FMT_FP8) {
          ldmatrix_x4(a, swz(kt, row, 2 * ks + (lane >> 4)));
          if constexpr (SP == 2) {
            mma_e4m3_k32(sacc[mt], a, QF(0, ks, 0), QF(0, ks, 1));
            mma_e4m3_k32(sacc2, a, QF(1, ks, 0), QF(1, ks, 1));
          } else {
            mma_e4m3_k32((ks & 1) ? sacc2 : sacc[mt], a, QF(0, ks, 0), QF(0, ks, 1));
          }
        } else {
          ldmatrix_x4(a, swz(kt + (ks >> 2) * (128 * 128), row, 2 * (ks & 3) + (lane >> 4)));
          mma_bf16_k16((ks & 1) ? sacc2 : sacc[mt], a, QF(0, ks, 0), QF(0, ks, 1));
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[mt][e] += sacc2[e];
    } else {
      const int r0 = kw + 16 * mt + g8, r1 = r0 + 8;
      const uint8_t* ksf = stg + TR::KTILE + TR::VTILE;
      const uint4 w0 = *reinterpret_cast<const uint4*>(stg + r0 * 64 + 16 * j);
      const uint4 w1 = *reinterpret_cast<const uint4*>(stg + r1 * 64 + 16 * j);
      const uint16_t sc0 = *reinterpret_cast<const uint16_t*>(ksf + r0 * 8 + 2 * j);
      const uint16_t sc1 = *reinterpret_cast<const uint16_t*>(ksf + r1 * 8 + 2 * j);
      uint32_t s0[2], s1[2], h;
      asm("{ .reg .b16 t; mov.b16 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h) : "h"(sc0));
      s0[0] = (h & 0xffffu) | (h << 16);
      s0[1] = (h >> 16) | (h & 0xffff0000u);
      asm("{ .reg .b16 t; mov.b16 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h) : "h"(sc1));
      s1[0] = (h & 0xffffu) | (h << 16);
      s1[1] = (h >> 16) | (h & 0xffff0000u);
      const uint32_t wa[4] = {w0.x, w0.y, w0.z, w0.w};
      const uint32_t wb[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int ks = 0; ks < TR::QKS; ++ks) {
        const int bi = 2 * ks;
        const int grp = bi >> 3;
        uint32_t x0 = e2m1x2_to_f16x2((wa[bi >> 2] >> (8 * (bi & 3))) & 0xffu);
        uint32_t x2 = e2m1x2_to_f16x2((wa[bi >> 2] >> (8 * ((bi + 1) & 3))) & 0xffu);
        uint32_t x1 = e2m1x2_to_f16x2((wb[bi >> 2] >> (8 * (bi & 3))) & 0xffu);
        uint32_t x3 = e2m1x2_to_f16x2((wb[bi >> 2] >> (8 * ((bi + 1) & 3))) & 0xffu);
        uint32_t a[4];
        __half2 t;
        t = __hmul2(*reinterpret_cast<__half2*>(&x0), *reinterpret_cast<const __half2*>(&s0[grp]));
        a[0] = *reinterpret_cast<uint32_t*>(&t);
        t = __hmul2(*reinterpret_cast<__half2*>(&x1), *reinterpret_cast<const __half2*>(&s1[grp]));
        a[1] = *reinterpret_cast<uint32_t*>(&t);
        t = __hmul2(*reinterpret_cast<__half2*>(&x2), *reinterpret_cast<const __half2*>(&s0[grp]));
        a[2] = *reinterpret_cast<uint32_t*>(&t);
        t = __hmul2(*reinterpret_cast<__half2*>(&x3), *reinterpret_cast<const __half2*>(&s1[grp]));
        a[3] = *reinterpret_cast<uint32_t*>(&t);
        if (nvr) {  // the product rounded to E4M3, as the Blackwell NVFP4 -> FP8 dequant does
#pragma unroll
          for (int q = 0; q < 4; ++q) a[q] = e4m3_round_f16x2(a[q]);
        }
        mma_f16_k16(sacc[mt], a, QF(0, ks, 0), QF(0, ks, 1));
      }
    }
  }
  }

  // ---------------- scale, mask, online softmax (per column, over this warp's keys)
  float alpha[2] = {0.f, 0.f};
  if (phases & 2u) {
  float ksc[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float v = 1.f;
      if constexpr (FMT == FMT_FP8)
        v = reinterpret_cast<const float*>(stg + TR::KTILE + TR::VTILE)[kw + 16 * mt + g8 + 8 * hh];
      ksc[mt][hh] = v;
    }
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const bool sel = (qmask >> qbit[c]) & 1u;
    float bmax = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int key = key0 + 16 * mt + g8 + 8 * hh;
        const bool vis = sel && key <= qlim[c];
        const float x = vis ? sacc[mt][c + 2 * hh] * ksc[mt][hh] * colf[c] : -INFINITY;
        sacc[mt][c + 2 * hh] = x;
        bmax = fmaxf(bmax, x);
      }
    bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 4));
    bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 8));
    bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 16));
    const float mnew = fmaxf(m_run[c], bmax);
    const float msub = (mnew == -INFINITY) ? 0.f : mnew;
    alpha[c] = ex2(m_run[c] - msub);
    float psum = 0.f;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float pv = ex2(sacc[mt][c + 2 * hh] - msub);
        sacc[mt][c + 2 * hh] = pv;
        psum += pv;
      }
    // per-lane partial row sum (this lane's keys); the 8 lanes of a column
    // add theirs up once, at the merge
    l_run[c] = l_run[c] * alpha[c] + psum;
    m_run[c] = mnew;
  }
  }

  // ---------------- P operand into this warp's shared tile
  __syncwarp();
  if (phases & 4u) {
  if constexpr (FMT == FMT_FP8) {
    // P' = p * vscale * 2^e, split into e4m3 hi + lo; tile [term][column][KW bytes]
    const float* vsc = reinterpret_cast<const float*>(stg + TR::KTILE + TR::VTILE + TR::KSC);
    float vmax = vsc[kw + lane];
#pragma unroll
    for (int i = 1; i < NT; ++i) vmax = fmaxf(vmax, vsc[kw + 32 * i + lane]);
    for (int off = 16; off > 0; off >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
    const int e = min(126, fit448(vmax));
    const float fe = (e >= -126) ? pow2i(e) : ldexpf(1.f, e);
    const int de = e - e_prev;
    const float resc = (de >= -126 && de <= 127) ? pow2i(de) : ldexpf(1.f, de);
    e_prev = e;
    // within each 32-key step, this lane's keys 16mt' + g8 + 8hh (mt' = 0, 1) sit in
    // bytes 2mt' + hh of word g8 of the column's row (keys j + 8i: bytes of b0,
    // keys 4 + j + 8i: bytes of b1, for lane j)
    uint32_t* psm32 = reinterpret_cast<uint32_t*>(psm);
#pragma unroll
    for (int ks = 0; ks < NT; ++ks) {
      float vs[2][2];
#pragma unroll
      for (int m2 = 0; m2 < 2; ++m2)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) vs[m2][hh] = vsc[kw + 32 * ks + 16 * m2 + g8 + 8 * hh] * fe;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t hw = 0, lw = 0;
#pragma unroll
        for (int m2 = 0; m2 < 2; ++m2) {
          const float x0 = sacc[2 * ks + m2][c] * vs[m2][0];
          const float x1 = sacc[2 * ks + m2][c + 2] * vs[m2][1];
          const uint16_t h = pack_e4m3x2(x0, x1);
          const float2 hv = e4m3x2_to_float2(h);
          const uint16_t l = pack_e4m3x2(x0 - hv.x, x1 - hv.y);
          hw |= (uint32_t)h << (16 * m2);
          lw |= (uint32_t)l << (16 * m2);
        }
        const int col = 2 * j + c;
        psm32[col * (KW / 4) + 8 * ks + g8] = hw;
        psm32[8 * (KW / 4) + col * (KW / 4) + 8 * ks + g8] = lw;
      }
    }
    // rescale the running output: softmax shift and the change of P scale
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const float f = alpha[c] * resc;
#pragma unroll
      for (int mm = 0; mm < 8; ++mm) {
        o[mm][c] *= f;
        o[mm][c + 2] *= f;
      }
    }
  } else {
    // P as one 16-bit term: bf16 for BF16 tiles, f16 for NVFP4 tiles; tile [column][KW]
    uint16_t* ps16 = reinterpret_cast<uint16_t*>(psm);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int kk = 16 * mt + g8 + 8 * hh;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col = 2 * j + c;
          const float pv = sacc[mt][c + 2 * hh];
          uint16_t bits;
          if constexpr (FMT == FMT_BF16) {
            __nv_bfloat16 x = __float2bfloat16_rn(pv);
            bits = *reinterpret_cast<uint16_t*>(&x);
          } else {
            __half x = __float2half_rn(pv);
            bits = *reinterpret_cast<uint16_t*>(&x);
          }
          ps16[col * KW + kk] = bits;
        }
      }
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int mm = 0; mm < 8; ++mm) {
        o[mm][c] *= alpha[c];
        o[mm][c + 2] *= alpha[c];
      }
    if constexpr (FMT == FMT_NVFP4) {
      // dequantize V rows 32w .. 32w+31 to f16 (exact) into the CTA's swizzled tile
      const uint8_t* vraw = stg + TR::KTILE;
      const uint8_t* vsf = stg + TR::KTILE + TR::VTILE + TR::KSC;
      const int key = 32 * warp + lane;
      const uint32_t vb = smem_u32(vdq);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint4 w = *reinterpret_cast<const uint4*>(vraw + key * 64 + 16 * q4);
        const uint16_t scp = *reinterpret_cast<const uint16_t*>(vsf + key * 8 + 2 * q4);
        uint32_t hsc;
        asm("{ .reg .b16 t; mov.b16 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(hsc) : "h"(scp));
        const uint32_t sA = (hsc & 0xffffu) | (hsc << 16), sB = (hsc >> 16) | (hsc & 0xffff0000u);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
        uint32_t out[16];
#pragma unroll
        for (int bi = 0; bi < 16; ++bi) {
          uint32_t x = e2m1x2_to_f16x2((ww[bi >> 2] >> (8 * (bi & 3))) & 0xffu);
          __half2 t = __hmul2(*reinterpret_cast<__half2*>(&x), *reinterpret_cast<const __half2*>(bi < 8 ? &sA : &sB));
          out[bi] = *reinterpret_cast<uint32_t*>(&t);
          if (nvr) out[bi] = e4m3_round_f16x2(out[bi]);
        }
        // 32 dims = d 32*q4 .. +31 -> f16 bytes 64*q4 .. +63 -> half (q4>>1), chunks 4*(q4&1) .. +3
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint32_t addr = swz(vb + (q4 >> 1) * (128 * 128), key, 4 * (q4 & 1) + cc);
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(out[4 * cc]), "r"(out[4 * cc + 1]),
                       "r"(out[4 * cc + 2]), "r"(out[4 * cc + 3]));
        }
      }
      if constexpr (NT > 1) {
        if (phases == kAllPhases) named_bar_sync(2, kConsumers);  // other warps' rows are read below
      }
    }
  }
  }
  __syncwarp();

  // ---------------- O^T += V^T P
  if (phases & 8u) {
  if constexpr (FMT == FMT_FP8) {
    const uint32_t vt = smem_u32(stg + TR::KTILE);
    const int cg = (g8 >> 1) | ((g8 & 1) << 2);  // this lane's 16-dim chunk
#pragma unroll
    for (int ks = 0; ks < NT; ++ks) {
      uint32_t bp[2][2];
#pragma unroll
      for (int sp = 0; sp < 2; ++sp) {
        const uint8_t* row = psm + sp * 8 * KW + g8 * KW + 32 * ks;
        bp[sp][0] = *reinterpret_cast<const uint32_t*>(row + 4 * j);
        bp[sp][1] = *reinterpret_cast<const uint32_t*>(row + 16 + 4 * j);
      }
      uint32_t A0[16], A2[16];
#pragma unroll
      for (int set = 0; set < 2; ++set) {
        uint4 raw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int key = kw + 32 * ks + 8 * i + 4 * set + j;
          const uint32_t addr = swz(vt, key, cg);
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(raw[i].x), "=r"(raw[i].y), "=r"(raw[i].z), "=r"(raw[i].w)
                       : "r"(addr));
        }
        uint32_t* A = set ? A2 : A0;
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
          uint32_t in[4], out[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            in[i] = (wd == 0) ? raw[i].x : (wd == 1) ? raw[i].y : (wd == 2) ? raw[i].z : raw[i].w;
          transpose4x4(in, out);
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) A[4 * wd + e2] = out[e2];
        }
      }
#pragma unroll
      for (int mm = 0; mm < 8; ++mm) {
        const uint32_t a[4] = {A0[2 * mm], A0[2 * mm + 1], A2[2 * mm], A2[2 * mm + 1]};
        mma_e4m3_k32(o[mm], a, bp[0][0], bp[0][1]);
        mma_e4m3_k32(o[mm], a, bp[1][0], bp[1][1]);
      }
    }
  } else {
    const uint16_t* ps16 = reinterpret_cast<const uint16_t*>(psm);
    const uint32_t vt = (FMT == FMT_BF16) ? smem_u32(stg + TR::KTILE) : smem_u32(vdq);
#pragma unroll
    for (int kk = 0; kk < KW / 16; ++kk) {
      const uint16_t* row = ps16 + g8 * KW + 16 * kk;
      const uint32_t bp0 = *reinterpret_cast<const uint32_t*>(row + 2 * j);
      const uint32_t bp1 = *reinterpret_cast<const uint32_t*>(row + 8 + 2 * j);
      const int key = kw + 16 * kk + (lane & 7) + 8 * ((lane >> 4) & 1);
#pragma unroll
      for (int mm = 0; mm < 8; ++mm) {
        const int d0 = 16 * mm + 8 * ((lane >> 3) & 1);
        uint32_t a[4];
        ldmatrix_x4_trans(a, swz(vt + (d0 >> 6) * (128 * 128), key, (d0 & 63) >> 3));
        if constexpr (FMT == FMT_BF16)
          mma_bf16_k16(o[mm], a, bp0, bp1);
        else
          mma_f16_k16(o[mm], a, bp0, bp1);
      }
    }
    if constexpr (FMT == FMT_NVFP4 && NT > 1) {
      if (phases == kAllPhases) named_bar_sync(2, kConsumers);  // before the tile is rewritten
    }
  }
  }
  __syncwarp();
}

#undef QF

__device__ __forceinline__ bool cta_dead(const int* flag) { return *reinterpret_cast<const volatile int*>(flag) != 0; }

__device__ __forceinline__ void set_dead(int* flag, DeviceStatus* st, int detail) {
  if (!cta_dead(flag)) raise_flag(st, FLAG_TIMEOUT, detail);
  *reinterpret_cast<volatile int*>(flag) = 1;
}

// Bounded warp-uniform wait that gives up at once when the CTA is winding down.
__device__ __forceinline__ bool ring_wait(uint64_t* bar, uint32_t parity, const int* dead) {
  if (cta_dead(dead)) return false;
  return mbar_wait_warp(bar, parity);
}

__device__ __noinline__ void merge_splits(const AttendParams& p, int sg, int nparts, int tid, bool write);

template <int FMT, int NT, int SP>
__device__ __forceinline__ void attend_producer(const CUtensorMap* tmk, const CUtensorMap* tmv, const AttendParams& p,
                                                uint8_t* base, uint64_t* full, uint64_t* empty, uint64_t* ifull,
                                                uint64_t* iempty, int* dead, ItemFacts* facts, int lane) {
  using TR = AttTraits<FMT>;
  using LY = AttLayout<FMT, NT, SP>;
  constexpr int NC = NT * 8;
  constexpr int NST = LY::NST;
  const BatchDev bt = p.batch;
  const int G = p.G;
  const int items = bt.S * G * p.splits;  // 32-bit: no 64-bit divisions below
  const int stride = gridDim.x;
  int bi = 0;  // blocks pushed through the ring
  int ii = 0;  // items published
  bool ok = true;
  bool waited = false;
#pragma unroll 1
  for (int it0 = blockIdx.x; it0 < items && ok; it0 += 32 * stride) {
    // selected-block counts of the next 32 items of this CTA, one per lane.  One
    // query token: the top-k keeps min(k, visible blocks) blocks, known from the
    // sequence length alone (a caller input, readable before the wait).
    const int my_it = it0 + lane * stride;
    int my_cnt = 0;
    if (p.direct && my_it < items) {
      const int T = bt.seq_len(my_it / p.splits / G);
      my_cnt = (T < 1 || T > bt.max_nb * kBlock) ? 0 : min(p.topk, (T - 1) / kBlock + 1);
    }
    if (!waited && my_it < items) {
      // the block-table row of this lane's item into L2 (caller input, readable now):
      // the physical-block lookups after the wait then hit
      const int32_t* rowp = bt.row(my_it / p.splits / G);
      for (int e = 0; e < bt.max_nb && e < 64 * 32; e += 32)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(rowp + e));
    }
    if (!waited) {
      // meanwhile the consumers fetch the block code; fetch the split merge's
      // (a pass over the first split's partials of the previous call, nothing written)
      merge_splits(p, 0, 1, lane, false);
      pdl_wait();  // the selection / union and the query fragments come from the preceding kernel
      waited = true;
    }
    if (!p.direct && my_it < items) my_cnt = p.u_count[my_it / p.splits];
#pragma unroll 1
    for (int t = 0; t < 32 && ok; ++t) {
      const int it = it0 + t * stride;
      if (it >= items) break;
      const int count = __shfl_sync(0xffffffffu, my_cnt, t);
      const int sg = it / p.splits, split = it - sg * p.splits;
      const int kb0 = split * p.bps;
      const int n = max(0, min(p.bps, count - kb0));
      const bool empty_sg = count <= 0;
      if (n == 0 && !(empty_sg && split == 0)) continue;  // nothing in this split
      const int s = sg / G, g = sg % G;
      const int T = bt.seq_len(s);
      int b = -1, phys = -1;
      uint32_t mask = 0;
      if (lane < n) {
        if (p.direct) {
          b = p.topk_idx[(size_t)sg * p.topk + kb0 + lane];
          mask = 1u;
        } else {
          b = p.u_ids[(size_t)sg * p.cap + kb0 + lane];
          mask = p.u_mask[(size_t)sg * p.cap + kb0 + lane];
        }
        if (b < 0 || T < 0 || b > (T - 1) / kBlock) {
          raise_flag(p.status, FLAG_BAD_SELECT, b);
          b = -1;
        } else {
          const int ph = bt.row(s)[b];
          if (ph < 0 || ph >= p.num_blocks) raise_flag(p.status, FLAG_BAD_BLOCK, ph);
          else phys = ph;
        }
      }
      // publish the item
      const int slot = (int)(ii & 1);
      const int use = ii >> 1;
      if (use > 0 && !ring_wait(&iempty[slot], (uint32_t)((use - 1) & 1), dead)) {
        set_dead(dead, p.status, (int)it);
        ok = false;
        break;
      }
      ItemFacts& f = facts[slot];
      if (lane < n) {
        f.sb[lane] = b;
        f.smask[lane] = mask;
        f.sok[lane] = phys >= 0 ? 1 : 0;
      }
      if (lane == 0) {
        f.sg = sg;
        f.split = split;
        f.n = n;
        f.count = count;
        f.empty_sg = empty_sg ? 1 : 0;
      }
      __syncwarp();
      if (lane == 0) {
        if (n > 0) {
          uint8_t* fd = base + LY::ITEM_OFF + (size_t)slot * LY::ISLOT;
          fence_proxy_async();
          mbar_expect_tx(&ifull[slot], (uint32_t)LY::FRAG);
          bulk_g2s(fd, p.frag + (size_t)sg * (LY::FRAGW / 4), (uint32_t)LY::FRAGW, &ifull[slot]);
          bulk_g2s(fd + LY::FRAGW, p.colf + (size_t)sg * NC, NC * 4, &ifull[slot]);
        } else {
          mbar_arrive(&ifull[slot]);
        }
      }
      ++ii;
      // its blocks, through the ring
#pragma unroll 1
      for (int k = 0; k < n; ++k) {
        const int ph = __shfl_sync(0xffffffffu, phys, k);
        const int st = (int)(bi % NST);
        const int ub = bi / NST;
        if (ub > 0 && !ring_wait(&empty[st], (uint32_t)((ub - 1) & 1), dead)) {
          set_dead(dead, p.status, (int)it);
          ok = false;
          break;
        }
        if (lane == 0) {
          if (ph >= 0) {
            uint8_t* stg = base + (size_t)st * LY::STAGE;
            const size_t tile_id = (size_t)ph * G + g;
            fence_proxy_async();
            mbar_expect_tx(&full[st], (uint32_t)LY::TILES);
            if constexpr (FMT == FMT_FP8) {
              tma_load_2d(stg, tmk, 0, (int)(tile_id * kBlock), &full[st]);
              tma_load_2d(stg + TR::KTILE, tmv, 0, (int)(tile_id * kBlock), &full[st]);
              bulk_g2s(stg + TR::KTILE + TR::VTILE, p.k_scale + tile_id * kBlock, TR::KSC, &full[st]);
              bulk_g2s(stg + TR::KTILE + TR::VTILE + TR::KSC, p.v_scale + tile_id * kBlock, TR::VSC, &full[st]);
            } else if constexpr (FMT == FMT_BF16) {
              tma_load_2d(stg, tmk, 0, (int)(tile_id * kBlock), &full[st]);
              tma_load_2d(stg + 128 * 128, tmk, 64, (int)(tile_id * kBlock), &full[st]);
              tma_load_2d(stg + TR::KTILE, tmv, 0, (int)(tile_id * kBlock), &full[st]);
              tma_load_2d(stg + TR::KTILE + 128 * 128, tmv, 64, (int)(tile_id * kBlock), &full[st]);
            } else {
              bulk_g2s(stg, p.k + tile_id * TR::KTILE, TR::KTILE, &full[st]);
              bulk_g2s(stg + TR::KTILE, p.v + tile_id * TR::VTILE, TR::VTILE, &full[st]);
              bulk_g2s(stg + TR::KTILE + TR::VTILE, p.k_sf + tile_id * TR::KSC, TR::KSC, &full[st]);
              bulk_g2s(stg + TR::KTILE + TR::VTILE + TR::KSC, p.v_sf + tile_id * TR::VSC, TR::VSC, &full[st]);
            }
          } else {
            mbar_arrive(&full[st]);  // rejected block: an empty phase keeps the ring in step
          }
        }
        ++bi;
      }
    }
  }
  if (!waited) pdl_wait();
  // end of the stream
  if (ok) {
    const int slot = (int)(ii & 1);
    const int use = ii >> 1;
    if (use > 0 && !ring_wait(&iempty[slot], (uint32_t)((use - 1) & 1), dead)) {
      set_dead(dead, p.status, -1);
    } else if (lane == 0) {
      facts[slot].n = -1;
      mbar_arrive(&ifull[slot]);
    }
    ++ii;
  }
  // before exiting, let the last copy into every stage and item slot land
  // (immediate in a healthy run: the consumers waited for all of them)
  if (lane == 0) {
    for (int st = 0; st < NST; ++st) {
      const int uses = bi > st ? (bi - 1 - st) / NST + 1 : 0;
      if (uses > 0) mbar_wait(&full[st], (uint32_t)((uses - 1) & 1), 2000);
    }
    for (int sl = 0; sl < 2; ++sl) {
      const int uses = ii > sl ? (ii - 1 - sl) / 2 + 1 : 0;
      if (uses > 0) mbar_wait(&ifull[sl], (uint32_t)((uses - 1) & 1), 2000);
    }
  }
}

// Atomic add at GPU scope with acquire-release semantics: the caller's earlier
// writes (and those its CTA barrier ordered before it) are visible to whoever
// reads the new count, and the old count it returns orders its later reads.
__device__ __forceinline__ int atomic_add_acq_rel(int* a, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
  return old;
}

// Merge of every split of one (sequence, group), by the CTA whose split
// finished last: out = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i.  One
// thread per 4 output dims of a column; the splits are read 8 at a time with
// every load of a group in flight together (one round trip per group).
__device__ __noinline__ void merge_splits(const AttendParams& p, int sg, int nparts, int tid, bool write) {
  const int G = p.G, Q = p.batch.Q, cols = p.geom.cols, H = G * p.r;
  const int s = sg / G, g = sg % G;
  const size_t pbase = (size_t)sg * p.splits;
#pragma unroll 1
  for (int e = tid; e < cols * 32; e += kConsumers) {
    const int col = e >> 5, d4 = (e & 31) * 4;
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int i0 = 0; i0 < nparts; i0 += 8) {
      float mi[8], li[8];
      float4 oi[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const size_t part = pbase + i0 + t;
        const bool ok = i0 + t < nparts;
        mi[t] = ok ? __ldcg(p.part_ml + (part * cols + col) * 2) : -INFINITY;
        li[t] = ok ? __ldcg(p.part_ml + (part * cols + col) * 2 + 1) : 0.f;
        oi[t] = ok ? __ldcg(reinterpret_cast<const float4*>(p.part_o + (part * cols + col) * 128 + d4))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float mn = M;
#pragma unroll
      for (int t = 0; t < 8; ++t) mn = fmaxf(mn, mi[t]);
      if (mn == -INFINITY) continue;
      const float a = ex2(M - mn);  // M = -inf: 0
      acc.x *= a;
      acc.y *= a;
      acc.z *= a;
      acc.w *= a;
      L *= a;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const float w = ex2(mi[t] - mn);  // -inf: 0
        acc.x += w * oi[t].x;
        acc.y += w * oi[t].y;
        acc.z += w * oi[t].z;
        acc.w += w * oi[t].w;
        L += w * li[t];
      }
      M = mn;
    }
    const float inv = (L > 0.f) ? __fdividef(1.f, L) : 0.f;
    if (!write) continue;
    const int qi = col_div(col, p.r), hh = col - qi * p.r;
    const size_t orow = (size_t)(s * Q + qi) * H + g * p.r + hh;
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + orow * 128 + d4) = pk;
    if (d4 == 0 && p.lse) p.lse[orow] = (L > 0.f) ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
  }
}

template <int FMT, int NT, int SP>
__device__ __forceinline__ void attend_consumer(const AttendParams& p, uint8_t* base, uint64_t* full, uint64_t* empty,
                                                uint64_t* ifull, uint64_t* iempty, int* dead, const ItemFacts* facts,
                                                int warp, int lane) {
  using LY = AttLayout<FMT, NT, SP>;
  constexpr int NST = LY::NST;
  constexpr int KG = LY::KG;       // warps sharing a column tile (key ranges)
  constexpr int KW = 32 * NT;      // keys of a warp
  const BatchDev bt = p.batch;
  const int G = p.G, Q = bt.Q;
  const int cols = p.geom.cols;
  const int H = G * p.r;
  const int g8 = lane >> 2, j = lane & 3;
  const int ct = warp / KG;         // this warp's column tile
  const int kw = (warp % KG) * KW;  // and its keys within a block
  const int tid = warp * 32 + lane;
  uint8_t* psm = base + LY::PSM + (size_t)warp * LY::PSM_WARP;
  uint8_t* vdq = base + LY::VDQ;
  float* om = reinterpret_cast<float*>(base + LY::MERGE);  // KG > 1: [4 warps][8 cols][kMergeRow]
  float* mls = om + (size_t)kWarps * 8 * kMergeRow;        // [4][8][2]: running max, row sum
  int* last_flag = reinterpret_cast<int*>(base + LY::MERGE + LY::MERGE_BYTES);
  int bi = 0;
  int pend_sg = -1, pend_np = 0, pend_old = 0;  // the previous item's split count (answer in thread 0)
  // Item -1 is a dry run before the grid dependency wait: the same code over
  // the first stage with every key masked and no global writes, so that the
  // instruction path is fetched while the preceding kernel still runs.
#pragma unroll 1
  for (int ii = -1;; ++ii) {
    const bool dry = ii < 0;
    const int slot = dry ? 0 : (int)(ii & 1);
    bool got = true;
    if (!dry) {
      got = ring_wait(&ifull[slot], (uint32_t)((ii >> 1) & 1), dead);
      if (!got) set_dead(dead, p.status, (int)ii);
    }
    if (named_bar_or(1, kConsumers, !got)) break;  // every consumer warp leaves together
    const ItemFacts& f = facts[slot];
    const int n = dry ? 1 : f.n;
    if (n < 0) break;
    const int sg = dry ? 0 : f.sg, split = dry ? 0 : f.split, count = dry ? 0 : f.count;
    const int s = sg / G, g = sg % G;
    const int T = dry ? 0 : bt.seq_len(s);
    const uint32_t* fr = reinterpret_cast<const uint32_t*>(base + LY::ITEM_OFF + (size_t)slot * LY::ISLOT);
    const float* cf = reinterpret_cast<const float*>(base + LY::ITEM_OFF + (size_t)slot * LY::ISLOT + LY::FRAGW);

    float colf[2], m_run[2], l_run[2];
    int qlim[2], qbit[2];
    float o[8][4];
    int e_prev = 0;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int col = ct * 8 + 2 * j + c;
      const int qi = col_div(col, p.r);
      colf[c] = (n > 0) ? cf[col] : 0.f;
      qlim[c] = (col < cols) ? T - Q + qi : -1;
      qbit[c] = (col < cols) ? qi : 0;
      m_run[c] = -INFINITY;
      l_run[c] = 0.f;
#pragma unroll
      for (int mm = 0; mm < 8; ++mm) o[mm][c] = o[mm][c + 2] = 0.f;
    }

#pragma unroll 1
    for (int k = 0; k < n; ++k) {
      const int st = dry ? 0 : (int)(bi % NST);
      bool have = true;
      if (!dry) {
        have = ring_wait(&full[st], (uint32_t)((bi / NST) & 1), dead);
        ++bi;
        if (!have) set_dead(dead, p.status, sg);
      }
      if constexpr (FMT == FMT_NVFP4 && NT > 1) {
        // the block's work has barriers among the consumers: decide together
        have = !named_bar_or(1, kConsumers, !have);
      }
      if (have && (dry || f.sok[k])) {
        attend_block<FMT, NT, SP>(base + (size_t)st * LY::STAGE, psm, vdq, fr, ct, colf, qlim, qbit,
                                  dry ? 0u : f.smask[k], (dry ? 0 : f.sb[k]) * kBlock + kw, kw, warp, lane, m_run,
                                  l_run, o, e_prev, dry ? (1u << warp) : kAllPhases, p.nv_round != 0);
      }
      __syncwarp();
      if (!dry && lane == 0) mbar_arrive(&empty[st]);
    }

    // ---------------- the item's result: its output rows when the (sequence, group)
    // fits this split, else its partial (o, m, l), merged by the last split
    const bool wdead = cta_dead(dead);
    const float oscale = (FMT == FMT_FP8) ? (e_prev >= -126 && e_prev <= 126 ? pow2i(-e_prev) : ldexpf(1.f, -e_prev))
                                           : ((FMT == FMT_NVFP4) ? p.v_global : 1.f);
    const bool whole = (count <= p.bps);
    const bool write = !dry;
    const size_t part = (size_t)sg * p.splits + split;
    float* po = p.part_o + part * cols * 128;
    float* pml = p.part_ml + part * cols * 2;
    float lsum[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v = l_run[c];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      lsum[c] = v;
    }
    if constexpr (KG == 1) {
      // this warp alone holds its columns: write them
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const float M = wdead ? -INFINITY : m_run[c];
        const float L = wdead ? 0.f : lsum[c];
        const int col = ct * 8 + 2 * j + c;
        if (col >= cols || !write) continue;
        const float fo = whole ? (L > 0.f ? __fdividef(oscale, L) : 0.f) : oscale;
        const int qi = col_div(col, p.r), hh = col - qi * p.r;
        const size_t orow = (size_t)(s * Q + qi) * H + g * p.r + hh;
#pragma unroll
        for (int mm = 0; mm < 8; ++mm)
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            int d;  // accumulator row 16mm + 8h2 + g8 -> output dim
            if constexpr (FMT == FMT_FP8) d = 16 * (((g8 & 1) << 2) | (g8 >> 1)) + 2 * mm + h2;
            else d = 16 * mm + 8 * h2 + g8;
            const float v = wdead ? 0.f : o[mm][c + 2 * h2] * fo;
            if (whole) static_cast<__nv_bfloat16*>(p.out)[orow * 128 + d] = __float2bfloat16_rn(v);
            else po[col * 128 + d] = v;
          }
        if (g8 == 0) {
          if (whole) {
            if (p.lse) p.lse[orow] = (L > 0.f) ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
          } else {
            pml[2 * col] = M;
            pml[2 * col + 1] = L;
          }
        }
      }
    } else {
      // the KG warps of a column tile hold different keys: merge them in shared
      // memory.  In the dry run, half of the warps take the stores and half the
      // merge loop, without barriers, so both parts are fetched at once.
      const bool seg_store = !dry || (warp & 1) == 0;
      const bool seg_merge = !dry || (warp & 1) == 1;
#pragma unroll
      for (int c = 0; c < 2 && seg_store; ++c) {
        const int cl = 2 * j + c;
        if (g8 == 0) {
          mls[(warp * 8 + cl) * 2] = wdead ? -INFINITY : m_run[c];
          mls[(warp * 8 + cl) * 2 + 1] = wdead ? 0.f : lsum[c];
        }
#pragma unroll
        for (int mm = 0; mm < 8; ++mm)
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2)
            om[(warp * 8 + cl) * kMergeRow + 16 * mm + 8 * h2 + g8] = o[mm][c + 2 * h2] * oscale;
      }
      if (!dry) named_bar_sync(1, kConsumers);
#pragma unroll 1
      for (int e = tid; e < NT * 8 * 128 && seg_merge; e += kConsumers) {
        const int tct = e >> 10, cl = (e >> 7) & 7, sl = e & 127;  // tile, column, accumulator row
        const int col = tct * 8 + cl;
        if (col >= cols) continue;
        int d;
        if constexpr (FMT == FMT_FP8) {
          const int g8s = sl & 7;
          d = 16 * (((g8s & 1) << 2) | (g8s >> 1)) + 2 * (sl >> 4) + ((sl >> 3) & 1);
        } else {
          d = sl;
        }
        float M = -INFINITY;
#pragma unroll
        for (int kq = 0; kq < KG; ++kq) M = fmaxf(M, mls[((tct * KG + kq) * 8 + cl) * 2]);
        float acc = 0.f, L = 0.f;
#pragma unroll
        for (int kq = 0; kq < KG; ++kq) {
          const float mw = mls[((tct * KG + kq) * 8 + cl) * 2];
          const float fw = (M == -INFINITY || mw == -INFINITY) ? 0.f : ex2(mw - M);
          L += fw * mls[((tct * KG + kq) * 8 + cl) * 2 + 1];
          acc += fw * om[((tct * KG + kq) * 8 + cl) * kMergeRow + sl];
        }
        if (!write) continue;
        if (whole) {
          const int qi = col_div(col, p.r), hh = col - qi * p.r;
          const size_t orow = (size_t)(s * Q + qi) * H + g * p.r + hh;
          static_cast<__nv_bfloat16*>(p.out)[orow * 128 + d] = __float2bfloat16_rn(L > 0.f ? __fdividef(acc, L) : 0.f);
          if (d == 0 && p.lse) p.lse[orow] = (L > 0.f) ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
        } else {
          po[col * 128 + d] = acc;
          if (d == 0) {
            pml[2 * col] = M;
            pml[2 * col + 1] = L;
          }
        }
      }
    }
    // ---------------- the split that finishes its (sequence, group) last merges all
    // of them.  The count is taken one item late: its atomic's answer is used
    // only after the next item, so nothing waits on it.
    if (!dry) named_bar_sync(1, kConsumers);  // every partial of this item written; the merge area is free again
    if (pend_sg >= 0) {
      if (tid == 0) *last_flag = (pend_old == pend_np - 1) ? 1 : 0;
      named_bar_sync(1, kConsumers);
      if (*last_flag) {
        __threadfence();
        merge_splits(p, pend_sg, pend_np, tid, true);
      }
      pend_sg = -1;
    }
    if (!whole && write) {
      pend_sg = sg;
      pend_np = (count + p.bps - 1) / p.bps;
      if (tid == 0) pend_old = atomic_add_acq_rel(p.sg_ctr + sg, 1);  // releases the CTA's partials
    }
    if (dry) {
      pdl_wait();  // the selection / union and the query fragments come from the preceding kernel
    } else if (lane == 0) {
      mbar_arrive(&iempty[slot]);
    }
  }
  if (pend_sg >= 0) {  // the last item's count
    if (tid == 0) *last_flag = (pend_old == pend_np - 1) ? 1 : 0;
    named_bar_sync(1, kConsumers);
    if (*last_flag) {
      __threadfence();
      merge_splits(p, pend_sg, pend_np, tid, true);
    }
  }
}

// 168 registers a thread: ten warps of two CTAs spread 3/3/2/2 over the four
// SM sub-partitions, 3 x 168 x 32 <= 16384 registers each.
template <int FMT, int NT, int SP>
__global__ void __maxnreg__(168)
    attend_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const AttendParams p) {
  using LY = AttLayout<FMT, NT, SP>;
  constexpr int NST = LY::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base + LY::BARS);
  uint64_t* empty = full + NST;
  uint64_t* ifull = empty + NST;
  uint64_t* iempty = ifull + 2;
  int* dead = reinterpret_cast<int*>(iempty + 2);
  ItemFacts* facts = reinterpret_cast<ItemFacts*>(base + LY::FACTS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kWarps);
    }
    for (int sl = 0; sl < 2; ++sl) {
      mbar_init(&ifull[sl], 1);
      mbar_init(&iempty[sl], kWarps);
    }
    *dead = 0;
    fence_mbar_init();
    if constexpr (FMT != FMT_NVFP4) {
      prefetch_tmap(&tmk);
      prefetch_tmap(&tmv);
    }
  }
  __syncthreads();
  // each role waits for the preceding kernel itself, after the work that does not need it
  if (warp == kWarps) attend_producer<FMT, NT, SP>(&tmk, &tmv, p, base, full, empty, ifull, iempty, dead, facts, lane);
  else attend_consumer<FMT, NT, SP>(p, base, full, empty, ifull, iempty, dead, facts, warp, lane);
}

cudaLaunchConfig_t pdl_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl, cudaLaunchAttribute* attr) {
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

template <int FMT, int NT, int SP>
cudaError_t launch_att(const CUtensorMap* tk, const CUtensorMap* tv, const AttendParams& p, int num_sms,
                       cudaStream_t st, bool pdl) {
  const size_t smem = AttLayout<FMT, NT, SP>::SMEM;
  auto kern = attend_kernel<FMT, NT, SP>;
  static int per_sm = 0;  // CTAs per SM for this instance (same on every device of one kind)
  if (per_sm == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    per_sm = n > 0 ? n : 1;
  }
  const long items = (long)p.batch.S * p.G * p.splits;
  long grid = (long)per_sm * (num_sms > 0 ? num_sms : 1);
  if (grid > items) grid = items;
  if (grid < 1) grid = 1;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_cfg(dim3((unsigned)grid), dim3(kThreads), smem, st, pdl, attr);
  CUtensorMap dummy = {};
  return cudaLaunchKernelEx(&cfg, kern, tk ? *tk : dummy, tv ? *tv : dummy, p);
}

template <int FMT>
cudaError_t launch_att_fmt(const CUtensorMap* tk, const CUtensorMap* tv, const AttendParams& p, int num_sms,
                           cudaStream_t st, bool pdl) {
  const int nt = p.geom.nt;
  if (p.geom.sp == 2) {
    if constexpr (FMT == FMT_FP8) {
      switch (nt) {
        case 1: return launch_att<FMT, 1, 2>(tk, tv, p, num_sms, st, pdl);
        case 2: return launch_att<FMT, 2, 2>(tk, tv, p, num_sms, st, pdl);
        case 4: return launch_att<FMT, 4, 2>(tk, tv, p, num_sms, st, pdl);
        default: return cudaErrorInvalidValue;
      }
    }
    return cudaErrorInvalidValue;
  }
  switch (nt) {
    case 1: return launch_att<FMT, 1, 1>(tk, tv, p, num_sms, st, pdl);
    case 2: return launch_att<FMT, 2, 1>(tk, tv, p, num_sms, st, pdl);
    case 4: return launch_att<FMT, 4, 1>(tk, tv, p, num_sms, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_attend(int fmt, const CUtensorMap* tk, const CUtensorMap* tv, const AttendParams& p, int num_sms,
                          cudaStream_t st, bool pdl) {
  switch (fmt) {
    case FMT_FP8: return launch_att_fmt<FMT_FP8>(tk, tv, p, num_sms, st, pdl);
    case FMT_BF16: return launch_att_fmt<FMT_BF16>(tk, tv, p, num_sms, st, pdl);
    case FMT_NVFP4: return launch_att_fmt<FMT_NVFP4>(tk, tv, p, num_sms, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace msa
