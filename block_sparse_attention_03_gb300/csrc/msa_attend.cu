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
// Work.  Unit = (sequence, group, split): the group's selected blocks (for
// several query tokens: the union of their selections) cut into splits of
// `bps` blocks, one CTA per unit, several CTAs per SM so that the hardware
// overlaps one CTA's loads with another's math.  Warp 0 fetches the unit's
// facts with parallel lane loads and thread 0 issues every block of the unit
// at once (one shared-memory stage per block: TMA tensor copies with the
// 128-byte swizzle for FP8 / BF16, bulk copies for NVFP4), together with the
// query fragments the preceding kernel prepared.  Warp w owns keys
// [32w, 32w+32) of every block with its own online softmax; at the end the
// four warps merge through shared memory (over the dead stages).  A (sequence,
// group) that fits one split writes its bf16 output and LSE directly;
// otherwise each split writes a partial and combine_kernel merges them by
// log-sum-exp (one warp per output row and head).
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

namespace msa {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kMergeRow = 132;  // padded row of the merge area (conflict-free stores)

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
__host__ __device__ constexpr size_t cmax(size_t a, size_t b) { return a > b ? a : b; }

// Blocks per unit (= stages): all of a unit's tiles are in flight at once.
template <int FMT, int NT>
__host__ __device__ constexpr int att_stages() {
  return FMT == FMT_BF16 ? 2 : (FMT == FMT_FP8 ? 2 : (NT == 1 ? 4 : 2));
}

template <int FMT, int NT, int SP>
struct AttLayout {
  using T = AttTraits<FMT>;
  static constexpr int NC = NT * 8;
  static constexpr int NST = att_stages<FMT, NT>();
  static constexpr size_t TILES = (size_t)T::KTILE + T::VTILE + T::KSC + T::VSC;
  static constexpr size_t STAGE = round_up(TILES, 1024);
  static constexpr size_t FRAGW = (size_t)SP * NT * T::QKS * 64 * 4;  // query fragment words
  static constexpr size_t FRAG_OFF = STAGE * NST;
  static constexpr size_t FRAG = FRAGW + NC * 4;                      // + column factors
  static constexpr size_t PSM = round_up(FRAG_OFF + FRAG, 16);        // per-warp P tiles
  static constexpr size_t PSM_WARP = 64 * NC;
  static constexpr size_t VDQ = PSM + kWarps * PSM_WARP;              // NVFP4 V^T f16 tiles
  static constexpr size_t VDQ_WARP = (FMT == FMT_NVFP4) ? 32 * 256 : 0;
  static constexpr size_t DATA_END = VDQ + kWarps * VDQ_WARP;
  static constexpr size_t MERGE_BYTES = (size_t)kWarps * NC * (kMergeRow + 2) * 4;  // aliases the data area
  static constexpr size_t BARS = round_up(cmax(DATA_END, MERGE_BYTES), 16);
  static constexpr size_t TOTAL = BARS + 8 * NST + 8 + 16 * NST + 16;
  static constexpr size_t SMEM = TOTAL + 1024;
};

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

template <int FMT, int NT, int SP>
__global__ void __launch_bounds__(kThreads)
    attend_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const AttendParams p) {
  using TR = AttTraits<FMT>;
  using LY = AttLayout<FMT, NT, SP>;
  constexpr int NC = NT * 8;
  constexpr int NST = LY::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base + LY::BARS);
  uint64_t* fbar = full + NST;
  int* sb = reinterpret_cast<int*>(fbar + 1);          // [NST] block ids
  uint32_t* smask = reinterpret_cast<uint32_t*>(sb + NST);
  int* sok = reinterpret_cast<int*>(smask + NST);      // [NST] 1: loaded
  int* sinfo = sok + NST;                              // n, count, empty

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BatchDev bt = p.batch;
  const int G = p.G, Q = bt.Q;
  const int cols = p.geom.cols;
  const int unit = blockIdx.x;
  const int sg = unit / p.splits, split = unit % p.splits;
  const int s = sg / G, g = sg % G;

  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) mbar_init(&full[st], 1);
    mbar_init(fbar, 1);
    fence_mbar_init();
    if constexpr (FMT != FMT_NVFP4) {
      prefetch_tmap(&tmk);
      prefetch_tmap(&tmv);
    }
  }
  pdl_wait();  // the selection / union, fragments and counters come from the preceding kernel
  const int T = bt.seq_len(s);

  // ---------------- warp 0: the unit's facts (parallel lane loads); thread 0 issues every copy
  if (warp == 0) {
    int entry = -1, count;
    if (p.direct) {
      entry = (lane < p.topk) ? p.topk_idx[(size_t)sg * p.topk + lane] : -1;
      count = __popc(__ballot_sync(0xffffffffu, entry >= 0));
    } else {
      count = p.u_count[sg];
    }
    const int kb0 = split * p.bps;
    int n = min(p.bps, count - kb0);
    const bool empty_sg = (count == 0);
    if (n < 0) n = 0;
    int b = -1, phys = -1;
    uint32_t mask = 0;
    if (lane < n) {
      if (p.direct) {
        mask = 1u;
      } else {
        b = p.u_ids[(size_t)sg * p.cap + kb0 + lane];
        mask = p.u_mask[(size_t)sg * p.cap + kb0 + lane];
      }
    }
    if (p.direct) b = __shfl_sync(0xffffffffu, entry, (kb0 + lane) & 31);
    if (lane < n) {
      if (b < 0 || T < 0 || b > (T - 1) / kBlock) {
        raise_flag(p.status, FLAG_BAD_SELECT, b);
        b = -1;
      } else {
        const int ph = bt.row(s)[b];
        if (ph < 0 || ph >= p.num_blocks) raise_flag(p.status, FLAG_BAD_BLOCK, ph);
        else phys = ph;
      }
      sb[lane] = b;
      smask[lane] = mask;
      sok[lane] = phys >= 0 ? 1 : 0;
    }
    if (lane == 0) {
      sinfo[0] = n;
      sinfo[1] = count;
      sinfo[2] = empty_sg ? 1 : 0;
      if (n > 0) {
        uint8_t* fd = base + LY::FRAG_OFF;
        mbar_expect_tx(fbar, (uint32_t)LY::FRAG);
        bulk_g2s(fd, p.frag + (size_t)sg * (LY::FRAGW / 4), (uint32_t)LY::FRAGW, fbar);
        bulk_g2s(fd + LY::FRAGW, p.colf + (size_t)sg * NC, NC * 4, fbar);
      }
    }
    for (int k = 0; k < n; ++k) {
      const int ph = __shfl_sync(0xffffffffu, phys, k);
      if (lane == 0 && ph >= 0) {
        uint8_t* stg = base + (size_t)k * LY::STAGE;
        const size_t tile_id = (size_t)ph * G + g;
        mbar_expect_tx(&full[k], (uint32_t)LY::TILES);
        if constexpr (FMT == FMT_FP8) {
          tma_load_2d(stg, &tmk, 0, (int)(tile_id * kBlock), &full[k]);
          tma_load_2d(stg + TR::KTILE, &tmv, 0, (int)(tile_id * kBlock), &full[k]);
          bulk_g2s(stg + TR::KTILE + TR::VTILE, p.k_scale + tile_id * kBlock, TR::KSC, &full[k]);
          bulk_g2s(stg + TR::KTILE + TR::VTILE + TR::KSC, p.v_scale + tile_id * kBlock, TR::VSC, &full[k]);
        } else if constexpr (FMT == FMT_BF16) {
          tma_load_2d(stg, &tmk, 0, (int)(tile_id * kBlock), &full[k]);
          tma_load_2d(stg + 128 * 128, &tmk, 64, (int)(tile_id * kBlock), &full[k]);
          tma_load_2d(stg + TR::KTILE, &tmv, 0, (int)(tile_id * kBlock), &full[k]);
          tma_load_2d(stg + TR::KTILE + 128 * 128, &tmv, 64, (int)(tile_id * kBlock), &full[k]);
        } else {
          bulk_g2s(stg, p.k + tile_id * TR::KTILE, TR::KTILE, &full[k]);
          bulk_g2s(stg + TR::KTILE, p.v + tile_id * TR::VTILE, TR::VTILE, &full[k]);
          bulk_g2s(stg + TR::KTILE + TR::VTILE, p.k_sf + tile_id * TR::KSC, TR::KSC, &full[k]);
          bulk_g2s(stg + TR::KTILE + TR::VTILE + TR::KSC, p.v_sf + tile_id * TR::VSC, TR::VSC, &full[k]);
        }
      }
    }
  }
  __syncthreads();
  pdl_launch_dependents();
  const int n = sinfo[0];
  const int count = sinfo[1];
  if (n == 0 && !(sinfo[2] && split == 0)) return;  // nothing in this split (the sequence's last splits)

  // ---------------- every warp: query fragments, softmax state
  const int g8 = lane >> 2, j = lane & 3;
  const int kw = 32 * warp;  // this warp's keys within a block
  uint8_t* psm = base + LY::PSM + (size_t)warp * LY::PSM_WARP;
  uint32_t bq[SP][NT][TR::QKS][2];
  float colf[NT][2];
  int qlim[NT][2], qbit[NT][2];
  float m_run[NT][2], l_run[NT][2];
  float o[8][NT][4];
  int e_prev = 0;
  bool dead = false;
  if (n > 0) {
    if (!mbar_wait_warp(fbar, 0)) {
      if (lane == 0) raise_flag(p.status, FLAG_TIMEOUT, unit);
      dead = true;
    }
  }
  if (n > 0 && !dead) {
    const uint32_t* fr = reinterpret_cast<const uint32_t*>(base + LY::FRAG_OFF);
    const float* cf = reinterpret_cast<const float*>(base + LY::FRAG_OFF + LY::FRAGW);
#pragma unroll
    for (int sp = 0; sp < SP; ++sp)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int ks = 0; ks < TR::QKS; ++ks)
#pragma unroll
          for (int rg = 0; rg < 2; ++rg) bq[sp][nt][ks][rg] = fr[(((sp * NT + nt) * TR::QKS + ks) * 2 + rg) * 32 + lane];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) colf[nt][c] = cf[nt * 8 + 2 * j + c];
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int col = nt * 8 + 2 * j + c;
      const int qi = col / p.r;
      qlim[nt][c] = (col < cols) ? T - Q + qi : -1;
      qbit[nt][c] = (col < cols) ? qi : 0;
      m_run[nt][c] = -INFINITY;
      l_run[nt][c] = 0.f;
#pragma unroll
      for (int mm = 0; mm < 8; ++mm) o[mm][nt][c] = o[mm][nt][c + 2] = 0.f;
    }

  for (int k = 0; k < n && !dead; ++k) {
    if (!sok[k]) continue;  // rejected block: nothing was copied, nothing to wait for
    if (!mbar_wait_warp(&full[k], 0)) {
      if (lane == 0) raise_flag(p.status, FLAG_TIMEOUT, unit);
      dead = true;
      break;
    }
    const uint8_t* stg = base + (size_t)k * LY::STAGE;
    const uint32_t qmask = smask[k];
    const int key0 = sb[k] * kBlock + kw;
    // ---------------- logits^T for this warp's 32 keys
    float sacc[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) sacc[mt][nt][0] = sacc[mt][nt][1] = sacc[mt][nt][2] = sacc[mt][nt][3] = 0.f;
    const uint32_t kt = smem_u32(stg);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      if constexpr (FMT == FMT_FP8 || FMT == FMT_BF16) {
        const int row = kw + 16 * mt + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int ks = 0; ks < TR::QKS; ++ks) {
          uint32_t a[4];
          if constexpr (FMT == FMT_FP8) {
            ldmatrix_x4(a, swz(kt, row, 2 * ks + (lane >> 4)));
#pragma unroll
            for (int sp = 0; sp < SP; ++sp)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) mma_e4m3_k32(sacc[mt][nt], a, bq[sp][nt][ks][0], bq[sp][nt][ks][1]);
          } else {
            ldmatrix_x4(a, swz(kt + (ks >> 2) * (128 * 128), row, 2 * (ks & 3) + (lane >> 4)));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16_k16(sacc[mt][nt], a, bq[0][nt][ks][0], bq[0][nt][ks][1]);
          }
        }
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
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_f16_k16(sacc[mt][nt], a, bq[0][nt][ks][0], bq[0][nt][ks][1]);
        }
      }
    }

    // ---------------- scale, mask, online softmax (per column, over this warp's keys)
    float ksc[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float v = 1.f;
        if constexpr (FMT == FMT_FP8)
          v = reinterpret_cast<const float*>(stg + TR::KTILE + TR::VTILE)[kw + 16 * mt + g8 + 8 * hh];
        ksc[mt][hh] = v;
      }
    float alpha[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const bool sel = (qmask >> qbit[nt][c]) & 1u;
        float bmax = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int key = key0 + 16 * mt + g8 + 8 * hh;
            const bool vis = sel && key <= qlim[nt][c];
            const float x = vis ? sacc[mt][nt][c + 2 * hh] * ksc[mt][hh] * colf[nt][c] : -INFINITY;
            sacc[mt][nt][c + 2 * hh] = x;
            bmax = fmaxf(bmax, x);
          }
        bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 4));
        bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 8));
        bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 16));
        const float mnew = fmaxf(m_run[nt][c], bmax);
        const float msub = (mnew == -INFINITY) ? 0.f : mnew;
        alpha[nt][c] = exp2f(m_run[nt][c] - msub);
        float psum = 0.f;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const float pv = exp2f(sacc[mt][nt][c + 2 * hh] - msub);
            sacc[mt][nt][c + 2 * hh] = pv;
            psum += pv;
          }
        psum += __shfl_xor_sync(0xffffffffu, psum, 4);
        psum += __shfl_xor_sync(0xffffffffu, psum, 8);
        psum += __shfl_xor_sync(0xffffffffu, psum, 16);
        l_run[nt][c] = l_run[nt][c] * alpha[nt][c] + psum;
        m_run[nt][c] = mnew;
      }

    // ---------------- P operand into this warp's shared tile, then B fragments
    __syncwarp();
    if constexpr (FMT == FMT_FP8) {
      // P' = p * vscale * 2^e, split into e4m3 hi + lo
      const float* vsc = reinterpret_cast<const float*>(stg + TR::KTILE + TR::VTILE + TR::KSC);
      float vmax = vsc[kw + lane];
      for (int off = 16; off > 0; off >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
      const int e = pow2_fit(vmax, 448.f);
      const float fe = ldexpf(1.f, e);
      const float resc = ldexpf(1.f, e - e_prev);
      e_prev = e;
      // this lane's keys 16mt + g8 + 8hh of a column sit in bytes 2mt + hh of
      // word g8 of that column's P row (keys j + 8i: bytes of b0, keys 4 + j + 8i:
      // bytes of b1, for lane j): one word per (column, term)
      float vs[2][2];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) vs[mt][hh] = vsc[kw + 16 * mt + g8 + 8 * hh] * fe;
      uint32_t* psm32 = reinterpret_cast<uint32_t*>(psm);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float hi[4], lo[4];
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
              split_e4m3(sacc[mt][nt][c + 2 * hh] * vs[mt][hh], hi[2 * mt + hh], lo[2 * mt + hh]);
          const int col = nt * 8 + 2 * j + c;
          psm32[col * 8 + g8] = (uint32_t)pack_e4m3x2(hi[0], hi[1]) | ((uint32_t)pack_e4m3x2(hi[2], hi[3]) << 16);
          psm32[NC * 8 + col * 8 + g8] =
              (uint32_t)pack_e4m3x2(lo[0], lo[1]) | ((uint32_t)pack_e4m3x2(lo[2], lo[3]) << 16);
        }
      // rescale the running output: softmax shift and the change of P scale
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const float f = alpha[nt][c] * resc;
#pragma unroll
          for (int mm = 0; mm < 8; ++mm) {
            o[mm][nt][c] *= f;
            o[mm][nt][c + 2] *= f;
          }
        }
    } else {
      // P as one 16-bit term: bf16 for BF16 tiles, f16 for NVFP4 tiles
      uint16_t* ps16 = reinterpret_cast<uint16_t*>(psm);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int kk = 16 * mt + g8 + 8 * hh;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const int col = nt * 8 + 2 * j + c;
              const float pv = sacc[mt][nt][c + 2 * hh];
              uint16_t bits;
              if constexpr (FMT == FMT_BF16) {
                __nv_bfloat16 x = __float2bfloat16_rn(pv);
                bits = *reinterpret_cast<uint16_t*>(&x);
              } else {
                __half x = __float2half_rn(pv);
                bits = *reinterpret_cast<uint16_t*>(&x);
              }
              ps16[col * 32 + kk] = bits;
            }
        }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int mm = 0; mm < 8; ++mm) {
            o[mm][nt][c] *= alpha[nt][c];
            o[mm][nt][c + 2] *= alpha[nt][c];
          }
      if constexpr (FMT == FMT_NVFP4) {
        // dequantize this warp's 32 V rows to f16 (exact) into a swizzled tile
        const uint8_t* vraw = stg + TR::KTILE;
        const uint8_t* vsf = stg + TR::KTILE + TR::VTILE + TR::KSC;
        uint8_t* vdq = base + LY::VDQ + (size_t)warp * LY::VDQ_WARP;
        const int key = kw + lane;
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
          }
          // 32 dims = d 32*q4 .. +31 -> f16 bytes 64*q4 .. +63 -> half (q4>>1), chunks 4*(q4&1) .. +3
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const uint32_t addr = swz(vb + (q4 >> 1) * (32 * 128), lane, 4 * (q4 & 1) + cc);
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(out[4 * cc]), "r"(out[4 * cc + 1]),
                         "r"(out[4 * cc + 2]), "r"(out[4 * cc + 3]));
          }
        }
      }
    }
    __syncwarp();

    // ---------------- O^T += V^T P
    if constexpr (FMT == FMT_FP8) {
      uint32_t bp[2][NT][2];
#pragma unroll
      for (int sp = 0; sp < 2; ++sp)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint8_t* row = psm + sp * NC * 32 + (nt * 8 + g8) * 32;
          bp[sp][nt][0] = *reinterpret_cast<const uint32_t*>(row + 4 * j);
          bp[sp][nt][1] = *reinterpret_cast<const uint32_t*>(row + 16 + 4 * j);
        }
      const uint32_t vt = smem_u32(stg + TR::KTILE);
      const int cg = (g8 >> 1) | ((g8 & 1) << 2);  // this lane's 16-dim chunk
      uint32_t A0[16], A2[16];
#pragma unroll
      for (int set = 0; set < 2; ++set) {
        uint4 raw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int key = kw + 8 * i + 4 * set + j;
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
          for (int i = 0; i < 4; ++i) in[i] = (wd == 0) ? raw[i].x : (wd == 1) ? raw[i].y : (wd == 2) ? raw[i].z : raw[i].w;
          transpose4x4(in, out);
#pragma unroll
          for (int e = 0; e < 4; ++e) A[4 * wd + e] = out[e];
        }
      }
#pragma unroll
      for (int mm = 0; mm < 8; ++mm) {
        const uint32_t a[4] = {A0[2 * mm], A0[2 * mm + 1], A2[2 * mm], A2[2 * mm + 1]};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_e4m3_k32(o[mm][nt], a, bp[0][nt][0], bp[0][nt][1]);
          mma_e4m3_k32(o[mm][nt], a, bp[1][nt][0], bp[1][nt][1]);
        }
      }
    } else {
      const uint16_t* ps16 = reinterpret_cast<const uint16_t*>(psm);
      uint32_t vt;
      int vrow0;
      if constexpr (FMT == FMT_BF16) {
        vt = smem_u32(stg + TR::KTILE);
        vrow0 = kw;
      } else {
        vt = smem_u32(base + LY::VDQ + (size_t)warp * LY::VDQ_WARP);
        vrow0 = 0;
      }
      constexpr int HALF = (FMT == FMT_BF16) ? 128 * 128 : 32 * 128;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t bp[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint16_t* row = ps16 + (nt * 8 + g8) * 32 + 16 * kk;
          bp[nt][0] = *reinterpret_cast<const uint32_t*>(row + 2 * j);
          bp[nt][1] = *reinterpret_cast<const uint32_t*>(row + 8 + 2 * j);
        }
        const int key = vrow0 + 16 * kk + (lane & 7) + 8 * ((lane >> 4) & 1);
#pragma unroll
        for (int mm = 0; mm < 8; ++mm) {
          const int d0 = 16 * mm + 8 * ((lane >> 3) & 1);
          uint32_t a[4];
          ldmatrix_x4_trans(a, swz(vt + (d0 >> 6) * HALF, key, (d0 & 63) >> 3));
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if constexpr (FMT == FMT_BF16)
              mma_bf16_k16(o[mm][nt], a, bp[nt][0], bp[nt][1]);
            else
              mma_f16_k16(o[mm][nt], a, bp[nt][0], bp[nt][1]);
          }
        }
      }
    }
    __syncwarp();
  }

  // ---------------- merge the four warps (over the dead stages), write output or partial
  const bool any_dead = __syncthreads_or(dead);
  if (any_dead) {
    if (threadIdx.x == 0) {  // bounded wait for copies still in flight before their buffers are reused
      mbar_wait(fbar, 0, 2000);
      for (int k = 0; k < n; ++k)
        if (sok[k]) mbar_wait(&full[k], 0, 2000);
    }
    __syncthreads();
  }
  float* om = reinterpret_cast<float*>(base);                 // [4][NC][kMergeRow], slot 16mm+8hh+g8
  float* mls = om + (size_t)kWarps * NC * kMergeRow;          // [4][NC][2]
  const float oscale = (FMT == FMT_FP8) ? ldexpf(1.f, -e_prev) : ((FMT == FMT_NVFP4) ? p.v_global : 1.f);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int col = nt * 8 + 2 * j + c;
      if (g8 == 0) {
        mls[(warp * NC + col) * 2] = dead ? -INFINITY : m_run[nt][c];
        mls[(warp * NC + col) * 2 + 1] = dead ? 0.f : l_run[nt][c];
      }
#pragma unroll
      for (int mm = 0; mm < 8; ++mm)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          om[(warp * NC + col) * kMergeRow + 16 * mm + 8 * hh + g8] = o[mm][nt][c + 2 * hh] * oscale;
    }
  __syncthreads();
  const bool whole = (count <= p.bps);  // the (sequence, group) fits this one split
  const int H = G * p.r;
  float* po = p.part_o + (size_t)unit * cols * 128;
  float* pml = p.part_ml + (size_t)unit * cols * 2;
  for (int idx = threadIdx.x; idx < cols * 128; idx += kThreads) {
    const int col = idx >> 7, d = idx & 127;
    int slot;  // merge-area position of output dim d (inverse of the accumulator row mapping)
    if constexpr (FMT == FMT_FP8) {
      const int cgd = d >> 4;
      const int g8d = ((cgd & 3) << 1) | (cgd >> 2);
      slot = 16 * ((d & 15) >> 1) + 8 * (d & 1) + g8d;
    } else {
      slot = d;
    }
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mls[(w * NC + col) * 2]);
    float acc = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = mls[(w * NC + col) * 2];
        const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
        acc += f * om[(w * NC + col) * kMergeRow + slot];
        L += f * mls[(w * NC + col) * 2 + 1];
      }
    }
    if (whole) {
      const int qi = col / p.r, hh = col % p.r;
      const size_t orow = (size_t)(s * Q + qi) * H + g * p.r + hh;
      static_cast<__nv_bfloat16*>(p.out)[orow * 128 + d] = __float2bfloat16_rn(L > 0.f ? acc / L : 0.f);
      if (d == 0 && p.lse) p.lse[orow] = (L > 0.f) ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
    } else {
      po[idx] = acc;
      if (d == 0) {
        pml[2 * col] = M;
        pml[2 * col + 1] = L;
      }
    }
  }
}

// out[row][h] = sum_k 2^(M_k - M) O_k / sum_k 2^(M_k - M) L_k over the splits of
// its (sequence, group); rows whose (sequence, group) fit one split were
// written by the attend itself.  One warp per (row, head); the loads of the
// partials are independent so they overlap.
__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
  pdl_wait();
  const int wg = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int H = p.G * p.r;
  if (wg >= p.S * p.Q * H) return;
  const int h = wg % H, sq = wg / H;
  const int s = sq / p.Q, i = sq % p.Q;
  const int g = h / p.r, hh = h % p.r;
  const int sg = s * p.G + g;
  int count;
  if (p.direct) {
    const int e = (lane < p.topk) ? p.topk_idx[(size_t)sg * p.topk + lane] : -1;
    count = __popc(__ballot_sync(0xffffffffu, e >= 0));
  } else {
    count = p.u_count[sg];
  }
  if (count <= p.bps) return;  // written by the attend
  const int nparts = (count + p.bps - 1) / p.bps;
  const int col = i * p.r + hh;
  const size_t ubase = (size_t)sg * p.splits;
  float M = -INFINITY;
  for (int k0 = 0; k0 < nparts; k0 += 32) {
    const int k = k0 + lane;
    const float mk = (k < nparts) ? __ldcg(p.part_ml + ((ubase + k) * p.cols + col) * 2) : -INFINITY;
    M = fmaxf(M, mk);
  }
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int k0 = 0; k0 < nparts; k0 += 32) {
      const int k = k0 + lane;
      float f = 0.f, lk = 0.f;
      if (k < nparts) {
        const float mk = __ldcg(p.part_ml + ((ubase + k) * p.cols + col) * 2);
        lk = __ldcg(p.part_ml + ((ubase + k) * p.cols + col) * 2 + 1);
        f = (mk == -INFINITY) ? 0.f : exp2f(mk - M);
      }
      float fl = f * lk;
      for (int o = 16; o > 0; o >>= 1) fl += __shfl_xor_sync(0xffffffffu, fl, o);
      L += fl;
      const int kn = min(32, nparts - k0);
#pragma unroll 8
      for (int t = 0; t < kn; ++t) {
        const float ft = __shfl_sync(0xffffffffu, f, t);
        const float4 v = __ldcg(reinterpret_cast<const float4*>(p.part_o + ((ubase + k0 + t) * p.cols + col) * 128) + lane);
        acc.x += ft * v.x;
        acc.y += ft * v.y;
        acc.z += ft * v.z;
        acc.w += ft * v.w;
      }
    }
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  const size_t orow = (size_t)sq * H + h;
  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out) + orow * 128 + 4 * lane;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(outp) = pk;
  if (lane == 0 && p.lse) p.lse[orow] = (L > 0.f) ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
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
cudaError_t launch_att(const CUtensorMap* tk, const CUtensorMap* tv, const AttendParams& p, cudaStream_t st, bool pdl) {
  const size_t smem = AttLayout<FMT, NT, SP>::SMEM;
  auto kern = attend_kernel<FMT, NT, SP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_cfg(dim3((unsigned)(p.batch.S * p.G * p.splits)), dim3(kThreads), smem, st, pdl, attr);
  CUtensorMap dummy = {};
  return cudaLaunchKernelEx(&cfg, kern, tk ? *tk : dummy, tv ? *tv : dummy, p);
}

template <int FMT>
cudaError_t launch_att_fmt(const CUtensorMap* tk, const CUtensorMap* tv, const AttendParams& p, cudaStream_t st,
                           bool pdl) {
  const int nt = p.geom.nt;
  if (p.geom.sp == 2) {
    if constexpr (FMT == FMT_FP8) {
      switch (nt) {
        case 1: return launch_att<FMT, 1, 2>(tk, tv, p, st, pdl);
        case 2: return launch_att<FMT, 2, 2>(tk, tv, p, st, pdl);
        case 4: return launch_att<FMT, 4, 2>(tk, tv, p, st, pdl);
        default: return cudaErrorInvalidValue;
      }
    }
    return cudaErrorInvalidValue;
  }
  switch (nt) {
    case 1: return launch_att<FMT, 1, 1>(tk, tv, p, st, pdl);
    case 2: return launch_att<FMT, 2, 1>(tk, tv, p, st, pdl);
    case 4: return launch_att<FMT, 4, 1>(tk, tv, p, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int attend_stages(int fmt, int nt) {
  if (fmt == FMT_FP8) return att_stages<FMT_FP8, 1>();
  if (fmt == FMT_BF16) return att_stages<FMT_BF16, 1>();
  return nt == 1 ? att_stages<FMT_NVFP4, 1>() : att_stages<FMT_NVFP4, 2>();
}

cudaError_t launch_attend(int fmt, const CUtensorMap* tk, const CUtensorMap* tv, const AttendParams& p, int num_sms,
                          cudaStream_t st, bool pdl) {
  (void)num_sms;
  switch (fmt) {
    case FMT_FP8: return launch_att_fmt<FMT_FP8>(tk, tv, p, st, pdl);
    case FMT_BF16: return launch_att_fmt<FMT_BF16>(tk, tv, p, st, pdl);
    case FMT_NVFP4: return launch_att_fmt<FMT_NVFP4>(tk, tv, p, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t st, bool pdl) {
  const int rows = p.S * p.Q * p.G * p.r;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_cfg(dim3((unsigned)((rows + 3) / 4)), dim3(128), 0, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace msa
