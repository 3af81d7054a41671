// Sparse attend over the selected blocks (split-K flash decoding) and the
// split combine.
//
// Definition (vLLM Day-0 blog, section "MSA 入门" and Figure 1): every query
// head of a GQA group attends, with exact softmax, to the keys of the blocks
// its group selected, at most k x 128 keys; logits are scaled by
// head_dim ** -0.5 (model page, MiniMaxM3SparseAttention: self.scaling).  With
// several new tokens per sequence (speculative verify) each token has its own
// selection and causal limit.
//
// Work decomposition.  Unit = (sequence, group, split): the union of the
// group's selected blocks (all query tokens of the sequence) is cut into
// splits of `bps` blocks.  A CTA of 4 warps loads every block of its split up
// front (one shared-memory stage per block: TMA tensor copies with the
// 128-byte swizzle for FP8 / BF16 tiles, 1-D bulk copies for NVFP4), and warp w
// handles keys [32w, 32w+32) of each block with its own online softmax, so
// the block loop has no CTA-wide barrier; the four warps' (max, sum, output)
// are merged once at the end and written as one partial.
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

template <int FMT>
struct AttTraits;
template <>
struct AttTraits<FMT_FP8> {
  static constexpr int KTILE = 128 * 128, VTILE = 128 * 128, KSC = 512, VSC = 512;
  static constexpr int NST = 2, QKS = 4;
};
template <>
struct AttTraits<FMT_BF16> {
  static constexpr int KTILE = 128 * 256, VTILE = 128 * 256, KSC = 0, VSC = 0;
  static constexpr int NST = 2, QKS = 8;
};
template <>
struct AttTraits<FMT_NVFP4> {
  static constexpr int KTILE = 128 * 64, VTILE = 128 * 64, KSC = 1024, VSC = 1024;
  static constexpr int NST = 4, QKS = 8;
};

template <int FMT>
struct AttLayout {
  using T = AttTraits<FMT>;
  static constexpr size_t STAGE = (size_t)T::KTILE + T::VTILE + T::KSC + T::VSC;  // multiple of 1024
  static constexpr size_t STAGES = STAGE * T::NST;
  static constexpr size_t PSM = STAGES;                                  // per-warp P tiles
  static constexpr size_t PSM_WARP = 2 * 32 * 32 * 2;                    // 4 KB
  static constexpr size_t VDQ = PSM + kWarps * PSM_WARP;                 // NVFP4 V^T f16 tiles
  static constexpr size_t VDQ_WARP = (FMT == FMT_NVFP4) ? 32 * 256 : 0;
  static constexpr size_t BARS = VDQ + kWarps * VDQ_WARP;
  static constexpr size_t STATE = BARS + 8 * T::NST;
  static constexpr size_t TOTAL = STATE + 4 * T::NST + 64;
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

// Key position inside a warp's 32-key FP8 P row so that b0/b1 are whole words:
// b0 of lane j holds keys {j, 8+j, 16+j, 24+j}, b1 keys {4+j, 12+j, 20+j, 28+j}.
__device__ __forceinline__ int p8_pos(int k) { return ((k & 4) ? 16 : 0) + 4 * (k & 3) + (k >> 3); }

template <int FMT, int NT, int SP>
__global__ void __launch_bounds__(kWarps * 32)
    attend_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const AttendParams p) {
  using TR = AttTraits<FMT>;
  using LY = AttLayout<FMT>;
  constexpr int NST = TR::NST;
  constexpr int NC = NT * 8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + LY::BARS);
  int* state = reinterpret_cast<int*>(base + LY::STATE);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g8 = lane >> 2, j = lane & 3;
  const BatchDev bt = p.batch;
  const int unit = blockIdx.x;
  const int sg = unit / p.splits, split = unit % p.splits;
  const int s = sg / p.G;
  const int cols = p.geom.cols;

  pdl_wait();
  const int count = p.u_count[sg];
  const int kb0 = split * p.bps;
  const int nblk = max(0, min(p.bps, count - kb0));
  float* pml = p.part_ml + (size_t)unit * cols * 2;
  if (nblk == 0) {
    for (int c = threadIdx.x; c < cols; c += blockDim.x) {
      pml[2 * c] = -INFINITY;
      pml[2 * c + 1] = 0.f;
    }
    pdl_launch_dependents();
    return;
  }
  const int T = bt.seq_lens[s];

  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) mbar_init(&bars[st], 1);
    fence_mbar_init();
    for (int k = 0; k < nblk; ++k) {
      const int b = p.u_ids[(size_t)sg * p.cap + kb0 + k];
      const int phys = bt.block_table[(size_t)s * bt.max_nb + b];
      if (phys < 0 || phys >= p.num_blocks) {
        raise_flag(p.status, FLAG_BAD_BLOCK, phys);
        state[k] = 0;
        continue;
      }
      state[k] = 1;
      uint8_t* stg = base + (size_t)k * LY::STAGE;
      const int g = sg % p.G;
      const size_t tile_id = (size_t)phys * p.G + g;
      if constexpr (FMT == FMT_FP8) {
        mbar_expect_tx(&bars[k], TR::KTILE + TR::VTILE + TR::KSC + TR::VSC);
        tma_load_2d(stg, &tmk, 0, (int)(tile_id * kBlock), &bars[k]);
        tma_load_2d(stg + TR::KTILE, &tmv, 0, (int)(tile_id * kBlock), &bars[k]);
        bulk_g2s(stg + TR::KTILE + TR::VTILE, p.k_scale + tile_id * kBlock, TR::KSC, &bars[k]);
        bulk_g2s(stg + TR::KTILE + TR::VTILE + TR::KSC, p.v_scale + tile_id * kBlock, TR::VSC, &bars[k]);
      } else if constexpr (FMT == FMT_BF16) {
        mbar_expect_tx(&bars[k], TR::KTILE + TR::VTILE);
        tma_load_2d(stg, &tmk, 0, (int)(tile_id * kBlock), &bars[k]);
        tma_load_2d(stg + 128 * 128, &tmk, 64, (int)(tile_id * kBlock), &bars[k]);
        tma_load_2d(stg + TR::KTILE, &tmv, 0, (int)(tile_id * kBlock), &bars[k]);
        tma_load_2d(stg + TR::KTILE + 128 * 128, &tmv, 64, (int)(tile_id * kBlock), &bars[k]);
      } else {
        mbar_expect_tx(&bars[k], TR::KTILE + TR::VTILE + TR::KSC + TR::VSC);
        bulk_g2s(stg, p.k + tile_id * TR::KTILE, TR::KTILE, &bars[k]);
        bulk_g2s(stg + TR::KTILE, p.v + tile_id * TR::VTILE, TR::VTILE, &bars[k]);
        bulk_g2s(stg + TR::KTILE + TR::VTILE, p.k_sf + tile_id * TR::KSC, TR::KSC, &bars[k]);
        bulk_g2s(stg + TR::KTILE + TR::VTILE + TR::KSC, p.v_sf + tile_id * TR::VSC, TR::VSC, &bars[k]);
      }
    }
  }
  __syncthreads();

  // query fragments and column factors of this (sequence, group)
  uint32_t bq[SP][NT][TR::QKS][2];
  {
    const uint32_t* fr = p.qfrag + (size_t)sg * p.geom.words_per_unit();
#pragma unroll
    for (int sp = 0; sp < SP; ++sp)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int ks = 0; ks < TR::QKS; ++ks)
#pragma unroll
          for (int rg = 0; rg < 2; ++rg)
            bq[sp][nt][ks][rg] = __ldg(fr + ((((sp * NT + nt) * TR::QKS + ks) * 2 + rg) * 32) + lane);
  }
  float colf[NT][2];
  int qlim[NT][2], qbit[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int col = nt * 8 + 2 * j + c;
      colf[nt][c] = __ldg(p.colf + (size_t)sg * NC + col);
      const int qi = col / p.r;
      qlim[nt][c] = (col < cols) ? T - bt.Q + qi : -1;
      qbit[nt][c] = (col < cols) ? qi : 0;
    }

  // running softmax state (log2 domain) and output accumulators O^T[d][col]
  float m_run[NT][2], l_run[NT][2];
  float o[8][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -INFINITY;
    l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
    for (int mm = 0; mm < 8; ++mm) o[mm][nt][0] = o[mm][nt][1] = o[mm][nt][2] = o[mm][nt][3] = 0.f;
  }
  int e_prev = 0;  // FP8: power-of-two scale of the P operand of the previous block
  uint8_t* psm = base + LY::PSM + (size_t)warp * LY::PSM_WARP;
  const int kw = 32 * warp;  // this warp's keys within a block
  bool dead = false;

  for (int k = 0; k < nblk; ++k) {
    if (!state[k]) continue;  // rejected block: nothing was copied, nothing to wait for
    const bool ok = mbar_wait_warp(&bars[k], 0);
    if (!ok) {
      if (lane == 0) raise_flag(p.status, FLAG_TIMEOUT, unit);
      dead = true;
      break;
    }
    const uint8_t* stg = base + (size_t)k * LY::STAGE;
    const int b = p.u_ids[(size_t)sg * p.cap + kb0 + k];
    const uint32_t qmask = p.u_mask[(size_t)sg * p.cap + kb0 + k];
    const int key0 = b * kBlock + kw;

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
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int kk = 16 * mt + g8 + 8 * hh;
          const float vs = vsc[kw + kk] * fe;
          const int pos = p8_pos(kk);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              float hi, lo;
              split_e4m3(sacc[mt][nt][c + 2 * hh] * vs, hi, lo);
              const int col = nt * 8 + 2 * j + c;
              const uint16_t pk = pack_e4m3x2(hi, lo);
              psm[col * 32 + pos] = (uint8_t)(pk & 0xff);
              psm[NC * 32 + col * 32 + pos] = (uint8_t)(pk >> 8);
            }
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

  // ---------------- merge the four warps' partials, write this split's partial
  const bool any_dead = __syncthreads_or(dead);
  if (any_dead) {
    // bounded wait for copies still in flight before their buffers are reused
    if (threadIdx.x == 0)
      for (int k = 0; k < nblk; ++k)
        if (state[k]) mbar_wait(&bars[k], 0, 2000);
    __syncthreads();
  }
  float* om = reinterpret_cast<float*>(base);            // [4][NC][128]
  float* mls = reinterpret_cast<float*>(base) + kWarps * NC * 128;  // [4][NC][2]
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
        for (int hh = 0; hh < 2; ++hh) {
          int d;
          if constexpr (FMT == FMT_FP8)
            d = 16 * ((g8 >> 1) | ((g8 & 1) << 2)) + 2 * mm + hh;
          else
            d = 16 * mm + g8 + 8 * hh;
          om[(warp * NC + col) * 128 + d] = o[mm][nt][c + 2 * hh] * oscale;
        }
    }
  __syncthreads();
  float* po = p.part_o + (size_t)unit * cols * 128;
  for (int idx = threadIdx.x; idx < cols * 128; idx += blockDim.x) {
    const int col = idx >> 7, d = idx & 127;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mls[(w * NC + col) * 2]);
    float acc = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = mls[(w * NC + col) * 2];
        const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
        acc += f * om[(w * NC + col) * 128 + d];
        L += f * mls[(w * NC + col) * 2 + 1];
      }
    }
    po[idx] = acc;
    if (d == 0) {
      pml[2 * col] = M;
      pml[2 * col + 1] = L;
    }
  }
  pdl_launch_dependents();
}

// out[row][h] = sum_k 2^(M_k - M) O_k / sum_k 2^(M_k - M) L_k ; lse in natural log
__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
  pdl_wait();
  const int warp_global = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int H = p.G * p.r;
  const int rows = p.S * p.Q * H;
  if (warp_global >= rows) return;
  const int h = warp_global % H;
  const int sq = warp_global / H;
  const int s = sq / p.Q, i = sq % p.Q;
  const int g = h / p.r, hh = h % p.r;
  const int col = i * p.r + hh;
  const size_t ubase = (size_t)(s * p.G + g) * p.splits;
  float M = -INFINITY;
  for (int k = 0; k < p.splits; ++k) M = fmaxf(M, p.part_ml[((ubase + k) * p.cols + col) * 2]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  if (M != -INFINITY) {
    for (int k = 0; k < p.splits; ++k) {
      const float mk = p.part_ml[((ubase + k) * p.cols + col) * 2];
      if (mk == -INFINITY) continue;
      const float f = exp2f(mk - M);
      L += f * p.part_ml[((ubase + k) * p.cols + col) * 2 + 1];
      const float4 v = *reinterpret_cast<const float4*>(p.part_o + ((ubase + k) * p.cols + col) * 128 + 4 * lane);
      acc.x += f * v.x;
      acc.y += f * v.y;
      acc.z += f * v.z;
      acc.w += f * v.w;
    }
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + ((size_t)sq * H + h) * 128 + 4 * lane;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(out) = pk;
  if (lane == 0 && p.lse) p.lse[(size_t)sq * H + h] = (L > 0.f) ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

template <int FMT, int NT, int SP>
cudaError_t launch_att(const CUtensorMap* tk, const CUtensorMap* tv, const AttendParams& p, cudaStream_t st, bool pdl) {
  const size_t smem = AttLayout<FMT>::SMEM;
  auto kern = attend_kernel<FMT, NT, SP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.batch.S * p.G * p.splits));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
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

int attend_max_stages(int fmt) {
  switch (fmt) {
    case FMT_FP8: return AttTraits<FMT_FP8>::NST;
    case FMT_BF16: return AttTraits<FMT_BF16>::NST;
    default: return AttTraits<FMT_NVFP4>::NST;
  }
}

cudaError_t launch_attend(int fmt, const CUtensorMap* tk, const CUtensorMap* tv, const AttendParams& p,
                          cudaStream_t st, bool pdl) {
  switch (fmt) {
    case FMT_FP8: return launch_att_fmt<FMT_FP8>(tk, tv, p, st, pdl);
    case FMT_BF16: return launch_att_fmt<FMT_BF16>(tk, tv, p, st, pdl);
    case FMT_NVFP4: return launch_att_fmt<FMT_NVFP4>(tk, tv, p, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t st, bool pdl) {
  const int rows = p.S * p.Q * p.G * p.r;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace msa
