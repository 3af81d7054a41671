// Sparse attend over the selected blocks (split-K flash decoding) with the
// split combine folded in.
//
// Definition (vLLM Day-0 blog, section "MSA 入门" and Figure 1): every query
// head of a GQA group attends, with exact softmax, to the keys of the blocks
// its group selected, at most k x 128 keys; logits are scaled by
// head_dim ** -0.5 (model page, MiniMaxM3SparseAttention: self.scaling).  With
// several new tokens per sequence (speculative verify) each token has its own
// selection and causal limit.
//
// Work.  Unit = (sequence, group, split): the group's selected blocks (for
// several query tokens: the union of their selections) cut into splits of
// `bps` blocks.  The grid is persistent.  Each CTA has three roles:
//  - warp 4, producer: takes units from a global counter and streams their K
//    and V tiles (and, with a unit's first block, its query fragments prepared
//    by the preceding kernel) into a ring of shared-memory stages, with TMA
//    tensor copies (128-byte swizzle) for FP8 / BF16 and bulk copies for NVFP4;
//  - warps 0-3, consumers: warp w owns keys [32w, 32w+32) of every block with
//    its own online softmax; at a unit's last block they park (max, sum,
//    output) in a merge slot and go on with the next unit;
//  - warp 5, finalizer: merges the four warps of a slot; an unsplit unit is
//    written as the final bf16 output and LSE, a split unit as a partial, and
//    the CTA that writes the last partial of a (sequence, group) merges all of
//    them by log-sum-exp (no separate combine launch).
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

constexpr int kWarps = 4;             // consumer warps
constexpr int kProducer = 4, kFinalizer = 5;
constexpr int kThreads = 32 * 6;
constexpr int kMergeRow = 132;        // padded row of a merge slot (conflict-free stores)

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

// what the producer tells the consumers about one stage
struct StageMeta {
  int unit;       // -1: no more work
  int k, n;       // block k of the unit's n blocks
  int b;          // logical block id
  uint32_t mask;  // query tokens that selected it
  int ok;         // 1: tiles loaded; 0: rejected block (no data); 2: empty unit (no keys at all)
  int expected;   // partials its (sequence, group) will receive
};

struct SlotHeader {
  int unit, expected, pad0, pad1;
};

__host__ __device__ constexpr size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <int FMT, int NT, int SP>
struct AttLayout {
  using T = AttTraits<FMT>;
  static constexpr int NC = NT * 8;
  static constexpr size_t FRAGW = (size_t)SP * NT * T::QKS * 64 * 4;  // query fragment words
  static constexpr size_t FRAG = FRAGW + NC * 4;                      // + column factors
  static constexpr size_t STAGE = round_up((size_t)T::KTILE + T::VTILE + T::KSC + T::VSC + FRAG, 1024);
  static constexpr int NST = (FMT == FMT_NVFP4) ? (NT == 1 ? 4 : 4) : (NT == 1 ? 2 : (FMT == FMT_FP8 ? 3 : 2));
  static constexpr int MSLOTS = (NT == 1) ? 2 : 1;
  static constexpr size_t PSM = STAGE * NST;                      // per-warp P tiles
  static constexpr size_t PSM_WARP = 64 * NC;
  static constexpr size_t VDQ = PSM + kWarps * PSM_WARP;          // NVFP4 V^T f16 tiles
  static constexpr size_t VDQ_WARP = (FMT == FMT_NVFP4) ? 32 * 256 : 0;
  static constexpr size_t SLOT_F = (size_t)kWarps * NC * (kMergeRow + 2);  // floats per merge slot
  static constexpr size_t MERGE = round_up(VDQ + kWarps * VDQ_WARP, 16);
  static constexpr size_t MERGE_BYTES = MSLOTS * (SLOT_F * 4 + 16);
  static constexpr size_t META = round_up(MERGE + MERGE_BYTES, 16);
  static constexpr size_t BARS = round_up(META + sizeof(StageMeta) * NST, 16);
  static constexpr size_t TOTAL = BARS + 8 * (2 * NST + 2 * MSLOTS) + 16;
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

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int FMT, int NT, int SP>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 2 : 1)
    attend_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const AttendParams p) {
  using TR = AttTraits<FMT>;
  using LY = AttLayout<FMT, NT, SP>;
  constexpr int NC = NT * 8;
  constexpr int NST = LY::NST;
  constexpr int MSLOTS = LY::MSLOTS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  StageMeta* meta = reinterpret_cast<StageMeta*>(base + LY::META);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + LY::BARS);
  uint64_t* empty = full + NST;
  uint64_t* mfull = empty + NST;
  uint64_t* mempty = mfull + MSLOTS;
  auto slot_f = [&](int ms) { return reinterpret_cast<float*>(base + LY::MERGE + ms * (LY::SLOT_F * 4 + 16)); };
  auto slot_h = [&](int ms) {
    return reinterpret_cast<SlotHeader*>(base + LY::MERGE + ms * (LY::SLOT_F * 4 + 16) + LY::SLOT_F * 4);
  };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BatchDev bt = p.batch;
  const int G = p.G, Q = bt.Q;
  const int cols = p.geom.cols;
  const int total_units = bt.S * G * p.splits;

  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kWarps);
    }
    for (int ms = 0; ms < MSLOTS; ++ms) {
      mbar_init(&mfull[ms], kWarps);
      mbar_init(&mempty[ms], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // selections / unions, fragments and counters come from the preceding kernel

  if (warp == kProducer) {
    // ============================== producer
    // Unit facts are fetched by the whole warp (parallel loads), one unit
    // ahead of the one whose blocks lane 0 is issuing.
    if constexpr (FMT != FMT_NVFP4) {
      if (lane == 0) {
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
      }
    }
    struct UnitFacts {
      int unit, sg, s, g, n, count, empty;  // unit < 0: no more work
      int b, phys;                          // lane k < n: block k of the unit
      uint32_t mask;
    };
    auto fetch = [&]() -> UnitFacts {
      UnitFacts f;
      for (;;) {
        int u = 0;
        if (lane == 0) u = atomicAdd(p.work_ctr, 1);
        u = __shfl_sync(0xffffffffu, u, 0);
        f.unit = u;
        if (u >= total_units) {
          f.unit = -1;
          return f;
        }
        const int sg = u / p.splits, split = u % p.splits;
        f.sg = sg;
        f.s = sg / G;
        f.g = sg % G;
        const int T = bt.seq_len(f.s);
        int entry = -1, count;
        if (p.direct) {
          entry = (lane < p.topk) ? p.topk_idx[(size_t)sg * p.topk + lane] : -1;
          count = __popc(__ballot_sync(0xffffffffu, entry >= 0));
        } else {
          count = p.u_count[sg];
        }
        f.count = count;
        const int kb0 = split * p.bps;
        f.n = min(p.bps, count - kb0);
        f.empty = (count == 0 && split == 0);
        if (f.n <= 0 && !f.empty) continue;  // nothing in this split: take the next unit
        if (f.empty) f.n = 1;
        f.b = -1;
        f.mask = 0;
        f.phys = -1;
        if (!f.empty) {
          int b;
          if (p.direct) {
            b = __shfl_sync(0xffffffffu, entry, (kb0 + lane) & 31);
            f.mask = 1u;
          } else {
            b = (lane < f.n) ? p.u_ids[(size_t)sg * p.cap + kb0 + lane] : -1;
            f.mask = (lane < f.n) ? p.u_mask[(size_t)sg * p.cap + kb0 + lane] : 0u;
          }
          if (lane < f.n) {
            if (b < 0 || b > (T - 1) / kBlock) {
              raise_flag(p.status, FLAG_BAD_SELECT, b);
              b = -1;
            } else {
              const int ph = bt.row(f.s)[b];
              if (ph < 0 || ph >= p.num_blocks) raise_flag(p.status, FLAG_BAD_BLOCK, ph);
              else f.phys = ph;
            }
          }
          f.b = b;
        }
        return f;
      }
    };
    int st = 0;
    long issued = 0;
    bool abort = false;
    auto acquire = [&]() -> bool {  // lane 0: wait until stage st is free
      if (issued >= NST) {
        const uint32_t par = (uint32_t)(((issued / NST) - 1) & 1);
        if (!mbar_wait(&empty[st], par)) {
          raise_flag(p.status, FLAG_TIMEOUT, -1);
          return false;
        }
      }
      return true;
    };
    UnitFacts nxt = fetch();
    while (nxt.unit >= 0 && !abort) {
      const UnitFacts cur = nxt;
      nxt = fetch();  // next unit's loads overlap this unit's issue
      const int expected = cur.empty ? 1 : (cur.count + p.bps - 1) / p.bps;
      for (int k = 0; k < cur.n; ++k) {
        const int b = __shfl_sync(0xffffffffu, cur.b, k);
        const int phys = __shfl_sync(0xffffffffu, cur.phys, k);
        const uint32_t mask = __shfl_sync(0xffffffffu, cur.mask, k);
        if (lane == 0) {
          if (!acquire()) abort = true;
          if (!abort) {
            StageMeta m;
            m.unit = cur.unit;
            m.k = k;
            m.n = cur.n;
            m.b = b;
            m.mask = mask;
            m.ok = cur.empty ? 2 : (phys >= 0 ? 1 : 0);
            m.expected = expected;
            meta[st] = m;
            uint8_t* stg = base + (size_t)st * LY::STAGE;
            const bool frag = (k == 0 && !cur.empty);
            uint32_t bytes = frag ? (uint32_t)LY::FRAG : 0u;
            if (m.ok == 1) bytes += TR::KTILE + TR::VTILE + TR::KSC + TR::VSC;
            if (bytes == 0) {
              mbar_arrive(&full[st]);  // nothing to copy: a plain arrive completes the phase
            } else {
              fence_proxy_async();
              mbar_expect_tx(&full[st], bytes);
              if (frag) {
                uint8_t* fd = stg + TR::KTILE + TR::VTILE + TR::KSC + TR::VSC;
                bulk_g2s(fd, p.frag + (size_t)cur.sg * (LY::FRAGW / 4), (uint32_t)LY::FRAGW, &full[st]);
                bulk_g2s(fd + LY::FRAGW, p.colf + (size_t)cur.sg * NC, NC * 4, &full[st]);
              }
              if (m.ok == 1) {
                const size_t tile_id = (size_t)phys * G + cur.g;
                if constexpr (FMT == FMT_FP8) {
                  tma_load_2d(stg, &tmk, 0, (int)(tile_id * kBlock), &full[st]);
                  tma_load_2d(stg + TR::KTILE, &tmv, 0, (int)(tile_id * kBlock), &full[st]);
                  bulk_g2s(stg + TR::KTILE + TR::VTILE, p.k_scale + tile_id * kBlock, TR::KSC, &full[st]);
                  bulk_g2s(stg + TR::KTILE + TR::VTILE + TR::KSC, p.v_scale + tile_id * kBlock, TR::VSC, &full[st]);
                } else if constexpr (FMT == FMT_BF16) {
                  tma_load_2d(stg, &tmk, 0, (int)(tile_id * kBlock), &full[st]);
                  tma_load_2d(stg + 128 * 128, &tmk, 64, (int)(tile_id * kBlock), &full[st]);
                  tma_load_2d(stg + TR::KTILE, &tmv, 0, (int)(tile_id * kBlock), &full[st]);
                  tma_load_2d(stg + TR::KTILE + 128 * 128, &tmv, 64, (int)(tile_id * kBlock), &full[st]);
                } else {
                  bulk_g2s(stg, p.k + tile_id * TR::KTILE, TR::KTILE, &full[st]);
                  bulk_g2s(stg + TR::KTILE, p.v + tile_id * TR::VTILE, TR::VTILE, &full[st]);
                  bulk_g2s(stg + TR::KTILE + TR::VTILE, p.k_sf + tile_id * TR::KSC, TR::KSC, &full[st]);
                  bulk_g2s(stg + TR::KTILE + TR::VTILE + TR::KSC, p.v_sf + tile_id * TR::VSC, TR::VSC, &full[st]);
                }
              }
            }
          }
        }
        abort = __shfl_sync(0xffffffffu, abort ? 1 : 0, 0) != 0;
        if (abort) break;
        st = (st + 1 == NST) ? 0 : st + 1;
        ++issued;
      }
    }
    if (lane == 0 && !abort && acquire()) {
      StageMeta m;
      m.unit = -1;
      m.k = m.n = m.b = 0;
      m.mask = 0;
      m.ok = 0;
      m.expected = 0;
      meta[st] = m;
      mbar_arrive(&full[st]);
    }
    pdl_launch_dependents();
    return;
  }

  if (warp == kFinalizer) {
    // ============================== finalizer
    const int H = G * p.r;
    for (int nfin = 0;; ++nfin) {
      const int ms = nfin % MSLOTS;
      if (!mbar_wait_warp(&mfull[ms], (uint32_t)((nfin / MSLOTS) & 1))) {
        if (lane == 0) raise_flag(p.status, FLAG_TIMEOUT, blockIdx.x);
        return;
      }
      const SlotHeader hd = *slot_h(ms);
      if (hd.unit < 0) return;
      const float* om = slot_f(ms);                         // [4][NC][kMergeRow]
      const float* mls = om + (size_t)kWarps * NC * kMergeRow;  // [4][NC][2]
      const int sg = hd.unit / p.splits;
      const int s = sg / G, g = sg % G;
      const bool whole = (p.splits == 1);
      float* po = p.part_o + (size_t)hd.unit * cols * 128;
      float* pml = p.part_ml + (size_t)hd.unit * cols * 2;
      for (int idx = lane; idx < cols * 128; idx += 32) {
        const int col = idx >> 7, d = idx & 127;
        int slot;  // merge-slot position of output dim d (inverse of the accumulator row mapping)
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
      __syncwarp();
      if (lane == 0) mbar_arrive(&mempty[ms]);  // the slot is free again
      if (whole) continue;
      __threadfence();
      int last = 0;
      if (lane == 0) last = (atomicAdd(p.sg_ctr + sg, 1) == hd.expected - 1);
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) continue;
      // ---------------- last partial of this (sequence, group): LSE merge of its splits
      __threadfence();
      const int nparts = hd.expected;
      const size_t ubase = (size_t)sg * p.splits;
      for (int col = 0; col < cols; ++col) {
        float M = -INFINITY;
        for (int k = 0; k < nparts; ++k) M = fmaxf(M, __ldcg(p.part_ml + ((ubase + k) * cols + col) * 2));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float L = 0.f;
        if (M != -INFINITY) {
          for (int k = 0; k < nparts; ++k) {
            const float mk = __ldcg(p.part_ml + ((ubase + k) * cols + col) * 2);
            if (mk == -INFINITY) continue;
            const float f = exp2f(mk - M);
            L += f * __ldcg(p.part_ml + ((ubase + k) * cols + col) * 2 + 1);
            const float4 v = __ldcg(reinterpret_cast<const float4*>(p.part_o + ((ubase + k) * cols + col) * 128) + lane);
            acc.x += f * v.x;
            acc.y += f * v.y;
            acc.z += f * v.z;
            acc.w += f * v.w;
          }
        }
        const float inv = (L > 0.f) ? 1.f / L : 0.f;
        const int qi = col / p.r, hh = col % p.r;
        const size_t orow = (size_t)(s * Q + qi) * H + g * p.r + hh;
        __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out) + orow * 128 + 4 * lane;
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo);
        pk.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(outp) = pk;
        if (lane == 0 && p.lse) p.lse[orow] = (L > 0.f) ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
      }
      if (lane == 0) p.sg_ctr[sg] = 0;  // ready for the next call
    }
  }

  // ============================== consumers (warps 0-3)
  const int g8 = lane >> 2, j = lane & 3;
  const int kw = 32 * warp;  // this warp's keys within a block
  uint8_t* psm = base + LY::PSM + (size_t)warp * LY::PSM_WARP;

  uint32_t bq[SP][NT][TR::QKS][2];
  float colf[NT][2];
  int qlim[NT][2], qbit[NT][2];
  float m_run[NT][2], l_run[NT][2];
  float o[8][NT][4];
  int e_prev = 0;
  int cur_unit = -1, T = 0;
  uint32_t full_bits = 0;
  int st = 0, nunits = 0;

  for (;;) {
    if (!mbar_wait_warp(&full[st], (full_bits >> st) & 1u)) {
      if (lane == 0) raise_flag(p.status, FLAG_TIMEOUT, blockIdx.x);
      break;
    }
    full_bits ^= 1u << st;
    const StageMeta mt_ = meta[st];
    const uint8_t* stg = base + (size_t)st * LY::STAGE;
    if (mt_.unit < 0) break;
    if (mt_.unit != cur_unit) {
      // ---------------- a new unit: its query fragments (copied with this stage) and a fresh softmax state
      cur_unit = mt_.unit;
      const int sg = cur_unit / p.splits;
      T = bt.seq_len(sg / G);
      if (mt_.ok != 2) {
        const uint32_t* fr = reinterpret_cast<const uint32_t*>(stg + TR::KTILE + TR::VTILE + TR::KSC + TR::VSC);
        const float* cf = reinterpret_cast<const float*>(stg + TR::KTILE + TR::VTILE + TR::KSC + TR::VSC + LY::FRAGW);
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
      e_prev = 0;
    }
    if (mt_.ok == 1) {
      const uint32_t qmask = mt_.mask;
      const int key0 = mt_.b * kBlock + kw;
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
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    st = (st + 1 == NST) ? 0 : st + 1;

    if (mt_.k == mt_.n - 1) {
      // ---------------- the unit's last block: park this warp's state in a merge slot
      const int ms = nunits % MSLOTS;
      if (nunits >= MSLOTS && !mbar_wait_warp(&mempty[ms], (uint32_t)(((nunits / MSLOTS) - 1) & 1))) {
        if (lane == 0) raise_flag(p.status, FLAG_TIMEOUT, blockIdx.x);
        break;
      }
      float* om = slot_f(ms);
      float* mls = om + (size_t)kWarps * NC * kMergeRow;
      const float oscale = (FMT == FMT_FP8) ? ldexpf(1.f, -e_prev) : ((FMT == FMT_NVFP4) ? p.v_global : 1.f);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col = nt * 8 + 2 * j + c;
          if (g8 == 0) {
            mls[(warp * NC + col) * 2] = m_run[nt][c];
            mls[(warp * NC + col) * 2 + 1] = l_run[nt][c];
          }
#pragma unroll
          for (int mm = 0; mm < 8; ++mm)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
              om[(warp * NC + col) * kMergeRow + 16 * mm + 8 * hh + g8] = o[mm][nt][c + 2 * hh] * oscale;
        }
      if (warp == 0 && lane == 0) {
        SlotHeader* h = slot_h(ms);
        h->unit = cur_unit;
        h->expected = mt_.expected;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&mfull[ms]);
      ++nunits;
    }
  }
  // no more units: tell the finalizer
  {
    const int ms = nunits % MSLOTS;
    if (nunits < MSLOTS || mbar_wait_warp(&mempty[ms], (uint32_t)(((nunits / MSLOTS) - 1) & 1))) {
      if (warp == 0 && lane == 0) slot_h(ms)->unit = -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&mfull[ms]);
    }
  }
  pdl_launch_dependents();
}

template <int FMT, int NT, int SP>
cudaError_t launch_att(const CUtensorMap* tk, const CUtensorMap* tv, const AttendParams& p, int num_sms,
                       cudaStream_t st, bool pdl) {
  const size_t smem = AttLayout<FMT, NT, SP>::SMEM;
  auto kern = attend_kernel<FMT, NT, SP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int units = p.batch.S * p.G * p.splits;
  const int grid = units < num_sms * per_sm ? units : num_sms * per_sm;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
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
