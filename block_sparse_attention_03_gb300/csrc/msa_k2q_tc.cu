// Key-block-major attend of prefill chunks on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory).
//
// What it computes (vLLM Day-0 blog, section "MSA 入门"): for every
// (token, head, slot) whose selected block b the token may see, the
// unnormalised softmax partial of the token's query against the block's keys
// t <= pos(token):
//   m = max_t x_t,  l = sum_t 2^(x_t - m),  o = sum_t 2^(x_t - m) v_t,
//   x_t = (q . k_t) * kscale_t * head_dim^-0.5 * log2(e),
// stored as (o / l in fp16 x 2^-ev, m, l, 2^ev); k2q_combine merges a token's
// slots by log-sum-exp (msa_k2q.cu).  The selection is inverted into lists
// (sequence, group, block) of (token, slot) entries, the key -> query CSR of
// the vLLM MiniMax-M3 model page ("vllm.models.minimax_m3.nvidia.model",
// build_k2q_csr), so that each item reads its block's K/V tile once for up to
// 128 / r tokens.
//
// Item = up to 128 / r entries of one list, as 128 MMA rows (entry, head):
//   S[128 x 128 keys] = Qop[128 x 128 dims] . K^T    (MMA 1: A, B in shared memory, K-major)
//   O[128 x 128 dims] = P[128 x 128 keys] . V        (MMA 2: A = P in TMEM, B = V MN-major)
// kind::f8f6f4, e4m3 x e4m3, fp32 accumulators in TMEM.  A bf16 query enters
// as two e4m3 terms (hi + lo, after a power-of-two scale per row, prepared
// once per (token, head) by the count pass); an e4m3 query as one.  P enters as
// hi + lo e4m3 terms of p * 2^e * vscale_t (2^e puts the block's largest V
// scale at most at 448), so that V's per-token scales fold into P; 2^e rides
// in the exponent of p, and l is summed at the same scale, so that o / l needs
// no further factor.  P is written into the S columns already read (hi and lo
// of each 32-key chunk side by side), where MMA 2 takes its A operand.
//
// One CTA per SM (all 512 TMEM columns), 9 warps:
//   warp 0     writes item headers (list facts, the entries by bulk copy) into
//              an 8-slot ring two items ahead of the K / V tiles, which it
//              copies (TMA, 128-byte swizzle, with the per-token scales) into a
//              4-stage ring; the facts of 32 items at a time are read by its 32
//              lanes together; it owns TMEM;
//   warps 1-4  group 0 and warps 5-8 group 1 take alternate items; each
//              thread owns one MMA row (TMEM lane).  Once its item's logits are
//              in TMEM a group starts the copies of its next item's query rows
//              (cp.async, a warp's 32 rows together, whole rows per
//              instruction) into the operand buffer MMA 1 has finished with,
//              turns S into P (max, exp2, sum, V scales, hi / lo split), and
//              its leader thread issues MMA 2; when O is ready the leader
//              issues the next item's MMA 1, and the group writes this item's
//              output: fp16 rows staged in the item's (now free) stage, one
//              bulk copy per entry (its r heads are adjacent in the partials),
//              after which the group's threads release the stage.  S (then P)
//              and O take 128 columns each per group.
// Every wait is bounded; a wait that gives up sets the timeout flag and the
// CTA stops issuing, drains what it issued and frees its TMEM.
#include "msa_device.cuh"
#include "msa_internal.h"
#include "msa_tcgen05.cuh"

namespace msa {

namespace {

constexpr int kTqStages = 4;               // K / V stages (two per group)
constexpr int kTqHdrs = 8;                 // header slots
constexpr int kTqAhead = 2;                // headers written this many items before their tiles
constexpr int kTqThreads = 288;
constexpr uint32_t kTqTile = 128 * 128;    // one e4m3 128 x 128 operand
constexpr uint32_t kTqScales = 128 * 4;
constexpr uint32_t kTqEnt = 136 * 4;       // an item's entries, copied from a 16-byte boundary
constexpr uint32_t kTqHdrW = 8;            // header words

constexpr uint32_t tq_round(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

struct TqLayout {
  static constexpr uint32_t OP = 0;                          // [group][hi, lo][16 KB] query operand
  static constexpr uint32_t ST = OP + 4 * kTqTile;           // the ring of stages
  static constexpr uint32_t S_K = 0, S_V = kTqTile, S_KS = 2 * kTqTile, S_VS = S_KS + kTqScales;
  // the output rows of an item, staged after MMA 2: 128 / r entries of r rows
  // of 256 bytes, 16 r bytes apart; with the rows' 16-byte chunks swizzled by
  // head (as in the partials) a warp's stores fall in different banks
  static constexpr uint32_t STAGE = tq_round(S_VS + kTqScales + 2048, 1024);
  static constexpr uint32_t HD = ST + kTqStages * STAGE;     // header slots: entries, then words
  static constexpr uint32_t HSLOT = kTqEnt + kTqHdrW * 4;
  static constexpr uint32_t BARS = tq_round(HD + kTqHdrs * HSLOT, 16);
  // kvfull[stages], kvempty[stages], hfull[slots], hempty[slots], sbar[2], obar[2], done[2]
  static constexpr uint32_t NBARS = 2 * kTqStages + 2 * kTqHdrs + 6;
  static constexpr uint32_t TSLOT = BARS + NBARS * 8;
  static constexpr uint32_t DEAD = TSLOT + 4;
  static constexpr uint32_t TOTAL = DEAD + 12;
  static constexpr uint32_t SMEM = TOTAL + 1024;             // 1024-byte alignment slack
};
static_assert(TqLayout::STAGE >= 32768 + 128 * 16, "an item's output rows fit its stage");

// Instruction descriptors: D fp32, A and B e4m3, M = N = 128, A K-major; B
// K-major (keys, MMA 1) or MN-major (V with the head dims contiguous, MMA 2).
constexpr uint32_t kIdescQK = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescPV = kIdescQK | (1u << 16);

// D (TMEM) = / += A (TMEM, K-major rows = lanes) x B (smem)^T, e4m3, fp32 accumulate.
__device__ __forceinline__ void mma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 8 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// 16-byte global -> shared copy (zero fill when !ok), completed by cp_async_wait.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(ok ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float tq_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (a, b) as two e4m3 terms, hi + lo, through f16 (a in the low byte of each):
// hi = f16(x) rounded to 3 mantissa bits by an integer add and mask (ties away
// from zero; exact in e4m3 from 2^-6 up, below which the conversion rounds it
// once more, to e4m3's subnormal step 2^-9), lo = e4m3(f16(x) - hi), the
// difference exact in f16.  |x| <= 448, so no half carries into the other.
__device__ __forceinline__ void split2_e4m3(float a, float b, uint32_t& hi, uint32_t& lo) {
  const uint32_t h2 = pack_f16x2(a, b);
  const uint32_t t2 = (h2 + 0x00400040u) & 0xff80ff80u;
  uint16_t h8, l8;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(h8) : "r"(t2));
  const __half2 d = __hsub2(*reinterpret_cast<const __half2*>(&h2), *reinterpret_cast<const __half2*>(&t2));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(l8) : "r"(*reinterpret_cast<const uint32_t*>(&d)));
  hi = h8;
  lo = l8;
}

// This thread's row of an item.
struct TqRow {
  int hs;       // header slot
  int st;       // K / V stage
  int valid;    // the row holds a real (entry, head)
  int pos;      // last key the row's token may see (-1: none)
  int key0;     // the block's first key
  int qrow;     // (token, head) query row
  long part;    // (token, slot, head) partial
};

__global__ void __launch_bounds__(kTqThreads, 1) k2q_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                                                             const __grid_constant__ CUtensorMap tmv,
                                                             const K2qParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using LY = TqLayout;
  uint64_t* kvfull = reinterpret_cast<uint64_t*>(base + LY::BARS);
  uint64_t* kvempty = kvfull + kTqStages;
  uint64_t* hfull = kvempty + kTqStages;
  uint64_t* hempty = hfull + kTqHdrs;
  uint64_t* sbar = hempty + kTqHdrs;
  uint64_t* obar = sbar + 2;
  uint64_t* done = obar + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(base + LY::TSLOT);
  int* dead = reinterpret_cast<int*>(base + LY::DEAD);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const BatchDev bt = p.batch;
  const int G = p.G, r = p.r, H = G * r, K = p.topk, Q = bt.Q;
  const int TPI = p.item_tokens;  // 128 / r
  const int lr = __ffs(r) - 1;
  const long L = (long)bt.S * G * bt.max_nb;
  const int items = p.item_off[L];
  const int i0 = (int)((long)blockIdx.x * items / gridDim.x);
  const int nj = (int)((long)(blockIdx.x + 1) * items / gridDim.x) - i0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTqStages; ++i) {
      mbar_init(&kvfull[i], 1);
      mbar_init(&kvempty[i], 128);  // the item's group, thread by thread
    }
    for (int i = 0; i < kTqHdrs; ++i) {
      mbar_init(&hfull[i], 1);
      mbar_init(&hempty[i], 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sbar[i], 1);
      mbar_init(&obar[i], 1);
      mbar_init(&done[i], 1);
    }
    *dead = 0;
    fence_mbar_init();
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  if (warp == 0) tmem_alloc(smem_u32(tslot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    // ---------------- headers, then (kTqAhead items later) tiles.  Step t
    // writes header t and copies the tiles of item t - kTqAhead; the tile
    // step reads the item's block from its header slot, which the producer
    // alone writes and does not reuse before header t - kTqAhead + kTqHdrs.
    int issued_h = 0, issued_k = 0;
    bool ok = true;
    auto fail = [&](int where) {
      if (!*reinterpret_cast<volatile int*>(dead)) raise_flag(p.status, FLAG_TIMEOUT, where);
      *reinterpret_cast<volatile int*>(dead) = 1;
      ok = false;
    };
    for (int t0 = 0; t0 < nj + kTqAhead && ok; t0 += 32) {
      int f_n = 0, f_s = 0, f_g = 0, f_b = 0, f_T = 0, f_e0 = 0, f_ph = -1;
      if (t0 + lane < nj) {
        const int it = i0 + t0 + lane;
        const int list = p.item_list[it];
        const int off = p.off[list];
        f_e0 = off + (it - p.item_off[list]) * TPI;
        f_n = min(TPI, off + p.cnt[list] - f_e0);
        f_s = (int)(list / ((long)G * bt.max_nb));
        f_g = (int)((list / bt.max_nb) % G);
        f_b = (int)(list % bt.max_nb);
        f_T = bt.seq_len(f_s);
        f_ph = bt.row(f_s)[f_b];
      }
      for (int t = 0; t < 32 && t0 + t < nj + kTqAhead; ++t) {
        const int n = __shfl_sync(0xffffffffu, f_n, t), s = __shfl_sync(0xffffffffu, f_s, t);
        const int g = __shfl_sync(0xffffffffu, f_g, t), b = __shfl_sync(0xffffffffu, f_b, t);
        const int T = __shfl_sync(0xffffffffu, f_T, t), e0 = __shfl_sync(0xffffffffu, f_e0, t);
        const int ph = __shfl_sync(0xffffffffu, f_ph, t);
        const int jh = t0 + t, jk = jh - kTqAhead;
        if (lane == 0) {
          if (jh < nj) {  // header jh
            const int hs = jh % kTqHdrs;
            if (jh >= kTqHdrs && (*reinterpret_cast<volatile int*>(dead) ||
                                  !mbar_wait_sleep(&hempty[hs], (uint32_t)(((jh / kTqHdrs) - 1) & 1)))) {
              fail(24);
            } else {
              uint8_t* hb = base + LY::HD + (size_t)hs * LY::HSLOT;
              int32_t* hw = reinterpret_cast<int32_t*>(hb + kTqEnt);
              const bool okb = ph >= 0 && ph < p.num_blocks && n > 0;
              if (!okb && n > 0) raise_flag(p.status, FLAG_BAD_BLOCK, ph);
              const int ea = e0 & ~3, nent = n > 0 ? n : 0;
              const uint32_t ebytes = (uint32_t)((e0 - ea + nent + 3) & ~3) * 4u;
              hw[0] = okb ? n : -nent;  // negative: the block is rejected, its entries get empty partials
              hw[1] = s;
              hw[2] = g;
              hw[3] = b;
              hw[4] = T;
              hw[5] = e0 - ea;
              hw[6] = okb ? (int)(((long)ph * G + g) * kBlock) : -1;  // the tile's first row
              fence_proxy_async();
              mbar_expect_tx(&hfull[hs], ebytes);
              if (ebytes > 0) bulk_g2s(hb, p.entries + ea, ebytes, &hfull[hs]);
              issued_h = jh + 1;
            }
          }
          if (ok && jk >= 0) {  // tiles of item jk
            const int st = jk % kTqStages;
            if (jk >= kTqStages && (*reinterpret_cast<volatile int*>(dead) ||
                                    !mbar_wait_sleep(&kvempty[st], (uint32_t)(((jk / kTqStages) - 1) & 1)))) {
              fail(20);
            } else {
              const int tile = reinterpret_cast<const int32_t*>(base + LY::HD + (size_t)(jk % kTqHdrs) * LY::HSLOT +
                                                                kTqEnt)[6];
              uint8_t* sb = base + LY::ST + (size_t)st * LY::STAGE;
              fence_proxy_async();
              if (tile >= 0) {
                mbar_expect_tx(&kvfull[st], 2 * kTqTile + 2 * kTqScales);
                tma_load_2d(sb + LY::S_K, &tmk, 0, tile, &kvfull[st]);
                tma_load_2d(sb + LY::S_V, &tmv, 0, tile, &kvfull[st]);
                bulk_g2s(sb + LY::S_KS, p.k_scale + tile, kTqScales, &kvfull[st]);
                bulk_g2s(sb + LY::S_VS, p.v_scale + tile, kTqScales, &kvfull[st]);
              } else {
                mbar_arrive(&kvfull[st]);  // a rejected block: nothing to copy
              }
              issued_k = jk + 1;
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
    }
    // a CTA that gave up waits (bounded) for the copies it issued
    if (lane == 0 && !ok) {
      for (int i = 0; i < kTqHdrs && i < issued_h; ++i) {
        const int jj = issued_h - 1 - i;
        mbar_wait_sleep(&hfull[jj % kTqHdrs], (uint32_t)((jj / kTqHdrs) & 1), 2000);
      }
      for (int i = 0; i < kTqStages && i < issued_k; ++i) {
        const int jj = issued_k - 1 - i;
        mbar_wait_sleep(&kvfull[jj % kTqStages], (uint32_t)((jj / kTqStages) & 1), 2000);
      }
    }
  } else {
    // ---------------- two groups of four warps, thread = MMA row
    const int grp = (warp - 1) >> 2;
    const int quarter = warp & 3;  // TMEM lanes 32 * quarter .. + 31
    const int m = 32 * quarter + lane;
    const bool leader = ((warp - 1) & 3) == 0 && lane == 0;
    const int bar_id = 1 + grp;
    uint8_t* op = base + LY::OP + (size_t)grp * 2 * kTqTile;
    const uint32_t op_s = smem_u32(op);
    const uint32_t tS = tmem + 256u * (uint32_t)grp, tO = tS + 128u;
    const uint32_t lsel = (uint32_t)(32 * quarter) << 16;
    const int terms = p.q_fp8 ? 1 : 2;
    const float qconst = p.q_scale * p.col_const;  // an e4m3 query's row factor
    const int hh = m & (r - 1);                     // this row's head within the group
    const uint32_t epitch = (uint32_t)r * 272u;     // staged output rows: bytes per entry

    // every thread of the group waits; the group agrees on the outcome
    auto gwait = [&](uint64_t* bar, uint32_t par, int where) -> bool {
      const bool ok = !*reinterpret_cast<volatile int*>(dead) && mbar_wait_sleep(bar, par);
      const bool bad = named_bar_or(bar_id, 128, !ok);
      if (bad && leader && !*reinterpret_cast<volatile int*>(dead)) {
        *reinterpret_cast<volatile int*>(dead) = 1;
        raise_flag(p.status, FLAG_TIMEOUT, where);
      }
      return !bad;
    };

    // Item j's header and this thread's row of it; for a real block, the
    // copies of the row's query into the operand buffer are started (the
    // warp's 32 rows together: two bf16-split rows of 256 bytes, or four e4m3
    // rows of 128, per instruction, each chunk straight to its swizzled
    // place).  Rejected items (block outside the cache) get empty partials and
    // release their header slot and stage here; the walk moves on to the
    // group's next item.  Returns the item taken, or nj.
    float rowf_n = 0.f;
    auto take = [&](int j, TqRow& rw) -> int {
      for (; j < nj; j += 2) {
        const int hs = j % kTqHdrs;
        if (!gwait(&hfull[hs], (uint32_t)((j / kTqHdrs) & 1), 21)) return nj;
        const uint8_t* hb = base + LY::HD + (size_t)hs * LY::HSLOT;
        const int32_t* hw = reinterpret_cast<const int32_t*>(hb + kTqEnt);
        const int n = hw[0], s = hw[1], g = hw[2], b = hw[3], T = hw[4], delta = hw[5];
        const int nr = (n < 0 ? -n : n) * r;
        rw.hs = hs;
        rw.st = j % kTqStages;
        rw.valid = m < nr;
        rw.key0 = b * kBlock;
        const int ent = rw.valid ? reinterpret_cast<const int32_t*>(hb)[delta + (m >> lr)] : 0;
        const long token = ent >> 5;
        const int head = g * r + hh;
        rw.part = (token * K + (ent & 31)) * H + head;
        rw.qrow = (int)(token * H + head);
        rw.pos = rw.valid ? T - Q + (int)(token - (long)s * Q) : -1;
        mbar_arrive(&hempty[hs]);  // the header is in registers
        if (n > 0) {
          uint8_t* wrows = op + (size_t)(32 * quarter) * 128;  // the warp's 32 operand rows
          if (p.q_fp8) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rho = 4 * i + (lane >> 3), c = lane & 7;
              const int qr = __shfl_sync(0xffffffffu, rw.qrow, rho);
              const int vd = __shfl_sync(0xffffffffu, rw.valid, rho);
              cp_async16(wrows + rho * 128 + ((c ^ (rho & 7)) << 4),
                         static_cast<const uint8_t*>(p.q) + (long)(vd ? qr : 0) * 128 + 16 * c, vd != 0);
            }
            rowf_n = rw.valid ? qconst : 0.f;
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int rho = 2 * i + (lane >> 4), c = lane & 15;
              const int qr = __shfl_sync(0xffffffffu, rw.qrow, rho);
              const int vd = __shfl_sync(0xffffffffu, rw.valid, rho);
              cp_async16(wrows + (c >> 3) * kTqTile + rho * 128 + (((c & 7) ^ (rho & 7)) << 4),
                         p.qsplit + (long)(vd ? qr : 0) * 256 + 16 * c, vd != 0);
            }
            rowf_n = rw.valid ? __ldg(p.qrowf + rw.qrow) : 0.f;
          }
          cp_async_commit();
          return j;
        }
        if (rw.valid) reinterpret_cast<float4*>(p.part_ml)[rw.part] = make_float4(-INFINITY, 0.f, 1.f, 0.f);
        mbar_arrive(&kvempty[rw.st]);  // no tiles to read: the stage goes straight back
      }
      return nj;
    };

    // the query operand is in place and the item's tiles are in: MMA 1
    auto start = [&](const TqRow& rw, int j) -> bool {
      cp_async_wait();
      fence_proxy_async();  // the MMA reads the operand through the async proxy
      tc_fence_before();
      if (!gwait(&kvfull[rw.st], (uint32_t)((j / kTqStages) & 1), 25)) return false;
      if (leader) {
        tc_fence_after();
        const uint32_t kt = smem_u32(base + LY::ST + (size_t)rw.st * LY::STAGE + LY::S_K);
#pragma unroll 1
        for (int term = 0; term < terms; ++term)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f8(tS, sw128_desc(op_s + term * kTqTile + 32 * k), sw128_desc(kt + 32 * k), kIdescQK,
                   (term | k) != 0);
        mma_commit(&sbar[grp]);
      }
      return true;
    };

    TqRow cur, nxt;
    int u = 0;  // items of this group whose MMAs ran (phases of sbar / obar)
    int j = take(grp, cur);
    float rowf = rowf_n;
    if (j < nj && !start(cur, j)) j = nj;
#pragma unroll 1
    while (j < nj) {
      if (!gwait(&sbar[grp], (uint32_t)(u & 1), 22)) break;
      tc_fence_after();
      // MMA 1 is done with the operand buffer: the next item's query rows go in
      const int jn = take(j + 2, nxt);
      const uint8_t* sb = base + LY::ST + (size_t)cur.st * LY::STAGE;
      const float* ks = reinterpret_cast<const float*>(sb + LY::S_KS);
      const float* vs = reinterpret_cast<const float*>(sb + LY::S_VS);
      // P's scale 2^e puts the block's largest V scale at most at 448 (2^e at
      // most 2^100, so that l cannot overflow); the fp16 partial o / l, at most
      // max |v| <= 448 x that scale, is brought under 32768 by 2^-ev
      float vmx = fmaxf(fmaxf(vs[lane], vs[lane + 32]), fmaxf(vs[lane + 64], vs[lane + 96]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) vmx = fmaxf(vmx, __shfl_xor_sync(0xffffffffu, vmx, o));
      const int e = min(100, fit448(vmx));
      int ev = 0;
      if (448.f * vmx > 32768.f) frexpf(448.f * vmx * (1.f / 32768.f), &ev);
      const bool full = cur.key0 + kBlock - 1 <= cur.pos;  // every key visible
      // ---- the row's max of s_t * kscale_t over its visible keys
      float mx = -INFINITY;
#pragma unroll 1
      for (int h = 0; h < 4; ++h) {
        float v[32];
        tmem_ld32(tS + lsel + 32 * h, v);
        tmem_ld_wait();
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        const int n0 = 32 * h;
        if (full) {
          const float4* k4 = reinterpret_cast<const float4*>(ks + n0);
#pragma unroll
          for (int n = 0; n < 32; n += 8) {
            const float4 ka = k4[n >> 2], kb = k4[(n >> 2) + 1];
            const float2 p0 = mul2(v[n], v[n + 1], ka.x, ka.y);
            const float2 p1 = mul2(v[n + 2], v[n + 3], ka.z, ka.w);
            const float2 p2 = mul2(v[n + 4], v[n + 5], kb.x, kb.y);
            const float2 p3 = mul2(v[n + 6], v[n + 7], kb.z, kb.w);
            m4[0] = max3(m4[0], p0.x, p0.y);
            m4[1] = max3(m4[1], p1.x, p1.y);
            m4[2] = max3(m4[2], p2.x, p2.y);
            m4[3] = max3(m4[3], p3.x, p3.y);
          }
        } else {
#pragma unroll
          for (int n = 0; n < 32; ++n) {
            const float sc = (cur.key0 + n0 + n <= cur.pos) ? v[n] * ks[n0 + n] : -INFINITY;
            m4[n & 3] = fmaxf(m4[n & 3], sc);
          }
        }
        mx = fmaxf(mx, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
      }
      const float m2 = mx * rowf;  // base-2 logit maximum (rowf > 0)
      // p_t 2^e = 2^(x_t - m + e): the exponent's offset, -inf rows kept at 0
      const float c0 = (mx == -INFINITY) ? 0.f : (float)e - m2;
      // ---- P'_t = p_t 2^e vscale_t as e4m3 hi + lo into the S columns read
      // (chunk h of 32 keys: hi at column 16h, lo at 16h + 8), l 2^e = sum p_t 2^e
      float l0 = 0.f, l1 = 0.f;
#pragma unroll 1
      for (int h = 0; h < 4; ++h) {
        float v[32];
        tmem_ld32(tS + lsel + 32 * h, v);
        tmem_ld_wait();
        const int n0 = 32 * h;
        uint32_t hw[8], lw[8];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {  // keys n0 + 4 q4 .. + 3: one word of each term
          const int n = n0 + 4 * q4;
          const float4 k4 = *reinterpret_cast<const float4*>(ks + n);
          const float4 v4 = *reinterpret_cast<const float4*>(vs + n);
          const float2 ta = mul2(v[4 * q4], v[4 * q4 + 1], k4.x, k4.y);
          const float2 tb = mul2(v[4 * q4 + 2], v[4 * q4 + 3], k4.z, k4.w);
          float x0 = fmaf(ta.x, rowf, c0), x1 = fmaf(ta.y, rowf, c0);
          float x2 = fmaf(tb.x, rowf, c0), x3 = fmaf(tb.y, rowf, c0);
          if (!full) {
            if (cur.key0 + n > cur.pos) x0 = -INFINITY;
            if (cur.key0 + n + 1 > cur.pos) x1 = -INFINITY;
            if (cur.key0 + n + 2 > cur.pos) x2 = -INFINITY;
            if (cur.key0 + n + 3 > cur.pos) x3 = -INFINITY;
          }
          const float p0 = tq_ex2(x0), p1 = tq_ex2(x1), p2 = tq_ex2(x2), p3 = tq_ex2(x3);
          l0 += p0 + p2;
          l1 += p1 + p3;
          const float2 pa = mul2(p0, p1, v4.x, v4.y);
          const float2 pb = mul2(p2, p3, v4.z, v4.w);
          uint32_t ha, la, hb, lb;
          split2_e4m3(pa.x, pa.y, ha, la);
          split2_e4m3(pb.x, pb.y, hb, lb);
          hw[q4] = ha | (hb << 16);
          lw[q4] = la | (lb << 16);
        }
        tmem_st8(tS + lsel + 16 * h, hw);
        tmem_st8(tS + lsel + 16 * h + 8, lw);
      }
      const float le = l0 + l1;  // l x 2^e
      tmem_st_wait();
      tc_fence_before();
      named_bar_sync(bar_id, 128);
      if (leader) {
        tc_fence_after();
        const uint32_t vt = smem_u32(sb + LY::S_V);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
          for (int term = 0; term < 2; ++term)
            mma_f8_ts(tO, tS + 16 * kk + 8 * term, sw128_desc_mn(vt + 4096 * kk), kIdescPV, (term | kk) != 0);
        mma_commit(&obar[grp]);
      }
      if (!gwait(&obar[grp], (uint32_t)(u & 1), 23)) break;
      tc_fence_after();
      ++u;
      // P has been read: the next item's MMA 1 overlaps this item's output
      if (jn < nj && !start(nxt, jn)) break;
      // ---- o / l x 2^-ev as fp16 rows, staged entry by entry in this item's
      // stage (its tiles, scales and header are no longer read), one bulk copy
      // per entry; then (m, l, 2^ev); the stage goes back to the producer once
      // the copies have read it
      const float inv = le > 0.f ? ldexpf(__frcp_rn(le), -ev) : 0.f;
      uint8_t* orow = base + LY::ST + (size_t)cur.st * LY::STAGE + (size_t)(m >> lr) * epitch + (size_t)hh * 256;
#pragma unroll 1
      for (int h = 0; h < 4; ++h) {
        float v[32];
        tmem_ld32(tO + lsel + 32 * h, v);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 w;
          w.x = pack_f16x2(v[8 * c] * inv, v[8 * c + 1] * inv);
          w.y = pack_f16x2(v[8 * c + 2] * inv, v[8 * c + 3] * inv);
          w.z = pack_f16x2(v[8 * c + 4] * inv, v[8 * c + 5] * inv);
          w.w = pack_f16x2(v[8 * c + 6] * inv, v[8 * c + 7] * inv);
          *reinterpret_cast<uint4*>(orow + 16 * ((4 * h + c) ^ hh)) = w;  // the partials' swizzle
        }
      }
      // the rows written here are read next by the bulk copies (and later
      // overwritten by the producer's copies): order them for the async proxy
      fence_proxy_async();
      __syncwarp();  // an entry's r rows are written by r lanes of one warp
      if (cur.valid && hh == 0) {
        bulk_s2g(reinterpret_cast<__half*>(p.part_o) + cur.part * 128, orow, (uint32_t)r * 256u);
        bulk_commit();
      }
      if (cur.valid)
        reinterpret_cast<float4*>(p.part_ml)[cur.part] = make_float4(m2, ldexpf(le, -e), ldexpf(1.f, ev), 0.f);
      bulk_wait_read();
      mbar_arrive(&kvempty[cur.st]);
      tc_fence_before();  // the O reads come before the next MMA 2 (ordered by the group's next barrier)
      j = jn;
      cur = nxt;
      rowf = rowf_n;
    }
    cp_async_wait();
    bulk_wait_all();
    // every MMA this leader issued has completed before TMEM is freed
    if (leader) {
      mma_commit(&done[grp]);
      mbar_wait_sleep(&done[grp], 0, 200000);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_k2q_attend(const CUtensorMap* tk, const CUtensorMap* tv, const K2qParams& p, int num_sms,
                              cudaStream_t st) {
  const size_t smem = TqLayout::SMEM;
  static bool ready = false;
  if (!ready) {
    cudaError_t e = cudaFuncSetAttribute(k2q_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k2q_tc_kernel, kTqThreads, smem);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    ready = true;  // one CTA per SM: it holds all 512 TMEM columns
  }
  k2q_tc_kernel<<<num_sms > 0 ? num_sms : 1, kTqThreads, smem, st>>>(*tk, *tv, p);
  return cudaGetLastError();
}

}  // namespace msa
