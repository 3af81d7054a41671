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
//   S[128 x 128 keys] = Qop[128 x 128 dims] . K^T       (MMA 1, K-major both)
//   O[128 x 128 dims] = P[128 x 128 keys] . V           (MMA 2, V MN-major)
// kind::f8f6f4, e4m3 x e4m3, fp32 accumulators in TMEM.  A bf16 query enters
// as two e4m3 terms (hi + lo, after a power-of-two scale per row, prepared
// once per (token, head) by the count pass); an e4m3 query as one.  P enters as
// hi + lo e4m3 terms of p * vscale_t * 2^e (2^e puts the block's largest V
// scale at most at 448), so that V's per-token scales fold into P.
//
// One CTA per SM (all 512 TMEM columns), 9 warps:
//   warp 0     copies items (header, entries, K / V tiles with the 128-byte
//              swizzle, per-token scales) into a 4-stage ring, the facts of 32
//              items at a time read by its 32 lanes together; owns TMEM;
//   warps 1-4  group 0 and warps 5-8 group 1 take alternate items; each
//              thread owns one MMA row (TMEM lane).  A group builds its
//              item's query operand, its leader thread issues MMA 1, the
//              threads turn S into P in the same shared buffer (max, exp2,
//              sum, V scales, hi / lo split), the leader issues MMA 2, and
//              while it runs the group loads its next item's query rows; the
//              next item's MMA 1 is issued before this item's output is
//              written.  S (128 columns) and O (128 columns) per group.
// Every wait is bounded; a wait that gives up sets the timeout flag and the
// CTA stops issuing, drains what it issued and frees its TMEM.
#include "msa_device.cuh"
#include "msa_internal.h"
#include "msa_tcgen05.cuh"

namespace msa {

namespace {

constexpr int kTqStages = 4;
constexpr int kTqThreads = 288;
constexpr uint32_t kTqTile = 128 * 128;   // one e4m3 128 x 128 operand
constexpr uint32_t kTqScales = 128 * 4;
constexpr uint32_t kTqEnt = 136 * 4;      // an item's entries, copied from a 16-byte boundary
constexpr uint32_t kTqHdr = 8 * 4;

constexpr uint32_t tq_round(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

struct TqLayout {
  static constexpr uint32_t OP = 0;                         // [group][hi, lo][16 KB]: query operand, then P
  static constexpr uint32_t ST = OP + 4 * kTqTile;          // the ring of stages
  static constexpr uint32_t S_K = 0, S_V = kTqTile, S_KS = 2 * kTqTile, S_VS = S_KS + kTqScales;
  static constexpr uint32_t S_ENT = S_VS + kTqScales, S_HDR = S_ENT + kTqEnt;
  static constexpr uint32_t STAGE = tq_round(S_HDR + kTqHdr, 1024);
  static constexpr uint32_t BARS = ST + kTqStages * STAGE;
  // kvfull[stages], kvempty[stages], sbar[2], obar[2], done[2]
  static constexpr uint32_t NBARS = 2 * kTqStages + 6;
  static constexpr uint32_t TSLOT = BARS + NBARS * 8;
  static constexpr uint32_t DEAD = TSLOT + 4;
  static constexpr uint32_t TOTAL = DEAD + 12;
  static constexpr uint32_t SMEM = TOTAL + 1024;            // 1024-byte alignment slack
};

// Instruction descriptors: D fp32, A and B e4m3, M = N = 128; A K-major; B
// K-major (keys, MMA 1) or MN-major (V with the head dims contiguous, MMA 2).
constexpr uint32_t kIdescQK = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescPV = kIdescQK | (1u << 16);

// Operand descriptor of an MN-major 128-byte-swizzled tile: 128-byte rows
// along K (one per key), 8-row groups 1024 bytes apart.  With 128 e4m3
// columns the tile is one swizzle atom wide, so only the K-direction group
// offset is used; both offsets hold it.
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3fffu) | ((uint64_t)(1024 >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ float tq_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// This thread's row of an item.
struct TqRow {
  int st;       // ring stage
  int valid;    // the row holds a real (entry, head)
  int pos;      // last key the row's token may see (-1: none)
  int key0;     // the block's first key
  long part;    // (token, head, slot) partial
  long qrow;    // (token, head) query row
};

__global__ void __launch_bounds__(kTqThreads, 1) k2q_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                                                             const __grid_constant__ CUtensorMap tmv,
                                                             const K2qParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using LY = TqLayout;
  uint64_t* kvfull = reinterpret_cast<uint64_t*>(base + LY::BARS);
  uint64_t* kvempty = kvfull + kTqStages;
  uint64_t* sbar = kvempty + kTqStages;
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
      mbar_init(&kvempty[i], 1);
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
    // ---------------- items into the ring
    int issued = 0;
    bool ok = true;
    for (int j0 = 0; j0 < nj && ok; j0 += 32) {
      int f_n = 0, f_s = 0, f_g = 0, f_b = 0, f_T = 0, f_e0 = 0, f_ph = -1;
      if (j0 + lane < nj) {
        const int it = i0 + j0 + lane;
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
      for (int t = 0; t < 32 && j0 + t < nj; ++t) {
        const int n = __shfl_sync(0xffffffffu, f_n, t), s = __shfl_sync(0xffffffffu, f_s, t);
        const int g = __shfl_sync(0xffffffffu, f_g, t), b = __shfl_sync(0xffffffffu, f_b, t);
        const int T = __shfl_sync(0xffffffffu, f_T, t), e0 = __shfl_sync(0xffffffffu, f_e0, t);
        const int ph = __shfl_sync(0xffffffffu, f_ph, t);
        const int j = j0 + t;
        if (lane == 0) {
          const int st = j % kTqStages;
          if (j >= kTqStages && (*reinterpret_cast<volatile int*>(dead) ||
                                 !mbar_wait(&kvempty[st], (uint32_t)(((j / kTqStages) - 1) & 1)))) {
            if (!*reinterpret_cast<volatile int*>(dead)) raise_flag(p.status, FLAG_TIMEOUT, 20);
            *reinterpret_cast<volatile int*>(dead) = 1;
            ok = false;
          } else {
            uint8_t* sb = base + LY::ST + (size_t)st * LY::STAGE;
            int32_t* hdr = reinterpret_cast<int32_t*>(sb + LY::S_HDR);
            const bool okb = ph >= 0 && ph < p.num_blocks && n > 0;
            if (!okb && n > 0) raise_flag(p.status, FLAG_BAD_BLOCK, ph);
            const int ea = e0 & ~3, nent = n > 0 ? n : 0;
            const uint32_t ebytes = (uint32_t)((e0 - ea + nent + 3) & ~3) * 4u;
            hdr[0] = okb ? n : -nent;  // negative: the block is rejected, its entries get empty partials
            hdr[1] = s;
            hdr[2] = g;
            hdr[3] = b;
            hdr[4] = T;
            hdr[5] = e0 - ea;
            fence_proxy_async();
            mbar_expect_tx(&kvfull[st], ebytes + (okb ? 2 * kTqTile + 2 * kTqScales : 0u));
            if (ebytes > 0) bulk_g2s(sb + LY::S_ENT, p.entries + ea, ebytes, &kvfull[st]);
            if (okb) {
              const int tile = (int)(((long)ph * G + g) * kBlock);
              tma_load_2d(sb + LY::S_K, &tmk, 0, tile, &kvfull[st]);
              tma_load_2d(sb + LY::S_V, &tmv, 0, tile, &kvfull[st]);
              bulk_g2s(sb + LY::S_KS, p.k_scale + tile, kTqScales, &kvfull[st]);
              bulk_g2s(sb + LY::S_VS, p.v_scale + tile, kTqScales, &kvfull[st]);
            }
            issued = j + 1;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
    }
    // a CTA that gave up waits (bounded) for the copies it issued
    if (lane == 0 && !ok) {
      for (int i = 0; i < kTqStages && i < issued; ++i) {
        const int jj = issued - 1 - i;
        mbar_wait(&kvfull[jj % kTqStages], (uint32_t)((jj / kTqStages) & 1), 2000);
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
    uint8_t* ohi = op + (size_t)m * 128;
    uint8_t* olo = ohi + kTqTile;
    const int sw = m & 7;

    // every thread of the group waits; the group agrees on the outcome
    auto gwait = [&](uint64_t* bar, uint32_t par, int where) -> bool {
      const bool ok = !*reinterpret_cast<volatile int*>(dead) && mbar_wait(bar, par);
      const bool bad = named_bar_or(bar_id, 128, !ok);
      if (bad && leader && !*reinterpret_cast<volatile int*>(dead)) {
        *reinterpret_cast<volatile int*>(dead) = 1;
        raise_flag(p.status, FLAG_TIMEOUT, where);
      }
      return !bad;
    };

    // Item j's stage and this thread's row of it, with the row's query loaded
    // into qv (hi, then lo for a bf16 query) and its factor into rowf.
    // Rejected items (block outside the cache) get empty partials and release
    // their stage here; the walk moves on to the group's next item.  Returns
    // the item taken, or nj.
    uint4 qv[16];
    float rowf_n = 0.f;
    auto take = [&](int j, TqRow& rw) -> int {
      for (; j < nj; j += 2) {
        const int st = j % kTqStages;
        if (!gwait(&kvfull[st], (uint32_t)((j / kTqStages) & 1), 21)) return nj;
        const uint8_t* sb = base + LY::ST + (size_t)st * LY::STAGE;
        const int32_t* hdr = reinterpret_cast<const int32_t*>(sb + LY::S_HDR);
        const int n = hdr[0], s = hdr[1], g = hdr[2], b = hdr[3], T = hdr[4], delta = hdr[5];
        const int nr = (n < 0 ? -n : n) * r;
        rw.st = st;
        rw.valid = m < nr;
        rw.key0 = b * kBlock;
        const int ent = rw.valid ? reinterpret_cast<const int32_t*>(sb + LY::S_ENT)[delta + (m >> lr)] : 0;
        const long token = ent >> 5;
        const int head = g * r + (m & (r - 1));
        rw.part = (token * H + head) * K + (ent & 31);
        rw.qrow = token * H + head;
        rw.pos = rw.valid ? T - Q + (int)(token - (long)s * Q) : -1;
        if (n > 0) {
          if (rw.valid) {
            if (p.q_fp8) {
              const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.q) + rw.qrow * 128);
#pragma unroll
              for (int c = 0; c < 8; ++c) qv[c] = __ldg(src + c);
              rowf_n = qconst;
            } else {
              const uint4* src = reinterpret_cast<const uint4*>(p.qsplit + rw.qrow * 256);
#pragma unroll
              for (int c = 0; c < 16; ++c) qv[c] = __ldg(src + c);
              rowf_n = __ldg(p.qrowf + rw.qrow);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) qv[c] = make_uint4(0u, 0u, 0u, 0u);
            rowf_n = 0.f;
          }
          return j;
        }
        if (rw.valid) reinterpret_cast<float4*>(p.part_ml)[rw.part] = make_float4(-INFINITY, 0.f, 1.f, 0.f);
        named_bar_sync(bar_id, 128);  // every row has read the stage
        if (leader) mbar_arrive(&kvempty[st]);
      }
      return nj;
    };

    // the loaded query rows into the operand (swizzled K-major rows), then MMA 1
    auto start = [&](const TqRow& rw) {
#pragma unroll
      for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(ohi + ((c ^ sw) << 4)) = qv[c];
      if (terms == 2) {
#pragma unroll
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(olo + ((c ^ sw) << 4)) = qv[8 + c];
      }
      fence_proxy_async();  // the MMA reads the operand through the async proxy
      tc_fence_before();
      named_bar_sync(bar_id, 128);
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
    };

    TqRow cur, nxt;
    int u = 0;  // items of this group whose MMAs ran (phases of sbar / obar)
    int j = take(grp, cur);
    float rowf = rowf_n;
    if (j < nj) start(cur);
#pragma unroll 1
    while (j < nj) {
      if (!gwait(&sbar[grp], (uint32_t)(u & 1), 22)) break;
      tc_fence_after();
      const uint8_t* sb = base + LY::ST + (size_t)cur.st * LY::STAGE;
      const float* ks = reinterpret_cast<const float*>(sb + LY::S_KS);
      const float* vs = reinterpret_cast<const float*>(sb + LY::S_VS);
      // P's scale 2^e puts the block's largest V scale at most at 448; the
      // fp16 partial o / l (at most max |v| <= 448 x that scale) is brought
      // under 32768 by 2^-ev
      float vmx = fmaxf(fmaxf(vs[lane], vs[lane + 32]), fmaxf(vs[lane + 64], vs[lane + 96]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) vmx = fmaxf(vmx, __shfl_xor_sync(0xffffffffu, vmx, o));
      const int e = min(126, fit448(vmx));
      const float fe = (e >= -126) ? pow2i(e) : ldexpf(1.f, e);
      int ev = 0;
      if (448.f * vmx > 32768.f) frexpf(448.f * vmx * (1.f / 32768.f), &ev);
      const bool full = cur.key0 + kBlock - 1 <= cur.pos;  // every key visible
      // ---- the row's max of s_t * kscale_t over its visible keys
      float mx = -INFINITY;
#pragma unroll 1
      for (int h = 0; h < 4; ++h) {
        float v[1][32];
        tmem_ld32(tS + lsel + 32 * h, v[0]);
        tmem_ld_wait();
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        {
          constexpr int q = 0;
          const int n0 = 32 * h;
          if (full) {
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
              const float sc = (cur.key0 + n0 + n <= cur.pos) ? v[q][n] * ks[n0 + n] : -INFINITY;
              m4[n & 3] = fmaxf(m4[n & 3], sc);
            }
          }
        }
        mx = fmaxf(mx, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
      }
      const float m2 = mx * rowf;                           // base-2 logit maximum (rowf > 0)
      const float msub = (mx == -INFINITY) ? 0.f : m2;
      // ---- p_t = 2^(x_t - m), l = sum p_t, P'_t = p_t vscale_t 2^e as e4m3 hi + lo
      float l0 = 0.f, l1 = 0.f;
#pragma unroll 1
      for (int h = 0; h < 4; ++h) {
        float v[1][32];
        tmem_ld32(tS + lsel + 32 * h, v[0]);
        tmem_ld_wait();
        constexpr int q = 0;
#pragma unroll
          for (int c16 = 0; c16 < 2; ++c16) {
            const int n0 = 32 * h + 16 * c16;  // first key of this 16-key chunk
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int n = n0 + 2 * i;
              const float2 t = mul2(v[q][16 * c16 + 2 * i], v[q][16 * c16 + 2 * i + 1], ks[n], ks[n + 1]);
              float x0 = fmaf(t.x, rowf, -msub), x1 = fmaf(t.y, rowf, -msub);
              if (!full) {
                if (cur.key0 + n > cur.pos) x0 = -INFINITY;
                if (cur.key0 + n + 1 > cur.pos) x1 = -INFINITY;
              }
              const float p0 = tq_ex2(x0), p1 = tq_ex2(x1);
              l0 += p0;
              l1 += p1;
              const float2 vf = mul2(vs[n], vs[n + 1], fe, fe);
              const float2 pp = mul2(p0, p1, vf.x, vf.y);
              const uint16_t hb = pack_e4m3x2(pp.x, pp.y);
              const float2 hv = e4m3x2_to_float2(hb);
              const uint16_t lb = pack_e4m3x2(pp.x - hv.x, pp.y - hv.y);
              if (i & 1) {
                hw[i >> 1] |= (uint32_t)hb << 16;
                lw[i >> 1] |= (uint32_t)lb << 16;
              } else {
                hw[i >> 1] = hb;
                lw[i >> 1] = lb;
              }
            }
            const int c = n0 >> 4;  // 16-byte chunk of the 128-key row
            *reinterpret_cast<uint4*>(ohi + ((c ^ sw) << 4)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(olo + ((c ^ sw) << 4)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
      }
      const float l = l0 + l1;
      fence_proxy_async();
      tc_fence_before();
      named_bar_sync(bar_id, 128);
      if (leader) {
        tc_fence_after();
        const uint32_t vt = smem_u32(sb + LY::S_V);
#pragma unroll
        for (int term = 0; term < 2; ++term)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f8(tO, sw128_desc(op_s + term * kTqTile + 32 * k), sw128_desc_mn(vt + 4096 * k), kIdescPV,
                   (term | k) != 0);
        mma_commit(&obar[grp]);
        mma_commit(&kvempty[cur.st]);  // the stage is free once MMA 2 has read V
      }
      // the group's next item: its stage and query rows, while MMA 2 runs
      const int jn = take(j + 2, nxt);
      if (!gwait(&obar[grp], (uint32_t)(u & 1), 23)) break;
      tc_fence_after();
      ++u;
      if (jn < nj) start(nxt);  // MMA 1 of the next item overlaps this item's output
      // ---- o / l x 2^-ev as fp16, with (m, l, 2^ev)
      const float inv = l > 0.f ? ldexpf(__frcp_rn(l), -e - ev) : 0.f;
      __half* dst = reinterpret_cast<__half*>(p.part_o) + cur.part * 128;
#pragma unroll 1
      for (int h = 0; h < 4; ++h) {
        float v[1][32];
        tmem_ld32(tO + lsel + 32 * h, v[0]);
        tmem_ld_wait();
        if (cur.valid) {
          constexpr int q = 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint4 w;
              w.x = pack_f16x2(v[q][8 * c] * inv, v[q][8 * c + 1] * inv);
              w.y = pack_f16x2(v[q][8 * c + 2] * inv, v[q][8 * c + 3] * inv);
              w.z = pack_f16x2(v[q][8 * c + 4] * inv, v[q][8 * c + 5] * inv);
              w.w = pack_f16x2(v[q][8 * c + 6] * inv, v[q][8 * c + 7] * inv);
              *reinterpret_cast<uint4*>(dst + 32 * h + 8 * c) = w;
            }
        }
      }
      if (cur.valid) reinterpret_cast<float4*>(p.part_ml)[cur.part] = make_float4(m2, l, ldexpf(1.f, ev), 0.f);
      tc_fence_before();  // the O reads come before the next MMA 2 (ordered by the group's next barrier)
      j = jn;
      cur = nxt;
      rowf = rowf_n;
    }
    // every MMA this leader issued has completed before TMEM is freed
    if (leader) {
      mma_commit(&done[grp]);
      mbar_wait(&done[grp], 0, 200000);
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
