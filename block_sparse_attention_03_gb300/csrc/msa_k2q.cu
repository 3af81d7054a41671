// Key-block-major attend of prefill chunks: the selection inverted into lists
// (the key -> query CSR `build_k2q_csr` of the vLLM MiniMax-M3 model page,
// "vllm.models.minimax_m3.nvidia.model") and the per-token merge of the
// per-block partials.
//
// Count: for every (token, group, slot) whose selected block is b, one more
// entry in list (sequence, group, b) -- taken token-fastest, so that a warp's
// lanes mostly share lists and one atomic serves each group of them.  Scan (one
// CTA): each list's first entry and first attend item (item_tokens = 128 / r
// entries an item: one MMA row per (token, head)); the same launch's other CTAs
// split each bf16 query row into the e4m3 hi + lo terms the attend's MMA reads.  Fill: every entry (token * 32 + slot)
// into its list, in arrival order (the per-entry results do not depend on
// it).  The attend (msa_k2q_tc.cu) reads each item's K/V tile once and writes
// one partial (o, m, l, 2^ev) per (token, head, slot); combine merges a
// token's slots by log-sum-exp: the exact softmax over all of the token's
// selected blocks (vLLM Day-0 blog, section "MSA 入门").
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {

namespace {

// Selection entry e = (token, group, slot): its list (sequence, group, block),
// or -1 for an empty slot (-1), a block the token cannot see, or a block an
// earlier slot of the same row already names (the last two flagged once, by
// the count pass; the softmax runs over the selected key set, each key once).
// Count, fill and combine agree.
// (Entries, rows and tokens are counted in 32 bits: make_plan keeps every
// partial index below 2^31.)
__device__ __forceinline__ long k2q_list(const K2qParams& p, int e, bool flag) {
  const BatchDev bt = p.batch;
  const int b = p.topk_idx[e];
  if (b < 0) return -1;
  const int row = e / p.topk;  // token * G + g
  const int token = row / p.G;
  const int s = token / bt.Q, g = row % p.G, i = token % bt.Q;
  const int T = bt.seq_len(s);
  bool bad = b >= bt.max_nb || T < bt.Q || T > bt.max_nb * kBlock || b > (T - bt.Q + i) / kBlock;
  const int slot = e - row * p.topk;
  for (int k = 0; k < slot && !bad; ++k) bad = p.topk_idx[(long)row * p.topk + k] == b;
  if (bad) {
    if (flag) raise_flag(p.status, FLAG_BAD_SELECT, b);
    return -1;
  }
  return ((long)s * p.G + g) * bt.max_nb + b;
}

// Entry x of the count and fill passes, token-fastest: the lanes of a warp take
// the same (group, slot) of 32 consecutive tokens, which often name the same
// block (the slots are ascending; nearby tokens share their own and the best
// blocks), so that one atomic serves each group of lanes with the same list.
__device__ __forceinline__ int k2q_entry_of(const K2qParams& p, int x, int ntok) {
  const int token = x % ntok, r = x / ntok;
  const int g = r % p.G, slot = r / p.G;
  return (token * p.G + g) * p.topk + slot;
}

__global__ void __launch_bounds__(256) k2q_count_kernel(const K2qParams p) {
  const BatchDev bt = p.batch;
  const int ntok = bt.S * bt.Q;
  const int n = ntok * p.G * p.topk;
  const int lane = threadIdx.x & 31;
  for (int x0 = blockIdx.x * blockDim.x + (threadIdx.x & ~31); x0 < n; x0 += gridDim.x * blockDim.x) {
    const int x = x0 + lane;  // the loop is warp-uniform
    const long key = x < n ? k2q_list(p, k2q_entry_of(p, x, ntok), true) : -1;
    const unsigned act = __ballot_sync(0xffffffffu, key >= 0);
    if (key >= 0) {
      const unsigned peers = __match_any_sync(act, (unsigned long long)key);
      if (lane == __ffs(peers) - 1) atomicAdd(&p.cnt[key], __popc(peers));
    }
  }
}

// The bf16 query split, by warps w0, w0 + 1, ... of nw (run by the scan
// launch's extra CTAs: it needs only the caller's queries, and the scan keeps one
// SM busy).
__device__ __forceinline__ void k2q_split_queries(const K2qParams& p, int w0, int nw) {
  // bf16 query rows (token, head), a warp each, lane l holding dims 4l .. 4l+3:
  // q x 2^e with the largest e that keeps the row's amax at most 448 (exact),
  // split into e4m3 hi + lo (together all 8 significant bits of bf16), and
  // the row factor 2^-e x col_const
  const BatchDev bt = p.batch;
  const int rows = bt.S * bt.Q * p.G * p.r;
  const int lane = threadIdx.x & 31;
  for (int row = w0 + (threadIdx.x >> 5); row < rows; row += nw) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p.q) + (long)row * 128) + lane);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    float amax = fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int ex = pow2_fit(amax, 448.f);
    const float ps = ldexpf(1.f, ex);
    float h[4], l[4];
    split_e4m3(a.x * ps, h[0], l[0]);
    split_e4m3(a.y * ps, h[1], l[1]);
    split_e4m3(b.x * ps, h[2], l[2]);
    split_e4m3(b.y * ps, h[3], l[3]);
    uint32_t* dst = reinterpret_cast<uint32_t*>(p.qsplit + (long)row * 256);
    dst[lane] = (uint32_t)pack_e4m3x2(h[0], h[1]) | ((uint32_t)pack_e4m3x2(h[2], h[3]) << 16);
    dst[32 + lane] = (uint32_t)pack_e4m3x2(l[0], l[1]) | ((uint32_t)pack_e4m3x2(l[2], l[3]) << 16);
    if (lane == 0) p.qrowf[row] = ldexpf(1.f, -ex) * p.col_const;
  }
}

// One CTA of 1024 threads: thread t owns the contiguous lists [t*L/1024, (t+1)*L/1024).
// CTA 0 scans; CTAs 1.. split the bf16 query rows meanwhile.
__global__ void __launch_bounds__(1024) k2q_scan_kernel(const K2qParams p) {
  __shared__ int se[64], si[64];  // the warp totals, then their inclusive scan
  if (blockIdx.x > 0) {
    k2q_split_queries(p, (blockIdx.x - 1) * 32, (gridDim.x - 1) * 32);
    return;
  }
  const BatchDev bt = p.batch;
  const long L = (long)bt.S * p.G * bt.max_nb;
  const int t = threadIdx.x;
  const long l0 = t * L / 1024, l1 = (t + 1) * L / 1024;
  int ne = 0, ni = 0;
  for (long i = l0; i < l1; ++i) {
    const int c = p.cnt[i];
    ne += c;
    ni += (c + p.item_tokens - 1) / p.item_tokens;
  }
  // inclusive scans of (entries, items) over the threads: within each warp by
  // shuffles, then over the 32 warp totals by warp 0
  const int lane = t & 31, warp = t >> 5;
  int xe = ne, xi = ni;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ye = __shfl_up_sync(0xffffffffu, xe, o), yi = __shfl_up_sync(0xffffffffu, xi, o);
    if (lane >= o) {
      xe += ye;
      xi += yi;
    }
  }
  if (lane == 31) {
    se[warp] = xe;
    si[warp] = xi;
  }
  __syncthreads();
  if (warp == 0) {
    int ve = se[lane], vi = si[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ye = __shfl_up_sync(0xffffffffu, ve, o), yi = __shfl_up_sync(0xffffffffu, vi, o);
      if (lane >= o) {
        ve += ye;
        vi += yi;
      }
    }
    se[32 + lane] = ve;  // inclusive over warps
    si[32 + lane] = vi;
  }
  __syncthreads();
  const int be = warp > 0 ? se[32 + warp - 1] : 0, bi = warp > 0 ? si[32 + warp - 1] : 0;
  int e0 = be + xe - ne, i0 = bi + xi - ni;
  for (long i = l0; i < l1; ++i) {
    const int c = p.cnt[i];
    const int items = (c + p.item_tokens - 1) / p.item_tokens;
    p.off[i] = e0;
    p.cur[i] = e0;
    p.item_off[i] = i0;
    for (int k = 0; k < items; ++k) p.item_list[i0 + k] = (int)i;  // the attend's item -> list map
    e0 += c;
    i0 += items;
  }
  if (t == 1023) p.item_off[L] = si[32 + 31];
}

__global__ void __launch_bounds__(256) k2q_fill_kernel(const K2qParams p) {
  const BatchDev bt = p.batch;
  const int ntok = bt.S * bt.Q;
  const int n = ntok * p.G * p.topk;
  const int lane = threadIdx.x & 31;
  for (int x0 = blockIdx.x * blockDim.x + (threadIdx.x & ~31); x0 < n; x0 += gridDim.x * blockDim.x) {
    const int x = x0 + lane;  // the loop is warp-uniform
    const int e = x < n ? k2q_entry_of(p, x, ntok) : 0;
    const long key = x < n ? k2q_list(p, e, false) : -1;
    const unsigned act = __ballot_sync(0xffffffffu, key >= 0);
    if (key >= 0) {
      // one cursor bump per group of lanes with the same list, each lane its place in it
      const unsigned peers = __match_any_sync(act, (unsigned long long)key);
      const int leader = __ffs(peers) - 1;
      int at = 0;
      if (lane == leader) at = atomicAdd(&p.cur[key], __popc(peers));
      at = __shfl_sync(peers, at, leader) + __popc(peers & ((1u << lane) - 1u));
      const int token = e / p.topk / p.G;
      const int slot = e % p.topk;
      p.entries[at] = token * 32 + slot;
    }
  }
}

__device__ __forceinline__ float k2q_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One warp per (token, head): the token's selected slots merged by
// log-sum-exp in base 2 (m and l come that way).  Every load of the row is
// issued at once: lane k < topk takes slot k's (m, l, 2^ev), and the two
// half-warps take the even and the odd slots' o / l rows, lane l holding the
// row's 16-byte chunk l % 16 (dims 8 ((l % 16) ^ (head % r)) .. + 7, the
// attend's swizzle) with one load a slot (32 slots at most).
template <int KMAX>
__global__ void __launch_bounds__(256) k2q_combine_kernel(const K2qParams p) {
  const BatchDev bt = p.batch;
  const int H = p.G * p.r;
  const int rows = bt.S * bt.Q * H;
  const int lane = threadIdx.x & 31, half = lane >> 4, d8 = 8 * (lane & 15);
  const int nw = gridDim.x * (blockDim.x >> 5);
  for (int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows; row += nw) {
    const int token = row / H;
    const int h = row % H, g = h / p.r;
    const int32_t* sel = p.topk_idx + ((long)token * p.G + g) * p.topk;
    // the entries the lists hold (k2q_list's rule), no others: the token's
    // visible blocks of a well-formed sequence
    const int s = token / bt.Q, i = token % bt.Q;
    const int T = bt.seq_len(s);
    const int last = (T < bt.Q || T > bt.max_nb * kBlock) ? -1 : min(bt.max_nb - 1, (T - bt.Q + i) / kBlock);
    // the lane's 16-byte chunk of every slot's row holds dims 8 ((lane % 16) ^
    // (head % r)) .. + 7 (the attend's swizzle, the same for all the row's slots)
    const uint4* orow = reinterpret_cast<const uint4*>(p.part_o + ((long)token * p.topk * H + h) * 128 + d8);
    uint4 ov[KMAX / 2];
#pragma unroll
    for (int q = 0; q < KMAX / 2; ++q) {  // slot 2q + half
      const int k = 2 * q + half;
      ov[q] = k < p.topk ? __ldcg(orow + (long)k * H * 16) : make_uint4(0u, 0u, 0u, 0u);
    }
    // slot lane's (m, l, 2^ev), loaded with the rest (in bounds for every slot;
    // used only for the slots the lists hold)
    const float4 ml = lane < p.topk
                          ? __ldcg(reinterpret_cast<const float4*>(p.part_ml) + ((long)token * p.topk + lane) * H + h)
                          : make_float4(-INFINITY, 0.f, 1.f, 0.f);
    float mk = -INFINITY, lk = 0.f, fk = 1.f;
    const int bl = lane < p.topk ? sel[lane] : -1;
    // a block an earlier slot already names has no list entry (k2q_list)
    const unsigned same = __match_any_sync(0xffffffffu, bl);
    if (lane < p.topk && bl >= 0 && bl <= last && (same & ((1u << lane) - 1u)) == 0u) {
      mk = ml.x;
      lk = ml.y;
      fk = ml.z;
    }
    float M = mk;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float wk = (mk == -INFINITY) ? 0.f : k2q_ex2(mk - M) * lk;
    const float wo = wk * fk;  // the weight of the stored o / l x 2^-ev
    float Lsum = wk;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < KMAX / 2; ++q) {
      const float w = __shfl_sync(0xffffffffu, wo, 2 * q + half);
      if (w != 0.f) {  // a slot left out may hold anything: select, do not multiply
        const __half2* hv = reinterpret_cast<const __half2*>(&ov[q]);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 f = __half22float2(hv[t]);
          acc[2 * t] += w * f.x;
          acc[2 * t + 1] += w * f.y;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], 16);
    const float inv = Lsum > 0.f ? __fdividef(1.f, Lsum) : 0.f;
    if (half == 0) {
      uint4 pk;
      pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      pk.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
      pk.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + (long)row * 128 + 8 * ((lane & 15) ^ (h % p.r))) =
          pk;
    }
    if (lane == 0 && p.lse) p.lse[row] = Lsum > 0.f ? (M + __log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_k2q_build(const K2qParams& p, int num_sms, cudaStream_t st) {
  const long L = (long)p.batch.S * p.G * p.batch.max_nb;
  cudaError_t e = cudaMemsetAsync(p.cnt, 0, (size_t)L * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  const long n = (long)p.batch.S * p.batch.Q * p.G * p.topk;
  long grid = (n + 255) / 256;
  if (grid > 4096) grid = 4096;
  if (grid < 1) grid = 1;
  k2q_count_kernel<<<(unsigned)grid, 256, 0, st>>>(p);
  // CTA 0 scans; with a bf16 query, 4 CTAs an SM more split its rows
  const long qrows = p.q_fp8 ? 0 : (long)p.batch.S * p.batch.Q * p.G * p.r;
  long qctas = (qrows + 31) / 32;
  if (qctas > 4L * num_sms) qctas = 4L * num_sms;
  k2q_scan_kernel<<<(unsigned)(1 + qctas), 1024, 0, st>>>(p);
  k2q_fill_kernel<<<(unsigned)grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_k2q_combine(const K2qParams& p, int num_sms, cudaStream_t st) {
  const long rows = (long)p.batch.S * p.batch.Q * p.G * p.r;
  long grid = (rows + 7) / 8;
  // eight CTAs an SM, each warp walking rows: with one row a warp, tens of
  // thousands of short CTAs spend the kernel turning CTAs over
  const long cap = 8L * (num_sms > 0 ? num_sms : 1);
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  if (p.topk <= 16) k2q_combine_kernel<16><<<(unsigned)grid, 256, 0, st>>>(p);
  else k2q_combine_kernel<32><<<(unsigned)grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace msa
