// Cache insert: the K, V and index key of new tokens quantized into the paged
// caches -- the step just before the path (vLLM Day-0 blog, section "QKV GEMM
// + norm + RoPE + KV 插入融合": K, V and the index key are quantized and written
// straight into their caches; "[M3] Enable FP8 sparse GQA", items 1 and 4: FP8
// values stored through the slot mapping).  The projections, norms and RoPE
// that precede it need weights and are not part of this library.
//
// One warp per token, its rows of 128 elements (K heads, V heads, index key)
// loaded together, four elements a lane: an 8-byte load of the bf16 row
// piece, the row's or the
// 16-group's absolute maximum by shuffles, one fp32 division per element, the
// hardware's round-to-nearest-even conversions (cvt ... satfinite e4m3x2 /
// e2m1x2), and coalesced stores of the codes.  The rules, fixed here because the
// pages give none:
//   BF16   the bits are copied;
//   FP8    scale = amax / 448 per (token, head) row (1 for an all-zero row),
//          code = e4m3(x / scale), sign kept;
//   NVFP4  with the cache's fp32 per-tensor scale g: per 16 elements
//          sf = e4m3(amax16 / (6 g)), code = e2m1(x / (sf * g)) (0 where
//          sf * g = 0), a code that rounds to zero stored as +0.
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {

namespace {

constexpr int kInsertWarps = 8;

// e2m1 codes of (lo, hi), round to nearest even, saturating at +-6: lo in the
// low nibble; a zero magnitude is returned as +0.
__device__ __forceinline__ uint32_t e2m1x2_code(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(r) : "f"(hi), "f"(lo));
  if ((r & 0x7u) == 0u) r &= 0xF0u;
  if ((r & 0x70u) == 0u) r &= 0x0Fu;
  return r;
}

// Quantize one row (raw: this lane's four bf16 elements) into the cache.
template <int FMT>
__device__ __forceinline__ void put_row(const uint2 raw, uint8_t* __restrict__ data, float* __restrict__ scale,
                                        uint8_t* __restrict__ sf, float g, long row, int lane) {
  if constexpr (FMT == FMT_BF16) {
    *reinterpret_cast<uint2*>(data + row * 256 + 8 * lane) = raw;
    return;
  }
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
  const float x[4] = {a.x, a.y, b.x, b.y};
  float m = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  if constexpr (FMT == FMT_FP8) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float s = m > 0.f ? __fdiv_rn(m, 448.f) : 1.f;
    const uint32_t c01 = pack_e4m3x2(__fdiv_rn(x[0], s), __fdiv_rn(x[1], s));
    const uint32_t c23 = pack_e4m3x2(__fdiv_rn(x[2], s), __fdiv_rn(x[3], s));
    *reinterpret_cast<uint32_t*>(data + row * 128 + 4 * lane) = c01 | (c23 << 16);
    if (lane == 0) scale[row] = s;
  } else {
    // the 16-element group of this lane: lanes 4q .. 4q + 3
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    const uint32_t sfc = pack_e4m3x2(__fdiv_rn(m, __fmul_rn(6.f, g)), 0.f) & 0xffu;
    const float den = __fmul_rn(e4m3_to_float((uint8_t)sfc), g);
    float y[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] = den > 0.f ? __fdiv_rn(x[i], den) : 0.f;
    const uint32_t c = e2m1x2_code(y[0], y[1]) | (e2m1x2_code(y[2], y[3]) << 8);
    *reinterpret_cast<uint16_t*>(data + row * 64 + 2 * lane) = (uint16_t)c;
    if ((lane & 3) == 0) sf[row * 8 + (lane >> 2)] = (uint8_t)sfc;
  }
}

// One warp per token: the loads of all its rows (H K heads, H V heads, the
// index key) are issued before any of them is quantized.  MAXH: the most
// heads an instance handles (4: sixteen row registers, four CTAs an SM).
template <int KVF, int IF, int MAXH>
__global__ void __launch_bounds__(32 * kInsertWarps, MAXH == 4 ? 4 : 2) insert_kernel(const InsertParams p) {
  constexpr int kMaxHeads = MAXH;
  const int lane = threadIdx.x & 31;
  const int H = p.H;
  const long nw = (long)gridDim.x * kInsertWarps;
  for (long t = (long)blockIdx.x * kInsertWarps + (threadIdx.x >> 5); t < p.num_tokens; t += nw) {
    const int slot = __ldg(p.slots + t);
    uint2 rk[kMaxHeads], rv[kMaxHeads], ri = make_uint2(0u, 0u);
#pragma unroll
    for (int h = 0; h < kMaxHeads; ++h) {
      if (h < H) {
        rk[h] = *reinterpret_cast<const uint2*>(p.k + (t * H + h) * kDim + 4 * lane);
        rv[h] = *reinterpret_cast<const uint2*>(p.v + (t * H + h) * kDim + 4 * lane);
      }
    }
    if (p.ik) ri = *reinterpret_cast<const uint2*>(p.ik + t * kDim + 4 * lane);
    if (slot < 0) continue;  // a padding token
    const int blk = slot >> 7, off = slot & 127;
    if (blk >= p.num_blocks) {
      if (lane == 0) raise_flag(p.status, FLAG_BAD_BLOCK, slot);
      continue;
    }
#pragma unroll
    for (int h = 0; h < kMaxHeads; ++h) {
      if (h < H) {
        const long row = ((long)blk * H + h) * kBlock + off;
        put_row<KVF>(rk[h], p.kc, p.ks, p.ksf, p.kg, row, lane);
        put_row<KVF>(rv[h], p.vc, p.vs, p.vsf, p.vg, row, lane);
      }
    }
    if (p.ik) put_row<IF>(ri, p.ic, p.is, p.isf, p.ig, (long)blk * kBlock + off, lane);
  }
}

template <int KVF>
cudaError_t launch_kv(const InsertParams& p, int num_sms, cudaStream_t st) {
  long grid = ((long)p.num_tokens + kInsertWarps - 1) / kInsertWarps;
  const long cap = (long)(num_sms > 0 ? num_sms : 1) * 16;  // the CTAs past those resident walk the rest
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  const bool h4 = p.H <= 4;
  switch (p.idx_fmt) {
    case FMT_BF16:
      if (h4) insert_kernel<KVF, FMT_BF16, 4><<<(unsigned)grid, 32 * kInsertWarps, 0, st>>>(p);
      else insert_kernel<KVF, FMT_BF16, 8><<<(unsigned)grid, 32 * kInsertWarps, 0, st>>>(p);
      break;
    case FMT_FP8:
      if (h4) insert_kernel<KVF, FMT_FP8, 4><<<(unsigned)grid, 32 * kInsertWarps, 0, st>>>(p);
      else insert_kernel<KVF, FMT_FP8, 8><<<(unsigned)grid, 32 * kInsertWarps, 0, st>>>(p);
      break;
    case FMT_NVFP4:
      if (h4) insert_kernel<KVF, FMT_NVFP4, 4><<<(unsigned)grid, 32 * kInsertWarps, 0, st>>>(p);
      else insert_kernel<KVF, FMT_NVFP4, 8><<<(unsigned)grid, 32 * kInsertWarps, 0, st>>>(p);
      break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_insert(const InsertParams& p, int num_sms, cudaStream_t st) {
  if (p.num_tokens == 0) return cudaSuccess;
  switch (p.kv_fmt) {
    case FMT_BF16: return launch_kv<FMT_BF16>(p, num_sms, st);
    case FMT_FP8: return launch_kv<FMT_FP8>(p, num_sms, st);
    case FMT_NVFP4: return launch_kv<FMT_NVFP4>(p, num_sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace msa
