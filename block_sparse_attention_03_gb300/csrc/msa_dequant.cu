// fp32 decode of stored cache elements (test hook msa_dequant_debug).
//
// Value definitions (vLLM Day-0 blog, section "MiniMax-M3.1 架构中的新特性" for
// NVFP4; "[M3] Enable FP8 sparse GQA" for the E4M3 KV cache):
//   BF16   the bits widened to fp32 (exact);
//   FP8    fp32(e4m3) * per-token fp32 scale, one round-to-nearest-even;
//   NVFP4  fp32(e2m1 * e4m3 block scale) * fp32 per-tensor scale; the inner
//          product is exact, so again one rounding.  With the cache's
//          MSA_NVFP4_E4M3_PRODUCT mode the product is first rounded to E4M3
//          (nearest even, saturating), as the Blackwell kernels' dequant does
//          ("NVIDIA Blackwell 优化的 MSA 内核").
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {

namespace {

__device__ __forceinline__ float e2m1_to_float(uint32_t nib) {
  const uint32_t h = e2m1x2_to_f16x2(nib & 0xfu);
  return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
}

// one thread per output element
__global__ void dequant_kernel(int fmt, int which, msa_cache_t c, const int32_t* phys, int32_t n, float* out) {
  const bool is_idx = which == 2;
  const int heads = is_idx ? 1 : c.num_kv_heads;
  const int D = 128;
  const size_t per_block = (size_t)heads * kBlock * D;
  const size_t total = per_block * n;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int bi = (int)(e / per_block);
    const size_t within = e % per_block;  // (head * 128 + token) * 128 + d
    const int d = (int)(within % D);
    const size_t ht = within / D;         // head * 128 + token
    const int pb = phys[bi];
    if (pb < 0 || pb >= c.num_blocks) {
      out[e] = __int_as_float(0x7fc00000);
      continue;
    }
    const size_t row = (size_t)pb * heads * kBlock + ht;  // global (block, head, token) row
    const void* data = is_idx ? c.idx : (which == 0 ? c.k : c.v);
    float v;
    if (fmt == FMT_BF16) {
      const uint16_t bits = static_cast<const uint16_t*>(data)[row * D + d];
      v = __uint_as_float((uint32_t)bits << 16);
    } else if (fmt == FMT_FP8) {
      const uint8_t code = static_cast<const uint8_t*>(data)[row * D + d];
      const float* sc = is_idx ? c.idx_scale : (which == 0 ? c.k_scale : c.v_scale);
      v = __fmul_rn(e4m3_to_float(code), sc[row]);
    } else {
      const uint8_t byte = static_cast<const uint8_t*>(data)[row * (D / 2) + d / 2];
      const uint8_t* sfp = static_cast<const uint8_t*>(is_idx ? c.idx_sf : (which == 0 ? c.k_sf : c.v_sf));
      const uint8_t sfc = sfp[row * (D / 16) + d / 16];
      const float gl = is_idx ? c.idx_global : (which == 0 ? c.k_global : c.v_global);
      float prod = __fmul_rn(e2m1_to_float((d & 1) ? (byte >> 4) : (byte & 0xf)), e4m3_to_float(sfc));
      if (c.nvfp4_mode == MSA_NVFP4_E4M3_PRODUCT) prod = e4m3_to_float((uint8_t)(pack_e4m3x2(prod, 0.f) & 0xffu));
      v = __fmul_rn(prod, gl);
    }
    out[e] = v;
  }
}

}  // namespace

cudaError_t launch_dequant(int fmt, int which, const msa_cache_t& c, const int32_t* phys, int32_t n, float* out,
                           cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const size_t total = (size_t)(which == 2 ? 1 : c.num_kv_heads) * kBlock * 128 * n;
  const unsigned grid = (unsigned)((total + 255) / 256 < 65535 ? (total + 255) / 256 : 65535);
  dequant_kernel<<<grid, 256, 0, st>>>(fmt, which, c, phys, n, out);
  return cudaGetLastError();
}

}  // namespace msa
