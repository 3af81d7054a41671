// Query-operand preparation: turns query rows into per-lane MMA B fragments.
//
// The indexer and the attend kernels compute S^T = Keys * Queries^T with the
// keys as the MMA "A" operand (rows = keys) and the queries as "B"
// (columns = query rows).  The queries of one unit (a sequence for the
// indexer, a (sequence, group) pair for the attend) are constant over the
// whole key scan, so their fragments are built once here:
//
//   e4m3 keys  (mma m16n8k32 e4m3): b0 = dims 32ks+4j..+3, b1 = dims 32ks+16+4j..+3
//   bf16 keys  (mma m16n8k16 bf16): b0 = dims 16ks+2j,+1,  b1 = dims 16ks+8+2j,+1
//   NVFP4 keys (mma m16n8k16 f16, dequantized in registers in a permuted
//               k order):           b0 = dims 32j+4ks,+1,  b1 = dims 32j+4ks+2,+3
// with lane = 4 * column + j.  A bf16 query meeting e4m3 keys is scaled by a
// power of two per column (exact) and split into hi + lo e4m3 terms, which
// together carry all 8 significant bits of bf16; the kernels run one MMA per
// term into the same accumulator.  The per-column factor (2^-e, the query's
// fp32 scale and a caller constant) is applied to the MMA result.
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {

namespace {

__device__ __forceinline__ float load_q(const void* q, int is_fp8, size_t idx) {
  if (is_fp8) return e4m3_to_float(static_cast<const uint8_t*>(q)[idx]);
  return __bfloat162float(static_cast<const __nv_bfloat16*>(q)[idx]);
}

constexpr int kMaxPrepCols = 64;

__global__ void __launch_bounds__(256) prep_kernel(const PrepParams p, int a, int u2, int b, int c2, int c) {
  __shared__ float qs[kMaxPrepCols][kDim + 1];
  __shared__ float cfac[kMaxPrepCols];
  __shared__ float pscale[kMaxPrepCols];
  const int unit = blockIdx.x;
  const FragGeom gm = p.geom;
  const int ncols_pad = gm.nt * 8;
  for (int i = threadIdx.x; i < ncols_pad * kDim; i += blockDim.x) {
    const int col = i / kDim, d = i % kDim;
    float v = 0.f;
    if (col < gm.cols) {
      const size_t row = (size_t)a * (unit / u2) + (size_t)b * (unit % u2) + (size_t)c * (col / c2) + (col % c2);
      v = load_q(p.q, p.q_is_fp8, row * kDim + d);
    }
    qs[col][d] = v;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int col = warp; col < ncols_pad; col += blockDim.x >> 5) {
    float m = 0.f;
    for (int d = lane; d < kDim; d += 32) m = fmaxf(m, fabsf(qs[col][d]));
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) {
      float base = p.q_is_fp8 ? p.q_scale : 1.f;
      int e = 0;
      if (p.key_fmt == FMT_FP8 && !p.q_is_fp8) e = pow2_fit(m, 448.f);
      if (p.key_fmt == FMT_NVFP4 && !p.q_is_fp8) e = pow2_fit(m, 16384.f);
      pscale[col] = ldexpf(1.f, e);
      cfac[col] = ldexpf(1.f, -e) * base * p.col_const;
    }
  }
  __syncthreads();
  if (threadIdx.x < ncols_pad) p.colf[(size_t)unit * ncols_pad + threadIdx.x] = cfac[threadIdx.x];
  const int words = gm.words_per_unit();
  uint32_t* out = p.frag + (size_t)unit * words;
  for (int w = threadIdx.x; w < words; w += blockDim.x) {
    // w = ((((sp * nt) + ntile) * ks + kstep) * 2 + reg) * 32 + ln
    const int ln = w & 31;
    const int reg = (w >> 5) & 1;
    const int kstep = (w >> 6) % gm.ks;
    const int ntile = ((w >> 6) / gm.ks) % gm.nt;
    const int sp = ((w >> 6) / gm.ks) / gm.nt;
    const int col = ntile * 8 + (ln >> 2), j = ln & 3;
    const float ps = pscale[col];
    uint32_t word = 0;
    if (p.key_fmt == FMT_FP8) {
      const int d0 = 32 * kstep + 16 * reg + 4 * j;
      if (p.q_is_fp8) {
        // raw e4m3 codes, unchanged
        for (int t = 0; t < 4; ++t) {
          const size_t row =
              (size_t)a * (unit / u2) + (size_t)b * (unit % u2) + (size_t)c * (col / c2) + (col % c2);
          uint32_t code = (col < gm.cols) ? static_cast<const uint8_t*>(p.q)[row * kDim + d0 + t] : 0u;
          word |= code << (8 * t);
        }
      } else {
        for (int t = 0; t < 4; t += 2) {
          float h0, l0, h1, l1;
          split_e4m3(qs[col][d0 + t] * ps, h0, l0);
          split_e4m3(qs[col][d0 + t + 1] * ps, h1, l1);
          const uint16_t pr = (sp == 0) ? pack_e4m3x2(h0, h1) : pack_e4m3x2(l0, l1);
          word |= (uint32_t)pr << (8 * t);
        }
      }
    } else if (p.key_fmt == FMT_BF16) {
      const int d0 = 16 * kstep + 8 * reg + 2 * j;
      word = pack_bf16x2(qs[col][d0], qs[col][d0 + 1]);
    } else {
      const int d0 = 32 * j + 4 * kstep + 2 * reg;
      word = pack_f16x2(qs[col][d0] * ps, qs[col][d0 + 1] * ps);
    }
    out[w] = word;
  }
}

}  // namespace

// Row of (unit, col) = a*(unit/u2) + b*(unit%u2) + c*(col/c2) + col%c2, set by
// the caller through PrepParams::units and the geometry; see launch_prep_rows.
cudaError_t launch_prep_rows(const PrepParams& p, int a, int u2, int b, int c2, int c, cudaStream_t st) {
  if (p.geom.nt * 8 > kMaxPrepCols) return cudaErrorInvalidValue;
  prep_kernel<<<p.units, 256, 0, st>>>(p, a, u2, b, c2, c);
  return cudaGetLastError();
}

}  // namespace msa
