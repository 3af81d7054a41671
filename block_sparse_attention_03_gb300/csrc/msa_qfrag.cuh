// Query-side MMA operand ("B" fragments) built in registers by each warp.
//
// The indexer and attend kernels compute S^T = Keys * Queries^T with keys as
// the MMA rows and the (few) query rows of one unit as the 8-wide column
// tiles.  Lane l = 4*n + j of a warp holds, for column n of each tile, the
// query values at the k positions the key operand puts in the same slots:
//   e4m3 keys  (mma m16n8k32 e4m3): b0 = dims 32ks+4j..+3,  b1 = dims 32ks+16+4j..+3
//   bf16 keys  (mma m16n8k16 bf16): b0 = dims 16ks+2j,+1,   b1 = dims 16ks+8+2j,+1
//   NVFP4 keys (mma m16n8k16 f16, keys dequantized in a permuted k order):
//                                   b0 = dims 32j+4ks,+1,   b1 = dims 32j+4ks+2,+3
// A bf16 query meeting e4m3 keys is scaled by a power of two per column
// (exact) and split into e4m3 hi + lo terms, which together carry all 8
// significant bits of bf16 (SP = 2: one MMA per term into one accumulator).
// A bf16 query meeting NVFP4 keys becomes f16 after a power-of-two scale that
// keeps it in f16's normal range.  E4M3 queries enter unchanged (e4m3 keys)
// or exactly widened (bf16 / f16).  The column factor (2^-e, the query's
// per-tensor scale and a caller constant) multiplies the MMA result.
#pragma once

#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {

__device__ __forceinline__ float q_elem(const void* q, bool q_fp8, size_t idx) {
  if (q_fp8) return e4m3_to_float(static_cast<const uint8_t*>(q)[idx]);
  return __bfloat162float(static_cast<const __nv_bfloat16*>(q)[idx]);
}

// dims held by slot (ks, reg, t) of lane j for a key format (t = element in the register)
template <int KEYFMT>
__device__ __forceinline__ int frag_dim(int ks, int reg, int t, int j) {
  if constexpr (KEYFMT == FMT_FP8) return 32 * ks + 16 * reg + 4 * j + t;        // t in 0..3
  else if constexpr (KEYFMT == FMT_BF16) return 16 * ks + 8 * reg + 2 * j + t;   // t in 0..1
  else return 32 * j + 4 * ks + 2 * reg + t;                                     // t in 0..1
}

// rows[nt]: element offset of column nt*8 + (lane>>2) in q (or -1 for padding).
template <int KEYFMT, int NT, int SP, int KS>
__device__ __forceinline__ void build_qfrag(const void* q, bool q_fp8, const long (&rows)[NT], float q_scale,
                                            float col_const, uint32_t (&bq)[SP][NT][KS][2], float (&colf)[NT][2],
                                            int lane) {
  const int j = lane & 3;
  constexpr int TPR = (KEYFMT == FMT_FP8) ? 4 : 2;  // elements per register
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const long row = rows[nt];
    float vals[KS][2][TPR];
    float amax = 0.f;
    if (KEYFMT == FMT_FP8 && !q_fp8) {
      // e4m3 keys, bf16 query: a register's 4 dims are contiguous and 8-byte
      // aligned (rows start at multiples of 4 elements): one 8-byte load each
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int rg = 0; rg < 2; ++rg) {
          uint2 w = make_uint2(0u, 0u);
          if (row >= 0)
            w = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(q) + (size_t)row +
                                                frag_dim<KEYFMT>(ks, rg, 0, j));
          const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
          const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
          const float f[4] = {a.x, a.y, b.x, b.y};
#pragma unroll
          for (int t = 0; t < TPR; ++t) {
            vals[ks][rg][t] = f[t];
            amax = fmaxf(amax, fabsf(f[t]));
          }
        }
    } else {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int rg = 0; rg < 2; ++rg)
#pragma unroll
          for (int t = 0; t < TPR; ++t) {
            const float v = (row >= 0) ? q_elem(q, q_fp8, (size_t)row + frag_dim<KEYFMT>(ks, rg, t, j)) : 0.f;
            vals[ks][rg][t] = v;
            amax = fmaxf(amax, fabsf(v));
          }
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int e = 0;
    if (!q_fp8 && KEYFMT == FMT_FP8) e = pow2_fit(amax, 448.f);
    if (!q_fp8 && KEYFMT == FMT_NVFP4) e = pow2_fit(amax, 16384.f);
    const float ps = ldexpf(1.f, e);
    const float cf = ldexpf(1.f, -e) * (q_fp8 ? q_scale : 1.f) * col_const;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int rg = 0; rg < 2; ++rg) {
        if constexpr (KEYFMT == FMT_FP8) {
          if (q_fp8) {
            uint32_t w = 0;
            if (row >= 0) {
              const uint8_t* qb = static_cast<const uint8_t*>(q) + row + frag_dim<KEYFMT>(ks, rg, 0, j);
#pragma unroll
              for (int t = 0; t < 4; ++t) w |= (uint32_t)qb[t] << (8 * t);
            }
            bq[0][nt][ks][rg] = w;
            if constexpr (SP == 2) bq[1][nt][ks][rg] = 0u;
          } else {
            float h[4], l[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) split_e4m3(vals[ks][rg][t] * ps, h[t], l[t]);
            bq[0][nt][ks][rg] = (uint32_t)pack_e4m3x2(h[0], h[1]) | ((uint32_t)pack_e4m3x2(h[2], h[3]) << 16);
            if constexpr (SP == 2)
              bq[1][nt][ks][rg] = (uint32_t)pack_e4m3x2(l[0], l[1]) | ((uint32_t)pack_e4m3x2(l[2], l[3]) << 16);
          }
        } else if constexpr (KEYFMT == FMT_BF16) {
          bq[0][nt][ks][rg] = pack_bf16x2(vals[ks][rg][0], vals[ks][rg][1]);
        } else {
          bq[0][nt][ks][rg] = pack_f16x2(vals[ks][rg][0] * ps, vals[ks][rg][1] * ps);
        }
      }
    // factor of the columns this lane's accumulators hold: nt*8 + 2j + c
#pragma unroll
    for (int c = 0; c < 2; ++c) colf[nt][c] = __shfl_sync(0xffffffffu, cf, 4 * (2 * j + c));
  }
}

}  // namespace msa

namespace msa {

// The same fragments written to global memory by a whole CTA (runtime
// geometry), for kernels that prepare them once per unit for a later kernel.
// qs: shared scratch of at least geom.nt*8 rows x (kDim+1) floats.
// row_of(col): element offset of query column col in q, or -1 (padding).
template <typename RowOf>
__device__ void write_qfrag(const void* q, bool q_fp8, RowOf row_of, float q_scale, float col_const, int key_fmt,
                            const FragGeom gm, float* qs, float* pscale, uint32_t* frag, float* colf) {
  const int ncols = gm.nt * 8;
  for (int i = threadIdx.x; i < ncols * kDim; i += blockDim.x) {
    const int col = i / kDim, d = i % kDim;
    const long row = row_of(col);
    qs[col * (kDim + 1) + d] = (row >= 0) ? q_elem(q, q_fp8, (size_t)row + d) : 0.f;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int col = warp; col < ncols; col += blockDim.x >> 5) {
    float m = 0.f;
    for (int d = lane; d < kDim; d += 32) m = fmaxf(m, fabsf(qs[col * (kDim + 1) + d]));
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) {
      int e = 0;
      if (key_fmt == FMT_FP8 && !q_fp8) e = pow2_fit(m, 448.f);
      if (key_fmt == FMT_NVFP4 && !q_fp8) e = pow2_fit(m, 16384.f);
      pscale[col] = ldexpf(1.f, e);
      colf[col] = ldexpf(1.f, -e) * (q_fp8 ? q_scale : 1.f) * col_const;
    }
  }
  __syncthreads();
  const int words = gm.words_per_unit();
  for (int w = threadIdx.x; w < words; w += blockDim.x) {
    // w = ((((sp * nt) + ntile) * ks + kstep) * 2 + reg) * 32 + ln
    const int ln = w & 31, reg = (w >> 5) & 1;
    const int kstep = (w >> 6) % gm.ks;
    const int ntile = ((w >> 6) / gm.ks) % gm.nt;
    const int sp = ((w >> 6) / gm.ks) / gm.nt;
    const int col = ntile * 8 + (ln >> 2), j = ln & 3;
    const float ps = pscale[col];
    const float* qc = qs + col * (kDim + 1);
    uint32_t word = 0;
    if (key_fmt == FMT_FP8) {
      const int d0 = 32 * kstep + 16 * reg + 4 * j;
      if (q_fp8) {
        const long row = row_of(col);
        for (int t = 0; t < 4; ++t) {
          const uint32_t code = (row >= 0) ? static_cast<const uint8_t*>(q)[row + d0 + t] : 0u;
          word |= code << (8 * t);
        }
        if (sp == 1) word = 0u;
      } else {
        for (int t = 0; t < 4; t += 2) {
          float h0, l0, h1, l1;
          split_e4m3(qc[d0 + t] * ps, h0, l0);
          split_e4m3(qc[d0 + t + 1] * ps, h1, l1);
          const uint16_t pr = (sp == 0) ? pack_e4m3x2(h0, h1) : pack_e4m3x2(l0, l1);
          word |= (uint32_t)pr << (8 * t);
        }
      }
    } else if (key_fmt == FMT_BF16) {
      const int d0 = 16 * kstep + 8 * reg + 2 * j;
      word = pack_bf16x2(qc[d0], qc[d0 + 1]);
    } else {
      const int d0 = 32 * j + 4 * kstep + 2 * reg;
      word = pack_f16x2(qc[d0] * ps, qc[d0 + 1] * ps);
    }
    frag[w] = word;
  }
}

}  // namespace msa
