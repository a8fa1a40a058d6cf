// prep_mma.cu -- fused chunk preparation for bf16 inputs on the tensor cores.
//
// One CTA (8 warps) per chunk of C = 128 tokens computes, following "PaTH
// Attention: Position Encoding via Accumulating Householder Transformations"
// (discussion slides), frames "A triangular representation makes paths
// computable" and "Backup: fix orientation before implementing UT products":
//
//   L   = strictLower(D W W^T)             bf16 MMA, exact fp32 products
//   X   = (I + L)^{-1}, U = X D            fp32, recursive doubling in smem
//   TK  = U strictLower(W K^T)             tf32 MMA
//   UW  = U W                              tf32 MMA
//   kr  = K - TK^T W                       tf32 MMA  -> workspace (bf16)
//   ngt = -(UW^T W)                        tf32 MMA  -> workspace (bf16)
//   sdt = log2(e) (scale (lower(Q K^T) - lower(Q W^T) TK) + gate), [j][i]
//   ql  = Q - lower(Q W^T) UW              tf32 MMA  -> workspace (fp32)
//
// Products whose operands are bf16 inputs (the four Gram blocks) use
// mma.m16n8k16 bf16 with fp32 accumulation and are exact.  Products with a
// computed fp32 operand round that operand to tf32 (2^-11 relative) and
// accumulate in fp32; the results are then rounded to bf16 (kr, ngt) or feed
// bf16 operands of the scan (ql), so the tf32 rounding stays below the
// rounding those outputs get anyway.  Warp w owns rows [16w, 16w + 16) of
// every C-row product; lower(Q W^T) never leaves registers (its accumulator
// fragments are re-laid out as tf32 A fragments with quad shuffles).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "prep_solve.cuh"

namespace pathattn {
namespace {

constexpr int kPC = 128;        // chunk length
constexpr int kPThreads = 256;  // 8 warps

template <int D>
struct PCfg {
  static constexpr int SW = D + 8;    // bf16 row stride of W, K (elements)
  static constexpr int SU = kPC + 4;  // fp32 stride of L / X / U (A-operand access)
  static constexpr int SK = kPC + 8;  // fp32 stride of strictLower(WK^T) / TK (B access)
  static constexpr int SD = D + 8;    // fp32 stride of UW (B access)
  static constexpr size_t kWBytes = size_t(kPC) * SW * 2;
  static constexpr size_t kUBytes = size_t(kPC) * (SU > SD ? SU : SD) * 4;
  static constexpr size_t kBBytes = size_t(kPC) * SK * 4;
  static constexpr size_t kSmem = 2 * kWBytes + kUBytes + kBBytes + 2 * kPC * 4;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t tf32r(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ uint32_t bf16_bits_to_f32(uint16_t h) {
  return static_cast<uint32_t>(h) << 16;
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// ---- fragment loads (g = lane / 4, t = lane % 4)
// bf16 A (16 x 16) of a row-major bf16 matrix s[row][col]
__device__ __forceinline__ void lda_bf16(uint32_t (&a)[4], const __nv_bfloat16* s, int S, int m0,
                                         int k0, int g, int t) {
  a[0] = *reinterpret_cast<const uint32_t*>(s + (m0 + g) * S + k0 + 2 * t);
  a[1] = *reinterpret_cast<const uint32_t*>(s + (m0 + g + 8) * S + k0 + 2 * t);
  a[2] = *reinterpret_cast<const uint32_t*>(s + (m0 + g) * S + k0 + 2 * t + 8);
  a[3] = *reinterpret_cast<const uint32_t*>(s + (m0 + g + 8) * S + k0 + 2 * t + 8);
}
// bf16 B (16 x 8) with B[k][n] = s[n][k]
__device__ __forceinline__ void ldb_bf16(uint32_t (&b)[2], const __nv_bfloat16* s, int S, int n0,
                                         int k0, int g, int t) {
  b[0] = *reinterpret_cast<const uint32_t*>(s + (n0 + g) * S + k0 + 2 * t);
  b[1] = *reinterpret_cast<const uint32_t*>(s + (n0 + g) * S + k0 + 2 * t + 8);
}
// tf32 A (16 x 8) of a row-major fp32 matrix s[m][k] (values already tf32)
__device__ __forceinline__ void lda_f32(uint32_t (&a)[4], const float* s, int S, int m0, int k0,
                                        int g, int t) {
  a[0] = __float_as_uint(s[(m0 + g) * S + k0 + t]);
  a[1] = __float_as_uint(s[(m0 + g + 8) * S + k0 + t]);
  a[2] = __float_as_uint(s[(m0 + g) * S + k0 + t + 4]);
  a[3] = __float_as_uint(s[(m0 + g + 8) * S + k0 + t + 4]);
}
// tf32 A (16 x 8) with A[m][k] = s[k][m] (fp32, values already tf32)
__device__ __forceinline__ void lda_f32_t(uint32_t (&a)[4], const float* s, int S, int m0, int k0,
                                          int g, int t) {
  a[0] = __float_as_uint(s[(k0 + t) * S + m0 + g]);
  a[1] = __float_as_uint(s[(k0 + t) * S + m0 + g + 8]);
  a[2] = __float_as_uint(s[(k0 + t + 4) * S + m0 + g]);
  a[3] = __float_as_uint(s[(k0 + t + 4) * S + m0 + g + 8]);
}
// tf32 B (8 x 8) of a row-major fp32 matrix s[k][n] (values already tf32)
__device__ __forceinline__ void ldb_f32(uint32_t (&b)[2], const float* s, int S, int n0, int k0,
                                        int g, int t) {
  b[0] = __float_as_uint(s[(k0 + t) * S + n0 + g]);
  b[1] = __float_as_uint(s[(k0 + t + 4) * S + n0 + g]);
}
// tf32 B (8 x 8) of a row-major bf16 matrix s[k][n] (exact in tf32)
__device__ __forceinline__ void ldb_bf16_as_tf32(uint32_t (&b)[2], const __nv_bfloat16* s, int S,
                                                 int n0, int k0, int g, int t) {
  const uint16_t* h = reinterpret_cast<const uint16_t*>(s);
  b[0] = bf16_bits_to_f32(h[(k0 + t) * S + n0 + g]);
  b[1] = bf16_bits_to_f32(h[(k0 + t + 4) * S + n0 + g]);
}
// bf16 A (16 x 16) straight from global memory rows (rows >= nrows read as 0)
__device__ __forceinline__ void lda_bf16_g(uint32_t (&a)[4], const __nv_bfloat16* rows, int D,
                                           int nrows, int m0, int k0, int g, int t) {
  const int r0 = m0 + g, r1 = m0 + g + 8;
  a[0] = r0 < nrows ? __ldg(reinterpret_cast<const unsigned int*>(rows + r0 * D + k0 + 2 * t)) : 0u;
  a[1] = r1 < nrows ? __ldg(reinterpret_cast<const unsigned int*>(rows + r1 * D + k0 + 2 * t)) : 0u;
  a[2] = r0 < nrows ? __ldg(reinterpret_cast<const unsigned int*>(rows + r0 * D + k0 + 2 * t + 8)) : 0u;
  a[3] = r1 < nrows ? __ldg(reinterpret_cast<const unsigned int*>(rows + r1 * D + k0 + 2 * t + 8)) : 0u;
}

// Accumulator fragments of a 16 x 8 tile (n-tile s of a 16-row strip) ->
// tf32 A fragment of k-slab s (same 8 columns).  Quad-local shuffles.
__device__ __forceinline__ void acc_to_a(uint32_t (&a)[4], const float (&c)[4], int g, int t) {
  const int srcA = g * 4 + (t >> 1), srcB = g * 4 + 2 + (t >> 1);
  const bool odd = t & 1;
  const float x0 = __shfl_sync(0xffffffffu, c[0], srcA), x1 = __shfl_sync(0xffffffffu, c[1], srcA);
  const float y0 = __shfl_sync(0xffffffffu, c[2], srcA), y1 = __shfl_sync(0xffffffffu, c[3], srcA);
  const float u0 = __shfl_sync(0xffffffffu, c[0], srcB), u1 = __shfl_sync(0xffffffffu, c[1], srcB);
  const float v0 = __shfl_sync(0xffffffffu, c[2], srcB), v1 = __shfl_sync(0xffffffffu, c[3], srcB);
  a[0] = tf32r(odd ? x1 : x0);
  a[1] = tf32r(odd ? y1 : y0);
  a[2] = tf32r(odd ? u1 : u0);
  a[3] = tf32r(odd ? v1 : v0);
}

template <int D, bool kGate>
__global__ void __launch_bounds__(kPThreads, 1)
    prep_mma_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                    const __nv_bfloat16* __restrict__ w, const float* __restrict__ beta,
                    const float* __restrict__ lam2, __nv_bfloat16* __restrict__ kr,
                    float* __restrict__ ql, __nv_bfloat16* __restrict__ ngt,
                    float* __restrict__ sdt, int T, int Np, float sl2) {
  using Cfg = PCfg<D>;
  constexpr int SW = Cfg::SW, SU = Cfg::SU, SK = Cfg::SK, SD = Cfg::SD;
  constexpr int NT = kPC / 8;  // n-tiles of a C-column product
  constexpr int ND = D / 8;    // n-tiles of a D-column product
  extern __shared__ __align__(16) uint8_t smem[];
  __nv_bfloat16* sW = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(smem + Cfg::kWBytes);
  float* sU = reinterpret_cast<float*>(smem + 2 * Cfg::kWBytes);
  float* sB = reinterpret_cast<float*>(smem + 2 * Cfg::kWBytes + Cfg::kUBytes);
  float* sBeta = reinterpret_cast<float*>(smem + 2 * Cfg::kWBytes + Cfg::kUBytes + Cfg::kBBytes);
  float* sLam = sBeta + kPC;

  const int ch = blockIdx.x, bh = ch / Np, n = ch - bh * Np, t0 = n * kPC;
  const int nrows = min(kPC, T - t0);  // real tokens in this chunk
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int m0 = warp * 16;
  const size_t row0 = static_cast<size_t>(bh) * T + t0;
  const __nv_bfloat16* Wg = w + row0 * D;
  const __nv_bfloat16* Kg = k + row0 * D;
  const __nv_bfloat16* Qg = q + row0 * D;

  // ---- stage W, K, beta (and the gate prefix) in shared memory; all 16-byte
  // copies in flight at once (cp.async), padding rows zero-filled
  for (int e = tid; e < kPC * D / 8; e += kPThreads) {
    const int r = e / (D / 8), c8 = e % (D / 8);
    __nv_bfloat16* dw = sW + r * SW + c8 * 8;
    __nv_bfloat16* dk = sK + r * SW + c8 * 8;
    if (r < nrows) {
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dw)),
                   "l"(Wg + r * D + c8 * 8) : "memory");
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dk)),
                   "l"(Kg + r * D + c8 * 8) : "memory");
    } else {
      *reinterpret_cast<uint4*>(dw) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(dk) = make_uint4(0, 0, 0, 0);
    }
  }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  if (tid < kPC) {
    sBeta[tid] = tid < nrows ? beta[row0 + tid] : 0.f;
    if (kGate) sLam[tid] = lam2[static_cast<size_t>(bh) * Np * kPC + t0 + tid];
  }
  __syncthreads();

  // ---- Gram blocks: L = strictLower(D W W^T) -> sU (fp32), strictLower(W K^T) -> sB (tf32)
  {
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < D; k0 += 16) {
      uint32_t a[4];
      lda_bf16(a, sW, SW, m0, k0, g, t);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        uint32_t b[2];
        ldb_bf16(b, sW, SW, j * 8, k0, g, t);
        mma_bf16(acc[j], a, b);
      }
    }
    const float b0 = sBeta[m0 + g], b1 = sBeta[m0 + g + 8];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int c = j * 8 + 2 * t, r0 = m0 + g, r1 = m0 + g + 8;
      sU[r0 * SU + c] = c < r0 ? acc[j][0] * b0 : 0.f;
      sU[r0 * SU + c + 1] = c + 1 < r0 ? acc[j][1] * b0 : 0.f;
      sU[r1 * SU + c] = c < r1 ? acc[j][2] * b1 : 0.f;
      sU[r1 * SU + c + 1] = c + 1 < r1 ? acc[j][3] * b1 : 0.f;
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < D; k0 += 16) {
      uint32_t a[4];
      lda_bf16(a, sW, SW, m0, k0, g, t);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        uint32_t b[2];
        ldb_bf16(b, sK, SW, j * 8, k0, g, t);
        mma_bf16(acc[j], a, b);
      }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int c = j * 8 + 2 * t, r0 = m0 + g, r1 = m0 + g + 8;
      sB[r0 * SK + c] = __uint_as_float(c < r0 ? tf32r(acc[j][0]) : 0u);
      sB[r0 * SK + c + 1] = __uint_as_float(c + 1 < r0 ? tf32r(acc[j][1]) : 0u);
      sB[r1 * SK + c] = __uint_as_float(c < r1 ? tf32r(acc[j][2]) : 0u);
      sB[r1 * SK + c + 1] = __uint_as_float(c + 1 < r1 ? tf32r(acc[j][3]) : 0u);
    }
  }
  __syncthreads();

  // ---- X = (I + L)^{-1}; U = X diag(beta), rounded to tf32
  invert_unit_lower<SU>(sU, tid);
  for (int e = tid; e < kPC * kPC; e += kPThreads) {
    const int i = e / kPC, c = e % kPC;
    sU[i * SU + c] = __uint_as_float(c <= i ? tf32r(sU[i * SU + c] * sBeta[c]) : 0u);
  }
  __syncthreads();

  // ---- TK = U strictLower(W K^T),  UW = U W   (U lower: k-slabs <= row)
  {
    float tk[NT][4], uw[ND][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) tk[j][0] = tk[j][1] = tk[j][2] = tk[j][3] = 0.f;
#pragma unroll
    for (int j = 0; j < ND; ++j) uw[j][0] = uw[j][1] = uw[j][2] = uw[j][3] = 0.f;
    const int kend = m0 + 16;
    for (int k0 = 0; k0 < kend; k0 += 8) {
      uint32_t a[4];
      lda_f32(a, sU, SU, m0, k0, g, t);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        uint32_t b[2];
        ldb_f32(b, sB, SK, j * 8, k0, g, t);
        mma_tf32(tk[j], a, b);
      }
#pragma unroll
      for (int j = 0; j < ND; ++j) {
        uint32_t b[2];
        ldb_bf16_as_tf32(b, sW, SW, j * 8, k0, g, t);
        mma_tf32(uw[j], a, b);
      }
    }
    __syncthreads();  // every warp is done reading U and strictLower(W K^T)
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int c = j * 8 + 2 * t, r0 = m0 + g, r1 = m0 + g + 8;
      sB[r0 * SK + c] = __uint_as_float(tf32r(tk[j][0]));
      sB[r0 * SK + c + 1] = __uint_as_float(tf32r(tk[j][1]));
      sB[r1 * SK + c] = __uint_as_float(tf32r(tk[j][2]));
      sB[r1 * SK + c + 1] = __uint_as_float(tf32r(tk[j][3]));
    }
#pragma unroll
    for (int j = 0; j < ND; ++j) {
      const int c = j * 8 + 2 * t, r0 = m0 + g, r1 = m0 + g + 8;
      sU[r0 * SD + c] = __uint_as_float(tf32r(uw[j][0]));
      sU[r0 * SD + c + 1] = __uint_as_float(tf32r(uw[j][1]));
      sU[r1 * SD + c] = __uint_as_float(tf32r(uw[j][2]));
      sU[r1 * SD + c + 1] = __uint_as_float(tf32r(uw[j][3]));
    }
  }
  __syncthreads();
  // now: sB = TK [t][j] (stride SK), sU = UW [t][n] (stride SD)

  // ---- kr = K - TK^T W   (TK^T[j][t] nonzero only for t > j)
  {
    float acc[ND][4];
#pragma unroll
    for (int j = 0; j < ND; ++j) {
      const int c = j * 8 + 2 * t, r0 = m0 + g, r1 = m0 + g + 8;
      acc[j][0] = __bfloat162float(sK[r0 * SW + c]);
      acc[j][1] = __bfloat162float(sK[r0 * SW + c + 1]);
      acc[j][2] = __bfloat162float(sK[r1 * SW + c]);
      acc[j][3] = __bfloat162float(sK[r1 * SW + c + 1]);
    }
    for (int k0 = m0; k0 < kPC; k0 += 8) {
      uint32_t a[4];
      lda_f32_t(a, sB, SK, m0, k0, g, t);
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] ^= 0x80000000u;  // -TK^T
#pragma unroll
      for (int j = 0; j < ND; ++j) {
        uint32_t b[2];
        ldb_bf16_as_tf32(b, sW, SW, j * 8, k0, g, t);
        mma_tf32(acc[j], a, b);
      }
    }
    __nv_bfloat16* out = kr + static_cast<size_t>(ch) * kPC * D;
#pragma unroll
    for (int j = 0; j < ND; ++j) {
      const int c = j * 8 + 2 * t, r0 = m0 + g, r1 = m0 + g + 8;
      *reinterpret_cast<__nv_bfloat162*>(out + r0 * D + c) = __floats2bfloat162_rn(acc[j][0], acc[j][1]);
      *reinterpret_cast<__nv_bfloat162*>(out + r1 * D + c) = __floats2bfloat162_rn(acc[j][2], acc[j][3]);
    }
  }

  // ---- ngt = -(UW^T W): rows n (D of them), columns f; K = chunk tokens
  {
    constexpr int kStrips = D / 16;             // 16-row strips of the D x D result
    constexpr int kSplit = 8 / kStrips;         // warps sharing one strip
    constexpr int kTiles = ND / kSplit;         // n-tiles per warp
    const int sm0 = (warp % kStrips) * 16, nt0 = (warp / kStrips) * kTiles;
    float acc[kTiles][4];
#pragma unroll
    for (int j = 0; j < kTiles; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    for (int k0 = 0; k0 < kPC; k0 += 8) {
      uint32_t a[4];
      lda_f32_t(a, sU, SD, sm0, k0, g, t);
#pragma unroll
      for (int j = 0; j < kTiles; ++j) {
        uint32_t b[2];
        ldb_bf16_as_tf32(b, sW, SW, (nt0 + j) * 8, k0, g, t);
        mma_tf32(acc[j], a, b);
      }
    }
    __nv_bfloat16* out = ngt + static_cast<size_t>(ch) * D * D;
#pragma unroll
    for (int j = 0; j < kTiles; ++j) {
      const int c = (nt0 + j) * 8 + 2 * t, r0 = sm0 + g, r1 = sm0 + g + 8;
      *reinterpret_cast<__nv_bfloat162*>(out + r0 * D + c) = __floats2bfloat162_rn(-acc[j][0], -acc[j][1]);
      *reinterpret_cast<__nv_bfloat162*>(out + r1 * D + c) = __floats2bfloat162_rn(-acc[j][2], -acc[j][3]);
    }
  }

  // ---- lower(Q W^T) (kept in registers) and Q K^T
  float pqk[NT][4];
  uint32_t aqw[NT][4];  // tf32 A fragments of lower(Q W^T), k-slab j = n-tile j
  {
    float pqw[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      pqw[j][0] = pqw[j][1] = pqw[j][2] = pqw[j][3] = 0.f;
      pqk[j][0] = pqk[j][1] = pqk[j][2] = pqk[j][3] = 0.f;
    }
#pragma unroll
    for (int k0 = 0; k0 < D; k0 += 16) {
      uint32_t a[4];
      lda_bf16_g(a, Qg, D, nrows, m0, k0, g, t);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        uint32_t b[2];
        ldb_bf16(b, sW, SW, j * 8, k0, g, t);
        mma_bf16(pqw[j], a, b);
        ldb_bf16(b, sK, SW, j * 8, k0, g, t);
        mma_bf16(pqk[j], a, b);
      }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int c = j * 8 + 2 * t, r0 = m0 + g, r1 = m0 + g + 8;
      pqw[j][0] = c <= r0 ? -pqw[j][0] : 0.f;  // negated: both uses subtract
      pqw[j][1] = c + 1 <= r0 ? -pqw[j][1] : 0.f;
      pqw[j][2] = c <= r1 ? -pqw[j][2] : 0.f;
      pqw[j][3] = c + 1 <= r1 ? -pqw[j][3] : 0.f;
      acc_to_a(aqw[j], pqw[j], g, t);
    }
  }

  // ---- diagonal logits: Q K^T - lower(Q W^T) TK, masked, scaled, gated, transposed
  {
    const int kslabs = (m0 + 16) / 8;  // lower(Q W^T)[i][s] nonzero only for s <= i
#pragma unroll
    for (int s = 0; s < NT; ++s) {
      if (s < kslabs) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          uint32_t b[2];
          ldb_f32(b, sB, SK, j * 8, s * 8, g, t);
          mma_tf32(pqk[j], aqw[s], b);
        }
      }
    }
    float* out = sdt + static_cast<size_t>(ch) * kPC * kPC;
    const int r0 = m0 + g, r1 = m0 + g + 8;
    const float l0 = kGate ? sLam[r0] : 0.f, l1 = kGate ? sLam[r1] : 0.f;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int c = j * 8 + 2 * t;
      const float g0 = kGate ? sLam[c] : 0.f, g1 = kGate ? sLam[c + 1] : 0.f;
      out[c * kPC + r0] = c <= r0 ? fmaf(pqk[j][0], sl2, l0 - g0) : -INFINITY;
      out[(c + 1) * kPC + r0] = c + 1 <= r0 ? fmaf(pqk[j][1], sl2, l0 - g1) : -INFINITY;
      out[c * kPC + r1] = c <= r1 ? fmaf(pqk[j][2], sl2, l1 - g0) : -INFINITY;
      out[(c + 1) * kPC + r1] = c + 1 <= r1 ? fmaf(pqk[j][3], sl2, l1 - g1) : -INFINITY;
    }
  }

  // ---- ql = Q - lower(Q W^T) UW
  {
    float acc[ND][4];
    const int r0 = m0 + g, r1 = m0 + g + 8;
#pragma unroll
    for (int j = 0; j < ND; ++j) {
      const int c = j * 8 + 2 * t;
      __nv_bfloat162 q0 = __floats2bfloat162_rn(0.f, 0.f), q1 = q0;
      if (r0 < nrows) q0 = *reinterpret_cast<const __nv_bfloat162*>(Qg + r0 * D + c);
      if (r1 < nrows) q1 = *reinterpret_cast<const __nv_bfloat162*>(Qg + r1 * D + c);
      acc[j][0] = __low2float(q0);
      acc[j][1] = __high2float(q0);
      acc[j][2] = __low2float(q1);
      acc[j][3] = __high2float(q1);
    }
    const int kslabs = (m0 + 16) / 8;
#pragma unroll
    for (int s = 0; s < NT; ++s) {
      if (s < kslabs) {
#pragma unroll
        for (int j = 0; j < ND; ++j) {
          uint32_t b[2];
          ldb_f32(b, sU, SD, j * 8, s * 8, g, t);
          mma_tf32(acc[j], aqw[s], b);
        }
      }
    }
    float* out = ql + static_cast<size_t>(ch) * kPC * D;
#pragma unroll
    for (int j = 0; j < ND; ++j) {
      const int c = j * 8 + 2 * t;
      *reinterpret_cast<float2*>(out + r0 * D + c) = make_float2(acc[j][0], acc[j][1]);
      *reinterpret_cast<float2*>(out + r1 * D + c) = make_float2(acc[j][2], acc[j][3]);
    }
  }
}

template <int D, bool kGate>
cudaError_t launch_one(const Geom& g, const Inputs& in, const Workspace& ws, cudaStream_t st) {
  using Cfg = PCfg<D>;
  auto kern = prep_mma_kernel<D, kGate>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cfg::kSmem));
  if (e != cudaSuccess) return e;
  kern<<<g.nch, kPThreads, Cfg::kSmem, st>>>(
      static_cast<const __nv_bfloat16*>(in.q), static_cast<const __nv_bfloat16*>(in.k),
      static_cast<const __nv_bfloat16*>(in.w), in.beta, ws.lam2,
      static_cast<__nv_bfloat16*>(ws.kr), ws.ql, static_cast<__nv_bfloat16*>(ws.ngt), ws.sdt,
      g.T, g.Np, in.scale * kLog2e);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep_mma(const Geom& g, const Inputs& in, const Workspace& ws,
                            cudaStream_t st) {
  if (g.C != kPC || !g.bf16) return cudaErrorInvalidValue;
  if (g.d == 128) return g.gate ? launch_one<128, true>(g, in, ws, st) : launch_one<128, false>(g, in, ws, st);
  if (g.d == 64) return g.gate ? launch_one<64, true>(g, in, ws, st) : launch_one<64, false>(g, in, ws, st);
  return cudaErrorInvalidValue;
}

}  // namespace pathattn
