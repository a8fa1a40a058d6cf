// prep_solve.cuh -- the unit-lower-triangular inverse X = (I + L)^{-1} of a
// 128 x 128 fp32 matrix in shared memory, used by the tensor-core chunk
// preparation (U = (I + strictLower(D W W^T))^{-1} D in "PaTH Attention: Position
// Encoding via Accumulating Householder Transformations", frame "A triangular
// representation makes paths computable").  Recursive doubling: 16 x 16
// diagonal blocks by substitution, then blocks of 16 on the CUDA cores and of
// 32 and 64 on the tensor cores (mma.sync tf32 with hi/lo splits, about fp32
// accuracy).  Block of 256 threads.
#pragma once
#include <cstdint>

namespace pathattn {
namespace solve {

constexpr int kPC = 128;        // matrix order
constexpr int kPThreads = 256;  // threads of the calling block

__device__ __forceinline__ uint32_t tf32r(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// One doubling level of the unit-lower-triangular inverse: for every pair of
// s x s diagonal blocks [[A, 0], [Cb, Dm]] whose inverses Ainv, Dinv are in
// place, overwrite Cb with -Dinv (Cb Ainv).  Thread t owns column t % s of one
// pair and rows i0, i0 + 4, ... of it, so the operand shared by its outputs is
// loaded once per k and the row operands come in as float4 broadcasts.
template <int S, int s>
__device__ __forceinline__ void invert_level(float* sU, int tid) {
  constexpr int kPer = s / 4;                  // outputs per thread
  constexpr int kPairs = kPC / (2 * s);
  const int jj = tid % s, rest = tid / s;
  const int p = rest % kPairs, i0 = rest / kPairs;
  const int r0 = p * 2 * s + s, c0 = p * 2 * s;
  float e[kPer];
#pragma unroll
  for (int r = 0; r < kPer; ++r) e[r] = 0.f;
  // E = Cb Ainv   (Ainv's upper part is zero, so every k can be summed)
#pragma unroll 4
  for (int kk = 0; kk < s; kk += 4) {
    const float a0 = sU[(c0 + kk) * S + c0 + jj], a1 = sU[(c0 + kk + 1) * S + c0 + jj];
    const float a2 = sU[(c0 + kk + 2) * S + c0 + jj], a3 = sU[(c0 + kk + 3) * S + c0 + jj];
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const float4 cv = *reinterpret_cast<const float4*>(sU + (r0 + i0 + 4 * r) * S + c0 + kk);
      e[r] = fmaf(cv.x, a0, fmaf(cv.y, a1, fmaf(cv.z, a2, fmaf(cv.w, a3, e[r]))));
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kPer; ++r) sU[(r0 + i0 + 4 * r) * S + c0 + jj] = e[r];
  __syncthreads();
  // F = -Dinv E   (Dinv's upper part is zero)
#pragma unroll
  for (int r = 0; r < kPer; ++r) e[r] = 0.f;
#pragma unroll 4
  for (int kk = 0; kk < s; kk += 4) {
    const float b0 = sU[(r0 + kk) * S + c0 + jj], b1 = sU[(r0 + kk + 1) * S + c0 + jj];
    const float b2 = sU[(r0 + kk + 2) * S + c0 + jj], b3 = sU[(r0 + kk + 3) * S + c0 + jj];
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const float4 dv = *reinterpret_cast<const float4*>(sU + (r0 + i0 + 4 * r) * S + r0 + kk);
      e[r] = fmaf(dv.x, b0, fmaf(dv.y, b1, fmaf(dv.z, b2, fmaf(dv.w, b3, e[r]))));
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kPer; ++r) sU[(r0 + i0 + 4 * r) * S + c0 + jj] = -e[r];
  __syncthreads();
}

// acc[nt] += A[m0:m0+16, k0:k1] * B[k0:k1, n0:n0+8 nt] on fp32 shared-memory
// matrices (row-major, strides SA / SB) with three tf32 products per term
// (hi*hi + hi*lo + lo*hi), which keeps about fp32 accuracy.
template <int NT, int SA, int SB>
__device__ __forceinline__ void mma_3xtf32(float (&acc)[NT][4], const float* A, int m0,
                                           const float* B, int n0, int k0, int k1, int g,
                                           int t, float sign) {
  for (int k = k0; k < k1; k += 8) {
    uint32_t ah[4], al[4];
    const float av[4] = {A[(m0 + g) * SA + k + t], A[(m0 + g + 8) * SA + k + t],
                         A[(m0 + g) * SA + k + t + 4], A[(m0 + g + 8) * SA + k + t + 4]};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float x = sign * av[u];
      ah[u] = tf32r(x);
      al[u] = tf32r(x - __uint_as_float(ah[u]));
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const float b0 = B[(k + t) * SB + n0 + 8 * j + g], b1 = B[(k + t + 4) * SB + n0 + 8 * j + g];
      uint32_t bh[2] = {tf32r(b0), tf32r(b1)};
      uint32_t bl[2] = {tf32r(b0 - __uint_as_float(bh[0])), tf32r(b1 - __uint_as_float(bh[1]))};
      mma_tf32(acc[j], al, bh);
      mma_tf32(acc[j], ah, bl);
      mma_tf32(acc[j], ah, bh);
    }
  }
}

// Doubling level on the tensor cores for s = 32 or 64: the same update as
// invert_level, E = Cb Ainv then Cb <- -Dinv E, with 16 x 8 output tiles
// spread over the 8 warps.
template <int S, int s>
__device__ __forceinline__ void invert_level_mma(float* sU, int warp, int g, int t) {
  constexpr int kPairs = kPC / (2 * s);
  constexpr int kMTiles = s / 16, kNTiles = s / 8;
  constexpr int kTilesPerPair = kMTiles * kNTiles;           // 16-row x 8-col tiles
  constexpr int kNT = kPairs * kTilesPerPair / 8;             // n-tiles per warp
  static_assert(kNT >= 1 && kNTiles % kNT == 0, "tile split");
  // warp -> (pair, m-tile, first n-tile)
  const int tile0 = warp * kNT;
  const int p = tile0 / kTilesPerPair, rem = tile0 % kTilesPerPair;
  const int mt = rem / kNTiles, nt0 = rem % kNTiles;
  const int r0 = p * 2 * s + s, c0 = p * 2 * s;
  float acc[kNT][4];
#pragma unroll
  for (int j = 0; j < kNT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  // E = Cb Ainv: A = rows r0 + 16 mt of Cb (columns c0..), B = Ainv (rows c0.., cols c0..);
  // Ainv is lower triangular, so rows k < 8 nt0 of it are zero in these columns
  mma_3xtf32<kNT, S, S>(acc, sU + c0, r0 + 16 * mt, sU + c0 * S + c0, 8 * nt0, 8 * nt0, s, g, t,
                        1.f);
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kNT; ++j) {
    const int c = c0 + 8 * (nt0 + j) + 2 * t, ra = r0 + 16 * mt + g;
    sU[ra * S + c] = acc[j][0];
    sU[ra * S + c + 1] = acc[j][1];
    sU[(ra + 8) * S + c] = acc[j][2];
    sU[(ra + 8) * S + c + 1] = acc[j][3];
    acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  }
  __syncthreads();
  // -Dinv E: A = Dinv (rows r0.., cols r0..), B = E (rows r0.., cols c0..); Dinv is
  // lower triangular, so columns k > 16 mt + 15 of these rows are zero
  mma_3xtf32<kNT, S, S>(acc, sU + r0, r0 + 16 * mt, sU + r0 * S + c0, 8 * nt0, 0, 16 * mt + 16, g,
                        t, -1.f);
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kNT; ++j) {
    const int c = c0 + 8 * (nt0 + j) + 2 * t, ra = r0 + 16 * mt + g;
    sU[ra * S + c] = acc[j][0];
    sU[ra * S + c + 1] = acc[j][1];
    sU[(ra + 8) * S + c] = acc[j][2];
    sU[(ra + 8) * S + c + 1] = acc[j][3];
  }
  __syncthreads();
}

// The 32 x 32 diagonal blocks of X = (I + L)^{-1} in place (L strictly lower
// on entry, stride S; only those blocks are read or written): the 16 x 16
// diagonal blocks by substitution, then one doubling level of 16 on the CUDA
// cores.  Ends with a block-wide barrier.
template <int S>
__device__ __forceinline__ void invert_diag32(float* sU, int tid) {
  {
    const int bb = tid >> 4, j = tid & 15, base = bb * 16;
    float x[16];
    if (tid < 128) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < i; ++k) s = fmaf(sU[(base + i) * S + base + k], x[k], s);
        x[i] = (i == j) ? 1.f : (i < j ? 0.f : -s);
      }
    }
    __syncthreads();
    if (tid < 128) {
#pragma unroll
      for (int i = 0; i < 16; ++i) sU[(base + i) * S + base + j] = x[i];
    }
    __syncthreads();
  }
  invert_level<S, 16>(sU, tid);
}

// X = (I + L)^{-1} in place (L strictly lower on entry, stride S), by
// recursive doubling: the 32 x 32 diagonal blocks as above, then levels of 32
// and 64 on the tensor cores.  Ends with a block-wide barrier.
template <int S>
__device__ __forceinline__ void invert_unit_lower(float* sU, int tid) {
  invert_diag32<S>(sU, tid);
  const int warp = tid >> 5, g = (tid & 31) >> 2, t = tid & 3;
  invert_level_mma<S, 32>(sU, warp, g, t);
  invert_level_mma<S, 64>(sU, warp, g, t);
}

}  // namespace solve
using solve::invert_diag32;
using solve::invert_unit_lower;
}  // namespace pathattn
