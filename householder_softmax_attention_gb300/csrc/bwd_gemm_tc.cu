// bwd_gemm_tc.cu -- batched small GEMMs of the backward's chunk pass on the
// sm_103a tensor cores.
//
//   C[z] = mask(sum_t alpha_t op(A_t[z]) op(B_t[z]) + (Add ? Add[z] : 0)),
//   z = 0 .. batch-1, up to kMaxTerms products t, and optionally
//   C2[z] = mask2(C[z] with rows or columns scaled by a per-item vector)
//
// fp32 row-major operands (M = 128 rows, N and every K_t in {64, 128}), one
// CTA of four warps per batch item; an operand flagged bf16 is an exact bf16
// array (half the bytes read, its lo products skipped).  Each fp32 operand enters the MMA as
// x_hi + x_lo with x_hi = bf16(x), x_lo = bf16(x - x_hi) (about 16
// significant bits; alpha_t is applied to A_t before the split, exactly for
// alpha = +-1); the three products hi*hi + hi*lo + lo*hi of every term
// accumulate in fp32 in one TMEM accumulator, so a sum of products costs one
// launch and one write of C.  Each K slice of 64 is converted into
// 128-byte-swizzled shared-memory tiles (op(A) K-major unless A is transposed,
// op(B) MN-major unless B is transposed, so that every global read is along
// a stored row), one thread issues the slice's twelve MMAs, and the next
// slice is written once they have completed.  The accumulator goes from TMEM
// (one row per thread) through shared memory, so that the epilogue (addend,
// mask) reads and writes in coalesced rows.  Three CTAs fit on an SM, so
// conversion, MMAs and epilogues of different batch items overlap.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace pathattn {
namespace {

constexpr int kM = 128, kKs = 64, kThreads = 128;
constexpr uint32_t kSliceA = kM * kKs * 2;      // one bf16 copy of an A slice
constexpr uint32_t kSliceB = kKs * 128 * 2;     // one bf16 copy of a B slice (N <= 128)
constexpr uint32_t kOffAlo = kSliceA, kOffBhi = 2 * kSliceA, kOffBlo = 2 * kSliceA + kSliceB;
constexpr size_t kSmemBytes = 2 * kSliceA + 2 * kSliceB + 1024 + 64;

struct GemmBars {
  uint64_t mma;
  uint32_t tmem_base;
  int abort_flag;
};

// Byte offset of (row, col) in a tile of `rows` stored rows whose columns are
// split into 64-column halves of rows * 128 bytes, 128-byte swizzled.
__device__ __forceinline__ uint32_t swz_off(int rows, int row, int col) {
  return (col >> 6) * (rows * 128) + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
         ((col & 7) << 1);
}

// Converts a stored tile (rows x cols fp32, global, leading dimension ld),
// times `mul`, into bf16 hi / lo swizzled tiles; each thread has four
// 8-column groups of loads in flight before it converts them.
__device__ __forceinline__ void load_split(const float* __restrict__ src, int ld, int rows, int cols,
                                           float mul, uint8_t* hi, uint8_t* lo) {
  const int groups = rows * cols / 8;  // a multiple of 4 * kThreads
  const int gpr = cols / 8;
  for (int g0 = threadIdx.x; g0 < groups; g0 += 4 * kThreads) {
    float4 a[4], b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int gi = g0 + u * kThreads, r = gi / gpr, c8 = gi - r * gpr;
      const float4* p = reinterpret_cast<const float4*>(src + static_cast<size_t>(r) * ld + c8 * 8);
      a[u] = __ldg(p);
      b[u] = __ldg(p + 1);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int gi = g0 + u * kThreads, r = gi / gpr, c8 = gi - r * gpr;
      const float v[8] = {mul * a[u].x, mul * a[u].y, mul * a[u].z, mul * a[u].w,
                          mul * b[u].x, mul * b[u].y, mul * b[u].z, mul * b[u].w};
      uint32_t h[4], l[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) split_hilo2(v[2 * e], v[2 * e + 1], h[e], l[e]);
      const uint32_t off = swz_off(rows, r, c8 * 8);
      *reinterpret_cast<uint4*>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
    }
  }
}

// An exact bf16 operand (rows x cols bf16, leading dimension ld) copied into
// the hi tile, its sign flipped by `neg`; it needs no lo part.
__device__ __forceinline__ void load_exact(const __nv_bfloat16* __restrict__ src, int ld, int rows,
                                           int cols, bool neg, uint8_t* hi) {
  const int groups = rows * cols / 8;
  const int gpr = cols / 8;
  const uint32_t flip = neg ? 0x80008000u : 0u;
  for (int g0 = threadIdx.x; g0 < groups; g0 += 4 * kThreads) {
    uint4 a[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int gi = g0 + u * kThreads, r = gi / gpr, c8 = gi - r * gpr;
      a[u] = __ldg(reinterpret_cast<const uint4*>(src + static_cast<size_t>(r) * ld + c8 * 8));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int gi = g0 + u * kThreads, r = gi / gpr, c8 = gi - r * gpr;
      *reinterpret_cast<uint4*>(hi + swz_off(rows, r, c8 * 8)) =
          make_uint4(a[u].x ^ flip, a[u].y ^ flip, a[u].z ^ flip, a[u].w ^ flip);
    }
  }
}

// Columns n0 .. n0 + 3 of row r with the triangular mask applied: mask 1
// keeps n <= r, mask 2 keeps n < r.
__device__ __forceinline__ float4 mask4(float4 o, int mask, int r, int n0) {
  const int lim = mask == 1 ? r : r - 1;
  if (n0 > lim) o.x = 0.f;
  if (n0 + 1 > lim) o.y = 0.f;
  if (n0 + 2 > lim) o.z = 0.f;
  if (n0 + 3 > lim) o.w = 0.f;
  return o;
}

template <int N>
__global__ void __launch_bounds__(kThreads, 3) gemm_tc_kernel(const __grid_constant__ TcGemmN g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  GemmBars* bars = reinterpret_cast<GemmBars*>(base + 2 * kSliceA + 2 * kSliceB);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const size_t z = blockIdx.x;
  if (threadIdx.x == 0) {
    mbar_init(&bars->mma, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem_base, N);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tb = bars->tmem_base;
  bool ok = true;
  int sl = 0;  // slices issued so far (phase of the MMA barrier)
  for (int t = 0; t < g.nterms && ok; ++t) {
    const TcTerm& tt = g.t[t];
    const float* Az = tt.A + z * tt.sA;
    const float* Bz = tt.B + z * tt.sB;
    const uint32_t id = idesc_bf16_f32(kM, N, tt.tA, !tt.tB);
    for (int k0 = 0; k0 < tt.K && ok; k0 += kKs, ++sl) {
      // op(A) slice: A[m][k0..] (K-major) or A[k0..][m] (MN-major), times alpha
      const size_t aoff = tt.tA ? static_cast<size_t>(k0) * tt.lda : static_cast<size_t>(k0);
      const int arows = tt.tA ? kKs : kM, acols = tt.tA ? kM : kKs;
      if (tt.aBf)
        load_exact(reinterpret_cast<const __nv_bfloat16*>(tt.A) + z * tt.sA + aoff, tt.lda, arows,
                   acols, tt.alpha < 0.f, base);
      else
        load_split(Az + aoff, tt.lda, arows, acols, tt.alpha, base, base + kOffAlo);
      // op(B) slice: B[k0..][n] (MN-major) or B[n][k0..] (K-major)
      const size_t boff = tt.tB ? static_cast<size_t>(k0) : static_cast<size_t>(k0) * tt.ldb;
      const int brows = tt.tB ? N : kKs, bcols = tt.tB ? kKs : N;
      if (tt.bBf)
        load_exact(reinterpret_cast<const __nv_bfloat16*>(tt.B) + z * tt.sB + boff, tt.ldb, brows,
                   bcols, false, base + kOffBhi);
      else
        load_split(Bz + boff, tt.ldb, brows, bcols, 1.f, base + kOffBhi, base + kOffBlo);
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncthreads();
      if (threadIdx.x == 0) {
        tc_fence_after_sync();
        const uint32_t a0 = smem_addr(base), b0 = smem_addr(base + kOffBhi);
#pragma unroll
        for (int term = 0; term < 3; ++term) {
          if ((term == 1 && tt.bBf) || (term == 2 && tt.aBf)) continue;   // zero lo parts
          const uint32_t at = a0 + (term == 2 ? kOffAlo : 0);
          const uint32_t bt = b0 + (term == 1 ? kSliceB : 0);
#pragma unroll
          for (int k = 0; k < kKs / 16; ++k) {
            const uint64_t ad = tt.tA ? sdesc_sw128(at + k * 2048, kKs * 128, 1024)
                                      : sdesc_sw128(at + k * 32, 16, 1024);
            const uint64_t bd = tt.tB ? sdesc_sw128(bt + k * 32, 16, 1024)
                                      : sdesc_sw128(bt + k * 2048, kKs * 128, 1024);
            mma_bf16_ss(tb, ad, bd, id, (sl > 0 || term > 0 || k > 0));
          }
        }
        mma_commit(&bars->mma);
      }
      // the slice's tiles are free (and, after the last, the accumulator final)
      // once its MMAs have completed
      ok = mbar_wait(&bars->mma, sl & 1, &bars->abort_flag, kWaitLimitNs);
      tc_fence_after_sync();
    }
  }
  if (ok) {
    // accumulator rows (one per thread) -> shared memory (the slice tiles are
    // free), 16-byte units of a row rotated by the row index; then the tile
    // goes out in row-major order, so that reads of Add and writes are coalesced
    const int m = warp * 32 + lane;
    const uint32_t lb = static_cast<uint32_t>(warp * 32) << 16;
    float4* stile = reinterpret_cast<float4*>(base);
    constexpr int kU = N / 4;  // 16-byte units per row
#pragma unroll
    for (int cc = 0; cc < N; cc += 32) {
      uint32_t v[32];
      tmem_ld_x32(tb + lb + cc, v);
#pragma unroll
      for (int u4 = 0; u4 < 8; ++u4) {
        const int j = cc / 4 + u4;
        stile[m * kU + (j ^ (m & 7))] =
            make_float4(__uint_as_float(v[4 * u4]), __uint_as_float(v[4 * u4 + 1]),
                        __uint_as_float(v[4 * u4 + 2]), __uint_as_float(v[4 * u4 + 3]));
      }
    }
    __syncthreads();
    float* Cz = g.Cm + z * g.sC;
    const float* Dz = g.Add ? g.Add + z * g.sAdd : nullptr;
#pragma unroll 4
    for (int idx = threadIdx.x; idx < kM * kU; idx += kThreads) {
      const int r = idx / kU, j = idx - r * kU;
      float4 o = stile[r * kU + (j ^ (r & 7))];
      if (Dz) {
        const float4 c = *reinterpret_cast<const float4*>(Dz + static_cast<size_t>(r) * g.ldadd + 4 * j);
        o.x += c.x; o.y += c.y; o.z += c.z; o.w += c.w;
      }
      if (g.mask != 0) o = mask4(o, g.mask, r, 4 * j);
      *reinterpret_cast<float4*>(Cz + static_cast<size_t>(r) * g.ldc + 4 * j) = o;
      if (g.C2) {
        const float* vz = g.vec + z * kM;
        if (g.c2op == 1) {
          const float b = vz[r];
          o.x *= b; o.y *= b; o.z *= b; o.w *= b;
        } else {
          const float4 b = *reinterpret_cast<const float4*>(vz + 4 * j);
          o.x *= b.x; o.y *= b.y; o.z *= b.z; o.w *= b.w;
        }
        if (g.c2mask != 0) o = mask4(o, g.c2mask, r, 4 * j);
        *reinterpret_cast<float4*>(g.C2 + z * g.sC + static_cast<size_t>(r) * g.ldc + 4 * j) = o;
      }
    }
  } else if (threadIdx.x == 0) {
    atomicExch(g.status, PATH_DEV_ERR_TIMEOUT);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tb, N);
  }
}

template <int N>
cudaError_t launch_n(const TcGemmN& g, cudaStream_t st) {
  auto kern = gemm_tc_kernel<N>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  kern<<<g.batch, kThreads, kSmemBytes, st>>>(g);
  return cudaGetLastError();
}

}  // namespace

bool gemm_tc_supported(const TcGemmN& g) {
  if (g.M != kM || (g.N != 64 && g.N != 128) || g.nterms < 1 || g.nterms > kMaxTerms ||
      g.ldc % 4 != 0 || (g.Add && g.ldadd % 4 != 0))
    return false;
  if (g.C2 && (!g.vec || (g.c2op != 1 && g.c2op != 2) || (g.c2op == 2 && g.N != kM)))
    return false;
  for (int t = 0; t < g.nterms; ++t) {
    const TcTerm& tt = g.t[t];
    if ((tt.K != 64 && tt.K != 128) || tt.lda % 8 != 0 || tt.ldb % 8 != 0) return false;
  }
  return true;
}

cudaError_t launch_gemm_tc(const TcGemmN& g, cudaStream_t st) {
  if (!gemm_tc_supported(g) || g.batch < 1) return cudaErrorInvalidValue;
  return g.N == 128 ? launch_n<128>(g, st) : launch_n<64>(g, st);
}

}  // namespace pathattn
