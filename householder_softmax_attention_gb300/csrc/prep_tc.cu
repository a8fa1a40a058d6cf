// prep_tc.cu -- chunk preparation for bf16 inputs (d = 64 or 128) on tcgen05.
//
// One CTA (8 warps) per chunk of C = 128 tokens; the outputs and their algebra
// are those listed in prep.cu (from "PaTH Attention: Position Encoding via
// Accumulating Householder Transformations", frames "A triangular
// representation makes paths computable" and "Backup: fix orientation before
// implementing UT products").  Phases:
//
//   P1  [W W^T | W K^T] = W [W; K]^T and [Q W^T | Q K^T] = Q [W; K]^T:
//       two MMAs of width 256 per k-step (exact fp32 products of bf16 inputs)
//   P2  L = strictLower(D W W^T) -> fp32 shared memory;
//       S = strictLower(W K^T) -> bf16 hi / lo tiles
//   P3  X = (I + L)^{-1} (prep_solve.cuh), U = X D -> bf16 hi / lo
//   P4  TK = U S (three hi/lo products), UW = U W (two)
//   P5  TK, UW -> bf16 hi / lo tiles, laid out as [TK | UW]
//   P6a kr' = TK^T W, ngt' = UW^T W   (two terms each; at d = 64 the
//       accumulator rows of ngt' past d are never read)
//       kr = K - kr', ngt = -ngt'
//   P6b [sd' | ql'] = -lower(Q W^T) [TK | UW]   (A from TMEM, three terms)
//       sdt = log2(e) (scale (Q K^T + sd') + gate) transposed, ql = Q + ql'
//
// A computed fp32 operand x enters an MMA as x_hi + x_lo with x_hi = bf16(x)
// and x_lo = bf16(x - x_hi) (about 16 significant bits); products of two
// computed operands drop only the lo*lo term.  All accumulation is fp32 in
// TMEM.  Every wait is bounded (records a timeout in the status word).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "ptx.cuh"
#include "prep_solve.cuh"

namespace pathattn {
namespace {

constexpr int kC = 128, kThreads = 256;
constexpr uint32_t kHalf = 16384;   // one 64-column half of a 128-row bf16 tile
constexpr uint32_t kTile = 32768;   // a 128 x 128 bf16 tile
// shared-memory regions (offsets from a 1024-aligned base)
constexpr uint32_t kRWK = 0;        // W | K stacked per half: half h at h * 32K (W 16K, K 16K)
constexpr uint32_t kRQS = 65536;    // Q (P1), then S hi/lo (P2-P4), then [TK|UW] hi (P5-P6)
constexpr uint32_t kRL = 131072;    // fp32 L/X (P2-P3, stride 132), then U hi/lo, then [TK|UW] lo
constexpr int kSL = kC + 4;
constexpr uint32_t kRMisc = kRL + kC * kSL * 4;   // beta, gate prefix, barriers
constexpr size_t kSmemBytes = kRMisc + 2 * kC * 4 + 64 + 1024;

struct Bars {
  uint64_t tma, mma;
  uint32_t tmem_base;
  int abort_flag;
};

// Byte offset of element (row, col) in a 128-row bf16 tile stored as two
// 128-byte-swizzled 64-column halves kHalf apart (K-major A/B rows = row, or
// MN-major rows = K index).
__device__ __forceinline__ uint32_t tile_off(int row, int col) {
  return (col >> 6) * kHalf + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) + ((col & 7) << 1);
}

// Writes 8 consecutive values (cols c8*8 .. +7 of `row`) as bf16 hi and lo
// parts into two tiles.
__device__ __forceinline__ void put_hilo8(uint8_t* hi_tile, uint8_t* lo_tile, int row, int c8,
                                          const float (&v)[8]) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * u]), h1 = __float2bfloat16_rn(v[2 * u + 1]);
    h[u] = pack_bf16x2(__bfloat162float(h0), __bfloat162float(h1));
    l[u] = pack_bf16x2(v[2 * u] - __bfloat162float(h0), v[2 * u + 1] - __bfloat162float(h1));
  }
  const uint32_t off = tile_off(row, c8 * 8);
  *reinterpret_cast<uint4*>(hi_tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo_tile + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ bool wait_mma(Bars* bars, uint32_t parity, int* status) {
  if (mbar_wait(&bars->mma, parity, &bars->abort_flag, kWaitLimitNs)) return true;
  bars->abort_flag = 1;
  atomicExch(status, PATH_DEV_ERR_TIMEOUT);
  return false;
}

template <int D, bool kGate>
__global__ void __launch_bounds__(kThreads, 1)
    prep_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_q, const float* __restrict__ beta, const float* __restrict__ lam2,
                   __nv_bfloat16* __restrict__ kr, float* __restrict__ ql,
                   __nv_bfloat16* __restrict__ ngt, float* __restrict__ sdt, int* status, int T,
                   int Np, float sl2) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  float* sL = reinterpret_cast<float*>(base + kRL);
  float* sBeta = reinterpret_cast<float*>(base + kRMisc);
  float* sLam = sBeta + kC;
  Bars* bars = reinterpret_cast<Bars*>(sLam + kC);

  const int ch = blockIdx.x, bh = ch / Np, n = ch - bh * Np, t0 = n * kC;
  const int nrows = min(kC, T - t0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, halfc = warp >> 2;  // TMEM lane quarter, column half
  const int row = quarter * 32 + lane;              // this thread's TMEM lane
  const size_t row0 = static_cast<size_t>(bh) * T + t0;

  if (tid == 0) {
    mbar_init(&bars->tma, 1);
    mbar_init(&bars->mma, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < kC) {
    sBeta[tid] = tid < nrows ? beta[row0 + tid] : 0.f;
    if (kGate) sLam[tid] = lam2[static_cast<size_t>(bh) * Np * kC + t0 + tid];
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tb = bars->tmem_base;
  const uint32_t lb = static_cast<uint32_t>(quarter * 32) << 16;
  uint32_t mma_phase = 0;
  bool ok = true;

  // ---- P1: TMA loads, then the Gram blocks
  if (tid == 0) {
    mbar_arrive_expect_tx(&bars->tma, 3 * kC * D * 2);
    for (int h = 0; h < D / 64; ++h) {
      tma_load_3d(base + kRWK + h * 2 * kHalf, &map_w, h * 64, t0, bh, &bars->tma);
      tma_load_3d(base + kRWK + h * 2 * kHalf + kHalf, &map_k, h * 64, t0, bh, &bars->tma);
      tma_load_3d(base + kRQS + h * kHalf, &map_q, h * 64, t0, bh, &bars->tma);
    }
    ok = mbar_wait(&bars->tma, 0, &bars->abort_flag, kWaitLimitNs);
    if (ok) {
      tc_fence_after_sync();
      constexpr uint32_t id = idesc_bf16_f32(128, 256, false, false);
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t kb = k >> 2, kk = (k & 3) * 32;
        const uint64_t bwk = sdesc_sw128(smem_addr(base + kRWK + kb * 2 * kHalf) + kk, 16, 1024);
        const uint64_t aw = sdesc_sw128(smem_addr(base + kRWK + kb * 2 * kHalf) + kk, 16, 1024);
        const uint64_t aq = sdesc_sw128(smem_addr(base + kRQS + kb * kHalf) + kk, 16, 1024);
        mma_bf16_ss(tb + 0, aw, bwk, id, k > 0);    // [W W^T | W K^T]
        mma_bf16_ss(tb + 256, aq, bwk, id, k > 0);  // [Q W^T | Q K^T]
      }
    } else {
      bars->abort_flag = 1;
      atomicExch(status, PATH_DEV_ERR_TIMEOUT);
    }
    mma_commit(&bars->mma);
  }
  ok = wait_mma(bars, mma_phase, status);
  mma_phase ^= 1;
  tc_fence_after_sync();

  // ---- P2: L (fp32, smem) and S = strictLower(W K^T) (bf16 hi/lo, MN-major B)
  {
    uint8_t* s_hi = base + kRQS;
    uint8_t* s_lo = base + kRQS + kTile;
    const float bt = sBeta[row];
#pragma unroll
    for (int cc = 0; cc < 64; cc += 32) {
      const int c0 = halfc * 64 + cc;
      uint32_t v[32];
      tmem_ld_x32(tb + lb + c0, v);
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const int c = c0 + u;
        sL[row * kSL + c] = c < row ? __uint_as_float(v[u]) * bt : 0.f;
      }
      tmem_ld_x32(tb + lb + 128 + c0, v);
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) {
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = c0 + g8 * 8 + u;
          x[u] = c < row ? __uint_as_float(v[g8 * 8 + u]) : 0.f;
        }
        put_hilo8(s_hi, s_lo, row, (c0 >> 3) + g8, x);
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();

  // ---- P3: X = (I + L)^{-1}, then U = X diag(beta) as bf16 hi/lo (K-major A)
  invert_unit_lower<kSL>(sL, tid);
  {
    // 2048 groups of 8 consecutive columns of one row; 8 groups per thread,
    // all read before the fp32 buffer is overwritten by the tiles
    float v[8][8];
#pragma unroll
    for (int gi = 0; gi < 8; ++gi) {
      const int grp = tid + gi * kThreads, i = grp >> 4, c8 = grp & 15;
      const float4 x0 = *reinterpret_cast<const float4*>(sL + i * kSL + c8 * 8);
      const float4 x1 = *reinterpret_cast<const float4*>(sL + i * kSL + c8 * 8 + 4);
      const float4 b0 = *reinterpret_cast<const float4*>(sBeta + c8 * 8);
      const float4 b1 = *reinterpret_cast<const float4*>(sBeta + c8 * 8 + 4);
      const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const float bs[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int u = 0; u < 8; ++u) v[gi][u] = c8 * 8 + u <= i ? xs[u] * bs[u] : 0.f;
    }
    __syncthreads();
    uint8_t* u_hi = base + kRL;
    uint8_t* u_lo = base + kRL + kTile;
#pragma unroll
    for (int gi = 0; gi < 8; ++gi) {
      const int grp = tid + gi * kThreads, i = grp >> 4, c8 = grp & 15;
      put_hilo8(u_hi, u_lo, i, c8, v[gi]);
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before_sync();
  __syncthreads();

  // ---- P4: TK = U S (hi*hi + hi*lo + lo*hi) -> cols [0,128); UW = U W -> [128,256)
  if (tid == 0 && ok) {
    tc_fence_after_sync();
    constexpr uint32_t id = idesc_bf16_f32(128, 128, false, true);
    constexpr uint32_t id_uw = idesc_bf16_f32(128, D, false, true);
    const uint32_t u_hi = smem_addr(base + kRL), u_lo = u_hi + kTile;
    const uint32_t s_hi = smem_addr(base + kRQS), s_lo = s_hi + kTile;
    const uint32_t w_b = smem_addr(base + kRWK);
    auto a_desc = [&](uint32_t t, int k) {
      return sdesc_sw128(t + (k >> 2) * kHalf + (k & 3) * 32, 16, 1024);
    };
    for (int term = 0; term < 3; ++term) {
      const uint32_t at = term == 2 ? u_lo : u_hi, bt = term == 1 ? s_lo : s_hi;
      for (int k = 0; k < kC / 16; ++k)
        mma_bf16_ss(tb + 0, a_desc(at, k), sdesc_sw128(bt + k * 2048, kHalf, 1024), id,
                    term > 0 || k > 0);
    }
    for (int term = 0; term < 2; ++term) {
      const uint32_t at = term == 0 ? u_hi : u_lo;
      for (int k = 0; k < kC / 16; ++k)
        mma_bf16_ss(tb + 128, a_desc(at, k), sdesc_sw128(w_b + k * 2048, 2 * kHalf, 1024), id_uw,
                    term > 0 || k > 0);
    }
    mma_commit(&bars->mma);
  } else if (tid == 0) {
    mma_commit(&bars->mma);
  }
  ok = wait_mma(bars, mma_phase, status) && ok;
  mma_phase ^= 1;
  tc_fence_after_sync();

  // ---- P5: [TK | UW] -> bf16 hi (region QS) and lo (region L) tiles, MN-major
  {
    uint8_t* hi = base + kRQS;   // TK at +0 (two halves), UW at +kTile
    uint8_t* lo = base + kRL;
#pragma unroll
    for (int cc = 0; cc < (halfc == 0 ? 128 : D); cc += 32) {
      const int c0 = halfc * 128 + cc;   // halfc 0: TK, 1: UW
      uint32_t v[32];
      tmem_ld_x32(tb + lb + c0, v);
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) {
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = __uint_as_float(v[g8 * 8 + u]);
        put_hilo8(hi + halfc * kTile, lo + halfc * kTile, row, (cc >> 3) + g8, x);
      }
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before_sync();
  __syncthreads();

  // ---- P6a: kr' = TK^T W and ngt' = UW^T W (A = the MN-major [TK | UW] tiles,
  // B = W): one output row per TMEM lane, so that the epilogue writes rows
  if (tid == 0 && ok) {
    tc_fence_after_sync();
    constexpr uint32_t id = idesc_bf16_f32(128, D, true, true);
    const uint32_t w_b = smem_addr(base + kRWK);
    const uint32_t b_hi = smem_addr(base + kRQS), b_lo = smem_addr(base + kRL);
    for (int part = 0; part < 2; ++part)        // TK^T W -> cols [0, D), UW^T W -> [128, 128 + D)
      for (int term = 0; term < 2; ++term) {    // hi, lo
        const uint32_t at = (term == 0 ? b_hi : b_lo) + part * kTile;
        for (int k = 0; k < kC / 16; ++k)
          mma_bf16_ss(tb + part * 128, sdesc_sw128(at + k * 2048, kHalf, 1024),
                      sdesc_sw128(w_b + k * 2048, 2 * kHalf, 1024), id, term > 0 || k > 0);
      }
    mma_commit(&bars->mma);
  } else if (tid == 0) {
    mma_commit(&bars->mma);
  }
  // meanwhile: -lower(Q W^T) -> bf16 hi / lo A operand in TMEM columns [256, 384)
  if (warp < 4) {
    uint32_t v[128];
    tmem_ld_x128(tb + lb + 256, v);
    uint32_t ph[64], pl[64];
#pragma unroll
    for (int u = 0; u < 64; ++u) {
      const int c = 2 * u;
      const float x0 = c <= row ? -__uint_as_float(v[c]) : 0.f;
      const float x1 = c + 1 <= row ? -__uint_as_float(v[c + 1]) : 0.f;
      const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
      ph[u] = pack_bf16x2(__bfloat162float(h0), __bfloat162float(h1));
      pl[u] = pack_bf16x2(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
    }
    tmem_st_x32(tb + lb + 256, *reinterpret_cast<uint32_t(*)[32]>(&ph[0]));
    tmem_st_x32(tb + lb + 288, *reinterpret_cast<uint32_t(*)[32]>(&ph[32]));
    tmem_st_x32(tb + lb + 320, *reinterpret_cast<uint32_t(*)[32]>(&pl[0]));
    tmem_st_x32(tb + lb + 352, *reinterpret_cast<uint32_t(*)[32]>(&pl[32]));
    tmem_st_wait();
  }
  ok = wait_mma(bars, mma_phase, status) && ok;
  mma_phase ^= 1;
  tc_fence_after_sync();
  // epilogue: kr[j][:] = K[j][:] - kr'[j][:] (half 0, row j = lane), ngt[n][:] =
  // -ngt'[n][:] (half 1, rows n < D): whole rows, 16 bytes per store
  if (halfc == 0) {
    const int j = row;
    uint4* out = reinterpret_cast<uint4*>(kr + (static_cast<size_t>(ch) * kC + j) * D);
    const uint8_t* kt = base + kRWK + kHalf;  // K rows inside the W|K halves
    for (int cc = 0; cc < D; cc += 32) {
      uint32_t v[32];
      tmem_ld_x32(tb + lb + cc, v);
#pragma unroll
      for (int u8 = 0; u8 < 32; u8 += 8) {
        const int f0 = cc + u8;  // features f0 .. f0 + 7: one 16-byte chunk of K's row j
        const uint32_t off =
            (f0 >> 6) * 2 * kHalf + j * 128 + ((((f0 & 63) >> 3) ^ (j & 7)) << 4);
        const uint4 kq = *reinterpret_cast<const uint4*>(kt + off);
        const uint32_t kw[4] = {kq.x, kq.y, kq.z, kq.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          o[e] = pack_bf16x2(__uint_as_float(kw[e] << 16) - __uint_as_float(v[u8 + 2 * e]),
                             __uint_as_float(kw[e] & 0xffff0000u) -
                                 __uint_as_float(v[u8 + 2 * e + 1]));
        out[f0 / 8] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  } else if (row < D) {
    const int n = row;
    uint4* out = reinterpret_cast<uint4*>(ngt + (static_cast<size_t>(ch) * D + n) * D);
    for (int cc = 0; cc < D; cc += 32) {
      uint32_t v[32];
      tmem_ld_x32(tb + lb + 128 + cc, v);
#pragma unroll
      for (int u8 = 0; u8 < 32; u8 += 8)
        out[(cc + u8) / 8] =
            make_uint4(pack_bf16x2(-__uint_as_float(v[u8]), -__uint_as_float(v[u8 + 1])),
                       pack_bf16x2(-__uint_as_float(v[u8 + 2]), -__uint_as_float(v[u8 + 3])),
                       pack_bf16x2(-__uint_as_float(v[u8 + 4]), -__uint_as_float(v[u8 + 5])),
                       pack_bf16x2(-__uint_as_float(v[u8 + 6]), -__uint_as_float(v[u8 + 7])));
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before_sync();
  __syncthreads();

  // Q again, into the W | K region (free from here on), for the final pass
  if (tid == 0) {
    mbar_arrive_expect_tx(&bars->tma, kC * D * 2);
    for (int h = 0; h < D / 64; ++h)
      tma_load_3d(base + kRWK + h * kHalf, &map_q, h * 64, t0, bh, &bars->tma);
  }

  // ---- P6b: [sd' | ql'] = -lower(Q W^T) [TK | UW], A from TMEM (hi, lo)
  if (tid == 0 && ok) {
    tc_fence_after_sync();
    constexpr uint32_t id = idesc_bf16_f32(128, kC + D, false, true);
    const uint32_t b_hi = smem_addr(base + kRQS), b_lo = smem_addr(base + kRL);
    for (int term = 0; term < 3; ++term) {
      const uint32_t acol = term == 2 ? 320 : 256;   // A: hi or lo
      const uint32_t bt = term == 1 ? b_lo : b_hi;
      for (int k = 0; k < kC / 16; ++k)
        mma_bf16_ts(tb + 0, tb + acol + k * 8, sdesc_sw128(bt + k * 2048, kHalf, 1024), id,
                    term > 0 || k > 0);
    }
    mma_commit(&bars->mma);
  } else if (tid == 0) {
    mma_commit(&bars->mma);
  }
  ok = wait_mma(bars, mma_phase, status) && ok;
  mma_phase ^= 1;
  tc_fence_after_sync();
  // epilogue: sdt[j][i] from Q K^T + sd' (half 0); ql[i][n] = Q[i][n] + ql' (half 1)
  {
    const int i = row;
    if (halfc == 0) {
      float* out = sdt + static_cast<size_t>(ch) * kC * kC + i;
      const float li = kGate ? sLam[i] : 0.f;
      for (int cc = 0; cc < 128; cc += 32) {
        uint32_t v[32], qk[32];
        tmem_ld_x32(tb + lb + cc, v);
        tmem_ld_x32(tb + lb + 384 + cc, qk);
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int j = cc + u;
          const float gj = kGate ? sLam[j] : 0.f;
          out[static_cast<size_t>(j) * kC] =
              j <= i ? fmaf(__uint_as_float(qk[u]) + __uint_as_float(v[u]), sl2, li - gj) : -INFINITY;
        }
      }
    } else {
      // ql' rows to shared memory (the lo tiles are dead once the MMA is done)
      float* sq = sL;
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t v[32];
        tmem_ld_x32(tb + lb + 128 + cc, v);
#pragma unroll
        for (int u = 0; u < 32; u += 4)
          *reinterpret_cast<float4*>(sq + i * kSL + cc + u) =
              make_float4(__uint_as_float(v[u]), __uint_as_float(v[u + 1]),
                          __uint_as_float(v[u + 2]), __uint_as_float(v[u + 3]));
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  // ql = Q + ql', one row per warp instruction: coalesced stores; Q from the
  // copy that landed during P6b (rows past T read as zero)
  if (!mbar_wait(&bars->tma, 1, &bars->abort_flag, kWaitLimitNs)) {
    bars->abort_flag = 1;
    atomicExch(status, PATH_DEV_ERR_TIMEOUT);
  }
  {
    const float* sq = sL;
    float* out = ql + static_cast<size_t>(ch) * kC * D;
    constexpr int kIter = kC * D / 4 / kThreads;  // 16 at d = 128
    uint2 qv[kIter];
#pragma unroll
    for (int r = 0; r < kIter; ++r) {
      const int e = tid + r * kThreads, i = e / (D / 4), n4 = (e % (D / 4)) * 4;
      qv[r] = *reinterpret_cast<const uint2*>(base + kRWK + tile_off(i, n4));
    }
#pragma unroll
    for (int r = 0; r < kIter; ++r) {
      const int e = tid + r * kThreads, i = e / (D / 4), n4 = (e % (D / 4)) * 4;
      float4 o = *reinterpret_cast<const float4*>(sq + i * kSL + n4);
      const __nv_bfloat162 q01 = *reinterpret_cast<const __nv_bfloat162*>(&qv[r].x);
      const __nv_bfloat162 q23 = *reinterpret_cast<const __nv_bfloat162*>(&qv[r].y);
      o.x += __low2float(q01);
      o.y += __high2float(q01);
      o.z += __low2float(q23);
      o.w += __high2float(q23);
      *reinterpret_cast<float4*>(out + i * D + n4) = o;
    }
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tb, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [BH][T][d] bf16 input seen as a 3D map with 128-byte-swizzled boxes of 64
// features x 128 tokens (tokens past T read as zero).
bool make_input_map(CUtensorMap* m, const void* ptr, int D, int T, int BH) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(T) * D * 2};
  cuuint32_t box[3] = {64, kC, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool kGate>
cudaError_t launch_one(const Geom& g, const Inputs& in, const Workspace& ws, int* status,
                       cudaStream_t st) {
  CUtensorMap mw, mk, mq;
  if (!make_input_map(&mw, in.w, D, g.T, g.BH) || !make_input_map(&mk, in.k, D, g.T, g.BH) ||
      !make_input_map(&mq, in.q, D, g.T, g.BH))
    return cudaErrorInvalidValue;
  auto kern = prep_tc_kernel<D, kGate>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  kern<<<g.nch, kThreads, kSmemBytes, st>>>(
      mw, mk, mq, in.beta, ws.lam2,
      static_cast<__nv_bfloat16*>(ws.kr), ws.ql, static_cast<__nv_bfloat16*>(ws.ngt), ws.sdt,
      status, g.T, g.Np, in.scale * kLog2e);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep_tc(const Geom& g, const Inputs& in, const Workspace& ws, int* status,
                           cudaStream_t st) {
  if (g.C != kC || !g.bf16) return cudaErrorInvalidValue;
  if (g.d == 128)
    return g.gate ? launch_one<128, true>(g, in, ws, status, st)
                  : launch_one<128, false>(g, in, ws, status, st);
  if (g.d == 64)
    return g.gate ? launch_one<64, true>(g, in, ws, status, st)
                  : launch_one<64, false>(g, in, ws, status, st);
  return cudaErrorInvalidValue;
}

}  // namespace pathattn
