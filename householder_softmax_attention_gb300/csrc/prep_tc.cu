// prep_tc.cu -- chunk preparation for bf16 inputs (d = 64 or 128) on tcgen05.
//
// One persistent CTA (8 warps) per SM walks chunks of C = 128 tokens; the
// outputs and their algebra are those listed in prep.cu (from "PaTH Attention: Position Encoding via
// Accumulating Householder Transformations", frames "A triangular
// representation makes paths computable" and "Backup: fix orientation before
// implementing UT products").  Phases:
//
//   P1  [W W^T | W K^T] = W [W; K]^T, then [Q W^T | Q K^T] = Q [W; K]^T:
//       MMAs of width 256 (exact fp32 products of bf16 inputs), committed
//       separately so that the second runs during P2 and P3
//   P2  the 32 x 32 diagonal blocks of L = strictLower(D W W^T) -> fp32
//   P3  U = X D, X = (I + L)^{-1}, as bf16 hi / lo tiles: the diagonal
//       blocks of X on the CUDA cores (prep_solve.cuh), the doubling levels
//       of 32 and 64 on tcgen05 through U_ba = -U_bb (W W^T)_ba U_aa;
//       S = strictLower(W K^T) -> bf16 hi / lo tiles over Q
//   P4  TK = U S (three hi/lo products), UW = U W (two)
//   P5  TK, UW -> bf16 hi / lo tiles, laid out as [TK | UW]
//   P6a kr' = TK^T W, ngt' = UW^T W   (two terms each; at d = 64 the
//       accumulator rows of ngt' past d are never read)
//       kr = K - kr', ngt = -ngt' (rows stored while P6b runs)
//   P6b [sd' | ql'] = -lower(Q W^T) [TK | UW]   (A from TMEM, three terms)
//       sdt = log2(e) (scale (Q K^T + sd') + gate) transposed, ql = Q + ql'
//
// Between chunks: the next chunk's W and K arrive by TMA while P6b runs, its
// Q once P6b has read the region Q goes to; the diagonal logits sdt of a
// chunk are held in registers and stored once the next chunk's Gram products
// have been issued, so that those stores drain while the tensor cores work.
//
// A computed fp32 operand x enters an MMA as x_hi + x_lo with x_hi = bf16(x)
// and x_lo = bf16(x - x_hi) (about 16 significant bits); products of two
// computed operands drop only the lo*lo term.  All accumulation is fp32 in
// TMEM.  Every wait is bounded (records a timeout in the status word).
#include <algorithm>

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
constexpr uint32_t kRE = kRL + kC * kSL * 4;      // inverse levels: E tiles, hi/lo (16 KB)
constexpr uint32_t kRMisc = kRE + 16384;          // beta, gate prefix, barriers
constexpr size_t kSmemBytes = kRMisc + 2 * kC * 4 + 64 + 1024;
static_assert(kRE % 1024 == 0, "swizzled tiles need 1024-byte alignment");

struct Bars {
  uint64_t tma, mma, mma_q;   // mma_q: the query Gram block of P1
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
  for (int u = 0; u < 4; ++u) split_hilo2(v[2 * u], v[2 * u + 1], h[u], l[u]);
  const uint32_t off = tile_off(row, c8 * 8);
  *reinterpret_cast<uint4*>(hi_tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo_tile + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ bool wait_mma(Bars* bars, uint32_t parity, int* status,
                                         uint64_t* bar = nullptr) {
  if (mbar_wait(bar ? bar : &bars->mma, parity, &bars->abort_flag, kWaitLimitNs)) return true;
  bars->abort_flag = 1;
  atomicExch(status, PATH_DEV_ERR_TIMEOUT);
  return false;
}

// The chunk's beta and gate prefix into shared memory (threads 0 .. kC-1).
template <bool kGate>
__device__ __forceinline__ void load_chunk_scalars(float* sBeta, float* sLam, const float* beta,
                                                   const float* lam2, int ch, int Np, int T,
                                                   int tid) {
  if (tid < kC) {
    const int bh = ch / Np, t0 = (ch - bh * Np) * kC;
    sBeta[tid] = t0 + tid < T ? beta[static_cast<size_t>(bh) * T + t0 + tid] : 0.f;
    if (kGate) sLam[tid] = lam2[static_cast<size_t>(bh) * Np * kC + t0 + tid];
  }
}

// TMA loads of a chunk's W and K rows (two 64-column halves each, stacked per
// half as W | K) and of its Q rows into their own region.
template <int D>
__device__ __forceinline__ void load_wk(uint8_t* base, const CUtensorMap* mw, const CUtensorMap* mk,
                                        int ch, int Np, uint64_t* bar) {
  const int bh = ch / Np, t0 = (ch - bh * Np) * kC;
  for (int h = 0; h < D / 64; ++h) {
    tma_load_3d(base + kRWK + h * 2 * kHalf, mw, h * 64, t0, bh, bar);
    tma_load_3d(base + kRWK + h * 2 * kHalf + kHalf, mk, h * 64, t0, bh, bar);
  }
}
template <int D>
__device__ __forceinline__ void load_q(uint8_t* base, const CUtensorMap* mq, int ch, int Np,
                                       uint64_t* bar) {
  const int bh = ch / Np, t0 = (ch - bh * Np) * kC;
  for (int h = 0; h < D / 64; ++h) tma_load_3d(base + kRQS + h * kHalf, mq, h * 64, t0, bh, bar);
}

// The last epilogue of a chunk, in three parts.  The chunk's Q rows, loaded
// from global memory before the last product is waited for (rows past T as
// zero; element group e = tid + r * kThreads holds row e / (D/4), features
// 4 (e % (D/4)) ..), so that their latency hides behind it:
template <int D>
__device__ __forceinline__ void load_q_rows(uint2 (&qv)[kC * D / 4 / kThreads],
                                            const __nv_bfloat16* __restrict__ q, int ch, int Np,
                                            int T, int tid) {
  const int bh = ch / Np, t0 = (ch - bh * Np) * kC;
  const __nv_bfloat16* qc = q + (static_cast<size_t>(bh) * T + t0) * D;
#pragma unroll
  for (int r = 0; r < kC * D / 4 / kThreads; ++r) {
    const int e = tid + r * kThreads, i = e / (D / 4), n4 = (e % (D / 4)) * 4;
    qv[r] = t0 + i < T ? __ldg(reinterpret_cast<const uint2*>(qc + static_cast<size_t>(i) * D + n4))
                       : make_uint2(0u, 0u);
  }
}
// ql = Q + ql' (ql' staged in shared memory), as coalesced rows:
template <int D>
__device__ __forceinline__ void store_ql(const uint2 (&qv)[kC * D / 4 / kThreads], const float* sq,
                                         float* __restrict__ ql, int ch, int tid) {
  float* out = ql + static_cast<size_t>(ch) * kC * D;
#pragma unroll
  for (int r = 0; r < kC * D / 4 / kThreads; ++r) {
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
// and the diagonal logits sdt[j][i] (64 keys j of row i per thread, -inf
// above the diagonal), coalesced over the rows i:
__device__ __forceinline__ void store_sdt(const float (&tv)[64], float* __restrict__ sdt, int ch,
                                          int row, int halfc) {
  float* out = sdt + static_cast<size_t>(ch) * kC * kC + row;
#pragma unroll
  for (int u = 0; u < 64; ++u) out[static_cast<size_t>(64 * halfc + u) * kC] = tv[u];
}

// CTA b prepares chunks b, b + gridDim.x, ... (gridDim.x at most the SM count).
template <int D, bool kGate>
__global__ void __launch_bounds__(kThreads, 1)
    prep_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_q, const uint8_t* w_raw, const uint8_t* k_raw,
                   const uint8_t* q_raw, const float* __restrict__ beta, const float* __restrict__ lam2,
                   __nv_bfloat16* __restrict__ kr, float* __restrict__ ql,
                   __nv_bfloat16* __restrict__ ngt, float* __restrict__ sdt,
                   __nv_bfloat16* __restrict__ uwn, int* status, int T, int Np, int nch,
                   float sl2, int wr) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  float* sL = reinterpret_cast<float*>(base + kRL);
  float* sBeta = reinterpret_cast<float*>(base + kRMisc);
  float* sLam = sBeta + kC;
  Bars* bars = reinterpret_cast<Bars*>(sLam + kC);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, halfc = warp >> 2;  // TMEM lane quarter, column half
  const int row = quarter * 32 + lane;              // this thread's TMEM lane
  const int grid = static_cast<int>(gridDim.x);
  const __nv_bfloat16* q_bf = reinterpret_cast<const __nv_bfloat16*>(q_raw);

  if (tid == 0) {
    mbar_init(&bars->tma, 1);
    mbar_init(&bars->mma, 1);
    mbar_init(&bars->mma_q, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
    // the first chunk's inputs
    mbar_arrive_expect_tx(&bars->tma, 3 * kC * D * 2);
    load_wk<D>(base, &map_w, &map_k, blockIdx.x, Np, &bars->tma);
    load_q<D>(base, &map_q, blockIdx.x, Np, &bars->tma);
  }
  load_chunk_scalars<kGate>(sBeta, sLam, beta, lam2, blockIdx.x, Np, T, tid);
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tb = bars->tmem_base;
  const uint32_t lb = static_cast<uint32_t>(quarter * 32) << 16;
  uint32_t mma_phase = 0, q_phase = 0, tma_phase = 0;
  bool ok = true, tma_pending = true;   // tma_pending: thread 0's view
  float tv[64];                         // the previous chunk's diagonal logits
  int prev = -1;

  for (int ch = blockIdx.x; ch < nch; ch += grid) {
  const int next = ch + grid;

  // ---- P1: the Gram blocks, once the inputs have landed
  if (tid == 0) {
    // the next chunk's rows into L2 (its TMA copies are issued late in this
    // chunk, so that they then read from L2)
    if (next < nch) {
      const int bh2 = next / Np, t2 = (next - bh2 * Np) * kC;
      const size_t off = (static_cast<size_t>(bh2) * T + t2) * D * 2;
      const uint32_t bytes = static_cast<uint32_t>(min(kC, T - t2)) * D * 2;
      // w has wr columns (wr = D, or r for partial PaTH)
      const size_t off_w = (static_cast<size_t>(bh2) * T + t2) * wr * 2;
      const uint32_t bytes_w = static_cast<uint32_t>(min(kC, T - t2)) * wr * 2;
      bulk_prefetch_l2(w_raw + off_w, bytes_w);
      bulk_prefetch_l2(k_raw + off, bytes);
      bulk_prefetch_l2(q_raw + off, bytes);
    }
    ok = ok && mbar_wait(&bars->tma, tma_phase, &bars->abort_flag, kWaitLimitNs);
    tma_pending = false;
    if (ok) {
      tc_fence_after_sync();
      constexpr uint32_t id = idesc_bf16_f32(128, 256, false, false);
      // [W W^T | W K^T], then [Q W^T | Q K^T] (it runs while the CUDA cores
      // work on P2 and the diagonal blocks of P3; Q is overwritten by S
      // only after its completion)
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t kb = k >> 2, kk = (k & 3) * 32;
        const uint64_t bwk = sdesc_sw128(smem_addr(base + kRWK + kb * 2 * kHalf) + kk, 16, 1024);
        mma_bf16_ss(tb + 0, bwk, bwk, id, k > 0);
      }
      mma_commit(&bars->mma);
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t kb = k >> 2, kk = (k & 3) * 32;
        const uint64_t bwk = sdesc_sw128(smem_addr(base + kRWK + kb * 2 * kHalf) + kk, 16, 1024);
        const uint64_t aq = sdesc_sw128(smem_addr(base + kRQS + kb * kHalf) + kk, 16, 1024);
        mma_bf16_ss(tb + 256, aq, bwk, id, k > 0);
      }
      mma_commit(&bars->mma_q);
    } else {
      bars->abort_flag = 1;
      atomicExch(status, PATH_DEV_ERR_TIMEOUT);
      mma_commit(&bars->mma);
      mma_commit(&bars->mma_q);
    }
  }
  tma_phase ^= 1;
  // the previous chunk's diagonal logits, while the Gram products run
  if (prev >= 0) store_sdt(tv, sdt, prev, row, halfc);
  __syncthreads();   // this chunk's beta / gate prefix
  ok = wait_mma(bars, mma_phase, status) && ok;
  mma_phase ^= 1;
  tc_fence_after_sync();

  // ---- P2: the 32 x 32 diagonal blocks of L (fp32, smem)
  if (halfc == quarter >> 1) {   // the warps whose columns hold their rows' diagonal block
    const float bt = sBeta[row];
    const int c0 = 32 * quarter;
    uint32_t v[32];
    tmem_ld_x32(tb + lb + c0, v);
#pragma unroll
    for (int u = 0; u < 32; u += 4) {
      float x[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = c0 + u + e < row ? __uint_as_float(v[u + e]) * bt : 0.f;
      *reinterpret_cast<float4*>(sL + row * kSL + c0 + u) = make_float4(x[0], x[1], x[2], x[3]);
    }
  }
  tc_fence_before_sync();
  __syncthreads();

  // ---- P3: U = X D with X = (I + L)^{-1}, as bf16 hi/lo tiles (K-major A).
  // With G = W W^T and L = strictLower(D G), every off-diagonal block of a
  // 2 x 2 split of a diagonal block of U follows from its diagonal blocks:
  // (I + L) X = I gives X_ba = -X_bb D_b G_ba X_aa, so U_ba = -U_bb G_ba U_aa.
  // The 32 x 32 diagonal blocks come from the CUDA cores (fp32); the levels of
  // 32 and 64 are two tensor-core products each, on hi/lo operands.
  invert_diag32<kSL>(sL, tid);
  uint8_t* const u_hi = base + kRL;
  uint8_t* const u_lo = base + kRL + kTile;
  {
    // row `row`, columns [64 halfc, 64 halfc + 64): the diagonal block X D,
    // G below it (the blocks the levels turn into U), zeros above
    float xd[32];
    const bool diag_here = (quarter >> 1) == halfc;
    if (diag_here) {
      const int c0 = 32 * quarter;
#pragma unroll
      for (int u = 0; u < 32; u += 4) {
        const float4 x = *reinterpret_cast<const float4*>(sL + row * kSL + c0 + u);
        const float4 b = *reinterpret_cast<const float4*>(sBeta + c0 + u);
        xd[u] = c0 + u <= row ? x.x * b.x : 0.f;
        xd[u + 1] = c0 + u + 1 <= row ? x.y * b.y : 0.f;
        xd[u + 2] = c0 + u + 2 <= row ? x.z * b.z : 0.f;
        xd[u + 3] = c0 + u + 3 <= row ? x.w * b.w : 0.f;
      }
    }
    __syncthreads();   // the fp32 blocks are read; the tiles overwrite them
    // S = strictLower(W K^T) -> bf16 hi/lo (MN-major B) over Q, once the query
    // Gram product that reads Q is done
    ok = wait_mma(bars, q_phase, status, &bars->mma_q) && ok;
    q_phase ^= 1;
    tc_fence_after_sync();
#pragma unroll
    for (int cc = 0; cc < 64; cc += 32) {
      const int c0 = halfc * 64 + cc;
      uint32_t v[32];
      tmem_ld_x32(tb + lb + 128 + c0, v);
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) {
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = c0 + g8 * 8 + u;
          x[u] = c < row ? __uint_as_float(v[g8 * 8 + u]) : 0.f;
        }
        put_hilo8(base + kRQS, base + kRQS + kTile, row, (c0 >> 3) + g8, x);
      }
    }
#pragma unroll
    for (int cc = 0; cc < 64; cc += 32) {
      const int c0 = halfc * 64 + cc, cb = c0 >> 5;
      float x[32];
      if (cb < quarter) {
        uint32_t v[32];
        tmem_ld_x32(tb + lb + c0, v);
#pragma unroll
        for (int u = 0; u < 32; ++u) x[u] = __uint_as_float(v[u]);
      } else if (cb == quarter) {
#pragma unroll
        for (int u = 0; u < 32; ++u) x[u] = xd[u];
      } else {
#pragma unroll
        for (int u = 0; u < 32; ++u) x[u] = 0.f;
      }
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8)
        put_hilo8(u_hi, u_lo, row, (c0 >> 3) + g8, *reinterpret_cast<const float(*)[8]>(&x[g8 * 8]));
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before_sync();
  __syncthreads();
  {
    constexpr uint32_t id64 = idesc_bf16_f32(128, 64, false, true);
    const uint32_t uh = smem_addr(u_hi), ul = smem_addr(u_lo), eb = smem_addr(base + kRE);
    auto a_desc = [&](uint32_t t, int k) {   // K-major A, k-step k of 16 columns
      return sdesc_sw128(t + (k >> 2) * kHalf + (k & 3) * 32, 16, 1024);
    };
    auto b_desc = [&](uint32_t t) { return sdesc_sw128(t, kHalf, 1024); };
    uint8_t* const e_tiles = base + kRE;
    // one round of MMAs issued by thread 0, then every thread waits for it
    auto mma_round = [&](auto&& body) {
      if (tid == 0) {
        if (ok) {
          tc_fence_after_sync();
          body();
        }
        mma_commit(&bars->mma);
      }
      ok = wait_mma(bars, mma_phase, status) && ok;
      mma_phase ^= 1;
      tc_fence_after_sync();
    };
    auto publish = [&]() {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before_sync();
      __syncthreads();
    };
    // Each product of a level is hi*hi + hi*lo + lo*hi; the first two share
    // A = hi, so they run as one MMA of width 128 whose B is the hi tile
    // followed by the lo tile (its second 64-wide atom at the lo tile's
    // offset): D[:, 0:64) = hi*hi (+ lo*hi, issued after it), D[:, 64:128)
    // = hi*lo, summed by the readers.  Two instructions per k-step, not three.
    constexpr uint32_t id128 = idesc_bf16_f32(128, 128, false, true);
    auto pair_b = [&](uint32_t hi, uint32_t lo_off) { return sdesc_sw128(hi, lo_off, 1024); };
    auto ld_sum32 = [&](uint32_t col, float (&x)[32]) {   // D[:, col] + D[:, col + 64]
      uint32_t v[32], w[32];
      tmem_ld_x32(tb + lb + col, v);
      tmem_ld_x32(tb + lb + col + 64, w);
#pragma unroll
      for (int u = 0; u < 32; ++u) x[u] = __uint_as_float(v[u]) + __uint_as_float(w[u]);
    };
    // level 32, pairs p = 0, 1 (a = rows 64p.., b = rows 64p + 32..):
    // E_p = G_ba U_aa -> TMEM cols [128p, 128p + 128) (cols 32.. of each half are zero)
    mma_round([&] {
      for (int p = 0; p < 2; ++p)
        for (int j = 0; j < 2; ++j) {
          const uint32_t bo = p * kHalf + (4 * p + j) * 2048;
          mma_bf16_ss(tb + 128 * p, a_desc(uh, 4 * p + j), pair_b(uh + bo, kTile), id128, j > 0);
          mma_bf16_ss(tb + 128 * p, a_desc(ul, 4 * p + j), b_desc(uh + bo), id64, 1);
        }
    });
    if (quarter & 1) {   // E_p rows are lanes of quarter 2p + 1 -> MN-major B tile
      const int p = quarter >> 1;
      float x32[32];
      ld_sum32(128 * p + 32 * halfc, x32);
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8)
        put_hilo8(e_tiles + p * 8192, e_tiles + p * 8192 + 4096, lane, 4 * halfc + g8,
                  *reinterpret_cast<const float(*)[8]>(&x32[g8 * 8]));
    }
    publish();
    // U_bb E_p -> TMEM cols [128p, 128p + 128)
    mma_round([&] {
      for (int p = 0; p < 2; ++p)
        for (int j = 0; j < 2; ++j) {
          const uint32_t be = eb + p * 8192 + j * 2048;
          mma_bf16_ss(tb + 128 * p, a_desc(uh, 4 * p + 2 + j), pair_b(be, 4096), id128, j > 0);
          mma_bf16_ss(tb + 128 * p, a_desc(ul, 4 * p + 2 + j), b_desc(be), id64, 1);
        }
    });
    if (quarter & 1) {   // U_ba = -U_bb E_p, 16 columns per warp
      const int p = quarter >> 1;
      uint32_t v[16], w[16];
      tmem_ld_x16(tb + lb + 128 * p + 16 * halfc, v);
      tmem_ld_x16(tb + lb + 128 * p + 64 + 16 * halfc, w);
#pragma unroll
      for (int g8 = 0; g8 < 2; ++g8) {
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          x[u] = -(__uint_as_float(v[g8 * 8 + u]) + __uint_as_float(w[g8 * 8 + u]));
        put_hilo8(u_hi, u_lo, row, 8 * p + 2 * halfc + g8, x);
      }
    }
    publish();
    // level 64: E = G_21 U_11 -> TMEM cols [0, 128)
    mma_round([&] {
      for (int j = 0; j < 4; ++j) {
        mma_bf16_ss(tb, a_desc(uh, j), pair_b(uh + j * 2048, kTile), id128, j > 0);
        mma_bf16_ss(tb, a_desc(ul, j), b_desc(uh + j * 2048), id64, 1);
      }
    });
    if (quarter >= 2) {
      float x32[32];
      ld_sum32(32 * halfc, x32);
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8)
        put_hilo8(e_tiles, e_tiles + 8192, row - 64, 4 * halfc + g8,
                  *reinterpret_cast<const float(*)[8]>(&x32[g8 * 8]));
    }
    publish();
    // U_22 E -> TMEM cols [128, 256)
    mma_round([&] {
      for (int j = 0; j < 4; ++j) {
        mma_bf16_ss(tb + 128, a_desc(uh, 4 + j), pair_b(eb + j * 2048, 8192), id128, j > 0);
        mma_bf16_ss(tb + 128, a_desc(ul, 4 + j), b_desc(eb + j * 2048), id64, 1);
      }
    });
    if (quarter >= 2) {   // U_21 = -U_22 E
      float x32[32];
      ld_sum32(128 + 32 * halfc, x32);
#pragma unroll
      for (int u = 0; u < 32; ++u) x32[u] = -x32[u];
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8)
        put_hilo8(u_hi, u_lo, row, 4 * halfc + g8, *reinterpret_cast<const float(*)[8]>(&x32[g8 * 8]));
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
      if (uwn != nullptr && halfc == 1) {
        // the low-rank transition form reads -(U W) as a bf16 operand
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          pk[u] = pack_bf16x2(-__uint_as_float(v[2 * u]), -__uint_as_float(v[2 * u + 1]));
        uint4* dst = reinterpret_cast<uint4*>(uwn + (static_cast<size_t>(ch) * kC + row) * D + cc);
#pragma unroll
        for (int u = 0; u < 4; ++u) dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
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
  // meanwhile: -lower(Q W^T) -> bf16 hi / lo A operand in TMEM columns [256, 384),
  // each warp 64 of its rows' 128 values; the hi / lo columns overlap the
  // source, so both warps of a lane quarter have read before either writes
  {
    uint32_t v[64];
    tmem_ld_x64(tb + lb + 256 + 64 * halfc, v);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    uint32_t ph[32], pl[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const int c = 64 * halfc + 2 * u;
      const float x0 = c <= row ? -__uint_as_float(v[2 * u]) : 0.f;
      const float x1 = c + 1 <= row ? -__uint_as_float(v[2 * u + 1]) : 0.f;
      split_hilo2(x0, x1, ph[u], pl[u]);
    }
    tmem_st_x32(tb + lb + 256 + 32 * halfc, ph);
    tmem_st_x32(tb + lb + 320 + 32 * halfc, pl);
    tmem_st_wait();
  }
  ok = wait_mma(bars, mma_phase, status) && ok;
  mma_phase ^= 1;
  tc_fence_after_sync();
  // epilogue, first half: this thread's output row as bf16 pairs in registers,
  // kr[j][:] = K[j][:] - kr'[j][:] (half 0, row j = lane), ngt[n][:] =
  // -ngt'[n][:] (half 1, rows n < D); stored while P6b runs
  uint32_t orow[D / 2];
  if (halfc == 0) {
    const int j = row;
    const uint8_t* kt = base + kRWK + kHalf;  // K rows inside the W|K halves
#pragma unroll
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
#pragma unroll
        for (int e = 0; e < 4; ++e)
          orow[f0 / 2 + e] = pack_bf16x2(__uint_as_float(kw[e] << 16) - __uint_as_float(v[u8 + 2 * e]),
                                         __uint_as_float(kw[e] & 0xffff0000u) -
                                             __uint_as_float(v[u8 + 2 * e + 1]));
      }
    }
  } else if (row < D) {
#pragma unroll
    for (int cc = 0; cc < D; cc += 32) {
      uint32_t v[32];
      tmem_ld_x32(tb + lb + 128 + cc, v);
#pragma unroll
      for (int u = 0; u < 16; ++u)
        orow[cc / 2 + u] = pack_bf16x2(-__uint_as_float(v[2 * u]), -__uint_as_float(v[2 * u + 1]));
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before_sync();
  __syncthreads();

  // the next chunk's W and K into the W | K region (free from here on)
  if (tid == 0 && next < nch && ok) {
    mbar_arrive_expect_tx(&bars->tma, 3 * kC * D * 2);
    load_wk<D>(base, &map_w, &map_k, next, Np, &bars->tma);
    tma_pending = true;
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
  // epilogue of P6a, second half: the kr / ngt rows, 32 bytes per store
  if (halfc == 0 || row < D) {
    uint32_t* out = halfc == 0
                        ? reinterpret_cast<uint32_t*>(kr + (static_cast<size_t>(ch) * kC + row) * D)
                        : reinterpret_cast<uint32_t*>(ngt + (static_cast<size_t>(ch) * D + row) * D);
#pragma unroll
    for (int u = 0; u < D / 2; u += 8) st_global_v8(out + u, &orow[u]);
  }
  uint2 qv[kC * D / 4 / kThreads];   // this chunk's Q rows, read while P6b runs
  load_q_rows<D>(qv, q_bf, ch, Np, T, tid);
  ok = wait_mma(bars, mma_phase, status) && ok;
  mma_phase ^= 1;
  tc_fence_after_sync();
  // the region of [TK | UW] hi is free: the next chunk's Q
  if (tid == 0 && next < nch && tma_pending) load_q<D>(base, &map_q, next, Np, &bars->tma);
  // last epilogue, read out of the tensor memory: the diagonal logits sdt[j][i]
  // from Q K^T + sd' for keys j in [64 halfc, 64 halfc + 64) into registers
  // (stored after the next chunk's Gram products have been issued), ql' for
  // features [D/2 halfc, D/2 (halfc + 1)) to shared memory (the lo tiles are
  // dead once the MMA is done) for the coalesced ql rows
  {
    const int i = row;
    const float li = kGate ? sLam[i] : 0.f;
#pragma unroll
    for (int cc = 0; cc < 64; cc += 32) {
      uint32_t v[32], qk[32];
      tmem_ld_x32(tb + lb + 64 * halfc + cc, v);
      tmem_ld_x32(tb + lb + 384 + 64 * halfc + cc, qk);
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const int j = 64 * halfc + cc + u;
        const float gj = kGate ? sLam[j] : 0.f;
        tv[cc + u] =
            j <= i ? fmaf(__uint_as_float(qk[u]) + __uint_as_float(v[u]), sl2, li - gj) : -INFINITY;
      }
    }
    float* sq = sL;
#pragma unroll
    for (int cc = (D / 2) * halfc; cc < (D / 2) * (halfc + 1); cc += 32) {
      uint32_t v[32];
      tmem_ld_x32(tb + lb + 128 + cc, v);
#pragma unroll
      for (int u = 0; u < 32; u += 4)
        *reinterpret_cast<float4*>(sq + i * kSL + cc + u) =
            make_float4(__uint_as_float(v[u]), __uint_as_float(v[u + 1]),
                        __uint_as_float(v[u + 2]), __uint_as_float(v[u + 3]));
    }
  }
  prev = ch;
  tc_fence_before_sync();
  __syncthreads();
  store_ql<D>(qv, sL, ql, ch, tid);
  // the tensor memory, the staging region and the chunk's beta / gate prefix
  // are free
  if (__syncthreads_or(bars->abort_flag != 0)) break;
  if (next < nch) load_chunk_scalars<kGate>(sBeta, sLam, beta, lam2, next, Np, T, tid);
  }  // chunks

  if (prev >= 0) store_sdt(tv, sdt, prev, row, halfc);
  // after an expired wait: copies still in flight land before the CTA exits
  if (tid == 0 && tma_pending) mbar_wait(&bars->tma, tma_phase, nullptr, kWaitLimitNs);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tb, 512);
  }
}

// The driver's tensor-map encoder, looked up once: a function-local static
// is initialised exactly once even when host threads make their first call
// at the same time.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    const bool found = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                        cudaEnableDefault, &qr) == cudaSuccess &&
                       qr == cudaDriverEntryPointSuccess;
    return found ? reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p) : nullptr;
  }();
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
  // w may have fewer columns than D (partial PaTH): its boxes then read zeros
  // past column wr, which makes every transition the identity there
  const int wr = in.wr > 0 ? in.wr : D;
  if (wr > D || wr % 64 != 0) return cudaErrorInvalidValue;
  if (!make_input_map(&mw, in.w, wr, g.T, g.BH) || !make_input_map(&mk, in.k, D, g.T, g.BH) ||
      !make_input_map(&mq, in.q, D, g.T, g.BH))
    return cudaErrorInvalidValue;
  auto kern = prep_tc_kernel<D, kGate>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = std::min(g.nch, std::max(sms, 1));   // one persistent CTA per SM
  kern<<<grid, kThreads, kSmemBytes, st>>>(
      mw, mk, mq, static_cast<const uint8_t*>(in.w), static_cast<const uint8_t*>(in.k),
      static_cast<const uint8_t*>(in.q), in.beta, ws.lam2,
      static_cast<__nv_bfloat16*>(ws.kr), ws.ql, static_cast<__nv_bfloat16*>(ws.ngt), ws.sdt,
      static_cast<__nv_bfloat16*>(ws.uwn), status, g.T, g.Np, g.nch, in.scale * kLog2e, wr);
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
