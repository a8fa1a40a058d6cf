// producer_mix_tc.cu -- the w / beta producer's mixing step on tcgen05 (bf16,
// R = 64).
//
// The slides' frame "PaTH inserts a learned transformation along every path"
// gives w_t from a low-rank projection, a width-3 causal convolution and an
// L2 normalization; with this library's readings (producer.cu)
//   z_t = cw_0 * p_{t-2} + cw_1 * p_{t-1} + cw_2 * p_t,   p_s = low_s Wu_h^T,
// and since every tap multiplies an output channel, the convolution folds
// into the weights:
//   z_t = [low_{t-2} | low_{t-1} | low_t] [cw_0 . Wu_h ; cw_1 . Wu_h ; cw_2 . Wu_h]^T,
// one product of width K = 3R per head.  The folded weights (bf16, one
// [d][3 * 64] tile per head) are made once per call by a small kernel.
//
// producer_mix_tc_kernel: one CTA per 128 tokens of one sequence and a group
// of heads.  The three row-shifted copies of the low-rank tile are three TMA
// loads at rows t0 - 2, t0 - 1, t0 of a per-sequence tensor map, so the rows
// before a sequence start read as zero (the causal padding).  Folded weights
// stream per head through a two-stage TMA ring; the product of head i
// accumulates in one of two TMEM buffers while the epilogue warps normalise
// head i - 1 (one token row per thread), write it as bf16 into one of two
// swizzled shared-memory tiles and store it with a TMA tensor store.
// Warps: 0 TMA, 1 TMEM + MMA issue, 2-5 epilogue (TMEM lane quarter = warp % 4;
// warp 2 lane 0 issues the stores).  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace pathattn {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kRows = 128;        // tokens per CTA
constexpr int kR = 64;            // rank of the low-rank projection
constexpr int kFoldK = 3 * kR;    // folded product width
constexpr int kHeadsPerCta = 8;
constexpr int kThreads = 192;
constexpr uint32_t kACopy = kRows * 128;  // one [128][64] bf16 copy (16 KB)

template <int D>
struct MixCfg {
  static constexpr uint32_t kBStage = 3 * D * 128;          // [D][192] as 3 halves
  static constexpr uint32_t kOut = (D / 64) * kRows * 128;  // [128][D] bf16
  static constexpr uint32_t kOffB = 3 * kACopy;
  static constexpr uint32_t kOffOut = kOffB + 2 * kBStage;
  static constexpr uint32_t kTmemCols = 2 * D;
  static constexpr size_t kSmemBytes = kOffOut + 2 * kOut + 1024 + 256;
};

struct MixBars {
  uint64_t a_full, b_full[2], b_empty[2], acc_full[2], acc_empty[2], final_done;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void mix_fail(MixBars* bars, int* status) {
  bars->abort_flag = 1;
  atomicExch(status, PATH_DEV_ERR_TIMEOUT);
}

// Epilogue helpers: one arrival per warp; barrier of the four epilogue warps
// (named barrier 2, 128 threads).
__device__ __forceinline__ void warp_arrive_mix(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
__device__ __forceinline__ void mix_bar() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int x, int y, int z,
                                             const void* src) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_addr(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Folded weights: bf[(h * D + c) * 192 + j * 64 + r] = cw[h * D + c][j] * Wu[h * D + c][r].
__global__ void __launch_bounds__(256) producer_fold_kernel(const bf16* __restrict__ Wu,
                                                            const float* __restrict__ cw,
                                                            bf16* __restrict__ bf, int rows) {
  const int i = blockIdx.x * 256 + threadIdx.x;  // (row, j, 8-column group)
  if (i >= rows * 3 * (kR / 8)) return;
  const int row = i / (3 * (kR / 8)), rem = i - row * 3 * (kR / 8);
  const int j = rem / (kR / 8), r0 = (rem - j * (kR / 8)) * 8;
  const float tap = cw[static_cast<size_t>(row) * 3 + j];
  const uint4 u = *reinterpret_cast<const uint4*>(Wu + static_cast<size_t>(row) * kR + r0);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    o[e] = pack_bf16x2(tap * __uint_as_float(w[e] << 16), tap * __uint_as_float(w[e] & 0xffff0000u));
  *reinterpret_cast<uint4*>(bf + static_cast<size_t>(row) * kFoldK + j * kR + r0) =
      make_uint4(o[0], o[1], o[2], o[3]);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    producer_mix_tc_kernel(const __grid_constant__ CUtensorMap map_low,
                           const __grid_constant__ CUtensorMap map_bf,
                           const __grid_constant__ CUtensorMap map_w, int* __restrict__ status,
                           int T, int H) {
  using Cfg = MixCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  MixBars* bars = reinterpret_cast<MixBars*>(base + Cfg::kOffOut + 2 * Cfg::kOut);
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t0 = blockIdx.x * kRows, b = blockIdx.y, h0 = blockIdx.z * kHeadsPerCta;
  const int nh = min(kHeadsPerCta, H - h0);
  const uint64_t LIM = kWaitLimitNs;

  if (threadIdx.x == 0) {
    mbar_init(&bars->a_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->b_full[s], 1);
      mbar_init(&bars->b_empty[s], 1);
      mbar_init(&bars->acc_full[s], 1);
      mbar_init(&bars->acc_empty[s], 4);
    }
    mbar_init(&bars->final_done, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&map_low);
    tma_prefetch_map(&map_bf);
  }
  if (warp == 2 && lane == 0) tma_prefetch_map(&map_w);
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tb = bars->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // the three row-shifted copies: rows t0 - 2 + j of this sequence
      // (rows before its start read as zero)
      mbar_arrive_expect_tx(&bars->a_full, 3 * kACopy);
      for (int j = 0; j < 3; ++j)
        tma_load_3d(base + j * kACopy, &map_low, 0, t0 - 2 + j, b, &bars->a_full);
      int last[2] = {-1, -1};
      bool ok = true;
      for (int i = 0; i < nh && ok; ++i) {
        const int s = i & 1;
        if (i >= 2) ok = mbar_wait(&bars->b_empty[s], ((i >> 1) - 1) & 1, abort_flag, LIM);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars->b_full[s], Cfg::kBStage);
        for (int j = 0; j < 3; ++j)
          tma_load_2d(base + Cfg::kOffB + s * Cfg::kBStage + j * (D * 128), &map_bf, j * kR,
                      (h0 + i) * D, &bars->b_full[s]);
        last[s] = (i >> 1) & 1;
      }
      if (!ok) mix_fail(bars, status);
      mbar_wait(&bars->a_full, 0, nullptr, LIM);
      for (int s = 0; s < 2; ++s)
        if (last[s] >= 0) mbar_wait(&bars->b_full[s], last[s], nullptr, LIM);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id = idesc_bf16_f32(128, D, false, false);
      const uint32_t a0 = smem_addr(base);
      bool ok = mbar_spin(&bars->a_full, 0, abort_flag, LIM);
      for (int i = 0; i < nh && ok; ++i) {
        const int s = i & 1;
        ok = mbar_spin(&bars->b_full[s], (i >> 1) & 1, abort_flag, LIM);
        if (ok && i >= 2) ok = mbar_spin(&bars->acc_empty[s], ((i >> 1) - 1) & 1, abort_flag, LIM);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t bb = smem_addr(base + Cfg::kOffB + s * Cfg::kBStage);
#pragma unroll
        for (int j = 0; j < 3; ++j)
#pragma unroll
          for (int k = 0; k < kR / 16; ++k)
            mma_bf16_ss(tb + s * D, sdesc_sw128(a0 + j * kACopy + k * 32, 16, 1024),
                        sdesc_sw128(bb + j * (D * 128) + k * 32, 16, 1024), id, (j > 0 || k > 0));
        mma_commit(&bars->acc_full[s]);
        mma_commit(&bars->b_empty[s]);
      }
      if (!ok) mix_fail(bars, status);
      mma_commit(&bars->final_done);
      mbar_wait(&bars->final_done, 0, nullptr, LIM);
    }
  } else {
    // epilogue: token row r of this tile, w = z / max(|z|, 1e-12)
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const bool leader = warp == 2 && lane == 0;
    const uint32_t lb = static_cast<uint32_t>(q4 * 32) << 16;
    bool ok = true;
    for (int i = 0; i < nh; ++i) {
      const int s = i & 1;
      ok = mbar_wait(&bars->acc_full[s], (i >> 1) & 1, abort_flag, LIM);
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t v[D];
#pragma unroll
      for (int cc = 0; cc < D; cc += 32)
        tmem_ld_x32(tb + lb + s * D + cc, *reinterpret_cast<uint32_t(*)[32]>(&v[cc]));
      tc_fence_before_sync();
      warp_arrive_mix(&bars->acc_empty[s]);
      float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
      for (int c = 0; c < D; c += 2) {
        ss0 = fmaf(__uint_as_float(v[c]), __uint_as_float(v[c]), ss0);
        ss1 = fmaf(__uint_as_float(v[c + 1]), __uint_as_float(v[c + 1]), ss1);
      }
      const float inv = 1.f / fmaxf(sqrtf(ss0 + ss1), 1e-12f);
      // the staging tile of head i - 2 has been read by its store
      if (leader) bulk_wait_read<1>();
      mix_bar();
      uint8_t* out = base + Cfg::kOffOut + s * Cfg::kOut;
#pragma unroll
      for (int c8 = 0; c8 < D / 8; ++c8) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(v[8 * c8 + 2 * e]) * inv,
                              __uint_as_float(v[8 * c8 + 2 * e + 1]) * inv);
        const uint32_t off = (c8 >> 3) * (kRows * 128) + r * 128 + (((c8 & 7) ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(out + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      fence_proxy_async_smem();
      mix_bar();
      if (leader) {
        // rows past the sequence end are outside the tensor map: not written
        for (int hh = 0; hh < D / 64; ++hh)
          tma_store_3d(&map_w, hh * 64, t0, b * H + h0 + i, out + hh * (kRows * 128));
        bulk_commit();
      }
    }
    if (!ok) mix_fail(bars, status);
    if (leader) bulk_wait<0>();
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tb, Cfg::kTmemCols);
  }
}

// The driver's tensor-map encoder, looked up once: a function-local static
// is initialised exactly once even when host threads make their first call
// at the same time.
PFN_cuTensorMapEncodeTiled_v12000 mix_encode_fn() {
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

// bf16 [z][rows][cols] row-major, 128-byte swizzled boxes of 64 columns x
// box_rows rows (rank 2 when zdim == 1 is not wanted: rank given).
bool mix_map(CUtensorMap* m, const void* ptr, int rank, uint64_t cols, uint64_t rows,
             uint64_t zdim, uint32_t box_rows) {
  auto enc = mix_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {cols, rows, zdim};
  cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides,
             box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_mix_t(const void* low, const void* Wu, const float* cw, void* bf, void* w,
                         int* status, int B, int T, int H, cudaStream_t st) {
  using Cfg = MixCfg<D>;
  const int rows = H * D;
  producer_fold_kernel<<<(rows * 3 * (kR / 8) + 255) / 256, 256, 0, st>>>(
      static_cast<const bf16*>(Wu), cw, static_cast<bf16*>(bf), rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap ml, mb, mw;
  if (!mix_map(&ml, low, 3, kR, T, B, kRows) || !mix_map(&mb, bf, 2, kFoldK, rows, 1, D) ||
      !mix_map(&mw, w, 3, D, T, static_cast<uint64_t>(B) * H, kRows))
    return cudaErrorInvalidValue;
  auto kern = producer_mix_tc_kernel<D>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(Cfg::kSmemBytes))) != cudaSuccess)
    return e;
  const dim3 grid((T + kRows - 1) / kRows, B, (H + kHeadsPerCta - 1) / kHeadsPerCta);
  kern<<<grid, kThreads, Cfg::kSmemBytes, st>>>(ml, mb, mw, status, T, H);
  return cudaGetLastError();
}

}  // namespace

bool producer_mix_tc_supported(int B, int T, int H, int d, int R) {
  return R == kR && (d == 64 || d == 128) && B <= 65535 && (H + kHeadsPerCta - 1) / kHeadsPerCta <= 65535;
}

size_t producer_fold_bytes(int H, int d) {
  return static_cast<size_t>(H) * d * kFoldK * sizeof(bf16);
}

cudaError_t launch_producer_mix_tc(const void* low, const void* Wu, const float* cw, void* bf,
                                   void* w, int* status, int B, int T, int H, int d,
                                   cudaStream_t st) {
  if (d == 128) return launch_mix_t<128>(low, Wu, cw, bf, w, status, B, T, H, st);
  if (d == 64) return launch_mix_t<64>(low, Wu, cw, bf, w, status, B, T, H, st);
  return cudaErrorInvalidValue;
}

}  // namespace pathattn
