// producer_tc.cu -- the w / beta producer's projection on tcgen05 (bf16).
//
// Same computation as producer.cu (slides' frame "PaTH inserts a learned
// transformation along every path"; OpenReview section "Model Architecture
// Details"; readings listed there):
//
// producer_proj_tc_kernel  128 tokens per CTA: acc = x [Wd ; Ub]^T, width
//     N = R + H (padded to 16), K = Dm in 64-column stages (TMA, three-stage
//     ring, 128-byte swizzle).  Epilogue, one thread per token row: the first
//     R columns to the bf16 workspace `low`, the last H to
//     beta = 2 sigmoid(. + b) in [B, H, T].
// Warps: 0 TMA producer, 1 TMEM allocation + MMA issue, 2-5 epilogue (TMEM
// lane quarter = warp % 4).  Every mbarrier wait is bounded and records a timeout in
// the status word.
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

constexpr int kThreadsTc = 192;
constexpr int kTileRows = 128;
constexpr int kStagesTc = 3;
constexpr uint32_t kABytes = 128 * 128;     // 128 rows x 64 bf16
constexpr uint32_t kStageTc = 2 * kABytes;  // A, then B (up to 128 rows)

struct ProjTcArgs {
  const float* bb;
  bf16* low;
  float* beta;
  int* status;
  int BT, T, Dm, H, R, NP;
};

struct TcBars {
  uint64_t full[kStagesTc], empty[kStagesTc], acc;
  uint32_t tmem;
  int abort_flag;
};

__device__ __forceinline__ void fail(TcBars* bars, int* status) {
  bars->abort_flag = 1;
  atomicExch(status, PATH_DEV_ERR_TIMEOUT);
}

__device__ __forceinline__ void finish(int warp, uint32_t tb, uint32_t ncols) {
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tb, ncols);
  }
}

// ---------------------------------------------------------------- projection
__global__ void __launch_bounds__(kThreadsTc, 1)
    producer_proj_tc_kernel(const __grid_constant__ CUtensorMap map_x,
                            const __grid_constant__ CUtensorMap map_wd,
                            const __grid_constant__ CUtensorMap map_ub, const ProjTcArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  TcBars* bars = reinterpret_cast<TcBars*>(base + kStagesTc * kStageTc);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int r0 = blockIdx.x * kTileRows, nk = p.Dm / 64, N = p.R + p.H;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesTc; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->acc, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  // rows N .. NP - 1 of every B stage are zero (never written by the copies)
  for (int x = threadIdx.x; x < kStagesTc * (p.NP - N) * 8; x += blockDim.x) {
    const int s = x / ((p.NP - N) * 8), rem = x % ((p.NP - N) * 8);
    *reinterpret_cast<uint4*>(base + s * kStageTc + kABytes + (N + rem / 8) * 128 + (rem % 8) * 16) =
        make_uint4(0u, 0u, 0u, 0u);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 1) {
    tmem_alloc(&bars->tmem, 128);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tb = bars->tmem;
  const uint64_t LIM = kWaitLimitNs;
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_map(&map_x);
      bool ok = true;
      int last[kStagesTc] = {-1, -1, -1};
      const uint32_t bytes = kABytes + static_cast<uint32_t>(N) * 128;
      for (int kc = 0; kc < nk && ok; ++kc) {
        const int s = kc % kStagesTc;
        if (kc >= kStagesTc)
          ok = mbar_wait(&bars->empty[s], ((kc / kStagesTc) - 1) & 1, &bars->abort_flag, LIM);
        if (!ok) break;
        uint8_t* st = base + s * kStageTc;
        mbar_arrive_expect_tx(&bars->full[s], bytes);
        tma_load_2d(st, &map_x, kc * 64, r0, &bars->full[s]);
        tma_load_2d(st + kABytes, &map_wd, kc * 64, 0, &bars->full[s]);
        tma_load_2d(st + kABytes + p.R * 128, &map_ub, kc * 64, 0, &bars->full[s]);
        last[s] = (kc / kStagesTc) & 1;
      }
      if (!ok) fail(bars, p.status);
      for (int s = 0; s < kStagesTc; ++s)
        if (last[s] >= 0) mbar_wait(&bars->full[s], last[s], nullptr, LIM);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id = idesc_bf16_f32(128, p.NP, false, false);
      bool ok = true;
      for (int kc = 0; kc < nk && ok; ++kc) {
        const int s = kc % kStagesTc;
        ok = mbar_wait(&bars->full[s], (kc / kStagesTc) & 1, &bars->abort_flag, LIM);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t a = smem_addr(base + s * kStageTc), b = a + kABytes;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16_ss(tb, sdesc_sw128(a + k * 32, 16, 1024), sdesc_sw128(b + k * 32, 16, 1024), id,
                      kc > 0 || k > 0);
        mma_commit(&bars->empty[s]);
      }
      if (!ok) fail(bars, p.status);
      mma_commit(&bars->acc);
      mbar_wait(&bars->acc, 0, nullptr, LIM);
    }
  } else {
    const int q = warp & 3, row = q * 32 + lane, grow = r0 + row;
    const bool ok = mbar_wait(&bars->acc, 0, &bars->abort_flag, LIM);
    if (ok) {
      tc_fence_after_sync();
      const uint32_t tl = tb + (static_cast<uint32_t>(q * 32) << 16);
      const int b = grow / p.T, t = grow % p.T;
      for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t v[32];
        tmem_ld_x32(tl + c0, v);
        if (grow >= p.BT) continue;
#pragma unroll
        for (int u = 0; u < 32; u += 8) {
          const int c = c0 + u;
          if (c + 8 <= p.R) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(v[u]), __uint_as_float(v[u + 1]));
            o.y = pack_bf16x2(__uint_as_float(v[u + 2]), __uint_as_float(v[u + 3]));
            o.z = pack_bf16x2(__uint_as_float(v[u + 4]), __uint_as_float(v[u + 5]));
            o.w = pack_bf16x2(__uint_as_float(v[u + 6]), __uint_as_float(v[u + 7]));
            *reinterpret_cast<uint4*>(p.low + static_cast<size_t>(grow) * p.R + c) = o;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int h = c + e - p.R;
              if (h >= 0 && h < p.H)
                p.beta[(static_cast<size_t>(b) * p.H + h) * p.T + t] =
                    2.f / (1.f + expf(-(__uint_as_float(v[u + e]) + p.bb[h])));
            }
          }
        }
      }
    } else {
      fail(bars, p.status);
    }
  }
  finish(warp, tb, 128);
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

// Row-major bf16 [rows][cols] seen with 128-byte-swizzled boxes of 64 columns
// x box_rows rows (rows outside the matrix read as zero).
bool map2d(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_producer_proj_tc(const void* x, const void* Wd, const void* Ub,
                                    const float* bb, void* low, float* beta, int* status, int B,
                                    int T, int Dm, int H, int R, cudaStream_t st) {
  const int BT = B * T, N = R + H, NP = (N + 15) / 16 * 16;
  if (NP > 128 || R % 8 != 0 || Dm % 64 != 0) return cudaErrorInvalidValue;
  CUtensorMap mx, md, mu;
  if (!map2d(&mx, x, Dm, BT, kTileRows) || !map2d(&md, Wd, Dm, R, R) ||
      !map2d(&mu, Ub, Dm, H, H))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + kStagesTc * kStageTc + sizeof(TcBars);
  cudaError_t e = cudaFuncSetAttribute(producer_proj_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const ProjTcArgs p{bb, static_cast<bf16*>(low), beta, status, BT, T, Dm, H, R, NP};
  producer_proj_tc_kernel<<<(BT + kTileRows - 1) / kTileRows, kThreadsTc, smem, st>>>(mx, md, mu,
                                                                                     p);
  return cudaGetLastError();
}

}  // namespace pathattn
