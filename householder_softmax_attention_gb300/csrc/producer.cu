// producer.cu -- the producer of PaTH's w and beta from the hidden states.
//
// "PaTH Attention: Position Encoding via Accumulating Householder
// Transformations" (slides, frame "PaTH inserts a learned transformation
// along every path"): w_t comes from a low-rank projection, a width-3
// convolution and an L2 normalization, and beta_t = 2 sigmoid(u^T x_t + b).
// The OpenReview discussion (section "Model Architecture Details") makes the
// normalization per head and the projection low-rank.  This library's
// readings: p = (x Wd^T) Wu^T without bias; causal depthwise convolution
// z_t = cw0 p_{t-2} + cw1 p_{t-1} + cw2 p_t (zero before the sequence start),
// no activation; w = z / max(|z|, 1e-12) per (token, head); one u and b per
// head.
//
// projection          low = x [Wd ; Ub]^T: bf16 on tcgen05 (producer_tc.cu),
//                     fp32 here (SIMT).  The first R columns are kept
//                     (workspace, in the input dtype), the last H become
//                     beta = 2 sigmoid(. + b) in [B, H, T].
// producer_mix_*_kernel per 112-token tile (bf16: and group of 4 heads, whose
//                       low rows plus 16 of history are loaded once): per
//                       head, p = low Wu_h^T (bf16: mma.sync in registers,
//                       Wu_h of the next head prefetched with cp.async), the
//                       causal convolution, the L2 normalization, and w in
//                       [B,H,T,d].
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace pathattn {
namespace {

using bf16 = __nv_bfloat16;

__device__ __forceinline__ void cp16_zfill(void* dst, const void* src, bool valid) {
  const int bytes = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8x8 bf16 matrices from shared memory; lane l supplies the address of
// row (l % 8) of matrix (l / 8).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const bf16* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}
// A fragment (16 x 16) at (m0, k0) of a row-major tile with stride S.
__device__ __forceinline__ void ldsm_a(uint32_t (&a)[4], const bf16* s, int S, int m0, int k0,
                                       int lane) {
  ldsm_x4(a, s + (m0 + (lane & 7) + ((lane >> 3) & 1) * 8) * S + k0 + (lane >> 4) * 8);
}
// B fragments of two n-tiles (n0 .. n0 + 15) x k16 from a row-major [n][k]
// tile: b[0], b[1] for n-tile n0, b[2], b[3] for n0 + 8.
__device__ __forceinline__ void ldsm_b2(uint32_t (&b)[4], const bf16* s, int S, int n0, int k0,
                                        int lane) {
  ldsm_x4(b, s + (n0 + (lane & 7) + (lane >> 4) * 8) * S + k0 + ((lane >> 3) & 1) * 8);
}

__device__ __forceinline__ float beta_of(float a) { return 2.f / (1.f + expf(-a)); }

struct ProdArgs {
  const void *x, *Wd, *Wu, *Ub;
  const float *cw, *bb;
  void* w;
  float* beta;
  void* low;  // [B*T][R] workspace: bf16 for bf16 inputs, else fp32
  int B, T, Dm, H, R;
};

__device__ __forceinline__ void store_proj(const ProdArgs& p, int row, int c, float v) {
  if (c < p.R) {
    static_cast<float*>(p.low)[static_cast<size_t>(row) * p.R + c] = v;
  } else {
    const int h = c - p.R, b = row / p.T, t = row % p.T;
    p.beta[(static_cast<size_t>(b) * p.H + h) * p.T + t] = beta_of(v + p.bb[h]);
  }
}

// ------------------------------------------------------------- projection
// fp32: one CTA per token, one thread per output column.
__global__ void __launch_bounds__(128) producer_proj_f32_kernel(const ProdArgs p) {
  extern __shared__ float xrow[];
  const int row = blockIdx.x, N = p.R + p.H;
  const float* x = static_cast<const float*>(p.x) + static_cast<size_t>(row) * p.Dm;
  for (int m = threadIdx.x; m < p.Dm; m += blockDim.x) xrow[m] = x[m];
  __syncthreads();
  for (int c = threadIdx.x; c < N; c += blockDim.x) {
    const float* wr = c < p.R ? static_cast<const float*>(p.Wd) + static_cast<size_t>(c) * p.Dm
                              : static_cast<const float*>(p.Ub) +
                                    static_cast<size_t>(c - p.R) * p.Dm;
    float s = 0.f;
    for (int m = 0; m < p.Dm; ++m) s = fmaf(xrow[m], wr[m], s);
    store_proj(p, row, c, s);
  }
}

// ----------------------------------------------------------------- mixing
constexpr int kOut = 112;            // output tokens per CTA (7 m-tiles)
constexpr int kLowRows = kOut + 16;  // plus one m-tile of history
constexpr int kHeadsPerCta = 4;

// bf16 shared memory: low [kLowRows][R + 8] bf16, Wu_h double-buffered
// [2][D][R + 8] bf16, halo [8 warps][2 rows][D] fp32, taps [4 heads][D][3] fp32.
template <int D>
__host__ __device__ inline int mix_bf16_smem_bytes(int R) {
  return (kLowRows + 2 * D) * (R + 8) * 2 + 8 * 2 * D * 4 + kHeadsPerCta * D * 3 * 4 +
         8 * 16 * (D + 8) * 2;  // + per-warp output staging [16][D + 8] bf16
}

// bf16: warp w computes p = low Wu_h^T for local rows 16 w .. 16 w + 15
// (warp 0: the 16 rows before the tile) in mma accumulators; the convolution
// takes rows r - 1, r - 2 from neighbouring lanes (shuffles) or, across the
// warp boundary, from the previous warp's last two rows in shared memory; the
// norm reduces over the 4 lanes that hold one row.
template <int D>
__global__ void __launch_bounds__(256, 2) producer_mix_bf16_kernel(const ProdArgs p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t4 = lane & 3;
  const int BT = p.B * p.T, R = p.R, LD = R + 8;
  const int r0 = blockIdx.x * kOut;
  const int h0 = blockIdx.y * kHeadsPerCta, h1 = min(p.H, h0 + kHeadsPerCta);
  bf16* lowb = reinterpret_cast<bf16*>(smem);
  bf16* wub = lowb + kLowRows * LD;
  float* halo = reinterpret_cast<float*>(smem + (kLowRows + 2 * D) * LD * 2);
  float* taps = halo + 8 * 2 * D;
  constexpr int OLD = D + 8;  // bf16 row stride of the output staging (conflict-free)
  bf16* stage = reinterpret_cast<bf16*>(taps + kHeadsPerCta * D * 3) + warp * 16 * OLD;
  const int n8 = R / 8;
  const int q0 = tid % n8, row0 = tid / n8;  // first 16-byte piece of this thread
  const int qstep = 256 % n8, rstep = 256 / n8;
  auto issue_wu = [&](int h, int buf) {
    const bf16* Wu = static_cast<const bf16*>(p.Wu) + static_cast<size_t>(h) * D * R;
    int q = q0, row = row0;
    while (row < D) {
      cp16_zfill(wub + (buf * D + row) * LD + 8 * q, Wu + static_cast<size_t>(row) * R + 8 * q,
                 true);
      q += qstep;
      row += rstep;
      if (q >= n8) {
        q -= n8;
        ++row;
      }
    }
    cp_commit();
  };
  {
    const bf16* low = static_cast<const bf16*>(p.low);
    int q = q0, lr = row0;
    while (lr < kLowRows) {
      const int grow = r0 - 16 + lr;
      const bool ok = grow >= 0 && grow < BT;
      cp16_zfill(lowb + lr * LD + 8 * q, low + static_cast<size_t>(ok ? grow : 0) * R + 8 * q, ok);
      q += qstep;
      lr += rstep;
      if (q >= n8) {
        q -= n8;
        ++lr;
      }
    }
    issue_wu(h0, 0);
    for (int x = tid; x < (h1 - h0) * D * 3; x += blockDim.x) {
      const int hh = x / (D * 3), r = x % (D * 3);  // source [h][c][k] -> [h][k][c]
      taps[hh * 3 * D + (r % 3) * D + r / 3] = p.cw[static_cast<size_t>(h0) * D * 3 + x];
    }
  }
  // the two rows this lane holds: local rows 16 w + g (A) and 16 w + g + 8 (B)
  const int growA = r0 - 16 + warp * 16 + g, growB = growA + 8;
  const int tA = growA >= 0 ? growA % p.T : 0;
  const int tB = growB >= 0 ? growB % p.T : 0;
  const float m1A = tA >= 1 ? 1.f : 0.f, m2A = tA >= 2 ? 1.f : 0.f;
  const float m1B = tB >= 1 ? 1.f : 0.f, m2B = tB >= 2 ? 1.f : 0.f;
  const unsigned full = 0xffffffffu;
  // rows this lane stores from the staging tile, as b * H * T + t (-1: none)
  constexpr int kStoreIters = 16 / (32 / (D / 8));
  int rowidx[kStoreIters];
#pragma unroll
  for (int k = 0; k < kStoreIters; ++k) {
    const int grow = r0 - 16 + warp * 16 + k * (32 / (D / 8)) + lane / (D / 8);
    rowidx[k] = (grow >= 0 && grow < BT) ? (grow / p.T) * p.H * p.T + grow % p.T : -1;
  }
  for (int h = h0; h < h1; ++h) {
    cp_wait<0>();
    __syncthreads();  // low, Wu_h and the taps landed; the halo is free again
    if (h + 1 < h1) issue_wu(h + 1, (h + 1 - h0) & 1);
    const bf16* wu = wub + ((h - h0) & 1) * D * LD;
    float acc[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
#pragma unroll
      for (int f = 0; f < 4; ++f) acc[n][f] = 0.f;
    for (int ks = 0; ks < R / 16; ++ks) {
      uint32_t a[4];
      ldsm_a(a, lowb, LD, warp * 16, ks * 16, lane);
#pragma unroll
      for (int n = 0; n < D / 8; n += 2) {
        uint32_t b[4];
        ldsm_b2(b, wu, LD, n * 8, ks * 16, lane);
        mma_bf16_16816(acc[n], a, b[0], b[1]);
        mma_bf16_16816(acc[n + 1], a, b[2], b[3]);
      }
    }
    // rows 14 and 15 of this warp's tile (lanes g = 6, 7, second half)
    if (g >= 6) {
#pragma unroll
      for (int n = 0; n < D / 8; ++n)
        *reinterpret_cast<float2*>(halo + (warp * 2 + g - 6) * D + n * 8 + 2 * t4) =
            make_float2(acc[n][2], acc[n][3]);
    }
    __syncthreads();
    const float* tp = taps + (h - h0) * D * 3;
    const float* prev = halo + (warp > 0 ? warp - 1 : 0) * 2 * D;  // rows 14, 15 before us
    float ssA = 0.f, ssB = 0.f;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const int c = n * 8 + 2 * t4;
      float up4[4], up8[4], r7[2], r6[2];
#pragma unroll
      for (int f = 0; f < 4; ++f) {
        up4[f] = __shfl_up_sync(full, acc[n][f], 4);
        up8[f] = __shfl_up_sync(full, acc[n][f], 8);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        r7[j] = __shfl_sync(full, acc[n][j], 28 + t4);
        r6[j] = __shfl_sync(full, acc[n][j], 24 + t4);
      }
      const float2 p14 = *reinterpret_cast<const float2*>(prev + c);
      const float2 p15 = *reinterpret_cast<const float2*>(prev + D + c);
      const float h14[2] = {p14.x, p14.y}, h15[2] = {p15.x, p15.y};
      const float2 k0 = *reinterpret_cast<const float2*>(tp + c);
      const float2 k1 = *reinterpret_cast<const float2*>(tp + D + c);
      const float2 k2 = *reinterpret_cast<const float2*>(tp + 2 * D + c);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float w0 = j ? k0.y : k0.x, w1 = j ? k1.y : k1.x, w2 = j ? k2.y : k2.x;
        // row A = g: r-1 = g-1 (or row 15 before), r-2 = g-2 (or rows 15 / 14 before)
        const float a1 = g >= 1 ? up4[j] : h15[j];
        const float a2 = g >= 2 ? up8[j] : (g == 1 ? h15[j] : h14[j]);
        // row B = g + 8: r-1 = g+7 (row 7 of the first half when g = 0)
        const float b1 = g >= 1 ? up4[2 + j] : r7[j];
        const float b2 = g >= 2 ? up8[2 + j] : (g == 1 ? r7[j] : r6[j]);
        const float zA = fmaf(w2, acc[n][j], fmaf(w1, m1A * a1, w0 * m2A * a2));
        const float zB = fmaf(w2, acc[n][2 + j], fmaf(w1, m1B * b1, w0 * m2B * b2));
        acc[n][j] = zA;
        acc[n][2 + j] = zB;
        ssA = fmaf(zA, zA, ssA);
        ssB = fmaf(zB, zB, ssB);
      }
    }
    ssA += __shfl_xor_sync(full, ssA, 1);
    ssA += __shfl_xor_sync(full, ssA, 2);
    ssB += __shfl_xor_sync(full, ssB, 1);
    ssB += __shfl_xor_sync(full, ssB, 2);
    const float invA = 1.f / fmaxf(sqrtf(ssA), 1e-12f), invB = 1.f / fmaxf(sqrtf(ssB), 1e-12f);
    // normalized rows through the warp's staging tile, then 16-byte stores
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      *reinterpret_cast<__nv_bfloat162*>(stage + g * OLD + n * 8 + 2 * t4) =
          __floats2bfloat162_rn(acc[n][0] * invA, acc[n][1] * invA);
      *reinterpret_cast<__nv_bfloat162*>(stage + (g + 8) * OLD + n * 8 + 2 * t4) =
          __floats2bfloat162_rn(acc[n][2] * invB, acc[n][3] * invB);
    }
    __syncwarp();
    if (warp > 0) {
      constexpr int CH = D / 8;        // 16-byte chunks per row
      constexpr int RPI = 32 / CH;     // rows per store instruction
      bf16* outp = static_cast<bf16*>(p.w);
#pragma unroll
      for (int k = 0; k < 16 / RPI; ++k) {
        const int rr = k * RPI + lane / CH, ch = lane % CH;
        if (rowidx[k] >= 0) {
          *reinterpret_cast<uint4*>(outp + (static_cast<size_t>(rowidx[k]) + static_cast<size_t>(h) * p.T) * D + ch * 8) =
              *reinterpret_cast<const uint4*>(stage + rr * OLD + ch * 8);
        }
      }
    }
    __syncwarp();
  }
}

// fp32 (small problems): one CTA per (112-token tile, head), SIMT.
template <int D>
__global__ void __launch_bounds__(256) producer_mix_f32_kernel(const ProdArgs p) {
  constexpr int PLD = D + 4, E = D / 32, kPre = kOut + 2;
  extern __shared__ __align__(16) float fsm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int BT = p.B * p.T, R = p.R;
  const int r0 = blockIdx.x * kOut, h = blockIdx.y;
  float* lowf = fsm;
  float* wuf = lowf + kPre * R;
  float* pre = wuf + D * R;
  const float* low = static_cast<const float*>(p.low);
  for (int x = tid; x < kPre * R; x += blockDim.x) {
    const int pr = x / R, r = x % R, grow = r0 - 2 + pr;
    lowf[x] = (grow >= 0 && grow < BT) ? low[static_cast<size_t>(grow) * R + r] : 0.f;
  }
  const float* Wu = static_cast<const float*>(p.Wu) + static_cast<size_t>(h) * D * R;
  for (int x = tid; x < D * R; x += blockDim.x) wuf[x] = Wu[x];
  __syncthreads();
  for (int x = tid; x < kPre * D; x += blockDim.x) {
    const int pr = x / D, c = x % D;
    float sum = 0.f;
    for (int r = 0; r < R; ++r) sum = fmaf(lowf[pr * R + r], wuf[c * R + r], sum);
    pre[pr * PLD + c] = sum;
  }
  __syncthreads();
  for (int i = 0; i < kOut / 8; ++i) {
    const int lr = warp * (kOut / 8) + i, grow = r0 + lr;
    if (grow >= BT) break;
    const int t = grow % p.T, b = grow / p.T;
    float z[E];
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = lane * E + e;
      const float* tp = p.cw + (static_cast<size_t>(h) * D + c) * 3;
      float v = tp[2] * pre[(lr + 2) * PLD + c];
      if (t >= 1) v = fmaf(tp[1], pre[(lr + 1) * PLD + c], v);
      if (t >= 2) v = fmaf(tp[0], pre[lr * PLD + c], v);
      z[e] = v;
      ss = fmaf(v, v, ss);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = 1.f / fmaxf(sqrtf(ss), 1e-12f);
    float* out = static_cast<float*>(p.w) + ((static_cast<size_t>(b) * p.H + h) * p.T + t) * D +
                 lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = z[e] * inv;
  }
}

template <int D>
cudaError_t launch_mix(const ProdArgs& p, bool bf16_in, cudaStream_t st) {
  const int BT = p.B * p.T, tiles = (BT + kOut - 1) / kOut;
  cudaError_t e;
  if (bf16_in) {
    auto kern = producer_mix_bf16_kernel<D>;
    const int smem = mix_bf16_smem_bytes<D>(p.R);
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
        cudaSuccess)
      return e;
    kern<<<dim3(tiles, (p.H + kHeadsPerCta - 1) / kHeadsPerCta), 256, smem, st>>>(p);
  } else {
    auto kern = producer_mix_f32_kernel<D>;
    const int smem = ((kOut + 2) * p.R + D * p.R + (kOut + 2) * (D + 4)) * 4;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
        cudaSuccess)
      return e;
    kern<<<dim3(tiles, p.H), 256, smem, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

size_t producer_workspace_bytes(int B, int T, int R, int H, int d) {
  const size_t low = align_up(static_cast<size_t>(B) * T * R * sizeof(float), 256);  // fp32 at most
  return low + producer_fold_bytes(H, d);
}

cudaError_t launch_producer(const void* x, const void* Wd, const void* Wu, const float* cw,
                            const void* Ub, const float* bb, void* w, float* beta, void* ws,
                            int* status, int B, int T, int Dm, int H, int d, int R, bool bf16_in,
                            cudaStream_t st) {
  float* low = static_cast<float*>(ws);
  void* fold = static_cast<char*>(ws) + align_up(static_cast<size_t>(B) * T * R * sizeof(float), 256);
  const ProdArgs p{x, Wd, Wu, Ub, cw, bb, w, beta, low, B, T, Dm, H, R};
  const int BT = B * T;
  cudaError_t e;
  if (bf16_in) {
    if ((e = launch_producer_proj_tc(x, Wd, Ub, bb, low, beta, status, B, T, Dm, H, R, st)) !=
        cudaSuccess)
      return e;
  } else {
    const int smem = Dm * 4;
    if ((e = cudaFuncSetAttribute(producer_proj_f32_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
        cudaSuccess)
      return e;
    producer_proj_f32_kernel<<<BT, 128, smem, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (bf16_in && producer_mix_tc_supported(B, T, H, d, R))
    return launch_producer_mix_tc(low, Wu, cw, fold, w, status, B, T, H, d, st);
  return d == 128 ? launch_mix<128>(p, bf16_in, st) : launch_mix<64>(p, bf16_in, st);
}

}  // namespace pathattn
