// prep.cu -- chunk preparation for the blockwise PaTH forward pass.
//
// For every chunk of C tokens (rows w_t^T of W, D = diag(beta)), following
// "PaTH Attention: Position Encoding via Accumulating Householder
// Transformations" (discussion slides), frames "A triangular representation
// makes paths computable" and "Backup: fix orientation before implementing
// UT products":
//   U    = (I + strictLower(D W W^T))^{-1} D          (forward substitution)
//   UW   = U W,  TK = U strictLower(W K^T)
//   kr   = K - TK^T W                 keys carried through H_{j+1} .. H_last
//   ql   = Q - lower(Q W^T) UW        queries carried through H_i .. H_first
//   ngt  = -(W^T UW)^T                so crossing the chunk backwards is
//                                     q^T F^T = q^T + q^T ngt^T
//   sdt  = log2(e) * (scale * (lower(Q K^T) - lower(Q W^T) TK) + gate),
//          stored transposed ([j][i]) with -inf above the diagonal
// and, for PaTH-FoX (frame "FoX adds a separate mechanism for forgetting"),
//   lam2 = log2(e) * inclusive cumsum of log f  (gate_ij = lam_i - lam_j).
//
// All arithmetic is fp32 (inputs widened exactly).  These SIMT kernels serve
// fp32 inputs; bf16 inputs go to the fused tensor-core kernel (prep_tc.cu).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace pathattn {
namespace {

__device__ __forceinline__ float load_elem(const void* p, size_t i, bool bf16) {
  return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i])
              : static_cast<const float*>(p)[i];
}
__device__ __forceinline__ void store_elem(void* p, size_t i, float v, bool bf16) {
  if (bf16)
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  else
    static_cast<float*>(p)[i] = v;
}

// An input tensor [BH][T][d] seen per chunk: (ch, token-in-chunk, column).
struct InTensor {
  const void* p;
  int T, d, C, Np;
  bool bf16;
  __device__ float operator()(int ch, int tok, int col) const {
    const int bh = ch / Np, n = ch - bh * Np, t = n * C + tok;
    if (t >= T) return 0.f;  // padding token
    return load_elem(p, (static_cast<size_t>(bh) * T + t) * d + col, bf16);
  }
};

// A per-chunk fp32 scratch matrix [ch][R][Cc].
struct Mat {
  const float* p;
  int R, Cc;
  __device__ float operator()(int ch, int r, int c) const {
    return p[(static_cast<size_t>(ch) * R + r) * Cc + c];
  }
};

// GEMM operand adapters: X(ch, mn, k) either directly or transposed.
// kContigK tells the tile loader which index is contiguous in memory.
template <class X>
struct Dir {
  X x;
  static constexpr bool kContigK = true;
  __device__ float operator()(int ch, int mn, int k) const { return x(ch, mn, k); }
};
template <class X>
struct Tr {
  X x;
  static constexpr bool kContigK = false;
  __device__ float operator()(int ch, int mn, int k) const { return x(ch, k, mn); }
};

// Batched tiled GEMM on the CUDA cores: for every chunk ch,
//   acc(m, n) = sum_k A(ch, m, k) * B(ch, n, k),   then ep(ch, m, n, acc).
// 64x64 output tile per block, 256 threads, 4x4 outputs per thread.
constexpr int kTile = 64, kKStep = 16;

template <class LA, class LB, class EP>
__global__ void __launch_bounds__(256) batched_gemm_kernel(int M, int N, int K, int tilesM,
                                                           int tilesN, LA la, LB lb, EP ep) {
  __shared__ float sA[kKStep][kTile + 4];
  __shared__ float sB[kKStep][kTile + 4];
  const int per_ch = tilesM * tilesN;
  const int ch = blockIdx.x / per_ch;
  const int rem = blockIdx.x - ch * per_ch;
  const int m0 = (rem / tilesN) * kTile, n0 = (rem % tilesN) * kTile;
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < K; k0 += kKStep) {
    for (int e = tid; e < kTile * kKStep; e += 256) {
      int mm, kk;
      if (LA::kContigK) { mm = e / kKStep; kk = e % kKStep; } else { kk = e / kTile; mm = e % kTile; }
      const int m = m0 + mm, k = k0 + kk;
      sA[kk][mm] = (m < M && k < K) ? la(ch, m, k) : 0.f;
      int nn, kb;
      if (LB::kContigK) { nn = e / kKStep; kb = e % kKStep; } else { kb = e / kTile; nn = e % kTile; }
      const int n = n0 + nn, kq = k0 + kb;
      sB[kb][nn] = (n < N && kq < K) ? lb(ch, n, kq) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kKStep; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = sA[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = sB[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
      if (m < M && n < N) ep(ch, m, n, acc[i][j]);
    }
}

template <class LA, class LB, class EP>
cudaError_t run_gemm(int nch, int M, int N, int K, LA la, LB lb, EP ep, cudaStream_t st) {
  const int tm = (M + kTile - 1) / kTile, tn = (N + kTile - 1) / kTile;
  const long long blocks = static_cast<long long>(nch) * tm * tn;
  batched_gemm_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(M, N, K, tm, tn, la, lb, ep);
  return cudaGetLastError();
}

// ------------------------------------------------------------ epilogues
struct BetaOf {
  const float* beta;
  int T, C, Np;
  __device__ float operator()(int ch, int tok) const {
    const int bh = ch / Np, n = ch - bh * Np, t = n * C + tok;
    return t < T ? beta[static_cast<size_t>(bh) * T + t] : 0.f;
  }
};

// strictLower(diag(beta) W W^T)
struct EpGramL {
  float* out;
  int C;
  BetaOf beta;
  __device__ void operator()(int ch, int i, int j, float acc) const {
    out[(static_cast<size_t>(ch) * C + i) * C + j] = j < i ? acc * beta(ch, i) : 0.f;
  }
};

// masked square store: keep j < i (strict) or j <= i
struct EpMasked {
  float* out;
  int C;
  bool strict;
  __device__ void operator()(int ch, int i, int j, float acc) const {
    const bool keep = strict ? (j < i) : (j <= i);
    out[(static_cast<size_t>(ch) * C + i) * C + j] = keep ? acc : 0.f;
  }
};

struct EpStoreF32 {
  float* out;
  int R, Cc;
  __device__ void operator()(int ch, int r, int c, float acc) const {
    out[(static_cast<size_t>(ch) * R + r) * Cc + c] = acc;
  }
};

// out = base(ch, r, c) - acc, stored as elem (bf16 or f32)
struct EpBaseMinus {
  void* out;
  bool out_bf16;
  int R, Cc;
  InTensor base;
  __device__ void operator()(int ch, int r, int c, float acc) const {
    store_elem(out, (static_cast<size_t>(ch) * R + r) * Cc + c, base(ch, r, c) - acc, out_bf16);
  }
};

struct EpNeg {
  void* out;
  bool out_bf16;
  int R, Cc;
  __device__ void operator()(int ch, int r, int c, float acc) const {
    store_elem(out, (static_cast<size_t>(ch) * R + r) * Cc + c, -acc, out_bf16);
  }
};

// Intra-chunk logits, log2 domain, transposed, masked.
struct EpDiag {
  float* sdt;
  const float* aqk;
  const float* lam2;  // may be null
  int C, Np, Tp;
  float scale_log2e;
  __device__ void operator()(int ch, int i, int j, float acc) const {
    float v = -INFINITY;
    if (j <= i) {
      v = (aqk[(static_cast<size_t>(ch) * C + i) * C + j] - acc) * scale_log2e;
      if (lam2) {
        const int bh = ch / Np, n = ch - bh * Np;
        const float* lg = lam2 + static_cast<size_t>(bh) * Tp + n * C;
        v += lg[i] - lg[j];
      }
    }
    sdt[(static_cast<size_t>(ch) * C + j) * C + i] = v;
  }
};

// ------------------------------------------------------------ triangular solve
// In place: lmat holds L = strictLower(D W W^T) of each chunk on entry and
// U = (I + L)^{-1} D on exit.  One block per chunk, thread j owns column j of
// X = (I + L)^{-1}:  x_jj = 1,  x_ij = -sum_{k=j}^{i-1} L_ik x_kj  (i > j).
__global__ void tri_solve_kernel(float* lmat, const float* beta, int C, int T, int Np) {
  extern __shared__ float sm[];
  float* sL = sm;                    // [C][C]
  float* sX = sm + C * C;            // [C][C]
  const int ch = blockIdx.x, j = threadIdx.x;
  float* Lg = lmat + static_cast<size_t>(ch) * C * C;
  for (int e = j; e < C * C; e += blockDim.x) sL[e] = Lg[e];
  __syncthreads();
  for (int i = 0; i < C; ++i) {
    float x;
    if (i < j) {
      x = 0.f;
    } else if (i == j) {
      x = 1.f;
    } else {
      const float* Li = sL + i * C;
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
      int k = j;
      for (; k + 3 < i; k += 4) {
        s0 = fmaf(Li[k], sX[k * C + j], s0);
        s1 = fmaf(Li[k + 1], sX[(k + 1) * C + j], s1);
        s2 = fmaf(Li[k + 2], sX[(k + 2) * C + j], s2);
        s3 = fmaf(Li[k + 3], sX[(k + 3) * C + j], s3);
      }
      for (; k < i; ++k) s0 = fmaf(Li[k], sX[k * C + j], s0);
      x = -((s0 + s1) + (s2 + s3));
    }
    sX[i * C + j] = x;
  }
  // U = X diag(beta): column j scaled by beta_j
  const int bh = ch / Np, n = ch - bh * Np, t = n * C + j;
  const float bj = t < T ? beta[static_cast<size_t>(bh) * T + t] : 0.f;
  for (int i = 0; i < C; ++i) Lg[i * C + j] = sX[i * C + j] * bj;
}

// ------------------------------------------------------------ gate prefix sum
// out[bh * out_stride + t] = mult * sum_{s<=t} logf[bh][s] for t < n_out;
// tokens at or past T (chunk padding) add 0.  Accumulated in fp64.
__global__ void gate_cumsum_kernel(const float* logf, float* out_base, int T, int Tp,
                                   size_t out_stride, double mult) {
  __shared__ double warp_tot[32];
  const int bh = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
  const int seg = (Tp + nt - 1) / nt;
  const int t0 = tid * seg;
  const float* lf = logf + static_cast<size_t>(bh) * T;
  double local = 0.0;
  for (int t = t0; t < t0 + seg && t < Tp; ++t) local += t < T ? static_cast<double>(lf[t]) : 0.0;
  // inclusive scan of per-thread totals across the block
  const int lane = tid & 31, wid = tid >> 5;
  double inc = local;
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_tot[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    double v = lane < (nt >> 5) ? warp_tot[lane] : 0.0;
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    warp_tot[lane] = v;
  }
  __syncthreads();
  double run = (inc - local) + (wid > 0 ? warp_tot[wid - 1] : 0.0);
  float* out = out_base + static_cast<size_t>(bh) * out_stride;
  for (int t = t0; t < t0 + seg && t < Tp; ++t) {
    run += t < T ? static_cast<double>(lf[t]) : 0.0;
    out[t] = static_cast<float>(run * mult);
  }
}

}  // namespace

cudaError_t launch_gate_prefix(const float* logf, float* out, int BH, int T, int n_out,
                               size_t out_stride, double mult, cudaStream_t st) {
  gate_cumsum_kernel<<<BH, 1024, 0, st>>>(logf, out, T, n_out, out_stride, mult);
  return cudaGetLastError();
}

cudaError_t launch_prep(const Geom& g, const Inputs& in, const Workspace& ws, int* dev_status,
                        cudaStream_t st, int* launches) {
  const int C = g.C, d = g.d, nch = g.nch;
  cudaError_t e;
  int n = 0;
  if (g.gate) {
    if ((e = launch_gate_prefix(in.logf, ws.lam2, g.BH, g.T, g.Tp, static_cast<size_t>(g.Tp),
                                1.4426950408889634, st)) != cudaSuccess)
      return e;
    ++n;
  }
  if (g.bf16) {
    e = launch_prep_tc(g, in, ws, dev_status, st);
    if (e != cudaSuccess) return e;
    if (launches) *launches = n + 1;
    return cudaSuccess;
  }
  const InTensor Q{in.q, g.T, d, C, g.Np, g.bf16}, K{in.k, g.T, d, C, g.Np, g.bf16},
      W{in.w, g.T, d, C, g.Np, g.bf16};
  const BetaOf beta{in.beta, g.T, C, g.Np};
  // Gram blocks of the chunk
  if ((e = run_gemm(nch, C, C, d, Dir<InTensor>{W}, Dir<InTensor>{W}, EpGramL{ws.lmat, C, beta}, st))) return e;
  if ((e = run_gemm(nch, C, C, d, Dir<InTensor>{W}, Dir<InTensor>{K}, EpMasked{ws.awk, C, true}, st))) return e;
  if ((e = run_gemm(nch, C, C, d, Dir<InTensor>{Q}, Dir<InTensor>{W}, EpMasked{ws.aqw, C, false}, st))) return e;
  if ((e = run_gemm(nch, C, C, d, Dir<InTensor>{Q}, Dir<InTensor>{K}, EpMasked{ws.aqk, C, false}, st))) return e;
  n += 4;
  // U = (I + L)^{-1} D
  {
    const size_t smem = static_cast<size_t>(2) * C * C * sizeof(float);
    if ((e = cudaFuncSetAttribute(tri_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem))))
      return e;
    tri_solve_kernel<<<nch, C, smem, st>>>(ws.lmat, in.beta, C, g.T, g.Np);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ++n;
  }
  const Mat U{ws.lmat, C, C}, AWK{ws.awk, C, C}, AQW{ws.aqw, C, C}, TK{ws.tk, C, C},
      UW{ws.uw, C, d};
  // UW = U W;  TK = U strictLower(W K^T)
  if ((e = run_gemm(nch, C, d, C, Dir<Mat>{U}, Tr<InTensor>{W}, EpStoreF32{ws.uw, C, d}, st))) return e;
  if ((e = run_gemm(nch, C, C, C, Dir<Mat>{U}, Tr<Mat>{AWK}, EpMasked{ws.tk, C, true}, st))) return e;
  // kr = K - TK^T W
  if ((e = run_gemm(nch, C, d, C, Tr<Mat>{TK}, Tr<InTensor>{W},
                    EpBaseMinus{ws.kr, g.bf16, C, d, K}, st)))
    return e;
  // ql = Q - lower(Q W^T) UW
  if ((e = run_gemm(nch, C, d, C, Dir<Mat>{AQW}, Tr<Mat>{UW}, EpBaseMinus{ws.ql, false, C, d, Q},
                    st)))
    return e;
  // ngt[n][k] = -(W^T UW)[k][n]
  if ((e = run_gemm(nch, d, d, C, Tr<Mat>{UW}, Tr<InTensor>{W}, EpNeg{ws.ngt, g.bf16, d, d}, st)))
    return e;
  // sdt = log2(e) (scale (lower(QK^T) - lower(QW^T) TK) + gate), transposed
  if ((e = run_gemm(nch, C, C, C, Dir<Mat>{AQW}, Tr<Mat>{TK},
                    EpDiag{ws.sdt, ws.aqk, g.gate ? ws.lam2 : nullptr, C, g.Np, g.Tp,
                           in.scale * kLog2e},
                    st)))
    return e;
  n += 6;
  if (launches) *launches = n;
  return cudaSuccess;
}

}  // namespace pathattn
