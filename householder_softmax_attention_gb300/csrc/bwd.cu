// bwd.cu -- backward pass of PaTH / PaTH-FoX attention (gradients of the
// outputs with respect to q, k, v, w, beta and log f).
//
// The pages time the forward and the backward together ("PaTH Attention:
// Position Encoding via Accumulating Householder Transformations", OpenReview
// discussion, section "Efficiency Evaluation") but spell out only the
// forward; the backward below is the derivative of the blockwise forward of
// the slides ("A triangular representation makes paths computable", "A
// right-to-left scan accumulates cross-block paths").  Per head, with chunks
// c < b, F_c = H_{first(c)} ... H_{last(c)} = I + ngt_c and
//   X_b^(b-1) = Ql_b,   X_b^(c-1) = X_b^(c) F_c^T        (query b crossing c)
//   S_bc = scale X_b^(c) Kr_c^T + gate,   S_bb = scale Adiag_b + gate.
// With dS = P (dP - D), D_i = dO_i . O_i - dlse_i:
//   dV_c  = sum_{b>=c} P_bc^T dO_b
//   dKr_c = scale sum_{b>c} dS_bc^T X_b^(c)
//   G_b^(c) = scale dS_bc Kr_c + G_b^(c-1) F_c  (c = 0 .. b-1),  dQl_b = G_b^(b-1)
//   dF_c  = sum_{b>c} G_b^(c-1)^T X_b^(c)
//   dAdiag_b = scale lower(dS_bb)
// and the chunk factors (UT transform) are differentiated chunk by chunk.
//
// Kernels (all fp32 arithmetic on the CUDA cores):
//   rowdot        D_i, and lse in the log2 domain
//   query walk    one warp per query row: walks X down (c = b-1 .. 0), storing
//                 X_b^(c); walks back up accumulating G, storing G_b^(c-1);
//                 writes dQl.  X and G are stored per (b, c) pair.
//   key pass      one warp per key row: the diagonal chunk from the prepared
//                 intra-chunk logits, then every later query chunk from the
//                 stored X: dV, dKr, lower(dS_cc), column sums of dS
//   dF            dF_c = sum_b G^T X over the stored pairs
//   chunk pass    batched GEMMs through the UT factors to dQ, dK, dW, dbeta
//   gate          dlog f_t = sum_{s >= t} (rowsum_s dS - colsum_s dS)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <initializer_list>
#include <type_traits>

#include "common.cuh"
#include "prep_solve.cuh"

namespace pathattn {
namespace {

using bf16 = __nv_bfloat16;

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const bf16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float x) { *p = x; }
__device__ __forceinline__ void stf(bf16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ uint32_t pack_bf16_pair(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ size_t pair_index(int b, int c) {
  return static_cast<size_t>(b) * (b - 1) / 2 + c;
}

constexpr int kRowWarps = 8;

// ------------------------------------------------------------------- rowdot
template <typename ET, int D>
__global__ void __launch_bounds__(kRowWarps * 32) bwd_rowdot_kernel(BwdParams p) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bh = blockIdx.y, t = blockIdx.x * kRowWarps + warp;
  if (t >= p.Tp) return;
  const size_t r = static_cast<size_t>(bh) * p.Tp + t;
  if (t >= p.T) {
    if (lane == 0) {
      p.dvec[r] = 0.f;
      p.lse2[r] = 0.f;
    }
    return;
  }
  const size_t row = (static_cast<size_t>(bh) * p.T + t) * D;
  const ET* o = static_cast<const ET*>(p.out) + row;
  const ET* go = static_cast<const ET*>(p.dout) + row;
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) s = fmaf(ldf(o + lane + 32 * e), ldf(go + lane + 32 * e), s);
  s = warp_sum(s);
  if (lane == 0) {
    const size_t it = static_cast<size_t>(bh) * p.T + t;
    p.dvec[r] = s - (p.dlse ? p.dlse[it] : 0.f);
    p.lse2[r] = p.lse[it] * kLog2e;
  }
}

// --------------------------------------------------------------- query walk
template <typename ET, int D>
__global__ void __launch_bounds__(kRowWarps * 32) bwd_query_kernel(BwdParams p) {
  constexpr int E = D / 32;
  __shared__ float sz[kRowWarps][D];
  __shared__ float sg[kRowWarps][D];
  __shared__ float sdo[kRowWarps][D];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bh = blockIdx.y, t = blockIdx.x * kRowWarps + warp;
  if (t >= p.Tp) return;  // warp-uniform; no block-wide barrier follows
  const int C = p.C, b = t / C, i = t - b * C;
  const size_t chb = static_cast<size_t>(bh) * p.Np + b;
  if (t >= p.T) {  // padded query: no gradient
#pragma unroll
    for (int e = 0; e < E; ++e) p.dql[(chb * C + i) * D + lane + 32 * e] = 0.f;
    return;
  }
  const ET* kr = static_cast<const ET*>(p.kr);
  const ET* ngt = static_cast<const ET*>(p.ngt);
  const ET* vv = static_cast<const ET*>(p.v) + static_cast<size_t>(bh) * p.T * D;
  ET* xs = static_cast<ET*>(p.xs) + static_cast<size_t>(bh) * p.npairs * C * D;
  ET* gs = static_cast<ET*>(p.gs) + static_cast<size_t>(bh) * p.npairs * C * D;
  float* z = sz[warp];
  float* gg = sg[warp];
  float* dor = sdo[warp];
  const ET* go = static_cast<const ET*>(p.dout) + (static_cast<size_t>(bh) * p.T + t) * D;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    dor[lane + 32 * e] = ldf(go + lane + 32 * e);
    z[lane + 32 * e] = p.ql[(chb * C + i) * D + lane + 32 * e];
  }
  __syncwarp();
  // walk down: store X_b^(c) as the element type, then cross chunk c
  for (int c = b - 1; c >= 0; --c) {
    ET* xr = xs + (pair_index(b, c) * C + i) * D;
#pragma unroll
    for (int e = 0; e < E; ++e) stf(xr + lane + 32 * e, z[lane + 32 * e]);
    if (c == 0) break;
    const ET* G = ngt + (static_cast<size_t>(bh) * p.Np + c) * D * D;
    float zn[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int n = lane + 32 * e;
      float acc = z[n];
      for (int kk = 0; kk < D; ++kk) acc = fmaf(z[kk], ldf(G + n * D + kk), acc);
      zn[e] = acc;
    }
    __syncwarp();
#pragma unroll
    for (int e = 0; e < E; ++e) z[lane + 32 * e] = zn[e];
    __syncwarp();
  }
  // walk up: G_b^(c) = scale dS_bc Kr_c + G_b^(c-1) F_c
  const size_t rt = static_cast<size_t>(bh) * p.Tp + t;
  const float lse2 = p.lse2[rt], Dv = p.dvec[rt];
  const float lrow = p.lam2 ? p.lam2[rt] : 0.f;
  // row sum of dS over the diagonal chunk (keys j <= i)
  float rs = 0.f;
  for (int j0 = 0; j0 <= i; j0 += 32) {
    const int j = j0 + lane;
    if (j <= i) {
      const float pr = exp2f(p.sdt[(chb * C + j) * C + i] - lse2);
      const ET* vj = vv + static_cast<size_t>(b * C + j) * D;
      float dp = 0.f;
      for (int m = 0; m < D; ++m) dp = fmaf(dor[m], ldf(vj + m), dp);
      rs += pr * (dp - Dv);
    }
  }
  float g[E];
#pragma unroll
  for (int e = 0; e < E; ++e) g[e] = 0.f;
  for (int c = 0; c < b; ++c) {
    const ET* xr = xs + (pair_index(b, c) * C + i) * D;
    __syncwarp();
#pragma unroll
    for (int e = 0; e < E; ++e) z[lane + 32 * e] = ldf(xr + lane + 32 * e);
    __syncwarp();
    const size_t chc = static_cast<size_t>(bh) * p.Np + c;
    float gn[E];
#pragma unroll
    for (int e = 0; e < E; ++e) gn[e] = 0.f;
    for (int j0 = 0; j0 < C; j0 += 32) {
      const int j = j0 + lane;
      const ET* kj = kr + (chc * C + j) * D;
      const ET* vj = vv + static_cast<size_t>(c * C + j) * D;
      float s = 0.f, dp = 0.f;
      for (int m = 0; m < D; ++m) {
        s = fmaf(z[m], ldf(kj + m), s);
        dp = fmaf(dor[m], ldf(vj + m), dp);
      }
      float s2 = s * p.scale_log2e;
      if (p.lam2) s2 += lrow - p.lam2[static_cast<size_t>(bh) * p.Tp + c * C + j];
      const float pr = exp2f(s2 - lse2);
      const float ds = pr * (dp - Dv);
      rs += ds;
      for (int u = 0; u < 32; ++u) {
        const float du = __shfl_sync(0xffffffffu, ds, u);
        const ET* ku = kr + (chc * C + j0 + u) * D;
#pragma unroll
        for (int e = 0; e < E; ++e) gn[e] = fmaf(du, ldf(ku + lane + 32 * e), gn[e]);
      }
    }
    if (c >= 1) {
      ET* gr = gs + (pair_index(b, c) * C + i) * D;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        stf(gr + lane + 32 * e, g[e]);
        gg[lane + 32 * e] = g[e];
      }
      __syncwarp();
      const ET* G = ngt + chc * D * D;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int n = lane + 32 * e;
        float acc = g[e];
        for (int kk = 0; kk < D; ++kk) acc = fmaf(gg[kk], ldf(G + kk * D + n), acc);
        g[e] = acc + p.scale * gn[e];
      }
      __syncwarp();
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) g[e] = p.scale * gn[e];
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) p.dql[(chb * C + i) * D + lane + 32 * e] = g[e];
  rs = warp_sum(rs);
  if (lane == 0) p.rowsum[rt] = rs;
}

// ----------------------------------------------------------------- key pass
template <typename ET, int D>
__global__ void __launch_bounds__(kRowWarps * 32) bwd_key_kernel(BwdParams p) {
  constexpr int E = D / 32;
  __shared__ float skr[kRowWarps][D];
  __shared__ float sv[kRowWarps][D];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bh = blockIdx.y, t = blockIdx.x * kRowWarps + warp;
  if (t >= p.Tp) return;
  const int C = p.C, c = t / C, jj = t - c * C;
  const size_t chc = static_cast<size_t>(bh) * p.Np + c;
  float* dkr = p.dkr + (chc * C + jj) * D;
  if (t >= p.T) {  // padded key: no gradient
#pragma unroll
    for (int e = 0; e < E; ++e) dkr[lane + 32 * e] = 0.f;
    return;
  }
  const ET* kr = static_cast<const ET*>(p.kr);
  const ET* vv = static_cast<const ET*>(p.v) + static_cast<size_t>(bh) * p.T * D;
  const ET* go = static_cast<const ET*>(p.dout) + static_cast<size_t>(bh) * p.T * D;
  const ET* xs = static_cast<const ET*>(p.xs) + static_cast<size_t>(bh) * p.npairs * C * D;
  float* kj = skr[warp];
  float* vj = sv[warp];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    kj[lane + 32 * e] = ldf(kr + (chc * C + jj) * D + lane + 32 * e);
    vj[lane + 32 * e] = ldf(vv + static_cast<size_t>(t) * D + lane + 32 * e);
  }
  __syncwarp();
  const float* lam2 = p.lam2 ? p.lam2 + static_cast<size_t>(bh) * p.Tp : nullptr;
  const float* lse2 = p.lse2 + static_cast<size_t>(bh) * p.Tp;
  const float* dvec = p.dvec + static_cast<size_t>(bh) * p.Tp;
  const float lcol = lam2 ? lam2[t] : 0.f;
  float dv[E], dk[E], cs = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) dv[e] = dk[e] = 0.f;
  // diagonal chunk: queries i >= jj
  for (int i0 = jj; i0 < C; i0 += 32) {
    const int i = i0 + lane, tq = c * C + i;
    const bool ok = i < C && tq < p.T;
    float pr = 0.f, ds = 0.f;
    if (ok) {
      const float s2 = p.sdt[(chc * C + jj) * C + i];
      pr = exp2f(s2 - lse2[tq]);
      const ET* gr = go + static_cast<size_t>(tq) * D;
      float dp = 0.f;
      for (int m = 0; m < D; ++m) dp = fmaf(ldf(gr + m), vj[m], dp);
      ds = pr * (dp - dvec[tq]);
      p.dad[(chc * C + i) * C + jj] = p.scale * ds;
    }
    cs += ds;
    const int n = min(32, min(C, p.T - c * C) - i0);
    for (int u = 0; u < n; ++u) {
      const float pu = __shfl_sync(0xffffffffu, pr, u);
      const ET* gr = go + static_cast<size_t>(c * C + i0 + u) * D;
#pragma unroll
      for (int e = 0; e < E; ++e) dv[e] = fmaf(pu, ldf(gr + lane + 32 * e), dv[e]);
    }
  }
  // later chunks from the stored walked queries
  for (int b = c + 1; b < p.Np; ++b) {
    const ET* xb = xs + pair_index(b, c) * C * D;
    for (int i0 = 0; i0 < C; i0 += 32) {
      if (b * C + i0 >= p.T) break;
      const int i = i0 + lane, tq = b * C + i;
      const bool ok = tq < p.T;
      float pr = 0.f, ds = 0.f;
      if (ok) {
        const ET* xr = xb + static_cast<size_t>(i) * D;
        const ET* gr = go + static_cast<size_t>(tq) * D;
        float s = 0.f, dp = 0.f;
        for (int m = 0; m < D; ++m) {
          s = fmaf(ldf(xr + m), kj[m], s);
          dp = fmaf(ldf(gr + m), vj[m], dp);
        }
        float s2 = s * p.scale_log2e;
        if (lam2) s2 += lam2[tq] - lcol;
        pr = exp2f(s2 - lse2[tq]);
        ds = pr * (dp - dvec[tq]);
      }
      cs += ds;
      const int n = min(32, p.T - (b * C + i0));
      for (int u = 0; u < n; ++u) {
        const float pu = __shfl_sync(0xffffffffu, pr, u);
        const float du = __shfl_sync(0xffffffffu, ds, u) * p.scale;
        const ET* gr = go + static_cast<size_t>(b * C + i0 + u) * D;
        const ET* xr = xb + static_cast<size_t>(i0 + u) * D;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          dv[e] = fmaf(pu, ldf(gr + lane + 32 * e), dv[e]);
          dk[e] = fmaf(du, ldf(xr + lane + 32 * e), dk[e]);
        }
      }
    }
  }
  cs = warp_sum(cs);
  ET* dvo = static_cast<ET*>(p.dv) + (static_cast<size_t>(bh) * p.T + t) * D;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    stf(dvo + lane + 32 * e, dv[e]);
    dkr[lane + 32 * e] = dk[e];
  }
  if (lane == 0) p.colsum[static_cast<size_t>(bh) * p.Tp + t] = cs;
}

// --------------------------------------------------------------------- dF
// dF_c = sum_{b>c} G_b^(c-1)^T X_b^(c); one block per chunk, thread-owned
// output entries, rows staged through shared memory 32 at a time.
template <typename ET, int D>
__global__ void __launch_bounds__(256) bwd_dF_kernel(BwdParams p) {
  constexpr int R = 32;
  constexpr int PER = D * D / 256;
  __shared__ float sgr[R][D];
  __shared__ float sxr[R][D];
  const int ch = blockIdx.x, bh = ch / p.Np, c = ch - bh * p.Np;
  const int C = p.C;
  const ET* xs = static_cast<const ET*>(p.xs) + static_cast<size_t>(bh) * p.npairs * C * D;
  const ET* gs = static_cast<const ET*>(p.gs) + static_cast<size_t>(bh) * p.npairs * C * D;
  float acc[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) acc[u] = 0.f;
  if (c >= 1) {
    for (int b = c + 1; b < p.Np; ++b) {
      const size_t base = pair_index(b, c) * C * D;
      const int rows = min(C, p.T - b * C);
      for (int r0 = 0; r0 < rows; r0 += R) {
        __syncthreads();
        for (int x = threadIdx.x; x < R * D; x += 256) {
          const int rr = x / D, cc = x % D;
          const bool ok = r0 + rr < rows;
          sgr[rr][cc] = ok ? ldf(gs + base + static_cast<size_t>(r0 + rr) * D + cc) : 0.f;
          sxr[rr][cc] = ok ? ldf(xs + base + static_cast<size_t>(r0 + rr) * D + cc) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < PER; ++u) {
          const int o = threadIdx.x + 256 * u, e = o / D, f = o % D;
          float a = acc[u];
          for (int rr = 0; rr < R; ++rr) a = fmaf(sgr[rr][e], sxr[rr][f], a);
          acc[u] = a;
        }
      }
    }
  }
  float* out = p.dF + static_cast<size_t>(ch) * D * D;
#pragma unroll
  for (int u = 0; u < PER; ++u) out[threadIdx.x + 256 * u] = acc[u];
}

// ---------------------------------------------------------- chunk helpers
// fp32 copies of w, k, q (zero rows past T) and beta (zero past T), per
// chunk.  Grid (groups of a head / 256, BH); a thread converts 8 consecutive
// elements of one row.
__device__ __forceinline__ void ld8(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void ld8(const bf16* p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[2 * e] = __uint_as_float(w[e] << 16);
    v[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
  }
}
__device__ __forceinline__ void st8(float* p, const float (&v)[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void st8(bf16* p, const float (&v)[8]) {
  uint4 u;
  u.x = pack_bf16_pair(v[0], v[1]);
  u.y = pack_bf16_pair(v[2], v[3]);
  u.z = pack_bf16_pair(v[4], v[5]);
  u.w = pack_bf16_pair(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = u;
}

template <typename ET>
__global__ void __launch_bounds__(256) bwd_chunk_inputs_kernel(BwdParams p, ChunkBufs cb) {
  const int g8 = p.d / 8;
  const int gi = blockIdx.x * 256 + threadIdx.x;
  if (gi >= p.Tp * g8) return;
  const int t = gi / g8, e = (gi - t * g8) * 8;
  for (int bh = blockIdx.y; bh < p.BH; bh += gridDim.y) {
  const size_t dst = (static_cast<size_t>(bh) * p.Tp + t) * p.d + e;
  float w[8], k[8], q[8];
  if (t < p.T) {
    const size_t src = (static_cast<size_t>(bh) * p.T + t) * p.d + e;
    ld8(static_cast<const ET*>(p.w) + src, w);
    ld8(static_cast<const ET*>(p.k) + src, k);
    ld8(static_cast<const ET*>(p.q) + src, q);
  } else {
#pragma unroll
    for (int u = 0; u < 8; ++u) w[u] = k[u] = q[u] = 0.f;
  }
  if constexpr (std::is_same<ET, bf16>::value) {   // exact bf16 copies
    st8(reinterpret_cast<bf16*>(cb.Wf) + dst, w);
    st8(reinterpret_cast<bf16*>(cb.Kf) + dst, k);
    st8(reinterpret_cast<bf16*>(cb.Qf) + dst, q);
  } else {
    st8(cb.Wf + dst, w);
    st8(cb.Kf + dst, k);
    st8(cb.Qf + dst, q);
  }
  if (e == 0)
    cb.bf[static_cast<size_t>(bh) * p.Tp + t] =
        t < p.T ? p.beta[static_cast<size_t>(bh) * p.T + t] : 0.f;
  }
}

// Batched C = mask(alpha op(A) op(B) + (acc ? C : 0)); 64 x 64 tiles, 4 x 4
// per thread.  op(A)(m, k) = tA ? A[k][m] : A[m][k]; op(B)(k, n) = tB ? B[n][k] : B[k][n].
// mask 0: none, 1: m >= n kept, 2: m > n kept (others written as 0).
struct GemmArg {
  const float* A;
  const float* B;
  float* Cm;
  long long sA, sB, sC;
  int lda, ldb, ldc, M, N, K, batch, mask;
  bool tA, tB, acc;
  float alpha;
};

__global__ void __launch_bounds__(256) gemm_batched_kernel(GemmArg g) {
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  for (int z = blockIdx.z; z < g.batch; z += gridDim.z) {
    const float* A = g.A + z * g.sA;
    const float* B = g.B + z * g.sB;
    float* Cm = g.Cm + z * g.sC;
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int s = 0; s < 4; ++s) acc[r][s] = 0.f;
    for (int k0 = 0; k0 < g.K; k0 += 16) {
      __syncthreads();
      for (int x = threadIdx.x; x < 1024; x += 256) {
        int mm, kk;
        if (g.tA) { kk = x / 64; mm = x % 64; } else { mm = x / 16; kk = x % 16; }
        As[kk][mm] = g.tA ? A[static_cast<size_t>(k0 + kk) * g.lda + m0 + mm]
                          : A[static_cast<size_t>(m0 + mm) * g.lda + k0 + kk];
        int nn, kb;
        if (g.tB) { nn = x / 16; kb = x % 16; } else { kb = x / 64; nn = x % 64; }
        Bs[kb][nn] = g.tB ? B[static_cast<size_t>(n0 + nn) * g.ldb + k0 + kb]
                          : B[static_cast<size_t>(k0 + kb) * g.ldb + n0 + nn];
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        float a[4], bv[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) a[r] = As[kk][ty * 4 + r];
#pragma unroll
        for (int s = 0; s < 4; ++s) bv[s] = Bs[kk][tx * 4 + s];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int s = 0; s < 4; ++s) acc[r][s] = fmaf(a[r], bv[s], acc[r][s]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int m = m0 + ty * 4 + r, n = n0 + tx * 4 + s;
        float* cp = Cm + static_cast<size_t>(m) * g.ldc + n;
        float v = g.alpha * acc[r][s] + (g.acc ? *cp : 0.f);
        if ((g.mask == 1 && m < n) || (g.mask == 2 && m <= n)) v = 0.f;
        *cp = v;
      }
  }
}

// Xi = (I + Lm)^{-1} for unit lower triangular I + Lm: forward substitution,
// one thread per column.
__global__ void bwd_tri_inv_kernel(const float* Lm, float* Xi, int C) {
  extern __shared__ float sl[];
  const int ch = blockIdx.x;
  const float* L = Lm + static_cast<size_t>(ch) * C * C;
  float* X = Xi + static_cast<size_t>(ch) * C * C;
  for (int x = threadIdx.x; x < C * C; x += blockDim.x) sl[x] = L[x];
  __syncthreads();
  float* col = sl + C * C;  // [C][C] solution, column j owned by thread j
  const int j = threadIdx.x;
  if (j < C) {
    for (int i = 0; i < C; ++i) {
      float v = (i == j) ? 1.f : 0.f;
      if (i > j)
        for (int k = j; k < i; ++k) v = fmaf(-sl[i * C + k], col[k * C + j], v);
      col[i * C + j] = v;
    }
  }
  __syncthreads();
  for (int x = threadIdx.x; x < C * C; x += blockDim.x) X[x] = col[x];
}

// The same inverse for C = 128 by recursive doubling (the forward
// preparation's solver, tensor cores for the 32- and 64-blocks); 256 threads.
constexpr int kSolveStride = 132;
// Also writes U = Xi diag(beta).
__global__ void __launch_bounds__(256) bwd_tri_inv128_kernel(const float* Lm, float* Xi,
                                                             const float* bf, float* Uo) {
  extern __shared__ float sl[];
  const size_t ch = blockIdx.x;
  const float* L = Lm + ch * 128 * 128;
  float* X = Xi + ch * 128 * 128;
  float* U = Uo + ch * 128 * 128;
  const float* be = bf + ch * 128;
  for (int x = threadIdx.x; x < 128 * 32; x += 256) {
    const int i = x >> 5, c4 = (x & 31) * 4;
    *reinterpret_cast<float4*>(sl + i * kSolveStride + c4) =
        *reinterpret_cast<const float4*>(L + i * 128 + c4);
  }
  __syncthreads();
  invert_unit_lower<kSolveStride>(sl, threadIdx.x);
  for (int x = threadIdx.x; x < 128 * 32; x += 256) {
    const int i = x >> 5, c4 = (x & 31) * 4;
    float4 v = *reinterpret_cast<const float4*>(sl + i * kSolveStride + c4);
    if (c4 > i) v.x = 0.f;
    if (c4 + 1 > i) v.y = 0.f;
    if (c4 + 2 > i) v.z = 0.f;
    if (c4 + 3 > i) v.w = 0.f;
    *reinterpret_cast<float4*>(X + i * 128 + c4) = v;
    const float4 b = *reinterpret_cast<const float4*>(be + c4);
    *reinterpret_cast<float4*>(U + i * 128 + c4) = make_float4(v.x * b.x, v.y * b.y, v.z * b.z, v.w * b.w);
  }
}

// Elementwise steps of the chunk pass, one block per chunk, 4 columns per
// thread and step.
//  op 0: Lm  = strictLower(beta_i GWW_ij)
//  op 1: U   = Xi diag(beta)  (and dXi = dU diag(beta) when `in` is dU)
//  op 2: BL  = diag(beta) dLm
__global__ void __launch_bounds__(256) bwd_chunk_elem_kernel(const float* in, float* out,
                                                             const float* bf, int C, int op) {
  const int ch = blockIdx.x;
  const float4* a = reinterpret_cast<const float4*>(in + static_cast<size_t>(ch) * C * C);
  float4* o = reinterpret_cast<float4*>(out + static_cast<size_t>(ch) * C * C);
  const float* be = bf + static_cast<size_t>(ch) * C;
  const int c4 = C / 4;
  for (int x = threadIdx.x; x < C * c4; x += blockDim.x) {
    const int i = x / c4, j = (x - i * c4) * 4;
    float4 v = a[x];
    if (op == 0) {
      const float bi = be[i];
      v.x = i > j ? bi * v.x : 0.f;
      v.y = i > j + 1 ? bi * v.y : 0.f;
      v.z = i > j + 2 ? bi * v.z : 0.f;
      v.w = i > j + 3 ? bi * v.w : 0.f;
    } else if (op == 1) {
      const float4 bj = *reinterpret_cast<const float4*>(be + j);
      v.x *= bj.x; v.y *= bj.y; v.z *= bj.z; v.w *= bj.w;
    } else {
      const float bi = be[i];
      v.x *= bi; v.y *= bi; v.z *= bi; v.w *= bi;
    }
    o[x] = v;
  }
}

// dbeta_j = sum_i Xi_ij dU_ij + sum_m dLm_jm GWW_jm (Xi lower, dLm strictly
// lower triangular); one block of 256 per chunk: the row sums by a warp per
// row, the column sums by all threads.
__global__ void __launch_bounds__(256) bwd_dbeta_kernel(const float* Xi, const float* dU,
                                                        const float* dLm, const float* GWW,
                                                        float* dbf, int C) {
  __shared__ float rows[128], cols[256];
  const int ch = blockIdx.x, tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const size_t o = static_cast<size_t>(ch) * C * C;
  for (int j = warp; j < C; j += 8) {
    float s = 0.f;
    for (int m = lane; m < j; m += 32) s = fmaf(dLm[o + j * C + m], GWW[o + j * C + m], s);
    s = warp_sum(s);
    if (lane == 0) rows[j] = s;
  }
  // column sums (Xi is lower triangular: rows r >= c): 256 / C threads per
  // column, each over every (256 / C)-th row, with independent partial sums
  // so that several loads are in flight
  const int nh = 256 / C, c = tid % C, h = tid / C;
  float a[4] = {0.f, 0.f, 0.f, 0.f};
  for (int i = h; i < C; i += 4 * nh) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = i + u * nh;
      if (r < C && r >= c) a[u] = fmaf(Xi[o + r * C + c], dU[o + r * C + c], a[u]);
    }
  }
  cols[tid] = (a[0] + a[1]) + (a[2] + a[3]);
  __syncthreads();
  if (tid < C) {
    float s = rows[tid];
    for (int q = 0; q < nh; ++q) s += cols[q * C + tid];
    dbf[static_cast<size_t>(ch) * C + tid] = s;
  }
}

// dq, dk, dw (input dtype) and dbeta from the chunk-pass buffers; grid as the
// inputs kernel.
template <typename ET>
__global__ void __launch_bounds__(256) bwd_chunk_outputs_kernel(BwdParams p, ChunkBufs cb) {
  const int g8 = p.d / 8;
  const int gi = blockIdx.x * 256 + threadIdx.x;
  if (gi >= p.T * g8) return;
  const int t = gi / g8, e = (gi - t * g8) * 8;
  for (int bh = blockIdx.y; bh < p.BH; bh += gridDim.y) {
  const size_t src = (static_cast<size_t>(bh) * p.Tp + t) * p.d + e;
  const size_t dst = (static_cast<size_t>(bh) * p.T + t) * p.d + e;
  float v[8];
  ld8(cb.dQf + src, v);
  st8(static_cast<ET*>(p.dq) + dst, v);
  ld8(cb.dKf + src, v);
  st8(static_cast<ET*>(p.dk) + dst, v);
  ld8(cb.dWf + src, v);
  st8(static_cast<ET*>(p.dw) + dst, v);
  if (e == 0)
    p.dbeta[static_cast<size_t>(bh) * p.T + t] = cb.dbf[static_cast<size_t>(bh) * p.Tp + t];
  }
}

// dlog f_t = sum_{s >= t, s < T} (rowsum_s - colsum_s) of dS (the row sum
// is dlse_s in exact arithmetic; taking both sums from the same dS keeps
// dlog f_0 = 0, as it is exactly): one block per head,
// tiles of 1024 walked from the end with a carried suffix sum.
__global__ void __launch_bounds__(1024) bwd_gate_kernel(BwdParams p) {
  __shared__ float wsum[32];
  __shared__ float carry_s;
  const int bh = blockIdx.x, lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  if (threadIdx.x == 0) carry_s = 0.f;
  __syncthreads();
  for (int end = p.T; end > 0; end -= 1024) {
    // position end - 1 - threadIdx.x (reverse order, so a prefix scan is a suffix scan)
    const int t = end - 1 - threadIdx.x;
    float v = 0.f;
    if (t >= 0) {
      const size_t r = static_cast<size_t>(bh) * p.Tp + t;
      v = p.rowsum[r] - p.colsum[r];
    }
    float x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      float w = wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      wsum[lane] = w;
    }
    __syncthreads();
    const float carry = carry_s;
    const float incl = x + (warp > 0 ? wsum[warp - 1] : 0.f) + carry;
    if (t >= 0) p.dlogf[static_cast<size_t>(bh) * p.T + t] = incl;
    __syncthreads();
    if (threadIdx.x == 0) carry_s = carry + wsum[31];
    __syncthreads();
  }
}

// Where the chunk-pass GEMMs run: bf16 inputs take the tensor-core kernel
// (fp32 operands as bf16 hi + lo), fp32 inputs the fp32 SIMT kernel.
struct GemmCtx {
  cudaStream_t st;
  bool tc;
  int* status;
  // operands held as bf16 copies (exact inputs), read as such by the
  // tensor-core products; no other path accepts them
  const float* bf_ops[3] = {nullptr, nullptr, nullptr};
  bool is_bf(const float* x) const {
    return x && (x == bf_ops[0] || x == bf_ops[1] || x == bf_ops[2]);
  }
};

cudaError_t gemm(const GemmCtx& gx, int batch, int M, int N, int K, float alpha, const float* A,
                 int lda, long long sA, bool tA, const float* B, int ldb, long long sB, bool tB,
                 float* Cm, int ldc, long long sC, bool acc, int mask) {
  cudaStream_t st = gx.st;
  GemmArg g{A, B, Cm, sA, sB, sC, lda, ldb, ldc, M, N, K, batch, mask, tA, tB, acc, alpha};
  const dim3 grid(N / 64, M / 64, batch < 65535 ? batch : 65535);
  gemm_batched_kernel<<<grid, 256, 0, st>>>(g);
  return cudaGetLastError();
}

// One product alpha op(A) op(B) with K = the shared dimension.
struct Term {
  float alpha;
  const float* A;
  int lda;
  long long sA;
  bool tA;
  const float* B;
  int ldb;
  long long sB;
  bool tB;
  int K;
};

// C = mask(sum of the terms + add) over the batch; add may be null or C.  The
// tensor-core kernel does it in one launch; the fp32 path copies add into C
// and accumulates the terms one GEMM at a time.
// A second output C2 (scaled copy of C, see TcGemmN) is written by the
// tensor-core kernel's epilogue, else by the elementwise kernel afterwards
// (op 0: strictLower(diag(vec) C), 1: C diag(vec), 2: diag(vec) C).
struct Out2 {
  float* C2 = nullptr;
  const float* vec = nullptr;
  int op = 0;
};
cudaError_t mgemm(const GemmCtx& gx, int batch, int M, int N, std::initializer_list<Term> terms,
                  float* Cm, int ldc, long long sC, const float* add, int mask,
                  Out2 o2 = Out2{}) {
  if (gx.tc) {
    TcGemmN g{};
    g.nterms = 0;
    for (const Term& t : terms) {
      if (g.nterms == kMaxTerms) return cudaErrorInvalidValue;
      TcTerm tt{t.A, t.B, t.sA, t.sB, t.lda, t.ldb, t.K, t.tA, t.tB, t.alpha};
      tt.aBf = gx.is_bf(t.A);
      tt.bBf = gx.is_bf(t.B);
      if (tt.aBf && t.alpha != 1.f && t.alpha != -1.f) return cudaErrorInvalidValue;
      g.t[g.nterms++] = tt;
    }
    g.Cm = Cm;
    g.Add = add;
    g.sC = g.sAdd = sC;
    g.ldc = g.ldadd = ldc;
    g.M = M;
    g.N = N;
    g.batch = batch;
    g.mask = mask;
    g.status = gx.status;
    if (o2.C2) {
      g.C2 = o2.C2;
      g.vec = o2.vec;
      g.c2op = o2.op == 1 ? 2 : 1;           // C diag(vec): columns; else rows
      g.c2mask = o2.op == 0 ? 2 : 0;         // op 0 is strictly lower
    }
    if (gemm_tc_supported(g)) return launch_gemm_tc(g, gx.st);
  }
  for (const Term& t : terms)
    if (gx.is_bf(t.A) || gx.is_bf(t.B)) return cudaErrorInvalidValue;
  cudaError_t e;
  if (add && add != Cm &&
      (e = cudaMemcpyAsync(Cm, add, static_cast<size_t>(batch) * sC * sizeof(float),
                           cudaMemcpyDeviceToDevice, gx.st)) != cudaSuccess)
    return e;
  const GemmCtx simt{gx.st, false, gx.status};
  bool acc = add != nullptr;
  for (const Term& t : terms) {
    if ((e = gemm(simt, batch, M, N, t.K, t.alpha, t.A, t.lda, t.sA, t.tA, t.B, t.ldb, t.sB, t.tB,
                  Cm, ldc, sC, acc, mask)) != cudaSuccess)
      return e;
    acc = true;
  }
  if (o2.C2) {
    if (M != N || ldc != M || sC != static_cast<long long>(M) * M) return cudaErrorInvalidValue;
    bwd_chunk_elem_kernel<<<batch, 256, 0, gx.st>>>(Cm, o2.C2, o2.vec, M, o2.op);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

template <typename ET, int D>
cudaError_t launch_bwd_t(const BwdParams& p, const ChunkBufs& cb, cudaStream_t st) {
  const int C = p.C;
  const dim3 rows_tp((p.Tp + kRowWarps - 1) / kRowWarps, p.BH);
  bwd_rowdot_kernel<ET, D><<<rows_tp, kRowWarps * 32, 0, st>>>(p);
  bwd_mark(p.ev, kBwdEvXwalk, st);
  cudaError_t e;
  if (p.bf16) {
    // bf16: the chunk pairs on the tensor cores
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_bwd_pairs_tc(p, p.status, st)) != cudaSuccess) return e;
  } else {
    bwd_query_kernel<ET, D><<<rows_tp, kRowWarps * 32, 0, st>>>(p);
    e = cudaMemsetAsync(p.dad, 0, static_cast<size_t>(p.nch) * C * C * 4, st);
    if (e != cudaSuccess) return e;
    bwd_key_kernel<ET, D><<<rows_tp, kRowWarps * 32, 0, st>>>(p);
    bwd_dF_kernel<ET, D><<<p.nch, 256, 0, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    for (int i = kBwdEvKey; i <= kBwdEvDf; ++i) bwd_mark(p.ev, i, st);
  }
  bwd_mark(p.ev, kBwdEvChunk, st);
  // ---- chunk pass (fp32, batched over chunks)
  const int nch = p.nch;
  GemmCtx gx{st, p.bf16, p.status};
  const long long cc = static_cast<long long>(C) * C, cd = static_cast<long long>(C) * D,
                  dd = static_cast<long long>(D) * D;
  bwd_chunk_inputs_kernel<ET><<<dim3((p.Tp * (D / 8) + 255) / 256, p.BH < 65535 ? p.BH : 65535), 256, 0, st>>>(p, cb);
  // bf16 inputs: W, K, Q are bf16 copies (padded to Tp), exact operands of the
  // tensor-core products
  const float *W = cb.Wf, *K = cb.Kf, *Q = cb.Qf;
  if (p.bf16) {
    gx.bf_ops[0] = W;
    gx.bf_ops[1] = K;
    gx.bf_ops[2] = Q;
  }
  // Products of [C][C] (cc) and [C][D] (cd) per-chunk matrices; a Term lists
  // alpha, A, its leading dimension and batch stride, whether it is
  // transposed, the same for B, and the shared dimension.
  auto CC = [&](float al, const float* A, bool tA, const float* B, bool tB) {
    return Term{al, A, C, cc, tA, B, C, cc, tB, C};
  };
  auto CD_DC = [&](float al, const float* A, bool tA, const float* B, bool tB) {  // [C][D] x [D][C]
    return Term{al, A, D, cd, tA, B, D, cd, tB, D};
  };
  auto CC_CD = [&](float al, const float* A, bool tA, const float* B) {  // [C][C] x [C][D]
    return Term{al, A, C, cc, tA, B, D, cd, false, C};
  };
  // forward factors
  // GWW = W W^T, Lm = strictLower(diag(beta) GWW)
  if ((e = mgemm(gx, nch, C, C, {CD_DC(1.f, W, false, W, true)}, cb.GWW, C, cc, nullptr, 0,
                 Out2{cb.Lm, cb.bf, 0})))
    return e;
  if (C == 128) {
    const int smem = 128 * kSolveStride * static_cast<int>(sizeof(float));
    if ((e = cudaFuncSetAttribute(bwd_tri_inv128_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
      return e;
    bwd_tri_inv128_kernel<<<nch, 256, smem, st>>>(cb.Lm, cb.Xi, cb.bf, cb.U);
  } else {
    const int tri_smem = 2 * C * C * static_cast<int>(sizeof(float));
    if ((e = cudaFuncSetAttribute(bwd_tri_inv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  tri_smem)) != cudaSuccess)
      return e;
    bwd_tri_inv_kernel<<<nch, C, tri_smem, st>>>(cb.Lm, cb.Xi, C);
    bwd_chunk_elem_kernel<<<nch, 256, 0, st>>>(cb.Xi, cb.U, cb.bf, C, 1);
  }
  if ((e = mgemm(gx, nch, C, C, {CD_DC(1.f, W, false, K, true)}, cb.Nm, C, cc, nullptr, 2)) ||
      (e = mgemm(gx, nch, C, C, {CC(1.f, cb.U, false, cb.Nm, false)}, cb.TK, C, cc, nullptr, 0)) ||
      (e = mgemm(gx, nch, C, D, {CC_CD(1.f, cb.U, false, W)}, cb.UW, D, cd, nullptr, 0)) ||
      (e = mgemm(gx, nch, C, C, {CD_DC(1.f, Q, false, W, true)}, cb.Mm, C, cc, nullptr, 1)))
    return e;
  const float *dQl = p.dql, *dKr = p.dkr, *dF = p.dF, *dA = p.dad;
  // dM = lower(-dQl UW^T - dA TK^T)
  if ((e = mgemm(gx, nch, C, C, {CD_DC(-1.f, dQl, false, cb.UW, true), CC(-1.f, dA, false, cb.TK, true)},
                 cb.dM, C, cc, nullptr, 1)))
    return e;
  // dQ = dQl + dA K + dM W
  if ((e = mgemm(gx, nch, C, D, {CC_CD(1.f, dA, false, K), CC_CD(1.f, cb.dM, false, W)}, cb.dQf, D,
                 cd, dQl, 0)))
    return e;
  // dTK = -W dKr^T - M^T dA ; dUW = -M^T dQl
  if ((e = mgemm(gx, nch, C, C, {CD_DC(-1.f, W, false, dKr, true), CC(-1.f, cb.Mm, true, dA, false)},
                 cb.dTK, C, cc, nullptr, 0)) ||
      (e = mgemm(gx, nch, C, D, {CC_CD(-1.f, cb.Mm, true, dQl)}, cb.dUW, D, cd, nullptr, 0)))
    return e;
  // dN = strictLower(U^T dTK); dK = dKr + dA^T Q + dN^T W
  if ((e = mgemm(gx, nch, C, C, {CC(1.f, cb.U, true, cb.dTK, false)}, cb.dN, C, cc, nullptr, 2)) ||
      (e = mgemm(gx, nch, C, D, {CC_CD(1.f, dA, true, Q), CC_CD(1.f, cb.dN, true, W)}, cb.dKf, D, cd,
                 dKr, 0)))
    return e;
  // P1 = W dF, P2 = W dF^T  ([C][D] x [D][D])
  if ((e = mgemm(gx, nch, C, D, {Term{1.f, W, D, cd, false, dF, D, dd, false, D}}, cb.P1, D, cd,
                 nullptr, 0)) ||
      (e = mgemm(gx, nch, C, D, {Term{1.f, W, D, cd, false, dF, D, dd, true, D}}, cb.P2, D, cd,
                 nullptr, 0)))
    return e;
  // dU = -P2 W^T + dTK N^T + dUW W^T, dXi = dU diag(beta)
  if ((e = mgemm(gx, nch, C, C,
                 {CD_DC(-1.f, cb.P2, false, W, true), CC(1.f, cb.dTK, false, cb.Nm, true),
                  CD_DC(1.f, cb.dUW, false, W, true)},
                 cb.dU, C, cc, nullptr, 0, Out2{cb.dXi, cb.bf, 1})))
    return e;
  // T1 = Xi^T dXi; dLm = strictLower(-T1 Xi^T), BL = diag(beta) dLm
  if ((e = mgemm(gx, nch, C, C, {CC(1.f, cb.Xi, true, cb.dXi, false)}, cb.T1, C, cc, nullptr, 0)) ||
      (e = mgemm(gx, nch, C, C, {CC(-1.f, cb.T1, false, cb.Xi, true)}, cb.dLm, C, cc, nullptr, 2,
                 Out2{cb.BL, cb.bf, 2})))
    return e;
  bwd_dbeta_kernel<<<nch, 256, 0, st>>>(cb.Xi, cb.dU, cb.dLm, cb.GWW, cb.dbf, C);
  // dW = -TK dKr - U P1 - U^T P2 + dM^T Q + dN K + U^T dUW + BL W + BL^T W
  if ((e = mgemm(gx, nch, C, D,
                 {CC_CD(-1.f, cb.TK, false, dKr), CC_CD(-1.f, cb.U, false, cb.P1),
                  CC_CD(-1.f, cb.U, true, cb.P2), CC_CD(1.f, cb.dM, true, Q),
                  CC_CD(1.f, cb.dN, false, K), CC_CD(1.f, cb.U, true, cb.dUW),
                  CC_CD(1.f, cb.BL, false, W), CC_CD(1.f, cb.BL, true, W)},
                 cb.dWf, D, cd, nullptr, 0)))
    return e;
  bwd_chunk_outputs_kernel<ET><<<dim3((p.T * (D / 8) + 255) / 256, p.BH < 65535 ? p.BH : 65535), 256, 0, st>>>(p, cb);
  if (p.dlogf) bwd_gate_kernel<<<p.BH, 1024, 0, st>>>(p);
  bwd_mark(p.ev, kBwdEvEnd, st);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_layout(const Geom& g, char* base, BwdParams* p, ChunkBufs* cb) {
  const size_t es = g.bf16 ? 2 : 4;
  const size_t nch = static_cast<size_t>(g.nch), C = g.C, d = g.d;
  const size_t BH = g.BH, Tp = g.Tp;
  const size_t npairs = static_cast<size_t>(g.Np) * (g.Np - 1) / 2;
  size_t off = 0;
  auto take = [&](size_t bytes) -> char* {
    char* q = base ? base + off : nullptr;
    off = align_up(off + bytes, 256);
    return q;
  };
  BwdParams b{};
  b.dvec = reinterpret_cast<float*>(take(BH * Tp * 4));
  b.lse2 = reinterpret_cast<float*>(take(BH * Tp * 4));
  b.colsum = reinterpret_cast<float*>(take(BH * Tp * 4));
  b.rowsum = reinterpret_cast<float*>(take(BH * Tp * 4));
  b.xs = take(BH * npairs * C * d * es);
  b.gs = take(BH * npairs * C * d * es);
  b.ds = g.bf16 ? take(BH * npairs * C * C * 2) : nullptr;
  b.dql = reinterpret_cast<float*>(take(nch * C * d * 4));
  b.dkr = reinterpret_cast<float*>(take(nch * C * d * 4));
  b.dF = reinterpret_cast<float*>(take(nch * d * d * 4));
  b.dad = reinterpret_cast<float*>(take(nch * C * C * 4));
  ChunkBufs c{};
  float** cd_bufs[] = {&c.Wf, &c.Kf, &c.Qf, &c.UW, &c.dUW, &c.P1, &c.P2, &c.dQf, &c.dKf, &c.dWf};
  for (float** q : cd_bufs) *q = reinterpret_cast<float*>(take(nch * C * d * 4));
  float** cc_bufs[] = {&c.GWW, &c.Lm, &c.Xi, &c.U, &c.Nm, &c.TK, &c.Mm, &c.dM,
                       &c.dTK, &c.dN, &c.dU, &c.dXi, &c.T1, &c.dLm, &c.BL};
  for (float** q : cc_bufs) *q = reinterpret_cast<float*>(take(nch * C * C * 4));
  c.bf = reinterpret_cast<float*>(take(nch * C * 4));
  c.dbf = reinterpret_cast<float*>(take(nch * C * 4));
  b.npairs = npairs;
  if (p) *p = b;
  if (cb) *cb = c;
  return off;
}

cudaError_t launch_bwd(const BwdParams& p, const ChunkBufs& cb, cudaStream_t st) {
  if (p.bf16) {
    if (p.d == 64) return launch_bwd_t<bf16, 64>(p, cb, st);
    return launch_bwd_t<bf16, 128>(p, cb, st);
  }
  if (p.d == 64) return launch_bwd_t<float, 64>(p, cb, st);
  return launch_bwd_t<float, 128>(p, cb, st);
}

}  // namespace pathattn
