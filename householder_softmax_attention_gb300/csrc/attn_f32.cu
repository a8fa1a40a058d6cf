// attn_f32.cu -- PaTH forward scan in fp32 on the CUDA cores (dtype f32).
//
// One warp per query row i of chunk b ("PaTH Attention ..." slides, frame
// "A right-to-left scan accumulates cross-block paths"):
//   1. the diagonal chunk's logits come precomputed (sdt, log2 domain);
//   2. z = ql_i (q_i carried through H_i .. H_first of its own chunk);
//   3. for c = b-1 .. 0: logits z . kr_j for the keys of chunk c, online
//      softmax and value accumulation; then cross chunk c backwards,
//      z <- z + z ngt_c^T  (= z F_c^T).
// Every lane owns d/32 columns of the output row.
#include <cuda_runtime.h>

#include "common.cuh"

namespace pathattn {
namespace {

__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr int kWarpsPerBlock = 8;

template <int D>
struct RowState {
  static constexpr int E = D / 32;
  float o[E];
  float m, l;
  __device__ void init() {
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
    m = -INFINITY;
    l = 0.f;
  }
  // Fold in up to 32 keys: this lane's log2-domain logit s2 (−inf if the
  // lane holds no key), value rows vbase[(0..cnt) * D].
  __device__ void consume(float s2, const float* vbase, int cnt, int lane) {
    const float gmax = warp_max(s2);
    const float m_new = fmaxf(m, gmax);
    if (m_new == -INFINITY) return;
    const float alpha = exp2f(m - m_new);
    const float p = exp2f(s2 - m_new);
    l = l * alpha + warp_sum(p);
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] *= alpha;
    for (int jj = 0; jj < cnt; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      const float* vr = vbase + static_cast<size_t>(jj) * D;
#pragma unroll
      for (int e = 0; e < E; ++e) o[e] = fmaf(pj, vr[lane + 32 * e], o[e]);
    }
    m = m_new;
  }
};

template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) attn_f32_kernel(
    const float* __restrict__ v, float* __restrict__ out, float* __restrict__ lse,
    const float* __restrict__ kr, const float* __restrict__ ql, const float* __restrict__ ngt,
    const float* __restrict__ sdt, const float* __restrict__ lam2, int T, int C, int Np,
    float scale_log2e) {
  constexpr int E = D / 32;
  __shared__ float sz[kWarpsPerBlock][D];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bh = blockIdx.y;
  const int t = blockIdx.x * kWarpsPerBlock + warp;
  if (t >= T) return;  // warp-uniform; no block-wide barrier follows
  const int Tp = Np * C;
  const int b = t / C, i = t - b * C;
  float* z = sz[warp];
  const float* vbh = v + static_cast<size_t>(bh) * T * D;
  RowState<D> st;
  st.init();
  // 1. diagonal chunk
  const size_t chb = static_cast<size_t>(bh) * Np + b;
  for (int j0 = 0; j0 <= i; j0 += 32) {
    const int j = j0 + lane;
    const float s2 = j <= i ? sdt[(chb * C + j) * C + i] : -INFINITY;
    st.consume(s2, vbh + static_cast<size_t>(b * C + j0) * D, min(32, i + 1 - j0), lane);
  }
  // 2. running query
#pragma unroll
  for (int e = 0; e < E; ++e) z[lane + 32 * e] = ql[(chb * C + i) * D + lane + 32 * e];
  __syncwarp();
  const float lrow = lam2 ? lam2[static_cast<size_t>(bh) * Tp + t] : 0.f;
  // 3. earlier chunks, nearest first
  for (int c = b - 1; c >= 0; --c) {
    const size_t chc = static_cast<size_t>(bh) * Np + c;
    for (int j0 = 0; j0 < C; j0 += 32) {
      const int j = j0 + lane;
      const float* kj = kr + (chc * C + j) * D;
      float s = 0.f;
      for (int mm = 0; mm < D; ++mm) s = fmaf(z[mm], kj[mm], s);
      float s2 = s * scale_log2e;
      if (lam2) s2 += lrow - lam2[static_cast<size_t>(bh) * Tp + c * C + j];
      st.consume(s2, vbh + static_cast<size_t>(c * C + j0) * D, 32, lane);
    }
    if (c > 0) {
      const float* G = ngt + chc * D * D;
      float zn[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int nn = lane + 32 * e;
        float acc = z[nn];
        for (int kk = 0; kk < D; ++kk) acc = fmaf(z[kk], G[nn * D + kk], acc);
        zn[e] = acc;
      }
      __syncwarp();
#pragma unroll
      for (int e = 0; e < E; ++e) z[lane + 32 * e] = zn[e];
      __syncwarp();
    }
  }
  const float inv = 1.f / st.l;
  float* orow = out + (static_cast<size_t>(bh) * T + t) * D;
#pragma unroll
  for (int e = 0; e < E; ++e) orow[lane + 32 * e] = st.o[e] * inv;
  if (lse && lane == 0) lse[static_cast<size_t>(bh) * T + t] = (st.m + log2f(st.l)) * kLn2;
}

}  // namespace

cudaError_t launch_attn_f32(const Geom& g, const Inputs& in, const Workspace& ws,
                            cudaStream_t st, int* launches) {
  const dim3 grid((g.T + kWarpsPerBlock - 1) / kWarpsPerBlock, g.BH);
  const float sl2 = in.scale * kLog2e;
  const auto* v = static_cast<const float*>(in.v);
  auto* out = static_cast<float*>(in.out);
  const auto* kr = static_cast<const float*>(ws.kr);
  const auto* ngt = static_cast<const float*>(ws.ngt);
  const float* lam2 = g.gate ? ws.lam2 : nullptr;
  if (g.d == 64)
    attn_f32_kernel<64><<<grid, kWarpsPerBlock * 32, 0, st>>>(v, out, in.lse, kr, ws.ql, ngt,
                                                              ws.sdt, lam2, g.T, g.C, g.Np, sl2);
  else
    attn_f32_kernel<128><<<grid, kWarpsPerBlock * 32, 0, st>>>(v, out, in.lse, kr, ws.ql, ngt,
                                                               ws.sdt, lam2, g.T, g.C, g.Np, sl2);
  if (launches) *launches = 1;
  return cudaGetLastError();
}

}  // namespace pathattn
