// decode.cu -- PaTH decoding over a cache of keys that every new token
// rewrites in place, and the prefill step that fills that cache.
//
// "PaTH Attention: Position Encoding via Accumulating Householder
// Transformations" (slides), frame "Decoding updates historical keys in
// place": when token t arrives, each cached key j < t becomes
// k_j - beta_t w_t (w_t^T k_j).  The cache then holds H_t .. H_{j+1} k_j, whose
// dot product with q_t is the PaTH logit, and a plain causal softmax over the
// cache gives the output of token t.  The FoX gate of frame "FoX adds a
// separate mechanism for forgetting" enters as lam_t - lam_j, with lam the
// inclusive prefix sum of log f kept beside the cache.
//
// decode_split_kernel   one CTA per (span of cached keys, head).  The fp32
//                       key rows and the value rows of the span stream through
//                       a ring of shared-memory stages with bulk copies that
//                       complete on mbarriers.  Each key row is refined in
//                       shared memory, written back with a bulk store, and its
//                       logit (k_j . q - beta (w . k_j)(w . q)) feeds an online
//                       softmax.  The CTA leaves (max, sum, o) of its span in a
//                       partial buffer.
// decode_combine_kernel merges the spans of a head with the new token's own
//                       term, writes out and lse, and appends k_t, v_t and
//                       lam_t to the cache.
// align_keys_kernel     after a prefill of T tokens the cache must hold every
//                       key carried to the prompt end, H_{T-1} .. H_{j+1} k_j.
//                       From the forward's chunk factors (kr_c: keys carried to
//                       the end of their chunk; F_c = H_first .. H_last =
//                       I + ngt_c) that is the row block kr_c G_c with
//                       G_c = F_{c+1} .. F_{last}, built from the last chunk
//                       backwards; each CTA owns 32 columns of G.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace pathattn {
namespace {

template <typename ET>
__device__ __forceinline__ float4 ld4(const ET* p);

template <>
__device__ __forceinline__ float4 ld4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

template <>
__device__ __forceinline__ float4 ld4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename ET>
__device__ __forceinline__ ET from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

template <int G>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int off = G / 2; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// ------------------------------------------------------------ decode: split
template <typename ET, int D>
struct DecCfg {
  static constexpr int kThreads = 256;
  static constexpr int kWarps = kThreads / 32;
  static constexpr int kLpk = D / 16;  // lanes per key row, 16 elements per lane
  static constexpr int kKeysPerWarp = 32 / kLpk;
  static constexpr int kTile = kWarps * kKeysPerWarp;  // key rows per stage
  static constexpr int kKBytes = kTile * D * 4;
  static constexpr int kVBytes = kTile * D * static_cast<int>(sizeof(ET));
  static constexpr int kStages = sizeof(ET) == 2 ? 4 : 3;
  static constexpr int kStageBytes = kKBytes + kVBytes;
  static constexpr int kRedOff = kStages * kStageBytes;
  static constexpr int kRedBytes = kWarps * (D + 2) * 4;
  static constexpr int kBarOff = (kRedOff + kRedBytes + 15) / 16 * 16;
  static constexpr int kSmem = kBarOff + kStages * 8;
};

// The lane's 16 elements of a row: float4 slots i * kLpk + g, i = 0..3, so
// the kLpk lanes of a key read 16 * kLpk consecutive bytes per slot.
template <typename ET, int D>
__device__ __forceinline__ void load_row(const ET* row, int g, float (&x)[16]) {
  constexpr int L = D / 16;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = ld4<ET>(row + 4 * (i * L + g));
    x[4 * i] = f.x; x[4 * i + 1] = f.y; x[4 * i + 2] = f.z; x[4 * i + 3] = f.w;
  }
}

template <typename ET, int D>
__global__ void __launch_bounds__(256, 2) decode_split_kernel(const DecodeParams p) {
  using Cfg = DecCfg<ET, D>;
  constexpr int L = Cfg::kLpk, S = Cfg::kStages, TK = Cfg::kTile;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);
  float* red = reinterpret_cast<float*>(smem + Cfg::kRedOff);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane % L, key = warp * Cfg::kKeysPerWarp + lane / L;
  const int split = blockIdx.x, bh = blockIdx.y;
  const int t = p.pos[bh / p.H];
  const bool pos_ok = t >= 0 && t < p.max_len;
  const int j0 = split * p.span;
  const int jend = pos_ok ? min(j0 + p.span, t) : j0;
  const int ntile = jend > j0 ? (jend - j0 + TK - 1) / TK : 0;
  float* kc = p.kcache + static_cast<size_t>(bh) * p.Tmax * D;
  const ET* vc = static_cast<const ET*>(p.vcache) + static_cast<size_t>(bh) * p.Tmax * D;
  const float* lamc = p.lamcache ? p.lamcache + static_cast<size_t>(bh) * p.Tmax : nullptr;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int tile, int stage) {
    const int r0 = j0 + tile * TK;
    const int n = min(TK, jend - r0);
    unsigned char* sk = smem + stage * Cfg::kStageBytes;
    const uint32_t kb = static_cast<uint32_t>(n) * D * 4u;
    const uint32_t vb = static_cast<uint32_t>(n) * D * static_cast<uint32_t>(sizeof(ET));
    mbar_arrive_expect_tx(&full[stage], kb + vb);
    bulk_load(sk, kc + static_cast<size_t>(r0) * D, kb, &full[stage]);
    bulk_load(sk + Cfg::kKBytes, vc + static_cast<size_t>(r0) * D, vb, &full[stage]);
  };
  int issued = 0;
  if (tid == 0)
    for (; issued < S && issued < ntile; ++issued) issue(issued, issued);

  float qv[16], wv[16];
  load_row<ET, D>(static_cast<const ET*>(p.q) + static_cast<size_t>(bh) * D, g, qv);
  load_row<ET, D>(static_cast<const ET*>(p.w) + static_cast<size_t>(bh) * D, g, wv);
  float wq = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) wq = fmaf(wv[e], qv[e], wq);
  wq = group_sum<L>(wq);
  const float beta = p.beta[bh];
  const float sl2 = p.scale * kLog2e;
  float lam_t = 0.f;
  if (lamc && pos_ok) lam_t = (t > 0 ? lamc[t - 1] : 0.f) + p.logf[bh];

  float m = -INFINITY, l = 0.f, o[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) o[e] = 0.f;
  bool failed = false;
  int it = 0;
  for (; it < ntile; ++it) {
    const int st = it % S;
    const int j = j0 + it * TK + key;
    const bool valid = j < jend;
    const float lam_j = (lamc && valid) ? lamc[j] : 0.f;
    const bool ok = mbar_wait(&full[st], static_cast<uint32_t>(it / S) & 1u, nullptr, kWaitLimitNs);
    float4* ks = reinterpret_cast<float4*>(smem + st * Cfg::kStageBytes) + key * (D / 4);
    float kk[16];
    float kd = 0.f, wk = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 x = ks[i * L + g];
      kk[4 * i] = x.x; kk[4 * i + 1] = x.y; kk[4 * i + 2] = x.z; kk[4 * i + 3] = x.w;
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      kd = fmaf(kk[e], qv[e], kd);
      wk = fmaf(kk[e], wv[e], wk);
    }
    kd = group_sum<L>(kd);
    wk = group_sum<L>(wk);
    const float c = beta * wk;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      ks[i * L + g] = make_float4(fmaf(-c, wv[4 * i], kk[4 * i]), fmaf(-c, wv[4 * i + 1], kk[4 * i + 1]),
                                  fmaf(-c, wv[4 * i + 2], kk[4 * i + 2]),
                                  fmaf(-c, wv[4 * i + 3], kk[4 * i + 3]));
    if (valid) {
      // refined key . q = k . q - beta (w . k)(w . q)
      const float s = fmaf(-c, wq, kd) * sl2 + (lam_t - lam_j) * kLog2e;
      float vv[16];
      load_row<ET, D>(reinterpret_cast<const ET*>(smem + st * Cfg::kStageBytes + Cfg::kKBytes) +
                          key * D, g, vv);
      const float mn = fmaxf(m, s);
      const float corr = ex2_approx(m - mn);
      const float pj = ex2_approx(s - mn);
      l = fmaf(l, corr, pj);
#pragma unroll
      for (int e = 0; e < 16; ++e) o[e] = fmaf(o[e], corr, pj * vv[e]);
      m = mn;
    }
    fence_proxy_async_smem();
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    if (tid == 0) {
      const int r0 = j0 + it * TK;
      const int n = min(TK, jend - r0);
      bulk_store(kc + static_cast<size_t>(r0) * D, smem + st * Cfg::kStageBytes,
                 static_cast<uint32_t>(n) * D * 4u);
      bulk_commit();
      // refill the stage of the previous tile once its store has read it
      if (it >= 1 && issued < ntile) {
        bulk_wait_read<1>();
        issue(issued, (it - 1) % S);
        ++issued;
      }
    }
  }
  if (tid == 0) {
    if (failed) {
      atomicExch(p.status, PATH_DEV_ERR_TIMEOUT);
      // let every load still in flight land before the CTA leaves
      for (int tl = it; tl < issued; ++tl)
        mbar_wait(&full[tl % S], static_cast<uint32_t>(tl / S) & 1u, nullptr, kWaitLimitNs);
    }
    bulk_wait<0>();
  }

  // merge the key groups of the warp, then the warps
#pragma unroll
  for (int off = L; off < 32; off <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
    const float mn = fmaxf(m, m2);
    const float a = m == -INFINITY ? 0.f : ex2_approx(m - mn);
    const float b = m2 == -INFINITY ? 0.f : ex2_approx(m2 - mn);
    l = l * a + l2 * b;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float o2 = __shfl_xor_sync(0xffffffffu, o[e], off);
      o[e] = o[e] * a + o2 * b;
    }
    m = mn;
  }
  float* rw = red + warp * (D + 2);
  if (lane < L) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) rw[2 + 4 * (i * L + lane) + c4] = o[4 * i + c4];
    if (lane == 0) {
      rw[0] = m;
      rw[1] = l;
    }
  }
  __syncthreads();
  if (tid < D) {
    float M = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < Cfg::kWarps; ++w2) M = fmaxf(M, red[w2 * (D + 2)]);
    float Lsum = 0.f, O = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < Cfg::kWarps; ++w2) {
      const float mw = red[w2 * (D + 2)];
      const float a = mw == -INFINITY ? 0.f : ex2_approx(mw - M);
      Lsum = fmaf(red[w2 * (D + 2) + 1], a, Lsum);
      O = fmaf(red[w2 * (D + 2) + 2 + tid], a, O);
    }
    float* pp = p.part + (static_cast<size_t>(bh) * p.nsplit + split) * (D + 2);
    pp[2 + tid] = O;
    if (tid == 0) {
      pp[0] = failed ? NAN : M;
      pp[1] = Lsum;
    }
  }
}

// ---------------------------------------------------------- decode: combine
template <typename ET, int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const DecodeParams p) {
  __shared__ float wsum[D / 32];
  const int bh = blockIdx.x, e = threadIdx.x;
  const int t = p.pos[bh / p.H];
  ET* out = static_cast<ET*>(p.out) + static_cast<size_t>(bh) * D;
  if (t < 0 || t >= p.max_len) {
    if (e == 0) {
      atomicExch(p.status, PATH_DEV_ERR_BAD_POS);
      if (p.lse) p.lse[bh] = NAN;
    }
    out[e] = from_f<ET>(NAN);
    return;
  }
  const size_t row = static_cast<size_t>(bh) * D + e;
  const ET ke = static_cast<const ET*>(p.k)[row], ve = static_cast<const ET*>(p.v)[row];
  const float kf = to_f(ke), vf = to_f(ve), qf = to_f(static_cast<const ET*>(p.q)[row]);
  float qk = qf * kf;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, off);
  if ((e & 31) == 0) wsum[e >> 5] = qk;
  __syncthreads();
  qk = 0.f;
#pragma unroll
  for (int w2 = 0; w2 < D / 32; ++w2) qk += wsum[w2];
  const float st = qk * (p.scale * kLog2e);  // the new key's own gate is 0
  const float* pp = p.part + static_cast<size_t>(bh) * p.nsplit * (D + 2);
  float M = st;
  bool bad = false;
  for (int s = 0; s < p.nsplit; ++s) {
    const float ms = pp[s * (D + 2)];
    bad |= ms != ms;
    M = fmaxf(M, ms);
  }
  float Lsum = ex2_approx(st - M);
  float O = Lsum * vf;
  for (int s = 0; s < p.nsplit; ++s) {
    const float ms = pp[s * (D + 2)];
    const float a = ms == -INFINITY ? 0.f : ex2_approx(ms - M);
    Lsum = fmaf(pp[s * (D + 2) + 1], a, Lsum);
    O = fmaf(pp[s * (D + 2) + 2 + e], a, O);
  }
  out[e] = from_f<ET>(bad ? NAN : O / Lsum);
  if (e == 0 && p.lse) p.lse[bh] = bad ? NAN : (M + log2f(Lsum)) * kLn2;
  // append the new token
  const size_t crow = (static_cast<size_t>(bh) * p.Tmax + t) * D + e;
  p.kcache[crow] = kf;
  static_cast<ET*>(p.vcache)[crow] = ve;
  if (e == 0 && p.lamcache) {
    float* lamc = p.lamcache + static_cast<size_t>(bh) * p.Tmax;
    lamc[t] = (t > 0 ? lamc[t - 1] : 0.f) + p.logf[bh];
  }
}

// ------------------------------------------------------- prefill: align keys
template <typename ET, int D, int C>
struct AlignCfg {
  static constexpr int kThreads = 256;
  static constexpr int kNB = 32;      // columns of G owned by one CTA
  static constexpr int kLd = D + 4;   // padded fp32 row stride of the kr and ngt tiles
  static constexpr int kKrOff = 0;
  static constexpr int kMOff = kKrOff + C * kLd * 4;
  static constexpr int kGOff = kMOff + D * kLd * 4;
  static constexpr int kSmem = kGOff + D * kNB * 4;
};

// Copies a [rows][D] row-major element tile into padded fp32 shared rows.
template <typename ET, int D>
__device__ __forceinline__ void stage_rows(float* dst, const ET* src, int rows, int ld) {
  constexpr int kPer = 4;  // elements per access
  const int n = rows * D / kPer;
  for (int x = threadIdx.x; x < n; x += blockDim.x) {
    const int r = x / (D / kPer), c = (x % (D / kPer)) * kPer;
    *reinterpret_cast<float4*>(dst + r * ld + c) = ld4<ET>(src + static_cast<size_t>(r) * D + c);
  }
}

template <typename ET, int D, int C>
__global__ void __launch_bounds__(256, 1)
    align_keys_kernel(const ET* kr, const ET* ngt, float* kcache, int T, int Np, int Tp,
                      int Tmax) {
  using Cfg = AlignCfg<ET, D, C>;
  constexpr int NB = Cfg::kNB, LD = Cfg::kLd;
  extern __shared__ __align__(128) unsigned char smem[];
  float* sKr = reinterpret_cast<float*>(smem + Cfg::kKrOff);
  float* sM = reinterpret_cast<float*>(smem + Cfg::kMOff);
  float* sG = reinterpret_cast<float*>(smem + Cfg::kGOff);
  const int tid = threadIdx.x, tc = tid & 7, tr = tid >> 3;
  const int cb = blockIdx.x, bh = blockIdx.y;
  const int col0 = cb * NB;
  const ET* krh = kr + static_cast<size_t>(bh) * Tp * D;
  const ET* ngh = ngt + static_cast<size_t>(bh) * Np * D * D;
  float* kch = kcache + static_cast<size_t>(bh) * Tmax * D;
  for (int x = tid; x < D * NB; x += blockDim.x) {
    const int r = x / NB, c = x % NB;
    sG[x] = r == col0 + c ? 1.f : 0.f;
  }
  for (int ch = Np - 1; ch >= 0; --ch) {
    __syncthreads();  // the previous chunk's readers of sKr / sM are done
    stage_rows<ET, D>(sKr, krh + static_cast<size_t>(ch) * C * D, C, LD);
    if (ch > 0) stage_rows<ET, D>(sM, ngh + static_cast<size_t>(ch) * D * D, D, LD);
    __syncthreads();
    // keys of chunk ch carried to the prompt end: kr_ch G
    {
      constexpr int R = C / 32;
      float acc[R][4];
#pragma unroll
      for (int i = 0; i < R; ++i)
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) acc[i][c4] = 0.f;
#pragma unroll 4
      for (int k = 0; k < D; ++k) {
        const float4 gk = *reinterpret_cast<const float4*>(sG + k * NB + 4 * tc);
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const float a = sKr[(tr + 32 * i) * LD + k];
          acc[i][0] = fmaf(a, gk.x, acc[i][0]);
          acc[i][1] = fmaf(a, gk.y, acc[i][1]);
          acc[i][2] = fmaf(a, gk.z, acc[i][2]);
          acc[i][3] = fmaf(a, gk.w, acc[i][3]);
        }
      }
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const int j = ch * C + tr + 32 * i;
        if (j < T)
          *reinterpret_cast<float4*>(kch + static_cast<size_t>(j) * D + col0 + 4 * tc) =
              make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      }
    }
    if (ch == 0) break;
    // G <- F_ch G = G + ngt_ch G
    {
      constexpr int R = D / 32;
      float acc[R][4];
#pragma unroll
      for (int i = 0; i < R; ++i)
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) acc[i][c4] = 0.f;
#pragma unroll 4
      for (int k = 0; k < D; ++k) {
        const float4 gk = *reinterpret_cast<const float4*>(sG + k * NB + 4 * tc);
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const float a = sM[(tr + 32 * i) * LD + k];
          acc[i][0] = fmaf(a, gk.x, acc[i][0]);
          acc[i][1] = fmaf(a, gk.y, acc[i][1]);
          acc[i][2] = fmaf(a, gk.z, acc[i][2]);
          acc[i][3] = fmaf(a, gk.w, acc[i][3]);
        }
      }
      __syncthreads();  // every read of the old G is done
#pragma unroll
      for (int i = 0; i < R; ++i) {
        float4* gp = reinterpret_cast<float4*>(sG + (tr + 32 * i) * NB + 4 * tc);
        float4 gv = *gp;
        gv.x += acc[i][0]; gv.y += acc[i][1]; gv.z += acc[i][2]; gv.w += acc[i][3];
        *gp = gv;
      }
    }
  }
}

template <typename ET, int D>
cudaError_t launch_decode_t(const DecodeParams& p, int BH, cudaStream_t st) {
  using Cfg = DecCfg<ET, D>;
  auto kern = decode_split_kernel<ET, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(p.nsplit, BH), Cfg::kThreads, Cfg::kSmem, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  decode_combine_kernel<ET, D><<<BH, D, 0, st>>>(p);
  return cudaGetLastError();
}

template <typename ET, int D, int C>
cudaError_t launch_align_t(const Geom& g, const Workspace& ws, float* kcache, int Tmax,
                           cudaStream_t st) {
  using Cfg = AlignCfg<ET, D, C>;
  auto kern = align_keys_kernel<ET, D, C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(D / Cfg::kNB, g.BH), Cfg::kThreads, Cfg::kSmem, st>>>(
      static_cast<const ET*>(ws.kr), static_cast<const ET*>(ws.ngt), kcache, g.T, g.Np, g.Tp,
      Tmax);
  return cudaGetLastError();
}

}  // namespace

int decode_tile_keys(int d) { return d == 128 ? DecCfg<float, 128>::kTile : DecCfg<float, 64>::kTile; }

cudaError_t launch_decode(const DecodeParams& p, int BH, int d, bool bf16, cudaStream_t st) {
  if (bf16)
    return d == 128 ? launch_decode_t<__nv_bfloat16, 128>(p, BH, st)
                    : launch_decode_t<__nv_bfloat16, 64>(p, BH, st);
  return d == 128 ? launch_decode_t<float, 128>(p, BH, st) : launch_decode_t<float, 64>(p, BH, st);
}

cudaError_t launch_align_keys(const Geom& g, const Workspace& ws, float* kcache, int Tmax,
                              cudaStream_t st) {
  if (g.bf16)
    return g.d == 128 ? launch_align_t<__nv_bfloat16, 128, 128>(g, ws, kcache, Tmax, st)
                      : launch_align_t<__nv_bfloat16, 64, 128>(g, ws, kcache, Tmax, st);
  return g.d == 128 ? launch_align_t<float, 128, 64>(g, ws, kcache, Tmax, st)
                    : launch_align_t<float, 64, 64>(g, ws, kcache, Tmax, st);
}

}  // namespace pathattn
