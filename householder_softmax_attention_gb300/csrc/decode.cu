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
//                       softmax.  Each CTA leaves (max, sum, o) of its span in
//                       a partial buffer.
//                       The CTA that finishes last for a head (an atomic
//                       ticket per head) merges the head's spans with the new
//                       token's own term, writes out and lse, and appends
//                       k_t, v_t and lam_t to the cache.
// align_keys_kernel     after a prefill of T tokens the cache must hold every
//                       key carried to the prompt end, H_{T-1} .. H_{j+1} k_j.
//                       From the forward's chunk factors (kr_c: keys carried to
//                       the end of their chunk; F_c = H_first .. H_last =
//                       I + ngt_c) that is the row block kr_c G_c with
//                       G_c = F_{c+1} .. F_{last}, built from the last chunk
//                       backwards; each CTA owns 32 columns of G (fp32 SIMT
//                       for fp32 inputs, mma.sync for bf16).
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

// ------------------------------------------------------------ decode: merge
// Run by the whole CTA that finished last for head bh: merges the spans'
// (max, sum, o) with the new token's own term (its gate is 0), writes out and
// lse, and appends k_t, v_t and lam_t.  scratch holds D / 32 floats.
template <typename ET, int D>
__device__ __forceinline__ void merge_head(const DecodeParams& p, int bh, int t, bool pos_ok,
                                           float* scratch) {
  const int e = threadIdx.x;
  ET* out = static_cast<ET*>(p.out) + static_cast<size_t>(bh) * D;
  if (!pos_ok) {
    if (e == 0) {
      atomicExch(p.status, PATH_DEV_ERR_BAD_POS);
      if (p.lse) p.lse[bh] = NAN;
    }
    if (e < D) out[e] = from_f<ET>(NAN);
    return;
  }
  const size_t row = static_cast<size_t>(bh) * D + (e < D ? e : 0);
  const ET ke = static_cast<const ET*>(p.k)[row], ve = static_cast<const ET*>(p.v)[row];
  const float kf = to_f(ke), vf = to_f(ve), qf = to_f(static_cast<const ET*>(p.q)[row]);
  float qk = e < D ? qf * kf : 0.f;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, off);
  if ((e & 31) == 0 && e < D) scratch[e >> 5] = qk;
  __syncthreads();
  if (e >= D) return;
  qk = 0.f;
#pragma unroll
  for (int w2 = 0; w2 < D / 32; ++w2) qk += scratch[w2];
  const float st = qk * (p.scale * kLog2e);
  // partials of other CTAs: read through L2
  const float* pp = p.part + static_cast<size_t>(bh) * p.nsplit * (D + 2);
  float M = st;
  bool bad = false;
  for (int s2 = 0; s2 < p.nsplit; ++s2) {
    const float ms = __ldcg(pp + s2 * (D + 2));
    bad |= ms != ms;
    M = fmaxf(M, ms);
  }
  float Lsum = ex2_approx(st - M);
  float O = Lsum * vf;
  for (int s2 = 0; s2 < p.nsplit; ++s2) {
    const float ms = __ldcg(pp + s2 * (D + 2));
    const float a = ms == -INFINITY ? 0.f : ex2_approx(ms - M);
    Lsum = fmaf(__ldcg(pp + s2 * (D + 2) + 1), a, Lsum);
    O = fmaf(__ldcg(pp + s2 * (D + 2) + 2 + e), a, O);
  }
  out[e] = from_f<ET>(bad ? NAN : O / Lsum);
  if (e == 0 && p.lse) p.lse[bh] = bad ? NAN : (M + log2f(Lsum)) * kLn2;
  const size_t crow = (static_cast<size_t>(bh) * p.Tmax + t) * D + e;
  p.kcache[crow] = kf;
  static_cast<ET*>(p.vcache)[crow] = ve;
  if (e == 0 && p.lamcache) {
    float* lamc = p.lamcache + static_cast<size_t>(bh) * p.Tmax;
    lamc[t] = (t > 0 ? lamc[t - 1] : 0.f) + p.logf[bh];
  }
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
  // the CTA that finishes last for this head merges all of its spans
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(p.counters + bh, 1) == p.nsplit - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  merge_head<ET, D>(p, bh, t, pos_ok, red);
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

// bf16 inputs: the same product on the tensor cores (mma.sync, bf16
// operands, fp32 accumulation), transposed so that the carried quantity is
// the operand A of both products: with X = (G[:, cols])^T (32 x D),
//   keys^T  = X kr_c^T            (phase B, X split into bf16 hi + lo)
//   X_next  = X + X ngt_c^T       (phase A, fp32 master in the accumulators)
// Each warp owns 16 keys of phase B and D / 8 / 8 column tiles of phase A;
// kr_c and ngt_c stream through two cp.async stages.
template <int D>
struct AlignTcCfg {
  static constexpr int kC = 128, kNB = 32, kThreads = 256;
  static constexpr int kLd = D + 8;  // bf16 row stride of the staged tiles (conflict-free)
  static constexpr int kKrBytes = kC * kLd * 2;
  static constexpr int kMBytes = D * kLd * 2;
  static constexpr int kStageBytes = kKrBytes + kMBytes;
  static constexpr int kXBytes = kNB * kLd * 2;
  static constexpr int kXOff = 2 * kStageBytes;  // X: [buffer][hi, lo]
  static constexpr int kOLd = 36;                // fp32 row stride of the output tile
  static constexpr int kOOff = kXOff + 4 * kXBytes;
  static constexpr int kSmem = kOOff + kC * kOLd * 4;
  static constexpr int kNA = D / 64;             // phase-A column tiles per warp
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A fragment (16 x 16) of a row-major bf16 shared tile s[row][k], stride S.
__device__ __forceinline__ void frag_a(uint32_t (&a)[4], const __nv_bfloat16* s, int S, int m0,
                                       int k0, int g, int t) {
  a[0] = *reinterpret_cast<const uint32_t*>(s + (m0 + g) * S + k0 + 2 * t);
  a[1] = *reinterpret_cast<const uint32_t*>(s + (m0 + g + 8) * S + k0 + 2 * t);
  a[2] = *reinterpret_cast<const uint32_t*>(s + (m0 + g) * S + k0 + 2 * t + 8);
  a[3] = *reinterpret_cast<const uint32_t*>(s + (m0 + g + 8) * S + k0 + 2 * t + 8);
}

template <int D>
__global__ void __launch_bounds__(256, 1)
    align_keys_tc_kernel(const __nv_bfloat16* kr, const __nv_bfloat16* ngt, float* kcache, int T,
                         int Np, int Tp, int Tmax) {
  using Cfg = AlignTcCfg<D>;
  constexpr int C = Cfg::kC, LD = Cfg::kLd, NA = Cfg::kNA, OLD = Cfg::kOLd;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t4 = lane & 3;
  const int cb = blockIdx.x, bh = blockIdx.y, col0 = cb * Cfg::kNB;
  const __nv_bfloat16* krh = kr + static_cast<size_t>(bh) * Tp * D;
  const __nv_bfloat16* ngh = ngt + static_cast<size_t>(bh) * Np * D * D;
  float* kch = kcache + static_cast<size_t>(bh) * Tmax * D;
  float* so = reinterpret_cast<float*>(smem + Cfg::kOOff);
  auto xbuf = [&](int buf, int lo) {
    return reinterpret_cast<__nv_bfloat16*>(smem + Cfg::kXOff + (2 * buf + lo) * Cfg::kXBytes);
  };
  auto issue = [&](int c, int stage) {
    __nv_bfloat16* skr = reinterpret_cast<__nv_bfloat16*>(smem + stage * Cfg::kStageBytes);
    __nv_bfloat16* sm = reinterpret_cast<__nv_bfloat16*>(smem + stage * Cfg::kStageBytes +
                                                         Cfg::kKrBytes);
    const __nv_bfloat16* gkr = krh + static_cast<size_t>(c) * C * D;
    const __nv_bfloat16* gm = ngh + static_cast<size_t>(c) * D * D;
    constexpr int P = D / 8;  // 16-byte pieces per row
    for (int x = tid; x < C * P; x += Cfg::kThreads)
      cp_async16(skr + (x / P) * LD + (x % P) * 8, gkr + (x / P) * D + (x % P) * 8);
    for (int x = tid; x < D * P; x += Cfg::kThreads)
      cp_async16(sm + (x / P) * LD + (x % P) * 8, gm + (x / P) * D + (x % P) * 8);
    cp_async_commit();
  };
  issue(Np - 1, 0);
  // X = (identity columns col0 .. col0 + 31)^T
  for (int x = tid; x < Cfg::kNB * D; x += Cfg::kThreads) {
    const int n = x / D, k = x % D;
    xbuf(0, 0)[n * LD + k] = __float2bfloat16_rn(k == col0 + n ? 1.f : 0.f);
    xbuf(0, 1)[n * LD + k] = __float2bfloat16_rn(0.f);
  }
  float xm[2][NA][4];  // fp32 master of this warp's phase-A tiles of X
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int j = 0; j < NA; ++j)
#pragma unroll
      for (int f = 0; f < 4; ++f) {
        const int n = mt * 16 + g + (f >= 2 ? 8 : 0);
        const int k = (warp * NA + j) * 8 + 2 * t4 + (f & 1);
        xm[mt][j][f] = k == col0 + n ? 1.f : 0.f;
      }
  for (int it = 0; it < Np; ++it) {
    const int c = Np - 1 - it, stage = it & 1;
    cp_async_wait_all();
    __syncthreads();  // stage `stage`, X buffer it & 1 and the drained output tile are ready
    if (c > 0) issue(c - 1, stage ^ 1);
    const __nv_bfloat16* skr =
        reinterpret_cast<const __nv_bfloat16*>(smem + stage * Cfg::kStageBytes);
    const __nv_bfloat16* sm =
        reinterpret_cast<const __nv_bfloat16*>(smem + stage * Cfg::kStageBytes + Cfg::kKrBytes);
    const __nv_bfloat16* xh = xbuf(it & 1, 0);
    const __nv_bfloat16* xl = xbuf(it & 1, 1);
    float ob[2][2][4];
    float xa[2][NA][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int f = 0; f < 4; ++f) ob[mt][j][f] = 0.f;
#pragma unroll
      for (int j = 0; j < NA; ++j)
#pragma unroll
        for (int f = 0; f < 4; ++f) xa[mt][j][f] = xm[mt][j][f];
    }
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t ah[2][4], al[2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        frag_a(ah[mt], xh, LD, mt * 16, ks * 16, g, t4);
        frag_a(al[mt], xl, LD, mt * 16, ks * 16, g, t4);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {  // phase B: keys warp * 16 + 8 j ..
        const __nv_bfloat16* row = skr + (warp * 16 + 8 * j + g) * LD + ks * 16 + 2 * t4;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(row);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(row + 8);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          mma16816(ob[mt][j], ah[mt], b0, b1);
          mma16816(ob[mt][j], al[mt], b0, b1);
        }
      }
#pragma unroll
      for (int j = 0; j < NA; ++j) {  // phase A: columns (warp * NA + j) * 8 ..
        const __nv_bfloat16* row = sm + ((warp * NA + j) * 8 + g) * LD + ks * 16 + 2 * t4;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(row);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(row + 8);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) mma16816(xa[mt][j], ah[mt], b0, b1);
      }
    }
    // keys of chunk c: so[key][n] = (X kr_c^T)[n][key]
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int key = warp * 16 + 8 * j + 2 * t4, n = mt * 16 + g;
        so[key * OLD + n] = ob[mt][j][0];
        so[(key + 1) * OLD + n] = ob[mt][j][1];
        so[key * OLD + n + 8] = ob[mt][j][2];
        so[(key + 1) * OLD + n + 8] = ob[mt][j][3];
      }
    // the carried product crosses chunk c
    __nv_bfloat16* nh = xbuf((it + 1) & 1, 0);
    __nv_bfloat16* nl = xbuf((it + 1) & 1, 1);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int j = 0; j < NA; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float x0 = xa[mt][j][2 * h], x1 = xa[mt][j][2 * h + 1];
          xm[mt][j][2 * h] = x0;
          xm[mt][j][2 * h + 1] = x1;
          const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
          const int n = mt * 16 + g + 8 * h, k = (warp * NA + j) * 8 + 2 * t4;
          *reinterpret_cast<__nv_bfloat162*>(nh + n * LD + k) = __halves2bfloat162(h0, h1);
          *reinterpret_cast<__nv_bfloat162*>(nl + n * LD + k) = __halves2bfloat162(
              __float2bfloat16_rn(x0 - __bfloat162float(h0)),
              __float2bfloat16_rn(x1 - __bfloat162float(h1)));
        }
    __syncthreads();
    for (int x = tid; x < C * 8; x += Cfg::kThreads) {
      const int r = x >> 3, q = x & 7, j = c * C + r;
      if (j < T)
        *reinterpret_cast<float4*>(kch + static_cast<size_t>(j) * D + col0 + 4 * q) =
            *reinterpret_cast<const float4*>(so + r * OLD + 4 * q);
    }
  }
}

template <int D>
cudaError_t launch_align_tc(const Geom& g, const Workspace& ws, float* kcache, int Tmax,
                            cudaStream_t st) {
  using Cfg = AlignTcCfg<D>;
  auto kern = align_keys_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(D / Cfg::kNB, g.BH), Cfg::kThreads, Cfg::kSmem, st>>>(
      static_cast<const __nv_bfloat16*>(ws.kr), static_cast<const __nv_bfloat16*>(ws.ngt), kcache,
      g.T, g.Np, g.Tp, Tmax);
  return cudaGetLastError();
}

template <typename ET, int D>
cudaError_t launch_decode_t(const DecodeParams& p, int BH, cudaStream_t st) {
  using Cfg = DecCfg<ET, D>;
  auto kern = decode_split_kernel<ET, D>;
  static bool attr_set[64] = {};  // once per device (setting it again is harmless)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  Cfg::kSmem)) != cudaSuccess)
      return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  kern<<<dim3(p.nsplit, BH), Cfg::kThreads, Cfg::kSmem, st>>>(p);
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
    return g.d == 128 ? launch_align_tc<128>(g, ws, kcache, Tmax, st)
                      : launch_align_tc<64>(g, ws, kcache, Tmax, st);
  return g.d == 128 ? launch_align_t<float, 128, 64>(g, ws, kcache, Tmax, st)
                    : launch_align_t<float, 64, 64>(g, ws, kcache, Tmax, st);
}

}  // namespace pathattn
