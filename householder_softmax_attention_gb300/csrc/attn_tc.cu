// attn_tc.cu -- PaTH forward scan on the sm_103a tensor cores (dtype bf16).
//
// One CTA per 128-row query tile (= one chunk b of one head).  The tile walks
// the key chunks backwards from the diagonal ("PaTH Attention ..." slides,
// frame "A right-to-left scan accumulates cross-block paths"):
//
//   diagonal   P_b = softmax-step(sdt_b)            (logits precomputed, fp32)
//   for c = b-1 .. 0:
//     [S | Qm] += Qw . [kr_c ; ngt_c]^T            one tcgen05 MMA (S zeroed
//                                                  first; no ngt for c = 0)
//     P_c = softmax-step(S)                        online softmax, lazy rescale
//     O  += P_{c+1} . V_{c+1}                      tcgen05, A = P from TMEM
//   O += P_0 . V_0;  out = O / l,  lse = (m + log2 l) ln 2
//
// Qm is the fp32 master of the running query (q_i carried through every
// transition crossed so far), held in TMEM and updated in place by the MMA;
// Qw is its bf16 copy, the A operand of the next step.  The transition is the
// dense d x d form of F_c^T = I - W^T U W from the chunk preparation.
//
// Warp roles (384 threads; 512 at d = 64):
//   warp 0      TMA producer: kr_c over ngt_c (one B tile), V (own ring)
//   warp 1      TMEM allocation; one thread issues the [S | Qm] MMAs
//   warp 2      one thread issues the O += P V MMAs
//   warps 4-7   softmax: one query row per thread (TMEM lane = row); at
//               d = 64 keys 0-63 of each step, warps 12-15 keys 64-127
//   warps 8-11  running-query conversion Qm -> Qw (and its initial load)
// TMEM columns: S [0,128), Qm (d), O (d), Qw (d/2, packed bf16x2), P (64).
// Every wait is bounded; on expiry the CTA records PATH_DEV_ERR_TIMEOUT in the
// status word, drains its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "ptx.cuh"

namespace pathattn {
namespace {

constexpr int kC = 128;       // chunk length = query tile = key tile
// 384 threads; at d = 64 (dense form) 512: each query row's logits are then
// split between two softmax warpgroups, 64 keys each (see below).
template <int D, bool kLR>
constexpr bool kSplitRows = D == 64 && !kLR;
template <int D, bool kLR>
constexpr int kThreadsOf = kSplitRows<D, kLR> ? 512 : 384;
// Tiles launch in groups of 4 heads: the group's kr, ngt and V chunks (12 MB
// per head at T = 16384, d = 128) then stay in L2 until its last tile has
// read them.  Measured at B = 2, H = 16, T = 16384, d = 128 (DRAM bytes per
// launch, ncu; floor 1.05 GB): groups of 16 heads 3.34 GB, 8 heads 1.83 GB,
// 4 heads 1.09 GB, 2 heads 1.06 GB; attention 1.986 / 1.914 / 1.891 / 1.891 ms.
constexpr int kHeadGroup = 4;
constexpr int kRegsLow = 56, kRegsSoftmax = 240, kRegsSoftmaxHalf = 168, kRegsQuery = 112;
static_assert(128 * (kRegsLow + kRegsSoftmax + kRegsQuery) <= 384 * 168, "register split");
static_assert(128 * (kRegsLow + 2 * kRegsSoftmaxHalf + kRegsQuery) <= 512 * 128,
              "register split, rows in two halves");

// D: head dimension; R: the coordinates the transitions act on (R = D for
// PaTH; R < D for partial PaTH, whose running query changes only in its
// first R coordinates and whose ngt_c vanishes outside its first R rows).
// kLR: the low-rank form of the transition (d = 64 only), see below.
template <int D, int R, bool kLR = false>
struct TcCfg {
  static_assert(R <= D && R % 64 == 0, "transition rank");
  static_assert(!kLR || (D == 64 && R == 64), "the low-rank form is built at d = 64");
  static constexpr int kHalves = D / 64;           // 64-column (128-byte) halves
  // One B tile per step stacks kr_c (kC rows) over the first R rows of ngt_c,
  // so that S = Qw kr^T and the transition Qm += Qw ngt^T are a single MMA
  // of width N = kC + R; tcgen05.mma pays a fixed cost per instruction below
  // N = 256.  Low-rank form: kr_c over W_c ([S | Y] = Qw [kr_c ; W_c]^T),
  // and -(U W)_c beside them, the B operand of Qm += Y (-(U W)_c).
  static constexpr int kKgRows = kLR ? 2 * kC : kC + R;
  static constexpr uint32_t kKgHalf = kKgRows * 128;  // one 64-column half
  static constexpr uint32_t kKgBytes = kHalves * kKgHalf;
  static constexpr uint32_t kUwBytes = kLR ? kC * D * 2 : 0;
  static constexpr uint32_t kStageBytes = kKgBytes + kUwBytes;
  static constexpr uint32_t kVBytes = kC * D * 2;
  // low-rank form: the bf16 copy of Y, A operand of the second product
  // (K-major, two 64-column halves)
  static constexpr uint32_t kYwBytes = kLR ? kC * kC * 2 : 0;
  static constexpr uint32_t kColS = 0;             // S and Qm are adjacent: one
  static constexpr uint32_t kColY = 128;           // (low-rank: S and Y)
  static constexpr uint32_t kColQm = kLR ? 256 : 128;  // accumulator of width kC + R
  static constexpr uint32_t kColO = kColQm + R;
  static constexpr uint32_t kColQw = kColO + D;
  static constexpr uint32_t kColP = kColQw + D / 2;
  // rows in two halves: the second half's O (its own reference max and sum)
  static constexpr uint32_t kColO2 = kColP + 64;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr size_t kTileBytes = 2 * (kStageBytes + kVBytes) + kYwBytes;
  // rows in two halves: the second half's (m, l) per row, after the barriers
  static constexpr size_t kXchOffset = kTileBytes + 1280;
  static constexpr size_t kSmemBytes =
      kTileBytes + 1024 /*align*/ + 1280 /*barriers, gate*/ + (D == 64 && !kLR ? 2 * kC * 4 : 0);
  static_assert(kColP + 64 <= kTmemCols, "TMEM budget");
  static_assert(kColO2 + D <= kTmemCols || D != 64 || kLR, "TMEM budget of the second O");
};

// Whether the first k-step of the fused logits MMA writes S alone (starting
// it from zero) instead of the softmax warps clearing S after reading it: one
// more MMA instruction per step, four fewer TMEM stores on the softmax path.
// Measured: 4% faster at d = 64 and 1.5-2% with the FoX gate, where the
// softmax weighs most; 2% slower for plain d = 128 (1.87 -> 1.90 ms at
// B=2 H=16 T=16384), whose step the tensor pipe bounds (kept on the
// clearing form).
template <int D, bool kGate>
constexpr bool kSplitFirst = D == 64 || kGate;

struct Bars {
  uint64_t kg_full[2], kg_empty[2], v_full[2], v_empty[2];
  uint64_t sq_ready, p_full, qk_done, pv_done, final_done;
  uint64_t yw_ready, q_done;  // low-rank form: Y converted; Qm += Y (-UW) done
  uint64_t gate_full[2], gate_empty[2];  // FoX: the gate ring below
  uint64_t xch_full;  // rows in two halves: the second half's (m, l) published
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) float gate[2][kC];  // FoX: log2-domain gate prefix of a key chunk
};

static_assert(sizeof(Bars) <= 1280, "barrier block size");

// The warp's tcgen05 stores / loads are fenced by each thread before this;
// the warp then arrives once.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

__device__ __forceinline__ void record_timeout(Bars* bars, int* status) {
  bars->abort_flag = 1;
  atomicExch(status, PATH_DEV_ERR_TIMEOUT);
}

// Row max / min of N values held as bit patterns: three-input max / min in
// four independent chains (a single chain would put every operation on the
// path).
template <int N>
__device__ __forceinline__ float row_max(const uint32_t (&x)[N]) {
  float m[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) m[u] = __uint_as_float(x[u]);
#pragma unroll
  for (int j = 4; j < N; j += 2)
    m[(j >> 1) & 3] = max3f(m[(j >> 1) & 3], __uint_as_float(x[j]), __uint_as_float(x[j + 1]));
  return max3f(m[0], m[1], fmaxf(m[2], m[3]));
}
template <int N>
__device__ __forceinline__ float row_min(const uint32_t (&x)[N]) {
  float m[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) m[u] = __uint_as_float(x[u]);
#pragma unroll
  for (int j = 4; j < N; j += 2)
    m[(j >> 1) & 3] = min3f(m[(j >> 1) & 3], __uint_as_float(x[j]), __uint_as_float(x[j + 1]));
  return min3f(m[0], m[1], fminf(m[2], m[3]));
}

// p_j = 2^(mul x_j - m) for N values held as bit patterns, as bf16 pairs in
// pk, returning their sum; the argument and the running sums go two values
// per instruction (four packed partial sums).
template <int N>
__device__ __forceinline__ float exp_row(const uint32_t (&x)[N], float mul, float m,
                                         uint32_t (&pk)[N / 2]) {
  const uint64_t mulv = f2(mul, mul), negm = f2(-m, -m);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    float a0, a1;
    f2_split(f2_fma(f2(__uint_as_float(x[j]), __uint_as_float(x[j + 1])), mulv, negm), a0, a1);
    const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
    acc[(j >> 1) & 3] = f2_add(acc[(j >> 1) & 3], f2(p0, p1));
    pk[j >> 1] = pack_bf16x2(p0, p1);
  }
  float s[8];
#pragma unroll
  for (int u = 0; u < 4; ++u) f2_split(acc[u], s[2 * u], s[2 * u + 1]);
  return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

// End of every role: all NT threads meet on named barrier 1, then warp 1
// (the allocating warp) frees TMEM.
template <int NT>
__device__ __forceinline__ void teardown(int warp, uint32_t tb, uint32_t ncols) {
  tc_fence_before_sync();
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tb, ncols);
  }
}

template <int D, bool kGate, int R, bool kLR>
__global__ void __launch_bounds__(kThreadsOf<D, kLR>, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap map_kr,
                   const __grid_constant__ CUtensorMap map_ng,
                   const __grid_constant__ CUtensorMap map_v,
                   const __grid_constant__ CUtensorMap map_uw, const float* __restrict__ ql,
                   const float* __restrict__ sdt, const float* __restrict__ lam2,
                   __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                   int* __restrict__ status, int T, int Np, int BH, float sl2) {
  using Cfg = TcCfg<D, R, kLR>;
  constexpr bool kSplit = kSplitRows<D, kLR>;
  constexpr int kNT = kThreadsOf<D, kLR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* s_kg = base;                                   // [2][kStageBytes]
  uint8_t* s_v = base + 2 * Cfg::kStageBytes;             // [2][kVBytes]
  uint8_t* s_yw = s_v + 2 * Cfg::kVBytes;                 // low-rank: [kYwBytes]
  Bars* bars = reinterpret_cast<Bars*>(base + Cfg::kTileBytes);
  // rows in two halves: the second half's m and l of each row
  float* xch_m = reinterpret_cast<float*>(base + Cfg::kXchOffset);
  float* xch_l = xch_m + kC;
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Tile order: heads in groups of kHeadGroup; inside a group, longest tiles
  // (largest b) first, interleaved over the group's heads.  Tiles of one head
  // that run together walk the same kr / ngt / V chunks, which then come
  // from L2; longest-first keeps the tail short.
  auto tile_of = [&](int ord, int& tb_, int& tbh) {
    const int per_group = kHeadGroup * Np;
    const int grp = ord / per_group, r = ord - grp * per_group;
    const int heads = min(kHeadGroup, BH - grp * kHeadGroup);
    tb_ = Np - 1 - r / heads;
    tbh = grp * kHeadGroup + r % heads;
  };
  int b, bh;
  tile_of(blockIdx.x, b, bh);
  const int Tp = Np * kC;
  const uint64_t LIM = kWaitLimitNs;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->kg_full[s], 1);
      mbar_init(&bars->kg_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    // the next [S | Qm] MMA may go once Qw is refreshed (4 running-query
    // warps) and S has been read and zeroed (4 softmax warps)
    mbar_init(&bars->sq_ready, kSplit ? 12 : 8);
    mbar_init(&bars->p_full, kSplit ? 8 : 4);  // one arrival per warp
    mbar_init(&bars->qk_done, 1);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->final_done, 2);  // one commit from each MMA-issuing thread
    mbar_init(&bars->yw_ready, 4);    // low-rank: the 4 running-query warps
    mbar_init(&bars->q_done, 1);
    mbar_init(&bars->xch_full, 4);  // rows in two halves: the second half's 4 warps
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->gate_full[s], 1);
      mbar_init(&bars->gate_empty[s], kSplit ? 8 : 4);  // the softmax warps, once read
    }
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&map_kr);
    tma_prefetch_map(&map_ng);
    tma_prefetch_map(&map_v);
    if (kLR) tma_prefetch_map(&map_uw);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tb = bars->tmem_base;

  // 384 threads launched at <= 168 registers each (64512); each warpgroup
  // re-sizes itself: 128 x 56 (producer / MMA / idle) + 128 x 240 (softmax) +
  // 128 x 112 (running query) = 52224.  The three warpgroups never rejoin:
  // each ends with its own copy of the teardown.
  if (warp < 4) {
    regs_dec<kRegsLow>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int last_kg[2] = {-1, -1}, last_v[2] = {-1, -1}, last_g[2] = {-1, -1};
      bool ok = true;
      for (int n = 0; n <= b && ok; ++n) {
        const int s = n & 1;
        if (n == max(b - 3, 0)) {
          // The tile one wave ahead (launch index + SM count) starts about
          // when this one ends, a few steps from here: its running query and
          // diagonal logits, written by the preparation and read once, into
          // L2 now, so that its first loads come from there, not from HBM.
          const int ord2 = blockIdx.x + static_cast<int>(sm_count());
          if (ord2 < static_cast<int>(gridDim.x)) {
            int b2, bh2;
            tile_of(ord2, b2, bh2);
            const size_t ch2 = static_cast<size_t>(bh2) * Np + b2;
            if (b2 > 0) bulk_prefetch_l2(ql + ch2 * kC * D, kC * D * 4);
            bulk_prefetch_l2(sdt + ch2 * kC * kC, kC * kC * 4);
          }
        }
        if (n < b) {
          const int c = b - 1 - n;
          if (n >= 2) ok = mbar_wait(&bars->kg_empty[s], ((n >> 1) - 1) & 1, abort_flag, LIM);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars->kg_full[s], Cfg::kStageBytes);
          uint8_t* stage = s_kg + s * Cfg::kStageBytes;
          for (int h = 0; h < Cfg::kHalves; ++h) {
            uint8_t* dst = stage + h * Cfg::kKgHalf;
            tma_load_2d(dst, &map_kr, h * 64, bh * Tp + c * kC, &bars->kg_full[s]);
            if constexpr (kLR)   // W_c, the input directions (rows past T read as zero)
              tma_load_3d(dst + kC * 128, &map_ng, h * 64, c * kC, bh, &bars->kg_full[s]);
            else
              tma_load_2d(dst + kC * 128, &map_ng, h * 64, (bh * Np + c) * D, &bars->kg_full[s]);
          }
          if constexpr (kLR)     // -(U W)_c, kC rows of D
            for (int h = 0; h < Cfg::kHalves; ++h)
              tma_load_2d(stage + Cfg::kKgBytes + h * (kC * 128), &map_uw, h * 64,
                          (bh * Np + c) * kC, &bars->kg_full[s]);
          last_kg[s] = (n >> 1) & 1;
          if (kGate) {
            // the key chunk's gate prefix (512 bytes) for the softmax warps
            if (n >= 2) ok = mbar_wait(&bars->gate_empty[s], ((n >> 1) - 1) & 1, abort_flag, LIM);
            if (!ok) break;
            mbar_arrive_expect_tx(&bars->gate_full[s], kC * 4);
            bulk_load(&bars->gate[s][0], lam2 + static_cast<size_t>(bh) * Tp + c * kC, kC * 4,
                      &bars->gate_full[s]);
            last_g[s] = (n >> 1) & 1;
          }
        }
        if (n >= 2) ok = mbar_wait(&bars->v_empty[s], ((n >> 1) - 1) & 1, abort_flag, LIM);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars->v_full[s], Cfg::kVBytes);
        for (int h = 0; h < Cfg::kHalves; ++h)
          tma_load_3d(s_v + s * Cfg::kVBytes + h * (kC * 128), &map_v, h * 64, (b - n) * kC, bh,
                      &bars->v_full[s]);
        last_v[s] = (n >> 1) & 1;
      }
      if (!ok) record_timeout(bars, status);
      // every copy this thread started has landed before the CTA may exit
      for (int s = 0; s < 2; ++s) {
        if (last_kg[s] >= 0) mbar_wait(&bars->kg_full[s], last_kg[s], nullptr, LIM);
        if (last_v[s] >= 0) mbar_wait(&bars->v_full[s], last_v[s], nullptr, LIM);
        if (last_g[s] >= 0) mbar_wait(&bars->gate_full[s], last_g[s], nullptr, LIM);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ logits issuer
    // [S | Qm] += Qw [kr_c ; ngt_c]^T for c = b-1 .. 0.  A second thread
    // (warp 2) issues O += P V: each waits only on its own barriers, so the
    // tensor pipe is fed while the other is blocked (one issuing thread spent
    // most of a step in barrier waits with the pipe idle).
    if (lane == 0) {
      const uint32_t tS = tb + Cfg::kColS, tQw = tb + Cfg::kColQw;
      constexpr uint32_t idS = idesc_bf16_f32(128, kC, false, false);       // S only
      constexpr uint32_t idSQ = idesc_bf16_f32(128, kC + R, false, false);  // [S | Qm]
      constexpr uint32_t idQ = idesc_bf16_f32(128, R, false, false);        // Qm only
      bool ok = true;
      for (int n = 0; n < b && ok; ++n) {
        const int c = b - 1 - n, s = n & 1;
        // the stage is usually loaded long before: check it first, then wait
        // for Qw and S (one barrier, the one that blocks)
        ok = mbar_spin(&bars->kg_full[s], (n >> 1) & 1, abort_flag, LIM);
        if (ok) ok = mbar_spin(&bars->sq_ready, n & 1, abort_flag, LIM);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t kg_a = smem_addr(s_kg + s * Cfg::kStageBytes);
        if constexpr (kLR) {
          // low-rank form: [S | Y] = Qw [kr_c ; W_c]^T from zero (width 2 kC;
          // S alone for the last chunk), then, once the running-query warps
          // have turned Y into bf16 in shared memory, Qm += Y (-(U W)_c)
          constexpr uint32_t idSY = idesc_bf16_f32(128, 2 * kC, false, false);
          constexpr uint32_t idQ2 = idesc_bf16_f32(128, D, false, true);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * Cfg::kKgHalf + (k & 3) * 32;
            mma_bf16_ts(tS, tQw + k * 8, sdesc_sw128(kg_a + off, 16, 1024), c > 0 ? idSY : idS,
                        k > 0);
          }
          mma_commit(&bars->qk_done);
          if (c > 0) {
            ok = mbar_spin(&bars->yw_ready, n & 1, abort_flag, LIM);
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t yw = smem_addr(s_yw), uw = kg_a + Cfg::kKgBytes;
#pragma unroll
            for (int k = 0; k < kC / 16; ++k)
              mma_bf16_ss(tb + Cfg::kColQm,
                          sdesc_sw128(yw + (k >> 2) * (kC * 128) + (k & 3) * 32, 16, 1024),
                          sdesc_sw128(uw + k * 2048, kC * 128, 1024), idQ2, 1);
            mma_commit(&bars->q_done);
          }
          mma_commit(&bars->kg_empty[s]);
          continue;
        }
        // the logits and the backward crossing of chunk c in one MMA of width
        // kC + R; the last chunk needs no crossing.  S starts from zero:
        // either the first k-step writes it alone (the crossing part
        // accumulating into Qm) or the softmax warps cleared it
        const uint32_t id = c > 0 ? idSQ : idS;
        int k = 0;
        if constexpr (kSplitFirst<D, kGate>) {
          mma_bf16_ts(tS, tQw, sdesc_sw128(kg_a, 16, 1024), idS, 0);
          if (c > 0) mma_bf16_ts(tS + kC, tQw, sdesc_sw128(kg_a + kC * 128, 16, 1024), idQ, 1);
          k = 1;
        }
#pragma unroll
        for (; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * Cfg::kKgHalf + (k & 3) * 32;
          mma_bf16_ts(tS, tQw + k * 8, sdesc_sw128(kg_a + off, 16, 1024), id, 1);
        }
        mma_commit(&bars->qk_done);
        mma_commit(&bars->kg_empty[s]);
      }
      if (!ok) record_timeout(bars, status);
      // this thread's MMAs complete before TMEM is released
      mma_commit(&bars->final_done);
      mbar_wait(&bars->final_done, 0, nullptr, LIM);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ PV issuer
    // O += P_{c+1} V_{c+1} for n = 0 .. b (the diagonal's P first)
    if (lane == 0) {
      const uint32_t tO = tb + Cfg::kColO, tP = tb + Cfg::kColP;
      constexpr uint32_t idPV = idesc_bf16_f32(128, D, false, true);
      bool ok = true;
      for (int n = 0; n <= b && ok; ++n) {
        const int s = n & 1;
        ok = mbar_spin(&bars->v_full[s], (n >> 1) & 1, abort_flag, LIM);
        if (ok) ok = mbar_spin(&bars->p_full, n & 1, abort_flag, LIM);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t v_a = smem_addr(s_v + s * Cfg::kVBytes);
#pragma unroll
        for (int k = 0; k < kC / 16; ++k) {
          // rows in two halves: keys 0-63 into O, keys 64-127 into O2
          const bool second = kSplit && k >= kC / 32;
          mma_bf16_ts(second ? tb + Cfg::kColO2 : tO, tP + k * 8,
                      sdesc_sw128(v_a + k * 2048, kC * 128, 1024), idPV,
                      (n > 0 || k > (second ? kC / 32 : 0)));
        }
        mma_commit(&bars->pv_done);
        if (n < b) mma_commit(&bars->v_empty[s]);
      }
      if (!ok) record_timeout(bars, status);
      mma_commit(&bars->final_done);
      mbar_wait(&bars->final_done, 0, nullptr, LIM);
    }
  }
    teardown<kNT>(warp, tb, Cfg::kTmemCols);
  } else if (warp < 8 || warp >= 12) {
    // ------------------------------------------------------------ softmax
    // One query row per thread (TMEM lane = row).  With rows in two halves
    // (d = 64), warps 4-7 take keys 0-63 and warps 12-15 keys 64-127 of the
    // same rows, each half with its own reference max m, sum l and output
    // accumulator (O, O2): the halves never wait on each other until the
    // epilogue, where the second half publishes (m, l) and the first merges.
    constexpr int NC = kSplit ? 64 : kC;   // keys of a step this thread handles
    if constexpr (kSplit) regs_inc<kRegsSoftmaxHalf>();
    else regs_inc<kRegsSoftmax>();
    const int h = kSplit && warp >= 12 ? 1 : 0;
    const int col0 = h * 64;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int t = b * kC + r;
    const uint32_t lb = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tS = tb + lb + Cfg::kColS, tP = tb + lb + Cfg::kColP;
    const uint32_t tO = tb + lb + (h ? Cfg::kColO2 : Cfg::kColO);
    uint32_t x[NC];
    float m_used, l = 0.f;
    // S is free for the first MMA: started from zero by it, or cleared here
    if constexpr (!kSplitFirst<D, kGate>) {
      uint32_t z[32];
#pragma unroll
      for (int u = 0; u < 32; ++u) z[u] = 0u;
#pragma unroll
      for (int cc = 0; cc < NC; cc += 32) tmem_st_x32(tS + col0 + cc, z);
      tmem_st_wait();
      tc_fence_before_sync();
    }
    warp_arrive(&bars->sq_ready);
    // diagonal chunk: precomputed log2-domain logits sdt[ch][j][i]
    {
      const float* sd = sdt + (static_cast<size_t>(bh) * Np + b) * kC * kC + r;
#pragma unroll
      for (int j = 0; j < NC; ++j) x[j] = __float_as_uint(__ldg(sd + (col0 + j) * kC));
      m_used = row_max(x);
      // a half whose keys all lie above the diagonal (rows below 64, second
      // half) holds only -inf: any finite reference gives it zero weight
      if (kSplit && m_used == -INFINITY) m_used = 0.f;
      uint32_t pk[NC / 2];
      l = exp_row(x, 1.f, m_used, pk);
#pragma unroll
      for (int cc = 0; cc < NC / 2; cc += 32)
        tmem_st_x32(tP + h * 32 + cc, *reinterpret_cast<uint32_t(*)[32]>(&pk[cc]));
      tmem_st_wait();
      tc_fence_before_sync();
      warp_arrive(&bars->p_full);
    }
    bool ok = true;
    // FoX: logits of the off-diagonal chunks are handled shifted by this row's
    // gate prefix, y_j = scale S_j - lam2_j (log2 units), so the reference max
    // is kept in that domain and lrow comes back for lse
    const float lrow = kGate ? lam2[static_cast<size_t>(bh) * Tp + t] : 0.f;
    if (kGate) m_used -= lrow;
    for (int n = 0; n < b; ++n) {
      // FoX: the chunk's gate prefix (loaded by the producer into the ring,
      // long before) is waited for here, off the path from S to P
      if (kGate) {
        ok = mbar_wait(&bars->gate_full[n & 1], (n >> 1) & 1, abort_flag, LIM);
        if (!ok) break;
      }
      ok = mbar_wait(&bars->qk_done, n & 1, abort_flag, LIM);
      if (!ok) break;
      {
      tc_fence_after_sync();
      // S is read; the next MMA starts it from zero, or it is cleared
      if constexpr (NC == 128) {
        tmem_ld_x128(tS, x);
      } else {
        tmem_ld_x64(tS + col0, x);
      }
      if constexpr (!kSplitFirst<D, kGate>) {
        uint32_t z[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) z[u] = 0u;
#pragma unroll
        for (int cc = 0; cc < NC; cc += 32) tmem_st_x32(tS + col0 + cc, z);
        tmem_st_wait();
      }
      tc_fence_before_sync();
      warp_arrive(&bars->sq_ready);
      float mx = -INFINITY;
      if (kGate) {
        // z_j = lam2_j - scale S_j = -y_j, two per instruction; max y = -min z
        const uint64_t* lg = reinterpret_cast<const uint64_t*>(&bars->gate[n & 1][col0]);
        const uint64_t nsl = f2(-sl2, -sl2);
#pragma unroll
        for (int j = 0; j < NC; j += 2) {
          float z0, z1;
          f2_split(f2_fma(f2(__uint_as_float(x[j]), __uint_as_float(x[j + 1])), nsl, lg[j >> 1]),
                   z0, z1);
          x[j] = __float_as_uint(z0);
          x[j + 1] = __float_as_uint(z1);
        }
        warp_arrive(&bars->gate_empty[n & 1]);
      }
      // The step's exponentials against the current reference max (gated: x
      // holds z = -y, scaled, log2 units; plain logits get the scale here).
      // Only when their sum shows that the logits grew past it (a term above
      // 2^9) is the row max taken and the reference moved (lazy rescaling);
      // otherwise the step needs no max at all.  NaN sums take that path too.
      const float mul = kGate ? -1.f : sl2;
      uint32_t pk[NC / 2];
      float ls = exp_row(x, mul, m_used, pk);
      bool need = false;
      float alpha = 1.f;
      if (!(ls <= 65536.f)) {
        if (kGate) {
          mx = -row_min(x);
        } else if (sl2 >= 0.f) {
          mx = row_max(x) * sl2;
        } else {
          mx = row_min(x) * sl2;
        }
        need = mx > m_used + 8.f;
        if (need) {
          alpha = ex2_approx(m_used - mx);
          m_used = mx;
          l *= alpha;
          ls = exp_row(x, mul, m_used, pk);
        }
      }
      l += ls;
      // P buffer and O are free once O += P_{c+1} V_{c+1} has completed
      ok = mbar_wait(&bars->pv_done, n & 1, abort_flag, LIM);
      if (!ok) break;
      {
      tc_fence_after_sync();
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          tmem_ld_x32(tO + cc, o);
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
          tmem_st_x32(tO + cc, o);
        }
      }
#pragma unroll
      for (int cc = 0; cc < NC / 2; cc += 32)
        tmem_st_x32(tP + h * 32 + cc, *reinterpret_cast<uint32_t(*)[32]>(&pk[cc]));
      tmem_st_wait();
      tc_fence_before_sync();
      warp_arrive(&bars->p_full);
      }  // pv_done
      }  // qk_done
    }
    // epilogue: out = O / l, lse = (m + log2 l) ln 2; with rows in two halves
    // the second half publishes (m, l) and the first merges the two partial
    // softmaxes (O and O2 weighted by 2^(m_h - M), M the larger reference)
    if (ok) ok = mbar_wait(&bars->pv_done, b & 1, abort_flag, LIM);
    if (kSplit && h == 1) {
      if (ok) {
        xch_m[r] = m_used;
        xch_l[r] = l;
        warp_arrive(&bars->xch_full);
      } else {
        record_timeout(bars, status);
      }
    } else {
      float s0 = 1.f, s1 = 0.f, M = m_used;
      if (kSplit && ok) {
        ok = mbar_wait(&bars->xch_full, 0, abort_flag, LIM);
        if (ok) {
          const float m1 = xch_m[r], l1 = xch_l[r];
          M = fmaxf(m_used, m1);
          s0 = ex2_approx(m_used - M);
          s1 = ex2_approx(m1 - M);
          l = l * s0 + l1 * s1;
        }
      }
      if (ok) {
        tc_fence_after_sync();
        const float inv = 1.f / l;
        __nv_bfloat16* orow = out + (static_cast<size_t>(bh) * T + t) * D;
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          tmem_ld_x32(tO + cc, o);
          if constexpr (kSplit) {
            uint32_t o2[32];
            tmem_ld_x32(tb + lb + Cfg::kColO2 + cc, o2);
#pragma unroll
            for (int u = 0; u < 32; ++u)
              o[u] = __float_as_uint(__uint_as_float(o[u]) * s0 + __uint_as_float(o2[u]) * s1);
          }
          uint32_t pk[16];
#pragma unroll
          for (int u = 0; u < 16; ++u)
            pk[u] = pack_bf16x2(__uint_as_float(o[2 * u]) * inv, __uint_as_float(o[2 * u + 1]) * inv);
          if (t < T) {
            uint4* dst = reinterpret_cast<uint4*>(orow + cc);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
        }
        if (lse && t < T) lse[static_cast<size_t>(bh) * T + t] = (M + lrow + log2f(l)) * kLn2;
      } else {
        record_timeout(bars, status);
      }
    }
    teardown<kNT>(warp, tb, Cfg::kTmemCols);
  } else {
    regs_dec<kRegsQuery>();
    // ------------------------------------------------------------ running query
    const int q4 = warp - 8;
    const int r = q4 * 32 + lane;
    const uint32_t lb = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tQm = tb + lb + Cfg::kColQm, tQw = tb + lb + Cfg::kColQw;
    if (b > 0) {
      const float4* qrow = reinterpret_cast<const float4*>(
          ql + ((static_cast<size_t>(bh) * Np + b) * kC + r) * D);
      uint32_t qw[D / 2];
#pragma unroll
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t m32[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 f = __ldg(qrow + cc / 4 + u);
          m32[4 * u] = __float_as_uint(f.x);
          m32[4 * u + 1] = __float_as_uint(f.y);
          m32[4 * u + 2] = __float_as_uint(f.z);
          m32[4 * u + 3] = __float_as_uint(f.w);
        }
        if (cc < R) tmem_st_x32(tQm + cc, m32);   // the rest never changes
#pragma unroll
        for (int u = 0; u < 16; ++u)
          qw[cc / 2 + u] = pack_bf16x2(__uint_as_float(m32[2 * u]), __uint_as_float(m32[2 * u + 1]));
      }
#pragma unroll
      for (int cc = 0; cc < D / 2; cc += 32)
        tmem_st_x32(tQw + cc, *reinterpret_cast<uint32_t(*)[32]>(&qw[cc]));
      tmem_st_wait();
      tc_fence_before_sync();
      warp_arrive(&bars->sq_ready);
      bool ok = true;
      for (int n = 0; n + 1 < b; ++n) {
        // Qm (and S) are final for this step once the fused MMA is done
        ok = mbar_wait(&bars->qk_done, n & 1, abort_flag, LIM);
        if (!ok) break;
        tc_fence_after_sync();
        if constexpr (kLR) {
          // Y (kC fp32 columns of this row) -> bf16 into the K-major,
          // 128-byte-swizzled A tile of the second product, 64 columns at a
          // time; then wait for Qm += Y (-UW) before refreshing Qw below
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t y64[64];
            tmem_ld_x64(tb + lb + Cfg::kColY + 64 * hh, y64);
            uint8_t* rowp = s_yw + hh * (kC * 128) + r * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(y64[8 * j]), __uint_as_float(y64[8 * j + 1]));
              v.y = pack_bf16x2(__uint_as_float(y64[8 * j + 2]), __uint_as_float(y64[8 * j + 3]));
              v.z = pack_bf16x2(__uint_as_float(y64[8 * j + 4]), __uint_as_float(y64[8 * j + 5]));
              v.w = pack_bf16x2(__uint_as_float(y64[8 * j + 6]), __uint_as_float(y64[8 * j + 7]));
              *reinterpret_cast<uint4*>(rowp + ((j ^ (r & 7)) << 4)) = v;
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          tc_fence_before_sync();
          warp_arrive(&bars->yw_ready);
          ok = mbar_wait(&bars->q_done, n & 1, abort_flag, LIM);
          if (!ok) break;
          tc_fence_after_sync();
        }
#pragma unroll
        for (int cc = 0; cc < R; cc += 64) {
          uint32_t m64[64];
          tmem_ld_x64(tQm + cc, m64);
#pragma unroll
          for (int u = 0; u < 32; ++u)
            qw[cc / 2 + u] = pack_bf16x2(__uint_as_float(m64[2 * u]), __uint_as_float(m64[2 * u + 1]));
        }
#pragma unroll
        for (int cc = 0; cc < R / 2; cc += 32)
          tmem_st_x32(tQw + cc, *reinterpret_cast<uint32_t(*)[32]>(&qw[cc]));
        tmem_st_wait();
        tc_fence_before_sync();
        warp_arrive(&bars->sq_ready);
      }
      if (!ok) record_timeout(bars, status);
    }
    teardown<kNT>(warp, tb, Cfg::kTmemCols);
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

// Row-major bf16 matrix viewed as [rows][cols] (2D) or [z][rows][cols] (3D),
// 128-byte swizzled boxes of 64 columns x box_rows rows.
bool make_map(CUtensorMap* m, const void* ptr, int rank, uint64_t cols, uint64_t rows,
              uint64_t zdim, uint32_t box_rows) {
  auto enc = encode_fn();
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

template <int D, bool kGate, int R = D, bool kLR = false>
cudaError_t launch_tc(const Geom& g, const Inputs& in, const Workspace& ws, int* status,
                      cudaStream_t st) {
  using Cfg = TcCfg<D, R, kLR>;
  CUtensorMap mkr, mng, mv, muw;
  if (!make_map(&mkr, ws.kr, 2, D, static_cast<uint64_t>(g.BH) * g.Tp, 1, kC) ||
      !make_map(&mv, in.v, 3, D, g.T, g.BH, kC))
    return cudaErrorInvalidValue;
  if constexpr (kLR) {
    // the input directions W ([BH][T][D], rows past T read as zero) and
    // -(U W) per chunk ([nch * kC][D]) from the preparation
    if (!ws.uwn || !make_map(&mng, in.w, 3, D, g.T, g.BH, kC) ||
        !make_map(&muw, ws.uwn, 2, D, static_cast<uint64_t>(g.nch) * kC, 1, kC))
      return cudaErrorInvalidValue;
  } else {
    // ngt_c is read as its first R rows (all D columns); no fourth operand
    if (!make_map(&mng, ws.ngt, 2, D, static_cast<uint64_t>(g.nch) * D, 1, R))
      return cudaErrorInvalidValue;
    muw = mv;
  }
  auto kern = attn_tc_kernel<D, kGate, R, kLR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cfg::kSmemBytes));
  if (e != cudaSuccess) return e;
  kern<<<g.nch, kThreadsOf<D, kLR>, Cfg::kSmemBytes, st>>>(
      mkr, mng, mv, muw, ws.ql, ws.sdt, kGate ? ws.lam2 : nullptr,
      static_cast<__nv_bfloat16*>(in.out), in.lse, status, g.T, g.Np, g.BH, in.scale * kLog2e);
  return cudaGetLastError();
}

// Diagnostics: one thread waits, with the library's bounded wait, on an
// mbarrier that nothing arrives at, and records the expiry like the kernels
// above do.  Used to check the timeout path without faulting the device.
__global__ void debug_wait_kernel(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, nullptr, limit_ns)) atomicExch(status, PATH_DEV_ERR_TIMEOUT);
  }
}

}  // namespace

cudaError_t launch_debug_wait(int* status, unsigned long long limit_ns, cudaStream_t st) {
  debug_wait_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_attn_tc(const Geom& g, const Inputs& in, const Workspace& ws, int* status,
                           cudaStream_t st, int* launches) {
  if (launches) *launches = 1;
  if (g.C != kC) return cudaErrorInvalidValue;
  if (in.wr > 0 && in.wr < g.d) {   // partial PaTH: transitions of rank 64 at d = 128
    if (g.d != 128 || in.wr != 64) return cudaErrorInvalidValue;
    return g.gate ? launch_tc<128, true, 64>(g, in, ws, status, st)
                  : launch_tc<128, false, 64>(g, in, ws, status, st);
  }
  if (g.lowrank) {   // the low-rank transition form, d = 64 only
    if (g.d != 64 || !ws.uwn) return cudaErrorInvalidValue;
    return g.gate ? launch_tc<64, true, 64, true>(g, in, ws, status, st)
                  : launch_tc<64, false, 64, true>(g, in, ws, status, st);
  }
  if (g.d == 128) return g.gate ? launch_tc<128, true>(g, in, ws, status, st)
                                : launch_tc<128, false>(g, in, ws, status, st);
  if (g.d == 64) return g.gate ? launch_tc<64, true>(g, in, ws, status, st)
                               : launch_tc<64, false>(g, in, ws, status, st);
  return cudaErrorInvalidValue;
}

}  // namespace pathattn
