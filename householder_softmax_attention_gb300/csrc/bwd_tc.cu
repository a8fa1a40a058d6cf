// bwd_tc.cu -- the chunk-pair part of the PaTH backward on the sm_103a tensor
// cores (dtype bf16, d = 64 or 128, chunk C = 128).
//
// With the forward's chunk factors (Ql_b, Kr_c, F_c = I + ngt_c, the
// diagonal logits) and, per query chunk b and key chunk c < b, the query
// carried backwards X_b^(c) (X_b^(b-1) = Ql_b, X_b^(c-1) = X_b^(c) F_c^T),
// the logits are S_bc = scale X_b^(c) Kr_c^T (+ gate) ("PaTH Attention ..."
// slides, frames "A triangular representation makes paths computable" and
// "A right-to-left scan accumulates cross-block paths").  Their derivative,
// with dS = P (dP - D), dP = dO V^T, D_i = dO_i . O_i - dlse_i:
//   dV_c     = sum_{b>=c} P_bc^T dO_b
//   dKr_c    = scale sum_{b>c} dS_bc^T X_b^(c)
//   G_b^(c)  = dS_bc Kr_c + G_b^(c-1) F_c   (c = 0 .. b-1),  dQl_b = scale G_b^(b-1)
//   dF_c     = scale sum_{b>c} G_b^(c-1)^T X_b^(c)
// Four kernels, each a tcgen05 pipeline (TMA ring -> one MMA-issuing thread
// -> TMEM accumulators -> warps that convert or apply the softmax):
//   xwalk   per query chunk b: X walked down c = b-1 .. 0 (X += Xw ngt_c^T,
//           fp32 master in TMEM; its bf16 copy Xw, in shared memory, is the
//           A operand and goes out by a TMA store), every X_b^(c) stored
//           (bf16) for the later kernels
//   key     per key chunk c: for b = c (diagonal logits from the
//           preparation) and b = c+1 .. N-1: S^T = Kr_c X_b^T and
//           dP^T = V_c dO_b^T, P and dS on 8 warps, dV += P^T dO_b and
//           dKr += dS^T X_b with P, dS in TMEM; dS_bc stored (bf16) for the
//           G walk, the diagonal's scale dS written in fp32, row and column
//           sums of dS for the gate
//   gwalk   per query chunk b: G walked up c = 0 .. b-1 (G += Gw ngt_c +
//           dS_bc Kr_c, Gw as Xw above), every G_b^(c-1) stored (bf16),
//           dQl_b written
//   dF      per chunk c: dF_c = sum_b G^T X over the stored pairs
// Every mbarrier wait is bounded; on expiry a CTA records a timeout in the
// status word, stops issuing, drains its copies and MMAs and frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>

#include "common.cuh"
#include "ptx.cuh"

namespace pathattn {
namespace {

using bf16 = __nv_bfloat16;
constexpr int kC = 128;
constexpr int kHeadGroup = 8;

__device__ __forceinline__ long long pair_row(int bh, size_t npairs, int b, int c) {
  return (static_cast<long long>(bh) * static_cast<long long>(npairs) +
          static_cast<long long>(b) * (b - 1) / 2 + c) * kC;
}

__device__ __forceinline__ void warp_arrive_one(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

__device__ __forceinline__ void set_timeout(volatile int* abort_flag, int* status) {
  *abort_flag = 1;
  atomicExch(status, PATH_DEV_ERR_TIMEOUT);
}

template <int NT>
__device__ __forceinline__ void teardown_all(int warp, uint32_t tb, uint32_t ncols) {
  tc_fence_before_sync();
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tb, ncols);
  }
}

// Tiles of a walk (one per query chunk b >= 1): heads in groups of
// kHeadGroup, longest walks first inside a group, so that walks of one head
// that run together read the same chunk factors from L2.
__device__ __forceinline__ void walk_tile(int ord, int Np, int BH, int nb, int* b, int* bh) {
  const int per_group = kHeadGroup * nb;
  const int grp = ord / per_group, r = ord - grp * per_group;
  const int heads = min(kHeadGroup, BH - grp * kHeadGroup);
  *b = Np - 1 - r / heads;
  *bh = grp * kHeadGroup + r % heads;
}

// Reads 32 fp32 TMEM columns, packs them as 16 bf16x2 words.
__device__ __forceinline__ void ld_pack32(uint32_t taddr, uint32_t (&pk)[16]) {
  uint32_t v[32];
  tmem_ld_x32(taddr, v);
#pragma unroll
  for (int u = 0; u < 16; ++u) pk[u] = pack_bf16x2(__uint_as_float(v[2 * u]), __uint_as_float(v[2 * u + 1]));
}

__device__ __forceinline__ void st_row16(bf16* dst, const uint32_t (&pk)[16]) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int u = 0; u < 4; ++u) d4[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
}

// ============================================================== X walk
// The bf16 copy of the running query lives in shared memory as a
// 128-byte-swizzled K-major tile: it is the A operand of the next crossing
// and, through a TMA tensor store, the stored X_b^(c).
template <int D>
struct XwCfg {
  static constexpr int kStages = 2;
  static constexpr uint32_t kNgBytes = D * D * 2;
  static constexpr uint32_t kXwBytes = kC * D * 2;
  static constexpr uint32_t kOffXw = kStages * kNgBytes;
  static constexpr uint32_t kTmemCols = D;
  static constexpr size_t kSmemBytes = kOffXw + kXwBytes + 1024 + 256;
};

struct XwBars {
  uint64_t full[2], empty[2];
  uint64_t xw_ready, mma_done, final_done;
  uint32_t tmem_base;
  int abort_flag;
};

// TMA tensor store of a shared-memory box to global (bulk group of the
// issuing thread); coordinates are never negative here.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_addr(src)), "r"(x), "r"(y)
               : "memory");
}

// Barrier of the four converting warps (named barrier 3, 128 threads).
__device__ __forceinline__ void convert_bar() { asm volatile("bar.sync 3, 128;" ::: "memory"); }

// Writes 32 packed bf16 (16 words, columns col0 .. col0 + 31) of row r into a
// swizzled K-major [128][D] tile (64-column halves of 16 KB).
__device__ __forceinline__ void put_row32(uint8_t* tile, int r, int col0, const uint32_t (&pk)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int c8 = (col0 >> 3) + q;
    const uint32_t off = (c8 >> 3) * (kC * 128) + r * 128 + (((c8 & 7) ^ (r & 7)) << 4);
    *reinterpret_cast<uint4*>(tile + off) = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
  }
}

// 192 threads: warp 0 TMA (ngt ring), warp 1 TMEM + MMA issue, warps 2-5
// convert the running query (TMEM lane quarter = warp % 4; warp 2 lane 0
// issues the stores).
template <int D>
__global__ void __launch_bounds__(192, 2)
    bwd_xwalk_tc_kernel(const __grid_constant__ CUtensorMap map_ng,
                        const __grid_constant__ CUtensorMap map_xs, const float* __restrict__ ql,
                        int* __restrict__ status, int Np, int BH, size_t npairs) {
  using Cfg = XwCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* s_ng = base;
  uint8_t* s_xw = base + Cfg::kOffXw;
  XwBars* bars = reinterpret_cast<XwBars*>(base + Cfg::kOffXw + Cfg::kXwBytes);
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int b, bh;
  walk_tile(blockIdx.x, Np, BH, Np - 1, &b, &bh);
  const uint64_t LIM = kWaitLimitNs;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->xw_ready, 1);
    mbar_init(&bars->mma_done, 1);
    mbar_init(&bars->final_done, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_map(&map_ng);
  if (warp == 2 && lane == 0) tma_prefetch_map(&map_xs);
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tb = bars->tmem_base;
  const int ncross = b - 1;  // chunks b-1 .. 1 are crossed

  if (warp == 0) {
    if (lane == 0) {
      int last[Cfg::kStages];
      for (int s = 0; s < Cfg::kStages; ++s) last[s] = -1;
      bool ok = true;
      for (int n = 0; n < ncross && ok; ++n) {
        const int c = b - 1 - n, s = n % Cfg::kStages;
        if (n >= Cfg::kStages)
          ok = mbar_wait(&bars->empty[s], ((n / Cfg::kStages) - 1) & 1, abort_flag, LIM);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars->full[s], Cfg::kNgBytes);
        for (int h = 0; h < D / 64; ++h)
          tma_load_2d(s_ng + s * Cfg::kNgBytes + h * (D * 128), &map_ng, h * 64,
                      (bh * Np + c) * D, &bars->full[s]);
        last[s] = (n / Cfg::kStages) & 1;
      }
      if (!ok) set_timeout(abort_flag, status);
      for (int s = 0; s < Cfg::kStages; ++s)
        if (last[s] >= 0) mbar_wait(&bars->full[s], last[s], nullptr, LIM);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id = idesc_bf16_f32(128, D, false, false);
      const uint32_t tX = tb;
      const uint32_t a0 = smem_addr(s_xw);
      bool ok = true;
      for (int n = 0; n < ncross && ok; ++n) {
        const int s = n % Cfg::kStages;
        ok = mbar_spin(&bars->full[s], (n / Cfg::kStages) & 1, abort_flag, LIM);
        if (ok) ok = mbar_spin(&bars->xw_ready, n & 1, abort_flag, LIM);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t bb = smem_addr(s_ng + s * Cfg::kNgBytes);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t offa = (k >> 2) * (kC * 128) + (k & 3) * 32;
          const uint32_t offb = (k >> 2) * (D * 128) + (k & 3) * 32;
          mma_bf16_ss(tX, sdesc_sw128(a0 + offa, 16, 1024), sdesc_sw128(bb + offb, 16, 1024), id, 1);
        }
        mma_commit(&bars->mma_done);
        mma_commit(&bars->empty[s]);
      }
      if (!ok) set_timeout(abort_flag, status);
      mma_commit(&bars->final_done);
      mbar_wait(&bars->final_done, 0, nullptr, LIM);
    }
  } else {
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const bool leader = warp == 2 && lane == 0;
    const uint32_t lb = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tX = tb + lb;
    // X_b^(b-1) = Ql_b
    {
      const float4* qrow =
          reinterpret_cast<const float4*>(ql + ((static_cast<size_t>(bh) * Np + b) * kC + r) * D);
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
        tmem_st_x32(tX + cc, m32);
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          pk[u] = pack_bf16x2(__uint_as_float(m32[2 * u]), __uint_as_float(m32[2 * u + 1]));
        put_row32(s_xw, r, cc, pk);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before_sync();
      convert_bar();
      if (leader) {
        const int prow = static_cast<int>(pair_row(bh, npairs, b, b - 1));
        for (int h = 0; h < D / 64; ++h) tma_store_2d(&map_xs, h * 64, prow, s_xw + h * (kC * 128));
        bulk_commit();
        mbar_arrive(&bars->xw_ready);
      }
    }
    bool ok = true;
    for (int n = 0; n < ncross; ++n) {
      const int c = b - 1 - n;  // chunk just crossed: X now holds X_b^(c-1)
      ok = mbar_wait(&bars->mma_done, n & 1, abort_flag, LIM);
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t pk[D / 2];
#pragma unroll
      for (int cc = 0; cc < D; cc += 32) ld_pack32(tX + cc, *reinterpret_cast<uint32_t(*)[16]>(&pk[cc / 2]));
      // the previous tile has been read by its store (and by the MMA, done)
      if (leader) bulk_wait_read<0>();
      convert_bar();
#pragma unroll
      for (int cc = 0; cc < D; cc += 32) put_row32(s_xw, r, cc, *reinterpret_cast<uint32_t(*)[16]>(&pk[cc / 2]));
      fence_proxy_async_smem();
      tc_fence_before_sync();
      convert_bar();
      if (leader) {
        const int prow = static_cast<int>(pair_row(bh, npairs, b, c - 1));
        for (int h = 0; h < D / 64; ++h) tma_store_2d(&map_xs, h * 64, prow, s_xw + h * (kC * 128));
        bulk_commit();
        mbar_arrive(&bars->xw_ready);
      }
    }
    if (!ok) set_timeout(abort_flag, status);
    // the stores complete before the CTA (and its shared memory) goes away
    if (leader) bulk_wait<0>();
  }
  teardown_all<192>(warp, tb, Cfg::kTmemCols);
}

// ============================================================== G walk
template <int D>
struct GwCfg {
  static constexpr int kStages = D == 128 ? 2 : 3;
  static constexpr uint32_t kNgBytes = D * D * 2;
  static constexpr uint32_t kDsBytes = kC * kC * 2;
  static constexpr uint32_t kKrBytes = kC * D * 2;
  static constexpr uint32_t kStageBytes = kDsBytes + kKrBytes + kNgBytes;
  static constexpr uint32_t kGwBytes = kC * D * 2;  // bf16 G, swizzled K-major
  static constexpr uint32_t kOffGw = kStages * kStageBytes;
  static constexpr uint32_t kTmemCols = D;
  static constexpr size_t kSmemBytes = kOffGw + kGwBytes + 1024 + 256;
};

struct GwBars {
  uint64_t full[3], empty[3];
  uint64_t gw_ready, mma_done, final_done;
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    bwd_gwalk_tc_kernel(const __grid_constant__ CUtensorMap map_ng,
                        const __grid_constant__ CUtensorMap map_ds,
                        const __grid_constant__ CUtensorMap map_kr,
                        const __grid_constant__ CUtensorMap map_gs, float* __restrict__ dql, int* __restrict__ status, int Np, int BH,
                        size_t npairs, float scale) {
  using Cfg = GwCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int b, bh;
  walk_tile(blockIdx.x, Np, BH, Np, &b, &bh);
  if (b == 0) {  // the first chunk crosses nothing: dQl = 0
    float4* o = reinterpret_cast<float4*>(dql + static_cast<size_t>(bh) * Np * kC * D);
    for (int x = threadIdx.x; x < kC * D / 4; x += blockDim.x) o[x] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* s_gw = base + Cfg::kOffGw;
  GwBars* bars = reinterpret_cast<GwBars*>(base + Cfg::kOffGw + Cfg::kGwBytes);
  volatile int* abort_flag = &bars->abort_flag;
  const int Tp = Np * kC;
  const uint64_t LIM = kWaitLimitNs;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->gw_ready, 1);
    mbar_init(&bars->mma_done, 1);
    mbar_init(&bars->final_done, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&map_ng);
    tma_prefetch_map(&map_ds);
    tma_prefetch_map(&map_kr);
  }
  if (warp == 2 && lane == 0) tma_prefetch_map(&map_gs);
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
      int last[Cfg::kStages];
      for (int s = 0; s < Cfg::kStages; ++s) last[s] = -1;
      bool ok = true;
      for (int c = 0; c < b && ok; ++c) {
        const int s = c % Cfg::kStages;
        if (c >= Cfg::kStages)
          ok = mbar_wait(&bars->empty[s], ((c / Cfg::kStages) - 1) & 1, abort_flag, LIM);
        if (!ok) break;
        uint8_t* st = base + s * Cfg::kStageBytes;
        mbar_arrive_expect_tx(&bars->full[s],
                              Cfg::kDsBytes + Cfg::kKrBytes + (c >= 1 ? Cfg::kNgBytes : 0));
        const int prow = static_cast<int>(pair_row(bh, npairs, b, c));
        for (int h = 0; h < 2; ++h)
          tma_load_2d(st + h * (kC * 128), &map_ds, h * 64, prow, &bars->full[s]);
        for (int h = 0; h < D / 64; ++h)
          tma_load_2d(st + Cfg::kDsBytes + h * (kC * 128), &map_kr, h * 64, bh * Tp + c * kC,
                      &bars->full[s]);
        if (c >= 1)
          for (int h = 0; h < D / 64; ++h)
            tma_load_2d(st + Cfg::kDsBytes + Cfg::kKrBytes + h * (D * 128), &map_ng, h * 64,
                        (bh * Np + c) * D, &bars->full[s]);
        last[s] = (c / Cfg::kStages) & 1;
      }
      if (!ok) set_timeout(abort_flag, status);
      for (int s = 0; s < Cfg::kStages; ++s)
        if (last[s] >= 0) mbar_wait(&bars->full[s], last[s], nullptr, LIM);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // G += dS_bc Kr_c: A = dS (queries x keys) read from the stored
      // [keys][queries] tile (MN-major), B = Kr_c (keys x D, MN-major).
      // G += Gw ngt_c: A = Gw (shared memory, K-major), B = ngt_c ([k][n], MN-major).
      constexpr uint32_t idK = idesc_bf16_f32(128, D, true, true);
      constexpr uint32_t idN = idesc_bf16_f32(128, D, false, true);
      const uint32_t tG = tb, gw = smem_addr(s_gw);
      bool ok = true;
      for (int c = 0; c < b && ok; ++c) {
        const int s = c % Cfg::kStages;
        ok = mbar_spin(&bars->full[s], (c / Cfg::kStages) & 1, abort_flag, LIM);
        // G_b^(c-1) has been read (and Gw written) before anything is added
        if (ok && c >= 1) ok = mbar_spin(&bars->gw_ready, (c - 1) & 1, abort_flag, LIM);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t sa = smem_addr(base + s * Cfg::kStageBytes);
#pragma unroll
        for (int k = 0; k < kC / 16; ++k)
          mma_bf16_ss(tG, sdesc_sw128(sa + k * 2048, kC * 128, 1024),
                      sdesc_sw128(sa + Cfg::kDsBytes + k * 2048, kC * 128, 1024), idK,
                      (c > 0 || k > 0));
        if (c >= 1) {
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_bf16_ss(tG, sdesc_sw128(gw + (k >> 2) * (kC * 128) + (k & 3) * 32, 16, 1024),
                        sdesc_sw128(sa + Cfg::kDsBytes + Cfg::kKrBytes + k * 2048, D * 128, 1024),
                        idN, 1);
        }
        mma_commit(&bars->mma_done);
        mma_commit(&bars->empty[s]);
      }
      if (!ok) set_timeout(abort_flag, status);
      mma_commit(&bars->final_done);
      mbar_wait(&bars->final_done, 0, nullptr, LIM);
    }
  } else {
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const bool leader = warp == 2 && lane == 0;
    const uint32_t lb = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tG = tb + lb;
    bool ok = true;
    for (int c = 0; c < b; ++c) {
      ok = mbar_wait(&bars->mma_done, c & 1, abort_flag, LIM);
      if (!ok) break;
      tc_fence_after_sync();
      if (c + 1 < b) {
        // G_b^(c) -> Gw (next step's A operand) and, by a TMA store, the
        // stored copy for dF; the previous Gw has been read by its store
        uint32_t pk[D / 2];
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) ld_pack32(tG + cc, *reinterpret_cast<uint32_t(*)[16]>(&pk[cc / 2]));
        if (leader) bulk_wait_read<0>();
        convert_bar();
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) put_row32(s_gw, r, cc, *reinterpret_cast<uint32_t(*)[16]>(&pk[cc / 2]));
        fence_proxy_async_smem();
        tc_fence_before_sync();
        convert_bar();
        if (leader) {
          const int prow = static_cast<int>(pair_row(bh, npairs, b, c + 1));
          for (int h = 0; h < D / 64; ++h) tma_store_2d(&map_gs, h * 64, prow, s_gw + h * (kC * 128));
          bulk_commit();
          mbar_arrive(&bars->gw_ready);
        }
      } else {
        float4* orow = reinterpret_cast<float4*>(
            dql + ((static_cast<size_t>(bh) * Np + b) * kC + r) * D);
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t v[32];
          tmem_ld_x32(tG + cc, v);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            orow[cc / 4 + u] = make_float4(scale * __uint_as_float(v[4 * u]),
                                           scale * __uint_as_float(v[4 * u + 1]),
                                           scale * __uint_as_float(v[4 * u + 2]),
                                           scale * __uint_as_float(v[4 * u + 3]));
        }
      }
    }
    if (!ok) set_timeout(abort_flag, status);
    if (leader) bulk_wait<0>();
  }
  teardown_all<192>(warp, tb, Cfg::kTmemCols);
}

// ============================================================== dF
template <int D>
struct DfCfg {
  static constexpr int kStages = D == 128 ? 3 : 4;
  static constexpr uint32_t kTile = kC * D * 2;
  static constexpr uint32_t kStageBytes = 2 * kTile;  // G then X
  static constexpr uint32_t kTmemCols = D;
  static constexpr size_t kSmemBytes = kStages * kStageBytes + 1024 + 256;
};

struct DfBars {
  uint64_t full[4], empty[4];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
};

// dF_c = scale sum_{b>c} G_b^(c-1)^T X_b^(c): A = G^T (features x queries)
// read from the stored [queries][D] tile (MN-major), B = X (queries x D,
// MN-major).  At D = 64 the MMA runs with M = 128: its second row block of A
// is read from the X tile (rows of no use); only lanes 0-63 are read out.
template <int D>
__global__ void __launch_bounds__(192, 1)
    bwd_dF_tc_kernel(const __grid_constant__ CUtensorMap map_gs,
                     const __grid_constant__ CUtensorMap map_xs, float* __restrict__ dF,
                     int* __restrict__ status, int Np, int BH, size_t npairs, float scale) {
  using Cfg = DfCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // chunks c = 1, 2, ... (longest sums first), then c = 0
  const int c = (blockIdx.x / BH + 1) % Np;
  const int bh = blockIdx.x % BH;
  const int steps = c >= 1 ? Np - 1 - c : 0;
  float* out = dF + (static_cast<size_t>(bh) * Np + c) * D * D;
  if (steps == 0) {
    float4* o = reinterpret_cast<float4*>(out);
    for (int x = threadIdx.x; x < D * D / 4; x += blockDim.x) o[x] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  DfBars* bars = reinterpret_cast<DfBars*>(base + Cfg::kStages * Cfg::kStageBytes);
  volatile int* abort_flag = &bars->abort_flag;
  const uint64_t LIM = kWaitLimitNs;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->done, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&map_gs);
    tma_prefetch_map(&map_xs);
  }
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
      int last[Cfg::kStages];
      for (int s = 0; s < Cfg::kStages; ++s) last[s] = -1;
      bool ok = true;
      for (int n = 0; n < steps && ok; ++n) {
        const int bq = c + 1 + n, s = n % Cfg::kStages;
        if (n >= Cfg::kStages)
          ok = mbar_wait(&bars->empty[s], ((n / Cfg::kStages) - 1) & 1, abort_flag, LIM);
        if (!ok) break;
        uint8_t* st = base + s * Cfg::kStageBytes;
        mbar_arrive_expect_tx(&bars->full[s], Cfg::kStageBytes);
        const int prow = static_cast<int>(pair_row(bh, npairs, bq, c));
        for (int h = 0; h < D / 64; ++h) {
          tma_load_2d(st + h * (kC * 128), &map_gs, h * 64, prow, &bars->full[s]);
          tma_load_2d(st + Cfg::kTile + h * (kC * 128), &map_xs, h * 64, prow, &bars->full[s]);
        }
        last[s] = (n / Cfg::kStages) & 1;
      }
      if (!ok) set_timeout(abort_flag, status);
      for (int s = 0; s < Cfg::kStages; ++s)
        if (last[s] >= 0) mbar_wait(&bars->full[s], last[s], nullptr, LIM);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id = idesc_bf16_f32(128, D, true, true);
      constexpr uint32_t lboA = kC * 128;
      bool ok = true;
      for (int n = 0; n < steps && ok; ++n) {
        const int s = n % Cfg::kStages;
        ok = mbar_spin(&bars->full[s], (n / Cfg::kStages) & 1, abort_flag, LIM);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t sa = smem_addr(base + s * Cfg::kStageBytes);
#pragma unroll
        for (int k = 0; k < kC / 16; ++k)
          mma_bf16_ss(tb, sdesc_sw128(sa + k * 2048, lboA, 1024),
                      sdesc_sw128(sa + Cfg::kTile + k * 2048, kC * 128, 1024), id,
                      (n > 0 || k > 0));
        mma_commit(&bars->empty[s]);
      }
      if (!ok) set_timeout(abort_flag, status);
      mma_commit(&bars->done);
      mbar_wait(&bars->done, 0, nullptr, LIM);
    }
  } else {
    const int q4 = warp & 3;
    const int e = q4 * 32 + lane;
    const uint32_t lb = static_cast<uint32_t>(q4 * 32) << 16;
    const bool ok = mbar_wait(&bars->done, 0, abort_flag, LIM);
    if (ok) {
      tc_fence_after_sync();
      if (q4 * 32 < D) {
        float4* orow = reinterpret_cast<float4*>(out + static_cast<size_t>(e) * D);
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t v[32];
          tmem_ld_x32(tb + lb + cc, v);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            orow[cc / 4 + u] = make_float4(scale * __uint_as_float(v[4 * u]),
                                           scale * __uint_as_float(v[4 * u + 1]),
                                           scale * __uint_as_float(v[4 * u + 2]),
                                           scale * __uint_as_float(v[4 * u + 3]));
        }
      }
    } else {
      set_timeout(abort_flag, status);
    }
  }
  teardown_all<192>(warp, tb, Cfg::kTmemCols);
}

// ============================================================== key pass
template <int D>
struct KeyCfg {
  static constexpr uint32_t kTile = kC * D * 2;          // [C][D] bf16
  static constexpr uint32_t kStageBytes = 2 * kTile;     // dO_b, X_b
  static constexpr uint32_t kVecBytes = kC * 4;          // one fp32 vector per query
  static constexpr uint32_t kOffKr = 0, kOffV = kTile, kOffStage = 2 * kTile;
  static constexpr uint32_t kOffVec = kOffStage + 2 * kStageBytes;  // [2][3][C] f32
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr size_t kSmemBytes = kOffVec + 2 * 3 * kVecBytes + 1024 + 1024;
};

struct KeyBars {
  uint64_t kv_full, full[2], empty[2];
  uint64_t s_full, dp_full, p_ready, ds_ready, p_consumed, ds_consumed, acc_done, final_done;
  uint32_t tmem_base;
  int abort_flag;
  float colpart[kC];
};

constexpr int kKeyThreads = 384;
constexpr int kKeyRegsLow = 56, kKeyRegsEw = 224;
static_assert(128 * kKeyRegsLow + 256 * kKeyRegsEw <= kKeyThreads * 168, "register split");

// 384 threads: warp 0 TMA, warp 1 TMEM + MMA issue, warps 2-3 idle, warps
// 4-7 and 8-11 the elementwise groups (queries 0-63 and 64-127 of the key
// row held by TMEM lane warp % 4 * 32 + lane).
template <int D, bool kGate>
__global__ void __launch_bounds__(kKeyThreads, 1)
    bwd_key_tc_kernel(const __grid_constant__ CUtensorMap map_kr,
                      const __grid_constant__ CUtensorMap map_v,
                      const __grid_constant__ CUtensorMap map_do,
                      const __grid_constant__ CUtensorMap map_xs, const float* __restrict__ sdt,
                      const float* __restrict__ lse2, const float* __restrict__ dvec,
                      const float* __restrict__ lam2, bf16* __restrict__ dsbuf,
                      float* __restrict__ dad, bf16* __restrict__ dv, float* __restrict__ dkr,
                      float* __restrict__ colsum, float* __restrict__ rowsum,
                      int* __restrict__ status, int T, int Np, int BH, size_t npairs,
                      float scale, float sl2) {
  using Cfg = KeyCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  KeyBars* bars = reinterpret_cast<KeyBars*>(base + Cfg::kOffVec + 2 * 3 * Cfg::kVecBytes);
  float* svec = reinterpret_cast<float*>(base + Cfg::kOffVec);  // [stage][lse2, dvec, lam2][C]
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // key chunks: heads in groups, the longest (smallest c) first in a group
  int c, bh;
  {
    const int per_group = kHeadGroup * Np;
    const int grp = blockIdx.x / per_group, r = blockIdx.x - grp * per_group;
    const int heads = min(kHeadGroup, BH - grp * kHeadGroup);
    c = r / heads;
    bh = grp * kHeadGroup + r % heads;
  }
  const int Tp = Np * kC;
  const int nsteps = Np - c;  // b = c (diagonal), c + 1, ..., Np - 1
  const uint64_t LIM = kWaitLimitNs;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_ready, 8);
    mbar_init(&bars->ds_ready, 8);
    mbar_init(&bars->p_consumed, 1);
    mbar_init(&bars->ds_consumed, 1);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->final_done, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&map_kr);
    tma_prefetch_map(&map_v);
    tma_prefetch_map(&map_do);
    tma_prefetch_map(&map_xs);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tb = bars->tmem_base;

  if (warp < 4) {
    regs_dec<kKeyRegsLow>();
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------ producer
      bool kv_issued = false;
      int last[2] = {-1, -1};
      bool ok = true;
      mbar_arrive_expect_tx(&bars->kv_full, 2 * Cfg::kTile);
      for (int h = 0; h < D / 64; ++h) {
        tma_load_2d(base + Cfg::kOffKr + h * (kC * 128), &map_kr, h * 64, bh * Tp + c * kC,
                    &bars->kv_full);
        tma_load_3d(base + Cfg::kOffV + h * (kC * 128), &map_v, h * 64, c * kC, bh,
                    &bars->kv_full);
      }
      kv_issued = true;
      for (int n = 0; n < nsteps && ok; ++n) {
        const int b = c + n, s = n & 1;
        if (n >= 2) ok = mbar_wait(&bars->empty[s], ((n >> 1) - 1) & 1, abort_flag, LIM);
        if (!ok) break;
        uint8_t* st = base + Cfg::kOffStage + s * Cfg::kStageBytes;
        float* vs = svec + s * 3 * kC;
        const uint32_t bytes = Cfg::kTile + (n >= 1 ? Cfg::kTile : 0) +
                               (kGate ? 3 : 2) * Cfg::kVecBytes;
        mbar_arrive_expect_tx(&bars->full[s], bytes);
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(st + h * (kC * 128), &map_do, h * 64, b * kC, bh, &bars->full[s]);
        if (n >= 1) {
          const int prow = static_cast<int>(pair_row(bh, npairs, b, c));
          for (int h = 0; h < D / 64; ++h)
            tma_load_2d(st + Cfg::kTile + h * (kC * 128), &map_xs, h * 64, prow, &bars->full[s]);
        }
        const size_t vo = static_cast<size_t>(bh) * Tp + static_cast<size_t>(b) * kC;
        bulk_load(vs, lse2 + vo, Cfg::kVecBytes, &bars->full[s]);
        bulk_load(vs + kC, dvec + vo, Cfg::kVecBytes, &bars->full[s]);
        if (kGate) bulk_load(vs + 2 * kC, lam2 + vo, Cfg::kVecBytes, &bars->full[s]);
        last[s] = (n >> 1) & 1;
      }
      if (!ok) set_timeout(abort_flag, status);
      if (kv_issued) mbar_wait(&bars->kv_full, 0, nullptr, LIM);
      for (int s = 0; s < 2; ++s)
        if (last[s] >= 0) mbar_wait(&bars->full[s], last[s], nullptr, LIM);
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------------------ MMA issue
      constexpr uint32_t idSS = idesc_bf16_f32(128, kC, false, false);  // S^T, dP^T
      constexpr uint32_t idAcc = idesc_bf16_f32(128, D, false, true);   // dV, dKr
      const uint32_t tS = tb + Cfg::kColS, tDP = tb + Cfg::kColDP;
      const uint32_t tDV = tb + Cfg::kColDV, tDK = tb + Cfg::kColDK;
      const uint32_t sKr = smem_addr(base + Cfg::kOffKr), sV = smem_addr(base + Cfg::kOffV);
      bool ok = mbar_spin(&bars->kv_full, 0, abort_flag, LIM);
      for (int n = 0; n < nsteps && ok; ++n) {
        const int s = n & 1;
        const uint32_t sDO = smem_addr(base + Cfg::kOffStage + s * Cfg::kStageBytes);
        const uint32_t sX = sDO + Cfg::kTile;
        ok = mbar_spin(&bars->full[s], (n >> 1) & 1, abort_flag, LIM);
        if (!ok) break;
        // Per step the pipe runs S^T, dP^T, dV, dKr back to back: P is made
        // from S while dP^T is computed, dS from dP while dV accumulates.
        if (n >= 1) {
          // S^T = Kr_c X_b^T once P of the previous step has been consumed
          ok = mbar_spin(&bars->p_consumed, (n - 1) & 1, abort_flag, LIM);
          if (!ok) break;
          tc_fence_after_sync();
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * (kC * 128) + (k & 3) * 32;
            mma_bf16_ss(tS, sdesc_sw128(sKr + off, 16, 1024), sdesc_sw128(sX + off, 16, 1024),
                        idSS, k > 0);
          }
        }
        mma_commit(&bars->s_full);
        if (n >= 1) {
          ok = mbar_spin(&bars->ds_consumed, (n - 1) & 1, abort_flag, LIM);
          if (!ok) break;
        }
        tc_fence_after_sync();
        // dP^T = V_c dO_b^T
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * (kC * 128) + (k & 3) * 32;
          mma_bf16_ss(tDP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO + off, 16, 1024),
                      idSS, k > 0);
        }
        mma_commit(&bars->dp_full);
        ok = mbar_spin(&bars->p_ready, n & 1, abort_flag, LIM);
        if (!ok) break;
        tc_fence_after_sync();
        // dV += P^T dO_b (P^T in TMEM: queries 0-63 at columns 0-31, 64-127 at 64-95)
#pragma unroll
        for (int k = 0; k < kC / 16; ++k)
          mma_bf16_ts(tDV, tS + (k >> 2) * 64 + (k & 3) * 8,
                      sdesc_sw128(sDO + k * 2048, kC * 128, 1024), idAcc, (n > 0 || k > 0));
        mma_commit(&bars->p_consumed);
        ok = mbar_spin(&bars->ds_ready, n & 1, abort_flag, LIM);
        if (!ok) break;
        tc_fence_after_sync();
        if (n >= 1) {
          // dKr += dS^T X_b
#pragma unroll
          for (int k = 0; k < kC / 16; ++k)
            mma_bf16_ts(tDK, tDP + (k >> 2) * 64 + (k & 3) * 8,
                        sdesc_sw128(sX + k * 2048, kC * 128, 1024), idAcc, (n > 1 || k > 0));
        }
        mma_commit(&bars->ds_consumed);
        mma_commit(&bars->empty[s]);
      }
      if (!ok) set_timeout(abort_flag, status);
      mma_commit(&bars->acc_done);
      mma_commit(&bars->final_done);
      mbar_wait(&bars->final_done, 0, nullptr, LIM);
    }
    // the register-split warpgroups do not rejoin: each has its own teardown
    teardown_all<kKeyThreads>(warp, tb, Cfg::kTmemCols);
  } else {
    regs_inc<kKeyRegsEw>();
    // ------------------------------------------------------------ elementwise
    const int g = (warp - 4) >> 2;  // query half
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;    // key row
    const int tk = c * kC + r;       // key token
    const uint32_t lb = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tS = tb + lb + Cfg::kColS + 64 * g, tDP = tb + lb + Cfg::kColDP + 64 * g;
    const size_t ch = static_cast<size_t>(bh) * Np + c;
    const float lamk = kGate ? lam2[static_cast<size_t>(bh) * Tp + tk] : 0.f;
    float csum = 0.f;
    bool ok = true;
    for (int n = 0; n < nsteps; ++n) {
      const int b = c + n, s = n & 1;
      const float* vs = svec + s * 3 * kC + 64 * g;
      uint32_t sv[64];
      if (n == 0) {
        const float4* srow = reinterpret_cast<const float4*>(sdt + (ch * kC + r) * kC + 64 * g);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float4 f = __ldg(srow + u);
          sv[4 * u] = __float_as_uint(f.x);
          sv[4 * u + 1] = __float_as_uint(f.y);
          sv[4 * u + 2] = __float_as_uint(f.z);
          sv[4 * u + 3] = __float_as_uint(f.w);
        }
      }
      // the stage's vectors (bulk copies) are read here: observe their barrier
      ok = mbar_wait(&bars->full[s], (n >> 1) & 1, abort_flag, LIM);
      if (ok) ok = mbar_wait(&bars->s_full, n & 1, abort_flag, LIM);
      if (!ok) break;
      tc_fence_after_sync();
      if (n >= 1) tmem_ld_x64(tS, sv);
      const int qlim = T - b * kC - 64 * g;  // columns j < qlim are real queries
      // P (kept in sv as fp32 bits) and its bf16 copy over S
      {
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          float x;
          if (n == 0) {
            x = __uint_as_float(sv[j]) - vs[j];
          } else if (kGate) {
            x = fmaf(__uint_as_float(sv[j]), sl2, vs[2 * kC + j] - lamk - vs[j]);
          } else {
            x = fmaf(__uint_as_float(sv[j]), sl2, -vs[j]);
          }
          float p = ex2_approx(x);
          if (j >= qlim) p = 0.f;
          sv[j] = __float_as_uint(p);
        }
#pragma unroll
        for (int u = 0; u < 32; ++u) pk[u] = pack_bf16x2(__uint_as_float(sv[2 * u]), __uint_as_float(sv[2 * u + 1]));
        tmem_st_x32(tS, pk);
        tmem_st_wait();
        tc_fence_before_sync();
        warp_arrive_one(&bars->p_ready);
      }
      // dS = P (dP - D) and its bf16 copy over dP
      ok = mbar_wait(&bars->dp_full, n & 1, abort_flag, LIM);
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t dp[64], dk[32];
      tmem_ld_x64(tDP, dp);
      float ds[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const float d = __uint_as_float(sv[j]) * (__uint_as_float(dp[j]) - vs[kC + j]);
        ds[j] = d;
        csum += d;
      }
#pragma unroll
      for (int u = 0; u < 32; ++u) dk[u] = pack_bf16x2(ds[2 * u], ds[2 * u + 1]);
      tmem_st_x32(tDP, dk);
      tmem_st_wait();
      tc_fence_before_sync();
      warp_arrive_one(&bars->ds_ready);
      if (n >= 1) {
        uint4* drow = reinterpret_cast<uint4*>(
            dsbuf + (pair_row(bh, npairs, b, c) + r) * kC + 64 * g);
#pragma unroll
        for (int u = 0; u < 8; ++u) drow[u] = make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
      } else {
        float* dcol = dad + ch * kC * kC + static_cast<size_t>(64 * g) * kC + r;
#pragma unroll
        for (int j = 0; j < 64; ++j) dcol[static_cast<size_t>(j) * kC] = scale * ds[j];
      }
      if (kGate) {
        // column sums over this warp's 32 key rows (row sums of dS, for the
        // gate): five rounds, each keeping half of the held columns and adding
        // the partner lane's copy of them; lane l ends with columns 2l, 2l + 1
#pragma unroll
        for (int w = 32, m = 16; w >= 2; w >>= 1, m >>= 1) {
          const bool hi = (lane & m) != 0;
#pragma unroll
          for (int i = 0; i < w; ++i) {
            const float keep = hi ? ds[w + i] : ds[i];
            const float give = hi ? ds[i] : ds[w + i];
            ds[i] = keep + __shfl_xor_sync(0xffffffffu, give, m);
          }
        }
        float* rs = rowsum + static_cast<size_t>(bh) * Tp + static_cast<size_t>(b) * kC + 64 * g;
        atomicAdd(rs + 2 * lane, ds[0]);
        atomicAdd(rs + 2 * lane + 1, ds[1]);
      }
    }
    // epilogue: dV (group 0) and dKr (group 1) rows of key r; column sums of dS
    if (ok) ok = mbar_wait(&bars->acc_done, 0, abort_flag, LIM);
    if (ok) {
      tc_fence_after_sync();
      if (g == 0) {
        // tcgen05.ld is warp-collective: every lane loads, real keys store
        bf16* orow = dv + (static_cast<size_t>(bh) * T + min(tk, T - 1)) * D;
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t pk[16];
          ld_pack32(tb + lb + Cfg::kColDV + cc, pk);
          if (tk < T) st_row16(orow + cc, pk);
        }
      } else {
        float4* orow = reinterpret_cast<float4*>(dkr + (ch * kC + r) * D);
        if (nsteps > 1) {
#pragma unroll
          for (int cc = 0; cc < D; cc += 32) {
            uint32_t v[32];
            tmem_ld_x32(tb + lb + Cfg::kColDK + cc, v);
#pragma unroll
            for (int u = 0; u < 8; ++u)
              orow[cc / 4 + u] = make_float4(scale * __uint_as_float(v[4 * u]),
                                             scale * __uint_as_float(v[4 * u + 1]),
                                             scale * __uint_as_float(v[4 * u + 2]),
                                             scale * __uint_as_float(v[4 * u + 3]));
          }
        } else {
#pragma unroll
          for (int u = 0; u < D / 4; ++u) orow[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        bars->colpart[r] = csum;
      }
    } else {
      set_timeout(abort_flag, status);
    }
    // both groups meet (named barrier 2, the 256 elementwise threads)
    asm volatile("bar.sync 2, 256;" ::: "memory");
    if (ok && g == 0) colsum[static_cast<size_t>(bh) * Tp + tk] = csum + bars->colpart[r];
    teardown_all<kKeyThreads>(warp, tb, Cfg::kTmemCols);
  }
}

// ============================================================== launch
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

// Row-major bf16 [rows][cols] (2D) or [z][rows][cols] (3D), 128-byte
// swizzled boxes of 64 columns x box_rows rows (rows past the end read zero).
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

template <typename K>
cudaError_t set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

template <int D, bool kGate>
cudaError_t launch_pairs_tc(const BwdParams& p, int* status, cudaStream_t st) {
  const uint64_t prow = static_cast<uint64_t>(p.BH) * p.npairs * kC;
  CUtensorMap mkr, mng, mv, mdo, mxs, mgs, mds;
  if (!make_map(&mkr, p.kr, 2, D, static_cast<uint64_t>(p.BH) * p.Tp, 1, kC) ||
      !make_map(&mng, p.ngt, 2, D, static_cast<uint64_t>(p.nch) * D, 1, D) ||
      !make_map(&mv, p.v, 3, D, p.T, p.BH, kC) || !make_map(&mdo, p.dout, 3, D, p.T, p.BH, kC))
    return cudaErrorInvalidValue;
  const bool pairs = p.Np >= 2;
  if (pairs && (!make_map(&mxs, p.xs, 2, D, prow, 1, kC) ||
                !make_map(&mgs, p.gs, 2, D, prow, 1, kC) ||
                !make_map(&mds, p.ds, 2, kC, prow, 1, kC)))
    return cudaErrorInvalidValue;
  if (!pairs) mxs = mgs = mds = mkr;  // never dereferenced: no chunk pairs
  cudaError_t e;
  if (pairs) {
    auto kx = bwd_xwalk_tc_kernel<D>;
    if ((e = set_smem(kx, XwCfg<D>::kSmemBytes)) != cudaSuccess) return e;
    kx<<<p.BH * (p.Np - 1), 192, XwCfg<D>::kSmemBytes, st>>>(mng, mxs, p.ql, status, p.Np, p.BH,
                                                              p.npairs);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  bwd_mark(p.ev, kBwdEvKey, st);
  if (kGate) {
    if ((e = cudaMemsetAsync(p.rowsum, 0, static_cast<size_t>(p.BH) * p.Tp * 4, st)) != cudaSuccess)
      return e;
  }
  auto kk = bwd_key_tc_kernel<D, kGate>;
  if ((e = set_smem(kk, KeyCfg<D>::kSmemBytes)) != cudaSuccess) return e;
  kk<<<p.nch, kKeyThreads, KeyCfg<D>::kSmemBytes, st>>>(
      mkr, mv, mdo, mxs, p.sdt, p.lse2, p.dvec, p.lam2, static_cast<bf16*>(p.ds), p.dad,
      static_cast<bf16*>(p.dv), p.dkr, p.colsum, p.rowsum, status, p.T, p.Np, p.BH, p.npairs,
      p.scale, p.scale_log2e);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bwd_mark(p.ev, kBwdEvGwalk, st);
  auto kg = bwd_gwalk_tc_kernel<D>;
  if ((e = set_smem(kg, GwCfg<D>::kSmemBytes)) != cudaSuccess) return e;
  kg<<<p.nch, 192, GwCfg<D>::kSmemBytes, st>>>(mng, mds, mkr, mgs, p.dql, status, p.Np, p.BH,
                                                p.npairs, p.scale);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bwd_mark(p.ev, kBwdEvDf, st);
  auto kf = bwd_dF_tc_kernel<D>;
  if ((e = set_smem(kf, DfCfg<D>::kSmemBytes)) != cudaSuccess) return e;
  kf<<<p.nch, 192, DfCfg<D>::kSmemBytes, st>>>(mgs, mxs, p.dF, status, p.Np, p.BH, p.npairs,
                                                p.scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pairs_tc(const BwdParams& p, int* status, cudaStream_t st) {
  if (!p.bf16 || p.C != kC) return cudaErrorInvalidValue;
  if (static_cast<long long>(p.BH) * static_cast<long long>(p.npairs) * kC >= INT_MAX ||
      static_cast<long long>(p.BH) * p.Tp >= INT_MAX)
    return cudaErrorInvalidValue;
  const bool gate = p.lam2 != nullptr;
  if (p.d == 128) return gate ? launch_pairs_tc<128, true>(p, status, st)
                              : launch_pairs_tc<128, false>(p, status, st);
  if (p.d == 64) return gate ? launch_pairs_tc<64, true>(p, status, st)
                             : launch_pairs_tc<64, false>(p, status, st);
  return cudaErrorInvalidValue;
}

}  // namespace pathattn
