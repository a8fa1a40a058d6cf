// common.cuh -- definitions shared by the PaTH forward kernels and the C ABI:
// problem geometry, the workspace layout, device status codes and the
// host-side launchers of each kernel family.
#pragma once
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace pathattn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device status word values (stored in a per-device int; 0 = fine).
constexpr int PATH_DEV_OK = 0;
constexpr int PATH_DEV_ERR_TIMEOUT = 1;
constexpr int PATH_DEV_ERR_BAD_POS = 2;  // a decoding position outside its bounds

// Time limit of every bounded wait inside the kernels.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

// Problem geometry.  Tokens are grouped into chunks of C; the last chunk is
// padded with beta = 0 tokens (H = I), which leaves every real logit as is.
struct Geom {
  int B, H, T, d, C;
  int BH;       // B * H
  int Np;       // chunks per head, ceil(T / C)
  int Tp;       // Np * C
  int nch;      // BH * Np
  bool bf16;    // element type of q, k, v, w, out (else fp32)
  bool gate;    // PaTH-FoX gate present
  // the low-rank transition form (bf16, d = 64): crossing chunk c as
  // q <- q + (q W_c^T)(-(U W)_c) instead of q <- q + q ngt_c^T
  bool lowrank = false;
};

// Workspace: every region 256-byte aligned.  Per chunk ch = bh * Np + n:
//   kr   [ch][C][d]   elem  boundary-adjusted keys (k_j through H_{j+1}..H_last)
//   ql   [ch][C][d]   f32   boundary-adjusted queries (q_i through H_i..H_first)
//   ngt  [ch][d][d]   elem  -(W^T U W)^T, so q_next = q + q ngt^T
//   sdt  [ch][C][C]   f32   intra-chunk log2-domain logits, [j][i], -inf for j > i
//   lam2 [bh][Tp]     f32   log2(e) * inclusive cumsum of log f (gate only)
//   uwn  [ch][C][d]   elem  -(U W), the low-rank transition form only
// and, for fp32 inputs only, the scratch of the SIMT preparation kernels:
//   lmat [ch][C][C] f32   strictLower(diag(beta) W W^T), then U
//   awk  [ch][C][C] f32   strictLower(W K^T)
//   aqw  [ch][C][C] f32   lower(Q W^T)
//   aqk  [ch][C][C] f32   lower(Q K^T)
//   tk   [ch][C][C] f32   U strictLower(W K^T)
//   uw   [ch][C][d] f32   U W
struct Workspace {
  void* kr;
  float* ql;
  void* ngt;
  float* sdt;
  float* lam2;
  void* uwn;
  float *lmat, *awk, *aqw, *aqk, *tk, *uw;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Lays out the workspace over `base` (may be null to only count bytes).
inline size_t workspace_layout(const Geom& g, char* base, Workspace* ws) {
  const size_t es = g.bf16 ? 2 : 4;
  const size_t nch = static_cast<size_t>(g.nch);
  const size_t C = g.C, d = g.d;
  size_t off = 0;
  auto take = [&](size_t bytes) -> char* {
    char* p = base ? base + off : nullptr;
    off = align_up(off + bytes, 256);
    return p;
  };
  Workspace w{};
  w.kr = take(nch * C * d * es);
  w.ql = reinterpret_cast<float*>(take(nch * C * d * 4));
  w.ngt = take(nch * d * d * es);
  w.sdt = reinterpret_cast<float*>(take(nch * C * C * 4));
  w.lam2 = g.gate ? reinterpret_cast<float*>(take(static_cast<size_t>(g.BH) * g.Tp * 4)) : nullptr;
  w.uwn = g.lowrank ? take(nch * C * d * es) : nullptr;
  if (g.bf16) {  // the fused tensor-core preparation keeps its intermediates on chip
    w.lmat = w.awk = w.aqw = w.aqk = w.tk = w.uw = nullptr;
    if (ws) *ws = w;
    return off;
  }
  w.lmat = reinterpret_cast<float*>(take(nch * C * C * 4));
  w.awk = reinterpret_cast<float*>(take(nch * C * C * 4));
  w.aqw = reinterpret_cast<float*>(take(nch * C * C * 4));
  w.aqk = reinterpret_cast<float*>(take(nch * C * C * 4));
  w.tk = reinterpret_cast<float*>(take(nch * C * C * 4));
  w.uw = reinterpret_cast<float*>(take(nch * C * d * 4));
  if (ws) *ws = w;
  return off;
}

struct Inputs {
  const void *q, *k, *v, *w;
  const float *beta, *logf;
  float scale;
  void* out;
  float* lse;
  // columns of w: 0 = d.  Partial PaTH (bf16) passes its u [B,H,T,r] as w
  // with wr = r; the preparation reads it with zeros in columns r .. d-1 and
  // the attention carries only the first r coordinates through transitions.
  int wr = 0;
};

// Kernel-family launchers (each returns the first launch error, if any).
// Chunk preparation: fills kr, ql, ngt, sdt (and lam2 when gated); bf16 runs
// one fused tcgen05 kernel per chunk, fp32 the SIMT kernels.
cudaError_t launch_prep(const Geom& g, const Inputs& in, const Workspace& ws, int* dev_status,
                        cudaStream_t st, int* launches);
// bf16, d = 64 or 128: the tcgen05 preparation (bounded waits report into dev_status)
cudaError_t launch_prep_tc(const Geom& g, const Inputs& in, const Workspace& ws, int* dev_status,
                           cudaStream_t st);
// fp32 attention over the prepared chunks (SIMT, fp32 throughout).
cudaError_t launch_attn_f32(const Geom& g, const Inputs& in, const Workspace& ws,
                            cudaStream_t st, int* launches);
// bf16 attention over the prepared chunks (tcgen05 / TMEM / TMA).
cudaError_t launch_attn_tc(const Geom& g, const Inputs& in, const Workspace& ws,
                           int* dev_status, cudaStream_t st, int* launches);
// Decoding over a key cache rewritten in place (decode.cu).  Per head bh:
//   q, k, v, w [bh][d] elem; beta, logf [bh] f32 (logf may be null)
//   kcache [bh][Tmax][d] f32; vcache [bh][Tmax][d] elem; lamcache [bh][Tmax] f32
//   pos [B] int32: position of the new token of each batch row
//   part [bh][nsplit][d + 2] f32 scratch: (max, sum, o) of each key span
// One launch; the last CTA of each head to finish merges its spans.
struct DecodeParams {
  const void *q, *k, *v, *w;
  const float *beta, *logf;
  float scale;
  float* kcache;
  void* vcache;
  float* lamcache;
  const int* pos;
  int H, Tmax, max_len;
  int nsplit, span;  // spans of `span` cached keys (a multiple of the tile)
  float* part;
  int* counters;  // [bh], zero before the launch: CTAs of the head that have finished
  void* out;
  float* lse;
  int* status;
};
// Key rows per pipeline stage of the decoding kernel (spans are multiples).
int decode_tile_keys(int d);
// One launch of the span kernel (counters must be zero).
cudaError_t launch_decode(const DecodeParams& p, int BH, int d, bool bf16, cudaStream_t st);
// Prefill: kcache rows j < T of each head <- key j carried to token T - 1,
// from the chunk factors kr and ngt of a prepared workspace.
cudaError_t launch_align_keys(const Geom& g, const Workspace& ws, float* kcache, int Tmax,
                              cudaStream_t st);
// w / beta producer (producer.cu): the projection, then the mixing step;
// the workspace holds `low` [B*T][R] (fp32 at most) and, for the tcgen05
// mixing kernel, the folded weights (producer_mix_tc.cu).
size_t producer_workspace_bytes(int B, int T, int R, int H, int d);
cudaError_t launch_producer(const void* x, const void* Wd, const void* Wu, const float* cw,
                            const void* Ub, const float* bb, void* w, float* beta, void* ws,
                            int* status, int B, int T, int Dm, int H, int d, int R, bool bf16_in,
                            cudaStream_t st);
// bf16 mixing on tcgen05 with the convolution folded into the weights (R = 64).
bool producer_mix_tc_supported(int B, int T, int H, int d, int R);
size_t producer_fold_bytes(int H, int d);
cudaError_t launch_producer_mix_tc(const void* low, const void* Wu, const float* cw, void* bf,
                                   void* w, int* status, int B, int T, int H, int d,
                                   cudaStream_t st);
// bf16 producer projection on tcgen05 (producer_tc.cu); `low` is [B*T][R] bf16.
cudaError_t launch_producer_proj_tc(const void* x, const void* Wd, const void* Ub,
                                    const float* bb, void* low, float* beta, int* status, int B,
                                    int T, int Dm, int H, int R, cudaStream_t st);
// Gate prefix: out[bh * out_stride + t] = mult * sum_{s<=t} logf[bh][s] for
// t < n_out (tokens at or past T add 0).
cudaError_t launch_gate_prefix(const float* logf, float* out, int BH, int T, int n_out,
                               size_t out_stride, double mult, cudaStream_t st);
// Backward pass (bwd.cu).  Geometry and pointers of one call; the forward
// preparation's workspace (kr, ql, ngt, sdt, lam2) comes first, then, from
// bwd_workspace_layout:
//   dvec, lse2, colsum, rowsum [bh][Tp] f32   D_i = dO_i . O_i - dlse_i,
//                                     lse log2(e), column and row sums of dS
//   xs, gs [bh][pair][C][d] elem      X_b^(c) and G_b^(c-1) of every chunk pair
//                                     c < b, pair = b (b - 1) / 2 + c
//   ds [bh][pair][C][C] bf16          dS_bc^T, [key][query] (bf16 inputs only)
//   dql, dkr [ch][C][d] f32           gradients of the boundary-adjusted queries / keys
//   dF [ch][d][d] f32                 gradient of the chunk transition F_c
//   dad [ch][C][C] f32                scale lower(dS_cc), [i][j]
struct BwdParams {
  const void *q, *k, *v, *w, *out, *dout;
  const float *beta, *lse, *dlse;
  float scale, scale_log2e;
  void *dq, *dk, *dv, *dw;
  float *dbeta, *dlogf;
  // forward preparation
  const void* kr;
  const float* ql;
  const void* ngt;
  const float* sdt;
  const float* lam2;
  // backward scratch
  float *dvec, *lse2, *colsum, *rowsum;
  void *xs, *gs, *ds;
  float *dql, *dkr, *dF, *dad;
  int* status;  // device status word (bounded waits of the tensor-core kernels)
  // optional timing: events recorded on the stream at the phase boundaries
  // (index kBwdEv* below), null when timing is off
  cudaEvent_t* ev;
  size_t npairs;
  int BH, T, Tp, Np, C, d, nch;
  bool bf16;
};
// Phase boundaries of one backward call (events 0 .. kBwdPhases):
// prep | rowdot | X walk | key pass | G walk | dF | chunk pass and gate.
constexpr int kBwdPhases = 7;
enum { kBwdEvPrep = 0, kBwdEvRowdot, kBwdEvXwalk, kBwdEvKey, kBwdEvGwalk, kBwdEvDf, kBwdEvChunk,
       kBwdEvEnd };
inline void bwd_mark(const cudaEvent_t* ev, int i, cudaStream_t st) {
  if (ev) cudaEventRecord(ev[i], st);
}
// fp32 scratch of the chunk pass ([ch][C][d] or [ch][C][C] or [ch][C]).
struct ChunkBufs {
  float *Wf, *Kf, *Qf, *UW, *dUW, *P1, *P2, *dQf, *dKf, *dWf;
  float *GWW, *Lm, *Xi, *U, *Nm, *TK, *Mm, *dM, *dTK, *dN, *dU, *dXi, *T1, *dLm, *BL;
  float *bf, *dbf;
};
// Lays out the backward scratch over `base` (null: count bytes only); the
// geometry and scratch pointers go to *p, the chunk-pass buffers to *cb.
size_t bwd_workspace_layout(const Geom& g, char* base, BwdParams* p, ChunkBufs* cb);
cudaError_t launch_bwd(const BwdParams& p, const ChunkBufs& cb, cudaStream_t st);
// bf16, d = 64 or 128, C = 128: the chunk-pair kernels on tcgen05 (bwd_tc.cu):
// fills xs, gs, ds, dql, dkr, dF, dad, dv, colsum, rowsum from dvec and lse2.
cudaError_t launch_bwd_pairs_tc(const BwdParams& p, int* status, cudaStream_t st);
// Batched C[z] = mask(sum_t alpha_t op(A_t[z]) op(B_t[z]) + Add[z]) for the
// backward's chunk pass on tcgen05 (bwd_gemm_tc.cu): fp32 row-major operands
// split into bf16 hi + lo, M = 128, N and every K_t in {64, 128}; op(X) = X^T
// when tX.  Add may be null (nothing added) or alias Cm.  mask 0: none,
// 1: keep n <= m, 2: keep n < m (others written as 0).
constexpr int kMaxTerms = 8;
struct TcTerm {
  const float* A;
  const float* B;
  long long sA, sB;
  int lda, ldb, K;
  bool tA, tB;
  float alpha;
  // operand stored as bf16 (pointer reinterpreted, leading dimension in
  // elements): exact in one bf16 part, so its lo products are skipped; a bf16
  // A needs alpha = +-1
  bool aBf = false, bBf = false;
};
struct TcGemmN {
  TcTerm t[kMaxTerms];
  int nterms;
  float* Cm;
  const float* Add;
  long long sC, sAdd;
  int ldc, ldadd, M, N, batch, mask;
  int* status;
  // optional second output, same layout as C: C2 = mask2(C scaled by the
  // batch item's vector: op 1 rows (vec[r]), op 2 columns (vec[n])), vec
  // holding M values per batch item
  float* C2 = nullptr;
  const float* vec = nullptr;
  int c2op = 0, c2mask = 0;
};
bool gemm_tc_supported(const TcGemmN& g);
cudaError_t launch_gemm_tc(const TcGemmN& g, cudaStream_t st);
// Diagnostics: a kernel whose bounded wait can only expire (sets *status).
cudaError_t launch_debug_wait(int* status, unsigned long long limit_ns, cudaStream_t st);

}  // namespace pathattn
