// api.cu -- the C ABI of libpathattn.so (declared in include/pathattn.h).
//
// Argument validation happens before any CUDA call.  Workspace comes from a
// per-device memory pool owned by the library (stream-ordered, cached across
// calls).  Kernels report bounded-wait expiry through a per-device status word.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/pathattn.h"
#include "common.cuh"

using namespace pathattn;

namespace {

constexpr int kVersion = 100;  // 0.1.0
constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  cudaMemPool_t pool = nullptr;
  int* status = nullptr;  // device int, 0 = fine
  int cc_major = 0, cc_minor = 0;
  int num_sms = 0;
  // copy streams of the host-buffer entry (non-blocking, created with the state)
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
};

// Form of the transition in the bf16 d = 64 forward (path_attn_set_transition_form):
// 0 dense (q <- q + q ngt^T), 1 low-rank (q <- q + (q W^T)(-(U W))).
std::atomic<int> g_transition_form{0};

// The low-rank form applies to bf16 problems at d = 64 when selected.
void apply_transition_form(Geom* g) {
  g->lowrank = g_transition_form.load() == 1 && g->bf16 && g->d == 64;
}

// Slices of (b, h) problems the host-buffer entry pipelines its copies over
// (at most this many).
constexpr int kHostSlices = 8;

// Heads per slice of the host-buffer entry, in order; returns the count.
// Fewer than 16 problems: up to four equal slices.  Otherwise a first and a
// last slice of BH/8 problems around middle slices of about BH/4: the copy
// of the first slice and the compute and copy-out of the last one are the
// parts of the call nothing overlaps, so they are kept small, while the
// middle slices stay large enough to fill the GPU.
int host_slice_plan(int BH, int* heads) {
  if (BH < 16) {
    const int nsl = BH < 4 ? BH : 4, per = (BH + nsl - 1) / nsl;
    int n = 0;
    for (int b0 = 0; b0 < BH; b0 += per) heads[n++] = std::min(per, BH - b0);
    return n;
  }
  const int edge = BH / 8, mid = BH - 2 * edge;
  const int n_mid = std::min(kHostSlices - 2, (mid + BH / 4 - 1) / (BH / 4));
  int n = 0;
  heads[n++] = edge;
  for (int i = 0; i < n_mid; ++i) heads[n++] = mid / n_mid + (i < mid % n_mid ? 1 : 0);
  heads[n++] = edge;
  return n;
}

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
thread_local char g_last_error[256] = "";

struct TimingRec {
  cudaEvent_t e0, e1, e2;
};
bool g_timing = false;
std::vector<TimingRec> g_timing_recs;
size_t g_timing_used = 0;
struct BwdTimingRec {
  cudaEvent_t ev[kBwdPhases + 1];
};
std::vector<BwdTimingRec> g_bwd_recs;
size_t g_bwd_used = 0;

// The next backward timing record (events created on first use), or null
// when timing is off or events cannot be created.
cudaEvent_t* next_bwd_rec() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_timing) return nullptr;
  if (g_bwd_used == g_bwd_recs.size()) {
    BwdTimingRec r{};
    for (auto& e : r.ev)
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_bwd_recs.push_back(r);
  }
  return g_bwd_recs[g_bwd_used++].ev;
}

int set_cuda_error(cudaError_t e) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return e == cudaErrorMemoryAllocation ? PATH_ERR_OOM : PATH_ERR_CUDA;
}

// Per-device library state, created on first use with that device current.
int device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return PATH_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    cudaDeviceProp prop;
    if ((e = cudaGetDeviceProperties(&prop, dev)) != cudaSuccess) return set_cuda_error(e);
    s.cc_major = prop.major;
    s.cc_minor = prop.minor;
    s.num_sms = prop.multiProcessorCount;
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    if ((e = cudaMemPoolCreate(&s.pool, &props)) != cudaSuccess) return set_cuda_error(e);
    uint64_t keep = UINT64_MAX;
    if ((e = cudaMemPoolSetAttribute(s.pool, cudaMemPoolAttrReleaseThreshold, &keep)) !=
        cudaSuccess)
      return set_cuda_error(e);
    if ((e = cudaMalloc(&s.status, sizeof(int))) != cudaSuccess) return set_cuda_error(e);
    if ((e = cudaMemset(s.status, 0, sizeof(int))) != cudaSuccess) return set_cuda_error(e);
    if ((e = cudaStreamCreateWithFlags(&s.copy_in, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&s.copy_out, cudaStreamNonBlocking)) != cudaSuccess)
      return set_cuda_error(e);
    s.ready = true;
  }
  *out = &s;
  return PATH_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int chunk_size(int d, int dtype) {
  if (dtype != PATH_DTYPE_F32 && dtype != PATH_DTYPE_BF16) return PATH_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PATH_ERR_UNSUPPORTED;
  return dtype == PATH_DTYPE_BF16 ? 128 : 64;
}

// Shape checks shared by every entry point; fills the geometry.
int make_geom(int B, int H, int T, int d, int dtype, bool gate, Geom* g) {
  if (B < 1 || H < 1 || T < 1) return PATH_ERR_INVALID_ARG;
  const int C = chunk_size(d, dtype);
  if (C < 0) return C;
  const long long BH = static_cast<long long>(B) * H;
  const long long Np = (static_cast<long long>(T) + C - 1) / C;
  const long long Tp = Np * C;
  // every operand and workspace index stays inside int32 row/column space
  if (BH * Tp * d > INT_MAX || BH * Np * d * d > INT_MAX || BH * Np > INT_MAX / 4)
    return PATH_ERR_UNSUPPORTED;
  g->B = B; g->H = H; g->T = T; g->d = d; g->C = C;
  g->BH = static_cast<int>(BH);
  g->Np = static_cast<int>(Np);
  g->Tp = static_cast<int>(Tp);
  g->nch = static_cast<int>(BH * Np);
  g->bf16 = dtype == PATH_DTYPE_BF16;
  g->gate = gate;
  return PATH_OK;
}

int check_device(const DeviceState* s) {
  // kernels are built for sm_103a only
  if (s->cc_major != 10 || s->cc_minor != 3) {
    std::snprintf(g_last_error, sizeof(g_last_error),
                  "libpathattn is built for sm_103a; this device is sm_%d%d", s->cc_major,
                  s->cc_minor);
    return PATH_ERR_UNSUPPORTED;
  }
  return PATH_OK;
}

// Prep, then (once `ev_v` has completed: the copy of v) attention, for the
// host-buffer entry's slices.
int run_forward_after(const Geom& g, const Inputs& in, char* ws_base, DeviceState* s,
                      cudaStream_t st, cudaEvent_t ev_v) {
  Workspace ws;
  workspace_layout(g, ws_base, &ws);
  cudaError_t e;
  if ((e = launch_prep(g, in, ws, s->status, st, nullptr)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(st, ev_v, 0)) != cudaSuccess)
    return set_cuda_error(e);
  if (g.bf16)
    e = launch_attn_tc(g, in, ws, s->status, st, nullptr);
  else
    e = launch_attn_f32(g, in, ws, st, nullptr);
  return e == cudaSuccess ? PATH_OK : set_cuda_error(e);
}

// Runs prep + attention for device pointers; `ws_base` must hold the layout.
int run_forward(const Geom& g, const Inputs& in, char* ws_base, DeviceState* s,
                cudaStream_t st) {
  Workspace ws;
  workspace_layout(g, ws_base, &ws);
  TimingRec* rec = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_timing) {
      if (g_timing_used == g_timing_recs.size()) {
        TimingRec r{};
        if (cudaEventCreate(&r.e0) == cudaSuccess && cudaEventCreate(&r.e1) == cudaSuccess &&
            cudaEventCreate(&r.e2) == cudaSuccess)
          g_timing_recs.push_back(r);
      }
      if (g_timing_used < g_timing_recs.size()) rec = &g_timing_recs[g_timing_used++];
    }
  }
  cudaError_t e;
  if (rec) cudaEventRecord(rec->e0, st);
  if ((e = launch_prep(g, in, ws, s->status, st, nullptr)) != cudaSuccess) return set_cuda_error(e);
  if (rec) cudaEventRecord(rec->e1, st);
  if (g.bf16)
    e = launch_attn_tc(g, in, ws, s->status, st, nullptr);
  else
    e = launch_attn_f32(g, in, ws, st, nullptr);
  if (e != cudaSuccess) return set_cuda_error(e);
  if (rec) cudaEventRecord(rec->e2, st);
  return PATH_OK;
}

}  // namespace

extern "C" {

const char* path_attn_status_string(int status) {
  switch (status) {
    case PATH_OK: return "PATH_OK";
    case PATH_ERR_INVALID_ARG: return "PATH_ERR_INVALID_ARG";
    case PATH_ERR_UNSUPPORTED: return "PATH_ERR_UNSUPPORTED";
    case PATH_ERR_CUDA: return "PATH_ERR_CUDA";
    case PATH_ERR_TIMEOUT: return "PATH_ERR_TIMEOUT";
    case PATH_ERR_OOM: return "PATH_ERR_OOM";
    default: return "PATH_ERR_UNKNOWN";
  }
}

const char* path_attn_last_error(void) { return g_last_error; }

int path_attn_version(void) { return kVersion; }

int path_attn_chunk_size(int d, int dtype) { return chunk_size(d, dtype); }

int path_attn_workspace_bytes(int B, int H, int T, int d, int dtype, int with_gate,
                              size_t* bytes) {
  if (!bytes) return PATH_ERR_INVALID_ARG;
  Geom g;
  const int rc = make_geom(B, H, T, d, dtype, with_gate != 0, &g);
  if (rc != PATH_OK) return rc;
  *bytes = workspace_layout(g, nullptr, nullptr);
  return PATH_OK;
}

int path_attn_launches_per_call(int d, int dtype, int with_gate) {
  const int C = chunk_size(d, dtype);
  if (C < 0) return C;
  const int prep = dtype == PATH_DTYPE_BF16 ? 1 : 11;
  return prep + (with_gate ? 1 : 0) + 1;
}

int path_attn_bwd_launches_per_call(int T, int d, int dtype, int with_gate) {
  const int C = chunk_size(d, dtype);
  if (C < 0) return C;
  if (T < 1) return PATH_ERR_INVALID_ARG;
  const int g = with_gate ? 1 : 0;
  if (dtype == PATH_DTYPE_BF16) {
    // chunk pass: input copies, 17 tensor-core products (the scaled second
    // outputs in their epilogues), inverse (with U), dbeta, outputs, gate scan
    const int chunk = 1 + 17 + 1 + 1 + 1 + g;
    // preparation (+ gate prefix), rowdot, [X walk], key pass, G walk, dF
    return (1 + g) + 1 + (T > C ? 1 : 0) + 3 + chunk;
  }
  // chunk pass: fp32 copies, 30 one-term GEMMs, 3 scaled copies, inverse,
  // U, dbeta, outputs, gate scan
  const int chunk = 1 + 30 + 3 + 1 + 1 + 1 + 1 + g;
  // SIMT preparation (+ gate prefix), rowdot, query walk, key pass, dF
  return (11 + g) + 1 + 3 + chunk;
}

int path_attn_fwd(const void* q, const void* k, const void* v, const void* w,
                  const float* beta, const float* logf, float scale, void* out, float* lse,
                  int B, int H, int T, int d, int dtype, void* stream) {
  if (!q || !k || !v || !w || !beta || !out) return PATH_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(w) || !aligned16(beta) ||
      !aligned16(out) || (logf && !aligned16(logf)) || (lse && !aligned16(lse)))
    return PATH_ERR_INVALID_ARG;
  if (!(scale == scale)) return PATH_ERR_INVALID_ARG;  // NaN scale
  Geom g;
  int rc = make_geom(B, H, T, d, dtype, logf != nullptr, &g);
  if (rc != PATH_OK) return rc;
  apply_transition_form(&g);
  DeviceState* s = nullptr;
  if ((rc = device_state(&s)) != PATH_OK) return rc;
  if ((rc = check_device(s)) != PATH_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = workspace_layout(g, nullptr, nullptr);
  void* ws = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, s->pool, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  Inputs in{q, k, v, w, beta, logf, scale, out, lse};
  rc = run_forward(g, in, static_cast<char*>(ws), s, st);
  e = cudaFreeAsync(ws, st);
  if (rc == PATH_OK && e != cudaSuccess) rc = set_cuda_error(e);
  return rc;
}

int path_attn_set_transition_form(int form) {
  if (form != 0 && form != 1) return PATH_ERR_INVALID_ARG;
  g_transition_form = form;
  return PATH_OK;
}

int path_attn_bwd_workspace_bytes(int B, int H, int T, int d, int dtype, int with_gate,
                                  size_t* bytes) {
  if (!bytes) return PATH_ERR_INVALID_ARG;
  Geom g;
  const int rc = make_geom(B, H, T, d, dtype, with_gate != 0, &g);
  if (rc != PATH_OK) return rc;
  *bytes = workspace_layout(g, nullptr, nullptr) + bwd_workspace_layout(g, nullptr, nullptr, nullptr);
  return PATH_OK;
}

int path_attn_bwd(const void* q, const void* k, const void* v, const void* w,
                  const float* beta, const float* logf, float scale, const void* out,
                  const float* lse, const void* dout, const float* dlse, void* dq, void* dk,
                  void* dv, void* dw, float* dbeta, float* dlogf, int B, int H, int T, int d,
                  int dtype, void* stream) {
  if (!q || !k || !v || !w || !beta || !out || !lse || !dout || !dq || !dk || !dv || !dw ||
      !dbeta)
    return PATH_ERR_INVALID_ARG;
  if ((logf != nullptr) != (dlogf != nullptr)) return PATH_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, w, beta, out, lse, dout, dq, dk, dv, dw, dbeta};
  for (const void* x : ptrs)
    if (!aligned16(x)) return PATH_ERR_INVALID_ARG;
  if ((logf && !aligned16(logf)) || (dlogf && !aligned16(dlogf)) || (dlse && !aligned16(dlse)))
    return PATH_ERR_INVALID_ARG;
  if (!(scale == scale)) return PATH_ERR_INVALID_ARG;
  Geom g;
  int rc = make_geom(B, H, T, d, dtype, logf != nullptr, &g);
  if (rc != PATH_OK) return rc;
  DeviceState* s = nullptr;
  if ((rc = device_state(&s)) != PATH_OK) return rc;
  if ((rc = check_device(s)) != PATH_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t fwd_bytes = workspace_layout(g, nullptr, nullptr);
  const size_t bytes = fwd_bytes + bwd_workspace_layout(g, nullptr, nullptr, nullptr);
  char* base = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&base), bytes, s->pool, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  Workspace ws;
  workspace_layout(g, base, &ws);
  BwdParams p;
  ChunkBufs cb;
  bwd_workspace_layout(g, base + fwd_bytes, &p, &cb);
  Inputs in{q, k, v, w, beta, logf, scale, nullptr, nullptr};
  p.ev = next_bwd_rec();
  bwd_mark(p.ev, kBwdEvPrep, st);
  e = launch_prep(g, in, ws, s->status, st, nullptr);
  bwd_mark(p.ev, kBwdEvRowdot, st);
  if (e == cudaSuccess) {
    p.q = q; p.k = k; p.v = v; p.w = w; p.out = out; p.dout = dout;
    p.beta = beta; p.lse = lse; p.dlse = dlse;
    p.scale = scale; p.scale_log2e = scale * kLog2e;
    p.dq = dq; p.dk = dk; p.dv = dv; p.dw = dw; p.dbeta = dbeta; p.dlogf = dlogf;
    p.kr = ws.kr; p.ql = ws.ql; p.ngt = ws.ngt; p.sdt = ws.sdt;
    p.lam2 = g.gate ? ws.lam2 : nullptr;
    p.BH = g.BH; p.T = g.T; p.Tp = g.Tp; p.Np = g.Np; p.C = g.C; p.d = g.d; p.nch = g.nch;
    p.bf16 = g.bf16;
    p.status = s->status;
    e = launch_bwd(p, cb, st);
  }
  if (e != cudaSuccess) rc = set_cuda_error(e);
  e = cudaFreeAsync(base, st);
  if (rc == PATH_OK && e != cudaSuccess) rc = set_cuda_error(e);
  return rc;
}

int path_attn_fwd_partial(const void* q, const void* k, const void* v, const void* w,
                          const float* beta, const float* logf, float scale, void* out,
                          float* lse, int B, int H, int T, int d, int r, int dtype, void* stream) {
  if (!q || !k || !v || (r > 0 && !w) || !beta || !out) return PATH_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(beta) || !aligned16(out) ||
      (logf && !aligned16(logf)) || (lse && !aligned16(lse)))
    return PATH_ERR_INVALID_ARG;
  if (!(scale == scale) || r < 0 || r > d) return PATH_ERR_INVALID_ARG;
  Geom g;
  int rc = make_geom(B, H, T, d, dtype, logf != nullptr, &g);
  if (rc != PATH_OK) return rc;
  DeviceState* s = nullptr;
  if ((rc = device_state(&s)) != PATH_OK) return rc;
  if ((rc = check_device(s)) != PATH_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (g.bf16 && d == 128 && r == 64 && aligned16(w)) {
    // rank-64 transitions at d = 128: the preparation reads u through a
    // tensor map of width r (zeros past it) and the attention carries only
    // the first r coordinates of the running query through the transitions
    void* ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, workspace_layout(g, nullptr, nullptr), s->pool, st);
    if (e != cudaSuccess) return set_cuda_error(e);
    Inputs in{q, k, v, w, beta, logf, scale, out, lse};
    in.wr = r;
    rc = run_forward(g, in, static_cast<char*>(ws), s, st);
    e = cudaFreeAsync(ws, st);
    if (rc == PATH_OK && e != cudaSuccess) rc = set_cuda_error(e);
    return rc;
  }
  const size_t es = g.bf16 ? 2 : 4;
  const size_t rows = static_cast<size_t>(g.BH) * T;
  const size_t wbytes = align_up(rows * d * es, 256);
  const size_t bytes = wbytes + workspace_layout(g, nullptr, nullptr);
  char* buf = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&buf), bytes, s->pool, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  // u widened with zeros: H_t is then the identity outside the first r dims
  if (r < d) e = cudaMemsetAsync(buf, 0, rows * d * es, st);
  if (e == cudaSuccess && r > 0)
    e = cudaMemcpy2DAsync(buf, d * es, w, static_cast<size_t>(r) * es, static_cast<size_t>(r) * es,
                          rows, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) {
    rc = set_cuda_error(e);
  } else {
    Inputs in{q, k, v, buf, beta, logf, scale, out, lse};
    rc = run_forward(g, in, buf + wbytes, s, st);
  }
  e = cudaFreeAsync(buf, st);
  if (rc == PATH_OK && e != cudaSuccess) rc = set_cuda_error(e);
  return rc;
}

int path_attn_fwd_host(const void* q, const void* k, const void* v, const void* w,
                       const float* beta, const float* logf, float scale, void* out,
                       float* lse, int B, int H, int T, int d, int dtype, void* stream) {
  if (!q || !k || !v || !w || !beta || !out) return PATH_ERR_INVALID_ARG;
  Geom g;
  int rc = make_geom(B, H, T, d, dtype, logf != nullptr, &g);
  if (rc != PATH_OK) return rc;
  DeviceState* s = nullptr;
  if ((rc = device_state(&s)) != PATH_OK) return rc;
  if ((rc = check_device(s)) != PATH_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The (b, h) problems are independent and contiguous in every array: the
  // call runs them in slices, copies of slice i + 1 in and of slice i - 1 out
  // on two copy streams while slice i computes on `stream`.  Within a slice,
  // q, k, w, beta (and log f) go first: the preparation starts once they have
  // landed, while v is still copying.
  int heads[kHostSlices];
  const int nsl = host_slice_plan(g.BH, heads);
  int per = 0;
  for (int i = 0; i < nsl; ++i) per = std::max(per, heads[i]);
  Geom gs;
  if ((rc = make_geom(1, per, T, d, dtype, logf != nullptr, &gs)) != PATH_OK) return rc;
  apply_transition_form(&gs);
  const size_t es = dtype == PATH_DTYPE_BF16 ? 2 : 4;
  const size_t xrow = static_cast<size_t>(T) * d * es, brow = static_cast<size_t>(T) * 4;
  const size_t nx = xrow * g.BH, nb = brow * g.BH;
  size_t off = 0;
  auto take = [&](size_t n) { size_t o = off; off = align_up(off + n, 256); return o; };
  const size_t oq = take(nx), ok_ = take(nx), ov = take(nx), ow = take(nx), ob = take(nb),
               olf = logf ? take(nb) : 0, oo = take(nx), ol = lse ? take(nb) : 0;
  const size_t io_bytes = off;
  const size_t ws_bytes = workspace_layout(gs, nullptr, nullptr);
  char* buf = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&buf), io_bytes + ws_bytes,
                                          s->pool, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  cudaEvent_t ev_start = nullptr, ev_in[kHostSlices] = {}, ev_qkw[kHostSlices] = {},
              ev_done[kHostSlices] = {}, ev_out = nullptr;
  auto mk = [](cudaEvent_t* ev) { return cudaEventCreateWithFlags(ev, cudaEventDisableTiming); };
  bool ok = (e = mk(&ev_start)) == cudaSuccess && (e = mk(&ev_out)) == cudaSuccess;
  for (int i = 0; ok && i < nsl; ++i)
    ok = (e = mk(&ev_in[i])) == cudaSuccess && (e = mk(&ev_qkw[i])) == cudaSuccess &&
         (e = mk(&ev_done[i])) == cudaSuccess;
  // the buffer exists on `stream` first; both copy streams start after that
  if (ok) ok = (e = cudaEventRecord(ev_start, st)) == cudaSuccess &&
               (e = cudaStreamWaitEvent(s->copy_in, ev_start, 0)) == cudaSuccess &&
               (e = cudaStreamWaitEvent(s->copy_out, ev_start, 0)) == cudaSuccess;
  auto h2d = [&](size_t o, const void* src, size_t n) {
    return cudaMemcpyAsync(buf + o, src, n, cudaMemcpyHostToDevice, s->copy_in);
  };
  auto d2h = [&](void* dst, size_t o, size_t n) {
    return cudaMemcpyAsync(dst, buf + o, n, cudaMemcpyDeviceToHost, s->copy_out);
  };
  auto hp = [](const void* p, size_t o) { return static_cast<const char*>(p) + o; };
  for (int i = 0, bh0 = 0; ok && i < nsl; bh0 += heads[i], ++i) {
    const int nbh = heads[i];
    const size_t x0 = xrow * bh0, xn = xrow * nbh, b0 = brow * bh0, bn = brow * nbh;
    ok = (e = h2d(oq + x0, hp(q, x0), xn)) == cudaSuccess &&
         (e = h2d(ok_ + x0, hp(k, x0), xn)) == cudaSuccess &&
         (e = h2d(ow + x0, hp(w, x0), xn)) == cudaSuccess &&
         (e = h2d(ob + b0, hp(beta, b0), bn)) == cudaSuccess &&
         (!logf || (e = h2d(olf + b0, hp(logf, b0), bn)) == cudaSuccess) &&
         (e = cudaEventRecord(ev_qkw[i], s->copy_in)) == cudaSuccess &&
         (e = h2d(ov + x0, hp(v, x0), xn)) == cudaSuccess &&
         (e = cudaEventRecord(ev_in[i], s->copy_in)) == cudaSuccess &&
         (e = cudaStreamWaitEvent(st, ev_qkw[i], 0)) == cudaSuccess;
    if (!ok) break;
    Geom gi = gs;
    if (nbh != per && (rc = make_geom(1, nbh, T, d, dtype, logf != nullptr, &gi)) != PATH_OK) break;
    apply_transition_form(&gi);
    Inputs in{buf + oq + x0, buf + ok_ + x0, buf + ov + x0, buf + ow + x0,
              reinterpret_cast<float*>(buf + ob + b0),
              logf ? reinterpret_cast<float*>(buf + olf + b0) : nullptr, scale,
              buf + oo + x0, lse ? reinterpret_cast<float*>(buf + ol + b0) : nullptr};
    if ((rc = run_forward_after(gi, in, buf + io_bytes, s, st, ev_in[i])) != PATH_OK) break;
    ok = (e = cudaEventRecord(ev_done[i], st)) == cudaSuccess &&
         (e = cudaStreamWaitEvent(s->copy_out, ev_done[i], 0)) == cudaSuccess &&
         (e = d2h(static_cast<char*>(out) + x0, oo + x0, xn)) == cudaSuccess &&
         (!lse || (e = d2h(reinterpret_cast<char*>(lse) + b0, ol + b0, bn)) == cudaSuccess);
  }
  if (rc == PATH_OK && !ok) rc = set_cuda_error(e);
  // whatever was queued on the copy streams finishes before the buffer is freed
  cudaError_t e2 = cudaEventRecord(ev_out, s->copy_out);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(st, ev_out, 0);
  cudaError_t e3 = cudaEventRecord(ev_start, s->copy_in);
  if (e3 == cudaSuccess) e3 = cudaStreamWaitEvent(st, ev_start, 0);
  if (rc == PATH_OK && (e2 != cudaSuccess || e3 != cudaSuccess))
    rc = set_cuda_error(e2 != cudaSuccess ? e2 : e3);
  e = cudaFreeAsync(buf, st);
  if (rc == PATH_OK && e != cudaSuccess) rc = set_cuda_error(e);
  e = cudaStreamSynchronize(st);
  if (rc == PATH_OK && e != cudaSuccess) rc = set_cuda_error(e);
  for (cudaEvent_t ev : {ev_start, ev_out})
    if (ev) cudaEventDestroy(ev);
  for (int i = 0; i < kHostSlices; ++i) {
    if (ev_in[i]) cudaEventDestroy(ev_in[i]);
    if (ev_qkw[i]) cudaEventDestroy(ev_qkw[i]);
    if (ev_done[i]) cudaEventDestroy(ev_done[i]);
  }
  return rc;
}

int path_attn_prefill(const void* q, const void* k, const void* v, const void* w,
                      const float* beta, const float* logf, float scale, void* out,
                      float* lse, float* kcache, void* vcache, float* lamcache, int Tmax,
                      int B, int H, int T, int d, int dtype, void* stream) {
  if (!q || !k || !v || !w || !beta || !out || !kcache || !vcache) return PATH_ERR_INVALID_ARG;
  if ((logf != nullptr) != (lamcache != nullptr)) return PATH_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(w) || !aligned16(beta) ||
      !aligned16(out) || (logf && !aligned16(logf)) || (lse && !aligned16(lse)) ||
      !aligned16(kcache) || !aligned16(vcache) || (lamcache && !aligned16(lamcache)))
    return PATH_ERR_INVALID_ARG;
  if (!(scale == scale) || Tmax < T) return PATH_ERR_INVALID_ARG;
  Geom g;
  int rc = make_geom(B, H, T, d, dtype, logf != nullptr, &g);
  if (rc != PATH_OK) return rc;
  DeviceState* s = nullptr;
  if ((rc = device_state(&s)) != PATH_OK) return rc;
  if ((rc = check_device(s)) != PATH_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = workspace_layout(g, nullptr, nullptr);
  void* ws = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, s->pool, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  Inputs in{q, k, v, w, beta, logf, scale, out, lse};
  rc = run_forward(g, in, static_cast<char*>(ws), s, st);
  if (rc == PATH_OK) {
    Workspace wsp;
    workspace_layout(g, static_cast<char*>(ws), &wsp);
    const size_t es = g.bf16 ? 2 : 4;
    const size_t row = static_cast<size_t>(d) * es;
    if ((e = launch_align_keys(g, wsp, kcache, Tmax, st)) != cudaSuccess ||
        (e = cudaMemcpy2DAsync(vcache, row * Tmax, v, row * T, row * T, g.BH,
                               cudaMemcpyDeviceToDevice, st)) != cudaSuccess ||
        (logf && (e = launch_gate_prefix(logf, lamcache, g.BH, T, T, static_cast<size_t>(Tmax),
                                         1.0, st)) != cudaSuccess))
      rc = set_cuda_error(e);
  }
  e = cudaFreeAsync(ws, st);
  if (rc == PATH_OK && e != cudaSuccess) rc = set_cuda_error(e);
  return rc;
}

int path_attn_decode_step(const void* q, const void* k, const void* v, const void* w,
                          const float* beta, const float* logf, float scale, float* kcache,
                          void* vcache, float* lamcache, const int* pos, int max_len,
                          void* out, float* lse, int B, int H, int Tmax, int d, int dtype,
                          void* stream) {
  if (!q || !k || !v || !w || !beta || !out || !kcache || !vcache || !pos)
    return PATH_ERR_INVALID_ARG;
  if ((logf != nullptr) != (lamcache != nullptr)) return PATH_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(w) || !aligned16(beta) ||
      !aligned16(out) || (logf && !aligned16(logf)) || (lse && !aligned16(lse)) ||
      !aligned16(kcache) || !aligned16(vcache) || (lamcache && !aligned16(lamcache)))
    return PATH_ERR_INVALID_ARG;
  if (!(scale == scale) || B < 1 || H < 1 || Tmax < 1 || max_len < 1 || max_len > Tmax)
    return PATH_ERR_INVALID_ARG;
  if (chunk_size(d, dtype) < 0) return chunk_size(d, dtype);
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 65535) return PATH_ERR_UNSUPPORTED;  // grid.y of the span kernel
  DeviceState* s = nullptr;
  int rc = device_state(&s);
  if (rc != PATH_OK) return rc;
  if ((rc = check_device(s)) != PATH_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // spans of whole tiles, about two CTAs per SM when there are few heads
  const int tile = decode_tile_keys(d);
  const long long tiles = std::max<long long>(1, (max_len - 1 + tile - 1) / tile);
  long long nsplit = std::max<long long>(1, 2LL * s->num_sms / BH);
  nsplit = std::min(nsplit, tiles);
  const long long per = (tiles + nsplit - 1) / nsplit;
  nsplit = (tiles + per - 1) / per;
  float* part = nullptr;
  const size_t part_bytes =
      align_up(static_cast<size_t>(BH) * nsplit * (d + 2) * sizeof(float), 256);
  const size_t cnt_bytes = static_cast<size_t>(BH) * sizeof(int);
  cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&part), part_bytes + cnt_bytes,
                                          s->pool, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  int* counters = reinterpret_cast<int*>(reinterpret_cast<char*>(part) + part_bytes);
  DecodeParams p{q, k, v, w, beta, logf, scale, kcache, vcache, lamcache, pos, H, Tmax, max_len,
                 static_cast<int>(nsplit), static_cast<int>(per * tile), part, counters, out, lse,
                 s->status};
  if ((e = cudaMemsetAsync(counters, 0, cnt_bytes, st)) != cudaSuccess ||
      (e = launch_decode(p, static_cast<int>(BH), d, dtype == PATH_DTYPE_BF16, st)) != cudaSuccess)
    rc = set_cuda_error(e);
  e = cudaFreeAsync(part, st);
  if (rc == PATH_OK && e != cudaSuccess) rc = set_cuda_error(e);
  return rc;
}

int path_producer_fwd(const void* x, const void* Wd, const void* Wu, const float* cw,
                      const void* Ub, const float* bb, void* w, float* beta, int B, int T,
                      int Dm, int H, int d, int R, int dtype, void* stream) {
  if (!x || !Wd || !Wu || !cw || !Ub || !bb || !w || !beta) return PATH_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wd) || !aligned16(Wu) || !aligned16(Ub) || !aligned16(w) ||
      !aligned16(beta) || (reinterpret_cast<uintptr_t>(cw) & 3u) ||
      (reinterpret_cast<uintptr_t>(bb) & 3u))
    return PATH_ERR_INVALID_ARG;
  if (dtype != PATH_DTYPE_F32 && dtype != PATH_DTYPE_BF16) return PATH_ERR_INVALID_ARG;
  if (B < 1 || T < 1 || H < 1 || Dm < 1 || R < 1) return PATH_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PATH_ERR_UNSUPPORTED;
  // tile shapes: Dm in 64-wide stages, R in 16-wide MMA steps, R + H columns
  // of one projection tile (padded to a multiple of 8)
  if (Dm % 64 != 0 || Dm > 32768 || R % 16 != 0 || R > 128 || R + H > 128)
    return PATH_ERR_UNSUPPORTED;
  const long long BT = static_cast<long long>(B) * T;
  if (BT > INT_MAX / 2 || BT * H > INT_MAX) return PATH_ERR_UNSUPPORTED;
  DeviceState* s = nullptr;
  int rc = device_state(&s);
  if (rc != PATH_OK) return rc;
  if ((rc = check_device(s)) != PATH_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&ws, producer_workspace_bytes(B, T, R, H, d), s->pool, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  if ((e = launch_producer(x, Wd, Wu, cw, Ub, bb, w, beta, ws, s->status, B, T, Dm, H, d, R,
                           dtype == PATH_DTYPE_BF16, st)) != cudaSuccess)
    rc = set_cuda_error(e);
  e = cudaFreeAsync(ws, st);
  if (rc == PATH_OK && e != cudaSuccess) rc = set_cuda_error(e);
  return rc;
}

int path_attn_device_status(int device, int clear) {
  int prev = 0;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return set_cuda_error(e);
  if ((e = cudaSetDevice(device)) != cudaSuccess) return set_cuda_error(e);
  DeviceState* s = nullptr;
  int rc = device_state(&s);
  int word = 0;
  if (rc == PATH_OK) {
    if ((e = cudaDeviceSynchronize()) != cudaSuccess ||
        (e = cudaMemcpy(&word, s->status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (clear && (e = cudaMemset(s->status, 0, sizeof(int))) != cudaSuccess))
      rc = set_cuda_error(e);
  }
  cudaSetDevice(prev);
  if (rc != PATH_OK) return rc;
  if (word == PATH_DEV_OK) return PATH_OK;
  return word == PATH_DEV_ERR_BAD_POS ? PATH_ERR_INVALID_ARG : PATH_ERR_TIMEOUT;
}

int path_attn_timing_enable(int enable) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_timing = enable != 0;
  g_timing_used = 0;
  g_bwd_used = 0;
  return PATH_OK;
}

int path_attn_bwd_timing_read(double* phase_ms, long* calls) {
  std::vector<BwdTimingRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    recs.assign(g_bwd_recs.begin(), g_bwd_recs.begin() + g_bwd_used);
  }
  double acc[kBwdPhases] = {};
  for (auto& r : recs) {
    cudaError_t e = cudaEventSynchronize(r.ev[kBwdPhases]);
    if (e != cudaSuccess) return set_cuda_error(e);
    for (int i = 0; i < kBwdPhases; ++i) {
      float x = 0;
      if ((e = cudaEventElapsedTime(&x, r.ev[i], r.ev[i + 1])) != cudaSuccess)
        return set_cuda_error(e);
      acc[i] += x;
    }
  }
  if (phase_ms)
    for (int i = 0; i < kBwdPhases; ++i) phase_ms[i] = acc[i];
  if (calls) *calls = static_cast<long>(recs.size());
  return PATH_OK;
}

int path_attn_timing_read(double* prep_ms, double* attn_ms, long* calls) {
  std::vector<TimingRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    recs.assign(g_timing_recs.begin(), g_timing_recs.begin() + g_timing_used);
  }
  double p = 0, a = 0;
  for (auto& r : recs) {
    cudaError_t e = cudaEventSynchronize(r.e2);
    if (e != cudaSuccess) return set_cuda_error(e);
    float x = 0, y = 0;
    if ((e = cudaEventElapsedTime(&x, r.e0, r.e1)) != cudaSuccess ||
        (e = cudaEventElapsedTime(&y, r.e1, r.e2)) != cudaSuccess)
      return set_cuda_error(e);
    p += x;
    a += y;
  }
  if (prep_ms) *prep_ms = p;
  if (attn_ms) *attn_ms = a;
  if (calls) *calls = static_cast<long>(recs.size());
  return PATH_OK;
}

int path_attn_debug_factors(const void* q, const void* k, const void* w, const float* beta,
                            const float* logf, float scale, int B, int H, int T, int d,
                            int dtype, void* kr, float* ql, void* ngt, float* sdt, float* lam2,
                            void* stream) {
  if (!q || !k || !w || !beta || !kr || !ql || !ngt || !sdt || (logf && !lam2))
    return PATH_ERR_INVALID_ARG;
  Geom g;
  int rc = make_geom(B, H, T, d, dtype, logf != nullptr, &g);
  if (rc != PATH_OK) return rc;
  DeviceState* s = nullptr;
  if ((rc = device_state(&s)) != PATH_OK) return rc;
  if ((rc = check_device(s)) != PATH_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = workspace_layout(g, nullptr, nullptr);
  void* base = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&base, bytes, s->pool, st);
  if (e != cudaSuccess) return set_cuda_error(e);
  Workspace ws;
  workspace_layout(g, static_cast<char*>(base), &ws);
  Inputs in{q, k, nullptr, w, beta, logf, scale, nullptr, nullptr};
  e = launch_prep(g, in, ws, s->status, st, nullptr);
  const size_t es = g.bf16 ? 2 : 4, nch = g.nch, C = g.C;
  if (e == cudaSuccess) e = cudaMemcpyAsync(kr, ws.kr, nch * C * d * es, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ql, ws.ql, nch * C * d * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ngt, ws.ngt, nch * d * d * es, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(sdt, ws.sdt, nch * C * C * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && logf)
    e = cudaMemcpyAsync(lam2, ws.lam2, static_cast<size_t>(g.BH) * g.Tp * 4,
                        cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) rc = set_cuda_error(e);
  e = cudaFreeAsync(base, st);
  if (rc == PATH_OK && e != cudaSuccess) rc = set_cuda_error(e);
  return rc;
}

int path_attn_debug_wait_timeout(unsigned long long limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 2000000000ull) return PATH_ERR_INVALID_ARG;
  DeviceState* s = nullptr;
  int rc = device_state(&s);
  if (rc != PATH_OK) return rc;
  if ((rc = check_device(s)) != PATH_OK) return rc;
  cudaError_t e = launch_debug_wait(s->status, limit_ns, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PATH_OK : set_cuda_error(e);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry: the workspace lives in a static device array.
namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[PATH_NOALLOC_SCRATCH_BYTES];
__device__ __align__(256) int g_noalloc_status;

struct NoAllocState {
  bool ready = false;
  char* scratch = nullptr;  // device address of g_noalloc_scratch
  int* status = nullptr;    // device address of g_noalloc_status
  int cc_major = 0, cc_minor = 0;
};
NoAllocState g_noalloc[kMaxDevices];

// Once per device, with that device current: check that the device is the
// one the library is built for (before anything loads the module holding the
// arrays), then look up the arrays' device addresses (host code may not use
// the symbols themselves as pointers).
int noalloc_setup(NoAllocState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) {
    std::snprintf(g_last_error, sizeof(g_last_error),
                  "libpathattn keeps state for devices 0 .. %d; the current device is %d",
                  kMaxDevices - 1, dev);
    return PATH_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  NoAllocState& s = g_noalloc[dev];
  if (!s.ready) {
    if ((e = cudaDeviceGetAttribute(&s.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&s.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
            cudaSuccess)
      return set_cuda_error(e);
    if (s.cc_major != 10 || s.cc_minor != 3) {
      std::snprintf(g_last_error, sizeof(g_last_error),
                    "libpathattn is built for sm_103a; this device is sm_%d%d", s.cc_major,
                    s.cc_minor);
      return PATH_ERR_UNSUPPORTED;
    }
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess) return set_cuda_error(e);
    s.scratch = static_cast<char*>(p);
    if ((e = cudaGetSymbolAddress(&p, g_noalloc_status)) != cudaSuccess) return set_cuda_error(e);
    s.status = static_cast<int*>(p);
    s.ready = true;
  }
  *out = &s;
  return PATH_OK;
}

}  // namespace

extern "C" int path_attn_fwd_noalloc(const void* q, const void* k, const void* v, const void* w,
                                     const float* beta, const float* logf, float scale,
                                     void* out, float* lse, int* status, int B, int H, int T,
                                     int d, int dtype, void* stream) {
  if (!q || !k || !v || !w || !beta || !out) return PATH_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(w) || !aligned16(beta) ||
      !aligned16(out) || (logf && !aligned16(logf)) || (lse && !aligned16(lse)) ||
      (status && (reinterpret_cast<uintptr_t>(status) & 3u)))
    return PATH_ERR_INVALID_ARG;
  if (!(scale == scale)) return PATH_ERR_INVALID_ARG;
  Geom g;
  int rc = make_geom(B, H, T, d, dtype, logf != nullptr, &g);
  if (rc != PATH_OK) return rc;
  const size_t bytes = workspace_layout(g, nullptr, nullptr);
  if (bytes > PATH_NOALLOC_SCRATCH_BYTES) {
    std::snprintf(g_last_error, sizeof(g_last_error),
                  "path_attn_fwd_noalloc: this problem needs %zu bytes of workspace; the static "
                  "scratch holds %zu",
                  bytes, static_cast<size_t>(PATH_NOALLOC_SCRATCH_BYTES));
    return PATH_ERR_UNSUPPORTED;
  }
  NoAllocState* s = nullptr;
  if ((rc = noalloc_setup(&s)) != PATH_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* word = status ? status : s->status;
  cudaError_t e = cudaMemsetAsync(word, 0, sizeof(int), st);
  if (e != cudaSuccess) return set_cuda_error(e);
  Workspace ws;
  workspace_layout(g, s->scratch, &ws);
  Inputs in{q, k, v, w, beta, logf, scale, out, lse};
  if ((e = launch_prep(g, in, ws, word, st, nullptr)) != cudaSuccess) return set_cuda_error(e);
  e = g.bf16 ? launch_attn_tc(g, in, ws, word, st, nullptr) : launch_attn_f32(g, in, ws, st, nullptr);
  if (e != cudaSuccess) return set_cuda_error(e);
  return PATH_OK;
}

extern "C" int path_attn_noalloc_status(int device, int clear) {
  int prev = 0;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return set_cuda_error(e);
  if ((e = cudaSetDevice(device)) != cudaSuccess) return set_cuda_error(e);
  NoAllocState* s = nullptr;
  int rc = noalloc_setup(&s);
  int word = 0;
  // a synchronous copy to a host int and a memset: nothing is allocated
  if (rc == PATH_OK &&
      ((e = cudaDeviceSynchronize()) != cudaSuccess ||
       (e = cudaMemcpy(&word, s->status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess ||
       (clear && (e = cudaMemset(s->status, 0, sizeof(int))) != cudaSuccess)))
    rc = set_cuda_error(e);
  cudaSetDevice(prev);
  if (rc != PATH_OK) return rc;
  return word == PATH_DEV_OK ? PATH_OK : PATH_ERR_TIMEOUT;
}
