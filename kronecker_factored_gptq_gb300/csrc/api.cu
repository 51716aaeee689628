// C ABI of libbakron.so: validation, workspace layout, the divide-and-conquer
// schedule over tile anti-diagonals, and the launch sequence.
//
// Schedule (summary page "FastKron: Efficient Quantization with
// Kronecker-Factored Hessians", section 3: process the first half of the
// anti-diagonals, propagate their error into the second half, process the
// second half).  The recursion runs over TILE anti-diagonals D = I + J of
// 128 x 128 tiles; every tile order with D increasing rounds an entry after
// all entries to its top-left, which Theorem 3.2 says leaves the result
// unchanged.  rec(D0, D1) with D1 - D0 == 1 is a leaf (all tiles of D in
// parallel, one CTA each); otherwise, with Dm = (D0 + D1) / 2:
//   rec(D0, Dm);
//   stage 1: for every row tile I with tiles in band P = [D0, Dm):
//            Y^T[J', I] = sum_{J in P_I, J <= J'} U_A^T[J', J] E[I, J]^T
//   stage 2: for every tile (I', J') in band Q = [Dm, D1):
//            W~[I', J'] -= sum_{I <= I'} U_B^T[I', I] Y^T[J', I]^T
//   rec(Dm, D1).
// Both stages are dense 128-tile products (the triangular diagonal blocks of
// the factors carry their zeros), listed as work items built here once per
// (M, N) and uploaded into the workspace.
#include <algorithm>
#include <climits>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "internal.cuh"

namespace bakron {
namespace {

constexpr int T = kTile;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Op {
  int kind;                // 0 = leaf, 1 = propagation
  int D, I0, ntiles;       // leaf
  int off1, n1, off2, n2;  // propagation: item ranges of stage 1 and stage 2
  int maxk1, maxk2;        // longest K range (tiles) of each stage
  double flops1, flops2;
};

struct Schedule {
  int M = 0, N = 0;
  std::vector<WorkItem> items;
  std::vector<Op> ops;
};

// Items of one stage are sorted longest-K first so the big tiles start early.
void sort_items(std::vector<WorkItem>& v, size_t from) {
  std::stable_sort(v.begin() + from, v.end(), [](const WorkItem& x, const WorkItem& y) {
    return (x.k1 - x.k0) > (y.k1 - y.k0);
  });
}

void build_prop(Schedule& s, int D0, int Dm, int D1) {
  const int M = s.M, N = s.N;
  Op op{};
  op.kind = 1;
  op.off1 = (int)s.items.size();
  double f1 = 0, f2 = 0;
  int mk1 = 0, mk2 = 0;
  for (int I = 0; I < M; ++I) {
    const int jlo = std::max(D0 - I, 0), jhi = std::min(Dm - I, N);
    if (jlo >= jhi) continue;
    for (int Jp = jlo; Jp < std::min(D1 - I, N); ++Jp) {
      const int lo = std::max(I, Dm - Jp), hi = std::min(M - 1, D1 - 1 - Jp);
      if (lo > hi) continue;  // no tile of Q in column Jp at or below row I
      const int k1 = std::min(jhi, Jp + 1);
      s.items.push_back(WorkItem{Jp, I, jlo, k1});
      f1 += 2.0 * T * T * T * (k1 - jlo);
      mk1 = std::max(mk1, k1 - jlo);
    }
  }
  sort_items(s.items, op.off1);
  op.n1 = (int)s.items.size() - op.off1;
  op.off2 = (int)s.items.size();
  for (int Ip = 0; Ip < M; ++Ip) {
    for (int Jp = std::max(Dm - Ip, 0); Jp < std::min(D1 - Ip, N); ++Jp) {
      const int ilo = std::max(std::max(0, D0 - Jp), D0 - N + 1);
      const int ihi = std::min(Ip, Dm - 1);
      if (ilo > ihi) continue;
      s.items.push_back(WorkItem{Ip, Jp, ilo, ihi + 1});
      f2 += 2.0 * T * T * T * (ihi + 1 - ilo);
      mk2 = std::max(mk2, ihi + 1 - ilo);
    }
  }
  sort_items(s.items, op.off2);
  op.n2 = (int)s.items.size() - op.off2;
  op.flops1 = f1;
  op.flops2 = f2;
  op.maxk1 = mk1;
  op.maxk2 = mk2;
  s.ops.push_back(op);
}

void build_rec(Schedule& s, int D0, int D1) {
  if (D1 - D0 <= 1) {
    Op op{};
    op.kind = 0;
    op.D = D0;
    op.I0 = std::max(0, D0 - s.N + 1);
    op.ntiles = std::min(D0, s.M - 1) - op.I0 + 1;
    s.ops.push_back(op);
    return;
  }
  const int Dm = (D0 + D1) / 2;
  build_rec(s, D0, Dm);
  build_prop(s, D0, Dm, D1);
  build_rec(s, Dm, D1);
}

const Schedule& get_schedule(int M, int N) {
  static std::mutex mu;
  static std::map<std::pair<int, int>, Schedule> cache;
  std::lock_guard<std::mutex> lk(mu);
  auto key = std::make_pair(M, N);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  Schedule s;
  s.M = M;
  s.N = N;
  build_rec(s, 0, M + N - 1);
  return cache.emplace(key, std::move(s)).first->second;
}

struct QLayout {
  int64_t M, N, Mp, Np;
  size_t status, sched, scale, wt, ehi, elo, yhi, ylo, lathi, latlo, lbthi, lbtlo, total;
};

QLayout quantize_layout(int64_t m, int64_t n) {
  QLayout L{};
  L.M = (m + T - 1) / T;
  L.N = (n + T - 1) / T;
  L.Mp = L.M * T;
  L.Np = L.N * T;
  const Schedule& s = get_schedule((int)L.M, (int)L.N);
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 1024); return o; };
  const size_t f = sizeof(float);
  L.status = take(256);
  L.sched = take(sizeof(WorkItem) * (s.items.size() + 1));
  L.scale = take(f * L.Mp);
  L.wt = take(f * L.Mp * L.Np);
  L.ehi = take(f * L.Mp * L.Np);
  L.elo = take(f * L.Mp * L.Np);
  L.yhi = take(f * L.Np * L.Mp);
  L.ylo = take(f * L.Np * L.Mp);
  L.lathi = take(f * L.Np * L.Np);
  L.latlo = take(f * L.Np * L.Np);
  L.lbthi = take(f * L.Mp * L.Mp);
  L.lbtlo = take(f * L.Mp * L.Mp);
  L.total = off;
  return L;
}

struct ALayout {
  size_t status, wt, ebuf, total;
};

ALayout antidiag_layout(int64_t m, int64_t n) {
  ALayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 1024); return o; };
  L.status = take(256);
  L.wt = take(sizeof(float) * m * n);
  L.ebuf = take(sizeof(float) * (m > 0 ? m : 1));
  L.total = off;
  return L;
}

struct PLayout {
  int64_t kp[2];
  size_t status, scal, items[2], C[2], Chi[2], Clo[2], Gihi[2], Gilo[2], GiThi[2], GiTlo[2],
      Thi[2], Tlo[2], total;
};

// Each factor has its own scratch: A and B are prepared concurrently.
PLayout prepare_layout(int64_t n, int64_t m) {
  PLayout L{};
  L.kp[0] = prepare_pad(n);
  L.kp[1] = prepare_pad(m);
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 1024); return o; };
  L.status = take(256);
  L.scal = take(256);
  for (int w = 0; w < 2; ++w) {
    const size_t kk = sizeof(float) * (size_t)L.kp[w] * (size_t)L.kp[w];
    L.items[w] = take(sizeof(WorkItem) * (size_t)(prepare_items_count(L.kp[w]) + 1));
    L.C[w] = take(kk);
    L.Chi[w] = take(kk);
    L.Clo[w] = take(kk);
    L.Gihi[w] = take(kk);
    L.Gilo[w] = take(kk);
    L.GiThi[w] = take(kk);
    L.GiTlo[w] = take(kk);
    L.Thi[w] = take(kk);
    L.Tlo[w] = take(kk);
  }
  L.total = off;
  return L;
}

// A second stream (and fork/join events) per device, created once, on which
// the B factor is prepared while A runs on the caller's stream.
struct AuxStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

cudaError_t aux_stream(AuxStream** out) {
  static std::mutex mu;
  static AuxStream per_dev[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  AuxStream& a = per_dev[dev];
  if (!a.s) {
    if ((e = cudaStreamCreateWithFlags(&a.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  *out = &a;
  return cudaSuccess;
}

#define TRY_CUDA(x)                                        \
  do {                                                     \
    cudaError_t e_ = (x);                                  \
    if (e_ != cudaSuccess) return BAKRON_ERR_CUDA;         \
  } while (0)

bakron_status finish(cudaStream_t s, const DevStatus* dst, DevStatus* host) {
  TRY_CUDA(cudaMemcpyAsync(host, dst, sizeof(DevStatus), cudaMemcpyDeviceToHost, s));
  TRY_CUDA(cudaStreamSynchronize(s));
  return (bakron_status)host->status;
}

bool valid_opts(const bakron_opts& o) {
  return (o.tile == 0 || o.tile == T) && (o.leaf_width == 0 || o.leaf_width == 1) &&
         (o.use_3xtf32 == 0 || o.use_3xtf32 == 1) && o.spin_budget_cycles >= 0 &&
         (o.fault_inject == 0 || o.fault_inject == 1);
}

// Per-launch CUDA events for bakron_opts.times.
struct PhaseTimer {
  bakron_phase_times* out;
  cudaStream_t s;
  std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>> rec;
  PhaseTimer(bakron_phase_times* o, cudaStream_t st) : out(o), s(st) {}
  ~PhaseTimer() {
    for (auto& r : rec) {
      cudaEventDestroy(r.second.first);
      cudaEventDestroy(r.second.second);
    }
  }
  cudaEvent_t begin() {
    if (!out) return nullptr;
    cudaEvent_t a;
    if (cudaEventCreate(&a) != cudaSuccess) return nullptr;
    cudaEventRecord(a, s);
    return a;
  }
  void end(int cat, cudaEvent_t a) {
    if (!out || !a) return;
    cudaEvent_t b;
    if (cudaEventCreate(&b) != cudaSuccess) { cudaEventDestroy(a); return; }
    cudaEventRecord(b, s);
    rec.push_back({cat, {a, b}});
  }
  void collect() {
    if (!out) return;
    for (auto& r : rec) {
      float ms = 0.f;
      cudaEventElapsedTime(&ms, r.second.first, r.second.second);
      switch (r.first) {
        case 0: out->leaf_ms += ms; out->leaf_launches++; break;
        case 1: out->prop1_ms += ms; out->prop_launches++; break;
        case 2: out->prop2_ms += ms; out->prop_launches++; break;
        default: out->other_ms += ms; out->other_launches++; break;
      }
    }
  }
};

bool sizes_ok(int64_t m, int64_t n) { return m >= 1 && n >= 1 && m <= (1 << 20) && n <= (1 << 20); }

}  // namespace
}  // namespace bakron

using namespace bakron;

extern "C" {

void bakron_default_opts(bakron_opts* o) {
  if (!o) return;
  std::memset(o, 0, sizeof(*o));
  o->tile = T;
  o->leaf_width = 1;
  o->use_3xtf32 = 1;
  o->spin_budget_cycles = 4000000000LL;
  o->fault_inject = 0;
  o->times = nullptr;
}

const char* bakron_status_string(int st) {
  switch (st) {
    case BAKRON_OK: return "ok";
    case BAKRON_ERR_INVALID_ARG: return "invalid argument";
    case BAKRON_ERR_NOT_PD: return "factor is not positive definite";
    case BAKRON_ERR_NONFINITE: return "non-finite input or intermediate value";
    case BAKRON_ERR_CODE_RANGE: return "code outside the int8 range";
    case BAKRON_ERR_TIMEOUT: return "bounded device wait timed out";
    case BAKRON_ERR_UNSUPPORTED: return "unsupported device or configuration";
    case BAKRON_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int bakron_version(void) { return 10000; }

int64_t bakron_kernel_launches(void) { return (int64_t)bakron::launches_so_far(); }

bakron_status bakron_workspace_size(int64_t m, int64_t n, const bakron_opts* opts, size_t* bytes) {
  if (!bytes || !sizes_ok(m, n)) return BAKRON_ERR_INVALID_ARG;
  if (opts && !valid_opts(*opts)) return BAKRON_ERR_INVALID_ARG;
  const QLayout q = quantize_layout(m, n);
  const ALayout a = antidiag_layout(m, n);
  *bytes = std::max(q.total, a.total);
  return BAKRON_OK;
}

bakron_status bakron_prepare_workspace_size(int64_t n, int64_t m, size_t* bytes) {
  if (!bytes || n < 0 || m < 0 || (n == 0 && m == 0) || n > (1 << 20) || m > (1 << 20))
    return BAKRON_ERR_INVALID_ARG;
  *bytes = prepare_layout(n, m).total;
  return BAKRON_OK;
}

bakron_status bakron_rowscale(const float* W, int64_t m, int64_t n, int qmax, float* scale,
                              void* stream) {
  if (!W || !scale || !sizes_ok(m, n) || qmax < 1) return BAKRON_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  TRY_CUDA(launch_rowscale(W, m, n, qmax, scale, s));
  TRY_CUDA(cudaStreamSynchronize(s));
  return BAKRON_OK;
}

bakron_status bakron_prepare(const float* A, int64_t n, float damp_A, const float* B, int64_t m,
                             float damp_B, float* UA, float* UB, float* LA, float* LB,
                             int64_t* info, void* ws, size_t ws_bytes, void* stream) {
  if (!A || n < 1 || !UA || !ws) return BAKRON_ERR_INVALID_ARG;
  if (B && (m < 1 || !UB)) return BAKRON_ERR_INVALID_ARG;
  if (!B) m = 0;
  if (!(damp_A >= 0.f) || !(damp_B >= 0.f)) return BAKRON_ERR_INVALID_ARG;
  if (n > (1 << 20) || m > (1 << 20)) return BAKRON_ERR_INVALID_ARG;
  const PLayout L = prepare_layout(n, m);
  if (ws_bytes < L.total) return BAKRON_ERR_INVALID_ARG;
  if (!prop_tc_supported()) return BAKRON_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  char* base = (char*)ws;
  DevStatus* st = (DevStatus*)(base + L.status);
  TRY_CUDA(cudaMemsetAsync(st, 0, sizeof(DevStatus), s));
  TRY_CUDA(cudaMemsetAsync(st->info, 0x7f, sizeof(st->info), s));
  AuxStream* aux = nullptr;
  if (B) {
    TRY_CUDA(aux_stream(&aux));
    TRY_CUDA(cudaEventRecord(aux->fork, s));
    TRY_CUDA(cudaStreamWaitEvent(aux->s, aux->fork, 0));
  }
  for (int which = 0; which < 2; ++which) {
    const float* X = which == 0 ? A : B;
    const int64_t k = which == 0 ? n : m;
    if (!X || k == 0) continue;
    PrepareFactorArgs pa{};
    pa.X = X; pa.k = k; pa.damp = which == 0 ? damp_A : damp_B;
    pa.U = which == 0 ? UA : UB;
    pa.L = which == 0 ? LA : LB;
    pa.C = (float*)(base + L.C[which]);
    pa.Chi = (float*)(base + L.Chi[which]);
    pa.Clo = (float*)(base + L.Clo[which]);
    pa.Gihi = (float*)(base + L.Gihi[which]);
    pa.Gilo = (float*)(base + L.Gilo[which]);
    pa.GiThi = (float*)(base + L.GiThi[which]);
    pa.GiTlo = (float*)(base + L.GiTlo[which]);
    pa.Thi = (float*)(base + L.Thi[which]);
    pa.Tlo = (float*)(base + L.Tlo[which]);
    pa.items = (WorkItem*)(base + L.items[which]);
    pa.scal = (float*)(base + L.scal) + which;
    pa.kp = L.kp[which];
    pa.which = which;
    pa.st = st;
    TRY_CUDA(run_prepare_factor(pa, which == 0 ? s : aux->s));
  }
  if (aux) {
    TRY_CUDA(cudaEventRecord(aux->join, aux->s));
    TRY_CUDA(cudaStreamWaitEvent(s, aux->join, 0));
  }
  DevStatus h{};
  bakron_status r = finish(s, st, &h);
  if (info) {
    for (int w = 0; w < 2; ++w) {
      const int64_t k = w == 0 ? n : m;
      const long long f = h.info[w];
      info[w] = (k > 0 && f >= 0 && f < k) ? (k - 1 - f) : -1;
    }
  }
  return r;
}

bakron_status bakron_quantize(const float* W, int64_t m, int64_t n, const float* UA, const float* UB,
                              const float* scale, int qmin, int qmax, float* V, int8_t* codes,
                              float* preround, const bakron_opts* opts_in, void* ws,
                              size_t ws_bytes, void* stream) {
  bakron_opts o;
  bakron_default_opts(&o);
  if (opts_in) o = *opts_in;
  if (!valid_opts(o)) return BAKRON_ERR_INVALID_ARG;
  if (!W || !UA || !UB || !scale || !V || !codes || !ws) return BAKRON_ERR_INVALID_ARG;
  if (!sizes_ok(m, n) || qmin > qmax) return BAKRON_ERR_INVALID_ARG;
  const QLayout L = quantize_layout(m, n);
  if (ws_bytes < L.total) return BAKRON_ERR_INVALID_ARG;
  if (o.use_3xtf32 && !prop_tc_supported()) return BAKRON_ERR_UNSUPPORTED;
  const Schedule& sch = get_schedule((int)L.M, (int)L.N);
  cudaStream_t s = (cudaStream_t)stream;
  char* base = (char*)ws;
  DevStatus* st = (DevStatus*)(base + L.status);
  WorkItem* items = (WorkItem*)(base + L.sched);
  float* sp = (float*)(base + L.scale);
  float* wt = (float*)(base + L.wt);
  float* ehi = (float*)(base + L.ehi);
  float* elo = (float*)(base + L.elo);
  float* yhi = (float*)(base + L.yhi);
  float* ylo = (float*)(base + L.ylo);
  float* lathi = (float*)(base + L.lathi);
  float* latlo = (float*)(base + L.latlo);
  float* lbthi = (float*)(base + L.lbthi);
  float* lbtlo = (float*)(base + L.lbtlo);
  if (o.times) std::memset(o.times, 0, sizeof(*o.times));
  PhaseTimer pt(o.times, s);

  TRY_CUDA(cudaMemsetAsync(st, 0, sizeof(DevStatus), s));
  if (!sch.items.empty())
    TRY_CUDA(cudaMemcpyAsync(items, sch.items.data(), sizeof(WorkItem) * sch.items.size(),
                             cudaMemcpyHostToDevice, s));
  {
    cudaEvent_t ev = pt.begin();
    TRY_CUDA(launch_check_finite(scale, m, st, s));
    TRY_CUDA(launch_pad_scale(scale, m, sp, L.Mp, s));
    TRY_CUDA(launch_pad_matrix(W, m, n, wt, L.Mp, L.Np, s));
    TRY_CUDA(launch_transpose_split(UA, n, lathi, latlo, L.Np, s));
    TRY_CUDA(launch_transpose_split(UB, m, lbthi, lbtlo, L.Mp, s));
    pt.end(3, ev);
  }
  LeafArgs la{};
  la.wt = wt; la.ldw = L.Np;
  la.lat_hi = lathi; la.lat_lo = latlo; la.lda = L.Np;
  la.lbt_hi = lbthi; la.lbt_lo = lbtlo; la.ldb = L.Mp;
  la.scale = sp;
  la.e_hi = ehi; la.e_lo = elo;
  la.V = V; la.codes = codes; la.preround = preround;
  la.m = m; la.n = n; la.qmin = qmin; la.qmax = qmax;
  la.st = st;
  PropArgs p1{};
  p1.A_hi = lathi; p1.A_lo = latlo; p1.lda = L.Np; p1.a_rows = L.Np;
  p1.B_hi = ehi; p1.B_lo = elo; p1.ldb = L.Np; p1.b_rows = L.Mp;
  p1.out_hi = yhi; p1.out_lo = ylo; p1.ldo = L.Mp;
  p1.stage = 1;
  p1.st = st;
  PropArgs p2{};
  p2.A_hi = lbthi; p2.A_lo = lbtlo; p2.lda = L.Mp; p2.a_rows = L.Mp;
  p2.B_hi = yhi; p2.B_lo = ylo; p2.ldb = L.Mp; p2.b_rows = L.Np;
  p2.wt = wt; p2.ldw = L.Np;
  p2.stage = 2;
  p2.st = st;
  for (const Op& op : sch.ops) {
    if (op.kind == 0) {
      la.D = op.D;
      la.I0 = op.I0;
      cudaEvent_t ev = pt.begin();
      TRY_CUDA(launch_leaf(la, op.ntiles, s));
      pt.end(0, ev);
    } else {
      p1.items = items + op.off1; p1.n_items = op.n1; p1.max_k = op.maxk1;
      p2.items = items + op.off2; p2.n_items = op.n2; p2.max_k = op.maxk2;
      cudaEvent_t ev = pt.begin();
      TRY_CUDA(o.use_3xtf32 ? launch_prop_tc(p1, s) : launch_prop_simt(p1, s));
      pt.end(1, ev);
      ev = pt.begin();
      TRY_CUDA(o.use_3xtf32 ? launch_prop_tc(p2, s) : launch_prop_simt(p2, s));
      pt.end(2, ev);
      if (o.times) o.times->prop_flops += op.flops1 + op.flops2;
    }
  }
  DevStatus h{};
  bakron_status r = finish(s, st, &h);
  pt.collect();
  return r;
}

bakron_status bakron_quantize_antidiag(const float* W, int64_t m, int64_t n, const float* UA,
                                       const float* UB, const float* scale, int qmin, int qmax,
                                       float* V, int8_t* codes, float* preround,
                                       const int8_t* guide_codes, float guide_tol,
                                       int64_t* overrides, const bakron_opts* opts_in, void* ws,
                                       size_t ws_bytes, void* stream) {
  bakron_opts o;
  bakron_default_opts(&o);
  if (opts_in) o = *opts_in;
  if (!valid_opts(o)) return BAKRON_ERR_INVALID_ARG;
  if (!W || !UA || !UB || !scale || !V || !codes || !ws) return BAKRON_ERR_INVALID_ARG;
  if (!sizes_ok(m, n) || qmin > qmax) return BAKRON_ERR_INVALID_ARG;
  if (guide_codes && !(guide_tol >= 0.f)) return BAKRON_ERR_INVALID_ARG;
  const ALayout L = antidiag_layout(m, n);
  if (ws_bytes < L.total) return BAKRON_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  char* base = (char*)ws;
  DevStatus* st = (DevStatus*)(base + L.status);
  TRY_CUDA(cudaMemsetAsync(st, 0, sizeof(DevStatus), s));
  TRY_CUDA(launch_check_finite(scale, m, st, s));
  TRY_CUDA(cudaMemcpyAsync(base + L.wt, W, sizeof(float) * m * n, cudaMemcpyDeviceToDevice, s));
  AntidiagArgs a{};
  a.wt = (float*)(base + L.wt);
  a.UA = UA; a.UB = UB; a.scale = scale;
  a.ebuf = (float*)(base + L.ebuf);
  a.V = V; a.codes = codes; a.preround = preround;
  a.guide = guide_codes; a.guide_tol = guide_tol;
  a.m = m; a.n = n; a.qmin = qmin; a.qmax = qmax;
  a.budget = o.spin_budget_cycles > 0 ? o.spin_budget_cycles : 4000000000LL;
  a.fault_inject = o.fault_inject;
  a.st = st;
  int unsupported = 0;
  TRY_CUDA(launch_antidiag(a, &unsupported, s));
  if (unsupported) {
    TRY_CUDA(cudaStreamSynchronize(s));
    return BAKRON_ERR_UNSUPPORTED;
  }
  DevStatus h{};
  bakron_status r = finish(s, st, &h);
  if (overrides) *overrides = (int64_t)h.overrides;
  return r;
}

}  // extern "C"
