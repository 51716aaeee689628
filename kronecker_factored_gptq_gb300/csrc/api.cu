// C ABI of libbakron.so: validation, workspace layout, the divide-and-conquer
// schedule over tile anti-diagonals, and the launch sequence.
//
// Schedule (summary page "FastKron: Efficient Quantization with
// Kronecker-Factored Hessians", section 3: process the first half of the
// anti-diagonals, propagate their error into the second half, process the
// second half).  The recursion runs over TILE anti-diagonals D = I + J of
// 128 x 128 tiles; every tile order with D increasing rounds an entry after
// all entries to its top-left, which Theorem 3.2 says leaves the result
// unchanged.
//
// The error reaches later tiles in the row-accumulator form: with
//   R[I, J'] = sum_{J <= J'} E[I, J] U_A[J, J']       (row I's accumulator)
// target (I', J') receives  W~[I', J'] -= sum_{I < I'} U_B[I, I']^T R[I, J']
// + U_B[I', I']^T R^-[I', J'], R^- the sum over J < J' only.  The library
// keeps R (transposed, R^T[J', I], in fp32 and split for the tensor cores)
// for the whole solve and builds it incrementally, so each row update
// E[I, J] U_A[J, J'] and each push of a complete R[I, J'] into a target is
// computed once:
//
//  * near products, on the critical stream between leaf D - 1 and leaf D,
//    for each target (I, J) of diagonal D: stage 1 adds the row updates
//    from diagonal D - 1 into R, E[I, J-1] U_A[J-1, J] into R[I, J] (now
//    R^-[I, J]) and the own term E[I-1, J] U_A[J, J] into R[I-1, J] (now
//    complete); stage 2 applies U_B[I-1, I]^T R[I-1, J] + U_B[I, I]^T R[I, J];
//  * propagation: rec(D0, D1) with D1 - D0 >= 2 and Dm = (D0 + D1) / 2 runs
//    rec(D0, Dm), then, for the sources [max(D0 - 1, 0), Dm - 1) and the
//    targets [Dm, D1): stage 1, the row updates from the source tiles E[I, J]
//    into the R tiles (I, J') of the target band; stage 2, the pushes of the
//    complete R tiles (I, J') of the source band into the targets (I', J')
//    below them; then rec(Dm, D1).  A (source, target) pair of either kind
//    with t - s >= 2 is handled by the one node whose split separates s + 1
//    from t; pairs with t - s = 1 are the near products.  The propagation
//    starts after the near products of diagonal Dm - 1 (the own terms that
//    complete the R tiles of diagonal Dm - 2), beside leaf Dm - 1: no
//    propagation sits between two leaves on the critical stream.
//
// Both stages are lists of dense 128-tile products (the triangular diagonal
// blocks of the factors carry their zeros):
//   stage 1: R^T[J', I] += sum_{J in the band, row I} U_A^T[J', J] E[I, J]^T
//   stage 2: W~[I', J'] -= sum_{I in the band, column J'} U_B^T[I', I] R^T[J', I]^T
// split by the tile anti-diagonal of the R tile (stage 1) or target (stage
// 2) into chunks [Dm, Dm+1), [Dm+1, Dm+2), [Dm+2, Dm+4), ...: every chunk is
// due at the near products of its first diagonal, which wait for it; the
// chunk due next runs on a high-priority stream, the later ones lower.  A
// chunk's two stages touch different tiles and go out as one launch.
#include <algorithm>
#include <climits>
#include <cstring>
#include <map>
#include <mutex>
#include <thread>
#include <utility>
#include <vector>

#include "internal.cuh"

namespace bakron {
namespace {

constexpr int T = kTile;
// Propagation lanes (three streams each).
constexpr int kMaxDepth = 24;
// A propagation chunk whose first target is at most this many leaves after
// the propagation's start runs at middle priority, a later one at the lowest.
#ifndef BAKRON_MID_SLACK
#define BAKRON_MID_SLACK 15
#endif
constexpr int kMidSlack = BAKRON_MID_SLACK;
// Chunks of priority class <= kFuseClass (0 urgent, 1 middle, 2 lowest; -1
// none) launch their row updates and pushes together (measured at 8192^2:
// all classes 17.77 ms, urgent and middle 17.78, none 17.88, urgent only
// 18.03; 4096^2 and 4096 x 14336 gain 1.4% with all classes).
#ifndef BAKRON_FUSE_CLASS
#define BAKRON_FUSE_CLASS 2
#endif
constexpr int kFuseClass = BAKRON_FUSE_CLASS;
// Source diagonals the near products reach back (diagonal D - 1); the
// propagations cover every pair further apart.
constexpr int kNear = 1;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Chunk {
  int off1, n1, maxk1;  // stage-1 items
  int off, n, maxk;     // stage-2 items
  int dlo, dhi;         // target tile anti-diagonals [dlo, dhi)
  double flops1, flops;
};

// Ops in the order the executor issues them: for each diagonal D, the near
// products into D (D >= 1), leaf D, then the propagation whose last source
// is D (the node split at D + 2), if there is one.
struct Op {
  int kind;                // 0 = leaf, 1 = propagation, 2 = near products
  int D;                   // leaf / near: the tile anti-diagonal; propagation:
                           // its last source diagonal (after whose leaf it starts)
  int I0, ntiles;          // leaf: first row tile and tile count
  int s0, s1;              // propagation: source diagonals [s0, s1)
  int depth;               // propagation: its lane (streams)
  int chunk0, nchunks;     // near: one chunk; propagation: its chunks
};

struct Schedule {
  int M = 0, N = 0, max_depth = 0;
  std::vector<WorkItem> items;
  std::vector<Op> ops;
  std::vector<Chunk> chunks;
};

// Items of one stage are sorted longest-K first so the big tiles start early.
void sort_items(std::vector<WorkItem>& v, size_t from) {
  std::stable_sort(v.begin() + from, v.end(), [](const WorkItem& x, const WorkItem& y) {
    return (x.k1 - x.k0) > (y.k1 - y.k0);
  });
}

// Propagation of the sources [S0, S1) into the targets [T0, T1) (T0 >= S1 + 1).
Op build_prop(Schedule& s, int S0, int S1, int T0, int T1, int depth) {
  const int M = s.M, N = s.N;
  Op op{};
  op.kind = 1;
  op.D = S1 - 1;
  op.s0 = S0;
  op.s1 = S1;
  op.depth = depth;
  s.max_depth = std::max(s.max_depth, depth);
  op.chunk0 = (int)s.chunks.size();
  // chunk boundaries over the target band [T0, T1)
  std::vector<std::pair<int, int>> bounds;
  for (int lo = T0, width = 1; lo < T1;) {
    const int hi = std::min(T1, lo + width);
    bounds.emplace_back(lo, hi);
    lo = hi;
    if (lo > T0 + 1) width *= 2;
  }
  auto chunk_of = [&](int d) {
    int c = 0;
    while (bounds[c].second <= d) ++c;
    return c;
  };
  std::vector<std::vector<WorkItem>> s1(bounds.size()), s2(bounds.size());
  // stage 1: R tile (I, J') of the target band += the source tiles of row I
  // (all at least two columns left of J')
  for (int I = 0; I < M; ++I) {
    const int jlo = std::max(S0 - I, 0), jhi = std::min(S1 - I, N);
    if (jlo >= jhi) continue;
    for (int Jp = std::max(T0 - I, 0); Jp < std::min(T1 - I, N); ++Jp) {
      const int c = chunk_of(I + Jp);
      s1[c].push_back(WorkItem{Jp, I, jlo, jhi});
    }
  }
  // stage 2: target (I', J') of the target band -= the complete R tiles of
  // column J' in the source band (all at least two rows above I')
  for (int Jp = 0; Jp < N; ++Jp) {
    const int ilo = std::max(S0 - Jp, 0), ihi = std::min(S1 - Jp, M);
    if (ilo >= ihi) continue;
    for (int Ip = std::max(T0 - Jp, 0); Ip < std::min(T1 - Jp, M); ++Ip) {
      const int c = chunk_of(Ip + Jp);
      s2[c].push_back(WorkItem{Ip, Jp, ilo, ihi});
    }
  }
  for (size_t ci = 0; ci < bounds.size(); ++ci) {
    Chunk c{};
    c.dlo = bounds[ci].first;
    c.dhi = bounds[ci].second;
    auto take = [&](const std::vector<WorkItem>& src, int& off, int& n, int& maxk, double& flops) {
      off = (int)s.items.size();
      for (const WorkItem& w : src) {
        s.items.push_back(w);
        maxk = std::max(maxk, w.k1 - w.k0);
        flops += 2.0 * T * T * T * (w.k1 - w.k0);
      }
      sort_items(s.items, off);
      n = (int)s.items.size() - off;
    };
    take(s1[ci], c.off1, c.n1, c.maxk1, c.flops1);
    take(s2[ci], c.off, c.n, c.maxk, c.flops);
    s.chunks.push_back(c);
  }
  op.nchunks = (int)s.chunks.size() - op.chunk0;
  return op;
}

// Near products into the tiles of diagonal D from diagonal D - 1, in the
// row-accumulator form: for a target (I, J) the stage-1 items add
// E[I, J-1] U_A[J-1, J] into R^T[J, I] and E[I-1, J] U_A[J, J] into
// R^T[J, I-1] (source columns J - 1 and J); the stage-2 item of (I, J) sums
// U_B^T[I, I''] R^T[J, I''] over the rows I'' = I - 1, I.  Targets of one
// diagonal sit in distinct columns J, so the R tiles of one launch are
// distinct.
Op build_near(Schedule& s, int D) {
  const int M = s.M, N = s.N;
  Op op{};
  op.kind = 2;
  op.D = D;
  op.chunk0 = (int)s.chunks.size();
  op.nchunks = 1;
  const int I0 = std::max(0, D - N + 1), I1 = std::min(D, M - 1);
  Chunk c{};
  c.dlo = D;
  c.dhi = D + 1;
  c.off1 = (int)s.items.size();
  for (int I = I0; I <= I1; ++I) {
    const int J = D - I;
    for (int k = 0; k <= kNear && I - k >= 0; ++k) {
      const int j0 = std::max(0, k == 0 ? J - kNear : J - kNear + k);
      const int j1 = k == 0 ? J : J + 1;   // exclusive
      if (j1 <= j0) continue;
      s.items.push_back(WorkItem{J, I - k, j0, j1});
      c.flops1 += 2.0 * T * T * T * (j1 - j0);
      c.maxk1 = std::max(c.maxk1, j1 - j0);
    }
  }
  c.n1 = (int)s.items.size() - c.off1;
  c.off = (int)s.items.size();
  for (int I = I0; I <= I1; ++I) {
    const int J = D - I;
    const int k0 = std::max(0, I - kNear), k1 = J >= 1 ? I + 1 : I;
    if (k1 <= k0) continue;
    s.items.push_back(WorkItem{I, J, k0, k1});
    c.flops += 2.0 * T * T * T * (k1 - k0);
    c.maxk = std::max(c.maxk, k1 - k0);
  }
  c.n = (int)s.items.size() - c.off;
  s.chunks.push_back(c);
  return op;
}

// The propagations of the recursion, each filed under its last source
// diagonal.  A wide source band is split into up to four parts of about
// kSplitWidth diagonals, propagated separately: both kinds of pairs are
// partitioned by their source diagonal (a row update by its error tile, a
// push by its accumulator tile), so each pair is still handled once and no
// work repeats, and each part starts right after the near products that
// follow its own last source.  The early parts of a wide band then run
// beside many leaves, and the part due at the band's first target has at
// most kSplitWidth-deep products (measured at 8192^2: width 16 17.8 ms,
// 8 and 32 17.9 ms, no split 18.0 ms).
#ifndef BAKRON_SPLIT_WIDTH
#define BAKRON_SPLIT_WIDTH 16
#endif
constexpr int kSplitWidth = BAKRON_SPLIT_WIDTH;   // 0: no split

void build_rec(Schedule& s, int D0, int D1, int depth, std::vector<std::vector<Op>>& prop_after,
               bool split) {
  if (D1 - D0 <= 1) return;
  const int Dm = (D0 + D1) / 2;
  build_rec(s, D0, Dm, depth + 1, prop_after, split);
  const int S0 = std::max(D0 - kNear, 0), S1 = Dm - kNear;
  if (S1 > S0) {
    const int w = S1 - S0;
    const int width = kSplitWidth > 0 ? kSplitWidth : 1;
    const int parts = split && kSplitWidth > 0 ? std::min(4, std::max(1, (w + width / 2) / width)) : 1;
    for (int p = 0; p < parts; ++p) {
      const int a = S0 + (int)((int64_t)w * p / parts), b = S0 + (int)((int64_t)w * (p + 1) / parts);
      if (b > a) prop_after[b - 1].push_back(build_prop(s, a, b, Dm, D1, depth));
    }
  }
  build_rec(s, Dm, D1, depth + 1, prop_after, split);
}

// Streams of each propagation ("lane", kept in Op.depth): the lowest lane
// whose previous propagation has finished.  A propagation's
// chunks all complete before the leaf of the last chunk's first target, and
// a propagation starts after the leaf of its last source, so a lane is free
// for a propagation starting after leaf D once its previous one's last chunk
// targets a diagonal <= D.  Returns false if more than kMaxLanes are needed.
bool assign_lanes(Schedule& s, int max_lanes) {
  std::vector<int> free_at;   // per lane: first leaf after which it is free
  int top = 0;
  for (Op& op : s.ops) {
    if (op.kind != 1) continue;
    int lane = -1;
    for (int l = 0; l < (int)free_at.size(); ++l)
      if (free_at[l] <= op.D) { lane = l; break; }
    if (lane < 0) {
      lane = (int)free_at.size();
      if (lane >= max_lanes) return false;
      free_at.push_back(0);
    }
    op.depth = lane;
    free_at[lane] = s.chunks[op.chunk0 + op.nchunks - 1].dlo;
    top = std::max(top, lane);
  }
  s.max_depth = top;
  return true;
}

void build_schedule(Schedule& s, int max_lanes) {
  for (int split = 1; split >= 0; --split) {
    s.items.clear();
    s.ops.clear();
    s.chunks.clear();
    s.max_depth = 0;
    const int ND = s.M + s.N - 1;
    std::vector<std::vector<Op>> prop_after(ND);
    build_rec(s, 0, ND, 0, prop_after, split != 0);
    for (int D = 0; D < ND; ++D) {
      // the propagations whose last source is diagonal D - 1 follow the near
      // products of diagonal D, which complete that diagonal's R tiles
      if (D >= 1) {
        s.ops.push_back(build_near(s, D));
        for (const Op& op : prop_after[D - 1]) s.ops.push_back(op);
      }
      Op leaf{};
      leaf.kind = 0;
      leaf.D = D;
      leaf.I0 = std::max(0, D - s.N + 1);
      leaf.ntiles = std::min(D, s.M - 1) - leaf.I0 + 1;
      s.ops.push_back(leaf);
    }
    if (assign_lanes(s, max_lanes)) return;
  }
}

// Propagation chunks whose updates of W~ a later writer of the same tiles
// must follow, each with the target range [dlo, dhi) it updates (tile
// anti-diagonals, or column tiles on the one-sided path).  Before a stream
// updates the diagonals [lo, hi) (a chunk's stage 2, the near products, a
// leaf) it waits for every listed chunk that overlaps them, so each W~ tile
// receives its updates in one fixed order and the fp32 result is the same on
// every run.  A chunk whose whole range lies inside [lo, hi) is then dropped:
// a writer after it overlaps [lo, hi) as well and follows it through the new
// writer's own event (or through the stream, for the leaf and the near
// products, which are the last writers of their diagonal).  A chunk that
// reaches past [lo, hi) stays listed for the writers of its other diagonals.
// The critical stream waits for a listed chunk once: its later work follows
// that wait in stream order, and a kernel launched with no event wait in
// front of it can start early (programmatic dependent launch).
struct PendingChunks {
  struct Item {
    cudaEvent_t ev;
    int dlo, dhi;
    bool crit_waited;
  };
  std::vector<Item> v;
  void add(cudaEvent_t ev, int dlo, int dhi) { v.push_back(Item{ev, dlo, dhi, false}); }
  cudaError_t order_before(cudaStream_t cs, int lo, int hi, bool critical = false) {
    size_t w = 0;
    for (size_t i = 0; i < v.size(); ++i) {
      const bool overlap = v[i].dlo < hi && v[i].dhi > lo;
      if (overlap && !(critical && v[i].crit_waited)) {
        const cudaError_t e = cudaStreamWaitEvent(cs, v[i].ev, 0);
        if (e != cudaSuccess) return e;
        if (critical) v[i].crit_waited = true;
      }
      if (!(overlap && v[i].dlo >= lo && v[i].dhi <= hi)) v[w++] = v[i];
    }
    v.resize(w);
    return cudaSuccess;
  }
};

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
  build_schedule(s, kMaxDepth);
  return cache.emplace(key, std::move(s)).first->second;
}

// Schedule of the one-sided (B = I) solve: divide and conquer over column
// tiles.  rows_rec(J0, J1) is a leaf (column tile J0 of every row tile) if
// J1 - J0 == 1; otherwise rows_rec(J0, Jm), the propagation
// W~[I, J'] -= sum_{J in [J0, Jm)} E[I, J] U_A[J, J'] for J' in [Jm, J1),
// rows_rec(Jm, J1).  The propagation is split by target column into chunks
// [Jm, Jm+1), [Jm+1, Jm+2), [Jm+2, Jm+4), ...: the first (what the next
// leaf needs) on the critical stream, the others deferred.
struct RowsOp {
  int kind;            // 0 = leaf, 1 = propagation
  int J, depth;        // leaf column tile; recursion depth
  int chunk0, nchunks;
};

struct RowsSchedule {
  int M = 0, N = 0, max_depth = 0;
  std::vector<WorkItem> items;
  std::vector<RowsOp> ops;
  std::vector<Chunk> chunks;   // stage-2 items only (off, n, maxk, dlo, dhi, flops)
};

void build_rows_rec(RowsSchedule& s, int J0, int J1, int depth) {
  if (J1 - J0 <= 1) {
    s.ops.push_back(RowsOp{0, J0, depth, 0, 0});
    return;
  }
  const int Jm = (J0 + J1) / 2;
  build_rows_rec(s, J0, Jm, depth + 1);
  RowsOp op{1, 0, depth, (int)s.chunks.size(), 0};
  s.max_depth = std::max(s.max_depth, depth);
  for (int lo = Jm, width = 1; lo < J1;) {
    const int hi = std::min(J1, lo + width);
    Chunk c{};
    c.dlo = lo;
    c.dhi = hi;
    c.off = (int)s.items.size();
    for (int Jp = lo; Jp < hi; ++Jp)
      for (int I = 0; I < s.M; ++I) s.items.push_back(WorkItem{I, Jp, J0, Jm});
    c.n = (int)s.items.size() - c.off;
    c.maxk = Jm - J0;
    c.flops = 2.0 * T * T * T * (double)(Jm - J0) * c.n;
    s.chunks.push_back(c);
    lo = hi;
    if (lo > Jm + 1) width *= 2;
  }
  op.nchunks = (int)s.chunks.size() - op.chunk0;
  s.ops.push_back(op);
  build_rows_rec(s, Jm, J1, depth + 1);
}

const RowsSchedule& get_rows_schedule(int M, int N) {
  static std::mutex mu;
  static std::map<std::pair<int, int>, RowsSchedule> cache;
  std::lock_guard<std::mutex> lk(mu);
  auto key = std::make_pair(M, N);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  RowsSchedule s;
  s.M = M;
  s.N = N;
  build_rows_rec(s, 0, N, 0);
  return cache.emplace(key, std::move(s)).first->second;
}

// The work lists of a solve on stream s: read in place from the caller's
// plan (after a header check that sets BAKRON_ERR_INVALID_ARG on a mismatch),
// or written into the workspace region ws_dst (kernel parameters, see
// fill_items).
cudaError_t stage_schedule(const void* plan, bool two_sided, int M, int N, WorkItem* ws_dst,
                           DevStatus* st, cudaStream_t s, const WorkItem** out) {
  const Schedule& sch = get_schedule(M, N);
  const RowsSchedule& rs = get_rows_schedule(M, N);
  if (plan) {
    cudaError_t e = launch_plan_check(plan, M, N, (int64_t)sch.items.size(), (int64_t)rs.items.size(),
                                      st, s);
    if (e != cudaSuccess) return e;
    const WorkItem* base = (const WorkItem*)((const char*)plan + kPlanHeaderBytes);
    *out = two_sided ? base : base + sch.items.size();
    return cudaSuccess;
  }
  *out = ws_dst;
  return two_sided ? fill_items(sch.items.data(), sch.items.size(), ws_dst, s)
                   : fill_items(rs.items.data(), rs.items.size(), ws_dst, s);
}

size_t plan_bytes(int M, int N) {
  return kPlanHeaderBytes +
         sizeof(WorkItem) * (get_schedule(M, N).items.size() + get_rows_schedule(M, N).items.size());
}

struct QLayout {
  int64_t M, N, Mp, Np;
  size_t status, sched, scale, zero, wt, ehi, elo, racc, rhi, rlo, lathi, latlo, lbthi, lbtlo, total;
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
  const RowsSchedule& rs = get_rows_schedule((int)L.M, (int)L.N);
  L.sched = take(sizeof(WorkItem) * (std::max(s.items.size(), rs.items.size()) + 1));
  // grid scales and zero points, padded rows x groups (at most one group per
  // 32 columns)
  const size_t ngmax = (size_t)std::max<int64_t>(1, (n + 31) / 32);
  L.scale = take(f * L.Mp * ngmax);
  L.zero = take(f * L.Mp * ngmax);
  L.wt = take(f * L.Mp * L.Np);
  L.ehi = take(f * L.Mp * L.Np);
  L.elo = take(f * L.Mp * L.Np);
  // the row accumulators R^T (Np x Mp): fp32 running sums, and split
  L.racc = take(f * L.Np * L.Mp);
  L.rhi = take(f * L.Np * L.Mp);
  L.rlo = take(f * L.Np * L.Mp);
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

// Streams of the factor preparation, per device, created once: four per
// factor (the chain, its lookahead, the bulk updates, the rows of G^{-1}), so
// the two factors are prepared side by side, plus fork/join events and a pool
// of reusable events.  Held under a lock for the whole (synchronous) call.
struct PrepStreams {
  cudaStream_t main[2] = {};       // high priority: the diagonal-block chains
  cudaStream_t side[2] = {};       // lower priority: lookahead panels and updates
  cudaStream_t bulk[2] = {};       // lowest priority: updates needed two steps later
  cudaStream_t inv[2] = {};        // lowest priority: the block rows of G^{-1}
  cudaEvent_t fork = nullptr, join = nullptr;
  std::vector<cudaEvent_t> events;
  std::mutex mu;
};

cudaError_t prep_streams(PrepStreams** out) {
  static std::mutex mu;
  static PrepStreams per_dev[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  PrepStreams& a = per_dev[dev];
  if (!a.main[0]) {
    int lo = 0, hi = 0;
    if ((e = cudaDeviceGetStreamPriorityRange(&lo, &hi)) != cudaSuccess) return e;
    for (int w = 0; w < 2; ++w) {
      if ((e = cudaStreamCreateWithPriority(&a.main[w], cudaStreamNonBlocking, hi)) != cudaSuccess)
        return e;
      if ((e = cudaStreamCreateWithPriority(&a.side[w], cudaStreamNonBlocking, (lo + hi) / 2)) !=
          cudaSuccess)
        return e;
      if ((e = cudaStreamCreateWithPriority(&a.bulk[w], cudaStreamNonBlocking, lo)) != cudaSuccess)
        return e;
      if ((e = cudaStreamCreateWithPriority(&a.inv[w], cudaStreamNonBlocking, lo)) != cudaSuccess)
        return e;
    }
    if ((e = cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  *out = &a;
  return cudaSuccess;
}

cudaError_t prep_events(PrepStreams* ps, size_t n) {
  while (ps->events.size() < n) {
    cudaEvent_t e;
    cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    if (r != cudaSuccess) return r;
    ps->events.push_back(e);
  }
  return cudaSuccess;
}

// Streams of the solve, per device, created once: a high-priority critical
// stream (leaves, near products; the one-sided path's urgent chunks) and per
// propagation lane an urgent stream (the chunk the next leaf waits for) just
// below it in priority, a middle-priority and a lowest-priority stream (the
// chunks due later), plus a pool of reusable events.  Calls are
// synchronous, so the pool is reused per call.
struct SolveStreams {
  cudaStream_t crit = nullptr;
  cudaStream_t urg[kMaxDepth] = {};
  cudaStream_t mid[kMaxDepth] = {};
  cudaStream_t side[kMaxDepth] = {};
  std::vector<cudaEvent_t> events;
  std::mutex mu;
};

// Stream sets per device: slot 0 serves the single-problem calls, slots
// 0 .. kSlots-1 the problems of a batch (one set per concurrent problem).
constexpr int kSlots = 8;

cudaError_t solve_streams(SolveStreams** out, int slot = 0) {
  static std::mutex mu;
  static SolveStreams per_dev[64][kSlots];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || slot < 0 || slot >= kSlots) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  SolveStreams& ss = per_dev[dev][slot];
  if (!ss.crit) {
    int lo = 0, hi = 0;
    if ((e = cudaDeviceGetStreamPriorityRange(&lo, &hi)) != cudaSuccess) return e;
    // greater priority = smaller number; urgent chunks one step below the
    // critical stream when the device has the levels
    const int urg = hi < lo ? hi + 1 : hi;
    const int mid = (urg + lo) / 2;
    cudaStream_t c = nullptr, u[kMaxDepth] = {}, md[kMaxDepth] = {}, sd[kMaxDepth] = {};
    e = cudaStreamCreateWithPriority(&c, cudaStreamNonBlocking, hi);
    for (int d = 0; d < kMaxDepth && e == cudaSuccess; ++d) {
      e = cudaStreamCreateWithPriority(&u[d], cudaStreamNonBlocking, urg);
      if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&md[d], cudaStreamNonBlocking, mid);
      if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&sd[d], cudaStreamNonBlocking, lo);
    }
    if (e != cudaSuccess) {
      if (c) cudaStreamDestroy(c);
      for (int d = 0; d < kMaxDepth; ++d) {
        if (u[d]) cudaStreamDestroy(u[d]);
        if (md[d]) cudaStreamDestroy(md[d]);
        if (sd[d]) cudaStreamDestroy(sd[d]);
      }
      return e;
    }
    for (int d = 0; d < kMaxDepth; ++d) {
      ss.urg[d] = u[d];
      ss.mid[d] = md[d];
      ss.side[d] = sd[d];
    }
    ss.crit = c;
  }
  *out = &ss;
  return cudaSuccess;
}

// After a failed enqueue: wait for whatever the call already queued on its
// stream set, so nothing of it still reads or writes the caller's memory or
// the workspace when the error is returned.
void drain_solve_streams(SolveStreams* ss) {
  cudaStreamSynchronize(ss->crit);
  for (int d = 0; d < kMaxDepth; ++d) {
    cudaStreamSynchronize(ss->urg[d]);
    cudaStreamSynchronize(ss->mid[d]);
    cudaStreamSynchronize(ss->side[d]);
  }
}

cudaError_t pool_event(SolveStreams* ss, size_t idx, cudaEvent_t* ev) {
  while (ss->events.size() <= idx) {
    cudaEvent_t e;
    cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    if (r != cudaSuccess) return r;
    ss->events.push_back(e);
  }
  *ev = ss->events[idx];
  return cudaSuccess;
}

#define TRY_CUDA(x)                                        \
  do {                                                     \
    cudaError_t e_ = (x);                                  \
    if (e_ != cudaSuccess) return BAKRON_ERR_CUDA;         \
  } while (0)

// After work was forked onto a solve stream set `ss`: on failure, wait for
// what is already queued there before returning the error.
#define TRY_SOLVE(x)                                       \
  do {                                                     \
    cudaError_t e_ = (x);                                  \
    if (e_ != cudaSuccess) {                               \
      drain_solve_streams(ss);                             \
      return BAKRON_ERR_CUDA;                              \
    }                                                      \
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

// Per-launch CUDA events for bakron_opts.times: a pair around a launch on
// the stream it is enqueued on.
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
  cudaEvent_t begin(cudaStream_t on = nullptr) {
    if (!out) return nullptr;
    cudaEvent_t a;
    if (cudaEventCreate(&a) != cudaSuccess) return nullptr;
    cudaEventRecord(a, on ? on : s);
    return a;
  }
  void end(int cat, cudaEvent_t a, cudaStream_t on = nullptr) {
    if (!out || !a) return;
    cudaEvent_t b;
    if (cudaEventCreate(&b) != cudaSuccess) { cudaEventDestroy(a); return; }
    cudaEventRecord(b, on ? on : s);
    rec.push_back({cat, {a, b}});
  }
  void adopt(PhaseTimer& other) {
    for (auto& r : other.rec) rec.push_back(r);
    other.rec.clear();
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
        case 4: out->near_ms += ms; out->near_launches++; break;
        default: out->other_ms += ms; out->other_launches++; break;
      }
    }
  }
};

bool sizes_ok(int64_t m, int64_t n) {
  return m >= 1 && n >= 1 && m <= (1 << 20) && n <= (1 << 20) &&
         ((m + T - 1) / T) * ((n + T - 1) / T) <= kMaxTiles;
}

// The one-sided solve (U_B = I): see RowsSchedule.  Arguments validated by
// bakron_quantize; the workspace layout is the two-sided one (its row
// accumulator and U_B^T regions stay unused).
// One problem of a batch: the stream set it runs on (locked by the caller),
// that set's event pool position, and what the call leaves for the caller:
// the event recorded at its end on the critical stream and its status block.
struct BatchCtx {
  SolveStreams* ss;
  size_t* nev;
  cudaEvent_t done;
  DevStatus* st;
};

// A validated grid: scale / zero point per (row, group of `group` columns).
struct GridIn {
  const float* scale;
  const float* zero;   // nullable: zero points of 0
  int64_t group, ng;
};

bakron_status quantize_rows(const float* W, int64_t m, int64_t n, const float* UA, const GridIn& gr,
                            int qmin, int qmax, float* V, int8_t* codes, float* preround,
                            const bakron_opts& o, void* ws, cudaStream_t s, BatchCtx* bctx) {
  const QLayout L = quantize_layout(m, n);
  const RowsSchedule& sch = get_rows_schedule((int)L.M, (int)L.N);
  SolveStreams* ss = bctx ? bctx->ss : nullptr;
  if (!ss) TRY_CUDA(solve_streams(&ss));
  std::unique_lock<std::mutex> slk(ss->mu, std::defer_lock);
  if (!bctx) slk.lock();
  size_t nev_own = 0;
  size_t& nev = bctx ? *bctx->nev : nev_own;
  auto next_event = [&](cudaEvent_t* ev) { return pool_event(ss, nev++, ev); };
  char* base = (char*)ws;
  DevStatus* st = (DevStatus*)(base + L.status);
  const WorkItem* items = (const WorkItem*)(base + L.sched);
  float* sp = (float*)(base + L.scale);
  float* zp = (float*)(base + L.zero);
  float* wt = (float*)(base + L.wt);
  float* ehi = (float*)(base + L.ehi);
  float* elo = (float*)(base + L.elo);
  float* lathi = (float*)(base + L.lathi);
  float* latlo = (float*)(base + L.latlo);
  if (o.times) std::memset(o.times, 0, sizeof(*o.times));
  cudaStream_t cs = ss->crit;
  {
    cudaEvent_t ev;
    TRY_SOLVE(next_event(&ev));
    TRY_SOLVE(cudaEventRecord(ev, s));
    TRY_SOLVE(cudaStreamWaitEvent(cs, ev, 0));
  }
  TRY_SOLVE(cudaMemsetAsync(st, 0, sizeof(DevStatus), cs));
  TRY_SOLVE(stage_schedule(o.plan, false, (int)L.M, (int)L.N, (WorkItem*)(base + L.sched), st, cs,
                           &items));
  PhaseTimer pt(o.times, cs);
  {
    cudaEvent_t ev = pt.begin();
    TRY_SOLVE(launch_check_finite(gr.scale, m * gr.ng, st, cs));
    TRY_SOLVE(launch_check_zero(gr.zero, m * gr.ng, qmin, qmax, st, cs));
    TRY_SOLVE(launch_pad_grid(gr.scale, gr.zero, m, gr.ng, sp, zp, L.Mp, cs));
    TRY_SOLVE(launch_pad_matrix(W, m, n, wt, L.Mp, L.Np, cs));
    TRY_SOLVE(launch_transpose_split(UA, n, lathi, latlo, L.Np, cs));
    pt.end(3, ev);
  }
  LeafArgs la{};
  la.wt = wt; la.ldw = L.Np;
  la.lat_hi = lathi; la.lat_lo = latlo; la.lda = L.Np;
  la.scale = sp;
  la.zero = zp;
  la.group = gr.group;
  la.ngroups = gr.ng;
  la.e_hi = ehi; la.e_lo = elo;
  la.round_lo = 1;
  la.V = V; la.codes = codes; la.preround = preround;
  la.m = m; la.n = n; la.qmin = qmin; la.qmax = qmax;
  la.st = st;
  PendingChunks pending;
  for (const RowsOp& op : sch.ops) {
    if (op.kind == 0) {
      TRY_SOLVE(pending.order_before(cs, op.J, op.J + 1, true));
      la.D = op.J;
      la.I0 = 0;
      la.pdl = op.J > 0;   // the first leaf reads the factor the kernel before it wrote
      cudaEvent_t ev = pt.begin();
      TRY_SOLVE(launch_rows_leaf(la, (int)L.M, cs));
      pt.end(0, ev);
      continue;
    }
    PropArgs p2{};
    p2.A_hi = ehi; p2.A_lo = elo; p2.lda = L.Np; p2.a_rows = L.Mp;
    p2.B_hi = lathi; p2.B_lo = latlo; p2.ldb = L.Np; p2.b_rows = L.Np;
    p2.wt = wt; p2.ldw = L.Np;
    p2.stage = 2;
    p2.st = st;
    if (op.nchunks > 0)
      TRY_SOLVE(pending.order_before(cs, sch.chunks[op.chunk0].dlo,
                                    sch.chunks[op.chunk0 + op.nchunks - 1].dhi, true));
    for (int c = 0; c < op.nchunks; ++c) {
      const Chunk& ch = sch.chunks[op.chunk0 + c];
      if (o.times) o.times->prop_flops += ch.flops;
      const bool urgent = c == 0;
      cudaStream_t cstr = urgent ? cs : ss->side[op.depth];
      if (c == 1) {
        // the deferred chunks start once the leaves they read have finished
        cudaEvent_t ev;
        TRY_SOLVE(next_event(&ev));
        TRY_SOLVE(cudaEventRecord(ev, cs));
        TRY_SOLVE(cudaStreamWaitEvent(cstr, ev, 0));
      }
      PhaseTimer side_pt(o.times, cstr);
      PhaseTimer* tm = urgent ? &pt : &side_pt;
      p2.items = items + ch.off; p2.n_items = ch.n; p2.max_k = ch.maxk;
      p2.pdl = urgent;
      cudaEvent_t ev = tm->begin();
      TRY_SOLVE(o.use_3xtf32 ? launch_prop_tc(p2, cstr) : launch_prop_simt(p2, cstr));
      tm->end(2, ev);
      if (!urgent) {
        pt.adopt(side_pt);
        cudaEvent_t done;
        TRY_SOLVE(next_event(&done));
        TRY_SOLVE(cudaEventRecord(done, cstr));
        pending.add(done, ch.dlo, ch.dhi);
      }
    }
  }
  {
    cudaEvent_t ev;
    TRY_SOLVE(next_event(&ev));
    TRY_SOLVE(cudaEventRecord(ev, cs));
    if (bctx) {
      bctx->done = ev;
      bctx->st = st;
      return BAKRON_OK;
    }
    TRY_SOLVE(cudaStreamWaitEvent(s, ev, 0));
  }
  DevStatus h{};
  bakron_status r = finish(s, st, &h);
  pt.collect();
  return r;
}

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
  o->plan = nullptr;
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

int bakron_version(void) { return 20000; }

int64_t bakron_kernel_launches(void) { return (int64_t)bakron::launches_so_far(); }

bakron_status bakron_schedule_export(int kind, int64_t M, int64_t N, int32_t* out, int64_t cap,
                                     int64_t* len) {
  try {
    if (!len || cap < 0 || (cap > 0 && !out)) return BAKRON_ERR_INVALID_ARG;
    if (kind == BAKRON_SCHEDULE_PREPARE ? (M < 1 || M > kMaxOrder / T)
                                        : (M < 1 || N < 1 || M > 8192 || N > 8192 || M * N > kMaxTiles))
      return BAKRON_ERR_INVALID_ARG;
    std::vector<int32_t> v;
    auto items = [&](const std::vector<WorkItem>& it) {
      for (const WorkItem& w : it) {
        v.push_back(w.r);
        v.push_back(w.c);
        v.push_back(w.k0);
        v.push_back(w.k1);
      }
    };
    auto chunks = [&](const std::vector<Chunk>& ch) {
      for (const Chunk& c : ch) {
        v.push_back(c.dlo);
        v.push_back(c.dhi);
        v.push_back(c.off1);
        v.push_back(c.n1);
        v.push_back(c.off);
        v.push_back(c.n);
      }
    };
    if (kind == BAKRON_SCHEDULE_SOLVE) {
      const Schedule& s = get_schedule((int)M, (int)N);
      v.push_back((int32_t)s.ops.size());
      v.push_back((int32_t)s.chunks.size());
      v.push_back((int32_t)s.items.size());
      for (const Op& op : s.ops) {
        // leaf: (0, D, I0, ntiles, 0, 0, 0); near: (2, D, 0, 0, 0, chunk, 1);
        // propagation: (1, last source, s0, s1, depth, chunk0, nchunks)
        int32_t rec[7] = {op.kind, op.D, 0, 0, 0, 0, 0};
        if (op.kind == 0) {
          rec[2] = op.I0;
          rec[3] = op.ntiles;
        } else {
          if (op.kind == 1) {
            rec[2] = op.s0;
            rec[3] = op.s1;
            rec[4] = op.depth;
          }
          rec[5] = op.chunk0;
          rec[6] = op.nchunks;
        }
        v.insert(v.end(), rec, rec + 7);
      }
      chunks(s.chunks);
      items(s.items);
    } else if (kind == BAKRON_SCHEDULE_ROWS) {
      const RowsSchedule& s = get_rows_schedule((int)M, (int)N);
      v.push_back((int32_t)s.ops.size());
      v.push_back((int32_t)s.chunks.size());
      v.push_back((int32_t)s.items.size());
      for (const RowsOp& op : s.ops) {
        const int32_t rec[7] = {op.kind, op.kind == 0 ? op.J : 0, 0, op.kind == 0 ? (int32_t)M : 0,
                                op.depth, op.kind == 1 ? op.chunk0 : 0, op.kind == 1 ? op.nchunks : 0};
        v.insert(v.end(), rec, rec + 7);
      }
      chunks(s.chunks);
      items(s.items);
    } else if (kind == BAKRON_SCHEDULE_PREPARE) {
      prepare_schedule_export(M, v);
    } else {
      return BAKRON_ERR_INVALID_ARG;
    }
    *len = (int64_t)v.size();
    if (cap >= *len && *len > 0) std::memcpy(out, v.data(), sizeof(int32_t) * v.size());
    return BAKRON_OK;
  } catch (...) {
    return BAKRON_ERR_INVALID_ARG;   // host allocation failure
  }
}

bakron_status bakron_workspace_size(int64_t m, int64_t n, const bakron_opts* opts, size_t* bytes) {
  try {
    if (!bytes || !sizes_ok(m, n)) return BAKRON_ERR_INVALID_ARG;
    if (opts && !valid_opts(*opts)) return BAKRON_ERR_INVALID_ARG;
    const QLayout q = quantize_layout(m, n);
    const ALayout a = antidiag_layout(m, n);
    *bytes = std::max(q.total, a.total);
    return BAKRON_OK;
  } catch (...) {
    return BAKRON_ERR_INVALID_ARG;   // host allocation failure
  }
}

bakron_status bakron_plan_size(int64_t m, int64_t n, size_t* bytes) {
  try {
    if (!bytes || !sizes_ok(m, n)) return BAKRON_ERR_INVALID_ARG;
    *bytes = plan_bytes((int)((m + T - 1) / T), (int)((n + T - 1) / T));
    return BAKRON_OK;
  } catch (...) {
    return BAKRON_ERR_INVALID_ARG;   // host allocation failure
  }
}

bakron_status bakron_plan_init(int64_t m, int64_t n, void* plan, size_t plan_bytes_given,
                               void* stream) {
  try {
    if (!plan || !sizes_ok(m, n) || ((uintptr_t)plan & 15)) return BAKRON_ERR_INVALID_ARG;
    const int M = (int)((m + T - 1) / T), N = (int)((n + T - 1) / T);
    if (plan_bytes_given < plan_bytes(M, N)) return BAKRON_ERR_INVALID_ARG;
    const Schedule& sch = get_schedule(M, N);
    const RowsSchedule& rs = get_rows_schedule(M, N);
    // the header as the first 16 work-item slots, then both lists
    std::vector<WorkItem> all(kPlanHeaderBytes / sizeof(WorkItem) + sch.items.size() +
                              rs.items.size());
    PlanHeader h{};
    h.magic = kPlanMagic;
    h.version = kPlanVersion;
    h.M = M;
    h.N = N;
    h.n_solve = (long long)sch.items.size();
    h.n_rows = (long long)rs.items.size();
    h.off_solve = (long long)(kPlanHeaderBytes / sizeof(WorkItem));
    h.off_rows = h.off_solve + h.n_solve;
    std::memcpy(all.data(), &h, sizeof(h));
    std::copy(sch.items.begin(), sch.items.end(), all.begin() + h.off_solve);
    std::copy(rs.items.begin(), rs.items.end(), all.begin() + h.off_rows);
    cudaStream_t s = (cudaStream_t)stream;
    TRY_CUDA(fill_items(all.data(), all.size(), (WorkItem*)plan, s));
    TRY_CUDA(cudaStreamSynchronize(s));
    return BAKRON_OK;
  } catch (...) {
    return BAKRON_ERR_INVALID_ARG;   // host allocation failure
  }
}

bakron_status bakron_prepare_workspace_size(int64_t n, int64_t m, size_t* bytes) {
  try {
    if (!bytes || n < 0 || m < 0 || (n == 0 && m == 0) || n > kMaxOrder || m > kMaxOrder)
      return BAKRON_ERR_INVALID_ARG;
    *bytes = prepare_layout(n, m).total;
    return BAKRON_OK;
  } catch (...) {
    return BAKRON_ERR_INVALID_ARG;   // host allocation failure
  }
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
  try {
    if (!A || n < 1 || !UA || !ws) return BAKRON_ERR_INVALID_ARG;
    if (B && (m < 1 || !UB)) return BAKRON_ERR_INVALID_ARG;
    if (!B) m = 0;
    if (!(damp_A >= 0.f) || !(damp_B >= 0.f)) return BAKRON_ERR_INVALID_ARG;
    if (n > kMaxOrder || m > kMaxOrder) return BAKRON_ERR_INVALID_ARG;
    const PLayout L = prepare_layout(n, m);
    if (ws_bytes < L.total) return BAKRON_ERR_INVALID_ARG;
    if (!prop_tc_supported()) return BAKRON_ERR_UNSUPPORTED;
    cudaStream_t s = (cudaStream_t)stream;
    char* base = (char*)ws;
    DevStatus* st = (DevStatus*)(base + L.status);
    TRY_CUDA(cudaMemsetAsync(st, 0, sizeof(DevStatus), s));
    TRY_CUDA(cudaMemsetAsync(st->info, 0x7f, sizeof(st->info), s));
    PrepStreams* ps = nullptr;
    TRY_CUDA(prep_streams(&ps));
    std::lock_guard<std::mutex> plk(ps->mu);
    const size_t ev_per = 5 * (size_t)(std::max(L.kp[0], L.kp[1]) / T + 1);
    TRY_CUDA(prep_events(ps, 2 * ev_per));
    TRY_CUDA(cudaEventRecord(ps->fork, s));
    // enqueue one factor's preparation on its own streams, after the fork
    auto enqueue = [&](int which) -> cudaError_t {
      const float* X = which == 0 ? A : B;
      const int64_t k = which == 0 ? n : m;
      cudaStream_t fs = ps->main[which];
      cudaError_t e;
      if ((e = cudaStreamWaitEvent(fs, ps->fork, 0)) != cudaSuccess) return e;
      // the other streams start after the factor's stream reaches this point
      cudaEvent_t start = ps->events[which * ev_per + ev_per - 1];
      if ((e = cudaEventRecord(start, fs)) != cudaSuccess) return e;
      for (cudaStream_t o : {ps->side[which], ps->bulk[which], ps->inv[which]})
        if ((e = cudaStreamWaitEvent(o, start, 0)) != cudaSuccess) return e;
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
      pa.side = ps->side[which];
      pa.bulk = ps->bulk[which];
      pa.inv = ps->inv[which];
      pa.ev = ps->events.data() + which * ev_per;
      if ((e = run_prepare_factor(pa, fs)) != cudaSuccess) return e;
      return cudaEventRecord(ps->events[which * ev_per + ev_per - 2], fs);
    };
    // Each factor's chain takes milliseconds of host time to enqueue, so with
    // two factors B is enqueued from a second host thread and both chains start
    // on the device together.
    cudaError_t err[2] = {cudaSuccess, cudaSuccess};
    const bool two = B && m > 0;
    if (two) {
      int dev = 0;
      TRY_CUDA(cudaGetDevice(&dev));
      std::thread tb;
      bool threaded = true;
      try {
        tb = std::thread([&] {
          err[1] = cudaSetDevice(dev);
          if (err[1] == cudaSuccess) err[1] = enqueue(1);
        });
      } catch (...) {
        threaded = false;   // no thread to be had: enqueue B after A
      }
      err[0] = enqueue(0);
      if (threaded) tb.join();
      else err[1] = enqueue(1);
    } else {
      err[0] = enqueue(0);
    }
    TRY_CUDA(err[0]);
    TRY_CUDA(err[1]);
    // join the chains back onto the caller's stream
    for (int which = 0; which < (two ? 2 : 1); ++which)
      TRY_CUDA(cudaStreamWaitEvent(s, ps->events[which * ev_per + ev_per - 2], 0));
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
  } catch (...) {
    return BAKRON_ERR_INVALID_ARG;   // host allocation failure
  }
}

}  // extern "C"

namespace bakron {
namespace {
bakron_status quantize_impl(const float* W, int64_t m, int64_t n, const float* UA, const float* UB,
                            const GridIn& gr, int qmin, int qmax, float* V, int8_t* codes,
                            float* preround, const bakron_opts* opts_in, void* ws, size_t ws_bytes,
                            void* stream, BatchCtx* bctx = nullptr) {
  bakron_opts o;
  bakron_default_opts(&o);
  if (opts_in) o = *opts_in;
  if (bctx) o.times = nullptr;
  if (!valid_opts(o)) return BAKRON_ERR_INVALID_ARG;
  if (!W || !UA || !gr.scale || !V || !codes || !ws) return BAKRON_ERR_INVALID_ARG;
  if (!sizes_ok(m, n) || qmin > qmax) return BAKRON_ERR_INVALID_ARG;
  const QLayout L = quantize_layout(m, n);
  if (ws_bytes < L.total) return BAKRON_ERR_INVALID_ARG;
  if (o.use_3xtf32 && !prop_tc_supported()) return BAKRON_ERR_UNSUPPORTED;
  if (!UB)
    return quantize_rows(W, m, n, UA, gr, qmin, qmax, V, codes, preround, o, ws,
                         (cudaStream_t)stream, bctx);
  const Schedule& sch = get_schedule((int)L.M, (int)L.N);
  cudaStream_t s = (cudaStream_t)stream;
  SolveStreams* ss = bctx ? bctx->ss : nullptr;
  if (!ss) TRY_CUDA(solve_streams(&ss));
  std::unique_lock<std::mutex> slk(ss->mu, std::defer_lock);
  if (!bctx) slk.lock();
  size_t nev_own = 0;
  size_t& nev = bctx ? *bctx->nev : nev_own;
  auto next_event = [&](cudaEvent_t* ev) { return pool_event(ss, nev++, ev); };
  char* base = (char*)ws;
  DevStatus* st = (DevStatus*)(base + L.status);
  const WorkItem* items = (const WorkItem*)(base + L.sched);
  float* sp = (float*)(base + L.scale);
  float* zp = (float*)(base + L.zero);
  float* wt = (float*)(base + L.wt);
  float* ehi = (float*)(base + L.ehi);
  float* elo = (float*)(base + L.elo);
  float* lathi = (float*)(base + L.lathi);
  float* latlo = (float*)(base + L.latlo);
  float* lbthi = (float*)(base + L.lbthi);
  float* lbtlo = (float*)(base + L.lbtlo);
  if (o.times) std::memset(o.times, 0, sizeof(*o.times));

  // fork onto the critical stream
  cudaStream_t cs = ss->crit;
  {
    cudaEvent_t ev;
    TRY_SOLVE(next_event(&ev));
    TRY_SOLVE(cudaEventRecord(ev, s));
    TRY_SOLVE(cudaStreamWaitEvent(cs, ev, 0));
  }
  TRY_SOLVE(cudaMemsetAsync(st, 0, sizeof(DevStatus), cs));
  TRY_SOLVE(stage_schedule(o.plan, true, (int)L.M, (int)L.N, (WorkItem*)(base + L.sched), st, cs,
                           &items));
  PhaseTimer pt(o.times, cs);
  {
    cudaEvent_t ev = pt.begin();
    TRY_SOLVE(launch_check_finite(gr.scale, m * gr.ng, st, cs));
    TRY_SOLVE(launch_check_zero(gr.zero, m * gr.ng, qmin, qmax, st, cs));
    TRY_SOLVE(launch_pad_grid(gr.scale, gr.zero, m, gr.ng, sp, zp, L.Mp, cs));
    TRY_SOLVE(launch_pad_matrix(W, m, n, wt, L.Mp, L.Np, cs));
    TRY_SOLVE(launch_transpose_split(UA, n, lathi, latlo, L.Np, cs));
    TRY_SOLVE(launch_transpose_split(UB, m, lbthi, lbtlo, L.Mp, cs));
    pt.end(3, ev);
  }
  LeafArgs la{};
  la.wt = wt; la.ldw = L.Np;
  la.lat_hi = lathi; la.lat_lo = latlo; la.lda = L.Np;
  la.lbt_hi = lbthi; la.lbt_lo = lbtlo; la.ldb = L.Mp;
  la.scale = sp;
  la.zero = zp;
  la.group = gr.group;
  la.ngroups = gr.ng;
  la.e_hi = ehi; la.e_lo = elo;
  la.round_lo = o.use_3xtf32;
  la.V = V; la.codes = codes; la.preround = preround;
  la.m = m; la.n = n; la.qmin = qmin; la.qmax = qmax;
  la.st = st;
  float* racc = (float*)(base + L.racc);
  float* rhi = (float*)(base + L.rhi);
  float* rlo = (float*)(base + L.rlo);
  // stage 1: R^T += U_A^T E^T (fp32 running sums, written back and split);
  // stage 2: W~ -= U_B^T R
  PropArgs p1{};
  p1.A_hi = lathi; p1.A_lo = latlo; p1.lda = L.Np; p1.a_rows = L.Np;
  p1.B_hi = ehi; p1.B_lo = elo; p1.ldb = L.Np; p1.b_rows = L.Mp;
  p1.out_hi = rhi; p1.out_lo = rlo; p1.acc = racc; p1.ldo = L.Mp;
  p1.stage = 1;
  p1.st = st;
  PropArgs p2{};
  p2.A_hi = lbthi; p2.A_lo = lbtlo; p2.lda = L.Mp; p2.a_rows = L.Mp;
  p2.B_hi = rhi; p2.B_lo = rlo; p2.ldb = L.Mp; p2.b_rows = L.Np;
  p2.wt = wt; p2.ldw = L.Np;
  p2.stage = 2;
  p2.st = st;
  auto launch = [&](PropArgs pa, int off, int nit, int maxk, cudaStream_t str) {
    pa.items = items + off; pa.n_items = nit; pa.max_k = maxk;
    pa.pdl = str == cs;
    return o.use_3xtf32 ? launch_prop_tc(pa, str) : launch_prop_simt(pa, str);
  };
  // R starts at zero: its fp32 sums are cleared on a lane stream beside the
  // first leaf; the critical stream waits before the first near products,
  // which every later writer of R follows
  cudaEvent_t ev_rzero = nullptr;
  {
    cudaEvent_t ev;
    TRY_SOLVE(next_event(&ev));
    TRY_SOLVE(cudaEventRecord(ev, cs));
    TRY_SOLVE(cudaStreamWaitEvent(ss->side[0], ev, 0));
    TRY_SOLVE(cudaMemsetAsync(racc, 0, sizeof(float) * (size_t)L.Np * (size_t)L.Mp, ss->side[0]));
    TRY_SOLVE(next_event(&ev_rzero));
    TRY_SOLVE(cudaEventRecord(ev_rzero, ss->side[0]));
  }
  // Writers of W~ tiles (pending) and of R tiles (rpending), each keyed by
  // the tile anti-diagonals they write; every later writer or reader of the
  // same diagonals waits for them (a fixed order of the updates).
  PendingChunks pending, rpending;
  cudaEvent_t ev_near1 = nullptr;   // after the last near products' stage 1
  bool first_near = true;
  auto enqueue = [&]() -> cudaError_t {
    cudaError_t e;
    for (const Op& op : sch.ops) {
      if (op.kind == 2) {
        // near products into diagonal op.D, after every chunk that writes
        // its R tiles (stage 1) or its W~ tiles
        const Chunk& ch = sch.chunks[op.chunk0];
        if (first_near) {
          if ((e = cudaStreamWaitEvent(cs, ev_rzero, 0)) != cudaSuccess) return e;
          first_near = false;
        }
        if ((e = rpending.order_before(cs, op.D, op.D + 1, true)) != cudaSuccess) return e;
        if ((e = pending.order_before(cs, op.D, op.D + 1, true)) != cudaSuccess) return e;
        if (o.times) o.times->prop_flops += ch.flops1 + ch.flops;
        if (ch.n1 > 0) {
          cudaEvent_t ev = pt.begin();
          if ((e = launch(p1, ch.off1, ch.n1, ch.maxk1, cs)) != cudaSuccess) return e;
          pt.end(4, ev);
        }
        if ((e = next_event(&ev_near1)) != cudaSuccess) return e;
        if ((e = cudaEventRecord(ev_near1, cs)) != cudaSuccess) return e;
        if (ch.n > 0) {
          cudaEvent_t ev = pt.begin();
          if ((e = launch(p2, ch.off, ch.n, ch.maxk, cs)) != cudaSuccess) return e;
          pt.end(4, ev);
        }
        continue;
      }
      if (op.kind == 0) {
        if ((e = pending.order_before(cs, op.D, op.D + 1, true)) != cudaSuccess) return e;
        la.D = op.D;
        la.I0 = op.I0;
        // the first leaf reads the factors the kernel directly before it
        // wrote; a leaf also waiting on deferred chunks (events) still waits
        // for them in full, the relaxation covers only the previous kernel on
        // this stream
        la.pdl = op.D > 0;
        cudaEvent_t ev = pt.begin();
        if ((e = launch_leaf(la, op.ntiles, cs)) != cudaSuccess) return e;
        pt.end(0, ev);
        continue;
      }
      // propagation: starts after the near products' stage 1 right before it
      // (its sources' leaves have run and its source band's R tiles are
      // complete).  Each chunk goes to a stream of the propagation's lane
      // chosen by its slack, the leaves between the propagation's start
      // (after leaf op.D) and its first target: the next leaf's chunk to the
      // urgent stream, the chunks due within kMidSlack leaves to a
      // middle-priority stream, the rest to the lowest; so far-off chunks of
      // a large propagation cannot hold the SMs that a near deadline needs.
      // The row updates (stage 1) and the pushes (stage 2) of a chunk write
      // different tiles and read nothing the other writes; they share the
      // class's stream (measured: separate streams were slower).
      cudaStream_t lane_str[3] = {ss->urg[op.depth], ss->mid[op.depth], ss->side[op.depth]};
      bool started[3] = {false, false, false};
      auto stream_for = [&](int k, cudaStream_t* out) -> cudaError_t {
        *out = lane_str[k];
        if (started[k]) return cudaSuccess;
        started[k] = true;
        return cudaStreamWaitEvent(*out, ev_near1, 0);
      };
      for (int c = 0; c < op.nchunks; ++c) {
        const Chunk& ch = sch.chunks[op.chunk0 + c];
        if (o.times) o.times->prop_flops += ch.flops1 + ch.flops;
        const int slack = ch.dlo - op.D - 1;
        const int k = slack <= 1 ? 0 : (slack <= kMidSlack ? 1 : 2);
        if (o.use_3xtf32 && k <= kFuseClass && ch.n1 > 0 && ch.n > 0) {
          // both stages in one launch (they touch different tiles), after the
          // earlier writers of the chunk's R and W~ tiles
          cudaStream_t cstr;
          if ((e = stream_for(k, &cstr)) != cudaSuccess) return e;
          if ((e = rpending.order_before(cstr, ch.dlo, ch.dhi)) != cudaSuccess) return e;
          if ((e = pending.order_before(cstr, ch.dlo, ch.dhi)) != cudaSuccess) return e;
          PropArgs a = p1, b = p2;
          a.items = items + ch.off1; a.n_items = ch.n1; a.max_k = ch.maxk1;
          b.items = items + ch.off; b.n_items = ch.n; b.max_k = ch.maxk;
          cudaEvent_t ev = pt.begin(cstr);
          if ((e = launch_prop_tc2(a, b, cstr)) != cudaSuccess) return e;
          pt.end(1, ev, cstr);
          cudaEvent_t done;
          if ((e = next_event(&done)) != cudaSuccess) return e;
          if ((e = cudaEventRecord(done, cstr)) != cudaSuccess) return e;
          rpending.add(done, ch.dlo, ch.dhi);
          pending.add(done, ch.dlo, ch.dhi);
          continue;
        }
        if (ch.n1 > 0) {
          cudaStream_t cstr;
          if ((e = stream_for(k, &cstr)) != cudaSuccess) return e;
          // after the earlier writers of the same R tiles (fixed order)
          if ((e = rpending.order_before(cstr, ch.dlo, ch.dhi)) != cudaSuccess) return e;
          cudaEvent_t ev = pt.begin(cstr);
          if ((e = launch(p1, ch.off1, ch.n1, ch.maxk1, cstr)) != cudaSuccess) return e;
          pt.end(1, ev, cstr);
          cudaEvent_t done;
          if ((e = next_event(&done)) != cudaSuccess) return e;
          if ((e = cudaEventRecord(done, cstr)) != cudaSuccess) return e;
          rpending.add(done, ch.dlo, ch.dhi);
        }
        if (ch.n > 0) {
          cudaStream_t cstr;
          if ((e = stream_for(k, &cstr)) != cudaSuccess) return e;
          // after the earlier updates of the same W~ tiles (fixed order)
          if ((e = pending.order_before(cstr, ch.dlo, ch.dhi)) != cudaSuccess) return e;
          cudaEvent_t ev = pt.begin(cstr);
          if ((e = launch(p2, ch.off, ch.n, ch.maxk, cstr)) != cudaSuccess) return e;
          pt.end(2, ev, cstr);
          cudaEvent_t done;
          if ((e = next_event(&done)) != cudaSuccess) return e;
          if ((e = cudaEventRecord(done, cstr)) != cudaSuccess) return e;
          pending.add(done, ch.dlo, ch.dhi);
        }
      }
    }
    return cudaSuccess;
  };
  if (enqueue() != cudaSuccess) {
    drain_solve_streams(ss);
    return BAKRON_ERR_CUDA;
  }
  // join back onto the caller's stream (every chunk was waited for by the
  // near products or the leaf of its diagonals, so the critical stream is
  // last)
  {
    cudaEvent_t ev;
    if (next_event(&ev) != cudaSuccess || cudaEventRecord(ev, cs) != cudaSuccess) {
      drain_solve_streams(ss);
      return BAKRON_ERR_CUDA;
    }
    if (bctx) {
      bctx->done = ev;
      bctx->st = st;
      return BAKRON_OK;
    }
    if (cudaStreamWaitEvent(s, ev, 0) != cudaSuccess) {
      drain_solve_streams(ss);
      return BAKRON_ERR_CUDA;
    }
  }
  DevStatus h{};
  bakron_status r = finish(s, st, &h);
  pt.collect();
  return r;
}


// The grid of a b-bit base quantizer: `group` columns per group (0 or >= n:
// one group per row; otherwise a multiple of 32).  Returns the group count,
// or -1 for an invalid group size.
int64_t grid_groups(int64_t n, int64_t group) {
  if (group <= 0 || group >= n) return 1;
  if (group % 32 != 0) return -1;
  return (n + group - 1) / group;
}
}  // namespace
}  // namespace bakron

extern "C" {

bakron_status bakron_quantize(const float* W, int64_t m, int64_t n, const float* UA, const float* UB,
                              const float* scale, int qmin, int qmax, float* V, int8_t* codes,
                              float* preround, const bakron_opts* opts, void* ws,
                              size_t ws_bytes, void* stream) {
  try {
    const GridIn gr{scale, nullptr, n, 1};
    return quantize_impl(W, m, n, UA, UB, gr, qmin, qmax, V, codes, preround, opts, ws, ws_bytes,
                         stream);
  } catch (...) {
    return BAKRON_ERR_INVALID_ARG;   // host allocation failure
  }
}

bakron_status bakron_quantize_grid(const float* W, int64_t m, int64_t n, const float* UA,
                                   const float* UB, const float* scale, const float* zero,
                                   int64_t group, int qmin, int qmax, float* V, int8_t* codes,
                                   float* preround, const bakron_opts* opts, void* ws,
                                   size_t ws_bytes, void* stream) {
  try {
    const int64_t ng = grid_groups(n, group);
    if (ng < 1 || !sizes_ok(m, n)) return BAKRON_ERR_INVALID_ARG;
    const GridIn gr{scale, zero, ng == 1 ? n : group, ng};
    return quantize_impl(W, m, n, UA, UB, gr, qmin, qmax, V, codes, preround, opts, ws, ws_bytes,
                         stream);
  } catch (...) {
    return BAKRON_ERR_INVALID_ARG;   // host allocation failure
  }
}

bakron_status bakron_grid_params(const float* W, int64_t m, int64_t n, int bits, int asymmetric,
                                 int64_t group, float* scale, float* zero, int* qmin, int* qmax,
                                 void* stream) {
  const int64_t ng = grid_groups(n, group);
  if (!W || !scale || !zero || !sizes_ok(m, n) || ng < 1 || bits < 2 || bits > 8 ||
      (asymmetric != 0 && asymmetric != 1))
    return BAKRON_ERR_INVALID_ARG;
  if (qmin) *qmin = asymmetric ? 0 : -(1 << (bits - 1));
  if (qmax) *qmax = asymmetric ? (1 << bits) - 1 : (1 << (bits - 1)) - 1;
  cudaStream_t s = (cudaStream_t)stream;
  TRY_CUDA(launch_grid_params(W, m, n, ng == 1 ? n : group, ng, bits, asymmetric, scale, zero, s));
  TRY_CUDA(cudaStreamSynchronize(s));
  return BAKRON_OK;
}

bakron_status bakron_batch_workspace_size(int count, const bakron_problem* p,
                                          const bakron_opts* opts, size_t* bytes) {
  try {
    if (count < 1 || !p || !bytes) return BAKRON_ERR_INVALID_ARG;
    size_t total = 0;
    for (int i = 0; i < count; ++i) {
      size_t b = 0;
      bakron_status st = bakron_workspace_size(p[i].m, p[i].n, opts, &b);
      if (st != BAKRON_OK) return st;
      total += (b + 1023) / 1024 * 1024;
    }
    *bytes = total;
    return BAKRON_OK;
  } catch (...) {
    return BAKRON_ERR_INVALID_ARG;   // host allocation failure
  }
}

bakron_status bakron_quantize_batch(int count, bakron_problem* p, const bakron_opts* opts, void* ws,
                                    size_t ws_bytes, void* stream) {
  try {
    size_t need = 0;
    bakron_status vs = bakron_batch_workspace_size(count, p, opts, &need);
    if (vs != BAKRON_OK) return vs;
    if (!ws || ws_bytes < need) return BAKRON_ERR_INVALID_ARG;
    for (int i = 0; i < count; ++i) {
      p[i].status = BAKRON_OK;
      if (grid_groups(p[i].n, p[i].group) < 1) return BAKRON_ERR_INVALID_ARG;
    }
    cudaStream_t s = (cudaStream_t)stream;
    const int nslots = std::min(count, kSlots);
    std::vector<SolveStreams*> sets(nslots, nullptr);
    std::vector<std::unique_lock<std::mutex>> locks;
    std::vector<size_t> nev(nslots, 0);
    for (int k = 0; k < nslots; ++k) {
      TRY_CUDA(solve_streams(&sets[k], k));
      locks.emplace_back(sets[k]->mu);
    }
    std::vector<BatchCtx> ctx(count);
    std::vector<int> enq(count, 0);
    std::vector<size_t> offs(count + 1, 0);
    for (int i = 0; i < count; ++i) {
      size_t b = 0;
      bakron_workspace_size(p[i].m, p[i].n, opts, &b);
      offs[i + 1] = offs[i] + (b + 1023) / 1024 * 1024;
    }
    (void)prop_tc_supported();   // cached before the enqueuing threads start
    int dev = 0;
    TRY_CUDA(cudaGetDevice(&dev));
    // one host thread per stream set enqueues its problems, so a launch queue
    // that fills up for one problem does not hold back the others
    auto enqueue_slot = [&](int k) {
      if (cudaSetDevice(dev) != cudaSuccess) {
        for (int i = k; i < count; i += nslots) p[i].status = BAKRON_ERR_CUDA;
        return;
      }
      for (int i = k; i < count; i += nslots) {
        const int64_t ng = grid_groups(p[i].n, p[i].group);
        const GridIn gr{p[i].scale, p[i].zero, ng == 1 ? p[i].n : p[i].group, ng};
        ctx[i].ss = sets[k];
        ctx[i].nev = &nev[k];
        const bakron_status st = quantize_impl(
            p[i].W, p[i].m, p[i].n, p[i].UA, p[i].UB, gr, p[i].qmin, p[i].qmax, p[i].V, p[i].codes,
            nullptr, opts, (char*)ws + offs[i], offs[i + 1] - offs[i], stream, &ctx[i]);
        p[i].status = st;
        enq[i] = st == BAKRON_OK;
      }
    };
    {
      std::vector<std::thread> th;
      int k = 1;
      try {
        for (; k < nslots; ++k) th.emplace_back(enqueue_slot, k);
      } catch (...) {
        // no more threads to be had: the remaining slots are enqueued here
      }
      enqueue_slot(0);
      for (int j = k; j < nslots; ++j) enqueue_slot(j);
      for (auto& t : th) t.join();
    }
    bakron_status first = BAKRON_OK;
    for (int i = 0; i < count; ++i)
      if (!enq[i] && first == BAKRON_OK) first = (bakron_status)p[i].status;
    // join every enqueued problem onto the caller's stream, then read the
    // status blocks
    std::vector<DevStatus> hs(count);
    for (int i = 0; i < count; ++i)
      if (enq[i]) TRY_CUDA(cudaStreamWaitEvent(s, ctx[i].done, 0));
    for (int i = 0; i < count; ++i)
      if (enq[i])
        TRY_CUDA(cudaMemcpyAsync(&hs[i], ctx[i].st, sizeof(DevStatus), cudaMemcpyDeviceToHost, s));
    TRY_CUDA(cudaStreamSynchronize(s));
    for (int i = 0; i < count; ++i)
      if (enq[i]) {
        p[i].status = hs[i].status;
        if (first == BAKRON_OK && hs[i].status != BAKRON_OK) first = (bakron_status)hs[i].status;
      }
    return first;
  } catch (...) {
    return BAKRON_ERR_INVALID_ARG;   // host allocation failure
  }
}

bakron_status bakron_quantize_antidiag(const float* W, int64_t m, int64_t n, const float* UA,
                                       const float* UB, const float* scale, int qmin, int qmax,
                                       float* V, int8_t* codes, float* preround,
                                       const int8_t* guide_codes, float guide_tol,
                                       int64_t* overrides, const bakron_opts* opts_in, void* ws,
                                       size_t ws_bytes, void* stream) {
  try {
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
  } catch (...) {
    return BAKRON_ERR_INVALID_ARG;   // host allocation failure
  }
}

}  // extern "C"
