// Leaf sweep: one tile anti-diagonal D of 128 x 128 tiles, one CTA per tile.
//
// A tile is solved as an NB x NB grid of S x S blocks (S = 16), block
// anti-diagonal ("level") by level; inside a block the entries are rounded
// anti-diagonal by anti-diagonal (the anti-diagonal variant of the summary
// page "FastKron: Efficient Quantization with Kronecker-Factored Hessians",
// section 3), one lane per block row and 32 / S blocks per warp, so a step
// needs no CTA barrier.  Any order that respects the entry partial order (an
// entry after every entry to its top-left) gives the GPTQ result, and this
// one does.
//
// Notation (tile-local): Ua, Ub the diagonal 128-blocks of U_A, U_B; E the
// scaled errors.  For blocks (I, J):
//   P[I,J] = sum_{J'' < J} E[I,J''] Ua[J'',J]        (row accumulator, left part)
//   R[I,J] = P[I,J] + E[I,J] Ua[J,J]                 (complete row accumulator)
//   x0[I,J] = W~[I,J] - sum_{I' < I} Ub[I',I]^T R[I',J]
// where W~ already holds every update from earlier tile anti-diagonals.  x0
// is what the block sweep starts from; the sweep applies the rest, the
// updates from the block's own rows, in the row-accumulator form
//   x(a,b) = x0(a,b) - sum_{a' < a} Ub(a',a) R(a',b) - Ub(a,a) R_part(a,b),
//   R(a,b) = P(a,b) + sum_{b' <= b} e(a,b') Ua(b',b),  R_part: the sum over
//   b' < b (the Ub[I,I]^T P[I,J] part of the block's own rows rides in the
//   accumulators, which start from P).
//
// Schedule, level k (blocks with I + J = k), two CTA barriers per level:
//   B(k):   the sweep warps run the block sweeps of level k (R, codes and
//           V); four other warps meanwhile apply the pushes of level k-1
//           that later levels need but level k+1 does not:
//           P[I,J'] += E[I,J] Ua[J,J'] for J' >= J + 2 and
//           W~[I',J] -= Ub[I,I']^T R[I,J] for I' >= I + 2;
//   prep(k+1): the pushes from the two neighbours on level k into each block
//           (I,J) of level k+1, P[I,J] += E[I,J-1] Ua[J-1,J] and
//           W~[I,J] -= Ub[I-1,I]^T R[I-1,J], one warp per product.
// R of level k lives in one of two slot sets (level parity), because the
// deferred pushes read it while level k+1 writes its own.
//
// Block sweep, lane = (block, row a): Ub(a', a) for a' < a lives in
// registers; r(a-1, b), completed by the row above in the previous step,
// arrives by a warp shuffle; the older r(a', b) of the rows above are read
// from shared memory (rT[b][a'], 16-byte loads); the pending r(a, b'') of the lane's own
// row live in registers FR[j] = r(a, j - a) (the step loop is unrolled
// completely, so every register index is static and a register lives only
// between the steps that use it); the diagonal-major copy
// Dg[b][t] = Ua(b, b + t) makes the row update a run of 16-byte loads.  With
// the step d static, the work of a step is cut to what its active lanes
// (rows d - S + 1 .. d) can use: the row update to t <= 2 S - 2 - d, the
// look-ahead to the rows a' <= d - 1.
#include "internal.cuh"

namespace bakron {

namespace {
constexpr int T = kTile;          // 128
constexpr int NTHR = 384;
constexpr int NWARP = NTHR / 32;
constexpr int NDEF = 4;           // warps of the deferred pushes during a sweep
constexpr size_t kSmemLimit = 232448;

template <int S>
struct Cfg {
  static constexpr int NB = T / S;          // blocks per tile edge
  static constexpr int BPW = 32 / S;        // blocks per warp in a sweep
  static constexpr int NF = 2 * S - 1;      // row accumulators, by step index
  static constexpr int PX = T + 4;          // tile pitch
  static constexpr int PP = S + 1;          // P^T block pitch
  static constexpr int PR = S + 4;          // rT pitch (16-byte rows)
  static constexpr int PU = S;              // U block pitch
  static constexpr int PC = S + 4;          // code block pitch (bytes)
  static constexpr int PD = S + 4;          // diagonal-major pitch (16-byte rows)
  static constexpr int RT_SLOT = (S + 1) * PR;   // + one all-zero row
  static constexpr int NSTEP = 2 * S - 1;
  static constexpr int NUA = NB * (NB - 1) / 2;  // upper off-diagonal Ua blocks
  static constexpr int NUB = NB * (NB + 1) / 2;  // upper Ub blocks (with diagonal)
  static constexpr int OFF_X = 0;
  static constexpr int OFF_P = OFF_X + T * PX;               // NB (NB-1) blocks (J >= 1)
  static constexpr int OFF_RT = OFF_P + NB * (NB - 1) * S * PP;   // 2 sets of NB slots
  static constexpr int OFF_D = OFF_RT + 2 * NB * RT_SLOT;    // NB diagonal blocks of Ua
  static constexpr int OFF_UA = OFF_D + NB * S * PD;
  static constexpr int OFF_UB = OFF_UA + NUA * S * PU;
  static constexpr int OFF_LA = OFF_UB + NUB * S * PU;
  static constexpr int OFF_LB = OFF_LA + T;
  static constexpr int OFF_CS = OFF_LB + T;                  // NB x [S][PC] int8 codes
  static constexpr int SMEM_FLOATS = OFF_CS + NB * S * PC / 4;
  static constexpr size_t SMEM = sizeof(float) * (size_t)SMEM_FLOATS;
  // block products: one warp, OPT outputs per lane (RPT rows x CPT columns)
  static constexpr int OPT = S * S / 32;
  static constexpr int CPT = OPT < 4 ? OPT : 4;
  static constexpr int RPT = OPT / CPT;
  static constexpr int TC = S / CPT;         // lanes along the columns
  static_assert(SMEM <= kSmemLimit, "leaf shared memory");
  static_assert(NB * S * PU <= NB * (NB - 1) * S * PP, "staging area");
  static_assert(RPT * CPT == OPT && (32 / TC) * RPT == S, "product tiling");
  static_assert(NB / BPW + NDEF <= NWARP, "a level leaves warps for the deferred pushes");

  // upper off-diagonal Ua block (J < J2) and upper Ub block (I <= I2)
  __device__ static __forceinline__ int ua_idx(int J, int J2) {
    return J * (2 * NB - J - 1) / 2 + (J2 - J - 1);
  }
  __device__ static __forceinline__ int ub_idx(int I, int I2) {
    return I * (2 * NB - I + 1) / 2 + (I2 - I);
  }
  __device__ static __forceinline__ int p_idx(int I, int J) { return I * (NB - 1) + (J - 1); }
};

// p-th pair (r, c) of the row-major enumeration of {r < c} (strict) or
// {r <= c} of an nb x nb grid.
__device__ __forceinline__ void decode_pair(int p, int nb, int strict, int& r, int& c) {
  int row = 0, cnt = nb - strict;
  while (p >= cnt) {
    p -= cnt;
    ++row;
    cnt = nb - row - strict;
  }
  r = row;
  c = row + strict + p;
}

// C(r, c) += sign * sum_k A(r, k) B(k, c) for one S x S block, one warp.
// Lane: rows tr + TR i (i < RPT), columns tc + TC u (u < CPT), so the eight
// lanes of a quarter warp read distinct 16-byte bank groups of A.  A
// row-major [r][k] with pitch S (16-byte loads along k), B(k, c) at
// B[k + c * ldbc] (VB: 16-byte loads along k, ldbc a multiple of 4), C(r, c)
// at C[r * ldcr + c].  TRI: A(r, k) = 0 for k > r.
template <int S, bool TRI, bool VB>
__device__ __forceinline__ void block_product(const float* __restrict__ A, const float* __restrict__ B,
                                              int ldbc, float* __restrict__ C, int ldcr, float sign,
                                              int lane) {
  using K = Cfg<S>;
  constexpr int RPT = K::RPT, CPT = K::CPT, TC = K::TC, TR = 32 / TC;
  const int tr = lane / TC, tc = lane % TC;
  float acc[RPT][CPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
#pragma unroll
    for (int u = 0; u < CPT; ++u) acc[i][u] = 0.f;
  const int kend = TRI ? min(S, (tr + TR * (RPT - 1) + 4) & ~3) : S;
#pragma unroll 2
  for (int k0 = 0; k0 < kend; k0 += 4) {
    float4 a4[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) a4[i] = *reinterpret_cast<const float4*>(A + (tr + TR * i) * S + k0);
    float bv[4][CPT];
    if constexpr (VB) {
#pragma unroll
      for (int u = 0; u < CPT; ++u) {
        const float4 b4 = *reinterpret_cast<const float4*>(B + (tc + TC * u) * ldbc + k0);
        bv[0][u] = b4.x; bv[1][u] = b4.y; bv[2][u] = b4.z; bv[3][u] = b4.w;
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int u = 0; u < CPT; ++u) bv[kk][u] = B[k0 + kk + (tc + TC * u) * ldbc];
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i)
#pragma unroll
      for (int u = 0; u < CPT; ++u) {
        acc[i][u] = fmaf(a4[i].x, bv[0][u], acc[i][u]);
        acc[i][u] = fmaf(a4[i].y, bv[1][u], acc[i][u]);
        acc[i][u] = fmaf(a4[i].z, bv[2][u], acc[i][u]);
        acc[i][u] = fmaf(a4[i].w, bv[3][u], acc[i][u]);
      }
  }
#pragma unroll
  for (int i = 0; i < RPT; ++i)
#pragma unroll
    for (int u = 0; u < CPT; ++u) {
      float* c = C + (tr + TR * i) * ldcr + tc + TC * u;
      *c = fmaf(sign, acc[i][u], *c);
    }
}

__device__ __forceinline__ int level_imin(int k, int nb) { return k < nb ? 0 : k - nb + 1; }
__device__ __forceinline__ int level_imax(int k, int nb) { return k < nb ? k : nb - 1; }

// The pushes of the blocks of level kp that level kp+1 does not need:
// P[I,J'] += E[I,J] Ua[J,J'] for J' >= J + 2 and W~[I',J] -= Ub[I,I']^T R[I,J]
// for I' >= I + 2.  Products are dealt to nwork warps in turn; this warp is
// worker wk.  rTp: the R^T slots of level kp.
template <int S>
__device__ __forceinline__ void deferred_pushes(int kp, int wk, int nwork, float* X, float* Pt,
                                                const float* rTp, const float* UaO, const float* UbB,
                                                int lane) {
  using K = Cfg<S>;
  constexpr int NB = K::NB;
  const int Ipmin = level_imin(kp, NB), Ipmax = level_imax(kp, NB);
  int pidx = 0, mine = wk;
  for (int I = Ipmin; I <= Ipmax; ++I) {
    const int J = kp - I, slot = I - Ipmin;
    for (int J2 = J + 2; J2 < NB; ++J2, ++pidx)
      if (pidx == mine) {
        block_product<S, false, true>(UaO + K::ua_idx(J, J2) * S * K::PU, X + (S * I) * K::PX + S * J, K::PX,
                                Pt + K::p_idx(I, J2) * S * K::PP, K::PP, 1.f, lane);
        mine += nwork;
      }
    for (int I2 = I + 2; I2 < NB; ++I2, ++pidx)
      if (pidx == mine) {
        block_product<S, false, true>(UbB + K::ub_idx(I, I2) * S * K::PU, rTp + slot * K::RT_SLOT, K::PR,
                                X + (S * I2) * K::PX + S * J, K::PX, -1.f, lane);
        mine += nwork;
      }
  }
}
}  // namespace

// PRE: also write the pre-rounding values (a.preround), a debug output kept
// out of the default instantiation for its register cost.  CHK: check every
// code against the int8 range; without it the grid guarantees the range
// (qmin >= -128, qmax <= 127 and integer zero points in [qmin, qmax], so a
// code c + z with c clamped to [qmin - z, qmax - z] lies in [qmin, qmax]).
template <int S, bool PRE, bool CHK>
__global__ void __launch_bounds__(NTHR, 1) leaf_kernel(LeafArgs a) {
  using K = Cfg<S>;
  constexpr int NB = K::NB, BPW = K::BPW, NF = K::NF, PX = K::PX, PP = K::PP, PR = K::PR,
                PU = K::PU, PC = K::PC, PD = K::PD, RT_SLOT = K::RT_SLOT, NSTEP = K::NSTEP;
  extern __shared__ __align__(16) float smem[];
  float* X = smem + K::OFF_X;     // [T][PX]: W~, then E block by block
  float* Pt = smem + K::OFF_P;    // NB (NB-1) x [S][PP]: P^T[I,J] (b, a), J >= 1
  float* rT0 = smem + K::OFF_RT;  // 2 x NB x [S+1][PR]: completed r(a, b) at [b][a]; then R^T
  float* Dg = smem + K::OFF_D;    // NB x [S][PD]: Dg[J][b][t] = Ua(SJ+b, SJ+b+t), 0 past the block
  float* UaO = smem + K::OFF_UA;  // NUA x [S][PU]: Ua(SJ+b, SJ2+b2) at [b2][b]
  float* UbB = smem + K::OFF_UB;  // NUB x [S][PU]: Ub(SI+a, SI2+a2) at [a2][a]
  float* lA = smem + K::OFF_LA;   // [T]: 1 / Ua(b, b)
  float* lB = smem + K::OFF_LB;   // [T]: 1 / Ub(a, a)
  signed char* CS = reinterpret_cast<signed char*>(smem + K::OFF_CS);  // NB x [S][PC] codes

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int Itile = a.I0 + blockIdx.x;
  const int Jtile = a.D - Itile;
  const int64_t i0 = (int64_t)Itile * T, j0 = (int64_t)Jtile * T;

  // ---- load: the upper blocks of Ua and Ub (16-byte loads, all of a
  // thread's issued before its first store), then the W~ tile.  The global
  // arrays hold U^T: a block is copied as it is stored (rows of U^T =
  // columns of U).  The factors were written at the start of the solve, so
  // they are read before waiting for the previous kernel (which writes W~).
  // blocks u < NB: Ua diagonal (staged in the P area); NB <= u < NB + NUA:
  // Ua upper off-diagonal; then Ub upper with diagonal.  Block of U^T at
  // (row S * c, column S * r) for the pair (r, c).
  float* stage = Pt;
  {
    constexpr int QPB = S * S / 4;   // 16-byte items per block
    constexpr int kItems = (NB + K::NUA + K::NUB) * QPB;
    constexpr int kIt = (kItems + NTHR - 1) / NTHR;
    float4 hv[kIt], lv[kIt];
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int idx = min(tid + it * NTHR, kItems - 1);   // the tail repeats the last item
      const int blk = idx / QPB, w = idx % QPB;
      const int r = w / (S / 4), q = (w % (S / 4)) * 4;
      int br, bc;
      const bool isA = blk < NB + K::NUA;
      if (blk < NB) { br = blk; bc = blk; }
      else if (isA) decode_pair(blk - NB, NB, 1, br, bc);
      else decode_pair(blk - NB - K::NUA, NB, 0, br, bc);
      const int64_t base = isA ? j0 : i0;
      const int64_t ld = isA ? a.lda : a.ldb;
      const int64_t g = (base + S * bc + r) * ld + base + S * br + q;
      hv[it] = *reinterpret_cast<const float4*>((isA ? a.lat_hi : a.lbt_hi) + g);
      lv[it] = *reinterpret_cast<const float4*>((isA ? a.lat_lo : a.lbt_lo) + g);
    }
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int idx = tid + it * NTHR;
      if (idx >= kItems) break;
      const int blk = idx / QPB, w = idx % QPB;
      const int r = w / (S / 4), q = (w % (S / 4)) * 4;
      float* dst = blk < NB ? stage + blk * S * PU
                            : (blk < NB + K::NUA ? UaO + (blk - NB) * S * PU
                                                 : UbB + (blk - NB - K::NUA) * S * PU);
      float4 v;
      v.x = hv[it].x + lv[it].x;
      v.y = hv[it].y + lv[it].y;
      v.z = hv[it].z + lv[it].z;
      v.w = hv[it].w + lv[it].w;
      *reinterpret_cast<float4*>(dst + r * PU + q) = v;
    }
  }
  for (int idx = tid; idx < 2 * NB * RT_SLOT; idx += NTHR) rT0[idx] = 0.f;
  __syncthreads();
  for (int idx = tid; idx < NB * S * PD; idx += NTHR) {
    const int J = idx / (S * PD), rem = idx - J * S * PD;
    const int b = rem / PD, t = rem % PD;
    Dg[idx] = (t < S && b + t < S) ? stage[J * S * PU + (b + t) * PU + b] : 0.f;
  }
  if (tid < T) {
    const int J = tid / S, b = tid % S;
    lA[tid] = 1.f / stage[J * S * PU + b * PU + b];
  } else if (tid < 2 * T) {
    const int I = (tid - T) / S, r = (tid - T) % S;
    lB[tid - T] = 1.f / UbB[K::ub_idx(I, I) * S * PU + r * PU + r];
  }
  __syncthreads();
  for (int idx = tid; idx < NB * (NB - 1) * S * PP; idx += NTHR) Pt[idx] = 0.f;
  grid_dep_wait();
  // W~: block (0, 0) now, the rest by the warps that do not sweep level 0
  // (they are idle until its barrier, and nothing else reads the tile before)
  if (tid < S * S / 4) {
    const int r = tid / (S / 4), c = (tid % (S / 4)) * 4;
    *reinterpret_cast<float4*>(X + r * PX + c) =
        *reinterpret_cast<const float4*>(a.wt + (i0 + r) * a.ldw + j0 + c);
  }
  __syncthreads();
  bool nonfinite = false, out_of_range = false;
  // E of one 16-byte group q of block (I, J), split, to the error arrays.  A
  // non-finite pre-rounding value gives a non-finite error (and so does an
  // error that overflows), so the check runs here, off the sweep's steps.
  auto write_e = [&](int I, int J, int q) {
    const int r = S * I + q / (S / 4), cc = S * J + (q % (S / 4)) * 4;
    const float4 e = *reinterpret_cast<const float4*>(X + r * PX + cc);
    nonfinite |= !isfinite(e.x) || !isfinite(e.y) || !isfinite(e.z) || !isfinite(e.w);
    float4 h, l;
    h.x = tf32_round(e.x); h.y = tf32_round(e.y); h.z = tf32_round(e.z); h.w = tf32_round(e.w);
    l.x = e.x - h.x; l.y = e.y - h.y; l.z = e.z - h.z; l.w = e.w - h.w;
    if (a.round_lo) {
      l.x = tf32_round(l.x); l.y = tf32_round(l.y); l.z = tf32_round(l.z); l.w = tf32_round(l.w);
    }
    const int64_t g = (i0 + r) * a.ldw + j0 + cc;
    *reinterpret_cast<float4*>(a.e_hi + g) = h;
    *reinterpret_cast<float4*>(a.e_lo + g) = l;
  };

  const float fqmin = (float)a.qmin, fqmax = (float)a.qmax;

  // Grid scale and zero point of the row and block this thread sweeps at
  // level kk (lane = (sub, row) of block slot BPW warp + sub; a slot past
  // the level's blocks takes the level's first block, an in-bounds address).
  // The padded grid is written at the start of the solve, like the factors,
  // and is read one level ahead so the load latency stays off the sweeps.
  auto grid_at = [&](int kk, float& sc, float& zc) {
    const int Imn = level_imin(kk, NB), nb = level_imax(kk, NB) - Imn + 1;
    const int slot = warp * BPW + lane / S;
    const int I = Imn + (slot < nb ? slot : 0);
    const int64_t gi = i0 + S * I + lane % S;
    int64_t grp = (j0 + S * (kk - I)) / a.group;
    if (grp > a.ngroups - 1) grp = a.ngroups - 1;
    sc = a.scale[gi * a.ngroups + grp];
    zc = a.zero[gi * a.ngroups + grp];
  };
  float sc_next = 1.f, zc_next = 0.f;
  if (warp < 1) grid_at(0, sc_next, zc_next);

  for (int k = 0; k < 2 * NB - 1; ++k) {
    if (k == 2 * NB - 2) grid_dep_launch();   // the next kernel may start setting up
    const int Imin = level_imin(k, NB), Imax = level_imax(k, NB);
    const int nblk = Imax - Imin + 1;
    const int nsw = (nblk + BPW - 1) / BPW;    // sweep warps of this level
    float* rTk = rT0 + (k & 1) * NB * RT_SLOT;
    const float sc = sc_next, zc = zc_next;
    if (k + 1 < 2 * NB - 1) {
      const int nbn = level_imax(k + 1, NB) - level_imin(k + 1, NB) + 1;
      if (warp < (nbn + BPW - 1) / BPW) grid_at(k + 1, sc_next, zc_next);
    }

    if (warp < nsw) {
      // ---- B. block sweeps: lane = (sub, row), block Imin + BPW warp + sub
      const int sub = lane / S, row = lane % S;
      const int slot = warp * BPW + sub;
      const bool live = slot < nblk;
      const int I = Imin + (live ? slot : 0), J = k - I;
      const float* Ubd = UbB + K::ub_idx(I, I) * S * PU;
      float ub[S];
#pragma unroll
      for (int c = 0; c < S / 4; ++c) {
        const float4 v = *reinterpret_cast<const float4*>(Ubd + row * PU + 4 * c);
        ub[4 * c + 0] = (4 * c + 0 < row - 1) ? v.x : 0.f;
        ub[4 * c + 1] = (4 * c + 1 < row - 1) ? v.y : 0.f;
        ub[4 * c + 2] = (4 * c + 2 < row - 1) ? v.z : 0.f;
        ub[4 * c + 3] = (4 * c + 3 < row - 1) ? v.w : 0.f;
      }
      ub[S - 1] = 0.f;   // a' < a - 1 <= S - 2
      // Ub(a-1, a): the row directly above, whose accumulator completes one
      // step before this row needs it, is kept out of the look-ahead sum
      const float ub1 = row > 0 ? Ubd[row * PU + row - 1] : 0.f;
      const float ubaa = Ubd[row * PU + row];
      const float lBa = lB[S * I + row];
      const int64_t gi = i0 + S * I + row;
      const bool row_real = live && gi < a.m;
      float* rs = rTk + slot * RT_SLOT;
      const float* Dj = Dg + J * S * PD;
      const float* lAj = lA + S * J;
      float* Xrow = X + (S * I + row) * PX + S * J;
      const int64_t jb0 = j0 + S * J;
      // sc, zc: the block's columns lie in one group of the grid (groups are
      // whole multiples of 32 columns, or the whole row)
      // centred code c = clamp(rint(x / s), qmin - z, qmax - z); stored c + z
      const float clo = fqmin - zc, chi = fqmax - zc;
      const float rinv = 1.f / sc;
      signed char* csr = CS + slot * S * PC + row * PC;
      float FR[NF];
#pragma unroll
      for (int j = 0; j < NF; ++j) FR[j] = 0.f;
      float pp = 0.f;   // column sum over rows a' < a - 1 for this step's column
      float rlast = 0.f;  // R(a, .) completed by this lane in the previous step
      // P(a, b) of the block (zero in block column 0) enters the accumulator
      // FR[a + b] one step before the lane reaches column b (row 0: here)
      const bool hasP = live && J >= 1;
      const float* Pa = Pt + K::p_idx(I, J >= 1 ? J : 1) * S * PP + row;   // P(a, b) at Pa[b PP]
      if (hasP && row == 0) FR[0] = Pa[0];

#pragma unroll
      for (int d = 0; d < NSTEP; ++d) {
        // straight-line step: inactive lanes compute on safe addresses and
        // their results are masked (e = 0, stores predicated)
        const int b = d - row;
        const bool act = live && (unsigned)b < (unsigned)S;
        const int bb = act ? b : 0;
        const float xin = Xrow[bb];
        const float la = lAj[bb];
        // P(a, b + 1) for the next column's accumulator
        float pnext = 0.f;
        if (d + 1 < NSTEP) {
          const bool pin = hasP && (unsigned)(b + 1) < (unsigned)S;
          pnext = Pa[(pin ? b + 1 : 0) * PP];
          pnext = pin ? pnext : 0.f;
        }
        // r(a-1, b): the row above completed column b in the previous step
        // (lane 0 of a block multiplies it by ub1 = 0)
        const float rprev = __shfl_up_sync(0xffffffffu, rlast, 1);
        // look-ahead: the column sum of the NEXT step (column b + 1) over
        // rows a' < a - 1, all completed by the previous step; it is off this
        // step's dependency chain.  A lane active next step has a <= d + 1,
        // so only the rows a' <= d - 1 can count (ub is zero past a - 2).
        // A lane inactive next step (bn outside 0 .. S-1) reads other shared
        // data here (at most 13 rows before the slot, 14 past it: still
        // inside the P, rT and Dg areas) and never uses the sum.
        const int bn = b + 1;
        const float* rc = rs + bn * PR;
        float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
        for (int c = 0; c < S / 4; ++c) {
          if (d + 1 < NSTEP && 4 * c <= d - 1) {
            const float4 v = *reinterpret_cast<const float4*>(rc + 4 * c);
            p0 = fmaf(ub[4 * c + 0], v.x, p0);
            p1 = fmaf(ub[4 * c + 1], v.y, p1);
            p2 = fmaf(ub[4 * c + 2], v.z, p2);
            if (c < S / 4 - 1) p3 = fmaf(ub[4 * c + 3], v.w, p3);
          }
        }
        // row b of the diagonal-major Ua (its S entries; the row's pad is
        // zero), read before this step's stores; entries t > 2 S - 2 - d
        // reach only columns past the block
        const float4* dr = reinterpret_cast<const float4*>(Dj + bb * PD);
        float4 dv[S / 4];
#pragma unroll
        for (int c = 0; c < S / 4; ++c)
          if (4 * c <= 2 * S - 2 - d) dv[c] = dr[c];
        const float x = xin - fmaf(ub1, rprev, pp) - ubaa * FR[d];
        pp = (p0 + p1) + (p2 + p3);
        // rounding decision on x * fl(1/s): within 2^-23 relative of x / s,
        // so it can differ from the correctly rounded quotient only within
        // 2e-5 grid units of a rounding boundary
        float c = rintf(x * rinv);
        c = fminf(fmaxf(c, clo), chi);
        const float e = act ? (x - sc * c) * lBa * la : 0.f;
        const float code = c + zc;
        if (CHK) out_of_range |= act && ((code < -128.f) || (code > 127.f));
        if (d + 1 < NSTEP) FR[d + 1] += pnext;
        FR[d] = fmaf(e, dv[0].x, FR[d]);
        rlast = FR[d];
        if (act) {
          Xrow[b] = e;
          // without CHK the grid keeps every code inside the int8 range
          csr[b] = (signed char)(int)(CHK ? fminf(fmaxf(code, -128.f), 127.f) : code);
          rs[b * PR + row] = FR[d];
        }
        if (PRE && act && row_real && jb0 + b < a.n) a.preround[gi * a.n + jb0 + b] = x;
        // pending accumulators of this row: FR[d + t] += e Ua(b, b + t)
#pragma unroll
        for (int c = 0; c < S / 4; ++c) {
          if (4 * c <= 2 * S - 2 - d) {
            const float4 v = dv[c];
            if (4 * c + 0 >= 1 && 4 * c + 0 <= 2 * S - 2 - d) FR[d + 4 * c + 0] = fmaf(e, v.x, FR[d + 4 * c + 0]);
            if (4 * c + 1 <= 2 * S - 2 - d) FR[d + 4 * c + 1] = fmaf(e, v.y, FR[d + 4 * c + 1]);
            if (4 * c + 2 <= 2 * S - 2 - d) FR[d + 4 * c + 2] = fmaf(e, v.z, FR[d + 4 * c + 2]);
            if (4 * c + 3 <= 2 * S - 2 - d) FR[d + 4 * c + 3] = fmaf(e, v.w, FR[d + 4 * c + 3]);
          }
        }
        __syncwarp();
      }
      // codes and V of this block row: one contiguous run per lane
      if (row_real) {
        const int64_t base = gi * a.n + jb0;
        const int nb = a.n - jb0 < S ? (int)(a.n - jb0) : S;
        if (nb == S && (a.n & 15) == 0) {
          if constexpr (S % 16 == 0) {
#pragma unroll
            for (int q = 0; q < S / 16; ++q) {
              uint4 w;
              w.x = *reinterpret_cast<const unsigned*>(csr + 16 * q + 0);
              w.y = *reinterpret_cast<const unsigned*>(csr + 16 * q + 4);
              w.z = *reinterpret_cast<const unsigned*>(csr + 16 * q + 8);
              w.w = *reinterpret_cast<const unsigned*>(csr + 16 * q + 12);
              reinterpret_cast<uint4*>(a.codes + base)[q] = w;
            }
          } else {
#pragma unroll
            for (int q = 0; q < S / 8; ++q) {
              uint2 w;
              w.x = *reinterpret_cast<const unsigned*>(csr + 8 * q + 0);
              w.y = *reinterpret_cast<const unsigned*>(csr + 8 * q + 4);
              reinterpret_cast<uint2*>(a.codes + base)[q] = w;
            }
          }
#pragma unroll
          for (int q = 0; q < S / 4; ++q) {
            float4 v;
            v.x = sc * ((float)csr[4 * q + 0] - zc);
            v.y = sc * ((float)csr[4 * q + 1] - zc);
            v.z = sc * ((float)csr[4 * q + 2] - zc);
            v.w = sc * ((float)csr[4 * q + 3] - zc);
            reinterpret_cast<float4*>(a.V + base)[q] = v;
          }
        } else {
          for (int t = 0; t < nb; ++t) {
            a.codes[base + t] = csr[t];
            a.V[base + t] = sc * ((float)csr[t] - zc);
          }
        }
      }
    } else if (k == 0) {
      // the rest of the W~ tile (everything but block (0, 0))
      for (int idx = tid - 32 * nsw; idx < T * T / 4; idx += NTHR - 32 * nsw) {
        const int r = idx >> 5, c = (idx & 31) * 4;
        if (r < S && c < S) continue;
        *reinterpret_cast<float4*>(X + r * PX + c) =
            *reinterpret_cast<const float4*>(a.wt + (i0 + r) * a.ldw + j0 + c);
      }
    } else if (warp >= nsw + NDEF) {
      // the errors of level k-1's blocks are final (later steps only read
      // them): out to the error arrays while this level sweeps
      const int kp = k - 1, Ipmin = level_imin(kp, NB), npb = level_imax(kp, NB) - Ipmin + 1;
      const int nthr = NTHR - 32 * (nsw + NDEF);
      for (int t = tid - 32 * (nsw + NDEF); t < npb * (S * S / 4); t += nthr) {
        const int I = Ipmin + t / (S * S / 4);
        write_e(I, kp - I, t % (S * S / 4));
      }
    } else if (k >= 1 && warp < nsw + NDEF) {
      // ---- deferred pushes of level k-1 into levels >= k+1, on NDEF of the
      // other warps (more would take issue and shared-memory bandwidth from
      // the latency-bound sweeps)
      deferred_pushes<S>(k - 1, warp - nsw, NDEF, X, Pt, rT0 + ((k - 1) & 1) * NB * RT_SLOT,
                         UaO, UbB, lane);
    }
    __syncthreads();

    // ---- prep(k+1): the neighbours' pushes into the blocks of level k+1,
    // one warp per product (the two products of a block write different
    // arrays)
    if (k + 1 < 2 * NB - 1) {
      const int kn = k + 1;
      const int Inmin = level_imin(kn, NB), Inmax = level_imax(kn, NB);
      const int nn = Inmax - Inmin + 1;
      for (int t = warp; t < 2 * nn; t += NWARP) {
        const int I = Inmin + (t >> 1), J = kn - I;
        if ((t & 1) == 0) {
          if (J >= 1)   // P[I,J] += E[I,J-1] Ua[J-1,J]  (the left neighbour, level k)
            block_product<S, false, true>(UaO + K::ua_idx(J - 1, J) * S * PU, X + (S * I) * PX + S * (J - 1),
                                    PX, Pt + K::p_idx(I, J) * S * PP, PP, 1.f, lane);
        } else if (I >= 1) {   // W~[I,J] -= Ub[I-1,I]^T R[I-1,J]  (the upper neighbour, level k)
          block_product<S, false, true>(UbB + K::ub_idx(I - 1, I) * S * PU,
                                  rTk + (I - 1 - Imin) * RT_SLOT, PR, X + (S * I) * PX + S * J, PX, -1.f, lane);
        }
      }
      __syncthreads();
    }
  }

  if (nonfinite) set_status(a.st, BAKRON_ERR_NONFINITE);
  if (out_of_range) set_status(a.st, BAKRON_ERR_CODE_RANGE);

  // write-out: the errors of the last level's block (the earlier levels'
  // went out while the next level swept)
  if (tid < S * S / 4) write_e(NB - 1, NB - 1, tid);
}

namespace {
constexpr int kLeafBlock = 16;
}  // namespace

cudaError_t launch_leaf(const LeafArgs& a, int n_tiles, cudaStream_t s) {
  constexpr int S = kLeafBlock;
  static std::atomic<unsigned long long> done[3];
  constexpr size_t smem = Cfg<S>::SMEM;
  cudaError_t e = ensure_smem_limit((const void*)leaf_kernel<S, false, false>, smem, done[0]);
  if (e == cudaSuccess) e = ensure_smem_limit((const void*)leaf_kernel<S, false, true>, smem, done[1]);
  if (e == cudaSuccess) e = ensure_smem_limit((const void*)leaf_kernel<S, true, true>, smem, done[2]);
  if (e != cudaSuccess) return e;
  count_launch();
  if (a.preround)
    return launch_kernel(leaf_kernel<S, true, true>, dim3(n_tiles), dim3(NTHR), smem, s, a.pdl != 0, a);
  if (a.qmin < -128 || a.qmax > 127)
    return launch_kernel(leaf_kernel<S, false, true>, dim3(n_tiles), dim3(NTHR), smem, s, a.pdl != 0, a);
  return launch_kernel(leaf_kernel<S, false, false>, dim3(n_tiles), dim3(NTHR), smem, s, a.pdl != 0, a);
}

}  // namespace bakron
