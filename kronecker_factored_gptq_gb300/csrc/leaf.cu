// Leaf sweep: one tile anti-diagonal D of 128 x 128 tiles, one CTA per tile.
//
// A tile is solved as a 4 x 4 grid of 32 x 32 blocks, block anti-diagonal by
// block anti-diagonal; inside a block the entries are rounded anti-diagonal
// by anti-diagonal (the anti-diagonal variant of the summary page "FastKron:
// Efficient Quantization with Kronecker-Factored Hessians", section 3), one
// warp per block and one lane per block row, so a step needs no CTA barrier.
// Any order that respects the entry partial order (an entry after every
// entry to its top-left) gives the GPTQ result, and this one does.
//
// Notation (tile-local): Ua, Ub the diagonal 128-blocks of U_A, U_B; E the
// scaled errors.  For blocks (I, J):
//   P[I,J] = sum_{J'' < J} E[I,J''] Ua[J'',J]        (row accumulator, left part)
//   R[I,J] = P[I,J] + E[I,J] Ua[J,J]                 (complete row accumulator)
//   x0[I,J] = W~[I,J] - sum_{I' < I} Ub[I',I]^T R[I',J] - Ub[I,I]^T P[I,J]
// where W~ already holds every update from earlier tile anti-diagonals and
// Ub[I,I]^T P includes the diagonal.  x0 is what the block sweep starts from;
// the sweep then applies the updates between entries of the block itself
// with the same row-accumulator form at entry level:
//   x(a,b) = x0(a,b) - sum_{a' < a} Ub(a',a) r(a',b) - Ub(a,a) r_part(a,b),
//   r(a,b) = sum_{b' <= b} e(a,b') Ua(b',b),  r_part: the sum over b' < b.
// Level k of the block sweep (blocks with I + J = k):
//   A. x0 for its blocks: W~ -= Ub[I,I]^T P[I,J]  (triangular block product);
//   B. block sweeps, 63 steps each, one warp per block;
//   C. R = P + r; pushes to later blocks: P[I,J'] += E[I,J] Ua[J,J'] (J' > J)
//      and W~[I',J] -= Ub[I,I']^T R[I,J] (I' > I).
// Phases are separated by CTA barriers (21 per tile).
//
// Block sweep, lane a = block row: Ub(a', a) for a' < a lives in registers;
// the completed r(a', b) of the rows above are read from shared memory
// (rT[b][a'], 16-byte loads); the pending r(a, b'') of the lane's own row
// live in a register window FR[j] = r(a, b0 + j), b0 = 4 kb - a, shifted by
// four registers every four steps (the step loop is unrolled by four, so
// every register index is static); the diagonal-major copy
// Dg[b][t] = Ua(b, b + t) makes the row update a run of 16-byte loads.
#include "internal.cuh"

namespace bakron {

namespace {
constexpr int T = kTile;          // 128
constexpr int S = 32;             // block edge
constexpr int NB = T / S;         // 4 blocks per tile edge
constexpr int NTHR = 384;
constexpr int NPAIR = NTHR / 64;   // warp pairs for the block products
constexpr int NF = S + 3;         // row-accumulator window: columns b0 .. b0 + 34, b0 >= -3 once active
constexpr int PX = T + 4;         // tile pitch
constexpr int PP = S + 1;         // P^T block pitch
constexpr int PR = S + 4;         // rT pitch (16-byte rows)
constexpr int PU = S;             // U block pitch (rows read whole, columns written lane by lane)
constexpr int PC = S + 4;         // code block pitch (bytes)
constexpr int PD = S + 4;         // diagonal-major pitch (16-byte rows)
constexpr int RT_SLOT = (S + 1) * PR;   // + one all-zero row
constexpr int NSTEP = 2 * S - 1;

constexpr int OFF_X = 0;
constexpr int OFF_P = OFF_X + T * PX;                  // 12 blocks (J >= 1)
constexpr int OFF_RT = OFF_P + NB * (NB - 1) * S * PP; // 4 slots
constexpr int OFF_D = OFF_RT + NB * RT_SLOT;           // 4 diagonal blocks of Ua
constexpr int OFF_UA = OFF_D + NB * S * PD;            // 6 upper off-diagonal blocks of Ua
constexpr int OFF_UB = OFF_UA + 6 * S * PU;            // 10 upper blocks of Ub (with diagonal)
constexpr int OFF_LA = OFF_UB + 10 * S * PU;
constexpr int OFF_CS = OFF_LA + T;                     // 4 x [S][PC] int8 codes
constexpr int SMEM_FLOATS = OFF_CS + NB * S * PC / 4;
constexpr size_t kLeafSmem = sizeof(float) * (size_t)SMEM_FLOATS;
static_assert(kLeafSmem <= 232448, "leaf shared memory");
static_assert(NB * S * PU <= NB * (NB - 1) * S * PP, "staging area");

// upper off-diagonal Ua block (J < J2) and upper Ub block (I <= I2)
__device__ __forceinline__ int ua_idx(int J, int J2) { return J * (7 - J) / 2 + (J2 - J - 1); }
__device__ __forceinline__ int ub_idx(int I, int I2) { return I * (9 - I) / 2 + (I2 - I); }
__device__ __forceinline__ int p_idx(int I, int J) { return I * (NB - 1) + (J - 1); }

// tile offsets (row of U^T, column of U^T) of the 20 loaded blocks:
// Ua diagonal (J, J) for J = 0..3; Ua (J, J2), J < J2, in ua_idx order;
// Ub (I, I2), I <= I2, in ub_idx order.  Row offset 32 * (J2 or I2),
// column offset 32 * (J or I).
__constant__ int kRow[20] = {0,  32, 64, 96,  32, 64, 96, 64, 96, 96,
                             0,  32, 64, 96,  32, 64, 96, 64, 96, 96};
__constant__ int kCol[20] = {0,  32, 64, 96,  0,  0,  0,  32, 32, 64,
                             0,  0,  0,  0,   32, 32, 32, 64, 64, 96};

// C(r, c) += sign * sum_k A(r, k) B(k, c) for one 32 x 32 block, 64 threads
// (lt in [0, 64)), each a 4 x 4 tile: rows 4 tr .. 4 tr + 3, columns
// tc + 8 u.  A row-major [r][k] with pitch PU (16-byte loads along k),
// B(k, c) at B[k + c * ldbc], C(r, c) at C[r * ldcr + c].  TRI: A(r, k) = 0
// for k > r, so the k loop stops at the warp's last row.
template <bool TRI>
__device__ __forceinline__ void block_product(const float* __restrict__ A, const float* __restrict__ B,
                                              int ldbc, float* __restrict__ C, int ldcr, float sign,
                                              int lt) {
  const int tr = lt >> 3, tc = lt & 7, r0 = 4 * tr;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[i][u] = 0.f;
  const int kend = TRI ? ((lt >> 5) + 1) * 16 : S;   // warp-uniform bound
#pragma unroll 2
  for (int k0 = 0; k0 < kend; k0 += 4) {
    float4 a4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a4[i] = *reinterpret_cast<const float4*>(A + (r0 + i) * PU + k0);
    float bv[4][4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int u = 0; u < 4; ++u) bv[kk][u] = B[k0 + kk + (tc + 8 * u) * ldbc];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc[i][u] = fmaf(a4[i].x, bv[0][u], acc[i][u]);
        acc[i][u] = fmaf(a4[i].y, bv[1][u], acc[i][u]);
        acc[i][u] = fmaf(a4[i].z, bv[2][u], acc[i][u]);
        acc[i][u] = fmaf(a4[i].w, bv[3][u], acc[i][u]);
      }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float* c = C + (r0 + i) * ldcr + tc + 8 * u;
      *c = fmaf(sign, acc[i][u], *c);
    }
}
}  // namespace

// PRE: also write the pre-rounding values (a.preround), a debug output kept
// out of the default instantiation for its register cost
template <bool PRE>
__global__ void __launch_bounds__(NTHR, 1) leaf_kernel(LeafArgs a) {
  extern __shared__ __align__(16) float smem[];
  float* X = smem + OFF_X;     // [T][PX]: W~, then E block by block
  float* Pt = smem + OFF_P;    // 12 x [S][PP]: P^T[I,J] (b, a), J >= 1
  float* rT = smem + OFF_RT;   // 4 x [S+1][PR]: completed r(a, b) at [b][a]; then R^T
  float* Dg = smem + OFF_D;    // 4 x [S][PD]: Dg[J][b][t] = Ua(32J+b, 32J+b+t), 0 past the block
  float* UaO = smem + OFF_UA;  // 6 x [S][PU]: Ua(32J+b, 32J2+b2) at [b2][b]
  float* UbB = smem + OFF_UB;  // 10 x [S][PU]: Ub(32I+a, 32I2+a2) at [a2][a]
  float* lA = smem + OFF_LA;   // [T]: 1 / Ua(b, b)
  signed char* CS = reinterpret_cast<signed char*>(smem + OFF_CS);  // 4 x [S][PC] codes

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int Itile = a.I0 + blockIdx.x;
  const int Jtile = a.D - Itile;
  const int64_t i0 = (int64_t)Itile * T, j0 = (int64_t)Jtile * T;

  // ---- load: W~ tile, the upper blocks of Ua and Ub (16-byte loads, several
  // in flight per thread).  The global arrays hold U^T: lane = row of the
  // shared block, so the transposing shared stores are conflict-free.
#pragma unroll 4
  for (int idx = tid; idx < T * T / 4; idx += NTHR) {
    const int r = idx >> 5, c = (idx & 31) * 4;
    *reinterpret_cast<float4*>(X + r * PX + c) =
        *reinterpret_cast<const float4*>(a.wt + (i0 + r) * a.ldw + j0 + c);
  }
  // 20 blocks of U^T copied as they are (rows of U^T = columns of U):
  // Ua diagonal blocks 0-3 (staged in the P area), Ua upper off-diagonal
  // blocks 4-9, Ub upper blocks 10-19.  Block u is the 32 x 32 block of U^T
  // at tile offsets (row kRow[u], column kCol[u]); a warp reads four whole
  // 128-byte rows per instruction, and all loads of a thread are issued
  // before the first store.
  float* stage = Pt;
  {
    constexpr int kItems = 20 * S * S / 4;
    constexpr int kIt = (kItems + NTHR - 1) / NTHR;   // items per thread
    float4 hv[kIt], lv[kIt];
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int idx = min(tid + it * NTHR, kItems - 1);   // the tail repeats the last item
      const int blk = idx >> 8, w = idx & 255;
      const int r = w >> 3, q = (w & 7) * 4;
      const bool isA = blk < 10;
      const int64_t base = isA ? j0 : i0;
      const int64_t ld = isA ? a.lda : a.ldb;
      const int64_t g = (base + kRow[blk] + r) * ld + base + kCol[blk] + q;
      hv[it] = *reinterpret_cast<const float4*>((isA ? a.lat_hi : a.lbt_hi) + g);
      lv[it] = *reinterpret_cast<const float4*>((isA ? a.lat_lo : a.lbt_lo) + g);
    }
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int idx = tid + it * NTHR;
      if (idx >= kItems) break;
      const int blk = idx >> 8, w = idx & 255;
      const int r = w >> 3, q = (w & 7) * 4;
      float* dst = blk < 4 ? stage + blk * S * PU
                           : (blk < 10 ? UaO + (blk - 4) * S * PU : UbB + (blk - 10) * S * PU);
      float4 v;
      v.x = hv[it].x + lv[it].x;
      v.y = hv[it].y + lv[it].y;
      v.z = hv[it].z + lv[it].z;
      v.w = hv[it].w + lv[it].w;
      *reinterpret_cast<float4*>(dst + r * PU + q) = v;
    }
  }
  for (int idx = tid; idx < NB * RT_SLOT; idx += NTHR) rT[idx] = 0.f;
  __syncthreads();
  for (int idx = tid; idx < NB * S * PD; idx += NTHR) {
    const int J = idx / (S * PD), rem = idx - J * S * PD;
    const int t = rem >> 5, b = rem & (S - 1);
    Dg[J * S * PD + b * PD + t] = (b + t < S) ? stage[J * S * PU + (b + t) * PU + b] : 0.f;
  }
  if (tid < T) {
    const int J = tid >> 5, b = tid & (S - 1);
    lA[tid] = 1.f / stage[J * S * PU + b * PU + b];
  }
  __syncthreads();
  for (int idx = tid; idx < NB * (NB - 1) * S * PP; idx += NTHR) Pt[idx] = 0.f;
  __syncthreads();

  const float fqmin = (float)a.qmin, fqmax = (float)a.qmax;
  bool nonfinite = false, out_of_range = false;
  const int pair = warp >> 1, lt = (warp & 1) * 32 + lane;

  for (int k = 0; k < 2 * NB - 1; ++k) {
    const int Imin = k < NB ? 0 : k - NB + 1;
    const int Imax = k < NB ? k : NB - 1;
    const int nblk = Imax - Imin + 1;

    // ---- A. x0 = W~ - Ub[I,I]^T P[I,J] for the blocks of this level with J >= 1
    if (pair < nblk) {
      const int I = Imin + pair, J = k - I;
      if (J >= 1)
        block_product<true>(UbB + ub_idx(I, I) * S * PU, Pt + p_idx(I, J) * S * PP, PP,
                            X + (S * I) * PX + S * J, PX, -1.f, lt);
    }
    __syncthreads();

    // ---- B. block sweeps
    if (warp < nblk) {
      const int I = Imin + warp, J = k - I;
      const int row = lane;
      const float* Ubd = UbB + ub_idx(I, I) * S * PU;
      float ub[S];
#pragma unroll
      for (int c = 0; c < S / 4; ++c) {
        const float4 v = *reinterpret_cast<const float4*>(Ubd + row * PU + 4 * c);
        ub[4 * c + 0] = (4 * c + 0 < row - 1) ? v.x : 0.f;
        ub[4 * c + 1] = (4 * c + 1 < row - 1) ? v.y : 0.f;
        ub[4 * c + 2] = (4 * c + 2 < row - 1) ? v.z : 0.f;
        ub[4 * c + 3] = (4 * c + 3 < row - 1) ? v.w : 0.f;
      }
      ub[S - 1] = 0.f;   // a' < a - 1 <= 30
      // Ub(a-1, a): the row directly above, whose accumulator completes one
      // step before this row needs it, is kept out of the look-ahead sum
      const float ub1 = row > 0 ? Ubd[row * PU + row - 1] : 0.f;
      const int rowm1 = row > 0 ? row - 1 : 0;
      const float ubaa = Ubd[row * PU + row];
      const float lB = 1.f / ubaa;
      const int64_t gi = i0 + S * I + row;
      const float sc = a.scale[gi];
      const bool row_real = gi < a.m;
      float* rs = rT + warp * RT_SLOT;
      const float* Dj = Dg + J * S * PD;
      const float* lAj = lA + S * J;
      float* Xrow = X + (S * I + row) * PX + S * J;
      const int64_t jb0 = j0 + S * J;
      const float rinv = 1.f / sc;
      signed char* csr = CS + warp * S * PC + row * PC;
      float FR[NF];
#pragma unroll
      for (int j = 0; j < NF; ++j) FR[j] = 0.f;
      float pp = 0.f;   // column sum over rows a' < a - 1 for this step's column

      for (int kb = 0; kb * 4 < NSTEP; ++kb) {
#pragma unroll
        for (int sg = 0; sg < 4; ++sg) {
          const int d = kb * 4 + sg;
          if (d >= NSTEP) break;
          // straight-line step: inactive lanes compute on safe addresses and
          // their results are masked (e = 0, stores predicated)
          const int b = d - row;
          const bool act = (unsigned)b < (unsigned)S;
          const int bb = act ? b : 0;
          const float xin = Xrow[bb];
          const float la = lAj[bb];
          // completed r(a-1, b) of the row above (previous step)
          const float rprev = rs[(act ? b : S) * PR + rowm1];
          // look-ahead: the column sum of the NEXT step (column b + 1) over
          // rows a' < a - 1, all completed by the previous step; it is off
          // this step's dependency chain
          const int bn = b + 1;
          const float* rc = rs + ((unsigned)bn < (unsigned)S ? bn : S) * PR;
          float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
          for (int c = 0; c < S / 4; ++c) {
            const float4 v = *reinterpret_cast<const float4*>(rc + 4 * c);
            p0 = fmaf(ub[4 * c + 0], v.x, p0);
            p1 = fmaf(ub[4 * c + 1], v.y, p1);
            p2 = fmaf(ub[4 * c + 2], v.z, p2);
            if (c < S / 4 - 1) p3 = fmaf(ub[4 * c + 3], v.w, p3);
          }
          // row b of the diagonal-major Ua, read before this step's stores
          const float4* dr = reinterpret_cast<const float4*>(Dj + bb * PD);
          float4 dv[PD / 4];
#pragma unroll
          for (int c = 0; c < PD / 4; ++c) dv[c] = dr[c];
          const float x = xin - fmaf(ub1, rprev, pp) - ubaa * FR[sg];
          pp = (p0 + p1) + (p2 + p3);
          // rounding decision on x * fl(1/s): within 2^-23 relative of x / s,
          // so it can differ from the correctly rounded quotient only within
          // 2e-5 grid units of a rounding boundary
          float c = rintf(x * rinv);
          c = fminf(fmaxf(c, fqmin), fqmax);
          const float e = act ? (x - sc * c) * lB * la : 0.f;
          nonfinite |= act && !isfinite(x);
          out_of_range |= act && ((c < -128.f) || (c > 127.f));
          FR[sg] = fmaf(e, dv[0].x, FR[sg]);
          if (act) {
            Xrow[b] = e;
            csr[b] = (signed char)(int)fminf(fmaxf(c, -128.f), 127.f);
            rs[b * PR + row] = FR[sg];
          }
          if (PRE && act && row_real && jb0 + b < a.n) a.preround[gi * a.n + jb0 + b] = x;
          // pending accumulators of this row: FR[sg + t] += e Ua(b, b + t),
          // first with the values loaded before the stores, then the rest
#pragma unroll
          for (int c = 0; c < PD / 4; ++c) {
            const float4 v = dv[c];
            if (4 * c + 0 >= 1 && sg + 4 * c + 0 < NF) FR[sg + 4 * c + 0] = fmaf(e, v.x, FR[sg + 4 * c + 0]);
            if (4 * c + 1 >= 1 && sg + 4 * c + 1 < NF) FR[sg + 4 * c + 1] = fmaf(e, v.y, FR[sg + 4 * c + 1]);
            if (4 * c + 2 >= 1 && sg + 4 * c + 2 < NF) FR[sg + 4 * c + 2] = fmaf(e, v.z, FR[sg + 4 * c + 2]);
            if (4 * c + 3 >= 1 && sg + 4 * c + 3 < NF) FR[sg + 4 * c + 3] = fmaf(e, v.w, FR[sg + 4 * c + 3]);
          }
          __syncwarp();
        }
#pragma unroll
        for (int j = 0; j < NF - 4; ++j) FR[j] = FR[j + 4];
#pragma unroll
        for (int j = NF - 4; j < NF; ++j) FR[j] = 0.f;
      }
      // codes and V of this block row: one contiguous run per lane
      if (row_real) {
        const int64_t base = gi * a.n + jb0;
        const int nb = a.n - jb0 < S ? (int)(a.n - jb0) : S;
        if (nb == S && (a.n & 15) == 0) {
          uint4 w[2];
          unsigned* wu = reinterpret_cast<unsigned*>(w);
#pragma unroll
          for (int q = 0; q < 8; ++q) wu[q] = *reinterpret_cast<const unsigned*>(csr + 4 * q);
          reinterpret_cast<uint4*>(a.codes + base)[0] = w[0];
          reinterpret_cast<uint4*>(a.codes + base)[1] = w[1];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 v;
            v.x = sc * (float)csr[4 * q + 0];
            v.y = sc * (float)csr[4 * q + 1];
            v.z = sc * (float)csr[4 * q + 2];
            v.w = sc * (float)csr[4 * q + 3];
            reinterpret_cast<float4*>(a.V + base)[q] = v;
          }
        } else {
          for (int t = 0; t < nb; ++t) {
            a.codes[base + t] = csr[t];
            a.V[base + t] = sc * (float)csr[t];
          }
        }
      }
      // R^T = P^T + r^T in place (lane = block row a owns column a)
      if (J >= 1) {
        const float* pb = Pt + p_idx(I, J) * S * PP;
#pragma unroll 8
        for (int b = 0; b < S; ++b) rs[b * PR + row] += pb[b * PP + row];
      }
    }
    __syncthreads();

    // ---- C. pushes from the blocks of this level, one block product per warp pair
    {
      int pidx = 0;
      for (int I = Imin; I <= Imax; ++I) {
        const int J = k - I, slot = I - Imin;
        for (int J2 = J + 1; J2 < NB; ++J2, ++pidx)
          if (pidx % NPAIR == pair)
            block_product<false>(UaO + ua_idx(J, J2) * S * PU, X + (S * I) * PX + S * J, PX,
                                 Pt + p_idx(I, J2) * S * PP, PP, 1.f, lt);
        for (int I2 = I + 1; I2 < NB; ++I2, ++pidx)
          if (pidx % NPAIR == pair)
            block_product<false>(UbB + ub_idx(I, I2) * S * PU, rT + slot * RT_SLOT, PR,
                                 X + (S * I2) * PX + S * J, PX, -1.f, lt);
      }
    }
    __syncthreads();
  }

  if (nonfinite) set_status(a.st, BAKRON_ERR_NONFINITE);
  if (out_of_range) set_status(a.st, BAKRON_ERR_CODE_RANGE);

  // write-out: scaled errors (split) for the propagation
  for (int idx = tid; idx < T * T; idx += NTHR) {
    const int r = idx >> 7, cc = idx & (T - 1);
    const float e = X[r * PX + cc];
    const float h = tf32_round(e);
    const int64_t g = (i0 + r) * a.ldw + j0 + cc;
    a.e_hi[g] = h;
    a.e_lo[g] = a.round_lo ? tf32_round(e - h) : e - h;
  }
}

cudaError_t launch_leaf(const LeafArgs& a, int n_tiles, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(leaf_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLeafSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(leaf_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kLeafSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  count_launch();
  if (a.preround)
    leaf_kernel<true><<<n_tiles, NTHR, kLeafSmem, s>>>(a);
  else
    leaf_kernel<false><<<n_tiles, NTHR, kLeafSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace bakron
