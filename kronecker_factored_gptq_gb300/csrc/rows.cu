// One-sided GPTQ: the B = I case of the BaKron problem.
//
// With B = I the rows of W are independent problems, each ordinary GPTQ with
// Hessian A (the ainews article on BaKron compares against this one-sided
// GPTQ, whose Hessian has the form A (x) I; Theorem 3.2 of the summary page
// "FastKron: Efficient Quantization with Kronecker-Factored Hessians" makes
// any column order that keeps each row left to right give the same result).
// Entry (i, j) has scaled error E_ij = (w~_ij - s_i c_ij) l^A_j and updates
// w~[i, j'] -= E_ij U_A[j, j'] for j' > j.
//
// The solve runs over column tiles of 128: a leaf quantizes one column tile
// of every row tile at once (one CTA per 128 x 128 tile), and a
// divide-and-conquer over column tiles pushes the error of the left half of
// the tiles into the right half with the tensor-core products of the
// two-sided solver (W~[I, J'] -= sum_J E[I, J] U_A[J, J']).
//
// Leaf, per tile: four 32-column blocks in turn.  (a) One thread per row
// sweeps the block's 32 columns; the pending updates from earlier columns of
// the block live in a 32-register window FR[t] = sum_{b' < t} e(b') Ua(b', t)
// (every register index static, the column loop fully unrolled); row b of Ua
// is read with 16-byte broadcast loads.  (b) All threads apply the block's
// error to the tile's later columns, X[:, later] -= E[:, block] Ua[block,
// later], with register tiles.
#include "internal.cuh"

namespace bakron {

namespace {
constexpr int T = kTile;           // 128
constexpr int CB = 32;             // column block of the sweep
constexpr int NTH = 256;
constexpr int PX = T + 4;          // pitch of the X and Ua tiles (16-byte rows)
constexpr int PC = T + 4;          // pitch of the code tile (bytes)
constexpr int OFF_X = 0;
constexpr int OFF_U = OFF_X + T * PX;          // Ua(r, c) of the diagonal block, row-major
constexpr int OFF_LA = OFF_U + T * PX;         // 1 / Ua(b, b)
constexpr int OFF_CS = OFF_LA + T;             // codes [T][PC]
constexpr int SMEM_FLOATS = OFF_CS + T * PC / 4;
constexpr size_t kRowsSmem = sizeof(float) * (size_t)SMEM_FLOATS;
static_assert(kRowsSmem <= 232448, "row leaf shared memory");
}  // namespace

template <bool PRE>
__global__ void __launch_bounds__(NTH, 1) rows_leaf_kernel(LeafArgs a) {
  extern __shared__ __align__(16) float smem[];
  float* X = smem + OFF_X;     // [T][PX]: W~, then E column by column
  float* U = smem + OFF_U;     // [T][PX]: Ua(r, c), zero below the diagonal
  float* lA = smem + OFF_LA;   // [T]
  signed char* CS = reinterpret_cast<signed char*>(smem + OFF_CS);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Itile = blockIdx.x, Jtile = a.D;
  const int64_t i0 = (int64_t)Itile * T, j0 = (int64_t)Jtile * T;

  // The factor block was written at the start of the solve: read it before
  // waiting for the previous kernel (which writes W~).  Global U_A^T rows
  // (= columns c of Ua) are read as float4 along r and written transposed:
  // a warp covers 32 consecutive c, so the shared stores are conflict-free.
  for (int idx = tid; idx < T * T / 4; idx += NTH) {
    const int c = idx & (T - 1), rq = (idx >> 7) * 4;
    const int64_t g = (j0 + c) * a.lda + j0 + rq;
    const float4 h = *reinterpret_cast<const float4*>(a.lat_hi + g);
    const float4 l = *reinterpret_cast<const float4*>(a.lat_lo + g);
    U[(rq + 0) * PX + c] = (rq + 0 <= c) ? h.x + l.x : 0.f;
    U[(rq + 1) * PX + c] = (rq + 1 <= c) ? h.y + l.y : 0.f;
    U[(rq + 2) * PX + c] = (rq + 2 <= c) ? h.z + l.z : 0.f;
    U[(rq + 3) * PX + c] = (rq + 3 <= c) ? h.w + l.w : 0.f;
  }
  grid_dep_wait();
#pragma unroll 4
  for (int idx = tid; idx < T * T / 4; idx += NTH) {
    const int r = idx >> 5, c = (idx & 31) * 4;
    *reinterpret_cast<float4*>(X + r * PX + c) =
        *reinterpret_cast<const float4*>(a.wt + (i0 + r) * a.ldw + j0 + c);
  }
  __syncthreads();
  if (tid < T) lA[tid] = 1.f / U[tid * PX + tid];
  __syncthreads();

  const float fqmin = (float)a.qmin, fqmax = (float)a.qmax;
  const bool wide = a.qmin < -128 || a.qmax > 127;
  bool out_of_range = false;
  const int row = tid;                       // sweep: threads 0..127, one row each

  for (int cb = 0; cb < T / CB; ++cb) {
    const int q = cb * CB;
    // ---- (a) sweep of columns q .. q + 31, one thread per row; the block's
    // columns lie in one group of the grid (groups are whole multiples of 32
    // columns, or the whole row)
    if (tid < T) {
      int64_t grp = (j0 + q) / a.group;
      if (grp > a.ngroups - 1) grp = a.ngroups - 1;
      const int64_t gidx = (i0 + row) * a.ngroups + grp;
      const float sc = a.scale[gidx], zc = a.zero[gidx];
      const float rinv = 1.f / sc;
      const float clo = fqmin - zc, chi = fqmax - zc;   // centred code range
      float* Xr = X + row * PX + q;
      float FR[CB];
#pragma unroll
      for (int t = 0; t < CB; ++t) FR[t] = 0.f;
      unsigned* cr = reinterpret_cast<unsigned*>(CS + row * PC + q);
      // four columns at a time: a 16-byte load of x0, a 16-byte store of e and
      // one 4-byte store of the codes (row pitch 132: the eight rows of a
      // quarter warp fall in distinct bank groups)
#pragma unroll
      for (int g = 0; g < CB / 4; ++g) {
        const float4 x4 = *reinterpret_cast<const float4*>(Xr + 4 * g);
        const float xg[4] = {x4.x, x4.y, x4.z, x4.w};
        float eg[4];
        unsigned cw = 0;
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          const int b = 4 * g + bb;
          const float x = xg[bb] - FR[b];
          float c = rintf(x * rinv);
          c = fminf(fmaxf(c, clo), chi);
          const float e = (x - sc * c) * lA[q + b];
          const float code = c + zc;
          if (wide) out_of_range |= (code < -128.f) || (code > 127.f);
          eg[bb] = e;
          short c8;   // saturating conversion to the int8 range
          asm("cvt.rzi.sat.s8.f32 %0, %1;" : "=h"(c8) : "f"(code));
          cw |= ((unsigned)c8 & 0xffu) << (8 * bb);
          if (PRE) {
            const int64_t gi = i0 + row, gj = j0 + q + b;
            if (gi < a.m && gj < a.n) a.preround[gi * a.n + gj] = x;
          }
          // FR[t] += e Ua(q + b, q + t) for the later columns of the block
          const float* ur = U + (q + b) * PX + q;
#pragma unroll
          for (int t4 = 0; t4 < CB / 4; ++t4) {
            if (4 * t4 + 3 > b) {
              const float4 u = *reinterpret_cast<const float4*>(ur + 4 * t4);
              if (4 * t4 + 0 > b) FR[4 * t4 + 0] = fmaf(e, u.x, FR[4 * t4 + 0]);
              if (4 * t4 + 1 > b) FR[4 * t4 + 1] = fmaf(e, u.y, FR[4 * t4 + 1]);
              if (4 * t4 + 2 > b) FR[4 * t4 + 2] = fmaf(e, u.z, FR[4 * t4 + 2]);
              FR[4 * t4 + 3] = fmaf(e, u.w, FR[4 * t4 + 3]);
            }
          }
        }
        *reinterpret_cast<float4*>(Xr + 4 * g) = make_float4(eg[0], eg[1], eg[2], eg[3]);
        cr[g] = cw;
        // keep the next group's loads from being hoisted here (registers)
        asm volatile("" ::: "memory");
      }
    }
    __syncthreads();
    // ---- (b) later columns of the tile: X[:, q+32 ..] -= E[:, q .. q+31] Ua[q.., q+32 ..],
    // in passes of at most 48 columns; thread: rows 8 tr .. 8 tr + 7,
    // columns cs + tc + 16 u (u < nc / 16)
    for (int cs = q + CB; cs < T; cs += 48) {
      const int nc = min(48, T - cs), nu = nc / 16;
      const int tr = tid >> 4, tc = tid & 15;
      float acc[8][3];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int u = 0; u < 3; ++u) acc[i][u] = 0.f;
#pragma unroll 2
      for (int k = 0; k < CB; k += 4) {
        float4 e4[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) e4[i] = *reinterpret_cast<const float4*>(X + (8 * tr + i) * PX + q + k);
#pragma unroll
        for (int u = 0; u < 3; ++u) {
          if (u < nu) {
            const int col = cs + tc + 16 * u;
            const float u0 = U[(q + k + 0) * PX + col], u1 = U[(q + k + 1) * PX + col];
            const float u2 = U[(q + k + 2) * PX + col], u3 = U[(q + k + 3) * PX + col];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              acc[i][u] = fmaf(e4[i].x, u0, acc[i][u]);
              acc[i][u] = fmaf(e4[i].y, u1, acc[i][u]);
              acc[i][u] = fmaf(e4[i].z, u2, acc[i][u]);
              acc[i][u] = fmaf(e4[i].w, u3, acc[i][u]);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 3; ++u)
        if (u < nu) {
          const int col = cs + tc + 16 * u;
#pragma unroll
          for (int i = 0; i < 8; ++i) X[(8 * tr + i) * PX + col] -= acc[i][u];
        }
    }
    __syncthreads();
  }
  if (out_of_range) set_status(a.st, BAKRON_ERR_CODE_RANGE);
  grid_dep_launch();

  // ---- write-out: E (split) for the propagation, codes and V (coalesced rows)
  bool nonfinite = false;
  for (int idx = tid; idx < T * T / 4; idx += NTH) {
    const int r = idx >> 5, cc = (idx & 31) * 4;
    const float4 e = *reinterpret_cast<const float4*>(X + r * PX + cc);
    nonfinite |= !isfinite(e.x) || !isfinite(e.y) || !isfinite(e.z) || !isfinite(e.w);
    float4 h, l;
    h.x = tf32_round(e.x); h.y = tf32_round(e.y); h.z = tf32_round(e.z); h.w = tf32_round(e.w);
    l.x = tf32_round(e.x - h.x); l.y = tf32_round(e.y - h.y);
    l.z = tf32_round(e.z - h.z); l.w = tf32_round(e.w - h.w);
    const int64_t g = (i0 + r) * a.ldw + j0 + cc;
    *reinterpret_cast<float4*>(a.e_hi + g) = h;
    *reinterpret_cast<float4*>(a.e_lo + g) = l;
  }
  if (nonfinite) set_status(a.st, BAKRON_ERR_NONFINITE);
  // codes and V: warp w writes rows w, w + 8, ...; lane = 4 consecutive columns
  for (int r = warp; r < T; r += NTH / 32) {
    const int64_t gi = i0 + r;
    if (gi >= a.m) continue;
    const int64_t jc = j0 + 4 * lane;
    int64_t grp = jc / a.group;
    if (grp > a.ngroups - 1) grp = a.ngroups - 1;
    const float s = a.scale[gi * a.ngroups + grp], z = a.zero[gi * a.ngroups + grp];
    const signed char* cr = CS + r * PC + 4 * lane;
    if (jc + 3 < a.n && (a.n & 3) == 0) {
      const int64_t base = gi * a.n + jc;
      *reinterpret_cast<unsigned*>(a.codes + base) = *reinterpret_cast<const unsigned*>(cr);
      *reinterpret_cast<float4*>(a.V + base) =
          make_float4(s * ((float)cr[0] - z), s * ((float)cr[1] - z), s * ((float)cr[2] - z),
                      s * ((float)cr[3] - z));
    } else {
      for (int t = 0; t < 4; ++t)
        if (jc + t < a.n) {
          a.codes[gi * a.n + jc + t] = cr[t];
          a.V[gi * a.n + jc + t] = s * ((float)cr[t] - z);
        }
    }
  }
}

cudaError_t launch_rows_leaf(const LeafArgs& a, int n_row_tiles, cudaStream_t s) {
  static std::atomic<unsigned long long> done[2];
  cudaError_t e = ensure_smem_limit((const void*)rows_leaf_kernel<false>, kRowsSmem, done[0]);
  if (e == cudaSuccess) e = ensure_smem_limit((const void*)rows_leaf_kernel<true>, kRowsSmem, done[1]);
  if (e != cudaSuccess) return e;
  count_launch();
  if (a.preround)
    return launch_kernel(rows_leaf_kernel<true>, dim3(n_row_tiles), dim3(NTH), kRowsSmem, s,
                         a.pdl != 0, a);
  return launch_kernel(rows_leaf_kernel<false>, dim3(n_row_tiles), dim3(NTH), kRowsSmem, s,
                       a.pdl != 0, a);
}

}  // namespace bakron
