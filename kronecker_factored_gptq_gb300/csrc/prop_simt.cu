// Propagation products on the fp32 FMA pipes: the exact-fp32 path, selected
// with bakron_opts.use_3xtf32 = 0 (prop_tc.cu holds the tensor-core path).
//
// One CTA per work item: a 128 x 128 output tile C[r][c] = sum_k A[r][k] B[c][k]
// over the item's K tiles, A and B read as (hi + lo) pairs, which restores
// their exact fp32 values.  Stage 1 stores C split into (hi, lo), after
// adding it to the fp32 accumulator when one is given (the row accumulators
// of the solve); stage 2 subtracts C from the working matrix W~.
#include "internal.cuh"

namespace bakron {

namespace {
constexpr int BM = 128, BN = 128, BK = 16, PAD = 4;
}

__global__ void __launch_bounds__(256) prop_simt_kernel(PropArgs p) {
  __shared__ __align__(16) float As[BK][BM + PAD];
  __shared__ __align__(16) float Bs[BK][BN + PAD];
  const WorkItem it = p.items[blockIdx.x];
  if (!item_in_bounds(it, p)) {
    if (threadIdx.x == 0) set_status(p.st, BAKRON_ERR_INVALID_ARG);
    return;
  }
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int64_t r0 = (int64_t)it.r * BM, c0 = (int64_t)it.c * BN;

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  const int lrow = tid >> 1;          // 0..127
  const int lk = (tid & 1) * 8;       // 0 or 8
  const int64_t kbeg = (int64_t)it.k0 * kTile, kend = (int64_t)it.k1 * kTile;
  for (int64_t k = kbeg; k < kend; k += BK) {
    {
      const int64_t ga = (r0 + lrow) * p.lda + k + lk;
      const float4 h0 = *reinterpret_cast<const float4*>(p.A_hi + ga);
      const float4 h1 = *reinterpret_cast<const float4*>(p.A_hi + ga + 4);
      const float4 l0 = *reinterpret_cast<const float4*>(p.A_lo + ga);
      const float4 l1 = *reinterpret_cast<const float4*>(p.A_lo + ga + 4);
      As[lk + 0][lrow] = h0.x + l0.x; As[lk + 1][lrow] = h0.y + l0.y;
      As[lk + 2][lrow] = h0.z + l0.z; As[lk + 3][lrow] = h0.w + l0.w;
      As[lk + 4][lrow] = h1.x + l1.x; As[lk + 5][lrow] = h1.y + l1.y;
      As[lk + 6][lrow] = h1.z + l1.z; As[lk + 7][lrow] = h1.w + l1.w;
      const int64_t gb = (c0 + lrow) * p.ldb + k + lk;
      const float4 g0 = *reinterpret_cast<const float4*>(p.B_hi + gb);
      const float4 g1 = *reinterpret_cast<const float4*>(p.B_hi + gb + 4);
      const float4 m0 = *reinterpret_cast<const float4*>(p.B_lo + gb);
      const float4 m1 = *reinterpret_cast<const float4*>(p.B_lo + gb + 4);
      Bs[lk + 0][lrow] = g0.x + m0.x; Bs[lk + 1][lrow] = g0.y + m0.y;
      Bs[lk + 2][lrow] = g0.z + m0.z; Bs[lk + 3][lrow] = g0.w + m0.w;
      Bs[lk + 4][lrow] = g1.x + m1.x; Bs[lk + 5][lrow] = g1.y + m1.y;
      Bs[lk + 6][lrow] = g1.z + m1.z; Bs[lk + 7][lrow] = g1.w + m1.w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t r = r0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
#pragma unroll
    for (int jh = 0; jh < 2; ++jh) {
      const int64_t c = c0 + jh * 64 + tx * 4;
      if (p.stage == 1) {
        if (p.acc) {   // running sum: acc += C, then split
          float4* ap = reinterpret_cast<float4*>(p.acc + r * p.ldo + c);
          const float4 a0 = *ap;
          acc[i][jh * 4 + 0] += a0.x; acc[i][jh * 4 + 1] += a0.y;
          acc[i][jh * 4 + 2] += a0.z; acc[i][jh * 4 + 3] += a0.w;
          *ap = make_float4(acc[i][jh * 4 + 0], acc[i][jh * 4 + 1], acc[i][jh * 4 + 2], acc[i][jh * 4 + 3]);
        }
        float4 h, l;
        h.x = tf32_round(acc[i][jh * 4 + 0]); l.x = acc[i][jh * 4 + 0] - h.x;
        h.y = tf32_round(acc[i][jh * 4 + 1]); l.y = acc[i][jh * 4 + 1] - h.y;
        h.z = tf32_round(acc[i][jh * 4 + 2]); l.z = acc[i][jh * 4 + 2] - h.z;
        h.w = tf32_round(acc[i][jh * 4 + 3]); l.w = acc[i][jh * 4 + 3] - h.w;
        *reinterpret_cast<float4*>(p.out_hi + r * p.ldo + c) = h;
        *reinterpret_cast<float4*>(p.out_lo + r * p.ldo + c) = l;
      } else {
        float4* w = reinterpret_cast<float4*>(p.wt + r * p.ldw + c);
        atomicAdd(w, make_float4(-acc[i][jh * 4 + 0], -acc[i][jh * 4 + 1], -acc[i][jh * 4 + 2],
                                 -acc[i][jh * 4 + 3]));
      }
    }
  }
}

cudaError_t launch_prop_simt(const PropArgs& p, cudaStream_t s) {
  if (p.n_items == 0) return cudaSuccess;
  count_launch();
  prop_simt_kernel<<<p.n_items, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace bakron
