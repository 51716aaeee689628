// Propagation products on the tcgen05 tensor cores with a 3xTF32 split.
//
// The two propagation stages of BaKron (summary page "FastKron: Efficient
// Quantization with Kronecker-Factored Hessians", section 3: the error of the
// first half of the anti-diagonals is pushed into the second half with dense
// products) are both "C[r][c] = sum_k A[r][k] B[c][k]" over lists of
// 128 x 128 output tiles with per-tile K ranges.  Each operand is stored
// pre-split, x = hi + lo with hi = tf32(x); the tensor core accumulates
//     C = A_hi B_hi + (A_hi B_lo + A_lo B_hi)
// dropping only A_lo B_lo (relative size 2^-22).
//
// Accuracy of the accumulation.  Inside one MMA chain the tensor core keeps
// the fp32 accumulator with truncating additions, so a chain of thousands
// of MMAs drifts far beyond fp32 rounding.  The chain is therefore cut after
// every 128-wide K tile: each K tile accumulates into a fresh TMEM buffer
// (the main A_hi B_hi products and the small correction products in separate
// buffers), and the epilogue warps add the finished buffer into fp32
// registers with round-to-nearest additions while the tensor core fills the
// other buffer of the pair.  The low parts this kernel writes for its own
// consumers are rounded to tf32 (round to nearest), so the tensor core reads
// them exactly.
//
// One CTA (8 warps) per work item:
//   warp 0, one thread: TMA producer, 3-stage ring of 32-wide K slices, each
//     stage holding A_hi, A_lo, B_hi, B_lo as 128 x 32 fp32 tiles with the
//     128-byte swizzle (64 KiB per stage);
//   warp 1, one thread: issues tcgen05.mma (M = N = 128, K = 8 per
//     instruction, 3 per K step) and commits each stage back to the producer
//     and each finished K tile to the epilogue;
//   warp 2: allocates / frees the 512 TMEM columns (main and correction
//     accumulators, two of each);
//   warps 4-7: epilogue, TMEM -> registers (warp 4 + q owns TMEM lanes
//     32q..32q+31, i.e. output rows) -> running fp32 sums -> global: stage 1
//     writes C split into (hi, lo) (or, with an fp32 accumulator, adds C to
//     it and writes the sum back and split), stage 2 subtracts C from W~,
//     stage 3 writes alpha C plainly (the factor accumulation).
// Every mbarrier wait is bounded (clock64 budget); on expiry the CTA records
// BAKRON_ERR_TIMEOUT, stops issuing, drains its own copies and MMAs (with a
// bound again), frees TMEM and returns.
#include "tc_common.cuh"

namespace bakron {

using namespace tc;

namespace {
constexpr int BM = 128, BN = 128, BKF = 32;      // tile rows, cols, K slice (floats)
constexpr int STAGES = 3;
constexpr uint32_t TILE_BYTES = BM * BKF * 4;    // 16 KiB
constexpr uint32_t STAGE_BYTES = 4 * TILE_BYTES; // A_hi, A_lo, B_hi, B_lo
constexpr size_t kSmem = (size_t)STAGES * STAGE_BYTES + 1024;
constexpr uint32_t TMEM_COLS = 512;             // main[2] at 0, 128; corr[2] at 256, 384
constexpr int SPC = kTile / BKF;                 // K slices per accumulation chunk
constexpr int NTHREADS = 256;
constexpr int SPITCH = BN + 4;                   // epilogue staging pitch (floats)
static_assert(4 * 32 * SPITCH * 4 <= STAGES * STAGE_BYTES, "epilogue staging fits the ring");

constexpr uint32_t kIdesc = tc::idesc_tf32(BM, BN);

}  // namespace

// Two item lists in one launch: CTAs [0, n_first) take list 0 (maps m0,
// arguments p0), the rest list 1 (m1, p1); a single list passes n_first =
// its length.
__global__ void __launch_bounds__(NTHREADS, 1)
    prop_tc_kernel(const __grid_constant__ CUtensorMap m0_ahi, const __grid_constant__ CUtensorMap m0_alo,
                   const __grid_constant__ CUtensorMap m0_bhi, const __grid_constant__ CUtensorMap m0_blo,
                   const __grid_constant__ CUtensorMap m1_ahi, const __grid_constant__ CUtensorMap m1_alo,
                   const __grid_constant__ CUtensorMap m1_bhi, const __grid_constant__ CUtensorMap m1_blo,
                   const __grid_constant__ PropArgs p0, const __grid_constant__ PropArgs p1, int n_first,
                   DevStatus* st) {
  const bool second = (int)blockIdx.x >= n_first;
  const PropArgs& p = second ? p1 : p0;
  const CUtensorMap& tm_ahi = second ? m1_ahi : m0_ahi;
  const CUtensorMap& tm_alo = second ? m1_alo : m0_alo;
  const CUtensorMap& tm_bhi = second ? m1_bhi : m0_bhi;
  const CUtensorMap& tm_blo = second ? m1_blo : m0_blo;
  const int item = second ? (int)blockIdx.x - n_first : (int)blockIdx.x;
  extern __shared__ __align__(1024) unsigned char dsm[];
  __shared__ __align__(8) unsigned long long bar_full[STAGES], bar_empty[STAGES];
  __shared__ __align__(8) unsigned long long acc_full[2], acc_empty[2], bar_done;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WorkItem it = p.items[item];
  if (!item_in_bounds(it, p)) {   // uniform over the CTA: nothing set up yet
    if (threadIdx.x == 0) set_status(st, BAKRON_ERR_INVALID_ARG);
    return;
  }
  const int nk = (it.k1 - it.k0) * SPC;     // K slices
  const int nc = it.k1 - it.k0;             // accumulation chunks (K tiles)
  // 1024-byte aligned stage ring
  const uint32_t base_raw = smem_u32(dsm);
  const uint32_t sbase = (base_raw + 1023u) & ~1023u;

  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_ahi) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_alo) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_bhi) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_blo) : "memory");
    abort_flag = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), 4);   // one arrival per epilogue warp
    }
    mbar_init(smem_u32(&bar_done), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_slot;
  volatile int* abortp = &abort_flag;
  // the operands (and, for stage 2, W~) come from the previous kernels
  grid_dep_wait();

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    const int kx0 = it.k0 * kTile;
    const int ya = it.r * BM, yb = it.c * BN;
    int issued = 0;
    for (int i = 0; i < nk; ++i) {
      const int s = i % STAGES;
      const uint32_t u = (uint32_t)(i / STAGES);
      if (i >= STAGES && !mbar_wait(smem_u32(&bar_empty[s]), (u & 1u) ^ 1u, abortp)) {
        set_status(st, BAKRON_ERR_TIMEOUT);
        *abortp = 1;
        break;
      }
      const uint32_t fb = smem_u32(&bar_full[s]);
      mbar_expect_tx(fb, STAGE_BYTES);
      const uint32_t sd = sbase + (uint32_t)s * STAGE_BYTES;
      const int x = kx0 + i * BKF;
      tma_load_2d(sd, &tm_ahi, fb, x, ya);
      tma_load_2d(sd + TILE_BYTES, &tm_alo, fb, x, ya);
      tma_load_2d(sd + 2 * TILE_BYTES, &tm_bhi, fb, x, yb);
      tma_load_2d(sd + 3 * TILE_BYTES, &tm_blo, fb, x, yb);
      ++issued;
    }
    // drain: every issued copy must have landed before the CTA may exit
    for (int i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i) {
      const int s = i % STAGES;
      const uint32_t u = (uint32_t)(i / STAGES);
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_u32(&bar_full[s]), u & 1u)) {
        if (clock64() - t0 > kBudget) { set_status(st, BAKRON_ERR_TIMEOUT); break; }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    for (int i = 0; i < nk; ++i) {
      const int c = i / SPC, b = c & 1;
      const bool first = (i % SPC) == 0;
      if (first && c >= 2 &&
          !mbar_wait(smem_u32(&acc_empty[b]), (uint32_t)((c / 2 - 1) & 1), abortp)) {
        set_status(st, BAKRON_ERR_TIMEOUT);
        *abortp = 1;
        break;
      }
      const int s = i % STAGES;
      const uint32_t u = (uint32_t)(i / STAGES);
      if (!mbar_wait(smem_u32(&bar_full[s]), u & 1u, abortp)) {
        set_status(st, BAKRON_ERR_TIMEOUT);
        *abortp = 1;
        break;
      }
      fence_after_sync();
      const uint32_t sd = sbase + (uint32_t)s * STAGE_BYTES;
      const uint64_t ahi = desc_sw128(sd), alo = desc_sw128(sd + TILE_BYTES);
      const uint64_t bhi = desc_sw128(sd + 2 * TILE_BYTES), blo = desc_sw128(sd + 3 * TILE_BYTES);
      const uint32_t tm_main = tmem + (uint32_t)(b * 128);
      const uint32_t tm_corr = tmem + 256u + (uint32_t)(b * 128);
#pragma unroll
      for (int j = 0; j < BKF / 8; ++j) {
        const uint64_t o = (uint64_t)(j * 32 >> 4);  // 8 tf32 = 32 bytes along K
        const uint32_t acc = (first && j == 0) ? 0u : 1u;
        mma_tf32(tm_main, ahi + o, bhi + o, kIdesc, acc);
        mma_tf32(tm_corr, ahi + o, blo + o, kIdesc, acc);
        mma_tf32(tm_corr, alo + o, bhi + o, kIdesc, 1u);
      }
      mma_commit(smem_u32(&bar_empty[s]));
      if ((i % SPC) == SPC - 1) mma_commit(smem_u32(&acc_full[b]));
    }
    mma_commit(smem_u32(&bar_done));
    grid_dep_launch();   // every MMA of this CTA is issued
  } else if (warp >= 4) {
    // ---------------- epilogue: running fp32 sums of the K-tile chunks
    const int q = warp - 4;                 // TMEM lane quarter (warp % 4)
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    if (p.stage == 1 && p.acc) {
      // the running sums this warp adds in at the end: into L2 now, while
      // the tensor core works (32 rows x 512 bytes, four 128-byte lines each)
      const float* ar = p.acc + ((int64_t)it.r * BM + q * 32 + lane) * p.ldo + (int64_t)it.c * BN;
#pragma unroll
      for (int l = 0; l < 4; ++l) asm volatile("prefetch.global.L2 [%0];" ::"l"(ar + 32 * l));
    }
    float acc[BN];
#pragma unroll
    for (int t = 0; t < BN; ++t) acc[t] = 0.f;
    bool ok = true;
    for (int c = 0; c < nc && ok; ++c) {
      const int b = c & 1;
      ok = mbar_wait(smem_u32(&acc_full[b]), (uint32_t)((c / 2) & 1), abortp);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      fence_after_sync();
#pragma unroll
      for (int g = 0; g < BN / 32; ++g) {
        float v[32];
        tmem_ld32(tmem + lane_off + (uint32_t)(b * 128 + g * 32), v);
#pragma unroll
        for (int t = 0; t < 32; ++t) acc[g * 32 + t] += v[t];
        tmem_ld32(tmem + lane_off + 256u + (uint32_t)(b * 128 + g * 32), v);
#pragma unroll
        for (int t = 0; t < 32; ++t) acc[g * 32 + t] += v[t];
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&acc_empty[b]))
                                  : "memory");
    }
    if (!ok) {
      set_status(st, BAKRON_ERR_TIMEOUT);
      *abortp = 1;
    }
    if (ok) {
      const int row = q * 32 + lane;
      if (p.stage != 2) {
        if (p.alpha != 0.f && p.alpha != 1.f) {
#pragma unroll
          for (int t = 0; t < BN; ++t) acc[t] *= p.alpha;
        }
        if (p.stage == 1 && p.tr_hi) {
          // transposed split store: lane = output row, so for each column the
          // 32 lanes of a warp write 32 consecutive floats
          const int64_t tcol = (int64_t)it.r * BM + row;
#pragma unroll
          for (int t = 0; t < BN; ++t) {
            const int64_t trow = (int64_t)it.c * BN + t;
            const float h = tf32_round(acc[t]);
            p.tr_hi[trow * p.ldt + tcol] = h;
            p.tr_lo[trow * p.ldt + tcol] = tf32_round(acc[t] - h);
          }
        }
      }
      // Coalesced write-out: each warp stages its 32 rows in the (now idle)
      // TMA ring, then writes whole 512-byte rows, so a store or atomic
      // instruction covers four 128-byte lines instead of 32 rows.  Every
      // MMA has completed (the last accumulator chunk was consumed), so no
      // copy or MMA touches the ring any more.
      float* stg = reinterpret_cast<float*>(dsm + (sbase - base_raw)) + q * 32 * SPITCH;
#pragma unroll
      for (int t = 0; t < BN / 4; ++t)
        *reinterpret_cast<float4*>(stg + lane * SPITCH + 4 * t) =
            make_float4(acc[4 * t + 0], acc[4 * t + 1], acc[4 * t + 2], acc[4 * t + 3]);
      __syncwarp();
      const int64_t grow0 = (int64_t)it.r * BM + q * 32;
      const int64_t gcol = (int64_t)it.c * BN + 4 * lane;
      if (p.stage == 1 && p.acc) {
        // running sums: acc += C (the fp32 tile), written back, then split;
        // all of the warp's loads in flight at once
        float4 a0[32];
#pragma unroll
        for (int rr = 0; rr < 32; ++rr)
          a0[rr] = *reinterpret_cast<const float4*>(p.acc + (grow0 + rr) * p.ldo + gcol);
#pragma unroll
        for (int rr = 0; rr < 32; ++rr) {
          float4 v = *reinterpret_cast<const float4*>(stg + rr * SPITCH + 4 * lane);
          v.x += a0[rr].x; v.y += a0[rr].y; v.z += a0[rr].z; v.w += a0[rr].w;
          *reinterpret_cast<float4*>(p.acc + (grow0 + rr) * p.ldo + gcol) = v;
          float4 h, l;
          h.x = tf32_round(v.x); l.x = tf32_round(v.x - h.x);
          h.y = tf32_round(v.y); l.y = tf32_round(v.y - h.y);
          h.z = tf32_round(v.z); l.z = tf32_round(v.z - h.z);
          h.w = tf32_round(v.w); l.w = tf32_round(v.w - h.w);
          *reinterpret_cast<float4*>(p.out_hi + (grow0 + rr) * p.ldo + gcol) = h;
          *reinterpret_cast<float4*>(p.out_lo + (grow0 + rr) * p.ldo + gcol) = l;
        }
      } else if (p.stage == 1) {
#pragma unroll 4
        for (int rr = 0; rr < 32; ++rr) {
          const float4 v = *reinterpret_cast<const float4*>(stg + rr * SPITCH + 4 * lane);
          float4 h, l;
          h.x = tf32_round(v.x); l.x = tf32_round(v.x - h.x);
          h.y = tf32_round(v.y); l.y = tf32_round(v.y - h.y);
          h.z = tf32_round(v.z); l.z = tf32_round(v.z - h.z);
          h.w = tf32_round(v.w); l.w = tf32_round(v.w - h.w);
          *reinterpret_cast<float4*>(p.out_hi + (grow0 + rr) * p.ldo + gcol) = h;
          *reinterpret_cast<float4*>(p.out_lo + (grow0 + rr) * p.ldo + gcol) = l;
        }
      } else if (p.stage == 3) {
#pragma unroll 4
        for (int rr = 0; rr < 32; ++rr) {
          const float4 v = *reinterpret_cast<const float4*>(stg + rr * SPITCH + 4 * lane);
          *reinterpret_cast<float4*>(p.wt + (grow0 + rr) * p.ldw + gcol) = v;
        }
      } else {
        // atomic: propagations of different recursion depths may update the
        // same tile concurrently (they run on different streams)
#pragma unroll 4
        for (int rr = 0; rr < 32; ++rr) {
          const float4 v = *reinterpret_cast<const float4*>(stg + rr * SPITCH + 4 * lane);
          atomicAdd(reinterpret_cast<float4*>(p.wt + (grow0 + rr) * p.ldw + gcol),
                    make_float4(-v.x, -v.y, -v.z, -v.w));
        }
      }
    }
  }
  __syncwarp();

  // all MMAs must have completed before TMEM is freed (bounded wait)
  if (warp == 2) {
    const long long t0 = clock64();
    bool done = true;
    while (!mbar_try_wait(smem_u32(&bar_done), 0u)) {
      if (clock64() - t0 > kBudget) { done = false; break; }
    }
    if (!__all_sync(0xffffffffu, done) && lane == 0) set_status(st, BAKRON_ERR_TIMEOUT);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    fence_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                 : "memory");
  }
}

namespace tc {
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

}  // namespace

bool encode_available() { return encode_fn() != nullptr; }

bool make_map(CUtensorMap* m, const float* ptr, int64_t rows, int64_t ld) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)ld, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * sizeof(float)};
  const cuuint32_t box[2] = {(cuuint32_t)BKF, (cuuint32_t)BM};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace tc

bool prop_tc_supported() {
  static std::atomic<int> cached{-1};
  const int c = cached.load(std::memory_order_acquire);
  if (c >= 0) return c == 1;
  int dev = 0, major = 0, minor = 0;
  bool ok = cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
            major == 10 && minor == 3 && tc::encode_available();
  if (!ok) (void)cudaGetLastError();
  cached.store(ok ? 1 : 0, std::memory_order_release);
  return ok;
}

namespace {
bool make_maps(CUtensorMap* m, const PropArgs& p) {
  return make_map(&m[0], p.A_hi, p.a_rows, p.lda) && make_map(&m[1], p.A_lo, p.a_rows, p.lda) &&
         make_map(&m[2], p.B_hi, p.b_rows, p.ldb) && make_map(&m[3], p.B_lo, p.b_rows, p.ldb);
}
}  // namespace

cudaError_t launch_prop_tc2(const PropArgs& a, const PropArgs& b, cudaStream_t s) {
  if (a.n_items + b.n_items == 0) return cudaSuccess;
  static std::atomic<unsigned long long> done;
  cudaError_t e = ensure_smem_limit((const void*)prop_tc_kernel, kSmem, done);
  if (e != cudaSuccess) return e;
  CUtensorMap ma[4], mb[4];
  if (!make_maps(ma, a)) return cudaErrorInvalidValue;
  if (b.n_items > 0) {
    if (!make_maps(mb, b)) return cudaErrorInvalidValue;
  } else {
    for (int i = 0; i < 4; ++i) mb[i] = ma[i];
  }
  count_launch();
  return launch_kernel(prop_tc_kernel, dim3((unsigned)(a.n_items + b.n_items)), dim3(NTHREADS), kSmem, s,
                       a.pdl != 0, ma[0], ma[1], ma[2], ma[3], mb[0], mb[1], mb[2], mb[3], a,
                       b.n_items > 0 ? b : a, a.n_items, a.st);
}

cudaError_t launch_prop_tc(const PropArgs& p, cudaStream_t s) {
  if (p.n_items == 0) return cudaSuccess;
  PropArgs none = p;
  none.n_items = 0;
  return launch_prop_tc2(p, none, s);
}

}  // namespace bakron
