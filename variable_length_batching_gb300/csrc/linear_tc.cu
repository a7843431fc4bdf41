// Single-side projections Y = X W^T (+ b) (+ R) on the tcgen05 tensor cores,
// bf16 operands, fp32 accumulation: the u, v and g Linear layers of the
// block ("DanLing NestedTensor" Eq. 1; projections are V W^T + b, section
// 3.3 "Dense work across valid positions") over the T packed single rows.
//
// Small problems: one CTA per 128 x 64 output tile (and per problem: u and
// v run in one launch).  Warp 0 streams 64-wide K blocks of X and W through a TMA ring
// of up to six stages, warp 1 issues the MMAs into a 64-column TMEM
// accumulator, and all four warps run the epilogue: TMEM -> +bias
// (+residual) -> global.  The grids are small (tens of CTAs for the
// block's projections), so each CTA's chain of copies sets the time: the
// ring holds every K block of a C_s = 384 contraction at once, and one
// round of copies replaces three.
//
// Large problems (the pair cells' GEMMs of the block backward, millions of
// rows): persistent CTAs, two per SM, each walking 128 x 128 output tiles
// (the N tiles of one row block consecutively, so they share its X rows in
// L2) through one TMA ring that runs on across tiles, into two TMEM
// accumulators used in turn: warps 2-5 write out one tile while warp 1
// accumulates the next.
#include "tc_ptx.cuh"

namespace nt {
namespace {

using namespace tc;

constexpr int kBM = 128, kBN = 64, kBK = 64;
constexpr int kThreads = 128;
constexpr uint32_t kXBytes = kBM * kBK * 2;           // 16 KB X block per stage
constexpr uint32_t kWBytes = kBN * kBK * 2;           // 8 KB W block per stage
constexpr uint32_t kStageBytes = kXBytes + kWBytes;   // a multiple of the 1 KB swizzle atom
constexpr uint32_t kTmemCols = kBN;                   // one fp32 accumulator column per output column
constexpr int kMaxStages = 6;
constexpr uint32_t kBarBytes = 256;

struct Bars {
  uint64_t full[kMaxStages], empty[kMaxStages], acc_full;
  uint32_t tmem_base;
  int abort;
};

struct Prob {
  const float* bias;
  const bf16* R;     // residual [M, N], or null
  void* Y;           // [M, N], fp32 or bf16
};

template <bool kOutF32>
__global__ void __launch_bounds__(kThreads)
linear_tc_kernel(const __grid_constant__ CUtensorMap tx0, const __grid_constant__ CUtensorMap tw0,
                 const __grid_constant__ CUtensorMap tx1, const __grid_constant__ CUtensorMap tw1, Prob p0, Prob p1,
                 int64_t M, int N, int K, int stages, unsigned int* status) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023) {
    pdl_wait();   // a kernel that waits on this one must also see the previous one done
    if (threadIdx.x == 0) flag_device(status, kDevCheck);
    return;
  }
  const CUtensorMap* tx = blockIdx.z == 0 ? &tx0 : &tx1;
  const CUtensorMap* tw = blockIdx.z == 0 ? &tw0 : &tw1;
  const Prob& pr = blockIdx.z == 0 ? p0 : p1;
  Bars& bar = *reinterpret_cast<Bars*>(smem + stages * kStageBytes);
  volatile int* abort_flag = &bar.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the N tiles of one M tile are consecutive blocks, so they run together
  // and read their X rows from L2 rather than each from HBM
  const int ntiles = N / kBN;
  const int64_t m0 = (int64_t)(blockIdx.x / ntiles) * kBM;
  const int n0 = (int)(blockIdx.x % ntiles) * kBN;
  const int nkb = K / kBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) { mbar_init(&bar.full[i], 1); mbar_init(&bar.empty[i], 1); }
    mbar_init(&bar.acc_full, 1);
    bar.abort = 0;
    fence_mbar_init();
    fence_async_shared();
  }
  if (warp == 1) tmem_alloc(&bar.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;
  // the set-up above overlaps the previous kernel's tail; its outputs (X, R)
  // are read only after it has completed
  pdl_wait();
  pdl_trigger();

  if (warp == 0 && lane == 0) {
    int issued = 0;
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb % stages;
      if (!mbar_wait(&bar.empty[st], ((kb / stages) & 1) ^ 1, abort_flag, status)) break;
      mbar_arrive_expect_tx(&bar.full[st], kStageBytes);
      tma_load_2d(smem + st * kStageBytes, tx, &bar.full[st], kb * kBK, (int)m0);
      tma_load_2d(smem + st * kStageBytes + kXBytes, tw, &bar.full[st], kb * kBK, n0);
      issued = kb + 1;
    }
    for (int kb = issued - stages; kb < issued; ++kb)
      if (kb >= 0) mbar_wait(&bar.full[kb % stages], (kb / stages) & 1, nullptr, status);
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16_f32(kBM, kBN);
    const uint32_t base = smem_u32(smem);
    for (int kb = 0; kb < nkb; ++kb) {
      const int st = kb % stages;
      if (!mbar_wait(&bar.full[st], (kb / stages) & 1, abort_flag, status)) break;
      tc_fence_after();
      const uint32_t a = base + st * kStageBytes, b = a + kXBytes;
      for (int k = 0; k < kBK / 16; ++k)
        mma_bf16(tmem, sdesc_k128(a + k * 32), sdesc_k128(b + k * 32), idesc, (kb > 0 || k > 0) ? 1u : 0u);
      mma_commit(&bar.empty[st]);
    }
    mma_commit(&bar.acc_full);
  }
  // epilogue: every warp, one accumulator row per thread
  const int r = warp * 32 + lane;
  const int64_t row = m0 + r;
  // the residual row does not depend on the MMAs: its loads are issued
  // before the accumulator wait and land while the tensor core works
  uint4 res[kBN / 8];
  const bool has_r = pr.R != nullptr && row < M;
  if (has_r) {
    const uint4* rp = reinterpret_cast<const uint4*>(pr.R + row * N + n0);
#pragma unroll
    for (int u = 0; u < kBN / 8; ++u) res[u] = rp[u];
  }
  if (mbar_wait_warp(&bar.acc_full, 0, abort_flag, status)) {
    tc_fence_after();
    __syncwarp();
    const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
#pragma unroll
    for (int g = 0; g < kBN / 32; ++g) {
      float v[32];
      tmem_ld32(tmem + lane_addr + 32 * g, v);
      tmem_ld_wait();
      if (row < M) {
        const int c0 = n0 + 32 * g;
        if (pr.bias) {
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] += pr.bias[c0 + c];
        }
        if (has_r) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 q4 = res[4 * g + u];
            const uint32_t w[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              v[8 * u + 2 * e] += bf16lo(w[e]);
              v[8 * u + 2 * e + 1] += bf16hi(w[e]);
            }
          }
        }
        if (kOutF32) {
          float* y = static_cast<float*>(pr.Y) + row * N + c0;
#pragma unroll
          for (int c = 0; c < 32; c += 4) *reinterpret_cast<float4*>(y + c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
        } else {
          bf16* y = static_cast<bf16*>(pr.Y) + row * N + c0;
#pragma unroll
          for (int c = 0; c < 32; c += 8)
            *reinterpret_cast<uint4*>(y + c) = make_uint4(pack_bf16x2(v[c], v[c + 1]), pack_bf16x2(v[c + 2], v[c + 3]),
                                                          pack_bf16x2(v[c + 4], v[c + 5]), pack_bf16x2(v[c + 6], v[c + 7]));
        }
      }
    }
  }
  if (warp == 1 && lane == 0) {
    // nothing may still be writing TMEM when it is released
    mbar_wait(&bar.acc_full, 0, nullptr, status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}


// ---------------------------------------------------------------- persistent

constexpr int kPN = 128;                                  // output columns per tile
constexpr uint32_t kPXBytes = kBM * kBK * 2;              // 16 KB
constexpr uint32_t kPWBytes = kPN * kBK * 2;              // 16 KB
constexpr uint32_t kPStageBytes = kPXBytes + kPWBytes;
constexpr uint32_t kPStgBytes = 32 * 64;                  // an epilogue warp's 32 rows x 64 bytes
constexpr int kPMaxStages = 6;

// One problem per tile: two CTAs per SM, each with a 3-stage ring, two
// 128-column accumulators used in turn and 4 epilogue warps.  Two problems
// (dual): one CTA per SM with a 5-stage ring, two accumulator pairs (all
// 512 columns) used in turn and 8 epilogue warps (each lane quadrant split
// into two column halves).
template <bool kDual>
struct PCfg {
  static constexpr int kStages = kDual ? 5 : 3;
  static constexpr int kEpiWarps = kDual ? 8 : 4;
  static constexpr int kThreads = (2 + kEpiWarps) * 32;
  static constexpr uint32_t kTmemCols = kDual ? 4 * kPN : 2 * kPN;
  static constexpr uint32_t kOffBar = kStages * kPStageBytes;
  static constexpr uint32_t kOffStg = kOffBar + 256;
  static constexpr uint32_t kSmemBytes = kOffStg + kEpiWarps * kPStgBytes + 1024;
  static constexpr int kCtasPerSm = kDual ? 1 : 2;
};

struct PBars {
  uint64_t full[kPMaxStages], empty[kPMaxStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(PBars) <= 256, "barrier block");

// kDual: two problems per output tile, A = X W^T (K) and B = X2 W2^T (K2),
// into one accumulator pair; Y = ReLU(A + bias) and Y2 = B where bf16(Y) >
// 0, both bf16.
template <bool kOutF32, bool kDual>
__global__ void __launch_bounds__(PCfg<kDual>::kThreads)
linear_tc_persistent_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw,
                            const __grid_constant__ CUtensorMap tx2, const __grid_constant__ CUtensorMap tw2, Prob pr,
                            bf16* Y2, int64_t M, int N, int K, int K2, unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  using C = PCfg<kDual>;
  constexpr int kPStages = C::kStages;
  PBars& bar = *reinterpret_cast<PBars*>(smem + C::kOffBar);
  volatile int* abort_flag = &bar.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = N / kPN, nkb = K / kBK;
  const int nkt = nkb + (kDual ? K2 / kBK : 0);        // k blocks per tile
  constexpr int kBufs = 2;                              // accumulators (pairs) in turn
  const int64_t tiles = (M + kBM - 1) / kBM * ntiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPStages; ++i) { mbar_init(&bar.full[i], 1); mbar_init(&bar.empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&bar.acc_full[i], 1); mbar_init(&bar.acc_empty[i], C::kEpiWarps); }
    mbar_init(&bar.mma_done, 1);
    bar.abort = 0;
    fence_mbar_init();
    fence_async_shared();
  }
  if (warp == 1) tmem_alloc(&bar.tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tx); prefetch_tmap(&tw);
      if (kDual) { prefetch_tmap(&tx2); prefetch_tmap(&tw2); }
      int64_t g = 0;                              // k blocks issued, over all tiles
      bool ok = true;
      for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        const int m0 = (int)(t / ntiles) * kBM, n0 = (int)(t % ntiles) * kPN;
        for (int kb = 0; kb < nkt; ++kb, ++g) {
          const int st = (int)(g % kPStages);
          if (!(ok = mbar_wait(&bar.empty[st], (uint32_t)((g / kPStages) & 1) ^ 1, abort_flag, status))) break;
          mbar_arrive_expect_tx(&bar.full[st], kPStageBytes);
          const bool second = kDual && kb >= nkb;
          const int kx = (second ? kb - nkb : kb) * kBK;
          tma_load_2d(smem + st * kPStageBytes, second ? &tx2 : &tx, &bar.full[st], kx, m0);
          tma_load_2d(smem + st * kPStageBytes + kPXBytes, second ? &tw2 : &tw, &bar.full[st], kx, n0);
        }
      }
      // drain the copies this thread issued
      for (int64_t k = g - kPStages; k < g; ++k)
        if (k >= 0) mbar_wait(&bar.full[k % kPStages], (uint32_t)((k / kPStages) & 1), nullptr, status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, kPN);
      const uint32_t base = smem_u32(smem);
      int64_t g = 0;
      int i = 0;                                  // tiles of this CTA
      bool ok = true;
      for (int64_t t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++i) {
        const int b = i % kBufs;
        // the accumulator is free once the epilogue has read tile i - kBufs out of it
        if (i >= kBufs &&
            !(ok = mbar_wait(&bar.acc_empty[b], (uint32_t)((i / kBufs) - 1) & 1, abort_flag, status)))
          break;
        tc_fence_after();
        for (int kb = 0; kb < nkt; ++kb, ++g) {
          const int st = (int)(g % kPStages);
          if (!(ok = mbar_wait(&bar.full[st], (uint32_t)((g / kPStages) & 1), abort_flag, status))) break;
          tc_fence_after();
          const uint32_t a = base + st * kPStageBytes, w = a + kPXBytes;
          // dual: the first problem into columns 0.., the second into kPN..
          const bool second = kDual && kb >= nkb;
          const uint32_t acc = tmem + (kDual ? b * 2 * kPN + (second ? kPN : 0) : b * kPN);
          const bool first_kb = second ? kb == nkb : kb == 0;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_bf16(acc, sdesc_k128(a + k * 32), sdesc_k128(w + k * 32), idesc, (!first_kb || k > 0) ? 1u : 0u);
          mma_commit(&bar.empty[st]);
        }
        if (ok) mma_commit(&bar.acc_full[b]);
      }
      mma_commit(&bar.mma_done);
      mbar_wait(&bar.mma_done, 0, nullptr, status);
    }
  } else {
    // epilogue: row (warp & 3) * 32 + lane of each tile.  Rows leave (and
    // mask or residual rows arrive) through the warp's 32 x 64-byte buffer in
    // shared memory, so that global accesses are 4 lanes x 16 bytes per row
    // instead of one lane per row; the 16-byte chunk c of row r sits at
    // chunk c ^ ((r >> 1) & 3), which keeps both access patterns free of
    // bank conflicts.
    const int q = warp & 3;                       // the TMEM lane quadrant this warp may read
    const int ew = warp - 2;                      // epilogue warp index
    const int hh = kDual ? ew >> 2 : 0;           // dual: its half of the tile's columns
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    uint8_t* stg = smem + C::kOffStg + ew * kPStgBytes;
    const int cr = lane >> 2, cc = lane & 3;     // coalesced role: rows cr + 8 i, chunk cc
    auto stg_at = [&](int r, int c) { return reinterpret_cast<uint4*>(stg + r * 64 + 16 * (c ^ ((r >> 1) & 3))); };
    // 32 rows x 64 bytes of the warp from the buffer to global rows row0 + r
    // (row-major, `pitch` bytes apart), rows >= M skipped
    auto flush = [&](uint8_t* g0, int64_t row0, size_t pitch) {
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = cr + 8 * i;
        const uint4 val = *stg_at(r, cc);
        if (row0 + r < M) *reinterpret_cast<uint4*>(g0 + (row0 + r) * pitch + 16 * cc) = val;
      }
      __syncwarp();
    };
    int i = 0;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
      const int b = i % kBufs;
      const int64_t row0 = (t / ntiles) * kBM + q * 32;   // the warp's first row
      const int n0 = (int)(t % ntiles) * kPN;
      // the residual or mask rows do not depend on the MMAs: their loads are
      // issued before the accumulator wait, 4 lanes per row (group gq, rows
      // cr + 8 j)
      uint4 rall[kPN / 8];
      if (!kDual && pr.R) {
#pragma unroll
        for (int gq = 0; gq < kPN / 32; ++gq)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int64_t rw = row0 + cr + 8 * j;
            rall[4 * gq + j] = rw < M ? *reinterpret_cast<const uint4*>(pr.R + rw * N + n0 + 32 * gq + 8 * cc)
                                      : make_uint4(0u, 0u, 0u, 0u);
          }
      }
      if (!mbar_wait_warp(&bar.acc_full[b], (uint32_t)(i / kBufs) & 1, abort_flag, status)) break;
      tc_fence_after();
      __syncwarp();
      if (kDual) {
#pragma unroll 1
        for (int gq = 2 * hh; gq < 2 * hh + 2; ++gq) {
          const int c0 = n0 + 32 * gq;
          float v[32];
          uint32_t hw[16];
          tmem_ld32_sync(tmem + lane_addr + b * 2 * kPN + 32 * gq, v);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float b0 = pr.bias ? pr.bias[c0 + 2 * c] : 0.f, b1 = pr.bias ? pr.bias[c0 + 2 * c + 1] : 0.f;
            hw[c] = pack_bf16x2(fmaxf(v[2 * c] + b0, 0.f), fmaxf(v[2 * c + 1] + b1, 0.f));
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) *stg_at(lane, c) = make_uint4(hw[4 * c], hw[4 * c + 1], hw[4 * c + 2], hw[4 * c + 3]);
          flush(reinterpret_cast<uint8_t*>(static_cast<bf16*>(pr.Y) + c0), row0, (size_t)N * 2);
          tmem_ld32_sync(tmem + lane_addr + b * 2 * kPN + kPN + 32 * gq, v);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            if (!(bf16lo(hw[c]) > 0.f)) v[2 * c] = 0.f;
            if (!(bf16hi(hw[c]) > 0.f)) v[2 * c + 1] = 0.f;
          }
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *stg_at(lane, c) = make_uint4(pack_bf16x2(v[8 * c], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                                          pack_bf16x2(v[8 * c + 4], v[8 * c + 5]),
                                          pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
          flush(reinterpret_cast<uint8_t*>(Y2 + c0), row0, (size_t)N * 2);
        }
      } else
#pragma unroll
      for (int gq = 0; gq < kPN / 32; ++gq) {
        const int c0 = n0 + 32 * gq;
        float v[32];
        tmem_ld32_sync(tmem + lane_addr + b * kPN + 32 * gq, v);
        uint4 rq[4];
        if (pr.R) {
          // the group's rows to one row per lane
#pragma unroll
          for (int j = 0; j < 4; ++j) *stg_at(cr + 8 * j, cc) = rall[4 * gq + j];
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 4; ++c) rq[c] = *stg_at(lane, c);
          __syncwarp();
        }
        if (pr.bias) {
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] += pr.bias[c0 + c];
        }
        if (pr.R) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t w[4] = {rq[u].x, rq[u].y, rq[u].z, rq[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              v[8 * u + 2 * e] += bf16lo(w[e]);
              v[8 * u + 2 * e + 1] += bf16hi(w[e]);
            }
          }
        }
        if (kOutF32) {
          // two rounds of 16 columns (64 bytes of fp32)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *stg_at(lane, c) = make_uint4(__float_as_uint(v[16 * h + 4 * c]), __float_as_uint(v[16 * h + 4 * c + 1]),
                                            __float_as_uint(v[16 * h + 4 * c + 2]),
                                            __float_as_uint(v[16 * h + 4 * c + 3]));
            flush(reinterpret_cast<uint8_t*>(static_cast<float*>(pr.Y) + c0 + 16 * h), row0, (size_t)N * 4);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *stg_at(lane, c) = make_uint4(pack_bf16x2(v[8 * c], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                                          pack_bf16x2(v[8 * c + 4], v[8 * c + 5]),
                                          pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
          flush(reinterpret_cast<uint8_t*>(static_cast<bf16*>(pr.Y) + c0), row0, (size_t)N * 2);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.acc_empty[b]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace

bool linear_tc_supported(int in_dtype, int64_t M, int N, int K) {
  return in_dtype == NT_BF16 && M > 0 && N % kBN == 0 && K % kBK == 0 && K > 0 && M < 0x7fffffffLL - kBM;
}

cudaError_t launch_linear_tc_dual(const void* X, const void* W, const float* bias, const void* X2, const void* W2,
                                  void* Y, void* Y2, int64_t M, int N, int K, int K2, unsigned int* status,
                                  cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  if (N % kPN != 0 || K % kBK != 0 || K2 % kBK != 0 || K <= 0 || K2 <= 0 || M >= 0x7fffffffLL - kBM)
    return cudaErrorInvalidValue;
  const int64_t ptiles = (M + kBM - 1) / kBM * (N / kPN);
  CUtensorMap px, pw, px2, pw2;
  if (!make_tmap_rows(&px, X, (uint64_t)K, (uint64_t)M, kBM) || !make_tmap_rows(&pw, W, (uint64_t)K, (uint64_t)N, kPN) ||
      !make_tmap_rows(&px2, X2, (uint64_t)K2, (uint64_t)M, kBM) ||
      !make_tmap_rows(&pw2, W2, (uint64_t)K2, (uint64_t)N, kPN))
    return cudaErrorInvalidValue;
  const Prob pp0 = Prob{bias, nullptr, Y};
  using C = PCfg<true>;
  const int grid = (int)min64(ptiles, (int64_t)C::kCtasPerSm * sm_count());
  auto kern = linear_tc_persistent_kernel<false, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, s, px, pw, px2, pw2, pp0, static_cast<bf16*>(Y2),
                 M, N, K, K2, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_linear_tc(int out_f32, const LinearProblem* probs, int nprob, int64_t M, int N, int K,
                             unsigned int* status, cudaStream_t s) {
  if (M == 0 || nprob == 0) return cudaSuccess;
  const int64_t ptiles = (M + kBM - 1) / kBM * (N / kPN);
  if (nprob == 1 && N % kPN == 0 && ptiles >= (int64_t)8 * sm_count()) {
    // large: persistent CTAs, two per SM
    const LinearProblem& lp = probs[0];
    CUtensorMap px, pw;
    if (!make_tmap_rows(&px, lp.X, (uint64_t)K, (uint64_t)M, kBM) ||
        !make_tmap_rows(&pw, lp.W, (uint64_t)K, (uint64_t)N, kPN))
      return cudaErrorInvalidValue;
    const Prob pp0 = Prob{lp.bias, static_cast<const bf16*>(lp.R), lp.Y};
    using C = PCfg<false>;
    const int grid = (int)min64(ptiles, (int64_t)C::kCtasPerSm * sm_count());
    auto kern = out_f32 ? linear_tc_persistent_kernel<true, false> : linear_tc_persistent_kernel<false, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, s, px, pw, px, pw, pp0, (bf16*)nullptr, M, N,
                   K, 0, status);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  CUtensorMap tx[2], tw[2];
  Prob pp[2];
  for (int i = 0; i < 2; ++i) {
    const LinearProblem& lp = probs[i < nprob ? i : 0];
    if (!make_tmap_rows(&tx[i], lp.X, (uint64_t)K, (uint64_t)M, kBM) ||
        !make_tmap_rows(&tw[i], lp.W, (uint64_t)K, (uint64_t)N, kBN))
      return cudaErrorInvalidValue;
    pp[i] = Prob{lp.bias, static_cast<const bf16*>(lp.R), lp.Y};
  }
  const int64_t blocks = (M + kBM - 1) / kBM * (N / kBN);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  dim3 grid((unsigned)blocks, 1, nprob);
  const int stages = min(K / kBK, kMaxStages);
  const uint32_t smem = stages * kStageBytes + kBarBytes;
  cudaError_t e;
  if (out_f32) {
    e = cudaFuncSetAttribute(linear_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(kMaxStages * kStageBytes + kBarBytes));
    if (e != cudaSuccess) return e;
    e = launch_pdl(linear_tc_kernel<true>, grid, dim3(kThreads), smem, s, tx[0], tw[0], tx[1], tw[1], pp[0], pp[1],
                   M, N, K, stages, status);
    if (e != cudaSuccess) return e;
  } else {
    e = cudaFuncSetAttribute(linear_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(kMaxStages * kStageBytes + kBarBytes));
    if (e != cudaSuccess) return e;
    e = launch_pdl(linear_tc_kernel<false>, grid, dim3(kThreads), smem, s, tx[0], tw[0], tx[1], tw[1], pp[0], pp[1],
                   M, N, K, stages, status);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace nt
