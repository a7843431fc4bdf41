// Weight gradients over the packed pair cells on the tcgen05 tensor cores,
// bf16 operands, fp32 accumulation:
//     G[m, n] = sum_p A[p, m] B[p, n]          (A: [P, M], B: [P, N], row-major,
//                                               rows lda and ldb elements apart)
//     c[m]    = sum_p A[p, m]                  (optional: the bias gradient)
// the contractions over all P cells that the backward of the pair
// transition needs ("DanLing NestedTensor" Eq. 1 second line: dW1 = dA^T
// LN(z), dW2 = dP~^T ReLU(A), db1 = sum dA, db2 = sum dP~).
//
// Both operands stay in their row-major cell layout: a 64-cell chunk of A
// is two TMA boxes of 64 columns x 64 cells (128-byte swizzle), which the
// MMA reads MN-major (M along the 128-byte rows, K = cells down them; the
// two 64-column atoms 8 KB apart, 8-cell groups 1 KB apart); B the same.
// The reduction runs over cells, so it is split: CTA (mt, nt, s) adds
// split s's chunks into a 128 x 128 TMEM accumulator and writes it to its
// own partial block; a second kernel sums the partials in split order, so
// the result does not depend on timing.
//
// Warps: 0 = TMA producer (3-stage ring), 1 = TMEM owner and MMA issuer,
// 2-3 = column sums of A from the staged tiles (each column by one of the
// CTAs that read the tile); then all four warps write the accumulator (one
// row per thread).
#include "tc_ptx.cuh"

namespace nt {
namespace {

using namespace tc;

constexpr int kBM = 128, kBN = 128, kBP = 64;         // G rows, G columns, cells per chunk
constexpr int kStages = 3;
constexpr int kThreads = 128;
constexpr uint32_t kABytes = kBP * kBM * 2;           // 16 KB: two 64-column boxes
constexpr uint32_t kBBytes = kBP * kBN * 2;           // 16 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kAtomBytes = kBP * 128;            // one 64-column box: 8 KB
// Room past the last stage: a descriptor reads only within its tile, and
// the slack keeps every address the MMA could form inside the allocation.
constexpr uint32_t kSlack = 12 * 1024;
constexpr uint32_t kOffBar = kStages * kStageBytes + kSlack;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;   // + barriers + alignment
constexpr uint32_t kTmemCols = kBN;

struct Bars {
  uint64_t full[kStages], empty[kStages], acc_full;
  uint32_t tmem_base;
  int abort;
};

// Shared-memory descriptor of an MN-major operand in the 128-byte swizzled
// layout: rows of 128 bytes along K, 8-row groups 1 KB apart (stride byte
// offset), 64-element atoms along M or N `atom_bytes` apart (leading byte
// offset).
__device__ __forceinline__ uint64_t sdesc_mn128(uint32_t saddr, uint32_t atom_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((atom_bytes >> 4) & 0x3FFFu) << 16;   // leading byte offset
  d |= (uint64_t)(1024u >> 4) << 32;                    // stride byte offset
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

template <int kTpp>
__global__ void __launch_bounds__(kThreads)
wgrad_tc_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb, int64_t P, int M,
                int N, int chunks_per_split, float* __restrict__ part, float* __restrict__ col_part,
                unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  Bars& bar = *reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort_flag = &bar.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x, nt = blockIdx.y, sp = blockIdx.z;
  const int64_t nchunks_all = (P + kBP - 1) / kBP;
  const int64_t c0 = (int64_t)sp * chunks_per_split;
  const int nch = (int)max64(0, min64((int64_t)chunks_per_split, nchunks_all - c0));
  // Column sums of the A tile, shared by the N / 128 CTAs that read it: CTA
  // nt takes column pairs [p_lo, p_hi) of the tile's 64, and each pair is
  // summed by kTpp consecutive threads (a power of two), thread `sub` taking
  // every kTpp-th cell; the pair's partials are added in sub order at the end.
  const int NT = N / kBN;
  const int p_lo = nt * 64 / NT, p_hi = (nt + 1) * 64 / NT, npairs = p_hi - p_lo;
  const bool sums = col_part != nullptr && npairs > 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar.full[i], 1);
      mbar_init(&bar.empty[i], 3);             // the MMAs' commit and the two column-sum warps
    }
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
  pdl_wait();
  pdl_trigger();

  float csum[2] = {0.f, 0.f};                   // this thread's share of its column pair's sums
  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&ta); prefetch_tmap(&tb);
      int issued = 0;
      for (int k = 0; k < nch; ++k) {
        const int st = k % kStages;
        if (!mbar_wait(&bar.empty[st], ((k / kStages) & 1) ^ 1, abort_flag, status)) break;
        uint8_t* a = smem + st * kStageBytes;
        const int p0 = (int)((c0 + k) * kBP);
        mbar_arrive_expect_tx(&bar.full[st], kStageBytes);
        tma_load_2d(a, &ta, &bar.full[st], mt * kBM, p0);
        tma_load_2d(a + kAtomBytes, &ta, &bar.full[st], mt * kBM + 64, p0);
        tma_load_2d(a + kABytes, &tb, &bar.full[st], nt * kBN, p0);
        tma_load_2d(a + kABytes + kAtomBytes, &tb, &bar.full[st], nt * kBN + 64, p0);
        issued = k + 1;
      }
      for (int k = issued - kStages; k < issued; ++k)
        if (k >= 0) mbar_wait(&bar.full[k % kStages], (k / kStages) & 1, nullptr, status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // both operands MN-major
      const uint32_t idesc = idesc_bf16_f32(kBM, kBN) | (1u << 15) | (1u << 16);
      const uint32_t base = smem_u32(smem);
      for (int k = 0; k < nch; ++k) {
        const int st = k % kStages;
        if (!mbar_wait(&bar.full[st], (k / kStages) & 1, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t a = base + st * kStageBytes, b = a + kABytes;
#pragma unroll
        for (int kk = 0; kk < kBP / 16; ++kk)      // 16 cells = 2 KB down the rows
          mma_bf16(tmem, sdesc_mn128(a + kk * 2048, kAtomBytes), sdesc_mn128(b + kk * 2048, kAtomBytes), idesc,
                   (k > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar.empty[st]);
      }
      mma_commit(&bar.acc_full);
    }
  } else {
    // column sums of the A tiles (one 32-bit word, a column pair, per cell)
    const int t = threadIdx.x - 64;             // 0..63
    const int pair = t / kTpp, sub = t % kTpp;
    const bool mine = sums && pair < npairs;
    const int col = 2 * (p_lo + pair);          // the pair's first column in the tile
    for (int k = 0; k < nch; ++k) {
      const int st = k % kStages;
      if (!mbar_wait_warp(&bar.full[st], (k / kStages) & 1, abort_flag, status)) break;
      if (mine) {
        const uint8_t* a = smem + st * kStageBytes;
        float e0 = 0.f, e1 = 0.f, o0 = 0.f, o1 = 0.f;   // two chains
#pragma unroll
        for (int i = 0; i < kBP / (2 * kTpp); ++i) {
          const int r = sub + 2 * kTpp * i;
          const uint32_t w = *reinterpret_cast<const uint32_t*>(a + swz128_offset(r, col, kBP));
          const uint32_t x = *reinterpret_cast<const uint32_t*>(a + swz128_offset(r + kTpp, col, kBP));
          e0 += bf16lo(w);
          e1 += bf16hi(w);
          o0 += bf16lo(x);
          o1 += bf16hi(x);
        }
        csum[0] += e0 + o0;
        csum[1] += e1 + o1;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.empty[st]);
    }
    // the pair's kTpp partials in sub order (the pair's threads share a
    // warp: kTpp is a power of two and pairs start at multiples of it)
    float tot0 = csum[0], tot1 = csum[1];
#pragma unroll
    for (int j = 1; j < kTpp; ++j) {
      const float a0 = __shfl_down_sync(0xffffffffu, csum[0], j);
      const float a1 = __shfl_down_sync(0xffffffffu, csum[1], j);
      tot0 += a0;
      tot1 += a1;
    }
    if (mine && sub == 0) {
      col_part[(int64_t)sp * M + mt * kBM + col] = tot0;
      col_part[(int64_t)sp * M + mt * kBM + col + 1] = tot1;
    }
  }

  // the partial block: row mt*128 + r of G, columns nt*128 .. +127
  const int r = warp * 32 + lane;
  float* out = part + ((int64_t)sp * M + mt * kBM + r) * N + nt * kBN;
  if (nch == 0) {
    for (int c = 0; c < kBN; c += 4) *reinterpret_cast<float4*>(out + c) = make_float4(0.f, 0.f, 0.f, 0.f);
  } else if (mbar_wait_warp(&bar.acc_full, 0, abort_flag, status)) {
    tc_fence_after();
    __syncwarp();
    const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
    for (int g = 0; g < kBN / 32; ++g) {
      float v[32];
      tmem_ld32_sync(tmem + lane_addr + 32 * g, v);
#pragma unroll
      for (int c = 0; c < 32; c += 4)
        *reinterpret_cast<float4*>(out + 32 * g + c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
    }
  }
  if (warp == 1 && lane == 0 && nch > 0) mbar_wait(&bar.acc_full, 0, nullptr, status);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// G = sum over the splits of the partial blocks, in split order; c likewise.
__global__ void wgrad_finish_kernel(const float* __restrict__ part, const float* __restrict__ col_part, int splits,
                                    int M, int N, float* __restrict__ G, float* __restrict__ c) {
  const int64_t MN = (int64_t)M * N;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < MN + (c ? M : 0);
       e += (int64_t)gridDim.x * blockDim.x) {
    float acc = 0.f;
    if (e < MN) {
      for (int s = 0; s < splits; ++s) acc += part[(int64_t)s * MN + e];
      G[e] = acc;
    } else {
      const int64_t m = e - MN;
      for (int s = 0; s < splits; ++s) acc += col_part[(int64_t)s * M + m];
      c[m] = acc;
    }
  }
}

// Splits of the cell range: about 304 CTAs in all (two per SM of a 152-SM
// GPU), each with at least 16 chunks.  A fixed count, not the device's, so
// the workspace size and the order of the final sum are the same on every
// GPU.
constexpr int64_t kTargetCtas = 304;
int wgrad_splits(int64_t P, int M, int N) {
  const int64_t chunks = (P + kBP - 1) / kBP;
  const int64_t tiles = (int64_t)(M / kBM) * (N / kBN);
  const int64_t s = min64(kTargetCtas / tiles, (chunks + 15) / 16);
  return (int)max64(1, s);
}

}  // namespace

bool wgrad_tc_supported(int64_t P, int M, int N) {
  return P > 0 && P < 0x7fffffffLL && M % kBM == 0 && N % kBN == 0 && M > 0 && N > 0;
}

size_t wgrad_tc_workspace_bytes(int64_t P, int M, int N) {
  const int s = wgrad_splits(P, M, N);
  return (size_t)s * ((size_t)M * N + M) * sizeof(float);
}

cudaError_t launch_wgrad_tc(const void* A, int lda, const void* B, int ldb, int64_t P, int M, int N, float* G,
                            float* colsum, void* workspace, unsigned int* status, cudaStream_t s) {
  CUtensorMap ta, tb;
  const uint64_t da[2] = {(uint64_t)M, (uint64_t)P}, db[2] = {(uint64_t)N, (uint64_t)P};
  const uint64_t sa[1] = {(uint64_t)lda * 2}, sb[1] = {(uint64_t)ldb * 2};
  const uint32_t box[2] = {64, (uint32_t)kBP};
  if (lda < M || ldb < N || !make_tmap_bf16(&ta, A, 2, da, sa, box) || !make_tmap_bf16(&tb, B, 2, db, sb, box))
    return cudaErrorInvalidValue;
  const int splits = wgrad_splits(P, M, N);
  const int64_t chunks = (P + kBP - 1) / kBP;
  const int cps = (int)((chunks + splits - 1) / splits);
  float* part = static_cast<float*>(workspace);
  float* col_part = colsum ? part + (int64_t)splits * M * N : nullptr;
  // threads per column pair: the largest power of two that lets every CTA's
  // share of the 64 pairs (at most ceil(64 / NT)) fit its 64 summing threads
  const int NT = N / kBN, most = (64 + NT - 1) / NT;
  int tpp = 1;
  while (tpp < 32 && 2 * tpp * most <= 64) tpp *= 2;
  auto kern = tpp >= 32 ? wgrad_tc_kernel<32> : tpp == 16 ? wgrad_tc_kernel<16> : tpp == 8 ? wgrad_tc_kernel<8>
            : tpp == 4 ? wgrad_tc_kernel<4> : tpp == 2 ? wgrad_tc_kernel<2> : wgrad_tc_kernel<1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(M / kBM, N / kBN, splits), dim3(kThreads), kSmemBytes, s, ta, tb, P, M, N, cps, part,
                 col_part, status);
  if (e != cudaSuccess) return e;
  const int64_t work = (int64_t)M * N + (colsum ? M : 0);
  wgrad_finish_kernel<<<(unsigned)min64((work + 255) / 256, (int64_t)sm_count() * 8), 256, 0, s>>>(
      part, col_part, splits, M, N, G, colsum);
  return cudaGetLastError();
}

}  // namespace nt
