// Backward of variable-length attention on the tcgen05 tensor cores, bf16 in
// / fp32 accumulate, head width 64 ("Variable-length attention and data
// packing", "What it is" / "How it works"; the causal and cross forms as in
// the forward).  Per segment and head, with P rebuilt from the forward's
// natural-log LSE (no running max: P = exp(scale s - lse) <= 1),
//     dP = dO V^T,  dS = P * (dP - D),  D = rowsum(dO * O)
//     dQ = scale dS K,   dK = scale dS^T Q,   dV = P^T dO.
// Two kernels, so that every output row has one owner and no atomics:
//
// dQ kernel (first): one CTA per (segment, 128-query tile, head), walking
// the key tiles of 64 the tile's queries see.  Its compute threads form D
// of their query rows from O and dO while the first S / dP are computed, use
// it, and write it out for the dK/dV kernel.
//   S  = Q K_j^T, dP = dO V_j^T          (M=128, N=64, K=64)  -> TMEM
//   dS -> bf16, written by the compute threads over dP's columns
//   dQ += dS K_j                          (A from TMEM, K_j MN-major)
//
// dK/dV kernel (second): one CTA per (segment, 128-key tile, head), walking the query
// tiles of 64 that see the tile's keys.  In the transposed frame (keys on
// the TMEM lanes) the per-query LSE and D are column constants, staged in
// shared memory by the producer warp beside each query tile.
//   S^T = K Q_i^T, dP^T = V dO_i^T        -> TMEM
//   P^T over S^T's columns, dS^T over dP^T's (bf16)
//   dV += P^T dO_i,  dK += dS^T Q_i       (A from TMEM, B MN-major)
//
// Warps: 0 = TMA producer, 1 = TMEM owner and MMA issuer (one elected lane
// issues), 2-9 = compute, two warps per TMEM lane quadrant, each taking 32
// of a tile's 64 columns.  256 TMEM columns and about 82 KB of shared memory
// per CTA: two CTAs share an SM.  Every wait is bounded.

#include "tc_ptx.cuh"

namespace nt {
namespace {

using namespace tc;

constexpr int kD = 64;
constexpr int kBM = 128;                       // rows held for the CTA's life
constexpr int kBN = 64;                        // rows of a streamed tile
constexpr int kStages = 3;
constexpr int kThreads = 10 * 32;
constexpr uint32_t kBigBytes = kBM * kD * 2;   // 16 KB
constexpr uint32_t kSmallBytes = kBN * kD * 2; // 8 KB
constexpr uint32_t kOffBig0 = 0;
constexpr uint32_t kOffBig1 = kBigBytes;
constexpr uint32_t kOffRing = 2 * kBigBytes;   // stage st: tile X at +16 KB st, tile Y 8 KB after
constexpr uint32_t kOffAux = kOffRing + kStages * 2 * kSmallBytes;
constexpr uint32_t kAuxBytes = 2 * kBN * 4;    // per stage: -lse (log2 units) and -D of 64 queries
constexpr uint32_t kOffBar = kOffAux + kStages * kAuxBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256;
// The dQ kernels stage no LSE/D; their O tile (128 rows, for D) sits where
// the dK/dV kernels keep those, and their barrier block follows it.
constexpr uint32_t kOffOQ = kOffAux;
constexpr uint32_t kOffBarQ = kOffOQ + kBigBytes;
constexpr uint32_t kSmemBytesQ = kOffBarQ + 256;
constexpr uint32_t kTmemCols = 256;
// S (or S^T) at 0, dP (or dP^T) at 64, accumulators at 128 (dQ or dV) and 192 (dK)
constexpr uint32_t kColS = 0, kColP = 64, kColAcc0 = 128, kColAcc1 = 192;
constexpr float kLog2e = 1.4426950408889634f;

struct Bars {
  uint64_t big_full;
  uint64_t full[kStages], empty[kStages], aux_full[kStages];
  uint64_t s_full, p_full, p_empty;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// TMEM column of the k-th 16-wide K chunk of an A operand that two compute
// warps wrote as bf16 pairs: tokens [32 g, 32 g + 32) packed into columns
// [32 g, 32 g + 16) of the base.
__device__ __forceinline__ uint32_t a_chunk(uint32_t base, int kk) {
  return base + 32u * (uint32_t)(kk >> 1) + 8u * (uint32_t)(kk & 1);
}

// D = rowsum(dO * O) of row r of the O and dO tiles (128-byte rows of 64
// bf16, 16-byte chunks XOR-swizzled by row as TMA's 128-byte swizzle leaves
// them), in the summation order of the D pass of the CUDA-core route: per
// 8-element chunk two fp32 sums over alternate elements, added, then the
// eight chunk sums pairwise.  So D does not depend on which route formed it.
__device__ __forceinline__ float row_dot64(const uint8_t* o_tile, const uint8_t* do_tile, int r) {
  float s[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int off = r * 128 + ((c ^ (r & 7)) << 4);
    const uint4 a = *reinterpret_cast<const uint4*>(o_tile + off);
    const uint4 b = *reinterpret_cast<const uint4*>(do_tile + off);
    const bf16* ea = reinterpret_cast<const bf16*>(&a);
    const bf16* eb = reinterpret_cast<const bf16*>(&b);
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      acc0 = fmaf(__bfloat162float(eb[e]), __bfloat162float(ea[e]), acc0);
      acc1 = fmaf(__bfloat162float(eb[e + 1]), __bfloat162float(ea[e + 1]), acc1);
    }
    s[c] = acc0 + acc1;
  }
  return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

// The dK/dV kernels start, by programmatic dependent launch, while the dQ
// kernel (which forms D) is still running: they read D only after
// griddepcontrol.wait, and every thread waits once more on its way out, so
// that no dK/dV CTA, and hence the grid, completes before the dQ kernel has.
struct WaitForPrimaryAtExit {
  __device__ ~WaitForPrimaryAtExit() { pdl_wait(); }
};

// The four MMAs of one M=128, N=64, K=64 product with both operands
// K-major in shared memory.
__device__ __forceinline__ void mma_kmajor(uint32_t d, uint32_t a_base, uint32_t b_base, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk)
    mma_bf16(d, sdesc_k128(a_base + kk * 32), sdesc_k128(b_base + kk * 32), idesc, kk > 0);
}

// D (+)= A (TMEM, bf16 pairs at `a_base`, 64 tokens of K) x B (a 64-token
// tile of shared memory read MN-major: token rows, 64 features).
__device__ __forceinline__ void mma_ts_mn(uint32_t d, uint32_t a_base, uint32_t b_base, uint32_t idesc,
                                          bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk)
    mma_bf16_ts(d, a_chunk(a_base, kk), sdesc_k128(b_base + kk * 2048), idesc, (accumulate || kk > 0) ? 1u : 0u);
}

// Output rows leave through shared memory: each compute thread writes its 32
// values (half a 128-byte row) into a [128 rows x 128 B] staging tile, 16-byte
// chunks XOR-swizzled by row, then the 256 compute threads copy whole rows
// out, eight threads per row, so that a warp's store covers four rows
// instead of 32 scattered half rows.
__device__ __forceinline__ void stage_row32(uint8_t* tile, int r, int g, const float* v, float mul) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * u] * mul, v[8 * u + 1] * mul);
    w.y = pack_bf16x2(v[8 * u + 2] * mul, v[8 * u + 3] * mul);
    w.z = pack_bf16x2(v[8 * u + 4] * mul, v[8 * u + 5] * mul);
    w.w = pack_bf16x2(v[8 * u + 6] * mul, v[8 * u + 7] * mul);
    *reinterpret_cast<uint4*>(tile + r * 128 + (((4 * g + u) ^ (r & 7)) << 4)) = w;
  }
}
// Rows [0, rows) of the staging tile to out rows first, first + 1, ... of head h.
__device__ __forceinline__ void copy_out(const uint8_t* tile, bf16* out, int64_t first, int rows, int H, int h,
                                         int ct) {
  for (int e = ct; e < rows * 8; e += 256) {
    const int r = e >> 3, c = e & 7;
    const uint4 w = *reinterpret_cast<const uint4*>(tile + r * 128 + ((c ^ (r & 7)) << 4));
    *reinterpret_cast<uint4*>(out + ((first + r) * H + h) * kD + 8 * c) = w;
  }
}

__device__ __forceinline__ void zero_rows(bf16* base, int64_t first, int rows, int H, int h) {
  for (int e = threadIdx.x; e < rows * (kD / 8); e += kThreads) {
    const int rr = e / (kD / 8), u = e % (kD / 8);
    *reinterpret_cast<uint4*>(base + ((first + rr) * H + h) * kD + 8 * u) = make_uint4(0u, 0u, 0u, 0u);
  }
}

__device__ __forceinline__ void init_bars(Bars& bar) {
  mbar_init(&bar.big_full, 1);
  for (int i = 0; i < kStages; ++i) {
    mbar_init(&bar.full[i], 1);
    mbar_init(&bar.empty[i], 1);
    mbar_init(&bar.aux_full[i], 32);
  }
  mbar_init(&bar.s_full, 1);
  mbar_init(&bar.p_full, 256);
  mbar_init(&bar.p_empty, 1);
  mbar_init(&bar.mma_done, 1);
  bar.abort = 0;
  fence_mbar_init();
  fence_async_shared();
}

// dQ kernel, one key tile: dS = P * (dP - D) for this thread's query row
// (segment-local index row_q) over columns [32 g, 32 g + 32), written as bf16
// pairs over dP's columns.  nL = -lse (log2 units, -inf for a row with no
// key or past the segment), nD = -D.
template <bool kCausal>
__device__ __forceinline__ void dq_tile(uint32_t lane_addr, int g, int j, int n_k, int row_q, int diag,
                                        float scale_log2, float nL, float nD) {
  int cnt = min(kBN, n_k - j * kBN);                   // visible keys: a prefix of the tile
  if (kCausal) cnt = max(0, min(cnt, row_q + diag - j * kBN + 1));
  const bool full = __all_sync(0xffffffffu, cnt >= 32 * g + 32);
  float sv[32], dp[32];
  tmem_ld32(lane_addr + kColS + 32 * g, sv);
  tmem_ld32(lane_addr + kColP + 32 * g, dp);
  tmem_ld_wait();
  uint32_t pk[16];
#pragma unroll
  for (int c = 0; c < 32; c += 2) {                    // packed fp32 pairs
    float x0, x1, p0, p1, e0, e1;
    ffma2(sv[c], sv[c + 1], scale_log2, scale_log2, nL, nL, x0, x1);
    p0 = ex2_approx(x0);
    p1 = ex2_approx(x1);
    if (!full) {
      if (32 * g + c >= cnt) p0 = 0.f;
      if (32 * g + c + 1 >= cnt) p1 = 0.f;
    }
    fadd2(dp[c], dp[c + 1], nD, nD, e0, e1);           // dP - D
    fmul2(p0, p1, e0, e1, e0, e1);
    pk[c / 2] = pack_bf16x2(e0, e1);
  }
  tmem_st16_sync(lane_addr + kColP + 32 * g, pk);
}

// dK/dV kernel, one query tile: P^T and dS^T = P^T * (dP^T - D) for this
// thread's key row over query columns [32 g, 32 g + 32), written as bf16
// pairs over S^T's and dP^T's columns.  aux holds this tile's staged -lse
// (log2 units) and, kBN floats on, -D, from column 32 g; causal: columns
// below cmin (relative to this half) are masked.
template <bool kCausal>
__device__ __forceinline__ void dkv_tile(uint32_t lane_addr, int g, int cmin, const float* aux, float scale_log2) {
  const bool full = !kCausal || __all_sync(0xffffffffu, cmin <= 0);
  float sv[32], dp[32];
  tmem_ld32(lane_addr + kColS + 32 * g, sv);
  tmem_ld32(lane_addr + kColP + 32 * g, dp);
  tmem_ld_wait();
  uint32_t pk[16], ds[16];
#pragma unroll
  for (int c = 0; c < 32; c += 4) {            // P^T, and dS^T = P^T * (dP^T - D), packed pairs
    const float4 L4 = *reinterpret_cast<const float4*>(aux + c);         // -lse
    const float4 D4 = *reinterpret_cast<const float4*>(aux + kBN + c);   // -D
    float x0, x1, x2, x3, p0, p1, p2, p3;
    ffma2(sv[c], sv[c + 1], scale_log2, scale_log2, L4.x, L4.y, x0, x1);
    ffma2(sv[c + 2], sv[c + 3], scale_log2, scale_log2, L4.z, L4.w, x2, x3);
    p0 = ex2_approx(x0);
    p1 = ex2_approx(x1);
    p2 = ex2_approx(x2);
    p3 = ex2_approx(x3);
    if (!full) {
      if (c < cmin) p0 = 0.f;
      if (c + 1 < cmin) p1 = 0.f;
      if (c + 2 < cmin) p2 = 0.f;
      if (c + 3 < cmin) p3 = 0.f;
    }
    pk[c / 2] = pack_bf16x2(p0, p1);
    pk[c / 2 + 1] = pack_bf16x2(p2, p3);
    fadd2(dp[c], dp[c + 1], D4.x, D4.y, x0, x1);
    fadd2(dp[c + 2], dp[c + 3], D4.z, D4.w, x2, x3);
    fmul2(p0, p1, x0, x1, x0, x1);
    fmul2(p2, p3, x2, x3, x2, x3);
    ds[c / 2] = pack_bf16x2(x0, x1);
    ds[c / 2 + 1] = pack_bf16x2(x2, x3);
  }
  tmem_st16_sync(lane_addr + kColS + 32 * g, pk);
  tmem_st16_sync(lane_addr + kColP + 32 * g, ds);
}

// ============================================================================ dQ
template <bool kCausal>
__global__ void __launch_bounds__(kThreads, 2)
attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_o, const float* __restrict__ lse,
                   float* __restrict__ Dbuf, const int32_t* __restrict__ cu_q,
                   const int32_t* __restrict__ cu_k, int B, int64_t T_q, int64_t T_k, int H, int QT,
                   float scale, bf16* __restrict__ dq, unsigned int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int64_t item = blockIdx.x;
  const int h = (int)(item % H);
  const int64_t rest = item / H;
  const int qi = kCausal ? QT - 1 - (int)(rest % QT) : (int)(rest % QT);
  const int b = (int)(rest / QT);
  if (b >= B) return;
  const int lo = cu_q[b], hi = cu_q[b + 1];
  const int klo = cu_k[b], khi = cu_k[b + 1];
  if (lo < 0 || hi < lo || hi > T_q || klo < 0 || khi < klo || khi > T_k) {
    if (threadIdx.x == 0 && qi == 0 && h == 0) flag_device(status, kDevCheck);
    return;
  }
  const int n = hi - lo, n_k = khi - klo;
  if (qi == QT - 1 && n > QT * kBM && threadIdx.x == 0 && h == 0) flag_device(status, kDevCheck);
  const int q0 = lo + qi * kBM;
  if (q0 >= hi) return;
  const int diag = n_k - n;                    // causal: query i sees keys j <= i + diag
  int nk = (n_k + kBN - 1) / kBN;
  if (kCausal) {
    const int last = min(qi * kBM + kBM - 1, n - 1) + diag;
    nk = last < 0 ? 0 : min(nk, last / kBN + 1);
  }
  if (nk == 0) {                               // no query here sees a key: no gradient
    zero_rows(dq, q0, min(kBM, hi - q0), H, h);
    return;
  }
  if (smem_u32(smem_raw) & 1023) {
    if (threadIdx.x == 0) flag_device(status, kDevCheck);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = smem_raw;
  Bars& bar = *reinterpret_cast<Bars*>(smem + kOffBarQ);
  volatile int* abort_flag = &bar.abort;
  if (threadIdx.x == 0) init_bars(bar);
  if (warp == 1) tmem_alloc(&bar.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();                               // the dK/dV kernel may start its set-up
  const uint32_t tmem = bar.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q); prefetch_tmap(&tm_do); prefetch_tmap(&tm_k); prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_o);
      mbar_arrive_expect_tx(&bar.big_full, 3 * kBigBytes);
      tma_load_3d(smem + kOffBig0, &tm_q, &bar.big_full, 0, h, q0);
      tma_load_3d(smem + kOffBig1, &tm_do, &bar.big_full, 0, h, q0);
      tma_load_3d(smem + kOffOQ, &tm_o, &bar.big_full, 0, h, q0);
      int issued = 0;
      for (int j = 0; j < nk; ++j) {
        const int st = j % kStages;
        if (!mbar_wait(&bar.empty[st], ((j / kStages) & 1) ^ 1, abort_flag, status)) break;
        uint8_t* ring = smem + kOffRing + st * 2 * kSmallBytes;
        mbar_arrive_expect_tx(&bar.full[st], 2 * kSmallBytes);
        tma_load_3d(ring, &tm_k, &bar.full[st], 0, h, klo + j * kBN);
        tma_load_3d(ring + kSmallBytes, &tm_v, &bar.full[st], 0, h, klo + j * kBN);
        issued = j + 1;
      }
      mbar_wait(&bar.big_full, 0, nullptr, status);
      for (int j = issued - kStages; j < issued; ++j)
        if (j >= 0) mbar_wait(&bar.full[j % kStages], (j / kStages) & 1, nullptr, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t id_kk = idesc_bf16_f32(128, kBN);
    const uint32_t id_mn = idesc_bf16_f32(128, kD) | (1u << 16);   // B MN-major
    const uint32_t q_base = smem_u32(smem + kOffBig0), do_base = smem_u32(smem + kOffBig1);
    const bool leader = elect_one();
    bool ok = mbar_wait_warp(&bar.big_full, 0, abort_flag, status);
    for (int j = 0; j < nk && ok; ++j) {
      const int st = j % kStages;
      const uint32_t kb = smem_u32(smem + kOffRing + st * 2 * kSmallBytes), vb = kb + kSmallBytes;
      if (!(ok = mbar_wait_warp(&bar.full[st], (j / kStages) & 1, abort_flag, status))) break;
      if (j > 0 && !(ok = mbar_wait_warp(&bar.p_empty, (j - 1) & 1, abort_flag, status))) break;
      tc_fence_after();
      if (leader) {
        mma_kmajor(tmem + kColS, q_base, kb, id_kk);       // S  = Q K_j^T
        mma_kmajor(tmem + kColP, do_base, vb, id_kk);      // dP = dO V_j^T
        mma_commit(&bar.s_full);
      }
      __syncwarp();
      if (!(ok = mbar_wait_warp(&bar.p_full, j & 1, abort_flag, status))) break;
      tc_fence_after();
      if (leader) {
        mma_ts_mn(tmem + kColAcc0, tmem + kColP, kb, id_mn, j > 0);   // dQ += dS K_j
        mma_commit(&bar.p_empty);
        mma_commit(&bar.empty[st]);
      }
      __syncwarp();
    }
    if (leader) mma_commit(&bar.mma_done);
    __syncwarp();
    mbar_wait_warp(&bar.mma_done, 0, nullptr, status);
  } else {
    // ------------------------------------------------------------ compute
    const int qd = warp & 3, g = (warp - 2) >> 2;
    const int r = qd * 32 + lane;
    const int64_t t = (int64_t)q0 + r;
    const uint32_t lane_addr = tmem + ((uint32_t)(qd * 32) << 16);
    const float scale_log2 = scale * kLog2e;
    // D of the row from the O and dO tiles (both threads of a row form it;
    // the first writes it for the dK/dV kernel); rows past the segment, and
    // rows that saw no key: P = 0 (lse -> +inf)
    bool ok = mbar_wait_warp(&bar.big_full, 0, abort_flag, status);
    float L = INFINITY, Dr = 0.f;
    if (ok && t < hi) {
      const float dv = row_dot64(smem + kOffOQ, smem + kOffBig1, r);
      if (g == 0) Dbuf[(int64_t)h * T_q + t] = dv;
      const float l = lse[(int64_t)h * T_q + t];
      if (l != -INFINITY) {
        L = l * kLog2e;
        Dr = dv;
      }
    }
    const float nL = -L, nD = -Dr;
    for (int j = 0; j < nk && ok; ++j) {
      if (!(ok = mbar_wait_warp(&bar.s_full, j & 1, abort_flag, status))) break;
      tc_fence_after();
      __syncwarp();
      dq_tile<kCausal>(lane_addr, g, j, n_k, qi * kBM + r, diag, scale_log2, nL, nD);
      tc_fence_before();
      mbar_arrive(&bar.p_full);
    }
    // Every compute warp reaches the named barrier, whether or not its waits
    // succeeded; the copy-out runs only if no wait of the CTA gave up.
    if (ok && mbar_wait_warp(&bar.p_empty, (nk - 1) & 1, abort_flag, status)) {
      tc_fence_after();
      __syncwarp();
      // every MMA has completed: the Q tile's buffer stages the dQ rows
      float acc[32];
      tmem_ld32(lane_addr + kColAcc0 + 32 * g, acc);
      tmem_ld_wait();
      stage_row32(smem + kOffBig0, r, g, acc, scale);
    }
    named_bar_sync(1, 256);
    if (!*abort_flag) copy_out(smem + kOffBig0, dq, q0, min(kBM, hi - q0), H, h, (int)threadIdx.x - 64);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ============================================================================ dK, dV
template <bool kCausal>
__global__ void __launch_bounds__(kThreads, 2)
attn_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                    const float* __restrict__ lse, const float* __restrict__ Dbuf, const int32_t* __restrict__ cu_q,
                    const int32_t* __restrict__ cu_k, int B, int64_t T_q, int64_t T_k, int H, int KT,
                    float scale, bf16* __restrict__ dk, bf16* __restrict__ dv, unsigned int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  WaitForPrimaryAtExit at_exit;
  const int64_t item = blockIdx.x;
  const int h = (int)(item % H);
  const int64_t rest = item / H;
  const int kt = (int)(rest % KT);             // causal: the first key tiles see the most queries
  const int b = (int)(rest / KT);
  if (b >= B) return;
  const int lo = cu_q[b], hi = cu_q[b + 1];
  const int klo = cu_k[b], khi = cu_k[b + 1];
  if (lo < 0 || hi < lo || hi > T_q || klo < 0 || khi < klo || khi > T_k) {
    if (threadIdx.x == 0 && kt == 0 && h == 0) flag_device(status, kDevCheck);
    return;
  }
  const int n = hi - lo, n_k = khi - klo;
  if (kt == KT - 1 && n_k > KT * kBM && threadIdx.x == 0 && h == 0) flag_device(status, kDevCheck);
  const int k0 = klo + kt * kBM;
  if (k0 >= khi) return;
  const int diag = n_k - n;                    // query i sees key j when i >= j - diag
  // the first query that sees any key of this tile, and the query tiles from there
  const int i_first = kCausal ? max(0, kt * kBM - diag) : 0;
  const int nq = i_first >= n ? 0 : (n - i_first + kBN - 1) / kBN;
  if (nq == 0) {                               // no query sees these keys: no gradient
    zero_rows(dk, k0, min(kBM, khi - k0), H, h);
    zero_rows(dv, k0, min(kBM, khi - k0), H, h);
    return;
  }
  if (smem_u32(smem_raw) & 1023) {
    if (threadIdx.x == 0) flag_device(status, kDevCheck);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = smem_raw;
  Bars& bar = *reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort_flag = &bar.abort;
  if (threadIdx.x == 0) init_bars(bar);
  if (warp == 1) tmem_alloc(&bar.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_k); prefetch_tmap(&tm_v); prefetch_tmap(&tm_q); prefetch_tmap(&tm_do);
      mbar_arrive_expect_tx(&bar.big_full, 2 * kBigBytes);
      tma_load_3d(smem + kOffBig0, &tm_k, &bar.big_full, 0, h, k0);
      tma_load_3d(smem + kOffBig1, &tm_v, &bar.big_full, 0, h, k0);
    }
    int issued = 0;
    for (int i = 0; i < nq; ++i) {
      const int st = i % kStages;
      if (!mbar_wait_warp(&bar.empty[st], ((i / kStages) & 1) ^ 1, abort_flag, status)) break;
      const int i0 = i_first + i * kBN;        // segment-local first query of the tile
      if (lane == 0) {
        uint8_t* ring = smem + kOffRing + st * 2 * kSmallBytes;
        mbar_arrive_expect_tx(&bar.full[st], 2 * kSmallBytes);
        tma_load_3d(ring, &tm_q, &bar.full[st], 0, h, lo + i0);
        tma_load_3d(ring + kSmallBytes, &tm_do, &bar.full[st], 0, h, lo + i0);
      }
      issued = i + 1;
      // -lse in log2 units (-inf where there is no query, or the query saw no
      // key, so that P = 0 there) and -D, one pair per query column; only the
      // compute threads wait for these, not the S^T / dP^T MMAs.  D is the dQ
      // kernel's.
      pdl_wait();
      float* aux = reinterpret_cast<float*>(smem + kOffAux + st * kAuxBytes);
      for (int c = lane; c < kBN; c += 32) {
        float nLc = -INFINITY, nDc = 0.f;
        if (i0 + c < n) {
          const int64_t t = (int64_t)lo + i0 + c;
          const float l = lse[(int64_t)h * T_q + t], dv = Dbuf[(int64_t)h * T_q + t];
          if (l != -INFINITY) {
            nLc = -l * kLog2e;
            nDc = -dv;
          }
        }
        aux[c] = nLc;
        aux[kBN + c] = nDc;
      }
      mbar_arrive(&bar.aux_full[st]);
    }
    if (lane == 0) {
      mbar_wait(&bar.big_full, 0, nullptr, status);
      for (int i = issued - kStages; i < issued; ++i)
        if (i >= 0) mbar_wait(&bar.full[i % kStages], (i / kStages) & 1, nullptr, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t id_kk = idesc_bf16_f32(128, kBN);
    const uint32_t id_mn = idesc_bf16_f32(128, kD) | (1u << 16);
    const uint32_t k_base = smem_u32(smem + kOffBig0), v_base = smem_u32(smem + kOffBig1);
    const bool leader = elect_one();
    bool ok = mbar_wait_warp(&bar.big_full, 0, abort_flag, status);
    for (int i = 0; i < nq && ok; ++i) {
      const int st = i % kStages;
      const uint32_t qb = smem_u32(smem + kOffRing + st * 2 * kSmallBytes), dob = qb + kSmallBytes;
      if (!(ok = mbar_wait_warp(&bar.full[st], (i / kStages) & 1, abort_flag, status))) break;
      if (i > 0 && !(ok = mbar_wait_warp(&bar.p_empty, (i - 1) & 1, abort_flag, status))) break;
      tc_fence_after();
      if (leader) {
        mma_kmajor(tmem + kColS, k_base, qb, id_kk);      // S^T  = K Q_i^T
        mma_kmajor(tmem + kColP, v_base, dob, id_kk);     // dP^T = V dO_i^T
        mma_commit(&bar.s_full);
      }
      __syncwarp();
      if (!(ok = mbar_wait_warp(&bar.p_full, i & 1, abort_flag, status))) break;
      tc_fence_after();
      if (leader) {
        mma_ts_mn(tmem + kColAcc0, tmem + kColS, dob, id_mn, i > 0);   // dV += P^T dO_i
        mma_ts_mn(tmem + kColAcc1, tmem + kColP, qb, id_mn, i > 0);    // dK += dS^T Q_i
        mma_commit(&bar.p_empty);
        mma_commit(&bar.empty[st]);
      }
      __syncwarp();
    }
    if (leader) mma_commit(&bar.mma_done);
    __syncwarp();
    mbar_wait_warp(&bar.mma_done, 0, nullptr, status);
  } else {
    // ------------------------------------------------------------ compute
    const int qd = warp & 3, g = (warp - 2) >> 2;
    const int r = qd * 32 + lane;
    const int jj = kt * kBM + r;               // segment-local key of this lane
    const uint32_t lane_addr = tmem + ((uint32_t)(qd * 32) << 16);
    const float scale_log2 = scale * kLog2e;
    bool ok = true;
    for (int i = 0; i < nq; ++i) {
      const int st = i % kStages;
      if (!(ok = mbar_wait_warp(&bar.s_full, i & 1, abort_flag, status))) break;
      // the aux values of this tile: acquire the producer lanes' writes
      if (!(ok = mbar_wait_warp(&bar.aux_full[st], (i / kStages) & 1, abort_flag, status))) break;
      tc_fence_after();
      __syncwarp();
      const int i0 = i_first + i * kBN;
      // causal: column c (query i0 + c) sees this key when c >= jj - diag - i0
      const int cmin = kCausal ? jj - diag - i0 - 32 * g : 0;   // relative to this half
      dkv_tile<kCausal>(lane_addr, g, cmin, reinterpret_cast<const float*>(smem + kOffAux + st * kAuxBytes) + 32 * g,
                        scale_log2);
      tc_fence_before();
      mbar_arrive(&bar.p_full);
    }
    // as in the dQ kernel: all compute warps meet at the named barrier
    if (ok && mbar_wait_warp(&bar.p_empty, (nq - 1) & 1, abort_flag, status)) {
      tc_fence_after();
      __syncwarp();
      // every MMA has completed: the K and V tiles' buffers stage dV and dK
      float acc[32];
      tmem_ld32(lane_addr + kColAcc0 + 32 * g, acc);
      tmem_ld_wait();
      stage_row32(smem + kOffBig1, r, g, acc, 1.0f);
      tmem_ld32(lane_addr + kColAcc1 + 32 * g, acc);
      tmem_ld_wait();
      stage_row32(smem + kOffBig0, r, g, acc, scale);
    }
    named_bar_sync(1, 256);
    if (!*abort_flag) {
      const int rows = min(kBM, khi - k0), ct = (int)threadIdx.x - 64;
      copy_out(smem + kOffBig1, dv, k0, rows, H, h, ct);
      copy_out(smem + kOffBig0, dk, k0, rows, H, h, ct);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}


// ============================================================================ persistent
// Persistent forms of the two kernels for short segments: two CTAs per SM
// take work items from a counter in the caller's workspace.  Lane 0 of
// the producer warp fetches the next item while the current one's ring is
// full and publishes it through a two-slot queue in shared memory; the next
// item's resident tiles are loaded once the current item's last S/dP MMA has
// completed, and its first accumulating MMA waits until the compute threads
// have read the accumulators out of TMEM ("acc free").  Output rows are
// stored directly (the resident buffers already hold the next item's tiles).
// Every barrier keeps its phase across items.

constexpr int kQueue = 2;

// One work item: segment b's 128-row tile t (keys for dK/dV, queries for dQ)
// for head h; n = streamed tiles; first = the first streamed token (segment
// local).  b < 0 ends the queue.
struct BItem {
  int b, t, h, n, first;
  int lo, hi, klo, khi;
};

struct PBars {
  uint64_t big_full, big_empty;
  uint64_t full[kStages], empty[kStages], aux_full[kStages];
  uint64_t s_full, p_full, p_empty, acc_free;
  uint64_t o_empty;                           // dQ: the compute threads have read D's rows
  uint64_t it_full[kQueue], it_empty[kQueue];
  uint64_t mma_done;
  BItem item[kQueue];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(PBars) <= 256, "barrier block");

__device__ __forceinline__ void init_pbars(PBars& bar) {
  mbar_init(&bar.big_full, 1);
  mbar_init(&bar.big_empty, 1);
  for (int i = 0; i < kStages; ++i) {
    mbar_init(&bar.full[i], 1);
    mbar_init(&bar.empty[i], 1);
    mbar_init(&bar.aux_full[i], 32);
  }
  mbar_init(&bar.s_full, 1);
  mbar_init(&bar.p_full, 256);
  mbar_init(&bar.p_empty, 1);
  mbar_init(&bar.acc_free, 256);
  mbar_init(&bar.o_empty, 256);
  for (int i = 0; i < kQueue; ++i) {
    mbar_init(&bar.it_full[i], 1);
    mbar_init(&bar.it_empty[i], 9);            // the MMA warp and eight compute warps
  }
  mbar_init(&bar.mma_done, 1);
  bar.abort = 0;
  fence_mbar_init();
  fence_async_shared();
}

// The next valid item from the counter.  kKV: items are (segment, 128-key
// tile, head) with the query tiles that see the keys; otherwise (segment,
// 128-query tile, head) with the key tiles the queries see.  Heads vary
// fastest.  An index whose tile lies past its segment's end moves the counter
// past the segment's other such indices (all invalid) in one atomicMax.
template <bool kKV, bool kCausal>
__device__ BItem fetch_bitem(unsigned int* next, unsigned int total, const int32_t* __restrict__ cu_q,
                             const int32_t* __restrict__ cu_k, int64_t T_q, int64_t T_k, int H, int NT,
                             volatile int* abort_flag, unsigned int* status) {
  BItem it;
  it.b = -1;
  while (!*abort_flag) {
    const unsigned int idx = atomicAdd(next, 1u);
    if (idx >= total) break;
    const int h = (int)(idx % (unsigned int)H);
    const unsigned int rest = idx / (unsigned int)H;
    // dQ, causal: the longest query tiles (largest index) of a segment first
    const int t = (!kKV && kCausal) ? NT - 1 - (int)(rest % (unsigned int)NT) : (int)(rest % (unsigned int)NT);
    const int b = (int)(rest / (unsigned int)NT);
    const int lo = cu_q[b], hi = cu_q[b + 1], klo = cu_k[b], khi = cu_k[b + 1];
    if (lo < 0 || hi < lo || hi > T_q || klo < 0 || khi < klo || khi > T_k) {
      if (t == 0 && h == 0) flag_device(status, kDevCheck);
      continue;
    }
    const int n = hi - lo, n_k = khi - klo;
    const int own = kKV ? n_k : n;              // rows this kind of item tiles
    const int diag = n_k - n;
    if (t == NT - 1 && own > NT * kBM && h == 0) flag_device(status, kDevCheck);
    const unsigned int seg0 = (unsigned int)b * (unsigned int)NT * (unsigned int)H;
    if (t * kBM >= own) {
      const unsigned int tiles = (unsigned int)((own + kBM - 1) / kBM);
      atomicMax(next, (!kKV && kCausal) ? seg0 + ((unsigned int)NT - tiles) * (unsigned int)H
                                        : seg0 + (unsigned int)NT * (unsigned int)H);
      continue;
    }
    int first = 0, cnt;
    if (kKV) {                                  // query tiles of 64 from the first query that sees a key here
      first = kCausal ? max(0, t * kBM - diag) : 0;
      cnt = first >= n ? 0 : (n - first + kBN - 1) / kBN;
    } else {                                    // key tiles of 64 the tile's queries see
      cnt = (n_k + kBN - 1) / kBN;
      if (kCausal) {
        const int last = min(t * kBM + kBM - 1, n - 1) + diag;
        cnt = last < 0 ? 0 : min(cnt, last / kBN + 1);
      }
    }
    it = BItem{b, t, h, cnt, first, lo, hi, klo, khi};
    break;
  }
  return it;
}

__device__ __forceinline__ bool publish_bitem(PBars& bar, int n, const BItem& it, volatile int* abort_flag,
                                              unsigned int* status) {
  const int slot = n % kQueue;
  if (!mbar_wait(&bar.it_empty[slot], ((n / kQueue) & 1) ^ 1, abort_flag, status)) return false;
  bar.item[slot] = it;
  mbar_arrive(&bar.it_full[slot]);
  return true;
}

// Item n for a consumer warp; lane 0 releases the slot once the warp holds it.
__device__ __forceinline__ bool take_bitem(PBars& bar, int n, volatile int* abort_flag, unsigned int* status,
                                           BItem& it) {
  const int slot = n % kQueue;
  if (!mbar_wait_warp(&bar.it_full[slot], (n / kQueue) & 1, abort_flag, status)) return false;
  it = bar.item[slot];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&bar.it_empty[slot]);
  return true;
}

// Broadcast lane 0's item to the warp.
__device__ __forceinline__ BItem shfl_bitem(BItem it) {
  int* f = reinterpret_cast<int*>(&it);
#pragma unroll
  for (int i = 0; i < 9; ++i) f[i] = __shfl_sync(0xffffffffu, f[i], 0);
  return it;
}

// The persistent kernels' output rows: a compute warp holds 32 rows (one per
// lane) x 32 columns of bf16, 64 bytes a row, with rows H * 128 bytes apart
// in the token-major tensor.  They leave through the warp's 2 KB buffer in
// shared memory, four lanes per row, so that each store instruction writes
// 8 rows x 64 contiguous bytes instead of 32 scattered pieces.  The 16-byte
// chunk c of row r sits at chunk c ^ ((r >> 1) & 3), which keeps the row-
// per-lane writes and the four-lanes-per-row reads free of bank conflicts.
// Rows r >= nrows (past the segment) are not written.
constexpr uint32_t kStgWarpBytes = 32 * 64;
constexpr uint32_t kSmemBytesP = kSmemBytes + 8 * kStgWarpBytes;   // the persistent dK/dV kernel
constexpr uint32_t kSmemBytesQP = kSmemBytesQ + 8 * kStgWarpBytes; // the persistent dQ kernel
// two CTAs per SM, each with the 1 KB the hardware reserves per CTA
static_assert(2 * (kSmemBytesQP + 1024) <= 228 * 1024, "two persistent dQ CTAs per SM");
__device__ __forceinline__ void staged_store_half32(uint8_t* stg, int lane, const float* v, float mul, bf16* dst0,
                                                    int64_t pitch, int nrows) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * c] * mul, v[8 * c + 1] * mul);
    w.y = pack_bf16x2(v[8 * c + 2] * mul, v[8 * c + 3] * mul);
    w.z = pack_bf16x2(v[8 * c + 4] * mul, v[8 * c + 5] * mul);
    w.w = pack_bf16x2(v[8 * c + 6] * mul, v[8 * c + 7] * mul);
    *reinterpret_cast<uint4*>(stg + lane * 64 + 16 * (c ^ ((lane >> 1) & 3))) = w;
  }
  __syncwarp();
  const int cr = lane >> 2, cc = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = cr + 8 * i;
    const uint4 w = *reinterpret_cast<const uint4*>(stg + r * 64 + 16 * (cc ^ ((r >> 1) & 3)));
    if (r < nrows) *reinterpret_cast<uint4*>(dst0 + r * pitch + 8 * cc) = w;
  }
  __syncwarp();
}
// The same rows as zeros (no buffer needed).
__device__ __forceinline__ void zero_rows32(int lane, bf16* dst0, int64_t pitch, int nrows) {
  const int cr = lane >> 2, cc = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = cr + 8 * i;
    if (r < nrows) *reinterpret_cast<uint4*>(dst0 + r * pitch + 8 * cc) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// ---------------------------------------------------------------------------- dK, dV persistent
template <bool kCausal>
__global__ void __launch_bounds__(kThreads, 2)
attn_bwd_dkv_persistent(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                        const float* __restrict__ lse, const float* __restrict__ Dbuf,
                        const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k, int B, int64_t T_q,
                        int64_t T_k, int H, int KT, float scale, bf16* __restrict__ dk, bf16* __restrict__ dv,
                        unsigned int* next, unsigned int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  WaitForPrimaryAtExit at_exit;
  if (smem_u32(smem_raw) & 1023) {
    if (threadIdx.x == 0) flag_device(status, kDevCheck);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = smem_raw;
  PBars& bar = *reinterpret_cast<PBars*>(smem + kOffBar);
  volatile int* abort_flag = &bar.abort;
  if (threadIdx.x == 0) init_pbars(bar);
  if (warp == 1) tmem_alloc(&bar.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;
  const unsigned int total = (unsigned int)B * (unsigned int)KT * (unsigned int)H;

  if (warp == 0) {
    // ------------------------------------------------------------ producer and scheduler
    // Lane 0 waits and issues the copies; the whole warp stages each query
    // tile's -lse and -D.  Lanes 1-31 learn of lane 0's progress through warp
    // shuffles, so they never poll a barrier.
    if (lane == 0) { prefetch_tmap(&tm_k); prefetch_tmap(&tm_v); prefetch_tmap(&tm_q); prefetch_tmap(&tm_do); }
    int gt = 0, kvc = 0, issued = 0;
    BItem cur;
    bool ok = true;
    if (lane == 0) {
      cur = fetch_bitem<true, kCausal>(next, total, cu_q, cu_k, T_q, T_k, H, KT, abort_flag, status);
      ok = publish_bitem(bar, 0, cur, abort_flag, status);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    cur = shfl_bitem(cur);
    for (int n = 0; ok && cur.b >= 0; ++n) {
      const int n_q = cur.hi - cur.lo;
      if (cur.n > 0) {
        if (lane == 0) {
          // K and V of this item once the previous item's last S^T / dP^T are computed
          ok = mbar_wait(&bar.big_empty, (kvc & 1) ^ 1, abort_flag, status);
          if (ok) {
            mbar_arrive_expect_tx(&bar.big_full, 2 * kBigBytes);
            tma_load_3d(smem + kOffBig0, &tm_k, &bar.big_full, 0, cur.h, cur.klo + cur.t * kBM);
            tma_load_3d(smem + kOffBig1, &tm_v, &bar.big_full, 0, cur.h, cur.klo + cur.t * kBM);
          }
        }
        if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
        ++kvc;
      }
      BItem nxt;
      nxt.b = -1;
      for (int i = 0; i <= cur.n && ok; ++i) {
        if (i == min(cur.n, kStages)) {         // the next item, while the ring is full
          if (lane == 0) {
            nxt = fetch_bitem<true, kCausal>(next, total, cu_q, cu_k, T_q, T_k, H, KT, abort_flag, status);
            ok = publish_bitem(bar, n + 1, nxt, abort_flag, status);
          }
          if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
          nxt = shfl_bitem(nxt);
        }
        if (i == cur.n) break;
        const int st = gt % kStages;
        const int i0 = cur.first + i * kBN;
        if (lane == 0) {
          ok = mbar_wait(&bar.empty[st], ((gt / kStages) & 1) ^ 1, abort_flag, status);
          if (ok) {
            uint8_t* ring = smem + kOffRing + st * 2 * kSmallBytes;
            mbar_arrive_expect_tx(&bar.full[st], 2 * kSmallBytes);
            tma_load_3d(ring, &tm_q, &bar.full[st], 0, cur.h, cur.lo + i0);
            tma_load_3d(ring + kSmallBytes, &tm_do, &bar.full[st], 0, cur.h, cur.lo + i0);
            issued = gt + 1;
          }
        }
        if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
        pdl_wait();                            // D is the dQ kernel's
        float* aux = reinterpret_cast<float*>(smem + kOffAux + st * kAuxBytes);
        for (int c = lane; c < kBN; c += 32) {
          float nLc = -INFINITY, nDc = 0.f;
          if (i0 + c < n_q) {
            const int64_t t = (int64_t)cur.lo + i0 + c;
            const float l = lse[(int64_t)cur.h * T_q + t], dvv = Dbuf[(int64_t)cur.h * T_q + t];
            if (l != -INFINITY) {
              nLc = -l * kLog2e;
              nDc = -dvv;
            }
          }
          aux[c] = nLc;
          aux[kBN + c] = nDc;
        }
        mbar_arrive(&bar.aux_full[st]);
        ++gt;
      }
      cur = nxt;
    }
    if (lane == 0) {
      if (kvc > 0) mbar_wait(&bar.big_full, (kvc - 1) & 1, nullptr, status);
      for (int j = issued - kStages; j < issued; ++j)
        if (j >= 0) mbar_wait(&bar.full[j % kStages], (j / kStages) & 1, nullptr, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t id_kk = idesc_bf16_f32(128, kBN);
    const uint32_t id_mn = idesc_bf16_f32(128, kD) | (1u << 16);
    const uint32_t k_base = smem_u32(smem + kOffBig0), v_base = smem_u32(smem + kOffBig1);
    const bool leader = elect_one();
    int gt = 0, kvc = 0;
    bool ok = true;
    BItem it;
    for (int n = 0; ok && (ok = take_bitem(bar, n, abort_flag, status, it)); ++n) {
      if (it.b < 0) break;
      if (it.n == 0) continue;
      if (!(ok = mbar_wait_warp(&bar.big_full, kvc & 1, abort_flag, status))) break;
      for (int i = 0; i < it.n && ok; ++i, ++gt) {
        const int st = gt % kStages;
        const uint32_t qb = smem_u32(smem + kOffRing + st * 2 * kSmallBytes), dob = qb + kSmallBytes;
        if (!(ok = mbar_wait_warp(&bar.full[st], (gt / kStages) & 1, abort_flag, status))) break;
        if (gt > 0 && !(ok = mbar_wait_warp(&bar.p_empty, (gt - 1) & 1, abort_flag, status))) break;
        tc_fence_after();
        if (leader) {
          mma_kmajor(tmem + kColS, k_base, qb, id_kk);      // S^T  = K Q_i^T
          mma_kmajor(tmem + kColP, v_base, dob, id_kk);     // dP^T = V dO_i^T
          mma_commit(&bar.s_full);
          if (i == it.n - 1) mma_commit(&bar.big_empty);  // K and V are free once these complete
        }
        __syncwarp();
        if (!(ok = mbar_wait_warp(&bar.p_full, gt & 1, abort_flag, status))) break;
        // the item's first accumulation overwrites dV, dK: the previous item's were read
        if (i == 0 && kvc > 0 && !(ok = mbar_wait_warp(&bar.acc_free, (kvc - 1) & 1, abort_flag, status))) break;
        tc_fence_after();
        if (leader) {
          mma_ts_mn(tmem + kColAcc0, tmem + kColS, dob, id_mn, i > 0);   // dV += P^T dO_i
          mma_ts_mn(tmem + kColAcc1, tmem + kColP, qb, id_mn, i > 0);    // dK += dS^T Q_i
          mma_commit(&bar.p_empty);
          mma_commit(&bar.empty[st]);
        }
        __syncwarp();
      }
      ++kvc;
    }
    if (leader) mma_commit(&bar.mma_done);
    __syncwarp();
    mbar_wait_warp(&bar.mma_done, 0, nullptr, status);
  } else {
    // ------------------------------------------------------------ compute
    const int qd = warp & 3, g = (warp - 2) >> 2;
    const int r = qd * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(qd * 32) << 16);
    const float scale_log2 = scale * kLog2e;
    uint8_t* stg = smem + kSmemBytes + (warp - 2) * kStgWarpBytes;   // this warp's output buffer
    int gt = 0;
    bool ok = true;
    BItem it;
    for (int n = 0; ok && (ok = take_bitem(bar, n, abort_flag, status, it)); ++n) {
      if (it.b < 0) break;
      const int n_q = it.hi - it.lo, n_k = it.khi - it.klo, diag = n_k - n_q;
      const int jj = it.t * kBM + r;             // segment-local key of this lane
      // the warp's rows: keys it.t * 128 + 32 qd + (0..31) of the segment
      const int nrows = min(32, max(0, n_k - (it.t * kBM + qd * 32)));
      const int64_t pitch = (int64_t)H * kD;
      const int64_t off0 = ((int64_t)(it.klo + it.t * kBM + qd * 32) * H + it.h) * kD + 32 * g;
      if (it.n == 0) {                           // no query sees these keys: no gradient
        zero_rows32(lane, dk + off0, pitch, nrows);
        zero_rows32(lane, dv + off0, pitch, nrows);
        continue;
      }
      for (int i = 0; i < it.n; ++i, ++gt) {
        const int st = gt % kStages;
        if (!(ok = mbar_wait_warp(&bar.s_full, gt & 1, abort_flag, status))) break;
        if (!(ok = mbar_wait_warp(&bar.aux_full[st], (gt / kStages) & 1, abort_flag, status))) break;
        tc_fence_after();
        __syncwarp();
        const int i0 = it.first + i * kBN;
        const int cmin = kCausal ? jj - diag - i0 - 32 * g : 0;
        dkv_tile<kCausal>(lane_addr, g, cmin,
                          reinterpret_cast<const float*>(smem + kOffAux + st * kAuxBytes) + 32 * g, scale_log2);
        tc_fence_before();
        mbar_arrive(&bar.p_full);
      }
      if (!ok) break;
      if (!(ok = mbar_wait_warp(&bar.p_empty, (gt - 1) & 1, abort_flag, status))) break;
      tc_fence_after();
      __syncwarp();
      float av[32], ak[32];
      tmem_ld32(lane_addr + kColAcc0 + 32 * g, av);
      tmem_ld32(lane_addr + kColAcc1 + 32 * g, ak);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&bar.acc_free);               // the next item may overwrite dV, dK
      staged_store_half32(stg, lane, av, 1.0f, dv + off0, pitch, nrows);
      staged_store_half32(stg, lane, ak, scale, dk + off0, pitch, nrows);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------- dQ persistent
template <bool kCausal>
__global__ void __launch_bounds__(kThreads, 2)
attn_bwd_dq_persistent(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o, const float* __restrict__ lse,
                       float* __restrict__ Dbuf,
                       const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k, int B, int64_t T_q,
                       int64_t T_k, int H, int QT, float scale, bf16* __restrict__ dq, unsigned int* next,
                       unsigned int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023) {
    if (threadIdx.x == 0) flag_device(status, kDevCheck);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = smem_raw;
  PBars& bar = *reinterpret_cast<PBars*>(smem + kOffBarQ);
  volatile int* abort_flag = &bar.abort;
  if (threadIdx.x == 0) init_pbars(bar);
  if (warp == 1) tmem_alloc(&bar.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_trigger();                               // the dK/dV kernel may start its set-up
  const uint32_t tmem = bar.tmem_base;
  const unsigned int total = (unsigned int)B * (unsigned int)QT * (unsigned int)H;

  if (warp == 0) {
    // ------------------------------------------------------------ producer and scheduler (lane 0)
    if (lane == 0) {
      prefetch_tmap(&tm_q); prefetch_tmap(&tm_do); prefetch_tmap(&tm_k); prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_o);
      int gt = 0, qc = 0, issued = 0;
      BItem cur = fetch_bitem<false, kCausal>(next, total, cu_q, cu_k, T_q, T_k, H, QT, abort_flag, status);
      bool ok = publish_bitem(bar, 0, cur, abort_flag, status);
      for (int n = 0; ok && cur.b >= 0; ++n) {
        if (cur.n > 0) {
          // Q, dO and O of this item once the previous item's last S / dP are
          // computed and its D has been read
          if (!(ok = mbar_wait(&bar.big_empty, (qc & 1) ^ 1, abort_flag, status))) break;
          if (!(ok = mbar_wait(&bar.o_empty, (qc & 1) ^ 1, abort_flag, status))) break;
          const int q0 = cur.lo + cur.t * kBM;
          mbar_arrive_expect_tx(&bar.big_full, 3 * kBigBytes);
          tma_load_3d(smem + kOffBig0, &tm_q, &bar.big_full, 0, cur.h, q0);
          tma_load_3d(smem + kOffBig1, &tm_do, &bar.big_full, 0, cur.h, q0);
          tma_load_3d(smem + kOffOQ, &tm_o, &bar.big_full, 0, cur.h, q0);
          ++qc;
        }
        BItem nxt;
        nxt.b = -1;
        for (int j = 0; j <= cur.n && ok; ++j) {
          if (j == min(cur.n, kStages)) {
            nxt = fetch_bitem<false, kCausal>(next, total, cu_q, cu_k, T_q, T_k, H, QT, abort_flag, status);
            if (!(ok = publish_bitem(bar, n + 1, nxt, abort_flag, status))) break;
          }
          if (j == cur.n) break;
          const int st = gt % kStages;
          if (!(ok = mbar_wait(&bar.empty[st], ((gt / kStages) & 1) ^ 1, abort_flag, status))) break;
          uint8_t* ring = smem + kOffRing + st * 2 * kSmallBytes;
          mbar_arrive_expect_tx(&bar.full[st], 2 * kSmallBytes);
          tma_load_3d(ring, &tm_k, &bar.full[st], 0, cur.h, cur.klo + j * kBN);
          tma_load_3d(ring + kSmallBytes, &tm_v, &bar.full[st], 0, cur.h, cur.klo + j * kBN);
          issued = gt + 1;
          ++gt;
        }
        cur = nxt;
      }
      if (qc > 0) mbar_wait(&bar.big_full, (qc - 1) & 1, nullptr, status);
      for (int j = issued - kStages; j < issued; ++j)
        if (j >= 0) mbar_wait(&bar.full[j % kStages], (j / kStages) & 1, nullptr, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t id_kk = idesc_bf16_f32(128, kBN);
    const uint32_t id_mn = idesc_bf16_f32(128, kD) | (1u << 16);
    const uint32_t q_base = smem_u32(smem + kOffBig0), do_base = smem_u32(smem + kOffBig1);
    const bool leader = elect_one();
    int gt = 0, qc = 0;
    bool ok = true;
    BItem it;
    for (int n = 0; ok && (ok = take_bitem(bar, n, abort_flag, status, it)); ++n) {
      if (it.b < 0) break;
      if (it.n == 0) continue;
      if (!(ok = mbar_wait_warp(&bar.big_full, qc & 1, abort_flag, status))) break;
      for (int j = 0; j < it.n && ok; ++j, ++gt) {
        const int st = gt % kStages;
        const uint32_t kb = smem_u32(smem + kOffRing + st * 2 * kSmallBytes), vb = kb + kSmallBytes;
        if (!(ok = mbar_wait_warp(&bar.full[st], (gt / kStages) & 1, abort_flag, status))) break;
        if (gt > 0 && !(ok = mbar_wait_warp(&bar.p_empty, (gt - 1) & 1, abort_flag, status))) break;
        tc_fence_after();
        if (leader) {
          mma_kmajor(tmem + kColS, q_base, kb, id_kk);       // S  = Q K_j^T
          mma_kmajor(tmem + kColP, do_base, vb, id_kk);      // dP = dO V_j^T
          mma_commit(&bar.s_full);
          if (j == it.n - 1) mma_commit(&bar.big_empty);   // Q and dO are free once these complete
        }
        __syncwarp();
        if (!(ok = mbar_wait_warp(&bar.p_full, gt & 1, abort_flag, status))) break;
        if (j == 0 && qc > 0 && !(ok = mbar_wait_warp(&bar.acc_free, (qc - 1) & 1, abort_flag, status))) break;
        tc_fence_after();
        if (leader) {
          mma_ts_mn(tmem + kColAcc0, tmem + kColP, kb, id_mn, j > 0);   // dQ += dS K_j
          mma_commit(&bar.p_empty);
          mma_commit(&bar.empty[st]);
        }
        __syncwarp();
      }
      ++qc;
    }
    if (leader) mma_commit(&bar.mma_done);
    __syncwarp();
    mbar_wait_warp(&bar.mma_done, 0, nullptr, status);
  } else {
    // ------------------------------------------------------------ compute
    const int qd = warp & 3, g = (warp - 2) >> 2;
    const int r = qd * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(qd * 32) << 16);
    const float scale_log2 = scale * kLog2e;
    uint8_t* stg = smem + kSmemBytesQ + (warp - 2) * kStgWarpBytes;  // this warp's output buffer
    int gt = 0, qc = 0;
    bool ok = true;
    BItem it;
    for (int n = 0; ok && (ok = take_bitem(bar, n, abort_flag, status, it)); ++n) {
      if (it.b < 0) break;
      const int n_q = it.hi - it.lo, n_k = it.khi - it.klo, diag = n_k - n_q;
      const int64_t t = (int64_t)it.lo + it.t * kBM + r;
      // the warp's rows: queries it.t * 128 + 32 qd + (0..31) of the segment
      const int nrows = (int)min64(32, max64(0, (int64_t)it.hi - (it.lo + it.t * kBM + qd * 32)));
      const int64_t pitch = (int64_t)H * kD;
      const int64_t off0 = ((int64_t)(it.lo + it.t * kBM + qd * 32) * H + it.h) * kD + 32 * g;
      if (it.n == 0) {                           // no query here sees a key: no gradient
        zero_rows32(lane, dq + off0, pitch, nrows);
        continue;
      }
      // D of the row from the item's O and dO tiles, as in the per-item
      // kernel, then the tiles may be reloaded as far as D is concerned;
      // rows past the segment, and rows that saw no key: P = 0 (-lse -> -inf)
      if (!(ok = mbar_wait_warp(&bar.big_full, qc & 1, abort_flag, status))) break;
      ++qc;
      float nL = -INFINITY, nD = 0.f;
      if (t < it.hi) {
        const float dvv = row_dot64(smem + kOffOQ, smem + kOffBig1, r);
        if (g == 0) Dbuf[(int64_t)it.h * T_q + t] = dvv;
        const float l = lse[(int64_t)it.h * T_q + t];
        if (l != -INFINITY) {
          nL = -l * kLog2e;
          nD = -dvv;
        }
      }
      mbar_arrive(&bar.o_empty);
      for (int j = 0; j < it.n; ++j, ++gt) {
        if (!(ok = mbar_wait_warp(&bar.s_full, gt & 1, abort_flag, status))) break;
        tc_fence_after();
        __syncwarp();
        dq_tile<kCausal>(lane_addr, g, j, n_k, it.t * kBM + r, diag, scale_log2, nL, nD);
        tc_fence_before();
        mbar_arrive(&bar.p_full);
      }
      if (!ok) break;
      if (!(ok = mbar_wait_warp(&bar.p_empty, (gt - 1) & 1, abort_flag, status))) break;
      tc_fence_after();
      __syncwarp();
      float acc[32];
      tmem_ld32(lane_addr + kColAcc0 + 32 * g, acc);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&bar.acc_free);               // the next item may overwrite dQ
      staged_store_half32(stg, lane, acc, scale, dq + off0, pitch, nrows);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

bool make_map_thd(CUtensorMap* map, const void* ptr, int64_t T, int H, uint32_t rows) {
  const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)H, (uint64_t)T};
  const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)H * kD * 2};
  const uint32_t box[3] = {(uint32_t)kD, 1, rows};
  return make_tmap_bf16(map, ptr, 3, dims, strides, box);
}

}  // namespace

bool attn_bwd_tc_supported(nt_dtype dt, int d) { return dt == NT_BF16 && d == kD; }

cudaError_t launch_attn_bwd_tc(const AttnBwdProblem& p, float* Dbuf, unsigned int* status, cudaStream_t s) {
  if (p.T_q == 0 || p.T_k == 0 || p.B == 0) return cudaErrorInvalidValue;   // the caller routes these
  CUtensorMap q128, do128, o128, k64, v64, k128, v128, q64, do64;
  if (!make_map_thd(&q128, p.q, p.T_q, p.H, kBM) || !make_map_thd(&do128, p.d_o, p.T_q, p.H, kBM) ||
      !make_map_thd(&o128, p.o, p.T_q, p.H, kBM) ||
      !make_map_thd(&k64, p.k, p.T_k, p.H, kBN) || !make_map_thd(&v64, p.v, p.T_k, p.H, kBN) ||
      !make_map_thd(&k128, p.k, p.T_k, p.H, kBM) || !make_map_thd(&v128, p.v, p.T_k, p.H, kBM) ||
      !make_map_thd(&q64, p.q, p.T_q, p.H, kBN) || !make_map_thd(&do64, p.d_o, p.T_q, p.H, kBN))
    return cudaErrorInvalidValue;
  const int QT = max(1, (p.max_len_q + kBM - 1) / kBM);
  const int KT = max(1, (p.max_len_k + kBM - 1) / kBM);
  const int64_t items_q = (int64_t)p.B * QT * p.H, items_k = (int64_t)p.B * KT * p.H;
  if (items_q > 0x7fffffffLL || items_k > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int slots = 2 * sm_count();
  cudaError_t e = cudaSuccess;
  // Persistent CTAs over a work counter where items are short (mean length
  // up to 768 tokens on the side a kernel tiles) and uneven (the longest
  // segment over 1.25 times the mean); one CTA per item otherwise, where the
  // hardware scheduler balances the work and the staged, row-contiguous
  // epilogue of the per-item kernels pays.
  // The counters are the caller's (two words of its workspace); without
  // them every kernel runs one CTA per item.
  const bool pkv = p.work && p.T_k <= (int64_t)768 * p.B && (int64_t)4 * p.max_len_k * p.B > (int64_t)5 * p.T_k;
  const bool pq = p.work && p.T_q <= (int64_t)768 * p.B && (int64_t)4 * p.max_len_q * p.B > (int64_t)5 * p.T_q;
  unsigned int* counters = p.work;
  if (pkv || pq) {
    e = cudaMemsetAsync(counters, 0, 2 * sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
  }
  // the dQ kernel forms D, which the dK/dV kernel reads
  if (pq) {
    auto kq = p.causal ? attn_bwd_dq_persistent<true> : attn_bwd_dq_persistent<false>;
    e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytesQP);
    if (e != cudaSuccess) return e;
    kq<<<(unsigned)min64(items_q, slots), kThreads, kSmemBytesQP, s>>>(q128, do128, k64, v64, o128, p.lse, Dbuf,
                                                                       p.cu_q, p.cu_k, p.B, p.T_q, p.T_k, p.H, QT,
                                                                       p.scale, (bf16*)p.dq, counters + 1, status);
  } else {
    auto kq = p.causal ? attn_bwd_dq_kernel<true> : attn_bwd_dq_kernel<false>;
    e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytesQ);
    if (e != cudaSuccess) return e;
    kq<<<(unsigned)items_q, kThreads, kSmemBytesQ, s>>>(q128, do128, k64, v64, o128, p.lse, Dbuf, p.cu_q, p.cu_k,
                                                        p.B, p.T_q, p.T_k, p.H, QT, p.scale, (bf16*)p.dq, status);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (pkv) {
    auto kkv = p.causal ? attn_bwd_dkv_persistent<true> : attn_bwd_dkv_persistent<false>;
    e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytesP);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kkv, dim3((unsigned)min64(items_k, slots)), dim3(kThreads), kSmemBytesP, s, k128, v128, q64, do64,
                   p.lse, (const float*)Dbuf, p.cu_q, p.cu_k, p.B, p.T_q, p.T_k, p.H, KT, p.scale, (bf16*)p.dk,
                   (bf16*)p.dv, counters, status);
    if (e != cudaSuccess) return e;
  } else {
    auto kkv = p.causal ? attn_bwd_dkv_kernel<true> : attn_bwd_dkv_kernel<false>;
    e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kkv, dim3((unsigned)items_k), dim3(kThreads), kSmemBytes, s, k128, v128, q64, do64, p.lse,
                   (const float*)Dbuf, p.cu_q, p.cu_k, p.B, p.T_q, p.T_k, p.H, KT, p.scale, (bf16*)p.dk,
                   (bf16*)p.dv, status);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace nt
