// Residual transition on the tcgen05 tensor cores, bf16 in / fp32 accumulate:
//     z~ = z + W2 ReLU(W1 LN(z) + b1) + b2        (one packed cell per row)
// or, with the SwiGLU update the paper measures (Eq. 1: h is a SwiGLU
// feature update; a template flag),
//     z~ = z + W2 (SiLU(W1 LN(z) + b1) * (W3 LN(z) + b3)) + b2.
// "DanLing NestedTensor" Eq. 1 second line; section 3.3 "Dense work across
// valid positions": the feature transform is a dense contraction over the
// sum N_i^2 packed rows, so it runs as a GEMM pair with the LayerNorm fused
// in front and the residual fused behind.
//
// Shape: C_z = 128, H_t = 128 * NC.  Persistent CTAs, one per SM; a tile is
// 256 packed rows handled as two 128-row sub-tiles that share every weight
// chunk (half the weight traffic of 128-row tiles).  Work goes out in units,
// round robin over the CTAs: F full tiles first, then the rows after them
// in half tiles of one 128-row sub-tile, when those fit in one wave (the
// launcher picks F); a unit's sub-tile 1 is idle in a half tile.
//
// Warp roles (14 warps):
//   warp 0        TMA producer: z tile (4 boxes of 64 x 128) into one of two
//                 input slots; weight chunks of 128 x 128 through a 3-stage
//                 ring, in the order W1(0), W2(0), W1(1), ...
//   warp 1        TMEM owner and MMA issuer (one thread).
//   warps 2-5     LayerNorm, in place on the tile in its input slot.
//   warps 6-9     epilogue of sub-tile 0; warps 10-13 of sub-tile 1: TMEM
//                 -> +b1, ReLU -> the bf16 hidden chunk written back over
//                 the columns it came from; at the end TMEM -> +b2 +
//                 residual -> bf16, staged in the tile's input slot -> TMA
//                 store.
// TMEM (512 columns): acc1[s] = GEMM1 chunk of sub-tile s at 128*s (and,
// once the epilogue has read it, the hidden chunk as bf16 pairs over its
// first columns), acc2[s] = output accumulator of sub-tile s at 256 + 128*s.
// GEMM2 takes the hidden chunk as its A operand straight from TMEM (B = the
// W2 chunk from shared memory), half by half as the epilogue writes it, so
// the hidden chunk never passes through shared memory; GEMM1 of the next
// chunk of a sub-tile waits until that sub-tile's GEMM2 has read it.  The
// shared memory this frees holds a second input slot: the next tile's z load
// and LayerNorm run while the current tile computes.  A slot is released by
// the tile's last GEMM1s and both sub-tiles' output stores.
// SwiGLU: hidden chunks are 64 units wide; a GEMM1 weight tile stacks those
// 64 rows of W1 (gate) over the same 64 rows of W3 (value), so one N = 128
// MMA leaves gate and value side by side in acc1, the epilogue writes the
// 64-wide product SiLU(gate + b1) * (value + b3) back over the gate, and
// GEMM2 contracts it with a 128 x 64 slice of W2 (K = 64).
// Every operand tile is K-major with the 128-byte swizzle that TMA writes.
//
// Fused block (a second template flag; "DanLing NestedTensor" Eq. 1 as one
// pass over the pair state): z never exists in HBM.  The LayerNorm warps
// build each tile as bf16(u[row] + v[col]) from the two projected single
// representations (fp32, L2-resident), with (row, col) of packed cell p
// found from the sample offsets; the output epilogue recomputes the
// same bf16 z for the residual; and after staging z~ for its TMA store the
// epilogue threads sum their feature column over the tile's cells, flushing
// one fp32 atomic add per pair row touched into m_acc (Eq. 4's column sum).
// HBM traffic per cell drops from 1,024 bytes (z written, read; z~
// written, read) to the 256 bytes of z~.
#include <cudaTypedefs.h>

#include "tc_ptx.cuh"

namespace nt {
namespace {

using namespace tc;

constexpr int kSubRows = 128;
constexpr int kTileRows = 2 * kSubRows;
constexpr int kCz = 128;
constexpr int kChunk = 128;
constexpr int kStages = 3;
constexpr int kThreads = 14 * 32;
constexpr uint32_t kBlockBytes = kSubRows * 128;          // one 64-column block: 16 KB
constexpr uint32_t kSubBytes = 2 * kBlockBytes;           // 128 x 128 bf16: 32 KB
constexpr uint32_t kABytes = 2 * kSubBytes;               // z / LN(z) tile: 64 KB (two slots)
constexpr uint32_t kWBytes = kChunk * kCz * 2;            // one weight chunk: 32 KB
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffW = kOffA + 2 * kABytes;
constexpr uint32_t kOffLN = kOffW + kStages * kWBytes;    // gamma, beta: 1 KB
constexpr uint32_t kOffBar = kOffLN + 2 * kCz * 4;
constexpr uint32_t kSmemBytes = kOffBar + 512 + 1024;     // + barriers + alignment slack

struct Bars {
  uint64_t z_full[2], a_full[2], a_empty[2];       // per input slot
  uint64_t g1_done[2], z2_full[2];                 // per input slot: last GEMM1s done, residual z reloaded
  uint64_t w_full[kStages], w_empty[kStages];
  uint64_t acc1_full[2], g2_done[2];               // per sub-tile
  uint64_t h_full[2][2];                           // per sub-tile, per half of the hidden chunk
  uint64_t acc2_full[2], acc2_empty[2];
  uint64_t out_ready[2];
  uint64_t colsum_done[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

// Inputs of the fused block: u, v (fp32, C_z wide), the partition's row
// splits and owners, the column offsets, and the fp32 accumulator of row sums.
struct FusedIn {
  const float* u;
  const float* v;
  const int64_t* row_start;
  const int32_t* row_sample;
  const int32_t* col_cu;
  int64_t T;
  float* m_acc;
  const int64_t* pair_off;   // B + 1 cell offsets of the samples
  const int32_t* cu;         // B + 1 row offsets
  const int32_t* col_len;    // M_i
  int B;
};

// Pair row and column single of packed cell p (< P): the sample by a binary
// search over the B cell offsets (the last one <= p, which steps past
// samples with no cells; a few steps, cached), then the row and column
// within the sample's N_i x M_i block by one division.
__device__ __forceinline__ void cell_of(const FusedIn& fz, int64_t p, int64_t& row, int64_t& vrow) {
  int lo = 0, hi = fz.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(fz.pair_off + mid) <= p) lo = mid; else hi = mid - 1;
  }
  const int64_t off = p - __ldg(fz.pair_off + lo);
  const int64_t m = __ldg(fz.col_len + lo);
  const int64_t a = off / m;
  row = __ldg(fz.cu + lo) + a;
  vrow = __ldg(fz.col_cu + lo) + (off - a * m);
}

// bf16 pairs of z = u[row] + v[col] for features [f0, f0 + 8) of cell p.
__device__ __forceinline__ uint4 fused_z8(const FusedIn& fz, int64_t row, int64_t vrow, int f0) {
  const float4 a0 = __ldg(reinterpret_cast<const float4*>(fz.u + row * kCz + f0));
  const float4 a1 = __ldg(reinterpret_cast<const float4*>(fz.u + row * kCz + f0 + 4));
  const float4 b0 = __ldg(reinterpret_cast<const float4*>(fz.v + vrow * kCz + f0));
  const float4 b1 = __ldg(reinterpret_cast<const float4*>(fz.v + vrow * kCz + f0 + 4));
  return make_uint4(pack_bf16x2(a0.x + b0.x, a0.y + b0.y), pack_bf16x2(a0.z + b0.z, a0.w + b0.w),
                    pack_bf16x2(a1.x + b1.x, a1.y + b1.y), pack_bf16x2(a1.z + b1.z, a1.w + b1.w));
}

// ReLU of a bf16 pair (max with +0 per half); rounding to bf16 keeps the
// sign, so this equals rounding ReLU(x) itself.
__device__ __forceinline__ uint32_t relu_bf16x2(uint32_t w) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(w), "r"(0u));
  return d;
}
// x * sigmoid(x) with sigmoid(x) = (1 + tanh(x / 2)) / 2 and tanh on the SFU
// (tanh.approx.f32, max relative error about 2^-11: below bf16's step).
__device__ __forceinline__ float silu_f(float x) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
  const float hx = 0.5f * x;
  return fmaf(hx, t, hx);
}
// Four consecutive fp32 bias values (zeros when there is no bias); b is
// 16-byte aligned and i a multiple of 4.
__device__ __forceinline__ float4 bias4(const float* __restrict__ b, int i) {
  return b ? __ldg(reinterpret_cast<const float4*>(b + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// First row and sub-tile count of work unit u: full tiles of 256 rows
// before F, half tiles of 128 rows after.
__device__ __forceinline__ void unit_rows(int64_t u, int64_t F, int64_t& row0, int& nsub) {
  if (u < F) {
    row0 = u * kTileRows;
    nsub = 2;
  } else {
    row0 = F * kTileRows + (u - F) * kSubRows;
    nsub = 1;
  }
}

template <bool kGLU, bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
transition_tc_kernel(const __grid_constant__ CUtensorMap tm_zin, const __grid_constant__ CUtensorMap tm_zout,
                     const __grid_constant__ CUtensorMap tm_w1, const __grid_constant__ CUtensorMap tm_w3,
                     const __grid_constant__ CUtensorMap tm_w2, const bf16* z_in, int64_t P, int H_t,
                     const float* __restrict__ gamma, const float* __restrict__ beta, float eps,
                     const float* __restrict__ b1, const float* __restrict__ b3, const float* __restrict__ b2,
                     const FusedIn fz, int64_t F, int64_t U, unsigned int* status) {
  // hidden units per chunk; GEMM2 contracts kHid per chunk
  constexpr int kHid = kGLU ? 64 : kChunk;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sA = smem + kOffA;
  uint8_t* sW = smem + kOffW;
  float* sGamma = reinterpret_cast<float*>(smem + kOffLN);
  float* sBeta = sGamma + kCz;
  Bars& bar = *reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort_flag = &bar.abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NC = H_t / kHid;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.z_full[i], 1);
      mbar_init(&bar.a_full[i], 128);
      // fused: the tile's last GEMM1s + both sub-tiles' output stores; otherwise
      // both output stores (the last GEMM1s release the slot for the residual
      // reload through g1_done, before the output)
      mbar_init(&bar.a_empty[i], kFused ? 3 : 2);
      mbar_init(&bar.g1_done[i], 1);
      mbar_init(&bar.z2_full[i], 1);
    }
    for (int i = 0; i < kStages; ++i) { mbar_init(&bar.w_full[i], 1); mbar_init(&bar.w_empty[i], 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar.acc1_full[s], 1); mbar_init(&bar.g2_done[s], 1);
      mbar_init(&bar.h_full[s][0], 128); mbar_init(&bar.h_full[s][1], 128);
      mbar_init(&bar.acc2_full[s], 1); mbar_init(&bar.acc2_empty[s], 128);
      mbar_init(&bar.out_ready[s], 128);
      mbar_init(&bar.colsum_done[s], 128);
    }
    mbar_init(&bar.mma_done, 1);
    bar.abort = 0;
    fence_mbar_init();
    fence_async_shared();
  }
  for (int i = threadIdx.x; i < kCz; i += kThreads) { sGamma[i] = gamma[i]; sBeta[i] = beta[i]; }
  if (warp == 1) tmem_alloc(&bar.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;
  // the set-up above overlaps the previous kernel's tail; z (or u and v) is
  // read, and z~ written, only after it has completed
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_zin); prefetch_tmap(&tm_w1); prefetch_tmap(&tm_w2); prefetch_tmap(&tm_zout);
      if (kGLU) prefetch_tmap(&tm_w3);
      int load_idx = 0;
      int last_j[2] = {-1, -1};                  // the last tile whose z each slot received
      int last_r[2] = {-1, -1};                  // the last tile whose residual each slot received
      // z of the unit at row zrow (zsub sub-tiles) into slot (zj & 1), completing on `bar_`
      auto load_z = [&](int64_t zrow, int zsub, int zj, uint64_t* bar_) {
        uint8_t* a = sA + (zj & 1) * kABytes;
        mbar_arrive_expect_tx(bar_, (uint32_t)zsub * kSubBytes);
        const int row0 = (int)zrow;
        for (int s = 0; s < zsub; ++s)
          for (int kb = 0; kb < 2; ++kb)
            tma_load_2d(a + s * kSubBytes + kb * kBlockBytes, &tm_zin, bar_, kb * 64, row0 + s * kSubRows);
      };
      // The residual z of tile zj comes back into its slot once the tile's
      // last GEMM1s have completed (they were the slot's last readers; GEMM2
      // takes its A operand from TMEM), so the output epilogue reads it from
      // shared memory.
      auto reload = [&](int64_t zrow, int zsub, int zj) -> bool {
        if (!mbar_wait(&bar.g1_done[zj & 1], (zj >> 1) & 1, abort_flag, status)) return false;
        load_z(zrow, zsub, zj, &bar.z2_full[zj & 1]);
        last_r[zj & 1] = zj;
        return true;
      };
      bool ok = true;
      int j = 0;
      int64_t prev_row = -1;
      int prev_sub = 0;
      for (int64_t u = blockIdx.x; u < U && ok; u += gridDim.x, ++j) {
        const int slot = j & 1;
        int64_t row0;
        int nsub;
        unit_rows(u, F, row0, nsub);
        if (!kFused) {   // the fused block builds its z tile in the LayerNorm warps
          if (!(ok = mbar_wait(&bar.a_empty[slot], ((j >> 1) & 1) ^ 1, abort_flag, status))) break;
          load_z(row0, nsub, j, &bar.z_full[slot]);
          last_j[slot] = j;
          if (prev_row >= 0 && !(ok = reload(prev_row, prev_sub, j - 1))) break;
          prev_row = row0;
          prev_sub = nsub;
        }
        // weights in consumption order: W1(c), W2(c), W1(c + 1), ...
        for (int q = 0; q < 2 * NC; ++q) {
          const bool w1 = (q & 1) == 0;
          const int c = q >> 1;
          const int stage = load_idx % kStages, round = load_idx / kStages;
          if (!(ok = mbar_wait(&bar.w_empty[stage], (round & 1) ^ 1, abort_flag, status))) break;
          uint8_t* dst = sW + stage * kWBytes;
          if (kGLU) {
            if (w1) {
              // rows 0-63: W1 (gate) rows of chunk c; rows 64-127: W3 (value) rows
              mbar_arrive_expect_tx(&bar.w_full[stage], kWBytes);
              for (int kb = 0; kb < 2; ++kb) {
                tma_load_2d(dst + kb * kBlockBytes, &tm_w1, &bar.w_full[stage], kb * 64, c * kHid);
                tma_load_2d(dst + kb * kBlockBytes + kBlockBytes / 2, &tm_w3, &bar.w_full[stage], kb * 64,
                            c * kHid);
              }
            } else {
              mbar_arrive_expect_tx(&bar.w_full[stage], kBlockBytes);    // W2[:, 64c : 64c + 64]
              tma_load_2d(dst, &tm_w2, &bar.w_full[stage], c * kHid, 0);
            }
          } else {
            mbar_arrive_expect_tx(&bar.w_full[stage], kWBytes);
            if (w1) {
              tma_load_2d(dst, &tm_w1, &bar.w_full[stage], 0, c * kChunk);
              tma_load_2d(dst + kBlockBytes, &tm_w1, &bar.w_full[stage], 64, c * kChunk);
            } else {
              tma_load_2d(dst, &tm_w2, &bar.w_full[stage], c * kChunk, 0);
              tma_load_2d(dst + kBlockBytes, &tm_w2, &bar.w_full[stage], c * kChunk + 64, 0);
            }
          }
          ++load_idx;
        }
      }
      if (ok && prev_row >= 0) reload(prev_row, prev_sub, j - 1);
      // drain: every copy this thread issued has landed before the CTA exits
      for (int sl = 0; sl < 2; ++sl) {
        if (last_j[sl] >= 0) mbar_wait(&bar.z_full[sl], (last_j[sl] >> 1) & 1, nullptr, status);
        if (last_r[sl] >= 0) mbar_wait(&bar.z2_full[sl], (last_r[sl] >> 1) & 1, nullptr, status);
      }
      for (int l = load_idx - kStages; l < load_idx; ++l)
        if (l >= 0) mbar_wait(&bar.w_full[l % kStages], (l / kStages) & 1, nullptr, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Per chunk c: GEMM1 of both sub-tiles (each once GEMM2 of chunk c - 1 on
    // that sub-tile has read the hidden chunk out of acc1), then GEMM2 of
    // both (each once the epilogue has written the hidden chunk over acc1).
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 128);
      const uint32_t w_base = smem_u32(sW);
      int load_idx = 0;
      int g2n[2] = {0, 0};                        // GEMM2s issued per sub-tile
      bool ok = true;
      int j = 0;
      auto take_w = [&](uint32_t* wsm) -> bool {
        const int stage = load_idx % kStages, round = load_idx / kStages;
        if (!mbar_wait(&bar.w_full[stage], round & 1, abort_flag, status)) return false;
        tc_fence_after();
        *wsm = w_base + stage * kWBytes;
        return true;
      };
      auto release_w = [&]() {
        mma_commit(&bar.w_empty[load_idx % kStages]);
        ++load_idx;
      };
      for (int64_t u = blockIdx.x; u < U && ok; u += gridDim.x, ++j) {
        const int slot = j & 1;
        const int nsub = u < F ? 2 : 1;
        const uint32_t a_base = smem_u32(sA + slot * kABytes);
        if (!(ok = mbar_wait(&bar.a_full[slot], (j >> 1) & 1, abort_flag, status))) break;
        tc_fence_after();
        for (int c = 0; c < NC && ok; ++c) {
          uint32_t wsm;
          if (!(ok = take_w(&wsm))) break;
          for (int s = 0; s < nsub; ++s) {
            // acc1[s] is free once the previous GEMM2 of sub-tile s has completed
            if (g2n[s] > 0 && !(ok = mbar_wait(&bar.g2_done[s], (g2n[s] - 1) & 1, abort_flag, status))) break;
            tc_fence_after();
            for (int k = 0; k < kCz / 16; ++k) {
              const uint32_t koff = (k >> 2) * kBlockBytes + (k & 3) * 32;
              mma_bf16(tmem + 128 * s, sdesc_k128(a_base + s * kSubBytes + koff), sdesc_k128(wsm + koff), idesc,
                       k > 0);
            }
            mma_commit(&bar.acc1_full[s]);
          }
          if (!ok) break;
          release_w();
          if (c == NC - 1)   // the slot's last reads by the tensor core
            mma_commit(kFused ? &bar.a_empty[slot] : &bar.g1_done[slot]);
          if (!(ok = take_w(&wsm))) break;
          const int it = j * NC + c;   // sub-tile 1 idles only in half tiles, which come last
          for (int s = 0; s < nsub; ++s) {
            if (c == 0 && !(ok = mbar_wait(&bar.acc2_empty[s], (j & 1) ^ 1, abort_flag, status))) break;
            // the hidden chunk as bf16 pairs in acc1[s] (16 hidden units = 8
            // columns), contracted half by half as the epilogue writes it
            for (int half = 0; half < 2 && ok; ++half) {
              if (!(ok = mbar_wait(&bar.h_full[s][half], it & 1, abort_flag, status))) break;
              tc_fence_after();
              for (int k = half * kHid / 32; k < (half + 1) * kHid / 32; ++k) {
                const uint32_t koff = (k >> 2) * kBlockBytes + (k & 3) * 32;
                mma_bf16_ts(tmem + 256 + 128 * s, tmem + 128 * s + 8 * k, sdesc_k128(wsm + koff), idesc,
                            (c > 0 || k > 0) ? 1u : 0u);
              }
            }
            if (!ok) break;
            mma_commit(&bar.g2_done[s]);
            ++g2n[s];
            if (c == NC - 1) mma_commit(&bar.acc2_full[s]);
          }
          if (!ok) break;
          release_w();
        }
      }
      // every MMA this thread issued has completed before TMEM is released
      mma_commit(&bar.mma_done);
      mbar_wait(&bar.mma_done, 0, nullptr, status);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ LayerNorm
    const int t = threadIdx.x - 64;   // 0..127: row t of each sub-tile
    // Without the fused prologue these warps also write each tile's output,
    // z~ = z + acc2 + b2, after the next tile's LayerNorm: the epilogue
    // warps then go straight from a tile's last hidden chunk to the next
    // tile's first.  The output is staged in the tile's own input slot (its
    // GEMM1s completed before acc2 did) for a TMA store; a slot's next
    // LayerNorm comes after its output in this order, so nothing waits on
    // itself.  Row r of acc2 is TMEM lane r: warp w reads quarter w & 3.
    const int r_out = (warp & 3) * 32 + lane;
    const uint32_t lane_out = (uint32_t)((warp & 3) * 32) << 16;
    const bool st_leader = threadIdx.x == 64;
    auto out_tile = [&](int64_t orow, int osub, int oj) -> bool {
      const int oslot = oj & 1;
#pragma unroll 1
      for (int so = 0; so < osub; ++so) {
        if (!mbar_wait_warp(&bar.acc2_full[so], oj & 1, abort_flag, status)) return false;
        tc_fence_after();
        __syncwarp();
        // the residual z is back in the slot (rows past P read as zeros); each
        // thread overwrites its own row's 16-byte chunks with the output
        uint8_t* hs = sA + oslot * kABytes + so * kSubBytes;
        if (so == 0 && !mbar_wait_warp(&bar.z2_full[oslot], (oj >> 1) & 1, abort_flag, status)) return false;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          // the group's residual first, so its shared-memory loads overlap the TMEM load
          uint32_t rw[16];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 q4 = *reinterpret_cast<const uint4*>(hs + swz128_offset(r_out, 32 * g + 8 * u, kSubRows));
            rw[4 * u] = q4.x; rw[4 * u + 1] = q4.y; rw[4 * u + 2] = q4.z; rw[4 * u + 3] = q4.w;
          }
          float v[32];
          tmem_ld32_sync(tmem + lane_out + 256 + 128 * so + 32 * g, v);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t o[4];
            const float4 bq0 = bias4(b2, 32 * g + 8 * u), bq1 = bias4(b2, 32 * g + 8 * u + 4);
            const float bb[8] = {bq0.x, bq0.y, bq0.z, bq0.w, bq1.x, bq1.y, bq1.z, bq1.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {      // (z + acc2) + b2, packed pairs
              const uint32_t zw = rw[4 * u + e];
              float y0, y1;
              fadd2(bf16lo(zw), bf16hi(zw), v[8 * u + 2 * e], v[8 * u + 2 * e + 1], y0, y1);
              fadd2(y0, y1, bb[2 * e], bb[2 * e + 1], y0, y1);
              o[e] = pack_bf16x2(y0, y1);
            }
            *reinterpret_cast<uint4*>(hs + swz128_offset(r_out, 32 * g + 8 * u, kSubRows)) =
                make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        tc_fence_before();
        mbar_arrive(&bar.acc2_empty[so]);
        fence_async_shared();
        mbar_arrive(&bar.out_ready[so]);
        const int64_t y = orow + so * kSubRows;
        if (st_leader && mbar_wait(&bar.out_ready[so], oj & 1, abort_flag, status) && y < P) {
          tma_store_2d(&tm_zout, hs, 0, (int)y);
          tma_store_2d(&tm_zout, hs + kBlockBytes, 64, (int)y);
          tma_store_commit();
        }
      }
      if (st_leader) {
        // the slot is reused once the stores have read it: two arrivals
        // (one per sub-tile of a full tile)
        tma_store_wait_read0();
        mbar_arrive(&bar.a_empty[oslot]);
        mbar_arrive(&bar.a_empty[oslot]);
      }
      __syncwarp();
      return true;
    };
    int64_t prev_row = -1;
    int prev_sub = 0;
    bool ok_out = true;
    int j = 0;
    for (int64_t u = blockIdx.x; u < U; u += gridDim.x, ++j) {
      const int slot = j & 1;
      int64_t row0;
      int nsub;
      unit_rows(u, F, row0, nsub);
      uint8_t* a = sA + slot * kABytes;
      if (kFused) {
        // the slot is free once its previous tile's GEMM1s and output stores
        // are done; then this thread writes row t of both sub-tiles:
        // z = bf16(u[row] + v[col])
        if (!mbar_wait(&bar.a_empty[slot], ((j >> 1) & 1) ^ 1, abort_flag, status)) break;
#pragma unroll 1
        for (int s = 0; s < nsub; ++s) {
          uint8_t* base = a + s * kSubBytes;
          const int64_t p = row0 + s * kSubRows + t;
          if (p < P) {
            int64_t row, vrow;
            cell_of(fz, p, row, vrow);
#pragma unroll 4
            for (int ci = 0; ci < 16; ++ci)
              *reinterpret_cast<uint4*>(base + swz128_offset(t, ci * 8, kSubRows)) = fused_z8(fz, row, vrow, ci * 8);
          } else {
#pragma unroll
            for (int ci = 0; ci < 16; ++ci)
              *reinterpret_cast<uint4*>(base + swz128_offset(t, ci * 8, kSubRows)) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      } else if (!mbar_wait(&bar.z_full[slot], (j >> 1) & 1, abort_flag, status)) {
        break;
      }
      {
        // this thread's two rows (row t of each sub-tile) side by side: two
        // independent chains, and one gamma / beta load serves both
        uint8_t* base[2] = {a, a + kSubBytes};
        float shift[2], mean[2], rstd[2];
        float s1a[2] = {0.f, 0.f}, s1b[2] = {0.f, 0.f}, s2a[2] = {0.f, 0.f}, s2b[2] = {0.f, 0.f};
#pragma unroll
        for (int s = 0; s < 2; ++s)
          shift[s] = bf16lo(*reinterpret_cast<const uint32_t*>(base[s] + swz128_offset(t, 0, kSubRows)));
#pragma unroll 4
        for (int ci = 0; ci < 16; ++ci) {
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const uint4 v = *reinterpret_cast<const uint4*>(base[s] + swz128_offset(t, ci * 8, kSubRows));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float d0, d1;
              fadd2(bf16lo(w[e]), bf16hi(w[e]), -shift[s], -shift[s], d0, d1);
              fadd2(s1a[s], s1b[s], d0, d1, s1a[s], s1b[s]);
              ffma2(d0, d1, d0, d1, s2a[s], s2b[s], s2a[s], s2b[s]);
            }
          }
        }
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const float s1 = s1a[s] + s1b[s], s2 = s2a[s] + s2b[s];
          const float m1 = s1 * (1.0f / kCz);
          mean[s] = shift[s] + m1;
          const float var = fmaxf(s2 * (1.0f / kCz) - m1 * m1, 0.f);
          rstd[s] = rsqrtf(var + eps);
        }
#pragma unroll 2
        for (int ci = 0; ci < 16; ++ci) {
          const float4 g0 = *reinterpret_cast<const float4*>(sGamma + ci * 8);
          const float4 g1 = *reinterpret_cast<const float4*>(sGamma + ci * 8 + 4);
          const float4 be0 = *reinterpret_cast<const float4*>(sBeta + ci * 8);
          const float4 be1 = *reinterpret_cast<const float4*>(sBeta + ci * 8 + 4);
          const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          const float bt[8] = {be0.x, be0.y, be0.z, be0.w, be1.x, be1.y, be1.z, be1.w};
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            uint8_t* p = base[s] + swz128_offset(t, ci * 8, kSubRows);
            const uint4 v = *reinterpret_cast<const uint4*>(p);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {   // ((x - mean) * rstd) * gamma + beta, packed pairs
              float y0, y1;
              fadd2(bf16lo(w[e]), bf16hi(w[e]), -mean[s], -mean[s], y0, y1);
              fmul2(y0, y1, rstd[s], rstd[s], y0, y1);
              ffma2(y0, y1, gg[2 * e], gg[2 * e + 1], bt[2 * e], bt[2 * e + 1], y0, y1);
              o[e] = pack_bf16x2(y0, y1);
            }
            *reinterpret_cast<uint4*>(p) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
      fence_async_shared();
      mbar_arrive(&bar.a_full[slot]);
      if (!kFused) {
        if (prev_row >= 0 && !(ok_out = out_tile(prev_row, prev_sub, j - 1))) break;
        prev_row = row0;
        prev_sub = nsub;
      }
    }
    if (!kFused) {
      if (ok_out && prev_row >= 0) out_tile(prev_row, prev_sub, j - 1);
      if (st_leader) tma_store_wait0();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int s = (warp - 6) >> 2;                 // sub-tile of this warpgroup
    const int qd = warp & 3;                       // TMEM lane quarter of this warp
    const int r = qd * 32 + lane;                  // row within the sub-tile
    const uint32_t lane_addr = (uint32_t)(qd * 32) << 16;
    const uint32_t acc1 = tmem + lane_addr + 128 * s;
    const bool leader = (warp == 6 + 4 * s) && lane == 0;
    int it = 0;
    int j = 0;
    bool ok = true;
    for (int64_t u = blockIdx.x; u < U && ok; u += gridDim.x, ++j) {
      const int slot = j & 1;
      int64_t row0;
      int nsub;
      unit_rows(u, F, row0, nsub);
      if (s >= nsub) continue;                     // sub-tile 1 of a half tile: idle
      for (int c = 0; c < NC; ++c, ++it) {
        if (!(ok = mbar_wait_warp(&bar.acc1_full[s], it & 1, abort_flag, status))) break;
        tc_fence_after();
        __syncwarp();   // tcgen05.ld is warp-collective: reconverge after the per-lane waits
        // the hidden chunk goes back over acc1 as bf16 pairs, each group into
        // columns this thread has already read
        if (kGLU) {
          // acc1 columns 0-63 hold the gate, 64-127 the value of hidden units
          // 64c .. 64c + 63: SiLU(gate + b1) * (value + b3) into columns 0-31
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            float gv[32], vv[32];
            tmem_ld32(acc1 + 32 * g, gv);
            tmem_ld32(acc1 + 64 + 32 * g, vv);
            tmem_ld_wait();
            uint32_t packed[16];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int col = c * kHid + 32 * g + 4 * q;
              const float4 bg = bias4(b1, col), bv = bias4(b3, col);
              float g4[4], v4[4];
              fadd2(gv[4 * q], gv[4 * q + 1], bg.x, bg.y, g4[0], g4[1]);
              fadd2(gv[4 * q + 2], gv[4 * q + 3], bg.z, bg.w, g4[2], g4[3]);
              fadd2(vv[4 * q], vv[4 * q + 1], bv.x, bv.y, v4[0], v4[1]);
              fadd2(vv[4 * q + 2], vv[4 * q + 3], bv.z, bv.w, v4[2], v4[3]);
#pragma unroll
              for (int e = 0; e < 2; ++e)
                packed[2 * q + e] = pack_bf16x2(silu_f(g4[2 * e]) * v4[2 * e], silu_f(g4[2 * e + 1]) * v4[2 * e + 1]);
            }
            tmem_st16_sync(acc1 + 16 * g, packed);
            tc_fence_before();
            mbar_arrive(&bar.h_full[s][g]);        // half g of the hidden chunk is in TMEM
          }
        } else if (!kFused) {
          // ReLU: the two halves, 64 columns read with one wait each
#pragma unroll 1
          for (int h2 = 0; h2 < 2; ++h2) {
            float v[64];
            tmem_ld64_sync(acc1 + 64 * h2, v);
            uint32_t packed[32];
#pragma unroll
            for (int q = 0; q < 16; ++q) {          // + b1 in packed pairs, ReLU on the bf16 pairs
              const float4 bb = bias4(b1, c * kChunk + 64 * h2 + 4 * q);
              float a0, a1, a2, a3;
              fadd2(v[4 * q], v[4 * q + 1], bb.x, bb.y, a0, a1);
              fadd2(v[4 * q + 2], v[4 * q + 3], bb.z, bb.w, a2, a3);
              packed[2 * q] = relu_bf16x2(pack_bf16x2(a0, a1));
              packed[2 * q + 1] = relu_bf16x2(pack_bf16x2(a2, a3));
            }
            tmem_st32_sync(acc1 + 32 * h2, packed);  // into columns this half has just read
            tc_fence_before();
            mbar_arrive(&bar.h_full[s][h2]);
          }
        } else {
          // ReLU in the fused block: per 32-column group (fewer live registers
          // beside the fused epilogue's)
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            float v[32];
            tmem_ld32(acc1 + 32 * g, v);
            tmem_ld_wait();
            uint32_t packed[16];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 bb = bias4(b1, c * kChunk + 32 * g + 4 * q);
              float a0, a1, a2, a3;
              fadd2(v[4 * q], v[4 * q + 1], bb.x, bb.y, a0, a1);
              fadd2(v[4 * q + 2], v[4 * q + 3], bb.z, bb.w, a2, a3);
              packed[2 * q] = relu_bf16x2(pack_bf16x2(a0, a1));
              packed[2 * q + 1] = relu_bf16x2(pack_bf16x2(a2, a3));
            }
            tmem_st16_sync(acc1 + 16 * g, packed);
            if (g & 1) {                            // groups 0-1, then 2-3: the two halves
              tc_fence_before();
              mbar_arrive(&bar.h_full[s][g >> 1]);
            }
          }
        }
      }
      if (!ok) break;
      if (!kFused) continue;                       // the LayerNorm warps write the output
      // output: z~ = z + acc2 + b2, staged in this tile's input slot (its
      // GEMM1s completed before acc2 did) for a TMA store
      if (!(ok = mbar_wait_warp(&bar.acc2_full[s], j & 1, abort_flag, status))) break;
      tc_fence_after();
      __syncwarp();
      uint8_t* hs = sA + slot * kABytes + s * kSubBytes;
      const int64_t row_g = row0 + s * kSubRows + r;
      const bool in_range = row_g < P;
      const bf16* zr = z_in + row_g * kCz;
      int64_t f_row = 0, f_vrow = 0;        // fused: the cell's pair row and column single
      if (kFused && in_range) cell_of(fz, row_g, f_row, f_vrow);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float v[32];
        tmem_ld32(tmem + lane_addr + 256 + 128 * s + 32 * g, v);
        tmem_ld_wait();
        uint32_t rw[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint4 q4 = make_uint4(0, 0, 0, 0);
          if (in_range) q4 = kFused ? fused_z8(fz, f_row, f_vrow, 32 * g + 8 * u)
                                    : *reinterpret_cast<const uint4*>(zr + 32 * g + 8 * u);
          rw[4 * u] = q4.x; rw[4 * u + 1] = q4.y; rw[4 * u + 2] = q4.z; rw[4 * u + 3] = q4.w;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t o[4];
          const float4 bq0 = bias4(b2, 32 * g + 8 * u), bq1 = bias4(b2, 32 * g + 8 * u + 4);
          const float bb[8] = {bq0.x, bq0.y, bq0.z, bq0.w, bq1.x, bq1.y, bq1.z, bq1.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {      // (z + acc2) + b2, packed pairs
            const uint32_t zw = rw[4 * u + e];
            float y0, y1;
            fadd2(bf16lo(zw), bf16hi(zw), v[8 * u + 2 * e], v[8 * u + 2 * e + 1], y0, y1);
            fadd2(y0, y1, bb[2 * e], bb[2 * e + 1], y0, y1);
            o[e] = pack_bf16x2(y0, y1);
          }
          *reinterpret_cast<uint4*>(hs + swz128_offset(r, 32 * g + 8 * u, kSubRows)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bar.acc2_empty[s]);
      fence_async_shared();
      mbar_arrive(&bar.out_ready[s]);
      const int64_t y = row0 + s * kSubRows;
      if (kFused) {
        // every thread reads the staged z~ tile: wait until it is complete
        if (!(ok = mbar_wait_warp(&bar.out_ready[s], j & 1, abort_flag, status))) break;
        if (leader && y < P) {
          tma_store_2d(&tm_zout, hs, 0, (int)y);
          tma_store_2d(&tm_zout, hs + kBlockBytes, 64, (int)y);
          tma_store_commit();
        }
        // Eq. 4's column sum: features fp and fp + 1 over half ch of the
        // sub-tile's cells (one 32-bit shared load per cell), one atomic add
        // per feature into m_acc per pair row touched.  The first cell's pair
        // row comes from the sample offsets (a few cached steps).
        const int fp = 2 * (r & 63), ch = r >> 6;
        const int cmax = y < P ? (int)min64(kSubRows, P - y) : 0;
        if (64 * ch < cmax) {
          const int c_end = min(cmax, 64 * ch + 64);
          int64_t row, vrow_unused;
          cell_of(fz, y + 64 * ch, row, vrow_unused);
          int64_t end = fz.row_start[row + 1];
          float acc0 = 0.f, acc1 = 0.f;
          for (int c = 64 * ch; c < c_end; ++c) {
            while (y + c >= end) {
              atomicAdd(fz.m_acc + row * kCz + fp, acc0);
              atomicAdd(fz.m_acc + row * kCz + fp + 1, acc1);
              acc0 = 0.f;
              acc1 = 0.f;
              ++row;
              end = fz.row_start[row + 1];
            }
            const uint32_t bits = *reinterpret_cast<const uint32_t*>(hs + swz128_offset(c, fp, kSubRows));
            acc0 += bf16lo(bits);
            acc1 += bf16hi(bits);
          }
          atomicAdd(fz.m_acc + row * kCz + fp, acc0);
          atomicAdd(fz.m_acc + row * kCz + fp + 1, acc1);
        }
        mbar_arrive(&bar.colsum_done[s]);
        if (leader) {
          // the slot is reused once the column sums and the store's reads are done
          const bool sums_done = mbar_wait(&bar.colsum_done[s], j & 1, abort_flag, status);
          if (y < P) tma_store_wait_read0();
          if (sums_done) {
            mbar_arrive(&bar.a_empty[slot]);
            if (nsub == 1) mbar_arrive(&bar.a_empty[slot]);   // for the idle sub-tile 1
          }
        }
      } else if (leader) {
        if (mbar_wait(&bar.out_ready[s], j & 1, abort_flag, status) && y < P) {
          tma_store_2d(&tm_zout, hs, 0, (int)y);
          tma_store_2d(&tm_zout, hs + kBlockBytes, 64, (int)y);
          tma_store_commit();
          tma_store_wait_read0();
        }
        mbar_arrive(&bar.a_empty[slot]);
      }
      __syncwarp();
    }
    if (kFused && leader) tma_store_wait0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 tensor map over a row-major [outer, inner] matrix, box {64, rows},
// 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t rows = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool transition_tc_supported(nt_dtype dt, int C_z, int H_t, bool glu) {
  const int unit = glu ? 64 : kChunk;
  return dt == NT_BF16 && C_z == kCz && H_t >= unit && H_t % unit == 0 && H_t <= 16384;
}

namespace {

cudaError_t launch_tc(const void* z_in, void* z_out, int64_t P, int C_z, int H_t, const float* gamma,
                      const float* beta, float eps, const void* W1, const float* b1, const void* W3,
                      const float* b3, const void* W2, const float* b2, const FusedIn* fused,
                      unsigned int* status, cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  if (P > 0x7fffffffLL - kTileRows) return cudaErrorInvalidValue;
  const bool glu = W3 != nullptr;
  if (fused) z_in = z_out;   // no z tensor: the unused input map is built over the output
  CUtensorMap m_zin, m_zout, m_w1, m_w3, m_w2;
  // SwiGLU: W1 and W3 are read as 64-row halves of a weight tile
  const uint32_t w_rows = glu ? 64 : 128;
  if (!make_map(&m_zin, z_in, C_z, (uint64_t)P) || !make_map(&m_zout, z_out, C_z, (uint64_t)P) ||
      !make_map(&m_w1, W1, C_z, H_t, w_rows) || !make_map(&m_w3, glu ? W3 : W1, C_z, H_t, w_rows) ||
      !make_map(&m_w2, W2, H_t, C_z))
    return cudaErrorInvalidValue;
  auto kern = fused ? (glu ? transition_tc_kernel<true, true> : transition_tc_kernel<false, true>)
                    : (glu ? transition_tc_kernel<true, false> : transition_tc_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  // Work units: S sub-tiles of 128 rows.  At most one sub-tile per SM: one
  // half tile per CTA.  Otherwise full tiles in whole waves of the grid and
  // the sub-tiles left in half tiles, when those fit in one more wave (the
  // slowest CTA then does one half tile more than the rest rather than one
  // full tile); else full tiles only.
  const int64_t S = (P + kSubRows - 1) / kSubRows;
  const int64_t tiles = (P + kTileRows - 1) / kTileRows;
  const int64_t sms = sm_count();
  int64_t grid, F, U;
  if (S <= sms) {
    grid = S;
    F = 0;
    U = S;
  } else {
    grid = min64(tiles, sms);
    const int64_t k = S / (2 * grid), H = S - 2 * k * grid;
    if (H <= grid) {
      F = k * grid;
      U = F + H;
    } else {
      F = tiles;
      U = tiles;
    }
  }
  const FusedIn none = {nullptr, nullptr, nullptr, nullptr, nullptr, 0, nullptr, nullptr, nullptr, nullptr, 0};
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), kSmemBytes, s, m_zin, m_zout, m_w1, m_w3, m_w2,
                    (const bf16*)z_in, P, H_t, gamma, beta, eps, b1, b3, b2, fused ? *fused : none, F, U, status);
}

}  // namespace

cudaError_t launch_transition_tc(const void* z_in, void* z_out, int64_t P, int C_z, int H_t,
                                 const float* gamma, const float* beta, float eps, const void* W1,
                                 const float* b1, const void* W3, const float* b3, const void* W2,
                                 const float* b2, unsigned int* status, cudaStream_t s) {
  return launch_tc(z_in, z_out, P, C_z, H_t, gamma, beta, eps, W1, b1, W3, b3, W2, b2, nullptr, status, s);
}

cudaError_t launch_block_fused_tc(const float* u, const float* v, const nt_partition* part, void* z_out, int C_z,
                                  int H_t, const float* gamma, const float* beta, float eps, const void* W1,
                                  const float* b1, const void* W3, const float* b3, const void* W2, const float* b2,
                                  float* m_acc, unsigned int* status, cudaStream_t s) {
  const FusedIn fz = {u,      v,        part->row_start, part->row_sample,     col_cu_of(part), part->T,
                      m_acc,  part->pair_off, part->cu_seqlens, col_lengths_of(part), part->B};
  return launch_tc(nullptr, z_out, part->P, C_z, H_t, gamma, beta, eps, W1, b1, W3, b3, W2, b2, &fz, status, s);
}

}  // namespace nt
