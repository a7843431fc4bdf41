// Variable-length attention on the tcgen05 tensor cores, bf16 in / fp32
// accumulate, head width 64 ("Variable-length attention and data packing",
// "What it is" / "How it works"): queries of segment i attend only to keys
// in [cu_i, cu_{i+1}), walked in key tiles of 128, with an online softmax.
//
// One CTA per (segment, 128-query tile, head).  The grid is sized from
// max_len (ceil(max_len / 128) query tiles per segment); CTAs whose tile
// starts past their segment's end exit at once, so no work list is needed.
// Warps: 0 = TMA producer (Q once, K and V tiles double-buffered through
// 3-D tensor maps over the token-major [T, H, d] tensors), 1 = TMEM owner
// and MMA issuer, 2-5 = softmax, one query row per thread.
//   S = Q K^T   (M=128, N=128, K=64)  -> TMEM columns [0, 128)
//   O_j = P V_j (M=128, N=64,  K=128) -> TMEM columns [128, 192); P is the
//   bf16 probability tile written by the softmax warps into shared memory
//   (K-major); V is read as an MN-major operand straight from its TMA tile.
// The running output stays in registers: O = O * exp(m_old - m_new) + O_j.
// Two CTAs fit on an SM (112 KB shared memory, 256 TMEM columns each), so
// one CTA's softmax overlaps the other's MMAs.
#include <cudaTypedefs.h>

#include "tc_ptx.cuh"

namespace nt {
namespace {

using namespace tc;

constexpr int kD = 64;
constexpr int kBQ = 128;
constexpr int kBK = 128;
constexpr int kThreads = 6 * 32;
constexpr uint32_t kTileBytes = 128 * kD * 2;     // 16 KB: 128 rows x 64 bf16
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;     // 2 stages
constexpr uint32_t kOffV = kOffK + 2 * kTileBytes; // 2 stages
constexpr uint32_t kOffP = kOffV + 2 * kTileBytes; // 128 x 128 bf16 = 32 KB
constexpr uint32_t kOffBar = kOffP + 2 * kTileBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256;   // two CTAs per SM: 2 x (112 KB + 1 KB reserved) fit
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColO = 128;

struct Bars {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full, s_empty, p_full, o_full;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

__global__ void __launch_bounds__(kThreads, 2)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const int32_t* __restrict__ cu, int B, int64_t T,
               int H, int QT, float scale_log2, bf16* __restrict__ o, float* __restrict__ lse,
               unsigned int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // (segment, query tile, head) of this CTA; heads vary fastest
  const int64_t item = blockIdx.x;
  const int h = (int)(item % H);
  const int64_t rest = item / H;
  const int qi = (int)(rest % QT);
  const int b = (int)(rest / QT);
  if (b >= B) return;
  const int lo = cu[b], hi = cu[b + 1];
  if (lo < 0 || hi < lo || hi > T) {
    if (threadIdx.x == 0 && qi == 0 && h == 0) flag_device(status, kDevCheck);
    return;
  }
  const int n = hi - lo;
  if (qi == QT - 1 && n > QT * kBQ && threadIdx.x == 0 && h == 0) flag_device(status, kDevCheck);
  const int q0 = lo + qi * kBQ;
  if (q0 >= hi) return;                       // CTA-uniform: nothing allocated yet
  const int nk = (n + kBK - 1) / kBK;

  if (smem_u32(smem_raw) & 1023) {               // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) flag_device(status, kDevCheck);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  uint8_t* sP = smem + kOffP;
  Bars& bar = *reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort_flag = &bar.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.k_full[i], 1); mbar_init(&bar.k_empty[i], 1);
      mbar_init(&bar.v_full[i], 1); mbar_init(&bar.v_empty[i], 1);
    }
    mbar_init(&bar.s_full, 1);
    mbar_init(&bar.s_empty, 128);
    mbar_init(&bar.p_full, 128);
    mbar_init(&bar.o_full, 1);
    mbar_init(&bar.mma_done, 1);
    bar.abort = 0;
    fence_mbar_init();
    fence_async_shared();
  }
  if (warp == 1) tmem_alloc(&bar.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q); prefetch_tmap(&tm_k); prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(&bar.q_full, kTileBytes);
      tma_load_3d(sQ, &tm_q, &bar.q_full, 0, h, q0);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < nk; ++j) {
        const int st = j & 1, rd = j >> 1;
        if (!mbar_wait(&bar.k_empty[st], (rd & 1) ^ 1, abort_flag, status)) break;
        mbar_arrive_expect_tx(&bar.k_full[st], kTileBytes);
        tma_load_3d(sK + st * kTileBytes, &tm_k, &bar.k_full[st], 0, h, lo + j * kBK);
        k_issued = j + 1;
        if (!mbar_wait(&bar.v_empty[st], (rd & 1) ^ 1, abort_flag, status)) break;
        mbar_arrive_expect_tx(&bar.v_full[st], kTileBytes);
        tma_load_3d(sV + st * kTileBytes, &tm_v, &bar.v_full[st], 0, h, lo + j * kBK);
        v_issued = j + 1;
      }
      // drain the copies this thread issued
      mbar_wait(&bar.q_full, 0, nullptr, status);
      for (int j = k_issued - 2; j < k_issued; ++j)
        if (j >= 0) mbar_wait(&bar.k_full[j & 1], (j >> 1) & 1, nullptr, status);
      for (int j = v_issued - 2; j < v_issued; ++j)
        if (j >= 0) mbar_wait(&bar.v_full[j & 1], (j >> 1) & 1, nullptr, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 128);
      const uint32_t id_o = idesc_bf16_f32(128, kD) | (1u << 16);   // B (= V) MN-major
      const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV), p_base = smem_u32(sP);
      bool ok = mbar_wait(&bar.q_full, 0, abort_flag, status);
      auto issue_pv = [&](int j) -> bool {
        if (!mbar_wait(&bar.p_full, j & 1, abort_flag, status)) return false;
        if (!mbar_wait(&bar.v_full[j & 1], (j >> 1) & 1, abort_flag, status)) return false;
        tc_fence_after();
        const uint32_t vb = v_base + (j & 1) * kTileBytes;
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint32_t pa = p_base + (kk >> 2) * kTileBytes + (kk & 3) * 32;
          mma_bf16(tmem + kColO, sdesc_k128(pa), sdesc_k128(vb + kk * 2048), id_o, kk > 0);
        }
        mma_commit(&bar.o_full);
        mma_commit(&bar.v_empty[j & 1]);
        return true;
      };
      for (int j = 0; j < nk && ok; ++j) {
        if (!(ok = mbar_wait(&bar.k_full[j & 1], (j >> 1) & 1, abort_flag, status))) break;
        if (j > 0 && !(ok = mbar_wait(&bar.s_empty, (j - 1) & 1, abort_flag, status))) break;
        tc_fence_after();
        const uint32_t kb = k_base + (j & 1) * kTileBytes;
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16(tmem + kColS, sdesc_k128(q_base + kk * 32), sdesc_k128(kb + kk * 32), id_s, kk > 0);
        mma_commit(&bar.s_full);
        mma_commit(&bar.k_empty[j & 1]);
        if (j > 0 && !(ok = issue_pv(j - 1))) break;
      }
      if (ok) issue_pv(nk - 1);
      mma_commit(&bar.mma_done);
      mbar_wait(&bar.mma_done, 0, nullptr, status);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int qd = warp & 3;
    const int r = qd * 32 + lane;                 // query row within the tile
    const uint32_t lane_addr = (uint32_t)(qd * 32) << 16;
    float m = -INFINITY, l = 0.f;
    float acc[kD];
#pragma unroll
    for (int c = 0; c < kD; ++c) acc[c] = 0.f;
    bool ok = true;
    for (int j = 0; j < nk; ++j) {
      if (!(ok = mbar_wait_warp(&bar.s_full, j & 1, abort_flag, status))) break;
      tc_fence_after();
      __syncwarp();
      const int kvalid = min(kBK, n - j * kBK);    // keys of this tile inside the segment
      // pass 1 over S in TMEM: the row maximum of the scaled scores
      float mx = -INFINITY;
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        float sv[32];
        tmem_ld32(tmem + lane_addr + kColS + 32 * g, sv);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (32 * g + c < kvalid) mx = fmaxf(mx, sv[c] * scale_log2);
      }
      const float m_new = fmaxf(m, mx);
      const float corr = exp2f(m - m_new);        // 0 on the first tile (m = -inf)
      if (j > 0) {
        // fold in O_{j-1} (relative to the previous max), then rescale; after
        // this wait PV_{j-1} is done, so P may be overwritten
        if (!(ok = mbar_wait_warp(&bar.o_full, (j - 1) & 1, abort_flag, status))) break;
        tc_fence_after();
        __syncwarp();
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          float ov[32];
          tmem_ld32(tmem + lane_addr + kColO + 32 * g, ov);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) acc[32 * g + c] = (acc[32 * g + c] + ov[c]) * corr;
        }
      }
      // pass 2: P = exp2(s - m_new) -> bf16 -> shared memory (K-major, two 64-key blocks)
      float rs = 0.f;
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        float sv[32];
        tmem_ld32(tmem + lane_addr + kColS + 32 * g, sv);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float p0 = (32 * g + c < kvalid) ? exp2f(sv[c] * scale_log2 - m_new) : 0.f;
          const float p1 = (32 * g + c + 1 < kvalid) ? exp2f(sv[c + 1] * scale_log2 - m_new) : 0.f;
          rs += p0 + p1;
          pk[c / 2] = pack_bf16x2(p0, p1);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4*>(sP + swz128_offset(r, 32 * g + 8 * u, 128)) =
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
      tc_fence_before();
      mbar_arrive(&bar.s_empty);
      l = l * corr + rs;
      m = m_new;
      fence_async_shared();
      mbar_arrive(&bar.p_full);
    }
    if (ok && mbar_wait_warp(&bar.o_full, (nk - 1) & 1, abort_flag, status)) {
      tc_fence_after();
      __syncwarp();
      float ov[kD];
      tmem_ld32(tmem + lane_addr + kColO, ov);
      tmem_ld32(tmem + lane_addr + kColO + 32, ov + 32);
      tmem_ld_wait();
      const int t = q0 + r;
      if (t < hi) {
        const float inv = 1.0f / l;
        bf16* op = o + ((int64_t)t * H + h) * kD;
#pragma unroll
        for (int u = 0; u < kD / 8; ++u) {
          uint4 w;
          w.x = pack_bf16x2((acc[8 * u] + ov[8 * u]) * inv, (acc[8 * u + 1] + ov[8 * u + 1]) * inv);
          w.y = pack_bf16x2((acc[8 * u + 2] + ov[8 * u + 2]) * inv, (acc[8 * u + 3] + ov[8 * u + 3]) * inv);
          w.z = pack_bf16x2((acc[8 * u + 4] + ov[8 * u + 4]) * inv, (acc[8 * u + 5] + ov[8 * u + 5]) * inv);
          w.w = pack_bf16x2((acc[8 * u + 6] + ov[8 * u + 6]) * inv, (acc[8 * u + 7] + ov[8 * u + 7]) * inv);
          *reinterpret_cast<uint4*>(op + 8 * u) = w;
        }
        if (lse) lse[(int64_t)h * T + t] = (m + log2f(l)) * 0.69314718055994531f;
      }
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

// 3-D bf16 map over a token-major [T, H, 64] tensor: box {64, 1, 128}
// (one head, 128 tokens), 128-byte swizzle.
bool make_map_thd(CUtensorMap* map, const void* ptr, int64_t T, int H) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
  cuuint32_t box[3] = {(cuuint32_t)kD, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool attn_tc_supported(nt_dtype dt, int d) { return dt == NT_BF16 && d == kD; }

cudaError_t launch_attn_tc(const void* q, const void* k, const void* v, const int32_t* cu, int32_t B, int64_t T,
                           int32_t max_len, int H, int d, float scale, void* o, float* lse,
                           unsigned int* status, cudaStream_t s) {
  if (T == 0 || B == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  if (!make_map_thd(&mq, q, T, H) || !make_map_thd(&mk, k, T, H) || !make_map_thd(&mv, v, T, H))
    return cudaErrorInvalidValue;
  const int QT = max(1, (max_len + kBQ - 1) / kBQ);
  const int64_t items = (int64_t)B * QT * H;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const float scale_log2 = scale * 1.4426950408889634f;
  attn_tc_kernel<<<(unsigned)items, kThreads, kSmemBytes, s>>>(mq, mk, mv, cu, B, T, H, QT, scale_log2, (bf16*)o,
                                                               lse, status);
  return cudaGetLastError();
}

}  // namespace nt
