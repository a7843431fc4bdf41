// Variable-length attention on the tcgen05 tensor cores, bf16 in / fp32
// accumulate, head width 64 ("Variable-length attention and data packing",
// "What it is" / "How it works"): queries of segment i attend only to keys
// in [cu_i, cu_{i+1}), walked in key tiles of 64, with an online softmax.
//
// One CTA per (segment, 128-query tile, head).  The grid is sized from
// max_len (ceil(max_len / 128) query tiles per segment); CTAs whose tile
// starts past their segment's end exit at once, so no work list is needed.
// Warps: 0 = TMA producer (K and V tiles of 64 tokens through a 3-stage ring,
// 3-D tensor maps over the token-major [T, H, d] tensors), 1 = TMEM owner and
// MMA issuer (the warp waits, one elected lane issues), 2-5 = softmax, one
// query row per thread.
//
// Every MMA takes its A operand from tensor memory, so shared memory only
// feeds the B operand (2 KB per MMA instead of 6 KB; with both operands in
// shared memory an N = 64 MMA is bound by shared-memory bandwidth):
//   Q   -> TMEM (the softmax threads load their query rows once)
//   S_j  = Q K_j^T  (M=128, N=64, K=64)  -> TMEM S (single buffer)
//   P_j  -> TMEM P[j & 1] (bf16, two per 32-bit column)
//   O   += P_j V_j   (M=128, N=64, K=64)  -> TMEM O
// The softmax threads read S_j into registers first and release the S
// buffer at once, so S_{j+1} is computed while they exponentiate S_j.  The
// running max moves only when a tile's max exceeds it by more than 8 (log2
// units), so O in TMEM is rescaled in place on those tiles only.  Full
// tiles take their exponentials two at a time on the SFU (f16x2 inputs).  Two CTAs fit on an SM (48 KB shared memory, 256 TMEM columns
// each, 224 of them used).
//
// Cross-attention takes the keys of query segment b from [cu_k[b], cu_k[b+1])
// ("DanLing NestedTensor" section 3.3: the output adopts the query
// structure).  The causal variant (a template flag) masks key j of a segment
// for query i when j > i + (n_k - n_q), the diagonal aligned to the segment's
// bottom-right corner: each CTA loads only the key tiles its last query row
// can see, tiles wholly under every row's diagonal run the unmasked path,
// and a query that sees no key gets zeros with lse = -inf.
#include "tc_ptx.cuh"

namespace nt {
namespace {

using namespace tc;

constexpr int kD = 64;
constexpr int kBQ = 128;
constexpr int kBK = 64;
constexpr int kStages = 3;
constexpr int kThreads = 6 * 32;
constexpr uint32_t kKVBytes = kBK * kD * 2;         // 8 KB
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kStages * kKVBytes;
constexpr uint32_t kOffBar = kOffV + kStages * kKVBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256;
constexpr uint32_t kTmemCols = 256;
// S at 0 (64 fp32 columns), O at 64 (64 fp32), P[b] at 128 + 32 b (64 keys as
// bf16 pairs), Q at 192 (64 features as bf16 pairs)
constexpr uint32_t kColS = 0, kColO = 64, kColP = 128, kColQ = 192;

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
  uint64_t s_full, s_free;
  uint64_t p_full[2], p_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

template <bool kCausal>
__global__ void __launch_bounds__(kThreads, 2)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const bf16* __restrict__ q, const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_k,
               int B, int64_t T, int64_t T_k, int H, int QT, float scale_log2, bf16* __restrict__ o,
               float* __restrict__ lse, unsigned int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // (segment, query tile, head) of this CTA; heads vary fastest
  const int64_t item = blockIdx.x;
  const int h = (int)(item % H);
  const int64_t rest = item / H;
  // causal: the longest query tiles (largest qi) are launched first
  const int qi = kCausal ? QT - 1 - (int)(rest % QT) : (int)(rest % QT);
  const int b = (int)(rest / QT);
  if (b >= B) return;
  const int lo = cu[b], hi = cu[b + 1];
  const int klo = cu_k[b], khi = cu_k[b + 1];
  if (lo < 0 || hi < lo || hi > T || klo < 0 || khi < klo || khi > T_k) {
    if (threadIdx.x == 0 && qi == 0 && h == 0) flag_device(status, kDevCheck);
    return;
  }
  const int n = hi - lo;                      // queries of the segment
  const int n_k = khi - klo;                  // keys of the segment
  if (qi == QT - 1 && n > QT * kBQ && threadIdx.x == 0 && h == 0) flag_device(status, kDevCheck);
  const int q0 = lo + qi * kBQ;
  if (q0 >= hi) return;                       // CTA-uniform: nothing allocated yet
  const int diag = n_k - n;                   // causal: query i sees keys j <= i + diag
  int nk = (n_k + kBK - 1) / kBK;
  if (kCausal) {
    const int last = min(qi * kBQ + kBQ - 1, n - 1) + diag;   // furthest key any row here sees
    nk = last < 0 ? 0 : min(nk, last / kBK + 1);
  }
  if (nk == 0) {
    // no row of this tile sees a key: zeros and lse = -inf, no pipeline
    const int rows = min(kBQ, hi - q0);
    for (int e = threadIdx.x; e < rows * (kD / 8); e += kThreads) {
      const int rr = e / (kD / 8), u = e % (kD / 8);
      *reinterpret_cast<uint4*>(o + ((int64_t)(q0 + rr) * H + h) * kD + 8 * u) = make_uint4(0u, 0u, 0u, 0u);
    }
    if (lse)
      for (int rr = threadIdx.x; rr < rows; rr += kThreads) lse[(int64_t)h * T + q0 + rr] = -INFINITY;
    return;
  }
  if (smem_u32(smem_raw) & 1023) {            // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) flag_device(status, kDevCheck);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Softmax threads fetch their query row now, so its global-memory latency
  // overlaps the barrier and TMEM set-up below (zeros past the segment's end).
  uint32_t qw[32];
  const int r = (warp & 3) * 32 + lane;       // query row within the tile (softmax warps)
  if (warp >= 2 && q0 + r < hi) {
    const uint4* qp = reinterpret_cast<const uint4*>(q + ((int64_t)(q0 + r) * H + h) * kD);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint4 w = __ldg(qp + u);
      qw[4 * u] = w.x; qw[4 * u + 1] = w.y; qw[4 * u + 2] = w.z; qw[4 * u + 3] = w.w;
    }
  } else {
#pragma unroll
    for (int u = 0; u < 32; ++u) qw[u] = 0u;
  }

  uint8_t* smem = smem_raw;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  Bars& bar = *reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort_flag = &bar.abort;

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 128);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar.k_full[i], 1); mbar_init(&bar.k_empty[i], 1);
      mbar_init(&bar.v_full[i], 1); mbar_init(&bar.v_empty[i], 1);
    }
    mbar_init(&bar.s_full, 1);
    mbar_init(&bar.s_free, 128);
    for (int i = 0; i < 2; ++i) { mbar_init(&bar.p_full[i], 128); mbar_init(&bar.p_empty[i], 1); }
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
      prefetch_tmap(&tm_k); prefetch_tmap(&tm_v);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < nk; ++j) {
        const int st = j % kStages, rd = j / kStages;
        if (!mbar_wait(&bar.k_empty[st], (rd & 1) ^ 1, abort_flag, status)) break;
        mbar_arrive_expect_tx(&bar.k_full[st], kKVBytes);
        tma_load_3d(sK + st * kKVBytes, &tm_k, &bar.k_full[st], 0, h, klo + j * kBK);
        k_issued = j + 1;
        if (!mbar_wait(&bar.v_empty[st], (rd & 1) ^ 1, abort_flag, status)) break;
        mbar_arrive_expect_tx(&bar.v_full[st], kKVBytes);
        tma_load_3d(sV + st * kKVBytes, &tm_v, &bar.v_full[st], 0, h, klo + j * kBK);
        v_issued = j + 1;
      }
      // drain the copies this thread issued
      for (int j = k_issued - kStages; j < k_issued; ++j)
        if (j >= 0) mbar_wait(&bar.k_full[j % kStages], (j / kStages) & 1, nullptr, status);
      for (int j = v_issued - kStages; j < v_issued; ++j)
        if (j >= 0) mbar_wait(&bar.v_full[j % kStages], (j / kStages) & 1, nullptr, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and waits; one elected lane issues.
    const uint32_t id_s = idesc_bf16_f32(128, kBK);
    const uint32_t id_o = idesc_bf16_f32(128, kD) | (1u << 16);   // B (= V) MN-major
    const uint32_t k_base = smem_u32(sK), v_base = smem_u32(sV);
    const bool leader = elect_one();
    bool ok = mbar_wait_warp(&bar.q_full, 0, abort_flag, status);
    // S_j into the single S buffer: needs K_j, and S_{j-1} read out by the softmax
    auto issue_s = [&](int j) -> bool {
      const int st = j % kStages;
      if (!mbar_wait_warp(&bar.k_full[st], (j / kStages) & 1, abort_flag, status)) return false;
      if (j > 0 && !mbar_wait_warp(&bar.s_free, (j - 1) & 1, abort_flag, status)) return false;
      tc_fence_after();
      if (leader) {
        const uint32_t kb = k_base + st * kKVBytes;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)      // 16 features = 8 packed TMEM columns of Q
          mma_bf16_ts(tmem + kColS, tmem + kColQ + 8 * kk, sdesc_k128(kb + kk * 32), id_s, kk > 0);
        mma_commit(&bar.s_full);
        mma_commit(&bar.k_empty[st]);
      }
      __syncwarp();
      return true;
    };
    if (ok) {
      tc_fence_after();
      ok = issue_s(0);
    }
    for (int j = 0; j < nk && ok; ++j) {
      if (j + 1 < nk && !(ok = issue_s(j + 1))) break;
      // P_j written (and O rescaled if needed) by the softmax
      if (!(ok = mbar_wait_warp(&bar.p_full[j & 1], (j >> 1) & 1, abort_flag, status))) break;
      const int st = j % kStages;
      if (!(ok = mbar_wait_warp(&bar.v_full[st], (j / kStages) & 1, abort_flag, status))) break;
      tc_fence_after();
      if (leader) {
        const uint32_t pt = tmem + kColP + 32 * (j & 1), vb = v_base + st * kKVBytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)    // 16 keys = 8 packed TMEM columns of P
          mma_bf16_ts(tmem + kColO, pt + 8 * kk, sdesc_k128(vb + kk * 2048), id_o, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar.p_empty[j & 1]);   // PV_j done: P[j&1] free, O holds tiles 0..j
        mma_commit(&bar.v_empty[st]);
      }
      __syncwarp();
    }
    if (leader) mma_commit(&bar.mma_done);
    __syncwarp();
    mbar_wait_warp(&bar.mma_done, 0, nullptr, status);
  } else {
    // ------------------------------------------------------------ softmax
    const int qd = warp & 3;
    const uint32_t lane_addr = (uint32_t)(qd * 32) << 16;
    // this row of Q -> TMEM
    tmem_st32_sync(tmem + lane_addr + kColQ, qw);
    tc_fence_before();
    mbar_arrive(&bar.q_full);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nk; ++j) {
      const int sb = j & 1;
      if (!(ok = mbar_wait_warp(&bar.s_full, j & 1, abort_flag, status))) break;
      tc_fence_after();
      __syncwarp();
      float sv[64];
      tmem_ld64_sync(tmem + lane_addr + kColS, sv);   // this row of S_j
      tc_fence_before();
      mbar_arrive(&bar.s_free);                      // the S buffer may take S_{j+1}
      // keys of this tile this row sees: a prefix [0, cnt) of the tile
      int cnt = min(kBK, n_k - j * kBK);
      if (kCausal) cnt = max(0, min(cnt, qi * kBQ + r + diag - j * kBK + 1));
      const bool full = kCausal ? __all_sync(0xffffffffu, cnt == kBK) : cnt == kBK;
      // row maximum of the raw scores (scale > 0)
      float mx = -INFINITY;
      if (full) {
        float pm[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) pm[u] = sv[u];
#pragma unroll
        for (int c = 8; c < 64; ++c) pm[c & 7] = fmaxf(pm[c & 7], sv[c]);
        mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])), fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < cnt) mx = fmaxf(mx, sv[c]);
      }
      // lazy running max: move it only when it grows by more than 8 (log2 units)
      const float cand = mx * scale_log2;
      float corr = 1.0f;
      const bool move = cand > m + 8.0f;
      if (move) {
        corr = ex2_approx(m - cand);              // 0 on the first tile (m = -inf)
        m = cand;
      }
      if (j > 0 && __any_sync(0xffffffffu, move)) {
        // rescale this warp's rows of O in TMEM once every earlier PV is done.
        // PV_{j-1} completes phase (j-1)>>1 of p_empty[(j-1)&1]; that barrier
        // is waited every other tile, so this wait is never two phases behind.
        if (!(ok = mbar_wait_warp(&bar.p_empty[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, status))) break;
        tc_fence_after();
        __syncwarp();
        float ov[64];
        tmem_ld64_sync(tmem + lane_addr + kColO, ov);
#pragma unroll
        for (int c = 0; c < 64; ++c) ov[c] *= corr;
        tmem_st32(tmem + lane_addr + kColO, ov);
        tmem_st32(tmem + lane_addr + kColO + 32, ov + 32);
        tmem_st_wait();
      }
      l *= corr;
      // P_j -> P[sb]; PV_{j-2} has finished reading that buffer
      if (j >= 2 && !(ok = mbar_wait_warp(&bar.p_empty[sb], ((j >> 1) & 1) ^ 1, abort_flag, status))) break;
      float rs = 0.f;
      uint32_t pk[32];
      if (full) {
        float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float x0 = fmaf(sv[c], scale_log2, -m), x1 = fmaf(sv[c + 1], scale_log2, -m);
          float p0, p1;
          ex2_f16x2(x0, x1, p0, p1);             // two exponentials per SFU instruction
          ps[(c >> 1) & 7] += p0 + p1;
          pk[c / 2] = pack_bf16x2(p0, p1);
        }
        rs = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      } else {
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float p0 = (c < cnt) ? ex2_approx(fmaf(sv[c], scale_log2, -m)) : 0.f;
          const float p1 = (c + 1 < cnt) ? ex2_approx(fmaf(sv[c + 1], scale_log2, -m)) : 0.f;
          rs += p0 + p1;
          pk[c / 2] = pack_bf16x2(p0, p1);
        }
      }
      tmem_st32_sync(tmem + lane_addr + kColP + 32 * sb, pk);
      l += rs;
      tc_fence_before();
      mbar_arrive(&bar.p_full[sb]);
    }
    if (ok && mbar_wait_warp(&bar.p_empty[(nk - 1) & 1], ((nk - 1) >> 1) & 1, abort_flag, status)) {
      tc_fence_after();
      __syncwarp();
      const int t = q0 + r;
      const float inv = l > 0.f ? 1.0f / l : 0.f;   // causal rows that see no key: zeros
      float ov[64];
      tmem_ld64_sync(tmem + lane_addr + kColO, ov);
      if (t < hi) {
        bf16* op = o + ((int64_t)t * H + h) * kD;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint4 w;
          w.x = pack_bf16x2(ov[8 * u] * inv, ov[8 * u + 1] * inv);
          w.y = pack_bf16x2(ov[8 * u + 2] * inv, ov[8 * u + 3] * inv);
          w.z = pack_bf16x2(ov[8 * u + 4] * inv, ov[8 * u + 5] * inv);
          w.w = pack_bf16x2(ov[8 * u + 6] * inv, ov[8 * u + 7] * inv);
          *reinterpret_cast<uint4*>(op + 8 * u) = w;
        }
        if (lse) lse[(int64_t)h * T + t] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
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

// 3-D map over a token-major [T, H, 64] tensor: box {64, 1, rows} (one head,
// `rows` tokens), 128-byte swizzle.
bool make_map_thd(CUtensorMap* map, const void* ptr, int64_t T, int H, uint32_t rows) {
  const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)H, (uint64_t)T};
  const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)H * kD * 2};
  const uint32_t box[3] = {(uint32_t)kD, 1, rows};
  return make_tmap_bf16(map, ptr, 3, dims, strides, box);
}

}  // namespace

bool attn_tc_supported(nt_dtype dt, int d) { return dt == NT_BF16 && d == kD; }

cudaError_t launch_attn_tc(const AttnProblem& p, unsigned int* status, cudaStream_t s) {
  if (p.T_q == 0 || p.B == 0) return cudaSuccess;
  if (p.T_k == 0) return cudaErrorInvalidValue;   // no key tensor to map; the caller routes this case
  CUtensorMap mk, mv;
  if (!make_map_thd(&mk, p.k, p.T_k, p.H, kBK) || !make_map_thd(&mv, p.v, p.T_k, p.H, kBK))
    return cudaErrorInvalidValue;
  const int QT = max(1, (p.max_len_q + kBQ - 1) / kBQ);
  const int64_t items = (int64_t)p.B * QT * p.H;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  auto kern = p.causal ? attn_tc_kernel<true> : attn_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const float scale_log2 = p.scale * 1.4426950408889634f;
  kern<<<(unsigned)items, kThreads, kSmemBytes, s>>>(mk, mv, (const bf16*)p.q, p.cu_q, p.cu_k, p.B, p.T_q, p.T_k,
                                                     p.H, QT, scale_log2, (bf16*)p.o, p.lse, status);
  return cudaGetLastError();
}

}  // namespace nt
