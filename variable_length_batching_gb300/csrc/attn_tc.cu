// Variable-length attention on the tcgen05 tensor cores, bf16 in / fp32
// accumulate, head width 64 ("Variable-length attention and data packing",
// "What it is" / "How it works"): queries of segment i attend only to keys
// in [cu_i, cu_{i+1}), walked in key tiles of 64, with an online softmax.
//
// A work item is (segment, 128-query tile, head).  Two schedules share the
// tile code below:
//   - one CTA per item (attn_item_kernel): the grid is sized from max_len;
//     CTAs whose tile starts past their segment's end exit at once.  With
//     long segments each CTA walks many key tiles and its set-up, Q load and
//     epilogue cost little.
//   - persistent CTAs (attn_persistent_kernel), four per SM, taking items
//     from a counter in the caller's workspace: the producer warp fetches
//     the next item while the current one's K/V ring is full, loads its Q as
//     soon as the current item's last S has been computed, and the next
//     item's first S is issued while the softmax warps write out the current
//     item's O.  With short segments this hides the per-item cost that
//     dominates one CTA per item.
//   The launcher picks by the mean segment length (and takes one CTA per
//   item when the caller gives no workspace).
//
// Warps: 0 = TMA producer (Q per item; K and V tiles of 64 tokens through a
// 2-stage ring, 3-D tensor maps over the token-major [T, H, d] tensors),
// 1 = TMEM owner and MMA issuer (the warp waits, one elected lane issues),
// 2-5 = softmax, one query row per thread.
//
// Four CTAs share an SM, so while one waits on its chain of hand-offs the
// others compute: each holds 128 TMEM columns and 48 KB of shared memory.
//   S_j  = Q K_j^T  (M=128, N=64, K=64)  -> TMEM S (64 columns)
//   P_j  -> written by the softmax threads over S's first 32 columns (bf16
//           pairs), after they have read S_j
//   O   += P_j V_j   (M=128, N=64, K=64; A from TMEM)  -> TMEM O
// S_{j+1} overwrites S/P, so it is issued once PV_j has completed.  The
// softmax reads S in two passes of 32 columns (row max, then exponentials)
// to stay within the registers four CTAs leave.  The running max moves only
// when a tile's max exceeds it by more than 8 (log2 units), so O in TMEM is
// rescaled in place on those tiles only; PV_{j-1} has completed by then
// (S_j was issued after it).  The softmax is bound by instruction issue, so
// full tiles use packed fp32 pairs for the exponent FMA and the row sums, a
// three-input max for the row maximum, and one SFU exponential per element.
//
// Cross-attention takes the keys of query segment b from [cu_k[b], cu_k[b+1])
// ("DanLing NestedTensor" section 3.3: the output adopts the query
// structure).  The causal variant (a template flag) masks key j of a segment
// for query i when j > i + (n_k - n_q), the diagonal aligned to the segment's
// bottom-right corner: each item loads only the key tiles its last query row
// can see, tiles wholly under every row's diagonal run the unmasked path,
// and a query that sees no key gets zeros with lse = -inf.
#include "tc_ptx.cuh"

namespace nt {
namespace {

using namespace tc;

constexpr int kD = 64;
constexpr int kBQ = 128;
constexpr int kBK = 64;
constexpr int kStages = 2;
constexpr int kThreads = 6 * 32;
constexpr uint32_t kQBytes = kBQ * kD * 2;          // 16 KB
constexpr uint32_t kKVBytes = kBK * kD * 2;         // 8 KB
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffV = kOffK + kStages * kKVBytes;
constexpr uint32_t kOffBar = kOffV + kStages * kKVBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256;
constexpr uint32_t kTmemCols = 128;
// S at 0 (64 fp32 columns; P over its first 32 as bf16 pairs), O at 64
constexpr uint32_t kColS = 0, kColO = 64;

constexpr int kQueue = 2;

// One work item: segment b's query tile qi for head h, with its offsets and
// key-tile count.  b < 0 ends the queue.
struct Item {
  int b, qi, h, nk;
  int lo, hi, klo, khi;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
  uint64_t s_full, p_full, p_empty;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct PBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
  uint64_t s_full, p_full, p_empty, o_free;
  uint64_t it_full[kQueue], it_empty[kQueue];
  uint64_t mma_done;
  Item item[kQueue];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(PBars) <= 256, "barrier block");

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// One key tile of the online softmax for this thread's query row: S_j is in
// TMEM at s_addr (64 fp32 columns), O at o_addr.  Writes P_j as bf16 pairs
// over S_j's first 32 columns and updates the running max m (log2 units)
// and the row sum l; rescales this warp's rows of O in place when m moves
// (the caller guarantees PV_{j-1} has completed).  row_q is the row's query
// index within its segment, diag = n_k - n_q.
template <bool kCausal>
__device__ __forceinline__ void softmax_tile(uint32_t s_addr, uint32_t o_addr, int j, int n_k, int row_q, int diag,
                                             float scale_log2, float& m, float& l) {
  // keys of this tile this row sees: a prefix [0, cnt) of the tile
  int cnt = min(kBK, n_k - j * kBK);
  if (kCausal) cnt = max(0, min(cnt, row_q + diag - j * kBK + 1));
  const bool full = kCausal ? __all_sync(0xffffffffu, cnt == kBK) : cnt == kBK;
  // pass 1: row maximum of the raw scores (scale > 0)
  float mx = -INFINITY;
#pragma unroll 1
  for (int g = 0; g < 2; ++g) {
    float sv[32];
    tmem_ld32(s_addr + 32 * g, sv);
    tmem_ld_wait();
    if (full) {
      float pm[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
      for (int c = 4; c < 28; c += 8) {
        pm[0] = max3f(pm[0], sv[c], sv[c + 1]);
        pm[1] = max3f(pm[1], sv[c + 2], sv[c + 3]);
        pm[2] = max3f(pm[2], sv[c + 4], sv[c + 5]);
        pm[3] = max3f(pm[3], sv[c + 6], sv[c + 7]);
      }
      pm[0] = max3f(pm[0], sv[28], sv[29]);
      pm[1] = max3f(pm[1], sv[30], sv[31]);
      mx = max3f(mx, max3f(pm[0], pm[1], pm[2]), pm[3]);
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (32 * g + c < cnt) mx = fmaxf(mx, sv[c]);
    }
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
    // rescale this warp's rows of O in TMEM: PV_{j-1} completed before S_j was issued
#pragma unroll 1
    for (int g = 0; g < 2; ++g) {
      float ov[32];
      tmem_ld32(o_addr + 32 * g, ov);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 32; ++c) ov[c] *= corr;
      tmem_st32(o_addr + 32 * g, ov);
    }
    tmem_st_wait();
  }
  l *= corr;
  // pass 2: P_j over S_j's first 32 columns; group g's 16 packed words go
  // to columns [16 g, 16 g + 16), whose scores this thread has already read
  float rs = 0.f;
#pragma unroll 1
  for (int g = 0; g < 2; ++g) {
    float sv[32];
    tmem_ld32(s_addr + 32 * g, sv);
    tmem_ld_wait();
    uint32_t pk[16];
    if (full) {
      // exponents and row sums in packed fp32 pairs (two pairs of
      // accumulators); exponentials on the SFU
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float x0, x1, p0, p1;
        ffma2(sv[c], sv[c + 1], scale_log2, scale_log2, -m, -m, x0, x1);
        p0 = ex2_approx(x0);
        p1 = ex2_approx(x1);
        if ((c >> 1) & 1) fadd2(ps[2], ps[3], p0, p1, ps[2], ps[3]);
        else fadd2(ps[0], ps[1], p0, p1, ps[0], ps[1]);
        pk[c / 2] = pack_bf16x2(p0, p1);
      }
      rs += (ps[0] + ps[1]) + (ps[2] + ps[3]);
    } else {
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        const float p0 = (32 * g + c < cnt) ? ex2_approx(fmaf(sv[c], scale_log2, -m)) : 0.f;
        const float p1 = (32 * g + c + 1 < cnt) ? ex2_approx(fmaf(sv[c + 1], scale_log2, -m)) : 0.f;
        rs += p0 + p1;
        pk[c / 2] = pack_bf16x2(p0, p1);
      }
    }
    tmem_st16_sync(s_addr + 16 * g, pk);
  }
  l += rs;
}

template <bool kCausal>
__global__ void __launch_bounds__(kThreads, 4)
attn_item_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_k,
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

  uint8_t* smem = smem_raw;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  Bars& bar = *reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort_flag = &bar.abort;

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar.k_full[i], 1); mbar_init(&bar.k_empty[i], 1);
      mbar_init(&bar.v_full[i], 1); mbar_init(&bar.v_empty[i], 1);
    }
    mbar_init(&bar.s_full, 1);
    mbar_init(&bar.p_full, 128);
    mbar_init(&bar.p_empty, 1);
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
      mbar_arrive_expect_tx(&bar.q_full, kQBytes);
      tma_load_3d(sQ, &tm_q, &bar.q_full, 0, h, q0);
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
      mbar_wait(&bar.q_full, 0, nullptr, status);
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
    const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV);
    const bool leader = elect_one();
    bool ok = mbar_wait_warp(&bar.q_full, 0, abort_flag, status);
    for (int j = 0; j < nk && ok; ++j) {
      // S_j: needs K_j, and S/P free (PV_{j-1} complete)
      const int st = j % kStages;
      if (!(ok = mbar_wait_warp(&bar.k_full[st], (j / kStages) & 1, abort_flag, status))) break;
      if (j > 0 && !(ok = mbar_wait_warp(&bar.p_empty, (j - 1) & 1, abort_flag, status))) break;
      tc_fence_after();
      if (leader) {
        const uint32_t kb = k_base + st * kKVBytes;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16(tmem + kColS, sdesc_k128(q_base + kk * 32), sdesc_k128(kb + kk * 32), id_s, kk > 0);
        mma_commit(&bar.s_full);
        mma_commit(&bar.k_empty[st]);
      }
      __syncwarp();
      // PV_j once the softmax has written P_j over S_j
      if (!(ok = mbar_wait_warp(&bar.p_full, j & 1, abort_flag, status))) break;
      if (!(ok = mbar_wait_warp(&bar.v_full[st], (j / kStages) & 1, abort_flag, status))) break;
      tc_fence_after();
      if (leader) {
        const uint32_t vb = v_base + st * kKVBytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)    // 16 keys = 8 packed TMEM columns of P
          mma_bf16_ts(tmem + kColO, tmem + kColS + 8 * kk, sdesc_k128(vb + kk * 2048), id_o,
                      (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar.p_empty);          // PV_j done: S/P free, O holds tiles 0..j
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
    const int r = qd * 32 + lane;                 // query row within the tile
    const uint32_t lane_addr = (uint32_t)(qd * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + kColS;
    // a warp whose 32 rows all lie past the segment's end keeps the
    // hand-offs but skips the arithmetic: its rows are never copied out
    const bool live = __any_sync(0xffffffffu, q0 + r < hi);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nk; ++j) {
      if (!(ok = mbar_wait_warp(&bar.s_full, j & 1, abort_flag, status))) break;
      tc_fence_after();
      __syncwarp();
      if (live)
        softmax_tile<kCausal>(s_addr, tmem + lane_addr + kColO, j, n_k, qi * kBQ + r, diag, scale_log2, m, l);
      tc_fence_before();
      mbar_arrive(&bar.p_full);
    }
    // The output rows leave through shared memory (the Q tile's buffer, free
    // once every MMA has completed): each thread stages its row, 16-byte
    // chunks XOR-swizzled by row, then the 128 softmax threads copy whole
    // rows out, eight per row.  Every softmax warp reaches the named barrier
    // whether or not its waits succeeded; the copy-out runs only if no wait
    // of the CTA gave up.
    if (ok && mbar_wait_warp(&bar.p_empty, (nk - 1) & 1, abort_flag, status)) {
      tc_fence_after();
      __syncwarp();
      const int t = q0 + r;
      const float inv = l > 0.f ? 1.0f / l : 0.f;   // causal rows that see no key: zeros
#pragma unroll 1
      for (int g = 0; g < 2 && live; ++g) {
        float ov[32];
        tmem_ld32(tmem + lane_addr + kColO + 32 * g, ov);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint4 w;
          w.x = pack_bf16x2(ov[8 * u] * inv, ov[8 * u + 1] * inv);
          w.y = pack_bf16x2(ov[8 * u + 2] * inv, ov[8 * u + 3] * inv);
          w.z = pack_bf16x2(ov[8 * u + 4] * inv, ov[8 * u + 5] * inv);
          w.w = pack_bf16x2(ov[8 * u + 6] * inv, ov[8 * u + 7] * inv);
          *reinterpret_cast<uint4*>(sQ + r * 128 + (((4 * g + u) ^ (r & 7)) << 4)) = w;
        }
      }
      if (t < hi && lse) lse[(int64_t)h * T + t] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
    named_bar_sync(1, 128);
    if (!*abort_flag) {
      const int rows = min(kBQ, hi - q0);
      for (int e = (int)threadIdx.x - 64; e < rows * 8; e += 128) {
        const int rr = e >> 3, c = e & 7;
        const uint4 w = *reinterpret_cast<const uint4*>(sQ + rr * 128 + ((c ^ (rr & 7)) << 4));
        *reinterpret_cast<uint4*>(o + ((int64_t)(q0 + rr) * H + h) * kD + 8 * c) = w;
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

// Item `n` of this CTA from queue slot n % kQueue; every consumer warp
// releases the slot (lane 0 arrives) once all its lanes hold the item.
__device__ __forceinline__ bool take_item(PBars& bar, int n, volatile int* abort_flag, unsigned int* status,
                                          Item& it) {
  const int slot = n % kQueue;
  if (!mbar_wait_warp(&bar.it_full[slot], (n / kQueue) & 1, abort_flag, status)) return false;
  it = bar.item[slot];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&bar.it_empty[slot]);
  return true;
}

// The next valid work item of the launch from the work counter (b = -1
// once the counter has passed every (segment, query tile, head)).  Indices
// run over (segment, query tile, head), heads fastest; an index whose query
// tile lies past its segment's end is skipped, and the counter is moved past
// every other such index of that segment at once (they are all invalid,
// whoever would take them), so a batch of short segments under a long
// max_len costs one atomic per segment rather than one per empty tile.
template <bool kCausal>
__device__ Item fetch_item(unsigned int* next, unsigned int total, const int32_t* __restrict__ cu,
                           const int32_t* __restrict__ cu_k, int64_t T, int64_t T_k, int H, int QT,
                           volatile int* abort_flag, unsigned int* status) {
  Item it;
  it.b = -1;
  while (!*abort_flag) {
    const unsigned int idx = atomicAdd(next, 1u);
    if (idx >= total) break;
    const int h = (int)(idx % (unsigned int)H);
    const unsigned int rest = idx / (unsigned int)H;
    // causal: the longest query tiles (largest qi) of a segment first
    const int qi = kCausal ? QT - 1 - (int)(rest % (unsigned int)QT) : (int)(rest % (unsigned int)QT);
    const int b = (int)(rest / (unsigned int)QT);
    const int lo = cu[b], hi = cu[b + 1], klo = cu_k[b], khi = cu_k[b + 1];
    if (lo < 0 || hi < lo || hi > T || klo < 0 || khi < klo || khi > T_k) {
      if (qi == 0 && h == 0) flag_device(status, kDevCheck);
      continue;
    }
    const int n_q = hi - lo, n_k = khi - klo;
    if (qi == QT - 1 && n_q > QT * kBQ && h == 0) flag_device(status, kDevCheck);
    if (lo + qi * kBQ >= hi) {                // no such query tile in this segment
      const unsigned int qt = (unsigned int)((n_q + kBQ - 1) / kBQ);   // the segment's query tiles
      const unsigned int seg0 = (unsigned int)b * (unsigned int)QT * (unsigned int)H;
      // non-causal: the invalid tiles are the segment's last QT - qt; causal
      // (tiles in reverse): its first QT - qt
      atomicMax(next, kCausal ? seg0 + ((unsigned int)QT - qt) * (unsigned int)H
                              : seg0 + (unsigned int)QT * (unsigned int)H);
      continue;
    }
    int nk = (n_k + kBK - 1) / kBK;
    if (kCausal) {
      const int last = min(qi * kBQ + kBQ - 1, n_q - 1) + (n_k - n_q);   // furthest key any row sees
      nk = last < 0 ? 0 : min(nk, last / kBK + 1);
    }
    it = Item{b, qi, h, nk, lo, hi, klo, khi};
    break;
  }
  return it;
}

// Publishes item n into queue slot n % kQueue once every consumer warp has
// taken the item that used the slot before.
__device__ __forceinline__ bool publish_item(PBars& bar, int n, const Item& it, volatile int* abort_flag,
                                             unsigned int* status) {
  const int slot = n % kQueue;
  if (!mbar_wait(&bar.it_empty[slot], ((n / kQueue) & 1) ^ 1, abort_flag, status)) return false;
  bar.item[slot] = it;
  mbar_arrive(&bar.it_full[slot]);
  return true;
}

template <bool kCausal>
__global__ void __launch_bounds__(kThreads, 4)
attn_persistent_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const int32_t* __restrict__ cu,
                       const int32_t* __restrict__ cu_k, int B, int64_t T, int64_t T_k, int H, int QT,
                       float scale_log2, bf16* __restrict__ o, float* __restrict__ lse, unsigned int* next,
                       unsigned int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023) {            // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) flag_device(status, kDevCheck);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = smem_raw;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  PBars& bar = *reinterpret_cast<PBars*>(smem + kOffBar);
  volatile int* abort_flag = &bar.abort;

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.q_empty, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar.k_full[i], 1); mbar_init(&bar.k_empty[i], 1);
      mbar_init(&bar.v_full[i], 1); mbar_init(&bar.v_empty[i], 1);
    }
    mbar_init(&bar.s_full, 1);
    mbar_init(&bar.p_full, 128);
    mbar_init(&bar.p_empty, 1);
    mbar_init(&bar.o_free, 128);
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(&bar.it_full[i], 1);
      mbar_init(&bar.it_empty[i], 5);          // MMA and four softmax warps
    }
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
  const unsigned int total = (unsigned int)B * (unsigned int)QT * (unsigned int)H;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // It also schedules: it publishes item n + 1 after issuing item n's Q and
    // first two K/V tiles, where it would otherwise wait for ring slots.
    if (lane == 0) {
      prefetch_tmap(&tm_q); prefetch_tmap(&tm_k); prefetch_tmap(&tm_v);
      int k_issued = 0, v_issued = 0, gt = 0;       // K / V tiles issued, tiles walked, over all items
      int qc = 0;                                   // Q tiles issued (items with key tiles)
      Item cur = fetch_item<kCausal>(next, total, cu, cu_k, T, T_k, H, QT, abort_flag, status);
      bool ok = publish_item(bar, 0, cur, abort_flag, status);
      for (int n = 0; ok && cur.b >= 0; ++n) {
        if (cur.nk > 0) {
          // Q of this item once the previous item's last S has been computed
          if (!(ok = mbar_wait(&bar.q_empty, (qc & 1) ^ 1, abort_flag, status))) break;
          mbar_arrive_expect_tx(&bar.q_full, kQBytes);
          tma_load_3d(sQ, &tm_q, &bar.q_full, 0, cur.h, cur.lo + cur.qi * kBQ);
          ++qc;
        }
        Item nxt;
        nxt.b = -1;
        const int nk = cur.nk;
        for (int j = 0; j <= nk && ok; ++j) {
          if (j == min(nk, kStages)) {          // the next item, while the ring is full
            nxt = fetch_item<kCausal>(next, total, cu, cu_k, T, T_k, H, QT, abort_flag, status);
            if (!(ok = publish_item(bar, n + 1, nxt, abort_flag, status))) break;
          }
          if (j == nk) break;
          const int st = gt % kStages;
          const uint32_t rd = (uint32_t)(gt / kStages);
          if (!(ok = mbar_wait(&bar.k_empty[st], (rd & 1) ^ 1, abort_flag, status))) break;
          mbar_arrive_expect_tx(&bar.k_full[st], kKVBytes);
          tma_load_3d(sK + st * kKVBytes, &tm_k, &bar.k_full[st], 0, cur.h, cur.klo + j * kBK);
          k_issued = gt + 1;
          if (!(ok = mbar_wait(&bar.v_empty[st], (rd & 1) ^ 1, abort_flag, status))) break;
          mbar_arrive_expect_tx(&bar.v_full[st], kKVBytes);
          tma_load_3d(sV + st * kKVBytes, &tm_v, &bar.v_full[st], 0, cur.h, cur.klo + j * kBK);
          v_issued = gt + 1;
          ++gt;
        }
        cur = nxt;
      }
      // drain the copies this thread issued
      if (qc > 0) mbar_wait(&bar.q_full, (qc - 1) & 1, nullptr, status);
      for (int j = k_issued - kStages; j < k_issued; ++j)
        if (j >= 0) mbar_wait(&bar.k_full[j % kStages], (uint32_t)(j / kStages) & 1, nullptr, status);
      for (int j = v_issued - kStages; j < v_issued; ++j)
        if (j >= 0) mbar_wait(&bar.v_full[j % kStages], (uint32_t)(j / kStages) & 1, nullptr, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t id_s = idesc_bf16_f32(128, kBK);
    const uint32_t id_o = idesc_bf16_f32(128, kD) | (1u << 16);   // B (= V) MN-major
    const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV);
    const bool leader = elect_one();
    int gt = 0;
    int qc = 0;
    bool ok = true;
    Item it;
    for (int n = 0; ok && (ok = take_item(bar, n, abort_flag, status, it)); ++n) {
      if (it.b < 0) break;
      if (it.nk == 0) continue;
      if (!(ok = mbar_wait_warp(&bar.q_full, qc & 1, abort_flag, status))) break;
      for (int j = 0; j < it.nk && ok; ++j, ++gt) {
        const int st = gt % kStages;
        const uint32_t rd = (uint32_t)(gt / kStages);
        // S_j: needs K_j, and S/P free (the previous tile's PV complete)
        if (!(ok = mbar_wait_warp(&bar.k_full[st], rd & 1, abort_flag, status))) break;
        if (gt > 0 && !(ok = mbar_wait_warp(&bar.p_empty, (uint32_t)(gt - 1) & 1, abort_flag, status))) break;
        tc_fence_after();
        if (leader) {
          const uint32_t kb = k_base + st * kKVBytes;
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            mma_bf16(tmem + kColS, sdesc_k128(q_base + kk * 32), sdesc_k128(kb + kk * 32), id_s, kk > 0);
          mma_commit(&bar.s_full);
          mma_commit(&bar.k_empty[st]);
          if (j == it.nk - 1) mma_commit(&bar.q_empty);   // Q is free once this S is computed
        }
        __syncwarp();
        // PV_j once the softmax has written P_j over S_j; the item's first PV
        // also waits until the previous item's O has been read
        if (!(ok = mbar_wait_warp(&bar.p_full, (uint32_t)gt & 1, abort_flag, status))) break;
        if (!(ok = mbar_wait_warp(&bar.v_full[st], rd & 1, abort_flag, status))) break;
        if (j == 0 && qc > 0 && !(ok = mbar_wait_warp(&bar.o_free, (qc - 1) & 1, abort_flag, status))) break;
        tc_fence_after();
        if (leader) {
          const uint32_t vb = v_base + st * kKVBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)    // 16 keys = 8 packed TMEM columns of P
            mma_bf16_ts(tmem + kColO, tmem + kColS + 8 * kk, sdesc_k128(vb + kk * 2048), id_o,
                        (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar.p_empty);          // PV_j done: S/P free, O holds tiles 0..j
          mma_commit(&bar.v_empty[st]);
        }
        __syncwarp();
      }
      ++qc;
    }
    if (leader) mma_commit(&bar.mma_done);
    __syncwarp();
    mbar_wait_warp(&bar.mma_done, 0, nullptr, status);
  } else {
    // ------------------------------------------------------------ softmax
    const int qd = warp & 3;
    const int r = qd * 32 + lane;                 // query row within the tile
    const uint32_t lane_addr = (uint32_t)(qd * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + kColS;
    int gt = 0;
    bool ok = true;
    Item it;
    for (int n = 0; ok && (ok = take_item(bar, n, abort_flag, status, it)); ++n) {
      if (it.b < 0) break;
      const int n_q = it.hi - it.lo, n_k = it.khi - it.klo, qi = it.qi;
      const int diag = n_k - n_q;                 // causal: query i sees keys j <= i + diag
      const int64_t t = (int64_t)it.lo + qi * kBQ + r;
      if (it.nk == 0) {
        // no row of this tile sees a key: zeros and lse = -inf
        if (t < it.hi) {
          uint4* op = reinterpret_cast<uint4*>(o + (t * H + it.h) * kD);
#pragma unroll
          for (int u = 0; u < kD / 8; ++u) op[u] = make_uint4(0u, 0u, 0u, 0u);
          if (lse) lse[(int64_t)it.h * T + t] = -INFINITY;
        }
        continue;
      }
      // a warp whose 32 rows all lie past the segment's end (the last query
      // tile of a segment) keeps the hand-offs but skips the arithmetic:
      // its P and O rows are never stored
      const bool live = __any_sync(0xffffffffu, t < it.hi);
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < it.nk; ++j, ++gt) {
        if (!(ok = mbar_wait_warp(&bar.s_full, (uint32_t)gt & 1, abort_flag, status))) break;
        tc_fence_after();
        __syncwarp();
        if (live)
          softmax_tile<kCausal>(s_addr, tmem + lane_addr + kColO, j, n_k, qi * kBQ + r, diag, scale_log2, m, l);
        tc_fence_before();
        mbar_arrive(&bar.p_full);
      }
      if (!ok) break;
      // O of this item is complete once its last PV has
      if (!(ok = mbar_wait_warp(&bar.p_empty, (uint32_t)(gt - 1) & 1, abort_flag, status))) break;
      tc_fence_after();
      __syncwarp();
      const float inv = l > 0.f ? 1.0f / l : 0.f;   // causal rows that see no key: zeros
#pragma unroll 1
      for (int g = 0; g < 2 && live; ++g) {
        float ov[32];
        tmem_ld32(tmem + lane_addr + kColO + 32 * g, ov);
        tmem_ld_wait();
        if (t < it.hi) {
          bf16* op = o + (t * H + it.h) * kD + 32 * g;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16x2(ov[8 * u] * inv, ov[8 * u + 1] * inv);
            w.y = pack_bf16x2(ov[8 * u + 2] * inv, ov[8 * u + 3] * inv);
            w.z = pack_bf16x2(ov[8 * u + 4] * inv, ov[8 * u + 5] * inv);
            w.w = pack_bf16x2(ov[8 * u + 6] * inv, ov[8 * u + 7] * inv);
            *reinterpret_cast<uint4*>(op + 8 * u) = w;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bar.o_free);                   // the next item's first PV may overwrite O
      if (t < it.hi && lse) lse[(int64_t)it.h * T + t] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
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
  CUtensorMap mq, mk, mv;
  if (!make_map_thd(&mq, p.q, p.T_q, p.H, kBQ) || !make_map_thd(&mk, p.k, p.T_k, p.H, kBK) ||
      !make_map_thd(&mv, p.v, p.T_k, p.H, kBK))
    return cudaErrorInvalidValue;
  const int QT = max(1, (p.max_len_q + kBQ - 1) / kBQ);
  const int64_t items = (int64_t)p.B * QT * p.H;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const float scale_log2 = p.scale * 1.4426950408889634f;
  cudaError_t e;
  // Short segments (few key tiles per item): persistent CTAs over the
  // caller's work counter; long ones, or no counter given: one CTA per item.
  // The crossover measured on the 65,536-token sweeps lies between mean
  // lengths of 512 and 1,024 tokens.
  if (p.work && p.T_q <= (int64_t)768 * p.B) {
    unsigned int* next = p.work;
    e = cudaMemsetAsync(next, 0, sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    auto kern = p.causal ? attn_persistent_kernel<true> : attn_persistent_kernel<false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = (int)min64(items, (int64_t)sm_count() * 4);
    kern<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, p.cu_q, p.cu_k, p.B, p.T_q, p.T_k, p.H, QT, scale_log2,
                                            (bf16*)p.o, p.lse, next, status);
  } else {
    auto kern = p.causal ? attn_item_kernel<true> : attn_item_kernel<false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)items, kThreads, kSmemBytes, s>>>(mq, mk, mv, p.cu_q, p.cu_k, p.B, p.T_q, p.T_k, p.H, QT,
                                                       scale_log2, (bf16*)p.o, p.lse, status);
  }
  return cudaGetLastError();
}

}  // namespace nt
