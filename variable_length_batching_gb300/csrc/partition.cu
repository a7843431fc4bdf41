// Partitions of a packed batch: exclusive scans of N_i and N_i^2 (sample
// offsets of singles and of square pairs) and the second-level row splits of
// the pair state.  "DanLing NestedTensor", section 3.1 Eq. 2 and Figure 2;
// section 3.2 Eq. 3; Appendix A "Structural invariants".  Rectangular pair
// states (section 3.2 "Consuming one logical axis", Eq. 4) add the column
// lengths M_i: the pair offsets scan N_i * M_i and rows are M_i cells long.
#include "nt_common.cuh"

namespace nt {
namespace {

constexpr int kScanThreads = 1024;

// One CTA scans the whole length vector in chunks of 1024 with a running
// carry; B is batch-sized metadata, so a single CTA is the right shape.
// cols == NULL: square pairs (M_i = N_i).  totals = {T, P, max_len, check,
// T_cols, max_col_len}; check bit 1: some length < 0, bit 2: T does not fit
// int32, bit 4: T_cols does not fit int32.
__global__ void __launch_bounds__(kScanThreads)
partition_scan_kernel(const int32_t* __restrict__ lengths, const int32_t* __restrict__ cols, int32_t B,
                      int32_t* __restrict__ cu, int32_t* __restrict__ cu_cols, int64_t* __restrict__ pair_off,
                      int64_t* __restrict__ totals, int64_t* host_totals) {
  __shared__ long long warp_n[32], warp_m[32], warp_nm[32];
  __shared__ int warp_max[32], warp_maxm[32];
  __shared__ long long carry_n, carry_m, carry_nm;
  __shared__ int carry_max, carry_maxm, bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) { carry_n = 0; carry_m = 0; carry_nm = 0; carry_max = 0; carry_maxm = 0; bad = 0; }
  __syncthreads();
  for (int base = 0; base < B; base += kScanThreads) {
    const int b = base + tid;
    long long n = 0, m = 0;
    if (b < B) {
      int nb = lengths[b];
      if (nb < 0) { atomicOr(&bad, 1); nb = 0; }
      int mb = cols ? cols[b] : nb;
      if (mb < 0) { atomicOr(&bad, 1); mb = 0; }
      n = nb;
      m = mb;
    }
    long long nm = n * m;
    int mx = (int)n, mxm = (int)m;
    // inclusive warp scans
    long long in_n = n, in_m = m, in_nm = nm;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      long long t1 = __shfl_up_sync(0xffffffffu, in_n, off);
      long long t2 = __shfl_up_sync(0xffffffffu, in_m, off);
      long long t3 = __shfl_up_sync(0xffffffffu, in_nm, off);
      if (lane >= off) { in_n += t1; in_m += t2; in_nm += t3; }
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      mxm = max(mxm, __shfl_xor_sync(0xffffffffu, mxm, off));
    }
    if (lane == 31) { warp_n[warp] = in_n; warp_m[warp] = in_m; warp_nm[warp] = in_nm; }
    if (lane == 0) { warp_max[warp] = mx; warp_maxm[warp] = mxm; }
    __syncthreads();
    if (warp == 0) {
      long long wn = warp_n[lane], wm_ = warp_m[lane], wnm = warp_nm[lane];
      int wx = warp_max[lane], wxm = warp_maxm[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        long long t1 = __shfl_up_sync(0xffffffffu, wn, off);
        long long t2 = __shfl_up_sync(0xffffffffu, wm_, off);
        long long t3 = __shfl_up_sync(0xffffffffu, wnm, off);
        if (lane >= off) { wn += t1; wm_ += t2; wnm += t3; }
        wx = max(wx, __shfl_xor_sync(0xffffffffu, wx, off));
        wxm = max(wxm, __shfl_xor_sync(0xffffffffu, wxm, off));
      }
      warp_n[lane] = wn;   // inclusive over warps
      warp_m[lane] = wm_;
      warp_nm[lane] = wnm;
      if (lane == 0) { warp_max[0] = wx; warp_maxm[0] = wxm; }
    }
    __syncthreads();
    const long long before_n = carry_n + (warp > 0 ? warp_n[warp - 1] : 0) + in_n - n;
    const long long before_m = carry_m + (warp > 0 ? warp_m[warp - 1] : 0) + in_m - m;
    const long long before_nm = carry_nm + (warp > 0 ? warp_nm[warp - 1] : 0) + in_nm - nm;
    if (b < B) {
      if (before_n > 0x7fffffffLL) atomicOr(&bad, 2);
      if (before_m > 0x7fffffffLL) atomicOr(&bad, 4);
      cu[b] = (int32_t)before_n;
      if (cu_cols) cu_cols[b] = (int32_t)before_m;
      pair_off[b] = before_nm;
    }
    __syncthreads();
    if (tid == 0) {
      carry_n += warp_n[31];
      carry_m += warp_m[31];
      carry_nm += warp_nm[31];
      carry_max = max(carry_max, warp_max[0]);
      carry_maxm = max(carry_maxm, warp_maxm[0]);
    }
    __syncthreads();
  }
  if (tid == 0) {
    if (carry_n > 0x7fffffffLL) bad |= 2;
    if (carry_m > 0x7fffffffLL) bad |= 4;
    cu[B] = (int32_t)carry_n;
    if (cu_cols) cu_cols[B] = (int32_t)carry_m;
    pair_off[B] = carry_nm;
    totals[0] = carry_n;
    totals[1] = carry_nm;
    totals[2] = carry_max;
    totals[3] = bad;
    if (cols) {
      totals[4] = carry_m;
      totals[5] = carry_maxm;
    }
    if (host_totals) {
      for (int i = 0; i < (cols ? 6 : 4); ++i) host_totals[i] = totals[i];
      __threadfence_system();
    }
  }
}

// Grid-stride over samples; the threads of a CTA walk the rows a of one
// sample: row_start[cu_i + a] = pair_off[i] + a * M_i (Eq. 3 with b = 0;
// Eq. 4 for rectangular states; M_i = N_i when cols is NULL).
__global__ void partition_rows_kernel(const int32_t* __restrict__ lengths, const int32_t* __restrict__ cols,
                                      const int32_t* __restrict__ cu,
                                      const int64_t* __restrict__ pair_off, int32_t B, int64_t T,
                                      int64_t P, int64_t* __restrict__ row_start,
                                      int32_t* __restrict__ row_sample) {
  for (int i = blockIdx.x; i < B; i += gridDim.x) {
    const int64_t n = lengths[i];
    const int64_t mcols = cols ? cols[i] : n;
    const int64_t c0 = cu[i];
    const int64_t o = pair_off[i];
    for (int64_t a = threadIdx.x; a < n; a += blockDim.x) {
      row_start[c0 + a] = o + a * mcols;
      row_sample[c0 + a] = i;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) row_start[T] = P;
}

// The same row splits with T and P read from the scan's device totals, so
// the kernel can follow the scan in the stream without a host round trip.
// Writes are bounded by the caller's capacity `cap` (rows of row_start
// beyond it, and negative offsets from invalid lengths, are skipped; the
// host reports the shortfall after reading the totals back).
__global__ void partition_rows_dev_kernel(const int32_t* __restrict__ lengths, const int32_t* __restrict__ cols,
                                          const int32_t* __restrict__ cu, const int64_t* __restrict__ pair_off,
                                          int32_t B, const int64_t* __restrict__ totals, int64_t cap,
                                          int64_t* __restrict__ row_start, int32_t* __restrict__ row_sample) {
  for (int i = blockIdx.x; i < B; i += gridDim.x) {
    const int64_t n = lengths[i];
    const int64_t mcols = cols ? cols[i] : n;
    const int64_t c0 = cu[i];
    const int64_t o = pair_off[i];
    for (int64_t a = threadIdx.x; a < n; a += blockDim.x) {
      const int64_t r = c0 + a;
      if (r >= 0 && r < cap) {
        row_start[r] = o + a * mcols;
        row_sample[r] = i;
      }
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const int64_t T = totals[0];
    if (T >= 0 && T <= cap) row_start[T] = totals[1];
  }
}

// Square partitions of small batches in one launch: one CTA scans N_i and
// N_i^2 (B <= 1024, one chunk) into shared memory, writes cu, pair_off and
// the totals, then its threads take rows t = tid, tid + 1024, ... below
// min(T, cap) and find the row's sample by binary search over the scanned
// offsets (the last i with cu_i <= t, so empty samples are passed over).
// Outputs and capacity rules are those of the scan followed by the row
// splits above.
constexpr int kFusedMaxB = kScanThreads;
constexpr int64_t kFusedMaxRows = 65536;

__global__ void __launch_bounds__(kScanThreads)
partition_fused_kernel(const int32_t* __restrict__ lengths, int32_t B, int64_t cap, int32_t* __restrict__ cu,
                       int64_t* __restrict__ pair_off, int64_t* __restrict__ totals,
                       int64_t* __restrict__ row_start, int32_t* __restrict__ row_sample, int64_t* host_totals) {
  __shared__ long long warp_n[32], warp_nm[32];
  __shared__ int warp_max[32];
  __shared__ long long s_cu[kFusedMaxB + 1], s_off[kFusedMaxB + 1];
  __shared__ int s_len[kFusedMaxB];
  __shared__ int bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) bad = 0;
  __syncthreads();
  long long n = 0;
  if (tid < B) {
    const int nb = lengths[tid];
    if (nb < 0) atomicOr(&bad, 1);
    n = nb < 0 ? 0 : nb;
  }
  const long long nm = n * n;
  long long in_n = n, in_nm = nm;
  int mx = (int)n;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long t1 = __shfl_up_sync(0xffffffffu, in_n, off);
    const long long t3 = __shfl_up_sync(0xffffffffu, in_nm, off);
    if (lane >= off) { in_n += t1; in_nm += t3; }
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  if (lane == 31) { warp_n[warp] = in_n; warp_nm[warp] = in_nm; }
  if (lane == 0) warp_max[warp] = mx;
  __syncthreads();
  if (warp == 0) {
    long long wn = warp_n[lane], wnm = warp_nm[lane];
    int wx = warp_max[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long t1 = __shfl_up_sync(0xffffffffu, wn, off);
      const long long t3 = __shfl_up_sync(0xffffffffu, wnm, off);
      if (lane >= off) { wn += t1; wnm += t3; }
      wx = max(wx, __shfl_xor_sync(0xffffffffu, wx, off));
    }
    warp_n[lane] = wn;
    warp_nm[lane] = wnm;
    if (lane == 0) warp_max[0] = wx;
  }
  __syncthreads();
  const long long before_n = (warp > 0 ? warp_n[warp - 1] : 0) + in_n - n;
  const long long before_nm = (warp > 0 ? warp_nm[warp - 1] : 0) + in_nm - nm;
  if (tid < B) {
    if (before_n > 0x7fffffffLL) atomicOr(&bad, 2);
    cu[tid] = (int32_t)before_n;
    pair_off[tid] = before_nm;
    s_cu[tid] = before_n;
    s_off[tid] = before_nm;
    s_len[tid] = (int)n;
  }
  const long long T = warp_n[31], P = warp_nm[31];
  __syncthreads();
  if (tid == 0) {
    if (T > 0x7fffffffLL) bad |= 2;
    cu[B] = (int32_t)T;
    pair_off[B] = P;
    totals[0] = T;
    totals[1] = P;
    totals[2] = warp_max[0];
    totals[3] = bad;
    if (T <= cap) row_start[T] = P;
    if (host_totals) {
      host_totals[0] = T;
      host_totals[1] = P;
      host_totals[2] = warp_max[0];
      host_totals[3] = bad;
      __threadfence_system();
    }
  }
  const long long rows = T < cap ? T : cap;
  for (long long t = tid; t < rows; t += kScanThreads) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    row_start[t] = s_off[lo] + (t - s_cu[lo]) * s_len[lo];
    row_sample[t] = lo;
  }
}

}  // namespace

bool partition_fused_fits(int32_t B, int64_t cap) { return B >= 1 && B <= kFusedMaxB && cap <= kFusedMaxRows; }

cudaError_t launch_partition_fused(const int32_t* lengths, int32_t B, int64_t cap, int32_t* cu, int64_t* pair_off,
                                   int64_t* totals, int64_t* row_start, int32_t* row_sample, int64_t* host_totals,
                                   cudaStream_t s) {
  partition_fused_kernel<<<1, kScanThreads, 0, s>>>(lengths, B, cap, cu, pair_off, totals, row_start, row_sample,
                                                    host_totals);
  return cudaGetLastError();
}

cudaError_t launch_partition_rows_dev(const int32_t* lengths, const int32_t* cols, const int32_t* cu,
                                      const int64_t* pair_off, int32_t B, const int64_t* totals, int64_t cap,
                                      int64_t* row_start, int32_t* row_sample, cudaStream_t s) {
  const int grid = B < 4096 ? (B > 0 ? B : 1) : 4096;
  partition_rows_dev_kernel<<<grid, 256, 0, s>>>(lengths, cols, cu, pair_off, B, totals, cap, row_start,
                                                 row_sample);
  return cudaGetLastError();
}

cudaError_t launch_partition_scan(const int32_t* lengths, const int32_t* cols, int32_t B, int32_t* cu,
                                  int32_t* cu_cols, int64_t* pair_off, int64_t* totals, int64_t* host_totals,
                                  cudaStream_t s) {
  partition_scan_kernel<<<1, kScanThreads, 0, s>>>(lengths, cols, B, cu, cu_cols, pair_off, totals, host_totals);
  return cudaGetLastError();
}

cudaError_t launch_partition_rows(const int32_t* lengths, const int32_t* cols, const int32_t* cu,
                                  const int64_t* pair_off, int32_t B, int64_t T, int64_t P, int64_t* row_start,
                                  int32_t* row_sample, cudaStream_t s) {
  const int grid = B < 4096 ? (B > 0 ? B : 1) : 4096;
  partition_rows_kernel<<<grid, 256, 0, s>>>(lengths, cols, cu, pair_off, B, T, P, row_start, row_sample);
  return cudaGetLastError();
}

}  // namespace nt
