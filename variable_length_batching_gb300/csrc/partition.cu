// Partitions of a packed batch: exclusive scans of N_i and N_i^2 (sample
// offsets of singles and of square pairs) and the second-level row splits of
// the pair state.  "DanLing NestedTensor", section 3.1 Eq. 2 and Figure 2;
// section 3.2 Eq. 3; Appendix A "Structural invariants".
#include "nt_common.cuh"

namespace nt {
namespace {

constexpr int kScanThreads = 1024;

// One CTA scans the whole length vector in chunks of 1024 with a running
// carry; B is batch-sized metadata, so a single CTA is the right shape.
// totals = {T, P, max_len, check}; check bit 1: some N_i < 0, bit 2: T does
// not fit int32.
__global__ void __launch_bounds__(kScanThreads)
partition_scan_kernel(const int32_t* __restrict__ lengths, int32_t B, int32_t* __restrict__ cu,
                      int64_t* __restrict__ pair_off, int64_t* __restrict__ totals) {
  __shared__ long long warp_n[32], warp_n2[32];
  __shared__ int warp_max[32];
  __shared__ long long carry_n, carry_n2;
  __shared__ int carry_max, bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) { carry_n = 0; carry_n2 = 0; carry_max = 0; bad = 0; }
  __syncthreads();
  for (int base = 0; base < B; base += kScanThreads) {
    const int b = base + tid;
    long long n = 0;
    if (b < B) {
      int nb = lengths[b];
      if (nb < 0) { atomicOr(&bad, 1); nb = 0; }
      n = nb;
    }
    long long n2 = n * n;
    int mx = (int)n;
    // inclusive warp scan
    long long in_n = n, in_n2 = n2;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      long long t1 = __shfl_up_sync(0xffffffffu, in_n, off);
      long long t2 = __shfl_up_sync(0xffffffffu, in_n2, off);
      if (lane >= off) { in_n += t1; in_n2 += t2; }
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    }
    if (lane == 31) { warp_n[warp] = in_n; warp_n2[warp] = in_n2; }
    if (lane == 0) warp_max[warp] = mx;
    __syncthreads();
    if (warp == 0) {
      long long wn = warp_n[lane], wn2 = warp_n2[lane];
      int wm = warp_max[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        long long t1 = __shfl_up_sync(0xffffffffu, wn, off);
        long long t2 = __shfl_up_sync(0xffffffffu, wn2, off);
        if (lane >= off) { wn += t1; wn2 += t2; }
        wm = max(wm, __shfl_xor_sync(0xffffffffu, wm, off));
      }
      warp_n[lane] = wn;   // inclusive over warps
      warp_n2[lane] = wn2;
      if (lane == 0) warp_max[0] = wm;
    }
    __syncthreads();
    const long long before_n = carry_n + (warp > 0 ? warp_n[warp - 1] : 0) + in_n - n;
    const long long before_n2 = carry_n2 + (warp > 0 ? warp_n2[warp - 1] : 0) + in_n2 - n2;
    if (b < B) {
      if (before_n > 0x7fffffffLL) atomicOr(&bad, 2);
      cu[b] = (int32_t)before_n;
      pair_off[b] = before_n2;
    }
    __syncthreads();
    if (tid == 0) {
      carry_n += warp_n[31];
      carry_n2 += warp_n2[31];
      carry_max = max(carry_max, warp_max[0]);
    }
    __syncthreads();
  }
  if (tid == 0) {
    if (carry_n > 0x7fffffffLL) bad |= 2;
    cu[B] = (int32_t)carry_n;
    pair_off[B] = carry_n2;
    totals[0] = carry_n;
    totals[1] = carry_n2;
    totals[2] = carry_max;
    totals[3] = bad;
  }
}

// Grid-stride over samples; the threads of a CTA walk the rows a of one
// sample: row_start[cu_i + a] = pair_off[i] + a * N_i (Eq. 3 with b = 0).
__global__ void partition_rows_kernel(const int32_t* __restrict__ lengths,
                                      const int32_t* __restrict__ cu,
                                      const int64_t* __restrict__ pair_off, int32_t B, int64_t T,
                                      int64_t P, int64_t* __restrict__ row_start,
                                      int32_t* __restrict__ row_sample) {
  for (int i = blockIdx.x; i < B; i += gridDim.x) {
    const int64_t n = lengths[i];
    const int64_t c0 = cu[i];
    const int64_t o = pair_off[i];
    for (int64_t a = threadIdx.x; a < n; a += blockDim.x) {
      row_start[c0 + a] = o + a * n;
      row_sample[c0 + a] = i;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) row_start[T] = P;
}

}  // namespace

cudaError_t launch_partition_scan(const int32_t* lengths, int32_t B, int32_t* cu, int64_t* pair_off,
                                  int64_t* totals, cudaStream_t s) {
  partition_scan_kernel<<<1, kScanThreads, 0, s>>>(lengths, B, cu, pair_off, totals);
  return cudaGetLastError();
}

cudaError_t launch_partition_rows(const int32_t* lengths, const int32_t* cu, const int64_t* pair_off,
                                  int32_t B, int64_t T, int64_t P, int64_t* row_start,
                                  int32_t* row_sample, cudaStream_t s) {
  const int grid = B < 4096 ? (B > 0 ? B : 1) : 4096;
  partition_rows_kernel<<<grid, 256, 0, s>>>(lengths, cu, pair_off, B, T, P, row_start, row_sample);
  return cudaGetLastError();
}

}  // namespace nt
