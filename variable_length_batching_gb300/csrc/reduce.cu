// Segmented column mean over the pair state ("DanLing NestedTensor" Eq. 1
// third line and Eq. 4, "Consuming one logical axis"):
//     m[cu_i + a] = (1/M_i) sum_b z[pair_off_i + a M_i + b]
// with M_i the row length (= N_i for square pairs; the rectangular variant
// divides by M_i, Appendix A.1), zero rows when M_i = 0.
// Every pair row's M_i cells are contiguous, so one CTA owns one pair row:
// its threads split the row's cells, each keeping a 16-byte feature vector
// of fp32 sums, then the cell groups are combined through shared memory.
// HBM-bound: reads P * C_z elements once, writes T * C_z.
#include "nt_common.cuh"

namespace nt {
namespace {

constexpr int kThreads = 128;

// kSq: also the weighted squared sum of Eq. 5's pair term ("DanLing
// NestedTensor" Appendix A.1), sum over the CTA's rows of beta_b * ||row's
// cells||^2 with beta_b = 1.5 - b / (2B): squares in fp32 per thread and row,
// the row's total over the CTA in fp32, the rows in double, into
// sq_part[blockIdx.x].
template <typename T, bool kSq>
__global__ void __launch_bounds__(kThreads, sizeof(T) == 2 ? 12 : 10)   // the kSq variants at the plain ones' occupancy
reduce_kernel(const T* __restrict__ z, const int32_t* __restrict__ row_len,
              const int32_t* __restrict__ row_sample, const int64_t* __restrict__ row_start,
              int64_t rows, int C_z, T* __restrict__ m, double* __restrict__ sq_part, int B) {
  pdl_wait();                                  // z comes from the kernel before
  pdl_trigger();
  extern __shared__ float part[];              // [groups][C_z], then kThreads squares (kSq)
  const int lanes = C_z / 8;                   // vectors per cell (<= kThreads)
  const int groups = kThreads / lanes;         // cells summed concurrently
  const int lane = threadIdx.x % lanes, grp = threadIdx.x / lanes;
  const bool active = grp < groups;
  float* sqs = part + groups * C_z;
  double cta_sq = 0.0;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const int bs = row_sample[r];
    const int64_t n = row_len[bs];
    // the row's Eq. 5 weight beta_b, formed in double before the row's loads
    // so that the (slow) fp64 division overlaps them
    double wrow = 0.0;
    if (kSq && threadIdx.x == 0) wrow = 1.5 - (double)bs / (2.0 * B);
    const T* zr = z + row_start[r] * C_z + lane * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float sq = 0.f;
    if (active) {
      int64_t b = grp;
      // two independent loads in flight per iteration
      for (; b + groups < n; b += 2 * groups) {
        float x0[8], x1[8];
        load8(zr + b * C_z, x0);
        load8(zr + (b + groups) * C_z, x1);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          acc[t] += x0[t] + x1[t];
          if (kSq) sq = fmaf(x1[t], x1[t], fmaf(x0[t], x0[t], sq));
        }
      }
      for (; b < n; b += groups) {
        float x0[8];
        load8(zr + b * C_z, x0);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          acc[t] += x0[t];
          if (kSq) sq = fmaf(x0[t], x0[t], sq);
        }
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) part[grp * C_z + lane * 8 + t] = acc[t];
    }
    if (kSq) sqs[threadIdx.x] = sq;
    __syncthreads();
    if (kSq && threadIdx.x < 32) {
      float v = 0.f;
      for (int i = threadIdx.x; i < kThreads; i += 32) v += sqs[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (threadIdx.x == 0) cta_sq += wrow * (double)v;
    }
    if (grp == 0) {
      float tot[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) tot[t] = part[lane * 8 + t];
      for (int g = 1; g < groups; ++g)
#pragma unroll
        for (int t = 0; t < 8; ++t) tot[t] += part[g * C_z + lane * 8 + t];
      const float inv = n > 0 ? 1.0f / (float)n : 0.f;
#pragma unroll
      for (int t = 0; t < 8; ++t) tot[t] *= inv;
      store8(m + r * C_z + lane * 8, tot);
    }
    __syncthreads();
  }
  if (kSq && threadIdx.x == 0) sq_part[blockIdx.x] = cta_sq;
}

// fp32 widths that are multiples of 4 but not of 8: one thread per feature.
__global__ void reduce_kernel_f32_scalar(const float* __restrict__ z, const int32_t* __restrict__ row_len,
                                         const int32_t* __restrict__ row_sample,
                                         const int64_t* __restrict__ row_start, int64_t rows, int C_z,
                                         float* __restrict__ m) {
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const int64_t n = row_len[row_sample[r]];
    const float* zr = z + row_start[r] * C_z;
    for (int c = threadIdx.x; c < C_z; c += blockDim.x) {
      float acc = 0.f;
      for (int64_t b = 0; b < n; ++b) acc += zr[b * C_z + c];
      m[r * C_z + c] = n > 0 ? acc / (float)n : 0.f;
    }
  }
}

// m = m_acc / M_i for every single row (zero when M_i = 0), in the I/O dtype:
// the division of the fused block's column sums (Eq. 4, then the mean).
template <typename TOut>
__global__ void mean_finish_kernel(const float* __restrict__ m_acc, const int32_t* __restrict__ row_len,
                                   const int32_t* __restrict__ row_sample, int64_t T, int C_z, TOut* __restrict__ m) {
  const int64_t vecs = T * (C_z / 4);
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < vecs; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / (C_z / 4);
    const int64_t n = row_len[row_sample[r]];
    const float inv = n > 0 ? 1.0f / (float)n : 0.f;
    const float4 a = reinterpret_cast<const float4*>(m_acc)[e];
    const float o[4] = {a.x * inv, a.y * inv, a.z * inv, a.w * inv};
#pragma unroll
    for (int t = 0; t < 4; ++t) m[4 * e + t] = from_f32<TOut>(o[t]);
  }
}

}  // namespace

cudaError_t launch_mean_finish(nt_dtype dt, const float* m_acc, const nt_partition* p, int C_z, void* m,
                               cudaStream_t s) {
  if (p->T == 0) return cudaSuccess;
  const int64_t vecs = p->T * (C_z / 4);
  const int grid = (int)min64((vecs + 255) / 256, (int64_t)sm_count() * 16);
  if (dt == NT_BF16)
    mean_finish_kernel<bf16><<<grid, 256, 0, s>>>(m_acc, col_lengths_of(p), p->row_sample, p->T, C_z, (bf16*)m);
  else
    mean_finish_kernel<float><<<grid, 256, 0, s>>>(m_acc, col_lengths_of(p), p->row_sample, p->T, C_z, (float*)m);
  return cudaGetLastError();
}

bool reduce_sq_supported(int C_z) { return C_z % 8 == 0 && C_z / 8 <= kThreads; }

cudaError_t launch_reduce(nt_dtype dt, const void* z, const nt_partition* p, int C_z, void* m,
                          cudaStream_t s, double* sq_part, int* sq_parts) {
  if (sq_parts) *sq_parts = 0;
  if (p->T == 0) return cudaSuccess;
  const int sms = sm_count();
  const int grid = (int)min64(min64(p->T, (int64_t)sms * 32), kReduceMaxGrid);
  const int32_t* cl = col_lengths_of(p);     // cells per pair row
  if (reduce_sq_supported(C_z)) {
    const int groups = kThreads / (C_z / 8);
    const size_t smem = sizeof(float) * (groups * C_z + (sq_part ? kThreads : 0));
    if (sq_parts && sq_part) *sq_parts = grid;
    if (dt == NT_BF16)
      return sq_part ? launch_pdl(reduce_kernel<bf16, true>, dim3(grid), dim3(kThreads), smem, s, (const bf16*)z, cl,
                                  p->row_sample, p->row_start, p->T, C_z, (bf16*)m, sq_part, p->B)
                     : launch_pdl(reduce_kernel<bf16, false>, dim3(grid), dim3(kThreads), smem, s, (const bf16*)z, cl,
                                  p->row_sample, p->row_start, p->T, C_z, (bf16*)m, (double*)nullptr, p->B);
    else
      return sq_part ? launch_pdl(reduce_kernel<float, true>, dim3(grid), dim3(kThreads), smem, s, (const float*)z,
                                  cl, p->row_sample, p->row_start, p->T, C_z, (float*)m, sq_part, p->B)
                     : launch_pdl(reduce_kernel<float, false>, dim3(grid), dim3(kThreads), smem, s, (const float*)z,
                                  cl, p->row_sample, p->row_start, p->T, C_z, (float*)m, (double*)nullptr, p->B);
  } else {
    reduce_kernel_f32_scalar<<<grid, 128, 0, s>>>((const float*)z, cl, p->row_sample,
                                                 p->row_start, p->T, C_z, (float*)m);
  }
  return cudaGetLastError();
}

}  // namespace nt
