// Pair construction by broadcast ("DanLing NestedTensor" Eq. 1 first line;
// section 3.2 "Creating axes through broadcasting"): the cells of pair row a
// of sample i are z[row_start[cu_i + a] + b] = u[cu_i + a] + v[ccu_i + b],
// b < M_i, where M_i and ccu are the column lengths and offsets (M_i = N_i
// and ccu = cu for square pairs; Eq. 4 for rectangular ones).  Only the
// sum N_i M_i valid cells are written; indices come from the partition
// tensors, not from materialised coordinate maps.
//
// HBM-bound: the kernel writes P * C_z elements and reads u, v (T * C_z
// fp32 each, L2-resident).  Each CTA owns kRows consecutive pair rows of one
// sample, so one load of v[cu_i + b] serves kRows output cells; stores are
// 16-byte vectors, consecutive threads on consecutive addresses.
#include "nt_common.cuh"

namespace nt {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 4;

// C_z with kThreads % (C_z / 8) == 0: a thread's 8-feature slice f is the
// same for every cell it writes, so the kRows u-vectors it adds are loaded
// once per row group and only v is read per cell.
template <typename TOut>
__global__ void __launch_bounds__(kThreads)
broadcast_fixed_slice_kernel(const float* __restrict__ u, const float* __restrict__ v,
                             const int32_t* __restrict__ lengths, const int32_t* __restrict__ cu,
                             const int32_t* __restrict__ col_lengths, const int32_t* __restrict__ col_cu,
                             const int32_t* __restrict__ row_sample, const int64_t* __restrict__ row_start,
                             int64_t T, int C_z, TOut* __restrict__ z) {
  pdl_wait();                                 // u and v come from the kernel before
  pdl_trigger();
  const int vecs = C_z / 8;
  const int f = (threadIdx.x % vecs) * 8;
  const int b_step = kThreads / vecs;
  for (int64_t g = blockIdx.x; g * kRows < T; g += gridDim.x) {
    const int64_t r0 = g * kRows;
    const int64_t r_end = min(r0 + kRows, T);
    int64_t r = r0;
    while (r < r_end) {
      // the rows [r, r1) of one sample inside this group
      const int i = row_sample[r];
      const int64_t r1 = min(r_end, (int64_t)cu[i] + lengths[i]);
      const int64_t n = col_lengths[i];      // cells per row
      const int64_t c0 = col_cu[i];          // first column single
      float uu[kRows][8];
      int64_t rs[kRows];
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        if (r + k < r1) {
          load8(u + (r + k) * C_z + f, uu[k]);
          rs[k] = row_start[r + k];
        }
      }
      for (int64_t b = threadIdx.x / vecs; b < n; b += b_step) {
        float vv[8];
        load8(v + (c0 + b) * C_z + f, vv);
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
          if (r + k < r1) {
            float o[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) o[t] = uu[k][t] + vv[t];
            store8_stream(z + (rs[k] + b) * C_z + f, o);
          }
        }
      }
      r = r1;
    }
  }
}

template <typename TOut>
__global__ void __launch_bounds__(kThreads)
broadcast_kernel(const float* __restrict__ u, const float* __restrict__ v,
                 const int32_t* __restrict__ lengths, const int32_t* __restrict__ cu,
                 const int32_t* __restrict__ col_lengths, const int32_t* __restrict__ col_cu,
                 const int32_t* __restrict__ row_sample, const int64_t* __restrict__ row_start,
                 int64_t T, int C_z, TOut* __restrict__ z) {
  const int vecs = C_z / 8;  // 8 features per thread-vector
  for (int64_t g = blockIdx.x; g * kRows < T; g += gridDim.x) {
    // rows [r0, r1) of one sample: a group never crosses a sample boundary,
    // it is cut at the sample's last row instead.
    const int64_t r0 = g * kRows;
    const int i = row_sample[r0];
    const int64_t r1 = min(r0 + kRows, (int64_t)cu[i] + lengths[i]);
    const int64_t n = col_lengths[i];
    const int64_t c0 = col_cu[i];
    const int64_t nrows = r1 - r0;
    for (int64_t e = threadIdx.x; e < n * vecs; e += kThreads) {
      const int64_t b = e / vecs;
      const int f = (int)(e - b * vecs) * 8;
      float vv[8];
      load8(v + (c0 + b) * C_z + f, vv);
      for (int64_t r = 0; r < nrows; ++r) {
        float uu[8];
        load8(u + (r0 + r) * C_z + f, uu);
#pragma unroll
        for (int t = 0; t < 8; ++t) uu[t] += vv[t];
        store8_stream(z + (row_start[r0 + r] + b) * C_z + f, uu);
      }
    }
    // rows of the next sample that fall into this group of kRows
    for (int64_t r = r1; r < min(r0 + kRows, T); ++r) {
      const int i2 = row_sample[r];
      const int64_t n2 = col_lengths[i2];
      const int64_t c2 = col_cu[i2];
      for (int64_t e = threadIdx.x; e < n2 * vecs; e += kThreads) {
        const int64_t b = e / vecs;
        const int f = (int)(e - b * vecs) * 8;
        float vv[8], uu[8];
        load8(v + (c2 + b) * C_z + f, vv);
        load8(u + r * C_z + f, uu);
#pragma unroll
        for (int t = 0; t < 8; ++t) uu[t] += vv[t];
        store8_stream(z + (row_start[r] + b) * C_z + f, uu);
      }
    }
  }
}

// fp32 output with widths that are multiples of 4 but not 8.
__global__ void __launch_bounds__(kThreads)
broadcast_kernel_f32x4(const float* __restrict__ u, const float* __restrict__ v,
                       const int32_t* __restrict__ col_lengths, const int32_t* __restrict__ col_cu,
                       const int32_t* __restrict__ row_sample, const int64_t* __restrict__ row_start,
                       int64_t T, int C_z, float* __restrict__ z) {
  const int vecs = C_z / 4;
  for (int64_t r = blockIdx.x; r < T; r += gridDim.x) {
    const int i = row_sample[r];
    const int64_t n = col_lengths[i];
    const int64_t c0 = col_cu[i];
    for (int64_t e = threadIdx.x; e < n * vecs; e += kThreads) {
      const int64_t b = e / vecs;
      const int f = (int)(e - b * vecs) * 4;
      float4 a = *reinterpret_cast<const float4*>(u + r * C_z + f);
      float4 c = *reinterpret_cast<const float4*>(v + (c0 + b) * C_z + f);
      *reinterpret_cast<float4*>(z + (row_start[r] + b) * C_z + f) =
          make_float4(a.x + c.x, a.y + c.y, a.z + c.z, a.w + c.w);
    }
  }
}

}  // namespace

cudaError_t launch_broadcast(nt_dtype dt, const float* u, const float* v, const nt_partition* p,
                             int C_z, void* z, cudaStream_t s) {
  if (p->T == 0) return cudaSuccess;
  const int sms = sm_count();
  const int32_t* cl = col_lengths_of(p);
  const int32_t* cc = col_cu_of(p);
  if (C_z % 8 == 0 && kThreads % (C_z / 8) == 0) {
    const int64_t groups = (p->T + kRows - 1) / kRows;
    const int grid = (int)min64(groups, (int64_t)sms * 16);
    if (dt == NT_BF16)
      return launch_pdl(broadcast_fixed_slice_kernel<bf16>, dim3(grid), dim3(kThreads), 0, s, u, v, p->lengths,
                        p->cu_seqlens, cl, cc, p->row_sample, p->row_start, p->T, C_z, (bf16*)z);
    else
      return launch_pdl(broadcast_fixed_slice_kernel<float>, dim3(grid), dim3(kThreads), 0, s, u, v, p->lengths,
                        p->cu_seqlens, cl, cc, p->row_sample, p->row_start, p->T, C_z, (float*)z);
  } else if (C_z % 8 == 0) {
    const int64_t groups = (p->T + kRows - 1) / kRows;
    const int grid = (int)min64(groups, (int64_t)sms * 16);
    if (dt == NT_BF16)
      broadcast_kernel<bf16><<<grid, kThreads, 0, s>>>(u, v, p->lengths, p->cu_seqlens, cl, cc, p->row_sample,
                                                       p->row_start, p->T, C_z, (bf16*)z);
    else
      broadcast_kernel<float><<<grid, kThreads, 0, s>>>(u, v, p->lengths, p->cu_seqlens, cl, cc, p->row_sample,
                                                        p->row_start, p->T, C_z, (float*)z);
  } else {
    const int grid = (int)min64(p->T, (int64_t)sms * 16);
    broadcast_kernel_f32x4<<<grid, kThreads, 0, s>>>(u, v, cl, cc, p->row_sample,
                                                     p->row_start, p->T, C_z, (float*)z);
  }
  return cudaGetLastError();
}

}  // namespace nt
