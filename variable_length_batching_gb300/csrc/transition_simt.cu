// Residual transition on fp32 CUDA cores: z~ = z + W2 ReLU(W1 LN(z) + b1) + b2
// per packed cell ("DanLing NestedTensor" Eq. 1 second line; section 3.2
// "Retaining structure through feature transformations"), or with the
// SwiGLU update the paper measures (W3 given): the hidden unit is
// SiLU(W1 x + b1) * (W3 x + b3).  Used for the fp32
// mode (no fp32 tensor-core path exists) and for widths the tensor-core
// kernel does not cover.  The cell-wise math never looks at the partition:
// every packed row is one independent cell.
#include "nt_common.cuh"

namespace nt {
namespace {

constexpr int kRowsPerCta = 8;   // one warp normalises one cell
constexpr int kThreads = 256;

__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

template <typename T, bool kGLU>
__global__ void __launch_bounds__(kThreads)
transition_simt_kernel(const T* z_in, T* z_out, int64_t P, int C_z,
                       int H_t, const float* __restrict__ gamma, const float* __restrict__ beta,
                       float eps, const T* __restrict__ W1, const float* __restrict__ b1,
                       const T* __restrict__ W3, const float* __restrict__ b3,
                       const T* __restrict__ W2, const float* __restrict__ b2) {
  extern __shared__ float smem[];
  float* xs = smem;                         // [kRowsPerCta][C_z]  LN(z)
  float* hs = smem + kRowsPerCta * C_z;     // [kRowsPerCta][H_t]  ReLU(W1 x + b1)
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int64_t r0 = (int64_t)blockIdx.x * kRowsPerCta; r0 < P; r0 += (int64_t)gridDim.x * kRowsPerCta) {
    const int nrows = (int)min64(kRowsPerCta, P - r0);
    // LayerNorm of one cell per warp: two passes over the row in smem.
    if (warp < nrows) {
      const T* zr = z_in + (r0 + warp) * C_z;
      float* xr = xs + warp * C_z;
      float sum = 0.f;
      for (int c = lane; c < C_z; c += 32) {
        float x = to_f32(zr[c]);
        xr[c] = x;
        sum += x;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      const float mean = sum / C_z;
      float sq = 0.f;
      for (int c = lane; c < C_z; c += 32) {
        float d = xr[c] - mean;
        sq += d * d;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
      const float rstd = rsqrtf(sq / C_z + eps);
      for (int c = lane; c < C_z; c += 32) xr[c] = (xr[c] - mean) * rstd * gamma[c] + beta[c];
    }
    __syncthreads();
    // hidden = ReLU(W1 x + b1), or SiLU(W1 x + b1) * (W3 x + b3): thread per
    // hidden unit, all rows at once.
    for (int h = threadIdx.x; h < H_t; h += kThreads) {
      float acc[kRowsPerCta], accv[kRowsPerCta];
#pragma unroll
      for (int r = 0; r < kRowsPerCta; ++r) { acc[r] = 0.f; accv[r] = 0.f; }
      const T* w = W1 + (int64_t)h * C_z;
      const T* w3 = kGLU ? W3 + (int64_t)h * C_z : nullptr;
      for (int c = 0; c < C_z; ++c) {
        const float wc = to_f32(w[c]);
#pragma unroll
        for (int r = 0; r < kRowsPerCta; ++r) acc[r] = fmaf(xs[r * C_z + c], wc, acc[r]);
        if (kGLU) {
          const float vc = to_f32(w3[c]);
#pragma unroll
          for (int r = 0; r < kRowsPerCta; ++r) accv[r] = fmaf(xs[r * C_z + c], vc, accv[r]);
        }
      }
      const float bias = b1 ? b1[h] : 0.f;
      const float bias3 = (kGLU && b3) ? b3[h] : 0.f;
#pragma unroll
      for (int r = 0; r < kRowsPerCta; ++r)
        hs[r * H_t + h] = kGLU ? silu(acc[r] + bias) * (accv[r] + bias3) : fmaxf(acc[r] + bias, 0.f);
    }
    __syncthreads();
    // z~ = z + W2 hidden + b2: thread per output feature.
    for (int c = threadIdx.x; c < C_z; c += kThreads) {
      float acc[kRowsPerCta];
#pragma unroll
      for (int r = 0; r < kRowsPerCta; ++r) acc[r] = 0.f;
      const T* w = W2 + (int64_t)c * H_t;
      for (int h = 0; h < H_t; ++h) {
        const float wh = to_f32(w[h]);
#pragma unroll
        for (int r = 0; r < kRowsPerCta; ++r) acc[r] = fmaf(hs[r * H_t + h], wh, acc[r]);
      }
      const float bias = b2 ? b2[c] : 0.f;
      for (int r = 0; r < nrows; ++r) {
        const int64_t idx = (r0 + r) * C_z + c;
        z_out[idx] = from_f32<T>(to_f32(z_in[idx]) + acc[r] + bias);
      }
    }
    __syncthreads();
  }
}

}  // namespace

size_t transition_simt_smem(int C_z, int H_t) {
  return sizeof(float) * kRowsPerCta * (size_t)(C_z + H_t);
}

namespace {

template <typename T, bool kGLU>
cudaError_t launch_t(const void* z_in, void* z_out, int64_t P, int C_z, int H_t, const float* gamma,
                     const float* beta, float eps, const void* W1, const float* b1, const void* W3,
                     const float* b3, const void* W2, const float* b2, cudaStream_t s) {
  const size_t smem = transition_simt_smem(C_z, H_t);
  const int sms = sm_count();
  const int64_t ctas = (P + kRowsPerCta - 1) / kRowsPerCta;
  const int grid = (int)min64(ctas, (int64_t)sms * 8);
  cudaError_t e = cudaFuncSetAttribute(transition_simt_kernel<T, kGLU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  transition_simt_kernel<T, kGLU><<<grid, kThreads, smem, s>>>((const T*)z_in, (T*)z_out, P, C_z, H_t, gamma, beta,
                                                               eps, (const T*)W1, b1, (const T*)W3, b3,
                                                               (const T*)W2, b2);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_transition_simt(nt_dtype dt, const void* z_in, void* z_out, int64_t P, int C_z,
                                   int H_t, const float* gamma, const float* beta, float eps,
                                   const void* W1, const float* b1, const void* W3, const float* b3,
                                   const void* W2, const float* b2, cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  if (dt == NT_BF16)
    return W3 ? launch_t<bf16, true>(z_in, z_out, P, C_z, H_t, gamma, beta, eps, W1, b1, W3, b3, W2, b2, s)
              : launch_t<bf16, false>(z_in, z_out, P, C_z, H_t, gamma, beta, eps, W1, b1, W3, b3, W2, b2, s);
  return W3 ? launch_t<float, true>(z_in, z_out, P, C_z, H_t, gamma, beta, eps, W1, b1, W3, b3, W2, b2, s)
            : launch_t<float, false>(z_in, z_out, P, C_z, H_t, gamma, beta, eps, W1, b1, W3, b3, W2, b2, s);
}

}  // namespace nt
