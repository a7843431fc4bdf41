// Small row-block projections Y = X W^T (+ b) (+ R) on fp32 CUDA cores:
// the single-side Linear layers of the block (u, v and g of "DanLing
// NestedTensor" Eq. 1), computed as V W^T + b on packed rows (section 3.3,
// "Dense work across valid positions").  These act on T = sum N_i single rows
// only, a small fraction of the block's work.
#include "nt_common.cuh"

namespace nt {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, kThreads = 256;

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(kThreads)
linear_kernel(LinearProblem p0, LinearProblem p1,
              int64_t M, int N, int K) {
  const LinearProblem& pr = blockIdx.z == 0 ? p0 : p1;
  const TIn* __restrict__ X = static_cast<const TIn*>(pr.X);
  const TIn* __restrict__ W = static_cast<const TIn*>(pr.W);
  const TIn* __restrict__ R = static_cast<const TIn*>(pr.R);
  TOut* __restrict__ Y = static_cast<TOut*>(pr.Y);
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;  // 16 x 16 threads, 4 x 4 outputs each
  const int64_t m0 = (int64_t)blockIdx.x * BM;
  const int n0 = blockIdx.y * BN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
    for (int l = 0; l < (BM * BK) / kThreads; ++l) {
      const int e = tid + l * kThreads;
      const int r = e / BK, c = e % BK;
      const int64_t gm = m0 + r;
      const int gk = k0 + c;
      As[c][r] = (gm < M && gk < K) ? to_f32(X[gm * K + gk]) : 0.f;
      const int gn = n0 + r;
      Bs[c][r] = (gn < N && gk < K) ? to_f32(W[(int64_t)gn * K + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= N) continue;
      float y = acc[i][j];
      if (pr.bias) y += pr.bias[gn];
      if (R) y += to_f32(R[gm * N + gn]);
      Y[gm * N + gn] = from_f32<TOut>(y);
    }
  }
}

}  // namespace

cudaError_t launch_linear(int in_dtype, int out_f32, const LinearProblem* probs, int nprob,
                          int64_t M, int N, int K, cudaStream_t s) {
  if (M == 0 || nprob == 0) return cudaSuccess;
  dim3 grid((unsigned)((M + BM - 1) / BM), (N + BN - 1) / BN, nprob);
  LinearProblem p1 = nprob > 1 ? probs[1] : probs[0];
  if (in_dtype == NT_BF16) {
    if (out_f32) linear_kernel<bf16, float><<<grid, kThreads, 0, s>>>(probs[0], p1, M, N, K);
    else linear_kernel<bf16, bf16><<<grid, kThreads, 0, s>>>(probs[0], p1, M, N, K);
  } else {
    linear_kernel<float, float><<<grid, kThreads, 0, s>>>(probs[0], p1, M, N, K);
  }
  return cudaGetLastError();
}

}  // namespace nt
