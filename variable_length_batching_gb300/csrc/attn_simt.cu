// Variable-length attention on fp32 CUDA cores ("Variable-length attention
// and data packing", "What it is" / "How it works"): query token t of segment
// i attends only to keys in [cu_i, cu_{i+1}), with an online (running-max)
// softmax so no score matrix is stored.  Used for the fp32 mode and head
// widths the tensor-core kernel does not cover.
//
// A CTA takes kBQ consecutive query tokens of the packed stream and one head;
// its key range is the union of the key segments those tokens attend to, and
// each thread skips the keys outside its own range (the block-diagonal mask of
// the page's "Core math" (C), applied per key instead of materialised).  For
// cross-attention the key segment of query segment b is [cu_k[b], cu_k[b+1])
// ("DanLing NestedTensor" section 3.3: the output takes the query structure);
// with the causal flag a query's range also ends at its diagonal, aligned to
// the segment's bottom-right corner.  A query with no key gets zeros and
// lse = -inf.
#include "nt_common.cuh"

namespace nt {
namespace {

constexpr int kBQ = 64;   // queries (= threads) per CTA

__device__ __forceinline__ int segment_of(const int32_t* __restrict__ cu, int B, int t) {
  // last i with cu[i] <= t; empty segments are skipped because cu[i+1] > t
  int lo = 0, hi = B;  // answer in [0, B-1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// keys staged in shared memory per step (K and V tiles, fp32, <= 32 KB)
template <int D> struct KeyTile { static constexpr int value = D > 64 ? 32 : 64; };

template <typename T, int D>
__global__ void __launch_bounds__(kBQ)
attn_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                 const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k, int B, int64_t Tq,
                 int64_t Tk, int H, float scale, bool causal, T* __restrict__ o, float* __restrict__ lse,
                 unsigned int* status) {
  constexpr int kBK = KeyTile<D>::value;
  __shared__ float Ks[kBK][D];
  __shared__ float Vs[kBK][D];
  __shared__ int range_lo, range_hi;
  const int h = blockIdx.y;
  const int64_t t = (int64_t)blockIdx.x * kBQ + threadIdx.x;
  bool valid = t < Tq;
  int my_lo = 0x7fffffff, my_hi = -1;
  if (threadIdx.x == 0) { range_lo = 0x7fffffff; range_hi = -1; }
  __syncthreads();
  float qr[D];
  if (valid) {
    const int seg = segment_of(cu_q, B, (int)t);
    const int qlo = cu_q[seg], qhi = cu_q[seg + 1];
    const int klo = cu_k[seg], khi = cu_k[seg + 1];
    if (qlo < 0 || qlo > t || qhi <= t || qhi > Tq || klo < 0 || khi < klo || khi > Tk) {
      // offsets inconsistent with the token counts: flag it and touch no key or output
      flag_device(status, kDevCheck);
      valid = false;
    } else {
      my_lo = klo;
      my_hi = khi;
      if (causal) {
        // key index j sees query index i when j <= i + (n_k - n_q)
        const int64_t last = (int64_t)klo + (t - qlo) + (int64_t)(khi - klo) - (qhi - qlo);
        my_hi = (int)max((int64_t)klo, min((int64_t)khi, last + 1));
      }
    }
  }
  if (valid) {
    if (my_hi > my_lo) {
      atomicMin(&range_lo, my_lo);
      atomicMax(&range_hi, my_hi);
    }
    const T* qp = q + (t * H + h) * D;
#pragma unroll
    for (int c = 0; c < D; ++c) qr[c] = to_f32(qp[c]) * scale;
  }
  __syncthreads();
  const int lo = range_lo, hi = range_hi;
  float mrun = -INFINITY, l = 0.f;
  float acc[D];
#pragma unroll
  for (int c = 0; c < D; ++c) acc[c] = 0.f;
  for (int kb = lo; kb < hi; kb += kBK) {
    const int nk = min(kBK, hi - kb);
    for (int e = threadIdx.x; e < nk * D; e += kBQ) {
      const int j = e / D, c = e % D;
      const int64_t src = ((int64_t)(kb + j) * H + h) * D + c;
      Ks[j][c] = to_f32(k[src]);
      Vs[j][c] = to_f32(v[src]);
    }
    __syncthreads();
    if (valid) {
      const int j0 = max(my_lo - kb, 0), j1 = min(my_hi - kb, nk);
      for (int j = j0; j < j1; ++j) {
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < D; ++c) s = fmaf(qr[c], Ks[j][c], s);
        if (s > mrun) {
          const float corr = expf(mrun - s);   // exp(-inf) = 0 on the first key
          l *= corr;
#pragma unroll
          for (int c = 0; c < D; ++c) acc[c] *= corr;
          mrun = s;
        }
        const float p = expf(s - mrun);
        l += p;
#pragma unroll
        for (int c = 0; c < D; ++c) acc[c] = fmaf(p, Vs[j][c], acc[c]);
      }
    }
    __syncthreads();
  }
  if (valid) {
    const float inv = l > 0.f ? 1.0f / l : 0.f;     // no visible key: zeros
    T* op = o + (t * H + h) * D;
#pragma unroll
    for (int c = 0; c < D; ++c) op[c] = from_f32<T>(acc[c] * inv);
    if (lse) lse[(int64_t)h * Tq + t] = l > 0.f ? mrun + logf(l) : -INFINITY;
  }
}

template <int D>
cudaError_t launch_d(nt_dtype dt, const AttnProblem& p, unsigned int* status, cudaStream_t s) {
  dim3 grid((unsigned)((p.T_q + kBQ - 1) / kBQ), p.H);
  if (dt == NT_BF16)
    attn_simt_kernel<bf16, D><<<grid, kBQ, 0, s>>>((const bf16*)p.q, (const bf16*)p.k, (const bf16*)p.v,
                                                  p.cu_q, p.cu_k, p.B, p.T_q, p.T_k, p.H, p.scale, p.causal,
                                                  (bf16*)p.o, p.lse, status);
  else
    attn_simt_kernel<float, D><<<grid, kBQ, 0, s>>>((const float*)p.q, (const float*)p.k, (const float*)p.v,
                                                   p.cu_q, p.cu_k, p.B, p.T_q, p.T_k, p.H, p.scale, p.causal,
                                                   (float*)p.o, p.lse, status);
  return cudaGetLastError();
}

}  // namespace

bool attn_simt_supported(int d) { return d == 32 || d == 64 || d == 128; }

cudaError_t launch_attn_simt(nt_dtype dt, const AttnProblem& p, unsigned int* status, cudaStream_t s) {
  if (p.T_q == 0) return cudaSuccess;
  switch (p.d) {
    case 32: return launch_d<32>(dt, p, status, s);
    case 64: return launch_d<64>(dt, p, status, s);
    case 128: return launch_d<128>(dt, p, status, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nt
