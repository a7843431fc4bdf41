// The sample-weighted squared loss of the single->pair->single block and
// the block's gradients, on CUDA cores (fp32 arithmetic; bf16 or fp32
// inputs; every gradient fp32).
//
// "DanLing NestedTensor" Appendix A.1, Eq. 5:
//     L = sum_i alpha_i ||X~_i||^2 / (C sum N_i) + sum_i beta_i ||P~_i||^2 / (C_p sum N_i^2),
//     alpha_i = 1 + i/B, beta_i = 1.5 - i/(2B)
// (S = 1: the packed layout is a leading one), and the chain rule of Eq. 1
// (section 3.4: the gradient flows from the eager loss back through the
// pair update, the reduction and the projections):
//     dM = dX~ W_g, dW_g = dX~^T M, db_g = sum dX~
//     dP~ = dP~_up + dM[row] / N          (the column mean's backward)
//     A = LN(z) W1^T + b1:  dH = dP~ W2, dA = dH [A > 0], dY = dA W1,
//       dW1 = dA^T LN(z), dW2 = dP~^T ReLU(A), db1 = sum dA, db2 = sum dP~
//     dz = dP~ + LayerNorm backward of dY (dgamma, dbeta on the way)
//     du[row] = sum over the row's cells of dz, dv[col] = sum over the column's
//     dW_a = du^T s, dW_b = dv^T s, ds = dX~ + du W_a + dv W_b
// z is rebuilt from u = s W_a^T and v = s W_b^T, rounded to the I/O dtype as
// the forward rounds it.  Square partitions only.
//
// bf16 with C_z = 128 and H_t a multiple of 128 takes the pair-cell part on
// the tensor cores, through the cells' row-major intermediates:
//   bwd_prep      per cell: LN(z) and dP~ as bf16 rows, the LayerNorm's mean
//                 and rstd
//   tcgen05 GEMMs H = ReLU(LN(z) W1^T + b1) and dA = (dP~ W2) where H > 0
//                 in one kernel (both accumulators per tile), dY = dA W1
//                 (linear_tc), dW1 = dA^T LN(z), dW2 = dP~^T H,
//                 db1, db2 (wgrad_tc: split over the cells)
//   bwd_ln_sums   per 32 x 32 cell item: the LayerNorm backward -> dz in
//                 registers, summed at once into row and column partials of
//                 du and dv (dz is not stored); dgamma, dbeta
//   sums_finish   du, dv from the partials in a fixed order
// The GEMM operands are bf16 (dP~ and dA rounded once); every accumulation
// is fp32.  fp32 I/O and other widths run the CUDA-core kernels below.
//
// Kernels:
//   eq5_partial / eq5_finish     the loss (per pair row, fixed-order final sum)
//                                and, optionally, its gradients dX~, dP~
//   rowmm                         Y = A W (+ A2 W2) (+ R) over the T single rows
//   gram                          G += A^T B over the T single rows (weight gradients)
//   colsum                        column sums over the T single rows (bias gradients)
//   trans_bwd_cells               per 32-cell tile: z, LayerNorm, A, dH, dA, dY over
//                                 64-unit hidden chunks, the LayerNorm backward -> dz;
//                                 dgamma, dbeta, db2
//   trans_bwd_weights             per (hidden chunk, cell range): dW1, dW2, db1
//   pair_rowcol_sum               du (row sums) and dv (column sums) of dz
#include "tc_ptx.cuh"

namespace nt {
namespace {

constexpr int kThreads = 256;
constexpr int kTC = 32;      // cells per tile
constexpr int kHC = 64;      // hidden units per chunk
constexpr int kCmax = 128;   // largest pair width the cell kernels hold
constexpr int kLossBlocks = 1024;   // CTAs (and double partial pairs) of the loss

// Sample of packed cell p: the last b with pair_off[b] <= p (steps past
// samples with no cells), then the row and column within its N x N block.
__device__ __forceinline__ void cell_coords(const int64_t* __restrict__ pair_off, const int32_t* __restrict__ cu,
                                            const int32_t* __restrict__ len, int B, int64_t p, int64_t& row,
                                            int64_t& col, int& n, int* sample = nullptr) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pair_off[mid] <= p) lo = mid; else hi = mid - 1;
  }
  n = len[lo];
  if (sample) *sample = lo;
  const int64_t off = p - pair_off[lo];
  const int64_t a = off / n;
  row = cu[lo] + a;
  col = cu[lo] + (off - a * n);
}

// 16 bytes of the I/O dtype as fp32: 8 bf16 or 4 fp32 values.
__device__ __forceinline__ void load_vec(const bf16* p, float* x) {
  const uint4 q = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void load_vec(const float* p, float* x) {
  const float4 q = *reinterpret_cast<const float4*>(p);
  x[0] = q.x; x[1] = q.y; x[2] = q.z; x[3] = q.w;
}

__device__ __forceinline__ float round_io(float x, float*) { return x; }
__device__ __forceinline__ float round_io(float x, bf16*) { return __bfloat162float(__float2bfloat16_rn(x)); }

// ---------------------------------------------------------------- the loss

// dL/dP~ = gp_b P~ for the cells of sample b: gp_b = 2 beta_b / (C_p P),
// beta_b = 1.5 - b / (2B), formed in double and rounded once to fp32 (the
// loss kernel and the fused loss + backward read the same value).
__device__ __forceinline__ float eq5_pair_scale(int b, int B, int Cp, int64_t P) {
  const double beta = 1.5 - (double)b / (2.0 * B);
  return (float)(2.0 * beta / ((double)Cp * P));
}

// Sum of alpha_b ||X~ row||^2 and of beta_b ||P~ row's cells||^2 over the
// CTA's rows, in double, into partial[blockIdx]; optionally writes
// dX~ = 2 alpha_b X~ / (C T) and dP~ = 2 beta_b P~ / (C_p P).  With the
// cells (zt given) the CTA takes one pair row at a time: X~ row and cells.
// Without them (the pair term then comes from the reduce, eq5_finish's extra
// partials) one warp takes one single row: lane 0 forms the row's weight in
// double, the row's squares are summed in fp32 by a fixed butterfly and
// added once, weighted, so no row waits on a CTA barrier behind one thread's
// fp64 divisions (which are slow here).
constexpr int kLossWarps = kThreads / 32;
template <typename T, bool kCells>
__global__ void __launch_bounds__(kThreads)
eq5_partial_kernel(const T* __restrict__ s_out, const T* __restrict__ zt, const int64_t* __restrict__ row_start,
                   const int32_t* __restrict__ row_sample, int B, int64_t Trows, int64_t P, int C, int Cp,
                   double* __restrict__ partial, float* __restrict__ ds_out, float* __restrict__ dz) {
  __shared__ double red[2][kLossWarps];
  __shared__ double s_ab[2];
  __shared__ float s_g[2];
  double ax = 0.0, ap = 0.0;
  if constexpr (!kCells) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t r = (int64_t)blockIdx.x * kLossWarps + warp; r < Trows; r += (int64_t)gridDim.x * kLossWarps) {
      double alpha = 0.0;
      float gx = 0.f;
      if (lane == 0) {
        alpha = 1.0 + (double)row_sample[r] / B;
        gx = (float)(2.0 * alpha / ((double)C * Trows));
      }
      gx = __shfl_sync(0xffffffffu, gx, 0);
      float sx = 0.f;
      for (int k = lane; k < C; k += 32) {
        const float x = to_f32(s_out[r * C + k]);
        sx = fmaf(x, x, sx);
        if (ds_out) ds_out[r * C + k] = gx * x;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sx += __shfl_xor_sync(0xffffffffu, sx, o);
      if (lane == 0) ax += alpha * (double)sx;
    }
  } else {
    for (int64_t r = blockIdx.x; r < Trows; r += gridDim.x) {
      // the row's weights and gradient scales, formed in double once per row
      if (threadIdx.x == 0) {
        const int b = row_sample[r];
        const double alpha = 1.0 + (double)b / B, beta = 1.5 - (double)b / (2.0 * B);
        s_ab[0] = alpha;
        s_ab[1] = beta;
        s_g[0] = (float)(2.0 * alpha / ((double)C * Trows));
        s_g[1] = eq5_pair_scale(b, B, Cp, P);
      }
      __syncthreads();
      const double alpha = s_ab[0], beta = s_ab[1];
      const float gx = s_g[0], gp = s_g[1];
      __syncthreads();                          // read before thread 0 writes the next row's
      float sx = 0.f;
      for (int k = threadIdx.x; k < C; k += kThreads) {
        const float x = to_f32(s_out[r * C + k]);
        sx += x * x;
        if (ds_out) ds_out[r * C + k] = gx * x;
      }
      ax += alpha * sx;
      // the row's cells: 16-byte loads (Cp is a multiple of 16 bytes' worth
      // of elements, so every row starts on a 16-byte boundary)
      constexpr int V = 16 / sizeof(T);
      const int64_t c0 = row_start[r] * Cp, c1 = row_start[r + 1] * Cp;
      float sp = 0.f;
      for (int64_t e = c0 + (int64_t)threadIdx.x * V; e < c1; e += (int64_t)kThreads * V) {
        float x[V];
        load_vec(zt + e, x);
#pragma unroll
        for (int i = 0; i < V; ++i) sp = fmaf(x[i], x[i], sp);
        if (dz) {
#pragma unroll
          for (int i = 0; i < V; i += 4)
            *reinterpret_cast<float4*>(dz + e + i) =
                make_float4(gp * x[i], gp * x[i + 1], gp * x[i + 2], gp * x[i + 3]);
        }
      }
      ap += beta * sp;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    ax += __shfl_xor_sync(0xffffffffu, ax, o);
    ap += __shfl_xor_sync(0xffffffffu, ap, o);
  }
  if ((threadIdx.x & 31) == 0) { red[0][threadIdx.x >> 5] = ax; red[1][threadIdx.x >> 5] = ap; }
  __syncthreads();
  if (threadIdx.x == 0) {
    double tx = 0.0, tp = 0.0;
    for (int w = 0; w < kThreads / 32; ++w) { tx += red[0][w]; tp += red[1][w]; }
    partial[2 * blockIdx.x] = tx;
    partial[2 * blockIdx.x + 1] = tp;
  }
}

// The partial sums in a fixed order (a pairwise tree over the partial
// index, one block of kLossBlocks threads), then Eq. 5's normalisations.
// extra: nextra further partials of the weighted pair term (the reduce's),
// thread i adding extra[i], extra[i + kLossBlocks], ... in that order.
__global__ void __launch_bounds__(kLossBlocks)
eq5_finish_kernel(const double* __restrict__ partial, int nblocks, int64_t Trows, int64_t P, int C, int Cp,
                  float* __restrict__ loss, const double* __restrict__ extra = nullptr, int nextra = 0) {
  __shared__ double sx[kLossBlocks], sp[kLossBlocks];
  const int i = threadIdx.x;
  sx[i] = i < nblocks ? partial[2 * i] : 0.0;
  double ep = i < nblocks ? partial[2 * i + 1] : 0.0;
  for (int k = i; k < nextra; k += kLossBlocks) ep += extra[k];
  sp[i] = ep;
  __syncthreads();
  for (int w = kLossBlocks / 2; w > 0; w >>= 1) {
    if (i < w) {
      sx[i] += sx[i + w];
      sp[i] += sp[i + w];
    }
    __syncthreads();
  }
  if (i != 0) return;
  const double tx = sx[0], tp = sp[0];
  double l = 0.0;
  if (Trows > 0) l += tx / ((double)C * Trows);
  if (P > 0) l += tp / ((double)Cp * P);
  *loss = (float)l;
}

// ------------------------------------------------------- the single rows side

// Register-tiled fp32 products over the T single rows: a CTA computes a 64 x
// 64 block of the output, each thread a 4 x 4 piece of it, from 16-deep
// slices of both operands staged in shared memory (16 FMAs per two 16-byte
// shared loads).
constexpr int kGT = 64, kGK = 16;

// Y[r, n] = R[r, n] + sum_k A[r, k] W[k, n] + sum_k A2[r, k] W2[k, n]
// (A, A2 fp32 [rows, K]; W, W2 [K, N] row-major in the I/O dtype; R fp32 or
// null; A2 and W2 may be null).  Grid (ceil(rows / 64), ceil(N / 64)): the
// rows on x, whose limit is 2^31 - 1 blocks.
template <typename T>
__global__ void __launch_bounds__(kThreads)
rowmm_kernel(const float* __restrict__ A, const T* __restrict__ W, const float* __restrict__ A2,
             const T* __restrict__ W2, const float* __restrict__ R, int64_t rows, int K, int N,
             float* __restrict__ Y) {
  __shared__ __align__(16) float as[kGK][kGT + 4];   // [k][row]
  __shared__ __align__(16) float ws[kGK][kGT + 4];   // [k][col]
  const int64_t r0 = (int64_t)blockIdx.x * kGT;
  const int n0 = blockIdx.y * kGT;
  const int tr = threadIdx.x >> 4, tc = threadIdx.x & 15;   // rows 4 tr .. 4 tr + 3, columns 4 tc ..
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  // steps of 16 k over one or two (A, W) pairs: A 64 rows x 16 k (four
  // consecutive k per thread, stored k-major), W 16 k x 64 columns (four
  // consecutive columns per thread); the next step's values are loaded into
  // registers while the current step's products run
  const int ksteps = (K + kGK - 1) / kGK, nsteps = (A2 ? 2 : 1) * ksteps;
  const int ra = threadIdx.x >> 2, ka = (threadIdx.x & 3) * 4;
  const int kw = threadIdx.x >> 4, cw = (threadIdx.x & 15) * 4;
  float na[4], nw[4];
  auto fetch = [&](int step) {
    const int pass = step / ksteps, k0 = (step % ksteps) * kGK;
    const float* Ap = pass ? A2 : A;
    const T* Wp = pass ? W2 : W;
    const int64_t r = r0 + ra;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      na[e] = (r < rows && k0 + ka + e < K) ? Ap[r * K + k0 + ka + e] : 0.f;
      nw[e] = (k0 + kw < K && n0 + cw + e < N) ? to_f32(Wp[(int64_t)(k0 + kw) * N + n0 + cw + e]) : 0.f;
    }
  };
  fetch(0);
  for (int step = 0; step < nsteps; ++step) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      as[ka + e][ra] = na[e];
      ws[kw][cw + e] = nw[e];
    }
    __syncthreads();
    if (step + 1 < nsteps) fetch(step + 1);
#pragma unroll
    for (int kk = 0; kk < kGK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&as[kk][4 * tr]);
      const float4 w = *reinterpret_cast<const float4*>(&ws[kk][4 * tc]);
      const float av[4] = {a.x, a.y, a.z, a.w}, wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t r = r0 + 4 * tr + i;
    if (r >= rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + 4 * tc + j;
      if (n < N) Y[r * N + n] = (R ? R[r * N + n] : 0.f) + acc[i][j];
    }
  }
}

// G[i, j] += sum_r A[r, i] B[r, j] over a range of the single rows (A fp32
// [rows, M], B [rows, N] fp32 or I/O dtype): grid (ceil(M / 64), ceil(N /
// 64), splits), one 64 x 64 block of G per CTA and range of rows, fp32
// atomics into G.
template <typename TB>
__global__ void __launch_bounds__(kThreads)
gram_kernel(const float* __restrict__ A, const TB* __restrict__ Bm, int64_t rows, int M, int N, int splits,
            float* __restrict__ G) {
  __shared__ __align__(16) float as[kGK][kGT + 4];   // [row][i]
  __shared__ __align__(16) float bs[kGK][kGT + 4];   // [row][j]
  const int i0 = blockIdx.x * kGT, j0 = blockIdx.y * kGT;
  const int64_t rlo = rows * blockIdx.z / splits, rhi = rows * (blockIdx.z + 1) / splits;
  const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  // 16 rows x 64 columns of each operand per step, four consecutive columns
  // per thread; the next step's values are loaded into registers while the
  // current step's products run
  const int rr = threadIdx.x >> 4, cc = (threadIdx.x & 15) * 4;
  float na[4], nb[4];
  auto fetch = [&](int64_t rb) {
    const int64_t r = rb + rr;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      na[e] = (r < rhi && i0 + cc + e < M) ? A[r * M + i0 + cc + e] : 0.f;
      nb[e] = (r < rhi && j0 + cc + e < N) ? to_f32(Bm[r * N + j0 + cc + e]) : 0.f;
    }
  };
  if (rlo < rhi) fetch(rlo);
  for (int64_t rb = rlo; rb < rhi; rb += kGK) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      as[rr][cc + e] = na[e];
      bs[rr][cc + e] = nb[e];
    }
    __syncthreads();
    if (rb + kGK < rhi) fetch(rb + kGK);
#pragma unroll
    for (int kk = 0; kk < kGK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&as[kk][4 * ti]);
      const float4 b = *reinterpret_cast<const float4*>(&bs[kk][4 * tj]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (i0 + 4 * ti + i < M && j0 + 4 * tj + j < N)
        atomicAdd(G + (int64_t)(i0 + 4 * ti + i) * N + j0 + 4 * tj + j, acc[i][j]);
}

// out[j] += sum_r A[r, j] over a range of rows (fp32 atomics).
__global__ void __launch_bounds__(kThreads)
colsum_kernel(const float* __restrict__ A, int64_t rows, int N, int splits, float* __restrict__ out) {
  const int64_t rlo = rows * blockIdx.y / splits, rhi = rows * (blockIdx.y + 1) / splits;
  for (int j = blockIdx.x * kThreads + threadIdx.x; j < N; j += gridDim.x * kThreads) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};                 // four loads in flight
    int64_t r = rlo;
    for (; r + 4 <= rhi; r += 4) {
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] += A[(r + i) * N + j];
    }
    for (; r < rhi; ++r) acc[0] += A[r * N + j];
    atomicAdd(out + j, (acc[0] + acc[1]) + (acc[2] + acc[3]));
  }
}

// du[t] = sum of dz over the cells of pair row t; dv[t] = sum of dz over
// the cells of column t (the same sample's rows).  One CTA per single row.
__global__ void __launch_bounds__(kThreads)
pair_rowcol_sum_kernel(const float* __restrict__ dz, const int32_t* __restrict__ cu,
                       const int64_t* __restrict__ pair_off, const int32_t* __restrict__ len,
                       const int32_t* __restrict__ row_sample, int64_t Trows, int C, float* __restrict__ du,
                       float* __restrict__ dv) {
  extern __shared__ float part[];            // [2][groups][C]
  const int groups = kThreads / C;
  const int f = threadIdx.x % C, g = threadIdx.x / C;
  for (int64_t t = blockIdx.x; t < Trows; t += gridDim.x) {
    const int b = row_sample[t];
    const int64_t n = len[b], a = t - cu[b], base = pair_off[b];
    float sr = 0.f, sc = 0.f;
    if (g < groups) {
      for (int64_t j = g; j < n; j += groups) {
        sr += dz[(base + a * n + j) * C + f];      // row a, column j
        sc += dz[(base + j * n + a) * C + f];      // row j, column a
      }
      part[g * C + f] = sr;
      part[(groups + g) * C + f] = sc;
    }
    __syncthreads();
    if (g == 0) {
      for (int q = 1; q < groups; ++q) { sr += part[q * C + f]; sc += part[(groups + q) * C + f]; }
      du[t * C + f] = sr;
      dv[t * C + f] = sc;
    }
    __syncthreads();
  }
}

// ------------------------------------------------------- the pair cells side

template <typename T>
struct CellArgs {
  const float* u;            // [T, C] fp32, s W_a^T
  const float* v;            // [T, C] fp32, s W_b^T
  const int64_t* pair_off;
  const int32_t* cu;
  const int32_t* len;
  int B;
  int64_t P;
  int C, H;
  const float* gamma;
  const float* beta;
  float eps;
  const T* W1;               // [H, C]
  const float* b1;           // [H] or null
  const T* W2;               // [C, H]
  const float* dM;           // [T, C] fp32: dX~ W_g
  const float* dz_up;        // [P, C] fp32 or null: gradient reaching P~ from downstream
};

// Loads one 32-cell tile: x-hat of the rebuilt z (rounded to the I/O dtype
// as the forward rounds it) and dP~ = dz_up + dM[row] / N.  Thread t owns
// cell t / 8 and features f = t % 8 + 8 j.  Cells past P get zeros.
template <typename T>
__device__ __forceinline__ void load_tile(const CellArgs<T>& a, int64_t p0, float* xh, float* dpt, float* rstd) {
  const int cell = threadIdx.x >> 3, sub = threadIdx.x & 7;
  const int64_t p = p0 + cell;
  const bool valid = p < a.P;
  float zv[kCmax / 8];
  float s1 = 0.f;
  int64_t row = 0, col = 0;
  int n = 1;
  if (valid) cell_coords(a.pair_off, a.cu, a.len, a.B, p, row, col, n);
  const int nf = (a.C - sub + 7) >> 3;
#pragma unroll
  for (int j = 0; j < kCmax / 8; ++j) {
    zv[j] = 0.f;
    if (j < nf && valid) {
      const int f = sub + 8 * j;
      zv[j] = round_io(a.u[row * a.C + f] + a.v[col * a.C + f], (T*)nullptr);
      s1 += zv[j];
    }
  }
  s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
  s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
  s1 += __shfl_xor_sync(0xffffffffu, s1, 4);
  const float mean = s1 / a.C;
  float s2 = 0.f;
#pragma unroll
  for (int j = 0; j < kCmax / 8; ++j)
    if (j < nf && valid) { const float d = zv[j] - mean; s2 += d * d; }
  s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
  s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
  s2 += __shfl_xor_sync(0xffffffffu, s2, 4);
  const float rs = rsqrtf(s2 / a.C + a.eps);
  const float inv_n = 1.0f / (float)n;
#pragma unroll
  for (int j = 0; j < kCmax / 8; ++j) {
    if (j < nf) {
      const int f = sub + 8 * j;
      xh[cell * a.C + f] = valid ? (zv[j] - mean) * rs : 0.f;
      float d = 0.f;
      if (valid) {
        d = a.dM[row * a.C + f] * inv_n;
        if (a.dz_up) d += a.dz_up[p * a.C + f];
      }
      dpt[cell * a.C + f] = d;
    }
  }
  if (sub == 0) rstd[cell] = valid ? rs : 0.f;
}

// A and dH of hidden chunk c for this thread's cell and its 8 hidden units
// (hg .. hg + 7): A = y W1^T + b1 with y = gamma x-hat + beta, dH = dP~ W2.
template <typename T>
__device__ __forceinline__ void chunk_a_dh(const CellArgs<T>& a, int c, const float* xh, const float* dpt,
                                           const float* w1c, const float* w2c, int cell, int hg, float* av,
                                           float* dh) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    av[i] = a.b1 ? a.b1[c * kHC + hg + i] : 0.f;
    dh[i] = 0.f;
  }
  for (int k = 0; k < a.C; ++k) {
    const float y = fmaf(a.gamma[k], xh[cell * a.C + k], a.beta[k]);
    const float g = dpt[cell * a.C + k];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      av[i] = fmaf(y, w1c[(hg + i) * (a.C + 1) + k], av[i]);
      dh[i] = fmaf(g, w2c[k * (kHC + 1) + hg + i], dh[i]);
    }
  }
}

// W1 rows [64 c, 64 c + 64) as w1c[h][k] (row stride C + 1) and W2 columns
// [64 c, 64 c + 64) as w2c[k][h] (row stride 65), in fp32.
template <typename T>
__device__ __forceinline__ void load_chunk(const CellArgs<T>& a, int c, float* w1c, float* w2c) {
  for (int e = threadIdx.x; e < kHC * a.C; e += kThreads) {
    const int h = e / a.C, k = e % a.C;
    w1c[h * (a.C + 1) + k] = to_f32(a.W1[(int64_t)(c * kHC + h) * a.C + k]);
  }
  for (int e = threadIdx.x; e < kHC * a.C; e += kThreads) {
    const int k = e / kHC, h = e % kHC;
    w2c[k * (kHC + 1) + h] = to_f32(a.W2[(int64_t)k * a.H + c * kHC + h]);
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
trans_bwd_cells_kernel(CellArgs<T> a, float* __restrict__ dz_out, float* __restrict__ dgamma,
                       float* __restrict__ dbeta, float* __restrict__ db2) {
  extern __shared__ float sm[];
  float* xh = sm;                               // [32][C]
  float* dpt = xh + kTC * a.C;                  // [32][C]
  float* dab = dpt + kTC * a.C;                 // [32][64] dA of the chunk
  float* w1c = dab + kTC * kHC;                 // [64][C + 1]
  float* w2c = w1c + kHC * (a.C + 1);           // [C][65]
  float* rstd = w2c + a.C * (kHC + 1);          // [32]
  const int cell = threadIdx.x >> 3, sub = threadIdx.x & 7, hg = sub * 8;
  const int nf = (a.C - sub + 7) >> 3;
  float pg[kCmax / 8], pb[kCmax / 8], pd[kCmax / 8];   // partial dgamma, dbeta, db2 of features sub + 8 j
#pragma unroll
  for (int j = 0; j < kCmax / 8; ++j) pg[j] = pb[j] = pd[j] = 0.f;
  const int nchunk = a.H / kHC;
  const int64_t ntiles = (a.P + kTC - 1) / kTC;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t p0 = tile * kTC;
    __syncthreads();                            // the previous tile's readers are done
    load_tile(a, p0, xh, dpt, rstd);
    float dy[kCmax / 8];
#pragma unroll
    for (int j = 0; j < kCmax / 8; ++j) dy[j] = 0.f;
    for (int c = 0; c < nchunk; ++c) {
      __syncthreads();                          // tile loaded / previous chunk's dA read
      load_chunk(a, c, w1c, w2c);
      __syncthreads();
      float av[8], dh[8];
      chunk_a_dh(a, c, xh, dpt, w1c, w2c, cell, hg, av, dh);
#pragma unroll
      for (int i = 0; i < 8; ++i) dab[cell * kHC + hg + i] = av[i] > 0.f ? dh[i] : 0.f;
      __syncthreads();
      // dY[cell][f] += sum_h dA[cell][h] W1[64 c + h][f], features f = sub + 8 j
      for (int h = 0; h < kHC; ++h) {
        const float d = dab[cell * kHC + h];
#pragma unroll
        for (int j = 0; j < kCmax / 8; ++j)
          if (j < nf) dy[j] = fmaf(d, w1c[h * (a.C + 1) + sub + 8 * j], dy[j]);
      }
    }
    // LayerNorm backward: dz = dP~ + rstd (dx - mean(dx) - xh mean(dx xh)), dx = dY gamma
    const float rs = rstd[cell];
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int j = 0; j < kCmax / 8; ++j)
      if (j < nf) {
        const int f = sub + 8 * j;
        const float dx = dy[j] * a.gamma[f];
        s1 += dx;
        s2 += dx * xh[cell * a.C + f];
      }
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 4);
    s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
    s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
    s2 += __shfl_xor_sync(0xffffffffu, s2, 4);
    const float m1 = s1 / a.C, m2 = s2 / a.C;
    const int64_t p = p0 + cell;
#pragma unroll
    for (int j = 0; j < kCmax / 8; ++j)
      if (j < nf) {
        const int f = sub + 8 * j;
        const float x = xh[cell * a.C + f];
        const float g = dpt[cell * a.C + f];
        if (p < a.P) dz_out[p * a.C + f] = g + rs * (dy[j] * a.gamma[f] - m1 - x * m2);
        pg[j] += dy[j] * x;
        pb[j] += dy[j];
        pd[j] += g;
      }
  }
  // this CTA's feature sums: over the four cells of each warp that share a
  // feature set (lanes sub, sub + 8, sub + 16, sub + 24), then one atomic per warp
#pragma unroll
  for (int j = 0; j < kCmax / 8; ++j) {
    float g = pg[j], b = pb[j], d = pd[j];
    g += __shfl_xor_sync(0xffffffffu, g, 8);  g += __shfl_xor_sync(0xffffffffu, g, 16);
    b += __shfl_xor_sync(0xffffffffu, b, 8);  b += __shfl_xor_sync(0xffffffffu, b, 16);
    d += __shfl_xor_sync(0xffffffffu, d, 8);  d += __shfl_xor_sync(0xffffffffu, d, 16);
    if (j < nf && (threadIdx.x & 31) < 8) {
      const int f = sub + 8 * j;
      atomicAdd(dgamma + f, g);
      atomicAdd(dbeta + f, b);
      atomicAdd(db2 + f, d);
    }
  }
}

// Weight gradients of hidden chunk c = blockIdx.x over the cell range of
// blockIdx.y: dW1[64 c + h][k] += sum_cells dA[h] y[k], dW2[k][64 c + h] +=
// sum_cells dP~[k] ReLU(A)[h], db1 += sum_cells dA.  Each thread keeps its
// outputs (o = t + 256 j of the 64 x C block of each) in registers over
// the range, then adds them with one atomic each.
template <typename T>
__global__ void __launch_bounds__(kThreads)
trans_bwd_weights_kernel(CellArgs<T> a, int splits, float* __restrict__ dW1, float* __restrict__ dW2,
                         float* __restrict__ db1) {
  extern __shared__ float sm[];
  float* xh = sm;                               // [32][C]
  float* dpt = xh + kTC * a.C;                  // [32][C]
  float* yb = dpt + kTC * a.C;                  // [32][C] y = gamma xh + beta
  float* dab = yb + kTC * a.C;                  // [32][64] dA
  float* hb = dab + kTC * kHC;                  // [32][64] ReLU(A)
  float* w1c = hb + kTC * kHC;                  // [64][C + 1]
  float* w2c = w1c + kHC * (a.C + 1);           // [C][65]
  float* rstd = w2c + a.C * (kHC + 1);          // [32]
  const int c = blockIdx.x;
  const int cell = threadIdx.x >> 3, hg = (threadIdx.x & 7) * 8;
  const int64_t ntiles = (a.P + kTC - 1) / kTC;
  const int64_t tlo = ntiles * blockIdx.y / splits, thi = ntiles * (blockIdx.y + 1) / splits;
  const int nout = kHC * a.C;                   // outputs of each of dW1, dW2 for the chunk
  float g1[kHC * kCmax / kThreads], g2[kHC * kCmax / kThreads];
#pragma unroll
  for (int j = 0; j < kHC * kCmax / kThreads; ++j) g1[j] = g2[j] = 0.f;
  float gb = 0.f;                               // db1 of hidden unit threadIdx.x (< 64)
  load_chunk(a, c, w1c, w2c);
  for (int64_t tile = tlo; tile < thi; ++tile) {
    __syncthreads();                            // chunk loaded / previous tile read
    load_tile(a, tile * kTC, xh, dpt, rstd);
    __syncthreads();
    for (int e = threadIdx.x; e < kTC * a.C; e += kThreads) {
      const int f = e % a.C;
      yb[e] = fmaf(a.gamma[f], xh[e], a.beta[f]);
    }
    float av[8], dh[8];
    chunk_a_dh(a, c, xh, dpt, w1c, w2c, cell, hg, av, dh);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      dab[cell * kHC + hg + i] = av[i] > 0.f ? dh[i] : 0.f;
      hb[cell * kHC + hg + i] = fmaxf(av[i], 0.f);
    }
    __syncthreads();
    // dW1 block element o = (h, k) = (o / C, o % C); dW2 block element o = (k, h) = (o / 64, o % 64)
#pragma unroll
    for (int j = 0; j < kHC * kCmax / kThreads; ++j) {
      const int o = threadIdx.x + kThreads * j;
      if (o < nout) {
        const int h1 = o / a.C, k1 = o % a.C;
        const int k2 = o / kHC, h2 = o % kHC;
        float s1 = 0.f, s2 = 0.f;
        for (int q = 0; q < kTC; ++q) {
          s1 = fmaf(dab[q * kHC + h1], yb[q * a.C + k1], s1);
          s2 = fmaf(dpt[q * a.C + k2], hb[q * kHC + h2], s2);
        }
        g1[j] += s1;
        g2[j] += s2;
      }
    }
    if (threadIdx.x < kHC)
      for (int q = 0; q < kTC; ++q) gb += dab[q * kHC + threadIdx.x];
  }
#pragma unroll
  for (int j = 0; j < kHC * kCmax / kThreads; ++j) {
    const int o = threadIdx.x + kThreads * j;
    if (o < nout) {
      const int h1 = o / a.C, k1 = o % a.C;
      const int k2 = o / kHC, h2 = o % kHC;
      atomicAdd(dW1 + (int64_t)(c * kHC + h1) * a.C + k1, g1[j]);
      atomicAdd(dW2 + (int64_t)k2 * a.H + c * kHC + h2, g2[j]);
    }
  }
  if (threadIdx.x < kHC) atomicAdd(db1 + c * kHC + threadIdx.x, gb);
}

template <typename T>
cudaError_t eq5_loss_t(const nt_partition* p, const void* s_out, int C_s, const void* zt, int C_z, float* loss,
                       float* ds_out, float* dz, double* partial, int nblocks, cudaStream_t s) {
  (zt ? eq5_partial_kernel<T, true> : eq5_partial_kernel<T, false>)<<<nblocks, kThreads, 0, s>>>(
      (const T*)s_out, (const T*)zt, p->row_start, p->row_sample, p->B, p->T, p->P, C_s, C_z, partial, ds_out, dz);
  eq5_finish_kernel<<<1, kLossBlocks, 0, s>>>(partial, nblocks, p->T, p->P, C_s, C_z, loss);
  return cudaGetLastError();
}

size_t cell_smem(int C, bool weights) {
  const size_t base = (size_t)kTC * C * 2 + (size_t)kTC * kHC + (size_t)kHC * (C + 1) + (size_t)C * (kHC + 1) + kTC;
  return sizeof(float) * (weights ? base + (size_t)kTC * C + (size_t)kTC * kHC : base);
}

cudaError_t cells_backward_tc(const BlockBwd& q, uint8_t* tcw, unsigned int* status, cudaStream_t s);

template <typename T>
cudaError_t block_backward_t(const BlockBwd& q, unsigned int* status, cudaStream_t s) {
  const nt_partition* p = q.part;
  const int C = q.C_z, Cs = q.C_s;
  const int64_t Trows = p->T;
  cudaError_t e;
  // dM = dX~ W_g ([T, C_s] x [C_s, C_z]); dW_g += dX~^T m; db_g += column sums of dX~
  if (Trows > 0) {
    rowmm_kernel<T><<<dim3((unsigned)((Trows + kGT - 1) / kGT), (C + kGT - 1) / kGT), kThreads, 0, s>>>(
        q.ds_out, (const T*)q.W_g, nullptr, nullptr, nullptr, Trows, Cs, C, q.dM);
    const int splits = (int)min64(64, (Trows + 255) / 256);
    gram_kernel<T><<<dim3((Cs + kGT - 1) / kGT, (C + kGT - 1) / kGT, splits), kThreads, 0, s>>>(q.ds_out, (const T*)q.m,
                                                                                      Trows, Cs, C, splits, q.dW_g);
    // the column sums in splits of about 32 rows: each thread's chain of
    // dependent loads and adds stays short
    const int csplits = (int)min64(1024, (Trows + 31) / 32);
    colsum_kernel<<<dim3((Cs + kThreads - 1) / kThreads, csplits), kThreads, 0, s>>>(q.ds_out, Trows, Cs, csplits,
                                                                                      q.db_g);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // the pair cells: dz, dgamma, dbeta, db2, then dW1, dW2, db1
  if (p->P > 0 && q.tc_ws) {
    if ((e = cells_backward_tc(q, static_cast<uint8_t*>(q.tc_ws), status, s)) != cudaSuccess) return e;
  } else if (p->P > 0) {
    CellArgs<T> a = {q.u, q.v, p->pair_off, p->cu_seqlens, p->lengths, p->B, p->P, C, q.H_t, q.gamma, q.beta,
                     q.eps, (const T*)q.W1, q.b1, (const T*)q.W2, q.dM, q.dz_up};
    const size_t sm1 = cell_smem(C, false), sm2 = cell_smem(C, true);
    e = cudaFuncSetAttribute(trans_bwd_cells_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(trans_bwd_weights_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = (p->P + kTC - 1) / kTC;
    const int grid1 = (int)min64(ntiles, (int64_t)sm_count() * 2);
    trans_bwd_cells_kernel<T><<<grid1, kThreads, sm1, s>>>(a, q.dz, q.dgamma, q.dbeta, q.db2);
    const int nchunk = q.H_t / kHC;
    const int splits = (int)max64(1, min64(ntiles, (int64_t)sm_count() * 2 / nchunk));
    trans_bwd_weights_kernel<T><<<dim3(nchunk, splits), kThreads, sm2, s>>>(a, splits, q.dW1, q.dW2, q.db1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // the broadcast: du, dv (already summed on the tensor-core route); dW_a += du^T s, dW_b += dv^T s;
  // ds = dX~ + du W_a + dv W_b
  if (Trows > 0) {
    if (!(p->P > 0 && q.tc_ws))
      pair_rowcol_sum_kernel<<<(unsigned)min64(Trows, 4096), kThreads, 2 * kThreads * sizeof(float), s>>>(
          q.dz, p->cu_seqlens, p->pair_off, p->lengths, p->row_sample, Trows, C, q.du, q.dv);
    const int splits = (int)min64(64, (Trows + 255) / 256);
    gram_kernel<T><<<dim3((C + kGT - 1) / kGT, (Cs + kGT - 1) / kGT, splits), kThreads, 0, s>>>(q.du, (const T*)q.s, Trows, C,
                                                                                     Cs, splits, q.dW_a);
    gram_kernel<T><<<dim3((C + kGT - 1) / kGT, (Cs + kGT - 1) / kGT, splits), kThreads, 0, s>>>(q.dv, (const T*)q.s, Trows, C,
                                                                                     Cs, splits, q.dW_b);
    rowmm_kernel<T><<<dim3((unsigned)((Trows + kGT - 1) / kGT), (Cs + kGT - 1) / kGT), kThreads, 0, s>>>(
        q.du, (const T*)q.W_a, q.dv, (const T*)q.W_b, q.ds_out, Trows, C, Cs, q.ds);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}


// ------------------------------------------------ the tensor-core route (bf16)

using tc::bf16hi;
using tc::bf16lo;
using tc::bulk_load;
using tc::fence_mbar_init;
using tc::fmul2;
using tc::fadd2;
using tc::ffma2;
using tc::mbar_arrive_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
using tc::mbar_wait_warp;
using tc::pack_bf16x2;

constexpr int kTcC = 128;          // pair width of the tensor-core route
// Per pair row t (sample b, row a: cells p0 + j, j < N contiguous), one CTA
// at a time: 16 threads per cell, thread q owning features 4q..4q+3 and
// 64+4q..64+4q+3, 16 cells per pass and two passes in flight per thread.
// The row's sample, u[t], dM[t] and Eq. 5's scale are read once per row;
// each cell's v, upstream gradient and outputs move 128 to 256 contiguous
// bytes per instruction.  Per cell: LN(z) as two bf16 parts, hi = bf16(y)
// and lo = bf16(y - hi), side by side in a row of 2 C_z (A = [hi | lo] [W1 |
// W1]^T carries y to about 16 bits, so A's sign, the ReLU's decision, is
// that of the fp32 y), and dP~ = dz_up + dM[row] / N as bf16, with z
// rebuilt bf16-rounded as the forward rounds it, and the LayerNorm's mean
// and rstd per cell for the LayerNorm backward.  With zt_up, dz_up is Eq.
// 5's gp_b z~, formed here as the loss forms it.
constexpr int kPrepThreads = 256;
constexpr int kPrepCells = kPrepThreads / 16;   // cells per pass

__global__ void __launch_bounds__(kPrepThreads, 4)
bwd_prep_kernel(const float* __restrict__ u, const float* __restrict__ v, const int64_t* __restrict__ pair_off,
                const int32_t* __restrict__ cu, const int32_t* __restrict__ len,
                const int32_t* __restrict__ row_sample, int B, int64_t T, int64_t P,
                const float* __restrict__ gamma, const float* __restrict__ beta, float eps,
                const float* __restrict__ dM, const float* __restrict__ dz_up, const bf16* __restrict__ zt_up,
                bf16* __restrict__ Y, bf16* __restrict__ dPt, float2* __restrict__ stats) {
  const int lane = threadIdx.x & 31, q = threadIdx.x & 15, slot = threadIdx.x >> 4;
  __shared__ float gsh[kTcC], bsh[kTcC];
  if (threadIdx.x < kTcC) {
    gsh[threadIdx.x] = gamma[threadIdx.x];
    bsh[threadIdx.x] = beta[threadIdx.x];
  }
  __syncthreads();
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    const int b = row_sample[t];
    const int n = len[b];
    const int64_t p0 = pair_off[b] + (t - cu[b]) * n;
    const float inv_n = 1.0f / (float)n;
    // Eq. 5's scale of the sample, formed in double by one lane per warp
    float gp = 0.f;
    if (zt_up) {
      if (lane == 0) gp = eq5_pair_scale(b, B, kTcC, P);
      gp = __shfl_sync(0xffffffffu, gp, 0);
    }
    float ur[8], mr[8];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float4 a4 = *reinterpret_cast<const float4*>(u + t * kTcC + 64 * h + 4 * q);
      const float4 m4 = *reinterpret_cast<const float4*>(dM + t * kTcC + 64 * h + 4 * q);
      ur[4 * h] = a4.x; ur[4 * h + 1] = a4.y; ur[4 * h + 2] = a4.z; ur[4 * h + 3] = a4.w;
      mr[4 * h] = m4.x; mr[4 * h + 1] = m4.y; mr[4 * h + 2] = m4.z; mr[4 * h + 3] = m4.w;
    }
    const int64_t col0 = cu[b];
    for (int j0 = 0; j0 < n; j0 += 2 * kPrepCells) {
      float z[2][8], up[2][8];
      bool ok[2];
      // loads of both cells first
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int j = j0 + c * kPrepCells + slot;
        ok[c] = j < n;
        const int64_t p = p0 + j;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int f = 64 * h + 4 * q;
          float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f), d4 = v4;
          if (ok[c]) {
            v4 = *reinterpret_cast<const float4*>(v + (col0 + j) * kTcC + f);
            if (zt_up) {
              const uint2 w = *reinterpret_cast<const uint2*>(zt_up + p * kTcC + f);
              d4 = make_float4(gp * bf16lo(w.x), gp * bf16hi(w.x), gp * bf16lo(w.y), gp * bf16hi(w.y));
            } else if (dz_up) {
              d4 = *reinterpret_cast<const float4*>(dz_up + p * kTcC + f);
            }
          }
          z[c][4 * h] = v4.x; z[c][4 * h + 1] = v4.y; z[c][4 * h + 2] = v4.z; z[c][4 * h + 3] = v4.w;
          up[c][4 * h] = d4.x; up[c][4 * h + 1] = d4.y; up[c][4 * h + 2] = d4.z; up[c][4 * h + 3] = d4.w;
        }
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float s1 = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          z[c][i] = round_io(ur[i] + z[c][i], (bf16*)nullptr);
          s1 += z[c][i];
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        const float mean = s1 * (1.0f / kTcC);
        float s2 = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float d = z[c][i] - mean;
          s2 = fmaf(d, d, s2);
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        const float rs = rsqrtf(s2 * (1.0f / kTcC) + eps);
        if (!ok[c]) continue;
        const int64_t p = p0 + j0 + c * kPrepCells + slot;
        if (q == 0) stats[p] = make_float2(mean, rs);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t yw[2], lw[2], gw[2];
          const float4 g4 = *reinterpret_cast<const float4*>(gsh + 64 * h + 4 * q);
          const float4 b4 = *reinterpret_cast<const float4*>(bsh + 64 * h + 4 * q);
          const float gm[4] = {g4.x, g4.y, g4.z, g4.w}, bt[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int i = 4 * h + e;
            const float y0 = fmaf((z[c][i] - mean) * rs, gm[e], bt[e]);
            const float y1 = fmaf((z[c][i + 1] - mean) * rs, gm[e + 1], bt[e + 1]);
            const float h0 = round_io(y0, (bf16*)nullptr), h1 = round_io(y1, (bf16*)nullptr);
            yw[e / 2] = pack_bf16x2(y0, y1);
            lw[e / 2] = pack_bf16x2(y0 - h0, y1 - h1);
            gw[e / 2] = pack_bf16x2(fmaf(mr[i], inv_n, up[c][i]), fmaf(mr[i + 1], inv_n, up[c][i + 1]));
          }
          const int f = 64 * h + 4 * q;
          *reinterpret_cast<uint2*>(Y + p * 2 * kTcC + f) = make_uint2(yw[0], yw[1]);
          *reinterpret_cast<uint2*>(Y + p * 2 * kTcC + kTcC + f) = make_uint2(lw[0], lw[1]);
          *reinterpret_cast<uint2*>(dPt + p * kTcC + f) = make_uint2(gw[0], gw[1]);
        }
      }
    }
  }
}

// ---------------------------------------- the LayerNorm and broadcast backward, fused

// The cells of sample b (N = N_b, c = ceil(N / 32)) are cut into c x c items
// of up to 32 rows (a row block) by 32 columns (a column chunk).  Slot bases
// follow from the partition's own scans, so no per-call table is built:
//   item slots of b:   [pair_off[b] / 1024 + cu[b] / 16 + b, the same for b + 1),
//                      at least c^2 of them (a CTA past the first c^2 exits);
//   partial rows of b: from pair_off[b] / 32 + cu[b], at least c N of them:
//                      du partial of (column chunk k, row a) and dv partial of
//                      (row block k, column a) at k N + a.
// Over the batch: at most P / 1024 + T / 16 + B items and P / 32 + T partial
// rows of each kind.
constexpr int kSumTile = 32;

__device__ __forceinline__ int64_t sum_item_base(const int64_t* pair_off, const int32_t* cu, int b) {
  return pair_off[b] / 1024 + cu[b] / 16 + b;
}
__device__ __forceinline__ int64_t sum_part_base(const int64_t* pair_off, const int32_t* cu, int b) {
  return pair_off[b] / kSumTile + cu[b];
}

// One CTA of 512 threads per item slot: 16 threads per column, thread q of
// a column owning features 4q..4q+3 and 64+4q..64+4q+3.  Per row of the
// item, its dY and upstream-gradient cells (32 contiguous cells each) and
// the row's u and dM are staged in shared memory by 1-D bulk copies, two
// rows per copy group and three groups in flight, issued by thread 0 once
// every thread has read the buffer (the group's barrier); the column's v
// stays in registers, so no per-row load waits on memory.  Per row the
// threads rebuild z = bf16(u + v), its LayerNorm mean and rstd, and form
// the LayerNorm backward in fp32 registers,
//     dz = dP~ + (dxhat - mean(dxhat) - xhat mean(dxhat xhat)) rstd,
//     dxhat = dY gamma, dP~ = dz_up + dM[row] / N
// (dz is never stored), and add dz into their column's sum over the item's rows; the
// item's 32 columns are summed per row, first over the warp's two columns
// (an exchange that leaves each lane 4 of the row's 128 features), then
// over the 16 warps in warp order through shared memory.  Fixed orders
// throughout, so du and dv are reproducible.  dgamma += dY xhat and dbeta
// += dY are reduced over the CTA the same way (the warp's two columns, then
// the warps in order), then added with one atomic per feature.  A copy wait that runs out flags the status word and
// ends the CTA once the copies it issued have landed (bounded as well).
constexpr int kSumThreads = 512;
constexpr int kSumWarps = kSumThreads / 32;
constexpr int kSumRows = 2;                                   // rows per copy group
constexpr int kSumBufs = 3;                                   // copy groups in flight
constexpr int kSumHalf = kSumTile * kTcC * 4;                 // 32 cells of fp32 features: 16 KB
constexpr int kSumStatBytes = 512;                             // the row's cells' (mean, rstd), from an even cell
// Staging of one row: dY, the upstream gradient (bf16 z~ on the one-call
// route, else fp32), u[row], dM[row], the statistics.  The row-sum buffer is
// double-buffered (one barrier per copy group instead of two: group k + 1
// writes the half that group k - 1's reduction read before group k's
// barrier); with the larger fp32 upstream that leaves room for two copy
// groups in flight instead of three.
template <bool kUpBf16>
struct SumLayout {
  static constexpr int kUpBytes = kUpBf16 ? kSumTile * kTcC * 2 : kSumHalf;
  static constexpr int kOffUp = kSumHalf;
  static constexpr int kOffU = kSumHalf + kUpBytes;
  static constexpr int kRowBytes = kOffU + 2 * kTcC * 4 + kSumStatBytes;
  static constexpr int kBufs = kUpBf16 ? kSumBufs : 2;       // copy groups in flight
  static constexpr int kRp = 2;                               // row-sum buffers
  static constexpr size_t kRpBytes = (size_t)kSumRows * kSumWarps * kTcC * 4;
  static constexpr size_t kSmem = (size_t)kBufs * kSumRows * kRowBytes + kRp * kRpBytes + kBufs * sizeof(uint64_t);
};
static_assert(kSumRows * kSumWarps * kTcC >= kSumWarps * 2 * kTcC, "the row-sum buffer holds the dgamma/dbeta tail");
static_assert(SumLayout<true>::kSmem <= 227 * 1024 && SumLayout<false>::kSmem <= 227 * 1024, "staging fits");

template <bool kUpBf16>
__global__ void __launch_bounds__(kSumThreads, 1)
bwd_ln_sums_kernel(const float* __restrict__ u, const float* __restrict__ v, const int64_t* __restrict__ pair_off,
                   const int32_t* __restrict__ cu, const int32_t* __restrict__ len, int B,
                   const float* __restrict__ gamma, const float2* __restrict__ stats, const float* __restrict__ dM,
                   const float* __restrict__ dz_up, const bf16* __restrict__ zt_up, const float* __restrict__ dY,
                   float* __restrict__ du_part, float* __restrict__ dv_part, float* __restrict__ dgamma,
                   float* __restrict__ dbeta, unsigned int* status) {
  extern __shared__ __align__(128) uint8_t sum_smem[];
  uint8_t* bufs = sum_smem;                                                        // [buf][row][dY | up]
  using L = SumLayout<kUpBf16>;
  float4* rp0 = reinterpret_cast<float4*>(sum_smem + (size_t)L::kBufs * kSumRows * L::kRowBytes);  // [row][warp][32]
  uint64_t* full = reinterpret_cast<uint64_t*>(sum_smem + (size_t)L::kBufs * kSumRows * L::kRowBytes + L::kRp * L::kRpBytes);
  __shared__ float gs[kTcC];
  __shared__ int abort_flag;
  const int64_t g = blockIdx.x;
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sum_item_base(pair_off, cu, mid) <= g) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int n = len[b];
  const int c = (n + kSumTile - 1) / kSumTile;
  const int64_t local = g - sum_item_base(pair_off, cu, b);
  if (local >= (int64_t)c * c) return;   // CTA-uniform, before any barrier
  const int rb = (int)(local / c), cc = (int)(local % c);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int q = threadIdx.x & 15, slot = threadIdx.x >> 4;
  const int j0 = cc * kSumTile, j = j0 + slot;
  const int ncols = min(n - j0, kSumTile);
  const bool cv = slot < ncols;
  const int a_lo = rb * kSumTile, a_hi = min(n, a_lo + kSumTile);
  const int ngroups = (a_hi - a_lo + kSumRows - 1) / kSumRows;
  const int64_t P0 = pair_off[b], t0 = cu[b], pb0 = sum_part_base(pair_off, cu, b);
  const float inv_n = 1.0f / (float)n;
  const float gp = zt_up ? eq5_pair_scale(b, B, kTcC, pair_off[B]) : 0.f;
  const uint32_t up_cell = zt_up ? kTcC * 2 : (dz_up ? kTcC * 4 : 0);   // upstream bytes per cell
  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kBufs; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  if (threadIdx.x < kTcC) gs[threadIdx.x] = gamma[threadIdx.x];
  __syncthreads();
  // copy group k: rows a_lo + 2k, a_lo + 2k + 1 into buffer k % 3
  auto issue = [&](int k) {
    const int buf = k % L::kBufs, a0 = a_lo + k * kSumRows, nr = min(kSumRows, a_hi - a0);
    // the stats copy starts at the even cell at or before the row's first
    // (8-byte entries, 16-byte copies) and ends at an even cell count: one
    // entry either side at most, inside the padded buffer
    uint32_t tx = 0;
    for (int r = 0; r < nr; ++r) {
      const int64_t p = P0 + (int64_t)(a0 + r) * n + j0;
      tx += (uint32_t)ncols * (kTcC * 4 + up_cell) + 2 * kTcC * 4 + (uint32_t)((((p + ncols + 1) & ~1LL) - (p & ~1LL)) * 8);
    }
    mbar_arrive_expect_tx(&full[buf], tx);
    for (int r = 0; r < nr; ++r) {
      const int64_t p = P0 + (int64_t)(a0 + r) * n + j0;
      uint8_t* dst = bufs + (size_t)(buf * kSumRows + r) * L::kRowBytes;
      const int64_t s0 = p & ~1LL;
      bulk_load(dst + L::kOffU + 2 * kTcC * 4, stats + s0, (uint32_t)((((p + ncols + 1) & ~1LL) - s0) * 8),
                &full[buf]);
      bulk_load(dst + L::kOffU, u + (t0 + a0 + r) * kTcC, kTcC * 4, &full[buf]);
      bulk_load(dst + L::kOffU + kTcC * 4, dM + (t0 + a0 + r) * kTcC, kTcC * 4, &full[buf]);
      bulk_load(dst, dY + p * kTcC, (uint32_t)ncols * kTcC * 4, &full[buf]);
      if (kUpBf16) bulk_load(dst + L::kOffUp, zt_up + p * kTcC, (uint32_t)ncols * up_cell, &full[buf]);
      else if (dz_up) bulk_load(dst + L::kOffUp, dz_up + p * kTcC, (uint32_t)ncols * up_cell, &full[buf]);
    }
  };
  if (threadIdx.x == 0)
    for (int k = 0; k < min(L::kBufs, ngroups); ++k) issue(k);
  float vv[8];          // the column's v, features 4q.. and 64+4q..
  {
    const float* vcol = v + (t0 + (cv ? j : j0)) * kTcC;
    const float4 v0 = *reinterpret_cast<const float4*>(vcol + 4 * q);
    const float4 v1 = *reinterpret_cast<const float4*>(vcol + 64 + 4 * q);
    vv[0] = v0.x; vv[1] = v0.y; vv[2] = v0.z; vv[3] = v0.w;
    vv[4] = v1.x; vv[5] = v1.y; vv[6] = v1.z; vv[7] = v1.w;
  }
  float cs[8], pg[8], pbt[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) { cs[k] = 0.f; pg[k] = 0.f; pbt[k] = 0.f; }
  const bool hi4 = (lane & 16) != 0;
  int k = 0;
  for (; k < ngroups; ++k) {
    const int buf = k % L::kBufs, a0 = a_lo + k * kSumRows, nr = min(kSumRows, a_hi - a0);
    float4* rp = rp0 + (size_t)(k % L::kRp) * (L::kRpBytes / sizeof(float4));
    // warp-uniform: the row arithmetic below has full-warp shuffles
    if (mbar_wait_warp(&full[buf], (uint32_t)(k / L::kBufs) & 1, &abort_flag, status)) {
      for (int r = 0; r < nr; ++r) {
        const uint8_t* sr = bufs + (size_t)(buf * kSumRows + r) * L::kRowBytes;
        const float* su = reinterpret_cast<const float*>(sr + L::kOffU);
        const float* sdm = su + kTcC;
        const int64_t pr0 = P0 + (int64_t)(a0 + r) * n + j0;      // the row's first cell
        const float2 st = reinterpret_cast<const float2*>(sdm + kTcC)[(pr0 & 1) + (cv ? slot : 0)];
        float dy[8], up[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) { dy[e] = 0.f; up[e] = 0.f; }
        if (cv) {
          const float4 y0 = *reinterpret_cast<const float4*>(sr + slot * kTcC * 4 + 16 * q);
          const float4 y1 = *reinterpret_cast<const float4*>(sr + slot * kTcC * 4 + 256 + 16 * q);
          dy[0] = y0.x; dy[1] = y0.y; dy[2] = y0.z; dy[3] = y0.w;
          dy[4] = y1.x; dy[5] = y1.y; dy[6] = y1.z; dy[7] = y1.w;
          if (kUpBf16) {
            const uint2 w0 = *reinterpret_cast<const uint2*>(sr + L::kOffUp + slot * kTcC * 2 + 8 * q);
            const uint2 w1 = *reinterpret_cast<const uint2*>(sr + L::kOffUp + slot * kTcC * 2 + 128 + 8 * q);
            up[0] = gp * bf16lo(w0.x); up[1] = gp * bf16hi(w0.x); up[2] = gp * bf16lo(w0.y); up[3] = gp * bf16hi(w0.y);
            up[4] = gp * bf16lo(w1.x); up[5] = gp * bf16hi(w1.x); up[6] = gp * bf16lo(w1.y); up[7] = gp * bf16hi(w1.y);
          } else if (dz_up) {
            const float4 u0 = *reinterpret_cast<const float4*>(sr + L::kOffUp + slot * kTcC * 4 + 16 * q);
            const float4 u1 = *reinterpret_cast<const float4*>(sr + L::kOffUp + slot * kTcC * 4 + 256 + 16 * q);
            up[0] = u0.x; up[1] = u0.y; up[2] = u0.z; up[3] = u0.w;
            up[4] = u1.x; up[5] = u1.y; up[6] = u1.z; up[7] = u1.w;
          }
        }
        // z rebuilt as the forward rounds it, x-hat from its kept mean and
        // rstd.  Elementwise work in fp32 pairs; a column past the sample's
        // end takes rstd = 1/N = 0, so its x-hat, dP~ and dz are exactly 0
        // (dy and up are 0 there already).
        float xh[8], gv[8], dx[8];
        {
          const float4 a0 = *reinterpret_cast<const float4*>(su + 4 * q);
          const float4 a1 = *reinterpret_cast<const float4*>(su + 64 + 4 * q);
          const float4 m0 = *reinterpret_cast<const float4*>(sdm + 4 * q);
          const float4 m1v = *reinterpret_cast<const float4*>(sdm + 64 + 4 * q);
          const float4 g0 = *reinterpret_cast<const float4*>(gs + 4 * q);
          const float4 g1 = *reinterpret_cast<const float4*>(gs + 64 + 4 * q);
          const float ua[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          const float ma[8] = {m0.x, m0.y, m0.z, m0.w, m1v.x, m1v.y, m1v.z, m1v.w};
          const float ga[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          const float in_c = cv ? inv_n : 0.f;
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            float z0, z1;
            fadd2(ua[i], ua[i + 1], vv[i], vv[i + 1], z0, z1);
            const uint32_t zw = pack_bf16x2(z0, z1);
            xh[i] = bf16lo(zw);
            xh[i + 1] = bf16hi(zw);
            ffma2(ma[i], ma[i + 1], in_c, in_c, up[i], up[i + 1], gv[i], gv[i + 1]);
            fmul2(dy[i], dy[i + 1], ga[i], ga[i + 1], dx[i], dx[i + 1]);
          }
        }
        const float mean = st.x, rs = cv ? st.y : 0.f;
        float m1a = 0.f, m1b = 0.f, m2a = 0.f, m2b = 0.f;
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          fadd2(xh[i], xh[i + 1], -mean, -mean, xh[i], xh[i + 1]);
          fmul2(xh[i], xh[i + 1], rs, rs, xh[i], xh[i + 1]);
          fadd2(m1a, m1b, dx[i], dx[i + 1], m1a, m1b);
          ffma2(dx[i], dx[i + 1], xh[i], xh[i + 1], m2a, m2b, m2a, m2b);
        }
        float m1 = m1a + m1b, m2 = m2a + m2b;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
          m1 += __shfl_xor_sync(0xffffffffu, m1, o);
          m2 += __shfl_xor_sync(0xffffffffu, m2, o);
        }
        m1 *= 1.0f / kTcC;
        m2 *= 1.0f / kTcC;
        float out[8];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          float t0, t1;
          fadd2(dx[i], dx[i + 1], -m1, -m1, t0, t1);                  // dxhat - mean(dxhat)
          ffma2(xh[i], xh[i + 1], -m2, -m2, t0, t1, t0, t1);          // - xhat mean(dxhat xhat)
          ffma2(t0, t1, rs, rs, gv[i], gv[i + 1], out[i], out[i + 1]);  // dP~ + (...) rstd
          fadd2(cs[i], cs[i + 1], out[i], out[i + 1], cs[i], cs[i + 1]);
          ffma2(dy[i], dy[i + 1], xh[i], xh[i + 1], pg[i], pg[i + 1], pg[i], pg[i + 1]);
          fadd2(pbt[i], pbt[i + 1], dy[i], dy[i + 1], pbt[i], pbt[i + 1]);
        }
        // the row over the warp's two columns (lane bit 4): the even column
        // keeps features 4q.. and adds the odd column's copy, the odd column
        // keeps 64+4q.. and adds the even column's
        float r4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float send = hi4 ? out[i] : out[i + 4];
          r4[i] = (hi4 ? out[i + 4] : out[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
        }
        rp[(r * kSumWarps + warp) * (kTcC / 4) + (hi4 ? 16 : 0) + q] = make_float4(r4[0], r4[1], r4[2], r4[3]);
      }
    }
    __syncthreads();
    if (abort_flag) break;   // read after the barrier: the same in every thread
    if (threadIdx.x == 0 && k + L::kBufs < ngroups) issue(k + L::kBufs);   // buffer k % kBufs has been read
    {
      const int f = threadIdx.x & (kTcC - 1), r = threadIdx.x / kTcC;
      if (r < nr) {
        const float* rr = reinterpret_cast<const float*>(rp + r * kSumWarps * (kTcC / 4));
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kSumWarps; ++w) acc += rr[w * kTcC + f];
        du_part[(pb0 + (int64_t)cc * n + a0 + r) * kTcC + f] = acc;
      }
    }
  }
  if (abort_flag) {
    // let the copies still in flight land before the CTA's shared memory goes
    if (threadIdx.x == 0)
      for (int k2 = k; k2 < min(k + L::kBufs, ngroups); ++k2)
        mbar_wait(&full[k2 % L::kBufs], (uint32_t)(k2 / L::kBufs) & 1, nullptr, status);
    return;
  }
  if (cv) {
    float* o = dv_part + (pb0 + (int64_t)rb * n + j) * kTcC;
    *reinterpret_cast<float4*>(o + 4 * q) = make_float4(cs[0], cs[1], cs[2], cs[3]);
    *reinterpret_cast<float4*>(o + 64 + 4 * q) = make_float4(cs[4], cs[5], cs[6], cs[7]);
  }
  // dgamma and dbeta over the item: the warp's two columns first (lane bit
  // 4), then the 16 warps in warp order through the row-sum buffer (once
  // the last group's reduction has read it), then one atomic per feature
  __syncthreads();
  float* red = reinterpret_cast<float*>(rp0);         // [warp][dgamma | dbeta][C]
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    pg[i] += __shfl_xor_sync(0xffffffffu, pg[i], 16);
    pbt[i] += __shfl_xor_sync(0xffffffffu, pbt[i], 16);
  }
  if (!hi4) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int f = 64 * (i >> 2) + 4 * q + (i & 3);
      red[(warp * 2) * kTcC + f] = pg[i];
      red[(warp * 2 + 1) * kTcC + f] = pbt[i];
    }
  }
  __syncthreads();
  if (threadIdx.x < 2 * kTcC) {
    const int which = threadIdx.x / kTcC, f = threadIdx.x % kTcC;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kSumWarps; ++w) acc += red[(w * 2 + which) * kTcC + f];
    atomicAdd((which ? dbeta : dgamma) + f, acc);
  }
}

// du[t] = sum over column chunks k of the du partials of row t, dv[t] = sum
// over row blocks k of the dv partials of column t, in k order.
__global__ void __launch_bounds__(kThreads)
sums_finish_kernel(const float* __restrict__ du_part, const float* __restrict__ dv_part,
                   const int64_t* __restrict__ pair_off, const int32_t* __restrict__ cu,
                   const int32_t* __restrict__ len, const int32_t* __restrict__ row_sample, int64_t T,
                   float* __restrict__ du, float* __restrict__ dv) {
  for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < T * kTcC; e += (int64_t)gridDim.x * kThreads) {
    const int64_t t = e / kTcC;
    const int f = (int)(e % kTcC);
    const int b = row_sample[t];
    const int n = len[b];
    const int c = (n + kSumTile - 1) / kSumTile;
    const int64_t base = sum_part_base(pair_off, cu, b) + (t - cu[b]);
    float su = 0.f, sv = 0.f;
    for (int k = 0; k < c; ++k) {
      su += du_part[(base + (int64_t)k * n) * kTcC + f];
      sv += dv_part[(base + (int64_t)k * n) * kTcC + f];
    }
    du[e] = su;
    dv[e] = sv;
  }
}

// out[c][r] = in[r][c] for a bf16 [R, Cc] matrix (the weights, once per call).
__global__ void transpose_bf16_kernel(const bf16* __restrict__ in, int R, int Cc, bf16* __restrict__ out) {
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < (int64_t)R * Cc;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(e / Cc), c = (int)(e % Cc);
    out[(int64_t)c * R + r] = in[e];
  }
}

// out[r] = [in[r] | in[r]] for a bf16 [R, Cc] matrix: W1 beside itself.
__global__ void twice_bf16_kernel(const bf16* __restrict__ in, int R, int Cc, bf16* __restrict__ out) {
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < (int64_t)R * Cc;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / Cc, c = e % Cc;
    out[r * 2 * Cc + c] = in[e];
    out[r * 2 * Cc + Cc + c] = in[e];
  }
}

// Byte offsets of the route's buffers in the workspace past the CUDA-core
// route's (each 256-byte aligned).
struct TcLayout {
  size_t Y, dPt, H, dA, stats, W1t, W2t, W1x2, du_part, dv_part, wg, end;
};
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
TcLayout tc_layout(int64_t P, int64_t T, int C, int H) {
  TcLayout L;
  size_t o = 0;
  L.Y = o; o = align256(o + (size_t)P * 2 * C * 2);   // [hi | lo] rows
  L.dPt = o; o = align256(o + (size_t)P * C * 2);
  L.H = o; o = align256(o + (size_t)P * H * 2);
  L.dA = o; o = align256(o + (size_t)P * H * 2);
  L.stats = o; o = align256(o + (size_t)P * 8 + 16);   // one entry of slack for the 16-byte copies
  L.W1t = o; o = align256(o + (size_t)C * H * 2);
  L.W2t = o; o = align256(o + (size_t)C * H * 2);
  L.W1x2 = o; o = align256(o + (size_t)2 * C * H * 2);
  const size_t part_rows = (size_t)(P / kSumTile + T + 1);
  L.du_part = o; o = align256(o + part_rows * C * 4);
  L.dv_part = o; o = align256(o + part_rows * C * 4);
  L.wg = o;
  const size_t w1 = wgrad_tc_workspace_bytes(P, H, C), w2 = wgrad_tc_workspace_bytes(P, C, H);
  o = align256(o + (w1 > w2 ? w1 : w2));
  L.end = o;
  return L;
}

cudaError_t cells_backward_tc(const BlockBwd& q, uint8_t* tcw, unsigned int* status, cudaStream_t s) {
  const nt_partition* p = q.part;
  const int C = q.C_z, H = q.H_t;
  const int64_t P = p->P;
  const TcLayout L = tc_layout(P, p->T, C, H);
  bf16* Y = reinterpret_cast<bf16*>(tcw + L.Y);
  bf16* dPt = reinterpret_cast<bf16*>(tcw + L.dPt);
  bf16* Hm = reinterpret_cast<bf16*>(tcw + L.H);
  bf16* dA = reinterpret_cast<bf16*>(tcw + L.dA);
  bf16* W1t = reinterpret_cast<bf16*>(tcw + L.W1t);
  bf16* W2t = reinterpret_cast<bf16*>(tcw + L.W2t);
  bf16* W1x2 = reinterpret_cast<bf16*>(tcw + L.W1x2);
  float2* stats = reinterpret_cast<float2*>(tcw + L.stats);
  float* du_part = reinterpret_cast<float*>(tcw + L.du_part);
  float* dv_part = reinterpret_cast<float*>(tcw + L.dv_part);
  void* wg = tcw + L.wg;
  const unsigned gt = (unsigned)min64(((int64_t)C * H + 255) / 256, 1024);
  transpose_bf16_kernel<<<gt, 256, 0, s>>>((const bf16*)q.W1, H, C, W1t);   // W1 [H, C] -> [C, H]
  transpose_bf16_kernel<<<gt, 256, 0, s>>>((const bf16*)q.W2, C, H, W2t);   // W2 [C, H] -> [H, C]
  twice_bf16_kernel<<<gt, 256, 0, s>>>((const bf16*)q.W1, H, C, W1x2);       // [W1 | W1], [H, 2C]
  bwd_prep_kernel<<<(unsigned)min64(p->T, (int64_t)sm_count() * 16), kPrepThreads, 0, s>>>(
      q.u, q.v, p->pair_off, p->cu_seqlens, p->lengths, p->row_sample, p->B, p->T, P, q.gamma, q.beta, q.eps, q.dM,
      q.dz_up, (const bf16*)q.zt_up, Y, dPt, stats);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // H = ReLU([hi | lo] [W1 | W1]^T + b1) and dA = (dP~ W2) where H > 0, per tile in one
  // kernel; dY = dA W1 (into the dz buffer)
  if ((e = launch_linear_tc_dual(Y, W1x2, q.b1, dPt, W2t, Hm, dA, P, H, 2 * C, C, status, s)) != cudaSuccess)
    return e;
  LinearProblem g3 = {dA, W1t, nullptr, nullptr, q.dz};
  if ((e = launch_linear_tc(1, &g3, 1, P, C, H, status, s)) != cudaSuccess) return e;
  // the LayerNorm backward and the broadcast's: du, dv (dz is not stored), dgamma, dbeta
  const int64_t items = P / 1024 + p->T / 16 + p->B;
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const bool up_bf16 = q.zt_up != nullptr;
  auto sums = up_bf16 ? bwd_ln_sums_kernel<true> : bwd_ln_sums_kernel<false>;
  const size_t sums_smem = up_bf16 ? SumLayout<true>::kSmem : SumLayout<false>::kSmem;
  if ((e = cudaFuncSetAttribute(sums, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sums_smem)) != cudaSuccess)
    return e;
  sums<<<(unsigned)items, kSumThreads, sums_smem, s>>>(
      q.u, q.v, p->pair_off, p->cu_seqlens, p->lengths, p->B, q.gamma, stats, q.dM, q.dz_up, (const bf16*)q.zt_up,
      q.dz, du_part, dv_part, q.dgamma, q.dbeta, status);
  sums_finish_kernel<<<(unsigned)min64((p->T * C + kThreads - 1) / kThreads, (int64_t)sm_count() * 8), kThreads, 0,
                       s>>>(du_part, dv_part, p->pair_off, p->cu_seqlens, p->lengths, p->row_sample, p->T, q.du,
                            q.dv);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // dW1 = dA^T LN(z) (the hi part, every other C_z block of the rows), db1 =
  // sum dA; dW2 = dP~^T H, db2 = sum dP~
  if ((e = launch_wgrad_tc(dA, H, Y, 2 * C, P, H, C, q.dW1, q.db1, wg, status, s)) != cudaSuccess) return e;
  return launch_wgrad_tc(dPt, C, Hm, H, P, C, H, q.dW2, q.db2, wg, status, s);
}

}  // namespace

bool block_bwd_supported(int C_z, int H_t) { return C_z >= 8 && C_z <= kCmax && H_t >= kHC && H_t % kHC == 0; }

bool block_bwd_tc(nt_dtype dt, int64_t P, int C_z, int H_t) {
  return dt == NT_BF16 && C_z == kTcC && H_t % 128 == 0 && P > 0 && linear_tc_supported(NT_BF16, P, H_t, C_z) &&
         linear_tc_supported(NT_BF16, P, C_z, H_t) && wgrad_tc_supported(P, H_t, C_z);
}

size_t block_bwd_workspace_bytes(nt_dtype dt, int64_t T, int64_t P, int C_z, int H_t) {
  const size_t base = align256((size_t)(5 * T + P) * (size_t)C_z * sizeof(float));
  return block_bwd_tc(dt, P, C_z, H_t) ? base + tc_layout(P, T, C_z, H_t).end : base;
}

cudaError_t launch_eq5_loss(nt_dtype dt, const nt_partition* p, const void* s_out, int C_s, const void* zt, int C_z,
                            float* loss, float* ds_out, float* dz, void* workspace, cudaStream_t s) {
  const int nblocks = (int)max64(1, min64(p->T, kLossBlocks));
  double* partial = static_cast<double*>(workspace);
  return dt == NT_BF16 ? eq5_loss_t<bf16>(p, s_out, C_s, zt, C_z, loss, ds_out, dz, partial, nblocks, s)
                       : eq5_loss_t<float>(p, s_out, C_s, zt, C_z, loss, ds_out, dz, partial, nblocks, s);
}

size_t eq5_loss_workspace_bytes() { return sizeof(double) * 2 * kLossBlocks; }

cudaError_t launch_eq5_loss_rows(nt_dtype dt, const nt_partition* p, const void* s_out, int C_s, int C_z,
                                 float* loss, const double* pair_sq, int npair, void* workspace, cudaStream_t s) {
  const int nblocks = (int)max64(1, min64(p->T, kLossBlocks));
  double* partial = static_cast<double*>(workspace);
  if (dt == NT_BF16)
    eq5_partial_kernel<bf16, false><<<nblocks, kThreads, 0, s>>>(
        (const bf16*)s_out, nullptr, p->row_start, p->row_sample, p->B, p->T, p->P, C_s, C_z, partial, nullptr,
        nullptr);
  else
    eq5_partial_kernel<float, false><<<nblocks, kThreads, 0, s>>>(
        (const float*)s_out, nullptr, p->row_start, p->row_sample, p->B, p->T, p->P, C_s, C_z, partial, nullptr,
        nullptr);
  eq5_finish_kernel<<<1, kLossBlocks, 0, s>>>(partial, nblocks, p->T, p->P, C_s, C_z, loss, pair_sq, npair);
  return cudaGetLastError();
}

cudaError_t launch_block_backward(nt_dtype dt, const BlockBwd& q, unsigned int* status, cudaStream_t s) {
  return dt == NT_BF16 ? block_backward_t<bf16>(q, status, s) : block_backward_t<float>(q, status, s);
}

}  // namespace nt
