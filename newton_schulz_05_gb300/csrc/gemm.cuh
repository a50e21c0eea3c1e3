// Batched fp32 SIMT GEMMs of the dense Newton-Schulz path in the fp32 mode
// (the fp16 mode runs on the tcgen05 tensor cores, tc_gemm.cu).
// D[b] = alpha * A[b] op(B[b]) + beta * C[b], all matrices row-major inside
// one per-slice workspace region (matrix b sits at base + b*stride):
//   A  [M, K]                      (K contiguous)
//   B  [N, K] for gemm_nt (K contiguous) or [K, N] for gemm_nn (N contiguous)
//   C  [M, N] (may be null when beta == 0), D [M, N]
// M and N must be multiples of 128 and K a multiple of 32 (the dense working
// buffers are zero-padded to multiples of 128).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "common.cuh"

namespace muon {

struct GemmBatch {
  int batch = 1;
  size_t stride_bytes = 0;
  int64_t M = 0, N = 0, K = 0;
  const void* A = nullptr;
  const void* B = nullptr;
  const void* C = nullptr;
  void* D = nullptr;
  float alpha = 1.f, beta = 0.f;
};

namespace gemm_detail {

template <typename T> __device__ __forceinline__ void store_out(T* p, float v) { *p = from_f<T>(v); }

// fp32 SIMT: 64x64x16 tiles, 256 threads, 4x4 outputs per thread.
template <bool BK, typename OT>
__global__ void __launch_bounds__(256) sgemm_kernel(GemmBatch p) {
  constexpr int BM = 64, BN = 64, BKT = 16;
  __shared__ __align__(16) float As[BKT][BM + 4];
  __shared__ __align__(16) float Bs[BKT][BN + 4];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
  const size_t boff = (size_t)blockIdx.z * p.stride_bytes;
  const float* A = reinterpret_cast<const float*>((const char*)p.A + boff);
  const float* B = reinterpret_cast<const float*>((const char*)p.B + boff);
  const int64_t K = p.K, N = p.N;
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < K; k0 += BKT) {
    {
      const int row = tid >> 2, kc = (tid & 3) * 4;
      const float4 a = *reinterpret_cast<const float4*>(A + (m0 + row) * K + k0 + kc);
      As[kc + 0][row] = a.x; As[kc + 1][row] = a.y; As[kc + 2][row] = a.z; As[kc + 3][row] = a.w;
      if (BK) {
        const float4 b = *reinterpret_cast<const float4*>(B + (n0 + row) * K + k0 + kc);
        Bs[kc + 0][row] = b.x; Bs[kc + 1][row] = b.y; Bs[kc + 2][row] = b.z; Bs[kc + 3][row] = b.w;
      } else {
        const int kr = tid >> 4, nc = (tid & 15) * 4;
        *reinterpret_cast<float4*>(&Bs[kr][nc]) =
            *reinterpret_cast<const float4*>(B + (k0 + kr) * N + n0 + nc);
      }
    }
    __syncthreads();
    #pragma unroll
    for (int kk = 0; kk < BKT; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
      #pragma unroll
      for (int i = 0; i < 4; ++i)
        #pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  const float* C = p.C ? reinterpret_cast<const float*>((const char*)p.C + boff) : nullptr;
  OT* D = reinterpret_cast<OT*>((char*)p.D + boff);
  #pragma unroll
  for (int i = 0; i < 4; ++i)
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t row = m0 + ty * 4 + i, col = n0 + tx * 4 + j;
      float v = p.alpha * acc[i][j];
      if (C && p.beta != 0.f) v = fmaf(p.beta, C[row * N + col], v);
      store_out(D + row * N + col, v);
    }
}

}  // namespace gemm_detail

template <typename IT, typename OT>
inline cudaError_t gemm_launch(const GemmBatch& p, bool bk, cudaStream_t s) {
  using namespace gemm_detail;
  static_assert(sizeof(IT) == 4, "the fp16 products run on tc_gemm");
  if (p.M % 128 || p.N % 128 || p.K % 32 || p.batch < 1) return cudaErrorInvalidValue;
  dim3 grid((unsigned)(p.N / 64), (unsigned)(p.M / 64), (unsigned)p.batch);
  if (bk) sgemm_kernel<true, OT><<<grid, 256, 0, s>>>(p);
  else sgemm_kernel<false, OT><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename IT, typename OT>
inline cudaError_t gemm_nt(const GemmBatch& p, cudaStream_t s) { return gemm_launch<IT, OT>(p, true, s); }
template <typename IT, typename OT>
inline cudaError_t gemm_nn(const GemmBatch& p, cudaStream_t s) { return gemm_launch<IT, OT>(p, false, s); }

}  // namespace muon
