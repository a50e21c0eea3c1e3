// Batched GEMMs of the dense Newton-Schulz path (warp-level MMA and fp32
// SIMT).  D[b] = alpha * A[b] op(B[b]) + beta * C[b], all matrices row-major
// inside one per-slice workspace region (matrix b sits at base + b*stride):
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

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <typename T> __device__ __forceinline__ void store_out(T* p, float v) { *p = from_f<T>(v); }

// fp16 operands, fp32 accumulation; 128x128x32 tiles, 8 warps (2 x 4),
// warp tile 64x32, two-stage cp.async pipeline.
template <bool BK, typename OT>
__global__ void __launch_bounds__(256) hgemm_kernel(GemmBatch p) {
  constexpr int BM = 128, BN = 128, BKT = 32, LDA = BKT + 8;
  constexpr int LDBN = BN + 8;
  __shared__ __align__(16) __half As[2][BM * LDA];
  __shared__ __align__(16) __half Bs[2][BK ? BN * LDA : BKT * LDBN];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp >> 2, wn = warp & 3;
  const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
  const size_t boff = (size_t)blockIdx.z * p.stride_bytes;
  const __half* A = reinterpret_cast<const __half*>((const char*)p.A + boff);
  const __half* B = reinterpret_cast<const __half*>((const char*)p.B + boff);
  const int64_t K = p.K, N = p.N;

  auto load = [&](int stage, int64_t k0) {
    #pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = tid + j * 256;
      const int row = c >> 2, col = (c & 3) * 8;
      cp_async16(&As[stage][row * LDA + col], A + (m0 + row) * K + k0 + col);
      if (BK) {
        cp_async16(&Bs[stage][row * LDA + col], B + (n0 + row) * K + k0 + col);
      } else {
        const int kr = c >> 4, nc = (c & 15) * 8;
        cp_async16(&Bs[stage][kr * LDBN + nc], B + (k0 + kr) * N + n0 + nc);
      }
    }
    cp_async_commit();
  };

  float acc[4][4][4];
  #pragma unroll
  for (int i = 0; i < 4; ++i)
    #pragma unroll
    for (int j = 0; j < 4; ++j)
      #pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;

  const int nk = (int)(K / BKT);
  load(0, 0);
  for (int kt = 0; kt < nk; ++kt) {
    if (kt + 1 < nk) {
      load((kt + 1) & 1, (int64_t)(kt + 1) * BKT);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const __half* as = As[kt & 1];
    const __half* bs = Bs[kt & 1];
    #pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t af[4][4], bf[4][2];
      #pragma unroll
      for (int mt = 0; mt < 4; ++mt)
        ldsm_x4(af[mt], as + (wm * 64 + mt * 16 + (lane & 15)) * LDA + ks * 16 + (lane >> 4) * 8);
      #pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t r[4];
        if (BK) {
          ldsm_x4(r, bs + (wn * 32 + np * 16 + (lane & 7) + (lane >> 4) * 8) * LDA + ks * 16 +
                         ((lane >> 3) & 1) * 8);
        } else {
          ldsm_x4_t(r, bs + (ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LDBN + wn * 32 +
                           np * 16 + (lane >> 4) * 8);
        }
        bf[2 * np][0] = r[0]; bf[2 * np][1] = r[1];
        bf[2 * np + 1][0] = r[2]; bf[2 * np + 1][1] = r[3];
      }
      #pragma unroll
      for (int mt = 0; mt < 4; ++mt)
        #pragma unroll
        for (int nt = 0; nt < 4; ++nt) mma16816(acc[mt][nt], af[mt], bf[nt][0], bf[nt][1]);
    }
    __syncthreads();
  }
  const __half* C = p.C ? reinterpret_cast<const __half*>((const char*)p.C + boff) : nullptr;
  OT* D = reinterpret_cast<OT*>((char*)p.D + boff);
  const int g = lane >> 2, t = lane & 3;
  #pragma unroll
  for (int mt = 0; mt < 4; ++mt)
    #pragma unroll
    for (int nt = 0; nt < 4; ++nt)
      #pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t row = m0 + wm * 64 + mt * 16 + g + h * 8;
        const int64_t col = n0 + wn * 32 + nt * 8 + 2 * t;
        float v0 = p.alpha * acc[mt][nt][2 * h], v1 = p.alpha * acc[mt][nt][2 * h + 1];
        if (C && p.beta != 0.f) {
          v0 = fmaf(p.beta, __half2float(C[row * N + col]), v0);
          v1 = fmaf(p.beta, __half2float(C[row * N + col + 1]), v1);
        }
        store_out(D + row * N + col, v0);
        store_out(D + row * N + col + 1, v1);
      }
}

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
  if (p.M % 128 || p.N % 128 || p.K % 32 || p.batch < 1) return cudaErrorInvalidValue;
  if constexpr (sizeof(IT) == 2) {
    dim3 grid((unsigned)(p.N / 128), (unsigned)(p.M / 128), (unsigned)p.batch);
    if (bk) hgemm_kernel<true, OT><<<grid, 256, 0, s>>>(p);
    else hgemm_kernel<false, OT><<<grid, 256, 0, s>>>(p);
  } else {
    dim3 grid((unsigned)(p.N / 64), (unsigned)(p.M / 64), (unsigned)p.batch);
    if (bk) sgemm_kernel<true, OT><<<grid, 256, 0, s>>>(p);
    else sgemm_kernel<false, OT><<<grid, 256, 0, s>>>(p);
  }
  return cudaGetLastError();
}

template <typename IT, typename OT>
inline cudaError_t gemm_nt(const GemmBatch& p, cudaStream_t s) { return gemm_launch<IT, OT>(p, true, s); }
template <typename IT, typename OT>
inline cudaError_t gemm_nn(const GemmBatch& p, cudaStream_t s) { return gemm_launch<IT, OT>(p, false, s); }

}  // namespace muon
