// Batched fp16 tcgen05 GEMM of the dense Newton-Schulz path (tc_gemm.cu).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace muon {

// D[b] = alpha * A[b] op(B[b]) + beta * C[b]; matrix b of each operand sits
// `stride` bytes after matrix b-1.
//   A  [M, K] fp16, K contiguous
//   B  [N, K] fp16, K contiguous (b_mn = 0)  or  [K, N], N contiguous (b_mn = 1)
//   C  [M, N] fp16 or null;  D [M, N] fp16 (d_f32 = 0) or fp32 (d_f32 = 1)
// sym = 1: the product is symmetric (M == N); only tiles on or above the
// diagonal are computed and each is mirrored, so every element has one writer.
// M must be a multiple of 128, N of 128, K of 64; every base address and
// `stride` a multiple of 16 bytes.
struct TcGemm {
  int64_t M = 0, N = 0, K = 0;
  int batch = 1;
  size_t stride = 0;
  const void* A = nullptr;
  const void* B = nullptr;
  const void* C = nullptr;
  void* D = nullptr;
  int d_f32 = 0;
  float alpha = 1.f, beta = 0.f;
  int sym = 0;
  int b_mn = 0;
  int* err = nullptr;   // device error word (bounded waits)
  const int* skip = nullptr;  // device flag: when set, the kernel returns at once
};

cudaError_t tc_gemm(const TcGemm& g, cudaStream_t s);
uint32_t tc_idesc_f16(int m, int n, int b_mn);
size_t tc_gemm_smem_bytes();

}  // namespace muon
