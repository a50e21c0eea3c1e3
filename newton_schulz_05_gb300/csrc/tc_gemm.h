// Batched fp16 tcgen05 GEMM of the dense Newton-Schulz path (tc_gemm.cu).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace muon {

// D[b] = alpha * A[b] op(B[b]) + diag * I, and optionally a second output
// D2[b] = alpha2 * A[b] op(B[b]) + diag2 * I from the same accumulator; matrix
// b of each operand sits `stride` bytes after matrix b-1.
//   A  [M, K] fp16, K contiguous
//   B  [N, K] fp16, K contiguous (b_mn = 0)  or  [K, N], N contiguous (b_mn = 1)
//   D  [M, N] fp16 (d_f32 = 0) or fp32 (d_f32 = 1);  D2 [M, N] fp16 or null
// I is the identity of [M, N] (ones where row == column).
// sym = 1: the product is symmetric (M == N); only tiles on or above the
// diagonal are computed and each is mirrored, so every element has one writer.
// M must be a multiple of 128, N of 128, K of 64; every base address and
// `stride` a multiple of 16 bytes; mirrored and second outputs are fp16.
struct TcGemm {
  int64_t M = 0, N = 0, K = 0;
  int batch = 1;
  size_t stride = 0;
  const void* A = nullptr;
  const void* B = nullptr;
  void* D = nullptr;
  void* D2 = nullptr;
  int d_f32 = 0;
  float alpha = 1.f, diag = 0.f;
  float alpha2 = 1.f, diag2 = 0.f;
  // optional per-slice factor of alpha and alpha2: the float at
  // alpha_base + b * alpha_stride (device) multiplies both for slice b
  const void* alpha_base = nullptr;
  size_t alpha_stride = 0;
  int sym = 0;
  int b_mn = 0;
  // fused parameter update (non-symmetric products only): with W set, the
  // epilogue writes W'[b] = W[b] (1 - lr wd) - lrs D[b] into parameter slice
  // b, of dtype bf16 (w_f32 = 0) or fp32, stored [wm, wn] or, with wtr, [wn, wm]
  // (D's rows past wm and columns past wn are padding), and stores no D
  void* const* W = nullptr;
  int w_f32 = 0, wtr = 0;
  int64_t wm = 0, wn = 0;
  float decay = 1.f, lrs = 0.f;
  int* err = nullptr;   // device error word (bounded waits); when set at the
                        // kernel's start, the kernel returns at once
  const int* skip = nullptr;  // device flag: when set, the kernel returns at once
  uint32_t wait_limit = 1u << 26;   // polls of a main-path wait before giving up
};

cudaError_t tc_gemm(const TcGemm& g, cudaStream_t s);
uint32_t tc_idesc_f16(int m, int n, int b_mn);
size_t tc_gemm_smem_bytes();

}  // namespace muon
