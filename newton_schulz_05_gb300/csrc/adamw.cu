// AdamW for the parameters Muon does not orthogonalise: 1-D tensors (biases,
// norm scales) and any other tensor the caller keeps off the Muon path.  The
// Paddle Muon sharding PR ("Support Muon sharding optimizer comm overlap")
// keeps separate 2-D and 1-D gradient buffers because the two kinds of
// parameters take different update rules; this is the 1-D rule.
//
// One launch updates every tensor (multi-tensor apply): block b takes chunk
// b of the concatenated element range, 4 elements per thread per iteration,
// 16-byte vector access when every base is aligned.  HBM traffic per element
// (bf16 parameters): G 2 + W 2 + W' 2 + m 4 + m' 4 + v 4 + v' 4 = 22 bytes.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace muon {

namespace {

constexpr int kAdamMaxTensors = 256;
constexpr int kAdamThreads = 256;
constexpr int kAdamChunk = kAdamThreads * 16;   // elements per block

struct AdamwParams {
  void* W[kAdamMaxTensors];
  const void* G[kAdamMaxTensors];
  float* M[kAdamMaxTensors];
  float* V[kAdamMaxTensors];
  int64_t numel[kAdamMaxTensors];
  int chunk_start[kAdamMaxTensors + 1];   // first chunk of each tensor
  int n;
  int vec;
  float lr, b1, b2, eps, decay;            // decay = 1 - lr * wd
  float inv_c1, inv_c2;                    // 1 / bias corrections
};

__device__ __forceinline__ void adam_one(float& w, float g, float& m, float& v,
                                         const AdamwParams& p) {
  m = fmaf(p.b1, m, (1.f - p.b1) * g);
  v = fmaf(p.b2, v, (1.f - p.b2) * g * g);
  const float mhat = m * p.inv_c1;
  const float vhat = v * p.inv_c2;
  w = fmaf(w, p.decay, -p.lr * (mhat / (sqrtf(vhat) + p.eps)));
}

template <typename PT>
__global__ void __launch_bounds__(kAdamThreads) adamw_kernel(const __grid_constant__ AdamwParams p) {
  // tensor of this chunk: the last t with chunk_start[t] <= blockIdx.x
  int lo = 0, hi = p.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.chunk_start[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
  }
  const int t = lo;
  const int64_t n = p.numel[t];
  const int64_t c0 = (int64_t)(blockIdx.x - p.chunk_start[t]) * kAdamChunk;
  const int64_t c1 = c0 + kAdamChunk < n ? c0 + kAdamChunk : n;
  PT* W = static_cast<PT*>(p.W[t]);
  const PT* G = static_cast<const PT*>(p.G[t]);
  float* M = p.M[t];
  float* V = p.V[t];
  for (int64_t i = c0 + 4 * threadIdx.x; i < c1; i += 4 * kAdamThreads) {
    if (p.vec && i + 3 < c1) {
      float w[4], g[4];
      float4 m = *reinterpret_cast<const float4*>(M + i);
      float4 v = *reinterpret_cast<const float4*>(V + i);
      if constexpr (sizeof(PT) == 2) {
        const uint2 uw = *reinterpret_cast<const uint2*>(W + i);
        const uint2 ug = *reinterpret_cast<const uint2*>(G + i);
        const float2 w01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&uw.x));
        const float2 w23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&uw.y));
        const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ug.x));
        const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ug.y));
        w[0] = w01.x; w[1] = w01.y; w[2] = w23.x; w[3] = w23.y;
        g[0] = g01.x; g[1] = g01.y; g[2] = g23.x; g[3] = g23.y;
      } else {
        const float4 uw = *reinterpret_cast<const float4*>(W + i);
        const float4 ug = *reinterpret_cast<const float4*>(G + i);
        w[0] = uw.x; w[1] = uw.y; w[2] = uw.z; w[3] = uw.w;
        g[0] = ug.x; g[1] = ug.y; g[2] = ug.z; g[3] = ug.w;
      }
      adam_one(w[0], g[0], m.x, v.x, p);
      adam_one(w[1], g[1], m.y, v.y, p);
      adam_one(w[2], g[2], m.z, v.z, p);
      adam_one(w[3], g[3], m.w, v.w, p);
      *reinterpret_cast<float4*>(M + i) = m;
      *reinterpret_cast<float4*>(V + i) = v;
      if constexpr (sizeof(PT) == 2) {
        uint2 u;
        __nv_bfloat162 a = __floats2bfloat162_rn(w[0], w[1]), b = __floats2bfloat162_rn(w[2], w[3]);
        u.x = *reinterpret_cast<uint32_t*>(&a);
        u.y = *reinterpret_cast<uint32_t*>(&b);
        *reinterpret_cast<uint2*>(W + i) = u;
      } else {
        *reinterpret_cast<float4*>(W + i) = make_float4(w[0], w[1], w[2], w[3]);
      }
    } else {
      for (int64_t j = i; j < i + 4 && j < c1; ++j) {
        float w = to_f(W[j]), m = M[j], v = V[j];
        adam_one(w, to_f(G[j]), m, v, p);
        M[j] = m;
        V[j] = v;
        W[j] = from_f<PT>(w);
      }
    }
  }
}

}  // namespace

}  // namespace muon

using namespace muon;

extern "C" muon_status muon_adamw_step(int n, void* const* params, const void* const* grads,
                                       float* const* exp_avg, float* const* exp_avg_sq,
                                       const int64_t* numel, int dtype, float lr, float beta1,
                                       float beta2, float eps, float wd, int step, void* stream) {
  if (n < 0 || (n > 0 && (!params || !grads || !exp_avg || !exp_avg_sq || !numel)))
    return MUON_ERR_INVALID_ARG;
  if (dtype != MUON_BF16 && dtype != MUON_F32) return MUON_ERR_DTYPE;
  if (step < 1 || !std::isfinite(lr) || !std::isfinite(beta1) || !std::isfinite(beta2) ||
      !std::isfinite(eps) || !std::isfinite(wd) || beta1 < 0.f || beta1 >= 1.f || beta2 < 0.f ||
      beta2 >= 1.f || eps < 0.f)
    return MUON_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (!params[i] || !grads[i] || !exp_avg[i] || !exp_avg_sq[i] || numel[i] < 0)
      return MUON_ERR_INVALID_ARG;
  if (fault_switch() == kFaultLaunch) return MUON_ERR_CUDA;
  NvtxRange range("muon_adamw_step");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t es = dtype == MUON_BF16 ? 2 : 4;
  AdamwParams p;
  p.lr = lr; p.b1 = beta1; p.b2 = beta2; p.eps = eps;
  p.decay = 1.f - lr * wd;
  p.inv_c1 = (float)(1.0 / (1.0 - std::pow((double)beta1, step)));
  p.inv_c2 = (float)(1.0 / (1.0 - std::pow((double)beta2, step)));
  for (int t0 = 0; t0 < n; t0 += kAdamMaxTensors) {
    const int cnt = n - t0 < kAdamMaxTensors ? n - t0 : kAdamMaxTensors;
    int chunks = 0, used = 0;
    int vec = 1;
    for (int i = 0; i < cnt; ++i) {
      if (numel[t0 + i] == 0) continue;
      const int64_t nc = (numel[t0 + i] + kAdamChunk - 1) / kAdamChunk;
      if ((int64_t)chunks + nc > (int64_t)1 << 30) return MUON_ERR_UNSUPPORTED_SHAPE;
      p.W[used] = params[t0 + i];
      p.G[used] = grads[t0 + i];
      p.M[used] = exp_avg[t0 + i];
      p.V[used] = exp_avg_sq[t0 + i];
      p.numel[used] = numel[t0 + i];
      p.chunk_start[used] = chunks;
      const uintptr_t a = reinterpret_cast<uintptr_t>(params[t0 + i]) |
                          reinterpret_cast<uintptr_t>(grads[t0 + i]);
      if (a % (4 * es) || (reinterpret_cast<uintptr_t>(exp_avg[t0 + i]) |
                           reinterpret_cast<uintptr_t>(exp_avg_sq[t0 + i])) % 16)
        vec = 0;
      chunks += (int)nc;
      ++used;
    }
    if (used == 0) continue;
    p.chunk_start[used] = chunks;
    p.n = used;
    p.vec = vec;
    if (dtype == MUON_BF16)
      adamw_kernel<__nv_bfloat16><<<chunks, kAdamThreads, 0, s>>>(p);
    else
      adamw_kernel<float><<<chunks, kAdamThreads, 0, s>>>(p);
    if (cudaGetLastError() != cudaSuccess) return MUON_ERR_CUDA;
  }
  return MUON_OK;
}
