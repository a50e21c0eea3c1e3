// Fused Muon step for skinny slice groups (min(M,N) <= 64), one launch per
// group: momentum, normalisation, T Newton-Schulz steps and the weight-decay
// update, with each slice resident on chip from its first load to its last
// store.
//
// Method (HyperParallel FSDP Muon RFC, mindspore hyper-parallel issue
// "HyperParallel FSDP Muon优化器性能优化 RFC"): section 3 batches the many
// small [24, 10240]-like parameters of equal trailing dims into one launch;
// section 1(1) feeds the gradient momentum to Newton-Schulz; section 6 adds
// decoupled weight decay to the update.
//
// GB300 design:
//   * one thread-block cluster per slice, C CTAs (<= 8), one CTA per SM;
//     CTA r owns a contiguous range of 32-column "superchunks" of the
//     working matrix X [m, n] (m = min(M, N); X = V^T when M > N);
//   * X lives in tensor memory (TMEM, 512 columns x 128 lanes x 4 B per SM)
//     between passes: every lane keeps, per superchunk, 4 registers per
//     8-row block in the layout of a warp-MMA fragment, so X never returns
//     to HBM: HBM traffic is G + M (read), M' (write), W (read + write),
//     14 bytes per element for bf16 parameters;
//   * X X^T and B X run on the tensor cores as m16n8k16 / m16n8k8 fp16 warp
//     MMAs with fp32 accumulation; B X needs X as the B operand, obtained
//     with movmatrix transposes of the 8x8 register blocks;
//   * the m x m Gram matrix is reduced deterministically: warps -> CTA in
//     shared memory, CTAs -> cluster through distributed shared memory in
//     rank order, so every CTA holds the same bits; A*A and B = b*A + c*A*A
//     are computed in fp32 by every CTA;
//   * the Frobenius norm is reduced the same way; V is kept as bf16 until
//     the norm is known, then X0 = fp16(V / (||V|| + eps)).
//   * W is prefetched into L2 (bulk prefetch) while the iteration runs.
#include <cooperative_groups.h>
#include <cstdio>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace muon {

namespace {

struct SkinnyParams {
  SlicePtrs ptrs;
  int m, n;          // working dims
  int tr;            // stored slice is [n, m] (working = transposed)
  int nsc;           // superchunks of 32 working columns
  int sc_per_cta, sc_per_warp;
  int cluster;
  int vec;           // vectorised global access allowed for every slice
  StepArgs st;
  float lrs;         // lr * scale
  float decay;       // 1 - lr * wd
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_h(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
}
__device__ __forceinline__ float2 unpack_h(uint32_t u) {
  return __half22float2(*reinterpret_cast<__half2*>(&u));
}
__device__ __forceinline__ uint32_t movt(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
  return d;
}
__device__ __forceinline__ void mma_k16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_k8(float* d, uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

// tensor memory: 32 lanes x 4 columns per warp access (lane = thread)
__device__ __forceinline__ void tm_ld4(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
__device__ __forceinline__ void tm_st4(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}
__device__ __forceinline__ void tm_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tm_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// 4 consecutive working columns c..c+3 of working row i of one slice.
template <typename PT>
struct Access {
  const SkinnyParams& p;
  __device__ __forceinline__ int64_t idx(int i, int c) const {
    return p.tr ? (int64_t)c * p.m + i : (int64_t)i * p.n + c;
  }
  // NC: read-only path (only for buffers this kernel never writes)
  template <bool NC>
  __device__ __forceinline__ void load(const PT* base, int i, int c, float* v) const {
    if (p.vec) {
      if (i < p.m && c < p.n) {
        if constexpr (sizeof(PT) == 2) {
          const uint2* a = reinterpret_cast<const uint2*>(base + idx(i, c));
          const uint2 u = NC ? __ldg(a) : *a;
          const float2 x = unpack_bf16(u.x), y = unpack_bf16(u.y);
          v[0] = x.x; v[1] = x.y; v[2] = y.x; v[3] = y.y;
        } else {
          const float4* a = reinterpret_cast<const float4*>(base + idx(i, c));
          const float4 u = NC ? __ldg(a) : *a;
          v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
        }
      } else {
        v[0] = v[1] = v[2] = v[3] = 0.f;
      }
    } else {
      #pragma unroll
      for (int e = 0; e < 4; ++e)
        v[e] = (i < p.m && c + e < p.n) ? to_f(base[idx(i, c + e)]) : 0.f;
    }
  }
  __device__ __forceinline__ void load_f32(const float* base, int i, int c, float* v) const {
    if (p.vec) {
      if (i < p.m && c < p.n) {
        const float4 u = *reinterpret_cast<const float4*>(base + idx(i, c));
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
      } else {
        v[0] = v[1] = v[2] = v[3] = 0.f;
      }
    } else {
      #pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = (i < p.m && c + e < p.n) ? base[idx(i, c + e)] : 0.f;
    }
  }
  __device__ __forceinline__ void store(PT* base, int i, int c, const float* v) const {
    if (p.vec) {
      if (i < p.m && c < p.n) {
        if constexpr (sizeof(PT) == 2) {
          uint2 u;
          u.x = pack_bf16(v[0], v[1]);
          u.y = pack_bf16(v[2], v[3]);
          *reinterpret_cast<uint2*>(base + idx(i, c)) = u;
        } else {
          *reinterpret_cast<float4*>(base + idx(i, c)) = make_float4(v[0], v[1], v[2], v[3]);
        }
      }
    } else {
      #pragma unroll
      for (int e = 0; e < 4; ++e)
        if (i < p.m && c + e < p.n) base[idx(i, c + e)] = from_f<PT>(v[e]);
    }
  }
  __device__ __forceinline__ void store_f32(float* base, int i, int c, const float* v) const {
    if (p.vec) {
      if (i < p.m && c < p.n)
        *reinterpret_cast<float4*>(base + idx(i, c)) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
      #pragma unroll
      for (int e = 0; e < 4; ++e)
        if (i < p.m && c + e < p.n) base[idx(i, c + e)] = v[e];
    }
  }
};

template <int MB, int NW>
struct SkinnySmem {
  static constexpr int MP = 8 * MB;
  static constexpr int NP = (MB + 1) / 2;
  static constexpr int MPX = 16 * NP;
  static constexpr size_t gram_w = 0;
  static constexpr size_t gram_c = gram_w + sizeof(float) * NW * MP * MP;
  static constexpr size_t afull = gram_c + sizeof(float) * 2 * MP * MP;
  static constexpr size_t bm = afull + sizeof(float) * MP * MP;
  static constexpr size_t misc = (bm + sizeof(__half) * MPX * MPX + 15) & ~size_t(15);
  static constexpr size_t total = misc + 64 * sizeof(float) + 16;
  // one CTA per SM: a second CTA on the SM would wait for tensor memory
  static constexpr size_t launch = total > 120 * 1024 ? total : 120 * 1024;
};

// Gram tiles: rows 16P..16P+15 (row blocks 2P, 2P+1) x row block J, J >= 2P.
__device__ __forceinline__ bool gram_covered(int i, int j) {
  const int I = i >> 3, J = j >> 3;
  return J >= ((I >> 1) << 1);
}

template <int MB>
__device__ __forceinline__ void gram_accum(float (&acc)[(MB + 1) / 2][MB][4],
                                           const uint32_t (&x)[MB][4]) {
  constexpr int NP = (MB + 1) / 2;
  #pragma unroll
  for (int k = 0; k < 2; ++k)
    #pragma unroll
    for (int P = 0; P < NP; ++P) {
      const uint32_t a0 = x[2 * P][2 * k], a2 = x[2 * P][2 * k + 1];
      const uint32_t a1 = (2 * P + 1 < MB) ? x[(2 * P + 1) % MB][2 * k] : 0u;
      const uint32_t a3 = (2 * P + 1 < MB) ? x[(2 * P + 1) % MB][2 * k + 1] : 0u;
      #pragma unroll
      for (int J = 2 * P; J < MB; ++J) mma_k16(acc[P][J], a0, a1, a2, a3, x[J][2 * k], x[J][2 * k + 1]);
    }
}

template <int MB, int NW, typename PT>
__global__ void __launch_bounds__(NW * 32, 1) skinny_kernel(const __grid_constant__ SkinnyParams p) {
  using S = SkinnySmem<MB, NW>;
  constexpr int MP = S::MP, NP = S::NP, MPX = S::MPX;
  constexpr int NT = NW * 32;
  constexpr int COLS_W = 512 / (NW / 4);
  extern __shared__ __align__(128) unsigned char smem[];
  float* gram_w = reinterpret_cast<float*>(smem + S::gram_w);
  float* gram_c = reinterpret_cast<float*>(smem + S::gram_c);
  float* afull = reinterpret_cast<float*>(smem + S::afull);
  __half* bm = reinterpret_cast<__half*>(smem + S::bm);
  float* red = reinterpret_cast<float*>(smem + S::misc);     // NW floats
  float* norm_slot = red + 32;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red + 48);

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int slice = blockIdx.x / p.cluster;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const Access<PT> acc_{p};
  const PT* G = static_cast<const PT*>(p.ptrs.G[slice]);
  PT* W = static_cast<PT*>(p.ptrs.W[slice]);
  float* Mo = p.ptrs.Mom[slice];
  float* Oout = p.ptrs.O[slice];
  const StepArgs& st = p.st;

  for (int e = tid; e < MPX * MPX; e += NT) bm[e] = __float2half_rn(0.f);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
                     smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t taddr_w = tbase + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)((warp >> 2) * COLS_W);

  const int jc0 = rank * p.sc_per_cta;
  const int jc1 = min(p.nsc, jc0 + p.sc_per_cta);
  const int j0 = jc0 + warp * p.sc_per_warp;
  const int j1 = min(jc1, j0 + p.sc_per_warp);
  const int nslot = max(0, j1 - j0);

  // ---- phase 1: momentum, V (bf16 in TMEM), sum of squares -------------------
  float ss = 0.f;
  for (int q = 0; q < nslot; ++q) {
    const int cb = (j0 + q) * 32;
    float gv[MB][2][4], mv[MB][2][4];
    #pragma unroll
    for (int rb = 0; rb < MB; ++rb)
      #pragma unroll
      for (int h = 0; h < 2; ++h) {
        acc_.template load<true>(G, rb * 8 + g, cb + h * 16 + 4 * t4, gv[rb][h]);
        acc_.load_f32(Mo, rb * 8 + g, cb + h * 16 + 4 * t4, mv[rb][h]);
      }
    uint32_t xr[MB][4];
    #pragma unroll
    for (int rb = 0; rb < MB; ++rb)
      #pragma unroll
      for (int h = 0; h < 2; ++h) {
        float vv[4];
        #pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float mm = fmaf(st.beta, mv[rb][h][e], gv[rb][h][e]);
          mv[rb][h][e] = mm;
          vv[e] = st.nesterov ? fmaf(st.beta, mm, gv[rb][h][e]) : mm;
          ss = fmaf(vv[e], vv[e], ss);
        }
        acc_.store_f32(Mo, rb * 8 + g, cb + h * 16 + 4 * t4, mv[rb][h]);
        xr[rb][2 * h] = pack_bf16(vv[0], vv[1]);
        xr[rb][2 * h + 1] = pack_bf16(vv[2], vv[3]);
      }
    #pragma unroll
    for (int rb = 0; rb < MB; ++rb) tm_st4(taddr_w + q * 4 * MB + 4 * rb, xr[rb]);
  }
  tm_wait_st();

  // ---- cluster-wide ||V||_F (fixed order) ------------------------------------
  #pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (tid == 0) {
    float s = 0.f;
    for (int w = 0; w < NW; ++w) s += red[w];
    norm_slot[0] = s;
  }
  cluster.sync();
  float tot = 0.f;
  for (int r = 0; r < p.cluster; ++r) tot += *cluster.map_shared_rank(norm_slot, r);
  const float inv = 1.f / (sqrtf(tot) + st.eps);

  // warm L2 with this CTA's parameter rows for the final update
  if (warp == NW - 1 && jc1 > jc0) {
    const size_t es = sizeof(PT);
    const int c0 = jc0 * 32, c1 = min(p.n, jc1 * 32);
    const int rows = p.tr ? 1 : p.m;
    for (int i = lane; i < rows; i += 32) {
      const char* a = reinterpret_cast<const char*>(W) +
                      (p.tr ? (size_t)c0 * p.m : (size_t)i * p.n + c0) * es;
      const size_t len = (size_t)(c1 - c0) * (p.tr ? p.m : 1) * es;
      const uintptr_t s0 = (reinterpret_cast<uintptr_t>(a) + 15) & ~uintptr_t(15);
      const uintptr_t s1 = (reinterpret_cast<uintptr_t>(a) + len) & ~uintptr_t(15);
      if (s1 > s0)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(s0),
                     "r"((uint32_t)(s1 - s0))
                     : "memory");
    }
  }

  auto epilogue = [&](int q, const float (&o)[MB][4][2]) {
    const int cb = (j0 + q) * 32;
    #pragma unroll
    for (int rb = 0; rb < MB; ++rb)
      #pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = rb * 8 + g, c = cb + h * 16 + 4 * t4;
        float w[4];
        acc_.template load<false>(W, i, c, w);
        const float ov[4] = {o[rb][2 * h][0], o[rb][2 * h][1], o[rb][2 * h + 1][0],
                             o[rb][2 * h + 1][1]};
        float wn[4];
        #pragma unroll
        for (int e = 0; e < 4; ++e) wn[e] = fmaf(w[e], p.decay, -p.lrs * ov[e]);
        acc_.store(W, i, c, wn);
        if (Oout) acc_.store_f32(Oout, i, c, ov);
      }
  };

  if (st.T == 0) {
    // O = V / (||V|| + eps)
    for (int q = 0; q < nslot; ++q) {
      uint32_t xr[MB][4];
      #pragma unroll
      for (int rb = 0; rb < MB; ++rb) tm_ld4(taddr_w + q * 4 * MB + 4 * rb, xr[rb]);
      tm_wait_ld();
      float o[MB][4][2];
      #pragma unroll
      for (int rb = 0; rb < MB; ++rb)
        #pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float2 f = unpack_bf16(xr[rb][r]);
          o[rb][r][0] = f.x * inv;
          o[rb][r][1] = f.y * inv;
        }
      epilogue(q, o);
    }
  } else {
    // ---- phase 2: X0 = fp16(V * inv) and its Gram partial --------------------
    float gacc[NP][MB][4];
    #pragma unroll
    for (int P = 0; P < NP; ++P)
      #pragma unroll
      for (int J = 0; J < MB; ++J)
        #pragma unroll
        for (int e = 0; e < 4; ++e) gacc[P][J][e] = 0.f;
    for (int q = 0; q < nslot; ++q) {
      uint32_t xr[MB][4];
      #pragma unroll
      for (int rb = 0; rb < MB; ++rb) tm_ld4(taddr_w + q * 4 * MB + 4 * rb, xr[rb]);
      tm_wait_ld();
      #pragma unroll
      for (int rb = 0; rb < MB; ++rb)
        #pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float2 f = unpack_bf16(xr[rb][r]);
          xr[rb][r] = pack_h(f.x * inv, f.y * inv);
        }
      #pragma unroll
      for (int rb = 0; rb < MB; ++rb) tm_st4(taddr_w + q * 4 * MB + 4 * rb, xr[rb]);
      gram_accum<MB>(gacc, xr);
    }
    tm_wait_st();

    for (int t = 0; t < st.T; ++t) {
      const bool last = t == st.T - 1;
      // warp partial -> shared memory
      float* gw = gram_w + warp * MP * MP;
      #pragma unroll
      for (int P = 0; P < NP; ++P)
        #pragma unroll
        for (int J = 2 * P; J < MB; ++J)
          #pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int row = 16 * P + 8 * hh + g;
            if (row < MP) {
              gw[row * MP + 8 * J + 2 * t4] = gacc[P][J][2 * hh];
              gw[row * MP + 8 * J + 2 * t4 + 1] = gacc[P][J][2 * hh + 1];
            }
          }
      __syncthreads();
      float* gc = gram_c + (t & 1) * MP * MP;
      for (int e = tid; e < MP * MP; e += NT) {
        if (!gram_covered(e / MP, e % MP)) continue;
        float s = 0.f;
        for (int w = 0; w < NW; ++w) s += gram_w[w * MP * MP + e];
        gc[e] = s;
      }
      cluster.sync();
      for (int e = tid; e < MP * MP; e += NT) {
        const int i = e / MP, j = e % MP;
        const int src = gram_covered(i, j) ? e : j * MP + i;
        float s = 0.f;
        for (int r = 0; r < p.cluster; ++r) s += cluster.map_shared_rank(gc, r)[src];
        afull[e] = s;
      }
      __syncthreads();
      for (int e = tid; e < MP * MP; e += NT) {
        const int i = e / MP, j = e % MP;
        float s = 0.f;
        #pragma unroll 8
        for (int k = 0; k < MP; ++k) s = fmaf(afull[i * MP + k], afull[k * MP + j], s);
        bm[i * MPX + j] = __float2half_rn(fmaf(st.b, afull[e], st.c * s));
      }
      __syncthreads();
      // B as the A operand of Y = B X: rows 16P.., k steps over row-block pairs
      uint32_t afr[NP][NP][4];
      #pragma unroll
      for (int P = 0; P < NP; ++P)
        #pragma unroll
        for (int kk = 0; kk < NP; ++kk) {
          const __half* r0 = bm + (16 * P + g) * MPX + 16 * kk + 2 * t4;
          const __half* r1 = r0 + 8 * MPX;
          afr[P][kk][0] = *reinterpret_cast<const uint32_t*>(r0);
          afr[P][kk][1] = *reinterpret_cast<const uint32_t*>(r1);
          afr[P][kk][2] = *reinterpret_cast<const uint32_t*>(r0 + 8);
          afr[P][kk][3] = *reinterpret_cast<const uint32_t*>(r1 + 8);
        }
      if (!last) {
        #pragma unroll
        for (int P = 0; P < NP; ++P)
          #pragma unroll
          for (int J = 0; J < MB; ++J)
            #pragma unroll
            for (int e = 0; e < 4; ++e) gacc[P][J][e] = 0.f;
      }
      for (int q = 0; q < nslot; ++q) {
        uint32_t xr[MB][4];
        #pragma unroll
        for (int rb = 0; rb < MB; ++rb) tm_ld4(taddr_w + q * 4 * MB + 4 * rb, xr[rb]);
        tm_wait_ld();
        float o[MB][4][2];
        #pragma unroll
        for (int r = 0; r < 4; ++r) {
          uint32_t xt[MB];
          #pragma unroll
          for (int J = 0; J < MB; ++J) xt[J] = movt(xr[J][r]);
          float y[NP][4];
          #pragma unroll
          for (int P = 0; P < NP; ++P) {
            y[P][0] = y[P][1] = y[P][2] = y[P][3] = 0.f;
            #pragma unroll
            for (int kk = 0; kk < NP; ++kk) {
              if (2 * kk + 1 < MB)
                mma_k16(y[P], afr[P][kk][0], afr[P][kk][1], afr[P][kk][2], afr[P][kk][3],
                        xt[2 * kk], xt[(2 * kk + 1) % MB]);
              else
                mma_k8(y[P], afr[P][kk][0], afr[P][kk][1], xt[2 * kk]);
            }
          }
          #pragma unroll
          for (int rb = 0; rb < MB; ++rb) {
            const float2 x = unpack_h(xr[rb][r]);
            o[rb][r][0] = fmaf(st.a, x.x, y[rb >> 1][(rb & 1) * 2]);
            o[rb][r][1] = fmaf(st.a, x.y, y[rb >> 1][(rb & 1) * 2 + 1]);
          }
        }
        if (last) {
          epilogue(q, o);
        } else {
          #pragma unroll
          for (int rb = 0; rb < MB; ++rb)
            #pragma unroll
            for (int r = 0; r < 4; ++r) xr[rb][r] = pack_h(o[rb][r][0], o[rb][r][1]);
          #pragma unroll
          for (int rb = 0; rb < MB; ++rb) tm_st4(taddr_w + q * 4 * MB + 4 * rb, xr[rb]);
          gram_accum<MB>(gacc, xr);
        }
      }
      tm_wait_st();
    }
  }
  // no CTA may leave while a cluster peer can still read its shared memory
  tc_fence_before();
  cluster.sync();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tbase) : "memory");
}

template <int MB, typename PT>
cudaError_t launch_mb(const Group& g, const SkinnyParams& prm, int nslices, cudaStream_t s) {
  constexpr int NW = MB <= 4 ? 16 : 8;
  using S = SkinnySmem<MB, NW>;
  auto kern = skinny_kernel<MB, NW, PT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)S::launch);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(nslices * g.cluster), 1, 1);
  cfg.blockDim = dim3(NW * 32, 1, 1);
  cfg.dynamicSmemBytes = S::launch;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)g.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

template <typename PT>
cudaError_t launch_pt(const Group& g, const SkinnyParams& prm, int ns, cudaStream_t s) {
  switch (g.mb) {
    case 1: return launch_mb<1, PT>(g, prm, ns, s);
    case 2: return launch_mb<2, PT>(g, prm, ns, s);
    case 3: return launch_mb<3, PT>(g, prm, ns, s);
    case 4: return launch_mb<4, PT>(g, prm, ns, s);
    case 6: return launch_mb<6, PT>(g, prm, ns, s);
    case 8: return launch_mb<8, PT>(g, prm, ns, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_skinny(const Group& g, const SlicePtrs& ptrs, int nslices, const StepArgs& st,
                          int* /*err_word*/, cudaStream_t s) {
  SkinnyParams prm;
  prm.ptrs = ptrs;
  prm.m = (int)g.m;
  prm.n = (int)g.n;
  prm.tr = g.tr;
  prm.nsc = (int)((g.n + 31) / 32);
  prm.sc_per_cta = g.sc_per_cta;
  prm.sc_per_warp = g.sc_per_warp;
  prm.cluster = g.cluster;
  prm.st = st;
  prm.lrs = st.lr * g.scale;
  prm.decay = 1.f - st.lr * st.wd;
  const size_t es = g.dtype == MUON_BF16 ? 2 : 4;
  int vec = (!g.tr && g.n % 4 == 0) ? 1 : 0;
  for (int i = 0; i < nslices && vec; ++i) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(ptrs.W[i]) | reinterpret_cast<uintptr_t>(ptrs.G[i]);
    if (a % (4 * es)) vec = 0;
    if (reinterpret_cast<uintptr_t>(ptrs.Mom[i]) % 16) vec = 0;
    if (ptrs.O[i] && reinterpret_cast<uintptr_t>(ptrs.O[i]) % 16) vec = 0;
  }
  prm.vec = vec;
  if (g.dtype == MUON_BF16) return launch_pt<__nv_bfloat16>(g, prm, nslices, s);
  return launch_pt<float>(g, prm, nslices, s);
}

}  // namespace muon
