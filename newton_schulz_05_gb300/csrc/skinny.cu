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
//     working matrix (m = min(M, N) rows; the slice is read transposed when
//     M > N);
//   * Newton-Schulz runs in Gram space (see skinny_kernel): one pass over
//     the slice forms V V^T, the T steps act on m x m matrices only, a
//     second pass applies O = Q X_0.  For m << n this removes 2(T-1) of the
//     2T passes over the long dimension and their syncs;
//   * between the passes V lives in tensor memory (TMEM, 512 columns x 128
//     lanes x 4 B per SM), 4 registers per 8-row block per lane in the layout
//     of a warp-MMA fragment, so the slice never returns to HBM: traffic is
//     G + M read, M' written, W read and W' written, 14 B per element for
//     bf16 parameters;
//   * V V^T and Q X_0 = (Q / (||V|| + eps)) V run on the tensor cores as
//     bf16 m16n8k16 / m16n8k8 warp MMAs with fp32 accumulation: the bf16 V
//     held in TMEM is the B operand of both (through movmatrix transposes of
//     its 8x8 register blocks for the second), the normalisation is folded
//     into the fp32 Q before it is rounded to bf16;
//   * ||V||^2 and V V^T are reduced deterministically: warps -> CTA in shared
//     memory, CTAs -> cluster through distributed shared memory in rank
//     order, so every CTA holds the same bits and computes the same Q in fp32;
//   * rows stream through a shared-memory ring of bulk copies when they are
//     16-byte aligned (G and M rows in pass 1, W rows in pass 2, the first W
//     stages issued by the warps the m x m recursion leaves idle); otherwise
//     gradient and momentum rows are prefetched into L2 a few superchunks
//     ahead and the parameter loads of the update are issued one superchunk
//     ahead.
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
  int staged;        // rows stream through the shared-memory ring (bulk copies)
  int* err;          // device error word (bounded waits)
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
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
}
__device__ __forceinline__ uint32_t movt(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
  return d;
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

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// bounded wait for the phase of parity `parity`: at most `limit` polls
// (zero: give up at once); false when the budget ran out
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint32_t limit = kWaitLimit) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
// one contiguous global -> shared copy, completion counted on `bar`
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
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

template <int MB, int NW, int ES>
struct SkinnySmem {
  static constexpr int MP = 8 * MB;
  static constexpr int NP = (MB + 1) / 2;
  static constexpr int MPX = 16 * NP;
  static constexpr size_t MAT = sizeof(float) * MP * MP;             // Gram partials
  // padded row of the m x m matrices: odd for distinct banks of column
  // reads, even for 8-byte row reads (the 2 x 2 register tiles, m <= 32)
  static constexpr int LDM = MB <= 4 ? MP + 2 : MP + 1;
  static constexpr size_t MATP = sizeof(float) * MP * LDM;             // m x m matrices
  // for m > 32 the five m x m matrices reuse the warp-partial region, dead
  // once the CTA partial is formed (NW = 8 >= 5); no ring is used there
  static constexpr bool ALIAS = MB > 4;
  static constexpr size_t gram_w = 0;                       // NW warp partials
  static constexpr size_t mat_a = ALIAS ? 0 : gram_w + NW * MAT;   // A_t
  static constexpr size_t mat_p = mat_a + MATP;              // P_t
  static constexpr size_t mat_q = mat_p + MATP;              // Q_t = P_{t-1} ... P_0
  static constexpr size_t mat_t1 = mat_q + MATP;             // scratch products
  static constexpr size_t mat_t2 = mat_t1 + MATP;
  static constexpr size_t gram_c = ALIAS ? gram_w + NW * MAT : mat_t2 + MATP;  // CTA partial
  static constexpr size_t qh = gram_c + MAT;                // bf16 Q, the MMA A operand
  static constexpr size_t bars = (qh + sizeof(__nv_bfloat16) * MPX * MPX + 15) & ~size_t(15);
  static constexpr size_t misc = bars + 12 * 8 + 12 * 4;    // 12 mbarriers, 12 counters
  static constexpr size_t ring = (misc + 64 * sizeof(float) + 16 + 127) & ~size_t(127);
  // ring of row stages (bulk copies), SW columns = one superchunk per warp;
  // row pitches padded so the fragment reads of a warp hit distinct banks.
  // Pass 1 stages hold G and M rows; pass 2 stages only W rows, two
  // superchunks per warp (2 SW columns: half the copies and half the stage
  // hand-offs of single-width stages).
  static constexpr int SW = 32 * NW;
  static constexpr int PITCH_G = SW * ES + (ES == 2 ? 32 : 64);
  static constexpr int PITCH_M = SW * 4 + 64;
  static constexpr size_t STAGE = (size_t)MP * (PITCH_G + PITCH_M);
  static constexpr int PITCH_W = 2 * SW * ES + (ES == 2 ? 32 : 64);
  static constexpr size_t STAGE_W = (size_t)MP * PITCH_W;
  static constexpr size_t BUDGET = 224 * 1024 > ring ? 224 * 1024 - ring : 0;
  static constexpr int FIT = (int)(BUDGET / STAGE);
  static constexpr bool STAGED = !ALIAS && FIT >= 2;
  static constexpr int NSTAGE = !STAGED ? 0 : (FIT >= 4 ? 4 : FIT);
  static constexpr size_t RING = STAGED ? NSTAGE * STAGE : 0;
  static constexpr int NSTAGE_W = !STAGED ? 0 : ((int)(RING / STAGE_W) >= 8 ? 8 : (int)(RING / STAGE_W));
  static constexpr size_t total = ring + RING;
  // one CTA per SM: a second CTA on the SM would wait for tensor memory
  static constexpr size_t launch = total > 120 * 1024 ? total : 120 * 1024;
  static_assert(!STAGED || (NSTAGE >= 2 && NSTAGE_W >= 2), "ring depth");
  static_assert(launch <= 227 * 1024, "shared memory");
};

// Gram tiles: rows 16P..16P+15 (row blocks 2P, 2P+1) x row block J, J >= 2P.
__device__ __forceinline__ bool gram_covered(int i, int j) {
  const int I = i >> 3, J = j >> 3;
  return J >= ((I >> 1) << 1);
}

__device__ __forceinline__ void mma_k16_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_k8_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

// X X^T partial of one superchunk (bf16 fragments, fp32 accumulation)
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
      for (int J = 2 * P; J < MB; ++J)
        mma_k16_bf16(acc[P][J], a0, a1, a2, a3, x[J][2 * k], x[J][2 * k + 1]);
    }
}

// Register tile of the m x m products: TB x TB outputs per thread, (MP/TB)^2
// threads busy, the smallest TB whose thread count fits the CTA.
template <int MP, int NT>
struct MatTile {
  static constexpr int TB = (MP / 2) * (MP / 2) <= NT ? 2 : ((MP + 2) / 3) * ((MP + 2) / 3) <= NT ? 3 : 4;
  static constexpr int NB = (MP + TB - 1) / TB;
  static_assert(NB * NB <= NT, "tile");
};

// D[i][j] = sum_k A[i][k] B[k][j]  (+ fused P epilogue when MODE == 1:
// D = c*(A A) + b*A + a*I, with B == A), MP x MP fp32 in shared memory with
// rows LDM floats apart (LDM = MP + 2 for the 2 x 2 tiles, else MP + 1).
//
// Every left operand of the recursion is symmetric in exact arithmetic (A_t,
// P_t and P_t A_t are polynomials in A_0), so with 2 x 2 tiles its column
// k is read as row k: both operands then come in 8-byte row reads.  The
// transposed read differs from the direct one by fp32 rounding only.
template <int MP, int NT, int MODE>
__device__ __forceinline__ void mat_mul(float* D, const float* A, const float* B, int tid,
                                        float a = 0.f, float b = 0.f, float c = 0.f) {
  using T = MatTile<MP, NT>;
  constexpr int TB = T::TB, NB = T::NB;
  constexpr int LDM = TB == 2 ? MP + 2 : MP + 1;
  if (tid >= NB * NB) return;
  const int i0 = (tid / NB) * TB, j0 = (tid % NB) * TB;
  float acc[TB][TB];
  #pragma unroll
  for (int x = 0; x < TB; ++x)
    #pragma unroll
    for (int y = 0; y < TB; ++y) acc[x][y] = 0.f;
  // fully unrolled for the small m of this kernel: every shared-memory load
  // of the product is issued before the dependent FMA chain runs
  #pragma unroll
  for (int k = 0; k < MP; ++k) {
    float av[TB], bv[TB];
    if constexpr (TB == 2) {
      // MP is a multiple of 8 and i0, j0 are even: both pairs exist
      const float2 ap = *reinterpret_cast<const float2*>(A + k * LDM + i0);
      const float2 bp = *reinterpret_cast<const float2*>(B + k * LDM + j0);
      av[0] = ap.x; av[1] = ap.y; bv[0] = bp.x; bv[1] = bp.y;
    } else {
      #pragma unroll
      for (int x = 0; x < TB; ++x) av[x] = (i0 + x < MP) ? A[(i0 + x) * LDM + k] : 0.f;
      #pragma unroll
      for (int y = 0; y < TB; ++y) bv[y] = (j0 + y < MP) ? B[k * LDM + j0 + y] : 0.f;
    }
    #pragma unroll
    for (int x = 0; x < TB; ++x)
      #pragma unroll
      for (int y = 0; y < TB; ++y) acc[x][y] = fmaf(av[x], bv[y], acc[x][y]);
  }
  #pragma unroll
  for (int x = 0; x < TB; ++x)
    #pragma unroll
    for (int y = 0; y < TB; ++y) {
      const int i = i0 + x, j = j0 + y;
      if (i < MP && j < MP) {
        float v = acc[x][y];
        if (MODE == 1) v = fmaf(c, v, fmaf(b, A[i * LDM + j], i == j ? a : 0.f));
        D[i * LDM + j] = v;
      }
    }
}

// The whole Muon step of one slice per cluster.
//
// Newton-Schulz in Gram space: with A_t = X_t X_t^T each step is
// X_{t+1} = P_t X_t, P_t = a I + b A_t + c A_t^2, a polynomial in A_t, hence
// symmetric and commuting with A_t, so A_{t+1} = P_t A_t P_t and
// X_T = (P_{T-1} ... P_0) X_0 = Q X_0.  The iteration is thus carried out
// exactly on m x m matrices: one pass over the slice forms A_0, the m x m
// recursion gives Q, one more pass applies O = Q X_0.
// STG: compile the row-streaming (ring) path; the direct path is the general
// fallback (transposed slices, unaligned rows, m > 32).  Separate
// instantiations keep the register budget of each path to itself.
template <int MB, int NW, typename PT, bool STG>
__global__ void __launch_bounds__(NW * 32, 1) skinny_kernel(const __grid_constant__ SkinnyParams p) {
  using S = SkinnySmem<MB, NW, (int)sizeof(PT)>;
  constexpr int MP = S::MP, NP = S::NP, MPX = S::MPX;
  constexpr int NT = NW * 32;
  constexpr int COLS_W = 512 / (NW / 4);
  constexpr int LOOKAHEAD = 3;   // superchunks prefetched into L2 ahead of use (direct path)
  constexpr int NSTG = S::NSTAGE > 0 ? S::NSTAGE : 1;
  constexpr int NSTW = S::NSTAGE_W > 0 ? S::NSTAGE_W : 1;
  extern __shared__ __align__(128) unsigned char smem[];
  float* gram_w = reinterpret_cast<float*>(smem + S::gram_w);
  float* gram_c = reinterpret_cast<float*>(smem + S::gram_c);
  float* mA = reinterpret_cast<float*>(smem + S::mat_a);
  float* mP = reinterpret_cast<float*>(smem + S::mat_p);
  float* mQ = reinterpret_cast<float*>(smem + S::mat_q);
  float* mT1 = reinterpret_cast<float*>(smem + S::mat_t1);
  float* mT2 = reinterpret_cast<float*>(smem + S::mat_t2);
  __nv_bfloat16* qh = reinterpret_cast<__nv_bfloat16*>(smem + S::qh);
  float* red = reinterpret_cast<float*>(smem + S::misc);     // NW floats
  float* norm_slot = red + 32;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red + 48);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::bars);  // pass-1 stage landed
  uint64_t* full_w = full + 4;                                      // pass-2 stage landed
  int* done_cnt = reinterpret_cast<int*>(smem + S::bars + 96);     // warps done with a stage
  int* done_w = done_cnt + 4;

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
  // a loss-scaled step whose gradients hold an inf or NaN changes nothing
  if (st.skip && *st.skip) return;

  for (int e = tid; e < MPX * MPX; e += NT) qh[e] = __float2bfloat16_rn(0.f);
  constexpr bool staged = S::STAGED && STG;
  if (tid == 0) {
    for (int b = 0; b < 12; ++b) { mbar_init(&full[b], 1); done_cnt[b] = 0; }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
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

  // slot q of warp w is superchunk jc0 + w + q*NW: at any moment the CTA's
  // warps stream one contiguous stretch of every row
  const int jc0 = rank * p.sc_per_cta;
  const int jc1 = min(p.nsc, jc0 + p.sc_per_cta);
  const int nslot = max(0, (jc1 - jc0 - warp + NW - 1) / NW);
  auto sc_col = [&](int q) { return (jc0 + warp + q * NW) * 32; };

  const int c_lo = jc0 * 32, c_hi = min(p.n, jc1 * 32);
  const int nstage = jc1 > jc0 ? (c_hi - c_lo + S::SW - 1) / S::SW : 0;   // pass-1 stages
  const int nstage_w = (nstage + 1) / 2;                                      // pass-2 stages
  // live: this thread stores results.  Cleared when one of its waits gave
  // up, or when the error word was set (by an earlier kernel of the step or
  // another cluster); the control flow, the cluster syncs and the waits for
  // copies in flight stay the same, only the stores stop.
  bool live = *static_cast<volatile int*>(p.err) == 0;
  // Rows [part*R, (part+1)*R) of stage k of pass `w2` (0: G and M rows,
  // columns [c_lo + k*SW, ...); 1: W rows, columns [c_lo + 2k*SW, ...)); one
  // warp issues them, one row per lane.  Part 0 posts the stage's byte count (copies of other parts may
  // land first: the phase cannot complete before that arrive).
  auto issue_stage = [&](int k, int w2, int part = 0, int nparts = 1) {
    if (!S::STAGED) return;
    const int width = w2 ? 2 * S::SW : S::SW;
    const int c0 = c_lo + k * width;
    const int cols = min(width, c_hi - c0);
    uint64_t* bar = w2 ? &full_w[k % NSTW] : &full[k % NSTG];
    unsigned char* base = smem + S::ring + (w2 ? (size_t)(k % NSTW) * S::STAGE_W : (size_t)(k % NSTG) * S::STAGE);
    if (part == 0 && lane == 0)
      mbar_expect_tx(bar, (uint32_t)(p.m * cols * ((int)sizeof(PT) + (w2 ? 0 : 4))));
    __syncwarp();
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    const int R = (p.m + nparts - 1) / nparts;
    const int r1 = min(p.m, (part + 1) * R);
    for (int i = part * R + lane; i < r1; i += 32) {
      const PT* src = w2 ? W : G;
      bulk_load(base + i * (w2 ? S::PITCH_W : S::PITCH_G), src + (size_t)i * p.n + c0,
                cols * (int)sizeof(PT), bar);
      if (!w2)
        bulk_load(base + MP * S::PITCH_G + i * S::PITCH_M, Mo + (size_t)i * p.n + c0, cols * 4, bar);
    }
  };
  // every warp calls this when done with stage k; the last one refills the
  // buffer with stage k + depth of the same pass
  auto release_stage = [&](int k, int w2) {
    __syncwarp();
    const int depth = w2 ? NSTW : NSTG;
    int last = 0;
    if (lane == 0) {
      int* cnt = w2 ? &done_w[k % NSTW] : &done_cnt[k % NSTG];
      __threadfence_block();
      if (atomicAdd(cnt, 1) == NW - 1) { *cnt = 0; last = 1; }
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last && k + depth < (w2 ? nstage_w : nstage)) issue_stage(k + depth, w2);
  };
  auto stage_wait = [&](int k, int w2) {
    uint64_t* bar = w2 ? &full_w[k % NSTW] : &full[k % NSTG];
    const uint32_t par = (uint32_t)((k / (w2 ? NSTW : NSTG)) & 1);
    if (!mbar_wait(bar, par, st.wait_limit)) {
      if (live) atomicExch(p.err, kDevErrTimeout);
      live = false;
      // the stage's copies are still owed to this buffer: wait for them
      // with the normal budget before it is read or refilled
      mbar_wait(bar, par);
    }
  };
  // L2 prefetch of one superchunk's gradient and momentum rows (direct path)
  auto prefetch_sc = [&](int q) {
    if (staged || !p.vec || q >= nslot) return;
    const int cb = sc_col(q);
    for (int i = lane; i < p.m; i += 32) {
      const size_t off = (size_t)i * p.n + cb;
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"(G + off));
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"(Mo + off));
    }
  };
  // the initial stages are issued by all warps, a few rows each (a bulk copy
  // takes tens of cycles to issue; spread out, no warp falls behind)
  if (staged) {
    const int ns0 = min(NSTG, nstage), parts = NW / NSTG;
    if (warp / parts < ns0) issue_stage(warp / parts, 0, warp % parts, parts);
  }
  for (int q = 0; q < LOOKAHEAD; ++q) prefetch_sc(q);

  static_assert(S::LDM == (MatTile<MP, NT>::TB == 2 ? MP + 2 : MP + 1), "m x m row pitch");
  // threads of the m x m recursion; SPLIT: the remaining warps are idle then
  constexpr int NB2 = MatTile<MP, NT>::NB * MatTile<MP, NT>::NB;
  constexpr int RT = 2 * NB2 <= NT ? (2 * NB2 + 31) / 32 * 32 : NT;
  constexpr bool SPLIT = staged && RT < NT;

  // ---- pass 1: momentum, V (bf16 in TMEM), sum of squares, Gram of V ----------
  float ss = 0.f;
  float gacc[NP][MB][4];
  #pragma unroll
  for (int P = 0; P < NP; ++P)
    #pragma unroll
    for (int J = 0; J < MB; ++J)
      #pragma unroll
      for (int e = 0; e < 4; ++e) gacc[P][J][e] = 0.f;
  const int npass = staged ? nstage : nslot;
  // staged path: rows start 16-byte aligned and columns are whole 4-groups,
  // so a lane's accesses reduce to a row base plus a column
  float* mo_row[MB];
  #pragma unroll
  for (int rb = 0; rb < MB; ++rb) mo_row[rb] = Mo + (size_t)(rb * 8 + g < p.m ? rb * 8 + g : 0) * p.n;
  auto row_ok = [&](int rb) { return rb * 8 + g < p.m; };
  for (int q = 0; q < npass; ++q) {
    const bool has = q < nslot;       // warp has a superchunk in this stage
    float gv[MB][2][4], mv[MB][2][4];
    if (staged) {
      stage_wait(q, 0);
      const unsigned char* base = smem + S::ring + (size_t)(q % NSTG) * S::STAGE;
      #pragma unroll
      for (int rb = 0; rb < MB; ++rb)
        #pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = rb * 8 + g;
          const int cl = warp * 32 + h * 16 + 4 * t4;   // column inside the stage
          const bool in = has && row_ok(rb) && sc_col(q) + h * 16 + 4 * t4 < p.n;
          if (in) {
            if constexpr (sizeof(PT) == 2) {
              const uint2 u = *reinterpret_cast<const uint2*>(base + i * S::PITCH_G + cl * 2);
              const float2 x = unpack_bf16(u.x), y = unpack_bf16(u.y);
              gv[rb][h][0] = x.x; gv[rb][h][1] = x.y; gv[rb][h][2] = y.x; gv[rb][h][3] = y.y;
            } else {
              const float4 u = *reinterpret_cast<const float4*>(base + i * S::PITCH_G + cl * 4);
              gv[rb][h][0] = u.x; gv[rb][h][1] = u.y; gv[rb][h][2] = u.z; gv[rb][h][3] = u.w;
            }
            const float4 u = *reinterpret_cast<const float4*>(base + MP * S::PITCH_G + i * S::PITCH_M + cl * 4);
            mv[rb][h][0] = u.x; mv[rb][h][1] = u.y; mv[rb][h][2] = u.z; mv[rb][h][3] = u.w;
          } else {
            #pragma unroll
            for (int e = 0; e < 4; ++e) gv[rb][h][e] = mv[rb][h][e] = 0.f;
          }
        }
      release_stage(q, 0);
    } else {
      prefetch_sc(q + LOOKAHEAD);
      const int cb = sc_col(q);
      #pragma unroll
      for (int rb = 0; rb < MB; ++rb)
        #pragma unroll
        for (int h = 0; h < 2; ++h) {
          acc_.template load<true>(G, rb * 8 + g, cb + h * 16 + 4 * t4, gv[rb][h]);
          acc_.load_f32(Mo, rb * 8 + g, cb + h * 16 + 4 * t4, mv[rb][h]);
        }
    }
    if (!has) continue;
    const int cb = sc_col(q);
    uint32_t xr[MB][4];
    #pragma unroll
    for (int rb = 0; rb < MB; ++rb)
      #pragma unroll
      for (int h = 0; h < 2; ++h) {
        float vv[4];
        #pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float gg = gv[rb][h][e] * st.gscale;
          const float mm = fmaf(st.beta, mv[rb][h][e], gg);
          mv[rb][h][e] = mm;
          vv[e] = st.nesterov ? fmaf(st.beta, mm, gg) : mm;
          ss = fmaf(vv[e], vv[e], ss);
        }
        if (staged) {
          const int c = cb + h * 16 + 4 * t4;
          if (live && row_ok(rb) && c < p.n)
            *reinterpret_cast<float4*>(mo_row[rb] + c) =
                make_float4(mv[rb][h][0], mv[rb][h][1], mv[rb][h][2], mv[rb][h][3]);
        } else if (live) {
          acc_.store_f32(Mo, rb * 8 + g, cb + h * 16 + 4 * t4, mv[rb][h]);
        }
        xr[rb][2 * h] = pack_bf16(vv[0], vv[1]);
        xr[rb][2 * h + 1] = pack_bf16(vv[2], vv[3]);
      }
    #pragma unroll
    for (int rb = 0; rb < MB; ++rb) tm_st4(taddr_w + q * 4 * MB + 4 * rb, xr[rb]);
    gram_accum<MB>(gacc, xr);
  }

  // warm L2 with this CTA's parameter rows for the final update, columns
  // [c0, end of the CTA's range); one warp
  auto prefetch_w_l2 = [&](int c0) {
    const size_t es = sizeof(PT);
    const int c1 = min(p.n, jc1 * 32);
    if (c1 <= c0) return;
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
  };
  // (with idle warps during the recursion, they warm it there instead)
  if (!SPLIT && warp == NW - 1 && jc1 > jc0) prefetch_w_l2(jc0 * 32);

  // ---- cluster-wide ||V||^2 and V V^T (fixed order: warps, then ranks) -----------
  __syncthreads();   // every pass-1 stage is consumed: the ring takes W rows
  {
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
  }
  #pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[warp] = ss;
  tm_wait_st();
  // The parameter rows of pass 2 start streaming while the reductions and
  // the m x m recursion run.  When the recursion leaves warps idle, those
  // warps issue the copies during it (issuing a bulk copy takes tens of
  // cycles, which would otherwise delay the reductions).
  if (staged && !SPLIT) {
    const int ns0 = min(NSTW, nstage_w), parts = NW / NSTW;
    if (warp / parts < ns0) issue_stage(warp / parts, 1, warp % parts, parts);
  }
  __syncthreads();
  for (int e = tid; e < MP * MP; e += NT) {
    if (!gram_covered(e / MP, e % MP)) continue;
    float s = 0.f;
    for (int w = 0; w < NW; ++w) s += gram_w[w * MP * MP + e];
    gram_c[e] = s;
  }
  if (tid == 0) {
    float s = 0.f;
    for (int w = 0; w < NW; ++w) s += red[w];
    norm_slot[0] = s;
  }
  cluster.sync();
  float tot = 0.f;
  for (int r = 0; r < p.cluster; ++r) tot += *cluster.map_shared_rank(norm_slot, r);
  const float inv = 1.f / (sqrtf(tot) + st.eps);
  for (int e = tid; e < MP * MP; e += NT) {
    const int i = e / MP, j = e % MP;
    const int src = gram_covered(i, j) ? e : j * MP + i;
    float s = 0.f;
    for (int r = 0; r < p.cluster; ++r) s += cluster.map_shared_rank(gram_c, r)[src];
    mA[i * S::LDM + j] = s * inv * inv;           // A_0 = X_0 X_0^T
    mQ[i * S::LDM + j] = i == j ? 1.f : 0.f;
  }
  __syncthreads();

  // ---- m x m recursion: P_t = aI + bA_t + cA_t^2;  Q <- P_t Q;  A <- P_t A_t P_t ----
  // The first RT threads run it, synchronised by a named barrier of their own
  // when that leaves warps over; those issue the parameter-row copies.
  auto rsync = [&]() {
    if constexpr (SPLIT) asm volatile("bar.sync 1, %0;\n" ::"n"(RT) : "memory");
    else __syncthreads();
  };
  if (!SPLIT || tid < RT) {
    for (int t = 0; t < st.T; ++t) {
      mat_mul<MP, NT, 1>(mP, mA, mA, tid, st.a, st.b, st.c);   // P = aI + bA + cA^2
      rsync();
      // Q <- P Q and P A on disjoint thread sets when both fit
      if (2 * NB2 <= NT) {
        if (tid < NB2) mat_mul<MP, NT, 0>(mT1, mP, mQ, tid);
        else if (t + 1 < st.T) mat_mul<MP, NT, 0>(mT2, mP, mA, tid - NB2);
      } else {
        mat_mul<MP, NT, 0>(mT1, mP, mQ, tid);
        if (t + 1 < st.T) mat_mul<MP, NT, 0>(mT2, mP, mA, tid);
      }
      rsync();
      { float* x = mQ; mQ = mT1; mT1 = x; }
      if (t + 1 < st.T) {
        mat_mul<MP, NT, 0>(mA, mT2, mP, tid);                    // A <- (P A) P
        rsync();
      }
    }
  } else {
    // one stage per idle warp, round robin; the last idle warp then warms L2
    // with the columns the ring does not hold yet
    constexpr int IW = (NT - RT) / 32;
    const int ns0 = min(NSTW, nstage_w);
    for (int k = warp - RT / 32; k < ns0; k += IW) issue_stage(k, 1);
    if (warp == NW - 1) prefetch_w_l2(c_lo + ns0 * 2 * S::SW);
    for (int t = 0; t < st.T; ++t) { float* x = mQ; mQ = mT1; mT1 = x; }
  }
  if constexpr (SPLIT) __syncthreads();
  // O = Q X_0 = (Q * inv) V; the bf16 A operand is the scaled Q.  When O is
  // not an output, the update's factor -lr s is folded in too, so that the
  // product is the update term itself: W' = W (1 - lr wd) + (-lr s inv Q) V
  // (ring-staged path)
  const bool fold = staged && Oout == nullptr;
  const float qscale = tot > 0.f ? (fold ? -p.lrs * inv : inv) : 0.f;
  for (int e = tid; e < MP * MP; e += NT) {
    const int i = e / MP, j = e % MP;
    qh[i * MPX + j] = __float2bfloat16_rn(mQ[i * S::LDM + j] * qscale);
  }
  __syncthreads();
  uint32_t afr[NP][NP][4];
  #pragma unroll
  for (int P = 0; P < NP; ++P)
    #pragma unroll
    for (int kk = 0; kk < NP; ++kk) {
      const __nv_bfloat16* r0 = qh + (16 * P + g) * MPX + 16 * kk + 2 * t4;
      const __nv_bfloat16* r1 = r0 + 8 * MPX;
      afr[P][kk][0] = *reinterpret_cast<const uint32_t*>(r0);
      afr[P][kk][1] = *reinterpret_cast<const uint32_t*>(r1);
      afr[P][kk][2] = *reinterpret_cast<const uint32_t*>(r0 + 8);
      afr[P][kk][3] = *reinterpret_cast<const uint32_t*>(r1 + 8);
    }

  // ---- pass 2: O = Q X_0 and W' = W (1 - lr wd) - lr s O -------------------------
  // a wait that gave up anywhere before the cluster sync (this cluster's
  // reduction included) leaves every parameter untouched
  live = live && *static_cast<volatile int*>(p.err) == 0;
  float wbuf[MB][2][4];
  auto load_w = [&](int q) {
    const int cb = sc_col(q);
    #pragma unroll
    for (int rb = 0; rb < MB; ++rb)
      #pragma unroll
      for (int h = 0; h < 2; ++h)
        acc_.template load<false>(W, rb * 8 + g, cb + h * 16 + 4 * t4, wbuf[rb][h]);
  };
  if (!staged && nslot > 0) load_w(0);
  // V of the next superchunk is read from tensor memory one iteration ahead
  uint32_t xn[MB][4];
  if (nslot > 0) {
    #pragma unroll
    for (int rb = 0; rb < MB; ++rb) tm_ld4(taddr_w + 4 * rb, xn[rb]);
  }
  for (int q = 0; q < npass; ++q) {
    const bool has = q < nslot;
    float wcur[MB][2][4];
    if (staged) {
      // superchunks q and q + 1 (q even) share one double-width stage
      const int k2 = q >> 1;
      if ((q & 1) == 0) stage_wait(k2, 1);
      const unsigned char* base = smem + S::ring + (size_t)(k2 % NSTW) * S::STAGE_W;
      #pragma unroll
      for (int rb = 0; rb < MB; ++rb)
        #pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = rb * 8 + g;
          const int cl = (q & 1) * S::SW + warp * 32 + h * 16 + 4 * t4;
          const bool in = has && row_ok(rb) && sc_col(q) + h * 16 + 4 * t4 < p.n;
          if (in) {
            if constexpr (sizeof(PT) == 2) {
              const uint2 u = *reinterpret_cast<const uint2*>(base + i * S::PITCH_W + cl * 2);
              const float2 x = unpack_bf16(u.x), y = unpack_bf16(u.y);
              wcur[rb][h][0] = x.x; wcur[rb][h][1] = x.y; wcur[rb][h][2] = y.x; wcur[rb][h][3] = y.y;
            } else {
              const float4 u = *reinterpret_cast<const float4*>(base + i * S::PITCH_W + cl * 4);
              wcur[rb][h][0] = u.x; wcur[rb][h][1] = u.y; wcur[rb][h][2] = u.z; wcur[rb][h][3] = u.w;
            }
          } else {
            #pragma unroll
            for (int e = 0; e < 4; ++e) wcur[rb][h][e] = 0.f;
          }
        }
      // the stage is handed back after its second superchunk (or the last)
      if ((q & 1) == 1 || q + 1 == npass) release_stage(k2, 1);
    } else {
      #pragma unroll
      for (int rb = 0; rb < MB; ++rb)
        #pragma unroll
        for (int h = 0; h < 2; ++h)
          #pragma unroll
          for (int e = 0; e < 4; ++e) wcur[rb][h][e] = wbuf[rb][h][e];
      if (q + 1 < nslot) load_w(q + 1);
    }
    if (!has) continue;
    tm_wait_ld();
    uint32_t xr[MB][4];
    #pragma unroll
    for (int rb = 0; rb < MB; ++rb)
      #pragma unroll
      for (int r = 0; r < 4; ++r) xr[rb][r] = xn[rb][r];
    if (q + 1 < nslot) {
      #pragma unroll
      for (int rb = 0; rb < MB; ++rb) tm_ld4(taddr_w + (q + 1) * 4 * MB + 4 * rb, xn[rb]);
    }
    float o[MB][4][2];
    #pragma unroll
    for (int r = 0; r < 4; ++r) {
      uint32_t xt[MB];
      #pragma unroll
      for (int J = 0; J < MB; ++J) xt[J] = movt(xr[J][r]);
      #pragma unroll
      for (int P = 0; P < NP; ++P) {
        float y[4] = {0.f, 0.f, 0.f, 0.f};
        #pragma unroll
        for (int kk = 0; kk < NP; ++kk) {
          if (2 * kk + 1 < MB)
            mma_k16_bf16(y, afr[P][kk][0], afr[P][kk][1], afr[P][kk][2], afr[P][kk][3], xt[2 * kk],
                    xt[(2 * kk + 1) % MB]);
          else
            mma_k8_bf16(y, afr[P][kk][0], afr[P][kk][1], xt[2 * kk]);
        }
        o[2 * P][r][0] = y[0];
        o[2 * P][r][1] = y[1];
        if (2 * P + 1 < MB) {
          o[(2 * P + 1) % MB][r][0] = y[2];
          o[(2 * P + 1) % MB][r][1] = y[3];
        }
      }
    }
    const int cb = sc_col(q);
    if (fold) {
      // o holds -lr s O: one multiply-add per parameter
      #pragma unroll
      for (int rb = 0; rb < MB; ++rb)
        #pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = cb + h * 16 + 4 * t4;
          if (live && row_ok(rb) && c < p.n) {
            float wn[4];
            wn[0] = fmaf(wcur[rb][h][0], p.decay, o[rb][2 * h][0]);
            wn[1] = fmaf(wcur[rb][h][1], p.decay, o[rb][2 * h][1]);
            wn[2] = fmaf(wcur[rb][h][2], p.decay, o[rb][2 * h + 1][0]);
            wn[3] = fmaf(wcur[rb][h][3], p.decay, o[rb][2 * h + 1][1]);
            PT* wp = W + (mo_row[rb] - Mo) + c;     // same row offset as the momentum
            if constexpr (sizeof(PT) == 2) {
              uint2 u;
              u.x = pack_bf16(wn[0], wn[1]);
              u.y = pack_bf16(wn[2], wn[3]);
              *reinterpret_cast<uint2*>(wp) = u;
            } else {
              *reinterpret_cast<float4*>(wp) = make_float4(wn[0], wn[1], wn[2], wn[3]);
            }
          }
        }
      continue;
    }
    #pragma unroll
    for (int rb = 0; rb < MB; ++rb)
      #pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = rb * 8 + g, c = cb + h * 16 + 4 * t4;
        const float ov[4] = {o[rb][2 * h][0], o[rb][2 * h][1], o[rb][2 * h + 1][0],
                             o[rb][2 * h + 1][1]};
        float wn[4];
        #pragma unroll
        for (int e = 0; e < 4; ++e) wn[e] = fmaf(wcur[rb][h][e], p.decay, -p.lrs * ov[e]);
        if (staged) {
          if (live && row_ok(rb) && c < p.n) {
            PT* wp = W + (mo_row[rb] - Mo) + c;     // same row offset as the momentum
            if constexpr (sizeof(PT) == 2) {
              uint2 u;
              u.x = pack_bf16(wn[0], wn[1]);
              u.y = pack_bf16(wn[2], wn[3]);
              *reinterpret_cast<uint2*>(wp) = u;
            } else {
              *reinterpret_cast<float4*>(wp) = make_float4(wn[0], wn[1], wn[2], wn[3]);
            }
            if (Oout)
              *reinterpret_cast<float4*>(Oout + (mo_row[rb] - Mo) + c) = make_float4(ov[0], ov[1], ov[2], ov[3]);
          }
        } else if (live) {
          acc_.store(W, i, c, wn);
          if (Oout) acc_.store_f32(Oout, i, c, ov);
        }
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
  using S = SkinnySmem<MB, NW, (int)sizeof(PT)>;
  auto kern = skinny_kernel<MB, NW, PT, false>;
  if constexpr (S::STAGED) {
    if (prm.staged) kern = skinny_kernel<MB, NW, PT, true>;
  }
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
                          int* err_word, cudaStream_t s) {
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
  // the ring needs 16-byte aligned row starts: rows of a multiple of 8
  // elements and 16-byte aligned slice bases
  int staged = (vec && g.n % 8 == 0 && g.mb <= 4) ? 1 : 0;
  for (int i = 0; i < nslices && staged; ++i) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(ptrs.W[i]) | reinterpret_cast<uintptr_t>(ptrs.G[i]) |
                        reinterpret_cast<uintptr_t>(ptrs.Mom[i]);
    if (a % 16) staged = 0;
  }
  prm.staged = staged;
  prm.err = err_word;
  if (g.dtype == MUON_BF16) return launch_pt<__nv_bfloat16>(g, prm, nslices, s);
  return launch_pt<float>(g, prm, nslices, s);
}

}  // namespace muon
