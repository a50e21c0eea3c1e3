// Batched fp16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA)
// for the dense Newton-Schulz products of one step, with the a, b terms of
// the polynomial folded into the operands so no product reads a third matrix:
//   A = X X^T, A2 = c X X^T + b I   (symmetric: upper tiles only, mirrored;
//                                    two outputs of one accumulator)
//   B' = A A2 + a I                 (symmetric; = b A + c A A + a I)
//   X' = B' X                       (B operand N-major; fp32 on the last step)
// D[b] = alpha * A[b] op(B[b]) + diag * I (and D2 = alpha2 * A op(B) + diag2 * I),
// fp32 accumulation in TMEM.
//
// One persistent CTA per SM, 6 warps:
//   warp 0    TMA producer: 128x64 A box and 256x64 B box per stage (or four
//             64x64 N-major boxes), 4-stage ring, 128-byte swizzle;
//   warp 1    allocates 512 TMEM columns (two 128x256 fp32 accumulators) and
//             one thread issues tcgen05.mma (M=128, N=256, K=16);
//   warps 2-5 epilogue: tcgen05.ld of their 32 TMEM lanes (rows), scaled rows
//             written to a shared-memory staging tile and sent to global
//             memory by TMA tensor stores (32 x 32 boxes; the mirror of a
//             symmetric tile as a transposed staging tile); the accumulator is
//             double-buffered so the epilogue of tile t overlaps the MMAs of
//             tile t+1.
// Every mbarrier wait is bounded; when a budget runs out the kernel records
// an error word, drains its own copies in flight and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_gemm.h"

namespace muon {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN * BK * 2;            // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr int NTHREADS = 192;
constexpr int EPI_BYTES = 8192;                 // staging bytes per epilogue warp

struct TcParams {
  int M, N, K;
  int tiles_m, tiles_n, tiles_per_batch, total_tiles;
  int d_f32;           // D in fp32 (else fp16)
  int has_d2;          // second fp16 output D2
  float alpha, diag;   // D  = alpha  * acc + diag  * I
  float alpha2, diag2; // D2 = alpha2 * acc + diag2 * I
  const char* alpha_base;   // optional per-slice factor of alpha and alpha2
  size_t alpha_stride;
  int sym;
  int b_mn;
  uint32_t idesc;      // M = 128, N = 256
  uint32_t idesc128;   // M = 128, N = 128: tiles with one 128-column half to compute
  int* err;
  const int* skip;
  uint32_t wait_limit;   // polls of a wait on the main path (drains: kWaitLimit)
  // fused parameter update (last product of the step): the epilogue applies
  // W' = W decay - lrs O to the parameter slices instead of storing O
  int fuse;
  int w_f32;           // parameter dtype fp32 (else bf16)
  int wm, wn;          // working dims of a slice (m rows of O, n columns)
  int wtr;             // the parameter is stored transposed ([n, m])
  int wvec;            // rows of every slice start 16-byte aligned (stored rows)
  float decay, lrs;
  void* W[kMaxSlicesPerLaunch];
};

// W' = W decay - lrs O on `cnt` consecutive stored elements row[0..cnt) with
// their O values o[0..cnt); 16-byte accesses when vec and cnt == 32
template <typename PT>
__device__ __forceinline__ void update_run(const TcParams& p, PT* row, const float* o, int cnt,
                                           bool vec) {
  if (vec && cnt == 32) {
    constexpr int E = 16 / sizeof(PT);   // elements per 16-byte access
    #pragma unroll
    for (int k = 0; k < 32 / E; ++k) {
      uint4 u = reinterpret_cast<const uint4*>(row)[k];
      PT* e = reinterpret_cast<PT*>(&u);
      #pragma unroll
      for (int i = 0; i < E; ++i) e[i] = from_f<PT>(fmaf(to_f(e[i]), p.decay, -p.lrs * o[k * E + i]));
      reinterpret_cast<uint4*>(row)[k] = u;
    }
  } else {
    #pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < cnt) row[j] = from_f<PT>(fmaf(to_f(row[j]), p.decay, -p.lrs * o[j]));
  }
}

constexpr int kTrPitch = 36;   // floats per row of the transposing tile (16-byte rows)

// W' = W decay - lrs O for the 32 x 32 outputs of working rows
// [row0, row0 + 32) (lane = row), columns [c0, c0 + 32) (o[] per lane) of
// slice W, stored [m, n], or [n, m] when transposed.  A transposed slice
// goes through a shared-memory tile (32 x kTrPitch floats, `tile`): lane j
// then updates stored row c0 + j, whose 32 elements of columns
// [row0, row0 + 32) are contiguous, so both orientations touch the
// parameters in 64-byte row pieces.  Called by all lanes of the warp.
template <typename PT>
__device__ __forceinline__ void fused_update(const TcParams& p, PT* W, int row0, int c0,
                                             float* o, float* tile) {
  const int lane = threadIdx.x & 31;
  if (!p.wtr) {
    const int r = row0 + lane;
    if (r < p.wm && c0 < p.wn) {
      const int cnt = p.wn - c0 < 32 ? p.wn - c0 : 32;
      update_run<PT>(p, W + (size_t)r * p.wn + c0, o, cnt, p.wvec != 0);
    }
    return;
  }
  // tile[j][i] = O(working row row0 + i, working column c0 + j)
  #pragma unroll
  for (int j = 0; j < 32; ++j) tile[j * kTrPitch + lane] = o[j];
  __syncwarp();
  const int k = c0 + lane;   // stored row
  if (k < p.wn && row0 < p.wm) {
    float t[32];
    #pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 x = reinterpret_cast<const float4*>(tile + lane * kTrPitch)[q];
      t[4 * q] = x.x; t[4 * q + 1] = x.y; t[4 * q + 2] = x.z; t[4 * q + 3] = x.w;
    }
    const int cnt = p.wm - row0 < 32 ? p.wm - row0 : 32;
    update_run<PT>(p, W + (size_t)k * p.wm + row0, t, cnt, p.wvec != 0);
  }
  __syncwarp();   // the tile is rewritten by the next chunk
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// bounded wait for the phase of parity `parity` to complete: at most
// `limit` polls (zero: give up at once)
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

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4, %5}], [%2];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];\n" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
// wait until at most n bulk groups of this thread still read shared memory
__device__ __forceinline__ void bulk_wait_read(int n) {
  if (n >= 3) asm volatile("cp.async.bulk.wait_group.read 3;\n" ::: "memory");
  else if (n == 1) asm volatile("cp.async.bulk.wait_group.read 1;\n" ::: "memory");
  else asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}
__device__ __forceinline__ void sts16(uint32_t a, __half h) {
  asm volatile("st.shared.b16 [%0], %1;\n" ::"r"(a), "h"(__half_as_ushort(h)) : "memory");
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// Staging tiles of 32 x 32 outputs, laid out as the TMA tensor store reads
// them with swizzling: fp16 tiles (64-byte rows) with the 64-byte pattern,
// 16-byte piece j of row r at position j ^ ((r >> 1) & 3); fp32 tiles
// (128-byte rows) with the 128-byte pattern, piece j at j ^ (r & 7).  The 32
// lanes of a warp (one row each) then spread over all shared-memory banks.
// Tiles start on 1024-byte boundaries.
__device__ __forceinline__ void stage_row_h(uint32_t tile, int r, const float* v) {
  #pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float* x = v + 8 * j;
    sts128(tile + r * 64 + ((j ^ ((r >> 1) & 3)) << 4), pack_h2(x[0], x[1]), pack_h2(x[2], x[3]),
           pack_h2(x[4], x[5]), pack_h2(x[6], x[7]));
  }
}
__device__ __forceinline__ void stage_row_f(uint32_t tile, int r, const float* v) {
  #pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float* x = v + 4 * j;
    sts128(tile + r * 128 + ((j ^ (r & 7)) << 4), __float_as_uint(x[0]), __float_as_uint(x[1]),
           __float_as_uint(x[2]), __float_as_uint(x[3]));
  }
}
// column r of a transposed fp16 staging tile (the mirror of row r): element
// (j, r) of the tile, in piece r / 8 of row j
__device__ __forceinline__ void stage_col_h(uint32_t tile, int r, const float* v) {
  const uint32_t within = (uint32_t)(r & 7) * 2;
  #pragma unroll
  for (int j = 0; j < 32; ++j)
    sts16(tile + j * 64 + ((((r >> 3) ^ ((j >> 1) & 3))) << 4) + within, __float2half_rn(v[j]));
}

// shared-memory matrix descriptor, 128-byte swizzle, sm_100 version bits
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;             // descriptor version
  d |= (uint64_t)2 << 61;             // SWIZZLE_128B
  return d;
}

__device__ __forceinline__ void mma_f16(uint32_t dtmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tm_ld32(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// tile index -> (batch, row tile I, col tile J); symmetric outputs only
// enumerate tiles whose second 128-column half reaches the diagonal.  Other
// products run down the columns (row tile fastest): the CTAs in flight then
// share a few column panels of B, read from DRAM once, and sweep the rows of
// A, which stay in L2 (for X' = B' X with X of [4096, 11008] the row-major
// order re-read X about eight times per slice)
__device__ __forceinline__ void tile_coords(const TcParams& p, int t, int& b, int& I, int& J) {
  b = t / p.tiles_per_batch;
  int r = t % p.tiles_per_batch;
  if (!p.sym) {
    I = r % p.tiles_m;
    J = r / p.tiles_m;
    return;
  }
  for (I = 0; I < p.tiles_m; ++I) {
    const int cnt = p.tiles_n - I / 2;
    if (r < cnt) { J = I / 2 + r; return; }
    r -= cnt;
  }
  I = 0; J = 0;  // unreachable for valid t
}

// Epilogue of one accumulator tile for the calling warp (all lanes): its
// 32 rows row0 + lane of 128-row block I, the BN columns from J * BN, read
// from tensor memory at `tacc`; scaled rows (plus the diagonal term) go to
// D (and D2) through the warp's staging slot and TMA tensor stores, a
// symmetric product's block above the diagonal also to its mirror, or, with
// a fused update, into the parameters.  ck counts the chunks staged so far.
__device__ __forceinline__ void epilogue_tile(const TcParams& p, const CUtensorMap* tmD,
                                              const CUtensorMap* tmD2, uint32_t tacc,
                                              unsigned char* epi_slot, int b, int I, int row0,
                                              int J, uint32_t& ck) {
  const int lane = threadIdx.x & 31;
  const uint32_t slot = smem_u32(epi_slot);
  // staging bytes of one 32-column chunk; the slot holds EPI_BYTES / that
  // many chunks in flight
  const int cbytes = (p.d_f32 ? 4096 : 2048) * (p.sym ? 2 : 1) * (p.has_d2 ? 2 : 1);
  const int nbuf = EPI_BYTES / cbytes;
  const int row = row0 + lane;
  float al = p.alpha, al2 = p.alpha2;
  if (p.alpha_base) {
    const float f = *reinterpret_cast<const float*>(p.alpha_base + (size_t)b * p.alpha_stride);
    al *= f;
    al2 *= f;
  }
  #pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    const int col0 = J * BN + c * 32;
    if (col0 >= p.N) continue;
    const int cblk = col0 / 128;
    if (p.sym && cblk < I) continue;  // lower block: written as a mirror by its owner
    const bool mirror = p.sym && cblk > I;
    float v[32], v2[32];
    tm_ld32(tacc + c * 32, v);
    const bool dg = row >= col0 && row < col0 + 32;   // the diagonal crosses this row
    #pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float d = (dg && col0 + j == row) ? 1.f : 0.f;
      v2[j] = fmaf(al2, v[j], d * p.diag2);
      v[j] = fmaf(al, v[j], d * p.diag);
    }
    if (p.fuse) {
      float* tile = reinterpret_cast<float*>(epi_slot);
      if (p.w_f32) fused_update<float>(p, static_cast<float*>(p.W[b]), row0, col0, v, tile);
      else fused_update<__nv_bfloat16>(p, static_cast<__nv_bfloat16*>(p.W[b]), row0, col0, v, tile);
      continue;
    }
    // the staging buffer of this chunk is free once the stores issued from
    // it nbuf chunks ago have read it
    if (lane == 0) bulk_wait_read(nbuf - 1);
    __syncwarp();
    const uint32_t buf = slot + (ck % nbuf) * cbytes;
    if (p.d_f32) {
      stage_row_f(buf, lane, v);
    } else {
      stage_row_h(buf, lane, v);
      if (mirror) stage_col_h(buf + 2048, lane, v);
      if (p.has_d2) {
        const uint32_t b2 = buf + (p.sym ? 4096 : 2048);
        stage_row_h(b2, lane, v2);
        if (mirror) stage_col_h(b2 + 2048, lane, v2);
      }
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tmD, buf, col0, row0, b);
      if (mirror) tma_store_3d(tmD, buf + 2048, row0, col0, b);
      if (p.has_d2) {
        const uint32_t b2 = buf + (p.sym ? 4096 : 2048);
        tma_store_3d(tmD2, b2, col0, row0, b);
        if (mirror) tma_store_3d(tmD2, b2 + 2048, row0, col0, b);
      }
      bulk_commit();
    }
    ++ck;
  }
}

__global__ void __launch_bounds__(NTHREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD2,
               const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* epi = smem + STAGES * STAGE_BYTES;      // 4 x EPI_BYTES staging
  uint64_t* full = reinterpret_cast<uint64_t*>(epi + 4 * EPI_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mdrain = tempty + 2;    // completion of every MMA this CTA issued
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdrain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], 1); mbar_init(&tempty[a], 4); }
    mbar_init(mdrain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
                     smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int kblocks = p.K / BK;
  // launched as a dependent of the previous kernel: the setup above overlaps
  // its tail; nothing global is touched before it has completed
  pdl_wait();
  // a skipped loss-scaled step computes nothing, nor does a step in which
  // an earlier kernel's wait gave up
  const bool skipped = (p.skip && *p.skip) || *static_cast<volatile int*>(p.err) != 0;

  auto fail = [&]() {
    *abort_flag = 1;
    atomicExch(p.err, kDevErrTimeout);
  };

  if (skipped) {
    // no role runs; only the teardown below
  } else if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      for (int t = blockIdx.x; t < p.total_tiles && !*abort_flag; t += gridDim.x) {
        int b, I, J;
        tile_coords(p, t, b, I, J);
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, p.wait_limit)) { fail(); break; }
          unsigned char* sa = smem + s * STAGE_BYTES;
          unsigned char* sb = sa + A_BYTES;
          mbar_expect_tx(&full[s], STAGE_BYTES);
          tma_load_3d(sa, &tmA, &full[s], kb * BK, I * BM, b);
          if (!p.b_mn) {
            tma_load_3d(sb, &tmB, &full[s], kb * BK, J * BN, b);
          } else {
            #pragma unroll
            for (int q = 0; q < BN / 64; ++q)
              tma_load_3d(sb + q * (64 * BK * 2), &tmB, &full[s], J * BN + q * 64, kb * BK, b);
          }
        }
      }
      // drain: every issued load must land before the CTA may exit
      const uint32_t last = it;
      for (uint32_t k = (last > STAGES ? last - STAGES : 0); k < last; ++k)
        if (!mbar_wait(&full[k % STAGES], (k / STAGES) & 1)) { fail(); break; }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, tl = 0;
      for (int t = blockIdx.x; t < p.total_tiles && !*abort_flag; t += gridDim.x, ++tl) {
        int b, I, J;
        tile_coords(p, t, b, I, J);
        // a 128-column half of the tile that no epilogue stores is not
        // computed: past N, or (symmetric) the block left of the diagonal
        const int n_lo = (p.sym && 2 * J < I) ? 128 : 0;
        const int n_hi = J * BN + BN > p.N ? p.N - J * BN : BN;
        const uint32_t idesc = n_hi - n_lo == BN ? p.idesc : p.idesc128;
        const uint32_t acc = tl & 1, aph = (tl >> 1) & 1;
        if (!mbar_wait(&tempty[acc], aph ^ 1, p.wait_limit)) { fail(); break; }
        tc_fence_after();
        const uint32_t dt = tmem + acc * BN + n_lo;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&full[s], ph, p.wait_limit)) { fail(); ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
          // K-major B: row n_lo of the tile starts n_lo * 128 bytes in (a
          // whole number of 1024-byte swizzle atoms); N-major B has n_lo = 0
          const uint32_t sb = sa + A_BYTES + n_lo * (BK * 2);
          #pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = sdesc(sa + k * 32, 16, 1024);
            const uint64_t bd = p.b_mn ? sdesc(sb + k * 2048, 64 * BK * 2, 1024)
                                       : sdesc(sb + k * 32, 16, 1024);
            mma_f16(dt, ad, bd, idesc, (kb | k) != 0);
          }
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
      }
      // every MMA issued above completes before the teardown releases the
      // tensor memory (on a wait that gave up, no epilogue may have waited)
      if (it > 0) {
        mma_commit(mdrain);
        if (!mbar_wait(mdrain, 0)) fail();
      }
    }
  } else {
    // epilogue warps 2..5: TMEM lane quarter q = warp % 4, 32 rows each
    const int q = warp & 3;
    uint32_t ck = 0, tl = 0;
    for (int t = blockIdx.x; t < p.total_tiles && !*abort_flag; t += gridDim.x, ++tl) {
      int b, I, J;
      tile_coords(p, t, b, I, J);
      const uint32_t acc = tl & 1, aph = (tl >> 1) & 1;
      if (!mbar_wait(&tfull[acc], aph, p.wait_limit)) { fail(); break; }
      tc_fence_after();
      epilogue_tile(p, &tmD, &tmD2, tmem + ((uint32_t)(q * 32) << 16) + acc * BN, epi + q * EPI_BYTES,
                    b, I, I * BM + q * 32, J, ck);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
    // every store has left shared memory and reached global memory
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem) : "memory");
}

// ---------------------------------------------------------------------------
// Pair kernel: the same products on CTA pairs (thread-block clusters of two
// CTAs on two SMs), with 2-SM MMAs (tcgen05.mma.cta_group::2, M = 256):
// a pair computes a 256 x 256 output tile; CTA r holds rows
// [256 I2 + 128 r, +128) of A and the B rows (K-major) or columns (N-major)
// [256 J + 128 r, +128) in its own shared memory, and its 128 x 256 fp32
// accumulator in its own tensor memory.  Per CTA and k-block a stage is
// 32 KB instead of 48 KB, so six stages are in flight instead of four and a
// CTA moves two thirds of the operand bytes per MMA flop.
//
// Roles per CTA (6 warps): warp 0 loads this CTA's operand halves into its
// own stages; the copies of both CTAs complete on CTA 0's `loaded` barrier,
// which CTA 0's producer arms with the bytes of both halves.  In CTA 0,
// warp 1 issues the pair's MMAs and releases stages and accumulators to both
// CTAs by multicast commits.  Warps 2-5 of both CTAs run the epilogue of
// their 128 rows and report to CTA 0's `tempty` barrier.
//
// Draining: CTA 1 cannot watch the barrier its copies complete on, so when
// its producer stops it stores how many stages it issued into CTA 0's
// shared memory and arrives on CTA 0's `peer_done`; CTA 0's producer then
// waits until every stage either CTA issued has landed (arming the stages
// only CTA 1 issued with CTA 1's bytes, and completing, for stages only CTA
// 0 issued, the bytes CTA 1 never sent) and arrives on CTA 1's `drained`.
// No CTA leaves with a copy in flight.
// A stage of the pair kernel spans PBOX 64-wide TMA boxes of K per operand
// (a 128-byte-swizzled box row holds 64 fp16), so that one barrier wait and
// one commit serve 4 * PBOX MMAs: with one box per stage that per-stage
// work held the tensor pipe's math to 77% of its busy time.  K is a
// multiple of PBK (the dense working dims are padded to 128); other
// products take the one-CTA kernel.
constexpr int PBOX = 2;                            // 64-wide K boxes per stage
constexpr int PBK = PBOX * BK;                     // K per stage
constexpr int PSTAGES = 3;
constexpr int PSUB = 128 * BK * 2;                 // 16 KB: one 64-wide box of A, or of this CTA's B half
constexpr int PA_BYTES = PBOX * PSUB;              // A of one stage
constexpr int PSTAGE_BYTES = 2 * PBOX * PSUB;      // A and this CTA's half of B

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::
                   : "memory");
}
// arrive on a barrier of another CTA of the cluster (shared::cluster address)
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];\n" ::"r"(cluster_addr) : "memory");
}
// the barrier's pending transaction count drops by `bytes` (bytes that will
// never arrive)
__device__ __forceinline__ void mbar_complete_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on a
// barrier of CTA 0 of the pair (shared::cluster address)
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map, uint32_t bar0,
                                                 int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5}], [%2];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar0), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void mma2_f16(uint32_t dtmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
// arrive on the barrier at this offset in both CTAs of the pair once every
// MMA issued so far by this thread has completed
__device__ __forceinline__ void mma2_commit_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;\n" ::"r"(smem_u32(bar)), "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void mma2_commit_local(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// pair tile index -> (batch, 256-row tile I2, 256-column tile J); symmetric
// outputs enumerate the tiles with J >= I2, other products run down the
// columns (as tile_coords)
__device__ __forceinline__ void pair_tile_coords(const TcParams& p, int t, int& b, int& I2, int& J) {
  b = t / p.tiles_per_batch;
  int r = t % p.tiles_per_batch;
  if (!p.sym) {
    I2 = r % p.tiles_m;
    J = r / p.tiles_m;
    return;
  }
  for (I2 = 0; I2 < p.tiles_n; ++I2) {
    const int cnt = p.tiles_n - I2;
    if (r < cnt) { J = I2 + r; return; }
    r -= cnt;
  }
  I2 = 0; J = 0;  // unreachable for valid t
}

__global__ void __launch_bounds__(NTHREADS, 1)
tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD2,
                    const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* epi = smem + PSTAGES * PSTAGE_BYTES;    // 4 x EPI_BYTES staging
  uint64_t* loaded = reinterpret_cast<uint64_t*>(epi + 4 * EPI_BYTES);  // CTA 0: both halves in
  uint64_t* empty = loaded + PSTAGES;    // stage free (multicast commit)
  uint64_t* tfull = empty + PSTAGES;     // accumulator ready (multicast commit)
  uint64_t* tempty = tfull + 2;          // CTA 0: accumulator drained by all 8 epilogue warps
  uint64_t* mdrain = tempty + 2;         // CTA 0: every MMA issued has completed
  uint64_t* peer_done = mdrain + 1;      // CTA 0: CTA 1's producer has stopped
  uint64_t* drained = peer_done + 1;     // CTA 1: every copy of the pair has landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drained + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* peer_issued = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);  // CTA 0
  volatile int* skip_flag = reinterpret_cast<volatile int*>(tmem_slot + 3);  // CTA 1: from CTA 0

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  if (threadIdx.x == 0) {
    for (int s = 0; s < PSTAGES; ++s) { mbar_init(&loaded[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], 1); mbar_init(&tempty[a], 8); }
    mbar_init(mdrain, 1);
    mbar_init(peer_done, 1);
    mbar_init(drained, 1);
    *abort_flag = 0;
    *peer_issued = 0;
    *skip_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  if (warp == 1) {
    // one warp of each CTA of the pair allocates, collectively
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
                     smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // barriers of both CTAs initialised before any remote access
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int kblocks = p.K / PBK;
  pdl_wait();
  // CTA 0 decides for the pair whether the step is skipped (a skipped
  // loss-scaled step, or a wait of the step that gave up), so that both
  // CTAs take the same path
  if (rank == 0 && threadIdx.x == 0) {
    const int sk = (p.skip && *p.skip) || *static_cast<volatile int*>(p.err) != 0;
    asm volatile("st.shared::cluster.u32 [%0], %1;\n" ::"r"(
                     mapa(smem_u32(const_cast<int*>(skip_flag)), 1)),
                 "r"(sk)
                 : "memory");
    *skip_flag = sk;
  }
  cluster_sync_all();
  const bool skipped = *skip_flag != 0;

  auto fail = [&]() {
    *abort_flag = 1;
    atomicExch(p.err, kDevErrTimeout);
  };

  if (skipped) {
    // no role runs; only the teardown below
  } else if (warp == 0) {
    if (lane == 0) {
      // producer: this CTA's halves of every stage
      uint32_t it = 0;
      for (int t = pair; t < p.total_tiles && !*abort_flag; t += npairs) {
        int b, I2, J;
        pair_tile_coords(p, t, b, I2, J);
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % PSTAGES;
          const uint32_t ph = (it / PSTAGES) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, p.wait_limit)) { fail(); ok = false; break; }
          unsigned char* sa = smem + s * PSTAGE_BYTES;
          unsigned char* sb = sa + PA_BYTES;
          const int row = I2 * 256 + (int)rank * 128;
          const int col = J * 256 + (int)rank * 128;
          if (rank == 0) mbar_expect_tx(&loaded[s], 2 * PSTAGE_BYTES);   // both halves
          const uint32_t bar0 = mapa(smem_u32(&loaded[s]), 0);
          #pragma unroll
          for (int h = 0; h < PBOX; ++h) {
            const int k0 = kb * PBK + h * BK;
            unsigned char* ha = sa + h * PSUB;
            unsigned char* hb = sb + h * PSUB;
            if (rank == 0) {
              tma_load_3d(ha, &tmA, &loaded[s], k0, row, b);
              if (!p.b_mn) {
                tma_load_3d(hb, &tmB, &loaded[s], k0, col, b);
              } else {
                #pragma unroll
                for (int q = 0; q < 2; ++q)
                  tma_load_3d(hb + q * (64 * BK * 2), &tmB, &loaded[s], col + q * 64, k0, b);
              }
            } else {
              tma_load_3d_pair(ha, &tmA, bar0, k0, row, b);
              if (!p.b_mn) {
                tma_load_3d_pair(hb, &tmB, bar0, k0, col, b);
              } else {
                #pragma unroll
                for (int q = 0; q < 2; ++q)
                  tma_load_3d_pair(hb + q * (64 * BK * 2), &tmB, bar0, col + q * 64, k0, b);
              }
            }
          }
        }
        if (!ok) break;
      }
      if (rank == 1) {
        // report the stages issued, then wait until CTA 0 has seen them land
        asm volatile("st.shared::cluster.u32 [%0], %1;\n" ::"r"(
                         mapa(smem_u32(const_cast<uint32_t*>(peer_issued)), 0)),
                     "r"(it)
                     : "memory");
        asm volatile("fence.acq_rel.cluster;\n" ::: "memory");
        mbar_arrive_remote(mapa(smem_u32(peer_done), 0));
        if (!mbar_wait(drained, 0)) fail();
      } else {
        if (!mbar_wait(peer_done, 0)) {
          fail();
        } else {
          asm volatile("fence.acq_rel.cluster;\n" ::: "memory");
          const uint32_t it1 = *peer_issued;
          const uint32_t hi = it > it1 ? it : it1;
          for (uint32_t k = (hi > PSTAGES ? hi - PSTAGES : 0); k < hi; ++k) {
            uint64_t* bar = &loaded[k % PSTAGES];
            if (k >= it) mbar_expect_tx(bar, PSTAGE_BYTES);       // CTA 1's half only
            else if (k >= it1) mbar_complete_tx(bar, PSTAGE_BYTES);  // CTA 1 never sent its half
            if (!mbar_wait(bar, (k / PSTAGES) & 1)) { fail(); break; }
          }
        }
        mbar_arrive_remote(mapa(smem_u32(drained), 1));
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // CTA 0: the pair's MMAs (M = 256, N = 256, K = 16)
      uint32_t it = 0, tl = 0;
      for (int t = pair; t < p.total_tiles && !*abort_flag; t += npairs, ++tl) {
        const uint32_t acc = tl & 1, aph = (tl >> 1) & 1;
        if (!mbar_wait(&tempty[acc], aph ^ 1, p.wait_limit)) { fail(); break; }
        tc_fence_after();
        const uint32_t dt = tmem + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % PSTAGES;
          const uint32_t ph = (it / PSTAGES) & 1;
          if (!mbar_wait(&loaded[s], ph, p.wait_limit)) { fail(); ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * PSTAGE_BYTES);
          const uint32_t sb = sa + PA_BYTES;
          #pragma unroll
          for (int k = 0; k < PBK / 16; ++k) {
            const uint32_t h = (uint32_t)(k / (BK / 16)) * PSUB;   // box of this K step
            const int kk = k % (BK / 16);
            const uint64_t ad = sdesc(sa + h + kk * 32, 16, 1024);
            const uint64_t bd = p.b_mn ? sdesc(sb + h + kk * 2048, 64 * BK * 2, 1024)
                                       : sdesc(sb + h + kk * 32, 16, 1024);
            mma2_f16(dt, ad, bd, p.idesc, (kb | k) != 0);
          }
          mma2_commit_both(&empty[s]);
        }
        if (!ok) break;
        mma2_commit_both(&tfull[acc]);
      }
      // every MMA issued above completes before either CTA releases its
      // shared or tensor memory
      if (it > 0) {
        mma2_commit_local(mdrain);
        if (!mbar_wait(mdrain, 0)) fail();
      }
    }
  } else {
    // epilogue warps 2..5 of both CTAs: TMEM lane quarter q, 32 rows each
    const int q = warp & 3;
    uint32_t ck = 0, tl = 0;
    for (int t = pair; t < p.total_tiles && !*abort_flag; t += npairs, ++tl) {
      int b, I2, J;
      pair_tile_coords(p, t, b, I2, J);
      const uint32_t acc = tl & 1, aph = (tl >> 1) & 1;
      if (!mbar_wait(&tfull[acc], aph, p.wait_limit)) { fail(); break; }
      tc_fence_after();
      const int I = 2 * I2 + (int)rank;    // 128-row block of this CTA
      if (I * BM < p.M)                    // past M: rows of zeros, nothing to store
        epilogue_tile(p, &tmD, &tmD2, tmem + ((uint32_t)(q * 32) << 16) + acc * BN,
                      epi + q * EPI_BYTES, b, I, I * BM + q * 32, J, ck);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa(smem_u32(&tempty[acc]), 0));
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // the peer's MMAs and remote accesses are done with this CTA
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, 512;\n" ::"r"(tmem) : "memory");
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D tensor map [batch][outer][inner]: MMA operands (fp16, 128-byte swizzle)
// and epilogue outputs (32 x 32 boxes: fp16 with the 64-byte swizzle, fp32
// with the 128-byte swizzle, matching the staging tiles)
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t batch,
              uint64_t row_bytes, uint64_t batch_bytes, uint32_t box_inner, uint32_t box_outer,
              bool f32 = false, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[3] = {inner, outer, batch};
  const cuuint64_t strides[2] = {row_bytes, batch_bytes};
  const cuuint32_t box[3] = {box_inner, box_outer, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
             const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

}  // namespace

uint32_t tc_idesc_f16(int m, int n, int b_mn) {
  uint32_t d = 0;
  d |= 1u << 4;                        // D format: f32
  d |= 0u << 7;                        // A format: f16
  d |= 0u << 10;                       // B format: f16
  d |= (uint32_t)(b_mn ? 1 : 0) << 16; // B major: 0 = K, 1 = MN
  d |= (uint32_t)(n >> 3) << 17;
  d |= (uint32_t)(m >> 4) << 24;
  return d;
}

size_t tc_gemm_smem_bytes() { return STAGES * STAGE_BYTES + 4 * EPI_BYTES + 1024 + 256; }

// the pair kernel for products with at least one 256-row tile and K a
// multiple of its stage, unless MUON_GEMM=single selects the one-CTA kernel
// (for comparisons)
static bool use_pair_kernel(const TcGemm& g) {
  if (g.M < 256 || g.K % PBK) return false;
  const char* e = std::getenv("MUON_GEMM");
  return !(e && std::strcmp(e, "single") == 0);
}

size_t tc_gemm_pair_smem_bytes() {
  return PSTAGES * PSTAGE_BYTES + 4 * EPI_BYTES + 1024 + 256;
}

// pairs of CTAs that can be resident at once (one CTA per SM), per device
static int max_pairs(size_t smem) {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 76);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_pair_kernel, &cfg) != cudaSuccess || n <= 0)
    n = num_sms() / 2;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

cudaError_t tc_gemm(const TcGemm& g, cudaStream_t s) {
  if (g.M % BM || g.N % 128 || g.K % BK || g.batch < 1 || (g.sym && g.M != g.N))
    return cudaErrorInvalidValue;
  const bool pair = use_pair_kernel(g);
  CUtensorMap ta, tb;
  if (!make_map(&ta, g.A, (uint64_t)g.K, (uint64_t)g.M, (uint64_t)g.batch, (uint64_t)g.K * 2,
                g.stride, BK, BM))
    return cudaErrorInvalidValue;
  const bool ok_b = g.b_mn
      ? make_map(&tb, g.B, (uint64_t)g.N, (uint64_t)g.K, (uint64_t)g.batch, (uint64_t)g.N * 2, g.stride,
                 64, BK)
      : make_map(&tb, g.B, (uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.batch, (uint64_t)g.K * 2, g.stride,
                 BK, pair ? 128 : BN);
  if (!ok_b) return cudaErrorInvalidValue;
  if (g.d_f32 && (g.sym || g.D2)) return cudaErrorInvalidValue;   // mirrors and D2 are fp16
  CUtensorMap td, td2;
  if (!make_map(&td, g.D, (uint64_t)g.N, (uint64_t)g.M, (uint64_t)g.batch,
                (uint64_t)g.N * (g.d_f32 ? 4 : 2), g.stride, 32, 32, g.d_f32 != 0,
                g.d_f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  if (g.D2) {
    if (!make_map(&td2, g.D2, (uint64_t)g.N, (uint64_t)g.M, (uint64_t)g.batch, (uint64_t)g.N * 2,
                  g.stride, 32, 32, false, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  } else {
    td2 = td;
  }
  TcParams p;
  p.M = (int)g.M; p.N = (int)g.N; p.K = (int)g.K;
  p.tiles_n = (int)((g.N + BN - 1) / BN);
  if (pair) {
    // 256 x 256 tiles; symmetric: the tiles with J >= I2
    p.tiles_m = (int)((g.M + 255) / 256);
    p.tiles_per_batch = g.sym ? p.tiles_n * (p.tiles_n + 1) / 2 : p.tiles_m * p.tiles_n;
  } else if (g.sym) {
    p.tiles_m = (int)(g.M / BM);
    int cnt = 0;
    for (int I = 0; I < p.tiles_m; ++I) cnt += p.tiles_n - I / 2;
    p.tiles_per_batch = cnt;
  } else {
    p.tiles_m = (int)(g.M / BM);
    p.tiles_per_batch = p.tiles_m * p.tiles_n;
  }
  p.total_tiles = p.tiles_per_batch * g.batch;
  p.d_f32 = g.d_f32;
  p.has_d2 = g.D2 ? 1 : 0;
  p.fuse = g.W ? 1 : 0;
  if (g.W) {
    if (g.batch > kMaxSlicesPerLaunch || g.sym || g.D2) return cudaErrorInvalidValue;
    p.w_f32 = g.w_f32; p.wm = (int)g.wm; p.wn = (int)g.wn; p.wtr = g.wtr;
    p.decay = g.decay; p.lrs = g.lrs;
    // 16-byte accesses along stored rows: wn (or wm when transposed)
    // elements per stored row
    int vec = 1;
    const size_t es = g.w_f32 ? 4 : 2;
    if ((size_t)(g.wtr ? g.wm : g.wn) * es % 16) vec = 0;
    for (int i = 0; i < g.batch; ++i) {
      p.W[i] = g.W[i];
      if (reinterpret_cast<uintptr_t>(g.W[i]) % 16) vec = 0;
    }
    p.wvec = vec;
  }
  p.alpha = g.alpha; p.diag = g.diag;
  p.alpha2 = g.alpha2; p.diag2 = g.diag2;
  p.alpha_base = static_cast<const char*>(g.alpha_base);
  p.alpha_stride = g.alpha_stride;
  p.sym = g.sym; p.b_mn = g.b_mn;
  p.idesc = pair ? tc_idesc_f16(256, BN, g.b_mn) : tc_idesc_f16(BM, BN, g.b_mn);
  p.idesc128 = tc_idesc_f16(BM, 128, g.b_mn);
  p.err = g.err;
  p.skip = g.skip;
  p.wait_limit = g.wait_limit;
  if (pair) {
    const size_t smem = tc_gemm_pair_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_pair_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int np = max_pairs(smem);
    const int pairs = p.total_tiles < np ? p.total_tiles : np;
    // thread-block clusters of two CTAs, launched as a dependent of the
    // previous kernel of the step
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, tc_gemm_pair_kernel, ta, tb, td, td2, p);
  }
  const size_t smem = tc_gemm_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = p.total_tiles < num_sms() ? p.total_tiles : num_sms();
  // a product always follows another kernel of the step: dependent launch
  return launch_k(tc_gemm_kernel, dim3(grid), dim3(NTHREADS), smem, s, true, ta, tb, td, td2, p);
}

}  // namespace muon
