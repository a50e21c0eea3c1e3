// Dense path of the Muon step: groups whose working matrix is too large for
// the fused on-chip kernel.  Per chunk of slices of one group:
//
//   front      M' = beta*M + G;  V = G + beta*M' | M'  -> V (fp32, working
//              layout [m_pad, n_pad], transposed when M > N), M' in place,
//              per-tile partial sums of V^2               (HBM-bound)
//   finalize   s = 1 / (sqrt(sum of partials) + eps) per slice
//   normalize  X0 = s*V in the iterate type
//   T x        A = X X^T;  B = b*A + c*A*A;  X <- a*X + B*X   (GEMMs)
//   epilogue   W' = W*(1 - lr*wd) - lr*scale*O  in the parameter layout
//
// With fp16 iterates and T > 0 V makes no round trip through memory.  The
// front writes the first iterate as X~ = fp16(V 2^-e) with a per-slice power
// of two e predicted from the slice's previous step, and the first Gram and
// update scale their products by f = 2^e / (||V|| + eps) (f^2 for the Gram),
// so that X~ stands for X0 = f X~.  finalize computes the slice's
// e = 8 floor(log2 ||V|| / 8) - 7, which keeps every |X~| below 2^15 and its
// typical element far above fp16's subnormals; a second pass of the front
// rewrites X~ from G and M' for the slices whose prediction missed.  The
// result never depends on the prediction.
//
// (HyperParallel FSDP Muon RFC, mindspore hyper-parallel issue
// "HyperParallel FSDP Muon优化器性能优化 RFC": section 1(1) momentum input,
// sections 2/3 batched slices, section 6 decoupled weight decay.)
//
// Working buffers are padded to multiples of 128 with zeros.  Zero rows and
// columns stay exactly zero under the iteration (A, B and the update of a
// zero row or column are zero), so padding changes no result.
#include <cstddef>
#include <cstdio>

#include "common.cuh"
#include "internal.h"
#include "gemm.cuh"
#include "tc_gemm.h"

namespace muon {

namespace {

constexpr int kNT = 256;

// per-slice scale slot of the dense path (in the slice's workspace)
struct ScaleSlot {
  float inv;    // 1 / (||V|| + eps)
  float f;      // 2^e / (||V|| + eps): X0 = f X~
  float f2;     // f^2, the first Gram's factor
  int redo;     // the front's exponent was not e: X~ is rewritten
  int e;        // exponent of X~ = fp16(V 2^-e)
};
constexpr int kExpMin = -100, kExpMax = 100;   // 2^-e stays a finite fp32
constexpr int kRedoBlocks = 148;               // blocks per slice of the redo pass

struct DenseBufs {
  float* V;        // [m_pad, n_pad] fp32: front output, then O
  void* X0;        // iterate ping
  void* X1;        // iterate pong
  void* A;         // [m_pad, m_pad]
  void* B;         // [m_pad, m_pad]
  float* part;     // front partial sums
  float* inv;      // per-slice 1/(||V|| + eps)
};

__device__ __forceinline__ void load4(const float* p, float* v) {
  const float4 u = *reinterpret_cast<const float4*>(p);
  v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float* v) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
__device__ __forceinline__ void store4(float* p, const float* v) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, const float* v) {
  uint2 u;
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// vec: every slice's rows start 16-byte aligned (n % 4 == 0, aligned
// bases): 4 consecutive elements per thread, 8-byte bf16 gradient loads (16-
// byte loads of 8 elements per thread measured slower on the dense set:
// 12.5 against 11.2 ms per step)
// OUT: kOutV writes V (fp32); kOutX writes X~ = fp16(V 2^-e) with the
// exponent predicted in exps[]; kOutRedo, for the slices whose prediction
// missed, recomputes V from G and M' (no momentum update, no partial sums)
// and writes X~ with the exact exponent.
enum { kOutV = 0, kOutX = 1, kOutRedo = 2 };

template <typename PT, int OUT>
__global__ void __launch_bounds__(kNT) front_kernel(
    const __grid_constant__ SlicePtrs ptrs, int64_t m, int64_t n, int64_t m_pad,
    int64_t n_pad, int tr, int vec, float beta, int nesterov, float gscale, const int* skip,
    const int* err, char* ws, size_t slice_ws, size_t off_V, size_t off_X, size_t off_part,
    size_t off_slot, const int* exps) {
  pdl_wait();
  // skipped loss-scaled step, or an earlier wait of the step gave up:
  // momentum untouched
  if ((skip && *skip) || *err) return;
  const int s = blockIdx.y;
  char* base = ws + (size_t)s * slice_ws;
  int e = 0;
  if (OUT == kOutRedo) {
    const ScaleSlot* slot = reinterpret_cast<const ScaleSlot*>(base + off_slot);
    if (!slot->redo) return;
    e = slot->e;
  } else if (OUT == kOutX) {
    e = min(max(exps[s], kExpMin), kExpMax);
  }
  const float xs = ldexpf(1.f, -e);   // exact power of two
  const int tiles_c = (int)(n_pad / kFrontTileC);
  float* V = reinterpret_cast<float*>(base + off_V);
  __half* X = reinterpret_cast<__half*>(base + off_X);
  float* part = reinterpret_cast<float*>(base + off_part);
  const PT* G = static_cast<const PT*>(ptrs.G[s]);
  float* Mo = ptrs.Mom[s];
  __shared__ float red[kNT / 32];
  __shared__ float tile[kFrontTileC][kFrontTileR + 1];
  float ss = 0.f;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // V of one element from its gradient g (scaled) and stored momentum
  // index; the momentum is updated in place unless this is the redo pass
  auto step = [&](float g, int64_t idx) {
    if (OUT == kOutRedo) {
      const float mm = Mo[idx];
      return nesterov ? fmaf(beta, mm, g) : mm;
    }
    const float mm = fmaf(beta, Mo[idx], g);
    Mo[idx] = mm;
    return nesterov ? fmaf(beta, mm, g) : mm;
  };
  auto put = [&](int64_t w, float v) {   // working-layout element w
    if (OUT == kOutV) V[w] = v;
    else X[w] = __float2half_rn(v * xs);
  };
  // one tile of the working layout, tile index bt
  auto do_tile = [&](int bt) {
    const int64_t i0 = (int64_t)(bt / tiles_c) * kFrontTileR;
    const int64_t k0 = (int64_t)(bt % tiles_c) * kFrontTileC;
    if (!tr && vec) {
      // working (i, k) = stored (i, k); 4 consecutive elements per thread
      for (int r = warp; r < kFrontTileR; r += kNT / 32) {
        const int64_t i = i0 + r;
        const int64_t k = k0 + 4 * lane;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (i < m && k < n) {
          const int64_t idx = i * n + k;
          float g[4], mo[4];
          load4(G + idx, g);
          const float4 mm4 = *reinterpret_cast<const float4*>(Mo + idx);
          mo[0] = mm4.x; mo[1] = mm4.y; mo[2] = mm4.z; mo[3] = mm4.w;
          #pragma unroll
          for (int q = 0; q < 4; ++q) {
            g[q] *= gscale;
            if (OUT != kOutRedo) mo[q] = fmaf(beta, mo[q], g[q]);
            v[q] = nesterov ? fmaf(beta, mo[q], g[q]) : mo[q];
            ss = fmaf(v[q], v[q], ss);
          }
          if (OUT != kOutRedo)
            *reinterpret_cast<float4*>(Mo + idx) = make_float4(mo[0], mo[1], mo[2], mo[3]);
        }
        if (OUT == kOutV) {
          *reinterpret_cast<float4*>(V + i * n_pad + k) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
          __half2 a = __floats2half2_rn(v[0] * xs, v[1] * xs), b = __floats2half2_rn(v[2] * xs, v[3] * xs);
          uint2 u;
          u.x = *reinterpret_cast<uint32_t*>(&a);
          u.y = *reinterpret_cast<uint32_t*>(&b);
          *reinterpret_cast<uint2*>(X + i * n_pad + k) = u;
        }
      }
    } else if (!tr) {
      // working (i, k) = stored (i, k); stored slice is [m, n]
      for (int r = warp; r < kFrontTileR; r += kNT / 32) {
        const int64_t i = i0 + r;
        for (int c = lane; c < kFrontTileC; c += 32) {
          const int64_t k = k0 + c;
          float v = 0.f;
          if (i < m && k < n) {
            const int64_t idx = i * n + k;
            v = step(to_f(G[idx]) * gscale, idx);
          }
          ss = fmaf(v, v, ss);
          put(i * n_pad + k, v);
        }
      }
    } else {
      // working (i, k) = stored (k, i); stored slice is [n, m]
      for (int c = warp; c < kFrontTileC; c += kNT / 32) {
        const int64_t k = k0 + c;
        const int64_t i = i0 + lane;
        float v = 0.f;
        if (i < m && k < n) {
          const int64_t idx = k * m + i;
          v = step(to_f(G[idx]) * gscale, idx);
        }
        ss = fmaf(v, v, ss);
        tile[c][lane] = v;
      }
      __syncthreads();
      for (int r = warp; r < kFrontTileR; r += kNT / 32)
        for (int c = lane; c < kFrontTileC; c += 32) put((i0 + r) * n_pad + k0 + c, tile[c][r]);
    }
  };
  if constexpr (OUT == kOutRedo) {
    // few blocks per slice, each walking the tiles of a mispredicted slice
    const int ntiles = (int)(m_pad / kFrontTileR) * tiles_c;
    for (int bt = blockIdx.x; bt < ntiles; bt += gridDim.x) {
      do_tile(bt);
      if (tr) __syncthreads();   // the next tile reuses tile[][]
    }
    return;
  } else {
    do_tile(blockIdx.x);
  }
  const float tot = block_sum<kNT>(ss, red);
  if (threadIdx.x == 0) part[blockIdx.x] = tot;
}

// ||V|| per slice from the front's partial sums; with exps (the fp16 first
// iterate X~ = fp16(V 2^-e)) also the slice's exponent e = 8 floor(log2
// ||V|| / 8) - 7, the factors f = 2^e / (||V|| + eps) and f^2, and whether
// the front's predicted exponent missed; e is stored back as the next step's
// prediction.  2^7 <= ||V|| 2^-e < 2^15 bounds every |X~| below fp16's
// largest value, and a prediction misses only when ||V|| crosses one of the
// 2^8-wide bins.
__global__ void __launch_bounds__(kNT) finalize_kernel(char* ws, size_t slice_ws,
                                                       size_t off_part, size_t off_slot,
                                                       int nblk, float eps, int* exps,
                                                       const int* err) {
  pdl_wait();
  if (*err) return;
  char* base = ws + (size_t)blockIdx.x * slice_ws;
  const float* part = reinterpret_cast<const float*>(base + off_part);
  __shared__ float red[kNT / 32];
  float ss = 0.f;
  for (int i = threadIdx.x; i < nblk; i += kNT) ss += part[i];
  const float tot = block_sum<kNT>(ss, red);
  if (threadIdx.x != 0) return;
  ScaleSlot* slot = reinterpret_cast<ScaleSlot*>(base + off_slot);
  const float nrm = sqrtf(tot);
  slot->inv = 1.f / (nrm + eps);
  if (!exps) return;
  int e = 0;
  if (nrm > 0.f && isfinite(nrm)) {
    int ex;
    frexpf(nrm, &ex);          // nrm = q 2^ex, q in [0.5, 1): floor(log2 nrm) = ex - 1
    const int L = ex - 1;
    const int q = L >= 0 ? L / 8 : -((-L + 7) / 8);   // floor(L / 8)
    e = min(max(8 * q - 7, kExpMin), kExpMax);
  }
  const float f = ldexpf(1.f, e) / (nrm + eps);
  slot->f = f;
  slot->f2 = f * f;
  slot->redo = exps[blockIdx.x] != e ? 1 : 0;
  slot->e = e;
  exps[blockIdx.x] = e;
}

// X0 = s*V in the iterate type; with T == 0 the scaled V is O itself.
template <typename IT>
__global__ void __launch_bounds__(kNT) normalize_kernel(char* ws, size_t slice_ws,
                                                        size_t off_V, size_t off_X,
                                                        size_t off_inv, int64_t count,
                                                        int in_place, const int* err) {
  pdl_wait();
  if (*err) return;
  char* base = ws + (size_t)blockIdx.y * slice_ws;
  float* V = reinterpret_cast<float*>(base + off_V);
  IT* X = reinterpret_cast<IT*>(base + off_X);
  const float s = *reinterpret_cast<const float*>(base + off_inv);
  const int64_t stride = (int64_t)gridDim.x * kNT * 4;
  for (int64_t i = ((int64_t)blockIdx.x * kNT + threadIdx.x) * 4; i < count; i += stride) {
    float4 v = *reinterpret_cast<const float4*>(V + i);
    v.x *= s; v.y *= s; v.z *= s; v.w *= s;
    if (in_place) {
      *reinterpret_cast<float4*>(V + i) = v;
    } else if constexpr (sizeof(IT) == 2) {
      uint2 u;
      __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
      u.x = *reinterpret_cast<uint32_t*>(&a);
      u.y = *reinterpret_cast<uint32_t*>(&b);
      *reinterpret_cast<uint2*>(X + i) = u;
    } else {
      *reinterpret_cast<float4*>(X + i) = v;
    }
  }
}

// W' = W*(1 - lr*wd) - lr*scale*O in the stored layout; O is read from the
// working layout (transposed when tr).  Optionally O is written out too.
template <typename PT>
__global__ void __launch_bounds__(kNT) epilogue_kernel(
    const __grid_constant__ SlicePtrs ptrs, int64_t M, int64_t N, int64_t n_pad, int tr, int vec,
    float decay, float lr_scale, const int* skip, const int* err, char* ws, size_t slice_ws,
    size_t off_O) {
  pdl_wait();
  // skipped loss-scaled step, or a wait of the step gave up: parameters untouched
  if ((skip && *skip) || *err) return;
  const int s = blockIdx.y;
  const float* O = reinterpret_cast<const float*>(ws + (size_t)s * slice_ws + off_O);
  PT* W = static_cast<PT*>(ptrs.W[s]);
  float* Oout = ptrs.O[s];
  if (!tr && vec) {
    // 32 rows x 128 columns per block, 4 consecutive elements per thread
    const int tiles_c4 = (int)((N + 127) / 128);
    const int64_t r0 = (int64_t)(blockIdx.x / tiles_c4) * 32;
    const int64_t c = (int64_t)(blockIdx.x % tiles_c4) * 128 + 4 * (threadIdx.x & 31);
    for (int j = threadIdx.x >> 5; j < 32; j += kNT / 32) {
      const int64_t r = r0 + j;
      if (r < M && c < N) {
        float o[4], w[4], wn[4];
        load4(O + r * n_pad + c, o);
        load4(W + r * N + c, w);
        #pragma unroll
        for (int e = 0; e < 4; ++e) wn[e] = fmaf(w[e], decay, -lr_scale * o[e]);
        store4(W + r * N + c, wn);
        if (Oout) store4(Oout + r * N + c, o);
      }
    }
    return;
  }
  __shared__ float tile[32][33];
  const int tiles_c = (int)((N + 31) / 32);
  const int64_t r0 = (int64_t)(blockIdx.x / tiles_c) * 32;
  const int64_t c0 = (int64_t)(blockIdx.x % tiles_c) * 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (tr) {
    // stored (r, c) = working (c, r): stage working rows c0.. as a tile
    for (int j = warp; j < 32; j += kNT / 32) {
      const int64_t wr = c0 + j, wc = r0 + lane;  // working row, col
      tile[j][lane] = O[wr * n_pad + wc];         // padded: always in range
    }
    __syncthreads();
  }
  for (int j = warp; j < 32; j += kNT / 32) {
    const int64_t r = r0 + j, c = c0 + lane;
    if (r < M && c < N) {
      const float o = tr ? tile[lane][j] : O[r * n_pad + c];
      const int64_t idx = r * N + c;
      const float w = to_f(W[idx]);
      W[idx] = from_f<PT>(fmaf(w, decay, -lr_scale * o));
      if (Oout) Oout[idx] = o;
    }
  }
}

struct Offsets {
  size_t V, X0, X1, A, A2, B, part, inv;
};

Offsets dense_offsets(const Group& g, int mode) {
  auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t mp = (size_t)g.m_pad, np = (size_t)g.n_pad;
  const size_t e = mode == MUON_MODE_FP32 ? 4 : 2;
  Offsets o;
  size_t p = 0;
  o.V = p;  p += a256(4 * mp * np);
  o.X0 = p; p += a256(e * mp * np);
  o.X1 = p; p += a256(e * mp * np);
  o.A = p;  p += a256(e * mp * mp);
  o.A2 = p; p += mode == MUON_MODE_FP32 ? 0 : a256(e * mp * mp);   // c A + b I (tensor-core path)
  o.B = p;  p += a256(e * mp * mp);
  o.part = p; p += a256(4 * (mp / kFrontTileR) * (np / kFrontTileC));
  o.inv = p; p += 256;
  return o;
}

template <typename IT>
cudaError_t run_dense(const Group& g, int mode, const SlicePtrs& ptrs, int ns,
                      const StepArgs& st, char* ws, int* exps, int* err_word, cudaStream_t s,
                      bool pdl_first) {
  const Offsets off = dense_offsets(g, mode);
  const size_t sws = g.slice_ws;
  const int64_t mp = g.m_pad, np = g.n_pad;
  const int nblk = (int)((mp / kFrontTileR) * (np / kFrontTileC));
  dim3 fgrid(nblk, ns);
  // vectorised access when every row of every slice starts 16-byte aligned
  const size_t es = g.dtype == MUON_BF16 ? 2 : 4;
  int vec = (g.n % 4 == 0 && g.N % 4 == 0) ? 1 : 0;
  for (int i = 0; i < ns && vec; ++i) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(ptrs.W[i]) | reinterpret_cast<uintptr_t>(ptrs.G[i]);
    if (a % (4 * es) || reinterpret_cast<uintptr_t>(ptrs.Mom[i]) % 16) vec = 0;
    if (ptrs.O[i] && reinterpret_cast<uintptr_t>(ptrs.O[i]) % 16) vec = 0;
  }

  // fp16 iterates and T > 0: the front writes the first iterate itself
  // (X~ = fp16(V 2^-e), see the header), and a second front pass fixes the
  // slices whose exponent was mispredicted; otherwise V, then X0 = s V
  const bool spec = sizeof(IT) == 2 && st.T > 0;
  auto front = [&](auto kern, bool pdl, dim3 grid) {
    return launch_k(kern, grid, dim3(kNT), 0, s, pdl, ptrs, g.m, g.n, mp, np, (int)g.tr, vec,
                    st.beta, st.nesterov, st.gscale, st.skip, (const int*)err_word, ws, sws,
                    off.V, off.X0, off.part, off.inv, (const int*)exps);
  };
  const bool bf = g.dtype == MUON_BF16;
  // every launch after the step's first may overlap the previous kernel's
  // tail (programmatic dependent launch; each kernel waits before reading)
  cudaError_t le;
  {
    NvtxRange r("muon::front_kernel");
    st.mark(MUON_KC_FRONT);
    if (spec)
      le = bf ? front(front_kernel<__nv_bfloat16, kOutX>, pdl_first, fgrid)
              : front(front_kernel<float, kOutX>, pdl_first, fgrid);
    else
      le = bf ? front(front_kernel<__nv_bfloat16, kOutV>, pdl_first, fgrid)
              : front(front_kernel<float, kOutV>, pdl_first, fgrid);
  }
  if (le != cudaSuccess) return le;
  {
    NvtxRange r("muon::finalize_kernel");
    st.mark(MUON_KC_NORM);
    le = launch_k(finalize_kernel, dim3(ns), dim3(kNT), 0, s, true, ws, sws, off.part, off.inv,
                  nblk, st.eps, spec ? exps : nullptr, (const int*)err_word);
  }
  if (le != cudaSuccess) return le;
  if (spec) {
    NvtxRange r("muon::front_kernel redo");
    st.mark(MUON_KC_NORM);
    const dim3 rgrid(nblk < kRedoBlocks ? nblk : kRedoBlocks, ns);
    le = bf ? front(front_kernel<__nv_bfloat16, kOutRedo>, true, rgrid)
            : front(front_kernel<float, kOutRedo>, true, rgrid);
  } else {
    const int64_t cnt = mp * np;
    int nb = (int)((cnt / 4 + kNT - 1) / kNT);
    if (nb > 1184) nb = 1184;
    NvtxRange r("muon::normalize_kernel");
    st.mark(MUON_KC_NORM);
    le = launch_k(normalize_kernel<IT>, dim3(nb, ns), dim3(kNT), 0, s, true, ws, sws, off.V,
                  off.X0, off.inv, cnt, st.T == 0 ? 1 : 0, (const int*)err_word);
  }
  if (le != cudaSuccess) return le;
  size_t xin = off.X0, xout = off.X1;
  // without O outputs the last product applies the parameter update itself
  // (a transposed slice through a transposing shared-memory tile in the
  // epilogue, so that its stored rows are read and written in 64-byte pieces)
  bool want_o = false;
  for (int i = 0; i < ns; ++i) want_o = want_o || ptrs.O[i] != nullptr;
  const bool fuse = sizeof(IT) == 2 && st.T > 0 && !want_o;
  const float decay = 1.f - st.lr * st.wd;
  const float lrs = st.lr * g.scale;
  if constexpr (sizeof(IT) == 2) {
    // fp16 operands: the three products on the tcgen05 tensor cores.  The
    // a and b terms of the step are folded into the operands, so that no
    // product reads a third matrix, and a X + B X = (B + a I) X.  Padded rows
    // and columns of X are zero, so the identity entries past m meet only
    // zeros.  The polynomial B + a I = c A A + b A + a I is formed from one
    // matrix when that is numerically safe:
    //   Y = c A + (b/2) I  (the Gram's only output),
    //   B + a I = Y Y / c + (a - b^2 / (4c)) I;
    // the constant b^2 / (4c) is 2.8 for the default coefficients against
    // a = 3.4 (CPU emulation: the same error as the two-output form).  When
    // b^2 / (4|c|) is large against the coefficients (or c = 0) the Gram
    // writes A and A2 = c A + b I instead and the product is A A2 + a I.
    const float ab = fabsf(st.b), ac = fabsf(st.c);
    const bool yform = st.c != 0.f && st.b * st.b / (4.f * ac) <= 2.9f * (1.45f * ac + ab);
    for (int t = 0; t < st.T; ++t) {
      const bool last = t == st.T - 1;
      TcGemm g1;
      g1.batch = ns; g1.stride = sws; g1.err = err_word; g1.skip = st.skip;
      g1.wait_limit = st.wait_limit;
      // Y = c X X^T + (b/2) I, or A = X X^T and A2 = c X X^T + b I (symmetric)
      g1.M = mp; g1.N = mp; g1.K = np;
      g1.A = ws + xin; g1.B = ws + xin; g1.D = ws + off.A; g1.sym = 1;
      if (yform) {
        g1.alpha = st.c; g1.diag = 0.5f * st.b;      // Y = c X X^T + (b/2) I
      } else {
        g1.D2 = ws + off.A2; g1.alpha2 = st.c; g1.diag2 = st.b;
      }
      if (t == 0) {   // X0 = f X~: the products of X~ scale by f^2
        g1.alpha_base = ws + off.inv + offsetof(ScaleSlot, f2);
        g1.alpha_stride = sws;
      }
      cudaError_t e;
      {
        NvtxRange r("muon::tc_gemm gram");
        st.mark(MUON_KC_GEMM);
        e = tc_gemm(g1, s);
      }
      if (e != cudaSuccess) return e;
      // B' = b A + c A A + a I (symmetric), as Y Y / c + (a - b^2/(4c)) I or
      // as A A2 + a I (A and A2 commute)
      TcGemm g2;
      g2.batch = ns; g2.stride = sws; g2.err = err_word; g2.skip = st.skip;
      g2.wait_limit = st.wait_limit;
      g2.M = mp; g2.N = mp; g2.K = mp;
      if (yform) {
        // B' = Y Y / c + (a - b^2 / (4c)) I
        g2.A = ws + off.A; g2.B = ws + off.A; g2.D = ws + off.B; g2.sym = 1;
        g2.alpha = 1.f / st.c;
        g2.diag = st.a - st.b * st.b / (4.f * st.c);
      } else {
        g2.A = ws + off.A; g2.B = ws + off.A2; g2.D = ws + off.B; g2.sym = 1;
        g2.diag = st.a;
      }
      {
        NvtxRange r("muon::tc_gemm poly");
        st.mark(MUON_KC_GEMM);
        e = tc_gemm(g2, s);
      }
      if (e != cudaSuccess) return e;
      // X' = B' X, X as an N-major B operand; fp32 O on the last step, or
      // there the update W' = W (1 - lr wd) - lr s O into the parameters
      TcGemm g3;
      g3.batch = ns; g3.stride = sws; g3.err = err_word; g3.skip = st.skip;
      g3.wait_limit = st.wait_limit;
      g3.M = mp; g3.N = np; g3.K = mp;
      g3.A = ws + off.B; g3.B = ws + xin; g3.b_mn = 1;
      g3.D = ws + (last ? off.V : xout); g3.d_f32 = last ? 1 : 0;
      if (t == 0) {   // X' = B' X0 = f (B' X~)
        g3.alpha_base = ws + off.inv + offsetof(ScaleSlot, f);
        g3.alpha_stride = sws;
      }
      if (last && fuse) {
        g3.W = ptrs.W;
        g3.w_f32 = g.dtype == MUON_F32 ? 1 : 0;
        g3.wm = g.m; g3.wn = g.n; g3.wtr = g.tr;
        g3.decay = decay; g3.lrs = lrs;
      }
      {
        NvtxRange r("muon::tc_gemm update");
        st.mark(MUON_KC_GEMM);
        e = tc_gemm(g3, s);
      }
      if (e != cudaSuccess) return e;
      const size_t tmp = xin; xin = xout; xout = tmp;
    }
  } else
  for (int t = 0; t < st.T; ++t) {
    const bool last = t == st.T - 1;
    GemmBatch gb;
    gb.batch = ns;
    gb.stride_bytes = sws;
    // A = X X^T                         [m_pad, m_pad], K = n_pad
    gb.M = mp; gb.N = mp; gb.K = np;
    gb.A = ws + xin; gb.B = ws + xin; gb.C = nullptr; gb.D = ws + off.A;
    gb.alpha = 1.f; gb.beta = 0.f;
    st.mark(MUON_KC_GEMM);
    cudaError_t e = gemm_nt<IT, IT>(gb, s);
    if (e != cudaSuccess) return e;
    // B = c*(A A) + b*A                 A symmetric: A A = A A^T
    gb.M = mp; gb.N = mp; gb.K = mp;
    gb.A = ws + off.A; gb.B = ws + off.A; gb.C = ws + off.A; gb.D = ws + off.B;
    gb.alpha = st.c; gb.beta = st.b;
    st.mark(MUON_KC_GEMM);
    e = gemm_nt<IT, IT>(gb, s);
    if (e != cudaSuccess) return e;
    // X' = B X + a*X                    [m_pad, n_pad], K = m_pad, X is N-major
    gb.M = mp; gb.N = np; gb.K = mp;
    gb.A = ws + off.B; gb.B = ws + xin; gb.C = ws + xin;
    gb.alpha = 1.f; gb.beta = st.a;
    st.mark(MUON_KC_GEMM);
    if (last) {
      gb.D = ws + off.V;
      e = gemm_nn<IT, float>(gb, s);
    } else {
      gb.D = ws + xout;
      e = gemm_nn<IT, IT>(gb, s);
    }
    if (e != cudaSuccess) return e;
    const size_t tmp = xin; xin = xout; xout = tmp;
  }
  const int tiles = (!g.tr && vec) ? (int)(((g.M + 31) / 32) * ((g.N + 127) / 128))
                                   : (int)(((g.M + 31) / 32) * ((g.N + 31) / 32));
  if (fuse) return cudaSuccess;   // the last product updated the parameters
  NvtxRange r("muon::epilogue_kernel");
  st.mark(MUON_KC_UPDATE);
  if (g.dtype == MUON_BF16)
    return launch_k(epilogue_kernel<__nv_bfloat16>, dim3(tiles, ns), dim3(kNT), 0, s, true, ptrs,
                    g.M, g.N, np, (int)g.tr, vec, decay, lrs, st.skip, (const int*)err_word, ws,
                    sws, off.V);
  return launch_k(epilogue_kernel<float>, dim3(tiles, ns), dim3(kNT), 0, s, true, ptrs, g.M, g.N,
                  np, (int)g.tr, vec, decay, lrs, st.skip, (const int*)err_word, ws, sws, off.V);
}

}  // namespace

// front, finalize, then the redo pass (fp16 iterates, T > 0) or normalize,
// 3 products per NS step, epilogue; in the tensor-core mode the last
// product applies the update (no epilogue launch)
int dense_launches(int ns_steps, int mode, int tr) {
  (void)tr;
  return (mode == MUON_MODE_TC16 && ns_steps > 0 ? 3 : 4) + 3 * ns_steps;
}

namespace {
// *found = 1 when any value of the chunk's gradients is inf or NaN
template <typename PT>
__global__ void __launch_bounds__(kNT) check_finite_kernel(const __grid_constant__ SlicePtrs ptrs,
                                                           int64_t count, int vec, int* found) {
  const PT* G = static_cast<const PT*>(ptrs.G[blockIdx.y]);
  int bad = 0;
  const int64_t stride = (int64_t)gridDim.x * kNT;
  if (vec) {
    for (int64_t i = ((int64_t)blockIdx.x * kNT + threadIdx.x) * 4; i < count; i += stride * 4) {
      float v[4];
      if (i + 3 < count) {
        load4(G + i, v);
      } else {
        for (int e = 0; e < 4; ++e) v[e] = i + e < count ? to_f(G[i + e]) : 0.f;
      }
      #pragma unroll
      for (int e = 0; e < 4; ++e) bad |= !isfinite(v[e]);
    }
  } else {
    for (int64_t i = (int64_t)blockIdx.x * kNT + threadIdx.x; i < count; i += stride)
      bad |= !isfinite(to_f(G[i]));
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) *found = 1;
}
}  // namespace

cudaError_t launch_check_finite(const Group& g, const SlicePtrs& ptrs, int nslices, int* found,
                                cudaStream_t s) {
  const int64_t count = g.M * g.N;
  const size_t es = g.dtype == MUON_BF16 ? 2 : 4;
  int vec = 1;
  for (int i = 0; i < nslices && vec; ++i)
    if (reinterpret_cast<uintptr_t>(ptrs.G[i]) % (4 * es)) vec = 0;
  int64_t per = (count + kNT * 16 - 1) / (kNT * 16);
  if (per > 64) per = 64;
  if (per < 1) per = 1;
  dim3 grid((unsigned)per, (unsigned)nslices);
  if (g.dtype == MUON_BF16)
    check_finite_kernel<__nv_bfloat16><<<grid, kNT, 0, s>>>(ptrs, count, vec, found);
  else
    check_finite_kernel<float><<<grid, kNT, 0, s>>>(ptrs, count, vec, found);
  return cudaGetLastError();
}

cudaError_t launch_dense_group_chunk(const Group& g, int mode, const SlicePtrs& ptrs,
                                     int nslices, const StepArgs& st, char* ws, int* exps,
                                     int* err_word, cudaStream_t s, bool pdl_first) {
  if (mode == MUON_MODE_FP32)
    return run_dense<float>(g, mode, ptrs, nslices, st, ws, exps, err_word, s, pdl_first);
  return run_dense<__half>(g, mode, ptrs, nslices, st, ws, exps, err_word, s, pdl_first);
}

}  // namespace muon
