// muon_step: validates its arguments, then enqueues, group by group, the
// launches of one Muon step on the caller's stream.  No allocation, no host
// synchronisation.  Skinny groups run the fused on-chip kernel (one launch
// per <= 512 slices); dense groups run the front / GEMM / epilogue sequence
// per chunk of slices that fits the workspace.
#include <cmath>
#include <cstring>

#include "internal.h"

using namespace muon;

namespace {

muon_status step_impl(const muon_plan_t* P, void* const* params, const void* const* grads,
                      float* const* momentum, float lr, float beta, float wd, int nesterov,
                      int ns_steps, const float* coeffs, void* workspace, size_t ws_bytes,
                      void* stream, float* const* ortho, float inv_scale = 1.f,
                      int* found_inf = nullptr, LaunchTimer* timer = nullptr) {
  if (!P) return MUON_ERR_INVALID_ARG;
  NvtxRange range(found_inf ? "muon_step_amp" : ortho ? "muon_step_ortho" : "muon_step");
  const int np = (int)P->shapes.size();
  if (np > 0 && (!params || !grads || !momentum)) return MUON_ERR_INVALID_ARG;
  for (int p = 0; p < np; ++p)
    if (!params[p] || !grads[p] || !momentum[p] || (ortho && !ortho[p])) return MUON_ERR_INVALID_ARG;
  if (ns_steps < 0 || ns_steps > 1000) return MUON_ERR_INVALID_ARG;
  if (!std::isfinite(lr) || !std::isfinite(beta) || !std::isfinite(wd)) return MUON_ERR_INVALID_ARG;
  if (!workspace) return MUON_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return MUON_ERR_ALIGNMENT;
  if (ws_bytes < P->ws_bytes) return MUON_ERR_WORKSPACE;
  StepArgs st;
  st.lr = lr; st.beta = beta; st.wd = wd; st.nesterov = nesterov ? 1 : 0;
  st.T = ns_steps;
  st.a = coeffs ? coeffs[0] : 3.4445f;
  st.b = coeffs ? coeffs[1] : -4.7750f;
  st.c = coeffs ? coeffs[2] : 2.0315f;
  if (!std::isfinite(st.a) || !std::isfinite(st.b) || !std::isfinite(st.c)) return MUON_ERR_INVALID_ARG;
  st.eps = P->opt.eps;
  if (!std::isfinite(inv_scale)) return MUON_ERR_INVALID_ARG;
  st.gscale = inv_scale;
  st.skip = found_inf;
  st.timer = timer;
  const int fault = fault_switch();
  if (fault == kFaultLaunch) return MUON_ERR_CUDA;
  if (fault == kFaultTimeout) st.wait_limit = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* err_word = reinterpret_cast<int*>(ws);
  char* body = ws + kHeaderBytes;

  SlicePtrs ptrs;
  auto fill = [&](const Group& g, int c0, int ns) {
    const size_t es = g.dtype == MUON_BF16 ? 2 : 4;
    const int64_t mn = g.M * g.N;
    for (int i = 0; i < ns; ++i) {
      const int p = g.slice_param[c0 + i];
      const int64_t off = g.slice_e[c0 + i] * mn;
      ptrs.W[i] = static_cast<char*>(params[p]) + off * es;
      ptrs.G[i] = static_cast<const char*>(grads[p]) + off * es;
      ptrs.Mom[i] = momentum[p] + off;
      ptrs.O[i] = ortho ? ortho[p] + off : nullptr;
    }
  };
  if (found_inf) {
    // loss-scaled step: every gradient value is checked before any state
    // changes; the kernels below return at once when the flag is set
    if (cudaMemsetAsync(found_inf, 0, sizeof(int), s) != cudaSuccess) return MUON_ERR_CUDA;
    for (const Group& g : P->groups)
      for (int c0 = 0; c0 < g.count(); c0 += kMaxSlicesPerLaunch) {
        const int ns = g.count() - c0 < kMaxSlicesPerLaunch ? g.count() - c0 : kMaxSlicesPerLaunch;
        fill(g, c0, ns);
        st.mark(MUON_KC_CHECK);
        if (launch_check_finite(g, ptrs, ns, found_inf, s) != cudaSuccess) return MUON_ERR_CUDA;
      }
  }
  // kernels after the step's first may overlap their predecessor's tail
  bool first = found_inf == nullptr;
  for (const Group& g : P->groups) {
    const int cnt = g.count();
    const int per = g.kernel == MUON_KERNEL_SKINNY ? kMaxSlicesPerLaunch : g.chunk;
    for (int c0 = 0; c0 < cnt; c0 += per) {
      const int ns = cnt - c0 < per ? cnt - c0 : per;
      fill(g, c0, ns);
      cudaError_t e;
      if (g.kernel == MUON_KERNEL_SKINNY) {
        NvtxRange r("muon::skinny_kernel");
        st.mark(MUON_KC_SKINNY);
        e = launch_skinny(g, ptrs, ns, st, err_word, s);
      } else {
        e = launch_dense_group_chunk(g, P->opt.mode, ptrs, ns, st, body,
                                     reinterpret_cast<int*>(ws + P->exp_off) + g.exp_base + c0,
                                     err_word, s, !first);
      }
      if (e != cudaSuccess) return MUON_ERR_CUDA;
      first = false;
    }
  }
  return MUON_OK;
}

}  // namespace

extern "C" {

muon_status muon_step(const muon_plan_t* P, void* const* params, const void* const* grads,
                      float* const* momentum, float lr, float beta, float wd, int nesterov,
                      int ns_steps, const float* coeffs, void* workspace, size_t ws_bytes,
                      void* stream) {
  return step_impl(P, params, grads, momentum, lr, beta, wd, nesterov, ns_steps, coeffs,
                   workspace, ws_bytes, stream, nullptr);
}

muon_status muon_step_ortho(const muon_plan_t* P, void* const* params,
                            const void* const* grads, float* const* momentum, float lr,
                            float beta, float wd, int nesterov, int ns_steps,
                            const float* coeffs, void* workspace, size_t ws_bytes,
                            void* stream, float* const* ortho) {
  if (!ortho) return MUON_ERR_INVALID_ARG;
  return step_impl(P, params, grads, momentum, lr, beta, wd, nesterov, ns_steps, coeffs,
                   workspace, ws_bytes, stream, ortho);
}

muon_status muon_step_amp(const muon_plan_t* P, void* const* params, const void* const* grads,
                          float* const* momentum, float lr, float beta, float wd, int nesterov,
                          int ns_steps, const float* coeffs, float inv_scale, int* found_inf,
                          void* workspace, size_t ws_bytes, void* stream) {
  if (!found_inf) return MUON_ERR_INVALID_ARG;
  return step_impl(P, params, grads, momentum, lr, beta, wd, nesterov, ns_steps, coeffs,
                   workspace, ws_bytes, stream, nullptr, inv_scale, found_inf);
}

muon_status muon_step_timed(const muon_plan_t* P, void* const* params, const void* const* grads,
                            float* const* momentum, float lr, float beta, float wd, int nesterov,
                            int ns_steps, const float* coeffs, void* workspace, size_t ws_bytes,
                            void* stream, muon_kernel_times* times) {
  if (!times) return MUON_ERR_INVALID_ARG;
  LaunchTimer timer;
  timer.stream = static_cast<cudaStream_t>(stream);
  const muon_status st = step_impl(P, params, grads, momentum, lr, beta, wd, nesterov, ns_steps,
                                   coeffs, workspace, ws_bytes, stream, nullptr, 1.f, nullptr,
                                   &timer);
  if (st != MUON_OK) return st;
  timer.mark(-1);   // end of the last launch
  if (timer.err != cudaSuccess) return MUON_ERR_CUDA;
  if (cudaStreamSynchronize(timer.stream) != cudaSuccess) return MUON_ERR_CUDA;
  for (int k = 0; k < MUON_KC_COUNT; ++k) { times->ms[k] = 0.f; times->launches[k] = 0; }
  for (size_t i = 0; i + 1 < timer.ev.size(); ++i) {
    const int c = timer.cls[i];
    if (c < 0 || c >= MUON_KC_COUNT) continue;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, timer.ev[i], timer.ev[i + 1]) != cudaSuccess) return MUON_ERR_CUDA;
    times->ms[c] += ms;
    times->launches[c] += 1;
  }
  return MUON_OK;
}

muon_status muon_workspace_error(const void* workspace, void* stream, int clear, int* code) {
  if (!workspace || !code) return MUON_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int h = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MUON_ERR_CUDA;
  if (cudaMemcpy(&h, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MUON_ERR_CUDA;
  if (clear && cudaMemset(const_cast<void*>(workspace), 0, sizeof(int)) != cudaSuccess)
    return MUON_ERR_CUDA;
  *code = h == 0 ? MUON_OK : MUON_ERR_DEVICE_TIMEOUT;
  return MUON_OK;
}

}  // extern "C"
