// Host planner and small C-ABI helpers of libmuon.
//
// Grouping follows the HyperParallel FSDP Muon RFC (mindspore hyper-parallel
// issue "HyperParallel FSDP Muon优化器性能优化 RFC"), section 3: parameters
// whose trailing dims agree are regrouped on the host into one batch so the
// device sees one batched launch sequence per shape instead of one per
// matrix; section 2: an [E, M, N] tensor contributes E independent slices.
// The plan is built once, on the host, with no device call.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <queue>
#include <utility>

#include "internal.h"

namespace muon {

int fault_switch() {
  const char* f = std::getenv("MUON_FAULT");
  if (!f || !*f) return kFaultNone;
  if (!std::strcmp(f, "alloc")) return kFaultAlloc;
  if (!std::strcmp(f, "launch")) return kFaultLaunch;
  if (!std::strcmp(f, "timeout")) return kFaultTimeout;
  return kFaultNone;
}

static bool log_enabled() {
  const char* v = std::getenv("MUON_LOG");
  return v && *v && std::strcmp(v, "0") != 0;
}

// update scale of a [M, N] slice, rounded once to float
static float update_scale(int64_t M, int64_t N, int mode) {
  if (mode == MUON_SCALE_RMS_MATCH) return (float)(0.2 * std::sqrt((double)(M > N ? M : N)));
  const double ratio = (double)M / (double)N;
  return (float)std::sqrt(ratio > 1.0 ? ratio : 1.0);
}

static int64_t round_up(int64_t x, int64_t k) { return (x + k - 1) / k * k; }
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t dense_slice_ws(const Group& g, int mode) {
  const size_t mp = (size_t)g.m_pad, np = (size_t)g.n_pad;
  const size_t e = mode == MUON_MODE_FP32 ? 4 : 2;   // iterate element size
  size_t b = 0;
  b += align256(4 * mp * np);       // V (front output), then O (last update)
  b += 2 * align256(e * mp * np);   // X ping-pong
  b += 2 * align256(e * mp * mp);   // A and B
  if (mode != MUON_MODE_FP32) b += align256(e * mp * mp);   // c A + b I
  const size_t nblk = (size_t)(mp / kFrontTileR) * (size_t)(np / kFrontTileC);
  b += align256(4 * nblk);          // front partial sums of squares
  b += 256;                         // per-slice 1/(||V|| + eps)
  return b;
}

// The fused skinny kernel keeps a whole slice on chip: each CTA of a
// cluster holds 32-column superchunks of the slice in tensor memory (512
// columns x 128 lanes x 4 bytes).  A superchunk of mb row blocks takes
// 4*mb tensor-memory columns per lane; nw/4 warps share a lane quarter.
static bool configure_skinny(Group& g, const muon_options& o) {
  if (o.mode != MUON_MODE_TC16 || o.skinny_max_m <= 0 || g.m > o.skinny_max_m || g.m > 64)
    return false;
  int mb = (int)((g.m + 7) / 8);
  static const int kSupported[] = {1, 2, 3, 4, 6, 6, 8, 8};
  mb = kSupported[mb - 1];
  const int nw = mb <= 4 ? 16 : 8;
  const int cols_per_warp = 512 / (nw / 4);
  const int cap_w = cols_per_warp / (4 * mb);
  const int64_t nsc = (g.n + 31) / 32;
  const int64_t cap_cta = (int64_t)nw * cap_w;
  const int64_t cluster = (nsc + cap_cta - 1) / cap_cta;
  if (cluster > 8) return false;
  g.mb = mb;
  g.nw = nw;
  g.cluster = (int)cluster;
  g.sc_per_cta = (int)((nsc + cluster - 1) / cluster);
  g.sc_per_warp = (g.sc_per_cta + nw - 1) / nw;
  return true;
}

}  // namespace muon

using namespace muon;

extern "C" {

void muon_options_default(muon_options* o) {
  if (!o) return;
  o->mode = MUON_MODE_TC16;
  o->eps = 1e-7f;
  o->workspace_cap = 0;
  o->skinny_max_m = 64;
  o->scale_mode = MUON_SCALE_SQRT_RATIO;
}

muon_status muon_plan(const muon_shape* shapes, int n, const muon_options* opt,
                      muon_plan_t** out) {
  if (!out || n < 0 || (n > 0 && !shapes)) return MUON_ERR_INVALID_ARG;
  *out = nullptr;
  muon_options o;
  muon_options_default(&o);
  if (opt) o = *opt;
  if (o.mode != MUON_MODE_TC16 && o.mode != MUON_MODE_FP32) return MUON_ERR_INVALID_ARG;
  if (!(o.eps >= 0.f)) return MUON_ERR_INVALID_ARG;
  if (o.scale_mode != MUON_SCALE_SQRT_RATIO && o.scale_mode != MUON_SCALE_RMS_MATCH)
    return MUON_ERR_INVALID_ARG;
  if (fault_switch() == kFaultAlloc) return MUON_ERR_NOMEM;

  muon_plan_s* P = new (std::nothrow) muon_plan_s();
  if (!P) return MUON_ERR_NOMEM;
  try {
  P->opt = o;
  P->shapes.assign(shapes, shapes + n);
  int slice = 0;
  for (int p = 0; p < n; ++p) {
    const muon_shape& sh = shapes[p];
    int64_t E, M, N;
    if (sh.ndim == 2) { E = 1; M = sh.dims[0]; N = sh.dims[1]; }
    else if (sh.ndim == 3) { E = sh.dims[0]; M = sh.dims[1]; N = sh.dims[2]; }
    else { delete P; return MUON_ERR_UNSUPPORTED_SHAPE; }
    if (E < 1 || M < 1 || N < 1) { delete P; return MUON_ERR_UNSUPPORTED_SHAPE; }
    if (sh.dtype != MUON_BF16 && sh.dtype != MUON_F32) { delete P; return MUON_ERR_DTYPE; }
    if (E > (int64_t)1 << 30 || M > ((int64_t)1 << 31) || N > ((int64_t)1 << 31)) {
      delete P; return MUON_ERR_UNSUPPORTED_SHAPE;
    }
    int g = -1;
    for (size_t k = 0; k < P->groups.size(); ++k) {
      const Group& G = P->groups[k];
      if (G.M == M && G.N == N && G.dtype == sh.dtype) { g = (int)k; break; }
    }
    if (g < 0) {
      Group G;
      G.M = M; G.N = N; G.dtype = sh.dtype;
      G.tr = M > N ? 1 : 0;
      G.m = G.tr ? N : M;
      G.n = G.tr ? M : N;
      G.scale = update_scale(M, N, o.scale_mode);
      P->groups.push_back(G);
      g = (int)P->groups.size() - 1;
    }
    P->param_first_slice.push_back(slice);
    for (int64_t e = 0; e < E; ++e, ++slice) {
      Group& G = P->groups[g];
      P->slice_group.push_back(g);
      P->slice_index.push_back(G.count());
      G.slice_param.push_back(p);
      G.slice_e.push_back(e);
    }
  }
  // dense groups: one exponent slot per slice, kept across calls in a
  // region after the body (the scale of each slice's first iterate)
  size_t nexp = 0;
  for (Group& G : P->groups) {
    if (configure_skinny(G, o)) {
      G.kernel = MUON_KERNEL_SKINNY;
      continue;
    }
    G.kernel = MUON_KERNEL_DENSE;
    G.exp_base = (int)nexp;
    nexp += (size_t)G.count();
  }
  const size_t exp_bytes = (4 * nexp + 255) / 256 * 256;
  size_t ws = 0;
  for (Group& G : P->groups) {
    if (G.kernel != MUON_KERNEL_DENSE) continue;
    G.m_pad = round_up(G.m, kDensePad);
    G.n_pad = round_up(G.n, kDensePad);
    G.slice_ws = dense_slice_ws(G, o.mode);
    int chunk = G.count();
    if (chunk > kMaxSlicesPerLaunch) chunk = kMaxSlicesPerLaunch;
    if (o.workspace_cap > kHeaderBytes + exp_bytes) {
      size_t fit = (o.workspace_cap - kHeaderBytes - exp_bytes) / G.slice_ws;
      if ((size_t)chunk > fit) chunk = fit < 1 ? 1 : (int)fit;
    } else if (o.workspace_cap > 0) {
      chunk = 1;
    }
    G.chunk = chunk;
    size_t need = (size_t)chunk * G.slice_ws;
    if (need > ws) ws = need;
  }
  P->exp_off = kHeaderBytes + ws;
  P->ws_bytes = kHeaderBytes + ws + exp_bytes;
  } catch (const std::bad_alloc&) {
    delete P;
    return MUON_ERR_NOMEM;
  }
  if (log_enabled()) {
    std::fprintf(stderr, "muon_plan: %d parameters, %d slices, %d groups, workspace %zu bytes\n",
                 n, (int)P->slice_group.size(), (int)P->groups.size(), P->ws_bytes);
    for (size_t k = 0; k < P->groups.size(); ++k) {
      const Group& G = P->groups[k];
      if (G.kernel == MUON_KERNEL_SKINNY)
        std::fprintf(stderr,
                     "muon_plan: group %zu [%lld,%lld] %s slices=%d m=%lld n=%lld tr=%d scale=%.9g "
                     "kernel=skinny cluster=%d\n",
                     k, (long long)G.M, (long long)G.N, G.dtype == MUON_BF16 ? "bf16" : "f32",
                     G.count(), (long long)G.m, (long long)G.n, G.tr, (double)G.scale, G.cluster);
      else
        std::fprintf(stderr,
                     "muon_plan: group %zu [%lld,%lld] %s slices=%d m=%lld n=%lld tr=%d scale=%.9g "
                     "kernel=dense chunk=%d slice_workspace=%zu\n",
                     k, (long long)G.M, (long long)G.N, G.dtype == MUON_BF16 ? "bf16" : "f32",
                     G.count(), (long long)G.m, (long long)G.n, G.tr, (double)G.scale, G.chunk,
                     G.slice_ws);
    }
  }
  *out = P;
  return MUON_OK;
}

muon_status muon_plan_workspace_bytes(const muon_plan_t* P, size_t* out) {
  if (!P || !out) return MUON_ERR_INVALID_ARG;
  *out = P->ws_bytes;
  return MUON_OK;
}

muon_status muon_plan_num_groups(const muon_plan_t* P, int* out) {
  if (!P || !out) return MUON_ERR_INVALID_ARG;
  *out = (int)P->groups.size();
  return MUON_OK;
}

muon_status muon_plan_num_slices(const muon_plan_t* P, int* out) {
  if (!P || !out) return MUON_ERR_INVALID_ARG;
  *out = (int)P->slice_group.size();
  return MUON_OK;
}

muon_status muon_plan_group(const muon_plan_t* P, int g, muon_group_info* out) {
  if (!P || !out || g < 0 || g >= (int)P->groups.size()) return MUON_ERR_INVALID_ARG;
  const Group& G = P->groups[g];
  out->M = G.M; out->N = G.N; out->m = G.m; out->n = G.n;
  out->dtype = G.dtype; out->count = G.count(); out->tr = G.tr;
  out->scale = G.scale; out->kernel = G.kernel;
  out->cluster = G.kernel == MUON_KERNEL_SKINNY ? G.cluster : 0;
  out->chunk = G.kernel == MUON_KERNEL_DENSE ? G.chunk : 0;
  return MUON_OK;
}

muon_status muon_plan_slice(const muon_plan_t* P, int param, int slice, int* group,
                            int* index) {
  if (!P || !group || !index || param < 0 || param >= (int)P->shapes.size())
    return MUON_ERR_INVALID_ARG;
  const muon_shape& sh = P->shapes[param];
  const int64_t E = sh.ndim == 3 ? sh.dims[0] : 1;
  if (slice < 0 || slice >= E) return MUON_ERR_INVALID_ARG;
  const int s = P->param_first_slice[param] + slice;
  *group = P->slice_group[s];
  *index = P->slice_index[s];
  return MUON_OK;
}

muon_status muon_plan_launches(const muon_plan_t* P, int ns_steps, int* out) {
  if (!P || !out || ns_steps < 0) return MUON_ERR_INVALID_ARG;
  int n = 0;
  for (const Group& G : P->groups) {
    const int c = G.count();
    if (G.kernel == MUON_KERNEL_SKINNY) {
      n += (c + kMaxSlicesPerLaunch - 1) / kMaxSlicesPerLaunch;
    } else {
      n += ((c + G.chunk - 1) / G.chunk) * dense_launches(ns_steps, P->opt.mode, G.tr);
    }
  }
  *out = n;
  return MUON_OK;
}

muon_status muon_plan_partition(const muon_plan_t* P, int world, int ns_steps,
                                double flops_per_s, double bytes_per_s, int* owner,
                                double* rank_load) {
  if (!P || !owner || world < 1 || ns_steps < 0) return MUON_ERR_INVALID_ARG;
  if (!std::isfinite(flops_per_s) || !(flops_per_s > 0.0) || !std::isfinite(bytes_per_s) ||
      !(bytes_per_s > 0.0))
    return MUON_ERR_INVALID_ARG;
  // per-group load: counts in 128-bit integers, one rounding to double each
  std::vector<double> group_load(P->groups.size());
  for (size_t k = 0; k < P->groups.size(); ++k) {
    const Group& G = P->groups[k];
    const unsigned __int128 m = (unsigned __int128)G.m, n = (unsigned __int128)G.n;
    const unsigned __int128 flops = (unsigned __int128)ns_steps * (4 * m * m * n + 2 * m * m * m);
    const unsigned __int128 bytes = m * n * (unsigned __int128)(G.dtype == MUON_BF16 ? 14 : 20);
    const double tf = (double)flops / flops_per_s;
    const double tb = (double)bytes / bytes_per_s;
    group_load[k] = tf > tb ? tf : tb;
  }
  const int ns = (int)P->slice_group.size();
  std::vector<int> order(ns);
  for (int s = 0; s < ns; ++s) order[s] = s;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    return group_load[P->slice_group[a]] > group_load[P->slice_group[b]];
  });
  // least loaded rank first, the lower rank among equals
  using Entry = std::pair<double, int>;
  std::priority_queue<Entry, std::vector<Entry>, std::greater<Entry>> heap;
  for (int r = 0; r < world; ++r) heap.push({0.0, r});
  for (int s : order) {
    Entry e = heap.top();
    heap.pop();
    owner[s] = e.second;
    e.first += group_load[P->slice_group[s]];
    heap.push(e);
  }
  if (rank_load) {
    while (!heap.empty()) {
      rank_load[heap.top().second] = heap.top().first;
      heap.pop();
    }
  }
  return MUON_OK;
}

void muon_plan_destroy(muon_plan_t* P) { delete P; }

const char* muon_status_string(muon_status s) {
  switch (s) {
    case MUON_OK: return "ok";
    case MUON_ERR_INVALID_ARG: return "invalid argument";
    case MUON_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (ndim must be 2 or 3, dims >= 1)";
    case MUON_ERR_DTYPE: return "unsupported dtype (bf16 or fp32)";
    case MUON_ERR_ALIGNMENT: return "workspace must be 256-byte aligned";
    case MUON_ERR_CUDA: return "CUDA runtime error";
    case MUON_ERR_DEVICE_TIMEOUT: return "device wait ran out of its budget";
    case MUON_ERR_WORKSPACE: return "workspace too small for the plan";
    case MUON_ERR_NOMEM: return "host memory allocation failed";
  }
  return "unknown status";
}

}  // extern "C"
