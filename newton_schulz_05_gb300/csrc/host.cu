// muon_step_host: one Muon step on parameters, gradients and momenta held in
// host memory.  The optimizer state of a large model can live in host memory
// (on a Grace-Blackwell node the GPU reaches it over NVLink-C2C); the step
// then streams it through a device staging buffer.
//
// The staging buffer is cut into nbuf = staging_bytes / unit_bytes buffers
// and the plan's slices into units that fit one (whole slices of one group,
// at most a dense chunk or one fused launch).  Unit k is copied in on its
// own stream, stepped on the caller's stream and copied out on a third
// stream, in buffer k % nbuf, so the copies of one unit overlap the kernels
// of its neighbours:
//
//   h2d stream   [in 0][in 1]      [in 2]      [in 3] ...
//   caller       .     [step 0]    [step 1]    [step 2] ...
//   d2h stream   .     .           [out 0]     [out 1] ...
//
// Buffer k % nbuf takes unit k + nbuf once unit k has been copied out, so
// the kernels never wait as long as a unit's copies in and out take together
// at most about nbuf - 1 times as long as its kernels.
//
// A unit's parameters, gradients and momenta go in (2 + 2 + 4 bytes per bf16
// element); its parameters and momenta come back (2 + 4).  Contiguous slices
// of one parameter move in one copy.
//
// muon_host_alloc gives the page-locked host memory for that state on
// transparent huge pages.  The state is read once per step, so every read
// is cold: on base pages (64 KiB on a Grace kernel) such reads out of some
// allocations ran at 30-140 GB/s where the link gives ~200 GB/s, on huge
// pages they keep the link's rate.
#include <sys/mman.h>
#include <unistd.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "internal.h"

using namespace muon;

namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxBufs = 16;   // staging buffers in rotation, at most
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Unit {
  int group;
  int i0, i1;                   // slices [i0, i1) of the group, in group order
  size_t bytes;                 // staging bytes (W, G and M regions)
};

// staging bytes of one slice of group g: W, G and M, each 256-byte aligned
size_t slice_stage_bytes(const Group& g) {
  const size_t es = g.dtype == MUON_BF16 ? 2 : 4;
  const size_t mn = (size_t)g.M * (size_t)g.N;
  return 2 * align_up(mn * es) + align_up(mn * 4);
}

muon_status make_units(const muon_plan_t* P, size_t part, std::vector<Unit>& units) {
  for (int gi = 0; gi < (int)P->groups.size(); ++gi) {
    const Group& g = P->groups[gi];
    const size_t per = slice_stage_bytes(g);
    if (per > part) return MUON_ERR_WORKSPACE;
    const int cap_n = g.kernel == MUON_KERNEL_SKINNY ? kMaxSlicesPerLaunch : g.chunk;
    int fit = (int)std::min<size_t>(part / per, (size_t)cap_n);
    if (fit < 1) fit = 1;
    for (int i0 = 0; i0 < g.count(); i0 += fit) {
      const int i1 = std::min(g.count(), i0 + fit);
      units.push_back(Unit{gi, i0, i1, per * (size_t)(i1 - i0)});
    }
  }
  return MUON_OK;
}

struct Copy {
  void* dst;
  const void* src;
  size_t bytes;
};

// one copy per run of slices that are contiguous on both sides
void add_run(std::vector<Copy>& v, void* dst, const void* src, size_t bytes, bool merge) {
  if (merge && !v.empty() && static_cast<char*>(v.back().dst) + v.back().bytes == dst &&
      static_cast<const char*>(v.back().src) + v.back().bytes == src) {
    v.back().bytes += bytes;
    return;
  }
  v.push_back(Copy{dst, src, bytes});
}

}  // namespace

namespace {

// the transparent-huge-page (PMD) size of the running kernel: 512 MiB on a
// 64 KiB-page Arm kernel, 2 MiB on x86-64
size_t huge_page_bytes() {
  static const size_t v = [] {
    unsigned long long x = 0;
    if (FILE* f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
      if (std::fscanf(f, "%llu", &x) != 1) x = 0;
      std::fclose(f);
    }
    return x >= 4096 && (x & (x - 1)) == 0 ? (size_t)x : (size_t)2 << 20;
  }();
  return v;
}

std::mutex g_host_mu;
std::unordered_map<void*, size_t>& host_allocs() {   // address -> mapped bytes
  static std::unordered_map<void*, size_t> m;
  return m;
}

}  // namespace

extern "C" muon_status muon_host_alloc(size_t bytes, void** out) {
  if (!out) return MUON_ERR_INVALID_ARG;
  *out = nullptr;
  if (bytes == 0) return MUON_ERR_INVALID_ARG;
  if (fault_switch() == kFaultAlloc) return MUON_ERR_NOMEM;
  const size_t hp = huge_page_bytes();
  if (bytes > SIZE_MAX - 2 * hp) return MUON_ERR_INVALID_ARG;
  const size_t len = (bytes + hp - 1) / hp * hp;
  // map one huge page more, then trim both ends to an aligned range
  const size_t span = len + hp;
  void* raw = mmap(nullptr, span, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (raw == MAP_FAILED) return MUON_ERR_NOMEM;
  const uintptr_t r = reinterpret_cast<uintptr_t>(raw);
  const uintptr_t a = (r + hp - 1) / hp * hp;
  if (a > r) munmap(raw, a - r);
  if (r + span > a + len) munmap(reinterpret_cast<void*>(a + len), r + span - (a + len));
  void* p = reinterpret_cast<void*>(a);
  // a hint only: without transparent huge pages the memory stays on base pages
  madvise(p, len, MADV_HUGEPAGE);
  // fault the pages in (huge pages where the kernel gives them) before the
  // driver pins them
  const long pg = sysconf(_SC_PAGESIZE);
  const size_t stride = pg > 0 ? (size_t)pg : 4096;
  for (size_t off = 0; off < len; off += stride) static_cast<volatile char*>(p)[off] = 0;
  if (cudaHostRegister(p, len, cudaHostRegisterPortable) != cudaSuccess) {
    cudaGetLastError();
    munmap(p, len);
    return MUON_ERR_CUDA;
  }
  {
    std::lock_guard<std::mutex> lock(g_host_mu);
    host_allocs()[p] = len;
  }
  *out = p;
  return MUON_OK;
}

extern "C" muon_status muon_host_free(void* p) {
  if (!p) return MUON_OK;
  size_t len = 0;
  {
    std::lock_guard<std::mutex> lock(g_host_mu);
    auto it = host_allocs().find(p);
    if (it == host_allocs().end()) return MUON_ERR_INVALID_ARG;
    len = it->second;
    host_allocs().erase(it);
  }
  const cudaError_t e = cudaHostUnregister(p);
  munmap(p, len);
  return e == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}

extern "C" muon_status muon_plan_host_unit_bytes(const muon_plan_t* P, size_t* out) {
  if (!P || !out) return MUON_ERR_INVALID_ARG;
  size_t m = 0;
  for (const Group& g : P->groups) m = std::max(m, slice_stage_bytes(g));
  *out = m;
  return MUON_OK;
}

extern "C" muon_status muon_step_host(const muon_plan_t* P, void* const* params,
                                      const void* const* grads, float* const* momentum,
                                      float lr, float beta, float wd, int nesterov, int ns_steps,
                                      const float* coeffs, void* workspace, size_t ws_bytes,
                                      void* staging, size_t staging_bytes, size_t unit_bytes,
                                      void* stream) {
  if (!P) return MUON_ERR_INVALID_ARG;
  const int np = (int)P->shapes.size();
  if (np > 0 && (!params || !grads || !momentum)) return MUON_ERR_INVALID_ARG;
  for (int p = 0; p < np; ++p)
    if (!params[p] || !grads[p] || !momentum[p]) return MUON_ERR_INVALID_ARG;
  if (ns_steps < 0 || ns_steps > 1000) return MUON_ERR_INVALID_ARG;
  if (!std::isfinite(lr) || !std::isfinite(beta) || !std::isfinite(wd)) return MUON_ERR_INVALID_ARG;
  if (!workspace || !staging) return MUON_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) | reinterpret_cast<uintptr_t>(staging)) & 255)
    return MUON_ERR_ALIGNMENT;
  if (ws_bytes < P->ws_bytes) return MUON_ERR_WORKSPACE;
  StepArgs st;
  st.lr = lr; st.beta = beta; st.wd = wd; st.nesterov = nesterov ? 1 : 0;
  st.T = ns_steps;
  st.a = coeffs ? coeffs[0] : 3.4445f;
  st.b = coeffs ? coeffs[1] : -4.7750f;
  st.c = coeffs ? coeffs[2] : 2.0315f;
  if (!std::isfinite(st.a) || !std::isfinite(st.b) || !std::isfinite(st.c)) return MUON_ERR_INVALID_ARG;
  st.eps = P->opt.eps;
  const size_t part = unit_bytes / kAlign * kAlign;
  if (part == 0) return MUON_ERR_INVALID_ARG;
  const int nbuf = (int)std::min<size_t>(staging_bytes / part, (size_t)kMaxBufs);
  if (nbuf < 2) return MUON_ERR_WORKSPACE;
  std::vector<Unit> units;
  muon_status ms = make_units(P, part, units);
  if (ms != MUON_OK) return ms;
  const int fault = fault_switch();
  if (fault == kFaultLaunch) return MUON_ERR_CUDA;
  if (fault == kFaultTimeout) st.wait_limit = 0;
  NvtxRange range("muon_step_host");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* err_word = reinterpret_cast<int*>(ws);
  char* body = ws + kHeaderBytes;
  char* stage[kMaxBufs];
  for (int b = 0; b < nbuf; ++b) stage[b] = static_cast<char*>(staging) + (size_t)b * part;

  // copy streams and events of this call, released when their work is done
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t entry = nullptr, in_done[kMaxBufs] = {}, step_done[kMaxBufs] = {},
              out_done[kMaxBufs] = {};
  auto release = [&]() {
    if (h2d) cudaStreamDestroy(h2d);
    if (d2h) cudaStreamDestroy(d2h);
    if (entry) cudaEventDestroy(entry);
    for (int b = 0; b < nbuf; ++b)
      for (cudaEvent_t e : {in_done[b], step_done[b], out_done[b]})
        if (e) cudaEventDestroy(e);
  };
  bool ok = cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&entry, cudaEventDisableTiming) == cudaSuccess;
  for (int b = 0; b < nbuf && ok; ++b)
    ok = cudaEventCreateWithFlags(&in_done[b], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&step_done[b], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&out_done[b], cudaEventDisableTiming) == cudaSuccess;
  // the copies start after the caller's earlier work on its stream
  ok = ok && cudaEventRecord(entry, s) == cudaSuccess &&
       cudaStreamWaitEvent(h2d, entry, 0) == cudaSuccess &&
       cudaStreamWaitEvent(d2h, entry, 0) == cudaSuccess;
  if (!ok) { release(); return MUON_ERR_CUDA; }

  std::vector<Copy> cin, cout;
  SlicePtrs ptrs;
  for (size_t k = 0; k < units.size() && ok; ++k) {
    const Unit& u = units[k];
    const Group& g = P->groups[u.group];
    const int b = (int)(k % nbuf);
    const size_t es = g.dtype == MUON_BF16 ? 2 : 4;
    const size_t mn = (size_t)g.M * (size_t)g.N;
    const int ns = u.i1 - u.i0;
    char* wreg = stage[b];
    char* greg = wreg + (size_t)ns * align_up(mn * es);
    char* mreg = greg + (size_t)ns * align_up(mn * es);
    // in-copies of W, G and M; out-copies of W' and M'
    cin.clear(); cout.clear();
    std::vector<Copy> cg, cm, ow, om;
    const bool contig = (mn * es) % kAlign == 0 && (mn * 4) % kAlign == 0;
    for (int j = 0; j < ns; ++j) {
      const int p = g.slice_param[u.i0 + j];
      const size_t e = (size_t)g.slice_e[u.i0 + j];
      char* dw = wreg + (size_t)j * align_up(mn * es);
      char* dg = greg + (size_t)j * align_up(mn * es);
      float* dm = reinterpret_cast<float*>(mreg + (size_t)j * align_up(mn * 4));
      char* hw = static_cast<char*>(params[p]) + e * mn * es;
      const char* hg = static_cast<const char*>(grads[p]) + e * mn * es;
      float* hm = momentum[p] + e * mn;
      add_run(cin, dw, hw, mn * es, contig);
      add_run(cg, dg, hg, mn * es, contig);
      add_run(cm, dm, hm, mn * 4, contig);
      add_run(ow, hw, dw, mn * es, contig);
      add_run(om, hm, dm, mn * 4, contig);
      ptrs.W[j] = dw;
      ptrs.G[j] = dg;
      ptrs.Mom[j] = dm;
      ptrs.O[j] = nullptr;
    }
    cin.insert(cin.end(), cg.begin(), cg.end());
    cin.insert(cin.end(), cm.begin(), cm.end());
    cout = ow;
    cout.insert(cout.end(), om.begin(), om.end());
    // in: after buffer b was last copied out
    ok = cudaStreamWaitEvent(h2d, out_done[b], 0) == cudaSuccess;
    for (const Copy& c : cin)
      ok = ok && cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyDefault, h2d) == cudaSuccess;
    ok = ok && cudaEventRecord(in_done[b], h2d) == cudaSuccess;
    // step the unit on the caller's stream
    ok = ok && cudaStreamWaitEvent(s, in_done[b], 0) == cudaSuccess;
    if (ok) {
      cudaError_t e;
      if (g.kernel == MUON_KERNEL_SKINNY)
        e = launch_skinny(g, ptrs, ns, st, err_word, s);
      else
        e = launch_dense_group_chunk(g, P->opt.mode, ptrs, ns, st, body,
                                     reinterpret_cast<int*>(ws + P->exp_off) + g.exp_base + u.i0,
                                     err_word, s, false);
      ok = e == cudaSuccess;
    }
    ok = ok && cudaEventRecord(step_done[b], s) == cudaSuccess;
    // out: after the unit's step
    ok = ok && cudaStreamWaitEvent(d2h, step_done[b], 0) == cudaSuccess;
    for (const Copy& c : cout)
      ok = ok && cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyDefault, d2h) == cudaSuccess;
    ok = ok && cudaEventRecord(out_done[b], d2h) == cudaSuccess;
  }
  // the caller's stream continues after every copy out
  for (int b = 0; b < nbuf && ok; ++b) ok = cudaStreamWaitEvent(s, out_done[b], 0) == cudaSuccess;
  release();
  return ok ? MUON_OK : MUON_ERR_CUDA;
}
