// Internal declarations shared by the host planner, the step driver and the
// kernel launchers of libmuon.  Not part of the public C ABI (include/muon.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "muon.h"

namespace muon {

constexpr size_t kHeaderBytes = 256;   // workspace header: device error word
constexpr int kMaxSlicesPerLaunch = 512;
constexpr int kDensePad = 128;         // dense working dims are padded to this
constexpr int kFrontTileR = 32;        // front kernel tile (working layout)
constexpr int kFrontTileC = 128;

// device error codes written into the workspace header
constexpr int kDevErrTimeout = 1;
// polls of an mbarrier before a bounded wait gives up (about a second or
// more); waits for a kernel's own copies in flight always use this budget
constexpr uint32_t kWaitLimit = 1u << 26;

// NVTX range over a scope (a step, a kernel launch): shows up in Nsight
// timelines; without a tool attached it costs a few nanoseconds
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// MUON_FAULT switch of this call: 0 none, else one of the kFault* values
enum { kFaultNone = 0, kFaultAlloc = 1, kFaultLaunch = 2, kFaultTimeout = 3 };
int fault_switch();

struct Group {
  int64_t M = 0, N = 0, m = 0, n = 0;
  int dtype = 0;
  int tr = 0;
  float scale = 1.f;
  int kernel = MUON_KERNEL_DENSE;
  std::vector<int> slice_param;  // parameter of each slice, group order
  std::vector<int64_t> slice_e;  // slice index inside that parameter
  int count() const { return (int)slice_param.size(); }
  // skinny kernel configuration
  int mb = 0;        // row blocks of 8 (padded m / 8)
  int nw = 0;        // warps per CTA
  int cluster = 0;   // CTAs per slice
  int sc_per_cta = 0, sc_per_warp = 0;  // 32-column superchunks
  // dense path
  int64_t m_pad = 0, n_pad = 0;
  int chunk = 0;           // slices per chunk
  size_t slice_ws = 0;     // workspace bytes per slice
  int exp_base = -1;       // index of the group's first slice in the exponent region
};

}  // namespace muon

struct muon_plan_s {
  std::vector<muon_shape> shapes;
  std::vector<int> param_first_slice;   // global slice id of (p, 0)
  std::vector<int> slice_group, slice_index;
  std::vector<muon::Group> groups;
  muon_options opt;
  size_t ws_bytes = 0;
  size_t exp_off = 0;   // exponent region: one int per dense slice, after the body
};

namespace muon {

// Per-slice pointers of one launch (passed by value as a kernel parameter).
struct SlicePtrs {
  void* W[kMaxSlicesPerLaunch];
  const void* G[kMaxSlicesPerLaunch];
  float* Mom[kMaxSlicesPerLaunch];
  float* O[kMaxSlicesPerLaunch];     // null entries: O not requested
};

// Events recorded before every kernel launch of a step (muon_step_timed):
// interval i, from event i to event i + 1, is the kernel of class cls[i].
struct LaunchTimer {
  cudaStream_t stream = nullptr;
  std::vector<cudaEvent_t> ev;
  std::vector<int> cls;
  cudaError_t err = cudaSuccess;
  void mark(int c) {
    cudaEvent_t e = nullptr;
    if (err == cudaSuccess) err = cudaEventCreate(&e);
    if (err == cudaSuccess) err = cudaEventRecord(e, stream);
    if (e) { ev.push_back(e); cls.push_back(c); }
  }
  ~LaunchTimer() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
};

struct StepArgs {
  float lr, beta, wd;
  int nesterov;
  int T;
  float a, b, c;
  float eps;
  float gscale = 1.f;          // gradients are multiplied by this (1/loss scale)
  const int* skip = nullptr;   // device flag: when set, the step changes nothing
  uint32_t wait_limit = kWaitLimit;   // polls of a bounded wait on the main path
  LaunchTimer* timer = nullptr;       // per-launch events (measurement only)
  void mark(int kernel_class) const {
    if (timer) timer->mark(kernel_class);
  }
};

size_t dense_slice_ws(const Group& g, int mode);

// launchers; each returns cudaSuccess or the launch error
cudaError_t launch_skinny(const Group& g, const SlicePtrs& ptrs, int nslices,
                          const StepArgs& st, int* err_word, cudaStream_t s);

// pdl_first: the chunk's first kernel may overlap the previous kernel on the
// stream (false for the first launch of a step).  exps: the exponent slots of
// the chunk's slices (device, kept across calls; any content is valid)
cudaError_t launch_dense_group_chunk(const Group& g, int mode, const SlicePtrs& ptrs,
                                     int nslices, const StepArgs& st, char* ws, int* exps,
                                     int* err_word, cudaStream_t s, bool pdl_first);

int dense_launches(int ns_steps, int mode, int tr);   // per chunk, step without O outputs

// Sets *found to 1 when any gradient value of the chunk is inf or NaN.
cudaError_t launch_check_finite(const Group& g, const SlicePtrs& ptrs, int nslices, int* found,
                                cudaStream_t s);

}  // namespace muon
