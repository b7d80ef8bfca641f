// Internal declarations shared by the host code and the CUDA kernels of libsfa.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "sfa.h"

struct CUctx_st;  // CUcontext

namespace sfa {

constexpr int kD = 64;          // head dimension (the only one supported)
constexpr int kMaxRungs = SFA_MAX_RUNGS;

// One call's key set, built on the host and passed to every kernel by value.
// Distances 0..W (W = -1: no window) plus n rungs.  Rung r reads, for query i
// with c[r] <= i, the row (1 - w[r]) * row[i - c[r]] + w[r] * row[i - c[r] + 1]
// (w = 0: the exact row i - c[r]).  Rungs are sorted by c ascending and every
// c[r] > W.  f[r] is the base offset (for dalpha = sum_k f_k dL/dd_k).
struct Plan {
  int32_t W;
  int32_t n;
  int32_t interp;  // 1: interpolated path (w may be nonzero, dalpha computed)
  int32_t c[kMaxRungs];
  float w[kMaxRungs];
  float f[kMaxRungs];
};

// A distance set written as runs of one step delta (delta divides T): run m
// holds the distances a[m] + delta * t, 0 <= t < len[m].  With i = r + delta u
// (r = i mod delta), run m sends the queries of residue class r to the keys
// of class rho = (r - a[m]) mod delta at compressed indices
// v in [u + e - len[m] + 1, u + e], e = floor((r - a[m]) / delta): a band, so
// a tile of queries meets a contiguous tile of keys (the band kernels).
constexpr int kMaxRuns = 128;
constexpr int kMaxBandDelta = 64;
struct BandPlan {
  int32_t delta;  // 0: the set is not served by the band kernels
  int32_t nruns;
  int32_t a[kMaxRuns];
  int32_t len[kMaxRuns];
};

// Pointers and sizes of one call, passed by value to every kernel.
// Tensor element type is bf16 or fp32 (a template parameter of the kernels).
struct AttnArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;       // forward output (read by the backward)
  const void* dO;
  const float* lse;    // [B, Hq, T]
  const void* rope;    // float2 [T][32] (cos, sin) or nullptr
  void* out_o;
  float* out_lse;
  void* dq;
  void* dk;
  void* dv;
  float* delta;        // workspace [B, Hq, T]
  double* dalpha_part; // workspace, one per backward key-side CTA
  float* dcorr;        // rung backward, G > 4: delta - sum_j P dP per query row (workspace [B, Hq, T])
  double* dalpha_out;  // device [2]: dL/dalpha, dL/dtheta (or nullptr)
  double alpha;
  const int32_t* pos;  // decode: device [B] query positions
  int32_t B, T, Hq, Hkv, lgG;  // G = 1 << lgG query heads per KV head
  int* status;         // device status word
  long long wait_cycles;  // limit of every bounded mbarrier wait, in SM clock cycles
  int32_t debug_skip;     // test injection: group whose loads CTA (0, 0) never issues, or -1
  int32_t band_tc05;      // band forward on tcgen05 (1) or mma.sync (0): sfa_set_option
};

// Default limit of a bounded mbarrier wait: ~1 s at the GB300's 2.07 GHz
// maximum SM clock.
constexpr long long kDefaultWaitCycles = 2000000000LL;

// Kernel launchers (stream is a cudaStream_t).
// The rung tensor-core kernels serve bf16 I/O with G = 4m (m = 1, 2, 4: groups
// of 4 query heads, m of them per KV head); everything else runs the fp32
// SIMT kernels (or the band kernels, for integer sets with a band plan).
inline bool use_tc(const sfa_desc* d) {
  const int G = d->Hq / d->Hkv;
  return d->dtype == SFA_BF16 && (G == 4 || G == 8 || G == 16);
}
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
// Workspace for the rotated keys the tensor-core kernels read (none when the
// caller supplies them in d->k_rot, or without RoPE).
inline size_t kr_bytes(const sfa_desc* d) {
  return d->rope && !d->k_rot ? align256((size_t)d->B * d->Hkv * d->T * 64 * 2) : 0;
}
int launch_rope_prep(const void* k, const void* rope, void* kr, int64_t rows, int T, void* stream);
int launch_forward_tc(const AttnArgs& a, const Plan& p, const void* kr, void* stream);
size_t backward_tc_workspace_bytes(const sfa_desc* d, const Plan& p, size_t* off_kr, size_t* off_qt,
                                   size_t* off_coef, size_t* off_corr);
int launch_backward_tc(const AttnArgs& a, const Plan& p, const void* kr, void* qt, void* coef,
                       void* stream);
int launch_forward(const AttnArgs& a, const Plan& p, int dtype, void* stream);
int launch_decode_int(const AttnArgs& a, const Plan& p, int dtype, void* stream);
int launch_backward(const AttnArgs& a, const Plan& p, int dtype, void* stream);
size_t backward_workspace_bytes(const sfa_desc* d, const Plan& p);
// Band kernels (bf16 I/O, G in {1, 2, 4, 8}, integer sets with a band plan).
int launch_band_forward(const AttnArgs& a, const BandPlan& p, const void* kr, void* stream);
size_t band_backward_workspace_bytes(const sfa_desc* d, size_t* off_kr, size_t* off_qt,
                                     size_t* off_stat);
int launch_band_backward(const AttnArgs& a, const BandPlan& p, const void* kr, void* qt,
                         void* stat, void* stream);

// Optional launch timing (sfa_api.cu): returns a record id or -1 when off.
// The CUDA context current on the calling thread, nullptr if none (sfa_api.cu).
::CUctx_st* current_context();
int timing_start(int kind, void* stream);
void timing_stop(int id, void* stream);

// Brackets one kernel launch with timing events (no-op while timing is off).
struct LaunchTimer {
  int id;
  void* stream;
  LaunchTimer(int kind, void* s) : id(timing_start(kind, s)), stream(s) {}
  ~LaunchTimer() { timing_stop(id, stream); }
};

// Host helpers (sfa_host.cpp).
int build_interp_plan(const sfa_desc* d, Plan* p);
int build_int_plan(const sfa_desc* d, Plan* p);
// Band plan of a sorted, distinct distance set (negative distances: later
// keys) for G query heads per KV head; p->delta = 0 when the band kernels
// would not pay.
int band_plan_of(const int32_t* s, int n, int T, int G, BandPlan* p);
int build_band_plan(const sfa_desc* d, BandPlan* p);
int validate_shape(const sfa_desc* d);

}  // namespace sfa
