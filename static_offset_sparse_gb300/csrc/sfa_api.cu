// C ABI device entry points of libsfa: argument checks, the per-call key plan,
// kernel launches and the device status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "sfa_internal.h"

namespace sfa {

// ---- TMA tensor maps (driver entry point, no libcuda link) -----------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int make_rows_map(CUtensorMap* m, const void* base, int64_t planes, int T, int box_rows, int box_h,
                  bool swizzle) {
  auto fn = encode_fn();
  if (!fn) return SFA_ERR_CUDA;
  const cuuint64_t dims[3] = {64, (cuuint64_t)T, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {128, (cuuint64_t)T * 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_h};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? SFA_OK
             : SFA_ERR_CUDA;
}

int make_band_map(CUtensorMap* m, const void* base, int64_t planes, int T, int delta, int box_rows,
                  int box_planes) {
  auto fn = encode_fn();
  if (!fn || delta <= 0 || T % delta) return SFA_ERR_CUDA;
  const cuuint64_t dims[4] = {64, (cuuint64_t)delta, (cuuint64_t)(T / delta), (cuuint64_t)planes};
  const cuuint64_t strides[3] = {128, (cuuint64_t)delta * 128, (cuuint64_t)T * 128};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, (cuuint32_t)box_planes};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? SFA_OK
             : SFA_ERR_CUDA;
}

int make_coef_map(CUtensorMap* m, const void* base, int64_t planes, int T, int NS, int words,
                  int box_slots, int box_q) {
  auto fn = encode_fn();
  if (!fn) return SFA_ERR_CUDA;
  const cuuint64_t rb = (cuuint64_t)words * 4;  // record bytes
  const cuuint64_t dims[4] = {(cuuint64_t)words, (cuuint64_t)NS, (cuuint64_t)T, (cuuint64_t)planes};
  const cuuint64_t strides[3] = {rb, (cuuint64_t)NS * rb, (cuuint64_t)T * NS * rb};
  const cuuint32_t box[4] = {(cuuint32_t)words, (cuuint32_t)box_slots, (cuuint32_t)box_q, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? SFA_OK
             : SFA_ERR_CUDA;
}

int launch_rope_table(int T, double theta, float* table, void* stream);

// Device status word: kernels record SFA_ERR_* codes here (bounded waits,
// index checks); sfa_get_device_status reads and clears it.
static __device__ int g_status;

// The CUDA context current on the calling thread (driver entry point, no
// libcuda link); nullptr if none is current or it cannot be read.
CUcontext current_context() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  });
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of g_status, cached per device together with the context it
// was looked up in (a new context, e.g. after cudaDeviceReset, looks it up
// again).
static int status_ptr(int** out) {
  static std::mutex mu;
  static int* cache[64] = {nullptr};
  static CUcontext owner[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SFA_ERR_CUDA;
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lock(mu);
  if (!ctx || !cache[dev] || owner[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return SFA_ERR_CUDA;
    cache[dev] = static_cast<int*>(p);
    owner[dev] = current_context();
  }
  *out = cache[dev];
  return SFA_OK;
}

// ---- launch timing --------------------------------------------------------
struct TimingRec {
  int kind;
  cudaEvent_t a, b;
};
static std::mutex g_tmu;
static std::vector<TimingRec> g_trec;
static bool g_timing = false;

int timing_start(int kind, void* stream) {
  std::lock_guard<std::mutex> lock(g_tmu);
  if (!g_timing) return -1;
  TimingRec r{kind, nullptr, nullptr};
  if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return -1;
  cudaEventRecord(r.a, (cudaStream_t)stream);
  g_trec.push_back(r);
  return (int)g_trec.size() - 1;
}

void timing_stop(int id, void* stream) {
  if (id < 0) return;
  std::lock_guard<std::mutex> lock(g_tmu);
  if (id < (int)g_trec.size()) cudaEventRecord(g_trec[id].b, (cudaStream_t)stream);
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Test injection (sfa_debug_inject): the bounded-wait limit and the group
// whose loads CTA (0, 0) of a rung tensor-core kernel never issues.
static std::mutex g_dbg_mu;
static long long g_dbg_wait = 0;  // 0: kDefaultWaitCycles
static int g_dbg_skip = -1;
// sfa_set_option values
static int g_opt_band_tc05 = 0;

static int fill_args(const sfa_desc* d, AttnArgs* a) {
  *a = AttnArgs{};
  a->B = d->B;
  a->T = d->T;
  a->Hq = d->Hq;
  a->Hkv = d->Hkv;
  a->lgG = __builtin_ctz((unsigned)(d->Hq / d->Hkv));
  a->rope = d->rope;
  a->alpha = d->alpha;
  {
    std::lock_guard<std::mutex> lock(g_dbg_mu);
    a->wait_cycles = g_dbg_wait > 0 ? g_dbg_wait : kDefaultWaitCycles;
    a->debug_skip = g_dbg_skip;
    a->band_tc05 = g_opt_band_tc05;
  }
  if (d->rope && !aligned16(d->rope)) return SFA_ERR_INVALID_ARG;
  if (d->k_rot && !aligned16(d->k_rot)) return SFA_ERR_INVALID_ARG;
  return status_ptr(&a->status);
}

// The rung kernels serve causal key sets; a signed (bidirectional) integer
// set, whose first rung distance is negative, runs the band kernels when it
// has a band plan and the SIMT kernels otherwise.
static bool tc_path(const sfa_desc* d, const Plan& p) {
  return use_tc(d) && (p.n == 0 || p.c[0] >= 0);
}

static size_t forward_workspace_bytes(const sfa_desc* d, const Plan& p, const BandPlan& bp) {
  return bp.delta > 0 || tc_path(d, p) ? kr_bytes(d) : 0;
}

// The plans of a call: an integer bf16 set with a band plan runs the band
// kernels (bp.delta > 0; p is then unused), anything else the rung plan p.
static int plan_call(const sfa_desc* d, int interp, Plan* p, BandPlan* bp) {
  bp->delta = 0;
  bp->nruns = 0;
  if (!interp) {
    int rc = build_band_plan(d, bp);
    if (rc != SFA_OK) return rc;
    if (bp->delta > 0) {
      p->W = -1;
      p->n = 0;
      p->interp = 0;
      return SFA_OK;
    }
  }
  const int rc = interp ? build_interp_plan(d, p) : build_int_plan(d, p);
  if (rc != SFA_OK) return rc;
  // the rung kernels give each group of four query heads a grid row: B Hq / 4
  // rows (B Hkv for G <= 4, which the shape check bounds; more for G = 8, 16)
  if (tc_path(d, *p) && (int64_t)d->B * (d->Hq / 4) > 65535) return SFA_ERR_UNSUPPORTED;
  return SFA_OK;
}

// Rotated keys for the tensor-core kernels: the caller's k_rot, the raw keys
// without RoPE, else K' written into scratch by the prep kernel.
static int rotated_keys(const sfa_desc* d, const void* k, void* scratch, void* stream,
                        const void** kr) {
  *kr = k;
  if (!d->rope) return SFA_OK;
  if (d->k_rot) {
    *kr = d->k_rot;
    return SFA_OK;
  }
  LaunchTimer tm(SFA_KERNEL_PREP, stream);
  int rc = launch_rope_prep(k, d->rope, scratch, (int64_t)d->B * d->Hkv * d->T, d->T, stream);
  *kr = scratch;
  return rc;
}

static int forward_common(const sfa_desc* d, int interp, const void* q, const void* k,
                          const void* v, void* o, float* lse, void* ws, size_t ws_bytes,
                          void* stream) {
  int rc = validate_shape(d);
  if (rc != SFA_OK) return rc;
  if (!q || !k || !v || !o || !lse) return SFA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return SFA_ERR_INVALID_ARG;
  Plan p;
  BandPlan bp;
  if ((rc = plan_call(d, interp, &p, &bp)) != SFA_OK) return rc;
  const size_t need = forward_workspace_bytes(d, p, bp);
  if (need && (!ws || !aligned16(ws))) return SFA_ERR_INVALID_ARG;
  if (ws_bytes < need) return SFA_ERR_CAPACITY;
  AttnArgs a;
  if ((rc = fill_args(d, &a)) != SFA_OK) return rc;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out_o = o;
  a.out_lse = lse;
  if (bp.delta == 0 && !tc_path(d, p)) return launch_forward(a, p, d->dtype, stream);
  const void* kr = nullptr;
  if ((rc = rotated_keys(d, k, ws, stream, &kr)) != SFA_OK) return rc;
  return bp.delta > 0 ? launch_band_forward(a, bp, kr, stream) : launch_forward_tc(a, p, kr, stream);
}

static size_t backward_bytes(const sfa_desc* d, const Plan& p, const BandPlan& bp) {
  size_t a, b, c, e;
  if (bp.delta > 0) return band_backward_workspace_bytes(d, &a, &b, &c);
  return tc_path(d, p) ? backward_tc_workspace_bytes(d, p, &a, &b, &c, &e) : backward_workspace_bytes(d, p);
}

static int backward_common(const sfa_desc* d, int interp, const void* q, const void* k,
                           const void* v, const void* o, const float* lse, const void* dO,
                           void* dq, void* dk, void* dv, double* dadt, void* ws,
                           size_t ws_bytes, void* stream) {
  int rc = validate_shape(d);
  if (rc != SFA_OK) return rc;
  if (d->Hq / d->Hkv > 16) return SFA_ERR_UNSUPPORTED;  // key-side smem budget
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !ws) return SFA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, o, dO, dq, dk, dv, ws};
  for (const void* x : ptrs)
    if (!aligned16(x)) return SFA_ERR_INVALID_ARG;
  Plan p;
  BandPlan bp;
  if ((rc = plan_call(d, interp, &p, &bp)) != SFA_OK) return rc;
  if (ws_bytes < backward_bytes(d, p, bp)) return SFA_ERR_CAPACITY;
  AttnArgs a;
  if ((rc = fill_args(d, &a)) != SFA_OK) return rc;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.dO = dO;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dalpha_out = interp ? dadt : nullptr;
  a.dalpha_part = static_cast<double*>(ws);
  char* w = static_cast<char*>(ws);
  if (bp.delta > 0) {
    size_t okr, oqt, ost;
    band_backward_workspace_bytes(d, &okr, &oqt, &ost);
    const void* kr = nullptr;
    if ((rc = rotated_keys(d, k, w + okr, stream, &kr)) != SFA_OK) return rc;
    return launch_band_backward(a, bp, kr, w + oqt, w + ost, stream);
  }
  if (tc_path(d, p)) {
    size_t okr, oqt, oco, ocr;
    backward_tc_workspace_bytes(d, p, &okr, &oqt, &oco, &ocr);
    a.dcorr = ocr ? reinterpret_cast<float*>(w + ocr) : nullptr;
    const void* kr = nullptr;
    if ((rc = rotated_keys(d, k, w + okr, stream, &kr)) != SFA_OK) return rc;
    return launch_backward_tc(a, p, kr, w + oqt, w + oco, stream);
  }
  const int TK = 128 >> a.lgG;
  const size_t nparts = (size_t)((d->T + TK - 1) / TK) * d->B * d->Hkv;
  a.delta = reinterpret_cast<float*>(w + align256(nparts * sizeof(double)));
  return launch_backward(a, p, d->dtype, stream);
}

}  // namespace sfa

using namespace sfa;

extern "C" {

int sfa_rope_table_bytes(int32_t T, size_t* bytes) {
  if (T <= 0 || !bytes) return SFA_ERR_INVALID_ARG;
  *bytes = (size_t)T * 32 * 2 * sizeof(float);
  return SFA_OK;
}

int sfa_rope_table(int32_t T, double theta, float* table, void* stream) {
  if (T <= 0 || T > (1 << 24) || !(theta > 0.0) || !table || !aligned16(table))
    return SFA_ERR_INVALID_ARG;
  return launch_rope_table(T, theta, table, stream);
}

int sfa_workspace_size(const sfa_desc* d, int interp, int backward, size_t* bytes) {
  if (!bytes) return SFA_ERR_INVALID_ARG;
  int rc = validate_shape(d);
  if (rc != SFA_OK) return rc;
  Plan p;
  BandPlan bp;
  if ((rc = plan_call(d, interp, &p, &bp)) != SFA_OK) return rc;
  *bytes = backward ? backward_bytes(d, p, bp) : forward_workspace_bytes(d, p, bp);
  return SFA_OK;
}

int sfa_forward(const sfa_desc* d, const void* q, const void* k, const void* v, void* o,
                float* lse, void* ws, size_t ws_bytes, void* stream) {
  return forward_common(d, 1, q, k, v, o, lse, ws, ws_bytes, stream);
}

int sfa_forward_int(const sfa_desc* d, const void* q, const void* k, const void* v, void* o,
                    float* lse, void* ws, size_t ws_bytes, void* stream) {
  return forward_common(d, 0, q, k, v, o, lse, ws, ws_bytes, stream);
}

int sfa_backward(const sfa_desc* d, const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dO, void* dq, void* dk, void* dv,
                 double* dalpha_dtheta, void* ws, size_t ws_bytes, void* stream) {
  return backward_common(d, 1, q, k, v, o, lse, dO, dq, dk, dv, dalpha_dtheta, ws, ws_bytes,
                         stream);
}

int sfa_backward_int(const sfa_desc* d, const void* q, const void* k, const void* v,
                     const void* o, const float* lse, const void* dO, void* dq, void* dk,
                     void* dv, void* ws, size_t ws_bytes, void* stream) {
  return backward_common(d, 0, q, k, v, o, lse, dO, dq, dk, dv, nullptr, ws, ws_bytes, stream);
}

int sfa_rope_keys(const sfa_desc* d, const void* k, void* k_rot, void* stream) {
  int rc = validate_shape(d);
  if (rc != SFA_OK) return rc;
  if (d->dtype != SFA_BF16) return SFA_ERR_UNSUPPORTED;
  if (!k || !k_rot || !d->rope || !aligned16(k) || !aligned16(k_rot) || !aligned16(d->rope))
    return SFA_ERR_INVALID_ARG;
  LaunchTimer tm(SFA_KERNEL_PREP, stream);
  return launch_rope_prep(k, d->rope, k_rot, (int64_t)d->B * d->Hkv * d->T, d->T, stream);
}

int sfa_decode_int(const sfa_desc* d, const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* pos, void* o, float* lse, void* stream) {
  int rc = validate_shape(d);
  if (rc != SFA_OK) return rc;
  if (!q || !k_cache || !v_cache || !pos || !o) return SFA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      ((uintptr_t)pos & 3u) || ((uintptr_t)lse & 3u))
    return SFA_ERR_INVALID_ARG;
  Plan p;
  if ((rc = build_int_plan(d, &p)) != SFA_OK) return rc;
  if (p.n > 0 && p.c[0] < 0) return SFA_ERR_INVALID_ARG;  // a cache has no future keys
  AttnArgs a;
  if ((rc = fill_args(d, &a)) != SFA_OK) return rc;
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.pos = pos;
  a.out_o = o;
  a.out_lse = lse;
  return launch_decode_int(a, p, d->dtype, stream);
}

int sfa_debug_inject(int64_t wait_cycles, int32_t skip_group) {
  if (wait_cycles < 0 || skip_group < -1) return SFA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_dbg_mu);
  g_dbg_wait = wait_cycles;
  g_dbg_skip = skip_group;
  return SFA_OK;
}

int sfa_set_option(int32_t option, int32_t value) {
  std::lock_guard<std::mutex> lock(g_dbg_mu);
  switch (option) {
    case SFA_OPT_BAND_FWD_TC05:
      if (value != 0 && value != 1) return SFA_ERR_INVALID_ARG;
      g_opt_band_tc05 = value;
      return SFA_OK;
    default:
      return SFA_ERR_INVALID_ARG;
  }
}

int sfa_timing_enable(int on) {
  std::lock_guard<std::mutex> lock(g_tmu);
  g_timing = on != 0;
  return SFA_OK;
}

int sfa_timing_read(double* ms, int64_t* launches, int n) {
  if (n < 0 || (n > 0 && (!ms || !launches))) return SFA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_tmu);
  for (int x = 0; x < n; ++x) {
    ms[x] = 0.0;
    launches[x] = 0;
  }
  int rc = SFA_OK;
  for (TimingRec& r : g_trec) {
    float t = 0.0f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      rc = SFA_ERR_CUDA;
    else if (r.kind >= 0 && r.kind < n) {
      ms[r.kind] += t;
      launches[r.kind] += 1;
    }
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  g_trec.clear();
  return rc;
}

int sfa_get_device_status(void* stream, int32_t* out) {
  if (!out) return SFA_ERR_INVALID_ARG;
  int* p = nullptr;
  int rc = status_ptr(&p);
  if (rc != SFA_OK) return rc;
  int v = 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(p, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return SFA_ERR_CUDA;
  *out = v;
  return SFA_OK;
}

}  // extern "C"
