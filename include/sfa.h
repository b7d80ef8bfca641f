/*
 * sfa.h - C ABI of libsfa: causal shared-offset sparse attention on one
 * NVIDIA GB300 (sm_103a), forward and backward.
 *
 * The operation ("Depth-Staggered Fibonacci Spacing for Sparse Attention",
 * method section): query i attends the keys at distances 0..W (a dense local
 * window, self included) and at rung distances d_k = alpha * f_k.  A rung
 * whose distance is not an integer reads the key/value row at real position
 * i - d_k by linear interpolation between rows floor(i - d_k) and
 * floor(i - d_k) + 1, which gives alpha a gradient.  RoPE rotates Q and K at
 * their own positions before the gather.  alpha = 0.5 + sigmoid(theta).
 * Integer offset lists (Fibonacci at integer alpha, power-of-2, the
 * Christoffel carry-word offsets of "Christoffel-Balanced Sparse Attention")
 * run through the same kernels as exact one-row gathers.
 *
 * Conventions shared by every entry point:
 *  - Tensors are contiguous [B, H, T, D] with D fastest; D must be 64.
 *    q, o, dO, dq: H = Hq.  k, v, dk, dv: H = Hkv.  Hq % Hkv == 0 and the
 *    group size G = Hq / Hkv is a power of two <= 32; query head h reads KV
 *    head h / G.  lse and delta are fp32 [B, Hq, T].  Sizes: 1 <= T <= 2^24,
 *    B * Hkv <= 65535, and for calls that run the rung kernels (bf16, G = 8
 *    or 16) B * Hq / 4 <= 65535; larger shapes return SFA_ERR_UNSUPPORTED.
 *  - All tensor pointers are device pointers, owned by the caller, 16-byte
 *    aligned.  Host arrays (base offsets, distance lists, outputs of the
 *    host builders) are read or written during the call and not retained.
 *  - The library never allocates device memory inside a call; scratch comes
 *    from the caller's workspace (see sfa_workspace_size).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Device entry points only enqueue work and return; they do not
 *    synchronise.  Asynchronous device-side errors are read with
 *    sfa_get_device_status.
 *  - Every function returns an sfa_status code.  On an argument error
 *    nothing is launched and no output is touched.
 *  - Gradients are of L = sum(O * dO) (no averaging).
 */
#ifndef SFA_H
#define SFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SFA_OK = 0,
  SFA_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad range */
  SFA_ERR_UNSUPPORTED = 2, /* valid but not implemented (D != 64, G not a power of two, ...) */
  SFA_ERR_CAPACITY = 3,    /* an output array or the workspace is too small */
  SFA_ERR_CUDA = 4,        /* a CUDA runtime call failed */
  SFA_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up (device status only) */
  SFA_ERR_DEVICE_BOUNDS = 6 /* a device-side index check failed (device status only) */
} sfa_status;

typedef enum { SFA_F32 = 0, SFA_BF16 = 1 } sfa_dtype;

typedef enum { SFA_SCHED_FIXED = 0, SFA_SCHED_LINEAR = 1, SFA_SCHED_COPRIME = 2 } sfa_schedule;

/* Maximum number of rungs (interpolated path) or of distances outside the
 * contiguous window prefix (integer path) in one call. */
#define SFA_MAX_RUNGS 256

/* One call's problem description. */
typedef struct {
  int32_t B, T, Hq, Hkv, D; /* D must be 64 */
  int32_t dtype;            /* sfa_dtype of q, k, v, o, dO, dq, dk, dv */
  /* interpolated path (sfa_forward / sfa_backward) */
  int32_t W;                /* window: distances 0..W, W >= 0 */
  double alpha;             /* rung scale, alpha > 0 (the method uses [0.5, 1.5]) */
  const int32_t* base;      /* host: base offsets f_k (> 0), n_base entries */
  int32_t n_base;
  /* integer path (sfa_forward_int / sfa_backward_int) */
  const int32_t* dist;      /* host: key distances, 0 and the window included; duplicates
                             * allowed; a negative distance is a future key (signed set) */
  int32_t n_dist;
  /* RoPE: device table written by sfa_rope_table for at least T positions
   * with D = 64, or NULL for no rotation. */
  const float* rope;
  /* Optional device [B, Hkv, T, 64] bf16: the rotated keys sfa_rope_keys wrote
   * for this k and this rope table, or NULL.  Calls that run the tensor-core
   * kernels (bf16 I/O: the rung kernels for G = 4, 8, 16 and the band kernels,
   * signed band sets included) then read it instead of
   * rotating K into their workspace (which shrinks accordingly), so one
   * rotation serves a layer's forward and backward.  Ignored otherwise. */
  const void* k_rot;
} sfa_desc;

/* ---- host builders (no GPU needed) ---------------------------------- */

/* First K terms of 1, 2, 3, 5, 8, ... (each the sum of the previous two),
 * the Fibonacci base of "Depth-Staggered Fibonacci Spacing for Sparse
 * Attention", method section.  1 <= K <= 40; out has K entries. */
int sfa_offsets_fib(int32_t K, int32_t* out);

/* 1, 2, 4, ..., 2^(K-1): the power-of-2 control base of the same page.
 * 1 <= K <= 31. */
int sfa_offsets_pow2(int32_t K, int32_t* out);

/* Christoffel carry word c[j] = floor((j+1)m/k) - floor(jm/k), j < k, in
 * 64-bit integer arithmetic ("Christoffel-Balanced Sparse Attention");
 * writes the offsets {j : c[j] = 1} ascending, preceded by 0 when
 * include_zero != 0.  0 < m <= k <= 2^30.  *n_out is always set to the
 * count; if it exceeds cap, nothing is written and SFA_ERR_CAPACITY is
 * returned. */
int sfa_offsets_christoffel(int32_t m, int32_t k, int32_t include_zero, int32_t* out,
                            int32_t cap, int32_t* n_out);

/* Per-layer alpha ("Depth-Staggered ...", method section): FIXED alpha = 1;
 * LINEAR alpha_l = 0.5 + l/(L-1); COPRIME: layer l takes the LINEAR value of
 * index (S*l mod L), gcd(S, L) = 1.  out has L entries.  1 <= L <= 4096. */
int sfa_alpha_schedule(int32_t L, int32_t kind, int32_t S, double* out);

/* The rung table the interpolated path uses (exposed for testing):
 * d = fl64(alpha * f) for each base entry; rungs with d <= W are dropped (they
 * lie in the window); c = ceil(d), w = c - d (fp64, then fp32).  Output is
 * sorted by c ascending; f_out holds the matching f.  *n_out always set;
 * SFA_ERR_CAPACITY if it exceeds cap. */
int sfa_rung_table(const int32_t* base, int32_t n_base, double alpha, int32_t W,
                   int32_t* c_out, float* w_out, float* f_out, int32_t cap, int32_t* n_out);

/* Sorted, de-duplicated integer distance set used by the integer path
 * (exposed for testing); |d| < 2^30.  *n_out always set; SFA_ERR_CAPACITY if
 * > cap. */
int sfa_int_distances(const int32_t* dist, int32_t n_dist, int32_t* out, int32_t cap,
                      int32_t* n_out);

/* How the integer path of a bf16 call lays out a distance set on the tensor
 * cores (exposed for testing and for callers choosing offset lists).  A set
 * that is a union of long arithmetic runs of one step delta (the
 * Christoffel offsets of "Christoffel-Balanced Sparse Attention" with
 * m | k: 0 and k/m - 1 + t k/m; a dense window: delta = 1) makes every
 * residue class of queries (mod delta) attend a contiguous band of keys of
 * one residue class per run: the band kernels run it as dense 64 x 64
 * tiles.  Distances are those of sfa_int_distances; distances with |d| >= T
 * are left out.  A negative distance (a later key of a signed set) is part of
 * a run like any other.  For each delta <= 64 dividing T the set is split into runs
 * a + delta t, 0 <= t < len (ascending a); the delta with the fewest 64-key
 * tiles per query tile of 64 / G positions, sum over runs of
 * ceil((64 / G + len - 1) / 64), is kept (smallest delta on ties).  Where the
 * rung kernels could take the set (G = 4 or 8, no negative distance) the plan
 * is used when the distance count is at least 8 times that tile count; for
 * G = 1 or 2 and for signed sets (whose alternative is the SIMT path) any
 * plan is used.
 * Writes *delta (0: no band plan; the set runs the rung kernels for G = 4, 8
 * or 16, the SIMT kernels otherwise), *n_runs, and run_start / run_len (cap
 * entries; SFA_ERR_CAPACITY if more runs).  G must be 1, 2, 4 or 8 for a
 * plan; a set without 0 has none. */
int sfa_band_plan(const int32_t* dist, int32_t n_dist, int32_t T, int32_t G, int32_t* delta,
                  int32_t* run_start, int32_t* run_len, int32_t cap, int32_t* n_runs);

/* ---- offset-schedule analysis and the shared power-law offset list ---- */

/* Distances reached through a stack of causal shared-offset layers
 * ("Christoffel-Balanced Sparse Attention": measure graph reachability
 * across layers, a single periodic mask may leave residue classes
 * unreached; "Depth-Staggered ...": coverage through the stack).  Layer l
 * (0-based) reads distances dist[layer_start[l]] .. dist[layer_start[l+1]-1],
 * each >= 0 (duplicates allowed).  After layers 1..l a distance d < T is
 * reached iff it is a sum of one distance of each of those layers; before
 * any layer only d = 0 is.  Writes hops[T]: the smallest l >= 0 after which
 * d is reached, -1 if never within the L layers; and, if covered != NULL,
 * covered[L]: the number of distances < T reached after exactly layers
 * 1..l.  layer_start has L + 1 non-decreasing entries starting at 0.
 * 1 <= L <= 4096, 1 <= T <= 2^24. */
int sfa_reach(const int32_t* dist, const int32_t* layer_start, int32_t L, int32_t T, int32_t* hops,
              int64_t* covered);

/* out[r] = number of d < T with hops[d] >= 0 and d mod M == r; 1 <= M <= T. */
int sfa_residue_classes(const int32_t* hops, int32_t T, int32_t M, int64_t* out);

/* Log2-binned histogram of a distance set (each distinct d with 0 <= d < T
 * counted once): bin 0 = {0}; bin b = [2^(b-1), 2^b) for 1 <= b < nb - 1;
 * bin nb - 1 takes every d >= 2^(nb-2).  nb >= 2; out has nb entries. */
int sfa_offset_histogram(const int32_t* dist, int32_t n, int32_t T, int32_t nb, int64_t* out);

/* Shared power-law offsets ("Critical power-law sparse attention",
 * integration point: m distances drawn from q(d) = d^-(1+sigma) /
 * sum_{v=1}^{floor(n/2)} v^-(1+sigma), d = 1..floor(n/2), deduplicated; here
 * one draw serves every query as causal keys i - d).  u holds the caller's m
 * uniforms in [0, 1).  Inverse CDF in fp64: c_d = sum_{v<=d} v^-(1+sigma)
 * in increasing v, Z = c_{floor(n/2)}; draw j is the smallest d with
 * c_d > u_j * Z.  Writes the distinct distances ascending; *n_out is always
 * set, SFA_ERR_CAPACITY (nothing written) if it exceeds cap.
 * 1 <= m, 2 <= n <= 2^26, sigma >= 0, 0 <= u_j < 1. */
int sfa_offsets_powerlaw(const double* u, int32_t m, double sigma, int32_t n, int32_t* out,
                         int32_t cap, int32_t* n_out);

const char* sfa_status_string(int status);

/* ---- device entry points ------------------------------------------- */

/* Bytes of the RoPE table for T positions (D = 64): T * 32 * 2 floats. */
int sfa_rope_table_bytes(int32_t T, size_t* bytes);

/* Fill `table` (device, sfa_rope_table_bytes(T)) with cos and sin of
 * phi(t, j) = t * theta^(-2j/64), t < T, j < 32, evaluated in fp64 and
 * stored fp32, laid out [T][32][2] = (cos, sin).  Rotation pairs are
 * (j, j + 32) ("rotate half").  theta > 0. */
int sfa_rope_table(int32_t T, double theta, float* table, void* stream);

/* RoPE-rotated keys for d->k_rot: writes k_rot [B, Hkv, T, 64] = k rotated
 * at each row's position by d->rope (fp32 rotation, one bf16 rounding).
 * bf16 only (SFA_ERR_UNSUPPORTED otherwise); d->rope must be set. */
int sfa_rope_keys(const sfa_desc* d, const void* k, void* k_rot, void* stream);

/* Workspace bytes a call needs: interp != 0 for sfa_forward / sfa_backward,
 * 0 for the integer path; backward != 0 for the backward calls.  The forward
 * keeps the RoPE-rotated keys there (bf16 I/O); the backward keeps them,
 * delta = rowsum(dO * O), the rotated queries and the per-(query, slot, head)
 * softmax terms its key-side kernel reads, and the per-block partial sums of
 * dL/dalpha.  The contents are scratch: nothing persists between calls. */
int sfa_workspace_size(const sfa_desc* d, int interp, int backward, size_t* bytes);

/* Interpolated-path forward.  Writes o [B,Hq,T,64] (d->dtype) and lse
 * (fp32 [B,Hq,T], natural log of the softmax denominator including the max
 * shift).  Keys for query i: window distances 0..min(W, i) and every rung
 * of sfa_rung_table with c_k <= i (a rung whose position precedes the
 * sequence is absent, not zero-filled).  ws must hold
 * sfa_workspace_size(d, 1, 0) bytes (may be NULL when that is 0). */
int sfa_forward(const sfa_desc* d, const void* q, const void* k, const void* v, void* o,
                float* lse, void* ws, size_t ws_bytes, void* stream);

/* Interpolated-path backward.  Inputs are those of the forward plus its
 * o and lse and the upstream gradient dO.  Writes dq, dk, dv (d->dtype) and,
 * if dalpha_dtheta != NULL, two device doubles: dL/dalpha and
 * dL/dtheta = dL/dalpha * (alpha - 0.5) * (1.5 - alpha).  At an integer
 * rung distance the alpha-derivative is the one-sided one from below
 * (the interpolation weight w = c - d with c held fixed).  ws must hold
 * sfa_workspace_size(d, 1) bytes. */
int sfa_backward(const sfa_desc* d, const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dO, void* dq, void* dk, void* dv,
                 double* dalpha_dtheta, void* ws, size_t ws_bytes, void* stream);

/* Integer-offset fast path ("Depth-Staggered ...", method section: integer
 * offsets as an exact gather; "Christoffel-Balanced Sparse Attention": keys
 * i - o kept when >= 0).  Keys for query i: i - s for every s in d->dist
 * with 0 <= i - s < T.  A negative s reads the future row i + |s| (signed
 * offsets for bidirectional attention, same page).  bf16 sets with a band plan
 * (sfa_band_plan; signed sets included) run the band kernels, other bf16 sets
 * without negative distances and with G = 4, 8 or 16 the rung kernels, every
 * other set the fp32 SIMT kernels.  Same outputs as sfa_forward / sfa_backward without the alpha
 * gradient. */
int sfa_forward_int(const sfa_desc* d, const void* q, const void* k, const void* v, void* o,
                    float* lse, void* ws, size_t ws_bytes, void* stream);
int sfa_backward_int(const sfa_desc* d, const void* q, const void* k, const void* v,
                     const void* o, const float* lse, const void* dO, void* dq, void* dk,
                     void* dv, void* ws, size_t ws_bytes, void* stream);

/* Incremental decode on the integer path: one new query per sequence
 * against a key/value cache ("Depth-Staggered ...": the method's efficiency
 * case is inference; "Christoffel-Balanced Sparse Attention": gather only
 * the allowed offsets of each query).
 *   q        [B, Hq, 64]     the queries, sequence b at position pos[b]
 *   k_cache  [B, Hkv, T, 64] raw (unrotated) keys; T = d->T is the capacity,
 *   v_cache  [B, Hkv, T, 64] rows 0..pos[b] of sequence b must be written
 *   pos      device int32 [B], 0 <= pos[b] < T (sequences may differ)
 *   o        [B, Hq, 64]     output (d->dtype)
 *   lse      fp32 [B, Hq]    natural-log softmax denominator, or NULL
 * Keys of sequence b: pos[b] - s for every s in d->dist with s <= pos[b]
 * (d->dist must contain 0 and no negative distance: a cache holds no future
 * keys; SFA_ERR_INVALID_ARG otherwise).  With d->rope the query is rotated at pos[b] and
 * each gathered key at its own position.  The result is row pos[b] of
 * sfa_forward_int over that sequence's prefix, computed in fp32.  No
 * workspace.  A position outside [0, T) is skipped on the device and
 * recorded as SFA_ERR_DEVICE_BOUNDS. */
int sfa_decode_int(const sfa_desc* d, const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* pos, void* o, float* lse, void* stream);

/* Allocation-free variant of sfa_forward (no counterpart on the pages; it
 * exists for callers that cannot allocate device memory: programs whose
 * allocator owns all device memory and bars raw cudaMalloc from libraries,
 * or that run under a hard memory budget).  Same arguments and results as
 * sfa_forward without ws / ws_bytes: the scratch lives in a file-scope device
 * array of SFA_STATIC_WS_BYTES that every GPU loading the library keeps until
 * the process exits.  Calls whose sfa_workspace_size(d, 1, 0) exceeds that
 * return SFA_ERR_CAPACITY and launch nothing (B * Hkv * T <= 65536 rows with
 * RoPE, e.g. B = 32, Hkv = 2, T = 1024; a call given d->k_rot needs no
 * scratch and has no such limit).  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress, that device current); make it
 * before any stream capture.  The address is kept with the context it belongs
 * to, and a call from a new context of that device (after cudaDeviceReset,
 * say) looks it up again, before launching.  Nothing is allocated or freed.  All
 * calls share the one array: calls that overlap on the GPU (other streams,
 * other threads) race on it; serialize them.  The array needs no clearing
 * (each call writes the scratch rows it reads). */
#define SFA_STATIC_WS_BYTES (8u << 20)
int sfa_forward_noalloc(const sfa_desc* d, const void* q, const void* k, const void* v, void* o,
                        float* lse, void* stream);

/* Per-kernel timing for measurement tools.  While enabled, every kernel the
 * library launches is bracketed by two CUDA events recorded on its own
 * stream.  sfa_timing_read waits for the recorded events, writes for each
 * kernel kind (index = sfa_kernel_kind) the summed milliseconds and the
 * launch count into arrays of n entries, and forgets the records.  Enabling
 * adds two event records per launch; nothing else changes. */
typedef enum {
  SFA_KERNEL_FWD = 0,
  SFA_KERNEL_BWD_Q = 1,
  SFA_KERNEL_BWD_KV = 2,
  SFA_KERNEL_DALPHA = 3,
  SFA_KERNEL_ROPE = 4,
  SFA_KERNEL_PREP = 5, /* RoPE-rotated bf16 copy of K for the tensor-core kernels */
  SFA_KERNEL_DECODE = 6,
  SFA_KERNEL_KINDS = 7
} sfa_kernel_kind;
int sfa_timing_enable(int on);
int sfa_timing_read(double* ms, int64_t* launches, int n);

/* Synchronise `stream`, return in *out the device status word (an
 * sfa_status recorded by a kernel's bounds check or bounded wait since the
 * last call, SFA_OK if none) and clear it. */
int sfa_get_device_status(void* stream, int32_t* out);

/* Kernel selection options (process-wide; read by every later call).
 * SFA_OPT_BAND_FWD_TC05: the band forward (integer sets with a band plan,
 * bf16) runs on the fifth-generation tensor cores with TMEM accumulators and
 * 128 query rows per CTA (1) or on the mma.sync kernel with 64 rows per CTA
 * (0, the default: faster on the Christoffel configuration, 42 against 56 us
 * per call on a GB300).  Both compute the same keys and are checked against
 * the same bounds; the option exists to compare them.  Returns
 * SFA_ERR_INVALID_ARG for an unknown option or value. */
typedef enum { SFA_OPT_BAND_FWD_TC05 = 0 } sfa_option;
int sfa_set_option(int32_t option, int32_t value);

/* Test injection for the bounded waits (no counterpart on the pages; for
 * tests of the failure path only).  Every mbarrier wait of the TMA-staged
 * kernels gives up after `wait_cycles` SM clock cycles (0 restores the
 * default of 2e9, about 1 s at 2.07 GHz); the CTA then records
 * SFA_ERR_TIMEOUT in the device status word, waits (bounded) for its own
 * loads in flight and leaves.  skip_group >= 0 makes CTA (0, 0) of the rung
 * tensor-core forward and query-side backward issue neither the expect_tx
 * nor the loads of that staged group (window chunks first, then rung pairs),
 * so its consumers' wait runs out with nothing in flight; -1 turns this off.
 * The setting is process-wide and read by every later call until changed;
 * the outputs of a call that timed out are undefined.  Returns
 * SFA_ERR_INVALID_ARG for wait_cycles < 0 or skip_group < -1. */
int sfa_debug_inject(int64_t wait_cycles, int32_t skip_group);

#ifdef __cplusplus
}
#endif

#endif /* SFA_H */
