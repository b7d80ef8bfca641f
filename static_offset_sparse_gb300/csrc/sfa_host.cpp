// Host-side builders of libsfa: offset lists, alpha schedules, rung tables and
// argument validation.  Integer work is exact (64-bit); the rung distances are
// fp64 products as the method defines them.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "sfa_internal.h"

extern "C" {

int sfa_offsets_fib(int32_t K, int32_t* out) {
  // "Depth-Staggered Fibonacci Spacing for Sparse Attention", method section:
  // base 1, 2, 3, 5, ... (15 terms reach 987).  Term 40 is 165580141 < 2^31.
  if (K < 1 || K > 40 || !out) return SFA_ERR_INVALID_ARG;
  int64_t a = 1, b = 2;
  for (int32_t j = 0; j < K; ++j) {
    out[j] = (int32_t)a;
    int64_t n = a + b;
    a = b;
    b = n;
  }
  return SFA_OK;
}

int sfa_offsets_pow2(int32_t K, int32_t* out) {
  // Same page, the reach-matched power-of-2 control base.
  if (K < 1 || K > 31 || !out) return SFA_ERR_INVALID_ARG;
  for (int32_t j = 0; j < K; ++j) out[j] = (int32_t)(1u << j);
  return SFA_OK;
}

int sfa_offsets_christoffel(int32_t m, int32_t k, int32_t include_zero, int32_t* out,
                            int32_t cap, int32_t* n_out) {
  // "Christoffel-Balanced Sparse Attention": c[j] = floor((j+1)m/k) - floor(jm/k).
  if (!n_out || m <= 0 || k <= 0 || m > k || k > (1 << 30)) return SFA_ERR_INVALID_ARG;
  std::vector<int32_t> o;
  o.reserve((size_t)m + 1);
  const int64_t M = m, Kp = k;
  for (int64_t j = 0; j < Kp; ++j) {
    int64_t cj = ((j + 1) * M) / Kp - (j * M) / Kp;  // both operands >= 0: floor
    if (cj == 1) o.push_back((int32_t)j);
  }
  if (include_zero && (o.empty() || o[0] != 0)) o.insert(o.begin(), 0);
  *n_out = (int32_t)o.size();
  if ((int64_t)o.size() > (int64_t)cap) return SFA_ERR_CAPACITY;
  if (!out && !o.empty()) return SFA_ERR_INVALID_ARG;
  std::copy(o.begin(), o.end(), out);
  return SFA_OK;
}

int sfa_alpha_schedule(int32_t L, int32_t kind, int32_t S, double* out) {
  // "Depth-Staggered ...", method section: fixed, linear ramp 0.5 .. 1.5, and
  // the coprime reassignment l -> S l mod L of the linear values.
  if (L < 1 || L > 4096 || !out) return SFA_ERR_INVALID_ARG;
  if (kind == SFA_SCHED_FIXED) {
    for (int32_t l = 0; l < L; ++l) out[l] = 1.0;
    return SFA_OK;
  }
  auto lin = [L](int64_t l) { return L > 1 ? 0.5 + (double)l / (double)(L - 1) : 1.0; };
  if (kind == SFA_SCHED_LINEAR) {
    for (int32_t l = 0; l < L; ++l) out[l] = lin(l);
    return SFA_OK;
  }
  if (kind == SFA_SCHED_COPRIME) {
    if (S <= 0) return SFA_ERR_INVALID_ARG;
    int64_t a = S, b = L;
    while (b) {
      int64_t t = a % b;
      a = b;
      b = t;
    }
    if (a != 1) return SFA_ERR_INVALID_ARG;
    for (int32_t l = 0; l < L; ++l) out[l] = lin(((int64_t)S * l) % L);
    return SFA_OK;
  }
  return SFA_ERR_INVALID_ARG;
}

int sfa_rung_table(const int32_t* base, int32_t n_base, double alpha, int32_t W,
                   int32_t* c_out, float* w_out, float* f_out, int32_t cap, int32_t* n_out) {
  if (!n_out || n_base < 0 || (n_base > 0 && !base) || W < -1) return SFA_ERR_INVALID_ARG;
  if (!(alpha > 0.0) || !std::isfinite(alpha)) return SFA_ERR_INVALID_ARG;
  struct R {
    int64_t c;
    double w;
    int32_t f;
  };
  std::vector<R> rs;
  for (int32_t j = 0; j < n_base; ++j) {
    if (base[j] <= 0) return SFA_ERR_INVALID_ARG;
    const double d = alpha * (double)base[j];  // fl64(alpha * f_k)
    if (!(d <= 2147483647.0)) return SFA_ERR_INVALID_ARG;
    if (d <= (double)W) continue;  // inside the window: the union keeps it once
    const double c = std::ceil(d);
    rs.push_back({(int64_t)c, c - d, base[j]});
  }
  std::stable_sort(rs.begin(), rs.end(), [](const R& a, const R& b) { return a.c < b.c; });
  *n_out = (int32_t)rs.size();
  if ((int64_t)rs.size() > (int64_t)cap) return SFA_ERR_CAPACITY;
  for (size_t j = 0; j < rs.size(); ++j) {
    if (c_out) c_out[j] = (int32_t)rs[j].c;
    if (w_out) w_out[j] = (float)rs[j].w;
    if (f_out) f_out[j] = (float)rs[j].f;
  }
  return SFA_OK;
}

int sfa_int_distances(const int32_t* dist, int32_t n_dist, int32_t* out, int32_t cap,
                      int32_t* n_out) {
  if (!n_out || n_dist < 0 || (n_dist > 0 && !dist)) return SFA_ERR_INVALID_ARG;
  std::vector<int32_t> s(dist, dist + n_dist);
  for (int32_t x : s)
    if (x <= -(1 << 30) || x >= (1 << 30)) return SFA_ERR_INVALID_ARG;
  std::sort(s.begin(), s.end());
  s.erase(std::unique(s.begin(), s.end()), s.end());
  *n_out = (int32_t)s.size();
  if ((int64_t)s.size() > (int64_t)cap) return SFA_ERR_CAPACITY;
  if (!out && !s.empty()) return SFA_ERR_INVALID_ARG;
  std::copy(s.begin(), s.end(), out);
  return SFA_OK;
}

int sfa_band_plan(const int32_t* dist, int32_t n_dist, int32_t T, int32_t G, int32_t* delta,
                  int32_t* run_start, int32_t* run_len, int32_t cap, int32_t* n_runs) {
  if (!delta || !n_runs || T <= 0 || G <= 0 || cap < 0) return SFA_ERR_INVALID_ARG;
  std::vector<int32_t> s((size_t)(n_dist > 0 ? n_dist : 0));
  int32_t n = 0;
  int rc = sfa_int_distances(dist, n_dist, s.data(), n_dist, &n);
  if (rc != SFA_OK) return rc;
  sfa::BandPlan p;
  sfa::band_plan_of(s.data(), n, T, G, &p);
  *delta = p.delta;
  *n_runs = p.nruns;
  if (p.nruns > cap) return SFA_ERR_CAPACITY;
  if (p.nruns > 0 && (!run_start || !run_len)) return SFA_ERR_INVALID_ARG;
  for (int32_t m = 0; m < p.nruns; ++m) {
    run_start[m] = p.a[m];
    run_len[m] = p.len[m];
  }
  return SFA_OK;
}

const char* sfa_status_string(int s) {
  switch (s) {
    case SFA_OK: return "ok";
    case SFA_ERR_INVALID_ARG: return "invalid argument";
    case SFA_ERR_UNSUPPORTED: return "unsupported configuration";
    case SFA_ERR_CAPACITY: return "output or workspace too small";
    case SFA_ERR_CUDA: return "CUDA runtime error";
    case SFA_ERR_TIMEOUT: return "device wait timed out";
    case SFA_ERR_DEVICE_BOUNDS: return "device index check failed";
    default: return "unknown status";
  }
}

}  // extern "C"

namespace sfa {

int validate_shape(const sfa_desc* d) {
  if (!d) return SFA_ERR_INVALID_ARG;
  if (d->B <= 0 || d->T <= 0 || d->Hq <= 0 || d->Hkv <= 0) return SFA_ERR_INVALID_ARG;
  if (d->dtype != SFA_F32 && d->dtype != SFA_BF16) return SFA_ERR_INVALID_ARG;
  if (d->D != kD) return SFA_ERR_UNSUPPORTED;
  if (d->Hq % d->Hkv != 0) return SFA_ERR_UNSUPPORTED;
  const int G = d->Hq / d->Hkv;
  if (G > 32 || (G & (G - 1)) != 0) return SFA_ERR_UNSUPPORTED;
  if (d->T > (1 << 24) || d->B > 65535 || (int64_t)d->B * d->Hkv > 65535)
    return SFA_ERR_UNSUPPORTED;  // grid y = B * Hkv
  return SFA_OK;
}

int build_interp_plan(const sfa_desc* d, Plan* p) {
  if (d->W < 0) return SFA_ERR_INVALID_ARG;
  int32_t n = 0;
  int rc = sfa_rung_table(d->base, d->n_base, d->alpha, d->W, p->c, p->w, p->f, kMaxRungs, &n);
  if (rc == SFA_ERR_CAPACITY) return SFA_ERR_UNSUPPORTED;
  if (rc != SFA_OK) return rc;
  p->W = d->W;
  p->n = n;
  p->interp = 1;
  return SFA_OK;
}

int build_int_plan(const sfa_desc* d, Plan* p) {
  if (d->n_dist <= 0 || !d->dist) return SFA_ERR_INVALID_ARG;
  std::vector<int32_t> s((size_t)d->n_dist);
  int32_t n = 0;
  int rc = sfa_int_distances(d->dist, d->n_dist, s.data(), d->n_dist, &n);
  if (rc != SFA_OK) return rc;
  s.resize((size_t)n);
  // Distance 0 (the query itself) must be present so that no query has an
  // empty key set, as the window of the method guarantees.
  const size_t z = (size_t)(std::lower_bound(s.begin(), s.end(), 0) - s.begin());
  if (z == s.size() || s[z] != 0) return SFA_ERR_INVALID_ARG;
  // The contiguous run 0..W runs as a window; every other distance is an
  // exact rung, ascending: negative ones (future keys of a signed,
  // bidirectional set) first, then those beyond the window.
  int32_t W = -1;
  size_t j = z;
  while (j < s.size() && s[j] == W + 1) {
    ++W;
    ++j;
  }
  const size_t nr = z + (s.size() - j);
  if (nr > (size_t)kMaxRungs) return SFA_ERR_UNSUPPORTED;
  p->W = W;
  p->n = (int32_t)nr;
  p->interp = 0;
  for (size_t r = 0; r < nr; ++r) {
    p->c[r] = r < z ? s[r] : s[j + (r - z)];
    p->w[r] = 0.0f;
    p->f[r] = 0.0f;
  }
  return SFA_OK;
}

// Band plan.  For each step delta <= 64 dividing T, the set splits into runs
// of step delta (a distance extends the run of s - delta when that is in the
// set); a query tile of 64 / G positions then meets ceil((64 / G + len - 1) /
// 64) key tiles of 64 rows per run.  The step with the fewest tiles wins
// (the smallest on ties).  Where the rung kernels could take the set (G = 4
// or 8, no negative distance) the plan is used when at least one product in
// eight is a wanted (query, key) pair, i.e. n >= 8 x tiles; elsewhere the
// alternative is the fp32 SIMT path, which every plan beats (measured down to
// the Fibonacci set at G = 1, 19 distances in 12 tiles: 0.38 against 0.75 ms),
// so any plan is used.  Distances with |d| >= T reach no key and are left
// out.  Signed (bidirectional) sets are runs like any other: a negative
// distance reads a later key, and the kernels clip every band to the
// sequence at both ends.
int band_plan_of(const int32_t* s0, int n, int T, int G, BandPlan* p) {
  p->delta = 0;
  p->nruns = 0;
  if (G != 1 && G != 2 && G != 4 && G != 8) return SFA_OK;
  if (n <= 0 || !std::binary_search(s0, s0 + n, 0)) return SFA_OK;  // no distance 0
  int first = 0, m = n;
  while (first < n && s0[first] <= -T) ++first;
  while (m > first && s0[m - 1] >= T) --m;
  const int32_t* s = s0 + first;
  m -= first;
  const int BU = 64 / G;
  int64_t best = -1;
  std::vector<int32_t> ra, rl, run_of((size_t)m);
  for (int delta = 1; delta <= kMaxBandDelta && delta <= T; ++delta) {
    if (T % delta) continue;
    ra.clear();
    rl.clear();
    for (int x = 0; x < m; ++x) {
      const int32_t prev = s[x] - delta;
      const int32_t* it = std::lower_bound(s, s + x, prev);
      if (it != s + x && *it == prev) {
        run_of[(size_t)x] = run_of[(size_t)(it - s)];
        ++rl[(size_t)run_of[(size_t)x]];
      } else {
        run_of[(size_t)x] = (int32_t)ra.size();
        ra.push_back(s[x]);
        rl.push_back(1);
      }
    }
    if (ra.size() > (size_t)kMaxRuns) continue;
    int64_t cost = 0;
    for (int32_t len : rl) cost += (BU + len - 1 + 63) / 64;
    if (best < 0 || cost < best) {
      best = cost;
      p->delta = delta;
      p->nruns = (int32_t)ra.size();
      std::copy(ra.begin(), ra.end(), p->a);
      std::copy(rl.begin(), rl.end(), p->len);
    }
  }
  const bool rung_ok = (G == 4 || G == 8) && s0[0] >= 0;
  if (best < 0 || (rung_ok && (int64_t)m < 8 * best)) {
    p->delta = 0;
    p->nruns = 0;
  }
  return SFA_OK;
}

int build_band_plan(const sfa_desc* d, BandPlan* p) {
  p->delta = 0;
  p->nruns = 0;
  if (d->dtype != SFA_BF16 || d->n_dist <= 0 || !d->dist) return SFA_OK;
  std::vector<int32_t> s((size_t)d->n_dist);
  int32_t n = 0;
  int rc = sfa_int_distances(d->dist, d->n_dist, s.data(), d->n_dist, &n);
  if (rc != SFA_OK) return rc;
  return band_plan_of(s.data(), n, d->T, d->Hq / d->Hkv, p);
}

}  // namespace sfa
