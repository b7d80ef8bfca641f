// Offset-schedule analysis (reachability through a stack of shared-offset
// layers, residue classes, offset histograms) and the shared power-law
// offset list.  Host code; declarations and definitions in include/sfa.h.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "sfa_internal.h"

namespace {

// dst |= src << s over a bitset of nw 64-bit words (bits past the end drop).
void or_shifted(uint64_t* dst, const uint64_t* src, int64_t nw, int64_t s) {
  const int64_t ws = s >> 6;
  const int bs = (int)(s & 63);
  if (ws >= nw) return;
  if (bs == 0) {
    for (int64_t w = nw - 1; w >= ws; --w) dst[w] |= src[w - ws];
  } else {
    for (int64_t w = nw - 1; w > ws; --w)
      dst[w] |= (src[w - ws] << bs) | (src[w - ws - 1] >> (64 - bs));
    dst[ws] |= src[0] << bs;
  }
}

}  // namespace

extern "C" int sfa_reach(const int32_t* dist, const int32_t* layer_start, int32_t L, int32_t T,
                         int32_t* hops, int64_t* covered) {
  if (!layer_start || !hops || L < 1 || L > 4096 || T < 1 || T > (1 << 24))
    return SFA_ERR_INVALID_ARG;
  if (layer_start[0] != 0) return SFA_ERR_INVALID_ARG;
  for (int32_t l = 0; l < L; ++l)
    if (layer_start[l + 1] < layer_start[l]) return SFA_ERR_INVALID_ARG;
  if (layer_start[L] > 0 && !dist) return SFA_ERR_INVALID_ARG;
  for (int32_t j = 0; j < layer_start[L]; ++j)
    if (dist[j] < 0) return SFA_ERR_INVALID_ARG;
  const int64_t nw = ((int64_t)T + 63) / 64;
  const uint64_t tail = (T % 64) ? ((uint64_t)1 << (T % 64)) - 1 : ~(uint64_t)0;
  std::vector<uint64_t> cur(nw, 0), nxt(nw), seen(nw, 0);
  cur[0] = seen[0] = 1;  // before any layer: distance 0
  for (int32_t d = 0; d < T; ++d) hops[d] = -1;
  hops[0] = 0;
  for (int32_t l = 0; l < L; ++l) {
    std::fill(nxt.begin(), nxt.end(), 0);
    for (int32_t j = layer_start[l]; j < layer_start[l + 1]; ++j)
      if (dist[j] < T) or_shifted(nxt.data(), cur.data(), nw, dist[j]);
    nxt[nw - 1] &= tail;
    int64_t cnt = 0;
    for (int64_t w = 0; w < nw; ++w) {
      cnt += __builtin_popcountll(nxt[w]);
      uint64_t fresh = nxt[w] & ~seen[w];
      seen[w] |= fresh;
      while (fresh) {
        const int b = __builtin_ctzll(fresh);
        hops[w * 64 + b] = l + 1;
        fresh &= fresh - 1;
      }
    }
    if (covered) covered[l] = cnt;
    cur.swap(nxt);
  }
  return SFA_OK;
}

extern "C" int sfa_residue_classes(const int32_t* hops, int32_t T, int32_t M, int64_t* out) {
  if (!hops || !out || T < 1 || M < 1 || M > T) return SFA_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(int64_t) * (size_t)M);
  for (int32_t d = 0; d < T; ++d)
    if (hops[d] >= 0) ++out[d % M];
  return SFA_OK;
}

extern "C" int sfa_offset_histogram(const int32_t* dist, int32_t n, int32_t T, int32_t nb,
                                    int64_t* out) {
  if (n < 0 || (n > 0 && !dist) || T < 1 || nb < 2 || !out) return SFA_ERR_INVALID_ARG;
  std::vector<int32_t> d;
  for (int32_t j = 0; j < n; ++j)
    if (dist[j] >= 0 && dist[j] < T) d.push_back(dist[j]);
  std::sort(d.begin(), d.end());
  d.erase(std::unique(d.begin(), d.end()), d.end());
  std::memset(out, 0, sizeof(int64_t) * (size_t)nb);
  for (int32_t x : d) {
    int b = 0;
    if (x > 0) b = std::min(nb - 1, 32 - __builtin_clz((unsigned)x));  // bit length
    ++out[b];
  }
  return SFA_OK;
}

extern "C" int sfa_offsets_powerlaw(const double* u, int32_t m, double sigma, int32_t n,
                                    int32_t* out, int32_t cap, int32_t* n_out) {
  if (!u || m < 1 || n < 2 || n > (1 << 26) || !(sigma >= 0.0) || !n_out) return SFA_ERR_INVALID_ARG;
  for (int32_t j = 0; j < m; ++j)
    if (!(u[j] >= 0.0 && u[j] < 1.0)) return SFA_ERR_INVALID_ARG;
  const int32_t Dmax = n / 2;
  std::vector<double> c((size_t)Dmax);
  double acc = 0.0;
  for (int32_t v = 1; v <= Dmax; ++v) {  // c_d, summed in increasing v
    acc += std::pow((double)v, -(1.0 + sigma));
    c[(size_t)v - 1] = acc;
  }
  const double Z = c[(size_t)Dmax - 1];
  std::vector<int32_t> d((size_t)m);
  for (int32_t j = 0; j < m; ++j) {  // smallest d with c_d > u_j Z
    const double t = u[j] * Z;
    d[(size_t)j] = (int32_t)(std::upper_bound(c.begin(), c.end(), t) - c.begin()) + 1;
    if (d[(size_t)j] > Dmax) d[(size_t)j] = Dmax;  // t >= Z cannot occur for u < 1, kept in range
  }
  std::sort(d.begin(), d.end());
  d.erase(std::unique(d.begin(), d.end()), d.end());
  *n_out = (int32_t)d.size();
  if (*n_out > cap) return SFA_ERR_CAPACITY;
  if (!out) return SFA_ERR_INVALID_ARG;
  std::copy(d.begin(), d.end(), out);
  return SFA_OK;
}
