// Host routing plan of sigma-routed sequence sharding (no device code).
//
// A long sequence is split over `world` ranks twice with the same chunk
// c = ceil(n / world): rank r holds the ORIGINAL tokens [r c, (r+1) c) of
// Q, K, V and of the output, and computes the SA rows of the PERMUTED
// positions [r c, (r+1) c) ("Core mechanism": sliding-window attention over
// the permuted order).  Those rows need the keys of the positions within the
// window, so rank r works on the span [r c - left, (r+1) c + right) clipped
// to [0, n): its local rows are the span's tokens, gathered from their
// owners by one all-to-all, and its own rows go back to their tokens' owners
// by a second one.
//
// The local rows are the span's tokens in ascending ORIGINAL order, and the
// local permutation maps each span position to its token's local row.  The
// relabelling is monotone, so the causal rule sigma(q) <= sigma(p)
// ("Theoretical properties") compares local rows exactly as it compares the
// original tokens, and the ordinary forward kernels run the local problem
// unchanged.  The local problem's windows are complete for the owned
// positions (their whole window lies in the span, or is cut by the sequence
// ends exactly as globally); the halo positions' rows are computed but not
// used.
#include <algorithm>
#include <vector>

#include "sa_internal.h"

namespace sa {

static void shard_bounds(int32_t n, int32_t window, int32_t world, int32_t rank, int64_t& c,
                         int64_t& own0, int64_t& own1, int64_t& s0, int64_t& s1) {
  const int64_t h = window / 2;
  c = (int64_t(n) + world - 1) / world;
  own0 = std::min<int64_t>(int64_t(rank) * c, n);
  own1 = std::min<int64_t>(own0 + c, n);
  s0 = std::max<int64_t>(0, own0 - h);
  s1 = std::min<int64_t>(n, own1 + h);
  if (own1 <= own0) s0 = s1 = own0;  // a rank beyond the end owns nothing
}

}  // namespace sa

using namespace sa;

extern "C" int32_t sa_shard_span(int32_t n, int32_t window, int32_t world, int32_t rank) {
  if (n < 1 || window < 1 || world < 1 || rank < 0 || rank >= world) return 0;
  int64_t c, o0, o1, s0, s1;
  shard_bounds(n, window, world, rank, c, o0, o1, s0, s1);
  return int32_t(s1 - s0);
}

extern "C" sa_status_t sa_shard_plan(const int32_t* perm_host, int32_t n, int32_t window,
                                     int32_t world, int32_t rank, int32_t* tokens,
                                     int32_t* local_perm, int32_t capacity,
                                     int32_t* span_begin, int32_t* own_begin,
                                     int32_t* own_end) {
  if (!perm_host || !tokens || !local_perm || !span_begin || !own_begin || !own_end)
    return fail(SA_ERR_INVALID_ARG, "sa_shard_plan: pointers must be non-NULL");
  if (n < 1 || window < 1 || world < 1 || rank < 0 || rank >= world)
    return fail(SA_ERR_INVALID_ARG, "sa_shard_plan: need n, window, world >= 1 and 0 <= rank < world");
  int64_t c, o0, o1, s0, s1;
  shard_bounds(n, window, world, rank, c, o0, o1, s0, s1);
  const int64_t m = s1 - s0;
  if (capacity < m)
    return fail(SA_ERR_INVALID_ARG, "sa_shard_plan: capacity %d below the span of %lld positions",
                capacity, (long long)m);
  // sigma must be a permutation: every entry in range, none repeated
  std::vector<unsigned char> seen(size_t(n), 0);
  for (int32_t p = 0; p < n; ++p) {
    const int32_t t = perm_host[p];
    if (t < 0 || t >= n || seen[size_t(t)])
      return fail(SA_ERR_BAD_PERM, "sa_shard_plan: perm is not a permutation (entry %d at %d)", t, p);
    seen[size_t(t)] = 1;
  }
  std::vector<int32_t> sorted(perm_host + s0, perm_host + s1);
  std::sort(sorted.begin(), sorted.end());
  for (int64_t i = 0; i < m; ++i) tokens[i] = sorted[size_t(i)];
  for (int64_t j = 0; j < m; ++j)
    local_perm[j] = int32_t(std::lower_bound(sorted.begin(), sorted.end(), perm_host[s0 + j]) -
                            sorted.begin());
  *span_begin = int32_t(s0);
  *own_begin = int32_t(o0);
  *own_end = int32_t(o1);
  return SA_OK;
}
