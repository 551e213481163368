// Host check of the MMA issuer's item decoding: KRanges must give, for every CTA
// and item of every schedule below, the k-steps [k0, k1) that get_item gives; and
// in split mode the fixup warps' piece count must be the CTA's item count.
// Prints "ok <items checked>" and exits 0, or the first disagreement and exits 1.
#include <cstdio>
#include <initializer_list>

#include "sg_sched.cuh"

using namespace sg;

static bool check(const Schedule& s, long long& n) {
  for (int32_t c = 0; c < s.grid; ++c) {
    const KRanges kr(s, c);
    const int32_t items = item_count(s, c);
    // split mode: a CTA's one item is its one k piece (the fixup warps count on it)
    if (s.split > 0 && sk_count(s, c) != items) {
      std::printf("split mode: sk_count %d != item_count %d (cta %d)\n", sk_count(s, c), items, c);
      return false;
    }
    for (int32_t i = 0; i < items; ++i) {
      const WorkItem w = get_item(s, c, i);
      int32_t k0 = -1, k1 = -1;
      kr.range(i, k0, k1);
      ++n;
      if (k0 != w.k0 || k1 != w.k1) {
        std::printf("mismatch: tiles %d x %d, k_steps %d, grid %d, split %d, cta %d, item %d: (%d, %d) vs (%d, %d)\n",
                    s.tiles_m, s.tiles_n, s.k_steps, s.grid, s.split, c, i, k0, k1, w.k0, w.k1);
        return false;
      }
    }
  }
  return true;
}

int main() {
  long long n = 0;
  const int32_t tms[] = {1, 2, 3, 7, 8, 16, 31, 64};
  const int32_t tns[] = {1, 2, 5, 16, 43, 64};
  const int32_t kss[] = {1, 2, 3, 32, 64, 127, 172};
  const int32_t ctas[] = {1, 2, 64, 74, 76, 148, 152, 304};
  for (int32_t tm : tms)
    for (int32_t tn : tns)
      for (int32_t ks : kss)
        for (int32_t g : ctas) {
          for (int fill = 0; fill < 2; ++fill)
            if (!check(make_schedule(tm, tn, ks, g, 4, tm < 8 ? tm : 8, fill != 0), n)) return 1;
          for (int32_t split : {1, 2, 3, 5, 9})
            if (!check(make_split_schedule(tm, tn, ks, split), n)) return 1;
        }
  std::printf("ok %lld\n", n);
  return 0;
}
