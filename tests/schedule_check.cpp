// Host-side check of the tensor-core kernel's work partition (the same inline
// functions the kernels use): the per-CTA ranges tile [0, T) exactly and in
// order, differ in length by at most one tile, and tc_owner inverts them.
#include <cstdio>

#include "decode_tc_launch.h"

using namespace pkv;

static int check(int64_t T, int64_t NW) {
  int64_t next = 0, minlen = T + 1, maxlen = -1;
  for (int64_t k = 0; k < NW; ++k) {
    const int64_t lo = tc_range_lo(k, T, NW), hi = tc_range_lo(k + 1, T, NW);
    if (lo != next || hi < lo) {
      std::printf("FAIL range T=%lld NW=%lld k=%lld\n", (long long)T, (long long)NW, (long long)k);
      return 1;
    }
    minlen = hi - lo < minlen ? hi - lo : minlen;
    maxlen = hi - lo > maxlen ? hi - lo : maxlen;
    for (int64_t x = lo; x < hi; x += (hi - lo + 2) / 3)
      if (tc_owner(x, T, NW) != k) {
        std::printf("FAIL owner T=%lld NW=%lld x=%lld\n", (long long)T, (long long)NW, (long long)x);
        return 1;
      }
    if (hi > lo && tc_owner(hi - 1, T, NW) != k) {
      std::printf("FAIL owner(last) T=%lld NW=%lld k=%lld\n", (long long)T, (long long)NW,
                  (long long)k);
      return 1;
    }
    next = hi;
  }
  if (next != T || maxlen - minlen > 1) {
    std::printf("FAIL cover/balance T=%lld NW=%lld\n", (long long)T, (long long)NW);
    return 1;
  }
  return 0;
}

int main() {
  int bad = 0;
  for (int64_t NW : {1, 7, 148, 152, 160, 1824})
    for (int64_t T : {1, 2, 15, 100, 511, 4096, 32768, 100003, 1048576, 20000017})
      bad |= check(T, NW);
  std::printf(bad ? "partition check FAILED\n" : "partition check ok\n");
  return bad;
}
