// Host-side check of the tensor-core kernel's work partition (the same inline
// functions the kernels use), compiled with g++:
//  * tc_range_lo / tc_owner split [0, V) evenly and tc_owner inverts them;
//  * the cost-weighted schedule: for random batches (empty, short and long
//    contexts), the CTAs' tile runs tile [0, T) exactly and in order, the unit
//    owner of every tile is the CTA whose run holds it, and each CTA's cost
//    (tiles + seg_cost per segment) stays within one pair of the even share;
//  * pieces: walking every CTA's segments the way the kernel does, each
//    partial segment (piece) takes a slot no other segment of its CTA takes;
//    for every piece, tc_pair_ctas names the CTAs cf .. cl of its pair, and
//    the merge's lookup (the non-empty CTAs of cf .. cl, slot 1 for cf and 0
//    for the others) names exactly the records written for every split
//    pair; no pair is both whole and split;
//  * the head piece: a piece is the one the CTA merges without publishing
//    (its pair's first tiles, slot 1) exactly when its CTA is cf, and it is
//    always that CTA's last segment.
#include <cstdio>
#include <algorithm>
#include <cstdlib>
#include <map>
#include <set>
#include <utility>
#include <vector>

#include "decode_tc_launch.h"

using namespace pkv;

static int check_even(int64_t T, int64_t NW) {
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

static uint64_t rng_state = 245;
static uint64_t rnd() {  // splitmix64
  uint64_t z = (rng_state += 0x9e3779b97f4a7c15ull);
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

// One batch: tiles per sequence n[i], Hkv KV heads, P CTAs, segment cost alpha.
static int check_weighted(const std::vector<int32_t>& n, int Hkv, int P, int alpha) {
  const int B = static_cast<int>(n.size());
  std::vector<int32_t> prefix(B + 1, 0);
  for (int i = 0; i < B; ++i) prefix[i + 1] = prefix[i] + n[i];
  const int64_t T = static_cast<int64_t>(Hkv) * prefix[B];
  const int64_t V = tc_vseq(prefix.data(), B, Hkv, alpha);
  auto fail = [&](const char* what, long long a, long long b) {
    std::printf("FAIL %s (%lld, %lld): B=%d Hkv=%d P=%d alpha=%d T=%lld\n", what, a, b, B, Hkv, P,
                alpha, (long long)T);
    return 1;
  };
  // pair of tile x and its unit
  std::vector<int64_t> pair_start, pair_n, pair_u0;
  for (int i = 0; i < B; ++i)
    for (int h = 0; h < Hkv; ++h) {
      pair_start.push_back(static_cast<int64_t>(Hkv) * prefix[i] + static_cast<int64_t>(h) * n[i]);
      pair_n.push_back(n[i]);
      pair_u0.push_back(tc_vseq(prefix.data(), i, Hkv, alpha) +
                        static_cast<int64_t>(h) * (n[i] + alpha) + alpha);
    }
  std::vector<int64_t> lo(P + 1);
  for (int c = 0; c <= P; ++c)
    lo[c] = tc_unit_to_tile(tc_range_lo(c, V, P), prefix.data(), B, Hkv, alpha);
  if (lo[0] != 0 || lo[P] != T) return fail("cover", lo[0], lo[P]);
  for (int c = 0; c < P; ++c)
    if (lo[c + 1] < lo[c]) return fail("order", c, lo[c]);
  // every tile: unit owner == run owner
  std::vector<int> run_owner(static_cast<size_t>(T));
  for (int c = 0; c < P; ++c)
    for (int64_t x = lo[c]; x < lo[c + 1]; ++x) run_owner[x] = c;
  const size_t npairs = pair_start.size();
  for (size_t q = 0; q < npairs; ++q)
    for (int64_t j = 0; j < pair_n[q]; ++j) {
      const int64_t x = pair_start[q] + j;
      if (tc_owner(pair_u0[q] + j, V, P) != run_owner[x]) return fail("unit owner", x, run_owner[x]);
    }
  // the kernel's segment walk: records written per pair, slots per CTA
  std::map<size_t, std::set<std::pair<int, int>>> written;  // pair -> {(cta, slot)}
  std::vector<int> whole_by(npairs, -1);
  size_t q = 0;
  for (int c = 0; c < P; ++c) {
    int64_t x = lo[c];
    int64_t segs = 0;
    bool used[2] = {false, false};
    while (x < lo[c + 1]) {
      while (q < npairs && pair_start[q] + pair_n[q] <= x) ++q;
      const int64_t ps = pair_start[q], pe = ps + pair_n[q];
      const int64_t x1 = pe < lo[c + 1] ? pe : lo[c + 1];
      ++segs;
      if (x == ps && x1 == pe) {
        whole_by[q] = c;
      } else {
        const int slot = x > ps ? 0 : 1;  // the kernel's rule
        if (used[slot]) return fail("slot reused", c, slot);
        used[slot] = true;
        written[q].insert({c, slot});
        // the kernel's view of the piece: its pair's CTAs, and whether it is
        // the head piece (merged by its own CTA)
        const TcSeg seg = tc_find_seg(x, lo[c + 1], prefix.data(), B, Hkv);
        if (seg.x0 != x || seg.x1 != x1 || seg.pstart != ps || seg.pend != pe)
          return fail("segment", c, x);
        int cf = -1, cl = -1;
        tc_pair_ctas(seg, prefix.data(), Hkv, alpha, V, P, &cf, &cl);
        const int ocf = static_cast<int>(tc_owner(pair_u0[q], V, P));
        const int ocl = static_cast<int>(tc_owner(pair_u0[q] + pair_n[q] - 1, V, P));
        if (cf != ocf || cl != ocl || c < cf || c > cl) return fail("pair ctas", c, cf);
        const bool head = cf == c;
        if (head != (slot == 1)) return fail("head piece slot", c, slot);
        if (head && x1 != lo[c + 1]) return fail("head piece not last", c, x1);
      }
      x = x1;
    }
    const int64_t cost = (lo[c + 1] - lo[c]) + alpha * segs;
    const int64_t share = V / P + 1;
    const int64_t longest = alpha + (B ? *std::max_element(n.begin(), n.end()) : 0);
    if (cost > share + 2 * longest + alpha) return fail("cost", c, cost);
  }
  // the merge's lookup of a split pair's records
  for (size_t r = 0; r < npairs; ++r) {
    if (pair_n[r] == 0) continue;
    const int cf = static_cast<int>(tc_owner(pair_u0[r], V, P));
    const int cl = static_cast<int>(tc_owner(pair_u0[r] + pair_n[r] - 1, V, P));
    if (cf == cl) {
      if (whole_by[r] != cf || written.count(r)) return fail("whole pair", (long long)r, cf);
      continue;
    }
    std::set<std::pair<int, int>> looked;
    for (int cc = cf; cc <= cl; ++cc) {
      if (tc_range_lo(cc, V, P) >= tc_range_lo(cc + 1, V, P)) continue;
      looked.insert({cc, cc == cf ? 1 : 0});
    }
    if (looked != written[r]) return fail("records", (long long)r, cf);
  }
  return 0;
}

int main() {
  int bad = 0;
  for (int64_t NW : {1, 7, 148, 152, 160, 1824})
    for (int64_t T : {1, 2, 15, 100, 511, 4096, 32768, 100003, 1048576, 20000017})
      bad |= check_even(T, NW);
  for (int trial = 0; trial < 400 && !bad; ++trial) {
    const int B = 1 + static_cast<int>(rnd() % (trial % 4 == 0 ? 512 : 40));
    const int Hkv = std::vector<int>{1, 2, 4, 8}[rnd() % 4];
    const int P = std::vector<int>{1, 2, 7, 152, 160}[rnd() % 5];
    const int alpha = std::vector<int>{0, 1, 16, 100}[rnd() % 4];
    std::vector<int32_t> n(B);
    for (int i = 0; i < B; ++i) {
      const uint64_t k = rnd() % 10;
      n[i] = k == 0 ? 0 : (k < 4 ? 1 + static_cast<int32_t>(rnd() % 8)
                                 : 1 + static_cast<int32_t>(rnd() % 600));
    }
    bad |= check_weighted(n, Hkv, P, alpha);
  }
  // uniform batches of the benchmark shapes
  bad |= check_weighted(std::vector<int32_t>(64, 64), 8, 152, 16);
  bad |= check_weighted(std::vector<int32_t>(256, 64), 8, 152, 16);
  bad |= check_weighted(std::vector<int32_t>(64, 64), 4, 152, 16);
  std::printf(bad ? "partition check FAILED\n" : "partition check ok\n");
  return bad;
}
