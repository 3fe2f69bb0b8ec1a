// Host-side check of the persistent decode's work schedule: every item has
// exactly one owner warp, no warp range is empty under the launch cap, the
// owner formula agrees with the ranges, and the (warp, stream) slots are
// distinct and in bounds -- for batches of one length and for ragged ones
// (rows of different lengths).  Also checks the device's division by a launch
// constant (fastdiv_mulshift: multiply by a rounded-up reciprocal, shift)
// against exact integer division, and the fp32 RoPE group anchors
// (anchor_turns) against the fp64 angle.  Built and run by
// test_schedule_host.py.
#include "../bit_kv_cache_07_gb300/csrc/kvq_internal.cuh"
#include <cmath>
#include <cstdio>
#include <set>
#include <vector>
using namespace kvq;
int main() {
  int bad = 0, cases = 0;
  for (int NS : {1, 2, 7, 32, 256}) for (int ng : {0, 1, 3, 31, 125}) for (int nt : {0, 1, 3, 12}) for (long long wq : {3328LL, 5376LL, 9984LL}) for (long long wt : {4096LL, 16384LL, 0LL}) {
    if (wt == 0) wt = wq;  // every item one group's weight (the quantized cache's schedule)
    if (ng + nt == 0) continue;
    DecodeParams p{}; p.ng = ng; p.nt = nt; p.n_items = ng + nt; p.wq = wq; p.wt = wt;
    p.wstream = ng * wq + nt * p.wt; p.wtot = NS * p.wstream;
    long long items = (long long)NS * p.n_items;
    for (long long nw0 : {1LL, 5LL, 37LL, 1824LL}) {
      long long nw = nw0; if (nw > items) nw = items; if (nw > 64LL * NS) nw = 64LL * NS;
      long long wmax = p.ng > 0 && p.wq > p.wt ? p.wq : p.wt; if (nw > p.wtot / wmax) nw = p.wtot / wmax; if (nw < 1) nw = 1;
      p.nwarps = (int)nw; ++cases;
      std::vector<int> own(items, -1);
      for (int i = 0; i < nw; ++i) {
        long long j0 = first_item_at(p, warp_x(p, i)), j1 = first_item_at(p, warp_x(p, i + 1));
        if (j0 >= j1) { printf("empty range NS=%d ng=%d nt=%d nw=%lld i=%d\n", NS, ng, nt, nw, i); ++bad; }
        for (long long j = j0; j < j1; ++j) { if (own[j] != -1) ++bad; own[j] = i; }
      }
      std::set<long long> slots;
      for (long long j = 0; j < items; ++j) {
        if (own[j] < 0) { printf("unowned item\n"); ++bad; continue; }
        if (owner_of(p, item_pos(p, j)) != own[j]) { printf("owner mismatch\n"); ++bad; }
      }
      for (int s = 0; s < NS; ++s) {
        std::set<int> ws;
        for (int k = 0; k < p.n_items; ++k) ws.insert(own[(long long)s * p.n_items + k]);
        int wf = owner_of(p, item_pos(p, (long long)s * p.n_items)), wl = owner_of(p, item_pos(p, (long long)s * p.n_items + p.n_items - 1));
        const StreamSpan sp = stream_span(p, s);  // positions from the stream's span (the kernel's stream ends)
        for (int k = 0; k < p.n_items; ++k)
          if (item_pos_in(p, sp, k) != item_pos(p, (long long)s * p.n_items + k)) { printf("span position\n"); ++bad; }
        if ((int)ws.size() != wl - wf + 1) { printf("count mismatch s=%d\n", s); ++bad; }
        for (int w : ws) { if (!slots.insert(w + s).second) { printf("slot clash\n"); ++bad; } if (w + s >= nw + NS) ++bad; }
      }
    }
  }
  // ragged batches: rows of different lengths, every row's streams laid end
  // to end with their own item counts; the same properties per stream
  {
    unsigned long long rs = 1234567ull;
    auto rr = [&]() { rs ^= rs << 13; rs ^= rs >> 7; rs ^= rs << 17; return rs; };
    for (int trial = 0; trial < 400; ++trial) {
      DecodeParams p{};
      static RaggedTables tab;
      p.ragged = 1;
      p.row_tokens = tab.tokens;
      p.row_j0 = tab.j0;
      p.row_x0 = tab.x0;
      p.geo.B = 1 + (int)(rr() % 40);
      p.geo.Hkv = 1 + (int)(rr() % 8);
      p.geo.NS = p.geo.B * p.geo.Hkv;
      p.geo.fp16_mode = trial % 7 == 0;
      p.geo.S = p.geo.fp16_mode ? 0 : (int)(rr() % 5);
      p.geo.R = p.geo.fp16_mode ? 0 : (int)(rr() % 70);
      p.wq = (trial & 1) ? 5376 : 9984;
      p.wt = trial % 3 == 1 ? p.wq : 8 * 128 * 4;  // equal item weights, or an fp16 item's bytes
      const int tmax = 1 + (int)(rr() % (trial % 3 == 0 ? 5000 : 300));
      for (int b = 0; b < p.geo.B; ++b) tab.tokens[b] = 1 + (int)(rr() % tmax);
      long long items;
      bool any_groups;
      plan_rows(p, &items, &any_groups);
      const int NS = p.geo.NS;
      long long nw = 1 + (long long)(rr() % 3000);
      if (nw > items) nw = items;
      if (nw > 64LL * NS) nw = 64LL * NS;
      const long long wmax = any_groups && p.wq > p.wt ? p.wq : p.wt;
      if (nw > p.wtot / wmax) nw = p.wtot / wmax;
      if (nw < 1) nw = 1;
      p.nwarps = (int)nw;
      p.fd_nwarps = make_fastdiv(p.nwarps);
      p.fd_wtot = make_fastdiv(p.wtot);
      ++cases;
      if (p.geo.B <= kInlineRows) {
        // the same schedule from inline tables (the pointers aimed at zeros)
        static RaggedTables zero;
        DecodeParams q = p;
        q.rows_inline = 1;
        for (int b = 0; b <= p.geo.B; ++b) {
          if (b < p.geo.B) q.in_tokens[b] = tab.tokens[b];
          q.in_j0[b] = tab.j0[b];
          q.in_x0[b] = tab.x0[b];
        }
        q.row_tokens = zero.tokens;
        q.row_j0 = zero.j0;
        q.row_x0 = zero.x0;
        for (long long i = 0; i <= nw; ++i)
          if (first_item_at(q, warp_x(q, i)) != first_item_at(p, warp_x(p, i))) { printf("inline range\n"); ++bad; }
        for (int s = 0; s < NS; ++s) {
          const StreamSpan a = stream_span(p, s), c = stream_span(q, s);
          if (a.first != c.first || a.x0 != c.x0 || a.n_items != c.n_items || a.ng != c.ng || a.k1 != c.k1) {
            printf("inline span\n");
            ++bad;
          }
        }
        for (long long jj = 0; jj < items; ++jj) {
          int s1, k1, s2, k2;
          locate_item(p, jj, &s1, &k1);
          locate_item(q, jj, &s2, &k2);
          if (s1 != s2 || k1 != k2) { printf("inline locate\n"); ++bad; }
        }
      }
      // items of every stream: their count and positions from the stream's own length
      long long j = 0;
      for (int s = 0; s < NS; ++s) {
        const StreamSpan sp = stream_span(p, s);
        int se, nq, w;
        window_counts(p.geo, p.row_tokens[s / p.geo.Hkv], &se, &nq, &w);
        if (sp.first != j || sp.ng != (p.geo.fp16_mode ? 0 : nq / 32) || sp.nt != (se + w + 7) / 8) {
          printf("ragged span s=%d\n", s);
          ++bad;
        }
        for (int k = 0; k < sp.n_items; ++k, ++j) {
          int s2, k2;
          locate_item(p, j, &s2, &k2);
          if (s2 != s || k2 != k) { printf("ragged locate j=%lld\n", j); ++bad; }
          if (item_pos(p, j) != sp.x0 + (k <= sp.ng ? k * p.wq : sp.ng * p.wq + (k - sp.ng) * p.wt)) ++bad;
          if (item_pos_in(p, sp, k) != item_pos(p, j)) { printf("ragged span position\n"); ++bad; }
        }
      }
      if (j != items) ++bad;
      // the device's warp search: (rows with an entry <= v) - 1 is row_at
      for (int t = 0; t < 64; ++t) {
        const long long vx = (long long)(rr() % (unsigned long long)p.wtot), vj = (long long)(rr() % (unsigned long long)items);
        int cx = 0, cj = 0;
        for (int r = 0; r < p.geo.B; ++r) { cx += p.row_x0[r] <= vx; cj += p.row_j0[r] <= vj; }
        if (cx - 1 != row_at(p.row_x0, p.geo.B, vx) || cj - 1 != row_at(p.row_j0, p.geo.B, vj)) { printf("row count\n"); ++bad; }
      }
      std::vector<int> own(items, -1);
      for (int i = 0; i < nw; ++i) {
        const long long j0 = first_item_at(p, warp_x(p, i)), j1 = first_item_at(p, warp_x(p, i + 1));
        if (j0 >= j1) { printf("ragged empty range trial=%d i=%d\n", trial, i); ++bad; }
        for (long long jj = j0; jj < j1; ++jj) { if (own[jj] != -1) ++bad; own[jj] = i; }
      }
      std::set<long long> slots;
      for (long long jj = 0; jj < items; ++jj) {
        if (own[jj] < 0) { printf("ragged unowned item\n"); ++bad; continue; }
        if (owner_of(p, item_pos(p, jj)) != own[jj]) { printf("ragged owner mismatch\n"); ++bad; }
      }
      for (int s = 0; s < NS; ++s) {
        const StreamSpan sp = stream_span(p, s);
        std::set<int> ws;
        for (int k = 0; k < sp.n_items; ++k) ws.insert(own[sp.first + k]);
        const int wf = owner_of(p, item_pos(p, sp.first)), wl = owner_of(p, item_pos(p, sp.first + sp.n_items - 1));
        if ((int)ws.size() != wl - wf + 1) { printf("ragged count mismatch s=%d\n", s); ++bad; }
        for (int w : ws) { if (!slots.insert(w + s).second) ++bad; if (w + s >= nw + NS) ++bad; }
      }
    }
  }
  // udiv: 32-bit when both operands fit, exact either way
  {
    unsigned long long us = 0x9E3779B97F4A7C15ull;
    auto ur = [&]() { us ^= us << 13; us ^= us >> 7; us ^= us << 17; return us; };
    for (int t = 0; t < 200000; ++t) {
      const int sx = (int)(ur() % 60), sd = (int)(ur() % 40);
      const long long x = (long long)(ur() >> (64 - 1 - sx) >> 1), d = (long long)(ur() >> (64 - 1 - sd) >> 1) + 1;
      if (udiv(x, d) != x / d) { printf("udiv %lld %lld\n", x, d); ++bad; break; }
    }
  }
  // multiply-shift division: exact for 0 <= x < 2^56, any d >= 1
  unsigned long long st = 88172645463325252ull;
  auto rnd = [&]() { st ^= st << 13; st ^= st >> 7; st ^= st << 17; return st; };
  auto check = [&](long long x, long long d) {
    ++cases;
    if (fastdiv_mulshift(x, make_fastdiv(d)) != x / d) {
      if (bad < 10) printf("fastdiv(%lld, %lld) wrong\n", x, d);
      ++bad;
    }
  };
  for (long long d = 1; d <= 300; ++d)  // every small divisor at the ends of the range
    for (long long x : {0LL, 1LL, d - 1, d, d + 1, kFastDivLimit - 1, kFastDivLimit - 1 - (kFastDivLimit - 1) % d,
                        kFastDivLimit - 2 - (kFastDivLimit - 1) % d})
      if (x >= 0) check(x, d);
  for (int e = 0; e < 48; ++e)  // powers of two and their neighbours
    for (long long d : {(1LL << e) - 1, 1LL << e, (1LL << e) + 1})
      if (d >= 1) { check(kFastDivLimit - 1, d); check((kFastDivLimit - 1) / d * d, d); check((kFastDivLimit - 1) / d * d - 1, d); }
  for (int i = 0; i < 2000000; ++i) {
    const long long d = (long long)(rnd() % ((i & 1) ? 5000ull : (1ull << 40))) + 1;
    long long x = (long long)(rnd() % (unsigned long long)kFastDivLimit);
    if (i % 3 == 0) x = (x / d) * d;                      // exact multiples
    if (i % 3 == 1 && (x / d) * d > 0) x = (x / d) * d - 1;  // just below one
    check(x, d);
  }
  // RoPE group anchors in fp32 (anchor_turns) against the fp64 angle
  double worst = 0.0;
  for (double base : {10000.0, 500000.0, 1e6}) for (int S : {0, 4, 128}) {
    DecodeParams p{};
    for (int i = 0; i < kHeadDim / 2; ++i) p.theta[i] = std::pow(base, -2.0 * i / (double)kHeadDim);
    float4 av[kHeadDim / 2];
    float ac[kHeadDim / 2];
    for (int j = 0; j < kHeadDim / 2; ++j) anchor_step(p.theta[j], S, &av[j], &ac[j]);
    for (int j = 0; j < kHeadDim / 2; ++j)
      for (int g : {0, 1, 2, 3, 31, 32, 33, 255, 256, 4095, 4096, 32767, 32768, 65534, 65535})
        for (int dg = 0; dg < 3; ++dg) {
          const int gg = g - dg * 7919 >= 0 ? g - dg * 7919 : g;
          const double exact = (double)(S + 32 * gg) * p.theta[j] / (2.0 * 3.14159265358979323846);
          double d = (double)anchor_turns(av[j], ac[j], gg) - (exact - std::floor(exact));
          d -= std::round(d);  // circular distance in turns
          ++cases;
          if (std::fabs(d) > worst) worst = std::fabs(d);
          if (std::fabs(d) > 1e-6) {
            if (bad < 10) printf("anchor j=%d g=%d S=%d base=%g off by %g turns\n", j, gg, S, base, d);
            ++bad;
          }
        }
  }
  printf("anchor worst %.3g turns\n", worst);
  // split-kernel grid widened to whole waves: the 1M-token NUQ layer's case,
  // then every combination of a small grid of shapes
  {
    int nq = 29, ns = 29;
    const int per = fill_waves_plan(32, 608, 32768, 1130, &nq, &ns);
    ++cases;
    if (nq != 38 || ns != 38 || per != 863) { printf("fill_waves 1M: %d %d %d\n", nq, ns, per); ++bad; }
  }
  for (int NS : {1, 8, 32, 200, 1024}) for (int ngroups : {1, 7, 64, 1000, 32768}) for (int f : {0, 1})
    for (long long resident : {152LL, 456LL, 608LL}) for (int q0 : {1, 5, 29, 64}) {
      if (q0 > ngroups) continue;
      const int gps0 = (ngroups + q0 - 1) / q0;
      int nq = (ngroups + gps0 - 1) / gps0, ns = nq + f;
      const int nq0 = nq;
      const int per = fill_waves_plan(NS, resident, ngroups, gps0, &nq, &ns);
      ++cases;
      // splits never drop, never exceed the cap or the groups, cover every group exactly once,
      // and a widened grid is no larger than the whole waves the old one started
      const long long waves = ((long long)NS * (nq0 + f) + resident - 1) / resident;
      if (nq < nq0 || nq > kMaxQSplits || nq > ngroups || ns != nq + f || (long long)per * nq < ngroups ||
          (long long)per * (nq - 1) >= ngroups || (nq > nq0 && (long long)NS * ns > waves * resident)) {
        printf("fill_waves NS=%d ngroups=%d f=%d res=%lld q0=%d -> %d\n", NS, ngroups, f, resident, q0, nq);
        ++bad;
      }
    }
  printf("cases %d bad %d\n", cases, bad);
  return bad != 0;
}
