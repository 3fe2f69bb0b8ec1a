// Host check of the InnerQ key-fragment layout of the persistent decode:
// k_offset_of inverts k_slot_of, each thread's key channels split 16 / 16
// between the two 64-channel groups with group 0 in k-steps 0-3, every
// channel is taken by exactly one (thread, k-step, element), and the stage
// swizzle iq_kswz is a chunk-granular bijection whose fragment reads are
// free of shared-memory bank conflicts.  Prints "bad <count>".
#include "../bit_kv_cache_07_gb300/csrc/kvq_decode_mma.cuh"
#include <cstdio>
#include <set>

using namespace kvq::mma;

template <int KB>
int check() {
  int bad = 0;
  std::set<int> seen;
  for (int tq = 0; tq < 4; ++tq)
    for (int o = 0; o < 32; ++o) {
      int s, e;
      k_slot_of<KB>(o, s, e);
      if (k_offset_of<KB>(s, e) != o) ++bad;
      const int c = iq_channel(tq, o);
      if ((c < 64) != (s < 4)) ++bad;  // group 0 in k-steps 0-3
      if ((c & 3) != (o & 3)) ++bad;   // the code's place in its 16-bit half
      seen.insert(c);
    }
  if ((int)seen.size() != 128) ++bad;
  constexpr int KROW = 128 * KB / 8, NB = KROW / 8;
  std::set<unsigned> chunks;
  for (unsigned off = 0; off < 32u * KROW; off += 16) {
    const unsigned m = iq_kswz<KB>(off);
    if (m % 16 || m >= 32u * KROW) ++bad;
    chunks.insert(m);
  }
  if ((int)chunks.size() != 32 * KROW / 16) ++bad;
  // the quad loads of one m-tile row half: lanes (gq, tq), rows gq, both group halves
  for (int half = 0; half < 2; ++half)
    for (int mt = 0; mt < 2; ++mt)
      for (int rr = 0; rr < 2; ++rr) {
        // a phase serves 128 bytes: NB-byte loads of 128 / NB lanes
        const int per_phase = 128 / NB;
        for (int p0 = 0; p0 < 32; p0 += per_phase) {
          std::set<unsigned> banks;
          for (int l = p0; l < p0 + per_phase; ++l) {
            const int gq = l >> 2, tq = l & 3;
            const unsigned r = 16 * mt + 8 * rr + gq;
            const unsigned off = iq_kswz<KB>(r * KROW + half * (KROW / 2) + NB * tq);
            for (unsigned b = 0; b < (unsigned)NB; b += 4) banks.insert(((off + b) / 4) % 32);
          }
          if ((int)banks.size() != per_phase * NB / 4) ++bad;
        }
      }
  return bad;
}

int main() {
  const int bad = check<2>() + check<4>() + check<8>();
  std::printf("bad %d\n", bad);
  return bad ? 1 : 0;
}
