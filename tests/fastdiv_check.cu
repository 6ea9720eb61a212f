// Host-side check of mp3d::FastDiv against integer division (run by tests/test_fastdiv.py).
#include "common.cuh"
#include <cstdio>
#include <random>
int main() {
  std::mt19937_64 rng(1);
  long bad = 0;
  for (uint32_t d = 1; d < 5000; ++d) {
    mp3d::FastDiv f(d);
    for (int k = 0; k < 2000; ++k) {
      int n = (int)(rng() & 0x7FFFFFFF);
      if (k < 50) n = k; if (k >= 50 && k < 100) n = 0x7FFFFFFF - (k - 50);
      if (f.div(n) != n / (int)d) { if (bad < 5) printf("bad d=%u n=%d\n", d, n); ++bad; }
    }
  }
  for (uint32_t d : {65537u, 1u<<20, 12544u, 200704u, 2147483647u, 1073741824u, 3000017u}) {
    mp3d::FastDiv f(d);
    for (int k = 0; k < 200000; ++k) { int n = (int)(rng() & 0x7FFFFFFF); if (f.div(n) != n / (int)d) ++bad; }
  }
  printf("bad=%ld\n", bad); return bad != 0;
}
