// Host-side check of the launch-time token walk (walk_grid, set_walk and
// TokenWalk from the library's own headers): for every (M, R) asked, each
// token is taken by exactly one cluster, every cluster takes at least one,
// and the grid respects the launch limits.  Built with nvcc and run on the
// CPU by tests/test_walk_host.py; no GPU is touched.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "attnres_launch.cuh"

using namespace attnres;

static int check(int M, unsigned gy, int tail, bool plain) {
  if (gy < 1 || gy > 65535) return 1;
  if (tail < 0 || (tail > 0 && (tail >= static_cast<int>(gy) || static_cast<int>(gy) > M))) return 2;
  Params p = {};
  p.M = M;
  p.tail = tail;
  set_walk(p, gy);
  std::vector<unsigned char> seen(static_cast<size_t>(M), 0);
  for (int c = 0; c < static_cast<int>(gy); ++c) {
    int taken = 0;
    const int m0 = plain ? TokenWalk<true>::first(p, c) : TokenWalk<false>::first(p, c);
    for (int m = m0; m < M;
         m = plain ? TokenWalk<true>::next(p, m, gy) : TokenWalk<false>::next(p, m, gy)) {
      if (m < 0) return 3;
      if (seen[m]++) return 4;   // a token taken twice
      ++taken;
    }
    if (taken == 0 && c < M) return 5;   // an idle cluster although tokens remain
  }
  for (int m = 0; m < M; ++m)
    if (!seen[m]) return 6;             // a token never taken
  return 0;
}

int main(int argc, char** argv) {
  const int Rs[] = {1, 2, 7, 50, 81, 108, 125, 130, 148, 152, 300, 1216, 4864};
  std::vector<int> Ms;
  for (int M = 1; M <= 3000; ++M) Ms.push_back(M);
  for (int M = 3001; M <= 200000; M += 997) Ms.push_back(M);
  const int extra[] = {4096, 8192, 16384, 32768, 65535, 65536, 70000, 131072, 1000000, 4000000};
  for (int M : extra) Ms.push_back(M);
  long cases = 0;
  for (int M : Ms) {
    for (int R : Rs) {
      unsigned gy = 0;
      int tail = 0;
      walk_grid(M, R, &gy, &tail);
      const int e = check(M, gy, tail, false);
      if (e) {
        std::printf("FAIL walk M=%d R=%d grid=%u tail=%d code=%d\n", M, R, gy, tail, e);
        return 1;
      }
      ++cases;
    }
    // the plain walk of the latency shapes: grid min(M, 65535), no tail
    const unsigned g = static_cast<unsigned>(M < 65535 ? M : 65535);
    if (M <= 200000 && check(M, g, 0, true)) {
      std::printf("FAIL plain M=%d\n", M);
      return 1;
    }
  }
  // pinned splits (tail_tokens): every tail below the grid, grids up to M
  for (int M = 1; M <= 300; ++M)
    for (int G = 1; G <= M; G += (G < 20 ? 1 : 7))
      for (int T = 0; T < G; T += (T < 10 ? 1 : 5)) {
        if (check(M, static_cast<unsigned>(G), T, false)) {
          std::printf("FAIL pinned M=%d grid=%d tail=%d\n", M, G, T);
          return 1;
        }
        ++cases;
      }
  std::printf("ok %ld cases\n", cases);
  return 0;
}
