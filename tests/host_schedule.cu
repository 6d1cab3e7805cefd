// Host-side checks of the prefill kernel's schedule and layout helpers
// (compiled by tests/test_host_schedule.py; nothing here runs on a GPU):
// the split schedule's pieces, the K order of S' in TMEM, and the shared
// memory and stage counts of every kernel shape.
#include <cstdio>
#include <vector>

#include "../state_space_sequence_06_b300/csrc/chunked.cuh"

static int failures = 0;
#define CHECK(cond, ...)            \
  do {                              \
    if (!(cond)) {                  \
      std::printf("FAIL: " __VA_ARGS__); \
      std::printf("\n");            \
      ++failures;                   \
    }                               \
  } while (0)

// Every chunk of every unit in exactly one piece; at most two pieces a
// range, the first of two ending its unit and the second starting the next.
static void check_split(int units, int64_t nch, int grid) {
  const int64_t total = (int64_t)units * nch;
  std::vector<int> seen((size_t)total, 0);
  for (int k = 0; k < grid; ++k) {
    int3 pc[2];
    const int n = m3::split_pieces(nch, total, grid, k, pc);
    const int64_t lo = (int64_t)k * total / grid, hi = (int64_t)(k + 1) * total / grid;
    CHECK(n >= (hi > lo ? 1 : 0) && n <= 2, "units %d nch %lld grid %d range %d: %d pieces", units, (long long)nch,
          grid, k, n);
    int64_t covered = 0;
    for (int i = 0; i < n; ++i) {
      CHECK(pc[i].x >= 0 && pc[i].x < units && pc[i].y >= 0 && pc[i].y < pc[i].z && pc[i].z <= nch,
            "range %d piece %d out of bounds", k, i);
      for (int c = pc[i].y; c < pc[i].z; ++c) ++seen[(size_t)(pc[i].x * nch + c)];
      covered += pc[i].z - pc[i].y;
    }
    CHECK(covered == hi - lo, "range %d covers %lld of %lld chunks", k, (long long)covered, (long long)(hi - lo));
    if (n == 2)
      CHECK(pc[0].z == nch && pc[1].y == 0 && pc[1].x == pc[0].x + 1, "range %d: pieces not at a unit boundary",
            k);
  }
  for (int64_t i = 0; i < total; ++i) CHECK(seen[(size_t)i] == 1, "chunk %lld covered %d times", (long long)i,
                                            seen[(size_t)i]);
}

// kperm is a permutation inside each block of 16 and matches the word
// placement of S -> S' (columns 8 g + 2 m + e at K position 4 m + 2 g + e).
static void check_kperm() {
  std::vector<int> hits(64, 0);
  for (int j = 0; j < 64; ++j) {
    const int kp = m3::kperm(j);
    CHECK(kp >= 0 && kp < 64 && kp / 16 == j / 16, "kperm(%d) = %d leaves its block", j, kp);
    if (kp >= 0 && kp < 64) ++hits[kp];
    const int l = j % 16, g = l / 8, m = (l % 8) / 2, e = l % 2;
    CHECK(kp % 16 == 4 * m + 2 * g + e, "kperm(%d) = %d, S -> S' puts it at %d", j, kp, 4 * m + 2 * g + e);
  }
  for (int i = 0; i < 64; ++i) CHECK(hits[i] == 1, "kperm hits %d %d times", i, hits[i]);
}

template <int N, int R, int Q, bool RE = false>
static void check_cfg(int want_nsf) {
  using C = m3::ChunkCfg<N, R, Q, RE>;
  CHECK(C::SMEM + C::STATIC_EST <= 232448, "N%d R%d: %d bytes of shared memory", N, R, C::SMEM + C::STATIC_EST);
  CHECK(C::NSF == want_nsf, "N%d R%d: %d full-pass stages, expected %d", N, R, C::NSF, want_nsf);
  CHECK(C::OFF_XB == C::NSF * C::STAGE && C::OFF_RT == C::OFF_XB + C::XB * C::XT_BYTES,
        "N%d R%d: X slots or R overlap the stages", N, R);
  // the state-only pass's three C-less stages fit in the CTA's shared memory
  // (that pass uses no X slots and no R, which follow the full pass's stages)
  CHECK(3 * C::SO_STRIDE <= C::SMEM - 1024, "N%d R%d: state-only stages overflow", N, R);
  CHECK(C::NT <= 1024 && C::NT % 32 == 0, "N%d R%d: %d threads", N, R, C::NT);
}

int main() {
  // the long workload's shape (32 units of 256 chunks on 148 SMs) and
  // ragged cases around it
  check_split(32, 256, 148);
  for (int units = 1; units <= 40; units += 3)
    for (int64_t nch = 4; nch <= 70; nch += 11)
      for (int grid = units + 1; grid <= 160 && (int64_t)units * nch / grid >= 4; grid += 7) check_split(units, nch, grid);
  check_kperm();
  check_cfg<128, 1, 64>(2);
  check_cfg<64, 1, 64>(3);
  check_cfg<128, 2, 32>(2);
  check_cfg<64, 2, 32>(2);
  check_cfg<64, 4, 16>(2);
  check_cfg<64, 8, 8>(2);
  check_cfg<128, 1, 64, true>(2);
  check_cfg<64, 4, 16, true>(2);
  std::printf("%s: %d failures\n", failures ? "FAILED" : "ok", failures);
  return failures ? 1 : 0;
}
