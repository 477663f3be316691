"""Host-side checks of the persistent attention kernels' work-item schedule
(item_index, item_kv_tiles, choose_group_sets in csrc/q3a_internal.h).

The schedule decides which (b, kv) group and query-tile pair every work item
is; if item_index were not a bijection some query rows would be computed twice
and others never. The functions are host/device inline code, so a small C++
driver compiled with g++ against the same header exercises exactly what the
kernels and launchers run, without a GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "qwen3_qk_norm_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

DRIVER = r"""
#include <cstdio>
#include <cstdlib>
#include <vector>
#include "q3a_internal.h"
using namespace q3a;

static int fails = 0;
#define CHECK(c, ...) do { if (!(c)) { ++fails; std::printf("FAIL " __VA_ARGS__); std::printf("\n"); } } while (0)

// the causal definition: the item's last token sits at position p0 + t_last and
// sees keys 0 .. p0 + t_last, i.e. every tile holding one of them
static int tiles_brute(int t0, int tok, int T, int p0, int keys) {
  int t_last = -1;
  for (int t = t0; t < t0 + tok && t < T; ++t) t_last = t;
  int n = 0;
  for (int k0 = 0; k0 <= p0 + t_last; k0 += keys) ++n;
  return n;
}

int main() {
  // 1. item_index is a bijection for every set count dividing the group count
  const int shapes[][2] = {{16, 32}, {64, 32}, {4, 8}, {3, 6}, {1, 1}, {32, 8}, {7, 12}, {128, 16}};
  for (auto& sh : shapes) {
    const int n_mt = sh[0], bk = sh[1];
    for (int sets = 1; sets <= 8; sets *= 2) {
      if (bk % sets) continue;
      std::vector<int> seen(n_mt * bk, 0);
      for (int i = 0; i < n_mt * bk; ++i) {
        const ItemIndex ix = item_index(i, n_mt, bk / sets);
        CHECK(ix.bk >= 0 && ix.bk < bk && ix.mt >= 0 && ix.mt < n_mt, "range %d %d", n_mt, bk);
        if (ix.bk >= 0 && ix.bk < bk && ix.mt >= 0 && ix.mt < n_mt) seen[ix.mt * bk + ix.bk]++;
        if (sets == 1) {
          // one set: plain longest first over all groups
          CHECK(ix.bk == i % bk && ix.mt == n_mt - 1 - i / bk, "one set order i=%d", i);
        }
        // within a set, m-tiles never increase (longest first)
        if (i > 0 && (i % ((bk / sets) * n_mt)) != 0) {
          const ItemIndex pv = item_index(i - 1, n_mt, bk / sets);
          CHECK(pv.mt >= ix.mt, "longest first within a set i=%d", i);
        }
        // the set count as a shift of the group count equals the division
        CHECK((bk >> __builtin_ctz(sets)) == bk / sets, "shift %d %d", bk, sets);
      }
      for (int v : seen) CHECK(v == 1, "bijection n_mt=%d bk=%d sets=%d", n_mt, bk, sets);
    }
  }
  // 2. item_kv_tiles against the definition
  for (int T : {1, 5, 64, 127, 128, 129, 300, 1024})
    for (int tok : {8, 32, 64, 256})
      for (int p0 : {0, 1, 127, 128, 3072})
        for (int t0 = 0; t0 < T; t0 += tok)
          CHECK(item_kv_tiles(t0, tok, T, p0, 128) == tiles_brute(t0, tok, T, p0, 128),
                "tiles T=%d tok=%d p0=%d t0=%d", T, tok, p0, t0);
  // 3. the replay's choices on the benchmarked shapes, and its invariants
  const int p_chunk[4] = {3072, 3072, 3072, 3072};
  // Qwen3-8B chunk: 16 m-tiles x 32 groups on 152 CTAs -> two sets
  CHECK(choose_group_sets(16, 4, 8, 64, 1024, p_chunk, 128, 152) == 2, "8B chunk");
  // the same prompt filled from position 0, and the plain 8B prefill -> one set
  CHECK(choose_group_sets(48, 4, 8, 64, 3072, nullptr, 128, 152) == 1, "8B fill");
  CHECK(choose_group_sets(64, 4, 8, 64, 4096, nullptr, 128, 152) == 1, "8B prefill");
  // gated chunk: 32 pair tiles x 8 groups on 76 pairs -> two sets
  CHECK(choose_group_sets(32, 4, 2, 32, 1024, p_chunk, 128, 76) == 2, "gated chunk");
  for (int B : {1, 2, 3, 4})
    for (int Hkv : {1, 2, 3, 4, 8})
      for (int n_mt : {1, 5, 16, 40})
        for (int workers : {1, 7, 76, 152}) {
          const int s = choose_group_sets(n_mt, B, Hkv, 64, n_mt * 64, nullptr, 128, workers);
          CHECK(s == 1 || s == 2 || s == 4 || s == 8, "power of two");
          CHECK((B * Hkv) % s == 0, "divides the group count");
        }
  // beyond the replay limit: one set
  CHECK(choose_group_sets(1 << 14, 4, 8, 64, 1 << 20, nullptr, 128, 152) == 1, "replay limit");
  std::printf("%s %d\n", fails ? "FAILED" : "OK", fails);
  return fails ? 1 : 0;
}
"""


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None or not os.path.isdir(CUDA_INC):
        pytest.skip("g++ or the CUDA headers are not available")
    d = tmp_path_factory.mktemp("schedule")
    src = d / "schedule_check.cpp"
    src.write_text(DRIVER)
    exe = d / "schedule_check"
    subprocess.run([gxx, "-std=c++17", "-O1", "-Wall", "-I", CSRC, "-I", CUDA_INC, str(src),
                    "-o", str(exe)], check=True)
    return str(exe)


def test_schedule_is_a_bijection_and_the_replay_choices_hold(driver):
    r = subprocess.run([driver], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip().startswith("OK"), r.stdout + r.stderr
