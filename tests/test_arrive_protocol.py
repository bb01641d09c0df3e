"""The split-KV arrival counters (csrc/pa_arrive.h) driven on the CPU: the header is
compiled as plain C++ with counters in host memory and compare-and-swap stand-ins,
including one that always fails so that the give-up path runs (it cannot be forced on
the GPU).  A pair of n pieces must see counts 1..n, whoever arrives; a counter left by
another call (another tag) or never written counts as zero; the completing arrival leaves
the counter at zero, so a replay with the same tag counts from zero again; and an arrival
whose compare-and-swaps keep failing returns -1 after its tries instead of looping."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_cache_149_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "pa_arrive.h"

struct Cas {
  unsigned long long operator()(unsigned long long* a, unsigned long long e, unsigned long long d) const {
    const unsigned long long old = *a;
    if (old == e) *a = d;
    return old;
  }
};
// another arrival slips in before each of the first `left` tries of this one
struct RacyCas {
  int* left;
  unsigned long long operator()(unsigned long long* a, unsigned long long e, unsigned long long d) const {
    if (*left > 0) {
      --*left;
      *a += 1;            // the other arrival's increment (same tag)
      return *a;
    }
    return Cas()(a, e, d);
  }
};
// every try finds the counter changed
struct NeverCas {
  unsigned long long operator()(unsigned long long* a, unsigned long long, unsigned long long) const {
    return ++*a;
  }
};
struct Load {
  unsigned long long operator()(unsigned long long* a) const { return *a; }
};

int main() {
  const unsigned long long tag = 0x123456789aull, other = 0x0fedcba987ull;
  unsigned long long ctr = 0xdeadbeefcafef00dull;             // never written
  // one call: 3 pieces
  for (int i = 0; i < 3; ++i) printf("a %d\n", pa::arrive_count(&ctr, tag, 3, Cas(), Load()));
  printf("after %llx\n", ctr);
  // the same call replayed (same tag)
  for (int i = 0; i < 3; ++i) printf("r %d\n", pa::arrive_count(&ctr, tag, 3, Cas(), Load()));
  // another call, another tag, 2 pieces
  for (int i = 0; i < 2; ++i) printf("o %d\n", pa::arrive_count(&ctr, other, 2, Cas(), Load()));
  printf("after2 %llx\n", ctr);
  // a counter left mid-count by another call: stale, counts as zero
  ctr = (other << 24) | 1;
  printf("s %d\n", pa::arrive_count(&ctr, tag, 4, Cas(), Load()));
  // contention: two other arrivals change the counter between this one's load and CAS
  ctr = tag << 24;
  int left = 2;
  printf("c %d\n", pa::arrive_count(&ctr, tag, 4, RacyCas{&left}, Load()));
  printf("cafter %llx\n", ctr);
  // give up after a bounded number of tries
  ctr = tag << 24;
  printf("g %d\n", pa::arrive_count(&ctr, tag, 2, NeverCas(), Load(), 8));
  printf("gafter %llx\n", ctr);
  return 0;
}
"""


@pytest.fixture(scope="module")
def run_program(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    d = tmp_path_factory.mktemp("arrive")
    src, exe = d / "arrive.cpp", d / "arrive"
    src.write_text(PROGRAM)
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return [line.split() for line in out.strip().splitlines()]


def values(lines, key):
    return [v for k, v in lines if k == key]


def test_counts_run_one_to_n_and_the_last_resets(run_program):
    tag = 0x123456789A
    assert values(run_program, "a") == ["1", "2", "3"]
    assert int(values(run_program, "after")[0], 16) == tag << 24


def test_a_replay_with_the_same_tag_counts_from_zero(run_program):
    assert values(run_program, "r") == ["1", "2", "3"]


def test_another_tag_is_stale(run_program):
    assert values(run_program, "o") == ["1", "2"]
    assert int(values(run_program, "after2")[0], 16) == 0x0FEDCBA987 << 24
    assert values(run_program, "s") == ["1"]


def test_retries_after_other_arrivals(run_program):
    tag = 0x123456789A
    assert values(run_program, "c") == ["3"]           # two others counted in first
    assert int(values(run_program, "cafter")[0], 16) == (tag << 24) | 3


def test_gives_up_after_its_tries(run_program):
    tag = 0x123456789A
    assert values(run_program, "g") == ["-1"]
    assert int(values(run_program, "gafter")[0], 16) == (tag << 24) + 8   # nothing of its own
