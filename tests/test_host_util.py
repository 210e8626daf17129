"""The launchers' one-time, per-device setup helper (csrc/host_util.h),
compiled on the host with g++ and driven with fake devices."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_decode_attention_fp8_gb300", "csrc")

PROGRAM = r"""
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>
#include "host_util.h"
using fp8mla::once_per_device;

int main() {
  std::atomic<uint64_t> done{0};
  int runs = 0;
  auto ok = [&] { ++runs; return 0; };
  if (once_per_device(done, 0, ok) != 0 || runs != 1) return 1;   // first call on device 0 runs
  if (once_per_device(done, 0, ok) != 0 || runs != 1) return 2;   // ... and only once
  if (once_per_device(done, 3, ok) != 0 || runs != 2) return 3;   // device 3 has its own bit
  if (once_per_device(done, 64, ok) != 0 || runs != 3) return 4;  // beyond the mask: every call
  if (once_per_device(done, 64, ok) != 0 || runs != 4) return 5;
  std::atomic<uint64_t> done2{0};
  int tries = 0;
  auto flaky = [&] { return ++tries == 1 ? 7 : 0; };              // fails once, then succeeds
  if (once_per_device(done2, 1, flaky) != 7) return 6;            // the failure is returned
  if (once_per_device(done2, 1, flaky) != 0 || tries != 2) return 7;  // and retried
  if (once_per_device(done2, 1, flaky) != 0 || tries != 2) return 8;
  // concurrent first calls: every caller succeeds, the bit ends set, setup ran at least once
  std::atomic<uint64_t> done3{0};
  std::atomic<int> n{0};
  std::vector<std::thread> ts;
  std::atomic<int> bad{0};
  for (int i = 0; i < 8; ++i)
    ts.emplace_back([&] { if (once_per_device(done3, 5, [&] { n.fetch_add(1); return 0; }) != 0) bad.fetch_add(1); });
  for (auto& t : ts) t.join();
  if (bad.load() != 0 || n.load() < 1 || (done3.load() & (1ull << 5)) == 0) return 9;
  std::puts("host util ok");
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="no C++ compiler")
def test_once_per_device(tmp_path):
    src = tmp_path / "t.cpp"
    exe = tmp_path / "t"
    src.write_text(PROGRAM)
    r = subprocess.run(["g++", "-std=c++17", "-O1", "-Wall", "-Werror", "-pthread", "-I", CSRC, str(src), "-o",
                        str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.returncode
    assert r.stdout.strip() == "host util ok"
