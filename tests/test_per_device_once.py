"""Host-side check of the per-device one-time set-up used by every launcher.

Kernel attributes (a dynamic shared-memory size above the default) and the SM
count belong to one device; the launchers remember them per device so that a
process driving several GPUs sets each one up. The bookkeeping is plain C++
(bit_rotated_kv_oscar_gb300/csrc/per_device_once.h) and is exercised here on the
CPU with made-up device indices: compiled with the host C++ compiler, no CUDA.
"""

import os
import shutil
import subprocess

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bit_rotated_kv_oscar_gb300",
                    "csrc")

PROGRAM = r"""
#include <cstdio>
#include <thread>
#include <vector>
#include "per_device_once.h"

#define CHECK(c) do { if (!(c)) { std::printf("FAIL line %d: %s\n", __LINE__, #c); return 1; } } while (0)

int main() {
  oscar::PerDeviceOnce once;
  int calls[oscar::kMaxDevices] = {};
  auto setup_for = [&](int dev, int result) { return [&calls, dev, result] { ++calls[dev]; return result; }; };
  // first call on device 0 runs the set-up, later ones do not
  CHECK(once.run_on(0, setup_for(0, 0)) == 0);
  CHECK(once.run_on(0, setup_for(0, 0)) == 0);
  CHECK(calls[0] == 1);
  // a second device runs its own set-up although device 0 is done
  CHECK(once.run_on(3, setup_for(3, 0)) == 0);
  CHECK(calls[3] == 1);
  // a failing set-up is reported and retried on the next call
  CHECK(once.run_on(5, setup_for(5, 7)) == 7);
  CHECK(once.run_on(5, setup_for(5, 0)) == 0);
  CHECK(once.run_on(5, setup_for(5, 0)) == 0);
  CHECK(calls[5] == 2);
  // device indices outside the table are refused without running the set-up
  CHECK(once.run_on(-1, setup_for(1, 0)) == -1);
  CHECK(once.run_on(oscar::kMaxDevices, setup_for(1, 0)) == -1);
  CHECK(calls[1] == 0);
  // many host threads on one fresh device: exactly one set-up
  std::vector<std::thread> ts;
  for (int i = 0; i < 16; ++i) ts.emplace_back([&] { once.run_on(9, setup_for(9, 0)); });
  for (auto& t : ts) t.join();
  CHECK(calls[9] == 1);
  // per-device values: computed once per device, device-specific
  oscar::PerDeviceValue v;
  int n = 0;
  CHECK(v.get(0, [&] { ++n; return 152; }) == 152);
  CHECK(v.get(0, [&] { ++n; return 999; }) == 152);
  CHECK(v.get(1, [&] { ++n; return 148; }) == 148);
  CHECK(n == 2);
  std::printf("OK\n");
  return 0;
}
"""


def test_per_device_once_bookkeeping(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "per_device_once_check.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "per_device_once_check"
    r = subprocess.run([cxx, "-std=c++17", "-O1", "-pthread", "-I", CSRC, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout + r.stderr
