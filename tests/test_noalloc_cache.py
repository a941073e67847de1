"""Key logic of the no-alloc entry point's address cache, on the CPU.

The library's fixed scratch array has one instance per CUDA context, so the
cached device address must be keyed on the context's unique id, never on the
device number alone: a device reset or a second context on the same device
gets a new id, misses the cache, and looks the address up again.  The cache is
plain C++ (csrc/noalloc_cache.h); this test compiles a small harness around it
with the host compiler and checks hits, misses, replacement and eviction.  No
GPU is touched.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "content_sparse_attention_shared_b300", "csrc")

HARNESS = r"""
#include <cstdio>
#include "noalloc_cache.h"
using rt::ContextAddressCache;
using rt::NoallocAddrs;
static int fails = 0;
#define CHECK(x) do { if (!(x)) { std::printf("FAIL %s\n", #x); ++fails; } } while (0)
static void* P(unsigned long v) { return reinterpret_cast<void*>(v); }
int main() {
  ContextAddressCache<4> c;
  CHECK(c.find(7) == nullptr);                 // nothing cached yet
  c.put(7, NoallocAddrs{P(0x1000), P(0x2000)});
  CHECK(c.find(7) && c.find(7)->scores == P(0x1000) && c.find(7)->status == P(0x2000));
  // same device, new context (e.g. after a reset): a different id misses
  CHECK(c.find(8) == nullptr);
  c.put(8, NoallocAddrs{P(0x3000), P(0x4000)});
  CHECK(c.find(8)->scores == P(0x3000));
  CHECK(c.find(7)->scores == P(0x1000));       // the old context keeps its own entry
  // replacing an entry keeps one slot per id
  c.put(7, NoallocAddrs{P(0x5000), P(0x6000)});
  CHECK(c.size() == 2 && c.find(7)->scores == P(0x5000));
  // eviction: the oldest entry goes first once full
  c.put(9, NoallocAddrs{P(0x10), P(0x20)});
  c.put(10, NoallocAddrs{P(0x30), P(0x40)});
  c.put(11, NoallocAddrs{P(0x50), P(0x60)});
  CHECK(c.size() == 4);
  CHECK(c.find(7) == nullptr);                 // inserted first, evicted first
  CHECK(c.find(8) && c.find(9) && c.find(10) && c.find(11));
  // id 0 is a valid key, distinct from "empty"
  ContextAddressCache<2> z;
  CHECK(z.find(0) == nullptr);
  z.put(0, NoallocAddrs{P(0x70), P(0x80)});
  CHECK(z.find(0) && z.find(0)->status == P(0x80));
  std::printf(fails ? "FAILED\n" : "OK\n");
  return fails ? 1 : 0;
}
"""


def test_context_keyed_cache(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "harness.cpp"
    exe = tmp_path / "harness"
    src.write_text(HARNESS)
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
    assert res.stdout.strip().endswith("OK")
