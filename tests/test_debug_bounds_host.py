"""Host tests of the bounds-checking build (DA_DEBUG_BOUNDS).

The predicate every checked device access goes through, da_index_ok(i, n)
from csrc/da_bounds.h, is plain C++: compiled here with g++ against a table of
boundary cases it must hold for 0 <= i < n and fail for every other i,
including the int64 extremes and negative n. The library's status string for
DA_ERR_DEVICE_BOUNDS is checked on the release build (no GPU call).
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "deformable_view_feature_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include "da_bounds.h"
int main() {
    struct Case { int64_t i, n; bool want; };
    const Case cases[] = {
        {0, 1, true}, {0, 0, false}, {-1, 5, false}, {4, 5, true}, {5, 5, false}, {6, 5, false},
        {INT64_MIN, 5, false}, {INT64_MAX, INT64_MAX, false}, {INT64_MAX - 1, INT64_MAX, true},
        {0, -3, false}, {-3, -3, false}, {2147483647LL, 2147483648LL, true},
        {2147483648LL, 2147483648LL, false}, {-2147483648LL, 2147483648LL, false},
    };
    int bad = 0;
    for (const Case &c : cases)
        if (da::da_index_ok(c.i, c.n) != c.want) {
            std::printf("da_index_ok(%lld, %lld) != %d\n", (long long)c.i, (long long)c.n, (int)c.want);
            ++bad;
        }
    // Brute force over a small square: exactly the pairs with 0 <= i < n.
    for (int64_t n = -4; n <= 8; ++n)
        for (int64_t i = -10; i <= 10; ++i)
            if (da::da_index_ok(i, n) != (i >= 0 && i < n)) ++bad;
    // The bits of the error word are distinct.
    const uint32_t bits[] = {da::kBoundsFeatRow, da::kBoundsOutput, da::kBoundsRecord, da::kBoundsAnchor,
                             da::kBoundsSample, da::kBoundsRowCount, da::kBoundsShared, da::kBoundsPixel};
    uint32_t seen = 0;
    for (uint32_t b : bits) { if (!b || (b & (b - 1)) || (seen & b)) ++bad; seen |= b; }
    std::printf(bad ? "FAIL\n" : "OK\n");
    return bad ? 1 : 0;
}
"""


def test_index_predicate_compiled_on_host(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    src = tmp_path / "bounds_check.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "bounds_check"
    subprocess.run([gxx, "-std=c++17", "-O2", "-Wall", "-Werror", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "OK"


def test_status_string():
    import deformable_view_feature_gb300 as da
    da.build.build()
    lib = da.load_library()
    assert lib.da_status_string(7) == b"DA_ERR_DEVICE_BOUNDS"
