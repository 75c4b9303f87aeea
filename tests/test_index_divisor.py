"""The kernels find their frame, tile and pixel row by dividing launch
indices by divisors fixed for a launch (the frame count, the frame's width,
its width in tiles) with one multiply-high and a shift; the host computes
the constants (make_index_divisor, hash_blocked_tsdf_gb300/csrc/
tsdf_internal.h, after Granlund and Montgomery, "Division by invariant
integers using multiplication", PLDI 1994).  Here the host code is compiled
on its own and the device's arithmetic, umulhi(2x, m) >> l, is repeated in
64-bit integers against exact division: every divisor up to 1,100 and large
ones up to 2^31 - 1, at indices from 0, around every multiple of the
divisor, random ones and the top of the index range, 2^31 - 1."""
import os
import subprocess

import pytest

from hash_blocked_tsdf_gb300 import _build

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include <random>
#include "tsdf_internal.h"

static uint32_t device_quotient(const tsdf::IndexDivisor& q, uint32_t x)
{
    const uint64_t hi = ((uint64_t)(x << 1) * (uint64_t)q.m) >> 32;   // __umulhi(2x, m)
    return (uint32_t)hi >> q.l;
}

int main()
{
    std::mt19937_64 rng(12345);
    const uint32_t top = 0x7FFFFFFFu;
    unsigned long long checked = 0, bad = 0;
    auto check = [&](const tsdf::IndexDivisor& q, uint32_t x) {
        ++checked;
        if (device_quotient(q, x) != x / q.d) {
            if (bad < 5) std::printf("mismatch d=%u x=%u\n", q.d, x);
            ++bad;
        }
    };
    std::vector<uint32_t> ds;
    for (uint32_t d = 1; d <= 1100; ++d) ds.push_back(d);
    for (uint32_t d : {1280u, 1920u, 3840u, 4096u, 65535u, 65536u, 65537u, 1u << 20,
                       (1u << 20) + 7, 1u << 30, (1u << 30) + 1, top - 1, top})
        ds.push_back(d);
    for (int i = 0; i < 200; ++i) ds.push_back(1 + (uint32_t)(rng() % top));
    for (uint32_t d : ds) {
        const tsdf::IndexDivisor q = tsdf::make_index_divisor(d);
        if (q.d != d || q.l > 31) { std::printf("bad constants d=%u\n", d); return 1; }
        for (uint32_t x = 0; x < 4096; ++x) check(q, x);
        for (uint32_t x = top - 4095; x != 0x80000000u; ++x) check(q, x);
        for (int i = 0; i < 4096; ++i) {
            const uint64_t k = rng() % ((uint64_t)top / d + 1);
            const uint64_t x = k * d;
            for (int64_t off = -1; off <= 1; ++off) {
                const int64_t y = (int64_t)x + off;
                if (y >= 0 && y <= (int64_t)top) check(q, (uint32_t)y);
            }
            if (x + d - 1 <= top) check(q, (uint32_t)(x + d - 1));
            check(q, (uint32_t)(rng() % ((uint64_t)top + 1)));
        }
    }
    std::printf("checked %llu mismatches %llu\n", checked, bad);
    return bad != 0;
}
"""


def test_index_divisor_matches_exact_division(tmp_path):
    src = tmp_path / "divisor_check.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "divisor_check"
    cuda_include = os.path.join(_build.cuda_home(), "include")
    if not os.path.exists(os.path.join(cuda_include, "cuda_runtime.h")):
        pytest.skip("CUDA headers not found")
    subprocess.run(["g++", "-std=c++17", "-O2", "-I", _build.CSRC, "-I", _build.INCLUDE,
                    "-I", cuda_include, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "mismatches 0" in out.stdout
