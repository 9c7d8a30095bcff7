"""Host-side layout logic of the kernels, compiled for the host and checked on the CPU:
how a fused decode layer cuts a pair's block list into per-CTA slices (CTA 0 free of
attention when its warps take the group top-k), the bound the shared-memory layout is
sized for, where the push merge applies and the tensor-memory tile descriptors."""
import os
import subprocess

import pytest

from block_sparse_long_pool_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_sparse_long_pool_gb300", "csrc")

HARNESS = r"""
#include <cstdio>
#include "select_layout.cuh"

int main()
{
    // every (k_tot, S, group): the slices tile [0, k_tot) in rank order, none longer than
    // fused_slice_max, CTA 0 empty when freed, and the others within one block of each other
    for (int k_tot = 0; k_tot <= 300; ++k_tot)
        for (int S = 1; S <= 16; S *= 2)
            for (int group = 0; group < 2; ++group) {
                const int mx = fused_slice_max(k_tot, S, group != 0);
                int next = 0, lo = 1 << 30, hi = -1;
                for (int r = 0; r < S; ++r) {
                    int i0, cap;
                    fused_slice(k_tot, S, r, group != 0, &i0, &cap);
                    if (cap < 0 || cap > mx || (cap > 0 && i0 != next)) {
                        printf("BAD k_tot=%d S=%d group=%d r=%d i0=%d cap=%d max=%d\n", k_tot, S, group, r, i0, cap, mx);
                        return 1;
                    }
                    if (group && S > 1 && r == 0 && cap != 0) {
                        printf("CTA0 k_tot=%d S=%d\n", k_tot, S);
                        return 1;
                    }
                    if (!(group && S > 1 && r == 0)) {
                        lo = cap < lo ? cap : lo;
                        hi = cap > hi ? cap : hi;
                    }
                    next = i0 + cap > next ? i0 + cap : next;
                }
                if (next != k_tot || (group && S > 1 && hi - lo > 1)) {
                    printf("COVER k_tot=%d S=%d group=%d next=%d lo=%d hi=%d\n", k_tot, S, group, next, lo, hi);
                    return 1;
                }
            }
    // the push merge: 8-row tiles up to 8 CTAs, 16-row tiles up to 4, never beyond 8
    printf("push %d %d %d %d %d\n", (int)merge_pushes<1>(8), (int)merge_pushes<1>(16), (int)merge_pushes<2>(4),
           (int)merge_pushes<2>(8), (int)merge_pushes<1>(1));
    // tensor-core instruction descriptor of kind::f16 (bf16 A/B, f32 D, M x N, majors)
    printf("idesc %08x %08x\n", tc_idesc_bf16(64, 16, 0, 0), tc_idesc_bf16(128, 16, 1, 0));
    return 0;
}
"""


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    d = tmp_path_factory.mktemp("layout")
    src = d / "harness.cu"
    src.write_text(HARNESS)
    exe = d / "harness"
    # the headers' device code is compiled for the library's target; only main() runs
    cmd = [build.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "--expt-relaxed-constexpr",
           "-I", os.path.join(ROOT, "include"), "-I", CSRC, str(src), "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    return out


def test_fused_slices_tile_the_list(harness):
    assert harness.returncode == 0, harness.stdout


def test_push_merge_applies_up_to_eight_ctas(harness):
    line = next(l for l in harness.stdout.splitlines() if l.startswith("push"))
    assert line.split()[1:] == ["1", "0", "1", "0", "0"]


def test_tensor_core_instruction_descriptors(harness):
    # bit 4: f32 accumulator; bits 7 and 10: bf16 A and B; bit 15: A MN-major;
    # bits 17-22: N / 8; bits 24-28: M / 16
    line = next(l for l in harness.stdout.splitlines() if l.startswith("idesc"))
    s_desc, o_desc = (int(x, 16) for x in line.split()[1:])
    assert s_desc == (1 << 4) | (1 << 7) | (1 << 10) | (2 << 17) | (4 << 24)
    assert o_desc == (1 << 4) | (1 << 7) | (1 << 10) | (1 << 15) | (2 << 17) | (8 << 24)
