"""The launch heuristics of the scan (channels per backward CTA, time
segments of the forward and the backward), compiled from the kernels' own
header with the host compiler: the configurations the documentation quotes
for the benchmark workloads."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "selective_state_space_ssm_gb300", "csrc")
CUDA_INC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")

PROGRAM = r'''
#include <cstdio>
#include "scan_args.cuh"
int main() {
    const int shapes[][3] = {{8, 1024, 1536}, {8, 2048, 4096}, {1, 65536, 2048}, {1, 64, 32}};
    for (const auto& s : shapes) {
        const int b = s[0], L = s[1], D = s[2];
        const int cw = ssm::bwd_channels(b, D);
        const int gf = ssm::fwd_segments(b, D, L);
        const int tiles = ssm::fwd_seg_tiles(L, gf);
        const int nt = (L + ssm::kFwdTile - 1) / ssm::kFwdTile;
        const int nseg_f = (nt + tiles - 1) / tiles;
        const int gb = ssm::bwd_segments(b, D, L, cw);
        const int nch = (L + ssm::kChunk - 1) / ssm::kChunk;
        const int sc = (nch + gb - 1) / gb;
        const int nseg_b = (nch + sc - 1) / sc;
        std::printf("%d %d %d %d %d %d\n", b, L, D, cw, nseg_f, nseg_b);
    }
    return 0;
}
'''


@pytest.fixture(scope="module")
def table(tmp_path_factory):
    if not shutil.which("g++") or not os.path.exists(os.path.join(CUDA_INC, "cuda.h")):
        pytest.skip("host compiler or CUDA headers missing")
    d = tmp_path_factory.mktemp("heur")
    src, exe = d / "h.cpp", d / "h"
    src.write_text(PROGRAM)
    subprocess.run(["g++", "-std=c++17", "-I", CSRC, "-I", CUDA_INC, str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    rows = [tuple(int(v) for v in line.split()) for line in out.strip().splitlines()]
    return {r[:3]: r[3:] for r in rows}


def test_benchmark_workload_runs_one_segment_with_32_channel_backward(table):
    # B8 L2048 D4096: 1024 CTAs of 32 channels fill the 152 SMs (>= 6 warps each)
    assert table[(8, 2048, 4096)] == (32, 1, 1)


def test_few_channel_workloads(table):
    # B8 L1024 D1536: 16-channel backward CTAs (twice the warps: 768, 5 per
    # SM) and 2 backward time segments; the forward (384 warps) is not split
    assert table[(8, 1024, 1536)] == (16, 1, 2)
    # B1 L65536 D2048: time segments in both passes (15 forward, 8 backward)
    assert table[(1, 65536, 2048)] == (16, 15, 8)
    # the tiny problem: too short to split
    assert table[(1, 64, 32)] == (16, 1, 1)
