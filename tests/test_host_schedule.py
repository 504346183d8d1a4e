"""Host-side launch schedules, without a GPU.

The streaming kernels read their launch-wide schedule from their arguments: the group (or tile)
count, each CTA's share of it, and the box-counter step of one grid-wide advance.  The library
computes these once on the host (stream_schedule, ring_schedule in csrc/tm_internal.h).  This test
compiles those functions into a small host program and checks them on random shapes against the
per-CTA definitions: CTA b of a grid of G takes groups b, b + G, ..., so it has
(ngroups - 1 - b) // G + 1 of them, and one advance moves G * group boxes, written in the mixed
radix of the grid's box counts (dim 0 fastest)."""
import os
import random
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")

PROGRAM = r"""
#include <cstdio>
#include <cstring>
#include "tm_internal.h"
using namespace tmk;
int main() {
    char kind;
    while (scanf(" %c", &kind) == 1) {
        if (kind == 'S') {
            unsigned long long nbox, nb[5];
            unsigned group, rank, grid;
            scanf("%llu %u %u %llu %llu %llu %llu %llu %u", &nbox, &group, &rank, &nb[0], &nb[1],
                  &nb[2], &nb[3], &nb[4], &grid);
            StreamArgs a;
            memset(&a, 0, sizeof(a));
            a.walk.nbox = nbox;
            a.walk.rank = rank;
            for (int i = 0; i < 5; i++) a.walk.grid_nb[i] = nb[i];
            a.group = group;
            stream_schedule(a, grid);
            printf("%llu %llu %u %u %u %u %u %u\n", (unsigned long long)a.ngroups,
                   (unsigned long long)a.n_base, a.n_rem, a.dstep[0], a.dstep[1], a.dstep[2],
                   a.dstep[3], a.dstep[4]);
        } else {
            unsigned long long ntiles, anb, bnb;
            unsigned grid;
            scanf("%llu %llu %llu %u", &ntiles, &anb, &bnb, &grid);
            RingArgs r;
            memset(&r, 0, sizeof(r));
            r.ntiles = ntiles;
            r.a_nb0 = anb;
            r.b_nb0 = bnb;
            ring_schedule(r, grid);
            printf("%llu %u %u %llu %u %llu\n", (unsigned long long)r.n_base, r.n_rem, r.a_d0,
                   (unsigned long long)r.a_d1, r.b_d0, (unsigned long long)r.b_d1);
        }
    }
    return 0;
}
"""


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None or not os.path.isdir(CUDA_INC):
        pytest.skip("needs g++ and the CUDA headers")
    d = tmp_path_factory.mktemp("sched")
    src, exe = d / "sched.cpp", d / "sched"
    src.write_text(PROGRAM)
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "async_bulk_tensor_tmap_gb300", "csrc"),
                    "-I", CUDA_INC, str(src), "-o", str(exe)], check=True)
    return str(exe)


def run(program, lines):
    r = subprocess.run([program], input="\n".join(lines) + "\n", capture_output=True, text=True,
                       check=True)
    return [list(map(int, ln.split())) for ln in r.stdout.splitlines()]


def digits(value, radix, rank):
    out = []
    for i in range(5):
        if i < rank:
            out.append(value % radix[i])
            value //= radix[i]
        else:
            out.append(0)
    return out


def test_stream_schedule_matches_the_per_cta_definitions(program):
    rng = random.Random(7)
    cases = []
    for _ in range(400):
        rank = rng.randint(1, 5)
        nb = [rng.randint(1, 300) if i < rank else 1 for i in range(5)]
        nbox = 1
        for v in nb:
            nbox *= v
        group = rng.choice([1, 2, 3, 4, 8, 16, 64])
        ngroups = -(-nbox // group)
        grid = rng.randint(1, min(ngroups, 1216))
        cases.append((nbox, group, rank, nb, grid))
    got = run(program, ["S %d %d %d %s %d" % (n, g, r, " ".join(map(str, nb)), gr)
                        for n, g, r, nb, gr in cases])
    for (nbox, group, rank, nb, grid), (ngroups, n_base, n_rem, *dstep) in zip(cases, got):
        assert ngroups == -(-nbox // group)
        for b in range(grid):
            assert n_base + (1 if b < n_rem else 0) == (ngroups - 1 - b) // grid + 1
        assert dstep == digits(grid * group, nb, rank)


def test_ring_schedule_matches_the_per_cta_definitions(program):
    rng = random.Random(11)
    cases = []
    for _ in range(400):
        anb, bnb = rng.randint(1, 200), rng.randint(1, 200)
        ntiles = rng.randint(1, 20000)
        grid = rng.randint(1, min(ntiles, 608))
        cases.append((ntiles, anb, bnb, grid))
    got = run(program, ["R %d %d %d %d" % c for c in cases])
    for (ntiles, anb, bnb, grid), (n_base, n_rem, a_d0, a_d1, b_d0, b_d1) in zip(cases, got):
        for b in range(grid):
            assert n_base + (1 if b < n_rem else 0) == (ntiles - 1 - b) // grid + 1
        assert (a_d0, a_d1, b_d0, b_d1) == (grid % anb, grid // anb, grid % bnb, grid // bnb)
