"""Host-side launch schedules, without a GPU.

The streaming kernels read their launch-wide schedule from their arguments: the full waves, the
tail split, and the box-counter step of one grid-wide advance.  The library computes these once on
the host (stream_schedule, ring_schedule in csrc/tm_internal.h), and the streaming kernel finds each
item's boxes with stream_item, which compiles for the host as well.  This test builds those
functions into a small host program and checks them on random shapes against the per-CTA
definitions: with grid CTAs and G boxes per stage, CTA c takes boxes (j * grid + c) * G .. + G - 1
of each full wave j, then q + (c < r) consecutive boxes of the R boxes left over (q = R // grid,
r = R % grid); one advance moves grid * G boxes, written in the mixed radix of the grid's box
counts (dim 0 fastest).  The program also checks that the items cover every box exactly once."""
import os
import random
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")

PROGRAM = r"""
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <vector>
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
            printf("%llu %llu %u %u %u %u %u %u %u\n", (unsigned long long)a.waves,
                   (unsigned long long)a.tail0, a.tail_q, a.tail_r, a.dstep[0], a.dstep[1],
                   a.dstep[2], a.dstep[3], a.dstep[4]);
            // every CTA's items: count, boxes, first and last box; coverage of [0, nbox)
            std::vector<unsigned char> seen(nbox, 0);
            bool ok = true;
            for (unsigned c = 0; c < grid; c++) {
                const unsigned long long n = stream_items(a, c);
                unsigned long long boxes = 0, first = 0, last = 0;
                for (unsigned long long i = 0; i < n; i++) {
                    uint64_t b0;
                    uint32_t cnt;
                    stream_item(a, c, grid, i, b0, cnt);
                    if (cnt < 1 || cnt > group || b0 + cnt > nbox) { ok = false; break; }
                    for (uint32_t j = 0; j < cnt; j++) ok = ok && seen[b0 + j]++ == 0;
                    if (i == 0) first = b0;
                    last = b0 + cnt - 1;
                    boxes += cnt;
                }
                printf("%llu %llu %llu %llu\n", n, boxes, first, last);
            }
            for (unsigned long long b = 0; b < nbox; b++) ok = ok && seen[b] == 1;
            printf("%d\n", ok ? 1 : 0);
        } else if (kind == 'D') {
            // the dynamic split's items: every CTA's static prefix, then fetches p = 0, 1, ...
            // until one starts past the items; prints whether every item is taken exactly once
            unsigned long long nitems, batch, taper;
            unsigned stages, grid;
            scanf("%llu %u %u %llu %llu", &nitems, &stages, &grid, &batch, &taper);
            StreamArgs a;
            memset(&a, 0, sizeof(a));
            a.nitems = nitems;
            a.stages = stages;
            a.batch = (uint32_t)batch;
            dyn_taper(a, grid, taper);
            std::vector<unsigned char> seen(nitems, 0);
            bool ok = true;
            const uint64_t prefix = (uint64_t)(stages + 1) * grid;
            for (unsigned c = 0; c < grid; c++)
                for (uint64_t dj = 0; dj <= stages; dj++) {
                    const uint64_t g = c + dj * grid;
                    if (g < nitems) ok = ok && seen[g]++ == 0;
                }
            unsigned long long fetches = 0, singles = 0;
            for (uint64_t p = 0;; p++) {
                uint64_t first, count;
                dyn_fetch(a, prefix, p, first, count);
                if (first >= nitems) break;
                fetches++;
                if (count == 1 && batch > 1) singles++;
                for (uint64_t g = first; g < first + count && g < nitems; g++) ok = ok && seen[g]++ == 0;
            }
            for (uint64_t g = 0; g < nitems; g++) ok = ok && seen[g] == 1;
            printf("%d %llu %llu %llu\n", ok ? 1 : 0, (unsigned long long)a.batched, fetches, singles);
        } else if (kind == 'P') {
            // stream_plan under GB300's shared-memory limits (228 KiB per SM, 227 KiB per CTA;
            // 1 KiB per CTA reserved, 1 KiB of stage alignment and 256 B of barriers kept back)
            unsigned long long nbox, box_bytes;
            unsigned span, reduce;
            scanf("%llu %llu %u %u", &nbox, &box_bytes, &span, &reduce);
            auto budget = [](uint32_t per_sm) -> size_t {
                const size_t share = 233472 / per_sm;
                const size_t cap = std::min<size_t>(232448, share > 1024 ? share - 1024 : 0);
                return cap > 2048 + 256 ? cap - 1024 - 256 : 0;
            };
            StreamArgs a;
            memset(&a, 0, sizeof(a));
            a.walk.nbox = nbox;
            a.walk.rank = 1;
            a.walk.grid_nb[0] = nbox;
            uint32_t grid = 0;
            size_t smem = 0;
            stream_plan(a, box_bytes, span, 152, budget, grid, smem, reduce != 0);
            printf("%u %u %u %u %u %zu %d\n", a.group, a.slot_bytes, a.stage_bytes, a.stages, grid,
                   smem, stream_small(a) ? 1 : 0);
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
    env = {k: v for k, v in os.environ.items() if not k.startswith("TM_")}  # the defaults
    r = subprocess.run([program], input="\n".join(lines) + "\n", capture_output=True, text=True,
                       check=True, env=env)
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


def expected_items(nbox, group, grid, c):
    """CTA c's items by the definition: (first box, box count) of each."""
    wave = grid * group
    waves = nbox // wave
    items = [((j * grid + c) * group, group) for j in range(waves)]
    rest = nbox - waves * wave
    q, r = divmod(rest, grid)
    cnt = q + (1 if c < r else 0)
    if cnt:
        items.append((waves * wave + c * q + min(c, r), cnt))
    return items


def test_stream_schedule_matches_the_per_cta_definitions(program):
    rng = random.Random(7)
    cases = []
    for _ in range(300):
        rank = rng.randint(1, 5)
        nb = [rng.randint(1, 40) if i < rank else 1 for i in range(5)]
        nbox = 1
        for v in nb:
            nbox *= v
        if nbox > 60000:
            continue
        group = rng.choice([1, 2, 3, 4, 8, 16, 64])
        ngroups = -(-nbox // group)
        grid = rng.randint(1, min(ngroups, 1216))
        cases.append((nbox, group, rank, nb, grid))
    # the bench's shapes: W3 (8192 boxes of 16 KiB, 2 a stage), W4 rank-3 (16384 and 32768 boxes,
    # 4 and 8 a stage), W5a (65536 boxes, 2 a stage) over 152 CTAs (one per SM) and 304; W3 through
    # 64 x 4 boxes (262144 boxes, 16 a stage) over 608 (four per SM)
    for grid in (152, 304):
        cases += [(8192, 2, 2, [128, 64, 1, 1, 1], grid), (16384, 4, 3, [16, 64, 16, 1, 1], grid),
                  (32768, 8, 3, [32, 64, 16, 1, 1], grid), (65536, 2, 2, [128, 512, 1, 1, 1], grid)]
    cases.append((262144, 16, 2, [128, 2048, 1, 1, 1], 608))
    got = run(program, ["S %d %d %d %s %d" % (n, g, r, " ".join(map(str, nb)), gr)
                        for n, g, r, nb, gr in cases])
    pos = 0
    for nbox, group, rank, nb, grid in cases:
        waves, tail0, q, r, *dstep = got[pos]
        per_cta = got[pos + 1:pos + 1 + grid]
        ok = got[pos + 1 + grid][0]
        pos += grid + 2
        assert ok == 1, (nbox, group, grid)
        assert (waves, tail0) == (nbox // (grid * group), nbox // (grid * group) * grid * group)
        assert (q, r) == divmod(nbox - tail0, grid)
        assert dstep == digits(grid * group, nb, rank)
        counts = []
        for c, (n, boxes, first, last) in enumerate(per_cta):
            want = expected_items(nbox, group, grid, c)
            assert n == len(want)
            assert boxes == sum(k for _, k in want)
            if want:
                assert (first, last) == (want[0][0], want[-1][0] + want[-1][1] - 1)
            counts.append(boxes)
        assert sum(counts) == nbox
        assert max(counts) - min(counts) <= 1  # no CTA has more than one box above another


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


def expected_plan(nbox, box_bytes, span, reduce):
    """The streaming launch shape by its stated rules: image slots rounded up to the swizzle
    period (1024 / 512 / 256 B, 128 B without); slots of at most 1 KiB take 16 KiB stages and 4 CTAs
    per SM, others 32 KiB stages and one CTA; as many stages as fit (reductions at most 4)."""
    period = {128: 1024, 64: 512, 32: 256}.get(span, 128)
    sl = -(-box_bytes // period) * period
    small = sl <= 1024
    group = min(max((16384 if small else 32768) // sl, 1), 64)
    slot = sl if group > 1 else box_bytes
    stage = -(-(group * slot) // 1024) * 1024

    def budget(per_sm):
        share = 233472 // per_sm
        cap = min(232448, share - 1024 if share > 1024 else 0)
        return cap - 1280 if cap > 2048 + 256 else 0

    per_sm = 4 if small else 1
    while per_sm > 1 and budget(per_sm) < 2 * stage:
        per_sm -= 1
    stages = min(budget(per_sm) // stage, 16, 4 if reduce else 16)
    grid = min(-(-nbox // group), 152 * per_sm)
    return [group, slot, stage, max(stages, 1), grid, max(stages, 1) * stage + 1024,
            1 if (group > 1 and slot <= 1024) else 0]


def test_stream_plan_launch_shapes(program):
    cases = [(8192, 16384, 128, 0),     # W3: 128 x 64 bf16 boxes, 128B swizzle
             (65536, 16384, 128, 1),    # W5a reduce-add: 128 x 32 fp32 boxes
             (262144, 512, 128, 0),     # W3 through 64 x 4 boxes: 512-byte images, 1 KiB slots
             (32768, 4096, 64, 0),      # W4 rank-3, 64B swizzle: 4 KiB boxes
             (16384, 8192, 128, 0),     # W4 rank-3, 128B swizzle: 8 KiB boxes
             (100, 256, 0, 0), (5000, 96, 32, 1), (7, 65536, 128, 0), (3, 200000, 0, 0),
             (999, 1024, 128, 0), (999, 1040, 128, 0)]
    got = run(program, ["P %d %d %d %d" % c for c in cases])
    for c, g in zip(cases, got):
        assert g == expected_plan(*c), (c, g)
    # the bench's shapes, spelled out
    assert got[0][:5] == [2, 16384, 32768, 7, 152] and got[0][6] == 0
    assert got[1][3] == 4                                  # reductions: four stages
    assert got[2][:5] == [16, 1024, 16384, 3, 608] and got[2][6] == 1
    assert got[3][:5] == [8, 4096, 32768, 7, 152] and got[3][6] == 0


def test_dynamic_split_takes_every_item_once(program):
    """The dynamic split's item map (csrc/tm_internal.h dyn_fetch, dyn_taper), which the streaming
    kernel follows: every CTA's static prefix of stages + 1 items, then the counter's fetches, whole
    batches until about taper x grid items are left and single items after, cover every item of
    the launch exactly once, on random launches and the bench's shapes."""
    rng = random.Random(13)
    cases = [(4096, 7, 152, 1, 4), (32768, 4, 152, 4, 4), (16384, 7, 152, 1, 4), (16384, 3, 608, 1, 4),
             (100, 7, 152, 4, 4), (1, 1, 1, 4, 4), (1065, 7, 152, 4, 0), (5000, 4, 152, 4, 100)]
    for _ in range(300):
        cases.append((rng.randint(1, 50000), rng.randint(1, 16), rng.randint(1, 700),
                      rng.choice([1, 2, 4, 8, 16]), rng.choice([0, 1, 2, 4, 8])))
    got = run(program, ["D %d %d %d %d %d" % c for c in cases])
    for (nitems, stages, grid, batch, taper), (ok, batched, fetches, singles) in zip(cases, got):
        assert ok == 1, (nitems, stages, grid, batch, taper)
        rest = max(nitems - (stages + 1) * grid, 0)
        if batch > 1:
            assert batched == (rest - min(rest, grid * taper)) // batch
            assert singles == rest - batched * batch  # the items after the batches go out singly
        else:
            assert batched == 0 and fetches == rest
