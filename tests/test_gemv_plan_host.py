"""The small-M GEMV's work planner, on the host (no GPU): which split each decode shape gets on a
152-SM GB300, and that every plan leaves the copy-warp ring the slots its compute warps need.

The planner chooses between whole row blocks per CTA (one launch) and the stream-K split (a second
pass that sums each row's partial sums in k order); both give the same bits, so the choice is a
matter of speed, measured on the GPU.  This test compiles the planner's own translation unit, links
it with stand-ins for the kernel launchers and runs it as a host program.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FMT = {"INT4_SYM": 0, "INT4_ASYM": 1, "INT8_SYM": 2, "INT2_ASYM": 3, "NF4": 4, "K4": 5}
MMA_X_GLOBAL, MMA_X_WHOLE, MMA_X_ROW1 = 0, 1, 2
PW = 6                                          # pairs of compute warps in the copy-warp kernel


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    exe = str(tmp_path_factory.mktemp("plan") / "probe")
    r = subprocess.run([nvcc, "-std=c++17", "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
                        "-gencode", "arch=compute_103a,code=sm_103a", "-o", exe,
                        os.path.join(ROOT, "tests", "gemv_plan_probe.cu"),
                        os.path.join(ROOT, "tests", "gemv_plan_stubs.cu")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]

    def run(fmt, M, N, K, group, a8=False, gated=False):
        out = subprocess.run([exe, str(FMT[fmt]), str(M), str(N), str(K), str(group), str(int(a8)), str(int(gated))],
                             capture_output=True, text=True, check=True).stdout.split()
        grid, cta_rows, launches, warp, slots, xmode, pairs = map(int, out)
        return dict(grid=grid, cta_rows=cta_rows, launches=launches, warp=bool(warp), slots=slots, xmode=xmode,
                    pairs=pairs)
    return run


def test_one_row_int4_shapes_of_the_8b_step(probe):
    # the per-warp kernel: whole row blocks for every linear of the step, the down projection
    # included (4 tiles a warp against 3 under the split, and no second pass)
    for N, K in [(14336, 4096), (4096, 4096), (1024, 4096), (4096, 14336)]:
        p = probe("INT4_ASYM", 1, N, K, 128)
        assert p["warp"] and p["cta_rows"] == 1 and p["launches"] == 1, (N, K, p)
    # a short, tall shape keeps the split: one row block of 14 tiles would give a warp 4 tiles
    # against 1
    p = probe("INT4_ASYM", 1, 1024, 14336, 128)
    assert p["warp"] and p["cta_rows"] == 0 and p["launches"] == 2


def test_copy_warp_splits(probe):
    # 2 rows of x: the down projection's CTAs own whole row blocks (2 pairs of tiles more than the
    # split, x still in shared memory beside the ring)
    p = probe("INT4_ASYM", 2, 4096, 14336, 128)
    assert p["cta_rows"] == 28 and p["launches"] == 1 and p["xmode"] == MMA_X_WHOLE
    # 8 rows: all of x would not fit beside the ring, so the split and its window of x
    p = probe("INT4_ASYM", 8, 4096, 14336, 128)
    assert p["cta_rows"] == 0 and p["launches"] == 2 and p["xmode"] == MMA_X_WHOLE
    # INT8 8192^2: whole row blocks would give a CTA 64 tiles, more than it holds partial sums for
    p = probe("INT8_SYM", 1, 8192, 8192, 128)
    assert p["cta_rows"] == 0 and p["launches"] == 2 and p["xmode"] == MMA_X_ROW1
    # INT2 and NF4 8192^2, W4A8 on the down projection: whole row blocks, one launch
    for args in [("INT2_ASYM", 1, 8192, 8192, 64), ("NF4", 1, 8192, 8192, 64)]:
        p = probe(*args)
        assert p["cta_rows"] > 0 and p["launches"] == 1 and p["xmode"] == MMA_X_ROW1, (args, p)
    p = probe("INT4_ASYM", 1, 4096, 14336, 128, a8=True)
    assert not p["warp"] and p["cta_rows"] > 0 and p["launches"] == 1


@pytest.mark.parametrize("fmt,group", [("INT4_ASYM", 128), ("INT4_SYM", 32), ("INT8_SYM", 128), ("INT2_ASYM", 64),
                                       ("NF4", 64), ("K4", 256)])
@pytest.mark.parametrize("M", [1, 2, 8])
@pytest.mark.parametrize("N,K", [(4096, 4096), (14336, 4096), (4096, 14336), (8192, 28672), (300, 2304)])
def test_every_copy_warp_plan_leaves_the_ring_its_slots(probe, fmt, group, M, N, K):
    # the kernel refuses (fault word, no work) a ring of no more slots than tile-taking warp pairs;
    # the planner must never hand it one, in any x mode
    if K % group or (fmt == "INT2_ASYM" and K % 64):
        pytest.skip("shape not valid for the format")
    for a8 in ([False, True] if fmt in ("INT4_ASYM", "INT4_SYM", "INT8_SYM") else [False]):
        p = probe(fmt, M, N, K, group, a8=a8)
        if p["warp"]:
            continue
        assert p["grid"] > 0, p
        assert p["slots"] >= PW + 2, (a8, p)
        assert 1 <= p["pairs"] <= PW
        assert p["xmode"] in (MMA_X_GLOBAL, MMA_X_WHOLE, MMA_X_ROW1)
        if p["xmode"] == MMA_X_ROW1:
            assert M == 1
