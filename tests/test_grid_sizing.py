"""Grid sizing of the persistent stream kernel (host logic, no GPU).

The kernel's CTAs wait on each other (a row's final polls tile keys that
other CTAs write), so a launch must never have more CTAs than the SMs the
calling context may use can hold at once. persistent_grid() in
csrc/dflash_internal.h makes that choice: SMs available x CTAs per SM, capped
by the number of pieces, and 0 (an error before any launch) when no CTA fits.
It is compiled here with the host compiler and checked case by case.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "speculative_decoding_verification_83_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

PROG = r"""
#include "dflash_internal.h"
#include <cstdio>
int main() {
  long long pieces, ctas;
  int sms, per_sm;
  while (scanf("%lld %d %d", &pieces, &sms, &per_sm) == 3)
    printf("%lld\n", dflash::persistent_grid(pieces, sms, per_sm));
  return 0;
}
"""

CASES = [
    # pieces, SMs available, CTAs per SM -> grid
    (12493, 152, 1, 152),      # the headline: one CTA per SM
    (12493, 100, 1, 100),      # a context limited to 100 SMs (green context)
    (12493, 152, 2, 304),      # two CTAs fit per SM
    (15, 152, 1, 15),          # fewer pieces than SMs: one CTA per piece
    (1, 152, 1, 1),
    (0, 152, 1, 1),            # nothing to stream still launches one CTA (it runs the finals)
    (12493, 0, 1, 0),          # no SM available: refused before launch
    (12493, 152, 0, 0),        # the kernel does not fit on an SM: refused
    (1 << 40, 152, 1, 152),
]


@pytest.fixture(scope="module")
def grid_prog(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None or not os.path.exists(os.path.join(CUDA_INC, "vector_types.h")):
        pytest.skip("no host C++ compiler or CUDA headers")
    d = tmp_path_factory.mktemp("grid")
    src = d / "grid.cpp"
    src.write_text(PROG)
    exe = d / "grid"
    subprocess.check_call([cxx, "-std=c++17", "-O1", "-I", CUDA_INC, "-I", CSRC, str(src), "-o", str(exe)])
    return str(exe)


def test_persistent_grid_cases(grid_prog):
    stdin = "".join(f"{p} {s} {c}\n" for p, s, c, _ in CASES)
    out = subprocess.run([grid_prog], input=stdin.encode(), stdout=subprocess.PIPE, check=True).stdout.decode()
    got = [int(x) for x in out.split()]
    assert got == [g for *_, g in CASES]


def test_grid_never_exceeds_resident_capacity(grid_prog):
    # every grid fits resident at once and is at least one CTA when any fits
    import itertools
    rows = list(itertools.product([0, 1, 7, 151, 152, 153, 5000], [0, 1, 76, 152], [0, 1, 2, 3]))
    stdin = "".join(f"{p} {s} {c}\n" for p, s, c in rows)
    out = subprocess.run([grid_prog], input=stdin.encode(), stdout=subprocess.PIPE, check=True).stdout.decode()
    for (p, s, c), g in zip(rows, (int(x) for x in out.split())):
        if s < 1 or c < 1:
            assert g == 0
        else:
            assert 1 <= g <= s * c and g <= max(1, p)
