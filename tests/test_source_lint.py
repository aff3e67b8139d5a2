"""Source checks of the CUDA kernels that need no GPU.

A warp collective with a full member mask (__shfl_*_sync, __any_sync, ...)
must be reached by every lane of the warp.  Writing one as the right operand
of || or && lets a lane skip it (short-circuit), and the lanes that do reach
it then wait for ever: the warp hangs.  These checks keep that form out."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCES = sorted(glob.glob(os.path.join(ROOT, "unpermute_combine_gb300", "csrc", "*.cu")) +
                 glob.glob(os.path.join(ROOT, "unpermute_combine_gb300", "csrc", "*.cuh")))
COLLECTIVE = r"__(shfl|shfl_up|shfl_down|shfl_xor|any|all|ballot|reduce_\w+|match_\w+)_sync"


def test_sources_found():
    assert len(SOURCES) >= 5


def test_no_warp_collective_behind_a_short_circuit():
    pat = re.compile(r"(\|\||&&|\?)\s*\(?\s*" + COLLECTIVE)
    bad = []
    for path in SOURCES:
        for n, line in enumerate(open(path), 1):
            if pat.search(line):
                bad.append(f"{os.path.basename(path)}:{n}: {line.strip()}")
    assert not bad, "warp collective behind ||, && or ?:\n" + "\n".join(bad)
