"""No kernel the library launches in production spills registers.

The fused step runs at the 128-register budget its 14 warps per SM allow;
a spill there turns register traffic into local-memory traffic on the path
that every token takes.  The build keeps ptxas's resource report
(-Xptxas -v) in _build/ptxas.log: every entry function compiled there without
the segment trace (-DMK_NO_TRACE variants of the fused kernel, and every
kernel of the other translation units) must report 0 bytes of spill stores
and loads.  The builds with the trace compiled in run only while a trace is
requested and are not checked.
"""
import os
import re

from decode_megakernel_05_gb300 import build, mk


def _sections():
    build.build()
    log = open(os.path.join(os.path.dirname(mk.library_path()), "ptxas.log")).read()
    out = []
    for sec in re.split(r"^==== ", log, flags=re.M)[1:]:
        head, _, body = sec.partition("\n")
        out.append((head, body))
    return out


def _entries(body):
    """(entry function, its spill line) for every entry compiled in a section."""
    res, cur = [], None
    for line in body.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            cur = m.group(1)
        elif cur and "spill stores" in line:
            res.append((cur, line.strip()))
            cur = None
    return res


def test_production_kernels_do_not_spill():
    secs = _sections()
    checked = 0
    fused = 0
    for head, body in secs:
        if head.startswith("mk_kernel.cu") and "-DMK_NO_TRACE" not in head:
            continue   # the build with the segment trace compiled in
        for fn, line in _entries(body):
            m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
            assert m, line
            assert m.group(1) == "0" and m.group(2) == "0", f"{head}: {fn}: {line}"
            checked += 1
            fused += "mk_decode_kernel" in fn
    assert fused == (len(build.VARIANTS) + len(build.LC_VARIANTS) + len(build.Q8_VARIANTS) +
                     len(build.Q8_LC_VARIANTS) + len(build.Q4_VARIANTS) + len(build.Q4_LC_VARIANTS)), fused
    assert checked > fused
