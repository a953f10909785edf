"""The C-ABI library builds for sm_103a, loads without a GPU, and exports every
function include/mk.h declares; the Python binding covers each one."""
import ctypes
import os
import re

from decode_megakernel_05_gb300 import mk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    lib = mk.load()
    names = declared_functions()
    assert len(names) >= 18, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in mk.h but not exported"
    bound = {n for n, _, _ in mk.SIGNATURES}
    assert set(names) == bound, set(names) ^ bound


def test_library_is_sm103a_and_self_contained():
    path = mk.library_path()
    assert os.path.exists(path)
    log = open(os.path.join(os.path.dirname(path), "ptxas.log")).read()
    assert "for 'sm_103a'" in log
    # the CUDA runtime is linked statically: no libcudart dependency to resolve at load time
    ctypes.CDLL(path)


def test_host_only_entry_points():
    assert mk.mk_strerror(mk.MK_ERR_DEVICE_TIMEOUT) == "device-side wait timed out"
    cfg = mk.mk_config(2, 256, 4, 2, 64, 688, 1024, 80, 1e-5, 1e4, 0)
    assert mk.mk_arena_bytes(cfg, None, 152) > 0
    bad = mk.mk_config(2, 256, 4, 3, 64, 688, 1024, 80, 1e-5, 1e4, 0)   # 4 % 3 != 0
    assert mk.mk_arena_bytes(bad, None, 150) == -1
    odd = mk.mk_config(2, 256, 4, 2, 96, 688, 1024, 80, 1e-5, 1e4, 0)   # head_dim 96 unsupported
    assert mk.mk_arena_bytes(odd, None, 152) == -1
    ragged = mk.mk_config(2, 3000, 24, 8, 128, 8192, 1024, 80, 1e-5, 1e4, 0)   # 3000 is not a multiple of 256
    assert mk.mk_arena_bytes(ragged, None, 152) == -1
    wide = mk.mk_config(2, 3072, 32, 8, 128, 8192, 1024, 80, 1e-5, 1e4, 0)     # layout fine; no kernel variant
    assert mk.mk_arena_bytes(wide, None, 152) > 0


def test_ring_slot_limit():
    """A consumer lane holds its share of a hidden-width tile in registers, so
    ring slots are 32 KB at most; larger requests are refused at planning."""
    cfg = mk.mk_config(2, 2048, 32, 8, 64, 8192, 1024, 80, 1e-5, 1e4, 1)
    assert mk.mk_arena_bytes(cfg, mk.tuning(slot_kib=32), 152) > 0
    assert mk.mk_arena_bytes(cfg, mk.tuning(slot_kib=16), 152) > 0
    assert mk.mk_arena_bytes(cfg, mk.tuning(slot_kib=64), 152) == -1


def test_every_kernel_build_is_in_the_library():
    """Each (head_dim, q heads per kv head, hidden/256) variant exists twice
    (without and with the segment trace), and so does each long-context and
    each weight-only INT8 / INT4 build."""
    from decode_megakernel_05_gb300 import build
    lib = mk.load()
    for hd, g, mh in build.VARIANTS:
        for pre in ("mk_kernel_ptr_", "mk_kernel_trace_ptr_"):
            assert hasattr(lib, f"{pre}{hd}_{g}_{mh}"), (pre, hd, g, mh)
    for hd, g, mh in build.LC_VARIANTS:
        for pre in ("mk_kernel_ptr_", "mk_kernel_trace_ptr_"):
            assert hasattr(lib, f"{pre}{hd}_{g}_{mh}_lc"), (pre, hd, g, mh)
    # the weight-only INT8 / INT4 builds, standard and long-context
    for table, sfx in ((build.Q8_VARIANTS, "_q8"), (build.Q8_LC_VARIANTS, "_lc_q8"),
                       (build.Q4_VARIANTS, "_q4"), (build.Q4_LC_VARIANTS, "_lc_q4")):
        for hd, g, mh in table:
            for pre in ("mk_kernel_ptr_", "mk_kernel_trace_ptr_"):
                assert hasattr(lib, f"{pre}{hd}_{g}_{mh}{sfx}"), (pre, hd, g, mh, sfx)


def test_no_closed_cuda_calls_in_sources():
    """The batched-memcpy family of CUDA calls is not used, and no source names it."""
    pat = re.compile(r"(cuda|cu)Memcpy(3D)?BatchAsync")
    for d in ("decode_megakernel_05_gb300", "include", "oracle", "synth", "tests"):
        for base, _, files in os.walk(os.path.join(ROOT, d)):
            for f in files:
                if f.endswith((".cu", ".h", ".c", ".cpp", ".py")) and f != "test_abi.py":
                    assert not pat.search(open(os.path.join(base, f), errors="ignore").read()), f


def test_binding_constants_match_header():
    """Every MK_DBG_* / MK_ERR_* / MK_OK number the header defines has the same
    value in the Python binding, and mk_info's and mk_tuning's fields are
    mirrored in order and width."""
    src = open(os.path.join(ROOT, "include", "mk.h")).read()
    defs = dict(re.findall(r"#define\s+(MK_(?:DBG|ERR)_[A-Z0-9_]+|MK_OK)\s+\(?(-?\d+)\)?", src))
    assert "MK_DBG_ATTN_BUILD" in defs and "MK_DBG_ATTN_TC_MIN" in defs
    for name, val in defs.items():
        if hasattr(mk, name):
            assert getattr(mk, name) == int(val), name
    assert all(hasattr(mk, n) for n in defs if n.startswith("MK_DBG_")), defs
    for name, cls in (("mk_info", mk.mk_info), ("mk_tuning", mk.mk_tuning)):
        end = src.index("} %s;" % name)
        body = src[src.rindex("typedef struct {", 0, end):end]
        body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
        fields = [f.strip() for decl in re.findall(r"int(?:32|64)_t\s+([^;]+);", body) for f in decl.split(",")]
        assert fields == [f for f, _ in cls._fields_], (name, fields)
        # and the widths: every field of these two structs is int32_t or int64_t
        widths = [w for decl_w, decl in re.findall(r"int(32|64)_t\s+([^;]+);", body) for w in [decl_w] * len(decl.split(","))]
        assert [8 if w == "64" else 4 for w in widths] == [mk.ctypes.sizeof(t) for _, t in cls._fields_], name
