"""The C ABI on a machine without a GPU: the library builds and loads, exports
every function include/verify_attn.h declares, sizes workspaces on the host,
and rejects bad arguments with its error codes before any device work."""
import ctypes
import os
import re

import pytest

import mla_speculative_decode_gb300 as va

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "verify_attn.h")

# fake, never dereferenced: the host checks run before any device access
A16 = 0x10000
A256 = 0x20000


@pytest.fixture(scope="module")
def lib():
    va.build()
    return va.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t)\s+(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("verify_attn_paged", "verify_attn_contiguous", "verify_attn_segmented",
              "verify_attn_defrag",
              "va_workspace_bytes", "va_init", "va_read_status", "va_auto_nsplit", "va_version",
              "va_set_partial_events"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_exports_nothing_else():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", va.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    syms = {l.split()[-1] for l in out.splitlines() if " T " in l}
    ours = {s for s in syms if s.startswith(("va_", "verify_attn"))}
    assert ours == set(declared_functions())


def test_version(lib):
    assert lib.va_version() == 100


def test_workspace_bytes_layout(lib):
    B, T, H, ns = 2, 16, 8, 5
    rows = B * T * H
    al = lambda x: (x + 255) // 256 * 256
    rbs = 2 * ((T * H + 255) // 256)   # 128-row blocks, rounded up to pairs
    want = 256 + al(B * T * 8) + al(B * rbs * ns * 2 * 4) + al(ns * rows * 4) + al(ns * rows * 512 * 2)
    assert va.workspace_bytes(B, T, H, ns) == want
    assert lib.va_workspace_bytes(0, 16, 8, 1) == 0
    assert lib.va_workspace_bytes(1, 65, 8, 1) == 0
    assert lib.va_workspace_bytes(1, 16, 8, 0) == 0


def _paged(lib, **over):
    a = dict(q=A16, kv=A16, num_slots=4096, stride=576, slot=A16, indptr=A16, prefix=A16,
             parent=A16, bits=None, B=1, T=4, H=8, scale=0.07, nsplit=4, flags=0, ws=A256,
             ws_bytes=1 << 30, out=A16, lse=A16, stream=None)
    a.update(over)
    return lib.verify_attn_paged(a["q"], a["kv"], a["num_slots"], a["stride"], a["slot"],
                                 a["indptr"], a["prefix"], a["parent"], a["bits"], a["B"], a["T"],
                                 a["H"], a["scale"], a["nsplit"], a["flags"], a["ws"],
                                 a["ws_bytes"], a["out"], a["lse"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(q=None), -1), (dict(kv=None), -1), (dict(slot=None), -1), (dict(indptr=None), -1),
    (dict(prefix=None), -1), (dict(ws=None), -1), (dict(out=None), -1), (dict(lse=None), -1),
    (dict(parent=None, bits=None), -1),
    (dict(B=0), -2), (dict(T=0), -2), (dict(T=65), -2), (dict(H=0), -2), (dict(num_slots=0), -2),
    (dict(stride=512), -2), (dict(nsplit=-1), -2), (dict(nsplit=1025), -2), (dict(flags=7), -2),
    (dict(flags=4), -2), (dict(flags=-1), -2),
    (dict(scale=float("nan")), -2),
    (dict(stride=580), -3), (dict(q=A16 + 8), -3), (dict(kv=A16 + 2), -3), (dict(out=A16 + 4), -3),
    (dict(ws=A256 + 16), -3), (dict(lse=A16 + 2), -3), (dict(slot=A16 + 2), -3),
    (dict(ws_bytes=1000), -4),
])
def test_paged_argument_errors(lib, over, code):
    assert _paged(lib, **over) == code


def test_valid_arguments_without_gpu_do_not_crash(lib):
    # no device (or no va_init): an error code, never a crash
    rc = _paged(lib)
    assert rc in (-5, -7)
    # every compute-path flag passes the argument checks, the one-SM
    # tensor-core shape (VA_PATH_TC_1SM = 3) included
    for flags in (0, 1, 2, 3):
        assert _paged(lib, flags=flags) in (-5, -7)
    assert rc in (-5, -7)


def test_contiguous_argument_errors(lib):
    f = lib.verify_attn_contiguous
    base = [A16, A16, 4096, 576, A16, A16, A16, None, 1, 4, 8, 0.07, 4, 0, A256, 1 << 30, A16, A16,
            None]
    assert f(*base) in (-5, -7)
    bad = list(base); bad[4] = None
    assert f(*bad) == -1
    bad = list(base); bad[4] = A16 + 4
    assert f(*bad) == -3
    bad = list(base); bad[15] = 10
    assert f(*bad) == -4


def _segmented(lib, **over):
    a = dict(q=A16, kv=A16, num_slots=4096, stride=576, indices=A16, indptr=A16, loc=A16,
             draft=None, mask=A16, mask_len=1000, parent=None, bits=None, B=1, T=4, H=8, scale=0.07, nsplit=4,
             flags=0, ws=A256, ws_bytes=1 << 30, out=A16, lse=A16, stream=None)
    a.update(over)
    return lib.verify_attn_segmented(a["q"], a["kv"], a["num_slots"], a["stride"], a["indices"],
                                     a["indptr"], a["loc"], a["draft"], a["mask"], a["mask_len"],
                                     a["parent"],
                                     a["bits"], a["B"], a["T"], a["H"], a["scale"], a["nsplit"],
                                     a["flags"], a["ws"], a["ws_bytes"], a["out"], a["lse"],
                                     a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(indices=None), -1), (dict(indptr=None), -1), (dict(loc=None), -1), (dict(q=None), -1),
    (dict(mask=None), -1), (dict(mask_len=-1), -2), (dict(T=65), -2), (dict(loc=A16 + 2), -3),
    (dict(indices=A16 + 2), -3), (dict(ws_bytes=1000), -4), (dict(draft=A16 + 8), -3),
])
def test_segmented_argument_errors(lib, over, code):
    assert _segmented(lib, **over) == code


def test_segmented_valid_arguments_without_gpu_do_not_crash(lib):
    assert _segmented(lib) in (-5, -7)
    assert _segmented(lib, mask=None, parent=A16) in (-5, -7)


def test_defrag_argument_errors(lib):
    f = lib.verify_attn_defrag
    base = [A16, 4096, 576, A16, A16, A16, None, 1, 100, None, None]
    assert f(*base) in (-5, -7)
    for i, code in ((0, -1), (3, -1), (4, -1), (5, -1)):
        bad = list(base); bad[i] = None
        assert f(*bad) == code
    bad = list(base); bad[7] = 0
    assert f(*bad) == -2
    bad = list(base); bad[2] = 584 + 4
    assert f(*bad) == -3
    bad = list(base); bad[0] = A16 + 8
    assert f(*bad) == -3


def test_read_status_null(lib):
    assert lib.va_read_status(None, None, None) == -1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import importlib
    monkeypatch.setattr(va, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(va, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        va.load()


def test_tree_accept_workspace_and_errors(lib):
    lib.va_tree_accept_workspace_bytes.restype = ctypes.c_size_t
    lib.va_tree_accept_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64]
    n = lib.va_tree_accept_workspace_bytes(8, 16, 129280)
    assert n > 256
    assert lib.va_tree_accept_workspace_bytes(0, 16, 100) == 0
    assert lib.va_tree_accept_workspace_bytes(1, 65, 100) == 0
    assert lib.va_tree_accept_workspace_bytes(1, 16, 0) == 0
    f = lib.va_tree_accept
    P = ctypes.c_void_p
    f.argtypes = [P, P, ctypes.c_int64, P, P, P, ctypes.c_int, ctypes.c_int, P, ctypes.c_size_t,
                  P, P, P, P, P]
    base = [A16, A16, 1000, A16, A16, None, 2, 8, A256, 1 << 20, A16, A16, None, A16, None]
    for i in (0, 1, 3, 4, 8, 10, 11, 13):
        bad = list(base); bad[i] = None
        assert f(*bad) == -1
    bad = list(base); bad[7] = 65
    assert f(*bad) == -2
    bad = list(base); bad[2] = 0
    assert f(*bad) == -2
    bad = list(base); bad[1] = A16 + 2
    assert f(*bad) == -3
    bad = list(base); bad[8] = A256 + 16
    assert f(*bad) == -3
    bad = list(base); bad[9] = 16
    assert f(*bad) == -4


def test_test_build_exports_its_gate_and_the_product_does_not():
    """libverifyattn_testhooks.so (VA_TEST_HOOKS) exports the product ABI plus
    the declarations of include/verify_attn_testhooks.h; the product library
    exports none of the test hooks."""
    import subprocess
    from mla_speculative_decode_gb300 import _builder
    th_path = _builder.build(testhooks=True)
    text = open(os.path.join(ROOT, "include", "verify_attn_testhooks.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    hooks = set(re.findall(r"^\s*(?:int|size_t)\s+(\w+)\s*\(", text, flags=re.M))
    assert hooks == {"va_test_set_gate"}

    def exported(path):
        out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True,
                             text=True, check=True).stdout
        return {l.split()[-1] for l in out.splitlines() if " T " in l}

    th = {s for s in exported(th_path) if s.startswith(("va_", "verify_attn"))}
    assert th == set(declared_functions()) | hooks
    assert not (exported(va.LIB_PATH) & hooks)


def _tree(lib, **over):
    a = dict(tok=A16, lp=A16, B=2, D=4, K=3, T=8, free=A16, cap=100, head=A16, par=A16,
             dtok=A16, depth=A16, loc=A16, status=None, stream=None)
    a.update(over)
    return lib.va_tree_build(a["tok"], a["lp"], a["B"], a["D"], a["K"], a["T"], a["free"],
                             a["cap"], a["head"], a["par"], a["dtok"], a["depth"], a["loc"],
                             a["status"], a["stream"])


def test_tree_build_rejects_bad_arguments_before_any_launch(lib):
    assert _tree(lib, tok=None) == -1
    assert _tree(lib, par=None) == -1
    assert _tree(lib, head=None) == -1            # a free list needs its head
    assert _tree(lib, loc=None) == -1
    assert _tree(lib, D=16) == -2 and _tree(lib, D=0) == -2
    assert _tree(lib, K=17) == -2 and _tree(lib, K=0) == -2
    assert _tree(lib, T=65) == -2 and _tree(lib, T=0) == -2
    assert _tree(lib, B=0) == -2
    # the candidate tree must hold T nodes: K=2, D=3 has 2 + 4 + 8 = 14
    assert _tree(lib, K=2, D=3, T=15) == -2
    assert _tree(lib, K=1, D=4, T=5) == -2
    assert _tree(lib, lp=A16 + 2) == -3
    assert _tree(lib, loc=A16 + 1) == -3


def _append(lib, **over):
    a = dict(pool=A16, num_slots=4096, stride=576, start=A16, prefix=A16, cap=A16, draft=A16,
             B=2, T=4, loc=A16, status=None)
    a.update(over)
    return lib.va_kv_append_contiguous(a["pool"], a["num_slots"], a["stride"], a["start"],
                                       a["prefix"], a["cap"], a["draft"], a["B"], a["T"],
                                       a["loc"], a["status"], None)


def _compact(lib, **over):
    a = dict(pool=A16, num_slots=4096, stride=576, start=A16, prefix=A16, cap=A16, alen=A16,
             nodes=A16, B=2, T=4, status=None)
    a.update(over)
    return lib.va_kv_compact_accepted(a["pool"], a["num_slots"], a["stride"], a["start"],
                                      a["prefix"], a["cap"], a["alen"], a["nodes"], a["B"], a["T"],
                                      a["status"], None)


@pytest.mark.parametrize("over,code", [
    (dict(pool=None), -1), (dict(start=None), -1), (dict(prefix=None), -1), (dict(cap=None), -1),
    (dict(draft=None), -1),
    (dict(B=0), -2), (dict(T=0), -2), (dict(T=65), -2), (dict(num_slots=0), -2),
    (dict(stride=512), -2),
    (dict(stride=580), -3), (dict(pool=A16 + 8), -3), (dict(start=A16 + 4), -3),
    (dict(draft=A16 + 8), -3), (dict(loc=A16 + 2), -3),
])
def test_append_contiguous_argument_errors(lib, over, code):
    assert _append(lib, **over) == code


@pytest.mark.parametrize("over,code", [
    (dict(pool=None), -1), (dict(alen=None), -1), (dict(nodes=None), -1), (dict(cap=None), -1),
    (dict(B=0), -2), (dict(T=65), -2), (dict(stride=100), -2),
    (dict(pool=A16 + 2), -3), (dict(alen=A16 + 2), -3), (dict(prefix=A16 + 1), -3),
])
def test_compact_accepted_argument_errors(lib, over, code):
    assert _compact(lib, **over) == code
