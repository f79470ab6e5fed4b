"""The C-ABI library builds, loads and exports every symbol include/megamoe.h
declares; host-side argument checks work without a GPU."""
import ctypes
import os
import re

import pytest

import moe_expert_layer_scan_gb300 as mm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "megamoe.h")).read()
    return sorted(set(re.findall(r"MM_API\s+[\w\s\*]+?\b(mm_\w+)\s*\(", hdr)))


@pytest.fixture(scope="module")
def lib():
    mm.build()
    return mm.lib()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for need in ("mm_create", "mm_set_options", "mm_workspace_bytes", "mm_run", "mm_get_status", "mm_destroy"):
        assert need in syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} not exported"


def test_binding_mirrors_the_c_names():
    for name in declared_symbols():
        assert hasattr(mm, name), f"binding lacks {name}"


def test_binding_constants_match_the_header():
    """Every policy, format and device-status value the header defines has the
    same name and value in the binding."""
    hdr = open(os.path.join(ROOT, "include", "megamoe.h")).read()
    defs = {n: int(v.strip("()").rstrip("u"), 0)
            for n, v in re.findall(r"#define\s+(MM_\w+)\s+(\(?-?(?:0x[0-9a-fA-F]+|\d+)u?\)?)", hdr)}
    wanted = [n for n in defs if re.match(r"MM_(TILES|SCHEDULE|WEIGHTS|DEV)_", n)]
    assert {"MM_TILES_AUTO", "MM_TILES_16", "MM_TILES_64", "MM_TILES_112", "MM_TILES_224"} <= set(wanted)
    for n in wanted:
        assert getattr(mm, n) == defs[n], n


def test_status_strings(lib):
    assert mm.mm_status_string(0) == "ok"
    assert mm.mm_status_string(3) == "workspace too small"


def test_create_rejects_bad_shapes_before_touching_the_device(lib):
    h = ctypes.c_void_p()
    assert lib.mm_create(None, 8, 512, 256, 2, 0) == 1                          # null out-pointer
    assert lib.mm_create(ctypes.byref(h), 0, 512, 256, 2, 0) == 1               # no experts
    assert lib.mm_create(ctypes.byref(h), 8, 500, 256, 2, 0) == 2               # H not a multiple of 128
    assert lib.mm_create(ctypes.byref(h), 8, 512, 200, 2, 0) == 2               # I not a multiple of 128
    assert lib.mm_create(ctypes.byref(h), 1020, 512, 256, 2, 5) == 2            # E + S > 1024
    assert lib.mm_create(ctypes.byref(h), 8, 512, 256, 16, 1) == 2              # topk + S > 16


def test_null_handle_calls_are_rejected(lib):
    n = ctypes.c_size_t()
    assert lib.mm_workspace_bytes(None, 4, ctypes.byref(n)) == 1
    assert lib.mm_set_options(None, 1.0, 0) == 1
    assert lib.mm_run(None, 1, *([None] * 10), 0, None) == 1
    lib.mm_destroy(None)


def test_binding_return_types():
    """Functions returning strings or nothing are not read back as status codes."""
    L = mm.lib()
    assert L.mm_status_string.restype is ctypes.c_char_p
    assert L.mm_profile_name.restype is ctypes.c_char_p
    assert L.mm_destroy.restype is None
    assert L.mm_run.restype is ctypes.c_int


PAGE_NAMES = ("MegaMoE research report", "MEGAMOE_SM90_DESIGN", "MEGAMOE_SM90_DEV", "pull request #411")


def declaration_comments():
    """(symbol, the comment block that documents it) for every MM_API
    declaration: the nearest comment above it, with only #defines, blank lines
    and the other declarations of the same group in between."""
    lines = open(os.path.join(ROOT, "include", "megamoe.h")).read().split("\n")
    out = []
    for i, line in enumerate(lines):
        m = re.match(r"MM_API\s+[\w\s\*]+?\b(mm_\w+)\s*\(", line)
        if not m:
            continue
        j = i - 1
        while j >= 0:
            t = lines[j].strip()
            if t.endswith("*/"):
                break
            prev_decl = t.startswith("MM_API") or (t.endswith(");") and not t.startswith("}"))
            cont = lines[j].startswith(" ") and not t.startswith("*") and not t.startswith("/*")
            if t == "" or t.startswith("#define") or prev_decl or cont:
                j -= 1
                continue
            j = -1
        if j < 0:
            out.append((m.group(1), None))
            continue
        k = j
        while k >= 0 and "/*" not in lines[k]:
            k -= 1
        out.append((m.group(1), "\n".join(lines[k:j + 1])))
    return out


def test_every_boundary_call_cites_its_passage():
    """Each declaration is documented by a comment that names the page (and
    section) defining the operation, or says that the pages have none."""
    decls = declaration_comments()
    assert {n for n, _ in decls} == set(declared_symbols())
    for name, comment in decls:
        assert comment is not None, f"{name}: no comment directly above the declaration"
        flat = " ".join(w for w in comment.split() if w not in ("/*", "*", "*/"))
        assert any(p in flat for p in PAGE_NAMES) or "no counterpart" in flat, \
            f"{name}: its comment names no page of the method"
