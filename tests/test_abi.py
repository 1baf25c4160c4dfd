"""CPU-only checks of the C ABI: the library loads, exports every function that
include/moe.h declares, and its host-side logic (sizes, layouts, argument
checks) behaves as documented.  No compute call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def pkg():
    from mixture_experts_layer_device_gb300 import build
    build.build()
    import mixture_experts_layer_device_gb300 as m
    return m


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["moe_route", "moe_forward", "moe_backward", "moe_quantize_mx", "moe_get_status"]:
        assert n in names


def test_library_exports_every_declared_symbol(pkg):
    L = ctypes.CDLL(pkg.LIB_PATH)
    for n in declared_functions():
        assert hasattr(L, n), n
    assert sorted(pkg.EXPORTS) == declared_functions()


def test_sizes_and_layout(pkg):
    cfg = pkg.config(256, 256, 128, 8, 2, 0, "bf16", pkg.MOE_FLAG_BACKWARD)
    assert pkg.moe_padded_rows(cfg) == ((256 * 2 + 127 * 8 + 127) // 128) * 128
    ws = pkg.moe_workspace_bytes(cfg)
    sv = pkg.moe_saved_bytes(cfg)
    assert ws > 0 and sv > 0
    off, nb = pkg.moe_buffer_info(cfg, 0, "o")
    assert off % 256 == 0 and nb == pkg.moe_padded_rows(cfg) * 256 * 2 and off + nb <= sv
    off, nb = pkg.moe_buffer_info(cfg, 1, "status")
    assert off == 0
    cfg_f = pkg.config(256, 256, 128, 8, 2, 0, "bf16", 0)
    assert pkg.moe_workspace_bytes(cfg_f) < ws          # backward buffers only with the flag
    with pytest.raises(RuntimeError):
        pkg.moe_buffer_info(cfg_f, 1, "dO")
    cmx = pkg.config(256, 256, 128, 8, 2, 0, "mxfp8", 0)
    off, nb = pkg.moe_buffer_info(cmx, 1, "xs_sf")
    assert nb == pkg.moe_padded_rows(cmx) * 256 // 32


def test_saved_wgrad_operands_by_format(pkg):
    """A training forward keeps the down wgrad's h operand as bf16 rows
    with BF16 experts and as column-blocked MXFP8 codes h^T with MXFP8 experts;
    the MXFP8 backward keeps dO and dGU only as codes."""
    T, d, m, E, k = 256, 256, 128, 8, 2
    bf = pkg.config(T, d, m, E, k, 0, "bf16", pkg.MOE_FLAG_BACKWARD)
    mx = pkg.config(T, d, m, E, k, 0, "mxfp8", pkg.MOE_FLAG_BACKWARD)
    rp = pkg.moe_padded_rows(mx)
    assert pkg.moe_buffer_info(bf, 0, "h")[1] == pkg.moe_padded_rows(bf) * m * 2
    for name in ("hT", "hT_sf"):
        with pytest.raises(RuntimeError):
            pkg.moe_buffer_info(bf, 0, name)
    assert pkg.moe_buffer_info(mx, 0, "hT")[1] == m * rp
    assert pkg.moe_buffer_info(mx, 0, "hT_sf")[1] == m * rp // 32
    with pytest.raises(RuntimeError):
        pkg.moe_buffer_info(mx, 0, "h")
    for name in ("dO", "dGU"):
        assert pkg.moe_buffer_info(bf, 1, name)[1] > 0
        with pytest.raises(RuntimeError):
            pkg.moe_buffer_info(mx, 1, name)
    assert pkg.moe_buffer_info(mx, 1, "dGUT")[1] == 2 * m * rp
    assert pkg.moe_buffer_info(mx, 1, "dGUq")[1] == rp * 2 * m
    assert pkg.moe_buffer_info(mx, 1, "tile_order")[1] == rp // 32 * 4


@pytest.mark.parametrize("bad,code", [
    (dict(d=100), -2), (dict(m=64), -2), (dict(k=9), -2), (dict(k=0), -1), (dict(E=2000), -2),
    (dict(T=0), -1), (dict(flags=8), -1), (dict(dtype=7), -1), (dict(m_shared=100), -2),
    (dict(ring_rows=256), -1),                          # the ring is MXFP8-only
    (dict(dtype=1, ring_rows=200), -2), (dict(dtype=1, ring_rows=-128), -1),
    (dict(dtype=1, ring_rows=256, gather_sms=65), -1), (dict(dtype=1, d=8448, ring_rows=256), -2),
    (dict(dtype=1, ring_rows=256, flags=4), -1),          # no pre-quantisation dump through the ring
])
def test_invalid_configs_rejected_on_host(pkg, bad, code):
    args = dict(T=64, d=256, m=128, E=8, k=2, m_shared=0, dtype=0, flags=0, ring_rows=0, gather_sms=0)
    args.update(bad)
    cfg = pkg.MoeConfig(*[args[n] for n in ("T", "d", "m", "E", "k", "m_shared", "dtype", "flags", "ring_rows",
                                            "gather_sms")])
    assert pkg.moe_workspace_bytes(cfg) == 0
    W = pkg.weights()
    assert pkg.moe_forward(cfg, 16, 16, W, 16, None, 16, 0) == code


def test_null_and_misaligned_pointers_rejected_on_host(pkg):
    cfg = pkg.config(64, 256, 128, 8, 2)
    W = pkg.weights(gu=1 << 20, dn=1 << 21)
    assert pkg.moe_forward(cfg, None, 16, W, 16, None, 16, 0) == -1
    assert pkg.moe_forward(cfg, 1 << 12, 1 << 12, W, 1 << 12, None, (1 << 12) + 4, 0) == -3
    assert pkg.moe_quantize_mx(16, 1, 100, 128, 0, 16, 16, 0) == -2
    assert pkg.moe_quantize_mx(8, 1, 128, 128, 0, 16, 16, 0) == -3
    # the layer-level weight entry: MXFP8 configs only, then the same checks
    mx = pkg.config(64, 256, 128, 8, 2, 0, "mxfp8")
    assert pkg.moe_quantize_weights(cfg, 16, 256, 256, 0, 16, 16, 0) == -1
    assert pkg.moe_quantize_weights(mx, None, 256, 256, 0, 16, 16, 0) == -1
    assert pkg.moe_quantize_weights(mx, 16, 100, 256, 1, 16, 16, 0) == -2
    assert pkg.moe_quantize_weights(mx, 8, 256, 256, 0, 16, 16, 0) == -3
    # backward without a backward-sized workspace
    assert pkg.moe_backward(cfg, 16, 16, W, 16, 16, 16, 16, 16, None, None, 16, 0) == -1


def test_debug_flag_accepted_unknown_flags_rejected(pkg):
    cfg = pkg.config(64, 256, 128, 8, 2, 0, "bf16", pkg.MOE_FLAG_BACKWARD | pkg.MOE_FLAG_DEBUG_STARVE)
    assert pkg.moe_workspace_bytes(cfg) == pkg.moe_workspace_bytes(pkg.config(64, 256, 128, 8, 2, 0, "bf16",
                                                                              pkg.MOE_FLAG_BACKWARD))
    assert pkg.moe_workspace_bytes(pkg.config(64, 256, 128, 8, 2, 0, "bf16", 8)) == 0


def test_dump_flag_adds_the_dump_buffers_only_with_mxfp8(pkg):
    T, d, m, E, k = 300, 256, 128, 8, 2
    for fmt in ("bf16", "mxfp8"):
        base = pkg.config(T, d, m, E, k, 0, fmt, pkg.MOE_FLAG_BACKWARD)
        dump = pkg.config(T, d, m, E, k, 0, fmt, pkg.MOE_FLAG_BACKWARD | pkg.MOE_FLAG_DEBUG_DUMP)
        if fmt == "bf16":
            assert pkg.moe_workspace_bytes(dump) == pkg.moe_workspace_bytes(base)
            with pytest.raises(Exception):
                pkg.moe_buffer_info(dump, 1, "h_dump")
            continue
        Rp = pkg.moe_padded_rows(dump)
        assert pkg.moe_buffer_info(dump, 1, "h_dump")[1] == Rp * m * 4
        assert pkg.moe_buffer_info(dump, 1, "dGU_dump")[1] == Rp * 2 * m * 2
        assert pkg.moe_workspace_bytes(dump) >= pkg.moe_workspace_bytes(base) + Rp * m * 6
        fwd_only = pkg.config(T, d, m, E, k, 0, fmt, pkg.MOE_FLAG_DEBUG_DUMP)
        pkg.moe_buffer_info(fwd_only, 1, "h_dump")
        with pytest.raises(Exception):
            pkg.moe_buffer_info(fwd_only, 1, "dGU_dump")


def test_scale_layout_calls_check_arguments_on_host(pkg):
    for f in (pkg.moe_prepare_scales, pkg.moe_canonical_scales):
        assert f(None, 128, 128, 1 << 12, 0) == -1
        assert f(1 << 12, 0, 128, 1 << 16, 0) == -1
        assert f(1 << 12, 128, 128, 1 << 12, 0) == -1          # same buffer
        assert f(1 << 12, 100, 128, 1 << 16, 0) == -2
        assert f(1 << 12, 128, 160, 1 << 16, 0) == -2
        assert f((1 << 12) + 4, 128, 128, 1 << 16, 0) == -3


def test_prepare_weights_checks_arguments_on_host(pkg):
    mx = pkg.config(64, 256, 128, 8, 2, 0, "mxfp8")
    P = 1 << 12
    assert pkg.moe_prepare_weights(mx, None, P, P, P, P, P, stream=0) == -1
    assert pkg.moe_prepare_weights(mx, P, P, None, P, P, P, stream=0) == -1          # MXFP8 needs codes + scales
    assert pkg.moe_prepare_weights(mx, P, P, P, P, P, P, P, P, None, None, stream=0) == -1   # gu_t without dn_t
    assert pkg.moe_prepare_weights(mx, P + 8, P, P, P, P, P, stream=0) == -3
    bad = pkg.config(64, 100, 128, 8, 2, 0, "mxfp8")
    assert pkg.moe_prepare_weights(bad, P, P, P, P, P, P, stream=0) == -2


def test_status_strings(pkg):
    L = pkg.lib()
    for c in range(-6, 1):
        assert L.moe_status_string(c).decode() == pkg.STATUS[c]


def test_ring_workspace_replaces_the_dispatch_buffer(pkg):
    """With a ring the workspace holds ring_rows dispatched rows (plus one row of
    codes per token) instead of every routed row; the saved activations do not
    change."""
    full = pkg.config(32768, 7168, 3072, 384, 6, 0, "mxfp8")
    ring = pkg.config(32768, 7168, 3072, 384, 6, 0, "mxfp8", ring_rows=8192, gather_sms=8)
    rows = pkg.moe_padded_rows(full)
    d = 7168
    with pytest.raises(RuntimeError):
        pkg.moe_buffer_info(ring, 1, "xs")
    saved = pkg.moe_workspace_bytes(full) - pkg.moe_workspace_bytes(ring)
    # the ring kernel also keeps the per-token codes (T rows) it gathers from
    assert saved >= (rows - 8192 - 32768) * d * (1 + 1 / 32) - 8192
    assert pkg.moe_saved_bytes(full) == pkg.moe_saved_bytes(ring)
    off, nb = pkg.moe_buffer_info(ring, 1, "ring")
    assert nb == 8192 * d


def _declarations():
    """(name, [parameter declarations]) of every function in the header."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(([^)]*)\)\s*;", src, flags=re.M):
        params = [p.strip() for p in m.group(2).replace("\n", " ").split(",")]
        out[m.group(1)] = [] if params == ["void"] else params
    return out


def _kind_of_decl(p):
    if "*" in p or p.startswith("moe_stream_t"):
        return "ptr"
    base = p.rsplit(None, 1)[0].replace("const", "").strip()
    return {"int": "int", "int32_t": "int", "int64_t": "i64", "size_t": "size", "float": "float"}[base]


def _kind_of_ctype(t):
    if t in (ctypes.c_void_p, ctypes.c_char_p) or issubclass(t, ctypes._Pointer):
        return "ptr"
    # c_int and c_int32 are the same type, as are c_size_t and c_ulong/c_uint64 on LP64
    return {ctypes.c_int: "int", ctypes.c_int64: "i64", ctypes.c_size_t: "size", ctypes.c_float: "float"}[t]


def test_binding_argtypes_match_the_header(pkg):
    L = pkg.lib()
    decls = _declarations()
    assert sorted(decls) == declared_functions()
    for name, params in decls.items():
        want = [_kind_of_decl(p) for p in params]
        got = [_kind_of_ctype(t) for t in getattr(L, name).argtypes]
        assert got == want, name


def _struct_fields(tag):
    """Field names of a `typedef struct { ... } tag;` in declaration order."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct \{([^}]*)\}\s*" + tag + r"\s*;", src).group(1)
    names = []
    for decl in filter(None, (x.strip() for x in body.split(";"))):
        first, *rest = decl.split(",")
        names.append(re.split(r"[\s\*]+", first.strip())[-1])   # type + first declarator
        names += [r.strip().lstrip("*").strip() for r in rest]   # further declarators
    return names


def test_binding_structs_match_the_header(pkg):
    assert [f[0] for f in pkg.MoeConfig._fields_] == _struct_fields("moe_config")
    assert [f[0] for f in pkg.MoeWeights._fields_] == _struct_fields("moe_weights")
    assert ctypes.sizeof(pkg.MoeConfig) == 11 * 4


def test_product_path_never_reaches_the_oracle():
    """The package imports nothing from oracle/; in bench.py only the CPU
    baseline and reference-arm helpers do."""
    import ast
    pkg_dir = os.path.join(ROOT, "mixture_experts_layer_device_gb300")
    for dirpath, _, files in os.walk(pkg_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", src, flags=re.M), f
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    users = set()
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if isinstance(node, ast.ImportFrom) and (node.module or "").split(".")[0] == "oracle":
                    users.add(fn.name)
                if isinstance(node, ast.Import) and any(a.name.split(".")[0] == "oracle" for a in node.names):
                    users.add(fn.name)
    assert users <= {"_prep_worker", "oracle_sample", "oracle_prepare", "oracle_step", "run_reference",
                     "cpu_baseline", "oracle_dw_time"}, users
    # the CPU baseline's helper is called from the CPU baseline only
    callers = {fn.name for fn in ast.walk(tree) if isinstance(fn, ast.FunctionDef)
               for node in ast.walk(fn) if isinstance(node, ast.Call)
               and getattr(node.func, "id", None) == "oracle_dw_time"}
    assert callers <= {"cpu_baseline"}, callers
    top = [n for n in tree.body if isinstance(n, (ast.Import, ast.ImportFrom))]
    assert not any("oracle" in ast.dump(n) for n in top)


def test_binding_raises_without_the_library(monkeypatch):
    import mixture_experts_layer_device_gb300 as m
    monkeypatch.setattr(m, "_lib", None)
    monkeypatch.setattr(m, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libmoe_gb300.so"))
    with pytest.raises(RuntimeError):
        m.lib()


def test_header_is_plain_c_and_links_from_c(pkg, tmp_path):
    """include/moe.h compiles as C99 and C++17, and a C program links against
    the library and calls a host-only entry point."""
    import shutil
    import subprocess
    gcc, gxx = shutil.which("gcc"), shutil.which("g++")
    if not gcc or not gxx:
        pytest.skip("no host C compiler")
    inc = os.path.join(ROOT, "include")
    for cc, lang, std in ((gcc, "c", "-std=c99"), (gxx, "c++", "-std=c++17")):
        r = subprocess.run([cc, std, "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-x", lang, HEADER],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
    src = tmp_path / "use_abi.c"
    src.write_text('#include <stdio.h>\n#include "moe.h"\n'
                   "int main(void) {\n"
                   "  moe_config c = {256, 256, 128, 8, 2, 0, MOE_BF16, MOE_FLAG_BACKWARD, 0, 0, 0.0f};\n"
                   "  size_t ws = moe_workspace_bytes(&c);\n"
                   "  c.k = 9; /* k > E */\n"
                   "  printf(\"%zu %zu\\n\", ws, moe_workspace_bytes(&c));\n"
                   "  return 0;\n}\n")
    exe = tmp_path / "use_abi"
    libdir = os.path.dirname(pkg.LIB_PATH)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", inc, str(src), "-o", str(exe), "-L", libdir,
                        "-l:" + os.path.basename(pkg.LIB_PATH), "-Wl,-rpath," + libdir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    ws, bad = (int(v) for v in r.stdout.split())
    cfg = pkg.config(256, 256, 128, 8, 2, 0, "bf16", pkg.MOE_FLAG_BACKWARD)
    assert ws == pkg.moe_workspace_bytes(cfg) > 0 and bad == 0
