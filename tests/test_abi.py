"""The C-ABI library loads, exports every entry point include/vas.h declares, and
rejects bad arguments on the host (no kernel is launched by these checks)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "vas.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\([^;{]*\)\s*;", text)
    return sorted(set(n for n in names if n not in ("if", "sizeof")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["paged_attn_fwd", "paged_attn_fwd_tree", "paged_attn_fwd_quant",
              "paged_attn_workspace_size", "spec_verify", "vas_last_device_error",
              "vas_pool_create", "vas_build_block_table", "vas_seq_rollback"]:
        assert n in names


def test_library_exports_every_declared_symbol(vas_lib):
    lib = ctypes.CDLL(vas_lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def _dims(vas_lib, **kw):
    d = dict(num_seqs=4, total_q_tokens=10, num_q_heads=32, num_kv_heads=8, head_dim=128,
             page_size=16, num_pages=100, max_pages_per_seq=10, kv_dtype=vas_lib.VAS_BF16, scale=0.0)
    d.update(kw)
    return vas_lib.vas_attn_dims(**d)


def test_workspace_queries(vas_lib):
    d = _dims(vas_lib)
    mn, rec = vas_lib.paged_attn_workspace_min(d), vas_lib.paged_attn_workspace_size(d)
    assert 0 < mn <= rec
    # partial capacity grows with the output rows
    d2 = _dims(vas_lib, total_q_tokens=1000)
    assert vas_lib.paged_attn_workspace_size(d2) > rec
    for bad in [dict(num_q_heads=30), dict(head_dim=96), dict(page_size=8), dict(kv_dtype=7),
                dict(num_seqs=-1)]:
        assert vas_lib.paged_attn_workspace_size(_dims(vas_lib, **bad)) == 0


def test_host_validation_without_launch(vas_lib):
    lib = vas_lib._lib
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: validation fails first
    d = _dims(vas_lib)
    null = P(0)
    st = lib.paged_attn_fwd(null, fake, fake, fake, fake, fake, fake, fake, ctypes.byref(d), fake,
                            1 << 30, null)
    assert st == vas_lib.VAS_E_INVALID_ARG
    st = lib.paged_attn_fwd(fake, fake, fake, fake, fake, fake, fake, fake,
                            ctypes.byref(_dims(vas_lib, head_dim=80)), fake, 1 << 30, null)
    assert st == vas_lib.VAS_E_UNSUPPORTED
    st = lib.paged_attn_fwd(fake, fake, fake, fake, fake, fake, fake, fake,
                            ctypes.byref(_dims(vas_lib, num_q_heads=33)), fake, 1 << 30, null)
    assert st == vas_lib.VAS_E_INVALID_ARG
    misaligned = P((1 << 20) + 8)
    st = lib.paged_attn_fwd(misaligned, fake, fake, fake, fake, fake, fake, fake, ctypes.byref(d),
                            fake, 1 << 30, null)
    assert st == vas_lib.VAS_E_INVALID_ARG
    st = lib.paged_attn_fwd(fake, fake, fake, fake, fake, fake, fake, fake, ctypes.byref(d), fake,
                            16, null)
    assert st == vas_lib.VAS_E_WORKSPACE
    # empty batch is a no-op
    assert lib.paged_attn_fwd(null, null, null, null, null, null, null, null,
                              ctypes.byref(_dims(vas_lib, num_seqs=0)), null, 0, null) == vas_lib.VAS_OK
    # the draft-tree entry point: a null or misaligned mask is refused on the host
    st = lib.paged_attn_fwd_tree(fake, fake, fake, fake, fake, fake, null, fake, fake,
                                 ctypes.byref(d), fake, 1 << 30, null)
    assert st == vas_lib.VAS_E_INVALID_ARG
    st = lib.paged_attn_fwd_tree(fake, fake, fake, fake, fake, fake, P((1 << 20) + 4), fake, fake,
                                 ctypes.byref(d), fake, 1 << 30, null)
    assert st == vas_lib.VAS_E_INVALID_ARG
    st = lib.paged_attn_fwd_tree(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                 ctypes.byref(d), fake, 16, null)
    assert st == vas_lib.VAS_E_WORKSPACE
    # quantised pools: only through paged_attn_fwd_quant, and only with both scale arrays
    for kv in (vas_lib.VAS_FP8_E4M3, vas_lib.VAS_INT8):
        dq = _dims(vas_lib, kv_dtype=kv)
        assert vas_lib.paged_attn_workspace_size(dq) == vas_lib.paged_attn_workspace_size(d)
        st = lib.paged_attn_fwd(fake, fake, fake, fake, fake, fake, fake, fake, ctypes.byref(dq),
                                fake, 1 << 30, null)
        assert st == vas_lib.VAS_E_INVALID_ARG
        st = lib.paged_attn_fwd_quant(fake, fake, fake, null, fake, fake, fake, fake, null, fake,
                                      fake, ctypes.byref(dq), fake, 1 << 30, null)
        assert st == vas_lib.VAS_E_INVALID_ARG
        st = lib.paged_attn_fwd_quant(fake, fake, fake, fake, P((1 << 20) + 4), fake, fake, fake,
                                      null, fake, fake, ctypes.byref(dq), fake, 1 << 30, null)
        assert st == vas_lib.VAS_E_INVALID_ARG
        st = lib.paged_attn_fwd_quant(fake, fake, fake, fake, fake, fake, fake, fake, null, fake,
                                      fake, ctypes.byref(dq), fake, 16, null)
        assert st == vas_lib.VAS_E_WORKSPACE
    st = lib.paged_attn_fwd_quant(fake, fake, fake, fake, fake, fake, fake, fake, null, fake, fake,
                                  ctypes.byref(d), fake, 1 << 30, null)
    assert st == vas_lib.VAS_E_INVALID_ARG  # bf16 pools take no scales
    # spec_verify argument checks
    assert lib.spec_verify(fake, fake, fake, 1, fake, fake, 4, 3, 0, null) == vas_lib.VAS_E_INVALID_ARG
    assert lib.spec_verify(null, fake, fake, 1, fake, fake, 4, 3, 10, null) == vas_lib.VAS_E_INVALID_ARG
    assert lib.spec_verify(fake, fake, fake, 1, fake, fake, -1, 3, 10, null) == vas_lib.VAS_E_INVALID_ARG
    assert lib.spec_verify(fake, null, null, 1, fake, fake, 4, 3, 10, null) == vas_lib.VAS_E_INVALID_ARG
    assert lib.spec_verify(null, null, null, 1, null, null, 0, 3, 10, null) == vas_lib.VAS_OK
    assert lib.vas_status_string(vas_lib.VAS_E_WORKSPACE) == b"workspace too small"


def test_host_validation_of_the_other_entry_points(vas_lib):
    """spec_verify_tree, vas_philox4x32_10 and paged_attn_fwd_static refuse bad arguments
    before any CUDA call."""
    lib = vas_lib._lib
    P = ctypes.c_void_p
    fake, null = P(1 << 20), P(0)
    tree = lambda B, n, V, p=fake, path=fake: lib.spec_verify_tree(p, fake, fake, fake, 1, fake,
                                                                 fake, path, B, n, V, null)
    assert tree(4, 0, 100) == vas_lib.VAS_E_INVALID_ARG      # no draft node
    assert tree(4, 256, 100) == vas_lib.VAS_E_INVALID_ARG    # more nodes than 255
    assert tree(-1, 4, 100) == vas_lib.VAS_E_INVALID_ARG
    assert tree(4, 4, 0) == vas_lib.VAS_E_INVALID_ARG
    assert tree(4, 4, 100, p=null) == vas_lib.VAS_E_INVALID_ARG
    assert tree(4, 4, 100, path=null) == vas_lib.VAS_E_INVALID_ARG
    assert tree(4, 1, 8 * 160 * 256 + 1) == vas_lib.VAS_E_UNSUPPORTED  # past 327680
    assert tree(4, 255, 1 << 22) == vas_lib.VAS_E_INVALID_ARG  # (n + 1) V past int32 / 2
    assert lib.spec_verify_tree(null, null, null, null, 1, null, null, null, 0, 4, 100,
                                null) == vas_lib.VAS_OK      # empty batch
    ph = lib.vas_philox4x32_10
    assert ph(fake, 1, 2, fake, -1, null) == vas_lib.VAS_E_INVALID_ARG
    assert ph(null, 1, 2, fake, 8, null) == vas_lib.VAS_E_INVALID_ARG
    assert ph(P((1 << 20) + 4), 1, 2, fake, 8, null) == vas_lib.VAS_E_INVALID_ARG
    assert ph(null, 1, 2, null, 0, null) == vas_lib.VAS_OK
    st = lib.paged_attn_fwd_static
    st.argtypes = [P] * 8 + [ctypes.POINTER(vas_lib.vas_attn_dims), P]
    st.restype = ctypes.c_int
    assert st(fake, fake, fake, fake, fake, fake, fake, fake,
              ctypes.byref(_dims(vas_lib, head_dim=80)), null) == vas_lib.VAS_E_UNSUPPORTED
    assert st(fake, fake, fake, fake, fake, fake, fake, fake,
              ctypes.byref(_dims(vas_lib, num_q_heads=33)), null) == vas_lib.VAS_E_INVALID_ARG
    big = _dims(vas_lib, num_seqs=2_000_000, total_q_tokens=2_000_000)
    assert st(fake, fake, fake, fake, fake, fake, fake, fake, ctypes.byref(big),
              null) == vas_lib.VAS_E_WORKSPACE               # past the 32 MiB array


def test_product_path_never_reaches_the_oracle():
    """Nothing in the package imports, loads or runs the oracle, and the oracle imports
    nothing from the CUDA path: the two share only the input generators."""
    import ast
    pkg = os.path.join(ROOT, "verify_attention_spec_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            path = os.path.join(dirpath, f)
            if f.endswith(".py"):
                tree = ast.parse(open(path).read())
                for node in ast.walk(tree):
                    if isinstance(node, ast.Import):
                        names = [n.name for n in node.names]
                    elif isinstance(node, ast.ImportFrom):
                        names = [node.module or ""]
                    else:
                        continue
                    assert not any(n.split(".")[0] == "oracle" for n in names), path
                text = open(path).read()
                assert "liboracle" not in text and "oracle.c" not in text, path
            elif f.endswith((".cu", ".cuh", ".cpp", ".h")):
                assert "oracle" not in open(path).read().lower(), path
    odir = os.path.join(ROOT, "oracle")
    for f in os.listdir(odir):
        path = os.path.join(odir, f)
        if f.endswith(".py"):
            for node in ast.walk(ast.parse(open(path).read())):
                if isinstance(node, (ast.Import, ast.ImportFrom)):
                    names = ([n.name for n in node.names] if isinstance(node, ast.Import)
                             else [node.module or ""])
                    assert not any(n.startswith("verify_attention_spec_gb300") for n in names), f
            assert "libvas" not in open(path).read(), f
        elif f.endswith((".c", ".h")):
            includes = [l for l in open(path) if l.lstrip().startswith("#include")]
            assert not any("vas" in l or "csrc" in l for l in includes), f


def test_binding_fails_loudly_without_library(tmp_path):
    """The product package raises when libvas.so is absent instead of falling back."""
    import subprocess
    import sys
    pkg = tmp_path / "verify_attention_spec_gb300"
    pkg.mkdir()
    src = os.path.join(ROOT, "verify_attention_spec_gb300")
    for f in ["__init__.py", "binding.py", "workloads.py", "_build.py"]:
        (pkg / f).write_text(open(os.path.join(src, f)).read())
    # the build script and the input generators import without the library ...
    code = ("from verify_attention_spec_gb300 import _build, workloads; "
            "import verify_attention_spec_gb300 as v; v.workloads.WORKLOADS['tiny']")
    res = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    # ... but the binding (and any compute entry point) refuses to run
    for code in ["import verify_attention_spec_gb300.binding",
                 "import verify_attention_spec_gb300 as v; v.paged_attn_fwd"]:
        res = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True,
                             text=True)
        assert res.returncode != 0 and "libvas.so" in res.stderr and "ImportError" in res.stderr
