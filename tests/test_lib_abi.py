"""The C-ABI library loads and exports every symbol include/ft.h declares; host-only calls work without a GPU."""
import ctypes
import os
import re

import pytest

from conftest import ROOT, read_golden


def declared_functions():
    src = open(os.path.join(ROOT, "include", "ft.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(ft_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ["ft_route", "ft_permute", "ft_cache_create", "ft_cache_step", "ft_cache_resize", "ft_expert_grouped",
              "ft_combine", "ft_stream_create", "ft_stream_layer", "ft_stream_destroy", "ft_qsplit"]:
        assert n in names


def test_library_exports_every_declared_symbol(ftlib):
    lib = ctypes.CDLL(ftlib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert missing == []
    assert sorted(ftlib.EXPORTED) == declared_functions()


def test_binding_constants_match_the_header(ftlib):
    src = open(os.path.join(ROOT, "include", "ft.h")).read()
    defines = {m[0]: m[1] for m in re.findall(r"^#define (FT_\w+) (.+)$", src, flags=re.M)}
    assert set(defines) >= {"FT_TC_WIDE_ASSIGNMENTS", "FT_NOALLOC_MAX_ELEMS"}
    for name, expr in defines.items():
        if name == "FT_H":
            continue
        assert getattr(ftlib, name) == eval(expr.replace("u", "")), name


def test_qsplit_table1(ftlib):
    ms = [1, 2, 3, 4, 6, 8, 16]
    for name, bp, bh, *qs in read_golden("table1_bandwidths.txt"):
        assert [ftlib.ft_qsplit(m, float(bp), float(bh)) for m in ms] == [int(q) for q in qs], name
    assert ftlib.ft_qsplit(0, 1.0, 2.0) == 0
    assert ftlib.ft_qsplit(7, 2.0, 2.0) == 7
    assert ftlib.ft_qsplit(7, 1e-12, 2.0) == 1
    assert ftlib.ft_qsplit(5, 1.0, 2.0) == 3   # 2.5 rounds half up


def test_expert_layouts(ftlib):
    # BF16, H=2048, I=512: three 2 MiB matrices, 6,291,456 bytes per expert
    L = ftlib.ft_expert_layout_get(ftlib.FT_W_BF16, 2048, 512)
    assert L.bytes == L.payload_bytes == 3 * 2048 * 512 * 2
    assert list(L.off_val) == [0, 2048 * 512 * 2, 2 * 2048 * 512 * 2]
    # NVFP4, H=4096, I=2048: values 3*4M, scales 3*512K, 12 bytes of matrix scales
    L = ftlib.ft_expert_layout_get(ftlib.FT_W_NVFP4, 4096, 2048)
    assert L.payload_bytes == 3 * 4096 * 2048 // 2 + 3 * 4096 * 2048 // 16 + 12
    assert abs(L.payload_bytes / 1e6 - 14.16) < 0.01
    # MXFP4, H=6144, I=2048: about 20.05 MB
    L = ftlib.ft_expert_layout_get(ftlib.FT_W_MXFP4, 6144, 2048)
    assert abs(L.payload_bytes / 1e6 - 20.05) < 0.01
    for wt in range(5):
        L = ftlib.ft_expert_layout_get(wt, 1024, 512)
        offs = [o for o in list(L.off_val) + list(L.off_scale) + [L.off_gscale] if o]
        assert all(o % 256 == 0 for o in offs) and L.bytes % 256 == 0
    with pytest.raises(ftlib.FTError):
        ftlib.ft_expert_layout_get(ftlib.FT_W_BF16, 100, 512)
    with pytest.raises(ftlib.FTError):
        ftlib.ft_expert_layout_get(9, 1024, 512)


def test_invalid_arguments_rejected_before_launch(ftlib):
    lib = ftlib.lib()
    s = None
    # bad k / E / T: FT_EINVAL, no device touched
    assert lib.ft_route(None, 4, 16, 0, None, None, s) == ftlib.FT_EINVAL
    assert lib.ft_route(None, 4, 16, 17, None, None, s) == ftlib.FT_EINVAL
    assert lib.ft_route(None, 4, 2000, 2, None, None, s) == ftlib.FT_EINVAL
    assert lib.ft_route(None, 0, 16, 2, None, None, s) == ftlib.FT_OK          # empty batch: no work
    assert lib.ft_permute(None, 2, 2, 1000, None, None, None, None, s) == ftlib.FT_EINVAL
    assert lib.ft_router_logits(None, 1, None, None, 3, 100, 16, None, s) == ftlib.FT_EINVAL
    assert lib.ft_combine(None, None, None, None, None, None, 2, 2, 6, 4, None, s) == ftlib.FT_EINVAL
    assert lib.ft_cache_create(None, None) == ftlib.FT_EINVAL
    assert lib.ft_cache_step(None, 0, None, 1.0, 0, None, None, None, s) == ftlib.FT_EINVAL
    assert lib.ft_expert_grouped(None, 1, 4, 2, 2048, 512, 16, 7, None, None, None, None, 0, 1, None, None, 0, s) \
        == ftlib.FT_EINVAL
    assert ftlib.ft_status_str(ftlib.FT_ESTATE) == "call not allowed in this state"


def test_expert_workspace_grows_with_the_batch(ftlib):
    """A workspace sized for a batch also serves every smaller batch (one buffer per layer object)."""
    lib = ftlib.lib()
    for H, I, k in ((2048, 512, 8), (512, 256, 4), (4096, 2048, 6), (6144, 2048, 8), (256, 128, 2)):
        prev = 0
        for T in list(range(1, 300)) + [511, 512, 1024, 2047, 2048, 4096, 8192]:
            w = lib.ft_expert_grouped_workspace(T, k, H, I)
            assert w >= prev, (H, I, k, T)
            assert w % 256 == 0
            prev = w


def test_header_compiles_as_c99_and_links(ftlib, tmp_path):
    """include/ft.h is a C header: a C99 program that includes it and calls a host-only
    entry point compiles with -pedantic and links against libft.so."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_ft.c"
    src.write_text('#include "ft.h"\n'
                   'int main(void) { return ft_qsplit(4, 50.0, 100.0) == 2 ? 0 : 1; }\n')
    exe = tmp_path / "use_ft"
    lib_dir = os.path.dirname(ftlib.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-L", lib_dir, "-l:libft.so", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert subprocess.run([str(exe)]).returncode == 0
