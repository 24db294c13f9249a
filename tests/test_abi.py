"""The C-ABI library without a GPU: it loads, exports every function include/adaln.h
declares, and its host-only logic (bucket rule, status names, argument checks that
return before any CUDA call) behaves as documented."""
import ctypes
import itertools
import os
import re
import subprocess

import pytest

import adaln_layernorm_modulate_gb300 as A
from oracle.bucket import bucket_batch as oracle_bucket_batch
from tests.test_bucket import brute_force, golden_rows

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "adaln.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(adaln_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(A.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = A.lib()
    out = subprocess.run(["nm", "-D", "--defined-only", A.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (adaln_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_debug_library_exports_every_declared_symbol():
    if not os.path.exists(A.DEBUG_LIB_PATH):
        pytest.skip("libadaln_debug.so not built")
    out = subprocess.run(["nm", "-D", "--defined-only", A.DEBUG_LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (adaln_\w+)", out))
    for name in declared_functions():
        assert name in exported, name


def test_release_library_has_no_debug_word():
    # The release build compiles the index checks away: adaln_debug_read answers
    # ADALN_ERR_UNSUPPORTED before any device work (and rejects nothing else first).
    word = ctypes.c_uint32(7)
    assert A.lib().adaln_debug_read(ctypes.addressof(word), 0) == 2
    assert A.lib().adaln_debug_read(None, 1) == 2
    assert word.value == 7
    with pytest.raises(A.AdalnError):
        A.adaln_debug_read()


def test_bucket_batch_matches_oracle_and_brute_force():
    for S, M_mem, M_comp, p in itertools.product(range(1, 24), (1, 5, 17, 64, 100),
                                                 (1, 9, 50, 333, 1000), (1, 2, 3)):
        want = brute_force(S, M_mem, M_comp, p)
        assert A.adaln_bucket_batch(S, M_mem, M_comp, p) == want
        assert oracle_bucket_batch(S, M_mem, M_comp, p) == want
    for S, M_mem, M_comp, p, B in golden_rows():
        assert A.adaln_bucket_batch(S, M_mem, M_comp, p) == B


def test_bucket_batch_large_and_invalid():
    cases = [(2, 2 ** 62, 2 ** 62, 61), (3, 2 ** 62, 2 ** 62, 40), (2 ** 40, 2 ** 62, 2 ** 62 - 1, 1),
             (65536, 2 ** 63 - 1, 2 ** 63 - 1, 3), (1, 2 ** 63 - 1, 5, 1000), (7, 10 ** 18, 10 ** 18, 21)]
    for c in cases:
        assert A.adaln_bucket_batch(*c) == oracle_bucket_batch(*c)
    for bad in ((0, 1, 1, 1), (1, 0, 1, 1), (1, 1, 0, 1), (1, 1, 1, 0), (-5, 1, 1, 2)):
        assert A.adaln_bucket_batch(*bad) == -1


def test_status_strings():
    for code, name in A.STATUS.items():
        assert A.adaln_status_string(code).startswith(name)
    assert "unknown" in A.adaln_status_string(99)


@pytest.mark.parametrize("D,dtype,want", [(7, 1, 2), (0, 1, 2), (16392, 0, 2), (100, 0, 2),
                                          (128, 5, 1), (128, -1, 1)])
def test_shape_and_dtype_checks(D, dtype, want):
    assert A.lib().adaln_fwd(16, 16, 16, 16, 16, 16, 1, 1, D, 1e-6, dtype, None) == want
    assert A.lib().adaln_bwd(16, 16, 16, 16, 16, 16, 16, 16, 256, 1 << 20, 1, 1, D, dtype, None) == want


def test_argument_checks_before_any_device_work():
    L = A.lib()
    # eps must be positive and finite; sizes non-negative
    assert L.adaln_fwd(16, 16, 16, 16, 16, 16, 1, 1, 64, 0.0, 1, None) == 1
    assert L.adaln_fwd(16, 16, 16, 16, 16, 16, 1, 1, 64, float("inf"), 1, None) == 1
    assert L.adaln_fwd(16, 16, 16, 16, 16, 16, -1, 1, 64, 1e-6, 1, None) == 1
    # empty problems are valid no-ops
    assert L.adaln_fwd(None, None, None, None, None, None, 0, 5, 64, 1e-6, 1, None) == 0
    # backward recomputing the statistics: eps, workspace
    assert L.adaln_bwd_recompute(16, 16, 16, 16, 16, 16, 256, 1 << 20, 1, 1, 64, 0.0, 1, None) == 1
    assert L.adaln_bwd_recompute(16, 16, 16, 16, 16, 16, None, 1 << 20, 1, 1, 64, 1e-6, 1, None) == 4
    # null and misaligned pointers
    assert L.adaln_fwd(None, 16, 16, 16, 16, 16, 1, 1, 64, 1e-6, 1, None) == 1
    assert L.adaln_fwd(24, 16, 16, 16, 16, 16, 1, 1, 64, 1e-6, 1, None) == 3
    assert L.adaln_fwd(16, 16, 16, 16, 18, 16, 1, 1, 64, 1e-6, 1, None) == 3
    # backward: missing / misaligned workspace
    assert L.adaln_bwd(16, 16, 16, 16, 16, 16, 16, 16, None, 1 << 20, 1, 1, 64, 1, None) == 4
    assert L.adaln_bwd(16, 16, 16, 16, 16, 16, 16, 16, 272, 1 << 20, 1, 1, 64, 1, None) == 3
    assert L.adaln_bwd(16, 16, 16, 16, 16, 16, 16, 16, 256, 100, 1, 1, 64, 1, None) == 4
    # packed calls: table pointers, rows without segments, int32 token limit
    assert L.adaln_fwd_varlen(16, 16, 16, 16, 16, 16, None, 16, 1, 5, 1, 64, 1e-6, 256, 1 << 20, 1, None) == 1
    assert L.adaln_fwd_varlen(16, 16, 16, 16, 16, 16, 16, None, 1, 5, 1, 64, 1e-6, 256, 1 << 20, 1, None) == 1
    assert L.adaln_fwd_varlen(16, 16, 16, 16, 16, 16, 16, 16, 0, 5, 1, 64, 1e-6, 256, 1 << 20, 1, None) == 1
    assert L.adaln_fwd_varlen(16, 16, 16, 16, 16, 16, 16, 16, 1, 2 ** 31, 1, 64, 1e-6, 256, 1 << 20, 1, None) == 1
    assert L.adaln_fwd_varlen(16, 16, 16, 16, 16, 16, 16, 16, 1, 5, 1, 64, 1e-6, 256, 16, 1, None) == 4
    assert L.adaln_bwd_varlen(16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 5, 1, 64, None, 0, 1, None) == 4
    assert L.adaln_read_status(None, None) == 4
    # rank-order gradient sum: world, size, pointers
    assert L.adaln_sum_ranks(16, 32, 0, 8, None) == 1
    assert L.adaln_sum_ranks(16, 32, 2, -1, None) == 1
    assert L.adaln_sum_ranks(16, 32, 2, 0, None) == 0
    assert L.adaln_sum_ranks(None, 32, 2, 8, None) == 1
    assert L.adaln_sum_ranks(16, 40, 2, 8, None) == 3
    assert L.adaln_sum_ranks(16, 32, 2, 2 ** 62, None) == 1


def test_workspace_size_rejects_bad_shapes():
    assert A.adaln_fwd_varlen_workspace_size(10, 2, 7, 1) == 0
    assert A.adaln_fwd_varlen_workspace_size(10, 2, 64, 1) > 0
    assert A.adaln_bwd_workspace_size(1, 1, 7, 1) == 0
    assert A.adaln_bwd_varlen_workspace_size(-1, 1, 1, 64, 1) == 0


def test_header_compiles_as_c_and_a_c_program_links(tmp_path):
    """include/adaln.h is a plain C header: a C99 program includes it, links libadaln and
    calls a host-only entry point."""
    import shutil
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    A.lib()  # the library is built
    src = tmp_path / "use_adaln.c"
    src.write_text('#include "adaln.h"\n'
                   "int main(void) {\n"
                   "    adaln_dtype d = ADALN_BF16;\n"
                   "    (void)d;\n"
                   "    return adaln_bucket_batch(256, 131072, 131072LL * 4096, 2) == 512 ? 0 : 1;\n"
                   "}\n")
    exe = tmp_path / "use_adaln"
    libdir = os.path.dirname(A.LIB_PATH)
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                    str(src), "-L", libdir, "-ladaln", "-Wl,-rpath," + libdir, "-o", str(exe)],
                   check=True, capture_output=True)
    assert subprocess.run([str(exe)]).returncode == 0
