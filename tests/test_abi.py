"""Host-side checks of the C-ABI (CPU only): the library loads, exports every
declared symbol, and rejects bad arguments before touching the GPU."""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ctr.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ctr_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from sparse_embeddings_feature_gb300 import ctr
    return ctr.lib()


def test_header_declares_the_path():
    names = declared_functions()
    for must in ("ctr_dedup", "ctr_embedding_bag_fwd", "ctr_embedding_bag_bwd_update", "ctr_dot_interaction",
                 "ctr_dot_interaction_bwd", "ctr_gather_rows", "ctr_check_status"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_library_is_sm103a_and_links_no_oracle(lib):
    from sparse_embeddings_feature_gb300 import ctr
    path = ctr.library_path()
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    assert "oracle_" not in out
    # the build compiles for sm_103a only, and the library on disk is the one those flags made
    from sparse_embeddings_feature_gb300 import build as B
    assert B.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert open(os.path.join(B.OUT_DIR, "fingerprint")).read() == B._fingerprint(
        os.environ.get("CTR_NVCC_EXTRA", "").split())


def test_status_strings(lib):
    from sparse_embeddings_feature_gb300 import ctr
    assert ctr.status_string(0) == "CTR_OK"
    assert ctr.status_string(-4) == "CTR_ERR_INDEX_OUT_OF_RANGE"
    assert ctr.status_string(-8) == "CTR_ERR_BAD_OFFSETS"
    assert lib.ctr_version() >= 100


def test_workspace_sizes_grow_with_the_batch(lib):
    from sparse_embeddings_feature_gb300 import ctr
    a = ctr.ctr_dedup_workspace_size(1000, 26, 10, 26 * 8_000_000)
    b = ctr.ctr_dedup_workspace_size(1_000_000, 26, 10, 26 * 8_000_000)
    assert 0 < a < b
    assert ctr.ctr_bwd_update_workspace_size(1000, 128) < ctr.ctr_bwd_update_workspace_size(10 ** 6, 128)
    assert ctr.ctr_embedding_bag_workspace_size() == 256
    assert ctr.ctr_interaction_workspace_size() == 256


def test_host_validation_rejects_bad_arguments(lib):
    # every case fails in host-side validation, before any CUDA call
    null = None
    b2t = (C.c_int32 * 1)(0)
    rb = (C.c_int64 * 2)(0, 10)
    bad_rb = (C.c_int64 * 2)(1, 10)
    st = lib.ctr_dedup(null, null, 1, 1, b2t, rb, 1, 0, null, null, null, null, null, null, null, null, 0, null)
    assert st == -1                                     # offsets / outputs missing
    dummy = C.c_void_p(256)
    st = lib.ctr_dedup(dummy, dummy, 1, 1, b2t, bad_rb, 1, 1, dummy, dummy, null, null, null, null, null, dummy,
                       1 << 20, null)
    assert st == -1                                     # row_base[0] != 0
    st = lib.ctr_dedup(dummy, dummy, 1000, 1, None, rb, 1, 1, dummy, dummy, null, null, null, null, null, dummy,
                       1 << 20, null)
    assert st == -1                                     # no bag_to_table
    st = lib.ctr_dedup(dummy, dummy, 1, 1, b2t, rb, 1, 1 << 31, dummy, dummy, null, null, null, null, null, dummy,
                       1 << 20, null)
    assert st == -2                                     # n_ids beyond int32 positions
    st = lib.ctr_dedup(dummy, dummy, 1, 1, b2t, rb, 1, 5, dummy, dummy, null, null, null, null, null, dummy, 16, null)
    assert st == -3                                     # workspace too small
    for phases in (0, 4):
        st = lib.ctr_dedup_phases(dummy, dummy, 1, 1, b2t, rb, 1, 5, dummy, dummy, null, null, null, null, null,
                                  phases, dummy, 1 << 20, null)
        assert st == -1                                 # no such part of the dedup
    st = lib.ctr_embedding_bag_fwd(dummy, 7, 16, 10, dummy, 0, 4, dummy, 1, 1, b2t, rb, 1, 0, dummy, 0, 16, 16,
                                   dummy, 256, null)
    assert st == -1                                     # bad dtype
    st = lib.ctr_embedding_bag_fwd(dummy, 0, 16, 10, dummy, 0, 4, dummy, 1, 1, b2t, rb, 1, 0, dummy, 0, 16, 16,
                                   C.c_void_p(100), 256, null)
    assert st == -3                                     # misaligned workspace
    st = lib.ctr_dot_interaction(null, 0, 4, 3, 8, dummy, dummy, 256, null)
    assert st == -1
    st = lib.ctr_embedding_bag_bwd_update(dummy, 16, 16, dummy, 1, 1, 0, dummy, dummy, dummy, dummy, 10, C.c_float(0.1),
                                          dummy, 0, 6, 10, null, dummy, 1 << 30, null)
    assert st == -2                                     # d not a multiple of 4
    st = lib.ctr_fill_table(null, 0, 10, 4, 0, 0, 1, C.c_float(1.0), null)
    assert st == -1


def test_product_code_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "sparse_embeddings_feature_gb300")
    pat = re.compile(r"^\s*(from\s+oracle|import\s+oracle)|liboracle|oracle\.oracle|oracle_[a-z]+\(", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not pat.search(text), f


def test_static_dedup_array_covers_every_row_count_at_its_id_limit(lib):
    # the allocation-free dedup keeps its scratch in a 48 MB array and accepts up to
    # 2^20 IDs: the dedup's workspace at 2^20 IDs must fit for any total row count
    # (it peaks on the presence-bitmap path at total rows = 64 x IDs)
    from sparse_embeddings_feature_gb300 import ctr
    n = 1 << 20
    static_bytes = 48 << 20
    counts = {1, 2, 1000, 64 * n - 1, 64 * n, 64 * n + 1, 1 << 32}
    counts |= {int(x) for x in __import__("numpy").geomspace(2, 1 << 32, 2000)}
    sizes = {t: ctr.ctr_dedup_workspace_size(n, 26, 131072, t) for t in counts}
    worst = max(sizes, key=sizes.get)
    assert sizes[worst] <= static_bytes, (worst, sizes[worst])
    assert worst == 64 * n
    st = lib.ctr_dedup_static(C.c_void_p(256), C.c_void_p(256), 1, 1, (C.c_int32 * 1)(0), (C.c_int64 * 2)(0, 10), 1,
                              C.c_int64(n + 1), None, None, None, None, None, None, None, None, None)
    assert st == -2                                     # beyond 2^20 IDs: refused before any CUDA call
