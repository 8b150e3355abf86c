"""The C-ABI library loads, exports every function its header declares, and
rejects bad host-side arguments before touching the GPU (no compute calls)."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from speculative_decode_mla_tree_gb300 import abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build_library()
    return abi.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "mla_tree.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(?:int|size_t|const char\*)\s+(\w+)\s*\(", src)))


def test_header_declares_the_abi():
    names = _declared()
    assert set(names) == set(abi.EXPORTS), names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def _signatures():
    """name -> (return type, [parameter types]) for every declaration."""
    src = open(os.path.join(ROOT, "include", "mla_tree.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for ret, name, params in re.findall(r"\b(int|size_t|const char\*)\s+(\w+)\s*\(([^)]*)\)\s*;", src):
        params = " ".join(params.split())
        types = [] if params in ("", "void") else [p.rsplit(" ", 1)[0].strip() for p in params.split(",")]
        out[name] = (ret, types)
    return out


def _ctype_of(c_type):
    """The ctypes class a C parameter type is passed as."""
    if "*" in c_type or c_type == "mt_stream_t":
        return ctypes.c_void_p
    return {"int": ctypes.c_int, "int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t,
            "float": ctypes.c_float}[c_type.replace("const ", "")]


def test_binding_matches_header_signatures(lib):
    """Every binding passes exactly the header's parameters, each with a
    ctypes type of the right width, and reads the right return type."""
    sigs = _signatures()
    assert set(sigs) == set(abi.EXPORTS)
    for name, (ret, types) in sigs.items():
        fn = getattr(lib, name)
        want_ret = {"int": ctypes.c_int, "size_t": ctypes.c_size_t, "const char*": ctypes.c_char_p}[ret]
        assert fn.restype is want_ret, name
        if name == "mla_tree_abi_version":
            continue  # no parameters; ctypes keeps its default argtypes
        assert fn.argtypes is not None and len(fn.argtypes) == len(types), (name, types)
        for i, (got, c_type) in enumerate(zip(fn.argtypes, types)):
            assert got is _ctype_of(c_type), (name, i, c_type, got)


def test_version_and_status_strings(lib):
    assert lib.mla_tree_abi_version() == 100
    for code in (0, -1, -2, -3, -4):
        assert lib.mla_tree_status_string(code).decode() not in ("", "unknown status")


def test_host_argument_checks(lib):
    null = None
    # verify: zero heads, negative sizes, bad path, non-finite scale
    args = [null, null, 0, null, 0, null, null, null, 0, null, 1, 1, 0, 1.0,
            null, null, null, 0, 0, 0, null, null]
    assert lib.mla_tree_verify(*args) == abi.MT_EINVAL
    args[12] = 8; args[19] = 3
    assert lib.mla_tree_verify(*args) == abi.MT_EINVAL
    args[19] = 0; args[13] = float("nan")
    assert lib.mla_tree_verify(*args) == abi.MT_EINVAL
    args[13] = 1.0; args[18] = 5000
    assert lib.mla_tree_verify(*args) == abi.MT_EINVAL
    # empty batch is a successful no-op
    args[18] = 0; args[10] = 0
    assert lib.mla_tree_verify(*args) == abi.MT_OK
    # null pointers with work to do
    args[10] = 1
    assert lib.mla_tree_verify(*args) == abi.MT_EINVAL
    # misaligned q (odd address) with otherwise plausible pointers
    fake = 4096
    args2 = [fake + 2, fake, 10, fake, 10, fake, fake, fake, 10, fake, 1, 1, 8, 1.0,
             fake, fake, fake, 1 << 20, 0, 0, null, null]
    assert lib.mla_tree_verify(*args2) == abi.MT_EINVAL
    # misaligned / too small workspace
    args2[0] = fake; args2[16] = fake + 8
    assert lib.mla_tree_verify(*args2) == abi.MT_EWORKSPACE
    args2[16] = fake; args2[17] = 16
    assert lib.mla_tree_verify(*args2) == abi.MT_EWORKSPACE
    # marshaling entry points
    assert lib.mla_tree_draft_kv_scatter(null, 100, null, 1, null, 10, null, null) == abi.MT_EINVAL
    assert lib.mla_tree_draft_kv_scatter(null, 576, null, 0, null, 10, null, null) == abi.MT_OK
    assert lib.mla_tree_kv_indices_build(null, 0, null, null, null, -1, 0, null, 0, null, null, null) == abi.MT_EINVAL
    assert lib.mla_tree_kv_indices_build(null, 0, null, null, null, 2, 4, null, 0, null, null, null) == abi.MT_EINVAL
    assert lib.tree_mask_pack(null, null, null, 0, 0, null, null, 0, null, null) == abi.MT_OK
    assert lib.tree_mask_pack(null, null, null, 1, 3, null, null, 0, null, null) == abi.MT_EINVAL
    assert lib.tree_mask_pack_bits(null, null, null, 0, 0, null, null, 0, null, null) == abi.MT_OK
    assert lib.tree_mask_pack_bits(null, null, null, 1, 3, null, null, 0, null, null) == abi.MT_EINVAL
    # fused marshaling: short row stride, null pointers, misaligned draft rows
    prep = [fake, 576, fake, fake, 4, fake, fake, fake, 1, 2, fake, 10, fake, 16, fake, fake, fake, 8,
            null, null]
    bad = list(prep); bad[1] = 100
    assert lib.mla_tree_prepare(*bad) == abi.MT_EINVAL
    bad = list(prep); bad[7] = null
    assert lib.mla_tree_prepare(*bad) == abi.MT_EINVAL
    bad = list(prep); bad[0] = fake + 8
    assert lib.mla_tree_prepare(*bad) == abi.MT_EINVAL
    bad = list(prep); bad[1] = 580
    assert lib.mla_tree_prepare(*bad) == abi.MT_EINVAL
    bad = list(prep); bad[8] = 0
    assert lib.mla_tree_prepare(*bad) == abi.MT_OK
    # validate mode: negative tolerance, missing diff, short workspace
    val = list(args2[:18]) + [0, 1e-2, fake, null, null]
    val[16] = fake; val[17] = 1 << 30
    bad = list(val); bad[19] = -1.0
    assert lib.mla_tree_verify_validate(*bad) == abi.MT_EINVAL
    bad = list(val); bad[20] = null
    assert lib.mla_tree_verify_validate(*bad) == abi.MT_EINVAL
    bad = list(val); bad[17] = 256
    assert lib.mla_tree_verify_validate(*bad) == abi.MT_EWORKSPACE
    assert (lib.mla_tree_verify_validate_workspace_bytes(2, 32, 8, 4) >
            lib.mla_tree_verify_workspace_bytes(2, 32, 8, 4) + 32 * 8 * 1024)
    # bit-form verify shares the verify checks
    args3 = list(args2); args3[16] = fake; args3[17] = 16
    assert lib.mla_tree_verify_bits(*args3) == abi.MT_EWORKSPACE
    args3[12] = 0
    assert lib.mla_tree_verify_bits(*args3) == abi.MT_EINVAL
    # the flags form: unknown flag bits, a misaligned word mask, then the
    # shared checks
    args4 = list(args2[:10]) + [abi.MASK_SKIP_PREFIX] + list(args2[10:])
    args4[17] = fake; args4[18] = 16
    assert lib.mla_tree_verify_masked(*args4) == abi.MT_EWORKSPACE
    bad = list(args4); bad[10] = 4
    assert lib.mla_tree_verify_masked(*bad) == abi.MT_EINVAL
    bad = list(args4); bad[10] = abi.MASK_BITS | abi.MASK_SKIP_PREFIX; bad[7] = fake + 2
    assert lib.mla_tree_verify_masked(*bad) == abi.MT_EINVAL


def test_workspace_size_grows_with_splits(lib):
    a = lib.mla_tree_verify_workspace_bytes(8, 128, 8, 1)
    b = lib.mla_tree_verify_workspace_bytes(8, 128, 8, 64)
    assert 0 < a < b
    assert b >= 64 * 128 * 8 * 513 * 4
    assert lib.mla_tree_verify_workspace_bytes(8, 128, 8, 5000) == 0


def test_unsplit_workspace_holds_no_partials(lib):
    """max_splits 1 (and the automatic choice when the rows alone fill the
    GPU, e.g. 32 requests x 64 nodes x 64 heads) needs only the per-token
    split counts: no kernel writes a partial then."""
    assert lib.mla_tree_verify_workspace_bytes(32, 2048, 64, 1) <= 2048 * 4 + 256
    assert lib.mla_tree_verify_workspace_bytes(32, 2048, 64, 0) <= 2048 * 4 + 256
    two = lib.mla_tree_verify_workspace_bytes(32, 2048, 64, 2)
    assert two >= 2 * 2048 * 64 * 513 * 4


def test_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(abi.MlaTreeError):
        abi._ptr(torch.zeros(4), None, "x")


def test_wait_limit_hook_arguments(lib):
    assert lib.mla_tree_test_wait_limits(-2, 0) == abi.MT_EINVAL
    assert lib.mla_tree_test_wait_limits(-1, -1) == abi.MT_EINVAL
    assert lib.mla_tree_test_wait_limits(3, 1000) == abi.MT_OK
    assert lib.mla_tree_test_wait_limits(-1, 0) == abi.MT_OK


def test_launch_count_many_requests(lib):
    """The tensor-core path takes any number of requests, in launches of at
    most 256 (plus the merge when splits are possible)."""
    assert lib.mla_tree_verify_launch_count(256, 256 * 16, 8, 100000, 1, 2) == 1
    assert lib.mla_tree_verify_launch_count(257, 257 * 16, 8, 100000, 1, 2) == 2
    assert lib.mla_tree_verify_launch_count(600, 600 * 16, 8, 100000, 4, 2) == 4


def test_launch_count_short_rows_need_no_merge(lib):
    """The warp-shuffle kernel splits a request across the grid only beyond
    256 keys: a call whose kv_indices are no longer launches one kernel."""
    assert lib.mla_tree_verify_launch_count(1, 9, 8, 30, 0, 0) == 1      # the live 9-node shape
    assert lib.mla_tree_verify_launch_count(1, 9, 8, 30, 64, 1) == 1
    assert lib.mla_tree_verify_launch_count(1, 9, 8, 5000, 64, 1) == 2
    assert lib.mla_tree_verify_launch_count(1, 9, 8, 5000, 1, 1) == 1
