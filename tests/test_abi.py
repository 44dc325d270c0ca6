"""The C-ABI library on the host: it builds, loads, exports every symbol the
public header declares, and its fail-closed validation rejects bad
arguments with the documented status before anything reaches a GPU.

Every call here has at least one invalid argument, so no call gets as far
as the CUDA runtime; the pointers are placeholders that are never
dereferenced.
"""

import ctypes
import os
import re

import pytest

from replication_token_warp_gb300 import build as kbuild
from replication_token_warp_gb300 import kvpub

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")

A = 0x10000          # 16-byte aligned placeholder address, never dereferenced


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kvpub.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = re.sub(r"#[^\n]*", "", text)
        names |= set(re.findall(r"\b(kvpub_\w+)\s*\(", text))
    return names


def test_header_declares_the_entry_points():
    want = {"kvpub_store_mla_fp8", "kvpub_store_mla_fp8_publish", "kvpub_store_mla_bf16",
            "kvpub_gather_insert",
            "kvpub_gather_workspace_bytes", "kvpub_epoch_advance", "kvpub_epoch_wait",
            "kvpub_last_error"}
    assert want <= declared_functions()


def test_library_exports_every_declared_symbol(lib):
    handle = ctypes.CDLL(kvpub.library_path())
    missing = [n for n in sorted(declared_functions()) if not hasattr(handle, n)]
    assert not missing
    assert set(declared_functions()) <= set(kvpub.SIGNATURES)


def test_workspace_bytes(lib):
    assert lib.kvpub_gather_workspace_bytes(0) == 0
    assert lib.kvpub_gather_workspace_bytes(-3) == 0
    assert lib.kvpub_gather_workspace_bytes(14336) == 14336 * 1408


def ptrs(n, base=A):
    arr = (ctypes.c_void_p * n)()
    for i in range(n):
        arr[i] = base + 0x100000 * (i + 1)
    return arr


def store_args(**over):
    a = dict(lat=A, ls=512, rope=A, rs=64, idx=A, is_=128, slots=A, T=16,
             mains=ptrs(2), idxs=ptrs(2), R=2, nb=4, bs=64, cnt=None)
    a.update(over)
    return [a["lat"], a["ls"], a["rope"], a["rs"], a["idx"], a["is_"], a["slots"], a["T"],
            a["mains"], a["idxs"], a["R"], a["nb"], a["bs"], a["cnt"]]


BAD = [
    ("R0", dict(R=0), 1),
    ("R9", dict(R=9, mains=ptrs(9), idxs=ptrs(9)), 3),
    ("block32", dict(bs=32), 1),
    ("negT", dict(T=-1), 1),
    ("nb0", dict(nb=0), 1),
    ("nb_huge", dict(nb=2 ** 62), 1),
    ("null_latent", dict(lat=None), 1),
    ("null_rope", dict(rope=None), 1),
    ("null_index", dict(idx=None), 1),
    ("null_slots", dict(slots=None), 1),
    ("misaligned_latent", dict(lat=A + 2), 2),
    ("misaligned_rope", dict(rope=A + 8), 2),
    ("misaligned_index", dict(idx=A + 4), 2),
    ("misaligned_slots", dict(slots=A + 4), 2),
    ("stride_not_x8", dict(ls=516), 2),
    ("stride_short", dict(rs=32), 1),
    ("null_cache_arrays", dict(mains=None), 1),
    ("null_cache", dict(idxs=(ctypes.c_void_p * 2)(A, None)), 1),
    ("misaligned_cache", dict(mains=(ctypes.c_void_p * 2)(A, A + 8)), 2),
    ("misaligned_counter", dict(cnt=A + 4), 2),
]


@pytest.mark.parametrize("name,over,status", BAD, ids=[b[0] for b in BAD])
def test_store_rejects_bad_arguments(lib, name, over, status):
    assert lib.kvpub_store_mla_fp8(*store_args(**over), None) == status
    assert kvpub.last_error() != ""
    assert lib.kvpub_gather_insert(*store_args(**over), A, 10 ** 9, None) == status
    assert lib.kvpub_store_mla_fp8_publish(*store_args(**over), A, A, None) == status
    assert lib.kvpub_store_mla_bf16(*store_args(**over), None) == status


def test_gather_rejects_small_or_missing_workspace(lib):
    assert lib.kvpub_gather_insert(*store_args(), A, 16 * 1408 - 1, None) == 5
    assert "workspace" in kvpub.last_error()
    assert lib.kvpub_gather_insert(*store_args(), None, 10 ** 9, None) == 5
    assert lib.kvpub_gather_insert(*store_args(), A + 8, 10 ** 9, None) == 2


def test_noalloc_rejects_bad_arguments_and_oversized_batches(lib):
    for name, over, status in BAD:
        assert lib.kvpub_gather_insert_noalloc(*store_args(**over), None) == status, name
    limit = kvpub.STATIC_GATHER_MAX_TOKENS
    assert lib.kvpub_gather_insert_noalloc(*store_args(T=limit + 1), None) == 5
    assert "static workspace limit" in kvpub.last_error()


def test_publish_rejects_bad_counters(lib):
    # invalid R keeps this call away from the GPU whatever the counters are
    assert lib.kvpub_store_mla_fp8_publish(*store_args(R=0), None, A, None) == 1
    assert lib.kvpub_store_mla_fp8_publish(*store_args(T=-1), A, None, None) == 1


def test_epoch_calls_reject_bad_arguments(lib):
    assert lib.kvpub_epoch_advance(None, None) == 1
    assert lib.kvpub_epoch_advance(A + 4, None) == 2
    assert lib.kvpub_epoch_wait(None, 1, 10, A, None) == 1
    assert lib.kvpub_epoch_wait(A, 1, 10, None, None) == 1
    assert lib.kvpub_epoch_wait(A + 4, 1, 10, A, None) == 2
    assert lib.kvpub_epoch_wait(A, 1, 0, A, None) == 1
    assert lib.kvpub_epoch_wait(A, 1, kvpub.MAX_POLLS + 1, A, None) == 1
    assert "max_polls" in kvpub.last_error()


def test_python_binding_raises_typed_errors(lib):
    with pytest.raises(kvpub.KvpubError) as e:
        kvpub.check(lib.kvpub_epoch_advance(None, None))
    assert e.value.status == 1 and "epoch" in e.value.message
