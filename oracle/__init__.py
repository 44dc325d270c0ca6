"""CPU oracle for the fused replicated KV-cache store.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library: the arithmetic lives in ``kvpub_oracle.c``
(scalar C, built here with gcc), and this module only builds it, loads it
with ctypes and marshals numpy arrays.

Every function follows "[Kernel][PCP] Publish replicated KV updates through
PyTorch symmetric memory" (vLLM #52863): Summary, the "AS-IS: gather then
insert" and "THIS PR: publish final rows directly" diagrams, and Design
(third bullet: final FP8 Main-KV and Indexer-K bytes).  The byte layout and
the quantisation rule are readings documented at the top of the C file.

Parity status: every function here is pinned by the tests in
``tests/test_oracle_*.py`` (closed forms, brute force over all bf16 inputs,
an independent library conversion, exact rational arithmetic, invariants).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvpub_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkvpub_oracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-Wall", "-Wextra"]

# Geometry of the stored bytes (the reading documented in kvpub_oracle.c).
LATENT_DIM = 512
ROPE_DIM = 64
INDEXER_DIM = 128
TILE = 128
BLOCK_SIZE = 64
MAIN_SLOT_BYTES = 656
INDEXER_SLOT_BYTES = 132
INDEXER_BLOCK_BYTES = BLOCK_SIZE * INDEXER_SLOT_BYTES
ROW_BF16 = LATENT_DIM + ROPE_DIM + INDEXER_DIM
MAIN_SLOT_BYTES_BF16 = 2 * (LATENT_DIM + ROPE_DIM)
INDEXER_SLOT_BYTES_BF16 = 2 * INDEXER_DIM

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build`` (gcc); return the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.kvo_e4m3_encode.argtypes = [ctypes.c_float]
        lib.kvo_e4m3_encode.restype = ctypes.c_uint8
        lib.kvo_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.kvo_e4m3_decode.restype = ctypes.c_double
        lib.kvo_quantize_tile.argtypes = [u16p, ctypes.c_int, u8p,
                                          ctypes.POINTER(ctypes.c_float)]
        lib.kvo_quantize_tile.restype = None
        common = [u16p, ctypes.c_int64, u16p, ctypes.c_int64, u16p, ctypes.c_int64,
                  i64p, ctypes.c_int64, ctypes.POINTER(u8p), ctypes.POINTER(u8p),
                  ctypes.c_int, ctypes.c_int64]
        lib.kvo_store_mla_fp8.argtypes = common + [i64p]
        lib.kvo_store_mla_fp8.restype = ctypes.c_int64
        lib.kvo_gather_insert.argtypes = common + [u16p, i64p]
        lib.kvo_gather_insert.restype = ctypes.c_int64
        lib.kvo_store_mla_bf16.argtypes = common + [i64p]
        lib.kvo_store_mla_bf16.restype = ctypes.c_int64
        _lib = lib
        return lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _as_bf16_bits(x: np.ndarray) -> np.ndarray:
    if x.dtype != np.uint16:
        raise TypeError("bf16 inputs are passed as their uint16 bit patterns")
    return x


def e4m3_encode(v: float) -> int:
    """One fp32 value -> its E4M3 code (RNE, saturating)."""
    return int(_load().kvo_e4m3_encode(float(v)))


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    """Element-wise e4m3_encode over a float32 array (scalar calls)."""
    lib = _load()
    flat = np.ascontiguousarray(v, dtype=np.float32).ravel()
    out = np.empty(flat.shape, dtype=np.uint8)
    enc = lib.kvo_e4m3_encode
    for i, x in enumerate(flat.tolist()):
        out[i] = enc(x)
    return out.reshape(np.shape(v))


def e4m3_decode(code: int) -> float:
    return float(_load().kvo_e4m3_decode(int(code) & 0xFF))


def quantize_tile(x_bits: np.ndarray):
    """One tile of bf16 bit patterns -> (codes uint8[n], scale float32)."""
    x = np.ascontiguousarray(_as_bf16_bits(x_bits))
    q = np.empty(x.shape[0], dtype=np.uint8)
    scale = ctypes.c_float()
    _load().kvo_quantize_tile(_ptr(x, ctypes.c_uint16), int(x.shape[0]),
                              _ptr(q, ctypes.c_uint8), ctypes.byref(scale))
    return q, np.float32(scale.value)


def _rows(x: np.ndarray, dim: int):
    x = _as_bf16_bits(x)
    if x.ndim != 2 or x.shape[1] < dim or x.strides[1] != 2:
        raise ValueError(f"expected [T, >= {dim}] bf16 rows with unit inner stride")
    return x, x.strides[0] // 2


def _cache_ptrs(caches):
    u8p = ctypes.POINTER(ctypes.c_uint8)
    arr = (u8p * len(caches))()
    for i, c in enumerate(caches):
        if c.dtype != np.uint8 or not c.flags.c_contiguous:
            raise TypeError("caches are contiguous uint8 arrays")
        arr[i] = _ptr(c, ctypes.c_uint8)
    return arr


def _check_caches(main_caches, indexer_caches, num_blocks):
    if len(main_caches) != len(indexer_caches) or not main_caches:
        raise ValueError("need the same number (>= 1) of Main and Indexer caches")
    for m, ix in zip(main_caches, indexer_caches):
        if m.nbytes < num_blocks * BLOCK_SIZE * MAIN_SLOT_BYTES:
            raise ValueError("Main cache too small")
        if ix.nbytes < num_blocks * INDEXER_BLOCK_BYTES:
            raise ValueError("Indexer cache too small")


def store_mla_fp8(kv_latent, k_rope, index_k, slot_mapping, main_caches,
                  indexer_caches, num_blocks):
    """Direct publication into every replica (modifies the caches in place).

    Returns (rows written per replica, invalid slot count).
    """
    lat, ls = _rows(kv_latent, LATENT_DIM)
    rope, rs = _rows(k_rope, ROPE_DIM)
    idx, ids = _rows(index_k, INDEXER_DIM)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T = slots.shape[0]
    if not (lat.shape[0] >= T and rope.shape[0] >= T and idx.shape[0] >= T):
        raise ValueError("fewer input rows than slot_mapping entries")
    _check_caches(main_caches, indexer_caches, num_blocks)
    inv = ctypes.c_int64()
    n = _load().kvo_store_mla_fp8(
        _ptr(lat, ctypes.c_uint16), ls, _ptr(rope, ctypes.c_uint16), rs,
        _ptr(idx, ctypes.c_uint16), ids, _ptr(slots, ctypes.c_int64), T,
        _cache_ptrs(main_caches), _cache_ptrs(indexer_caches), len(main_caches),
        int(num_blocks), ctypes.byref(inv))
    return int(n), int(inv.value)


def gather_insert(kv_latent, k_rope, index_k, slot_mapping, main_caches,
                  indexer_caches, num_blocks):
    """The unfused fallback: gather all rows, then insert once per replica."""
    lat, ls = _rows(kv_latent, LATENT_DIM)
    rope, rs = _rows(k_rope, ROPE_DIM)
    idx, ids = _rows(index_k, INDEXER_DIM)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T = slots.shape[0]
    _check_caches(main_caches, indexer_caches, num_blocks)
    ws = np.empty(max(T, 1) * ROW_BF16, dtype=np.uint16)
    inv = ctypes.c_int64()
    n = _load().kvo_gather_insert(
        _ptr(lat, ctypes.c_uint16), ls, _ptr(rope, ctypes.c_uint16), rs,
        _ptr(idx, ctypes.c_uint16), ids, _ptr(slots, ctypes.c_int64), T,
        _cache_ptrs(main_caches), _cache_ptrs(indexer_caches), len(main_caches),
        int(num_blocks), _ptr(ws, ctypes.c_uint16), ctypes.byref(inv))
    return int(n), int(inv.value)


def store_mla_bf16(kv_latent, k_rope, index_k, slot_mapping, main_caches, indexer_caches,
                   num_blocks):
    """Unquantised variant: the bf16 rows stored as they are into every
    replica (Main slot 1152 B, Indexer slot 256 B).  Returns (rows written
    per replica, invalid slot count)."""
    lat, ls = _rows(kv_latent, LATENT_DIM)
    rope, rs = _rows(k_rope, ROPE_DIM)
    idx, ids = _rows(index_k, INDEXER_DIM)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T = slots.shape[0]
    if not (lat.shape[0] >= T and rope.shape[0] >= T and idx.shape[0] >= T):
        raise ValueError("fewer input rows than slot_mapping entries")
    if len(main_caches) != len(indexer_caches) or not main_caches:
        raise ValueError("need the same number (>= 1) of Main and Indexer caches")
    for m, ix in zip(main_caches, indexer_caches):
        if (m.nbytes < num_blocks * BLOCK_SIZE * MAIN_SLOT_BYTES_BF16
                or ix.nbytes < num_blocks * BLOCK_SIZE * INDEXER_SLOT_BYTES_BF16):
            raise ValueError("cache too small")
    inv = ctypes.c_int64()
    n = _load().kvo_store_mla_bf16(
        _ptr(lat, ctypes.c_uint16), ls, _ptr(rope, ctypes.c_uint16), rs,
        _ptr(idx, ctypes.c_uint16), ids, _ptr(slots, ctypes.c_int64), T,
        _cache_ptrs(main_caches), _cache_ptrs(indexer_caches), len(main_caches),
        int(num_blocks), ctypes.byref(inv))
    return int(n), int(inv.value)


def new_caches_bf16(num_replicas: int, num_blocks: int, guard: int = 0xA5):
    """Fresh guard-filled host caches of the bf16 variant: (main, indexer)."""
    main = [np.full(num_blocks * BLOCK_SIZE * MAIN_SLOT_BYTES_BF16, guard, np.uint8)
            for _ in range(num_replicas)]
    idx = [np.full(num_blocks * BLOCK_SIZE * INDEXER_SLOT_BYTES_BF16, guard, np.uint8)
           for _ in range(num_replicas)]
    return main, idx


def new_caches(num_replicas: int, num_blocks: int, guard: int = 0xA5):
    """Fresh guard-filled host caches: (main list, indexer list)."""
    main = [np.full(num_blocks * BLOCK_SIZE * MAIN_SLOT_BYTES, guard, np.uint8)
            for _ in range(num_replicas)]
    idx = [np.full(num_blocks * INDEXER_BLOCK_BYTES, guard, np.uint8)
           for _ in range(num_replicas)]
    return main, idx
