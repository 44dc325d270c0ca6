"""Run a fast subset of the oracle pins against one oracle build (a .so).

Usage: python oracle_mutant_check.py LIB.so
Exit status 0 if every pin holds, 1 if one fails (a crash also counts as
detection).  Used by test_oracle_mutants.py on deliberately broken copies
of the oracle; the pins are the same facts as in test_oracle_*.py: the
nearest-code brute force, the hand-derived rows, the pairs where a
reciprocal multiply and a true division give different codes, the
slot-layout extents with padded and invalid slots, gather-then-insert equal
to direct publication, and the bf16 layout against numpy indexing.
"""

import ctypes
import os
import struct
import sys
from fractions import Fraction

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import hand_rows  # noqa: E402
from e4m3_ref import nearest_code, nearest_codes, rn_f32  # noqa: E402
from replication_token_warp_gb300 import inputs  # noqa: E402


def load(path):
    lib = ctypes.CDLL(path)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.kvo_e4m3_encode.argtypes = [ctypes.c_float]
    lib.kvo_e4m3_encode.restype = ctypes.c_uint8
    lib.kvo_quantize_tile.argtypes = [u16p, ctypes.c_int, u8p, ctypes.POINTER(ctypes.c_float)]
    lib.kvo_store_mla_fp8.argtypes = [u16p, ctypes.c_int64, u16p, ctypes.c_int64, u16p,
                                      ctypes.c_int64, i64p, ctypes.c_int64,
                                      ctypes.POINTER(u8p), ctypes.POINTER(u8p), ctypes.c_int,
                                      ctypes.c_int64, i64p]
    lib.kvo_store_mla_fp8.restype = ctypes.c_int64
    lib.kvo_gather_insert.argtypes = lib.kvo_store_mla_fp8.argtypes[:-1] + [u16p, i64p]
    lib.kvo_gather_insert.restype = ctypes.c_int64
    lib.kvo_store_mla_bf16.argtypes = lib.kvo_store_mla_fp8.argtypes
    lib.kvo_store_mla_bf16.restype = ctypes.c_int64
    return lib


def ptr(a, t):
    return a.ctypes.data_as(ctypes.POINTER(t))


def store(lib, lat, rope, idx, slots, R, nb, guard=0xA5, how="fp8"):
    """One oracle call: how = "fp8" (direct), "gather" (gather-then-insert)
    or "bf16" (the unquantised layout).  Returns (main, indexer, n, invalid)."""
    main_bytes, idx_bytes = (nb * 64 * 1152, nb * 64 * 256) if how == "bf16" else \
        (nb * 64 * 656, nb * 8448)
    main = [np.full(main_bytes, guard, np.uint8) for _ in range(R)]
    ixc = [np.full(idx_bytes, guard, np.uint8) for _ in range(R)]
    u8p = ctypes.POINTER(ctypes.c_uint8)
    mp = (u8p * R)(*[ptr(m, ctypes.c_uint8) for m in main])
    ip = (u8p * R)(*[ptr(x, ctypes.c_uint8) for x in ixc])
    lat, rope, idx = (np.ascontiguousarray(a) for a in (lat, rope, idx))
    slots = np.ascontiguousarray(slots, np.int64)
    inv = ctypes.c_int64()
    args = [ptr(lat, ctypes.c_uint16), lat.shape[1], ptr(rope, ctypes.c_uint16), rope.shape[1],
            ptr(idx, ctypes.c_uint16), idx.shape[1], ptr(slots, ctypes.c_int64), slots.shape[0],
            mp, ip, R, nb]
    if how == "gather":
        ws = np.empty(max(1, slots.shape[0]) * 704, np.uint16)
        n = lib.kvo_gather_insert(*args, ptr(ws, ctypes.c_uint16), ctypes.byref(inv))
    elif how == "bf16":
        n = lib.kvo_store_mla_bf16(*args, ctypes.byref(inv))
    else:
        n = lib.kvo_store_mla_fp8(*args, ctypes.byref(inv))
    return main, ixc, n, inv.value


def check_encoder(lib):
    v = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    got = np.array([lib.kvo_e4m3_encode(float(x)) for x in v.tolist()], np.uint8)
    with np.errstate(invalid="ignore"):
        want = nearest_codes(v.astype(np.float64))
    return np.array_equal(got, want)


def check_hand_rows(lib):
    for row in hand_rows.load()["rows"]:
        lat = hand_rows.build_bf16(row["latent"], 512)[None]
        rope = hand_rows.build_bf16(row["rope"], 64)[None]
        idx = hand_rows.build_bf16(row["index_k"], 128)[None]
        s = int(row["slot"])
        main, ixc, n, inv = store(lib, lat, rope, idx, np.array([s]), 1, 4)
        ex = row["expect"]
        m = main[0][s * 656:(s + 1) * 656]
        if not np.array_equal(m[:512], hand_rows.build_codes(ex["latent_codes"], 512)):
            return False
        scales = [int.from_bytes(m[512 + 4 * j:516 + 4 * j].tobytes(), "little") for j in range(4)]
        if scales != [int(b, 16) for b in ex["latent_scale_bits"]]:
            return False
        if m[528:].tobytes() != rope[0].astype("<u2").tobytes():
            return False
        blk, off = divmod(s, 64)
        b = ixc[0][blk * 8448:(blk + 1) * 8448]
        if not np.array_equal(b[off * 128:(off + 1) * 128],
                              hand_rows.build_codes(ex["index_codes"], 128)):
            return False
        if int.from_bytes(b[8192 + 4 * off:8196 + 4 * off].tobytes(), "little") != \
                int(ex["index_scale_bits"], 16):
            return False
    return True


def check_true_division(lib):
    import torch
    pos = (np.arange(0x0001, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    found = 0
    for amax_bits in range(0x3800, 0x4400, 3):
        a = np.float32((np.uint32(amax_bits) << 16).view(np.float32))
        s = np.float32(max(a, np.float32(1e-4))) / np.float32(448)
        x = pos[pos <= a]
        with np.errstate(all="ignore"):
            q_div, q_rcp = x / s, x * (np.float32(1) / s)
        differ = np.nonzero(q_div != q_rcp)[0]
        if differ.size == 0:
            continue
        c_div = torch.from_numpy(q_div[differ]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        c_rcp = torch.from_numpy(q_rcp[differ]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        for i in np.nonzero(c_div != c_rcp)[0]:
            xb = int(x.view(np.uint32)[differ[i]] >> 16)
            tile = np.zeros(128, np.uint16)
            tile[0], tile[1] = amax_bits, xb
            q = np.empty(128, np.uint8)
            sc = ctypes.c_float()
            lib.kvo_quantize_tile(ptr(tile, ctypes.c_uint16), 128, ptr(q, ctypes.c_uint8),
                                  ctypes.byref(sc))
            xv = struct.unpack("<f", struct.pack("<I", xb << 16))[0]
            if q[1] != nearest_code(rn_f32(Fraction(xv) / Fraction(float(sc.value)))):
                return False
            found += 1
            if found >= 16:
                return True
    return found > 0


def check_layout(lib):
    w = inputs.make(0)
    cap = w.num_blocks * 64
    slots = w.slot_mapping.copy()
    slots[[1, 4]] = [cap, -5]
    a_main, a_ix, n, inv = store(lib, w.kv_latent, w.k_rope, w.index_k, slots, 1, w.num_blocks,
                                 0xA5)
    b_main, b_ix, _, _ = store(lib, w.kv_latent, w.k_rope, w.index_k, slots, 1, w.num_blocks,
                               0x5A)
    em = np.zeros(cap * 656, bool)
    ei = np.zeros(w.num_blocks * 8448, bool)
    valid = [s for s in slots.tolist() if 0 <= s < cap]
    for s in valid:
        em[s * 656:(s + 1) * 656] = True
        blk, off = divmod(s, 64)
        ei[blk * 8448 + off * 128: blk * 8448 + (off + 1) * 128] = True
        ei[blk * 8448 + 8192 + 4 * off: blk * 8448 + 8196 + 4 * off] = True
    changed_m = (a_main[0] != 0xA5) | (b_main[0] != 0x5A)
    changed_i = (a_ix[0] != 0xA5) | (b_ix[0] != 0x5A)
    return (n == len(valid) and inv == 2 and np.array_equal(changed_m, em)
            and np.array_equal(changed_i, ei))


def _padded_workload():
    w = inputs.make(1)                      # decode batch: 64 rows, 4 padded
    slots = w.slot_mapping.copy()
    cap = w.num_blocks * 64
    slots[[3, 10]] = [cap + 7, -3]          # two invalid slots besides the padding
    return w, slots


def check_gather(lib):
    """Gather-then-insert leaves the same bytes and counts as direct
    publication, in every one of 3 replicas."""
    w, slots = _padded_workload()
    a = store(lib, w.kv_latent, w.k_rope, w.index_k, slots, 3, w.num_blocks)
    b = store(lib, w.kv_latent, w.k_rope, w.index_k, slots, 3, w.num_blocks, how="gather")
    if a[2:] != b[2:] or a[3] != 2:
        return False
    return all(np.array_equal(x, y) for x, y in zip(a[0] + a[1], b[0] + b[1]))


def check_bf16(lib):
    """bf16 layout: each written slot holds its row's little-endian bytes
    (Main = latent | rope at s * 1152, Indexer = index_k at s * 256), in
    every replica, and nothing else changes (two guard values)."""
    w, slots = _padded_workload()
    R, nb = 2, w.num_blocks
    a_main, a_ix, n, inv = store(lib, w.kv_latent, w.k_rope, w.index_k, slots, R, nb, 0xA5, "bf16")
    b_main, b_ix, _, _ = store(lib, w.kv_latent, w.k_rope, w.index_k, slots, R, nb, 0x5A, "bf16")
    ok = [t for t, s in enumerate(slots.tolist()) if 0 <= s < nb * 64]
    if n != len(ok) or inv != 2:
        return False
    want_main = np.full(nb * 64 * 1152, 0xA5, np.uint8).reshape(nb * 64, 1152)
    want_ix = np.full(nb * 64 * 256, 0xA5, np.uint8).reshape(nb * 64, 256)
    for t in ok:
        s = slots[t]
        want_main[s] = np.frombuffer(w.kv_latent[t].astype("<u2").tobytes() +
                                     w.k_rope[t].astype("<u2").tobytes(), np.uint8)
        want_ix[s] = np.frombuffer(w.index_k[t].astype("<u2").tobytes(), np.uint8)
    for r in range(R):
        if not (np.array_equal(a_main[r], want_main.ravel()) and
                np.array_equal(a_ix[r], want_ix.ravel())):
            return False
        changed = (a_main[r] != 0xA5) | (b_main[r] != 0x5A)
        if int(changed.sum()) != 1152 * len(ok):
            return False
    return True


def main(path):
    lib = load(path)
    for check in (check_encoder, check_hand_rows, check_true_division, check_layout,
                  check_gather, check_bf16):
        if not check(lib):
            print(f"pin failed: {check.__name__}")
            return 1
    print("all pins hold")
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1]))
