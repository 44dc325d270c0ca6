"""The oracle's pins catch plausible mistakes: each mutant below is a copy of
oracle/kvpub_oracle.c with one planted error, built here with the oracle's
own compiler flags and checked by oracle_mutant_check.py in a subprocess
(a crash counts as caught).  The unmodified oracle must pass the same
checks, so a mutant's failure is the mistake's doing.

Mistakes planted (all on the CPU, in the oracle only): a wrong scale divisor,
a wrong floor, multiplying by a reciprocal, ties rounded up, truncation, a
dropped sign, the subnormal spacing, the Main-row field order, interleaved
Indexer rows, an Indexer-scale offset, an amax taken across tile borders,
ignoring NaN, an off-by-one slot bound, counting padding as invalid; in
gather-then-insert a shifted workspace field, inserting into the first
replica only and counting invalid slots once per replica; in the bf16
layout a wrong Main or Indexer slot stride and the rope written over the
latent.
"""

import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
CHECK = os.path.join(HERE, "oracle_mutant_check.py")

MUTANTS = {
    "scale_divisor_447": ("scale = m / 448.0f;", "scale = m / 447.0f;"),
    "floor_1e-3": ("(amax < 1e-4f) ? 1e-4f : amax", "(amax < 1e-3f) ? 1e-3f : amax"),
    "reciprocal_multiply": ("float quotient = bf16_to_f32(x[i]) / scale;",
                            "float quotient = bf16_to_f32(x[i]) * (1.0f / scale);"),
    "ties_up": ("if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;",
                "if (frac >= 0.5) r += 1.0;"),
    "truncate": ("if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;", ""),
    "drop_sign": ("uint8_t sign = (f32_to_bits(v) >> 31) ? 0x80 : 0x00;", "uint8_t sign = 0;"),
    "subnormal_spacing": ("if (E < -6) E = -6;", "if (E < -7) E = -7;"),
    "fields_swapped": ("#define KVO_MAIN_SCALES_AT 512\n#define KVO_MAIN_ROPE_AT 528",
                       "#define KVO_MAIN_SCALES_AT 640\n#define KVO_MAIN_ROPE_AT 512"),
    "indexer_interleaved": ("memcpy(block + off * KVO_INDEXER_DIM, b->idx_codes, KVO_INDEXER_DIM);",
                            "memcpy(indexer_cache + s * 132, b->idx_codes, KVO_INDEXER_DIM);"),
    "indexer_scale_offset": ("memcpy(block + KVO_IDX_SCALES_AT + off * 4, b->idx_scale, 4);",
                             "memcpy(block + KVO_IDX_SCALES_AT + off * 4 + (off < 63 ? 4 : 0), "
                             "b->idx_scale, 4);"),
    "amax_across_tiles": ("kvo_quantize_tile(latent + j * KVO_TILE, KVO_TILE,",
                          "kvo_quantize_tile(latent + j * KVO_TILE, KVO_TILE + (j < 3 ? 1 : 0),"),
    "nan_ignored": ("if (has_nan) {", "if (0) {"),
    "slot_bound_off_by_one": ("return s >= 0 && s < num_slots;", "return s >= 0 && s <= num_slots;"),
    "gather_workspace_rope_shifted": ("memcpy(w + KVO_LATENT_DIM, k_rope + t * rope_stride",
                                      "memcpy(w + KVO_LATENT_DIM + 1, k_rope + t * rope_stride"),
    "gather_first_replica_only": ("insert_row(&b, s, main_caches[r], indexer_caches[r]);",
                                  "insert_row(&b, s, main_caches[0], indexer_caches[0]);"),
    "gather_invalid_per_replica": ("if (r == 0 && s != -1) ++invalid;", "if (s != -1) ++invalid;"),
    "bf16_main_stride": ("uint8_t *m = main_caches[r] + s * KVO_MAIN_SLOT_BF16;",
                         "uint8_t *m = main_caches[r] + s * 1024;"),
    "bf16_rope_before_latent": ("put_le16(m + 2 * KVO_LATENT_DIM + 2 * i, k_rope[t * rope_stride + i]);",
                                "put_le16(m + 2 * i, k_rope[t * rope_stride + i]);"),
    "bf16_indexer_stride": ("uint8_t *x = indexer_caches[r] + s * KVO_IDX_SLOT_BF16;",
                            "uint8_t *x = indexer_caches[r] + s * 128;"),
    "padding_counted": ("if (s != -1) ++invalid;\n            continue;\n        }\n"
                        "        make_row_bytes(kv_latent",
                        "++invalid;\n            continue;\n        }\n        make_row_bytes(kv_latent"),
}


def _build(src_text, out_dir, name):
    c = os.path.join(out_dir, f"{name}.c")
    so = os.path.join(out_dir, f"lib{name}.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *oracle._CFLAGS, "-o", so, c, "-lm"], check=True,
                   capture_output=True)
    return so


def _check(so):
    return subprocess.run([sys.executable, CHECK, so], capture_output=True, text=True,
                          timeout=300)


@pytest.fixture(scope="module")
def source():
    with open(oracle._SRC) as f:
        return f.read()


def test_unmodified_oracle_passes_the_checks(source, tmp_path):
    res = _check(_build(source, str(tmp_path), "original"))
    assert res.returncode == 0, res.stdout + res.stderr


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(source, tmp_path, name):
    old, new = MUTANTS[name]
    assert old in source, f"mutation site of {name} no longer exists"
    res = _check(_build(source.replace(old, new, 1), str(tmp_path), name))
    assert res.returncode != 0, f"mutant {name} passed every pin"
