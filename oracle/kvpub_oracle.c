/*
 * kvpub oracle: a plain, slow, scalar CPU statement of the fused replicated
 * KV-cache store.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and
 * the benchmark's CPU-baseline leg are the only callers.  The GPU library
 * shares no code, header or table with this file.
 *
 * What it computes (sources, by page title and section):
 *  - "[Kernel][PCP] Publish replicated KV updates through PyTorch symmetric
 *    memory" (vLLM #52863), Summary and the "THIS PR: publish final rows
 *    directly" diagram: every producer quantises its final Main-KV and
 *    Indexer-K rows once and stores the final bytes into every replica.
 *  - same page, Design, third bullet: the cache-store writes final FP8
 *    Main-KV (fp8_ds_mla) and FP8 Indexer-K bytes.
 *  - same page, "Correctness and current-head validation": padded and
 *    invalid slots are handled and guard bytes are checked, so a skipped
 *    slot writes nothing and no byte outside a written slot row changes.
 *  - same page, "AS-IS: gather then insert" diagram: the fallback first
 *    gathers the update tensors, then each rank inserts the gathered rows
 *    into its own cache (kvo_gather_insert below).
 *
 * Readings where the pages are silent (all in fp32, as the workload states):
 *  - a quantisation tile is 128 consecutive elements; amax = max |x| over
 *    the tile; scale = max(amax, 1e-4f) / 448.0f (one correctly rounded
 *    fp32 division); every element is stored as e4m3(x / scale), the
 *    quotient again one correctly rounded fp32 division.
 *  - e4m3 is the OCP OFP8 E4M3 ("fn") format: bias 7, no infinities, the
 *    single NaN mantissa 111 at exponent 1111; conversion rounds to nearest
 *    with ties to the even code and saturates finite overflow and +-Inf to
 *    +-448; NaN encodes as 0x7F; the sign of zero is kept.
 *  - a tile that contains a NaN has a NaN amax (max propagates NaN), its
 *    scale is stored as the quiet NaN 0x7FFFFFFF and every code is 0x7F.
 *  - Main slot row (656 bytes): 512 fp8 codes of the latent, the 4 tile
 *    scales as little-endian fp32, then the 64 rope bf16 values copied
 *    verbatim (little-endian).
 *  - Indexer cache, per block of 64 slots (8448 bytes): 64 rows of 128 fp8
 *    codes, then 64 little-endian fp32 scales.
 *  - slot s is written iff 0 <= s < num_blocks * 64; -1 is padding; any
 *    other value is invalid, skipped and counted.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math (no contraction, so every
 * fp32 operation is one IEEE operation).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define KVO_LATENT_DIM 512
#define KVO_ROPE_DIM 64
#define KVO_INDEXER_DIM 128
#define KVO_TILE 128
#define KVO_BLOCK 64
#define KVO_MAIN_SLOT 656       /* 512 + 4*4 + 64*2 */
#define KVO_MAIN_SCALES_AT 512
#define KVO_MAIN_ROPE_AT 528
#define KVO_IDX_BLOCK 8448      /* 64 * (128 + 4) */
#define KVO_IDX_SCALES_AT 8192  /* 64 * 128 */
#define KVO_ROW_BF16 704        /* 512 + 64 + 128 bf16 values */

static float bits_to_f32(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t f32_to_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/* bf16 -> fp32 is exact: the 16 bits are the top half of the fp32 word. */
static float bf16_to_f32(uint16_t b) { return bits_to_f32((uint32_t)b << 16); }

/* Little-endian byte writers, independent of the host's byte order. */
static void put_le32(uint8_t *p, uint32_t v) {
    p[0] = (uint8_t)(v & 0xFFu);
    p[1] = (uint8_t)((v >> 8) & 0xFFu);
    p[2] = (uint8_t)((v >> 16) & 0xFFu);
    p[3] = (uint8_t)((v >> 24) & 0xFFu);
}

static void put_le16(uint8_t *p, uint16_t v) {
    p[0] = (uint8_t)(v & 0xFFu);
    p[1] = (uint8_t)((v >> 8) & 0xFFu);
}

/*
 * fp32 -> OCP E4M3 (fn) with round-to-nearest-even and saturation.
 *
 * Representable magnitudes: subnormals m * 2^-9 (m = 1..7) and normals
 * 2^E * (1 + m/8) for E = -6..8, excluding exponent field 15 with m = 7
 * (the NaN code), so the largest finite value is 448.  On [2^E, 2^(E+1))
 * the spacing of the grid is 2^(E-3); below 2^-6 it is 2^-9, the same as
 * the first normal binade.  The magnitude is divided by that spacing
 * (exact: a power of two, done in double), rounded to the nearest integer
 * with ties to even, and multiplied back.  Whatever lands at or above 448,
 * and every input >= 448 (Inf included), is the saturated code 0x7E.
 */
uint8_t kvo_e4m3_encode(float v) {
    if (v != v) return 0x7F;
    uint8_t sign = (f32_to_bits(v) >> 31) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a == 0.0) return sign;

    int e2;
    (void)frexp(a, &e2);          /* a = f * 2^e2 with f in [0.5, 1) */
    int E = e2 - 1;               /* floor(log2 a) */
    if (E < -6) E = -6;           /* subnormal range shares 2^-9 spacing */
    double spacing = ldexp(1.0, E - 3);
    double n = a / spacing;       /* exact */
    double r = floor(n);
    double frac = n - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    double val = r * spacing;
    if (val >= 448.0) return (uint8_t)(sign | 0x7E);
    if (val == 0.0) return sign;

    uint8_t code;
    if (val < ldexp(1.0, -6)) {
        code = (uint8_t)(val / ldexp(1.0, -9));   /* exponent field 0 */
    } else {
        int ev;
        double f = frexp(val, &ev);               /* val = f * 2^ev */
        int exp_unbiased = ev - 1;
        int mant = (int)((2.0 * f - 1.0) * 8.0);  /* exact: val on grid */
        code = (uint8_t)(((exp_unbiased + 7) << 3) | mant);
    }
    return (uint8_t)(sign | code);
}

/* E4M3 (fn) -> value, from the format definition (used by the tests). */
double kvo_e4m3_decode(uint8_t c) {
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) mag = ldexp((double)m, -9);
    else mag = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/*
 * One quantisation tile: amax over the tile, the tile scale, the codes.
 * x holds n bf16 values with element stride 1.
 */
void kvo_quantize_tile(const uint16_t *x, int n, uint8_t *q, float *scale_out) {
    float amax = 0.0f;
    int has_nan = 0;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(bf16_to_f32(x[i]));
        if (a != a) has_nan = 1;
        else if (a > amax) amax = a;
    }
    float scale;
    if (has_nan) {
        scale = bits_to_f32(0x7FFFFFFFu);
    } else {
        float m = (amax < 1e-4f) ? 1e-4f : amax;
        scale = m / 448.0f;
    }
    for (int i = 0; i < n; ++i) {
        float quotient = bf16_to_f32(x[i]) / scale;
        q[i] = kvo_e4m3_encode(quotient);
    }
    *scale_out = scale;
}

/* The final bytes of one token row: 656 Main bytes and 132 Indexer bytes. */
typedef struct {
    uint8_t main_row[KVO_MAIN_SLOT];
    uint8_t idx_codes[KVO_INDEXER_DIM];
    uint8_t idx_scale[4];
} kvo_row_bytes;

static void make_row_bytes(const uint16_t *latent, const uint16_t *rope,
                           const uint16_t *index_k, kvo_row_bytes *out) {
    for (int j = 0; j < KVO_LATENT_DIM / KVO_TILE; ++j) {
        float scale;
        kvo_quantize_tile(latent + j * KVO_TILE, KVO_TILE,
                          out->main_row + j * KVO_TILE, &scale);
        put_le32(out->main_row + KVO_MAIN_SCALES_AT + 4 * j, f32_to_bits(scale));
    }
    for (int i = 0; i < KVO_ROPE_DIM; ++i)
        put_le16(out->main_row + KVO_MAIN_ROPE_AT + 2 * i, rope[i]);
    float iscale;
    kvo_quantize_tile(index_k, KVO_INDEXER_DIM, out->idx_codes, &iscale);
    put_le32(out->idx_scale, f32_to_bits(iscale));
}

/* Place one row's final bytes at slot s of one replica. */
static void insert_row(const kvo_row_bytes *b, int64_t s, uint8_t *main_cache,
                       uint8_t *indexer_cache) {
    memcpy(main_cache + s * KVO_MAIN_SLOT, b->main_row, KVO_MAIN_SLOT);
    int64_t blk = s / KVO_BLOCK;
    int64_t off = s % KVO_BLOCK;
    uint8_t *block = indexer_cache + blk * KVO_IDX_BLOCK;
    memcpy(block + off * KVO_INDEXER_DIM, b->idx_codes, KVO_INDEXER_DIM);
    memcpy(block + KVO_IDX_SCALES_AT + off * 4, b->idx_scale, 4);
}

static int slot_is_written(int64_t s, int64_t num_slots) {
    return s >= 0 && s < num_slots;
}

/*
 * Direct publication: quantise every row once, store it into every replica.
 * Strides are in bf16 elements.  Returns the number of rows written (per
 * replica); *invalid_out (if not NULL) receives the count of slots that are
 * neither -1 nor in range.
 */
int64_t kvo_store_mla_fp8(const uint16_t *kv_latent, int64_t latent_stride,
                          const uint16_t *k_rope, int64_t rope_stride,
                          const uint16_t *index_k, int64_t index_stride,
                          const int64_t *slot_mapping, int64_t num_tokens,
                          uint8_t *const *main_caches,
                          uint8_t *const *indexer_caches, int num_replicas,
                          int64_t num_blocks, int64_t *invalid_out) {
    int64_t num_slots = num_blocks * KVO_BLOCK;
    int64_t written = 0, invalid = 0;
    kvo_row_bytes b;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (!slot_is_written(s, num_slots)) {
            if (s != -1) ++invalid;
            continue;
        }
        make_row_bytes(kv_latent + t * latent_stride, k_rope + t * rope_stride,
                       index_k + t * index_stride, &b);
        for (int r = 0; r < num_replicas; ++r)
            insert_row(&b, s, main_caches[r], indexer_caches[r]);
        ++written;
    }
    if (invalid_out) *invalid_out = invalid;
    return written;
}

/*
 * Gather then insert: step 1 collects every token's bf16 update row into
 * the workspace (latent | rope | index_k, 704 values per row); step 2, once
 * per replica, quantises each gathered row whose slot is written and
 * inserts it.  The bytes it leaves equal kvo_store_mla_fp8's.
 * workspace must hold num_tokens * 704 uint16 values.
 */
int64_t kvo_gather_insert(const uint16_t *kv_latent, int64_t latent_stride,
                          const uint16_t *k_rope, int64_t rope_stride,
                          const uint16_t *index_k, int64_t index_stride,
                          const int64_t *slot_mapping, int64_t num_tokens,
                          uint8_t *const *main_caches,
                          uint8_t *const *indexer_caches, int num_replicas,
                          int64_t num_blocks, uint16_t *workspace,
                          int64_t *invalid_out) {
    for (int64_t t = 0; t < num_tokens; ++t) {
        uint16_t *w = workspace + t * KVO_ROW_BF16;
        memcpy(w, kv_latent + t * latent_stride, KVO_LATENT_DIM * 2);
        memcpy(w + KVO_LATENT_DIM, k_rope + t * rope_stride, KVO_ROPE_DIM * 2);
        memcpy(w + KVO_LATENT_DIM + KVO_ROPE_DIM, index_k + t * index_stride,
               KVO_INDEXER_DIM * 2);
    }
    int64_t num_slots = num_blocks * KVO_BLOCK;
    int64_t written = 0, invalid = 0;
    kvo_row_bytes b;
    for (int r = 0; r < num_replicas; ++r) {
        for (int64_t t = 0; t < num_tokens; ++t) {
            int64_t s = slot_mapping[t];
            if (!slot_is_written(s, num_slots)) {
                if (r == 0 && s != -1) ++invalid;
                continue;
            }
            const uint16_t *w = workspace + t * KVO_ROW_BF16;
            make_row_bytes(w, w + KVO_LATENT_DIM, w + KVO_LATENT_DIM + KVO_ROPE_DIM,
                           &b);
            insert_row(&b, s, main_caches[r], indexer_caches[r]);
            if (r == 0) ++written;
        }
    }
    if (invalid_out) *invalid_out = invalid;
    return written;
}

/*
 * Unquantised (bf16) cache variant of direct publication: the same rows,
 * slots and replicas, with the bytes stored as they arrive.  Covers the BF16
 * main/indexer cache cases of "[Feature][KV Connector] Support QSA HiSparse
 * in disaggregated serving", Validation.  Reading of the slot layout:
 *   Main slot (1152 bytes) = 512 latent bf16 | 64 rope bf16, little-endian,
 *   at s * 1152;  Indexer slot (256 bytes) = 128 bf16 at s * 256.
 */
#define KVO_MAIN_SLOT_BF16 1152
#define KVO_IDX_SLOT_BF16 256

int64_t kvo_store_mla_bf16(const uint16_t *kv_latent, int64_t latent_stride,
                           const uint16_t *k_rope, int64_t rope_stride,
                           const uint16_t *index_k, int64_t index_stride,
                           const int64_t *slot_mapping, int64_t num_tokens,
                           uint8_t *const *main_caches,
                           uint8_t *const *indexer_caches, int num_replicas,
                           int64_t num_blocks, int64_t *invalid_out) {
    int64_t num_slots = num_blocks * KVO_BLOCK;
    int64_t written = 0, invalid = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (!slot_is_written(s, num_slots)) {
            if (s != -1) ++invalid;
            continue;
        }
        for (int r = 0; r < num_replicas; ++r) {
            uint8_t *m = main_caches[r] + s * KVO_MAIN_SLOT_BF16;
            for (int i = 0; i < KVO_LATENT_DIM; ++i)
                put_le16(m + 2 * i, kv_latent[t * latent_stride + i]);
            for (int i = 0; i < KVO_ROPE_DIM; ++i)
                put_le16(m + 2 * KVO_LATENT_DIM + 2 * i, k_rope[t * rope_stride + i]);
            uint8_t *x = indexer_caches[r] + s * KVO_IDX_SLOT_BF16;
            for (int i = 0; i < KVO_INDEXER_DIM; ++i)
                put_le16(x + 2 * i, index_k[t * index_stride + i]);
        }
        ++written;
    }
    if (invalid_out) *invalid_out = invalid;
    return written;
}
