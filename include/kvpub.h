/*
 * kvpub: fused replicated KV-cache store for GB300 (sm_103a).
 *
 * The operation is the direct publication described on "[Kernel][PCP]
 * Publish replicated KV updates through PyTorch symmetric memory" (vLLM
 * #52863), Summary and the "THIS PR: publish final rows directly" diagram.
 * Each producer quantises its final Main-KV and Indexer-K rows once, then
 * stores the final FP8 bytes into every replica of the paged cache (Design,
 * third bullet). That replaces the "AS-IS: gather then insert" path, which
 * is kept here as kvpub_gather_insert. All R replicas live in this GPU's own
 * memory.
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument is a device pointer unless its comment says
 *    "host".
 *  - The caller owns and allocates all memory: inputs, caches, workspace and
 *    counters. The one exception is kvpub_gather_insert_noalloc, whose
 *    workspace is a fixed array inside the library. These entry points
 *    allocate nothing and never synchronise. Their only state is the calling
 *    thread's last error message and, per device, cached launch geometry
 *    (SM count, resident blocks per kernel).
 *  - Work is enqueued on `stream`. NULL means the legacy default stream.
 *  - kvpub_store_mla_fp8, kvpub_store_mla_bf16, kvpub_store_mla_fp8_publish,
 *    kvpub_gather_insert, kvpub_epoch_advance and kvpub_epoch_wait may be
 *    captured into a CUDA graph. Kernel parameters hold the pointers by
 *    value, so a replay reuses the same buffers.
 *  - Validation is fail-closed. Every check runs on the host before
 *    anything is enqueued. On any validation error nothing is launched, no
 *    byte changes, and kvpub_last_error() says why.
 *  - KVPUB_ERR_CUDA means the CUDA runtime refused a launch (or the device
 *    query before it). A single-launch call then has enqueued nothing.
 *    kvpub_gather_insert and kvpub_gather_insert_noalloc enqueue 1 + R
 *    launches in turn and stop at the first refusal, so the launches before
 *    it may already be on the stream. The stream is then in an error state
 *    that the caller must handle anyway.
 *
 * Byte layout of one slot. The pages name the format (fp8_ds_mla Main-KV,
 * FP8 Indexer-K) but not its bytes. The reading used here is this:
 *  - Quantisation: tiles of 128 consecutive elements. Per tile,
 *    amax = max |x|, and scale = max(amax, 1e-4f) / 448.0f is one correctly
 *    rounded fp32 division. Each element is stored as the E4M3 (OCP "fn")
 *    code of x / scale: another correctly rounded fp32 division, then
 *    round-to-nearest-even with saturation to +-448. Signed zero is kept,
 *    and NaN encodes as 0x7F.
 *  - A NaN anywhere in a tile makes its scale the quiet NaN 0x7FFFFFFF and
 *    all of its codes 0x7F.
 *  - Main cache: num_blocks * 64 slots of KVPUB_MAIN_SLOT_BYTES = 656 bytes,
 *    slot s at byte s * 656. The row holds:
 *      [0, 512)   E4M3 codes of the 512 latent values (4 tiles);
 *      [512, 528) the 4 tile scales, little-endian fp32;
 *      [528, 656) the 64 rope bf16 values, copied verbatim.
 *  - Indexer cache: num_blocks blocks of KVPUB_INDEXER_BLOCK_BYTES = 8448
 *    bytes (132 per slot). Slot s = 64 * blk + off is stored as:
 *      byte blk*8448 + off*128        the 128 E4M3 codes (1 tile);
 *      byte blk*8448 + 8192 + off*4   its fp32 scale.
 *
 * Slots: slot_mapping[t] is an int64. -1 marks a padded token, which is
 * skipped. A value outside [0, num_blocks * 64) is invalid: it is skipped
 * too and counted. Nothing is written for a skipped token. Its input row may
 * still be read, because some rows are loaded together with their slot, so
 * every one of the num_tokens input rows must be readable. Slots must be
 * distinct. If two tokens name the same slot, the bytes left there are
 * unspecified.
 *
 * Cache reads: no byte outside the written slots changes. An fp8 store
 * launch of at least SMs x 8 tokens whose slots are not contiguous runs
 * (kvpub_store_mla_fp8, kvpub_store_mla_fp8_publish, and the inserts of the
 * gather-then-insert calls) may read, into L2 and never back to the caller,
 * the 32-byte sectors that a written slot shares with its neighbours: the
 * Main sector holding the slot's first or last 16 bytes, and the Indexer
 * sector holding its scale. Those reads keep each partial sector write from
 * costing DRAM a read-modify-write.
 */
#ifndef KVPUB_H
#define KVPUB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so callers need no CUDA header. */
struct CUstream_st;
typedef struct CUstream_st *kvpub_stream_t;

typedef enum {
    KVPUB_OK = 0,
    KVPUB_ERR_INVALID_ARG = 1,       /* null pointer, bad size or stride     */
    KVPUB_ERR_ALIGNMENT = 2,         /* pointer or stride not 16-byte aligned */
    KVPUB_ERR_TOO_MANY_REPLICAS = 3, /* num_replicas > KVPUB_MAX_REPLICAS     */
    KVPUB_ERR_CUDA = 4,              /* the CUDA runtime reported an error    */
    KVPUB_ERR_WORKSPACE = 5          /* workspace missing or too small        */
} kvpub_status;

#define KVPUB_MAX_REPLICAS 8
#define KVPUB_BLOCK_SIZE 64
#define KVPUB_LATENT_DIM 512
#define KVPUB_ROPE_DIM 64
#define KVPUB_INDEXER_DIM 128
#define KVPUB_QUANT_TILE 128
#define KVPUB_MAIN_SLOT_BYTES 656
#define KVPUB_INDEXER_SLOT_BYTES 132
#define KVPUB_INDEXER_BLOCK_BYTES (KVPUB_BLOCK_SIZE * KVPUB_INDEXER_SLOT_BYTES)
#define KVPUB_GATHER_ROW_BYTES 1408  /* (512 + 64 + 128) bf16 */
#define KVPUB_MAIN_SLOT_BYTES_BF16 1152     /* (512 + 64) bf16 */
#define KVPUB_INDEXER_SLOT_BYTES_BF16 256   /* 128 bf16 */
#define KVPUB_MAX_POLLS (1ull << 24)
#define KVPUB_STATIC_GATHER_MAX_TOKENS 4096

/*
 * Fused direct publication. One launch stores every token's final Main-KV
 * and Indexer-K bytes into all num_replicas replicas. Source: "[Kernel][PCP]
 * Publish replicated KV updates through PyTorch symmetric memory", Summary,
 * the "THIS PR" diagram, and Design bullet 3.
 *
 *  kv_latent     bf16 [num_tokens, >= 512], row stride latent_stride.
 *  k_rope        bf16 [num_tokens, >= 64], row stride rope_stride.
 *  index_k       bf16 [num_tokens, >= 128], row stride index_stride.
 *                Strides are counted in elements and must be multiples of
 *                8, at least the row width. Base pointers must be 16-byte
 *                aligned. The element stride is 1. The three inputs may be
 *                views of one buffer.
 *  slot_mapping  int64 [num_tokens], 8-byte aligned. See above for -1 and
 *                invalid slots.
 *  num_tokens    >= 0. With 0 the call does nothing, and the input and
 *                slot pointers may be NULL.
 *  main_caches, indexer_caches
 *                HOST arrays of num_replicas device pointers, each 16-byte
 *                aligned. Main cache r holds num_blocks * 64 * 656 bytes and
 *                Indexer cache r holds num_blocks * 8448 bytes. The arrays
 *                are read during the call only.
 *  num_replicas  1..KVPUB_MAX_REPLICAS. 0 or less is KVPUB_ERR_INVALID_ARG;
 *                more is KVPUB_ERR_TOO_MANY_REPLICAS.
 *  num_blocks    >= 1.  block_size must be KVPUB_BLOCK_SIZE (64).
 *  invalid_count NULL, or a device uint64 counter. The call atomically adds
 *                the number of invalid (not -1, out-of-range) slots to it.

 */
kvpub_status kvpub_store_mla_fp8(
    const void *kv_latent, int64_t latent_stride,
    const void *k_rope, int64_t rope_stride,
    const void *index_k, int64_t index_stride,
    const int64_t *slot_mapping, int64_t num_tokens,
    void *const *main_caches, void *const *indexer_caches, int num_replicas,
    int64_t num_blocks, int block_size,
    unsigned long long *invalid_count, kvpub_stream_t stream);

/*
 * Unquantised (bf16) cache variant of the same publication. It has the same
 * rows, slots, replicas, launch and failure rules as kvpub_store_mla_fp8,
 * but the bytes are stored as they arrive, with no scales. Source: the BF16
 * main/indexer cache cases listed under Validation on "[Feature][KV
 * Connector] Support QSA HiSparse in disaggregated serving", published as
 * on "[Kernel][PCP] Publish replicated KV updates through PyTorch symmetric
 * memory", Summary.
 *
 * Layout (a reading; the pages give none):
 *  - Main cache r: num_blocks * 64 slots of KVPUB_MAIN_SLOT_BYTES_BF16 =
 *    1152 bytes. Slot s at byte s * 1152 holds the 512 latent bf16 values,
 *    then the 64 rope bf16 values.
 *  - Indexer cache r: slots of KVPUB_INDEXER_SLOT_BYTES_BF16 = 256 bytes.
 *    Slot s at byte s * 256 holds the 128 Indexer-K bf16 values.
 * Arguments are as in kvpub_store_mla_fp8, with these cache sizes.
 */
kvpub_status kvpub_store_mla_bf16(
    const void *kv_latent, int64_t latent_stride,
    const void *k_rope, int64_t rope_stride,
    const void *index_k, int64_t index_stride,
    const int64_t *slot_mapping, int64_t num_tokens,
    void *const *main_caches, void *const *indexer_caches, int num_replicas,
    int64_t num_blocks, int block_size,
    unsigned long long *invalid_count, kvpub_stream_t stream);

/*
 * Fused publication followed by the epoch advance. This is the same store
 * as kvpub_store_mla_fp8. The launch's last block to finish then makes all
 * stores visible at GPU scope and adds 1 to *epoch. One launch per layer
 * replaces a store launch plus a fence launch. Source: "[Perf][PCP] Fuse
 * direct-KV publication fence" (vLLM #54030), its summary of moving the
 * epoch onto the device and cutting two launches per fence to one.
 *
 *  epoch       device uint64, advanced by exactly 1 per call (also when
 *              num_tokens is 0 or every slot is padded).
 *  done_count  device uint32, zero before the first call. The kernel
 *              counts finished blocks in it and resets it to zero, so it
 *              stays ready for the next call or graph replay. Calls that
 *              share one done_count must not run concurrently.
 *  Other arguments are as in kvpub_store_mla_fp8.
 *
 * This is the choice for eager (non-graph) loops, where the host's cost per
 * launch dominates. Inside a CUDA graph, kvpub_store_mla_fp8 followed by
 * kvpub_epoch_advance is faster: the graph removes the launch cost, and the
 * separate one-thread epoch launch costs less than this kernel's end-of-grid
 * counter round trip.
 */
kvpub_status kvpub_store_mla_fp8_publish(
    const void *kv_latent, int64_t latent_stride,
    const void *k_rope, int64_t rope_stride,
    const void *index_k, int64_t index_stride,
    const int64_t *slot_mapping, int64_t num_tokens,
    void *const *main_caches, void *const *indexer_caches, int num_replicas,
    int64_t num_blocks, int block_size,
    unsigned long long *invalid_count, unsigned long long *epoch,
    unsigned int *done_count, kvpub_stream_t stream);

/* Workspace bytes kvpub_gather_insert needs: num_tokens * 1408 (0 if < 0). */
size_t kvpub_gather_workspace_bytes(int64_t num_tokens);

/*
 * The unfused reference path: gather, then insert. Source: "[Kernel][PCP]
 * Publish replicated KV updates through PyTorch symmetric memory", the
 * "AS-IS: gather then insert" diagram.
 *  - Step 1, one launch: copy every token's bf16 row (latent | rope |
 *    index_k, 1408 bytes) into the workspace. On one GPU this stands in for
 *    the AllGather of the update tensors.
 *  - Step 2, one launch per replica: quantise the gathered rows and insert
 *    them into that replica.
 * The bytes left in the caches equal kvpub_store_mla_fp8's.
 *
 *  workspace       device buffer of at least
 *                  kvpub_gather_workspace_bytes(num_tokens) bytes, 16-byte
 *                  aligned. Its contents on return are unspecified.
 *  workspace_bytes its size. Too small gives KVPUB_ERR_WORKSPACE.
 *  Other arguments are as in kvpub_store_mla_fp8. invalid_count is advanced
 *  once per call, not once per replica.
 */
kvpub_status kvpub_gather_insert(
    const void *kv_latent, int64_t latent_stride,
    const void *k_rope, int64_t rope_stride,
    const void *index_k, int64_t index_stride,
    const int64_t *slot_mapping, int64_t num_tokens,
    void *const *main_caches, void *const *indexer_caches, int num_replicas,
    int64_t num_blocks, int block_size,
    unsigned long long *invalid_count,
    void *workspace, size_t workspace_bytes, kvpub_stream_t stream);

/*
 * Allocation-free gather-then-insert. It has no counterpart on the pages: it
 * is kvpub_gather_insert for callers that cannot allocate device memory. Such
 * callers include:
 *  - a serving loop whose device memory is planned and reserved once at
 *    start-up, so that nothing may be allocated while requests run;
 *  - a plugin inside another runtime that owns all device memory;
 *  - code on a latency-critical path, where cudaMalloc may synchronise the
 *    device and stall every other stream.
 * Its bytes equal kvpub_gather_insert's. The only difference is the
 * workspace: a fixed array of KVPUB_STATIC_GATHER_MAX_TOKENS rows of 1408
 * bytes (5.5 MiB) inside this library, not caller memory. Every GPU that
 * loads the library holds that array until the process exits.
 *
 *  - num_tokens above KVPUB_STATIC_GATHER_MAX_TOKENS gives
 *    KVPUB_ERR_WORKSPACE, and nothing is launched.
 *  - Every call looks up the array's device address for the current device
 *    (a host-side lookup; nothing is cached, so the call stays valid after a
 *    cudaDeviceReset, which reloads the array at another address). The
 *    first call on a device may load the library's device code there: make
 *    it before any stream capture on that device.
 *  - Every call uses the same array. Calls that can overlap on the GPU (on
 *    different streams, or issued from several threads without ordering)
 *    race on it and corrupt each other's rows. Issue them on one stream.
 *  - No element of the array needs to start at zero. Each call writes every
 *    workspace row before it reads it.
 *  - It calls no cudaMalloc, no cudaFree and no allocating library routine.
 * Other arguments, and the failure statuses, are as in kvpub_gather_insert.
 */
kvpub_status kvpub_gather_insert_noalloc(
    const void *kv_latent, int64_t latent_stride,
    const void *k_rope, int64_t rope_stride,
    const void *index_k, int64_t index_stride,
    const int64_t *slot_mapping, int64_t num_tokens,
    void *const *main_caches, void *const *indexer_caches, int num_replicas,
    int64_t num_blocks, int block_size,
    unsigned long long *invalid_count, kvpub_stream_t stream);

/*
 * Device-resident publication epoch: one single-thread launch. It makes
 * every earlier store on the stream visible at GPU scope (a release), then
 * adds 1 to *epoch. The counter lives in device memory, so a captured
 * graph advances it on every replay. Sources: "[Perf][PCP] Fuse direct-KV
 * publication fence" (vLLM #54030), Motivation and its summary of the
 * device epoch. "[Kernel][PCP] Publish replicated KV updates through
 * PyTorch symmetric memory", Design bullet 4 (device-epoch barrier).
 *
 *  epoch  device uint64, 8-byte aligned. The caller initialises it.
 */
kvpub_status kvpub_epoch_advance(unsigned long long *epoch, kvpub_stream_t stream);

/*
 * Bounded acquire-wait on a device epoch: one single-thread launch. It
 * polls *epoch with acquire loads until *epoch >= target, or until it has
 * polled max_polls times. It then writes 0 (reached) or 1 (timed out) to
 * *status. It never traps. This is the consumer half of the release/acquire
 * barrier: "[Kernel][PCP] Publish replicated KV updates through PyTorch
 * symmetric memory", Summary (one release/acquire barrier after
 * publication).
 *
 *  epoch      device uint64 counter, as above.
 *  max_polls  1 .. KVPUB_MAX_POLLS (2^24); other values are
 *             KVPUB_ERR_INVALID_ARG. Polls are about 64 ns apart, so the
 *             longest wait is on the order of a second.
 *  status     device uint32 result word.
 * The wait must not depend on a kernel that cannot run alongside it. On
 * one stream, the epoch is either already advanced or never will be.
 */
kvpub_status kvpub_epoch_wait(const unsigned long long *epoch,
                              unsigned long long target,
                              unsigned long long max_polls,
                              unsigned int *status, kvpub_stream_t stream);

/* The calling thread's last error message ("" after a successful call). */
const char *kvpub_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVPUB_H */
