// libkvpub: the fused replicated fp8 KV-cache store and its companions,
// hand-written for GB300 (sm_103a).  The C ABI is declared in kvpub.h.
//
// Direct publication ("[Kernel][PCP] Publish replicated KV updates through
// PyTorch symmetric memory", Summary and the "THIS PR" diagram): one launch
// reads each token row once, quantises it in registers and stores the final
// bytes to all R replicas.  The work is HBM-bound (1408 bytes read and
// 788 * R bytes written per row); no tensor cores, no shared memory.

#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include <atomic>

#include "kvpub.h"
#include "quant.cuh"

namespace kvpub {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kThreads = kWarpsPerBlock * 32;
// The row loop is tuned for 4 resident blocks of kThreads threads per SM,
// which needs at most 64 registers a thread.  The compiler gets there by
// itself for most instantiations.  The few it would give more registers
// (3 blocks per SM) are held to it explicitly: the bf16 store with one
// replica and the fused publish with two or three, each 3-4 % faster so.
// A minimum of 0 blocks leaves the choice to the compiler (an explicit 1
// would let it spend up to 255 registers).
template <int R> constexpr int kBf16MinBlocks = (R == 1) ? 4 : 0;
template <int R> constexpr int kPublishMinBlocks = (R == 2 || R == 3) ? 4 : 0;
// Block size of a launch too small to give every SM a block of kWarpsPerBlock rows.
constexpr int kSmallBlockWarps = 2;
constexpr unsigned long long kMaxPolls = KVPUB_MAX_POLLS;

struct Replicas {
    uint8_t *main[KVPUB_MAX_REPLICAS];
    uint8_t *indexer[KVPUB_MAX_REPLICAS];
};

struct StoreArgs {
    const uint16_t *latent;
    const uint16_t *rope;
    const uint16_t *index_k;
    int64_t latent_stride;   // elements
    int64_t rope_stride;
    int64_t index_stride;
    const int64_t *slot_mapping;
    int64_t num_tokens;
    int64_t num_slots;
    unsigned long long *invalid_count;
    Replicas rep;
};

__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ld_stream8(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// Stores are cache-streaming (evict-first): nothing written here is read
// again by this launch.
__device__ __forceinline__ void st16(void *p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ void st8(void *p, uint2 v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// Plain store, for the gather workspace that the insert launches read back.
__device__ __forceinline__ void st16_keep(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ void st4(void *p, uint32_t v) {
    asm volatile("st.global.cs.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Every kernel here is launched with programmatic stream serialization, so
// its blocks may be scheduled while the previous kernel on the stream is
// still finishing.  Each kernel waits, before it touches memory, until that
// kernel has completed and its memory is visible, so nothing is read or
// written out of stream order; only the launch latency overlaps.
__device__ __forceinline__ void wait_previous_kernel() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// One token row's inputs as this lane holds them.
struct RowRegs {
    uint4 x0, x1;   // latent elements [16 l, 16 l + 16)
    uint2 xi;       // Indexer-K elements [4 l, 4 l + 4)
    uint4 tail;     // lanes 1..8: rope chunk l - 1
};

__device__ __forceinline__ void load_row(const StoreArgs &a, int64_t t, int lane, RowRegs &v) {
    const uint8_t *lat = reinterpret_cast<const uint8_t *>(a.latent + t * a.latent_stride);
    v.x0 = ld_stream16(lat + 32 * lane);
    v.x1 = ld_stream16(lat + 32 * lane + 16);
    v.xi = ld_stream8(reinterpret_cast<const uint8_t *>(a.index_k + t * a.index_stride) +
                      8 * lane);
    v.tail = make_uint4(0u, 0u, 0u, 0u);
    if (lane >= 1 && lane <= 8)
        v.tail = ld_stream16(reinterpret_cast<const uint8_t *>(a.rope + t * a.rope_stride) +
                             16 * (lane - 1));
}

__device__ __forceinline__ bool slot_written(int64_t s, int64_t num_slots) {
    return s >= 0 && s < num_slots;
}

// Quantise one row held in registers and store it to every replica.  All
// lanes of the warp call this together (s is warp-uniform).
template <int R>
__device__ __forceinline__ void publish_row(const StoreArgs &a, const RowRegs &v, int64_t s,
                                            int lane) {
    // amax: latent tile (8 lanes) in the low half, Indexer-K (32 lanes) high.
    uint32_t m_lat = absmax_bf16x2(absmax_bf16x2(v.x0.x, v.x0.y), absmax_bf16x2(v.x0.z, v.x0.w));
    m_lat = __vmaxu2(m_lat, absmax_bf16x2(absmax_bf16x2(v.x1.x, v.x1.y),
                                          absmax_bf16x2(v.x1.z, v.x1.w)));
    const uint32_t m_idx = halves_max(absmax_bf16x2(v.xi.x, v.xi.y));
    uint32_t packed = halves_max(m_lat) | (m_idx << 16);
    packed = __vmaxu2(packed, __shfl_xor_sync(kFullMask, packed, 1));
    packed = __vmaxu2(packed, __shfl_xor_sync(kFullMask, packed, 2));
    packed = __vmaxu2(packed, __shfl_xor_sync(kFullMask, packed, 4));
    const float s_lat = tile_scale(packed & 0xffffu);
    packed = __vmaxu2(packed, __shfl_xor_sync(kFullMask, packed, 8));
    packed = __vmaxu2(packed, __shfl_xor_sync(kFullMask, packed, 16));
    const float s_idx = tile_scale(packed >> 16);

    const TileDivisor d_lat = tile_divisor(s_lat);
    const TileDivisor d_idx = tile_divisor(s_idx);
    const uint4 q_lat = make_uint4(quant4(v.x0.x, v.x0.y, d_lat), quant4(v.x0.z, v.x0.w, d_lat),
                                   quant4(v.x1.x, v.x1.y, d_lat), quant4(v.x1.z, v.x1.w, d_lat));
    const uint32_t q_idx = quant4(v.xi.x, v.xi.y, d_idx);

    // lane 0 carries the 4 tile scales (row bytes 512..527); lanes 1..8
    // carry the rope (bytes 528..655).
    const float s1 = __shfl_sync(kFullMask, s_lat, 8);
    const float s2 = __shfl_sync(kFullMask, s_lat, 16);
    const float s3 = __shfl_sync(kFullMask, s_lat, 24);
    uint4 tail = v.tail;
    if (lane == 0)
        tail = make_uint4(__float_as_uint(s_lat), __float_as_uint(s1), __float_as_uint(s2),
                          __float_as_uint(s3));

    const int64_t main_off = s * KVPUB_MAIN_SLOT_BYTES;
    const int64_t blk = s >> 6, off = s & 63;
    const int64_t idx_off = blk * KVPUB_INDEXER_BLOCK_BYTES + off * KVPUB_INDEXER_DIM;
    const int64_t idx_scale_off = blk * KVPUB_INDEXER_BLOCK_BYTES +
                                  KVPUB_BLOCK_SIZE * KVPUB_INDEXER_DIM + off * 4;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        uint8_t *row = a.rep.main[r] + main_off;
        st16(row + 16 * lane, q_lat);
        if (lane <= 8) st16(row + 512 + 16 * lane, tail);
        uint8_t *ib = a.rep.indexer[r];
        st4(ib + idx_off + 4 * lane, q_idx);
        if (lane == 0) st4(ib + idx_scale_off, __float_as_uint(s_idx));
    }
}

// Unquantised (bf16) cache variant: the row's bytes stored as they arrive.
// Main slot s = latent | rope at s * 1152; Indexer slot s = index_k at
// s * 256.  The lanes hold the row exactly as load_row left it.
template <int R>
__device__ __forceinline__ void copy_row_bf16(const StoreArgs &a, const RowRegs &v, int64_t s,
                                              int lane) {
    const int64_t main_off = s * KVPUB_MAIN_SLOT_BYTES_BF16 + 32 * lane;
    const int64_t rope_off = s * KVPUB_MAIN_SLOT_BYTES_BF16 + 2 * KVPUB_LATENT_DIM +
                             16 * (lane - 1);
    const int64_t idx_off = s * KVPUB_INDEXER_SLOT_BYTES_BF16 + 8 * lane;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        uint8_t *m = a.rep.main[r];
        st16(m + main_off, v.x0);
        st16(m + main_off + 16, v.x1);
        if (lane >= 1 && lane <= 8) st16(m + rope_off, v.tail);
        st8(a.rep.indexer[r] + idx_off, v.xi);
    }
}

// The fp8 slot layout leaves two 32-byte sectors of every written row and
// replica only partly written: the Main row's last (even s) or first (odd s)
// 16 bytes share a sector with the neighbouring slot, and the 4-byte Indexer
// scale shares one with 7 others.  When the neighbours are written in the
// same launch (contiguous prefill runs) L2 merges the parts into whole
// sectors.  When they are not (slots scattered over a large cache), each
// part-written sector costs DRAM a read-modify-write late, among the
// write-backs; fetching those sectors into L2 a row ahead instead makes the
// stores land on valid sectors (on the 706,624-slot capacity batch, L2's
// read-modify-writes fall from about one per row and replica to none, and
// the launch takes about 10 % less time).  Lanes 0..R-1 fetch the Main
// sectors and lanes R..2R-1 the scale sectors of replicas 0..R-1.
template <int R>
__device__ __forceinline__ void prefetch_part_sectors(const StoreArgs &a, int64_t s, int lane) {
    const uint8_t *p = nullptr;
    if (lane < R) {
        p = a.rep.main[lane] + s * KVPUB_MAIN_SLOT_BYTES + ((s & 1) ? -16 : 640);
    } else if (lane < 2 * R) {
        p = a.rep.indexer[lane - R] + (s >> 6) * KVPUB_INDEXER_BLOCK_BYTES +
            KVPUB_BLOCK_SIZE * KVPUB_INDEXER_DIM + (s & 56) * 4;
    }
    if (p != nullptr) asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

// Grid-stride over token rows, one warp per row.  The next row's slot and
// inputs are loaded before the current row is quantised, so each warp keeps
// two rows of loads in flight; the next row's inputs are read only if its
// slot is written.
//
// kPrefetch (large launches of the fp8 store only): the warp also reads the
// slots of its first row's two neighbours in the batch, in the same load
// instruction as that row's slot.  If neither holds the neighbouring slot
// (the rows are not a contiguous run), the warp prefetches the part-written
// sectors of every row it stores (see prefetch_part_sectors); in contiguous
// runs those prefetches would only add reads.
template <int R, bool kFp8, bool kPrefetch>
__device__ __forceinline__ void publish_rows(const StoreArgs &a) {
    const int lane = threadIdx.x & 31;
    const int64_t num_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (t >= a.num_tokens) return;
    // The warp's first row is loaded together with its slot instead of after
    // it: one memory latency less at the start of every launch, which is most
    // of a decode batch's time.  A padded row's inputs may be read this way
    // (they exist: the caller passes num_tokens rows); nothing is written.
    RowRegs cur;
    load_row(a, t, lane, cur);
    int64_t s;
    bool pf = false;
    if (kPrefetch) {
        // lanes 0, 1, 2 read the slots of rows t-1, t, t+1 (clamped to the
        // batch, so a missing neighbour reads row t itself and never matches)
        int64_t tn = t - 1 + (lane < 2 ? lane : 2);
        tn = tn < 0 ? 0 : (tn >= a.num_tokens ? a.num_tokens - 1 : tn);
        const int64_t v = a.slot_mapping[tn];
        s = __shfl_sync(kFullMask, v, 1);
        const int64_t s_prev = __shfl_sync(kFullMask, v, 0);
        const int64_t s_succ = __shfl_sync(kFullMask, v, 2);
        pf = !(s_prev == s - 1 || s_succ == s + 1);
        if (pf && slot_written(s, a.num_slots)) prefetch_part_sectors<R>(a, s, lane);
    } else {
        s = a.slot_mapping[t];
    }
    while (true) {
        const int64_t t_next = t + num_warps;
        int64_t s_next = -1;
        RowRegs nxt;
        if (t_next < a.num_tokens) {
            s_next = a.slot_mapping[t_next];
            if (slot_written(s_next, a.num_slots)) {
                load_row(a, t_next, lane, nxt);
                if (kPrefetch && pf) prefetch_part_sectors<R>(a, s_next, lane);
            }
        }
        if (slot_written(s, a.num_slots)) {
            if (kFp8) publish_row<R>(a, cur, s, lane);
            else copy_row_bf16<R>(a, cur, s, lane);
        } else if (s != -1 && lane == 0 && a.invalid_count != nullptr) {
            atomicAdd(a.invalid_count, 1ull);
        }
        if (t_next >= a.num_tokens) break;
        t = t_next;
        s = s_next;
        cur = nxt;
    }
}

// kPrefetch is true for launches of kThreads-thread blocks (at least
// SMs x kWarpsPerBlock rows) and false for the small-block launches of
// latency-bound batches, which get a kernel without the prefetch code.
template <int R, bool kPrefetch>
__global__ void __launch_bounds__(kThreads) store_mla_fp8_kernel(const StoreArgs a) {
    wait_previous_kernel();
    publish_rows<R, true, kPrefetch>(a);
}

template <int R>
__global__ void __launch_bounds__(kThreads, kBf16MinBlocks<R>)
store_mla_bf16_kernel(const StoreArgs a) {
    wait_previous_kernel();
    publish_rows<R, false, false>(a);
}

__device__ __forceinline__ void release_add_epoch(unsigned long long *epoch) {
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" :: "l"(epoch) : "memory");
}

// Store, then the last block to finish publishes the epoch.
template <int R, bool kPrefetch>
__global__ void __launch_bounds__(kThreads, kPublishMinBlocks<R>)
store_mla_fp8_publish_kernel(const StoreArgs a, unsigned long long *epoch,
                             unsigned int *done_count) {
    wait_previous_kernel();
    publish_rows<R, true, kPrefetch>(a);
    // The barrier orders every thread's stores before thread 0's counter
    // update; that update is an acq_rel atomic at GPU scope, so it releases
    // the whole block's stores and, in the last block, acquires every other
    // block's.  (The same barrier-then-one-thread pattern as a grid-wide
    // sync, with the fence folded into the atomic.)
    __syncthreads();
    // Every store of this block is issued: the next kernel on the stream may
    // be scheduled now rather than when this block exits after the counter
    // round trip (its own wait still holds it until this grid completes).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        unsigned int prev;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                     : "=r"(prev) : "l"(done_count) : "memory");
        if (prev == gridDim.x - 1) {
            // Ready for the next call or replay, which reads the counter only
            // after this grid has completed: a plain store is enough.
            asm volatile("st.relaxed.gpu.global.u32 [%0], 0;" :: "l"(done_count) : "memory");
            release_add_epoch(epoch);
        }
    }
}

// Gather step of the unfused path: every token's bf16 row into one
// 1408-byte workspace row (latent | rope | index_k).
__global__ void __launch_bounds__(kThreads)
gather_rows_kernel(const StoreArgs a, uint8_t *workspace) {
    wait_previous_kernel();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t num_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t t = warp; t < a.num_tokens; t += num_warps) {
        uint8_t *w = workspace + t * KVPUB_GATHER_ROW_BYTES;
        const uint8_t *lat = reinterpret_cast<const uint8_t *>(a.latent + t * a.latent_stride);
        const uint8_t *rope = reinterpret_cast<const uint8_t *>(a.rope + t * a.rope_stride);
        const uint8_t *idx = reinterpret_cast<const uint8_t *>(a.index_k + t * a.index_stride);
        // 88 chunks of 16 bytes: 64 latent, 8 rope, 16 Indexer-K.
        for (int c = lane; c < 88; c += 32) {
            const uint8_t *src = c < 64 ? lat + 16 * c
                                : c < 72 ? rope + 16 * (c - 64)
                                         : idx + 16 * (c - 72);
            st16_keep(w + 16 * c, ld_stream16(src));
        }
    }
}

// The one-thread epoch kernel lets the next kernel on the stream be
// scheduled at once (griddepcontrol.launch_dependents) instead of when it
// exits.  The next kernel's blocks then become resident while this one is
// still waiting for the store before it; their own wait still holds them
// until this kernel has completed and its increment is visible.  In a graph
// of store + epoch launches this takes the launch of the next store's grid
// off the critical path (61-layer prefill step 0.750 -> 0.735 ms).  The
// store kernels do not trigger early: there the next grid's blocks would
// only compete with the running one for SM slots (measured slower).
__global__ void epoch_advance_kernel(unsigned long long *epoch) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    wait_previous_kernel();
    release_add_epoch(epoch);
}

__global__ void epoch_wait_kernel(const unsigned long long *epoch, unsigned long long target,
                                  unsigned long long max_polls, unsigned int *status) {
    wait_previous_kernel();
    unsigned int st = 1u;
    for (unsigned long long i = 0; i < max_polls; ++i) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(epoch) : "memory");
        if (v >= target) {
            st = 0u;
            break;
        }
        __nanosleep(64);
    }
    *status = st;
}

// ---------------------------------------------------------------- host side

thread_local char g_last_error[512] = "";

kvpub_status fail(kvpub_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

kvpub_status ok() {
    g_last_error[0] = '\0';
    return KVPUB_OK;
}

bool aligned(const void *p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

kvpub_status check_rows(const void *p, int64_t stride, int64_t dim, int64_t num_tokens,
                        const char *name) {
    if (p == nullptr) return fail(KVPUB_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned(p, 16)) return fail(KVPUB_ERR_ALIGNMENT, "%s is not 16-byte aligned", name);
    if (stride < dim)
        return fail(KVPUB_ERR_INVALID_ARG, "%s row stride %lld < %lld", name, (long long)stride,
                    (long long)dim);
    if (stride % 8 != 0)
        return fail(KVPUB_ERR_ALIGNMENT, "%s row stride %lld is not a multiple of 8 elements",
                    name, (long long)stride);
    if (num_tokens > 0 && stride > INT64_MAX / 2 / num_tokens)
        return fail(KVPUB_ERR_INVALID_ARG, "%s spans more than 2^62 bytes", name);
    return KVPUB_OK;
}

struct Validated {
    StoreArgs args;
    int num_replicas;
};

kvpub_status validate(const void *kv_latent, int64_t latent_stride, const void *k_rope,
                      int64_t rope_stride, const void *index_k, int64_t index_stride,
                      const int64_t *slot_mapping, int64_t num_tokens,
                      void *const *main_caches, void *const *indexer_caches, int num_replicas,
                      int64_t num_blocks, int block_size, unsigned long long *invalid_count,
                      Validated *out, int64_t main_slot_bytes = KVPUB_MAIN_SLOT_BYTES) {
    if (num_replicas < 1) return fail(KVPUB_ERR_INVALID_ARG, "num_replicas %d < 1", num_replicas);
    if (num_replicas > KVPUB_MAX_REPLICAS)
        return fail(KVPUB_ERR_TOO_MANY_REPLICAS, "num_replicas %d > %d", num_replicas,
                    KVPUB_MAX_REPLICAS);
    if (block_size != KVPUB_BLOCK_SIZE)
        return fail(KVPUB_ERR_INVALID_ARG, "block_size %d != %d", block_size, KVPUB_BLOCK_SIZE);
    if (num_tokens < 0)
        return fail(KVPUB_ERR_INVALID_ARG, "num_tokens %lld < 0", (long long)num_tokens);
    if (num_blocks < 1 ||
        num_blocks > INT64_MAX / (KVPUB_BLOCK_SIZE * main_slot_bytes))
        return fail(KVPUB_ERR_INVALID_ARG, "num_blocks %lld out of range", (long long)num_blocks);
    if (main_caches == nullptr || indexer_caches == nullptr)
        return fail(KVPUB_ERR_INVALID_ARG, "cache pointer arrays are NULL");
    if (invalid_count != nullptr && !aligned(invalid_count, 8))
        return fail(KVPUB_ERR_ALIGNMENT, "invalid_count is not 8-byte aligned");
    Replicas rep{};
    for (int r = 0; r < num_replicas; ++r) {
        if (main_caches[r] == nullptr || indexer_caches[r] == nullptr)
            return fail(KVPUB_ERR_INVALID_ARG, "cache pointer of replica %d is NULL", r);
        if (!aligned(main_caches[r], 16) || !aligned(indexer_caches[r], 16))
            return fail(KVPUB_ERR_ALIGNMENT, "cache of replica %d is not 16-byte aligned", r);
        rep.main[r] = static_cast<uint8_t *>(main_caches[r]);
        rep.indexer[r] = static_cast<uint8_t *>(indexer_caches[r]);
    }
    if (num_tokens > 0) {
        kvpub_status st;
        if ((st = check_rows(kv_latent, latent_stride, KVPUB_LATENT_DIM, num_tokens,
                             "kv_latent")) != KVPUB_OK)
            return st;
        if ((st = check_rows(k_rope, rope_stride, KVPUB_ROPE_DIM, num_tokens, "k_rope")) !=
            KVPUB_OK)
            return st;
        if ((st = check_rows(index_k, index_stride, KVPUB_INDEXER_DIM, num_tokens,
                             "index_k")) != KVPUB_OK)
            return st;
        if (slot_mapping == nullptr) return fail(KVPUB_ERR_INVALID_ARG, "slot_mapping is NULL");
        if (!aligned(slot_mapping, 8))
            return fail(KVPUB_ERR_ALIGNMENT, "slot_mapping is not 8-byte aligned");
    }
    out->args.latent = static_cast<const uint16_t *>(kv_latent);
    out->args.rope = static_cast<const uint16_t *>(k_rope);
    out->args.index_k = static_cast<const uint16_t *>(index_k);
    out->args.latent_stride = latent_stride;
    out->args.rope_stride = rope_stride;
    out->args.index_stride = index_stride;
    out->args.slot_mapping = slot_mapping;
    out->args.num_tokens = num_tokens;
    out->args.num_slots = num_blocks * KVPUB_BLOCK_SIZE;
    out->args.invalid_count = invalid_count;
    out->args.rep = rep;
    out->num_replicas = num_replicas;
    return KVPUB_OK;
}

// SM count and, per kernel, resident blocks per SM; both cached per device.
constexpr int kMaxDevices = 64;

std::atomic<int> g_sm_count[kMaxDevices];

kvpub_status current_device(int *dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return fail(KVPUB_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (*dev < 0 || *dev >= kMaxDevices)
        return fail(KVPUB_ERR_CUDA, "device %d out of range", *dev);
    return KVPUB_OK;
}

kvpub_status sm_count(int dev, int *out) {
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return fail(KVPUB_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    *out = n;
    return KVPUB_OK;
}

// A grid-stride pass over num_tokens rows (one warp per row): one block per
// kWarpsPerBlock rows, capped at the blocks that fit on the GPU at once, so
// every launch is a single wave.  A launch with fewer rows than SMs x
// kWarpsPerBlock would leave SMs idle; it takes blocks of kSmallBlockWarps
// warps instead, which spreads its rows over 4x as many SMs.  Such a launch
// (a decode batch) is latency-bound, and each SM's load path then serves
// fewer rows (measured: a 64-row store 1.91 -> 1.76 us).  All its blocks fit
// at once too: at most SMs x 4 blocks of 64 threads.
struct LaunchShape {
    int grid;
    int threads;
};

template <typename Kernel>
kvpub_status one_wave_grid(Kernel kernel, std::atomic<int> *resident, int64_t num_tokens,
                           LaunchShape *shape) {
    int dev = 0, sms = 0;
    kvpub_status st = current_device(&dev);
    if (st != KVPUB_OK) return st;
    if ((st = sm_count(dev, &sms)) != KVPUB_OK) return st;
    if (num_tokens < static_cast<int64_t>(sms) * kWarpsPerBlock) {
        const int64_t want = (num_tokens + kSmallBlockWarps - 1) / kSmallBlockWarps;
        shape->grid = static_cast<int>(want < 1 ? 1 : want);
        shape->threads = kSmallBlockWarps * 32;
        return KVPUB_OK;
    }
    int per_sm = resident[dev].load(std::memory_order_relaxed);
    if (per_sm == 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
        if (e != cudaSuccess)
            return fail(KVPUB_ERR_CUDA, "occupancy query: %s", cudaGetErrorString(e));
        if (per_sm < 1) per_sm = 1;
        resident[dev].store(per_sm, std::memory_order_relaxed);
    }
    int64_t want = (num_tokens + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const int64_t cap = static_cast<int64_t>(sms) * per_sm;
    if (want > cap) want = cap;
    shape->grid = static_cast<int>(want);
    shape->threads = kThreads;
    return KVPUB_OK;
}

kvpub_status launched(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(KVPUB_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
    return ok();
}

// Launch with programmatic stream serialization (see wait_previous_kernel).
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), int grid, int threads, cudaStream_t stream,
                   Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <template <int> class Launch, typename... Args>
kvpub_status dispatch_replicas(int r, Args &&...args) {
    switch (r) {
        case 1: return Launch<1>::go(args...);
        case 2: return Launch<2>::go(args...);
        case 3: return Launch<3>::go(args...);
        case 4: return Launch<4>::go(args...);
        case 5: return Launch<5>::go(args...);
        case 6: return Launch<6>::go(args...);
        case 7: return Launch<7>::go(args...);
        default: return Launch<8>::go(args...);
    }
}

// Launches of kThreads-thread blocks take the kernel with the part-sector
// prefetch; the small-block launches of latency-bound batches the one
// without (see publish_rows).
template <int R>
struct LaunchStore {
    static std::atomic<int> resident[kMaxDevices];
    static kvpub_status go(cudaStream_t stream, const StoreArgs &a) {
        LaunchShape sh;
        kvpub_status st =
            one_wave_grid(store_mla_fp8_kernel<R, true>, resident, a.num_tokens, &sh);
        if (st != KVPUB_OK) return st;
        (void)cudaGetLastError();
        if (sh.threads == kThreads)
            (void)launch(store_mla_fp8_kernel<R, true>, sh.grid, sh.threads, stream, a);
        else
            (void)launch(store_mla_fp8_kernel<R, false>, sh.grid, sh.threads, stream, a);
        return launched("store_mla_fp8");
    }
};
template <int R>
std::atomic<int> LaunchStore<R>::resident[kMaxDevices];

template <int R>
struct LaunchStoreBf16 {
    static std::atomic<int> resident[kMaxDevices];
    static kvpub_status go(cudaStream_t stream, const StoreArgs &a) {
        LaunchShape sh;
        kvpub_status st = one_wave_grid(store_mla_bf16_kernel<R>, resident, a.num_tokens, &sh);
        if (st != KVPUB_OK) return st;
        (void)cudaGetLastError();
        (void)launch(store_mla_bf16_kernel<R>, sh.grid, sh.threads, stream, a);
        return launched("store_mla_bf16");
    }
};
template <int R>
std::atomic<int> LaunchStoreBf16<R>::resident[kMaxDevices];

template <int R>
struct LaunchPublish {
    static std::atomic<int> resident[kMaxDevices];
    static kvpub_status go(cudaStream_t stream, const StoreArgs &a, unsigned long long *epoch,
                           unsigned int *done) {
        LaunchShape sh;
        kvpub_status st =
            one_wave_grid(store_mla_fp8_publish_kernel<R, true>, resident, a.num_tokens, &sh);
        if (st != KVPUB_OK) return st;
        (void)cudaGetLastError();
        if (sh.threads == kThreads)
            (void)launch(store_mla_fp8_publish_kernel<R, true>, sh.grid, sh.threads, stream, a,
                         epoch, done);
        else
            (void)launch(store_mla_fp8_publish_kernel<R, false>, sh.grid, sh.threads, stream, a,
                         epoch, done);
        return launched("store_mla_fp8_publish");
    }
};
template <int R>
std::atomic<int> LaunchPublish<R>::resident[kMaxDevices];

std::atomic<int> g_gather_resident[kMaxDevices];

// Gather every row into the workspace, then one insert launch per replica
// that quantises the gathered rows (the insert is the store kernel with one
// replica, reading the workspace rows).
kvpub_status gather_then_insert(const Validated &v, uint8_t *ws, cudaStream_t s) {
    LaunchShape sh;
    kvpub_status st = one_wave_grid(gather_rows_kernel, g_gather_resident, v.args.num_tokens, &sh);
    if (st != KVPUB_OK) return st;
    (void)cudaGetLastError();
    (void)launch(gather_rows_kernel, sh.grid, sh.threads, s, v.args, ws);
    if ((st = launched("gather_rows")) != KVPUB_OK) return st;
    StoreArgs ins = v.args;
    const uint16_t *w16 = reinterpret_cast<const uint16_t *>(ws);
    ins.latent = w16;
    ins.rope = w16 + KVPUB_LATENT_DIM;
    ins.index_k = w16 + KVPUB_LATENT_DIM + KVPUB_ROPE_DIM;
    ins.latent_stride = ins.rope_stride = ins.index_stride = KVPUB_GATHER_ROW_BYTES / 2;
    for (int r = 0; r < v.num_replicas; ++r) {
        ins.rep = Replicas{};
        ins.rep.main[0] = v.args.rep.main[r];
        ins.rep.indexer[0] = v.args.rep.indexer[r];
        ins.invalid_count = (r == 0) ? v.args.invalid_count : nullptr;
        if ((st = LaunchStore<1>::go(s, ins)) != KVPUB_OK) return st;
    }
    return ok();
}

}  // namespace
}  // namespace kvpub

using namespace kvpub;

extern "C" kvpub_status kvpub_store_mla_fp8(
    const void *kv_latent, int64_t latent_stride, const void *k_rope, int64_t rope_stride,
    const void *index_k, int64_t index_stride, const int64_t *slot_mapping, int64_t num_tokens,
    void *const *main_caches, void *const *indexer_caches, int num_replicas, int64_t num_blocks,
    int block_size, unsigned long long *invalid_count, kvpub_stream_t stream) {
    Validated v;
    kvpub_status st = validate(kv_latent, latent_stride, k_rope, rope_stride, index_k,
                               index_stride, slot_mapping, num_tokens, main_caches,
                               indexer_caches, num_replicas, num_blocks, block_size,
                               invalid_count, &v);
    if (st != KVPUB_OK) return st;
    if (num_tokens == 0) return ok();
    return dispatch_replicas<LaunchStore>(v.num_replicas, (cudaStream_t)stream, v.args);
}

extern "C" kvpub_status kvpub_store_mla_bf16(
    const void *kv_latent, int64_t latent_stride, const void *k_rope, int64_t rope_stride,
    const void *index_k, int64_t index_stride, const int64_t *slot_mapping, int64_t num_tokens,
    void *const *main_caches, void *const *indexer_caches, int num_replicas, int64_t num_blocks,
    int block_size, unsigned long long *invalid_count, kvpub_stream_t stream) {
    Validated v;
    kvpub_status st = validate(kv_latent, latent_stride, k_rope, rope_stride, index_k,
                               index_stride, slot_mapping, num_tokens, main_caches,
                               indexer_caches, num_replicas, num_blocks, block_size,
                               invalid_count, &v, KVPUB_MAIN_SLOT_BYTES_BF16);
    if (st != KVPUB_OK) return st;
    if (num_tokens == 0) return ok();
    return dispatch_replicas<LaunchStoreBf16>(v.num_replicas, (cudaStream_t)stream, v.args);
}

extern "C" kvpub_status kvpub_store_mla_fp8_publish(
    const void *kv_latent, int64_t latent_stride, const void *k_rope, int64_t rope_stride,
    const void *index_k, int64_t index_stride, const int64_t *slot_mapping, int64_t num_tokens,
    void *const *main_caches, void *const *indexer_caches, int num_replicas, int64_t num_blocks,
    int block_size, unsigned long long *invalid_count, unsigned long long *epoch,
    unsigned int *done_count, kvpub_stream_t stream) {
    Validated v;
    kvpub_status st = validate(kv_latent, latent_stride, k_rope, rope_stride, index_k,
                               index_stride, slot_mapping, num_tokens, main_caches,
                               indexer_caches, num_replicas, num_blocks, block_size,
                               invalid_count, &v);
    if (st != KVPUB_OK) return st;
    if (epoch == nullptr || done_count == nullptr)
        return fail(KVPUB_ERR_INVALID_ARG, "epoch or done_count is NULL");
    if (!aligned(epoch, 8) || !aligned(done_count, 4))
        return fail(KVPUB_ERR_ALIGNMENT, "epoch or done_count is misaligned");
    return dispatch_replicas<LaunchPublish>(v.num_replicas, (cudaStream_t)stream, v.args, epoch,
                                            done_count);
}

extern "C" size_t kvpub_gather_workspace_bytes(int64_t num_tokens) {
    if (num_tokens <= 0) return 0;
    return static_cast<size_t>(num_tokens) * KVPUB_GATHER_ROW_BYTES;
}

extern "C" kvpub_status kvpub_gather_insert(
    const void *kv_latent, int64_t latent_stride, const void *k_rope, int64_t rope_stride,
    const void *index_k, int64_t index_stride, const int64_t *slot_mapping, int64_t num_tokens,
    void *const *main_caches, void *const *indexer_caches, int num_replicas, int64_t num_blocks,
    int block_size, unsigned long long *invalid_count, void *workspace, size_t workspace_bytes,
    kvpub_stream_t stream) {
    Validated v;
    kvpub_status st = validate(kv_latent, latent_stride, k_rope, rope_stride, index_k,
                               index_stride, slot_mapping, num_tokens, main_caches,
                               indexer_caches, num_replicas, num_blocks, block_size,
                               invalid_count, &v);
    if (st != KVPUB_OK) return st;
    if (num_tokens == 0) return ok();
    if (workspace == nullptr) return fail(KVPUB_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned(workspace, 16))
        return fail(KVPUB_ERR_ALIGNMENT, "workspace is not 16-byte aligned");
    if (workspace_bytes < kvpub_gather_workspace_bytes(num_tokens))
        return fail(KVPUB_ERR_WORKSPACE, "workspace holds %zu bytes, %zu needed", workspace_bytes,
                    kvpub_gather_workspace_bytes(num_tokens));
    return gather_then_insert(v, static_cast<uint8_t *>(workspace), (cudaStream_t)stream);
}

extern "C" kvpub_status kvpub_epoch_advance(unsigned long long *epoch, kvpub_stream_t stream) {
    if (epoch == nullptr) return fail(KVPUB_ERR_INVALID_ARG, "epoch is NULL");
    if (!aligned(epoch, 8)) return fail(KVPUB_ERR_ALIGNMENT, "epoch is not 8-byte aligned");
    (void)cudaGetLastError();
    (void)launch(epoch_advance_kernel, 1, 1, (cudaStream_t)stream, epoch);
    return launched("epoch_advance");
}

extern "C" kvpub_status kvpub_epoch_wait(const unsigned long long *epoch,
                                         unsigned long long target,
                                         unsigned long long max_polls, unsigned int *status,
                                         kvpub_stream_t stream) {
    if (epoch == nullptr || status == nullptr)
        return fail(KVPUB_ERR_INVALID_ARG, "epoch or status is NULL");
    if (!aligned(epoch, 8) || !aligned(status, 4))
        return fail(KVPUB_ERR_ALIGNMENT, "epoch or status is misaligned");
    if (max_polls < 1 || max_polls > kMaxPolls)
        return fail(KVPUB_ERR_INVALID_ARG, "max_polls %llu outside [1, %llu]", max_polls,
                    kMaxPolls);
    (void)cudaGetLastError();
    (void)launch(epoch_wait_kernel, 1, 1, (cudaStream_t)stream, epoch, target, max_polls, status);
    return launched("epoch_wait");
}

extern "C" const char *kvpub_last_error(void) { return g_last_error; }

// ------------------------------------------- allocation-free gather-insert
//
// kvpub_gather_insert with its workspace in a fixed array inside this
// library instead of caller memory, for callers that cannot allocate device
// memory.  Every GPU that loads the library holds the array
// (KVPUB_STATIC_GATHER_MAX_TOKENS rows of 1408 bytes, 5.5 MiB) until the
// process exits.  Host code cannot use the array's name as a device address:
// every call looks the address up for the current device.  The address is
// not cached, because it belongs to the device's context: after a
// cudaDeviceReset the array is reloaded at another address, and a cached
// one would point at freed memory.

static __device__ __align__(256) uint8_t
    g_static_gather_workspace[KVPUB_STATIC_GATHER_MAX_TOKENS * KVPUB_GATHER_ROW_BYTES];

namespace kvpub {
namespace {

kvpub_status static_gather_workspace(uint8_t **out) {
    int dev = 0;
    kvpub_status st = current_device(&dev);
    if (st != KVPUB_OK) return st;
    void *addr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&addr, g_static_gather_workspace);
    if (e != cudaSuccess || addr == nullptr)
        return fail(KVPUB_ERR_CUDA, "cudaGetSymbolAddress(static workspace) on device %d: %s",
                    dev, cudaGetErrorString(e));
    *out = static_cast<uint8_t *>(addr);
    return KVPUB_OK;
}

}  // namespace
}  // namespace kvpub

extern "C" kvpub_status kvpub_gather_insert_noalloc(
    const void *kv_latent, int64_t latent_stride, const void *k_rope, int64_t rope_stride,
    const void *index_k, int64_t index_stride, const int64_t *slot_mapping, int64_t num_tokens,
    void *const *main_caches, void *const *indexer_caches, int num_replicas, int64_t num_blocks,
    int block_size, unsigned long long *invalid_count, kvpub_stream_t stream) {
    Validated v;
    kvpub_status st = validate(kv_latent, latent_stride, k_rope, rope_stride, index_k,
                               index_stride, slot_mapping, num_tokens, main_caches,
                               indexer_caches, num_replicas, num_blocks, block_size,
                               invalid_count, &v);
    if (st != KVPUB_OK) return st;
    if (num_tokens > KVPUB_STATIC_GATHER_MAX_TOKENS)
        return fail(KVPUB_ERR_WORKSPACE,
                    "num_tokens %lld exceeds the static workspace limit of %d tokens",
                    (long long)num_tokens, KVPUB_STATIC_GATHER_MAX_TOKENS);
    if (num_tokens == 0) return ok();
    uint8_t *ws = nullptr;
    if ((st = static_gather_workspace(&ws)) != KVPUB_OK) return st;
    // Nothing in the array has to start at zero: the gather writes every
    // row that the inserts then read, all in stream order.
    return gather_then_insert(v, ws, (cudaStream_t)stream);
}
