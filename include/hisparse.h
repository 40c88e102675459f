/*
 * hisparse.h -- C ABI of a GB300 (sm_103a) library for the decode hot path of
 * HiSparse ("HiSparse: Scaling Sparse-Attention Decoding with Hierarchical KV
 * Cache Management", as summarised on marsggbo.github.io, 2026-09-23).
 *
 * The method (summary §3): every request keeps its full per-layer KV history in
 * a host-DRAM pool (pinned; the authoritative copy).  The GPU holds only a
 * fixed B-slot hot buffer per (request, layer) with page-table and recency
 * metadata.  Each decode layer: the indexer hands over k logical positions;
 * RESOLVE looks them up in the hot buffer, fetches the misses from the host
 * pool into evicted slots and publishes the physical slot of every selected
 * position (§5); sparse attention reads exactly those slots (§3 step (4));
 * the new token's KV is written through to the host pool (§3 step (5)).
 *
 * Conventions for every call:
 *   - Pointers named d_* are device pointers (or device-visible managed memory)
 *     owned by the caller; the library never frees them.  Host pointers are
 *     named h_* or src/dst with the rule stated at the call.
 *   - Alignment of device arguments (the kernels move them with vector loads and
 *     stores): d_q, d_out, d_rec and d_kv 16 bytes, d_pos 8 bytes, d_topk and
 *     d_locs 4 bytes.  A misaligned pointer returns HS_ERR_ARG.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Calls marked CAPTURABLE only enqueue kernels on `stream`: no allocation,
 *     no host synchronisation, no read of device data by the host.  They may be
 *     captured in a CUDA graph and replayed.  Each request of a pool is used from one
 *     stream at a time; disjoint request ranges (the *_range calls) may run on
 *     different streams concurrently.
 *   - Return value: HS_OK (0) or a negative hs_status.  Argument errors found on
 *     the host return at once and enqueue nothing.  Errors that only the device
 *     can see (a bad position in a top-k list, an append out of range, a timed
 *     out wait) set bits in the pool's device error word; the kernel skips the
 *     offending entry; hs_stats reports them and returns HS_ERR_DEVICE_FLAG.
 */
#ifndef HISPARSE_H
#define HISPARSE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct hs_pool hs_pool; /* opaque; owns all pool, buffer and metadata memory */

enum hs_status {
  HS_OK = 0,
  HS_ERR_CONFIG = -1,      /* hs_config rejected (see hs_pool_create) */
  HS_ERR_ALLOC_HOST = -2,  /* pinned host allocation failed */
  HS_ERR_ALLOC_DEV = -3,   /* device allocation failed */
  HS_ERR_ARG = -4,         /* a call argument is out of range or NULL */
  HS_ERR_CUDA = -5,        /* a CUDA runtime call failed */
  HS_ERR_DEVICE_FLAG = -6, /* hs_stats: a kernel recorded an error bit */
  HS_ERR_SCRATCH = -7      /* hs_sparse_attn_noalloc: the call needs more than its fixed scratch */
};

enum hs_policy {
  HS_POLICY_LRU = 0,          /* summary §4-§5: evict the least recently used, update in place */
  HS_POLICY_FIFO = 1,         /* §4: evict the earliest inserted */
  HS_POLICY_RANDOM = 2,       /* §4: evict at random (counter-based hash, reproducible) */
  HS_POLICY_SWAP_VANILLA = 3  /* §4: keep only the current top-k, no hot set */
};

enum hs_layout {
  HS_LAYOUT_MLA = 0, /* one shared latent of head_dim_qk bf16 per token; V = its first head_dim_v values */
  HS_LAYOUT_GQA = 1  /* per token num_kv_heads blocks of [K (head_dim_qk) | V (head_dim_v)] bf16 */
};

/* bits of the device error word */
enum hs_device_error {
  HS_DEVERR_RANGE = 1,    /* a top-k entry outside [0, capacity) other than -1 */
  HS_DEVERR_DUP = 2,      /* a top-k entry repeating an earlier one in the same list */
  HS_DEVERR_CLOCK = 4,    /* the 32-bit recency clock of a (request, layer) would wrap */
  HS_DEVERR_APPEND = 8,   /* an append position outside [shared_prefix, capacity), or on a host
                             page not reserved (hs_reserve) */
  HS_DEVERR_LOC = 16,     /* an attention slot index outside [0, rows) */
  HS_DEVERR_TIMEOUT = 32, /* a bounded wait inside a kernel gave up */
  HS_DEVERR_PAGE = 64,    /* a miss fetch read a position whose host page is not reserved (the
                             slot keeps its old contents) */
  HS_DEVERR_SLOTS = 128   /* a resolve or append on a (request, layer) whose device buffer holds
                             fewer than top_k slots (device_pool_slots > 0 and not reserved):
                             the call changed nothing for it and its locations are -1 */
};

typedef struct {
  int32_t num_requests;   /* R >= 1 */
  int32_t num_layers;     /* L >= 1 */
  int64_t capacity;       /* C: positions per (request, layer), prefill plus appends */
  int64_t shared_prefix;  /* positions [0, shared_prefix) are ONE history shared by all requests
                             (read-only for appends); 0 = every request owns its whole history */
  int32_t layout;         /* hs_layout */
  int32_t num_q_heads;    /* Hq */
  int32_t num_kv_heads;   /* GQA: KV heads per token (Hq % num_kv_heads == 0); MLA: 1 */
  int32_t head_dim_qk;    /* MLA 576, GQA 128 */
  int32_t head_dim_v;     /* MLA 512, GQA 128 */
  int32_t top_k;          /* k, 1 <= k <= buffer_slots, k <= 4096 (shared-memory hash) */
  int32_t buffer_slots;   /* B: hot-buffer slots per (request, layer), <= 16384 */
  int32_t policy;         /* hs_policy */
  uint64_t seed;          /* key of HS_POLICY_RANDOM */
  int32_t io_chunk_bytes; /* bytes one thread moves per batch of loads in a miss fetch:
                             16..128, a power of two dividing the record size (summary §5: the
                             per-thread transfer size of the swap-in is a tuned knob) */
  int32_t log_steps;      /* >0: keep per-step miss counts of the first log_steps resolves */
  int32_t fetch_in_attention; /* 0: hs_resolve copies the misses into their slots (summary §5).
                                 1: hs_resolve only decides; the next hs_sparse_attn of the layer
                                 reads the missing records straight from the host history while it
                                 gathers the resident ones from HBM, and writes them to their
                                 slots, so the host-link transfer overlaps the HBM-bound attention.
                                 Copies left pending when no attention follows are finished by the
                                 next hs_resolve or hs_append_writethrough of that layer.  Needs
                                 the GQA layout. */
  int32_t host_page_tokens;   /* positions per host page (summary §8, the memory layer allocates
                                 the host pool in pages): 0 = automatic (1024, or the largest power
                                 of two <= 1024 dividing shared_prefix); else a power of two that
                                 divides shared_prefix */
  int32_t host_on_demand;     /* 0: every page of [0, capacity) is reserved at pool creation.
                                 1: pages are reserved on demand: by hs_prefill_write for the
                                 positions it writes and by hs_reserve ahead of appends; a
                                 request's private pages return to the pool with hs_release. */
  int32_t buffer_page_slots;  /* slots per device buffer page: 0 = automatic (the smallest power of
                                 two >= 16 that cuts B into at most 64 pages); else a power of two
                                 with ceil(B / buffer_page_slots) <= 64 */
  int64_t device_pool_slots;  /* summary §8, the coordinator allocates and grows the per-request,
                                 per-layer device cache on demand.  0: every (request, layer) buffer
                                 holds all B slots from creation.  > 0: the device cache pool holds
                                 this many slots (rounded up to whole pages); a buffer holds only
                                 the pages hs_reserve gave it -- min(B, max(end, top_k)) slots
                                 rounded up to a page -- and
                                 resolve and append use its slots [0, that count) alone.  With the
                                 growth kept ahead of the positions a request uses, every result is
                                 identical to the full buffer's. */
  double host_to_device_ratio; /* > 0: the pinned host history may hold at most this many times the
                                  device cache pool's bytes; reservations beyond fail with
                                  HS_ERR_ALLOC_HOST.  0: no bound. */
  int32_t early_fetch;        /* summary §5 step 4 (the swap-in), started before the decision ends.
                                 0: each hs_resolve cluster fetches its misses once it has chosen
                                 the victims.  1: every hs_resolve launch also runs one cluster of
                                 fetch CTAs per request, which do the whole miss fetch.  From the
                                 launch's start they copy the records that look missing (from the
                                 slot each position was last installed in: a device map position
                                 -> slot, confirmed by the slot's tag) from the host history into
                                 a device scratch, up to about top_k / 4 per (request, layer).
                                 Once the deciding CTAs have chosen the victims, the fetch CTAs
                                 install every miss in its slot: from the scratch when they have
                                 it, else from the host.  Results are identical to mode 0.  Extra
                                 device memory per (layer, request): 4 x capacity bytes for the
                                 map, the scratch (about top_k / 4 records) and 4 x top_k bytes.
                                 Needs fetch_in_attention = 0. */
} hs_config;

/* Record size in bytes for a configuration (MLA: 2*head_dim_qk; GQA: 2*kv_heads*(qk+v)). */
int64_t hs_record_bytes(const hs_config* cfg);

/*
 * Create a pool on `cuda_device` (summary §3, §8 "memory layer").
 *   - Host history: pinned, device-mapped pages of host_page_tokens records, carved from large
 *     pinned slabs.  A device page table [R][L][ceil(capacity / page)] maps every (request, layer,
 *     position) to its page.  The pages of [0, shared_prefix) are one copy per layer, mapped into
 *     every request's table.
 *   - Hot buffers in HBM: one device cache pool of pages of buffer_page_slots slots x rec bytes; a
 *     device slot table [L][R][ceil(B / page)] maps each (layer, request, slot) to its page.  Tags
 *     [L][R][B] (-1 = empty), stamps (0 = empty), per-(request, layer) clock (starts at 1),
 *     counters and attention workspace.  All slots start empty.
 * With host_on_demand = 0 every host page is reserved here; else none is.  With
 * device_pool_slots = 0 every buffer gets all its pages here; else none does.  Synchronous, not
 * capturable.  Errors: HS_ERR_CONFIG, HS_ERR_ALLOC_HOST, HS_ERR_ALLOC_DEV, HS_ERR_CUDA.
 * Environment HS_FAULT=alloc_host|alloc_dev makes the named allocation fail (for tests).
 */
int hs_pool_create(const hs_config* cfg, int cuda_device, hs_pool** out);

/* Free everything the pool owns.  Synchronises the device.  NULL is accepted. */
int hs_pool_destroy(hs_pool* pool);

/* Cold start: empty every slot, reset clocks, counters, error word and step log.  CAPTURABLE. */
int hs_pool_reset(hs_pool* pool, void* stream);

/*
 * Prefill write (summary §3 step (1)): copy n records from `src` (host or device memory,
 * [n][rec] bytes) into the host history of (req, layer) at positions [pos0, pos0 + n).
 * Positions below shared_prefix go to the shared history whatever `req` is.  Reserves the pages
 * it writes (synchronously), then enqueues the copy on `stream`; the caller keeps `src` alive
 * until the stream reaches this point.  Writes only the host pool; the hot buffer is filled on
 * demand by hs_resolve (a device buffer grown on demand grows only by hs_reserve).
 * Errors: HS_ERR_ARG, HS_ERR_ALLOC_HOST, HS_ERR_CUDA.
 */
int hs_prefill_write(hs_pool* pool, int req, int layer, int64_t pos0, int64_t n, const void* src,
                     void* stream);

/*
 * Write-through append (summary §3 step (5)): for every request r, record d_rec[r] (bf16,
 * [R][rec] bytes, device) becomes position d_pos[r] (int64 [R], device) of (r, layer): it is
 * stored to the host history (16-byte stores through the device mapping) and into the hot
 * buffer -- in the slot already holding d_pos[r] if any, else the slot the policy would evict
 * first over all B slots -- with stamp = clock, clock += 1.  Positions outside
 * [shared_prefix, capacity) set HS_DEVERR_APPEND and are skipped.  CAPTURABLE.
 */
int hs_append_writethrough(hs_pool* pool, int layer, const int64_t* d_pos, const void* d_rec, void* stream);

/*
 * Fused RESOLVE (summary §5).  The summary runs one CTA per request; here a thread-block cluster
 * serves each request: every CTA of the cluster computes the whole decision below from the same
 * inputs, then writes its share of the slots and fetches its share of the misses, so one request's
 * host copies are spread over several SMs.  The cluster holds the largest of 8, 4 or 2 CTAs for
 * which every request's cluster fits on the GPU at once (fixed at hs_pool_create), else 1.
 * The decision: hash the k positions of d_topk[r]
 * (int32 [R][k], device; -1 = padding) in shared memory, probe all B slots for hits, choose
 * the m victims among the slots holding no selected position (smallest eviction key, then
 * lowest slot; victims in ascending slot order take the misses in top-k order), update the
 * recency stamps in place (hits to MRU in top-k order, misses after the hits), fetch each
 * missing record from the pinned host history with 16-byte loads straight into its slot,
 * and write d_locs[r][i] = slot of d_topk[r][i] (-1 for padding or invalid entries; int32
 * [R][k], device).  Updates hits/misses/host-byte counters.  With early_fetch = 1 a second cluster
 * per request does the whole miss fetch, starting at the launch's start (see hs_config).
 * CAPTURABLE.
 */
int hs_resolve(hs_pool* pool, int layer, const int32_t* d_topk, int32_t* d_locs, void* stream);

/*
 * hs_append_writethrough followed by hs_resolve for the same layer, fused into one kernel (the
 * append's slot choice and the resolve's decision are made by the same resolve cluster): results,
 * state and counters are identical to the two calls in sequence.  Arguments as for those calls.
 * CAPTURABLE.
 */
int hs_append_resolve(hs_pool* pool, int layer, const int64_t* d_pos, const void* d_rec, const int32_t* d_topk,
                      int32_t* d_locs, void* stream);

/*
 * Sparse attention over resolved slots (summary §3 step (4)): for request r and query head h,
 *   out[r][h] = sum_i softmax_i(scale * <q[r][h], K(row_i)>) V(row_i)
 * over the entries i with d_locs[r][i] >= 0, in top-k order, with K/V taken from the record
 * layout (MLA: K = the latent, V = its first head_dim_v values; GQA: KV head h/(Hq/Hkv)).
 * d_q: bf16 [R][Hq][head_dim_qk]; d_out: fp32 [R][Hq][head_dim_v]; both device.
 * kv_base == NULL: rows are the hot-buffer slots of `layer` (kv_rows ignored).  Otherwise
 * kv_base is a caller-owned device array [R][kv_rows][rec] and d_locs index its rows
 * (fully resident KV: used to check the exactness property).  A request with no valid entry
 * gets zeros.  Entries >= rows set HS_DEVERR_LOC and are skipped.  The reduction order
 * depends only on the top-k order, so the result is bit-identical whichever slots hold the
 * records.  Enqueued directly after hs_resolve / hs_append_resolve of the same layer on the same
 * stream (nothing of this pool in between), the attention of a request may start as soon as that
 * request's resolve is done, before the rest of the resolve; results are the same either way.
 * CAPTURABLE.
 */
int hs_sparse_attn(hs_pool* pool, int layer, const void* d_q, const int32_t* d_locs, const void* kv_base,
                   int64_t kv_rows, float scale, float* d_out, void* stream);

/* Size of the fixed device scratch that hs_sparse_attn_noalloc uses on every GPU (8 MiB + 64 KiB). */
#define HS_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u + 64u * 1024u)

/*
 * Sparse attention over caller-resident KV that allocates nothing.  The paper has no counterpart:
 * this is a convenience of this library for callers that must not call cudaMalloc at all, for
 * example code inside an inference engine whose own allocator owns all device memory, or a
 * process that must keep its device footprint fixed after start-up.  Creating a pool would
 * allocate the host history and the hot buffers; this call needs none of that.
 *
 * It computes exactly what hs_sparse_attn computes with a non-NULL kv_base, with the same
 * kernels and the same split plan, so the two give bit-identical outputs: for request r and query
 * head h, softmax(scale * <q, K(row)>)-weighted V over the rows d_locs[r][i] >= 0 of d_kv, in
 * top-k order.  Only these fields of *cfg are read: num_requests, layout, num_q_heads,
 * num_kv_heads, head_dim_qk, head_dim_v, top_k (pool settings such as fetch_in_attention are
 * ignored).
 *   d_q    : bf16 [R][Hq][head_dim_qk], device          d_locs : int32 [R][k], device
 *   d_kv   : bf16 [R][kv_rows][record], device, 16-byte aligned
 *   d_out  : fp32 [R][Hq][head_dim_v], device
 * The split partials live in one file-scope device array of HS_NOALLOC_SCRATCH_BYTES per GPU,
 * loaded with the library and held until the process exits.  A shape whose partials do not fit
 * returns HS_ERR_SCRATCH before anything is enqueued (about R * splits * Hq * (head_dim_v + 2) * 4
 * bytes; splits <= number of SMs / R).  Each call first clears the combine tickets and the error
 * word it uses and fills d_out with NaN.
 * The first call on a device (with that device current) looks up the scratch's device address
 * and raises the kernels' shared-memory limits; make that first call before any stream capture.
 * Every call on a device shares the one array and finds the previous call's leftovers there:
 * calls that may overlap on the GPU (different streams without ordering) race and corrupt each
 * other's results.  Rows outside [0, kv_rows) are skipped and not reported.  A bounded wait inside
 * a kernel that gives up (about a second without progress, a stalled GPU) leaves the affected
 * requests' outputs NaN; there is no pool whose error word could report it.
 * Errors: HS_ERR_ARG, HS_ERR_CONFIG, HS_ERR_SCRATCH, HS_ERR_CUDA.
 */
int hs_sparse_attn_noalloc(const hs_config* cfg, const void* d_q, const int32_t* d_locs, const void* d_kv,
                           int64_t kv_rows, float scale, float* d_out, void* stream);

/*
 * Request-range forms (summary §3: requests are independent; each one's layers stay in order).
 * They act on requests [r0, r0 + nreq) only; d_topk, d_locs, d_pos, d_rec, d_q and d_out hold
 * rows for those requests, the first row being request r0.  hs_resolve_range fuses the
 * write-through append when d_pos and d_rec are both non-NULL (both NULL: plain resolve).
 * hs_sparse_attn_range reads the hot buffer.  Calls on disjoint ranges touch disjoint state, so
 * two micro-batches of one pool can run on two streams and overlap one's host-link fetch with the
 * other's HBM-bound attention.  Errors: HS_ERR_ARG for an empty or out-of-range span.  CAPTURABLE.
 */
int hs_resolve_range(hs_pool* pool, int layer, int r0, int nreq, const int64_t* d_pos, const void* d_rec,
                     const int32_t* d_topk, int32_t* d_locs, void* stream);
int hs_sparse_attn_range(hs_pool* pool, int layer, int r0, int nreq, const void* d_q, const int32_t* d_locs,
                         float scale, float* d_out, void* stream);

typedef struct {
  uint64_t hits;
  uint64_t misses;
  uint64_t appends;
  uint64_t host_bytes;  /* bytes fetched from the host history by hs_resolve */
  uint32_t error_bits;  /* OR of all hs_device_error bits */
  uint32_t resolves;    /* hs_resolve calls counted on (request 0, layer 0) */
} hs_totals;

/*
 * Read the device counters (synchronises the device; not capturable).  Any output may be NULL.
 *   h_counters : uint64 [R][L][4]  (hits, misses, appends, host_bytes) per (request, layer)
 *   h_errors   : uint32 [R][L]     error bits per (request, layer)
 *   h_step_log : uint32 [log_steps][R][L] misses of the t-th resolve of (r, l)
 * reset != 0 zeroes the counters, error bits and step log afterwards (not the cache state).
 * Returns HS_ERR_DEVICE_FLAG when any error bit is set, after filling the outputs.
 */
int hs_stats(hs_pool* pool, hs_totals* totals, uint64_t* h_counters, uint32_t* h_errors, uint32_t* h_step_log,
             int reset);

/*
 * Inspection (synchronous, not capturable): copy the metadata of `layer` to host memory.
 *   h_tag: int32 [R][B]; h_stamp: uint32 [R][B]; h_clock: uint32 [R]; any may be NULL.
 */
int hs_read_state(hs_pool* pool, int layer, int32_t* h_tag, uint32_t* h_stamp, uint32_t* h_clock);

/* Inspection: copy the hot buffer of (req, layer), [B][rec] bytes, to host memory `dst`; slots
 * the buffer does not hold read as zeros. */
int hs_read_buffer(hs_pool* pool, int req, int layer, void* dst);

/* Inspection: copy n records of the host history of (req, layer) from position pos0 to `dst`;
 * positions on pages not reserved read as zeros. */
int hs_read_history(hs_pool* pool, int req, int layer, int64_t pos0, int64_t n, void* dst);

/*
 * Memory layer (summary §8: paged host pool and device cache pool, grown on demand): reserve the
 * host pages of (req, layer) that cover positions [0, end) -- layer = -1: every layer -- so that
 * appends up to `end` have somewhere to go, and (device_pool_slots > 0) grow its device buffer to
 * min(B, max(end, top_k)) slots rounded up to a page.  Pages of the shared prefix are reserved
 * once per layer.  Nothing is reserved when the call fails.  Synchronous (it updates the device
 * tables); call it outside captured graphs, before the decode steps that use those positions.
 * Errors: HS_ERR_ARG, HS_ERR_ALLOC_HOST, HS_ERR_ALLOC_DEV (device cache pool exhausted), HS_ERR_CUDA.
 */
int hs_reserve(hs_pool* pool, int req, int layer, int64_t end);

/*
 * End request `req` (every layer): its private host pages, and with device_pool_slots > 0 its
 * device buffer pages, return to the free lists for reuse by later reservations; the shared prefix
 * stays.  Its buffers are emptied (tags -1, stamps 0, clock 1, resolve count 0, error bits 0, no
 * copies pending), so a new request in this index starts cold; its counters are kept.  The
 * request's history reads as zeros afterwards.  Synchronises the device first.
 * Errors: HS_ERR_ARG, HS_ERR_CUDA.
 */
int hs_release(hs_pool* pool, int req);

/*
 * Test hook for the bounded waits (not for production use): the next launch of each kernel named in
 * `kernels` leaves one mbarrier arrival out, so that the wait for it gives up after its limit (about
 * one second) instead of completing.  The kernel then reports HS_DEVERR_TIMEOUT (hs_stats) and
 * returns; its outputs for that launch are undefined, and the cache state of a resolve that gave up
 * no longer matches its history (call hs_pool_reset).  The context stays usable.
 *   HS_STALL_ATTN    : the 64-head shared-latent tensor-core attention (the producers' arrival on
 *                      the first ring slot), consumed by the next launch of that kernel
 *   HS_STALL_RESOLVE : the resolve (the arrival that completes the early miss copies), consumed by
 *                      the next resolve launch that stages early copies
 *   HS_STALL_FETCH   : the resolve's fetch CTAs (early_fetch = 1): the deciding CTAs of the
 *                      launch's first request never signal that the victims are chosen, so that
 *                      request's fetch CTAs give up waiting and install nothing.  Consumed by the
 *                      next resolve launch with fetch CTAs.
 * Host-side only (takes effect at launch, also when the launch is captured).  Errors: HS_ERR_ARG.
 */
enum { HS_STALL_ATTN = 1, HS_STALL_RESOLVE = 2, HS_STALL_FETCH = 4 };
int hs_debug_stall_next(hs_pool* pool, int kernels);

/* Host memory of the pool: pages mapped in some table, pages on the free list, pinned bytes held. */
int hs_host_usage(hs_pool* pool, int64_t* pages_in_use, int64_t* pages_free, int64_t* bytes_pinned);

/* Device cache pool: pages held by some buffer, pages free, slots per page. */
int hs_device_usage(hs_pool* pool, int64_t* pages_in_use, int64_t* pages_free, int64_t* page_slots);

#ifdef __cplusplus
}
#endif

#endif /* HISPARSE_H */
