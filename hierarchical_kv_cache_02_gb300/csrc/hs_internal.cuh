// Internal declarations shared by the translation units of libhisparse.
// Layouts (all row-major):
//   host history   pages of 2^page_shift records (pinned, device-mapped), found through the page
//                  table [R][L][max_pages] of device addresses (0 = not reserved); the pages of
//                  the shared prefix appear in every request's table
//   hot buffer     [L][R][B][rec]                                        (HBM)
//   tag / stamp    [L][R][B]  int32 (-1 empty) / uint32 (0 empty)
//   state          [L][R]     {clock, nres, err, pad}
//   counters       [L][R][4]  uint64 hits, misses, appends, host_bytes
//   step log       [log_steps][L][R] uint32
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "hisparse.h"

struct hs_rl_state {
  uint32_t clock;  // next stamp; starts at 1, 0 marks an empty slot
  uint32_t nres;   // resolves done: the step counter of the random key
  uint32_t err;    // hs_device_error bits
  uint32_t pad;
};

struct hs_host_pages;  // host-side page allocator and the host mirror of the page table
struct hs_dev_pages;   // device cache pool allocator and the host mirror of the slot table
constexpr int kMaxSlotPages = 64;  // device buffer pages per (request, layer)

// A miss the resolve left to the attention (fetch-in-attention mode): the device address of its
// record in the mapped host history (0: nothing pending for this top-k entry) and its slot.
struct hs_pending {
  uint64_t src;
  int32_t slot;
  int32_t pos;
};

struct hs_pool {
  hs_config cfg;
  int device;
  int num_sms;
  int64_t rec;           // record bytes
  uint64_t* page_table;  // device [R][L][max_pages]: device address of each host page, 0 = none
  int64_t max_pages;     // pages per (request, layer): ceil(capacity / page size)
  int page_shift;        // log2 of the records per page
  hs_host_pages* host;
  uint8_t* buf;          // the device cache pool: pages of slot_page slots x rec bytes
  uint64_t* slot_table;  // device [L][R][slot_pages]: device address of each buffer page, 0 = none
  int32_t* slot_cap;     // device [L][R]: slots the buffer holds, min(B, pages x slot_page)
  int slot_pages;        // pages per buffer: ceil(B / slot_page), <= kMaxSlotPages
  int slot_shift;        // log2 of the slots per page
  hs_dev_pages* dev;
  int32_t* tag;
  uint32_t* stamp;
  hs_rl_state* state;
  unsigned long long* counters;
  uint32_t* step_log;
  uint32_t* err_global;  // attention-side error bits
  hs_pending* pend;      // [L][R][k] misses the attention still has to fetch
  uint32_t* pend_live;   // [L][R] 1 while such a list is outstanding
  float* attn_part;      // split partials
  uint32_t* attn_ticket; // [R][attn_tickets_per_req]: per-group split tickets, then the pending-list count
  int attn_max_splits;
  int resolve_cs;        // CTAs per request in the resolve cluster
  int attn_tickets_per_req;
  size_t attn_part_floats;
  int debug_stall;       // HS_STALL_* bits: the next such launch leaves one barrier arrival out (test hook)
  // [L][R][2] resolve launches and resolve CTAs finished per (layer, request): an attention that
  // directly follows the resolve of its layer waits for its request's CTAs only (see k_attn_gqa)
  uint32_t* res_count;
  int last_res_layer;            // layer of the last launch if it was a whole-batch resolve, else -1
  cudaStream_t last_res_stream;  // and its stream
  int resolve_ctas;              // resolve CTAs per request and launch: cs, or 2 cs with fetch CTAs
  // early fetch (cfg.early_fetch = 1), else all null:
  int32_t* pos_slot;   // [L][R][C] slot each position was last installed in (a hint: a position is
                       // resident iff that slot is below the buffer's slot count and carries its tag)
  int32_t* fslot;      // [L][R][k] slot + 1 of each missing top-k entry of a launch (0: none), written
                       // by the deciding CTAs for the fetch CTAs; all 0 again when the launch ends
  uint32_t* fdec;      // [L][R] deciding CTAs of the launch that have written their share
  uint32_t* ffin;      // [L][R] CTAs of the launch finished (the last one clears fslot and fdec)
  uint8_t* fscratch;   // [L][R][cs x fetch_rows][rec] records fetched ahead of the decision
  int fetch_rows;      // scratch rows of one fetch CTA
};

// ---- small device helpers -------------------------------------------------

// splitmix64 output function at counter n (Steele, Lea, Flood 2014): mix(seed + n * gamma)
__device__ __forceinline__ uint64_t hs_splitmix_at(uint64_t seed, uint64_t n) {
  uint64_t z = seed + n * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// eviction key of a slot; smaller keys are evicted first, ties by lower slot
__device__ __forceinline__ uint32_t hs_evict_key(int policy, int32_t tag, uint32_t stamp, uint64_t seed,
                                                 uint32_t nres, int R, int r, int L, int l, int B, int j) {
  if (policy == HS_POLICY_RANDOM) {
    if (tag < 0) return 0u;
    uint64_t n = (((uint64_t)nres * (uint64_t)R + (uint64_t)r) * (uint64_t)L + (uint64_t)l) * (uint64_t)B + (uint64_t)j;
    return 1u + (uint32_t)(hs_splitmix_at(seed, n) >> 33);
  }
  return stamp;
}

// device address of position p of (r, l) in the mapped host history, or null when its page is not
// reserved
__device__ __forceinline__ uint8_t* hs_page_addr(const uint64_t* pt, int64_t max_pages, int shift, int64_t rec,
                                                 int L, int r, int l, int64_t p) {
  const uint64_t page = pt[((int64_t)r * L + l) * max_pages + (p >> shift)];
  if (page == 0ull) return nullptr;
  return (uint8_t*)page + (p & ((1ll << shift) - 1)) * rec;
}

// The same through one (request, layer) row of the table: a copy in shared memory, or the row in
// global memory when it is longer than a kernel caches.
constexpr int kPageRowCache = 1024;  // entries a kernel keeps in shared memory (8 KB)
__device__ __forceinline__ uint8_t* hs_page_row_addr(const uint64_t* row, int shift, int64_t rec, int64_t p) {
  const uint64_t page = row[p >> shift];
  if (page == 0ull) return nullptr;
  return (uint8_t*)page + (p & ((1ll << shift) - 1)) * rec;
}
// Copy the row of (r, l) into `cache` when it fits; returns the row to use.  Needs a barrier
// between this and the first use.
__device__ __forceinline__ const uint64_t* hs_page_row(const uint64_t* pt, int64_t max_pages, int L, int r, int l,
                                                       uint64_t* cache) {
  const uint64_t* row = pt + ((int64_t)r * L + l) * max_pages;
  if (max_pages > kPageRowCache) return row;
  for (int64_t i = threadIdx.x; i < max_pages; i += blockDim.x) cache[i] = row[i];
  return cache;
}

// Slot j of a buffer whose page row (device addresses of its pages) is `row`.
__device__ __forceinline__ uint8_t* hs_slot_addr(const uint64_t* row, int shift, int64_t rec, int j) {
  return (uint8_t*)(uintptr_t)row[j >> shift] + (int64_t)(j & ((1 << shift) - 1)) * rec;
}

// Finish the host -> slot copies that a resolve in fetch-in-attention mode left pending for
// (r, l) and that no attention has completed.  The entries [k*part/nparts, k*(part+1)/nparts) are
// copied by this CTA, one warp per record; `slots` is the buffer's page row.
__device__ __forceinline__ void hs_copy_pending(const hs_pending* pend, int k, int64_t rec, const uint64_t* slots,
                                                int slot_shift, int part, int nparts) {
  const int e0 = (int)((int64_t)k * part / nparts), e1 = (int)((int64_t)k * (part + 1) / nparts);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int nv = (int)(rec / 16);
  for (int i = e0 + warp; i < e1; i += nw) {
    const hs_pending e = pend[i];
    if (e.src == 0ull) continue;
    const uint4* src = (const uint4*)e.src;
    uint4* dst = (uint4*)hs_slot_addr(slots, slot_shift, rec, e.slot);
    for (int v = lane; v < nv; v += 32) dst[v] = src[v];
  }
}

// Alignment the kernels' vector accesses need: 16 bytes for queries, outputs and appended records
// (16-byte loads and stores), 8 for positions, 4 for top-k lists and slot lists.
inline bool hs_aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1u)) == 0; }

// Programmatic dependent launch: the hot-path kernels are launched so that the next kernel of the
// stream may start its launch while this one drains.  Every kernel waits for its predecessor's
// completion (and memory) before touching global memory, then lets its own successor launch.
__device__ __forceinline__ void hs_pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Raise a kernel's dynamic shared-memory limit to `bytes`, never lower it: pools of different
// configurations in one process share the kernel's attribute, and a later pool that needs less must
// not break the launches of an earlier one that needs more.
template <typename K>
inline cudaError_t hs_raise_smem_limit(K kern, int bytes) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, (const void*)kern);
  if (e != cudaSuccess) return e;
  if (fa.maxDynamicSharedSizeBytes >= bytes) return cudaSuccess;
  return cudaFuncSetAttribute((const void*)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// ---- phase stamps (built only with -DHS_PHASE_TRACE, for the phase tables of the profiles) ----
// Thread 0 of each of the first 256 CTAs of a launch records %globaltimer at numbered points of a
// kernel into `table` ([256][64], a device array of the kernel's translation unit, read out by its
// hs_phase_*_read function).  The normal build compiles the stamps away.
#ifdef HS_PHASE_TRACE
#define HS_PHASE(table, ev, cond)                                                                \
  do {                                                                                          \
    const unsigned _c = blockIdx.x + gridDim.x * blockIdx.y;                                    \
    if ((cond) && _c < 256u) {                                                                  \
      unsigned long long _t;                                                                    \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(_t));                                    \
      table[_c][ev] = _t;                                                                       \
    }                                                                                           \
  } while (0)
#else
#define HS_PHASE(table, ev, cond) \
  do {                            \
  } while (0)
#endif

// ---- launchers (defined in the kernel translation units) -------------------
int hs_launch_resolve(hs_pool* pool, int layer, int r0, int nreq, const int64_t* d_pos, const void* d_rec,
                      const int32_t* d_topk, int32_t* d_locs, cudaStream_t st);
int hs_launch_append(hs_pool* pool, int layer, const int64_t* d_pos, const void* d_rec, cudaStream_t st);
int hs_launch_attn(hs_pool* pool, int layer, int r0, int nreq, const void* d_q, const int32_t* d_locs,
                   const void* kv_base, int64_t kv_rows, float scale, float* d_out, cudaStream_t st);
// attention workspace requirement for a configuration (floats, splits, groups)
void hs_attn_workspace(const hs_config* cfg, int num_sms, size_t* floats, int* max_splits, int* tickets_per_req);
bool hs_attn_supported(const hs_config* cfg);
bool hs_attn_can_fetch(const hs_config* cfg);  // the attention can take over the miss fetch
int hs_attn_prepare(const hs_config* cfg, int num_sms);
int hs_resolve_prepare(hs_pool* pool);
size_t hs_resolve_smem_bytes(const hs_config* cfg);
// Dynamic shared memory of a resolve CTA at most: 227 KB less the kernel's static shared memory
// (about 29 KB) and the staging area's alignment slack.
constexpr size_t kResolveDynSmemCap = 196 * 1024;
