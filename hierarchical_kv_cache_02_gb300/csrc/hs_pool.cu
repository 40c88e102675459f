// Host side of the C ABI: configuration checks, pool memory, prefill, stats and inspection.
// The memory layer follows the HiSparse summary §3 and §8: a pinned host pool holds the
// authoritative KV history; HBM holds only B slots per (request, layer) plus metadata.  The host
// pool is paged: fixed-size pages carved from large pinned, device-mapped slabs, found by the
// kernels through a device page table, reserved up front or on demand and returned to a free list.
// The hot buffers are paged the same way in one device cache pool: a (request, layer) buffer holds
// all its pages from creation, or grows page by page as its context grows (§8: the coordinator
// allocates and grows the per-request, per-layer device cache on demand).
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "hs_internal.cuh"

namespace {

bool fault_requested(const char* what) {
  const char* f = getenv("HS_FAULT");
  return f != nullptr && strstr(f, what) != nullptr;
}

bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

// records per host page: the configured power of two, or 1024, or the largest power of two <= 1024
// that divides the shared prefix (a page never mixes shared and private positions)
int64_t page_tokens_for(const hs_config* c) {
  if (c->host_page_tokens > 0) return c->host_page_tokens;
  int64_t pt = 1024;
  while (c->shared_prefix > 0 && c->shared_prefix % pt != 0) pt >>= 1;
  return pt;
}

int check_config(const hs_config* c) {
  if (c == nullptr) return HS_ERR_ARG;
  if (c->num_requests < 1 || c->num_layers < 1) return HS_ERR_CONFIG;
  if (c->capacity < 1 || c->capacity > (int64_t)INT32_MAX) return HS_ERR_CONFIG;
  if (c->shared_prefix < 0 || c->shared_prefix > c->capacity) return HS_ERR_CONFIG;
  if (c->layout != HS_LAYOUT_MLA && c->layout != HS_LAYOUT_GQA) return HS_ERR_CONFIG;
  if (c->num_q_heads < 1 || c->num_kv_heads < 1 || c->head_dim_qk < 1 || c->head_dim_v < 1) return HS_ERR_CONFIG;
  if (c->layout == HS_LAYOUT_MLA && (c->num_kv_heads != 1 || c->head_dim_v > c->head_dim_qk)) return HS_ERR_CONFIG;
  if (c->num_q_heads % c->num_kv_heads != 0) return HS_ERR_CONFIG;
  if (c->top_k < 1 || c->top_k > c->buffer_slots || c->buffer_slots > 16384) return HS_ERR_CONFIG;
  if (c->top_k > 4096) return HS_ERR_CONFIG;  // the resolve holds a thread's four top-k entries in registers
  if (c->policy < HS_POLICY_LRU || c->policy > HS_POLICY_SWAP_VANILLA) return HS_ERR_CONFIG;
  if (c->log_steps < 0) return HS_ERR_CONFIG;
  int64_t rec = hs_record_bytes(c);
  if (rec <= 0 || rec % 16 != 0) return HS_ERR_CONFIG;
  if (!is_pow2(c->io_chunk_bytes) || c->io_chunk_bytes < 16 || c->io_chunk_bytes > 128 || rec % c->io_chunk_bytes != 0)
    return HS_ERR_CONFIG;
  if (!hs_attn_supported(c)) return HS_ERR_CONFIG;
  if (hs_resolve_smem_bytes(c) > kResolveDynSmemCap) return HS_ERR_CONFIG;
  if (c->fetch_in_attention != 0 && (c->fetch_in_attention != 1 || !hs_attn_can_fetch(c))) return HS_ERR_CONFIG;
  if (c->host_page_tokens < 0 || c->host_page_tokens > (1 << 20) ||
      (c->host_page_tokens > 0 && !is_pow2(c->host_page_tokens)))
    return HS_ERR_CONFIG;
  if (c->shared_prefix > 0 && c->shared_prefix % page_tokens_for(c) != 0) return HS_ERR_CONFIG;
  if (c->host_on_demand != 0 && c->host_on_demand != 1) return HS_ERR_CONFIG;
  if (c->buffer_page_slots < 0 || c->buffer_page_slots > (1 << 20) ||
      (c->buffer_page_slots > 0 && (!is_pow2(c->buffer_page_slots) ||
                                    (c->buffer_slots + c->buffer_page_slots - 1) / c->buffer_page_slots > kMaxSlotPages)))
    return HS_ERR_CONFIG;
  if (c->device_pool_slots < 0) return HS_ERR_CONFIG;
  if (!(c->host_to_device_ratio >= 0.0) || c->host_to_device_ratio > 1e12) return HS_ERR_CONFIG;  // rejects NaN
  if (c->early_fetch != 0 && (c->early_fetch != 1 || c->fetch_in_attention != 0)) return HS_ERR_CONFIG;
  return HS_OK;
}

// slots per device buffer page: the configured power of two, or the smallest power of two >= 16
// that cuts B into at most kMaxSlotPages pages
int64_t slot_page_for(const hs_config* c) {
  if (c->buffer_page_slots > 0) return c->buffer_page_slots;
  int64_t ps = 16;
  while ((c->buffer_slots + ps - 1) / ps > kMaxSlotPages) ps <<= 1;
  return ps;
}

template <typename T>
int dev_alloc(T** p, size_t count) {
  *p = nullptr;
  if (count == 0) return HS_OK;
  if (fault_requested("alloc_dev")) return HS_ERR_ALLOC_DEV;
  if (cudaMalloc((void**)p, count * sizeof(T)) != cudaSuccess) {
    *p = nullptr;
    cudaGetLastError();
    return HS_ERR_ALLOC_DEV;
  }
  return HS_OK;
}

}  // namespace

// Pinned host pages and the host mirror of the page table.
struct hs_host_pages {
  int64_t page_tokens = 0, page_bytes = 0, shared_pages = 0;
  std::vector<std::pair<uint8_t*, uint8_t*>> slabs;       // (host, device) of each pinned slab
  std::vector<size_t> slab_bytes;
  std::vector<std::pair<uint8_t*, uint8_t*>> free_pages;  // (host, device)
  std::vector<uint8_t*> host_pt;                          // [R][L][max_pages] host address, null = none
  std::vector<uint64_t> dev_pt;                           // the same pages' device addresses
  int64_t pages_in_use = 0;
};

// The device cache pool: pages of page_slots slots, and the host mirror of the slot table.
struct hs_dev_pages {
  int64_t page_slots = 0, page_bytes = 0, total_pages = 0;
  bool on_demand = false;               // device_pool_slots > 0: buffers grow page by page
  std::vector<int64_t> free_pages;      // page indices; the next one handed out is at the back
  std::vector<uint64_t> table;          // [L][R][slot_pages] device address of each page, 0 = none
  std::vector<int32_t> npages;          // [L][R] pages each buffer holds (its first ones, in order)
  int64_t pages_in_use = 0;
};

namespace {

int host_alloc(uint8_t** h, uint8_t** d, size_t bytes) {
  *h = nullptr;
  *d = nullptr;
  if (bytes == 0) return HS_OK;
  if (fault_requested("alloc_host")) return HS_ERR_ALLOC_HOST;
  if (cudaHostAlloc((void**)h, bytes, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
    *h = nullptr;
    cudaGetLastError();
    return HS_ERR_ALLOC_HOST;
  }
  if (cudaHostGetDevicePointer((void**)d, *h, 0) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  return HS_OK;
}

void free_pool(hs_pool* p) {
  if (p == nullptr) return;
  if (p->host != nullptr) {
    for (auto& sl : p->host->slabs) cudaFreeHost(sl.first);
    delete p->host;
  }
  delete p->dev;
  cudaFree(p->page_table);
  cudaFree(p->slot_table);
  cudaFree(p->slot_cap);
  cudaFree(p->buf);
  cudaFree(p->tag);
  cudaFree(p->stamp);
  cudaFree(p->state);
  cudaFree(p->counters);
  cudaFree(p->step_log);
  cudaFree(p->err_global);
  cudaFree(p->res_count);
  cudaFree(p->attn_part);
  cudaFree(p->attn_ticket);
  cudaFree(p->pend);
  cudaFree(p->pend_live);
  cudaFree(p->pos_slot);
  cudaFree(p->fslot);
  cudaFree(p->fdec);
  cudaFree(p->ffin);
  cudaFree(p->fscratch);
  delete p;
}

__global__ void k_reset(int32_t* tag, uint32_t* stamp, size_t nslots, hs_rl_state* state, size_t nrl) {
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t j = i; j < nslots; j += stride) {
    tag[j] = -1;
    stamp[j] = 0u;
  }
  for (size_t j = i; j < nrl; j += stride) {
    hs_rl_state s;
    s.clock = 1u;
    s.nres = 0u;
    s.err = 0u;
    s.pad = 0u;
    state[j] = s;
  }
}

size_t slots_total(const hs_pool* p) {
  return (size_t)p->cfg.num_layers * p->cfg.num_requests * p->cfg.buffer_slots;
}

size_t rl_total(const hs_pool* p) { return (size_t)p->cfg.num_layers * p->cfg.num_requests; }

int do_reset(hs_pool* p, cudaStream_t st) {
  p->last_res_layer = -1;
  size_t ns = slots_total(p), nrl = rl_total(p);
  int blocks = (int)std::min<size_t>((ns + 255) / 256, (size_t)p->num_sms * 8);
  k_reset<<<blocks, 256, 0, st>>>(p->tag, p->stamp, ns, p->state, nrl);
  if (cudaMemsetAsync(p->counters, 0, nrl * 4 * sizeof(unsigned long long), st) != cudaSuccess) return HS_ERR_CUDA;
  if (p->step_log && cudaMemsetAsync(p->step_log, 0, (size_t)p->cfg.log_steps * nrl * sizeof(uint32_t), st) != cudaSuccess)
    return HS_ERR_CUDA;
  if (cudaMemsetAsync(p->err_global, 0, sizeof(uint32_t), st) != cudaSuccess) return HS_ERR_CUDA;
  if (p->pend_live && cudaMemsetAsync(p->pend_live, 0, nrl * sizeof(uint32_t), st) != cudaSuccess) return HS_ERR_CUDA;
  if (cudaMemsetAsync(p->attn_ticket, 0, (size_t)p->cfg.num_requests * p->attn_tickets_per_req * sizeof(uint32_t), st) !=
      cudaSuccess)
    return HS_ERR_CUDA;
  if (p->fslot != nullptr &&
      (cudaMemsetAsync(p->fslot, 0, nrl * p->cfg.top_k * sizeof(int32_t), st) != cudaSuccess ||
       cudaMemsetAsync(p->fdec, 0, nrl * sizeof(uint32_t), st) != cudaSuccess ||
       cudaMemsetAsync(p->ffin, 0, nrl * sizeof(uint32_t), st) != cudaSuccess))
    return HS_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

// Pinned slabs.  The GPU reads scattered host rows faster from few large mappings than from many
// small ones: on the 16-request, 32-layer GQA decode workload (17 GB of history) one slab for the
// whole reservation decodes as fast as flat arrays, while one 516 MB slab per (request, layer) cost
// 4-15% (slower miss copies).  So a reservation made at creation takes a single slab; a slab made
// on demand is at least kSlabMin and at least a quarter of what is already pinned (few slabs as the
// pool grows, at most a quarter over-reserved), never more pages than the page table could still take.
constexpr size_t kSlabMin = (size_t)256 << 20;

// bytes of the device cache pool (the base of host_to_device_ratio)
int64_t dev_pool_bytes(const hs_pool* p) { return p->dev->total_pages * p->dev->page_bytes; }

// n more pages on the free list
int grow_free_pages(hs_pool* p, int64_t n) {
  hs_host_pages& h = *p->host;
  while ((int64_t)h.free_pages.size() < n) {
    const int64_t want = n - (int64_t)h.free_pages.size();
    const int64_t R = p->cfg.num_requests, L = p->cfg.num_layers;  // distinct pages: shared ones once per layer
    const int64_t room = L * h.shared_pages + R * L * (p->max_pages - h.shared_pages) - h.pages_in_use -
                         (int64_t)h.free_pages.size();
    size_t pinned = 0;
    for (size_t b : h.slab_bytes) pinned += b;
    const int64_t min_pages = std::max<int64_t>(1, (int64_t)(std::max(kSlabMin, pinned / 4) / (size_t)h.page_bytes));
    int64_t np = std::max(want, std::min(min_pages, room));
    if (p->cfg.host_to_device_ratio > 0.0) {  // the host pool's bound relative to the device cache pool
      const double limit = p->cfg.host_to_device_ratio * (double)dev_pool_bytes(p);
      const int64_t allow = (int64_t)((limit - (double)pinned) / (double)h.page_bytes);
      if (allow < want) return HS_ERR_ALLOC_HOST;
      np = std::min(np, allow);
    }
    uint8_t *hp = nullptr, *dp = nullptr;
    int rc = host_alloc(&hp, &dp, (size_t)(np * h.page_bytes));
    if (rc != HS_OK) {
      if (hp) cudaFreeHost(hp);
      return rc;
    }
    h.slabs.push_back({hp, dp});
    h.slab_bytes.push_back((size_t)(np * h.page_bytes));
    for (int64_t i = np - 1; i >= 0; --i) h.free_pages.push_back({hp + i * h.page_bytes, dp + i * h.page_bytes});
  }
  return HS_OK;
}

// host pages of (req, layer) among [pg0, pg1) that have none yet
int64_t host_pages_missing(const hs_pool* p, int req, int layer, int64_t pg0, int64_t pg1) {
  const hs_host_pages& h = *p->host;
  int64_t need = 0;
  for (int64_t g = pg0; g < std::min(pg1, p->max_pages); ++g)
    if (h.host_pt[((int64_t)req * p->cfg.num_layers + layer) * p->max_pages + g] == nullptr) ++need;
  return need;
}

// Give every missing page of pages [pg0, pg1) of (req, layer) a page; the shared prefix's pages are
// one per layer, mapped into every request's table.  Updates the host mirror only; *changed is set
// when an entry changed.
int reserve_pages(hs_pool* p, int req, int layer, int64_t pg0, int64_t pg1, bool* changed) {
  hs_host_pages& h = *p->host;
  const int R = p->cfg.num_requests, L = p->cfg.num_layers;
  pg1 = std::min(pg1, p->max_pages);
  const int64_t need = host_pages_missing(p, req, layer, pg0, pg1);
  if (need == 0) return HS_OK;
  int rc = grow_free_pages(p, need);
  if (rc != HS_OK) return rc;
  for (int64_t g = pg0; g < pg1; ++g) {
    const int64_t e = ((int64_t)req * L + layer) * p->max_pages + g;
    if (h.host_pt[e] != nullptr) continue;
    const auto pg = h.free_pages.back();
    h.free_pages.pop_back();
    ++h.pages_in_use;
    const int r0 = g < h.shared_pages ? 0 : req, r1 = g < h.shared_pages ? R : req + 1;
    for (int r = r0; r < r1; ++r) {  // a shared page appears in every request's table
      const int64_t er = ((int64_t)r * L + layer) * p->max_pages + g;
      h.host_pt[er] = pg.first;
      h.dev_pt[er] = (uint64_t)(uintptr_t)pg.second;
    }
    *changed = true;
  }
  return HS_OK;
}

// device buffer pages (req, layer) needs to cover positions [0, end): min(B, max(end, k)) slots
int64_t dev_pages_missing(const hs_pool* p, int req, int layer, int64_t end) {
  const hs_dev_pages& d = *p->dev;
  if (!d.on_demand) return 0;
  const int64_t want = std::min<int64_t>(p->cfg.buffer_slots, std::max<int64_t>(end, p->cfg.top_k));
  const int64_t np = (want + d.page_slots - 1) / d.page_slots;
  return std::max<int64_t>(0, np - d.npages[(int64_t)layer * p->cfg.num_requests + req]);
}

// Grow the buffer of (req, layer) by `n` pages from the free list (the caller checked they exist).
void grow_buffer(hs_pool* p, int req, int layer, int64_t n, bool* changed) {
  hs_dev_pages& d = *p->dev;
  const int64_t rl = (int64_t)layer * p->cfg.num_requests + req;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t pg = d.free_pages.back();
    d.free_pages.pop_back();
    d.table[rl * p->slot_pages + d.npages[rl]] = (uint64_t)(uintptr_t)(p->buf + pg * d.page_bytes);
    ++d.npages[rl];
    ++d.pages_in_use;
    *changed = true;
  }
}

// Reserve, for request `req` and layers [l0, l1), host pages [pg0, pg1) and (dev_end >= 0) device
// slots covering positions [0, dev_end); all or nothing.
int reserve_range(hs_pool* p, int req, int l0, int l1, int64_t pg0, int64_t pg1, int64_t dev_end, bool* changed) {
  int64_t host_need = 0, dev_need = 0;
  for (int l = l0; l < l1; ++l) {
    host_need += host_pages_missing(p, req, l, pg0, pg1);
    if (dev_end >= 0) dev_need += dev_pages_missing(p, req, l, dev_end);
  }
  if (dev_need > (int64_t)p->dev->free_pages.size()) return HS_ERR_ALLOC_DEV;
  int rc = grow_free_pages(p, host_need);
  if (rc != HS_OK) return rc;
  for (int l = l0; l < l1; ++l) {
    rc = reserve_pages(p, req, l, pg0, pg1, changed);  // cannot fail: the free list holds enough
    if (rc != HS_OK) return rc;
    if (dev_end >= 0) grow_buffer(p, req, l, dev_pages_missing(p, req, l, dev_end), changed);
  }
  return HS_OK;
}

// Both tables to the device, after every kernel that may read them has finished.
int upload_tables(hs_pool* p) {
  const hs_dev_pages& d = *p->dev;
  std::vector<int32_t> cap(d.npages.size());
  for (size_t i = 0; i < cap.size(); ++i)
    cap[i] = (int32_t)std::min<int64_t>(p->cfg.buffer_slots, d.npages[i] * d.page_slots);
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(p->page_table, p->host->dev_pt.data(), p->host->dev_pt.size() * sizeof(uint64_t),
                 cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(p->slot_table, d.table.data(), d.table.size() * sizeof(uint64_t), cudaMemcpyHostToDevice) !=
          cudaSuccess ||
      cudaMemcpy(p->slot_cap, cap.data(), cap.size() * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  return HS_OK;
}

// A released request starts cold: empty slots, clock 1, no resolves, no errors, nothing pending.
__global__ void k_release(int32_t* tag, uint32_t* stamp, hs_rl_state* state, uint32_t* pend_live, int R, int L, int B,
                          int req) {
  const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x, stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = i0; i < (size_t)L * B; i += stride) {
    const size_t e = ((i / B) * R + req) * B + i % B;
    tag[e] = -1;
    stamp[e] = 0u;
  }
  for (size_t l = i0; l < (size_t)L; l += stride) {
    hs_rl_state s;
    s.clock = 1u;
    s.nres = 0u;
    s.err = 0u;
    s.pad = 0u;
    state[l * R + req] = s;
    if (pend_live != nullptr) pend_live[l * R + req] = 0u;
  }
}

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

}  // namespace

extern "C" int64_t hs_record_bytes(const hs_config* c) {
  if (c == nullptr) return -1;
  if (c->layout == HS_LAYOUT_MLA) return 2 * (int64_t)c->head_dim_qk;
  return 2 * (int64_t)c->num_kv_heads * ((int64_t)c->head_dim_qk + c->head_dim_v);
}

extern "C" int hs_pool_create(const hs_config* cfg, int cuda_device, hs_pool** out) {
  if (out == nullptr) return HS_ERR_ARG;
  *out = nullptr;
  int rc = check_config(cfg);
  if (rc != HS_OK) return rc;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || cuda_device < 0 || cuda_device >= ndev) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  DeviceGuard guard(cuda_device);
  hs_pool* p = new hs_pool();
  memset(p, 0, sizeof(*p));
  p->last_res_layer = -1;
  p->cfg = *cfg;
  p->device = cuda_device;
  cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, cuda_device);
  p->rec = hs_record_bytes(cfg);
  const size_t R = cfg->num_requests, L = cfg->num_layers, B = cfg->buffer_slots;
  // the device cache pool and its slot table (first: the host pool's bound refers to its size)
  p->dev = new hs_dev_pages();
  hs_dev_pages& d = *p->dev;
  d.page_slots = slot_page_for(cfg);
  d.page_bytes = d.page_slots * p->rec;
  d.on_demand = cfg->device_pool_slots > 0;
  p->slot_pages = (int)((B + d.page_slots - 1) / d.page_slots);
  p->slot_shift = 0;
  while ((1ll << p->slot_shift) < d.page_slots) ++p->slot_shift;
  d.total_pages = d.on_demand ? (cfg->device_pool_slots + d.page_slots - 1) / d.page_slots
                              : (int64_t)(L * R) * p->slot_pages;
  d.table.assign(L * R * (size_t)p->slot_pages, 0ull);
  d.npages.assign(L * R, 0);
  rc = dev_alloc(&p->buf, (size_t)(d.total_pages * d.page_bytes));
  if (rc == HS_OK) rc = dev_alloc(&p->slot_table, d.table.size());
  if (rc == HS_OK) rc = dev_alloc(&p->slot_cap, L * R);
  if (rc == HS_OK) {
    if (d.on_demand) {  // every page free, page 0 handed out first
      for (int64_t i = d.total_pages - 1; i >= 0; --i) d.free_pages.push_back(i);
    } else {  // buffer (l, r) holds pages [(l R + r) P, (l R + r + 1) P): the flat [L][R][B] layout
      for (size_t rl = 0; rl < L * R; ++rl) {
        for (int i = 0; i < p->slot_pages; ++i)
          d.table[rl * p->slot_pages + i] = (uint64_t)(uintptr_t)(p->buf + ((int64_t)rl * p->slot_pages + i) * d.page_bytes);
        d.npages[rl] = p->slot_pages;
      }
      d.pages_in_use = d.total_pages;
    }
  }
  // host pages and their table
  p->host = new hs_host_pages();
  p->host->page_tokens = page_tokens_for(cfg);
  p->host->page_bytes = p->host->page_tokens * p->rec;
  p->host->shared_pages = cfg->shared_prefix / p->host->page_tokens;
  p->page_shift = 0;
  while ((1ll << p->page_shift) < p->host->page_tokens) ++p->page_shift;
  p->max_pages = (cfg->capacity + p->host->page_tokens - 1) / p->host->page_tokens;
  p->host->host_pt.assign(R * L * (size_t)p->max_pages, nullptr);
  p->host->dev_pt.assign(R * L * (size_t)p->max_pages, 0ull);
  if (rc == HS_OK) rc = dev_alloc(&p->page_table, R * L * (size_t)p->max_pages);
  if (rc == HS_OK && cfg->host_on_demand == 0) {  // every page of [0, capacity) now, from one slab
    const int64_t sp = p->host->shared_pages;
    rc = grow_free_pages(p, (int64_t)L * sp + (int64_t)(R * L) * (p->max_pages - sp));  // all of them
    bool changed = false;
    for (int r = 0; rc == HS_OK && r < (int)R; ++r)
      for (int l = 0; rc == HS_OK && l < (int)L; ++l) rc = reserve_pages(p, r, l, 0, p->max_pages, &changed);
  }
  if (rc == HS_OK) rc = upload_tables(p);
  if (rc == HS_OK) rc = dev_alloc(&p->tag, L * R * B);
  if (rc == HS_OK) rc = dev_alloc(&p->stamp, L * R * B);
  if (rc == HS_OK) rc = dev_alloc(&p->state, L * R);
  if (rc == HS_OK) rc = dev_alloc(&p->counters, L * R * 4);
  if (rc == HS_OK) rc = dev_alloc(&p->step_log, (size_t)cfg->log_steps * L * R);
  if (rc == HS_OK) rc = dev_alloc(&p->err_global, 1);
  if (rc == HS_OK) rc = dev_alloc(&p->res_count, L * R * 2);
  if (rc == HS_OK && cudaMemset(p->res_count, 0, L * R * 2 * sizeof(uint32_t)) != cudaSuccess) rc = HS_ERR_CUDA;
  if (rc == HS_OK) {
    hs_attn_workspace(cfg, p->num_sms, &p->attn_part_floats, &p->attn_max_splits, &p->attn_tickets_per_req);
    rc = dev_alloc(&p->attn_part, p->attn_part_floats);
  }
  if (rc == HS_OK) rc = dev_alloc(&p->attn_ticket, R * (size_t)p->attn_tickets_per_req);
  if (rc == HS_OK && cfg->fetch_in_attention) {
    rc = dev_alloc(&p->pend, L * R * (size_t)cfg->top_k);
    if (rc == HS_OK) rc = dev_alloc(&p->pend_live, L * R);
  }
  if (rc == HS_OK) rc = hs_resolve_prepare(p);
  p->resolve_ctas = p->resolve_cs;
  if (rc == HS_OK && cfg->early_fetch) {
    // the position -> slot map (every entry -1: no position installed yet), the miss slots and
    // counters (cleared by do_reset), and about top_k / 4 scratch records per (layer, request)
    // fetch CTAs per request: as many as deciding CTAs (one per request measured far slower: a
    // single SM cannot keep enough of a request's records in flight)
    const int fpr = p->resolve_cs;
    p->resolve_ctas = p->resolve_cs + fpr;
    p->fetch_rows = (cfg->top_k + 4 * fpr - 1) / (4 * fpr);
    rc = dev_alloc(&p->pos_slot, L * R * (size_t)cfg->capacity);
    if (rc == HS_OK && cudaMemset(p->pos_slot, 0xff, L * R * (size_t)cfg->capacity * sizeof(int32_t)) != cudaSuccess)
      rc = HS_ERR_CUDA;
    if (rc == HS_OK) rc = dev_alloc(&p->fslot, L * R * (size_t)cfg->top_k);
    if (rc == HS_OK) rc = dev_alloc(&p->fdec, L * R);
    if (rc == HS_OK) rc = dev_alloc(&p->ffin, L * R);
    if (rc == HS_OK) rc = dev_alloc(&p->fscratch, L * R * (size_t)fpr * p->fetch_rows * (size_t)p->rec);
  }
  if (rc == HS_OK) rc = hs_attn_prepare(cfg, p->num_sms);
  if (rc == HS_OK) rc = do_reset(p, 0);
  if (rc == HS_OK && cudaDeviceSynchronize() != cudaSuccess) rc = HS_ERR_CUDA;
  if (rc != HS_OK) {
    cudaGetLastError();
    free_pool(p);
    return rc;
  }
  *out = p;
  return HS_OK;
}

extern "C" int hs_pool_destroy(hs_pool* pool) {
  if (pool == nullptr) return HS_OK;
  DeviceGuard guard(pool->device);
  cudaDeviceSynchronize();
  free_pool(pool);
  return HS_OK;
}

extern "C" int hs_pool_reset(hs_pool* pool, void* stream) {
  if (pool == nullptr) return HS_ERR_ARG;
  DeviceGuard guard(pool->device);
  return do_reset(pool, (cudaStream_t)stream);
}

extern "C" int hs_prefill_write(hs_pool* pool, int req, int layer, int64_t pos0, int64_t n, const void* src,
                                void* stream) {
  if (pool == nullptr || src == nullptr) return HS_ERR_ARG;
  const hs_config& c = pool->cfg;
  if (req < 0 || req >= c.num_requests || layer < 0 || layer >= c.num_layers) return HS_ERR_ARG;
  if (pos0 < 0 || n < 0 || pos0 + n > c.capacity) return HS_ERR_ARG;
  if (n == 0) return HS_OK;
  DeviceGuard guard(pool->device);
  hs_host_pages& h = *pool->host;
  const int64_t pt = h.page_tokens, rec = pool->rec;
  bool changed = false;
  int rc = reserve_range(pool, req, layer, layer + 1, pos0 / pt, (pos0 + n + pt - 1) / pt, -1, &changed);
  if (rc != HS_OK) return rc;
  if (changed && (rc = upload_tables(pool)) != HS_OK) return rc;
  const uint8_t* s = (const uint8_t*)src;
  cudaStream_t st = (cudaStream_t)stream;
  pool->last_res_layer = -1;
  for (int64_t a = pos0; a < pos0 + n;) {  // one copy per page
    const int64_t b = std::min(pos0 + n, (a / pt + 1) * pt);
    uint8_t* dst = h.host_pt[((int64_t)req * c.num_layers + layer) * pool->max_pages + a / pt] + (a % pt) * rec;
    if (cudaMemcpyAsync(dst, s, (size_t)((b - a) * rec), cudaMemcpyDefault, st) != cudaSuccess) return HS_ERR_CUDA;
    s += (b - a) * rec;
    a = b;
  }
  return HS_OK;
}

extern "C" int hs_reserve(hs_pool* pool, int req, int layer, int64_t end) {
  if (pool == nullptr) return HS_ERR_ARG;
  const hs_config& c = pool->cfg;
  if (req < 0 || req >= c.num_requests || layer < -1 || layer >= c.num_layers) return HS_ERR_ARG;
  if (end < 0 || end > c.capacity) return HS_ERR_ARG;
  DeviceGuard guard(pool->device);
  const int64_t pg1 = (end + pool->host->page_tokens - 1) / pool->host->page_tokens;
  bool changed = false;
  int rc = reserve_range(pool, req, layer < 0 ? 0 : layer, layer < 0 ? c.num_layers : layer + 1, 0, pg1, end, &changed);
  if (rc == HS_OK && changed) rc = upload_tables(pool);
  return rc;
}

extern "C" int hs_release(hs_pool* pool, int req) {
  if (pool == nullptr || req < 0 || req >= pool->cfg.num_requests) return HS_ERR_ARG;
  DeviceGuard guard(pool->device);
  if (cudaDeviceSynchronize() != cudaSuccess) return HS_ERR_CUDA;  // no kernel reads them any more
  hs_host_pages& h = *pool->host;
  const int L = pool->cfg.num_layers;
  bool changed = false;
  for (int l = 0; l < L; ++l) {
    for (int64_t g = h.shared_pages; g < pool->max_pages; ++g) {
      const int64_t e = ((int64_t)req * L + l) * pool->max_pages + g;
      if (h.host_pt[e] == nullptr) continue;
      h.free_pages.push_back({h.host_pt[e], (uint8_t*)(uintptr_t)h.dev_pt[e]});
      h.host_pt[e] = nullptr;
      h.dev_pt[e] = 0ull;
      --h.pages_in_use;
      changed = true;
    }
  }
  hs_dev_pages& d = *pool->dev;
  const int R = pool->cfg.num_requests;
  if (d.on_demand) {
    for (int l = 0; l < L; ++l) {
      const int64_t rl = (int64_t)l * R + req;
      for (int i = d.npages[rl] - 1; i >= 0; --i) {
        uint64_t& e = d.table[rl * pool->slot_pages + i];
        d.free_pages.push_back((int64_t)(((uint8_t*)(uintptr_t)e - pool->buf) / d.page_bytes));
        e = 0ull;
        --d.pages_in_use;
        changed = true;
      }
      d.npages[rl] = 0;
    }
  }
  const int B = pool->cfg.buffer_slots;
  k_release<<<std::min(pool->num_sms * 4, (L * B + 255) / 256), 256>>>(pool->tag, pool->stamp, pool->state,
                                                                       pool->pend_live, R, L, B, req);
  if (cudaGetLastError() != cudaSuccess) return HS_ERR_CUDA;
  if (changed) return upload_tables(pool);  // synchronises after the reset
  return cudaDeviceSynchronize() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

extern "C" int hs_device_usage(hs_pool* pool, int64_t* pages_in_use, int64_t* pages_free, int64_t* page_slots) {
  if (pool == nullptr) return HS_ERR_ARG;
  const hs_dev_pages& d = *pool->dev;
  if (pages_in_use) *pages_in_use = d.pages_in_use;
  if (pages_free) *pages_free = d.on_demand ? (int64_t)d.free_pages.size() : 0;
  if (page_slots) *page_slots = d.page_slots;
  return HS_OK;
}

extern "C" int hs_debug_stall_next(hs_pool* pool, int kernels) {
  if (pool == nullptr || (kernels & ~(HS_STALL_ATTN | HS_STALL_RESOLVE | HS_STALL_FETCH)) != 0) return HS_ERR_ARG;
  pool->debug_stall |= kernels;
  return HS_OK;
}

extern "C" int hs_host_usage(hs_pool* pool, int64_t* pages_in_use, int64_t* pages_free, int64_t* bytes_pinned) {
  if (pool == nullptr) return HS_ERR_ARG;
  const hs_host_pages& h = *pool->host;
  size_t b = 0;
  for (size_t x : h.slab_bytes) b += x;
  if (pages_in_use) *pages_in_use = h.pages_in_use;
  if (pages_free) *pages_free = (int64_t)h.free_pages.size();
  if (bytes_pinned) *bytes_pinned = (int64_t)b;
  return HS_OK;
}

extern "C" int hs_append_writethrough(hs_pool* pool, int layer, const int64_t* d_pos, const void* d_rec,
                                      void* stream) {
  if (pool == nullptr || d_pos == nullptr || d_rec == nullptr) return HS_ERR_ARG;
  if (!hs_aligned(d_pos, 8) || !hs_aligned(d_rec, 16)) return HS_ERR_ARG;
  if (layer < 0 || layer >= pool->cfg.num_layers) return HS_ERR_ARG;
  DeviceGuard guard(pool->device);
  return hs_launch_append(pool, layer, d_pos, d_rec, (cudaStream_t)stream);
}

extern "C" int hs_resolve(hs_pool* pool, int layer, const int32_t* d_topk, int32_t* d_locs, void* stream) {
  if (pool == nullptr || d_topk == nullptr || d_locs == nullptr) return HS_ERR_ARG;
  if (!hs_aligned(d_topk, 4) || !hs_aligned(d_locs, 4)) return HS_ERR_ARG;
  if (layer < 0 || layer >= pool->cfg.num_layers) return HS_ERR_ARG;
  DeviceGuard guard(pool->device);
  return hs_launch_resolve(pool, layer, 0, pool->cfg.num_requests, nullptr, nullptr, d_topk, d_locs,
                           (cudaStream_t)stream);
}

extern "C" int hs_append_resolve(hs_pool* pool, int layer, const int64_t* d_pos, const void* d_rec,
                                 const int32_t* d_topk, int32_t* d_locs, void* stream) {
  if (pool == nullptr || d_pos == nullptr || d_rec == nullptr || d_topk == nullptr || d_locs == nullptr)
    return HS_ERR_ARG;
  if (!hs_aligned(d_pos, 8) || !hs_aligned(d_rec, 16) || !hs_aligned(d_topk, 4) || !hs_aligned(d_locs, 4))
    return HS_ERR_ARG;
  if (layer < 0 || layer >= pool->cfg.num_layers) return HS_ERR_ARG;
  DeviceGuard guard(pool->device);
  return hs_launch_resolve(pool, layer, 0, pool->cfg.num_requests, d_pos, d_rec, d_topk, d_locs,
                           (cudaStream_t)stream);
}

extern "C" int hs_resolve_range(hs_pool* pool, int layer, int r0, int nreq, const int64_t* d_pos, const void* d_rec,
                                const int32_t* d_topk, int32_t* d_locs, void* stream) {
  if (pool == nullptr || d_topk == nullptr || d_locs == nullptr) return HS_ERR_ARG;
  if ((d_pos == nullptr) != (d_rec == nullptr)) return HS_ERR_ARG;
  if (!hs_aligned(d_pos, 8) || !hs_aligned(d_rec, 16) || !hs_aligned(d_topk, 4) || !hs_aligned(d_locs, 4))
    return HS_ERR_ARG;
  if (layer < 0 || layer >= pool->cfg.num_layers) return HS_ERR_ARG;
  if (r0 < 0 || nreq < 1 || r0 + nreq > pool->cfg.num_requests) return HS_ERR_ARG;
  DeviceGuard guard(pool->device);
  return hs_launch_resolve(pool, layer, r0, nreq, d_pos, d_rec, d_topk, d_locs, (cudaStream_t)stream);
}

extern "C" int hs_sparse_attn(hs_pool* pool, int layer, const void* d_q, const int32_t* d_locs,
                              const void* kv_base, int64_t kv_rows, float scale, float* d_out, void* stream) {
  if (pool == nullptr || d_q == nullptr || d_locs == nullptr || d_out == nullptr) return HS_ERR_ARG;
  if (!hs_aligned(d_q, 16) || !hs_aligned(d_out, 16) || !hs_aligned(d_locs, 4)) return HS_ERR_ARG;
  if (layer < 0 || layer >= pool->cfg.num_layers) return HS_ERR_ARG;
  if (kv_base != nullptr && (kv_rows < 1 || kv_rows > (int64_t)INT32_MAX)) return HS_ERR_ARG;
  DeviceGuard guard(pool->device);
  return hs_launch_attn(pool, layer, 0, pool->cfg.num_requests, d_q, d_locs, kv_base, kv_rows, scale, d_out,
                        (cudaStream_t)stream);
}

extern "C" int hs_sparse_attn_range(hs_pool* pool, int layer, int r0, int nreq, const void* d_q, const int32_t* d_locs,
                                    float scale, float* d_out, void* stream) {
  if (pool == nullptr || d_q == nullptr || d_locs == nullptr || d_out == nullptr) return HS_ERR_ARG;
  if (!hs_aligned(d_q, 16) || !hs_aligned(d_out, 16) || !hs_aligned(d_locs, 4)) return HS_ERR_ARG;
  if (layer < 0 || layer >= pool->cfg.num_layers) return HS_ERR_ARG;
  if (r0 < 0 || nreq < 1 || r0 + nreq > pool->cfg.num_requests) return HS_ERR_ARG;
  DeviceGuard guard(pool->device);
  return hs_launch_attn(pool, layer, r0, nreq, d_q, d_locs, nullptr, 0, scale, d_out, (cudaStream_t)stream);
}

extern "C" int hs_stats(hs_pool* pool, hs_totals* totals, uint64_t* h_counters, uint32_t* h_errors,
                        uint32_t* h_step_log, int reset) {
  if (pool == nullptr) return HS_ERR_ARG;
  DeviceGuard guard(pool->device);
  const int R = pool->cfg.num_requests, L = pool->cfg.num_layers;
  const size_t nrl = (size_t)R * L;
  if (cudaDeviceSynchronize() != cudaSuccess) return HS_ERR_CUDA;
  std::vector<unsigned long long> cnt(nrl * 4);
  std::vector<hs_rl_state> st(nrl);
  std::vector<uint32_t> log((size_t)pool->cfg.log_steps * nrl);
  uint32_t eg = 0;
  if (cudaMemcpy(cnt.data(), pool->counters, cnt.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost) !=
          cudaSuccess ||
      cudaMemcpy(st.data(), pool->state, st.size() * sizeof(hs_rl_state), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(&eg, pool->err_global, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return HS_ERR_CUDA;
  if (!log.empty() && cudaMemcpy(log.data(), pool->step_log, log.size() * sizeof(uint32_t), cudaMemcpyDeviceToHost) !=
                          cudaSuccess)
    return HS_ERR_CUDA;
  hs_totals t;
  memset(&t, 0, sizeof t);
  t.error_bits = eg;
  // device layout [L][R]; the API layout is [R][L]
  for (int r = 0; r < R; ++r) {
    for (int l = 0; l < L; ++l) {
      size_t d = (size_t)l * R + r, a = (size_t)r * L + l;
      t.hits += cnt[d * 4 + 0];
      t.misses += cnt[d * 4 + 1];
      t.appends += cnt[d * 4 + 2];
      t.host_bytes += cnt[d * 4 + 3];
      t.error_bits |= st[d].err;
      if (h_counters)
        for (int x = 0; x < 4; ++x) h_counters[a * 4 + x] = cnt[d * 4 + x];
      if (h_errors) h_errors[a] = st[d].err;
      if (h_step_log)
        for (int s = 0; s < pool->cfg.log_steps; ++s) h_step_log[(size_t)s * nrl + a] = log[(size_t)s * nrl + d];
    }
  }
  t.resolves = st[0].nres;
  if (totals) *totals = t;
  if (reset) {
    cudaMemset(pool->counters, 0, nrl * 4 * sizeof(unsigned long long));
    if (!log.empty()) cudaMemset(pool->step_log, 0, log.size() * sizeof(uint32_t));
    cudaMemset(pool->err_global, 0, sizeof(uint32_t));
    for (auto& s : st) s.err = 0;
    cudaMemcpy(pool->state, st.data(), st.size() * sizeof(hs_rl_state), cudaMemcpyHostToDevice);
    if (cudaDeviceSynchronize() != cudaSuccess) return HS_ERR_CUDA;
  }
  return t.error_bits ? HS_ERR_DEVICE_FLAG : HS_OK;
}

extern "C" int hs_read_state(hs_pool* pool, int layer, int32_t* h_tag, uint32_t* h_stamp, uint32_t* h_clock) {
  if (pool == nullptr || layer < 0 || layer >= pool->cfg.num_layers) return HS_ERR_ARG;
  DeviceGuard guard(pool->device);
  const size_t R = pool->cfg.num_requests, B = pool->cfg.buffer_slots;
  if (cudaDeviceSynchronize() != cudaSuccess) return HS_ERR_CUDA;
  const size_t off = (size_t)layer * R * B;
  if (h_tag && cudaMemcpy(h_tag, pool->tag + off, R * B * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return HS_ERR_CUDA;
  if (h_stamp && cudaMemcpy(h_stamp, pool->stamp + off, R * B * sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return HS_ERR_CUDA;
  if (h_clock) {
    std::vector<hs_rl_state> st(R);
    if (cudaMemcpy(st.data(), pool->state + (size_t)layer * R, R * sizeof(hs_rl_state), cudaMemcpyDeviceToHost) !=
        cudaSuccess)
      return HS_ERR_CUDA;
    for (size_t r = 0; r < R; ++r) h_clock[r] = st[r].clock;
  }
  return HS_OK;
}

extern "C" int hs_read_buffer(hs_pool* pool, int req, int layer, void* dst) {
  if (pool == nullptr || dst == nullptr) return HS_ERR_ARG;
  if (req < 0 || req >= pool->cfg.num_requests || layer < 0 || layer >= pool->cfg.num_layers) return HS_ERR_ARG;
  DeviceGuard guard(pool->device);
  const int64_t R = pool->cfg.num_requests, B = pool->cfg.buffer_slots, rec = pool->rec;
  if (cudaDeviceSynchronize() != cudaSuccess) return HS_ERR_CUDA;
  const hs_dev_pages& d = *pool->dev;
  const int64_t rl = (int64_t)layer * R + req;
  for (int i = 0; i < pool->slot_pages; ++i) {  // page by page; pages the buffer lacks read as zeros
    const int64_t j0 = i * d.page_slots, n = std::min<int64_t>(d.page_slots, B - j0);
    uint8_t* out = (uint8_t*)dst + j0 * rec;
    if (i < d.npages[rl]) {
      const void* src = (const void*)(uintptr_t)d.table[rl * pool->slot_pages + i];
      if (cudaMemcpy(out, src, (size_t)(n * rec), cudaMemcpyDeviceToHost) != cudaSuccess) return HS_ERR_CUDA;
    } else {
      memset(out, 0, (size_t)(n * rec));
    }
  }
  return HS_OK;
}

extern "C" int hs_read_history(hs_pool* pool, int req, int layer, int64_t pos0, int64_t n, void* dst) {
  if (pool == nullptr || dst == nullptr) return HS_ERR_ARG;
  const hs_config& c = pool->cfg;
  if (req < 0 || req >= c.num_requests || layer < 0 || layer >= c.num_layers) return HS_ERR_ARG;
  if (pos0 < 0 || n < 0 || pos0 + n > c.capacity) return HS_ERR_ARG;
  DeviceGuard guard(pool->device);
  if (cudaDeviceSynchronize() != cudaSuccess) return HS_ERR_CUDA;
  const hs_host_pages& h = *pool->host;
  const int64_t pt = h.page_tokens, rec = pool->rec;
  uint8_t* d = (uint8_t*)dst;
  for (int64_t p = pos0; p < pos0 + n;) {  // page by page; pages not reserved read as zeros
    const int64_t b = std::min(pos0 + n, (p / pt + 1) * pt);
    const uint8_t* page = h.host_pt[((int64_t)req * c.num_layers + layer) * pool->max_pages + p / pt];
    if (page != nullptr)
      memcpy(d, page + (p % pt) * rec, (size_t)((b - p) * rec));
    else
      memset(d, 0, (size_t)((b - p) * rec));
    d += (b - p) * rec;
    p = b;
  }
  return HS_OK;
}
