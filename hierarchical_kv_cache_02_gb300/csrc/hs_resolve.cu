// Fused RESOLVE and write-through APPEND kernels.
//
// RESOLVE follows the fused kernel of the HiSparse summary (§5), one CTA per (request, layer):
//   (1) build a shared-memory hash table of the k selected positions;
//   (2) probe every hot-buffer slot in parallel: hit, or a candidate for eviction;
//   (3) parallel scans: rank hits and misses in top-k order, select the m victims (radix select
//       on the eviction key, then an ordered compaction), update the recency stamps in place
//       (hits to MRU in top-k order, misses after the hits);
//   (4) fetch the missing records straight from the pinned host history with 16-byte
//       non-coherent vector loads into the claimed slots, a tuned number of bytes per thread;
//   (5) publish the page-table update and the dense vector of physical slots (locs).
// APPEND is step (5) of the decode flow in §3: the new token's record is written through to
// the host history and installed in the hot buffer.
#include <cuda_runtime.h>
#include <stdint.h>

#include "hs_internal.cuh"

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

struct ResolveArgs {
  const int32_t* topk;  // [R][k]
  int32_t* locs;        // [R][k]
  int32_t* tag;         // layer slice [R][B]
  uint32_t* stamp;      // layer slice [R][B]
  hs_rl_state* state;   // layer slice [R]
  unsigned long long* counters;  // layer slice [R][4]
  uint32_t* step_log;   // [log_steps][L][R] or null
  const uint8_t* hist_shared;
  const uint8_t* hist_priv;
  uint8_t* buf;         // layer slice [R][B][rec]
  int64_t C, P0, priv_tokens, rec;
  uint64_t seed;
  int R, L, layer, B, k, policy, log_steps, ht_bits;
};

__device__ __forceinline__ uint32_t ht_hash(int32_t p, int bits) { return ((uint32_t)p * 0x9E3779B1u) >> (32 - bits); }

// Exclusive scan of one uint32 per thread over the CTA; *total receives the sum.
__device__ __forceinline__ uint32_t cta_exclusive_scan(uint32_t v, uint32_t* wbuf, uint32_t* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wbuf[w] = x;
  __syncthreads();
  if (w == 0) {
    uint32_t s = wbuf[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    wbuf[lane] = s;  // inclusive prefix over warps
  }
  __syncthreads();
  const uint32_t base = w > 0 ? wbuf[w - 1] : 0u;
  *total = wbuf[kWarps - 1];
  __syncthreads();
  return base + x - v;
}

__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Move the m missing records host -> slots.  One work item = NV contiguous 16-byte vectors of one
// record; ITEMS work items per thread are loaded before any of their stores.
template <int NV>
__device__ void fetch_misses(const ResolveArgs& a, int r, int m, const int32_t* miss_pos, const int32_t* victims) {
  constexpr int ITEMS = NV >= 8 ? 1 : 2;
  const int64_t chunk = NV * 16;
  const int cpr = (int)(a.rec / chunk);
  const int total = m * cpr;
  for (int w0 = threadIdx.x; w0 < total; w0 += ITEMS * kThreads) {
    uint4 v[ITEMS][NV];
    uint4* dst[ITEMS];
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int w = w0 + it * kThreads;
      dst[it] = nullptr;
      if (w < total) {
        const int q = w / cpr, c = w - q * cpr;
        const uint4* src = (const uint4*)(hs_hist_addr(a.hist_shared, a.hist_priv, a.P0, a.priv_tokens, a.rec, a.L, r,
                                                       a.layer, miss_pos[q]) + c * chunk);
        dst[it] = (uint4*)(a.buf + ((int64_t)r * a.B + victims[q]) * a.rec + c * chunk);
#pragma unroll
        for (int u = 0; u < NV; ++u) v[it][u] = ld_nc_v4(src + u);
      }
    }
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      if (dst[it] != nullptr) {
#pragma unroll
        for (int u = 0; u < NV; ++u) dst[it][u] = v[it][u];
      }
    }
  }
}

template <int NV>
__global__ void __launch_bounds__(kThreads, 1) k_resolve(ResolveArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  const int k = a.k, B = a.B;
  const int ht_size = 1 << a.ht_bits;
  int32_t* ht_key = (int32_t*)smem;                 // [ht_size]
  int32_t* ht_val = ht_key + ht_size;               // [ht_size] smallest top-k index of the key
  int32_t* hit_slot = ht_val + ht_size;             // [k]: slot of a hit, -1 miss, -2 invalid
  int32_t* miss_idx = hit_slot + k;                 // [k]: top-k index of the q-th miss
  int32_t* miss_pos = miss_idx + k;                 // [k]: position of the q-th miss
  int32_t* victims = miss_pos + k;                  // [k]: q-th victim slot (ascending)
  uint8_t* slot_hit = (uint8_t*)(victims + k);      // [B]
  __shared__ uint32_t wbuf[kWarps];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t sel_digit, sel_need, err_bits;

  const int32_t* topk = a.topk + (int64_t)r * k;
  int32_t* locs = a.locs + (int64_t)r * k;
  int32_t* tag = a.tag + (int64_t)r * B;
  uint32_t* stamp = a.stamp + (int64_t)r * B;
  const hs_rl_state st = a.state[r];
  const uint32_t clock = st.clock;

  if (tid == 0) err_bits = ((uint64_t)clock + (uint64_t)k >= 0xFFFFFFFFull) ? (uint32_t)HS_DEVERR_CLOCK : 0u;
  for (int x = tid; x < ht_size; x += kThreads) {
    ht_key[x] = -1;
    ht_val[x] = 0x7fffffff;
  }
  for (int j = tid; j < B; j += kThreads) slot_hit[j] = 0;
  __syncthreads();

  // (1) hash the selected positions; a key keeps the smallest top-k index that carries it
  for (int i = tid; i < k; i += kThreads) {
    const int32_t s = topk[i];
    if (s == -1) continue;
    if (s < 0 || (int64_t)s >= a.C) {
      atomicOr(&err_bits, (uint32_t)HS_DEVERR_RANGE);
      continue;
    }
    uint32_t h = ht_hash(s, a.ht_bits);
    while (true) {
      const int32_t prev = atomicCAS(&ht_key[h], -1, s);
      if (prev == -1 || prev == s) {
        atomicMin(&ht_val[h], i);
        break;
      }
      h = (h + 1) & (uint32_t)(ht_size - 1);
    }
  }
  __syncthreads();
  for (int i = tid; i < k; i += kThreads) {
    const int32_t s = topk[i];
    int32_t state = -2;
    if (s >= 0 && (int64_t)s < a.C) {
      uint32_t h = ht_hash(s, a.ht_bits);
      while (ht_key[h] != s) h = (h + 1) & (uint32_t)(ht_size - 1);
      if (ht_val[h] == i) {
        state = -1;
      } else {
        atomicOr(&err_bits, (uint32_t)HS_DEVERR_DUP);
      }
    }
    hit_slot[i] = state;
  }
  __syncthreads();

  // (2) probe every slot
  for (int j = tid; j < B; j += kThreads) {
    const int32_t t = tag[j];
    if (t < 0) continue;
    uint32_t h = ht_hash(t, a.ht_bits);
    while (true) {
      const int32_t key = ht_key[h];
      if (key == t) {
        hit_slot[ht_val[h]] = j;
        slot_hit[j] = 1;
        break;
      }
      if (key == -1) break;
      h = (h + 1) & (uint32_t)(ht_size - 1);
    }
  }
  __syncthreads();

  // (3a) rank hits and misses in top-k order; stamp hits; list misses
  const int kpt = (k + kThreads - 1) / kThreads;
  const int i0 = min(k, tid * kpt), i1 = min(k, i0 + kpt);
  uint32_t local = 0;
  for (int i = i0; i < i1; ++i) {
    const int32_t hs = hit_slot[i];
    local += hs >= 0 ? 1u : (hs == -1 ? 0x10000u : 0u);
  }
  uint32_t tot;
  uint32_t pre = cta_exclusive_scan(local, wbuf, &tot);
  const int h = (int)(tot & 0xffffu), m = (int)(tot >> 16);
  {
    uint32_t a_rank = pre & 0xffffu, q_rank = pre >> 16;
    for (int i = i0; i < i1; ++i) {
      const int32_t hs = hit_slot[i];
      if (hs >= 0) {
        if (a.policy != HS_POLICY_FIFO) stamp[hs] = clock + a_rank;
        locs[i] = hs;
        ++a_rank;
      } else if (hs == -1) {
        miss_idx[q_rank] = i;
        miss_pos[q_rank] = topk[i];
        ++q_rank;
      } else {
        locs[i] = -1;
      }
    }
  }

  // (3b) victims: the m candidates with the smallest (key, slot)
  const int ncand = B - h;
  const bool take_all = (m == ncand);
  uint32_t T = 0u, need_eq = 0u;
  if (m > 0 && !take_all) {
    uint32_t prefix = 0u, mask = 0u, need = (uint32_t)m;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      if (tid < 256) hist[tid] = 0u;
      __syncthreads();
      for (int j = tid; j < B; j += kThreads) {
        if (slot_hit[j]) continue;
        const uint32_t key = hs_evict_key(a.policy, tag[j], stamp[j], a.seed, st.nres, a.R, r, a.L, a.layer, B, j);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        uint32_t s = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) s += hist[tid * 8 + b];
        uint32_t c = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          uint32_t y = __shfl_up_sync(0xffffffffu, c, o);
          if (tid >= o) c += y;
        }
        const uint32_t excl = c - s;
        if (excl < need && need <= c) {
          uint32_t run = excl;
          for (int b = 0; b < 8; ++b) {
            const uint32_t hb = hist[tid * 8 + b];
            if (run + hb >= need) {
              sel_digit = (uint32_t)(tid * 8 + b);
              sel_need = need - run;
              break;
            }
            run += hb;
          }
        }
      }
      __syncthreads();
      prefix |= sel_digit << shift;
      mask |= 255u << shift;
      need = sel_need;
      __syncthreads();
    }
    T = prefix;
    need_eq = need;
  }

  // (3c) ordered compaction of the victims (ascending slot) and install the misses
  if (m > 0) {
    const int bpt = (B + kThreads - 1) / kThreads;
    const int j0 = min(B, tid * bpt), j1 = min(B, j0 + bpt);
    uint32_t cnt = 0;
    for (int j = j0; j < j1; ++j) {
      if (slot_hit[j]) continue;
      if (take_all) {
        cnt += 1u;
      } else {
        const uint32_t key = hs_evict_key(a.policy, tag[j], stamp[j], a.seed, st.nres, a.R, r, a.L, a.layer, B, j);
        cnt += key < T ? 1u : (key == T ? 0x10000u : 0u);
      }
    }
    uint32_t tot2;
    const uint32_t pre2 = cta_exclusive_scan(cnt, wbuf, &tot2);
    uint32_t less_b = pre2 & 0xffffu, eq_b = pre2 >> 16;
    // keys are read before any write of this phase: every slot is owned by one thread
    for (int j = j0; j < j1; ++j) {
      if (slot_hit[j]) continue;
      bool victim;
      uint32_t q;
      if (take_all) {
        victim = true;
        q = less_b++;
      } else {
        const uint32_t key = hs_evict_key(a.policy, tag[j], stamp[j], a.seed, st.nres, a.R, r, a.L, a.layer, B, j);
        if (key < T) {
          victim = true;
          q = less_b + min(eq_b, need_eq);
          ++less_b;
        } else if (key == T) {
          victim = eq_b < need_eq;
          q = less_b + eq_b;
          ++eq_b;
        } else {
          victim = false;
          q = 0;
        }
      }
      if (victim) {
        const int i = miss_idx[q];
        tag[j] = miss_pos[q];
        stamp[j] = a.policy == HS_POLICY_FIFO ? clock + q : clock + (uint32_t)h + q;
        locs[i] = j;
        victims[q] = j;
      } else if (a.policy == HS_POLICY_SWAP_VANILLA) {
        tag[j] = -1;
        stamp[j] = 0u;
      }
    }
  } else if (a.policy == HS_POLICY_SWAP_VANILLA) {
    for (int j = tid; j < B; j += kThreads) {
      if (!slot_hit[j]) {
        tag[j] = -1;
        stamp[j] = 0u;
      }
    }
  }
  __syncthreads();

  // (4) fetch the misses from the host history
  if (m > 0) fetch_misses<NV>(a, r, m, miss_pos, victims);

  // (5) clock and counters
  if (tid == 0) {
    hs_rl_state ns = st;
    ns.clock = clock + (uint32_t)k;
    ns.nres = st.nres + 1u;
    ns.err = st.err | err_bits;
    a.state[r] = ns;
    unsigned long long* c = a.counters + (int64_t)r * 4;
    c[0] += (unsigned long long)h;
    c[1] += (unsigned long long)m;
    c[3] += (unsigned long long)m * (unsigned long long)a.rec;
    if (a.step_log != nullptr && st.nres < (uint32_t)a.log_steps)
      a.step_log[((int64_t)st.nres * a.L + a.layer) * a.R + r] = (uint32_t)m;
  }
}

struct AppendArgs {
  const int64_t* pos;    // [R]
  const uint8_t* rec_in; // [R][rec]
  int32_t* tag;
  uint32_t* stamp;
  hs_rl_state* state;
  unsigned long long* counters;
  uint8_t* hist_shared;
  uint8_t* hist_priv;
  uint8_t* buf;
  int64_t C, P0, priv_tokens, rec;
  uint64_t seed;
  int R, L, layer, B, policy;
};

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads) k_append(AppendArgs a) {
  const int r = blockIdx.x, tid = threadIdx.x;
  const int64_t p = a.pos[r];
  const hs_rl_state st = a.state[r];
  if (p < a.P0 || p < 0 || p >= a.C) {
    if (tid == 0) a.state[r].err = st.err | (uint32_t)HS_DEVERR_APPEND;
    return;
  }
  int32_t* tag = a.tag + (int64_t)r * a.B;
  uint32_t* stamp = a.stamp + (int64_t)r * a.B;
  int found = 0x7fffffff;
  unsigned long long best = ~0ull;
  for (int j = tid; j < a.B; j += kAppendThreads) {
    const int32_t t = tag[j];
    if (t == (int32_t)p) found = min(found, j);
    const uint32_t key = hs_evict_key(a.policy, t, stamp[j], a.seed, st.nres, a.R, r, a.L, a.layer, a.B, j);
    const unsigned long long kj = ((unsigned long long)key << 32) | (unsigned)j;
    best = kj < best ? kj : best;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    found = min(found, __shfl_xor_sync(0xffffffffu, found, o));
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
    best = y < best ? y : best;
  }
  __shared__ int s_found[kAppendThreads / 32];
  __shared__ unsigned long long s_best[kAppendThreads / 32];
  __shared__ int s_slot;
  if ((tid & 31) == 0) {
    s_found[tid >> 5] = found;
    s_best[tid >> 5] = best;
  }
  __syncthreads();
  if (tid == 0) {
    int f = s_found[0];
    unsigned long long b = s_best[0];
    for (int w = 1; w < kAppendThreads / 32; ++w) {
      f = min(f, s_found[w]);
      b = s_best[w] < b ? s_best[w] : b;
    }
    s_slot = f != 0x7fffffff ? f : (int)(b & 0xffffffffull);
  }
  __syncthreads();
  const int slot = s_slot;
  const uint4* src = (const uint4*)(a.rec_in + (int64_t)r * a.rec);
  uint4* dh = (uint4*)(a.hist_priv + (((int64_t)r * a.L + a.layer) * a.priv_tokens + (p - a.P0)) * a.rec);
  uint4* db = (uint4*)(a.buf + ((int64_t)r * a.B + slot) * a.rec);
  const int nv = (int)(a.rec / 16);
  for (int x = tid; x < nv; x += kAppendThreads) {
    const uint4 v = src[x];
    dh[x] = v;
    db[x] = v;
  }
  if (tid == 0) {
    tag[slot] = (int32_t)p;
    stamp[slot] = st.clock;
    hs_rl_state ns = st;
    ns.clock = st.clock + 1u;
    if ((uint64_t)st.clock + 1u >= 0xFFFFFFFFull) ns.err |= (uint32_t)HS_DEVERR_CLOCK;
    a.state[r] = ns;
    a.counters[(int64_t)r * 4 + 2] += 1ull;
  }
}

int ht_bits_for(int k) {
  int bits = 1;
  while ((1 << bits) < 2 * k) ++bits;
  return bits;
}

}  // namespace

size_t hs_resolve_smem_bytes(const hs_config* c) {
  const size_t ht = (size_t)1 << ht_bits_for(c->top_k);
  return ht * 8 + (size_t)c->top_k * 16 + (size_t)c->buffer_slots;
}

int hs_launch_resolve(hs_pool* p, int layer, const int32_t* d_topk, int32_t* d_locs, cudaStream_t st) {
  const hs_config& c = p->cfg;
  const int64_t R = c.num_requests, B = c.buffer_slots;
  ResolveArgs a;
  a.topk = d_topk;
  a.locs = d_locs;
  a.tag = p->tag + (int64_t)layer * R * B;
  a.stamp = p->stamp + (int64_t)layer * R * B;
  a.state = p->state + (int64_t)layer * R;
  a.counters = p->counters + (int64_t)layer * R * 4;
  a.step_log = c.log_steps > 0 ? p->step_log : nullptr;
  a.hist_shared = p->dmap_shared;
  a.hist_priv = p->dmap_priv;
  a.buf = p->buf + (int64_t)layer * R * B * p->rec;
  a.C = c.capacity;
  a.P0 = c.shared_prefix;
  a.priv_tokens = p->priv_tokens;
  a.rec = p->rec;
  a.seed = c.seed;
  a.R = c.num_requests;
  a.L = c.num_layers;
  a.layer = layer;
  a.B = c.buffer_slots;
  a.k = c.top_k;
  a.policy = c.policy;
  a.log_steps = c.log_steps;
  a.ht_bits = ht_bits_for(c.top_k);
  const size_t smem = hs_resolve_smem_bytes(&c);
  switch (c.io_chunk_bytes) {
    case 16: k_resolve<1><<<c.num_requests, kThreads, smem, st>>>(a); break;
    case 32: k_resolve<2><<<c.num_requests, kThreads, smem, st>>>(a); break;
    case 64: k_resolve<4><<<c.num_requests, kThreads, smem, st>>>(a); break;
    default: k_resolve<8><<<c.num_requests, kThreads, smem, st>>>(a); break;
  }
  return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

// Kernel attributes are set once at pool creation so that the launches stay capturable.
int hs_resolve_prepare(const hs_config* c) {
  const int smem = (int)hs_resolve_smem_bytes(c);
  cudaError_t e;
  switch (c->io_chunk_bytes) {
    case 16: e = cudaFuncSetAttribute(k_resolve<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); break;
    case 32: e = cudaFuncSetAttribute(k_resolve<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); break;
    case 64: e = cudaFuncSetAttribute(k_resolve<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); break;
    default: e = cudaFuncSetAttribute(k_resolve<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); break;
  }
  return e == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

int hs_launch_append(hs_pool* p, int layer, const int64_t* d_pos, const void* d_rec, cudaStream_t st) {
  const hs_config& c = p->cfg;
  const int64_t R = c.num_requests, B = c.buffer_slots;
  AppendArgs a;
  a.pos = d_pos;
  a.rec_in = (const uint8_t*)d_rec;
  a.tag = p->tag + (int64_t)layer * R * B;
  a.stamp = p->stamp + (int64_t)layer * R * B;
  a.state = p->state + (int64_t)layer * R;
  a.counters = p->counters + (int64_t)layer * R * 4;
  a.hist_shared = p->dmap_shared;
  a.hist_priv = p->dmap_priv;
  a.buf = p->buf + (int64_t)layer * R * B * p->rec;
  a.C = c.capacity;
  a.P0 = c.shared_prefix;
  a.priv_tokens = p->priv_tokens;
  a.rec = p->rec;
  a.seed = c.seed;
  a.R = c.num_requests;
  a.L = c.num_layers;
  a.layer = layer;
  a.B = c.buffer_slots;
  a.policy = c.policy;
  k_append<<<c.num_requests, kAppendThreads, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}
