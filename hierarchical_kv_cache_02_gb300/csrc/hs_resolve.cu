// Fused RESOLVE and write-through APPEND kernels.
//
// RESOLVE follows the fused kernel of the HiSparse summary (§5), which runs one CTA per (request,
// layer).  Here a thread-block cluster serves each request of a launch: every CTA of the cluster
// computes the whole decision from the same inputs, then takes its share of the writes and of the
// host copies, so the copies of one request are spread over several SMs.  The steps:
//   (1) build a shared-memory hash table of the k selected positions;
//   (2) probe every hot-buffer slot in parallel: hit, or a candidate for eviction;
//   (3) parallel scans: rank hits and misses in top-k order, select the m victims (a bitmap over
//       the eviction keys when they are distinct, else a radix select on them; then an ordered
//       compaction), update the recency stamps in place
//       (hits to MRU in top-k order, misses after the hits);
//   (4) fetch the missing records straight from the pinned host history with 16-byte
//       non-coherent vector loads into the claimed slots, a tuned number of bytes per thread.
//       The first misses of each CTA are requested as soon as the miss list is known, with
//       asynchronous 16-byte copies into a shared-memory staging area, so the host link is busy
//       while the victims are still being chosen; they reach their slots once the victims are known;
//   (5) publish the page-table update and the dense vector of physical slots (locs).
// APPEND is step (5) of the decode flow in §3: the new token's record is written through to
// the host history and installed in the hot buffer.
// A buffer grown on demand (§8) holds slots [0, cap) only: both kernels probe, evict and install
// there alone, and refuse a (request, layer) with fewer than k slots (HS_DEVERR_SLOTS).
#include <cuda_runtime.h>
#include <stdint.h>

#include "hs_internal.cuh"

#ifdef HS_PHASE_TRACE
// phase stamps of k_resolve (see HS_PHASE); read and cleared by the two calls below
__device__ unsigned long long hs_phase_res[256][64];
extern "C" int hs_phase_resolve_read(void* host) {
  return (int)cudaMemcpyFromSymbol(host, hs_phase_res, sizeof(hs_phase_res));
}
extern "C" int hs_phase_resolve_clear() {
  static unsigned long long zero[256][64];
  return (int)cudaMemcpyToSymbol(hs_phase_res, zero, sizeof(zero));
}
#endif

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
  const uint64_t* pt;   // host page table [R][L][max_pages]
  uint32_t* err_global; // pool-wide error word (errors found outside the deciding CTA)
  const uint64_t* spt;  // layer slice [R][spp] of the slot table: device address of each buffer page
  const int32_t* scap;  // layer slice [R]: slots each buffer holds
  int64_t C, P0, max_pages, rec;
  int page_shift, sshift, spp;
  uint64_t seed;
  hs_pending* pend;      // fetch-in-attention mode: layer slice [R][k], else null
  uint32_t* pend_live;   // layer slice [R]
  const int64_t* app_pos;  // fused write-through append before the resolve: [R] positions, or null
  const uint8_t* app_rec;  // [R][rec] new records
  int R, L, layer, B, k, policy, log_steps, ht_bits, cs;  // R: all requests of the pool
  int r0;  // first request of this launch: topk, locs and the append inputs are indexed from it
  int stage_off, stage_recs;  // staging area for early miss copies: byte offset in shared memory, records
  int stall;                  // test hook (hs_debug_stall_next): leave the early copies' arrival out
  uint32_t* res_count;        // layer slice [R][2]: launches, CTAs finished (per request)
  int nreq;                   // requests of this launch: CTAs [0, nreq cs) decide, the rest fetch
  // early fetch (null when off): layer slices of the position -> slot map [R][C], the slot of each
  // missing top-k entry (+1; 0 none) [R][k], the deciding CTAs done [R], all CTAs finished [R] and
  // the scratch [R][cs x fetch_rows][rec]
  int32_t* pos_slot;
  int32_t* fslot;
  uint32_t* fdec;
  uint32_t* ffin;
  uint8_t* fscratch;
  int fetch_rows;             // scratch rows of one fetch CTA
  int fpr;                    // fetch CTAs per request
  int fstall;                 // test hook: the fetch CTAs of the launch's first request do not wait
};

__device__ __forceinline__ uint32_t ht_hash(int32_t p, int bits) { return ((uint32_t)p * 0x9E3779B1u) >> (32 - bits); }

// Exclusive scan of one uint32 per thread over the CTA; *total receives the sum.
// kTrailing = false leaves out the last barrier, which only keeps wbuf from being rewritten while
// it is read: for a caller that passes another barrier before its next scan.
template <bool kTrailing = true>
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
    uint32_t s = lane < kWarps ? wbuf[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kWarps) wbuf[lane] = s;  // inclusive prefix over warps
  }
  __syncthreads();
  const uint32_t base = w > 0 ? wbuf[w - 1] : 0u;
  *total = wbuf[kWarps - 1];
  if (kTrailing) __syncthreads();
  return base + x - v;
}

__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// mbarrier and bulk-copy helpers for the early miss copies
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init1(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar)) : "memory");
}
// wait for phase `parity` of `bar`, at most about one second (%globaltimer); false when it gave up
__device__ __forceinline__ bool mbar_wait_1s(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((it & 63u) == 0u) {
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (it == 0u) t0 = t;
      else if (t - t0 > 1000000000ull) return false;
    }
  }
}
// one bulk copy global -> this CTA's shared memory, completing on `bar` (16-byte aligned, size a
// multiple of 16)
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Copy misses [q0, q1) host -> slots.  A warp moves one chunk of 32 x NV lane-contiguous 16-byte
// vectors of one record per item (coalesced 512-byte rows); ITEMS items are loaded before any store.
template <int NV>
__device__ void fetch_misses(const ResolveArgs& a, int q0, int q1, const uint64_t* s_src, const int32_t* victims,
                             const uint64_t* slots) {
  constexpr int ITEMS = NV >= 8 ? 1 : 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int vpr = (int)(a.rec / 16);            // vectors per record
  const int cpr = (vpr + 32 * NV - 1) / (32 * NV);
  const int total = (q1 - q0) * cpr;
  for (int w0 = warp; w0 < total; w0 += ITEMS * kWarps) {
    uint4 v[ITEMS][NV];
    const uint4* src[ITEMS];
    uint4* dst[ITEMS];
    int vbase[ITEMS];
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int w = w0 + it * kWarps;
      dst[it] = nullptr;
      if (w < total) {
        const int q = q0 + w / cpr, c = w % cpr;
        src[it] = (const uint4*)s_src[q - q0];
        if (src[it] == nullptr) continue;  // page not reserved (flagged): the slot keeps its contents
        dst[it] = (uint4*)hs_slot_addr(slots, a.sshift, a.rec, victims[q]);
        vbase[it] = c * 32 * NV + lane;
#pragma unroll
        for (int u = 0; u < NV; ++u) {
          const int vi = vbase[it] + 32 * u;
          if (vi < vpr) v[it][u] = ld_nc_v4(src[it] + vi);
        }
      }
    }
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      if (dst[it] != nullptr) {
#pragma unroll
        for (int u = 0; u < NV; ++u) {
          const int vi = vbase[it] + 32 * u;
          if (vi < vpr) dst[it][vi] = v[it][u];
        }
      }
    }
  }
}

// The m victims are the candidates with the smallest (key, slot).  Radix select over the key range
// of the candidates (key - min, 11-bit digits from the top) finds the threshold T and how many
// candidates with key == T (lowest slots first) complete the set.  Passes alternate between two
// histograms and two selection words, both zero on entry: each thread clears the bins it has read,
// so a histogram is zero again two passes later and a pass needs no barrier to clear one.
__device__ __noinline__ void select_threshold(const uint32_t* key32, const uint8_t* flag, int B, uint32_t m, uint32_t lo,
                                             uint32_t hi, uint32_t* wbuf, uint32_t (*hist)[2048], uint32_t (*sel)[2],
                                             uint32_t* T_out, uint32_t* need_out) {
  // lo, hi: the smallest and largest candidate key (found by the probe)
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t range = hi - lo;
  int shift = range == 0u ? 0 : 32 - __clz(range);
  uint64_t prefix = 0;
  uint32_t need = m;
  for (int pass = 0; shift > 0; ++pass) {
    const int width = shift < 11 ? shift : 11;
    shift -= width;
    const int nb = 1 << width;
    uint32_t* h = hist[pass & 1];
    uint32_t* sl = sel[pass & 1];
    for (int base = tid & ~31; base < B; base += kThreads) {
      const int j = base + lane;
      uint32_t digit = 0xffffffffu;
      if (j < B && !(flag[j] & 1u)) {
        const uint64_t v = (uint64_t)(key32[j] - lo);
        if ((v >> (shift + width)) == prefix) digit = (uint32_t)(v >> shift) & (uint32_t)(nb - 1);
      }
      // the lanes sharing the first counted lane's digit add once (empty slots and old stamps crowd
      // into a few bins); the others add one each
      const uint32_t part = __ballot_sync(0xffffffffu, digit != 0xffffffffu);
      if (part != 0u) {
        const uint32_t d0 = __shfl_sync(0xffffffffu, digit, __ffs(part) - 1);
        const uint32_t same = __ballot_sync(0xffffffffu, digit == d0);
        if (digit == d0) {
          if (lane == __ffs(same) - 1) atomicAdd(&h[digit], (uint32_t)__popc(same));
        } else if (digit != 0xffffffffu) {
          atomicAdd(&h[digit], 1u);
        }
      }
    }
    __syncthreads();
    HS_PHASE(hs_phase_res, 14 + 2 * (pass & 1), threadIdx.x == 0 && pass < 2);  // pass's histogram complete
    // bins [BPT tid, BPT tid + BPT): find the bin where the running count reaches `need`
    constexpr int BPT = 2048 / kThreads;
    const int b0 = BPT * tid;
    uint32_t c[BPT], csum = 0u;
#pragma unroll
    for (int u = 0; u < BPT; ++u) {
      c[u] = 0u;
      if (b0 + u < nb) {
        c[u] = h[b0 + u];
        h[b0 + u] = 0u;  // only this thread reads this bin
      }
      csum += c[u];
    }
    uint32_t tot;
    // no trailing barrier: the one below comes before the next pass's scan rewrites wbuf
    const uint32_t excl = cta_exclusive_scan<false>(csum, wbuf, &tot);
    if (excl < need && need <= excl + csum) {
      uint32_t run = excl;
#pragma unroll
      for (int u = 0; u < BPT; ++u) {
        if (run < need && need <= run + c[u]) {
          sl[0] = (uint32_t)(b0 + u);
          sl[1] = need - run;
        }
        run += c[u];
      }
    }
    __syncthreads();
    HS_PHASE(hs_phase_res, 15 + 2 * (pass & 1), threadIdx.x == 0 && pass < 2);  // pass's bin found
    prefix = (prefix << width) | sl[0];
    need = sl[1];
  }
  *T_out = lo + (uint32_t)prefix;
  *need_out = need;
}

// The same threshold in one pass when the candidates' nonzero keys are all distinct: the recency
// stamps of LRU, FIFO and swap-vanilla (every stamp a resolve or append hands out is new; 0 marks an
// empty slot).  Each nonzero key sets bit (key - lo) of a bitmap over [lo, lo + kDenseSpan) (the
// radix select's histograms, zero on entry); the zero keys are counted.  Then T is the
// (m - zeros)-th set bit (need_eq = 1), found by a block scan of the words' bit counts, or T = 0 with
// need_eq = m when the empty slots alone suffice.  Returns false, with the bitmap cleared again, when
// a nonzero key lies outside the window: the radix select then runs.
constexpr uint32_t kDenseSpan = 2u * 2048u * 32u;  // bits in the two histograms
__device__ __noinline__ bool select_dense(const uint32_t* key32, const uint8_t* flag, int B, uint32_t m, uint32_t lo,
                                          uint32_t* wbuf, uint32_t (*hist)[2048], uint32_t (*sel)[2], uint32_t* s_cnt,
                                          uint32_t* T_out, uint32_t* need_out) {
  // s_cnt[0]: zero keys, s_cnt[1]: keys outside the window (both 0 on entry)
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t* bmw = &hist[0][0];
  constexpr int U = 4;  // slots a thread loads before it sets any bit
  for (int base = tid & ~31; base < B; base += U * kThreads) {
    uint32_t key[U];
    bool cand[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = base + u * kThreads + lane;
      cand[u] = j < B && !(flag[j] & 1u);
      key[u] = cand[u] ? key32[j] : 0u;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t d = key[u] - lo;
      const bool zero = cand[u] && key[u] == 0u, out = cand[u] && key[u] != 0u && (key[u] < lo || d >= kDenseSpan);
      if (cand[u] && key[u] != 0u && !out) atomicOr(&bmw[d >> 5], 1u << (d & 31u));
      const uint32_t zb = __ballot_sync(0xffffffffu, zero), ob = __ballot_sync(0xffffffffu, out);
      if (lane == 0 && (zb | ob) != 0u) {
        if (zb) atomicAdd(&s_cnt[0], (uint32_t)__popc(zb));
        if (ob) atomicAdd(&s_cnt[1], (uint32_t)__popc(ob));
      }
    }
  }
  __syncthreads();
  HS_PHASE(hs_phase_res, 14, threadIdx.x == 0);
  if (s_cnt[1] != 0u) {
    for (int x = tid; x < 2 * 2048; x += kThreads) bmw[x] = 0u;
    __syncthreads();
    return false;
  }
  const uint32_t z = s_cnt[0];
  if (m <= z) {
    *T_out = 0u;
    *need_out = m;
    return true;
  }
  const uint32_t m2 = m - z;  // the m2-th smallest nonzero key
  constexpr int WPT = 2 * 2048 / kThreads;  // bitmap words per thread
  uint32_t w[WPT], c = 0u;
#pragma unroll
  for (int u = 0; u < WPT; ++u) {
    w[u] = bmw[WPT * tid + u];
    c += (uint32_t)__popc(w[u]);
  }
  // the thread's exclusive prefix of set bits: a warp scan, the warps' totals through wbuf, and a scan
  // of those in every warp
  uint32_t incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wbuf[tid >> 5] = incl;
  __syncthreads();
  uint32_t wincl = lane < kWarps ? wbuf[lane] : 0u;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, wincl, o);
    if (lane >= o) wincl += y;
  }
  const uint32_t wpre = __shfl_sync(0xffffffffu, wincl, tid >> 5) - wbuf[tid >> 5];  // the warps before
  const uint32_t excl = wpre + incl - c;
  if (excl < m2 && m2 <= excl + c) {
    uint32_t run = excl;
#pragma unroll
    for (int u = 0; u < WPT; ++u) {
      const uint32_t pc = (uint32_t)__popc(w[u]);
      if (run < m2 && m2 <= run + pc) {
        uint32_t x = w[u];
        for (uint32_t t = m2 - run - 1u; t > 0u; --t) x &= x - 1u;
        sel[0][0] = (uint32_t)(32 * (WPT * tid + u)) + (uint32_t)(__ffs(x) - 1);
      }
      run += pc;
    }
  }
  __syncthreads();
  HS_PHASE(hs_phase_res, 15, threadIdx.x == 0);
  *T_out = lo + sel[0][0];
  *need_out = 1u;
  return true;
}

// A resolve CTA's last act: once every thread's writes (locs, metadata, fetched rows) are done, count
// the CTA as finished for its request, with release ordering (an attention that waits for the count
// then reads those writes).  With fetch CTAs, the last CTA of the request's launch to get here first
// clears the request's miss slots and counters for the next launch: every other CTA counted itself
// after its last use of them.
__device__ __forceinline__ void count_finished(const ResolveArgs& a, int r) {
  __syncthreads();
  if (a.fslot != nullptr) {
    __shared__ int s_last;
    if (threadIdx.x == 0) {
      __threadfence();
      s_last = atomicAdd(&a.ffin[r], 1u) == (uint32_t)(a.cs + a.fpr - 1);
      __threadfence();
    }
    __syncthreads();
    if (s_last) {
      for (int i = threadIdx.x; i < a.k; i += kThreads) a.fslot[(int64_t)r * a.k + i] = 0;
      if (threadIdx.x == 0) {
        a.fdec[r] = 0u;
        a.ffin[r] = 0u;
      }
      __syncthreads();
    }
  }
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&a.res_count[2 * r + 1], 1u);
  }
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr int kFetchUnroll = 8;  // 16-byte loads a lane of a fetch CTA has in flight per record

// A fetch CTA (early fetch) does all of the miss fetch for its share [e0, e1) of the request's top-k
// list, starting at the launch's start:
//   (1) it lists the entries that look missing: those whose position's last slot (the position ->
//       slot map) is not below the buffer's slot count or no longer carries the position's tag (a
//       hint only: the decision is what counts);
//   (2) until every deciding CTA has written its share, it copies those records from the host
//       history into its scratch rows, at most fetch_rows of them;
//   (3) it waits (bounded) for the deciding CTAs, reads the slot each actual miss of its share was
//       given, and copies the record there: from its scratch row when it has it (HBM to HBM), else
//       from the host.
// A record it fetched that the decision did not count as a miss (a repeat, the position the fused
// append has just installed) only costs the link transfer.  A wait that gives up flags the resolve
// and installs nothing (the cache state then no longer matches the history).
__device__ void early_fetch_cta(const ResolveArgs& a, int r, int crank) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = a.k;
  const int cap = a.scap[r];
  if (min(a.B, cap) < k) return;  // too few slots: the deciding CTAs change nothing
  const int e0 = (int)((int64_t)k * crank / a.fpr), e1 = (int)((int64_t)k * (crank + 1) / a.fpr), ne = e1 - e0;
  int32_t* lst = (int32_t*)smem;  // [ne]: the share's apparent misses (top-k indices)
  int32_t* srow = lst + ne;       // [ne]: scratch row holding entry e0 + x, or -1
  int32_t* inst = srow + ne;      // [ne]: the share's actual misses (top-k indices)
  int32_t* islot = inst + ne;     // [ne]: and their slots
  __shared__ int s_n, s_m, s_go;
  const int32_t* topk = a.topk + (int64_t)(r - a.r0) * k;
  const int32_t* tag = a.tag + (int64_t)r * a.B;
  const int32_t* ps = a.pos_slot + (int64_t)r * a.C;
  const uint32_t* dec = a.fdec + r;
  if (tid == 0) {
    s_n = 0;
    s_m = 0;
  }
  for (int x = tid; x < ne; x += kThreads) srow[x] = -1;
  __syncthreads();
  // (1)
  for (int ib = e0 + 32 * warp; ib < e1; ib += kThreads) {
    const int i = ib + lane;
    bool miss = false;
    if (i < e1) {
      const int32_t p = topk[i];
      if (p >= 0 && (int64_t)p < a.C) {
        const int32_t s = __ldcg(ps + p);
        miss = !(s >= 0 && s < cap && __ldcg(tag + s) == p);
      }
    }
    const uint32_t bm = __ballot_sync(0xffffffffu, miss);
    int base = 0;
    if (lane == 0 && bm != 0u) base = atomicAdd(&s_n, __popc(bm));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (miss) lst[base + __popc(bm & ((1u << lane) - 1u))] = i;
  }
  __syncthreads();
  HS_PHASE(hs_phase_res, 21, tid == 0);
  const int n = min(s_n, a.fetch_rows);
  const uint64_t* row = a.pt + ((int64_t)r * a.L + a.layer) * a.max_pages;
  const int row0 = crank * a.fetch_rows;  // this CTA's first row in the request's scratch
  uint8_t* scratch = a.fscratch + (int64_t)r * a.fpr * a.fetch_rows * a.rec;
  const int vpr = (int)(a.rec / 16);
  // one record -> dst by the calling warp, kFetchUnroll 16-byte loads per lane in flight
  auto copy_rec = [&](uint4* dst, const uint4* src, bool from_host) {
    for (int v0 = 0; v0 < vpr; v0 += 32 * kFetchUnroll) {
      uint4 t[kFetchUnroll];
#pragma unroll
      for (int u = 0; u < kFetchUnroll; ++u) {
        const int v = v0 + 32 * u + lane;
        if (v < vpr) t[u] = from_host ? ld_nc_v4(src + v) : __ldcg(src + v);
      }
#pragma unroll
      for (int u = 0; u < kFetchUnroll; ++u) {
        const int v = v0 + 32 * u + lane;
        if (v < vpr) dst[v] = t[u];
      }
    }
  };
  // (2)
  for (int x = warp; x < n; x += kWarps) {
    uint32_t decided = 0u;
    if (lane == 0) decided = ld_acquire_gpu(dec) >= (uint32_t)a.cs ? 1u : 0u;
    if (__shfl_sync(0xffffffffu, decided, 0) != 0u) break;
    const int i = lst[x];
    const uint4* src = (const uint4*)hs_page_row_addr(row, a.page_shift, a.rec, topk[i]);
    if (src == nullptr) continue;  // not reserved: the deciding CTA flags it
    copy_rec((uint4*)(scratch + (int64_t)(row0 + x) * a.rec), src, true);
    __syncwarp();
    if (lane == 0) srow[i - e0] = row0 + x;
  }
  // (3)
  if (tid == 0) {
    bool ok = ld_acquire_gpu(dec) >= (uint32_t)a.cs;
    if (!ok) {
      const uint64_t t0 = global_ns();
      do {
        __nanosleep(256);
        ok = ld_acquire_gpu(dec) >= (uint32_t)a.cs;
      } while (!ok && global_ns() - t0 < 1000000000ull);
    }
    if (!ok) atomicOr(a.err_global, (uint32_t)HS_DEVERR_TIMEOUT);
    s_go = ok ? 1 : 0;
  }
  __syncthreads();
  HS_PHASE(hs_phase_res, 23, tid == 0);
  if (s_go == 0) return;
  const int32_t* fs = a.fslot + (int64_t)r * k;
  for (int ib = e0 + 32 * warp; ib < e1; ib += kThreads) {
    const int i = ib + lane;
    const int32_t v = i < e1 ? __ldcg(fs + i) : 0;
    const uint32_t bm = __ballot_sync(0xffffffffu, v != 0);
    int base = 0;
    if (lane == 0 && bm != 0u) base = atomicAdd(&s_m, __popc(bm));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (v != 0) {
      const int x = base + __popc(bm & ((1u << lane) - 1u));
      inst[x] = i;
      islot[x] = v - 1;
    }
  }
  __syncthreads();
  const uint64_t* slots = a.spt + (int64_t)r * a.spp;
  for (int x = warp; x < s_m; x += kWarps) {
    const int i = inst[x];
    const int sr = srow[i - e0];
    const uint4* src = sr >= 0 ? (const uint4*)(scratch + (int64_t)sr * a.rec)
                               : (const uint4*)hs_page_row_addr(row, a.page_shift, a.rec, topk[i]);
    if (src == nullptr) continue;  // not reserved (flagged by the deciding CTA)
    copy_rec((uint4*)hs_slot_addr(slots, a.sshift, a.rec, islot[x]), src, sr < 0);
  }
}

template <int NV>
__global__ void __launch_bounds__(kThreads, 1) k_resolve(ResolveArgs a) {
  // CTAs [0, nreq cs) decide, one cluster per request; with early fetch, CTAs [nreq cs, 2 nreq cs)
  // are the requests' fetch CTAs, in clusters of the same size that never use the cluster barrier
  const bool fetcher = (int)blockIdx.x >= a.nreq * a.cs;
  const int b = fetcher ? (int)blockIdx.x - a.nreq * a.cs : (int)blockIdx.x;
  if (fetcher && b >= a.nreq * a.fpr) return;  // a cluster's padding: no request, nothing counted
  const int r = a.r0 + (fetcher ? b / a.fpr : b / a.cs);
  const int crank = fetcher ? b % a.fpr : b % a.cs;  // rank among the request's deciding (fetch) CTAs
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the launch is counted for its requests before the next kernel may start
  if (!fetcher && crank == 0 && threadIdx.x == 0) {
    atomicAdd(&a.res_count[2 * r], 1u);
    __threadfence();
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (fetcher) {
    HS_PHASE(hs_phase_res, 0, threadIdx.x == 0);
    early_fetch_cta(a, r, crank);
    HS_PHASE(hs_phase_res, 22, threadIdx.x == 0);
    count_finished(a, r);
    return;
  }
  HS_PHASE(hs_phase_res, 0, threadIdx.x == 0);
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x;
  const int k = a.k, BK = a.B;              // BK: the configured B (the random key's counter)
  const int32_t* topk = a.topk + (int64_t)(r - a.r0) * k;
  int32_t* tag = a.tag + (int64_t)r * BK;
  uint32_t* stamp = a.stamp + (int64_t)r * BK;
  const uint64_t* slots_g = a.spt + (int64_t)r * a.spp;
  // The loads that start the resolve go out together before any of them is used: the buffer's slot
  // count, this thread's first slots' tags and stamps and top-k entries, the new position, the
  // buffer's slot-page row, the host page-table row and the (request, layer) state.
  constexpr int kBatch = 4;  // slots and top-k entries a thread loads up front (k <= 4 x kThreads)
  const int cap = a.scap[r];
  int32_t tb[kBatch], tk[kBatch];
  uint32_t sb[kBatch];
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    const int j = tid + u * kThreads;
    tb[u] = j < BK ? tag[j] : -1;  // slots past the buffer's B are never used
    sb[u] = j < BK ? stamp[j] : 0u;
    tk[u] = j < k ? topk[j] : -1;
  }
  const int64_t app_p = a.app_pos != nullptr ? a.app_pos[r - a.r0] : -1;
  const uint64_t v_slots = tid < a.spp ? slots_g[tid] : 0ull;
  const bool pt_cached = a.max_pages <= kPageRowCache;  // the row fits in shared memory
  const uint64_t v_pt =
      (pt_cached && tid < a.max_pages) ? a.pt[((int64_t)r * a.L + a.layer) * a.max_pages + tid] : 0ull;
  const hs_rl_state st = a.state[r];
  const int B = min(BK, cap);               // slots this buffer holds: all work is over [0, B)
  const int ht_size = 1 << a.ht_bits;
  int32_t* ht_key = (int32_t*)smem;                 // [ht_size]
  int32_t* ht_val = ht_key + ht_size;               // [ht_size] smallest top-k index of the key
  int32_t* hit_slot = ht_val + ht_size;             // [k]: slot of a hit, -1 miss, -2 invalid
  int32_t* erank = hit_slot + k;                    // [k]: rank of a hit among hits
  int32_t* miss_idx = erank + k;                    // [k]: top-k index of the q-th miss
  int32_t* miss_pos = miss_idx + k;                 // [k]: position of the q-th miss
  int32_t* victims = miss_pos + k;                  // [k]: q-th victim slot (ascending)
  uint32_t* key32 = (uint32_t*)(victims + k);       // [B]: eviction key
  uint8_t* flag = (uint8_t*)(key32 + B);            // [B]: bit 0 hit, bit 1 victim
  __shared__ uint32_t wbuf[kWarps];
  __shared__ uint32_t hist[2][2048];  // the victim select's histograms, zero outside the select
  __shared__ uint32_t sel[2][2];
  __shared__ uint32_t s_cmask[kWarps][16][2];  // compaction: each warp's round masks (B <= 16384)
  __shared__ uint32_t err_bits;
  __shared__ __align__(8) uint64_t bar_stage;  // the early miss copies (one phase per launch)

  int32_t* locs = a.locs + (int64_t)(r - a.r0) * k;
  if (B < k) {
    // too few slots for a step (a buffer not grown): nothing changes; the locations are -1 and the
    // fused append is skipped too (same decision in every CTA of the cluster: no barrier is reached)
    for (int i = crank * kThreads + tid; i < k; i += a.cs * kThreads) locs[i] = -1;
    if (crank == 0 && tid == 0) {
      uint32_t e = (uint32_t)HS_DEVERR_SLOTS;
      if (a.app_pos != nullptr) {
        const int64_t p = a.app_pos[r - a.r0];
        if (p < a.P0 || p < 0 || p >= a.C ||
            hs_page_addr(a.pt, a.max_pages, a.page_shift, a.rec, a.L, r, a.layer, p) == nullptr)
          e |= (uint32_t)HS_DEVERR_APPEND;
      }
      a.state[r].err = st.err | e;
    }
    count_finished(a, r);
    return;
  }
  __shared__ uint64_t s_slots[kMaxSlotPages];  // this buffer's page row (first used after the decision)
  if (tid < a.spp) s_slots[tid] = v_slots;
  __shared__ int s_app_slot;
  __shared__ unsigned long long s_best[kWarps];
  __shared__ int s_found[kWarps];
  __shared__ uint64_t s_pt[kPageRowCache];
  // this (request, layer)'s row of the host page table, cached for the early copies and phase B (the
  // decision's barriers order it before the first use; the pointer is recomputed where it is used
  // rather than kept live)
  if (pt_cached && tid < a.max_pages) s_pt[tid] = v_pt;
  auto pt_row = [&]() -> const uint64_t* {
    return pt_cached ? s_pt : a.pt + ((int64_t)r * a.L + a.layer) * a.max_pages;
  };

  // fetch-in-attention mode: copies a previous resolve left to an attention that never ran are
  // finished first (they target slots this decision may reuse); the cluster barrier below orders
  // them before this resolve rewrites the pending list
  if (a.pend != nullptr && a.pend_live[r] != 0u)
    hs_copy_pending(a.pend + (int64_t)r * k, k, a.rec, slots_g, a.sshift, crank, a.cs);

  // ---------------- phase A: every CTA of the cluster computes the whole decision ----------------
  // The hash table and the select's histograms are cleared while the first loads are in flight.  The
  // hash is then built while the append's slot search reduces, so the two share their barriers, and
  // the probe reuses the tags and stamps loaded at the start.
  // fused write-through append (hs_append_resolve): the new position takes the slot that already
  // holds it, else the slot with the smallest eviction key over the buffer's slots; stamp = clock, clock
  // += 1; the resolve below then sees that state
  // The new position loaded with the rest; its host page is requested by thread 0 once the position
  // has arrived and checked only after the hash, so no thread waits for the two loads in a row here.
  int app_slot = -1;
  uint4* app_dh = nullptr;  // the append's place in the host history (known after the hash)
  __shared__ uint32_t s_dups, s_klo, s_khi, s_dcnt[2];
  __shared__ unsigned long long s_app_page;
  if (tid == 0) {
    err_bits = 0u;
    mbar_init1(&bar_stage);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_dups = 0u;
    s_klo = 0xffffffffu;
    s_khi = 0u;
    s_dcnt[0] = 0u;
    s_dcnt[1] = 0u;
  }
  for (int x = tid; x < ht_size; x += kThreads) {
    ht_key[x] = -1;
    ht_val[x] = 0x7fffffff;
  }
  for (int x = tid; x < 2 * 2048; x += kThreads) hist[x >> 11][x & 2047] = 0u;
  // the append position must lie in [shared_prefix, capacity) and on a reserved host page
  const bool app_try = a.app_pos != nullptr && app_p >= a.P0 && app_p >= 0 && app_p < a.C;
  unsigned long long app_page = 0ull;  // requested here, used after the hash
  if (tid == 0 && app_try)
    app_page = a.pt[((int64_t)r * a.L + a.layer) * a.max_pages + (app_p >> a.page_shift)];
  __syncthreads();

  HS_PHASE(hs_phase_res, 1, tid == 0);
  // (1) hash the selected positions; a key keeps the smallest top-k index that carries it.  Entries
  // start as misses (-1) or invalid (-2); repeats are sorted out below only when an insert met its key.
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    const int i = tid + u * kThreads;
    if (i >= k) break;
    const int32_t sv = tk[u];
    int32_t state = -2;
    if (sv >= 0 && (int64_t)sv < a.C) {
      uint32_t hh = ht_hash(sv, a.ht_bits);
      while (true) {
        const int32_t prev = atomicCAS(&ht_key[hh], -1, sv);
        if (prev == -1 || prev == sv) {
          atomicMin(&ht_val[hh], i);
          if (prev == sv) s_dups = 1u;
          break;
        }
        hh = (hh + 1) & (uint32_t)(ht_size - 1);
      }
      state = -1;
    } else if (sv != -1) {
      atomicOr(&err_bits, (uint32_t)HS_DEVERR_RANGE);
    }
    hit_slot[i] = state;
  }
  HS_PHASE(hs_phase_res, 10, tid == 0);  // this thread's hash inserts done
  // the append's slot search over the tags and stamps already loaded (and the rest of the slots)
  if (app_try) {
    int found = 0x7fffffff;
    unsigned long long best = ~0ull;
    auto visit = [&](int j, int32_t t, uint32_t sj) {
      if (t == (int32_t)app_p) found = min(found, j);
      const uint32_t key = hs_evict_key(a.policy, t, sj, a.seed, st.nres, a.R, r, a.L, a.layer, BK, j);
      const unsigned long long kj = ((unsigned long long)key << 32) | (unsigned)j;
      best = kj < best ? kj : best;
    };
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = tid + u * kThreads;
      if (j < B) visit(j, tb[u], sb[u]);
    }
    for (int j = tid + kBatch * kThreads; j < B; j += kThreads) visit(j, tag[j], stamp[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      found = min(found, __shfl_xor_sync(0xffffffffu, found, o));
      const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
      best = y < best ? y : best;
    }
    if ((tid & 31) == 0) {
      s_found[tid >> 5] = found;
      s_best[tid >> 5] = best;
    }
  }
  HS_PHASE(hs_phase_res, 11, tid == 0);  // this warp's append search reduced
  __syncthreads();  // the hash table and the append's per-warp results are complete
  HS_PHASE(hs_phase_res, 12, tid == 0);
  if (tid == 0) {
    s_app_page = app_page;
    if (a.app_pos != nullptr && app_page == 0ull) atomicOr(&err_bits, (uint32_t)HS_DEVERR_APPEND);
  }
  if (app_try && tid < 32) {  // one warp combines the warps' results
    int f = tid < kWarps ? s_found[tid] : 0x7fffffff;
    unsigned long long bb = tid < kWarps ? s_best[tid] : ~0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      f = min(f, __shfl_xor_sync(0xffffffffu, f, o));
      const unsigned long long y = __shfl_xor_sync(0xffffffffu, bb, o);
      bb = y < bb ? y : bb;
    }
    if (tid == 0) s_app_slot = f != 0x7fffffff ? f : (int)(bb & 0xffffffffull);
  }
  if (s_dups != 0u) {  // a repeated position: only its first occurrence (smallest index) is valid
    for (int i = tid; i < k; i += kThreads) {
      if (hit_slot[i] != -1) continue;
      const int32_t sv = topk[i];
      uint32_t hh = ht_hash(sv, a.ht_bits);
      while (ht_key[hh] != sv) hh = (hh + 1) & (uint32_t)(ht_size - 1);
      if (ht_val[hh] != i) {
        hit_slot[i] = -2;
        atomicOr(&err_bits, (uint32_t)HS_DEVERR_DUP);
      }
    }
  }
  __syncthreads();  // the append's slot and the sorted-out repeats are known
  if (app_try && s_app_page != 0ull) {
    app_dh = (uint4*)((uint8_t*)(uintptr_t)s_app_page + (app_p & ((1ll << a.page_shift) - 1)) * a.rec);
    app_slot = s_app_slot;
  }
  const uint32_t clock = st.clock + (app_slot >= 0 ? 1u : 0u);  // the resolve's clock
  if (tid == 0 && (uint64_t)clock + (uint64_t)k >= 0xFFFFFFFFull) atomicOr(&err_bits, (uint32_t)HS_DEVERR_CLOCK);

  HS_PHASE(hs_phase_res, 2, tid == 0);
  // (2) probe every slot; keep its eviction key and the candidates' key range (the tags and stamps of
  // a thread's first kBatch slots are the ones loaded at the start).
  uint32_t klo = 0xffffffffu, khi = 0u;
  auto probe_slot = [&](int j, int32_t tj, uint32_t sj) {
    const bool is_app = j == app_slot;
    const int32_t t = is_app ? (int32_t)app_p : tj;
    const uint32_t stj = is_app ? st.clock : sj;
    uint8_t f = 0;
    if (t >= 0) {
      uint32_t h = ht_hash(t, a.ht_bits);
      while (true) {
        const int32_t key = ht_key[h];
        if (key == t) {
          hit_slot[ht_val[h]] = j;
          f = 1;
          break;
        }
        if (key == -1) break;
        h = (h + 1) & (uint32_t)(ht_size - 1);
      }
    }
    flag[j] = f;
    const uint32_t key = hs_evict_key(a.policy, t, stj, a.seed, st.nres, a.R, r, a.L, a.layer, BK, j);
    key32[j] = key;
    if (f == 0) {
      klo = min(klo, key);
      khi = max(khi, key);
    }
  };
  {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = tid + u * kThreads;
      if (j < B) probe_slot(j, tb[u], sb[u]);
    }
    for (int j = tid + kBatch * kThreads; j < B; j += kThreads) probe_slot(j, tag[j], stamp[j]);
  }
  HS_PHASE(hs_phase_res, 13, tid == 0);  // this thread's probes done
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    klo = min(klo, __shfl_xor_sync(0xffffffffu, klo, o));
    khi = max(khi, __shfl_xor_sync(0xffffffffu, khi, o));
  }
  if ((tid & 31) == 0) {
    atomicMin(&s_klo, klo);
    atomicMax(&s_khi, khi);
  }
  __syncthreads();
  // every old tag and stamp this CTA needs has been read and used: the cluster's writes may follow
  if (a.cs > 1) cluster_arrive_relaxed();

  HS_PHASE(hs_phase_res, 3, tid == 0);
  // (3a) rank hits and misses in top-k order; list the misses.  Each warp takes a run of consecutive
  // entries, 32 at a time, and ranks its lanes by ballot.
  const int lane = tid & 31;
  const uint32_t below = (1u << lane) - 1u;  // the lanes before this one
  const int kchunk = (((k + kWarps - 1) / kWarps) + 31) & ~31;
  const int i0 = min(k, (tid >> 5) * kchunk), i1 = min(k, i0 + kchunk);
  uint32_t local = 0;
  for (int ib = i0; ib < i1; ib += 32) {
    const int i = ib + lane;
    const int32_t hs = i < i1 ? hit_slot[i] : -2;
    local += (uint32_t)__popc(__ballot_sync(0xffffffffu, hs >= 0)) +
             ((uint32_t)__popc(__ballot_sync(0xffffffffu, hs == -1)) << 16);
  }
  uint32_t tot;
  const uint32_t pre = __shfl_sync(0xffffffffu, cta_exclusive_scan(lane == 0 ? local : 0u, wbuf, &tot), 0);
  const int h = (int)(tot & 0xffffu), m = (int)(tot >> 16);
  {
    uint32_t a_rank = pre & 0xffffu, q_rank = pre >> 16;
    for (int ib = i0; ib < i1; ib += 32) {
      const int i = ib + lane;
      const int32_t hs = i < i1 ? hit_slot[i] : -2;
      const uint32_t bh = __ballot_sync(0xffffffffu, hs >= 0), bm = __ballot_sync(0xffffffffu, hs == -1);
      if (hs >= 0) {
        erank[i] = (int32_t)(a_rank + (uint32_t)__popc(bh & below));
      } else if (hs == -1) {
        const uint32_t q = q_rank + (uint32_t)__popc(bm & below);
        miss_idx[q] = i;
        miss_pos[q] = topk[i];
      }
      a_rank += (uint32_t)__popc(bh);
      q_rank += (uint32_t)__popc(bm);
    }
  }

  HS_PHASE(hs_phase_res, 4, tid == 0);
  // (4, early) this CTA's first misses start crossing the host link now; the victims are chosen
  // meanwhile and the staged records reach their slots in phase B.  One bulk copy per record (lane 0
  // of warp e mod 32 issues record e), completing on bar_stage: each issuer adds its record's bytes
  // to the barrier's transaction count before its copy, and thread 0 arrives once every issuer has
  // (after the select's barriers), so the phase completes when every staged record has landed.
  // Bulk copies leave the load units free, where 16-byte copies from host memory filled their queues
  // and held the issuing threads back from the select.
  const int q0 = (int)((int64_t)m * crank / a.cs), q1 = (int)((int64_t)m * (crank + 1) / a.cs);
  // 128-byte aligned (the launch adds the slack), like the host records
  uint8_t* stage = (uint8_t*)(((uintptr_t)(smem + a.stage_off) + 127u) & ~(uintptr_t)127u);
  const int nstage = a.pend == nullptr ? min(q1 - q0, a.stage_recs) : 0;
  if (nstage > 0) {
    __syncthreads();  // the miss list is complete
    if ((tid & 31) == 0) {
      const uint64_t* row = pt_row();
      for (int e = tid >> 5; e < nstage; e += kWarps) {
        const uint8_t* src = hs_page_row_addr(row, a.page_shift, a.rec, miss_pos[q0 + e]);
        if (src != nullptr) {
          mbar_expect(&bar_stage, (uint32_t)a.rec);
          bulk_copy_g2s(stage + (int64_t)e * a.rec, src, (uint32_t)a.rec, &bar_stage);
        }
      }
    }
  }

  HS_PHASE(hs_phase_res, 5, tid == 0);
  // (3b) threshold of the m smallest candidate keys
  const int ncand = B - h;
  const bool take_all = (m == ncand);
  uint32_t T = 0u, need_eq = 0u;
  if (m > 0 && !take_all) {
    // distinct nonzero keys (every policy but random): one bitmap pass over a window that ends at the
    // largest key (or starts at the smallest when no slot is empty), else the radix select
    const uint32_t lo = s_klo != 0u ? s_klo : (s_khi >= kDenseSpan ? s_khi - (kDenseSpan - 1u) : 1u);
    const bool dense = a.policy != HS_POLICY_RANDOM && s_khi - lo < kDenseSpan &&
                       select_dense(key32, flag, B, (uint32_t)m, lo, wbuf, hist, sel, s_dcnt, &T, &need_eq);
    if (!dense) select_threshold(key32, flag, B, (uint32_t)m, s_klo, s_khi, wbuf, hist, sel, &T, &need_eq);
  }
  if (nstage > 0) {
    __syncthreads();  // every early copy has been issued (with its bytes expected)
    if (tid == 0 && a.stall == 0) mbar_arrive1(&bar_stage);
  }

  HS_PHASE(hs_phase_res, 6, tid == 0);
  // (3c) ordered compaction: the q-th victim in ascending slot order.  A slot is a victim when its
  // key is below T, or equals T and fewer than need_eq slots below it do; each warp takes a run of
  // consecutive slots, 32 at a time, and ranks its lanes by ballot.
  if (m > 0) {
    const int chunk = (((B + kWarps - 1) / kWarps) + 31) & ~31;
    const int j0 = min(B, (tid >> 5) * chunk), j1 = min(B, j0 + chunk);
    auto classify = [&](int j, bool& lt, bool& eq) {
      lt = false;
      eq = false;
      if (j < j1 && !(flag[j] & 1u)) {
        if (take_all) {
          lt = true;
        } else {
          const uint32_t key = key32[j];
          lt = key < T;
          eq = key == T;
        }
      }
    };
    // the counting pass keeps each 32-slot round's masks (below T, equal to T) for the placing pass
    uint32_t(*masks)[2] = s_cmask[tid >> 5];
    uint32_t cnt = 0;
    for (int jb = j0, it = 0; jb < j1; jb += 32, ++it) {
      bool lt, eq;
      classify(jb + lane, lt, eq);
      const uint32_t bl = __ballot_sync(0xffffffffu, lt), be = __ballot_sync(0xffffffffu, eq);
      if (lane == 0) {
        masks[it][0] = bl;
        masks[it][1] = be;
      }
      cnt += (uint32_t)__popc(bl) + ((uint32_t)__popc(be) << 16);
    }
    uint32_t tot2;
    const uint32_t pre2 = __shfl_sync(0xffffffffu, cta_exclusive_scan(lane == 0 ? cnt : 0u, wbuf, &tot2), 0);
    HS_PHASE(hs_phase_res, 18, tid == 0);  // compaction counts scanned
    uint32_t less_b = pre2 & 0xffffu, eq_b = pre2 >> 16;
    for (int jb = j0, it = 0; jb < j1; jb += 32, ++it) {
      const uint32_t bl = masks[it][0], be = masks[it][1];
      if (((bl | be) >> lane) & 1u) {
        const uint32_t lb = less_b + (uint32_t)__popc(bl & below), eb = eq_b + (uint32_t)__popc(be & below);
        int q = -1;
        if ((bl >> lane) & 1u) {
          q = (int)(lb + min(eb, need_eq));
        } else if (eb < need_eq) {
          q = (int)(lb + eb);
        }
        if (q >= 0) {
          const int j = jb + lane;
          victims[q] = j;
          flag[j] |= 2u;
        }
      }
      less_b += (uint32_t)__popc(bl);
      eq_b += (uint32_t)__popc(be);
    }
  }
  HS_PHASE(hs_phase_res, 19, tid == 0);  // this thread's victims placed
  // every CTA of the request has read the old tags and stamps before anyone writes them
  __syncthreads();
  HS_PHASE(hs_phase_res, 20, tid == 0);
  if (a.cs > 1) cluster_wait();
  HS_PHASE(hs_phase_res, 7, tid == 0);

  // ---------------- phase B: this CTA's share of the writes and of the fetch ----------------
  {
    const int e0 = (int)((int64_t)k * crank / a.cs), e1 = (int)((int64_t)k * (crank + 1) / a.cs);
    for (int i = e0 + tid; i < e1; i += kThreads) {
      const int32_t hs = hit_slot[i];
      if (hs >= 0) {
        if (a.policy != HS_POLICY_FIFO) stamp[hs] = clock + (uint32_t)erank[i];
        locs[i] = hs;
      } else if (hs == -2) {
        locs[i] = -1;
      }
      if (a.pend != nullptr && hs != -1) a.pend[(int64_t)r * k + i] = hs_pending{0ull, -1, -1};
    }
    for (int q = q0 + tid; q < q1; q += kThreads) {
      const int j = victims[q];
      tag[j] = miss_pos[q];
      if (a.pos_slot != nullptr) a.pos_slot[(int64_t)r * a.C + miss_pos[q]] = j;
      stamp[j] = a.policy == HS_POLICY_FIFO ? clock + (uint32_t)q : clock + (uint32_t)h + (uint32_t)q;
      locs[miss_idx[q]] = j;
      if (a.pend != nullptr) {
        // the record's host address, resolved once here; a page not reserved leaves nothing pending
        const uint8_t* src = hs_page_row_addr(pt_row(), a.page_shift, a.rec, miss_pos[q]);
        if (src == nullptr) atomicOr(a.err_global, (uint32_t)HS_DEVERR_PAGE);
        a.pend[(int64_t)r * k + miss_idx[q]] = hs_pending{(uint64_t)(uintptr_t)src, src ? j : -1, miss_pos[q]};
      }
    }
    if (a.policy == HS_POLICY_SWAP_VANILLA) {
      const int s0 = (int)((int64_t)B * crank / a.cs), s1 = (int)((int64_t)B * (crank + 1) / a.cs);
      for (int j = s0 + tid; j < s1; j += kThreads) {
        if (flag[j] == 0u) {
          tag[j] = -1;
          stamp[j] = 0u;
        }
      }
    }
    // the fused append's own writes (CTA 0): the record to the host history always; slot, tag and
    // stamp unless the resolve reuses or empties that slot now, the stamp only where no hit restamps it
    if (app_slot >= 0 && crank == 0) {
      const uint4* src = (const uint4*)(a.app_rec + (int64_t)(r - a.r0) * a.rec);
      uint4* dh = app_dh;
      // the slot is rewritten by the resolve when it is a victim now, or emptied by swap-vanilla
      // when it holds no selected position
      const bool evicted = (flag[app_slot] & 2u) != 0u ||
                           (a.policy == HS_POLICY_SWAP_VANILLA && (flag[app_slot] & 1u) == 0u);
      const bool restamped = (flag[app_slot] & 1u) != 0u && a.policy != HS_POLICY_FIFO;
      uint4* db = (uint4*)hs_slot_addr(s_slots, a.sshift, a.rec, app_slot);
      const int nv = (int)(a.rec / 16);
      for (int x = tid; x < nv; x += kThreads) {
        const uint4 v = src[x];
        dh[x] = v;
        if (!evicted) db[x] = v;
      }
      if (tid == 0 && !evicted) {
        tag[app_slot] = (int32_t)app_p;
        if (a.pos_slot != nullptr) a.pos_slot[(int64_t)r * a.C + app_p] = app_slot;
        if (!restamped) stamp[app_slot] = st.clock;
      }
    }
    HS_PHASE(hs_phase_res, 8, tid == 0);
    // (4) fetch this CTA's share of the misses from the host history (or leave it to the attention,
    // or to the fetch CTAs: they are told each miss's slot, once every deciding CTA has written its
    // share)
    if (a.fslot != nullptr) {
      for (int q = q0 + tid; q < q1; q += kThreads) {
        if (hs_page_row_addr(pt_row(), a.page_shift, a.rec, miss_pos[q]) == nullptr)
          atomicOr(a.err_global, (uint32_t)HS_DEVERR_PAGE);
        a.fslot[(int64_t)r * k + miss_idx[q]] = victims[q] + 1;
      }
      __syncthreads();
      if (tid == 0 && !(a.fstall != 0 && r == a.r0)) {
        __threadfence();
        atomicAdd(&a.fdec[r], 1u);
      }
    } else if (a.pend == nullptr && q1 > q0) {
      // host addresses of this CTA's misses, resolved once (in the hash table's space: dead by now)
      uint64_t* s_src = (uint64_t*)ht_key;
      const uint64_t* row = pt_row();
      for (int q = q0 + tid; q < q1; q += kThreads) {
        const uint8_t* src = hs_page_row_addr(row, a.page_shift, a.rec, miss_pos[q]);
        if (src == nullptr) atomicOr(a.err_global, (uint32_t)HS_DEVERR_PAGE);
        s_src[q - q0] = (uint64_t)(uintptr_t)src;
      }
      // the rest straight from the host, then the staged ones from shared memory
      __syncthreads();
      fetch_misses<NV>(a, q0 + nstage, q1, s_src + nstage, victims, s_slots);
      if (nstage > 0) {
        // the staged records have landed (bounded: a wait that gives up flags the resolve and skips
        // the staged records, after a second bounded wait for copies still in flight)
        bool landed = mbar_wait_1s(&bar_stage, 0u);
        if (!landed) {
          atomicOr(a.err_global, (uint32_t)HS_DEVERR_TIMEOUT);
          mbar_wait_1s(&bar_stage, 0u);
        }
        const int vpr = (int)(a.rec / 16);
        for (int x = tid; landed && x < nstage * vpr; x += kThreads) {
          const int e = x / vpr, v = x - e * vpr;
          if (s_src[e] == 0ull) continue;  // page not reserved (flagged): nothing was staged
          *((uint4*)hs_slot_addr(s_slots, a.sshift, a.rec, victims[q0 + e]) + v) = *((const uint4*)(stage + (int64_t)e * a.rec) + v);
        }
      }
    }
  }

  HS_PHASE(hs_phase_res, 9, tid == 0);
  // (5) clock and counters
  if (crank == 0 && tid == 0) {
    hs_rl_state ns = st;
    ns.clock = clock + (uint32_t)k;
    ns.nres = st.nres + 1u;
    ns.err = st.err | err_bits;
    a.state[r] = ns;
    unsigned long long* c = a.counters + (int64_t)r * 4;
    c[0] += (unsigned long long)h;
    c[1] += (unsigned long long)m;
    if (app_slot >= 0) c[2] += 1ull;
    c[3] += (unsigned long long)m * (unsigned long long)a.rec;
    if (a.step_log != nullptr && st.nres < (uint32_t)a.log_steps)
      a.step_log[((int64_t)st.nres * a.L + a.layer) * a.R + r] = (uint32_t)m;
    if (a.pend != nullptr) a.pend_live[r] = 1u;
  }
  count_finished(a, r);
}

struct AppendArgs {
  const int64_t* pos;    // [R]
  const uint8_t* rec_in; // [R][rec]
  int32_t* tag;
  uint32_t* stamp;
  hs_rl_state* state;
  unsigned long long* counters;
  const uint64_t* pt;    // host page table [R][L][max_pages]
  uint32_t* err_global;
  const uint64_t* spt;   // layer slice [R][spp] of the slot table
  const int32_t* scap;   // layer slice [R]: slots each buffer holds
  int64_t C, P0, max_pages, rec;
  int page_shift, sshift, spp;
  uint64_t seed;
  const hs_pending* pend;  // fetch-in-attention mode: layer slice [R][k], else null
  uint32_t* pend_live;
  int32_t* pos_slot;       // early fetch: layer slice [R][C] of the position -> slot map, else null
  int R, L, layer, B, policy, k;
};

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads) k_append(AppendArgs a) {
  hs_pdl_enter();
  const int r = blockIdx.x, tid = threadIdx.x;
  if (a.pend != nullptr && a.pend_live[r] != 0u) {
    // finish the copies a previous resolve left pending before this append may overwrite a slot
    hs_copy_pending(a.pend + (int64_t)r * a.k, a.k, a.rec, a.spt + (int64_t)r * a.spp, a.sshift, 0, 1);
    __syncthreads();
    if (tid == 0) a.pend_live[r] = 0u;
  }
  const int64_t p = a.pos[r];
  const hs_rl_state st = a.state[r];
  uint4* dh = (p >= a.P0 && p >= 0 && p < a.C)
                  ? (uint4*)hs_page_addr(a.pt, a.max_pages, a.page_shift, a.rec, a.L, r, a.layer, p)
                  : nullptr;
  if (dh == nullptr) {  // outside [shared_prefix, capacity), or its host page is not reserved
    if (tid == 0) a.state[r].err = st.err | (uint32_t)HS_DEVERR_APPEND;
    return;
  }
  const int B = min(a.B, a.scap[r]);  // slots this buffer holds
  if (B < a.k) {                      // too few for a step: nothing changes
    if (tid == 0) a.state[r].err = st.err | (uint32_t)HS_DEVERR_SLOTS;
    return;
  }
  int32_t* tag = a.tag + (int64_t)r * a.B;
  uint32_t* stamp = a.stamp + (int64_t)r * a.B;
  int found = 0x7fffffff;
  unsigned long long best = ~0ull;
  for (int j = tid; j < B; j += kAppendThreads) {
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
  uint4* db = (uint4*)hs_slot_addr(a.spt + (int64_t)r * a.spp, a.sshift, a.rec, slot);
  const int nv = (int)(a.rec / 16);
  for (int x = tid; x < nv; x += kAppendThreads) {
    const uint4 v = src[x];
    dh[x] = v;
    db[x] = v;
  }
  if (tid == 0) {
    tag[slot] = (int32_t)p;
    if (a.pos_slot != nullptr) a.pos_slot[(int64_t)r * a.C + p] = slot;
    stamp[slot] = st.clock;
    hs_rl_state ns = st;
    ns.clock = st.clock + 1u;
    if ((uint64_t)st.clock + 1u >= 0xFFFFFFFFull) ns.err |= (uint32_t)HS_DEVERR_CLOCK;
    a.state[r] = ns;
    a.counters[(int64_t)r * 4 + 2] += 1ull;
  }
}

// Early miss copies: 32 KB per CTA is what the host link moves in the ~10 us the victims take to
// choose, with 64 CTAs fetching; a larger area issues more copies than the link drains and holds the
// decision back (measured on the GQA decode workload with 16-byte copies: 16 KB +4%, 32 KB +6%, 96 KB
// -1% per layer-step; with bulk copies, whose issue waits once a few are in flight from host memory:
// 96 KB -5% on the GQA workload, -8% on the stress batch).  HS_STAGE_KB builds another size.
#ifndef HS_STAGE_KB
#define HS_STAGE_KB 32
#endif
constexpr size_t kStageBytes = (size_t)HS_STAGE_KB * 1024;
constexpr size_t kDynSmemCap = kResolveDynSmemCap;

// Shared memory of the decision's arrays with a hash table of 2^bits entries.
size_t decision_smem(const hs_config* c, int bits) {
  return ((size_t)1 << bits) * 8 + (size_t)c->top_k * 24 + (size_t)c->buffer_slots * 5;
}

// Hash table of the selected positions: at most a quarter full where that leaves room for the early
// miss copies, else at most half full.  Every probe of a slot whose tag is not selected runs to an
// empty entry, and a warp waits for its longest chain: on the batch-8 shared-latent workload a half
// full table made the probe pass 2.6 us of a ~21 us decision.
int ht_bits_for(const hs_config* c) {
  int bits = 1;
  while ((1 << bits) < 2 * c->top_k) ++bits;
  return decision_smem(c, bits + 1) + kStageBytes <= kDynSmemCap ? bits + 1 : bits;
}

}  // namespace

size_t hs_resolve_smem_bytes(const hs_config* c) { return decision_smem(c, ht_bits_for(c)); }

namespace {

// Dynamic shared memory of a resolve launch: the decision's arrays, then (misses copied by the
// resolve) a staging area for the early miss copies, up to kStageBytes within kDynSmemCap in all.
size_t resolve_launch_smem(const hs_config* c, int* stage_off, int* stage_recs) {
  const size_t base = (hs_resolve_smem_bytes(c) + 127) & ~(size_t)127;
  const size_t rec = (size_t)hs_record_bytes(c);
  size_t room = base < kDynSmemCap ? kDynSmemCap - base : 0;
  room = room < kStageBytes ? room : kStageBytes;
  *stage_off = (int)base;
  *stage_recs = (c->fetch_in_attention || c->early_fetch) ? 0 : (int)(room / rec);
  return base + (size_t)*stage_recs * rec + (*stage_recs > 0 ? 128 : 0);  // + alignment slack
}

template <int NV>
cudaError_t launch_resolve_nv(const ResolveArgs* a, int nreq, int cs, size_t smem, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  // the fetch CTAs follow the deciding ones, rounded up to whole clusters
  const int nf = a->fslot != nullptr ? (nreq * a->fpr + cs - 1) / cs * cs : 0;
  cfg.gridDim = dim3((unsigned)(nreq * cs + nf), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_resolve<NV>, *a);
}

template <int NV>
int prepare_nv(const hs_config* c, int num_sms, int* cs_out) {
  int stage_off, stage_recs;
  const int smem = (int)resolve_launch_smem(c, &stage_off, &stage_recs);
  if (hs_raise_smem_limit(k_resolve<NV>, smem) != cudaSuccess) return HS_ERR_CUDA;
  // the same (largest) shared-memory carveout as the attention kernels, so the SMs keep their
  // L1/shared split from one kernel of a decode step to the next
  if (cudaFuncSetAttribute(k_resolve<NV>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return HS_ERR_CUDA;
  // largest cluster (<= 8 CTAs per request) that lets every request's cluster be resident at once
  *cs_out = 1;
  for (int cs = 8; cs >= 2; cs /= 2) {
    if (cs * c->num_requests > num_sms) continue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(c->num_requests * cs), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_resolve<NV>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (n >= c->num_requests) {
      *cs_out = cs;
      break;
    }
  }
  return HS_OK;
}

}  // namespace

int hs_launch_resolve(hs_pool* p, int layer, int r0, int nreq, const int64_t* d_pos, const void* d_rec,
                      const int32_t* d_topk, int32_t* d_locs, cudaStream_t st) {
  const hs_config& c = p->cfg;
  const int64_t R = c.num_requests, B = c.buffer_slots;
  ResolveArgs a{};
  a.topk = d_topk;
  a.locs = d_locs;
  a.tag = p->tag + (int64_t)layer * R * B;
  a.stamp = p->stamp + (int64_t)layer * R * B;
  a.state = p->state + (int64_t)layer * R;
  a.counters = p->counters + (int64_t)layer * R * 4;
  a.step_log = c.log_steps > 0 ? p->step_log : nullptr;
  a.pt = p->page_table;
  a.err_global = p->err_global;
  a.spt = p->slot_table + (int64_t)layer * R * p->slot_pages;
  a.scap = p->slot_cap + (int64_t)layer * R;
  a.sshift = p->slot_shift;
  a.spp = p->slot_pages;
  a.C = c.capacity;
  a.P0 = c.shared_prefix;
  a.max_pages = p->max_pages;
  a.page_shift = p->page_shift;
  a.rec = p->rec;
  a.seed = c.seed;
  a.R = c.num_requests;
  a.L = c.num_layers;
  a.layer = layer;
  a.B = c.buffer_slots;
  a.k = c.top_k;
  a.policy = c.policy;
  a.log_steps = c.log_steps;
  a.ht_bits = ht_bits_for(&c);
  a.cs = p->resolve_cs;
  a.pend = p->pend != nullptr ? p->pend + (int64_t)layer * R * c.top_k : nullptr;
  a.pend_live = p->pend_live != nullptr ? p->pend_live + (int64_t)layer * R : nullptr;
  a.app_pos = d_pos;
  a.app_rec = (const uint8_t*)d_rec;
  a.r0 = r0;
  a.nreq = nreq;
  a.res_count = p->res_count + (int64_t)layer * R * 2;
  if (p->fslot != nullptr) {
    a.pos_slot = p->pos_slot + (int64_t)layer * R * c.capacity;
    a.fslot = p->fslot + (int64_t)layer * R * c.top_k;
    a.fdec = p->fdec + (int64_t)layer * R;
    a.ffin = p->ffin + (int64_t)layer * R;
    a.fpr = p->resolve_ctas - p->resolve_cs;
    a.fscratch = p->fscratch + (int64_t)layer * R * a.fpr * p->fetch_rows * p->rec;
    a.fetch_rows = p->fetch_rows;
    if ((p->debug_stall & HS_STALL_FETCH) != 0) {  // test hook
      a.fstall = 1;
      p->debug_stall &= ~HS_STALL_FETCH;
    }
  }
  // an attention launched right after a whole-batch resolve of its layer on the same stream may
  // wait for its own request's resolve CTAs instead of the whole grid
  p->last_res_layer = (r0 == 0 && nreq == R) ? layer : -1;
  p->last_res_stream = st;
  const size_t smem = resolve_launch_smem(&c, &a.stage_off, &a.stage_recs);
  if (a.stage_recs > 0 && a.pend == nullptr && (p->debug_stall & HS_STALL_RESOLVE) != 0) {  // test hook
    a.stall = 1;
    p->debug_stall &= ~HS_STALL_RESOLVE;
  }
  cudaError_t e;
  switch (c.io_chunk_bytes) {
    case 16: e = launch_resolve_nv<1>(&a, nreq, a.cs, smem, st); break;
    case 32: e = launch_resolve_nv<2>(&a, nreq, a.cs, smem, st); break;
    case 64: e = launch_resolve_nv<4>(&a, nreq, a.cs, smem, st); break;
    default: e = launch_resolve_nv<8>(&a, nreq, a.cs, smem, st); break;
  }
  return e == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

// Kernel attributes and the cluster size are fixed once at pool creation; launches stay capturable.
int hs_resolve_prepare(hs_pool* p) {
  const hs_config* c = &p->cfg;
  switch (c->io_chunk_bytes) {
    case 16: return prepare_nv<1>(c, p->num_sms, &p->resolve_cs);
    case 32: return prepare_nv<2>(c, p->num_sms, &p->resolve_cs);
    case 64: return prepare_nv<4>(c, p->num_sms, &p->resolve_cs);
    default: return prepare_nv<8>(c, p->num_sms, &p->resolve_cs);
  }
}

int hs_launch_append(hs_pool* p, int layer, const int64_t* d_pos, const void* d_rec, cudaStream_t st) {
  p->last_res_layer = -1;
  const hs_config& c = p->cfg;
  const int64_t R = c.num_requests, B = c.buffer_slots;
  AppendArgs a;
  a.pos = d_pos;
  a.rec_in = (const uint8_t*)d_rec;
  a.tag = p->tag + (int64_t)layer * R * B;
  a.stamp = p->stamp + (int64_t)layer * R * B;
  a.state = p->state + (int64_t)layer * R;
  a.counters = p->counters + (int64_t)layer * R * 4;
  a.pt = p->page_table;
  a.err_global = p->err_global;
  a.spt = p->slot_table + (int64_t)layer * R * p->slot_pages;
  a.scap = p->slot_cap + (int64_t)layer * R;
  a.sshift = p->slot_shift;
  a.spp = p->slot_pages;
  a.C = c.capacity;
  a.P0 = c.shared_prefix;
  a.max_pages = p->max_pages;
  a.page_shift = p->page_shift;
  a.rec = p->rec;
  a.seed = c.seed;
  a.R = c.num_requests;
  a.L = c.num_layers;
  a.layer = layer;
  a.B = c.buffer_slots;
  a.policy = c.policy;
  a.k = c.top_k;
  a.pend = p->pend != nullptr ? p->pend + (int64_t)layer * R * c.top_k : nullptr;
  a.pend_live = p->pend_live != nullptr ? p->pend_live + (int64_t)layer * R : nullptr;
  a.pos_slot = p->pos_slot != nullptr ? p->pos_slot + (int64_t)layer * R * c.capacity : nullptr;
  k_append<<<c.num_requests, kAppendThreads, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}
