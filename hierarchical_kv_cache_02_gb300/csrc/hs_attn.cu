// Sparse attention over resolved slots (HiSparse summary §3 step (4): the physical slots
// published by RESOLVE go to the sparse-attention backend, which gathers exactly those records).
//
// Kernels in this file:
//   * k_attn_gqa: GQA records, one CTA per (request, KV head); bulk-copy producers and consumers
//     on mma.sync in a transposed form (tokens on the MMA's row side);
//   * k_attn_mla_pipe: shared-latent records with 64 query heads on tcgen05 tensor cores, the
//     accumulators in tensor memory, Q loaded once by TMA and the tiles streamed through a ring by
//     16-byte cp.async; split partials merged by k_combine_wide;
//   * k_attn_cc: CUDA-core fallback for other shared-latent head counts (a producer warp gathers
//     whole records with cp.async.bulk into a 3-stage ring; consumers reduce 32 logits per lane
//     with a transposed butterfly and keep an online softmax in base 2).
// In every kernel a split is a fixed range of top-k entries and all reductions run in a fixed
// order, so the result depends only on the top-k order, never on which slot holds a record:
// cold, warm and fully-resident runs are bit-identical.  Partials are combined in split order
// by the last CTA to finish (atomic ticket, no waiting) or by k_combine_wide.
#include <cuda.h>  // CUtensorMap (the encoder is reached through the runtime's driver entry point)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <new>

#include "hs_internal.cuh"

#ifdef HS_PHASE_TRACE
// phase stamps of k_attn_mla_pipe (see HS_PHASE); read and cleared by the two calls below
__device__ unsigned long long hs_phase_attn[256][64];
extern "C" int hs_phase_attn_read(void* host) {
  return (int)cudaMemcpyFromSymbol(host, hs_phase_attn, sizeof(hs_phase_attn));
}
extern "C" int hs_phase_attn_clear() {
  static unsigned long long zero[256][64];
  return (int)cudaMemcpyToSymbol(hs_phase_attn, zero, sizeof(zero));
}
#endif

namespace {

constexpr int kStages = 3;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnArgs {
  const uint16_t* q;     // [R][Hq][DK] bf16
  const int32_t* locs;   // [R][k]
  const uint8_t* kv;     // caller rows (kv_pt null): row (r, loc) at kv + (r * rows + loc) * rec
  const uint64_t* kv_pt; // hot-buffer rows: [R][kv_pages] device address of each buffer page
  const int32_t* kv_cap; // hot-buffer rows: [R] rows each buffer holds (<= rows)
  int kv_pages, kv_shift;
  float* out;            // [R][Hq][DV]
  float* part;           // [R][S][Hq][DV]
  float* ml;             // [R][S][Hq][2]
  uint32_t* ticket;      // [R][groups + 1]: split tickets per group, then the pending-list count
  uint32_t* err;
  int64_t rows, rec;     // rows: per request (the configured B for the hot buffer)
  int64_t kstride, vdelta;  // K of KV block g at g * kstride, V at K + vdelta (bytes)
  float qscale;             // scale * log2(e)
  int R, Hq, k, S, chunk, groups;  // R: requests in this launch (the grid), starting at r0
  int r0;                   // first request: q, locs and out are indexed from it, pool state absolutely
  // fetch-in-attention mode (hot-buffer rows only): misses still to copy from the host history
  const hs_pending* pend;   // [R][k] host address and slot of a miss still to copy (src 0: none); null: none
  uint32_t* pend_live;      // [R]
  int L, layer;
  int stall;                // test hook (hs_debug_stall_next): leave the first ring slot's arrival out
  // set when the launch directly follows the whole-batch resolve of its layer on its stream: that
  // resolve's [R][2] counters (launches, CTAs finished) and its CTAs per request
  const uint32_t* res_count;
  int res_cs;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Rows of request r.  A hot buffer is paged (a row of page addresses); caller rows are contiguous
// and take the form of one page of 2^31 rows, so every kernel addresses both the same way:
// row `loc` lives at pg[loc >> shift] + (loc mod 2^shift) * rec.
__device__ __forceinline__ void rows_setup(const AttnArgs& a, int r, uint64_t* s_pg) {
  if (a.kv_pt != nullptr) {
    for (int i = threadIdx.x; i < a.kv_pages; i += blockDim.x) s_pg[i] = a.kv_pt[(int64_t)r * a.kv_pages + i];
  } else if (threadIdx.x == 0) {
    s_pg[0] = (uint64_t)(uintptr_t)(a.kv + (int64_t)r * a.rows * a.rec);
  }
}
__device__ __forceinline__ int64_t rows_of(const AttnArgs& a, int r) {
  return a.kv_cap != nullptr ? min(a.rows, (int64_t)a.kv_cap[r]) : a.rows;
}
__device__ __forceinline__ uint8_t* row_addr(const uint64_t* s_pg, int shift, int64_t rec, int32_t loc) {
  return (uint8_t*)(uintptr_t)s_pg[loc >> shift] + (int64_t)(loc & (int32_t)((1u << shift) - 1u)) * rec;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar`; give up after ~1 s or when another warp raised *abort.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile uint32_t* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*abort) return false;
      if (global_ns() - t0 > 1000000000ull) return false;
    }
  }
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 32 partial sums per lane -> lane l holds the warp-wide sum of value l.
__device__ __forceinline__ float reduce32_transposed(float (&v)[32], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int off = 16 >> step;
    const int n = 32 >> step;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

// Combine the split partials of heads [h0, h0 + nh) of request r, in split order, one warp.
// Split weights come from lanes over splits (parallel loads, warp reductions); the partial rows
// are then accumulated with the loads of 4 splits issued together.
template <int DV>
__device__ __forceinline__ void combine_heads(const AttnArgs& a, int r, int h0, int nh, int lane) {
  constexpr int DW = DV / 128;  // float4 per lane per row
  for (int x = 0; x < nh; ++x) {
    const int h = h0 + x;
    float mloc = -INFINITY;
    for (int s2 = lane; s2 < a.S; s2 += 32)
      mloc = fmaxf(mloc, __ldcg(&a.ml[(((int64_t)r * a.S + s2) * a.Hq + h) * 2]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
    const float M = mloc;
    float acc[DW][4];
#pragma unroll
    for (int u = 0; u < DW; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
    float den = 0.f;
    if (M != -INFINITY) {
      for (int c0 = 0; c0 < a.S; c0 += 32) {
        float w = 0.f, lw = 0.f;
        const int s2 = c0 + lane;
        if (s2 < a.S) {
          const int64_t ph = ((int64_t)r * a.S + s2) * a.Hq + h;
          const float ms = __ldcg(&a.ml[ph * 2]);
          w = ms == -INFINITY ? 0.f : exp2f(ms - M);
          lw = w * __ldcg(&a.ml[ph * 2 + 1]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
        den += lw;
        const int ns = min(32, a.S - c0);
        for (int b0 = 0; b0 < ns; b0 += 4) {
          float4 v[4][DW];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (b0 + j < ns) {
              const float4* po = (const float4*)(a.part + (((int64_t)r * a.S + c0 + b0 + j) * a.Hq + h) * DV);
#pragma unroll
              for (int u = 0; u < DW; ++u) v[j][u] = __ldcg(&po[lane + 32 * u]);
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float wj = __shfl_sync(0xffffffffu, w, (b0 + j) & 31);
            if (b0 + j < ns) {
#pragma unroll
              for (int u = 0; u < DW; ++u) {
                acc[u][0] = fmaf(wj, v[j][u].x, acc[u][0]);
                acc[u][1] = fmaf(wj, v[j][u].y, acc[u][1]);
                acc[u][2] = fmaf(wj, v[j][u].z, acc[u][2]);
                acc[u][3] = fmaf(wj, v[j][u].w, acc[u][3]);
              }
            }
          }
        }
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    float4* out = (float4*)(a.out + ((int64_t)(r - a.r0) * a.Hq + h) * DV);
#pragma unroll
    for (int u = 0; u < DW; ++u)
      out[lane + 32 * u] = make_float4(acc[u][0] * inv, acc[u][1] * inv, acc[u][2] * inv, acc[u][3] * inv);
  }
}

// Combine of NH heads at once (up to 32 splits): lane s holds split s's running max and sum for
// every head, so the weights take one round of loads; the partial rows are then read in batches of
// up to four splits for all NH heads together.  Larger split counts use combine_heads.
template <int DV, int NH>
__device__ __forceinline__ void combine_heads_wide(const AttnArgs& a, int r, int h0, int lane) {
  constexpr int DW = DV / 128;
  constexpr int JB = NH * DW >= 8 ? 2 : 4;  // splits per batch of loads, bounded by registers
  float m[NH], l[NH], w[NH], den[NH], acc[NH][DW][4];
  const bool mine = lane < a.S;
#pragma unroll
  for (int x = 0; x < NH; ++x) {
    const int64_t ph = ((int64_t)r * a.S + lane) * a.Hq + h0 + x;
    m[x] = mine ? __ldcg(&a.ml[ph * 2]) : -INFINITY;
    l[x] = mine ? __ldcg(&a.ml[ph * 2 + 1]) : 0.f;
  }
#pragma unroll
  for (int x = 0; x < NH; ++x) {
    float M = m[x];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    w[x] = (M == -INFINITY || m[x] == -INFINITY) ? 0.f : exp2f(m[x] - M);
    float d = w[x] * l[x];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    den[x] = d;
#pragma unroll
    for (int u = 0; u < DW; ++u) acc[x][u][0] = acc[x][u][1] = acc[x][u][2] = acc[x][u][3] = 0.f;
  }
  for (int b0 = 0; b0 < a.S; b0 += JB) {
    float4 v[JB][NH][DW];
#pragma unroll
    for (int j = 0; j < JB; ++j) {
      if (b0 + j < a.S) {
#pragma unroll
        for (int x = 0; x < NH; ++x) {
          const float4* po = (const float4*)(a.part + (((int64_t)r * a.S + b0 + j) * a.Hq + h0 + x) * DV);
#pragma unroll
          for (int u = 0; u < DW; ++u) v[j][x][u] = __ldcg(&po[lane + 32 * u]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < JB; ++j) {
      if (b0 + j < a.S) {
#pragma unroll
        for (int x = 0; x < NH; ++x) {
          const float wj = __shfl_sync(0xffffffffu, w[x], b0 + j);
#pragma unroll
          for (int u = 0; u < DW; ++u) {
            acc[x][u][0] = fmaf(wj, v[j][x][u].x, acc[x][u][0]);
            acc[x][u][1] = fmaf(wj, v[j][x][u].y, acc[x][u][1]);
            acc[x][u][2] = fmaf(wj, v[j][x][u].z, acc[x][u][2]);
            acc[x][u][3] = fmaf(wj, v[j][x][u].w, acc[x][u][3]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int x = 0; x < NH; ++x) {
    const float inv = den[x] > 0.f ? 1.f / den[x] : 0.f;
    float4* out = (float4*)(a.out + ((int64_t)(r - a.r0) * a.Hq + h0 + x) * DV);
#pragma unroll
    for (int u = 0; u < DW; ++u)
      out[lane + 32 * u] =
          make_float4(acc[x][u][0] * inv, acc[x][u][1] * inv, acc[x][u][2] * inv, acc[x][u][3] * inv);
  }
}

template <int DK, int DV, int G, int NW>
struct AttnCfg {
  static constexpr int T = 32 / G;      // tokens per stage
  static constexpr int DKW = DK / 64;   // bf16 pairs per lane of a K row
  static constexpr int DVW = DV / 64;   // bf16 pairs per lane of a V row
  static constexpr int THREADS = (NW + 1) * 32;
  static_assert(G * T == 32, "G must divide 32");
  static_assert(DK % 64 == 0 && DV % 64 == 0, "head dims must be multiples of 64");
};

template <int DK, int DV, int G, int NW>
__global__ void __launch_bounds__(AttnCfg<DK, DV, G, NW>::THREADS) k_attn_cc(AttnArgs a) {
  hs_pdl_enter();
  using C = AttnCfg<DK, DV, G, NW>;
  constexpr int T = C::T, DKW = C::DKW, DVW = C::DVW;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ uint32_t tok_mask[kStages];
  __shared__ uint32_t abort_flag;
  __shared__ uint32_t is_last;
  __shared__ uint64_t s_pg[kMaxSlotPages];

  const int split = blockIdx.x, r = a.r0 + (int)blockIdx.y, grp = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = split * a.chunk;
  const int t1 = min(a.k, t0 + a.chunk);
  const int nst = (t1 - t0 + T - 1) / T;
  const int64_t rec = a.rec;
  const int32_t* locs = a.locs + (int64_t)(r - a.r0) * a.k;
  const int64_t rows_r = rows_of(a, r);

  rows_setup(a, r, s_pg);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1u);
      mbar_init(&empty_bar[s], (uint32_t)NW);
    }
    abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  float m_run[G], l_run[G], o[G][DVW][2];
  const int g = grp * NW + warp;  // KV block of this consumer warp

  if (warp == NW) {
    // ---------------- producer: gather records into the ring ----------------
    if (lane == 0) {
      uint32_t bad = 0u;
      int issued = 0;
      for (int st = 0; st < nst; ++st) {
        const int b = st % kStages;
        if (st >= kStages) {
          if (!mbar_wait_bounded(&empty_bar[b], (uint32_t)((st / kStages - 1) & 1), &abort_flag)) {
            *(volatile uint32_t*)&abort_flag = 1u;
            atomicOr(a.err, (uint32_t)HS_DEVERR_TIMEOUT);
            break;
          }
        }
        uint32_t mask = 0u, nvalid = 0u;
        int32_t lc[T];
#pragma unroll
        for (int j = 0; j < T; ++j) {
          const int idx = t0 + st * T + j;
          int32_t loc = idx < t1 ? locs[idx] : -1;
          if (loc < -1 || (int64_t)loc >= rows_r) {
            bad = 1u;
            loc = -1;
          }
          lc[j] = loc;
          if (loc >= 0) {
            mask |= 1u << j;
            ++nvalid;
          }
        }
        tok_mask[b] = mask;
        mbar_arrive_expect_tx(&full_bar[b], nvalid * (uint32_t)rec);
        uint8_t* dst = smem + (size_t)b * T * rec;
#pragma unroll
        for (int j = 0; j < T; ++j) {
          if (lc[j] >= 0)
            bulk_g2s(dst + (size_t)j * rec, row_addr(s_pg, a.kv_shift, rec, lc[j]), (uint32_t)rec, &full_bar[b]);
        }
        issued = st + 1;
      }
      if (bad) atomicOr(a.err, (uint32_t)HS_DEVERR_LOC);
      if (abort_flag) {
        // let copies already issued land before the CTA can retire
        for (int st = max(0, issued - kStages); st < issued; ++st) {
          volatile uint32_t never = 0u;
          mbar_wait_bounded(&full_bar[st % kStages], (uint32_t)((st / kStages) & 1), &never);
        }
      }
    }
  } else {
    // ---------------- consumers: one KV block, G query heads ----------------
    float qf[G][DKW][2];
    const int hbase = g * G;
#pragma unroll
    for (int x = 0; x < G; ++x) {
      const uint32_t* qw = (const uint32_t*)(a.q + ((int64_t)(r - a.r0) * a.Hq + hbase + x) * DK);
#pragma unroll
      for (int u = 0; u < DKW; ++u) {
        const uint32_t w = qw[lane + 32 * u];
        qf[x][u][0] = bf_lo(w) * a.qscale;
        qf[x][u][1] = bf_hi(w) * a.qscale;
      }
      m_run[x] = -INFINITY;
      l_run[x] = 0.f;
#pragma unroll
      for (int u = 0; u < DVW; ++u) o[x][u][0] = o[x][u][1] = 0.f;
    }
    const int64_t koff = (int64_t)g * a.kstride;
    const int64_t voff = koff + a.vdelta;
    const int my_x = lane / T, my_j = lane % T;
    for (int st = 0; st < nst; ++st) {
      const int b = st % kStages;
      if (!mbar_wait_bounded(&full_bar[b], (uint32_t)((st / kStages) & 1), &abort_flag)) {
        *(volatile uint32_t*)&abort_flag = 1u;
        atomicOr(a.err, (uint32_t)HS_DEVERR_TIMEOUT);
        break;
      }
      const uint32_t mask = tok_mask[b];
      const uint8_t* stage = smem + (size_t)b * T * rec;
      float s[32];
#pragma unroll
      for (int j = 0; j < T; ++j) {
        const uint32_t* kw = (const uint32_t*)(stage + j * rec + koff);
        uint32_t w[DKW];
#pragma unroll
        for (int u = 0; u < DKW; ++u) w[u] = kw[lane + 32 * u];
#pragma unroll
        for (int x = 0; x < G; ++x) {
          float acc = 0.f;
#pragma unroll
          for (int u = 0; u < DKW; ++u) {
            acc = fmaf(qf[x][u][0], bf_lo(w[u]), acc);
            acc = fmaf(qf[x][u][1], bf_hi(w[u]), acc);
          }
          s[x * T + j] = acc;
        }
      }
      float logit = reduce32_transposed(s, lane);
      if (!((mask >> my_j) & 1u)) logit = -INFINITY;
      float smax = logit;
#pragma unroll
      for (int off = T / 2; off > 0; off >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, off));
      float mnew_mine = fmaxf(m_run[my_x], smax);
      const float p = mnew_mine == -INFINITY ? 0.f : exp2f(logit - mnew_mine);
      float psum = p;
#pragma unroll
      for (int off = T / 2; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
#pragma unroll
      for (int x = 0; x < G; ++x) {
        const float mnew = __shfl_sync(0xffffffffu, mnew_mine, x * T);
        const float ps = __shfl_sync(0xffffffffu, psum, x * T);
        const float alpha = mnew == -INFINITY ? 1.f : exp2f(m_run[x] - mnew);
        m_run[x] = mnew;
        l_run[x] = l_run[x] * alpha + ps;
#pragma unroll
        for (int u = 0; u < DVW; ++u) {
          o[x][u][0] *= alpha;
          o[x][u][1] *= alpha;
        }
      }
#pragma unroll
      for (int j = 0; j < T; ++j) {
        if (!((mask >> j) & 1u)) continue;
        const uint32_t* vw = (const uint32_t*)(stage + j * rec + voff);
        uint32_t w[DVW];
#pragma unroll
        for (int u = 0; u < DVW; ++u) w[u] = vw[lane + 32 * u];
#pragma unroll
        for (int x = 0; x < G; ++x) {
          const float pj = __shfl_sync(0xffffffffu, p, x * T + j);
#pragma unroll
          for (int u = 0; u < DVW; ++u) {
            o[x][u][0] = fmaf(pj, bf_lo(w[u]), o[x][u][0]);
            o[x][u][1] = fmaf(pj, bf_hi(w[u]), o[x][u][1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[b]);
    }
    if (!abort_flag) {
      // split partial: unnormalised o, running max (base 2) and sum
#pragma unroll
      for (int x = 0; x < G; ++x) {
        const int64_t ph = ((int64_t)r * a.S + split) * a.Hq + hbase + x;
        float2* po = (float2*)(a.part + ph * DV);
#pragma unroll
        for (int u = 0; u < DVW; ++u) po[lane + 32 * u] = make_float2(o[x][u][0], o[x][u][1]);
        if (lane == 0) {
          a.ml[ph * 2 + 0] = m_run[x];
          a.ml[ph * 2 + 1] = l_run[x];
        }
      }
    }
  }
  __threadfence();  // every writer publishes its partials before the ticket
  __syncthreads();
  if (abort_flag) return;
  if (threadIdx.x == 0) {
    const uint32_t t = atomicAdd(&a.ticket[(int64_t)r * (a.groups + 1) + grp], 1u);
    is_last = (t == (uint32_t)(a.S - 1)) ? 1u : 0u;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  if (warp < NW) {
    if (a.S <= 32)
      combine_heads_wide<DV, G>(a, r, g * G, lane);
    else
      combine_heads<DV>(a, r, g * G, G, lane);
  }
  if (threadIdx.x == 0) a.ticket[(int64_t)r * (a.groups + 1) + grp] = 0u;
}

// ---- tensor-core variant for GQA records ----------------------------------------
//
// A KV block (one KV head) serves G <= 8 query heads.  Per 16-token tile a consumer warp runs the
// transposed products, so that tokens and value dims fill the MMA's 16-row side and the few heads
// sit on its 8-column side:
//   S^T[16 tokens x 8] = K[16 x 128] . Q^T[128 x 8]
//   O^T[128 x 8]      += V^T[128 x 16] . P^T[16 x 8]
// on mma.sync m16n8k16 (bf16 in, fp32 accumulate): 8 + 8 MMAs per tile.  K and V^T fragments come
// from the staged records with ldmatrix (plain for K, transposed for V); each staged record is
// padded by 16 bytes so the eight rows of every 8x8 matrix fall in distinct banks.  P is carried
// as a bf16 high part plus a bf16 remainder (~16 mantissa bits): for G <= 4 the remainders ride in
// columns G..2G-1 of the same MMA (Q^T repeats its heads there, so those columns see the same
// scores), for G = 8 they take a second MMA.  P^T's fragments come from the score fragments by an
// in-register 8x8 transpose (movmatrix).

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

constexpr int kMmaTile = 16;  // tokens per stage

// ---- GQA, one CTA per (request, KV head, split) ------------------------------------------
//
// Each CTA gathers one KV head's 512-byte K|V slice of every selected record (128 CTAs for 16
// requests x 8 KV heads; a split of the top-k list only when requests x KV heads leave SMs idle).
// Its eight consumer warps take the 16-token stages round robin (warp w: stages w, w + 8, ...),
// each through its own kGqaStages buffers, and only compute.  Each consumer has a producer warp
// that requests its stages in order, one 512-byte bulk copy per token (lanes 0-15), on the
// buffer's full mbarrier, and waits for the consumer to hand the buffer back through its empty
// mbarrier (all waits bounded).  Issuing a bulk copy costs the issuing warp tens of nanoseconds, so
// the copies are spread over eight warps and kept out of the consumers' instruction streams.  Rows
// of padding entries are zero-filled instead, so the math needs no masking of V.  The per-tile
// math is the transposed MMA form described above.  At the end the consumers' (max, sum, O) are
// merged through shared memory in warp order, so the reduction order is fixed by the top-k order
// alone; with one split the CTA writes the final output, otherwise a partial that the last split of
// the (request, KV head) combines.
//
// FETCH (misses copied inside the attention): the resolve only decided, and left {host address,
// slot} for every miss.  A producer requests a pending row of its stage straight from the mapped host
// history by bulk copy, like the resident rows from HBM, on the same full mbarrier, so the host-link
// transfer overlaps the HBM gather and the math; it leaves the row's hot-buffer address beside the
// stage, and the consumer, once the stage has landed, writes the row back to that slot (each CTA its
// own KV head's slice).  The last CTA of a request to finish clears the request's pending flag.
constexpr int kGqaWarps = 8;           // consumer warps
constexpr int kGqaProducers = 8;       // producer warps, one per consumer
constexpr int kGqaStages = 3;          // buffers per consumer warp
constexpr int kGqaRow = 512 + 16;      // staged slice (K 256 B | V 256 B) + 16 B pad for ldmatrix

__device__ __forceinline__ float fast_exp2(float x) {  // 2^x; -inf gives +0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The dependency on the resolve just before: by default the whole resolve grid (programmatic
// dependent launch).  When the launch directly follows the whole-batch resolve of its layer
// (a.res_count set), a CTA waits only for the resolve CTAs of its own request: every resolve CTA
// counts itself finished after its writes (release), the resolve counts its launch for each request
// before any CTA of this kernel may start, and thread 0 waits until the finished count reaches the
// request's CTAs times its launches (acquire, bounded).  The resolve's CTAs are all resident before
// this kernel starts, so the wait cannot block them.  The bulk copies then read through the async
// proxy what the resolve wrote through the generic one, hence the proxy fence.
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void attn_enter(const AttnArgs& a, int r, uint32_t* err) {
  if (a.res_count == nullptr) {
    hs_pdl_enter();
    return;
  }
  if (threadIdx.x == 0) {
    const uint32_t target = (uint32_t)a.res_cs * ld_acquire_u32(&a.res_count[2 * r]);
    uint64_t t0 = 0;
    for (uint32_t it = 0; ld_acquire_u32(&a.res_count[2 * r + 1]) < target; ++it) {
      __nanosleep(64);
      if ((it & 63u) == 0u) {
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (it == 0u) {
          t0 = t;
        } else if (t - t0 > 1000000000ull) {
          atomicOr(err, (uint32_t)HS_DEVERR_TIMEOUT);
          break;
        }
      }
    }
  }
  __syncthreads();
  asm volatile("fence.proxy.async.global;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int G, bool FETCH>
__global__ void __launch_bounds__((kGqaWarps + kGqaProducers) * 32, 1) k_attn_gqa(AttnArgs a) {
  attn_enter(a, a.r0 + (int)blockIdx.y, a.err);
  constexpr int T = kMmaTile, D = 128, NW = kGqaWarps, NS = kGqaStages, RW = kGqaRow;
  constexpr bool kStuff = G <= 4;        // P remainders ride in columns G..2G-1 of the same MMA
  constexpr int kCols = kStuff ? 2 * G : G;
  constexpr int DP = D + 4;              // row stride of the merge area (conflict-free stores)
  static_assert(G == 1 || G == 2 || G == 4 || G == 8, "1, 2, 4 or 8 query heads per KV head");
  static_assert(NW * kCols * DP * 4 <= NW * NS * T * RW, "merge area fits in the buffers");
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[NW][NS];
  __shared__ __align__(8) uint64_t empty[NW][NS];
  __shared__ float s_m[NW][8], s_l[NW][8], s_fin[8][2];
  __shared__ uint32_t s_mask[NW][NS];  // valid tokens of the stage in each buffer (bit j: token j)
  // FETCH: the stage's tokens copied from the host history (bit j: token j) and the hot-buffer
  // address of each one's slice, which the consumer writes the landed row back to
  __shared__ uint32_t s_pmask[FETCH ? NW : 1][NS];
  __shared__ uint64_t s_pdst[FETCH ? NW : 1][NS][FETCH ? kMmaTile : 1];
  __shared__ uint32_t is_last, abort_flag, use_pend;
  __shared__ uint64_t s_pg[kMaxSlotPages];

  const int split = blockIdx.x, r = a.r0 + (int)blockIdx.y, g = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grow = lane >> 2, tig = lane & 3;
  const int t0 = split * a.chunk;
  const int n = min(a.k, t0 + a.chunk) - t0;
  const int nst = (n + T - 1) / T;
  const int64_t rec = a.rec;
  if (threadIdx.x == 0) {
    use_pend = (FETCH && a.pend != nullptr && a.pend_live[r] != 0u) ? 1u : 0u;
    for (int w = 0; w < NW; ++w)
      for (int b = 0; b < NS; ++b) {
        mbar_init(&full[w][b], 1u);
        mbar_init(&empty[w][b], 1u);
      }
    abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool pend_on = FETCH && use_pend != 0u;

  // consumer state: columns c0, c1 of the 8-wide MMA side (head c % G; high part, remainder or
  // zero padding, see above), running max / sum per column, O^T accumulators
  const int c0 = 2 * tig, c1 = 2 * tig + 1;
  float ot[8][4];
#pragma unroll
  for (int m = 0; m < 8; ++m) ot[m][0] = ot[m][1] = ot[m][2] = ot[m][3] = 0.f;
  float mr0 = -INFINITY, mr1 = -INFINITY, lp0 = 0.f, lp1 = 0.f;

  if (warp >= NW) {
    // ---------------- producers: producer pw fills consumer pw's buffers, stage by stage ----------------
    const int w = warp - NW;
    const int ni = w < nst ? (nst - w + NW - 1) / NW : 0;
    const int64_t goff = (int64_t)g * a.kstride;  // KV head g's slice of a row
    const int rows_r = (int)rows_of(a, r);
    bool ok = true;
    int issued = 0;
    // the slot (and, FETCH, the host address of a pending record, 0 if none) of token `lane` of
    // stage i, read from global memory two stages before use; invalid slots become padding
    const int32_t* locs_r = a.locs + (int64_t)(r - a.r0) * a.k + t0;
    const hs_pending* pend_r = pend_on ? a.pend + (int64_t)r * a.k + t0 : nullptr;
    auto load_raw = [&](int i, int32_t& l, uint64_t& q) {
      const int x = (w + NW * i) * T + lane;
      const bool in = i < ni && lane < T && x < n;
      l = in ? locs_r[x] : -1;
      q = (FETCH && in && pend_on) ? pend_r[x].src : 0ull;
    };
    auto stage_info = [&](int32_t l, uint64_t q, int32_t& loc, uint64_t& pp, uint32_t& vmask, uint32_t& pmask) {
      if (l < -1 || l >= rows_r) {
        atomicOr(a.err, (uint32_t)HS_DEVERR_LOC);
        l = -1;
      }
      loc = l;
      pp = (FETCH && l >= 0) ? q : 0ull;
      vmask = __ballot_sync(0xffffffffu, lane < T && loc >= 0);
      pmask = FETCH ? __ballot_sync(0xffffffffu, lane < T && pp != 0ull) : 0u;
    };
    // the first three stages' slots are requested before the page row, so the loads overlap
    int32_t raw_l0, raw_l1, raw_l2;
    uint64_t raw_q0, raw_q1, raw_q2;
    load_raw(0, raw_l0, raw_q0);
    load_raw(1, raw_l1, raw_q1);
    load_raw(2, raw_l2, raw_q2);
    {  // the page row, filled by the producers for the producers
      const int pt = (int)threadIdx.x - NW * 32;
      if (a.kv_pt != nullptr) {
        if (pt < a.kv_pages) s_pg[pt] = a.kv_pt[(int64_t)r * a.kv_pages + pt];
      } else if (pt == 0) {
        s_pg[0] = (uint64_t)(uintptr_t)(a.kv + (int64_t)r * a.rows * rec);
      }
      asm volatile("bar.sync 2, %0;" ::"n"(kGqaProducers * 32) : "memory");
    }
    int32_t loc;
    uint64_t pp;
    uint32_t vmask, pmask;
    stage_info(raw_l0, raw_q0, loc, pp, vmask, pmask);
    raw_l0 = raw_l2;
    raw_q0 = raw_q2;
    for (int i = 0; i < ni; ++i) {
      const int b = i % NS;
      if (i >= NS) {
        bool okw = true;
        if (lane == 0) okw = mbar_wait_bounded(&empty[w][b], (uint32_t)((i / NS - 1) & 1), &abort_flag);
        if (__shfl_sync(0xffffffffu, okw ? 1 : 0, 0) == 0) {
          ok = false;
          break;
        }
      }
      uint8_t* dst = smem + ((size_t)(w * NS + b) * T) * RW;
      if (lane == 0) s_mask[w][b] = vmask;
      if (vmask != 0xffffu) {
        // padding rows (and the tail past the chunk) read as zeros
        for (uint32_t zm = ~vmask & 0xffffu; zm != 0u; zm &= zm - 1u)
          *(uint4*)(dst + (__ffs(zm) - 1) * RW + lane * 16) = make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();
      }
      if (FETCH) {
        // a pending row comes straight from the host history, by bulk copy like the resident rows;
        // the consumer writes it back to its hot-buffer slot once the stage has landed
        if (lane == 0) s_pmask[w][b] = pmask;
        if (pp != 0ull) s_pdst[w][b][lane] = (uint64_t)(uintptr_t)(row_addr(s_pg, a.kv_shift, rec, loc) + goff);
        __syncwarp();
      }
      if (lane == 0) mbar_arrive_expect_tx(&full[w][b], (uint32_t)__popc(vmask) * 512u);
      __syncwarp();
      if (loc >= 0) {
        const uint8_t* src = (FETCH && pp != 0ull) ? (const uint8_t*)(uintptr_t)pp + goff
                                                   : row_addr(s_pg, a.kv_shift, rec, loc) + goff;
        bulk_g2s(dst + lane * RW, src, 512u, &full[w][b]);
      }
      int32_t loc2;
      uint64_t pp2;
      uint32_t vmask2, pmask2;
      stage_info(raw_l1, raw_q1, loc2, pp2, vmask2, pmask2);
      raw_l1 = raw_l0;
      raw_q1 = raw_q0;
      load_raw(i + 3, raw_l0, raw_q0);
      loc = loc2;
      pp = pp2;
      vmask = vmask2;
      pmask = pmask2;
      issued = i + 1;
    }
    if (!ok && lane == 0) {
      *(volatile uint32_t*)&abort_flag = 1u;
      atomicOr(a.err, (uint32_t)HS_DEVERR_TIMEOUT);
      // let this warp's copies already requested (the last use of each buffer) land before retiring
      volatile uint32_t never = 0u;
      for (int i = max(0, issued - NS); i < issued; ++i)
        mbar_wait_bounded(&full[w][i % NS], (uint32_t)((i / NS) & 1), &never);
    }
  } else {
    // ---------------- consumers: warp w takes stages w, w + NW, ... ----------------
    const int ni = warp < nst ? (nst - warp + NW - 1) / NW : 0;
    const uint32_t ring_u = smem_u32(smem) + (uint32_t)(warp * NS * T * RW);
    uint32_t qb[8][2];
    {
      const bool qon = grow < kCols;
      const uint32_t* qw =
          (const uint32_t*)(a.q + ((int64_t)(r - a.r0) * a.Hq + (int64_t)g * G + (grow % G)) * D);
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2) {
        qb[s2][0] = qon ? qw[s2 * 8 + tig] : 0u;
        qb[s2][1] = qon ? qw[s2 * 8 + 4 + tig] : 0u;
      }
    }
    const uint32_t k_lane = (uint32_t)((lane & 15) * RW + (lane >> 4) * 16);
    const uint32_t v_lane = (uint32_t)(((lane & 7) + ((lane >> 4) << 3)) * RW + 256 + ((lane >> 3) & 1) * 16);
    for (int i = 0; i < ni; ++i) {
      const int b = i % NS;
      if (!mbar_wait_bounded(&full[warp][b], (uint32_t)((i / NS) & 1), &abort_flag)) {
        *(volatile uint32_t*)&abort_flag = 1u;
        atomicOr(a.err, (uint32_t)HS_DEVERR_TIMEOUT);
        break;
      }
      const uint32_t mask = s_mask[warp][b];
      const uint32_t base = ring_u + (uint32_t)(b * T * RW);
      if (FETCH) {
        // the stage's rows fetched from the host go back to their hot-buffer slots (each CTA its KV
        // head's slice): 512 coalesced bytes a row
        const uint8_t* stage_rows = smem + (size_t)(warp * NS + b) * T * RW;
        for (uint32_t pm = s_pmask[warp][b]; pm != 0u; pm &= pm - 1u) {
          const int j = __ffs(pm) - 1;
          *((uint4*)(uintptr_t)s_pdst[warp][b][j] + lane) = *((const uint4*)(stage_rows + j * RW) + lane);
        }
      }
      // S^T = K Q^T in four independent MMA chains (k-steps s, s + 4)
      float sacc[4][4];
#pragma unroll
      for (int c = 0; c < 4; ++c) sacc[c][0] = sacc[c][1] = sacc[c][2] = sacc[c][3] = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2) {
        uint32_t x0, x1, x2, x3;
        ldsm_x4(base + k_lane + s2 * 32, x0, x1, x2, x3);
        mma_bf16(sacc[s2 & 3], x0, x1, x2, x3, qb[s2][0], qb[s2][1]);
      }
      float sv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) sv[e] = (sacc[0][e] + sacc[1][e]) + (sacc[2][e] + sacc[3][e]);
      const bool va = ((mask >> grow) & 1u) != 0u, vb = ((mask >> (grow + 8)) & 1u) != 0u;
      const float x00 = va ? sv[0] * a.qscale : -INFINITY;
      const float x01 = va ? sv[1] * a.qscale : -INFINITY;
      const float x10 = vb ? sv[2] * a.qscale : -INFINITY;
      const float x11 = vb ? sv[3] * a.qscale : -INFINITY;
      float mx0 = fmaxf(x00, x10), mx1 = fmaxf(x01, x11);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(mr0, mx0), mn1 = fmaxf(mr1, mx1);
      // a column with no valid token yet keeps max -inf: its weights are zero, its scale one
      const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
      const float p00 = fast_exp2(x00 - ms0), p10 = fast_exp2(x10 - ms0);
      const float p01 = fast_exp2(x01 - ms1), p11 = fast_exp2(x11 - ms1);
      if (__any_sync(0xffffffffu, mn0 != mr0 || mn1 != mr1)) {
        const float al0 = fast_exp2(mr0 - ms0), al1 = fast_exp2(mr1 - ms1);
        lp0 *= al0;
        lp1 *= al1;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          ot[m][0] *= al0;
          ot[m][1] *= al1;
          ot[m][2] *= al0;
          ot[m][3] *= al1;
        }
      }
      mr0 = mn0;
      mr1 = mn1;
      lp0 += p00 + p10;
      lp1 += p01 + p11;
      uint32_t bh0, bh1, bl0 = 0u, bl1 = 0u;
      {
        const float h00 = __bfloat162float(__float2bfloat16_rn(p00)), h01 = __bfloat162float(__float2bfloat16_rn(p01));
        const float h10 = __bfloat162float(__float2bfloat16_rn(p10)), h11 = __bfloat162float(__float2bfloat16_rn(p11));
        if (kStuff) {
          const float y00 = c0 < G ? h00 : (c0 < 2 * G ? p00 - h00 : 0.f);
          const float y01 = c1 < G ? h01 : (c1 < 2 * G ? p01 - h01 : 0.f);
          const float y10 = c0 < G ? h10 : (c0 < 2 * G ? p10 - h10 : 0.f);
          const float y11 = c1 < G ? h11 : (c1 < 2 * G ? p11 - h11 : 0.f);
          bh0 = movm_t(pack_bf16(y00, y01));
          bh1 = movm_t(pack_bf16(y10, y11));
        } else {
          bh0 = movm_t(pack_bf16(h00, h01));
          bh1 = movm_t(pack_bf16(h10, h11));
          bl0 = movm_t(pack_bf16(p00 - h00, p01 - h01));
          bl1 = movm_t(pack_bf16(p10 - h10, p11 - h11));
        }
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        uint32_t x0, x1, x2, x3;
        ldsm_x4_t(base + v_lane + m * 32, x0, x1, x2, x3);
        mma_bf16(ot[m], x0, x1, x2, x3, bh0, bh1);
        if (!kStuff) mma_bf16(ot[m], x0, x1, x2, x3, bl0, bl1);
      }
      __syncwarp();  // every lane is done with buffer b before it is handed back
      if (lane == 0) mbar_arrive(&empty[warp][b]);
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lp0 += __shfl_xor_sync(0xffffffffu, lp0, o);
      lp1 += __shfl_xor_sync(0xffffffffu, lp1, o);
    }
    if (grow == 0) {
      if (c0 < G) {
        s_m[warp][c0] = mr0;
        s_l[warp][c0] = lp0;
      }
      if (c1 < G) {
        s_m[warp][c1] = mr1;
        s_l[warp][c1] = lp1;
      }
    }
  }
  __syncthreads();  // (A) stats in place, no buffer read any more
  if (abort_flag) return;
  if (pend_on && threadIdx.x == 0) {
    // every CTA of the request has written its slices of the fetched rows back: the list is done
    uint32_t* cnt = &a.ticket[(int64_t)r * (a.groups + 1) + a.groups];
    const uint32_t t = atomicAdd(cnt, 1u);
    if (t == (uint32_t)(a.S * a.groups - 1)) {
      *cnt = 0u;
      a.pend_live[r] = 0u;
    }
  }
  // merge: each consumer column scaled by exp2(m_w - M) into red[w][c][.]; the producer warp's
  // lanes h < G compute the per-head max M and normaliser
  float* red = (float*)smem;
  if (warp < NW) {
    float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      M0 = fmaxf(M0, s_m[w][c0 % G]);
      M1 = fmaxf(M1, s_m[w][c1 % G]);
    }
    const float w0 = mr0 == -INFINITY ? 0.f : exp2f(mr0 - M0);
    const float w1 = mr1 == -INFINITY ? 0.f : exp2f(mr1 - M1);
    if (c0 < kCols) {
      float* rw = red + ((size_t)warp * kCols + c0) * DP;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        rw[16 * m + grow] = ot[m][0] * w0;
        rw[16 * m + grow + 8] = ot[m][2] * w0;
      }
    }
    if (c1 < kCols) {
      float* rw = red + ((size_t)warp * kCols + c1) * DP;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        rw[16 * m + grow] = ot[m][1] * w1;
        rw[16 * m + grow + 8] = ot[m][3] * w1;
      }
    }
  } else if (warp == NW && lane < G) {
    float M = -INFINITY, den = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, s_m[w][lane]);
#pragma unroll
    for (int w = 0; w < NW; ++w) den += s_m[w][lane] == -INFINITY ? 0.f : s_l[w][lane] * exp2f(s_m[w][lane] - M);
    s_fin[lane][0] = M;
    s_fin[lane][1] = den;
  }
  __syncthreads();  // (B)
  // sum over warps in warp order (high part, then remainder); one thread per (head, value)
  for (int e = (int)threadIdx.x; e < G * D; e += (NW + kGqaProducers) * 32) {
    const int h = e / D, d = e % D;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      acc += red[((size_t)w * kCols + h) * DP + d];
      if (kStuff) acc += red[((size_t)w * kCols + h + G) * DP + d];
    }
    const float den = s_fin[h][1];
    const int hq = g * G + h;
    if (a.S == 1) {
      a.out[((int64_t)(r - a.r0) * a.Hq + hq) * D + d] = den > 0.f ? acc / den : 0.f;
    } else {
      const int64_t ph = ((int64_t)r * a.S + split) * a.Hq + hq;
      a.part[ph * D + d] = acc;
      if (d == 0) *(float2*)(a.ml + ph * 2) = make_float2(s_fin[h][0], den);
    }
  }
  if (a.S == 1) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t t = atomicAdd(&a.ticket[(int64_t)r * (a.groups + 1) + g], 1u);
    is_last = (t == (uint32_t)(a.S - 1)) ? 1u : 0u;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  if (warp == 0) {
    if (a.S <= 32)
      combine_heads_wide<D, G>(a, r, g * G, lane);
    else
      combine_heads<D>(a, r, g * G, G, lane);
  }
  if (threadIdx.x == 0) a.ticket[(int64_t)r * (a.groups + 1) + g] = 0u;
}

constexpr int kMlaHeads = 64;  // query heads of the shared-latent tensor-core kernel


// Split partials of the tensor-core shared-latent kernel, merged in split order: one warp per
// (request, head, 128-dim quarter of the value), lane = 4 consecutive dims.  Every split's partial row
// is requested first, then the splits' maxima and sums, so the two round trips to memory overlap
// rather than follow one another.  The same arithmetic as combine_heads_wide, so the result is
// identical.
__global__ void __launch_bounds__(256, 2) k_combine_wide(AttnArgs a) {
  HS_PHASE(hs_phase_attn, 57, threadIdx.x == 0);  // combine CTA resident
  hs_pdl_enter();
  HS_PHASE(hs_phase_attn, 58, threadIdx.x == 0);  // the attention grid is complete
  constexpr int DV = 512, JB = 24;  // splits requested at once (one round trip up to 24 splits)
  const int r = a.r0 + (int)blockIdx.x;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = (int)blockIdx.y * 2 + (w >> 2), c = w & 3;
  if (h >= a.Hq) return;
  const float4* p = (const float4*)(a.part + ((int64_t)r * a.S * a.Hq + h) * DV) + 32 * c + lane;
  const int64_t step = (int64_t)a.Hq * (DV / 4);  // float4s from one split's partial to the next
  float4 v[JB];
#pragma unroll
  for (int j = 0; j < JB; ++j)
    if (j < a.S) v[j] = __ldcg(p + j * step);
  const bool mine = lane < a.S;  // lane j holds split j's max and sum (S <= 32)
  const int64_t phl = ((int64_t)r * a.S + lane) * a.Hq + h;
  const float m = mine ? __ldcg(&a.ml[phl * 2]) : -INFINITY;
  const float l = mine ? __ldcg(&a.ml[phl * 2 + 1]) : 0.f;
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float wt = (M == -INFINITY || m == -INFINITY) ? 0.f : exp2f(m - M);
  float den = wt * l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int b0 = 0; b0 < a.S; b0 += JB) {
    if (b0 > 0) {
#pragma unroll
      for (int j = 0; j < JB; ++j)
        if (b0 + j < a.S) v[j] = __ldcg(p + (b0 + j) * step);
    }
#pragma unroll
    for (int j = 0; j < JB; ++j) {
      if (b0 + j < a.S) {
        const float wj = __shfl_sync(0xffffffffu, wt, b0 + j);
        acc.x = fmaf(wj, v[j].x, acc.x);
        acc.y = fmaf(wj, v[j].y, acc.y);
        acc.z = fmaf(wj, v[j].z, acc.z);
        acc.w = fmaf(wj, v[j].w, acc.w);
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  ((float4*)(a.out + ((int64_t)(r - a.r0) * a.Hq + h) * DV))[32 * c + lane] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  HS_PHASE(hs_phase_attn, 59, threadIdx.x == 0);  // this CTA's rows written
}

// ---- shared-latent records on tcgen05 tensor cores (64 heads), pipelined over tiles --------
//
// One CTA per (request, split of the top-k list); a split is walked in tiles of up to 128 tokens
// (the last one ragged: its missing rows are zero-filled and get zero weight).  Per tile, with the
// tokens on the MMA's 128-row side and the 64 heads on its N side:
//   S^T[128 x 64]  = K[128 x 576] . Q^T      36 tcgen05.mma (K = 16 each) into a TMEM S buffer
//   O^T[512 x 64] += V^T[512 x 128] . P^T    4 row tiles x 8 k-steps into TMEM columns 128-383
// Q (all 576 dims of the 64 heads, 72 KB, loaded once by TMA) stays in shared memory for the whole
// split.  The records stream through a ring of four 32 KB slots, each holding two 64-dim blocks of a
// tile (128 rows x 128 B per block) in the 128-byte swizzled layout the MMA reads.  Six producer
// warps fill a slot with 16-byte cp.async copies straight into that layout: one warp instruction
// moves four whole 128-byte lines (rows 4q..4q+3, lane -> row 4q + lane / 8, chunk lane % 8, stored at
// chunk (lane % 8) XOR (row % 8)), so the loads are fully coalesced.  In a split of several tiles every
// tile is gathered twice: its nine blocks for the scores (five slot loads: dims 512-575 alone, then
// 0-127, ..., 384-511), then its eight value blocks for the value product (four slot loads), which the
// first pass has just brought into L2.  The load order is
//   K(0), K(1), V(0), K(2), V(1), ..., K(n-1), V(n-2), V(n-1),
// and one thread of warp 8 consumes the loads in that order, issuing S(0), S(1), PV(0), S(2), PV(1),
// ..., so the scores of tile i+1 are computed while the softmax of tile i runs.  (Alternating the
// slot loads of K(i+1) and V(i) measured slower: the value product of tile i then waits for its
// softmax while holding slots, and its products arrive one 128-row tile at a time.)  A value
// product takes two 128-row tiles of O^T at a time and interleaves their k-steps, so consecutive
// products accumulate into different TMEM columns (measured: 90 instead of 125 cycles a product).
// A split of one tile loads only K(0): the slot of dims 512-575 is released after the scores, the
// four slots of dims 0-511 stay in place for the value product.
// Why this shape (measured on this GPU, per SM): a tcgen05.mma costs its issuing thread 51-75 cycles
// whatever its size up to N = 128, so 128-token tiles (68 products per 128 tokens) beat 64-token tiles
// with M = 64 products (104); in a split of several tiles, holding a tile's value blocks (128 KB beside
// Q) from its score pass to its value pass would stall the next tile's loads; TMA tile::gather4 builds the same
// layout but completes only about 60 of its 512-byte gathers per microsecond (32 GB/s), while 16-byte
// cp.async reaches about 42 GB/s from HBM and 50 GB/s from L2; a ring with one in-order consumer
// never waits on a slot two loads ahead (two consumers of one ring can, and an mbarrier parity test
// then passes a phase early).
// Roles: warps 9-14 produce (each lane keeps the record addresses of its rows of a tile in registers;
// the first tile's slot indices are requested before the setup barrier, each later tile's a tile
// ahead); warp 8 allocates TMEM and one of its threads issues the MMAs, releasing each ring slot by
// a commit once its products are done; the partial is stored as the last tile's value product
// completes each 128 rows of it; warps 0-7 run the softmax as two warpgroups, warpgroup g on heads 32g..32g+31, each thread on one
// token (= TMEM lane).  S alternates between two TMEM buffers (columns 0-63, 64-127).  The running
// max of a head is raised only when a score exceeds it by more than 2^8 (softmax is shift-invariant;
// weights stay <= 256, exact in bf16's range), and only then is its O^T column rescaled in TMEM.
// Weights are rounded to bf16 for the MMA and the normaliser sums the same rounded weights.  Partials
// (O, max, sum) per split are combined by k_combine_wide in split order.  Every wait is bounded; a
// CTA that gives up writes no partial.
constexpr int kUTok = 128, kUHeads = 64, kUDim = 576;
constexpr int kUQ = kUHeads * kUDim * 2;   // 73728 B: Q, nine 64-dim blocks of 64 heads x 128 B
constexpr int kUP = kUTok * kUHeads * 2;   // 16384 B: the weights P of one tile
constexpr int kUBlk = kUTok * 128;         // 16384 B: one 64-dim block of a tile
constexpr int kUSlot = 2 * kUBlk;          // a ring slot holds two blocks
constexpr int kURing = 4;                  // ring slots
constexpr int kUWarpMma = 8, kUWarpProd = 9, kUProd = 6;  // MMA warp, first producer warp, producers
constexpr int kURowsPerLane = (32 + kUProd - 1) / kUProd;  // rows of a tile per producer lane
constexpr int kUThreads = (kUWarpProd + kUProd) * 32;
constexpr int kUTmemO = 128;               // first TMEM column of O^T (after the two S buffers)
constexpr float kULazy = 8.f;              // log2 headroom before the max is raised
constexpr size_t kUSmem = (size_t)kUQ + kUP + (size_t)kURing * kUSlot + 1024;  // + 1 KB alignment

// one lane of the (fully active) warp
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// 16-byte cp.async; src_bytes = 0 writes zeros (nothing is read)
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// one arrival on *bar once every cp.async this thread issued before has landed
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint64_t umma_sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout = 0) {
  // start address, leading / stride byte offsets (16-byte units), descriptor version 1, layout type
  // (0: no swizzle; 2: 128-byte swizzle, atoms 1024-byte aligned so the base offset is 0)
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)layout << 61);
}
// TMA load of one box of a 2-D tensor map at element coordinates (x, y) into shared memory at dst
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ uint32_t umma_idesc_bf16(int M, int N, int a_mn, int b_mn) {
  // fp32 accumulator, bf16 A and B, operand majors, N / 8, M / 16
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
               "l"(a), "l"(b), "r"(id), "r"(acc)
               : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 32 consecutive TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t x[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]),
        "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]), "=r"(x[15]),
        "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), "=r"(x[21]), "=r"(x[22]), "=r"(x[23]),
        "=r"(x[24]), "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(x[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
      "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
      "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
      "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
      "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// barrier of one softmax warpgroup (ids 1 and 2; 0 is __syncthreads)
__device__ __forceinline__ void wg_sync(int g) { asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory"); }

// 32 partial maxima per lane -> lane l holds the warp-wide max of value l (transposed butterfly)
__device__ __forceinline__ float reduce32_max_transposed(float (&v)[32], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int off = 16 >> step;
    const int n = 32 >> step;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, off));
    }
  }
  return v[0];
}

// bounded wait of a whole warp: lane 0 waits, the result is the warp's
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort) {
  bool w = true;
  if ((threadIdx.x & 31) == 0) w = mbar_wait_bounded(bar, parity, abort);
  return __shfl_sync(0xffffffffu, w ? 1 : 0, 0) != 0;
}

__global__ void __launch_bounds__(kUThreads, 1) k_attn_mla_pipe(AttnArgs a, const __grid_constant__ CUtensorMap qmap) {
  // Until the grid dependency is met (programmatic dependent launch: the preceding kernel may still
  // be running) the CTA touches only what no kernel of this library writes: its barriers, TMEM and
  // the buffer's slot-page row (changed only by host calls between launches).  The slot indices and
  // the queries are read after the wait.
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // Q and the ring start 1024-byte aligned (the period of the 128-byte swizzle); the launch adds 1 KB
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + kUQ;
  uint8_t* sP = sRing + kURing * kUSlot;
  __shared__ __align__(8) uint64_t bar_full[kURing], bar_empty[kURing];
  __shared__ __align__(8) uint64_t bar_q, bar_s[2], bar_p, bar_pv, bar_fin, bar_o[4];
  __shared__ uint32_t s_tmem, abort_flag;
  __shared__ uint32_t s_need[2][2][4];            // [parity][warpgroup][warp]
  __shared__ uint32_t s_resc[2];                  // [warpgroup]: some head's max was raised this tile
  __shared__ __align__(16) float s_m[2][32];      // [warpgroup][head]: running max (base 2)
  __shared__ __align__(16) float s_alpha[2][32];  // [warpgroup][head]: rescale of this tile
  __shared__ __align__(16) float s_max[2][4][32]; // [warpgroup][warp][head]: per-warp tile max
  __shared__ __align__(16) float s_sum[2][4][32]; // [warpgroup][warp][head]: per-warp tile weight sum
  __shared__ uint64_t s_pg[kMaxSlotPages];

  const int split = blockIdx.x, r = a.r0 + (int)blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = split * a.chunk;
  const int n = min(a.k, t0 + a.chunk) - t0;
  const int nt = (n + kUTok - 1) / kUTok;
  // a split of one tile keeps the four slots of its value blocks from the score pass to the value
  // product (nothing else is loaded after them); longer splits re-read the values from L2
  const bool hold = nt == 1;
  if (tid == 0) {
    for (int s = 0; s < kURing; ++s) {
      mbar_init(&bar_full[s], (uint32_t)(kUProd * 32));  // every producer thread, once its copies land
      mbar_init(&bar_empty[s], 1u);                      // one MMA commit
    }
    mbar_init(&bar_q, 1u);
    mbar_init(&bar_s[0], 1u);
    mbar_init(&bar_s[1], 1u);
    mbar_init(&bar_p, 256u);  // every softmax thread, once its weights are in place
    mbar_init(&bar_pv, 1u);
    mbar_init(&bar_fin, 1u);
    for (int mt = 0; mt < 4; ++mt) mbar_init(&bar_o[mt], 1u);  // value rows 128 mt.. of the last tile done
    abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < 64) s_m[tid >> 5][tid & 31] = -INFINITY;
  rows_setup(a, r, s_pg);
  const int64_t rows_r = rows_of(a, r);
  if (warp == kUWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&s_tmem))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  attn_enter(a, r, a.err);
  HS_PHASE(hs_phase_attn, 0, threadIdx.x == 0);
  const int32_t* locs = a.locs + (int64_t)(r - a.r0) * a.k + t0;
  // producers: this lane's rows of a tile are 4 (pw + kUProd e) + lane / 8; the first tile's slot
  // indices are requested before the setup barrier
  const int pw = warp - kUWarpProd, crow = lane >> 3, cch = lane & 7;
  int32_t lfirst[kURowsPerLane];
  if (warp >= kUWarpProd) {
#pragma unroll
    for (int e = 0; e < kURowsPerLane; ++e) {
      const int q = pw + kUProd * e, x = 4 * q + crow;
      lfirst[e] = (q < 32 && x < n) ? locs[x] : -1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = s_tmem;
  const uint32_t sq_u = smem_u32(sQ), ring_u = smem_u32(sRing), sp_u = smem_u32(sP);
  HS_PHASE(hs_phase_attn, 1, tid == 0);

  if (warp >= kUWarpProd) {
    // ---------------- producers: Q once by TMA, then the tiles' blocks through the ring ----------------
    if (pw == 0 && lane == 0) {
      mbar_arrive_expect_tx(&bar_q, (uint32_t)kUQ);
      for (int kb = 0; kb < 9; ++kb)
        tma_load_2d(sq_u + (uint32_t)(kb * 8192), &qmap, kb * 64, (r - a.r0) * kUHeads, &bar_q);
    }
    bool ok = true, bad = false;
    // record addresses (0: padding, invalid, or past the split) of this lane's rows, for the tile
    // whose scores are being gathered and for the one whose values are
    uint64_t rows_k[kURowsPerLane], rows_v[kURowsPerLane];
    int u = 0;  // loads issued
    // one slot load: blocks kb0 (and kb0 + 1 when two) of a tile whose rows are `rows`
    auto load = [&](const uint64_t (&rows)[kURowsPerLane], int kb0, int nblk) -> bool {
      const int slot = u % kURing;
      if (u >= kURing && !warp_wait(&bar_empty[slot], (uint32_t)((u / kURing - 1) & 1), &abort_flag)) return false;
      const uint32_t sbase = ring_u + (uint32_t)(slot * kUSlot);
      for (int b = 0; b < nblk; ++b) {
        const int coff = (kb0 + b) * 128 + cch * 16;
#pragma unroll
        for (int e = 0; e < kURowsPerLane; ++e) {
          const int q = pw + kUProd * e;
          if (q < 32) {
            const int row = 4 * q + crow;
            const uint64_t src = rows[e];
            cp_async16_zfill(sbase + (uint32_t)(b * kUBlk + row * 128 + ((cch ^ (row & 7)) << 4)),
                             src != 0ull ? (const void*)(uintptr_t)(src + coff) : (const void*)a.q,
                             src != 0ull ? 16u : 0u);
          }
        }
      }
      HS_PHASE(hs_phase_attn, 2 + u, lane == 0 && pw == 0 && u < 18);  // load u issued
      if (!(a.stall != 0 && u == 0)) cp_async_arrive_noinc(&bar_full[slot]);
      ++u;
      return true;
    };
    int32_t lcur[kURowsPerLane];  // slot indices of this lane's rows of the tile about to be loaded
#pragma unroll
    for (int e = 0; e < kURowsPerLane; ++e) lcur[e] = lfirst[e];
    for (int i = 0; ok && i <= nt; ++i) {
      if (i < nt) {
#pragma unroll
        for (int e = 0; e < kURowsPerLane; ++e) {
          int32_t loc = lcur[e];
          if (loc < -1 || (int64_t)loc >= rows_r) {
            bad = true;
            loc = -1;
          }
          rows_k[e] = loc >= 0 ? (uint64_t)(uintptr_t)row_addr(s_pg, a.kv_shift, a.rec, loc) : 0ull;
        }
        // the next tile's slot indices are requested now, a tile ahead of their use
#pragma unroll
        for (int e = 0; e < kURowsPerLane; ++e) {
          const int q = pw + kUProd * e, x = (i + 1) * kUTok + 4 * q + crow;
          lcur[e] = (i + 1 < nt && q < 32 && x < n) ? locs[x] : -1;
        }
      }
      // scores: all 9 blocks, the last one first, so that blocks 0-7 (the values) fill whole slots
      if (i < nt) {
        ok = load(rows_k, 8, 1);
        for (int p = 0; ok && p < 4; ++p) ok = load(rows_k, 2 * p, 2);
      }
      // values of the tile before; a split of one tile keeps its value blocks from the score pass
      if (i >= 1 && !hold)
        for (int p = 0; ok && p < 4; ++p) ok = load(rows_v, 2 * p, 2);
#pragma unroll
      for (int e = 0; e < kURowsPerLane; ++e) rows_v[e] = rows_k[e];
    }
    if (bad) atomicOr(a.err, (uint32_t)HS_DEVERR_LOC);
    if (!ok && lane == 0) {
      *(volatile uint32_t*)&abort_flag = 1u;
      atomicOr(a.err, (uint32_t)HS_DEVERR_TIMEOUT);
    }
    // every copy this thread issued lands in shared memory before the CTA may exit (the MMA issuer
    // may have given up before consuming the last loads); Q likewise
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (pw == 0 && lane == 0) {
      volatile uint32_t never = 0u;
      mbar_wait_bounded(&bar_q, 0u, &never);
    }
  } else if (warp == kUWarpMma) {
    // ---------------- MMA issuer: S(0), S(1), PV(0), S(2), PV(1), ... ----------------
    const uint32_t id_s = umma_idesc_bf16(128, 64, 0, 0), id_o = umma_idesc_bf16(128, 64, 1, 0);
    // operand descriptors, built once: a score k-step moves 32 B inside an operand (2 in the
    // descriptor's address field, 16-byte units), a value k-step of 16 tokens 2 KB (128); no carry:
    // shared addresses stay below 256 KB
    const uint64_t dq0 = umma_sdesc(sq_u, 16, 1024, 2);         // Q block 0, K-major swizzled
    const uint64_t dk0 = umma_sdesc(ring_u, 16, 1024, 2);       // ring slot 0 as a K operand
    // V^T MN-major from the same bytes: LBO = 16 KB between a slot's two 64-dim blocks, SBO = 1 KB
    // between 8-token groups; P K-major swizzled like Q (two 8 KB blocks of 64 tokens; a k-step of
    // 16 tokens moves 32 B inside a block)
    const uint64_t dv0 = umma_sdesc(ring_u, kUBlk, 1024, 2);
    const uint64_t dp = umma_sdesc(sp_u, 16, 1024, 2);
    constexpr uint64_t kSlotStep = kUSlot >> 4, kBlkStep = kUBlk >> 4, kQStep = 8192 >> 4;
    bool ok = warp_wait(&bar_q, 0u, &abort_flag);
    int u = 0;  // loads consumed
    auto take = [&]() -> int {  // wait for the next load; returns its slot, or -1
      const int slot = u % kURing;
      if (!warp_wait(&bar_full[slot], (uint32_t)((u / kURing) & 1), &abort_flag)) return -1;
      // the producers' copies are generic-proxy writes; the tensor cores read through the async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_after();
      return slot;
    };
    for (int i = 0; ok && i <= nt; ++i) {
      const int j = i - 1;  // the tile whose value product is issued in this round
      if (i < nt) {
        const uint32_t dS = tb + (uint32_t)((i & 1) * 64);
        for (int p = 0; ok && p < 5; ++p) {
          const int slot = take();
          if (slot < 0) {
            ok = false;
            break;
          }
          HS_PHASE(hs_phase_attn, 20 + u, lane == 0 && u < 18);  // load u landed, its score products issued
          if (elect_one()) {
            // load 0 of a tile is block 8, load p >= 1 blocks 2(p-1) and 2(p-1)+1
            for (int b = 0; b < (p == 0 ? 1 : 2); ++b) {
              const int kb = p == 0 ? 8 : 2 * (p - 1) + b;
              const uint64_t dk = dk0 + (uint64_t)slot * kSlotStep + (uint64_t)b * kBlkStep;
              const uint64_t dq = dq0 + (uint64_t)kb * kQStep;
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                umma_bf16(dS, dk + (uint64_t)(2 * ks), dq + (uint64_t)(2 * ks), id_s, (p | ks) != 0 ? 1u : 0u);
            }
            if (p == 0 || !hold) umma_commit(&bar_empty[slot]);
            HS_PHASE(hs_phase_attn, 38 + i, p == 4 && i < 2);  // scores of tile i complete (issued)
            if (p == 4) umma_commit(&bar_s[i & 1]);
          }
          __syncwarp();
          ++u;
        }
      }
      if (ok && j >= 0) {
        // the values of tile j (a split of one tile: still in place from its score pass)
        ok = warp_wait(&bar_p, (uint32_t)(j & 1), &abort_flag);
        if (ok) tc_fence_after();
        HS_PHASE(hs_phase_attn, 51, lane == 0 && j == 0);  // the MMA thread saw the weights of tile 0
        // two 128-row tiles of O^T at a time, their k-steps interleaved so that consecutive products
        // accumulate into different TMEM columns
        for (int pr = 0; ok && pr < 2; ++pr) {
          int sl[2];
          for (int x = 0; ok && x < 2; ++x) {
            // held: value blocks 2mt, 2mt+1 are score load 1 + mt of the split's only tile, still in place
            sl[x] = hold ? (1 + 2 * pr + x) % kURing : take();
            if (sl[x] < 0) ok = false;
            if (!hold) ++u;
          }
          if (!ok) break;
          if (elect_one()) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint64_t dpk = dp + (uint64_t)((ks >> 2) * kQStep + 2 * (ks & 3));
#pragma unroll
              for (int x = 0; x < 2; ++x)
                umma_bf16(tb + (uint32_t)(kUTmemO + 64 * (2 * pr + x)), dv0 + (uint64_t)sl[x] * kSlotStep + (uint64_t)(128 * ks),
                          dpk, id_o, (j | ks) != 0 ? 1u : 0u);
            }
            if (!hold) {
              umma_commit(&bar_empty[sl[0]]);
              umma_commit(&bar_empty[sl[1]]);
            }
            if (pr == 1) umma_commit(&bar_pv);
            if (j == nt - 1) {  // the epilogue reads these rows meanwhile
              umma_commit(&bar_o[2 * pr]);
              umma_commit(&bar_o[2 * pr + 1]);
            }
            HS_PHASE(hs_phase_attn, 40 + j, pr == 1 && j < 3);  // value product of tile j issued
            HS_PHASE(hs_phase_attn, 53 + 2 * pr, j == 0);        // its value rows 256 pr.. issued (tile 0)
          }
          __syncwarp();
        }
      }
    }
    if (!ok && lane == 0) {
      *(volatile uint32_t*)&abort_flag = 1u;
      atomicOr(a.err, (uint32_t)HS_DEVERR_TIMEOUT);
    }
    // every product issued has completed before the accumulator can be released
    if (elect_one()) umma_commit(&bar_fin);
    __syncwarp();
    {
      volatile uint32_t never = 0u;
      warp_wait(&bar_fin, 0u, &never);
    }
  } else {
    // ---------------- softmax: warpgroup g = heads 32g..32g+31, thread = token = TMEM lane ----------------
    // Every thread of a warpgroup passes the same sequence of its barrier: a wait that gives up only
    // marks the thread (ok = false: no TMEM access, zero weights), so a barrier never misses a thread.
    const int g = warp >> 2, wq = warp & 3, tok = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    float lsum = 0.f;  // warp 0 of the warpgroup: running weight sum of head 32g + lane
    bool ok = true;
    for (int i = 0; i < nt; ++i) {
      if (ok) ok = mbar_wait_bounded(&bar_s[i & 1], (uint32_t)((i >> 1) & 1), &abort_flag);
      tc_fence_after();
      HS_PHASE(hs_phase_attn, 43 + i, tid == 0 && i < 3);  // softmax saw the scores of tile i
      const int x = i * kUTok + tok;
      const int32_t lx = x < n ? locs[x] : -1;
      const bool valid = ok && lx >= 0 && (int64_t)lx < rows_r;
      float v[32];
      if (ok) tmem_ld32(tb + lane_base + (uint32_t)((i & 1) * 64 + 32 * g), v);
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) v[jj] = valid ? v[jj] * a.qscale : -INFINITY;
      bool need = false;
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const float4 m4 = *(const float4*)&s_m[g][4 * j4];
        need |= v[4 * j4] > m4.x + kULazy;
        need |= v[4 * j4 + 1] > m4.y + kULazy;
        need |= v[4 * j4 + 2] > m4.z + kULazy;
        need |= v[4 * j4 + 3] > m4.w + kULazy;
      }
      const int par = i & 1;
      const bool need_w = __any_sync(0xffffffffu, need);
      if (lane == 0) s_need[par][g][wq] = need_w ? 1u : 0u;
      wg_sync(g);
      const bool any = (s_need[par][g][0] | s_need[par][g][1] | s_need[par][g][2] | s_need[par][g][3]) != 0u;
      bool resc = false;
      if (any) {
        // exact tile max per head; warp 0 of the warpgroup raises the running max where needed
        float t[32];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) t[jj] = v[jj];
        s_max[g][wq][lane] = reduce32_max_transposed(t, lane);  // head 32g + lane over this warp's tokens
        wg_sync(g);
        if (wq == 0) {
          const float tm = fmaxf(fmaxf(s_max[g][0][lane], s_max[g][1][lane]), fmaxf(s_max[g][2][lane], s_max[g][3][lane]));
          const float mo = s_m[g][lane];
          const float mn = tm > mo + kULazy ? tm : mo;
          // a head with nothing accumulated yet has zero sums and accumulators: nothing to scale
          const float al = (mn == mo || mo == -INFINITY) ? 1.f : fast_exp2(mo - mn);
          s_alpha[g][lane] = al;
          s_m[g][lane] = mn;
          lsum *= al;
          const bool rw = __any_sync(0xffffffffu, al != 1.f);
          if (lane == 0) s_resc[g] = rw ? 1u : 0u;
        }
        wg_sync(g);
        resc = s_resc[g] != 0u;
      }
      // the previous tile's value product is complete: P may be rewritten and O^T rescaled
      if (ok && i >= 1) ok = mbar_wait_bounded(&bar_pv, (uint32_t)((i - 1) & 1), &abort_flag);
      tc_fence_after();
      if (resc && ok && i >= 1) {
#pragma unroll 1
        for (int mt = 0; mt < 4; ++mt) {
          float o[32];
          const uint32_t ta = tb + lane_base + (uint32_t)(kUTmemO + 64 * mt + 32 * g);
          tmem_ld32(ta, o);
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) o[jj] *= s_alpha[g][jj];
          tmem_st32(ta, o);
        }
      }
      // weights (bf16)
      uint32_t pk[16];
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const float4 m4 = *(const float4*)&s_m[g][4 * j4];
        pk[2 * j4] = pack_bf16(valid ? fast_exp2(v[4 * j4] - m4.x) : 0.f, valid ? fast_exp2(v[4 * j4 + 1] - m4.y) : 0.f);
        pk[2 * j4 + 1] =
            pack_bf16(valid ? fast_exp2(v[4 * j4 + 2] - m4.z) : 0.f, valid ? fast_exp2(v[4 * j4 + 3] - m4.w) : 0.f);
      }
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        v[2 * jj] = __uint_as_float(pk[jj] << 16);  // the rounded weights, as the MMA sees them
        v[2 * jj + 1] = __uint_as_float(pk[jj] & 0xffff0000u);
      }
      // P (the value product's B operand, K-major): two blocks of 64 tokens, each 64 head rows of
      // 128 B, 128-byte swizzled like Q (tokens 8c..8c+7 of head h in the 16-byte chunk c XOR (h mod 8)).
      // A warp's store of one head writes 64 contiguous bytes of its row: no bank conflict.
      {
        uint8_t* pblk = sP + (tok >> 6) * 8192 + (tok & 7) * 2;
        const int c = (tok & 63) >> 3;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int h0 = 32 * g + 2 * jj;
          *(uint16_t*)(pblk + h0 * 128 + ((c ^ (h0 & 7)) << 4)) = (uint16_t)(pk[jj] & 0xffffu);
          *(uint16_t*)(pblk + (h0 + 1) * 128 + ((c ^ ((h0 + 1) & 7)) << 4)) = (uint16_t)(pk[jj] >> 16);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P is read by the tensor cores
      tc_fence_before();
      mbar_arrive(&bar_p);
      HS_PHASE(hs_phase_attn, 46 + i, tid == 0 && i < 3);  // weights of tile i written
      // this tile's weight sums per head: this warp's tokens, then the four warps in order
      s_sum[g][wq][lane] = reduce32_transposed(v, lane);
      wg_sync(g);
      if (wq == 0) lsum += (s_sum[g][0][lane] + s_sum[g][1][lane]) + (s_sum[g][2][lane] + s_sum[g][3][lane]);
    }
    HS_PHASE(hs_phase_attn, 49, tid == 0);
    // the partial, 128 value rows at a time as the last tile's value product completes them: O^T
    // rows (value dims) of this thread, the warpgroup's heads; a warp stores 32 consecutive dims
    const int64_t ph0 = ((int64_t)r * a.S + split) * a.Hq + 32 * g;
#pragma unroll 1
    for (int mt = 0; mt < 4; ++mt) {
      if (ok) ok = mbar_wait_bounded(&bar_o[mt], 0u, &abort_flag);
      tc_fence_after();
      HS_PHASE(hs_phase_attn, 56, tid == 0 && mt == 0);  // value rows 0-127 of the last tile complete
      if (ok && abort_flag == 0u) {
        float o[32];
        tmem_ld32(tb + lane_base + (uint32_t)(kUTmemO + 64 * mt + 32 * g), o);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) a.part[(ph0 + jj) * 512 + mt * 128 + tok] = o[jj];
      }
    }
    if (!ok) {
      *(volatile uint32_t*)&abort_flag = 1u;
      atomicOr(a.err, (uint32_t)HS_DEVERR_TIMEOUT);
    }
    // max and sum last: a split that gave up leaves them unwritten
    if (ok && abort_flag == 0u && wq == 0) *(float2*)(a.ml + (ph0 + lane) * 2) = make_float2(s_m[g][lane], lsum);
    HS_PHASE(hs_phase_attn, 50, tid == 0);  // partial written
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kUWarpMma) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tb) : "memory");
}

// ---- dispatch ----------------------------------------------------------------

struct Plan {
  int kind;  // 0: CUDA-core shared-latent, 1: GQA per KV head, 4: shared-latent on tcgen05
  int NW, G, T, groups, S, chunk;
  int fetch;  // 1: the GQA kernel also copies the misses the resolve left pending
  size_t smem;
};


bool plan_for(const hs_config* c, int num_sms, Plan* pl) {
  const int64_t rec = hs_record_bytes(c);
  int per_cta_wave;
  if (c->layout == HS_LAYOUT_GQA) {
    if (c->head_dim_qk != 128 || c->head_dim_v != 128) return false;
    const int G = c->num_q_heads / c->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return false;
    pl->G = G;
    pl->T = kMmaTile;
    pl->kind = 1;
    pl->NW = kGqaWarps;
    pl->groups = c->num_kv_heads;  // one KV head per CTA
    pl->fetch = c->fetch_in_attention != 0;
    pl->smem = (size_t)kGqaWarps * kGqaStages * kMmaTile * kGqaRow;
    per_cta_wave = 1;  // one CTA per SM: the staging buffers hold most of the shared memory
  } else if (c->head_dim_qk == 576 && c->head_dim_v == 512 && c->num_q_heads == kMlaHeads) {
    // tcgen05 kernel: Q resident, the tiles streamed through the ring.  One CTA per SM; splits of any
    // multiple of 16 tokens (a ragged last tile reads zero rows), at least 64 tokens each so that a
    // CTA's Q load (72 KB) does not outweigh its records, at most 32 per request (the wide combine)
    pl->kind = 4;
    pl->fetch = 0;
    pl->NW = 8;
    pl->G = kMlaHeads;
    pl->groups = 1;
    pl->T = 16;
    pl->smem = kUSmem;
    int S = num_sms / c->num_requests;
    const int max_s = (c->top_k + 63) / 64;
    S = S < 1 ? 1 : (S > max_s ? max_s : S);
    S = S > 32 ? 32 : S;
    int chunk = (c->top_k + S - 1) / S;
    chunk = (chunk + 15) / 16 * 16;
    pl->chunk = chunk;
    pl->S = (c->top_k + chunk - 1) / chunk;
    return pl->smem <= 227 * 1024;
  } else {
    if (c->head_dim_qk != 576 || c->head_dim_v != 512) return false;
    if (c->num_q_heads % 8 != 0) return false;
    pl->kind = 0;
    pl->fetch = 0;
    pl->NW = 8;
    pl->G = 1;
    pl->groups = c->num_q_heads / 8;
    pl->T = 32 / pl->G;
    pl->smem = (size_t)kStages * pl->T * (size_t)rec;
    per_cta_wave = 2;
  }
  const int per_split = c->num_requests * pl->groups;
  int S = per_cta_wave * num_sms / per_split;
  const int max_s = (c->top_k + pl->T - 1) / pl->T;
  S = S < 1 ? 1 : (S > max_s ? max_s : S);
  int chunk = (c->top_k + S - 1) / S;
  chunk = (chunk + pl->T - 1) / pl->T * pl->T;
  pl->chunk = chunk;
  pl->S = (c->top_k + chunk - 1) / chunk;

  return pl->smem <= 220 * 1024;
}

template <typename K>
cudaError_t launch_kernel(K kern, const AttnArgs* a, const Plan& pl, int threads, cudaStream_t st) {
  if (a == nullptr) {  // preparation, once: the dynamic shared-memory limit and the largest carveout
    cudaError_t e = hs_raise_smem_limit(kern, (int)pl.smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.S, a->R, pl.groups);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, *a);
}



typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime; null if unavailable.
EncodeFn tensor_map_encoder() {
  static const EncodeFn fn = []() -> EncodeFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        f == nullptr || q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return (EncodeFn)f;
  }();
  return fn;
}

// Q of the launch's requests as a 2-D tensor (rows = request x head, 576 bf16 each) in boxes of 64
// dims x 64 heads, 128-byte swizzled: the tensor-core kernel's Q operand layout.  False (and Q by
// cp.async) when the encoder is missing or refuses the address.
bool encode_q_map(CUtensorMap* m, const void* q, int nreq) {
  const EncodeFn fn = tensor_map_encoder();
  if (fn == nullptr || q == nullptr || ((uintptr_t)q & 15u) != 0) return false;
  const cuuint64_t gdim[2] = {(cuuint64_t)kUDim, (cuuint64_t)nreq * kUHeads};
  const cuuint64_t gstride[1] = {(cuuint64_t)kUDim * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kUHeads}, estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), gdim, gstride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t dispatch(const hs_config& c, const AttnArgs* a, const Plan& pl, cudaStream_t st) {
  if (pl.kind == 4) {
    cudaError_t e = cudaSuccess;
    if (a == nullptr) {  // preparation: shared-memory limit and carveout
      e = hs_raise_smem_limit(k_attn_mla_pipe, (int)pl.smem);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attn_mla_pipe, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    } else {
      // Q through a tensor map of the launch's queries, encoded for this launch
      CUtensorMap qm;
      memset(&qm, 0, sizeof(qm));
      if (!encode_q_map(&qm, a->q, a->R)) return cudaErrorNotSupported;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(pl.S, a->R, pl.groups);
      cfg.blockDim = dim3(kUThreads, 1, 1);
      cfg.dynamicSmemBytes = pl.smem;
      cfg.stream = st;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, k_attn_mla_pipe, *a, qm);
    }
    if (e == cudaSuccess && a == nullptr)
      e = cudaFuncSetAttribute(k_combine_wide, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess || a == nullptr) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a->R, (a->Hq + 1) / 2, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_combine_wide, *a);
  }
  if (pl.kind == 0) return launch_kernel(k_attn_cc<576, 512, 1, 8>, a, pl, AttnCfg<576, 512, 1, 8>::THREADS, st);
  if (pl.fetch) {
    switch (pl.G) {
      case 1: return launch_kernel(k_attn_gqa<1, true>, a, pl, (kGqaWarps + kGqaProducers) * 32, st);
      case 2: return launch_kernel(k_attn_gqa<2, true>, a, pl, (kGqaWarps + kGqaProducers) * 32, st);
      case 4: return launch_kernel(k_attn_gqa<4, true>, a, pl, (kGqaWarps + kGqaProducers) * 32, st);
      default: return launch_kernel(k_attn_gqa<8, true>, a, pl, (kGqaWarps + kGqaProducers) * 32, st);
    }
  }
  switch (pl.G) {
    case 1: return launch_kernel(k_attn_gqa<1, false>, a, pl, (kGqaWarps + kGqaProducers) * 32, st);
    case 2: return launch_kernel(k_attn_gqa<2, false>, a, pl, (kGqaWarps + kGqaProducers) * 32, st);
    case 4: return launch_kernel(k_attn_gqa<4, false>, a, pl, (kGqaWarps + kGqaProducers) * 32, st);
    default: return launch_kernel(k_attn_gqa<8, false>, a, pl, (kGqaWarps + kGqaProducers) * 32, st);
  }
}

}  // namespace

bool hs_attn_can_fetch(const hs_config* c) {
  hs_config f = *c;
  f.fetch_in_attention = 1;
  Plan pl;
  return plan_for(&f, 152, &pl) && pl.kind == 1;
}

bool hs_attn_supported(const hs_config* c) {
  Plan pl;
  return plan_for(c, 152, &pl);
}

void hs_attn_workspace(const hs_config* c, int num_sms, size_t* floats, int* max_splits, int* tickets_per_req) {
  Plan pl;
  plan_for(c, num_sms, &pl);
  *max_splits = pl.S;
  *tickets_per_req = pl.groups + 1;  // one per group, then the pending-list count
  *floats = (size_t)c->num_requests * pl.S * c->num_q_heads * ((size_t)c->head_dim_v + 2);
}

int hs_launch_attn(hs_pool* p, int layer, int r0, int nreq, const void* d_q, const int32_t* d_locs,
                   const void* kv_base, int64_t kv_rows, float scale, float* d_out, cudaStream_t st) {
  const hs_config& c = p->cfg;
  Plan pl;
  if (!plan_for(&c, p->num_sms, &pl)) return HS_ERR_CONFIG;
  if (kv_base != nullptr && ((uintptr_t)kv_base & 15u) != 0) return HS_ERR_ARG;
  AttnArgs a{};
  a.q = (const uint16_t*)d_q;
  a.locs = d_locs;
  if (kv_base == nullptr) {  // the layer's hot buffers, through the slot table
    a.kv_pt = p->slot_table + (int64_t)layer * c.num_requests * p->slot_pages;
    a.kv_cap = p->slot_cap + (int64_t)layer * c.num_requests;
    a.kv_pages = p->slot_pages;
    a.kv_shift = p->slot_shift;
    a.rows = c.buffer_slots;
  } else {
    a.kv = (const uint8_t*)kv_base;
    a.kv_pages = 1;
    a.kv_shift = 31;
    a.rows = kv_rows;
  }
  a.out = d_out;
  a.part = p->attn_part;
  a.ml = p->attn_part + (size_t)c.num_requests * pl.S * c.num_q_heads * c.head_dim_v;
  a.ticket = p->attn_ticket;
  a.err = p->err_global;
  a.rec = p->rec;
  if (c.layout == HS_LAYOUT_GQA) {
    a.kstride = 2 * (int64_t)(c.head_dim_qk + c.head_dim_v);
    a.vdelta = 2 * (int64_t)c.head_dim_qk;
  } else {
    a.kstride = 0;
    a.vdelta = 0;
  }
  a.qscale = scale * kLog2e;
  a.R = nreq;
  a.r0 = r0;
  a.Hq = c.num_q_heads;
  a.k = c.top_k;
  a.S = pl.S;
  a.chunk = pl.chunk;
  a.groups = pl.groups;
  const bool hot = kv_base == nullptr;
  a.pend = (hot && p->pend != nullptr) ? p->pend + (int64_t)layer * c.num_requests * c.top_k : nullptr;
  a.pend_live = (hot && p->pend_live != nullptr) ? p->pend_live + (int64_t)layer * c.num_requests : nullptr;
  a.L = c.num_layers;
  a.layer = layer;
  if (pl.kind == 4 && (p->debug_stall & HS_STALL_ATTN) != 0) {  // test hook, consumed by this launch
    a.stall = 1;
    p->debug_stall &= ~HS_STALL_ATTN;
  }
  // directly after the whole-batch resolve of this layer on this stream (GQA or 64-head shared-latent
  // kernel, misses copied by the resolve): wait for each request's own resolve CTAs rather than the
  // whole resolve grid
#ifndef HS_ATTN_WAIT_WHOLE_GRID  // build option: always wait for the whole resolve grid
  if ((pl.kind == 1 || pl.kind == 4) && !pl.fetch && kv_base == nullptr && r0 == 0 && nreq == c.num_requests &&
      p->last_res_layer == layer && p->last_res_stream == st) {
    a.res_count = p->res_count + (int64_t)layer * c.num_requests * 2;
    a.res_cs = p->resolve_ctas;
  }
#endif
  p->last_res_layer = -1;
  return dispatch(c, &a, pl, st) == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

int hs_attn_prepare(const hs_config* c, int num_sms) {
  Plan pl;
  if (!plan_for(c, num_sms, &pl)) return HS_ERR_CONFIG;
  return dispatch(*c, nullptr, pl, 0) == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

// ---- attention without any allocation --------------------------------------------------
//
// For callers that may not allocate device memory at all: an inference engine whose own
// allocator owns every byte of HBM, or a process that must not grow its footprint after start-up.
// Their attention runs the same kernels as hs_sparse_attn, but the split partials, the combine
// tickets and the error word live in this fixed file-scope array instead of a pool.  Every GPU
// that loads the library holds it until the process exits.

#include <mutex>

namespace {

constexpr size_t kNoAllocTicketBytes = 64 * 1024;  // the error word, then up to 16380 tickets
constexpr size_t kNoAllocTicketOff = 16;            // tickets start here (the error word is at 0)
constexpr size_t kNoAllocPartBytes = (size_t)HS_NOALLOC_SCRATCH_BYTES - kNoAllocTicketBytes;
static __device__ __align__(256) unsigned char hs_noalloc_scratch[HS_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices];  // device address of hs_noalloc_scratch on each device
int g_noalloc_sms[kMaxDevices];

// Once per device, with that device current: the scratch's device address (host code only has a
// stand-in symbol) and the kernels' shared-memory limits are fixed here.
int noalloc_setup(int dev, const hs_config* c, void** ptr, int* sms) {
  if (dev < 0 || dev >= kMaxDevices) return HS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, hs_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return HS_ERR_CUDA;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
      cudaGetLastError();
      return HS_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
    g_noalloc_sms[dev] = n;
  }
  *ptr = g_noalloc_ptr[dev];
  *sms = g_noalloc_sms[dev];
  // the kernel for this configuration may not have had its shared-memory limit raised yet
  return hs_attn_prepare(c, *sms);
}

}  // namespace

extern "C" int hs_sparse_attn_noalloc(const hs_config* cfg, const void* d_q, const int32_t* d_locs,
                                      const void* d_kv, int64_t kv_rows, float scale, float* d_out, void* stream) {
  if (cfg == nullptr || d_q == nullptr || d_locs == nullptr || d_kv == nullptr || d_out == nullptr) return HS_ERR_ARG;
  if (kv_rows < 1 || kv_rows > (int64_t)INT32_MAX || ((uintptr_t)d_kv & 15u) != 0) return HS_ERR_ARG;
  if (!hs_aligned(d_q, 16) || !hs_aligned(d_out, 16) || !hs_aligned(d_locs, 4)) return HS_ERR_ARG;
  // only the documented fields decide the kernel and its split plan: the rest of *cfg (pool
  // settings such as fetch_in_attention) is ignored
  hs_config c;
  memset(&c, 0, sizeof(c));
  c.num_requests = cfg->num_requests;
  c.num_layers = 1;
  c.layout = cfg->layout;
  c.num_q_heads = cfg->num_q_heads;
  c.num_kv_heads = cfg->num_kv_heads;
  c.head_dim_qk = cfg->head_dim_qk;
  c.head_dim_v = cfg->head_dim_v;
  c.top_k = cfg->top_k;
  if (c.num_requests < 1 || c.top_k < 1 || c.num_q_heads < 1 || c.num_kv_heads < 1 ||
      c.num_q_heads % c.num_kv_heads != 0)
    return HS_ERR_CONFIG;
  if (c.layout == HS_LAYOUT_MLA && c.num_kv_heads != 1) return HS_ERR_CONFIG;
  if (!hs_attn_supported(&c)) return HS_ERR_CONFIG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  void* scratch = nullptr;
  int sms = 0;
  int rc = noalloc_setup(dev, &c, &scratch, &sms);
  if (rc != HS_OK) return rc;
  Plan pl;
  if (!plan_for(&c, sms, &pl)) return HS_ERR_CONFIG;
  const size_t o_floats = (size_t)c.num_requests * pl.S * c.num_q_heads * c.head_dim_v;
  const size_t ml_floats = (size_t)c.num_requests * pl.S * c.num_q_heads * 2;
  const size_t tickets = (size_t)c.num_requests * (pl.groups + 1);
  if ((o_floats + ml_floats) * sizeof(float) > kNoAllocPartBytes ||
      kNoAllocTicketOff + tickets * sizeof(uint32_t) > kNoAllocTicketBytes)
    return HS_ERR_SCRATCH;
  uint8_t* base = (uint8_t*)scratch;
  uint32_t* err = (uint32_t*)base;  // fixed offset: the error word comes first
  uint32_t* ticket = (uint32_t*)(base + kNoAllocTicketOff);
  float* part = (float*)(base + kNoAllocTicketBytes);
  float* ml = part + o_floats;
  cudaStream_t st = (cudaStream_t)stream;
  // The error word and the tickets start at zero (a call whose wait gave up may have left tickets
  // raised).  The split statistics and the output start as NaN (all bits set): a CTA whose bounded
  // wait gave up writes neither, so its request's output stays NaN (the combine of a NaN statistic
  // gives NaN) instead of an earlier call's values.
  if (cudaMemsetAsync(base, 0, kNoAllocTicketOff + tickets * sizeof(uint32_t), st) != cudaSuccess ||
      cudaMemsetAsync(ml, 0xff, ml_floats * sizeof(float), st) != cudaSuccess ||
      cudaMemsetAsync(d_out, 0xff, (size_t)c.num_requests * c.num_q_heads * c.head_dim_v * sizeof(float), st) !=
          cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  AttnArgs a{};
  a.q = (const uint16_t*)d_q;
  a.locs = d_locs;
  a.kv = (const uint8_t*)d_kv;
  a.kv_pages = 1;
  a.kv_shift = 31;
  a.rows = kv_rows;
  a.out = d_out;
  a.part = part;
  a.ml = ml;
  a.ticket = ticket;
  a.err = err;
  a.rec = hs_record_bytes(&c);
  if (c.layout == HS_LAYOUT_GQA) {
    a.kstride = 2 * (int64_t)(c.head_dim_qk + c.head_dim_v);
    a.vdelta = 2 * (int64_t)c.head_dim_qk;
  } else {
    a.kstride = 0;
    a.vdelta = 0;
  }
  a.qscale = scale * kLog2e;
  a.R = c.num_requests;
  a.Hq = c.num_q_heads;
  a.k = c.top_k;
  a.S = pl.S;
  a.chunk = pl.chunk;
  a.groups = pl.groups;
  return dispatch(c, &a, pl, st) == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}
