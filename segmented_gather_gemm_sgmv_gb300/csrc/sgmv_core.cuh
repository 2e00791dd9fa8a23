// sgmv_core.cuh -- the segment scheduler and the CUDA-core shrink / expand / fused kernels.
//
// Operation (Punica Guide: Multi-Tenant LoRA Serving with SGMV; section "The Heterogeneous
// Batching Bottleneck", equation y_i = x_i W0 + (alpha/r) x_i A_k B_k; section "The SGMV
// Mathematical Formulation", segments [s_i, s_{i+1}) bound to one adapter each):
//     v[t]  = x[t] . A_k            shrink  (h_in -> r)
//     y[t] += scale * v[t] . B_k    expand  (r -> h_out)
//
// GB300 design (not the pages' Ampere design):
//  * Scheduler, in every CTA: the segment table is staged in shared memory and every segment
//    with an adapter is hashed by adapter id, so that all rows of one adapter -- even rows of
//    non-adjacent segments -- form one group whose weights are streamed once per call.  A
//    group is cut into work items of at most `rmax` rows.  All CTAs derive the same item list;
//    cluster q runs items q, q+G, q+2G, ...  (The pages' "pre-sorted segment descriptors" and
//    "one threadblock per segment", section "Hardware-Level Optimizations in SGMV".)
//  * One item runs on one thread-block cluster of C CTAs.  CTA c owns the c-th slice of h_in
//    (shrink, split-K) and of h_out (expand).  Its weight slices stream through a ring of
//    shared-memory stages filled by 1-D bulk copies (TMA) that one producer warp issues; the
//    eight consumer warps compute on the CUDA cores in fp32.
//  * The r-wide partial products of the C CTAs are summed through distributed shared memory
//    in a fixed order (deterministic), so the intermediate v never leaves the cluster in the
//    fused path.
//  * Every wait is bounded (globaltimer); a wait that runs out flags the CTA, sets the
//    library's device error word and lets the kernel run to its end without touching global
//    memory again.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sgmv_ptx.cuh"

namespace sgmv {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kStatusTimeout = -5;         // SGMV_ETIMEOUT

enum Mode : int { kFused = 0, kShrink = 1, kExpand = 2 };

// Barrier slots after the 2*nstages ring barriers.
enum Bar : int { kXFull = 0, kXFree, kYFull, kYFree, kDesc0, kDesc1, kVReady0, kVReady1, kNever,
                 kNumFixedBars };

struct Params {
  void* y;
  const void* x;
  float* v_out;
  const float* v_in;
  const void* const* A_ptrs;
  const void* const* B_ptrs;
  const int32_t* seg_starts;
  const int32_t* seg_adapter;
  int* err;  // library device error word
  int32_t S, layer, h_in, h_out;
  float scale;
  int32_t C;            // CTAs per item (cluster size for shrink / fused)
  int32_t nstages;      // ring stages
  int32_t stage_bytes;  // bytes per ring stage
  int32_t rmax;         // rows per work item
  int32_t kc_max, nc_max;  // widest h_in / h_out slice of one CTA (elements)
  int32_t wmax;            // widest B row segment one expand pass covers (elements)
  int32_t hash_slots;      // power of two > 1.5*S
  uint32_t off_bars, off_ctl, off_desc, off_tab, off_vpart, off_vfull, off_red, off_xs, off_ys,
      off_ring;
  uint32_t xs_row_bytes, ys_row_bytes;
  int32_t desc_ints;
  uint64_t wait_limit_ns;
  int32_t inject_stall;
};

// ---- element types ---------------------------------------------------------------------
template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kVec = 4;  // elements per 16 bytes
  __device__ static __forceinline__ void load16(const void* p, float (&o)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
  __device__ static __forceinline__ float load1(const void* p) {
    return *reinterpret_cast<const float*>(p);
  }
  __device__ static __forceinline__ void store16(void* p, const float (&o)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
  }
};
template <>
struct Elem<__half> {
  static constexpr int kVec = 8;
  __device__ static __forceinline__ void load16(const void* p, float (&o)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      o[2 * i] = f.x;
      o[2 * i + 1] = f.y;
    }
  }
  __device__ static __forceinline__ float load1(const void* p) {
    return __half2float(*reinterpret_cast<const __half*>(p));
  }
  __device__ static __forceinline__ void store16(void* p, const float (&o)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __floats2half2_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ static __forceinline__ void load16(const void* p, float (&o)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // bf16 -> fp32 is exact: the bf16 bits are the high half
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static __forceinline__ float load1(const void* p) {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
  }
  __device__ static __forceinline__ void store16(void* p, const float (&o)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// ---- bounded waits ----------------------------------------------------------------------
struct Waiter {
  volatile int* abort;  // CTA-wide flag in shared memory
  int* err;
  uint64_t limit;

  // Returns false (without waiting) once the CTA has given up, or when the bound runs out.
  template <bool kCluster>
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
    if (*abort) return false;
    if (kCluster ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    while (true) {
#pragma unroll 1
      for (int i = 0; i < 8; ++i)
        if (kCluster ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
      if (*abort) return false;
      if (now_ns() - t0 > limit) {
        *abort = 1;
        atomicExch(err, kStatusTimeout);
        return false;
      }
    }
  }
  __device__ __forceinline__ bool ok() const { return *abort == 0; }
};

// ---- slices and chunking (identical arithmetic on the producer and consumer sides) -------
static __device__ __forceinline__ void slice_of(int n, int C, int c, int& lo, int& hi) {
  const int units = n >> 3;  // slices start on multiples of 8 elements (16-byte aligned)
  lo = (units * c / C) << 3;
  hi = (units * (c + 1) / C) << 3;
}

template <typename T, int R>
struct Chunking {
  int kc, nc;     // this CTA's h_in / h_out slice width
  int kb, nA;     // A rows per chunk, number of A chunks
  int passes;     // expand passes
  __device__ __forceinline__ void init(const Params& p, int kc_, int nc_) {
    kc = kc_;
    nc = nc_;
    kb = p.stage_bytes / (R * (int)sizeof(T));
    nA = (kc + kb - 1) / kb;
    passes = (nc + p.wmax - 1) / p.wmax;
  }
  __device__ __forceinline__ int pass_width(const Params& p, int pass) const {
    return min(p.wmax, nc - pass * p.wmax);
  }
  __device__ __forceinline__ static int row_stride(int w) {  // padded B row in a stage
    return w * (int)sizeof(T) + 16;
  }
  __device__ __forceinline__ int pass_rows(const Params& p, int w) const {  // B rows / chunk
    return min(R, p.stage_bytes / row_stride(w));
  }
};

// ---- scheduler ------------------------------------------------------------------------
// Exclusive scan of `cnt(i)` over i in [0, n) into out[0..n] (out[n] = total), all threads.
template <typename F>
__device__ void block_exclusive_scan(int n, int* out, int* wsum, F cnt) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kThreads / 32;
  const int per = (n + kThreads - 1) / kThreads;
  const int lo = min(tid * per, n), hi = min(lo + per, n);
  int local = 0;
  for (int i = lo; i < hi; ++i) local += cnt(i);
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int v = wsum[w];
      wsum[w] = run;
      run += v;
    }
    wsum[kWarps] = run;
  }
  __syncthreads();
  int off = wsum[warp] + incl - local;
  for (int i = lo; i < hi; ++i) {
    out[i] = off;
    off += cnt(i);
  }
  if (tid == 0) out[n] = wsum[kWarps];
  __syncthreads();
}

static __device__ __forceinline__ uint32_t hash_slot(int k, int mask) {
  return ((static_cast<uint32_t>(k) * 0x9E3779B1u) >> 12) & static_cast<uint32_t>(mask);
}

// Builds, in shared memory: starts[0..S], adapters[0..S-1], base[0..S] where base is the
// exclusive prefix of "work items led by segment i".  Segment i leads its group when it is the
// first non-empty segment of its adapter; its group gets ceil(rows / rmax) items.
// `scratch` (transient) holds slot[S] and the hash table (3 * hash_slots ints).
static __device__ void build_schedule(const Params& p, int* starts, int* adapters, int* base,
                               int* scratch, int* wsum) {
  const int tid = threadIdx.x;
  const int S = p.S, HS = p.hash_slots;
  int* slot = scratch;
  int* hkey = slot + S;
  int* hlead = hkey + HS;
  int* hcnt = hlead + HS;
  for (int i = tid; i <= S; i += kThreads) starts[i] = __ldg(p.seg_starts + i);
  for (int i = tid; i < S; i += kThreads) adapters[i] = __ldg(p.seg_adapter + i);
  for (int h = tid; h < HS; h += kThreads) {
    hkey[h] = -1;
    hlead[h] = 0x7fffffff;
    hcnt[h] = 0;
  }
  __syncthreads();
  for (int i = tid; i < S; i += kThreads) {
    const int k = adapters[i];
    const int len = starts[i + 1] - starts[i];
    int h = -1;
    if (k >= 0 && len > 0) {
      h = static_cast<int>(hash_slot(k, HS - 1));
      while (true) {  // at most S distinct keys in HS > 1.5 S slots: terminates
        const int prev = atomicCAS(&hkey[h], -1, k);
        if (prev == -1 || prev == k) break;
        h = (h + 1) & (HS - 1);
      }
      atomicMin(&hlead[h], i);
      atomicAdd(&hcnt[h], len);
    }
    slot[i] = h;
  }
  __syncthreads();
  const int rmax = p.rmax;
  block_exclusive_scan(S, base, wsum, [&](int i) {
    const int h = slot[i];
    return (h >= 0 && hlead[h] == i) ? (hcnt[h] + rmax - 1) / rmax : 0;
  });
}

// One warp: turns item t into {adapter, rows, row ids...} in d (d[0]=k, d[1]=R, d[2..]=rows).
static __device__ void decode_item(const Params& p, int t, const int* starts, const int* adapters,
                            const int* base, int* d) {
  const int lane = threadIdx.x & 31;
  const int S = p.S;
  int lo = 0, hi = S - 1;  // largest i with base[i] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int lead = lo;
  const int k = adapters[lead];
  const int p_lo = (t - base[lead]) * p.rmax;
  const int p_hi = p_lo + p.rmax;
  int pos = 0;
  for (int jb = lead; jb < S && pos < p_hi; jb += 32) {
    const int j = jb + lane;
    int len = 0;
    if (j < S && adapters[j] == k) len = max(starts[j + 1] - starts[j], 0);
    int incl = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int seg_lo = pos + incl - len;
    const int a = max(seg_lo, p_lo), b = min(pos + incl, p_hi);
    for (int q = a; q < b; ++q) d[2 + q - p_lo] = starts[j] + (q - seg_lo);
    pos += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) {
    d[0] = k;
    d[1] = max(0, min(pos, p_hi) - p_lo);
  }
  __syncwarp();
}

// ---- the kernel ------------------------------------------------------------------------
template <typename T, int R, int MODE>
struct Kernel {
  using E = Elem<T>;
  static constexpr int kVec = E::kVec;
  static constexpr int kCpr = R / kVec;          // 16-byte chunks per A row
  static constexpr int kKLanes = kConsumers / kCpr;
  static constexpr int kEb = sizeof(T);
  static_assert(kCpr >= 1 && kCpr <= 32, "rank / vector width");

  struct Smem {
    uint8_t* base;
    const Params* p;
    __device__ uint32_t bar(int i) const {
      return smem_addr(base + p->off_bars) + 8u * static_cast<uint32_t>(i);
    }
    __device__ uint32_t full(int s) const { return bar(s); }
    __device__ uint32_t empty(int s) const { return bar(p->nstages + s); }
    __device__ uint32_t fixed(int b) const { return bar(2 * p->nstages + b); }
    __device__ uint8_t* stage(int s) const {
      return base + p->off_ring + static_cast<uint32_t>(s) * p->stage_bytes;
    }
    __device__ int* desc(int b) const {
      return reinterpret_cast<int*>(base + p->off_desc) + b * p->desc_ints;
    }
    __device__ float* vpart(int b) const {
      return reinterpret_cast<float*>(base + p->off_vpart) + b * p->rmax * R;
    }
    __device__ float* vfull() const { return reinterpret_cast<float*>(base + p->off_vfull); }
    __device__ float* red() const { return reinterpret_cast<float*>(base + p->off_red); }
    __device__ uint8_t* xs() const { return base + p->off_xs; }
    __device__ uint8_t* ys() const { return base + p->off_ys; }
  };

  // ------------------------------------------------------------------ producer warp ----
  __device__ static void producer(const Params& p, const Smem& sm, const Waiter& w,
                                  const int* starts, const int* adapters, const int* base,
                                  int q, int G, int n_my, int crank, int k0, int n0,
                                  const Chunking<T, R>& ch) {
    const int lane = threadIdx.x & 31;
    const uint64_t pol_w = policy_evict_first();  // weights: streamed once per call
    const uint64_t pol_a = policy_evict_last();   // activations: reused by the C CTAs
    const int NST = p.nstages;
    uint32_t g = 0;  // ring chunk counter
    for (int li = 0; li < n_my; ++li) {
      const int t = q + li * G;
      int* d = sm.desc(li & 1);
      decode_item(p, t, starts, adapters, base, d);
      if (lane == 0) mbar_arrive(sm.fixed(kDesc0 + (li & 1)));
      const int k = d[0];
      const int nrow = min(max(d[1], 0), p.rmax);
      const T* Ak = nullptr;
      const T* Bk = nullptr;
      if (MODE != kExpand) {
        Ak = static_cast<const T*>(p.A_ptrs[k]) + static_cast<size_t>(p.layer) * p.h_in * R;
      }
      if (MODE != kShrink) {
        Bk = static_cast<const T*>(p.B_ptrs[k]) + static_cast<size_t>(p.layer) * R * p.h_out;
      }
      // ---- x rows (shrink, fused) or v rows (expand) into xs
      if (li > 0 && lane == 0) w.wait<false>(sm.fixed(kXFree), (li - 1) & 1);
      __syncwarp();
      {
        const uint32_t row_bytes = (MODE == kExpand) ? R * 4u : ch.kc * kEb;
        if (lane == 0) mbar_arrive_expect_tx(sm.fixed(kXFull), w.ok() ? nrow * row_bytes : 0u);
        __syncwarp();
        for (int i = lane; i < nrow && row_bytes > 0 && w.ok(); i += 32) {
          const int row = d[2 + i];
          const void* src = (MODE == kExpand)
                                ? static_cast<const void*>(p.v_in + static_cast<size_t>(row) * R)
                                : static_cast<const void*>(static_cast<const T*>(p.x) +
                                                           static_cast<size_t>(row) * p.h_in + k0);
          bulk_g2s(smem_addr(sm.xs() + i * p.xs_row_bytes), src, row_bytes, sm.fixed(kXFull),
                   pol_a);
        }
      }
      // ---- A chunks
      if (MODE != kExpand) {
        for (int j = 0; j < ch.nA; ++j, ++g) {
          const int s = g % NST;
          if (lane == 0) {
            if (g >= (uint32_t)NST) w.wait<false>(sm.empty(s), ((g / NST) - 1) & 1);
            const int rows = min(ch.kb, ch.kc - j * ch.kb);
            const uint32_t bytes = rows * R * kEb;
            mbar_arrive_expect_tx(sm.full(s), w.ok() ? bytes : 0u);
            if (w.ok())
              bulk_g2s(smem_addr(sm.stage(s)), Ak + static_cast<size_t>(k0 + j * ch.kb) * R,
                       bytes, sm.full(s), pol_w);
          }
        }
      }
      // ---- y rows
      if (MODE != kShrink) {
        if (li > 0 && lane == 0) w.wait<false>(sm.fixed(kYFree), (li - 1) & 1);
        __syncwarp();
        const uint32_t row_bytes = ch.nc * kEb;
        if (lane == 0) mbar_arrive_expect_tx(sm.fixed(kYFull), w.ok() ? nrow * row_bytes : 0u);
        __syncwarp();
        for (int i = lane; i < nrow && row_bytes > 0 && w.ok(); i += 32) {
          const int row = d[2 + i];
          bulk_g2s(smem_addr(sm.ys() + i * p.ys_row_bytes),
                   static_cast<const T*>(p.y) + static_cast<size_t>(row) * p.h_out + n0,
                   row_bytes, sm.fixed(kYFull), pol_a);
        }
        // ---- B chunks: pass by pass, `cb` rows of the pass's column window per chunk
        for (int pass = 0; pass < ch.passes; ++pass) {
          const int wdt = ch.pass_width(p, pass);
          const int cb = ch.pass_rows(p, wdt);
          const int stride = Chunking<T, R>::row_stride(wdt);
          for (int c0 = 0; c0 < R; c0 += cb, ++g) {
            const int s = g % NST;
            const int rows = min(cb, R - c0);
            if (lane == 0) {
              if (g >= (uint32_t)NST) w.wait<false>(sm.empty(s), ((g / NST) - 1) & 1);
              mbar_arrive_expect_tx(sm.full(s), w.ok() ? rows * wdt * kEb : 0u);
            }
            __syncwarp();
            for (int rr = lane; rr < rows && w.ok(); rr += 32) {
              bulk_g2s(smem_addr(sm.stage(s) + rr * stride),
                       Bk + static_cast<size_t>(c0 + rr) * p.h_out + n0 + pass * p.wmax,
                       wdt * kEb, sm.full(s), pol_w);
            }
            __syncwarp();
          }
        }
      }
    }
  }

  // --------------------------------------------------------------- consumer warps ----
  template <int RB>
  __device__ static void consume_item(const Params& p, const Smem& sm, const Waiter& w,
                                      int li, uint32_t& g, const int* d, int nrow, int crank,
                                      int k0, int n0, const Chunking<T, R>& ch) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NST = p.nstages;
    float acc[RB][kVec];
    float* vfull = sm.vfull();

    if (MODE != kExpand) {
      // ----------------------------------------------------------- shrink (split-K)
#pragma unroll
      for (int i = 0; i < RB; ++i)
#pragma unroll
        for (int j = 0; j < kVec; ++j) acc[i][j] = 0.f;
      w.wait<false>(sm.fixed(kXFull), li & 1);
      const int cc = tid % kCpr, kl = tid / kCpr;
      const uint8_t* xs = sm.xs();
      const int xs_row = p.xs_row_bytes;
      for (int j = 0; j < ch.nA; ++j, ++g) {
        const int s = g % NST;
        w.wait<false>(sm.full(s), (g / NST) & 1);
        const int kr0 = j * ch.kb;
        const int rows = min(ch.kb, ch.kc - kr0);
        const uint8_t* st = sm.stage(s);
        for (int kk = kl; kk < rows; kk += kKLanes) {
          float a[kVec];
          E::load16(st + (kk * R + cc * kVec) * kEb, a);
#pragma unroll
          for (int i = 0; i < RB; ++i) {
            const float xv = E::load1(xs + i * xs_row + (kr0 + kk) * kEb);
#pragma unroll
            for (int e = 0; e < kVec; ++e) acc[i][e] = fmaf(xv, a[e], acc[i][e]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty(s));
      }
      if (MODE == kFused) {  // xs is no longer read (shrink-only releases it after writing v,
        __syncwarp();        // since the producer may rewrite this descriptor after that)
        if (lane == 0) mbar_arrive(sm.fixed(kXFree));
      }
      // reduce over the k-lanes of the warp (lanes with equal cc), then over warps
#pragma unroll
      for (int o = kCpr; o < 32; o <<= 1)
#pragma unroll
        for (int i = 0; i < RB; ++i)
#pragma unroll
          for (int e = 0; e < kVec; ++e) acc[i][e] += __shfl_xor_sync(0xffffffffu, acc[i][e], o);
      float* red = sm.red();
      if (lane < kCpr) {
#pragma unroll
        for (int i = 0; i < RB; ++i)
#pragma unroll
          for (int e = 0; e < kVec; ++e)
            red[(warp * p.rmax + i) * R + lane * kVec + e] = acc[i][e];
      }
      named_bar(1, kConsumers);
      float* vp = sm.vpart(li & 1);
      for (int t = tid; t < RB * R; t += kConsumers) {
        const int i = t / R, c = t % R;
        float s = 0.f;
#pragma unroll
        for (int ww = 0; ww < kConsumerWarps; ++ww) s += red[(ww * p.rmax + i) * R + c];
        vp[i * R + c] = s;
      }
      named_bar(1, kConsumers);
      // ----------------------------------------------------- cluster all-reduce of v
      const uint32_t vready = sm.fixed(kVReady0 + (li & 1));
      if (tid == 0) {
        fence_acq_rel_cluster();
        for (int c = 0; c < p.C; ++c) mbar_arrive_remote(vready, c);
      }
      w.wait<true>(vready, (li >> 1) & 1);
      const uint32_t vp_addr = smem_addr(vp);
      for (int t = tid; t < nrow * R; t += kConsumers) {
        float s = 0.f;
        for (int c = 0; c < p.C; ++c) s += ld_cluster_f32(cluster_map(vp_addr + 4u * t, c));
        if (MODE == kFused) {
          vfull[t] = s * p.scale;
        } else {  // shrink: CTA (row mod C) writes the row
          const int i = t / R;
          if ((i % p.C) == crank && w.ok())
            p.v_out[static_cast<size_t>(d[2 + i]) * R + (t % R)] = s;
        }
      }
      named_bar(1, kConsumers);
      if (MODE == kShrink) {
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.fixed(kXFree));
      }
    } else {
      // ------------------------------------------------------------- expand only
      w.wait<false>(sm.fixed(kXFull), li & 1);
      for (int t = tid; t < nrow * R; t += kConsumers) {
        const int i = t / R, c = t % R;
        vfull[t] = p.scale * reinterpret_cast<const float*>(sm.xs() + i * p.xs_row_bytes)[c];
      }
      named_bar(1, kConsumers);
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.fixed(kXFree));
    }

    if (MODE != kShrink) {
      // ------------------------------------------------------- expand over the N slice
      bool y_ready = false;
      for (int pass = 0; pass < ch.passes; ++pass) {
        const int wdt = ch.pass_width(p, pass);
        const int cb = ch.pass_rows(p, wdt);
        const int stride = Chunking<T, R>::row_stride(wdt);
        const int nch = wdt / kVec;
        int cl_n = 1;
        while (cl_n < 32 && nch * cl_n * 2 <= kConsumers) cl_n <<= 1;
        const int my_ch = tid / cl_n, cl = tid % cl_n;
        const bool active = my_ch < nch;
#pragma unroll
        for (int i = 0; i < RB; ++i)
#pragma unroll
          for (int e = 0; e < kVec; ++e) acc[i][e] = 0.f;
        for (int c0 = 0; c0 < R; c0 += cb, ++g) {
          const int s = g % NST;
          const int rows = min(cb, R - c0);
          w.wait<false>(sm.full(s), (g / NST) & 1);
          if (active) {
            const uint8_t* st = sm.stage(s) + my_ch * 16;
            for (int c = cl; c < rows; c += cl_n) {
              float b[kVec];
              E::load16(st + c * stride, b);
#pragma unroll
              for (int i = 0; i < RB; ++i) {
                const float vv = vfull[i * R + c0 + c];
#pragma unroll
                for (int e = 0; e < kVec; ++e) acc[i][e] = fmaf(vv, b[e], acc[i][e]);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(sm.empty(s));
        }
        for (int o = 1; o < cl_n; o <<= 1)
#pragma unroll
          for (int i = 0; i < RB; ++i)
#pragma unroll
            for (int e = 0; e < kVec; ++e) acc[i][e] += __shfl_xor_sync(0xffffffffu, acc[i][e], o);
        if (!y_ready) {
          w.wait<false>(sm.fixed(kYFull), li & 1);
          y_ready = true;
        }
        if (active && cl == 0 && w.ok()) {
          const int col = pass * p.wmax + my_ch * kVec;
#pragma unroll
          for (int i = 0; i < RB; ++i) {
            if (i < nrow) {
              float yo[kVec];
              E::load16(sm.ys() + i * p.ys_row_bytes + col * kEb, yo);
#pragma unroll
              for (int e = 0; e < kVec; ++e) yo[e] += acc[i][e];
              E::store16(static_cast<T*>(p.y) + static_cast<size_t>(d[2 + i]) * p.h_out + n0 + col,
                         yo);
            }
          }
        }
      }
      if (!y_ready) w.wait<false>(sm.fixed(kYFull), li & 1);
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.fixed(kYFree));
    }
  }

  __device__ static void consumer(const Params& p, const Smem& sm, const Waiter& w, int n_my,
                                  int crank, int k0, int n0, const Chunking<T, R>& ch) {
    uint32_t g = 0;
    for (int li = 0; li < n_my; ++li) {
      w.wait<false>(sm.fixed(kDesc0 + (li & 1)), (li >> 1) & 1);
      const int* d = sm.desc(li & 1);
      const int nrow = min(max(d[1], 0), p.rmax);
      if (nrow <= 1)
        consume_item<1>(p, sm, w, li, g, d, nrow, crank, k0, n0, ch);
      else if (nrow <= 2)
        consume_item<2>(p, sm, w, li, g, d, nrow, crank, k0, n0, ch);
      else if (nrow <= 4)
        consume_item<4>(p, sm, w, li, g, d, nrow, crank, k0, n0, ch);
      else
        consume_item<8>(p, sm, w, li, g, d, nrow, crank, k0, n0, ch);
    }
  }

  __device__ static void run(const Params& p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Smem sm{smem, &p};
    const int tid = threadIdx.x, warp = tid >> 5;
    const int C = p.C;
    const int crank = static_cast<int>(blockIdx.x) % C;
    const int q = static_cast<int>(blockIdx.x) / C;
    const int G = static_cast<int>(gridDim.x) / C;
    int* ctl = reinterpret_cast<int*>(smem + p.off_ctl);
    int* starts = reinterpret_cast<int*>(smem + p.off_tab);
    int* adapters = starts + (p.S + 1);
    int* base = adapters + p.S;

    if (tid == 0) {
      for (int s = 0; s < p.nstages; ++s) {
        mbar_init(sm.full(s), 1);
        mbar_init(sm.empty(s), kConsumerWarps);
      }
      mbar_init(sm.fixed(kXFull), 1);
      mbar_init(sm.fixed(kXFree), kConsumerWarps);
      mbar_init(sm.fixed(kYFull), 1);
      mbar_init(sm.fixed(kYFree), kConsumerWarps);
      mbar_init(sm.fixed(kDesc0), 1);
      mbar_init(sm.fixed(kDesc1), 1);
      mbar_init(sm.fixed(kVReady0), C);
      mbar_init(sm.fixed(kVReady1), C);
      mbar_init(sm.fixed(kNever), 1);
      ctl[0] = 0;
      fence_mbar_init();
    }
    build_schedule(p, starts, adapters, base, reinterpret_cast<int*>(smem + p.off_ring),
                   ctl + 4);
    fence_proxy_async();  // the ring held the hash table: order before bulk copies land
    __syncthreads();
    if (MODE != kExpand) cluster_sync_all();  // peers' barriers are initialised

    const Waiter w{reinterpret_cast<volatile int*>(ctl), p.err, p.wait_limit_ns};
    if (p.inject_stall) w.wait<false>(sm.fixed(kNever), 0);  // nothing completes it

    const int n_items = base[p.S];
    const int n_my = (q < n_items) ? (n_items - q + G - 1) / G : 0;
    int k0 = 0, k1 = 0, n0 = 0, n1 = 0;
    slice_of(p.h_in, C, crank, k0, k1);
    slice_of(p.h_out, C, crank, n0, n1);
    Chunking<T, R> ch;
    ch.init(p, MODE == kExpand ? 0 : k1 - k0, MODE == kShrink ? 0 : n1 - n0);

    if (warp == kConsumerWarps) {
      producer(p, sm, w, starts, adapters, base, q, G, n_my, crank, k0, n0, ch);
    } else {
      consumer(p, sm, w, n_my, crank, k0, n0, ch);
    }
    __syncthreads();
    if (!w.ok()) {  // gave up: let every bulk copy already issued land before the CTA exits
      const uint64_t t0 = now_ns();
      while (now_ns() - t0 < 200000ull) __nanosleep(1000);
    }
    if (MODE != kExpand) cluster_sync_all();  // no CTA leaves while peers read its smem
  }
};

template <typename T, int R, int MODE>
__global__ void __launch_bounds__(kThreads, 2) sgmv_kernel(const __grid_constant__ Params p) {
  Kernel<T, R, MODE>::run(p);
}

}  // namespace sgmv
